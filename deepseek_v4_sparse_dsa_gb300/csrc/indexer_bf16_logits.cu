// Indexer kernel instantiations: bf16 logits (see indexer_kernel.cuh).
#include "indexer_kernel.cuh"

namespace dsa {

DSA_INDEXER_VARIANT(bf16_logits, false, false)

}  // namespace dsa
