// Indexer kernel instantiations: fp8 logits (see indexer_kernel.cuh).
#include "indexer_kernel.cuh"

namespace dsa {

DSA_INDEXER_VARIANT(fp8_logits, true, false)

}  // namespace dsa
