// Indexer kernel instantiations: bf16 topk (see indexer_kernel.cuh).
#include "indexer_kernel.cuh"

namespace dsa {

DSA_INDEXER_VARIANT(bf16_topk, false, true)

}  // namespace dsa
