// Indexer kernel instantiations: fp8 topk (see indexer_kernel.cuh).
#include "indexer_kernel.cuh"

namespace dsa {

DSA_INDEXER_VARIANT(fp8_topk, true, true)

}  // namespace dsa
