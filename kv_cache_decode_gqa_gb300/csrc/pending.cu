// Launchers whose kernels are not compiled into this build yet: each reports
// cudaErrorNotSupported, which the C ABI turns into KVD_ERR_UNSUPPORTED.
#include "kvd_internal.h"

namespace kvd {
cudaError_t launch_indexer_scores(const IndexerParams &, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t launch_topk(const IndexerParams &, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace kvd
