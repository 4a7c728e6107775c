// gdn_prefill.cu -- chunked prefill (work in progress).
#include "gdn_common.cuh"
#include "gdn_launch.h"
namespace gdn {
size_t prefill_scratch_bytes(int, int, int, long long) { return 0; }
cudaError_t launch_prefill(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace gdn
