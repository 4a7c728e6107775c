// gdn_noalloc.cu -- gdn_prefill_noalloc: the chunked prefill for callers that
// cannot hand the library a device workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// layer: a step running under a strict memory budget, an allocator that
// forbids new device allocations after start-up, a host framework that gives
// the layer no allocation hook.  This entry point
// takes the same inputs and outputs as gdn_prefill but no workspace: its
// scratch (the device status word and the device-built segment list) lives in
// one file-scope device array of GDN_NOALLOC_SCRATCH_BYTES bytes, which every
// GPU that loads the library holds until the process exits.
//
// Nothing here allocates: no cudaMalloc, no cudaFree, no allocating library
// routine.  The array's device address is looked up with cudaGetSymbolAddress
// once per context (its name is only a host-side stand-in in host code).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_trace.h"
#include "gdn_launch.h"

namespace {

constexpr size_t kScratchBytes = GDN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// status word (256 B) + the unsplit work lists for up to GDN_NOALLOC_MAX_SEQS sequences
static __device__ __align__(256) unsigned char g_prefill_scratch[kScratchBytes];

static_assert(256 + 256 + ((16 + 32 * (size_t)GDN_NOALLOC_MAX_SEQS + 255) / 256) * 256 <= kScratchBytes,
              "the fixed scratch must hold the work list of GDN_NOALLOC_MAX_SEQS sequences");

std::mutex g_mu;
struct ScratchCache {
  unsigned long long ctx_id = 0;   // the context the address belongs to (0: none yet)
  void* addr = nullptr;
};
ScratchCache g_cache[kMaxDevices];

using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);

// Id of the calling thread's current context (0 if there is none or the
// driver cannot say).
unsigned long long current_context_id() {
  static PfnCtxGetCurrent get_current = nullptr;
  static PfnCtxGetId get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PfnCtxGetCurrent>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PfnCtxGetId>(f);
    looked_up = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_prefill_scratch in the current context.  It is looked
// up with cudaGetSymbolAddress on the first call in a context and cached
// under the context's id, so a context that was rebuilt (after a
// cudaDeviceReset, say) gets the address of its own copy of the array.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchCache& c = g_cache[dev];
  const unsigned long long id = current_context_id();
  if (c.addr == nullptr || id == 0 || id != c.ctx_id) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_prefill_scratch);   // also makes the primary context current
    if (e != cudaSuccess) return e;
    c.addr = addr;
    c.ctx_id = current_context_id();
  }
  *out = c.addr;
  return cudaSuccess;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" gdn_status gdn_prefill_noalloc(const gdn_dims* d, const void* qkv, const void* z,
                                          const void* a, const void* b, const float* A_log,
                                          const float* dt_bias, const void* conv_w,
                                          const float* norm_w, const int32_t* cu_seqlens,
                                          int n_seqs, long long total_tokens, float* conv_state,
                                          float* ssm_state, void* out, int32_t* device_status,
                                          void* stream) {
  gdn::TraceRange trace_range("gdn_prefill_noalloc");
  if (!d) return GDN_ERR_INVALID_ARG;
  if (d->h_k <= 0 || d->h_v <= 0 || d->h_v % d->h_k != 0 || d->d_k <= 0 || d->d_v <= 0 ||
      d->conv_w <= 0 || d->chunk <= 0 || !(d->l2_eps >= 0.0f) || !(d->rms_eps >= 0.0f) ||
      !isfinite(d->l2_eps) || !isfinite(d->rms_eps))
    return GDN_ERR_INVALID_ARG;
  const int G = d->h_v / d->h_k;
  if (d->d_k != gdn::kD || d->d_v != gdn::kD || d->conv_w != gdn::kConvW || d->chunk != gdn::kChunk ||
      !(G == 1 || G == 2 || G == 4) || d->h_k > 64)
    return GDN_ERR_UNSUPPORTED;
  if (n_seqs < 0 || total_tokens < 0 || total_tokens > (1LL << 31) - 1) return GDN_ERR_INVALID_ARG;
  if (n_seqs > GDN_NOALLOC_MAX_SEQS) return GDN_ERR_UNSUPPORTED;   // the fixed scratch holds no more
  if (n_seqs == 0 || total_tokens == 0) return GDN_OK;
  if (!aligned16(qkv) || !aligned16(z) || !aligned16(a) || !aligned16(b) || !aligned16(A_log) ||
      !aligned16(dt_bias) || !aligned16(conv_w) || !aligned16(norm_w) || !aligned16(cu_seqlens) ||
      !aligned16(conv_state) || !aligned16(ssm_state) || !aligned16(out))
    return GDN_ERR_INVALID_ARG;
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u)) return GDN_ERR_INVALID_ARG;
  const size_t need = 256 + gdn::prefill_scratch_bytes_unsplit(n_seqs);
  if (need > kScratchBytes) return GDN_ERR_UNSUPPORTED;

  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return GDN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  gdn::PrefillArgs p;
  p.qkv = static_cast<const uint16_t*>(qkv);
  p.z = static_cast<const uint16_t*>(z);
  p.a = static_cast<const uint16_t*>(a);
  p.b = static_cast<const uint16_t*>(b);
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.conv_w = static_cast<const uint16_t*>(conv_w);
  p.norm_w = norm_w;
  p.cu_seqlens = cu_seqlens;
  p.conv_state = conv_state;
  p.ssm_state = ssm_state;
  p.out = static_cast<uint16_t*>(out);
  p.status = static_cast<int32_t*>(scratch);
  p.scratch = static_cast<char*>(scratch) + 256;
  p.scratch_bytes = kScratchBytes - 256;
  p.n_seqs = n_seqs;
  p.h_k = d->h_k;
  p.h_v = d->h_v;
  p.total_tokens = total_tokens;
  p.l2_eps = d->l2_eps;
  p.rms_eps = d->rms_eps;
  // the array keeps the previous call's contents: only the status word must
  // start at zero (the work lists are rewritten in full by the call)
  if (cudaMemsetAsync(scratch, 0, 256, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (gdn::launch_prefill(p, s, /*allow_split=*/false) != cudaSuccess) return GDN_ERR_CUDA;
  if (device_status &&
      cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}
