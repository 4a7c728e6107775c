// gdn_api.cu -- the extern "C" surface of libgdn: validation and launch.
//
// Every entry point validates its arguments on the host before it touches
// the device; on any failure it returns a status and launches nothing.
// Checks that need device data (cu_seqlens contents, slot indices) run in
// the kernels and report through a device status word.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <new>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_trace.h"
#include "gdn_launch.h"

namespace {

constexpr int kVersion = 310;  // 0.3.1: the decode step from host buffers

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool ptr_ok(const void* p) { return p != nullptr && aligned16(p); }

// Shape sanity (INVALID_ARG) first, then the compiled fast path (UNSUPPORTED).
gdn_status check_dims(const gdn_dims* d) {
  if (!d) return GDN_ERR_INVALID_ARG;
  if (d->h_k <= 0 || d->h_v <= 0 || d->h_v % d->h_k != 0 || d->d_k <= 0 ||
      d->d_v <= 0 || d->conv_w <= 0 || d->chunk <= 0)
    return GDN_ERR_INVALID_ARG;
  if (!(d->l2_eps >= 0.0f) || !(d->rms_eps >= 0.0f) || !isfinite(d->l2_eps) ||
      !isfinite(d->rms_eps))
    return GDN_ERR_INVALID_ARG;
  const int G = d->h_v / d->h_k;
  if (d->d_k != gdn::kD || d->d_v != gdn::kD || d->conv_w != gdn::kConvW ||
      d->chunk != gdn::kChunk || !(G == 1 || G == 2 || G == 4) || d->h_k > 64)
    return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

long long channels(const gdn_dims* d) {
  return 2LL * d->h_k * d->d_k + (long long)d->h_v * d->d_v;
}

}  // namespace

extern "C" {

int gdn_version(void) { return kVersion; }

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: null or misaligned pointer, bad size or inconsistent dims";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: dims outside the compiled fast path (d_k = d_v = 128, conv_w = 4, chunk = 64, h_v/h_k in {1,2,4}, h_k <= 64)";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing or smaller than gdn_workspace_bytes()";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA runtime call failed";
    case GDN_ERR_DEVICE_TIMEOUT: return "GDN_ERR_DEVICE_TIMEOUT: a bounded device-side wait gave up";
    case GDN_ERR_DEVICE_BOUNDS: return "GDN_ERR_DEVICE_BOUNDS: cu_seqlens or a slot index out of range";
  }
  return "unknown gdn_status";
}

size_t gdn_state_bytes(const gdn_dims* d) {
  if (!d || d->h_k <= 0 || d->h_v <= 0 || d->d_k <= 0 || d->d_v <= 0 || d->conv_w <= 0 ||
      d->h_v % d->h_k != 0)
    return 0;
  const size_t ssm = (size_t)d->h_v * d->d_v * d->d_k * sizeof(float);
  const size_t conv = (size_t)(d->conv_w - 1) * (size_t)channels(d) * sizeof(float);
  return ssm + conv;
}

size_t gdn_workspace_bytes(const gdn_dims* d, int n_seqs, long long total_tokens) {
  if (check_dims(d) != GDN_OK || n_seqs < 0 || total_tokens < 0) return 0;
  return 256 + gdn::prefill_scratch_bytes(n_seqs, d->h_k, d->h_v, total_tokens);
}

long long gdn_prefill_segment_tokens(const gdn_dims* d, int n_seqs, long long total_tokens) {
  if (check_dims(d) != GDN_OK || n_seqs < 0 || total_tokens < 0) return -1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  return gdn::prefill_segment_tokens(n_seqs, d->h_v, total_tokens, sms);
}

long long gdn_prefill_segment_tokens_for(const gdn_dims* d, int n_seqs, long long total_tokens,
                                         int sms) {
  if (check_dims(d) != GDN_OK || n_seqs < 0 || total_tokens < 0 || sms <= 0) return -1;
  return gdn::prefill_segment_tokens(n_seqs, d->h_v, total_tokens, sms);
}

gdn_status gdn_prefill(const gdn_dims* dims, const void* qkv, const void* z, const void* a,
                       const void* b, const float* A_log, const float* dt_bias,
                       const void* conv_w, const float* norm_w, const int32_t* cu_seqlens,
                       int n_seqs, long long total_tokens, float* conv_state,
                       float* ssm_state, void* out, void* workspace, size_t workspace_bytes,
                       void* stream) {
  gdn::TraceRange trace_range("gdn_prefill");
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (n_seqs < 0 || total_tokens < 0 || total_tokens > (1LL << 31) - 1)
    return GDN_ERR_INVALID_ARG;
  if (n_seqs == 0 || total_tokens == 0) return GDN_OK;
  if (!ptr_ok(qkv) || !ptr_ok(z) || !ptr_ok(a) || !ptr_ok(b) || !ptr_ok(A_log) ||
      !ptr_ok(dt_bias) || !ptr_ok(conv_w) || !ptr_ok(norm_w) || !ptr_ok(cu_seqlens) ||
      !ptr_ok(conv_state) || !ptr_ok(ssm_state) || !ptr_ok(out))
    return GDN_ERR_INVALID_ARG;
  const size_t need = gdn_workspace_bytes(dims, n_seqs, total_tokens);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return GDN_ERR_WORKSPACE;

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
  p.status = static_cast<int32_t*>(workspace);
  p.scratch = static_cast<char*>(workspace) + 256;
  p.scratch_bytes = workspace_bytes - 256;
  p.n_seqs = n_seqs;
  p.h_k = dims->h_k;
  p.h_v = dims->h_v;
  p.total_tokens = total_tokens;
  p.l2_eps = dims->l2_eps;
  p.rms_eps = dims->rms_eps;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, 256, s) != cudaSuccess) return GDN_ERR_CUDA;
  return gdn::launch_prefill(p, s) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // extern "C"

namespace {

// Host checks shared by the decode entry points; fills p on success.  `steps`
// tokens per sequence per launch (1 for the single step).
gdn_status decode_args(const gdn_dims* dims, const void* qkv, const void* z, const void* a,
                       const void* b, const float* A_log, const float* dt_bias,
                       const void* conv_w, const float* norm_w, const int32_t* slot, int n_slots,
                       int batch, int steps, float* conv_state, float* ssm_state, void* out,
                       int out_dtype, float* ssm_trace, float* conv_trace,
                       int32_t* device_status, gdn::DecodeArgs& p) {
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (batch < 0 || n_slots < 0 || steps < 1 || steps > GDN_DECODE_MAX_STEPS ||
      (out_dtype != GDN_DTYPE_BF16 && out_dtype != GDN_DTYPE_F32))
    return GDN_ERR_INVALID_ARG;
  if ((long long)batch * dims->h_k > 0x7fffffffLL || (long long)batch * steps > 0x7fffffffLL)
    return GDN_ERR_INVALID_ARG;
  if (batch > 0 && (n_slots < 1 || (!slot && n_slots < batch))) return GDN_ERR_INVALID_ARG;
  if (batch > 0 && (!ptr_ok(qkv) || !ptr_ok(z) || !ptr_ok(a) || !ptr_ok(b) || !ptr_ok(A_log) ||
                    !ptr_ok(dt_bias) || !ptr_ok(conv_w) || !ptr_ok(norm_w) ||
                    !ptr_ok(conv_state) || !ptr_ok(ssm_state) || !ptr_ok(out)))
    return GDN_ERR_INVALID_ARG;
  if ((slot && !aligned16(slot)) || (ssm_trace && !aligned16(ssm_trace)) ||
      (conv_trace && !aligned16(conv_trace)))
    return GDN_ERR_INVALID_ARG;
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u))
    return GDN_ERR_INVALID_ARG;
  p.qkv = static_cast<const uint16_t*>(qkv);
  p.z = static_cast<const uint16_t*>(z);
  p.a = static_cast<const uint16_t*>(a);
  p.b = static_cast<const uint16_t*>(b);
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.conv_w = static_cast<const uint16_t*>(conv_w);
  p.norm_w = norm_w;
  p.slot = slot;
  p.conv_state = conv_state;
  p.ssm_state = ssm_state;
  p.out = out;
  p.status = device_status;
  p.n_slots = n_slots;
  p.batch = batch;
  p.h_k = dims->h_k;
  p.h_v = dims->h_v;
  p.l2_eps = dims->l2_eps;
  p.rms_eps = dims->rms_eps;
  p.steps = steps;
  p.ssm_trace = ssm_trace;
  p.conv_trace = conv_trace;
  return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status gdn_decode_step(const gdn_dims* dims, const void* qkv, const void* z,
                           const void* a, const void* b, const float* A_log,
                           const float* dt_bias, const void* conv_w, const float* norm_w,
                           const int32_t* slot, int n_slots, int batch, float* conv_state,
                           float* ssm_state, void* out, int out_dtype,
                           int32_t* device_status, void* stream) {
  gdn::TraceRange trace_range("gdn_decode_step");
  gdn::DecodeArgs p;
  const gdn_status st = decode_args(dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, slot,
                                    n_slots, batch, 1, conv_state, ssm_state, out, out_dtype,
                                    nullptr, nullptr, device_status, p);
  if (st != GDN_OK || batch == 0) return st;
  return gdn::launch_decode(p, out_dtype == GDN_DTYPE_F32, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

static_assert(GDN_DECODE_MAX_STEPS == gdn::kDecodeMaxSteps, "the header's token limit is the kernel's");

gdn_status gdn_decode_multi(const gdn_dims* dims, const void* qkv, const void* z, const void* a,
                            const void* b, const float* A_log, const float* dt_bias,
                            const void* conv_w, const float* norm_w, const int32_t* slot,
                            int n_slots, int batch, int steps, float* conv_state, float* ssm_state,
                            void* out, int out_dtype, float* ssm_trace, float* conv_trace,
                            int32_t* device_status, void* stream) {
  gdn::TraceRange trace_range("gdn_decode_multi");
  gdn::DecodeArgs p;
  const gdn_status st = decode_args(dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, slot,
                                    n_slots, batch, steps, conv_state, ssm_state, out, out_dtype,
                                    ssm_trace, conv_trace, device_status, p);
  if (st != GDN_OK || batch == 0) return st;
  return gdn::launch_decode_multi(p, out_dtype == GDN_DTYPE_F32, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

}  // extern "C"

namespace {

// The device staging area of gdn_decode_step_host: the step's qkv, z, a, b and
// its output, each 256-byte aligned.
struct DecodeHostLayout {
  size_t qkv, z, a, b, out, total;
};
size_t round256(size_t x) { return (x + 255) & ~size_t(255); }
bool decode_host_layout(const gdn_dims* d, int batch, int out_dtype, DecodeHostLayout& l) {
  if (check_dims(d) != GDN_OK || batch < 0 || (out_dtype != GDN_DTYPE_BF16 && out_dtype != GDN_DTYPE_F32))
    return false;
  const size_t B = (size_t)(batch > 0 ? batch : 1);
  const size_t cc = 2ull * d->h_k * d->d_k + (size_t)d->h_v * d->d_v, zv = (size_t)d->h_v * d->d_v;
  size_t off = 0;
  l.qkv = off; off = round256(off + B * cc * 2);
  l.z = off;   off = round256(off + B * zv * 2);
  l.a = off;   off = round256(off + B * d->h_v * 2);
  l.b = off;   off = round256(off + B * d->h_v * 2);
  l.out = off; off = round256(off + B * zv * (out_dtype == GDN_DTYPE_F32 ? 4 : 2));
  l.total = off;
  return true;
}

// The device address of `bytes` of page-locked host memory at p, or null when
// p is not page-locked host memory the device can address (pageable memory,
// device memory, null): both its first and its last byte must be.
const void* mapped_host(const void* p, size_t bytes) {
  if (!p || bytes == 0) return nullptr;
  cudaPointerAttributes first, last;
  if (cudaPointerGetAttributes(&first, p) != cudaSuccess ||
      cudaPointerGetAttributes(&last, static_cast<const char*>(p) + bytes - 1) != cudaSuccess) {
    cudaGetLastError();   // a refused query leaves no sticky error behind
    return nullptr;
  }
  if (first.type != cudaMemoryTypeHost || last.type != cudaMemoryTypeHost || !first.devicePointer ||
      !last.devicePointer ||
      static_cast<const char*>(last.devicePointer) - static_cast<const char*>(first.devicePointer) !=
          (ptrdiff_t)(bytes - 1))
    return nullptr;
  return first.devicePointer;
}

}  // namespace

extern "C" {

size_t gdn_decode_step_host_workspace_bytes(const gdn_dims* dims, int batch, int out_dtype) {
  DecodeHostLayout l;
  return decode_host_layout(dims, batch, out_dtype, l) ? l.total : 0;
}

gdn_status gdn_decode_step_host(const gdn_dims* dims, const void* qkv, const void* z, const void* a,
                                const void* b, const float* A_log, const float* dt_bias,
                                const void* conv_w, const float* norm_w, const int32_t* slot,
                                int n_slots, int batch, float* conv_state, float* ssm_state, void* out,
                                int out_dtype, int32_t* device_status, void* workspace,
                                size_t workspace_bytes, void* stream) {
  gdn::TraceRange trace_range("gdn_decode_step_host");
  DecodeHostLayout l;
  if (!decode_host_layout(dims, batch, out_dtype, l)) {
    const gdn_status st = check_dims(dims);
    return st != GDN_OK ? st : GDN_ERR_INVALID_ARG;
  }
  if (batch == 0) return GDN_OK;
  if (!qkv || !z || !a || !b || !out) return GDN_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < l.total)
    return GDN_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  // every argument checked, against the staging buffers, before anything is enqueued
  gdn::DecodeArgs p;
  const gdn_status st = decode_args(dims, ws + l.qkv, ws + l.z, ws + l.a, ws + l.b, A_log, dt_bias, conv_w,
                                    norm_w, slot, n_slots, batch, 1, conv_state, ssm_state, ws + l.out,
                                    out_dtype, nullptr, nullptr, device_status, p);
  if (st != GDN_OK) return st;
  const size_t B = (size_t)batch;
  const size_t cc = 2ull * dims->h_k * dims->d_k + (size_t)dims->h_v * dims->d_v;
  const size_t zv = (size_t)dims->h_v * dims->d_v, hv = (size_t)dims->h_v;
  const size_t out_bytes = B * zv * (out_dtype == GDN_DTYPE_F32 ? 4 : 2);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Page-locked buffers are read and written by the step's kernel in place, over
  // the host link: no staging copies, whose fixed cost per copy is several
  // microseconds.  Any other host memory goes through the staging area.
  const void* mq = mapped_host(qkv, B * cc * 2);
  const void* mz = mapped_host(z, B * zv * 2);
  const void* ma = mapped_host(a, B * hv * 2);
  const void* mb = mapped_host(b, B * hv * 2);
  void* mo = const_cast<void*>(mapped_host(out, out_bytes));
  if (mq && mz && ma && mb && mo && ((reinterpret_cast<uintptr_t>(mq) | reinterpret_cast<uintptr_t>(mz) |
                                      reinterpret_cast<uintptr_t>(ma) | reinterpret_cast<uintptr_t>(mb) |
                                      reinterpret_cast<uintptr_t>(mo)) & 15u) == 0) {
    p.qkv = static_cast<const uint16_t*>(mq);
    p.z = static_cast<const uint16_t*>(mz);
    p.a = static_cast<const uint16_t*>(ma);
    p.b = static_cast<const uint16_t*>(mb);
    p.out = mo;
    return gdn::launch_decode(p, out_dtype == GDN_DTYPE_F32, s) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  }
  if (cudaMemcpyAsync(ws + l.qkv, qkv, B * cc * 2, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(ws + l.z, z, B * zv * 2, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(ws + l.a, a, B * hv * 2, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(ws + l.b, b, B * hv * 2, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (gdn::launch_decode(p, out_dtype == GDN_DTYPE_F32, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaMemcpyAsync(out, ws + l.out, out_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

}  // extern "C"

// A captured chain of single decode steps: the graph and its executable form.
struct gdn_decode_graph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

extern "C" {

gdn_status gdn_decode_graph_create(const gdn_dims* dims, int steps, const void* qkv, const void* z,
                                   const void* a, const void* b, const float* A_log,
                                   const float* dt_bias, const void* conv_w, const float* norm_w,
                                   const int32_t* slot, int n_slots, int batch, float* conv_state,
                                   float* ssm_state, void* out, int out_dtype,
                                   int32_t* device_status, gdn_decode_graph** graph) {
  gdn::TraceRange trace_range("gdn_decode_graph_create");
  if (!graph) return GDN_ERR_INVALID_ARG;
  *graph = nullptr;
  if (steps < 1 || steps > (1 << 20) || batch < 1) return GDN_ERR_INVALID_ARG;
  gdn::DecodeArgs p;
  gdn_status st = decode_args(dims, qkv, z, a, b, A_log, dt_bias, conv_w, norm_w, slot, n_slots,
                              batch, 1, conv_state, ssm_state, out, out_dtype, nullptr, nullptr,
                              device_status, p);
  if (st != GDN_OK) return st;
  const bool f32 = out_dtype == GDN_DTYPE_F32;

  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return GDN_ERR_CUDA;
  cudaError_t err = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
  if (err != cudaSuccess) {
    cudaStreamDestroy(s);
    return GDN_ERR_CUDA;
  }
  // the whole chain as one persistent launch (the state rows stay on chip
  // through every step), then the conv state after the last step
  err = gdn::launch_decode_chain(p, steps, f32, s);
  if (err == cudaSuccess) err = gdn::launch_decode_chain_conv_state(p, p.qkv, steps, s);
  cudaGraph_t g = nullptr;
  const cudaError_t end = cudaStreamEndCapture(s, &g);
  cudaStreamDestroy(s);
  if (err != cudaSuccess || end != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return GDN_ERR_CUDA;
  }
  cudaGraphExec_t x = nullptr;
  if (cudaGraphInstantiate(&x, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    cudaGetLastError();
    return GDN_ERR_CUDA;
  }
  gdn_decode_graph* h = new (std::nothrow) gdn_decode_graph{g, x};
  if (!h) {
    cudaGraphExecDestroy(x);
    cudaGraphDestroy(g);
    return GDN_ERR_CUDA;
  }
  *graph = h;
  return GDN_OK;
}

gdn_status gdn_decode_graph_launch(gdn_decode_graph* graph, void* stream) {
  gdn::TraceRange trace_range("gdn_decode_graph_launch");
  if (!graph) return GDN_ERR_INVALID_ARG;
  return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

void gdn_decode_graph_destroy(gdn_decode_graph* graph) {
  if (!graph) return;
  cudaGraphExecDestroy(graph->exec);
  cudaGraphDestroy(graph->graph);
  delete graph;
}

}  // extern "C"

namespace {

gdn_status state_copy(const gdn_dims* dims, const float* src_conv, const float* src_ssm,
                      int src_slots, const int32_t* src_slot, float* dst_conv, float* dst_ssm,
                      int dst_slots, const int32_t* dst_slot, int n, int32_t* device_status,
                      void* stream) {
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (n < 0 || n > 65535) return GDN_ERR_INVALID_ARG;
  if (n == 0) return GDN_OK;
  const bool zero = src_ssm == nullptr;
  if (dst_slots < 1 || (!dst_slot && dst_slots < n)) return GDN_ERR_INVALID_ARG;
  if (!ptr_ok(dst_conv) || !ptr_ok(dst_ssm) || (dst_slot && !aligned16(dst_slot)))
    return GDN_ERR_INVALID_ARG;
  if (!zero) {
    if (src_slots < 1 || (!src_slot && src_slots < n)) return GDN_ERR_INVALID_ARG;
    if (!ptr_ok(src_conv) || !ptr_ok(src_ssm) || (src_slot && !aligned16(src_slot)))
      return GDN_ERR_INVALID_ARG;
  }
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u))
    return GDN_ERR_INVALID_ARG;
  gdn::StateCopyArgs p;
  p.src_conv = zero ? nullptr : src_conv;
  p.src_ssm = zero ? nullptr : src_ssm;
  p.src_idx = zero ? nullptr : src_slot;
  p.dst_conv = dst_conv;
  p.dst_ssm = dst_ssm;
  p.dst_idx = dst_slot;
  p.status = device_status;
  p.conv_floats = (long long)(dims->conv_w - 1) * channels(dims);
  p.ssm_floats = (long long)dims->h_v * dims->d_v * dims->d_k;
  p.src_slots = zero ? 0 : src_slots;
  p.dst_slots = dst_slots;
  p.n = n;
  return gdn::launch_state_copy(p, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

}  // namespace

extern "C" {

gdn_status gdn_state_copy(const gdn_dims* dims, const float* src_conv_state,
                          const float* src_ssm_state, int src_slots, const int32_t* src_slot,
                          float* dst_conv_state, float* dst_ssm_state, int dst_slots,
                          const int32_t* dst_slot, int n, int32_t* device_status, void* stream) {
  gdn::TraceRange trace_range("gdn_state_copy");
  if (!src_conv_state || !src_ssm_state) return GDN_ERR_INVALID_ARG;
  return state_copy(dims, src_conv_state, src_ssm_state, src_slots, src_slot, dst_conv_state,
                    dst_ssm_state, dst_slots, dst_slot, n, device_status, stream);
}

gdn_status gdn_state_reset(const gdn_dims* dims, float* conv_state, float* ssm_state, int n_slots,
                           const int32_t* slot, int n, int32_t* device_status, void* stream) {
  gdn::TraceRange trace_range("gdn_state_reset");
  return state_copy(dims, nullptr, nullptr, 0, nullptr, conv_state, ssm_state, n_slots, slot, n,
                    device_status, stream);
}

gdn_status gdn_read_device_status(const void* status_word, void* stream, int32_t* code) {
  gdn::TraceRange trace_range("gdn_read_device_status");
  if (!status_word || !code || (reinterpret_cast<uintptr_t>(status_word) & 3u))
    return GDN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, status_word, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  *code = v;
  return GDN_OK;
}

}  // extern "C"

// ---- the dense projections around the layer ----
namespace {

// The checks both projections share: dims as every call, a hidden size the
// GEMM's K-blocks and stores handle, h_v a multiple of 8 (the a and b column
// runs of the input projection are 16-byte stores), and an int-sized problem.
gdn_status check_proj(const gdn_dims* d, int hidden, long long tokens, int32_t* device_status) {
  gdn_status st = check_dims(d);
  if (st != GDN_OK) return st;
  if (hidden <= 0 || tokens < 0 || tokens > (1LL << 31) - 1) return GDN_ERR_INVALID_ARG;
  if (hidden % 64 != 0 || hidden > 65536 || d->h_v % 8 != 0) return GDN_ERR_UNSUPPORTED;
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u)) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status gdn_in_proj(const gdn_dims* dims, int hidden, long long tokens, const void* x,
                       const void* w_in, void* qkv, void* z, void* a, void* b,
                       int32_t* device_status, void* stream) {
  gdn::TraceRange trace_range("gdn_in_proj");
  gdn_status st = check_proj(dims, hidden, tokens, device_status);
  if (st != GDN_OK) return st;
  if (tokens == 0) return GDN_OK;
  if (!ptr_ok(x) || !ptr_ok(w_in) || !ptr_ok(qkv) || !ptr_ok(z) || !ptr_ok(a) || !ptr_ok(b))
    return GDN_ERR_INVALID_ARG;
  const int Cc = (int)channels(dims), Cv = dims->h_v * dims->d_v;
  gdn::GemmArgs g;
  g.A = static_cast<const uint16_t*>(x);
  g.B = static_cast<const uint16_t*>(w_in);
  g.M = (int)tokens;
  g.N = Cc + Cv + 2 * dims->h_v;
  g.K = hidden;
  g.nseg = 4;
  g.seg[0] = gdn::GemmOut{static_cast<uint16_t*>(qkv), Cc, 0, Cc};
  g.seg[1] = gdn::GemmOut{static_cast<uint16_t*>(z), Cv, Cc, Cv};
  g.seg[2] = gdn::GemmOut{static_cast<uint16_t*>(a), dims->h_v, Cc + Cv, dims->h_v};
  g.seg[3] = gdn::GemmOut{static_cast<uint16_t*>(b), dims->h_v, Cc + Cv + dims->h_v, dims->h_v};
  g.status = device_status;
  return gdn::launch_gemm(g, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_out_proj(const gdn_dims* dims, int hidden, long long tokens, const void* o,
                        const void* w_out, void* y, int32_t* device_status, void* stream) {
  gdn::TraceRange trace_range("gdn_out_proj");
  gdn_status st = check_proj(dims, hidden, tokens, device_status);
  if (st != GDN_OK) return st;
  if (tokens == 0) return GDN_OK;
  if (!ptr_ok(o) || !ptr_ok(w_out) || !ptr_ok(y)) return GDN_ERR_INVALID_ARG;
  gdn::GemmArgs g;
  g.A = static_cast<const uint16_t*>(o);
  g.B = static_cast<const uint16_t*>(w_out);
  g.M = (int)tokens;
  g.N = hidden;
  g.K = dims->h_v * dims->d_v;
  g.nseg = 1;
  g.seg[0] = gdn::GemmOut{static_cast<uint16_t*>(y), hidden, 0, hidden};
  g.status = device_status;
  return gdn::launch_gemm(g, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // extern "C"
