// gdn_host.cu -- gdn_prefill from host buffers, with the host link pipelined
// against the compute.
//
// A prefill whose inputs and output live in host memory is bound by the host
// link: at 32K tokens the inputs are 0.8 GB and the output 0.27 GB, several
// times the time of the layer itself.  The packed tokens are therefore cut
// into segments and fed as a chunked-prefill scheduler would (each segment a
// gdn_prefill call whose sequences start from the states the previous segment
// left), while two library copy streams move segment i+1's inputs in and
// segment i-1's output out during segment i's compute:
//
//   h2d stream   : in[i % 2]  <- host inputs of segment i   (after compute i-2 read it)
//   caller stream: gdn_prefill(segment i) into out[i % 2]   (after h2d i and d2h i-2)
//   d2h stream   : host output of segment i <- out[i % 2]   (after compute i)
//
// and the caller's stream finally waits for the last copies, so work enqueued
// on it afterwards sees the whole call complete.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_trace.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr long long kDefaultSegTokens = 5120;   // fastest of 1024 .. 8192 at 32K tokens

struct CopyStreams {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t entry = nullptr, in_done[2] = {}, comp_done[2] = {}, out_done[2] = {};
};
std::mutex g_copy_mu;
CopyStreams g_copy[kMaxDevices];

cudaError_t copy_streams_locked(int dev, CopyStreams*& out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CopyStreams& cs = g_copy[dev];
  if (!cs.ready) {
    cudaError_t e = cudaStreamCreateWithFlags(&cs.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&cs.d2h, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&cs.entry, cudaEventDisableTiming);
    for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
      e = cudaEventCreateWithFlags(&cs.in_done[k], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&cs.comp_done[k], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&cs.out_done[k], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return e;
    cs.ready = true;
  }
  out = &cs;
  return cudaSuccess;
}

// Keeps the first nonzero device status of any segment: *acc = *seg unless
// *acc already holds one.
__global__ void status_fold_kernel(int32_t* acc, const int32_t* seg) {
  if (*acc == 0 && *seg != 0) *acc = *seg;
}

// Small host arrays reach the device as kernel parameters: copied at launch,
// so nothing host-side has to outlive the call and nothing waits on the host.
constexpr int kIntsPerLaunch = 2048;
struct IntBlock {
  int32_t v[kIntsPerLaunch];
};
__global__ void put_ints_kernel(int32_t* dst, int n, const IntBlock blk) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = blk.v[i];
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The segment length a call uses: seg_tokens, 0 meaning the default, never
// more than the tokens there are.
long long effective_seg(int seg_tokens, long long T) {
  long long seg = seg_tokens > 0 ? seg_tokens : kDefaultSegTokens;
  return (T > 0 && seg > T) ? T : seg;
}

// cu_seqlens as the prefill needs it: 0 first, non-decreasing, T last.
bool cu_valid(const int32_t* cu, int n_seqs, long long T) {
  if (!cu || n_seqs < 0 || cu[0] != 0 || cu[n_seqs] != T) return false;
  for (int j = 0; j < n_seqs; ++j)
    if (cu[j + 1] < cu[j]) return false;
  return true;
}

// Segment i: tokens [s0, s1) and the sequences ja .. ja + nj - 1 holding them
// (from the one holding token s0 to the one holding token s1 - 1; empty
// sequences between them come along with no tokens, empty ones at a boundary
// are skipped, which leaves their states as they are, as a call over them would).
struct SegPlan {
  long long s0, s1;
  int ja, nj;
};

void plan_segments(const int32_t* cu, long long T, long long seg, std::vector<SegPlan>& out) {
  out.clear();
  int j = 0;
  for (long long s0 = 0; s0 < T; s0 += seg) {
    SegPlan g;
    g.s0 = s0;
    g.s1 = s0 + seg < T ? s0 + seg : T;
    while (cu[j + 1] <= g.s0) ++j;   // the sequence holding token s0
    int jb = j;
    while (cu[jb + 1] < g.s1) ++jb;  // the sequence holding token s1 - 1
    g.ja = j;
    g.nj = jb - j + 1;
    out.push_back(g);
  }
}

struct HostLayout {
  long long seg;             // tokens per segment
  int nseg;
  size_t cu, in_qkv[2], in_z[2], in_a[2], in_b[2], out[2], pws, pws_bytes, total;
};

bool host_layout(const gdn_dims* d, int n_seqs, long long T, int seg_tokens, HostLayout& l) {
  if (!d || n_seqs < 0 || T < 0 || seg_tokens < 0 || (seg_tokens > 0 && seg_tokens < 64)) return false;
  l.seg = effective_seg(seg_tokens, T);
  const long long nseg = T > 0 ? (T + l.seg - 1) / l.seg : 0;
  if (nseg > (1 << 24)) return false;
  l.nseg = (int)nseg;
  const size_t cc = 2ull * d->h_k * d->d_k + (size_t)d->h_v * d->d_v;
  const size_t zv = (size_t)d->h_v * d->d_v;
  const size_t S = (size_t)(l.seg > 0 ? l.seg : 1);
  size_t off = 256;   // the accumulated device status word
  l.cu = off;   // per segment: its local cu_seqlens, 16-byte aligned
  off = align256(off + 4 * ((size_t)n_seqs + 6 * (size_t)l.nseg + 8));
  for (int k = 0; k < 2; ++k) {
    l.in_qkv[k] = off; off = align256(off + S * cc * 2);
    l.in_z[k] = off;   off = align256(off + S * zv * 2);
    l.in_a[k] = off;   off = align256(off + S * d->h_v * 2);
    l.in_b[k] = off;   off = align256(off + S * d->h_v * 2);
    l.out[k] = off;    off = align256(off + S * zv * 2);
  }
  l.pws = off;
  l.pws_bytes = gdn_workspace_bytes(d, n_seqs > 0 ? n_seqs : 1, (long long)S);
  if (l.pws_bytes == 0) return false;
  l.total = off + l.pws_bytes;
  return true;
}

}  // namespace

extern "C" {

long long gdn_prefill_host_segments(const int32_t* cu_seqlens, int n_seqs, long long total_tokens,
                                    int seg_tokens, long long* seg_info, long long max_segs) {
  if (total_tokens < 0 || seg_tokens < 0 || (seg_tokens > 0 && seg_tokens < 64) || max_segs < 0 ||
      (max_segs > 0 && !seg_info) || !cu_valid(cu_seqlens, n_seqs, total_tokens))
    return -1;
  std::vector<SegPlan> segs;
  plan_segments(cu_seqlens, total_tokens, effective_seg(seg_tokens, total_tokens), segs);
  for (size_t i = 0; i < segs.size() && (long long)i < max_segs; ++i) {
    seg_info[4 * i + 0] = segs[i].s0;
    seg_info[4 * i + 1] = segs[i].s1;
    seg_info[4 * i + 2] = segs[i].ja;
    seg_info[4 * i + 3] = segs[i].nj;
  }
  return (long long)segs.size();
}

size_t gdn_prefill_host_workspace_bytes(const gdn_dims* dims, int n_seqs, long long total_tokens,
                                        int seg_tokens) {
  HostLayout l;
  if (!host_layout(dims, n_seqs, total_tokens, seg_tokens, l)) return 0;
  return l.total;
}

gdn_status gdn_prefill_host(const gdn_dims* dims, const void* qkv, const void* z, const void* a,
                            const void* b, const float* A_log, const float* dt_bias,
                            const void* conv_w, const float* norm_w, const int32_t* cu_seqlens,
                            int n_seqs, long long total_tokens, float* conv_state,
                            float* ssm_state, void* out, int seg_tokens, void* workspace,
                            size_t workspace_bytes, void* stream) {
  gdn::TraceRange trace_range("gdn_prefill_host");
  // dims as gdn_prefill checks them (an empty problem launches nothing)
  const gdn_status dst = gdn_prefill(dims, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                     nullptr, nullptr, nullptr, 0, 0, nullptr, nullptr, nullptr,
                                     nullptr, 0, nullptr);
  if (dst != GDN_OK) return dst;
  HostLayout l;
  if (!host_layout(dims, n_seqs, total_tokens, seg_tokens, l)) return GDN_ERR_INVALID_ARG;
  if (!cu_valid(cu_seqlens, n_seqs, total_tokens)) return GDN_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < l.total)
    return GDN_ERR_WORKSPACE;
  if (n_seqs == 0 || total_tokens == 0) return GDN_OK;
  // every check a segment's gdn_prefill makes on these, made before anything is
  // enqueued, so that an invalid argument launches nothing
  auto dev_ok = [](const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!qkv || !z || !a || !b || !out || !dev_ok(A_log) || !dev_ok(dt_bias) || !dev_ok(conv_w) ||
      !dev_ok(norm_w) || !dev_ok(conv_state) || !dev_ok(ssm_state))
    return GDN_ERR_INVALID_ARG;

  const size_t cc = 2ull * dims->h_k * dims->d_k + (size_t)dims->h_v * dims->d_v;
  const size_t zv = (size_t)dims->h_v * dims->d_v, hv = (size_t)dims->h_v;
  const size_t conv_per_seq = (size_t)(dims->conv_w - 1) * cc;
  const size_t ssm_per_seq = zv * dims->d_k;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // per-segment sequence ranges and local cu_seqlens, planned on the host
  std::vector<SegPlan> segs;
  plan_segments(cu_seqlens, total_tokens, l.seg, segs);
  if ((int)segs.size() != l.nseg) return GDN_ERR_INVALID_ARG;
  std::vector<size_t> cu_off(segs.size());   // int32 index of each segment's cu_seqlens
  std::vector<int32_t> cu_all;
  cu_all.reserve((size_t)n_seqs + 6 * (size_t)l.nseg + 8);
  for (size_t i = 0; i < segs.size(); ++i) {
    const SegPlan& g = segs[i];
    while (cu_all.size() % 4) cu_all.push_back(0);   // gdn_prefill wants 16-byte-aligned cu_seqlens
    cu_off[i] = cu_all.size();
    cu_all.push_back(0);
    for (int q = g.ja; q < g.ja + g.nj; ++q) {
      const long long e = cu_seqlens[q + 1] < g.s1 ? cu_seqlens[q + 1] : g.s1;
      cu_all.push_back((int32_t)(e - g.s0));
    }
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_copy_mu);
  CopyStreams* cs = nullptr;
  if (copy_streams_locked(dev, cs) != cudaSuccess) return GDN_ERR_CUDA;

  int32_t* acc_status = reinterpret_cast<int32_t*>(ws);
  int32_t* cu_dev = reinterpret_cast<int32_t*>(ws + l.cu);
  gdn_status st = GDN_OK;
  bool forked = false;
  auto cuda_ok = [&](cudaError_t e) {
    if (e != cudaSuccess && st == GDN_OK) st = GDN_ERR_CUDA;
    return st == GDN_OK;
  };
  // the copy streams start after the caller's earlier work (the staging buffers
  // and the states may still be in use by it)
  if (cuda_ok(cudaMemsetAsync(ws, 0, 256, s))) {
    for (size_t o = 0; o < cu_all.size() && st == GDN_OK; o += kIntsPerLaunch) {
      const int n = (int)(cu_all.size() - o < (size_t)kIntsPerLaunch ? cu_all.size() - o : kIntsPerLaunch);
      IntBlock blk;
      for (int q = 0; q < n; ++q) blk.v[q] = cu_all[o + (size_t)q];
      put_ints_kernel<<<1, 256, 0, s>>>(cu_dev + o, n, blk);
      cuda_ok(cudaGetLastError());
    }
  }
  if (st == GDN_OK && cuda_ok(cudaEventRecord(cs->entry, s)) &&
      cuda_ok(cudaStreamWaitEvent(cs->h2d, cs->entry, 0)) &&
      cuda_ok(cudaStreamWaitEvent(cs->d2h, cs->entry, 0)))
    forked = true;

  const char* hq = static_cast<const char*>(qkv);
  const char* hz = static_cast<const char*>(z);
  const char* ha = static_cast<const char*>(a);
  const char* hb = static_cast<const char*>(b);
  char* ho = static_cast<char*>(out);
  for (int i = 0; i < l.nseg && st == GDN_OK; ++i) {
    const SegPlan& g = segs[(size_t)i];
    const int k = i & 1;
    const size_t n = (size_t)(g.s1 - g.s0);
    const size_t t0 = (size_t)g.s0;
    // inputs of segment i, once compute i-2 has read the buffer
    if (i >= 2 && !cuda_ok(cudaStreamWaitEvent(cs->h2d, cs->comp_done[k], 0))) break;
    if (!cuda_ok(cudaMemcpyAsync(ws + l.in_qkv[k], hq + t0 * cc * 2, n * cc * 2, cudaMemcpyHostToDevice, cs->h2d)) ||
        !cuda_ok(cudaMemcpyAsync(ws + l.in_z[k], hz + t0 * zv * 2, n * zv * 2, cudaMemcpyHostToDevice, cs->h2d)) ||
        !cuda_ok(cudaMemcpyAsync(ws + l.in_a[k], ha + t0 * hv * 2, n * hv * 2, cudaMemcpyHostToDevice, cs->h2d)) ||
        !cuda_ok(cudaMemcpyAsync(ws + l.in_b[k], hb + t0 * hv * 2, n * hv * 2, cudaMemcpyHostToDevice, cs->h2d)) ||
        !cuda_ok(cudaEventRecord(cs->in_done[k], cs->h2d)))
      break;
    // compute, once the inputs are in and the d2h of segment i-2 has drained out[k]
    if (!cuda_ok(cudaStreamWaitEvent(s, cs->in_done[k], 0))) break;
    if (i >= 2 && !cuda_ok(cudaStreamWaitEvent(s, cs->out_done[k], 0))) break;
    st = gdn_prefill(dims, ws + l.in_qkv[k], ws + l.in_z[k], ws + l.in_a[k], ws + l.in_b[k], A_log,
                     dt_bias, conv_w, norm_w, cu_dev + cu_off[(size_t)i], g.nj, (long long)n,
                     conv_state + (size_t)g.ja * conv_per_seq, ssm_state + (size_t)g.ja * ssm_per_seq,
                     ws + l.out[k], ws + l.pws, l.pws_bytes, stream);
    if (st != GDN_OK) break;
    status_fold_kernel<<<1, 1, 0, s>>>(acc_status, reinterpret_cast<const int32_t*>(ws + l.pws));
    if (!cuda_ok(cudaGetLastError()) || !cuda_ok(cudaEventRecord(cs->comp_done[k], s))) break;
    // output of segment i back to the host
    if (!cuda_ok(cudaStreamWaitEvent(cs->d2h, cs->comp_done[k], 0)) ||
        !cuda_ok(cudaMemcpyAsync(ho + t0 * zv * 2, ws + l.out[k], n * zv * 2, cudaMemcpyDeviceToHost, cs->d2h)) ||
        !cuda_ok(cudaEventRecord(cs->out_done[k], cs->d2h)))
      break;
  }
  // join: the caller's stream waits for everything the copy streams were given
  if (forked) {
    if (cudaEventRecord(cs->in_done[0], cs->h2d) != cudaSuccess ||
        cudaStreamWaitEvent(s, cs->in_done[0], 0) != cudaSuccess ||
        cudaEventRecord(cs->out_done[0], cs->d2h) != cudaSuccess ||
        cudaStreamWaitEvent(s, cs->out_done[0], 0) != cudaSuccess) {
      if (st == GDN_OK) st = GDN_ERR_CUDA;
    }
  }
  return st;
}

}  // extern "C"
