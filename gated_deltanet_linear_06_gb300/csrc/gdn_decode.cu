// gdn_decode.cu -- one decode step of the Gated DeltaNet layer (sm_103a).
//
// The step is bound by HBM: per sequence it reads and writes the fp32 SSM
// state, h_v x 128 x 128 x 4 B = 2 MiB at 32 value heads, against ~40 KiB of
// activations and conv state.  So the kernel is built around streaming the
// state exactly once each way:
//   - one CTA per (sequence, key head) owns the q/k conv channels of that key
//     head and the v channels of its G value heads, so the conv state it
//     reads and rewrites belongs to no other CTA;
//   - a warp updates one state row at a time, each lane holding 4 consecutive
//     fp32 columns (one 128-bit load and one 128-bit store per lane per row,
//     512 contiguous bytes per warp), with batches of 8 rows in flight and
//     the next batch prefetched while the current one is updated;
//   - loads and stores use the streaming cache hint, since the state is
//     touched once per step;
//   - the conv, the norms and the gates run before the first row is needed,
//     while the first batch of rows is already in flight.
//
// Per state row i (S_i: row i of S, d_k wide):
//   S_i <- exp(g) S_i;  u = beta (v_i - S_i . k^);  S_i <- S_i + u k^;  o_i = S_i . q^
// which is exp(g) S (I - beta k^ k^T) + beta v k^T followed by o = S q^.
//
// Bit-identity: every value a sequence produces depends only on its own
// inputs, through reductions in a fixed order (butterfly shuffles over fixed
// lanes); batch size and batch neighbours change only which CTA runs it.
#include "gdn_common.cuh"
#include "gdn_launch.h"
#include "../../include/gdn.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerBatch = 8;
constexpr int kBatchesPerHead = kD / (kWarps * kRowsPerBatch);  // 2

__device__ __forceinline__ float dot4(const float4& s, const float (&v)[4]) {
  float acc = s.x * v[0];
  acc = fmaf(s.y, v[1], acc);
  acc = fmaf(s.z, v[2], acc);
  acc = fmaf(s.w, v[3], acc);
  return acc;
}

template <int G, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(DecodeArgs p) {
  constexpr int kBatches = G * kBatchesPerHead;
  const int bidx = blockIdx.x / p.h_k;
  const int kh = blockIdx.x - bidx * p.h_k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Cq = p.h_k * kD;
  const int Cc = 2 * Cq + p.h_v * kD;

  int s = bidx;
  if (p.slot) {
    s = p.slot[bidx];
    if (s < 0 || s >= p.n_slots) {
      if (tid == 0) record_status(p.status, GDN_ERR_DEVICE_BOUNDS);
      return;
    }
  }

  __shared__ float sq[kD], sk[kD], sv[G][kD], so[G][kD];
  __shared__ float s_decay[G], s_beta[G], s_rstd[G];
  __shared__ float s_rq, s_rk;

  // state rows of value head kh*G + vh, row r: base + (vh*kD + r)*kD
  float* const S_base = p.ssm_state + ((size_t)s * p.h_v + (size_t)kh * G) * kD * kD;
  auto row_ptr = [&](int nb, int j) -> float4* {
    const int vh = nb / kBatchesPerHead;
    const int r = warp * (kBatchesPerHead * kRowsPerBatch) + (nb % kBatchesPerHead) * kRowsPerBatch + j;
    return reinterpret_cast<float4*>(S_base + ((size_t)vh * kD + r) * kD) + lane;
  };

  float4 cur[kRowsPerBatch];
#pragma unroll
  for (int j = 0; j < kRowsPerBatch; ++j) cur[j] = __ldcs(row_ptr(0, j));

  // ---- conv + SiLU over this CTA's channels, conv-state shift ----
  {
    float* cs = p.conv_state + (size_t)s * (kConvW - 1) * Cc;
    const uint16_t* x = p.qkv + (size_t)bidx * Cc;
    for (int ci = tid; ci < (2 + G) * kD; ci += kThreads) {
      int c;
      if (ci < kD) c = kh * kD + ci;
      else if (ci < 2 * kD) c = Cq + kh * kD + (ci - kD);
      else c = 2 * Cq + kh * G * kD + (ci - 2 * kD);
      const float s0 = cs[c], s1 = cs[Cc + c], s2 = cs[2 * Cc + c];
      const float xt = bf16_to_f32(x[c]);
      const uint2 wr = *reinterpret_cast<const uint2*>(p.conv_w + (size_t)c * kConvW);
      const float w0 = bf16_to_f32(wr.x & 0xffffu), w1 = bf16_to_f32(wr.x >> 16);
      const float w2 = bf16_to_f32(wr.y & 0xffffu), w3 = bf16_to_f32(wr.y >> 16);
      float y = w0 * s0;
      y = fmaf(w1, s1, y);
      y = fmaf(w2, s2, y);
      y = fmaf(w3, xt, y);
      y = silu(y);
      cs[c] = s1;
      cs[Cc + c] = s2;
      cs[2 * Cc + c] = xt;
      if (ci < kD) sq[ci] = y;
      else if (ci < 2 * kD) sk[ci - kD] = y;
      else sv[(ci - 2 * kD) / kD][(ci - 2 * kD) % kD] = y;
    }
  }
  __syncthreads();

  // ---- L2 norms of q and k, gates ----
  if (warp == 0 || warp == 1) {
    const float* v = warp == 0 ? sq : sk;
    const float4 x4 = reinterpret_cast<const float4*>(v)[lane];
    float ss = x4.x * x4.x;
    ss = fmaf(x4.y, x4.y, ss);
    ss = fmaf(x4.z, x4.z, ss);
    ss = fmaf(x4.w, x4.w, ss);
    ss = warp_sum(ss);
    if (lane == 0) {
      const float r = rsqrtf(ss + p.l2_eps);
      if (warp == 0) s_rq = r * rsqrtf((float)kD);
      else s_rk = r;
    }
  } else if (warp == 2 && lane < G) {
    const int h = kh * G + lane;
    const float av = bf16_to_f32(p.a[(size_t)bidx * p.h_v + h]);
    const float bv = bf16_to_f32(p.b[(size_t)bidx * p.h_v + h]);
    const float g = -__expf(p.A_log[h]) * softplus(av + p.dt_bias[h]);
    s_decay[lane] = __expf(g);
    s_beta[lane] = sigmoid(bv);
  }
  __syncthreads();

  float qh[4], kk[4];
  {
    const float rq = s_rq, rk = s_rk;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qh[i] = sq[4 * lane + i] * rq;
      kk[i] = sk[4 * lane + i] * rk;
    }
  }

  // ---- the state stream ----
#pragma unroll
  for (int nb = 0; nb < kBatches; ++nb) {
    float4 nxt[kRowsPerBatch];
    if (nb + 1 < kBatches) {
#pragma unroll
      for (int j = 0; j < kRowsPerBatch; ++j) nxt[j] = __ldcs(row_ptr(nb + 1, j));
    }
    const int vh = nb / kBatchesPerHead;
    const int r0 = warp * (kBatchesPerHead * kRowsPerBatch) + (nb % kBatchesPerHead) * kRowsPerBatch;
    const float decay = s_decay[vh], beta = s_beta[vh];
    float red[kRowsPerBatch];
#pragma unroll
    for (int j = 0; j < kRowsPerBatch; ++j) {
      cur[j].x *= decay; cur[j].y *= decay; cur[j].z *= decay; cur[j].w *= decay;
      red[j] = dot4(cur[j], kk);
    }
#pragma unroll
    for (int j = 0; j < kRowsPerBatch; ++j) red[j] = warp_sum(red[j]);
#pragma unroll
    for (int j = 0; j < kRowsPerBatch; ++j) {
      const float u = beta * (sv[vh][r0 + j] - red[j]);
      cur[j].x = fmaf(u, kk[0], cur[j].x);
      cur[j].y = fmaf(u, kk[1], cur[j].y);
      cur[j].z = fmaf(u, kk[2], cur[j].z);
      cur[j].w = fmaf(u, kk[3], cur[j].w);
      __stcs(row_ptr(nb, j), cur[j]);
      red[j] = dot4(cur[j], qh);
    }
#pragma unroll
    for (int j = 0; j < kRowsPerBatch; ++j) red[j] = warp_sum(red[j]);
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < kRowsPerBatch; ++j) so[vh][r0 + j] = red[j];
    }
    if (nb + 1 < kBatches) {
#pragma unroll
      for (int j = 0; j < kRowsPerBatch; ++j) cur[j] = nxt[j];
    }
  }
  __syncthreads();

  // ---- gated RMSNorm over d_v of each value head ----
  if (warp < G) {
    const float4 o4 = reinterpret_cast<const float4*>(so[warp])[lane];
    float ss = o4.x * o4.x;
    ss = fmaf(o4.y, o4.y, ss);
    ss = fmaf(o4.z, o4.z, ss);
    ss = fmaf(o4.w, o4.w, ss);
    ss = warp_sum(ss);
    if (lane == 0) s_rstd[warp] = rsqrtf(ss * (1.0f / kD) + p.rms_eps);
  }
  __syncthreads();
  for (int i = tid; i < G * kD; i += kThreads) {
    const int vh = i / kD, r = i % kD;
    const size_t o_idx = ((size_t)bidx * p.h_v + (size_t)kh * G + vh) * kD + r;
    const float zz = bf16_to_f32(p.z[o_idx]);
    const float val = so[vh][r] * s_rstd[vh] * p.norm_w[r] * silu(zz);
    if (OUT_F32) reinterpret_cast<float*>(p.out)[o_idx] = val;
    else reinterpret_cast<uint16_t*>(p.out)[o_idx] = f32_to_bf16(val);
  }
}

// p.steps decode steps per sequence in one launch: the state rows are read
// once, taken through every token in registers and written once (plus, when
// p.ssm_trace is set, once per token into the trace), so the HBM traffic per
// token falls by the number of tokens.  Every step repeats the single-step
// kernel's arithmetic in its order -- the conv window shift, the norms' lane
// split and butterflies, the gates, each row's decay, dot products, update and
// output dot, the gated RMSNorm -- so k tokens here give, bit for bit, what k
// successive single steps give.
template <int G, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 2) decode_multi_kernel(DecodeArgs p) {
  constexpr int kBatches = G * kBatchesPerHead;
  const int bidx = blockIdx.x / p.h_k;
  const int kh = blockIdx.x - bidx * p.h_k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Cq = p.h_k * kD;
  const int Cc = 2 * Cq + p.h_v * kD;
  const int K = p.steps;

  int s = bidx;
  if (p.slot) {
    s = p.slot[bidx];
    if (s < 0 || s >= p.n_slots) {
      if (tid == 0) record_status(p.status, GDN_ERR_DEVICE_BOUNDS);
      return;
    }
  }

  __shared__ float sq[kDecodeMaxSteps][kD], sk[kDecodeMaxSteps][kD];
  __shared__ float sv[kDecodeMaxSteps][G][kD], so[kDecodeMaxSteps][G][kD];
  __shared__ float s_decay[kDecodeMaxSteps][G], s_beta[kDecodeMaxSteps][G], s_rstd[kDecodeMaxSteps][G];
  __shared__ float s_rq[kDecodeMaxSteps], s_rk[kDecodeMaxSteps];

  // state rows of value head kh*G + vh, row r: base + (vh*kD + r)*kD
  float* const S_base = p.ssm_state + ((size_t)s * p.h_v + (size_t)kh * G) * kD * kD;
  auto row_of = [&](int nb, int j) {
    return warp * (kBatchesPerHead * kRowsPerBatch) + (nb % kBatchesPerHead) * kRowsPerBatch + j;
  };
  auto row_ptr = [&](int nb, int j) -> float4* {
    const int vh = nb / kBatchesPerHead;
    return reinterpret_cast<float4*>(S_base + ((size_t)vh * kD + row_of(nb, j)) * kD) + lane;
  };
  auto trace_ptr = [&](int t, int nb, int j) -> float4* {
    const int vh = nb / kBatchesPerHead;
    float* base = p.ssm_trace + (((size_t)bidx * K + t) * p.h_v + (size_t)kh * G + vh) * kD * kD;
    return reinterpret_cast<float4*>(base + (size_t)row_of(nb, j) * kD) + lane;
  };

  float4 cur[kRowsPerBatch];
#pragma unroll
  for (int j = 0; j < kRowsPerBatch; ++j) cur[j] = __ldcs(row_ptr(0, j));

  // ---- conv + SiLU over this CTA's channels for every token, the window shifting
  //      one token at a time ----
  {
    float* cs = p.conv_state + (size_t)s * (kConvW - 1) * Cc;
    for (int ci = tid; ci < (2 + G) * kD; ci += kThreads) {
      int c;
      if (ci < kD) c = kh * kD + ci;
      else if (ci < 2 * kD) c = Cq + kh * kD + (ci - kD);
      else c = 2 * Cq + kh * G * kD + (ci - 2 * kD);
      float s0 = cs[c], s1 = cs[Cc + c], s2 = cs[2 * Cc + c];
      const uint2 wr = *reinterpret_cast<const uint2*>(p.conv_w + (size_t)c * kConvW);
      const float w0 = bf16_to_f32(wr.x & 0xffffu), w1 = bf16_to_f32(wr.x >> 16);
      const float w2 = bf16_to_f32(wr.y & 0xffffu), w3 = bf16_to_f32(wr.y >> 16);
      for (int t = 0; t < K; ++t) {
        const float xt = bf16_to_f32(p.qkv[((size_t)bidx * K + t) * Cc + c]);
        float y = w0 * s0;
        y = fmaf(w1, s1, y);
        y = fmaf(w2, s2, y);
        y = fmaf(w3, xt, y);
        y = silu(y);
        s0 = s1;
        s1 = s2;
        s2 = xt;
        if (p.conv_trace) {
          float* ct = p.conv_trace + ((size_t)bidx * K + t) * (kConvW - 1) * Cc;
          ct[c] = s0;
          ct[Cc + c] = s1;
          ct[2 * Cc + c] = s2;
        }
        if (ci < kD) sq[t][ci] = y;
        else if (ci < 2 * kD) sk[t][ci - kD] = y;
        else sv[t][(ci - 2 * kD) / kD][(ci - 2 * kD) % kD] = y;
      }
      cs[c] = s0;
      cs[Cc + c] = s1;
      cs[2 * Cc + c] = s2;
    }
  }
  __syncthreads();

  // ---- L2 norms of q and k (a warp per token and vector), gates ----
  for (int pr = warp; pr < 2 * K; pr += kWarps) {
    const int t = pr >> 1;
    const float* v = (pr & 1) ? sk[t] : sq[t];
    const float4 x4 = reinterpret_cast<const float4*>(v)[lane];
    float ss = x4.x * x4.x;
    ss = fmaf(x4.y, x4.y, ss);
    ss = fmaf(x4.z, x4.z, ss);
    ss = fmaf(x4.w, x4.w, ss);
    ss = warp_sum(ss);
    if (lane == 0) {
      const float r = rsqrtf(ss + p.l2_eps);
      if (pr & 1) s_rk[t] = r;
      else s_rq[t] = r * rsqrtf((float)kD);
    }
  }
  for (int i = tid; i < K * G; i += kThreads) {
    const int t = i / G, g = i - t * G;
    const int h = kh * G + g;
    const size_t ab = ((size_t)bidx * K + t) * p.h_v + h;
    const float gg = -__expf(p.A_log[h]) * softplus(bf16_to_f32(p.a[ab]) + p.dt_bias[h]);
    s_decay[t][g] = __expf(gg);
    s_beta[t][g] = sigmoid(bf16_to_f32(p.b[ab]));
  }
  __syncthreads();

  // ---- the state stream: each batch of rows through every token ----
#pragma unroll
  for (int nb = 0; nb < kBatches; ++nb) {
    float4 nxt[kRowsPerBatch];
    if (nb + 1 < kBatches) {
#pragma unroll
      for (int j = 0; j < kRowsPerBatch; ++j) nxt[j] = __ldcs(row_ptr(nb + 1, j));
    }
    const int vh = nb / kBatchesPerHead;
    const int r0 = row_of(nb, 0);
#pragma unroll 1
    for (int t = 0; t < K; ++t) {
      float qh[4], kk[4];
      const float rq = s_rq[t], rk = s_rk[t];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        qh[i] = sq[t][4 * lane + i] * rq;
        kk[i] = sk[t][4 * lane + i] * rk;
      }
      const float decay = s_decay[t][vh], beta = s_beta[t][vh];
      float red[kRowsPerBatch];
#pragma unroll
      for (int j = 0; j < kRowsPerBatch; ++j) {
        cur[j].x *= decay; cur[j].y *= decay; cur[j].z *= decay; cur[j].w *= decay;
        red[j] = dot4(cur[j], kk);
      }
#pragma unroll
      for (int j = 0; j < kRowsPerBatch; ++j) red[j] = warp_sum(red[j]);
#pragma unroll
      for (int j = 0; j < kRowsPerBatch; ++j) {
        const float u = beta * (sv[t][vh][r0 + j] - red[j]);
        cur[j].x = fmaf(u, kk[0], cur[j].x);
        cur[j].y = fmaf(u, kk[1], cur[j].y);
        cur[j].z = fmaf(u, kk[2], cur[j].z);
        cur[j].w = fmaf(u, kk[3], cur[j].w);
        if (p.ssm_trace) __stcs(trace_ptr(t, nb, j), cur[j]);
        red[j] = dot4(cur[j], qh);
      }
#pragma unroll
      for (int j = 0; j < kRowsPerBatch; ++j) red[j] = warp_sum(red[j]);
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < kRowsPerBatch; ++j) so[t][vh][r0 + j] = red[j];
      }
    }
#pragma unroll
    for (int j = 0; j < kRowsPerBatch; ++j) __stcs(row_ptr(nb, j), cur[j]);
    if (nb + 1 < kBatches) {
#pragma unroll
      for (int j = 0; j < kRowsPerBatch; ++j) cur[j] = nxt[j];
    }
  }
  __syncthreads();

  // ---- gated RMSNorm over d_v of each (token, value head) ----
  for (int pr = warp; pr < K * G; pr += kWarps) {
    const int t = pr / G, vh = pr - t * G;
    const float4 o4 = reinterpret_cast<const float4*>(so[t][vh])[lane];
    float ss = o4.x * o4.x;
    ss = fmaf(o4.y, o4.y, ss);
    ss = fmaf(o4.z, o4.z, ss);
    ss = fmaf(o4.w, o4.w, ss);
    ss = warp_sum(ss);
    if (lane == 0) s_rstd[t][vh] = rsqrtf(ss * (1.0f / kD) + p.rms_eps);
  }
  __syncthreads();
  for (int i = tid; i < K * G * kD; i += kThreads) {
    const int t = i / (G * kD), rem = i - t * (G * kD);
    const int vh = rem / kD, r = rem - vh * kD;
    const size_t o_idx = (((size_t)bidx * K + t) * p.h_v + (size_t)kh * G + vh) * kD + r;
    const float zz = bf16_to_f32(p.z[o_idx]);
    const float val = so[t][vh][r] * s_rstd[t][vh] * p.norm_w[r] * silu(zz);
    if (OUT_F32) reinterpret_cast<float*>(p.out)[o_idx] = val;
    else reinterpret_cast<uint16_t*>(p.out)[o_idx] = f32_to_bf16(val);
  }
}

template <int G>
cudaError_t launch_multi_g(const DecodeArgs& p, bool out_f32, cudaStream_t stream) {
  const dim3 grid((unsigned)(p.batch * p.h_k)), block(kThreads);
  if (out_f32) decode_multi_kernel<G, true><<<grid, block, 0, stream>>>(p);
  else decode_multi_kernel<G, false><<<grid, block, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_g(const DecodeArgs& p, bool out_f32, cudaStream_t stream) {
  const dim3 grid((unsigned)(p.batch * p.h_k)), block(kThreads);
  if (out_f32) decode_kernel<G, true><<<grid, block, 0, stream>>>(p);
  else decode_kernel<G, false><<<grid, block, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_multi(const DecodeArgs& p, bool out_f32, cudaStream_t stream) {
  if (p.steps < 1 || p.steps > kDecodeMaxSteps) return cudaErrorInvalidValue;
  switch (p.h_v / p.h_k) {
    case 1: return launch_multi_g<1>(p, out_f32, stream);
    case 2: return launch_multi_g<2>(p, out_f32, stream);
    case 4: return launch_multi_g<4>(p, out_f32, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(const DecodeArgs& p, bool out_f32, cudaStream_t stream) {
  switch (p.h_v / p.h_k) {
    case 1: return launch_g<1>(p, out_f32, stream);
    case 2: return launch_g<2>(p, out_f32, stream);
    case 4: return launch_g<4>(p, out_f32, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
