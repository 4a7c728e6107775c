// gdn_decode.cu -- one decode step of the Gated DeltaNet layer (sm_103a).
//
// The step is bound by HBM: per sequence it reads and writes the fp32 SSM
// state, h_v x 128 x 128 x 4 B = 2 MiB at 32 value heads, against ~40 KiB of
// activations and conv state.  So the kernel is built around streaming the
// state exactly once each way:
//   - one CTA per (sequence, key head) owns the q/k conv channels of that key
//     head and the v channels of its G value heads, so the conv state it
//     reads and rewrites belongs to no other CTA;
//   - a warp updates 8 state rows at a time, 8 lanes per row: lane 8*rr + q
//     holds, for each of two groups of 4 rows, row 4*gi + rr at the columns of
//     the float4 chunks q, q + 8, q + 16, q + 24, so each 128-bit warp load or
//     store covers 4 whole 128-byte row segments; the next batch of rows is
//     prefetched while the current one is updated;
//   - the d_k reductions are an in-lane sum of 16 products in packed fp32x2
//     arithmetic and a 3-level butterfly over the row's 8 lanes, which serves
//     4 rows with each shuffle;
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
#include <atomic>

#include "gdn_common.cuh"
#include "gdn_launch.h"
#include "../../include/gdn.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerBatch = 8;
constexpr int kBatchesPerHead = kD / (kWarps * kRowsPerBatch);  // 2

// A warp's batch of 8 state rows: v[gi][i] is row 4*gi + rr, float4 chunk q + 8*i
// (lane = 8*rr + q).  The 8 chunk indices of a row are the row's 8 lanes.
struct RowBatch {
  float4 v[2][4];
};

// Columns of a lane: float4 chunks q + 8*i, i < 4, as 8 float2 pairs.
struct LaneCols {
  float2 c[8];
};

__device__ __forceinline__ void load_lane_cols(LaneCols& x, const float* vec, int q) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = reinterpret_cast<const float4*>(vec)[q + 8 * i];
    x.c[2 * i] = make_float2(f.x, f.y);
    x.c[2 * i + 1] = make_float2(f.z, f.w);
  }
}

// rows: the batch's first row; row stride kD floats
__device__ __forceinline__ void load_rows(RowBatch& R, const float* rows, int rr, int q) {
#pragma unroll
  for (int gi = 0; gi < 2; ++gi)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      R.v[gi][i] = __ldcs(reinterpret_cast<const float4*>(rows + (size_t)(4 * gi + rr) * kD) + q + 8 * i);
}

__device__ __forceinline__ void store_rows(float* rows, const RowBatch& R, int rr, int q) {
#pragma unroll
  for (int gi = 0; gi < 2; ++gi)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      __stcs(reinterpret_cast<float4*>(rows + (size_t)(4 * gi + rr) * kD) + q + 8 * i, R.v[gi][i]);
}

// 16-byte asynchronous copy global -> shared (L2 only), its commit and wait.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float2 lo2(const float4& f) { return make_float2(f.x, f.y); }
__device__ __forceinline__ float2 hi2(const float4& f) { return make_float2(f.z, f.w); }

// The lane's 16 products of a row with x, summed in a fixed order.
__device__ __forceinline__ float lane_dot(const float4 (&r)[4], const LaneCols& x) {
  float2 acc = __fmul2_rn(lo2(r[0]), x.c[0]);
  acc = __ffma2_rn(hi2(r[0]), x.c[1], acc);
#pragma unroll
  for (int i = 1; i < 4; ++i) {
    acc = __ffma2_rn(lo2(r[i]), x.c[2 * i], acc);
    acc = __ffma2_rn(hi2(r[i]), x.c[2 * i + 1], acc);
  }
  return acc.x + acc.y;
}

// One token on a batch of rows.  With d_k = S_i . k^ and d_q = S_i . q^ taken
// from the state before the token:
//   u = beta (v_i - e^g d_k);   S_i <- e^g S_i + u k^;   o_i = e^g d_q + u (k^ . q^)
// which is S <- e^g S (I - beta k^ k^T) + beta v k^T followed by o = S q^, with the
// output dot moved before the update so that both dots share one butterfly (a
// 3-level xor butterfly over the row's 8 lanes: every lane of the row ends with the
// same bits).  v[gi] is v at the lane's row of group gi; kq = k^ . q^.
__device__ __forceinline__ void rows_token(RowBatch& R, const LaneCols& kk, const LaneCols& qh,
                                           float decay, float beta, float kq, const float (&v)[2],
                                           float (&o)[2]) {
  float dk[2], dq[2];
#pragma unroll
  for (int gi = 0; gi < 2; ++gi) {
    dk[gi] = lane_dot(R.v[gi], kk);
    dq[gi] = lane_dot(R.v[gi], qh);
  }
#pragma unroll
  for (int m = 1; m < 8; m <<= 1)
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
      dk[gi] += __shfl_xor_sync(0xffffffffu, dk[gi], m);
      dq[gi] += __shfl_xor_sync(0xffffffffu, dq[gi], m);
    }
  const float2 d2 = make_float2(decay, decay);
#pragma unroll
  for (int gi = 0; gi < 2; ++gi) {
    const float u = beta * fmaf(-decay, dk[gi], v[gi]);
    o[gi] = fmaf(u, kq, decay * dq[gi]);
    const float2 u2 = make_float2(u, u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = __ffma2_rn(lo2(R.v[gi][i]), d2, __fmul2_rn(u2, kk.c[2 * i]));
      const float2 b = __ffma2_rn(hi2(R.v[gi][i]), d2, __fmul2_rn(u2, kk.c[2 * i + 1]));
      R.v[gi][i] = make_float4(a.x, a.y, b.x, b.y);
    }
  }
}

// Norms of one token's q and k and their dot (a warp; lane holds 4 consecutive
// elements): rq = 1/sqrt(sum q^2 + eps) / sqrt(d_k), rk = 1/sqrt(sum k^2 + eps),
// kq = (q . k) rq rk = k^ . q^.
__device__ __forceinline__ void token_norms(const float* qv, const float* kv, int lane, float eps,
                                            float& rq, float& rk, float& kq) {
  const float4 a = reinterpret_cast<const float4*>(qv)[lane];
  const float4 b = reinterpret_cast<const float4*>(kv)[lane];
  float sq = a.x * a.x, sk = b.x * b.x, qk = a.x * b.x;
  sq = fmaf(a.y, a.y, sq); sk = fmaf(b.y, b.y, sk); qk = fmaf(a.y, b.y, qk);
  sq = fmaf(a.z, a.z, sq); sk = fmaf(b.z, b.z, sk); qk = fmaf(a.z, b.z, qk);
  sq = fmaf(a.w, a.w, sq); sk = fmaf(b.w, b.w, sk); qk = fmaf(a.w, b.w, qk);
  sq = warp_sum(sq);
  sk = warp_sum(sk);
  qk = warp_sum(qk);
  rq = rsqrtf(sq + eps) * rsqrtf((float)kD);
  rk = rsqrtf(sk + eps);
  kq = qk * rq * rk;
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

  __shared__ __align__(16) float sq[kD], sk[kD], sv[G][kD], so[G][kD];
  __shared__ float s_decay[G], s_beta[G], s_rstd[G];
  __shared__ float s_rq, s_rk, s_kq;

  // state rows of value head kh*G + vh, row r: base + (vh*kD + r)*kD; batch nb
  // of a warp covers rows batch_row0(nb) .. + 7 of value head nb / kBatchesPerHead
  float* const S_base = p.ssm_state + ((size_t)s * p.h_v + (size_t)kh * G) * kD * kD;
  const int rr = lane >> 3, q = lane & 7;
  auto batch_row0 = [&](int nb) {
    return warp * (kBatchesPerHead * kRowsPerBatch) + (nb % kBatchesPerHead) * kRowsPerBatch;
  };
  auto batch_rows = [&](int nb) -> float* {
    return S_base + ((size_t)(nb / kBatchesPerHead) * kD + batch_row0(nb)) * kD;
  };

  RowBatch cur;
  load_rows(cur, batch_rows(0), rr, q);

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

  // ---- L2 norms of q and k and k^ . q^, gates ----
  if (warp == 0) {
    float rq, rk, kq;
    token_norms(sq, sk, lane, p.l2_eps, rq, rk, kq);
    if (lane == 0) {
      s_rq = rq;
      s_rk = rk;
      s_kq = kq;
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
  if (tid < kD) {
    sq[tid] *= s_rq;
    sk[tid] *= s_rk;
  }
  __syncthreads();

  LaneCols qh, kk;
  load_lane_cols(qh, sq, q);
  load_lane_cols(kk, sk, q);
  const float kq = s_kq;

  // ---- the state stream ----
#pragma unroll 1
  for (int nb = 0; nb < kBatches; ++nb) {
    RowBatch nxt;
    if (nb + 1 < kBatches) load_rows(nxt, batch_rows(nb + 1), rr, q);
    const int vh = nb / kBatchesPerHead;
    const int r0 = batch_row0(nb);
    const float v[2] = {sv[vh][r0 + rr], sv[vh][r0 + 4 + rr]};
    float o[2];
    rows_token(cur, kk, qh, s_decay[vh], s_beta[vh], kq, v, o);
    store_rows(batch_rows(nb), cur, rr, q);
    if (q == 0) {
      so[vh][r0 + rr] = o[0];
      so[vh][r0 + 4 + rr] = o[1];
    }
    if (nb + 1 < kBatches) cur = nxt;
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
// Bytes of dynamic shared memory of decode_multi_kernel: each warp's staging
// area for its next batch of rows, [8 chunks of the lane][32 lanes] float4.
constexpr int kMultiStageBytes = kWarps * 8 * 32 * 16;

template <int G, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 3) decode_multi_kernel(DecodeArgs p) {
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

  __shared__ __align__(16) float sq[kDecodeMaxSteps][kD], sk[kDecodeMaxSteps][kD];
  __shared__ __align__(16) float sv[kDecodeMaxSteps][G][kD], so[kDecodeMaxSteps][G][kD];
  __shared__ float s_decay[kDecodeMaxSteps][G], s_beta[kDecodeMaxSteps][G], s_rstd[kDecodeMaxSteps][G];
  __shared__ float s_rq[kDecodeMaxSteps], s_rk[kDecodeMaxSteps], s_kq[kDecodeMaxSteps];

  // state rows of value head kh*G + vh, row r: base + (vh*kD + r)*kD (the same
  // batches of rows as the single step)
  float* const S_base = p.ssm_state + ((size_t)s * p.h_v + (size_t)kh * G) * kD * kD;
  const int rr = lane >> 3, q = lane & 7;
  auto batch_row0 = [&](int nb) {
    return warp * (kBatchesPerHead * kRowsPerBatch) + (nb % kBatchesPerHead) * kRowsPerBatch;
  };
  auto batch_rows = [&](int nb) -> float* {
    return S_base + ((size_t)(nb / kBatchesPerHead) * kD + batch_row0(nb)) * kD;
  };
  auto trace_rows = [&](int t, int nb) -> float* {
    const int vh = nb / kBatchesPerHead;
    float* base = p.ssm_trace + (((size_t)bidx * K + t) * p.h_v + (size_t)kh * G + vh) * kD * kD;
    return base + (size_t)batch_row0(nb) * kD;
  };
  // The next batch of rows waits in shared memory, not in registers: each lane
  // copies its own 8 chunks asynchronously and later reads back only what it
  // copied, so the registers go to a third CTA per SM instead.
  extern __shared__ float4 stage_all[];
  float4* const stage = stage_all + warp * (8 * 32) + lane;
  auto stage_batch = [&](int nb) {
    const float* rows = batch_rows(nb);
#pragma unroll
    for (int gi = 0; gi < 2; ++gi)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        cp_async16(stage + (4 * gi + i) * 32,
                   reinterpret_cast<const float4*>(rows + (size_t)(4 * gi + rr) * kD) + q + 8 * i);
    cp_async_commit();
  };
  auto take_batch = [&](RowBatch& R) {
    cp_async_wait_all();
#pragma unroll
    for (int gi = 0; gi < 2; ++gi)
#pragma unroll
      for (int i = 0; i < 4; ++i) R.v[gi][i] = stage[(4 * gi + i) * 32];
  };

  stage_batch(0);

  // ---- gates of every (token, value head): their loads overlap the conv's ----
  for (int i = tid; i < K * G; i += kThreads) {
    const int t = i / G, g = i - t * G;
    const int h = kh * G + g;
    const size_t ab = ((size_t)bidx * K + t) * p.h_v + h;
    const float gg = -__expf(p.A_log[h]) * softplus(bf16_to_f32(p.a[ab]) + p.dt_bias[h]);
    s_decay[t][g] = __expf(gg);
    s_beta[t][g] = sigmoid(bf16_to_f32(p.b[ab]));
  }

  // ---- conv + SiLU over this CTA's channels for every token, the window shifting
  //      one token at a time; every channel's inputs are loaded before any is used ----
  {
    constexpr int kIt = ((2 + G) * kD + kThreads - 1) / kThreads;   // channels per thread
    float* cs = p.conv_state + (size_t)s * (kConvW - 1) * Cc;
    int cidx[kIt];
    float s0[kIt], s1[kIt], s2[kIt];
    uint2 wr[kIt];
    float xs[kIt][kDecodeMaxSteps];
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int ci = tid + it * kThreads;
      cidx[it] = -1;
      if (ci >= (2 + G) * kD) continue;
      const int c = ci < kD ? kh * kD + ci : ci < 2 * kD ? Cq + kh * kD + (ci - kD) : 2 * Cq + kh * G * kD + (ci - 2 * kD);
      cidx[it] = c;
      s0[it] = cs[c];
      s1[it] = cs[Cc + c];
      s2[it] = cs[2 * Cc + c];
      wr[it] = *reinterpret_cast<const uint2*>(p.conv_w + (size_t)c * kConvW);
#pragma unroll
      for (int t = 0; t < kDecodeMaxSteps; ++t)
        if (t < K) xs[it][t] = bf16_to_f32(p.qkv[((size_t)bidx * K + t) * Cc + c]);
    }
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int c = cidx[it];
      if (c < 0) continue;
      const int ci = tid + it * kThreads;
      const float w0 = bf16_to_f32(wr[it].x & 0xffffu), w1 = bf16_to_f32(wr[it].x >> 16);
      const float w2 = bf16_to_f32(wr[it].y & 0xffffu), w3 = bf16_to_f32(wr[it].y >> 16);
      float a0 = s0[it], a1 = s1[it], a2 = s2[it];
#pragma unroll
      for (int t = 0; t < kDecodeMaxSteps; ++t) {
        if (t >= K) break;
        const float xt = xs[it][t];
        float y = w0 * a0;
        y = fmaf(w1, a1, y);
        y = fmaf(w2, a2, y);
        y = fmaf(w3, xt, y);
        y = silu(y);
        a0 = a1;
        a1 = a2;
        a2 = xt;
        if (p.conv_trace) {
          float* ct = p.conv_trace + ((size_t)bidx * K + t) * (kConvW - 1) * Cc;
          ct[c] = a0;
          ct[Cc + c] = a1;
          ct[2 * Cc + c] = a2;
        }
        if (ci < kD) sq[t][ci] = y;
        else if (ci < 2 * kD) sk[t][ci - kD] = y;
        else sv[t][(ci - 2 * kD) / kD][(ci - 2 * kD) % kD] = y;
      }
      cs[c] = a0;
      cs[Cc + c] = a1;
      cs[2 * Cc + c] = a2;
    }
  }
  __syncthreads();

  // ---- L2 norms of q and k and k^ . q^ (a warp per token) ----
  static_assert(kDecodeMaxSteps <= kWarps, "a warp per token");
  if (warp < K) {
    float rq, rk, kq;
    token_norms(sq[warp], sk[warp], lane, p.l2_eps, rq, rk, kq);
    if (lane == 0) {
      s_rq[warp] = rq;
      s_rk[warp] = rk;
      s_kq[warp] = kq;
    }
  }
  __syncthreads();
  for (int i = tid; i < K * kD; i += kThreads) {
    const int t = i / kD, c = i - t * kD;
    sq[t][c] *= s_rq[t];
    sk[t][c] *= s_rk[t];
  }
  __syncthreads();

  // ---- the state stream: each batch of rows through every token ----
#pragma unroll 1
  for (int nb = 0; nb < kBatches; ++nb) {
    RowBatch cur;
    take_batch(cur);
    const int vh = nb / kBatchesPerHead;
    const int r0 = batch_row0(nb);
#pragma unroll 1
    for (int t = 0; t < K; ++t) {
      LaneCols qh, kk;
      load_lane_cols(qh, sq[t], q);
      load_lane_cols(kk, sk[t], q);
      const float v[2] = {sv[t][vh][r0 + rr], sv[t][vh][r0 + 4 + rr]};
      float o[2];
      rows_token(cur, kk, qh, s_decay[t][vh], s_beta[t][vh], s_kq[t], v, o);
      // the staging area is free again once the first token has consumed the
      // values read from it: refill it with the next batch
      if (t == 0 && nb + 1 < kBatches) stage_batch(nb + 1);
      if (p.ssm_trace) store_rows(trace_rows(t, nb), cur, rr, q);
      if (q == 0) {
        so[t][vh][r0 + rr] = o[0];
        so[t][vh][r0 + 4 + rr] = o[1];
      }
    }
    store_rows(batch_rows(nb), cur, rr, q);
  }
  // this thread's z values for the output below, all loaded at once (its
  // output rows share one d_v index, so one norm weight)
  constexpr int kOut = kDecodeMaxSteps * G * kD / kThreads;
  float zv[kOut];
#pragma unroll
  for (int k = 0; k < kOut; ++k) {
    const int i = tid + k * kThreads;
    zv[k] = 0.0f;
    if (i < K * G * kD) {
      const int t = i / (G * kD), rem = i - t * (G * kD);
      const int vh = rem / kD, r = rem - vh * kD;
      zv[k] = bf16_to_f32(p.z[(((size_t)bidx * K + t) * p.h_v + (size_t)kh * G + vh) * kD + r]);
    }
  }
  static_assert(kThreads % kD == 0, "a thread's outputs share one d_v index");
  const float nw = p.norm_w[tid % kD];
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
#pragma unroll
  for (int k = 0; k < kOut; ++k) {
    const int i = tid + k * kThreads;
    if (i >= K * G * kD) break;
    const int t = i / (G * kD), rem = i - t * (G * kD);
    const int vh = rem / kD, r = rem - vh * kD;
    const size_t o_idx = (((size_t)bidx * K + t) * p.h_v + (size_t)kh * G + vh) * kD + r;
    const float val = so[t][vh][r] * s_rstd[t][vh] * nw * silu(zv[k]);
    if (OUT_F32) reinterpret_cast<float*>(p.out)[o_idx] = val;
    else reinterpret_cast<uint16_t*>(p.out)[o_idx] = f32_to_bf16(val);
  }
}

// ---- a captured chain of steps, in one launch ----
//
// A chain of `steps` decode steps whose tokens are all known when it is
// launched (gdn_decode_graph: the caller fills the step-major buffers first)
// runs as one persistent launch.  A cluster of two CTAs owns one (sequence,
// value head), each CTA 64 of its 128 state rows, 8 per warp -- the same
// batches of 8 rows and lane layout as decode_kernel -- and keeps them in
// registers through every step: the state crosses HBM once per launch instead of
// once per step, and a step costs only its token's activations.
//
// Nothing outside a cluster is shared between steps: a step's conv window is
// the raw inputs of the three tokens before it, which each thread keeps in
// registers for its channels (from the conv state before the first step), so
// no CTA writes the conv state during the chain; a small kernel writes it once
// after the last step.  Each CTA conv-filters and normalises q and k (its key
// head's 256 channels, recomputed by every CTA of the key head) and the 64 v
// channels of its rows.  The gated RMSNorm needs all 128 outputs of the head:
// each CTA forms the lane partial sums of o^2 that lanes 16 h .. 16 h + 15 of
// the single step form, writes them into both CTAs' shared memory, and after a
// cluster barrier both run the single step's butterfly over all 32 partials.
// Every value is therefore computed by the same operations in the same order
// as in decode_kernel: the chain gives bit for bit what the same single steps
// give.  The next step's activations are loaded while a step computes.
constexpr int kChainRows = kD / 2;   // state rows of a value head per CTA
constexpr int kChainChannels = 2 * kD + kChainRows;   // conv channels a CTA filters

template <int G, bool OUT_F32>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 2)
    decode_chain_kernel(DecodeArgs p, int steps) {
  const int half = blockIdx.x & 1;
  const int pair = blockIdx.x >> 1;
  const int bidx = pair / p.h_v;
  const int h = pair - bidx * p.h_v;
  const int kh = h / G, vh = h - kh * G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Cq = p.h_k * kD;
  const int Cc = 2 * Cq + p.h_v * kD;
  // per-step strides of the step-major buffers, in elements
  const size_t qkv_step = (size_t)p.batch * Cc, z_step = (size_t)p.batch * p.h_v * kD;
  const size_t ab_step = (size_t)p.batch * p.h_v;

  int s = bidx;
  if (p.slot) {   // both CTAs of the cluster see the same slot and leave together
    s = p.slot[bidx];
    if (s < 0 || s >= p.n_slots) {
      if (tid == 0 && half == 0) record_status(p.status, GDN_ERR_DEVICE_BOUNDS);
      return;
    }
  }

  __shared__ __align__(16) float sq[kD], sk[kD], sv[kChainRows], so[kChainRows];
  __shared__ float s_part[2][32];   // by step parity: the peer may be a step ahead
  __shared__ float s_decay, s_beta, s_rstd, s_rq, s_rk, s_kq;

  // this thread's conv channels (ci < kChainChannels): q and k of the key head,
  // v of this half's rows; taps, and the window of raw inputs before the step
  int chn[2];
  float w[2][kConvW], win[2][kConvW - 1];
  const float* cs = p.conv_state + (size_t)s * (kConvW - 1) * Cc;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int ci = tid + j * kThreads;
    chn[j] = -1;
    if (ci < kChainChannels) {
      const int c = ci < kD ? kh * kD + ci
                            : ci < 2 * kD ? Cq + kh * kD + (ci - kD) : 2 * Cq + h * kD + kChainRows * half + (ci - 2 * kD);
      chn[j] = c;
      const uint2 wr = *reinterpret_cast<const uint2*>(p.conv_w + (size_t)c * kConvW);
      w[j][0] = bf16_to_f32(wr.x & 0xffffu);
      w[j][1] = bf16_to_f32(wr.x >> 16);
      w[j][2] = bf16_to_f32(wr.y & 0xffffu);
      w[j][3] = bf16_to_f32(wr.y >> 16);
#pragma unroll
      for (int r = 0; r < kConvW - 1; ++r) win[j][r] = cs[(size_t)r * Cc + c];
    }
  }
  const float A_exp_h = __expf(p.A_log[h]);   // as the single step forms it
  const float dtb = p.dt_bias[h];
  const int r_out = kChainRows * half + tid;   // this thread's output row (tid < 64)
  const float nw = tid < kChainRows ? p.norm_w[r_out] : 0.0f;

  // the state rows of this warp, in registers for the whole chain
  const int rr = lane >> 3, q = lane & 7;
  float* const rows = p.ssm_state + (((size_t)s * p.h_v + h) * kD + kChainRows * half + 8 * warp) * kD;
  RowBatch cur;
  load_rows(cur, rows, rr, q);

  // step 0's activations; later steps' are loaded one step ahead
  auto load_x = [&](int t, float (&x)[2], float& av, float& bv, float& zz) {
    const uint16_t* xq = p.qkv + (size_t)t * qkv_step + (size_t)bidx * Cc;
#pragma unroll
    for (int j = 0; j < 2; ++j) x[j] = chn[j] >= 0 ? bf16_to_f32(xq[chn[j]]) : 0.0f;
    const size_t ab = (size_t)t * ab_step + (size_t)bidx * p.h_v + h;
    av = (warp == 2 && lane == vh) ? bf16_to_f32(p.a[ab]) : 0.0f;
    bv = (warp == 2 && lane == vh) ? bf16_to_f32(p.b[ab]) : 0.0f;
    zz = tid < kChainRows ? bf16_to_f32(p.z[(size_t)t * z_step + ((size_t)bidx * p.h_v + h) * kD + r_out]) : 0.0f;
  };
  float x[2], av, bv, zz;
  load_x(0, x, av, bv, zz);

#pragma unroll 1
  for (int t = 0; t < steps; ++t) {
    float nx[2] = {0.0f, 0.0f}, nav = 0.0f, nbv = 0.0f, nzz = 0.0f;
    if (t + 1 < steps) load_x(t + 1, nx, nav, nbv, nzz);

    // ---- conv + SiLU, the window shifting by one token ----
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (chn[j] < 0) continue;
      const int ci = tid + j * kThreads;
      float y = w[j][0] * win[j][0];
      y = fmaf(w[j][1], win[j][1], y);
      y = fmaf(w[j][2], win[j][2], y);
      y = fmaf(w[j][3], x[j], y);
      y = silu(y);
      win[j][0] = win[j][1];
      win[j][1] = win[j][2];
      win[j][2] = x[j];
      if (ci < kD) sq[ci] = y;
      else if (ci < 2 * kD) sk[ci - kD] = y;
      else sv[ci - 2 * kD] = y;
    }
    __syncthreads();

    // ---- L2 norms of q and k and k^ . q^, the gates of value head h ----
    if (warp == 0) {
      float rq, rk, kq;
      token_norms(sq, sk, lane, p.l2_eps, rq, rk, kq);
      if (lane == 0) {
        s_rq = rq;
        s_rk = rk;
        s_kq = kq;
      }
    } else if (warp == 2 && lane == vh) {
      const float g = -A_exp_h * softplus(av + dtb);
      s_decay = __expf(g);
      s_beta = sigmoid(bv);
    }
    __syncthreads();
    if (tid < kD) {
      sq[tid] *= s_rq;
      sk[tid] *= s_rk;
    }
    __syncthreads();

    // ---- this warp's 8 rows through the token ----
    {
      LaneCols qh, kk;
      load_lane_cols(qh, sq, q);
      load_lane_cols(kk, sk, q);
      const float v[2] = {sv[8 * warp + rr], sv[8 * warp + 4 + rr]};
      float o[2];
      rows_token(cur, kk, qh, s_decay, s_beta, s_kq, v, o);
      if (q == 0) {
        so[8 * warp + rr] = o[0];
        so[8 * warp + 4 + rr] = o[1];
      }
    }
    __syncthreads();

    // ---- gated RMSNorm: the single step's 32 lane partials, 16 from each CTA ----
    if (warp == 0 && lane < 16) {
      const float4 o4 = reinterpret_cast<const float4*>(so)[lane];
      float ss = o4.x * o4.x;
      ss = fmaf(o4.y, o4.y, ss);
      ss = fmaf(o4.z, o4.z, ss);
      ss = fmaf(o4.w, o4.w, ss);
      float* mine = &s_part[t & 1][16 * half + lane];
      *mine = ss;
      const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(mine));
      uint32_t remote;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(half ^ 1));
      asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(ss) : "memory");
    }
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (warp == 0) {
      const float ss = warp_sum(s_part[t & 1][lane]);
      if (lane == 0) s_rstd = rsqrtf(ss * (1.0f / kD) + p.rms_eps);
    }
    __syncthreads();
    if (tid < kChainRows) {
      const size_t o_idx = (size_t)t * z_step + ((size_t)bidx * p.h_v + h) * kD + r_out;
      const float val = so[tid] * s_rstd * nw * silu(zz);
      if (OUT_F32) reinterpret_cast<float*>(p.out)[o_idx] = val;
      else reinterpret_cast<uint16_t*>(p.out)[o_idx] = f32_to_bf16(val);
    }
    x[0] = nx[0];
    x[1] = nx[1];
    av = nav;
    bv = nbv;
    zz = nzz;
  }
  store_rows(rows, cur, rr, q);
}

// The conv state after a chain of `steps` steps: the raw inputs of its last
// conv_w - 1 positions (rows of the starting conv state where the chain is
// shorter than that).
__global__ void __launch_bounds__(256) decode_chain_conv_state_kernel(DecodeArgs p, const uint16_t* qkv0,
                                                                      int steps) {
  const int Cc = 2 * p.h_k * kD + p.h_v * kD;
  const int bidx = blockIdx.y, c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= Cc) return;
  int s = bidx;
  if (p.slot) {
    s = p.slot[bidx];
    if (s < 0 || s >= p.n_slots) return;   // the step kernels recorded it
  }
  float* cs = p.conv_state + (size_t)s * (kConvW - 1) * Cc;
  float v[kConvW - 1];
#pragma unroll
  for (int r = 0; r < kConvW - 1; ++r) {
    const int pos = steps - (kConvW - 1) + r;
    v[r] = pos >= 0 ? bf16_to_f32(qkv0[((size_t)pos * p.batch + bidx) * Cc + c])
                    : cs[(size_t)(kConvW - 1 + pos) * Cc + c];
  }
#pragma unroll
  for (int r = 0; r < kConvW - 1; ++r) cs[(size_t)r * Cc + c] = v[r];
}

template <int G, bool OUT_F32>
cudaError_t launch_chain_go(const DecodeArgs& p, int steps, cudaStream_t stream) {
  decode_chain_kernel<G, OUT_F32><<<dim3((unsigned)(2 * p.batch * p.h_v)), dim3(kThreads), 0, stream>>>(p, steps);
  return cudaGetLastError();
}

template <int G, bool OUT_F32>
cudaError_t launch_multi_go(const DecodeArgs& p, cudaStream_t stream) {
  // the staging area takes the block's shared memory past the default 48 KiB;
  // the attribute is set once per device and instantiation
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
  if (!bit || !(done.load(std::memory_order_acquire) & bit)) {
    err = cudaFuncSetAttribute(decode_multi_kernel<G, OUT_F32>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kMultiStageBytes);
    if (err != cudaSuccess) return err;
    done.fetch_or(bit, std::memory_order_release);
  }
  decode_multi_kernel<G, OUT_F32>
      <<<dim3((unsigned)(p.batch * p.h_k)), dim3(kThreads), kMultiStageBytes, stream>>>(p);
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_multi_g(const DecodeArgs& p, bool out_f32, cudaStream_t stream) {
  return out_f32 ? launch_multi_go<G, true>(p, stream) : launch_multi_go<G, false>(p, stream);
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
  // one token and no trace: the single-step kernel (same layouts, same arithmetic)
  if (p.steps == 1 && !p.ssm_trace && !p.conv_trace) return launch_decode(p, out_f32, stream);
  switch (p.h_v / p.h_k) {
    case 1: return launch_multi_g<1>(p, out_f32, stream);
    case 2: return launch_multi_g<2>(p, out_f32, stream);
    case 4: return launch_multi_g<4>(p, out_f32, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_chain(const DecodeArgs& p, int steps, bool out_f32, cudaStream_t stream) {
  if (steps < 1 || (long long)p.batch * p.h_v * 2 > 0x7fffffffLL) return cudaErrorInvalidValue;
  switch (p.h_v / p.h_k) {
    case 1: return out_f32 ? launch_chain_go<1, true>(p, steps, stream) : launch_chain_go<1, false>(p, steps, stream);
    case 2: return out_f32 ? launch_chain_go<2, true>(p, steps, stream) : launch_chain_go<2, false>(p, steps, stream);
    case 4: return out_f32 ? launch_chain_go<4, true>(p, steps, stream) : launch_chain_go<4, false>(p, steps, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_chain_conv_state(const DecodeArgs& p, const uint16_t* qkv0, int steps,
                                           cudaStream_t stream) {
  const int Cc = 2 * p.h_k * kD + p.h_v * kD;
  decode_chain_conv_state_kernel<<<dim3((unsigned)((Cc + 255) / 256), (unsigned)p.batch), 256, 0, stream>>>(
      p, qkv0, steps);
  return cudaGetLastError();
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
