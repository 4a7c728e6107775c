// gdn_prefill.cu -- chunked prefill of the Gated DeltaNet layer (sm_103a).
//
// One CTA per (sequence, value head) walks that sequence in chunks of C = 64
// tokens, keeping the head's state S (d_v x d_k = 128 x 128, fp32) in tensor
// memory across chunks.  Per chunk, with q^, k^, v the conv+SiLU+normalised
// inputs, gamma_t = sum_{s<=t} g_s the cumulative log-decay inside the chunk
// and S0 the state before it (the chunked WY/UT form of the gated delta rule):
//
//   A    = strictly-lower(beta_t e^{gamma_t - gamma_s} k^_t.k^_s)
//   T    = (I + A)^{-1}                                   (CUDA cores, fp32)
//   W^T  = K^T (T diag(beta e^gamma))^T                   MMA  M128 N64 K64
//   U^T  = V^T (T diag(beta))^T                           MMA  M128 N64 K64
//   Vn^T = U^T - S0 W^T                                   MMA  M128 N64 K128
//   O^T  = e^gamma (S0 Q^T)  +  Vn^T P^T,                 MMA  M128 N64 K128 / K64
//          P = lower(q^_t.k^_s e^{gamma_t - gamma_s})
//   S    = e^{gamma_C} S0 + (Vn^T diag(e^{gamma_C-gamma})) K   MMA M128 N128 K64
//   [K; Q] K^T (the Gram matrices feeding A and P)        MMA  M128 N64 K128
//
// then the gated RMSNorm epilogue writes bf16 out.  Every exponential is of a
// non-positive difference, so a chunk whose decay underflows fp32 stays finite.
//
// The Gram product takes its operands in fp16, all others in bf16.  q^ and k^
// are unit-bounded, so fp16 cannot overflow there, and its 3 extra mantissa
// bits matter: when q^_t . k^_t nearly cancels, a token's output is small and
// the RMSNorm magnifies the rounding of these dot products (bf16 Gram operands
// alone put the 4096-token output error at ~9e-3 of its maximum; fp16 halves
// it).
//
// Operands are bf16 tiles in shared memory with the 128-byte swizzle; the
// accumulators are fp32 in tensor memory (512 columns: Gram 64, W 64, U/Vn
// 64, O1 64, O2 64, S 128).  The K^ tile serves both as a K-major operand
// (rows = tokens) and, read MN-major, as K^T / the B operand of the state
// update, so no transposed copy is written.  A partial last chunk is padded
// with tokens whose k, q, v, beta and g are zero, which leave S unchanged.
//
// The conv state is rewritten by a second, small kernel after this one, so no
// CTA overwrites conv-state rows that another CTA of the same sequence still
// reads.
#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_launch.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int C = kChunk;

// ---- shared memory map (bytes from a 1024-aligned base) ----
constexpr uint32_t OFF_KQ = 0;        // [kb0: K^ | Q^][kb1: K^ | Q^], 8 KB each (64 rows x 128 B)
constexpr uint32_t OFF_V = 32768;     // V [t][d_v], 64-column blocks 8 KB apart
constexpr uint32_t OFF_S = 49152;     // S bf16 [d_v][d_k], K blocks 16 KB apart
constexpr uint32_t OFF_WN = 81920;    // -W [t][d_k], K blocks 8 KB apart
constexpr uint32_t OFF_VN = 98304;    // Vn^T [d_v][t]
constexpr uint32_t OFF_VNS = 114688;  // Vn^T diag(e^{gamma_C - gamma}) [d_v][t]
constexpr uint32_t OFF_TB = 131072;   // T diag(beta) [t][s]
constexpr uint32_t OFF_TW = 139264;   // T diag(beta e^gamma) [t][s]
constexpr uint32_t OFF_P = 147456;    // P [t][s]
constexpr uint32_t OFF_KQ16 = OFF_VN; // fp16 copy of the KQ tile for the Gram MMA; aliases Vn^T
                                      // and its scaled copy, which are dead while it is live
constexpr uint32_t OFF_F32 = 155648;  // fp32: A [64][65] + T [64][65], or O staging [64][129]
constexpr int LDA = 65, LDO = 129;
constexpr uint32_t F32_BYTES = 2 * 64 * LDA * 4;
constexpr uint32_t OFF_CW = OFF_F32 + F32_BYTES;  // conv weights fp32 [3][128][4]
constexpr uint32_t OFF_NW = OFF_CW + 3 * 128 * 4 * 4;
constexpr uint32_t OFF_GATE = OFF_NW + 128 * 4;   // gam, beta, e^gam, e^{gamC-gam}: 4 x 64 fp32
constexpr uint32_t SMEM_USED = OFF_GATE + 4 * 64 * 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024

// ---- tensor memory columns ----
constexpr uint32_t TM_G = 0, TM_W = 64, TM_U = 128, TM_O1 = 192, TM_O2 = 256, TM_Z = 384;
constexpr uint32_t TM_COLS = 512;

constexpr uint64_t D_K = tc::sdesc_sw128(16, 1024);         // K-major tiles
constexpr uint64_t D_MN_KQ = tc::sdesc_sw128(16384, 1024);  // K^ read MN-major
constexpr uint64_t D_MN_V = tc::sdesc_sw128(8192, 1024);    // V read MN-major
constexpr uint32_t ID_KK = tc::idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_GRAM = tc::idesc_f16(128, 64, 0, 0);
constexpr uint32_t ID_MN_A = tc::idesc_bf16(128, 64, 1, 0);
constexpr uint32_t ID_MN_B = tc::idesc_bf16(128, 128, 0, 1);

constexpr long long kWaitBudget = 1LL << 31;  // clock cycles (~1 s) before a wait gives up

struct Smem {
  uint8_t* base;
  uint32_t addr;  // shared-window address of base
  __device__ float* f32(uint32_t off) const { return reinterpret_cast<float*>(base + off); }
};

__device__ __forceinline__ void store_bf16x4(uint8_t* tile, uint32_t off, float a, float b, float c,
                                             float d) {
  uint2 v;
  v.x = pack_bf16x2(a, b);
  v.y = pack_bf16x2(c, d);
  *reinterpret_cast<uint2*>(tile + off) = v;
}

__device__ __forceinline__ void store_f16x4(uint8_t* tile, uint32_t off, float a, float b, float c,
                                            float d) {
  uint2 v;
  v.x = pack_f16x2(a, b);
  v.y = pack_f16x2(c, d);
  *reinterpret_cast<uint2*>(tile + off) = v;
}

__device__ __forceinline__ void store_bf16x8(uint8_t* tile, uint32_t off, const float* x) {
  uint4 v;
  v.x = pack_bf16x2(x[0], x[1]);
  v.y = pack_bf16x2(x[2], x[3]);
  v.z = pack_bf16x2(x[4], x[5]);
  v.w = pack_bf16x2(x[6], x[7]);
  *reinterpret_cast<uint4*>(tile + off) = v;
}

// Every thread calls this; all agree on the verdict.
__device__ bool cu_seqlens_valid(const PrefillArgs& p) {
  int bad = 0;
  for (int i = threadIdx.x; i <= p.n_seqs; i += blockDim.x) {
    const int c = p.cu_seqlens[i];
    if (c < 0 || c > p.total_tokens) bad = 1;
    if (i == 0 && c != 0) bad = 1;
    if (i > 0 && c < p.cu_seqlens[i - 1]) bad = 1;
    if (i == p.n_seqs && c != p.total_tokens) bad = 1;
  }
  return !__syncthreads_or(bad);
}

// Block-wide sync that also orders tensor-memory traffic and makes generic
// smem writes visible to the tensor core.
__device__ __forceinline__ void sync_for_mma() {
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(PrefillArgs p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t mbar;
  __shared__ uint32_t tmem_base_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (!cu_seqlens_valid(p)) {
    if (tid == 0) record_status(p.status, GDN_ERR_DEVICE_BOUNDS);
    return;
  }
  const int n = blockIdx.x / p.h_v, h = blockIdx.x % p.h_v;
  const int G = p.h_v / p.h_k, kh = h / G;
  const int start = p.cu_seqlens[n];
  const int len = p.cu_seqlens[n + 1] - start;
  if (len <= 0) return;
  const int Cq = p.h_k * kD, Cc = 2 * Cq + p.h_v * kD;

  Smem sm;
  {
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    sm.base = smem_raw + pad;
    sm.addr = raw + pad;
  }
  float* cw = sm.f32(OFF_CW);      // [blk][i][4]
  float* nw = sm.f32(OFF_NW);
  float* gam = sm.f32(OFF_GATE);
  float* bet = gam + 64;
  float* eg = gam + 128;
  float* egc = gam + 192;
  float* Af = sm.f32(OFF_F32);
  float* Tf = Af + 64 * LDA;
  float* Ost = Af;                  // aliases A and T (used at different times)

  if (tid == 0) tc::mbar_init(&mbar, 1);
  if (warp == 0) tc::tmem_alloc(&tmem_base_s, TM_COLS);
  for (int e = tid; e < 3 * kD; e += kThreads) {
    const int blk = e / kD, i = e % kD;
    const int ch = blk == 0 ? kh * kD + i : blk == 1 ? Cq + kh * kD + i : 2 * Cq + h * kD + i;
    const uint2 w = *reinterpret_cast<const uint2*>(p.conv_w + (size_t)ch * kConvW);
    cw[e * 4 + 0] = bf16_to_f32(w.x & 0xffffu);
    cw[e * 4 + 1] = bf16_to_f32(w.x >> 16);
    cw[e * 4 + 2] = bf16_to_f32(w.y & 0xffffu);
    cw[e * 4 + 3] = bf16_to_f32(w.y >> 16);
  }
  if (tid < kD) nw[tid] = p.norm_w[tid];
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_s;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  const int row = 32 * (warp & 3) + lane;   // TMEM lane this thread reads
  const int half = warp >> 2;               // which half of the columns

  float* S_glob = p.ssm_state + ((size_t)n * p.h_v + h) * kD * kD;
  // initial state: fp32 into TMEM, bf16 into the S operand tile
  {
    const float4* src = reinterpret_cast<const float4*>(S_glob + (size_t)row * kD + half * 64);
#pragma unroll
    for (int c32 = 0; c32 < 2; ++c32) {
      float v[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 x = src[c32 * 8 + q];
        v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
      }
      tc::tmem_st32(tmem + lane_base + TM_Z + half * 64 + c32 * 32, v);
#pragma unroll
      for (int m = 0; m < 4; ++m)
        store_bf16x8(sm.base + OFF_S, tc::sw128_off(row, half * 64 + c32 * 32 + 8 * m, 16384), v + 8 * m);
    }
  }

  const float A_exp = __expf(p.A_log[h]);
  const float dtb = p.dt_bias[h];
  const float qscale = rsqrtf((float)kD);
  uint32_t phase = 0;
  bool aborted = false;

  auto wait_mma = [&]() -> bool {
    const bool ok = tc::mbar_wait(&mbar, phase, kWaitBudget);
    phase ^= 1u;
    const bool all_ok = __syncthreads_and(ok);
    tc::fence_after_sync();
    return all_ok;
  };

  for (int t0 = 0; t0 < len && !aborted; t0 += C) {
    const int L = min(C, len - t0);

    // ---- gates and their cumulative sums (warp 0) ----
    if (warp == 0) {
      float g2[2], b2[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int t = lane + 32 * u;
        g2[u] = 0.0f;
        b2[u] = 0.0f;
        if (t < L) {
          const size_t pidx = (size_t)(start + t0 + t) * p.h_v + h;
          g2[u] = -A_exp * softplus(bf16_to_f32(p.a[pidx]) + dtb);
          b2[u] = sigmoid(bf16_to_f32(p.b[pidx]));
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, g2[u], off);
          if (lane >= off) g2[u] += y;
        }
      }
      g2[1] += __shfl_sync(0xffffffffu, g2[0], 31);
      const float gC = __shfl_sync(0xffffffffu, g2[1], 31);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int t = lane + 32 * u;
        gam[t] = g2[u];
        bet[t] = b2[u];
        eg[t] = __expf(g2[u]);
        egc[t] = __expf(gC - g2[u]);
      }
    }

    // ---- conv + SiLU + L2 norms -> K^, Q^, V tiles (all warps) ----
    for (int t = warp; t < C; t += kThreads / 32) {
      float y[3][4];
      if (t < L) {
#pragma unroll
        for (int blk = 0; blk < 3; ++blk)
#pragma unroll
          for (int e = 0; e < 4; ++e) y[blk][e] = 0.0f;
#pragma unroll
        for (int j = 0; j < kConvW; ++j) {
          const int tau = t0 + t - (kConvW - 1) + j;   // position in the sequence
#pragma unroll
          for (int blk = 0; blk < 3; ++blk) {
            const int ch = (blk == 0 ? kh * kD : blk == 1 ? Cq + kh * kD : 2 * Cq + h * kD) + 4 * lane;
            float x[4];
            if (tau >= 0) {
              const uint2 r = *reinterpret_cast<const uint2*>(p.qkv + (size_t)(start + tau) * Cc + ch);
              x[0] = bf16_to_f32(r.x & 0xffffu); x[1] = bf16_to_f32(r.x >> 16);
              x[2] = bf16_to_f32(r.y & 0xffffu); x[3] = bf16_to_f32(r.y >> 16);
            } else {
              const float4 r = *reinterpret_cast<const float4*>(
                  p.conv_state + ((size_t)n * (kConvW - 1) + (kConvW - 1 + tau)) * Cc + ch);
              x[0] = r.x; x[1] = r.y; x[2] = r.z; x[3] = r.w;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float w = cw[(blk * kD + 4 * lane + e) * 4 + j];
              y[blk][e] = j == 0 ? w * x[e] : fmaf(w, x[e], y[blk][e]);
            }
          }
        }
#pragma unroll
        for (int blk = 0; blk < 3; ++blk)
#pragma unroll
          for (int e = 0; e < 4; ++e) y[blk][e] = silu(y[blk][e]);
        float sq = y[0][0] * y[0][0], sk = y[1][0] * y[1][0];
#pragma unroll
        for (int e = 1; e < 4; ++e) {
          sq = fmaf(y[0][e], y[0][e], sq);
          sk = fmaf(y[1][e], y[1][e], sk);
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        const float rq = rsqrtf(sq + p.l2_eps) * qscale, rk = rsqrtf(sk + p.l2_eps);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          y[0][e] *= rq;
          y[1][e] *= rk;
        }
      } else {
#pragma unroll
        for (int blk = 0; blk < 3; ++blk)
#pragma unroll
          for (int e = 0; e < 4; ++e) y[blk][e] = 0.0f;
      }
      store_bf16x4(sm.base + OFF_KQ, tc::sw128_off(t, 4 * lane, 16384), y[1][0], y[1][1], y[1][2], y[1][3]);
      store_bf16x4(sm.base + OFF_KQ + 8192, tc::sw128_off(t, 4 * lane, 16384), y[0][0], y[0][1], y[0][2], y[0][3]);
      store_bf16x4(sm.base + OFF_V, tc::sw128_off(t, 4 * lane, 8192), y[2][0], y[2][1], y[2][2], y[2][3]);
      store_f16x4(sm.base + OFF_KQ16, tc::sw128_off(t, 4 * lane, 16384), y[1][0], y[1][1], y[1][2], y[1][3]);
      store_f16x4(sm.base + OFF_KQ16 + 8192, tc::sw128_off(t, 4 * lane, 16384), y[0][0], y[0][1], y[0][2], y[0][3]);
    }
    sync_for_mma();

    // ---- Gram matrices [K; Q] K^T and O1 = S0 Q^T ----
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t kb = k >> 2, ks = (k & 3) * 32;
        const uint32_t a = sm.addr + OFF_KQ16 + kb * 16384 + ks;
        tc::mma_bf16(tmem + TM_G, tc::sdesc_at(D_K, a), tc::sdesc_at(D_K, a), ID_GRAM, k > 0);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t kb = k >> 2, ks = (k & 3) * 32;
        tc::mma_bf16(tmem + TM_O1, tc::sdesc_at(D_K, sm.addr + OFF_S + kb * 16384 + ks),
                     tc::sdesc_at(D_K, sm.addr + OFF_KQ + kb * 16384 + 8192 + ks), ID_KK, k > 0);
      }
      tc::mma_commit(&mbar);
    }
    // meanwhile: pre-scale the fp32 state by the chunk's total decay
    {
      const float dC = eg[C - 1];
#pragma unroll
      for (int c32 = 0; c32 < 2; ++c32) {
        float v[32];
        const uint32_t ta = tmem + lane_base + TM_Z + half * 64 + c32 * 32;
        tc::tmem_ld32(ta, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= dC;
        tc::tmem_st32(ta, v);
      }
    }
    if (!wait_mma()) { aborted = true; break; }

    // ---- A (fp32, warps 0-1) and P (bf16 tile, warps 2-3) from the Gram rows ----
    if (warp < 4) {
      float v[32];
      const int t = row & 63;
      const float gt = gam[t];
#pragma unroll
      for (int c32 = 0; c32 < 2; ++c32) {
        tc::tmem_ld32(tmem + lane_base + TM_G + c32 * 32, v);
        if (warp < 2) {
          const float bt = bet[t];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int s = c32 * 32 + i;
            Af[t * LDA + s] = s < t ? bt * __expf(gt - gam[s]) * v[i] : 0.0f;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int s = c32 * 32 + i;
            v[i] = s <= t ? v[i] * __expf(gt - gam[s]) : 0.0f;
          }
#pragma unroll
          for (int m = 0; m < 4; ++m)
            store_bf16x8(sm.base + OFF_P, tc::sw128_off(t, c32 * 32 + 8 * m, 0), v + 8 * m);
        }
      }
    }
    __syncthreads();

    // ---- T = (I + A)^{-1}: 16 x 16 diagonal blocks, then block rows ----
    if (tid < 64) {
      const int b = tid >> 4, c = tid & 15;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float acc = (r == c) ? 1.0f : 0.0f;
#pragma unroll
        for (int s = 0; s < r; ++s) acc = fmaf(-Af[(16 * b + r) * LDA + 16 * b + s], x[s], acc);
        x[r] = acc;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) Tf[(16 * b + r) * LDA + 16 * b + c] = x[r];
    } else {
      // zero the blocks above the diagonal
      for (int e = tid - 64; e < 6 * 256; e += kThreads - 64) {
        const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
        const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        Tf[(16 * bi + r) * LDA + 16 * bj + c] = 0.0f;
      }
    }
    __syncthreads();
#pragma unroll 1
    for (int d = 1; d < 4; ++d) {
      const int tasks = 64 * (4 - d);
      if (tid < tasks) {
        const int j = tid >> 6, i = j + d, c = (tid >> 2) & 15, qr = tid & 3;
        // M[4qr + r][c] = sum_{k=j}^{i-1} A_ik T_kj
        float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int kb = j; kb < i; ++kb) {
#pragma unroll
          for (int s = 0; s < 16; ++s) {
            const float tv = Tf[(16 * kb + s) * LDA + 16 * j + c];
#pragma unroll
            for (int r = 0; r < 4; ++r)
              m[r] = fmaf(Af[(16 * i + 4 * qr + r) * LDA + 16 * kb + s], tv, m[r]);
          }
        }
        float mf[16];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int r = 0; r < 4; ++r) mf[4 * q + r] = __shfl_sync(0xffffffffu, m[r], (lane & ~3) | q);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int rr = 4 * qr + r;
          float acc = 0.0f;
#pragma unroll
          for (int q = 0; q < 16; ++q) acc = fmaf(Tf[(16 * i + rr) * LDA + 16 * i + q], mf[q], acc);
          Tf[(16 * i + rr) * LDA + 16 * j + c] = -acc;
        }
      }
      __syncthreads();
    }
    // T diag(beta) and T diag(beta e^gamma) as bf16 tiles [t][s]
    for (int e = tid; e < 64 * 8; e += kThreads) {
      const int t = e >> 3, c8 = (e & 7) * 8;
      float xb[8], xw[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float tv = Tf[t * LDA + c8 + q];
        xb[q] = tv * bet[c8 + q];
        xw[q] = xb[q] * eg[c8 + q];
      }
      store_bf16x8(sm.base + OFF_TB, tc::sw128_off(t, c8, 0), xb);
      store_bf16x8(sm.base + OFF_TW, tc::sw128_off(t, c8, 0), xw);
    }
    sync_for_mma();

    // ---- W^T = K^T Tw^T and U^T = V^T Tb^T ----
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tc::mma_bf16(tmem + TM_W, tc::sdesc_at(D_MN_KQ, sm.addr + OFF_KQ + k * 2048),
                     tc::sdesc_at(D_K, sm.addr + OFF_TW + k * 32), ID_MN_A, k > 0);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tc::mma_bf16(tmem + TM_U, tc::sdesc_at(D_MN_V, sm.addr + OFF_V + k * 2048),
                     tc::sdesc_at(D_K, sm.addr + OFF_TB + k * 32), ID_MN_A, k > 0);
      }
      tc::mma_commit(&mbar);
    }
    if (!wait_mma()) { aborted = true; break; }

    // ---- -W tile [t][d_k] from W^T (lane = d_k index) ----
    {
      float v[32];
      tc::tmem_ld32(tmem + lane_base + TM_W + half * 32, v);
      uint8_t* wn = sm.base + OFF_WN;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int t = half * 32 + i;
        *reinterpret_cast<uint16_t*>(wn + tc::sw128_off(t, row, 8192)) = f32_to_bf16(-v[i]);
      }
    }
    sync_for_mma();

    // ---- Vn^T = U^T - S0 W^T ----
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t kb = k >> 2, ks = (k & 3) * 32;
        tc::mma_bf16(tmem + TM_U, tc::sdesc_at(D_K, sm.addr + OFF_S + kb * 16384 + ks),
                     tc::sdesc_at(D_K, sm.addr + OFF_WN + kb * 8192 + ks), ID_KK, 1u);
      }
      tc::mma_commit(&mbar);
    }
    if (!wait_mma()) { aborted = true; break; }

    // ---- Vn^T tiles (plain and decay-weighted), row = d_v index ----
    {
      float v[32], vs[32];
      tc::tmem_ld32(tmem + lane_base + TM_U + half * 32, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) vs[i] = v[i] * egc[half * 32 + i];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t off = tc::sw128_off(row, half * 32 + 8 * m, 0);
        store_bf16x8(sm.base + OFF_VN, off, v + 8 * m);
        store_bf16x8(sm.base + OFF_VNS, off, vs + 8 * m);
      }
    }
    sync_for_mma();

    // ---- O2 = Vn^T P^T and S += Vn^T diag(e^{gC-g}) K ----
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tc::mma_bf16(tmem + TM_O2, tc::sdesc_at(D_K, sm.addr + OFF_VN + k * 32),
                     tc::sdesc_at(D_K, sm.addr + OFF_P + k * 32), ID_KK, k > 0);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tc::mma_bf16(tmem + TM_Z, tc::sdesc_at(D_K, sm.addr + OFF_VNS + k * 32),
                     tc::sdesc_at(D_MN_KQ, sm.addr + OFF_KQ + k * 2048), ID_MN_B, 1u);
      }
      tc::mma_commit(&mbar);
    }
    if (!wait_mma()) { aborted = true; break; }

    // ---- new S -> bf16 operand tile; O = e^gamma O1 + O2 -> fp32 staging ----
    {
#pragma unroll
      for (int c32 = 0; c32 < 2; ++c32) {
        float v[32];
        tc::tmem_ld32(tmem + lane_base + TM_Z + half * 64 + c32 * 32, v);
#pragma unroll
        for (int m = 0; m < 4; ++m)
          store_bf16x8(sm.base + OFF_S, tc::sw128_off(row, half * 64 + c32 * 32 + 8 * m, 16384), v + 8 * m);
      }
      float o1[32], o2[32];
      tc::tmem_ld32(tmem + lane_base + TM_O1 + half * 32, o1);
      tc::tmem_ld32(tmem + lane_base + TM_O2 + half * 32, o2);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int t = half * 32 + i;
        Ost[t * LDO + row] = fmaf(eg[t], o1[i], o2[i]);
      }
    }
    __syncthreads();

    // ---- gated RMSNorm epilogue: warp per token ----
    for (int t = warp; t < L; t += kThreads / 32) {
      float o[4];
      float ss = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[e] = Ost[t * LDO + lane + 32 * e];
        ss = fmaf(o[e], o[e], ss);
      }
      ss = warp_sum(ss);
      const float rstd = rsqrtf(ss * (1.0f / kD) + p.rms_eps);
      const size_t obase = ((size_t)(start + t0 + t) * p.h_v + h) * kD;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = lane + 32 * e;
        const float zz = bf16_to_f32(p.z[obase + i]);
        p.out[obase + i] = f32_to_bf16(o[e] * rstd * nw[i] * silu(zz));
      }
    }
    __syncthreads();
  }

  if (aborted) {
    if (tid == 0) record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
  } else {
    // final state back to global memory
    float4* dst = reinterpret_cast<float4*>(S_glob + (size_t)row * kD + half * 64);
#pragma unroll
    for (int c32 = 0; c32 < 2; ++c32) {
      float v[32];
      tc::tmem_ld32(tmem + lane_base + TM_Z + half * 64 + c32 * 32, v);
#pragma unroll
      for (int q = 0; q < 8; ++q) dst[c32 * 8 + q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TM_COLS);
}

// The last conv_w - 1 raw inputs of each sequence become its conv state
// (rows of the old state fill in when the sequence is shorter than that).
__global__ void __launch_bounds__(256) conv_state_kernel(PrefillArgs p) {
  if (!cu_seqlens_valid(p)) return;
  const int Cc = 2 * p.h_k * kD + p.h_v * kD;
  const int n = blockIdx.y, c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= Cc) return;
  const int start = p.cu_seqlens[n], len = p.cu_seqlens[n + 1] - start;
  float* cs = p.conv_state + (size_t)n * (kConvW - 1) * Cc;
  float v[kConvW - 1];
#pragma unroll
  for (int r = 0; r < kConvW - 1; ++r) {
    const int pos = len - (kConvW - 1) + r;
    v[r] = pos >= 0 ? bf16_to_f32(p.qkv[(size_t)(start + pos) * Cc + c]) : cs[(size_t)(kConvW - 1 + pos) * Cc + c];
  }
#pragma unroll
  for (int r = 0; r < kConvW - 1; ++r) cs[(size_t)r * Cc + c] = v[r];
}

}  // namespace

size_t prefill_scratch_bytes(int, int, int, long long) { return 0; }

cudaError_t launch_prefill(const PrefillArgs& p, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  prefill_kernel<<<(unsigned)(p.n_seqs * p.h_v), kThreads, SMEM_BYTES, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int Cc = 2 * p.h_k * kD + p.h_v * kD;
  conv_state_kernel<<<dim3((unsigned)((Cc + 255) / 256), (unsigned)p.n_seqs), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
