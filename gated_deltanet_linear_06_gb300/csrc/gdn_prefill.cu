// gdn_prefill.cu -- chunked prefill of the Gated DeltaNet layer (sm_103a):
// the launcher, the work list, the combine pass of segmented sequences, the
// conv-state update, and the single-pass kernel.
//
// gdn_prefill runs the split path (gdn_prefill_split.cu): a chunk-parallel
// prep pass writes per-chunk records to the workspace, then state scans walk
// the chunks.  The single-pass kernel below does everything in one CTA per
// (sequence, value head) with no records, for callers without a workspace
// (gdn_prefill_noalloc); the arithmetic is the same.
//
// The single pass walks a sequence in chunks of C = 64
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
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_launch.h"
#include "gdn_tc.cuh"
#include "gdn_prefill.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 512;   // 16 warps: 4 per TMEM lane quarter
static_assert(kThreads / 32 * 4 == C, "the conv stage gives each warp a quad of a chunk's tokens");

// ---- shared memory map (bytes from a 1024-aligned base) ----
struct Lay {
  static constexpr uint32_t KQ = 0;        // [kb0: K^ | Q^][kb1: K^ | Q^], 8 KB each (64 rows x 128 B)
  static constexpr uint32_t V = 32768;     // V [t][d_v], 64-column blocks 8 KB apart
  static constexpr uint32_t S = 49152;     // S bf16 [d_v][d_k], K blocks 16 KB apart
  static constexpr uint32_t VN = 81920;    // Vn^T [d_v][t]
  static constexpr uint32_t VNS = 98304;   // Vn^T diag(e^{gamma_C - gamma}) [d_v][t]
  static constexpr uint32_t KQ16 = VN;     // fp16 copy of KQ for the Gram MMA (dead before Vn^T is written)
  static constexpr uint32_t WN = 114688;   // -W [d_k][t] (read MN-major)
  static constexpr uint32_t TB = 131072;   // T diag(beta) [t][s]
  static constexpr uint32_t TW = 139264;   // T diag(beta e^gamma) [t][s]
  static constexpr uint32_t P = 147456;    // P [t][s]
  static constexpr uint32_t F32 = 155648;  // fp32: the solve's A, then T over it (17 KB)
};
constexpr uint32_t F32_BYTES = 2 * UT_BYTES;
// Staging of a chunk's raw inputs, loaded by TMA (2-D tensor maps over qkv and z):
// the raw q, k and v rows of tokens t0-3 .. t0+63 (bf16, one [67][128] box per
// block) land over -W, T, P and the fp32 area, which are dead from the last MMA of
// the previous chunk to the end of this chunk's conv stage; z ([64][128]) lands in
// the fp32 area's tail between the state-correction MMA and the epilogue.
struct Map : Lay {
  using L_ = Lay;
  static constexpr uint32_t CW = L_::F32 + F32_BYTES;   // conv weights fp32 [3][tap][128]
  static constexpr uint32_t NW = CW + 3 * 128 * 4 * 4;
  static constexpr uint32_t GATE = NW + 128 * 4;        // gam, beta, e^gam, e^{gamC-gam}
  static constexpr uint32_t USED = GATE + 4 * 64 * 4;
  static constexpr uint32_t BYTES = USED + 1024;        // slack to align the base to 1024
  static constexpr uint32_t RAW = L_::WN;               // [q | k | v blocks]
  static constexpr uint32_t RAW_END = RAW + 3 * RAW_BLK;
  static constexpr uint32_t OST = L_::VN;               // O staging fp32 [64][128]
  static constexpr uint32_t Z = RAW_END;                // z bf16 [64][128]
  static_assert(RAW_END <= L_::F32 + F32_BYTES, "raw staging past the fp32 area");
  static_assert(RAW % 128 == 0 && RAW_BLK % 128 == 0 && RAW_END % 128 == 0, "TMA destinations need 128-B alignment");
  static_assert(Z + 64 * 128 * 2 <= CW, "z staging overlaps the conv weights");
  static_assert(OST + 64 * LDO * 4 <= L_::WN, "O staging overlaps -W");
  static_assert(BYTES <= 227 * 1024, "shared memory");
};

// ---- tensor memory columns ----
constexpr uint32_t TM_G = 0, TM_W = 64, TM_U = 128, TM_O1 = 192, TM_O2 = 256, TM_Z = 384;
constexpr uint32_t TM_COLS = 512;

// One thread: the raw q, k and v rows of tokens t0-3 .. t0+63 of a sequence
// starting at packed row `start` (rows before the sequence are fetched too and
// ignored: the conv reads the carried conv state for them).
__device__ __forceinline__ void stage_raw(const CUtensorMap* tm_qkv, uint8_t* raw, uint64_t* mbar, int start,
                                          int t0, int kh, int h, int Cq) {
  mbar_expect_tx(mbar, 3 * RAW_BLK);
  const int y = start + t0 - (kConvW - 1);
  tma_load_2d(raw, tm_qkv, kh * kD, y, mbar);
  tma_load_2d(raw + RAW_BLK, tm_qkv, Cq + kh * kD, y, mbar);
  tma_load_2d(raw + 2 * RAW_BLK, tm_qkv, 2 * Cq + h * kD, y, mbar);
}

// Every thread calls this; all agree on the answer.
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



__global__ void __launch_bounds__(kThreads, 1)
    fused_kernel(const PrefillArgs p, const __grid_constant__ CUtensorMap tm_qkv,
                 const __grid_constant__ CUtensorMap tm_z) {
  using M = Map;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t mbar;      // MMA completion
  __shared__ __align__(8) uint64_t mbar_raw;  // raw q|k|v rows of a chunk landed
  __shared__ __align__(8) uint64_t mbar_z;    // z of a chunk landed
  __shared__ uint32_t tmem_base_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = blockIdx.x / p.h_v, h = blockIdx.x % p.h_v;
  if (u >= p.seg_list[0]) return;
  const Seg sg = load_seg(p.seg_list, u);
  const int n = sg.n;
  const int G = p.h_v / p.h_k, kh = h / G;
  const int start = p.cu_seqlens[n];
  const int seg_end = sg.begin + sg.len;          // token positions within the sequence
  const int Cq = p.h_k * kD, Cc = 2 * Cq + p.h_v * kD;

  // the state: read at the start, written back at the end (one segment per sequence)
  float* ssm = p.ssm_state + ((size_t)n * p.h_v + h) * kD * kD;

  const Smem sm = smem_aligned(smem_raw);
  float* cw = sm.f32(M::CW);      // [blk][tap][i]
  float* nw = sm.f32(M::NW);
  float* gam = sm.f32(M::GATE);
  float* bet = gam + 64;
  float* eg = gam + 128;
  float* egc = gam + 192;
  float* Af = sm.f32(M::F32);   // A, then T over it (the solve runs in place)
  const float* Tf = Af;
  float* Ost = sm.f32(M::OST);      // aliases the Vn tiles (used after them)

  if (tid == 0) {
    tc::mbar_init(&mbar, 1);
    tc::mbar_init(&mbar_raw, 1);
    tc::mbar_init(&mbar_z, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base_s, TM_COLS);
  for (int e = tid; e < 3 * kD; e += kThreads) {   // tap-major: cw[blk][tap][channel]
    const int blk = e / kD, i = e % kD;
    const int ch = blk == 0 ? kh * kD + i : blk == 1 ? Cq + kh * kD + i : 2 * Cq + h * kD + i;
    const uint2 w = *reinterpret_cast<const uint2*>(p.conv_w + (size_t)ch * kConvW);
    cw[(blk * 4 + 0) * kD + i] = bf16_to_f32(w.x & 0xffffu);
    cw[(blk * 4 + 1) * kD + i] = bf16_to_f32(w.x >> 16);
    cw[(blk * 4 + 2) * kD + i] = bf16_to_f32(w.y & 0xffffu);
    cw[(blk * 4 + 3) * kD + i] = bf16_to_f32(w.y >> 16);
  }
  if (tid < kD) nw[tid] = p.norm_w[tid];
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_s;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  const int row = 32 * (warp & 3) + lane;   // TMEM lane this thread reads
  const int part = warp >> 2;               // which quarter of a lane quarter's columns

  // initial state: fp32 into TMEM, bf16 into the operand tile
  {
    const int col0 = part * 32;
    float v[32];
    const float4* src = reinterpret_cast<const float4*>(ssm + (size_t)row * kD + col0);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 x = src[q];
      v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
    }
    tc::tmem_st32(tmem + lane_base + TM_Z + col0, v);
#pragma unroll
    for (int m = 0; m < 4; ++m)
      store_bf16x8(sm.base + M::S, tc::sw128_off(row, col0 + 8 * m, 16384), v + 8 * m);
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

  if (tid == 32) stage_raw(&tm_qkv, sm.base + M::RAW, &mbar_raw, start, sg.begin, kh, h, Cq);
  // gate inputs of the next chunk, prefetched into warp 0's registers
  float a_nx[2] = {0.0f, 0.0f}, b_nx[2] = {0.0f, 0.0f};
  if (warp == 0) {
#pragma unroll
    for (int uu = 0; uu < 2; ++uu) {
      const int t = sg.begin + lane + 32 * uu;
      if (t < seg_end) {
        const size_t pidx = (size_t)(start + t) * p.h_v + h;
        a_nx[uu] = bf16_to_f32(p.a[pidx]);
        b_nx[uu] = bf16_to_f32(p.b[pidx]);
      }
    }
  }
  uint32_t chunk_parity = 0;
  // bulk copies in flight (uniform across the CTA), waited for on the time-out path
  bool raw_pending = true, z_pending = false;
  for (int t0 = sg.begin; t0 < seg_end && !aborted; t0 += C, chunk_parity ^= 1u) {
    const int L = min(C, seg_end - t0);

    // ---- gates and their cumulative sums (warp 0) ----
    if (warp == 0) {
      float g2[2], b2[2];
#pragma unroll
      for (int uu = 0; uu < 2; ++uu) {
        const int t = lane + 32 * uu;
        g2[uu] = t < L ? -A_exp * softplus_gate(a_nx[uu] + dtb) : 0.0f;
        b2[uu] = t < L ? sigmoid_gate(b_nx[uu]) : 0.0f;
      }
      // prefetch the next chunk's gate inputs
#pragma unroll
      for (int uu = 0; uu < 2; ++uu) {
        const int t = t0 + C + lane + 32 * uu;
        if (t < seg_end) {
          const size_t pidx = (size_t)(start + t) * p.h_v + h;
          a_nx[uu] = bf16_to_f32(p.a[pidx]);
          b_nx[uu] = bf16_to_f32(p.b[pidx]);
        }
      }
#pragma unroll
      for (int uu = 0; uu < 2; ++uu) {
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, g2[uu], off);
          if (lane >= off) g2[uu] += y;
        }
      }
      g2[1] += __shfl_sync(0xffffffffu, g2[0], 31);
      const float gC = __shfl_sync(0xffffffffu, g2[1], 31);
#pragma unroll
      for (int uu = 0; uu < 2; ++uu) {
        const int t = lane + 32 * uu;
        gam[t] = g2[uu];
        bet[t] = b2[uu];
        eg[t] = __expf(g2[uu]);
        egc[t] = __expf(gC - g2[uu]);
      }
    }

    if (!__syncthreads_and(tc::mbar_wait(&mbar_raw, chunk_parity, kWaitBudget))) { aborted = true; break; }
    raw_pending = false;

    // ---- conv + SiLU + L2 norms -> K^, Q^, V tiles.  Warp w takes tokens 4w .. 4w+3
    //      of every block and a lane 4 channels of them, so each raw row is read once
    //      for all the taps that use it and the four tokens are independent work ----
    {
      const int tq = 4 * warp;
#pragma unroll
      for (int blk = 0; blk < 3; ++blk) {
        float w[kConvW][4];
#pragma unroll
        for (int j = 0; j < kConvW; ++j) {
          const float4 w4 = reinterpret_cast<const float4*>(cw + (blk * 4 + j) * kD)[lane];
          w[j][0] = w4.x; w[j][1] = w4.y; w[j][2] = w4.z; w[j][3] = w4.w;
        }
        float y[4][4];
        conv_quad_staged(sm.base + M::RAW + blk * RAW_BLK,
                         p.conv_state + (size_t)n * (kConvW - 1) * Cc +
                             (blk == 0 ? kh * kD : blk == 1 ? Cq + kh * kD : 2 * Cq + h * kD) + 4 * lane,
                         Cc, t0, L, tq, lane, w, y);
        if (blk < 2) {
          float rn[4];
          l2_rnorm4(y, p.l2_eps, blk == 0 ? qscale : 1.0f, lane, rn);
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) y[i][e] *= rn[i];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = tq + i;
          if (blk == 2) {
            store_bf16x4(sm.base + M::V, tc::sw128_off(t, 4 * lane, 8192), y[i][0], y[i][1], y[i][2], y[i][3]);
          } else {
            const uint32_t o16 = tc::sw128_off(t, 4 * lane, 16384) + (blk == 0 ? 8192u : 0u);
            store_bf16x4(sm.base + M::KQ, o16, y[i][0], y[i][1], y[i][2], y[i][3]);
            store_f16x4(sm.base + M::KQ16, o16, y[i][0], y[i][1], y[i][2], y[i][3]);
          }
        }
      }
    }
    sync_for_mma();

    // ---- Gram matrices [K; Q] K^T (fp16) and, in the output pass, O1 = S0 Q^T ----
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t kb = k >> 2, ks = (k & 3) * 32;
        const uint32_t a = sm.addr + M::KQ16 + kb * 16384 + ks;
        tc::mma_bf16(tmem + TM_G, tc::sdesc_at(D_K, a), tc::sdesc_at(D_K, a), ID_GRAM, k > 0);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t kb = k >> 2, ks = (k & 3) * 32;
        tc::mma_bf16(tmem + TM_O1, tc::sdesc_at(D_K, sm.addr + M::S + kb * 16384 + ks),
                     tc::sdesc_at(D_K, sm.addr + M::KQ + kb * 16384 + 8192 + ks), ID_KK, k > 0);
      }
      tc::mma_commit(&mbar);
    }
    // meanwhile: pre-scale the fp32 state by the chunk's total decay
    {
      const float dC = eg[C - 1];
      float v[32];
      const uint32_t ta = tmem + lane_base + TM_Z + part * 32;
      tc::tmem_ld32(ta, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= dC;
      tc::tmem_st32(ta, v);
    }
    if (!wait_mma()) { aborted = true; break; }

    // ---- A (fp32, lanes 0-63, below its diagonal: the solve reads nothing
    //      else) and P (bf16 tile, lanes 64-127) from the Gram rows; warps w and
    //      w+4 share a lane quarter and split its 64 columns ----
    {
      float v[16];
      const int t = row & 63;
      const float gt = gam[t];
      const int c0 = part * 16;
      tc::tmem_ld16(tmem + lane_base + TM_G + c0, v);
      if ((warp & 3) < 2) {
        const float bt = bet[t];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float a[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) a[e] = bt * __expf(gt - gam[c0 + 4 * m + e]) * v[4 * m + e];
          ut_st4(Af, t, c0 + 4 * m, a[0], a[1], a[2], a[3]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int s = c0 + i;
          v[i] = keep_if_le(v[i] * __expf(gt - gam[s]), s, t);
        }
#pragma unroll
        for (int m = 0; m < 2; ++m)
          store_bf16x8(sm.base + M::P, tc::sw128_off(t, c0 + 8 * m, 0), v + 8 * m);
      }
    }
    __syncthreads();

    // ---- T = (I + A)^{-1} ----
    solve_unit_lower<kThreads>(Af, tid, 0);
    // T diag(beta) and T diag(beta e^gamma) as bf16 tiles [t][s]
    for (int e = tid; e < 64 * 8; e += kThreads) {
      const int t = e >> 3, c8 = (e & 7) * 8;
      float xb[8], xw[8];
      const float4 lo = ut_ld4(Tf, t, c8), hi = ut_ld4(Tf, t, c8 + 4);
      const float tv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        xb[q] = keep_if_le(tv[q], c8 + q, t) * bet[c8 + q];   // T is zero above its diagonal
        xw[q] = xb[q] * eg[c8 + q];
      }
      store_bf16x8(sm.base + M::TB, tc::sw128_off(t, c8, 0), xb);
      store_bf16x8(sm.base + M::TW, tc::sw128_off(t, c8, 0), xw);
    }
    sync_for_mma();

    // ---- W^T = K^T Tw^T and U^T = V^T Tb^T ----
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tc::mma_bf16(tmem + TM_W, tc::sdesc_at(D_MN_KQ, sm.addr + M::KQ + k * 2048),
                     tc::sdesc_at(D_K, sm.addr + M::TW + k * 32), ID_MN_A, k > 0);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tc::mma_bf16(tmem + TM_U, tc::sdesc_at(D_MN_V, sm.addr + M::V + k * 2048),
                     tc::sdesc_at(D_K, sm.addr + M::TB + k * 32), ID_MN_A, k > 0);
      }
      tc::mma_commit(&mbar);
    }
    if (!wait_mma()) { aborted = true; break; }

    // ---- -W tile [d_k][t] from W^T (lane = d_k index: 32 contiguous bytes a thread) ----
    {
      float v[16];
      tc::tmem_ld16(tmem + lane_base + TM_W + part * 16, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = -v[i];
#pragma unroll
      for (int m = 0; m < 2; ++m) store_bf16x8(sm.base + M::WN, tc::sw128_off(row, part * 16 + 8 * m, 0), v + 8 * m);
    }
    sync_for_mma();

    // ---- Vn^T = U^T - S0 W^T ----
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t kb = k >> 2, ks = (k & 3) * 32;
        tc::mma_bf16(tmem + TM_U, tc::sdesc_at(D_K, sm.addr + M::S + kb * 16384 + ks),
                     tc::sdesc_at(D_MN_W, sm.addr + M::WN + k * 2048), ID_KMN, 1u);
      }
      tc::mma_commit(&mbar);
    }
    if (!wait_mma()) { aborted = true; break; }

    // ---- z of the chunk -> smem (TMA; read by the epilogue) ----
    if (tid == 32) {
      mbar_expect_tx(&mbar_z, 64 * 256);
      tma_load_2d(sm.base + M::Z, &tm_z, h * kD, start + t0, &mbar_z);
    }
    z_pending = true;

    // ---- Vn^T tiles (plain and decay-weighted), row = d_v index ----
    {
      float v[16], vs[16];
      tc::tmem_ld16(tmem + lane_base + TM_U + part * 16, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) vs[i] = v[i] * egc[part * 16 + i];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint32_t off = tc::sw128_off(row, part * 16 + 8 * m, 0);
        store_bf16x8(sm.base + M::VN, off, v + 8 * m);
        store_bf16x8(sm.base + M::VNS, off, vs + 8 * m);
      }
    }
    sync_for_mma();

    // ---- O2 = Vn^T P^T and S += Vn^T diag(e^{gC-g}) K ----
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tc::mma_bf16(tmem + TM_O2, tc::sdesc_at(D_K, sm.addr + M::VN + k * 32),
                     tc::sdesc_at(D_K, sm.addr + M::P + k * 32), ID_KK, k > 0);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tc::mma_bf16(tmem + TM_Z, tc::sdesc_at(D_K, sm.addr + M::VNS + k * 32),
                     tc::sdesc_at(D_MN_KQ, sm.addr + M::KQ + k * 2048), ID_MN_B, 1u);
      }
      tc::mma_commit(&mbar);
    }
    if (!wait_mma()) { aborted = true; break; }
    // the next chunk's raw rows land while this chunk finishes
    if (tid == 32 && t0 + C < seg_end) stage_raw(&tm_qkv, sm.base + M::RAW, &mbar_raw, start, t0 + C, kh, h, Cq);
    raw_pending = t0 + C < seg_end;

    // ---- new state -> bf16 operand tile; O = e^gamma O1 + O2 -> fp32 staging ----
    {
      float v[32];
      tc::tmem_ld32(tmem + lane_base + TM_Z + part * 32, v);
#pragma unroll
      for (int m = 0; m < 4; ++m)
        store_bf16x8(sm.base + M::S, tc::sw128_off(row, part * 32 + 8 * m, 16384), v + 8 * m);
      float o1[16], o2[16];
      tc::tmem_ld16(tmem + lane_base + TM_O1 + part * 16, o1);
      tc::tmem_ld16(tmem + lane_base + TM_O2 + part * 16, o2);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = part * 16 + i;
        Ost[t * LDO + row] = fmaf(eg[t], o1[i], o2[i]);
      }
    }
    if (!__syncthreads_and(tc::mbar_wait(&mbar_z, chunk_parity, kWaitBudget))) { aborted = true; break; }
    z_pending = false;

    // ---- gated RMSNorm epilogue: warp per token, 4 channels per lane ----
    for (int t = warp; t < L; t += kThreads / 32) {
      const float4 o4 = reinterpret_cast<const float4*>(Ost + t * LDO)[lane];
      float ss = o4.x * o4.x;
      ss = fmaf(o4.y, o4.y, ss);
      ss = fmaf(o4.z, o4.z, ss);
      ss = fmaf(o4.w, o4.w, ss);
      ss = warp_sum(ss);
      const float rstd = rsqrtf(ss * (1.0f / kD) + p.rms_eps);
      const uint2 zr = *reinterpret_cast<const uint2*>(sm.base + M::Z + t * 256 + lane * 8);
      const float4 w4 = reinterpret_cast<const float4*>(nw)[lane];
      float g[4] = {bf16_to_f32(zr.x & 0xffffu), bf16_to_f32(zr.x >> 16), bf16_to_f32(zr.y & 0xffffu),
                    bf16_to_f32(zr.y >> 16)};
      silu4(g);
      uint2 o;
      o.x = pack_bf16x2(o4.x * rstd * w4.x * g[0], o4.y * rstd * w4.y * g[1]);
      o.y = pack_bf16x2(o4.z * rstd * w4.z * g[2], o4.w * rstd * w4.w * g[3]);
      *reinterpret_cast<uint2*>(p.out + ((size_t)(start + t0 + t) * p.h_v + h) * kD + 4 * lane) = o;
    }
    __syncthreads();
  }

  if (aborted) {
    if (tid == 0) record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
    // let this CTA's own bulk copies finish (bounded) before its smem goes away
    if (raw_pending) tc::mbar_wait(&mbar_raw, chunk_parity, kWaitBudget);
    if (z_pending) tc::mbar_wait(&mbar_z, chunk_parity, kWaitBudget);
  } else {
    // final state back to global memory
    float4* dst = reinterpret_cast<float4*>(ssm + (size_t)row * kD + part * 32);
    float v[32];
    tc::tmem_ld32(tmem + lane_base + TM_Z + part * 32, v);
#pragma unroll
    for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TM_COLS);
}

// The work list: every sequence split into segments of p.seg_tokens (the last
// one ragged; a sequence of at most that many tokens is one segment), and the
// list of sequences with more than one segment.  On the split path it also
// numbers the chunks of all sequences (a record slot per chunk): chunk_off[n]
// is the first chunk of sequence n and chunk_list[c] the (sequence, first
// token) of chunk c.  Validates cu_seqlens first: on a violation the lists
// stay empty and the status word says why.
__global__ void __launch_bounds__(256) seg_list_kernel(PrefillArgs p) {
  __shared__ int s_cnt[256], s_ch[256];
  __shared__ int s_base, s_mbase, s_cbase;
  if (!cu_seqlens_valid(p)) {
    if (threadIdx.x == 0) {
      record_status(p.status, GDN_ERR_DEVICE_BOUNDS);
      p.seg_list[0] = 0;
      p.multi_list[0] = 0;
    }
    if (p.chunk_list)
      for (int c = threadIdx.x; c < p.max_chunks; c += blockDim.x) p.chunk_list[c] = make_int2(-1, 0);
    return;
  }
  if (threadIdx.x == 0) { s_base = 0; s_mbase = 0; s_cbase = 0; }
  __syncthreads();
  for (int n0 = 0; n0 < p.n_seqs; n0 += 256) {
    const int n = n0 + threadIdx.x;
    int nsig = 0, len = 0, st = 0, nch = 0;
    if (n < p.n_seqs) {
      st = p.cu_seqlens[n];
      len = p.cu_seqlens[n + 1] - st;
      nsig = len <= 0 ? 0 : (len + p.seg_tokens - 1) / p.seg_tokens;
      nch = len <= 0 ? 0 : (len + C - 1) / C;
    }
    // inclusive scans over the tile of segment counts (bits 0-21) with
    // multi-segment flags (bits 22-30), and of chunk counts
    s_cnt[threadIdx.x] = nsig | ((nsig > 1 ? 1 : 0) << 22);
    s_ch[threadIdx.x] = nch;
    __syncthreads();
    for (int off = 1; off < 256; off <<= 1) {
      const int v = threadIdx.x >= off ? s_cnt[threadIdx.x - off] : 0;
      const int w = threadIdx.x >= off ? s_ch[threadIdx.x - off] : 0;
      __syncthreads();
      s_cnt[threadIdx.x] += v;
      s_ch[threadIdx.x] += w;
      __syncthreads();
    }
    const int incl = s_cnt[threadIdx.x], incl_ch = s_ch[threadIdx.x];
    const int seg_off = s_base + (incl & 0x3FFFFF) - nsig;
    const int m_off = s_mbase + (incl >> 22) - (nsig > 1 ? 1 : 0);
    const int ch_off = s_cbase + incl_ch - nch;
    const int k0 = st / p.seg_tokens;
    if (p.chunk_off && n < p.n_seqs) p.chunk_off[n] = ch_off;
    for (int sg = 0; sg < nsig; ++sg) {
      int* e = p.seg_list + 4 + 8 * (seg_off + sg);
      e[0] = n;
      e[1] = sg * p.seg_tokens;
      e[2] = min(p.seg_tokens, len - sg * p.seg_tokens);
      e[3] = sg;
      e[4] = nsig;
      e[5] = k0;
      e[6] = ch_off + sg * (p.seg_tokens / C);
    }
    if (nsig > 1) {
      int* e = p.multi_list + 4 + 4 * m_off;
      e[0] = n;
      e[1] = k0;
      e[2] = nsig;
    }
    __syncthreads();
    if (threadIdx.x == 255) {
      s_base += incl & 0x3FFFFF;
      s_mbase += incl >> 22;
      s_cbase += incl_ch;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.seg_list[0] = s_base;
    p.multi_list[0] = s_mbase;
    if (p.chunk_off) p.chunk_off[p.n_seqs] = s_cbase;
  }
  if (!p.chunk_list) return;
  __syncthreads();   // chunk_off is complete (and visible to the whole block)
  const int n_chunks = s_cbase;
  for (int c = threadIdx.x; c < p.max_chunks; c += blockDim.x) {
    int2 e = make_int2(-1, 0);
    if (c < n_chunks) {
      // the last sequence whose first chunk is <= c (empty sequences share their successor's offset)
      int lo = 0, hi = p.n_seqs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.chunk_off[mid] <= c) lo = mid; else hi = mid - 1;
      }
      e = make_int2(lo, (c - p.chunk_off[lo]) * C);
    }
    p.chunk_list[c] = e;
  }
}

// The last conv_w - 1 raw inputs of each sequence become its conv state
// (rows of the old state fill in when the sequence is shorter than that).
__global__ void __launch_bounds__(256) conv_state_kernel(PrefillArgs p) {
  if (*p.status == GDN_ERR_DEVICE_BOUNDS) return;   // cu_seqlens rejected by the list kernel
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

namespace {
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
size_t align1024(size_t x) { return (x + 1023) & ~(size_t)1023; }
struct ScratchLayout {
  size_t seg_list, multi_list, xfer, xzero, chunk_off, chunk_list, rec_kq, rec_v, total;
  long long max_chunks;
};
// The scratch of one call.  The split path (records = true) has room for a
// segment per 1024 tokens, their transfer maps, the chunk index and the
// per-chunk records; the single-pass path needs only the unsplit work list,
// whose size depends on n_seqs alone.
ScratchLayout scratch_layout(int n_seqs, int h_k, int h_v, long long total_tokens, bool records) {
  const long long slots = records ? total_tokens / kSegTokens : 0;   // the single pass never segments
  const long long units = slots + n_seqs;   // segments: sum of ceil(T_n / L) <= T / L + N
  ScratchLayout l;
  l.seg_list = 0;
  l.multi_list = align256(16 + (size_t)units * 32);
  l.xfer = l.multi_list + align256(16 + (size_t)slots * 16);
  l.xzero = l.xfer + (size_t)slots * h_v * 3 * kD * kD * sizeof(float);
  size_t end = l.xzero + align256((size_t)slots * h_v * sizeof(int));
  l.max_chunks = records ? total_tokens / C + n_seqs : 0;
  l.chunk_off = align256(end);
  l.chunk_list = l.chunk_off + (records ? align256((size_t)(n_seqs + 1) * 4) : 0);
  l.rec_kq = align1024(l.chunk_list + (size_t)l.max_chunks * 8);
  l.rec_v = l.rec_kq + (size_t)l.max_chunks * h_k * kRecKQ;
  end = l.rec_v + (size_t)l.max_chunks * h_v * kRecV;
  l.total = records ? end : l.xzero + align256((size_t)slots * h_v * sizeof(int));
  return l;
}
}  // namespace

size_t prefill_scratch_bytes(int n_seqs, int h_k, int h_v, long long total_tokens) {
  return scratch_layout(n_seqs, h_k, h_v, total_tokens, true).total;
}

size_t prefill_scratch_bytes_unsplit(int n_seqs) { return scratch_layout(n_seqs, 0, 0, 0, false).total; }

// Segment length L: whole chunks, at least kSegTokens (which sizes the
// workspace), at least two segments, and only when one CTA per (sequence,
// value head) would leave the GPU short (sequences x h_v < 4 x SMs) and some
// sequence could be longer than L.  L minimises a cost model of the scans, as
// if all tokens were one sequence: with s = ceil(T / L) segments of L / C
// chunks, the output scan runs ceil(s h_v / SMs) waves of CTAs each walking
// L / C chunks, the transfer scan ceil((s - 1) h_v / SMs) such waves (two
// tracks, two CTAs per SM), and the combine s - 1 dependent steps of about 1.5
// chunk-times.  Measured at 32K tokens, 32 value heads, 152 SMs: the model's
// choice, 3648 tokens (9 segments), 1.10 ms a call; 4096: 1.14; 2368: 1.14;
// 2048: 1.19; 1024: 1.27; 8192: 1.22.
long long prefill_segment_tokens(int n_seqs, int h_v, long long total_tokens, int sms) {
  if (n_seqs <= 0 || h_v <= 0 || sms <= 0 || (long long)n_seqs * h_v >= 4LL * sms || total_tokens <= kSegTokens)
    return 0;
  long long seg_len = kSegTokens;
  double best = 1e300;
  for (long long s = 2; s <= 64; ++s) {
    long long L = (total_tokens + s - 1) / s;
    L = std::max<long long>((L + C - 1) / C * C, kSegTokens);
    const long long segs = (total_tokens + L - 1) / L;
    const long long waves = (segs * h_v + sms - 1) / sms + ((segs - 1) * h_v + sms - 1) / sms;
    const double cost = (double)waves * (double)(L / C) + 1.5 * (double)(segs - 1);
    if (cost < best - 1e-9 || (cost < best + 1e-9 && L > seg_len)) {
      best = cost;
      seg_len = L;
    }
  }
  return total_tokens > seg_len ? seg_len : 0;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows][cols] array, box [box_rows][box_cols].
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                 uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A segmented call runs as kHeadGroups groups of key heads (with their value
// heads), each on its own stream: every head's passes are independent of the
// other heads', so one group's combine pass -- a chain of dependent steps on
// one CTA per head -- and the passes' last partial waves overlap other groups'
// work.  A kernel timeline shows the groups' prep passes running one after
// another and the scans after them: the dispatcher hands out pending CTAs in the
// order their grids became eligible.  Measured slower, each time because the SMs
// are busy in both phases and reordering only moves work around:
//   - stream priorities to run the first group ahead (a pending high-priority
//     combine CTA needs a whole SM and holds back the rest);
//   - chaining the groups' prep passes, 1.14 -> 1.28 ms at 32K tokens;
//   - the transfer scans on high-priority streams, beside the later prep passes
//     (those slowed by about as much as they absorbed, and the last group's
//     chain then queued behind the other groups' output scans), 1.14 -> 1.29 ms;
//     again once the transfer scan skipped its decayed prefix (12 us a group),
//     with the transfer and combine passes alone on high-priority streams forked
//     after each prep pass, 0.768 -> 0.797 ms (slow decay 0.988 -> 1.102 ms).
// The first group runs on the caller's stream, the others on side streams, per
// device, created on first use and kept for the life of the process; the
// caller's stream forks to them through one event and joins back through one
// event per side stream.  Enqueueing is serialised by a mutex, so concurrent
// calls on one device also share (and are ordered on) the side streams.
constexpr int kHeadGroups = 4;
constexpr int kMaxDevices = 64;
struct SideStreams {
  bool ready = false;
  cudaStream_t s[kHeadGroups - 1] = {};
  cudaEvent_t fork = nullptr, join[kHeadGroups - 1] = {};
};
std::mutex g_side_mu;
SideStreams g_side[kMaxDevices];

cudaError_t side_streams_locked(int dev, SideStreams*& out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  SideStreams& ss = g_side[dev];
  if (!ss.ready) {
    cudaError_t e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming);
    for (int i = 0; i < kHeadGroups - 1 && e == cudaSuccess; ++i) {
      e = cudaStreamCreateWithFlags(&ss.s[i], cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.join[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return e;   // a partial set is created again next time (the handles made so far leak)
    ss.ready = true;
  }
  out = &ss;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& p_in, cudaStream_t stream, bool allow_split) {
  PrefillArgs p = p_in;
  p.kh0 = 0;
  p.nkh = p.h_k;
  p.h0 = 0;
  p.nh = p.h_v;
  const ScratchLayout l = scratch_layout(p.n_seqs, p.h_k, p.h_v, p.total_tokens, allow_split);
  char* scratch = static_cast<char*>(p.scratch);
  p.seg_list = reinterpret_cast<int*>(scratch + l.seg_list);
  p.multi_list = reinterpret_cast<int*>(scratch + l.multi_list);
  p.xfer = reinterpret_cast<float*>(scratch + l.xfer);
  p.xzero = reinterpret_cast<int*>(scratch + l.xzero);
  p.chunk_off = allow_split ? reinterpret_cast<int*>(scratch + l.chunk_off) : nullptr;
  p.chunk_list = allow_split ? reinterpret_cast<int2*>(scratch + l.chunk_list) : nullptr;
  p.rec_kq = allow_split ? reinterpret_cast<uint8_t*>(scratch + l.rec_kq) : nullptr;
  p.rec_v = allow_split ? reinterpret_cast<uint8_t*>(scratch + l.rec_v) : nullptr;
  p.max_chunks = (int)l.max_chunks;
  cudaError_t e;
  const int Cc_ = 2 * p.h_k * kD + p.h_v * kD;
  CUtensorMap tm_qkv, tm_z;
  if (!make_map_2d(&tm_qkv, p.qkv, (uint64_t)Cc_, (uint64_t)p.total_tokens, kD, RAW_BOX_ROWS) ||
      !make_map_2d(&tm_z, p.z, (uint64_t)p.h_v * kD, (uint64_t)p.total_tokens, kD, C))
    return cudaErrorInvalidValue;
  if (!allow_split) {
    // one fused pass per (sequence, value head): no records, no segments
    if ((e = cudaFuncSetAttribute(fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)Map::BYTES)) != cudaSuccess)
      return e;
    p.seg_tokens = 0x40000000;
    seg_list_kernel<<<1, 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fused_kernel<<<(unsigned)p.n_seqs * (unsigned)p.h_v, kThreads, Map::BYTES, stream>>>(p, tm_qkv, tm_z);
  } else {
    // Split long sequences into segments scanned in parallel only when one CTA
    // per (sequence, value head) would leave the GPU short of work: the
    // transfer pass that makes segments independent is a second scan.
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long long seg_len = prefill_segment_tokens(p.n_seqs, p.h_v, p.total_tokens, sms);
    const bool segment = seg_len > 0;
    p.seg_tokens = segment ? (int)seg_len : 0x40000000;
    const long long slots = segment ? p.total_tokens / seg_len : 0;   // >= the segment boundaries
    const unsigned units = (unsigned)(slots + p.n_seqs);
    seg_list_kernel<<<1, 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // head groups on forked streams when there is a combine pass to hide
    const int groups = (slots > 0 && p.h_k % kHeadGroups == 0) ? kHeadGroups : 1;
    std::unique_lock<std::mutex> lock(g_side_mu, std::defer_lock);
    SideStreams* ss = nullptr;
    cudaStream_t st[kHeadGroups] = {stream};
    int forked = 1;   // streams that the caller's stream must join again
    if (groups > 1) {
      lock.lock();
      if ((e = side_streams_locked(dev, ss)) != cudaSuccess) return e;
      if ((e = cudaEventRecord(ss->fork, stream)) != cudaSuccess) return e;
      for (int g = 1; g < groups; ++g) {
        st[g] = ss->s[g - 1];
        if ((e = cudaStreamWaitEvent(st[g], ss->fork, 0)) != cudaSuccess) break;
        forked = g + 1;
      }
    }
    PrefillArgs pg[kHeadGroups];
    for (int g = 0; g < groups; ++g) {
      pg[g] = p;
      pg[g].nkh = p.h_k / groups;
      pg[g].kh0 = g * pg[g].nkh;
      pg[g].nh = pg[g].nkh * (p.h_v / p.h_k);
      pg[g].h0 = pg[g].kh0 * (p.h_v / p.h_k);
    }
    // On an error part-way, the streams already forked still join the caller's
    // stream, so that nothing enqueued on it afterwards overtakes their work.
    for (int g = 0; g < groups && e == cudaSuccess; ++g)
      e = launch_prefill_prep(pg[g], (unsigned)l.max_chunks, tm_qkv, st[g]);
    if (slots > 0) {   // some sequence may be longer than one segment
      for (int g = 0; g < groups && e == cudaSuccess; ++g) e = launch_prefill_scan(pg[g], true, units, tm_z, st[g]);
      for (int g = 0; g < groups && e == cudaSuccess; ++g) e = launch_prefill_combine(pg[g], (unsigned)slots, st[g]);
    }
    for (int g = 0; g < groups && e == cudaSuccess; ++g) e = launch_prefill_scan(pg[g], false, units, tm_z, st[g]);
    for (int g = 1; g < forked; ++g) {
      cudaError_t j = cudaEventRecord(ss->join[g - 1], st[g]);
      if (j == cudaSuccess) j = cudaStreamWaitEvent(stream, ss->join[g - 1], 0);
      if (e == cudaSuccess) e = j;
    }
    if (e != cudaSuccess) return e;
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  conv_state_kernel<<<dim3((unsigned)((Cc_ + 255) / 256), (unsigned)p.n_seqs), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
