// gdn_prefill_split.cu -- the chunked prefill as a chunk-parallel prep pass
// followed by state scans (sm_103a).
//
// In the chunked WY/UT form of the gated delta rule, most of a 64-token
// chunk's work does not depend on the state S0 entering it: the conv, SiLU
// and L2 norms, the gates and their cumulative sums gamma, the Gram products
// [K^; Q^] K^T, A and P, T = (I + A)^{-1}, and W = T diag(beta e^gamma) K^.
// What does depend on S0 is short and all tensor-core work:
//
//   Vn^T = V^T (T diag beta)^T + S0 (-W)^T        U, then the correction
//   O^T  = e^gamma (S0 Q^T) + Vn^T P^T            (output pass)
//   S    = e^{gamma_C} S0 + (Vn^T diag(e^{gamma_C - gamma})) K^
//
// The prep pass therefore computes the state-free part of every chunk of
// every sequence at once, one CTA per (chunk, key head) -- the q/k conv and
// the Gram product are shared by the value heads that read that key head --
// and stores it as per-chunk records (tiles in their shared-memory layout).
// The scan passes walk the chunks of each (segment, value head) in order and
// do only the products above, the record tiles of later chunks loading by
// bulk copies while the current chunk computes; in the output pass the gated
// RMSNorm epilogue of a chunk runs while the tensor core works on the next.
//
// The transfer pass (segments of a long sequence) runs the same scan in two
// independent tracks per segment: S from 0 with the real inputs, and X from
// the identity with v = 0, which yields the segment's affine map S_end =
// S_start X + S_end(0); the combine pass then chains the maps into every
// segment's true start state.
#include <cuda.h>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_launch.h"
#include "gdn_prefill.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

// ============================== prep pass ==============================

constexpr int kPrepThreads = 256;
constexpr int kPrepWarps = kPrepThreads / 32;
constexpr int kMaxG = 4;   // value heads per key head on the compiled path
// Shared memory (bytes from a 1024-aligned base), sized for three CTAs per SM:
// two raw staging blocks (k, then the bf16 K^ tile of the W products; q, then
// the v rows of the value heads in turn), the fp16 [K^ | Q^] tile of the Gram
// product and the gates.  The value heads then run in the Gram tile's space,
// two at a time, one per slot.
struct PrepLay {
  static constexpr uint32_t KQ16 = 0;       // fp16 [K^ | Q^], 64-column blocks 16 KB apart; then two head slots
  static constexpr uint32_t RAW = 34816;    // staging block b at RAW + b * RAW_STRIDE
  static constexpr uint32_t RAW_STRIDE = (RAW_BLK + 1023) / 1024 * 1024;
  static constexpr uint32_t KB = RAW;       // bf16 K^ [t][d_k], 64-column blocks 8 KB apart (head phase)
  static constexpr uint32_t GATE = RAW + RAW_STRIDE + RAW_BLK;   // per value head: fp32 gamma, beta, e^gamma [64]
  static constexpr uint32_t BYTES = GATE + kMaxG * 3 * 64 * 4 + 1024;   // + slack to align the base
  // Slot e of the head area, at AREA + e * UT_BYTES: a value head's A, T over it
  // (fp32, 17 KB), then T diag(beta e^gamma), then -W [d_k][t]
  static constexpr uint32_t AREA = KQ16;
};
static_assert(2 * UT_BYTES <= PrepLay::RAW - PrepLay::KQ16, "two head slots fit the Gram tile's space");
static_assert(16384 <= RAW_BLK, "the K^ tile fits a staging block");
static_assert(16384 <= UT_BYTES && UT_BYTES % 1024 == 0, "-W fits a slot; slots keep the tiles' alignment");
static_assert(PrepLay::RAW % 1024 == 0 && RAW_BLK % 128 == 0, "TMA destinations need 128-byte alignment");
static_assert(3 * (PrepLay::BYTES + 1024) <= 228 * 1024, "three prep CTAs per SM");
constexpr uint32_t TP_G = 0, TP_W = 64, TP_COLS = 128;   // TMEM: Gram [K^;Q^]K^T, W^T of the current head

// This lane's 4 channels ch .. ch+3 of the conv weight as stored (bf16 [channel][tap]),
// and unpacked to w[tap][channel].
struct ConvW4 {
  uint4 u0, u1;   // channels ch, ch+1 | ch+2, ch+3
};
__device__ __forceinline__ ConvW4 conv_weights_load(const uint16_t* conv_w, int ch) {
  return {*reinterpret_cast<const uint4*>(conv_w + (size_t)ch * kConvW),
          *reinterpret_cast<const uint4*>(conv_w + (size_t)(ch + 2) * kConvW)};
}
__device__ __forceinline__ void conv_weights(const ConvW4& cw, float (&w)[kConvW][4]) {
  const uint32_t wv[8] = {cw.u0.x, cw.u0.y, cw.u0.z, cw.u0.w, cw.u1.x, cw.u1.y, cw.u1.z, cw.u1.w};
#pragma unroll
  for (int e = 0; e < 4; ++e)
#pragma unroll
    for (int j = 0; j < kConvW; ++j) {
      const int k = e * kConvW + j;   // channel e, tap j
      w[j][e] = bf16_to_f32((k & 1) ? (wv[k >> 1] >> 16) : (wv[k >> 1] & 0xffffu));
    }
}

// Bounded wait for a shared-memory counter that other threads of the CTA
// raise (after a block-scope fence) to reach n; acquire ordering on success.
__device__ __forceinline__ bool wait_count(const int* ctr, int n) {
  const long long t0 = clock64();
  while (*reinterpret_cast<const volatile int*>(ctr) < n)
    if (clock64() - t0 > kWaitBudget) return false;
  __threadfence_block();
  return true;
}

// One CTA per (chunk, key head): the state-free part of the chunk for the G
// value heads that read this key head, stored as records.  Three CTAs share an
// SM, so one CTA's waits (a raw block in flight, a product, a barrier behind
// its slowest warp) leave the issue slots to the other two; within a CTA two
// groups of four warps each take every other value head and the v conv of the
// others, so that one group's solve, which keeps only a few warps busy, runs
// beside the other's conv.
__global__ void __launch_bounds__(kPrepThreads, 3)
    prep_kernel(const PrefillArgs p, const __grid_constant__ CUtensorMap tm_qkv) {
  using L_ = PrepLay;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t mbar;       // the Gram product done
  __shared__ __align__(8) uint64_t mb_raw[2];  // a staging block's raw rows landed
  __shared__ __align__(8) uint64_t mb_w[2];    // a value head's W product done (per group)
  __shared__ int raw_read[2];                  // warps done reading a staging block (cumulative)
  __shared__ int raw_issued[2];                // raw loads issued into a staging block
  __shared__ int w_read;                       // value heads whose W^T has been read out of TMEM
  __shared__ uint32_t tmem_base_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x / p.nkh, kh = p.kh0 + blockIdx.x % p.nkh;
  if (*p.status == GDN_ERR_DEVICE_BOUNDS) return;   // cu_seqlens rejected by the list kernel
  const int2 ce = p.chunk_list[c];
  if (ce.x < 0 || ce.x >= p.n_seqs) return;          // past the last chunk
  const int n = ce.x, t0 = ce.y;
  const int start = p.cu_seqlens[n], len = p.cu_seqlens[n + 1] - start;
  const int L = min(C, len - t0);
  const int G = p.h_v / p.h_k;
  const int Cq = p.h_k * kD, Cc = 2 * Cq + p.h_v * kD;
  const float* cs_seq = p.conv_state + (size_t)n * (kConvW - 1) * Cc;   // this sequence's carried conv state
  uint8_t* rkq = p.rec_kq + ((size_t)c * p.h_k + kh) * kRecKQ;

  const Smem sm = smem_aligned(smem_raw);

  if (tid == 0) {
    tc::mbar_init(&mbar, 1);
    tc::mbar_init(&mb_w[0], 1);
    tc::mbar_init(&mb_w[1], 1);
    w_read = 0;
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&mb_raw[b], 1);
      raw_read[b] = 0;
      raw_issued[b] = 1;   // k and q, issued below
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base_s, TP_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_s;
  const int quarter = warp & 3;   // TMEM lane quarter
  const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
  const int row = 32 * quarter + lane;
  const int y_raw = start + t0 - (kConvW - 1);      // first staged row (a chunk and its halo)
  // Staging block 0 takes the k rows (later the bf16 K^ tile), block 1 the q
  // rows and then the v rows of each value head in turn.
  auto raw_blk = [&](int b) { return sm.base + L_::RAW + b * L_::RAW_STRIDE; };
  if (tid == 32) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      mbar_expect_tx(&mb_raw[b], RAW_BLK);
      tma_load_2d(raw_blk(b), &tm_qkv, (b == 0 ? Cq : 0) + kh * kD, y_raw, &mb_raw[b]);
    }
  }
  // the k rows (block 0) or the q rows (block 1), each block's first load; on a
  // time-out the copy stays pending for the exit path
  auto wait_raw = [&](int b) -> bool { return __syncthreads_and(tc::mbar_wait(&mb_raw[b], 0, kWaitBudget)); };
  // the v rows of value head kh*G + g into block 1 (its earlier rows read)
  auto load_v = [&](int g) {
    tc::fence_proxy_async();
    mbar_expect_tx(&mb_raw[1], RAW_BLK);
    tma_load_2d(raw_blk(1), &tm_qkv, 2 * Cq + (kh * G + g) * kD, y_raw, &mb_raw[1]);
    __threadfence_block();
    atomicAdd(&raw_issued[1], 1);   // the other group may wait for this count
  };
  // Each warp done reading the q rows counts itself out; the last one issues
  // the first value head's v rows into the block.
  auto release_q = [&]() {
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&raw_read[1], 1) == kPrepWarps - 1) {
        __threadfence_block();
        load_v(0);
      }
    }
  };
  bool ok = true;
  // this lane's k and q conv weights, in flight while the gates run
  const ConvW4 cw_kq[2] = {conv_weights_load(p.conv_w, Cq + kh * kD + 4 * lane),
                           conv_weights_load(p.conv_w, kh * kD + 4 * lane)};

  // ---- gates and their cumulative sums, warp g for value head kh*G + g (meanwhile
  //      the raw rows land); the scan passes get e^gamma and e^{gamma_C - gamma} ----
  if (warp < G) {
    const int h = kh * G + warp;
    const float A_exp = __expf(p.A_log[h]);
    const float dtb = p.dt_bias[h];
    float g2[2], b2[2];
#pragma unroll
    for (int uu = 0; uu < 2; ++uu) {
      const int t = lane + 32 * uu;
      if (t < L) {
        const size_t pidx = (size_t)(start + t0 + t) * p.h_v + h;
        g2[uu] = -A_exp * softplus_gate(bf16_to_f32(p.a[pidx]) + dtb);
        b2[uu] = sigmoid_gate(bf16_to_f32(p.b[pidx]));
      } else {
        g2[uu] = 0.0f;
        b2[uu] = 0.0f;
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
    float* gam = sm.f32(L_::GATE + warp * 3 * 64 * 4);
    float* rg = reinterpret_cast<float*>(p.rec_v + ((size_t)c * p.h_v + h) * kRecV + kRecGate);
#pragma unroll
    for (int uu = 0; uu < 2; ++uu) {
      const int t = lane + 32 * uu;
      const float e1 = __expf(g2[uu]);
      gam[t] = g2[uu];
      gam[64 + t] = b2[uu];
      gam[128 + t] = e1;
      rg[t] = e1;
      rg[64 + t] = __expf(gC - g2[uu]);
    }
  }

  // ---- conv + SiLU + L2 norms, q then k: into the fp16 Gram tile, and in bf16
  //      straight into the record ----
  static_assert(C / 4 == 2 * kPrepWarps, "each warp takes two token quads of each block");
  const float qscale = rsqrtf((float)kD);
  // This lane's 4 columns (4 lane .. 4 lane + 3) in row tq + i of a tile in the
  // 128-byte swizzle: tq is a multiple of 4 whose bits 0-2 are the same for
  // every quad a warp takes, so the row-within-atom part of the offset is fixed
  // per thread (quad_off) and the rest is (tq >> 3) * 1024 (tc::sw128_off, with
  // the tile's 64-column block stride kb_stride).
  auto quad_off = [&](int tq, int i, uint32_t kb_stride) -> uint32_t {
    const int r7 = (tq & 7) + i;
    return (uint32_t)(lane >> 4) * kb_stride + (uint32_t)r7 * 128u +
           ((uint32_t)(((lane >> 1) & 7) ^ r7) << 4) + ((uint32_t)(lane & 1) << 3);
  };
  uint32_t qk_off[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) qk_off[i] = quad_off(4 * warp, i, 16384);
  // q first (block 1), so that its block is free for the first value head's v
  // rows, loading behind the k conv
#pragma unroll
  for (int bi = 0; bi < 2; ++bi) {
    const int blk = 1 - bi;   // 0: k, 1: q
    if (!wait_raw(blk)) {
      ok = false;
      break;
    }
    const int ch = (blk == 0 ? Cq : 0) + kh * kD + 4 * lane;
    float w[kConvW][4];
    conv_weights(cw_kq[blk], w);
#pragma unroll 1
    for (int qd = 0; qd < 2; ++qd) {
      const int tq = 4 * (warp + kPrepWarps * qd);
      float y[4][4];
      conv_quad_staged(raw_blk(blk), cs_seq + ch, Cc, t0, L, tq, lane, w, y);
      float rn[4];
      l2_rnorm4(y, p.l2_eps, blk == 0 ? 1.0f : qscale, lane, rn);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 r2 = make_float2(rn[i], rn[i]);
        const float2 a = __fmul2_rn(make_float2(y[i][0], y[i][1]), r2);
        const float2 b = __fmul2_rn(make_float2(y[i][2], y[i][3]), r2);
        const uint32_t o16 = qk_off[i] + (uint32_t)(tq >> 3) * 1024u + (blk == 0 ? 0u : 8192u);
        store_f16x4(sm.base + L_::KQ16, o16, a.x, a.y, b.x, b.y);
        store_bf16x4(rkq, o16, a.x, a.y, b.x, b.y);
      }
    }
    if (blk == 1) release_q();
  }
  sync_for_mma();   // the Gram tile is written
  if (ok && tid == 0) {
    // Gram [K^; Q^] K^T in fp16 (rows 0-63: K^K^T, 64-127: Q^K^T)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t a = sm.addr + L_::KQ16 + (k >> 2) * 16384 + (k & 3) * 32;
      tc::mma_bf16(tmem + TP_G, tc::sdesc_at(D_K, a), tc::sdesc_at(D_K, a), ID_GRAM, k > 0);
    }
    tc::mma_commit(&mbar);
  }

  if (ok) {
    // the bf16 K^ tile of the W products, back from this CTA's record into block
    // 0, whose k rows every warp has read (64-column blocks 16 KB apart there,
    // 8 KB here)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = tid + j * kPrepThreads, kb = i >> 9, off = (i & 511) * 16;
      *reinterpret_cast<uint4*>(sm.base + L_::KB + kb * 8192 + off) =
          __ldcg(reinterpret_cast<const uint4*>(rkq + kb * 16384 + off));
    }
  }
  sync_for_mma();   // the K^ tile is written (the W products read it)

  // ---- two groups of four warps from here on (e = 0: warps 0-3, e = 1: warps
  //      4-7), each on its own named barrier (1 + e) and with its own slot of
  //      the head area.  Step g of group e is value head g (A, P, the solve, T
  //      diag(beta), W) when g % 2 == e, else the v conv of value head g, so
  //      that each group does about half of both kinds of work.  The v rows of
  //      the heads pass through staging block 1 in head order, each load issued
  //      by the group that read the previous one; the W^T products take the
  //      TMEM columns TP_W in head order, each issued once the group of the
  //      head before has read its W^T out. ----
  const int grp = warp >> 2, gtid = tid & 127, gwarp = warp & 3;
  const int bar = 1 + grp;
  float* M = sm.f32(L_::AREA + grp * UT_BYTES);   // A, T over it, then T diag(beta e^gamma), then -W
  uint8_t* wn = sm.base + L_::AREA + grp * UT_BYTES;
  const uint32_t tw = sm.addr + L_::AREA + grp * UT_BYTES;
  const uint32_t tm_w = tmem + TP_W;
  // one thread's bounded wait for a shared counter to reach n, then a barrier of
  // the group that tells everyone whether it did
  auto group_wait_count = [&](const int* ctr, int n) -> bool {
    bool got = true;
    if (gtid == 0) got = wait_count(ctr, n);
    return group_sync_and<128>(bar, got);
  };
  bool gram_waited = false;
  uint32_t wphase = 0;
  int heads = 0;   // value heads this group has done
#pragma unroll 1
  for (int g = 0; g < G && ok; ++g) {
    const int h = kh * G + g;
    uint8_t* rv = p.rec_v + ((size_t)c * p.h_v + h) * kRecV;
    if ((g & 1) != grp) {
      // ---- the v conv of value head g, straight into its record, from block 1
      //      (its rows the (g + 2)-th load into the block: q, then v_0 .. v_g) ----
      const int ch = 2 * Cq + h * kD + 4 * lane;
      const ConvW4 cw_v = conv_weights_load(p.conv_w, ch);
      ok = group_wait_count(&raw_issued[1], 2 + g);
      if (ok) ok = group_sync_and<128>(bar, tc::mbar_wait(&mb_raw[1], (1 + g) & 1, kWaitBudget));
      if (!ok) break;
      float w[kConvW][4];
      conv_weights(cw_v, w);
      uint8_t* vh = rv + kRecVH;
      uint32_t v_off[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v_off[i] = quad_off(4 * gwarp, i, 8192);
#pragma unroll 1
      for (int qd = 0; qd < 4; ++qd) {
        const int tq = 4 * (gwarp + 4 * qd);
        float y[4][4];
        conv_quad_staged(raw_blk(1), cs_seq + ch, Cc, t0, L, tq, lane, w, y);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          store_bf16x4(vh, v_off[q] + (uint32_t)(tq >> 3) * 1024u, y[q][0], y[q][1], y[q][2], y[q][3]);
      }
      group_sync<128>(bar);   // every warp of the group has read the block
      if (gtid == 0 && g + 1 < G) load_v(g + 1);
      continue;
    }
    // ---- value head g ----
    if (!gram_waited) {   // the Gram product (and its tile's space is free)
      ok = group_sync_and<128>(bar, tc::mbar_wait(&mbar, 0, kWaitBudget));
      tc::fence_after_sync();
      gram_waited = true;
      if (!ok) break;
    }
    const float* gam = sm.f32(L_::GATE + g * 3 * 64 * 4);
    const float* bet = gam + 64;
    const float* eg = gam + 128;
    if (heads >= 1) {   // this group's previous -W tile has left its slot
      if (gtid == 0) bulk_wait_read();
      group_sync<128>(bar);
    }
    // ---- A (fp32, below its diagonal: the solve reads nothing else) and P
    //      (bf16, stored straight into the record) from the Gram rows: lane
    //      quarters 0-1 hold K^K^T rows, 2-3 Q^K^T rows; P's rows 0-31 are
    //      zero right of column 31 ----
    {
      uint8_t* prec = rv + kRecP;
      const int t = row & 63;
      const float gt = gam[t];
      const float bt = bet[t];
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        const int c0 = 32 * hf;
        if (t < 32 && hf == 1) {
          if (quarter >= 2) {
#pragma unroll
            for (int m = 0; m < 4; ++m)
              *reinterpret_cast<uint4*>(prec + tc::sw128_off(t, c0 + 8 * m, 0)) = make_uint4(0, 0, 0, 0);
          }
          continue;
        }
        float v[32];
        tc::tmem_ld32(tmem + lane_base + TP_G + c0, v);
        if (quarter < 2) {
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            float a[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) a[e] = bt * __expf(gt - gam[c0 + 4 * m + e]) * v[4 * m + e];
            ut_st4(M, t, c0 + 4 * m, a[0], a[1], a[2], a[3]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int s = c0 + i;
            v[i] = keep_if_le(v[i] * __expf(gt - gam[s]), s, t);
          }
#pragma unroll
          for (int m = 0; m < 4; ++m) store_bf16x8(prec, tc::sw128_off(t, c0 + 8 * m, 0), v + 8 * m);
        }
      }
    }
    group_sync<128>(bar);   // A is written

    // ---- T = (I + A)^{-1} in place; T diag(beta) -> record, T diag(beta e^gamma)
    //      over T once every thread has read its rows ----
    solve_unit_lower<128>(M, gtid, bar);
    {
      uint4 tw8[4];   // this thread's T diag(beta e^gamma) groups, bf16, held across the barrier
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int e = gtid + q4 * 128, t = e >> 3, c8 = (e & 7) * 8;
        const float4 lo = ut_ld4(M, t, c8), hi = ut_ld4(M, t, c8 + 4);
        const float tv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        float xb[8], xw[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          xb[q] = keep_if_le(tv[q], c8 + q, t) * bet[c8 + q];   // T is zero above its diagonal
          xw[q] = xb[q] * eg[c8 + q];
        }
        store_bf16x8(rv + kRecTB, tc::sw128_off(t, c8, 0), xb);
        tw8[q4] = make_uint4(pack_bf16x2(xw[0], xw[1]), pack_bf16x2(xw[2], xw[3]), pack_bf16x2(xw[4], xw[5]),
                             pack_bf16x2(xw[6], xw[7]));
      }
      group_sync<128>(bar);   // T is read
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int e = gtid + q4 * 128, t = e >> 3, c8 = (e & 7) * 8;
        *reinterpret_cast<uint4*>(wn + tc::sw128_off(t, c8, 0)) = tw8[q4];
      }
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    // the W^T columns are free once value head g - 1's W^T has been read out
    ok = group_wait_count(&w_read, g);
    tc::fence_after_sync();
    if (!ok) break;
    if (gtid == 0) {
      // W^T = K^T (T diag(beta e^gamma))^T
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc::mma_bf16(tm_w, tc::sdesc_at(D_MN_V, sm.addr + L_::KB + k * 2048), tc::sdesc_at(D_K, tw + k * 32),
                     ID_MN_A, k > 0);
      tc::mma_commit(&mb_w[grp]);
    }
    ok = group_sync_and<128>(bar, tc::mbar_wait(&mb_w[grp], wphase, kWaitBudget));
    wphase ^= 1u;
    tc::fence_after_sync();
    if (!ok) break;

    // ---- -W tile [d_k][t] over T diag(beta e^gamma), which the product has
    //      consumed: a thread's TMEM lane is its d_k row, each 32 columns 64
    //      contiguous bytes ----
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {
      float v[32];
      tc::tmem_ld32(tm_w + lane_base + 32 * hf, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = -v[i];
#pragma unroll
      for (int m = 0; m < 4; ++m) store_bf16x8(wn, tc::sw128_off(row, 32 * hf + 8 * m, 0), v + 8 * m);
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();   // W^T is read before the next head's product overwrites it
    group_sync<128>(bar);
    tc::fence_after_sync();
    if (gtid == 0) {
      __threadfence_block();
      atomicAdd(&w_read, 1);
      bulk_store(rv + kRecWN, wn, 16384);
      bulk_commit();
    }
    ++heads;
  }
  ok = __syncthreads_and(ok);

  if (gtid == 0) bulk_wait_read();   // the record copies have read this CTA's shared memory
  if (tid == 0) {
    if (!ok) record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
    // a raw copy still in flight after a time-out must land before the shared
    // memory goes away: each load into a block was issued after the one before
    // it had landed, so only the last one can be pending
    for (int b = 0; b < 2; ++b) tc::mbar_wait(&mb_raw[b], (raw_issued[b] - 1) & 1, kWaitBudget);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TP_COLS);
}

// ============================== output pass ==============================

// The output pass, warp-specialised.  One CTA per (segment, value head): 16
// worker warps (4 per TMEM lane quarter) make the operand tiles from the
// accumulators, stage O and run the gated RMSNorm epilogue; one more warp
// issues the tensor-core products and another the bulk copies (issuing a copy
// can stall, and the products are on the chain).  They meet on mbarriers, so
// the per-chunk chain is only
//   [U, Vn^T] -> Vn^T tiles -> [state update] -> state tile -> next [U, Vn^T]
// while O1 = S0 Q^T, O2 = Vn^T P^T, the O staging and the epilogue run beside
// it (O1 double-buffered in TMEM).  Every wait is bounded; the workers agree on
// a time-out at their own barriers.
constexpr int kOutWorkers = 512;              // 16 warps
constexpr int kOutThreads = kOutWorkers + 64; // + the MMA warp and the copy warp
static_assert(kOutWorkers / 32 * 4 == C, "the epilogue gives each worker warp 4 of a chunk's tokens");
struct ScanLay {
  static constexpr uint32_t S = 0;          // S bf16 [d_v][d_k], K blocks 16 KB apart
  static constexpr uint32_t KQ = 32768;     // two [K^ | Q^] buffers
  static constexpr uint32_t KQ_BUF = 32768;
  static constexpr uint32_t WN = 98304;     // -W | V^ | T diag(beta): the record's first 40 KB, one copy
  static constexpr uint32_t VH = WN + kRecVH;
  static constexpr uint32_t TB = WN + kRecTB;
  static constexpr uint32_t P = WN + 40960;
  static constexpr uint32_t GT = P + 8192;  // three gate buffers: e^gamma [64], e^{gamma_C - gamma} [64]
  static constexpr uint32_t Z = GT + 2048;  // two z buffers, bf16 [64][128]
  static constexpr uint32_t VN = Z + 32768;     // Vn^T [d_v][t]
  static constexpr uint32_t VNS = VN + 16384;   // Vn^T diag(e^{gamma_C - gamma})
  static constexpr uint32_t OST = VN;           // O fp32 [64][LDO], over VN and VNS once they are consumed
  static constexpr uint32_t NW = VNS + 16384;   // RMSNorm weight
  static constexpr uint32_t BYTES = NW + 512 + 1024;
};
static_assert(ScanLay::WN % 1024 == 0 && ScanLay::VH % 1024 == 0 && ScanLay::TB % 1024 == 0 &&
                  ScanLay::VN % 1024 == 0 && ScanLay::VNS % 1024 == 0 && ScanLay::KQ % 1024 == 0 &&
                  ScanLay::P % 1024 == 0,
              "operand tiles need 1024-byte alignment");
static_assert(ScanLay::Z % 128 == 0, "TMA destination alignment");
static_assert(ScanLay::OST + 64 * LDO * 4 <= ScanLay::NW, "O staging overlaps the norm weight");
static_assert(ScanLay::BYTES <= 227 * 1024, "shared memory");
// TMEM columns: S, U / Vn^T, O1 (two buffers), O2
constexpr uint32_t TS_S = 0, TS_U = 128, TS_O1 = 192, TS_O2 = 320, TS_COLS = 512;

// Block-wide sync for the tensor core that also ANDs a per-thread flag.
__device__ __forceinline__ bool sync_for_mma_and(bool ok) {
  tc::fence_proxy_async();
  tc::fence_before_sync();
  const bool all = __syncthreads_and(ok);
  tc::fence_after_sync();
  return all;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(mbar)) : "memory");
}

// A worker warp's signal: its generic smem writes and tensor-memory traffic are
// ordered before the arrival (one per warp).
__device__ __forceinline__ void warp_signal(uint64_t* mbar, int lane) {
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive(mbar);
}

__global__ void __launch_bounds__(kOutThreads, 1)
    output_kernel(const PrefillArgs p, const __grid_constant__ CUtensorMap tm_z) {
  using M = ScanLay;
  extern __shared__ uint8_t smem_raw[];
  // copies landed
  __shared__ __align__(8) uint64_t mb_kq[2], mb_a, mb_g[3], mb_p, mb_z[2];
  // products done: [U, Vn^T]; [state update] (and O1 before it); [O2] (and all before)
  __shared__ __align__(8) uint64_t mb_b1, mb_b2, mb_o;
  // worker warps done (16 arrivals): Vn^T tiles, state tile, O read, epilogue
  __shared__ __align__(8) uint64_t mb_vn, mb_s, mb_or, mb_ep;
  __shared__ __align__(8) uint64_t mb_fin;   // after a time-out: every product issued has finished
  __shared__ uint32_t tmem_base_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = blockIdx.x / p.nh, h = p.h0 + blockIdx.x % p.nh;
  if (u >= p.seg_list[0]) return;
  const Seg sg = load_seg(p.seg_list, u);
  const int n = sg.n;
  const int G = p.h_v / p.h_k, kh = h / G;
  const int start = p.cu_seqlens[n];
  const int seg_end = sg.begin + sg.len;
  const int nch = (sg.len + C - 1) / C;

  // where the state comes from and goes to (the caller's state is row-major,
  // the workspace slots tiled)
  const float* S_init;
  float* S_final;
  float* ssm = p.ssm_state + ((size_t)n * p.h_v + h) * kD * kD;
  const bool init_tiled = sg.nsig > 1;
  if (sg.nsig == 1) {
    S_init = ssm;
    S_final = ssm;
  } else {
    S_init = sg.sigma == 0 ? xfer_ptr(p, sg.k0, h, 2) : xfer_ptr(p, sg.k0 + sg.sigma - 1, h, 1);
    S_final = sg.sigma == sg.nsig - 1 ? ssm : nullptr;
  }

  const Smem sm = smem_aligned(smem_raw);
  float* Ost = sm.f32(M::OST);
  float* nw = sm.f32(M::NW);
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&mb_kq[i], 1);
      tc::mbar_init(&mb_z[i], 1);
    }
    for (int i = 0; i < 3; ++i) tc::mbar_init(&mb_g[i], 1);
    tc::mbar_init(&mb_a, 1);
    tc::mbar_init(&mb_p, 1);
    tc::mbar_init(&mb_b1, 1);
    tc::mbar_init(&mb_b2, 1);
    tc::mbar_init(&mb_o, 1);
    tc::mbar_init(&mb_fin, 1);
    tc::mbar_init(&mb_vn, kOutWorkers / 32);
    tc::mbar_init(&mb_s, kOutWorkers / 32);
    tc::mbar_init(&mb_or, kOutWorkers / 32);
    tc::mbar_init(&mb_ep, kOutWorkers / 32);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base_s, TS_COLS);
  if (tid < kD) nw[tid] = p.norm_w[tid];
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_s;
  auto wt = [&](uint64_t* mb, uint32_t k) -> bool {   // the k-th completion of mb (parity k & 1)
    return tc::mbar_wait(mb, k & 1u, kWaitBudget);
  };
  bool ok = true;

  if (warp == kOutWorkers / 32) {
    // ================= the MMA warp (one lane) =================
    // Each wait below is for a completion whose successor needs something this
    // lane issues only afterwards, so the barrier is never two phases on.
    if (lane == 0) {
      uint32_t issued_mma = 0;
      // U = V^T (T diag beta)^T needs only the records: each chunk's is issued
      // ahead, before the state tile it waits for
      auto issue_u = [&](int j) -> bool {
        if (!wt(&mb_a, j)) return false;
        tc::fence_after_sync();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_bf16(tmem + TS_U, tc::sdesc_at(D_MN_V, sm.addr + M::VH + k * 2048),
                       tc::sdesc_at(D_K, sm.addr + M::TB + k * 32), ID_MN_A, k > 0);
        ++issued_mma;
        return true;
      };
      ok = issue_u(0);
      for (int j = 0; j < nch && ok; ++j) {
        const uint32_t kq = sm.addr + M::KQ + (j & 1) * M::KQ_BUF;
        // this chunk's [K^ | Q^] and the workers' state tile
        if (!(wt(&mb_kq[j & 1], j >> 1) && wt(&mb_s, j))) { ok = false; break; }
        tc::fence_after_sync();
        // [Vn^T = U + S0 (-W)^T]
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t kb = k >> 2, ks = (k & 3) * 32;
          tc::mma_bf16(tmem + TS_U, tc::sdesc_at(D_K, sm.addr + M::S + kb * 16384 + ks),
                       tc::sdesc_at(D_MN_W, sm.addr + M::WN + k * 2048), ID_KMN, 1u);
        }
        tc::mma_commit(&mb_b1);
        // O1 = S0 Q^T into its buffer, which the workers read at chunk j - 2 (the
        // wait for that read was the O2 wait of chunk j - 1)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t kb = k >> 2, ks = (k & 3) * 32;
          tc::mma_bf16(tmem + TS_O1 + 64 * (j & 1), tc::sdesc_at(D_K, sm.addr + M::S + kb * 16384 + ks),
                       tc::sdesc_at(D_K, kq + kb * 16384 + 8192 + ks), ID_KK, k > 0);
        }
        // the workers' Vn^T tiles, and P
        if (!(wt(&mb_vn, j) && wt(&mb_p, j))) { ok = false; break; }
        tc::fence_after_sync();
        // [S += Vn^T diag(e^{gamma_C - gamma}) K^]
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_bf16(tmem + TS_S, tc::sdesc_at(D_K, sm.addr + M::VNS + k * 32),
                       tc::sdesc_at(D_MN_KQ, kq + k * 2048), ID_MN_B, 1u);
        tc::mma_commit(&mb_b2);
        // O2 = Vn^T P^T, once the workers have read O2 of chunk j - 1
        if (j >= 1 && !wt(&mb_or, j - 1)) { ok = false; break; }
        tc::fence_after_sync();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_bf16(tmem + TS_O2, tc::sdesc_at(D_K, sm.addr + M::VN + k * 32),
                       tc::sdesc_at(D_K, sm.addr + M::P + k * 32), ID_KK, k > 0);
        tc::mma_commit(&mb_o);
        // the next chunk's U (TS_U was read for the Vn^T tiles)
        if (j + 1 < nch && !issue_u(j + 1)) { ok = false; break; }
      }
      if (!ok) {
        record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
        // the products issued finish (bounded) before the tensor memory is freed
        if (issued_mma > 0) {
          tc::mma_commit(&mb_fin);
          wt(&mb_fin, 0);
        }
      }
    }
    __syncwarp();
  } else if (warp == kOutWorkers / 32 + 1) {
    // ================= the copy warp (one lane) =================
    // Every buffer is refilled once a product barrier shows its last reader done:
    // -W | V^ | T diag(beta) after [U, Vn^T] (b1); P and the [K^ | Q^] buffer after
    // O2 (o), which follows the state update, O1 and -- through the MMA warp's own
    // waits -- the workers' O read of the previous chunk (its gates) and their
    // previous epilogue (its z).  The successor of each completion waited for needs
    // a copy issued after the wait, so the barrier is never two phases on.
    if (lane == 0) {
      auto rec_kq = [&](int j) { return p.rec_kq + ((size_t)(sg.c0 + j) * p.h_k + kh) * kRecKQ; };
      auto rec_v = [&](int j) { return p.rec_v + ((size_t)(sg.c0 + j) * p.h_v + h) * kRecV; };
      uint32_t i_kq[2] = {0, 0}, i_a = 0, i_g0 = 0, i_g1 = 0, i_g2 = 0, i_p = 0, i_z[2] = {0, 0};   // copies issued
      auto load_kq = [&](int j) {
        bulk_load(sm.base + M::KQ + (j & 1) * M::KQ_BUF, rec_kq(j), kRecKQ, &mb_kq[j & 1]);
        ++i_kq[j & 1];
      };
      auto load_a = [&](int j) {
        bulk_load(sm.base + M::WN, rec_v(j), kRecP, &mb_a);
        ++i_a;
      };
      auto load_g = [&](int j) {
        const int q = j % 3;
        bulk_load(sm.base + M::GT + q * 512, rec_v(j) + kRecGate, kRecGateBytes, &mb_g[q]);
        if (q == 0) ++i_g0; else if (q == 1) ++i_g1; else ++i_g2;
      };
      auto load_p = [&](int j) {
        bulk_load(sm.base + M::P, rec_v(j) + kRecP, 8192, &mb_p);
        ++i_p;
      };
      auto load_z = [&](int j) {
        mbar_expect_tx(&mb_z[j & 1], C * kD * 2);
        tma_load_2d(sm.base + M::Z + (j & 1) * 16384, &tm_z, h * kD, start + sg.begin + C * j, &mb_z[j & 1]);
        ++i_z[j & 1];
      };
      load_a(0);
      load_kq(0);
      load_g(0);
      load_p(0);
      load_z(0);
      if (nch > 1) {
        load_kq(1);
        load_g(1);
        load_z(1);
      }
      for (int j = 0; j + 1 < nch; ++j) {
        if (!wt(&mb_b1, j)) { ok = false; break; }
        load_a(j + 1);
        if (!wt(&mb_o, j)) { ok = false; break; }
        load_p(j + 1);
        if (j >= 1) load_z(j + 1);
        if (j + 2 < nch) {
          load_kq(j + 2);
          load_g(j + 2);
        }
      }
      if (!ok) {
        record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
        // the copies this CTA started land (bounded) before its shared memory goes away
        auto drain = [&](uint64_t* mb, uint32_t issued) {
          if (issued > 0) wt(mb, issued - 1);
        };
        drain(&mb_kq[0], i_kq[0]);
        drain(&mb_kq[1], i_kq[1]);
        drain(&mb_a, i_a);
        drain(&mb_g[0], i_g0);
        drain(&mb_g[1], i_g1);
        drain(&mb_g[2], i_g2);
        drain(&mb_p, i_p);
        drain(&mb_z[0], i_z[0]);
        drain(&mb_z[1], i_z[1]);
      }
    }
    __syncwarp();
  } else {
    // ================= the worker warps =================
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const int row = 32 * (warp & 3) + lane;   // TMEM lane this thread reads
    const int part = warp >> 2;               // which quarter of a lane quarter's columns
    // the initial state: bf16 into the operand tile, and into TMEM in fp32 already
    // scaled by the first chunk's total decay (the state update adds to e^{gamma_C} S0;
    // each chunk's end scales for the next one)
    ok = wt(&mb_g[0], 0);
    {
      const float dC0 = sm.f32(M::GT)[C - 1];
      const int col0 = part * 32;
      float v[32];
      load_state_row(S_init, init_tiled, row, col0, v);
#pragma unroll
      for (int m = 0; m < 4; ++m) store_bf16x8(sm.base + M::S, tc::sw128_off(row, col0 + 8 * m, 16384), v + 8 * m);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= dC0;
      tc::tmem_st32(tmem + lane_base + TS_S + col0, v);
    }
    warp_signal(&mb_s, lane);

    for (int j = 0; j < nch; ++j) {
      const float* eg = sm.f32(M::GT + (j % 3) * 512);
      const float* egc = eg + 64;
      // ---- Vn^T tiles, plain and decay-weighted, row = d_v index ----
      ok = wt(&mb_b1, j) && wt(&mb_g[j % 3], j / 3) && ok;
      tc::fence_after_sync();
      {
        float v[16], vs[16];
        tc::tmem_ld16(tmem + lane_base + TS_U + part * 16, v);
        // (the multiplies two per packed fp32x2 instruction, each rounding as
        // the scalar one would, here and below)
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          const float4 e4 = *reinterpret_cast<const float4*>(egc + part * 16 + i);
          const float2 a = __fmul2_rn(make_float2(v[i], v[i + 1]), make_float2(e4.x, e4.y));
          const float2 b = __fmul2_rn(make_float2(v[i + 2], v[i + 3]), make_float2(e4.z, e4.w));
          vs[i] = a.x; vs[i + 1] = a.y; vs[i + 2] = b.x; vs[i + 3] = b.y;
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint32_t off = tc::sw128_off(row, part * 16 + 8 * m, 0);
          store_bf16x8(sm.base + M::VN, off, v + 8 * m);
          store_bf16x8(sm.base + M::VNS, off, vs + 8 * m);
        }
      }
      warp_signal(&mb_vn, lane);
      // ---- the new state -> bf16 operand tile, and in TMEM scaled by the next
      //      chunk's total decay ----
      ok = wt(&mb_b2, j) && ok;
      tc::fence_after_sync();
      if (j + 1 < nch) {
        ok = wt(&mb_g[(j + 1) % 3], (j + 1) / 3) && ok;
        const float dC = sm.f32(M::GT + ((j + 1) % 3) * 512)[C - 1];
        float v[32];
        const uint32_t ta = tmem + lane_base + TS_S + part * 32;
        tc::tmem_ld32(ta, v);
#pragma unroll
        for (int m = 0; m < 4; ++m)
          store_bf16x8(sm.base + M::S, tc::sw128_off(row, part * 32 + 8 * m, 16384), v + 8 * m);
        const float2 dC2 = make_float2(dC, dC);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 a = __fmul2_rn(make_float2(v[i], v[i + 1]), dC2);
          v[i] = a.x; v[i + 1] = a.y;
        }
        tc::tmem_st32(ta, v);
        warp_signal(&mb_s, lane);
      }
      // ---- O = e^gamma O1 + O2 -> fp32 staging (over the Vn^T tiles, consumed) ----
      ok = wt(&mb_o, j) && ok;
      tc::fence_after_sync();
      {
        float o1[16], o2[16];
        tc::tmem_ld16(tmem + lane_base + TS_O1 + 64 * (j & 1) + part * 16, o1);
        tc::tmem_ld16(tmem + lane_base + TS_O2 + part * 16, o2);
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const int t = part * 16 + i;
          const float2 o = __ffma2_rn(make_float2(eg[t], eg[t + 1]), make_float2(o1[i], o1[i + 1]),
                                      make_float2(o2[i], o2[i + 1]));
          Ost[t * LDO + row] = o.x;
          Ost[(t + 1) * LDO + row] = o.y;
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&mb_or);
      if (!group_sync_and<kOutWorkers>(1, ok)) { ok = false; break; }   // the O staging is complete
      // ---- the gated RMSNorm epilogue, a warp per 4 tokens and 4 channels per lane ----
      ok = wt(&mb_z[j & 1], j >> 1) && ok;
      {
        const int t0e = sg.begin + C * j, Le = min(C, seg_end - t0e);
        const uint8_t* zb = sm.base + M::Z + (j & 1) * 16384;
        const int tq = 4 * warp;
        float o[4][4], ss[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 o4 = reinterpret_cast<const float4*>(Ost + (tq + i) * LDO)[lane];
          o[i][0] = o4.x; o[i][1] = o4.y; o[i][2] = o4.z; o[i][3] = o4.w;
        }
#pragma unroll
        for (int i = 0; i < 4; i += 2) {   // tokens i and i + 1, each summed in channel order
          float2 q = __fmul2_rn(make_float2(o[i][0], o[i + 1][0]), make_float2(o[i][0], o[i + 1][0]));
#pragma unroll
          for (int e = 1; e < 4; ++e)
            q = __ffma2_rn(make_float2(o[i][e], o[i + 1][e]), make_float2(o[i][e], o[i + 1][e]), q);
          ss[i] = q.x;
          ss[i + 1] = q.y;
        }
        const float r = rsqrtf(warp_sum4(ss, lane) * (1.0f / kD) + p.rms_eps);
        const float4 w4 = reinterpret_cast<const float4*>(nw)[lane];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float rstd = __shfl_sync(0xffffffffu, r, token_lane(i));
          const uint2 zr = *reinterpret_cast<const uint2*>(zb + (tq + i) * 256 + lane * 8);
          float g[4] = {bf16_to_f32(zr.x & 0xffffu), bf16_to_f32(zr.x >> 16), bf16_to_f32(zr.y & 0xffffu),
                        bf16_to_f32(zr.y >> 16)};
          silu4(g);
          const float2 r2 = make_float2(rstd, rstd);
          const float2 p0 = __fmul2_rn(__fmul2_rn(__fmul2_rn(make_float2(o[i][0], o[i][1]), r2),
                                                  make_float2(w4.x, w4.y)), make_float2(g[0], g[1]));
          const float2 p1 = __fmul2_rn(__fmul2_rn(__fmul2_rn(make_float2(o[i][2], o[i][3]), r2),
                                                  make_float2(w4.z, w4.w)), make_float2(g[2], g[3]));
          uint2 ov;
          ov.x = pack_bf16x2(p0.x, p0.y);
          ov.y = pack_bf16x2(p1.x, p1.y);
          if (tq + i < Le)
            *reinterpret_cast<uint2*>(p.out + ((size_t)(start + t0e + tq + i) * p.h_v + h) * kD + 4 * lane) = ov;
        }
      }
      if (!group_sync_and<kOutWorkers>(1, ok)) { ok = false; break; }   // the O staging and z are read
      __syncwarp();
      if (lane == 0) mbar_arrive(&mb_ep);
    }
    if (!ok) {
      if (tid == 0) record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
    } else if (S_final != nullptr) {
      // final state back to the caller (the last segment of a sequence)
      float v[32];
      tc::tmem_ld32(tmem + lane_base + TS_S + part * 32, v);
      store_state_row(S_final, false, row, part * 32, v);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TS_COLS);
}

// ============================== transfer pass ==============================

// The transfer pass as two independent tracks per (non-last segment, value
// head), one CTA each, so two fit on an SM:
//   track S: S from 0 with the real inputs   -> the segment's end state S_end(0)
//   track X: X from the identity with v = 0   -> the segment's map X
// Per chunk, track S: U = V^T (T diag beta)^T, Vn^T = U + S (-W)^T, S <-
// e^{gamma_C} S + (Vn^T diag(e^{gamma_C - gamma})) K^; track X the same with
// v = 0 (no U).
//
// Warp-specialised like the output pass: 8 worker warps make the Vn^T and state
// tiles from the accumulators, one warp issues the tensor-core products and one
// the bulk copies; they meet on mbarriers.  The chain per chunk is [S (-W)^T] ->
// Vn^T tile -> [state update] -> state tile; U of the next chunk, which needs
// only its records, is issued while the state tile is made.  Each wait is for a
// completion whose successor needs something issued only after the wait, so a
// barrier is never two phases on.
constexpr int kXferWorkers = 256;                 // 8 warps: 2 per TMEM lane quarter
constexpr float kNegligibleLogDecay = -160.0f;    // e^-160 < 1e-69

// The last chunk j (0 <= j < n) of a segment such that the gamma_C of chunks
// j .. n-1 sum to less than kNegligibleLogDecay, or -1.  rec: the gate-bearing
// record of the segment's first chunk, stride bytes between chunks.  Every
// thread of the block calls it and gets the same answer.  Each gamma_C <= 0, so
// the suffix sums fall as j falls and the chunks are scanned from the end, a
// block-sized tile at a time, until the sum crosses the bound.
__device__ int decayed_prefix(const uint8_t* rec, size_t stride, int n) {
  __shared__ float s_warp[32];
  __shared__ int s_found;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = (blockDim.x + 31) >> 5;
  float run = 0.0f;   // the sum over the tiles already scanned (the same on every thread)
  int found = -1;
  for (int base = n - 1; base >= 0 && found < 0; base -= (int)blockDim.x) {
    const int j = base - tid;   // thread i takes the i-th chunk from the tile's end
    float g = 0.0f;
    if (j >= 0) {
      const float e = *reinterpret_cast<const float*>(rec + (size_t)j * stride + kRecGate + (C - 1) * 4);
      g = e > 0.0f ? __logf(e) : -INFINITY;
    }
    // inclusive prefix sum over the tile in thread order
    float x = g;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    float before = 0.0f;
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    const float suffix = run + before + x;   // T_j for this thread's chunk
    // the sums fall with the thread index: count those still above the bound
    const int above = __syncthreads_count(j >= 0 && suffix >= kNegligibleLogDecay);
    if (above < (int)blockDim.x && base - above >= 0) found = base - above;
    float tile = 0.0f;
    for (int w = 0; w < nw; ++w) tile += s_warp[w];
    run += tile;
    __syncthreads();   // s_warp is rewritten by the next tile
  }
  if (tid == 0) s_found = found;
  __syncthreads();
  return s_found;
}
constexpr int kXferThreads = kXferWorkers + 64;   // + the MMA warp and the copy warp
struct XferLay {
  static constexpr uint32_t ST = 0;          // the tracked state, bf16 [128][128], K blocks 16 KB apart
  static constexpr uint32_t KH = 32768;      // K^ [K^ kb0 | K^ kb1]
  static constexpr uint32_t WN = 49152;      // -W | V^ | T diag(beta) (track X: -W only)
  static constexpr uint32_t VH = WN + kRecVH;
  static constexpr uint32_t TB = WN + kRecTB;
  static constexpr uint32_t GT = WN + kRecP; // two gate buffers of 512 B (chunk j in buffer j & 1)
  static constexpr uint32_t VN = GT + 1024;  // Vn^T diag(e^{gamma_C - gamma}) [d_v][t]
  static constexpr uint32_t BYTES = VN + 16384 + 1024;
};
static_assert(XferLay::VN % 1024 == 0 && XferLay::TB % 1024 == 0, "operand tiles need 1024-byte alignment");
static_assert(2 * (XferLay::BYTES + 1024) <= 228 * 1024, "two transfer CTAs per SM");
constexpr uint32_t TX_ST = 0, TX_V = 128, TX_COLS = 256;   // TMEM: the state, its Vn^T

__global__ void __launch_bounds__(kXferThreads, 2) xfer_kernel(const PrefillArgs p) {
  using L_ = XferLay;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t mb_k, mb_a, mb_g[2];   // copies landed
  __shared__ __align__(8) uint64_t mb_b1, mb_b2, mb_fin;  // products done (mb_fin: after a time-out)
  __shared__ __align__(8) uint64_t mb_vn, mb_s;           // worker warps done (8 arrivals)
  __shared__ uint32_t tmem_base_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool track_x = (blockIdx.x & 1) != 0;
  const int cu = blockIdx.x >> 1;
  const int u = cu / p.nh, h = p.h0 + cu % p.nh;
  if (u >= p.seg_list[0]) return;
  const Seg sg = load_seg(p.seg_list, u);
  if (sg.sigma == sg.nsig - 1) return;   // the last segment needs no transfer map
  const int G = p.h_v / p.h_k, kh = h / G;

  // ---- the decayed prefix of the segment ----
  // Chunk c's transition of the state, e^{gamma_C} prod_t (I - beta_t k^_t k^_t^T),
  // has 2-norm at most e^{gamma_C} (beta in (0, 1), |k^| <= 1).  So whatever the
  // state holds before chunk j reaches the segment's end shrunk by at least
  // e^{T_j}, T_j = the sum of gamma_C over chunks j .. end.  Where T_j <
  // kNegligibleLogDecay that is below 1e-69 of its size, far under the smallest
  // fp32 value: track S can start at the last such chunk from zero (the result
  // then differs from the full scan by rounding only), and track X, the whole
  // product, is zero.  Each chunk's e^{gamma_C} is its gate record's
  // last e^gamma (0 once it underflows, read as -inf).
  const int nch_all = (sg.len + C - 1) / C;
  const int j0 = decayed_prefix(p.rec_v + ((size_t)sg.c0 * p.h_v + h) * kRecV, (size_t)p.h_v * kRecV, nch_all);
  if (track_x) {   // the combine pass skips steps whose map is zero
    if (tid == 0) p.xzero[(size_t)(sg.k0 + sg.sigma) * p.h_v + h] = j0 >= 0 ? 1 : 0;
    if (j0 >= 0) {   // X = 0: the zero map as its bf16 hi / lo tiles
      uint4* xt = reinterpret_cast<uint4*>(xfer_ptr(p, sg.k0 + sg.sigma, h, 0));
      for (int i = tid; i < 65536 / 16; i += kXferThreads) xt[i] = make_uint4(0, 0, 0, 0);
      return;
    }
  }
  const int jb = j0 > 0 ? j0 : 0;   // track S's first chunk
  const int nch = nch_all - jb;
  const int c0 = sg.c0 + jb;

  const Smem sm = smem_aligned(smem_raw);
  if (tid == 0) {
    tc::mbar_init(&mb_k, 1);
    tc::mbar_init(&mb_a, 1);
    tc::mbar_init(&mb_g[0], 1);
    tc::mbar_init(&mb_g[1], 1);
    tc::mbar_init(&mb_b1, 1);
    tc::mbar_init(&mb_b2, 1);
    tc::mbar_init(&mb_fin, 1);
    tc::mbar_init(&mb_vn, kXferWorkers / 32);
    tc::mbar_init(&mb_s, kXferWorkers / 32);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base_s, TX_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_s;
  auto wt = [&](uint64_t* mb, uint32_t k) -> bool {   // the k-th completion of mb (parity k & 1)
    return tc::mbar_wait(mb, k & 1u, kWaitBudget);
  };
  auto rec_kq = [&](int j) { return p.rec_kq + ((size_t)(c0 + j) * p.h_k + kh) * kRecKQ; };
  auto rec_v = [&](int j) { return p.rec_v + ((size_t)(c0 + j) * p.h_v + h) * kRecV; };
  bool ok = true;

  if (warp == kXferWorkers / 32) {
    // ================= the MMA warp (one lane) =================
    if (lane == 0) {
      bool issued = false;
      auto issue_u = [&](int j) -> bool {   // track S: U = V^T (T diag beta)^T into TX_V
        if (!wt(&mb_a, j)) return false;
        tc::fence_after_sync();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_bf16(tmem + TX_V, tc::sdesc_at(D_MN_V, sm.addr + L_::VH + k * 2048),
                       tc::sdesc_at(D_K, sm.addr + L_::TB + k * 32), ID_MN_A, k > 0);
        issued = true;
        return true;
      };
      if (!track_x) ok = issue_u(0);
      for (int j = 0; j < nch && ok; ++j) {
        // the workers' state tile (track X: and this chunk's -W)
        if (!(wt(&mb_s, j) && (!track_x || wt(&mb_a, j)))) { ok = false; break; }
        tc::fence_after_sync();
        // [Vn^T = U + S (-W)^T]   (track X: X (-W)^T)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t kb = k >> 2, ks = (k & 3) * 32;
          tc::mma_bf16(tmem + TX_V, tc::sdesc_at(D_K, sm.addr + L_::ST + kb * 16384 + ks),
                       tc::sdesc_at(D_MN_W, sm.addr + L_::WN + k * 2048), ID_KMN, track_x ? (k > 0) : 1u);
        }
        issued = true;
        tc::mma_commit(&mb_b1);
        // the workers' Vn^T tile, and K^
        if (!(wt(&mb_vn, j) && wt(&mb_k, j))) { ok = false; break; }
        tc::fence_after_sync();
        // [state += Vn^T diag(e^{gamma_C - gamma}) K^]
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_bf16(tmem + TX_ST, tc::sdesc_at(D_K, sm.addr + L_::VN + k * 32),
                       tc::sdesc_at(D_MN_V, sm.addr + L_::KH + k * 2048), ID_MN_B, 1u);
        tc::mma_commit(&mb_b2);
        // the next chunk's U (TX_V was read for the Vn^T tile)
        if (!track_x && j + 1 < nch && !issue_u(j + 1)) { ok = false; break; }
      }
      if (!ok) {
        record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
        if (issued) {   // the products issued finish (bounded) before the tensor memory is freed
          tc::mma_commit(&mb_fin);
          wt(&mb_fin, 0);
        }
      }
    }
    __syncwarp();
  } else if (warp == kXferWorkers / 32 + 1) {
    // ================= the copy warp (one lane) =================
    // -W | V^ | T diag(beta) refills after [S (-W)^T] (b1), K^ after the state
    // update (b2), which also follows the Vn^T tile that last read the gates two
    // chunks back.
    if (lane == 0) {
      uint32_t i_k = 0, i_a = 0, i_g0 = 0, i_g1 = 0;   // copies issued
      auto load_k = [&](int j) {   // the K^ halves of the [K^ | Q^] record
        mbar_expect_tx(&mb_k, 16384);
        bulk_copy(sm.base + L_::KH, rec_kq(j), 8192, &mb_k);
        bulk_copy(sm.base + L_::KH + 8192, rec_kq(j) + 16384, 8192, &mb_k);
        ++i_k;
      };
      auto load_a = [&](int j) {   // track S: -W | V^ | T diag(beta); track X: -W
        bulk_load(sm.base + L_::WN, rec_v(j), track_x ? 16384u : kRecP, &mb_a);
        ++i_a;
      };
      auto load_g = [&](int j) {
        bulk_load(sm.base + L_::GT + (j & 1) * 512, rec_v(j) + kRecGate, kRecGateBytes, &mb_g[j & 1]);
        if (j & 1) ++i_g1; else ++i_g0;
      };
      load_g(0);
      if (nch > 1) load_g(1);
      load_k(0);
      load_a(0);
      for (int j = 0; j + 1 < nch; ++j) {
        if (!wt(&mb_b1, j)) { ok = false; break; }
        load_a(j + 1);
        if (!wt(&mb_b2, j)) { ok = false; break; }
        load_k(j + 1);
        if (j + 2 < nch) load_g(j + 2);
      }
      if (!ok) {
        record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
        // the copies this CTA started land (bounded) before its shared memory goes away
        auto drain = [&](uint64_t* mb, uint32_t n_issued) {
          if (n_issued > 0) wt(mb, n_issued - 1);
        };
        drain(&mb_k, i_k);
        drain(&mb_a, i_a);
        drain(&mb_g[0], i_g0);
        drain(&mb_g[1], i_g1);
      }
    }
    __syncwarp();
  } else {
    // ================= the worker warps =================
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const int row = 32 * (warp & 3) + lane;   // TMEM lane this thread reads
    const int hf = warp >> 2;                 // which half of the lane quarter's columns
    // the initial state -- S = 0 or X = I -- as the bf16 operand tile, and in TMEM
    // scaled by the first chunk's total decay
    ok = wt(&mb_g[0], 0);
    if (ok) {
      const float dC0 = sm.f32(L_::GT)[C - 1];
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int col0 = 64 * hf + 32 * c2;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = (track_x && col0 + i == row) ? 1.0f : 0.0f;
#pragma unroll
        for (int m = 0; m < 4; ++m) store_bf16x8(sm.base + L_::ST, tc::sw128_off(row, col0 + 8 * m, 16384), v + 8 * m);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= dC0;
        tc::tmem_st32(tmem + lane_base + TX_ST + col0, v);
      }
      warp_signal(&mb_s, lane);
    }
    for (int j = 0; j < nch && ok; ++j) {
      const float* egc = sm.f32(L_::GT + (j & 1) * 512) + 64;
      // ---- Vn^T diag(e^{gamma_C - gamma}) tile, row = d_v index ----
      if (!(wt(&mb_b1, j) && wt(&mb_g[j & 1], j >> 1))) { ok = false; break; }
      tc::fence_after_sync();
      {
        float v[32];
        tc::tmem_ld32(tmem + lane_base + TX_V + 32 * hf, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= egc[32 * hf + i];
#pragma unroll
        for (int m = 0; m < 4; ++m) store_bf16x8(sm.base + L_::VN, tc::sw128_off(row, 32 * hf + 8 * m, 0), v + 8 * m);
      }
      warp_signal(&mb_vn, lane);
      // ---- the new state -> bf16 operand tile, and in TMEM scaled by the next chunk's
      //      decay (after the last chunk the accumulator is read out below) ----
      if (!wt(&mb_b2, j)) { ok = false; break; }
      tc::fence_after_sync();
      if (j + 1 < nch) {
        if (!wt(&mb_g[(j + 1) & 1], (j + 1) >> 1)) { ok = false; break; }
        const float dC = sm.f32(L_::GT + ((j + 1) & 1) * 512)[C - 1];
#pragma unroll 1
        for (int c2 = 0; c2 < 2; ++c2) {
          const int col0 = 64 * hf + 32 * c2;
          float v[32];
          const uint32_t ta = tmem + lane_base + TX_ST + col0;
          tc::tmem_ld32(ta, v);
#pragma unroll
          for (int m = 0; m < 4; ++m) store_bf16x8(sm.base + L_::ST, tc::sw128_off(row, col0 + 8 * m, 16384), v + 8 * m);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= dC;
          tc::tmem_st32(ta, v);
        }
        warp_signal(&mb_s, lane);
      }
    }
    if (!ok) {
      if (lane == 0) record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
    } else if (!track_x) {
      // S_end(0), fp32 in tiled order
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int col0 = 64 * hf + 32 * c2;
        float v[32];
        tc::tmem_ld32(tmem + lane_base + TX_ST + col0, v);
        store_state_row(xfer_ptr(p, sg.k0 + sg.sigma, h, 1), true, row, col0, v);
      }
    } else {
      // X as bf16 hi / lo tiles for the combine pass's tensor-core products
      uint8_t* xt = reinterpret_cast<uint8_t*>(xfer_ptr(p, sg.k0 + sg.sigma, h, 0));
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int col0 = 64 * hf + 32 * c2;
        float v[32], lo[32];
        tc::tmem_ld32(tmem + lane_base + TX_ST + col0, v);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {   // X - bf16(X), exact in fp32
          float r0, r1;
          round_bf16x2(v[i], v[i + 1], r0, r1);
          lo[i] = v[i] - r0;
          lo[i + 1] = v[i + 1] - r1;
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint32_t off = tc::sw128_off(row, col0 + 8 * m, 16384);
          store_bf16x8(xt, off, v + 8 * m);
          store_bf16x8(xt + 32768, off, lo + 8 * m);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TX_COLS);
}

// ============================== combine pass ==============================

// Chains the transfer maps of a multi-segment sequence into every segment's
// true start state, one CTA per (sequence, value head):
//   S_{sigma+1} = S_sigma X_sigma + S_sigma^0,
// written over slot sigma's end state after saving the initial state (so the
// output pass never reads a state that the last segment's CTA is writing).
//
// The products run on the tensor core with fp32 accumulation.  S is split
// into three bf16 parts (s1 = bf16(S), s2 = bf16(S - s1), s3 = bf16(S - s1 -
// s2), which sum to S exactly) and X into two (X_hi, X_lo); TMEM starts at
// S^0 and accumulates s1 X_hi + s2 X_hi + s3 X_hi + s1 X_lo.  The terms left
// out are below 2^-16 of |S||X| per step.  A map that is exactly the identity
// (no writes, no decay) gives back S bit for bit.
//
// The accumulator is double-buffered in TMEM, so while the tensor core runs a
// step's products the threads load the next step's S^0 into the other buffer
// and store the previous step's result: per step the chain is only the
// products, the read-back and the split into the next operands.  The warp that
// issues the products does its share of that after its split instead, when the
// other warps' stores have drained (behind them it would hold up the step).
constexpr int kCombThreads = 512;
struct CombLay {
  static constexpr uint32_t XB = 0;               // two map buffers: [X_hi 32 KB | X_lo 32 KB]
  static constexpr uint32_t XB_BYTES = 65536;
  static constexpr uint32_t S1 = 2 * XB_BYTES;    // s1, s2, s3: bf16 [row][k], K blocks 16 KB apart
  static constexpr uint32_t S2 = S1 + 32768;
  static constexpr uint32_t S3 = S2 + 32768;
  static constexpr uint32_t BYTES = S3 + 32768 + 1024;
};
static_assert(CombLay::BYTES <= 227 * 1024, "shared memory");
constexpr uint32_t TC_COLS = 256;   // two accumulator buffers

__global__ void __launch_bounds__(kCombThreads, 1) combine_kernel(const PrefillArgs p) {
  using L_ = CombLay;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t mb_x[2];   // map buffers landed
  __shared__ __align__(8) uint64_t mb_mma;
  __shared__ uint32_t tmem_base_s;
  const int u = blockIdx.x / p.nh, h = p.h0 + blockIdx.x % p.nh;
  if (u >= p.multi_list[0]) return;
  const int* e = p.multi_list + 4 + 4 * u;
  const int n = e[0], k0 = e[1], nsig = e[2];
  const int steps = nsig - 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = 32 * (warp & 3) + lane, col0 = 32 * (warp >> 2);   // TMEM lane = state row, 32 columns
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  // Where every map of the sequence is exactly zero, each S_{sigma+1} is its
  // S_sigma^0, which slot sigma already holds: only the initial state is saved.
  int nonzero = 0;
  for (int sg = tid; sg < steps; sg += kCombThreads) nonzero |= p.xzero[(size_t)(k0 + sg) * p.h_v + h] == 0;
  if (!__syncthreads_or(nonzero)) {
    float v[32];
    load_state_row(p.ssm_state + ((size_t)n * p.h_v + h) * kD * kD, false, row, col0, v);
    store_state_row(xfer_ptr(p, k0, h, 2), true, row, col0, v);
    return;
  }
  const Smem sm = smem_aligned(smem_raw);
  if (tid == 0) {
    tc::mbar_init(&mb_x[0], 1);
    tc::mbar_init(&mb_x[1], 1);
    tc::mbar_init(&mb_mma, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base_s, TC_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_s;
  // copies issued / waited per buffer (the same on every thread: tid 32 issues
  // under conditions every thread evaluates alike)
  int issued[2] = {1, steps > 1 ? 1 : 0}, waited[2] = {0, 0};
  if (tid == 32) {
    bulk_load(sm.base + L_::XB, xfer_ptr(p, k0, h, 0), L_::XB_BYTES, &mb_x[0]);
    if (steps > 1) bulk_load(sm.base + L_::XB + L_::XB_BYTES, xfer_ptr(p, k0 + 1, h, 0), L_::XB_BYTES, &mb_x[1]);
  }
  // S0 = the initial state: saved, and split into the operand tiles
  auto split_store = [&](const float (&v)[32]) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      float a[8], b[8], c[8];
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        round_bf16x2(v[8 * m + i], v[8 * m + i + 1], a[i], a[i + 1]);
        const float r0 = v[8 * m + i] - a[i], r1 = v[8 * m + i + 1] - a[i + 1];
        round_bf16x2(r0, r1, b[i], b[i + 1]);
        c[i] = r0 - b[i];
        c[i + 1] = r1 - b[i + 1];
      }
      const uint32_t off = tc::sw128_off(row, col0 + 8 * m, 16384);
      store_bf16x8(sm.base + L_::S1, off, a);
      store_bf16x8(sm.base + L_::S2, off, b);
      store_bf16x8(sm.base + L_::S3, off, c);
    }
  };
  {
    float v[32];
    load_state_row(p.ssm_state + ((size_t)n * p.h_v + h) * kD * kD, false, row, col0, v);
    store_state_row(xfer_ptr(p, k0, h, 2), true, row, col0, v);
    split_store(v);
  }
  // buffer 0 starts at S^0 of the first segment; b then holds the next one's
  float b[32];
  load_state_row(xfer_ptr(p, k0, h, 1), true, row, col0, b);
  tc::tmem_st32(tmem + lane_base + col0, b);
  if (steps > 1) load_state_row(xfer_ptr(p, k0 + 1, h, 1), true, row, col0, b);
  float v[32];   // the last step's result, stored while the next step's products run
  uint32_t phase = 0;
  bool ok = true;
#pragma unroll 1
  for (int sg = 0; sg < steps; ++sg) {
    const uint32_t acc = tmem + (uint32_t)(sg & 1) * 128;
    ok = tc::mbar_wait(&mb_x[sg & 1], (uint32_t)((sg >> 1) & 1), kWaitBudget);
    if (!sync_for_mma_and(ok)) { ok = false; break; }   // also: the S parts and this accumulator are in place
    ++waited[sg & 1];
    if (tid == 0) {
      const uint32_t xb = sm.addr + L_::XB + (sg & 1) * L_::XB_BYTES;
      const uint32_t a_of[4] = {L_::S1, L_::S2, L_::S3, L_::S1};
      const uint32_t b_of[4] = {0u, 0u, 0u, 32768u};
#pragma unroll
      for (int pass = 0; pass < 4; ++pass)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t kb = k >> 2, ks = (k & 3) * 32;
          tc::mma_bf16(acc, tc::sdesc_at(D_K, sm.addr + a_of[pass] + kb * 16384 + ks),
                       tc::sdesc_at(D_MN_KQ, xb + b_of[pass] + k * 2048), ID_MN_B, 1u);
        }
      tc::mma_commit(&mb_mma);
    }
    // meanwhile: the last step's result out, the next step's S^0 into the other buffer
    // (whose previous products were read back last step)
    auto hand_off = [&](int done) {   // results of steps < done are out
      if (done > 0) store_state_row(xfer_ptr(p, k0 + done - 1, h, 1), true, row, col0, v);
      if (sg + 1 < steps) {
        tc::tmem_st32(tmem + (uint32_t)((sg + 1) & 1) * 128 + lane_base + col0, b);
        if (sg + 2 < steps) load_state_row(xfer_ptr(p, k0 + sg + 2, h, 1), true, row, col0, b);
      }
    };
    if (warp != 0) hand_off(sg);
    ok = tc::mbar_wait(&mb_mma, phase, kWaitBudget);
    phase ^= 1u;
    if (!__syncthreads_and(ok)) { ok = false; break; }
    tc::fence_after_sync();
    // the map buffer and the S parts are free again
    if (sg + 2 < steps) {
      if (tid == 32) bulk_load(sm.base + L_::XB + (sg & 1) * L_::XB_BYTES, xfer_ptr(p, k0 + sg + 2, h, 0),
                               L_::XB_BYTES, &mb_x[sg & 1]);
      ++issued[sg & 1];
    }
    tc::tmem_ld32(acc + lane_base + col0, v);
    split_store(v);   // the next step's operands
    if (warp == 0) hand_off(sg + 1);
  }
  if (ok && steps > 0 && warp != 0) store_state_row(xfer_ptr(p, k0 + steps - 1, h, 1), true, row, col0, v);
  if (!ok) {
    if (tid == 0) record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
    // the map copies this CTA started must land (bounded) before its smem goes away
    for (int q = 0; q < 2; ++q)
      for (; waited[q] < issued[q]; ++waited[q]) tc::mbar_wait(&mb_x[q], (uint32_t)(waited[q] & 1), kWaitBudget);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TC_COLS);
}

}  // namespace

cudaError_t launch_prefill_prep(const PrefillArgs& p, unsigned max_chunks, const CUtensorMap& tm_qkv,
                                cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)PrepLay::BYTES);
  if (e != cudaSuccess) return e;
  prep_kernel<<<max_chunks * (unsigned)p.nkh, kPrepThreads, PrepLay::BYTES, stream>>>(p, tm_qkv);
  return cudaGetLastError();
}

cudaError_t launch_prefill_combine(const PrefillArgs& p, unsigned max_multi, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)CombLay::BYTES);
  if (e != cudaSuccess) return e;
  combine_kernel<<<max_multi * (unsigned)p.nh, kCombThreads, CombLay::BYTES, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prefill_scan(const PrefillArgs& p, bool transfer, unsigned units, const CUtensorMap& tm_z,
                                cudaStream_t stream) {
  cudaError_t e;
  if (transfer) {   // two tracks per (segment, value head)
    if ((e = cudaFuncSetAttribute(xfer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)XferLay::BYTES)) != cudaSuccess)
      return e;
    xfer_kernel<<<2 * units * (unsigned)p.nh, kXferThreads, XferLay::BYTES, stream>>>(p);
  } else {
    if ((e = cudaFuncSetAttribute(output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)ScanLay::BYTES)) != cudaSuccess)
      return e;
    output_kernel<<<units * (unsigned)p.nh, kOutThreads, ScanLay::BYTES, stream>>>(p, tm_z);
  }
  return cudaGetLastError();
}

}  // namespace gdn
