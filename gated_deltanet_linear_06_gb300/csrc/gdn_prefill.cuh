// gdn_prefill.cuh -- pieces shared by the prefill kernels: operand
// descriptors, tile stores, bulk copies, the work list, the per-chunk records
// and the unit-lower-triangular solve of the chunked WY/UT form.
#pragma once
#include <cuda.h>

#include "gdn_common.cuh"
#include "gdn_launch.h"
#include "gdn_tc.cuh"

namespace gdn {

constexpr int C = kChunk;
constexpr int kSegTokens = 1024;   // shortest segment a long sequence is split into (sizes the workspace)
constexpr int LDO = 128;   // fp32 row stride of the O staging [64][LDO]

// ---- tcgen05 operand and instruction descriptors ----
constexpr uint64_t D_K = tc::sdesc_sw128(16, 1024);         // K-major tiles
constexpr uint64_t D_MN_KQ = tc::sdesc_sw128(16384, 1024);  // K^ of a [K^ | Q^] tile read MN-major
constexpr uint64_t D_MN_V = tc::sdesc_sw128(8192, 1024);    // a [64][128] tile (blocks 8 KB apart) read MN-major
// -W stored [d_k][t]: 128 rows of one 64-column atom, read MN-major as the B
// operand (N = t); a K = 16 step advances 16 rows (2 KB)
constexpr uint64_t D_MN_W = tc::sdesc_sw128(8192, 1024);
constexpr uint32_t ID_KK = tc::idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_GRAM = tc::idesc_f16(128, 64, 0, 0);
constexpr uint32_t ID_MN_A = tc::idesc_bf16(128, 64, 1, 0);
constexpr uint32_t ID_MN_B = tc::idesc_bf16(128, 128, 0, 1);
constexpr uint32_t ID_KMN = tc::idesc_bf16(128, 64, 0, 1);   // A K-major, B MN-major, N = 64

constexpr long long kWaitBudget = 1LL << 31;  // clock cycles (~1 s) before a wait gives up

// ---- per-chunk records (prep pass -> scan passes), in the workspace ----
// Tiles are stored byte for byte in their shared-memory layout (128-byte
// swizzle, 1024-byte atoms), so a scan pass moves them with plain bulk copies.
// Per (chunk, key head):   bf16 [K^ | Q^] tile, 64-column blocks 16 KB apart.
constexpr uint32_t kRecKQ = 32768;
// Per (chunk, value head):
constexpr uint32_t kRecWN = 0;         // -W [d_k][t] bf16 (one 64-column atom)
constexpr uint32_t kRecVH = 16384;     // V^ [t][d_v] bf16 (conv + SiLU), blocks 8 KB apart
constexpr uint32_t kRecTB = 32768;     // T diag(beta) [t][s] bf16
constexpr uint32_t kRecP = 40960;      // P [t][s] bf16
constexpr uint32_t kRecGate = 49152;   // fp32 e^gamma [64], e^{gamma_C - gamma} [64]
constexpr uint32_t kRecGateBytes = 512;
constexpr uint32_t kRecV = 50176;      // record size (multiple of 1024)
static_assert(kRecGate + kRecGateBytes <= kRecV && kRecV % 1024 == 0, "value record layout");

// Raw inputs of a chunk staged in shared memory by a 2-D TMA load: the q, k or
// v rows of tokens t0-3 .. t0+63 (a chunk and its conv halo), one
// [67 rows][128 bf16] box per 128-channel block.
constexpr uint32_t RAW_BOX_ROWS = C + kConvW - 1;
constexpr uint32_t RAW_BLK = RAW_BOX_ROWS * 256;

struct Smem {
  uint8_t* base;
  uint32_t addr;  // shared-window address of base
  __device__ float* f32(uint32_t off) const { return reinterpret_cast<float*>(base + off); }
};

// The dynamic shared memory rounded up to a 1024-byte boundary (swizzle atoms).
__device__ __forceinline__ Smem smem_aligned(uint8_t* raw_base) {
  const uint32_t raw = tc::smem_u32(raw_base);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  return Smem{raw_base + pad, raw + pad};
}

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

// The prefill's gates with the fast exp, log and divide.  softplus(x) =
// max(x, 0) + log(1 + e^{-|x|}): __logf of 1 + e^{-|x|} is off by well under
// 1e-6 absolute, where g = -e^{A_log} softplus(.) needs about 1e-3 relative.
// sigmoid clamps the exponent at 80 so that the denominator stays below 2^126,
// where the fast divide is exact to a few ulp (sigma(-80) < 2e-35 either way).
__device__ __forceinline__ float softplus_gate(float x) {
  return fmaxf(x, 0.0f) + __logf(1.0f + __expf(-fabsf(x)));
}
__device__ __forceinline__ float sigmoid_gate(float x) {
  return __fdividef(1.0f, 1.0f + __expf(fminf(-x, 80.0f)));
}

// x where s <= t, else +0, by masking the bits: no compare-and-select, which
// next to the exp of the decay factor measured about three times slower.
__device__ __forceinline__ float keep_if_le(float x, int s, int t) {
  return __uint_as_float(__float_as_uint(x) & (uint32_t)((s - t - 1) >> 31));
}

// SiLU of four values through the hyperbolic tangent: with h = x / 2,
// sigma(x) = (1 + tanh h) / 2, so x sigma(x) = h + h tanh(h) -- one
// special-function operation (tanh.approx, relative error about 2^-11) and two
// more per value.  The error it adds, at most |h| 2^-11, stays below the bf16
// rounding of the result wherever the result is not much smaller than x.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// SiLU(x) = h + h tanh(h) with h = x / 2, two elements per packed fp32x2 op
// (each element rounds as the scalar fmul and fma would).
__device__ __forceinline__ void silu4(float (&x)[4]) {
#pragma unroll
  for (int pp = 0; pp < 2; ++pp) {
    const float2 h = __fmul2_rn(make_float2(x[2 * pp], x[2 * pp + 1]), make_float2(0.5f, 0.5f));
    const float2 r = __ffma2_rn(h, make_float2(tanh_approx(h.x), tanh_approx(h.y)), h);
    x[2 * pp] = r.x;
    x[2 * pp + 1] = r.y;
  }
}

// Conv + SiLU of the 4 tokens tq .. tq+3 of a chunk starting at position t0
// of its sequence, over this lane's 4 channels, from a staged raw block (row r
// = position t0 - 3 + r).  Positions before the sequence read the carried conv
// state instead (cs: its 3 fp32 rows at this lane's channels, row stride
// cs_stride floats); padding tokens (tq + i >= L) come out zero.  w[j][e] is
// tap j of channel e (tap 3 multiplies the current token).
__device__ __forceinline__ void conv_quad_staged(const uint8_t* raw_blk, const float* cs, size_t cs_stride, int t0,
                                                 int L, int tq, int lane, const float (&w)[kConvW][4],
                                                 float (&y)[4][4]) {
  constexpr int kRows = 4 + kConvW - 1;
  float2 x[kRows][2];   // channel pairs (0, 1) and (2, 3)
  auto staged_row = [&](int r) {
    const uint2 v2 = *reinterpret_cast<const uint2*>(raw_blk + (tq + r) * 256 + lane * 8);
    x[r][0] = make_float2(bf16_to_f32(v2.x & 0xffffu), bf16_to_f32(v2.x >> 16));
    x[r][1] = make_float2(bf16_to_f32(v2.y & 0xffffu), bf16_to_f32(v2.y >> 16));
  };
  // rows kConvW - 1 .. kRows - 1 hold the chunk's tokens tq .. tq + 3, which lie
  // in the sequence; only the halo rows before them can lie before it
#pragma unroll
  for (int r = kConvW - 1; r < kRows; ++r) staged_row(r);
#pragma unroll
  for (int r = 0; r < kConvW - 1; ++r) {
    const int tau = t0 + tq - (kConvW - 1) + r;   // position in the sequence
    if (tau >= 0) {
      staged_row(r);
    } else {
      const float4 v4 = *reinterpret_cast<const float4*>(cs + (size_t)(kConvW - 1 + tau) * cs_stride);
      x[r][0] = make_float2(v4.x, v4.y);
      x[r][1] = make_float2(v4.z, v4.w);
    }
  }
  // taps in order, two channels per packed fp32x2 multiply-add (each channel
  // rounds as the scalar chain w0 x0, fma(w1, x1, .), ... would)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
      float2 acc = __fmul2_rn(make_float2(w[0][2 * pp], w[0][2 * pp + 1]), x[i][pp]);
#pragma unroll
      for (int j = 1; j < kConvW; ++j)
        acc = __ffma2_rn(make_float2(w[j][2 * pp], w[j][2 * pp + 1]), x[i + j][pp], acc);
      y[i][2 * pp] = acc.x;
      y[i][2 * pp + 1] = acc.y;
    }
    silu4(y[i]);
  }
  // padding tokens of a partial chunk are zero (as SiLU of a zero conv would
  // leave them); the same on the whole warp, taken in a sequence's last chunk only
  if (tq + 4 > L) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (tq + i >= L) y[i][0] = y[i][1] = y[i][2] = y[i][3] = 0.0f;
  }
}

// Sums over the warp of four per-token partial sums (one per lane and token):
// the first two butterfly steps hand half of the sums to the partner lane, so
// a lane ends with the full sum of token 2 (lane bit 4) + (lane bit 3), added
// in the same tree as warp_sum.  token_lane(i) is a lane holding token i's sum.
__device__ __forceinline__ float warp_sum4(const float (&s)[4], int lane) {
  const bool hi16 = (lane & 16) != 0, hi8 = (lane & 8) != 0;
  float k0 = hi16 ? s[2] : s[0], k1 = hi16 ? s[3] : s[1];
  const float s0 = hi16 ? s[0] : s[2], s1 = hi16 ? s[1] : s[3];
  k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
  k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
  float tot = hi8 ? k1 : k0;
  tot += __shfl_xor_sync(0xffffffffu, hi8 ? k0 : k1, 8);
  tot += __shfl_xor_sync(0xffffffffu, tot, 4);
  tot += __shfl_xor_sync(0xffffffffu, tot, 2);
  tot += __shfl_xor_sync(0xffffffffu, tot, 1);
  return tot;
}
__device__ __forceinline__ int token_lane(int i) { return ((i >> 1) << 4) | ((i & 1) << 3); }

// Sums of squares of four tokens' 128 channels (each lane holding 4 channels
// of each token) -> 1/sqrt(sum + eps) * scale for token i, on every lane.
__device__ __forceinline__ void l2_rnorm4(const float (&y)[4][4], float eps, float scale, int lane,
                                          float (&rn)[4]) {
  float ss[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ss[i] = y[i][0] * y[i][0];
#pragma unroll
    for (int e = 1; e < 4; ++e) ss[i] = fmaf(y[i][e], y[i][e], ss[i]);
  }
  const float r = rsqrtf(warp_sum4(ss, lane) + eps) * scale;
#pragma unroll
  for (int i = 0; i < 4; ++i) rn[i] = __shfl_sync(0xffffffffu, r, token_lane(i));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(mbar)), "r"(bytes)
               : "memory");
}

// One 2-D TMA tile load: the box at column x, row y of the tensor map lands at
// smem_dst and reports its bytes to mbar.  Rows outside the tensor read as zero.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* tm, int x, int y, uint64_t* mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(tc::smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(tc::smem_u32(mbar))
      : "memory");
}

// Bulk copy global -> shared that reports its bytes to mbar (the caller posts
// the expected byte count); both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_copy(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          tc::smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(tc::smem_u32(mbar))
      : "memory");
}

// One bulk copy with its own expected-byte count.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* mbar) {
  mbar_expect_tx(mbar, bytes);
  bulk_copy(smem_dst, gmem_src, bytes, mbar);
}

// Bulk copy shared -> global in the issuing thread's current bulk group.
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(tc::smem_u32(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The issuing thread's bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... and have completed.

// Block-wide sync that also orders tensor-memory traffic and makes generic
// smem writes visible to the tensor core (and to bulk copies).
__device__ __forceinline__ void sync_for_mma() {
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

// One segment of the work list (built on the device from cu_seqlens).
struct Seg {
  int n, begin, len, sigma, nsig, k0, c0;   // sequence, token range within it, segment index/count,
                                            // the sequence's first boundary slot, the segment's
                                            // first chunk record
};

__device__ __forceinline__ Seg load_seg(const int* list, int u) {
  const int* e = list + 4 + 8 * u;
  return Seg{e[0], e[1], e[2], e[3], e[4], e[5], e[6]};
}

// Transfer matrices of boundary slot k, value head h, 64 KB each: the map X
// (as two bf16 tiles, X_hi = bf16(X) and X_lo = bf16(X - X_hi), rows = first
// index, 64-column blocks 16 KB apart), S (fp32 end state from zero,
// overwritten by the combine pass with the true start state of the next
// segment), and the sequence's initial state (fp32, first slot only); the
// fp32 states in tiled order (tiled_off).
__device__ __forceinline__ float* xfer_ptr(const PrefillArgs& p, int k, int h, int part) {
  return p.xfer + (((size_t)k * p.h_v + h) * 3 + part) * (size_t)(kD * kD);
}

// fp32 128 x 128 states kept in the workspace (the transfer pass's end
// states, the combine pass's start states, a saved initial state) are stored
// in TMEM-native order: the 4-column group q of row r at float offset
// (q * 128 + r) * 4, so a warp holding 32 consecutive rows (one TMEM lane
// each) moves 512 contiguous bytes per 16-byte access.  The caller's
// ssm_state is row-major.
__device__ __forceinline__ size_t tiled_off(int r, int q) { return ((size_t)q * kD + r) * 4; }

// This thread's row r, columns col0 .. col0+31 of a state, tiled or row-major.
__device__ __forceinline__ void load_state_row(const float* base, bool tiled, int r, int col0, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 x = *reinterpret_cast<const float4*>(
        base + (tiled ? tiled_off(r, (col0 >> 2) + q) : (size_t)r * kD + col0 + 4 * q));
    v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
  }
}
__device__ __forceinline__ void store_state_row(float* base, bool tiled, int r, int col0, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    *reinterpret_cast<float4*>(base + (tiled ? tiled_off(r, (col0 >> 2) + q) : (size_t)r * kD + col0 + 4 * q)) =
        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// Barrier over the NT threads of a group: bar_id 0 is the whole CTA
// (__syncthreads), others a named barrier that exactly those threads use.
// (Ids 1 and 2 are the only named barriers used, as immediates.)
template <int NT>
__device__ __forceinline__ void group_sync(int bar_id) {
  if (bar_id == 0)
    __syncthreads();
  else if (bar_id == 1)
    asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
  else
    asm volatile("bar.sync 2, %0;" ::"n"(NT) : "memory");
}

// The same, returning whether every thread of the group passed ok.
template <int NT>
__device__ __forceinline__ bool group_sync_and(int bar_id, bool ok) {
  if (bar_id == 0) return __syncthreads_and(ok);
  uint32_t r;
  if (bar_id == 1)
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"((uint32_t)ok), "n"(NT)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 2, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"((uint32_t)ok), "n"(NT)
        : "memory");
  return r != 0;
}

// ---- the UT solve's fp32 64 x 64 matrices (A, T) ----
// Row-major with rows UT_LD = 68 floats apart: a warp reading or writing one
// 16-byte column group of 8 consecutive rows, or 8 column groups of one row,
// touches 32 distinct banks, and every element's offset is its row's base plus
// a constant (no per-access index arithmetic).
constexpr int UT_LD = 68;
constexpr uint32_t UT_BYTES = 64 * UT_LD * 4;
__device__ __forceinline__ int ut_idx(int t, int s) { return t * UT_LD + s; }
// columns s4 .. s4+3 of row t (s4 a multiple of 4)
__device__ __forceinline__ float4 ut_ld4(const float* M, int t, int s4) {
  return *reinterpret_cast<const float4*>(M + ut_idx(t, s4));
}
__device__ __forceinline__ void ut_st4(float* M, int t, int s4, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(M + ut_idx(t, s4)) = make_float4(a, b, c, d);
}

// acc[r][e] += sum_{k < nk} X[xr[r]][xc + k] Y[yr + k][yc + e] for two rows
// (R = 2) or one, the sum in increasing k; nk a multiple of 8, xc and yc
// multiples of 4.  Column pairs run as packed fp32x2 multiply-adds, each
// element rounding as fmaf would; Y's rows are taken 8 at a time.
template <int R>
__device__ __forceinline__ void ut_rowquad(const float* X, const int (&xr)[R], int xc, const float* Y, int yr,
                                           int yc, int nk, float (&acc)[R][4]) {
  float2 a2[R][2];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    a2[r][0] = make_float2(acc[r][0], acc[r][1]);
    a2[r][1] = make_float2(acc[r][2], acc[r][3]);
  }
  const float* Xb[R];
#pragma unroll
  for (int r = 0; r < R; ++r) Xb[r] = X + ut_idx(xr[r], xc);
  const float* Yb = Y + ut_idx(yr, yc);
#pragma unroll 1
  for (int k8 = 0; k8 < nk; k8 += 8, Yb += 8 * UT_LD) {
    float xk[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float4 x0 = *reinterpret_cast<const float4*>(Xb[r] + k8);
      const float4 x1 = *reinterpret_cast<const float4*>(Xb[r] + k8 + 4);
      xk[r][0] = x0.x; xk[r][1] = x0.y; xk[r][2] = x0.z; xk[r][3] = x0.w;
      xk[r][4] = x1.x; xk[r][5] = x1.y; xk[r][6] = x1.z; xk[r][7] = x1.w;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 y4 = *reinterpret_cast<const float4*>(Yb + j * UT_LD);
      const float2 ylo = make_float2(y4.x, y4.y), yhi = make_float2(y4.z, y4.w);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float2 x2 = make_float2(xk[r][j], xk[r][j]);
        a2[r][0] = __ffma2_rn(x2, ylo, a2[r][0]);
        a2[r][1] = __ffma2_rn(x2, yhi, a2[r][1]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    acc[r][0] = a2[r][0].x; acc[r][1] = a2[r][0].y;
    acc[r][2] = a2[r][1].x; acc[r][3] = a2[r][1].y;
  }
}

// T = (I + A)^{-1} for a strictly lower 64 x 64 matrix A, in place: M holds A
// (read only below its diagonal) on entry and T on return, both in the layout
// above.  With L = I + A partitioned into blocks, [L11 0; L21 L22]^{-1} =
// [T11 0; -T22 L21 T11, T22], applied twice:
//   1. the four 16 x 16 diagonal blocks by forward substitution (a column per
//      thread, 64 threads), written over A's diagonal blocks once every
//      thread has read them;
//   2. 16 -> 32: T10 = -T11 (A10 T00), T32 = -T33 (A32 T22);
//   3. 32 -> 64: T[32:64][0:32] = -T[32:64][32:64] (A[32:64][0:32] T[0:32][0:32]).
// Each product's left factor is staged in a block above the diagonal, where A
// holds nothing and the inverse is zero, and each product's result goes over
// the block of A that the previous step consumed.  On return M holds the
// inverse on and below its diagonal; above it, the 16 x 16 diagonal blocks are
// exactly +0 (forward substitution) and the other blocks hold staging data, so
// whoever reads T takes T[t][s] = 0 for s > t.  The products run as 128 units
// of one or two rows x 4 columns, so every output's sum has the same order
// whatever the thread count NT (>= 128); the unit -> thread maps keep each
// warp's loop bounds uniform.  tid: the thread's index in its group of NT;
// bar_id: the group's named barrier (0 for the whole CTA).  Every thread of the
// group calls it; it ends with a group barrier.
template <int NT>
__device__ __forceinline__ void solve_unit_lower(float* M, int tid, int bar_id) {
  static_assert(NT >= 128 && NT % 32 == 0, "the products use 128 threads");
  const float* Af = M;
  float* Tf = M;
  const int b = tid >> 4, c = tid & 15;
  float x[16];
  if (tid < 64) {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float a[16];
#pragma unroll
      for (int q = 0; 4 * q < r; ++q) {
        const float4 a4 = ut_ld4(Af, 16 * b + r, 16 * b + 4 * q);
        a[4 * q] = a4.x; a[4 * q + 1] = a4.y; a[4 * q + 2] = a4.z; a[4 * q + 3] = a4.w;
      }
      float acc = (r == c) ? 1.0f : 0.0f;
#pragma unroll
      for (int s = 0; s < r; ++s) acc = fmaf(-a[s], x[s], acc);
      x[r] = acc;
    }
  }
  group_sync<NT>(bar_id);   // every thread has read the diagonal blocks of A
  if (tid < 64) {
#pragma unroll
    for (int r = 0; r < 16; ++r) Tf[ut_idx(16 * b + r, 16 * b + c)] = x[r];
  }
  group_sync<NT>(bar_id);
  // 16 -> 32; unit u: column group u & 3, row (u >> 2) & 15, pair u >> 6
  const int u = tid;
  const int s_cq = u & 3, s_r = (u >> 2) & 15, s_i = 2 * (u >> 6) + 1, s_j = s_i - 1;
  if (u < 128) {   // A_ij T_jj -> the zero block (j, i)
    float acc[1][4] = {{0.0f, 0.0f, 0.0f, 0.0f}};
    const int xr[1] = {16 * s_i + s_r};
    ut_rowquad<1>(Af, xr, 16 * s_j, Tf, 16 * s_j, 16 * s_j + 4 * s_cq, 16, acc);
    ut_st4(Tf, 16 * s_j + s_r, 16 * s_i + 4 * s_cq, acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
  }
  group_sync<NT>(bar_id);
  if (u < 128) {   // T_ij = -T_ii (A_ij T_jj)
    float acc[1][4] = {{0.0f, 0.0f, 0.0f, 0.0f}};
    const int xr[1] = {16 * s_i + s_r};
    ut_rowquad<1>(Tf, xr, 16 * s_i, Tf, 16 * s_j, 16 * s_i + 4 * s_cq, 16, acc);
    ut_st4(Tf, 16 * s_i + s_r, 16 * s_j + 4 * s_cq, -acc[0][0], -acc[0][1], -acc[0][2], -acc[0][3]);
  }
  group_sync<NT>(bar_id);
  // 32 -> 64; unit u: rows r0 = 16 rh + (u >> 2) & 7 and r0 + 8, column group
  // 4 ch + (u & 3), with ch = (u >> 5) & 1 and rh = u >> 6
  const int rh = (u >> 6) & 1, ch = (u >> 5) & 1;
  const int r0 = 16 * rh + ((u >> 2) & 7), cq = 4 * ch + (u & 3);
  if (u < 128) {   // A[32:64][0:32] T[0:32][0:32] -> T[0:32][32:64]; T[0:16][16:32] is staging, skipped
    float acc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
    const int xr[2] = {32 + r0, 40 + r0};
    const int k0 = 16 * ch;
    ut_rowquad<2>(Af, xr, k0, Tf, k0, 4 * cq, 32 - k0, acc);
#pragma unroll
    for (int r = 0; r < 2; ++r) ut_st4(Tf, r0 + 8 * r, 32 + 4 * cq, acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  }
  group_sync<NT>(bar_id);
  if (u < 128) {   // -T[32:64][32:64] (...) -> T[32:64][0:32]; T[32:48][48:64] is staging, skipped
    float acc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
    const int xr[2] = {32 + r0, 40 + r0};
    ut_rowquad<2>(Tf, xr, 32, Tf, 0, 32 + 4 * cq, rh ? 32 : 16, acc);
#pragma unroll
    for (int r = 0; r < 2; ++r)
      ut_st4(Tf, 32 + r0 + 8 * r, 4 * cq, -acc[r][0], -acc[r][1], -acc[r][2], -acc[r][3]);
  }
  group_sync<NT>(bar_id);
}

// Launchers of the split prefill (prep pass, then the scan passes).
cudaError_t launch_prefill_prep(const PrefillArgs& p, unsigned max_chunks, const CUtensorMap& tm_qkv,
                                cudaStream_t stream);
cudaError_t launch_prefill_combine(const PrefillArgs& p, unsigned max_multi, cudaStream_t stream);
cudaError_t launch_prefill_scan(const PrefillArgs& p, bool transfer, unsigned units, const CUtensorMap& tm_z,
                                cudaStream_t stream);

}  // namespace gdn
