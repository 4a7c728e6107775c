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
constexpr int kSegTokens = 1024;   // segment length when long sequences are split
constexpr int LDA = 65, LDO = 128;   // fp32 row strides: A and T [64][LDA], O staging [64][LDO]

// ---- tcgen05 operand and instruction descriptors ----
constexpr uint64_t D_K = tc::sdesc_sw128(16, 1024);         // K-major tiles
constexpr uint64_t D_MN_KQ = tc::sdesc_sw128(16384, 1024);  // K^ of a [K^ | Q^] tile read MN-major
constexpr uint64_t D_MN_V = tc::sdesc_sw128(8192, 1024);    // a [64][128] tile (blocks 8 KB apart) read MN-major
constexpr uint32_t ID_KK = tc::idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_GRAM = tc::idesc_f16(128, 64, 0, 0);
constexpr uint32_t ID_MN_A = tc::idesc_bf16(128, 64, 1, 0);
constexpr uint32_t ID_MN_B = tc::idesc_bf16(128, 128, 0, 1);

constexpr long long kWaitBudget = 1LL << 31;  // clock cycles (~1 s) before a wait gives up

// ---- per-chunk records (prep pass -> scan passes), in the workspace ----
// Tiles are stored byte for byte in their shared-memory layout (128-byte
// swizzle, 1024-byte atoms), so a scan pass moves them with plain bulk copies.
// Per (chunk, key head):   bf16 [K^ | Q^] tile, 64-column blocks 16 KB apart.
constexpr uint32_t kRecKQ = 32768;
// Per (chunk, value head):
constexpr uint32_t kRecWN = 0;         // -W [t][d_k] bf16, blocks 8 KB apart
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

// Four SiLUs with one reciprocal: with d_i = 1 + e^{-x_i}, 1/d_1 =
// d_2 d_3 d_4 / (d_1 d_2 d_3 d_4), and so on.  Inputs are clamped at -20 so the
// product stays below 2^126 (|silu(x)| < 4.2e-8 for x < -20, which the clamp
// replaces by silu(-20)); this takes the special-function unit from two
// operations per SiLU to 1.25.
__device__ __forceinline__ void silu4(float (&x)[4]) {
  float d[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = 1.0f + __expf(-fmaxf(x[i], -20.0f));
  const float d01 = d[0] * d[1], d23 = d[2] * d[3];
  const float r = __fdividef(1.0f, d01 * d23);   // approximate reciprocal (product < 2^126)
  const float r01 = r * d23, r23 = r * d01;   // 1/(d0 d1), 1/(d2 d3)
  x[0] *= r01 * d[1];
  x[1] *= r01 * d[0];
  x[2] *= r23 * d[3];
  x[3] *= r23 * d[2];
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
  float x[kRows][4];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int tau = t0 + tq - (kConvW - 1) + r;   // position in the sequence
    if (tau >= 0) {
      const uint2 v2 = *reinterpret_cast<const uint2*>(raw_blk + (tq + r) * 256 + lane * 8);
      x[r][0] = bf16_to_f32(v2.x & 0xffffu); x[r][1] = bf16_to_f32(v2.x >> 16);
      x[r][2] = bf16_to_f32(v2.y & 0xffffu); x[r][3] = bf16_to_f32(v2.y >> 16);
    } else {
      const float4 v4 = *reinterpret_cast<const float4*>(cs + (size_t)(kConvW - 1 + tau) * cs_stride);
      x[r][0] = v4.x; x[r][1] = v4.y; x[r][2] = v4.z; x[r][3] = v4.w;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float acc = w[0][e] * x[i][e];
#pragma unroll
      for (int j = 1; j < kConvW; ++j) acc = fmaf(w[j][e], x[i + j][e], acc);
      y[i][e] = tq + i < L ? acc : 0.0f;   // padding tokens of a partial chunk are zero
    }
    silu4(y[i]);
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
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

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

// One block diagonal d = i - j of T (blocks (j + d, j), j = 0 .. 3 - d), over
// NT threads, each with up to ceil(256 (4 - d) / NT) outputs in flight:
//   M_ij = sum_{k=j}^{i-1} A_ik T_kj   (into the scratch Mf),
//   T_ij = -T_ii M_ij.
template <int NT, int D>
__device__ __forceinline__ void solve_block_diagonal(const float* Af, float* Tf, float* Mf, int tid, int bar_id) {
  constexpr int kOuts = 256 * (4 - D), kPer = (kOuts + NT - 1) / NT;
  float m[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int o = tid + u * NT;
    m[u] = 0.0f;
    if (kPer * NT == kOuts || o < kOuts) {
      const int j = o >> 8, i = j + D, r = (o >> 4) & 15, c = o & 15;
#pragma unroll
      for (int k2 = 0; k2 < D; ++k2) {
        const int kb = j + k2;
#pragma unroll
        for (int s = 0; s < 16; ++s)
          m[u] = fmaf(Af[(16 * i + r) * LDA + 16 * kb + s], Tf[(16 * kb + s) * LDA + 16 * j + c], m[u]);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u)
    if (kPer * NT == kOuts || tid + u * NT < kOuts) Mf[tid + u * NT] = m[u];
  group_sync<NT>(bar_id);
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int o = tid + u * NT;
    if (kPer * NT == kOuts || o < kOuts) {
      const int j = o >> 8, i = j + D, r = (o >> 4) & 15, c = o & 15;
      float acc = 0.0f;
#pragma unroll
      for (int q = 0; q < 16; ++q) acc = fmaf(Tf[(16 * i + r) * LDA + 16 * i + q], Mf[(j << 8) + (q << 4) + c], acc);
      m[u] = -acc;
    }
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int o = tid + u * NT;
    if (kPer * NT == kOuts || o < kOuts) {
      const int j = o >> 8, i = j + D, r = (o >> 4) & 15, c = o & 15;
      Tf[(16 * i + r) * LDA + 16 * j + c] = m[u];
    }
  }
  group_sync<NT>(bar_id);
}

// T = (I + A)^{-1} for a strictly lower 64 x 64 matrix A (fp32, row stride
// LDA): the 16 x 16 diagonal blocks by forward substitution, a column per
// thread, then the blocks below them one block diagonal at a time, each
// product spread over the NT threads of a group (Mf: 3 x 16 x 16 fp32
// scratch; tid: the thread's index in the group; bar_id: the group's barrier,
// 0 for the whole CTA).  Every thread of the group calls it; it ends with a
// group barrier.
template <int NT>
__device__ __forceinline__ void solve_unit_lower(const float* Af, float* Tf, float* Mf, int tid, int bar_id) {
  static_assert(NT >= 64 && NT % 32 == 0, "the diagonal blocks use 64 threads");
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
    for (int e = tid - 64; e < 6 * 256; e += NT - 64) {
      const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
      const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
      const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
      Tf[(16 * bi + r) * LDA + 16 * bj + c] = 0.0f;
    }
  }
  group_sync<NT>(bar_id);
  solve_block_diagonal<NT, 1>(Af, Tf, Mf, tid, bar_id);
  solve_block_diagonal<NT, 2>(Af, Tf, Mf, tid, bar_id);
  solve_block_diagonal<NT, 3>(Af, Tf, Mf, tid, bar_id);
}

// Launchers of the split prefill (prep pass, then the scan passes).
cudaError_t launch_prefill_prep(const PrefillArgs& p, unsigned max_chunks, const CUtensorMap& tm_qkv,
                                cudaStream_t stream);
cudaError_t launch_prefill_combine(const PrefillArgs& p, unsigned max_multi, cudaStream_t stream);
cudaError_t launch_prefill_scan(const PrefillArgs& p, bool transfer, unsigned units, const CUtensorMap& tm_z,
                                cudaStream_t stream);

}  // namespace gdn
