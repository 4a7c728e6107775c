// gdn_gemm.cu -- the layer's input and output projections (sm_103a): one
// persistent tcgen05 GEMM, D = A B^T with bf16 operands and fp32 accumulation.
//
// The Gated DeltaNet layer sits between two dense projections in the hybrid
// models the pages run ("Serving large language models on our own stack",
// section "Qwen3.5-35B-A3B from a real GGUF"; llmxabe README, architecture
// paragraph: three Gated DeltaNet layers per gated-attention layer).  The
// input projection maps the hidden state x [T][hidden] to the layer's
// inputs q|k|v, z, a and b; the output projection maps the gated-norm output
// o [T][h_v d_v] back to [T][hidden].  Both are A [M][K] times B [N][K]^T
// (B in the nn.Linear layout, output features by input features), and the
// epilogue writes each run of output columns straight into its destination
// array -- for the input projection the layer's own qkv, z, a and b buffers,
// in the layouts gdn_prefill and gdn_decode_step read -- so nothing is copied
// or reshaped between the projection and the layer.
//
// Kernel shape: one CTA per SM walks 128 x 256 output tiles (row-major tile
// order: the CTAs of a wave share A's rows and read all of B, which stays in
// L2).  Six warps, meeting on mbarriers:
//   warp 0   one thread issues the 2-D TMA loads of A [128 x 64] and B
//            [256 x 64] K-blocks (128-byte swizzle) into a 4-stage ring;
//   warp 1   one thread issues tcgen05.mma (M 128, N 256, K 16) into a TMEM
//            accumulator and commits each stage back to the loader;
//   warps 2-5  read the finished accumulator (each its own TMEM lane
//            quarter), round to bf16 and store.
// The accumulator is double-buffered (2 x 256 of the 512 TMEM columns), so a
// tile's epilogue overlaps the next tile's products.  Rows past M and columns
// past N read as zeros (TMA fill) and are not stored; K past the array reads
// zeros too.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_launch.h"
#include "gdn_prefill.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int GBM = 128, GBN = 256, GBK = 64, GSTAGES = 4;
constexpr uint32_t GA_BYTES = GBM * GBK * 2;          // one A K-block (16 KB)
constexpr uint32_t GB_BYTES = GBN * GBK * 2;          // one B K-block (32 KB)
constexpr uint32_t GSTAGE_BYTES = GA_BYTES + GB_BYTES;
constexpr uint32_t GSMEM_BYTES = GSTAGES * GSTAGE_BYTES + 1024;   // + slack to align the base
constexpr int GTHREADS = 192;
constexpr uint32_t GTMEM_COLS = 2 * GBN;
constexpr uint32_t G_IDESC = tc::idesc_bf16(GBM, GBN, 0, 0);
constexpr uint64_t G_DESC = tc::sdesc_sw128(16, 1024);   // K-major, 8-row groups 1 KB apart
static_assert(GSMEM_BYTES <= 227 * 1024, "shared memory");
static_assert(GA_BYTES % 1024 == 0 && GSTAGE_BYTES % 1024 == 0, "swizzle atoms are 1024-byte aligned");

struct GemmParams {
  int M, N, K;
  int nseg;
  GemmOut seg[kGemmMaxSegs];
  int32_t* status;
};

__device__ __forceinline__ void mbar_arrive(uint64_t* mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(mbar)) : "memory");
}

// Eight consecutive output columns starting at col (a multiple of 8) of one
// row: into the destination run that holds them, as one 16-byte store.
__device__ __forceinline__ void store_group(const GemmParams& p, int row, int col, const float* v) {
  if (col >= p.N) return;
#pragma unroll
  for (int i = 0; i < kGemmMaxSegs; ++i) {
    if (i >= p.nseg) break;
    const GemmOut& s = p.seg[i];
    if (col >= s.col0 && col < s.col0 + s.ncols) {
      uint4 u;
      u.x = pack_bf16x2(v[0], v[1]);
      u.y = pack_bf16x2(v[2], v[3]);
      u.z = pack_bf16x2(v[4], v[5]);
      u.w = pack_bf16x2(v[6], v[7]);
      *reinterpret_cast<uint4*>(s.ptr + (size_t)row * (size_t)s.ld + (col - s.col0)) = u;
      return;
    }
  }
}

__global__ void __launch_bounds__(GTHREADS, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[GSTAGES];    // a stage's A and B landed
  __shared__ __align__(8) uint64_t empty[GSTAGES];   // a stage's products completed (slot free)
  __shared__ __align__(8) uint64_t tfull[2];         // an accumulator's tile is complete
  __shared__ __align__(8) uint64_t tempty[2];        // an accumulator has been read out
  __shared__ uint32_t tmem_base_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Smem sm = smem_aligned(smem_raw);
  if (threadIdx.x == 0) {
    for (int s = 0; s < GSTAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&tfull[a], 1);
      tc::mbar_init(&tempty[a], 4);   // one arrival per epilogue warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base_s, GTMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_s;

  const int n_nt = (p.N + GBN - 1) / GBN;
  const int tiles = ((p.M + GBM - 1) / GBM) * n_nt;
  const int kblocks = (p.K + GBK - 1) / GBK;

  if (warp == 0) {
    // ---- loader ----
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_a)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b)) : "memory");
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int m0 = (t / n_nt) * GBM, n0 = (t % n_nt) * GBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!tc::mbar_wait(&empty[s], ph ^ 1u, kWaitBudget)) {
            record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          uint8_t* dst = sm.base + s * GSTAGE_BYTES;
          mbar_expect_tx(&full[s], GSTAGE_BYTES);
          tma_load_2d(dst, &tm_a, kb * GBK, m0, &full[s]);
          tma_load_2d(dst + GA_BYTES, &tm_b, kb * GBK, n0, &full[s]);
          if (++s == GSTAGES) { s = 0; ph ^= 1u; }
        }
      }
      // take every slot once more: the products' releases have all landed
      // before the CTA can exit
      for (int i = 0; i < GSTAGES && ok; ++i) {
        if (!tc::mbar_wait(&empty[s], ph ^ 1u, kWaitBudget)) {
          record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
          break;
        }
        if (++s == GSTAGES) { s = 0; ph ^= 1u; }
      }
    }
  } else if (warp == 1) {
    // ---- tensor-core issue ----
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      int it = 0;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++it) {
        const int acc = it & 1;
        if (!tc::mbar_wait(&tempty[acc], ((uint32_t)(it >> 1) & 1u) ^ 1u, kWaitBudget)) {
          record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + (uint32_t)acc * GBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!tc::mbar_wait(&full[s], ph, kWaitBudget)) {
            record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a = sm.addr + s * GSTAGE_BYTES, b = a + GA_BYTES;
#pragma unroll
          for (int k = 0; k < GBK / 16; ++k)
            tc::mma_bf16(d, tc::sdesc_at(G_DESC, a + 32 * k), tc::sdesc_at(G_DESC, b + 32 * k), G_IDESC,
                         (kb | k) != 0);
          tc::mma_commit(&empty[s]);   // the slot frees once these products have read it
          if (++s == GSTAGES) { s = 0; ph ^= 1u; }
        }
        if (ok) tc::mma_commit(&tfull[acc]);
      }
    }
  } else {
    // ---- epilogue: TMEM -> bf16 -> global ----
    const int q = warp & 3;   // the TMEM lane quarter this warp may read
    int it = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
      const int acc = it & 1;
      if (!tc::mbar_wait(&tfull[acc], (uint32_t)(it >> 1) & 1u, kWaitBudget)) {
        record_status(p.status, GDN_ERR_DEVICE_TIMEOUT);
        break;
      }
      tc::fence_after_sync();
      const int m0 = (t / n_nt) * GBM, n0 = (t % n_nt) * GBN;
      const int row = m0 + 32 * q + lane;
      const uint32_t taddr = tmem + (uint32_t)acc * GBN + ((uint32_t)(32 * q) << 16);
#pragma unroll 1
      for (int c = 0; c < GBN; c += 32) {
        float v[32];
        tc::tmem_ld32(taddr + (uint32_t)c, v);
        if (row < p.M) {
#pragma unroll
          for (int g = 0; g < 4; ++g) store_group(p, row, n0 + c + 8 * g, v + 8 * g);
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, GTMEM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 gemm_map_encoder() {
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

// K-major bf16 operand [rows][K]: boxes of 64 K-elements (128 bytes, the
// swizzle span) by box_rows rows, 128-byte swizzle, zeros outside.
bool make_operand_map(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = gemm_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)GBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0 || g.nseg <= 0 || g.nseg > kGemmMaxSegs) return cudaErrorInvalidValue;
  CUtensorMap tm_a, tm_b;
  if (!make_operand_map(&tm_a, g.A, (uint64_t)g.K, (uint64_t)g.M, GBM) ||
      !make_operand_map(&tm_b, g.B, (uint64_t)g.K, (uint64_t)g.N, GBN))
    return cudaErrorInvalidValue;
  GemmParams p;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.nseg = g.nseg;
  for (int i = 0; i < kGemmMaxSegs; ++i) p.seg[i] = i < g.nseg ? g.seg[i] : GemmOut{nullptr, 0, 0, 0};
  p.status = g.status;
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)GSMEM_BYTES)) != cudaSuccess)
    return e;
  const long long tiles = (long long)((g.M + GBM - 1) / GBM) * ((g.N + GBN - 1) / GBN);
  const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
  gemm_bf16_kernel<<<grid, GTHREADS, GSMEM_BYTES, stream>>>(tm_a, tm_b, p);
  return cudaGetLastError();
}

}  // namespace gdn
