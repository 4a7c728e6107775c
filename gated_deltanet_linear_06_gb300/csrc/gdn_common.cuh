// gdn_common.cuh -- small device helpers shared by the libgdn kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kD = 128;       // d_k = d_v of the compiled fast path
constexpr int kConvW = 4;     // conv width
constexpr int kChunk = 64;    // prefill chunk

__device__ __forceinline__ float bf16_to_f32(uint16_t v) {
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

// Round-to-nearest-even fp32 -> bf16 bit pattern.
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Two fp32 values -> bf16x2 (lo in bits 0-15), round to nearest even, in one
// packed conversion: the same bits as converting each value alone, at several
// times the throughput of two single conversions.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The same for fp16x2.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// a and b rounded to bf16 (returned as fp32), with one packed conversion.
__device__ __forceinline__ void round_bf16x2(float a, float b, float& ra, float& rb) {
  const uint32_t r = pack_bf16x2(a, b);
  ra = __uint_as_float(r << 16);
  rb = __uint_as_float(r & 0xffff0000u);
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + __expf(-x)); }

__device__ __forceinline__ float sigmoid(float x) { return 1.0f / (1.0f + __expf(-x)); }

// log(1 + e^x) without overflow: max(x, 0) + log1p(e^{-|x|}).
__device__ __forceinline__ float softplus(float x) {
  return fmaxf(x, 0.0f) + log1pf(__expf(-fabsf(x)));
}

// Sum over the 32 lanes in a fixed butterfly order: every lane ends with the
// same value, and the order depends on nothing but the lane layout.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// Device status word: keep the first error recorded.
__device__ __forceinline__ void record_status(int32_t* word, int32_t code) {
  if (word) atomicCAS(reinterpret_cast<int*>(word), 0, code);
}

}  // namespace gdn
