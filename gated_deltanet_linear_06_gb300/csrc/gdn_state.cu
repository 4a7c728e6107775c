// gdn_state.cu -- copies of whole per-sequence states between caller-owned state
// pools, and resets of pool slots.
//
// A sequence's recurrent state is its conv state [W-1][Cc] and its SSM state
// [h_v][d_v][d_k], both fp32.  A snapshot is an exact copy of those bytes into
// another slot or another pool (a bank), and a restore is the copy back: the
// prefix-sharing pattern of "xwen" (README, batch mode: the shared prefix is
// prefilled once, its state kept, and every item restores it before its own
// tail) and the state "snapshot banks" of "Our own inference runtime" (section
// "What it is").  Since a copy is bit-exact, restore-and-continue reproduces the
// uninterrupted run bit for bit.
//
// The copy is a pure HBM stream: each CTA moves 32 KiB of one slot pair with
// 128-bit loads and stores, eight independent loads in flight per thread before
// the first store; grid = (chunks per slot, pairs).
#include "gdn_common.cuh"
#include "gdn_launch.h"
#include "../../include/gdn.h"

namespace gdn {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kVecPerThread = 8;
constexpr int kVecPerCta = kCopyThreads * kVecPerThread;  // float4 per CTA (32 KiB)

__global__ void __launch_bounds__(kCopyThreads) state_copy_kernel(StateCopyArgs p) {
  const int i = blockIdx.y;
  const int d = p.dst_idx ? p.dst_idx[i] : i;
  int s = i;
  if (p.src_ssm && p.src_idx) s = p.src_idx[i];
  if (d < 0 || d >= p.dst_slots || (p.src_ssm && (s < 0 || s >= p.src_slots))) {
    if (threadIdx.x == 0 && blockIdx.x == 0) record_status(p.status, GDN_ERR_DEVICE_BOUNDS);
    return;
  }
  const long long conv_vec = p.conv_floats / 4, ssm_vec = p.ssm_floats / 4;
  const long long total = conv_vec + ssm_vec;
  const long long base = (long long)blockIdx.x * kVecPerCta + threadIdx.x;

  // element e of the slot's state: conv state first, then the SSM state
  auto src_at = [&](long long e) -> const float4* {
    return e < conv_vec ? reinterpret_cast<const float4*>(p.src_conv + (size_t)s * p.conv_floats) + e
                        : reinterpret_cast<const float4*>(p.src_ssm + (size_t)s * p.ssm_floats) + (e - conv_vec);
  };
  auto dst_at = [&](long long e) -> float4* {
    return e < conv_vec ? reinterpret_cast<float4*>(p.dst_conv + (size_t)d * p.conv_floats) + e
                        : reinterpret_cast<float4*>(p.dst_ssm + (size_t)d * p.ssm_floats) + (e - conv_vec);
  };

  float4 v[kVecPerThread];
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const long long e = base + (long long)k * kCopyThreads;
    v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.src_ssm && e < total) v[k] = __ldg(src_at(e));
  }
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const long long e = base + (long long)k * kCopyThreads;
    if (e < total) *dst_at(e) = v[k];
  }
}

}  // namespace

cudaError_t launch_state_copy(const StateCopyArgs& p, cudaStream_t stream) {
  if (p.n <= 0) return cudaSuccess;
  const long long total = (p.conv_floats + p.ssm_floats) / 4;
  const long long chunks = (total + kVecPerCta - 1) / kVecPerCta;
  if (chunks > 0x7fffffffLL || p.n > 65535) return cudaErrorInvalidValue;
  state_copy_kernel<<<dim3((unsigned)chunks, (unsigned)p.n), kCopyThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
