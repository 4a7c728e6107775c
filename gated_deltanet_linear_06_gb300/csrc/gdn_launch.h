// gdn_launch.h -- argument packs and launchers of the libgdn kernels
// (internal to the library; the public surface is include/gdn.h).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

struct DecodeArgs {
  const uint16_t* qkv;     // bf16 [batch][Cc]
  const uint16_t* z;       // bf16 [batch][h_v][128]
  const uint16_t* a;       // bf16 [batch][h_v]
  const uint16_t* b;       // bf16 [batch][h_v]
  const float* A_log;      // [h_v]
  const float* dt_bias;    // [h_v]
  const uint16_t* conv_w;  // bf16 [Cc][4]
  const float* norm_w;     // [128]
  const int32_t* slot;     // nullable [batch]
  float* conv_state;       // [n_slots][3][Cc]
  float* ssm_state;        // [n_slots][h_v][128][128]
  void* out;               // [batch][h_v][128], bf16 or fp32
  int32_t* status;         // nullable device word
  int n_slots, batch, h_k, h_v;
  float l2_eps, rms_eps;
  // multi-token decode (launch_decode_multi): tokens per sequence, the token-major
  // activations above then being [batch][steps][...], and the nullable traces of
  // the states after every token
  int steps;
  float* ssm_trace;        // [batch][steps][h_v][128][128]
  float* conv_trace;       // [batch][steps][3][Cc]
};

struct PrefillArgs {
  const uint16_t* qkv;     // bf16 [T][Cc]
  const uint16_t* z;       // bf16 [T][h_v][128]
  const uint16_t* a;       // bf16 [T][h_v]
  const uint16_t* b;       // bf16 [T][h_v]
  const float* A_log;
  const float* dt_bias;
  const uint16_t* conv_w;  // bf16 [Cc][4]
  const float* norm_w;
  const int32_t* cu_seqlens;  // device [n_seqs + 1]
  float* conv_state;       // [n_seqs][3][Cc]
  float* ssm_state;        // [n_seqs][h_v][128][128]
  uint16_t* out;           // bf16 [T][h_v][128]
  int32_t* status;         // device word (workspace offset 0)
  void* scratch;           // workspace beyond the status word
  size_t scratch_bytes;
  // set by the launcher, inside the scratch area:
  int seg_tokens;          // segment length (sequences up to this long are one segment)
  int* seg_list;           // [count, pad x3][units][8]: the segments of every sequence
  int* multi_list;         // [count, pad x3][slots][4]: sequences longer than one segment
  float* xfer;             // per boundary slot and value head: transfer map, end state, initial state
  int* xzero;              // per boundary slot and value head: 1 where the transfer map is exactly zero
  int* chunk_off;          // [n_seqs + 1]: first chunk record of each sequence (split path; else null)
  int2* chunk_list;        // [max_chunks]: (sequence, first token) of each chunk record, sequence -1 past the end
  uint8_t* rec_kq;         // [max_chunks][h_k] per-chunk key/query tile records
  uint8_t* rec_v;          // [max_chunks][h_v] per-chunk value-head records
  int max_chunks;          // chunk records the workspace holds: total_tokens / 64 + n_seqs
  // the heads one launch of the prep / scan / combine passes covers (a call may
  // run as several head groups): key heads kh0 .. kh0+nkh-1, value heads
  // h0 .. h0+nh-1
  int kh0, nkh, h0, nh;
  int n_seqs, h_k, h_v;
  long long total_tokens;
  float l2_eps, rms_eps;
};

// Slot-to-slot copies of whole states (conv state then SSM state of a slot).
// Pair i copies source slot src_idx[i] (i when src_idx is null) to destination
// slot dst_idx[i] (i when null); with src_conv = src_ssm = null it zeroes the
// destination slot instead.  Slot indices are checked on the device.
struct StateCopyArgs {
  const float* src_conv;
  const float* src_ssm;
  const int32_t* src_idx;
  float* dst_conv;
  float* dst_ssm;
  const int32_t* dst_idx;
  int32_t* status;
  long long conv_floats;  // per slot: (W-1) * Cc
  long long ssm_floats;   // per slot: h_v * d_v * d_k
  int src_slots, dst_slots, n;
};

// Dense projection D = A B^T (bf16 operands, fp32 accumulation, bf16 out):
// A [M][K] and B [N][K] row-major (K contiguous, K % 8 == 0, 16-byte aligned
// bases).  The N output columns are split into runs: columns col0 ..
// col0+ncols-1 go to ptr[row * ld + (col - col0)] (col0, ncols, ld multiples
// of 8, ptr 16-byte aligned).
constexpr int kGemmMaxSegs = 4;
struct GemmOut {
  uint16_t* ptr;
  long long ld;
  int col0, ncols;
};
struct GemmArgs {
  const uint16_t* A;
  const uint16_t* B;
  int M, N, K;
  int nseg;
  GemmOut seg[kGemmMaxSegs];
  int32_t* status;         // nullable device word (bounded waits that give up)
};
cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream);

// Host launchers: enqueue on `stream`, return the launch error (or
// cudaSuccess).  Dims are validated by the caller.
cudaError_t launch_decode(const DecodeArgs& p, bool out_f32, cudaStream_t stream);
// p.steps tokens per sequence in one launch (1 <= steps <= kDecodeMaxSteps).
constexpr int kDecodeMaxSteps = 8;
cudaError_t launch_decode_multi(const DecodeArgs& p, bool out_f32, cudaStream_t stream);
// A chain of `steps` single steps in one persistent launch: p's activations
// and output are the chain's step-major buffers ([steps][batch][...]).  The
// state rows stay in registers through the chain; the conv state is read (the
// window before the first step) but not written --
// launch_decode_chain_conv_state writes it afterwards.  The results are
// bit-identical to `steps` launch_decode calls.
cudaError_t launch_decode_chain(const DecodeArgs& p, int steps, bool out_f32, cudaStream_t stream);
cudaError_t launch_decode_chain_conv_state(const DecodeArgs& p, const uint16_t* qkv0, int steps,
                                           cudaStream_t stream);
// n <= 65535 pairs per launch.
cudaError_t launch_state_copy(const StateCopyArgs& p, cudaStream_t stream);
// allow_split = false keeps every sequence in one segment (no transfer maps in
// the scratch); the scratch then needs only prefill_scratch_bytes_unsplit().
cudaError_t launch_prefill(const PrefillArgs& p, cudaStream_t stream, bool allow_split = true);
size_t prefill_scratch_bytes(int n_seqs, int h_k, int h_v, long long total_tokens);
size_t prefill_scratch_bytes_unsplit(int n_seqs);
// The segment length gdn_prefill splits long sequences into on a GPU with `sms`
// SMs, or 0 when it does not split (a whole number of chunks, >= 1024 tokens).
long long prefill_segment_tokens(int n_seqs, int h_v, long long total_tokens, int sms);

}  // namespace gdn
