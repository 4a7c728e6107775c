/*
 * gdn.h -- C ABI of libgdn, the Gated DeltaNet layer on NVIDIA GB300 (sm_103a).
 *
 * The layer.  The source pages name it as the linear-attention layer of
 * hybrid Qwen3.x-style models ("Serving large language models on our own
 * stack", section "Qwen3.5-35B-A3B from a real GGUF"; "Our own inference
 * runtime", section "What it is") and fix its serving properties: a
 * fixed-size recurrent state per sequence, constant regardless of position
 * (llmxabe README, architecture paragraph: ~60 MiB per sequence over 30
 * layers, i.e. 2 MiB fp32 per layer at 32 x 128 x 128), carried across
 * chunked prefill and decode (llmxabe README, the worker diagram:
 * "chunked-prefill scheduler"), and a decode that is bit-identical whether a
 * sequence runs alone or batched with others (llmxabe README, status and
 * "Accuracy is a hard gate" paragraphs).  The pages print no formula; the
 * layer computed here is the gated delta rule, per token t of a sequence:
 *
 *   y_t   = silu(causal depthwise conv_W(x)_t)      over the mixed q|k|v channels
 *   q^    = q / sqrt(|q|^2 + l2_eps) / sqrt(d_k),    k^ = k / sqrt(|k|^2 + l2_eps)
 *   g     = -exp(A_log[h]) * softplus(a_t[h] + dt_bias[h]),   beta = sigmoid(b_t[h])
 *   S_t   = exp(g) S_{t-1} (I - beta k^ k^T) + beta v k^T     (S: d_v x d_k, fp32)
 *   o_t   = S_t q^
 *   out_t = o_t / sqrt(mean(o_t^2) + rms_eps) * norm_w * silu(z_t[h])
 *
 * Value head h reads key head h / (h_v / h_k).  The conv weight w[c][W-1]
 * multiplies the current token and w[c][0] the oldest; there is no conv bias.
 *
 * Conventions for every call:
 *   - The caller owns all memory.  The library never allocates or frees
 *     device memory and never synchronises (gdn_read_device_status is the one
 *     call that waits; gdn_prefill_host from pageable host memory may wait in
 *     the runtime's copies).  The only resources it creates are, once per
 *     device, the side streams and events of gdn_prefill's head groups and of
 *     gdn_prefill_host's copies, and the CUDA graph a gdn_decode_graph handle
 *     owns until it is destroyed.
 *   - Calls are asynchronous on the given stream (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  The returned status covers
 *     host-side validation and the launch only.  Device-side checks
 *     (cu_seqlens contents, slot indices, bounded waits) write a code into a
 *     device status word instead of faulting; read it with
 *     gdn_read_device_status.
 *   - On GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED or GDN_ERR_WORKSPACE nothing
 *     was launched and no buffer was touched.  GDN_ERR_CUDA can follow part of
 *     a call's launches; the outputs and states are then undefined.
 *   - All device pointers must be 16-byte aligned.  Tensors are dense and
 *     row-major in the shapes given below.
 *   - Activations (qkv, z, a, b), conv weights and the prefill output are
 *     bf16 (raw uint16 bit patterns).  A_log, dt_bias, norm_w and both
 *     states are fp32.
 *   - The only dims compiled are d_k = d_v = 128, conv_w = 4, chunk = 64,
 *     h_v / h_k in {1, 2, 4}, h_k <= 64; anything else returns
 *     GDN_ERR_UNSUPPORTED.
 *   - No exception crosses this boundary.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,    /* null or misaligned pointer, bad size, inconsistent dims */
  GDN_ERR_UNSUPPORTED = 2,    /* dims outside the compiled fast path */
  GDN_ERR_WORKSPACE = 3,      /* workspace missing or smaller than gdn_workspace_bytes */
  GDN_ERR_CUDA = 4,           /* a CUDA runtime call failed (launch, attribute, copy) */
  GDN_ERR_DEVICE_TIMEOUT = 5, /* device word: a bounded device-side wait gave up */
  GDN_ERR_DEVICE_BOUNDS = 6   /* device word: cu_seqlens or a slot index out of range */
} gdn_status;

/* Layer dimensions.  d_k / d_v: key / value head size; conv_w: conv width;
 * chunk: prefill chunk length; the epsilons of the two norms. */
typedef struct gdn_dims {
  int h_k;
  int h_v;
  int d_k;
  int d_v;
  int conv_w;
  int chunk;
  float l2_eps;
  float rms_eps;
} gdn_dims;

enum { GDN_DTYPE_BF16 = 0, GDN_DTYPE_F32 = 1 };

/* Library version: major * 10000 + minor * 100 + patch. */
int gdn_version(void);

/* Human-readable name of a status code (static storage, never NULL). */
const char* gdn_status_string(gdn_status status);

/* Bytes of carried state per sequence: the fp32 SSM state
 * [h_v][d_v][d_k] plus the fp32 conv state [conv_w - 1][Cc], with
 * Cc = 2 h_k d_k + h_v d_v.  A snapshot of a sequence is a copy of these
 * bytes (the pages' state "snapshot banks": "Our own inference runtime",
 * section "What it is").  Returns 0 for invalid dims. */
size_t gdn_state_bytes(const gdn_dims* dims);

/* Device workspace gdn_prefill needs for this problem (>= 256 bytes; holds
 * the device status word at offset 0).  Returns 0 for invalid arguments. */
size_t gdn_workspace_bytes(const gdn_dims* dims, int n_seqs, long long total_tokens);

/* The segment length, in tokens, that gdn_prefill on the current device splits
 * the sequences of this problem into: a multiple of the chunk (64), at least
 * 1024, chosen from the token count, the value heads and the SM count; 0 when
 * the call splits nothing (enough sequences to fill the GPU, or too few
 * tokens); -1 for invalid arguments or when no device can be queried.  A
 * chunked-prefill scheduler can use it to align its own boundaries; segments
 * never change results beyond rounding. */
long long gdn_prefill_segment_tokens(const gdn_dims* dims, int n_seqs, long long total_tokens);
/* The same choice for a GPU with `sms` SMs, without touching a device (for
 * schedulers that plan ahead, and for tests); -1 for invalid arguments. */
long long gdn_prefill_segment_tokens_for(const gdn_dims* dims, int n_seqs, long long total_tokens,
                                         int sms);

/*
 * Chunked prefill over cu_seqlens-packed variable-length sequences.
 *
 * Runs the layer over every token of n_seqs sequences packed back to back
 * (no padding), each starting from its carried states, and leaves the
 * states after its last token in place -- so a long prompt can be fed in
 * segments, as a chunked-prefill scheduler does (llmxabe README, worker
 * diagram), and a segment continues exactly where the previous one stopped.
 *
 *   qkv        bf16 [total_tokens][Cc]            channel order q | k | v (input)
 *   z          bf16 [total_tokens][h_v][d_v]      output-gate input (input)
 *   a, b       bf16 [total_tokens][h_v]           decay / write-gate inputs (input)
 *   A_log      fp32 [h_v];  dt_bias fp32 [h_v]    (input)
 *   conv_w     bf16 [Cc][conv_w]                  (input)
 *   norm_w     fp32 [d_v]                         RMSNorm weight, shared by heads (input)
 *   cu_seqlens int32 [n_seqs + 1], DEVICE memory, cu_seqlens[0] = 0,
 *              non-decreasing, cu_seqlens[n_seqs] = total_tokens.  Violations
 *              are caught on the device: the call then writes nothing and sets
 *              GDN_ERR_DEVICE_BOUNDS in the status word.
 *   conv_state fp32 [n_seqs][conv_w - 1][Cc]      in/out: raw inputs of the last
 *              conv_w - 1 tokens, oldest first (zeros = fresh sequence)
 *   ssm_state  fp32 [n_seqs][h_v][d_v][d_k]       in/out (zeros = fresh sequence)
 *   out        bf16 [total_tokens][h_v][d_v]      (output)
 *   workspace  device buffer of >= gdn_workspace_bytes(dims, n_seqs,
 *              total_tokens) bytes, 256-byte aligned; its status word is reset
 *              by the call itself.
 * Empty sequences are allowed and leave their states unchanged.  n_seqs = 0
 * or total_tokens = 0 launches nothing and returns GDN_OK.
 *
 * Streams: when some sequence is split into segments (few sequences, so one
 * CTA per (sequence, value head) would leave the GPU short) and h_k is a
 * multiple of 4, the call runs as 4 groups of key heads: the first on `stream`,
 * the others on side streams of the library that wait for `stream` through an
 * event and that `stream` waits for again before the call's last kernel.  Work
 * enqueued on `stream` afterwards therefore sees the call complete, as with a
 * single-stream call; it also works under stream capture.  Concurrent calls
 * on one device from several host threads share the side streams (and are
 * ordered on them).
 */
gdn_status gdn_prefill(const gdn_dims* dims, const void* qkv, const void* z,
                       const void* a, const void* b, const float* A_log,
                       const float* dt_bias, const void* conv_w,
                       const float* norm_w, const int32_t* cu_seqlens,
                       int n_seqs, long long total_tokens, float* conv_state,
                       float* ssm_state, void* out, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * One decode step for a batch of sequences, one token each.
 *
 * Per sequence this is the same arithmetic in the same order whatever the
 * batch size or the batch's other members: a sequence decodes bit-identically
 * alone or batched (llmxabe README, "Accuracy is a hard gate" paragraph).
 *
 *   qkv  bf16 [batch][Cc];  z bf16 [batch][h_v][d_v];  a, b bf16 [batch][h_v]
 *   A_log, dt_bias, conv_w, norm_w   as for gdn_prefill
 *   slot       NULL: batch entry i uses state i of the arrays below.
 *              Else int32 [batch] DEVICE memory: entry i uses state slot[i],
 *              0 <= slot[i] < n_slots, all distinct.  An out-of-range entry
 *              is skipped on the device (its out row is left untouched) and
 *              GDN_ERR_DEVICE_BOUNDS is written to *device_status if given.
 *   n_slots    number of states in the arrays (>= batch when slot is NULL).
 *   conv_state fp32 [n_slots][conv_w - 1][Cc]   in/out
 *   ssm_state  fp32 [n_slots][h_v][d_v][d_k]    in/out
 *   out        [batch][h_v][d_v], bf16 or fp32 per out_dtype (output)
 *   device_status  NULL or a device int32 word that device checks write into
 *              (never cleared by this call).
 * batch = 0 launches nothing and returns GDN_OK.
 */
gdn_status gdn_decode_step(const gdn_dims* dims, const void* qkv, const void* z,
                           const void* a, const void* b, const float* A_log,
                           const float* dt_bias, const void* conv_w,
                           const float* norm_w, const int32_t* slot,
                           int n_slots, int batch, float* conv_state,
                           float* ssm_state, void* out, int out_dtype,
                           int32_t* device_status, void* stream);

/*
 * gdn_decode_step with the step's activations and output in HOST memory, for a
 * serving loop that keeps each step's tokens on the host (llmxabe README,
 * worker diagram: the worker owns the host side of every step).  The step
 * runs on `stream` as gdn_decode_step does (same bits).  When all five host
 * buffers are page-locked memory the device can address, its kernel reads the
 * inputs and writes the output in place over the host link (no copies);
 * otherwise qkv, z, a and b are first copied into the workspace and the output
 * is copied to `out` after the step, on `stream`.
 *
 *   qkv, z, a, b   HOST, layouts as for gdn_decode_step; page-locked memory
 *                  (cudaHostAlloc, torch pin_memory) is used in place,
 *                  pageable memory still works (the copies then block the
 *                  calling thread)
 *   out            HOST [batch][h_v][d_v], bf16 or fp32 per out_dtype (output;
 *                  written once the stream reaches the end of the call)
 *   A_log, dt_bias, conv_w, norm_w, slot, conv_state, ssm_state, device_status
 *                  DEVICE, as for gdn_decode_step
 *   workspace      DEVICE, 256-byte aligned, >= the bytes below (staging for
 *                  the step's inputs and output when they are copied; not
 *                  touched by other calls)
 * The host buffers are read and written when the stream executes the call:
 * leave the inputs unchanged and do not read `out` until the stream has passed
 * it (as with any asynchronous copy).  Every argument is checked before
 * anything is enqueued.  batch = 0 does nothing and returns GDN_OK.
 */
size_t gdn_decode_step_host_workspace_bytes(const gdn_dims* dims, int batch, int out_dtype);
gdn_status gdn_decode_step_host(const gdn_dims* dims, const void* qkv, const void* z,
                                const void* a, const void* b, const float* A_log,
                                const float* dt_bias, const void* conv_w,
                                const float* norm_w, const int32_t* slot, int n_slots,
                                int batch, float* conv_state, float* ssm_state, void* out,
                                int out_dtype, int32_t* device_status, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * gdn_prefill with the activations in HOST memory: the call copies the inputs
 * in and the output out itself, overlapping the host link with the compute.
 *
 * The packed tokens are cut into segments of seg_tokens (0: 5120) tokens, fed
 * as a chunked-prefill scheduler would (llmxabe README, worker diagram): each
 * segment is one gdn_prefill call whose sequences continue from the states the
 * previous segment left.  Two library copy streams move segment i+1's inputs
 * host->device and segment i-1's output device->host while segment i computes.
 * The result equals those gdn_prefill calls made one after another (a segment
 * boundary inside a sequence changes rounding only, as any chunked prefill).
 *
 *   qkv, z, a, b   HOST bf16, layouts as for gdn_prefill; pinned (page-locked)
 *                  memory lets the copies overlap, pageable memory still works
 *   A_log, dt_bias, conv_w, norm_w   DEVICE, as for gdn_prefill
 *   cu_seqlens     HOST int32 [n_seqs + 1], read during the call (checked on
 *                  the host: 0 first, non-decreasing, total_tokens last)
 *   conv_state, ssm_state            DEVICE, in/out, as for gdn_prefill
 *   out            HOST bf16 [total_tokens][h_v][d_v] (output)
 *   seg_tokens     0 or >= 64
 *   workspace      DEVICE, 256-byte aligned, >= gdn_prefill_host_workspace_bytes();
 *                  the int32 at offset 0 holds the first nonzero device status of
 *                  any segment (read it with gdn_read_device_status)
 * Everything is ordered after the caller's earlier work on `stream`, and work
 * enqueued on `stream` afterwards sees the output in host memory.  Not for
 * stream capture.  Concurrent calls on one device share the copy streams.
 */
size_t gdn_prefill_host_workspace_bytes(const gdn_dims* dims, int n_seqs, long long total_tokens,
                                        int seg_tokens);
/*
 * The segments gdn_prefill_host cuts a batch into (host only, no device use):
 * returns their count, or -1 for invalid arguments (cu_seqlens as for
 * gdn_prefill_host, seg_tokens 0 or >= 64), and writes the first max_segs of
 * them to seg_info as {first token, end token, first sequence, sequence
 * count}.  Segment i covers tokens [i * seg, min((i + 1) * seg, total)) and the
 * sequences from the one holding its first token to the one holding its last;
 * an empty sequence at a segment boundary belongs to no segment (its states
 * stay as they are).
 */
long long gdn_prefill_host_segments(const int32_t* cu_seqlens, int n_seqs, long long total_tokens,
                                    int seg_tokens, long long* seg_info, long long max_segs);
gdn_status gdn_prefill_host(const gdn_dims* dims, const void* qkv, const void* z, const void* a,
                            const void* b, const float* A_log, const float* dt_bias,
                            const void* conv_w, const float* norm_w, const int32_t* cu_seqlens,
                            int n_seqs, long long total_tokens, float* conv_state,
                            float* ssm_state, void* out, int seg_tokens, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * Copy whole sequence states between slots of caller-owned state pools:
 * snapshot a prefix's state into a bank and restore it later, or fork one
 * sequence's state into several ("xwen" README, batch mode: the shared prefix
 * is prefilled once and restored for every item; "Our own inference runtime",
 * section "What it is": state "snapshot banks").  The copy is exact, so
 * decoding or prefilling from a restored state gives, bit for bit, what the
 * uninterrupted run gives.
 *
 *   src_conv_state, src_ssm_state  fp32 [src_slots][W-1][Cc], [src_slots][h_v][d_v][d_k]
 *   dst_conv_state, dst_ssm_state  fp32 [dst_slots][...] the same per-slot layout (output)
 *   src_slot, dst_slot  NULL (pair i uses slot i; the pool then needs >= n slots)
 *              or int32 [n] DEVICE arrays of slot indices.  A pair whose index is
 *              out of range is skipped on the device and GDN_ERR_DEVICE_BOUNDS is
 *              written to *device_status if given.
 *   n          pairs, 0 .. 65535 (0 launches nothing)
 * The source and destination slots of one call must not overlap, and no
 * destination slot may appear twice (the copies run concurrently).  Any dims
 * gdn_decode_step accepts; other dims return the same status it does.
 */
gdn_status gdn_state_copy(const gdn_dims* dims, const float* src_conv_state,
                          const float* src_ssm_state, int src_slots, const int32_t* src_slot,
                          float* dst_conv_state, float* dst_ssm_state, int dst_slots,
                          const int32_t* dst_slot, int n, int32_t* device_status, void* stream);

/*
 * Zero the conv and SSM states of n slots of a state pool: the start of a new
 * sequence in a reused slot.  Arguments as for gdn_state_copy's destination.
 */
gdn_status gdn_state_reset(const gdn_dims* dims, float* conv_state, float* ssm_state, int n_slots,
                           const int32_t* slot, int n, int32_t* device_status, void* stream);

/*
 * A CUDA graph of `steps` successive gdn_decode_step calls, for small batches
 * whose steps are launch-bound (three sequences decode a step in a few
 * microseconds of HBM time).  The buffers are bound when the graph is
 * created; the caller refills them between launches.
 *
 *   qkv  bf16 [steps][batch][Cc];  z bf16 [steps][batch][h_v][d_v];
 *   a, b bf16 [steps][batch][h_v]     step t's tokens at [t]
 *   out        [steps][batch][h_v][d_v], bf16 or fp32 per out_dtype
 *   the rest   as for gdn_decode_step (the states advance by `steps` tokens
 *              per launch)
 *   steps 1 .. 2^20, batch >= 1
 *   *graph     receives the handle (NULL on failure)
 * gdn_decode_graph_launch enqueues one run of all the steps on `stream`;
 * results are bit-identical to the same gdn_decode_step calls made one by
 * one.  gdn_decode_graph_destroy frees the handle (NULL is a no-op); the
 * caller must not destroy a graph with a launch still in flight.
 */
typedef struct gdn_decode_graph gdn_decode_graph;

gdn_status gdn_decode_graph_create(const gdn_dims* dims, int steps, const void* qkv, const void* z,
                                   const void* a, const void* b, const float* A_log,
                                   const float* dt_bias, const void* conv_w, const float* norm_w,
                                   const int32_t* slot, int n_slots, int batch, float* conv_state,
                                   float* ssm_state, void* out, int out_dtype,
                                   int32_t* device_status, gdn_decode_graph** graph);
gdn_status gdn_decode_graph_launch(gdn_decode_graph* graph, void* stream);
void gdn_decode_graph_destroy(gdn_decode_graph* graph);

/*
 * Self-test of the device-side failure path.  Launches one CTA whose threads
 * wait, with the kernels' bounded wait and a budget of budget_cycles clock
 * cycles (1 .. 2^31; about 2 GHz), on a shared-memory barrier that nothing
 * completes.  The wait gives up, GDN_ERR_DEVICE_TIMEOUT is written to
 * *device_status (a device int32, left alone if it already holds a code) and
 * the kernel exits; the context stays usable.  The status returned covers the
 * launch only.
 */
gdn_status gdn_selftest_wait_timeout(int32_t* device_status, long long budget_cycles, void* stream);

/* Most tokens per sequence one gdn_decode_multi call takes. */
#define GDN_DECODE_MAX_STEPS 8

/*
 * `steps` decode steps per sequence in one call: multi-token decode, or the
 * verification pass of speculative decoding (the draft tokens of every
 * sequence at once).  The result is bit-identical to `steps` successive
 * gdn_decode_step calls on the same tokens -- every step repeats that call's
 * arithmetic in its order -- while each state is read and written once per
 * call instead of once per token.
 *
 *   qkv  bf16 [batch][steps][Cc];  z bf16 [batch][steps][h_v][d_v];
 *   a, b bf16 [batch][steps][h_v]  (token t of sequence i at [i][t])
 *   A_log, dt_bias, conv_w, norm_w, slot, n_slots, conv_state, ssm_state,
 *   device_status   as for gdn_decode_step; the states end after the last token
 *   steps      1 .. GDN_DECODE_MAX_STEPS
 *   out        [batch][steps][h_v][d_v], bf16 or fp32 per out_dtype (output)
 *   ssm_trace  NULL, or fp32 [batch][steps][h_v][d_v][d_k]: the SSM state after
 *              each token (for rolling back to the last accepted draft token);
 *              it costs one more state write per token
 *   conv_trace NULL, or fp32 [batch][steps][conv_w - 1][Cc]: the conv state
 *              after each token
 * batch = 0 launches nothing and returns GDN_OK.
 */
gdn_status gdn_decode_multi(const gdn_dims* dims, const void* qkv, const void* z,
                            const void* a, const void* b, const float* A_log,
                            const float* dt_bias, const void* conv_w, const float* norm_w,
                            const int32_t* slot, int n_slots, int batch, int steps,
                            float* conv_state, float* ssm_state, void* out, int out_dtype,
                            float* ssm_trace, float* conv_trace, int32_t* device_status,
                            void* stream);

/*
 * Prefill for callers that cannot allocate device memory.
 *
 * The source pages have no counterpart to this call: it exists for callers
 * that cannot hand the library a device workspace at the point where they run
 * the layer -- for instance a step recorded under a strict memory budget, an
 * allocator that forbids new device allocations after start-up, or a host
 * framework that gives the layer no allocation hook.  It computes the same
 * prefill as gdn_prefill (same arguments, layouts and outputs) and allocates
 * nothing: its scratch -- the device status word and the segment list --
 * lives in one fixed device array of GDN_NOALLOC_SCRATCH_BYTES bytes inside
 * the library, which every GPU that loads the library holds until the process
 * exits.
 *
 * Limits and behaviour:
 *   - n_seqs above GDN_NOALLOC_MAX_SEQS returns GDN_ERR_UNSUPPORTED without
 *     launching (the fixed array holds no more).
 *   - Sequences are never split into parallel segments (that needs transfer
 *     maps far larger than the fixed array), so a batch of few long sequences
 *     runs slower than through gdn_prefill; the results agree within the
 *     prefill tolerance.
 *   - The first call in a CUDA context looks up the array's device address
 *     (once per context, with that context's device current) and caches it
 *     under the context's id, so a context rebuilt after cudaDeviceReset looks
 *     it up again; make that first call before any stream capture.
 *   - All calls share the one array, which keeps the previous call's
 *     contents; each call clears the status word itself.  Calls whose work
 *     overlaps on the GPU (other streams, other host threads, concurrent
 *     graph launches) race on the array and must be serialised by the caller.
 *   - device_status: NULL, or a device int32 word that receives a copy of the
 *     call's status word (GDN_OK or the first device-side error) in stream
 *     order, for gdn_read_device_status.  With NULL the device-side errors of
 *     the call are lost: a rejected cu_seqlens (GDN_ERR_DEVICE_BOUNDS, nothing
 *     written, so out and the states keep their old contents) or a bounded
 *     wait that gave up (GDN_ERR_DEVICE_TIMEOUT) goes only to the library's
 *     internal word, which the next call clears.
 */
#define GDN_NOALLOC_MAX_SEQS 32768
#define GDN_NOALLOC_SCRATCH_BYTES 1049344 /* status word + segment list for GDN_NOALLOC_MAX_SEQS */

gdn_status gdn_prefill_noalloc(const gdn_dims* dims, const void* qkv, const void* z,
                               const void* a, const void* b, const float* A_log,
                               const float* dt_bias, const void* conv_w,
                               const float* norm_w, const int32_t* cu_seqlens,
                               int n_seqs, long long total_tokens, float* conv_state,
                               float* ssm_state, void* out, int32_t* device_status,
                               void* stream);

/*
 * The dense projections around the layer.  In the hybrid models the pages
 * run, every Gated DeltaNet layer sits between an input projection of the
 * hidden state and an output projection back to it ("Serving large language
 * models on our own stack", section "Qwen3.5-35B-A3B from a real GGUF";
 * llmxabe README, architecture paragraph: three Gated DeltaNet layers per
 * gated-attention layer).  Both are y = x w^T on the tensor cores, with bf16
 * operands, fp32 accumulation and the result rounded to bf16 (nearest even).
 * Weights are in the output-features-by-input-features layout.
 *
 * gdn_in_proj writes its output columns straight into the layer's input
 * buffers, in the layouts gdn_prefill and gdn_decode_step read, so nothing is
 * copied between the projection and the layer:
 *   x      bf16 [tokens][hidden]                    (input)
 *   w_in   bf16 [Cc + h_v d_v + 2 h_v][hidden]      rows in the order: the Cc
 *          mixed q|k|v conv channels, z (value head major), a (h_v), b (h_v)
 *   qkv    bf16 [tokens][Cc];  z bf16 [tokens][h_v][d_v];
 *   a, b   bf16 [tokens][h_v]                       (outputs)
 *
 * gdn_out_proj maps the layer's output to the hidden size:
 *   o      bf16 [tokens][h_v][d_v]                  (the gdn_prefill / bf16 decode output)
 *   w_out  bf16 [hidden][h_v d_v]
 *   y      bf16 [tokens][hidden]                    (output)
 *
 * hidden: a multiple of 64, at most 65536 (else GDN_ERR_UNSUPPORTED); h_v a
 * multiple of 8; tokens 0 .. 2^31 - 1 (0 launches nothing); dims as for
 * gdn_prefill.  device_status: NULL or a device int32 word that a bounded
 * wait that gave up writes GDN_ERR_DEVICE_TIMEOUT into.  The kernel keeps one
 * CTA per SM resident for the call and uses all of its tensor memory.
 */
gdn_status gdn_in_proj(const gdn_dims* dims, int hidden, long long tokens, const void* x,
                       const void* w_in, void* qkv, void* z, void* a, void* b,
                       int32_t* device_status, void* stream);
gdn_status gdn_out_proj(const gdn_dims* dims, int hidden, long long tokens, const void* o,
                        const void* w_out, void* y, int32_t* device_status, void* stream);

/* Waits for the stream, then reads a device status word (the first 4 bytes
 * of a prefill workspace, or a decode device_status word) into *code:
 * GDN_OK or the first device-side error recorded.  Returns GDN_ERR_CUDA if
 * the copy or the wait failed. */
gdn_status gdn_read_device_status(const void* status_word, void* stream,
                                  int32_t* code);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
