/*
 * gdn.h -- C ABI of the Gated DeltaNet (GDN) linear-attention layer core for
 * NVIDIA GB300 (sm_103a).
 *
 * The layer core sits between the input projections and out_proj of a GDN
 * layer of the hybrid DeltaNet/GQA models Qwen3.6-27B and Qwen3-Coder-Next:
 *
 *   mixed_qkv --conv1d+SiLU--> [q | k | v] --l2norm(q,k), gates g/beta-->
 *   gated delta rule (chunked prefill or per-token decode) --> o
 *   --RMSNormGated(o, z)--> out
 *
 * Definitions follow the cortex commit "feat(stage-8c): linear-attention layer
 * (Qwen3-Next GatedDeltaNet)" (sections "Block", "Discretisation", "Delta rule
 * (recurrent, per-token)", "Output", "State (GatedDeltaNetState)") and the
 * NxD-Inference PR "Add Qwen3.6-27B hybrid DeltaNet/GQA contrib model and vLLM
 * serving path" (Summary: chunked context encoding, token generation, GDN
 * recurrent and convolution state checkpoints for hybrid prefix caching).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers marked (device) are CUDA device pointers; (host) are host memory.
 *   The caller owns every buffer.  The library allocates no device memory:
 *   scratch is a caller-sized workspace (see gdn_chunk_prefill_workspace_size).
 *   Its persistent objects are two: a fixed scratch array compiled into the
 *   library for gdn_chunk_prefill_noalloc, and three CUDA streams per device
 *   context that gdn_layer_prefill_host creates on its first call there
 *   (released with the context).
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream), except where a call says it synchronises.
 * - Tensors are dense, row-major, in the shapes given per argument.  Device
 *   pointers must be 16-byte aligned (GDN_ERR_ALIGN otherwise).
 * - Arguments are validated before anything is launched.  On any error
 *   nothing is written and nothing is launched.  No C++ exception crosses the
 *   ABI.  GDN_ERR_CUDA means a launch failed: gdn_last_cuda_error() returns
 *   the cudaError_t of the calling thread's last failure.
 * - `dtype` gives the element type of the activations (x, y, qkv, z, a, b, o,
 *   out), the conv weight, the conv state and the RMSNormGated weight.  A_log,
 *   dt_bias, g, beta and the recurrent state are always float32.
 * - Dimensions: H_k query/key heads, H_v value heads (a multiple of H_k),
 *   head dims d_k = d_v = D, conv kernel width conv_k = 4,
 *   conv_dim = 2*H_k*d_k + H_v*d_v.  Value head h reads key head
 *   h / (H_v / H_k) (repeat_interleave order).
 * - Supported: D in {16, 128} for GDN_F32; D = 128 for GDN_BF16 (the tensor-
 *   core path); conv_k = 4.  Other shapes return GDN_ERR_UNSUPPORTED.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* NULL where a buffer is required, bad size or flag */
    GDN_ERR_ALIGN = 2,       /* a device pointer is not 16-byte aligned          */
    GDN_ERR_UNSUPPORTED = 3, /* dims the kernels do not cover                     */
    GDN_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required        */
    GDN_ERR_CUDA = 5,        /* a CUDA call or launch failed                      */
    GDN_ERR_TIMEOUT = 6      /* a bounded device-side wait gave up                */
} gdn_status_t;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype_t;

typedef struct {
    int32_t H_k, H_v, d_k, d_v, conv_k;
} gdn_dims_t;

/* flags of gdn_chunk_prefill / gdn_recurrent_decode */
#define GDN_QK_L2NORM 1u /* l2-normalise q and k per head (eps 1e-6 inside the sqrt) */
/* gdn_chunk_prefill only, tensor-core path (bf16, d = 128): form each chunk's
 * (I + A)^-1 as the Neumann-style product (I + N)(I + N^2)...(I + N^32),
 * N = -A, instead of the direct solve.  NxD-Inference Qwen3.6-27B PR, "Known
 * limitations" (a faster Neumann-style path against the stable direct solve).
 * Exact in exact arithmetic (A is nilpotent) but unstable when the chunk's
 * inverse is far from the identity (slow decay, correlated keys); shipped to
 * compare the two.  Other paths: GDN_ERR_UNSUPPORTED. */
#define GDN_SOLVE_NEUMANN 2u
/* gdn_chunk_prefill (and the calls built on it): the chunk size C, in flag
 * bits 8..15 -- GDN_CHUNK(16), GDN_CHUNK(32) or GDN_CHUNK(64); the field left
 * at 0 means 64.  Any C gives the per-token rule's result up to rounding
 * (cortex GatedDeltaNet commit, "Performance note": chunk_size=64 is one
 * choice of the chunked algorithm); it trades per-chunk matrix work (which
 * grows with C) against the number of sequential chunk steps.  Both paths take
 * all three.  The tensor-core path (bf16, d = 128) keeps its tiles at 64 rows:
 * a chunk of 16 or 32 tokens fills the first rows of its tile, so it costs
 * about what a chunk of 64 does, and the call runs in more workspace segments
 * (the same workspace size), between which the state crosses through
 * final_state, which these chunk sizes require there (else
 * GDN_ERR_UNSUPPORTED).  Other values: GDN_ERR_INVALID_ARG. */
#define GDN_CHUNK(c) ((((uint32_t)(c)) & 0xffu) << 8)

/* Text for a status code (static storage, never NULL). */
const char* gdn_status_string(gdn_status_t status);

/* cudaError_t of the calling thread's last GDN_ERR_CUDA (0 if none). */
int gdn_last_cuda_error(void);

/* ABI version: (major << 16) | minor. */
int gdn_version(void);

/*
 * Number of checkpoint rows for packed sequences: sum_i floor(L_i / every),
 * L_i = cu_seqlens[i+1] - cu_seqlens[i].  cu_seqlens (host) has n_seq + 1
 * entries.  Returns -1 on invalid input (NULL, n_seq < 1, every < 0,
 * decreasing offsets).  every == 0 returns 0.
 */
int64_t gdn_ckpt_count(const int32_t* cu_seqlens, int32_t n_seq, int32_t every);

/*
 * Validates packed-sequence offsets that live on the device: cu_seqlens[0] == 0,
 * non-decreasing, cu_seqlens[n_seq] == T_tot.  SYNCHRONISES `stream` (copies the
 * n_seq + 1 offsets to the host).  Returns GDN_OK or GDN_ERR_INVALID_ARG.
 * The compute calls below do not read offsets on the host; on the device they
 * clamp every sequence to [0, T_tot) so bad offsets cannot make them access
 * memory out of bounds, but the results are then meaningless.
 */
gdn_status_t gdn_check_cu_seqlens(const int32_t* cu_seqlens, int32_t n_seq, int64_t T_tot,
                                  void* stream);

/*
 * SYNCHRONISES `stream`, then reports failures that happened on the device
 * after the calls above returned: GDN_ERR_TIMEOUT if a kernel of this library
 * gave up one of its bounded waits (about 1 s each) since the last call -- its
 * outputs are then incomplete -- and clears that record; GDN_ERR_CUDA if the
 * stream holds a CUDA error; GDN_OK otherwise.
 */
gdn_status_t gdn_sync_status(void* stream);

/*
 * Prefill depthwise causal conv1d (width conv_k = 4) with state prepend and
 * optional SiLU, over packed sequences.
 * Defined by: cortex GatedDeltaNet commit, "Block" (depthwise causal Conv1d
 * (k=4) with state-aware prepend; SiLU) and "State" (conv_state, the
 * left-padded tail of raw inputs); NxD-Inference Qwen3.6-27B PR, Summary
 * (convolution state checkpoints).
 *
 *   x          (device) [T_tot, conv_dim]            raw mixed_qkv
 *   w          (device) [conv_dim, 4]                tap 3 multiplies the current token
 *   cu_seqlens (device) [n_seq + 1] int32, or NULL for one sequence of T_tot tokens
 *   conv_state_in  (device) [n_seq, conv_dim, 3] or NULL (zeros): the 3 raw inputs
 *                  preceding each sequence, column 0 oldest
 *   conv_state_out (device) [n_seq, conv_dim, 3] or NULL: the 3 newest raw inputs of
 *                  [state_in | x] per sequence (bit copies).  May alias conv_state_in.
 *   ckpt_every     0 (off) or a positive multiple of 64: conv_ckpt_out row r holds the
 *                  conv state after m*ckpt_every tokens of a sequence, m = 1..floor(L/N),
 *                  rows in sequence order (gdn_ckpt_count rows), [rows, conv_dim, 3]
 *   ckpt_rows      rows allocated in conv_ckpt_out; rows past it are never written;
 *                  with 0 rows conv_ckpt_out may be NULL
 *   apply_silu     nonzero: y = silu(conv)
 *   y          (device) [T_tot, conv_dim]  (must not alias x)
 * Arithmetic: f32 accumulation; y is rounded once to `dtype`.
 */
gdn_status_t gdn_conv1d_fwd(const void* x, const void* w, const int32_t* cu_seqlens,
                            int32_t n_seq, int64_t T_tot, const void* conv_state_in,
                            void* conv_state_out, int32_t ckpt_every, void* conv_ckpt_out,
                            int64_t ckpt_rows, int32_t apply_silu, void* y, gdn_dims_t dims, gdn_dtype_t dtype,
                            void* stream);

/*
 * Decode conv update for B sequences, one token each.
 * Defined by: cortex GatedDeltaNet commit, "Block" and "State" (as above).
 *   x          (device) [B, conv_dim]
 *   w          (device) [conv_dim, 4]
 *   conv_state (device) [B, conv_dim, 3], updated in place: shifted left by one
 *              column, x appended as column 2
 *   y          (device) [B, conv_dim] = silu(w . [state | x]) (or without SiLU)
 */
gdn_status_t gdn_conv1d_update(const void* x, const void* w, void* conv_state, int32_t B,
                               int32_t apply_silu, void* y, gdn_dims_t dims, gdn_dtype_t dtype,
                               void* stream);

/*
 * Workspace bytes gdn_chunk_prefill needs for these sizes (0 = none; then
 * `workspace` may be NULL).
 */
size_t gdn_chunk_prefill_workspace_size(int32_t n_seq, int64_t T_tot, gdn_dims_t dims,
                                        gdn_dtype_t dtype);

/*
 * The layer core -- conv1d + SiLU, chunked delta rule, RMSNormGated, as in
 * gdn_conv1d_fwd, gdn_chunk_prefill and gdn_rmsnorm_gated -- for ONE sequence
 * whose activations and output are in page-locked host memory (the pages have
 * no counterpart; this is the host-buffer form of the three calls).  The tokens
 * run in gdn_layer_prefill_host_pieces pieces of at most
 * gdn_layer_prefill_host_piece tokens, cut at multiples of 64 (when T is a
 * whole number of full pieces the last is cut into 3/4 and 1/4, so little work
 * remains after the last copy in).  A piece's inputs are copied to the device
 * while earlier pieces compute and its output is copied back while later ones
 * do; the copies, each piece's conv and chunk-local kernels, and the state
 * chain + RMSNormGated run on three internal streams of the library and
 * `stream`, starting after the work already queued on `stream` and joined back
 * to it.  The conv state and the recurrent state carry from piece to piece on
 * the device, so the result equals gdn_layer_prefill's (and the three device
 * calls') bit for bit.
 *   h_qkv      (host, page-locked) [T, conv_dim]    dtype
 *   h_z        (host, page-locked) [T, H_v*d_v]     dtype
 *   h_a, h_b   (host, page-locked) [T, H_v]         dtype
 *   conv_w     (device) [conv_dim, 4] dtype;  norm_w (device) [d_v] dtype
 *   A_log, dt_bias (device) [H_v] f32
 *   initial_state  (device) [1, H_v, d_k, d_v] f32, or NULL (zeros)
 *   final_state    (device) [1, H_v, d_k, d_v] f32, required; may alias initial_state
 *   conv_state_in  (device) [1, conv_dim, 3] dtype, or NULL (zeros)
 *   conv_state_out (device) [1, conv_dim, 3] dtype, required; may alias conv_state_in
 *   scale      0 -> d_k^-1/2;  flags: GDN_QK_L2NORM;  norm_eps > 0 (the layer uses 1e-6)
 *   h_out      (host, page-locked) [T, H_v*d_v] dtype
 *   workspace  (device) >= gdn_layer_prefill_host_workspace_size(T, dims, dtype) bytes
 * Host buffers that are not page-locked: GDN_ERR_INVALID_ARG.  No checkpoints.
 * Make the first call on a device before any stream capture (it creates the
 * three internal streams).  h_out is complete once `stream` reaches this point.
 */
size_t gdn_layer_prefill_host_workspace_size(int64_t T, gdn_dims_t dims, gdn_dtype_t dtype);
int64_t gdn_layer_prefill_host_piece(int64_t T, gdn_dims_t dims, gdn_dtype_t dtype);
int64_t gdn_layer_prefill_host_pieces(int64_t T, gdn_dims_t dims, gdn_dtype_t dtype);
gdn_status_t gdn_layer_prefill_host(const void* h_qkv, const void* h_z, const void* h_a,
                                    const void* h_b, const void* conv_w, const float* A_log,
                                    const float* dt_bias, const void* norm_w, int64_t T,
                                    const float* initial_state, float* final_state,
                                    const void* conv_state_in, void* conv_state_out, float scale,
                                    uint32_t flags, float norm_eps, void* h_out, void* workspace,
                                    size_t ws_bytes, gdn_dims_t dims, gdn_dtype_t dtype,
                                    void* stream);

/*
 * Self-test of the failure-detection path (the pages have no counterpart):
 * launches one CTA whose bounded wait on an mbarrier that nothing arrives at
 * gives up after limit_ns nanoseconds (clamped to [1 us, 1 s]) and sets the
 * device error word, as a kernel's timed-out wait does.  gdn_sync_status then
 * returns GDN_ERR_TIMEOUT and clears the word.  Nothing faults or traps; the
 * context stays usable.  Asynchronous on `stream`.
 */
gdn_status_t gdn_selftest_bounded_wait(int64_t limit_ns, void* stream);

/*
 * Number of kernel launches one gdn_chunk_prefill call with these sizes and
 * flags issues (for profiling and launch accounting; the library has no paper
 * counterpart for it): on the tensor-core path, a chunk-offsets kernel when
 * cu_seqlens is given (has_cu_seqlens != 0), then an intra and a chain kernel
 * per workspace segment (more segments for GDN_CHUNK(16) and GDN_CHUNK(32);
 * the other flag bits do not matter).  0 for T_tot == 0 or invalid dims.
 */
int32_t gdn_chunk_prefill_launches(int32_t n_seq, int64_t T_tot, int32_t has_cu_seqlens, gdn_dims_t dims,
                                   gdn_dtype_t dtype, uint32_t flags);

/*
 * Chunked gated delta rule (chunk size 64, WY/UT form) over packed sequences.
 * Defined by: cortex GatedDeltaNet commit, "Discretisation" (g, beta in f32),
 * "Block" (L2norm on q,k), "Delta rule (recurrent, per-token)" (the result is
 * that of the per-token rule; "Performance note": the chunked algorithm with
 * chunk_size=64 keeps the same surface); NxD-Inference Qwen3.6-27B PR, Summary
 * (chunked context encoding; recurrent state checkpoints).
 *
 * Per sequence and value head h (key head kh = h / (H_v/H_k)), token by token:
 *   q^ = scale * l2norm(q), k^ = l2norm(k)       (l2norm only with GDN_QK_L2NORM)
 *   g = -exp(A_log[h]) * softplus(a + dt_bias[h]), beta = sigmoid(b)
 *   S <- exp(g) S;  delta = beta (v - S^T k^);  S <- S + k^ delta^T;  o = S^T q^
 *
 *   qkv        (device) [T_tot, conv_dim]   post-conv activations, channels [q|k|v]
 *   a, b       (device) [T_tot, H_v]        gate inputs, or NULL when g/beta are given
 *   A_log, dt_bias (device) [H_v] f32       or NULL when g/beta are given
 *   g, beta    (device) [T_tot, H_v] f32    precomputed gates, or both NULL
 *   cu_seqlens (device) [n_seq + 1] int32 or NULL (one sequence)
 *   initial_state (device) [n_seq, H_v, d_k, d_v] f32 or NULL (zeros)
 *   final_state   (device) [n_seq, H_v, d_k, d_v] f32 or NULL; may alias initial_state
 *               (required on the tensor-core path with GDN_CHUNK(16) or (32))
 *   ckpt_every  0 or a positive multiple of 64; state_ckpt_out (device)
 *               [gdn_ckpt_count rows, H_v, d_k, d_v] f32: state after m*ckpt_every tokens
 *   ckpt_rows   rows allocated in state_ckpt_out; rows past it are never written;
 *               with 0 rows state_ckpt_out may be NULL
 *   scale       query scale; 0 means d_k^-1/2
 *   flags       GDN_QK_L2NORM, optionally | GDN_SOLVE_NEUMANN | GDN_CHUNK(c), or 0
 *   o          (device) [T_tot, H_v, d_v]   (dtype)
 *   workspace  (device) >= gdn_chunk_prefill_workspace_size bytes, or NULL if that is 0
 */
gdn_status_t gdn_chunk_prefill(const void* qkv, const void* a, const void* b, const float* A_log,
                               const float* dt_bias, const float* g, const float* beta,
                               const int32_t* cu_seqlens, int32_t n_seq, int64_t T_tot,
                               const float* initial_state, float* final_state, int32_t ckpt_every,
                               float* state_ckpt_out, int64_t ckpt_rows, float scale, uint32_t flags, void* o,
                               void* workspace, size_t ws_bytes, gdn_dims_t dims,
                               gdn_dtype_t dtype, void* stream);

/*
 * gdn_chunk_prefill without a workspace, for callers that cannot allocate
 * device memory.  The pages have no counterpart for this call: it exists for
 * library users whose device memory is owned by someone else -- for example a
 * plugin inside a host runtime that has partitioned all device memory up front,
 * or a serving loop that must not allocate on its hot path -- and who therefore
 * cannot provide the scratch gdn_chunk_prefill_workspace_size asks for.
 *
 * The scratch is a fixed 24 MiB array compiled into this library: every GPU
 * that loads the library holds it until the process exits.  Arguments and
 * results are those of gdn_chunk_prefill, with these differences:
 *   - only the tensor-core path: dtype GDN_BF16 and d_k = d_v = 128
 *     (GDN_ERR_UNSUPPORTED otherwise; gdn_chunk_prefill needs no workspace for
 *     the other shapes);
 *   - final_state is required (it carries the state between the call's
 *     segments); it may alias initial_state;
 *   - limits: n_seq <= 16384 and H_v * 58,368 bytes must fit in the array
 *     (H_v <= 430); calls beyond them return GDN_ERR_WORKSPACE;
 *   - the first call on a device looks up the array's device address (once per
 *     device, with that device current); make that first call before any
 *     stream capture;
 *   - all calls share the one array: calls whose kernels overlap on the GPU
 *     (other streams, other host threads) race and corrupt each other's
 *     results.  Nothing in the array has to start at zero -- every value a
 *     call reads is written earlier in the same call -- so the contents left
 *     by the previous call do no harm.
 * The arithmetic is the same as gdn_chunk_prefill's; the chunks are processed
 * in smaller segments (more kernel launches).
 */
gdn_status_t gdn_chunk_prefill_noalloc(const void* qkv, const void* a, const void* b,
                                       const float* A_log, const float* dt_bias, const float* g,
                                       const float* beta, const int32_t* cu_seqlens, int32_t n_seq,
                                       int64_t T_tot, const float* initial_state, float* final_state,
                                       int32_t ckpt_every, float* state_ckpt_out, int64_t ckpt_rows,
                                       float scale, uint32_t flags, void* o, gdn_dims_t dims,
                                       gdn_dtype_t dtype, void* stream);

/*
 * One recurrent decode step for B sequences (one token each), state in place.
 * Defined by: cortex GatedDeltaNet commit, "Delta rule (recurrent, per-token)",
 * "Discretisation", "Block" (L2norm on q,k); NxD-Inference Qwen3.6-27B PR,
 * Summary (token generation kernel).
 *   qkv    (device) [B, conv_dim]  post-conv activations of this step
 *   a, b   (device) [B, H_v] and A_log, dt_bias (device) [H_v] f32, or g, beta
 *          (device) [B, H_v] f32 (as in gdn_chunk_prefill)
 *   state  (device) [B, H_v, d_k, d_v] f32, read and rewritten in place
 *   scale, flags as in gdn_chunk_prefill
 *   o      (device) [B, H_v, d_v]
 */
gdn_status_t gdn_recurrent_decode(const void* qkv, const void* a, const void* b,
                                  const float* A_log, const float* dt_bias, const float* g,
                                  const float* beta, float* state, int32_t B, float scale,
                                  uint32_t flags, void* o, gdn_dims_t dims, gdn_dtype_t dtype,
                                  void* stream);

/*
 * One fused decode step of the layer core: conv update + SiLU (as
 * gdn_conv1d_update), gates and l2 norms, the recurrent rule (as
 * gdn_recurrent_decode) and RMSNormGated (as gdn_rmsnorm_gated) for one token
 * of each of B sequences, in one kernel (one CTA per sequence and key head;
 * for batches whose B*H_k is at most half the SM count, one CTA per sequence
 * and value head, the value heads of a key head as a thread-block cluster,
 * with the same results bit for bit).
 * Defined by the passages of those three calls; the fusion has no counterpart
 * on the pages beyond the hybrid cache they describe (NxD-Inference PR "Add
 * Qwen3.6-27B hybrid DeltaNet/GQA contrib model and vLLM serving path",
 * Summary: GDN recurrent and convolution state per cache slot).
 *   x          (device) [B, conv_dim]      dtype (pre-conv mixed_qkv of the token)
 *   conv_w     (device) [conv_dim, 4]      dtype
 *   conv_state (device) [n_slots, conv_dim, 3] dtype, updated in place
 *   z          (device) [B, H_v*d_v]       dtype
 *   a, b       (device) [B, H_v]           dtype;  A_log, dt_bias (device) [H_v] f32
 *   state      (device) [n_slots, H_v, d_k, d_v] f32, updated in place
 *   norm_w     (device) [d_v] dtype;  norm_eps > 0 (the layer uses 1e-6)
 *   slots      (device) [B] int32 cache slot of each sequence, or NULL (slot b);
 *              the slots of one call must be distinct and < n_slots (not checked
 *              on the device: an out-of-range slot is out of bounds)
 *   scale, flags as gdn_recurrent_decode;  out (device) [B, H_v*d_v] dtype
 * H_v / H_k <= 8.  Results equal the three separate calls up to the rounding
 * order of the norm's sum of squares.
 */
gdn_status_t gdn_decode_step(const void* x, const void* conv_w, void* conv_state, const void* z,
                             const void* a, const void* b, const float* A_log,
                             const float* dt_bias, float* state, const void* norm_w,
                             float norm_eps, const int32_t* slots, int32_t B, float scale,
                             uint32_t flags, void* out, gdn_dims_t dims, gdn_dtype_t dtype,
                             void* stream);

/*
 * Speculative decoding, the verification pass: K draft tokens of each of B
 * sequences through the fused decode step (conv update + SiLU, gates, l2
 * norms, recurrent rule, RMSNormGated), token after token, in one kernel.  The
 * pages name multi-token (MTP) speculative decoding as missing (NxD-Inference
 * Qwen3.6-27B PR, "Known limitations"); each token is the recurrent rule of the
 * cortex commit's "Delta rule (recurrent, per-token)".  The states are read
 * from cache slot slots[b][0] and the conv state and recurrent state after
 * draft token t are written to slot slots[b][t + 1], so accepting the first j
 * draft tokens of sequence b is continuing from slot slots[b][j] (nothing is
 * copied); slot slots[b][0] itself is only read unless it is repeated later in
 * the row.  Each value head's state is read once and written K times.
 *   x          (device) [B, K, conv_dim]  dtype (pre-conv mixed_qkv of the draft tokens)
 *   z          (device) [B, K, H_v*d_v];  a, b (device) [B, K, H_v]   dtype
 *   conv_w, A_log, dt_bias, norm_w, norm_eps, scale, flags as gdn_decode_step
 *   conv_state (device) [n_slots, conv_dim, 3] dtype;  state (device) [n_slots, H_v, d_k, d_v] f32
 *   slots      (device) [B, K + 1] int32, required: the slots of all rows distinct
 *              (slots[b][K] may equal slots[b][0]) and < n_slots (not checked on
 *              the device: an out-of-range slot is out of bounds)
 *   out        (device) [B, K, H_v*d_v] dtype
 * 1 <= K <= 16 (K = 0 or B = 0: nothing to do), H_v / H_k <= 8.  Every output
 * and every state equals that of K successive gdn_decode_step calls, bit for bit.
 * Batches whose B*H_k is at most half the SM count run, like the fused step,
 * one CTA per sequence and value head (clustered per key head), with the same
 * results.
 */
gdn_status_t gdn_decode_verify(const void* x, const void* conv_w, void* conv_state, const void* z,
                               const void* a, const void* b, const float* A_log,
                               const float* dt_bias, float* state, const void* norm_w,
                               float norm_eps, const int32_t* slots, int32_t B, int32_t K,
                               float scale, uint32_t flags, void* out, gdn_dims_t dims,
                               gdn_dtype_t dtype, void* stream);

/*
 * gdn_chunk_prefill followed by RMSNormGated of its output (as
 * gdn_rmsnorm_gated): out = RMSNormGated(o, z) with weight norm_w.  The rule
 * writes o into `out` and the norm kernel normalises it in place, so no o
 * buffer is needed.  Defined by the passages of the two calls (cortex
 * GatedDeltaNet commit, "Output": RMSNormGated(core_attn_out, z)).
 *   arguments before z: as gdn_chunk_prefill (workspace:
 *               gdn_chunk_prefill_workspace_size bytes)
 *   z          (device) [T_tot, H_v*d_v] dtype;  norm_w (device) [d_v] dtype
 *   norm_eps   > 0 (the layer uses 1e-6)
 *   out        (device) [T_tot, H_v*d_v] dtype
 * Results equal gdn_chunk_prefill then gdn_rmsnorm_gated, bit for bit.
 * Kernel launches: gdn_chunk_prefill_launches + 1.
 */
gdn_status_t gdn_chunk_prefill_norm(const void* qkv, const void* a, const void* b, const float* A_log,
                                    const float* dt_bias, const float* g, const float* beta,
                                    const int32_t* cu_seqlens, int32_t n_seq, int64_t T_tot,
                                    const float* initial_state, float* final_state, int32_t ckpt_every,
                                    float* state_ckpt_out, int64_t ckpt_rows, float scale, uint32_t flags,
                                    const void* z, const void* norm_w, float norm_eps, void* out,
                                    void* workspace, size_t ws_bytes, gdn_dims_t dims, gdn_dtype_t dtype,
                                    void* stream);

/*
 * The layer core on device buffers in one call: conv1d + SiLU (as
 * gdn_conv1d_fwd, with its state and checkpoint outputs), the chunked rule (as
 * gdn_chunk_prefill) and RMSNormGated (as gdn_rmsnorm_gated), for packed
 * sequences.  Defined by the passages of those three calls: cortex
 * GatedDeltaNet commit, "Block" and "Output" (the order conv -> rule ->
 * RMSNormGated(core_attn_out, z)); the fusion has no counterpart on the pages
 * beyond the chunked kernel of the NxD-Inference Qwen3.6-27B PR, Summary.
 * bf16 with d_k = 128 (the tensor-core path): the conv runs inside the chunk
 * kernels -- each chunk's tiles of x and their 3-token halo (or the
 * sequence's conv state) are convolved in shared memory, so the conv output
 * never goes to device memory -- and the same kernels write the conv state and
 * checkpoints, unless conv_state_out is conv_state_in (then a pass after them
 * does).  Otherwise it is gdn_conv1d_fwd (into the workspace) followed by
 * gdn_chunk_prefill_norm.
 *   x          (device) [T_tot, conv_dim]   raw (pre-conv) mixed_qkv
 *   z          (device) [T_tot, H_v*d_v];  a, b (device) [T_tot, H_v]    dtype
 *   conv_w     (device) [conv_dim, 4];  norm_w (device) [d_v]            dtype
 *   A_log, dt_bias (device) [H_v] f32;  norm_eps > 0 (the layer uses 1e-6)
 *   cu_seqlens, n_seq, T_tot, initial_state, final_state  as gdn_chunk_prefill
 *   conv_state_in, conv_state_out   as gdn_conv1d_fwd
 *   ckpt_every  0 or a positive multiple of 64, for both checkpoint outputs:
 *               state_ckpt_out [rows, H_v, d_k, d_v] f32 (as gdn_chunk_prefill) and
 *               conv_ckpt_out [rows, conv_dim, 3] dtype (as gdn_conv1d_fwd);
 *               ckpt_rows rows allocated in each (with 0, both may be NULL)
 *   scale, flags  as gdn_chunk_prefill (GDN_QK_L2NORM, optionally | GDN_SOLVE_NEUMANN)
 *   out        (device) [T_tot, H_v*d_v]   dtype
 *   workspace  (device) >= gdn_layer_prefill_workspace_size bytes, 16-byte
 *              aligned (tensor-core path: the chunk intermediates and the conv'd
 *              q tiles the state chain reads; otherwise the conv output)
 * Results equal those of the three separate calls bit for bit.  Kernel
 * launches: gdn_layer_prefill_launches (with conv_state_out not conv_state_in;
 * one more in place on the tensor-core path).
 */
size_t gdn_layer_prefill_workspace_size(int32_t n_seq, int64_t T_tot, gdn_dims_t dims, gdn_dtype_t dtype);
int32_t gdn_layer_prefill_launches(int32_t n_seq, int64_t T_tot, int32_t has_cu_seqlens, gdn_dims_t dims,
                                   gdn_dtype_t dtype, uint32_t flags);
gdn_status_t gdn_layer_prefill(const void* x, const void* z, const void* a, const void* b, const void* conv_w,
                               const float* A_log, const float* dt_bias, const void* norm_w, float norm_eps,
                               const int32_t* cu_seqlens, int32_t n_seq, int64_t T_tot,
                               const float* initial_state, float* final_state, const void* conv_state_in,
                               void* conv_state_out, int32_t ckpt_every, float* state_ckpt_out,
                               void* conv_ckpt_out, int64_t ckpt_rows, float scale, uint32_t flags, void* out,
                               void* workspace, size_t ws_bytes, gdn_dims_t dims, gdn_dtype_t dtype,
                               void* stream);

/*
 * RMSNormGated over each value head.
 * Defined by: cortex GatedDeltaNet commit, "Output": RMSNormGated(core_attn_out, z).
 *   out[t, h*d_v + j] = w[j] * o[t,h,j] / sqrt(mean_j o[t,h,j]^2 + eps) * silu(z[t, h*d_v + j])
 *   o   (device) [T, H_v, d_v];  z, out (device) [T, H_v*d_v];  w (device) [d_v]
 *   eps > 0 (the layer uses 1e-6).  out may alias o.
 */
gdn_status_t gdn_rmsnorm_gated(const void* o, const void* z, const void* w, float eps, int64_t T,
                               void* out, gdn_dims_t dims, gdn_dtype_t dtype, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GDN_H_ */
