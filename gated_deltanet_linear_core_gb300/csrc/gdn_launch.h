// Host-side launchers of the GDN kernels (one translation unit per kernel
// family).  Arguments are already validated by the C ABI layer in gdn_api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

#include <cudaTypedefs.h>

namespace gdn {

struct ConvArgs {
    const void* x;
    const void* w;
    const int32_t* cu;
    int n_seq;
    int64_t T;
    int C;  // conv_dim
    const void* state_in;
    void* state_out;
    int ckpt_every;
    void* ckpt;
    int64_t ckpt_rows;
    int silu;
    void* y;
    int fused_state;  // set by launch_conv1d_fwd: the tile kernel writes the state and checkpoints
};
cudaError_t launch_conv1d_fwd(const ConvArgs& a, gdn_dtype_t dt, cudaStream_t s);
// Only the conv state after each sequence and the conv checkpoints (no y): the
// state pass of launch_conv1d_fwd, for callers that compute y elsewhere.
cudaError_t launch_conv1d_state(const ConvArgs& a, gdn_dtype_t dt, cudaStream_t s);
cudaError_t launch_conv1d_update(const void* x, const void* w, void* state, int B, int C,
                                 int silu, void* y, gdn_dtype_t dt, cudaStream_t s);

struct DeltaArgs {
    const void* qkv;  // [T, conv_dim]
    const void* a;
    const void* b;
    const float* A_log;
    const float* dt_bias;
    const float* g;
    const float* beta;
    const int32_t* cu;
    int n_seq;
    int64_t T;
    int H_k, H_v, D;
    const float* S0;
    float* S_final;
    int ckpt_every;
    float* ckpt;
    int64_t ckpt_rows;
    float scale;
    int l2norm;
    void* o;  // [T, H_v, D]
    int neumann;  // chunk inverse by the Neumann-style product (tensor-core path)
    int chunk;    // tokens per chunk: 16, 32 or 64 (0: 64)
    // Conv1d + SiLU inside the chunk kernels (tensor-core path): with conv_w
    // set, qkv is the raw conv input x and the kernels compute y themselves
    // from x, these taps ([conv_dim][4]) and the sequences' conv states before
    // their first tokens ([n_seq][conv_dim][3], null: zeros).
    const void* conv_w;
    const void* conv_state0;
    // ... and, when set, the kernels also write the conv state after each
    // sequence ([n_seq][conv_dim][3]; never the conv_state0 array) and the
    // conv checkpoints ([ckpt_rows][conv_dim][3], every ckpt_every tokens)
    void* conv_state_out;
    void* conv_ckpt;
};
// Chunked prefill on CUDA cores (f32 arithmetic; any supported D and dtype).
cudaError_t launch_chunk_ffma(const DeltaArgs& a, gdn_dtype_t dt, cudaStream_t s);
// Recurrent decode: T = B tokens, sequence i = token i, state in place (S0 == S_final).
cudaError_t launch_recurrent_decode(const DeltaArgs& a, gdn_dtype_t dt, cudaStream_t s);

// Fused decode step: conv update, gates, recurrence and RMSNormGated for one
// token per sequence; conv state and state in place at slots[b] (or b).
struct DecodeStepArgs {
    const void* x;         // [B, conv_dim]
    const void* conv_w;    // [conv_dim, 4]
    void* conv_state;      // [slots, conv_dim, 3]
    const void *z, *a, *b; // [B, H_v*D], [B, H_v], [B, H_v]
    const float *A_log, *dt_bias;
    float* state;          // [slots, H_v, D, D]
    const void* norm_w;    // [D]
    const int32_t* slots;  // [B] or null
    int B, H_k, H_v, D;
    float scale, eps;
    int l2norm;
    void* out;             // [B, H_v*D]
};
cudaError_t launch_decode_step(const DecodeStepArgs& a, gdn_dtype_t dt, cudaStream_t s);

// K draft tokens per sequence from the states in slot slots[b][0]; the conv
// state and the recurrent state after draft token t go to slot slots[b][t + 1].
struct DecodeVerifyArgs {
    const void* x;         // [B, K, conv_dim]
    const void* conv_w;    // [conv_dim, 4]
    void* conv_state;      // [slots, conv_dim, 3]
    const void *z, *a, *b; // [B, K, H_v*D], [B, K, H_v], [B, K, H_v]
    const float *A_log, *dt_bias;
    float* state;          // [slots, H_v, D, D]
    const void* norm_w;    // [D]
    const int32_t* slots;  // [B, K + 1]
    int B, K, H_k, H_v, D;
    float scale, eps;
    int l2norm;
    void* out;             // [B, K, H_v*D]
};
constexpr int kVerifyMaxK = 16;
cudaError_t launch_decode_verify(const DecodeVerifyArgs& a, gdn_dtype_t dt, cudaStream_t s);

// cuTensorMapEncodeTiled from the driver (nullptr if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensormap_encoder();
// Unique id of the calling thread's current CUDA context, 0 if there is none
// (or the driver cannot tell).  Caches of device objects key on it, so that a
// context destroyed and created again (a device reset) never reuses objects of
// the old one.
unsigned long long current_context_id();

// Chunked prefill on tcgen05 tensor cores (bf16 operands, f32 state, D = 128)
// in two kernels: the state-independent work of every chunk in parallel (into
// `workspace`), then the sequential state recurrence.
size_t chunk_split_workspace_bytes(int n_seq, int64_t T, int H_v);
// ... when the conv is computed inside the kernels (DeltaArgs::conv_w): the
// same plus the conv'd q tiles of each segment's chunks and key heads.
size_t chunk_split_conv_workspace_bytes(int n_seq, int64_t T, int H_k, int H_v);
cudaError_t launch_chunk_split(const DeltaArgs& a, void* workspace, size_t ws_bytes,
                               cudaStream_t s);
// The same with the chunk offsets and intra kernels on s_pre and the chain on
// s_chain after ev_pre (recorded on s_pre, waited on s_chain); with more than
// one workspace segment everything runs on s_chain after ev_pre.
cudaError_t launch_chunk_split_two(const DeltaArgs& a, void* workspace, size_t ws_bytes, cudaStream_t s_pre,
                                   cudaStream_t s_chain, cudaEvent_t ev_pre);
// Kernel launches launch_chunk_split issues: chunk offsets, then intra + chain per segment
// (chunk: tokens per chunk, 16, 32 or 64).
int chunk_split_launches(int n_seq, int64_t T, int H_v, bool has_cu, int chunk);

// The same chunked prefill with its scratch in a fixed device array of the
// library (gdn_chunk_prefill_noalloc): no allocation; final_state required.
bool chunk_split_static_fits(int n_seq, int H_v);
cudaError_t launch_chunk_split_static(const DeltaArgs& a, cudaStream_t s);

// Reads (synchronising `s`) and clears the library's device error word.
cudaError_t read_and_clear_device_error(cudaStream_t s, int* flags);
// One CTA whose bounded wait runs out after limit_ns and sets the error word.
cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, cudaStream_t s);
// The same for the conv kernels' own error word.
cudaError_t read_and_clear_conv_error(cudaStream_t s, int* flags);

cudaError_t launch_rmsnorm_gated(const void* o, const void* z, const void* w, float eps, int64_t T,
                                 int H, int D, void* out, gdn_dtype_t dt, cudaStream_t s);

// The layer core for one sequence streamed from page-locked host memory
// (gdn_layer_prefill_host).
struct HostLayerArgs {
    const void *h_qkv, *h_z, *h_a, *h_b;  // host, page-locked
    const void* conv_w;
    const float *A_log, *dt_bias;
    const void* norm_w;
    int64_t T;
    int H_k, H_v, D;
    const float* initial_state;
    float* final_state;
    const void* conv_state_in;
    void* conv_state_out;
    float scale, eps;
    int l2norm;
    void* h_out;  // host, page-locked
};
size_t layer_prefill_host_workspace_bytes(int64_t T, int H_k, int H_v, int D, int es, bool tensor_core);
int64_t layer_prefill_host_piece(int64_t T, int H_k, int H_v, int D, int es, bool tensor_core);
int64_t layer_prefill_host_pieces(int64_t T, int H_k, int H_v, int D, int es, bool tensor_core);
cudaError_t launch_layer_prefill_host(const HostLayerArgs& h, gdn_dtype_t dt, void* workspace, cudaStream_t s);

}  // namespace gdn
