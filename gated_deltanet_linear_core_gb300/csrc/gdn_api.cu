// C ABI of the GDN layer core: argument validation and dispatch.
//
// Every entry point validates all of its arguments on the host before it
// launches anything; no device memory is read here (except in
// gdn_check_cu_seqlens, which says so).  No exception crosses the ABI.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <vector>

#include "gdn.h"
#include "gdn_launch.h"

namespace {

thread_local int g_last_cuda_error = 0;

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_n(const void* p, size_t n) {
    return p == nullptr || (reinterpret_cast<uintptr_t>(p) % n) == 0;
}
size_t elem_size(gdn_dtype_t dt) { return dt == GDN_BF16 ? 2 : 4; }

gdn_status_t check_dims(const gdn_dims_t& d, gdn_dtype_t dt) {
    if (dt != GDN_F32 && dt != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (d.H_k <= 0 || d.H_v <= 0 || d.d_k <= 0 || d.d_v <= 0 || d.conv_k <= 0)
        return GDN_ERR_INVALID_ARG;
    if (d.H_v % d.H_k != 0) return GDN_ERR_INVALID_ARG;
    if (d.conv_k != 4) return GDN_ERR_UNSUPPORTED;
    if (d.d_k != d.d_v) return GDN_ERR_UNSUPPORTED;
    if (d.d_k != 16 && d.d_k != 128) return GDN_ERR_UNSUPPORTED;
    if ((int64_t)d.H_v * d.d_v > (1 << 24) || (int64_t)d.H_k * d.d_k > (1 << 24))
        return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

int64_t conv_dim_of(const gdn_dims_t& d) { return 2LL * d.H_k * d.d_k + (int64_t)d.H_v * d.d_v; }

gdn_status_t cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return GDN_OK;
    g_last_cuda_error = (int)e;
    return GDN_ERR_CUDA;
}

gdn_status_t check_ckpt(int32_t every, const void* ckpt, int64_t rows) {
    if (every < 0) return GDN_ERR_INVALID_ARG;
    if (every > 0) {
        if (every % 64 != 0) return GDN_ERR_INVALID_ARG;
        // a buffer is needed only when rows are allocated (a call whose sequences are
        // all shorter than the cadence has none)
        if (rows < 0 || (ckpt == nullptr && rows > 0)) return GDN_ERR_INVALID_ARG;
    }
    return GDN_OK;
}

gdn_status_t check_seqs(const int32_t* cu, int32_t n_seq, int64_t T) {
    if (T < 0 || T > (int64_t)INT32_MAX) return GDN_ERR_INVALID_ARG;
    if (cu == nullptr) return n_seq == 1 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (n_seq < 1 || n_seq > (1 << 24)) return GDN_ERR_INVALID_ARG;
    if (!aligned_n(cu, 4)) return GDN_ERR_ALIGN;
    return GDN_OK;
}

// gates: either (a, b, A_log, dt_bias) or (g, beta)
gdn_status_t check_gates(const void* a, const void* b, const float* A_log, const float* dt_bias,
                         const float* g, const float* beta, gdn_dtype_t dt) {
    const bool raw = a && b && A_log && dt_bias;
    const bool pre = g && beta;
    if (!raw && !pre) return GDN_ERR_INVALID_ARG;
    if (!aligned_n(a, elem_size(dt)) || !aligned_n(b, elem_size(dt)) || !aligned_n(A_log, 4) ||
        !aligned_n(dt_bias, 4) || !aligned_n(g, 4) || !aligned_n(beta, 4))
        return GDN_ERR_ALIGN;
    return GDN_OK;
}

}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status_t s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument";
        case GDN_ERR_ALIGN: return "device pointer not 16-byte aligned";
        case GDN_ERR_UNSUPPORTED: return "unsupported dimensions";
        case GDN_ERR_WORKSPACE: return "workspace missing or too small";
        case GDN_ERR_CUDA: return "CUDA error";
        case GDN_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

int gdn_last_cuda_error(void) { return g_last_cuda_error; }

int gdn_version(void) { return (1 << 16) | 0; }

int64_t gdn_ckpt_count(const int32_t* cu, int32_t n_seq, int32_t every) {
    if (cu == nullptr || n_seq < 1 || every < 0) return -1;
    if (every == 0) return 0;
    int64_t r = 0;
    for (int32_t i = 0; i < n_seq; ++i) {
        if (cu[i + 1] < cu[i]) return -1;
        r += (int64_t)(cu[i + 1] - cu[i]) / every;
    }
    return r;
}

gdn_status_t gdn_check_cu_seqlens(const int32_t* cu, int32_t n_seq, int64_t T, void* stream) {
    if (cu == nullptr || n_seq < 1 || T < 0) return GDN_ERR_INVALID_ARG;
    std::vector<int32_t> h((size_t)n_seq + 1);
    cudaError_t e = cudaMemcpyAsync(h.data(), cu, sizeof(int32_t) * h.size(),
                                    cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_status(e);
    if (h[0] != 0 || h[(size_t)n_seq] != T) return GDN_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_seq; ++i)
        if (h[(size_t)i + 1] < h[(size_t)i]) return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

gdn_status_t gdn_sync_status(void* stream) {
    int flags = 0, cflags = 0;
    cudaError_t e = gdn::read_and_clear_device_error((cudaStream_t)stream, &flags);
    if (e == cudaSuccess) e = gdn::read_and_clear_conv_error((cudaStream_t)stream, &cflags);
    if (e != cudaSuccess) return cuda_status(e);
    return ((flags | cflags) & 1) ? GDN_ERR_TIMEOUT : GDN_OK;
}

size_t gdn_layer_prefill_host_workspace_size(int64_t T, gdn_dims_t dims, gdn_dtype_t dtype) {
    if (check_dims(dims, dtype) != GDN_OK || T <= 0 || T > (int64_t)INT32_MAX) return 0;
    return gdn::layer_prefill_host_workspace_bytes(T, dims.H_k, dims.H_v, dims.d_k, (int)elem_size(dtype),
                                                   dtype == GDN_BF16 && dims.d_k == 128);
}

int64_t gdn_layer_prefill_host_piece(int64_t T, gdn_dims_t dims, gdn_dtype_t dtype) {
    if (check_dims(dims, dtype) != GDN_OK || T <= 0 || T > (int64_t)INT32_MAX) return 0;
    return gdn::layer_prefill_host_piece(T, dims.H_k, dims.H_v, dims.d_k, (int)elem_size(dtype),
                                         dtype == GDN_BF16 && dims.d_k == 128);
}

int64_t gdn_layer_prefill_host_pieces(int64_t T, gdn_dims_t dims, gdn_dtype_t dtype) {
    if (check_dims(dims, dtype) != GDN_OK || T <= 0 || T > (int64_t)INT32_MAX) return 0;
    return gdn::layer_prefill_host_pieces(T, dims.H_k, dims.H_v, dims.d_k, (int)elem_size(dtype),
                                          dtype == GDN_BF16 && dims.d_k == 128);
}

namespace {
bool page_locked(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost;
}
}  // namespace

gdn_status_t gdn_layer_prefill_host(const void* h_qkv, const void* h_z, const void* h_a,
                                    const void* h_b, const void* conv_w, const float* A_log,
                                    const float* dt_bias, const void* norm_w, int64_t T,
                                    const float* initial_state, float* final_state,
                                    const void* conv_state_in, void* conv_state_out, float scale,
                                    uint32_t flags, float norm_eps, void* h_out, void* workspace,
                                    size_t ws_bytes, gdn_dims_t dims, gdn_dtype_t dtype,
                                    void* stream) {
    gdn_status_t st = check_dims(dims, dtype);
    if (st != GDN_OK) return st;
    if (T < 0 || T > (int64_t)INT32_MAX) return GDN_ERR_INVALID_ARG;
    if (flags & ~GDN_QK_L2NORM) return GDN_ERR_INVALID_ARG;
    if (!isfinite(scale) || !isfinite(norm_eps) || norm_eps <= 0.f) return GDN_ERR_INVALID_ARG;
    if (conv_w == nullptr || A_log == nullptr || dt_bias == nullptr || norm_w == nullptr ||
        final_state == nullptr || conv_state_out == nullptr)
        return GDN_ERR_INVALID_ARG;
    if (T > 0 && (h_qkv == nullptr || h_z == nullptr || h_a == nullptr || h_b == nullptr || h_out == nullptr))
        return GDN_ERR_INVALID_ARG;
    if (!aligned16(conv_w) || !aligned16(norm_w) || !aligned_n(A_log, 4) || !aligned_n(dt_bias, 4) ||
        !aligned16(initial_state) || !aligned16(final_state) || !aligned16(conv_state_in) ||
        !aligned16(conv_state_out) || !aligned16(workspace))
        return GDN_ERR_ALIGN;
    if (T > 0 && !(page_locked(h_qkv) && page_locked(h_z) && page_locked(h_a) && page_locked(h_b) &&
                   page_locked(h_out)))
        return GDN_ERR_INVALID_ARG;
    const size_t need = gdn_layer_prefill_host_workspace_size(T, dims, dtype);
    if (need > 0 && (workspace == nullptr || ws_bytes < need)) return GDN_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) {
        // no tokens: the states pass through (conv state pass, then the empty prefill)
        gdn::ConvArgs c;
        memset(&c, 0, sizeof(c));
        c.w = conv_w; c.n_seq = 1; c.C = (int)conv_dim_of(dims);
        c.state_in = conv_state_in; c.state_out = conv_state_out; c.silu = 1;
        cudaError_t e = gdn::launch_conv1d_fwd(c, dtype, s);
        if (e != cudaSuccess) return cuda_status(e);
        gdn::DeltaArgs d;
        memset(&d, 0, sizeof(d));
        d.A_log = A_log; d.dt_bias = dt_bias; d.n_seq = 1;
        d.H_k = dims.H_k; d.H_v = dims.H_v; d.D = dims.d_k;
        d.S0 = initial_state; d.S_final = final_state; d.scale = 1.f;
        return cuda_status(gdn::launch_chunk_ffma(d, dtype, s));
    }
    gdn::HostLayerArgs h;
    h.h_qkv = h_qkv; h.h_z = h_z; h.h_a = h_a; h.h_b = h_b;
    h.conv_w = conv_w; h.A_log = A_log; h.dt_bias = dt_bias; h.norm_w = norm_w;
    h.T = T; h.H_k = dims.H_k; h.H_v = dims.H_v; h.D = dims.d_k;
    h.initial_state = initial_state; h.final_state = final_state;
    h.conv_state_in = conv_state_in; h.conv_state_out = conv_state_out;
    h.scale = scale == 0.f ? 1.0f / sqrtf((float)dims.d_k) : scale;
    h.eps = norm_eps;
    h.l2norm = (flags & GDN_QK_L2NORM) != 0;
    h.h_out = h_out;
    return cuda_status(gdn::launch_layer_prefill_host(h, dtype, workspace, s));
}

gdn_status_t gdn_decode_step(const void* x, const void* conv_w, void* conv_state, const void* z,
                             const void* a, const void* b, const float* A_log,
                             const float* dt_bias, float* state, const void* norm_w,
                             float norm_eps, const int32_t* slots, int32_t B, float scale,
                             uint32_t flags, void* out, gdn_dims_t dims, gdn_dtype_t dtype,
                             void* stream) {
    gdn_status_t st = check_dims(dims, dtype);
    if (st != GDN_OK) return st;
    if (B < 0 || (int64_t)B * dims.H_v > INT32_MAX) return GDN_ERR_INVALID_ARG;
    if (dims.H_v / dims.H_k > 8) return GDN_ERR_UNSUPPORTED;
    if (flags & ~GDN_QK_L2NORM) return GDN_ERR_INVALID_ARG;
    if (!isfinite(scale) || !isfinite(norm_eps) || norm_eps <= 0.f) return GDN_ERR_INVALID_ARG;
    if (B > 0 && (x == nullptr || conv_w == nullptr || conv_state == nullptr || z == nullptr ||
                  a == nullptr || b == nullptr || A_log == nullptr || dt_bias == nullptr ||
                  state == nullptr || norm_w == nullptr || out == nullptr))
        return GDN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(conv_w) || !aligned16(conv_state) || !aligned16(z) ||
        !aligned_n(a, elem_size(dtype)) || !aligned_n(b, elem_size(dtype)) || !aligned_n(A_log, 4) ||
        !aligned_n(dt_bias, 4) || !aligned16(state) || !aligned16(norm_w) || !aligned_n(slots, 4) ||
        !aligned16(out))
        return GDN_ERR_ALIGN;
    gdn::DecodeStepArgs d;
    memset(&d, 0, sizeof(d));
    d.x = x; d.conv_w = conv_w; d.conv_state = conv_state; d.z = z; d.a = a; d.b = b;
    d.A_log = A_log; d.dt_bias = dt_bias; d.state = state; d.norm_w = norm_w; d.slots = slots;
    d.B = B; d.H_k = dims.H_k; d.H_v = dims.H_v; d.D = dims.d_k;
    d.scale = scale == 0.f ? 1.0f / sqrtf((float)dims.d_k) : scale;
    d.eps = norm_eps;
    d.l2norm = (flags & GDN_QK_L2NORM) != 0;
    d.out = out;
    return cuda_status(gdn::launch_decode_step(d, dtype, (cudaStream_t)stream));
}

gdn_status_t gdn_decode_verify(const void* x, const void* conv_w, void* conv_state, const void* z,
                               const void* a, const void* b, const float* A_log,
                               const float* dt_bias, float* state, const void* norm_w,
                               float norm_eps, const int32_t* slots, int32_t B, int32_t K,
                               float scale, uint32_t flags, void* out, gdn_dims_t dims,
                               gdn_dtype_t dtype, void* stream) {
    gdn_status_t st = check_dims(dims, dtype);
    if (st != GDN_OK) return st;
    if (B < 0 || K < 0 || K > gdn::kVerifyMaxK || (int64_t)B * K * dims.H_v > INT32_MAX)
        return GDN_ERR_INVALID_ARG;
    if (dims.H_v / dims.H_k > 8) return GDN_ERR_UNSUPPORTED;
    if (flags & ~GDN_QK_L2NORM) return GDN_ERR_INVALID_ARG;
    if (!isfinite(scale) || !isfinite(norm_eps) || norm_eps <= 0.f) return GDN_ERR_INVALID_ARG;
    if (B > 0 && K > 0 &&
        (x == nullptr || conv_w == nullptr || conv_state == nullptr || z == nullptr || a == nullptr ||
         b == nullptr || A_log == nullptr || dt_bias == nullptr || state == nullptr ||
         norm_w == nullptr || slots == nullptr || out == nullptr))
        return GDN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(conv_w) || !aligned16(conv_state) || !aligned16(z) ||
        !aligned_n(a, elem_size(dtype)) || !aligned_n(b, elem_size(dtype)) || !aligned_n(A_log, 4) ||
        !aligned_n(dt_bias, 4) || !aligned16(state) || !aligned16(norm_w) || !aligned_n(slots, 4) ||
        !aligned16(out))
        return GDN_ERR_ALIGN;
    gdn::DecodeVerifyArgs d;
    memset(&d, 0, sizeof(d));
    d.x = x; d.conv_w = conv_w; d.conv_state = conv_state; d.z = z; d.a = a; d.b = b;
    d.A_log = A_log; d.dt_bias = dt_bias; d.state = state; d.norm_w = norm_w; d.slots = slots;
    d.B = B; d.K = K; d.H_k = dims.H_k; d.H_v = dims.H_v; d.D = dims.d_k;
    d.scale = scale == 0.f ? 1.0f / sqrtf((float)dims.d_k) : scale;
    d.eps = norm_eps;
    d.l2norm = (flags & GDN_QK_L2NORM) != 0;
    d.out = out;
    return cuda_status(gdn::launch_decode_verify(d, dtype, (cudaStream_t)stream));
}

gdn_status_t gdn_selftest_bounded_wait(int64_t limit_ns, void* stream) {
    if (limit_ns < 1000) limit_ns = 1000;
    if (limit_ns > 1000000000) limit_ns = 1000000000;
    return cuda_status(gdn::launch_bounded_wait_selftest((uint64_t)limit_ns, (cudaStream_t)stream));
}

gdn_status_t gdn_conv1d_fwd(const void* x, const void* w, const int32_t* cu_seqlens, int32_t n_seq,
                            int64_t T_tot, const void* conv_state_in, void* conv_state_out,
                            int32_t ckpt_every, void* conv_ckpt_out, int64_t ckpt_rows,
                            int32_t apply_silu, void* y, gdn_dims_t dims, gdn_dtype_t dtype,
                            void* stream) {
    gdn_status_t st = check_dims(dims, dtype);
    if (st != GDN_OK) return st;
    if ((st = check_seqs(cu_seqlens, n_seq, T_tot)) != GDN_OK) return st;
    if ((st = check_ckpt(ckpt_every, conv_ckpt_out, ckpt_rows)) != GDN_OK) return st;
    if (w == nullptr || (T_tot > 0 && (x == nullptr || y == nullptr))) return GDN_ERR_INVALID_ARG;
    if (x != nullptr && x == y) return GDN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || !aligned16(conv_state_in) ||
        !aligned16(conv_state_out) || !aligned16(conv_ckpt_out))
        return GDN_ERR_ALIGN;
    gdn::ConvArgs a;
    a.x = x; a.w = w; a.cu = cu_seqlens; a.n_seq = n_seq; a.T = T_tot;
    a.C = (int)conv_dim_of(dims);
    a.state_in = conv_state_in; a.state_out = conv_state_out;
    a.ckpt_every = ckpt_every; a.ckpt = ckpt_every > 0 ? conv_ckpt_out : nullptr;
    a.ckpt_rows = ckpt_rows; a.silu = apply_silu != 0; a.y = y;
    return cuda_status(gdn::launch_conv1d_fwd(a, dtype, (cudaStream_t)stream));
}

gdn_status_t gdn_conv1d_update(const void* x, const void* w, void* conv_state, int32_t B,
                               int32_t apply_silu, void* y, gdn_dims_t dims, gdn_dtype_t dtype,
                               void* stream) {
    gdn_status_t st = check_dims(dims, dtype);
    if (st != GDN_OK) return st;
    if (B < 0 || B > INT32_MAX / 2) return GDN_ERR_INVALID_ARG;
    if (B > 0 && (x == nullptr || w == nullptr || conv_state == nullptr || y == nullptr))
        return GDN_ERR_INVALID_ARG;
    if (x != nullptr && x == y) return GDN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(conv_state) || !aligned16(y))
        return GDN_ERR_ALIGN;
    return cuda_status(gdn::launch_conv1d_update(x, w, conv_state, B, (int)conv_dim_of(dims),
                                                 apply_silu != 0, y, dtype, (cudaStream_t)stream));
}

size_t gdn_chunk_prefill_workspace_size(int32_t n_seq, int64_t T_tot, gdn_dims_t dims,
                                        gdn_dtype_t dtype) {
    if (check_dims(dims, dtype) != GDN_OK || n_seq < 1 || T_tot <= 0) return 0;
    if (dtype != GDN_BF16 || dims.d_k != 128) return 0;  // the CUDA-core path needs none
    return gdn::chunk_split_workspace_bytes(n_seq, T_tot, dims.H_v);
}

int32_t gdn_chunk_prefill_launches(int32_t n_seq, int64_t T_tot, int32_t has_cu_seqlens, gdn_dims_t dims,
                                   gdn_dtype_t dtype, uint32_t flags) {
    if (check_dims(dims, dtype) != GDN_OK || n_seq < 1 || T_tot <= 0) return 0;
    if (dtype != GDN_BF16 || dims.d_k != 128) return 1;  // the CUDA-core path: one kernel
    return gdn::chunk_split_launches(n_seq, T_tot, dims.H_v, has_cu_seqlens != 0, (int)((flags >> 8) & 0xffu));
}

namespace {
// gdn_chunk_prefill, and with norm_out set (== o) the same followed by
// RMSNormGated(o, norm_z) in place over norm_out.
gdn_status_t chunk_prefill_impl(const void* qkv, const void* a, const void* b, const float* A_log,
                                const float* dt_bias, const float* g, const float* beta,
                                const int32_t* cu_seqlens, int32_t n_seq, int64_t T_tot,
                                const float* initial_state, float* final_state, int32_t ckpt_every,
                                float* state_ckpt_out, int64_t ckpt_rows, float scale, uint32_t flags, void* o,
                                void* workspace, size_t ws_bytes, gdn_dims_t dims, gdn_dtype_t dtype,
                                void* stream, const void* norm_z, const void* norm_w, float norm_eps,
                                void* norm_out) {
    gdn_status_t st = check_dims(dims, dtype);
    if (st != GDN_OK) return st;
    if ((st = check_seqs(cu_seqlens, n_seq, T_tot)) != GDN_OK) return st;
    if ((st = check_ckpt(ckpt_every, state_ckpt_out, ckpt_rows)) != GDN_OK) return st;
    if (T_tot > 0 && (st = check_gates(a, b, A_log, dt_bias, g, beta, dtype)) != GDN_OK) return st;
    if (flags & ~(GDN_QK_L2NORM | GDN_SOLVE_NEUMANN | GDN_CHUNK(0xff))) return GDN_ERR_INVALID_ARG;
    const int chunk = ((flags >> 8) & 0xffu) == 0 ? 64 : (int)((flags >> 8) & 0xffu);
    if (chunk != 16 && chunk != 32 && chunk != 64) return GDN_ERR_INVALID_ARG;
    const bool tensor_core = dtype == GDN_BF16 && dims.d_k == 128;
    if ((flags & GDN_SOLVE_NEUMANN) && !tensor_core) return GDN_ERR_UNSUPPORTED;
    // shorter chunks on the tensor-core path run in more workspace segments,
    // between which the state crosses through final_state
    if (chunk != 64 && tensor_core && T_tot > 0 && final_state == nullptr) return GDN_ERR_UNSUPPORTED;
    if (!isfinite(scale)) return GDN_ERR_INVALID_ARG;
    if (T_tot > 0 && (qkv == nullptr || o == nullptr)) return GDN_ERR_INVALID_ARG;
    if (!aligned16(qkv) || !aligned16(o) || !aligned16(initial_state) || !aligned16(final_state) ||
        !aligned16(state_ckpt_out))
        return GDN_ERR_ALIGN;
    const size_t need = gdn_chunk_prefill_workspace_size(n_seq, T_tot, dims, dtype);
    if (need > 0 && (workspace == nullptr || ws_bytes < need)) return GDN_ERR_WORKSPACE;
    if ((int64_t)n_seq * dims.H_v * 8 > INT32_MAX) return GDN_ERR_UNSUPPORTED;

    gdn::DeltaArgs d;
    memset(&d, 0, sizeof(d));
    d.qkv = qkv; d.a = a; d.b = b; d.A_log = A_log; d.dt_bias = dt_bias;
    const bool pre = g && beta;
    d.g = pre ? g : nullptr; d.beta = pre ? beta : nullptr;
    d.cu = cu_seqlens; d.n_seq = n_seq; d.T = T_tot;
    d.H_k = dims.H_k; d.H_v = dims.H_v; d.D = dims.d_k;
    d.S0 = initial_state; d.S_final = final_state;
    d.ckpt_every = ckpt_every; d.ckpt = ckpt_every > 0 ? state_ckpt_out : nullptr;
    d.ckpt_rows = ckpt_rows;
    d.scale = scale == 0.f ? 1.0f / sqrtf((float)dims.d_k) : scale;
    d.l2norm = (flags & GDN_QK_L2NORM) != 0;
    d.neumann = (flags & GDN_SOLVE_NEUMANN) != 0;
    d.chunk = chunk;
    d.o = o;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = need > 0 ? gdn::launch_chunk_split(d, workspace, ws_bytes, s) : gdn::launch_chunk_ffma(d, dtype, s);
    if (e == cudaSuccess && norm_out != nullptr)
        e = gdn::launch_rmsnorm_gated(o, norm_z, norm_w, norm_eps, T_tot, dims.H_v, dims.d_v, norm_out, dtype, s);
    return cuda_status(e);
}
}  // namespace

gdn_status_t gdn_chunk_prefill(const void* qkv, const void* a, const void* b, const float* A_log,
                               const float* dt_bias, const float* g, const float* beta,
                               const int32_t* cu_seqlens, int32_t n_seq, int64_t T_tot,
                               const float* initial_state, float* final_state, int32_t ckpt_every,
                               float* state_ckpt_out, int64_t ckpt_rows, float scale,
                               uint32_t flags, void* o, void* workspace, size_t ws_bytes,
                               gdn_dims_t dims, gdn_dtype_t dtype, void* stream) {
    return chunk_prefill_impl(qkv, a, b, A_log, dt_bias, g, beta, cu_seqlens, n_seq, T_tot, initial_state,
                              final_state, ckpt_every, state_ckpt_out, ckpt_rows, scale, flags, o, workspace,
                              ws_bytes, dims, dtype, stream, nullptr, nullptr, 0.f, nullptr);
}

gdn_status_t gdn_chunk_prefill_norm(const void* qkv, const void* a, const void* b, const float* A_log,
                                    const float* dt_bias, const float* g, const float* beta,
                                    const int32_t* cu_seqlens, int32_t n_seq, int64_t T_tot,
                                    const float* initial_state, float* final_state, int32_t ckpt_every,
                                    float* state_ckpt_out, int64_t ckpt_rows, float scale, uint32_t flags,
                                    const void* z, const void* norm_w, float norm_eps, void* out,
                                    void* workspace, size_t ws_bytes, gdn_dims_t dims, gdn_dtype_t dtype,
                                    void* stream) {
    if (!isfinite(norm_eps) || norm_eps <= 0.f || norm_w == nullptr) return GDN_ERR_INVALID_ARG;
    if (T_tot > 0 && z == nullptr) return GDN_ERR_INVALID_ARG;
    if (!aligned16(z) || !aligned16(norm_w)) return GDN_ERR_ALIGN;
    return chunk_prefill_impl(qkv, a, b, A_log, dt_bias, g, beta, cu_seqlens, n_seq, T_tot, initial_state,
                              final_state, ckpt_every, state_ckpt_out, ckpt_rows, scale, flags, out, workspace,
                              ws_bytes, dims, dtype, stream, z, norm_w, norm_eps, T_tot > 0 ? out : nullptr);
}

size_t gdn_layer_prefill_workspace_size(int32_t n_seq, int64_t T_tot, gdn_dims_t dims, gdn_dtype_t dtype) {
    if (check_dims(dims, dtype) != GDN_OK || n_seq < 1 || T_tot <= 0 || T_tot > (int64_t)INT32_MAX) return 0;
    // tensor-core path: the conv runs inside the chunk kernels (no y buffer)
    if (dtype == GDN_BF16 && dims.d_k == 128) return gdn::chunk_split_conv_workspace_bytes(n_seq, T_tot, dims.H_k, dims.H_v);
    return ((size_t)T_tot * (size_t)conv_dim_of(dims) * elem_size(dtype) + 255) & ~(size_t)255;
}

int32_t gdn_layer_prefill_launches(int32_t n_seq, int64_t T_tot, int32_t has_cu_seqlens, gdn_dims_t dims,
                                   gdn_dtype_t dtype, uint32_t flags) {
    if (check_dims(dims, dtype) != GDN_OK || n_seq < 1 || T_tot <= 0) return 0;
    // the chunked rule and the norm, and the conv (on the tensor-core path it
    // runs in the chunk kernels, which with conv_state_out not conv_state_in
    // also write the conv state)
    const bool tc = dtype == GDN_BF16 && dims.d_k == 128;
    return (tc ? 1 : 2) + gdn_chunk_prefill_launches(n_seq, T_tot, has_cu_seqlens, dims, dtype, flags);
}

gdn_status_t gdn_layer_prefill(const void* x, const void* z, const void* a, const void* b, const void* conv_w,
                               const float* A_log, const float* dt_bias, const void* norm_w, float norm_eps,
                               const int32_t* cu_seqlens, int32_t n_seq, int64_t T_tot,
                               const float* initial_state, float* final_state, const void* conv_state_in,
                               void* conv_state_out, int32_t ckpt_every, float* state_ckpt_out,
                               void* conv_ckpt_out, int64_t ckpt_rows, float scale, uint32_t flags, void* out,
                               void* workspace, size_t ws_bytes, gdn_dims_t dims, gdn_dtype_t dtype,
                               void* stream) {
    gdn_status_t st = check_dims(dims, dtype);
    if (st != GDN_OK) return st;
    if ((st = check_seqs(cu_seqlens, n_seq, T_tot)) != GDN_OK) return st;
    if ((st = check_ckpt(ckpt_every, state_ckpt_out, ckpt_rows)) != GDN_OK) return st;
    if ((st = check_ckpt(ckpt_every, conv_ckpt_out, ckpt_rows)) != GDN_OK) return st;
    if (!isfinite(norm_eps) || norm_eps <= 0.f) return GDN_ERR_INVALID_ARG;
    if (conv_w == nullptr || norm_w == nullptr || A_log == nullptr || dt_bias == nullptr) return GDN_ERR_INVALID_ARG;
    if (T_tot > 0 && (x == nullptr || z == nullptr || a == nullptr || b == nullptr || out == nullptr))
        return GDN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(z) || !aligned16(norm_w) || !aligned16(out) || !aligned16(workspace))
        return GDN_ERR_ALIGN;
    const size_t need = gdn_layer_prefill_workspace_size(n_seq, T_tot, dims, dtype);
    if (need > 0 && (workspace == nullptr || ws_bytes < need)) return GDN_ERR_WORKSPACE;
    if (T_tot > 0 && dtype == GDN_BF16 && dims.d_k == 128) {
        // tensor-core path: conv1d + SiLU, the conv state and the conv
        // checkpoints inside the chunk kernels (the state in place: by a pass
        // after them), then RMSNormGated
        if ((st = check_gates(a, b, A_log, dt_bias, nullptr, nullptr, dtype)) != GDN_OK) return st;
        if (flags & ~(GDN_QK_L2NORM | GDN_SOLVE_NEUMANN | GDN_CHUNK(0xff))) return GDN_ERR_INVALID_ARG;
        const uint32_t c = (flags >> 8) & 0xffu;
        if (c != 0 && c != 16 && c != 32 && c != 64) return GDN_ERR_INVALID_ARG;
        // shorter chunks: more segments, the state crossing them through final_state
        if (c == 16 || c == 32) {
            if (final_state == nullptr) return GDN_ERR_UNSUPPORTED;
        }
        if (!isfinite(scale)) return GDN_ERR_INVALID_ARG;
        if (!aligned16(conv_w) || !aligned16(conv_state_in) || !aligned16(conv_state_out) ||
            !aligned16(conv_ckpt_out) || !aligned16(initial_state) || !aligned16(final_state) ||
            !aligned16(state_ckpt_out))
            return GDN_ERR_ALIGN;
        if ((int64_t)n_seq * dims.H_v * 8 > INT32_MAX) return GDN_ERR_UNSUPPORTED;
        gdn::DeltaArgs d;
        memset(&d, 0, sizeof(d));
        d.qkv = x; d.a = a; d.b = b; d.A_log = A_log; d.dt_bias = dt_bias;
        d.cu = cu_seqlens; d.n_seq = n_seq; d.T = T_tot;
        d.H_k = dims.H_k; d.H_v = dims.H_v; d.D = dims.d_k;
        d.S0 = initial_state; d.S_final = final_state;
        d.ckpt_every = ckpt_every; d.ckpt = ckpt_every > 0 ? state_ckpt_out : nullptr;
        d.ckpt_rows = ckpt_rows;
        d.scale = scale == 0.f ? 1.0f / sqrtf((float)dims.d_k) : scale;
        d.l2norm = (flags & GDN_QK_L2NORM) != 0;
        d.neumann = (flags & GDN_SOLVE_NEUMANN) != 0;
        d.chunk = c == 0 ? 64 : (int)c;
        d.o = out;
        d.conv_w = conv_w;
        d.conv_state0 = conv_state_in;
        // the kernels write the conv state and checkpoints unless the state is
        // updated in place (the kernels of other chunks still read it)
        const bool in_place = conv_state_out != nullptr && conv_state_out == conv_state_in;
        if (!in_place) {
            d.conv_state_out = conv_state_out;
            d.conv_ckpt = ckpt_every > 0 ? conv_ckpt_out : nullptr;
        }
        cudaStream_t s = (cudaStream_t)stream;
        cudaError_t e = gdn::launch_chunk_split(d, workspace, ws_bytes, s);
        if (e == cudaSuccess && in_place) {
            gdn::ConvArgs c;
            memset(&c, 0, sizeof(c));
            c.x = x; c.w = conv_w; c.cu = cu_seqlens; c.n_seq = n_seq; c.T = T_tot;
            c.C = (int)conv_dim_of(dims);
            c.state_in = conv_state_in; c.state_out = conv_state_out;
            c.ckpt_every = ckpt_every; c.ckpt = ckpt_every > 0 ? conv_ckpt_out : nullptr;
            c.ckpt_rows = ckpt_rows; c.silu = 1;
            e = gdn::launch_conv1d_state(c, dtype, s);
        }
        if (e == cudaSuccess)
            e = gdn::launch_rmsnorm_gated(out, z, norm_w, norm_eps, T_tot, dims.H_v, dims.d_v, out, dtype, s);
        return cuda_status(e);
    }
    const size_t ybytes = T_tot > 0 ? ((size_t)T_tot * (size_t)conv_dim_of(dims) * elem_size(dtype) + 255) &
                                          ~(size_t)255
                                    : 0;
    void* y = T_tot > 0 ? workspace : nullptr;
    void* cws = need > ybytes ? static_cast<uint8_t*>(workspace) + ybytes : nullptr;
    st = gdn_conv1d_fwd(x, conv_w, cu_seqlens, n_seq, T_tot, conv_state_in, conv_state_out, ckpt_every,
                        conv_ckpt_out, ckpt_rows, 1, y, dims, dtype, stream);
    if (st != GDN_OK) return st;
    return gdn_chunk_prefill_norm(y, a, b, A_log, dt_bias, nullptr, nullptr, cu_seqlens, n_seq, T_tot,
                                  initial_state, final_state, ckpt_every, state_ckpt_out, ckpt_rows, scale, flags,
                                  z, norm_w, norm_eps, out, cws, need - ybytes, dims, dtype, stream);
}

gdn_status_t gdn_chunk_prefill_noalloc(const void* qkv, const void* a, const void* b,
                                       const float* A_log, const float* dt_bias, const float* g,
                                       const float* beta, const int32_t* cu_seqlens, int32_t n_seq,
                                       int64_t T_tot, const float* initial_state, float* final_state,
                                       int32_t ckpt_every, float* state_ckpt_out, int64_t ckpt_rows,
                                       float scale, uint32_t flags, void* o, gdn_dims_t dims,
                                       gdn_dtype_t dtype, void* stream) {
    gdn_status_t st = check_dims(dims, dtype);
    if (st != GDN_OK) return st;
    if (dtype != GDN_BF16 || dims.d_k != 128) return GDN_ERR_UNSUPPORTED;
    if ((st = check_seqs(cu_seqlens, n_seq, T_tot)) != GDN_OK) return st;
    if ((st = check_ckpt(ckpt_every, state_ckpt_out, ckpt_rows)) != GDN_OK) return st;
    if (T_tot > 0 && (st = check_gates(a, b, A_log, dt_bias, g, beta, dtype)) != GDN_OK) return st;
    if (flags & ~GDN_QK_L2NORM) return GDN_ERR_INVALID_ARG;
    if (!isfinite(scale)) return GDN_ERR_INVALID_ARG;
    if (final_state == nullptr) return GDN_ERR_INVALID_ARG;
    if (T_tot > 0 && (qkv == nullptr || o == nullptr)) return GDN_ERR_INVALID_ARG;
    if (!aligned16(qkv) || !aligned16(o) || !aligned16(initial_state) || !aligned16(final_state) ||
        !aligned16(state_ckpt_out))
        return GDN_ERR_ALIGN;
    if (!gdn::chunk_split_static_fits(n_seq, dims.H_v)) return GDN_ERR_WORKSPACE;
    if (T_tot == 0) {
        // nothing to compute: the final state of every (empty) sequence is its initial state
        const size_t bytes = (size_t)n_seq * dims.H_v * dims.d_k * dims.d_v * sizeof(float);
        cudaError_t e = initial_state != nullptr
                            ? (initial_state == final_state
                                   ? cudaSuccess
                                   : cudaMemcpyAsync(final_state, initial_state, bytes,
                                                     cudaMemcpyDeviceToDevice, (cudaStream_t)stream))
                            : cudaMemsetAsync(final_state, 0, bytes, (cudaStream_t)stream);
        return cuda_status(e);
    }
    gdn::DeltaArgs d;
    memset(&d, 0, sizeof(d));
    d.qkv = qkv; d.a = a; d.b = b; d.A_log = A_log; d.dt_bias = dt_bias;
    const bool pre = g && beta;
    d.g = pre ? g : nullptr; d.beta = pre ? beta : nullptr;
    d.cu = cu_seqlens; d.n_seq = n_seq; d.T = T_tot;
    d.H_k = dims.H_k; d.H_v = dims.H_v; d.D = dims.d_k;
    d.S0 = initial_state; d.S_final = final_state;
    d.ckpt_every = ckpt_every; d.ckpt = ckpt_every > 0 ? state_ckpt_out : nullptr;
    d.ckpt_rows = ckpt_rows;
    d.scale = scale == 0.f ? 1.0f / sqrtf((float)dims.d_k) : scale;
    d.l2norm = (flags & GDN_QK_L2NORM) != 0;
    d.o = o;
    return cuda_status(gdn::launch_chunk_split_static(d, (cudaStream_t)stream));
}

gdn_status_t gdn_recurrent_decode(const void* qkv, const void* a, const void* b,
                                  const float* A_log, const float* dt_bias, const float* g,
                                  const float* beta, float* state, int32_t B, float scale,
                                  uint32_t flags, void* o, gdn_dims_t dims, gdn_dtype_t dtype,
                                  void* stream) {
    gdn_status_t st = check_dims(dims, dtype);
    if (st != GDN_OK) return st;
    if (B < 0 || (int64_t)B * dims.H_v > INT32_MAX) return GDN_ERR_INVALID_ARG;
    if (B > 0 && (st = check_gates(a, b, A_log, dt_bias, g, beta, dtype)) != GDN_OK) return st;
    if (flags & ~GDN_QK_L2NORM) return GDN_ERR_INVALID_ARG;
    if (!isfinite(scale)) return GDN_ERR_INVALID_ARG;
    if (B > 0 && (qkv == nullptr || state == nullptr || o == nullptr)) return GDN_ERR_INVALID_ARG;
    if (!aligned16(qkv) || !aligned16(state) || !aligned16(o)) return GDN_ERR_ALIGN;
    gdn::DeltaArgs d;
    memset(&d, 0, sizeof(d));
    d.qkv = qkv; d.a = a; d.b = b; d.A_log = A_log; d.dt_bias = dt_bias;
    const bool pre = g && beta;
    d.g = pre ? g : nullptr; d.beta = pre ? beta : nullptr;
    d.n_seq = B; d.T = B;
    d.H_k = dims.H_k; d.H_v = dims.H_v; d.D = dims.d_k;
    d.S0 = state; d.S_final = state;
    d.scale = scale == 0.f ? 1.0f / sqrtf((float)dims.d_k) : scale;
    d.l2norm = (flags & GDN_QK_L2NORM) != 0;
    d.o = o;
    return cuda_status(gdn::launch_recurrent_decode(d, dtype, (cudaStream_t)stream));
}

gdn_status_t gdn_rmsnorm_gated(const void* o, const void* z, const void* w, float eps, int64_t T,
                               void* out, gdn_dims_t dims, gdn_dtype_t dtype, void* stream) {
    gdn_status_t st = check_dims(dims, dtype);
    if (st != GDN_OK) return st;
    if (T < 0 || !(eps > 0.f) || !isfinite(eps)) return GDN_ERR_INVALID_ARG;
    if (w == nullptr || (T > 0 && (o == nullptr || z == nullptr || out == nullptr)))
        return GDN_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(z) || !aligned16(w) || !aligned16(out)) return GDN_ERR_ALIGN;
    return cuda_status(gdn::launch_rmsnorm_gated(o, z, w, eps, T, dims.H_v, dims.d_v, out, dtype,
                                                 (cudaStream_t)stream));
}

}  // extern "C"
