// Depthwise causal conv1d (width 4) + SiLU for the GDN layer core.
//
// cortex commit "feat(stage-8c): linear-attention layer (Qwen3-Next
// GatedDeltaNet)", "Block": depthwise causal Conv1d (k=4) with state-aware
// prepend; SiLU.  "State": conv_state holds the left-padded tail of raw inputs
// (here its 3 newest columns, column 0 oldest).  NxD-Inference PR "Add
// Qwen3.6-27B hybrid DeltaNet/GQA contrib model and vLLM serving path",
// Summary: convolution state checkpoints for hybrid prefix caching.
//
// The conv is HBM-bound (about 4 bytes of traffic per bf16 channel-token and
// 4 FMAs).  Each thread owns one 16-byte channel vector (8 bf16 or 4 f32
// channels) of a run of kTok tokens.  A run inside one sequence issues all of
// its kTok + 3 row loads at once (the 3 halo rows are the previous run's last
// rows, mostly L2 hits) and then writes kTok outputs, so every thread has one
// memory round trip; coalesced 128-bit accesses (a warp covers 512 contiguous
// bytes of a token row).  Runs that touch a sequence start take the general
// path, which walks the tokens with the three previous inputs in registers.
#include "gdn_common.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr int kTok = 8;       // tokens per thread
constexpr int kThreads = 128;

template <typename T>
__device__ __forceinline__ void load_state_col(const T* __restrict__ st, int64_t seq, int C, int c0,
                                               int col, float* dst) {
    constexpr int V = Vec16<T>::N;
#pragma unroll
    for (int e = 0; e < V; ++e) dst[e] = to_f(st[((int64_t)seq * C + c0 + e) * 3 + col]);
}

template <typename T>
__device__ __forceinline__ void conv_out(const float (&w)[Vec16<T>::N][4], const float* w0,
                                         const float* w1, const float* w2, const float* cur,
                                         int silu, T* __restrict__ dst) {
    constexpr int V = Vec16<T>::N;
    float out[V];
#pragma unroll
    for (int e = 0; e < V; ++e) {
        float acc = w[e][0] * w0[e];
        acc = fmaf(w[e][1], w1[e], acc);
        acc = fmaf(w[e][2], w2[e], acc);
        acc = fmaf(w[e][3], cur[e], acc);
        out[e] = silu ? silu_fast(acc) : acc;
    }
    store16(dst, out);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) conv1d_fwd_kernel(ConvArgs a) {
    constexpr int V = Vec16<T>::N;
    const int nvec = a.C / V;
    const int cv = blockIdx.y * blockDim.x + threadIdx.x;
    if (cv >= nvec) return;
    const int C = a.C;
    const int c0 = cv * V;
    const T* __restrict__ x = static_cast<const T*>(a.x);
    const T* __restrict__ st = static_cast<const T*>(a.state_in);
    T* __restrict__ y = static_cast<T*>(a.y);

    float w[V][4];
    {
        const T* wp = static_cast<const T*>(a.w) + (int64_t)c0 * 4;
        float tmp[4 * V];
#pragma unroll
        for (int i = 0; i < 4; ++i) load16(wp + i * V, tmp + i * V);
#pragma unroll
        for (int e = 0; e < V; ++e)
#pragma unroll
            for (int j = 0; j < 4; ++j) w[e][j] = tmp[e * 4 + j];
    }

    const int64_t t0 = (int64_t)blockIdx.x * kTok;
    const int64_t t1 = t0 + kTok < a.T ? t0 + kTok : a.T;
    int seq = seq_of_token(a.cu, a.n_seq, t0);
    int64_t s, e;
    seq_bounds(a.cu, seq, a.T, s, e);

    if (t0 - 3 >= s && t0 + kTok <= e) {
        // the run and its halo lie inside one sequence: one round trip
        uint4 raw[kTok + 3];
#pragma unroll
        for (int j = 0; j < kTok + 3; ++j)
            raw[j] = __ldg(reinterpret_cast<const uint4*>(x + (t0 - 3 + j) * C + c0));
        float r0[V], r1[V], r2[V], r3[V];
        unpack16<T>(raw[0], r0);
        unpack16<T>(raw[1], r1);
        unpack16<T>(raw[2], r2);
#pragma unroll
        for (int j = 0; j < kTok; ++j) {
            unpack16<T>(raw[j + 3], r3);
            conv_out<T>(w, r0, r1, r2, r3, a.silu, y + (t0 + j) * C + c0);
#pragma unroll
            for (int q = 0; q < V; ++q) {
                r0[q] = r1[q];
                r1[q] = r2[q];
                r2[q] = r3[q];
            }
        }
        return;
    }

    float win[3][V];  // inputs at t-3, t-2, t-1
    bool need_init = true;
    int64_t t = t0;
    while (t < t1) {
        while (t >= e && seq + 1 < a.n_seq) {
            ++seq;
            seq_bounds(a.cu, seq, a.T, s, e);
            need_init = true;
        }
        if (need_init) {
            const int64_t ss = s < t ? s : t;  // clamp (only differs for invalid offsets)
#pragma unroll
            for (int j = 1; j <= 3; ++j) {
                float* dst = win[3 - j];
                const int64_t p = t - j;
                if (p >= ss) {
                    load16(x + p * C + c0, dst);
                } else if (st != nullptr) {
                    load_state_col(st, seq, C, c0, (int)(3 - (ss - p)), dst);
                } else {
#pragma unroll
                    for (int q = 0; q < V; ++q) dst[q] = 0.f;
                }
            }
            need_init = false;
        }
        const int64_t lim = e < t1 ? e : t1;
        if (t + 4 <= lim) {
            // four tokens inside one sequence: issue the loads together
            float c[4][V];
#pragma unroll
            for (int u = 0; u < 4; ++u) load16_stream(x + (t + u) * C + c0, c[u]);
            conv_out<T>(w, win[0], win[1], win[2], c[0], a.silu, y + t * C + c0);
            conv_out<T>(w, win[1], win[2], c[0], c[1], a.silu, y + (t + 1) * C + c0);
            conv_out<T>(w, win[2], c[0], c[1], c[2], a.silu, y + (t + 2) * C + c0);
            conv_out<T>(w, c[0], c[1], c[2], c[3], a.silu, y + (t + 3) * C + c0);
#pragma unroll
            for (int q = 0; q < V; ++q) {
                win[0][q] = c[1][q];
                win[1][q] = c[2][q];
                win[2][q] = c[3][q];
            }
            t += 4;
        } else {
            float c[V];
            load16_stream(x + t * C + c0, c);
            conv_out<T>(w, win[0], win[1], win[2], c, a.silu, y + t * C + c0);
#pragma unroll
            for (int q = 0; q < V; ++q) {
                win[0][q] = win[1][q];
                win[1][q] = win[2][q];
                win[2][q] = c[q];
            }
            t += 1;
        }
    }
}

// Conv state after a sequence (and its checkpoints): the 3 newest raw inputs
// of [state_in | x].  One thread per (sequence, 16-byte channel vector); each
// thread reads every state value it needs before writing, so state_out may
// alias state_in.  Values are bit copies (bf16 -> f32 -> bf16 is exact).
template <typename T>
__global__ void __launch_bounds__(kThreads) conv1d_state_kernel(ConvArgs a) {
    constexpr int V = Vec16<T>::N;
    const int nvec = a.C / V;
    const int cv = blockIdx.y * blockDim.x + threadIdx.x;
    if (cv >= nvec) return;
    const int C = a.C;
    const int c0 = cv * V;
    const int seq = blockIdx.x;
    const T* __restrict__ x = static_cast<const T*>(a.x);
    const T* st = static_cast<const T*>(a.state_in);
    int64_t s, e;
    seq_bounds(a.cu, seq, a.T, s, e);
    const int64_t L = e - s;

    if (a.state_out != nullptr) {
        float v[3][V];
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int64_t p = L - 3 + j;
            if (p >= 0) {
                load16(x + (s + p) * C + c0, v[j]);
            } else if (st != nullptr) {
                load_state_col(st, seq, C, c0, (int)(3 + p), v[j]);
            } else {
#pragma unroll
                for (int q = 0; q < V; ++q) v[j][q] = 0.f;
            }
        }
        // [c][3] layout: 3V contiguous elements = three 16-byte vectors
        float flat[3 * V];
#pragma unroll
        for (int q = 0; q < V; ++q)
#pragma unroll
            for (int j = 0; j < 3; ++j) flat[q * 3 + j] = v[j][q];
        T* dst = static_cast<T*>(a.state_out) + ((int64_t)seq * C + c0) * 3;
#pragma unroll
        for (int i = 0; i < 3; ++i) store16(dst + i * V, flat + i * V);
    }

    if (a.ckpt_every > 0 && a.ckpt != nullptr) {
        const int64_t row0 = ckpt_row0(a.cu, seq, a.T, a.ckpt_every);
        for (int64_t m = 1; m * a.ckpt_every <= L; ++m) {
            const int64_t row = row0 + m - 1;
            if (row >= a.ckpt_rows) break;
            float v[3][V];
#pragma unroll
            for (int j = 0; j < 3; ++j) load16(x + (s + m * a.ckpt_every - 3 + j) * C + c0, v[j]);
            float flat[3 * V];
#pragma unroll
            for (int q = 0; q < V; ++q)
#pragma unroll
                for (int j = 0; j < 3; ++j) flat[q * 3 + j] = v[j][q];
            T* dst = static_cast<T*>(a.ckpt) + (row * C + c0) * 3;
#pragma unroll
            for (int i = 0; i < 3; ++i) store16(dst + i * V, flat + i * V);
        }
    }
}

// Decode: one token per sequence, conv state shifted in place.
template <typename T>
__global__ void __launch_bounds__(kThreads) conv1d_update_kernel(const T* __restrict__ x,
                                                                 const T* __restrict__ w,
                                                                 T* __restrict__ state, int C,
                                                                 int silu, T* __restrict__ y) {
    constexpr int V = Vec16<T>::N;
    const int cv = blockIdx.y * blockDim.x + threadIdx.x;
    if (cv >= C / V) return;
    const int c0 = cv * V;
    const int64_t b = blockIdx.x;
    float wt[4 * V], cur[V], flat[3 * V];
#pragma unroll
    for (int i = 0; i < 4; ++i) load16(w + (int64_t)c0 * 4 + i * V, wt + i * V);
    load16(x + b * C + c0, cur);
    T* sp = state + (b * C + c0) * 3;
#pragma unroll
    for (int i = 0; i < 3; ++i) load16(sp + i * V, flat + i * V);
    float out[V], nst[3 * V];
#pragma unroll
    for (int q = 0; q < V; ++q) {
        float acc = wt[q * 4 + 0] * flat[q * 3 + 0];
        acc = fmaf(wt[q * 4 + 1], flat[q * 3 + 1], acc);
        acc = fmaf(wt[q * 4 + 2], flat[q * 3 + 2], acc);
        acc = fmaf(wt[q * 4 + 3], cur[q], acc);
        out[q] = silu ? silu_f(acc) : acc;
        nst[q * 3 + 0] = flat[q * 3 + 1];
        nst[q * 3 + 1] = flat[q * 3 + 2];
        nst[q * 3 + 2] = cur[q];
    }
    store16(y + b * C + c0, out);
#pragma unroll
    for (int i = 0; i < 3; ++i) store16(sp + i * V, nst + i * V);
}

template <typename T>
cudaError_t conv_fwd_t(const ConvArgs& a, cudaStream_t s) {
    constexpr int V = Vec16<T>::N;
    const int nvec = a.C / V;
    const dim3 blk(kThreads);
    if (a.T > 0) {
        const dim3 grid((unsigned)((a.T + kTok - 1) / kTok), (nvec + kThreads - 1) / kThreads);
        conv1d_fwd_kernel<T><<<grid, blk, 0, s>>>(a);
    }
    if (a.state_out != nullptr || (a.ckpt_every > 0 && a.ckpt != nullptr)) {
        const dim3 grid2((unsigned)a.n_seq, (nvec + kThreads - 1) / kThreads);
        conv1d_state_kernel<T><<<grid2, blk, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv1d_fwd(const ConvArgs& a, gdn_dtype_t dt, cudaStream_t s) {
    return dt == GDN_BF16 ? conv_fwd_t<bf16>(a, s) : conv_fwd_t<float>(a, s);
}

cudaError_t launch_conv1d_update(const void* x, const void* w, void* state, int B, int C,
                                 int silu, void* y, gdn_dtype_t dt, cudaStream_t s) {
    if (B == 0) return cudaSuccess;
    const dim3 blk(kThreads);
    if (dt == GDN_BF16) {
        const dim3 grid(B, (C / 8 + kThreads - 1) / kThreads);
        conv1d_update_kernel<bf16><<<grid, blk, 0, s>>>(
            (const bf16*)x, (const bf16*)w, (bf16*)state, C, silu, (bf16*)y);
    } else {
        const dim3 grid(B, (C / 4 + kThreads - 1) / kThreads);
        conv1d_update_kernel<float><<<grid, blk, 0, s>>>(
            (const float*)x, (const float*)w, (float*)state, C, silu, (float*)y);
    }
    return cudaGetLastError();
}

}  // namespace gdn
