// Shared device helpers of the GDN layer-core kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------- scalar conversion
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// ---------------------------------------------------------------- 16-byte vectors
// VecN<T>::N elements of T fill one 16-byte (128-bit) access.
template <typename T> struct Vec16 { static constexpr int N = 16 / sizeof(T); };

// The Vec16<T>::N values of one 16-byte vector as f32 (bf16 -> f32 is exact).
template <typename T>
__device__ __forceinline__ void unpack16(uint4 u, float* out) {
    if constexpr (sizeof(T) == 4) {
        out[0] = __uint_as_float(u.x); out[1] = __uint_as_float(u.y);
        out[2] = __uint_as_float(u.z); out[3] = __uint_as_float(u.w);
    } else {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            out[2 * i] = __uint_as_float(w[i] << 16);
            out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
}

template <typename T>
__device__ __forceinline__ void load16(const T* __restrict__ p, float* out) {
    unpack16<T>(*reinterpret_cast<const uint4*>(p), out);
}

// Streaming variant: no L1 allocation (data read once).
template <typename T>
__device__ __forceinline__ void load16_stream(const T* __restrict__ p, float* out) {
    unpack16<T>(__ldcs(reinterpret_cast<const uint4*>(p)), out);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <typename T>
__device__ __forceinline__ void store16(T* __restrict__ p, const float* in) {
    uint4 u;
    if constexpr (sizeof(T) == 4) {
        u.x = __float_as_uint(in[0]); u.y = __float_as_uint(in[1]);
        u.z = __float_as_uint(in[2]); u.w = __float_as_uint(in[3]);
    } else {
        u.x = pack_bf16x2(in[0], in[1]); u.y = pack_bf16x2(in[2], in[3]);
        u.z = pack_bf16x2(in[4], in[5]); u.w = pack_bf16x2(in[6], in[7]);
    }
    *reinterpret_cast<uint4*>(p) = u;
}

// ---------------------------------------------------------------- dependent launch
// Programmatic dependent launch: a kernel launched with launch_pdl may have
// its CTAs placed while the previous kernel on the stream is still finishing;
// pdl_wait() blocks until that kernel has completed and its writes are
// visible, so every kernel calls it before touching global memory.
// pdl_trigger() lets the next kernel's CTAs be placed once every CTA of this
// grid has started.  Both are no-ops without a programmatic dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- math
// Full-precision CUDA math functions only (no hand-written approximations).
__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }
// SiLU with the hardware exponential and an approximate divide (a few ulp of
// f32; the exponent is clamped so the divisor stays finite and below 2^126).
__device__ __forceinline__ float silu_fast(float x) {
    return __fdividef(x, 1.0f + __expf(fminf(-x, 80.0f)));
}
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// SiLU of a pair as x sigma(x) = h (1 + tanh h), h = x / 2, with the hardware
// tanh (one special-function op per element; its relative error, a few 1e-4 at
// most, is below bf16 rounding, so this is used where the result is bf16).
__device__ __forceinline__ float2 silu2_tanh(float2 x) {
    const float2 h = __fmul2_rn(x, make_float2(0.5f, 0.5f));
    return __ffma2_rn(h, make_float2(tanh_approx(h.x), tanh_approx(h.y)), h);
}
// SiLU of a pair: the tanh form for bf16 results, the exponential form for f32.
template <typename T>
__device__ __forceinline__ float2 silu2(float2 x) {
    if constexpr (sizeof(T) == 2) return silu2_tanh(x);
    else return make_float2(silu_fast(x.x), silu_fast(x.y));
}
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

// ---------------------------------------------------------------- depthwise conv1d (k = 4)
// cortex commit "feat(stage-8c): linear-attention layer", "Block": depthwise
// causal conv (k = 4), then SiLU.  The helpers below are the conv's whole
// arithmetic, shared by every kernel that computes it, so that they agree bit
// for bit.  w is [C][4] (tap 0 multiplies the oldest input); taps are held as
// (channel 2k, channel 2k + 1) pairs per tap.
// Taps of the Vec16<T>::N channels from c0; raw[i] is the 16-byte vector of w
// from element 4 c0 + i Vec16<T>::N on.
template <typename T>
__device__ __forceinline__ void conv_taps(const uint4 (&raw)[4], float2 (&taps)[Vec16<T>::N / 2][4]) {
    constexpr int V = Vec16<T>::N;
    float tmp[4 * V];
#pragma unroll
    for (int i = 0; i < 4; ++i) unpack16<T>(raw[i], tmp + i * V);
#pragma unroll
    for (int k = 0; k < V / 2; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j) taps[k][j] = make_float2(tmp[(2 * k) * 4 + j], tmp[(2 * k + 1) * 4 + j]);
}
template <typename T>
__device__ __forceinline__ void load_conv_taps(const T* __restrict__ w, int64_t c0,
                                               float2 (&taps)[Vec16<T>::N / 2][4]) {
    uint4 raw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) raw[i] = *reinterpret_cast<const uint4*>(w + c0 * 4 + i * Vec16<T>::N);
    conv_taps<T>(raw, taps);
}
// bf16 taps of the two channel pairs from c0 (c0 even): raw = w[4 c0 .. 4 c0 + 16)
__device__ __forceinline__ void conv_taps_bf16_2(const uint4 (&raw)[2], float2 (&taps)[2][4]) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        float t[8];
        unpack16<bf16>(raw[k], t);
#pragma unroll
        for (int j = 0; j < 4; ++j) taps[k][j] = make_float2(t[j], t[4 + j]);
    }
}

// NP channel pairs of outputs at token t from the inputs at t-3 (x0) .. t
// (x3): w0 x0 + w1 x1 + w2 x2 + w3 x3 in that order, in packed f32x2
// arithmetic, then SiLU when `silu`.  Each channel's result does not depend
// on NP.
template <int NP, typename T>
__device__ __forceinline__ void conv4_pairs(const float2 (&w)[NP][4], const float* x0, const float* x1,
                                            const float* x2, const float* x3, int silu, float* out) {
#pragma unroll
    for (int k = 0; k < NP; ++k) {
        float2 acc = __fmul2_rn(w[k][0], make_float2(x0[2 * k], x0[2 * k + 1]));
        acc = __ffma2_rn(w[k][1], make_float2(x1[2 * k], x1[2 * k + 1]), acc);
        acc = __ffma2_rn(w[k][2], make_float2(x2[2 * k], x2[2 * k + 1]), acc);
        acc = __ffma2_rn(w[k][3], make_float2(x3[2 * k], x3[2 * k + 1]), acc);
        if (silu) acc = silu2<T>(acc);
        out[2 * k] = acc.x;
        out[2 * k + 1] = acc.y;
    }
}

// One 16-byte vector of outputs at token t from the inputs at t-3 (x0) .. t (x3).
template <typename T>
__device__ __forceinline__ void conv4_vec(const float2 (&w)[Vec16<T>::N / 2][4], const float* x0,
                                          const float* x1, const float* x2, const float* x3, int silu,
                                          float* out) {
    conv4_pairs<Vec16<T>::N / 2, T>(w, x0, x1, x2, x3, silu, out);
}

// softplus with the identity branch above 20 (cortex unit test "softplus small/large branches")
__device__ __forceinline__ float softplus_f(float x) { return x > 20.0f ? x : log1pf(expf(x)); }

// g = -exp(A_log) * softplus(a + dt_bias), computed in f32 (cortex "Discretisation")
__device__ __forceinline__ float gate_g(float a, float A_log, float dt_bias) {
    return -expf(A_log) * softplus_f(a + dt_bias);
}

// ---------------------------------------------------------------- packed sequences
// Clamped bounds of sequence i: 0 <= start <= end <= T.  cu == nullptr means
// one sequence [0, T).
__device__ __forceinline__ void seq_bounds(const int32_t* __restrict__ cu, int i, int64_t T,
                                           int64_t& start, int64_t& end) {
    if (cu == nullptr) { start = 0; end = T; return; }
    int64_t s = cu[i], e = cu[i + 1];
    s = s < 0 ? 0 : (s > T ? T : s);
    e = e < s ? s : (e > T ? T : e);
    start = s; end = e;
}

// Largest i in [0, n_seq) with cu[i] <= t (binary search; cu non-decreasing).
__device__ __forceinline__ int seq_of_token(const int32_t* __restrict__ cu, int n_seq, int64_t t) {
    if (cu == nullptr) return 0;
    int lo = 0, hi = n_seq - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Checkpoint row offset of sequence i: sum_{j<i} floor(L_j / every).
__device__ __forceinline__ int64_t ckpt_row0(const int32_t* __restrict__ cu, int i, int64_t T,
                                             int every) {
    int64_t r = 0;
    for (int j = 0; j < i; ++j) {
        int64_t s, e;
        seq_bounds(cu, j, T, s, e);
        r += (e - s) / every;
    }
    return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace gdn
