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
// 4 FMAs).  A CTA takes a tile of 64 tokens x 512 bytes of channels: one TMA
// copy brings the tile and its 3-token halo (negative rows read as zeros)
// into shared memory, so x is read 67/64 times; each thread then owns one
// 16-byte channel vector (8 bf16 or 4 f32 channels) of 8 tokens and writes
// them with coalesced 128-bit stores (a warp covers a 512-byte token row).
// Inputs before a sequence's first token come from its conv state (or are
// zero), not from the tile.
#include "gdn_common.cuh"
#include "gdn_launch.h"
#include "tc_ptx.cuh"

namespace gdn {

__device__ int g_conv_error;  // bit 0: a bounded wait gave up

namespace {

constexpr int kThreads = 128;  // decode and state kernels
constexpr int kTT = 64;        // tokens per tile
constexpr int kRowBytes = 512;  // bytes of channels per tile row
constexpr int kTileThreads = 256;
constexpr uint64_t kConvWaitNs = 1000000000ull;

template <typename T>
__device__ __forceinline__ void load_state_col(const T* __restrict__ st, int64_t seq, int C, int c0,
                                               int col, float* dst) {
    constexpr int V = Vec16<T>::N;
#pragma unroll
    for (int e = 0; e < V; ++e) dst[e] = to_f(st[((int64_t)seq * C + c0 + e) * 3 + col]);
}

// One 16-byte vector of outputs from the inputs at t-3..t, stored at dst.
template <typename T>
__device__ __forceinline__ void conv_out2(const float2 (&w)[Vec16<T>::N / 2][4], const float* x0,
                                          const float* x1, const float* x2, const float* x3, int silu,
                                          T* __restrict__ dst) {
    float out[Vec16<T>::N];
    conv4_vec<T>(w, x0, x1, x2, x3, silu, out);
    store16(dst, out);
}

template <typename T>
__global__ void __launch_bounds__(kTileThreads, 3) conv1d_fwd_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                  ConvArgs a) {
    constexpr int V = Vec16<T>::N;
    constexpr int TC = kRowBytes / (int)sizeof(T);  // channels per tile
    __shared__ alignas(128) uint8_t tile[(kTT + 3) * kRowBytes];
    __shared__ alignas(8) uint64_t bar;
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, cg = tid & 31, tg = tid >> 5;
    const int64_t t0 = (int64_t)blockIdx.x * kTT;
    const int cbase = blockIdx.y * TC;
    if (tid == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
        tc::mbar_arrive_expect_tx(&bar, (kTT + 3) * kRowBytes);
        tc::tma_load_2d(tile, &xmap, &bar, cbase, (int)(t0 - 3));  // row r of the tile = token t0 - 3 + r
    }
    __syncthreads();
    // while the copy is in flight: weights and the sequence of the first token
    const int C = a.C;
    const int c0 = cbase + cg * V;
    const bool cv = c0 < C;
    float2 w[V / 2][4];  // (channel 2k, channel 2k + 1) x tap
    if (cv) load_conv_taps(static_cast<const T*>(a.w), c0, w);
    const int64_t tb = t0 + 8 * tg;
    const int64_t te = tb + 8 < a.T ? tb + 8 : a.T;
    int seq = 0;
    int64_t s = 0, e = a.T;
    if (tb < a.T) {
        seq = seq_of_token(a.cu, a.n_seq, tb);
        seq_bounds(a.cu, seq, a.T, s, e);
    }
    const bool landed = tc::mbar_wait(&bar, 0, kConvWaitNs);
    if (!landed) {
        if (tid == 0) atomicOr(&g_conv_error, 1);
        return;
    }
    if (!cv || tb >= a.T) return;
    const T* st = static_cast<const T*>(a.state_in);
    T* __restrict__ y = static_cast<T*>(a.y);
    auto row = [&](int64_t p, float* dst) {  // input of token p (p >= t0 - 3) from the tile
        unpack16<T>(*reinterpret_cast<const uint4*>(tile + (p - t0 + 3) * kRowBytes + cg * 16), dst);
    };
    // One sequence and no aliasing (fused_state): the run holding the last
    // token writes the conv state, and the run holding token m N - 1 the m-th
    // checkpoint -- the 3 raw inputs ending there, from the tile (its halo
    // reaches back 3 tokens) or, for a sequence shorter than 3, from state_in
    // (zeros without one).  Values are bit copies.
    auto write3 = [&](int64_t last, T* dst) {
        float flat[3 * V];  // [channel][3] order of the state
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int64_t p = last - 2 + j;
            float v[V];
            if (p >= 0) {
                row(p, v);
            } else if (st != nullptr) {
                load_state_col(st, 0, C, c0, (int)(3 + p), v);
            } else {
#pragma unroll
                for (int q = 0; q < V; ++q) v[q] = 0.f;
            }
#pragma unroll
            for (int q = 0; q < V; ++q) flat[q * 3 + j] = v[q];
        }
#pragma unroll
        for (int i = 0; i < 3; ++i) store16(dst + i * V, flat + i * V);
    };
    auto fused_state = [&]() {
        if (!a.fused_state) return;
        if (a.state_out != nullptr && a.T - 1 < te)
            write3(a.T - 1, static_cast<T*>(a.state_out) + (int64_t)c0 * 3);
        if (a.ckpt_every > 0 && a.ckpt != nullptr) {
            for (int64_t m = (tb + a.ckpt_every) / a.ckpt_every; m * a.ckpt_every - 1 < te; ++m) {
                if (m - 1 >= a.ckpt_rows) break;
                write3(m * a.ckpt_every - 1, static_cast<T*>(a.ckpt) + ((m - 1) * C + c0) * 3);
            }
        }
    };
    if (tb - 3 >= s && te <= e) {
        // the run and its halo lie inside one sequence
        float r0[V], r1[V], r2[V], r3[V];
        row(tb - 3, r0);
        row(tb - 2, r1);
        row(tb - 1, r2);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (tb + j >= te) break;
            row(tb + j, r3);
            conv_out2<T>(w, r0, r1, r2, r3, a.silu, y + (tb + j) * C + c0);
#pragma unroll
            for (int q = 0; q < V; ++q) {
                r0[q] = r1[q];
                r1[q] = r2[q];
                r2[q] = r3[q];
            }
        }
        fused_state();
        return;
    }
    // a sequence starts inside the run or its halo
    for (int64_t t = tb; t < te; ++t) {
        while (t >= e && seq + 1 < a.n_seq) {
            ++seq;
            seq_bounds(a.cu, seq, a.T, s, e);
        }
        float in[4][V];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int64_t p = t - 3 + m;
            if (p >= s) {
                row(p, in[m]);
            } else if (st != nullptr) {
                load_state_col(st, seq, C, c0, (int)(3 - (s - p)), in[m]);
            } else {
#pragma unroll
                for (int q = 0; q < V; ++q) in[m][q] = 0.f;
            }
        }
        conv_out2<T>(w, in[0], in[1], in[2], in[3], a.silu, y + t * C + c0);
    }
    fused_state();
}

// Conv state after a sequence (and its checkpoints): the 3 newest raw inputs
// of [state_in | x].  One thread per (sequence, 16-byte channel vector); each
// thread reads every state value it needs before writing, so state_out may
// alias state_in.  Values are bit copies (bf16 -> f32 -> bf16 is exact).
template <typename T>
__global__ void __launch_bounds__(kThreads) conv1d_state_kernel(ConvArgs a) {
    constexpr int V = Vec16<T>::N;
    pdl_wait();
    pdl_trigger();
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
cudaError_t conv_fwd_t(const ConvArgs& args, cudaStream_t s) {
    constexpr int V = Vec16<T>::N;
    // one sequence whose state_out does not alias state_in: the tile kernel
    // writes the state and checkpoints (no tile reads what another writes);
    // otherwise a second pass does, after every tile has read state_in
    ConvArgs a = args;
    a.fused_state = a.cu == nullptr && a.T > 0 && (a.state_in == nullptr || a.state_in != a.state_out);
    constexpr int TC = kRowBytes / (int)sizeof(T);
    const int nvec = a.C / V;
    const dim3 blk(kThreads);
    if (a.T > 0) {
        // x as a [T][C] tensor; a box is one tile with its halo
        const PFN_cuTensorMapEncodeTiled_v12000 enc = tensormap_encoder();
        if (enc == nullptr) return cudaErrorNotSupported;
        CUtensorMap xmap;
        cuuint64_t gdim[2] = {(cuuint64_t)a.C, (cuuint64_t)a.T};
        cuuint64_t gstr[1] = {(cuuint64_t)a.C * sizeof(T)};
        cuuint32_t box[2] = {(cuuint32_t)TC, (cuuint32_t)(kTT + 3)};
        cuuint32_t es[2] = {1, 1};
        if (enc(&xmap, sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                const_cast<void*>(a.x), gdim, gstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        const dim3 grid((unsigned)((a.T + kTT - 1) / kTT), (unsigned)((a.C + TC - 1) / TC));
        const cudaError_t e = launch_pdl(conv1d_fwd_kernel<T>, grid, dim3(kTileThreads), 0, s, xmap, a);
        if (e != cudaSuccess) return e;
    }
    if (!a.fused_state && (a.state_out != nullptr || (a.ckpt_every > 0 && a.ckpt != nullptr))) {
        const dim3 grid2((unsigned)a.n_seq, (nvec + kThreads - 1) / kThreads);
        const cudaError_t e = launch_pdl(conv1d_state_kernel<T>, grid2, blk, 0, s, a);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t read_and_clear_conv_error(cudaStream_t s, int* flags) {
    int hf = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&hf, g_conv_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    *flags = hf;
    if (hf != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_conv_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

cudaError_t launch_conv1d_fwd(const ConvArgs& a, gdn_dtype_t dt, cudaStream_t s) {
    return dt == GDN_BF16 ? conv_fwd_t<bf16>(a, s) : conv_fwd_t<float>(a, s);
}

cudaError_t launch_conv1d_state(const ConvArgs& a, gdn_dtype_t dt, cudaStream_t s) {
    if (a.T == 0 || (a.state_out == nullptr && (a.ckpt_every <= 0 || a.ckpt == nullptr))) return cudaSuccess;
    const int V = dt == GDN_BF16 ? 8 : 4;
    const dim3 grid((unsigned)a.n_seq, (unsigned)((a.C / V + kThreads - 1) / kThreads));
    const cudaError_t e = dt == GDN_BF16 ? launch_pdl(conv1d_state_kernel<bf16>, grid, dim3(kThreads), 0, s, a)
                                         : launch_pdl(conv1d_state_kernel<float>, grid, dim3(kThreads), 0, s, a);
    return e != cudaSuccess ? e : cudaGetLastError();
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
