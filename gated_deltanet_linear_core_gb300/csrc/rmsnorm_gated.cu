// RMSNormGated for the GDN layer core.
//
// cortex commit "feat(stage-8c): linear-attention layer (Qwen3-Next
// GatedDeltaNet)", "Output": RMSNormGated(core_attn_out, z), per value head:
//     out = w * o / sqrt(mean(o^2) + eps) * silu(z)
//
// HBM-bound (read o and z, write out: 6 bytes per bf16 element).  A group of
// D/V lanes owns one (token, head) row, each lane one 16-byte vector of o, z
// and out; the sum of squares is reduced with warp shuffles inside the group.
#include "gdn_common.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

template <typename T, int D>
__global__ void __launch_bounds__(256) rmsnorm_gated_kernel(const T* o,  // may alias out
                                                            const T* __restrict__ z,
                                                            const T* __restrict__ w, float eps,
                                                            int64_t rows, T* out) {
    pdl_wait();
    pdl_trigger();
    constexpr int V = Vec16<T>::N;
    constexpr int TPR = D / V;  // lanes per row
    static_assert(TPR >= 1 && TPR <= 32 && (32 % TPR) == 0, "row must fit a warp");
    constexpr int RPW = 32 / TPR;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t row = warp * RPW + lane / TPR;
    const int c0 = (lane % TPR) * V;
    const bool valid = row < rows;

    float ov[V], zv[V], wv[V];
    if (valid) {
        load16_stream(o + row * D + c0, ov);
        load16_stream(z + row * D + c0, zv);
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) ov[i] = zv[i] = 0.f;
    }
    load16(w + c0, wv);
    // channel pairs in packed f32x2 arithmetic
    float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < V; i += 2) {
        const float2 o2 = make_float2(ov[i], ov[i + 1]);
        ss2 = __ffma2_rn(o2, o2, ss2);
    }
    float ss = ss2.x + ss2.y;
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float rs = rsqrtf(ss / (float)D + eps);
    float res[V];
#pragma unroll
    for (int i = 0; i < V; i += 2) {
        const float2 g = silu2<T>(make_float2(zv[i], zv[i + 1]));
        const float2 r = __fmul2_rn(__fmul2_rn(make_float2(wv[i], wv[i + 1]),
                                               __fmul2_rn(make_float2(ov[i], ov[i + 1]), make_float2(rs, rs))),
                                    g);
        res[i] = r.x;
        res[i + 1] = r.y;
    }
    if (valid) store16(out + row * D + c0, res);
}

template <typename T>
cudaError_t norm_t(const void* o, const void* z, const void* w, float eps, int64_t T_, int H,
                   int D, void* out, cudaStream_t s) {
    const int64_t rows = T_ * H;
    if (rows == 0) return cudaSuccess;
    constexpr int V = Vec16<T>::N;
    const int64_t rows_per_block = (int64_t)(256 / 32) * (32 / (D / V));
    const unsigned grid = (unsigned)((rows + rows_per_block - 1) / rows_per_block);
    if (D == 128)
        return launch_pdl(rmsnorm_gated_kernel<T, 128>, dim3(grid), dim3(256), 0, s, (const T*)o, (const T*)z,
                          (const T*)w, eps, rows, (T*)out);
    return launch_pdl(rmsnorm_gated_kernel<T, 16>, dim3(grid), dim3(256), 0, s, (const T*)o, (const T*)z,
                      (const T*)w, eps, rows, (T*)out);
}

}  // namespace

cudaError_t launch_rmsnorm_gated(const void* o, const void* z, const void* w, float eps,
                                 int64_t T, int H, int D, void* out, gdn_dtype_t dt,
                                 cudaStream_t s) {
    return dt == GDN_BF16 ? norm_t<bf16>(o, z, w, eps, T, H, D, out, s)
                          : norm_t<float>(o, z, w, eps, T, H, D, out, s);
}

}  // namespace gdn
