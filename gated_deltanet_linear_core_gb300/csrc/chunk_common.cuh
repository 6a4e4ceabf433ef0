// Device helpers shared by the tensor-core chunked-prefill kernels.
#pragma once

#include <cuda_fp16.h>

#include "gdn_common.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace tc {

// The tensor-core operands the kernels form themselves (W, U, P, the state S,
// U') are fp16: 11 significant bits against bf16's 8, the same MMA rate.
// bf16 activations (q, k, v) are converted to fp16 in shared memory where
// they meet those operands in one product (exact for |x| in [2^-14, 65504]).
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Eight fp16 values of one 16-byte vector as f32.
__device__ __forceinline__ void unpack8_h(uint4 u, float* out) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        out[2 * i] = f.x;
        out[2 * i + 1] = f.y;
    }
}

// Eight bf16 values of one 16-byte vector re-encoded as fp16.
__device__ __forceinline__ uint4 bf16x8_to_h(uint4 u) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = pack_h2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// Re-encodes `bytes` (a multiple of 16 * nthreads) of bf16 at p as fp16 in
// place, thread t of nthreads taking every nthreads-th 16-byte vector.
__device__ __forceinline__ void bf16_to_h_inplace(uint8_t* p, int bytes, int t, int nthreads) {
    uint4* v = reinterpret_cast<uint4*>(p);
    for (int e = t; e < bytes / 16; e += nthreads) v[e] = bf16x8_to_h(v[e]);
}

// Writes n (multiple of 8) floats as fp16 into row `row` of a 128-byte-row
// swizzled block, starting at column c0 (multiple of 8, c0 + n <= 64).
__device__ __forceinline__ void store_row_h(uint8_t* blk, int row, int c0, const float* v, int n) {
#pragma unroll
    for (int g = 0; g < n / 8; ++g) {
        uint4 u;
        u.x = pack_h2(v[8 * g + 0], v[8 * g + 1]);
        u.y = pack_h2(v[8 * g + 2], v[8 * g + 3]);
        u.z = pack_h2(v[8 * g + 4], v[8 * g + 5]);
        u.w = pack_h2(v[8 * g + 6], v[8 * g + 7]);
        *reinterpret_cast<uint4*>(blk + sw128_off(row, c0 + 8 * g)) = u;
    }
}

// Writes n (multiple of 8) floats as bf16 into row `row` of a 128-byte-row
// swizzled block, starting at column c0 (multiple of 8, c0 + n <= 64).
__device__ __forceinline__ void store_row_bf16(uint8_t* blk, int row, int c0, const float* v,
                                               int n) {
#pragma unroll
    for (int g = 0; g < n / 8; ++g) {
        uint4 u;
        u.x = pack_bf16x2(v[8 * g + 0], v[8 * g + 1]);
        u.y = pack_bf16x2(v[8 * g + 2], v[8 * g + 3]);
        u.z = pack_bf16x2(v[8 * g + 4], v[8 * g + 5]);
        u.w = pack_bf16x2(v[8 * g + 6], v[8 * g + 7]);
        *reinterpret_cast<uint4*>(blk + sw128_off(row, c0 + 8 * g)) = u;
    }
}

// Sum of squares of 32 elements (four 16-byte chunks) of a 128-element bf16
// row stored as two 128-byte swizzled rows; part p (0..3) covers chunks
// 4(p&1)..4(p&1)+3 of block p>>1, visited in a bank-conflict-free order.
__device__ __forceinline__ float row_sumsq_part(const uint8_t* blk0, const uint8_t* blk1, int row,
                                                int part) {
    const uint4* p = reinterpret_cast<const uint4*>(((part >> 1) ? blk1 : blk0) + row * 128);
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int chunk = ((part & 1) * 4 + ((q + (part >> 1) * 2) & 3)) ^ (row & 7);
        const uint4 u = p[chunk];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
            s = fmaf(lo, lo, s);
            s = fmaf(hi, hi, s);
        }
    }
    return s;
}

}  // namespace tc
}  // namespace gdn
