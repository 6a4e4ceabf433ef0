// Device helpers shared by the tensor-core chunked-prefill kernels.
#pragma once

#include "gdn_common.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace tc {

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
