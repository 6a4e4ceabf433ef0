// Chunked gated delta rule in two tcgen05 kernels.
//
// The result is that of the per-token rule of the cortex commit "feat(stage-8c):
// linear-attention layer (Qwen3-Next GatedDeltaNet)", "Delta rule (recurrent,
// per-token)", computed with the chunked algorithm (chunk_size=64) its
// "Performance note" names; NxD-Inference PR "Add Qwen3.6-27B hybrid
// DeltaNet/GQA contrib model and vLLM serving path": chunked context encoding,
// recurrent-state checkpoints, and the direct (not Neumann-style) solve.
//
// Of the per-chunk work only two products depend on the state S carried from
// chunk to chunk.  With G the chunk-local cumulative decay, rq / rk the
// l2-norm factors of raw q / k rows and T' = (I + A)^-1:
//   intra (independent per chunk, all chunks of all heads in parallel):
//     D1 = [K; Q] K^T,  A = beta rk e^{G_i-G_j} rk k.k (j<i),  P = rq e^{G_i-G_j} rk q.k (j<=i)
//     W^T = K^T (T' diag(beta e^G rk))^T,  U^T = V^T (T' diag(beta))^T
//     -> workspace: W (row-major), U^T, P (bf16) and e^G rq, e^{G_n-G_j} rk, e^{G_n} (f32)
//   chain (sequential per sequence and value head):
//     U'^T = U^T - S^T W^T;  O^T = (S^T Q^T) diag(e^G rq) + U'^T P^T
//     S^T <- e^{G_n} S^T + U'^T diag(e^{G_n-G_j} rk) K
// The chunks of a call are processed in segments (a range of chunk indices
// over all sequences) whose intermediates fit in the workspace and, at the
// default size, in L2; the state crosses segments through final_state (or a
// workspace carry).  Every wait is bounded (1 s); a CTA that gives up sets
// the device error word, lets its copies land, frees its TMEM and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "chunk_common.cuh"
#include "gdn_launch.h"

namespace gdn {

__device__ int g_device_error;  // bit 0: a bounded wait gave up

namespace {

using namespace tc;

constexpr int C = 64;
constexpr int D = 128;
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr size_t kSegBytes = 128ull << 20;  // workspace intermediates per segment

// per (chunk, value head) unit in the workspace
constexpr size_t U_WT = 16384, U_UT = 16384, U_P = 8192, U_VEC = 1024;
constexpr size_t UNIT_BYTES = U_WT + U_UT + U_P + U_VEC;

struct Layout {
    int64_t segc;    // chunks per segment
    int64_t n_seg;
    size_t off_wt, off_ut, off_p, off_vec, off_coff, off_carry, carry_bytes, total;
};

Layout layout_of(int n_seq, int64_t T, int H_v) {
    Layout L;
    const int64_t max_chunks = T / C + n_seq;
    int64_t segc = (int64_t)(kSegBytes / ((size_t)H_v * UNIT_BYTES));
    if (segc < 1) segc = 1;
    if (segc > max_chunks) segc = max_chunks;
    if (segc > 65535) segc = 65535;  // grid.y of the intra kernel
    L.segc = segc;
    L.n_seg = (max_chunks + segc - 1) / segc;
    const size_t U = (size_t)segc * H_v;
    L.off_wt = 0;
    L.off_ut = L.off_wt + U * U_WT;
    L.off_p = L.off_ut + U * U_UT;
    L.off_vec = L.off_p + U * U_P;
    L.off_coff = L.off_vec + U * U_VEC;
    L.off_carry = (L.off_coff + 4 * ((size_t)n_seq + 1) + 255) & ~(size_t)255;
    L.carry_bytes = L.n_seg > 1 ? (size_t)n_seq * H_v * D * D * 4 : 0;
    L.total = L.off_carry + L.carry_bytes;
    return L;
}

struct Work {
    bf16* wt;       // W, [U][64][128] (row i of W = 128 d-values)
    bf16* ut;       // [U][128][64]
    bf16* p;        // [U][64][64]
    float* vec;     // [U][256]: e^G rq (0..63), e^{G_n-G_j} rk (64..127), e^{G_n} (128)
    int32_t* coff;  // [n_seq + 1] chunk offsets
    float* carry;   // state between segments (final_state or workspace), may be null
};

// coff[i] = number of chunks of sequences 0..i-1 (one block, any n_seq)
__global__ void __launch_bounds__(1024) chunk_offsets_kernel(const int32_t* cu, int n_seq, int64_t T,
                                                             int32_t* coff) {
    __shared__ int32_t wsum[32];
    __shared__ int32_t base;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        base = 0;
        coff[0] = 0;
    }
    __syncthreads();
    for (int i0 = 0; i0 < n_seq; i0 += 1024) {
        const int i = i0 + tid;
        int v = 0;
        if (i < n_seq) {
            int64_t s, e;
            seq_bounds(cu, i, T, s, e);
            v = (int)((e - s + C - 1) / C);
        }
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        const int incl = x + (warp > 0 ? wsum[warp - 1] : 0);
        if (i < n_seq) coff[i + 1] = base + incl;
        __syncthreads();
        if (tid == 1023) base += incl;
        __syncthreads();
    }
}

// ============================================================== intra kernel
constexpr int NT_I = 256;
constexpr int IS_KQ = 0;                       // [cb0: K | Q][cb1: K | Q]; Q halves reused for B_W, B_U
constexpr int IS_V = IS_KQ + 32768;
constexpr int IS_A = IS_V + 16384;             // A, f32 [64][68]
constexpr int A_PITCH = 68;
constexpr int IS_F = IS_A + 64 * A_PITCH * 4;  // factor tables, then T' and block temporaries
constexpr int IS_VEC = IS_F + 32768;           // G, e^G, beta, dec, rk, rq, misc, fw
constexpr int IS_BAR = IS_VEC + 8 * 64 * 4;
constexpr int IS_TOTAL = IS_BAR + 64;
constexpr int ISMEM = IS_TOTAL + 1024;
constexpr uint32_t TI_D1 = 0, TI_DW = 64, TI_DU = 128, TI_COLS = 256;

__global__ void __launch_bounds__(NT_I, 2)
chunk_intra_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap wmap,
                   DeltaArgs a, Work w, int64_t C0) {
    const int h = blockIdx.x;
    const int64_t gc = C0 + blockIdx.y;
    const int n_seq = a.n_seq;
    if (gc >= w.coff[n_seq]) return;  // past the last chunk of the call
    int lo_s = 0, hi_s = n_seq - 1;   // sequence of chunk gc
    while (lo_s < hi_s) {
        const int mid = (lo_s + hi_s + 1) >> 1;
        if ((int64_t)w.coff[mid] <= gc) lo_s = mid; else hi_s = mid - 1;
    }
    const int seq = lo_s;
    const int64_t lc = gc - w.coff[seq];
    int64_t s0, s1;
    seq_bounds(a.cu, seq, a.T, s0, s1);
    const int64_t L = s1 - s0;
    const int64_t t0 = s0 + lc * C;
    const int n = (int)(L - lc * C < C ? L - lc * C : C);
    const int kh = h / (a.H_v / a.H_k);
    const int xq = kh * D, xk = a.H_k * D + kh * D, xv = 2 * a.H_k * D + h * D;
    const int64_t u = (gc - C0) * a.H_v + h;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* kq = sm + IS_KQ;
    uint8_t* vv = sm + IS_V;
    float* Gs = reinterpret_cast<float*>(sm + IS_VEC);
    float* eGs = Gs + 64;
    float* Bs = Gs + 128;
    float* DECs = Gs + 192;
    float* RKs = Gs + 256;
    float* RQs = Gs + 320;
    float* misc = Gs + 384;
    float* FWs = Gs + 448;
    float* Am = reinterpret_cast<float*>(sm + IS_A);
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + IS_BAR);
    uint64_t* bar_mma = bar_tma + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_tma + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lo = (uint32_t)(quarter * 32) << 16;
    constexpr float kLog2e = 1.4426950408889634f;

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_tma, 6 * 8192);
        const int y = (int)t0;
        tma_load_2d(kq, &qmap, bar_tma, xk, y);
        tma_load_2d(kq + 16384, &qmap, bar_tma, xk + 64, y);
        tma_load_2d(kq + 8192, &qmap, bar_tma, xq, y);
        tma_load_2d(kq + 24576, &qmap, bar_tma, xq + 64, y);
        tma_load_2d(vv, &qmap, bar_tma, xv, y);
        tma_load_2d(vv + 8192, &qmap, bar_tma, xv + 64, y);
    }
    if (warp == 0) {
        tmem_alloc(tslot, TI_COLS);
        tmem_relinquish();
    }
    // gates (log2 domain) and in-warp cumulative sums
    if (tid < 64) {
        float g = 0.f, bt = 0.f;
        if (tid < n) {
            const int64_t gi = (t0 + tid) * a.H_v + h;
            if (a.g != nullptr) {
                g = a.g[gi];
                bt = a.beta[gi];
            } else {
                g = gate_g(to_f(static_cast<const bf16*>(a.a)[gi]), a.A_log[h], a.dt_bias[h]);
                bt = sigmoid_f(to_f(static_cast<const bf16*>(a.b)[gi]));
            }
        }
        float x = g * kLog2e;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        Gs[tid] = x;
        Bs[tid] = bt;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *tslot;
    bool ok = __syncthreads_and(mbar_wait(bar_tma, 0, kWaitNs));
    bool mma_pending = false;
    uint32_t mma_phase = 0;
    if (ok) {
        if (tid >= 32 && tid < 64) Gs[tid] += Gs[31];
        {   // l2-norm factors: 128 rows (k then q) x 2 halves of 64 elements
            const int r = tid >> 1, hh = tid & 1, rr = r & 63;
            const bool isk = r < 64;
            const uint8_t* b0 = isk ? kq : kq + 8192;
            const uint8_t* b1 = isk ? kq + 16384 : kq + 24576;
            float ss = row_sumsq_part(b0, b1, rr, 2 * hh) + row_sumsq_part(b0, b1, rr, 2 * hh + 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            if (hh == 0) {
                float f = isk ? 1.f : a.scale;
                if (a.l2norm) f = f / sqrtf(ss + 1e-6f);
                (isk ? RKs : RQs)[rr] = f;
            }
        }
        __syncthreads();
        if (tid < 64) {
            const float Gn = Gs[n - 1];
            const float eg = exp2f(Gs[tid]);
            eGs[tid] = eg;
            FWs[tid] = Bs[tid] * eg * RKs[tid];
            DECs[tid] = tid < n ? exp2f(Gn - Gs[tid]) : 0.f;
            if (tid == 0) misc[0] = exp2f(Gn);
        }
        {   // decay-and-norm factor tables: thread t fills 16 entries of row t/4
            float* FA = reinterpret_cast<float*>(sm + IS_F);
            float* FP = FA + 64 * 64;
            const int i = tid >> 2, j0 = (tid & 3) * 16;
            const float Gi = Gs[i], fa = Bs[i] * RKs[i], fq = RQs[i];
            const bool live = i < n;
#pragma unroll
            for (int g4 = 0; g4 < 4; ++g4) {
                const int j = j0 + 4 * g4;
                const float4 G4 = *reinterpret_cast<const float4*>(Gs + j);
                const float4 R4 = *reinterpret_cast<const float4*>(RKs + j);
                const float gj[4] = {G4.x, G4.y, G4.z, G4.w}, rj[4] = {R4.x, R4.y, R4.z, R4.w};
                float va[4], vp[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float e = (live && j + q <= i) ? exp2f(fminf(Gi - gj[q], 0.f)) : 0.f;
                    vp[q] = fq * rj[q] * e;
                    va[q] = (j + q < i) ? fa * rj[q] * e : 0.f;
                }
                *reinterpret_cast<float4*>(FA + ftab(i, j)) = make_float4(va[0], va[1], va[2], va[3]);
                *reinterpret_cast<float4*>(FP + ftab(i, j)) = make_float4(vp[0], vp[1], vp[2], vp[3]);
            }
        }
        __syncthreads();
        // D1 = [K; Q] K^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t akq = smem_u32(kq);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                mma_bf16(tb + TI_D1, sdesc_sw128(akq + off, 16, 1024),
                         sdesc_sw128(akq + off, 16, 1024), idesc_bf16_f32(128, 64, 0, 0), k > 0);
            }
            mma_commit(bar_mma);
        }
        mma_pending = true;
        ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase, kWaitNs));
    }
    if (ok) {
        mma_phase ^= 1;
        mma_pending = false;
        tc_fence_after();
        {   // A (rows 0-63 -> shared, f32) and P (rows 64-127 -> workspace, bf16)
            float d1[32];
            tmem_ld32(tb + lo + TI_D1 + 32 * half, d1);
            tmem_wait_ld();
            const int i = row & 63;
            const float* F = reinterpret_cast<const float*>(sm + IS_F) + (row < 64 ? 0 : 64 * 64);
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4) {
                const float4 f = *reinterpret_cast<const float4*>(F + ftab(i, 32 * half + 4 * g4));
                d1[4 * g4 + 0] *= f.x;
                d1[4 * g4 + 1] *= f.y;
                d1[4 * g4 + 2] *= f.z;
                d1[4 * g4 + 3] *= f.w;
            }
            if (row < 64) {
#pragma unroll
                for (int g4 = 0; g4 < 8; ++g4)
                    *reinterpret_cast<float4*>(&Am[i * A_PITCH + 32 * half + 4 * g4]) =
                        make_float4(d1[4 * g4], d1[4 * g4 + 1], d1[4 * g4 + 2], d1[4 * g4 + 3]);
            } else {
                bf16* pp = w.p + u * (U_P / 2) + i * 64 + 32 * half;
#pragma unroll
                for (int g = 0; g < 4; ++g) store16(pp + 8 * g, d1 + 8 * g);
            }
        }
        __syncthreads();
        {   // T' = (I + A)^-1 blocked by 16 (see the fused kernel's derivation)
            float* Tm = reinterpret_cast<float*>(sm + IS_F);
            float* Mt = Tm + 64 * A_PITCH;
            if (tid < 64) {
                const int r0 = (tid >> 4) * 16, cl = tid & 15;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const float* Ar = &Am[(r0 + r) * A_PITCH + r0];
                    float acc = (r == cl) ? 1.f : 0.f;
#pragma unroll
                    for (int q = 0; q < r; ++q) acc = fmaf(-Ar[q], x[q], acc);
                    x[r] = acc;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Tm[(r0 + r) * A_PITCH + r0 + cl] = x[r];
            } else {
                for (int e = tid - 64; e < 6 * 256; e += NT_I - 64) {
                    const int blk = e >> 8, r = (e >> 4) & 15, cc = e & 15;
                    const int br = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
                    const int bc = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
                    Tm[(br * 16 + r) * A_PITCH + bc * 16 + cc] = 0.f;
                }
            }
            __syncthreads();
            for (int dd = 1; dd < 4; ++dd) {
                const int nstrip = (4 - dd) * 64;
                if (tid < nstrip) {
                    const int bl = tid >> 6, r = (tid >> 2) & 15, q4 = (tid & 3) * 4;
                    const float* Ar = &Am[((bl + dd) * 16 + r) * A_PITCH];
                    const float* Tc = &Tm[bl * 16 + q4];
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int k = bl * 16; k < (bl + dd) * 16; k += 4) {
                        const float4 a4 = *reinterpret_cast<const float4*>(Ar + k);
                        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 t4 = *reinterpret_cast<const float4*>(Tc + (k + q) * A_PITCH);
                            acc.x = fmaf(av[q], t4.x, acc.x);
                            acc.y = fmaf(av[q], t4.y, acc.y);
                            acc.z = fmaf(av[q], t4.z, acc.z);
                            acc.w = fmaf(av[q], t4.w, acc.w);
                        }
                    }
                    *reinterpret_cast<float4*>(&Mt[(bl << 8) + r * 16 + q4]) = acc;
                }
                __syncthreads();
                if (tid < nstrip) {
                    const int bl = tid >> 6, r = (tid >> 2) & 15, q4 = (tid & 3) * 4;
                    const int a0 = (bl + dd) * 16;
                    const float* Ta = &Tm[(a0 + r) * A_PITCH + a0];
                    const float* Mb = &Mt[(bl << 8) + q4];
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < 16; k += 4) {
                        const float4 a4 = *reinterpret_cast<const float4*>(Ta + k);
                        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 m4 = *reinterpret_cast<const float4*>(Mb + (k + q) * 16);
                            acc.x = fmaf(av[q], m4.x, acc.x);
                            acc.y = fmaf(av[q], m4.y, acc.y);
                            acc.z = fmaf(av[q], m4.z, acc.z);
                            acc.w = fmaf(av[q], m4.w, acc.w);
                        }
                    }
                    *reinterpret_cast<float4*>(&Tm[(a0 + r) * A_PITCH + bl * 16 + q4]) =
                        make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
                }
                __syncthreads();
            }
            // B_W = T' diag(beta e^G rk), B_U = T' diag(beta) into the (consumed) Q halves
            {
                const int which = tid >> 7, i = (tid >> 1) & 63, c0 = (tid & 1) * 32;
                const float* Ti = &Tm[i * A_PITCH + c0];
                const float* Fc = (which == 0 ? FWs : Bs) + c0;
                float vals[32];
#pragma unroll
                for (int g4 = 0; g4 < 8; ++g4) {
                    const float4 t4 = *reinterpret_cast<const float4*>(Ti + 4 * g4);
                    const float4 f4 = *reinterpret_cast<const float4*>(Fc + 4 * g4);
                    vals[4 * g4 + 0] = t4.x * f4.x;
                    vals[4 * g4 + 1] = t4.y * f4.y;
                    vals[4 * g4 + 2] = t4.z * f4.z;
                    vals[4 * g4 + 3] = t4.w * f4.w;
                }
                store_row_bf16(kq + (which == 0 ? 8192 : 24576), i, c0, vals, 32);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // W^T = K^T B_W^T,  U^T = V^T B_U^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t akq = smem_u32(kq), av = smem_u32(vv);
            const uint32_t bw = smem_u32(kq + 8192), bu = smem_u32(kq + 24576);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mma_bf16(tb + TI_DW, sdesc_sw128(akq + k * 2048, 16384, 1024),
                         sdesc_sw128(bw + k * 32, 16, 1024), idesc_bf16_f32(128, 64, 1, 0), k > 0);
                mma_bf16(tb + TI_DU, sdesc_sw128(av + k * 2048, 8192, 1024),
                         sdesc_sw128(bu + k * 32, 16, 1024), idesc_bf16_f32(128, 64, 1, 0), k > 0);
            }
            mma_commit(bar_mma);
        }
        mma_pending = true;
        ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase, kWaitNs));
    }
    if (ok) {
        mma_pending = false;
        tc_fence_after();
        {   // W (row-major, staged 128B-swizzled in the consumed V tile, stored by TMA)
            // and U^T rows (bf16, 32 columns per thread)
            float v32[32];
            tmem_ld32(tb + lo + TI_DW + 32 * half, v32);
            tmem_wait_ld();
            uint8_t* stg = vv + (row >> 6) * 8192;
            const int dc = row & 63;
#pragma unroll
            for (int q = 0; q < 32; ++q)
                *reinterpret_cast<bf16*>(stg + sw128_off(32 * half + q, dc)) = __float2bfloat16_rn(v32[q]);
            tmem_ld32(tb + lo + TI_DU + 32 * half, v32);
            tmem_wait_ld();
            bf16* dst = w.ut + u * (U_UT / 2) + row * 64 + 32 * half;
#pragma unroll
            for (int g = 0; g < 4; ++g) store16(dst + 8 * g, v32 + 8 * g);
            fence_async_smem();
        }
        if (tid < 64) {
            float* vec = w.vec + u * (U_VEC / 4);
            vec[tid] = eGs[tid] * RQs[tid];
            vec[64 + tid] = DECs[tid] * RKs[tid];
            if (tid == 0) vec[128] = misc[0];
        }
    } else if (tid == 0) {
        atomicOr(&g_device_error, 1);
        if (mma_pending) mbar_wait(bar_mma, mma_phase, kWaitNs);
        mbar_wait(bar_tma, 0, kWaitNs);
    }
    tc_fence_before();
    __syncthreads();
    if (ok && tid == 0) {
        tma_store_2d(&wmap, vv, 0, (int)(u * 64));
        tma_store_2d(&wmap, vv + 8192, 64, (int)(u * 64));
        bulk_commit();
        bulk_wait_all();
    }
    if (warp == 0) tmem_dealloc(tb, TI_COLS);
}

// ============================================================== chain kernel
constexpr int NT_C = 512;
constexpr int CS_ST = 0;                           // S^T bf16 [v][d], 2 blocks of 16 KB
constexpr int STAGE = 74752;  // [W|Q] 32K (per 64-column block: W rows, Q rows) | UT 16K | P 8K | K 16K | vec 1K
constexpr int CS_STAGE = CS_ST + 32768;
constexpr int SG_WQ = 0, SG_UT = 32768, SG_P = 49152, SG_K = 57344, SG_VEC = 73728;
constexpr int CS_UTC = CS_STAGE + 2 * STAGE;       // U'^T bf16 (then the O staging tile)
constexpr int CS_UTD = CS_UTC + 16384;             // U'^T diag(e^{G_n-G_j} rk)
constexpr int CS_BAR = CS_UTD + 16384;
constexpr int CS_TOTAL = CS_BAR + 64;
constexpr int CSMEM = CS_TOTAL + 1024;
static_assert(CSMEM <= 232448, "chain kernel shared memory");
// TMEM: the chunk's state increment, two buffers of [(W S)^T | (Q S)^T] and two
// of U'^T P^T.  The f32 state itself lives in registers: thread (v, cg) holds
// S[d][v] for d in [32 cg, 32 cg + 32).
constexpr uint32_t TC_DS = 0, TC_WQS = 128, TC_O = 384, TC_COLS = 512;

// Per chunk: MMA(S^T W^T, S^T Q^T) -> U' -> MMA(state update, U'^T P^T) -> state
// read-back (bf16 operand for the next chunk, the next chunk's decay applied in
// TMEM) -> the next chunk's first MMAs are issued -> this chunk's O epilogue
// runs while they execute.
__global__ void __launch_bounds__(NT_C, 1)
chunk_chain_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                   const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap utmap,
                   const __grid_constant__ CUtensorMap pmap, DeltaArgs a, Work w, int64_t C0,
                   int64_t segc) {
    const int h = blockIdx.x % a.H_v;
    const int seq = blockIdx.x / a.H_v;
    const int64_t cs = w.coff[seq], ce = w.coff[seq + 1];
    const int64_t c_lo = cs > C0 ? cs : C0, c_hi = ce < C0 + segc ? ce : C0 + segc;
    const int64_t sbase = ((int64_t)seq * a.H_v + h) * D * D;
    const int tid = threadIdx.x, warp = tid >> 5;
    if (c_lo >= c_hi) {
        // no chunk of this sequence in this segment; an empty sequence's final
        // state is its initial state (written once, by the first segment)
        if (cs == ce && C0 == 0 && a.S_final != nullptr && a.S_final != a.S0)
            for (int e = tid; e < D * D; e += NT_C)
                a.S_final[sbase + e] = a.S0 != nullptr ? a.S0[sbase + e] : 0.f;
        return;
    }
    const int quarter = warp & 3, cg = warp >> 2;
    const int row = quarter * 32 + (tid & 31);
    const uint32_t lo = (uint32_t)(quarter * 32) << 16;
    const int kh = h / (a.H_v / a.H_k);
    const int xq = kh * D, xk = a.H_k * D + kh * D;
    int64_t s0, s1;
    seq_bounds(a.cu, seq, a.T, s0, s1);
    const int64_t L = s1 - s0;
    int64_t ck_row0 = 0;
    if (a.ckpt_every > 0 && a.ckpt != nullptr) ck_row0 = ckpt_row0(a.cu, seq, a.T, a.ckpt_every);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + CS_BAR);  // [0], [1]
    uint64_t* bar_mma = bar_tma + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_tma + 3);

    if (tid == 0) {
        mbar_init(&bar_tma[0], 1);
        mbar_init(&bar_tma[1], 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, TC_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *tslot;

    int issued0 = 0, issued1 = 0, consumed0 = 0, consumed1 = 0;
    auto issue = [&](int64_t gcc) {
        const int b = (int)((gcc - c_lo) & 1);
        uint8_t* st = sm + CS_STAGE + b * STAGE;
        const int y = (int)(s0 + (gcc - cs) * C);
        const int64_t uu = (gcc - C0) * a.H_v + h;
        mbar_arrive_expect_tx(&bar_tma[b], STAGE);
        tma_load_2d(st + SG_WQ, &wmap, &bar_tma[b], 0, (int)(uu * 64));
        tma_load_2d(st + SG_WQ + 16384, &wmap, &bar_tma[b], 64, (int)(uu * 64));
        tma_load_2d(st + SG_WQ + 8192, &qmap, &bar_tma[b], xq, y);
        tma_load_2d(st + SG_WQ + 24576, &qmap, &bar_tma[b], xq + 64, y);
        tma_load_2d(st + SG_UT, &utmap, &bar_tma[b], 0, (int)(uu * 128));
        tma_load_2d(st + SG_P, &pmap, &bar_tma[b], 0, (int)(uu * 64));
        tma_load_2d(st + SG_K, &qmap, &bar_tma[b], xk, y);
        tma_load_2d(st + SG_K + 8192, &qmap, &bar_tma[b], xk + 64, y);
        bulk_load(st + SG_VEC, w.vec + uu * (int64_t)(U_VEC / 4), (uint32_t)U_VEC, &bar_tma[b]);
        if (b) ++issued1; else ++issued0;
    };
    auto wait_stage = [&](int64_t gcc) -> bool {  // every thread, in chunk order
        const int b = (int)((gcc - c_lo) & 1);
        const bool r = mbar_wait(&bar_tma[b], (uint32_t)((b ? consumed1 : consumed0) & 1), kWaitNs);
        if (r) {
            if (b) ++consumed1; else ++consumed0;
        }
        return r;
    };
    auto issue_mma45 = [&](int64_t gcc) {  // thread 0: [(W S)^T | (Q S)^T] of chunk gcc, one N=128 MMA
        const int b = (int)((gcc - c_lo) & 1);
        uint8_t* st = sm + CS_STAGE + b * STAGE;
        tc_fence_after();
        const uint32_t ast = smem_u32(sm + CS_ST), bwq = smem_u32(st + SG_WQ);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
            mma_bf16(tb + TC_WQS + 128 * b, sdesc_sw128(ast + off, 16, 1024),
                     sdesc_sw128(bwq + off, 16, 1024), idesc_bf16_f32(128, 128, 0, 0), k > 0);
        }
        mma_commit(bar_mma);
    };
    if (tid == 0) {
        issue(c_lo);
        if (c_lo + 1 < c_hi) issue(c_lo + 1);
    }

    // initial state of this segment: the sequence's initial state at its first
    // chunk, else what the previous segment left in the carry
    float sv[32];
    {
        const float* src = (c_lo == cs) ? a.S0 : w.carry;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            sv[j] = src != nullptr ? src[sbase + (int64_t)(32 * cg + j) * D + row] : 0.f;
        store_row_bf16(sm + CS_ST + (cg >> 1) * 16384, row, (cg & 1) * 32, sv, 32);
    }
    bool ok = __syncthreads_and(wait_stage(c_lo));
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    uint32_t mma_phase = 0;
    bool mma_pending = false;
    if (ok && tid == 0) issue_mma45(c_lo);
    mma_pending = ok;

    for (int64_t gcc = c_lo; ok && gcc < c_hi; ++gcc) {
        const int b = (int)((gcc - c_lo) & 1);
        uint8_t* st = sm + CS_STAGE + b * STAGE;
        const float* vs = reinterpret_cast<const float*>(st + SG_VEC);
        const int64_t lc = gcc - cs;
        const int64_t t0 = s0 + lc * C;
        const int n = (int)(L - lc * C < C ? L - lc * C : C);
        const int i0 = 16 * cg;

        if (tid == 0) bulk_wait_read_all();  // the previous O tile store has left U'^T's buffer
        ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase, kWaitNs));
        if (!ok) break;
        mma_phase ^= 1;
        mma_pending = false;
        tc_fence_after();

        // U'^T = U^T - (W S)^T (bf16, and scaled by e^{G_n-G_j} rk_j)
        float erq[16];  // e^{G_i} rq_i of this thread's O rows (the stage is reloaded below)
        const float eGn = vs[128];
        {
            const int j0 = 16 * cg;
            float ws[16], ui[16];
            tmem_ld16(tb + lo + TC_WQS + 128 * b + j0, ws);
            const uint8_t* urow = st + SG_UT;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                float t8[8];
                load16(reinterpret_cast<const bf16*>(urow + sw128_off(row, j0 + 8 * g)), t8);
#pragma unroll
                for (int e = 0; e < 8; ++e) ui[8 * g + e] = t8[e];
            }
#pragma unroll
            for (int q = 0; q < 16; ++q) erq[q] = vs[i0 + q];
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) ui[j] -= ws[j];
            store_row_bf16(sm + CS_UTC, row, j0, ui, 16);
#pragma unroll
            for (int j = 0; j < 16; ++j) ws[j] = ui[j] * vs[64 + j0 + j];
            store_row_bf16(sm + CS_UTD, row, j0, ws, 16);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // dS^T = U'^T_dec K  (M = v, N = d, K = j);  O_P^T = U'^T P^T  (N = i)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t autd = smem_u32(sm + CS_UTD), aut = smem_u32(sm + CS_UTC);
            const uint32_t bk = smem_u32(st + SG_K), bp = smem_u32(st + SG_P);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mma_bf16(tb + TC_DS, sdesc_sw128(autd + k * 32, 16, 1024),
                         sdesc_sw128(bk + k * 2048, 8192, 1024), idesc_bf16_f32(128, 128, 0, 1), k > 0);
                mma_bf16(tb + TC_O + 64 * b, sdesc_sw128(aut + k * 32, 16, 1024),
                         sdesc_sw128(bp + k * 32, 16, 1024), idesc_bf16_f32(128, 64, 0, 0), k > 0);
            }
            mma_commit(bar_mma);
        }
        mma_pending = true;
        ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase, kWaitNs));
        if (!ok) break;
        mma_phase ^= 1;
        mma_pending = false;
        tc_fence_after();
        if (tid == 0 && gcc + 2 < c_hi) issue(gcc + 2);  // this chunk's stage is consumed

        // S <- e^{G_n} S + dS (registers) -> bf16 S^T operand (and checkpoint)
        const bool more = gcc + 1 < c_hi;
        bool landed = true;
        {
            const int64_t done = lc * C + n;
            float* ck = nullptr;
            if (a.ckpt_every > 0 && a.ckpt != nullptr && done % a.ckpt_every == 0) {
                const int64_t crow = ck_row0 + done / a.ckpt_every - 1;
                if (crow < a.ckpt_rows) ck = a.ckpt + (crow * a.H_v + h) * D * D;
            }
            float ds[32];
            tmem_ld32(tb + lo + TC_DS + 32 * cg, ds);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) sv[j] = fmaf(eGn, sv[j], ds[j]);
            store_row_bf16(sm + CS_ST + (cg >> 1) * 16384, row, (cg & 1) * 32, sv, 32);
            if (ck != nullptr)
#pragma unroll
                for (int j = 0; j < 32; ++j) ck[(int64_t)(32 * cg + j) * D + row] = sv[j];
            if (more) landed = wait_stage(gcc + 1);
        }
        fence_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(landed);
        if (!ok) break;
        if (more && tid == 0) issue_mma45(gcc + 1);
        mma_pending = more;

        // O = (Q S) diag(e^G rq) + P U' of this chunk, while the next chunk's MMAs run
        {
            tc_fence_after();
            float qs[16], po[16];
            tmem_ld16(tb + lo + TC_WQS + 128 * b + 64 + i0, qs);
            tmem_ld16(tb + lo + TC_O + 64 * b + i0, po);
            tmem_wait_ld();
            if (n == C) {
                uint8_t* stg = sm + CS_UTC + (row >> 6) * 8192;
                const int cc = row & 63;
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    *reinterpret_cast<bf16*>(stg + sw128_off(i0 + q, cc)) =
                        __float2bfloat16_rn(erq[q] * qs[q] + po[q]);
                fence_async_smem();
                __syncthreads();
                if (tid == 0) {
                    tma_store_2d(&omap, sm + CS_UTC, h * D, (int)t0);
                    tma_store_2d(&omap, sm + CS_UTC + 8192, h * D + 64, (int)t0);
                    bulk_commit();
                }
            } else {
                bf16* o = static_cast<bf16*>(a.o) + (t0 * a.H_v + h) * D + row;
                const int64_t ostride = (int64_t)a.H_v * D;
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    if (i0 + q < n) o[(i0 + q) * ostride] = __float2bfloat16_rn(erq[q] * qs[q] + po[q]);
            }
        }
        tc_fence_before();
        __syncthreads();
    }

    if (ok) {
        float* dst = a.S_final != nullptr ? a.S_final : w.carry;
        if (dst != nullptr)
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[sbase + (int64_t)(32 * cg + j) * D + row] = sv[j];
    } else if (tid == 0) {
        atomicOr(&g_device_error, 1);
        if (mma_pending) mbar_wait(bar_mma, mma_phase, kWaitNs);
        for (int k = consumed0; k < issued0; ++k) mbar_wait(&bar_tma[0], (uint32_t)(k & 1), kWaitNs);
        for (int k = consumed1; k < issued1; ++k) mbar_wait(&bar_tma[1], (uint32_t)(k & 1), kWaitNs);
    }
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, TC_COLS);
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensormap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

namespace {

bool encode2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensormap_encoder();
    if (enc == nullptr) return false;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstr[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstr, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t chunk_split_workspace_bytes(int n_seq, int64_t T, int H_v) {
    return layout_of(n_seq, T, H_v).total;
}

cudaError_t launch_chunk_split(const DeltaArgs& a, void* workspace, size_t ws_bytes, cudaStream_t s) {
    const Layout Ly = layout_of(a.n_seq, a.T, a.H_v);
    if (workspace == nullptr || ws_bytes < Ly.total) return cudaErrorInvalidValue;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    Work w;
    w.wt = reinterpret_cast<bf16*>(ws + Ly.off_wt);
    w.ut = reinterpret_cast<bf16*>(ws + Ly.off_ut);
    w.p = reinterpret_cast<bf16*>(ws + Ly.off_p);
    w.vec = reinterpret_cast<float*>(ws + Ly.off_vec);
    w.coff = reinterpret_cast<int32_t*>(ws + Ly.off_coff);
    w.carry = Ly.carry_bytes ? reinterpret_cast<float*>(ws + Ly.off_carry) : nullptr;
    if (a.S_final != nullptr) w.carry = a.S_final;

    const uint64_t conv_dim = 2ull * a.H_k * D + (uint64_t)a.H_v * D;
    const uint64_t U = (uint64_t)Ly.segc * a.H_v;
    CUtensorMap qmap, omap, wtmap, utmap, pmap;
    if (!encode2d(&qmap, a.qkv, conv_dim, (uint64_t)a.T, 64, 64) ||
        !encode2d(&omap, a.o, (uint64_t)a.H_v * D, (uint64_t)a.T, 64, 64) ||
        !encode2d(&wtmap, w.wt, 128, U * 64, 64, 64) || !encode2d(&utmap, w.ut, 64, U * 128, 64, 128) ||
        !encode2d(&pmap, w.p, 64, U * 64, 64, 64))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(chunk_intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ISMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(chunk_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, CSMEM);
    if (e != cudaSuccess) return e;

    chunk_offsets_kernel<<<1, 1024, 0, s>>>(a.cu, a.n_seq, a.T, w.coff);
    for (int64_t seg = 0; seg < Ly.n_seg; ++seg) {
        const int64_t C0 = seg * Ly.segc;
        chunk_intra_kernel<<<dim3((unsigned)a.H_v, (unsigned)Ly.segc), NT_I, ISMEM, s>>>(qmap, wtmap, a, w, C0);
        chunk_chain_kernel<<<(unsigned)(a.n_seq * a.H_v), NT_C, CSMEM, s>>>(qmap, omap, wtmap, utmap,
                                                                          pmap, a, w, C0, Ly.segc);
    }
    return cudaGetLastError();
}

cudaError_t read_and_clear_device_error(cudaStream_t s, int* flags) {
    int hf = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&hf, g_device_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    *flags = hf;
    if (hf != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

}  // namespace gdn

// ===================================================================== no-allocation variant
// gdn_chunk_prefill_noalloc runs the same two kernels with their scratch in a
// fixed array that is part of the library image, for callers that cannot
// allocate device memory.  Smaller segments than the workspace variant (the
// array is 24 MiB) mean more launches; the arithmetic is the same.
namespace gdn {

namespace {

constexpr size_t kStaticScratchBytes = 24ull << 20;
constexpr int kStaticMaxSeq = 16384;

static __device__ __align__(256) uint8_t g_prefill_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[128];  // device address of g_prefill_scratch, per device ordinal

}  // namespace

bool chunk_split_static_fits(int n_seq, int H_v) {
    const size_t coff_bytes = ((size_t)4 * (kStaticMaxSeq + 1) + 255) & ~(size_t)255;
    return n_seq >= 1 && n_seq <= kStaticMaxSeq &&
           (size_t)H_v * UNIT_BYTES <= kStaticScratchBytes - coff_bytes;
}

cudaError_t launch_chunk_split_static(const DeltaArgs& a, cudaStream_t s) {
    if (!chunk_split_static_fits(a.n_seq, a.H_v) || a.S_final == nullptr) return cudaErrorInvalidValue;
    // set-up once per device, with that device current: the host-side name of
    // the array is not a device address
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    uint8_t* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (g_scratch_ptr[dev] == nullptr) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_prefill_scratch);
            if (e != cudaSuccess) return e;
            g_scratch_ptr[dev] = p;
        }
        base = static_cast<uint8_t*>(g_scratch_ptr[dev]);
    }
    // layout inside the fixed array: chunk offsets, then as many chunks per
    // segment as fit; final_state carries the state between segments
    const size_t coff_bytes = ((size_t)4 * (kStaticMaxSeq + 1) + 255) & ~(size_t)255;
    const int64_t max_chunks = a.T / C + a.n_seq;
    int64_t segc = (int64_t)((kStaticScratchBytes - coff_bytes) / ((size_t)a.H_v * UNIT_BYTES));
    if (segc > max_chunks) segc = max_chunks;
    if (segc > 65535) segc = 65535;
    const int64_t n_seg = (max_chunks + segc - 1) / segc;
    const size_t U = (size_t)segc * a.H_v;
    Work w;
    w.coff = reinterpret_cast<int32_t*>(base);
    w.wt = reinterpret_cast<bf16*>(base + coff_bytes);
    w.ut = reinterpret_cast<bf16*>(base + coff_bytes + U * U_WT);
    w.p = reinterpret_cast<bf16*>(base + coff_bytes + U * (U_WT + U_UT));
    w.vec = reinterpret_cast<float*>(base + coff_bytes + U * (U_WT + U_UT + U_P));
    w.carry = a.S_final;

    const uint64_t conv_dim = 2ull * a.H_k * D + (uint64_t)a.H_v * D;
    CUtensorMap qmap, omap, wtmap, utmap, pmap;
    if (!encode2d(&qmap, a.qkv, conv_dim, (uint64_t)a.T, 64, 64) ||
        !encode2d(&omap, a.o, (uint64_t)a.H_v * D, (uint64_t)a.T, 64, 64) ||
        !encode2d(&wtmap, w.wt, 128, U * 64, 64, 64) || !encode2d(&utmap, w.ut, 64, U * 128, 64, 128) ||
        !encode2d(&pmap, w.p, 64, U * 64, 64, 64))
        return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(chunk_intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ISMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(chunk_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, CSMEM);
    if (e != cudaSuccess) return e;
    chunk_offsets_kernel<<<1, 1024, 0, s>>>(a.cu, a.n_seq, a.T, w.coff);
    for (int64_t seg = 0; seg < n_seg; ++seg) {
        const int64_t C0 = seg * segc;
        chunk_intra_kernel<<<dim3((unsigned)a.H_v, (unsigned)segc), NT_I, ISMEM, s>>>(qmap, wtmap, a, w, C0);
        chunk_chain_kernel<<<(unsigned)(a.n_seq * a.H_v), NT_C, CSMEM, s>>>(qmap, omap, wtmap, utmap,
                                                                          pmap, a, w, C0, segc);
    }
    return cudaGetLastError();
}

}  // namespace gdn
