// Chunked gated delta rule on tcgen05 tensor cores: bf16 operands in shared
// memory, f32 accumulators and the f32 recurrent state in tensor memory (TMEM).
//
// The result is that of the per-token rule of the cortex commit "feat(stage-8c):
// linear-attention layer (Qwen3-Next GatedDeltaNet)", "Delta rule (recurrent,
// per-token)", computed with the chunked algorithm its "Performance note" names
// (chunk_size=64, same surface).  NxD-Inference PR "Add Qwen3.6-27B hybrid
// DeltaNet/GQA contrib model and vLLM serving path": chunked context encoding,
// recurrent-state checkpoints; its "Known limitations" contrast a stable
// direct-solve path with a Neumann-style one -- the triangular system here is
// solved directly (forward substitution in f32).
//
// Per chunk of n <= 64 tokens, with G the chunk-local cumulative decay, raw
// q, k rows and their l2-norm factors rq (scale included) and rk:
//   D1 = [K; Q] K^T                      (one M=128 MMA: k.k and q.k)
//   A_ij = beta_i e^{G_i-G_j} rk_i rk_j k_i.k_j  (j < i)
//   P_ij = e^{G_i-G_j} rq_i rk_j q_i.k_j         (j <= i)
//   T' = (I + A)^-1                      (CUDA cores, f32)
//   W^T = K^T (T' diag(beta e^G rk))^T,  U^T = V^T (T' diag(beta))^T
//   U'^T = U^T - S^T W^T
//   O^T = diag-scaled (S^T Q^T) + U'^T P^T
//   S^T <- e^{G_n} S^T + (U'^T diag(e^{G_n-G_j} rk_j)) K
// The value dimension (128) sits on the TMEM lanes for every product, so each
// MMA is M=128 and thread v of the 128-thread CTA owns state column v.
// Operands K, Q, V come straight from global memory by TMA in the 128-byte
// swizzled layout and are read K-major or MN-major as each product needs; the
// computed operands (P, T' factors, W^T, U'^T, S^T) are written by the threads
// that own their rows.  Every exponent is G_i - G_j with i >= j or G itself
// (<= 0), so nothing overflows.
//
// One CTA per (sequence, value head); sequential over the sequence's chunks,
// with the next chunk's tiles prefetched by TMA.  Every wait is bounded
// (1 s); a CTA that gives up sets the library's device error word, waits
// (bounded) for its copies in flight, frees its TMEM and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_common.cuh"
#include "gdn_launch.h"
#include "tc_ptx.cuh"

namespace gdn {

__device__ int g_device_error;  // bit 0: a bounded wait gave up

namespace {

using namespace tc;

constexpr int C = 64;
constexpr int D = 128;
constexpr int NT = 128;
constexpr uint64_t kWaitNs = 1000000000ull;

// shared memory map, byte offsets from a 1024-aligned base
constexpr int KQ_BYTES = 32768;  // [cb0: K rows 0-63 | Q rows 0-63][cb1: K | Q], cb = 64 d-columns
constexpr int V_BYTES = 16384;   // [cb0: 64 rows][cb1: 64 rows]
constexpr int SM_KQ = 0;
constexpr int SM_V = SM_KQ + 2 * KQ_BYTES;
constexpr int SM_P = SM_V + 2 * V_BYTES;  // P [i][j]        K-major B operand
constexpr int SM_BW = SM_P + 8192;        // T' * beta e^G rk  [i][j]
constexpr int SM_BU = SM_BW + 8192;       // T' * beta         [i][j]
constexpr int SM_WT = SM_BU + 8192;       // W^T [d][i]       MN-major B operand
constexpr int SM_ST = SM_WT + 16384;      // S^T [v][d] bf16  K-major A operand (2 blocks)
constexpr int SM_UT = SM_ST + 32768;      // U'^T [v][j]      K-major A operand
constexpr int SM_UTD = SM_UT + 16384;     // U'^T diag(e^{G_n-G_j} rk_j)
constexpr int SM_A = SM_UTD + 16384;      // A matrix, f32
constexpr int A_PITCH = 68;
constexpr int SM_VEC = SM_A + 64 * A_PITCH * 4;  // G, e^G, beta, dec, rk, rq, misc, fw
constexpr int SM_BAR = SM_VEC + 8 * 64 * 4;
constexpr int SM_TOTAL = SM_BAR + 64;
constexpr int SMEM_BYTES = SM_TOTAL + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");

// TMEM columns
constexpr uint32_t T_S = 0, T_D1 = 128, T_DW = 192, T_DU = 256, T_DWS = 320, T_DQS = 384,
                   T_DO = 448;
constexpr uint32_t TMEM_COLS = 512;

constexpr uint32_t ID_N64_KK = idesc_bf16_f32(128, 64, 0, 0);
constexpr uint32_t ID_N64_MK = idesc_bf16_f32(128, 64, 1, 0);
constexpr uint32_t ID_N64_KM = idesc_bf16_f32(128, 64, 0, 1);
constexpr uint32_t ID_N128_KM = idesc_bf16_f32(128, 128, 0, 1);

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

// Element (i, j) of a 64 x 64 f32 table whose float4 groups are XOR-swizzled
// by row, so that a warp reading one float4 per row hits distinct banks.
__device__ __forceinline__ int ftab(int i, int j) {
    return i * 64 + ((((j >> 2) ^ (i & 15)) & 15) << 2) + (j & 3);
}

// Sum of squares of a 128-element bf16 row stored as two 128-byte swizzled rows.
__device__ __forceinline__ float row_sumsq(const uint8_t* blk0, const uint8_t* blk1, int row) {
    float s = 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const uint4* p = reinterpret_cast<const uint4*>((half ? blk1 : blk0) + row * 128);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint4 u = p[q ^ (row & 7)];  // same chunks, bank-conflict-free order
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
                s = fmaf(lo, lo, s);
                s = fmaf(hi, hi, s);
            }
        }
    }
    return s;
}

__global__ void __launch_bounds__(NT, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                DeltaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float* Gs = reinterpret_cast<float*>(sm + SM_VEC);
    float* eGs = Gs + 64;
    float* Bs = Gs + 128;
    float* DECs = Gs + 192;
    float* RKs = Gs + 256;
    float* RQs = Gs + 320;
    float* misc = Gs + 384;
    float* FWs = Gs + 448;  // beta_j e^{G_j} rk_j
    float* Am = reinterpret_cast<float*>(sm + SM_A);
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + SM_BAR);  // [0], [1]
    uint64_t* bar_mma = bar_tma + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_tma + 3);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x % a.H_v;
    const int seq = blockIdx.x / a.H_v;
    const int kh = h / (a.H_v / a.H_k);
    int64_t s0, s1;
    seq_bounds(a.cu, seq, a.T, s0, s1);
    const int64_t L = s1 - s0;
    const int nchunks = (int)((L + C - 1) / C);
    const int xq = kh * D, xk = a.H_k * D + kh * D, xv = 2 * a.H_k * D + h * D;
    int64_t ck_row0 = 0;
    if (a.ckpt_every > 0 && a.ckpt != nullptr) ck_row0 = ckpt_row0(a.cu, seq, a.T, a.ckpt_every);

    if (tid == 0) {
        mbar_init(&bar_tma[0], 1);
        mbar_init(&bar_tma[1], 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        prefetch_tmap(&qmap);
        prefetch_tmap(&omap);
    }
    if (warp == 0) {
        tmem_alloc(tslot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *tslot;
    const uint32_t lo = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lane quarter

    int issued0 = 0, issued1 = 0;      // TMA issues per buffer (thread 0)
    int consumed0 = 0, consumed1 = 0;  // completed TMA phases waited on, per buffer
    auto issue_tma = [&](int c) {
        const int b = c & 1;
        const int y = (int)(s0 + (int64_t)c * C);
        uint8_t* kq = sm + SM_KQ + b * KQ_BYTES;
        uint8_t* vv = sm + SM_V + b * V_BYTES;
        mbar_arrive_expect_tx(&bar_tma[b], 6 * 8192);
        tma_load_2d(kq, &qmap, &bar_tma[b], xk, y);
        tma_load_2d(kq + 16384, &qmap, &bar_tma[b], xk + 64, y);
        tma_load_2d(kq + 8192, &qmap, &bar_tma[b], xq, y);
        tma_load_2d(kq + 24576, &qmap, &bar_tma[b], xq + 64, y);
        tma_load_2d(vv, &qmap, &bar_tma[b], xv, y);
        tma_load_2d(vv + 8192, &qmap, &bar_tma[b], xv + 64, y);
        if (b) ++issued1; else ++issued0;
    };
    if (tid == 0) {
        if (nchunks > 0) issue_tma(0);
        if (nchunks > 1) issue_tma(1);
    }

    // initial state: thread v owns column v of S (row v of S^T)
    const int64_t sbase = ((int64_t)seq * a.H_v + h) * D * D;
    for (int c0 = 0; c0 < D; c0 += 32) {
        float sv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
            sv[j] = a.S0 != nullptr ? a.S0[sbase + (int64_t)(c0 + j) * D + tid] : 0.f;
        tmem_st32(tb + lo + T_S + c0, sv);
        store_row_bf16(sm + SM_ST + (c0 >> 6) * 16384, tid, c0 & 63, sv, 32);
    }
    tmem_wait_st();
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // raw gate inputs of a chunk's token `tid` (tid < 64), loaded one chunk ahead
    float ga = 0.f, gb = 0.f;
    auto load_gates = [&](int cc) {
        ga = 0.f;
        gb = 0.f;
        const int64_t tok = (int64_t)cc * C + tid;
        if (tid < 64 && tok < L) {
            const int64_t gi = (s0 + tok) * a.H_v + h;
            if (a.g != nullptr) {
                ga = a.g[gi];
                gb = a.beta[gi];
            } else {
                ga = to_f(static_cast<const bf16*>(a.a)[gi]);
                gb = to_f(static_cast<const bf16*>(a.b)[gi]);
            }
        }
    };
    if (nchunks > 0) load_gates(0);
    const float A_log_h = a.g == nullptr ? a.A_log[h] : 0.f;
    const float dt_bias_h = a.g == nullptr ? a.dt_bias[h] : 0.f;
    constexpr float kLog2e = 1.4426950408889634f;

    uint32_t mma_phase = 0;
    bool mma_pending = false;
    bool ok = true;
    int c = 0;
    for (; c < nchunks; ++c) {
        const int b = c & 1;
        const int64_t t0 = s0 + (int64_t)c * C;
        const int n = (int)(L - (int64_t)c * C < C ? L - (int64_t)c * C : C);
        uint8_t* kq = sm + SM_KQ + b * KQ_BYTES;
        uint8_t* vv = sm + SM_V + b * V_BYTES;

        // ---- gates (log2 domain) and their in-warp cumulative sums (tokens 0-31, 32-63)
        if (tid < 64) {
            float g = 0.f, bt = 0.f;
            if (tid < n) {
                if (a.g != nullptr) {
                    g = ga;
                    bt = gb;
                } else {
                    g = gate_g(ga, A_log_h, dt_bias_h);
                    bt = sigmoid_f(gb);
                }
            }
            if (c + 1 < nchunks) load_gates(c + 1);  // lands while this chunk computes
            float x = g * kLog2e;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            Gs[tid] = x;
            Bs[tid] = bt;
        }
        ok = mbar_wait(&bar_tma[b], (uint32_t)((b ? consumed1 : consumed0) & 1), kWaitNs);
        ok = __syncthreads_and(ok);
        if (!ok) break;
        if (b) ++consumed1; else ++consumed0;
        if (tid >= 32 && tid < 64) Gs[tid] += Gs[31];
        // l2-norm factors from the tiles
        {
            const bool isk = tid < 64;
            const int r = isk ? tid : tid - 64;
            const float ss = isk ? row_sumsq(kq, kq + 16384, r) : row_sumsq(kq + 8192, kq + 24576, r);
            float f = isk ? 1.f : a.scale;
            if (a.l2norm) f = f / sqrtf(ss + 1e-6f);
            (isk ? RKs : RQs)[r] = f;
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
        // decay-and-norm factor tables for A and P: thread t fills half of row t/2
        {
            float* FA = reinterpret_cast<float*>(sm + SM_UT);
            float* FP = FA + 64 * 64;
            const int i = tid >> 1, j0 = (tid & 1) * 32;
            const float Gi = Gs[i], fa = Bs[i] * RKs[i], fq = RQs[i];
            const bool live = i < n;
#pragma unroll 2
            for (int g4 = 0; g4 < 8; ++g4) {
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

        // ---- MMA 1: D1 = [K; Q] K^T   (M=128 rows: k_i then q_i; N=64: k_j)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t akq = smem_u32(kq);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                mma_bf16(tb + T_D1, sdesc_sw128(akq + off, 16, 1024),
                         sdesc_sw128(akq + off, 16, 1024), ID_N64_KK, k > 0);
            }
            mma_commit(bar_mma);
        }
        mma_pending = true;
        ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase, kWaitNs));
        if (!ok) break;
        mma_phase ^= 1;
        mma_pending = false;
        tc_fence_after();

        // ---- A (rows 0-63, f32) and P (rows 64-127, bf16 operand) = D1 * factor table
        {
            float d1[64];
            tmem_ld32(tb + lo + T_D1, d1);
            tmem_ld32(tb + lo + T_D1 + 32, d1 + 32);
            tmem_wait_ld();
            const int i = tid & 63;
            const float* F = reinterpret_cast<const float*>(sm + SM_UT) + (tid < 64 ? 0 : 64 * 64);
#pragma unroll
            for (int g4 = 0; g4 < 16; ++g4) {
                const float4 f = *reinterpret_cast<const float4*>(F + ftab(i, 4 * g4));
                d1[4 * g4 + 0] *= f.x;
                d1[4 * g4 + 1] *= f.y;
                d1[4 * g4 + 2] *= f.z;
                d1[4 * g4 + 3] *= f.w;
            }
            if (tid < 64) {
#pragma unroll
                for (int g4 = 0; g4 < 16; ++g4)
                    *reinterpret_cast<float4*>(&Am[i * A_PITCH + 4 * g4]) =
                        make_float4(d1[4 * g4], d1[4 * g4 + 1], d1[4 * g4 + 2], d1[4 * g4 + 3]);
            } else {
                store_row_bf16(sm + SM_P, i, 0, d1, 64);
            }
        }
        fence_async_smem();
        __syncthreads();

        // ---- T' = (I + A)^-1, blocked by 16 (f32): the four diagonal blocks by
        //      forward substitution, then by block distance d = 1, 2, 3:
        //      T'_{b+d,b} = -T'_{b+d,b+d} sum_{c=b}^{b+d-1} A_{b+d,c} T'_{c,b}
        {
            float* Tm = reinterpret_cast<float*>(sm + SM_UT);  // [64][A_PITCH]
            float* Mt = Tm + 64 * A_PITCH;                     // <= 3 blocks of 16 x 16
            if (tid == 0) bulk_wait_read_all();  // the previous O tile store has left B_W/B_U
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
                // strictly upper blocks are zero: (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
                for (int e = tid - 64; e < 6 * 256; e += 64) {
                    const int blk = e >> 8, r = (e >> 4) & 15, cc = e & 15;
                    const int br = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
                    const int bc = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
                    Tm[(br * 16 + r) * A_PITCH + bc * 16 + cc] = 0.f;
                }
            }
            __syncthreads();
            for (int dd = 1; dd < 4; ++dd) {
                const int nel = (4 - dd) * 256;
                for (int e = tid; e < nel; e += NT) {
                    const int bl = e >> 8, r = (e >> 4) & 15, cc = e & 15;
                    const float* Ar = &Am[((bl + dd) * 16 + r) * A_PITCH];
                    const float* Tc = &Tm[bl * 16 + cc];
                    float acc = 0.f;
                    for (int k = bl * 16; k < (bl + dd) * 16; ++k) acc = fmaf(Ar[k], Tc[k * A_PITCH], acc);
                    Mt[e] = acc;
                }
                __syncthreads();
                for (int e = tid; e < nel; e += NT) {
                    const int bl = e >> 8, r = (e >> 4) & 15, cc = e & 15;
                    const int a0 = (bl + dd) * 16;
                    const float* Ta = &Tm[(a0 + r) * A_PITCH + a0];
                    const float* Mb = &Mt[(bl << 8) + cc];
                    float acc = 0.f;
#pragma unroll
                    for (int k = 0; k < 16; ++k) acc = fmaf(Ta[k], Mb[k * 16], acc);
                    Tm[(a0 + r) * A_PITCH + bl * 16 + cc] = -acc;
                }
                __syncthreads();
            }
            // B_W = T' diag(beta e^G rk) (threads 0-63), B_U = T' diag(beta) (64-127), bf16
            {
                const int i = tid & 63;
                const float* Ti = &Tm[i * A_PITCH];
                const float* Fc = tid < 64 ? FWs : Bs;
                float row[64];
#pragma unroll
                for (int g4 = 0; g4 < 16; ++g4) {
                    const float4 t4 = *reinterpret_cast<const float4*>(Ti + 4 * g4);
                    const float4 f4 = *reinterpret_cast<const float4*>(Fc + 4 * g4);
                    row[4 * g4 + 0] = t4.x * f4.x;
                    row[4 * g4 + 1] = t4.y * f4.y;
                    row[4 * g4 + 2] = t4.z * f4.z;
                    row[4 * g4 + 3] = t4.w * f4.w;
                }
                store_row_bf16(sm + (tid < 64 ? SM_BW : SM_BU), i, 0, row, 64);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- MMA 2, 3: W^T = K^T B_W^T,  U^T = V^T B_U^T   (M = d or v, N = i, K = j)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t akq = smem_u32(kq), av = smem_u32(vv);
            const uint32_t bw = smem_u32(sm + SM_BW), bu = smem_u32(sm + SM_BU);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mma_bf16(tb + T_DW, sdesc_sw128(akq + k * 2048, 16384, 1024),
                         sdesc_sw128(bw + k * 32, 16, 1024), ID_N64_MK, k > 0);
                mma_bf16(tb + T_DU, sdesc_sw128(av + k * 2048, 8192, 1024),
                         sdesc_sw128(bu + k * 32, 16, 1024), ID_N64_MK, k > 0);
            }
            mma_commit(bar_mma);
        }
        mma_pending = true;
        ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase, kWaitNs));
        if (!ok) break;
        mma_phase ^= 1;
        mma_pending = false;
        tc_fence_after();

        // ---- W^T -> bf16 operand (row d = tid)
        {
            float w[64];
            tmem_ld32(tb + lo + T_DW, w);
            tmem_ld32(tb + lo + T_DW + 32, w + 32);
            tmem_wait_ld();
            store_row_bf16(sm + SM_WT, tid, 0, w, 64);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- MMA 4, 5: (W S)^T = S^T W^T,  (Q S)^T = S^T Q^T   (M = v, N = i, K = d)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t ast = smem_u32(sm + SM_ST), bwt = smem_u32(sm + SM_WT);
            const uint32_t akq = smem_u32(kq);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                mma_bf16(tb + T_DWS, sdesc_sw128(ast + off, 16, 1024),
                         sdesc_sw128(bwt + k * 2048, 16384, 1024), ID_N64_KM, k > 0);
                mma_bf16(tb + T_DQS, sdesc_sw128(ast + off, 16, 1024),
                         sdesc_sw128(akq + 8192 + off, 16, 1024), ID_N64_KK, k > 0);
            }
            mma_commit(bar_mma);
        }
        mma_pending = true;
        ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase, kWaitNs));
        if (!ok) break;
        mma_phase ^= 1;
        mma_pending = false;
        tc_fence_after();

        // ---- U'^T = U^T - (W S)^T (two bf16 copies); S^T *= e^{G_n} in TMEM
        {
            float u[64], ws[64];
            tmem_ld32(tb + lo + T_DU, u);
            tmem_ld32(tb + lo + T_DU + 32, u + 32);
            tmem_ld32(tb + lo + T_DWS, ws);
            tmem_ld32(tb + lo + T_DWS + 32, ws + 32);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 64; ++j) u[j] -= ws[j];
            store_row_bf16(sm + SM_UT, tid, 0, u, 64);
#pragma unroll
            for (int j = 0; j < 64; ++j) ws[j] = u[j] * DECs[j] * RKs[j];
            store_row_bf16(sm + SM_UTD, tid, 0, ws, 64);
            const float eGn = misc[0];
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                float sv[32];
                tmem_ld32(tb + lo + T_S + c0, sv);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) sv[j] *= eGn;
                tmem_st32(tb + lo + T_S + c0, sv);
            }
            tmem_wait_st();
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- MMA 6: S^T += U'^T_dec K  (M = v, N = d, K = j);  MMA 7: O_P^T = U'^T P^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t autd = smem_u32(sm + SM_UTD), aut = smem_u32(sm + SM_UT);
            const uint32_t akq = smem_u32(kq), bp = smem_u32(sm + SM_P);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mma_bf16(tb + T_S, sdesc_sw128(autd + k * 32, 16, 1024),
                         sdesc_sw128(akq + k * 2048, 16384, 1024), ID_N128_KM, 1);
                mma_bf16(tb + T_DO, sdesc_sw128(aut + k * 32, 16, 1024),
                         sdesc_sw128(bp + k * 32, 16, 1024), ID_N64_KK, k > 0);
            }
            mma_commit(bar_mma);
        }
        mma_pending = true;
        ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase, kWaitNs));
        if (!ok) break;
        mma_phase ^= 1;
        mma_pending = false;
        tc_fence_after();
        // this chunk's tiles are consumed: prefetch chunk c + 2 into the buffer
        if (tid == 0 && c + 2 < nchunks) issue_tma(c + 2);

        // ---- O = e^G rq (Q S) + P U'  (thread v writes column v of this chunk's O)
        {
            float qs[64], po[64];
            tmem_ld32(tb + lo + T_DQS, qs);
            tmem_ld32(tb + lo + T_DQS + 32, qs + 32);
            tmem_ld32(tb + lo + T_DO, po);
            tmem_ld32(tb + lo + T_DO + 32, po + 32);
            tmem_wait_ld();
            if (n == C) {
                // stage the 64 x 128 tile (128B-swizzled, in the B_W/B_U buffers, free
                // until the next solve) and write it with two TMA stores
                uint8_t* stg = sm + SM_BW + (tid >> 6) * 8192;
                const int cc = tid & 63;
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    *reinterpret_cast<bf16*>(stg + sw128_off(i, cc)) =
                        __float2bfloat16_rn(eGs[i] * RQs[i] * qs[i] + po[i]);
                fence_async_smem();
                __syncthreads();
                if (tid == 0) {
                    tma_store_2d(&omap, sm + SM_BW, h * D, (int)t0);
                    tma_store_2d(&omap, sm + SM_BW + 8192, h * D + 64, (int)t0);
                    bulk_commit();
                }
            } else {
                bf16* o = static_cast<bf16*>(a.o) + (t0 * a.H_v + h) * D + tid;
                const int64_t ostride = (int64_t)a.H_v * D;
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (i < n) o[i * ostride] = __float2bfloat16_rn(eGs[i] * RQs[i] * qs[i] + po[i]);
            }
        }
        // ---- new state -> bf16 S^T operand (and checkpoint)
        {
            const int64_t done = (int64_t)c * C + n;
            float* ck = nullptr;
            if (a.ckpt_every > 0 && a.ckpt != nullptr && done % a.ckpt_every == 0) {
                const int64_t row = ck_row0 + done / a.ckpt_every - 1;
                if (row < a.ckpt_rows) ck = a.ckpt + (row * a.H_v + h) * D * D;
            }
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                float sv[32];
                tmem_ld32(tb + lo + T_S + c0, sv);
                tmem_wait_ld();
                store_row_bf16(sm + SM_ST + (c0 >> 6) * 16384, tid, c0 & 63, sv, 32);
                if (ck != nullptr)
#pragma unroll
                    for (int j = 0; j < 32; ++j) ck[(int64_t)(c0 + j) * D + tid] = sv[j];
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    if (ok) {
        if (a.S_final != nullptr) {
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                float sv[32];
                tmem_ld32(tb + lo + T_S + c0, sv);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) a.S_final[sbase + (int64_t)(c0 + j) * D + tid] = sv[j];
            }
        }
    } else if (tid == 0) {
        atomicOr(&g_device_error, 1);
        // let copies and MMAs still in flight land before the memory is released
        if (mma_pending) mbar_wait(bar_mma, mma_phase, kWaitNs);
        for (int k = consumed0; k < issued0; ++k) mbar_wait(&bar_tma[0], (uint32_t)(k & 1), kWaitNs);
        for (int k = consumed1; k < issued1; ++k) mbar_wait(&bar_tma[1], (uint32_t)(k & 1), kWaitNs);
    }
    if (tid == 0) bulk_wait_all();  // O tile stores complete before the CTA's memory goes
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, TMEM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

}  // namespace

bool chunk_tc_supported(const DeltaArgs& a, gdn_dtype_t dt) {
    return dt == GDN_BF16 && a.D == D && a.T > 0 && a.qkv != nullptr && encode_fn() != nullptr;
}

cudaError_t launch_chunk_tc(const DeltaArgs& a, cudaStream_t s) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    const uint64_t conv_dim = 2ull * a.H_k * D + (uint64_t)a.H_v * D;
    CUtensorMap map;
    cuuint64_t gdim[2] = {conv_dim, (cuuint64_t)a.T};
    cuuint64_t gstr[1] = {conv_dim * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t es[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.qkv), gdim, gstr, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    CUtensorMap omap;
    cuuint64_t odim[2] = {(cuuint64_t)a.H_v * D, (cuuint64_t)a.T};
    cuuint64_t ostr[1] = {(cuuint64_t)a.H_v * D * 2};
    if (enc(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.o, odim, ostr, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(a.n_seq * a.H_v);
    if (grid == 0) return cudaSuccess;
    chunk_tc_kernel<<<grid, NT, SMEM_BYTES, s>>>(map, omap, a);
    return cudaGetLastError();
}

cudaError_t read_and_clear_device_error(cudaStream_t s, int* flags) {
    int h = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&h, g_device_error, sizeof(int), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    *flags = h;
    if (h != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

}  // namespace gdn
