// Recurrent (per-token) gated delta rule for decode, state updated in place.
//
// cortex commit "feat(stage-8c): linear-attention layer (Qwen3-Next
// GatedDeltaNet)", "Delta rule (recurrent, per-token)":
//     state *= exp(g); kv_mem = state^T k; delta = (v - kv_mem) * beta;
//     state += outer(k, delta); out = state^T q
// with q, k l2-normalised ("Block": L2norm on q,k) and g = -exp(A_log) *
// softplus(a + dt_bias), beta = sigmoid(b) in f32 ("Discretisation").
// NxD-Inference PR "Add Qwen3.6-27B hybrid DeltaNet/GQA contrib model and vLLM
// serving path", Summary: the token-generation kernel.
//
// Decode is HBM-bound: each (sequence, value head) state is D x D f32
// (64 KiB at D = 128) and must be read and written once per token.  Both
// products the rule needs come from the OLD state in one pass:
//     kv_mem = e^g S^T k,   out = e^g S^T q + (k . q) delta
// so one CTA per (sequence, head) streams its state into registers with
// coalesced 128-bit loads (a warp reads one 512-byte state row), reduces S^T k
// and S^T q across warps through shared memory, and writes the updated state
// e^g S + k delta^T straight from the same registers.
#include "gdn_common.cuh"
#include "gdn_launch.h"

namespace gdn {
namespace {

template <typename T, int D, int NW>
__global__ void __launch_bounds__(NW * 32, (D >= 128 ? 2 : 1))
recurrent_decode_kernel(DeltaArgs a) {
    constexpr int NT = NW * 32;
    constexpr int TPR = D / 4;         // threads per state row (float4 each)
    constexpr int RPP = NT / TPR;      // rows per pass
    constexpr int PASSES = D / RPP;    // rows per thread
    static_assert(NT % TPR == 0 && D % RPP == 0, "layout");

    const int unit = blockIdx.x;
    const int b = unit / a.H_v;
    const int h = unit - b * a.H_v;
    const int kh = h / (a.H_v / a.H_k);
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int cq = tid % TPR;
    const int r0 = tid / TPR;

    float* __restrict__ S = a.S_final + ((int64_t)b * a.H_v + h) * D * D;

    // 1. stream the state in (independent of everything else)
    float4 s[PASSES];
#pragma unroll
    for (int p = 0; p < PASSES; ++p)
        s[p] = __ldcs(reinterpret_cast<const float4*>(S + (int64_t)(r0 + p * RPP) * D) + cq);

    __shared__ __align__(16) float qs[D], ks[D], vs[D], ds[D];
    __shared__ __align__(16) float red[2][RPP][D];
    __shared__ float gb[2];

    const int conv_dim = 2 * a.H_k * D + a.H_v * D;
    const T* row = static_cast<const T*>(a.qkv) + (int64_t)b * conv_dim;
    for (int i = tid; i < D; i += NT) {
        qs[i] = to_f(row[kh * D + i]);
        ks[i] = to_f(row[a.H_k * D + kh * D + i]);
        vs[i] = to_f(row[2 * a.H_k * D + h * D + i]);
    }
    if (tid == 0) {
        const int64_t gi = (int64_t)b * a.H_v + h;
        if (a.g != nullptr) {
            gb[0] = a.g[gi];
            gb[1] = a.beta[gi];
        } else {
            gb[0] = gate_g(to_f(static_cast<const T*>(a.a)[gi]), a.A_log[h], a.dt_bias[h]);
            gb[1] = sigmoid_f(to_f(static_cast<const T*>(a.b)[gi]));
        }
    }
    __syncthreads();

    // 2. norms (every warp computes them redundantly; no extra barrier)
    float sq = 0.f, sk = 0.f, sqk = 0.f;
    for (int i = lane; i < D; i += 32) {
        sq = fmaf(qs[i], qs[i], sq);
        sk = fmaf(ks[i], ks[i], sk);
        sqk = fmaf(qs[i], ks[i], sqk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    sqk = warp_sum(sqk);
    float rq = a.scale, rk = 1.f;
    if (a.l2norm) {
        rq = a.scale / sqrtf(sq + 1e-6f);
        rk = 1.f / sqrtf(sk + 1e-6f);
    }
    const float kq = sqk * rq * rk;  // k^ . q^

    // 3. partial S^T k^ and S^T q^ over this thread's rows
    float mk[4] = {0.f, 0.f, 0.f, 0.f}, mq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int i = r0 + p * RPP;
        const float kv = ks[i] * rk, qv = qs[i] * rq;
        mk[0] = fmaf(s[p].x, kv, mk[0]); mk[1] = fmaf(s[p].y, kv, mk[1]);
        mk[2] = fmaf(s[p].z, kv, mk[2]); mk[3] = fmaf(s[p].w, kv, mk[3]);
        mq[0] = fmaf(s[p].x, qv, mq[0]); mq[1] = fmaf(s[p].y, qv, mq[1]);
        mq[2] = fmaf(s[p].z, qv, mq[2]); mq[3] = fmaf(s[p].w, qv, mq[3]);
    }
    *reinterpret_cast<float4*>(&red[0][r0][cq * 4]) = make_float4(mk[0], mk[1], mk[2], mk[3]);
    *reinterpret_cast<float4*>(&red[1][r0][cq * 4]) = make_float4(mq[0], mq[1], mq[2], mq[3]);
    __syncthreads();

    const float eg = expf(gb[0]);
    const float bt = gb[1];
    for (int j = tid; j < D; j += NT) {
        float m = 0.f, pq = 0.f;
#pragma unroll
        for (int r = 0; r < RPP; ++r) {
            m += red[0][r][j];
            pq += red[1][r][j];
        }
        const float delta = bt * (vs[j] - eg * m);
        ds[j] = delta;
        const float out = eg * pq + kq * delta;
        static_cast<T*>(a.o)[((int64_t)b * a.H_v + h) * D + j] = from_f<T>(out);
    }
    __syncthreads();

    // 4. S <- e^g S + k^ delta^T, written from registers
    const float4 d4 = *reinterpret_cast<const float4*>(&ds[cq * 4]);
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int i = r0 + p * RPP;
        const float kv = ks[i] * rk;
        float4 n;
        n.x = fmaf(kv, d4.x, eg * s[p].x);
        n.y = fmaf(kv, d4.y, eg * s[p].y);
        n.z = fmaf(kv, d4.z, eg * s[p].z);
        n.w = fmaf(kv, d4.w, eg * s[p].w);
        __stcs(reinterpret_cast<float4*>(S + (int64_t)i * D) + cq, n);
    }
}

template <typename T>
cudaError_t decode_t(const DeltaArgs& a, cudaStream_t s) {
    const unsigned units = (unsigned)(a.T * a.H_v);
    if (units == 0) return cudaSuccess;
    if (a.D == 128)
        recurrent_decode_kernel<T, 128, 8><<<units, 256, 0, s>>>(a);
    else
        recurrent_decode_kernel<T, 16, 1><<<units, 32, 0, s>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- fused decode step
// conv update + SiLU -> gates, l2 norms -> recurrence -> RMSNormGated for one
// token per sequence.  One CTA per (sequence, key head): it owns every conv
// channel of that key head (q, k and the r = H_v / H_k value heads' v), so it
// reads their old conv state and writes the shifted state in place with no
// other CTA touching them; it then runs the recurrence of its r value heads
// one after the other, each streaming its state once through registers as
// above, with the RMSNormGated of the head's output row as the epilogue.
// The conv output is rounded to the activation dtype before the rule, as the
// separate calls round y.
template <typename T, int D, int NW, int RMAX>
__global__ void __launch_bounds__(NW * 32, (D >= 128 ? 2 : 1))
decode_step_kernel(DecodeStepArgs a) {
    constexpr int NT = NW * 32;
    constexpr int TPR = D / 4;
    constexpr int RPP = NT / TPR;
    constexpr int PASSES = D / RPP;
    static_assert(NT % TPR == 0 && D % RPP == 0 && NT >= D, "layout");

    const int b = blockIdx.x / a.H_k;
    const int kh = blockIdx.x - b * a.H_k;
    const int r = a.H_v / a.H_k;
    const int64_t slot = a.slots != nullptr ? a.slots[b] : b;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cq = tid % TPR;
    const int r0 = tid / TPR;
    const int C = 2 * a.H_k * D + a.H_v * D;

    __shared__ __align__(16) float qs[D], ks[D], vs[RMAX][D], ds[D], os[D];
    __shared__ __align__(16) float red[2][RPP][D];
    __shared__ float gb[RMAX][2];
    __shared__ float wsum[NW];

    // the first head's state streams in while the conv runs
    float4 s[PASSES];
    auto load_state = [&](int j) {
        const float* S = a.state + (slot * a.H_v + kh * r + j) * D * D;
#pragma unroll
        for (int p = 0; p < PASSES; ++p)
            s[p] = __ldcs(reinterpret_cast<const float4*>(S + (int64_t)(r0 + p * RPP) * D) + cq);
    };
    load_state(0);

    // 1. conv update of the group's channels: q, k, then the r heads' v, one
    //    16-byte vector of channels per thread (x, 3 state and 4 weight
    //    vectors loaded together; [c][3] and [c][4] keep V channels contiguous)
    {
        constexpr int V = Vec16<T>::N;
        const T* x = static_cast<const T*>(a.x) + (int64_t)b * C;
        const T* w = static_cast<const T*>(a.conv_w);
        T* cs = static_cast<T*>(a.conv_state) + slot * C * 3;
        const int nvec = (2 + r) * D / V;
        for (int e = tid; e < nvec; e += NT) {
            const int grp = (e * V) / D, i0 = e * V - grp * D;
            const int c0 = grp == 0 ? kh * D + i0
                         : grp == 1 ? a.H_k * D + kh * D + i0
                                    : 2 * a.H_k * D + (kh * r + grp - 2) * D + i0;
            float xv[V], st[3 * V], wt[4 * V];
            load16(x + c0, xv);
#pragma unroll
            for (int k = 0; k < 3; ++k) load16(cs + (int64_t)c0 * 3 + k * V, st + k * V);
#pragma unroll
            for (int k = 0; k < 4; ++k) load16(w + (int64_t)c0 * 4 + k * V, wt + k * V);
            float* dst = grp == 0 ? qs + i0 : grp == 1 ? ks + i0 : vs[grp - 2] + i0;
            float nst[3 * V];
#pragma unroll
            for (int q = 0; q < V; ++q) {
                float acc = wt[q * 4] * st[q * 3];
                acc = fmaf(wt[q * 4 + 1], st[q * 3 + 1], acc);
                acc = fmaf(wt[q * 4 + 2], st[q * 3 + 2], acc);
                acc = fmaf(wt[q * 4 + 3], xv[q], acc);
                dst[q] = to_f(from_f<T>(silu_f(acc)));
                nst[q * 3] = st[q * 3 + 1];
                nst[q * 3 + 1] = st[q * 3 + 2];
                nst[q * 3 + 2] = xv[q];
            }
#pragma unroll
            for (int k = 0; k < 3; ++k) store16(cs + (int64_t)c0 * 3 + k * V, nst + k * V);
        }
        if (tid < r) {
            const int h = kh * r + tid;
            const int64_t gi = (int64_t)b * a.H_v + h;
            gb[tid][0] = gate_g(to_f(static_cast<const T*>(a.a)[gi]), a.A_log[h], a.dt_bias[h]);
            gb[tid][1] = sigmoid_f(to_f(static_cast<const T*>(a.b)[gi]));
        }
    }
    __syncthreads();
    float sq = 0.f, sk = 0.f, sqk = 0.f;
    for (int i = lane; i < D; i += 32) {
        sq = fmaf(qs[i], qs[i], sq);
        sk = fmaf(ks[i], ks[i], sk);
        sqk = fmaf(qs[i], ks[i], sqk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    sqk = warp_sum(sqk);
    float rq = a.scale, rk = 1.f;
    if (a.l2norm) {
        rq = a.scale / sqrtf(sq + 1e-6f);
        rk = 1.f / sqrtf(sk + 1e-6f);
    }
    const float kq = sqk * rq * rk;

    // 2. the r value heads in turn
    for (int j = 0; j < r; ++j) {
        const int h = kh * r + j;
        float* __restrict__ S = a.state + (slot * a.H_v + h) * D * D;
        float mk[4] = {0.f, 0.f, 0.f, 0.f}, mq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int p = 0; p < PASSES; ++p) {
            const int i = r0 + p * RPP;
            const float kv = ks[i] * rk, qv = qs[i] * rq;
            mk[0] = fmaf(s[p].x, kv, mk[0]); mk[1] = fmaf(s[p].y, kv, mk[1]);
            mk[2] = fmaf(s[p].z, kv, mk[2]); mk[3] = fmaf(s[p].w, kv, mk[3]);
            mq[0] = fmaf(s[p].x, qv, mq[0]); mq[1] = fmaf(s[p].y, qv, mq[1]);
            mq[2] = fmaf(s[p].z, qv, mq[2]); mq[3] = fmaf(s[p].w, qv, mq[3]);
        }
        *reinterpret_cast<float4*>(&red[0][r0][cq * 4]) = make_float4(mk[0], mk[1], mk[2], mk[3]);
        *reinterpret_cast<float4*>(&red[1][r0][cq * 4]) = make_float4(mq[0], mq[1], mq[2], mq[3]);
        __syncthreads();
        const float eg = expf(gb[j][0]);
        const float bt = gb[j][1];
        float o2 = 0.f;
        for (int c = tid; c < D; c += NT) {
            float m = 0.f, pq = 0.f;
#pragma unroll
            for (int rr = 0; rr < RPP; ++rr) {
                m += red[0][rr][c];
                pq += red[1][rr][c];
            }
            const float delta = bt * (vs[j][c] - eg * m);
            ds[c] = delta;
            const float o = to_f(from_f<T>(eg * pq + kq * delta));  // o as the separate call stores it
            os[c] = o;
            o2 = fmaf(o, o, o2);
        }
        o2 = warp_sum(o2);
        if (lane == 0) wsum[warp] = o2;
        __syncthreads();
        // S <- e^g S + k^ delta^T, written from registers
        const float4 d4 = *reinterpret_cast<const float4*>(&ds[cq * 4]);
#pragma unroll
        for (int p = 0; p < PASSES; ++p) {
            const int i = r0 + p * RPP;
            const float kv = ks[i] * rk;
            float4 n;
            n.x = fmaf(kv, d4.x, eg * s[p].x);
            n.y = fmaf(kv, d4.y, eg * s[p].y);
            n.z = fmaf(kv, d4.z, eg * s[p].z);
            n.w = fmaf(kv, d4.w, eg * s[p].w);
            __stcs(reinterpret_cast<float4*>(S + (int64_t)i * D) + cq, n);
        }
        // the registers are free: the next head's state streams in during
        // this head's norm epilogue
        if (j + 1 < r) load_state(j + 1);
        // RMSNormGated of the head's output row
        float tot = 0.f;
#pragma unroll
        for (int ww = 0; ww < NW; ++ww) tot += wsum[ww];
        const float rs = rsqrtf(tot / (float)D + a.eps);
        const T* z = static_cast<const T*>(a.z) + ((int64_t)b * a.H_v + h) * D;
        T* out = static_cast<T*>(a.out) + ((int64_t)b * a.H_v + h) * D;
        const T* nw = static_cast<const T*>(a.norm_w);
        for (int c = 2 * tid; c < D; c += 2 * NT) {
            const float2 g = silu2<T>(make_float2(to_f(z[c]), to_f(z[c + 1])));
            const float2 res = __fmul2_rn(__fmul2_rn(make_float2(to_f(nw[c]), to_f(nw[c + 1])),
                                                     __fmul2_rn(make_float2(os[c], os[c + 1]), make_float2(rs, rs))),
                                          g);
            out[c] = from_f<T>(res.x);
            out[c + 1] = from_f<T>(res.y);
        }
        __syncthreads();  // red, ds, os and wsum are reused by the next head
    }
}

// Thread-block cluster helpers: barrier phases over the CTAs of a cluster, and
// a 16-byte store into the same shared-memory variable of another CTA of it.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_cluster_v4(const void* local, uint32_t rank, float4 v) {
    const uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(ra), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

// The fused decode step for small batches: one CTA per (sequence, value head),
// r times the CTAs of decode_step_kernel, so that a few sequences still spread
// over many SMs.  The r value heads of a key head form a thread-block cluster;
// its first CTA owns the q and k conv channels (it reads their old conv state,
// writes the shifted one in place and sends the conv outputs to the others
// through distributed shared memory), and every CTA owns its head's v
// channels.  Per head the arithmetic and its order are decode_step_kernel's,
// so states and outputs are the same bit for bit.
template <typename T, int D, int NW>
__global__ void __launch_bounds__(NW * 32, (D >= 128 ? 2 : 1))
decode_step_head_kernel(DecodeStepArgs a) {
    constexpr int NT = NW * 32;
    constexpr int TPR = D / 4;
    constexpr int RPP = NT / TPR;
    constexpr int PASSES = D / RPP;
    static_assert(NT % TPR == 0 && D % RPP == 0 && NT >= D, "layout");

    const int r = a.H_v / a.H_k;
    const int b = blockIdx.x / a.H_v;
    const int h = blockIdx.x - b * a.H_v;
    const int kh = h / r, rank = h - kh * r;  // rank in the key head's cluster
    const bool cl = r > 1;
    if (cl) cluster_arrive_relaxed();  // this CTA has started (waited for before any remote store)
    const int64_t slot = a.slots != nullptr ? a.slots[b] : b;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cq = tid % TPR;
    const int r0 = tid / TPR;
    const int C = 2 * a.H_k * D + a.H_v * D;

    __shared__ __align__(16) float qs[D], ks[D], vs[D], ds[D], os[D];
    __shared__ __align__(16) float red[2][RPP][D];
    __shared__ float gb[2];
    __shared__ float wsum[NW];

    // the head's state streams in while the conv runs
    float* __restrict__ S = a.state + (slot * a.H_v + h) * D * D;
    float4 s[PASSES];
#pragma unroll
    for (int p = 0; p < PASSES; ++p)
        s[p] = __ldcs(reinterpret_cast<const float4*>(S + (int64_t)(r0 + p * RPP) * D) + cq);

    // 1. conv update of the channels this CTA owns (q and k in the first CTA
    //    of the cluster, then the head's v), as in decode_step_kernel
    {
        constexpr int V = Vec16<T>::N;
        const T* x = static_cast<const T*>(a.x) + (int64_t)b * C;
        const T* w = static_cast<const T*>(a.conv_w);
        T* cs = static_cast<T*>(a.conv_state) + slot * C * 3;
        const int g0 = rank == 0 ? 0 : 2;
        const int nvec = (3 - g0) * D / V;
        for (int e = tid; e < nvec; e += NT) {
            const int grp = g0 + (e * V) / D, i0 = e * V - (grp - g0) * D;
            const int c0 = grp == 0 ? kh * D + i0 : grp == 1 ? a.H_k * D + kh * D + i0 : 2 * a.H_k * D + h * D + i0;
            float xv[V], st[3 * V], wt[4 * V];
            load16(x + c0, xv);
#pragma unroll
            for (int k = 0; k < 3; ++k) load16(cs + (int64_t)c0 * 3 + k * V, st + k * V);
#pragma unroll
            for (int k = 0; k < 4; ++k) load16(w + (int64_t)c0 * 4 + k * V, wt + k * V);
            float* dst = grp == 0 ? qs + i0 : grp == 1 ? ks + i0 : vs + i0;
            float nst[3 * V];
#pragma unroll
            for (int q = 0; q < V; ++q) {
                float acc = wt[q * 4] * st[q * 3];
                acc = fmaf(wt[q * 4 + 1], st[q * 3 + 1], acc);
                acc = fmaf(wt[q * 4 + 2], st[q * 3 + 2], acc);
                acc = fmaf(wt[q * 4 + 3], xv[q], acc);
                dst[q] = to_f(from_f<T>(silu_f(acc)));
                nst[q * 3] = st[q * 3 + 1];
                nst[q * 3 + 1] = st[q * 3 + 2];
                nst[q * 3 + 2] = xv[q];
            }
#pragma unroll
            for (int k = 0; k < 3; ++k) store16(cs + (int64_t)c0 * 3 + k * V, nst + k * V);
        }
        if (tid == 0) {
            const int64_t gi = (int64_t)b * a.H_v + h;
            gb[0] = gate_g(to_f(static_cast<const T*>(a.a)[gi]), a.A_log[h], a.dt_bias[h]);
            gb[1] = sigmoid_f(to_f(static_cast<const T*>(a.b)[gi]));
        }
    }
    __syncthreads();
    if (cl) {
        // q and k from the first CTA to the others, once every CTA has started
        cluster_wait();
        if (rank == 0) {
            for (int e = tid; e < (r - 1) * (D / 2); e += NT) {
                const int dst = 1 + e / (D / 2), i = e % (D / 2);
                const float* src = i < D / 4 ? qs + 4 * i : ks + 4 * (i - D / 4);
                st_cluster_v4(src, (uint32_t)dst, *reinterpret_cast<const float4*>(src));
            }
        }
        cluster_sync();
    }
    float sq = 0.f, sk = 0.f, sqk = 0.f;
    for (int i = lane; i < D; i += 32) {
        sq = fmaf(qs[i], qs[i], sq);
        sk = fmaf(ks[i], ks[i], sk);
        sqk = fmaf(qs[i], ks[i], sqk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    sqk = warp_sum(sqk);
    float rq = a.scale, rk = 1.f;
    if (a.l2norm) {
        rq = a.scale / sqrtf(sq + 1e-6f);
        rk = 1.f / sqrtf(sk + 1e-6f);
    }
    const float kq = sqk * rq * rk;

    // 2. the recurrence of head h, then RMSNormGated of its output row
    float mk[4] = {0.f, 0.f, 0.f, 0.f}, mq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int i = r0 + p * RPP;
        const float kv = ks[i] * rk, qv = qs[i] * rq;
        mk[0] = fmaf(s[p].x, kv, mk[0]); mk[1] = fmaf(s[p].y, kv, mk[1]);
        mk[2] = fmaf(s[p].z, kv, mk[2]); mk[3] = fmaf(s[p].w, kv, mk[3]);
        mq[0] = fmaf(s[p].x, qv, mq[0]); mq[1] = fmaf(s[p].y, qv, mq[1]);
        mq[2] = fmaf(s[p].z, qv, mq[2]); mq[3] = fmaf(s[p].w, qv, mq[3]);
    }
    *reinterpret_cast<float4*>(&red[0][r0][cq * 4]) = make_float4(mk[0], mk[1], mk[2], mk[3]);
    *reinterpret_cast<float4*>(&red[1][r0][cq * 4]) = make_float4(mq[0], mq[1], mq[2], mq[3]);
    __syncthreads();
    const float eg = expf(gb[0]);
    const float bt = gb[1];
    float o2 = 0.f;
    for (int c = tid; c < D; c += NT) {
        float m = 0.f, pq = 0.f;
#pragma unroll
        for (int rr = 0; rr < RPP; ++rr) {
            m += red[0][rr][c];
            pq += red[1][rr][c];
        }
        const float delta = bt * (vs[c] - eg * m);
        ds[c] = delta;
        const float o = to_f(from_f<T>(eg * pq + kq * delta));  // o as the separate call stores it
        os[c] = o;
        o2 = fmaf(o, o, o2);
    }
    o2 = warp_sum(o2);
    if (lane == 0) wsum[warp] = o2;
    __syncthreads();
    const float4 d4 = *reinterpret_cast<const float4*>(&ds[cq * 4]);
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int i = r0 + p * RPP;
        const float kv = ks[i] * rk;
        float4 n;
        n.x = fmaf(kv, d4.x, eg * s[p].x);
        n.y = fmaf(kv, d4.y, eg * s[p].y);
        n.z = fmaf(kv, d4.z, eg * s[p].z);
        n.w = fmaf(kv, d4.w, eg * s[p].w);
        __stcs(reinterpret_cast<float4*>(S + (int64_t)i * D) + cq, n);
    }
    float tot = 0.f;
#pragma unroll
    for (int ww = 0; ww < NW; ++ww) tot += wsum[ww];
    const float rs = rsqrtf(tot / (float)D + a.eps);
    const T* z = static_cast<const T*>(a.z) + ((int64_t)b * a.H_v + h) * D;
    T* out = static_cast<T*>(a.out) + ((int64_t)b * a.H_v + h) * D;
    const T* nw = static_cast<const T*>(a.norm_w);
    for (int c = 2 * tid; c < D; c += 2 * NT) {
        const float2 g = silu2<T>(make_float2(to_f(z[c]), to_f(z[c + 1])));
        const float2 res = __fmul2_rn(__fmul2_rn(make_float2(to_f(nw[c]), to_f(nw[c + 1])),
                                                 __fmul2_rn(make_float2(os[c], os[c + 1]), make_float2(rs, rs))),
                                      g);
        out[c] = from_f<T>(res.x);
        out[c + 1] = from_f<T>(res.y);
    }
}

template <typename K, typename Args>
cudaError_t launch_cluster(K kernel, unsigned grid, unsigned block, size_t smem, unsigned cluster, cudaStream_t s,
                           const Args& a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = cluster;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

int device_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

template <typename T>
cudaError_t decode_step_t(const DecodeStepArgs& a, cudaStream_t s) {
    const unsigned units = (unsigned)(a.B * a.H_k);
    if (units == 0) return cudaSuccess;
    const int r = a.H_v / a.H_k;
    if (r > 8) return cudaErrorNotSupported;
    // same thread layout (and so the same summation order of S^T k and S^T q)
    // as the recurrent decode kernel: the fused step's state is bit-identical
    // to the separate calls'
    // at most one (sequence, key head) unit per two SMs: one clustered CTA per
    // value head instead (27B at B = 1: 12.0 against 16.4 us per step; from
    // B = 8 the per-key-head CTAs are faster)
    if ((int64_t)units * 2 <= device_sms()) {
        const unsigned heads = (unsigned)(a.B * a.H_v);
        return a.D == 128 ? launch_cluster(decode_step_head_kernel<T, 128, 8>, heads, 256, 0, (unsigned)r, s, a)
                          : launch_cluster(decode_step_head_kernel<T, 16, 1>, heads, 32, 0, (unsigned)r, s, a);
    }
    if (a.D == 128)
        decode_step_kernel<T, 128, 8, 8><<<units, 256, 0, s>>>(a);
    else
        decode_step_kernel<T, 16, 1, 8><<<units, 32, 0, s>>>(a);
    return cudaGetLastError();
}

// K draft tokens of speculative decoding checked in one pass: per sequence,
// the conv update, gates, l2 norms, recurrence and RMSNormGated of tokens
// 0..K-1 in order, from the states in slot slots[b][0], writing the conv state
// and the recurrent state after token t to slot slots[b][t + 1] (so that
// accepting j draft tokens is choosing slot slots[b][j], with no copy).  One
// CTA per (sequence, key head) as in the fused step, with its thread layout and
// arithmetic order, so every state and output equals that of K fused steps;
// the state of each value head is read once and written K times.
template <typename T, int D, int NW>
__global__ void __launch_bounds__(NW * 32, (D >= 128 ? 2 : 1))
decode_verify_kernel(DecodeVerifyArgs a) {
    constexpr int NT = NW * 32;
    constexpr int TPR = D / 4;
    constexpr int RPP = NT / TPR;
    constexpr int PASSES = D / RPP;
    constexpr int V = Vec16<T>::N;
    static_assert(NT % TPR == 0 && D % RPP == 0 && NT >= D, "layout");

    const int b = blockIdx.x / a.H_k;
    const int kh = blockIdx.x - b * a.H_k;
    const int r = a.H_v / a.H_k, K = a.K;
    const int32_t* sl = a.slots + (int64_t)b * (K + 1);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cq = tid % TPR;
    const int r0 = tid / TPR;
    const int C = 2 * a.H_k * D + a.H_v * D;

    extern __shared__ __align__(16) float vsm[];
    float* qs = vsm;                  // [K][D]
    float* ks = qs + K * D;           // [K][D]
    float* vs = ks + K * D;           // [K][r][D]
    float* zs = vs + K * r * D;       // [K][r][D]: the gate input z
    float* ds = zs + K * r * D;       // [D]
    float* os = ds + D;               // [D]
    float* red = os + D;              // [2][RPP][D]
    float* gb = red + 2 * RPP * D;    // [K][r][2]: g, beta
    float* nrm = gb + 2 * K * r;      // [K][3]: rq, rk, k.q rq rk
    float* wsum = nrm + 3 * K;        // [NW]

    const int64_t s_in = sl[0];
    float4 s[PASSES];
    auto load_state = [&](int j) {
        const float* S = a.state + (s_in * a.H_v + kh * r + j) * D * D;
#pragma unroll
        for (int p = 0; p < PASSES; ++p)
            s[p] = __ldcs(reinterpret_cast<const float4*>(S + (int64_t)(r0 + p * RPP) * D) + cq);
    };
    // a value head's state into L2 ahead of its register loads (which wait for
    // the registers: the conv's window first, then the previous head)
    auto prefetch_state = [&](int j) {
        const char* S = reinterpret_cast<const char*>(a.state + (s_in * a.H_v + kh * r + j) * D * D);
        for (int off = tid * 128; off < D * D * 4; off += NT * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(S + off));
    };
    prefetch_state(0);

    // 1. conv over the K tokens: q, k, then the r heads' v, one 16-byte vector
    //    of channels per thread; the window slides over [state | x_0 .. x_{K-1}]
    {
        const T* x = static_cast<const T*>(a.x) + (int64_t)b * K * C;
        const T* w = static_cast<const T*>(a.conv_w);
        T* cs = static_cast<T*>(a.conv_state);
        const int nvec = (2 + r) * D / V;
        for (int e = tid; e < nvec; e += NT) {
            const int grp = (e * V) / D, i0 = e * V - grp * D;
            const int c0 = grp == 0 ? kh * D + i0
                         : grp == 1 ? a.H_k * D + kh * D + i0
                                    : 2 * a.H_k * D + (kh * r + grp - 2) * D + i0;
            float st[3 * V], wt[4 * V];
#pragma unroll
            for (int k = 0; k < 3; ++k) load16(cs + (s_in * C + c0) * 3 + k * V, st + k * V);
#pragma unroll
            for (int k = 0; k < 4; ++k) load16(w + (int64_t)c0 * 4 + k * V, wt + k * V);
            float* dst = grp == 0 ? qs + i0 : grp == 1 ? ks + i0 : vs + (grp - 2) * D + i0;
            const int tstride = grp < 2 ? D : r * D;
            for (int t = 0; t < K; ++t) {
                float xv[V];
                load16(x + (int64_t)t * C + c0, xv);
#pragma unroll
                for (int q = 0; q < V; ++q) {
                    float acc = wt[q * 4] * st[q * 3];
                    acc = fmaf(wt[q * 4 + 1], st[q * 3 + 1], acc);
                    acc = fmaf(wt[q * 4 + 2], st[q * 3 + 2], acc);
                    acc = fmaf(wt[q * 4 + 3], xv[q], acc);
                    dst[t * tstride + q] = to_f(from_f<T>(silu_f(acc)));
                    st[q * 3] = st[q * 3 + 1];  // the window moves one token
                    st[q * 3 + 1] = st[q * 3 + 2];
                    st[q * 3 + 2] = xv[q];
                }
                T* out_cs = cs + ((int64_t)sl[t + 1] * C + c0) * 3;
#pragma unroll
                for (int k = 0; k < 3; ++k) store16(out_cs + k * V, st + k * V);
            }
        }
        for (int e = tid; e < K * r; e += NT) {
            const int t = e / r, j = e - t * r;
            const int h = kh * r + j;
            const int64_t gi = ((int64_t)b * K + t) * a.H_v + h;
            gb[2 * e] = gate_g(to_f(static_cast<const T*>(a.a)[gi]), a.A_log[h], a.dt_bias[h]);
            gb[2 * e + 1] = sigmoid_f(to_f(static_cast<const T*>(a.b)[gi]));
        }
        // z of the CTA's r heads for the K tokens (contiguous r * D per token),
        // staged once so that the K * r norm epilogues do not wait on DRAM
        const T* zg = static_cast<const T*>(a.z) + ((int64_t)b * K * a.H_v + kh * r) * D;
        for (int e = tid; e < K * r * D / V; e += NT) {
            const int t = (e * V) / (r * D), o = e * V - t * r * D;
            float zv[V];
            load16(zg + (int64_t)t * a.H_v * D + o, zv);
#pragma unroll
            for (int q = 0; q < V; ++q) zs[t * r * D + o + q] = zv[q];
        }
    }
    __syncthreads();
    // the first value head's state streams in while the norms are formed (the
    // conv's K-token window needs the registers before)
    load_state(0);
    // l2 norms of each token's q and k (each warp sums the whole row, lanes
    // strided, as the fused step does)
    for (int t = warp; t < K; t += NW) {
        float sq = 0.f, sk = 0.f, sqk = 0.f;
        for (int i = lane; i < D; i += 32) {
            sq = fmaf(qs[t * D + i], qs[t * D + i], sq);
            sk = fmaf(ks[t * D + i], ks[t * D + i], sk);
            sqk = fmaf(qs[t * D + i], ks[t * D + i], sqk);
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        sqk = warp_sum(sqk);
        float rq = a.scale, rk = 1.f;
        if (a.l2norm) {
            rq = a.scale / sqrtf(sq + 1e-6f);
            rk = 1.f / sqrtf(sk + 1e-6f);
        }
        if (lane == 0) {
            nrm[3 * t] = rq;
            nrm[3 * t + 1] = rk;
            nrm[3 * t + 2] = sqk * rq * rk;
        }
    }
    __syncthreads();

    // 2. the r value heads in turn, each through the K tokens in registers
    for (int j = 0; j < r; ++j) {
        const int h = kh * r + j;
        if (j > 0) load_state(j);
        if (j + 1 < r) prefetch_state(j + 1);
        for (int t = 0; t < K; ++t) {
            const float rq = nrm[3 * t], rk = nrm[3 * t + 1], kq = nrm[3 * t + 2];
            const float* kt = ks + t * D;
            const float* qt = qs + t * D;
            float mk[4] = {0.f, 0.f, 0.f, 0.f}, mq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int p = 0; p < PASSES; ++p) {
                const int i = r0 + p * RPP;
                const float kv = kt[i] * rk, qv = qt[i] * rq;
                mk[0] = fmaf(s[p].x, kv, mk[0]); mk[1] = fmaf(s[p].y, kv, mk[1]);
                mk[2] = fmaf(s[p].z, kv, mk[2]); mk[3] = fmaf(s[p].w, kv, mk[3]);
                mq[0] = fmaf(s[p].x, qv, mq[0]); mq[1] = fmaf(s[p].y, qv, mq[1]);
                mq[2] = fmaf(s[p].z, qv, mq[2]); mq[3] = fmaf(s[p].w, qv, mq[3]);
            }
            *reinterpret_cast<float4*>(&red[r0 * D + cq * 4]) = make_float4(mk[0], mk[1], mk[2], mk[3]);
            *reinterpret_cast<float4*>(&red[(RPP + r0) * D + cq * 4]) = make_float4(mq[0], mq[1], mq[2], mq[3]);
            __syncthreads();
            const float eg = expf(gb[2 * (t * r + j)]);
            const float bt = gb[2 * (t * r + j) + 1];
            const float* vt = vs + (t * r + j) * D;
            float o2 = 0.f;
            for (int c = tid; c < D; c += NT) {
                float m = 0.f, pq = 0.f;
#pragma unroll
                for (int rr = 0; rr < RPP; ++rr) {
                    m += red[rr * D + c];
                    pq += red[(RPP + rr) * D + c];
                }
                const float delta = bt * (vt[c] - eg * m);
                ds[c] = delta;
                const float o = to_f(from_f<T>(eg * pq + kq * delta));
                os[c] = o;
                o2 = fmaf(o, o, o2);
            }
            o2 = warp_sum(o2);
            if (lane == 0) wsum[warp] = o2;
            __syncthreads();
            // S <- e^g S + k^ delta^T, kept in registers and written to slot t + 1
            float* S = a.state + ((int64_t)sl[t + 1] * a.H_v + h) * D * D;
            const float4 d4 = *reinterpret_cast<const float4*>(&ds[cq * 4]);
#pragma unroll
            for (int p = 0; p < PASSES; ++p) {
                const int i = r0 + p * RPP;
                const float kv = kt[i] * rk;
                float4 n;
                n.x = fmaf(kv, d4.x, eg * s[p].x);
                n.y = fmaf(kv, d4.y, eg * s[p].y);
                n.z = fmaf(kv, d4.z, eg * s[p].z);
                n.w = fmaf(kv, d4.w, eg * s[p].w);
                s[p] = n;
                __stcs(reinterpret_cast<float4*>(S + (int64_t)i * D) + cq, n);
            }
            float tot = 0.f;
#pragma unroll
            for (int ww = 0; ww < NW; ++ww) tot += wsum[ww];
            const float rs = rsqrtf(tot / (float)D + a.eps);
            const int64_t row = ((int64_t)b * K + t) * a.H_v + h;
            const float* z = zs + (t * r + j) * D;
            T* out = static_cast<T*>(a.out) + row * D;
            const T* nw = static_cast<const T*>(a.norm_w);
            for (int c = 2 * tid; c < D; c += 2 * NT) {
                const float2 g = silu2<T>(make_float2(z[c], z[c + 1]));
                const float2 res = __fmul2_rn(__fmul2_rn(make_float2(to_f(nw[c]), to_f(nw[c + 1])),
                                                         __fmul2_rn(make_float2(os[c], os[c + 1]), make_float2(rs, rs))),
                                              g);
                out[c] = from_f<T>(res.x);
                out[c + 1] = from_f<T>(res.y);
            }
            __syncthreads();  // red, ds, os and wsum are reused by the next token
        }
    }
}

// Verification for small batches: one CTA per (sequence, value head), the r
// value heads of a key head as a thread-block cluster, as the small-batch
// decode step.  The first CTA of the cluster convolves q and k over the K
// tokens (writing their conv states to the slots) and sends them to the others
// through distributed shared memory; every CTA convolves its head's v and runs
// its head through the K tokens with decode_verify_kernel's arithmetic, so the
// states and outputs are the same bit for bit.
template <typename T, int D, int NW>
__global__ void __launch_bounds__(NW * 32, (D >= 128 ? 2 : 1))
decode_verify_head_kernel(DecodeVerifyArgs a) {
    constexpr int NT = NW * 32;
    constexpr int TPR = D / 4;
    constexpr int RPP = NT / TPR;
    constexpr int PASSES = D / RPP;
    constexpr int V = Vec16<T>::N;
    static_assert(NT % TPR == 0 && D % RPP == 0 && NT >= D, "layout");

    const int r = a.H_v / a.H_k, K = a.K;
    const int b = blockIdx.x / a.H_v;
    const int h = blockIdx.x - b * a.H_v;
    const int kh = h / r, rank = h - kh * r;  // rank in the key head's cluster
    const bool cl = r > 1;
    if (cl) cluster_arrive_relaxed();  // this CTA has started (waited for before any remote store)
    const int32_t* sl = a.slots + (int64_t)b * (K + 1);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cq = tid % TPR;
    const int r0 = tid / TPR;
    const int C = 2 * a.H_k * D + a.H_v * D;

    extern __shared__ __align__(16) float vsm[];
    float* qs = vsm;                  // [K][D]
    float* ks = qs + K * D;           // [K][D]
    float* vs = ks + K * D;           // [K][D]
    float* zs = vs + K * D;           // [K][D]: the gate input z
    float* ds = zs + K * D;           // [D]
    float* os = ds + D;               // [D]
    float* red = os + D;              // [2][RPP][D]
    float* gb = red + 2 * RPP * D;    // [K][2]: g, beta
    float* nrm = gb + 2 * K;          // [K][3]: rq, rk, k.q rq rk
    float* wsum = nrm + 3 * K;        // [NW]

    const int64_t s_in = sl[0];
    {   // the head's state into L2 ahead of its register loads
        const char* S = reinterpret_cast<const char*>(a.state + (s_in * a.H_v + h) * D * D);
        for (int off = tid * 128; off < D * D * 4; off += NT * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(S + off));
    }
    // 1. conv over the K tokens of the channels this CTA owns (q and k in the
    //    first CTA of the cluster, then the head's v)
    {
        const T* x = static_cast<const T*>(a.x) + (int64_t)b * K * C;
        const T* w = static_cast<const T*>(a.conv_w);
        T* cs = static_cast<T*>(a.conv_state);
        const int g0 = rank == 0 ? 0 : 2;
        const int nvec = (3 - g0) * D / V;
        for (int e = tid; e < nvec; e += NT) {
            const int grp = g0 + (e * V) / D, i0 = e * V - (grp - g0) * D;
            const int c0 = grp == 0 ? kh * D + i0 : grp == 1 ? a.H_k * D + kh * D + i0 : 2 * a.H_k * D + h * D + i0;
            float st[3 * V], wt[4 * V];
#pragma unroll
            for (int k = 0; k < 3; ++k) load16(cs + (s_in * C + c0) * 3 + k * V, st + k * V);
#pragma unroll
            for (int k = 0; k < 4; ++k) load16(w + (int64_t)c0 * 4 + k * V, wt + k * V);
            float* dst = (grp == 0 ? qs : grp == 1 ? ks : vs) + i0;
            for (int t = 0; t < K; ++t) {
                float xv[V];
                load16(x + (int64_t)t * C + c0, xv);
#pragma unroll
                for (int q = 0; q < V; ++q) {
                    float acc = wt[q * 4] * st[q * 3];
                    acc = fmaf(wt[q * 4 + 1], st[q * 3 + 1], acc);
                    acc = fmaf(wt[q * 4 + 2], st[q * 3 + 2], acc);
                    acc = fmaf(wt[q * 4 + 3], xv[q], acc);
                    dst[t * D + q] = to_f(from_f<T>(silu_f(acc)));
                    st[q * 3] = st[q * 3 + 1];  // the window moves one token
                    st[q * 3 + 1] = st[q * 3 + 2];
                    st[q * 3 + 2] = xv[q];
                }
                T* out_cs = cs + ((int64_t)sl[t + 1] * C + c0) * 3;
#pragma unroll
                for (int k = 0; k < 3; ++k) store16(out_cs + k * V, st + k * V);
            }
        }
        for (int t = tid; t < K; t += NT) {
            const int64_t gi = ((int64_t)b * K + t) * a.H_v + h;
            gb[2 * t] = gate_g(to_f(static_cast<const T*>(a.a)[gi]), a.A_log[h], a.dt_bias[h]);
            gb[2 * t + 1] = sigmoid_f(to_f(static_cast<const T*>(a.b)[gi]));
        }
        const T* zg = static_cast<const T*>(a.z) + ((int64_t)b * K * a.H_v + h) * D;
        for (int e = tid; e < K * D / V; e += NT) {
            const int t = (e * V) / D, o = e * V - t * D;
            float zv[V];
            load16(zg + (int64_t)t * a.H_v * D + o, zv);
#pragma unroll
            for (int q = 0; q < V; ++q) zs[t * D + o + q] = zv[q];
        }
    }
    __syncthreads();
    if (cl) {
        // q and k of the K tokens from the first CTA to the others
        cluster_wait();
        if (rank == 0) {
            const int per = K * D / 2;  // float4s of qs and ks (contiguous)
            for (int e = tid; e < (r - 1) * per; e += NT) {
                const int dst = 1 + e / per, i = e - (dst - 1) * per;
                st_cluster_v4(qs + 4 * i, (uint32_t)dst, *reinterpret_cast<const float4*>(qs + 4 * i));
            }
        }
        cluster_sync();
    }
    float4 s[PASSES];
    {
        const float* S = a.state + (s_in * a.H_v + h) * D * D;
#pragma unroll
        for (int p = 0; p < PASSES; ++p)
            s[p] = __ldcs(reinterpret_cast<const float4*>(S + (int64_t)(r0 + p * RPP) * D) + cq);
    }
    for (int t = warp; t < K; t += NW) {
        float sq = 0.f, sk = 0.f, sqk = 0.f;
        for (int i = lane; i < D; i += 32) {
            sq = fmaf(qs[t * D + i], qs[t * D + i], sq);
            sk = fmaf(ks[t * D + i], ks[t * D + i], sk);
            sqk = fmaf(qs[t * D + i], ks[t * D + i], sqk);
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        sqk = warp_sum(sqk);
        float rq = a.scale, rk = 1.f;
        if (a.l2norm) {
            rq = a.scale / sqrtf(sq + 1e-6f);
            rk = 1.f / sqrtf(sk + 1e-6f);
        }
        if (lane == 0) {
            nrm[3 * t] = rq;
            nrm[3 * t + 1] = rk;
            nrm[3 * t + 2] = sqk * rq * rk;
        }
    }
    __syncthreads();

    // 2. the head through the K tokens, its state in registers
    for (int t = 0; t < K; ++t) {
        const float rq = nrm[3 * t], rk = nrm[3 * t + 1], kq = nrm[3 * t + 2];
        const float* kt = ks + t * D;
        const float* qt = qs + t * D;
        float mk[4] = {0.f, 0.f, 0.f, 0.f}, mq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int p = 0; p < PASSES; ++p) {
            const int i = r0 + p * RPP;
            const float kv = kt[i] * rk, qv = qt[i] * rq;
            mk[0] = fmaf(s[p].x, kv, mk[0]); mk[1] = fmaf(s[p].y, kv, mk[1]);
            mk[2] = fmaf(s[p].z, kv, mk[2]); mk[3] = fmaf(s[p].w, kv, mk[3]);
            mq[0] = fmaf(s[p].x, qv, mq[0]); mq[1] = fmaf(s[p].y, qv, mq[1]);
            mq[2] = fmaf(s[p].z, qv, mq[2]); mq[3] = fmaf(s[p].w, qv, mq[3]);
        }
        *reinterpret_cast<float4*>(&red[r0 * D + cq * 4]) = make_float4(mk[0], mk[1], mk[2], mk[3]);
        *reinterpret_cast<float4*>(&red[(RPP + r0) * D + cq * 4]) = make_float4(mq[0], mq[1], mq[2], mq[3]);
        __syncthreads();
        const float eg = expf(gb[2 * t]);
        const float bt = gb[2 * t + 1];
        const float* vt = vs + t * D;
        float o2 = 0.f;
        for (int c = tid; c < D; c += NT) {
            float m = 0.f, pq = 0.f;
#pragma unroll
            for (int rr = 0; rr < RPP; ++rr) {
                m += red[rr * D + c];
                pq += red[(RPP + rr) * D + c];
            }
            const float delta = bt * (vt[c] - eg * m);
            ds[c] = delta;
            const float o = to_f(from_f<T>(eg * pq + kq * delta));
            os[c] = o;
            o2 = fmaf(o, o, o2);
        }
        o2 = warp_sum(o2);
        if (lane == 0) wsum[warp] = o2;
        __syncthreads();
        float* S = a.state + ((int64_t)sl[t + 1] * a.H_v + h) * D * D;
        const float4 d4 = *reinterpret_cast<const float4*>(&ds[cq * 4]);
#pragma unroll
        for (int p = 0; p < PASSES; ++p) {
            const int i = r0 + p * RPP;
            const float kv = kt[i] * rk;
            float4 n;
            n.x = fmaf(kv, d4.x, eg * s[p].x);
            n.y = fmaf(kv, d4.y, eg * s[p].y);
            n.z = fmaf(kv, d4.z, eg * s[p].z);
            n.w = fmaf(kv, d4.w, eg * s[p].w);
            s[p] = n;
            __stcs(reinterpret_cast<float4*>(S + (int64_t)i * D) + cq, n);
        }
        float tot = 0.f;
#pragma unroll
        for (int ww = 0; ww < NW; ++ww) tot += wsum[ww];
        const float rs = rsqrtf(tot / (float)D + a.eps);
        const int64_t row = ((int64_t)b * K + t) * a.H_v + h;
        const float* z = zs + t * D;
        T* out = static_cast<T*>(a.out) + row * D;
        const T* nw = static_cast<const T*>(a.norm_w);
        for (int c = 2 * tid; c < D; c += 2 * NT) {
            const float2 g = silu2<T>(make_float2(z[c], z[c + 1]));
            const float2 res = __fmul2_rn(__fmul2_rn(make_float2(to_f(nw[c]), to_f(nw[c + 1])),
                                                     __fmul2_rn(make_float2(os[c], os[c + 1]), make_float2(rs, rs))),
                                          g);
            out[c] = from_f<T>(res.x);
            out[c + 1] = from_f<T>(res.y);
        }
        __syncthreads();  // red, ds, os and wsum are reused by the next token
    }
}

template <int D, int NW>
size_t verify_head_smem_bytes(int K) {
    constexpr int RPP = NW * 32 / (D / 4);
    return sizeof(float) * ((size_t)4 * K * D + 2 * D + 2 * RPP * D + 2 * K + 3 * K + NW);
}

template <int D, int NW>
size_t verify_smem_bytes(int K, int r) {
    constexpr int RPP = NW * 32 / (D / 4);
    return sizeof(float) * ((size_t)2 * K * D + (size_t)2 * K * r * D + 2 * D + 2 * RPP * D + 2 * K * r + 3 * K + NW);
}

template <typename T>
cudaError_t decode_verify_t(const DecodeVerifyArgs& a, cudaStream_t s) {
    const unsigned units = (unsigned)(a.B * a.H_k);
    if (units == 0 || a.K == 0) return cudaSuccess;
    const int r = a.H_v / a.H_k;
    if (r > 8 || a.K > kVerifyMaxK) return cudaErrorNotSupported;
    if ((int64_t)units * 2 <= device_sms()) {
        // few (sequence, key head) units: one clustered CTA per value head (27B,
        // B = 1, K = 4: 21.8 against 34.8 us; from B = 8 the per-key-head CTAs
        // are faster)
        const unsigned heads = (unsigned)(a.B * a.H_v);
        if (a.D == 128) {
            const size_t smem = verify_head_smem_bytes<128, 8>(a.K);
            cudaError_t e = cudaFuncSetAttribute(decode_verify_head_kernel<T, 128, 8>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            return e != cudaSuccess ? e
                                    : launch_cluster(decode_verify_head_kernel<T, 128, 8>, heads, 256, smem,
                                                     (unsigned)r, s, a);
        }
        const size_t smem = verify_head_smem_bytes<16, 1>(a.K);
        cudaError_t e = cudaFuncSetAttribute(decode_verify_head_kernel<T, 16, 1>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        return e != cudaSuccess ? e
                                : launch_cluster(decode_verify_head_kernel<T, 16, 1>, heads, 32, smem, (unsigned)r, s, a);
    }
    if (a.D == 128) {
        const size_t smem = verify_smem_bytes<128, 8>(a.K, r);
        cudaError_t e = cudaFuncSetAttribute(decode_verify_kernel<T, 128, 8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        decode_verify_kernel<T, 128, 8><<<units, 256, smem, s>>>(a);
    } else {
        const size_t smem = verify_smem_bytes<16, 1>(a.K, r);
        cudaError_t e = cudaFuncSetAttribute(decode_verify_kernel<T, 16, 1>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        decode_verify_kernel<T, 16, 1><<<units, 32, smem, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_step(const DecodeStepArgs& a, gdn_dtype_t dt, cudaStream_t s) {
    return dt == GDN_BF16 ? decode_step_t<bf16>(a, s) : decode_step_t<float>(a, s);
}

cudaError_t launch_decode_verify(const DecodeVerifyArgs& a, gdn_dtype_t dt, cudaStream_t s) {
    return dt == GDN_BF16 ? decode_verify_t<bf16>(a, s) : decode_verify_t<float>(a, s);
}

cudaError_t launch_recurrent_decode(const DeltaArgs& a, gdn_dtype_t dt, cudaStream_t s) {
    return dt == GDN_BF16 ? decode_t<bf16>(a, s) : decode_t<float>(a, s);
}

}  // namespace gdn
