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

}  // namespace

cudaError_t launch_recurrent_decode(const DeltaArgs& a, gdn_dtype_t dt, cudaStream_t s) {
    return dt == GDN_BF16 ? decode_t<bf16>(a, s) : decode_t<float>(a, s);
}

}  // namespace gdn
