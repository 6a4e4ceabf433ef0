// gdn_layer_prefill_host: the layer core (conv1d + SiLU -> chunked delta rule
// -> RMSNormGated) for one sequence whose activations live in page-locked host
// memory.  The tokens run in pieces, each through four streams:
//   copy-in:   piece p's inputs
//   pre:       conv1d of piece p, then the chunk-local (intra) kernels
//   caller's:  the state chain of piece p (in order, carrying the state), RMSNormGated
//   copy-out:  piece p's output
// so the copies, the chunk-parallel work of piece p + 1 and the sequential
// chain of piece p overlap; only the chain and the norm are serial per piece.
// The conv state and the recurrent state carry from piece to piece in place on
// the device.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr int kMaxDev = 128;
std::mutex g_host_mu;
cudaStream_t g_copy_in[kMaxDev], g_copy_out[kMaxDev], g_pre[kMaxDev];
unsigned long long g_stream_ctx[kMaxDev];  // context the streams of a device belong to

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// pieces in flight: piece p reuses the buffers of piece p - kSlots
constexpr int kSlots = 3;

struct Slot {
    size_t qkv, z, y, o, out;  // byte offsets in the workspace
};

struct HostLayout {
    int64_t piece;  // tokens per piece (a multiple of 64 unless the whole sequence is one piece)
    size_t a, b;    // the whole sequence's gate inputs (copied once)
    size_t cst[2];  // conv state between pieces, alternating (never read and written by one call)
    Slot slot[kSlots];
    size_t chunk_ws[kSlots], chunk_ws_bytes, total;
};

HostLayout host_layout(int64_t T, int H_k, int H_v, int D, int es, bool tensor_core) {
    HostLayout L;
    // about 16 pieces of a multiple of 64 tokens, at least 512 (a short
    // sequence is one piece)
    int64_t p = T;
    if (T > 1024) {
        p = (T + 15) / 16;
        p = ((p + 63) / 64) * 64;
        if (p < 512) p = 512;
    }
    L.piece = p;
    const size_t C = (size_t)(2 * H_k + H_v) * D, O = (size_t)H_v * D;
    size_t off = 0;
    L.a = off; off = align256(off + (size_t)T * H_v * es);
    L.b = off; off = align256(off + (size_t)T * H_v * es);
    for (int i = 0; i < 2; ++i) {
        L.cst[i] = off;
        off = align256(off + (size_t)(2 * H_k + H_v) * D * 3 * es);
    }
    for (int s = 0; s < kSlots; ++s) {
        Slot& q = L.slot[s];
        q.qkv = off; off = align256(off + (size_t)p * C * es);
        q.z = off;   off = align256(off + (size_t)p * O * es);
        q.y = off;   off = align256(off + (size_t)p * C * es);
        q.o = off;   off = align256(off + (size_t)p * O * es);
        q.out = off; off = align256(off + (size_t)p * O * es);
    }
    L.chunk_ws_bytes = tensor_core ? align256(chunk_split_workspace_bytes(1, p, H_v)) : 0;
    for (int s = 0; s < kSlots; ++s) {
        L.chunk_ws[s] = off;
        off += L.chunk_ws_bytes;
    }
    L.total = off;
    return L;
}

// Piece plan: pieces of L.piece tokens, except that when the sequence is a
// whole number (>= 2) of full pieces the last one is cut into 3/4 and 1/4
// (multiples of 64): after the last copy in, only the small last piece's
// kernels and copy out remain.
struct PiecePlan {
    int64_t full;  // leading pieces of L.piece tokens
    int64_t tail[2];
    int n_tail;
};

PiecePlan piece_plan(int64_t T, int64_t P) {
    PiecePlan q;
    q.n_tail = 0;
    q.full = (T + P - 1) / P;
    const int64_t quarter = (P / 4) & ~(int64_t)63;
    if (T > P && T % P == 0 && quarter >= 64) {
        q.full = T / P - 1;
        q.tail[0] = P - quarter;
        q.tail[1] = quarter;
        q.n_tail = 2;
    }
    return q;
}

int64_t plan_count(const PiecePlan& q) { return q.full + q.n_tail; }

// tokens [t0, t0 + tp) of piece p
void plan_span(const PiecePlan& q, int64_t T, int64_t P, int64_t p, int64_t& t0, int64_t& tp) {
    if (p < q.full) {
        t0 = p * P;
        tp = T - t0 < P ? T - t0 : P;
        return;
    }
    t0 = q.full * P;
    for (int64_t i = 0; i < p - q.full; ++i) t0 += q.tail[i];
    tp = q.tail[p - q.full];
}

cudaError_t copy_streams(cudaStream_t* in, cudaStream_t* out, cudaStream_t* pre) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_host_mu);
    // created once per device context: after a device reset the old handles
    // belong to a destroyed context and new streams are made
    unsigned long long ctx = current_context_id();
    if (ctx == 0) {
        if ((e = cudaFree(nullptr)) != cudaSuccess) return e;  // makes the device's context current
        ctx = current_context_id();
    }
    if (g_copy_in[dev] == nullptr || ctx != g_stream_ctx[dev]) {
        e = cudaStreamCreateWithFlags(&g_copy_in[dev], cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&g_copy_out[dev], cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&g_pre[dev], cudaStreamNonBlocking);
        if (e != cudaSuccess) {
            g_copy_in[dev] = nullptr;
            return e;
        }
        g_stream_ctx[dev] = ctx;
    }
    *in = g_copy_in[dev];
    *out = g_copy_out[dev];
    *pre = g_pre[dev];
    return cudaSuccess;
}

}  // namespace

size_t layer_prefill_host_workspace_bytes(int64_t T, int H_k, int H_v, int D, int es, bool tensor_core) {
    return T > 0 ? host_layout(T, H_k, H_v, D, es, tensor_core).total : 0;
}

int64_t layer_prefill_host_piece(int64_t T, int H_k, int H_v, int D, int es, bool tensor_core) {
    return host_layout(T, H_k, H_v, D, es, tensor_core).piece;
}

int64_t layer_prefill_host_pieces(int64_t T, int H_k, int H_v, int D, int es, bool tensor_core) {
    return T > 0 ? plan_count(piece_plan(T, host_layout(T, H_k, H_v, D, es, tensor_core).piece)) : 0;
}

cudaError_t launch_layer_prefill_host(const HostLayerArgs& h, gdn_dtype_t dt, void* workspace,
                                      cudaStream_t s) {
    const int es = dt == GDN_BF16 ? 2 : 4;
    const bool tc = dt == GDN_BF16 && h.D == 128;
    const HostLayout L = host_layout(h.T, h.H_k, h.H_v, h.D, es, tc);
    const size_t C = (size_t)(2 * h.H_k + h.H_v) * h.D, O = (size_t)h.H_v * h.D;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t cin, cout, pre;
    cudaError_t e = copy_streams(&cin, &cout, &pre);
    if (e != cudaSuccess) return e;
    constexpr int NEV = 5 * kSlots + 1;
    cudaEvent_t ev[NEV];  // in (qkv), in (z), comp, out, pre per slot; start
    int made = 0;
    for (; made < NEV && e == cudaSuccess; ++made)
        e = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming);
    cudaEvent_t* ev_in = ev;
    cudaEvent_t* ev_comp = ev + kSlots;
    cudaEvent_t* ev_out = ev + 2 * kSlots;
    cudaEvent_t* ev_pre = ev + 3 * kSlots;
    cudaEvent_t* ev_inz = ev + 4 * kSlots;
    cudaEvent_t ev_start = ev[5 * kSlots];
    // the other streams start after whatever the caller queued on `s`
    if (e == cudaSuccess) e = cudaEventRecord(ev_start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cin, ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cout, ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pre, ev_start, 0);
    // the gate inputs of the whole sequence (small) in two copies
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(ws + L.a, h.h_a, (size_t)h.T * h.H_v * es, cudaMemcpyHostToDevice, cin);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(ws + L.b, h.h_b, (size_t)h.T * h.H_v * es, cudaMemcpyHostToDevice, cin);
    const PiecePlan plan = piece_plan(h.T, L.piece);
    const int64_t n_piece = plan_count(plan);
    for (int64_t p = 0; p < n_piece && e == cudaSuccess; ++p) {
        const int sl = (int)(p % kSlots);
        const Slot& q = L.slot[sl];
        int64_t t0, tp;
        plan_span(plan, h.T, L.piece, p, t0, tp);
        const uint8_t* hq = static_cast<const uint8_t*>(h.h_qkv);
        // inputs of piece p, once piece p - kSlots (same slot) has finished with the
        // slot's buffers and chunk workspace
        if (p >= kSlots) e = cudaStreamWaitEvent(cin, ev_comp[sl], 0);
        // qkv first, on its own event: the conv and the chunk kernels need only it,
        // and only the norm waits for z
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(ws + q.qkv, hq + (size_t)t0 * C * es, (size_t)tp * C * es, cudaMemcpyHostToDevice, cin);
        if (e == cudaSuccess) e = cudaEventRecord(ev_in[sl], cin);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(ws + q.z, static_cast<const uint8_t*>(h.h_z) + (size_t)t0 * O * es,
                                (size_t)tp * O * es, cudaMemcpyHostToDevice, cin);
        if (e == cudaSuccess) e = cudaEventRecord(ev_inz[sl], cin);
        // conv and the chunk-local kernels on the pre stream once the inputs are in
        if (e == cudaSuccess) e = cudaStreamWaitEvent(pre, ev_in[sl], 0);
        if (e == cudaSuccess) {
            ConvArgs c;
            c.x = ws + q.qkv; c.w = h.conv_w; c.cu = nullptr; c.n_seq = 1; c.T = tp; c.C = (int)C;
            // piece p reads the state piece p - 1 wrote and writes the other buffer
            // (the last piece writes conv_state_out), so no conv call has its
            // state_out aliasing its state_in
            c.state_in = p == 0 ? h.conv_state_in : ws + L.cst[(p - 1) & 1];
            c.state_out = p == n_piece - 1 ? h.conv_state_out : ws + L.cst[p & 1];
            c.ckpt_every = 0; c.ckpt = nullptr; c.ckpt_rows = 0; c.silu = 1; c.y = ws + q.y;
            e = launch_conv1d_fwd(c, dt, pre);
        }
        if (e == cudaSuccess) {
            DeltaArgs d = {};
            d.qkv = ws + q.y; d.a = ws + L.a + (size_t)t0 * h.H_v * es;
            d.b = ws + L.b + (size_t)t0 * h.H_v * es; d.A_log = h.A_log; d.dt_bias = h.dt_bias;
            d.cu = nullptr; d.n_seq = 1; d.T = tp; d.H_k = h.H_k; d.H_v = h.H_v; d.D = h.D;
            d.S0 = p == 0 ? h.initial_state : h.final_state;
            d.S_final = h.final_state;
            d.scale = h.scale; d.l2norm = h.l2norm; d.o = ws + q.o;
            // the chain (and the norm after it) on the caller's stream, once the
            // output slot has been copied out
            if (e == cudaSuccess && p >= kSlots) e = cudaStreamWaitEvent(s, ev_out[sl], 0);
            if (e == cudaSuccess) {
                if (tc) {
                    e = launch_chunk_split_two(d, ws + L.chunk_ws[sl], L.chunk_ws_bytes, pre, s, ev_pre[sl]);
                } else {
                    e = cudaEventRecord(ev_pre[sl], pre);
                    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_pre[sl], 0);
                    if (e == cudaSuccess) e = launch_chunk_ffma(d, dt, s);
                }
            }
        }
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_inz[sl], 0);
        if (e == cudaSuccess)
            e = launch_rmsnorm_gated(ws + q.o, ws + q.z, h.norm_w, h.eps, tp, h.H_v, h.D, ws + q.out, dt, s);
        if (e == cudaSuccess) e = cudaEventRecord(ev_comp[sl], s);
        // output of piece p
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cout, ev_comp[sl], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<uint8_t*>(h.h_out) + (size_t)t0 * O * es, ws + q.out,
                                (size_t)tp * O * es, cudaMemcpyDeviceToHost, cout);
        if (e == cudaSuccess) e = cudaEventRecord(ev_out[sl], cout);
    }
    // join: the caller's stream waits for the last copies out
    for (int sl = 0; sl < kSlots && e == cudaSuccess; ++sl)
        if (n_piece > sl) e = cudaStreamWaitEvent(s, ev_out[(n_piece - 1 - sl) % kSlots], 0);
    for (int i = 0; i < made; ++i) cudaEventDestroy(ev[i]);  // released once complete
    return e;
}

}  // namespace gdn
