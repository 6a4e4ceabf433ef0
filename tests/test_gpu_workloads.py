"""GPU parity of the whole layer core on the five workloads, at full size.

Where the full oracle is affordable (tiny f32, the 4096-token 27B prefill) it
runs over every head; for the batched decode, the varlen Coder-Next prefill
and the 262144-token prefill the GPU runs the full workload and the oracle
recomputes sampled sequences or value heads one by one (heads, sequences and
conv channels are independent, so the sample is exact).  Conv state and conv
checkpoints are bit copies of raw inputs and are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_core_gb300 as gdn
import oracle
import workloads as W
from gpu_util import TOL, assert_close, head_channels, host, oracle_heads_prefill, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _dims(s):
    return gdn.GDNDims(s.H_k, s.H_v, s.d_k, s.d_v)


def _run_prefill(inp, shape, ckpt_every=0):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    r = gdn.gdn_layer_prefill(d["mixed_qkv"], d["z"], d["a"], d["b"], d["conv_w"], d["A_log"],
                              d["dt_bias"], d["norm_w"], _dims(shape), cu_seqlens=d["cu_seqlens"],
                              initial_state=d["S0"], conv_state=d["conv_state0"],
                              ckpt_every=ckpt_every)
    torch.cuda.synchronize()
    return r


def _check_conv_state_bytes(inp, r, shape, ckpt_every=0):
    """Conv state / checkpoints are the 3 newest raw inputs (state_in prepended)."""
    cu = inp["cu_seqlens"].tolist()
    x = inp["mixed_qkv"]
    got = r["conv_state"].cpu()
    row = 0
    for i in range(len(cu) - 1):
        s, e = cu[i], cu[i + 1]
        L = e - s
        ext = x[s:e].T  # [C, L]
        if L < 3:
            head = (inp["conv_state0"][i] if inp["conv_state0"] is not None
                    else torch.zeros((shape.conv_dim, 3), dtype=x.dtype))
            ext = torch.cat([head, ext], dim=1)
        assert torch.equal(got[i], ext[:, -3:]), f"conv state of sequence {i}"
        if ckpt_every:
            for m in range(1, L // ckpt_every + 1):
                assert torch.equal(r["conv_ckpt"][row].cpu(),
                                   x[s + m * ckpt_every - 3:s + m * ckpt_every].T), \
                    f"conv ckpt {row}"
                row += 1


def test_tiny_f32_layer():
    w = W.WORKLOADS["tiny_f32"]
    s = w.shape
    inp = W.workload_inputs(w.name)
    r = _run_prefill(inp, s)
    f = W.to_f64
    ref = oracle.layer_prefill(f(inp["mixed_qkv"]), f(inp["z"]), f(inp["a"]), f(inp["b"]),
                               f(inp["conv_w"]), f(inp["A_log"]), f(inp["dt_bias"]),
                               f(inp["norm_w"]), s.H_k, s.H_v, s.d_k, s.d_v)
    assert_close("out", host(r["out"]), ref["out"], TOL[torch.float32])
    assert_close("S", host(r["final_state"]), ref["S"], TOL[torch.float32], per_head_axis=1)
    assert np.array_equal(host(r["conv_state"]), ref["conv_state"])


def test_qwen36_27b_prefill_layer():
    w = W.WORKLOADS["qwen36_27b_prefill"]
    s = w.shape
    inp = W.workload_inputs(w.name)
    r = _run_prefill(inp, s)
    f = W.to_f64
    ref = oracle.layer_prefill(f(inp["mixed_qkv"]), f(inp["z"]), f(inp["a"]), f(inp["b"]),
                               f(inp["conv_w"]), f(inp["A_log"]), f(inp["dt_bias"]),
                               f(inp["norm_w"]), s.H_k, s.H_v, s.d_k, s.d_v)
    tol = TOL[torch.bfloat16]
    out = host(r["out"])
    assert_close("out", out, ref["out"], tol)
    assert_close("out per head", out.reshape(-1, s.H_v, s.d_v), ref["out"].reshape(-1, s.H_v, s.d_v),
                 tol, per_head_axis=1)
    assert_close("S", host(r["final_state"]), ref["S"], tol, per_head_axis=1)
    assert np.array_equal(host(r["conv_state"]), ref["conv_state"])


def test_qwen36_27b_decode_64x256():
    w = W.WORKLOADS["qwen36_27b_decode"]
    s = w.shape
    inp = W.workload_inputs(w.name)
    dims = _dims(s)
    dev = {k: v.cuda() for k, v in inp.items()}
    S = dev["S0"].clone()
    cs = dev["conv_state0"].clone()
    outs = []
    for t in range(w.decode_steps):
        outs.append(gdn.gdn_layer_decode(dev["qkv"][t], dev["z"][t], dev["a"][t], dev["b"][t],
                                         dev["conv_w"], dev["A_log"], dev["dt_bias"],
                                         dev["norm_w"], dims, S, cs))
    torch.cuda.synchronize()
    outs = torch.stack(outs)  # [steps, B, H_v*d_v]
    # oracle on sampled sequences, every step
    f = W.to_f64
    seqs = [0, 17, 42, 63]
    S_ref = f(inp["S0"][seqs])
    cs_ref = f(inp["conv_state0"][seqs])
    tol = TOL[torch.bfloat16]
    for t in range(w.decode_steps):
        out_ref, S_ref, cs_ref, _ = oracle.layer_decode_step(
            f(inp["qkv"][t, seqs]), f(inp["z"][t, seqs]), f(inp["a"][t, seqs]),
            f(inp["b"][t, seqs]), f(inp["conv_w"]), f(inp["A_log"]), f(inp["dt_bias"]),
            f(inp["norm_w"]), s.H_k, s.H_v, s.d_k, s.d_v, S_ref, cs_ref)
        e = rel_l2(host(outs[t, seqs]), out_ref)
        assert e <= tol, f"step {t}: out rel-L2 {e:.3e}"
    assert_close("S final", host(S[seqs]), S_ref, tol, per_head_axis=1)
    assert np.array_equal(host(cs[seqs]), cs_ref)
    assert torch.isfinite(outs).all() and torch.isfinite(S).all()


def test_coder_next_varlen_resumed_prefill():
    w = W.WORKLOADS["coder_next_varlen"]
    s = w.shape
    L = np.array(w.lengths)
    assert L.sum() == 32768 and len(L) == 8 and np.any(L % 64 != 0)
    inp = W.workload_inputs(w.name)
    r = _run_prefill(inp, s)
    _check_conv_state_bytes(inp, r, s)
    heads = [0, 13, 31]
    refs = oracle_heads_prefill(inp, s, heads)
    tol = TOL[torch.bfloat16]
    out = r["out"].view(-1, s.H_v, s.d_v)
    for h in heads:
        ref = refs[h]
        assert_close(f"out head {h}", host(out[:, h]), ref["out"], tol)
        assert_close(f"S head {h}", host(r["final_state"][:, h]), ref["S"][:, 0], tol,
                     per_head_axis=0)
        assert np.array_equal(host(r["conv_state"][:, head_channels(s, h)]), ref["conv_state"])
    assert torch.isfinite(r["out"]).all() and torch.isfinite(r["final_state"]).all()


# one decode step's output row of one head (128 bf16 values), config-4 tail
STEP_TOL = 2.5e-2


@pytest.mark.slow
def test_qwen36_27b_long_prefill_ckpts_then_decode():
    w = W.WORKLOADS["qwen36_27b_long"]
    s = w.shape
    inp = W.workload_inputs(w.name)
    r = _run_prefill(inp, s, ckpt_every=w.ckpt_every)
    assert r["state_ckpt"].shape[0] == 64 and r["conv_ckpt"].shape[0] == 64
    _check_conv_state_bytes(inp, r, s, ckpt_every=w.ckpt_every)
    heads = [5, 40]
    refs = oracle_heads_prefill(inp, s, heads, ckpt_every=w.ckpt_every)
    tol = TOL[torch.bfloat16]
    out = r["out"].view(-1, s.H_v, s.d_v)
    for h in heads:
        ref = refs[h]
        assert_close(f"out head {h}", host(out[:, h]), ref["out"], tol)
        assert_close(f"S head {h}", host(r["final_state"][:, h]), ref["S"][:, 0], tol)
        assert_close(f"ckpts head {h}", host(r["state_ckpt"][:, h]), ref["S_ckpt"][:, 0], tol,
                     per_head_axis=0)
        assert np.array_equal(host(r["conv_ckpt"][:, head_channels(s, h)]), ref["conv_ckpt"])
    # the last checkpoint is the final state (4096 divides 262144)
    assert torch.equal(r["state_ckpt"][-1], r["final_state"][0])
    assert torch.isfinite(r["out"]).all()
    del inp["mixed_qkv"], inp["z"]
    # 128 decode steps (B = 1) from the final states
    dec = W.decode_inputs(s, w.dtype, 1, w.decode_steps, seed=w.seed + 100)
    dims = _dims(s)
    dd = {k: v.cuda() for k, v in dec.items()}
    S, cs = r["final_state"].clone(), r["conv_state"].clone()
    p = {k: inp[k].cuda() for k in ("conv_w", "A_log", "dt_bias", "norm_w")}
    outs = []
    for t in range(w.decode_steps):
        outs.append(gdn.gdn_layer_decode(dd["qkv"][t], dd["z"][t], dd["a"][t], dd["b"][t],
                                         p["conv_w"], p["A_log"], p["dt_bias"], p["norm_w"],
                                         dims, S, cs))
    torch.cuda.synchronize()
    outs = torch.stack(outs)[:, 0].view(w.decode_steps, s.H_v, s.d_v)
    f = W.to_f64
    for h in heads:
        ch = head_channels(s, h)
        S_h, cs_h = refs[h]["S"], refs[h]["conv_state"]
        ref_steps = []
        for t in range(w.decode_steps):
            o_ref, S_h, cs_h, _ = oracle.layer_decode_step(
                f(dec["qkv"][t][:, ch]), f(dec["z"][t][:, h * s.d_v:(h + 1) * s.d_v]),
                f(dec["a"][t][:, h:h + 1]), f(dec["b"][t][:, h:h + 1]), f(inp["conv_w"][ch]),
                f(inp["A_log"][h:h + 1]), f(inp["dt_bias"][h:h + 1]), f(inp["norm_w"]), 1, 1,
                s.d_k, s.d_v, S_h, cs_h)
            ref_steps.append(o_ref[0])
        # rel-L2 per output tensor (this head's 128-step decode output) at the
        # bf16 tolerance, and every single step -- one head's 128-value output
        # row -- within STEP_TOL: a row carries the bf16 roundings of the conv
        # output, o and out on its own, and those alone, applied to the
        # oracle's exact states, put single rows of these two heads at up to
        # 1.05e-2 and 1.99e-2
        got, ref = host(outs[:, h]), np.stack(ref_steps)
        worst = max(rel_l2(got[t], ref[t]) for t in range(len(ref)))
        e = assert_close(f"decode out head {h}", got, ref, tol)
        print(f"decode head {h}: rel-L2 {e:.2e}, worst single step {worst:.2e}")
        assert worst <= STEP_TOL, f"decode head {h}: worst single step rel-L2 {worst:.3e} > {STEP_TOL:.1e}"
        assert_close(f"decode S head {h}", host(S[0, h]), S_h[0, 0], tol)


def _host_prefill(inp, shape):
    pin = {k: inp[k].pin_memory() for k in ("mixed_qkv", "z", "a", "b")}
    dev = {k: (inp[k].cuda() if inp[k] is not None else None)
           for k in ("conv_w", "A_log", "dt_bias", "norm_w", "S0", "conv_state0")}
    r = gdn.gdn_layer_prefill_host(pin["mixed_qkv"], pin["z"], pin["a"], pin["b"], dev["conv_w"],
                                   dev["A_log"], dev["dt_bias"], dev["norm_w"], _dims(shape),
                                   initial_state=dev["S0"], conv_state_in=dev["conv_state0"])
    torch.cuda.synchronize()
    gdn.gdn_sync_status()
    return r


@pytest.mark.parametrize("T,init", [(4096, True), (3000, True), (64, True), (1, True), (513, False),
                                    (1100, True), (5000, False)])
def test_host_streamed_prefill_equals_device_prefill(T, init):
    """gdn_layer_prefill_host (pinned host buffers, pieces of 64-aligned tokens,
    copies overlapped with the kernels) gives the device path's result bit for
    bit -- the pieces cut at chunk boundaries and the states carry exactly --
    and matches the oracle on sampled heads; one token, a piece and one token,
    more tokens than the 4096-token cut, and zero initial states included."""
    shape = W.QWEN36_27B
    inp = W.layer_inputs(shape, torch.bfloat16, [T], seed=31, init_state=init)
    dims = _dims(shape)
    piece = gdn._lib.load().gdn_layer_prefill_host_piece(T, gdn._dims(dims), gdn._lib.GDN_BF16)
    assert piece % 64 == 0 or piece == T
    r_h = _host_prefill(inp, shape)
    r_d = _run_prefill(inp, shape)
    assert torch.equal(r_h["out"], r_d["out"].cpu())
    assert torch.equal(r_h["final_state"].cpu(), r_d["final_state"].cpu())
    assert torch.equal(r_h["conv_state"].cpu(), r_d["conv_state"].cpu())
    heads = [0, shape.H_v - 1]
    ref = oracle_heads_prefill(inp, shape, heads)
    for h in heads:
        sl = slice(h * shape.d_v, (h + 1) * shape.d_v)
        assert rel_l2(host(r_h["out"])[:, sl], ref[h]["out"]) <= TOL[torch.bfloat16]


def _resume_inputs(inp, r, lengths, N, m):
    """Inputs of the run resumed from checkpoint m[i] (token m[i] * N) of each
    sequence of an uninterrupted run r with checkpoints every N tokens: the
    remaining tokens, the state checkpoint as initial state and the conv
    checkpoint (the 3 raw inputs before the resume point) as conv state."""
    cu = [0] + list(np.cumsum(lengths))
    rows0 = [0] + list(np.cumsum([L // N for L in lengths]))
    keep, rest, rows = [], [], []
    for i, L in enumerate(lengths):
        assert 1 <= m[i] <= L // N
        keep.append(torch.arange(cu[i] + m[i] * N, cu[i + 1]))
        rest.append(L - m[i] * N)
        rows.append(rows0[i] + m[i] - 1)
    idx = torch.cat(keep)
    res = {k: inp[k][idx] for k in ("mixed_qkv", "z", "a", "b")}
    for k in ("conv_w", "A_log", "dt_bias", "norm_w"):
        res[k] = inp[k]
    res["cu_seqlens"] = W.cu_seqlens_of(rest)
    res["S0"] = r["state_ckpt"][rows].cpu()
    res["conv_state0"] = r["conv_ckpt"][rows].cpu()
    return res, idx, rest, rows0


@pytest.mark.parametrize("lengths,N,m", [
    ([3000], 64, [1]),
    ([3000], 192, [7]),
    ([4096], 1024, [3]),
    ([1000, 2500, 640], 128, [2, 19, 5]),  # the last sequence resumes at its end
], ids=["N64-first", "N192-mid", "N1024-last", "varlen-N128"])
def test_resume_from_checkpoint_is_bit_identical(lengths, N, m):
    """Prefix reuse: resuming each sequence from its mid-sequence checkpoint (state
    and conv checkpoints of an uninterrupted run) gives the uninterrupted run's
    remaining outputs, final states, conv states and later checkpoints bit for
    bit, whatever the alignment of the checkpoint cadence with the chunks."""
    shape = W.QWEN36_27B
    inp = W.layer_inputs(shape, torch.bfloat16, lengths, seed=41, init_state=True)
    r = _run_prefill(inp, shape, ckpt_every=N)
    res, idx, rest, rows0 = _resume_inputs(inp, r, lengths, N, m)
    r2 = _run_prefill(res, shape, ckpt_every=N)
    assert torch.equal(r2["out"], r["out"][idx.cuda()])
    assert torch.equal(r2["final_state"], r["final_state"])
    assert torch.equal(r2["conv_state"], r["conv_state"])
    row = 0
    for i, L in enumerate(lengths):
        later = L // N - m[i]
        assert later == rest[i] // N
        if later:
            a0 = rows0[i] + m[i]
            assert torch.equal(r2["state_ckpt"][row:row + later], r["state_ckpt"][a0:a0 + later])
            assert torch.equal(r2["conv_ckpt"][row:row + later], r["conv_ckpt"][a0:a0 + later])
        row += later
    assert torch.isfinite(r["out"]).all()
