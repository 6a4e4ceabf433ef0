"""Seeded random layer configurations on the GPU against the f64 oracle.

Each case draws its own head counts (H_k in 1..4, r = H_v / H_k in 1..4), packed
sequence lengths (empty, 1..3 tokens, around one and two chunks), checkpoint
cadence, chunk size (16, 32, 64), solve form and whether the call resumes
from initial states.  The one-call layer prefill must equal the three separate
calls bit for bit and the oracle (cortex GatedDeltaNet commit, "Block",
"Delta rule (recurrent, per-token)", "Output") within the dtype's tolerance;
the conv state and checkpoints are raw inputs and must match exactly.  Three
fused decode steps then continue every sequence from the prefill's states:
their states against the oracle's single-token steps, their output rows
against the same steps with the conv output and the rule's output rounded to
the activation dtype, as the calls hand them on, both at the dtype's
tolerance.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_core_gb300 as gdn
import oracle
import workloads as W
from gpu_util import TOL, assert_close, host, oracle_step_in_activation_dtype, rounded_to

pytestmark = pytest.mark.gpu

LENGTH_POOL = [0, 1, 2, 3, 17, 63, 64, 65, 100, 128, 129, 191, 200, 257, 300]
DECODE_STEPS = 3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def draw_case(seed: int, dtype: torch.dtype) -> dict:
    """The configuration of case `seed`: a pure function of the seed."""
    g = np.random.default_rng(1000 + seed)
    H_k = int(g.choice([1, 2, 4]))
    r = int(g.integers(1, 5))
    d = 128 if dtype == torch.bfloat16 else int(g.choice([16, 128]))
    n_seq = int(g.integers(1, 7))
    lengths = [int(x) for x in g.choice(LENGTH_POOL, size=n_seq)]
    if sum(lengths) == 0:
        lengths[0] = 65
    chunk = int(g.choice([16, 32, 64]))
    return {
        "shape": W.GDNShape(H_k=H_k, H_v=H_k * r, d_k=d, d_v=d),
        "lengths": lengths,
        "ckpt_every": int(g.choice([0, 64, 128])),
        "chunk": chunk,
        "solve": "neumann" if dtype == torch.bfloat16 and chunk == 64 and g.random() < 0.25 else "direct",
        "init_state": bool(g.random() < 0.6),
    }


def _dims(s):
    return gdn.GDNDims(s.H_k, s.H_v, s.d_k, s.d_v)


CASES = [(torch.bfloat16, i) for i in range(30)] + [(torch.float32, i) for i in range(30, 40)]


@pytest.mark.parametrize("dtype,seed", CASES, ids=[f"{'bf16' if d == torch.bfloat16 else 'f32'}-{i}" for d, i in CASES])
def test_random_layer_case(dtype, seed):
    c = draw_case(seed, dtype)
    s, lengths, N = c["shape"], c["lengths"], len(c["lengths"])
    inp = W.layer_inputs(s, dtype, lengths, seed=2000 + seed, init_state=c["init_state"])
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    dims = _dims(s)
    args = (d["mixed_qkv"], d["z"], d["a"], d["b"], d["conv_w"], d["A_log"], d["dt_bias"], d["norm_w"], dims)
    kw = dict(cu_seqlens=d["cu_seqlens"], initial_state=d["S0"], conv_state=d["conv_state0"],
              ckpt_every=c["ckpt_every"], solve=c["solve"], chunk=c["chunk"])
    one = gdn.gdn_layer_prefill(*args, **kw)
    sep = gdn.gdn_layer_prefill(*args, return_intermediates=True, **kw)
    torch.cuda.synchronize()
    gdn.gdn_sync_status()
    for k in ("out", "final_state", "conv_state", "state_ckpt", "conv_ckpt"):
        if sep[k] is None:
            assert one[k] is None, k
        else:
            assert torch.equal(one[k], sep[k]), f"{k}: the one-call prefill differs from the separate calls"

    f = W.to_f64
    ref = oracle.layer_prefill(f(inp["mixed_qkv"]), f(inp["z"]), f(inp["a"]), f(inp["b"]), f(inp["conv_w"]),
                               f(inp["A_log"]), f(inp["dt_bias"]), f(inp["norm_w"]), s.H_k, s.H_v, s.d_k, s.d_v,
                               cu_seqlens=inp["cu_seqlens"].numpy(),
                               S0=None if inp["S0"] is None else f(inp["S0"]),
                               conv_state0=None if inp["conv_state0"] is None else f(inp["conv_state0"]),
                               ckpt_every=c["ckpt_every"])
    tol = TOL[dtype]
    e_pre = assert_close("out", host(one["out"]), ref["out"], tol)
    assert_close("final state", host(one["final_state"]), ref["S"], tol)
    assert np.array_equal(host(one["conv_state"]), ref["conv_state"]), "conv state"
    if ref["S_ckpt"] is not None and ref["S_ckpt"].shape[0]:
        assert_close("state checkpoints", host(one["state_ckpt"]), ref["S_ckpt"], tol)
        assert np.array_equal(host(one["conv_ckpt"]), ref["conv_ckpt"]), "conv checkpoints"
    for i, L in enumerate(lengths):
        if L == 0:
            # an empty sequence passes its states through unchanged
            S_in = inp["S0"][i] if inp["S0"] is not None else torch.zeros_like(one["final_state"][i].cpu())
            assert torch.equal(one["final_state"][i].cpu(), S_in)

    # fused decode steps from the prefill's states, every sequence at once
    dec = W.decode_inputs(s, dtype, N, DECODE_STEPS, seed=3000 + seed)
    dd = {k: v.cuda() for k, v in dec.items()}
    S, cs = one["final_state"].clone(), one["conv_state"].clone()
    outs = []
    for t in range(DECODE_STEPS):
        outs.append(gdn.gdn_decode_step(dd["qkv"][t], dd["z"][t], dd["a"][t], dd["b"][t], d["conv_w"],
                                        d["A_log"], d["dt_bias"], d["norm_w"], dims, S, cs))
    torch.cuda.synchronize()
    gdn.gdn_sync_status()
    # the output rows of a few steps against the oracle with y and o rounded
    # as the calls hand them on: one 128-value row carries those roundings on
    # its own (up to ~2e-2 rel-L2 for single rows), which a tensor of a few
    # rows does not average out; the states against the plain oracle
    rnd = rounded_to(dtype)
    S_r, cs_r, S_a, cs_a, refs = ref["S"], ref["conv_state"], ref["S"], ref["conv_state"], []
    for t in range(DECODE_STEPS):
        step = (f(dec["qkv"][t]), f(dec["z"][t]), f(dec["a"][t]), f(dec["b"][t]), f(inp["conv_w"]),
                f(inp["A_log"]), f(inp["dt_bias"]), f(inp["norm_w"]))
        _, S_r, cs_r, _ = oracle.layer_decode_step(*step, s.H_k, s.H_v, s.d_k, s.d_v, S_r, cs_r)
        o_a, S_a, cs_a = oracle_step_in_activation_dtype(*step, s, S_a, cs_a, rnd)
        refs.append(o_a)
    e_out = assert_close("decode out", host(torch.stack(outs)), np.stack(refs), tol)
    e_S = assert_close("decode state", host(S), S_r, tol)
    print(f"case {seed}: prefill out {e_pre:.2e}, decode out {e_out:.2e}, decode state {e_S:.2e}")
    assert np.array_equal(host(cs), cs_r), "decode conv state"
