"""GPU parity of the one-call entry points: gdn_layer_prefill (conv, chunked
rule, RMSNormGated; its scratch in one workspace) and gdn_chunk_prefill_norm
(the rule's output normalised in place in `out`).

Against the three separate calls on the same inputs: every output bit for bit
(the same kernels on the same values).  Against the f64 oracle: the dtype's
tolerance.  The cases reach both chain forms of the tensor-core path -- a head
split into two 64-column CTAs (few sequences) and one CTA per head (more
(sequence, head) pairs than SMs) -- ragged tails, empty and 1..3-token
sequences, checkpoints, the conv state updated in place, the Neumann-style
solve and the CUDA-core path.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_core_gb300 as gdn
import oracle
import workloads as W
from gpu_util import TOL, assert_close, host, oracle_heads_prefill

pytestmark = pytest.mark.gpu

SHAPE_27B = W.GDNShape(H_k=16, H_v=48, d_k=128, d_v=128)
SMALL_128 = W.GDNShape(H_k=2, H_v=6, d_k=128, d_v=128)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _dims(s):
    return gdn.GDNDims(s.H_k, s.H_v, s.d_k, s.d_v)


def _run(inp, shape, one_call, ckpt_every=0, solve="direct"):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    r = gdn.gdn_layer_prefill(d["mixed_qkv"], d["z"], d["a"], d["b"], d["conv_w"], d["A_log"], d["dt_bias"],
                              d["norm_w"], _dims(shape), cu_seqlens=d["cu_seqlens"], initial_state=d["S0"],
                              conv_state=d["conv_state0"], ckpt_every=ckpt_every,
                              return_intermediates=not one_call, solve=solve)
    torch.cuda.synchronize()
    gdn.gdn_sync_status()
    return r


def _compare_with_separate(fz, sp):
    for k in ("out", "final_state", "conv_state", "state_ckpt", "conv_ckpt"):
        if sp[k] is None:
            assert fz[k] is None, k
        else:
            assert torch.equal(fz[k], sp[k]), f"{k} differs from the separate calls"
    assert torch.isfinite(fz["out"].float()).all()


def _oracle(inp, shape, ckpt_every=0):
    f = W.to_f64
    return oracle.layer_prefill(f(inp["mixed_qkv"]), f(inp["z"]), f(inp["a"]), f(inp["b"]), f(inp["conv_w"]),
                                f(inp["A_log"]), f(inp["dt_bias"]), f(inp["norm_w"]), shape.H_k, shape.H_v,
                                shape.d_k, shape.d_v, cu_seqlens=inp["cu_seqlens"].numpy(),
                                S0=None if inp["S0"] is None else f(inp["S0"]),
                                conv_state0=None if inp["conv_state0"] is None else f(inp["conv_state0"]),
                                ckpt_every=ckpt_every)


def test_one_sequence_27b_heads_ragged_tail():
    # 48 value heads x 2 column slices = 96 chain CTAs; 1000 tokens: 15 full
    # chunks and a 40-token tail stored row by row
    inp = W.layer_inputs(SHAPE_27B, torch.bfloat16, [1000], seed=31, init_state=True)
    fz = _run(inp, SHAPE_27B, one_call=True, ckpt_every=256)
    sp = _run(inp, SHAPE_27B, one_call=False, ckpt_every=256)
    _compare_with_separate(fz, sp)
    ref = _oracle(inp, SHAPE_27B, ckpt_every=256)
    tol = TOL[torch.bfloat16]
    assert_close("out", host(fz["out"]), ref["out"], tol)
    assert_close("out per head", host(fz["out"]).reshape(-1, SHAPE_27B.H_v, SHAPE_27B.d_v),
                 ref["out"].reshape(-1, SHAPE_27B.H_v, SHAPE_27B.d_v), tol, per_head_axis=1)
    assert_close("S", host(fz["final_state"]), ref["S"], tol, per_head_axis=1)


def test_many_sequences_one_cta_per_head():
    # 4 x 48 x 2 > 152 SMs: one chain CTA per (sequence, head); sequences
    # shorter than a chunk, exactly one chunk, and with a ragged tail
    lengths = [70, 1, 300, 64]
    inp = W.layer_inputs(SHAPE_27B, torch.bfloat16, lengths, seed=32, init_state=True)
    fz = _run(inp, SHAPE_27B, one_call=True, ckpt_every=64)
    sp = _run(inp, SHAPE_27B, one_call=False, ckpt_every=64)
    _compare_with_separate(fz, sp)
    ref = _oracle(inp, SHAPE_27B, ckpt_every=64)
    tol = TOL[torch.bfloat16]
    assert_close("out", host(fz["out"]), ref["out"], tol)
    assert_close("S", host(fz["final_state"]), ref["S"], tol, per_head_axis=1)
    assert_close("S ckpt", host(fz["state_ckpt"]), ref["S_ckpt"], tol)


@pytest.mark.parametrize("lengths", [[1, 63, 64, 65, 0, 200, 3], [130, 70]], ids=["edge", "two"])
def test_small_heads_varlen(lengths):
    # few (sequence, head) pairs: every head split into two chain CTAs; empty
    # sequences and sequences of 1..3 tokens
    inp = W.layer_inputs(SMALL_128, torch.bfloat16, lengths, seed=33, init_state=True)
    fz = _run(inp, SMALL_128, one_call=True)
    sp = _run(inp, SMALL_128, one_call=False)
    _compare_with_separate(fz, sp)
    ref = _oracle(inp, SMALL_128)
    assert_close("out", host(fz["out"]), ref["out"], TOL[torch.bfloat16])


def test_many_short_sequences_conv_inside_the_chunk_kernels():
    # 40 packed sequences of 0-150 tokens (many shorter than the conv's 3-token
    # window, some empty, several with a checkpoint): the intra kernel takes
    # each sequence's conv state at its first chunk and writes the conv state
    # and checkpoints at its last; everything equals the separate calls
    g = np.random.default_rng(38)
    lengths = [int(x) for x in g.choice([0, 1, 2, 3, 4, 63, 64, 65, 127, 128, 150], size=40)]
    inp = W.layer_inputs(SMALL_128, torch.bfloat16, lengths, seed=38, init_state=True)
    fz = _run(inp, SMALL_128, one_call=True, ckpt_every=64)
    sp = _run(inp, SMALL_128, one_call=False, ckpt_every=64)
    _compare_with_separate(fz, sp)
    ref = _oracle(inp, SMALL_128, ckpt_every=64)
    assert_close("out", host(fz["out"]), ref["out"], TOL[torch.bfloat16])
    assert_close("S", host(fz["final_state"]), ref["S"], TOL[torch.bfloat16], per_head_axis=1)
    assert np.array_equal(host(fz["conv_state"]), ref["conv_state"])


def test_more_sequences_than_the_longest_first_order_covers():
    # 1500 packed sequences (0-69 tokens): above 1024 the chunk-offsets kernel
    # leaves the chain's CTAs in sequence order instead of longest first; one
    # 128-column chain CTA per (sequence, head); every result against the
    # separate calls bit for bit and against the oracle
    g = np.random.default_rng(39)
    lengths = [int(x) for x in g.integers(0, 70, size=1500)]
    inp = W.layer_inputs(SMALL_128, torch.bfloat16, lengths, seed=39, init_state=True)
    fz = _run(inp, SMALL_128, one_call=True, ckpt_every=64)
    sp = _run(inp, SMALL_128, one_call=False, ckpt_every=64)
    _compare_with_separate(fz, sp)
    ref = _oracle(inp, SMALL_128, ckpt_every=64)
    assert_close("out", host(fz["out"]), ref["out"], TOL[torch.bfloat16])
    assert_close("S", host(fz["final_state"]), ref["S"], TOL[torch.bfloat16], per_head_axis=1)
    assert np.array_equal(host(fz["conv_state"]), ref["conv_state"])


@pytest.mark.parametrize("H_k,H_v,lengths", [(16, 128, [300, 212]), (64, 64, [200]), (2, 32, [130, 1, 66])],
                         ids=["r8-128heads", "r1-64heads", "r16"])
def test_head_counts_beyond_the_workloads(H_k, H_v, lengths):
    # 128 value heads (r = 8: 256 chain CTAs as 128-column CTAs), 64 key heads
    # at r = 1, and r = 16 (beyond what the decode kernels take): the layer call
    # against the separate calls bit for bit and against the oracle
    shape = W.GDNShape(H_k=H_k, H_v=H_v, d_k=128, d_v=128)
    inp = W.layer_inputs(shape, torch.bfloat16, lengths, seed=40 + H_k, init_state=True)
    fz = _run(inp, shape, one_call=True, ckpt_every=128)
    sp = _run(inp, shape, one_call=False, ckpt_every=128)
    _compare_with_separate(fz, sp)
    ref = _oracle(inp, shape, ckpt_every=128)
    tol = TOL[torch.bfloat16]
    assert_close("out", host(fz["out"]), ref["out"], tol)
    assert_close("S", host(fz["final_state"]), ref["S"], tol, per_head_axis=1)
    if ref["S_ckpt"] is not None and ref["S_ckpt"].shape[0]:
        assert_close("S ckpt", host(fz["state_ckpt"]), ref["S_ckpt"], tol)
    assert np.array_equal(host(fz["conv_state"]), ref["conv_state"])


def test_conv_state_in_place_equals_out_of_place():
    # bf16 with d = 128 runs the conv inside the chunk kernels, which then also
    # write the conv state and checkpoints -- unless the state is updated in
    # place, where a pass after them does; empty and 1..3-token sequences take
    # their state from conv_state0
    lengths = [1, 63, 0, 200, 3, 130]
    inp = W.layer_inputs(SMALL_128, torch.bfloat16, lengths, seed=37, init_state=True)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    args = (d["mixed_qkv"], d["z"], d["a"], d["b"], d["conv_w"], d["A_log"], d["dt_bias"], d["norm_w"],
            _dims(SMALL_128))
    kw = dict(cu_seqlens=d["cu_seqlens"], initial_state=d["S0"], ckpt_every=64)
    cs = d["conv_state0"].clone()
    ref = gdn.gdn_layer_prefill(*args, conv_state=d["conv_state0"], **kw)
    got = gdn.gdn_layer_prefill(*args, conv_state=cs, conv_state_out=cs, **kw)
    torch.cuda.synchronize()
    gdn.gdn_sync_status()
    assert got["conv_state"].data_ptr() == cs.data_ptr()
    for k in ("out", "final_state", "conv_state", "state_ckpt", "conv_ckpt"):
        assert torch.equal(got[k], ref[k]), k
    sp = _run(inp, SMALL_128, one_call=False, ckpt_every=64)
    _compare_with_separate(ref, sp)


def test_neumann_solve_in_the_layer_call():
    inp = W.layer_inputs(SMALL_128, torch.bfloat16, [257], seed=34, init_state=False)
    fz = _run(inp, SMALL_128, one_call=True, solve="neumann")
    sp = _run(inp, SMALL_128, one_call=False, solve="neumann")
    _compare_with_separate(fz, sp)


@pytest.mark.parametrize("shape", [W.TINY, SMALL_128], ids=["d16", "d128"])
def test_cuda_core_path_f32(shape):
    # f32: conv, the CUDA-core rule and the norm kernel in turn
    inp = W.layer_inputs(shape, torch.float32, [65, 3, 128], seed=35, init_state=True)
    fz = _run(inp, shape, one_call=True)
    sp = _run(inp, shape, one_call=False)
    _compare_with_separate(fz, sp)
    ref = _oracle(inp, shape)
    assert_close("out", host(fz["out"]), ref["out"], TOL[torch.float32])


def test_empty_call_passes_the_states_through():
    inp = W.layer_inputs(SMALL_128, torch.bfloat16, [0, 0], seed=36, init_state=True)
    fz = _run(inp, SMALL_128, one_call=True)
    assert fz["out"].numel() == 0
    assert torch.equal(fz["final_state"].cpu(), inp["S0"])
    assert torch.equal(fz["conv_state"].cpu(), inp["conv_state0"])


def test_chunk_prefill_norm_one_sequence_without_offsets():
    # the form the layer call uses for one sequence: no cu_seqlens, no offsets kernel
    inp = W.layer_inputs(SHAPE_27B, torch.bfloat16, [1100], seed=37, init_state=True)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    dims = _dims(SHAPE_27B)
    y = gdn.gdn_conv1d_fwd(d["mixed_qkv"], d["conv_w"], dims, None, d["conv_state0"], None)
    S1 = torch.empty_like(d["S0"])
    S2 = torch.empty_like(d["S0"])
    out = gdn.gdn_chunk_prefill_norm(y, d["z"], d["norm_w"], dims, d["a"], d["b"], d["A_log"], d["dt_bias"],
                                     initial_state=d["S0"], final_state=S1)
    o = gdn.gdn_chunk_prefill(y, dims, d["a"], d["b"], d["A_log"], d["dt_bias"], initial_state=d["S0"],
                              final_state=S2)
    ref = gdn.gdn_rmsnorm_gated(o, d["z"], d["norm_w"], dims)
    torch.cuda.synchronize()
    gdn.gdn_sync_status()
    assert torch.equal(S1, S2)
    _compare_with_separate({"out": out, "final_state": S1, "conv_state": None, "state_ckpt": None,
                            "conv_ckpt": None},
                           {"out": ref, "final_state": S2, "conv_state": None, "state_ckpt": None,
                            "conv_ckpt": None})


@pytest.mark.parametrize("dtype,shape", [(torch.bfloat16, SMALL_128), (torch.float32, SMALL_128),
                                         (torch.float32, W.TINY)], ids=["bf16-tensor-core", "f32-d128", "f32-d16"])
def test_packed_sequences_equal_separate_calls(dtype, shape):
    """A packed (cu_seqlens) call equals one call per sequence, bit for bit:
    rows past a sequence's last token (the next sequence's tokens when packed,
    zeros when alone) enter only through factors that are exactly zero."""
    lengths = [70, 1, 200, 64]
    every = 64
    inp = W.layer_inputs(shape, dtype, lengths, seed=38, init_state=True)
    packed = _run(inp, shape, one_call=True, ckpt_every=every)
    cu = inp["cu_seqlens"].tolist()
    row = 0
    for i, L in enumerate(lengths):
        one = {k: inp[k][cu[i]:cu[i + 1]] for k in ("mixed_qkv", "z", "a", "b")}
        for k in ("conv_w", "A_log", "dt_bias", "norm_w"):
            one[k] = inp[k]
        one["cu_seqlens"] = W.cu_seqlens_of([L])
        one["S0"] = inp["S0"][i:i + 1]
        one["conv_state0"] = inp["conv_state0"][i:i + 1]
        r = _run(one, shape, one_call=True, ckpt_every=every)
        assert torch.equal(r["out"], packed["out"][cu[i]:cu[i + 1]]), f"out of sequence {i}"
        assert torch.equal(r["final_state"][0], packed["final_state"][i]), f"state of sequence {i}"
        assert torch.equal(r["conv_state"][0], packed["conv_state"][i]), f"conv state of sequence {i}"
        n_ck = L // every
        if n_ck:
            assert torch.equal(r["state_ckpt"], packed["state_ckpt"][row:row + n_ck]), f"ckpts of sequence {i}"
            assert torch.equal(r["conv_ckpt"], packed["conv_ckpt"][row:row + n_ck]), f"conv ckpts of sequence {i}"
        row += n_ck


@pytest.mark.parametrize("world", [2, 4])
def test_head_shards_equal_the_full_call(world):
    """Head sharding (tensor parallel over key heads): each shard's call on its
    slices equals the full call's slice bit for bit; no exchange inside the
    core.  The shards run one after another on this GPU."""
    s = SHAPE_27B
    inp = W.layer_inputs(s, torch.bfloat16, [600, 400], seed=39, init_state=True)
    full = _run(inp, s, one_call=True, ckpt_every=256)
    # the full call itself against the oracle, on one value head of each shard
    tol = TOL[torch.bfloat16]
    heads = [gdn.head_shard(_dims(s), r, world).h0 for r in range(world)]
    out = full["out"].view(-1, s.H_v, s.d_v)
    for h, ref in oracle_heads_prefill(inp, s, heads, ckpt_every=256).items():
        assert_close(f"out head {h}", host(out[:, h]), ref["out"], tol)
        assert_close(f"S head {h}", host(full["final_state"][:, h]), ref["S"][:, 0], tol)
        assert_close(f"ckpts head {h}", host(full["state_ckpt"][:, h]), ref["S_ckpt"][:, 0], tol)
    for r in range(world):
        sh = gdn.head_shard(_dims(s), r, world)
        zc = slice(sh.h0 * s.d_v, sh.h1 * s.d_v)
        part_in = {"mixed_qkv": inp["mixed_qkv"][:, sh.channels].contiguous(), "z": inp["z"][:, zc].contiguous(),
                   "a": inp["a"][:, sh.h0:sh.h1].contiguous(), "b": inp["b"][:, sh.h0:sh.h1].contiguous(),
                   "conv_w": inp["conv_w"][sh.channels].contiguous(), "A_log": inp["A_log"][sh.h0:sh.h1].contiguous(),
                   "dt_bias": inp["dt_bias"][sh.h0:sh.h1].contiguous(), "norm_w": inp["norm_w"],
                   "cu_seqlens": inp["cu_seqlens"], "S0": inp["S0"][:, sh.h0:sh.h1].contiguous(),
                   "conv_state0": inp["conv_state0"][:, sh.channels].contiguous()}
        shape = W.GDNShape(sh.dims.H_k, sh.dims.H_v, s.d_k, s.d_v)
        part = _run(part_in, shape, one_call=True, ckpt_every=256)
        ch = sh.channels.cuda()
        assert torch.equal(part["out"], full["out"][:, zc]), f"out of shard {r}"
        assert torch.equal(part["final_state"], full["final_state"][:, sh.h0:sh.h1]), f"state of shard {r}"
        assert torch.equal(part["state_ckpt"], full["state_ckpt"][:, sh.h0:sh.h1]), f"ckpts of shard {r}"
        assert torch.equal(part["conv_state"], full["conv_state"][:, ch]), f"conv state of shard {r}"
        assert torch.equal(part["conv_ckpt"], full["conv_ckpt"][:, ch]), f"conv ckpts of shard {r}"


@pytest.mark.parametrize("H_k,H_v", [(4, 4), (2, 4), (1, 8)], ids=["r1", "r2", "r8"])
def test_head_ratios_prefill_then_fused_decode(H_k, H_v):
    """Value heads per key head r = 1, 2 and 8 (the fused decode CTA's
    largest): the layer prefill on the tensor-core path against the oracle,
    then two fused decode steps from the prefill's own states against the
    oracle started from those same states (so the decode kernel is measured
    alone, not the bf16 prefill's state error carried into it)."""
    s = W.GDNShape(H_k=H_k, H_v=H_v, d_k=128, d_v=128)
    lengths = [130, 70]
    inp = W.layer_inputs(s, torch.bfloat16, lengths, seed=43, init_state=True)
    r = _run(inp, s, one_call=True)
    ref = _oracle(inp, s)
    tol = TOL[torch.bfloat16]
    assert_close("out", host(r["out"]), ref["out"], tol)
    assert_close("S", host(r["final_state"]), ref["S"], tol, per_head_axis=1)
    f = W.to_f64
    dec = W.decode_inputs(s, torch.bfloat16, len(lengths), 2, seed=44)
    S, cs = r["final_state"].clone(), r["conv_state"].clone()
    S_ref, cs_ref = host(r["final_state"]), host(r["conv_state"])
    dev = {k: v.cuda() for k, v in dec.items()}
    p = {k: inp[k].cuda() for k in ("conv_w", "A_log", "dt_bias", "norm_w")}
    for t in range(2):
        out = gdn.gdn_decode_step(dev["qkv"][t], dev["z"][t], dev["a"][t], dev["b"][t], p["conv_w"], p["A_log"],
                                  p["dt_bias"], p["norm_w"], _dims(s), S, cs)
        torch.cuda.synchronize()
        out_ref, S_ref, cs_ref, _ = oracle.layer_decode_step(
            f(dec["qkv"][t]), f(dec["z"][t]), f(dec["a"][t]), f(dec["b"][t]), f(inp["conv_w"]), f(inp["A_log"]),
            f(inp["dt_bias"]), f(inp["norm_w"]), s.H_k, s.H_v, s.d_k, s.d_v, S_ref, cs_ref)
        assert_close(f"decode out, step {t}", host(out), out_ref, tol)
    assert_close("decode S", host(S), S_ref, tol, per_head_axis=1)
    assert np.array_equal(host(cs), cs_ref)
