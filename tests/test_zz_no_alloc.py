"""gdn_chunk_prefill_noalloc: the chunked prefill for callers that cannot
allocate device memory (its scratch is a fixed array inside the library, and
the caller passes every output).  Its arithmetic is that of gdn_chunk_prefill
-- the workspace entry point -- with the state carried between its shorter
segments in f32, so on two calls in a row (the second after the first has left
its own contents in the shared array) outputs, final states and checkpoints
must equal the workspace entry point's bit for bit, and sampled value heads
must match the oracle within the bf16 tolerance.  This file is collected last
so a run that stops at the first failure has run every other test first."""
import pytest
import torch

import gated_deltanet_linear_core_gb300 as gdn
import oracle
import workloads as W
from gpu_util import TOL, assert_close, host

pytestmark = pytest.mark.gpu

# (shape, sequence lengths, seed, checkpoint interval): the second case needs
# several segments of the fixed array (48 value heads) and carries its state
# between them
CASES = [
    (W.GDNShape(2, 6, 128, 128), [1, 63, 64, 200, 0, 130], 71, 64),
    (W.QWEN36_27B, [1000, 1500, 37], 72, 512),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def test_noalloc_prefill_matches_the_workspace_entry_point_twice():
    for shape, lengths, seed, every in CASES:
        inp = W.layer_inputs(shape, torch.bfloat16, lengths, seed=seed, init_state=True)
        d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
        dims = gdn.GDNDims(shape.H_k, shape.H_v, shape.d_k, shape.d_v)
        N, T = len(lengths), sum(lengths)
        rows = gdn.gdn_ckpt_count(inp["cu_seqlens"], every)
        sdims = (shape.H_v, shape.d_k, shape.d_v)

        S_ref = torch.empty((N,) + sdims, device="cuda")
        ck_ref = torch.empty((rows,) + sdims, device="cuda")
        o_ref = gdn.gdn_chunk_prefill(d["mixed_qkv"], dims, d["a"], d["b"], d["A_log"],
                                      d["dt_bias"], cu_seqlens=d["cu_seqlens"],
                                      initial_state=d["S0"], final_state=S_ref, ckpt_every=every,
                                      state_ckpt_out=ck_ref)
        # every output preallocated by the caller
        o = torch.full((T, shape.H_v, shape.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        S = torch.full((N,) + sdims, float("nan"), device="cuda")
        ck = torch.full((rows,) + sdims, float("nan"), device="cuda")
        gdn.gdn_chunk_prefill_noalloc(d["mixed_qkv"], dims, o, S, d["a"], d["b"], d["A_log"],
                                      d["dt_bias"], cu_seqlens=d["cu_seqlens"],
                                      initial_state=d["S0"], ckpt_every=every,
                                      state_ckpt_out=ck)
        gdn.gdn_sync_status()
        assert torch.equal(o, o_ref), "o differs from the workspace entry point"
        assert torch.equal(S, S_ref), "final state differs from the workspace entry point"
        assert torch.equal(ck, ck_ref), "checkpoints differ from the workspace entry point"
        # sampled value heads against the oracle (heads are independent)
        tol = TOL[torch.bfloat16]
        f = W.to_f64
        heads = [0, shape.H_v - 1]
        q, k, v = oracle.split_qkv(f(inp["mixed_qkv"]), shape.H_k, shape.H_v, shape.d_k, shape.d_v)
        g, beta = oracle.gates(f(inp["a"]), f(inp["b"]), f(inp["A_log"]), f(inp["dt_bias"]))
        r = shape.H_v // shape.H_k
        for h in heads:
            o_h, S_h, ck_h = oracle.delta_rule(q[:, h // r:h // r + 1], k[:, h // r:h // r + 1],
                                               v[:, h:h + 1], g[:, h:h + 1], beta[:, h:h + 1],
                                               inp["cu_seqlens"].numpy(), f(inp["S0"])[:, h:h + 1],
                                               None, True, every)
            assert_close(f"o head {h}", host(o[:, h]), o_h[:, 0], tol)
            assert_close(f"final state head {h}", host(S[:, h]), S_h[:, 0], tol)
            assert_close(f"checkpoints head {h}", host(ck[:, h]), ck_h[:, 0], tol)


def test_noalloc_rejects_calls_beyond_its_limits():
    shape = W.GDNShape(2, 4, 128, 128)
    dims = gdn.GDNDims(2, 4, 128, 128)
    qkv = torch.zeros((64, shape.conv_dim), dtype=torch.bfloat16, device="cuda")
    gates = torch.zeros((64, 4), dtype=torch.bfloat16, device="cuda")
    par = torch.zeros(4, device="cuda")
    o = torch.empty((64, 4, 128), dtype=torch.bfloat16, device="cuda")
    S = torch.empty((1, 4, 128, 128), device="cuda")
    with pytest.raises(gdn.GDNError, match="INVALID_ARG"):  # final_state is required
        gdn.gdn_chunk_prefill_noalloc(qkv, dims, o, None, gates, gates, par, par)
    with pytest.raises(gdn.GDNError, match="UNSUPPORTED"):  # tensor-core shapes only
        gdn.gdn_chunk_prefill_noalloc(qkv.float(), dims, o.float(), S, gates.float(),
                                      gates.float(), par, par)
