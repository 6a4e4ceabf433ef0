"""gdn_chunk_prefill_noalloc: the chunked prefill for callers that cannot
allocate device memory (its scratch is a fixed array inside the library, and
the caller passes every output).  Checked against gdn_chunk_prefill -- the
workspace entry point -- on two calls in a row, the second after the first has
left its own contents in the shared array.  This file is collected last so a
run that stops at the first failure has run every other test first."""
import pytest
import torch

import gated_deltanet_linear_core_gb300 as gdn
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
        tol = TOL[torch.bfloat16]
        assert_close("o", host(o), host(o_ref), tol)
        assert_close("final state", host(S), host(S_ref), tol)
        assert_close("checkpoints", host(ck), host(ck_ref), tol)


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
