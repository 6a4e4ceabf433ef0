"""Head sharding of the layer core (CPU): the partition `head_shard` computes,
and the property it rests on -- heads, their conv channels and their states
are independent through the whole core -- checked on the oracle, in one
process and across two gloo ranks that each run their shard and gather the
outputs.  The GPU counterpart is in test_gpu_layer_call.py."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import gated_deltanet_linear_core_gb300 as gdn
import oracle
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SHAPE = W.GDNShape(H_k=4, H_v=8, d_k=16, d_v=16)


def _dims(s):
    return gdn.GDNDims(s.H_k, s.H_v, s.d_k, s.d_v)


@pytest.mark.parametrize("world", [1, 2, 4, 8, 16])
def test_shards_partition_heads_and_channels(world):
    dims = gdn.GDNDims(16, 48, 128, 128)
    seen = torch.zeros(dims.conv_dim, dtype=torch.int64)
    heads = []
    for r in range(world):
        sh = gdn.head_shard(dims, r, world)
        assert sh.dims.H_k * world == dims.H_k and sh.dims.H_v * world == dims.H_v
        assert sh.dims.conv_dim == sh.channels.numel()
        seen[sh.channels] += 1
        heads += list(range(sh.h0, sh.h1))
        assert sh.h0 == sh.kh0 * 3 and sh.h1 == sh.kh1 * 3
    assert bool((seen == 1).all())
    assert heads == list(range(dims.H_v))


def test_invalid_shardings_are_refused():
    dims = gdn.GDNDims(16, 48, 128, 128)
    for rank, world in [(0, 3), (2, 2), (-1, 2), (0, 0), (0, 32)]:
        with pytest.raises(ValueError):
            gdn.head_shard(dims, rank, world)


def _shard_inputs(inp, sh, s):
    """The slices of a layer's inputs one shard reads."""
    d = sh.dims
    zc = slice(sh.h0 * s.d_v, sh.h1 * s.d_v)
    out = {"mixed_qkv": inp["mixed_qkv"][:, sh.channels], "z": inp["z"][:, zc],
           "a": inp["a"][:, sh.h0:sh.h1], "b": inp["b"][:, sh.h0:sh.h1],
           "conv_w": inp["conv_w"][sh.channels], "A_log": inp["A_log"][sh.h0:sh.h1],
           "dt_bias": inp["dt_bias"][sh.h0:sh.h1], "norm_w": inp["norm_w"], "cu_seqlens": inp["cu_seqlens"],
           "S0": inp["S0"][:, sh.h0:sh.h1], "conv_state0": inp["conv_state0"][:, sh.channels]}
    assert d.conv_dim == out["mixed_qkv"].shape[1]
    return out


def _oracle(inp, s):
    f = W.to_f64
    return oracle.layer_prefill(f(inp["mixed_qkv"]), f(inp["z"]), f(inp["a"]), f(inp["b"]), f(inp["conv_w"]),
                                f(inp["A_log"]), f(inp["dt_bias"]), f(inp["norm_w"]), s.H_k, s.H_v, s.d_k, s.d_v,
                                cu_seqlens=inp["cu_seqlens"].numpy(), S0=f(inp["S0"]),
                                conv_state0=f(inp["conv_state0"]), ckpt_every=64)


def _check_shard(full, part, sh, s):
    zc = slice(sh.h0 * s.d_v, sh.h1 * s.d_v)
    assert np.array_equal(part["out"], full["out"][:, zc])
    assert np.array_equal(part["S"], full["S"][:, sh.h0:sh.h1])
    assert np.array_equal(part["S_ckpt"], full["S_ckpt"][:, sh.h0:sh.h1])
    assert np.array_equal(part["conv_state"], full["conv_state"][:, sh.channels.numpy()])
    assert np.array_equal(part["conv_ckpt"], full["conv_ckpt"][:, sh.channels.numpy()])


@pytest.mark.parametrize("world", [2, 4])
def test_oracle_shards_equal_the_full_layer(world):
    inp = W.layer_inputs(SHAPE, torch.float32, [70, 130], seed=41, init_state=True)
    full = _oracle(inp, SHAPE)
    for r in range(world):
        sh = gdn.head_shard(_dims(SHAPE), r, world)
        part = _oracle(_shard_inputs(inp, sh, SHAPE), W.GDNShape(sh.dims.H_k, sh.dims.H_v, SHAPE.d_k, SHAPE.d_v))
        _check_shard(full, part, sh, SHAPE)


def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = W.layer_inputs(SHAPE, torch.float32, [70, 130], seed=42, init_state=True)
    sh = gdn.head_shard(_dims(SHAPE), rank, world)
    part = _oracle(_shard_inputs(inp, sh, SHAPE), W.GDNShape(sh.dims.H_k, sh.dims.H_v, SHAPE.d_k, SHAPE.d_v))
    # the only exchange: gathering each rank's output columns, as the layer's
    # out_proj all-reduce would combine them
    mine = torch.from_numpy(np.ascontiguousarray(part["out"]))
    got = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(got, mine)
    if rank == 0:
        full = _oracle(inp, SHAPE)
        assert np.array_equal(torch.cat(got, dim=1).numpy(), full["out"])
        open(os.path.join(out_dir, "ok"), "w").write("ok")
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_each_run_their_shard(tmp_path):
    mp.start_processes(_rank, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    assert (tmp_path / "ok").exists()
