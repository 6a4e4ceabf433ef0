"""Benchmark of the GDN layer core on GB300.

Prints ONE JSON line (rank 0).  A call is one pass of the layer core's
prefill path -- one gdn_layer_prefill call: conv1d + SiLU, the chunked rule,
RMSNormGated -- over the Qwen3.6-27B prefill workload (B=1, T=4096, 16 QK / 48 V heads,
d=128, bf16 activations, f32 state); a timed step is --calls such calls, each
on its own copy of the inputs (a ring of 16 copies, so every call starts with
its inputs out of L2).  `value` is prefill tokens/s with inputs resident in
HBM; the same line carries the other prefill workloads (Coder-Next varlen with
resumed states; the 262144-token sequence with checkpoints every 4096 tokens
and its 128-step decode tail) under "prefill_workloads", the decode path (the
27B decode workload: 64 sequences, one token each per step) under "decode",
each with the roofline of its dominant kernel, one rank's call under head
sharding over 2, 4 and 8 ranks ("head_shards"), the end-to-end rate through
host buffers ("e2e"), the oracle's CPU rate on all cores and on one
("cpu_baseline") and the SM clocks seen while timing.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same per-GPU workload (replicas:
the layer core has no exchange step), so scaling is weak and `value` is the
sum over ranks of tokens divided by the slowest rank's time.
`--impl reference` times the CPU oracle on a bounded sample of the same
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "GDN prefill tokens/s and decode tokens/s per layer; % tensor-core / HBM roofline"
PREFILL = "qwen36_27b_prefill"
DECODE = "qwen36_27b_decode"
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2
RING = 16  # input copies the headline prefill step cycles through
FLOP_PER_TOKEN_HEAD = 5 * 64 * 128 + 6 * 128 * 128  # 139,264 (chunked delta rule, C=64, d=128)


def chunk_bytes_per_token(s: W.GDNShape) -> int:
    """Algorithmic bytes of the chunk stage per token (bf16): post-conv q, k, v
    and the gate inputs a, b read, o written."""
    return 2 * (s.conv_dim + 2 * s.H_v + s.H_v * s.d_v)


def decode_kernel_bytes_per_seq(s: W.GDNShape) -> int:
    """Algorithmic bytes of the recurrent-decode kernel per sequence-step: read
    and write each f32 state once, read q/k/v (bf16) and a, b, write o."""
    state = s.H_v * 2 * s.d_k * s.d_v * 4
    return state + (s.conv_dim + 2 * s.H_v + s.H_v * s.d_v) * 2


def decode_step_bytes_per_seq(s: W.GDNShape) -> int:
    """Algorithmic bytes of one fused decode step per sequence: the f32 state
    and the bf16 conv state read and written once, the token's qkv, z, a, b
    read and its output written (the conv weight, shared by all sequences, is
    left out)."""
    state = s.H_v * 2 * s.d_k * s.d_v * 4
    conv_state = 2 * s.conv_dim * 3 * 2
    return state + conv_state + (s.conv_dim + s.z_dim + 2 * s.H_v + s.H_v * s.d_v) * 2


def verify_bytes_per_seq(s: W.GDNShape, K: int) -> int:
    """Algorithmic bytes of one K-token verification per sequence: the f32
    state and the bf16 conv state read once and written after every draft
    token, the tokens' qkv, z, a, b read and their outputs written."""
    state = s.H_v * s.d_k * s.d_v * 4
    conv_state = s.conv_dim * 3 * 2
    return (1 + K) * (state + conv_state) + K * (s.conv_dim + s.z_dim + 2 * s.H_v + s.H_v * s.d_v) * 2


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def traffic_record(kernel: str):
    """DRAM bytes per launch from the committed ncu summary of `kernel`, valid
    only while the kernel's source is unchanged (sha256 recorded with it)."""
    path = os.path.join(ROOT, "profiles", f"ncu_traffic_{kernel}.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            m = re.match(r"^(\w+)\s*=\s*(\S+)", line.strip())
            if m:
                kv[m.group(1)] = m.group(2)
    src = os.path.join(ROOT, "gated_deltanet_linear_core_gb300", "csrc", kv.get("source", ""))
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != kv.get("source_sha256"):
            return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled every 200 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.rows = []
        self.proc = None
        self.marks = []
        args = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                "-lms", "200"]
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            if uuid and not uuid.startswith("GPU-"):
                uuid = "GPU-" + uuid
            args += ["-i", uuid]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(args, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append((time.time(), parts))

    def mark(self, on: bool):
        self.marks.append((time.time(), on))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        spans, start = [], None
        for t, on in self.marks:
            if on:
                start = t
            elif start is not None:
                spans.append((start - 0.25, t + 0.25))
                start = None
        rows = [p for t, p in self.rows if any(a <= t <= b for a, b in spans)] or \
            [p for _, p in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist, dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return None, 0, 1, 0


def max_over_ranks(dist, x: float, dev) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, dev):
    if dist is not None:
        dist.barrier(device_ids=[dev.index] if dev.type == "cuda" else None)


# --------------------------------------------------------------------------- other prefill workloads
def prefill_workload(gdn, name, args, dev, stream, flush, clocks, pk, steps, warmup):
    """Time gdn_layer_prefill on the named workload (device-resident inputs, its
    own cu_seqlens, initial states and checkpoint cadence), calls back to back
    (the inputs are larger than L2); then the chunk stage alone (gdn_chunk_prefill on the conv output)
    for its tensor-peak fraction; for a workload with a decode tail, the fused
    decode steps that follow from the prefill's final states.  Returns (dict,
    launches)."""
    w = W.WORKLOADS[name]
    s = w.shape
    dims = gdn.GDNDims(s.H_k, s.H_v, s.d_k, s.d_v)
    t_gen = time.perf_counter()
    inp = W.workload_inputs(name)
    t_gen = time.perf_counter() - t_gen
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    T = int(inp["mixed_qkv"].shape[0])
    n = len(w.lengths)
    cu = d["cu_seqlens"] if n > 1 else None
    host_cu = inp["cu_seqlens"]
    rows = gdn.gdn_ckpt_count(host_cu, w.ckpt_every) if w.ckpt_every else 0
    out = torch.empty((T, s.H_v * s.d_v), dtype=w.dtype, device=dev)
    Sf = torch.empty((n, s.H_v, s.d_k, s.d_v), dtype=torch.float32, device=dev)
    csf = torch.empty((n, s.conv_dim, 3), dtype=w.dtype, device=dev)
    Sck = torch.empty((rows, s.H_v, s.d_k, s.d_v), dtype=torch.float32, device=dev) if rows else None
    cck = torch.empty((rows, s.conv_dim, 3), dtype=w.dtype, device=dev) if rows else None
    ws = torch.empty(gdn.gdn_layer_prefill_workspace_size(n, T, dims, w.dtype), dtype=torch.uint8, device=dev)

    def call():
        gdn.gdn_layer_prefill(d["mixed_qkv"], d["z"], d["a"], d["b"], d["conv_w"], d["A_log"], d["dt_bias"],
                              d["norm_w"], dims, cu_seqlens=cu, initial_state=d["S0"],
                              conv_state=d["conv_state0"], ckpt_every=w.ckpt_every, out=out, final_state=Sf,
                              conv_state_out=csf, workspace=ws, state_ckpt_out=Sck, conv_ckpt_out=cck)

    def timed(fn, k_steps, gap=False):
        # gap: an L2 flush before each timed call, which also keeps the host's
        # launches ahead of a short call (back to back, a one-sequence decode
        # step would time the host's launch path)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k_steps)]
        torch.cuda.synchronize(dev)
        clocks.mark(True)
        for k in range(k_steps):
            if gap:
                flush.zero_()
            ev[k][0].record(stream)
            fn()
            ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark(False)
        return [a_.elapsed_time(b_) for a_, b_ in ev]

    for _ in range(warmup):
        call()
    ms = timed(call, steps)
    launches = steps * gdn.gdn_layer_prefill_launches(n, T, dims, w.dtype, cu_seqlens=cu is not None)
    # the chunk stage alone, on the conv output of the same inputs
    y = torch.empty_like(d["mixed_qkv"])
    gdn.gdn_conv1d_fwd(d["mixed_qkv"], d["conv_w"], dims, cu, d["conv_state0"], torch.empty_like(csf), y=y)
    o = torch.empty((T, s.H_v, s.d_v), dtype=w.dtype, device=dev)
    cws = torch.empty(gdn.gdn_chunk_prefill_workspace_size(n, T, dims, w.dtype), dtype=torch.uint8, device=dev)

    def chunk():
        gdn.gdn_chunk_prefill(y, dims, d["a"], d["b"], d["A_log"], d["dt_bias"], cu_seqlens=cu,
                              initial_state=d["S0"], final_state=Sf, ckpt_every=w.ckpt_every,
                              state_ckpt_out=Sck, o=o, workspace=cws)

    chunk()
    cms = timed(chunk, steps)
    launches += 1 + steps * gdn.gdn_chunk_prefill_launches(n, T, dims, w.dtype, cu_seqlens=cu is not None)
    del y
    c_avg = statistics.mean(cms) / 1e3
    flops = FLOP_PER_TOKEN_HEAD * T * s.H_v
    res = {
        "workload": name, "tokens_per_call": T, "sequences": n, "H_k": s.H_k, "H_v": s.H_v,
        "ckpt_every": w.ckpt_every, "initial_states": w.init_state,
        "value": round(T / (statistics.mean(ms) / 1e3), 1), "unit": "tokens/s",
        "ms_per_call": round(statistics.mean(ms), 4), "calls": steps,
        "call": "gdn_layer_prefill (the chunk kernels with conv1d + SiLU inside, rmsnorm_gated)",
        "chunk_prefill_ms": round(c_avg * 1e3, 4),
        "roofline": {"kernel": "gdn_chunk_prefill", "bound": "tensor",
                     "achieved": round(flops / c_avg / 1e12, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(flops / c_avg / 1e12 / pk["bf16_tflops"], 4),
                     "frac_of_sustained": round(flops / c_avg / 1e12 / pk["bf16_tflops_sustained"], 4),
                     "algorithmic_flop_per_launch": flops},
        "l2": "calls back to back; inputs larger than L2 (a flush right before a call would leave its "
              "own dirty lines for the call to write back)",
        "input_generation_s": round(t_gen, 1),
    }
    if w.decode_steps and w.decode_batch:
        # the decode tail: fused steps of one token per sequence from the final states
        dec = W.decode_inputs(s, w.dtype, w.decode_batch, w.decode_steps, seed=w.seed + 100)
        dd = {k: v.to(dev) for k, v in dec.items()}
        Sd, csd = Sf.clone(), csf.clone()
        outd = torch.empty((w.decode_batch, s.H_v * s.d_v), dtype=w.dtype, device=dev)
        it = iter(range(w.decode_steps))

        def dstep():
            t = next(it)
            gdn.gdn_decode_step(dd["qkv"][t], dd["z"][t], dd["a"][t], dd["b"][t], d["conv_w"], d["A_log"],
                                d["dt_bias"], d["norm_w"], dims, Sd, csd, out=outd)

        dms = timed(dstep, w.decode_steps, gap=True)
        launches += w.decode_steps
        dbytes = w.decode_batch * decode_step_bytes_per_seq(s)
        res["decode_tail"] = {
            "batch": w.decode_batch, "steps": w.decode_steps,
            "value": round(w.decode_batch * w.decode_steps / (sum(dms) / 1e3), 1), "unit": "tokens/s",
            "ms_per_step": round(statistics.mean(dms), 4), "call": "gdn_decode_step (one kernel per step)",
            "hbm_frac": round(dbytes / (statistics.mean(dms) / 1e3) / 1e9 / pk["hbm_gbs"], 4),
            "note": "one sequence per step, L2 flushed before each: launch-latency bound (6.5 MB per step)"}
    del d, inp
    torch.cuda.empty_cache()
    return res, launches


# --------------------------------------------------------------------------- our arm
def run_ours(args):
    import gated_deltanet_linear_core_gb300 as gdn
    from gated_deltanet_linear_core_gb300 import build as gbuild
    gbuild.build()

    dist, rank, world, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    pk = peaks()

    wp = W.WORKLOADS[PREFILL]
    s = wp.shape
    dims = gdn.GDNDims(s.H_k, s.H_v, s.d_k, s.d_v)
    inp = W.workload_inputs(PREFILL)
    T = int(inp["mixed_qkv"].shape[0])
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    # RING copies of the per-call inputs: call i of a step reads copy i % RING,
    # last touched RING - 1 calls (> 2 GB of traffic) earlier, so every call
    # starts with its inputs out of the 129 MB L2
    ring = [{k: d[k].clone() for k in ("mixed_qkv", "z", "a", "b")} for _ in range(RING)]
    ring_out = [torch.empty((T, s.H_v * s.d_v), dtype=wp.dtype, device=dev) for _ in range(RING)]
    y = torch.empty_like(d["mixed_qkv"])
    conv_out = torch.empty((1, s.conv_dim, 3), dtype=wp.dtype, device=dev)
    S = torch.empty((1, s.H_v, s.d_k, s.d_v), dtype=torch.float32, device=dev)
    o = torch.empty((T, s.H_v, s.d_v), dtype=wp.dtype, device=dev)
    out = torch.empty((T, s.H_v * s.d_v), dtype=wp.dtype, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    lws = torch.empty(gdn.gdn_layer_prefill_workspace_size(1, T, dims, wp.dtype), dtype=torch.uint8, device=dev)
    cws = torch.empty(gdn.gdn_chunk_prefill_workspace_size(1, T, dims, wp.dtype), dtype=torch.uint8, device=dev)

    def prefill_step(ev=None):
        # the headline step: args.calls gdn_layer_prefill calls of one 4096-token
        # sequence each, over the ring of input copies; events only at its ends
        if ev:
            ev[0].record(stream)
        for i in range(args.calls):
            x = ring[i % RING]
            gdn.gdn_layer_prefill(x["mixed_qkv"], x["z"], x["a"], x["b"], d["conv_w"], d["A_log"], d["dt_bias"],
                                  d["norm_w"], dims, out=ring_out[i % RING], final_state=S,
                                  conv_state_out=conv_out, workspace=lws)
        if ev:
            ev[3].record(stream)

    def staged_step(ev):
        # the same kernels as three calls with events between them, for the
        # per-call times (an event between two kernels keeps the second from
        # being placed early, so these steps are a little longer)
        ev[0].record(stream)
        gdn.gdn_conv1d_fwd(d["mixed_qkv"], d["conv_w"], dims, None, None, conv_out, y=y)
        ev[1].record(stream)
        gdn.gdn_chunk_prefill(y, dims, d["a"], d["b"], d["A_log"], d["dt_bias"], final_state=S, o=o,
                              workspace=cws)
        ev[2].record(stream)
        gdn.gdn_rmsnorm_gated(o, d["z"], d["norm_w"], dims, out=out)
        ev[3].record(stream)

    clocks = ClockSampler(local)
    launches = 0

    # ---- prefill, device-resident inputs
    for _ in range(args.warmup):
        flush.zero_()
        prefill_step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    clocks.mark(True)
    for k in range(args.steps):
        flush.zero_()  # L2 flush between steps, outside the timed events
        prefill_step(evs[k])
    torch.cuda.synchronize(dev)
    clocks.mark(False)
    barrier(dist, dev)
    chunk_launches = gdn.gdn_chunk_prefill_launches(1, T, dims, wp.dtype, cu_seqlens=None)
    # the chunk kernels (conv1d + SiLU and the conv state inside them), the norm
    step_launches = gdn.gdn_layer_prefill_launches(1, T, dims, wp.dtype, cu_seqlens=None)
    launches += args.steps * args.calls * step_launches
    step_ms = [e[0].elapsed_time(e[3]) for e in evs]

    # per-call times
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    clocks.mark(True)
    for k in range(args.steps):
        flush.zero_()
        staged_step(sev[k])
    torch.cuda.synchronize(dev)
    clocks.mark(False)
    # the three calls: conv (one kernel: one sequence, no cu_seqlens, state_out
    # apart from state_in, so the tiles write the conv state), chunk, norm
    launches += args.steps * (2 + chunk_launches)
    conv_ms = [e[0].elapsed_time(e[1]) for e in sev]
    chunk_ms = [e[1].elapsed_time(e[2]) for e in sev]
    norm_ms = [e[2].elapsed_time(e[3]) for e in sev]

    # the conv and RMSNormGated calls alone, back to back over the ring of input
    # copies (each call's inputs out of L2, as in the headline step; in the
    # staged pass the norm reads o straight after the chunk kernel wrote it,
    # much of it from L2): their HBM rooflines.  A flush right before a call
    # would leave ~126 MB of the flush's own dirty lines for the call to write
    # back; back to back, each call writes back what earlier calls left, as in
    # a running layer.
    ring_o = [torch.empty_like(o) for _ in range(RING)]
    for r_o in ring_o:
        r_o.copy_(o)

    def alone(fn):
        for i in range(RING):
            fn(i)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        torch.cuda.synchronize(dev)
        clocks.mark(True)
        for k in range(args.steps):
            ev[k][0].record(stream)
            for i in range(args.calls):
                fn(i % RING)
            ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark(False)
        return statistics.mean(a_.elapsed_time(b_) for a_, b_ in ev) / 1e3 / args.calls

    y_ring = [torch.empty_like(y) for _ in range(RING)]
    conv_alone = alone(lambda i: gdn.gdn_conv1d_fwd(ring[i]["mixed_qkv"], d["conv_w"], dims, None, None, conv_out,
                                                    y=y_ring[i]))
    del y_ring
    norm_alone = alone(lambda i: gdn.gdn_rmsnorm_gated(ring_o[i], ring[i]["z"], d["norm_w"], dims, out=ring_out[i]))
    del ring_o
    launches += 2 * (args.steps * args.calls + RING)
    # algorithmic bytes: conv reads x and writes y (2 B each per channel-token)
    # plus the conv state out; the norm reads o and z and writes out
    conv_bytes = T * s.conv_dim * 2 * 2 + s.conv_dim * 3 * 2
    norm_bytes = T * s.H_v * s.d_v * 2 * 3
    hbm_alone = {
        kname: {"kernel": kname, "bound": "hbm", "ms": round(t * 1e3, 4),
                "achieved": round(nb / t / 1e9, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(nb / t / 1e9 / pk["hbm_gbs"], 4), "algorithmic_bytes_per_launch": nb,
                "l2": f"back to back over {RING} input copies (each call's inputs out of L2)"}
        for kname, t, nb in (("gdn_conv1d_fwd", conv_alone, conv_bytes),
                             ("gdn_rmsnorm_gated", norm_alone, norm_bytes))}

    # ---- head sharding: the first rank's shard of a tensor-parallel group of
    # 2, 4 and 8 ranks (head_shard), timed like the conv and norm above over the
    # shard's slices of the input copies.  The ranks of a group run their own
    # heads at the same time on their own GPUs, with no exchange inside the
    # core, so the group takes one shard's time per call.
    full_call_ms = statistics.mean(step_ms) / args.calls
    head_shards = {}
    for tp in (2, 4, 8):
        sh = gdn.head_shard(dims, 0, tp)
        ch = sh.channels.to(dev)
        zc = slice(sh.h0 * s.d_v, sh.h1 * s.d_v)
        sring = [{"mixed_qkv": x["mixed_qkv"][:, ch].contiguous(), "z": x["z"][:, zc].contiguous(),
                  "a": x["a"][:, sh.h0:sh.h1].contiguous(), "b": x["b"][:, sh.h0:sh.h1].contiguous()}
                 for x in ring]
        s_w = d["conv_w"][ch].contiguous()
        s_alog, s_dtb = d["A_log"][sh.h0:sh.h1].contiguous(), d["dt_bias"][sh.h0:sh.h1].contiguous()
        s_out = [torch.empty((T, (sh.h1 - sh.h0) * s.d_v), dtype=wp.dtype, device=dev) for _ in range(RING)]
        s_S = torch.empty((1, sh.h1 - sh.h0, s.d_k, s.d_v), dtype=torch.float32, device=dev)
        s_cs = torch.empty((1, ch.numel(), 3), dtype=wp.dtype, device=dev)
        s_ws = torch.empty(gdn.gdn_layer_prefill_workspace_size(1, T, sh.dims, wp.dtype), dtype=torch.uint8,
                           device=dev)
        t_sh = alone(lambda i: gdn.gdn_layer_prefill(
            sring[i]["mixed_qkv"], sring[i]["z"], sring[i]["a"], sring[i]["b"], s_w, s_alog, s_dtb, d["norm_w"],
            sh.dims, out=s_out[i], final_state=s_S, conv_state_out=s_cs, workspace=s_ws))
        launches += (args.steps * args.calls + RING) * gdn.gdn_layer_prefill_launches(1, T, sh.dims, wp.dtype,
                                                                                      cu_seqlens=False)
        head_shards[f"tp{tp}"] = {
            "key_heads": sh.dims.H_k, "value_heads": sh.dims.H_v, "ms_per_call": round(t_sh * 1e3, 4),
            "group_tokens_per_s": round(T / t_sh, 1),
            "speedup_over_one_gpu": round(full_call_ms / (t_sh * 1e3), 3)}
        del sring, s_out, s_ws
    torch.cuda.empty_cache()

    total_s = max_over_ranks(dist, sum(step_ms) / 1e3, dev)
    value = world * T * args.calls * args.steps / total_s
    chunk_avg = sum(chunk_ms) / len(chunk_ms) / 1e3

    # the same chunk stage with each chunk's (I + A)^-1 formed as the
    # Neumann-style product instead of the direct solve (GDN_SOLVE_NEUMANN)
    def neumann_chunk():
        gdn.gdn_chunk_prefill(y, dims, d["a"], d["b"], d["A_log"], d["dt_bias"], final_state=S,
                              o=o, solve="neumann")

    for _ in range(args.warmup):
        flush.zero_()
        neumann_chunk()
    nev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    clocks.mark(True)
    for k in range(args.steps):
        flush.zero_()
        nev[k][0].record(stream)
        neumann_chunk()
        nev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(False)
    launches += args.steps * chunk_launches
    neumann_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in nev)
    chunk_solve = {"direct_ms": round(chunk_avg * 1e3, 4), "neumann_ms": round(neumann_ms, 4),
                   "call": "gdn_chunk_prefill, flags GDN_QK_L2NORM vs | GDN_SOLVE_NEUMANN"}

    # chunk-size sweep on the tensor-core path (bf16; a chunk of 16 or 32 tokens
    # fills the first rows of a 64-row tile, over more workspace segments)
    tc_sweep = {}
    for c in (16, 32, 64):
        def tc_chunk():
            gdn.gdn_chunk_prefill(y, dims, d["a"], d["b"], d["A_log"], d["dt_bias"], final_state=S, o=o, chunk=c)
        for _ in range(args.warmup):
            flush.zero_()
            tc_chunk()
        cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        torch.cuda.synchronize(dev)
        clocks.mark(True)
        for k in range(args.steps):
            flush.zero_()
            cev[k][0].record(stream)
            tc_chunk()
            cev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark(False)
        launches += args.steps * gdn.gdn_chunk_prefill_launches(1, T, dims, wp.dtype, cu_seqlens=None, chunk=c)
        ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in cev)
        tc_sweep[str(c)] = {"ms": round(ms, 4), "tokens_per_s": round(T / (ms / 1e3), 1),
                            "launches": gdn.gdn_chunk_prefill_launches(1, T, dims, wp.dtype, cu_seqlens=None,
                                                                       chunk=c)}

    # and on the CUDA-core path (f32 arithmetic): the same workload in f32
    yf = y.float()
    af, bf_ = d["a"].float(), d["b"].float()
    of = torch.empty((T, s.H_v, s.d_v), dtype=torch.float32, device=dev)
    sweep = {}
    for c in (16, 32, 64):
        def ffma_chunk():
            gdn.gdn_chunk_prefill(yf, dims, af, bf_, d["A_log"], d["dt_bias"], final_state=S, o=of, chunk=c)
        ffma_chunk()
        cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
        torch.cuda.synchronize(dev)
        for k in range(3):
            flush.zero_()
            cev[k][0].record(stream)
            ffma_chunk()
            cev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        launches += 3  # the timed calls (one kernel each)
        ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in cev)
        sweep[str(c)] = {"ms": round(ms, 4), "tokens_per_s": round(T / (ms / 1e3), 1)}
    del yf, af, bf_, of
    chunk_sweep = {"tensor_core": {"path": "tcgen05 (bf16 operands, f32 state)", "by_chunk": tc_sweep},
                   "cuda_core": {"path": "CUDA-core (f32 FFMA), f32 copies of the workload", "by_chunk": sweep},
                   "call": "gdn_chunk_prefill, flags | GDN_CHUNK(c)"}
    flops = FLOP_PER_TOKEN_HEAD * T * s.H_v
    achieved_tf = flops / chunk_avg / 1e12
    ncu_bytes = traffic_record("chunk_prefill")
    # the chunk stage's intensity is below the ridge, so HBM co-binds: the
    # tensor fraction it could reach at full bandwidth is min(1, BW * I / peak)
    cbytes = chunk_bytes_per_token(s) * T
    intensity = flops / cbytes
    roofline = {"kernel": "gdn_chunk_prefill", "bound": "tensor", "achieved": round(achieved_tf, 2),
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved_tf / pk["bf16_tflops"], 4),
                "peak_source": pk["source"] + " (bf16 burst)",
                "frac_of_sustained": round(achieved_tf / pk["bf16_tflops_sustained"], 4),
                "traffic": ncu_bytes, "algorithmic_flop_per_launch": flops,
                "hbm": {"algorithmic_bytes_per_launch": cbytes,
                        "algorithmic_gbs": round(cbytes / chunk_avg / 1e9, 1),
                        "frac": round(cbytes / chunk_avg / 1e9 / pk["hbm_gbs"], 4),
                        "dram_gbs": None if ncu_bytes is None else round(ncu_bytes / chunk_avg / 1e9, 1),
                        "dram_frac": None if ncu_bytes is None else round(ncu_bytes / chunk_avg / 1e9 / pk["hbm_gbs"], 4)},
                "ceiling_frac": round(min(1.0, pk["hbm_gbs"] * 1e9 * intensity / (pk["bf16_tflops"] * 1e12)), 4)}

    # ---- decode (64 sequences x one token per step)
    wd = W.WORKLOADS[DECODE]
    B = wd.decode_batch
    nd = min(wd.decode_steps, args.decode_steps)
    dinp = W.workload_inputs(DECODE)
    dd = {k: v.to(dev) for k, v in dinp.items()}
    Sd = dd["S0"].clone()
    csd = dd["conv_state0"].clone()
    yd = torch.empty((B, s.conv_dim), dtype=wd.dtype, device=dev)
    od = torch.empty((B, s.H_v, s.d_v), dtype=wd.dtype, device=dev)
    outd = torch.empty((B, s.H_v * s.d_v), dtype=wd.dtype, device=dev)

    def decode_step(t, ev=None):
        if ev:
            ev[0].record(stream)
        gdn.gdn_conv1d_update(dd["qkv"][t], dd["conv_w"], csd, dims, y=yd)
        if ev:
            ev[1].record(stream)
        gdn.gdn_recurrent_decode(yd, Sd, dims, dd["a"][t], dd["b"][t], dd["A_log"], dd["dt_bias"],
                                 o=od)
        if ev:
            ev[2].record(stream)
        gdn.gdn_rmsnorm_gated(od, dd["z"][t], dd["norm_w"], dims, out=outd)
        if ev:
            ev[3].record(stream)

    for t in range(min(args.warmup, nd)):
        decode_step(t)
    devs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nd)]
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    clocks.mark(True)
    for t in range(nd):
        decode_step(t, devs[t])
    torch.cuda.synchronize(dev)
    clocks.mark(False)
    barrier(dist, dev)
    launches += nd * 3
    dstep_ms = [e[0].elapsed_time(e[3]) for e in devs]
    dker_ms = [e[1].elapsed_time(e[2]) for e in devs]
    dbytes = B * decode_kernel_bytes_per_seq(s)
    dker_avg = sum(dker_ms) / len(dker_ms) / 1e3
    d_gbs = dbytes / dker_avg / 1e9

    # the same steps as one fused kernel per step (gdn_decode_step), from the
    # same initial states
    Sd.copy_(dd["S0"])
    csd.copy_(dd["conv_state0"])

    def fused_step(t):
        gdn.gdn_decode_step(dd["qkv"][t], dd["z"][t], dd["a"][t], dd["b"][t], dd["conv_w"],
                            dd["A_log"], dd["dt_bias"], dd["norm_w"], dims, Sd, csd, out=outd)

    for t in range(min(args.warmup, nd)):
        fused_step(t)
    Sd.copy_(dd["S0"])
    csd.copy_(dd["conv_state0"])
    fevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(nd)]
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    clocks.mark(True)
    for t in range(nd):
        fevs[t][0].record(stream)
        fused_step(t)
        fevs[t][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(False)
    barrier(dist, dev)
    launches += nd
    fstep_ms = [a_.elapsed_time(b_) for a_, b_ in fevs]
    # the same nd steps captured as one CUDA graph and replayed, as a serving
    # loop runs its decode step: one kernel per step, launched from the graph
    # with no host and no event between steps (the states carry on from replay
    # to replay); the per-step events above add their own gap to every step
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize(dev)
    with torch.cuda.graph(graph):
        for t in range(nd):
            fused_step(t)
    GR = 4
    for _ in range(2):
        graph.replay()
    gev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    clocks.mark(True)
    gev[0].record(torch.cuda.current_stream(dev))
    for _ in range(GR):
        graph.replay()
    gev[1].record(torch.cuda.current_stream(dev))
    torch.cuda.synchronize(dev)
    clocks.mark(False)
    barrier(dist, dev)
    launches += nd * (GR + 2)
    g_step_ms = gev[0].elapsed_time(gev[1]) / (GR * nd)
    del graph
    ftotal = max_over_ranks(dist, g_step_ms * nd / 1e3, dev)
    fbytes = B * decode_step_bytes_per_seq(s)
    f_gbs = fbytes / (g_step_ms / 1e3) / 1e9
    # speculative-decoding verification: K draft tokens per sequence per call,
    # states read from one cache slot and written to K others
    KV = 4
    nv = nd // KV
    S_pool = torch.empty(((KV + 1) * B,) + tuple(Sd.shape[1:]), dtype=torch.float32, device=dev)
    cs_pool = torch.empty(((KV + 1) * B,) + tuple(csd.shape[1:]), dtype=csd.dtype, device=dev)
    S_pool[:B].copy_(dd["S0"])
    cs_pool[:B].copy_(dd["conv_state0"])
    vslots = (torch.arange(KV + 1, device=dev, dtype=torch.int32)[None, :] * B +
              torch.arange(B, device=dev, dtype=torch.int32)[:, None]).contiguous()
    vin = [{k: dd[k][KV * i:KV * (i + 1)].transpose(0, 1).contiguous() for k in ("qkv", "z", "a", "b")}
           for i in range(nv)]
    vout = torch.empty((B, KV, s.H_v * s.d_v), dtype=wd.dtype, device=dev)

    def verify_call(i):
        v = vin[i]
        gdn.gdn_decode_verify(v["qkv"], v["z"], v["a"], v["b"], dd["conv_w"], dd["A_log"],
                              dd["dt_bias"], dd["norm_w"], dims, S_pool, cs_pool, vslots, out=vout)

    for i in range(min(args.warmup, nv)):
        verify_call(i)
    vevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(nv)]
    torch.cuda.synchronize(dev)
    clocks.mark(True)
    for i in range(nv):
        vevs[i][0].record(stream)
        verify_call(i)
        vevs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(False)
    launches += nv
    vms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in vevs)
    vbytes = B * verify_bytes_per_seq(s, KV)
    v_gbs = vbytes / (vms / 1e3) / 1e9
    verify = {
        "draft_tokens": KV, "value": round(world * B * KV / (vms / 1e3), 1), "unit": "tokens/s",
        "ms_per_call": round(vms, 4), "calls": nv, "call": "gdn_decode_verify (one kernel per call)",
        "roofline": {"kernel": "gdn_decode_verify", "bound": "hbm", "achieved": round(v_gbs, 1),
                     "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(v_gbs / pk["hbm_gbs"], 4),
                     "peak_source": pk["source"] + " (HBM copy)",
                     "traffic": traffic_record("decode_verify"),
                     "algorithmic_bytes_per_launch": vbytes},
    }

    decode = {
        "workload": DECODE, "value": round(world * B * nd / ftotal, 1), "unit": "tokens/s",
        "ms_per_step": round(g_step_ms, 4), "steps": nd, "batch": B,
        "call": "gdn_decode_step (one fused kernel per step)",
        "timing": f"{nd} steps as one CUDA graph, replayed {GR} times (event pair around the replays)",
        "ms_per_step_with_events": round(sum(fstep_ms) / nd, 4),
        "roofline": {"kernel": "gdn_decode_step", "bound": "hbm", "achieved": round(f_gbs, 1),
                     "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(f_gbs / pk["hbm_gbs"], 4),
                     "peak_source": pk["source"] + " (HBM copy)",
                     "traffic": traffic_record("decode_step"),
                     "algorithmic_bytes_per_launch": fbytes},
        "separate_calls": {
            "value": round(world * B * nd / max_over_ranks(dist, sum(dstep_ms) / 1e3, dev), 1),
            "ms_per_step": round(sum(dstep_ms) / nd, 4),
            "per_kernel_ms": {"conv1d_update": round(statistics.mean(
                [e[0].elapsed_time(e[1]) for e in devs]), 4),
                "recurrent_decode": round(dker_avg * 1e3, 4),
                "rmsnorm_gated": round(statistics.mean([e[2].elapsed_time(e[3]) for e in devs]), 4)},
            "roofline": {"kernel": "gdn_recurrent_decode", "bound": "hbm",
                         "achieved": round(d_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(d_gbs / pk["hbm_gbs"], 4),
                         "peak_source": pk["source"] + " (HBM copy)",
                         "traffic": traffic_record("recurrent_decode"),
                         "algorithmic_bytes_per_launch": dbytes},
        },
        "verify": verify,
        "l2": "steps back to back, no flush: the states (201 MB, read and written every step) are "
              "larger than L2, and each step writes back what the previous one left in it",
    }

    # ---- the other prefill workloads: packed sequences with resumed states,
    # and the 262144-token sequence with checkpoints and its decode tail
    workloads = {}
    if not args.no_extra_workloads:
        for wname, k_steps in (("coder_next_varlen", args.steps), ("qwen36_27b_long", min(args.steps, 5))):
            r_w, l_w = prefill_workload(gdn, wname, args, dev, stream, flush, clocks, pk, k_steps, 3)
            workloads[wname] = r_w
            launches += l_w

    # ---- end to end through the C-ABI call with pinned host buffers
    # (gdn_layer_prefill_host: the copies in and out run inside the call,
    # overlapped piece by piece with the kernels)
    names = ("mixed_qkv", "z", "a", "b")
    hin = {k: inp[k].pin_memory() for k in names}
    hout = torch.empty((T, s.H_v * s.d_v), dtype=wp.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in hin.values())
    d2h = hout.numel() * hout.element_size()
    S_h = torch.empty((1, s.H_v, s.d_k, s.d_v), dtype=torch.float32, device=dev)
    cst_h = torch.empty((1, s.conv_dim, 3), dtype=wp.dtype, device=dev)
    ws_h = torch.empty(gdn._lib.load().gdn_layer_prefill_host_workspace_size(
        T, gdn._dims(dims), gdn._lib.GDN_BF16), dtype=torch.uint8, device=dev)
    host_pieces = gdn._lib.load().gdn_layer_prefill_host_pieces(T, gdn._dims(dims), gdn._lib.GDN_BF16)

    def e2e_step():
        gdn.gdn_layer_prefill_host(hin["mixed_qkv"], hin["z"], hin["a"], hin["b"], d["conv_w"],
                                   d["A_log"], d["dt_bias"], d["norm_w"], dims, h_out=hout,
                                   final_state=S_h, conv_state_out=cst_h, workspace=ws_h)

    for _ in range(args.warmup):
        e2e_step()
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    clocks.mark(True)
    for k in range(args.steps):
        flush.zero_()
        eev[k][0].record(stream)
        e2e_step()
        eev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(False)
    barrier(dist, dev)
    # per piece: conv, the chunk kernels, the norm
    piece_launches = 2 + gdn.gdn_chunk_prefill_launches(
        1, gdn._lib.load().gdn_layer_prefill_host_piece(T, gdn._dims(dims), gdn._lib.GDN_BF16),
        dims, wp.dtype, cu_seqlens=None)
    launches += args.steps * host_pieces * piece_launches
    e_total = max_over_ranks(dist, sum(a.elapsed_time(b) for a, b in eev) / 1e3, dev)
    e2e = {"value": round(world * T * args.steps / e_total, 1), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(e_total * 1e3 / args.steps, 4),
           "call": f"gdn_layer_prefill_host, {host_pieces} pieces"}
    clocks.stop()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp, s, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_s * 1e3 / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) activations, random layer parameters)",
            "config": {"workload": PREFILL, "tokens_per_call": T, "calls_per_step": args.calls,
                       "tokens_per_step": T * args.calls, "H_k": s.H_k, "H_v": s.H_v,
                       "d_k": s.d_k, "d_v": s.d_v, "chunk": 64, "state": "f32",
                       "l2": f"each call reads one of {RING} input copies ({RING} x 135 MB), last read "
                             f"{RING - 1} calls earlier; L2 also flushed (512 MiB write) between steps",
                       "parallelism": f"replicas x{world}"},
            "call": "gdn_layer_prefill (the chunk kernels with conv1d + SiLU inside, rmsnorm_gated)",
            "chunk_solve": chunk_solve,
            "chunk_sweep": chunk_sweep,
            "per_kernel_ms": {"conv1d_fwd": round(statistics.mean(conv_ms), 4),
                              "chunk_prefill": round(statistics.mean(chunk_ms), 4),
                              "rmsnorm_gated": round(statistics.mean(norm_ms), 4)},
            "roofline": roofline,
            "hbm_kernels": hbm_alone,
            "prefill_workloads": workloads,
            "head_shards": {"workload": PREFILL, "rank": 0, "calls": args.steps * args.calls,
                            "note": "one rank's shard timed on this GPU; the group's ranks run theirs "
                                    "at the same time on their own GPUs, so the group takes one shard's "
                                    "time per call",
                            **head_shards},
            "decode": decode,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": launches,
            "clocks": clocks.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def cpu_baseline(inp, s, seconds):
    """The oracle (as it stands) over the whole prefill workload (all tokens,
    all heads), repeated until `seconds` of host time have passed, on this
    host's cores."""
    import oracle
    f = W.to_f64
    args = [f(inp[k]) for k in ("mixed_qkv", "z", "a", "b")]
    params = [f(inp[k]) for k in ("conv_w", "A_log", "dt_bias", "norm_w")]
    T = args[0].shape[0]
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle.layer_prefill(*args, *params, s.H_k, s.H_v, s.d_k, s.d_v)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    # one core: a bounded prefix of the same workload (the rule's cost per token
    # does not depend on the position)
    n1 = 512
    a1 = [x[:n1] for x in args]
    t1 = time.perf_counter()
    oracle.layer_prefill(*a1, *params, s.H_k, s.H_v, s.d_k, s.d_v, nthreads=1)
    t1 = time.perf_counter() - t1
    return {"value": round(passes * T / dt, 2), "unit": "tokens/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{passes} passes over the whole {PREFILL} workload ({T} tokens, all "
                      f"{s.H_v} heads), f64, {dt:.1f} s",
            "one_core": {"value": round(n1 / t1, 2), "unit": "tokens/s", "cores": 1,
                         "sample": f"the first {n1} tokens of {PREFILL} (all {s.H_v} heads), f64, "
                                   f"{t1:.1f} s"}}


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The CPU oracle timed as the reference implementation, on a bounded
    sample per step of the same workload."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    wp = W.WORKLOADS[PREFILL]
    s = wp.shape
    inp = W.workload_inputs(PREFILL)
    tokens = args.ref_tokens
    f = W.to_f64
    params = [f(inp[k]) for k in ("conv_w", "A_log", "dt_bias", "norm_w")]
    T = int(inp["mixed_qkv"].shape[0])

    def step(k):
        t0 = (k * tokens) % max(1, T - tokens)
        xs = [f(inp[n][t0:t0 + tokens]) for n in ("mixed_qkv", "z", "a", "b")]
        a = time.perf_counter()
        oracle.layer_prefill(*xs, *params, s.H_k, s.H_v, s.d_k, s.d_v)
        return time.perf_counter() - a

    for k in range(args.warmup):
        step(k)
    times = [step(k) for k in range(args.steps)]
    total = sum(times)
    value = tokens * args.steps / total
    cores = oracle.max_threads()
    sample = (f"{tokens} tokens per step (all {s.H_v} heads) of {PREFILL}, f64 oracle, "
              f"{cores} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) activations, random layer parameters)",
        "config": {"workload": PREFILL, "tokens_per_step": tokens, "H_k": s.H_k, "H_v": s.H_v,
                   "d_k": s.d_k, "d_v": s.d_v},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-steps", type=int, default=256)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-tokens", type=int, default=4096)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--calls", type=int, default=64,
                    help="gdn_layer_prefill calls (4096-token sequences) per timed prefill step")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="skip the varlen and 262144-token prefill workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
