"""Benchmark of the GDN mixer hot path on GB300 (one JSON line on rank 0).

Headline workload: batched decode, 128 sequences x 1 token, H_k = 16, H_v = 32,
d_k = d_v = 128, conv width 4, bf16 activations / conv state, f32 recurrent state.  One
step is one gdn_decode_batched call (conv + SiLU + L2, gates, gated delta rule, gated
RMSNorm: one fused kernel launch) over the 128 sequences.  Steps rotate over 4 state pools
(4 x 256 MiB), so every step streams its state from HBM rather than L2.

Also reported (key "modes"): the ragged verify of 128 sequences with k ~ U{2..16}, the
accepted-draft fold after it, the decode step on half-width (fp16) state pools, the
8192-token chunked prefill and the mixed serving step, each with its own throughput and
roofline fraction.

`--impl reference` times the fp64 CPU oracle on this host's cores on a bounded sample of
the same workload.  Under torchrun every rank runs an independent replica (the mixer has
no cross-sequence exchange); value = all ranks' tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN decode tokens/s @128 seqs + HBM GB/s % of peak; prefill tokens/s + tensor %"
N_SEQ = 128
POOLS = 4
REF_SAMPLE = 16  # sequences per reference-arm step
HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0

# Algorithmic bytes of one decode step (every byte the method must move once):
#   per token: state read + write 2*32*128*128*4 = 4,194,304; conv state read + write
#   2*8192*4*2 = 131,072; qkv 8192*2 + z 4096*2 + a, b 2*32*2 + y 4096*2 = 32,896;
#   per launch: conv_w 8192*4*4 + A_log, dt_bias 2*32*4 + norm_w 128*4 = 131,840.
DECODE_BYTES_PER_TOKEN = 4_194_304 + 131_072 + 32_896
WEIGHT_BYTES = 131_840


def verify_bytes(ks, state_elem: int = 4) -> int:
    """Algorithmic bytes of one ragged verify launch (no conv intermediates)."""
    state = 32 * 128 * 128 * state_elem
    return int(sum(state + k * state + 131_072 + k * 32_896 for k in ks) + WEIGHT_BYTES)


def prefill_flops(T: int, C: int = 64) -> float:
    """Dense-contraction flops of the chunked form per full 64-token chunk (H_k = 16, H_v = 32,
    d = 128): 2*H_k*2*C^2*d (QK^T, KK^T) + 2*H_v*(C^2 d + 2 C^2 d + 3 C d^2)."""
    per_chunk = 2 * 16 * 2 * C * C * 128 + 2 * 32 * (C * C * 128 + 2 * C * C * 128 + 3 * C * 128 * 128)
    return per_chunk * (T / C)


def prefill_bytes(T: int) -> int:
    """qkv + z + a, b in, y out (bf16), plus weights; state starts and ends in HBM."""
    per_tok = 8192 * 2 + 4096 * 2 + 2 * 32 * 2 + 4096 * 2
    return T * per_tok + 2 * 2 * 1024 * 1024 + 2 * 8192 * 4 * 2 + WEIGHT_BYTES


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, BF16_FALLBACK_TFLOPS, "fallback"


def _kernel_sources_hash() -> str:
    """Hash of the decode kernel's sources without their comments and blank lines, so
    that a comment edit does not disown the counters captured on the same code."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_deltanet_layer_conv1d_gb300", "csrc")
    for name in ("recurrent.cu", "common.cuh"):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def ncu_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "gdn_recurrent_decode_128seq.md")
    try:
        with open(path) as f:
            txt = f.read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_sources_sha256_16:\s*([0-9a-f]+)", txt)
    m_t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not (m_hash and m_t) or m_hash.group(1) != _kernel_sources_hash():
        return None
    return float(m_t.group(1))


def slowest_rank(ms: float, device=None) -> float:
    """The largest of every rank's time: replicas finish when the slowest one does."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job units per second: every rank's units over the slowest rank's time."""
    return units_per_rank * world / (ms * 1e-3)


class ClockSampler:
    """nvidia-smi clock / throttle samples while the GPU works."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm
class DecodeBench:
    def __init__(self, device, seed=0):
        import torch

        from gated_deltanet_layer_conv1d_gb300 import device as dev
        from gated_deltanet_layer_conv1d_gb300 import gdn
        from gated_deltanet_layer_conv1d_gb300 import workloads as wl
        self.torch, self.gdn = torch, gdn
        self.w = wl.batched_decode(n=N_SEQ, steps=POOLS, seed=seed)
        w = self.w
        self.dims = dev.dims_of(w.shape)
        self.weights = dev.weights_to(w, device)
        # POOLS independent slot pools of 128 sequences each, one per rotating step
        h_pool, conv_pool, _ = dev.states_to(w, device, n_slots=N_SEQ)
        self.h_pool = h_pool.repeat(POOLS, 1, 1, 1).contiguous()
        self.conv_pool = conv_pool.repeat(POOLS, 1, 1).contiguous()
        self.n_slots = POOLS * N_SEQ
        self.slots = [torch.arange(p * N_SEQ, (p + 1) * N_SEQ, dtype=torch.int32, device=device)
                      for p in range(POOLS)]
        self.inputs = [dev.tokens_to(t, torch.bfloat16, device) for t in [w.tokens] + w.steps]
        self.y = torch.empty((N_SEQ, 4096), dtype=torch.bfloat16, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.stream = torch.cuda.current_stream(device)

    def step(self, i: int):
        p = i % POOLS
        self.gdn.gdn_decode_batched(self.dims, self.weights, self.inputs[p], N_SEQ, self.h_pool,
                                    self.conv_pool, self.n_slots, self.slots[p], self.y, None,
                                    self.status, self.stream)

    def e2e(self, steps: int, warmup: int):
        """The same step end to end: every step's inputs come in from pinned host memory and
        its y goes back to pinned host memory, as a serving loop runs it.  Each step's
        inputs travel as one block ([qkv | z | a | b] rows) on an input-copy stream and its
        y on an output-copy stream, overlapping the neighbouring steps' kernels; two device
        input and output buffers alternate."""
        torch = self.torch
        dev = self.y.device
        n = N_SEQ
        widths = {"qkv": 8192, "z": 4096, "a": 32, "b": 32}
        offs, o = {}, 0
        for k, wdt in widths.items():
            offs[k] = o
            o += n * wdt
        total = o

        def views(block):
            return self.gdn.Inputs(*[block[offs[k]:offs[k] + n * widths[k]].view(n, widths[k])
                                     for k in ("qkv", "z", "a", "b")])

        host_blocks = []
        for x in self.inputs:  # one pinned block per rotating pool
            hb = torch.empty(total, dtype=torch.bfloat16).pin_memory()
            for k in widths:
                hb[offs[k]:offs[k] + n * widths[k]].copy_(getattr(x, k).reshape(-1).cpu())
            host_blocks.append(hb)
        dev_blocks = [torch.empty(total, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        dev_in = [views(b) for b in dev_blocks]
        ys = [torch.empty_like(self.y) for _ in range(2)]
        y_host = [torch.empty(self.y.shape, dtype=self.y.dtype).pin_memory() for _ in range(2)]
        h2d = total * 2
        d2h = self.y.numel() * self.y.element_size()
        cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_ready = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        released = [torch.cuda.Event() for _ in range(2)]

        def one(i):
            b = i & 1
            with torch.cuda.stream(cin):
                if i >= 2:
                    cin.wait_event(released[b])  # step i-2 is done with buffers b
                dev_blocks[b].copy_(host_blocks[i % POOLS], non_blocking=True)
                in_ready[b].record(cin)
            self.stream.wait_event(in_ready[b])
            self.gdn.gdn_decode_batched(self.dims, self.weights, dev_in[b], N_SEQ, self.h_pool,
                                        self.conv_pool, self.n_slots, self.slots[i % POOLS],
                                        ys[b], None, self.status, self.stream)
            computed[b].record(self.stream)
            with torch.cuda.stream(cout):
                cout.wait_event(computed[b])
                y_host[b].copy_(ys[b], non_blocking=True)
                released[b].record(cout)

        for i in range(warmup):
            one(i)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(cin)  # before the first input copy
        for i in range(steps):
            one(i)
        t1.record(cout)  # after the last result copy, which follows every kernel
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / steps
        return ms, h2d, d2h

    def check_status(self):
        s = int(self.status.item())
        if s != 0:
            raise RuntimeError(f"device status {s}: {self.gdn.status_string(s)}")


def time_loop(torch, stream, fn, steps, warmup):
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def time_graph(torch, stream, fn, calls=50, reps=4):
    """GPU time per call of `fn(i, st)`, from `calls` calls captured in one CUDA graph (on a
    side stream, as capture requires) and replayed `reps` times on `stream`: no host launch
    overhead in the timed region, which for a 10 us GEMM launched from Python would
    otherwise dominate."""
    side = torch.cuda.Stream(stream.device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(3):
            fn(i, side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for i in range(calls):
            fn(i, side)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (calls * reps)


def verify_mode(device, steps, hbm_peak, warmup=3, n=N_SEQ, h16=False):
    """The 128-sequence ragged verify; h16: on fp16 state pools and intermediates."""
    import torch

    from gated_deltanet_layer_conv1d_gb300 import device as dev
    from gated_deltanet_layer_conv1d_gb300 import gdn
    from gated_deltanet_layer_conv1d_gb300 import workloads as wl
    w = wl.ragged_verify(n=n)
    ks = [int(k) for k in w.lens]
    h_pool, conv_pool, slots = dev.states_to(w, device)
    sdt = torch.float16 if h16 else torch.float32
    if h16:
        h_pool = h_pool.half()
    inter = torch.empty((n, 15, 32, 128, 128), dtype=sdt, device=device)
    hsz = 32 * 128 * 128 * (2 if h16 else 4)
    tables = dev.wy_tables_to(ks, [h_pool.data_ptr() + i * hsz for i in range(n)],
                              [[inter[i, t].data_ptr() for t in range(15)] for i in range(n)],
                              device)
    inp = dev.tokens_to(w.tokens, torch.bfloat16, device)
    y = torch.empty((sum(ks), 4096), dtype=torch.bfloat16, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    dims, weights = dev.dims_of(w.shape), dev.weights_to(w, device)
    stream = torch.cuda.current_stream(device)

    run = gdn.gdn_verify_multi_h16 if h16 else gdn.gdn_verify_multi

    def fn(i):
        run(dims, weights, inp, n, ks, tables, conv_pool, n, slots, None, y, None, status, stream)

    ms = time_loop(torch, stream, fn, steps, warmup)
    assert int(status.item()) == 0
    byts = verify_bytes(ks, 2 if h16 else 4)
    gbs = byts / (ms * 1e-3) / 1e9
    return {"workload": f"ragged_verify_{n}seq_k2to16" + ("_fp16_state_pool" if h16 else ""),
            "tokens_per_step": sum(ks),
            "ms_per_step": round(ms, 4), "value": round(sum(ks) / (ms * 1e-3), 1),
            "unit": "tokens/s", "gpu_launches_per_step": 1,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "traffic": None,
                         "algorithmic_bytes": byts}}


def decode_h16_mode(device, steps, hbm_peak, warmup=3):
    """Batched decode of 128 sequences on half-width (fp16) state pools: the same step as
    the headline, with half the state bytes.  Four rotating pools (4 x 128 MiB), as there."""
    import torch

    from gated_deltanet_layer_conv1d_gb300 import device as dev
    from gated_deltanet_layer_conv1d_gb300 import gdn
    from gated_deltanet_layer_conv1d_gb300 import workloads as wl
    w = wl.batched_decode(n=N_SEQ, steps=POOLS)
    dims, weights = dev.dims_of(w.shape), dev.weights_to(w, device)
    h_pool, conv_pool, _ = dev.states_to(w, device, n_slots=N_SEQ)
    h16 = h_pool.half().repeat(POOLS, 1, 1, 1).contiguous()
    conv_pool = conv_pool.repeat(POOLS, 1, 1).contiguous()
    slots = [torch.arange(q * N_SEQ, (q + 1) * N_SEQ, dtype=torch.int32, device=device)
             for q in range(POOLS)]
    inputs = [dev.tokens_to(t, torch.bfloat16, device) for t in [w.tokens] + w.steps]
    y = torch.empty((N_SEQ, 4096), dtype=torch.bfloat16, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)

    def fn(i):
        q = i % POOLS
        gdn.gdn_decode_batched_h16(dims, weights, inputs[q], N_SEQ, h16, conv_pool,
                                   POOLS * N_SEQ, slots[q], y, None, status, stream)

    ms = time_loop(torch, stream, fn, steps, warmup)
    assert int(status.item()) == 0
    byts = N_SEQ * (DECODE_BYTES_PER_TOKEN - 2 * 1024 * 1024) + WEIGHT_BYTES
    gbs = byts / (ms * 1e-3) / 1e9
    return {"workload": "batched_decode_128seq_1tok_fp16_state_pool", "tokens_per_step": N_SEQ,
            "ms_per_step": round(ms, 4), "value": round(N_SEQ / (ms * 1e-3), 1),
            "unit": "tokens/s", "gpu_launches_per_step": 1, "state_dtype": "f16",
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "traffic": None,
                         "algorithmic_bytes": byts}}


def fold_mode(device, steps, hbm_peak, warmup=3, n=N_SEQ):
    """The accepted-draft fold after a 128-sequence ragged verify (k ~ U{2..16}), m_i ~
    U{1..k_i} accepted; the fold is repeated on the same verify output (it is idempotent)."""
    import torch

    from gated_deltanet_layer_conv1d_gb300 import device as dev
    from gated_deltanet_layer_conv1d_gb300 import gdn
    from gated_deltanet_layer_conv1d_gb300 import workloads as wl
    w = wl.ragged_verify(n=n)
    ks = [int(k) for k in w.lens]
    rng = np.random.default_rng(1)
    m = [int(rng.integers(1, k + 1)) for k in ks]
    h_pool, conv_pool, slots = dev.states_to(w, device)
    inter = torch.empty((n, 15, 32, 128, 128), dtype=torch.float32, device=device)
    ci = torch.empty((n, 15, 8192, 4), dtype=torch.bfloat16, device=device)
    hsz = 32 * 128 * 128 * 4
    tables = dev.wy_tables_to(ks, [h_pool.data_ptr() + i * hsz for i in range(n)],
                              [[inter[i, t].data_ptr() for t in range(15)] for i in range(n)],
                              device)
    inp = dev.tokens_to(w.tokens, torch.bfloat16, device)
    y = torch.empty((sum(ks), 4096), dtype=torch.bfloat16, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    dims, weights = dev.dims_of(w.shape), dev.weights_to(w, device)
    stream = torch.cuda.current_stream(device)
    gdn.gdn_verify_multi(dims, weights, inp, n, ks, tables, conv_pool, n, slots, ci, y, None,
                         status, stream)
    acc = torch.tensor(m, dtype=torch.int32, device=device)

    def fn(i):
        gdn.gdn_fold_accepted(dims, n, ks, acc, tables, conv_pool, n, slots, ci,
                              gdn.GDN_DTYPE_BF16, status, stream)

    ms = time_loop(torch, stream, fn, steps, warmup)
    assert int(status.item()) == 0
    rolled = sum(1 for k, a in zip(ks, m) if a < k)
    byts = rolled * 2 * (2 * 1024 * 1024 + 8192 * 4 * 2) + n * 4
    gbs = byts / (ms * 1e-3) / 1e9
    return {"workload": f"accepted_fold_{n}seq_k2to16", "sequences_rolled_back": rolled,
            "ms_per_step": round(ms, 4), "value": round(n / (ms * 1e-3), 1),
            "unit": "sequences/s", "gpu_launches_per_step": 1,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "traffic": None,
                         "algorithmic_bytes": byts}}


def woa_mode(device, steps, hbm_peak, warmup=3, n=N_SEQ):
    """A speculative step of 128 sequences (k ~ U{2..16} drafts, m ~ U{1..k} accepted) in
    the two forms: the write-on-accept verify, its fold and the flag clear, against the
    verify that writes every intermediate state plus the copy fold."""
    import torch

    from gated_deltanet_layer_conv1d_gb300 import device as dev
    from gated_deltanet_layer_conv1d_gb300 import gdn
    from gated_deltanet_layer_conv1d_gb300 import workloads as wl
    w = wl.ragged_verify(n=n)
    ks = [int(k) for k in w.lens]
    rng = np.random.default_rng(1)
    m = [int(rng.integers(1, k + 1)) for k in ks]
    h_pool, conv_pool, slots = dev.states_to(w, device)
    inter = torch.empty((n, 15, 32, 128, 128), dtype=torch.float32, device=device)
    ci = torch.empty((n, 15, 8192, 4), dtype=torch.bfloat16, device=device)
    hsz = 32 * 128 * 128 * 4
    tables = dev.wy_tables_to(ks, [h_pool.data_ptr() + i * hsz for i in range(n)],
                              [[inter[i, t].data_ptr() for t in range(15)] for i in range(n)],
                              device)
    inp = dev.tokens_to(w.tokens, torch.bfloat16, device)
    y = torch.empty((sum(ks), 4096), dtype=torch.bfloat16, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    dims, weights = dev.dims_of(w.shape), dev.weights_to(w, device)
    stream = torch.cuda.current_stream(device)
    words = gdn.gdn_woa_stash_seq_floats(dims, gdn.GDN_DTYPE_BF16)
    stash = torch.empty((n, words), dtype=torch.float32, device=device)
    flag = torch.zeros(1, dtype=torch.int32, device=device)
    acc = torch.tensor(m, dtype=torch.int32, device=device)

    def woa(i):
        gdn.gdn_verify_woa(dims, weights, inp, n, ks, tables, conv_pool, n, slots, stash, n,
                           flag, y, None, status, stream)
        gdn.gdn_woa_fold(dims, n, acc, tables, conv_pool, n, slots, stash, flag,
                         gdn.GDN_DTYPE_BF16, status, stream)
        gdn.gdn_woa_clear(flag, stream)

    def copy(i):
        gdn.gdn_verify_multi(dims, weights, inp, n, ks, tables, conv_pool, n, slots, ci, y,
                             None, status, stream)
        gdn.gdn_fold_accepted(dims, n, ks, acc, tables, conv_pool, n, slots, ci,
                              gdn.GDN_DTYPE_BF16, status, stream)

    ms_woa = time_loop(torch, stream, woa, steps, warmup)
    assert int(status.item()) == 0
    ms_copy = time_loop(torch, stream, copy, steps, warmup)
    assert int(status.item()) == 0
    # algorithmic bytes of the write-on-accept step, per sequence: the verify reads the state
    # and conv state, its inputs and outputs, and writes the stash (per token alpha, k_hat,
    # delta, the raw row); the fold reads the state, the accepted tokens' factors and raw
    # rows, the conv state, and writes the state and conv state
    state, conv_b, io = 2 * 1024 * 1024, 8192 * 4 * 2, 32896
    per_tok = 32 * 4 + 16 * 128 * 4 + 32 * 128 * 4 + 8192 * 2
    byts = sum(state + conv_b + k * io + k * per_tok +
               2 * state + a * (per_tok - 8192 * 2) + min(a, 4) * 8192 * 2 + 2 * conv_b
               for k, a in zip(ks, m))
    gbs = byts / (ms_woa * 1e-3) / 1e9
    return {"workload": f"speculative_step_{n}seq_k2to16_write_on_accept",
            "tokens_per_step": sum(ks), "ms_per_step": round(ms_woa, 4),
            "value": round(sum(ks) / (ms_woa * 1e-3), 1), "unit": "tokens/s",
            "gpu_launches_per_step": 3,
            "copy_form_ms_per_step": round(ms_copy, 4),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "traffic": None,
                         "algorithmic_bytes": byts}}


def prefill_mode(device, steps, tc_peak, warmup=2, f32=False):
    """The 1 x 8192-token prefill; f32: the token-sequential f32 option (the 1e-4 class),
    timed beside the tensor-core form."""
    import torch

    from gated_deltanet_layer_conv1d_gb300 import device as dev
    from gated_deltanet_layer_conv1d_gb300 import gdn
    from gated_deltanet_layer_conv1d_gb300 import workloads as wl
    T = 8192
    w = wl.long_prefill(T)
    h_pool, conv_pool, slots = dev.states_to(w, device)
    hp = torch.tensor([h_pool.data_ptr()], dtype=torch.int64, device=device)
    cu = torch.tensor([0, T], dtype=torch.int32, device=device)
    dims, weights = dev.dims_of(w.shape), dev.weights_to(w, device)
    if f32:
        dims.prefill_precision = gdn.GDN_PREFILL_F32
    inp = dev.tokens_to(w.tokens, torch.bfloat16, device)
    y = torch.empty((T, 4096), dtype=torch.bfloat16, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    wsb = gdn.gdn_prefill_workspace_bytes(dims, 1, T, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=device) if wsb else None
    stream = torch.cuda.current_stream(device)

    def fn(i):
        gdn.gdn_prefill_chunked(dims, weights, inp, 1, cu, T, T, hp, conv_pool, 1, slots, y,
                                None, ws, status, stream)

    ms = time_loop(torch, stream, fn, steps, warmup)
    assert int(status.item()) == 0
    fl = prefill_flops(T)
    tfs = fl / (ms * 1e-3) / 1e12
    if f32:
        return {"workload": f"long_prefill_{T}tok_f32_token_sequential", "tokens_per_step": T,
                "ms_per_step": round(ms, 4), "value": round(T / (ms * 1e-3), 1),
                "unit": "tokens/s", "state_error_class": "1e-4"}
    return {"workload": f"long_prefill_{T}tok_chunk64", "tokens_per_step": T,
            "ms_per_step": round(ms, 4), "value": round(T / (ms * 1e-3), 1), "unit": "tokens/s",
            "roofline": {"bound": "tensor", "achieved": round(tfs, 2), "peak": tc_peak,
                         "unit": "TFLOP/s", "frac": round(tfs / tc_peak, 4), "traffic": None,
                         "algorithmic_flops": fl,
                         "hbm_GBps": round(prefill_bytes(T) / (ms * 1e-3) / 1e9, 1)}}


PREFILL_FLOPS_PER_TOKEN = prefill_flops(64) / 64


def proj_mode(device, steps, tc_peak, hbm_peak, warmup=3):
    """The bf16 projections around the mixer, hidden width 2048: in_proj (-> [Q|K|V|Z|b|a],
    12352 outputs) and out_proj (4096 -> 2048) at 8192 tokens (tensor-bound) and at 128
    tokens (one decode step of 128 sequences: weight-streaming, HBM-bound).  Operand sets
    rotate so every call reads more than L2 holds.  `ms` is the library call as a caller
    makes it (back-to-back calls on one stream); `graph_ms` the same calls replayed from a
    CUDA graph; cuBLAS (torch.matmul) on the same operands is timed beside from a CUDA
    graph too (`cublas_ms`), since at 128 tokens its eager loop times Python's dispatch,
    not the GPU."""
    import torch

    from gated_deltanet_layer_conv1d_gb300 import device as dev
    from gated_deltanet_layer_conv1d_gb300 import gdn
    from gated_deltanet_layer_conv1d_gb300 import workloads as wl
    dims = dev.dims_of(wl.FULL)
    width = gdn.gdn_in_proj_width(dims)
    H, vd = wl.HIDDEN, wl.FULL.z_dim
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    g = torch.Generator(device=device).manual_seed(0)

    def rnd(*shape, scale=1.0):
        return (torch.randn(*shape, generator=g, device=device) * scale).to(torch.bfloat16)

    out = {}
    for name, T, K, N in (("in_proj", 8192, H, width), ("out_proj", 8192, vd, H),
                          ("in_proj", 128, H, width), ("out_proj", 128, vd, H)):
        per_set = (T * K + N * K + T * N) * 2
        sets = max(1, -(-160 * 2**20 // per_set))
        a = [rnd(T, K) for _ in range(sets)]
        b = [rnd(N, K, scale=K ** -0.5) for _ in range(sets)]
        c = [torch.empty((T, N), dtype=torch.bfloat16, device=device) for _ in range(sets)]

        def ours(i, st=stream):
            q = i % sets
            gdn.gdn_proj_gemm(a[q], b[q], c[q], status, st)

        def cublas(i, st=None):
            q = i % sets
            torch.matmul(a[q], b[q].t(), out=c[q])  # on the current stream

        ms = time_loop(torch, stream, ours, steps, warmup)
        assert int(status.item()) == 0
        ms_graph = time_graph(torch, stream, ours, calls=20 if T >= 1024 else 50)
        assert int(status.item()) == 0
        ms_cublas = time_graph(torch, stream, cublas, calls=20 if T >= 1024 else 50)
        fl = 2.0 * T * K * N
        byts = per_set
        r = {"M": T, "N": N, "K": K, "ms": round(ms, 4), "graph_ms": round(ms_graph, 4),
             "cublas_ms": round(ms_cublas, 4), "cublas_timing": "cuda_graph_replay"}
        tfs = fl / (ms * 1e-3) / 1e12
        gbs = byts / (ms * 1e-3) / 1e9
        if T >= 1024:
            r["roofline"] = {"bound": "tensor", "achieved": round(tfs, 1), "peak": tc_peak,
                             "unit": "TFLOP/s", "frac": round(tfs / tc_peak, 4),
                             "traffic": None, "algorithmic_flops": fl}
        else:
            r["roofline"] = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                             "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "traffic": None,
                             "algorithmic_bytes": byts}
        out[f"{name}_{T}tok"] = r
    return {"workload": f"bf16 projections, hidden {H}, H_k 16, H_v 32, d 128",
            "gpu_launches_per_call": 1, "calls": out}


def proj128_profile(device, steps, warmup=3):
    """Only the two 128-token projection calls of proj_mode, eager: warmup + steps calls
    of in_proj, then of out_proj (for profiler captures)."""
    import torch

    from gated_deltanet_layer_conv1d_gb300 import device as dev
    from gated_deltanet_layer_conv1d_gb300 import gdn
    from gated_deltanet_layer_conv1d_gb300 import workloads as wl
    dims = dev.dims_of(wl.FULL)
    width = gdn.gdn_in_proj_width(dims)
    H, vd = wl.HIDDEN, wl.FULL.z_dim
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    g = torch.Generator(device=device).manual_seed(0)
    for K, N in ((H, width), (vd, H)):
        a = (torch.randn(128, K, generator=g, device=device)).to(torch.bfloat16)
        b = (torch.randn(N, K, generator=g, device=device) * K ** -0.5).to(torch.bfloat16)
        c = torch.empty((128, N), dtype=torch.bfloat16, device=device)
        for _ in range(warmup + steps):
            gdn.gdn_proj_gemm(a, b, c, status, stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0


def layer_mode(device, steps, warmup=3):
    """The whole layer around the mixer, hidden width 2048, bf16 between the steps:
    hidden -> in_proj -> mixer (reading the in_proj rows in place) -> out_proj, as one
    decode step of 128 sequences (rotating state pools larger than L2) and as the prefill
    of one 8192-token sequence.  Three launches per decode step; the prefill's are the
    projections plus the mixer's own."""
    import torch

    from gated_deltanet_layer_conv1d_gb300 import device as dev
    from gated_deltanet_layer_conv1d_gb300 import gdn
    from gated_deltanet_layer_conv1d_gb300 import workloads as wl
    out = {}
    stream = torch.cuda.current_stream(device)
    status = torch.zeros(1, dtype=torch.int32, device=device)

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(device, torch.bfloat16)

    # ---- decode: 128 sequences x 1 token
    w = wl.batched_decode(n=N_SEQ, steps=1)
    P = wl.projections(N_SEQ * POOLS, seed=5)
    dims, weights = dev.dims_of(w.shape), dev.weights_to(w, device)
    width = gdn.gdn_in_proj_width(dims)
    h_pool, conv_pool, _ = dev.states_to(w, device, n_slots=N_SEQ)
    h_pool = h_pool.repeat(POOLS, 1, 1, 1).contiguous()
    conv_pool = conv_pool.repeat(POOLS, 1, 1).contiguous()
    slots = [torch.arange(q * N_SEQ, (q + 1) * N_SEQ, dtype=torch.int32, device=device)
             for q in range(POOLS)]
    hidden = bf(P.hidden).view(POOLS, N_SEQ, wl.HIDDEN)
    w_in, w_out = bf(P.w_in), bf(P.w_out)
    rows = torch.empty((N_SEQ, width), dtype=torch.bfloat16, device=device)
    inputs = gdn.in_proj_inputs(dims, rows)
    y = torch.empty((N_SEQ, w.shape.z_dim), dtype=torch.bfloat16, device=device)
    o = torch.empty((N_SEQ, wl.HIDDEN), dtype=torch.bfloat16, device=device)

    def dec(i):
        q = i % POOLS
        gdn.gdn_in_proj(dims, hidden[q], w_in, rows, status, stream)
        gdn.gdn_decode_batched(dims, weights, inputs, N_SEQ, h_pool, conv_pool, POOLS * N_SEQ,
                               slots[q], y, None, status, stream)
        gdn.gdn_out_proj(dims, y, w_out, o, status, stream)

    ms = time_loop(torch, stream, dec, steps, warmup)
    assert int(status.item()) == 0
    out["decode_128seq_1tok"] = {"ms_per_step": round(ms, 4),
                                 "value": round(N_SEQ / (ms * 1e-3), 1), "unit": "tokens/s",
                                 "gpu_launches_per_step": 3}
    del h_pool, conv_pool

    # ---- prefill: one sequence of 8192 tokens
    T = 8192
    w = wl.long_prefill(T)
    P = wl.projections(T, seed=6)
    h_pool, conv_pool, slots1 = dev.states_to(w, device)
    hp = torch.tensor([h_pool.data_ptr()], dtype=torch.int64, device=device)
    cu = torch.tensor([0, T], dtype=torch.int32, device=device)
    weights = dev.weights_to(w, device)
    hidden, w_in, w_out = bf(P.hidden), bf(P.w_in), bf(P.w_out)
    rows = torch.empty((T, width), dtype=torch.bfloat16, device=device)
    inputs = gdn.in_proj_inputs(dims, rows)
    y = torch.empty((T, w.shape.z_dim), dtype=torch.bfloat16, device=device)
    o = torch.empty((T, wl.HIDDEN), dtype=torch.bfloat16, device=device)
    ws = torch.empty(gdn.gdn_prefill_workspace_bytes(dims, 1, T, T), dtype=torch.uint8,
                     device=device)

    def pre(i):
        gdn.gdn_in_proj(dims, hidden, w_in, rows, status, stream)
        gdn.gdn_prefill_chunked(dims, weights, inputs, 1, cu, T, T, hp, conv_pool, 1, slots1, y,
                                None, ws, status, stream)
        gdn.gdn_out_proj(dims, y, w_out, o, status, stream)

    ms = time_loop(torch, stream, pre, max(3, steps // 20), 2)
    assert int(status.item()) == 0
    out["prefill_1x8192tok"] = {"ms_per_step": round(ms, 4), "value": round(T / (ms * 1e-3), 1),
                                "unit": "tokens/s"}
    return {"workload": f"GDN layer: in_proj -> mixer -> out_proj, hidden {wl.HIDDEN}, "
                        "H_k 16, H_v 32, d 128, bf16 activations", "steps": out}


def mixed_mode(device, steps, hbm_peak, tc_peak):
    """Mixed serving step: 32 sequences prefilling U{512..4096} tokens on one stream next to
    a 96-sequence ragged verify (k ~ U{2..16}) on another; tokens/s over both."""
    import torch

    from gated_deltanet_layer_conv1d_gb300 import device as dev
    from gated_deltanet_layer_conv1d_gb300 import gdn
    from gated_deltanet_layer_conv1d_gb300 import workloads as wl
    pre, ver = wl.mixed_serving()
    dims, weights = dev.dims_of(pre.shape), dev.weights_to(pre, device)
    # prefill side
    ph, pc, ps = dev.states_to(pre, device)
    hsz = 32 * 128 * 128 * 4
    php = torch.tensor([ph.data_ptr() + i * hsz for i in range(pre.n)], dtype=torch.int64,
                       device=device)
    cu = torch.from_numpy(pre.cu_seqlens).to(device)
    T = int(pre.lens.sum())
    Lmax = int(pre.lens.max())
    pin = dev.tokens_to(pre.tokens, torch.bfloat16, device)
    py = torch.empty((T, 4096), dtype=torch.bfloat16, device=device)
    ws = torch.empty(gdn.gdn_prefill_workspace_bytes(dims, pre.n, T, Lmax), dtype=torch.uint8,
                     device=device)
    # verify side
    ks = [int(k) for k in ver.lens]
    vh, vc, vs = dev.states_to(ver, device)
    inter = torch.empty((ver.n, 15, 32, 128, 128), dtype=torch.float32, device=device)
    tables = dev.wy_tables_to(ks, [vh.data_ptr() + i * hsz for i in range(ver.n)],
                              [[inter[i, t].data_ptr() for t in range(15)] for i in range(ver.n)],
                              device)
    vin = dev.tokens_to(ver.tokens, torch.bfloat16, device)
    vy = torch.empty((sum(ks), 4096), dtype=torch.bfloat16, device=device)
    status = torch.zeros(2, dtype=torch.int32, device=device)
    main = torch.cuda.current_stream(device)
    s_pre, s_ver = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def fn(i):
        fork = torch.cuda.Event()
        fork.record(main)
        s_pre.wait_event(fork)
        s_ver.wait_event(fork)
        gdn.gdn_prefill_chunked(dims, weights, pin, pre.n, cu, T, Lmax, php, pc, pre.n, ps, py,
                                None, ws, status[0:1], s_pre)
        gdn.gdn_verify_multi(dims, weights, vin, ver.n, ks, tables, vc, ver.n, vs, None, vy,
                             None, status[1:2], s_ver)
        for st in (s_pre, s_ver):
            done = torch.cuda.Event()
            done.record(st)
            main.wait_event(done)

    def prefill_alone(i):
        gdn.gdn_prefill_chunked(dims, weights, pin, pre.n, cu, T, Lmax, php, pc, pre.n, ps, py,
                                None, ws, status[0:1], main)

    def verify_alone(i):
        gdn.gdn_verify_multi(dims, weights, vin, ver.n, ks, tables, vc, ver.n, vs, None, vy,
                             None, status[1:2], main)

    ms = time_loop(torch, main, fn, steps, 2)
    ms_pre = time_loop(torch, main, prefill_alone, steps, 2)
    ms_ver = time_loop(torch, main, verify_alone, steps, 2)
    assert int(status.abs().sum().item()) == 0
    tokens = T + sum(ks)
    fl = PREFILL_FLOPS_PER_TOKEN * T
    b_pre, b_ver = prefill_bytes(T), verify_bytes(ks)
    byts = b_ver + b_pre

    def frac(work, ms_, peak, scale):
        return round(work / (ms_ * 1e-3) / scale / peak, 4)

    return {"workload": "mixed_32prefill_U512to4096_96verify_k2to16", "tokens_per_step": tokens,
            "prefill_tokens": T, "verify_tokens": sum(ks), "ms_per_step": round(ms, 4),
            "value": round(tokens / (ms * 1e-3), 1), "unit": "tokens/s", "streams": 2,
            "roofline": {"tensor": {"achieved": round(fl / (ms * 1e-3) / 1e12, 2),
                                    "peak": tc_peak, "unit": "TFLOP/s",
                                    "frac": round(fl / (ms * 1e-3) / 1e12 / tc_peak, 4)},
                         "hbm": {"achieved": round(byts / (ms * 1e-3) / 1e9, 1),
                                 "peak": hbm_peak, "unit": "GB/s",
                                 "frac": round(byts / (ms * 1e-3) / 1e9 / hbm_peak, 4)}},
            # each part alone on one stream, same calls and sizes: the step's time against
            # their sum shows what running them side by side saves
            "parts": {"prefill": {"ms": round(ms_pre, 4), "tokens": T,
                                  "tensor_frac": frac(fl, ms_pre, tc_peak, 1e12),
                                  "hbm_frac": frac(b_pre, ms_pre, hbm_peak, 1e9)},
                      "verify": {"ms": round(ms_ver, 4), "tokens": sum(ks),
                                 "hbm_frac": frac(b_ver, ms_ver, hbm_peak, 1e9)},
                      "sum_ms": round(ms_pre + ms_ver, 4)}}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_baseline_decode(n_seq=N_SEQ, tokens=4, seconds=10.0):
    """The fp64 oracle on this host's cores: n_seq sequences x `tokens` decode tokens of
    the headline workload (one oracle call per sequence, sequences on OpenMP threads),
    repeated from the same states until `seconds` have passed; then a quarter of the
    sequences the same way on one thread for half as long."""
    import oracle
    from gated_deltanet_layer_conv1d_gb300 import workloads as wl
    oracle.build()
    w = wl.batched_decode(n=n_seq, steps=tokens, seed=0)
    steps = [w.tokens] + w.steps
    seqs = []
    for i in range(n_seq):
        tok = {k: np.stack([s[k][i] for s in steps]) for k in ("qkv", "z", "a", "b")}
        seqs.append(dict(tok, conv_state=w.conv0[i], H=w.H0[i]))
    s = w.shape
    dims = oracle.Dims(s.n_k_heads, s.n_v_heads, s.d_k, s.d_v, s.d_conv,
                       float(np.float32(s.q_scale)), float(np.float32(s.l2_eps)),
                       float(np.float32(s.norm_eps)))
    cores = oracle.max_threads()

    def run(batch, budget):
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle.mixer_batch(dims, w.weights, batch)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= budget:
                return reps, dt

    reps, dt = run(seqs, seconds)
    n1 = max(1, n_seq // 4)
    oracle.set_threads(1)
    reps1, dt1 = run(seqs[:n1], seconds / 2)
    oracle.set_threads(cores)
    return {"value": round(reps * n_seq * tokens / dt, 2), "unit": "tokens/s", "cores": cores,
            "kind": "oracle", "cpu_model": cpu_model(),
            "single_thread_value": round(reps1 * n1 * tokens / dt1, 2),
            "sample": f"{n_seq} sequences x {tokens} decode tokens of the 128-sequence "
                      f"workload, {reps} times ({dt:.1f} s on {cores} threads); {n1} of them "
                      f"{reps1} times on one thread ({dt1:.1f} s); fp64"}


def cpu_baseline_prefill(tokens=8192, seconds=10.0):
    """The fp64 oracle's token loop over the first `tokens` tokens of the 8192-token
    prefill workload (one sequence, so one thread), repeated until `seconds` have passed."""
    import oracle
    from gated_deltanet_layer_conv1d_gb300 import workloads as wl
    oracle.build()
    w = wl.long_prefill(8192)
    s = w.shape
    dims = oracle.Dims(s.n_k_heads, s.n_v_heads, s.d_k, s.d_v, s.d_conv,
                       float(np.float32(s.q_scale)), float(np.float32(s.l2_eps)),
                       float(np.float32(s.norm_eps)))
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.mixer(dims, w.weights, *(w.tokens[k][:tokens] for k in ("qkv", "z", "a", "b")),
                     w.conv0[0], w.H0[0])
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    return {"value": round(reps * tokens / dt, 2), "unit": "tokens/s", "cores": 1,
            "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{tokens} of the 8192 tokens, {reps} times (fp64 token loop, "
                      f"{dt:.1f} s)"}


def run_reference(args):
    """The fp64 oracle as it stands, on this host's cores: each step is a bounded sample of
    the headline workload (REF_SAMPLE sequences x 1 decode token, sequences on OpenMP
    threads); tokens/s is per token, so it compares with the GPU arm's value."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from gated_deltanet_layer_conv1d_gb300 import workloads as wl
    oracle.build()
    w = wl.batched_decode(n=N_SEQ, steps=1, seed=0)
    seqs = [dict(qkv=w.tokens["qkv"][i:i + 1], z=w.tokens["z"][i:i + 1],
                 a=w.tokens["a"][i:i + 1], b=w.tokens["b"][i:i + 1], conv_state=w.conv0[i],
                 H=w.H0[i]) for i in range(REF_SAMPLE)]
    s = w.shape
    dims = oracle.Dims(s.n_k_heads, s.n_v_heads, s.d_k, s.d_v, s.d_conv,
                       float(np.float32(s.q_scale)), float(np.float32(s.l2_eps)),
                       float(np.float32(s.norm_eps)))
    for _ in range(args.warmup):
        oracle.mixer_batch(dims, w.weights, seqs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.mixer_batch(dims, w.weights, seqs)
    dt = time.perf_counter() - t0
    v = REF_SAMPLE * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * dt / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy PCG64)",
            "config": {"workload": "batched_decode_128seq_1tok_Hk16_Hv32_d128",
                       "global_batch": N_SEQ, "seq_len": 1, "parallelism": "single"},
            "cpu_baseline": {"value": round(v, 2), "unit": "tokens/s",
                             "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"each step: {REF_SAMPLE} of the 128 sequences x 1 "
                                       f"decode token"},
            "e2e": {"value": round(v, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def mode_summary(modes: dict) -> dict:
    """{mode: [ms per step, throughput, roofline fraction]} for every mode that ran (the
    projections and the layer steps by call)."""
    out = {}
    for name, m in modes.items():
        if "ms_per_step" in m:
            rf = m.get("roofline", {})
            frac = rf.get("frac") if "frac" in rf else rf.get("tensor", {}).get("frac")
            out[name] = [m["ms_per_step"], m.get("value"), frac]
        for part, pm in m.get("parts", {}).items():
            if isinstance(pm, dict) and "ms" in pm:
                tok = pm.get("tokens")
                out[f"{name}.{part}"] = [pm["ms"], round(tok / pm["ms"] * 1e3, 1) if tok else None,
                                         pm.get("tensor_frac", pm.get("hbm_frac"))]
        for sub in ("calls", "steps"):
            for cname, c in m.get(sub, {}).items():
                ms = c.get("ms", c.get("ms_per_step"))
                out[cname] = [ms, c.get("value"), c.get("roofline", {}).get("frac")]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--no-modes", action="store_true", help="skip the verify / prefill lines")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--profile", nargs="?", const="decode", default=None,
                    choices=["decode", "verify", "verify-small", "verify16", "verify16-small",
                             "prefill", "mixed", "proj", "proj128", "layer", "fold", "decode16",
                             "woa"],
                    help="only one timed loop of one mode (for profiler captures); "
                         "verify-small runs 32 sequences; verify16 runs on fp16 state pools")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    from gated_deltanet_layer_conv1d_gb300 import gdn
    gdn.lib()

    hbm_peak, tc_peak, peak_src = peaks()
    if args.profile == "proj128":
        proj128_profile(device, args.steps, warmup=args.warmup)
        if rank == 0:
            print(json.dumps({"profile_run": "proj128"}))
        return
    if args.profile == "proj":
        r = proj_mode(device, args.steps, tc_peak, hbm_peak, warmup=args.warmup)
        if rank == 0:
            print(json.dumps({"profile_run": "proj", "calls": r["calls"]}))
        return
    if args.profile in ("fold", "decode16", "woa"):
        if args.profile == "fold":
            r = fold_mode(device, args.steps, hbm_peak, warmup=args.warmup)
        elif args.profile == "woa":
            r = woa_mode(device, args.steps, hbm_peak, warmup=args.warmup)
        else:
            r = decode_h16_mode(device, args.steps, hbm_peak, warmup=args.warmup)
        if rank == 0:
            print(json.dumps({"profile_run": args.profile, "ms_per_step": r["ms_per_step"]}))
        return
    if args.profile == "layer":
        r = layer_mode(device, args.steps, warmup=args.warmup)
        if rank == 0:
            print(json.dumps({"profile_run": "layer", "steps": r["steps"]}))
        return
    if args.profile in ("verify", "verify-small", "verify16", "verify16-small", "prefill",
                        "mixed"):
        if args.profile == "prefill":
            r = prefill_mode(device, args.steps, tc_peak, warmup=args.warmup)
        elif args.profile == "mixed":
            r = mixed_mode(device, args.steps, hbm_peak, tc_peak)
        else:
            r = verify_mode(device, args.steps, hbm_peak, warmup=args.warmup,
                            n=32 if args.profile.endswith("-small") else N_SEQ,
                            h16=args.profile.startswith("verify16"))
        if rank == 0:
            out = {"profile_run": args.profile, "ms_per_step": r["ms_per_step"]}
            if "parts" in r:
                out["parts"] = r["parts"]
            print(json.dumps(out))
        return
    bench = DecodeBench(device)
    for i in range(args.warmup):
        bench.step(i)
    torch.cuda.synchronize()
    bench.check_status()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(bench.stream)
    for i in range(args.steps):
        bench.step(i)
    e1.record(bench.stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms_total = e0.elapsed_time(e1)
    if args.profile:
        sampler.stop()
        bench.check_status()
        if rank == 0:
            print(json.dumps({"profile_run": True, "ms_per_step": ms_total / args.steps}))
        return
    # keep the same work running until the clock record spans at least 1.5 s
    soak_t0 = time.perf_counter()
    i = 0
    while time.perf_counter() - soak_t0 < max(0.0, 1.5 - ms_total / 1e3):
        bench.step(i)
        i += 1
        if i % 200 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    sampler.stop()
    bench.check_status()

    ms_total = slowest_rank(ms_total, device)
    ms_step = ms_total / args.steps
    value = replica_throughput(N_SEQ * args.steps, world, ms_total)
    step_bytes = N_SEQ * DECODE_BYTES_PER_TOKEN + WEIGHT_BYTES
    achieved = step_bytes / (ms_step * 1e-3) / 1e9  # one kernel launch per step
    e2e_ms, h2d, d2h = bench.e2e(max(20, args.steps // 4), 5)
    e2e_ms = slowest_rank(e2e_ms, device)
    e2e = {"value": round(replica_throughput(N_SEQ, world, e2e_ms), 1), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(e2e_ms, 4)}

    modes = {}
    if not args.no_modes and rank == 0:
        modes["ragged_verify"] = verify_mode(device, max(10, min(200, args.steps // 10)), hbm_peak)
        modes["accepted_fold"] = fold_mode(device, 50, hbm_peak)
        modes["speculative_step_write_on_accept"] = woa_mode(device, 50, hbm_peak)
        modes["decode_fp16_state"] = decode_h16_mode(device, 200, hbm_peak)
        modes["ragged_verify_fp16_state"] = verify_mode(device, max(10, min(200, args.steps // 10)),
                                                        hbm_peak, h16=True)
        modes["chunked_prefill"] = prefill_mode(device, 5, tc_peak)
        modes["prefill_f32_option"] = prefill_mode(device, 3, tc_peak, f32=True)
        if world == 1 and not args.no_cpu:
            modes["chunked_prefill"]["cpu_baseline"] = cpu_baseline_prefill()
        modes["mixed_serving"] = mixed_mode(device, 3, hbm_peak, tc_peak)
        modes["projections"] = proj_mode(device, 20, tc_peak, hbm_peak)
        modes["layer"] = layer_mode(device, 100)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline_decode()
    if world > 1:
        dist.barrier()
    if rank == 0:
        traffic = ncu_traffic()
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded numpy PCG64; bf16 activations, f32 state)",
            "config": {"workload": "batched_decode_128seq_1tok_Hk16_Hv32_d128",
                       "global_batch": N_SEQ * world, "seq_len": 1,
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": f"inputs larger than L2: {POOLS} rotating 256 MiB state pools"},
            "gpu_launches": args.steps,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                         "traffic": traffic, "peak_source": peak_src,
                         "algorithmic_bytes": step_bytes, "kernel": "gdn_recurrent_kernel"},
            "clocks": sampler.summary(),
            "e2e": e2e,
            "cpu_baseline": cpu,
            "modes": modes,
        }
        # One compact line per mode at the very end, so that the last few hundred bytes of the
        # output carry every mode's time, throughput and roofline fraction.
        line["summary"] = mode_summary(modes)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
