#!/usr/bin/env python
"""Benchmark of the fused decode GEMV path on GB300.

One step = one pass over every operation of the hot path at full size, each through
the C ABI (weights resident in HBM, ~357 MB per step, more than the 129 MB L2, so
every launch streams its weights from HBM):

  f16 4096x4096  residual add in place through a [32,128] view      (1 launch)
  f16 4096x4096  sigmoid tail                                        (1)
  Q8_0 11008x4096  silu(y) * m                                      (1)
  Q4_0 decode-layer chain, d_model 4096, ffn 14336: q, k, v, o+add,
       up, gate silu*up, down+add, beta sigmoid (M=32): q, k, v and beta
       sharing x in one gemv_multi, o+add, gate and up in one gemv_glu,
       down+add                                                         (4)
  signed FWHT(1024) prologue + f16 5120x5120 + add in place, 1 column (1)
  the same with a batch of 8 columns                                 (1)

value = algorithmic bytes of the step (W + x + aux + dst, each once) / step time, GB/s,
with the step captured in a CUDA graph (launches chained with programmatic dependent
launch) and replayed.  Also reported: per-kernel CUDA-event durations and the roofline
of the dominant kernel, microseconds per decode layer (the step's 4 launches, the 8
fused launches, the 13 unfused ones), the epilogue cost against the tail-free GEMV, an end-to-end number through host buffers,
SM clocks during the timed region, and the fp64 CPU oracle timed on the host cores.
Under "next_rows": the layer chain with the gated dual GEMV (7 launches), the same
layer in Q4_K, the dual GEMV against its two separate launches, split K on and off for
GEMVs with few rows, and the cost of the RMS-normalisation prologue.

Launch: python bench.py [--gpus N --steps K --warmup W] [--impl reference]
(N > 1 under torch.distributed.run; every rank runs the same step on its own GPU.)
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused GEMV HBM GB/s & % of GB300 peak; µs per decode layer chain"
UNIT = "GB/s"
WORKLOAD = ("decode_step: f16 4096x4096 add-in-place via [32,128] view + sigmoid; "
            "Q8_0 11008x4096 silu*m; Q4_0 decode-layer chain (d_model 4096, ffn 14336, 8 GEMVs in 4 "
            "launches: multi q/k/v/beta, o+add, glu gate*up, down+add); "
            "signed FWHT(1024) + f16 5120x5120 add-in-place, ncols 1 and 8")
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------------------- workload spec

def step_spec():
    """(name, wtype, M, K, epilogue, ncols, fwht) for every launch of one step, in order."""
    F16, Q8, Q4 = 1, 2, 3
    NONE, SIG, SILU_MUL, ADD = 0, 1, 3, 4
    d, f = 4096, 14336
    return [
        ("f16_add_view", F16, 4096, 4096, ADD, 1, False),
        ("f16_sigmoid", F16, 4096, 4096, SIG, 1, False),
        ("q8_0_silu_mul", Q8, 11008, 4096, SILU_MUL, 1, False),
        ("chain_q", Q4, d, d, NONE, 1, False),
        ("chain_k", Q4, d, d, NONE, 1, False),
        ("chain_v", Q4, d, d, NONE, 1, False),
        ("chain_o_add", Q4, d, d, ADD, 1, False),
        ("chain_up", Q4, f, d, NONE, 1, False),
        ("chain_gate_silu_mul", Q4, f, d, SILU_MUL, 1, False),
        ("chain_down_add", Q4, d, f, ADD, 1, False),
        ("chain_beta_sigmoid", Q4, 32, d, SIG, 1, False),
        ("fwht_f16_add_n1", F16, 5120, 5120, ADD, 1, True),
        ("fwht_f16_add_n8", F16, 5120, 5120, ADD, 8, True),
    ]


def row_bytes(wt, K):
    return {0: 4 * K, 1: 2 * K, 2: (K // 32) * 34, 3: (K // 32) * 18}[wt]


def algo_bytes(wt, M, K, epi, ncols, fwht):
    """W once + x once + aux once (read) + dst once (write)."""
    b = M * row_bytes(wt, K) + ncols * K * 4 + ncols * M * 4
    if epi in (3, 4):
        b += ncols * M * 4
    if fwht:
        b += 1024 * 4
    return b


WT_NAME = {0: "f32", 1: "f16", 2: "q8_0", 3: "q4_0"}
CHAIN_NAMES = ["chain_q", "chain_k", "chain_v", "chain_o_add", "chain_up", "chain_gate_silu_mul",
               "chain_down_add", "chain_beta_sigmoid"]
# The step runs the layer's eight GEMVs as four launches: q, k, v and the sigmoid head
# sharing x (gemv_multi), o + residual add, gate and up in one pass with silu(gate) * up
# (gemv_glu), down + residual add.  Measured on GB300 (us per layer, two weight sets
# alternating): 42.1 for these four and 53.3 for the eight calls as separate launches.
LAYER_UNITS = {
    "layer_qkv_beta": ["chain_q", "chain_k", "chain_v", "chain_beta_sigmoid"],
    "layer_o_add": ["chain_o_add"],
    "layer_gate_up": ["chain_gate_silu_mul", "chain_up"],
    "layer_down_add": ["chain_down_add"],
}
LAYER_KEYS = {"layer_qkv_beta": "gemv_stream_kernel<q4_0,1,ext>", "layer_o_add": "gemv_stream_kernel<q4_0,1>",
              "layer_gate_up": "gemv_stream_kernel<q4_0,1,ext>", "layer_down_add": "gemv_stream_kernel<q4_0,1>"}


# ----------------------------------------------------------------------------- GPU arm

class Step:
    """Device buffers and the list of ABI calls of one step."""

    def __init__(self, G, torch, seed0=0, layer_seed=100):
        from decode_gemv_epilogue_gb300 import synth
        self.G, self.torch = G, torch
        dev = torch.device("cuda")
        up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        spec = step_spec()
        self.spec = spec
        self.W = {}
        for i, (name, wt, M, K, epi, nc, fw) in enumerate(spec):
            seed = (layer_seed + i) if name.startswith("chain_") else (seed0 + 10 * i)
            self.W[name] = up(synth.weights(wt, M, K, seed=seed))
        self.x4096 = up(synth.normal(4096, seed=seed0 + 1))
        self.r4096 = up(synth.normal(4096, seed=seed0 + 2))
        self.xsig = up(synth.normal(4096, seed=seed0 + 3))
        self.xq8 = up(synth.normal(4096, seed=seed0 + 4))
        self.m = up(synth.normal(11008, seed=seed0 + 5))
        self.gate_out = torch.empty(11008, device=dev)
        self.sig_out = torch.empty(4096, device=dev)
        # chain
        self.cx = up(synth.normal(4096, seed=seed0 + 6))
        self.ca = up(synth.normal(4096, seed=seed0 + 7))
        # the layer's residual: the o-proj add reads r0 (N(0,1), as the workload draws it) and
        # writes r, which gate/up read and down adds to in place; so every step starts from
        # the same distribution instead of feeding its output back (which would grow
        # without bound and end in Inf/NaN after a few steps)
        self.cr0 = up(synth.normal(4096, seed=seed0 + 8))
        self.cr = self.cr0.clone()
        self.cq, self.ck, self.cv = (torch.empty(4096, device=dev) for _ in range(3))
        self.cup = torch.empty(14336, device=dev)
        self.cg = torch.empty(14336, device=dev)
        self.cbeta = torch.empty(32, device=dev)
        # FWHT + f16 5120
        self.signs = up(synth.rademacher(1024, seed=seed0 + 9))
        self.fx1 = up(synth.normal(5120, seed=seed0 + 10))
        self.fr1 = up(synth.normal(5120, seed=seed0 + 11))
        self.fx8 = up(synth.normal(8 * 5120, seed=seed0 + 12))
        self.fr8 = up(synth.normal(8 * 5120, seed=seed0 + 13))
        # transform-once prologue: x' of each batch goes to a caller workspace
        self.ws1 = torch.empty(5120, device=dev)
        self.ws8 = torch.empty(8 * 5120, device=dev)
        self.bytes = {n: algo_bytes(wt, M, K, e, nc, fw) for (n, wt, M, K, e, nc, fw) in spec}
        self.step_bytes = sum(self.bytes.values())
        self.keys = {}
        for (n, wt, M, K, e, nc, fw) in spec:
            x_any = self.fx8 if nc > 1 else (self.fx1 if K == 5120 else self.cg if K == 14336 else self.cx)
            aux_any = self.fr8 if nc > 1 else self.gate_out
            ws = (self.ws8 if nc > 1 else self.ws1) if fw else None
            path, _ = G.plan(self.W[n], wt, x_any, M, K, e, aux_any, aux_any, ncols=nc,
                             fwht_signs=self.signs if fw else None, fwht_block=1024 if fw else 0, fwht_workspace=ws)
            if path < 0:
                raise RuntimeError("plan failed for %s: %s" % (n, G.status_string(path)))
            kind = {G.PATH_STREAM: "gemv_stream_kernel", G.PATH_TC: "gemv_tc_kernel"}.get(path, "gemv_generic_kernel")
            self.keys[n] = ("fwht_signed_kernel+" if fw else "") + "%s<%s,%d>" % (kind, WT_NAME[wt], nc)
        # the step's launch units: every call on its own, except the layer's eight GEMVs,
        # which run as four launches (LAYER_UNITS)
        self.unit_names = [n for (n, *_r) in spec if n not in CHAIN_NAMES]
        self.unit_names[3:3] = list(LAYER_UNITS)
        wb = lambda n: self.W[n].numel()
        d, f = 4096, 14336
        self.bytes["layer_qkv_beta"] = sum(wb(n) for n in LAYER_UNITS["layer_qkv_beta"]) + 4 * d + 4 * (3 * d + 32)
        self.bytes["layer_o_add"] = wb("chain_o_add") + 4 * d + 2 * 4 * d
        self.bytes["layer_gate_up"] = wb("chain_gate_silu_mul") + wb("chain_up") + 4 * d + 4 * f
        self.bytes["layer_down_add"] = wb("chain_down_add") + 4 * f + 2 * 4 * d
        self.keys.update(LAYER_KEYS)
        self.step_bytes = sum(self.bytes[n] for n in self.unit_names)
        # kernels launched per step (a prologue call launches the transform, then the GEMV)
        self.kernels_per_step = (sum(2 if fw else 1 for (n, wt, M, K, e, nc, fw) in spec if n not in CHAIN_NAMES)
                                 + len(LAYER_UNITS))

    def call_specs(self):
        """(name, arguments, keyword arguments) of the step's gemv_fused_ex calls, on the
        buffers the step holds now."""
        W = self.W
        return [
            ("f16_add_view", (W["f16_add_view"], 1, self.x4096, 4096, 4096, 4, self.r4096, self.r4096),
             {"view": (32, 128)}),
            ("f16_sigmoid", (W["f16_sigmoid"], 1, self.xsig, 4096, 4096, 1, None, self.sig_out), {}),
            ("q8_0_silu_mul", (W["q8_0_silu_mul"], 2, self.xq8, 11008, 4096, 3, self.m, self.gate_out), {}),
            ("chain_q", (W["chain_q"], 3, self.cx, 4096, 4096, 0, None, self.cq), {}),
            ("chain_k", (W["chain_k"], 3, self.cx, 4096, 4096, 0, None, self.ck), {}),
            ("chain_v", (W["chain_v"], 3, self.cx, 4096, 4096, 0, None, self.cv), {}),
            ("chain_o_add", (W["chain_o_add"], 3, self.ca, 4096, 4096, 4, self.cr0, self.cr), {}),
            ("chain_up", (W["chain_up"], 3, self.cr, 14336, 4096, 0, None, self.cup), {}),
            ("chain_gate_silu_mul", (W["chain_gate_silu_mul"], 3, self.cr, 14336, 4096, 3, self.cup, self.cg), {}),
            ("chain_down_add", (W["chain_down_add"], 3, self.cg, 4096, 14336, 4, self.cr, self.cr), {}),
            ("chain_beta_sigmoid", (W["chain_beta_sigmoid"], 3, self.cx, 32, 4096, 1, None, self.cbeta), {}),
            ("fwht_f16_add_n1", (W["fwht_f16_add_n1"], 1, self.fx1, 5120, 5120, 4, self.fr1, self.fr1),
             {"fwht_signs": self.signs, "fwht_block": 1024, "fwht_workspace": self.ws1}),
            ("fwht_f16_add_n8", (W["fwht_f16_add_n8"], 1, self.fx8, 5120, 5120, 4, self.fr8, self.fr8),
             {"ncols": 8, "fwht_signs": self.signs, "fwht_block": 1024, "fwht_workspace": self.ws8}),
        ]

    def calls(self, pdl=True, stream=None):
        G = self.G
        return [(name, (lambda a=a, kw=kw: G.gemv_fused_ex(*a, pdl=pdl, stream=stream, **kw)))
                for (name, a, kw) in self.call_specs()]

    def layer_call(self, unit, Wl, prepare=False, pdl=True):
        """One of the layer's four launches on weight set Wl: issued now, or (prepare) planned
        once and returned (gf_prepare*)."""
        G, d, f = self.G, 4096, 14336
        if unit == "layer_qkv_beta":
            items = [(Wl["chain_q"], d, 0, None, self.cq), (Wl["chain_k"], d, 0, None, self.ck),
                     (Wl["chain_v"], d, 0, None, self.cv), (Wl["chain_beta_sigmoid"], 32, 1, None, self.cbeta)]
            return (G.prepare_multi if prepare else G.gemv_multi)(items, 3, self.cx, d, pdl=pdl)
        if unit == "layer_gate_up":
            fn = G.prepare_glu if prepare else G.gemv_glu
            return fn(Wl["chain_gate_silu_mul"], Wl["chain_up"], 3, self.cr, f, d, self.cg, pdl=pdl, split_k=False)
        fn = G.prepare if prepare else G.gemv_fused_ex
        if unit == "layer_o_add":
            return fn(Wl["chain_o_add"], 3, self.ca, d, d, 4, self.cr0, self.cr, pdl=pdl, split_k=False)
        return fn(Wl["chain_down_add"], 3, self.cg, d, f, 4, self.cr, self.cr, pdl=pdl, split_k=False)

    def prepared(self, pdl=True):
        """The step's launch units planned once (gf_prepare*), in order."""
        G = self.G
        one = {name: G.prepare(*a, pdl=pdl, **kw) for (name, a, kw) in self.call_specs() if name not in CHAIN_NAMES}
        for u in LAYER_UNITS:
            one[u] = self.layer_call(u, self.W, prepare=True, pdl=pdl)
        return [(n, one[n]) for n in self.unit_names]

    def unit_calls(self, pdl=True):
        """(name, fn) per launch unit: fn issues it on the current stream."""
        G = self.G
        return [(n, (lambda h=h: G.launch_prepared([h]))) for n, h in self.prepared(pdl)]

    # the end-to-end leg: every per-step activation in one device arena laid out as
    # [results only | residuals (read and written in place) | inputs only], mirrored by a
    # pinned host buffer, so a step is one host->device copy of the residuals and inputs
    # and one device->host copy of the results and residuals
    def pack_for_e2e(self):
        torch = self.torch
        res_only = ["sig_out", "gate_out", "cq", "ck", "cv", "cbeta"]
        inplace = ["r4096", "cr", "fr1", "fr8"]
        inputs = ["x4096", "xsig", "xq8", "m", "cx", "ca", "cr0", "fx1", "fx8"]
        names = res_only + inplace + inputs
        sizes = [getattr(self, n).numel() for n in names]
        total = sum(sizes)
        arena = torch.empty(total, device="cuda")
        host = torch.empty(total, dtype=torch.float32, pin_memory=True)
        off = 0
        spans = {}
        for n, k in zip(names, sizes):
            view = arena[off:off + k]
            view.copy_(getattr(self, n))
            host[off:off + k].copy_(view.cpu())
            setattr(self, n, view)
            spans[n] = (off, off + k)
            off += k
        in_lo = spans[inplace[0]][0]            # residuals + inputs: host -> device
        out_hi = spans[inplace[-1]][1]          # results + residuals: device -> host
        return arena, host, (in_lo, total), (0, out_hi)


def max_over_ranks(ms, dist=None, device=None):
    """The timed region's length as the slowest rank saw it (all ranks get the max)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world, step_bytes, ms_per_step):
    """Replicas: every rank runs the whole step, so the job moves world * step_bytes."""
    return world * step_bytes / (ms_per_step * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [t.strip() for t in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash():
    """Hash of the library's sources with comments and blank lines left out (a change to a
    comment leaves the kernels, and so their counters, as they were)."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_gemv_epilogue_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, fn)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = [re.sub(r"//.*$", "", l).rstrip() for l in text.splitlines()]
        h.update(fn.encode())
        h.update("\n".join(l for l in lines if l.strip()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """dram read+write bytes per launch from the committed ncu summary, if it still
    matches the kernel source (profiles/traffic.txt: key, bytes, source hash)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel_key and parts[2] == src:
                return float(parts[1])
    return None


def gpu_arm(args, rank, world, local_rank):
    import torch
    import __graft_entry__ as ge
    ge.build()
    from decode_gemv_epilogue_gb300 import gemvfuse as G

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if dist is not None:
            dist.barrier()

    step = Step(G, torch)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    calls = step.unit_calls(pdl=True)
    sampler = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)

    with torch.cuda.stream(s):
        for _ in range(max(args.warmup, 3)):
            for _, fn in calls:
                fn()
    s.synchronize()
    assert G.device_status(reset=True) == 0
    # capture one step in a CUDA graph (launches chained with programmatic dependencies)
    graph = torch.cuda.CUDAGraph()
    mode = "cuda_graph+pdl"
    try:
        with torch.cuda.graph(graph, stream=s):
            for _, fn in calls:
                fn()
        graph.replay()
        s.synchronize()
    except Exception as e:  # report and fall back to eager launches
        graph = None
        mode = "eager+pdl (graph capture failed: %s)" % str(e).splitlines()[0][:120]

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            for _, fn in calls:
                fn()

    sampler.start()
    with torch.cuda.stream(s):
        soak_end = time.time() + 1.0
        while time.time() < soak_end:
            for _ in range(50):
                run_step()
            s.synchronize()
    # ---------------------------------------------------------------- timed region
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    G.repair_count(reset=True)  # (synchronises) counted over the timed steps only
    barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        ev0.record(s)
        for _ in range(args.steps):
            run_step()
        ev1.record(s)
    s.synchronize()
    torch.cuda.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    sampler.stop()
    ms = max_over_ranks(ms, dist, torch.device("cuda"))
    ms_per_step = ms / args.steps
    value = whole_job_gbs(world, step.step_bytes, ms_per_step)

    # row chunks the integer-path kernels handed to their fp32 repair during the timed steps
    # (0 for the workload's inputs: a repair reads the chunk's weights twice)
    step_repairs = G.repair_count(reset=True)
    # ---------------------------------------------------------------- per-kernel durations
    per_call = launch_durations(G, torch, step, s, args)
    nl = len(calls)
    per_kernel = {}
    for name, ms_i in per_call.items():
        key = step.keys[name]
        d = per_kernel.setdefault(key, {"launches_per_step": 0, "ms_per_step": 0.0, "bytes_per_step": 0})
        d["launches_per_step"] += 1
        d["ms_per_step"] += ms_i
        d["bytes_per_step"] += step.bytes[name]
    total_k = sum(d["ms_per_step"] for d in per_kernel.values())
    for d in per_kernel.values():
        d["share"] = round(d["ms_per_step"] / total_k, 4)
        d["gbs"] = round(d["bytes_per_step"] / (d["ms_per_step"] * 1e-3) / 1e9, 1)
    dom = max(per_kernel, key=lambda k: per_kernel[k]["ms_per_step"])
    peak, peak_kind = measured_peaks()
    dk = per_kernel[dom]
    achieved = dk["gbs"]
    traffic = ncu_traffic(dom)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else
                "fallback 6.8 TB/s", "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": traffic,
                "algorithmic_bytes_per_launch": round(dk["bytes_per_step"] / dk["launches_per_step"]),
                "launch_us": round(1e3 * dk["ms_per_step"] / dk["launches_per_step"], 3),
                "timing": "CUDA events around a CUDA graph of back-to-back PDL launches of each launch type "
                          "over rotating weight copies (> 2x L2 where the weights allow); per-launch mean"}
    per_workload = {n: {"us": round(1e3 * per_call[n], 3), "bytes": step.bytes[n],
                        "gbs": round(step.bytes[n] / (per_call[n] * 1e-3) / 1e9, 1),
                        "frac_of_peak": round(step.bytes[n] / (per_call[n] * 1e-3) / 1e9 / peak, 4)}
                    for n in per_call}
    # the FWHT + f16 5120x5120 call at every batch width 1..8
    per_workload["fwht_f16_add_ncols_1_to_8"] = fwht_ncols_measure(G, torch, step, s, args, peak)

    # ---------------------------------------------------------------- decode-layer chain
    chain = chain_measure(G, torch, step, s, args)
    # ---------------------------------------------------------------- epilogue cost
    epi_cost = epilogue_cost(G, torch, s)
    # ---------------------------------------------------------------- rows beyond the step
    nxt = next_rows_measure(G, torch, step, s, args, peak)
    # ---------------------------------------------------------------- end to end (host buffers)
    e2e = e2e_measure(G, torch, step, s, args)
    assert G.device_status() == 0, "a kernel reported a bounded-wait timeout"

    launches = step.kernels_per_step * args.steps
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; weight distributions of the workload; weights resident in HBM)",
        "config": {"workload": WORKLOAD, "model": None, "bytes_per_step": step.step_bytes,
                   "l2": "inputs larger than L2: %.0f MB of weights per step vs 129 MB L2; each launch "
                         "reads a distinct weight buffer" % (step.step_bytes / 1e6),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "launch_mode": mode, "abi_calls_per_step": nl, "kernel_launches_per_step": step.kernels_per_step,
                   "prologue": "signed FWHT once per call into a caller workspace (fwht_signed_kernel), "
                               "then the GEMV, PDL-chained",
                   "soak_s_before_timing": 1.0},
        "roofline": roofline,
        "pct_of_peak": round(100 * value / world / peak, 2),
        "gpu_launches": launches,
        "us_per_layer": chain["step_form_us"], "launches_per_layer": len(LAYER_UNITS),
        "us_per_layer_8_launches": chain["fused_us"],
        "us_per_layer_unfused": chain["unfused_us"], "launches_per_layer_unfused": 13,
        "chain": chain, "epilogue_cost": epi_cost, "per_kernel": per_kernel, "per_workload": per_workload,
        "next_rows": nxt, "repairs_in_timed_steps": step_repairs,
        "e2e": e2e, "clocks": sampler.summary(),
    }
    if dist is not None:
        dist.destroy_process_group()
    return out


def launch_durations(G, torch, step, s, args):
    """Per-launch device time of every launch of the step: for each launch, a CUDA graph
    of back-to-back launches (chained with programmatic dependent launch, as in the step)
    cycling through copies of its weights -- enough copies to exceed 2x L2 when the
    weights allow, at most 32 -- timed with CUDA events on the launch stream."""
    out = {}
    specs = {n: (a, kw) for (n, a, kw) in step.call_specs()}
    for name in step.unit_names:
        mats = LAYER_UNITS.get(name, [name])
        nbytes = sum(step.W[n].numel() for n in mats)
        ncopy = int(min(32, max(2, -(-2 * L2_BYTES // nbytes))))
        W0 = {n: step.W[n] for n in mats}
        copies = [W0] + [{n: W0[n].clone() for n in mats} for _ in range(ncopy - 1)]
        if name in LAYER_UNITS:
            fn = lambda Wl, name=name: step.layer_call(name, Wl)
        else:
            a, kw = specs[name]
            fn = lambda Wl, name=name, a=a, kw=kw: G.gemv_fused_ex(Wl[name], *a[1:], pdl=True, **kw)

        def run_all():
            for Wc in copies:
                fn(Wc)

        with torch.cuda.stream(s):
            run_all()
        s.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            run_all()
        reps = max(3, min(20, args.steps // 20))
        with torch.cuda.stream(s):
            gr.replay()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(reps):
                gr.replay()
            e1.record(s)
        s.synchronize()
        out[name] = e0.elapsed_time(e1) / (reps * ncopy)
        del gr, copies
    return out


def fwht_ncols_measure(G, torch, step, s, args, peak):
    """The signed-FWHT(1024) + f16 5120x5120 + in-place residual call for every batch width
    1..8 (the workload's ncols = 1..8), as the step issues it (transform once into the
    workspace, then the GEMV, PDL-chained): per width the mean device time over a CUDA graph
    of back-to-back calls cycling through weight copies (> 2x L2), the algorithmic bytes,
    GB/s and the fraction of the measured HBM peak."""
    M = K = 5120
    W0 = step.W["fwht_f16_add_n8"]
    ncopy = int(min(32, max(2, -(-2 * L2_BYTES // W0.numel()))))
    copies = [W0] + [W0.clone() for _ in range(ncopy - 1)]
    reps = max(3, min(20, args.steps // 20))
    out = {}
    for nc in range(1, 9):
        x, r, ws = step.fx8[:nc * K], step.fr8[:nc * M], step.ws8[:nc * K]

        def run_all(nc=nc, x=x, r=r, ws=ws):
            for Wc in copies:
                G.gemv_fused_ex(Wc, 1, x, M, K, 4, r, r, ncols=nc, fwht_signs=step.signs, fwht_block=1024,
                                fwht_workspace=ws, pdl=True)

        with torch.cuda.stream(s):
            run_all()
        s.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            run_all()
        with torch.cuda.stream(s):
            gr.replay()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(reps):
                gr.replay()
            e1.record(s)
        s.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / (reps * ncopy)
        path, _ = G.plan(W0, 1, x, M, K, 4, r, r, ncols=nc, fwht_signs=step.signs, fwht_block=1024,
                         fwht_workspace=ws)
        b = algo_bytes(1, M, K, 4, nc, True)
        gbs = b / (us * 1e-6) / 1e9
        out["ncols_%d" % nc] = {"us": round(us, 3), "bytes": b, "gbs": round(gbs, 1),
                                "frac_of_peak": round(gbs / peak, 4),
                                "kernel": {G.PATH_STREAM: "gemv_stream_kernel", G.PATH_TC: "gemv_tc_kernel"}.get(
                                    path, "gemv_generic_kernel")}
        del gr
    del copies
    return out


def second_layer(torch, step):
    """A second set of the layer's weights (seeded apart from the step's), so that timed
    layers alternate between two sets and nothing stays in L2."""
    from decode_gemv_epilogue_gb300 import synth
    if not hasattr(step, "_layer2"):
        shapes = {n: (M, K) for (n, wt, M, K, e, nc, fw) in step_spec() if n in CHAIN_NAMES}
        dev = torch.device("cuda")
        step._layer2 = {n: torch.from_numpy(synth.weights(3, shapes[n][0], shapes[n][1], seed=300 + i)).to(dev)
                        for i, n in enumerate(CHAIN_NAMES)}
    return step._layer2


def chain_measure(G, torch, step, s, args):
    """Microseconds per decode layer: the step's four launches, the 8 fused
    launches and the 13-launch unfused chain (separate GEMV, add, silu, mul, sigmoid
    kernels), each captured in a CUDA graph, two layers' weights alternating so nothing
    stays in L2."""
    dev = torch.device("cuda")
    names = ["chain_q", "chain_k", "chain_v", "chain_o_add", "chain_up", "chain_gate_silu_mul",
             "chain_down_add", "chain_beta_sigmoid"]
    layers = [{n: step.W[n] for n in names}, second_layer(torch, step)]
    x, a, r, r0 = step.cx, step.ca, step.cr, step.cr0
    q, k, v, u, g, beta = step.cq, step.ck, step.cv, step.cup, step.cg, step.cbeta
    y4 = torch.empty(4096, device=dev)
    y14 = torch.empty(14336, device=dev)

    def fused(Wl):
        G.gemv_fused_ex(Wl["chain_q"], 3, x, 4096, 4096, 0, None, q, pdl=True)
        G.gemv_fused_ex(Wl["chain_k"], 3, x, 4096, 4096, 0, None, k, pdl=True)
        G.gemv_fused_ex(Wl["chain_v"], 3, x, 4096, 4096, 0, None, v, pdl=True)
        G.gemv_fused_ex(Wl["chain_o_add"], 3, a, 4096, 4096, 4, r0, r, pdl=True)
        G.gemv_fused_ex(Wl["chain_up"], 3, r, 14336, 4096, 0, None, u, pdl=True)
        G.gemv_fused_ex(Wl["chain_gate_silu_mul"], 3, r, 14336, 4096, 3, u, g, pdl=True)
        G.gemv_fused_ex(Wl["chain_down_add"], 3, g, 4096, 14336, 4, r, r, pdl=True)
        G.gemv_fused_ex(Wl["chain_beta_sigmoid"], 3, x, 32, 4096, 1, None, beta, pdl=True)

    def unfused(Wl):
        G.gemv_fused(Wl["chain_q"], 3, x, 4096, 4096, 0, None, q)
        G.gemv_fused(Wl["chain_k"], 3, x, 4096, 4096, 0, None, k)
        G.gemv_fused(Wl["chain_v"], 3, x, 4096, 4096, 0, None, v)
        G.gemv_fused(Wl["chain_o_add"], 3, a, 4096, 4096, 0, None, y4)
        G.elementwise(G.EW_ADD, y4, r0, r, 4096)
        G.gemv_fused(Wl["chain_up"], 3, r, 14336, 4096, 0, None, u)
        G.gemv_fused(Wl["chain_gate_silu_mul"], 3, r, 14336, 4096, 0, None, y14)
        G.elementwise(G.EW_SILU, y14, None, y14, 14336)
        G.elementwise(G.EW_MUL, y14, u, g, 14336)
        G.gemv_fused(Wl["chain_down_add"], 3, g, 4096, 14336, 0, None, y4)
        G.elementwise(G.EW_ADD, y4, r, r, 4096)
        G.gemv_fused(Wl["chain_beta_sigmoid"], 3, x, 32, 4096, 0, None, beta)
        G.elementwise(G.EW_SIGMOID, beta, None, beta, 32)

    res = {}
    reps = max(20, min(args.steps, 500))
    for label, fn in (("fused", fused), ("unfused", unfused)):
        with torch.cuda.stream(s):
            fn(layers[0]); fn(layers[1])
        s.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            fn(layers[0])
            fn(layers[1])
        for _ in range(3):
            gr.replay()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(reps):
                gr.replay()
            e1.record(s)
        s.synchronize()
        res[label + "_us"] = round(1e3 * e0.elapsed_time(e1) / (2 * reps), 3)
    # the step's form: four launches
    res["step_form_us"] = round(graph_us(torch, s, lambda i: [step.layer_call(u, layers[i]) for u in LAYER_UNITS],
                                         2, reps), 3)
    layer_bytes = sum(step.bytes[n] for n in names)
    res["layer_bytes"] = layer_bytes
    res["step_form_bytes"] = sum(step.bytes[u] for u in LAYER_UNITS)
    res["fused_gbs"] = round(layer_bytes / (res["fused_us"] * 1e-6) / 1e9, 1)
    res["step_form_gbs"] = round(res["step_form_bytes"] / (res["step_form_us"] * 1e-6) / 1e9, 1)
    res["layers_timed"] = 2 * reps
    return res


def graph_us(torch, s, issue, nsets, reps):
    """Mean microseconds per weight set of issue(i) for i < nsets, replayed in a CUDA
    graph on stream s (after one warm replay), CUDA events on s."""
    with torch.cuda.stream(s):
        for i in range(nsets):
            issue(i)
    s.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        for i in range(nsets):
            issue(i)
    with torch.cuda.stream(s):
        gr.replay()
    s.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(reps):
            gr.replay()
        e1.record(s)
    s.synchronize()
    del gr
    return 1e3 * e0.elapsed_time(e1) / (reps * nsets)


def next_rows_measure(G, torch, step, s, args, peak):
    """The gated dual GEMV, split K and the RMS-normalisation prologue, each timed as
    graph-replayed PDL launches cycling through enough weight copies to exceed 2x L2."""
    from decode_gemv_epilogue_gb300 import synth
    dev = torch.device("cuda")
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    reps = max(5, min(40, args.steps // 20))
    out = {}

    def copies_for(nbytes):
        return int(min(32, max(2, -(-2 * L2_BYTES // nbytes))))

    # 1. decode-layer chain with gate and up in one launch (7 launches per layer)
    names = ["chain_q", "chain_k", "chain_v", "chain_o_add", "chain_up", "chain_gate_silu_mul",
             "chain_down_add", "chain_beta_sigmoid"]
    shapes = {n: (M, K) for (n, wt, M, K, e, nc, fw) in step_spec() if n in names}
    layers = [{n: step.W[n] for n in names}, second_layer(torch, step)]
    x, a, r, r0 = step.cx, step.ca, step.cr, step.cr0
    q, k, v, g, beta = step.cq, step.ck, step.cv, step.cg, step.cbeta

    def glu_layer(i):
        Wl = layers[i]
        G.gemv_fused_ex(Wl["chain_q"], 3, x, 4096, 4096, 0, None, q, pdl=True)
        G.gemv_fused_ex(Wl["chain_k"], 3, x, 4096, 4096, 0, None, k, pdl=True)
        G.gemv_fused_ex(Wl["chain_v"], 3, x, 4096, 4096, 0, None, v, pdl=True)
        G.gemv_fused_ex(Wl["chain_o_add"], 3, a, 4096, 4096, 4, r0, r, pdl=True)
        G.gemv_glu(Wl["chain_gate_silu_mul"], Wl["chain_up"], 3, r, 14336, 4096, g, pdl=True)
        G.gemv_fused_ex(Wl["chain_down_add"], 3, g, 4096, 14336, 4, r, r, pdl=True)
        G.gemv_fused_ex(Wl["chain_beta_sigmoid"], 3, x, 32, 4096, 1, None, beta, pdl=True)

    us = graph_us(torch, s, glu_layer, 2, max(20, min(args.steps, 500)))
    # bytes: the 8 matrices, x/a/r reads, q/k/v/g/beta writes, r read+write twice
    lb = sum(step.W[n].numel() for n in names) + 4 * (4096 * 3 + 4096 * 3 + 2 * 4096 * 2 + 14336 * 2 + 32)
    out["chain_glu"] = {"us_per_layer": round(us, 3), "launches_per_layer": 7, "layer_bytes": lb,
                        "gbs": round(lb / (us * 1e-6) / 1e9, 1)}

    # 1a. q, k and v stored as one 12288 x 4096 matrix (a layout choice of the caller:
    # one launch reads all three), with the gated dual GEMV: 5 launches per layer
    qkv = [torch.cat([layers[l]["chain_q"], layers[l]["chain_k"], layers[l]["chain_v"]]) for l in range(2)]
    qkv_out = torch.empty(3 * 4096, device=dev)

    def qkv_layer(i):
        Wl = layers[i]
        G.gemv_fused_ex(qkv[i], 3, x, 3 * 4096, 4096, 0, None, qkv_out, pdl=True)
        G.gemv_fused_ex(Wl["chain_o_add"], 3, a, 4096, 4096, 4, r0, r, pdl=True)
        G.gemv_glu(Wl["chain_gate_silu_mul"], Wl["chain_up"], 3, r, 14336, 4096, g, pdl=True)
        G.gemv_fused_ex(Wl["chain_down_add"], 3, g, 4096, 14336, 4, r, r, pdl=True)
        G.gemv_fused_ex(Wl["chain_beta_sigmoid"], 3, x, 32, 4096, 1, None, beta, pdl=True)

    us5 = graph_us(torch, s, qkv_layer, 2, max(20, min(args.steps, 500)))
    out["chain_qkv_glu"] = {"us_per_layer": round(us5, 3), "launches_per_layer": 5, "layer_bytes": lb,
                            "gbs": round(lb / (us5 * 1e-6) / 1e9, 1),
                            "note": "q, k, v weights concatenated into one matrix by the caller"}
    del qkv

    # 1a'. q, k, v and the sigmoid head in one gemv_multi launch (the matrices stay separate
    # buffers), o, the gated dual GEMV and down: 4 launches per layer
    def multi_layer(i):
        Wl = layers[i]
        G.gemv_multi([(Wl["chain_q"], 4096, 0, None, q), (Wl["chain_k"], 4096, 0, None, k),
                      (Wl["chain_v"], 4096, 0, None, v), (Wl["chain_beta_sigmoid"], 32, 1, None, beta)],
                     3, x, 4096, pdl=True)
        G.gemv_fused_ex(Wl["chain_o_add"], 3, a, 4096, 4096, 4, r0, r, pdl=True)
        G.gemv_glu(Wl["chain_gate_silu_mul"], Wl["chain_up"], 3, r, 14336, 4096, g, pdl=True)
        G.gemv_fused_ex(Wl["chain_down_add"], 3, g, 4096, 14336, 4, r, r, pdl=True)

    us4 = graph_us(torch, s, multi_layer, 2, max(20, min(args.steps, 500)))
    out["chain_multi_glu"] = {"us_per_layer": round(us4, 3), "launches_per_layer": 4, "layer_bytes": lb,
                              "gbs": round(lb / (us4 * 1e-6) / 1e9, 1),
                              "note": "q, k, v and the sigmoid head in one gemv_multi launch (separate buffers)"}

    # 1b. the same layer in Q4_K (a format the pages' decode-layer measurements name),
    # 8 launches and 7 with the dual GEMV
    layers_k = [{n: up(synth.weights(4, shapes[n][0], shapes[n][1], seed=700 + 10 * l + i))
                 for i, n in enumerate(names)} for l in range(2)]

    def k_layer(i, glu):
        Wl = layers_k[i]
        G.gemv_fused_ex(Wl["chain_q"], 4, x, 4096, 4096, 0, None, q, pdl=True)
        G.gemv_fused_ex(Wl["chain_k"], 4, x, 4096, 4096, 0, None, k, pdl=True)
        G.gemv_fused_ex(Wl["chain_v"], 4, x, 4096, 4096, 0, None, v, pdl=True)
        G.gemv_fused_ex(Wl["chain_o_add"], 4, a, 4096, 4096, 4, r0, r, pdl=True)
        if glu:
            G.gemv_glu(Wl["chain_gate_silu_mul"], Wl["chain_up"], 4, r, 14336, 4096, g, pdl=True)
        else:
            G.gemv_fused_ex(Wl["chain_up"], 4, r, 14336, 4096, 0, None, step.cup, pdl=True)
            G.gemv_fused_ex(Wl["chain_gate_silu_mul"], 4, r, 14336, 4096, 3, step.cup, g, pdl=True)
        G.gemv_fused_ex(Wl["chain_down_add"], 4, g, 4096, 14336, 4, r, r, pdl=True)
        G.gemv_fused_ex(Wl["chain_beta_sigmoid"], 4, x, 32, 4096, 1, None, beta, pdl=True)

    G.repair_count(reset=True)
    us8 = graph_us(torch, s, lambda i: k_layer(i, False), 2, max(20, min(args.steps, 500)))
    us7 = graph_us(torch, s, lambda i: k_layer(i, True), 2, max(20, min(args.steps, 500)))
    lbk = sum(layers_k[0][n].numel() for n in names) + 4 * (4096 * 3 + 4096 * 3 + 2 * 4096 * 2 + 14336 * 3 + 32)
    out["chain_q4_k_repairs"] = G.repair_count(reset=True)
    out["chain_q4_k"] = {"us_per_layer": round(us8, 3), "launches_per_layer": 8,
                         "us_per_layer_glu": round(us7, 3), "launches_per_layer_glu": 7, "layer_bytes": lbk,
                         "gbs": round(lbk / (us8 * 1e-6) / 1e9, 1)}
    del layers_k

    # 2. the FFN gate/up pair: one dual launch vs up, then gate with the silu*mul tail
    Wg0, Wu0 = step.W["chain_gate_silu_mul"], step.W["chain_up"]
    nset = copies_for(2 * Wg0.numel())
    pairs = [(Wg0, Wu0)] + [(Wg0.clone(), Wu0.clone()) for _ in range(nset - 1)]
    u_tmp = torch.empty(14336, device=dev)
    t_glu = graph_us(torch, s, lambda i: G.gemv_glu(pairs[i][0], pairs[i][1], 3, r, 14336, 4096, g, pdl=True),
                     nset, reps)

    def two(i):
        G.gemv_fused_ex(pairs[i][1], 3, r, 14336, 4096, 0, None, u_tmp, pdl=True)
        G.gemv_fused_ex(pairs[i][0], 3, r, 14336, 4096, 3, u_tmp, g, pdl=True)

    t_two = graph_us(torch, s, two, nset, reps)
    gb = 2 * Wg0.numel() + 4 * (4096 + 14336)
    out["glu_q4_0_14336x4096"] = {"dual_us": round(t_glu, 3), "two_launch_us": round(t_two, 3),
                                  "dual_gbs": round(gb / (t_glu * 1e-6) / 1e9, 1),
                                  "dual_frac_of_peak": round(gb / (t_glu * 1e-6) / 1e9 / peak, 4)}
    del pairs

    # 3. split K for GEMVs with few rows
    for label, wt, M, K, epi in (("q4_0_32x4096_sigmoid", 3, 32, 4096, 1), ("f16_64x14336_none", 1, 64, 14336, 0)):
        base = up(synth.weights(wt, M, K, seed=600))
        nset = copies_for(base.numel())
        Ws = [base] + [base.clone() for _ in range(nset - 1)]
        xv = up(synth.normal(K, seed=601))
        dst = torch.empty(M, device=dev)
        res = {}
        for split in (True, False):
            _, info = G.plan(Ws[0], wt, xv, M, K, epi, None, dst, split_k=split)
            t = graph_us(torch, s, lambda i: G.gemv_fused_ex(Ws[i], wt, xv, M, K, epi, None, dst, pdl=True,
                                                              split_k=split), nset, reps)
            res["split%d_us" % info["split"]] = round(t, 3)
        b = base.numel() + 4 * (K + M)
        res["bytes"] = b
        out["split_k_" + label] = res
        del Ws

    # 4. RMS-normalisation prologue cost against the same GEMV without it
    for label, wt, M, K in (("f16_4096x4096", 1, 4096, 4096), ("q4_0_14336x4096", 3, 14336, 4096)):
        base = up(synth.weights(wt, M, K, seed=610))
        nset = copies_for(base.numel())
        Ws = [base] + [base.clone() for _ in range(nset - 1)]
        xv = up(synth.normal(K, seed=611))
        gam = up(1.0 + 0.1 * synth.normal(K, seed=612))
        dst = torch.empty(M, device=dev)
        t0 = graph_us(torch, s, lambda i: G.gemv_fused_ex(Ws[i], wt, xv, M, K, 0, None, dst, pdl=True), nset, reps)
        t1 = graph_us(torch, s, lambda i: G.gemv_fused_ex(Ws[i], wt, xv, M, K, 0, None, dst, pdl=True,
                                                           rms_norm_weight=gam, rms_norm_eps=1e-6), nset, reps)
        out["rms_norm_" + label] = {"plain_us": round(t0, 3), "with_norm_us": round(t1, 3),
                                    "cost": round(t1 / t0 - 1.0, 4)}
        del Ws
    return out


def epilogue_cost(G, torch, s):
    """Fused tail vs the tail-free GEMV of the same shape (per-launch CUDA-event mean over
    launches cycling through enough weight copies to exceed L2)."""
    from decode_gemv_epilogue_gb300 import synth
    dev = torch.device("cuda")
    out = {}
    for label, wt, M, K, epi in (("f16_4096_add", 1, 4096, 4096, 4), ("q8_0_11008_silu_mul", 2, 11008, 4096, 3),
                                 ("q4_0_14336_silu_mul", 3, 14336, 4096, 3)):
        base = torch.from_numpy(synth.weights(wt, M, K, seed=500)).to(dev)
        ncopy = max(2, int(2 * L2_BYTES // base.numel()) + 1)
        Ws = [base.clone() for _ in range(ncopy)]
        x = torch.from_numpy(synth.normal(K, seed=501)).to(dev)
        aux = torch.from_numpy(synth.normal(M, seed=502)).to(dev)
        dst = torch.empty(M, device=dev)
        times = {}
        for e in (0, epi):
            def run(Wc, e=e):
                G.gemv_fused(Wc, wt, x, M, K, e, aux if e in (3, 4) else None, aux if e == 4 else dst)
            with torch.cuda.stream(s):
                for Wc in Ws:
                    run(Wc)
            s.synchronize()
            reps = 4
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                e0.record(s)
                for _ in range(reps):
                    for Wc in Ws:
                        run(Wc)
                e1.record(s)
            s.synchronize()
            times[e] = e0.elapsed_time(e1) / (reps * len(Ws))
        out[label] = {"none_us": round(1e3 * times[0], 3), "fused_us": round(1e3 * times[epi], 3),
                      "cost": round(times[epi] / times[0] - 1.0, 4)}
        del Ws
    return out


def e2e_measure(G, torch, step, s, args):
    """The same step through the public API from pinned host memory: every step copies its
    activations host->device (one copy), runs the step's prepared calls (the layer as its
    four launches) and copies every result back (one copy); the two copies are the
    library's staging copies (gf_prepare_copy), recorded with the calls as one CUDA graph,
    so a step is one gf_graph_launch."""
    arena, host, (i0, i1), (o0, o1) = step.pack_for_e2e()
    d_in, h_in = arena[i0:i1], host[i0:i1]
    d_out, h_out = arena[o0:o1], host[o0:o1]
    bi = h_in.numel() * h_in.element_size()
    bo = h_out.numel() * h_out.element_size()
    assert bi % 16 == 0 and bo % 16 == 0 and (i0 * 4) % 16 == 0, "staging ranges must be 16-byte granular"
    # the decode loop's calls, planned once on the step's buffers (gf_prepare), between
    # the upload and the download (the download waits for the last GEMV through PDL)
    prepared = [h for _, h in step.prepared(pdl=True)]
    calls = [G.prepare_copy(d_in, h_in, bi)] + prepared + [G.prepare_copy(h_out, d_out, bo, pdl=True)]
    graph = G.Graph(calls)
    reps = max(5, min(args.steps, 200))
    st = s.cuda_stream

    def one():
        graph.launch(stream=st)

    with torch.cuda.stream(s):
        for _ in range(3):
            one()
    s.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(reps):
            one()
        e1.record(s)
    s.synchronize()
    wall = time.perf_counter() - t0
    ms = e0.elapsed_time(e1) / reps
    return {"value": round(step.step_bytes / (ms * 1e-3) / 1e9, 1), "unit": UNIT, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "ms_per_step": round(ms, 6), "wall_ms_per_step": round(1e3 * wall / reps, 6),
            "steps": reps, "launch_mode": "the step's calls prepared once (gf_prepare, gf_prepare_multi, "
                                          "gf_prepare_glu) with the upload from and the download to pinned host "
                                          "memory (gf_prepare_copy: copy kernels) recorded as one graph "
                                          "(gf_graph_create, programmatic dependent launch inside); per step one "
                                          "gf_graph_launch"}


# ----------------------------------------------------------------------------- CPU oracle

_ORACLE_INPUTS = {}


def _oracle_inputs(seed0=0):
    """Seeded inputs of every launch of the step (generated once per process)."""
    from decode_gemv_epilogue_gb300 import synth
    if seed0 not in _ORACLE_INPUTS:
        items = []
        for i, (name, wt, M, K, epi, nc, fw) in enumerate(step_spec()):
            raw = synth.weights(wt, M, K, seed=seed0 + 10 * i)
            X = synth.normal(nc * K, seed=seed0 + 1).reshape(nc, K)
            aux = synth.normal(nc * M, seed=seed0 + 2).reshape(nc, M) if epi in (3, 4) else None
            s = synth.rademacher(1024, seed=seed0 + 9) if fw else None
            items.append((raw, X, aux, s))
        _ORACLE_INPUTS[seed0] = items
    return _ORACLE_INPUTS[seed0]


def oracle_step(frac, seed0=0, part=(0, 1)):
    """Run the fp64 oracle on a row sample (every frac-th row) of every launch of the
    step -- of that sample, share `part` = (w, n): the w-th of n contiguous row ranges of
    each launch; returns (algorithmic bytes of the share, seconds of oracle work)."""
    from oracle import fwht as ofwht
    from oracle import gemv as ogemv
    w, n = part
    total_b, total_t = 0, 0.0
    for (name, wt, M, K, epi, nc, fw), (raw, X, aux, s) in zip(step_spec(), _oracle_inputs(seed0)):
        rows = np.array_split(np.arange(0, M, frac), n)[w]
        if rows.size == 0:
            continue
        t = time.perf_counter()
        if fw:
            X = np.stack([ofwht.fwht_signed(X[c], s, 1024) for c in range(nc)])
        for r0 in range(0, rows.size, 2048):
            ogemv.gemv(raw, wt, X, M, K, epi, aux, rows=rows[r0:r0 + 2048])
        total_t += time.perf_counter() - t
        total_b += algo_bytes(wt, rows.size, K, epi, nc, fw)
    return total_b, total_t


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_part(w, n, frac, nsteps, barrier, q):
    """One process of the row-parallel oracle: its inputs first (untimed), then nsteps
    steps of its row share, each started together with the other processes."""
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    _oracle_inputs()
    spans = []
    for _ in range(nsteps):
        barrier.wait()
        t0 = time.monotonic()
        oracle_step(frac, part=(w, n))
        spans.append((t0, time.monotonic()))
    q.put((w, spans))


def oracle_parallel(frac, nsteps, nproc=None):
    """The oracle (as it stands, one thread per process) over nproc processes, each a
    contiguous share of every launch's sampled rows; per step the wall time from the
    common start to the last process's end.  Processes are spawned (no inherited CUDA
    state).  Returns (per-step seconds, processes)."""
    import multiprocessing as mp
    n = nproc or host_cores()
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(n)
    q = ctx.Queue()
    procs = [ctx.Process(target=_oracle_part, args=(w, n, frac, nsteps, barrier, q), daemon=True) for w in range(n)]
    for p in procs:
        p.start()
    res = [q.get(timeout=1800) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    spans = [r[1] for r in res]
    per_step = [max(sp[i][1] for sp in spans) - min(sp[i][0] for sp in spans) for i in range(nsteps)]
    return per_step, n


def cpu_baseline(reps=3):
    """The oracle over every row of every launch of the step, `reps` times: row-parallel
    over every host core (the reported value) and on one core (~10 s)."""
    b1, t1 = 0, 0.0
    for _ in range(reps):
        bi, ti = oracle_step(1)
        b1 += bi
        t1 += ti
    per_step, n = oracle_parallel(1, reps)
    tn = sum(per_step)
    return {"value": round(b1 / tn / 1e9, 4), "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": "%d full decode steps (every row of every launch, %.0f MB of algorithmic bytes each), "
                      "numpy fp64 oracle, row-parallel: %d processes of one thread, each a contiguous share of "
                      "every launch's rows" % (reps, b1 / reps / 1e6, n),
            "seconds": round(tn, 2),
            "one_core": {"value": round(b1 / t1 / 1e9, 4), "cores": 1, "seconds": round(t1, 2)}}


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    frac = 16
    tb = sum(algo_bytes(wt, np.arange(0, M, frac).size, K, epi, nc, fw)
             for (name, wt, M, K, epi, nc, fw) in step_spec())
    per_step, n = oracle_parallel(frac, max(args.warmup, 0) + args.steps)
    wall = sum(per_step[max(args.warmup, 0):])
    value = tb * args.steps / wall / 1e9
    cb = {"value": round(value, 4), "unit": UNIT, "cores": n, "kind": "oracle",
          "sample": "every 16th row of every launch of one decode step per step (%d steps), row-parallel over "
                    "%d processes of one thread" % (args.steps, n)}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * wall / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": "1/16 of the rows of each launch"},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------- profiling cases

PROFILE_CASES = ("q4_0_glu_14336x4096", "q4_0_multi_qkv_head", "q4_0_down_add_4096x14336", "q4_0_o_add_4096x4096",
                 "q8_0_silu_mul_11008x4096", "f16_add_4096x4096", "fwht_f16_add_5120x5120_n1",
                 "fwht_f16_add_5120x5120_n8")


def profile_case(name, launches=6):
    """A small workload for per-kernel ncu captures: one call of the decode step, issued
    `launches` times (no graph, no timing) over enough weight copies that the weights
    exceed L2; a few hundred MB on the device."""
    import torch
    import __graft_entry__ as ge
    ge.build()
    from decode_gemv_epilogue_gb300 import gemvfuse as G
    from decode_gemv_epilogue_gb300 import synth
    dev = torch.device("cuda")
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    d, f = 4096, 14336
    x, a = up(synth.normal(d, seed=1)), up(synth.normal(d, seed=2))
    r0, r = up(synth.normal(d, seed=3)), torch.empty(d, device=dev)
    xf = up(synth.normal(f, seed=4))
    signs = up(synth.rademacher(1024, seed=5))

    def copies(wt, M, K, nbytes_per):
        n = max(2, -(-2 * L2_BYTES // nbytes_per))
        return [up(synth.weights(wt, M, K, seed=10 + i)) for i in range(n)]

    if name == "q4_0_glu_14336x4096":
        Wg = copies(3, f, d, 2 * row_bytes(3, d) * f)
        Wu = [up(synth.weights(3, f, d, seed=50 + i)) for i in range(len(Wg))]
        g = torch.empty(f, device=dev)
        fn = lambda i: G.gemv_glu(Wg[i % len(Wg)], Wu[i % len(Wg)], 3, x, f, d, g, split_k=False)
    elif name == "q4_0_multi_qkv_head":
        Ws = [[up(synth.weights(3, M, d, seed=10 + 4 * i + j)) for j, M in enumerate((d, d, d, 32))] for i in range(6)]
        outs = [torch.empty(M, device=dev) for M in (d, d, d, 32)]
        fn = lambda i: G.gemv_multi([(Ws[i % 6][j], M, e, None, outs[j])
                                     for j, (M, e) in enumerate(((d, 0), (d, 0), (d, 0), (32, 1)))], 3, x, d)
    elif name == "q4_0_down_add_4096x14336":
        Ws = copies(3, d, f, row_bytes(3, f) * d)
        fn = lambda i: G.gemv_fused_ex(Ws[i % len(Ws)], 3, xf, d, f, 4, r, r, split_k=False)
    elif name == "q4_0_o_add_4096x4096":
        Ws = copies(3, d, d, row_bytes(3, d) * d)
        fn = lambda i: G.gemv_fused_ex(Ws[i % len(Ws)], 3, a, d, d, 4, r0, r, split_k=False)
    elif name == "q8_0_silu_mul_11008x4096":
        Ws = copies(2, 11008, d, row_bytes(2, d) * 11008)
        m, gout = up(synth.normal(11008, seed=6)), torch.empty(11008, device=dev)
        fn = lambda i: G.gemv_fused_ex(Ws[i % len(Ws)], 2, x, 11008, d, 3, m, gout)
    elif name == "f16_add_4096x4096":
        Ws = copies(1, d, d, row_bytes(1, d) * d)
        rr = up(synth.normal(d, seed=7))
        fn = lambda i: G.gemv_fused_ex(Ws[i % len(Ws)], 1, x, d, d, 4, rr, rr, view=(32, 128))
    elif name.startswith("fwht_f16_add_5120x5120_n"):
        nc = int(name.rsplit("n", 1)[1])
        Ws = copies(1, 5120, 5120, row_bytes(1, 5120) * 5120)
        X = up(synth.normal(nc * 5120, seed=8))
        rr = up(synth.normal(nc * 5120, seed=9))
        ws = torch.empty(nc * 5120, device=dev)
        fn = lambda i: G.gemv_fused_ex(Ws[i % len(Ws)], 1, X, 5120, 5120, 4, rr, rr, ncols=nc, fwht_signs=signs,
                                       fwht_block=1024, fwht_workspace=ws)
    else:
        raise SystemExit("unknown profile case %r (one of %s)" % (name, ", ".join(PROFILE_CASES)))
    for i in range(launches):
        fn(i)
    torch.cuda.synchronize()
    assert G.device_status() == 0
    print(json.dumps({"profile_case": name, "launches": launches}))
    return 0


# ----------------------------------------------------------------------------- main

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", choices=PROFILE_CASES,
                    help="run one call of the step a few times (a small workload for ncu) and exit")
    args = ap.parse_args(argv)
    if args.profile_case:
        return profile_case(args.profile_case)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and "WORLD_SIZE" in os.environ:
        print("warning: --gpus %d but WORLD_SIZE %d" % (args.gpus, world), file=sys.stderr)
    if args.impl == "reference":
        out = reference_arm(args, rank, world)
        if out is not None:
            print(json.dumps(out))
        return 0
    out = gpu_arm(args, rank, world, local_rank)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline()
        print(json.dumps(out))
    return 0


if __name__ == "__main__":
    sys.exit(main())
