"""Benchmark of the quantized sparse MoE FFN layer (one JSON line on rank 0).

Default workload: decode, T=1 token through 40 independent Qwen3.6-35B-A3B
shaped MoE layers (H=2048, 256 experts, top-8 + shared expert, I=512, Q8_0
weights, 34.4 GB resident).  One step = one pass of the whole hot path
(route -> group -> FFN with SwiGLU and combine) over the 40 layers, in
sequence, captured in a CUDA graph.  Metric: MoE-layer tokens/s = T * 40 /
step time.  Inputs are synthetic, seeded, drawn on the device before the
timed region; the 1.3 GB of expert weights a step touches is ~10x the L2,
so no flush is needed.

The metric is quoted on T=1 decode and on T=4096 prefill: the default line
also carries a "prefill" object for one T=4096 layer (Zipf-offset routing,
Q8_0), measured in the same run with the same protocol.

Protocol per workload: W warm-up replays, then exactly K graph replays
between two events (ms_per_step, value), then --replays further replays
each timed alone ("replays": median and spread), with the routing ids
hashed after every replay and required identical (the output-hash check of
"Ember: packed Q8 decode"); the oracle is timed on the host at all cores and
at one thread (cpu_baseline).

Other workloads (--workload): prefill (T=4096, Zipf-skewed routing, one
layer), batched16 / batched64 / batched1 (affine 4-bit, 40 layers), gemv
(Llama-3.2-1B Q8_0 projections).

--impl reference times the fp64 CPU oracle on the host cores, on a bounded
sample of the same workload, and reports it in the same metric.
Multi-GPU (torchrun): replicas only, each rank runs its own copy; the time is
the max over ranks and value = all ranks' tokens / that time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

Q8_EXPERT_BYTES = {  # per expert, H=2048, I=512
    synth.Q8_0: (2 * 512 * 2048 + 2 * 512 * 64 * 2, 2048 * 512 + 2048 * 16 * 2),
    synth.AFFINE4_G64: (1024 * 1024 + 1024 * 32 * 4, 2048 * 256 + 2048 * 8 * 4),
}
ROUTER_BYTES = 256 * 2048 * 4

WORKLOADS = {
    "decode": dict(shape=synth.QWEN, T=1, layers=40, zipf=None,
                   desc="decode T=1, 40 layers, H=2048, E=256, top-8 + shared, "
                        "I=512, Q8_0"),
    "batched1": dict(shape=synth.QWEN_A4, T=1, layers=40, zipf=None,
                     desc="batched decode T=1, 40 layers, affine-4 g64"),
    "batched16": dict(shape=synth.QWEN_A4, T=16, layers=40, zipf=None,
                      desc="batched decode T=16, 40 layers, affine-4 g64"),
    "batched64": dict(shape=synth.QWEN_A4, T=64, layers=40, zipf=None,
                      desc="batched decode T=64, 40 layers, affine-4 g64"),
    "prefill": dict(shape=synth.QWEN, T=4096, layers=1, zipf="noise",
                    desc="prefill T=4096, 1 layer, Zipf-offset routing, Q8_0"),
    "prefill_a4": dict(shape=synth.QWEN_A4, T=4096, layers=1, zipf="noise",
                       desc="prefill T=4096, 1 layer, Zipf-offset routing, affine-4 g64"),
    "gemv": dict(gemv="f16", desc="Q8_0 GEMV batch 1, Llama-3.2-1B projection shapes "
                                  "(2048x2048, 512x2048, 8192x2048, 2048x8192, 128256x2048)"),
    "gemv_layer": dict(gemv="f16", shapes="layer",
                       desc="Q8_0 GEMV batch 1, one Llama-3.2-1B layer's projections with "
                            "shared-activation stacking (QKV 3072x2048, O 2048x2048, gate_up "
                            "16384x2048, down 2048x8192) and the LM head 128256x2048"),
    "gemv_i8": dict(gemv="i8", desc="Q8_0 GEMV batch 1 on the int8-quantized activation, "
                                    "Llama-3.2-1B projection shapes"),
}


def measured_traffic(workload):
    """DRAM bytes per launch of the workload's dominant kernel (group) from the
    committed ncu capture, or None when its sources changed since."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "ffn_dram_traffic.json")
    if not os.path.exists(p):
        return None
    ent = json.load(open(p)).get(workload)
    if not ent:
        return None
    m = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_sparse_moe_gb300", "csrc")
    for f in ent["sources"]:
        m.update(open(os.path.join(csrc, f), "rb").read())
    return ent["bytes_per_launch"] if m.hexdigest() == ent["sources_sha256"] else None


def rank_max(x, dev, world):
    """The largest of x over all ranks (x itself for one rank): every rank's
    timed region is bracketed by the same barriers, so the job takes as long
    as its slowest rank."""
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.item()


def job_value(world, units_per_rank, ms):
    """Whole-job throughput: the units all ranks processed per second of the
    slowest rank's time."""
    return world * units_per_rank / (ms / 1e3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d.get("bf16_tflops"), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------- ours

def fnv1a64(data: bytes) -> str:
    """FNV-1a 64-bit hash (the output hash of the Ember page's method)."""
    h = 0xcbf29ce484222325
    for b in data:
        h = ((h ^ b) * 0x100000001b3) & 0xFFFFFFFFFFFFFFFF
    return f"fnv1a64:{h:016x}"


def replay_stats(graph, stream, fwds, n):
    """Each of n further graph replays timed alone (its own event pair on the
    launching stream), and the routing ids of every layer hashed after each
    replay: all replays must route identically ("Ember: packed Q8 decode",
    method paragraph: every accepted trial shares one output hash).  The
    check compares a BLAKE2b digest of each replay's ids; the FNV-1a 64 hash
    of the first replay's ids is reported as the output hash."""
    import hashlib
    times, digests, first = [], set(), None
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for a, b in evs:
        with torch.cuda.stream(stream):
            a.record(stream)
            graph.replay()
            b.record(stream)
        stream.synchronize()
        ids = torch.cat([f.topk_idx.reshape(-1) for f in fwds]).cpu().numpy().tobytes()
        digests.add(hashlib.blake2b(ids, digest_size=16).hexdigest())
        if first is None:
            first = ids
        times.append(a.elapsed_time(b))
    if len(digests) != 1:
        raise RuntimeError(f"routing differed across replays: {len(digests)} distinct outputs")
    t = np.array(times)
    return {"n": n, "median_ms": float(np.median(t)), "p10_ms": float(np.percentile(t, 10)),
            "p90_ms": float(np.percentile(t, 90)), "routing_hash": fnv1a64(first),
            "hash_equal_over_replays": True}


def build_layers(qsm, wl, device, seed, fuse=True, gated=False, sel_only=False):
    shape = wl["shape"]
    layers, xs, fwds, syn = [], [], [], []
    for l in range(wl["layers"]):
        Lg = synth.draw_layer(shape, device, seed=seed, layer=l, zipf=wl["zipf"])
        syn.append(Lg)
        sg = synth.draw_shared_gate(shape.H, device, seed, l) if gated else None
        L = qsm.Layer.from_synth(Lg, sg)
        layers.append(L)
        xs.append(synth.draw_x(wl["T"], shape.H, device, seed, l))
        fwds.append(qsm.MoEForward(L, wl["T"], device, fuse_route_group=fuse,
                                   bias_select_only=sel_only))
    return layers, xs, fwds, syn


class ChunkedLayer:
    """One layer through moe_layer_forward in chunks, outputs and workspace
    allocated once."""

    def __init__(self, qsm, L, T, chunk, device, sel_only=False):
        self.qsm, self.L, self.chunk, self.sel_only = qsm, L, chunk, sel_only
        self.y = torch.empty((T, L.H), dtype=torch.bfloat16, device=device)
        self.idx = torch.empty((T, L.k), dtype=torch.int32, device=device)
        self.w = torch.empty((T, L.k), dtype=torch.float32, device=device)
        self.ws = torch.zeros(qsm.layer_workspace_bytes(L, T, chunk), dtype=torch.uint8,
                              device=device)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=device)

    def __call__(self, x, stream=None):
        self.qsm.moe_layer_forward(self.L, x, self.chunk, True, self.sel_only, y=self.y,
                                   topk_idx=self.idx,
                                   topk_w=self.w, workspace=self.ws,
                                   dev_status=self.dev_status, stream=stream)
        return self.y


def touched_bytes(layers, fwds, qtype):
    """Distinct touched experts (from the device routing) + shared +
    router + x + y, per step."""
    gu, dn = Q8_EXPERT_BYTES[qtype]
    total = 0
    n_exp = 0
    for L, f in zip(layers, fwds):
        ne = int(torch.unique(f.topk_idx).numel())
        n_exp += ne
        T = f.T
        total += (ne + 1) * (gu + dn) + ROUTER_BYTES + 2 * T * L.H * 2
    return total, n_exp


def run_ours(args, wl, rank, world):
    import quantized_sparse_moe_gb300 as qsm
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    layers, xs, fwds, syn = build_layers(qsm, wl, dev, seed=0,
                                         fuse=args.route_group == "fused",
                                         gated=args.gated_shared,
                                         sel_only=args.bias_select_only)
    T, nL = wl["T"], wl["layers"]
    stream = torch.cuda.Stream(device=dev)

    calls = fwds
    if args.chunk:  # the whole layer per call, in chunks of args.chunk tokens
        calls = [ChunkedLayer(qsm, L, T, args.chunk, dev, args.bias_select_only)
                 for L in layers]

    def step(s):
        for f, x in zip(calls, xs):
            f(x, stream=s)

    # warm-up (also builds the library and fixes the routing)
    with torch.cuda.stream(stream):
        step(stream)
    if args.chunk:  # the unchunked calls give the routing counts for the bytes
        with torch.cuda.stream(stream):
            for f, x in zip(fwds, xs):
                f(x, stream=stream)
    torch.cuda.synchronize()
    for f in list(fwds) + (list(calls) if args.chunk else []):
        assert f.dev_status.item() == 0, "device status set"
    graph = torch.cuda.CUDAGraph()
    n0 = qsm.launch_count()
    with torch.cuda.graph(graph, stream=stream):
        step(torch.cuda.current_stream())
    launches_per_step = qsm.launch_count() - n0
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks, torch.cuda.stream(stream):
        time.sleep(0.25)
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = rank_max(ev0.elapsed_time(ev1) / args.steps, dev, world)
    value = job_value(world, T * nL, ms)
    replays = replay_stats(graph, stream, fwds, args.replays)

    # dominant launch pair: the expert FFN (gate_up+SwiGLU, down+combine),
    # bracketed per layer by event nodes inside a captured graph so the
    # elapsed times are pure device time on the FFN's stream
    def graph_event():
        # an event-record node inside the captured graph (timing enabled)
        return torch.cuda.Event(enable_timing=True, external=True)

    one_launch = fwds[0].decode_ws is not None and not args.chunk
    evs = [(graph_event(), graph_event()) for _ in range(nL)]
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        s2 = torch.cuda.current_stream()
        for (a, b), f, x, L in zip(evs, fwds, xs, layers):
            if one_launch:  # the whole layer is the one launch
                a.record(s2)
                f(x, stream=s2)
                b.record(s2)
                continue
            qsm.moe_route(x, L.w_router, L.k, L.logit_bias, f.renormalize, f.topk_idx,
                          f.topk_w, f.route_ws, f.dev_status, s2)
            qsm.moe_group_tokens(f.topk_idx, L.E, f.grouping.tile_rows,
                                 f.grouping, f.dev_status, s2)
            a.record(s2)
            qsm.moe_ffn_forward(L, x, f.topk_idx, f.topk_w, f.grouping, f.y,
                                False, f.ffn_ws, f.dev_status, s2)
            b.record(s2)
    ffn_ms = []
    with torch.cuda.stream(stream):
        for rep in range(5):
            g2.replay()
            torch.cuda.synchronize()
            ffn_ms.append(sum(a.elapsed_time(b) for a, b in evs) / nL)
    ffn_ms = min(ffn_ms)
    qtype = wl["shape"].qtype
    step_bytes, n_exp = touched_bytes(layers, fwds, qtype)
    gu, dn = Q8_EXPERT_BYTES[qtype]
    ffn_bytes_per_layer = (n_exp / nL + 1) * (gu + dn) + 2 * T * 2048 * 2
    if one_launch:
        ffn_bytes_per_layer += ROUTER_BYTES
    hbm, _, peak_kind = peaks()
    # DRAM bytes per FFN call (ncu), or per layer launch for the one-launch path
    traffic = measured_traffic(wl.get("name", args.workload) + ("_one_launch" if one_launch else ""))
    if args.chunk:
        # the dominant launch group is the whole chunked layer call
        ffn_ms = ms / nL
        traffic = None
    elif one_launch:
        # the timed step is nL back-to-back launches of this one kernel (the
        # event-bracketed replay above breaks their programmatic overlap)
        ffn_ms = ms / nL

    # end to end through the public API: pinned host x in, host y out
    xh = torch.stack(xs).cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    xd = torch.empty_like(xs[0]).new_empty((nL,) + tuple(xs[0].shape))
    yd = torch.empty_like(xd)  # the step's outputs, read back in one copy
    e_ms = []
    for rep in range(args.warmup + args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e0.record(stream)
        with torch.cuda.stream(stream):
            xd.copy_(xh, non_blocking=True)
            for l, f in enumerate(calls):
                if args.chunk:
                    yd[l].copy_(f(xd[l], stream=stream), non_blocking=True)
                else:
                    f(xd[l], stream=stream, out=yd[l])
            yh.copy_(yd, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
        t1 = time.perf_counter()
        if rep >= args.warmup:
            e_ms.append((t1 - t0) * 1e3)
    e2e_ms = rank_max(statistics.median(e_ms), dev, world)

    achieved = ffn_bytes_per_layer / (ffn_ms / 1e3) / 1e9
    # algorithmic FLOPs per layer: expert matmuls (k routed + shared per
    # token, gate_up 2*2I*H + down 2*H*I) and the router (2*E*H per token)
    sh = wl["shape"]
    flops_layer = (2.0 * T * (sh.k + 1) * 3 * sh.H * sh.I + 2.0 * T * sh.E * sh.H)
    _, tc_peak, _ = peaks()
    t_hbm = step_bytes / (hbm * 1e9)
    t_tc = flops_layer * nL / (tc_peak * 1e12)
    bound = "tensor" if t_tc > t_hbm else "hbm"
    result = {
        "metric": "MoE-layer tokens/s",
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "q8_0/affine4 weights, f16 MMA inputs, f32 accumulate",
        "data": "synthetic (seeded; random-init weights of the layer shapes)",
        "config": {"workload": wl["desc"], "tokens_per_layer": T,
                   "layers": nL, "parallelism": f"replicas x{world}",
                   "route_group": ("one launch per layer" if one_launch else
                                   args.route_group if T <= 8 else "separate"),
                   "chunk_tokens": args.chunk or None,
                   "workspace_bytes_per_layer": int(
                       calls[0].ws.numel() if args.chunk else
                       fwds[0].decode_ws.numel() if one_launch else
                       fwds[0].route_ws.numel() + fwds[0].ffn_ws.numel()),
                   "l2": "inputs larger than L2 (touched weights per step "
                         f"{step_bytes / 1e9:.2f} GB)"},
        "layer_roofline": {
            "bound": bound, "touched_bytes_per_step": step_bytes,
            "flops_per_step": flops_layer * nL,
            "floor_ms": max(t_hbm, t_tc) * 1e3,
            "hbm_frac": t_hbm / (ms / 1e3), "tensor_frac": t_tc / (ms / 1e3),
            "frac": max(t_hbm, t_tc) / (ms / 1e3),
            "peak_gbs": hbm, "peak_tflops": tc_peak, "peak_kind": peak_kind},
        "roofline": ({
            "kernel": ("moe_decode_layer (router, selection, gate_up+SwiGLU, "
                       "down+combine in one launch)" if one_launch else
                       "moe_ffn_forward (gate_up+SwiGLU "
                       + ("streamed by one CTA per SM" if T > 8 else "d1") + ", d2 down+combine)"),
            "bound": "hbm", "achieved": achieved, "peak": hbm,
            "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
            "bytes_per_launch": ffn_bytes_per_layer,
            "launch_ms": ffn_ms, "peak_kind": peak_kind} if T <= 64 else {
            "kernel": ("moe_ffn_forward (prep, gate_up GEMM, down GEMM, finalize)"
                       if not args.chunk else
                       f"moe_layer_forward in chunks of {args.chunk} tokens "
                       "(route, group, FFN per chunk)"),
            "bound": "tensor",
            "achieved": (flops_layer - 2.0 * T * sh.E * sh.H) / (ffn_ms / 1e3) / 1e12,
            "peak": tc_peak, "unit": "TFLOP/s",
            "frac": (flops_layer - 2.0 * T * sh.E * sh.H) / (ffn_ms / 1e3) / 1e12 / tc_peak,
            "traffic": traffic, "flops_per_launch": flops_layer - 2.0 * T * sh.E * sh.H,
            "launch_ms": ffn_ms, "peak_kind": peak_kind}),
        "e2e": {"value": job_value(world, T * nL, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": xh.numel() * 2,
                "d2h_bytes_per_step": yh.numel() * 2, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks.summary(),
        "replays": dict(replays, tokens_per_s_at_median=job_value(world, T * nL, replays["median_ms"])),
    }
    return result, (syn, fwds, xs)


# ----------------------------------------------------------- CPU oracle

class OracleSampler:
    """The fp64 oracle on the host cores over a bounded sample of the
    workload: up to max_layers of its layers (weights copied to the host
    once), each call one full layer (route, group, expert FFNs, combine) for
    the layer's tokens (prefill: a fixed sample of 64 tokens of the full
    routing)."""

    def __init__(self, wl, layers_dev, xs_dev, max_layers=4):
        import oracle
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        from _helpers import bits16, oracle_q
        self.oracle = oracle
        self.layers = []
        T = wl["T"]
        for Lg, x in list(zip(layers_dev, xs_dev))[:max_layers]:
            toks = np.arange(T, dtype=np.int32)
            if T > 64:
                toks = np.random.default_rng(0).choice(T, 64, replace=False).astype(np.int32)
            self.layers.append(dict(
                q=[oracle_q(t) for t in (Lg.gate_up, Lg.down, Lg.shared_gate_up,
                                         Lg.shared_down)],
                x=bits16(x), wr=Lg.w_router.cpu().numpy(),
                bias=None if Lg.logit_bias is None else Lg.logit_bias.cpu().numpy(),
                k=Lg.shape.k, E=Lg.shape.E, toks=toks))

    def run(self, budget_s, threads=None):
        """Calls cycling over the sampled layers until budget_s seconds of
        oracle time; returns (tokens/s, seconds, calls).  threads: OpenMP
        threads for this run (default: all host cores)."""
        orc = self.oracle
        all_cores = orc.max_threads()
        orc.set_threads(threads or all_cores)
        try:
            return self._run(budget_s)
        finally:
            orc.set_threads(all_cores)

    def _run(self, budget_s):
        orc = self.oracle
        tokens, t_used, calls = 0, 0.0, 0
        while t_used < budget_s:
            L = self.layers[calls % len(self.layers)]
            t0 = time.perf_counter()
            idx, w = orc.route(L["x"], L["wr"], L["k"], L["bias"])
            orc.group(idx, L["E"], 8)
            orc.moe_layer(L["x"], idx, w, *L["q"], tokens=L["toks"])
            t_used += time.perf_counter() - t0
            tokens += len(L["toks"])
            calls += 1
        return tokens / t_used, t_used, calls

    def baseline(self, budget_s, budget_1t_s):
        """cpu_baseline object: all host cores, and one thread."""
        cores = self.oracle.max_threads()
        v, t, calls = self.run(budget_s)
        v1, t1, calls1 = self.run(budget_1t_s, threads=1)
        return {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                "sample": self.describe(t, calls),
                "one_thread": {"value": v1, "unit": "tokens/s", "cores": 1,
                               "sample": self.describe(t1, calls1)},
                "speedup_all_cores": v / v1 if v1 > 0 else None}

    def describe(self, seconds, calls):
        return (f"{len(self.layers)} layer(s) of the workload, {calls} call(s) cycling "
                f"over them, {seconds:.1f} s of fp64 oracle (route, group, expert "
                f"FFNs, combine; {len(self.layers[0]['toks'])} token(s) per call)")


def run_reference(args, wl, rank, world):
    if rank != 0:
        return None
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    Ls = [synth.draw_layer(wl["shape"], dev, seed=0, layer=l, zipf=wl["zipf"])
          for l in range(min(wl["layers"], 2))]
    xs = [synth.draw_x(wl["T"], wl["shape"].H, dev, 0, l) for l in range(len(Ls))]
    sampler = OracleSampler(wl, Ls, xs, max_layers=2)
    del Ls
    # each step a bounded sample: the whole run stays within about 90 s
    step_s = min(6.0, max(0.05, 90.0 / (args.warmup + args.steps)))
    vals, secs, calls = [], 0.0, 0
    for s in range(args.warmup + args.steps):
        v, t, c = sampler.run(step_s)
        if s >= args.warmup:
            vals.append(v)
            secs += t
            calls += c
    value = statistics.median(vals)
    prefill = None
    if args.workload == "decode" and not args.no_prefill:
        # the prefill workload of the same metric, on a bounded sample
        pwl = WORKLOADS["prefill"]
        PL = [synth.draw_layer(pwl["shape"], dev, seed=0, layer=0, zipf=pwl["zipf"])]
        px = [synth.draw_x(pwl["T"], pwl["shape"].H, dev, 0, 0)]
        psampler = OracleSampler(pwl, PL, px, max_layers=1)
        del PL
        pv, pt, pc = psampler.run(min(20.0, max(5.0, step_s * args.steps)))
        prefill = {"value": pv, "unit": "tokens/s", "config": {"workload": pwl["desc"],
                                                               "tokens_per_layer": pwl["T"],
                                                               "layers": 1},
                   "cpu_baseline": {"value": pv, "unit": "tokens/s",
                                    "cores": psampler.oracle.max_threads(), "kind": "oracle",
                                    "sample": psampler.describe(pt, pc)},
                   "e2e": {"value": pv, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}}
    out = {
        "impl": "reference", "metric": "MoE-layer tokens/s", "value": value,
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl["desc"], "tokens_per_layer": wl["T"],
                   "layers": wl["layers"]},
        "cpu_baseline": {"value": value, "unit": "tokens/s",
                         "cores": sampler.oracle.max_threads(), "kind": "oracle",
                         "sample": sampler.describe(secs, calls) +
                                   f"; {step_s:.2f} s per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    if prefill is not None:
        out["prefill"] = prefill
    return out



# --------------------------------------------------------------- GEMV sweep

def gemv_metric(wl):
    if wl.get("shapes") == "layer":
        return ("Q8_0 GEMV weight GB/s (one GEMV per stacked projection of a layer and the "
                "LM head per step)")
    return "Q8_0 GEMV weight GB/s (one GEMV per projection shape per step)"


def run_gemv(args, wl, rank, world):
    """One step = one batch-1 GEMV per Llama-3.2-1B projection shape.  The
    matrices that fit in L2 rotate over copies so a step's weights exceed
    four times the L2 (129 MB); the LM head alone is larger than L2."""
    import quantized_sparse_moe_gb300 as qsm
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    i8 = wl["gemv"] == "i8"
    shapes = list((synth.GEMV_LAYER_SHAPES if wl.get("shapes") == "layer"
                   else synth.GEMV_SHAPES).items())
    small = sum(n * k for name, (n, k) in shapes if name != "lm_head") * 34 // 32
    R = max(1, -(-4 * 129_000_000 // small))  # copies of the L2-sized matrices
    mats = {}
    for name, (n, k) in shapes:
        copies = 1 if name == "lm_head" else R
        mats[name] = [synth.draw_gemv(n, k, dev, seed=c, name=name) for c in range(copies)]
    step_bytes = sum(n * k * 34 // 32 + 2 * (n + k) for name, (n, k) in shapes)
    ys = {name: torch.empty(n, dtype=torch.bfloat16, device=dev) for name, (n, _) in shapes}
    qbuf = {k: (torch.empty(k, dtype=torch.int8, device=dev),
                torch.empty(k // 32, dtype=torch.float32, device=dev))
            for k in {k for _, (_, k) in shapes}}
    stream = torch.cuda.Stream(device=dev)

    def one(name, c, s):
        x, q, d = mats[name][c % len(mats[name])]
        if i8:
            qx, dx = qbuf[q.shape[1]]
            qsm.q8_quantize_x(x, qx, dx, stream=s)
            qsm.q8_gemv_i8(qx, dx, q, d, ys[name], stream=s)
        else:
            qsm.q8_gemv(x, q, d, ys[name], stream=s)

    def step(c, s):
        for name, _ in shapes:
            one(name, c, s)

    with torch.cuda.stream(stream):
        for c in range(R):
            step(c, stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    n0 = qsm.launch_count()
    with torch.cuda.graph(graph, stream=stream):
        for c in range(R):
            step(c, torch.cuda.current_stream())
    launches_per_replay = qsm.launch_count() - n0
    replays = max(1, -(-args.steps // R))
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    with ClockSampler(dev.index) as clocks, torch.cuda.stream(stream):
        time.sleep(0.25)
        ev0.record(stream)
        for _ in range(replays):
            graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = rank_max(ev0.elapsed_time(ev1) / (replays * R), dev, world)
    # per shape: a graph of its R rotations, timed alone
    per_shape = {}
    for name, (n, k) in shapes:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for c in range(R):
                one(name, c, torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(20):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / (20 * R)
        by = n * k * 34 // 32
        per_shape[name] = {"N": n, "K": k, "us": us, "GB/s": by / (us * 1e-6) / 1e9}
    hbm, _, peak_kind = peaks()
    top = max(per_shape, key=lambda k: per_shape[k]["us"])
    # end to end: pinned host x in, host y out, each step
    xh = {name: mats[name][0][0].cpu().pin_memory() for name, _ in shapes}
    yh = {name: torch.empty_like(ys[name], device="cpu").pin_memory() for name, _ in shapes}
    xd = {name: torch.empty_like(mats[name][0][0]) for name, _ in shapes}
    e_ms = []
    for r in range(args.warmup + min(args.steps, 200)):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for name, _ in shapes:
                xd[name].copy_(xh[name], non_blocking=True)
                _, q, d = mats[name][r % len(mats[name])]
                x = xd[name]
                if i8:
                    qx, dx = qbuf[q.shape[1]]
                    qsm.q8_quantize_x(x, qx, dx, stream=stream)
                    qsm.q8_gemv_i8(qx, dx, q, d, ys[name], stream=stream)
                else:
                    qsm.q8_gemv(x, q, d, ys[name], stream=stream)
                yh[name].copy_(ys[name], non_blocking=True)
        stream.synchronize()
        if r >= args.warmup:
            e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_ms = rank_max(statistics.median(e_ms), dev, world)
    result = {
        "metric": gemv_metric(wl),
        "value": job_value(world, step_bytes, ms) / 1e9, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("int8 activation codes x int8 weight codes, s32 block sums, f32 scales"
                  if i8 else "q8_0 weights, f16 MMA inputs, f32 accumulate"),
        "data": "synthetic (seeded)",
        "config": {"workload": wl["desc"], "rotating_copies": R,
                   "l2": f"weights per step {step_bytes / 1e6:.0f} MB, L2-sized matrices "
                         f"rotate over {R} copies"},
        "per_shape": per_shape,
        "roofline": {"kernel": f"{'q8_gemv_i8' if i8 else 'q8_gemv'} {top} "
                               f"({per_shape[top]['N']}x{per_shape[top]['K']})",
                     "bound": "hbm", "achieved": per_shape[top]["GB/s"], "peak": hbm,
                     "unit": "GB/s", "frac": per_shape[top]["GB/s"] / hbm,
                     # DRAM bytes of one LM-head launch (ncu), int8-activation mode not captured
                     "traffic": measured_traffic("gemv") if not i8 and top == "lm_head" else None,
                     "bytes_per_launch": per_shape[top]["N"] * per_shape[top]["K"] * 34 // 32,
                     "launch_ms": per_shape[top]["us"] / 1e3, "peak_kind": peak_kind},
        "step_roofline": {"bytes_per_step": step_bytes, "frac": step_bytes / (ms * 1e-3) / 1e9 / hbm},
        "e2e": {"value": job_value(world, step_bytes, e2e_ms) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": sum(2 * k for _, (_, k) in shapes),
                "d2h_bytes_per_step": sum(2 * n for _, (n, _) in shapes), "ms_per_step": e2e_ms},
        "gpu_launches": launches_per_replay * replays,
        "clocks": clocks.summary(),
    }
    return result, mats


def gemv_cpu_baseline(wl, mats, budget_s=12.0):
    """The fp64 oracle GEMV over the same shapes (copy 0), cycling until the
    budget; GB/s of weights."""
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from _helpers import bits16
    host = {name: (bits16(m[0][0].cpu()), m[0][1].cpu().numpy(), bits16(m[0][2].cpu()))
            for name, m in mats.items()}
    t_used, by, calls = 0.0, 0, 0
    i8 = wl["gemv"] == "i8"
    while t_used < budget_s:
        for name, (x, q, d) in host.items():
            t0 = time.perf_counter()
            if i8:
                qx, dx = oracle.q8_quantize_x(x)
                oracle.q8_gemv_i8(qx, dx, q, d)
            else:
                oracle.q8_gemv(x, q, d)
            t_used += time.perf_counter() - t0
            by += q.size * 34 // 32
            calls += 1
    return {"value": by / t_used / 1e9, "unit": "GB/s", "cores": oracle.max_threads(),
            "kind": "oracle", "sample": f"{calls} GEMVs over the five shapes, "
                                         f"{t_used:.1f} s of fp64 oracle"}

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--route-group", default="fused", choices=["fused", "separate"],
                    help="for T <= 8: one fused route+group launch, or the two "
                         "separate launches")
    ap.add_argument("--gated-shared", action="store_true",
                    help="sigmoid-gated shared expert (a random gate vector per layer)")
    ap.add_argument("--bias-select-only", action="store_true",
                    help="the logit bias selects experts but leaves the weights")
    ap.add_argument("--chunk", type=int, default=0,
                    help="run each layer through moe_layer_forward in chunks of "
                         "this many tokens (chunked prefill)")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the layer count (profiling runs only)")
    ap.add_argument("--replays", type=int, default=100,
                    help="graph replays timed one by one after the K timed steps "
                         "(median and routing-hash check)")
    ap.add_argument("--no-prefill", action="store_true",
                    help="decode workload: leave out the T=4096 prefill object")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group("nccl")
    wl = dict(WORKLOADS[args.workload])
    if args.layers:
        wl["layers"] = args.layers
        wl["desc"] += f" (layer count overridden: {args.layers})"
    if args.chunk:
        wl["desc"] += f", chunks of {args.chunk} tokens"
    if args.gated_shared:
        wl["desc"] += ", gated shared expert"
    if args.bias_select_only:
        wl["desc"] += ", selection-only logit bias"
    if "gemv" in wl:
        if args.impl == "reference":
            res = None
            if rank == 0:
                import quantized_sparse_moe_gb300  # noqa: F401 (device init only)
                dev = torch.device("cuda", 0)
                shapes = (synth.GEMV_LAYER_SHAPES if wl.get("shapes") == "layer"
                          else synth.GEMV_SHAPES)
                mats = {name: [synth.draw_gemv(n, k, dev, seed=0, name=name)]
                        for name, (n, k) in shapes.items()}
                cb = gemv_cpu_baseline(wl, mats, budget_s=min(60.0, max(
                    5.0, 90.0 * args.steps / (args.steps + args.warmup))))
                res = {"impl": "reference", "metric": gemv_metric(wl),
                       "value": cb["value"], "unit": "GB/s",
                       "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                       "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                       "dtype": "f64", "data": "synthetic", "config": {"workload": wl["desc"]},
                       "cpu_baseline": cb, "e2e": {"value": cb["value"], "unit": "GB/s",
                                                   "h2d_bytes_per_step": 0,
                                                   "d2h_bytes_per_step": 0}}
        else:
            res, mats = run_gemv(args, wl, rank, world)
            if rank == 0 and not args.no_cpu_baseline:
                res["cpu_baseline"] = gemv_cpu_baseline(wl, mats)
    elif args.impl == "reference":
        res = run_reference(args, wl, rank, world)
    else:
        res, (syn, fwds, xs) = run_ours(args, wl, rank, world)
        if rank == 0 and not args.no_cpu_baseline:
            sampler = OracleSampler(wl, syn, xs, max_layers=4)
            res["cpu_baseline"] = sampler.baseline(10.0, 4.0)
        del syn, fwds, xs
        if args.workload == "decode" and not args.no_prefill and not args.layers:
            # the metric is quoted on T=1 decode and T=4096 prefill: the
            # prefill layer is measured in the same run, same protocol
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
            pwl = dict(WORKLOADS["prefill"], name="prefill")
            pres, (psyn, pfwds, pxs) = run_ours(args, pwl, rank, world)
            if rank == 0 and not args.no_cpu_baseline:
                psampler = OracleSampler(pwl, psyn, pxs, max_layers=1)
                pres["cpu_baseline"] = psampler.baseline(10.0, 4.0)
            for key in ("metric", "n_gpus", "steps", "warmup", "higher_is_better",
                        "scaling", "vs_baseline", "data"):
                pres.pop(key, None)
            res["prefill"] = pres
    if rank == 0 and res is not None:
        print(json.dumps(res))
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
