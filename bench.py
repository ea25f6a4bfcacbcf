#!/usr/bin/env python
"""Benchmark of the lookahead sparse decode hot path on one GB300 (or N replicas).

Workload: Qwen3-8B decode shape - 36 layers, batch 32, 32 query / 8 KV heads,
head dim 128, bf16, context 32768 (2048 blocks of 16), budget 2048 tokens (128
blocks), 4 lookahead queries, fetch cap 0.02 x budget = 2 blocks per KV head per
step, 64 planted hot blocks per head, AR(1) query drift (rho 0.9).  Inputs are
synthetic (seeded counter-based generator), resident in HBM / page-locked host
memory before the timed region; the per-layer key cache (2 GiB) is far larger
than L2, so no flush is needed between steps.

One step = one decode step = all 36 layers x (score, top-K, capped diff, host
gather, sparse attention) over the whole batch.  Metric: layer-steps/s (plus the
achieved HBM GB/s of the path and of the dominant kernel, block scoring).

Defaults: max-dot scoring; the `overlap` launch order (each layer's gather on a
side stream beside the previous layer's attention); the host tier in one
cudaHostAlloc allocation holding 8 layers of distinct data (layer l reads buffer
l mod 8, 4 GiB each), read once through the SMs before the pre-roll; 32 timed
steps.  The timed steps are one captured CUDA graph.  The
JSON line also reports the pooled-key scoring and cross-step pipeline variants,
the fused look-ahead attention, the host-link roofline of the gather, per-layer
prediction agreement, an end-to-end run with host copies, clocks and the CPU
oracle baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun every rank runs its own replica on its own GPU (independent
requests, no data-path collective): weak scaling, value = all ranks' layer-steps
over the max time.  ``--impl reference`` times the CPU oracle on the host cores
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time


def _impl_from_argv():
    for i, a in enumerate(sys.argv):
        if a == "--impl" and i + 1 < len(sys.argv):
            return sys.argv[i + 1]
        if a.startswith("--impl="):
            return a.split("=", 1)[1]
    return None


# The CPU oracle's numpy products are small: on the 16-core host of a GB300 node
# its BLAS ran a layer-step about 2.5x faster with one thread than with all cores.
# The oracle runs in this process only under --impl reference, so that arm takes
# one thread unless the environment says otherwise (set before numpy loads).
if _impl_from_argv() == "reference":
    for _k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(_k, "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse decode layer-steps/sec and achieved HBM GB/s (% of GB300 peak)"
UNIT = "layer-steps/s"
# ncu DRAM traffic of one scoring launch, per scorer kernel, with the hash of the
# kernel source it was taken on
PROFILE_TRAFFIC = {"mma": os.path.join(ROOT, "profiles", "score_blocks_traffic.json"),
                   "tc": os.path.join(ROOT, "profiles", "score_blocks_tc_traffic.json")}
KERNEL_SOURCE = {"mma": "score.cu", "tc": "score_tc.cu"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="oasis", choices=["oasis", "reference"])
    ap.add_argument("--layers", type=int, default=36, help="model layers (36 = Qwen3-8B)")
    ap.add_argument("--batch", type=int, default=32)
    ap.add_argument("--ctx", type=int, default=32768)
    ap.add_argument("--host-layers", type=int, default=8,
                    help="distinct host-tier layers (layer l uses buffer l mod N; 0 = as many as 60%% of the "
                         "available host memory holds); 8 layers (32 GiB) gave ~15%% more layer-steps/s than 29 on the same box")
    ap.add_argument("--preroll", type=int, default=40,
                    help="untimed decode steps run first, so the timed steps see a warmed-up resident set")
    ap.add_argument("--copy", default="overlap", choices=["overlap", "fork", "pipe", "gather", "carry", "lag"],
                    help="gather: one gather launch per layer after its selection, one stream; "
                         "overlap: gather of layer l on a side stream beside the attention of layer l-1; "
                         "carry: the host copy of layer l rides in layer l+1's scoring launch; "
                         "lag: cross-step pipeline, attention over the previous step's selection; "
                         "pipe: scorers back to back, each layer's selection, gather and attention on a side stream")
    ap.add_argument("--score-ctas", type=int, default=-1,
                    help="scorer CTAs per SM (0 = as many as fit; -1 = 2 with --copy pipe, else 0)")
    ap.add_argument("--scoring", default="maxdot", choices=["maxdot", "pooled"],
                    help="maxdot: scan of the full keys; pooled: scan of the min/max pooled keys")
    ap.add_argument("--workload", default="qwen3_8b_decode",
                    choices=["qwen3_8b_decode", "tiny", "llama31_8b_long", "qwen3_32b", "long_output"],
                    help="the timed configuration (--layers/--batch/--ctx apply to qwen3_8b_decode)")
    ap.add_argument("--ratio", default="0.01", help="fetch ratio of qwen3_32b: a number or 'all'")
    ap.add_argument("--phys-layers", type=int, default=0,
                    help="layers of distinct keys and pools in HBM (layer l uses l mod N; 0 = all, or 12 for "
                         "long_output, whose 36 layers of keys do not fit)")
    ap.add_argument("--no-pooled", action="store_true", help="skip the pooled-scoring variant")
    ap.add_argument("--score-kernel", default="tc", choices=["tc", "mma"],
                    help="max-dot scorer: TMA + tcgen05 with TMEM accumulators (default) or mma.sync from registers")
    ap.add_argument("--dynamic-scorer", action="store_true",
                    help="max-dot scoring with chunks from an atomic counter (oasis_score_blocks_dynamic)")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the cross-step pipeline and fused look-ahead attention measurements")
    ap.add_argument("--host-alloc", default="cuda", choices=["cuda", "thp", "thp_layers", "cuda_layers"],
                    help="host tier on transparent huge pages registered with CUDA, or from cudaHostAlloc; "
                         "*_layers: one allocation per host layer")
    ap.add_argument("--no-warm-host", action="store_true",
                    help="skip the one-time zero-copy read of the host tier before the pre-roll")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-hostlink", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-worker", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--ref-pairs", type=int, default=1,
                    help="(request, KV head) pairs the reference arm times per step")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the short measurements of the other synthetic configurations")
    ap.add_argument("--no-host-fit", action="store_true",
                    help="skip the headline re-measured with as many host-tier layers as fit")
    ap.add_argument("--cpu-heads", type=int, default=12,
                    help="(request, KV head) pairs the CPU baseline times (about 0.3 s each on the Qwen3-8B decode shape)")
    return ap.parse_args()


def workload(args):
    from sparse_decode_attention_oasis_gb300 import synthetic as syn

    if args.workload == "tiny":
        return syn.tiny()
    if args.workload == "llama31_8b_long":
        return syn.llama31_8b_long()
    if args.workload == "qwen3_32b":
        return syn.qwen3_32b(ratio=None if args.ratio == "all" else float(args.ratio))
    if args.workload == "long_output":
        return syn.long_output()
    return syn.qwen3_8b_decode(B=args.batch, L=args.layers, ctx=args.ctx)


def l2_note(w, scoring) -> str:
    per_block = 2 * w.d * 2 if scoring == "pooled" else w.bs * w.d * 2
    nbytes = sum(w.nb(b) for b in range(w.B)) * w.Hkv * per_block
    what = "pooled keys" if scoring == "pooled" else "keys"
    rel = "larger than" if nbytes > 129 * 2 ** 20 else "smaller than (the workload is launch-bound)"
    return f"inputs {rel} L2 ({nbytes / 2 ** 30:.2f} GiB of {what} per layer)"


def planned_layers(args, w):
    """(HBM layers, host-tier layers) the GPU arm plans for the workload (layer l uses
    HBM buffer l mod the first and host buffer l mod the second)."""
    l_phys = args.phys_layers or (min(12, w.L) if w.name == "long_output" else w.L)
    return l_phys, min(host_layers_for(w, args.host_layers), l_phys)


def config_dict(args, w, l_phys, l_host, score_ctas, world=1):
    """The `config` of the JSON line; the reference arm reports the same one."""
    return {"workload": workload_desc(w), "l2": l2_note(w, args.scoring),
            "scoring": args.scoring, "copy": args.copy, "score_ctas_per_sm": score_ctas,
            "host_tier_layers": l_host, "host_tier_aliased": l_host < w.L,
            "hbm_layers": l_phys, "hbm_layers_aliased": l_phys < w.L,
            "host_alloc": args.host_alloc,
            "dynamic_scorer": bool(getattr(args, "dynamic_scorer", False)),
            "score_kernel": getattr(args, "score_kernel", "tc"),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def workload_desc(w) -> str:
    ctx = f"{w.ctx[0]}" if min(w.ctx) == max(w.ctx) else f"{min(w.ctx)}-{max(w.ctx)} (+1 token per step)"
    hot = (f"{w.n_hot}-block hot set drifting through {w.n_pool} planted blocks/head (AR(1) rho_u {w.rho_u})"
           if w.hot_mode == "drift" else f"{w.n_hot} planted hot blocks/head")
    return (f"{w.name}: {w.L} layers, batch {w.B}, {w.Hq}/{w.Hkv} heads, d {w.d}, bf16, ctx {ctx}, "
            f"block {w.bs}, budget {w.Kb * w.bs} tokens ({w.Kb} blocks), {w.n_la} lookahead queries, "
            f"fetch cap {w.C} blocks/head/step, {hot}")


# --------------------------------------------------------------------------- CPU oracle timing
def cpu_sample(args, nheads: int, step: int = 0, warm: int = 0):
    """Time the oracle's layer-step on `nheads` sampled (request, KV head) pairs of layer 0,
    after `warm` untimed ones (first-call costs of the process).

    Returns seconds per head (the oracle as it stands, numpy float64/exact).
    """
    import numpy as np

    from oracle import oasis_ref as ref
    from sparse_decode_attention_oasis_gb300 import synthetic as syn

    w = workload(args)
    rng = np.random.default_rng(1234 + step)
    picks = [(int(rng.integers(w.B)), int(rng.integers(w.Hkv))) for _ in range(nheads + warm)]
    G = w.G
    total = 0.0
    for i, (b, h) in enumerate(picks):
        Kh, Vh = syn.head_kv(w, 0, b, h)
        qh, qlah = syn.head_queries(w, 0, b, h, step)
        sub = syn.Workload("sub", L=1, B=1, Hq=G, Hkv=1, ctx=[w.ctx[b]], Kb=w.Kb, C=w.C, n_la=w.n_la,
                           nb_max=w.nb_max)
        K = Kh[None, None]
        V = Vh[None, None]
        host = syn.host_tier_from_kv(sub, K, V)
        res = syn.initial_resident(w, 0, b, h)
        b2s = np.full((1, 1, w.nb_max), -1, np.int32)
        s2b = np.full((1, 1, w.P), -1, np.int32)
        lu = np.full((1, 1, w.P), -1, np.int32)
        for p, x in enumerate(res):
            s2b[0, 0, p] = x
            b2s[0, 0, x] = p
        kp, vp = syn.pools_from_tables(sub, host, s2b)
        q = qh[None]
        qla = qlah[None]
        t0 = time.perf_counter()
        ref.layer_step(K, qla, q, [w.ctx[b]], host, kp, vp, b2s, s2b, lu, w.Kb, w.C, step)
        if i >= warm:
            total += time.perf_counter() - t0
    return total / nheads


def _cpu_worker_sec_per_head(args, heads: int, threads: int) -> float:
    """Seconds per head of the oracle sample, in a fresh process with `threads` BLAS threads."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(threads)
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker", str(heads), "--layers", str(args.layers),
           "--batch", str(args.batch), "--ctx", str(args.ctx), "--workload", args.workload, "--ratio", str(args.ratio)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("cpu baseline worker failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])["sec_per_head"]


def cpu_baseline(args, heads: int):
    """Time the oracle sample with one BLAS thread and with all host cores; report
    the faster as `value` (`cores` = the threads it used) and both."""
    cores = os.cpu_count() or 1
    w = workload(args)
    n1, nall = 4 * heads, max(1, heads // 3)
    one = _cpu_worker_sec_per_head(args, n1, 1)
    allc = _cpu_worker_sec_per_head(args, nall, cores)
    best, used = (one, 1) if one <= allc else (allc, cores)
    per = w.B * w.Hkv
    return {"value": 1.0 / (best * per), "unit": UNIT, "cores": used, "kind": "oracle",
            "value_1_thread": 1.0 / (one * per), f"value_{cores}_threads": 1.0 / (allc * per),
            "sample": f"(request, KV head) pairs of layer 0 of the {w.name} workload, one full layer-step each "
                      f"(exact scoring, top-K, capped diff, LRU slots, fp64 attention), after one untimed pair: "
                      f"{n1} pairs with one BLAS thread ({n1 * one:.1f} s of oracle time), {nall} with {cores} "
                      f"({nall * allc:.1f} s); layer-step time = time per pair x {per} pairs; the oracle is numpy "
                      f"arithmetic driven by one Python thread"}


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"oasis_bench_clocks_rank{index}_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append(parts)
        if not rows:
            return None
        idxs = sorted(set(r[0] for r in rows))
        mine = [r for r in rows if r[0] == str(self.index)] if len(idxs) > 1 else rows
        sm = [float(r[1]) for r in mine if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in mine if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in mine:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(mine)}


# --------------------------------------------------------------------------- helpers
class GraphEvents:
    """Timing events recorded as nodes of a captured CUDA graph.

    cudaEventRecordWithFlags(..., cudaEventRecordExternal) during stream capture
    adds an event-record node; after a replay, cudaEventElapsedTime between two
    such events gives the device time between the nodes.
    """

    def __init__(self, n):
        import ctypes

        self.ct = ctypes
        lib = None
        for name in ("libcudart.so.13", "libcudart.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None:
            raise RuntimeError("libcudart not found")
        self.lib = lib
        lib.cudaEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        lib.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        lib.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p, ctypes.c_void_p]
        lib.cudaEventDestroy.argtypes = [ctypes.c_void_p]
        self.pool = []
        for _ in range(n):
            h = ctypes.c_void_p()
            if lib.cudaEventCreate(ctypes.byref(h)) != 0:
                raise RuntimeError("cudaEventCreate failed")
            self.pool.append(h)
        self.used = []
        self.names = {"score", "topk"}

    def __call__(self, name, stream):
        if name not in self.names:
            return
        h = self.pool[len(self.used)]
        if self.lib.cudaEventRecordWithFlags(h, self.ct.c_void_p(stream.cuda_stream), 1) != 0:
            raise RuntimeError("cudaEventRecordWithFlags failed")
        self.used.append((name, h))

    def durations(self):
        out = {"score": [], "topk": [], "diff": [], "assign": [], "copy": [], "gather": [], "attn": []}
        prev = None
        for name, h in self.used:
            if prev is not None and prev[0] in out:
                ms = self.ct.c_float()
                if self.lib.cudaEventElapsedTime(self.ct.byref(ms), prev[1], h) == 0:
                    out[prev[0]].append(ms.value)
            prev = (name, h)
        return out

    def close(self):
        for h in self.pool:
            self.lib.cudaEventDestroy(h)


class KernelMarks:
    """CUDA events recorded before/after each kernel of the decode step, per stream.

    ``names`` limits the marks recorded (the timed region records only the two
    around the scoring kernel, so the measurement barely perturbs the schedule).
    """

    def __init__(self, n, names=None):
        import torch

        self.pool = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        self.used = []
        self.names = names

    def __call__(self, name, stream):
        if self.names is not None and name not in self.names:
            return
        ev = self.pool[len(self.used)]
        ev.record(stream)
        self.used.append((name, stream, ev))

    def durations(self):
        """Per kernel name, the list of launch durations in ms (consecutive marks on one stream)."""
        out = {"score": [], "topk": [], "diff": [], "assign": [], "copy": [], "gather": [], "attn": []}
        last = {}
        for name, stream, ev in self.used:
            key = id(stream)
            if key in last and last[key][0] in out:
                out[last[key][0]].append(last[key][1].elapsed_time(ev))
            last[key] = (name, ev)
        return out


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(world: int, layers: int, steps: int, max_ms: float) -> float:
    """Whole-job layer-steps/s: every rank runs its own replica of the workload."""
    return world * layers * steps / (max_ms / 1000.0)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash(kernel: str = "tc") -> str:
    """Hash of a scoring kernel's code with comments and blank lines removed."""
    src = os.path.join(ROOT, "sparse_decode_attention_oasis_gb300", "csrc", KERNEL_SOURCE[kernel])
    code = []
    for line in open(src, encoding="utf-8"):
        line = line.split("//", 1)[0].strip()
        if line:
            code.append(line)
    return hashlib.sha256("\n".join(code).encode()).hexdigest()[:16]


def score_traffic_per_launch(kernel: str = "tc"):
    """ncu dram bytes of one score launch (full workload), if captured for this kernel source."""
    path = PROFILE_TRAFFIC[kernel]
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    if d.get("source_sha256_16") != kernel_source_hash(kernel):
        return None
    return d.get("bytes_per_launch_full")


def algorithmic_bytes(w, attended_per_head=None, scoring="maxdot"):
    """Algorithmic HBM bytes of one layer-step, split by kernel.

    The scorer reads every valid block's keys (4 KiB) or, with pooled scoring,
    its two pooled rows (512 B), plus the queries, and writes 8 B per block.
    Attention reads the K and V of the attended blocks: ``attended_per_head``
    (measured) or, if not given, the full budget Kb.
    """
    H = w.B * w.Hkv
    ctx_blocks = sum(w.nb(b) for b in range(w.B)) * w.Hkv
    per_block = 2 * w.d * 2 if scoring == "pooled" else w.bs * w.d * 2
    score = ctx_blocks * per_block + w.B * w.n_la * w.Hq * w.d * 2 + ctx_blocks * 8
    topk = ctx_blocks * 8 + H * (w.Kb + 1) * 4
    na = w.Kb if attended_per_head is None else attended_per_head
    attn = int(H * na * w.bs * w.d * 2 * 2) + w.B * w.Hq * w.d * (2 + 4)
    gather_hbm = H * w.C * w.bs * w.d * 2 * 2
    return {"score": score, "topk": topk, "attn": attn, "gather_hbm": gather_hbm,
            "total": score + topk + attn + gather_hbm}


def measure_agreement(st, qla_layers, q_layers, q_prev_layers):
    """Fraction of the exact top-K blocks of the true query that a predictor selects.

    Per layer, over all heads: the lookahead queries' top-K ("lookahead"), the
    previous step's true query ("previous_token"), and the exact blocks the
    attention actually reads (lookahead set and resident, "attended").  At K =
    Kb (the budget) and K = 20 (the top-20 of Figure 4).
    """
    import torch

    from sparse_decode_attention_oasis_gb300.engine import AgreementProbe

    out = {}
    for K in (st.shape.Kb, 20):
        probe = AgreementProbe(st, K=K)
        per_layer = {"lookahead": [], "previous_token": [], "attended": []}
        for l in range(st.w.L):
            c = probe.run(l, qla_layers[l], q_layers[l], q_prev_layers[l])
            la, prev = c["la"].sum(dim=(0, 1)).tolist(), c["prev"].sum(dim=(0, 1)).tolist()
            per_layer["lookahead"].append(la[0] / la[2])
            per_layer["attended"].append(la[1] / la[2])
            per_layer["previous_token"].append(prev[0] / prev[2])
        torch.cuda.synchronize()
        out[f"K{K}"] = {k: {"mean": round(sum(v) / len(v), 4), "min": round(min(v), 4)}
                        for k, v in per_layer.items()}
        del probe
    return out


def measure_hostlink(st, qla0, dev):
    """Host-link roofline of the gather: fetch-all into an emptied layer vs a pinned memcpy.

    Layer 0's resident set is emptied and the fetch cap raised to the budget, so
    the gather copies every selected block (Kb x 8 KiB per head) from the host
    tier; its CUDA-event time gives GB/s, compared with cudaMemcpy of 1 GiB from
    page-locked memory (the measured host-link peak on this machine).
    """
    import torch

    from sparse_decode_attention_oasis_gb300 import binding as B

    w, s, sc = st.w, st.shape, st.scratch
    main = torch.cuda.current_stream(dev)
    best = {"gather": None, "copy": None}
    for rep in range(6):
        which = "gather" if rep % 2 == 0 else "copy"
        st.b2sl[0].fill_(-1)
        st.s2bl[0].fill_(-1)
        st.lul[0].fill_(-1)
        B.oasis_score_blocks(s, st.Kl[0], st.ctx, qla0[0], sc.scores, sc.err, main)
        B.oasis_topk_select(s, sc.scores, st.Kl[0], qla0[0], st.ctx, sc.sel, sc.nsel, main)
        B.oasis_fetch_diff_capped(s, sc.scores, st.Kl[0], qla0[0], st.ctx, sc.sel, sc.nsel, st.b2sl[0], w.Kb,
                                  sc.fetch, sc.nfetch, main)
        if which == "copy":  # the table half first, untimed: the copy kernel alone is timed
            B.oasis_assign_slots(s, sc.sel, sc.nsel, sc.fetch, sc.nfetch, st.b2sl[0], st.s2bl[0], st.lul[0],
                                 st.step_dev, sc.err, main)
        torch.cuda.synchronize()
        nfetch = int(sc.nfetch.sum().item())
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main)
        if which == "gather":
            B.oasis_gather_h2d(s, st.hostl[0], sc.sel, sc.nsel, sc.fetch, sc.nfetch, st.b2sl[0], st.s2bl[0],
                               st.lul[0], st.step_dev, st.kpl[0], st.vpl[0], sc.err, main)
        else:
            B.oasis_copy_fetched(s, st.hostl[0], sc.fetch, sc.nfetch, st.b2sl[0], st.kpl[0], st.vpl[0], sc.err,
                                 main)
        e1.record(main)
        torch.cuda.synchronize()
        gbs = nfetch * 2 * w.bs * w.d * 2 / (e0.elapsed_time(e1) / 1000.0) / 1e9
        best[which] = gbs if best[which] is None else max(best[which], gbs)
    src = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    peak = 0.0
    for rep in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main)
        dst.copy_(src, non_blocking=True)
        e1.record(main)
        torch.cuda.synchronize()
        peak = max(peak, (1 << 30) / (e0.elapsed_time(e1) / 1000.0) / 1e9)
    del src, dst
    return {"kernel": "gather_h2d (fetch-all, one layer)", "bound": "host link", "achieved": best["gather"],
            "peak": peak, "peak_kind": "measured: pinned cudaMemcpy H2D of 1 GiB", "unit": "GB/s",
            "frac": best["gather"] / peak, "bytes_per_launch": nfetch * 2 * w.bs * w.d * 2,
            "copy_fetched_achieved": best["copy"], "copy_fetched_frac": best["copy"] / peak}


# --------------------------------------------------------------------------- reference arm
def run_reference(args, rank):
    """The CPU oracle as the reference arm: each timed step runs one full oracle
    layer-step on `--ref-pairs` sampled (request, KV head) pairs of layer 0; the
    layer-steps/s of the whole workload is extrapolated from the time per pair."""
    if rank != 0:
        return
    w = workload(args)
    pairs = max(1, args.ref_pairs)
    per_step = []
    t_all = time.perf_counter()
    for s in range(args.warmup + args.steps):
        t = cpu_sample(args, pairs, step=s)
        if s >= args.warmup:
            per_step.append(t * pairs)
    wall = time.perf_counter() - t_all
    sec_per_head = sum(per_step) / (len(per_step) * pairs)
    value = 1.0 / (sec_per_head * w.B * w.Hkv)
    try:
        cores = int(os.environ.get("OPENBLAS_NUM_THREADS", ""))
    except ValueError:
        cores = os.cpu_count() or 1
    l_phys, l_host = planned_layers(args, w)
    score_ctas = args.score_ctas if args.score_ctas >= 0 else (2 if args.copy == "pipe" else 0)
    heads = w.B * w.Hkv
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup,
            # the time each timed step actually took (the sample), not the extrapolation
            "ms_per_step": 1000.0 * sum(per_step) / len(per_step),
            "extrapolated": True, "pairs_per_step": pairs, "pairs_timed": pairs * args.steps,
            "ms_per_step_extrapolated": 1000.0 * w.L / value,
            "run_wall_s": round(wall, 2),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(args, w, l_phys, l_host, score_ctas),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{pairs} (request, KV head) pair(s) of layer 0 per timed step, one full "
                                       f"oracle layer-step each; layer-steps/s extrapolated from the time per pair "
                                       f"x {heads} pairs per layer-step; cores = BLAS threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm
def host_layers_for(w, requested: int) -> int:
    """Layers of distinct host-tier data (layer l reads buffer l mod this).  A
    request of 0 takes as many as 60% of the available host memory holds."""
    per_layer = w.B * w.Hkv * w.nb_max * 2 * w.bs * w.d * 2
    avail = None
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                avail = int(line.split()[1]) * 1024
    except OSError:
        pass
    fit = w.L if avail is None else max(1, int(0.6 * avail // per_layer))
    return max(1, min(w.L, fit, requested or w.L))


def launches_per_step(st, copy):
    """Kernels of this library one decode step launches (the graph's own LRU-clock
    increment is a PyTorch kernel and is not counted)."""
    s = st.shape
    G = s.Hq // s.Hkv
    nsplit = st.scratch.ws_bytes // (s.B * s.Hkv * G * (s.d + 2) * 4)
    attn = 1 if nsplit <= 1 else 2  # split-K partials, then the combine kernel
    select = 1 if st.fused_select else 2  # top-K and diff in one launch, or two
    per_layer = 1 + select + 1 + attn  # score (maybe carrying a copy), selection, gather or assign, attention
    return st.w.L * per_layer + (1 if copy == "carry" else 0)


def make_state(args, w, dev, l_phys, l_host, scoring="maxdot"):
    """A filled, warmed DecodeState; the host tier shrinks if page-locked memory runs out."""
    import torch

    from sparse_decode_attention_oasis_gb300.engine import DecodeState

    while True:
        try:
            st = DecodeState(w, device=dev, l_phys=l_phys, l_host=l_host, scoring=scoring,
                             host_alloc=args.host_alloc)
            break
        except RuntimeError:
            if l_host <= 2:
                raise
            l_host = max(2, l_host // 2)
            torch.cuda.empty_cache()
    st.dynamic_scorer = args.dynamic_scorer
    st.fill_synthetic()
    st.warm_host_tier()
    return st


def device_queries(w, dev, nsteps):
    """q [n][L][B][Hq][d] and q_la [n][L][B][n_la][Hq][d] (bf16, device) of decode steps 0..n-1."""
    import torch

    from sparse_decode_attention_oasis_gb300 import synthetic as syn

    qs = [syn.QueryStreamTorch(w, l, dev) for l in range(w.L)]
    q_dev = torch.empty((nsteps, w.L, w.B, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    qla_dev = torch.empty((nsteps, w.L, w.B, w.n_la, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    for s_ in range(nsteps):
        for l in range(w.L):
            qb, qlab = qs[l].next()
            q_dev[s_, l].copy_(qb)
            qla_dev[s_, l].copy_(qlab)
    return q_dev, qla_dev


def token_appends(w, dev, n=16):
    """(k_new, v_new) pairs, bf16 [L][B][Hkv][d], for workloads whose context grows."""
    import torch

    if w.name != "long_output":
        return None
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    k_app = torch.randn((n, w.L, w.B, w.Hkv, w.d), generator=gen, device=dev).to(torch.bfloat16)
    v_app = torch.randn((n, w.L, w.B, w.Hkv, w.d), generator=gen, device=dev).to(torch.bfloat16)
    return [(k_app[i], v_app[i]) for i in range(n)]


def exact_topk_turnover(st, q_steps, K=64, layer=0):
    """Mean fraction of the exact top-K blocks of the true queries (the a1 score of
    the true query, then top-K) that change from one decode step to the next, over
    all heads of `layer`; q_steps: that layer's true queries of consecutive steps."""
    import torch

    from sparse_decode_attention_oasis_gb300 import binding as B
    from sparse_decode_attention_oasis_gb300.engine import AgreementProbe

    probe = AgreementProbe(st, K=K)
    prev, tos = None, []
    counts = torch.empty((st.shape.B, st.shape.Hkv, 3), dtype=torch.int32, device=st.device)
    for q in q_steps:
        probe._topk(probe.shape1, layer, q, "exact", torch.cuda.current_stream(st.device))
        cur = (probe.sel["exact"].clone(), probe.nsel["exact"].clone())
        if prev is not None:
            B.oasis_set_agreement(probe.shape, cur[0], cur[1], prev[0], prev[1], None, counts, probe.err)
            c = counts.sum(dim=(0, 1)).tolist()
            tos.append(1.0 - c[0] / c[2])
        prev = cur
    torch.cuda.synchronize(st.device)
    return sum(tos) / len(tos) if tos else None


def light_measure(args, st, q_dev, qla_dev, start, preroll, steps, appends, world, dev):
    """Eager pre-roll steps, then `steps` timed steps as one graph (event nodes around
    the scorer), then two eager steps that count attended and fetched blocks."""
    import torch

    w = st.w
    L = w.L
    main = torch.cuda.current_stream(dev)
    n_in = q_dev.shape[0]

    def eager(s_, **kw):
        if appends is not None:
            st.append_step(*appends[s_ % len(appends)], stream=main)
        k = s_ % n_in
        st.decode_step(s_, qla_dev[k], q_dev[k], main=main, side=main, copy=args.copy, **kw)

    for k in range(preroll):
        eager(start + k)
    torch.cuda.synchronize()
    first = start + preroll
    marks = GraphEvents(L * steps * 3 + 16)
    marks.names = {"score", "topk", "end"}
    ts_first = first % n_in
    if ts_first + steps > n_in:
        ts_first = 0
    # the graph's LRU clock starts at `first`; its inputs are steps ts_first.. of the query buffers
    ms, clk = _timed_graph_at(st, first, ts_first, q_dev, qla_dev, steps, args.copy, appends, world, dev, marks)
    durs = marks.durations()
    score_ms, topk_ms = durs["score"], durs["topk"]
    marks.close()
    attended = torch.zeros((), dtype=torch.int64, device=dev)
    fetched = torch.zeros((), dtype=torch.int64, device=dev)
    nxt = first + steps
    for k in range(2):
        eager(nxt + k, count=attended, fetched=fetched)
    torch.cuda.synchronize()
    err = st.error_word()
    att = float(attended.item()) / (2 * L * w.B * w.Hkv)
    fetched_step = float(fetched.item()) / 2 * 2 * w.bs * w.d * 2
    ab = algorithmic_bytes(w, att, st.scoring)
    peak = measured_peaks()[0]
    path = ab["total"] * L * steps / (ms / 1000.0) / 1e9
    sc_avg = sum(score_ms) / len(score_ms)
    return {"value": aggregate_value(world, L, steps, ms), "unit": UNIT, "steps": steps,
            "ms_per_step": ms / steps, "path_hbm_gbs": path, "path_hbm_frac": path / peak,
            "scorer_us": round(1000.0 * sc_avg, 2),
            "topk_diff_us_p50": round(1000.0 * statistics.median(topk_ms), 2) if topk_ms else None,
            "scorer_frac": ab["score"] / (sc_avg / 1000.0) / 1e9 / peak,
            "attended_blocks_per_head": round(att, 2), "fetched_bytes_per_step": int(fetched_step),
            "fetched_gbs": fetched_step / (ms / steps / 1000.0) / 1e9,
            "clocks": clk, "device_error_word": err}, nxt + 2


def _timed_graph_at(st, lru_first, in_first, q_dev, qla_dev, steps, copy, appends, world, dev, marks):
    import torch

    from sparse_decode_attention_oasis_gb300.engine import StepGraph

    ts = range(in_first, in_first + steps)
    outs = [torch.empty((st.w.L, st.w.B, st.w.Hq, st.w.d), dtype=torch.float32, device=dev) for _ in range(2)]
    app = None if appends is None else [appends[s_ % len(appends)] for s_ in ts]
    g = StepGraph(st, lru_first, [qla_dev[s_] for s_ in ts], [q_dev[s_] for s_ in ts],
                  [outs[k % 2] for k in range(steps)], mark=marks, copy=copy, appends=app)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index or 0)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    with torch.cuda.stream(g.stream):
        e0.record(g.stream)
        g.replay()
        e1.record(g.stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    del g
    return reduce_max(e0.elapsed_time(e1), world, dev), clk


def measure_other_configs(args, dev, world):
    """Short measurements of the other synthetic configurations, each on its own state
    (layers aliased in HBM and in the host tier to bound set-up time; every aliased
    buffer is far larger than L2): Llama-3.1-8B 128K, the Qwen3-32B fetch-ratio sweep
    and long-output decode with its drifting hot set."""
    import gc

    import torch

    from sparse_decode_attention_oasis_gb300 import synthetic as syn

    out = {}
    steps, pre = 8, 8
    plans = [("llama31_8b_long", syn.llama31_8b_long(), 8, 4, None),
             ("qwen3_32b_ratio_sweep", syn.qwen3_32b(ratio=0.01), 8, 4, [0.01, 0.02, 0.05, 0.10, 0.20, None]),
             ("long_output", syn.long_output(), 6, 4, None)]
    for name, w, l_phys, l_host, ratios in plans:
        t0 = time.time()
        try:
            st = make_state(args, w, dev, l_phys, min(l_host, l_phys))
            n_in = pre + steps + 2
            q_dev, qla_dev = device_queries(w, dev, n_in)
            appends = token_appends(w, dev)
            entry = {"workload": workload_desc(w), "hbm_layers": st.L_phys, "host_tier_layers": st.L_host,
                     "aliased": True, "setup_s": round(time.time() - t0, 1)}
            if name == "long_output":
                heads = [(b, h) for b in range(0, w.B, 8) for h in range(w.Hkv)]
                entry["hot_set_turnover"] = round(syn.hot_set_turnover(w, 0, 64, heads=heads), 4)
                entry["exact_top64_turnover"] = round(
                    exact_topk_turnover(st, [q_dev[k, 0] for k in range(8)], K=64), 4)
            runs = {}
            s0 = 0
            for ratio in (ratios or ["cfg"]):
                if ratio != "cfg":
                    w.C = syn.fetch_cap_from_ratio(ratio, w.Kb)
                key = "cfg" if ratio == "cfg" else ("fetch_all" if ratio is None else f"ratio_{ratio}")
                r, s0 = light_measure(args, st, q_dev, qla_dev, s0, pre, steps, appends, world, dev)
                r["fetch_cap"] = w.C
                runs[key] = r
            entry.update(runs["cfg"] if list(runs) == ["cfg"] else {"ratios": runs})
            out[name] = entry
        except Exception as e:  # one configuration failing does not lose the others
            out[name] = {"unavailable": f"{type(e).__name__}: {str(e)[-300:]}"}
        finally:
            st = q_dev = qla_dev = appends = None
            gc.collect()
            torch.cuda.empty_cache()
            empty = getattr(torch._C, "_host_emptyCache", None)
            if empty is not None:
                empty()
    return out


def measure_host_fit(args, st, q_dev, qla_dev, start, world, dev):
    """The headline workload again with as many host-tier layers as 60% of the
    available host memory holds (less aliasing of host data, more page-locked memory)."""
    fit = host_layers_for(st.w, 0)
    if fit <= st.L_host:
        return {"host_tier_layers": st.L_host, "skipped": "no more host layers fit than the headline uses"}
    t0 = time.time()
    while True:
        try:
            st.rebuild_host_tier(fit)
            break
        except RuntimeError:
            if fit <= st.L_host:
                raise
            fit = max(st.L_host, fit * 3 // 4)
    rebuild = time.time() - t0
    t1 = time.time()
    st.warm_host_tier()
    warm = time.time() - t1
    r, _ = light_measure(args, st, q_dev, qla_dev, start, 8, args.steps, None, world, dev)
    r.update({"host_tier_layers": st.L_host, "host_tier_aliased": st.L_host < st.w.L,
              "rebuild_s": round(rebuild, 1), "host_tier_warm_s": round(warm, 2)})
    return r


def measure_spans(st, first_step, qla_steps, q_steps, out_dev, copy, appends, steps=3):
    """Kernel spans of `steps` decode steps captured as one CUDA graph with the span
    trace on (no event nodes between kernels), replayed once."""
    import torch

    from sparse_decode_attention_oasis_gb300.engine import KernelTrace, StepGraph

    L = st.w.L
    tr = KernelTrace(capacity=max(64, 2 * L * steps), device=st.device)
    tr.start()
    try:
        g = StepGraph(st, first_step, qla_steps, q_steps, [out_dev] * steps, copy=copy, appends=appends)
    finally:
        tr.stop()
    with torch.cuda.stream(g.stream):
        g.replay()
    torch.cuda.synchronize()
    sp = tr.spans()
    del g, tr
    torch.cuda.synchronize()
    return sp


def summarize_spans(sp, L, steps, copy, gather_bytes=None, link_gbs=None):
    """Per-kind span statistics (us) and, for the overlap order, the gaps of the
    critical path between consecutive kernels of a layer."""
    import numpy as np

    def stats(x):
        x = np.asarray(x, dtype=np.float64)
        if x.size == 0:
            return None
        return {"p50": round(float(np.median(x)), 2), "mean": round(float(x.mean()), 2),
                "max": round(float(x.max()), 2), "n": int(x.size)}

    out = {"source": f"per-launch spans (earliest block start to latest block end, %globaltimer) of {steps} "
                     f"decode steps captured as one CUDA graph with the span trace on and no event nodes, "
                     f"replayed once", "steps": steps, "kernel_us": {}}
    for name, (a, b) in sp.items():
        if len(a):
            out["kernel_us"][name] = stats((b - a) / 1000.0)
    score_name = "score" if len(sp["score"][0]) else "score_pooled"
    S0, S1 = (x / 1000.0 for x in sp[score_name])
    if len(S0) > 1:
        out["layer_period_us"] = stats(np.diff(S0))
    n = L * steps
    if copy == "overlap" and all(len(sp[k][0]) == n for k in (score_name, "select", "gather", "attn")):
        T0, T1 = (x / 1000.0 for x in sp["select"])
        G0, G1 = (x / 1000.0 for x in sp["gather"])
        A0, A1 = (x / 1000.0 for x in sp["attn"])
        prev = [i for i in range(n) if i % L]  # attention of layer l-1 runs beside the gather of layer l
        nxt = range(n - 1)
        out["gaps_us"] = {
            "score_end_to_select_start": stats(T0 - S1),
            "select_end_to_gather_start": stats(G0 - T1),
            "select_end_to_attn_prev_start": stats([A0[i - 1] - T1[i] for i in prev]),
            "gather_end_to_next_score_start": stats([S0[i + 1] - G1[i] for i in nxt]),
            "next_score_start_after_gather_and_attn_prev": stats(
                [S0[i + 1] - max(G1[i], A1[i - 1]) for i in nxt if i % L]),
        }
    if gather_bytes and len(sp["gather"][0]):
        g_us = (sp["gather"][1] - sp["gather"][0]) / 1000.0
        gbs = gather_bytes / (g_us * 1e3)
        out["decode_gather_gbs"] = stats(gbs)
        if link_gbs:
            out["decode_gather_link_frac_p50"] = round(float(np.median(gbs)) / link_gbs, 4)
            out["decode_gather_link_frac_of_mean_time"] = round(gather_bytes / (float(g_us.mean()) * 1e3) / link_gbs, 4)
    return out


def run_gpu(args, rank, world, local_rank):
    import numpy as np
    import torch

    from sparse_decode_attention_oasis_gb300 import build as _build
    from sparse_decode_attention_oasis_gb300 import synthetic as syn
    from sparse_decode_attention_oasis_gb300.engine import DecodeState

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the path has no CPU fallback)")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if local_rank == 0:
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    w = workload(args)
    L = w.L
    l_phys, l_host = planned_layers(args, w)
    t0 = time.time()
    while True:
        try:
            st = DecodeState(w, device=dev, l_phys=l_phys, l_host=l_host, scoring=args.scoring,
                             host_alloc=args.host_alloc)
            break
        except RuntimeError:
            if l_host <= 2:
                raise
            l_host = max(2, l_host // 2)
            torch.cuda.empty_cache()
    alloc_s = time.time() - t0
    st.dynamic_scorer = args.dynamic_scorer
    st.fill_synthetic()
    torch.cuda.synchronize()
    gen_s = time.time() - t0
    warm_s = None
    if not args.no_warm_host:
        t1 = time.time()
        st.warm_host_tier()
        warm_s = time.time() - t1

    pre = args.preroll
    nsteps = pre + args.warmup + args.steps
    qs = [syn.QueryStreamTorch(w, l, dev) for l in range(L)]
    q_dev = torch.empty((nsteps, L, w.B, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    qla_dev = torch.empty((nsteps, L, w.B, w.n_la, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    for s in range(nsteps):
        for l in range(L):
            qb, qlab = qs[l].next()
            q_dev[s, l].copy_(qb)
            qla_dev[s, l].copy_(qlab)
    first = pre + args.warmup
    # the growing context of long-output decode: one new token per request and layer per step
    appends = None
    if args.workload == "long_output":
        gen = torch.Generator(device=dev)
        gen.manual_seed(7)
        n_app = 16
        k_app = torch.randn((n_app, L, w.B, w.Hkv, w.d), generator=gen, device=dev).to(torch.bfloat16)
        v_app = torch.randn((n_app, L, w.B, w.Hkv, w.d), generator=gen, device=dev).to(torch.bfloat16)
        appends = [(k_app[i], v_app[i]) for i in range(n_app)]

    def app(s_):
        return None if appends is None else appends[s_ % len(appends)]

    def app_list(steps_):
        return None if appends is None else [app(s_) for s_ in steps_]

    def eager_step(s_, qla, q, **kw):
        if appends is not None:
            st.append_step(*app(s_), stream=main)
        st.decode_step(s_, qla, q, **kw)

    q_host = q_dev[first:].cpu().pin_memory()      # inputs of the timed steps, for the end-to-end pass
    qla_host = qla_dev[first:].cpu().pin_memory()
    torch.cuda.synchronize()

    score_ctas = args.score_ctas if args.score_ctas >= 0 else (2 if args.copy == "pipe" else 0)
    from sparse_decode_attention_oasis_gb300 import binding as _B

    _B.oasis_set_option(_B.OPT_SCORE_CTAS_PER_SM, score_ctas)
    _B.oasis_set_option(_B.OPT_SCORE_KERNEL, _B.SCORE_KERNEL_TC if args.score_kernel == "tc" else _B.SCORE_KERNEL_MMA)
    main = torch.cuda.current_stream(dev)
    side = main  # the overlap mode makes its own side stream; the others run on one stream
    out_dev = torch.empty((L, w.B, w.Hq, w.d), dtype=torch.float32, device=dev)

    def step(s, mark=None, qla=None, q=None):
        eager_step(s, qla if qla is not None else qla_dev[s], q if q is not None else q_dev[s],
                       out_layers=out_dev, main=main, side=side, mark=mark, copy=args.copy)

    for s in range(pre + args.warmup):
        step(s)
    torch.cuda.synchronize()
    errw = st.error_word()

    # the timed steps, captured once as a CUDA graph (inputs already in HBM, the LRU
    # clock advanced by the graph); events around every scoring launch are graph nodes
    from sparse_decode_attention_oasis_gb300.engine import StepGraph

    marks = GraphEvents(L * args.steps * 2 + 16)
    out_steps = [torch.empty((L, w.B, w.Hq, w.d), dtype=torch.float32, device=dev) for _ in range(2)]
    ts = range(first, first + args.steps)
    graph = StepGraph(st, first, [qla_dev[s] for s in ts], [q_dev[s] for s in ts],
                      [out_steps[k % 2] for k in range(args.steps)], mark=marks, copy=args.copy,
                      appends=app_list(ts))
    gstream = graph.stream
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(gstream):
        ev0.record(gstream)
        graph.replay()
        ev1.record(gstream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    ms = reduce_max(ev0.elapsed_time(ev1), world, dev)
    score_ms = marks.durations()["score"]
    errw |= st.error_word()
    del graph
    torch.cuda.synchronize()
    marks.close()

    # the same kind of steps issued eagerly from Python (one stream), timed as a whole
    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nxt = first + args.steps
    e_a.record(main)
    for k in range(3):
        s_k = first + k % args.steps
        eager_step(nxt + k, qla_dev[s_k], q_dev[s_k], out_layers=out_dev, main=main, side=main,
                       copy=args.copy)
    e_b.record(main)
    torch.cuda.synchronize()
    eager_ms = e_a.elapsed_time(e_b) / 3
    nxt += 3

    # per-kernel device time: one decode step captured with an event node around
    # every kernel (no host in the loop), replayed 3 times
    iso = GraphEvents(L * 10 + 16)
    iso.names = {"score", "topk", "diff", "end", "assign", "copy", "gather", "gather_end", "attn", "attn_end"}
    g_iso = StepGraph(st, nxt, [qla_dev[first]], [q_dev[first]], [out_dev], mark=iso, copy=args.copy,
                      appends=app_list([nxt]))
    kernel_ms = {k: [] for k in ("score", "topk", "diff", "assign", "copy", "gather", "attn")}
    for k in range(3):
        with torch.cuda.stream(g_iso.stream):
            g_iso.replay()
        torch.cuda.synchronize()
        for name, v in iso.durations().items():
            kernel_ms[name] += v
    nxt += 3
    del g_iso
    torch.cuda.synchronize()
    iso.close()
    # the same launch order without event nodes: kernel spans from the span trace
    span_steps = 3
    span_ts = [first + k % args.steps for k in range(span_steps)]
    spans_raw = measure_spans(st, nxt, [qla_dev[s_] for s_ in span_ts], [q_dev[s_] for s_ in span_ts], out_dev,
                              args.copy, app_list([nxt + k for k in range(span_steps)]), steps=span_steps)
    nxt += span_steps
    # attended blocks (selected and resident) per head, counted on eager steps
    attended = torch.zeros((), dtype=torch.int64, device=dev)
    fetched = torch.zeros((), dtype=torch.int64, device=dev)
    for k in range(2):
        s_k = first + k % args.steps
        eager_step(nxt + k, qla_dev[s_k], q_dev[s_k], out_layers=out_dev, main=main, side=main,
                   count=attended, fetched=fetched, copy=args.copy)
    torch.cuda.synchronize()
    nxt += 2
    attended_per_head = float(attended.item()) / (2 * L * w.B * w.Hkv)
    fetched_bytes_per_step = float(fetched.item()) / 2 * 2 * w.bs * w.d * 2

    # prediction agreement per layer (Figure 6 / Figure 4 analogue), one step, untimed
    agreement = measure_agreement(st, qla_dev[first], q_dev[first], q_dev[first - 1])

    # end to end: every step copies its queries from pinned host memory into the
    # graph's input buffers, replays the one-step graph and copies the outputs back
    e2e = None
    if not args.no_e2e:
        q_in = torch.empty_like(q_dev[0])
        qla_in = torch.empty_like(qla_dev[0])
        out_e2e = torch.empty((L, w.B, w.Hq, w.d), dtype=torch.float32, device=dev)
        out_host = torch.empty((L, w.B, w.Hq, w.d), dtype=torch.float32, pin_memory=True)
        g1 = StepGraph(st, nxt, [qla_in], [q_in], [out_e2e], copy=args.copy, appends=app_list([nxt]))
        nrep = args.steps
        # one untimed read of every staged input (a serving loop reuses warm pinned buffers)
        with torch.cuda.stream(g1.stream):
            for k in range(args.steps):
                q_in.copy_(q_host[k], non_blocking=True)
                qla_in.copy_(qla_host[k], non_blocking=True)
            out_host.copy_(out_e2e, non_blocking=True)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nrep)]
        t0 = time.perf_counter()
        with torch.cuda.stream(g1.stream):
            for k in range(nrep):
                ev[k][0].record(g1.stream)
                q_in.copy_(q_host[k % args.steps], non_blocking=True)
                qla_in.copy_(qla_host[k % args.steps], non_blocking=True)
                ev[k][1].record(g1.stream)
                g1.replay()
                ev[k][2].record(g1.stream)
                out_host.copy_(out_e2e, non_blocking=True)
                ev[k][3].record(g1.stream)
                g1.stream.synchronize()
        e2e_s = reduce_max(time.perf_counter() - t0, world, dev)
        bi = q_in.numel() * 2 + qla_in.numel() * 2
        bo = out_host.numel() * 4
        part = [sum(e[i].elapsed_time(e[i + 1]) for e in ev) / nrep for i in range(3)]
        e2e = {"value": aggregate_value(world, L, nrep, 1000.0 * e2e_s), "unit": UNIT, "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": bo, "ms_per_step": 1000.0 * e2e_s / nrep,
               "device_ms": {"h2d": round(part[0], 3), "step": round(part[1], 3), "d2h": round(part[2], 3)}}
        nxt += nrep

    # the pooled-key scoring path (f1) on the same state: a short eager pre-roll under
    # the new scorer, then the same timed steps captured as one graph
    pooled = None
    if args.scoring == "maxdot" and not args.no_pooled:
        st.set_scoring("pooled")
        for k in range(8):
            s_k = first + k % args.steps
            eager_step(nxt + k, qla_dev[s_k], q_dev[s_k], out_layers=out_dev, main=main, side=main,
                           copy=args.copy)
        nxt += 8
        pmarks = GraphEvents(L * args.steps * 2 + 16)
        pgraph = StepGraph(st, nxt, [qla_dev[s] for s in ts], [q_dev[s] for s in ts],
                           [out_steps[k % 2] for k in range(args.steps)], mark=pmarks, copy=args.copy,
                           appends=app_list(ts))
        nxt += args.steps
        torch.cuda.synchronize()
        pa, pb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(pgraph.stream):
            pa.record(pgraph.stream)
            pgraph.replay()
            pb.record(pgraph.stream)
        torch.cuda.synchronize()
        pms = reduce_max(pa.elapsed_time(pb), world, dev)
        pscore = pmarks.durations()["score"]
        del pgraph
        torch.cuda.synchronize()
        pmarks.close()
        pab = algorithmic_bytes(w, attended_per_head, "pooled")
        pavg = sum(pscore) / len(pscore)
        pach = pab["score"] / (pavg / 1000.0) / 1e9
        ppath = pab["total"] * L * args.steps / (pms / 1000.0) / 1e9
        pooled = {"value": aggregate_value(world, L, args.steps, pms), "unit": UNIT,
                  "ms_per_step": pms / args.steps,
                  "path_hbm_gbs": ppath, "path_hbm_frac": ppath / measured_peaks()[0],
                  "path_bytes_per_layer_step": pab,
                  "score_kernel": {"kernel": "score_pooled_kernel", "avg_launch_ms": pavg,
                                   "bytes_per_launch": pab["score"], "achieved_gbs": pach,
                                   "frac": pach / measured_peaks()[0]}}
        errw |= st.error_word()
        st.set_scoring("maxdot")

    # the cross-step pipeline (f4): attention over the previous step's selection;
    # a short eager pre-roll in that order, then the same timed steps as one graph
    lag = None
    if not args.no_variants:
        for k in range(4):
            s_k = first + k % args.steps
            eager_step(nxt + k, qla_dev[s_k], q_dev[s_k], out_layers=out_dev, main=main, side=main,
                           copy="lag")
        nxt += 4
        lgraph = StepGraph(st, nxt, [qla_dev[s] for s in ts], [q_dev[s] for s in ts],
                           [out_steps[k % 2] for k in range(args.steps)], copy="lag", appends=app_list(ts))
        nxt += args.steps
        torch.cuda.synchronize()
        la_, lb_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(lgraph.stream):
            la_.record(lgraph.stream)
            lgraph.replay()
            lb_.record(lgraph.stream)
        torch.cuda.synchronize()
        lms = reduce_max(la_.elapsed_time(lb_), world, dev)
        del lgraph
        lag = {"value": aggregate_value(world, L, args.steps, lms), "unit": UNIT, "ms_per_step": lms / args.steps}
        errw |= st.error_word()

    # fused look-ahead attention (f2): one launch per layer for the true and the n_la
    # draft queries over the same resident blocks, against the plain attention launch
    la_attn = None
    if not args.no_variants:
        sc = st.scratch
        out_la = torch.empty((w.B, w.n_la, w.Hq, w.d), dtype=torch.float32, device=dev)
        times = {"plain": [], "fused": []}
        for rep in range(4):
            for kind in ("plain", "fused"):
                e0_, e1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0_.record(main)
                for l in range(L):
                    if kind == "plain":
                        st._attend(l, q_dev[first][l], sc, main, out_dev[l])
                    else:
                        st.attend_lookahead(l, q_dev[first][l], qla_dev[first][l], sc, out_dev[l], out_la, main)
                e1_.record(main)
                torch.cuda.synchronize()
                if rep:
                    times[kind].append(e0_.elapsed_time(e1_) * 1000.0 / L)
        la_attn = {"plain_us_per_layer": round(sum(times["plain"]) / len(times["plain"]), 2),
                   "fused_us_per_layer": round(sum(times["fused"]) / len(times["fused"]), 2),
                   "rows_per_kv_head": {"plain": w.G, "fused": (1 + w.n_la) * w.G}}

    hostlink = measure_hostlink(st, qla_dev[first], dev) if not args.no_hostlink else None
    if hostlink is not None and kernel_ms["gather"]:
        # the gather of the timed decode step itself: fetched bytes per layer over its launch time
        per_layer = fetched_bytes_per_step / L
        g_mean = sum(kernel_ms["gather"]) / len(kernel_ms["gather"])
        g_p50 = statistics.median(kernel_ms["gather"])
        hostlink["decode_gather"] = {
            "bytes_per_launch": int(per_layer), "mean_us": round(1000.0 * g_mean, 2),
            "p50_us": round(1000.0 * g_p50, 2), "max_us": round(1000.0 * max(kernel_ms["gather"]), 2),
            "achieved_gbs_mean": per_layer / (g_mean / 1000.0) / 1e9,
            "achieved_gbs_p50": per_layer / (g_p50 / 1000.0) / 1e9,
            "frac_mean": per_layer / (g_mean / 1000.0) / 1e9 / hostlink["peak"],
            "frac_p50": per_layer / (g_p50 / 1000.0) / 1e9 / hostlink["peak"],
            "source": "gather launches of the per-kernel timing graph (3 replays x layers)"}
    kernel_spans = summarize_spans(spans_raw, L, span_steps, args.copy, gather_bytes=fetched_bytes_per_step / L,
                                   link_gbs=hostlink["peak"] if hostlink else None)
    if hostlink is not None and "decode_gather" in hostlink and "gather" in kernel_spans["kernel_us"]:
        gs = kernel_spans["kernel_us"]["gather"]
        per_layer = fetched_bytes_per_step / L
        hostlink["decode_gather"].update({
            "span_p50_us": gs["p50"], "span_mean_us": gs["mean"],
            "span_frac_p50": per_layer / (gs["p50"] * 1e3) / hostlink["peak"],
            "span_frac_mean": per_layer / (gs["mean"] * 1e3) / hostlink["peak"],
            "span_source": "gather spans of the traced graph (no event nodes)"})

    launches = launches_per_step(st, args.copy)
    # exact top-64 turnover of the true queries from one step to the next (layer 0)
    top64_turnover = exact_topk_turnover(st, [q_dev[first + k, 0] for k in range(min(8, args.steps))], K=64)

    # the headline workload again with more host-tier layers, then the other configurations
    host_fit = None
    if world == 1 and not args.no_host_fit and args.workload == "qwen3_8b_decode":
        try:
            host_fit = measure_host_fit(args, st, q_dev, qla_dev, nxt, world, dev)
        except Exception as e:
            host_fit = {"unavailable": f"{type(e).__name__}: {str(e)[-300:]}"}
    errw |= st.error_word()
    other = None
    if world == 1 and not args.no_other_configs and args.workload == "qwen3_8b_decode":
        import gc

        st = graph = g1 = None
        q_dev = qla_dev = q_host = qla_host = None
        gc.collect()
        torch.cuda.empty_cache()
        other = measure_other_configs(args, dev, world)

    if rank != 0:
        return
    ab = algorithmic_bytes(w, attended_per_head, args.scoring)
    peak, peak_kind = measured_peaks()
    score_avg_ms = sum(score_ms) / len(score_ms)
    achieved = ab["score"] / (score_avg_ms / 1000.0) / 1e9
    value = aggregate_value(world, L, args.steps, ms)
    path_gbs = ab["total"] * L * args.steps / (ms / 1000.0) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(args, w, l_phys, l_host, score_ctas, world),
        "path_hbm_gbs": path_gbs, "path_hbm_frac": path_gbs / peak,
        "roofline": {"kernel": "score_blocks_pooled" if args.scoring == "pooled" else
                     ("score_blocks_tc" if args.score_kernel == "tc" else "score_blocks"),
                     "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": score_traffic_per_launch(args.score_kernel) if args.scoring == "maxdot" else None,
                     "bytes_per_launch": ab["score"],
                     "avg_launch_ms": score_avg_ms},
        "kernel_times_source": "a separate one-step CUDA graph of the same launch order with an event-record "
                               "node around every kernel, replayed 3 times; the nodes perturb the schedule, so "
                               "these per-kernel figures need not add up to ms_per_step",
        "kernel_avg_us": {k: round(1000.0 * sum(v) / len(v), 2) for k, v in kernel_ms.items() if v},
        "kernel_p50_us": {k: round(1000.0 * statistics.median(v), 2) for k, v in kernel_ms.items() if v},
        "kernel_max_us": {k: round(1000.0 * max(v), 2) for k, v in kernel_ms.items() if v},
        "kernel_spans": kernel_spans,
        "attended_blocks_per_head": round(attended_per_head, 2),
        "fetched_bytes_per_step": int(fetched_bytes_per_step),
        "timed_steps": [pre + args.warmup, pre + args.warmup + args.steps - 1],
        "ms_per_step_eager_python": eager_ms,
        "gpu_launches": launches * args.steps,
        "copy_mode": args.copy,
        "hostlink": hostlink,
        "true_query_top64_turnover": None if top64_turnover is None else round(top64_turnover, 4),
        "host_tier_fit": host_fit,
        "other_configs": other,
        "prediction_agreement": agreement,
        "pooled_scoring": pooled,
        "lag_pipeline": lag,
        "lookahead_attention": la_attn,
        "clocks": clk,
        "e2e": e2e,
        "device_error_word": errw,
        "setup_s": round(gen_s, 1), "alloc_s": round(alloc_s, 1),
        "host_tier_warm_s": None if warm_s is None else round(warm_s, 2),
        "score_kernel": "tcgen05 (TMA ring, TMEM accumulators)" if args.score_kernel == "tc" else "mma.sync",
    }
    if not args.no_cpu_baseline and world == 1:
        try:
            line["cpu_baseline"] = cpu_baseline(args, args.cpu_heads)
        except Exception as e:  # the GPU measurement stands without it
            line["cpu_baseline"] = {"unavailable": f"{type(e).__name__}: {str(e)[-300:]}"}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.cpu_worker:
        print(json.dumps({"sec_per_head": cpu_sample(args, args.cpu_worker, warm=1)}), flush=True)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch

        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch

            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
