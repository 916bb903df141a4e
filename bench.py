#!/usr/bin/env python
"""Benchmark of the fused decode-and-multiply hot path on GB300.

One step = one pass of the dictionary-path hot path over one token batch of
the switch-c2048-shaped MoE FFN layer (E=2048 experts, d_model=2080,
d_ff=6144, ternary weights with P(0)=0.886 dictionary-coded: ~0.76 bits per
weight of codewords, ~0.81 stored with row starts, block lengths and row
scales; T=4096 bf16 tokens, top-1 Zipf(1.0) routing): route (top-1 + softmax
gate) -> bucket tokens by expert -> fused decode-multiply of every touched
expert's wi with ReLU -> fused decode-multiply of wo with the gate applied.
Inputs are resident in HBM; each step streams the touched experts' compressed
weights (about 2.5 GB, 20x the L2), so no L2 flush is needed.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import os

# The CPU oracle timings use one BLAS thread; set before numpy loads.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import csv
import dataclasses
import hashlib
import io
import json
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

CFG = synth.SWITCH_C2048
T_MAIN = 4096
TC_MIN_TOKENS = 32      # experts with this many tokens take the tensor-core kernel ...
TC_MIN_SLOTS = 256      # ... in launches with at least this many token slots
METRIC = "MoE-layer tokens/s and compressed-stream HBM GB/s (% of GB300 peak) at 1 GPU"
UNIT = "tokens/s"
WORKLOAD = (f"{CFG.name} MoE FFN layer: E={CFG.E}, d_model={CFG.d_model}, d_ff={CFG.d_ff}, T={T_MAIN} bf16 tokens, "
            f"top-1 Zipf(s={CFG.zipf_s}) routing, ternary P(0)={CFG.p0} dictionary-coded (2^16 entries, "
            f"256-weight blocks), seed {CFG.seed}")


# ---------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (the job is as slow as its slowest rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        if not self.out:
            return None
        rows = [r for r in csv.reader(io.StringIO(self.out)) if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_traffic(kernel_file: str, key: str):
    """Per-launch DRAM bytes from the committed ncu summary, if the kernel source is unchanged since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[key]
        with open(os.path.join(ROOT, kernel_file), "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
        if rec.get("source_sha256") != digest:
            return None
        return rec.get("dram_bytes_per_launch")
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------- workload
def native_synth():
    import ctypes
    lib = ctypes.CDLL(os.path.join(ROOT, "synth", "libsynth.so"))
    lib.synth_ternary_rows.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int64,
                                       ctypes.c_uint32, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    lib.synth_ternary_rows.restype = None
    return lib


def build_dict_layer(cfg, device):
    from decode_matvec_gb300.layers import DictLayer
    lib = native_synth()
    thr = synth.zero_threshold(cfg.p0)

    def tern(matrix):
        def fill(e, out):
            rows, cols = out.shape
            lib.synth_ternary_rows(cfg.seed, e, matrix, cols, thr, 0, rows, out.ctypes.data)
        return fill

    def scale(matrix):
        rows = synth.dict_matrix_shape(cfg, matrix)[0]
        return lambda e: synth.row_scales(cfg.seed, e, matrix, rows)

    return DictLayer(cfg.p0, cfg.E, cfg.d_model, cfg.d_ff, tern(synth.WI), tern(synth.WO), scale(synth.WI),
                     scale(synth.WO), device=device)


class DictStep:
    """Device buffers and one step of the dictionary hot path for one token batch."""

    def __init__(self, layer, cfg, T, rank, device):
        import torch
        self.layer, self.T = layer, T
        # rank r > 0 gets its own independent batch (weak scaling)
        rcfg = dataclasses.replace(cfg, seed=cfg.seed + 7919 * rank)
        self.logits_host = synth.layer_logits(rcfg, T)
        self.x_host = synth.layer_tokens(rcfg, T)
        self.x = torch.from_numpy(self.x_host.view(np.int16).copy()).to(device)
        self.logits = torch.from_numpy(self.logits_host).to(device)
        self.ids = torch.empty((T, 1), dtype=torch.int32, device=device)
        self.gates = torch.empty((T, 1), dtype=torch.float32, device=device)
        self.y = torch.empty((T, layer.d_model), dtype=torch.int16, device=device)
        import decode_matvec_gb300 as Q
        self.Q = Q
        self.ws = torch.empty(Q.qmoe_moe_layer_ws_size(layer.E, layer.d_model, layer.d_ff, T, 1), dtype=torch.uint8,
                              device=device)

    def run(self, stream=None):
        Q, L = self.Q, self.layer
        Q.qmoe_route(self.logits, 1, self.ids, self.gates, stream=stream)
        Q.qmoe_moe_layer(L.dictionary, L.wi, L.wo, self.x, self.ids, self.gates, self.y, self.ws, y_is_f32=False,
                         stream=stream)

    launches_per_step = 6   # route, plan, wi CUDA-core + tensor-core kernels, wo CUDA-core + tensor-core kernels


def time_steps(step, K, W, world):
    """K timed steps after W warm-up steps, bracketed by barriers; returns (seconds, {p10, p50, p90} ms)."""
    import torch
    st = torch.cuda.current_stream()
    for _ in range(W):
        step.run()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    # one event between consecutive steps: the first and last bracket the K steps, the others give
    # the per-step distribution
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    ev[0].record(st)
    for i in range(K):
        step.run()
        ev[i + 1].record(st)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    per = np.array([ev[i].elapsed_time(ev[i + 1]) for i in range(K)])
    dist = {q: float(np.percentile(per, v)) for q, v in (("p10", 10), ("p50", 50), ("p90", 90))}
    return ev[0].elapsed_time(ev[K]) / 1000.0, dist


def time_phases(step, K):
    """Per-kernel device time over K steps from phase events recorded by the library."""
    import torch
    Q = step.Q
    st = torch.cuda.current_stream()
    rec = []
    pool = []
    for _ in range(K):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        for e in ev:
            e.record(st)        # torch creates the CUDA event on first record
        pool.append(ev)
    torch.cuda.synchronize()
    for i in range(K):
        ev = pool[i]
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        Q.qmoe_set_phase_events(ev)
        r0.record(st)
        Q.qmoe_route(step.logits, 1, step.ids, step.gates)
        r1.record(st)
        L = step.layer
        Q.qmoe_moe_layer(L.dictionary, L.wi, L.wo, step.x, step.ids, step.gates, step.y, step.ws, y_is_f32=False)
        rec.append((r0, r1, ev))
    Q.qmoe_set_phase_events(None)
    torch.cuda.synchronize()
    out = {"route": 0.0, "plan": 0.0, "wi": 0.0, "wi_tc": 0.0, "wo": 0.0, "wo_tc": 0.0}
    for r0, r1, ev in rec:
        out["route"] += r0.elapsed_time(r1) / 1000.0
        out["plan"] += ev[0].elapsed_time(ev[1]) / 1000.0
        out["wi"] += ev[1].elapsed_time(ev[2]) / 1000.0
        out["wi_tc"] += ev[2].elapsed_time(ev[3]) / 1000.0
        out["wo"] += ev[3].elapsed_time(ev[4]) / 1000.0
        out["wo_tc"] += ev[4].elapsed_time(ev[5]) / 1000.0
    return {k: v / K for k, v in out.items()}


def time_e2e(step, K, W):
    """The same step through the public API with host buffers, pipelined the way a serving loop runs
    it: step i's inputs (x, router logits) go host -> device on one copy stream while step i - 1
    computes, and step i - 1's output goes device -> host on another; inputs and outputs are double
    buffered.  Every step's copies are inside the timed region."""
    import torch
    Q, L = step.Q, step.layer
    x_pin = torch.from_numpy(step.x_host.view(np.int16).copy()).pin_memory()
    lg_pin = torch.from_numpy(step.logits_host).pin_memory()
    comp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    bufs = [dict(x=torch.empty_like(step.x), lg=torch.empty_like(step.logits), y=torch.empty_like(step.y),
                 y_pin=torch.empty(tuple(step.y.shape), dtype=torch.int16).pin_memory()) for _ in range(2)]
    in_ready = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    for s_ in range(2):
        computed[s_].record(comp)
        out_done[s_].record(comp)

    def issue(i):
        s_ = i % 2
        b = bufs[s_]
        with torch.cuda.stream(h2d):
            h2d.wait_event(computed[s_])             # step i - 2 has finished reading these inputs
            b["x"].copy_(x_pin, non_blocking=True)
            b["lg"].copy_(lg_pin, non_blocking=True)
            in_ready[s_].record(h2d)
        comp.wait_event(in_ready[s_])
        comp.wait_event(out_done[s_])                # step i - 2's output has been copied out
        Q.qmoe_route(b["lg"], 1, step.ids, step.gates, stream=comp)
        Q.qmoe_moe_layer(L.dictionary, L.wi, L.wo, b["x"], step.ids, step.gates, b["y"], step.ws, y_is_f32=False,
                         stream=comp)
        computed[s_].record(comp)
        with torch.cuda.stream(d2h):
            d2h.wait_event(computed[s_])
            b["y_pin"].copy_(b["y"], non_blocking=True)
            out_done[s_].record(d2h)

    for i in range(W):
        issue(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    h2d.wait_event(e0)
    d2h.wait_event(e0)
    for i in range(K):
        issue(i)
    comp.wait_event(out_done[(K - 1) % 2])
    e1.record(comp)
    torch.cuda.synchronize()
    bi = x_pin.numel() * 2 + lg_pin.numel() * 4
    bo = bufs[0]["y_pin"].numel() * 2
    return e0.elapsed_time(e1) / 1000.0 / K, bi, bo


# ---------------------------------------------------------------- CPU oracle timing
def sampled_parity(step, cfg, tokens):
    """The timed layer call again with fp32 output; for a few sampled tokens, the normwise relative
    error against the float64 oracle layer computed from the seeded ternary weights and row scales
    themselves (so dictionary, encoder, decoder and product are all checked)."""
    import torch
    from oracle import moe as M
    from oracle import products as P
    Q, L = step.Q, step.layer
    y32 = torch.empty((step.T, L.d_model), dtype=torch.float32, device=step.x.device)
    Q.qmoe_route(step.logits, 1, step.ids, step.gates)
    Q.qmoe_moe_layer(L.dictionary, L.wi, L.wo, step.x, step.ids, step.gates, y32, step.ws, y_is_f32=True)
    status = Q.qmoe_check_status()
    y = y32.cpu().numpy()
    rid, rg = M.route(step.logits_host, 1)
    x = synth.bf16_to_f64(step.x_host)
    lib = native_synth()                     # the seeded ternary generator (checked against synth's definition)
    thr = synth.zero_threshold(cfg.p0)
    worst = 0.0
    for t in tokens:
        e = int(rid[t, 0])
        w = []
        for m in (synth.WI, synth.WO):
            rows, cols = synth.dict_matrix_shape(cfg, m)
            tern = np.zeros((rows, cols), np.int8)
            lib.synth_ternary_rows(cfg.seed, e, m, cols, thr, 0, rows, tern.ctypes.data)
            s = synth.row_scales(cfg.seed, e, m, rows).view(np.float16).astype(np.float64)
            w.append(tern.astype(np.float64) * s[:, None])
        ref = rg[t, 0] * M.relu_expert(x[t:t + 1], w[0], w[1])[0]
        worst = max(worst, P.normwise_rel_err(y[t], ref))
    return {"max_normwise_rel_err": worst, "tolerance": 2e-3, "status_ok": status == Q.QMOE_OK,
            "routing_equal": bool(np.array_equal(step.ids.cpu().numpy(), rid)),
            "sample": f"tokens {list(tokens)}: fp32-mode output against the float64 oracle from the seeded "
                      "ternary weights (max |y - ref| / max |ref| per token)"}


class OracleSampler:
    """Times the CPU oracle on bounded samples of the layer: decode + float64 product of a
    64-row slice of one touched expert's matrix for that expert's tokens.  Inputs are
    oracle-encoded from the seeded weights outside the timed part."""

    ROWS = 64

    def __init__(self, cfg, T, seed=0):
        from oracle import codec as C
        from oracle import dictionary as D
        from oracle import moe as M
        self.C, self.M = C, M
        self.cfg, self.T = cfg, T
        self.words = D.build(cfg.p0)
        self.table = C.entry_table(self.words)
        logits = synth.layer_logits(cfg, T)
        self.ids = np.argmax(logits, axis=1) if cfg.top_k == 1 else M.route(logits, cfg.top_k)[0]
        self.counts = np.bincount(np.asarray(self.ids).reshape(-1), minlength=cfg.E)
        self.touched = np.nonzero(self.counts)[0]
        self.x = synth.bf16_to_f64(synth.activations_bf16(cfg.seed, T, cfg.d_model))
        self.rng = np.random.default_rng(seed)
        self.total_weights = int(len(self.touched)) * 2 * cfg.d_model * cfg.d_ff

    def step(self):
        """One sample; returns (seconds, weights decoded)."""
        cfg = self.cfg
        e = int(self.rng.choice(self.touched))
        matrix = int(self.rng.integers(0, 2))
        rows, cols = synth.dict_matrix_shape(cfg, matrix)
        r0 = int(self.rng.integers(0, rows - self.ROWS + 1))
        tern = synth.ternary_rows(cfg.seed, e, matrix, cols, cfg.p0, r0, self.ROWS)
        codes, off = self.C.encode(tern, self.words, table=self.table)
        scale = synth.row_scales(cfg.seed, e, matrix, rows)[r0:r0 + self.ROWS]
        n_e = int(self.counts[e])
        xin = self.x[:n_e, :cols] if matrix == 0 else synth.bf16_to_f64(synth.activations_bf16(e, n_e, cols))
        t0 = time.perf_counter()
        w = self.C.decode(codes, off, self.words, scale, self.ROWS, cols)
        _ = xin @ w.T
        return time.perf_counter() - t0, self.ROWS * cols

    def sample(self, budget_s=None, n_steps=None):
        """(timed seconds, weights, samples) over a bounded run."""
        secs, weights, n = 0.0, 0, 0
        t_start = time.perf_counter()
        while True:
            s, w = self.step()
            secs += s
            weights += w
            n += 1
            if n_steps is not None and n >= n_steps:
                break
            if budget_s is not None and time.perf_counter() - t_start > budget_s:
                break
        return secs, weights, n


def host_cores() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


_WORKER = {}


def _sampler_init(cfg_name, T, seed0):
    import multiprocessing as mp
    cfg = {c.name: c for c in (synth.SWITCH_BASE_128, synth.SWITCH_LARGE_128, synth.SWITCH_C2048)}[cfg_name]
    ident = mp.current_process()._identity
    _WORKER["sampler"] = OracleSampler(cfg, T, seed=seed0 + (ident[0] if ident else 0))


def _sampler_task(budget_s):
    return _WORKER["sampler"].sample(budget_s=budget_s)


def _sampler_one(_):
    return _WORKER["sampler"].step()


def oracle_baseline(cfg, T, budget_1, budget_n, cores=None):
    """The oracle's throughput on the workload, extrapolated from 64-row slices of touched experts: once
    on one core, once on every host core (a spawn pool, one sampler per process, all sampling at the
    same time; the aggregate rate is the sum of the processes' rates)."""
    import multiprocessing as mp
    cores = cores or host_cores()
    one = OracleSampler(cfg, T)
    one.step()
    s1, w1, n1 = one.sample(budget_s=budget_1)
    total = one.total_weights
    out = {"unit": UNIT, "kind": "oracle", "extrapolated": True,
           "single_core": {"value": T / (total / (w1 / s1)), "cores": 1, "samples": n1, "weights": w1,
                           "seconds": s1}}
    if cores > 1:
        with mp.get_context("spawn").Pool(cores, initializer=_sampler_init, initargs=(cfg.name, T, 1000)) as pool:
            pool.map(_sampler_task, [0.5] * cores)          # warm-up: every process decodes once
            res = pool.map(_sampler_task, [budget_n] * cores)
        rate = sum(w / s for s, w, n in res)
        n_all, w_all = sum(r[2] for r in res), sum(r[1] for r in res)
    else:
        rate, n_all, w_all = w1 / s1, n1, w1
    out.update({"value": T / (total / rate), "cores": cores,
                "sample": (f"{n_all} slices of {OracleSampler.ROWS} rows of touched experts' wi/wo ({w_all} weights; "
                           f"decode + float64 product for the expert's tokens) on {cores} host cores at once, "
                           f"extrapolated to the {len(one.touched)} touched experts ({total} weights) of the "
                           f"T={T} batch; single_core: the same on one core")})
    return out


# ---------------------------------------------------------------- the oracle on whole workloads
def _dict_expert_task(args):
    """The oracle's MoE expert on one seeded expert: decode wi and wo (host-encoded codewords) and the
    float64 product h = bf16(relu(Wi x)), o = Wo h for the expert's tokens; returns timed seconds."""
    from oracle import codec as C
    from oracle import moe as M
    import decode_matvec_gb300 as Q
    cfg_name, e, xs, words = args
    cfg = {c.name: c for c in (synth.SWITCH_BASE_128, synth.SWITCH_LARGE_128, synth.SWITCH_C2048)}[cfg_name]
    lib = native_synth()
    thr = synth.zero_threshold(cfg.p0)
    mats = []
    for m in (synth.WI, synth.WO):
        rows, cols = synth.dict_matrix_shape(cfg, m)
        tern = np.empty((rows, cols), np.int8)
        lib.synth_ternary_rows(cfg.seed, e, m, cols, thr, 0, rows, tern.ctypes.data)
        codes, off = Q.qmoe_pack(tern, words)
        mats.append((codes, off, synth.row_scales(cfg.seed, e, m, rows), rows, cols))
    t0 = time.perf_counter()
    wi = C.decode(mats[0][0], mats[0][1], words, mats[0][2], mats[0][3], mats[0][4])
    wo = C.decode(mats[1][0], mats[1][1], words, mats[1][2], mats[1][3], mats[1][4])
    _ = M.relu_expert(xs, wi, wo)
    return time.perf_counter() - t0


def _rvq_expert_task(args):
    """The oracle's SwiGLU expert on one seeded expert: decode gate/up/down (host-encoded indices) and
    the float64 transform-aware product for the expert's tokens; returns timed seconds."""
    from oracle import rvq as R
    import decode_matvec_gb300 as Q
    seed, e, shapes, cb, xs = args
    parts = []
    for m, (rows, cols) in enumerate(shapes):
        w = synth.rvq_weight(seed, e, m, rows, cols)
        so, si = synth.rvq_signs(seed, e, m, rows, cols)
        idx, sc = Q.rvq_pack(w, so, si, cb)
        parts.append((idx, sc, so, si))
    t0 = time.perf_counter()
    trip = [(R.decode(idx, cb, sc), so, si) for idx, sc, so, si in parts]
    _ = R.swiglu_expert(xs, *trip)
    return time.perf_counter() - t0


def oracle_full_rows(cores=None):
    """The oracle on the whole of three workloads (every touched expert, every token), on every host
    core: linear 1024x4096 (T = 1, 8, 32), switch-base-128 (T = 512) and the OLMoE-shaped two-stage RVQ
    layer (T = 1, 32).  Inputs are the seeded weights, encoded by the library's host encoders (which the
    tests pin byte for byte to the oracle's encoders) outside the timed part; the timed part is the
    oracle's decode and float64 product.  tokens_per_s = T / (timed CPU seconds / cores)."""
    import multiprocessing as mp
    from oracle import codec as C
    from oracle import moe as M
    from oracle import products as P
    import decode_matvec_gb300 as Q
    cores = cores or host_cores()
    rows = []
    # linear layer: one matrix, all its tokens
    lc = synth.LINEAR_1024x4096
    words, _ = Q.qmoe_encode_dictionary(lc.p0)
    tern = synth.ternary_matrix(lc.seed, 0, 0, lc.rows, lc.cols, lc.p0)
    codes, off = Q.qmoe_pack(tern, words)
    sc = synth.row_scales(lc.seed, 0, 0, lc.rows)
    for T in lc.tokens:
        x = synth.bf16_to_f64(synth.activations_bf16(lc.seed, T, lc.cols))
        t0 = time.perf_counter()
        W = C.decode(codes, off, words, sc, lc.rows, lc.cols)
        _ = P.matmul_xwt(x, W)
        secs = time.perf_counter() - t0
        rows.append({"workload": f"{lc.name}, T={T}", "tokens_per_s": T / secs, "cpu_seconds": secs, "cores": 1,
                     "sample": "the whole call (one matrix, every token) on one core"})
    with mp.get_context("spawn").Pool(cores) as pool:
        cfg = synth.SWITCH_BASE_128
        T = cfg.tokens[0]
        ids = M.route(synth.layer_logits(cfg, T), 1)[0][:, 0]
        x = synth.bf16_to_f64(synth.layer_tokens(cfg, T))
        w2, _ = Q.qmoe_encode_dictionary(cfg.p0)
        tasks = [(cfg.name, int(e), x[ids == e], w2) for e in np.unique(ids)]
        t0 = time.perf_counter()
        secs = pool.map(_dict_expert_task, tasks)
        wall = time.perf_counter() - t0
        rows.append({"workload": f"{cfg.name} MoE layer, T={T}", "tokens_per_s": T / (sum(secs) / cores),
                     "cpu_seconds": sum(secs), "cores": cores, "wall_seconds_with_untimed_encoding": wall,
                     "sample": f"the whole layer call: all {len(tasks)} touched experts, every token"})
        rc = synth.OLMOE_RVQ
        cb = np.load(os.path.join(ROOT, "tests", "golden", "olmoe_rvq_codebooks.npy")).view(np.uint16)
        shapes = [synth.rvq_matrix_shape(rc, m) for m in (synth.GATE, synth.UP, synth.DOWN)]
        for T in rc.tokens:
            ids = M.route(synth.layer_logits(rc, T), rc.top_k)[0]
            x = synth.bf16_to_f64(synth.layer_tokens(rc, T))
            tasks = [(rc.seed, int(e), shapes, cb, x[np.nonzero((ids == e).any(axis=1))[0]]) for e in np.unique(ids)]
            t0 = time.perf_counter()
            secs = pool.map(_rvq_expert_task, tasks)
            wall = time.perf_counter() - t0
            rows.append({"workload": f"{rc.name} SwiGLU MoE layer, T={T}", "tokens_per_s": T / (sum(secs) / cores),
                         "cpu_seconds": sum(secs), "cores": cores, "wall_seconds_with_untimed_encoding": wall,
                         "sample": f"the whole layer call: all {len(tasks)} touched experts, every token "
                                   "(the slot combine, a few multiply-adds per output, is not timed)"})
    return rows


# ---------------------------------------------------------------- extra rows
def _time_calls(fn, n=50, warm=5):
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1000.0 / n


def _dict_layer_row(layer, cfg, T, device, peak, note=""):
    st = DictStep(layer, cfg, T, 0, device)
    t = _time_calls(st.run)
    t_graph = _graph_time(st.run)
    phases = {k: v * 1e3 for k, v in time_phases(st, 20).items()}
    touched = np.unique(st.ids.cpu().numpy().reshape(-1))
    sb = layer.stream_bytes(touched)
    return {"workload": f"{cfg.name} MoE layer (E={cfg.E}, d={cfg.d_model}, f={cfg.d_ff}, p0={cfg.p0}), T={T}{note}",
            "tokens_per_s": T / t, "ms_per_call": t * 1e3, "touched_experts": int(len(touched)),
            "stream_bytes": sb, "stream_gbs": sb / t / 1e9, "stream_pct_of_hbm_peak": 100.0 * sb / t / 1e9 / peak,
            "ms_per_call_cuda_graph": t_graph * 1e3, "phase_ms": phases}


def _rotating_dict_row(layer, cfg, T, device, peak, replicas=1, batches=1, n=60):
    """The layer call cycling over `replicas` device copies of the layer's weights (each call streams
    weights that the previous calls did not leave in L2) or over `batches` token batches (different
    routing, so mostly different experts): an HBM figure for layers or batches that fit in L2."""
    import types
    views = [layer]
    for _ in range(replicas - 1):
        views.append(types.SimpleNamespace(dictionary=layer.dictionary, wi=layer.wi_host.to_device(device),
                                           wo=layer.wo_host.to_device(device), E=layer.E, d_model=layer.d_model,
                                           d_ff=layer.d_ff))
    steps = [DictStep(v, cfg, T, b, device) for v in views for b in range(batches)]
    for st_ in steps:
        st_.run()
    calls = [st_.run for st_ in steps]
    t = _time_calls(lambda it=iter(range(1 << 30)): calls[next(it) % len(calls)](), n=n, warm=len(calls))
    sb = float(np.mean([layer.stream_bytes(np.unique(st_.ids.cpu().numpy().reshape(-1))) for st_ in steps]))
    what = f"{replicas} weight copies" if replicas > 1 else f"{batches} token batches"
    out = {"workload": f"{cfg.name} MoE layer (E={cfg.E}, d={cfg.d_model}, f={cfg.d_ff}, p0={cfg.p0}), T={T}, "
                       f"cycling over {what}",
           "tokens_per_s": T / t, "ms_per_call": t * 1e3, "stream_bytes": sb, "stream_gbs": sb / t / 1e9,
           "stream_pct_of_hbm_peak": 100.0 * sb / t / 1e9 / peak,
           "resident_bytes_cycled": sb * len(steps)}
    del views, steps
    return out


def _graph_time(step, n=50, warm=5):
    """Time of `step` replayed from a CUDA graph (host launch overhead removed)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    t = _time_calls(graph.replay, n=n, warm=warm)
    del graph
    return t


def _rvq_phases(call, K=20):
    """Device time of rvq_moe_layer's phases (library phase events), averaged over K calls."""
    import torch
    import decode_matvec_gb300 as Q
    st = torch.cuda.current_stream()
    pool = []
    for _ in range(K):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        for e in ev:
            e.record(st)        # torch creates the CUDA event on first record
        pool.append(ev)
    torch.cuda.synchronize()
    for ev in pool:
        Q.qmoe_set_phase_events(ev)
        call()
    Q.qmoe_set_phase_events(None)
    torch.cuda.synchronize()
    names = ("plan_and_in_transform", "gate_up", "swiglu_and_down_in_transform", "down", "out_transform")
    return {n: sum(ev[i].elapsed_time(ev[i + 1]) for ev in pool) / K for i, n in enumerate(names)}


def _rvq_rows(device, peak, cfg=None):
    """The OLMoE-shaped RVQ layer at T = 1 and 32.  With cfg.freq_stages, expert e's matrices have
    rvq_stage_allocation(popularity)[e] stages (3 / 2 / 1 by popularity thirds, mean 2 bits per
    weight) and the router uses the layer's fixed popularity."""
    import torch
    import decode_matvec_gb300 as Q
    from decode_matvec_gb300.layers import pack_e8p_set, pack_rvq_set
    cfg = cfg or synth.OLMOE_RVQ
    golden = os.path.join(ROOT, "tests", "golden")
    e8p = cfg.vq == "e8p"
    if e8p:
        cb = np.zeros((0, 256, 8), dtype=np.uint16)
        stages = None
    elif cfg.freq_stages:
        cb = np.load(os.path.join(golden, "olmoe_rvq_codebooks3.npy")).view(np.uint16)
        stages = Q.rvq_stage_allocation(synth.zipf_popularity(cfg.seed, cfg.E, cfg.zipf_s), cfg.stages)
    else:
        cb = np.load(os.path.join(golden, "olmoe_rvq_codebooks.npy")).view(np.uint16)
        stages = None
    sets = []
    for m in (synth.GATE, synth.UP, synth.DOWN):
        rows, cols = synth.rvq_matrix_shape(cfg, m)
        wfn = lambda e, m=m, r=rows, c=cols: synth.rvq_weight(cfg.seed, e, m, r, c)   # noqa: E731
        sfn = lambda e, m=m, r=rows, c=cols: synth.rvq_signs(cfg.seed, e, m, r, c)    # noqa: E731
        sets.append(pack_e8p_set(cfg.E, rows, cols, wfn, sfn, device=device) if e8p else
                    pack_rvq_set(cfg.E, rows, cols, cb, wfn, sfn, device=device, stages=stages))
    out = []
    for T in cfg.tokens:
        lg = torch.from_numpy(synth.layer_logits(cfg, T)).to(device)
        x = torch.from_numpy(synth.layer_tokens(cfg, T).view(np.int16).copy()).to(device)
        ids = torch.empty((T, cfg.top_k), dtype=torch.int32, device=device)
        gates = torch.empty((T, cfg.top_k), dtype=torch.float32, device=device)
        y = torch.empty((T, cfg.d_model), dtype=torch.int16, device=device)
        ws = torch.empty(Q.rvq_moe_layer_ws_size(cfg.E, cfg.d_model, cfg.d_ff, T, cfg.top_k), dtype=torch.uint8,
                         device=device)

        def step():
            Q.qmoe_route(lg, cfg.top_k, ids, gates)
            Q.rvq_moe_layer(sets[0], sets[1], sets[2], x, ids, gates, y, ws, y_is_f32=False)
        t = _time_calls(step)
        t_graph = _graph_time(step)
        phases = _rvq_phases(lambda: Q.rvq_moe_layer(sets[0], sets[1], sets[2], x, ids, gates, y, ws,
                                                     y_is_f32=False))
        touched = np.unique(ids.cpu().numpy().reshape(-1))
        sb = 1024 if e8p else 2 * 256 * 8 * cb.shape[0]
        for e in touched:
            s_e = 2 if stages is None else int(stages[e])
            sb += sum(r * (c // 8) * s_e + r * 2 + r + c for r, c in
                      (synth.rvq_matrix_shape(cfg, m) for m in (synth.GATE, synth.UP, synth.DOWN)))
        label = "E8P lattice code, 16 bits per 8 weights" if e8p else "2-stage RVQ d=8" if stages is None else \
            "RVQ d=8, 3/2/1 stages by popularity thirds (2 bits mean)"
        out.append({"workload": f"{cfg.name} SwiGLU MoE layer (E={cfg.E}, d={cfg.d_model}, f={cfg.d_ff}, top-8, "
                                f"{label}), T={T}" + (" (tcgen05 path)" if T * cfg.top_k >= 16 else ""),
                    "tokens_per_s": T / t, "ms_per_call": t * 1e3, "touched_experts": int(len(touched)),
                    "stream_bytes": int(sb), "stream_gbs": sb / t / 1e9,
                    "stream_pct_of_hbm_peak": 100.0 * sb / t / 1e9 / peak, "phase_ms": phases,
                    "ms_per_call_cuda_graph": t_graph * 1e3})
    return out


def extra_rows(layer, device, peak):
    """The other workloads, measured in the same run (all bf16 outputs)."""
    import torch
    import decode_matvec_gb300 as Q
    rows = []

    def guarded(fn):
        try:
            r = fn()
            rows.extend(r if isinstance(r, list) else [r])
        except Exception as exc:  # a failing extra row must not hide the headline line
            rows.append({"error": f"{type(exc).__name__}: {exc}"})

    for T in (64, 1):
        guarded(lambda T=T: _dict_layer_row(layer, CFG, T, device, peak,
                                            " (one batch, repeated: L2-resident, a latency figure)" if T == 1 else
                                            " (one batch, repeated: partly L2-resident)"))
        # HBM figure: 16 token batches in turn (each call mostly touches experts the last did not)
        guarded(lambda T=T: _rotating_dict_row(layer, CFG, T, device, peak, batches=16))
    for cfg in (synth.SWITCH_BASE_128, synth.SWITCH_LARGE_128):
        def one(cfg=cfg):
            small = build_dict_layer(cfg, device)
            r = [_dict_layer_row(small, cfg, T, device, peak, " (layer fits in L2: not an HBM figure)")
                 for T in cfg.tokens]
            # HBM figure: copies of the layer's weights in turn, more than twice the L2 in all
            per = small.total_bytes()
            reps = max(2, int(np.ceil(2.2 * 129e6 / per)))
            r += [_rotating_dict_row(small, cfg, T, device, peak, replicas=reps) for T in cfg.tokens]
            del small
            return r
        guarded(one)
    guarded(lambda: _rvq_rows(device, peak))
    guarded(lambda: _rvq_rows(device, peak, synth.OLMOE_RVQ_FREQ))
    guarded(lambda: _rvq_rows(device, peak, synth.OLMOE_E8P))

    def linear():
        lc = synth.LINEAR_1024x4096
        lib = native_synth()
        tern = np.empty((lc.rows, lc.cols), np.int8)
        lib.synth_ternary_rows(lc.seed, 0, 0, lc.cols, synth.zero_threshold(lc.p0), 0, lc.rows, tern.ctypes.data)
        words, _ = Q.qmoe_encode_dictionary(lc.p0)
        codes, off = Q.qmoe_pack(tern, words)
        d = Q.Dictionary(words, device=device)
        m = Q.MatrixSet.from_host(codes, off, synth.row_scales(lc.seed, 0, 0, lc.rows), lc.rows, lc.cols,
                                  device=device)
        out = []
        sb = 2 * len(codes) + 4 * len(off) + 2 * lc.rows
        reps = int(np.ceil(2.2 * 129e6 / sb))
        copies = [m] + [Q.MatrixSet.from_host(codes, off, synth.row_scales(lc.seed, 0, 0, lc.rows), lc.rows, lc.cols,
                                              device=device) for _ in range(reps - 1)]
        peak_ = peak
        for T in lc.tokens:
            x = torch.from_numpy(synth.activations_bf16(lc.seed, T, lc.cols).view(np.int16).copy()).to(device)
            y = torch.empty((T, lc.rows), dtype=torch.int16, device=device)
            t = _time_calls(lambda: Q.qmoe_expert_matvec(d, m, x, y, y_is_f32=False), n=200, warm=10)
            out.append({"workload": f"{lc.name}, T={T} (one copy, repeated: L2-resident, a latency figure)",
                        "tokens_per_s": T / t, "us_per_call": t * 1e6, "stream_bytes": sb})
            it = iter(range(1 << 30))
            t2 = _time_calls(lambda: Q.qmoe_expert_matvec(d, copies[next(it) % reps], x, y, y_is_f32=False),
                             n=2 * reps, warm=reps)
            out.append({"workload": f"{lc.name}, T={T}, cycling over {reps} copies of the matrix ({reps * sb / 1e6:.0f} MB)",
                        "tokens_per_s": T / t2, "us_per_call": t2 * 1e6, "stream_bytes": sb,
                        "stream_gbs": sb / t2 / 1e9, "stream_pct_of_hbm_peak": 100.0 * sb / t2 / 1e9 / peak_})
        del copies
        return out
    guarded(linear)

    def device_encoder():
        # qmoe_pack_device on c2048-shaped wi matrices (6144 x 2080), against the host encoder
        cfg = CFG
        lib = native_synth()
        rows_, cols_ = synth.dict_matrix_shape(cfg, synth.WI)
        tern = np.empty((rows_, cols_), np.int8)
        lib.synth_ternary_rows(cfg.seed, 0, synth.WI, cols_, synth.zero_threshold(cfg.p0), 0, rows_, tern.ctypes.data)
        words = layer.words
        t0 = time.perf_counter()
        hc, ho = Q.qmoe_pack(tern, words)
        host_s = time.perf_counter() - t0
        tt = torch.from_numpy(tern).to(device)
        codes = torch.zeros(rows_ * cols_ // 2, dtype=torch.int16, device=device)
        off = torch.zeros(ho.size, dtype=torch.int32, device=device)
        ws = torch.empty(Q.qmoe_pack_device_ws_size(rows_, cols_), dtype=torch.uint8, device=device)
        t = _time_calls(lambda: Q.qmoe_pack_device(layer.dictionary, tt, codes, off, ws), n=20, warm=3)
        same = (Q.qmoe_check_status() == Q.QMOE_OK and
                np.array_equal(off.cpu().numpy().view(np.uint32), ho) and
                np.array_equal(codes[:hc.size].cpu().numpy().view(np.uint16), hc))
        w = rows_ * cols_
        return {"workload": f"device encoder qmoe_pack_device, {cfg.name} wi matrix {rows_}x{cols_} "
                            f"(p0={cfg.p0}, 256-weight blocks)",
                "weights_per_s": w / t, "ms_per_matrix": t * 1e3,
                "host_encoder_weights_per_s": w / host_s, "host_encoder_threads": 1,
                "equal_to_host_encoder": bool(same)}
    guarded(device_encoder)
    guarded(lambda: _dense_baseline_row(layer, device))
    guarded(lambda: _materialise_row(layer, device, 64))
    return rows


def _expert_view(Q, ms, host, e):
    """A count-1 matrix descriptor for expert e of a device matrix set."""
    return ms.expert(e, host.code_base)


def _materialise_row(layer, device, T):
    """The unfused alternative: decode each touched expert's wi and wo to dense fp32 in HBM
    (qmoe_decode_dense), then cuBLAS GEMMs; replayed from a CUDA graph."""
    import torch
    import decode_matvec_gb300 as Q
    cfg = CFG
    st = DictStep(layer, cfg, T, 0, device)
    st.run()
    ids = st.ids.view(-1)
    x = st.x.view(torch.bfloat16).float()
    gates = st.gates.view(-1)
    touched = torch.unique(ids).tolist()
    wi_d = torch.empty((cfg.d_ff, cfg.d_model), dtype=torch.float32, device=device)
    wo_d = torch.empty((cfg.d_model, cfg.d_ff), dtype=torch.float32, device=device)
    plan = [(torch.nonzero(ids == e).view(-1), _expert_view(Q, layer.wi, layer.wi_host, e),
             _expert_view(Q, layer.wo, layer.wo_host, e)) for e in touched]
    y = torch.zeros((T, cfg.d_model), dtype=torch.float32, device=device)

    def step():
        y.zero_()
        for idx, vi, vo in plan:
            Q.qmoe_decode_dense(layer.dictionary, vi, wi_d)
            h = torch.relu(x.index_select(0, idx) @ wi_d.t()).to(torch.bfloat16).float()
            Q.qmoe_decode_dense(layer.dictionary, vo, wo_d)
            y.index_add_(0, idx, (h @ wo_d.t()) * gates.index_select(0, idx).unsqueeze(1))

    side = torch.cuda.Stream(device=device)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    t = _time_calls(graph.replay, n=20, warm=3)
    ok = Q.qmoe_check_status() == Q.QMOE_OK
    fused = _time_calls(st.run, n=50, warm=5)
    return {"workload": f"materialise-then-GEMM baseline: {cfg.name} layer, T={T} (qmoe_decode_dense to fp32 in HBM "
                        f"per touched expert, then cuBLAS; CUDA graph)",
            "tokens_per_s": T / t, "ms_per_step": t * 1e3, "touched_experts": len(touched),
            "fused_ms_per_step": fused * 1e3, "status_ok": ok}


def _dense_baseline_row(layer, device):
    """The same layer step with uncompressed bf16 weights: per touched expert, cuBLAS GEMMs
    h = relu(x_e Wi_e^T), o = h Wo_e^T, gated scatter into y; replayed from a CUDA graph so that
    launch overhead is not timed.  The dense weights are fresh ternary draws with the layer's p0 and
    shapes (their values do not change the time), only for the experts this batch touches."""
    import torch
    cfg = CFG
    st = DictStep(layer, cfg, T_MAIN, 0, device)
    st.run()
    ids = st.ids.view(-1)
    x = st.x.view(torch.bfloat16)
    gates = st.gates.view(-1)
    touched = torch.unique(ids).tolist()
    g = torch.Generator(device=device)
    g.manual_seed(cfg.seed)

    def ternary(rows, cols):
        u = torch.rand((rows, cols), generator=g, device=device)
        w = torch.where(u < cfg.p0, 0.0, torch.where(u < (1 + cfg.p0) / 2, -1.0, 1.0))
        return w.to(torch.bfloat16)

    experts = []
    for e in touched:
        idx = torch.nonzero(ids == e).view(-1)
        experts.append((idx, ternary(cfg.d_ff, cfg.d_model), ternary(cfg.d_model, cfg.d_ff)))
    y = torch.zeros((T_MAIN, cfg.d_model), dtype=torch.float32, device=device)

    def step():
        y.zero_()
        for idx, wi, wo in experts:
            xe = x.index_select(0, idx)
            h = torch.relu(xe @ wi.t())
            o = (h @ wo.t()).float() * gates.index_select(0, idx).unsqueeze(1)
            y.index_add_(0, idx, o)

    side = torch.cuda.Stream(device=device)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    t = _time_calls(graph.replay, n=20, warm=3)
    dense_bytes = len(experts) * 2 * cfg.d_ff * cfg.d_model * 2
    del experts, graph
    torch.cuda.empty_cache()
    return {"workload": f"dense bf16 baseline: {cfg.name} layer step with uncompressed weights, T={T_MAIN} "
                        f"(cuBLAS per-expert GEMMs, CUDA graph)",
            "tokens_per_s": T_MAIN / t, "ms_per_step": t * 1e3, "touched_experts": len(touched),
            "dense_weight_bytes": dense_bytes, "dense_weight_gbs": dense_bytes / t / 1e9,
            "dense_ms_at_hbm_peak": dense_bytes / (hbm_peak()[0] * 1e9) * 1e3}


# ---------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="skip the extra rows and shorten the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--experts", type=int, default=None,
                    help="profiling case: keep only this many experts of the c2048-shaped layer")
    ap.add_argument("--tokens", type=int, default=None, help="profiling case: token batch size")
    ap.add_argument("--dict-rows", action="store_true",
                    help="profiling case: only the switch-base-128 / switch-large-128 layer rows, one JSON line")
    ap.add_argument("--rvq-rows", nargs="?", const="all", default=None, choices=("all", "rvq", "freq", "e8p"),
                    help="profiling case: only the OLMoE-shaped VQ layer rows (T=1 and T=32) of one code or all, "
                         "one JSON line")
    args = ap.parse_args()
    global CFG, T_MAIN, WORKLOAD
    if args.experts or args.tokens:
        CFG = dataclasses.replace(CFG, E=args.experts or CFG.E)
        T_MAIN = args.tokens or T_MAIN
        WORKLOAD = WORKLOAD.replace("E=2048", f"E={CFG.E}").replace("T=4096", f"T={T_MAIN}") + \
            " (reduced profiling case)"
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_setup()

    if args.impl == "reference":
        if rank != 0:
            return 0
        # the CPU oracle as it stands, on every host core: a step is the decode + float64 product of one
        # 64-row slice of a touched expert's matrix (a bounded sample of the layer); the metric is
        # extrapolated from the slices' rate to the whole layer call
        import multiprocessing as mp
        cores = host_cores()
        probe = OracleSampler(CFG, T_MAIN)
        with mp.get_context("spawn").Pool(cores, initializer=_sampler_init, initargs=(CFG.name, T_MAIN, 2000)) as pool:
            pool.map(_sampler_one, range(max(args.warmup, cores)), chunksize=1)
            t0 = time.perf_counter()
            res = pool.map(_sampler_one, range(args.steps), chunksize=1)
            wall = time.perf_counter() - t0
        weights = sum(w for _, w in res)
        secs = sum(t for t, _ in res)                          # timed decode + product, summed over processes
        rate = weights / (secs / cores)                        # weights per second with every core decoding
        layer_s = probe.total_weights / rate
        value = T_MAIN / layer_s
        cpu = {"value": value, "unit": UNIT, "kind": "oracle", "cores": cores, "extrapolated": True,
               "sample": (f"{args.steps} slices of {OracleSampler.ROWS} rows ({weights} weights: decode + float64 "
                          f"product for the expert's tokens; {secs:.2f} s of timed work, {wall:.2f} s of wall time "
                          f"with the untimed slice encoding) spread over {cores} host cores; extrapolated "
                          f"to the {len(probe.touched)} touched experts ({probe.total_weights} weights) of the "
                          f"T={T_MAIN} batch ({layer_s:.1f} s per layer call)")}
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps, "wall_seconds": wall,
                "step": f"one {OracleSampler.ROWS}-row slice (a bounded sample of the layer call)",
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "impl": "reference", "extrapolated": True,
                "config": {"workload": WORKLOAD, "tokens": T_MAIN},
                "cpu_baseline": cpu,
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    if args.dict_rows:
        if rank == 0:
            pk = hbm_peak()[0]
            rows = []
            for cfg in (synth.SWITCH_BASE_128, synth.SWITCH_LARGE_128):
                small = build_dict_layer(cfg, device)
                rows += [_dict_layer_row(small, cfg, T, device, pk, " (layer fits in L2: not an HBM figure)")
                         for T in cfg.tokens]
                del small
            print(json.dumps({"workload": "switch-base-128 / switch-large-128 layer rows (profiling case)",
                              "rows": rows}))
        return 0
    if args.rvq_rows:
        if rank == 0:
            pk = hbm_peak()[0]
            pick = {"rvq": [synth.OLMOE_RVQ], "freq": [synth.OLMOE_RVQ_FREQ], "e8p": [synth.OLMOE_E8P],
                    "all": [synth.OLMOE_RVQ, synth.OLMOE_RVQ_FREQ, synth.OLMOE_E8P]}[args.rvq_rows]
            print(json.dumps({"workload": "olmoe-shaped VQ layer rows (profiling case)",
                              "rows": [r for c in pick for r in _rvq_rows(device, pk, c)]}))
        return 0
    t_setup = time.time()
    layer = build_dict_layer(CFG, device)
    setup_s = time.time() - t_setup
    step = DictStep(layer, CFG, T_MAIN, rank, device)

    with ClockSampler(local if world > 1 else 0) as clk:
        secs, step_dist = time_steps(step, args.steps, args.warmup, world)
    secs = max_over_ranks(secs, world)
    ms_per_step = secs / args.steps * 1e3
    value = T_MAIN * world / (secs / args.steps)

    ids = step.ids.cpu().numpy().reshape(-1)
    touched = np.unique(ids)
    phases = time_phases(step, min(args.steps, 50))
    stream_bytes = layer.stream_bytes(touched)
    counts = np.bincount(ids, minlength=CFG.E)
    # experts with >= 32 tokens run on the tensor-core kernel (large launches only)
    hot = counts >= TC_MIN_TOKENS if T_MAIN >= TC_MIN_SLOTS else np.zeros(CFG.E, bool)
    kern = {}
    # the CUDA-core launches, one per matrix (which kernel each takes: the library's own choice)
    import decode_matvec_gb300 as Q
    wi_k, wo_k, _ = Q.qmoe_moe_layer_kernels(CFG.E, CFG.d_model, CFG.d_ff, T_MAIN, 1)
    ex = np.nonzero((counts > 0) & ~hot)[0]
    n_tok = int(counts[ex].sum())
    for label, host, k_id, secs_k in (("wi", layer.wi_host, wi_k, phases["wi"]), ("wo", layer.wo_host, wo_k, phases["wo"])):
        act = n_tok * (CFG.d_model * 2 + CFG.d_ff * 2)            # wi: x in, h out; wo: h in, y out
        b = sum(host.expert_bytes(int(e)) for e in ex) + act + 3 * 65536
        # the CUDA-core kernels read only the row starts, not the block lengths
        unread = sum(host.expert_offset_bytes_unread_by_cuda_cores(int(e)) for e in ex)
        kern[f"{Q.KERNEL_NAMES[k_id]} ({label})"] = {
            "experts": int(len(ex)), "tokens": n_tok, "launches_per_step": 1, "ms_per_step": secs_k * 1e3,
            "algorithmic_bytes_per_step": int(b), "achieved_gbs": (b / secs_k / 1e9) if secs_k > 0 else None,
            "bytes_read_per_step": int(b - unread),
            "achieved_gbs_on_bytes_read": (b - unread) / secs_k / 1e9 if secs_k > 0 else None}
    ex = np.nonzero(hot)[0]
    n_tok = int(counts[ex].sum())
    secs_k = phases["wi_tc"] + phases["wo_tc"]
    b = layer.stream_bytes(ex) + n_tok * (2 * CFG.d_model * 2 + 2 * CFG.d_ff * 2)
    kern["dict_tc_kernel (wi, wo)"] = {"experts": int(len(ex)), "tokens": n_tok, "launches_per_step": 2,
                                       "ms_per_step": secs_k * 1e3, "algorithmic_bytes_per_step": int(b),
                                       "achieved_gbs": (b / secs_k / 1e9) if secs_k > 0 else None}
    dom = max(kern, key=lambda k: kern[k]["ms_per_step"])
    peak, peak_kind = hbm_peak()
    achieved = kern[dom]["achieved_gbs"]
    e2e_s, bi, bo = time_e2e(step, max(10, args.steps // 4), 3)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "ms_per_step_distribution": step_dist,
        "config": {"workload": WORKLOAD, "tokens": T_MAIN, "activations": "bf16 in/out, fp32 accumulate",
                   "touched_experts": int(len(touched)),
                   "l2": "inputs larger than L2: each step streams the touched experts' compressed weights "
                         f"({stream_bytes / 1e9:.2f} GB) against a 129 MB L2",
                   "parallelism": f"{world} independent replicas (one token batch per GPU)"},
        "stream_gbs": stream_bytes / (secs / args.steps) / 1e9,
        "stream_pct_of_hbm_peak": 100.0 * stream_bytes / (secs / args.steps) / 1e9 / peak,
        # the dense bf16 bytes of the touched experts' weights the step replaces, per second; and the
        # stored bits per weight of those experts (codes, block offsets, row scales)
        "decoded_weight_gbs": len(touched) * 2 * CFG.d_model * CFG.d_ff * 2 / (secs / args.steps) / 1e9,
        "effective_bits_per_weight": 8.0 * stream_bytes / (len(touched) * 2 * CFG.d_model * CFG.d_ff),
        # ... with the canonical dictionary (2^16 entries x 8 bytes) counted once against the same weights
        "effective_bits_per_weight_with_dictionary":
            8.0 * (stream_bytes + 65536 * 8) / (len(touched) * 2 * CFG.d_model * CFG.d_ff),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "peak_kind": "measured (MEASURED_PEAKS hbm_gbs)" if peak_kind == "measured" else "fallback",
                     "unit": "GB/s", "frac": achieved / peak,
                     "frac_on_bytes_read": (kern[dom].get("achieved_gbs_on_bytes_read") or achieved) / peak,
                     "traffic": kernel_traffic("decode_matvec_gb300/csrc/dict_kernels.cu", dom),
                     "kernels": kern, "phase_ms": {k: v * 1e3 for k, v in phases.items()}},
        "e2e": {"value": T_MAIN / e2e_s, "unit": UNIT, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo},
        "gpu_launches": DictStep.launches_per_step * args.steps,
        "clocks": clk.summary(),
        "setup_seconds": setup_s,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(CFG, T_MAIN, 3.0 if args.quick else 8.0, 3.0 if args.quick else 10.0)
        line["parity"] = sampled_parity(step, CFG, (0, T_MAIN // 2, T_MAIN - 1))
    if rank == 0 and not args.quick:
        line["rows"] = extra_rows(layer, device, peak)
        if world == 1 and not args.no_cpu_baseline:
            try:
                line["cpu_oracle_full_workloads"] = oracle_full_rows()
            except Exception as exc:  # the oracle rows must not hide the headline line
                line["cpu_oracle_full_workloads"] = [{"error": f"{type(exc).__name__}: {exc}"}]
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
