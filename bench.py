"""Benchmark: paged split-KV decode attention on one GB300 (or N, one process per GPU).

A step is one pass of the hot path over one batch: append the step's new positions
into the paged pools (nbx_paged_kv_append), then split-KV decode attention for every
query row (nbx_paged_decode_attn: split plan, per-split partials, fixed-order merge).
Inputs are synthetic and seeded (workloads/), resident in HBM before timing starts.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

Prints ONE JSON line. value = K/V bytes read per step / device time per step (GB/s).
The L2 is flushed before every timed step, outside the timed events: a buffer of twice
its size is written, then read back, so no input and no dirty line is cached when the step starts. `--impl reference` times the float64 CPU oracle on this host instead.
"""

from __future__ import annotations

import os

# Each process of the CPU oracle leg runs one BLAS thread (the leg runs one process per core).
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import re
import json
import math
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "paged decode attn µs/step and KV-read GB/s (% of GB300 HBM peak)"
DEFAULT_CONFIG = "single_row"
KERNEL_SOURCES = ("paged_split_kv_append_gb300/csrc/decode_kernels.cuh",
                  "paged_split_kv_append_gb300/csrc/nbx_device.cuh",
                  "paged_split_kv_append_gb300/csrc/nbx_tcgen05.cuh",
                  "paged_split_kv_append_gb300/csrc/decode_common.cu",
                  "paged_split_kv_append_gb300/csrc/decode_mma.cu")


# ------------------------------------------------------------------------------------------ shared set-up
def session_for_case(case: "wl.Case", device, fill_nan: bool = True, prefill: bool = True):
    """The device state of one workload: pools prefilled through nbx_paged_kv_append with every
    position but the step's, and the step's inputs (queries, tables, lengths, new tokens)."""
    from paged_split_kv_append_gb300.session import PagedDecodeSession
    cfg = case.cfg
    sess = PagedDecodeSession(num_pages=case.num_pages, h_kv=cfg.h_kv, page_tokens=cfg.page_tokens, d=cfg.d,
                              pool_dtype=cfg.pool_dtype, batch=cfg.batch, rows=cfg.rows, h_q=cfg.h_q,
                              max_seq_len=case.max_seq_len, device=device, fill_nan=fill_nan,
                              q_dtype=cfg.q_dtype)
    sess.k_scale, sess.v_scale = case.k_scale, case.v_scale
    if prefill:
        idx, slots = case.prefill_index()
        sess.prefill(case.k_raw, case.v_raw, idx, slots)
    sidx, sslots = case.step_index()
    ii = torch.from_numpy(sidx).to(case.k_raw.device)
    sess.set_inputs(case.q, case.block_table, case.lens, case.k_raw.index_select(0, ii),
                    case.v_raw.index_select(0, ii), sslots, case.scale, case.k_scale, case.v_scale)
    return sess


def measured_peaks():
    """(HBM GB/s, dense bf16 TFLOP/s burst, source): the driver's measurement, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def attention_flops(case) -> float:
    """Algorithmic FLOPs of the step's attention: per (sequence, row, query head) that sees n keys,
    2*d*n for q.K^T and 2*d*n for P.V."""
    cfg = case.cfg
    n_vis = 0
    for L in case.lens.tolist():
        for r in range(cfg.rows):
            n_vis += min(max(int(L) - cfg.rows + r + 1, 0), int(L))
    return 4.0 * cfg.d * cfg.h_q * n_vis


_SOURCE_TOKEN = re.compile(r'"(?:\\.|[^"\\\n])*"|//[^\n]*|/\*.*?\*/', re.S)


def _code_only(text: str) -> str:
    """The source without its comments, blank lines and runs of whitespace (string literals, such as
    inline PTX, kept): what decides the compiled kernel."""
    text = _SOURCE_TOKEN.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", text)
    return "\n".join(line for line in (" ".join(raw.split()) for raw in text.splitlines()) if line)


def kernel_source_hash() -> str:
    """Identifies the kernel code the committed ncu counters were taken on; a change to comments
    alone keeps it."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, n_kv_bytes: int):
    """DRAM bytes per decode launch from the committed ncu summary, scaled to this workload's
    K/V bytes, or None when the kernel source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "decode_partial_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    ent = d.get("workloads", {}).get(workload)
    if not ent:
        return None
    return int(ent["dram_bytes_per_launch"] * n_kv_bytes / ent["kv_bytes"])


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return False
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)
        return False

    def summary(self):
        rows = getattr(self, "rows", [])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        busy = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------------------ CPU oracle leg
def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine() or "unknown"


class OracleGroups:
    """The float64 oracle on a fixed list of (sequence, KV head) groups, in one process.

    Set-up (not timed) builds the oracle's own pools with every prefill position of the groups'
    heads. A timed sample runs the groups in turn: the oracle's append of the sequence's new
    positions (this head) and attention for all of the group's query rows and heads."""

    def __init__(self, spec: dict):
        import oracle.paged as op
        self.op = op
        self.spec = spec
        P, dt = spec["page_tokens"], spec["pool_dtype"]
        shape = (spec["num_pages"], spec["h_kv"], P, spec["d"])
        self.kp = op.new_pool(*shape, dt)     # untouched pages of other heads stay unallocated
        self.vp = op.new_pool(*shape, dt)
        self.elt = {"f32": 4, "bf16": 2, "e4m3": 1}[dt]
        for g in spec["groups"]:
            L, n_new, hk = g["len"], g["n_new"], g["hk"]
            slots = (g["bt"][np.arange(L) // P].astype(np.int64) * P + np.arange(L) % P).astype(np.int32)
            g["slots"] = slots
            op.append(self.kp[:, hk:hk + 1], g["k"][:L - n_new, None], slots[:L - n_new], P, dt, spec["k_scale"])
            op.append(self.vp[:, hk:hk + 1], g["v"][:L - n_new, None], slots[:L - n_new], P, dt, spec["v_scale"])
        self.cursor = 0

    def sample(self, budget_s: float):
        """Run groups until about budget_s seconds passed; returns (K/V bytes, seconds, groups)."""
        op, sp = self.op, self.spec
        P, dt, G = sp["page_tokens"], sp["pool_dtype"], sp["h_q"] // sp["h_kv"]
        done, n = 0, 0
        t0 = time.perf_counter()
        while sp["groups"]:
            g = sp["groups"][self.cursor]
            L, n_new, hk = g["len"], g["n_new"], g["hk"]
            op.append(self.kp[:, hk:hk + 1], g["k"][L - n_new:, None], g["slots"][L - n_new:], P, dt, sp["k_scale"])
            op.append(self.vp[:, hk:hk + 1], g["v"][L - n_new:, None], g["slots"][L - n_new:], P, dt, sp["v_scale"])
            heads = [(0, r, h) for r in range(sp["rows"]) for h in range(hk * G, (hk + 1) * G)]
            op.decode_attention(g["q"][None], self.kp, self.vp, dt, g["bt"][None], np.array([L]), P, sp["scale"],
                                sp["k_scale"], sp["v_scale"], heads=heads)
            done += L * sp["d"] * self.elt * 2
            n += 1
            self.cursor = (self.cursor + 1) % len(sp["groups"])
            el = time.perf_counter() - t0
            if el >= budget_s:
                return done, el, n
        return 0, time.perf_counter() - t0, 0


def _oracle_worker(spec, conn):
    """One oracle process: build, report ready, then run one timed sample per request."""
    leg = OracleGroups(spec)
    conn.send("ready")
    while True:
        budget = conn.recv()
        if budget is None:
            break
        conn.send(leg.sample(budget))
    conn.close()


class OracleLeg:
    """The float64 CPU oracle as the CPU baseline, on every core of this host: the step's
    (sequence, KV head) groups are dealt, longest first, to one spawned process per core (each
    with one BLAS thread), and a timed sample runs all of them for the same wall-clock budget."""

    def __init__(self, case: "wl.Case", workers: int = 0):
        cfg = case.cfg
        groups = [(b, hk) for b in range(cfg.batch) for hk in range(cfg.h_kv) if int(case.lens[b]) > 0]
        groups.sort(key=lambda x: -int(case.lens[x[0]]))
        self.case = case
        self.workers = max(1, min(workers or host_cores(), len(groups) or 1))
        q = case.q.float().cpu().numpy()
        k_raw, v_raw = case.k_raw.cpu().numpy(), case.v_raw.cpu().numpy()
        specs = []
        for w in range(self.workers):
            mine = []
            for b, hk in groups[w::self.workers]:
                lo, hi = int(case.tok_offset[b]), int(case.tok_offset[b + 1])
                mine.append({"b": b, "hk": hk, "len": int(case.lens[b]), "n_new": int(case.n_new[b]),
                             "bt": case.block_table[b].copy(), "k": np.ascontiguousarray(k_raw[lo:hi, hk]),
                             "v": np.ascontiguousarray(v_raw[lo:hi, hk]), "q": q[b]})
            specs.append({"rows": cfg.rows, "h_q": cfg.h_q, "h_kv": cfg.h_kv, "d": cfg.d,
                          "page_tokens": cfg.page_tokens, "pool_dtype": cfg.pool_dtype, "num_pages": case.num_pages,
                          "scale": case.scale, "k_scale": case.k_scale, "v_scale": case.v_scale, "groups": mine})
        import multiprocessing as mp
        ctx = mp.get_context("spawn")     # never fork a process that holds a CUDA context
        self.conns, self.procs = [], []
        for spec in specs:
            parent, child = ctx.Pipe()
            proc = ctx.Process(target=_oracle_worker, args=(spec, child), daemon=True)
            proc.start()
            child.close()
            self.conns.append(parent)
            self.procs.append(proc)
        for c in self.conns:
            if c.recv() != "ready":
                raise RuntimeError("oracle worker failed to start")
        self.n_groups = len(groups)

    def sample(self, budget_s: float):
        """All workers run for about budget_s seconds; returns (K/V bytes, wall seconds, groups)."""
        t0 = time.perf_counter()
        for c in self.conns:
            c.send(budget_s)
        res = [c.recv() for c in self.conns]
        wall = time.perf_counter() - t0
        return sum(r[0] for r in res), wall, sum(r[2] for r in res)

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
            except (OSError, BrokenPipeError):
                pass
        for p in self.procs:
            p.join(timeout=30)

    def describe(self, groups: int) -> str:
        cfg = self.case.cfg
        return (f"{groups} (sequence, KV head) groups of the {cfg.name} step (of {self.n_groups} per step; each: "
                f"the oracle's append of the sequence's new positions and attention for its "
                f"{cfg.rows * cfg.group} query rows x heads), float64 numpy, {self.workers} processes "
                f"of one thread, groups dealt longest first")


# ------------------------------------------------------------------------------------------ GPU leg
def flush_l2(buf: torch.Tensor, sink: torch.Tensor):
    """Evict the L2 before a timed step: write the whole buffer (twice the L2 size), then read it
    back. The write evicts every input; the read evicts the write's own dirty lines, so their
    write-back to HBM happens here and not inside the timed region."""
    buf.add_(1)
    sink.add_(buf.sum())


def replica_seed(cfg, rank: int) -> int:
    """Seed of rank `rank`'s replica: every rank draws its own batch of the same workload (weak
    scaling; the path has no exchange step, so the ranks share nothing but the timing reduction)."""
    return cfg.seed + 1000 * rank


def pack_inputs(sess, dev):
    """Move the step's device inputs into one packed device buffer (sections 256-byte aligned) and
    return it with a pinned host copy of the same layout, so the inputs of a step travel in one
    host-to-device copy. The session's tensors become views of the packed buffer."""
    names = ("q", "block_table", "seq_lens", "new_k", "new_v", "new_slots")
    tensors = [(n, getattr(sess, n)) for n in names if getattr(sess, n) is not None]
    offs, total = [], 0
    for _, t in tensors:
        offs.append(total)
        total += -(-(t.numel() * t.element_size()) // 256) * 256
    dev_buf = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
    host_buf = torch.empty(max(total, 256), dtype=torch.uint8, pin_memory=True)
    for (n, t), o in zip(tensors, offs):
        nb = t.numel() * t.element_size()
        view = dev_buf[o:o + nb].view(t.dtype).view(t.shape)
        view.copy_(t)
        host_buf[o:o + nb].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
        setattr(sess, n, view)
    return dev_buf, host_buf, total


def time_fixed_shift(sess, steps: int, flush, sink, stream):
    """The fixed-shift ablation of a tensor-core window: its bounds pass and the decode call with the
    bounds (precomputed outside the timed decode), each timed like the decode call (graph replays)."""
    import paged_split_kv_append_gb300 as nbx
    with torch.cuda.stream(stream):
        qn, kv = nbx.nbx_paged_decode_bounds(sess.q, sess.k_pool, sess.v_pool, sess.block_table, sess.seq_lens,
                                             sess.max_seq_len, sess.k_scale, sess.v_scale, status=sess.status,
                                             stream=stream)

        def fixed():
            nbx.nbx_paged_decode_attn_fixed_shift(sess.q, sess.k_pool, sess.v_pool, sess.block_table, sess.seq_lens,
                                                  sess.max_seq_len, sess.scale, qn, kv, sess.k_scale, sess.v_scale,
                                                  out=sess.out, workspace=sess.workspace, status=sess.status,
                                                  stream=stream)

        def bounds():
            nbx.nbx_paged_decode_bounds(sess.q, sess.k_pool, sess.v_pool, sess.block_table, sess.seq_lens,
                                        sess.max_seq_len, sess.k_scale, sess.v_scale, status=sess.status,
                                        stream=stream)
        out = {}
        for name, fn in (("fixed_shift_decode_us", fixed), ("bounds_us", bounds)):
            fn()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            for a, b in evs:
                flush_l2(flush, sink)
                a.record(stream)
                g.replay()
                b.record(stream)
            stream.synchronize()
            out[name] = round(sum(a.elapsed_time(b) for a, b in evs) / steps * 1e3, 3)
    if sess.status_bits() != 0:
        raise RuntimeError(f"device status {sess.status_bits():#x} after the fixed-shift ablation")
    return out


def time_case(case, dev, steps: int, warmup: int, flush, sink, stream, e2e_steps: int = 0):
    """Time one workload's step (a CUDA-graph replay of append + decode) and its decode call alone
    (plan + partial + merge: a CUDA-graph replay, the device time of the three kernels, and the same
    call launched eagerly, which adds the host's launch gaps), each with the L2 flushed before every
    timed iteration; with e2e_steps, also the step end to end through the public API with host
    buffers."""
    sess = session_for_case(case, dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 1)):      # also configures the kernels before capture
            sess.step(stream=stream)
    stream.synchronize()
    if sess.status_bits() != 0:
        raise RuntimeError(f"device status {sess.status_bits():#x} after warm-up")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        sess.step(stream=stream)
    dgraph = torch.cuda.CUDAGraph()          # the decode call alone
    with torch.cuda.graph(dgraph, stream=stream):
        sess.decode(stream=stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush_l2(flush, sink)
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        for i in range(steps):               # the decode call alone, same flush discipline
            flush_l2(flush, sink)
            kev[i][0].record(stream)
            dgraph.replay()
            kev[i][1].record(stream)
        for i in range(steps):               # and launched eagerly
            flush_l2(flush, sink)
            eev[i][0].record(stream)
            sess.decode(stream=stream)
            eev[i][1].record(stream)
    stream.synchronize()
    if sess.status_bits() != 0:
        raise RuntimeError(f"device status {sess.status_bits():#x} after the timed steps")
    step_ms = [a.elapsed_time(b) for a, b in ev]
    dec_ms = [a.elapsed_time(b) for a, b in kev]
    eager_ms = [a.elapsed_time(b) for a, b in eev]
    # our kernels per call: append (when the step has new tokens), plan, partial, and the merge when
    # some sequence can have more than one split
    decode_launches = 2 + (1 if case.max_seq_len > 256 else 0)
    step_launches = decode_launches + (1 if (sess.new_k is not None and sess.new_k.shape[0] > 0) else 0)
    r = dict(step_ms=step_ms, ms_per_step=sum(step_ms) / len(step_ms), dec_ms=sum(dec_ms) / len(dec_ms),
             eager_ms=sum(eager_ms) / len(eager_ms), launches=(step_launches + 2 * decode_launches) * steps,
             partial=partial_kernel_name(case.cfg))
    if "mma" in r["partial"] and not e2e_steps:
        r["fixed_shift"] = time_fixed_shift(sess, steps, flush, sink, stream)
    if e2e_steps:
        # end to end: one H2D copy of the step's packed inputs from pinned memory, the step through
        # the public API, one D2H copy of the output, per step
        dev_buf, host_buf, h2d = pack_inputs(sess, dev)
        host_out = torch.empty(sess.out.shape, dtype=sess.out.dtype, pin_memory=True)
        e2e_ms = []
        with torch.cuda.stream(stream):
            for _ in range(e2e_steps):
                flush_l2(flush, sink)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                dev_buf.copy_(host_buf, non_blocking=True)
                sess.step(stream=stream)
                host_out.copy_(sess.out, non_blocking=True)
                b.record(stream)
                stream.synchronize()
                e2e_ms.append(a.elapsed_time(b))
        if sess.status_bits() != 0:
            raise RuntimeError(f"device status {sess.status_bits():#x} after the end-to-end steps")
        r.update(e2e_ms=sum(e2e_ms) / len(e2e_ms), h2d=h2d, d2h=host_out.numel() * host_out.element_size())
    del graph, sess
    return r


def roofline(case, dec_ms: float, peaks) -> dict:
    """The roof that bounds the decode call: tensor throughput when the step's arithmetic intensity
    (FLOPs per K/V byte) is above the ridge of the two measured peaks, else HBM bandwidth."""
    peak, tflops_peak, peak_kind = peaks
    kv = case.kv_bytes()
    flops = attention_flops(case)
    achieved_gbs = kv / (dec_ms * 1e-3) / 1e9
    if kv and flops / kv > tflops_peak * 1e12 / (peak * 1e9):
        tf = flops / (dec_ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": round(tf, 2), "peak": tflops_peak, "unit": "TFLOP/s",
                "frac": round(tf / tflops_peak, 4),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json bf16_tflops, dense bf16 burst)",
                "algorithmic_flops_per_launch": int(flops), "kv_gbs": round(achieved_gbs, 2)}
    return {"bound": "hbm", "achieved": round(achieved_gbs, 2), "peak": peak, "unit": "GB/s",
            "frac": round(achieved_gbs / peak, 4), "frac_of_nominal_8000": round(achieved_gbs / 8000.0, 4),
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s", "kv_gbs": round(achieved_gbs, 2)}


# the pages' own figure next to the one workload it matches (other hardware: context, not a target)
CONTEXT = {"verify": "TensorFold PR #1219 (rows-first grid): 16 query rows over 32k keys, 7.62 -> 4.67 ms "
                     "on GB10 (other hardware and model; context only)"}


def run_gpu(args, rank: int, world: int):
    dev = torch.device("cuda", torch.cuda.current_device())
    cfg = wl.CONFIGS[args.config]
    case = wl.make_case(cfg, device=dev, seed=replica_seed(cfg, rank))
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.zeros(max(2 * l2, 1 << 20) // 4, dtype=torch.float32, device=dev)
    sink = torch.zeros(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        r = time_case(case, dev, args.steps, args.warmup, flush, sink, stream,
                      e2e_steps=max(3, min(args.steps, 50)))
    barrier(world)
    torch.cuda.synchronize()
    kv_bytes = case.kv_bytes()
    out = dict(case=case, kv_bytes=kv_bytes, total_bytes=all_reduce_sum(float(kv_bytes), world),
               ms_per_step=all_reduce_max(r["ms_per_step"], world), dec_ms=all_reduce_max(r["dec_ms"], world),
               eager_ms=all_reduce_max(r["eager_ms"], world),
               e2e_ms=all_reduce_max(r["e2e_ms"], world), h2d=r["h2d"], d2h=r["d2h"], clocks=clocks.summary(),
               launches=r["launches"], step_ms=r["step_ms"], partial=r["partial"])
    # every other workload, timed the same way (one GPU only: they are not replicas)
    per = {}
    if world == 1 and args.per_config:
        peaks = measured_peaks()
        steps = max(10, min(args.steps, 200))
        for name in wl.FULL_CONFIGS:
            if name == args.config:
                continue
            c = wl.make_case(wl.CONFIGS[name], device=dev, seed=wl.CONFIGS[name].seed)
            with ClockSampler(dev.index) as clk:
                rr = time_case(c, dev, steps, args.warmup, flush, sink, stream)
            roof = roofline(c, rr["dec_ms"], peaks)
            per[name] = {"partial_kernel": rr["partial"], "steps": steps, "us_per_step": round(rr["ms_per_step"] * 1e3, 3),
                         "step_kv_gbs": round(c.kv_bytes() / (rr["ms_per_step"] * 1e-3) / 1e9, 2),
                         "decode_us": round(rr["dec_ms"] * 1e3, 3),
                         "decode_eager_us": round(rr["eager_ms"] * 1e3, 3), "kv_bytes": int(c.kv_bytes()),
                         "roofline": {**roof, "traffic": profiled_traffic(name, c.kv_bytes())},
                         "clocks": clk.summary()}
            if "fixed_shift" in rr:
                per[name]["fixed_shift_ablation"] = {
                    **rr["fixed_shift"],
                    "what": "decode call with the fixed-shift softmax (maxdiffusion PR #477) where the score bound "
                            "passes the gate, bounds precomputed; bounds_us is the pass that computes them"}
            if name in CONTEXT:
                per[name]["context"] = CONTEXT[name]
            del c
            torch.cuda.empty_cache()
    out["per_config"] = per
    return out


def partial_kernel_name(cfg) -> str:
    import paged_split_kv_append_gb300 as nbx
    code = {"f32": nbx.NBX_F32, "bf16": nbx.NBX_BF16, "e4m3": nbx.NBX_E4M3}
    kind = nbx.nbx_paged_decode_partial_kernel(code[cfg.q_dtype], code[cfg.pool_dtype], cfg.rows, cfg.h_q, cfg.h_kv,
                                               cfg.d, 1, cfg.page_tokens)
    return "decode_partial_kernel" if kind == nbx.PARTIAL_SIMT else "decode_partial_mma_kernel"


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def all_reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def all_reduce_sum(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def config_block(case, args, arm: str = "gpu"):
    cfg = case.cfg
    kind = cfg.lens[0]
    if kind == "fixed":
        vals = list(cfg.lens[1])
        lens = f"fixed {vals[:4]}{'...' if len(vals) > 4 else ''}"
    elif kind == "uniform":
        lens = f"uniform[{cfg.lens[1]},{cfg.lens[2]}]"
    else:
        lens = f"log-uniform[{cfg.lens[1]},{cfg.lens[2]}]"
    return {"workload": cfg.name, "batch": cfg.batch, "rows": cfg.rows, "h_q": cfg.h_q, "h_kv": cfg.h_kv,
            "d": cfg.d, "page_tokens": cfg.page_tokens, "kv_dtype": cfg.pool_dtype, "q_dtype": cfg.q_dtype,
            "seq_lens": f"{lens} seed {cfg.seed}", "kv_bytes_per_step": int(case.kv_bytes()),
            "l2": "flushed before every timed step, outside the events: a 2x-L2 buffer written, then read back (no input and no dirty line in L2 when the step starts)" if arm == "gpu"
            else "n/a (CPU)",
            "step": "append of the step's new positions + split plan + split-KV partial + fixed-order merge"
            if arm == "gpu" else "the oracle's append of the new positions + float64 attention, bounded sample",
            "timing": "CUDA events per step around a CUDA-graph replay of the step; the roofline's decode call "
                      "(plan + partial + merge) likewise around a graph replay of the call alone, with the eagerly "
                      "launched call's time beside it (us_per_launch_eager)" if arm == "gpu"
            else "wall clock (time.perf_counter) around each sample"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(wl.CONFIGS))
    ap.add_argument("--impl", default="nbx", choices=["nbx", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work in the CPU leg")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="time only --config, not the other workloads")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args)
        return

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    import paged_split_kv_append_gb300 as nbx
    nbx.build()

    r = run_gpu(args, rank, world)
    case = r["case"]
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    peaks = measured_peaks()
    ms = r["ms_per_step"]
    value = r["total_bytes"] / (ms * 1e-3) / 1e9
    roof = roofline(case, r["dec_ms"], peaks)
    traffic = profiled_traffic(case.cfg.name, r["kv_bytes"])
    cpu_bytes, cpu_s, cpu_desc, cores = 0, 0.0, "skipped", 0
    if args.cpu_budget > 0:
        leg = OracleLeg(wl.make_case(case.cfg, device="cpu"))
        try:
            cpu_bytes, cpu_s, n_groups = leg.sample(args.cpu_budget)
            cpu_desc, cores = leg.describe(n_groups), leg.workers
        finally:
            leg.close()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 6),
        "us_per_step": round(ms * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded: workloads/)",
        "config": config_block(case, args),
        "roofline": {"kernel": f"decode call (plan_kernel + {r['partial']} + decode_merge_kernel)", **roof,
                     "us_per_launch": round(r["dec_ms"] * 1e3, 3),
                     "us_per_launch_eager": round(r["eager_ms"] * 1e3, 3), "traffic": traffic,
                     "algorithmic_bytes_per_launch": int(r["kv_bytes"])},
        "per_config": r["per_config"],
        "cpu_baseline": {"value": round(cpu_bytes / cpu_s / 1e9, 4) if cpu_s > 0 else None, "unit": "GB/s",
                         "cores": cores, "cpu_model": cpu_model(), "host_cores": host_cores(), "kind": "oracle",
                         "sample": cpu_desc, "seconds": round(cpu_s, 3)},
        "e2e": {"value": round(r["total_bytes"] / (r["e2e_ms"] * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(r["e2e_ms"], 6), "h2d_bytes_per_step": int(r["h2d"]),
                "d2h_bytes_per_step": int(r["d2h"])},
        "gpu_launches": int(r["launches"]),
        "clocks": r["clocks"],
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The reference arm: the float64 CPU oracle, as it stands, on every core of this host; every step
    a bounded sample of the workload's step, sized so the whole run takes about two minutes."""
    cfg = wl.CONFIGS[args.config]
    leg = OracleLeg(wl.make_case(cfg, device="cpu"))
    try:
        per_step = min(2.0, max(0.05, 120.0 / max(1, args.steps + args.warmup)))
        for _ in range(args.warmup):
            leg.sample(per_step)
        tot_bytes, tot_s, tot_groups = 0, 0.0, 0
        for _ in range(args.steps):
            b, s, g = leg.sample(per_step)
            tot_bytes += b
            tot_s += s
            tot_groups += g
    finally:
        leg.close()
    value = tot_bytes / tot_s / 1e9 if tot_s > 0 else None
    v = round(value, 4) if value else None
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_s / max(1, args.steps) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded: workloads/)",
        "config": config_block(leg.case, args, arm="oracle"),
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": leg.workers, "cpu_model": cpu_model(),
                         "host_cores": host_cores(), "kind": "oracle",
                         "sample": f"per step ~{per_step:.3f} s: " + leg.describe(tot_groups // max(1, args.steps))},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
