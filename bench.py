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

# The CPU oracle leg is single-threaded and says so (its BLAS calls are matrix-vector products).
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
                  "paged_split_kv_append_gb300/csrc/decode_common.cu",
                  "paged_split_kv_append_gb300/csrc/decode_mma.cu")


# ------------------------------------------------------------------------------------------ shared set-up
def session_for_case(case: "wl.Case", device, fill_nan: bool = True, prefill: bool = True, widen: bool = True):
    """The device state of one workload: pools prefilled through nbx_paged_kv_append with every
    position but the step's, and the step's inputs (queries, tables, lengths, new tokens).
    widen=False sizes the workspace without room for the bf16 copies of an fp8 pool."""
    from paged_split_kv_append_gb300.session import PagedDecodeSession
    cfg = case.cfg
    sess = PagedDecodeSession(num_pages=case.num_pages, h_kv=cfg.h_kv, page_tokens=cfg.page_tokens, d=cfg.d,
                              pool_dtype=cfg.pool_dtype, batch=cfg.batch, rows=cfg.rows, h_q=cfg.h_q,
                              max_seq_len=case.max_seq_len, device=device, fill_nan=fill_nan,
                              q_dtype=cfg.q_dtype, widen=widen)
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
class OracleLeg:
    """The float64 CPU oracle run on this host as the CPU baseline. Set-up (not timed) builds
    the oracle's own pools with every prefill position. A timed sample is a bounded part of the
    step: (sequence, KV head) groups taken in order, each with the oracle's append of that
    sequence's new positions and attention for all of the group's query rows and heads."""

    def __init__(self, case: "wl.Case"):
        import oracle.paged as op
        self.op = op
        self.case = case
        cfg = case.cfg
        self.kp = op.new_pool(case.num_pages, cfg.h_kv, cfg.page_tokens, cfg.d, cfg.pool_dtype)
        self.vp = op.new_pool(case.num_pages, cfg.h_kv, cfg.page_tokens, cfg.d, cfg.pool_dtype)
        self.q = case.q.float().cpu().numpy()
        self.k_new, self.v_new, self.s_new = [], [], []
        for b in range(cfg.batch):
            L, n_new = int(case.lens[b]), int(case.n_new[b])
            lo, hi = int(case.tok_offset[b]), int(case.tok_offset[b + 1])
            slots = wl.slots_for(case.block_table, cfg.page_tokens, b, np.arange(L, dtype=np.int64))
            kk = case.k_raw[lo:hi].cpu().numpy()
            vv = case.v_raw[lo:hi].cpu().numpy()
            op.append(self.kp, kk[:L - n_new], slots[:L - n_new], cfg.page_tokens, cfg.pool_dtype, case.k_scale)
            op.append(self.vp, vv[:L - n_new], slots[:L - n_new], cfg.page_tokens, cfg.pool_dtype, case.v_scale)
            self.k_new.append(kk[L - n_new:].copy())
            self.v_new.append(vv[L - n_new:].copy())
            self.s_new.append(slots[L - n_new:].copy())
        self.cursor = 0
        self.elt = {"f32": 4, "bf16": 2, "e4m3": 1}[cfg.pool_dtype]

    def sample(self, budget_s: float):
        """Run groups until about budget_s seconds passed; returns (K/V bytes, seconds, groups)."""
        op, case, cfg = self.op, self.case, self.case.cfg
        G = cfg.group
        n_groups = cfg.batch * cfg.h_kv
        done, groups = 0, 0
        t0 = time.perf_counter()
        while True:
            b, hk = divmod(self.cursor, cfg.h_kv)
            if hk == 0:
                op.append(self.kp, self.k_new[b], self.s_new[b], cfg.page_tokens, cfg.pool_dtype, case.k_scale)
                op.append(self.vp, self.v_new[b], self.s_new[b], cfg.page_tokens, cfg.pool_dtype, case.v_scale)
            heads = [(0, r, h) for r in range(cfg.rows) for h in range(hk * G, (hk + 1) * G)]
            op.decode_attention(self.q[b:b + 1], self.kp, self.vp, cfg.pool_dtype, case.block_table[b:b + 1],
                                case.lens[b:b + 1], cfg.page_tokens, case.scale, case.k_scale, case.v_scale,
                                heads=heads)
            done += int(case.lens[b]) * cfg.d * self.elt * 2
            groups += 1
            self.cursor = (self.cursor + 1) % n_groups
            el = time.perf_counter() - t0
            if el >= budget_s:
                return done, el, groups

    def describe(self, groups: int) -> str:
        cfg = self.case.cfg
        return (f"{groups} (sequence, KV head) groups of the {cfg.name} step (of {cfg.batch * cfg.h_kv} per step; "
                f"each: the oracle's append of the sequence's new positions and attention for its "
                f"{cfg.rows * cfg.group} query rows x heads), float64 numpy, 1 thread")


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


def run_gpu(args, rank: int, world: int):
    import paged_split_kv_append_gb300 as nbx
    dev = torch.device("cuda", torch.cuda.current_device())
    cfg = wl.CONFIGS[args.config]
    seed = replica_seed(cfg, rank)
    case = wl.make_case(cfg, device=dev, seed=seed)
    sess = session_for_case(case, dev)
    torch.cuda.synchronize()
    kv_bytes = case.kv_bytes()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.zeros(max(2 * l2, 1 << 20) // 4, dtype=torch.float32, device=dev)
    sink = torch.zeros(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    # warm-up (also configures the kernels before capture)
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 1)):
            sess.step(stream=stream)
    stream.synchronize()
    if sess.status_bits() != 0:
        raise RuntimeError(f"device status {sess.status_bits():#x} after warm-up")

    # the step as a CUDA graph: append + plan + partial, replayed per timed step
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        sess.step(stream=stream)
    # our kernels per call: append (when the step has new tokens), plan, partial, and the merge
    # when some sequence can have more than one split
    merge = 1 if case.max_seq_len > 256 else 0
    widen = 1 if partial_kernel_name(cfg).startswith("widen") else 0
    decode_launches = 2 + merge + widen
    launches_per_step = decode_launches + (1 if (sess.new_k is not None and sess.new_k.shape[0] > 0) else 0)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush_l2(flush, sink)
                ev[i][0].record(stream)
                graph.replay()
                ev[i][1].record(stream)
            # the dominant kernel alone (plan + partial, no append), same flush discipline
            for i in range(args.steps):
                flush_l2(flush, sink)
                kev[i][0].record(stream)
                sess.decode(stream=stream)
                kev[i][1].record(stream)
        stream.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    dec_ms = [a.elapsed_time(b) for a, b in kev]
    if sess.status_bits() != 0:
        raise RuntimeError(f"device status {sess.status_bits():#x} after the timed steps")
    ms_per_step = sum(step_ms) / len(step_ms)
    dec_ms_mean = sum(dec_ms) / len(dec_ms)

    # end to end through the public API with host buffers: H2D of the step's inputs from pinned
    # memory, the step, D2H of the output, per step
    host_in = {k: t.cpu().pin_memory() for k, t in (("q", sess.q), ("bt", sess.block_table),
                                                       ("lens", sess.seq_lens), ("nk", sess.new_k),
                                                       ("nv", sess.new_v), ("ns", sess.new_slots))
               if t is not None}
    host_out = torch.empty(sess.out.shape, dtype=sess.out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out.numel() * host_out.element_size()
    dst = {"q": sess.q, "bt": sess.block_table, "lens": sess.seq_lens, "nk": sess.new_k, "nv": sess.new_v,
           "ns": sess.new_slots}
    e2e_steps = max(3, min(args.steps, 50))
    e2e_ms = []
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            flush_l2(flush, sink)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for k, t in host_in.items():
                dst[k].copy_(t, non_blocking=True)
            sess.step(stream=stream)
            host_out.copy_(sess.out, non_blocking=True)
            b.record(stream)
            stream.synchronize()
            e2e_ms.append(a.elapsed_time(b))
    e2e_ms_mean = sum(e2e_ms) / len(e2e_ms)

    t_max = all_reduce_max(ms_per_step, world)
    dec_max = all_reduce_max(dec_ms_mean, world)
    e2e_max = all_reduce_max(e2e_ms_mean, world)
    total_bytes = all_reduce_sum(float(kv_bytes), world)
    return dict(case=case, kv_bytes=kv_bytes, total_bytes=total_bytes, ms_per_step=t_max, dec_ms=dec_max,
                e2e_ms=e2e_max, h2d=h2d, d2h=d2h, clocks=clocks.summary(),
                launches=(launches_per_step + decode_launches) * args.steps, step_ms=step_ms,
                partial=partial_kernel_name(cfg))


def partial_kernel_name(cfg) -> str:
    import paged_split_kv_append_gb300 as nbx
    code = {"f32": nbx.NBX_F32, "bf16": nbx.NBX_BF16, "e4m3": nbx.NBX_E4M3}
    kind = nbx.nbx_paged_decode_partial_kernel(code[cfg.q_dtype], code[cfg.pool_dtype], cfg.rows, cfg.h_q, cfg.h_kv,
                                               cfg.d, 1, cfg.page_tokens)
    if kind == nbx.PARTIAL_TCGEN05_WIDENED:
        return "widen_kernel + decode_partial_mma_kernel"
    return "decode_partial_mma_kernel" if kind == nbx.PARTIAL_TCGEN05 else "decode_partial_kernel"


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
            "timing": "CUDA events per step around a CUDA-graph replay of the step" if arm == "gpu"
            else "wall clock (time.perf_counter) around each sample"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(wl.CONFIGS))
    ap.add_argument("--impl", default="nbx", choices=["nbx", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work in the CPU leg")
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
    peak, tflops_peak, peak_kind = measured_peaks()
    ms = r["ms_per_step"]
    value = r["total_bytes"] / (ms * 1e-3) / 1e9
    dec_achieved = r["kv_bytes"] / (r["dec_ms"] * 1e-3) / 1e9
    flops = attention_flops(case)
    # the roof that bounds the decode call: tensor throughput when the step's arithmetic intensity
    # (FLOPs per K/V byte) is above the ridge of the two measured peaks, else HBM bandwidth
    tensor_bound = flops / r["kv_bytes"] > tflops_peak * 1e12 / (peak * 1e9)
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": round(flops / (r["dec_ms"] * 1e-3) / 1e12, 2), "peak": tflops_peak,
                "unit": "TFLOP/s", "frac": round(flops / (r["dec_ms"] * 1e-3) / 1e12 / tflops_peak, 4),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json bf16_tflops, dense bf16 burst)",
                "algorithmic_flops_per_launch": int(flops)}
    else:
        roof = {"bound": "hbm", "achieved": round(dec_achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(dec_achieved / peak, 4), "frac_of_nominal_8000": round(dec_achieved / 8000.0, 4),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s"}
    traffic = profiled_traffic(case.cfg.name, r["kv_bytes"])
    if args.cpu_budget > 0:
        leg = OracleLeg(wl.make_case(case.cfg, device="cpu"))
        cpu_bytes, cpu_s, n_groups = leg.sample(args.cpu_budget)
        cpu_desc = leg.describe(n_groups)
    else:
        cpu_bytes, cpu_s, cpu_desc = 0, 0.0, "skipped"
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
                     "us_per_launch": round(r["dec_ms"] * 1e3, 3), "traffic": traffic,
                     "algorithmic_bytes_per_launch": int(r["kv_bytes"]),
                     "kv_gbs": round(dec_achieved, 2)},
        "cpu_baseline": {"value": round(cpu_bytes / cpu_s / 1e9, 4) if cpu_s > 0 else None, "unit": "GB/s",
                         "cores": 1, "kind": "oracle", "sample": cpu_desc,
                         "seconds": round(cpu_s, 3)},
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
    """The reference arm: the float64 CPU oracle, as it stands, on this host's cores; every step a
    bounded sample of the workload's step, sized so the whole run takes about two minutes."""
    cfg = wl.CONFIGS[args.config]
    leg = OracleLeg(wl.make_case(cfg, device="cpu"))
    per_step = min(2.0, max(0.02, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        leg.sample(per_step)
    tot_bytes, tot_s, tot_groups = 0, 0.0, 0
    for _ in range(args.steps):
        b, s, g = leg.sample(per_step)
        tot_bytes += b
        tot_s += s
        tot_groups += g
    value = tot_bytes / tot_s / 1e9 if tot_s > 0 else None
    v = round(value, 4) if value else None
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_s / max(1, args.steps) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded: workloads/)",
        "config": config_block(leg.case, args, arm="oracle"),
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"per step ~{per_step:.3f} s: " + leg.describe(tot_groups // max(1, args.steps))},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
