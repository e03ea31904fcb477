"""Benchmark: fused mask + top-k / top-p / min-p sample at B=256, V=128,256 f32.

One step = one `sample` call over one batch of synthetic decode logits with a
per-row grammar mask applied on load (the bitmask apply, max / argmax,
temperature softmax normaliser, keep-threshold and Gumbel-max draw, all in one
kernel).  The standalone bitmask apply and the exact top-k are timed in the
same run and reported under "per_op".

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun (N > 1) every rank runs its own batch (replicas: the rows of a
decode batch are independent), a barrier brackets the timed region and rank 0
prints one JSON line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
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

import workloads  # noqa: E402

METRIC = "rows/s and achieved HBM GB/s, fused mask+top-k/p/min-p sample, B=256 V=128256"
B, V = 256, 128256
MASK_DENSITY = 0.7
SAMPLE_LAUNCHES = 1  # kernels one sample call launches at B=256 (one CTA per row)
N_BUFFERS = 4  # inputs rotate over 4 device copies (each 135 MB > L2)


def algorithmic_bytes(B, V, esize, mask=True):
    """Logit bytes read once + mask bytes + per-row outputs (8 B token)."""
    return B * V * esize + (B * ((V + 31) // 32) * 4 if mask else 0) + B * 8


# DRAM bytes (read + write) per sample call on the headline workload, from an
# ncu capture of the kernel on that workload (dram__bytes_read.sum +
# dram__bytes_write.sum, one launch).  They hold only for the kernel sources
# they were taken on: a changed source reports null.
TRAFFIC_SOURCES = ('tsa_sample_row.cuh', 'tsa_sample_row.cu', 'tsa_sample_row_spec_f32.cu', 'tsa_sample_common.cuh',
                   'tsa_select.cuh', 'tsa_device.cuh', 'tsa_host.h')
TRAFFIC = {"sha256": "086f2f2cf85c1a65d115506c81d0f56311784ce73d46a005d44010f8d98d448b",
           "bytes": 135_547_904 + 3_009_280}


def sample_traffic():
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "top_sampling_apply_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return TRAFFIC["bytes"] if h.hexdigest() == TRAFFIC["sha256"] else None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workload
def make_inputs(seed=0):
    case = workloads.decode_batch("combined", mask_density=MASK_DENSITY, B=B, V=V, seed=seed)
    return case


REF_BUDGET_S = 120.0  # wall-clock the reference arm's timed steps may take


def reference_rows_per_step(steps, cores, sec_per_row_core, budget_s=REF_BUDGET_S, cap=B):
    """Rows of the batch the oracle handles per reference step: a multiple of
    the core count (one row per thread per round), as many rounds as fit
    `steps` steps into `budget_s` seconds, at least one round and at most
    the whole batch."""
    rounds = int(budget_s / max(1e-9, steps * sec_per_row_core))
    return max(1, min(cap, cores * max(1, rounds)))


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, on the host cores, on
    a bounded sample of the same workload and the same metric.  Each step is
    a sample of the batch's rows sized so that all steps end within a few
    minutes.  Under several ranks only rank 0 runs it."""
    import oracle

    if rank != 0:
        return None
    case = make_inputs()
    nthreads = os.cpu_count() or 1
    T, K, P, MP = (case.temperature, case.top_k, case.top_p, case.min_p)
    # calibrate: one row per thread (also the first warm-up step)
    t0 = time.perf_counter()
    oracle.sample(case.logits[:nthreads], T, K, P, MP, seed=0, offset=0,
                  bitmask=case.bitmask[:nthreads], nthreads=nthreads)
    per_row_core = time.perf_counter() - t0
    rows = reference_rows_per_step(args.steps, nthreads, per_row_core)
    x = case.logits[:rows]
    m = case.bitmask[:rows]
    for w in range(1, args.warmup):
        oracle.sample(x, T, K, P, MP, seed=w, offset=w, bitmask=m, nthreads=nthreads)
    t0 = time.perf_counter()
    for s in range(args.steps):
        oracle.sample(x, T, K, P, MP, seed=s, offset=s, bitmask=m, nthreads=nthreads)
    dt = (time.perf_counter() - t0) / args.steps
    rps = rows / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": rps, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": headline_config(world),
        "cpu_baseline": {"value": rps, "unit": "rows/s", "cores": nthreads, "kind": "oracle",
                         "sample": "%d of the 256 rows per step, full sort per row" % rows},
        "e2e": {"value": rps, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def headline_config(world):
    """The headline workload's `config`, the same on both arms."""
    return {"workload": "decode batch B=256 V=128256 f32 logits 3N(0,1)+Zipf(1.1) "
                        "log-rank head, per-row mask density 0.7 fused on load, "
                        "T=1 top_k=50 top_p=0.9 min_p=0.05, seed=offset=step",
            "rows_per_gpu": B, "vocab": V,
            "l2": "inputs larger than L2 (135 MB per step), rotated over %d buffers" % N_BUFFERS,
            "parallelism": "replicas" if world > 1 else "single"}


def cpu_baseline_sample():
    """The oracle timed on the host cores on a bounded sample (64 rows x 4
    draws of the same workload), reported beside the GPU number, with the
    same oracle on one thread (16 rows x 2 draws) beside it."""
    import oracle

    case = make_inputs()
    nthreads = os.cpu_count() or 1

    def rate(rows, reps, nt):
        x, m = case.logits[:rows], case.bitmask[:rows]
        oracle.sample(x[:nt], 1.0, 50, 0.9, 0.05, seed=0, bitmask=m[:nt], nthreads=nt)  # warm-up
        t0 = time.perf_counter()
        for s in range(reps):
            oracle.sample(x, 1.0, 50, 0.9, 0.05, seed=s, offset=s, bitmask=m, nthreads=nt)
        return rows * reps / (time.perf_counter() - t0)

    all_cores = rate(64, 4, nthreads)
    one = rate(16, 2, 1)
    return {"value": all_cores, "unit": "rows/s", "cores": nthreads, "kind": "oracle",
            "sample": "%d rows x %d draws of the B=256 V=128256 masked combined workload" % (64, 4),
            "single_thread": {"value": one, "unit": "rows/s", "cores": 1,
                              "sample": "16 rows x 2 draws of the same workload"}}


class GraphSteps:
    """fn(i) for i in range(n), captured once into CUDA graphs (blocks of up to
    64 calls) so that Python launch overhead stays out of device timings."""

    def __init__(self, fn, n, block=64):
        self.graphs = []
        i = 0
        while i < n:
            m = min(block, n - i)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for j in range(i, i + m):
                    fn(j)
            self.graphs.append(g)
            i += m

    def replay(self):
        for g in self.graphs:
            g.replay()


def time_op(fn, iters, stream, warm=3):
    """Average device time of fn(i) over `iters` calls replayed from CUDA
    graphs, CUDA events on the launching stream, synchronised on both sides."""
    for i in range(warm):
        fn(i)
    torch.cuda.synchronize()
    gs = GraphSteps(fn, iters)
    gs.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    gs.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def per_op_breakdown(tsa, dev, stream, hbm_peak):
    """Every other row of the path, timed in the same run (not in the headline
    timed region)."""
    out = {}
    # the five unmasked decode modes
    base = workloads.decode_batch("greedy", mask_density=None, B=B, V=V)
    bufs = [base.logits.to(dev) for _ in range(N_BUFFERS)]
    nbytes = algorithmic_bytes(B, V, 4, mask=False)
    for mode, (T, K, P, MP) in workloads.DECODE_MODES.items():
        ms = time_op(lambda i: tsa.sample(bufs[i % N_BUFFERS], T, K, P, MP, seed=i, offset=i), 40,
                     stream)
        out["decode_" + mode] = {"ms": ms, "rows_per_s": B / ms * 1e3,
                                 "GB_per_s": nbytes / ms / 1e6,
                                 "frac_hbm": nbytes / ms / 1e6 / hbm_peak}
    # standalone in-place bitmask apply on the same batch
    mcase = workloads.decode_batch("greedy", mask_density=MASK_DENSITY, B=B, V=V)
    mask = mcase.bitmask.to(dev)
    ms = time_op(lambda i: tsa.apply_token_bitmask(bufs[i % N_BUFFERS], mask), 40, stream)
    disallowed = int((~torch.from_numpy(np.unpackbits(mcase.bitmask.numpy().view(np.uint8), axis=1,
                                                      bitorder="little")[:, :V].astype(bool))).sum())
    mb = mask.numel() * 4 + disallowed * 4
    out["apply_token_bitmask"] = {"ms": ms, "GB_per_s": mb / ms / 1e6,
                                  "bytes": mb, "note": "mask read + -inf writes only"}
    # selective log-softmax of the masked batch at one index a row (one read of the rows)
    idx = (torch.arange(B, device=dev, dtype=torch.int64) * 7919) % V
    ms = time_op(lambda i: tsa.selective_log_softmax(bufs[i % N_BUFFERS], idx, 1.0, bitmask=mask), 40, stream)
    lb = B * V * 4 + mask.numel() * 4 + B * 12
    out["selective_log_softmax"] = {"ms": ms, "rows_per_s": B / ms * 1e3, "GB_per_s": lb / ms / 1e6,
                                    "frac_hbm": lb / ms / 1e6 / hbm_peak}
    del bufs
    # f1's sequential top-p and f3's inverse-CDF draw on the masked combined batch
    cc = workloads.decode_batch("combined", mask_density=MASK_DENSITY, B=B, V=V)
    cx = [cc.logits.to(dev) for _ in range(N_BUFFERS)]
    cm = cc.bitmask.to(dev)
    Tc, Kc, Pc, Mc = cc.temperature, cc.top_k, cc.top_p, cc.min_p
    nbytes_m = algorithmic_bytes(B, V, 4, mask=True)
    ms = time_op(lambda i: tsa.sample(cx[i % N_BUFFERS], Tc, Kc, Pc, Mc, seed=i, offset=i, bitmask=cm,
                                      sequential=True), 40, stream)
    out["sequential_combined_mask"] = {"ms": ms, "rows_per_s": B / ms * 1e3, "GB_per_s": nbytes_m / ms / 1e6,
                                       "note": "three reads of the batch: top-k cut, survivors' mask, filters"}
    u = torch.rand(B, device=dev)
    ms = time_op(lambda i: tsa.sample_icdf(cx[i % N_BUFFERS], u, Tc, Kc, Pc, Mc, bitmask=cm), 40, stream)
    out["icdf_combined_mask"] = {"ms": ms, "rows_per_s": B / ms * 1e3, "GB_per_s": nbytes_m / ms / 1e6,
                                 "note": "the sample call, then one more read of the batch"}
    allowed = torch.from_numpy(np.unpackbits(cc.bitmask.numpy().view(np.uint8), axis=1,
                                             bitorder="little")[:, :V].astype(bool)).to(dev)
    ms = time_op(lambda i: tsa.bitmask_from_allowed(allowed), 40, stream)
    ab = B * V + B * ((V + 31) // 32) * 4
    out["bitmask_from_allowed"] = {"ms": ms, "GB_per_s": ab / ms / 1e6, "frac_hbm": ab / ms / 1e6 / hbm_peak}
    del cx, allowed
    # the dense lm-head fused with top-k: V=248,320, H=5,120, bf16 random weights
    lw = torch.empty(248320, 5120, dtype=torch.bfloat16, device=dev)
    lw.normal_(0.0, 0.02, generator=torch.Generator(device=dev).manual_seed(0))
    lh = torch.randn(4, 5120, device=dev, generator=torch.Generator(device=dev).manual_seed(1)).to(torch.bfloat16)
    for M, k in ((1, 50), (4, 50), (1, 2048)):
        ms = time_op(lambda i: tsa.lm_head_topk(lh[:M], lw, k), 20, stream)
        wb = lw.numel() * 2
        out["lm_head_topk_m%d_k%d" % (M, k)] = {"ms": ms, "GB_per_s": wb / ms / 1e6,
                                                 "frac_hbm": wb / ms / 1e6 / hbm_peak}
    del lw
    # exact top-k at V=248,320
    for k in (50, 2048):
        x, _ = workloads.topk_large(k)
        xs = [x.to(dev) for _ in range(N_BUFFERS)]
        ms = time_op(lambda i: tsa.topk(xs[i % N_BUFFERS], k), 40, stream)
        tb = x.numel() * 4 + x.shape[0] * k * 12
        out["topk_k%d" % k] = {"ms": ms, "GB_per_s": tb / ms / 1e6, "frac_hbm": tb / ms / 1e6 / hbm_peak}
    # heterogeneous bf16 batch and large peaked bf16 batch
    h = workloads.hetero_batch()
    hx = [h.logits.to(dev) for _ in range(N_BUFFERS)]
    hm = h.bitmask.to(dev)
    hp = [p.to(dev) for p in (h.temperature, h.top_k, h.top_p, h.min_p)]
    ms = time_op(lambda i: tsa.sample(hx[i % N_BUFFERS], *hp, seed=i, offset=i, bitmask=hm), 40, stream)
    hb = h.B * h.V * 2 + hm.numel() * 4 + h.B * 24
    out["hetero_bf16"] = {"ms": ms, "rows_per_s": h.B / ms * 1e3, "GB_per_s": hb / ms / 1e6,
                          "frac_hbm": hb / ms / 1e6 / hbm_peak}
    del hx
    pk = workloads.peaked_batch()
    px = [pk.logits.to(dev) for _ in range(3)]
    pm = pk.bitmask.to(dev)
    ms = time_op(lambda i: tsa.sample(px[i % 3], 0.8, 0, 0.95, 0.05, seed=i, offset=i, bitmask=pm), 40,
                 stream)
    pb = pk.B * pk.V * 2 + pm.numel() * 4 + pk.B * 8
    out["peaked_bf16"] = {"ms": ms, "rows_per_s": pk.B / ms * 1e3, "GB_per_s": pb / ms / 1e6,
                          "frac_hbm": pb / ms / 1e6 / hbm_peak}
    return out


def _profile_hetero(tsa, dev):
    h = workloads.hetero_batch()
    x, m = h.logits.to(dev), h.bitmask.to(dev)
    p = [v.to(dev) for v in (h.temperature, h.top_k, h.top_p, h.min_p)]
    return lambda i: tsa.sample(x, *p, seed=i, offset=i, bitmask=m)


def _profile_peaked(tsa, dev, flat_only=False):
    pk = workloads.peaked_batch()
    x, m = pk.logits.to(dev), pk.bitmask.to(dev)
    if flat_only:  # the batch's flat rows alone (all 0.0), one CTA each
        rows = torch.tensor(pk.info["flat_rows"], device=dev)
        x, m = x[rows].contiguous(), m[rows].contiguous()
        reps = (128 + x.shape[0] - 1) // x.shape[0]  # at least 128 rows: the one-CTA-per-row kernel
        x, m = x.repeat(reps, 1), m.repeat(reps, 1)
    return lambda i: tsa.sample(x, 0.8, 0, 0.95, 0.05, seed=i, offset=i, bitmask=m)


def _profile_topk(tsa, dev, k):
    x, _ = workloads.topk_large(k)
    x = x.to(dev)
    return lambda i: tsa.topk(x, k)


def _profile_mask(tsa, dev):
    c = workloads.decode_batch("greedy", mask_density=MASK_DENSITY, B=B, V=V)
    x, m = c.logits.to(dev), c.bitmask.to(dev)
    return lambda i: tsa.apply_token_bitmask(x, m)


def _profile_split(tsa, dev):
    c = workloads.decode_batch("combined", mask_density=MASK_DENSITY, B=B, V=V, rows=32)
    x, m = c.logits.to(dev), c.bitmask.to(dev)
    return lambda i: tsa.sample(x, c.temperature, c.top_k, c.top_p, c.min_p, seed=i, offset=i, bitmask=m)


def _profile_lm_head(tsa, dev):
    w = torch.empty(248320, 5120, dtype=torch.bfloat16, device=dev)
    w.normal_(0.0, 0.02, generator=torch.Generator(device=dev).manual_seed(0))
    h = torch.randn(1, 5120, device=dev, generator=torch.Generator(device=dev).manual_seed(1)).to(torch.bfloat16)
    return lambda i: tsa.lm_head_topk(h, w, 50)


def _profile_decode_variant(tsa, dev, kind):
    c = workloads.decode_batch("combined", mask_density=MASK_DENSITY, B=B, V=V)
    x, m = c.logits.to(dev), c.bitmask.to(dev)
    if kind == "icdf":
        u = torch.rand(B, device=dev, generator=torch.Generator(device=dev).manual_seed(2))
        return lambda i: tsa.sample_icdf(x, u, c.temperature, c.top_k, c.top_p, c.min_p, bitmask=m)
    if kind == "pack":
        allowed = torch.from_numpy(np.unpackbits(c.bitmask.numpy().view(np.uint8), axis=1,
                                                 bitorder="little")[:, :V].astype(bool)).to(dev)
        return lambda i: tsa.bitmask_from_allowed(allowed)
    return lambda i: tsa.sample(x, c.temperature, c.top_k, c.top_p, c.min_p, seed=i, offset=i, bitmask=m,
                                sequential=True)


# --profile --op NAME: one per-op workload, run eagerly for a profiler
PROFILE_OPS = {
    "sample": None,  # the decode batch of --mode (and --no-mask)
    "hetero": _profile_hetero,  # heterogeneous bf16 B=1,024 V=32,000
    "peaked": _profile_peaked,  # peaked bf16 B=512 V=256,000
    "peaked_flat": lambda tsa, dev: _profile_peaked(tsa, dev, True),  # its flat rows, repeated to >= 128
    "topk50": lambda tsa, dev: _profile_topk(tsa, dev, 50),  # exact top-k, B=8 V=248,320
    "topk2048": lambda tsa, dev: _profile_topk(tsa, dev, 2048),
    "mask": _profile_mask,  # in-place bitmask apply on the decode batch
    "split": _profile_split,  # 32 decode rows: the split-row kernels and their merge
    "lm_head": _profile_lm_head,  # dense lm-head fused top-k, V=248,320 H=5,120 M=1 k=50
    "icdf": lambda tsa, dev: _profile_decode_variant(tsa, dev, "icdf"),  # inverse-CDF draw, decode batch
    "sequential": lambda tsa, dev: _profile_decode_variant(tsa, dev, "sequential"),  # sequential top-p
    "pack": lambda tsa, dev: _profile_decode_variant(tsa, dev, "pack"),  # bitmask_from_allowed, decode allow-set
}


def max_over_ranks(x, dev):
    """The largest value of x over all ranks, returned on every rank (x itself
    without a process group).  NCCL reduces on the GPU, gloo on the host."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    on = dev if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=on)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="skip per_op and cpu_baseline")
    ap.add_argument("--profile", action="store_true",
                    help="eager warm-up + steps only (for a profiler); prints the step time")
    ap.add_argument("--mode", default="combined", choices=list(workloads.DECODE_MODES),
                    help="with --profile: the decode mode to run")
    ap.add_argument("--no-mask", action="store_true", help="with --profile: run without the mask")
    ap.add_argument("--op", default="sample", choices=list(PROFILE_OPS),
                    help="with --profile: the workload to run (sample: the decode batch in --mode)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = world > 1
    if dist:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl" if args.impl == "ours" else "gloo")

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line))
        if dist:
            torch.distributed.destroy_process_group()
        return

    import __graft_entry__

    if rank == 0 or not dist:
        __graft_entry__.build()
    if dist:
        torch.distributed.barrier()
    import top_sampling_apply_gb300 as tsa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    hbm_peak, peak_kind = peaks()

    case = make_inputs(seed=rank)
    xs = [case.logits.to(dev) for _ in range(N_BUFFERS)]
    masks = [case.bitmask.to(dev) for _ in range(N_BUFFERS)]
    T, K, P, MP = case.temperature, case.top_k, case.top_p, case.min_p
    if args.profile:
        T, K, P, MP = workloads.DECODE_MODES[args.mode]
        if args.no_mask:
            masks = [None] * N_BUFFERS
    out = torch.empty(B, dtype=torch.int64, device=dev)

    def step(i):
        j = i % N_BUFFERS
        tsa.sample(xs[j], T, K, P, MP, seed=i, offset=i, bitmask=masks[j], out=out)

    if args.profile and args.op != "sample":
        del xs, masks
        step = PROFILE_OPS[args.op](tsa, dev)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if args.profile:
        t0 = time.perf_counter()
        for i in range(args.steps):
            step(args.warmup + i)
        torch.cuda.synchronize()
        print(json.dumps({"profile_steps": args.steps,
                          "ms_per_step_wall": (time.perf_counter() - t0) / args.steps * 1e3}))
        return
    timed = GraphSteps(lambda i: step(args.warmup + i), args.steps)
    preload = GraphSteps(step, 64)
    clocks = ClockSampler(local)
    clocks.start()
    t_end = time.perf_counter() + 0.5  # sustained load before the timed region
    while time.perf_counter() < t_end:
        preload.replay()
        torch.cuda.synchronize()
    if dist:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    timed.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        torch.distributed.barrier()
    ms = e0.elapsed_time(e1) / args.steps
    time.sleep(0.15)
    clk = clocks.stop()
    ms = max_over_ranks(ms, dev)
    assert tsa.device_status() == 0

    nbytes = algorithmic_bytes(B, V, 4, mask=True)
    achieved = nbytes / ms / 1e6  # GB/s
    rows_per_s = world * B / ms * 1e3

    # end to end through the public call: pinned host inputs -> device ->
    # sample -> tokens back to the host, every step
    h_logits = case.logits.pin_memory()
    h_mask = case.bitmask.pin_memory()
    h_tok = torch.empty(B, dtype=torch.int64).pin_memory()
    d_x = torch.empty_like(xs[0])
    d_m = torch.empty_like(masks[0])

    def e2e_step(i):
        d_x.copy_(h_logits, non_blocking=True)
        d_m.copy_(h_mask, non_blocking=True)
        tsa.sample(d_x, T, K, P, MP, seed=i, offset=i, bitmask=d_m, out=out)
        h_tok.copy_(out, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_iters = max(10, args.steps // 4)
    if dist:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(e2e_iters):
        e2e_step(i)
        torch.cuda.current_stream(dev).synchronize()
    e2e_ms = (time.perf_counter() - t0) / e2e_iters * 1e3
    e2e_ms = max_over_ranks(e2e_ms, dev)

    per_op = None
    cpu_base = None
    if rank == 0 and not args.no_extras:
        per_op = per_op_breakdown(tsa, dev, stream, hbm_peak)
        if world == 1:
            cpu_base = cpu_baseline_sample()
    if rank == 0:
        line = {
            "metric": METRIC, "value": rows_per_s, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": headline_config(world),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": sample_traffic(),
                         "kernel": "sample_row_kernel<f32> (one CTA per row)",
                         "peak_kind": peak_kind,
                         "bytes_per_launch": nbytes},
            "cpu_baseline": cpu_base,
            "e2e": {"value": world * B / e2e_ms * 1e3, "unit": "rows/s",
                    "h2d_bytes_per_step": h_logits.numel() * 4 + h_mask.numel() * 4,
                    "d2h_bytes_per_step": B * 8, "ms_per_step": e2e_ms},
            "gpu_launches": SAMPLE_LAUNCHES * args.steps,
            "clocks": clk,
            "per_op": per_op,
        }
        print(json.dumps(line))
    if dist:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
