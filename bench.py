"""Benchmark of the block-sparse attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic inputs:
  * block-sparse prefill (bsattn_prefill, mask compaction fused in the kernel) on the
    workload the headline metric is quoted on: B=2, H=8, S=4096, d=128 bf16, top-16 block
    mask with tril and dense last rows, causal (seed 0: 9850 active 64x64 block pairs);
  * GQA varlen sparse decode (bsattn_decode_varlen) on 8 sequences, 32 q-heads / 8 kv-heads,
    d=128 bf16, cache_seqlens uniform in [8192, 65536], 64 selected blocks per (b, kv-head).

value = effective TFLOP/s of the prefill over active block pairs (4*64*64*d FLOPs each),
summed over ranks; the decode's HBM GB/s over the K/V bytes of the valid tokens it reads is
reported beside it.  L2 is flushed before each of the two timed kernels, outside the events:
a 256 MiB write evicts everything, then a 256 MiB read replaces the flush's dirty lines with
clean ones, so that no kernel pays for writing back the flush buffer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synthetic  # noqa: E402

PREFILL = synthetic.PREFILL_CONFIGS["C2"]
DECODE = synthetic.DECODE_CONFIGS["C5"]
METRIC = "block-sparse attn effective TFLOP/s (active blocks) & decode HBM GB/s, % of roofline"
WORKLOAD = ("prefill B=2 H=8 S=4096 d=128 bf16 top-16+tril+dense-last causal (seed 0) + "
            "GQA varlen sparse decode B=8 Hq=32 Hkv=8 d=128 bf16 seqlens U[8192,65536] "
            "64 blocks/(b,kv-head)")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


def traffic_record(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source: the hash covers the kernel's .cu file and the inline helpers it
    includes (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    names = rec["source"] if isinstance(rec["source"], list) else [rec["source"]]
    h = hashlib.sha256()
    try:
        for name in names:
            with open(os.path.join(ROOT, "block_sparse_attention_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    digest = h.hexdigest()[:16]
    return rec["bytes_per_launch"] if digest == rec.get("source_sha256_16") else None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms; only the samples whose
    timestamps fall inside the timed window are summarised."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons, power = [], [], set(), []
        for arrived, ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = arrived
            if not (t0 <= ts <= t1):
                continue
            try:
                sm.append(float(parts[2]))
                smax.append(float(parts[3]))
                power.append(float(parts[4]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_median": statistics.median(power) if power else None}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist.get_rank(), world, int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(units_per_rank_per_step: float, steps: int, world: int, max_seconds: float):
    """Whole-job throughput: units processed by all ranks / the slowest rank's time."""
    return units_per_rank_per_step * steps * world / max_seconds


# ---------------------------------------------------------------------------- workloads

def build_inputs(mask_builder):
    """Seeded inputs; the block mask comes from `mask_builder` (the library's host builder
    on the GPU arm, the oracle's own builder on the CPU arms)."""
    q, k, v, scores = synthetic.prefill_inputs(PREFILL)
    mask = torch.as_tensor(mask_builder(scores, int(PREFILL.param), PREFILL.dense_last,
                                        PREFILL.tril))
    dq, dk, dv, sl, idx = synthetic.decode_inputs(DECODE)
    return (q, k, v, mask), (dq, dk, dv, sl, idx)


def prefill_flops(mask, causal=True) -> float:
    nq = mask.shape[2]
    keep = torch.ones(nq, mask.shape[3], dtype=torch.bool)
    if causal:
        keep = keep.tril()
    pairs = int(((mask != 0) & keep).sum())
    return pairs * 4.0 * 64 * 64 * PREFILL.d, pairs


def decode_bytes(sl, idx, d=DECODE.d, elt=2) -> float:
    total = 0
    for b in range(idx.shape[0]):
        n = int(sl[b])
        for g in range(idx.shape[1]):
            for t in idx[b, g].tolist():
                if t >= 0 and t * 64 < n:
                    total += min(64, n - t * 64)
    return total * d * elt * 2.0            # K and V


# ---------------------------------------------------------------------------- GPU arm

def run_gpu(args):
    import block_sparse_attention_gb300 as bsa
    rank, world, local = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    bsa.load()
    (q, k, v, mask), (dq, dk, dv, sl, idx) = build_inputs(bsa.bsattn_mask_from_topk)
    flops, pairs = prefill_flops(mask)
    dbytes = decode_bytes(sl, idx)

    gq, gk, gv, gm = (t.to(dev) for t in (q, k, v, mask))
    gdq, gdk, gdv, gsl, gidx = (t.to(dev) for t in (dq, dk, dv, sl, idx))
    out = torch.empty_like(gq)
    dout = torch.empty_like(gdq)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    # a second buffer, read (not written) after each flush, so that L2 holds clean lines when
    # a timed kernel starts: the flush's own dirty lines are written back outside the events
    clean = torch.ones(32 << 20, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    ns = bsa.bsattn_decode_default_splits(DECODE.B, DECODE.Hkv, DECODE.max_sel, DECODE.d)

    def cold_l2(i):
        flush.fill_(i & 0xFF)
        clean.max()

    def step(ev, i):
        ev[0].record(stream)
        bsa.bsattn_prefill(gq, gk, gv, gm, True, out=out)
        ev[1].record(stream)
        cold_l2(i + 1)
        ev[2].record(stream)
        bsa.bsattn_decode_varlen(gdq, gdk, gdv, gsl, gidx, ns, out=dout)
        ev[3].record(stream)

    clocks = ClockSampler(local)
    clocks.start()
    for i in range(args.warmup):
        cold_l2(i)
        step([torch.cuda.Event(enable_timing=True) for _ in range(4)], i)
    torch.cuda.synchronize()
    time.sleep(0.3)            # let the sampler start before the timed window

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    w0 = time.time()
    for i in range(args.steps):
        cold_l2(i)
        step(evs[i], i)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    clk = clocks.stop(w0, time.time())
    pre_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[2].elapsed_time(e[3]) for e in evs]
    step_ms = [a + b for a, b in zip(pre_ms, dec_ms)]
    dev_s = max_over_ranks(sum(step_ms) / 1e3, world, dev)
    pre_s = max_over_ranks(sum(pre_ms) / 1e3, world, dev)
    dec_s = max_over_ranks(sum(dec_ms) / 1e3, world, dev)
    status = bsa.bsattn_get_device_status(bsa.workspace(dev, "prefill", 256)) | \
        bsa.bsattn_get_device_status(bsa.workspace(dev, "decode", 256))

    # ---- end to end through the public API with host buffers (pinned), copies timed
    hp = [t.pin_memory() for t in (q, k, v, mask)]
    hdq, hsl, hidx = (t.pin_memory() for t in (dq, sl, idx))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hdout = torch.empty(dout.shape, dtype=dout.dtype).pin_memory()
    dq_dev, sl_dev, idx_dev = torch.empty_like(gdq), torch.empty_like(gsl), torch.empty_like(gidx)
    e2e_steps = max(3, min(args.steps, 50))
    h2d_pre = sum(t.numel() * t.element_size() for t in hp)
    h2d_dec = sum(t.numel() * t.element_size() for t in (hdq, hsl, hidx))
    d2h_pre, d2h_dec = hout.numel() * 2, hdout.numel() * 2
    e_pre, e_dec = [], []
    for i in range(e2e_steps + 2):
        cold_l2(i)
        a, bq, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(stream)
        tq, tk, tv, tm = (t.to(dev, non_blocking=True) for t in hp)
        bsa.bsattn_prefill(tq, tk, tv, tm, True, out=out)
        hout.copy_(out, non_blocking=True)
        bq.record(stream)
        dq_dev.copy_(hdq, non_blocking=True)
        sl_dev.copy_(hsl, non_blocking=True)
        idx_dev.copy_(hidx, non_blocking=True)
        bsa.bsattn_decode_varlen(dq_dev, gdk, gdv, sl_dev, idx_dev, ns, out=dout)
        hdout.copy_(dout, non_blocking=True)
        c.record(stream)
        torch.cuda.synchronize()
        if i >= 2:
            e_pre.append(a.elapsed_time(bq))
            e_dec.append(bq.elapsed_time(c))
    e_pre_s = max_over_ranks(sum(e_pre) / 1e3, world, dev)
    e_dec_s = max_over_ranks(sum(e_dec) / 1e3, world, dev)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    pk, kind = peaks()
    tflops = aggregate(flops, args.steps, world, pre_s) / 1e12
    per_launch_pre = pre_s / args.steps
    per_launch_dec = dec_s / args.steps
    ach_pre = flops / per_launch_pre / 1e12
    ach_dec = dbytes / per_launch_dec / 1e9
    line = {
        "metric": METRIC,
        "value": round(tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dev_s / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V, uniform block scores; see synthetic/)",
        "config": {"workload": WORKLOAD, "active_block_pairs": pairs,
                   "prefill_gflop_per_step": round(flops / 1e9, 3),
                   "decode_bytes_per_step": int(dbytes), "decode_num_splits": ns,
                   "l2": "flushed before each timed kernel (256 MiB write, then a 256 MiB read so the lines are clean; outside the events)",
                   "inputs": "resident in HBM when the timed region starts",
                   "parallelism": f"replicas x{world} (no collective)"},
        "roofline": {"bound": "tensor", "achieved": round(ach_pre, 2),
                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(ach_pre / pk["bf16_tflops"], 4),
                     "traffic": traffic_record("prefill"),
                     "kernel": "prefill_kernel<128,bf16>", "peak_source": f"{kind} bf16 burst"},
        "decode": {"value": round(aggregate(dbytes, args.steps, world, dec_s) / 1e9, 1),
                   "unit": "GB/s", "ms_per_launch": round(per_launch_dec * 1e3, 4),
                   "roofline": {"bound": "hbm", "achieved": round(ach_dec, 1),
                                "peak": pk["hbm_gbs"], "unit": "GB/s",
                                "frac": round(ach_dec / pk["hbm_gbs"], 4),
                                "traffic": traffic_record("decode"),
                                "kernel": "decode_kernel<128,bf16>",
                                "peak_source": f"{kind} copy bandwidth"}},
        "prefill_ms_per_launch": round(per_launch_pre * 1e3, 4),
        "e2e": {"value": round(aggregate(flops, e2e_steps, world, e_pre_s) / 1e12, 3),
                "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d_pre),
                "d2h_bytes_per_step": int(d2h_pre),
                "decode": {"value": round(aggregate(dbytes, e2e_steps, world, e_dec_s) / 1e9, 1),
                           "unit": "GB/s", "h2d_bytes_per_step": int(h2d_dec),
                           "d2h_bytes_per_step": int(d2h_dec),
                           "note": "KV cache device-resident across decode steps"}},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
        "device_status": status,
        "wall_s": round(wall, 3),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(q, k, v, target_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- CPU arms

def oracle_rows_sample(mask, rows_per_head, seed):
    """Query rows (b, h, [rows]) to run through the oracle: whole 64-row query blocks,
    drawn across all heads so the sample follows the workload's length mix."""
    import numpy as np
    rng = np.random.default_rng(seed)
    B, H, nq, _ = mask.shape
    picks = []
    for b in range(B):
        for h in range(H):
            blocks = rng.choice(nq, size=max(1, rows_per_head // 64), replace=False)
            rows = [r for qb in blocks for r in range(int(qb) * 64, int(qb) * 64 + 64)]
            picks.append((b, h, rows))
    return picks


def oracle_sample_flops(mask, picks, causal=True) -> float:
    """Effective FLOPs of the sampled rows in the metric's unit (active pairs x 4*64*d / 64
    per row)."""
    total = 0.0
    for b, h, rows in picks:
        for qb in sorted({r // 64 for r in rows}):
            n_rows = sum(1 for r in rows if r // 64 == qb)
            row = mask[b, h, qb]
            pairs = int((row[: qb + 1] != 0).sum()) if causal else int((row != 0).sum())
            total += pairs * 4.0 * 64 * PREFILL.d * n_rows
    return total


def time_oracle_sample(q, k, v, mask, picks):
    import oracle
    t0 = time.perf_counter()
    for b, h, rows in picks:
        oracle.prefill_rows(q, k, v, mask, True, b, h, rows)
    return time.perf_counter() - t0


def cpu_baseline(q, k, v, target_s=10.0, seed=0):
    """The oracle, as it stands, on whole 64-row query blocks drawn at random (seeded) from
    every head of the workload, until `target_s` seconds of CPU work are done."""
    import numpy as np
    import oracle
    oracle.build()
    _, _, _, scores = synthetic.prefill_inputs(PREFILL)
    mask = torch.from_numpy(oracle.mask_from_topk(scores, int(PREFILL.param), PREFILL.dense_last,
                                                  PREFILL.tril))
    rng = np.random.default_rng(seed)
    B, H, nq, _ = mask.shape
    t_total, flops, blocks = 0.0, 0.0, 0
    while t_total < target_s:
        b, h, qb = int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(nq))
        picks = [(b, h, list(range(qb * 64, min(qb * 64 + 64, PREFILL.S))))]
        t_total += time_oracle_sample(q, k, v, mask, picks)
        flops += oracle_sample_flops(mask, picks)
        blocks += 1
    return {"value": round(flops / t_total / 1e12, 6), "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{blocks} random 64-row query blocks ({blocks * 64} rows) of the prefill "
                      f"workload, fp64, {t_total:.1f} s of oracle time"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    (q, k, v, mask), _ = build_inputs(oracle.mask_from_topk)
    # each step: one query block per head, drawn afresh (a bounded sample of the workload)
    for i in range(args.warmup):
        time_oracle_sample(q, k, v, mask, oracle_rows_sample(mask, 64, 1000 + i))
    tot_t, tot_f, rows = 0.0, 0.0, 0
    for i in range(args.steps):
        picks = oracle_rows_sample(mask, 64, i)
        tot_t += time_oracle_sample(q, k, v, mask, picks)
        tot_f += oracle_sample_flops(mask, picks)
        rows += sum(len(r) for _, _, r in picks)
    val = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": "TFLOP/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s",
                             "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"per step one 64-row query block of each of the 16 "
                                       f"prefill heads ({rows} rows over {args.steps} steps)"},
            "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["bsattn", "reference"], default="bsattn")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
