"""Benchmark of the block-sparse attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic inputs:
  * block-sparse prefill (bsattn_prefill, mask compaction fused in the kernel) on the largest
    prefill workload: B=1, H=32, S=16384, d=128 bf16, threshold-0.9 block mask (~10 %
    density) with tril and dense last rows, causal (seed 0: 120402 active 64x64 block pairs);
  * GQA varlen sparse decode (bsattn_decode_varlen) on 8 sequences, 32 q-heads / 8 kv-heads,
    d=128 bf16, cache_seqlens uniform in [8192, 65536], 64 selected blocks per (b, kv-head).

value = effective TFLOP/s of the prefill over active block pairs (4*64*64*d FLOPs each),
summed over ranks; the decode's HBM GB/s over the K/V bytes of the valid tokens it reads is
reported beside it.  L2 is flushed before each of the two timed kernels, outside the events:
a 256 MiB write evicts everything, then a 256 MiB read replaces the flush's dirty lines with
clean ones, so that no kernel pays for writing back the flush buffer.

After the timed steps, every workload of the set (the four prefill shapes and the decode) is
timed on its own the same way, and (unless --no-parity) compared on every output element
with the fp64 oracle: the `configs` object of the JSON line.  SM clocks and throttle reasons
are sampled in-process through NVML (about every millisecond) during each phase.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--no-parity]

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synthetic  # noqa: E402

HEADLINE = "C3"
PREFILL = synthetic.PREFILL_CONFIGS[HEADLINE]
DECODE = synthetic.DECODE_CONFIGS["C5"]
METRIC = "block-sparse attn effective TFLOP/s (active blocks) & decode HBM GB/s, % of roofline"
WORKLOAD = ("prefill B=1 H=32 S=16384 d=128 bf16 threshold-0.9 (~10% blocks)+tril+dense-last "
            "causal (seed 0) + GQA varlen sparse decode B=8 Hq=32 Hkv=8 d=128 bf16 seqlens "
            "U[8192,65536] 64 blocks/(b,kv-head)")
DESCRIBE = {
    "C1": "prefill B=1 H=2 S=512 d=64 fp16 top-3+tril causal",
    "C2": "prefill B=2 H=8 S=4096 d=128 bf16 top-16+tril+dense-last causal",
    "C3": "prefill B=1 H=32 S=16384 d=128 bf16 threshold-0.9+tril+dense-last causal",
    "C4": "prefill B=4 H=16 S=8192 d=64 fp16 threshold-0.75 non-causal",
    "C5": "GQA varlen sparse decode B=8 Hq=32 Hkv=8 d=128 bf16, 64 blocks/(b,kv-head)",
    "C3/128": "prefill B=1 H=32 S=16384 d=128 bf16 threshold-0.9+tril+dense-last causal on 128-token "
              "blocks (the 128-row kernel)",
}
TOL = {torch.float16: 1e-2, torch.bfloat16: 2e-2}
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


def source_digest(paths) -> str:
    """Hash of the code in the given source files, comments, indentation and blank lines left
    out: a record taken on a kernel stays valid through comment edits, not through code edits."""
    h = hashlib.sha256()
    for path in paths:
        with open(path) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for line in src.splitlines():
            line = line.strip()
            if line:
                h.update(line.encode() + b"\n")
    return h.hexdigest()[:16]


def traffic_record(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    kernel code and on this workload: the hash covers the code of the kernel's .cu file and of
    the inline helpers it includes (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("config") != workload:
        return None
    names = rec["source"] if isinstance(rec["source"], list) else [rec["source"]]
    try:
        digest = source_digest([os.path.join(ROOT, "block_sparse_attention_gb300", "csrc", name)
                                for name in names])
    except OSError:
        return None
    return rec["bytes_per_launch"] if digest == rec.get("source_sha256_16") else None


class ClockSampler:
    """SM clock, power and clock-event (throttle) reasons read in-process through NVML (a
    read-only query) about every millisecond by a background thread; each named phase of the
    run keeps the samples taken while it ran."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        self.samples = []          # (perf_counter, sm_mhz, reasons, power_w or None)
        self.phases = {}
        self.error = None
        self.max_mhz = None
        self._stop = threading.Event()
        self.thread = None
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            self.handle = self._handle(cuda_index)
            try:
                self.reasons_fn = self.nv.nvmlDeviceGetCurrentClocksEventReasons
            except AttributeError:                      # older drivers: the previous name
                self.reasons_fn = self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint(0)
            if self.nv.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
        except OSError as e:
            self.error = str(e)

    def _handle(self, cuda_index):
        want = str(torch.cuda.get_device_properties(cuda_index).uuid).lower().replace("gpu-", "")
        n = ctypes.c_uint(0)
        if self.nv.nvmlDeviceGetCount_v2(ctypes.byref(n)) != 0:
            raise OSError("nvmlDeviceGetCount failed")
        for i in range(n.value):
            h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByIndex_v2(i, ctypes.byref(h)) != 0:
                continue
            buf = ctypes.create_string_buffer(96)
            if self.nv.nvmlDeviceGetUUID(h, buf, 96) != 0:
                continue
            if buf.value.decode().lower().replace("gpu-", "") == want:
                return h
        raise OSError("no NVML device with this GPU's UUID")

    def _loop(self):
        clk, rs, pw = ctypes.c_uint(0), ctypes.c_ulonglong(0), ctypes.c_uint(0)
        n = 0
        while not self._stop.is_set():
            t = time.perf_counter()
            if self.nv.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0 and \
                    self.reasons_fn(self.handle, ctypes.byref(rs)) == 0:
                power = None
                if n % 20 == 0 and self.nv.nvmlDeviceGetPowerUsage(self.handle, ctypes.byref(pw)) == 0:
                    power = pw.value / 1000.0
                self.samples.append((t, float(clk.value), int(rs.value), power))
            n += 1
            time.sleep(0.0005)

    def start(self):
        if self.error is None:
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()

    def phase(self, name, t0, t1):
        self.phases[name] = (t0, t1)

    def stop(self):
        self._stop.set()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, names):
        if self.error is not None:
            return {name: {"sm_mhz": None, "reasons": [f"nvml: {self.error}"], "samples": 0}
                    for name in names}
        out = {}
        for name in names:
            t0, t1 = self.phases.get(name, (0.0, -1.0))
            sel = [s for s in self.samples if t0 <= s[0] <= t1]
            reasons = set()
            for s in sel:
                for bit, label in self.REASONS.items():
                    if s[2] & bit:
                        reasons.add(label)
            power = [s[3] for s in sel if s[3] is not None]
            out[name] = {"sm_mhz": statistics.median([s[1] for s in sel]) if sel else None,
                         "sm_min_mhz": min(s[1] for s in sel) if sel else None,
                         "reasons": sorted(reasons), "samples": len(sel),
                         "power_w_median": statistics.median(power) if power else None}
        return out


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

def prefill_case(cfg, mask_builder):
    """Seeded inputs of a prefill configuration; the block mask comes from `mask_builder`
    (a function (scores, cfg) -> mask)."""
    q, k, v, scores = synthetic.prefill_inputs(cfg)
    return q, k, v, torch.as_tensor(mask_builder(scores, cfg))


def library_mask(scores, cfg):
    import block_sparse_attention_gb300 as bsa
    if cfg.rule == "topk":
        return bsa.bsattn_mask_from_topk(scores, int(cfg.param), cfg.dense_last, cfg.tril)
    return bsa.bsattn_mask_from_threshold(scores, cfg.param, cfg.dense_last, cfg.tril)


def oracle_mask(scores, cfg):
    import oracle
    if cfg.rule == "topk":
        return oracle.mask_from_topk(scores, int(cfg.param), cfg.dense_last, cfg.tril)
    return oracle.mask_from_threshold(scores, cfg.param, cfg.dense_last, cfg.tril)


def prefill_flops(mask, cfg, block=64):
    """Effective FLOPs: 4*64*64*d per visited 64x64 tile pair (a 128-token entry stands for its
    four tiles, of which the causal rule keeps those on or below the diagonal)."""
    m = torch.as_tensor(mask) != 0
    if block == 128:
        m = m.repeat_interleave(2, dim=2).repeat_interleave(2, dim=3)
        n = -(-cfg.S // 64)
        m = m[:, :, :n, :n]
    nq = m.shape[2]
    keep = torch.ones(nq, m.shape[3], dtype=torch.bool)
    if cfg.causal:
        keep = keep.tril()
    pairs = int((m & keep).sum())
    return pairs * 4.0 * 64 * 64 * cfg.d, pairs


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

class L2Flush:
    """Leaves L2 holding clean lines of an unrelated buffer: a 256 MiB write evicts
    everything, then a 256 MiB read replaces the write's dirty lines."""

    def __init__(self, dev):
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.clean = torch.ones(32 << 20, dtype=torch.int64, device=dev)

    def __call__(self, i):
        self.flush.fill_(i & 0xFF)
        self.clean.max()


def pipelined(n, host_in, dev_in, compute, dev_out, host_out, dev):
    """Runs n steps, each copying `host_in` (pinned) into device buffer set i % 2, computing into
    dev_out[i % 2] and copying that back into host_out[i % 2], on three streams so that the
    copies of one step overlap the computation of its neighbours.  Returns the elapsed ms from
    the first input copy to the last output copy (CUDA events)."""
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(s_in)
    for i in range(n):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_cmp[b])         # step i-2 no longer reads buffer set b
            for d, h in zip(dev_in[b], host_in):
                d.copy_(h, non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev_in[b])
            if i >= 2:
                s_cmp.wait_event(ev_out[b])        # step i-2's output has left dev_out[b]
            compute(b)
            ev_cmp[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[b])
            host_out[b].copy_(dev_out[b], non_blocking=True)
            ev_out[b].record(s_out)
    s_out.wait_event(ev_in[(n - 1) % 2])
    end.record(s_out)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def time_calls(fn, stream, flush, reps, warm=3):
    """Median CUDA-event time (ms) of fn(), each call after an L2 flush outside the events."""
    for i in range(warm):
        flush(i)
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for i, (a, b) in enumerate(evs):
        flush(i + 1)
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def run_gpu(args):
    import block_sparse_attention_gb300 as bsa
    rank, world, local = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    bsa.load()
    q, k, v, mask = prefill_case(PREFILL, library_mask)
    flops, pairs = prefill_flops(mask, PREFILL)
    dq, dk, dv, sl, idx = synthetic.decode_inputs(DECODE)
    dbytes = decode_bytes(sl, idx)

    gq, gk, gv, gm = (t.to(dev) for t in (q, k, v, mask))
    gdq, gdk, gdv, gsl, gidx = (t.to(dev) for t in (dq, dk, dv, sl, idx))
    out = torch.empty_like(gq)
    dout = torch.empty_like(gdq)
    cold_l2 = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    ns = bsa.bsattn_decode_default_splits(DECODE.B, DECODE.Hkv, DECODE.max_sel, DECODE.d)
    ns_page = bsa.bsattn_num_splits_heuristic(
        DECODE.B * DECODE.Hkv, torch.cuda.get_device_properties(dev).multi_processor_count,
        DECODE.max_sel, 1, DECODE.max_sel * 64 * 2 * DECODE.d * 2, True, 128)

    def step(ev, i):
        ev[0].record(stream)
        bsa.bsattn_prefill(gq, gk, gv, gm, PREFILL.causal, out=out)
        ev[1].record(stream)
        cold_l2(i + 1)
        ev[2].record(stream)
        bsa.bsattn_decode_varlen(gdq, gdk, gdv, gsl, gidx, ns, out=dout)
        ev[3].record(stream)

    clocks = ClockSampler(local)
    clocks.start()
    t_w0 = time.perf_counter()
    for i in range(args.warmup):
        cold_l2(i)
        step([torch.cuda.Event(enable_timing=True) for _ in range(4)], i)
    torch.cuda.synchronize()
    clocks.phase("warmup", t_w0, time.perf_counter())

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        cold_l2(i)
        step(evs[i], i)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(world)
    clocks.phase("timed", t0, t1)
    wall = t1 - t0
    pre_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[2].elapsed_time(e[3]) for e in evs]
    step_ms = [a + b for a, b in zip(pre_ms, dec_ms)]
    dev_s = max_over_ranks(sum(step_ms) / 1e3, world, dev)
    pre_s = max_over_ranks(sum(pre_ms) / 1e3, world, dev)
    dec_s = max_over_ranks(sum(dec_ms) / 1e3, world, dev)
    status = bsa.bsattn_get_device_status(bsa.workspace(dev, "prefill", 256)) | \
        bsa.bsattn_get_device_status(bsa.workspace(dev, "decode", 256))

    # ---- end to end through the public API with host buffers (pinned), copies timed: every step
    # copies its inputs in and its output back; steps are pipelined over three streams (inputs of
    # step i+1 in, step i computing, output of step i-1 out), with two device buffer sets
    hp = [t.pin_memory() for t in (q, k, v, mask)]
    hdec = [t.pin_memory() for t in (dq, sl, idx)]
    houts = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    hdouts = [torch.empty(dout.shape, dtype=dout.dtype).pin_memory() for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 50))
    h2d_pre = sum(t.numel() * t.element_size() for t in hp)
    h2d_dec = sum(t.numel() * t.element_size() for t in hdec)
    d2h_pre, d2h_dec = out.numel() * 2, dout.numel() * 2
    pin = [[torch.empty_like(t, device=dev) for t in hp] for _ in range(2)]
    pout = [out, torch.empty_like(out)]
    din = [[torch.empty_like(t, device=dev) for t in hdec] for _ in range(2)]
    dpout = [dout, torch.empty_like(dout)]

    def prefill_step(b):
        tq, tk, tv, tm = pin[b]
        bsa.bsattn_prefill(tq, tk, tv, tm, PREFILL.causal, out=pout[b])

    def decode_step(b):
        tq, tsl, tidx = din[b]
        bsa.bsattn_decode_varlen(tq, gdk, gdv, tsl, tidx, ns, out=dpout[b])

    t_e0 = time.perf_counter()
    pipelined(3, hp, pin, prefill_step, pout, houts, dev)             # warm-up
    e_pre_ms = pipelined(e2e_steps, hp, pin, prefill_step, pout, houts, dev)
    # the decode's copies are a few KB: its steps run one after another on one stream (copies in,
    # kernel, copy back), all enqueued ahead so that no host gap falls inside a step's events
    dec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(e2e_steps + 2)]
    torch.cuda.synchronize()
    for i, (a, c) in enumerate(dec_ev):
        a.record(stream)
        for d, h in zip(din[0], hdec):
            d.copy_(h, non_blocking=True)
        decode_step(0)
        hdouts[i % 2].copy_(dpout[0], non_blocking=True)
        c.record(stream)
    torch.cuda.synchronize()
    e_dec_ms = sum(a.elapsed_time(c) for a, c in dec_ev[2:])
    clocks.phase("e2e", t_e0, time.perf_counter())
    e_pre_s = max_over_ranks(e_pre_ms / 1e3, world, dev)
    e_dec_s = max_over_ranks(e_dec_ms / 1e3, world, dev)
    del pin, din, hp

    # ---- every workload of the set on its own (rank 0), plus a copy as long as the decode's
    per_cfg, outputs = {}, {}
    pk, kind = peaks()
    if rank == 0:
        t_c0 = time.perf_counter()
        reps = max(5, min(args.steps, 50))
        for name in ("C1", "C2", "C3", "C4"):
            cfg = synthetic.PREFILL_CONFIGS[name]
            if name == HEADLINE:
                cq, ck, cv, cm, cgq, cgk, cgv, cgm, cflops, cpairs = (
                    q, k, v, mask, gq, gk, gv, gm, flops, pairs)
            else:
                cq, ck, cv, cm = prefill_case(cfg, library_mask)
                cflops, cpairs = prefill_flops(cm, cfg)
                cgq, cgk, cgv, cgm = (t.to(dev) for t in (cq, ck, cv, cm))
            cout = torch.empty_like(cgq)
            ms = time_calls(lambda: bsa.bsattn_prefill(cgq, cgk, cgv, cgm, cfg.causal, out=cout),
                            stream, cold_l2, reps)
            outputs[name] = (cfg, cq, ck, cv, cm, cout.cpu())
            ach = cflops / (ms / 1e3) / 1e12
            per_cfg[name] = {"workload": DESCRIBE[name], "ms": round(ms, 4),
                             "active_block_pairs": cpairs, "gflop": round(cflops / 1e9, 3),
                             "value": round(ach, 2), "unit": "TFLOP/s",
                             "frac": round(ach / pk["bf16_tflops"], 4)}
            del cgq, cgk, cgv, cgm, cout
        # the largest workload's shape and rule on 128-token blocks: the 128-row kernel
        cfg = PREFILL
        n128 = -(-cfg.S // 128)
        scores128 = synthetic.block_scores(cfg.B, cfg.H, n128, n128, seed=0)
        m128 = torch.as_tensor(library_mask(scores128, cfg))
        cflops, cpairs = prefill_flops(m128, cfg, block=128)
        gm128 = m128.to(dev)
        cout = torch.empty_like(gq)
        ms = time_calls(lambda: bsa.bsattn_prefill(gq, gk, gv, gm128, cfg.causal, out=cout,
                                                   block_size=128), stream, cold_l2, reps)
        outputs["C3/128"] = (cfg, q, k, v, m128, cout.cpu(), scores128)
        ach = cflops / (ms / 1e3) / 1e12
        per_cfg["C3/128"] = {"workload": DESCRIBE["C3/128"], "ms": round(ms, 4),
                             "active_tile_pairs": cpairs, "gflop": round(cflops / 1e9, 3),
                             "value": round(ach, 2), "unit": "TFLOP/s",
                             "frac": round(ach / pk["bf16_tflops"], 4)}
        del gm128, cout
        ms = time_calls(lambda: bsa.bsattn_decode_varlen(gdq, gdk, gdv, gsl, gidx, ns, out=dout),
                        stream, cold_l2, reps)
        ms_page = time_calls(lambda: bsa.bsattn_decode_varlen(gdq, gdk, gdv, gsl, gidx, ns_page,
                                                               out=dout), stream, cold_l2, reps)
        outputs["C5"] = dout.cpu()
        ach = dbytes / (ms / 1e3) / 1e9
        per_cfg["C5"] = {"workload": DESCRIBE["C5"], "ms": round(ms, 4),
                         "bytes": int(dbytes), "value": round(ach, 1), "unit": "GB/s",
                         "frac": round(ach / pk["hbm_gbs"], 4), "num_splits": ns,
                         "num_splits_rule": "one wave of resident CTAs (library default)",
                         "page_heuristic": {"num_splits": ns_page,
                                            "ms": round(ms_page, 4),
                                            "value": round(dbytes / (ms_page / 1e3) / 1e9, 1)}}
        # the same byte count moved by a plain device copy and read by a plain reduction: the
        # practical ceiling of a transfer this short on this GPU
        src = torch.empty(int(dbytes) // 2, dtype=torch.uint8, device=dev).fill_(1)
        dst = torch.empty_like(src)
        rd = torch.empty(int(dbytes) // 4, dtype=torch.float32, device=dev).fill_(1.0)
        ms_copy = time_calls(lambda: dst.copy_(src), stream, cold_l2, reps)
        ms_read = time_calls(lambda: rd.sum(), stream, cold_l2, reps)
        per_cfg["C5"]["same_size_transfers"] = {
            "copy": {"bytes_moved": 2 * src.numel(), "ms": round(ms_copy, 4),
                     "GB/s": round(2 * src.numel() / (ms_copy / 1e3) / 1e9, 1)},
            "read": {"bytes_moved": 4 * rd.numel(), "ms": round(ms_read, 4),
                     "GB/s": round(4 * rd.numel() / (ms_read / 1e3) / 1e9, 1)},
            "note": "torch copy_ and sum over as many bytes as the decode reads, each after "
                    "the same L2 flush"}
        del src, dst, rd
        clocks.phase("configs", t_c0, time.perf_counter())
    clocks.stop()

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    tflops = aggregate(flops, args.steps, world, pre_s) / 1e12
    per_launch_pre = pre_s / args.steps
    per_launch_dec = dec_s / args.steps
    ach_pre = flops / per_launch_pre / 1e12
    ach_dec = dbytes / per_launch_dec / 1e9
    phases = clocks.summary(["warmup", "timed", "e2e", "configs"])
    timed = phases.get("timed", {})
    clk = {"sm_mhz": timed.get("sm_mhz"), "sm_max_mhz": clocks.max_mhz,
           "reasons": timed.get("reasons", []), "samples": timed.get("samples", 0),
           "power_w_median": timed.get("power_w_median"), "source": "NVML in-process, ~1 kHz",
           "phases": phases}
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
                   "decode_num_splits_rule": "library default: one wave of resident CTAs",
                   "l2": "flushed before each timed kernel (256 MiB write, then a 256 MiB read "
                         "so the lines are clean; outside the events); the prefill's inputs "
                         "(402 MB) are also larger than L2",
                   "inputs": "resident in HBM when the timed region starts",
                   "parallelism": f"replicas x{world} (no collective)"},
        "roofline": {"bound": "tensor", "achieved": round(ach_pre, 2),
                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(ach_pre / pk["bf16_tflops"], 4),
                     "traffic": traffic_record("prefill", HEADLINE),
                     "kernel": "prefill_kernel<128,bf16>",
                     "peak_source": f"{kind} bf16 burst (kernel timed alone)"},
        "decode": {"value": round(aggregate(dbytes, args.steps, world, dec_s) / 1e9, 1),
                   "unit": "GB/s", "ms_per_launch": round(per_launch_dec * 1e3, 4),
                   "roofline": {"bound": "hbm", "achieved": round(ach_dec, 1),
                                "peak": pk["hbm_gbs"], "unit": "GB/s",
                                "frac": round(ach_dec / pk["hbm_gbs"], 4),
                                "traffic": traffic_record("decode", "C5"),
                                "kernel": "decode_kernel<128,bf16>",
                                "peak_source": f"{kind} copy bandwidth"}},
        "prefill_ms_per_launch": round(per_launch_pre * 1e3, 4),
        "e2e": {"value": round(aggregate(flops, e2e_steps, world, e_pre_s) / 1e12, 3),
                "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d_pre),
                "d2h_bytes_per_step": int(d2h_pre), "steps": e2e_steps,
                "h2d_GBps": round(h2d_pre * e2e_steps / e_pre_s / 1e9, 1),
                "note": "every step copies Q/K/V/mask in from pinned host memory and the output "
                        "back; steps pipelined over three streams with two device buffer sets; "
                        "L2 not flushed",
                "decode": {"value": round(aggregate(dbytes, e2e_steps, world, e_dec_s) / 1e9, 1),
                           "unit": "GB/s", "h2d_bytes_per_step": int(h2d_dec),
                           "d2h_bytes_per_step": int(d2h_dec),
                           "note": "q, cache_seqlens and block_indices in, the output back, one "
                                   "step at a time; KV cache device-resident across decode "
                                   "steps"}},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
        "device_status": status,
        "wall_s": round(wall, 3),
        "configs": per_cfg,
    }
    if world == 1 and not args.no_parity:
        line["parity"] = parity(outputs, per_cfg, (dq, dk, dv, sl, idx))
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(q, k, v, target_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)


def parity(outputs, per_cfg, decode_in):
    """Every output element of every workload against the fp64 oracle (on the same rounded
    inputs and the same block masks); adds max_err / tolerance to each config."""
    import numpy as np
    import oracle
    oracle.build()
    res = {}
    for name in ("C1", "C2", "C3", "C4"):
        cfg, q, k, v, mask, got = outputs[name]
        want_mask = oracle_mask(synthetic.prefill_inputs(cfg)[3], cfg)
        same_mask = bool(np.array_equal(np.asarray(mask), want_mask))
        t0 = time.perf_counter()
        want = oracle.prefill(q, k, v, want_mask, cfg.causal)
        t_or = time.perf_counter() - t0
        err = float(np.abs(got.double().numpy() - want).max())
        per_cfg[name].update({"max_err": err, "tol": TOL[cfg.dtype],
                              "pass": err <= TOL[cfg.dtype] and same_mask,
                              "mask_bit_exact": same_mask, "oracle_s": round(t_or, 2)})
        res[name] = per_cfg[name]["pass"]
    cfg, q, k, v, mask, got, scores128 = outputs["C3/128"]
    want_mask = oracle_mask(scores128, cfg)
    same_mask = bool(np.array_equal(np.asarray(mask), want_mask))
    t0 = time.perf_counter()
    want = oracle.prefill(q, k, v, want_mask, cfg.causal, block=128)
    t_or = time.perf_counter() - t0
    err = float(np.abs(got.double().numpy() - want).max())
    per_cfg["C3/128"].update({"max_err": err, "tol": TOL[cfg.dtype],
                              "pass": err <= TOL[cfg.dtype] and same_mask,
                              "mask_bit_exact": same_mask, "oracle_s": round(t_or, 2)})
    res["C3/128"] = per_cfg["C3/128"]["pass"]
    dq, dk, dv, sl, idx = decode_in
    t0 = time.perf_counter()
    want = oracle.decode_varlen(dq, dk, dv, sl, idx)
    t_or = time.perf_counter() - t0
    err = float(np.abs(outputs["C5"].double().numpy() - want).max())
    per_cfg["C5"].update({"max_err": err, "tol": TOL[DECODE.dtype],
                          "pass": err <= TOL[DECODE.dtype], "oracle_s": round(t_or, 2)})
    res["C5"] = per_cfg["C5"]["pass"]
    return {"all_pass": all(res.values()), "elements": "every output element",
            "oracle_cores": oracle.num_threads()}


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


def oracle_sample_flops(mask, picks, causal=PREFILL.causal) -> float:
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
        oracle.prefill_rows(q, k, v, mask, PREFILL.causal, b, h, rows)
    return time.perf_counter() - t0


def cpu_baseline(q, k, v, target_s=10.0, seed=0):
    """The oracle, as it stands, on whole 64-row query blocks drawn at random (seeded) from
    every head of the workload, until `target_s` seconds of CPU work are done."""
    import numpy as np
    import oracle
    oracle.build()
    _, _, _, scores = synthetic.prefill_inputs(PREFILL)
    mask = torch.from_numpy(oracle_mask(scores, PREFILL))
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
    q, k, v, mask = prefill_case(PREFILL, oracle_mask)
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
                             "sample": f"per step one 64-row query block of each of the "
                                       f"{PREFILL.B * PREFILL.H} prefill heads ({rows} rows "
                                       f"over {args.steps} steps)"},
            "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["bsattn", "reference"], default="bsattn")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parity", action="store_true",
                    help="skip the every-element oracle comparison of the workloads")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
