#!/usr/bin/env python3
"""Benchmark of the XOR-swizzle data-movement path on GB300.

One step = the headline workload: Swizzle<5,2,5> relayout of 131072 int8
tiles of 64 x 128 (1 GiB of random bytes from seed 4; groups of 4 bytes move
intact), forward (logical -> swizzled) then inverse (swizzled -> logical),
through the C ABI.  The metric is algorithmic bytes moved (read + write,
2 x 1 GiB per launch) per second.

Timing: W untimed warm-up steps, then exactly K timed steps back to back,
bracketed by a barrier and a device synchronisation and timed by one CUDA
event pair on the launch stream.  Every buffer is 1 GiB, larger than the
126 MB L2, so no step finds the previous one's data in L2 (no flush).  SM
clocks and throttle reasons are sampled (NVML, else nvidia-smi) during the
timed steps.

The JSON line also carries:
  roofline      the relayout kernel's achieved GB/s against the measured HBM
                copy bandwidth (MEASURED_PEAKS.json), with the DRAM traffic per
                launch from the committed ncu summary when it matches the
                current kernel source;
  e2e           the same metric through the C ABI on pinned HOST buffers: the
                forward launch reads the host input and the inverse launch
                writes the host output over the host link, inside the timed
                region; a copy-engine pipeline of the same step is reported
                beside it;
  cpu_baseline  the CPU oracle on the same workload: single thread on a
                bounded sample of tiles, and the whole workload split over
                every host core (spawned processes); the 125-set sweep on a
                64 MiB sample; every other row on a bounded sample;
  rows          every other row of the path measured in the same run: the
                64 MiB bf16 relayout (L2-assisted), the small relayout, the
                uint16 sweep, the fp32 / fp16 / fp64 (and 1-byte) transposes
                with each staging, the bank profiler (skip with --no-rows).

--impl reference times the CPU oracle as the reference arm.
--gpus N without torchrun relaunches itself under torch.distributed.run.
Multi-GPU: every rank runs the same per-GPU workload (weak scaling, no
collective on the data path); value = all ranks' bytes / max time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

MiB = 1 << 20
GB = 1e9
METRIC = "relayout/transpose GB/s (read+write) & % of GB300 HBM peak; smem bank conflicts"
TILES, ROWS, COLS, ESIZE = 131072, 64, 128, 1
B, M, S = 5, 2, 5
WORKLOAD = ("Swizzle<5,2,5> relayout forward then inverse of 131072 int8 tiles of 64x128 "
            "(1 GiB, random bytes from seed 4)")
N_BYTES = TILES * ROWS * COLS * ESIZE                 # 1 GiB
LAUNCH_BYTES = 2 * N_BYTES                            # each launch reads and writes 1 GiB
STEP_BYTES = 2 * LAUNCH_BYTES                         # forward launch + inverse launch
HEADLINE_KERNEL = "relayout_vec_kernel<1,1,false,false> 131072x64x128 int8 Sw<5,2,5>"
# the 64 MiB bf16 workload (its output stays in L2): a row of the bench
BF16 = dict(tiles=4096, rows=128, cols=64, esize=2, bms=(3, 4, 3))


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-rows", action="store_true", help="skip the per-row measurements")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--case", default=None,
                   help="run one kernel case for a profiler and exit: relayout, relayout_bf16, relayout_bms, staging_probe, "
                        "relayout_staged, relayout_tma, transposes, transpose_u8, transpose_relayout, bank_profile")
    p.add_argument("--n", type=int, default=0, help="--case size (matrix edge / elements / patterns)")
    p.add_argument("--bms", default="1,1,1", help="--case relayout_bms: B,M,S (several sets separated by ';')")
    p.add_argument("--reps", type=int, default=2, help="--case launches per kernel")
    p.add_argument("--width", type=int, default=4, help="--case bank_profile: access bytes per lane")
    p.add_argument("--launcher-check", action="store_true",
                   help="check the multi-rank launch on CPU (gloo): each rank reports a fixed time, rank 0 "
                        "prints the world size and the slowest rank's time; no GPU, no bench line")
    return p.parse_args()


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def source_hash(*names) -> str:
    """Hash of the code in the named sources, comments and blank space
    removed: a comment edit does not make a committed ncu record stale."""
    import re
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "xor_swizzle_movement_gb300", "csrc", n), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def committed_traffic(kernel_key: str, src_hash: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel_key]
        if e.get("source_hash") == src_hash:
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """SM clocks, power and clock-event (throttle) reasons during the timed
    region.  Polls NVML every 1 ms through ctypes when the driver's library
    is present (read-only queries), else runs nvidia-smi at its fastest
    interval (50 ms).  Only samples taken between the region's start and end
    are kept."""

    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # clock-event reason bits of NVML's public API
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_slowdown"}
    NVML_CLOCK_SM = 1

    def __init__(self, gpu_id: str | None):
        self.rows = []          # (t, sm_mhz, max_mhz, power_w, {reasons})
        self.proc = None
        self.gpu_id = gpu_id
        self.source = None
        self._stop = threading.Event()
        self.thread = None

    # -- NVML --------------------------------------------------------------
    def _nvml_open(self):
        import ctypes
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return None
        if nv.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        ok = False
        if self.gpu_id:
            ok = nv.nvmlDeviceGetHandleByUUID(self.gpu_id.encode(), ctypes.byref(h)) == 0
        if not ok:
            idx = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0]
            ok = idx.isdigit() and nv.nvmlDeviceGetHandleByIndex_v2(int(idx), ctypes.byref(h)) == 0
        if not ok:
            nv.nvmlShutdown()
            return None
        reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        return nv, h, reasons_fn

    def _nvml_poll(self, nv, h, reasons_fn):
        import ctypes
        clk, mx, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        # the maximum clock is a fixed property and its query is slow: once
        top = mx.value if nv.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0 else None
        k = 0
        while not self._stop.is_set():
            t = time.perf_counter()
            sm = clk.value if nv.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(clk)) == 0 else None
            bits = rs.value if reasons_fn is not None and reasons_fn(h, ctypes.byref(rs)) == 0 else 0
            pw = None
            if k % 8 == 0 and nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0:
                pw = mw.value / 1000.0
            names = {n for b, n in self.REASON_BITS.items() if bits & b}
            self.rows.append((t, sm, top, pw, names))
            k += 1
            self._stop.wait(0.001)
        nv.nvmlShutdown()

    # -- nvidia-smi ----------------------------------------------------------
    def _smi_read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        for line in self.proc.stdout:
            p = [x.strip() for x in line.split(",")]
            if len(p) >= 8:
                self.rows.append((time.perf_counter(), num(p[0]), num(p[1]), num(p[2]),
                                  {names[i] for i in range(4) if p[4 + i].lower() == "active"}))

    def start(self):
        nvml = self._nvml_open()
        if nvml is not None:
            self.source = "nvml, 1 ms"
            # let the polling thread take the interpreter lock often while the
            # main thread launches (the default switch interval is 5 ms)
            self._switch = sys.getswitchinterval()
            sys.setswitchinterval(0.0005)
            self.thread = threading.Thread(target=self._nvml_poll, args=nvml, daemon=True)
            self.thread.start()
            return
        cmd = ["nvidia-smi", f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.source = "nvidia-smi, 50 ms"
        self.thread = threading.Thread(target=self._smi_read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.rows and time.time() - t0 < 5:
            time.sleep(0.02)

    def stop(self, t0: float, t1: float):
        """Summary of the samples taken in [t0, t1] (time.perf_counter)."""
        if self.thread is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        if self.proc is not None:
            time.sleep(0.06)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self._stop.set()
        self.thread.join(timeout=5)
        if getattr(self, "_switch", None):
            sys.setswitchinterval(self._switch)
        rows = [r for r in list(self.rows) if t0 <= r[0] <= t1]
        if not rows and self.proc is not None:   # region shorter than one nvidia-smi interval
            after = [r for r in list(self.rows) if r[0] > t1]
            rows = after[:1]
        sm = [r[1] for r in rows if r[1] is not None]
        mx = [r[2] for r in rows if r[2] is not None]
        pw = [r[3] for r in rows if r[3] is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(set().union(*[r[4] for r in rows])) if rows else [],
                "samples": len(rows), "source": self.source,
                "power_w_max": max(pw) if pw else None}


# ----------------------------------------------------------------------------


def reduce_max_ms(torch, total_ms: float, dist, device) -> float:
    """The slowest rank's timed milliseconds (all ranks get it)."""
    t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(world: int, bytes_per_step: int, steps: int, max_total_ms: float) -> float:
    """Whole-job GB/s: every rank moved bytes_per_step per step (weak scaling),
    timed by the slowest rank."""
    return world * bytes_per_step * steps / (max_total_ms * 1e-3) / GB


def make_flush(torch, dev):
    w = torch.empty(512 * MiB, dtype=torch.uint8, device=dev)
    r = torch.ones(512 * MiB // 4, dtype=torch.float32, device=dev)

    def flush():
        w.fill_(1)
        r.sum()
    return flush


def timed_launches(torch, fn, reps, flush, warm=3):
    """fn() launches kernels on the current stream; returns per-rep ms (events),
    L2 flushed before each rep."""
    st = torch.cuda.current_stream()
    for _ in range(warm):
        flush()
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        flush()
        a.record(st)
        fn()
        b.record(st)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def back_to_back_ms(torch, fn, reps=10, groups=3, warm=2):
    """Mean ms per launch over `reps` back-to-back launches (best of `groups`).
    For inputs larger than L2, where no launch finds the previous one's data
    in L2; avoids the ~2 us quantum of single-launch event timings."""
    st = torch.cuda.current_stream()
    for _ in range(warm):
        fn()
    best = None
    for _ in range(groups):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(reps):
            fn()
        b.record(st)
        b.synchronize()
        ms = a.elapsed_time(b) / reps
        best = ms if best is None else min(best, ms)
    return best


def staging_patterns(esize, variant):
    """Warp-wide shared-memory access patterns (byte addresses of lanes 0..31)
    of the transpose stagings: the first fill store and the first drain load
    of warp 0, as the kernels index their tiles; returns
    {access: (addresses, access_bytes)}."""
    if esize in (4, 8):
        n = 128 // esize                 # unit edge
        vpe = 16 // esize                # elements per 16-byte vector
        pitch = n + 1 if variant == 2 else n

        def phys(ir, ic):
            return ic ^ ir if variant == 0 else ic
        fill = [esize * ((lane >> 3) * pitch + phys(lane >> 3, (lane & 7) * vpe)) for lane in range(32)]
        drain = [esize * (((lane & 7) * vpe) * pitch + phys((lane & 7) * vpe, lane >> 3)) for lane in range(32)]
        return {"fill_store": (fill, esize), "drain_load": (drain, esize)}
    # 16-bit: 128-byte rows (144 with padding), 16-byte chunks
    pitch_b = 144 if variant == 2 else 128

    def chunk(row, ch):
        return ch ^ (row & 7) if variant in (0, 3) else ch
    fill = [(lane >> 3) * pitch_b + 16 * chunk(lane >> 3, lane & 7) for lane in range(32)]
    rows = [(lane >> 3) * 8 + (lane & 7) for lane in range(32)]     # ldmatrix.x4 row addresses
    drain = [r * pitch_b + 16 * chunk(r, 0) for r in rows]
    return {"fill_store": (fill, 16), "drain_ldmatrix": (drain, 16)}


def measure_rows(torch, swz, dev, flush, peak):
    """Each remaining row of the path at its full size (inputs drawn on the GPU
    from the row's seed).  Inputs larger than L2 are timed back to back; the
    2 MiB relayout is timed with L2 flushed (cold) and as a CUDA graph of 20
    steps (warm, no launch gaps)."""
    out = {}
    gen = torch.Generator(device=dev)

    def rand_bytes(n, seed):
        gen.manual_seed(seed)
        return torch.randint(0, 256, (n,), dtype=torch.uint8, device=dev, generator=gen)

    def summary(ms, nbytes):
        gbs = nbytes / (ms * 1e-3) / GB
        return {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 3)}

    def flushed_median(fn, nbytes):
        """Median of 20 single launches, each after an L2 flush and timed by
        its own event pair (event resolution about 2 us)."""
        return summary(statistics.median(timed_launches(torch, fn, 20, flush)), nbytes)

    # small relayout: 256 fp16 tiles 64x64, Swizzle<3,3,3>, forward then inverse (4 MiB moved per launch)
    src = rand_bytes(256 * 64 * 64 * 2, 0)
    a, b = torch.empty_like(src), torch.empty_like(src)

    def small_step():
        swz.swz_relayout(a, src, 256, 64, 64, 2, 3, 3, 3, 0)
        swz.swz_relayout(b, a, 256, 64, 64, 2, 3, 3, 3, 1)
    cold = statistics.mean(timed_launches(torch, small_step, 100, flush))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            small_step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(20):
            small_step()
    warm = back_to_back_ms(torch, graph.replay, reps=10) / 20
    def small_step_tma():
        swz.swz_relayout_tma(a, src, 256, 64, 64, 2, 3, 3, 3, 0)
        swz.swz_relayout_tma(b, a, 256, 64, 64, 2, 3, 3, 3, 1)
    cold_tma = statistics.mean(timed_launches(torch, small_step_tma, 100, flush))
    # the floor for a step this small: the same two dependent 2 MiB moves as
    # plain device-to-device copies (cudaMemcpyAsync), timed the same two ways
    def copy_step():
        a.copy_(src)
        b.copy_(a)
    copy_cold = statistics.mean(timed_launches(torch, copy_step, 100, flush))
    with torch.cuda.stream(side):
        for _ in range(3):
            copy_step()
    torch.cuda.current_stream().wait_stream(side)
    cgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cgraph):
        for _ in range(20):
            copy_step()
    copy_warm = back_to_back_ms(torch, cgraph.replay, reps=10) / 20
    out["relayout_fp16_64x64_sw333_2MiB"] = {
        "cold_l2": summary(cold, 8 * src.numel()), "warm_l2_graph": summary(warm, 8 * src.numel()),
        "tma_cold_l2": summary(cold_tma, 8 * src.numel()),
        "copy_floor_cold_l2": summary(copy_cold, 8 * src.numel()),
        "copy_floor_warm_l2_graph": summary(copy_warm, 8 * src.numel()),
        "note": "one step = forward + inverse, 8 MiB moved; too small for HBM: launch- and L2-bound. "
                "copy_floor: the same two dependent 2 MiB moves by cudaMemcpyAsync"}
    del src, a, b, graph, cgraph

    # the 64 MiB bf16 workload: Swizzle<3,4,3> relayout of 4096 tiles of 128 x 64
    # (N(0,1) from seed 1), forward then inverse, L2 flushed before every step
    # (one event pair per step).  64 MiB of output stays in the 126 MB L2, so
    # the inverse reads much of the forward's output from L2: L2-assisted.
    import numpy as np
    from xor_swizzle_movement_gb300 import inputs
    nt, nr, nc, ne = BF16["tiles"], BF16["rows"], BF16["cols"], BF16["esize"]
    bq, mq, sq = BF16["bms"]
    host = inputs.bf16_normal(nt * nr * nc, seed=1)
    src = torch.from_numpy(host.view(np.int16)).to(dev)
    a, b = torch.empty_like(src), torch.empty_like(src)

    def bf16_step():
        swz.swz_relayout(a, src, nt, nr, nc, ne, bq, mq, sq, 0)
        swz.swz_relayout(b, a, nt, nr, nc, ne, bq, mq, sq, 1)
    step_ms = statistics.mean(timed_launches(torch, bf16_step, 200, flush))
    torch.cuda.synchronize()
    assert torch.equal(b, src), "bf16 relayout round trip failed"
    moved = 4 * src.numel() * ne
    # what bounds it: the fixed cost of an event-timed launch after the flush
    # (one 16 KiB tile), and the same kernel copying 32 MiB that stays in L2
    one = statistics.mean(timed_launches(
        torch, lambda: swz.swz_relayout(a, src, 1, nr, nc, ne, bq, mq, sq, 0), 100, flush))
    half = src[: src.numel() // 2]
    l2_sw = back_to_back_ms(torch, lambda: swz.swz_relayout(a[: half.numel()], half, nt // 2, nr, nc, ne,
                                                            bq, mq, sq, 0), reps=50)
    out["relayout_bf16_4096x128x64_sw343_64MiB"] = {
        "step": summary(step_ms, moved),
        "note": "forward + inverse, L2 flushed before each step; L2-assisted: the 64 MiB output stays in "
                "the 126 MB L2, so the fraction is not an HBM figure",
        "one_tile_launch_after_flush_ms": round(one, 4),
        "l2_resident_32MiB_forward": summary(l2_sw, 2 * half.numel() * ne)}
    del src, a, b, half

    # the same Swizzle<3,3,3> fp16 64x64 tiles over 1 GiB: register path vs the TMA 128-byte mode
    src = rand_bytes(1 << 30, 4)
    dst = torch.empty_like(src)
    nt = (1 << 30) // 8192
    r = {}
    for name, fn in (("register", swz.swz_relayout), ("tma_128B", swz.swz_relayout_tma)):
        for d in (0, 1):
            ms = back_to_back_ms(torch, lambda: fn(dst, src, nt, 64, 64, 2, 3, 3, 3, d))
            r[f"{name}_{'forward' if d == 0 else 'inverse'}"] = summary(ms, 2 << 30)
    out["relayout_fp16_64x64_sw333_1GiB"] = r
    # Swizzle<2,4,2> on the same buffer: the TMA 128-byte mode with 32-byte atoms
    r = {}
    for name, fn in (("register", swz.swz_relayout), ("tma_128B_atom32B", swz.swz_relayout_tma)):
        for d in (0, 1):
            ms = back_to_back_ms(torch, lambda: fn(dst, src, nt, 64, 64, 2, 2, 4, 2, d))
            r[f"{name}_{'forward' if d == 0 else 'inverse'}"] = summary(ms, 2 << 30)
    r["tma_path"] = swz.swz_relayout_tma_path(dst, src, nt, 64, 64, 2, 2, 4, 2, 0)
    out["relayout_fp16_64x64_sw242_1GiB"] = r
    del src, dst

    src = rand_bytes(1 << 30, 4)
    dst = torch.empty_like(src)
    n_tiles = (1 << 30) // (64 * 128)
    out["relayout_int8_64x128_sw525_1GiB_flushed"] = {
        "forward_flushed_median_20": flushed_median(
            lambda: swz.swz_relayout(dst, src, n_tiles, 64, 128, 1, 5, 2, 5, 0), 2 << 30),
        "note": "the headline's forward launch, each after an L2 flush, timed by its own event pair"}

    # one 1 GiB uint16 buffer, every (B, M, S) with B 1..5, M 0..4, S B..7, forward
    n = 1 << 29
    res = []
    for Bq in range(1, 6):
        for Mq in range(0, 5):
            for Sq in range(Bq, 8):
                ms = back_to_back_ms(torch, lambda: swz.swz_relayout(dst, src, 1, 1, n, 2, Bq, Mq, Sq, 0),
                                     reps=3, groups=2, warm=1)
                res.append(((2 << 30) / (ms * 1e-3) / GB, (Bq, Mq, Sq)))
    res.sort()
    vals = [r[0] for r in res]
    out["relayout_uint16_1GiB_sweep125"] = {
        "min": {"GB/s": round(vals[0], 1), "BMS": res[0][1]},
        "median_GB/s": round(statistics.median(vals), 1),
        "max": {"GB/s": round(vals[-1], 1), "BMS": res[-1][1]},
        "min_frac_of_hbm": round(vals[0] / peak, 3)}

    # negative SShift on the same buffer, forward: one parameter set per relayout path
    neg = {}
    for label, (Bq, Mq, Sq) in (("whole_vectors_sw33m3", (3, 3, -3)), ("lane_map_sw20m1", (2, 0, -1)),
                                ("warp_shuffles_sw30m4", (3, 0, -4)), ("cosets_of_4_sw31m7", (3, 1, -7)),
                                ("cosets_of_2_sw42m9", (4, 2, -9)), ("cosets_of_8_sw40m9", (4, 0, -9)),
                                ("warp_shuffles_lane_map_sw30m2", (3, 0, -2)),
                                ("cosets_lane_map_sw160m2", (16, 0, -2))):
        ms = back_to_back_ms(torch, lambda: swz.swz_relayout(dst, src, 1, 1, n, 2, Bq, Mq, Sq, 0),
                             reps=3, groups=2, warm=1)
        neg[label] = summary(ms, 2 << 30)
    neg["note"] = "1 GiB uint16 as one tile, forward; the path each set takes is in its label"
    # every negative set of the sweep's ranges with the read field in the lanes
    # (B 1..5, M below log2 V, S -1..-5), uint16 and int8, forward
    sweep = []
    for esize, lv in ((2, 3), (1, 4)):
        ne = (1 << 30) // esize
        for Bq in range(1, 6):
            for Mq in range(lv):
                for Sq in range(-1, -6, -1):
                    ms = back_to_back_ms(torch, lambda: swz.swz_relayout(dst, src, 1, 1, ne, esize, Bq, Mq, Sq, 0),
                                         reps=3, groups=2, warm=1)
                    sweep.append(((2 << 30) / (ms * 1e-3) / GB, (esize, Bq, Mq, Sq)))
    sweep.sort()
    sv = [v for v, _ in sweep]
    neg["sweep_175"] = {
        "min": {"GB/s": round(sv[0], 1), "esize_BMS": sweep[0][1]},
        "median_GB/s": round(statistics.median(sv), 1),
        "max": {"GB/s": round(sv[-1], 1), "esize_BMS": sweep[-1][1]},
        "below_0.96_of_hbm": sum(1 for v in sv if v < 0.96 * peak),
        "lowest_5": [[round(v / peak, 3), list(k)] for v, k in sweep[:5]]}
    out["relayout_uint16_1GiB_negative_shift"] = neg
    del src, dst

    # transposes, with the bank model's prediction for each staging's warp accesses
    pat_rows, pat_keys = [], []
    for esize, variants in ((4, (0, 1, 2)), (2, (0, 3, 1, 2)), (8, (0, 1, 2))):
        for v in variants:
            for access, (addrs, width) in staging_patterns(esize, v).items():
                pat_rows.append((addrs, width))
                pat_keys.append((esize, v, access))
    ways_model = {}
    for width in sorted({w for _, w in pat_rows}):
        idx = [i for i, (_, w) in enumerate(pat_rows) if w == width]
        pats = torch.tensor([pat_rows[i][0] for i in idx], dtype=torch.int32, device=dev)
        wy = torch.empty(len(idx), dtype=torch.int32, device=dev)
        wf = torch.empty(len(idx), dtype=torch.int32, device=dev)
        swz.swz_bank_profile(pats, None, len(idx), width, wy, wf)
        for j, i in enumerate(idx):
            ways_model[pat_keys[i]] = int(wy[j].item())

    def transpose_rows(name, n, esize, variants, seed):
        s_ = rand_bytes(n * n * esize, seed)
        d_ = torch.empty_like(s_)
        r = {}
        for v, vname in variants:
            ms = back_to_back_ms(torch, lambda: swz.swz_transpose(d_, s_, n, n, esize, v))
            r[vname] = summary(ms, 2 * n * n * esize)
            r[vname]["flushed_median_20"] = flushed_median(
                lambda: swz.swz_transpose(d_, s_, n, n, esize, v), 2 * n * n * esize)
            r[vname]["bank_model_ways"] = {acc: ways_model[(esize, v, acc)]
                                           for (e_, v_, acc) in pat_keys if e_ == esize and v_ == v}
        out[name] = r

    transpose_rows("transpose_fp32_8192", 8192, 4, [(0, "swizzled_sw505"), (1, "unswizzled"), (2, "padded_33")], 2)
    transpose_rows("transpose_fp16_16384", 16384, 2,
                   [(0, "swizzled_sw343_ldmatrix"), (3, "tma_swizzle128b"), (1, "unswizzled"), (2, "padded")], 3)
    transpose_rows("transpose_fp64_8192", 8192, 8, [(0, "swizzled_sw404"), (1, "unswizzled"), (2, "padded_17")], 4)

    # the same swizzled fp32 kernel when the output rows are not 32 KiB apart:
    # 8256 x 8192 (output pitch 33 KiB) and 16384 x 16384 (64 KiB)
    pitch = {}
    for r_, c_ in ((8256, 8192), (16384, 16384)):
        s_ = rand_bytes(r_ * c_ * 4, 2)
        d_ = torch.empty_like(s_)
        ms = back_to_back_ms(torch, lambda: swz.swz_transpose(d_, s_, r_, c_, 4, 0))
        pitch[f"{r_}x{c_}_output_pitch_{r_ * 4}B"] = summary(ms, 2 * r_ * c_ * 4)
        del s_, d_
    out["transpose_fp32_swizzled_output_pitch"] = pitch

    # tiles that are not whole 16-byte vectors (not a configured workload): 256 MiB
    # each, staged in shared memory (aligned pointers) or element by element
    # (a source 2 bytes off 16-byte alignment)
    rag = {}
    nb = (256 * MiB) // 120 * 120
    s_ = rand_bytes(nb + 64, 4)
    d_ = torch.empty_like(s_)
    for name, args_ in (("u8_tile24_sw201", (nb // 24, 1, 24, 1, 2, 0, 1)),
                        ("u8_tile24_sw123_4byte_units", (nb // 24, 1, 24, 1, 1, 2, 3)),
                        ("u16_tile3x4_sw201", (nb // 24, 3, 4, 2, 2, 0, 1)),
                        ("u32_tile30_sw105", (nb // 120, 1, 30, 4, 1, 0, 5))):
        ms = back_to_back_ms(torch, lambda: swz.swz_relayout(d_, s_[:nb], *args_, 0))
        rag[name] = summary(ms, 2 * nb)
    # 16-bit 64 x 64 tiles, Swizzle<3,3,3>, 240 MiB (larger than L2), with pointers off 16-byte alignment
    nu = 240 * MiB
    for name, so, do in (("u16_64x64_sw333_source_plus_2B", 2, 0), ("u16_64x64_sw333_destination_plus_2B", 0, 2),
                         ("u16_64x64_sw333_source_plus_6B_destination_plus_10B", 6, 10)):
        s_off, d_off = s_[so:so + nu], d_[do:do + nu]
        ms = back_to_back_ms(torch, lambda: swz.swz_relayout(d_off, s_off, nu // 8192, 64, 64, 2, 3, 3, 3, 0))
        rag[name] = summary(ms, 2 * nu)
    out["relayout_ragged_or_unaligned"] = rag
    del s_, d_, s_off, d_off

    # 1-byte elements (not a configured workload): 16384 x 16384 bytes, the
    # swizzled 128 x 128 byte tiles against the element-wise unswizzled staging
    s_ = rand_bytes(16384 * 16384, 4)
    d_ = torch.empty_like(s_)
    u8 = {}
    for v, vname in ((0, "swizzled_byte_sw347"), (1, "unswizzled")):
        ms = back_to_back_ms(torch, lambda: swz.swz_transpose(d_, s_, 16384, 16384, 1, v))
        u8[vname] = summary(ms, 2 * 16384 * 16384)
    out["transpose_u8_16384"] = u8
    del s_, d_

    # transpose fused with the relayout: a 64 x 2^21 bf16 matrix (256 MiB) into K-major 128 x 64
    # tiles under Swizzle<3,4,3>, in one pass, against the transpose and the relayout apart
    kr, kc = 64, 1 << 21
    s_ = rand_bytes(kr * kc * 2, 1)
    d_ = torch.empty_like(s_)
    t_ = torch.empty_like(s_)
    fused = back_to_back_ms(torch, lambda: swz.swz_transpose_relayout(d_, s_, kr, kc, 2, 8192, 3, 4, 3))

    def two_pass():
        swz.swz_transpose(t_, s_, kr, kc, 2, 0)
        swz.swz_relayout(d_, t_, kr * kc // 8192, 128, 64, 2, 3, 4, 3, 0)
    two = back_to_back_ms(torch, two_pass)
    plain = back_to_back_ms(torch, lambda: swz.swz_transpose(t_, s_, kr, kc, 2, 0))
    nb = kr * kc * 2
    out["transpose_relayout_bf16_64x2M_kmajor_sw343"] = {
        "fused": summary(fused, 2 * nb), "transpose_alone": summary(plain, 2 * nb),
        "two_pass": {"ms": round(two, 4), "speedup_of_fused": round(two / fused, 2)}}
    del s_, d_, t_

    # bank profiler: 2^22 random aligned 4-byte patterns (512 MiB of addresses)
    npat = 1 << 22
    gen.manual_seed(5)
    pats = (torch.randint(0, 228 * 1024 // 4, (npat, 32), dtype=torch.int32, device=dev, generator=gen) * 4)
    ways = torch.empty(npat, dtype=torch.int32, device=dev)
    wf = torch.empty(npat, dtype=torch.int32, device=dev)
    def profile_row(width, act):
        # bytes per pattern: 128 of addresses and 4 of mask read, 8 of results written
        per = 136 + (4 if act is not None else 0)
        ms = back_to_back_ms(torch, lambda: swz.swz_bank_profile(pats, act, npat, width, ways, wf))
        gbs = npat * per / (ms * 1e-3) / GB
        return {"ms": round(ms, 4), "Gpatterns/s": round(npat / (ms * 1e-3) / 1e9, 3), "GB/s": round(gbs, 1),
                "frac_of_hbm": round(gbs / peak, 3)}
    out["bank_profile_4M_patterns_w4"] = profile_row(4, None)
    masks = torch.randint(-(1 << 31), 1 << 31, (npat,), dtype=torch.int64, device=dev, generator=gen).to(torch.int32)
    other = {"w4_masked": profile_row(4, masks)}
    for width in (1, 2, 8, 16):
        pats.bitwise_and_(~(width - 1))  # addresses aligned to the width (all are multiples of 4)
        other[f"w{width}"] = profile_row(width, None)
    pats.add_(2)  # every 4-byte access straddles two words: the word-key path
    other["w4_all_unaligned"] = profile_row(4, None)
    out["bank_profile_4M_patterns_other_widths"] = other
    del pats, masks, ways, wf

    # batched slice collision: 2^27 64-bit masks (1 GiB in, 1 GiB out), Swizzle<3,4,3>
    nm = 1 << 27
    gen.manual_seed(6)
    masks = torch.randint(0, 1 << 62, (nm,), dtype=torch.int64, device=dev, generator=gen)
    coll = torch.empty_like(masks)
    ms = back_to_back_ms(torch, lambda: swz.swz_slice_collision_batch(masks, nm, 3, 4, 3, coll))
    out["slice_collision_128M_masks"] = {**summary(ms, 16 * nm), "Gmasks/s": round(nm / (ms * 1e-3) / 1e9, 2)}
    del masks, coll
    return out


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


# The oracle over every host core: spawned worker processes (no CUDA state is
# inherited) attach to the input in shared memory and each runs the oracle,
# unchanged, on its own run of tiles: the oracle's outer loop split across
# processes.
_POOL = {}


def _pool_init(shm_name, nbytes):
    import numpy as np
    from multiprocessing import shared_memory
    shm = shared_memory.SharedMemory(name=shm_name)
    _POOL["shm"] = shm
    _POOL["buf"] = np.ndarray((nbytes,), dtype=np.uint8, buffer=shm.buf)


def _pool_job(job):
    """('pair' | 'fwd', dtype, e0, e1, tile, B, M, S): forward (then inverse,
    for 'pair') relayout of elements [e0, e1) of the shared buffer viewed as
    dtype; ('transpose', dtype, r0, r1, cols): transpose of rows [r0, r1) of a
    row-major matrix with `cols` columns at the start of the buffer."""
    import numpy as np
    import oracle
    kind, dtype = job[0], np.dtype(job[1])
    view = _POOL["buf"].view(dtype)
    if kind == "transpose":
        _, _, r0, r1, cols = job
        oracle.transpose(view[r0 * cols:r1 * cols].reshape(r1 - r0, cols))
        return (r1 - r0) * cols
    _, _, e0, e1, te, b, m, s = job
    out = oracle.relayout(view[e0:e1], tile_elems=te, B=b, M=m, S=s, direction=0)
    if kind == "pair":
        oracle.relayout(out, tile_elems=te, B=b, M=m, S=s, direction=1)
    return e1 - e0


def _timed_rounds(fn, seconds):
    t_end = time.perf_counter() + seconds
    times = []
    while True:
        t0 = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t0)
        if time.perf_counter() > t_end:
            return times


def cpu_baseline(host_src, seconds=10.0, seconds_all=5.0, sweep_el=1 << 25, sample_scale=1,
                 sample_tiles=4096):
    """The CPU oracle, as it stands, on the headline workload (forward then
    inverse): single thread on a bounded sample of `sample_tiles` tiles for
    about `seconds`, then the whole workload split over every core of this
    process's affinity set for about `seconds_all`.  Also the relayout
    sweep's 125 parameter sets on a 64 MiB uint16 sample, over all cores and
    single-threaded on three of them; and every other row's workload on a
    bounded sample, single thread and over all cores.  `sample_scale`
    divides the other rows' samples (tests)."""
    import numpy as np
    import multiprocessing as mp
    from multiprocessing import shared_memory
    import oracle
    from xor_swizzle_movement_gb300 import inputs
    te = ROWS * COLS
    n_tiles = host_src.size // te
    sample_tiles = min(sample_tiles, n_tiles)
    part = host_src[: sample_tiles * te]
    times = _timed_rounds(lambda: oracle.relayout(
        oracle.relayout(part, tile_elems=te, B=B, M=M, S=S, direction=0),
        tile_elems=te, B=B, M=M, S=S, direction=1), seconds)
    mean = sum(times) / len(times)
    moved = 4 * part.nbytes
    res = {"value": round(moved / mean / GB, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"forward + inverse of {sample_tiles} of the {n_tiles} tiles, {len(times)} repetitions, "
                     f"{mean * 1e3:.1f} ms each, single thread",
           "cpu_model": cpu_model()}

    cores = len(os.sched_getaffinity(0))
    band = max(8, 256 // sample_scale)                   # transpose rows per worker
    bf = BF16["tiles"] * BF16["rows"] * BF16["cols"] * BF16["esize"]
    nbytes = max(host_src.nbytes, sweep_el * 2, band * cores * 8192 * 8, band * cores * 16384 * 2, bf)
    shm = shared_memory.SharedMemory(create=True, size=nbytes)

    def wall(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0
    try:
        buf = np.ndarray((nbytes,), dtype=np.uint8, buffer=shm.buf)
        u16 = buf.view(np.uint16)
        with mp.get_context("spawn").Pool(cores, initializer=_pool_init, initargs=(shm.name, nbytes)) as pool:
            # the headline workload, tiles split into 4 runs per core
            buf[:host_src.size] = host_src.reshape(-1)
            n_runs = 4 * cores
            cuts = [n_tiles * i // n_runs for i in range(n_runs + 1)]
            jobs = [("pair", "u1", cuts[i] * te, cuts[i + 1] * te, te, B, M, S)
                    for i in range(n_runs) if cuts[i + 1] > cuts[i]]
            pool.map(_pool_job, jobs)                    # warm: every worker has loaded the oracle
            t_all = _timed_rounds(lambda: pool.map(_pool_job, jobs), seconds_all)
            m_all = sum(t_all) / len(t_all)
            res["all_cores"] = {"value": round(4 * host_src.nbytes / m_all / GB, 3), "unit": "GB/s", "cores": cores,
                                "sample": f"whole workload, {len(t_all)} repetitions, {m_all * 1e3:.1f} ms each, "
                                          f"{len(jobs)} runs of tiles over {cores} processes"}
            # the relayout sweep: one 2^25-element tile (a prefix of the 2^29-element buffer; every
            # swizzle period divides it), forward, all 125 parameter sets
            u16[:sweep_el] = inputs.uint16_bits(sweep_el, seed=4)
            combos = [(b, m, s) for b in range(1, 6) for m in range(5) for s in range(b, 8)]
            sweep_jobs = [("fwd", "<u2", 0, sweep_el, sweep_el, b, m, s) for (b, m, s) in combos]
            t_sweep = wall(lambda: pool.map(_pool_job, sweep_jobs, chunksize=1))
            one = {}
            for (b, m, s) in ((1, 4, 7), (3, 3, 3), (5, 2, 5)):
                t = wall(lambda: oracle.relayout(u16[:sweep_el], tile_elems=sweep_el, B=b, M=m, S=s, direction=0))
                one[f"{b},{m},{s}"] = round(2 * sweep_el * 2 / t / GB, 3)
            res["sweep125_uint16"] = {
                "all_cores_GB/s": round(len(combos) * 2 * sweep_el * 2 / t_sweep / GB, 3), "cores": cores,
                "single_thread_GB/s": one,
                "sample": f"forward relayout of a {sweep_el * 2 / MiB:g} MiB prefix of the 1 GiB buffer, "
                          f"{len(combos)} parameter sets"}

            # every other row: one run on one core, then one band per core at once
            other = {}

            def row(name, moved_one, run_one, moved_all, all_jobs, sample):
                pool.map(_pool_job, all_jobs)            # warm
                other[name] = {"single_thread_GB/s": round(moved_one / wall(run_one) / GB, 3),
                               "all_cores_GB/s": round(moved_all / wall(lambda: pool.map(_pool_job, all_jobs)) / GB, 3),
                               "cores": cores, "sample": sample}
            small = inputs.uint16_bits(256 * 4096, seed=0)
            u16[:small.size] = small
            cut = [256 * i // cores for i in range(cores + 1)]
            row("relayout_fp16_64x64_sw333_2MiB", 4 * small.nbytes,
                lambda: oracle.relayout(oracle.relayout(u16[:small.size], tile_elems=4096, B=3, M=3, S=3, direction=0),
                                        tile_elems=4096, B=3, M=3, S=3, direction=1),
                4 * small.nbytes,
                [("pair", "<u2", cut[i] * 4096, cut[i + 1] * 4096, 4096, 3, 3, 3)
                 for i in range(cores) if cut[i + 1] > cut[i]],
                "whole workload, forward + inverse; all cores: its 256 tiles split over the cores")
            hb = inputs.bf16_normal(bf // 2, seed=1)
            u16[:hb.size] = hb
            bt = BF16["tiles"]
            bte = BF16["rows"] * BF16["cols"]
            bq, mq, sq = BF16["bms"]
            cut = [bt * i // cores for i in range(cores + 1)]
            one_tiles = max(16, 512 // sample_scale)
            row("relayout_bf16_4096x128x64_sw343_64MiB", 4 * one_tiles * bte * 2,
                lambda: oracle.relayout(oracle.relayout(u16[:one_tiles * bte], tile_elems=bte, B=bq, M=mq, S=sq,
                                                        direction=0), tile_elems=bte, B=bq, M=mq, S=sq, direction=1),
                4 * bf,
                [("pair", "<u2", cut[i] * bte, cut[i + 1] * bte, bte, bq, mq, sq)
                 for i in range(cores) if cut[i + 1] > cut[i]],
                f"forward + inverse; single thread {one_tiles} of the {bt} tiles; all cores: the whole workload")
            for name, n, esize, dt, gen in (
                    ("transpose_fp32_8192", 8192, 4, "<u4", lambda k: inputs.f32_uniform(k, seed=2).view(np.uint32)),
                    ("transpose_fp16_16384", 16384, 2, "<u2", lambda k: inputs.f16_bits_no_nan(k, seed=3)),
                    ("transpose_fp64_8192", 8192, 8, "<u8",
                     lambda k: inputs.random_bytes(8 * k, seed=4).view(np.uint64))):
                rows = min(n, band * cores)
                view = buf.view(np.dtype(dt))
                view[:rows * n] = gen(rows * n)
                row(name, 2 * band * n * esize, lambda: oracle.transpose(view[:band * n].reshape(band, n)),
                    2 * rows * n * esize,
                    [("transpose", dt, r0, min(rows, r0 + band), n) for r0 in range(0, rows, band)],
                    f"{band} rows; all cores: {rows} rows of the {n} in bands of {band}")
            res["other_rows"] = other
    finally:
        shm.close()
        shm.unlink()
    return res


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, single thread, on a
    bounded sample of the headline workload's tiles per step (at most 4096,
    fewer when K + W steps would take over about a minute)."""
    rank, world, _ = dist_info()
    if rank != 0:
        return
    from xor_swizzle_movement_gb300 import inputs
    import oracle
    te = ROWS * COLS
    probe_tiles = 256
    host = inputs.random_bytes(4096 * te, seed=4)   # the first 4096 tiles of the 1 GiB buffer
    probe = host[: probe_tiles * te]
    t0 = time.perf_counter()
    oracle.relayout(oracle.relayout(probe, tile_elems=te, B=B, M=M, S=S, direction=0),
                    tile_elems=te, B=B, M=M, S=S, direction=1)
    per_tile = (time.perf_counter() - t0) / probe_tiles
    budget = 60.0 / max(1, args.steps + args.warmup)
    sample_tiles = int(max(16, min(4096, budget / per_tile)))
    part = host[: sample_tiles * te]
    step_bytes = 4 * part.nbytes
    for _ in range(args.warmup):
        oracle.relayout(oracle.relayout(part, tile_elems=te, B=B, M=M, S=S, direction=0),
                        tile_elems=te, B=B, M=M, S=S, direction=1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        f = oracle.relayout(part, tile_elems=te, B=B, M=M, S=S, direction=0)
        oracle.relayout(f, tile_elems=te, B=B, M=M, S=S, direction=1)
    dt = time.perf_counter() - t0
    value = step_bytes * args.steps / dt / GB
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample_tiles": sample_tiles},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{sample_tiles} of {TILES} tiles per step, forward + inverse, single thread"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_case(args):
    """Launch one kernel case `reps` times (no timing): the command a profiler wraps."""
    import torch
    import xor_swizzle_movement_gb300 as swz
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    swz.lib()
    gen = torch.Generator(device=dev)
    gen.manual_seed(4)

    def rand_bytes(n):
        return torch.randint(0, 256, (n,), dtype=torch.uint8, device=dev, generator=gen)

    done = []
    if args.case == "relayout":            # the headline workload, forward + inverse
        nbytes = (args.n or N_BYTES) // (ROWS * COLS) * (ROWS * COLS)
        src = rand_bytes(nbytes)
        a, b = torch.empty_like(src), torch.empty_like(src)
        nt = nbytes // (ROWS * COLS * ESIZE)
        for _ in range(args.reps):
            swz.swz_relayout(a, src, nt, ROWS, COLS, ESIZE, B, M, S, 0)
            swz.swz_relayout(b, a, nt, ROWS, COLS, ESIZE, B, M, S, 1)
        done.append(f"relayout int8 {nt} tiles of 64x128 Sw<5,2,5> fwd+inv")
    elif args.case == "relayout_bf16":     # the 64 MiB bf16 workload, forward + inverse
        nt, nr, nc, ne = BF16["tiles"], BF16["rows"], BF16["cols"], BF16["esize"]
        src = rand_bytes(nt * nr * nc * ne)
        a, b = torch.empty_like(src), torch.empty_like(src)
        for _ in range(args.reps):
            swz.swz_relayout(a, src, nt, nr, nc, ne, *BF16["bms"], 0)
            swz.swz_relayout(b, a, nt, nr, nc, ne, *BF16["bms"], 1)
        done.append("relayout bf16 64 MiB Sw<3,4,3> fwd+inv")
    elif args.case == "relayout_bms":      # one uint16 buffer as one tile, forward, per parameter set
        n = args.n or (1 << 27)
        src = rand_bytes(2 * n)
        dst = torch.empty_like(src)
        for bms in args.bms.split(";"):
            Bq, Mq, Sq = (int(v) for v in bms.split(","))
            for _ in range(args.reps):
                swz.swz_relayout(dst, src, 1, 1, n, 2, Bq, Mq, Sq, 0)
            done.append(f"relayout uint16 n={n} Sw<{Bq},{Mq},{Sq}>")
    elif args.case == "relayout_staged":   # ragged 24-byte tiles staged in shared memory
        nbytes = (args.n or (256 << 20)) // 24 * 24
        src = rand_bytes(nbytes)
        dst = torch.empty_like(src)
        for _ in range(args.reps):
            swz.swz_relayout(dst, src, nbytes // 24, 3, 4, 2, 2, 0, 1, 0)     # uint16 3 x 4, Sw<2,0,1>
            swz.swz_relayout(dst, src, nbytes // 24, 1, 24, 1, 1, 2, 3, 0)    # int8 24, Sw<1,2,3>
            swz.swz_relayout(dst, src, nbytes // 24, 1, 24, 1, 2, 0, 1, 0)    # int8 24, Sw<2,0,1>: 1-byte units
        done.append(f"relayout staged bytes={nbytes}")
    elif args.case == "transposes":        # every staging of the fp32 / fp16 / fp64 transposes
        for esize, n, variants in ((4, args.n or 8192, (0, 1, 2)), (2, args.n or 8192, (0, 3, 1, 2)),
                                   (8, (args.n or 8192) // 2, (0, 1, 2))):
            src = rand_bytes(n * n * esize)
            dst = torch.empty_like(src)
            for v in variants:
                for _ in range(args.reps):
                    swz.swz_transpose(dst, src, n, n, esize, v)
                done.append(f"transpose esize={esize} n={n} variant={v}")
            del src, dst
    elif args.case == "relayout_tma":      # 16-bit 64 x 64 tiles, Swizzle<3,3,3> on the TMA 128-byte mode
        nbytes = args.n or (256 << 20)
        src = rand_bytes(nbytes)
        a, b = torch.empty_like(src), torch.empty_like(src)
        for _ in range(args.reps):
            swz.swz_relayout_tma(a, src, nbytes // 8192, 64, 64, 2, 3, 3, 3, 0)
            swz.swz_relayout_tma(b, a, nbytes // 8192, 64, 64, 2, 3, 3, 3, 1)
        done.append(f"relayout_tma fwd+inv bytes={nbytes}")
    elif args.case == "transpose_u8":  # n x n bytes, swizzled and unswizzled stagings
        n = args.n or 8192
        src = rand_bytes(n * n)
        dst = torch.empty_like(src)
        for v in (0, 1):
            for _ in range(args.reps):
                swz.swz_transpose(dst, src, n, n, 1, v)
            done.append(f"transpose esize=1 n={n} variant={v}")
    elif args.case == "transpose_relayout":  # 64 x n bf16 into K-major 128 x 64 Swizzle<3,4,3> tiles
        cols = args.n or (1 << 20)
        src = rand_bytes(64 * cols * 2)
        dst = torch.empty_like(src)
        for _ in range(args.reps):
            swz.swz_transpose_relayout(dst, src, 64, cols, 2, 8192, 3, 4, 3)
        done.append(f"transpose_relayout 64 x {cols}")
    elif args.case == "staging_probe":     # every transpose staging on registers, then with global traffic
        # two shapes: persistent CTAs that repeat the staging (4 per SM, `iters` rounds), and one round
        # per CTA over as many CTAs as the 8192^2 fp32 transpose launches (16384)
        iters = args.n or 64
        shapes = [(iters, torch.cuda.get_device_properties(dev).multi_processor_count * 4), (1, 16384)]
        gbytes = 256 << 20                 # larger than L2: the streamed data comes from DRAM
        gsrc, gdst = rand_bytes(gbytes), torch.empty(gbytes, dtype=torch.uint8, device=dev)
        stagings = [(4, 0), (4, 1), (4, 2), (2, 0), (2, 1), (2, 2), (2, 3), (8, 0), (8, 1), (8, 2), (1, 0)]
        for it_, ctas in shapes:
            for mode in ("shared_only", "with_global"):
                for esize, v in stagings:
                    for _ in range(args.reps):
                        if mode == "shared_only":
                            swz.swz_staging_probe(esize, v, it_, ctas)     # no global access at all
                        else:
                            swz.swz_staging_probe(esize, v, it_, ctas, gsrc=gsrc, gdst=gdst, gbytes=gbytes)
                    done.append(f"staging_probe esize={esize} variant={v} {mode} iters={it_} ctas={ctas}")
    elif args.case == "bank_profile":
        n = args.n or (1 << 20)
        width = args.width
        pats = torch.randint(0, 228 * 1024 // width, (n, 32), dtype=torch.int32, device=dev, generator=gen) * width
        w = torch.empty(n, dtype=torch.int32, device=dev)
        f = torch.empty(n, dtype=torch.int32, device=dev)
        for _ in range(args.reps):
            swz.swz_bank_profile(pats, None, n, width, w, f)
        done.append(f"bank_profile n={n} width={width}")
    else:
        raise SystemExit(f"unknown --case {args.case}")
    torch.cuda.synchronize()
    print(json.dumps({"case": args.case, "launched": done, "reps": args.reps}), flush=True)


def relaunch_command(argv, n_gpus: int, port: int):
    """The torch.distributed.run command that runs this script on n_gpus
    ranks of one node (used when --gpus N > 1 is given without torchrun)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n_gpus}",
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]


def _free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def e2e_host_abi(torch, swz, host_in, steps: int):
    """The step through the C ABI on pinned host buffers: the forward launch
    reads the host input over the host link, the inverse launch writes the
    host output.  Consecutive steps alternate between two streams (and two
    device buffers and two host outputs).  Step k's forward waits for step
    k - 1's forward and step k's inverse for step k - 1's inverse, so the
    launches pair up: step k's forward (reading the host) runs beside step
    k - 1's inverse (writing it), both directions of the link carry data at
    once, and two inverses never share the device-to-host direction.  (The
    library runs relayouts on host buffers on a grid sized for the link, so
    the two kernels fit on the GPU together.)  Returns seconds per step (CUDA
    events) and checks both outputs."""
    dev = torch.cuda.current_device()
    phys = [torch.empty(N_BYTES, dtype=torch.uint8, device=dev) for _ in range(2)]
    outs = [torch.zeros(N_BYTES, dtype=torch.uint8).pin_memory() for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    fwd_done = [torch.cuda.Event(), torch.cuda.Event()]
    inv_done = [torch.cuda.Event(), torch.cuda.Event()]
    main = torch.cuda.current_stream()

    def run(n):
        for k in range(n):
            st, j = streams[k % 2], k % 2
            if k > 0:
                st.wait_event(fwd_done[1 - j])   # the previous step's forward has finished
            swz.swz_relayout(phys[j], host_in.data_ptr(), TILES, ROWS, COLS, ESIZE, B, M, S, 0, stream=st)
            fwd_done[j].record(st)
            if k > 0:
                st.wait_event(inv_done[1 - j])   # the previous step's inverse has finished
            swz.swz_relayout(outs[j].data_ptr(), phys[j], TILES, ROWS, COLS, ESIZE, B, M, S, 1, stream=st)
            inv_done[j].record(st)
    for st in streams:
        st.wait_stream(main)
    run(2)
    for st in streams:
        main.wait_stream(st)
    torch.cuda.synchronize()
    for o in outs:
        o.zero_()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for st in streams:
        st.wait_stream(main)
    run(steps)
    for st in streams:
        main.wait_stream(st)
    e1.record(main)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, host_in), "end-to-end round trip through host buffers failed"
    return e0.elapsed_time(e1) * 1e-3 / steps


def e2e_copy_engine(torch, swz, host_in, src, steps_per_graph=4, n_chunks=8, replays=3):
    """The same step fed by the copy engines: each step's input goes in by
    chunks over three streams (copy in / relayout forward + inverse / copy
    out), consecutive steps alternate between two buffer sets, and several
    steps form one CUDA graph.  Returns seconds per step (host clock) and the
    plain copy rates."""
    ct = TILES // n_chunks
    ce = ct * ROWS * COLS * ESIZE
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    buf_sets = [tuple(torch.empty_like(src) for _ in range(3)) for _ in range(2)]
    out_hosts = [torch.empty_like(host_in).pin_memory() for _ in range(2)]
    ev = {key: [[torch.cuda.Event() for _ in range(n_chunks)] for _ in range(steps_per_graph)]
          for key in ("in", "run", "out")}

    def enqueue():
        for k in range(steps_per_graph):
            d_in_k, phys_k, back_k = buf_sets[k % 2]
            out_k = out_hosts[k % 2]
            for c in range(n_chunks):
                sl = slice(c * ce, (c + 1) * ce)
                if k >= 2:
                    s_in.wait_event(ev["run"][k - 2][c])   # that step's relayout has read d_in
                with torch.cuda.stream(s_in):
                    d_in_k[sl].copy_(host_in[sl], non_blocking=True)
                    ev["in"][k][c].record(s_in)
                s_run.wait_event(ev["in"][k][c])
                if k >= 2:
                    s_run.wait_event(ev["out"][k - 2][c])  # that step's copy-out has read back
                with torch.cuda.stream(s_run):
                    swz.swz_relayout(phys_k[sl], d_in_k[sl], ct, ROWS, COLS, ESIZE, B, M, S, 0, stream=s_run)
                    swz.swz_relayout(back_k[sl], phys_k[sl], ct, ROWS, COLS, ESIZE, B, M, S, 1, stream=s_run)
                    ev["run"][k][c].record(s_run)
                s_out.wait_event(ev["run"][k][c])
                with torch.cuda.stream(s_out):
                    out_k[sl].copy_(back_k[sl], non_blocking=True)
                    ev["out"][k][c].record(s_out)

    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=cap):
        for s_ in (s_in, s_run, s_out):
            s_.wait_stream(cap)
        enqueue()
        for s_ in (s_in, s_run, s_out):
            cap.wait_stream(s_)
    for o in out_hosts:
        o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(replays):
        graph.replay()
    torch.cuda.synchronize()
    per_step = (time.perf_counter() - t0) / (replays * steps_per_graph)
    for o in out_hosts:
        assert torch.equal(o, host_in), "copy-engine end-to-end round trip failed"
    d_in, out_host = buf_sets[1][0], out_hosts[0]
    t0 = time.perf_counter()
    for _ in range(2):
        d_in.copy_(host_in, non_blocking=True)
    torch.cuda.synchronize()
    h2d = 2 * N_BYTES / (time.perf_counter() - t0) / GB
    t0 = time.perf_counter()
    for _ in range(2):
        out_host.copy_(d_in, non_blocking=True)
    torch.cuda.synchronize()
    d2h = 2 * N_BYTES / (time.perf_counter() - t0) / GB
    del buf_sets, out_hosts, graph
    return per_step, {"h2d": round(h2d, 1), "d2h": round(d2h, 1)}


def launcher_check():
    """The multi-rank plumbing without a GPU: a gloo process group over the
    ranks the launcher started, each rank's time 10 + 5 * rank ms, the
    max-over-ranks reduction and rank 0's report."""
    import torch
    import torch.distributed as dist
    rank, world, _ = dist_info()
    if world > 1:
        dist.init_process_group("gloo")
    mx = 10.0 + 5.0 * rank
    if world > 1:
        mx = reduce_max_ms(torch, mx, dist, torch.device("cpu"))
        dist.barrier()
    if rank == 0:
        print(json.dumps({"launcher_check": True, "world": world, "max_ms": mx,
                          "value": throughput(world, STEP_BYTES, 1, mx)}), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.case:
        run_case(args)
        return
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: run this same command under torch.distributed.run
        cmd = relaunch_command(sys.argv[1:], args.gpus, _free_port())
        raise SystemExit(subprocess.call(cmd))
    if args.launcher_check:
        launcher_check()
        return
    if args.impl == "reference":
        run_reference(args)
        return
    rank, world, local = dist_info()
    import numpy as np
    import torch
    import xor_swizzle_movement_gb300 as swz
    from xor_swizzle_movement_gb300 import inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    swz.lib()
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist

    peak, peak_kind = peaks()
    host = inputs.random_bytes(N_BYTES, seed=4)
    host_t = torch.from_numpy(host).pin_memory()
    src = host_t.to(dev)
    phys = torch.empty_like(src)
    back = torch.empty_like(src)
    stream = torch.cuda.current_stream()

    def step():
        swz.swz_relayout(phys, src, TILES, ROWS, COLS, ESIZE, B, M, S, 0)
        swz.swz_relayout(back, phys, TILES, ROWS, COLS, ESIZE, B, M, S, 1)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert torch.equal(back, src), "relayout round trip failed"

    gpu_id = None
    try:
        gpu_id = str(torch.cuda.get_device_properties(dev).uuid)
        if gpu_id and not gpu_id.startswith("GPU-"):
            gpu_id = "GPU-" + gpu_id
    except Exception:
        gpu_id = None
    clocks = ClockSampler(gpu_id)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    # one event pair around the K steps: an event between launches would keep
    # the next launch from starting under this one's last wave (programmatic
    # dependent launch); every buffer is larger than L2, so no flush
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    wall1 = time.perf_counter()
    wall = wall1 - wall0
    clk = clocks.stop(wall0, wall1)
    total_ms = e0.elapsed_time(e1)
    if pg:
        total_ms = reduce_max_ms(torch, total_ms, pg, dev)
    ms_per_step = total_ms / args.steps
    value = throughput(world, STEP_BYTES, args.steps, total_ms)

    # each direction on its own, 20 launches back to back (not part of the value)
    fwd_ms = back_to_back_ms(torch, lambda: swz.swz_relayout(phys, src, TILES, ROWS, COLS, ESIZE, B, M, S, 0),
                             reps=20)
    inv_ms = back_to_back_ms(torch, lambda: swz.swz_relayout(back, phys, TILES, ROWS, COLS, ESIZE, B, M, S, 1),
                             reps=20)

    # roofline of the relayout kernel: both launches of a step are that kernel
    # (Swizzle<5,2,5> is its own inverse), so its mean launch duration over the
    # timed region is the step time / 2
    avg_launch_s = ms_per_step / 2 * 1e-3
    achieved = LAUNCH_BYTES / avg_launch_s / GB
    src_hash = source_hash("swz_relayout.cu", "swz_common.cuh")
    traffic = committed_traffic(HEADLINE_KERNEL, src_hash)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 3), "traffic": traffic,
                "algorithmic_bytes_per_launch": LAUNCH_BYTES,
                "peak_kind": f"{peak_kind} HBM copy bandwidth", "kernel": "relayout_vec_kernel<1,1,false,false>",
                "mean_launch_ms": round(avg_launch_s * 1e3, 5),
                "back_to_back_ms": {"forward": round(fwd_ms, 5), "inverse": round(inv_ms, 5),
                                    "note": "20 launches of one direction, outside the timed region"}}

    # end to end through the C ABI on pinned host buffers (the headline e2e),
    # and the copy-engine pipeline of the same step for context
    e2e_s = e2e_host_abi(torch, swz, host_t, steps=16)
    ce_s, copy_rates = e2e_copy_engine(torch, swz, host_t, src)
    e2e = {"value": round(STEP_BYTES / e2e_s / GB, 1), "unit": "GB/s",
           "h2d_bytes_per_step": N_BYTES, "d2h_bytes_per_step": N_BYTES,
           "ms_per_step": round(e2e_s * 1e3, 4), "steps": 16,
           "how": "swz_relayout forward reading the pinned host input, inverse writing the pinned host "
                  "output (kernels on host memory over the host link); consecutive steps on two streams, "
                  "each forward paired with the previous step's inverse",
           "copy_engine_pipeline": {"value": round(STEP_BYTES / ce_s / GB, 1), "unit": "GB/s",
                                    "ms_per_step": round(ce_s * 1e3, 4),
                                    "how": "cudaMemcpyAsync chunks in and out over three streams around "
                                           "the two launches, 4 steps per CUDA graph"},
           "copy_GB/s": copy_rates}

    rows = None
    if not args.no_rows and rank == 0:
        del phys, back
        rows = measure_rows(torch, swz, dev, make_flush(torch, dev), peak)

    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": {"workload": WORKLOAD, "tiles": TILES, "rows": ROWS, "cols": COLS, "elem_bytes": ESIZE,
                       "swizzle_BMS": [B, M, S], "step": "forward launch + inverse launch",
                       "bytes_per_step": STEP_BYTES,
                       "l2": "inputs larger than L2 (three 1 GiB buffers against a 126 MB L2); no flush",
                       "parallelism": f"replicas x{world}"},
            "frac_of_hbm_peak": round(value / world / peak, 3),
            "roofline": roofline, "e2e": e2e, "gpu_launches": 2 * args.steps,
            "clocks": clk, "wall_s_timed_loop": round(wall, 3)}
    if rows is not None:
        line["rows"] = rows
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(host)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
