#!/usr/bin/env python
"""Benchmark: causal bf16 ring attention, forward + backward, N = 131072,
16 heads, d = 128, P = 32 virtual hosts, on one GB300 per process.

One step = ra_ring_fwd + ra_ring_bwd over the whole sequence (every row of
the hot path).  Inputs are seeded synthetic tensors resident in HBM (each of
Q, K, V, dO is 512 MiB, larger than L2, so no flush is needed between steps).
Prints one JSON line (rank 0).  With --impl reference the fp64 CPU oracle is
timed on a bounded sample of the same workload instead.

Multi-GPU: the workload does not exchange data between GPUs (the ring is
emulated inside one GPU), so N processes run N independent replicas; the
step time is the maximum over ranks and the value sums the work of all ranks.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal attention TFLOP/s fwd+bwd at 128K bf16 d=128; % of GB300 BF16 peak"
WORKLOAD = dict(B=1, N=131072, Hq=16, Hkv=16, d=128, P=32, causal=True, cid=3, dtype=torch.bfloat16,
                q_scale=1.0, v_outlier_frac=0.0, precise=False)
WORKLOAD_NAME = "bf16 causal ring attention fwd+bwd, B1 H16 N131072 d128, P32 virtual hosts of 4096"
WORKLOAD_OVERRIDDEN = False


def algo_flops(B, N, Hq, d, causal=True):
    """Causal-adjusted algorithmic flops: fwd 4*B*H*N^2*d/2 (two products of
    2*N*N*d over the visible half), bwd 2.5x fwd (five products, two of them
    shared with the forward)."""
    fwd = 4.0 * B * Hq * N * N * d / (2.0 if causal else 1.0)
    return fwd, 2.5 * fwd


def row_flops(i, d, causal=True, N=None):
    """Algorithmic flops of one query row in fwd+bwd: 14 * d * (keys seen)."""
    keys = (i + 1) if causal else N
    return 4.0 * d * keys * 3.5


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(burst=float(p["bf16_tflops"]), sustained=float(p["bf16_tflops_sustained"]),
                    hbm=float(p["hbm_gbs"]), source="measured (MEASURED_PEAKS.json)")
    except Exception:
        return dict(burst=1900.0, sustained=1700.0, hbm=6800.0, source="fallback")


def kernel_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, only if it was
    taken on the current kernel source (sha256 of the .cu file) and the
    workload is the one it was captured on."""
    import hashlib
    if WORKLOAD_OVERRIDDEN:
        return None
    src = {"tc_bwd": "ra_bwd_tc.cu", "tc_fwd": "ra_fwd_tc.cu"}[kernel]
    path = os.path.join(ROOT, "blockwise_exact_attention_ra_gb300", "csrc", src)
    sha = hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]
    table = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(table):
        return None
    for line in open(table):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel and parts[1] == sha:
            return float(parts[2])
    return None


class HostArena:
    """Page-locked host memory for the end-to-end leg: one anonymous mapping
    advised for transparent huge pages and registered with cudaHostRegister.
    On the Grace hosts of these GB300 machines buffers from cudaHostAlloc sometimes
    copy at ~20 GB/s once the host's memory has been through heavy use, while
    huge-page-backed registered memory kept 67-211 GB/s in every state tried;
    the two-stream pipeline hides copies at either rate.  Falls back to ordinary
    pinned tensors when the mapping or the registration is refused."""

    def __init__(self, nbytes):
        import ctypes
        import mmap
        self.kind = "cudaHostAlloc"
        self.buf = None
        self.off = 0
        align = 1 << 30
        try:
            m = mmap.mmap(-1, nbytes + align, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
            base = ctypes.addressof(ctypes.c_char.from_buffer(m))
            start = (base + align - 1) & ~(align - 1)
            libc = ctypes.CDLL("libc.so.6", use_errno=True)
            libc.madvise.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
            libc.madvise(start, nbytes, 14)  # MADV_HUGEPAGE
            t = torch.frombuffer(m, dtype=torch.uint8, count=nbytes, offset=start - base)
            t.fill_(0)
            if int(torch.cuda.cudart().cudaHostRegister(start, nbytes, 0)) != 0:
                raise RuntimeError("cudaHostRegister refused")
            self.map, self.buf, self.kind = m, t, "registered huge pages"
        except Exception:
            self.buf = None

    def tensor(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        if self.buf is None or self.off + n > self.buf.numel():
            return torch.empty(shape, dtype=dtype, pin_memory=True)
        t = self.buf[self.off:self.off + n].view(dtype).view(shape)
        self.off += (n + 255) & ~255
        return t


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.dev)], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def _parse(self, lines):
        sm, mx, reasons = [], [], set()
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return sm, mx, reasons

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.seek(0)
        sm, mx, reasons = self._parse(self.file)
        after = False
        if not sm:
            # a timed region shorter than nvidia-smi's start-up and first
            # interval leaves no sample: take one right after it, and say so
            try:
                out = subprocess.run(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                      "-i", str(self.dev)], capture_output=True, text=True, timeout=20).stdout
            except Exception:
                out = ""
            sm, mx, reasons = self._parse(out.splitlines())
            after = True
        if not sm:
            return None
        res = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
               "reasons": sorted(reasons)}
        if after:
            res["sampled_after_region"] = True
        return res


L2_BYTES = 129 * 2**20  # GB300 last-level cache


def l2_note(B, N, Hq, Hkv, d, es=2):
    """How the timed steps stand to L2: each input tensor's size (es bytes per element)."""
    q_mib = B * N * Hq * d * es / 2**20
    kv_mib = B * N * Hkv * d * es / 2**20
    sizes = (f"Q, K, V, dO {q_mib:.0f} MiB each" if Hq == Hkv else
             f"Q, dO {q_mib:.0f} MiB, K, V {kv_mib:.0f} MiB each")
    if min(q_mib, kv_mib) * 2**20 > L2_BYTES:
        return f"inputs larger than L2 ({sizes}); no flush"
    return f"inputs not larger than L2 ({sizes}); no flush, so timings include L2 reuse across steps"


def max_over_ranks(x, device):
    """Max of a per-rank float over all ranks (identity on one process)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world_size, flop_per_step_per_rank, ms_per_step):
    """Whole-job TFLOP/s: every rank runs one replica's step; the step takes
    the slowest rank's time."""
    return world_size * flop_per_step_per_rank / (ms_per_step * 1e-3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def cpu_oracle_sample(q, k, v, do, rows, causal, scale):
    """Run the oracle (fwd + bwd incl. dK/dV contributions) on `rows`; returns
    (seconds, algorithmic flops of those rows)."""
    import oracle
    heads = sorted({h for _, h, _ in rows})
    group = q.shape[2] // k.shape[2]   # query heads per key/value head
    hk = {}
    for h in heads:
        g = h // group
        hk[h] = tuple(t.float().cpu().numpy().astype(np.float64)
                      for t in (q[:, :, h:h + 1], k[:, :, g:g + 1], v[:, :, g:g + 1], do[:, :, h:h + 1]))
    t0 = time.perf_counter()
    for h in heads:
        qq, kk, vv, dd = hk[h]
        sel = [(b, 0, i) for b, hh, i in rows if hh == h]
        oracle.attention_rows(qq, kk, vv, sel, causal, scale, do=dd, want_kv_grads=True)
    dt = time.perf_counter() - t0
    N = q.shape[1]
    fl = sum(row_flops(i, q.shape[3], causal, N) for _, _, i in rows)
    return dt, fl


def oracle_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = [x.get("num_threads") for x in info if x.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def sample_rows(N, Hq, count, seed):
    g = torch.Generator().manual_seed(seed)
    h = int(torch.randint(Hq, (1,), generator=g))
    idx = torch.randint(N, (count,), generator=g)
    return [(0, h, int(i)) for i in idx]


def bench_config(ws):
    """The `config` object of the JSON line, the same for both arms."""
    W = WORKLOAD
    f32 = W["dtype"] == torch.float32
    return {"workload": WORKLOAD_NAME, "B": W["B"], "N": W["N"], "Hq": W["Hq"], "Hkv": W["Hkv"], "d": W["d"],
            "P": W["P"], "causal": W["causal"],
            "l2": l2_note(W["B"], W["N"], W["Hq"], W["Hkv"], W["d"], 4 if f32 else 2),
            "parallelism": "replicas" if ws > 1 else "single GPU"}


def run_reference(args, ws, rank):
    """Reference arm: the fp64 oracle on the host cores, bounded row samples."""
    if rank != 0:
        return
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    W = WORKLOAD
    q, k, v, do = make_tensors(W["B"], W["N"], W["Hq"], W["Hkv"], W["d"], W["dtype"], "cpu",
                               1000 + W["cid"], W["q_scale"], W["v_outlier_frac"], with_do=True)
    scale = W["d"] ** -0.5
    times, flops = [], []
    for s in range(args.warmup + args.steps):
        rows = sample_rows(W["N"], W["Hq"], min(args.ref_rows, W["N"]), 500 + s)
        dt, fl = cpu_oracle_sample(q, k, v, do, rows, W["causal"], scale)
        if s >= args.warmup:
            times.append(dt)
            flops.append(fl)
    value = sum(flops) / sum(times) / 1e12
    cores = oracle_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": bench_config(ws),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.ref_rows} seeded query rows of one head per step, fwd+bwd "
                                   f"(incl. their dK/dV contributions), fp64 numpy",
                         "extrapolated_full_step_s": sum(algo_flops(W["B"], W["N"], W["Hq"], W["d"], W["causal"]))
                         / (value * 1e12),
                         "extrapolation": "the workload's algorithmic flops at the sampled rows' rate"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_named_workload(ra, cid, dev, stream, steps, warmup, peaks):
    """One of the five named workloads through ra_ring_fwd (+ ra_ring_bwd when
    the workload has a backward), with its own seeded inputs, mask and
    numerics (workload 4: two-term fp16 P and dS), outputs in fp32; device
    time with CUDA events on the launching stream."""
    from blockwise_exact_attention_ra_gb300.inputs import WORKLOADS, make_config
    c = WORKLOADS[cid]
    B, N, Hq, Hkv, d, P = c["B"], c["N"], c["Hq"], c["Hkv"], c["d"], c["P"]
    causal, bwd, precise = c["causal"], c["bwd"], cid == 4
    scale = d ** -0.5
    q, k, v, do = make_config(cid, dev, with_do=bwd)
    o = torch.empty(B, N, Hq, d, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
    sh = ra.shape_of(q, k)
    wsf = torch.empty(max(16, ra.ra_ring_fwd_workspace_bytes(ra._dt(q), sh, P)), dtype=torch.uint8, device=dev)
    if bwd:
        dq = torch.empty(B, N, Hq, d, dtype=torch.float32, device=dev)
        dk = torch.empty(B, N, Hkv, d, dtype=torch.float32, device=dev)
        dv = torch.empty(B, N, Hkv, d, dtype=torch.float32, device=dev)
        wsb = torch.empty(max(16, ra.ra_ring_bwd_workspace_bytes(ra._dt(q), ra.RA_F32, sh, P)), dtype=torch.uint8,
                          device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3 * steps)]
    for s_ in range(warmup + steps):
        t = s_ - warmup
        if t >= 0:
            ev[3 * t].record(stream)
        ra.ra_ring_fwd(q, k, v, P, causal, scale, o, lse, wsf, stream, precise=precise)
        if t >= 0:
            ev[3 * t + 1].record(stream)
        if bwd:
            ra.ra_ring_bwd(q, k, v, o, do, lse, P, causal, scale, dq, dk, dv, wsb, stream, precise=precise)
        if t >= 0:
            ev[3 * t + 2].record(stream)
    torch.cuda.synchronize(dev)
    ra.ra_sync_status(stream)
    f_ms = sum(ev[3 * i].elapsed_time(ev[3 * i + 1]) for i in range(steps)) / steps
    b_ms = sum(ev[3 * i + 1].elapsed_time(ev[3 * i + 2]) for i in range(steps)) / steps
    ffl, bfl = algo_flops(B, N, Hq, d, causal)
    if not bwd:
        bfl = 0.0
    res = {"workload": c["name"] + (" (forward)" if not bwd else " (fwd+bwd)")
           + (", two-term fp16 P and dS" if precise else ""),
           "steps": steps, "warmup": warmup, "ms_per_step": f_ms + b_ms,
           "tflops": (ffl + bfl) / ((f_ms + b_ms) * 1e-3) / 1e12,
           "fwd_ms": f_ms, "fwd_tflops": ffl / (f_ms * 1e-3) / 1e12}
    if bwd:
        res.update(bwd_ms=b_ms, bwd_tflops=bfl / (b_ms * 1e-3) / 1e12)
    if c["dtype"] != torch.float32:
        res["frac_of_peak"] = res["tflops"] / peaks["sustained"]
    return res


def run_ours(args, ws, rank, local):
    import blockwise_exact_attention_ra_gb300 as ra
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    W = WORKLOAD
    B, N, Hq, Hkv, d, P = W["B"], W["N"], W["Hq"], W["Hkv"], W["d"], W["P"]
    causal, precise, f32 = W["causal"], W["precise"], W["dtype"] == torch.float32
    scale = d ** -0.5
    q, k, v, do = make_tensors(B, N, Hq, Hkv, d, W["dtype"], dev, 1000 + W["cid"] + 17 * rank, W["q_scale"],
                               W["v_outlier_frac"])
    o = torch.empty(B, N, Hq, d, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
    dq = torch.empty(B, N, Hq, d, dtype=torch.float32, device=dev)
    dk = torch.empty(B, N, Hkv, d, dtype=torch.float32, device=dev)
    dv = torch.empty(B, N, Hkv, d, dtype=torch.float32, device=dev)
    sh = ra.shape_of(q, k)
    wsf = torch.empty(max(16, ra.ra_ring_fwd_workspace_bytes(ra._dt(q), sh, P)), dtype=torch.uint8, device=dev)
    wsb = torch.empty(max(16, ra.ra_ring_bwd_workspace_bytes(ra._dt(q), ra.RA_F32, sh, P)),
                      dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        ra.ra_ring_fwd(q, k, v, P, causal, scale, o, lse, wsf, stream, precise=precise)
        if ev is not None:
            ev.record(stream)
        ra.ra_ring_bwd(q, k, v, o, do, lse, P, causal, scale, dq, dk, dv, wsb, stream, precise=precise)

    for _ in range(args.warmup):
        step()
    ra.ra_sync_status(stream)

    fwd_fl, bwd_fl = algo_flops(B, N, Hq, d, causal)
    n_ev = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    clocks = ClockSampler(local)
    launches0 = ra.ra_launch_count()
    ra.ra_kernel_timing(1)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        starts[s].record(stream)
        step(mids[s])
        ends[s].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if ws > 1:
        torch.distributed.barrier()
    ra.ra_sync_status(stream)
    launches = ra.ra_launch_count() - launches0
    total_ms = t_start.elapsed_time(t_end)
    fwd_ms = sum(s.elapsed_time(m) for s, m in zip(starts, mids)) / args.steps
    bwd_ms = sum(m.elapsed_time(e) for m, e in zip(mids, ends)) / args.steps
    kfwd, kbwd = (ra.RA_KERNEL_FWD_F32, ra.RA_KERNEL_BWD_F32) if f32 else (ra.RA_KERNEL_FWD_TC, ra.RA_KERNEL_BWD_TC)
    ktime = {kid: ra.ra_kernel_timing_read(kid) for kid in (kfwd, kbwd)}
    ra.ra_kernel_timing(0)

    ms_step = max_over_ranks(total_ms / args.steps, dev)
    value = job_value(ws, fwd_fl + bwd_fl, ms_step)
    peaks = load_peaks()

    # dominant kernel: the one with the larger share of device time
    fwd_k_ms, fwd_n = ktime[kfwd]
    bwd_k_ms, bwd_n = ktime[kbwd]
    kf, kb = ("f32_fwd", "f32_bwd") if f32 else ("tc_fwd", "tc_bwd")
    if f32:
        # fp32 CUDA-core kernels: bound by FMA issue; peak = SMs x 128 fp32
        # lanes x 2 flops x the highest SM clock seen
        mhz = (clk or {}).get("sm_max_mhz") or 2070.0
        peak = torch.cuda.get_device_properties(dev).multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12
        peak_source = f"derived: SMs x 128 fp32 FMA lanes x 2 flops x {mhz:.0f} MHz"
    else:
        peak = peaks["sustained"]
        peak_source = peaks["source"] + ", bf16 sustained (dense fp16 runs at the bf16 rate)"
    kern = {
        kf: {"avg_ms": fwd_k_ms / max(fwd_n, 1), "launches": fwd_n, "flop_per_launch": fwd_fl},
        kb: {"avg_ms": bwd_k_ms / max(bwd_n, 1), "launches": bwd_n, "flop_per_launch": bwd_fl},
    }
    for kk in kern.values():
        kk["tflops"] = kk["flop_per_launch"] / (kk["avg_ms"] * 1e-3) / 1e12
        kk["frac_of_peak"] = kk["tflops"] / peak
    dom = kb if bwd_k_ms >= fwd_k_ms else kf
    roof = {"bound": "alu" if f32 else "tensor", "kernel": dom, "achieved": kern[dom]["tflops"], "peak": peak,
            "unit": "TFLOP/s", "frac": kern[dom]["tflops"] / peak,
            "traffic": None if f32 else kernel_traffic(dom), "peak_source": peak_source}

    # the striped (load-balanced) causal layout on the same tensors: same
    # algorithmic work, every virtual host with an equal share
    striped = None
    if not args.no_striped:
        def step_striped(ev=None):
            ra.ra_ring_fwd(q, k, v, P, True, scale, o, lse, wsf, stream, striped=True)
            if ev is not None:
                ev.record(stream)
            ra.ra_ring_bwd(q, k, v, o, do, lse, P, True, scale, dq, dk, dv, wsb, stream, striped=True)
        for _ in range(args.warmup):
            step_striped()
        torch.cuda.synchronize(dev)
        sa = [torch.cuda.Event(enable_timing=True) for _ in range(3 * args.steps)]
        for s_ in range(args.steps):
            sa[3 * s_].record(stream)
            step_striped(sa[3 * s_ + 1])
            sa[3 * s_ + 2].record(stream)
        torch.cuda.synchronize(dev)
        ra.ra_sync_status(stream)
        f_ms = sum(sa[3 * i].elapsed_time(sa[3 * i + 1]) for i in range(args.steps)) / args.steps
        b_ms = sum(sa[3 * i + 1].elapsed_time(sa[3 * i + 2]) for i in range(args.steps)) / args.steps
        striped = {"layout": "striped rows (host i local row l = position l*P + i)",
                   "tflops": (fwd_fl + bwd_fl) / ((f_ms + b_ms) * 1e-3) / 1e12,
                   "fwd_tflops": fwd_fl / (f_ms * 1e-3) / 1e12, "bwd_tflops": bwd_fl / (b_ms * 1e-3) / 1e12}

    # variable per-host lengths (dynamic masking): the same tensors through the
    # varlen entry points, (a) with every host full, whose cost over the plain
    # ring is the price of the masking, and (b) with seeded ragged lengths in
    # [S/2, S], timed against the flops of causal attention over the valid tokens
    varlen = None
    if not args.no_varlen:
        S = N // P
        g = torch.Generator().manual_seed(4321 + rank)
        ragged = torch.randint(S // 2, S + 1, (P,), generator=g, dtype=torch.int32)

        def time_varlen(hl):
            def one(ev=None):
                ra.ra_ring_fwd_varlen(q, k, v, P, hl, True, scale, o, lse, wsf, stream)
                if ev is not None:
                    ev.record(stream)
                ra.ra_ring_bwd_varlen(q, k, v, o, do, lse, P, hl, True, scale, dq, dk, dv, wsb, stream)
            for _ in range(args.warmup):
                one()
            torch.cuda.synchronize(dev)
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(3 * args.steps)]
            for s_ in range(args.steps):
                evs[3 * s_].record(stream)
                one(evs[3 * s_ + 1])
                evs[3 * s_ + 2].record(stream)
            torch.cuda.synchronize(dev)
            ra.ra_sync_status(stream)
            f = sum(evs[3 * i].elapsed_time(evs[3 * i + 1]) for i in range(args.steps)) / args.steps
            b_ = sum(evs[3 * i + 1].elapsed_time(evs[3 * i + 2]) for i in range(args.steps)) / args.steps
            return f, b_

        full = torch.full((P,), S, dtype=torch.int32, device=dev)
        f_ms, b_ms = time_varlen(full)
        L = int(ragged.sum())
        rf_ms, rb_ms = time_varlen(ragged.to(dev))
        lf, lb = algo_flops(B, L, Hq, d)
        varlen = {"full_lengths": {"tflops": (fwd_fl + bwd_fl) / ((f_ms + b_ms) * 1e-3) / 1e12,
                                   "ms_per_step": f_ms + b_ms, "fwd_ms": f_ms, "bwd_ms": b_ms,
                                   "overhead_vs_plain": (f_ms + b_ms) / (fwd_ms + bwd_ms) - 1.0},
                  "ragged": {"host_len": "seeded uniform in [S/2, S] per host", "valid_tokens": L,
                             "ms_per_step": rf_ms + rb_ms, "fwd_ms": rf_ms, "bwd_ms": rb_ms,
                             "tflops_on_valid_tokens": (lf + lb) / ((rf_ms + rb_ms) * 1e-3) / 1e12}}

    # blockwise feed-forward layer at the same model width (d_model = Hq * d,
    # hidden 4 d_model, all B * N tokens, blocks of 16384 tokens): forward and
    # backward timed separately; algorithmic flops count the layer's products
    # (2 forward, 4 backward), not the backward's recomputation of h
    ffn = None
    if not args.no_ffn:
        from blockwise_exact_attention_ra_gb300.inputs import make_ffn
        T, dm = B * N, Hq * d
        dh, blk = 4 * dm, min(16384, B * N)
        fx, fw1, fw2, fdy = make_ffn(T, dm, dh, torch.bfloat16, dev, 777 + rank)
        fy = torch.empty(T, dm, dtype=torch.bfloat16, device=dev)
        fdx = torch.empty(T, dm, dtype=torch.bfloat16, device=dev)
        fdw1 = torch.empty(dh, dm, dtype=torch.float32, device=dev)
        fdw2 = torch.empty(dm, dh, dtype=torch.float32, device=dev)
        fws = torch.empty(ra.ra_ffn_workspace_bytes(ra.RA_BF16, T, dm, dh, blk, True), dtype=torch.uint8,
                          device=dev)
        for _ in range(args.warmup):
            ra.ra_ffn_fwd(fx, fw1, fw2, blk, fy, fws, stream)
            ra.ra_ffn_bwd(fx, fw1, fw2, fdy, blk, fdx, fdw1, fdw2, fws, stream)
        torch.cuda.synchronize(dev)
        fe = [torch.cuda.Event(enable_timing=True) for _ in range(3 * args.steps)]
        ra.ra_kernel_timing(1)
        for s_ in range(args.steps):
            fe[3 * s_].record(stream)
            ra.ra_ffn_fwd(fx, fw1, fw2, blk, fy, fws, stream)
            fe[3 * s_ + 1].record(stream)
            ra.ra_ffn_bwd(fx, fw1, fw2, fdy, blk, fdx, fdw1, fdw2, fws, stream)
            fe[3 * s_ + 2].record(stream)
        torch.cuda.synchronize(dev)
        gemm_ms, gemm_n = ra.ra_kernel_timing_read(ra.RA_KERNEL_GEMM_TC)
        ra.ra_kernel_timing(0)
        ra.ra_sync_status(stream)
        f_ms = sum(fe[3 * i].elapsed_time(fe[3 * i + 1]) for i in range(args.steps)) / args.steps
        b_ms = sum(fe[3 * i + 1].elapsed_time(fe[3 * i + 2]) for i in range(args.steps)) / args.steps
        unit = 2.0 * T * dm * dh   # one of the layer's products
        ffn = {"shape": {"tokens": T, "d_model": dm, "d_hidden": dh, "block": blk, "dtype": "bf16"},
               "fwd_ms": f_ms, "bwd_ms": b_ms,
               "fwd_tflops": 2 * unit / (f_ms * 1e-3) / 1e12, "bwd_tflops": 4 * unit / (b_ms * 1e-3) / 1e12,
               "bwd_executed_tflops": 5 * unit / (b_ms * 1e-3) / 1e12,
               "gemm_launches": gemm_n, "gemm_avg_tflops": 7 * args.steps * unit / (gemm_ms * 1e-3) / 1e12,
               "frac_of_peak_fwd": 2 * unit / (f_ms * 1e-3) / 1e12 / peaks["sustained"]}
        del fx, fw1, fw2, fdy, fy, fdx, fdw1, fdw2, fws

    # end to end through the public C-ABI call with host buffers: every step
    # uploads its q, k, v, dO from pinned host memory and downloads O, LSE, dQ,
    # dK, dV (bf16) to pinned host memory.  Steps alternate between two streams
    # and two workspaces so that one step's copies overlap the other's kernels.
    e2e = None
    if not args.no_e2e:
        qel, kvel = B * N * Hq * d, B * N * Hkv * d
        # inputs q, k, v, dO (bf16) and two output sets O, LSE (fp32), dQ, dK, dV (bf16)
        arena = HostArena(2 * (2 * qel + 2 * kvel) + 2 * (4 * qel + 4 * kvel + 4 * B * Hq * N) + 64 * 256)
        host_in = []
        for t in (q, k, v, do):
            h_ = arena.tensor(tuple(t.shape), t.dtype)
            h_.copy_(t)
            host_in.append(h_)
        host_out = [[arena.tensor((B, N, Hq, d), torch.bfloat16), arena.tensor((B, Hq, N), torch.float32),
                     arena.tensor((B, N, Hq, d), torch.bfloat16), arena.tensor((B, N, Hkv, d), torch.bfloat16),
                     arena.tensor((B, N, Hkv, d), torch.bfloat16)] for _ in range(2)]
        hws = ra.ra_ring_step_host_workspace_bytes(ra.RA_BF16, ra.RA_BF16, ra.RA_BF16, sh, P)
        wsh = [torch.empty(hws, dtype=torch.uint8, device=dev) for _ in range(2)]
        sts = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]

        def e2e_steps(n):
            for i in range(n):
                ra.ra_ring_step_host(*host_in, P, True, scale, *host_out[i % 2], wsh[i % 2], sts[i % 2])

        main = torch.cuda.current_stream(dev)
        for st_ in sts:
            st_.wait_stream(main)
        e2e_steps(max(1, args.warmup))
        for st_ in sts:
            main.wait_stream(st_)
        torch.cuda.synchronize(dev)
        if ws > 1:
            torch.distributed.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(main)
        for st_ in sts:
            st_.wait_event(a)
        e2e_steps(args.steps)
        for st_ in sts:
            main.wait_stream(st_)
        b.record(main)
        torch.cuda.synchronize(dev)
        ra.ra_sync_status(main)
        e_ms = max_over_ranks(a.elapsed_time(b) / args.steps, dev)
        h2d_bytes = sum(t.numel() * t.element_size() for t in host_in)
        d2h_bytes = sum(t.numel() * t.element_size() for t in host_out[0])
        # what sets the pace: the same steps again with the library's event
        # timing on, which brackets every copy group and every kernel on its own
        # stream (a separate pass, so the timed steps above carry no events)
        ra.ra_kernel_timing(1)
        e2e_steps(args.steps)
        for st_ in sts:
            main.wait_stream(st_)
        torch.cuda.synchronize(dev)
        part = {name: ra.ra_kernel_timing_read(kid)[0] / args.steps for name, kid in
                (("h2d", ra.RA_COPY_H2D), ("d2h", ra.RA_COPY_D2H), ("fwd", ra.RA_KERNEL_FWD_TC),
                 ("bwd", ra.RA_KERNEL_BWD_TC))}
        ra.ra_kernel_timing(0)
        kern_ms, copy_ms = part["fwd"] + part["bwd"], part["h2d"] + part["d2h"]
        e2e = {"value": job_value(ws, fwd_fl + bwd_fl, e_ms), "unit": "TFLOP/s",
               "ms_per_step": e_ms,
               "h2d_bytes_per_step": h2d_bytes,
               "d2h_bytes_per_step": d2h_bytes,
               "api": "ra_ring_step_host (host buffers, pinned), two streams alternating",
               "host_memory": arena.kind,
               "breakdown": {
                   "h2d_ms_per_step": part["h2d"], "d2h_ms_per_step": part["d2h"],
                   "h2d_gbs": h2d_bytes / (part["h2d"] * 1e-3) / 1e9 if part["h2d"] > 0 else None,
                   "d2h_gbs": d2h_bytes / (part["d2h"] * 1e-3) / 1e9 if part["d2h"] > 0 else None,
                   "kernel_ms_per_step": kern_ms, "copy_ms_per_step": copy_ms,
                   # kernels set the pace while a step takes no longer than its
                   # kernels (within 5%); beyond that the copies are not hidden
                   "bound_by": "kernels" if e_ms <= 1.05 * kern_ms else "copies",
                   "how": "CUDA events around each copy group and each attention kernel on its own stream, "
                          "a second pass of the same steps"}}
        del wsh

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        n_rows = min(args.cpu_rows, N)
        rows = sample_rows(N, Hq, n_rows, 4242)
        dt, fl = cpu_oracle_sample(q, k, v, do, rows, causal, scale)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle_threads(), "kind": "oracle",
               "extrapolated_full_step_s": (fwd_fl + bwd_fl) / (fl / dt),
               "extrapolation": "the workload's algorithmic flops at the sampled rows' rate",
               "sample": f"{n_rows} seeded query rows of one head, fwd+bwd incl. their dK/dV "
                         f"contributions, fp64 numpy; {dt:.1f} s"}

    # the other named workloads, each with its own inputs, mask and numerics,
    # timed the same way with a few steps (1M tokens: one step of ~30 s)
    others = None
    if ws == 1 and not args.no_workloads and not WORKLOAD_OVERRIDDEN:
        del q, k, v, do, o, lse, dq, dk, dv, wsf, wsb
        torch.cuda.empty_cache()
        others = {}
        for cid, (st_, wu_) in {1: (10, 3), 2: (5, 3), 4: (2, 1), 5: (1, 1)}.items():
            try:
                others[str(cid)] = time_named_workload(ra, cid, dev, stream, st_, wu_, peaks)
            except Exception as exc:  # one workload's failure must not lose the line
                others[str(cid)] = {"error": f"{type(exc).__name__}: {exc}"[:300]}
            torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32" if f32 else "bf16", "data": "synthetic",
            "config": bench_config(ws),
            "pct_of_peak": value / ws / peak,
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "fwd_tflops": fwd_fl / (fwd_ms * 1e-3) / 1e12, "bwd_tflops": bwd_fl / (bwd_ms * 1e-3) / 1e12,
            "kernels": kern, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "striped": striped, "varlen": varlen, "ffn": ffn,
            "other_workloads": others,
            "gpu_launches": launches, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-striped", action="store_true", help="skip the striped-layout measurement")
    ap.add_argument("--no-varlen", action="store_true", help="skip the variable-length measurement")
    ap.add_argument("--no-ffn", action="store_true", help="skip the blockwise feed-forward measurement")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other named workloads (1, 2, 4, 5; the 1M-token one holds ~165 GB for ~1 min)")
    ap.add_argument("--cpu-rows", type=int, default=3072)
    ap.add_argument("--ref-rows", type=int, default=1024)
    ap.add_argument("--config", type=int, choices=[1, 2, 3, 4, 5], default=None,
                    help="one of the five named workloads (default: 3, the metric's); 4 runs with the "
                         "two-term fp16 P and dS its outlier inputs need; the striped, variable-length, "
                         "feed-forward and end-to-end legs belong to workload 3 and are skipped for the others")
    ap.add_argument("--N", type=int, default=None, help="override N (profiling on a smaller case)")
    ap.add_argument("--heads", type=int, default=None, help="override the (query) head count")
    ap.add_argument("--hkv", type=int, default=None, help="override the key/value head count (GQA)")
    ap.add_argument("--P", type=int, default=None, help="override the number of virtual hosts")
    args = ap.parse_args()
    global WORKLOAD_NAME, WORKLOAD_OVERRIDDEN
    if args.config is not None:
        from blockwise_exact_attention_ra_gb300.inputs import WORKLOADS
        c = WORKLOADS[args.config]
        WORKLOAD.update(B=c["B"], N=c["N"], Hq=c["Hq"], Hkv=c["Hkv"], d=c["d"], P=c["P"], causal=c["causal"],
                        cid=args.config, dtype=c["dtype"], q_scale=c["q_scale"],
                        v_outlier_frac=c["v_outlier_frac"], precise=args.config == 4)
        if args.config != 3:
            WORKLOAD_NAME = (f"workload {args.config}: {c['name']} fwd+bwd, virtual hosts of {c['N'] // c['P']}"
                             + (", two-term fp16 P and dS" if args.config == 4 else ""))
            WORKLOAD_OVERRIDDEN = True
            args.no_striped = args.no_varlen = args.no_ffn = args.no_e2e = True
    if args.N or args.heads or args.hkv or args.P:
        WORKLOAD["N"] = args.N or WORKLOAD["N"]
        WORKLOAD["Hq"] = WORKLOAD["Hkv"] = args.heads or WORKLOAD["Hq"]
        WORKLOAD["Hkv"] = args.hkv or WORKLOAD["Hkv"]
        WORKLOAD["P"] = args.P or WORKLOAD["P"]
        W = WORKLOAD
        heads = f"H{W['Hq']}" if W["Hq"] == W["Hkv"] else f"Hq{W['Hq']} Hkv{W['Hkv']}"
        WORKLOAD_NAME = (f"bf16 causal ring attention fwd+bwd, B1 {heads} N{W['N']} d128, "
                         f"P{W['P']} virtual hosts of {W['N'] // W['P']} (override of the bench workload)")
        WORKLOAD_OVERRIDDEN = True
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)


if __name__ == "__main__":
    main()
