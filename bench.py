"""Benchmark of the convrot INT8 linear on one GB300 (or N independent replicas).

A step is one pass of the whole hot path on the DiT attention-projection
workload: X fp32 [4608, 3072] (1% outliers x40) is packed once with G = 256
(rotation, row absmax, quantization) and one grouped tensor-core GEMM computes
the three [3072, 3072] linears (Q, K, V) with the fused reconstruction.
Weights are prepared offline (untimed). The step runs as the library's two
stream-ordered calls (pack, grouped GEMM) so that CUDA events also time the
dominant GEMM kernel alone; the e2e leg times the one-call convrot_linear API
with host buffers, host<->device copies included.

Metric: INT8-equivalent tera-operations per second (2*M*N*K summed over the
linears, per step time). L2 is flushed (256 MiB write) before every timed
step. Also reported: the pack-only sweep (X fp32 [4096, 3072], every G) in
GB/s, the roofline of the GEMM kernel, SM clocks sampled during the timed
region, and the CPU oracle timed on a bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from int8_hadamard_rotated_gb300 import workloads  # noqa: E402

METRIC = "convrot INT8 linear TOPS (% INT8 TC peak); pack GB/s (% HBM peak)"
UNIT = "TOPS"
WORKLOAD = "dit_qkv"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def config_dict(w, n_gpus):
    return {
        "workload": f"{w.name}: X fp32 [{w.M},{w.K}] G={w.G} -> {len(w.Ns)} linears "
                    f"[{w.Ns[0]},{w.K}] sharing one pack (grouped GEMM)",
        "M": w.M, "K": w.K, "N": list(w.Ns), "G": w.G, "x_dtype": w.x_dtype,
        "l2": "flushed before every timed step (256 MiB write)",
        "parallelism": "replicas" if n_gpus > 1 else "single",
    }


def data_desc(w):
    return (f"synthetic: seeded PCG64({w.seed}); X ~ N(0,1) with {w.outlier_frac:.0%} "
            f"element outliers x{w.outlier_mult:g}; W ~ N(0,{w.w_std}); b ~ N(0,{w.b_std})")


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ---------------------------------------------------------------------------

def oracle_sample_seconds(case, w, rows, prepared):
    import oracle
    X = case.X[:rows]
    t0 = time.perf_counter()
    Qx, s_x = oracle.pack(X, w.G)
    for (Qw, s_w), b in zip(prepared, case.bs):
        oracle.reconstruct(oracle.gemm_s32(Qx, Qw), s_x, s_w, b)
    return time.perf_counter() - t0


def cpu_baseline(case, w, budget_s=10.0):
    """Time the oracle as it stands on a sample of the workload's rows, growing
    the sample until it takes about `budget_s` (or covers all rows)."""
    import oracle
    prepared = [oracle.prepare_weight(W, w.G) for W in case.Ws]
    rows = 64
    t = oracle_sample_seconds(case, w, rows, prepared)
    while t < budget_s / 4 and rows < w.M:
        rows = min(w.M, rows * 4)
        t = oracle_sample_seconds(case, w, rows, prepared)
    ops = 2.0 * rows * sum(w.Ns) * w.K
    try:
        cores = len(os.sched_getaffinity(0))
    except Exception:
        cores = os.cpu_count() or 1
    return {"value": ops / t / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"oracle pack + {len(w.Ns)} int32 GEMMs + reconstruction on the first "
                      f"{rows} of {w.M} rows ({t:.2f} s; numpy/BLAS on all host cores)"}


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def gemm_traffic(kernel_src_hash):
    """DRAM bytes per GEMM launch from the committed ncu summary, if it was
    taken on the current kernel source (its `traffic_json:` line)."""
    p = os.path.join(ROOT, "profiles", "gemm_dit_qkv.md")
    try:
        with open(p) as f:
            for line in f:
                if line.startswith("traffic_json:"):
                    d = json.loads(line.split(":", 1)[1])
                    if d.get("gemm_src_sha256") == kernel_src_hash:
                        return d.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


GEMM_SOURCES = ("gemm.cu", "gemm_common.cuh", "common.cuh")


def source_hash():
    """SHA-256 of the GEMM kernel's sources (gemm.cu, gemm_common.cuh and
    common.cuh, concatenated in that order)."""
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "int8_hadamard_rotated_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def bench_lib():
    """The benchmark's own measurement kernels (libconvrot_bench.so, built
    beside libconvrot.so): a size-matched streaming copy and a probe of the
    legacy s8 tensor instruction. Neither is part of the library."""
    import ctypes
    from int8_hadamard_rotated_gb300 import build
    L = ctypes.CDLL(build.BENCH_LIB_PATH)
    L.bench_probe_int8_mma_rate.restype = ctypes.c_int
    L.bench_probe_int8_mma_rate.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
    L.bench_copy_ceiling.restype = ctypes.c_int
    L.bench_copy_ceiling.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    return L


def int8_mma_rate(iters=20000):
    """TOPS of the legacy mma.sync s8 instruction on the current device."""
    import ctypes
    out = ctypes.c_double(0.0)
    st = bench_lib().bench_probe_int8_mma_rate(int(iters), ctypes.byref(out))
    if st != 0:
        raise RuntimeError(f"bench_probe_int8_mma_rate failed: {st}")
    return float(out.value)


def copy_ceiling_us(X, out_bytes, flush, stream, reps=20, ctas_per_sm=8):
    """Mean time of the size-matched copy of X fp32 [M, K] -> out_bytes per
    element + one fp32 word per row, L2 flushed before each launch like the
    pack it is the ceiling for."""
    import torch
    M, K = X.shape
    out = torch.empty((M, K * out_bytes), dtype=torch.uint8, device=X.device)
    sc = torch.empty((M,), dtype=torch.float32, device=X.device)
    L = bench_lib()

    def run():
        st = L.bench_copy_ceiling(X.data_ptr(), M, K, out_bytes, out.data_ptr(), sc.data_ptr(), ctas_per_sm,
                                  stream.cuda_stream)
        if st != 0:
            raise RuntimeError(f"bench_copy_ceiling failed: {st}")
    for _ in range(3):
        run()
    ev = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) for a, b in ev])) * 1e3


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value over the ranks (the slowest rank's time); x itself
    with one rank. Every rank must call it (a collective)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tops(ops_per_rank: float, ms_per_step: float, world: int) -> float:
    """Whole-job throughput in TOPS: the units every rank processed in a step
    (the same on each: weak scaling) over the slowest rank's step time."""
    return world * ops_per_rank / (ms_per_step * 1e-3) / 1e12


def run_gpu(args, rank, world, local_rank):
    import torch
    from int8_hadamard_rotated_gb300 import build, ops

    build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    w = workloads.get(WORKLOAD)
    case = workloads.make_case(w)
    peaks, peak_kind = load_peaks()

    # resident inputs and offline weight preparation (untimed)
    X = torch.from_numpy(case.X).to(dev)
    q16s, scales, biases, plans = [], [], [], []
    for W, b in zip(case.Ws, case.bs):
        q8, s_w, q16 = ops.convrot_prepare_weight(torch.from_numpy(W).to(dev), w.G)
        q16s.append(q16)
        scales.append(s_w)
        biases.append(torch.from_numpy(b).to(dev))
        plans.append(ops.convrot_weight_chunks(q8))   # exact-chunk plan, also offline
    Ys = [torch.empty((w.M, n), dtype=torch.float32, device=dev) for n in w.Ns]
    Qx16 = torch.empty((w.M, w.K), dtype=torch.float16, device=dev)
    s_x = torch.empty((w.M,), dtype=torch.float32, device=dev)
    wdesc = ops.make_weights(q16s, scales, biases, Ys, plans)
    sync_ws = torch.empty((ops.GEMM_SYNC_BYTES,), dtype=torch.uint8, device=dev)  # GEMM hand-over words
    L = ops.lib()
    sp = stream.cuda_stream
    flush = torch.empty((L2_FLUSH_BYTES,), dtype=torch.uint8, device=dev)

    def step():
        st = L.convrot_pack_activations_f16(X.data_ptr(), ops.F32, w.M, w.K, w.G,
                                            Qx16.data_ptr(), s_x.data_ptr(), sp)
        if st:
            raise ops.ConvrotError(st, "pack")
        return st

    def gemm():
        st = L.convrot_linear_packed(Qx16.data_ptr(), s_x.data_ptr(), w.M, w.K, wdesc, len(q16s),
                                     sync_ws.data_ptr(), ops.GEMM_SYNC_BYTES, sp)
        if st:
            raise ops.ConvrotError(st, "gemm")

    for _ in range(args.warmup):
        flush.zero_()
        step()
        gemm()
    torch.cuda.synchronize()

    # The step is timed as a whole (events only around it, so the GEMM can be
    # launched as a programmatic dependent of the pack); the two kernels are
    # then timed alone on the same stream for the roofline and pack figures.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for k in range(args.steps):
        flush.zero_()
        ev[k][0].record(stream)
        step()
        gemm()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    status = ops.convrot_device_status()
    if status != ops.OK:
        raise ops.ConvrotError(status, "device status")
    step_ms = np.array([e[0].elapsed_time(e[1]) for e in ev])

    def time_alone(fn, reps):
        evs = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        return np.array([a.elapsed_time(b) for a, b in evs])

    reps_alone = max(10, min(args.steps, 200))
    step()
    gemm_ms = time_alone(gemm, reps_alone)
    pack_ms = time_alone(step, reps_alone)
    ms_step = max_over_ranks(float(step_ms.mean()), world, dev)
    ops_step = float(w.gemm_ops)
    value = job_tops(ops_step, ms_step, world)

    gemm_tflops = ops_step / (gemm_ms.mean() * 1e-3) / 1e12
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # the pack's algorithmic bytes: fp32 X in, one int8 code per element and
    # one fp32 scale per row out; the step's pack writes its codes as
    # binary16 (the GEMM's operand), so it moves M*K more bytes than that
    fused_pack_bytes = w.M * w.K * 4 + w.M * w.K + w.M * 4
    fused_pack_moved = w.M * w.K * 4 + w.M * w.K * 2 + w.M * 4
    roofline = {
        "bound": "tensor", "kernel": "convrot_gemm_kernel (tcgen05 kind::f16, exact int32)",
        "achieved": round(gemm_tflops, 2), "peak": peak_tf, "unit": "TFLOP/s",
        "frac": round(gemm_tflops / peak_tf, 4),
        "peak_kind": f"{peak_kind} bf16 dense burst (fp16 nominal = bf16 nominal)",
        "ops_per_launch": int(ops_step),
        "traffic": gemm_traffic(source_hash()),
    }

    # ---- e2e: one convrot_linear_host call with host buffers ----------------
    # X and the outputs in pinned host memory; the library copies row chunks
    # in and out on two copy streams while it packs and multiplies.
    X_host = torch.from_numpy(case.X).pin_memory()
    Y_host = [torch.empty((w.M, n), dtype=torch.float32).pin_memory() for n in w.Ns]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    n_total = sum(w.Ns)
    ws = torch.empty((ops.convrot_linear_host_workspace_size(w.M, w.K, ops.F32, n_total, 0),),
                     dtype=torch.uint8, device=dev)
    wdesc2 = ops.make_weights(q16s, scales, biases, Y_host, plans)
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        st = L.convrot_linear_host(X_host.data_ptr(), ops.F32, w.M, w.K, w.G, wdesc2, len(q16s), 0,
                                   ws.data_ptr(), ws.numel(), sp, s_in.cuda_stream, s_out.cuda_stream)
        if st:
            raise ops.ConvrotError(st, "convrot_linear_host")

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    e2e = {"value": job_tops(ops_step, e2e_ms, world), "unit": UNIT,
           "h2d_bytes_per_step": int(X_host.numel() * 4),
           "d2h_bytes_per_step": int(sum(y.numel() * 4 for y in Y_host)),
           "ms_per_step": e2e_ms,
           "api": "convrot_linear_host (one call; pinned host X and Y, chunked copies overlapped with compute)"}
    # check parity of the e2e output against the timed path's output
    step(); gemm()
    torch.cuda.synchronize()
    Yt = [y.cpu() for y in Ys]

    # ---- pack-only sweep (X fp32 [4096, 3072], every G) -------------------
    pw = workloads.get("pack_sweep")
    pcase = workloads.make_case(pw)
    Xp = torch.from_numpy(pcase.X).to(dev)
    Qp = torch.empty((pw.M, pw.K), dtype=torch.int8, device=dev)
    sp_x = torch.empty((pw.M,), dtype=torch.float32, device=dev)
    pack_bytes = pw.M * pw.K * 4 + pw.M * pw.K + pw.M * 4
    sweep = {}
    reps = 20
    for G in pw.groups:
        for _ in range(3):
            L.convrot_pack_activations(Xp.data_ptr(), ops.F32, pw.M, pw.K, G, Qp.data_ptr(), sp_x.data_ptr(), sp)
        times = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            st = L.convrot_pack_activations(Xp.data_ptr(), ops.F32, pw.M, pw.K, G, Qp.data_ptr(),
                                            sp_x.data_ptr(), sp)
            b.record(stream)
            if st:
                raise ops.ConvrotError(st, "pack sweep")
            times.append((a, b))
        torch.cuda.synchronize()
        ms = float(np.mean([a.elapsed_time(b) for a, b in times]))
        gbs = pack_bytes / (ms * 1e-3) / 1e9
        sweep[str(G)] = {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4)}
    # the same packs back to back over rotating buffers (together more than
    # 4x L2, so no launch finds its input in L2): kernel throughput without
    # the launch latency that an isolated launch after a flush includes
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (126 << 20))
    nbuf = max(2, -(-4 * l2 // (pw.M * pw.K * 4)))
    Xr = [Xp.clone() for _ in range(nbuf)]
    Qr = [torch.empty_like(Qp) for _ in range(nbuf)]
    sr = [torch.empty_like(sp_x) for _ in range(nbuf)]
    passes = 3
    for G in pw.groups:
        def run_all():
            for i in range(nbuf):
                st = L.convrot_pack_activations(Xr[i].data_ptr(), ops.F32, pw.M, pw.K, G, Qr[i].data_ptr(),
                                                sr[i].data_ptr(), sp)
                if st:
                    raise ops.ConvrotError(st, "pack sweep")
        run_all()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(passes):
            run_all()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / (passes * nbuf)
        gbs = pack_bytes / (ms * 1e-3) / 1e9
        sweep[str(G)]["back_to_back"] = {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
                                         "buffers": nbuf}
    # the size-matched copy over the same rotating buffers: the back-to-back ceiling
    bl = bench_lib()

    def copy_all():
        for i in range(nbuf):
            st = bl.bench_copy_ceiling(Xr[i].data_ptr(), pw.M, pw.K, 1, Qr[i].data_ptr(), sr[i].data_ptr(), 8, sp)
            if st != 0:
                raise RuntimeError(f"bench_copy_ceiling failed: {st}")
    copy_all()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(passes):
        copy_all()
    b.record(stream)
    torch.cuda.synchronize()
    cc_b2b = a.elapsed_time(b) / (passes * nbuf) * 1e3  # us
    del Xr, Qr, sr
    # long rows: the MLP pair's repack input, X fp32 [4608, 12288] -> binary16 codes
    ML, KL = 4608, 12288
    gen = torch.Generator(device=dev)
    gen.manual_seed(4)
    Xl = torch.randn((ML, KL), generator=gen, device=dev)
    Ql = torch.empty((ML, KL), dtype=torch.float16, device=dev)
    sl = torch.empty((ML,), dtype=torch.float32, device=dev)
    large_bytes = ML * KL * 4 + ML * KL * 2 + ML * 4
    for _ in range(3):
        L.convrot_pack_activations_f16(Xl.data_ptr(), ops.F32, ML, KL, 256, Ql.data_ptr(), sl.data_ptr(), sp)
    times = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        st = L.convrot_pack_activations_f16(Xl.data_ptr(), ops.F32, ML, KL, 256, Ql.data_ptr(), sl.data_ptr(), sp)
        b.record(stream)
        if st:
            raise ops.ConvrotError(st, "pack long rows")
        times.append((a, b))
    torch.cuda.synchronize()
    ms = float(np.mean([a.elapsed_time(b) for a, b in times]))
    gbs = large_bytes / (ms * 1e-3) / 1e9
    large = {"workload": f"X fp32 [{ML},{KL}] ~N(0,1) seed 4, G=256 -> binary16 codes + s",
             "bytes": large_bytes, "us": round(ms * 1e3, 2), "GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
             "copy_ceiling_us": round(copy_ceiling_us(Xl, 2, flush, stream), 2),
             "copy_ceiling_note": "size-matched copy (fp32 in, 2 B per element + 4 B per row out), same flush protocol"}
    del Xl, Ql, sl

    # ---- the DiT MLP pair on the device (convrot_mlp) ---------------------
    mlp = mlp_leg(dev, flush, peak_tf, hbm, peak_kind, with_cpu=(world == 1 and rank == 0 and not args.no_cpu_baseline))

    nxt = next_rows_legs(X, w, dev, flush, hbm, q16s, scales, biases, plans, ops_step)

    library = library_gemm_same_shape(w, dev, flush, float(gemm_ms.mean() * 1e3)) if args.library_gemm else None
    # context for "% INT8 TC peak": the legacy 8-bit integer tensor instruction's
    # rate on this GPU (tcgen05 has no 8-bit integer kind here)
    int8_rate = int8_mma_rate(20000)
    small = small_configs_in_graph(dev) if args.small_configs else None

    # the size-matched copies: the same bytes as the packs, no arithmetic
    cc_sweep = copy_ceiling_us(Xp, 1, flush, stream)
    cc_step = copy_ceiling_us(X, 2, flush, stream)
    pack_us = float(pack_ms.mean()) * 1e3
    pack = {
        "workload": f"pack_sweep: X fp32 [{pw.M},{pw.K}] 0.5% channel outliers x30 -> int8 + s",
        "bytes_per_launch": pack_bytes, "bound": "hbm", "peak": hbm, "unit": "GB/s",
        "peak_kind": f"{peak_kind} HBM copy", "by_group": sweep,
        "by_group_note": "us/GB/s/frac: isolated launches, L2 flushed before each (launch latency included); "
                         "back_to_back: consecutive launches over rotating buffers larger than 4x L2",
        "copy_ceiling": {"what": "size-matched streaming copy (fp32 in, 1 B per element + 4 B per row out), "
                                 "same flush protocol, no pack arithmetic",
                         "us": round(cc_sweep, 2), "GB/s": round(pack_bytes / (cc_sweep * 1e-6) / 1e9, 1),
                         "frac": round(pack_bytes / (cc_sweep * 1e-6) / 1e9 / hbm, 4),
                         "back_to_back_us": round(cc_b2b, 2),
                         "back_to_back_frac": round(pack_bytes / (cc_b2b * 1e-6) / 1e9 / hbm, 4)},
        "fused_step_pack": {"us": round(pack_us, 2),
                            "bytes": fused_pack_bytes,
                            "bytes_note": "algorithmic: fp32 X in, int8 codes + fp32 row scales out",
                            "GB/s": round(fused_pack_bytes / (pack_us * 1e-6) / 1e9, 1),
                            "frac": round(fused_pack_bytes / (pack_us * 1e-6) / 1e9 / hbm, 4),
                            "bytes_moved": fused_pack_moved,
                            "moved_note": "the codes are written as binary16, the GEMM's operand",
                            "frac_moved": round(fused_pack_moved / (pack_us * 1e-6) / 1e9 / hbm, 4),
                            "copy_ceiling_us": round(cc_step, 2),
                            "copy_ceiling_note": "size-matched copy of the moved bytes (fp32 in, 2 B per "
                                                 "element + 4 B per row out), same flush protocol",
                            "frac_of_copy_ceiling": round(cc_step / pack_us, 4)},
        "long_rows": large,
    }

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8", "data": data_desc(w), "config": config_dict(w, world),
        "roofline": roofline, "pack": pack, "mlp_chain": mlp, "next_rows": nxt, "e2e": e2e,
        "gpu_launches": 2 * args.steps,  # pack + grouped GEMM per timed step
        "clocks": clocks,
        "timing": {"step_ms_median": float(np.median(step_ms)), "pack_us_mean_alone": float(pack_ms.mean() * 1e3),
                   "gemm_us_mean_alone": float(gemm_ms.mean() * 1e3), "wall_s_timed_loop": wall},
        "e2e_parity_max_abs_diff": float(max((a - b).abs().max().item() for a, b in zip(Yt, Y_host))),
    }
    result["int8_mma_sync_probe"] = {
        "TOPS": round(int8_rate, 1),
        "what": "register-only mma.sync m16n8k32 s8 x s8 -> s32 on every SM (the only 8-bit integer tensor "
                "instruction on sm_103a)",
        "gemm_achieved_over_it": round(gemm_tflops / int8_rate, 3)}
    if library is not None:
        result["library_gemm_same_shape"] = library
    if small is not None:
        result["small_configs_in_graph"] = small
    return result, case, w


def mlp_leg(dev, flush, peak_tf, hbm, peak_kind, with_cpu=True, reps=10):
    """The DiT MLP pair (X fp32 [4608, 3072] -> up [12288, 3072] -> GELU ->
    down [3072, 12288], G = 256) as a leg of its own: the whole convrot_mlp
    call, its four launches timed alone (the pack, the up GEMM with GELU in
    its epilogue, the repack of H, the down GEMM; and the other placement of
    GELU, a plain up GEMM and the repack with GELU), the rooflines of the two
    GEMMs (tensor) and of the repack (HBM, on the algorithmic bytes: fp32 H
    in, int8 codes and row scales out), the call end to end with host
    buffers, the split-SwiGLU pair (gate and up [12288, 3072] sharing the
    pack), and the oracle chain on a row sample of the host cores. L2 is
    flushed before every timed launch; CUDA events on the launching stream."""
    import torch
    from int8_hadamard_rotated_gb300 import ops
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    L = ops.lib()
    mw = workloads.get("dit_mlp")
    mcase = workloads.make_case(mw)
    M, K, N_up, N_down, G = mw.M, mw.K, mw.Ns[0], mw.Ns[1], mw.G
    Xm = torch.from_numpy(mcase.X).to(dev)
    mlp_w = []
    for W, b in zip(mcase.Ws, mcase.bs):
        q8, s_w, q16 = ops.convrot_prepare_weight(torch.from_numpy(W).to(dev), G)
        mlp_w.append((q16, s_w, torch.from_numpy(b).to(dev), ops.convrot_weight_chunks(q8)))
        del q8
    Ym = torch.empty((M, N_down), dtype=torch.float32, device=dev)
    wsm = torch.empty((ops.convrot_mlp_workspace_size(M, K, N_up),), dtype=torch.uint8, device=dev)

    def timed(fn, n=reps):
        for _ in range(3):
            fn()
        ev = []
        for _ in range(n):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            ev.append((a, b))
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in ev])) * 1e3  # us

    chain = lambda: ops.convrot_mlp(Xm, G, mlp_w[0], ops.ACT_GELU, G, mlp_w[1], Y=Ym, workspace=wsm, stream=stream)
    t_chain = timed(chain)
    ops_up = 2.0 * M * N_up * K
    ops_down = 2.0 * M * N_down * N_up

    # the four launches alone, on the same buffers
    Qx = torch.empty((M, K), dtype=torch.float16, device=dev)
    sx = torch.empty((M,), dtype=torch.float32, device=dev)
    H = torch.empty((M, N_up), dtype=torch.float32, device=dev)
    Qh = torch.empty((M, N_up), dtype=torch.float16, device=dev)
    sh = torch.empty((M,), dtype=torch.float32, device=dev)
    sync_ws = torch.zeros((ops.GEMM_SYNC_BYTES,), dtype=torch.uint8, device=dev)
    wup = ops.make_weights([mlp_w[0][0]], [mlp_w[0][1]], [mlp_w[0][2]], [H], [mlp_w[0][3]])
    wdn = ops.make_weights([mlp_w[1][0]], [mlp_w[1][1]], [mlp_w[1][2]], [Ym], [mlp_w[1][3]])

    def chk(st, what):
        if st:
            raise ops.ConvrotError(st, what)
    t_pack = timed(lambda: chk(L.convrot_pack_activations_f16(Xm.data_ptr(), ops.F32, M, K, G, Qx.data_ptr(),
                                                               sx.data_ptr(), sp), "pack"))
    t_up = timed(lambda: chk(L.convrot_linear_packed_act(Qx.data_ptr(), sx.data_ptr(), M, K, wup, 1, ops.ACT_GELU,
                                                         sync_ws.data_ptr(), ops.GEMM_SYNC_BYTES, sp), "up GEMM + GELU"))
    t_repack = timed(lambda: chk(L.convrot_pack_activations_f16(H.data_ptr(), ops.F32, M, N_up, G, Qh.data_ptr(),
                                                                 sh.data_ptr(), sp), "repack"))
    # the other placement of GELU: in the repack (convrot_pack_gelu_f16), after a plain up GEMM
    t_up_plain = timed(lambda: chk(L.convrot_linear_packed(Qx.data_ptr(), sx.data_ptr(), M, K, wup, 1,
                                                           sync_ws.data_ptr(), ops.GEMM_SYNC_BYTES, sp), "up GEMM"))
    t_gelu_repack = timed(lambda: chk(L.convrot_pack_gelu_f16(H.data_ptr(), M, N_up, G, Qh.data_ptr(), sh.data_ptr(),
                                                              sp), "GELU repack"))
    t_down = timed(lambda: chk(L.convrot_linear_packed(Qh.data_ptr(), sh.data_ptr(), M, N_up, wdn, 1,
                                                       sync_ws.data_ptr(), ops.GEMM_SYNC_BYTES, sp), "down GEMM"))
    repack_bytes = M * N_up * 4 + M * N_up + M * 4   # algorithmic: fp32 H in, int8 codes + fp32 scales out
    tf = lambda ops_, us: ops_ / (us * 1e-6) / 1e12
    gbs = lambda b_, us: b_ / (us * 1e-6) / 1e9
    roof = {
        "gemm_up_gelu": {"bound": "tensor", "us": round(t_up, 2), "achieved": round(tf(ops_up, t_up), 1),
                         "peak": peak_tf, "unit": "TFLOP/s", "frac": round(tf(ops_up, t_up) / peak_tf, 4)},
        "gemm_down": {"bound": "tensor", "us": round(t_down, 2), "achieved": round(tf(ops_down, t_down), 1),
                      "peak": peak_tf, "unit": "TFLOP/s", "frac": round(tf(ops_down, t_down) / peak_tf, 4)},
        "repack": {"bound": "hbm", "us": round(t_repack, 2), "bytes": repack_bytes,
                   "achieved": round(gbs(repack_bytes, t_repack), 1), "peak": hbm, "unit": "GB/s",
                   "frac": round(gbs(repack_bytes, t_repack) / hbm, 4)},
        "pack": {"bound": "hbm", "us": round(t_pack, 2)},
        "peak_kind": f"{peak_kind} (bf16 dense burst; HBM copy)",
    }
    del Qx, Qh, sh

    # end to end: pinned host X in, Y back to pinned host memory, inside the events
    Xh = torch.from_numpy(mcase.X).pin_memory()
    Yh = torch.empty((M, N_down), dtype=torch.float32).pin_memory()
    Xd = torch.empty_like(Xm)

    def e2e_call():
        Xd.copy_(Xh, non_blocking=True)
        ops.convrot_mlp(Xd, G, mlp_w[0], ops.ACT_GELU, G, mlp_w[1], Y=Ym, workspace=wsm, stream=stream)
        Yh.copy_(Ym, non_blocking=True)
    t_seq = timed(e2e_call, n=5)

    # the same through convrot_mlp_host: row chunks whose copies in and out run on two copy
    # streams, overlapping the other chunks' compute (the library default is 1536 rows)
    copy_in, copy_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    Yh2 = torch.empty_like(Yh).pin_memory()

    def host_call(rows):
        wsh = torch.empty((ops.convrot_mlp_host_workspace_size(M, K, ops.F32, N_up, N_down, rows),),
                          dtype=torch.uint8, device=dev)
        return lambda: ops.convrot_mlp_host(Xh, G, mlp_w[0], ops.ACT_GELU, G, mlp_w[1], Y=Yh2, chunk_rows=rows,
                                            workspace=wsh, stream=stream, copy_in_stream=copy_in,
                                            copy_out_stream=copy_out)
    by_rows = {rows: timed(host_call(rows), n=5) for rows in (1152, 1536, 2304)}
    t_e2e = timed(host_call(0), n=5)
    e2e = {"value": round((ops_up + ops_down) / (t_e2e * 1e-6) / 1e12, 2), "unit": "TOPS", "us": round(t_e2e, 2),
           "h2d_bytes_per_step": int(Xh.numel() * 4), "d2h_bytes_per_step": int(Yh.numel() * 4),
           "api": "convrot_mlp_host (one call; pinned host X and Y, row chunks of 1536 whose copies overlap "
                  "the other chunks' compute)",
           "us_by_chunk_rows": {str(r): round(t, 2) for r, t in by_rows.items()},
           "sequential": {"us": round(t_seq, 2), "TOPS": round((ops_up + ops_down) / (t_seq * 1e-6) / 1e12, 2),
                          "api": "copy X host->device, one convrot_mlp call, copy Y device->host"}}
    # the pipelined result equals the one-call result
    host_call(0)()
    e2e_call()
    torch.cuda.synchronize()
    e2e["parity_max_abs_diff_vs_one_call"] = float((Yh2 - Yh).abs().max().item())
    del Yh2
    del Xh, Yh, Xd

    # split SwiGLU: gate and up [12288, 3072] sharing the pack, h = silu(gate) * up
    rng = workloads.rng_for(5)
    Wg = torch.from_numpy(workloads.weights(rng, N_up, K)).to(dev)
    q8, sg, qg = ops.convrot_prepare_weight(Wg, G)
    gate = (qg, sg, torch.from_numpy(workloads.biases(rng, N_up)).to(dev), ops.convrot_weight_chunks(q8))
    del q8, Wg
    t_sw = timed(lambda: ops.convrot_mlp(Xm, G, (gate, mlp_w[0]), ops.ACT_SWIGLU, G, mlp_w[1], Y=Ym, workspace=wsm,
                                         stream=stream))
    ops_sw = 2.0 * ops_up + ops_down
    swiglu = {"workload": f"X fp32 [{M},{K}] -> gate and up [{N_up},{K}] (one pack, one GEMM, h = silu(gate) * up "
                          f"in its epilogue) -> repack -> down [{N_down},{N_up}], one convrot_mlp call",
              "us": round(t_sw, 2), "TOPS": round(ops_sw / (t_sw * 1e-6) / 1e12, 2), "ops_per_call": int(ops_sw)}
    del gate

    out = {"workload": f"dit_mlp: X fp32 [{M},{K}] -> up [{N_up},{K}] + GELU (in the up GEMM's epilogue) -> "
                       f"repack -> down [{N_down},{N_up}], G={G}, one convrot_mlp call",
           "ms": round(t_chain * 1e-3, 4), "TOPS": round((ops_up + ops_down) / (t_chain * 1e-6) / 1e12, 2),
           "frac": round((ops_up + ops_down) / (t_chain * 1e-6) / 1e12 / peak_tf, 4),
           "ops_per_call": int(ops_up + ops_down),
           "parts_us": {"pack": round(t_pack, 2), "up_gemm_gelu": round(t_up, 2), "repack": round(t_repack, 2),
                        "down_gemm": round(t_down, 2)},
           "gelu_placement_us": {"in_the_up_gemm_epilogue": {"up_gemm": round(t_up, 2), "repack": round(t_repack, 2)},
                                 "in_the_repack": {"up_gemm": round(t_up_plain, 2),
                                                   "repack": round(t_gelu_repack, 2)}},
           "roofline": roof, "e2e": e2e, "swiglu": swiglu}
    if with_cpu:
        out["cpu_baseline"] = mlp_cpu_baseline(mcase, mw)
    del Xm, mlp_w, Ym, wsm, H
    return out


def mlp_cpu_baseline(case, w, rows=256):
    """The oracle MLP chain (pack, int32 GEMM, reconstruction, GELU, repack,
    int32 GEMM, reconstruction) on the first `rows` rows, weights prepared
    by the oracle beforehand (offline in the method, not timed)."""
    import oracle
    G = w.G
    (Qu, su), (Qd, sd) = [oracle.prepare_weight(W, G) for W in case.Ws]
    X = case.X[:rows]
    t0 = time.perf_counter()
    H = oracle.gelu(oracle.linear(X, Qu, su, case.bs[0], G))
    oracle.linear(H, Qd, sd, case.bs[1], G)
    t = time.perf_counter() - t0
    ops_ = 2.0 * rows * (w.Ns[0] * w.K + w.Ns[1] * w.Ns[0])
    try:
        cores = len(os.sched_getaffinity(0))
    except Exception:
        cores = os.cpu_count() or 1
    return {"value": ops_ / t / 1e12, "unit": "TOPS", "cores": cores, "kind": "oracle",
            "sample": f"oracle MLP chain on the first {rows} of {w.M} rows ({t:.2f} s; numpy/BLAS on all host cores)"}


def small_configs_in_graph(dev, replays=5):
    """The small workloads (tiny and UNet-like), one convrot_linear call each
    (pack + GEMM), timed inside a captured CUDA graph so that launch overhead
    is amortized: the graph holds one call per set of input, output and
    workspace buffers, with enough sets (more than 4x L2 in total) that no
    call finds its data in L2 from the call before. Context, not the step."""
    import torch
    from int8_hadamard_rotated_gb300 import ops
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (126 << 20))
    out = {}
    for name in ("tiny", "unet"):
        w = workloads.get(name)
        case = workloads.make_case(w)
        preps = [ops.convrot_prepare_weight(torch.from_numpy(W).to(dev), w.G) for W in case.Ws]
        q16s, scales = [p[2] for p in preps], [p[1] for p in preps]
        biases = [torch.from_numpy(b).to(dev) for b in case.bs]
        plans = [ops.convrot_weight_chunks(p[0]) for p in preps]
        X0 = torch.from_numpy(case.X).to(dev)
        per_set = X0.numel() * X0.element_size() + sum(w.M * n * 4 for n in w.Ns)
        nsets = int(min(256, max(2, -(-4 * l2 // per_set))))
        Xs = [X0.clone() for _ in range(nsets)]
        Ys = [[torch.empty((w.M, n), dtype=torch.float32, device=dev) for n in w.Ns] for _ in range(nsets)]
        wss = [torch.empty((ops.convrot_linear_workspace_size(w.M, w.K),), dtype=torch.uint8, device=dev)
               for _ in range(nsets)]
        descs = [ops.make_weights(q16s, scales, biases, Ys[i], plans) for i in range(nsets)]

        def calls():
            for i in range(nsets):
                ops.convrot_linear(Xs[i], w.G, q16s, scales, biases, Ys=Ys[i], workspace=wss[i], weights=descs[i])
        calls()                      # warm-up outside the graph (configures the kernels)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            calls()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(replays):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        status = ops.convrot_device_status()
        if status != ops.OK:
            raise ops.ConvrotError(status, "device status")
        us = a.elapsed_time(b) * 1e3 / (replays * nsets)
        out[name] = {"workload": f"X {'fp16' if name == 'unet' else 'fp32'} [{w.M},{w.K}] G={w.G} -> "
                                 f"{len(w.Ns)} linear(s) N={list(w.Ns)}",
                     "us_per_call": round(us, 3), "TOPS": round(w.gemm_ops / (us * 1e-6) / 1e12, 2),
                     "calls_per_graph": nsets}
        del Xs, Ys, wss, descs, g
    return out


def next_rows_legs(X, w, dev, flush, hbm, q16s, scales, biases, plans, ops_step, reps=20):
    """Context for the rows beyond the step, each on the DiT input and timed
    like the step's parts (L2 flushed before every launch, CUDA events on the
    launching stream, mean over `reps`): the pack with the modulation prologue
    (RMS norm, per-channel weight, (x + x*scale) + shift) beside the plain
    pack of the same X; the one-call linear with an input scale beside the
    plain one-call linear; the three projections as W4A4 linears (packed
    signed 4-bit weights read by the S8 x S4 GEMM). Not part of the step."""
    import torch
    from int8_hadamard_rotated_gb300 import ops

    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    L = ops.lib()
    M, K = X.shape

    def timed(fn):
        for _ in range(3):
            fn()
        ev = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            ev.append((a, b))
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in ev])) * 1e3  # us

    # f2: modulation prologue fused into the pack (int8 codes)
    wv, sc, sh = (torch.from_numpy(v).to(dev) for v in workloads.modulation(workloads.rng_for(11), K))
    Q = torch.empty((M, K), dtype=torch.int8, device=dev)
    s = torch.empty((M,), dtype=torch.float32, device=dev)
    t_pro = timed(lambda: ops.convrot_pack_prologue(X, w.G, rmsnorm=True, weight=wv, scale=sc, shift=sh,
                                                    Q_x=Q, s_x=s, stream=stream))
    t_plain = timed(lambda: ops.convrot_pack_activations(X, w.G, Q_x=Q, s_x=s, stream=stream))
    pro_bytes = M * K * 4 + M * K + M * 4 + 3 * K * 4
    f2 = {"workload": f"X fp32 [{M},{K}], G={w.G}: RMS norm, weight, (x + x*scale) + shift, then the pack -> int8 + s",
          "bound": "hbm", "bytes": pro_bytes, "us": round(t_pro, 2),
          "GB/s": round(pro_bytes / (t_pro * 1e-6) / 1e9, 1), "frac": round(pro_bytes / (t_pro * 1e-6) / 1e9 / hbm, 4),
          "plain_pack_us": round(t_plain, 2)}
    del Q, s

    # f4: input scale (scaled pack, then the GEMM that unscales before the bias)
    Ys = [torch.empty((M, q.shape[0]), dtype=torch.float32, device=dev) for q in q16s]
    ws = torch.empty((ops.convrot_linear_workspace_size(M, K),), dtype=torch.uint8, device=dev)
    wdesc = ops.make_weights(q16s, scales, biases, Ys, plans)
    t_lin = timed(lambda: ops.convrot_linear(X, w.G, q16s, scales, biases, Ys=Ys, workspace=ws, stream=stream,
                                             weights=wdesc))
    t_scaled = timed(lambda: ops.convrot_linear_scaled(X, w.G, 0.37, q16s, scales, biases, Ys=Ys, workspace=ws,
                                                       stream=stream, weights=wdesc))
    f4 = {"workload": f"{w.name}: one convrot_linear_scaled call, input scale 0.37", "bound": "tensor",
          "us": round(t_scaled, 2), "TOPS": round(ops_step / (t_scaled * 1e-6) / 1e12, 2),
          "plain_linear_us": round(t_lin, 2), "plain_linear_TOPS": round(ops_step / (t_lin * 1e-6) / 1e12, 2)}
    del Ys, ws

    # f3: W4A4 linears -- the three projections with packed signed 4-bit
    # weights (0.5 B per weight, read as they are by the S8 x S4 GEMM)
    rng4 = workloads.rng_for(12)
    P4 = [torch.from_numpy(workloads.packed_int4(rng4, q.shape[0], K)).to(dev) for q in q16s]
    s4 = [torch.from_numpy((0.001 + 0.01 * rng4.random(q.shape[0])).astype(np.float32)).to(dev) for q in q16s]
    Y4 = [torch.empty((M, q.shape[0]), dtype=torch.float32, device=dev) for q in q16s]
    w4desc = ops.make_weights(P4, s4, biases, Y4)
    Q16 = torch.empty((M, K), dtype=torch.float16, device=dev)
    sx = torch.empty((M,), dtype=torch.float32, device=dev)
    sync_ws = torch.zeros((ops.GEMM_SYNC_BYTES,), dtype=torch.uint8, device=dev)
    ops.convrot_pack_activations_f16(X, w.G, Q_x16=Q16, s_x=sx, stream=stream)

    def gemm_w4():
        st = L.convrot_linear_packed(Q16.data_ptr(), sx.data_ptr(), M, K, w4desc, len(P4), sync_ws.data_ptr(),
                                     ops.GEMM_SYNC_BYTES, sp)
        if st:
            raise ops.ConvrotError(st, "convrot_linear_packed (W4A4)")
    t_g4 = timed(gemm_w4)
    ws4 = torch.empty((ops.convrot_linear_workspace_size(M, K),), dtype=torch.uint8, device=dev)
    t_l4 = timed(lambda: ops.convrot_linear(X, w.G, P4, s4, biases, Ys=Y4, workspace=ws4, stream=stream,
                                            weights=w4desc))
    n_w = sum(q.shape[0] for q in q16s)
    f3 = {"workload": f"{w.name}: three W4A4 projections [{q16s[0].shape[0]},{K}] (packed signed 4-bit weights, "
                      "F32 row scales) sharing one pack",
          "bound": "tensor", "gemm_us": round(t_g4, 2), "gemm_TOPS": round(ops_step / (t_g4 * 1e-6) / 1e12, 2),
          "linear_us": round(t_l4, 2), "linear_TOPS": round(ops_step / (t_l4 * 1e-6) / 1e12, 2),
          "weight_bytes_read_per_launch": int(n_w * K // 2),
          "weight_bytes_binary16_gemm": int(n_w * K * 2),
          "note": "the S8 x S4 GEMM reads the packed bytes (TMA) and widens them to exact binary16 "
                  "codes in shared memory; no expanded copy of the weights exists"}
    del P4, Y4, ws4, Q16
    return {"f2_pack_prologue": f2, "f4_input_scale": f4, "f3_w4a4_linear": f3,
            "note": "isolated launches, L2 flushed before each (launch latency included); "
                    "frac against the measured HBM copy peak"}


def library_gemm_same_shape(w, dev, flush, ours_us, reps=20):
    """Context for the GEMM roofline: cuBLAS (through torch.mm) on the same
    shape, M x sum(N) x K with binary16 operands and fp32 output, L2 flushed
    before each call like the timed steps. Not part of the step."""
    import torch
    n = sum(w.Ns)
    a = torch.randn(w.M, w.K, device=dev).half()
    b = torch.randn(n, w.K, device=dev).half()
    try:
        fn = lambda: torch.mm(a, b.t(), out_dtype=torch.float32)
        fn()
    except (TypeError, RuntimeError) as e:
        return {"unavailable": f"torch.mm with out_dtype: {type(e).__name__}"}
    for _ in range(3):
        flush.zero_()
        fn()
    ev = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        ev.append((e0, e1))
    torch.cuda.synchronize()
    us = float(np.mean([x.elapsed_time(y) for x, y in ev])) * 1e3
    ops = 2.0 * w.M * n * w.K
    return {"kernel": "cuBLAS binary16 x binary16 -> fp32 (torch.mm, out_dtype=float32), no reconstruction",
            "shape": [w.M, n, w.K], "us": round(us, 2), "TFLOP/s": round(ops / (us * 1e-6) / 1e12, 1),
            "ours_gemm_us": round(ours_us, 2)}


def run_reference(args, rank):
    """The oracle as the reference arm: each step is the oracle on a bounded
    sample (the first 256 rows) of the same workload."""
    if rank != 0:
        return None
    import oracle
    w = workloads.get(WORKLOAD)
    case = workloads.make_case(w)
    rows = 256
    prepared = [oracle.prepare_weight(W, w.G) for W in case.Ws]
    for _ in range(args.warmup):
        oracle_sample_seconds(case, w, rows, prepared)
    times = [oracle_sample_seconds(case, w, rows, prepared) for _ in range(args.steps)]
    t = float(np.mean(times))
    ops_step = 2.0 * rows * sum(w.Ns) * w.K
    v = ops_step / t / 1e12
    try:
        cores = len(os.sched_getaffinity(0))
    except Exception:
        cores = os.cpu_count() or 1
    return {
        "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": data_desc(w),
        "config": config_dict(w, 1), "impl": "reference",
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"oracle on the first {rows} of {w.M} rows per step"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-library-gemm", dest="library_gemm", action="store_false",
                    help="skip timing cuBLAS on the GEMM's shape (context for the roofline)")
    ap.add_argument("--no-small-configs", dest="small_configs", action="store_false",
                    help="skip the tiny and UNet-like configs timed inside a CUDA graph")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        res = run_reference(args, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res, case, w = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            res["cpu_baseline"] = cpu_baseline(case, w)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
