#!/usr/bin/env python
"""Throughput of the tcgen05 GEMM library on one or more GB300s.

One step = one pass of the whole GEMM path over the headline workload:
D = A B^T for bf16 8192^3 and for block-scaled MXFP8 8192^3 (the two halves
of the headline metric; the MXFP8 GEMM also exercises the scale-factor path).
``value`` is the whole job's algorithmic TFLOP/s (2 M N K per GEMM, summed
over the step and over all ranks) with inputs already resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle, as it stands

Timing: W untimed warm-up steps, then K steps bracketed by a barrier and a
device synchronise on both sides, CUDA events on the launching stream, max
over ranks.  The operands (256 MiB of bf16, 128 MiB of E4M3) are larger
than the 129 MB L2, so no flush is needed between steps.  Multi-GPU runs are
weak-scaled replicas: every rank multiplies its own copy of the workload and
no data-path collective exists (the barrier and the max-reduction of the
elapsed time are the only inter-rank traffic).
"""
from __future__ import annotations

import argparse
import csv
import datetime
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1000 * 1000   # GB300 L2 (about 129 MB)
METRIC = "GEMM TFLOP/s and % of dense tensor peak (bf16 & MXFP8, 8192³) on 1 GB300"
HEADLINE = ("square_8192", "mxfp8_8192")
FP8_OVER_BF16 = 2.0   # nominal dense FP8 / BF16 tensor ratio (4.5 vs 2.25 PFLOP/s)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------- utilities

def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="headline",
                    help="headline (bf16 8192^3 + MXFP8 8192^3) or one named workload")
    ap.add_argument("--variant", type=int, default=0, help="kernel variant (0 = auto)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-library-context", action="store_true",
                    help="skip the cuBLAS context figures measured after the timed region")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    """Hash of the CUDA sources, to tell whether stored ncu counters still
    describe the kernels being timed."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_gemm_blackwell_tcgen05_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name in PERSISTENT_KERNEL_SOURCES:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


# The sources of the persistent tcgen05 kernels and their launcher: the DRAM
# counters stored under profiles/ hold while these are unchanged.
PERSISTENT_KERNEL_SOURCES = ("ptx.cuh", "kernel_common.cuh", "gemm_kernels.cuh", "launch_ws.cuh",
                             "gemm_host.h", "gemm_bf16.cu", "gemm_mxfp8.cu")


def stored_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    if t.get("source_hash") != kernel_source_hash():
        return None
    ent = t.get("kernels", {}).get(kernel_key)
    return None if ent is None else ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples around the timed region,
    every 10 ms, each with its host timestamp.  sm_mhz is the median over the
    samples taken inside the timed region's wall-clock window; with none
    there, over the samples under load (the board drawing at least 30% of its
    power limit -- nvidia-smi averages power.draw over a window longer than a
    short region, so short regions rarely show it), else over all samples.
    The counts are reported too."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
             "power.limit,timestamp")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.buf = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None

    @staticmethod
    def _stamp(x):
        try:
            return datetime.datetime.strptime(x.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self, window=None):
        """Stop sampling and summarise; window = (start, end) of the timed
        region in host seconds since the epoch (time.time())."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 10]
        if not rows:
            return None
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        pairs = [(num(r[1]), num(r[3]), num(r[9])) for r in rows]
        sm = [c for c, _, _ in pairs if c is not None]
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        power = [w for _, w, _ in pairs if w is not None]
        pmax = max(power) if power else None
        loaded = [c for c, w, lim in pairs
                  if c is not None and w is not None and lim is not None and w >= 0.3 * lim]
        inside = []
        if window is not None:
            for r, (c, _, _) in zip(rows, pairs):
                ts = self._stamp(r[10]) if len(r) > 10 else None
                if c is not None and ts is not None and window[0] <= ts <= window[1]:
                    inside.append(c)
        return {"sm_mhz": statistics.median(inside or loaded or sm) if sm else None,
                "samples_in_region": len(inside),
                "sm_mhz_all_samples": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "active_masks": sorted({r[4].strip() for r in rows}),
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": pmax}


def tensor_peak_choice(region_s: float, clk) -> tuple[str, str]:
    """Which measured tensor peak a kernel timed in this region is held to:
    the sustained one (cuBLAS back to back for seconds under the power cap)
    only when the timed region itself ran for a second or more with the
    power cap active; otherwise the burst one."""
    capped = bool(clk) and "sw_power_cap" in (clk.get("reasons") or [])
    if region_s >= 1.0 and capped:
        return "sustained", f"timed region {region_s:.2f} s with sw_power_cap active"
    return "burst", (f"timed region {region_s:.3f} s" + (", sw_power_cap active" if capped
                                                        else ", no sw_power_cap"))


def dist_setup(want_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ the workload

def workload_list(name: str):
    import gemm_inputs as gi
    names = HEADLINE if name == "headline" else (name,)
    for n in names:
        if n not in gi.WORKLOADS:
            raise SystemExit(f"unknown workload {n}; known: headline, {', '.join(gi.WORKLOADS)}")
    return [gi.WORKLOADS[n] for n in names]


def host_operands(w, pinned: bool = True):
    """Seeded inputs on the host (page-locked when a GPU will copy them): the
    GEMM operands, then the epilogue's C and bias when the workload has them."""
    import gemm_inputs as gi
    ops = gi.workload_operands(w.name) + tuple(t for t in gi.epilogue_operands(w) if t is not None)
    return tuple(t.pin_memory() for t in ops) if pinned else ops


def n_gemm_operands(w) -> int:
    return {"quant": 1, "bf16": 2, "mxfp8": 4}[w.kind]


def alg_bytes(w) -> int:
    import gemm_inputs as gi
    if w.kind == "quant":
        return 4 * w.M * w.K + w.M * w.K + w.M * ((w.K + 31) // 32)
    spec = gi.epilogue_spec(w)
    out = 4 if spec and spec["out"] == "f32" else 2
    extra = 0
    if spec:
        extra += w.M * w.N * out if spec["beta"] != 0.0 else 0
        extra += w.N * {"none": 0, "bf16": 2, "f32": 4}[spec["bias"]]
    if w.kind == "bf16":
        return 2 * (w.M * w.K + w.N * w.K) + out * w.M * w.N + extra
    nblk = (w.K + 31) // 32
    return w.M * w.K + w.N * w.K + (w.M + w.N) * nblk + out * w.M * w.N + extra


class Problem:
    """Device buffers of one workload plus the call that runs it."""

    def __init__(self, w, host, variant, device):
        import torch

        import dense_gemm_blackwell_tcgen05_gb300 as g
        import gemm_inputs as gi
        self.w = w
        self.tiled = w.kind == "mxfp8" and w.sf_layout == "tiled"
        self.rows_dev = None
        if self.tiled:
            # the same scale bytes, rearranged on the host into the tiled layout
            # the GEMM takes (what a caller keeps its scales in for this path)
            A, SFA, B, SFB = host[:4]
            self.rows_dev = (SFA.to(device), SFB.to(device))   # row-major twin (context only)
            tiles = (gi.tile_scales(SFA, w.M, w.K), gi.tile_scales(SFB, w.N, w.K))
            if SFA.is_pinned():
                tiles = tuple(t.pin_memory() for t in tiles)
            host = (A, tiles[0], B, tiles[1]) + tuple(host[4:])
        self.host = host
        self.dev = tuple(t.to(device, non_blocking=False) for t in host)
        self.spec = gi.epilogue_spec(w)
        self.variant = variant if variant else w.variant
        if w.kind == "quant":
            pitch = max(16, ((w.K + 31) // 32 + 15) // 16 * 16)
            self.D = torch.empty(w.M, w.K, dtype=torch.uint8, device=device)       # codes
            self.SF = torch.zeros(w.M, pitch, dtype=torch.uint8, device=device)
            self.D_host = torch.empty(w.M, w.K, dtype=torch.uint8).pin_memory()
        else:
            out_dt = torch.float32 if self.spec and self.spec["out"] == "f32" else torch.bfloat16
            self.out_dtype = out_dt
            self.D = torch.empty(w.M, w.N, dtype=out_dt, device=device)
            self.D_host = torch.empty(w.M, w.N, dtype=out_dt).pin_memory()
        self.ws = (g.streamk_workspace(w.kind == "mxfp8", self.variant, device)
                   if w.schedule == "streamk" else None)
        self._epi = {}

    def epilogue(self, tensors):
        """The GemmEpilogue for this set of device tensors (cached per set)."""
        import dense_gemm_blackwell_tcgen05_gb300 as g
        key = tuple(t.data_ptr() for t in tensors)
        if key not in self._epi:
            sp = self.spec
            it = iter(tensors)
            C = next(it) if sp["beta"] != 0.0 else None
            bias = next(it) if sp["bias"] != "none" else None
            self._epi[key] = g.make_epilogue(sp["alpha"], sp["beta"], C, bias, sp["act"],
                                             self.out_dtype)
        return self._epi[key]

    def new_outputs(self):
        """A second set of output buffers (the pipelined end-to-end loop)."""
        import torch
        if self.w.kind == "quant":
            return (torch.empty_like(self.D), torch.zeros_like(self.SF))
        return (torch.empty_like(self.D),)

    def launch(self, stream_handle: int, bufs=None, outs=None) -> int:
        import dense_gemm_blackwell_tcgen05_gb300 as g
        w = self.w
        b = self.dev if bufs is None else bufs
        k = n_gemm_operands(w)
        ops, epi_t = b[:k], b[k:]
        if w.kind == "quant":
            (X,) = ops
            Q, SF = (self.D, self.SF) if outs is None else outs
            return g.gemm_mxfp8_quantize(X.data_ptr(), w.M, w.K, X.stride(0), Q.data_ptr(),
                                         Q.stride(0), SF.data_ptr(), SF.stride(0), stream_handle)
        D, v = (self.D if outs is None else outs[0]), self.variant
        if w.kind == "bf16":
            A, B = ops
            args = (A.data_ptr(), B.data_ptr(), D.data_ptr(), w.M, w.N, w.K, A.stride(0),
                    B.stride(0), D.stride(0))
            if self.spec:
                return g.gemm_bf16_fused(v, *args, self.epilogue(epi_t), stream_handle)
            if self.ws is not None:
                return g.gemm_bf16_streamk(v, *args, self.ws.data_ptr(), self.ws.numel(),
                                           stream_handle)
            return g.gemm_bf16_variant(v, *args, stream_handle)
        A, SFA, B, SFB = ops
        if self.tiled:
            return g.gemm_mxfp8_tiled(v, A.data_ptr(), B.data_ptr(), SFA.data_ptr(), SFB.data_ptr(),
                                      D.data_ptr(), w.M, w.N, w.K, A.stride(0), B.stride(0),
                                      D.stride(0), stream_handle)
        args = (A.data_ptr(), B.data_ptr(), SFA.data_ptr(), SFB.data_ptr(), D.data_ptr(), w.M,
                w.N, w.K, A.stride(0), B.stride(0), SFA.stride(0), SFB.stride(0), D.stride(0))
        if self.spec:
            return g.gemm_mxfp8_fused(v, *args, self.epilogue(epi_t), stream_handle)
        if self.ws is not None:
            return g.gemm_mxfp8_streamk(v, *args, self.ws.data_ptr(), self.ws.numel(),
                                        stream_handle)
        return g.gemm_mxfp8_variant(v, *args, stream_handle)

    def h2d_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.host)

    def d2h_bytes(self) -> int:
        return self.D.numel() * self.D.element_size()


# ------------------------------------------------------------ CPU oracle leg

def oracle_entries(w, host, n: int) -> float:
    """Run the oracle on the first `n` entries of D in row-major order; seconds."""
    import numpy as np
    import torch

    import gemm_inputs as gi
    import oracle
    ncols = w.K if w.kind == "quant" else w.N
    t = np.arange(n, dtype=np.int64)
    r, c = t // ncols, t % ncols
    rows = int(r[-1]) + 1
    k = n_gemm_operands(w)
    ops, epi_t = host[:k], host[k:]
    t0 = time.perf_counter()
    if w.kind == "quant":
        (X,) = ops
        oracle.mxfp8_quantize(X.numpy()[:rows])
        return time.perf_counter() - t0
    if w.kind == "bf16":
        A, B = ops
        P, _ = oracle.gemm_bf16_entries(gi.bf16_codes(A[:rows]), gi.bf16_codes(B), r, c)
    else:
        A, SFA, B, SFB = ops
        P, _ = oracle.gemm_mxfp8_entries(A[:rows].numpy(), B.numpy(), SFA[:rows].numpy(),
                                         SFB.numpy(), r, c)
    spec = gi.epilogue_spec(w)
    if spec:
        it = iter(epi_t)
        dec = lambda t: t.double().numpy() if t.dtype != torch.bfloat16 else \
            oracle.bf16_to_f64(gi.bf16_codes(t))
        ri, ci = torch.from_numpy(r), torch.from_numpy(c)
        C = dec(next(it)[ri, ci])[None, :] if spec["beta"] != 0.0 else None
        bias = dec(next(it)[ci]) if spec["bias"] != "none" else None
        oracle.epilogue(np.asarray(P).reshape(1, -1), spec["alpha"], spec["beta"], C, bias,
                        {"none": 0, "relu": 1, "gelu": 2}[spec["act"]])
    return time.perf_counter() - t0


def plan_oracle_sample(works, hosts, seconds: float):
    """Entries per workload so that one pass of the sample takes about `seconds`."""
    plan = []
    for w, h in zip(works, hosts):
        total = w.M * (w.K if w.kind == "quant" else w.N)
        probe = min(total, 4096 if w.kind != "quant" else 65536)
        t1 = max(oracle_entries(w, h, probe) / probe, 1e-9)
        n = int(max(1, min(total, (seconds / len(works)) / t1)))
        plan.append(n)
    return plan


def oracle_pass(works, hosts, plan):
    secs = 0.0
    flops = 0
    for w, h, n in zip(works, hosts, plan):
        secs += oracle_entries(w, h, n)
        flops += n * 5 + (n + 31) // 32 if w.kind == "quant" else 2 * n * w.K   # quantiser: bytes
    return flops, secs


def step_unit(works):
    """The step's amount per pass, its unit and scale: algorithmic FLOPs in
    TFLOP/s when any GEMM is in the step, else algorithmic bytes in GB/s."""
    flops = sum(w.flops for w in works)
    if flops:
        return flops, "TFLOP/s", 1e12
    return sum(alg_bytes(w) for w in works), "GB/s", 1e9


def workload_text(works) -> str:
    """The config's workload name, the same string in both arms."""
    return " + ".join(f"{w.name} {w.M}x{w.N}x{w.K} {w.kind}" for w in works)


def sample_text(works, plan) -> str:
    return "; ".join(f"first {n} of {w.M * w.N} outputs (row-major) of {w.name} "
                     f"({w.M}x{w.N}x{w.K} {w.kind})" for w, n in zip(works, plan))


# --------------------------------------------------------------- the arms

def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    works = workload_list(args.workload)
    hosts = [host_operands(w, pinned=False) for w in works]
    oracle.default()
    budget = 150.0 / max(1, args.steps + args.warmup)
    plan = plan_oracle_sample(works, hosts, budget)
    for _ in range(args.warmup):
        oracle_pass(works, hosts, plan)
    flops = 0
    secs = 0.0
    for _ in range(args.steps):
        f, s = oracle_pass(works, hosts, plan)
        flops += f
        secs += s
    _, unit, scale = step_unit(works)
    value = flops / secs / scale
    cores = oracle.num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_text(works), "parallelism": "none (CPU)"},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": sample_text(works, plan) + " per step"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def blocked_scales(sf, rows: int, K: int):
    """UE8M0 scales [rows, >= K/32] in cuBLASLt's block-scaled layout (the tiled layout of
    gemm_inputs.tile_scales: 128-row x 4-block tiles of 512 bytes), shaped [R, C] and typed
    as torch._scaled_mm takes them.  Context leg only."""
    import torch

    import gemm_inputs as gi
    R, C = (rows + 127) // 128 * 128, ((K + 31) // 32 + 3) // 4 * 4
    return gi.tile_scales(sf, rows, K).view(R, C).view(torch.float8_e8m0fnu)


def library_context(probs, stream, n: int, flush_buf, flush_each):
    """cuBLAS on the same device operands, for context: torch.matmul for plain bf16 and
    torch._scaled_mm (block-scaled E4M3) for plain MXFP8 workloads (the stream-K ones
    included: cuBLAS picks its own schedule for the shape).  Measured after the
    timed region, alternating with our own kernel (two rounds of n launches each, same
    flush policy), so both see the same clocks.  No step of the path calls these."""
    import torch

    import dense_gemm_blackwell_tcgen05_gb300 as g
    out = {}
    for j, p in enumerate(probs):
        w = p.w
        if w.kind not in ("bf16", "mxfp8") or p.spec:
            continue
        try:
            if w.kind == "bf16":
                A, B = p.dev[:2]
                lib_name = "torch.matmul (cuBLAS)"
                lib = lambda A=A, B=B: torch.matmul(A, B.t())
            else:
                A, SFA, B, SFB = p.dev[:4]
                if p.tiled:   # already the layout cuBLASLt takes
                    R = lambda n: (n + 127) // 128 * 128
                    C = ((w.K + 31) // 32 + 3) // 4 * 4
                    sa = SFA.view(R(w.M), C).view(torch.float8_e8m0fnu)
                    sb = SFB.view(R(w.N), C).view(torch.float8_e8m0fnu)
                else:
                    sa, sb = blocked_scales(SFA, w.M, w.K), blocked_scales(SFB, w.N, w.K)
                a8, b8 = A.view(torch.float8_e4m3fn), B.view(torch.float8_e4m3fn)
                lib_name = "torch._scaled_mm (cuBLASLt, block-scaled E4M3)"
                lib = lambda a8=a8, b8=b8, sa=sa, sb=sb: torch._scaled_mm(
                    a8, b8.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16)
            with torch.cuda.stream(stream):
                rc = p.launch(stream.cuda_stream)
                if rc != g.GEMM_OK:
                    raise g.GemmError(rc, w.name)
                ref = lib()
            torch.cuda.synchronize()
            same = bool(torch.equal(ref.view(torch.int16), p.D.view(torch.int16)))

            def timed(f):
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                total = 0.0
                with torch.cuda.stream(stream):
                    if flush_each[j]:
                        for _ in range(n):
                            flush_buf.zero_()
                            s.record(stream)
                            f()
                            e.record(stream)
                            e.synchronize()
                            total += s.elapsed_time(e)
                    else:
                        s.record(stream)
                        for _ in range(n):
                            f()
                        e.record(stream)
                        e.synchronize()
                        total = s.elapsed_time(e)
                return total / n

            ours_f = lambda: p.launch(stream.cuda_stream)
            t_ours, t_lib = [], []
            for _ in range(2):
                t_ours.append(timed(ours_f))
                t_lib.append(timed(lib))
            out[w.name] = {"library": lib_name,
                           "library_tflops": w.flops / (min(t_lib) / 1e3) / 1e12,
                           "ours_tflops": w.flops / (min(t_ours) / 1e3) / 1e12,
                           "launches": 2 * n, "bitwise_equal_to_ours": same}
            if p.tiled:
                # our row-major-scale entry point on the same operands
                SAr, SBr = p.rows_dev
                rows_f = lambda: g.gemm_mxfp8_variant(
                    0, A.data_ptr(), B.data_ptr(), SAr.data_ptr(), SBr.data_ptr(), p.D.data_ptr(),
                    w.M, w.N, w.K, A.stride(0), B.stride(0), SAr.stride(0), SBr.stride(0),
                    p.D.stride(0), stream.cuda_stream)
                t_rows = [timed(rows_f) for _ in range(2)]
                out[w.name]["ours_row_major_scales_tflops"] = w.flops / (min(t_rows) / 1e3) / 1e12
        except Exception as exc:   # a torch without block-scaled _scaled_mm, for instance
            out[w.name] = {"unavailable": repr(exc)[:200]}
    return out


def run_ours(args, rank, world, local):
    import torch

    import dense_gemm_blackwell_tcgen05_gb300 as g
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    g.load()
    works = workload_list(args.workload)
    hosts = [host_operands(w) for w in works]
    probs = [Problem(w, h, args.variant, device) for w, h in zip(works, hosts)]
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    step_flops, unit, scale = step_unit(works)

    def step():
        for p in probs:
            rc = p.launch(sh)
            if rc != g.GEMM_OK:
                raise g.GemmError(rc, p.w.name)

    # ---- warm-up (also the correctness gate of the watchdog status) ----
    for _ in range(max(3, args.warmup)):
        step()
    st = g.gemm_last_status(sh)
    if st != g.GEMM_OK:
        raise g.GemmError(st, "warm-up")

    # ---- device-resident timed region ----
    # A one-kernel step runs its K launches back to back between two events
    # (an event between kernels would keep the next launch from overlapping the
    # previous kernel's tail), so the region's time is also that kernel's.  A
    # step of several kernels records an event pair around every launch inside
    # the region, which gives each kernel's duration under the same clocks.
    # Workloads whose inputs fit in L2 get a 512 MiB write before each launch
    # (outside their events) and are timed by their kernels' events alone.
    flush_each = [p.h2d_bytes() < L2_BYTES for p in probs]
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=device) if any(flush_each) else None
    per_launch = any(flush_each) or len(probs) > 1
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)

    def launches(n, starts=None, ends=None):
        for i in range(n):
            for j, p in enumerate(probs):
                if flush_each[j]:
                    flush_buf.zero_()
                if starts is not None:
                    starts[j][i].record(stream)
                rc = p.launch(sh)
                if ends is not None:
                    ends[j][i].record(stream)
                if rc != g.GEMM_OK:
                    raise g.GemmError(rc, p.w.name)

    def event_grid(n):
        return [[torch.cuda.Event(enable_timing=True) for _ in range(n)] for _ in probs]

    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(device)
    clocks.start()
    time.sleep(0.3)   # let the sampler attach before the first timed kernel
    starts = ends = None
    if per_launch:
        starts, ends = event_grid(args.steps), event_grid(args.steps)
    wall0 = time.time()
    t0.record(stream)
    launches(args.steps, starts, ends)
    t1.record(stream)
    torch.cuda.synchronize(device)
    wall1 = time.time()
    barrier(world)
    clk = clocks.stop((wall0, wall1))
    st = g.gemm_last_status(sh)
    if st != g.GEMM_OK:
        raise g.GemmError(st, "timed region")
    if per_launch:
        kern_ms = [statistics.fmean(s.elapsed_time(e) for s, e in zip(starts[j], ends[j]))
                   for j in range(len(probs))]
    # The same events around a one-element fill after the same flush: the floor
    # this protocol puts under any launch (context for the small workloads).
    event_floor_us = None
    if any(flush_each):
        tiny = torch.zeros(1, device=device)
        floor = []
        for _ in range(20):
            flush_buf.zero_()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            tiny.zero_()
            a1.record(stream)
            a1.synchronize()
            floor.append(a0.elapsed_time(a1))
        event_floor_us = 1e3 * statistics.median(floor)
    # Context for the same workloads, outside the timed region: the mean time
    # per launch of 1000 back-to-back launches with no flush between them (the
    # operands stay in L2), the figure a caller sees in a loop of small GEMMs.
    back_to_back_us = None
    if any(flush_each):
        back_to_back_us = {}
        for j, p in enumerate(probs):
            if not flush_each[j]:
                continue
            for _ in range(3):
                p.launch(sh)
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            for _ in range(1000):
                rc = p.launch(sh)
                if rc != g.GEMM_OK:
                    raise g.GemmError(rc, p.w.name)
            b1.record(stream)
            b1.synchronize()
            back_to_back_us[p.w.name] = 1e3 * b0.elapsed_time(b1) / 1000
        st = g.gemm_last_status(sh)
        if st != g.GEMM_OK:
            raise g.GemmError(st, "back-to-back launches")
    if any(flush_each):
        elapsed_ms = max_over_ranks(args.steps * sum(kern_ms), world)
    else:
        elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world)
    if not per_launch:
        kern_ms = [elapsed_ms / args.steps]   # one kernel per step: the region's own time
    value = world * args.steps * step_flops / (elapsed_ms / 1e3) / scale

    # ---- end to end through the C ABI from pinned host buffers ----
    # Every step copies its inputs from pinned host memory, runs the step's
    # calls and copies its results (the whole D, and the scales for the
    # quantiser) back, all inside the timed region.  Steps are pipelined the
    # way a serving loop would run them: inputs, compute and results each on a
    # stream of their own, with two device buffer sets, so that step i+1's
    # inputs arrive while step i computes and step i-1's results leave.
    e2e_steps = max(1, args.e2e_steps)
    h2d = sum(p.h2d_bytes() for p in probs)
    d2h = sum(p.d2h_bytes() for p in probs)
    nbuf = 2
    staging = [[tuple(torch.empty_like(t, device=device) for t in p.host) for p in probs]
               for _ in range(nbuf)]
    outs = [[(p.D, p.SF) if p.w.kind == "quant" else (p.D,) for p in probs]] + \
           [[p.new_outputs() for p in probs] for _ in range(nbuf - 1)]
    s_in, s_comp, s_out = (torch.cuda.Stream(device) for _ in range(3))

    def e2e_run(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_comp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            b = i % nbuf
            if i >= nbuf:
                s_in.wait_event(ev_comp[i - nbuf])      # buffer set b no longer read
            with torch.cuda.stream(s_in):
                for buf, p in zip(staging[b], probs):
                    for dst, src in zip(buf, p.host):
                        dst.copy_(src, non_blocking=True)
            ev_in[i].record(s_in)
            s_comp.wait_event(ev_in[i])
            if i >= nbuf:
                s_comp.wait_event(ev_out[i - nbuf])     # outputs b already copied out
            for buf, out, p in zip(staging[b], outs[b], probs):
                rc = p.launch(s_comp.cuda_stream, buf, out)
                if rc != g.GEMM_OK:
                    raise g.GemmError(rc, p.w.name)
            ev_comp[i].record(s_comp)
            s_out.wait_event(ev_comp[i])
            with torch.cuda.stream(s_out):
                for out, p in zip(outs[b], probs):
                    p.D_host.copy_(out[0], non_blocking=True)
            ev_out[i].record(s_out)
        return ev_out[n - 1]

    e2e_run(nbuf)   # warm the streams and buffers
    barrier(world)
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_comp.wait_event(e0)
    s_out.wait_event(e0)
    last = e2e_run(e2e_steps)
    s_out.wait_event(last)
    e1.record(s_out)
    torch.cuda.synchronize(device)
    barrier(world)
    st = g.gemm_last_status(s_comp.cuda_stream)
    if st != g.GEMM_OK:
        raise g.GemmError(st, "end-to-end region")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = world * e2e_steps * step_flops / (e2e_ms / 1e3) / scale

    # ---- roofline of each kernel (the first workload's kernel dominates) ----
    peaks, peak_src = load_peaks()
    region_s = elapsed_ms / 1e3
    choice, why = tensor_peak_choice(region_s, clk)
    bf16_peaks = {"burst": peaks["bf16_tflops"],
                  "sustained": peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])}
    kernels = {}
    for p, ms in zip(probs, kern_ms):
        w = p.w
        tflops = w.flops / (ms / 1e3) / 1e12
        gbs = alg_bytes(w) / (ms / 1e3) / 1e9
        ent = {}
        if (w.kind == "bf16" and w.K >= 256) or w.kind == "mxfp8":
            ratio = FP8_OVER_BF16 if w.kind == "mxfp8" else 1.0
            bound, ach, pk, kunit = "tensor", tflops, bf16_peaks[choice] * ratio, "TFLOP/s"
            ent = {"frac_burst": tflops / (bf16_peaks["burst"] * ratio),
                   "frac_sustained": tflops / (bf16_peaks["sustained"] * ratio)}
        else:
            bound, ach, pk, kunit = "hbm", gbs, peaks["hbm_gbs"], "GB/s"
        key = f"{w.name}/variant{args.variant}"
        kernels[w.name] = {"bound": bound, "achieved": ach, "peak": pk, "unit": kunit,
                           "frac": ach / pk, **ent, "traffic": stored_traffic(key),
                           "ms_per_launch": ms, "tflops": tflops, "alg_bytes": alg_bytes(w)}
    dom = max(range(len(probs)), key=lambda j: kern_ms[j])
    roof = {k: kernels[works[dom].name][k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    roof["kernel"] = works[dom].name
    if roof["bound"] == "hbm":
        roof["peak_source"] = f"{peak_src} (hbm_gbs)"
    else:
        name = {"burst": "bf16_tflops", "sustained": "bf16_tflops_sustained"}[choice]
        roof["peak_source"] = (f"{peak_src} ({name if peak_src == 'measured' else 'fallback ' + choice}"
                               f"{' x2 for FP8' if works[dom].kind == 'mxfp8' else ''})")
        roof["peak_choice"] = f"{choice}: {why}"

    # ---- cuBLAS on the same operands, for context (after the timed region) ----
    libctx = None
    if rank == 0 and not args.no_library_context:
        libctx = library_context(probs, stream, min(args.steps, 100), flush_buf, flush_each)
        st = g.gemm_last_status(sh)
        if st != g.GEMM_OK:
            raise g.GemmError(st, "library context")

    # ---- CPU baseline: the oracle as it stands, bounded sample, rank 0 at N=1 ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.default()
        plan = plan_oracle_sample(works, hosts, args.cpu_seconds)
        f, s = oracle_pass(works, hosts, plan)
        cpu = {"value": f / s / scale, "unit": unit, "cores": oracle.num_threads(),
               "kind": "oracle", "sample": sample_text(works, plan), "seconds": s}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "+".join(sorted({"bf16" if w.kind == "bf16" else "e4m3" for w in works})) + "->f32",
            "data": "synthetic (seeded; bf16 N(0,1)*0.5, MXFP8 quantised from N(0,1)"
                    + ("; MXFP8 scales passed in the tiled layout" if any(p.tiled for p in probs) else "")
                    + ")",
            "config": {"workload": workload_text(works),
                       "variant": args.variant,
                       "l2": ("512 MiB write before each launch of a workload whose inputs fit "
                              "in L2; its kernels' event time only" if any(flush_each)
                              else "operands larger than L2, no flush"),
                       "event_floor_us": event_floor_us,
                       "back_to_back_us": back_to_back_us,
                       "parallelism": f"replicas x{world} (no data-path collective)"},
            "roofline": roof,
            "kernels": kernels,
            "cpu_baseline": cpu,
            "library_context": libctx,
            "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": args.steps * len(probs),   # in the timed region (value)
            "device": {"name": torch.cuda.get_device_name(device),
                       "sm_count": torch.cuda.get_device_properties(device).multi_processor_count},
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    rank, world, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world)
        return run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
