"""Benchmark of the scaled-precision GEMM hot path on one GB300.

Default workload ``prefill`` (one "step"): the FP8 E4M3 row-scaled
linear_add layer at T in {1024, 4096, 8192} for the two weight shapes
(K=17408, N=5120) and (K=6144, N=5120), and the NVFP4 block-scaled layers at
the same T: linear_add at both weight shapes and linear_swiglu at (K=5120,
N=34816).  For each of the fifteen cases a step quantizes the bf16
activations (FP8: E4M3 codes with per-row scales; NVFP4: the global scale,
then E2M1 codes with blocked E4M3 scales) and runs the GEMM with its fused
epilogue (bf16 residual add, or SwiGLU over interleaved gate/up columns).
Weights are quantized once, outside the timed region, as a deployment does
offline.  L2 is flushed (a 512 MB write, read back) before every case,
outside the CUDA-event brackets; the reported time is the sum of the
bracketed segments.

The GEMMs go through the library's workspace entry points (a workspace of
spg_gemm_workspace_bytes per case, allocated once), so the route may split
the last partial wave along K where its cost model says that pays.

Metric: TFLOP/s = sum(2 T N K) / step time, plus each case's GEMM-only rate
and its fraction of the dense tensor peak of its format (FP8, or FP4 for
NVFP4), and the roofline of the longest GEMM of each format.

Other workloads (--workload): fp8_linear_add (the six FP8 cases alone),
fp8_swiglu (T in {1024, 4096}, K=5120, N=34816 and the plain-linear widths
14336/16384/34816), nvfp4 (linear_add and linear_swiglu at T in {256, 1024,
4096, 8192}), fp8_tensor (the per-tensor training shapes), decode
(linear_add at narrow T: FP8 T in {1, 16, 64, 128}, NVFP4 T in {1, 2, 4};
its roofline is the HBM copy peak).  ``--impl reference`` times the CPU
oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "scaled GEMM TFLOP/s and % of GB300 FP8/FP4 tensor peak at T=1024/4096/8192"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal dense ratios to bf16 (2.25 PF): fp8 4.5 PF, fp4 13.5 PF
NOMINAL_RATIO = {"fp8": 2.0, "fp4": 6.0, "bf16": 1.0}
L2_FLUSH_BYTES = 512 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return {"hbm_gbs": float(d.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
                    "bf16_tflops": float(d.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
                    "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained",
                                                         d.get("bf16_tflops", 1700.0))),
                    "source": "measured"}
        except Exception:
            pass
    return dict(FALLBACK_PEAKS, source="fallback")


# ------------------------------------------------------------ ranks
def job_throughput(ms_local, flops_per_rank, world, dist=None, device=None):
    """Whole-job throughput of a replica run (weak scaling): every rank does
    `flops_per_rank` of work and the job lasts as long as its slowest rank.
    Returns (the max over ranks of `ms_local`, all ranks' TFLOP/s)."""
    ms = float(ms_local)
    if dist is not None and world > 1:
        import torch
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, flops_per_rank * world / (ms * 1e-3) / 1e12


# ------------------------------------------------------------ workloads
def workload_cases(name):
    if name == "prefill":
        # The headline workload: FP8 row-scaled linear_add and NVFP4
        # linear_add / linear_swiglu at the three prefill widths, so one step
        # exercises both flavours of the metric.
        cases = workload_cases("fp8_linear_add")
        for T in (1024, 4096, 8192):
            cases += [dict(kind="nvfp4", T=T, K=17408, N=5120, epi="add"),
                      dict(kind="nvfp4", T=T, K=6144, N=5120, epi="add"),
                      dict(kind="nvfp4", T=T, K=5120, N=34816, epi="swiglu")]
        return cases
    if name == "fp8_linear_add":
        return [dict(kind="fp8", T=T, K=K, N=5120, epi="add", w_std=0.02)
                for T in (1024, 4096, 8192) for K in (17408, 6144)]
    if name == "fp8_swiglu":
        cases = [dict(kind="fp8", T=T, K=5120, N=34816, epi="swiglu", w_std=1.0) for T in (1024, 4096)]
        cases += [dict(kind="fp8", T=T, K=5120, N=N, epi="linear", w_std=1.0)
                  for T in (1024, 4096) for N in (14336, 16384, 34816)]
        return cases
    if name == "nvfp4":
        cases = []
        for T in (256, 1024, 4096, 8192):
            cases += [dict(kind="nvfp4", T=T, K=17408, N=5120, epi="add"),
                      dict(kind="nvfp4", T=T, K=6144, N=5120, epi="add"),
                      dict(kind="nvfp4", T=T, K=5120, N=34816, epi="swiglu")]
        return cases
    if name == "decode":
        # Narrow T (decode and small batches) at the linear_add widths: the
        # weights stream once, so these are HBM-bound (swapped FP8 tile with
        # the K split; NVFP4: the GEMV at T <= 2 or K <= 8192, else one-CTA
        # tiles with the K split inside clusters).
        cases = [dict(kind="fp8", T=T, K=K, N=5120, epi="add", w_std=0.02)
                 for T in (1, 16, 64, 128) for K in (17408, 6144)]
        cases += [dict(kind="nvfp4", T=T, K=K, N=5120, epi="add")
                  for T in (1, 2, 4, 16, 64, 128) for K in (17408, 6144)]
        return cases
    if name == "fp8_tensor":
        return [dict(kind="tensor", layout=l, M=M, N=N, K=K, batch=b) for (l, M, N, K, b) in [
            ("NT", 2048, 6912, 1536, 1), ("NT", 2048, 1536, 6912, 1), ("NN", 2048, 1536, 6912, 1),
            ("NN", 2048, 6912, 1536, 1), ("TN", 6912, 1536, 2048, 1), ("TN", 1536, 6912, 2048, 1),
            ("NT", 512, 512, 512, 1), ("NT", 4096, 4096, 4096, 1), ("NT", 8192, 8192, 8192, 1),
            ("NT", 64, 8192, 2048, 1), ("NT", 1024, 1536, 2048, 1), ("NT", 1024, 1024, 2048, 8),
            ("NT", 512, 512, 512, 64)]]
    raise SystemExit(f"unknown workload {name}")


def case_flops(c):
    if c["kind"] == "tensor":
        return 2.0 * c["M"] * c["N"] * c["K"] * c["batch"]
    return 2.0 * c["T"] * c["N"] * c["K"]


def case_bytes(c):
    """Algorithmic HBM bytes of the GEMM launch (inputs read once, output written once)."""
    if c["kind"] == "tensor":
        return c["batch"] * (c["M"] * c["K"] + c["N"] * c["K"] + 2 * c["M"] * c["N"]) + 8
    T, N, K = c["T"], c["N"], c["K"]
    n_out = N // 2 if c["epi"] == "swiglu" else N
    res = 2 * T * N if c["epi"] == "add" else 0
    if c["kind"] == "nvfp4":
        return T * K // 2 + N * K // 2 + (T + N) * K // 16 + 8 + 2 * T * n_out + res
    return T * K + N * K + 4 * (T + N) + 2 * T * n_out + res


def case_name(c):
    if c["kind"] == "tensor":
        return f"tensor_{c['layout']}_b{c['batch']}_{c['M']}x{c['N']}x{c['K']}"
    return f"{c['kind']}_{c['epi']}_T{c['T']}_K{c['K']}_N{c['N']}"


def gemm_source_hash():
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "scaled_precision_gemm_gb300", "csrc")
    for f in sorted(glob.glob(os.path.join(csrc, "gemm_*"))) + [os.path.join(csrc, "ptx.cuh")]:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(case):
    """DRAM bytes per launch recorded from ncu for this case, or None when no
    capture exists or the GEMM sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = gemm_source_hash()
    for line in open(path):
        parts = line.split()
        if len(parts) == 3 and not line.startswith("#") and parts[0] == case and parts[2] == cur:
            return int(parts[1])
    return None


# ------------------------------------------------------------ clocks
class ClockSampler:
    """Samples the SM clock and the clock-event reasons of the benchmarked GPU
    during the timed region with read-only NVML queries (ctypes) every 2 ms;
    falls back to nvidia-smi if NVML cannot be opened."""
    REASON_BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown",
                   0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, device_index=0):
        import threading
        self.samples = []
        self.reasons = set()
        self.stop_ev = threading.Event()
        self.thread = None
        self.max_mhz = None
        self.nvml = None
        self.handle = None
        self.device_index = device_index
        # optional per-sample record of the SM clock (the JSON line carries
        # the summary either way)
        self.path = os.environ.get("SPG_CLOCKS_CSV") or None
        try:
            self._open_nvml()
        except Exception:
            self.nvml = None

    def _open_nvml(self):
        import ctypes
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(self.device_index)
        ok = False
        uuid = str(getattr(props, "uuid", ""))
        for cand in (uuid, "GPU-" + uuid):
            if cand and lib.nvmlDeviceGetHandleByUUID(cand.encode(), ctypes.byref(h)) == 0:
                ok = True
                break
        if not ok:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            idx = int(vis.split(",")[self.device_index]) if vis and vis.split(",")[0].isdigit() \
                else self.device_index
            if lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) != 0:
                raise RuntimeError("no NVML handle")
        self.nvml, self.handle = lib, h
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def _poll(self):
        import ctypes
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self.stop_ev.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0:
                self.samples.append(float(clk.value))
            if self._reason_fn(self.handle, ctypes.byref(rs)) == 0:
                for bit, name in self.REASON_BITS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(0.002)

    def start(self):
        import threading
        if self.nvml is None:
            return
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()

    def stop(self):
        if self.nvml is None or self.thread is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.stop_ev.set()
        self.thread.join()
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"]}
        if self.path:
            try:
                os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
                with open(self.path, "w") as f:
                    f.write("sm_mhz\n" + "\n".join(str(v) for v in self.samples) + "\n")
            except OSError:
                pass
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": "NVML, 2 ms polling during the timed steps"}


# ------------------------------------------------------------ GPU arm
def run_gpu(args):
    import torch

    import scaled_precision_gemm_gb300 as spg
    from scaled_precision_gemm_gb300 import build as spg_build
    from synthetic_inputs import normal_bf16

    spg_build.build()
    spg.load_library()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    def to_dev_bf16(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    cases = workload_cases(args.workload)
    if args.case:
        cases = [c for c in cases if case_name(c) == args.case]
        if not cases:
            raise SystemExit(f"no case {args.case} in workload {args.workload}")
    # synthetic inputs, generated once per distinct shape (largest T, sliced)
    inputs = {}
    for c in cases:
        if c["kind"] == "tensor":
            key = ("tensor", c["layout"], c["M"], c["N"], c["K"], c["batch"])
            if key not in inputs:
                a_shape = (c["batch"], c["K"], c["M"]) if c["layout"][0] == "T" else (c["batch"], c["M"], c["K"])
                b_shape = (c["batch"], c["K"], c["N"]) if c["layout"][1] == "N" else (c["batch"], c["N"], c["K"])
                a = to_dev_bf16(normal_bf16(a_shape, seed=0))
                b = to_dev_bf16(normal_bf16(b_shape, seed=1))
                inputs[key] = (a, b)
            continue
        kx = ("x", c["K"])
        if kx not in inputs:
            tmax = max(cc["T"] for cc in cases if cc["kind"] != "tensor" and cc["K"] == c["K"])
            inputs[kx] = to_dev_bf16(normal_bf16((tmax, c["K"]), seed=0))
        kw = ("w", c["kind"], c["K"], c["N"])
        if kw not in inputs:
            w = to_dev_bf16(normal_bf16((c["N"], c["K"]), seed=1, std=c.get("w_std", 1.0)))
            if c["kind"] == "fp8":
                inputs[kw] = spg.quantize_fp8_rows(w)            # offline weight quantization
            else:
                gw = spg.nvfp4_global_scale(w)
                inputs[kw] = (*spg.quantize_nvfp4(w, gw), gw)
            del w
        kr = ("r", c["N"])
        if c["epi"] == "add" and kr not in inputs:
            tmax = max(cc["T"] for cc in cases if cc["kind"] != "tensor" and cc["N"] == c["N"])
            inputs[kr] = to_dev_bf16(normal_bf16((tmax, c["N"]), seed=2))
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_words = flush.view(torch.float32)
    scratch = torch.empty(4, dtype=torch.float32, device=dev)

    # Per case: preallocated buffers, quant(x, res) (activation quantization of
    # the given device activations) and gemm() (the GEMM with its fused
    # epilogue, reading what quant() wrote).  `launches` counts library kernels.
    class Case:
        pass

    prepared = []
    for c in cases:
        k = Case()
        k.c = c
        if c["kind"] == "tensor":
            a, b = inputs[("tensor", c["layout"], c["M"], c["N"], c["K"], c["batch"])]
            k.x, k.res = a, None
            ac = torch.empty(a.shape, dtype=torch.uint8, device=dev)
            bc = torch.empty(b.shape, dtype=torch.uint8, device=dev)
            sa = torch.empty(1, dtype=torch.float32, device=dev)
            sb = torch.empty(1, dtype=torch.float32, device=dev)
            k.out = torch.empty((c["batch"], c["M"], c["N"]), dtype=torch.bfloat16, device=dev)
            spg.quantize_fp8_tensor(b, bc, sb, scratch)   # weight-side operand, offline
            k.ws = spg.gemm_workspace("fp8_tensor", c["M"], c["N"], c["K"], "linear", c["batch"],
                                      device=dev)
            k.quant = lambda x, res, ac=ac, sa=sa: spg.quantize_fp8_tensor(x, ac, sa, scratch)
            k.gemm = lambda c=c, ac=ac, sa=sa, bc=bc, sb=sb, out=k.out, k=k: spg.fp8_tensor_gemm(
                c["layout"], ac, sa, bc, sb, c["M"], c["N"], c["K"], batch=c["batch"], out=out,
                workspace=k.ws)
            k.launches = 3
            prepared.append(k)
            continue
        T, K, N = c["T"], c["K"], c["N"]
        k.x = inputs[("x", K)][:T]
        n_out = N // 2 if c["epi"] == "swiglu" else N
        k.out = torch.empty((T, n_out), dtype=torch.bfloat16, device=dev)
        k.res = inputs[("r", N)][:T] if c["epi"] == "add" else None
        k.res_dev = k.res
        # The library's workspace (allocated once, like any deployment would):
        # lets the route split the last partial wave along K where that pays.
        k.ws = spg.gemm_workspace("fp8_rowscaled" if c["kind"] == "fp8" else "nvfp4", T, N, K,
                                  c["epi"], device=dev)
        if c["kind"] == "fp8":
            W, sw = inputs[("w", "fp8", K, N)]
            A = torch.empty((T, K), dtype=torch.uint8, device=dev)
            sa = torch.empty((T,), dtype=torch.float32, device=dev)
            k.quant = lambda x, res, A=A, sa=sa, k=k: (spg.quantize_fp8_rows(x, A, sa),
                                                       setattr(k, "res_dev", res))
            k.gemm = lambda A=A, sa=sa, W=W, sw=sw, k=k, epi=c["epi"]: spg.fp8_rowscaled_gemm(
                A, sa, W, sw, residual=k.res_dev, epilogue=epi, out=k.out, workspace=k.ws)
            k.launches = 2
        else:
            Wc, sfW, gW = inputs[("w", "nvfp4", K, N)]
            A = torch.empty((T, K // 2), dtype=torch.uint8, device=dev)
            sfA = torch.empty((spg.nvfp4_sf_bytes(T, K),), dtype=torch.uint8, device=dev)
            gA = torch.empty((1,), dtype=torch.float32, device=dev)

            def quant(x, res, A=A, sfA=sfA, gA=gA, k=k):
                spg.quantize_nvfp4_act(x, gA, A, sfA, scratch)
                k.res_dev = res
            k.quant = quant
            k.gemm = lambda A=A, sfA=sfA, gA=gA, Wc=Wc, sfW=sfW, gW=gW, k=k, epi=c["epi"]: \
                spg.nvfp4_gemm(A, sfA, gA, Wc, sfW, gW, residual=k.res_dev, epilogue=epi,
                               out=k.out, workspace=k.ws)
            # one quantizer kernel (one CTA, or one cluster) for activations of
            # up to 512 Ki elements, else amax + quantize (plus one memset);
            # then the GEMM
            k.launches = 2 if T * K <= 512 * 1024 else 3
        prepared.append(k)

    # Warm the library (first-call set-up: shared-memory limits, device error
    # word) eagerly, then capture each case's activation quantization and GEMM
    # as two CUDA graphs so the timed region measures device time only.
    for k in prepared:
        k.quant(k.x, k.res)
        k.gemm()
    torch.cuda.synchronize()
    use_graphs = not args.no_graphs
    if use_graphs:
        for k in prepared:
            k.g_quant = torch.cuda.CUDAGraph()
            with torch.cuda.graph(k.g_quant):
                k.quant(k.x, k.res)
            k.g_gemm = torch.cuda.CUDAGraph()
            with torch.cuda.graph(k.g_gemm):
                k.gemm()
        torch.cuda.synchronize()

    def one_step(timed):
        """Run every case once; returns (segment events, gemm-only events, launches)."""
        seg, gem, launches = [], [], 0
        for k in prepared:
            # L2 flush, outside the brackets: write a buffer larger than L2,
            # then read it back so the lines left behind are clean (the GEMM
            # is not charged for writing the flush's dirty lines back).
            flush.zero_()
            flush_words.sum()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e2 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if use_graphs:
                k.g_quant.replay()
            else:
                k.quant(k.x, k.res)
            e1.record(stream)
            if use_graphs:
                k.g_gemm.replay()
            else:
                k.gemm()
            e2.record(stream)
            seg.append((e0, e2))
            gem.append((e1, e2))
            launches += k.launches
        return seg, gem, launches

    for _ in range(args.warmup):
        one_step(False)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    all_seg, all_gemm, launches = [], [], 0
    for _ in range(args.steps):
        s, g, nl = one_step(True)
        all_seg.append(s)
        all_gemm.append(g)
        launches += nl
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()

    step_ms = [sum(a.elapsed_time(b) for a, b in s) for s in all_seg]
    flops_step = sum(case_flops(k.c) for k in prepared)
    total_ms, value = job_throughput(sum(step_ms), flops_step * args.steps, world, dist, dev)

    peaks = load_peaks()
    per_case = []
    for i, k in enumerate(prepared):
        c = k.c
        gms = statistics.median(all_gemm[k][i][0].elapsed_time(all_gemm[k][i][1])
                                for k in range(args.steps))
        sms = statistics.median(all_seg[k][i][0].elapsed_time(all_seg[k][i][1])
                                for k in range(args.steps))
        dtype = "fp4" if c["kind"] == "nvfp4" else "fp8"
        peak = peaks["bf16_tflops"] * NOMINAL_RATIO[dtype]
        tf = case_flops(c) / (gms * 1e-3) / 1e12
        per_case.append({"case": case_name(c), "gemm_us": round(gms * 1e3, 2),
                         "step_us": round(sms * 1e3, 2), "gemm_tflops": round(tf, 1),
                         "frac_of_peak": round(tf / peak, 4),
                         "gemm_gbs": round(case_bytes(c) / (gms * 1e-3) / 1e9, 1)})
    # Dominant kernel: the case with the longest GEMM; the same figures for
    # the longest GEMM of each flavour (FP8 against the FP8 peak, NVFP4
    # against the FP4 peak).
    def roofline_of(i):
        dc = prepared[i].c
        dtype = "fp4" if dc["kind"] == "nvfp4" else "fp8"
        dom_ms = per_case[i]["gemm_us"] * 1e-3
        traffic = recorded_traffic(case_name(dc))
        if args.workload == "decode":
            # weight-streaming cases: bytes against the HBM copy peak
            ach_gbs = case_bytes(dc) / (dom_ms * 1e-3) / 1e9
            return {"bound": "hbm", "kernel": case_name(dc), "achieved": round(ach_gbs, 1),
                    "peak": round(peaks["hbm_gbs"], 1), "unit": "GB/s",
                    "frac": round(ach_gbs / peaks["hbm_gbs"], 4), "traffic": traffic,
                    "peak_source": f"{peaks['source']} HBM copy {peaks['hbm_gbs']} GB/s",
                    "algorithmic_bytes": case_bytes(dc)}
        dom_peak = peaks["bf16_tflops"] * NOMINAL_RATIO[dtype]
        achieved = case_flops(dc) / (dom_ms * 1e-3) / 1e12
        return {"bound": "tensor", "kernel": case_name(dc), "achieved": round(achieved, 1),
                "peak": round(dom_peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / dom_peak, 4), "traffic": traffic,
                "peak_source": f"{peaks['source']} bf16 burst {peaks['bf16_tflops']} TFLOP/s x "
                               f"nominal {dtype}:bf16 ratio {NOMINAL_RATIO[dtype]}",
                "algorithmic_bytes": case_bytes(dc), "algorithmic_flops": case_flops(dc)}

    dom_i = max(range(len(per_case)), key=lambda i: per_case[i]["gemm_us"])
    roofline = roofline_of(dom_i)
    by_flavour = {}
    for flav, kinds in (("fp8", ("fp8", "tensor")), ("fp4", ("nvfp4",))):
        idx = [i for i, k in enumerate(prepared) if k.c["kind"] in kinds]
        if idx and args.workload != "decode":
            r = roofline_of(max(idx, key=lambda i: per_case[i]["gemm_us"]))
            fl = sum(case_flops(prepared[i].c) for i in idx)
            us = sum(per_case[i]["gemm_us"] for i in idx)
            r["all_cases_tflops"] = round(fl / (us * 1e-6) / 1e12, 1)
            r["all_cases_frac"] = round(r["all_cases_tflops"] / r["peak"], 4)
            by_flavour[flav] = r

    # ---------------- e2e: host buffers through the public API
    e2e = None if args.no_e2e else run_e2e(args, spg, torch, dev, prepared, inputs, dist, world)

    dtype_line = {"nvfp4": "e2m1", "decode": "e4m3/e2m1",
                  "prefill": "e4m3/e2m1"}.get(args.workload, "e4m3")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_line, "data": "synthetic",
        "config": {"workload": args.workload,
                   "cases": [case_name(k.c) for k in prepared],
                   "step": "activation quantization + GEMM with fused epilogue per case",
                   "l2": "flushed (512 MB write, then read back so no dirty lines remain) "
                         "before every case, outside the timed brackets",
                   "api": "workspace entry points (workspace sized by spg_gemm_workspace_bytes, "
                          "allocated once; the route may split the last partial wave along K)",
                   "launch": "CUDA graph replay per case" if use_graphs else "eager",
                   "inputs": "bf16 N(0,1) activations/residual; weights N(0,0.02) for FP8 "
                             "linear_add, N(0,1) otherwise (splitmix64 "
                             "Box-Muller, seeds 0/1/2); weights quantized once offline"},
        "roofline": roofline,
        "roofline_by_flavour": by_flavour,
        "per_case": per_case,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
        "wall_s_timed": round(wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.workload, rows=args.cpu_rows)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def bind_host_near_gpu(torch, dev):
    """Run this process on the CPUs the GPU's PCI device reports as local
    (sysfs local_cpulist), so the pinned host buffers allocated next are
    first touched, hence placed, in that NUMA node's memory.  Returns what
    was done, for the JSON line; leaves the affinity alone when the device
    or its CPU list cannot be read or shares no CPU with the allowed set."""
    props = torch.cuda.get_device_properties(dev)
    try:
        bus = "%04x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
    except AttributeError:
        return {"bound": False, "why": "no PCI id in the device properties"}
    base = os.path.join("/sys/bus/pci/devices", bus)
    try:
        text = open(os.path.join(base, "local_cpulist")).read().strip()
        node = open(os.path.join(base, "numa_node")).read().strip()
    except OSError:
        return {"bound": False, "pci": bus, "why": "no local_cpulist"}
    local = set()
    for part in text.split(","):
        if "-" in part:
            a, b = part.split("-")
            local.update(range(int(a), int(b) + 1))
        elif part:
            local.add(int(part))
    allowed = os.sched_getaffinity(0)
    use = allowed & local
    if not use:
        return {"bound": False, "pci": bus, "numa_node": node, "why": "no allowed local CPU"}
    if use != allowed:
        try:
            os.sched_setaffinity(0, use)
        except OSError as e:
            return {"bound": False, "pci": bus, "numa_node": node, "why": f"sched_setaffinity: {e}"}
    return {"bound": True, "pci": bus, "numa_node": node, "cpus": len(use),
            "changed": use != allowed}


def run_e2e(args, spg, torch, dev, prepared, inputs, dist=None, world=1):
    """Same workload through the public API with HOST buffers: per case the
    bf16 activations (and residual) are copied from pinned host memory, the
    step runs on those device copies, and the bf16 output is copied back to
    pinned host memory; all copies are inside the timed region.  Copies run
    on two copy streams, ordered by events, so case i+1's inputs travel
    while case i computes and case i-1's output travels back."""
    h2d = d2h = 0
    prev_affinity = os.sched_getaffinity(0)
    host_affinity = bind_host_near_gpu(torch, dev)
    for k in prepared:
        k.x_host = k.x.cpu().pin_memory()
        k.res_host = None if k.res is None else k.res.cpu().pin_memory()
        k.out_host = torch.empty(k.out.shape, dtype=k.out.dtype).pin_memory()
        k.out_host.zero_()  # first touch here, in the bound node's memory
        k.x_d = torch.empty_like(k.x)
        k.res_d = None if k.res is None else torch.empty_like(k.res)
        h2d += k.x_host.numel() * 2 + (0 if k.res_host is None else k.res_host.numel() * 2)
        d2h += k.out_host.numel() * 2
    try:
        os.sched_setaffinity(0, prev_affinity)  # the pages stay where they were placed
    except OSError:
        pass
    compute = torch.cuda.current_stream(dev)
    s_h2d = torch.cuda.Stream(dev)
    s_d2h = torch.cuda.Stream(dev)
    n = len(prepared)
    ev = lambda: torch.cuda.Event()
    done_compute = [None] * n
    done_d2h = [None] * n

    def issue_h2d(i):
        k = prepared[i]
        if done_compute[i] is not None:          # buffer still read by the previous step
            s_h2d.wait_event(done_compute[i])
        with torch.cuda.stream(s_h2d):
            k.x_d.copy_(k.x_host, non_blocking=True)
            if k.res_d is not None:
                k.res_d.copy_(k.res_host, non_blocking=True)
        e = ev()
        e.record(s_h2d)
        return e

    def e2e_step():
        ready = issue_h2d(0)
        for i, k in enumerate(prepared):
            nxt = issue_h2d(i + 1) if i + 1 < n else None
            compute.wait_event(ready)
            if done_d2h[i] is not None:          # output buffer still being read back
                compute.wait_event(done_d2h[i])
            k.quant(k.x_d, k.res_d)
            k.gemm()
            done_compute[i] = ev()
            done_compute[i].record(compute)
            s_d2h.wait_event(done_compute[i])
            with torch.cuda.stream(s_d2h):
                k.out_host.copy_(k.out, non_blocking=True)
            done_d2h[i] = ev()
            done_d2h[i].record(s_d2h)
            ready = nxt

    e2e_step()
    torch.cuda.synchronize()
    reps = max(1, min(args.steps, 3))
    t0 = time.perf_counter()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    for st in (s_h2d, s_d2h):      # copies start after the opening event
        st.wait_stream(compute)
    for _ in range(reps):
        e2e_step()
    for st in (s_h2d, s_d2h):
        compute.wait_stream(st)
    e1.record(compute)
    torch.cuda.synchronize()
    wall_ms = (time.perf_counter() - t0) * 1e3 / reps
    for k in prepared:          # restore the device-resident inputs
        k.quant(k.x, k.res)
    flops = sum(case_flops(k.c) for k in prepared)
    ms, value = job_throughput(e0.elapsed_time(e1) / reps, flops, world, dist, dev)
    return {"value": round(value, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 3), "wall_ms_per_step": round(wall_ms, 3),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "copies": "two copy streams overlapping compute (pinned host buffers)",
            "host_affinity": host_affinity}


# ------------------------------------------------------------ CPU oracle
_CPU_INPUTS = {}


def _cpu_case_inputs(c, rows):
    """Oracle-side inputs of one case (weights quantized once, cached)."""
    import oracle
    from synthetic_inputs import normal_bf16

    key = (case_name(c), rows)
    if key in _CPU_INPUTS:
        return _CPU_INPUTS[key]
    if c["kind"] == "tensor":
        K, N = c["K"], c["N"]
        B, sB = oracle.quantize_fp8_tensor(normal_bf16((N, K), seed=1))
        d = dict(x=normal_bf16((rows, K), seed=0), B=B, sB=sB)
    else:
        K, N = c["K"], c["N"]
        w = normal_bf16((N, K), seed=1, std=c.get("w_std", 1.0))
        d = dict(x=normal_bf16((rows, K), seed=0),
                 res=normal_bf16((rows, N), seed=2) if c["epi"] == "add" else None)
        if c["kind"] == "fp8":
            d["W"], d["sw"] = oracle.quantize_fp8_rows(w)
        else:
            d["gw"] = oracle.nvfp4_global_scale(w)
            d["W"], d["sfW"] = oracle.quantize_nvfp4(w, d["gw"])
    _CPU_INPUTS[key] = d
    return d


def cpu_baseline(workload, rows=32):
    """The oracle as it stands, on the host cores, on a bounded sample of the
    workload: for every case, the activation quantizer and the exact-integer
    GEMM with its epilogue on `rows` activation rows (all N columns).  Weight
    quantization is offline and untimed, as on the GPU side."""
    import oracle

    oracle.build()
    cases = workload_cases(workload)
    cores = os.cpu_count() or 1
    done_flops = 0.0
    t_total = 0.0
    for c in cases:
        d = _cpu_case_inputs(c, rows)
        t0 = time.perf_counter()
        if c["kind"] == "tensor":
            A, sA = oracle.quantize_fp8_tensor(d["x"])
            oracle.fp8_tensor_gemm("NT", A, sA, d["B"], d["sB"], rows, c["N"], c["K"])
        elif c["kind"] == "fp8":
            A, sa = oracle.quantize_fp8_rows(d["x"])
            oracle.fp8_rowscaled_gemm(A, sa, d["W"], d["sw"], d["res"], c["epi"])
        else:
            ga = oracle.nvfp4_global_scale(d["x"])
            A, sfA = oracle.quantize_nvfp4(d["x"], ga)
            oracle.nvfp4_gemm(A, sfA, ga, d["W"], d["sfW"], d["gw"], d["res"], c["epi"])
        t_total += time.perf_counter() - t0
        done_flops += 2.0 * rows * c["N"] * c["K"]
    return {"value": round(done_flops / t_total / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{rows} activation rows (all N) of each of the {len(cases)} cases of "
                      f"{workload}: activation quantization + exact GEMM + epilogue; "
                      f"{t_total:.1f} s of CPU work on {cores} threads"}


def run_reference(args):
    """Reference arm: the CPU oracle timed on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    per_step = []
    rows = args.ref_rows
    for _ in range(args.warmup):
        cpu_baseline(args.workload, rows=rows)
    base = None
    flops = work_s = 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        base = cpu_baseline(args.workload, rows=rows)
        per_step.append(time.perf_counter() - t0)
        flops += sum(2.0 * rows * c["N"] * c["K"] * c.get("batch", 1)
                     for c in workload_cases(args.workload))
        work_s += per_step[-1]
    value = round(flops / work_s / 1e12, 6)
    base["value"] = value
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * sum(per_step) / len(per_step), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int64 exact dot products, fp64 scales", "data": "synthetic",
            "config": {"workload": args.workload}, "impl": "reference",
            "cpu_baseline": dict(base),
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_host_overhead(args):
    """Host time per eager GEMM call through the C ABI (ctypes, arguments
    marshalled once): the library's argument checks, route selection,
    tensor-map set-up and the launch itself, with the tensor-map cache on and
    off.  Calls are enqueued in batches of 100 (each batch well inside the
    launch queue) and the device is synchronised between batches, outside the
    host timer."""
    import ctypes
    import torch

    import scaled_precision_gemm_gb300 as spg
    from scaled_precision_gemm_gb300 import build as spg_build

    spg_build.build()
    lib = spg.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    vp = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    out = {}
    shapes = [("fp8", 16, 17408, 5120), ("fp8", 8192, 17408, 5120),
              ("nvfp4", 1, 17408, 5120), ("nvfp4", 8192, 17408, 5120)]
    for kind, T, K, N in shapes:
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        kbytes = K if kind == "fp8" else K // 2
        A = torch.randint(0, 0x70, (T, kbytes), dtype=torch.uint8, device=dev, generator=g)
        W = torch.randint(0, 0x70, (N, kbytes), dtype=torch.uint8, device=dev, generator=g)
        res = torch.zeros((T, N), dtype=torch.bfloat16, device=dev)
        Y = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
        ws = spg.gemm_workspace("fp8_rowscaled" if kind == "fp8" else "nvfp4", T, N, K, "add",
                                device=dev)
        wsn = 0 if ws is None else ws.numel()
        if kind == "fp8":
            sa = torch.full((T,), 1e-3, device=dev)
            sw = torch.full((N,), 1e-3, device=dev)
            fn = lib.fp8_rowscaled_gemm_ws
            cargs = (vp(A), vp(sa), vp(W), vp(sw), None, None, vp(res), vp(Y), T, N, K, 1,
                     vp(ws), wsn, stream)
        else:
            sfA = torch.full((spg.nvfp4_sf_bytes(T, K),), 0x38, dtype=torch.uint8, device=dev)
            sfW = torch.full((spg.nvfp4_sf_bytes(N, K),), 0x38, dtype=torch.uint8, device=dev)
            g1 = torch.ones(4, device=dev)
            fn = lib.nvfp4_gemm_ws
            cargs = (vp(A), vp(sfA), vp(g1), vp(W), vp(sfW), vp(g1), None, None, vp(res), vp(Y),
                     T, N, K, 1, vp(ws), wsn, stream)
        name = f"{kind}_add_T{T}_K{K}_N{N}"
        route = spg.select_route("fp8_rowscaled" if kind == "fp8" else "nvfp4", T, N, K, "add",
                                 workspace=True)
        res_d = {"variant": route["variant"], "swap_ab": route["swap_ab"]}
        for mode in ("cache_on", "cache_off"):
            lib.spg_debug_set_tmap_cache(1 if mode == "cache_on" else 0)
            for _ in range(20):
                assert fn(*cargs) == 0
            torch.cuda.synchronize()
            per = []
            for _ in range(10):
                t0 = time.perf_counter()
                for _ in range(100):
                    fn(*cargs)
                per.append((time.perf_counter() - t0) / 100 * 1e6)
                torch.cuda.synchronize()
            res_d[mode + "_us"] = round(statistics.median(per), 2)
        lib.spg_debug_set_tmap_cache(1)
        out[name] = res_d
    # the cost of the ctypes call itself: a host-only entry point
    n0 = time.perf_counter()
    for _ in range(10000):
        lib.spg_version()
    out["ctypes_call_floor_us"] = round((time.perf_counter() - n0) / 10000 * 1e6, 3)
    print(json.dumps({"host_overhead": out}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="spg", choices=["spg", "reference"])
    ap.add_argument("--workload", default="prefill",
                    choices=["prefill", "fp8_linear_add", "fp8_swiglu", "nvfp4", "fp8_tensor",
                             "decode"])
    ap.add_argument("--cpu-rows", type=int, default=32,
                    help="activation rows per case in the CPU-oracle baseline sample")
    ap.add_argument("--ref-rows", type=int, default=4,
                    help="activation rows per case in each step of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graphs", action="store_true",
                    help="launch eagerly in the timed region instead of replaying CUDA graphs")
    ap.add_argument("--case", default=None, help="run only this case of the workload")
    ap.add_argument("--host-overhead", action="store_true",
                    help="only measure host time per eager GEMM call (tensor-map cache on/off)")
    args = ap.parse_args()
    if args.host_overhead:
        run_host_overhead(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
