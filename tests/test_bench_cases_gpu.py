"""Every case the benchmark times, compared with the CPU oracle in the launch
configuration the benchmark uses.

The cases come from ``bench.workload_cases`` itself (every workload), so a
case added to the benchmark is covered here by construction.  Each GEMM runs
through the workspace entry point with a workspace of the size the library
asks for, exactly as the benchmark calls it, so the route under test is the
one that was timed: the persistent schedule over all tiles, the grouped
raster, the split of the last partial wave (along K, with its per-chunk
finish) and, at narrow T, the swapped tile or the GEMV.

Inputs are the benchmark's synthetic tensors (same shapes, distributions and
seeds), quantized by the ORACLE; the GPU GEMM gets those codes and scales.
Outputs are checked on sampled rows (every N column) against
|y - ref| <= 8e-3 |ref| + 1e-3 rms(ref): rows 0, 1, 127, 128, 255, 256, the
last 256 rows' edges, and one row of every 256-row block, so every pair
tile -- including those of the split last wave -- is sampled.  Output and
workspace sit between guard bands that must stay untouched, and the output is
prefilled with NaN so an unwritten element fails.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
import scaled_precision_gemm_gb300 as spg
from synthetic_inputs import normal_bf16
from tests.gpu_common import DEV, cuda, cuda_bf16, to_f64
from tests.helpers import assert_within_tol, sf_rowmajor_to_blocked

pytestmark = pytest.mark.gpu
GUARD = 256
WS_FILL = 0x5A
WORKLOADS = ("prefill", "fp8_linear_add", "fp8_swiglu", "nvfp4", "decode", "fp8_tensor")


def _all_cases():
    seen, out = set(), []
    for wl in WORKLOADS:
        for c in bench.workload_cases(wl):
            name = bench.case_name(c)
            if name not in seen:
                seen.add(name)
                out.append(c)
    return out


# grouped by operand shape so the cached inputs below are reused
CASES = sorted(_all_cases(), key=lambda c: (c["kind"] == "tensor", c.get("K", 0), c.get("N", 0),
                                            c["kind"], c.get("T", 0)))
_CACHE = {}
_CACHE_LIMIT = 3 << 30


def _nbytes(v):
    if isinstance(v, np.ndarray):
        return v.nbytes
    if isinstance(v, (tuple, list)):
        return sum(_nbytes(e) for e in v)
    return 0


def _cached(key, make):
    """Host inputs, generated once and kept while they fit in a few GB."""
    if key not in _CACHE:
        v = make()
        while _CACHE and sum(_nbytes(e) for e in _CACHE.values()) + _nbytes(v) > _CACHE_LIMIT:
            _CACHE.pop(next(iter(_CACHE)))
        _CACHE[key] = v
    return _CACHE[key]


def sample_rows(T, seed=0):
    if T <= 160:
        return np.arange(T, dtype=np.int64)
    rows = {0, 1, 127, 128, 255, 256, T - 256, T - 129, T - 128, T - 1, T // 2}
    rng = np.random.default_rng(seed + T)
    for b0 in range(0, T, 256):
        rows.add(int(rng.integers(b0, min(T, b0 + 256))))
    return np.array(sorted(r for r in rows if 0 <= r < T), np.int64)


def _guarded(n, dtype, fill):
    buf = torch.full((n + 2 * GUARD,), fill, dtype=dtype, device=DEV)
    return buf, buf[GUARD:GUARD + n]


def _check_guards(buf, fill_ok):
    g = torch.cat([buf[:GUARD], buf[-GUARD:]])
    assert fill_ok(g), "write outside the buffer"


def _workspace(kind, T, N, K, epi, batch=1):
    n = spg.gemm_workspace_bytes(kind, T, N, K, epi, batch)
    if n <= 0:
        return None, None
    buf, ws = _guarded(n, torch.uint8, WS_FILL)
    return buf, ws


def _out(T, n_out, batch=1):
    buf, flat = _guarded(batch * T * n_out, torch.bfloat16, float("nan"))
    view = flat.view(batch, T, n_out) if batch > 1 else flat.view(T, n_out)
    return buf, view


def _finish(out_buf, ws_buf):
    torch.cuda.synchronize()
    _check_guards(out_buf, lambda g: bool(torch.isnan(g.float()).all()))
    if ws_buf is not None:
        _check_guards(ws_buf, lambda g: bool((g == WS_FILL).all()))
    assert spg.last_device_error() == 0


def _x(K, T_max):
    return _cached(("x", K, T_max), lambda: normal_bf16((T_max, K), seed=0))


def _t_max(c):
    return max(cc["T"] for cc in CASES if cc["kind"] == c["kind"] and cc["K"] == c["K"])


def _res(c):
    if c["epi"] != "add":
        return None
    t_max = max(cc["T"] for cc in CASES if cc["kind"] != "tensor" and cc["N"] == c["N"])
    return _cached(("r", c["N"], t_max), lambda: normal_bf16((t_max, c["N"]), seed=2))[:c["T"]]


def run_fp8_case(c):
    T, K, N, epi = c["T"], c["K"], c["N"], c["epi"]
    x = _x(K, _t_max(c))[:T]
    A, sa = oracle.quantize_fp8_rows(x)
    W, sw = _cached(("wfp8", K, N, c.get("w_std", 1.0)), lambda: oracle.quantize_fp8_rows(
        normal_bf16((N, K), seed=1, std=c.get("w_std", 1.0))))
    res = _res(c)
    n_out = N // 2 if epi == "swiglu" else N
    ob, y = _out(T, n_out)
    wb, ws = _workspace("fp8_rowscaled", T, N, K, epi)
    spg.fp8_rowscaled_gemm(cuda(A), cuda(sa), cuda(W), cuda(sw),
                           residual=None if res is None else cuda_bf16(np.ascontiguousarray(res)),
                           epilogue=epi, out=y, workspace=ws)
    _finish(ob, wb)
    rows = sample_rows(T)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, epi, rows=rows)
    return to_f64(y[torch.from_numpy(rows).to(DEV)]), ref


def run_nvfp4_case(c):
    T, K, N, epi = c["T"], c["K"], c["N"], c["epi"]
    x = np.ascontiguousarray(_x(K, _t_max(c))[:T])
    gA = oracle.nvfp4_global_scale(x)
    A, sfA = oracle.quantize_nvfp4(x, gA)

    def make_w():
        w = normal_bf16((N, K), seed=1, std=c.get("w_std", 1.0))
        gW = oracle.nvfp4_global_scale(w)
        Wc, sfW = oracle.quantize_nvfp4(w, gW)
        return Wc, sfW, gW, sf_rowmajor_to_blocked(sfW, N, K)

    Wc, sfW, gW, sfW_blocked = _cached(("wnv", K, N), make_w)
    res = _res(c)
    n_out = N // 2 if epi == "swiglu" else N
    ob, y = _out(T, n_out)
    wb, ws = _workspace("nvfp4", T, N, K, epi)
    spg.nvfp4_gemm(cuda(A), cuda(sf_rowmajor_to_blocked(sfA, T, K)),
                   torch.tensor([gA], dtype=torch.float32, device=DEV), cuda(Wc), cuda(sfW_blocked),
                   torch.tensor([gW], dtype=torch.float32, device=DEV),
                   residual=None if res is None else cuda_bf16(np.ascontiguousarray(res)),
                   epilogue=epi, out=y, workspace=ws)
    _finish(ob, wb)
    rows = sample_rows(T)
    ref = oracle.nvfp4_gemm(A, sfA, gA, Wc, sfW, gW, res, epi, rows=rows)
    return to_f64(y[torch.from_numpy(rows).to(DEV)]), ref


def run_tensor_case(c):
    layout, M, N, K, batch = c["layout"], c["M"], c["N"], c["K"], c["batch"]
    a_shape = (batch, K, M) if layout[0] == "T" else (batch, M, K)
    b_shape = (batch, K, N) if layout[1] == "N" else (batch, N, K)
    A, sA = oracle.quantize_fp8_tensor(normal_bf16(a_shape, seed=0))
    B, sB = oracle.quantize_fp8_tensor(normal_bf16(b_shape, seed=1))
    A, B = A.reshape(-1), B.reshape(-1)
    ob, y = _out(M, N, batch)
    wb, ws = _workspace("fp8_tensor", M, N, K, "linear", batch)
    spg.fp8_tensor_gemm(layout, cuda(A), torch.tensor([sA], dtype=torch.float32, device=DEV),
                        cuda(B), torch.tensor([sB], dtype=torch.float32, device=DEV), M, N, K,
                        batch=batch, out=y, workspace=ws)
    _finish(ob, wb)
    rows = sample_rows(M)
    ref = oracle.fp8_tensor_gemm(layout, A, sA, B, sB, M, N, K, batch=batch, rows=rows)
    yy = to_f64(y.view(batch, M, N)[:, torch.from_numpy(rows).to(DEV), :])
    return yy, ref


@pytest.mark.parametrize("case", CASES, ids=[bench.case_name(c) for c in CASES])
def test_bench_case_matches_oracle(case):
    if case["kind"] == "fp8":
        y, ref = run_fp8_case(case)
    elif case["kind"] == "nvfp4":
        y, ref = run_nvfp4_case(case)
    else:
        y, ref = run_tensor_case(case)
    assert not np.isnan(y).any(), "unwritten output element"
    assert_within_tol(y, ref, bench.case_name(case))
