"""Workspace entry points (K split of the last partial wave of two-SM tiles)
against the CPU oracle.

The split changes only the order of the fp32 sums, so the bar is the same
element-wise tolerance as for the plain route.  Besides parity: the result
repeats bit for bit (each chunk's last piece adds all pieces in split order,
whatever order they arrive in), the workspace needs no initialisation and is
left with its counters at zero, nothing is written outside it, a CUDA graph
replays it, and a workspace that is too small falls back to the plain route.
"""
import numpy as np
import pytest
import torch

import oracle
import scaled_precision_gemm_gb300 as spg
from synthetic_inputs import normal_bf16, random_codes
from tests.gpu_common import DEV, cuda, cuda_bf16, to_f64
from tests.helpers import assert_within_tol, sf_rowmajor_to_blocked

pytestmark = pytest.mark.gpu
GUARD = 256
PATTERN = 0xA5


@pytest.fixture(params=["auto", "2sm", "2sm192", "2sm160", "2sm128"])
def variant(request, monkeypatch):
    """Pair tile width; the K split is forced for the last partial wave."""
    monkeypatch.setenv("SPG_FORCE_TAIL", "k")
    if request.param == "auto":
        monkeypatch.delenv("SPG_FORCE_VARIANT", raising=False)
    else:
        monkeypatch.setenv("SPG_FORCE_VARIANT", request.param)
    return request.param


def workspace_for(kind, T, N, K, epi="linear", batch=1, fill=PATTERN, exact=True):
    """Workspace of the size the library asks for (pattern-filled, never
    zeroed) between two guard bands; returns (whole buffer, workspace view,
    route).  exact=False: the size may cover other routes (the per-tensor
    GEMM's size covers both B layouts), so the counters are not located."""
    r = spg.select_route(kind, T, N, K, epi, batch, workspace=True)
    n = spg.gemm_workspace_bytes(kind, T, N, K, epi, batch)
    if exact:
        assert n == r["workspace_bytes"]
    else:
        assert n >= r["workspace_bytes"]
        r = dict(r, split_k=1)
    buf = torch.full((n + 2 * GUARD,), fill, dtype=torch.uint8, device=DEV)
    return buf, buf[GUARD:GUARD + n], r


def check_workspace(buf, n, r, epi="linear"):
    g = torch.cat([buf[:GUARD], buf[GUARD + n:]])
    assert bool((g == PATTERN).all()), "write outside the workspace"
    if r["split_k"] > 1:
        # every completed call leaves the arrival counters at zero
        cw = 64 if epi == "swiglu" else 32
        counter_bytes = 2 * 4 * (r["block_n"] // cw) * 8  # per tile: CTA x quarter x chunk
        per_tile = r["split_k"] * 2 * 128 * r["block_n"] * 4 + counter_bytes
        tail_tiles = n // per_tile
        assert tail_tiles * per_tile == n
        counters = buf[GUARD + n - counter_bytes * tail_tiles:GUARD + n]
        assert bool((counters == 0).all()), "arrival counters not reset"


def fp8_inputs(T, N, K, seed, w_std=1.0):
    A, sa = oracle.quantize_fp8_rows(normal_bf16((T, K), seed=seed))
    W, sw = oracle.quantize_fp8_rows(normal_bf16((N, K), seed=seed + 1, std=w_std))
    return A, sa, W, sw


def run_fp8_ws(A, sa, W, sw, res, epi, ws, bias=None, bias_scale=None):
    y = spg.fp8_rowscaled_gemm(cuda(A), cuda(sa), cuda(W), cuda(sw),
                               residual=None if res is None else cuda_bf16(res), epilogue=epi,
                               bias=bias, bias_scale=bias_scale, workspace=ws)
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    return y


# ------------------------------------------------------------------- FP8
@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
@pytest.mark.parametrize("T,N,K", [(1, 16, 1024), (64, 528, 4096), (65, 264, 1040),
                                   (200, 272, 2304), (257, 784, 1296), (520, 1040, 1296)])
def test_fp8_splitk_ragged(T, N, K, epi, variant):
    A, sa, W, sw = fp8_inputs(T, N, K, seed=T + N + K)
    res = normal_bf16((T, N), seed=3) if epi == "add" else None
    buf, ws, r = workspace_for("fp8_rowscaled", T, N, K, epi)
    if epi == "swiglu" and N % 16:
        with pytest.raises(spg.SpgError, match="UNSUPPORTED_SHAPE"):
            run_fp8_ws(A, sa, W, sw, res, epi, ws)
        return
    y = run_fp8_ws(A, sa, W, sw, res, epi, ws)
    check_workspace(buf, ws.numel(), r, epi)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, epi)
    assert_within_tol(to_f64(y), ref, f"fp8 split-K {epi} {T}x{N}x{K} ({r['split_k']} pieces)")


def test_fp8_splitk_taken_for_narrow_t(monkeypatch):
    monkeypatch.delenv("SPG_FORCE_VARIANT", raising=False)
    monkeypatch.delenv("SPG_FORCE_TAIL", raising=False)
    # the default narrow-T route: the swapped tile split inside clusters
    r = spg.select_route("fp8_rowscaled", 64, 528, 16384, "linear", workspace=True)
    assert r["variant"] == 8 and r["split_k"] > 1 and r["workspace_bytes"] == 0
    # the unswapped pair tile splits through the workspace
    monkeypatch.setenv("SPG_FORCE_VARIANT", "2sm")
    r = spg.select_route("fp8_rowscaled", 64, 528, 16384, "linear", workspace=True)
    assert r["block_m"] == 256 and r["split_k"] > 1 and r["workspace_bytes"] > 0


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
def test_fp8_splitk_bias(epi, kind, monkeypatch):
    monkeypatch.setenv("SPG_FORCE_TAIL", "k")
    T, N, K = 96, 528, 3072
    A, sa, W, sw = fp8_inputs(T, N, K, seed=11)
    if kind == "bf16":
        b = normal_bf16((N,), seed=12, std=2.0)
        bs, bt, bst = None, cuda_bf16(b), None
    else:
        b = random_codes((N,), seed=12, exclude=(0x7F, 0xFF))
        bs = np.float32(0.0625)
        bt, bst = cuda(b), torch.tensor([bs], dtype=torch.float32, device=DEV)
    res = normal_bf16((T, N), seed=13) if epi == "add" else None
    buf, ws, r = workspace_for("fp8_rowscaled", T, N, K, epi)
    assert r["split_k"] > 1
    y = run_fp8_ws(A, sa, W, sw, res, epi, ws, bias=bt, bias_scale=bst)
    check_workspace(buf, ws.numel(), r, epi)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, epi, bias=b, bias_scale=bs)
    assert_within_tol(to_f64(y), ref, f"fp8 split-K bias {kind} {epi}")


def test_fp8_splitk_repeats_bit_for_bit_and_reuses_workspace(monkeypatch):
    """Same bits on every call (fixed summation order), on a workspace that
    was never zeroed and is reused across calls."""
    monkeypatch.setenv("SPG_FORCE_TAIL", "k")
    T, N, K = 128, 1024, 8192
    A, sa, W, sw = fp8_inputs(T, N, K, seed=21)
    res = normal_bf16((T, N), seed=22)
    buf, ws, r = workspace_for("fp8_rowscaled", T, N, K, "add", fill=0xFF)
    assert r["split_k"] == 4
    buf[:GUARD] = PATTERN
    buf[GUARD + ws.numel():] = PATTERN
    ys = [run_fp8_ws(A, sa, W, sw, res, "add", ws).clone() for _ in range(5)]
    check_workspace(buf, ws.numel(), r)
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, "add")
    assert_within_tol(to_f64(ys[0]), ref, "fp8 split-K repeat")
    # the plain route computes the same GEMM (sums in another order)
    y_plain = spg.fp8_rowscaled_gemm(cuda(A), cuda(sa), cuda(W), cuda(sw),
                                     residual=cuda_bf16(res), epilogue="add")
    torch.cuda.synchronize()
    assert_within_tol(to_f64(y_plain), ref, "fp8 plain route")


def test_fp8_splitk_cuda_graph_replay(monkeypatch):
    """A captured launch keeps its call number; the counters it leaves at zero
    let every replay count its pieces afresh."""
    monkeypatch.setenv("SPG_FORCE_TAIL", "k")
    T, N, K = 64, 784, 4096
    A, sa, W, sw = fp8_inputs(T, N, K, seed=31)
    buf, ws, r = workspace_for("fp8_rowscaled", T, N, K)
    dA, dsa, dW, dsw = cuda(A), cuda(sa), cuda(W), cuda(sw)
    out = torch.empty((T, N), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        spg.fp8_rowscaled_gemm(dA, dsa, dW, dsw, out=out, workspace=ws)  # warm-up, sets attributes
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        spg.fp8_rowscaled_gemm(dA, dsa, dW, dsw, out=out, workspace=ws)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw)
    first = None
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert spg.last_device_error() == 0
        assert_within_tol(to_f64(out), ref, "fp8 split-K graph replay")
        first = out.clone() if first is None else first
        assert torch.equal(out.view(torch.int16), first.view(torch.int16))
    check_workspace(buf, ws.numel(), r)


def test_fp8_small_workspace_falls_back(monkeypatch):
    monkeypatch.setenv("SPG_FORCE_TAIL", "k")
    T, N, K = 64, 528, 4096
    A, sa, W, sw = fp8_inputs(T, N, K, seed=41)
    small = torch.zeros(16, dtype=torch.uint8, device=DEV)
    y = run_fp8_ws(A, sa, W, sw, None, "linear", small)
    assert bool((small == 0).all())
    assert_within_tol(to_f64(y), oracle.fp8_rowscaled_gemm(A, sa, W, sw), "fp8 fallback")


def test_fp8_multiwave_tail_split_sampled(monkeypatch):
    """80 pair tiles on 76 pairs: one whole wave, then 4 tiles split along K."""
    monkeypatch.setenv("SPG_FORCE_TAIL", "k")
    monkeypatch.setenv("SPG_FORCE_VARIANT", "2sm")
    T, N, K = 1024, 5120, 2048
    r = spg.select_route("fp8_rowscaled", T, N, K, "add", workspace=True)
    if r["grid"] != 152:
        pytest.skip("schedule written for 152 SMs")
    assert r["tiles"] == 80 and r["split_k"] > 1
    A, sa, W, sw = fp8_inputs(T, N, K, seed=51, w_std=0.05)
    res = normal_bf16((T, N), seed=52)
    buf, ws, r = workspace_for("fp8_rowscaled", T, N, K, "add")
    y = run_fp8_ws(A, sa, W, sw, res, "add", ws)
    check_workspace(buf, ws.numel(), r)
    rows = np.array([0, 1, 127, 128, 255, 256, 511, 700, 1023], np.int64)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, "add", rows=rows)
    assert_within_tol(to_f64(y[torch.from_numpy(rows).to(DEV)]), ref, "fp8 multi-wave K split")


@pytest.mark.parametrize("epi", ["add", "swiglu"])
def test_fp8_narrow_t_full_size_sampled(epi):
    """T = 256 with the full K and N of the linear_add and SwiGLU workloads,
    in the route the selector picks (no pin)."""
    T, K, N = (256, 17408, 5120) if epi == "add" else (256, 5120, 34816)
    A, sa, W, sw = fp8_inputs(T, N, K, seed=61, w_std=0.02)
    res = normal_bf16((T, N), seed=62) if epi == "add" else None
    buf, ws, r = workspace_for("fp8_rowscaled", T, N, K, epi)
    y = run_fp8_ws(A, sa, W, sw, res, epi, ws if ws.numel() else None)
    check_workspace(buf, ws.numel(), r, epi)
    rows = np.array([0, 1, 31, 32, 100, 127, 128, 200, 255], np.int64)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, epi, rows=rows)
    assert_within_tol(to_f64(y[torch.from_numpy(rows).to(DEV)]), ref, f"fp8 T=256 {epi}")


# ----------------------------------------------------------------- NVFP4
def nvfp4_inputs(T, N, K, seed):
    x = normal_bf16((T, K), seed=seed)
    w = normal_bf16((N, K), seed=seed + 1)
    gA = oracle.nvfp4_global_scale(x)
    gW = oracle.nvfp4_global_scale(w)
    A, sfA = oracle.quantize_nvfp4(x, gA)
    W, sfW = oracle.quantize_nvfp4(w, gW)
    return A, sfA, gA, W, sfW, gW


def run_nvfp4_ws(A, sfA, gA, W, sfW, gW, res, epi, ws, bias=None, bias_scale=None):
    T, N, K = A.shape[0], W.shape[0], 2 * A.shape[1]
    y = spg.nvfp4_gemm(cuda(A), cuda(sf_rowmajor_to_blocked(sfA, T, K)),
                       torch.tensor([gA], dtype=torch.float32, device=DEV),
                       cuda(W), cuda(sf_rowmajor_to_blocked(sfW, N, K)),
                       torch.tensor([gW], dtype=torch.float32, device=DEV),
                       residual=None if res is None else cuda_bf16(res), epilogue=epi,
                       bias=bias, bias_scale=bias_scale, workspace=ws)
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    return y


@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
@pytest.mark.parametrize("T,N,K", [(1, 16, 2048), (64, 512, 4096), (200, 272, 2304),
                                   (333, 400, 3072)])
@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("kernel", ["2sm_cp", "2sm_st", "2sm_mc"])
def test_nvfp4_splitk_ragged(T, N, K, epi, bias, kernel, monkeypatch):
    monkeypatch.setenv("SPG_FORCE_TAIL", "k")
    monkeypatch.setenv("SPG_FORCE_VARIANT", kernel)
    A, sfA, gA, W, sfW, gW = nvfp4_inputs(T, N, K, seed=T + N)
    res = normal_bf16((T, N), seed=71) if epi == "add" else None
    b = normal_bf16((N,), seed=72, std=2.0) if bias else None
    buf, ws, r = workspace_for("nvfp4", T, N, K, epi)
    assert r["split_k"] > 1
    y = run_nvfp4_ws(A, sfA, gA, W, sfW, gW, res, epi, ws,
                     bias=None if b is None else cuda_bf16(b))
    check_workspace(buf, ws.numel(), r, epi)
    ref = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, epi, bias=b)
    assert_within_tol(to_f64(y), ref, f"nvfp4 split-K {epi} {T}x{N}x{K}")


def test_nvfp4_narrow_t_full_size_sampled():
    T, K, N = 256, 17408, 5120
    A, sfA, gA, W, sfW, gW = nvfp4_inputs(T, N, K, seed=81)
    res = normal_bf16((T, N), seed=82)
    buf, ws, r = workspace_for("nvfp4", T, N, K, "add")
    y = run_nvfp4_ws(A, sfA, gA, W, sfW, gW, res, "add", ws if ws.numel() else None)
    check_workspace(buf, ws.numel(), r)
    rows = np.array([0, 1, 31, 32, 100, 127, 128, 200, 255], np.int64)
    ref = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, "add", rows=rows)
    assert_within_tol(to_f64(y[torch.from_numpy(rows).to(DEV)]), ref, "nvfp4 T=256 add")


# ------------------------------------------------------------ per-tensor
@pytest.mark.parametrize("layout", ["NT", "NN", "TN"])
@pytest.mark.parametrize("M,N,K,batch", [(64, 512, 4096, 1), (144, 272, 1024, 2)])
def test_tensor_splitk(layout, M, N, K, batch, monkeypatch):
    # the pair tile (the selector may prefer one-CTA tiles at these sizes)
    monkeypatch.setenv("SPG_FORCE_VARIANT", "2sm")
    monkeypatch.setenv("SPG_FORCE_TAIL", "k")
    a_shape = (batch, K, M) if layout[0] == "T" else (batch, M, K)
    b_shape = (batch, K, N) if layout[1] == "N" else (batch, N, K)
    A, sA = oracle.quantize_fp8_tensor(normal_bf16(a_shape, seed=91))
    B, sB = oracle.quantize_fp8_tensor(normal_bf16(b_shape, seed=92))
    A = A.reshape(-1)
    B = B.reshape(-1)
    assert spg.select_route("fp8_tensor", M, N, K, "linear", batch, workspace=True)["split_k"] > 1
    buf, ws, r = workspace_for("fp8_tensor", M, N, K, "linear", batch, exact=False)
    y = spg.fp8_tensor_gemm(layout, cuda(A), torch.tensor([sA], dtype=torch.float32, device=DEV),
                            cuda(B), torch.tensor([sB], dtype=torch.float32, device=DEV), M, N, K,
                            batch=batch, workspace=ws)
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    check_workspace(buf, ws.numel(), r)
    ref = oracle.fp8_tensor_gemm(layout, A, sA, B, sB, M, N, K, batch=batch)
    assert_within_tol(to_f64(y).reshape(batch, M, N), ref, f"tensor split-K {layout}")
