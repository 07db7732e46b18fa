"""Swapped narrow-T tile of the FP8 row-scaled GEMM (and of the per-tensor
GEMM at narrow M, layout NT) against the CPU oracle.

For T <= 128 the weights can take the MMA's 256-row side and the tokens its
N side (the accumulator is Y transposed; the epilogue writes it back as
Y [T, N]).  The scales, bias and residual enter in the same order as in the
unswapped epilogue, so the bar is the usual element-wise tolerance; with a
K split the result still repeats bit for bit and the workspace counters are
left at zero.  With fewer weight tiles than CTA pairs (every shape here) the
K split runs inside clusters of 2 x split_k CTAs and needs no workspace.
"""
import numpy as np
import pytest
import torch

import oracle
import scaled_precision_gemm_gb300 as spg
from synthetic_inputs import normal_bf16, random_codes
from tests.gpu_common import DEV, cuda, cuda_bf16, to_f64
from tests.helpers import assert_within_tol
from tests.test_splitk_gpu import GUARD, PATTERN, check_workspace, fp8_inputs, workspace_for

pytestmark = pytest.mark.gpu


@pytest.fixture
def swap(monkeypatch):
    monkeypatch.setenv("SPG_FORCE_VARIANT", "swap")
    monkeypatch.delenv("SPG_FORCE_TAIL", raising=False)


def run(A, sa, W, sw, res, epi, ws=None, bias=None, bias_scale=None):
    y = spg.fp8_rowscaled_gemm(cuda(A), cuda(sa), cuda(W), cuda(sw),
                               residual=None if res is None else cuda_bf16(res), epilogue=epi,
                               bias=bias, bias_scale=bias_scale, workspace=ws)
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    return y


@pytest.mark.parametrize("epi", ["linear", "add"])
@pytest.mark.parametrize("T", [1, 16, 33, 64, 65, 100, 128])
@pytest.mark.parametrize("N,K", [(264, 1040), (528, 4096), (1040, 2064)])
@pytest.mark.parametrize("with_ws", [False, True])
def test_swap_ragged(T, N, K, epi, with_ws, swap):
    A, sa, W, sw = fp8_inputs(T, N, K, seed=T * 7 + N + K)
    res = normal_bf16((T, N), seed=T + 5) if epi == "add" else None
    r = spg.select_route("fp8_rowscaled", T, N, K, epi, workspace=with_ws)
    assert r["swap_ab"] == 1 and r["block_m"] == 256 and r["block_n"] == (64 if T <= 64 else 128)
    if with_ws:
        buf, ws, r = workspace_for("fp8_rowscaled", T, N, K, epi)
        y = run(A, sa, W, sw, res, epi, ws if ws.numel() else None)
        check_workspace(buf, ws.numel(), r, epi)
    else:
        # no workspace: whole tiles, or (fewer tiles than pairs) the K split
        # inside clusters, which needs none
        assert r["workspace_bytes"] == 0 and (r["split_k"] == 1 or r["variant"] == 8), r
        y = run(A, sa, W, sw, res, epi)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, epi)
    assert_within_tol(to_f64(y), ref, f"fp8 swap {epi} {T}x{N}x{K} ({r['split_k']} pieces)")


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
@pytest.mark.parametrize("epi", ["linear", "add"])
def test_swap_bias(epi, kind, swap, monkeypatch):
    monkeypatch.setenv("SPG_FORCE_TAIL", "k")  # split although K is short
    T, N, K = 48, 784, 3072
    A, sa, W, sw = fp8_inputs(T, N, K, seed=17)
    if kind == "bf16":
        b = normal_bf16((N,), seed=18, std=2.0)
        bs, bt, bst = None, cuda_bf16(b), None
    else:
        b = random_codes((N,), seed=18, exclude=(0x7F, 0xFF))
        bs = np.float32(0.125)
        bt, bst = cuda(b), torch.tensor([bs], dtype=torch.float32, device=DEV)
    res = normal_bf16((T, N), seed=19) if epi == "add" else None
    buf, ws, r = workspace_for("fp8_rowscaled", T, N, K, epi)
    assert r["swap_ab"] == 1 and r["split_k"] > 1
    y = run(A, sa, W, sw, res, epi, ws, bias=bt, bias_scale=bst)
    check_workspace(buf, ws.numel(), r, epi)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, epi, bias=b, bias_scale=bs)
    assert_within_tol(to_f64(y), ref, f"fp8 swap bias {kind} {epi}")


def test_swap_splitk_repeats_and_matches_unswapped(swap, monkeypatch):
    """Same bits on every call on a never-zeroed, reused workspace; the
    unswapped route computes the same GEMM within the tolerance."""
    T, N, K = 100, 1024, 8192
    A, sa, W, sw = fp8_inputs(T, N, K, seed=23)
    res = normal_bf16((T, N), seed=24)
    buf, ws, r = workspace_for("fp8_rowscaled", T, N, K, "add", fill=0xFF)
    assert r["swap_ab"] == 1 and r["split_k"] == 4
    buf[:GUARD] = PATTERN
    buf[GUARD + ws.numel():] = PATTERN
    ys = [run(A, sa, W, sw, res, "add", ws).clone() for _ in range(5)]
    check_workspace(buf, ws.numel(), r, "add")
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, "add")
    assert_within_tol(to_f64(ys[0]), ref, "fp8 swap repeat")
    monkeypatch.setenv("SPG_FORCE_VARIANT", "2sm128")
    y_plain = run(A, sa, W, sw, res, "add")
    assert_within_tol(to_f64(y_plain), ref, "fp8 unswapped route")
    d = np.abs(to_f64(y_plain) - to_f64(ys[0])).max()
    assert d <= 0.02 * np.abs(ref).max()


def test_swap_cuda_graph_replay(swap):
    T, N, K = 16, 1536, 4096
    A, sa, W, sw = fp8_inputs(T, N, K, seed=33)
    buf, ws, r = workspace_for("fp8_rowscaled", T, N, K)
    assert r["swap_ab"] == 1 and r["split_k"] > 1
    dA, dsa, dW, dsw = cuda(A), cuda(sa), cuda(W), cuda(sw)
    out = torch.empty((T, N), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        spg.fp8_rowscaled_gemm(dA, dsa, dW, dsw, out=out, workspace=ws)
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
        assert_within_tol(to_f64(out), ref, "fp8 swap graph replay")
        first = out.clone() if first is None else first
        assert torch.equal(out.view(torch.int16), first.view(torch.int16))
    check_workspace(buf, ws.numel(), r)


@pytest.mark.parametrize("T", [1, 16, 64, 128])
def test_swap_full_size_sampled(T, swap):
    """The linear_add workload's full K and N at narrow T, sampled rows."""
    N, K = 5120, 17408
    A, sa, W, sw = fp8_inputs(T, N, K, seed=71 + T, w_std=0.02)
    res = normal_bf16((T, N), seed=72)
    buf, ws, r = workspace_for("fp8_rowscaled", T, N, K, "add")
    assert r["swap_ab"] == 1
    y = run(A, sa, W, sw, res, "add", ws if ws.numel() else None)
    check_workspace(buf, ws.numel(), r, "add")
    rows = np.unique(np.array([0, 1, 15, 31, 32, 63, 64, 100, 127]) % T).astype(np.int64)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, "add", rows=rows)
    assert_within_tol(to_f64(y[torch.from_numpy(rows).to(DEV)]), ref, f"fp8 swap T={T} add")


# ------------------------------------------------------------ per-tensor
def tensor_run(layout, A, sA, B, sB, M, N, K, ws=None, bias=None, bias_scale=None):
    y = spg.fp8_tensor_gemm(layout, cuda(A), torch.tensor([sA], dtype=torch.float32, device=DEV),
                            cuda(B), torch.tensor([sB], dtype=torch.float32, device=DEV), M, N, K,
                            workspace=ws, bias=bias, bias_scale=bias_scale)
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    return to_f64(y).reshape(M, N)


def tensor_operands(layout, M, N, K, seed):
    a = normal_bf16((K, M) if layout[0] == "T" else (M, K), seed=seed)
    b = normal_bf16((K, N) if layout[1] == "N" else (N, K), seed=seed + 1)
    A, sA = oracle.quantize_fp8_tensor(a)
    B, sB = oracle.quantize_fp8_tensor(b)
    return A.reshape(-1), sA, B.reshape(-1), sB


@pytest.mark.parametrize("M", [1, 16, 33, 64, 100, 128])
@pytest.mark.parametrize("N,K", [(136, 256), (1040, 2064), (8192, 2048)])
@pytest.mark.parametrize("with_ws", [False, True])
def test_tensor_swap_nt(M, N, K, with_ws, swap):
    """Per-tensor NT at narrow M takes the swapped tile (B's rows on the MMA's
    256-row side, scaled by sA * sB)."""
    A, sA, B, sB = tensor_operands("NT", M, N, K, seed=M * 3 + N + K)
    r = spg.select_route("fp8_tensor", M, N, K, "linear", workspace=with_ws)
    assert r["swap_ab"] == 1 and r["block_n"] == (64 if M <= 64 else 128)
    if with_ws:
        buf, ws, r = workspace_for("fp8_tensor", M, N, K, exact=False)
        y = tensor_run("NT", A, sA, B, sB, M, N, K, ws)
        check_workspace(buf, ws.numel(), r)
    else:
        y = tensor_run("NT", A, sA, B, sB, M, N, K)
    ref = oracle.fp8_tensor_gemm("NT", A, sA, B, sB, M, N, K).reshape(M, N)
    assert_within_tol(y, ref, f"tensor swap NT {M}x{N}x{K}")


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
def test_tensor_swap_bias(kind, swap):
    M, N, K = 48, 784, 1024
    A, sA, B, sB = tensor_operands("NT", M, N, K, seed=91)
    if kind == "bf16":
        b = normal_bf16((N,), seed=92, std=2.0)
        bs, bt, bst = None, cuda_bf16(b), None
    else:
        b = random_codes((N,), seed=92, exclude=(0x7F, 0xFF))
        bs = np.float32(0.125)
        bt, bst = cuda(b), torch.tensor([bs], dtype=torch.float32, device=DEV)
    y = tensor_run("NT", A, sA, B, sB, M, N, K, bias=bt, bias_scale=bst)
    ref = oracle.fp8_tensor_gemm("NT", A, sA, B, sB, M, N, K, bias=b, bias_scale=bs).reshape(M, N)
    assert_within_tol(y, ref, f"tensor swap bias {kind}")


@pytest.mark.parametrize("layout", ["NN", "TN", "TT"])
def test_tensor_narrow_other_layouts(layout):
    """Narrow M with an M-major A or an N-major B: the unswapped tiles."""
    M, N, K = 64, 528, 1024
    A, sA, B, sB = tensor_operands(layout, M, N, K, seed=95)
    y = tensor_run(layout, A, sA, B, sB, M, N, K)
    if layout == "TT":
        Bt = B.reshape(N, K).T.reshape(-1)
        ref = oracle.fp8_tensor_gemm("TN", A, sA, Bt, sB, M, N, K)
    else:
        ref = oracle.fp8_tensor_gemm(layout, A, sA, B, sB, M, N, K)
    assert_within_tol(y, ref.reshape(M, N), f"tensor narrow {layout}")
