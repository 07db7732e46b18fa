"""NVFP4 GEMV route (decode-sized T <= 4, CUDA cores) against the CPU oracle.

The GEMV takes each 16-element block's dot product exactly (int8 holding
twice the E2M1 values) and sums the scaled blocks in fp32, so it differs
from the oracle's exact sum only by fp32 rounding: the usual element-wise
tolerance.  Ragged N (not a multiple of the 4 warps x 2 rows of a CTA), all
three epilogues, both bias kinds, T = 1..4, and the full linear_add /
SwiGLU widths on sampled tokens.
"""
import numpy as np
import pytest
import torch

import oracle
import scaled_precision_gemm_gb300 as spg
from synthetic_inputs import normal_bf16, random_codes
from tests.gpu_common import DEV, cuda, cuda_bf16, to_f64
from tests.helpers import assert_within_tol
from tests.test_gemm_gpu import nvfp4_inputs, run_nvfp4

pytestmark = pytest.mark.gpu


@pytest.fixture
def gemv_route(monkeypatch):
    """The GEMV pinned (the default route for T <= 4 as well)."""
    monkeypatch.setenv("SPG_FORCE_VARIANT", "gemv")
    monkeypatch.delenv("SPG_FORCE_TAIL", raising=False)


@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
@pytest.mark.parametrize("T", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", [(8, 256), (16, 512), (136, 768), (1040, 4352)])
def test_gemv_ragged(T, N, K, epi, gemv_route):
    r = spg.select_route("nvfp4", T, N, K, epi)
    assert r["variant"] == 4 and r["grid"] == (N // 2 + 3) // 4
    A, sfA, gA, W, sfW, gW = nvfp4_inputs(T, N, K, seed=T * 31 + N + K)
    res = normal_bf16((T, N), seed=T + 9) if epi == "add" else None
    if epi == "swiglu" and N % 16:
        with pytest.raises(spg.SpgError, match="UNSUPPORTED_SHAPE"):
            run_nvfp4(A, sfA, gA, W, sfW, gW, res, epi)
        return
    y = run_nvfp4(A, sfA, gA, W, sfW, gW, res, epi)
    ref = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, epi)
    assert_within_tol(to_f64(y), ref, f"nvfp4 gemv {epi} {T}x{N}x{K}")


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
def test_gemv_bias(epi, kind, gemv_route):
    T, N, K = 3, 272, 1024
    A, sfA, gA, W, sfW, gW = nvfp4_inputs(T, N, K, seed=5)
    if kind == "bf16":
        b = normal_bf16((N,), seed=6, std=2.0)
        bs, bt, bst = None, cuda_bf16(b), None
    else:
        b = random_codes((N,), seed=6, exclude=(0x7F, 0xFF))
        bs = np.float32(0.125)
        bt, bst = cuda(b), torch.tensor([bs], dtype=torch.float32, device=DEV)
    res = normal_bf16((T, N), seed=7) if epi == "add" else None
    from tests.helpers import sf_rowmajor_to_blocked
    y = spg.nvfp4_gemm(cuda(A), cuda(sf_rowmajor_to_blocked(sfA, T, K)),
                       torch.tensor([gA], dtype=torch.float32, device=DEV),
                       cuda(W), cuda(sf_rowmajor_to_blocked(sfW, N, K)),
                       torch.tensor([gW], dtype=torch.float32, device=DEV),
                       residual=None if res is None else cuda_bf16(res), epilogue=epi,
                       bias=bt, bias_scale=bst)
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    ref = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, epi, bias=b, bias_scale=bs)
    assert_within_tol(to_f64(y), ref, f"nvfp4 gemv bias {kind} {epi}")


@pytest.mark.parametrize("T", [1, 4])
def test_gemv_matches_tile_route(T, monkeypatch):
    """The GEMV and the pair tile compute the same GEMM (sums in another
    order); the GEMV repeats bit for bit."""
    N, K = 528, 2048
    A, sfA, gA, W, sfW, gW = nvfp4_inputs(T, N, K, seed=40 + T)
    res = normal_bf16((T, N), seed=41)
    monkeypatch.setenv("SPG_FORCE_VARIANT", "gemv")
    ys = [run_nvfp4(A, sfA, gA, W, sfW, gW, res, "add").clone() for _ in range(3)]
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))
    monkeypatch.setenv("SPG_FORCE_VARIANT", "2sm_st")
    y_tile = run_nvfp4(A, sfA, gA, W, sfW, gW, res, "add")
    ref = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, "add")
    assert_within_tol(to_f64(ys[0]), ref, "gemv")
    assert_within_tol(to_f64(y_tile), ref, "pair tile")


@pytest.mark.parametrize("epi", ["add", "swiglu"])
@pytest.mark.parametrize("T", [1, 4])
def test_gemv_full_size(T, epi, gemv_route):
    """The linear_add (K=17408, N=5120) and SwiGLU (K=5120, N=34816) widths."""
    K, N = (17408, 5120) if epi == "add" else (5120, 34816)
    A, sfA, gA, W, sfW, gW = nvfp4_inputs(T, N, K, seed=50 + T)
    res = normal_bf16((T, N), seed=51) if epi == "add" else None
    assert spg.select_route("nvfp4", T, N, K, epi)["variant"] == 4
    y = run_nvfp4(A, sfA, gA, W, sfW, gW, res, epi)
    ref = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, epi)
    assert_within_tol(to_f64(y), ref, f"nvfp4 gemv full {epi} T={T}")
