"""Fused bias on the three GEMMs against the CPU oracle (bf16 bias, and E4M3
bias storage dequantized with bias_scale), with every epilogue and tile shape."""
import numpy as np
import pytest
import torch

import oracle
import scaled_precision_gemm_gb300 as spg
from synthetic_inputs import normal_bf16, random_codes
from tests.gpu_common import DEV, cuda, cuda_bf16, to_f64
from tests.helpers import assert_within_tol, sf_rowmajor_to_blocked

pytestmark = pytest.mark.gpu


def _bias(kind, N, seed):
    if kind == "bf16":
        b = normal_bf16((N,), seed=seed, std=2.0)
        return b, None, cuda_bf16(b), None
    b = random_codes((N,), seed=seed, exclude=(0x7F, 0xFF))
    s = np.float32(0.0625)
    return b, s, cuda(b), torch.tensor([s], dtype=torch.float32, device=DEV)


@pytest.fixture(params=["auto", "2sm", "2sm192", "1sm256"])
def variant(request, monkeypatch):
    if request.param == "auto":
        monkeypatch.delenv("SPG_FORCE_VARIANT", raising=False)
    else:
        monkeypatch.setenv("SPG_FORCE_VARIANT", request.param)
    return request.param


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
@pytest.mark.parametrize("T,N,K", [(65, 272, 400), (300, 1088, 1040)])
def test_fp8_rowscaled_bias(T, N, K, epi, kind, variant):
    A, sa = oracle.quantize_fp8_rows(normal_bf16((T, K), seed=1))
    W, sw = oracle.quantize_fp8_rows(normal_bf16((N, K), seed=2))
    b, bs, bt, bst = _bias(kind, N, seed=3)
    res = normal_bf16((T, N), seed=4) if epi == "add" else None
    y = spg.fp8_rowscaled_gemm(cuda(A), cuda(sa), cuda(W), cuda(sw),
                               residual=None if res is None else cuda_bf16(res), epilogue=epi,
                               bias=bt, bias_scale=bst)
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, epi, bias=b, bias_scale=bs)
    assert_within_tol(to_f64(y), ref, f"fp8 bias {kind} {epi}")


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
@pytest.mark.parametrize("nv_variant", ["auto", "1sm128", "2sm_cp", "2sm_st", "2sm_mc"])
def test_nvfp4_bias(epi, kind, nv_variant, monkeypatch):
    if nv_variant == "auto":
        monkeypatch.delenv("SPG_FORCE_VARIANT", raising=False)
    else:
        monkeypatch.setenv("SPG_FORCE_VARIANT", nv_variant)
    T, N, K = 520, 784, 768
    x = normal_bf16((T, K), seed=5)
    w = normal_bf16((N, K), seed=6)
    gA = oracle.nvfp4_global_scale(x)
    gW = oracle.nvfp4_global_scale(w)
    A, sfA = oracle.quantize_nvfp4(x, gA)
    W, sfW = oracle.quantize_nvfp4(w, gW)
    b, bs, bt, bst = _bias(kind, N, seed=7)
    res = normal_bf16((T, N), seed=8) if epi == "add" else None
    y = spg.nvfp4_gemm(cuda(A), cuda(sf_rowmajor_to_blocked(sfA, T, K)),
                       torch.tensor([gA], dtype=torch.float32, device=DEV), cuda(W),
                       cuda(sf_rowmajor_to_blocked(sfW, N, K)),
                       torch.tensor([gW], dtype=torch.float32, device=DEV),
                       residual=None if res is None else cuda_bf16(res), epilogue=epi,
                       bias=bt, bias_scale=bst)
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    ref = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, epi, bias=b, bias_scale=bs)
    assert_within_tol(to_f64(y), ref, f"nvfp4 bias {kind} {epi}")


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
@pytest.mark.parametrize("layout", ["NT", "NN", "TN"])
def test_tensor_bias_broadcast_over_batch(layout, kind):
    M, N, K, batch = 144, 272, 160, 2
    a_shape = (batch, K, M) if layout[0] == "T" else (batch, M, K)
    b_shape = (batch, K, N) if layout[1] == "N" else (batch, N, K)
    A, sA = oracle.quantize_fp8_tensor(normal_bf16(a_shape, seed=9))
    B, sB = oracle.quantize_fp8_tensor(normal_bf16(b_shape, seed=10))
    A = A.reshape(-1)
    B = B.reshape(-1)
    b, bs, bt, bst = _bias(kind, N, seed=11)
    y = spg.fp8_tensor_gemm(layout, cuda(A), torch.tensor([sA], dtype=torch.float32, device=DEV),
                            cuda(B), torch.tensor([sB], dtype=torch.float32, device=DEV), M, N, K,
                            batch=batch, bias=bt, bias_scale=bst)
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    ref = oracle.fp8_tensor_gemm(layout, A, sA, B, sB, M, N, K, batch=batch, bias=b, bias_scale=bs)
    assert_within_tol(to_f64(y).reshape(batch, M, N), ref, f"tensor bias {layout} {kind}")
