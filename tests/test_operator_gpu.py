"""The activation operators (bf16 activations in, quantized inside the call)
against the CPU oracle.

The oracle quantizes the same bf16 activations (NVFP4: global scale, block
scales, codes; FP8: row scales, codes) and multiplies them with the
oracle-quantized weights; the operator's output must meet the element-wise
tolerance of the GEMM tests.  The operator's codes are by definition those
of the library's quantizers, so its output must also equal, bit for bit,
the library's own quantize-then-GEMM sequence on the same route -- and the
single fused NVFP4 decode kernel (pinned; each CTA cluster quantizes the
activations itself) against the quantizer kernels followed by the GEMV.  Output buffers are NaN-filled with NaN guard bands.
"""
import numpy as np
import pytest
import torch

import oracle
import scaled_precision_gemm_gb300 as spg
from synthetic_inputs import normal_bf16, random_codes
from tests.gpu_common import DEV, cuda, cuda_bf16, to_f64
from tests.helpers import assert_within_tol, sf_rowmajor_to_blocked
from tests.test_gemm_gpu import check_guards, guarded_out

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def default_route(monkeypatch):
    for v in ("SPG_FORCE_VARIANT", "SPG_FORCE_TAIL", "SPG_FORCE_GROUP_M"):
        monkeypatch.delenv(v, raising=False)


@pytest.fixture(params=["sequence", "fused"])
def nv_form(request, monkeypatch):
    """The NVFP4 operator as two kernels (the default) or, at T <= 4, as the
    single fused decode kernel (pinned)."""
    if request.param == "fused":
        monkeypatch.setenv("SPG_FORCE_VARIANT", "gemv_fused")
    return request.param


def nv_weights(N, K, seed):
    w = normal_bf16((N, K), seed=seed)
    gW = oracle.nvfp4_global_scale(w)
    W, sfW = oracle.quantize_nvfp4(w, gW)
    return W, sfW, gW


def nv_device_weights(W, sfW, gW, N, K):
    return (cuda(W), cuda(sf_rowmajor_to_blocked(sfW, N, K)),
            torch.tensor([gW], dtype=torch.float32, device=DEV))


def nv_reference(x, W, sfW, gW, res, epi, rows=None, bias=None, bias_scale=None):
    gA = oracle.nvfp4_global_scale(x)
    A, sfA = oracle.quantize_nvfp4(x, gA)
    return oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, epi, rows=rows, bias=bias,
                             bias_scale=bias_scale)


def nv_library_sequence(xd, Wd, sfWd, gWd, resd, epi, T, N, K, fused, monkeypatch,
                        bias=None, bias_scale=None):
    """The library's quantizers, then its GEMM with the operator's workspace
    (for the fused kernel: the GEMV, whose sums it shares)."""
    gA = spg.nvfp4_global_scale(xd)
    A, sfA = spg.quantize_nvfp4(xd, gA)
    if fused:
        monkeypatch.setenv("SPG_FORCE_VARIANT", "gemv")
    y = spg.nvfp4_gemm(A, sfA, gA, Wd, sfWd, gWd, residual=resd, epilogue=epi, bias=bias,
                       bias_scale=bias_scale,
                       workspace=spg.gemm_workspace("nvfp4", T, N, K, epi, device=DEV))
    if fused:
        monkeypatch.setenv("SPG_FORCE_VARIANT", "gemv_fused")
    return y


def run_nv_operator(xd, Wd, sfWd, gWd, resd, epi, T, N, bias=None, bias_scale=None):
    n_out = N // 2 if epi == "swiglu" else N
    buf, out = guarded_out(T, n_out)
    y = spg.nvfp4_linear_bf16(xd, Wd, sfWd, gWd, residual=resd, epilogue=epi, out=out,
                              bias=bias, bias_scale=bias_scale)
    torch.cuda.synchronize()
    check_guards(buf)
    assert spg.last_device_error() == 0
    return y


@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 64, 200])
@pytest.mark.parametrize("N,K", [(144, 768), (1040, 4352), (16400, 512)])
def test_nvfp4_operator(T, N, K, epi, nv_form, monkeypatch):
    fused = nv_form == "fused" and T <= 4
    assert (spg.act_workspace_bytes("nvfp4", T, N, K, epi) == 0) == fused
    x = normal_bf16((T, K), seed=T * 7 + N + K)
    W, sfW, gW = nv_weights(N, K, seed=N + 1)
    res = normal_bf16((T, N), seed=T + 3) if epi == "add" else None
    xd = cuda_bf16(x)
    Wd, sfWd, gWd = nv_device_weights(W, sfW, gW, N, K)
    resd = None if res is None else cuda_bf16(res)
    y = run_nv_operator(xd, Wd, sfWd, gWd, resd, epi, T, N)
    assert_within_tol(to_f64(y), nv_reference(x, W, sfW, gW, res, epi),
                      f"nvfp4 operator {epi} {T}x{N}x{K}")
    seq = nv_library_sequence(xd, Wd, sfWd, gWd, resd, epi, T, N, K, fused, monkeypatch)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), seq.view(torch.int16))


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
@pytest.mark.parametrize("T,N,K", [(2, 16400, 512), (64, 272, 1024)])
def test_nvfp4_operator_bias(T, N, K, epi, kind, nv_form):
    x = normal_bf16((T, K), seed=11)
    W, sfW, gW = nv_weights(N, K, seed=12)
    if kind == "bf16":
        b = normal_bf16((N,), seed=13, std=2.0)
        bs, bt, bst = None, cuda_bf16(b), None
    else:
        b = random_codes((N,), seed=13, exclude=(0x7F, 0xFF))
        bs = np.float32(0.125)
        bt, bst = cuda(b), torch.tensor([bs], dtype=torch.float32, device=DEV)
    res = normal_bf16((T, N), seed=14) if epi == "add" else None
    xd = cuda_bf16(x)
    Wd, sfWd, gWd = nv_device_weights(W, sfW, gW, N, K)
    resd = None if res is None else cuda_bf16(res)
    y = run_nv_operator(xd, Wd, sfWd, gWd, resd, epi, T, N, bias=bt, bias_scale=bst)
    ref = nv_reference(x, W, sfW, gW, res, epi, bias=b, bias_scale=bs)
    assert_within_tol(to_f64(y), ref, f"nvfp4 operator bias {kind} {epi}")


def test_nvfp4_operator_special_activations(nv_form, monkeypatch):
    """Activations with an all-zero block, a block whose scale underflows to
    zero, an all-zero token and an all-zero tensor (global scale 1)."""
    T, N, K = 2, 16400, 1024
    fused = nv_form == "fused"
    x = normal_bf16((T, K), seed=21).view(np.uint16).copy()
    x[0, 16:32] = 0                                  # zero block
    xf = (x[0].astype(np.uint32) << 16).view(np.float32) * np.float32(1e-7)
    x[0, 64:80] = (xf.view(np.uint32)[64:80] >> 16).astype(np.uint16)   # tiny block (truncated to bf16)
    x[1] = 0                                         # zero token
    W, sfW, gW = nv_weights(N, K, seed=22)
    Wd, sfWd, gWd = nv_device_weights(W, sfW, gW, N, K)
    for xx in (x, np.zeros_like(x)):
        xd = cuda_bf16(xx)
        y = run_nv_operator(xd, Wd, sfWd, gWd, None, "linear", T, N)
        assert_within_tol(to_f64(y), nv_reference(xx, W, sfW, gW, None, "linear"),
                          "nvfp4 operator special blocks")
        seq = nv_library_sequence(xd, Wd, sfWd, gWd, None, "linear", T, N, K, fused,
                                  monkeypatch)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), seq.view(torch.int16))


@pytest.mark.parametrize("T,K,N,epi", [(1, 17408, 5120, "add"), (1, 6144, 5120, "add"),
                                       (4, 6144, 5120, "add"), (2, 5120, 34816, "swiglu"),
                                       (4, 5120, 34816, "swiglu"), (64, 17408, 5120, "add")])
def test_nvfp4_operator_full_size(T, K, N, epi, nv_form):
    x = normal_bf16((T, K), seed=31)
    W, sfW, gW = nv_weights(N, K, seed=32)
    res = normal_bf16((T, N), seed=33) if epi == "add" else None
    xd = cuda_bf16(x)
    Wd, sfWd, gWd = nv_device_weights(W, sfW, gW, N, K)
    resd = None if res is None else cuda_bf16(res)
    y = run_nv_operator(xd, Wd, sfWd, gWd, resd, epi, T, N)
    rows = np.unique(np.array([0, T // 2, T - 1]))
    ref = nv_reference(x, W, sfW, gW, res, epi, rows=rows)
    assert_within_tol(to_f64(y[torch.from_numpy(rows).to(DEV)]), ref,
                      f"nvfp4 operator {epi} {T}x{N}x{K}")


# ------------------------------------------------------------------ FP8
@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
@pytest.mark.parametrize("T", [1, 16, 64, 200])
def test_fp8_operator(T, epi):
    N, K = 272, 1280
    x = normal_bf16((T, K), seed=T + 41)
    w = normal_bf16((N, K), seed=42)
    W, sw = oracle.quantize_fp8_rows(w)
    res = normal_bf16((T, N), seed=43) if epi == "add" else None
    n_out = N // 2 if epi == "swiglu" else N
    buf, out = guarded_out(T, n_out)
    xd, Wd, swd = cuda_bf16(x), cuda(W), cuda(sw)
    resd = None if res is None else cuda_bf16(res)
    y = spg.fp8_rowscaled_linear_bf16(xd, Wd, swd, residual=resd, epilogue=epi, out=out)
    torch.cuda.synchronize()
    check_guards(buf)
    assert spg.last_device_error() == 0
    A, sa = oracle.quantize_fp8_rows(x)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, epi)
    assert_within_tol(to_f64(y), ref, f"fp8 operator {epi} {T}x{N}x{K}")
    Ad, sad = spg.quantize_fp8_rows(xd)
    seq = spg.fp8_rowscaled_gemm(Ad, sad, Wd, swd, residual=resd, epilogue=epi,
                                 workspace=spg.gemm_workspace("fp8_rowscaled", T, N, K, epi,
                                                              device=DEV))
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), seq.view(torch.int16))


def test_fp8_operator_full_size_sampled():
    T, K, N = 16, 17408, 5120
    x = normal_bf16((T, K), seed=51)
    w = normal_bf16((N, K), seed=52, std=0.02)
    W, sw = oracle.quantize_fp8_rows(w)
    res = normal_bf16((T, N), seed=53)
    y = spg.fp8_rowscaled_linear_bf16(cuda_bf16(x), cuda(W), cuda(sw), residual=cuda_bf16(res),
                                      epilogue="add")
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    rows = np.array([0, 7, 15])
    A, sa = oracle.quantize_fp8_rows(x)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, "add", rows=rows)
    assert_within_tol(to_f64(y[torch.from_numpy(rows).to(DEV)]), ref, "fp8 operator full size")


# --------------------------------------------------------------- errors
def test_operator_errors():
    T, N, K = 64, 272, 1280
    x = cuda_bf16(normal_bf16((T, K), seed=61))
    W, sw = oracle.quantize_fp8_rows(normal_bf16((N, K), seed=62))
    Wd, swd = cuda(W), cuda(sw)
    need = spg.act_workspace_bytes("fp8_rowscaled", T, N, K)
    assert need >= T * K + 4 * T
    small = torch.empty((T * K,), dtype=torch.uint8, device=DEV)
    with pytest.raises(spg.SpgError, match="INVALID_ARG"):
        spg.fp8_rowscaled_linear_bf16(x, Wd, swd, workspace=small)
    # an unaligned activation base
    flat = torch.empty((T * K + 8,), dtype=torch.bfloat16, device=DEV)
    xu = flat[1:1 + T * K].view(T, K)
    with pytest.raises(spg.SpgError, match="MISALIGNED"):
        spg.fp8_rowscaled_linear_bf16(xu, Wd, swd)
    # NVFP4 K must be a multiple of 256
    Wn, sfWn, gWn = nv_weights(N, 320, seed=63)
    with pytest.raises(spg.SpgError, match="UNSUPPORTED_SHAPE"):
        spg.nvfp4_linear_bf16(cuda_bf16(normal_bf16((T, 320), seed=64)),
                              *nv_device_weights(Wn, sfWn, gWn, N, 320))
    assert spg.last_device_error() == 0
