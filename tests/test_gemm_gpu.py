"""GPU GEMMs against the CPU oracle.

Inputs are quantized by the ORACLE (never by the CUDA path) and the same codes
and scales are fed to both sides.  Outputs must satisfy
|y - ref| <= 8e-3 |ref| + 1e-3 rms(ref) element by element.  Small shapes are
compared in full (several tiles plus ragged tails in T, N and K); the full
workload shapes are compared on sampled rows, in the launch configuration the
bench times.  Every output buffer is prefilled with NaN and surrounded by NaN
guard bands, so an unwritten element or a write out of bounds fails.
"""
import numpy as np
import pytest
import torch

import oracle
import scaled_precision_gemm_gb300 as spg
from synthetic_inputs import normal_bf16
from tests.gpu_common import DEV, cuda, cuda_bf16, to_f64
from tests.helpers import assert_within_tol, sf_rowmajor_to_blocked

pytestmark = pytest.mark.gpu
GUARD = 64
VARIANTS = ["auto", "2sm", "2sm192", "2sm160", "2sm128", "1sm256", "1sm128"]


@pytest.fixture(params=VARIANTS)
def variant(request, monkeypatch):
    """Pin the FP8 tile shape: two-SM 256 x {256, 192, 160, 128}, one-CTA 128 x {256, 128}.

    A pin the shape cannot take (SwiGLU needs 64-column multiples; an N-major B
    needs the 256-wide pair tile) falls back to the selector's choice."""
    if request.param == "auto":
        monkeypatch.delenv("SPG_FORCE_VARIANT", raising=False)
    else:
        monkeypatch.setenv("SPG_FORCE_VARIANT", request.param)
    return request.param


def guarded_out(rows, cols, batch=1):
    n = batch * rows * cols
    buf = torch.full((n + 2 * GUARD,), float("nan"), dtype=torch.bfloat16, device=DEV)
    view = buf[GUARD:GUARD + n].view(batch, rows, cols) if batch > 1 else \
        buf[GUARD:GUARD + n].view(rows, cols)
    return buf, view


def check_guards(buf):
    g = torch.cat([buf[:GUARD], buf[-GUARD:]])
    assert torch.isnan(g.float()).all(), "write outside the output buffer"


def fp8_inputs(T, N, K, w_std=1.0, seed=0):
    x = normal_bf16((T, K), seed=seed)
    w = normal_bf16((N, K), seed=seed + 1, std=w_std)
    A, sa = oracle.quantize_fp8_rows(x)
    W, sw = oracle.quantize_fp8_rows(w)
    return A, sa, W, sw


def run_fp8(A, sa, W, sw, res, epi):
    T, N = A.shape[0], W.shape[0]
    n_out = N // 2 if epi == "swiglu" else N
    buf, out = guarded_out(T, n_out)
    y = spg.fp8_rowscaled_gemm(cuda(A), cuda(sa), cuda(W), cuda(sw),
                               residual=None if res is None else cuda_bf16(res),
                               epilogue=epi, out=out)
    torch.cuda.synchronize()
    check_guards(buf)
    assert spg.last_device_error() == 0
    return to_f64(y)


# ------------------------------------------------------------------- FP8
def test_fp8_config_small_linear():
    """T=64, K=256, N=128 plain linear, A and W N(0,1)."""
    A, sa, W, sw = fp8_inputs(64, 128, 256)
    y = run_fp8(A, sa, W, sw, None, "linear")
    assert_within_tol(y, oracle.fp8_rowscaled_gemm(A, sa, W, sw), "fp8 64x128x256")


@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
@pytest.mark.parametrize("T,N,K", [(1, 16, 16), (63, 136, 112), (65, 264, 400), (257, 528, 1040),
                                   (130, 256, 4096), (300, 1040, 272), (520, 784, 640)])
def test_fp8_ragged(T, N, K, epi, variant):
    A, sa, W, sw = fp8_inputs(T, N, K, seed=T + N + K)
    res = normal_bf16((T, N), seed=2) if epi == "add" else None
    if epi == "swiglu" and N % 16:
        # SwiGLU needs whole gate/up pairs in 16-byte output rows: rejected on the host
        with pytest.raises(spg.SpgError, match="UNSUPPORTED_SHAPE"):
            run_fp8(A, sa, W, sw, res, epi)
        return
    y = run_fp8(A, sa, W, sw, res, epi)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, epi)
    assert_within_tol(y, ref, f"fp8 {epi} {T}x{N}x{K}")


def test_fp8_identity_onehot_linearity():
    K = N = 256
    A, _, _, _ = fp8_inputs(96, N, K)
    sa = np.float32(2.0) ** np.arange(-6, 90, dtype=np.float32)[:96] / np.float32(2.0 ** 40)
    Wid = np.zeros((N, K), np.uint8)
    np.fill_diagonal(Wid, 0x38)
    ones = np.ones(N, np.float32)
    y = run_fp8(A, sa, Wid, ones, None, "linear")
    ref = oracle.fp8_rowscaled_gemm(A, sa, Wid, ones)
    # power-of-two row scales: every output is an E4M3 value times 2^j, exact in bf16
    assert np.array_equal(y, ref)
    _, _, W, sw = fp8_inputs(1, 136, K, seed=5)
    onehot = np.zeros((1, K), np.uint8)
    onehot[0, 77] = 0x38
    y1 = run_fp8(onehot, np.ones(1, np.float32), W, sw, None, "linear")
    assert_within_tol(y1, oracle.fp8_rowscaled_gemm(onehot, np.ones(1, np.float32), W, sw))
    y2 = run_fp8(A, sa * 2, Wid, ones, None, "linear")
    assert np.array_equal(y2, 2 * y)


def _sample_rows(T, n=12, seed=0):
    rng = np.random.default_rng(seed)
    rows = {0, 1, 127, 128, T - 1, T // 2}
    rows |= set(rng.integers(0, T, n).tolist())
    return np.array(sorted(r for r in rows if r < T), np.int64)


@pytest.mark.parametrize("T,K,N", [(1024, 17408, 5120), (4096, 6144, 5120)])
def test_fp8_linear_add_full_size_sampled(T, K, N):
    A, sa, W, sw = fp8_inputs(T, N, K, w_std=0.02)
    res = normal_bf16((T, N), seed=2)
    buf, out = guarded_out(T, N)
    y = spg.fp8_rowscaled_gemm(cuda(A), cuda(sa), cuda(W), cuda(sw), residual=cuda_bf16(res),
                               epilogue="add", out=out)
    torch.cuda.synchronize()
    check_guards(buf)
    assert not torch.isnan(y.float()).any()
    rows = _sample_rows(T)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, res, "add", rows=rows)
    assert_within_tol(to_f64(y[torch.from_numpy(rows).to(DEV)]), ref, f"fp8 add {T}x{N}x{K}")


@pytest.mark.parametrize("T,N,epi", [(1024, 34816, "swiglu"), (1024, 14336, "linear")])
def test_fp8_k5120_full_size_sampled(T, N, epi):
    K = 5120
    A, sa, W, sw = fp8_inputs(T, N, K)
    n_out = N // 2 if epi == "swiglu" else N
    buf, out = guarded_out(T, n_out)
    y = spg.fp8_rowscaled_gemm(cuda(A), cuda(sa), cuda(W), cuda(sw), epilogue=epi, out=out)
    torch.cuda.synchronize()
    check_guards(buf)
    assert not torch.isnan(y.float()).any()
    rows = _sample_rows(T, n=6)
    ref = oracle.fp8_rowscaled_gemm(A, sa, W, sw, None, epi, rows=rows)
    assert_within_tol(to_f64(y[torch.from_numpy(rows).to(DEV)]), ref, f"fp8 {epi} {T}x{N}")


# ----------------------------------------------------------------- NVFP4
@pytest.fixture(params=["auto", "1sm128", "2sm_cp", "2sm_st", "2sm_mc"])
def nv_variant(request, monkeypatch):
    """Pin the NVFP4 kernel: two-SM 256x256 with its scales copied into TMEM
    by the tensor core (2sm_cp) or written by warps (2sm_st), the cluster of
    two one-CTA tiles sharing the weight tile by multicast (2sm_mc), or the one-CTA
    128x128 tile."""
    if request.param == "auto":
        monkeypatch.delenv("SPG_FORCE_VARIANT", raising=False)
    else:
        monkeypatch.setenv("SPG_FORCE_VARIANT", request.param)
    return request.param


def nvfp4_inputs(T, N, K, seed=0):
    x = normal_bf16((T, K), seed=seed)
    w = normal_bf16((N, K), seed=seed + 1)
    gA = oracle.nvfp4_global_scale(x)
    gW = oracle.nvfp4_global_scale(w)
    A, sfA = oracle.quantize_nvfp4(x, gA)
    W, sfW = oracle.quantize_nvfp4(w, gW)
    return A, sfA, gA, W, sfW, gW


def run_nvfp4(A, sfA, gA, W, sfW, gW, res, epi):
    T, N, K = A.shape[0], W.shape[0], 2 * A.shape[1]
    n_out = N // 2 if epi == "swiglu" else N
    buf, out = guarded_out(T, n_out)
    y = spg.nvfp4_gemm(cuda(A), cuda(sf_rowmajor_to_blocked(sfA, T, K)),
                       torch.tensor([gA], dtype=torch.float32, device=DEV),
                       cuda(W), cuda(sf_rowmajor_to_blocked(sfW, N, K)),
                       torch.tensor([gW], dtype=torch.float32, device=DEV),
                       residual=None if res is None else cuda_bf16(res), epilogue=epi, out=out)
    torch.cuda.synchronize()
    check_guards(buf)
    assert spg.last_device_error() == 0
    return y


@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
@pytest.mark.parametrize("T,N,K", [(64, 128, 256), (128, 256, 512), (200, 272, 1280),
                                   (1, 16, 256), (333, 400, 2304), (520, 784, 768)])
def test_nvfp4_ragged(T, N, K, epi, nv_variant):
    A, sfA, gA, W, sfW, gW = nvfp4_inputs(T, N, K, seed=T + N)
    res = normal_bf16((T, N), seed=2) if epi == "add" else None
    y = run_nvfp4(A, sfA, gA, W, sfW, gW, res, epi)
    ref = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, epi)
    assert_within_tol(to_f64(y), ref, f"nvfp4 {epi} {T}x{N}x{K}")


def test_nvfp4_uniform_scales_and_linearity(nv_variant):
    # all block scales equal: isolates the E2M1 data path from the scale layout
    T, N, K = 128, 128, 512
    rng = np.random.default_rng(3)
    A = rng.integers(0, 256, (T, K // 2), dtype=np.uint8)
    W = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sfA = np.full((T, K // 16), 0x38, np.uint8)
    sfW = np.full((N, K // 16), 0x38, np.uint8)
    y = run_nvfp4(A, sfA, 1.0, W, sfW, 1.0, None, "linear")
    ref = oracle.nvfp4_gemm(A, sfA, 1.0, W, sfW, 1.0)
    assert_within_tol(to_f64(y), ref, "nvfp4 uniform scales")
    y2 = run_nvfp4(A, sfA, 2.0, W, sfW, 1.0, None, "linear")
    assert torch.equal(y2.float(), 2 * y.float())


@pytest.mark.parametrize("T,K,N,epi", [(256, 17408, 5120, "add"), (1024, 6144, 5120, "add"),
                                       (1024, 5120, 34816, "swiglu"), (64, 17408, 5120, "add"),
                                       (128, 5120, 34816, "swiglu")])
def test_nvfp4_full_size_sampled(T, K, N, epi):
    A, sfA, gA, W, sfW, gW = nvfp4_inputs(T, N, K)
    res = normal_bf16((T, N), seed=2) if epi == "add" else None
    y = run_nvfp4(A, sfA, gA, W, sfW, gW, res, epi)
    assert not torch.isnan(y.float()).any()
    rows = _sample_rows(T, n=6)
    ref = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, epi, rows=rows)
    assert_within_tol(to_f64(y[torch.from_numpy(rows).to(DEV)]), ref, f"nvfp4 {epi} {T}x{N}x{K}")


# --------------------------------------------------------- per-tensor FP8
def tensor_inputs(layout, M, N, K, batch, seed):
    a_shape = (batch, K, M) if layout[0] == "T" else (batch, M, K)
    b_shape = (batch, K, N) if layout[1] == "N" else (batch, N, K)
    a = normal_bf16(a_shape, seed=seed)
    b = normal_bf16(b_shape, seed=seed + 1)
    A, sA = oracle.quantize_fp8_tensor(a)
    B, sB = oracle.quantize_fp8_tensor(b)
    return A.reshape(-1), sA, B.reshape(-1), sB


def run_tensor(layout, A, sA, B, sB, M, N, K, batch, strideA=None, strideB=None):
    buf, out = guarded_out(M, N, batch)
    y = spg.fp8_tensor_gemm(layout, cuda(A), torch.tensor([sA], dtype=torch.float32, device=DEV), cuda(B),
                            torch.tensor([sB], dtype=torch.float32, device=DEV), M, N, K, batch=batch,
                            strideA=strideA, strideB=strideB, out=out)
    torch.cuda.synchronize()
    check_guards(buf)
    assert spg.last_device_error() == 0
    return to_f64(y).reshape(batch, M, N)


@pytest.mark.parametrize("layout", ["NT", "NN", "TN", "TT"])
@pytest.mark.parametrize("M,N,K,batch", [(144, 272, 160, 1), (64, 128, 512, 2), (256, 528, 1040, 1),
                                         (16, 16, 16, 3), (400, 784, 384, 2)])
def test_tensor_layouts(layout, M, N, K, batch, variant):
    A, sA, B, sB = tensor_inputs(layout, M, N, K, batch, seed=M + N + K)
    y = run_tensor(layout, A, sA, B, sB, M, N, K, batch)
    # the oracle's layout letters are NT / NN / TN; TT is A^T . B^T, i.e. TN with B as [N, K]
    ol = {"NT": "NT", "NN": "NN", "TN": "TN", "TT": None}[layout]
    if ol is None:
        # C = A^T B^T: transpose B on the host into [K, N] and use TN
        Bt = B.reshape(batch, N, K).transpose(0, 2, 1).reshape(-1)
        ref = oracle.fp8_tensor_gemm("TN", A, sA, Bt, sB, M, N, K, batch=batch)
    else:
        ref = oracle.fp8_tensor_gemm(ol, A, sA, B, sB, M, N, K, batch=batch)
    assert_within_tol(y, ref, f"tensor {layout} {M}x{N}x{K}x{batch}")


@pytest.mark.parametrize("layout", ["NT", "NN"])
def test_tensor_broadcast_stride0(layout, variant):
    M, N, K, batch = 128, 256, 256, 3
    A, sA, B, sB = tensor_inputs(layout, M, N, K, batch, seed=11)
    B0 = B[: N * K]
    y = run_tensor(layout, A, sA, B0, sB, M, N, K, batch, strideB=0)
    ref = oracle.fp8_tensor_gemm(layout, A, sA, B0, sB, M, N, K, batch=batch, strideB=0)
    assert_within_tol(y, ref, "broadcast B")


@pytest.mark.parametrize("layout,M,N,K,batch", [
    ("NT", 512, 512, 512, 1), ("NT", 64, 8192, 2048, 1), ("NT", 1024, 1536, 2048, 1),
    ("NT", 2048, 6912, 1536, 1), ("NN", 2048, 1536, 6912, 1), ("TN", 6912, 1536, 2048, 1),
    ("NT", 512, 512, 512, 64), ("NT", 1024, 1024, 2048, 8), ("NT", 4096, 4096, 4096, 1)])
def test_tensor_workload_shapes_sampled(layout, M, N, K, batch):
    A, sA, B, sB = tensor_inputs(layout, M, N, K, batch, seed=7)
    y = run_tensor(layout, A, sA, B, sB, M, N, K, batch)
    assert not np.isnan(y).any()
    rows = _sample_rows(M, n=4)
    ref = oracle.fp8_tensor_gemm(layout, A, sA, B, sB, M, N, K, batch=batch, rows=rows)
    assert_within_tol(y[:, rows, :], ref, f"tensor {layout} {M}x{N}x{K}x{batch}")


@pytest.mark.parametrize("epi", ["add", "swiglu"])
def test_nvfp4_pair_kernels_agree_and_repeat(epi, monkeypatch):
    """The two NVFP4 pair kernels differ only in how the scale factors reach
    TMEM, so their outputs must agree bit for bit -- on every one of many
    repeated launches (a missed ordering between the scale stores, the
    residual copies or the accumulator hand-over shows up as a run that
    differs).  Shapes with short K give frequent tile changes."""
    T, N, K = 4096, 5120, 5120
    A, sfA, gA, W, sfW, gW = nvfp4_inputs(T, N, K, seed=91)
    res = normal_bf16((T, N), seed=92) if epi == "add" else None
    dA, dW = cuda(A), cuda(W)
    dsA, dsW = cuda(sf_rowmajor_to_blocked(sfA, T, K)), cuda(sf_rowmajor_to_blocked(sfW, N, K))
    tgA = torch.tensor([gA], dtype=torch.float32, device=DEV)
    tgW = torch.tensor([gW], dtype=torch.float32, device=DEV)
    dr = None if res is None else cuda_bf16(res)
    monkeypatch.setenv("SPG_FORCE_VARIANT", "2sm_cp")
    base = spg.nvfp4_gemm(dA, dsA, tgA, dW, dsW, tgW, residual=dr, epilogue=epi).clone()
    monkeypatch.setenv("SPG_FORCE_VARIANT", "2sm_st")
    for _ in range(12):
        y = spg.nvfp4_gemm(dA, dsA, tgA, dW, dsW, tgW, residual=dr, epilogue=epi)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), base.view(torch.int16))
    assert spg.last_device_error() == 0
    rows = _sample_rows(T, n=4)
    ref = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, epi, rows=rows)
    assert_within_tol(to_f64(base[torch.from_numpy(rows).to(DEV)]), ref, f"nvfp4 {epi} repeat")


@pytest.mark.parametrize("epi", ["add", "swiglu"])
def test_nvfp4_multicast_kernel_repeats(epi, monkeypatch):
    """The multicast-cluster NVFP4 kernel (one-CTA MMAs, weight tile shared
    by multicast, scales stored by each CTA's own warps) gives the same bits
    on every one of many launches -- a missed ordering between the scale
    stores, the two producers' multicast copies, the residual copies or the
    accumulator hand-back shows up as a launch that differs -- and matches
    the oracle."""
    T, N, K = 4096, 5120, 5120
    A, sfA, gA, W, sfW, gW = nvfp4_inputs(T, N, K, seed=93)
    res = normal_bf16((T, N), seed=94) if epi == "add" else None
    dA, dW = cuda(A), cuda(W)
    dsA, dsW = cuda(sf_rowmajor_to_blocked(sfA, T, K)), cuda(sf_rowmajor_to_blocked(sfW, N, K))
    tgA = torch.tensor([gA], dtype=torch.float32, device=DEV)
    tgW = torch.tensor([gW], dtype=torch.float32, device=DEV)
    dr = None if res is None else cuda_bf16(res)
    monkeypatch.setenv("SPG_FORCE_VARIANT", "2sm_mc")
    assert spg.select_route("nvfp4", T, N, K, epi)["variant"] == 5
    base = spg.nvfp4_gemm(dA, dsA, tgA, dW, dsW, tgW, residual=dr, epilogue=epi).clone()
    for _ in range(12):
        y = spg.nvfp4_gemm(dA, dsA, tgA, dW, dsW, tgW, residual=dr, epilogue=epi)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), base.view(torch.int16))
    assert spg.last_device_error() == 0
    rows = _sample_rows(T, n=4)
    ref = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, epi, rows=rows)
    assert_within_tol(to_f64(base[torch.from_numpy(rows).to(DEV)]), ref, f"nvfp4 mc {epi} repeat")
