"""NVFP4 one-CTA tiles with the K split inside thread-block clusters (route
variant 7) against the CPU oracle.

Every tile is reduced by split_k CTAs of one cluster, which sum their pieces
through distributed shared memory in split order; only the order of the fp32
sums differs from the plain route, so the bar is the same element-wise
tolerance.  Besides parity: the result repeats bit for bit, needs no
workspace, and replays inside a CUDA graph.
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


@pytest.fixture(params=["1sm_cks", "1sm256_cks"])
def kernel(request, monkeypatch):
    monkeypatch.setenv("SPG_FORCE_VARIANT", request.param)
    return request.param


def nvfp4_inputs(T, N, K, seed):
    x = normal_bf16((T, K), seed=seed)
    w = normal_bf16((N, K), seed=seed + 1)
    gA = oracle.nvfp4_global_scale(x)
    gW = oracle.nvfp4_global_scale(w)
    A, sfA = oracle.quantize_nvfp4(x, gA)
    W, sfW = oracle.quantize_nvfp4(w, gW)
    return A, sfA, gA, W, sfW, gW


def device_inputs(A, sfA, gA, W, sfW, gW):
    T, N, K = A.shape[0], W.shape[0], 2 * A.shape[1]
    return (cuda(A), cuda(sf_rowmajor_to_blocked(sfA, T, K)),
            torch.tensor([gA], dtype=torch.float32, device=DEV),
            cuda(W), cuda(sf_rowmajor_to_blocked(sfW, N, K)),
            torch.tensor([gW], dtype=torch.float32, device=DEV))


def run(dev_in, res, epi, bias=None):
    y = spg.nvfp4_gemm(*dev_in, residual=res, epilogue=epi, bias=bias)
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    return y


def expect_cluster_route(T, N, K, epi, kernel):
    r = spg.select_route("nvfp4", T, N, K, epi)
    assert r["variant"] == 7 and r["block_m"] == 128, r
    assert r["block_n"] == (256 if kernel == "1sm256_cks" else 128), r
    assert 2 <= r["split_k"] <= 4 and r["workspace_bytes"] == 0, r
    tiles = -(-T // 128) * -(-N // r["block_n"])
    assert r["grid"] == tiles * r["split_k"] <= torch.cuda.get_device_properties(0).multi_processor_count
    return r


@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
@pytest.mark.parametrize("T,N,K", [(1, 16, 4096), (64, 512, 6144), (200, 272, 8192),
                                   (129, 384, 4352), (333, 400, 4096), (256, 640, 6144)])
@pytest.mark.parametrize("bias", [False, True])
def test_cluster_split_ragged(T, N, K, epi, bias, kernel):
    r = expect_cluster_route(T, N, K, epi, kernel)
    A, sfA, gA, W, sfW, gW = nvfp4_inputs(T, N, K, seed=T + N + K)
    res = normal_bf16((T, N), seed=91) if epi == "add" else None
    b = normal_bf16((N,), seed=92, std=2.0) if bias else None
    y = run(device_inputs(A, sfA, gA, W, sfW, gW), None if res is None else cuda_bf16(res), epi,
            None if b is None else cuda_bf16(b))
    ref = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, epi, bias=b)
    assert_within_tol(to_f64(y), ref, f"nvfp4 cluster split {r['split_k']} {epi} {T}x{N}x{K}")


def test_cluster_split_repeats_bit_for_bit(kernel):
    T, N, K = 100, 1024, 8192
    expect_cluster_route(T, N, K, "add", kernel)
    dev_in = device_inputs(*nvfp4_inputs(T, N, K, seed=5))
    res = cuda_bf16(normal_bf16((T, N), seed=6))
    y0 = run(dev_in, res, "add")
    for _ in range(20):
        assert torch.equal(run(dev_in, res, "add"), y0)


def test_cluster_split_cuda_graph_replay(kernel):
    T, N, K = 48, 768, 6144
    expect_cluster_route(T, N, K, "linear", kernel)
    dev_in = device_inputs(*nvfp4_inputs(T, N, K, seed=7))
    y_eager = run(dev_in, None, "linear")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run(dev_in, None, "linear")  # warm-up (tensor maps, kernel attributes)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        y = spg.nvfp4_gemm(*dev_in, epilogue="linear")
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    assert torch.equal(y, y_eager)


@pytest.mark.parametrize("T", [16, 64, 128, 256])
@pytest.mark.parametrize("epi", ["add", "swiglu"])
def test_cluster_split_full_size_sampled(T, epi, kernel):
    """Narrow T at the bench's K = 17408 (linear_add N = 5120; SwiGLU at
    N = 2048, whose tiles still fit one split wave), sampled rows against the
    oracle."""
    K = 17408
    N = 5120 if epi == "add" else 2048
    tiles = -(-T // 128) * -(-N // (256 if kernel == "1sm256_cks" else 128))
    if 2 * tiles > torch.cuda.get_device_properties(0).multi_processor_count:
        pytest.skip("too many tiles for a split in one wave")
    expect_cluster_route(T, N, K, epi, kernel)
    A, sfA, gA, W, sfW, gW = nvfp4_inputs(T, N, K, seed=T + 3)
    res = normal_bf16((T, N), seed=93) if epi == "add" else None
    y = run(device_inputs(A, sfA, gA, W, sfW, gW), None if res is None else cuda_bf16(res), epi)
    rows = np.unique(np.array([0, 1, 31, 32, 63, T // 2, 127, 128, 200, T - 1], np.int64) % T)
    ref = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, res, epi, rows=rows)
    assert_within_tol(to_f64(y[torch.from_numpy(rows).to(DEV)]), ref,
                      f"nvfp4 cluster split T={T} {epi}")
