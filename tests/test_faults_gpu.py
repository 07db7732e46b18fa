"""Failure detection without a GPU fault.

Every in-kernel wait is bounded in time.  With the test hook
spg_debug_inject_stall, the epilogue of every GEMM kernel waits on a barrier
that nothing arrives on (a flag nothing sets), under a 20 ms bound: the wait
runs out, the kernel records the code in the device error word, the producer
and MMA roles see the abort flag, drain the copies and MMAs in flight, free
tensor memory and return.  The host must read SPG_ERR_TIMEOUT and the context
must stay usable for a correct call right after.
"""
import numpy as np
import pytest
import torch

import oracle
import scaled_precision_gemm_gb300 as spg
from synthetic_inputs import normal_bf16
from tests.gpu_common import DEV, cuda, to_f64
from tests.helpers import assert_within_tol

pytestmark = pytest.mark.gpu

INJECTED = 0x106


def _inputs(T, N, K):
    A, sa = oracle.quantize_fp8_rows(normal_bf16((T, K), seed=0))
    W, sw = oracle.quantize_fp8_rows(normal_bf16((N, K), seed=1))
    return A, sa, W, sw


def test_wait_timeout_is_reported_and_context_survives(monkeypatch):
    monkeypatch.setenv("SPG_FORCE_VARIANT", "1sm256")
    T, N, K = 512, 512, 4096
    A, sa, W, sw = _inputs(T, N, K)
    args = (cuda(A), cuda(sa), cuda(W), cuda(sw))
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    spg.set_wait_timeout_ns(20_000_000)
    spg.debug_inject_stall(True)
    try:
        spg.fp8_rowscaled_gemm(*args)
        code = spg.last_device_error_code()
    finally:
        spg.debug_inject_stall(False)
        spg.set_wait_timeout_ns(2_000_000_000)
    assert code == INJECTED, hex(code)
    assert spg.last_device_error() == 0          # reading the code cleared it
    # the context is intact: the same call now completes and is correct
    y = spg.fp8_rowscaled_gemm(*args)
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    assert_within_tol(to_f64(y), oracle.fp8_rowscaled_gemm(A, sa, W, sw), "after time-out")


def _nvfp4_inputs(T, N, K):
    from tests.helpers import sf_rowmajor_to_blocked
    x, w = normal_bf16((T, K), seed=0), normal_bf16((N, K), seed=1)
    gA, gW = oracle.nvfp4_global_scale(x), oracle.nvfp4_global_scale(w)
    A, sfA = oracle.quantize_nvfp4(x, gA)
    W, sfW = oracle.quantize_nvfp4(w, gW)
    dev = (cuda(A), cuda(sf_rowmajor_to_blocked(sfA, T, K)),
           torch.tensor([gA], dtype=torch.float32, device=DEV), cuda(W),
           cuda(sf_rowmajor_to_blocked(sfW, N, K)),
           torch.tensor([gW], dtype=torch.float32, device=DEV))
    return (A, sfA, gA, W, sfW, gW), dev


@pytest.mark.parametrize("variant", ["2sm", "swap", "2sm_cp", "2sm_st", "2sm_mc"])
def test_pair_kernel_timeout_is_reported_and_context_survives(variant, monkeypatch):
    """The same check on the two-SM kernels: both CTAs' epilogues stall, every
    wait of the pair runs out or sees the abort, the two producers settle
    their copies on the leader's barriers and the pair exits cleanly."""
    monkeypatch.setenv("SPG_FORCE_VARIANT", variant)
    if variant in ("2sm", "swap"):
        T, N, K = (64, 1024, 4096) if variant == "swap" else (512, 512, 4096)
        A, sa, W, sw = _inputs(T, N, K)
        args = (cuda(A), cuda(sa), cuda(W), cuda(sw))
        call = lambda: spg.fp8_rowscaled_gemm(*args)
        ref = lambda: oracle.fp8_rowscaled_gemm(A, sa, W, sw)
        assert spg.select_route("fp8_rowscaled", T, N, K)["swap_ab"] == (variant == "swap")
    else:
        T, N, K = 512, 512, 4096
        host, dev = _nvfp4_inputs(T, N, K)
        call = lambda: spg.nvfp4_gemm(*dev)
        ref = lambda: oracle.nvfp4_gemm(*host)
        assert spg.select_route("nvfp4", T, N, K)["variant"] == {"2sm_cp": 0, "2sm_st": 3,
                                                                 "2sm_mc": 5}[variant]
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    spg.set_wait_timeout_ns(20_000_000)
    spg.debug_inject_stall(True)
    try:
        call()
        code = spg.last_device_error_code()
    finally:
        spg.debug_inject_stall(False)
        spg.set_wait_timeout_ns(2_000_000_000)
    # In the warp-stored-scale kernels the stalled epilogue warps are also the
    # scale writers, so the MMA issuer's wait for the first stage's scales
    # (0x102, ring slot full) and the producer's wait for a ring slot the
    # MMAs never free (0x101, ring slot free) start at about the same time as
    # the injected wait and run out with it; whichever expires first is
    # recorded.
    expected = {INJECTED, 0x101, 0x102} if variant in ("2sm_st", "2sm_mc") else {INJECTED}
    assert code in expected, hex(code)
    assert spg.last_device_error() == 0
    y = call()
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    assert_within_tol(to_f64(y), ref(), f"{variant} after time-out")


def test_cluster_split_timeout_is_reported_and_context_survives(monkeypatch):
    """The NVFP4 one-CTA tiles with the K split inside clusters: every CTA's
    epilogue stalls, so none reaches the reduction; each still gives its
    arrivals on its peers' barriers on the way out and waits (bounded) for
    theirs, so no CTA leaves while a peer may still write into it."""
    monkeypatch.delenv("SPG_FORCE_VARIANT", raising=False)
    T, N, K = 64, 512, 6144
    host, dev = _nvfp4_inputs(T, N, K)
    r = spg.select_route("nvfp4", T, N, K)
    assert r["variant"] == 7 and r["split_k"] == 3, r
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    spg.set_wait_timeout_ns(20_000_000)
    spg.debug_inject_stall(True)
    try:
        spg.nvfp4_gemm(*dev)
        code = spg.last_device_error_code()
    finally:
        spg.debug_inject_stall(False)
        spg.set_wait_timeout_ns(2_000_000_000)
    assert code == INJECTED, hex(code)
    assert spg.last_device_error() == 0
    y = spg.nvfp4_gemm(*dev)
    torch.cuda.synchronize()
    assert spg.last_device_error() == 0
    assert_within_tol(to_f64(y), oracle.nvfp4_gemm(*host), "cluster split after time-out")


def test_status_codes_are_distinct_for_host_errors():
    with pytest.raises(spg.SpgError) as e:
        spg.fp8_rowscaled_gemm(torch.zeros((4, 24), dtype=torch.uint8, device=DEV),
                               torch.ones(4, device=DEV),
                               torch.zeros((8, 24), dtype=torch.uint8, device=DEV),
                               torch.ones(8, device=DEV))
    assert e.value.status == 2          # K % 16
