"""The allocation-free per-tensor FP8 quantizer, called through the C ABI.

Some callers cannot allocate device memory for the amax scratch that
spg_quantize_fp8_tensor takes (latency-critical paths where an allocator call
may block or fail, programs under a device-memory budget that forbids new
allocations, foreign-language callers without a device allocator);
spg_quantize_fp8_tensor_noalloc keeps that scratch in a static device array
inside the library.  Its codes and scale must equal those of
the scratch-taking entry point bit for bit, on two calls in a row with
different inputs (so a stale scratch from the first call would show), and it
must reject inputs beyond its stated maximum.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import scaled_precision_gemm_gb300 as spg
from synthetic_inputs import normal_bf16

pytestmark = pytest.mark.gpu


def _bf16(shape, seed, std):
    bits = normal_bf16(shape, seed=seed, std=std)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_quantizer_matches_scratch_entry_point_twice():
    lib = spg.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # first call: a large tensor (many partial maxima); second: a small one
    for shape, seed, std in [((1536, 6912), 31, 3.0), ((24, 520), 32, 0.5)]:
        x = _bf16(shape, seed, std)
        codes = torch.empty(shape, dtype=torch.uint8, device="cuda")
        scale = torch.empty(4, dtype=torch.float32, device="cuda")
        st = lib.spg_quantize_fp8_tensor_noalloc(_p(x), x.numel(), _p(codes), _p(scale), stream)
        assert st == 0, spg.status_string(st)
        ref_codes, ref_scale = spg.quantize_fp8_tensor(x)
        torch.cuda.synchronize()
        assert scale[0].item() == ref_scale.item()
        assert torch.equal(codes, ref_codes)
    assert spg.last_device_error() == 0


def test_noalloc_quantizer_rejects_oversize_input():
    lib = spg.load_library()
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    codes = torch.empty(16, dtype=torch.uint8, device="cuda")
    scale = torch.empty(4, dtype=torch.float32, device="cuda")
    too_big = 4096 * 65536 + 8
    st = lib.spg_quantize_fp8_tensor_noalloc(_p(x), too_big, _p(codes), _p(scale), None)
    assert spg.status_string(st) == "SPG_ERR_UNSUPPORTED_SHAPE"
