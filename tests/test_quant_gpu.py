"""GPU quantizers against the CPU oracle: codes and scales bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import scaled_precision_gemm_gb300 as spg
from synthetic_inputs import bf16_bits_to_f32, f32_to_bf16_bits, normal_bf16
from tests.gpu_common import DEV, cuda_bf16
from tests.helpers import sf_blocked_to_rowmajor

pytestmark = pytest.mark.gpu


def _special_rows(x):
    xf = bf16_bits_to_f32(x).copy()
    if xf.shape[0] > 4:
        xf[1] = 0.0                         # all-zero row
        xf[2] = 0.0
        xf[2, -1] = -5.0                    # a single non-zero at the end
        xf[3] *= 1e-30                      # tiny values (subnormal codes)
        xf[4] *= 3e4
    return f32_to_bf16_bits(xf)


@pytest.mark.parametrize("rows,K", [(1, 8), (7, 40), (64, 256), (129, 5120), (33, 17408),
                                    (5, 24576)])
def test_fp8_rows_bit_exact(rows, K):
    x = _special_rows(normal_bf16((rows, K), seed=rows * 7 + K))
    codes, scales = spg.quantize_fp8_rows(cuda_bf16(x))
    oc, os_ = oracle.quantize_fp8_rows(x)
    got = codes.cpu().numpy()
    assert np.array_equal(scales.cpu().numpy(), os_)
    bad = np.argwhere(got != oc)
    assert bad.size == 0, f"{len(bad)} codes differ, first {bad[:5].tolist()}"


@pytest.mark.parametrize("shape", [(16,), (3, 40), (257, 96), (1024, 1536)])
def test_fp8_tensor_bit_exact(shape):
    x = normal_bf16(shape, seed=sum(shape))
    codes, scale = spg.quantize_fp8_tensor(cuda_bf16(x))
    oc, os_ = oracle.quantize_fp8_tensor(x)
    assert scale.item() == float(os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


def test_fp8_tensor_all_zero():
    x = np.zeros((4, 64), np.uint16)
    codes, scale = spg.quantize_fp8_tensor(cuda_bf16(x))
    assert scale.item() == 1.0 and not codes.cpu().numpy().any()


@pytest.mark.parametrize("rows,K", [(1, 64), (128, 256), (129, 5120), (300, 6144), (37, 17408)])
def test_nvfp4_bit_exact(rows, K):
    x = normal_bf16((rows, K), seed=rows + 3 * K)
    xf = bf16_bits_to_f32(x).copy()
    xf[0, 16:32] = 0.0                   # an all-zero block
    if rows > 2:
        xf[2, :16] *= 1e-7               # a block whose scale underflows
    x = f32_to_bf16_bits(xf)
    g = spg.nvfp4_global_scale(cuda_bf16(x))
    og = oracle.nvfp4_global_scale(x)
    assert g.item() == float(og)
    codes, sf = spg.quantize_nvfp4(cuda_bf16(x), g)
    oc, osf = oracle.quantize_nvfp4(x, og)
    assert np.array_equal(codes.cpu().numpy(), oc)
    blocked = sf.cpu().numpy()
    assert np.array_equal(sf_blocked_to_rowmajor(blocked, rows, K), osf)
    # padding rows of the blocked layout are zero
    mask = np.ones(blocked.size, bool)
    r = np.arange(rows)[:, None]
    c = np.arange(K // 16)[None, :]
    kt = K // 64
    mask[((r // 128) * kt + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)] = False
    assert not blocked[mask].any()


def test_nvfp4_explicit_global_scale():
    # the quantizer takes g as an input: with g = 1 it is the one-level scheme
    x = normal_bf16((8, 128), seed=99)
    g = torch.ones(1, dtype=torch.float32, device=DEV)
    codes, sf = spg.quantize_nvfp4(cuda_bf16(x), g)
    oc, osf = oracle.quantize_nvfp4(x, 1.0)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(sf_blocked_to_rowmajor(sf.cpu().numpy(), 8, 128), osf)
