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


# ---------------------------------------------------------------------------
# Quotients x / s placed exactly on and around the points where a code's
# rounding changes (ties to even), in the subnormal E4M3 range, and behind a
# subnormal scale: any encoder that forms the quotient other than as one
# IEEE-rounded division fails here first.

def _bf16_rows(rows_f32):
    return f32_to_bf16_bits(np.asarray(rows_f32, np.float32))


def test_fp8_rows_quotients_on_rounding_points():
    e4m3_mid = [1.0625, 1.1875, 1.3125, 1.4375, 1.5625, 1.6875, 1.8125, 1.9375]
    rows = []
    for j in range(-6, 7):
        scale = 2.0 ** j
        r = [448.0 * scale]                                    # amax: s = 2^j exactly
        for m in e4m3_mid:
            for e in range(-5, 9):                             # every normal E4M3 binade
                v = m * 2.0 ** e * scale
                if v < 448.0 * scale:
                    r += [v, -v]
        r += [464.0 * scale * 0.999, 0.0, -0.0]                # near the saturation midpoint
        r += [0.9375 * 2.0 ** -6 * scale, 2.0 ** -10 * scale, 3 * 2.0 ** -10 * scale]  # subnormal E4M3
        rows.append(r)
    width = max(len(r) for r in rows)
    width = (width + 7) // 8 * 8
    x = np.zeros((len(rows), width), np.float32)
    for i, r in enumerate(rows):
        x[i, :len(r)] = r
    xb = _bf16_rows(x)
    codes, scales = spg.quantize_fp8_rows(cuda_bf16(xb))
    oc, os_ = oracle.quantize_fp8_rows(xb)
    assert np.array_equal(scales.cpu().numpy(), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


def test_fp8_rows_many_scales_and_a_subnormal_scale():
    """16M quotients over 4096 rows of different scales (so x * fl(1/s)
    lands within a few ulp of a midpoint for some of them), a row whose
    scale is subnormal (its reciprocal overflows), and rows whose small
    values fall in the subnormal E4M3 range."""
    rows, K = 4096, 4096
    x = bf16_bits_to_f32(normal_bf16((rows, K), seed=4242)).copy()
    rng = np.random.default_rng(7)
    x *= (2.0 ** rng.uniform(-20, 20, size=(rows, 1))).astype(np.float32)
    x[0] = 0.0
    x[0, :16] = 1e-39 * np.arange(1, 17)                       # subnormal bf16 values, subnormal s
    x[1, 1:] *= 1e-4                                           # quotients below 2^-6
    x[1, 0] = 1000.0
    xb = f32_to_bf16_bits(x)
    codes, scales = spg.quantize_fp8_rows(cuda_bf16(xb))
    oc, os_ = oracle.quantize_fp8_rows(xb)
    assert np.array_equal(scales.cpu().numpy(), os_)
    bad = np.argwhere(codes.cpu().numpy() != oc)
    assert bad.size == 0, f"{len(bad)} codes differ, first {bad[:5].tolist()}"
    # the per-tensor and delayed encoders share the code path
    ct, st = spg.quantize_fp8_tensor(cuda_bf16(xb))
    oct_, ost = oracle.quantize_fp8_tensor(xb)
    assert st.item() == float(ost) and np.array_equal(ct.cpu().numpy(), oct_)


def test_nvfp4_quotients_on_rounding_points():
    """Blocks whose E4M3 scale decodes to a power of two (g = 1), so x / d is
    exactly an E2M1 rounding point (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) or a
    representable value, in both signs."""
    pts = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 0.125]
    K = 64
    rows = []
    for k in range(-8, 9):
        d = 2.0 ** k
        for sign in (1.0, -1.0):
            blk = [6.0 * d * sign] + [sign * p * d for p in pts]    # amax_b = 6d -> sf = d
            blk = (blk + [0.0] * 16)[:16]
            rows.append(blk * (K // 16))
    x = _bf16_rows(np.array(rows, np.float32))
    g = torch.ones(1, dtype=torch.float32, device=DEV)
    codes, sf = spg.quantize_nvfp4(cuda_bf16(x), g)
    oc, osf = oracle.quantize_nvfp4(x, 1.0)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(sf_blocked_to_rowmajor(sf.cpu().numpy(), len(rows), K), osf)


def test_nvfp4_many_blocks_bit_exact():
    rows, K = 2048, 8192
    x = bf16_bits_to_f32(normal_bf16((rows, K), seed=777)).copy()
    rng = np.random.default_rng(8)
    x *= (2.0 ** rng.uniform(-8, 8, size=(rows, K // 16, 1))).astype(np.float32).repeat(16, 2).reshape(rows, K)
    xb = f32_to_bf16_bits(x)
    g = spg.nvfp4_global_scale(cuda_bf16(xb))
    og = oracle.nvfp4_global_scale(xb)
    assert g.item() == float(og)
    codes, sf = spg.quantize_nvfp4(cuda_bf16(xb), g)
    oc, osf = oracle.quantize_nvfp4(xb, og)
    bad = np.argwhere(codes.cpu().numpy() != oc)
    assert bad.size == 0, f"{len(bad)} code bytes differ, first {bad[:5].tolist()}"
    assert np.array_equal(sf_blocked_to_rowmajor(sf.cpu().numpy(), rows, K), osf)


@pytest.mark.parametrize("rows,K", [(1, 64), (3, 1024), (4, 17408), (7, 5120), (5, 17408),
                                    (64, 2048), (30, 17408), (85, 6144), (129, 5120),
                                    (130, 6144), (128, 17408)])
def test_nvfp4_act_quantizer(rows, K):
    """Global scale + block quantizer in one call: one CTA up to 73,728
    elements, one cluster up to 512 Ki elements, the two-pass kernels beyond;
    bit-exact against the oracle and identical to the two calls, padding
    scale rows zero."""
    x = normal_bf16((rows, K), seed=rows * 5 + K)
    xf = bf16_bits_to_f32(x).copy()
    xf[0, :16] = 0.0                           # an all-zero block
    if rows > 1:
        xf[1, 16:32] *= 1e-7                   # a block whose scale underflows
    x = f32_to_bf16_bits(xf)
    xd = cuda_bf16(x)
    codes, sf, g = spg.quantize_nvfp4_act(xd)
    og = oracle.nvfp4_global_scale(x)
    assert g.item() == float(og)
    oc, osf = oracle.quantize_nvfp4(x, og)
    assert np.array_equal(codes.cpu().numpy(), oc)
    blocked = sf.cpu().numpy()
    assert np.array_equal(sf_blocked_to_rowmajor(blocked, rows, K), osf)
    g2 = spg.nvfp4_global_scale(xd)
    c2, s2 = spg.quantize_nvfp4(xd, g2)
    assert torch.equal(codes, c2) and torch.equal(sf, s2)
    assert spg.last_device_error() == 0
