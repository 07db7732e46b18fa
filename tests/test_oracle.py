"""Pins of the CPU oracle against facts fixed outside it (no GPU).

Each pin comes from something other than the oracle's own code: the golden
fixtures worked by hand from the format definitions, PyTorch's float8_e4m3fn
conversion (a library routine), a binade-wise numpy formulation of E2M1
rounding, exact rational arithmetic with ``fractions`` on tiny shapes, and
algebraic invariants (identity, one-hot, linearity, power-of-two scaling).
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from synthetic_inputs import bf16_bits_to_f32, f32_to_bf16_bits, normal_bf16, random_codes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def torch_e4m3_values(codes):
    c = torch.tensor(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return c.to(torch.float64).numpy()


def torch_e4m3_encode(x_f32):
    t = torch.tensor(np.asarray(x_f32, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def e2m1_binade_round(q):
    """E2M1 round-to-nearest-even written per binade with numpy's half-even round.

    [0,2): step 0.5; [2,4): step 1; [4,6]: step 2; above 6 saturates."""
    q = np.asarray(q, np.float64)
    a = np.abs(q)
    out = np.where(a < 2.0, np.round(a * 2.0) / 2.0,
                   np.where(a < 4.0, np.round(a), 2.0 * np.round(a / 2.0)))
    out = np.minimum(out, 6.0)
    return np.where(np.signbit(q), -out, out)


E2M1_CODE_OF = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}


# ---------------------------------------------------------------- decode
def test_e4m3_decode_all_codes_match_torch():
    ours = oracle.e4m3_table()
    ref = torch_e4m3_values(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    assert sorted(np.flatnonzero(nan).tolist()) == [0x7F, 0xFF]


def test_e4m3_golden_facts():
    for code, val in _lines("e4m3fn_facts.txt"):
        v = oracle.e4m3_value(int(code, 16))
        if val == "nan":
            assert np.isnan(v), code
        else:
            assert v == float(val) and np.signbit(v) == val.startswith("-"), code
    finite = oracle.e4m3_table()
    assert np.nanmax(finite) == 448.0 and np.nanmin(finite) == -448.0


def test_e2m1_golden_table():
    for code, val in _lines("e2m1_values.txt"):
        v = oracle.e2m1_value(int(code))
        assert v == float(val) and np.signbit(v) == val.startswith("-"), code


# ---------------------------------------------------------------- encode
def _e4m3_probe_values():
    mags = np.array(sorted(set(abs(v) for v in oracle.e4m3_table() if np.isfinite(v))))
    mids = (mags[:-1] + mags[1:]) / 2.0
    pts = np.concatenate([mags, mids])
    f = pts.astype(np.float32)
    nudged = np.concatenate([f, np.nextafter(f, np.float32(0)), np.nextafter(f, np.float32(1e9))])
    rng = np.random.default_rng(1)
    rand = (rng.standard_normal(20000) * np.exp2(rng.integers(-12, 9, 20000))).astype(np.float32)
    allv = np.concatenate([nudged, -nudged, rand]).astype(np.float32)
    return allv[np.abs(allv) < 464.0]


def test_e4m3_encode_matches_torch_rne():
    xs = _e4m3_probe_values()
    ours = np.array([oracle.e4m3_encode(float(x)) for x in xs], np.uint8)
    ref = torch_e4m3_encode(xs)
    bad = np.flatnonzero(ours != ref)
    assert bad.size == 0, [(float(xs[i]), int(ours[i]), int(ref[i])) for i in bad[:10]]


def test_e4m3_encode_saturates_and_roundtrips():
    for x, code in [(448.0, 0x7E), (449.0, 0x7E), (470.0, 0x7E), (1e30, 0x7E), (-1e30, 0xFE),
                    (-460.0, 0xFE), (-0.0, 0x80), (-1e-12, 0x80), (1e-12, 0x00)]:
        assert oracle.e4m3_encode(x) == code, x
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_value(c)) == c


def test_e2m1_golden_ties():
    for x, code in _lines("e2m1_rne_ties.txt"):
        assert oracle.e2m1_encode(float(x)) == int(code), x


def test_e2m1_encode_matches_binade_rounding():
    rng = np.random.default_rng(2)
    grid = np.arange(-7.5, 7.5, 0.03125)
    xs = np.concatenate([grid, rng.uniform(-8, 8, 5000), rng.standard_normal(2000) * 0.3])
    for x in xs:
        code = oracle.e2m1_encode(float(x))
        ref = e2m1_binade_round(x)
        assert oracle.e2m1_value(code) == ref, x
        assert (code >> 3) == int(np.signbit(x)), x


def test_encoders_monotone():
    xs = np.linspace(-500, 500, 4001)
    v = [oracle.e4m3_value(oracle.e4m3_encode(x)) for x in xs]
    assert all(b >= a for a, b in zip(v, v[1:]))
    xs = np.linspace(-7, 7, 2801)
    v = [oracle.e2m1_value(oracle.e2m1_encode(x)) for x in xs]
    assert all(b >= a for a, b in zip(v, v[1:]))


# ------------------------------------------------------- FP8 quantizers
def test_fp8_rows_golden():
    rows = list(_lines("fp8_rows_worked_example.txt"))
    x0 = [float(v) for v in rows[0][1:]]
    c0 = [int(v, 16) for v in rows[1][1:]]
    s0 = float(rows[2][1])
    x1 = [float(v) for v in rows[3][1:]]
    c1 = [int(v, 16) for v in rows[4][1:]]
    x = f32_to_bf16_bits(np.array([x0, x1], np.float32))
    codes, scales = oracle.quantize_fp8_rows(x)
    assert codes[0].tolist() == c0 and codes[1].tolist() == c1
    assert scales[0] == np.float32(s0)
    assert scales[1] == np.float32(3) / np.float32(448)


def _fp8_rows_torch(x_bits):
    x = torch.tensor(bf16_bits_to_f32(x_bits))
    amax = x.abs().amax(dim=1, keepdim=True)
    s = torch.where(amax == 0, torch.ones_like(amax), amax / 448.0)
    q = x / s
    return q.to(torch.float8_e4m3fn).view(torch.uint8).numpy(), s[:, 0].numpy()


def test_fp8_rows_match_torch_conversion():
    x = normal_bf16((37, 200), seed=5)
    xf = bf16_bits_to_f32(x).copy()
    xf[3] = 0.0                       # all-zero row
    xf[4] = 0.0
    xf[4, 17] = -3.0                  # one non-zero element
    xf[5] *= 1e-30                    # tiny row (bf16 has fp32 range)
    xf[6] *= 3e4                      # large row
    x = f32_to_bf16_bits(xf)
    codes, scales = oracle.quantize_fp8_rows(x)
    rc, rs = _fp8_rows_torch(x)
    assert np.array_equal(scales, rs)
    assert np.array_equal(codes, rc)
    assert scales[3] == 1.0 and not codes[3].any()


def test_fp8_rows_invariants():
    x = normal_bf16((16, 512), seed=7)
    codes, scales = oracle.quantize_fp8_rows(x)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    table = oracle.e4m3_table()
    for r in range(16):
        i = np.argmax(np.abs(xf[r]))
        assert codes[r, i] in (0x7E, 0xFE)
        deq = table[codes[r]] * scales[r]
        # half a grid step of E4M3 at each magnitude: 2^-4 relative (normal
        # range) or 2^-10 * s absolute (subnormal range)
        bound = np.maximum(np.abs(xf[r]) * 2.0 ** -4, 2.0 ** -10 * scales[r]) * (1 + 1e-6)
        assert np.all(np.abs(deq - xf[r]) <= bound)
    for j in (-3, 1, 5):
        xs = f32_to_bf16_bits(bf16_bits_to_f32(x) * np.float32(2.0 ** j))
        c2, s2 = oracle.quantize_fp8_rows(xs)
        assert np.array_equal(c2, codes)
        assert np.array_equal(s2, scales * np.float32(2.0 ** j))


def test_fp8_tensor_matches_torch_conversion():
    x = normal_bf16((9, 333), seed=11)
    codes, s = oracle.quantize_fp8_tensor(x)
    xt = torch.tensor(bf16_bits_to_f32(x))
    st = xt.abs().amax() / 448.0
    ref = (xt / st).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert s == np.float32(st.item())
    assert np.array_equal(codes, ref)
    z, sz = oracle.quantize_fp8_tensor(np.zeros((3, 16), np.uint16))
    assert sz == 1.0 and not z.any()


# ----------------------------------------------------- NVFP4 quantizer
def test_nvfp4_golden_worked_example():
    rows = list(_lines("nvfp4_worked_example.txt"))
    g = float(rows[0][1])
    x = np.array([float(v) for r in rows[1:4] for v in r[1:]], np.float32).reshape(1, 48)
    sf_ref = [int(v, 16) for v in rows[4][1:]]
    codes_ref = [int(v) for r in rows[5:8] for v in r[1:]]
    packed_ref = [int(v, 16) for r in rows[8:11] for v in r[1:]]
    xb = f32_to_bf16_bits(x)
    assert np.array_equal(bf16_bits_to_f32(xb), x)   # the example is bf16-exact
    gg = oracle.nvfp4_global_scale(xb)
    assert gg == np.float32(g)
    codes, sf = oracle.quantize_nvfp4(xb, gg)
    assert sf[0].tolist() == sf_ref
    assert codes[0].tolist() == packed_ref
    unpacked = [(b >> (4 * h)) & 0xF for b in codes[0] for h in (0, 1)]
    assert unpacked == codes_ref


def test_nvfp4_matches_torch_and_binade_composition():
    x = normal_bf16((12, 256), seed=13)
    xf = bf16_bits_to_f32(x).copy()
    xf[2, 32:48] = 0.0                # an all-zero block
    xf[3, :16] *= 1e-6                # a block whose scale underflows E4M3
    x = f32_to_bf16_bits(xf)
    xf = bf16_bits_to_f32(x)
    g = oracle.nvfp4_global_scale(x)
    assert g == np.float32(np.abs(xf).max()) / np.float32(2688.0)
    codes, sf = oracle.quantize_nvfp4(x, g)
    xt = torch.tensor(xf).reshape(12, 16, 16)
    amax_b = xt.abs().amax(dim=2)
    t = (amax_b / 6.0) / torch.tensor(g)
    sf_ref = t.to(torch.float8_e4m3fn)
    assert np.array_equal(sf, sf_ref.view(torch.uint8).numpy())
    d = sf_ref.to(torch.float32) * torch.tensor(g)
    q = torch.where(d[..., None] == 0, torch.zeros_like(xt), xt / d[..., None])
    val = e2m1_binade_round(q.numpy().astype(np.float64)).reshape(12, 256)
    unpacked = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(12, 256)
    table = oracle.e2m1_table()
    assert np.array_equal(table[unpacked], val)


def test_nvfp4_invariants():
    x = normal_bf16((8, 512), seed=17)
    g = oracle.nvfp4_global_scale(x)
    codes, sf = oracle.quantize_nvfp4(x, g)
    xf = bf16_bits_to_f32(x).astype(np.float64).reshape(8, 32, 16)
    e4 = oracle.e4m3_table()
    e2 = oracle.e2m1_table()
    vals = e2[np.stack([codes & 0xF, codes >> 4], -1).reshape(8, 32, 16)]
    d = (e4[sf].astype(np.float32) * np.float32(g)).astype(np.float64)[..., None]
    # the block maximum always lands on +-6
    imax = np.argmax(np.abs(xf), axis=2)
    assert np.all(np.abs(np.take_along_axis(vals, imax[..., None], 2)) == 6.0)
    # dequant error within the grid spacing of its binade (1 d at most)
    q = np.abs(xf) / d
    step = np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    assert np.all(np.abs(vals * d - xf) <= np.maximum(step / 2, q - 6) * d * (1 + 1e-6))
    # the largest block scale of the tensor is 448 (the global scale maps it there)
    assert e4[sf].max() == 448.0
    # scaling the tensor by 2^j scales g by 2^j and leaves codes and sf unchanged
    for j in (-4, 3):
        xs = f32_to_bf16_bits(bf16_bits_to_f32(x) * np.float32(2.0 ** j))
        g2 = oracle.nvfp4_global_scale(xs)
        assert g2 == g * np.float32(2.0 ** j)
        c2, s2 = oracle.quantize_nvfp4(xs, g2)
        assert np.array_equal(c2, codes) and np.array_equal(s2, sf)


# ---------------------------------------------------------------- GEMMs
def _frac_e4m3(code):
    v = torch_e4m3_values([code])[0]
    return Fraction(float(v))


def _frac_e2m1(code):
    return Fraction(float(e2m1_binade_round(E2M1_VALUES[code])))


E2M1_VALUES = [0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6]


@pytest.mark.parametrize("T,N,K", [(3, 5, 32), (1, 1, 16), (4, 2, 48)])
def test_fp8_gemm_exact_vs_fractions(T, N, K):
    A = random_codes((T, K), seed=T * 100 + K, exclude=(0x7F, 0xFF))
    W = random_codes((N, K), seed=N * 1000 + K, exclude=(0x7F, 0xFF))
    sa = np.float32(np.linspace(0.5, 3.0, T))
    sw = np.float32(np.linspace(0.01, 0.2, N))
    out, acc = oracle.fp8_rowscaled_gemm(A, sa, W, sw, return_acc=True)
    for t in range(T):
        for n in range(N):
            exact = sum(_frac_e4m3(A[t, k]) * _frac_e4m3(W[n, k]) for k in range(K))
            assert Fraction(acc[t, n]) == exact
            ref = float(exact) * float(sa[t]) * float(sw[n])
            assert abs(out[t, n] - ref) <= 1e-15 * abs(ref) + 1e-300


def test_fp8_gemm_extreme_magnitudes_exact():
    K = 17408
    A = np.full((1, K), 0x7E, np.uint8)     # 448
    W = np.full((2, K), 0xFE, np.uint8)     # -448
    W[1, ::2] = 0x01                        # 2^-9 subnormal
    out, acc = oracle.fp8_rowscaled_gemm(A, np.ones(1, np.float32), W, np.ones(2, np.float32),
                                         return_acc=True)
    assert acc[0, 0] == -448.0 * 448.0 * K
    assert Fraction(acc[0, 1]) == Fraction(K // 2) * 448 * Fraction(1, 512) + (K // 2) * 448 * -448


def test_fp8_gemm_identity_and_onehot():
    K = 64
    A = random_codes((7, K), seed=3, exclude=(0x7F, 0xFF))
    sa = np.float32(np.linspace(0.25, 4, 7))
    Wid = np.zeros((K, K), np.uint8)
    np.fill_diagonal(Wid, 0x38)                # 1.0
    y = oracle.fp8_rowscaled_gemm(A, sa, Wid, np.ones(K, np.float32))
    deq = torch_e4m3_values(A.reshape(-1)).reshape(7, K) * sa[:, None].astype(np.float64)
    assert np.array_equal(y, deq)
    W = random_codes((9, K), seed=4, exclude=(0x7F, 0xFF))
    sw = np.float32(np.linspace(0.5, 1.5, 9))
    for k in (0, 17, K - 1):
        A1 = np.zeros((1, K), np.uint8)
        A1[0, k] = 0x38
        y = oracle.fp8_rowscaled_gemm(A1, np.ones(1, np.float32), W, sw)
        assert np.array_equal(y[0], torch_e4m3_values(W[:, k]) * sw.astype(np.float64))


def test_fp8_gemm_linearity_residual_and_swiglu():
    from scipy.special import expit
    T, N, K = 5, 12, 96
    x = normal_bf16((T, K), seed=0)
    w = normal_bf16((N, K), seed=1)
    A, sa = oracle.quantize_fp8_rows(x)
    W, sw = oracle.quantize_fp8_rows(w)
    y = oracle.fp8_rowscaled_gemm(A, sa, W, sw)
    assert np.array_equal(oracle.fp8_rowscaled_gemm(A, sa * 2, W, sw), 2 * y)
    assert np.array_equal(oracle.fp8_rowscaled_gemm(A, sa, W, sw * 4), 4 * y)
    zero = np.zeros((T, N), np.uint16)
    assert np.array_equal(oracle.fp8_rowscaled_gemm(A, sa, W, sw, zero, "add"), y)
    r = normal_bf16((T, N), seed=2)
    ya = oracle.fp8_rowscaled_gemm(A, sa, W, sw, r, "add")
    assert np.array_equal(ya, y + bf16_bits_to_f32(r).astype(np.float64))
    ys = oracle.fp8_rowscaled_gemm(A, sa, W, sw, epilogue="swiglu")
    gate, up = y[:, 0::2], y[:, 1::2]
    ref = gate * expit(gate) * up
    assert ys.shape == (T, N // 2)
    np.testing.assert_allclose(ys, ref, rtol=1e-13, atol=1e-300)
    sub = oracle.fp8_rowscaled_gemm(A, sa, W, sw, r, "add", rows=[4, 1])
    assert np.array_equal(sub, ya[[4, 1]])


def test_nvfp4_gemm_exact_vs_fractions():
    T, N, K = 3, 4, 64
    A = random_codes((T, K // 2), seed=21)
    W = random_codes((N, K // 2), seed=22)
    sfA = random_codes((T, K // 16), seed=23, exclude=tuple(range(0x60, 0x100)))
    sfW = random_codes((N, K // 16), seed=24, exclude=tuple(range(0x60, 0x100)))
    gA, gW = np.float32(0.75), np.float32(1.5)
    out, acc = oracle.nvfp4_gemm(A, sfA, gA, W, sfW, gW, return_acc=True)

    def elem(codes, sf, r, k):
        c = (int(codes[r, k // 2]) >> (4 * (k & 1))) & 0xF
        return Fraction(E2M1_VALUES[c]) * _frac_e4m3(sf[r, k // 16])

    for t in range(T):
        for n in range(N):
            exact = sum(elem(A, sfA, t, k) * elem(W, sfW, n, k) for k in range(K))
            assert Fraction(acc[t, n]) == exact
            assert out[t, n] == float(exact) * 0.75 * 1.5


def test_nvfp4_gemm_identity_linearity():
    K = 32
    x = normal_bf16((6, K), seed=31)
    gA = oracle.nvfp4_global_scale(x)
    A, sfA = oracle.quantize_nvfp4(x, gA)
    Wc = np.zeros((K, K // 2), np.uint8)
    for n in range(K):
        Wc[n, n // 2] |= 0x2 << (4 * (n & 1))  # E2M1 code 2 = 1.0 at column n
    sfW = np.full((K, K // 16), 0x38, np.uint8)   # E4M3 1.0
    y = oracle.nvfp4_gemm(A, sfA, gA, Wc, sfW, np.float32(1.0))
    e2 = np.array(E2M1_VALUES, np.float64)
    e4 = torch_e4m3_values(np.arange(256))
    deq = e2[np.stack([A & 0xF, A >> 4], -1).reshape(6, K)] * np.repeat(e4[sfA], 16, axis=1)
    assert np.array_equal(y, deq * float(gA))
    y2 = oracle.nvfp4_gemm(A, sfA, gA * 2, Wc, sfW, np.float32(1.0))
    assert np.array_equal(y2, 2 * y)


@pytest.mark.parametrize("layout", ["NT", "NN", "TN"])
def test_tensor_gemm_layouts_vs_fractions(layout):
    M, N, K, batch = 3, 4, 32, 2
    A = random_codes((batch, M * K), seed=41, exclude=(0x7F, 0xFF))
    B = random_codes((batch, N * K), seed=42, exclude=(0x7F, 0xFF))
    sA, sB = np.float32(0.5), np.float32(3.0)
    out = oracle.fp8_tensor_gemm(layout, A, sA, B, sB, M, N, K, batch=batch)
    for b in range(batch):
        a = A[b].reshape((K, M) if layout[0] == "T" else (M, K))
        bb = B[b].reshape((K, N) if layout[1] == "N" else (N, K))
        aM = a.T if layout[0] == "T" else a          # logical [M, K]
        bN = bb.T if layout[1] == "N" else bb         # logical [N, K]
        for m in range(M):
            for n in range(N):
                exact = sum(_frac_e4m3(aM[m, k]) * _frac_e4m3(bN[n, k]) for k in range(K))
                assert out[b, m, n] == float(exact) * 1.5
    # stride 0 broadcasts B across the batch
    o0 = oracle.fp8_tensor_gemm(layout, A, sA, B[0], sB, M, N, K, batch=batch, strideB=0)
    o1 = oracle.fp8_tensor_gemm(layout, A[1], sA, B[0], sB, M, N, K, batch=1)
    assert np.array_equal(o0[1], o1[0])


# ------------------------------------------------------------ fused bias
def test_bias_alone_bf16_and_fp8():
    """A = 0 leaves exactly the bias: bf16 values, or E4M3 x bias_scale rounded to fp32."""
    T, N, K = 3, 24, 32
    A = np.zeros((T, K), np.uint8)
    W = random_codes((N, K), seed=51, exclude=(0x7F, 0xFF))
    sa = np.ones(T, np.float32)
    sw = np.float32(np.linspace(0.5, 2, N))
    b16 = normal_bf16((N,), seed=52, std=3.0)
    y = oracle.fp8_rowscaled_gemm(A, sa, W, sw, bias=b16)
    assert np.array_equal(y, np.broadcast_to(bf16_bits_to_f32(b16).astype(np.float64), (T, N)))
    b8 = random_codes((N,), seed=53, exclude=(0x7F, 0xFF))
    scale = np.float32(0.37)
    y = oracle.fp8_rowscaled_gemm(A, sa, W, sw, bias=b8, bias_scale=scale)
    ref = (torch_e4m3_values(b8).astype(np.float32) * scale).astype(np.float64)
    assert np.array_equal(y, np.broadcast_to(ref, (T, N)))


def test_bias_is_added_after_scales_and_before_epilogue():
    from scipy.special import expit
    T, N, K = 4, 16, 64
    x = normal_bf16((T, K), seed=61)
    w = normal_bf16((N, K), seed=62)
    A, sa = oracle.quantize_fp8_rows(x)
    W, sw = oracle.quantize_fp8_rows(w)
    b = normal_bf16((N,), seed=63)
    bf = bf16_bits_to_f32(b).astype(np.float64)
    y = oracle.fp8_rowscaled_gemm(A, sa, W, sw)
    yb = oracle.fp8_rowscaled_gemm(A, sa, W, sw, bias=b)
    np.testing.assert_allclose(yb - y, np.broadcast_to(bf, (T, N)), rtol=0, atol=1e-12)
    r = normal_bf16((T, N), seed=64)
    ya = oracle.fp8_rowscaled_gemm(A, sa, W, sw, r, "add", bias=b)
    np.testing.assert_allclose(ya, yb + bf16_bits_to_f32(r), rtol=1e-15)
    ys = oracle.fp8_rowscaled_gemm(A, sa, W, sw, epilogue="swiglu", bias=b)
    g, u = yb[:, 0::2], yb[:, 1::2]
    np.testing.assert_allclose(ys, g * expit(g) * u, rtol=1e-13)
    # the same bias on the NVFP4 and per-tensor GEMMs
    gA = oracle.nvfp4_global_scale(x)
    gW = oracle.nvfp4_global_scale(w)
    An, sfA = oracle.quantize_nvfp4(x, gA)
    Wn, sfW = oracle.quantize_nvfp4(w, gW)
    d = oracle.nvfp4_gemm(An, sfA, gA, Wn, sfW, gW, bias=b) - oracle.nvfp4_gemm(An, sfA, gA, Wn, sfW, gW)
    np.testing.assert_allclose(d, np.broadcast_to(bf, (T, N)), rtol=0, atol=1e-12)
    At, sAt = oracle.quantize_fp8_tensor(x)
    Bt, sBt = oracle.quantize_fp8_tensor(w)
    d = (oracle.fp8_tensor_gemm("NT", At, sAt, Bt, sBt, T, N, K, bias=b)
         - oracle.fp8_tensor_gemm("NT", At, sAt, Bt, sBt, T, N, K))
    np.testing.assert_allclose(d[0], np.broadcast_to(bf, (T, N)), rtol=0, atol=1e-12)


# ------------------------------------------------------- delayed scaling
def test_delayed_scaling_ring_sequence():
    """Each call uses the scale published by the previous one; the next scale
    is max(history)/448 over the last H amaxes (worked sequence)."""
    ring = oracle.DelayedScaleRing(history=3, initial_scale=1.0)
    mags = [2.0, 8.0, 0.5, 0.25, 0.25]
    xs = [f32_to_bf16_bits(np.array([m, -m / 2, 0.0, m / 4], np.float32)) for m in mags]
    used = []
    for x in xs:
        codes, s = ring.step(x)
        used.append(float(s))
        # codes are exactly E4M3(x / s) with the scale in force
        xf = torch.tensor(bf16_bits_to_f32(x)) / torch.tensor(np.float32(s))
        assert np.array_equal(codes, xf.to(torch.float8_e4m3fn).view(torch.uint8).numpy()) \
            or np.abs(bf16_bits_to_f32(x)).max() / s > 448  # saturated values differ from torch
    f = lambda a: float(np.float32(a) / np.float32(448))
    # window of 3: after 2 -> 2/448; after 8 -> 8/448; after .5 -> 8/448; after .25 -> 8/448
    # (8 still in window), after .25 -> .5/448 (8 left the window)
    assert used == [1.0, f(2), f(8), f(8), f(8)]
    assert float(ring.scale[0]) == f(0.5)
    assert ring.hist.tolist() == [0.25, 0.25, 0.5] and int(ring.idx[0]) == 2


def test_delayed_scaling_saturates_when_amax_grows():
    ring = oracle.DelayedScaleRing(history=2, initial_scale=float(np.float32(1) / np.float32(448)))
    x = f32_to_bf16_bits(np.array([1.0, 2.0, -4.0, 0.5], np.float32))
    codes, s = ring.step(x)
    # the scale in force maps 1.0 to 448: larger magnitudes saturate to +-448
    assert codes.tolist() == [0x7E, 0x7E, 0xFE, 0x76]
    assert float(ring.scale[0]) == float(np.float32(4) / np.float32(448))
