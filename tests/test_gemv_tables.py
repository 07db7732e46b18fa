"""The NVFP4 GEMV's decode tables, read from its source and checked against
the E2M1 definition (OCP MX formats: sign, 2 exponent bits with bias 1, one
mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6).  The kernel turns four
codes into four int8 holding twice their values with three byte permutes;
emulating those permutes here on every 4-code group checks the constants
and the selector arithmetic without a GPU."""
import os
import re

import pytest

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "scaled_precision_gemm_gb300", "csrc", "gemv_nvfp4.cuh")


def e2m1_value(code):
    s = -1.0 if code & 8 else 1.0
    e, m = (code >> 1) & 3, code & 1
    return s * (m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2))


def byte_perm(x, y, sel):
    """CUDA __byte_perm with selectors below 8: byte i of the result is byte
    (nibble i of sel) of the 8-byte value y:x."""
    b = [(x >> (8 * i)) & 0xFF for i in range(4)] + [(y >> (8 * i)) & 0xFF for i in range(4)]
    return sum(b[(sel >> (4 * i)) & 7] << (8 * i) for i in range(4))


def kernel_decoder():
    src = open(SRC).read()
    body = src[src.index("e2m1x4_to_s8x2(uint32_t codes16)"):]
    body = body[:body.index("}")]
    pos = re.search(r"pos = __byte_perm\((0x[0-9A-Fa-f]+)u, (0x[0-9A-Fa-f]+)u, mag\)", body)
    neg = re.search(r"neg = __byte_perm\((0x[0-9A-Fa-f]+)u, (0x[0-9A-Fa-f]+)u, mag\)", body)
    sel = re.search(r"__byte_perm\(pos, neg, (0x[0-9A-Fa-f]+)u \| \(\(codes16 >> 1\) & "
                    r"(0x[0-9A-Fa-f]+)u\)\)", body)
    assert pos and neg and sel, "decode tables not found in the kernel source"
    p0, p1 = int(pos.group(1), 16), int(pos.group(2), 16)
    n0, n1 = int(neg.group(1), 16), int(neg.group(2), 16)
    base, smask = int(sel.group(1), 16), int(sel.group(2), 16)

    def decode(codes16):
        mag = codes16 & 0x7777
        return byte_perm(byte_perm(p0, p1, mag), byte_perm(n0, n1, mag),
                         base | ((codes16 >> 1) & smask))
    return decode


def s8(word, i):
    v = (word >> (8 * i)) & 0xFF
    return v - 256 if v & 0x80 else v


def test_every_code_decodes_to_twice_its_value():
    decode = kernel_decoder()
    for code in range(16):
        for lane in range(4):  # the code in each of the four nibbles
            word = decode(code << (4 * lane))
            assert s8(word, lane) == 2 * e2m1_value(code), (code, lane)


@pytest.mark.parametrize("seed", range(4))
def test_mixed_groups_decode_elementwise(seed):
    import random
    rnd = random.Random(seed)
    decode = kernel_decoder()
    for _ in range(2000):
        codes = [rnd.randrange(16) for _ in range(4)]
        word = decode(sum(c << (4 * i) for i, c in enumerate(codes)))
        assert [s8(word, i) for i in range(4)] == [2 * e2m1_value(c) for c in codes]


def test_block_products_fit_int32_exactly():
    # |2a|, |2w| <= 12, 16 products per block: |sum| <= 2304 < 2^24 (exact in
    # fp32 after the int -> float conversion)
    assert 16 * 12 * 12 < 2 ** 24
