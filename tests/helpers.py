"""Shared helpers of the test suite (host-side marshalling and the tolerance)."""
import numpy as np

from synthetic_inputs import bf16_bits_to_f32


def tol_violations(y, ref):
    """Elements breaking |y - ref| <= 8e-3 |ref| + 1e-3 rms(ref) (the GEMM parity bound)."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    bound = 8e-3 * np.abs(ref) + 1e-3 * rms
    bad = ~(np.abs(y - ref) <= bound)
    return int(bad.sum()), float(np.max(np.abs(y - ref) / np.maximum(bound, 1e-300))) if ref.size else 0.0


def assert_within_tol(y, ref, what=""):
    n, worst = tol_violations(y, ref)
    assert n == 0, f"{what}: {n} elements outside tolerance (worst ratio {worst:.3g})"


def sf_rowmajor_to_blocked(sf_rm: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Place a row-major [rows, K/16] scale matrix into the blocked layout.

    Written from the layout definition: tiles of 128 rows x 4 scales (512
    bytes), tile rows outermost, K-tiles innermost; inside a tile (r, c) is at
    byte (r % 32) * 16 + (r // 32) * 4 + c.  Padding is zero."""
    rows_pad = (rows + 127) // 128 * 128
    kt = (K + 63) // 64
    out = np.zeros(rows_pad * kt * 4, np.uint8)
    r = np.arange(rows)[:, None]
    c = np.arange(K // 16)[None, :]
    off = ((r // 128) * kt + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)
    out[off] = sf_rm
    return out


def sf_blocked_to_rowmajor(blocked: np.ndarray, rows: int, K: int) -> np.ndarray:
    kt = (K + 63) // 64
    r = np.arange(rows)[:, None]
    c = np.arange(K // 16)[None, :]
    off = ((r // 128) * kt + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)
    return np.asarray(blocked)[off]


def bf16_to_f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)
