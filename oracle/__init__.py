"""CPU oracle for the scaled low-precision linear-layer GEMM (test infrastructure).

This package is TEST INFRASTRUCTURE.  Only the tests, the smoke check and the
CPU-baseline leg of the bench may import it.  The library product never calls
it, and it shares no code with the CUDA path: the arithmetic lives in
``spg_oracle.c`` (plain C, fp32 steps as single IEEE operations, exact 64-bit
integer dot products), and this module only marshals numpy arrays.

Functions and the passages they follow:

* ``e4m3_value`` / ``e2m1_value`` / ``e4m3_encode`` / ``e2m1_encode`` -- code
  decode from the format definitions and round-to-nearest-even saturating
  encode (ninfer PR #167 opening paragraph names FP8 E4M3; ninfer PR #160 body
  names E2M1 codes with an E4M3 scale per 16 elements).
* ``quantize_fp8_rows`` -- one fp32 scale per row, s = amax/448 (ninfer PR #167,
  "What actually changes": row-scaled A8 activations and row-scaled weights).
* ``quantize_fp8_tensor`` -- one scale per tensor (AstrAI fp8 gemm.cuh commit
  log, the quantize bullets).
* ``DelayedScaleRing`` -- delayed scaling from an amax history ring (AstrAI fp8
  gemm.cuh commit log, scale-ring bullets).
* ``nvfp4_global_scale`` / ``quantize_nvfp4`` -- two-level NVFP4 scaling (ninfer
  PR #160 body).
* ``fp8_rowscaled_gemm`` / ``nvfp4_gemm`` -- Y = dequant(A) dequant(W)^T with the
  epilogues linear / linear_add / linear_swiglu (ninfer PR #167 opening
  paragraph; the SwiGLU pairing reading: W rows 2j = gate_j, 2j+1 = up_j).
* ``fp8_tensor_gemm`` -- per-tensor FP8 GEMM, layouts NT / NN / TN, batch
  strides with stride 0 broadcasting (AstrAI fp8 gemm.cuh commit log, first
  bullet).
* ``bias=`` / ``bias_scale=`` on the three GEMMs -- fused bias per output column
  after the scales, bf16 or E4M3 x bias_scale (AstrAI fp8 gemm.cuh commit log,
  bias bullets).

Every pin of these functions is in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spg_oracle.c")
_LIB = os.path.join(_HERE, "libspg_oracle.so")
_lock = threading.Lock()
_lib = None

EPI = {"linear": 0, "add": 1, "linear_add": 1, "swiglu": 2, "linear_swiglu": 2}


def build(force: bool = False) -> str:
    """Compile the oracle's C source into ``libspg_oracle.so`` beside it."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            c = ctypes
            i64, f32, u32 = c.c_int64, c.c_float, c.c_uint32
            vp = c.c_void_p
            lib.spg_oracle_e4m3_value.restype = c.c_double
            lib.spg_oracle_e4m3_value.argtypes = [u32]
            lib.spg_oracle_e2m1_value.restype = c.c_double
            lib.spg_oracle_e2m1_value.argtypes = [u32]
            lib.spg_oracle_e4m3_encode.restype = u32
            lib.spg_oracle_e4m3_encode.argtypes = [c.c_double]
            lib.spg_oracle_e2m1_encode.restype = u32
            lib.spg_oracle_e2m1_encode.argtypes = [c.c_double]
            lib.spg_oracle_quantize_fp8_rows.argtypes = [vp, i64, i64, vp, vp]
            lib.spg_oracle_quantize_fp8_tensor.argtypes = [vp, i64, vp, vp]
            lib.spg_oracle_fp8_delayed_step.argtypes = [vp, i64, vp, vp, c.c_int, vp, vp, vp]
            lib.spg_oracle_nvfp4_global_scale.restype = f32
            lib.spg_oracle_nvfp4_global_scale.argtypes = [vp, i64]
            lib.spg_oracle_quantize_nvfp4.argtypes = [vp, i64, i64, f32, vp, vp]
            lib.spg_oracle_fp8_rowscaled_gemm.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64,
                                                          c.c_int, vp, i64, vp, vp]
            lib.spg_oracle_nvfp4_gemm.argtypes = [vp, vp, f32, vp, vp, f32, vp, i64, i64, i64,
                                                  c.c_int, vp, i64, vp, vp]
            lib.spg_oracle_fp8_tensor_gemm.argtypes = [c.c_char, c.c_char, i64, vp, i64, f32, vp,
                                                       i64, f32, i64, i64, i64, vp, i64, vp]
            lib.spg_oracle_fp8_rowscaled_gemm_bias.argtypes = [vp, vp, vp, vp, vp, c.c_int, f32, vp,
                                                               i64, i64, i64, c.c_int, vp, i64, vp,
                                                               vp]
            lib.spg_oracle_nvfp4_gemm_bias.argtypes = [vp, vp, f32, vp, vp, f32, vp, c.c_int, f32,
                                                       vp, i64, i64, i64, c.c_int, vp, i64, vp, vp]
            lib.spg_oracle_fp8_tensor_gemm_bias.argtypes = [c.c_char, c.c_char, i64, vp, i64, f32,
                                                            vp, i64, f32, vp, c.c_int, f32, i64,
                                                            i64, i64, vp, i64, vp]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _bf16_bits(x) -> np.ndarray:
    """Accept bf16 bit patterns as uint16 (numpy has no bfloat16 dtype)."""
    x = np.asarray(x)
    if x.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as their uint16 bit patterns")
    return np.ascontiguousarray(x)


# ----------------------------------------------------------------- codes
def e4m3_value(code: int) -> float:
    return _load().spg_oracle_e4m3_value(int(code))


def e2m1_value(code: int) -> float:
    return _load().spg_oracle_e2m1_value(int(code))


def e4m3_encode(x: float) -> int:
    return int(_load().spg_oracle_e4m3_encode(float(x)))


def e2m1_encode(x: float) -> int:
    return int(_load().spg_oracle_e2m1_encode(float(x)))


def e4m3_table() -> np.ndarray:
    """fp64 value of every E4M3FN code 0..255 (NaN at 0x7F and 0xFF)."""
    return np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e2m1_table() -> np.ndarray:
    """fp64 value of every E2M1 code 0..15."""
    return np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


# ------------------------------------------------------------ quantizers
def quantize_fp8_rows(x_bf16: np.ndarray):
    """bf16 bits [R, K] -> (codes u8 [R, K], scales f32 [R])."""
    x = _bf16_bits(x_bf16)
    R, K = x.shape
    codes = np.empty((R, K), np.uint8)
    scales = np.empty((R,), np.float32)
    _load().spg_oracle_quantize_fp8_rows(_ptr(x), R, K, _ptr(codes), _ptr(scales))
    return codes, scales


def quantize_fp8_tensor(x_bf16: np.ndarray):
    """bf16 bits (any shape) -> (codes u8 same shape, scale f32 scalar)."""
    x = _bf16_bits(x_bf16)
    codes = np.empty(x.shape, np.uint8)
    scale = np.empty((1,), np.float32)
    _load().spg_oracle_quantize_fp8_tensor(_ptr(x), x.size, _ptr(codes), _ptr(scale))
    return codes, np.float32(scale[0])


class DelayedScaleRing:
    """Amax-history ring for delayed per-tensor scaling (state kept on the host)."""

    def __init__(self, history: int, initial_scale: float = 1.0):
        self.hist = np.zeros(history, np.float32)
        self.idx = np.zeros(1, np.int32)
        self.scale = np.array([initial_scale], np.float32)

    def step(self, x_bf16):
        """Quantize x with the current scale, then fold amax(x) into the ring.
        Returns (codes, scale_used)."""
        x = _bf16_bits(x_bf16)
        codes = np.empty(x.shape, np.uint8)
        used = np.empty(1, np.float32)
        _load().spg_oracle_fp8_delayed_step(_ptr(x), x.size, _ptr(codes), _ptr(self.hist),
                                            self.hist.size, _ptr(self.idx), _ptr(self.scale),
                                            _ptr(used))
        return codes, np.float32(used[0])


def nvfp4_global_scale(x_bf16: np.ndarray) -> np.float32:
    x = _bf16_bits(x_bf16)
    return np.float32(_load().spg_oracle_nvfp4_global_scale(_ptr(x), x.size))


def quantize_nvfp4(x_bf16: np.ndarray, g: float):
    """bf16 bits [R, K] with global scale g -> (codes u8 [R, K/2], sf u8 [R, K/16] row-major)."""
    x = _bf16_bits(x_bf16)
    R, K = x.shape
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    codes = np.empty((R, K // 2), np.uint8)
    sf = np.empty((R, K // 16), np.uint8)
    _load().spg_oracle_quantize_nvfp4(_ptr(x), R, K, float(np.float32(g)), _ptr(codes), _ptr(sf))
    return codes, sf


# ----------------------------------------------------------------- GEMMs
def _rows_arg(rows, T):
    if rows is None:
        return None, T
    r = _c(rows, np.int64)
    if r.size and (r.min() < 0 or r.max() >= T):
        raise IndexError("row index out of range")
    return r, r.size


def _bias_args(bias, bias_scale, N):
    """(pointer array, kind, scale): bias bf16 bits uint16 [N] (kind 1), or
    E4M3 codes uint8 [N] with an fp32 bias_scale (kind 2)."""
    if bias is None:
        return None, 0, 0.0
    b = np.ascontiguousarray(bias)
    assert b.shape == (N,)
    if bias_scale is None:
        if b.dtype != np.uint16:
            raise TypeError("a bf16 bias is passed as uint16 bit patterns")
        return b, 1, 0.0
    if b.dtype != np.uint8:
        raise TypeError("an fp8 bias is passed as uint8 E4M3 codes")
    return b, 2, float(np.float32(bias_scale))


def fp8_rowscaled_gemm(A, sa, W, sw, residual=None, epilogue="linear", rows=None,
                       return_acc=False, bias=None, bias_scale=None):
    """Y [len(rows) or T, N_out] fp64 = epilogue(dequant(A) dequant(W)^T [+ bias])."""
    A = _c(A, np.uint8); W = _c(W, np.uint8)
    sa = _c(sa, np.float32); sw = _c(sw, np.float32)
    T, K = A.shape
    N, K2 = W.shape
    assert K == K2 and sa.shape == (T,) and sw.shape == (N,)
    epi = EPI[epilogue]
    res = None
    if epi == 1:
        res = _bf16_bits(residual).reshape(T, N)
    r, nr = _rows_arg(rows, T)
    n_out = N // 2 if epi == 2 else N
    out = np.empty((nr, n_out), np.float64)
    acc = np.empty((nr, N), np.float64) if return_acc else None
    bb, bk, bs = _bias_args(bias, bias_scale, N)
    _load().spg_oracle_fp8_rowscaled_gemm_bias(_ptr(A), _ptr(sa), _ptr(W), _ptr(sw), _ptr(bb), bk, bs,
                                               _ptr(res), T, N, K, epi, _ptr(r), nr, _ptr(out),
                                               _ptr(acc))
    return (out, acc) if return_acc else out


def nvfp4_gemm(A, sfA, gA, W, sfW, gW, residual=None, epilogue="linear", rows=None,
               return_acc=False, bias=None, bias_scale=None):
    """A codes [T, K/2], sfA row-major [T, K/16]; same for W [N, ...]."""
    A = _c(A, np.uint8); W = _c(W, np.uint8)
    sfA = _c(sfA, np.uint8); sfW = _c(sfW, np.uint8)
    T, Kh = A.shape
    N, Kh2 = W.shape
    K = 2 * Kh
    assert Kh == Kh2 and sfA.shape == (T, K // 16) and sfW.shape == (N, K // 16)
    epi = EPI[epilogue]
    res = None
    if epi == 1:
        res = _bf16_bits(residual).reshape(T, N)
    r, nr = _rows_arg(rows, T)
    n_out = N // 2 if epi == 2 else N
    out = np.empty((nr, n_out), np.float64)
    acc = np.empty((nr, N), np.float64) if return_acc else None
    bb, bk, bs = _bias_args(bias, bias_scale, N)
    _load().spg_oracle_nvfp4_gemm_bias(_ptr(A), _ptr(sfA), float(np.float32(gA)), _ptr(W),
                                       _ptr(sfW), float(np.float32(gW)), _ptr(bb), bk, bs,
                                       _ptr(res), T, N, K, epi, _ptr(r), nr, _ptr(out), _ptr(acc))
    return (out, acc) if return_acc else out


def fp8_tensor_gemm(layout: str, A, sA, B, sB, M, N, K, batch=1, strideA=None, strideB=None,
                    rows=None, bias=None, bias_scale=None):
    """C [batch, M (or len(rows)), N] fp64 for layout 'NT', 'NN' or 'TN'.

    A / B are flat u8 buffers; matrix b starts at b*strideA / b*strideB
    elements (defaults: dense packing; 0 broadcasts)."""
    if layout not in ("NT", "NN", "TN"):
        raise ValueError("layout must be NT, NN or TN")
    A = _c(A, np.uint8).reshape(-1); B = _c(B, np.uint8).reshape(-1)
    strideA = M * K if strideA is None else strideA
    strideB = N * K if strideB is None else strideB
    assert A.size >= (batch - 1) * strideA + M * K and B.size >= (batch - 1) * strideB + N * K
    r, nr = _rows_arg(rows, M)
    out = np.empty((batch, nr, N), np.float64)
    bb, bk, bs = _bias_args(bias, bias_scale, N)
    _load().spg_oracle_fp8_tensor_gemm_bias(layout[0].encode(), layout[1].encode(), batch,
                                            _ptr(A), strideA, float(np.float32(sA)), _ptr(B),
                                            strideB, float(np.float32(sB)), _ptr(bb), bk, bs, M, N,
                                            K, _ptr(r), nr, _ptr(out))
    return out

