"""Thin Python binding of the scaled-precision GEMM library (``libspg.so``).

Argument marshalling only: every function checks tensor dtypes, shapes and
devices, passes raw device pointers and the current CUDA stream to the C ABI
declared in ``include/spg.h``, and raises :class:`SpgError` on a non-zero
status.  All arithmetic runs in the library's CUDA kernels.  There is no
fallback: if the shared library is missing the import of any entry point
fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "SpgError", "EPILOGUES", "load_library", "library_path",
    "quantize_fp8_rows", "quantize_fp8_tensor", "quantize_fp8_tensor_noalloc",
    "fp8_scale_ring", "quantize_fp8_tensor_delayed",
    "nvfp4_global_scale", "quantize_nvfp4", "quantize_nvfp4_act",
    "nvfp4_sf_bytes", "nvfp4_sf_offset", "fp8_rowscaled_gemm", "nvfp4_gemm", "fp8_tensor_gemm",
    "act_workspace_bytes", "act_workspace", "fp8_rowscaled_linear_bf16", "nvfp4_linear_bf16",
    "select_route", "last_device_error", "set_wait_timeout_ns", "status_string",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libspg.so")
_lock = threading.Lock()
_lib = None

EPILOGUES = {"linear": 0, "add": 1, "linear_add": 1, "swiglu": 2, "linear_swiglu": 2}
KINDS = {"fp8_rowscaled": 0, "nvfp4": 1, "fp8_tensor": 2}
STATUS = {0: "SPG_OK", 1: "SPG_ERR_INVALID_ARG", 2: "SPG_ERR_UNSUPPORTED_SHAPE",
          3: "SPG_ERR_MISALIGNED", 4: "SPG_ERR_CUDA", 5: "SPG_ERR_TIMEOUT"}


class SpgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class Route(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("block_m", ctypes.c_int32),
                ("block_n", ctypes.c_int32), ("block_k", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("acc_buffers", ctypes.c_int32),
                ("group_m", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("tiles", ctypes.c_int64), ("smem_bytes", ctypes.c_int32),
                ("variant", ctypes.c_int32), ("split_n", ctypes.c_int32),
                ("split_k", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64),
                ("swap_ab", ctypes.c_int32), ("reserved", ctypes.c_int32)]


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load ``libspg.so`` (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "scaled_precision_gemm_gb300.build.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64
        st = ctypes.c_int
        sig = {
            "spg_status_string": (ctypes.c_char_p, [i32]),
            "spg_version": (i32, []),
            "spg_set_wait_timeout_ns": (None, [u64]),
            "spg_debug_inject_stall": (None, [i32]),
            "spg_debug_reload_env": (None, []),
            "spg_debug_set_tmap_cache": (None, [i32]),
            "spg_debug_tmap_cache_stats": (None, [ctypes.POINTER(ctypes.c_uint64),
                                                  ctypes.POINTER(ctypes.c_uint64)]),
            "spg_last_device_error": (st, [vp]),
            "spg_last_device_error_code": (st, [vp, ctypes.POINTER(ctypes.c_uint32)]),
            "spg_quantize_fp8_rows": (st, [vp, i64, i64, vp, vp, vp]),
            "spg_quantize_fp8_tensor": (st, [vp, i64, vp, vp, vp, vp]),
            "spg_quantize_fp8_tensor_noalloc": (st, [vp, i64, vp, vp, vp]),
            "spg_nvfp4_global_scale": (st, [vp, i64, vp, vp, vp]),
            "spg_fp8_scale_ring_bytes": (ctypes.c_size_t, [i32]),
            "spg_fp8_scale_ring_init": (st, [vp, i32, ctypes.c_float, vp]),
            "spg_quantize_fp8_tensor_delayed": (st, [vp, i64, vp, vp, vp, i32, vp]),
            "spg_quantize_nvfp4": (st, [vp, i64, i64, vp, vp, vp, vp]),
            "spg_quantize_nvfp4_act": (st, [vp, i64, i64, vp, vp, vp, vp, vp]),
            "spg_nvfp4_sf_bytes": (ctypes.c_size_t, [i64, i64]),
            "spg_nvfp4_sf_offset": (i64, [i64, i64, i64]),
            "fp8_rowscaled_gemm": (st, [vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp]),
            "nvfp4_gemm": (st, [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp]),
            "fp8_tensor_gemm": (st, [ctypes.c_char, ctypes.c_char, i64, vp, i64, vp, vp, i64, vp,
                                     vp, i64, i64, i64, i64, vp]),
            "spg_select_route": (st, [i32, i64, i64, i64, i32, i64, ctypes.POINTER(Route)]),
            "fp8_rowscaled_gemm_bias": (st, [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32,
                                             vp]),
            "nvfp4_gemm_bias": (st, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32,
                                     vp]),
            "fp8_tensor_gemm_bias": (st, [ctypes.c_char, ctypes.c_char, i64, vp, i64, vp, vp, i64,
                                          vp, vp, vp, vp, i64, i64, i64, i64, vp]),
            "spg_select_route_ws": (st, [i32, i64, i64, i64, i32, i64, ctypes.POINTER(Route)]),
            "spg_gemm_workspace_bytes": (i64, [i32, i64, i64, i64, i32, i64]),
            "fp8_rowscaled_gemm_ws": (st, [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32,
                                           vp, i64, vp]),
            "nvfp4_gemm_ws": (st, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32,
                                   vp, i64, vp]),
            "fp8_tensor_gemm_ws": (st, [ctypes.c_char, ctypes.c_char, i64, vp, i64, vp, vp, i64,
                                        vp, vp, vp, vp, i64, i64, i64, i64, vp, i64, vp]),
            "spg_act_workspace_bytes": (i64, [i32, i64, i64, i64, i32]),
            "fp8_rowscaled_linear_bf16": (st, [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32,
                                               vp, i64, vp]),
            "nvfp4_linear_bf16": (st, [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp,
                                       i64, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


_FORCE_VARS = ("SPG_FORCE_VARIANT", "SPG_FORCE_TAIL", "SPG_FORCE_GROUP_M")
_forced_seen = None


def _lib_for_call():
    """The library, after telling it when the route-pinning variables changed
    (it reads them once and caches them; tests pin routes by setting them)."""
    global _forced_seen
    lib = load_library()
    cur = tuple(os.environ.get(v) for v in _FORCE_VARS)
    if cur != _forced_seen:
        lib.spg_debug_reload_env()
        _forced_seen = cur
    return lib


def tmap_cache_stats():
    """(hits, misses) of the library's tensor-map cache."""
    h, m = ctypes.c_uint64(0), ctypes.c_uint64(0)
    load_library().spg_debug_tmap_cache_stats(ctypes.byref(h), ctypes.byref(m))
    return int(h.value), int(m.value)


def status_string(s: int) -> str:
    return load_library().spg_status_string(int(s)).decode()


def _check(status: int, where: str):
    if status != 0:
        raise SpgError(status, where)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, dim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dimensions")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ---------------------------------------------------------------- control
def set_wait_timeout_ns(ns: int):
    load_library().spg_set_wait_timeout_ns(int(ns))


def debug_inject_stall(enable: bool):
    """Test hook: make one-CTA GEMM launches stall on a barrier nothing arrives on."""
    load_library().spg_debug_inject_stall(1 if enable else 0)


def last_device_error(device=None) -> int:
    """Synchronize the current stream and return (and clear) the device error status."""
    s = torch.cuda.current_stream(device)
    return int(load_library().spg_last_device_error(ctypes.c_void_p(s.cuda_stream)))


def last_device_error_code(device=None) -> int:
    """Synchronize, then return (and clear) the raw code of the first in-kernel wait that ran out."""
    s = torch.cuda.current_stream(device)
    code = ctypes.c_uint32(0)
    load_library().spg_last_device_error_code(ctypes.c_void_p(s.cuda_stream), ctypes.byref(code))
    return int(code.value)


def select_route(kind, T, N, K, epilogue="linear", batch=1, workspace=False) -> dict:
    """Route of the plain entry points, or (workspace=True) of the workspace
    entry points given a large enough workspace."""
    r = Route()
    k = KINDS[kind] if isinstance(kind, str) else int(kind)
    e = EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue)
    lib = _lib_for_call()
    fn = lib.spg_select_route_ws if workspace else lib.spg_select_route
    _check(fn(k, T, N, K, e, batch, ctypes.byref(r)), "spg_select_route")
    return {f: getattr(r, f) for f, _ in Route._fields_}


def gemm_workspace_bytes(kind, T, N, K, epilogue="linear", batch=1) -> int:
    """Bytes of workspace that let the workspace entry points split K."""
    k = KINDS[kind] if isinstance(kind, str) else int(kind)
    e = EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue)
    return int(_lib_for_call().spg_gemm_workspace_bytes(k, T, N, K, e, batch))


def gemm_workspace(kind, T, N, K, epilogue="linear", batch=1, device="cuda"):
    """A workspace tensor (uint8) sized for this GEMM, or None when its route
    does not split K."""
    n = gemm_workspace_bytes(kind, T, N, K, epilogue, batch)
    return torch.empty(n, dtype=torch.uint8, device=device) if n > 0 else None


# ------------------------------------------------------------- quantizers
def quantize_fp8_rows(x: torch.Tensor, codes=None, scales=None):
    """bf16 [R, K] -> (E4M3 codes uint8 [R, K], fp32 row scales [R])."""
    _need(x, "x", torch.bfloat16, 2)
    R, K = x.shape
    codes = torch.empty((R, K), dtype=torch.uint8, device=x.device) if codes is None else codes
    scales = torch.empty((R,), dtype=torch.float32, device=x.device) if scales is None else scales
    _need(codes, "codes", torch.uint8)
    _need(scales, "scales", torch.float32)
    _check(load_library().spg_quantize_fp8_rows(_ptr(x), R, K, _ptr(codes), _ptr(scales),
                                                 _stream(x)), "spg_quantize_fp8_rows")
    return codes, scales


def quantize_fp8_tensor(x: torch.Tensor, codes=None, scale=None, amax_scratch=None):
    """bf16 (any shape) -> (E4M3 codes uint8 same shape, fp32 scale [1] on device)."""
    _need(x, "x", torch.bfloat16)
    dev = x.device
    codes = torch.empty(x.shape, dtype=torch.uint8, device=dev) if codes is None else codes
    scale = torch.empty((1,), dtype=torch.float32, device=dev) if scale is None else scale
    scratch = (torch.empty((4,), dtype=torch.float32, device=dev)
               if amax_scratch is None else amax_scratch)
    _check(load_library().spg_quantize_fp8_tensor(_ptr(x), x.numel(), _ptr(codes), _ptr(scale),
                                                   _ptr(scratch), _stream(x)),
           "spg_quantize_fp8_tensor")
    return codes, scale


def quantize_fp8_tensor_noalloc(x: torch.Tensor, codes: torch.Tensor, scale: torch.Tensor):
    """Per-tensor FP8 quantizer whose scratch is the library's static device
    array; the caller passes preallocated codes and scale, nothing is allocated."""
    _need(x, "x", torch.bfloat16)
    _need(codes, "codes", torch.uint8)
    _need(scale, "scale", torch.float32)
    _check(load_library().spg_quantize_fp8_tensor_noalloc(_ptr(x), x.numel(), _ptr(codes),
                                                          _ptr(scale), _stream(x)),
           "spg_quantize_fp8_tensor_noalloc")
    return codes, scale


def fp8_scale_ring(history: int, initial_scale: float = 1.0, device="cuda") -> torch.Tensor:
    """A device amax-history ring for delayed scaling, initialised on `device`."""
    n = int(load_library().spg_fp8_scale_ring_bytes(int(history))) // 4
    ring = torch.empty((max(n, 4) + 3) // 4 * 4, dtype=torch.float32, device=device)
    _check(load_library().spg_fp8_scale_ring_init(_ptr(ring), int(history), float(initial_scale),
                                                  _stream(ring)), "spg_fp8_scale_ring_init")
    return ring


def quantize_fp8_tensor_delayed(x: torch.Tensor, ring: torch.Tensor, history: int, codes=None,
                                scale_used=None):
    """Encode x with the ring's current scale, fold amax(x) into the ring.
    Returns (codes, scale_used)."""
    _need(x, "x", torch.bfloat16)
    _need(ring, "ring", torch.float32)
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device) if codes is None else codes
    scale_used = (torch.empty((4,), dtype=torch.float32, device=x.device)
                  if scale_used is None else scale_used)
    _check(load_library().spg_quantize_fp8_tensor_delayed(_ptr(x), x.numel(), _ptr(codes),
                                                          _ptr(scale_used), _ptr(ring),
                                                          int(history), _stream(x)),
           "spg_quantize_fp8_tensor_delayed")
    return codes, scale_used


def nvfp4_global_scale(x: torch.Tensor, g=None, amax_scratch=None):
    """bf16 tensor -> fp32 [1] device scalar g = amax / 2688."""
    _need(x, "x", torch.bfloat16)
    g = torch.empty((1,), dtype=torch.float32, device=x.device) if g is None else g
    scratch = (torch.empty((4,), dtype=torch.float32, device=x.device)
               if amax_scratch is None else amax_scratch)
    _check(load_library().spg_nvfp4_global_scale(_ptr(x), x.numel(), _ptr(g), _ptr(scratch),
                                                  _stream(x)), "spg_nvfp4_global_scale")
    return g


def nvfp4_sf_bytes(rows: int, K: int) -> int:
    return int(load_library().spg_nvfp4_sf_bytes(rows, K))


def nvfp4_sf_offset(row: int, kb: int, K: int) -> int:
    return int(load_library().spg_nvfp4_sf_offset(row, kb, K))


def quantize_nvfp4(x: torch.Tensor, g: torch.Tensor, codes=None, sf=None):
    """bf16 [R, K] with device scalar g -> (packed E2M1 codes [R, K/2], blocked E4M3 scales)."""
    _need(x, "x", torch.bfloat16, 2)
    _need(g, "g", torch.float32)
    R, K = x.shape
    codes = (torch.empty((R, K // 2), dtype=torch.uint8, device=x.device)
             if codes is None else codes)
    sf = (torch.empty((max(nvfp4_sf_bytes(R, K), 16),), dtype=torch.uint8, device=x.device)
          if sf is None else sf)
    _check(load_library().spg_quantize_nvfp4(_ptr(x), R, K, _ptr(g), _ptr(codes), _ptr(sf),
                                              _stream(x)), "spg_quantize_nvfp4")
    return codes, sf


# ------------------------------------------------------------------ GEMMs
def quantize_nvfp4_act(x: torch.Tensor, g=None, codes=None, sf=None, amax_scratch=None):
    """bf16 [R, K] -> (packed E2M1 codes [R, K/2], blocked E4M3 scales, fp32 [1] g):
    the global scale and the block quantizer in one call (one kernel for small x)."""
    _need(x, "x", torch.bfloat16, 2)
    R, K = x.shape
    g = torch.empty((1,), dtype=torch.float32, device=x.device) if g is None else g
    codes = (torch.empty((R, K // 2), dtype=torch.uint8, device=x.device)
             if codes is None else codes)
    sf = (torch.empty((nvfp4_sf_bytes(R, K),), dtype=torch.uint8, device=x.device)
          if sf is None else sf)
    scratch = (torch.empty((4,), dtype=torch.float32, device=x.device)
               if amax_scratch is None else amax_scratch)
    _need(g, "g", torch.float32)
    _check(load_library().spg_quantize_nvfp4_act(_ptr(x), R, K, _ptr(g), _ptr(scratch),
                                                 _ptr(codes), _ptr(sf), _stream(x)),
           "spg_quantize_nvfp4_act")
    return codes, sf, g


def _epi(epilogue) -> int:
    return EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue)


def _check_bias(bias, bias_scale, N):
    """bias: bf16 [N], or uint8 E4M3 codes [N] with an fp32 [1] bias_scale."""
    if bias is None:
        if bias_scale is not None:
            raise ValueError("bias_scale without bias")
        return
    if bias_scale is None:
        _need(bias, "bias", torch.bfloat16, 1)
    else:
        _need(bias, "bias", torch.uint8, 1)
        _need(bias_scale, "bias_scale", torch.float32)
    if bias.shape[0] != N:
        raise ValueError("bias must have N elements")


def _ws(workspace):
    if workspace is None:
        return None, 0
    _need(workspace, "workspace", torch.uint8, 1)
    return _ptr(workspace), workspace.numel()


def fp8_rowscaled_gemm(A, sa, W, sw, residual=None, epilogue="linear", out=None, bias=None,
                       bias_scale=None, workspace=None):
    """Y = epilogue((A . W^T) * sa[:, None] * sw[None, :] [+ bias]) in bf16.

    workspace (uint8 device tensor, see gemm_workspace) selects the
    workspace entry point, which may split K over the last partial wave."""
    _need(A, "A", torch.uint8, 2)
    _need(W, "W", torch.uint8, 2)
    _need(sa, "sa", torch.float32, 1)
    _need(sw, "sw", torch.float32, 1)
    T, K = A.shape
    N = W.shape[0]
    e = _epi(epilogue)
    if W.shape[1] != K or sa.shape[0] != T or sw.shape[0] != N:
        raise ValueError("shape mismatch")
    if e == 1:
        _need(residual, "residual", torch.bfloat16, 2)
        if tuple(residual.shape) != (T, N):
            raise ValueError("residual must be [T, N]")
    n_out = N // 2 if e == 2 else N
    out = torch.empty((T, n_out), dtype=torch.bfloat16, device=A.device) if out is None else out
    _need(out, "out", torch.bfloat16, 2)
    _check_bias(bias, bias_scale, N)
    lib = _lib_for_call()
    res = _ptr(residual if e == 1 else None)
    if workspace is not None:
        wp, wn = _ws(workspace)
        st = lib.fp8_rowscaled_gemm_ws(_ptr(A), _ptr(sa), _ptr(W), _ptr(sw),
                                                  _ptr(bias), _ptr(bias_scale), res, _ptr(out),
                                                  T, N, K, e, wp, wn, _stream(A))
    elif bias is None:
        st = lib.fp8_rowscaled_gemm(_ptr(A), _ptr(sa), _ptr(W), _ptr(sw), res,
                                               _ptr(out), T, N, K, e, _stream(A))
    else:
        st = lib.fp8_rowscaled_gemm_bias(_ptr(A), _ptr(sa), _ptr(W), _ptr(sw),
                                                    _ptr(bias), _ptr(bias_scale), res, _ptr(out),
                                                    T, N, K, e, _stream(A))
    _check(st, "fp8_rowscaled_gemm")
    return out


def nvfp4_gemm(A, sfA, gA, W, sfW, gW, residual=None, epilogue="linear", out=None, bias=None,
               bias_scale=None, workspace=None):
    """Y = epilogue(block-scaled NVFP4 product * gA * gW [+ bias]) in bf16; A/W packed [rows, K/2]."""
    for t, n, d in ((A, "A", torch.uint8), (W, "W", torch.uint8), (sfA, "sfA", torch.uint8),
                    (sfW, "sfW", torch.uint8), (gA, "gA", torch.float32),
                    (gW, "gW", torch.float32)):
        _need(t, n, d)
    T, Kh = A.shape
    N = W.shape[0]
    K = 2 * Kh
    e = _epi(epilogue)
    if W.shape[1] != Kh:
        raise ValueError("shape mismatch")
    if sfA.numel() < nvfp4_sf_bytes(T, K) or sfW.numel() < nvfp4_sf_bytes(N, K):
        raise ValueError("scale buffers smaller than the blocked layout")
    if e == 1:
        _need(residual, "residual", torch.bfloat16, 2)
        if tuple(residual.shape) != (T, N):
            raise ValueError("residual must be [T, N]")
    n_out = N // 2 if e == 2 else N
    out = torch.empty((T, n_out), dtype=torch.bfloat16, device=A.device) if out is None else out
    _need(out, "out", torch.bfloat16, 2)
    _check_bias(bias, bias_scale, N)
    lib = _lib_for_call()
    res = _ptr(residual if e == 1 else None)
    if workspace is not None:
        wp, wn = _ws(workspace)
        st = lib.nvfp4_gemm_ws(_ptr(A), _ptr(sfA), _ptr(gA), _ptr(W), _ptr(sfW),
                                          _ptr(gW), _ptr(bias), _ptr(bias_scale), res, _ptr(out),
                                          T, N, K, e, wp, wn, _stream(A))
    elif bias is None:
        st = lib.nvfp4_gemm(_ptr(A), _ptr(sfA), _ptr(gA), _ptr(W), _ptr(sfW), _ptr(gW),
                                       res, _ptr(out), T, N, K, e, _stream(A))
    else:
        st = lib.nvfp4_gemm_bias(_ptr(A), _ptr(sfA), _ptr(gA), _ptr(W), _ptr(sfW),
                                            _ptr(gW), _ptr(bias), _ptr(bias_scale), res,
                                            _ptr(out), T, N, K, e, _stream(A))
    _check(st, "nvfp4_gemm")
    return out


_ACT_KINDS = {"fp8_rowscaled": 0, "nvfp4": 1}


def act_workspace_bytes(kind, T, N, K, epilogue="linear") -> int:
    """Bytes of workspace the activation operators take (0: none needed)."""
    return int(_lib_for_call().spg_act_workspace_bytes(_ACT_KINDS[kind], T, N, K,
                                                       _epi(epilogue)))


def act_workspace(kind, T, N, K, epilogue="linear", device="cuda"):
    """A workspace tensor (uint8) for the activation operators, or None when
    the call needs none."""
    n = act_workspace_bytes(kind, T, N, K, epilogue)
    return torch.empty((n,), dtype=torch.uint8, device=device) if n > 0 else None


def _act_common(X, N, epilogue, residual, out, bias, bias_scale):
    _need(X, "X", torch.bfloat16, 2)
    T, K = X.shape
    e = _epi(epilogue)
    if e == 1:
        _need(residual, "residual", torch.bfloat16, 2)
        if tuple(residual.shape) != (T, N):
            raise ValueError("residual must be [T, N]")
    n_out = N // 2 if e == 2 else N
    out = torch.empty((T, n_out), dtype=torch.bfloat16, device=X.device) if out is None else out
    _need(out, "out", torch.bfloat16, 2)
    _check_bias(bias, bias_scale, N)
    return T, K, e, out


def fp8_rowscaled_linear_bf16(X, W, sw, residual=None, epilogue="linear", out=None, bias=None,
                              bias_scale=None, workspace=None):
    """The FP8 row-scaled operator on bf16 activations X [T, K]: per-row
    quantization of X, then the GEMM (workspace: act_workspace(...), made
    here when not given)."""
    _need(W, "W", torch.uint8, 2)
    _need(sw, "sw", torch.float32)
    N = W.shape[0]
    T, K, e, out = _act_common(X, N, epilogue, residual, out, bias, bias_scale)
    if W.shape[1] != K:
        raise ValueError("shape mismatch")
    if workspace is None:
        workspace = act_workspace("fp8_rowscaled", T, N, K, epilogue, device=X.device)
    wp, wn = _ws(workspace)
    st = _lib_for_call().fp8_rowscaled_linear_bf16(
        _ptr(X), _ptr(W), _ptr(sw), _ptr(bias), _ptr(bias_scale),
        _ptr(residual if e == 1 else None), _ptr(out), T, N, K, e, wp, wn, _stream(X))
    _check(st, "fp8_rowscaled_linear_bf16")
    return out


def nvfp4_linear_bf16(X, W, sfW, gW, residual=None, epilogue="linear", out=None, bias=None,
                      bias_scale=None, workspace=None):
    """The NVFP4 operator on bf16 activations X [T, K]: global scale, block
    quantization of X, then the block-scaled GEMM -- one kernel at T <= 4
    (workspace: act_workspace(...), made here when not given)."""
    for t, n, d in ((W, "W", torch.uint8), (sfW, "sfW", torch.uint8), (gW, "gW", torch.float32)):
        _need(t, n, d)
    N = W.shape[0]
    T, K, e, out = _act_common(X, N, epilogue, residual, out, bias, bias_scale)
    if 2 * W.shape[1] != K:
        raise ValueError("shape mismatch")
    if sfW.numel() < nvfp4_sf_bytes(N, K):
        raise ValueError("weight scale buffer smaller than the blocked layout")
    if workspace is None:
        workspace = act_workspace("nvfp4", T, N, K, epilogue, device=X.device)
    wp, wn = _ws(workspace)
    st = _lib_for_call().nvfp4_linear_bf16(
        _ptr(X), _ptr(W), _ptr(sfW), _ptr(gW), _ptr(bias), _ptr(bias_scale),
        _ptr(residual if e == 1 else None), _ptr(out), T, N, K, e, wp, wn, _stream(X))
    _check(st, "nvfp4_linear_bf16")
    return out


def fp8_tensor_gemm(layout: str, A, sA, B, sB, M, N, K, batch=1, strideA=None, strideB=None,
                    out=None, strideC=None, bias=None, bias_scale=None, workspace=None):
    """C[b] = bf16(sA*sB*opA(A[b]) opB(B[b])), layout in {'NT','NN','TN','TT'}.

    A / B are flat (or any contiguous) uint8 buffers; matrix b starts at
    b*strideA / b*strideB elements (default: dense; 0 broadcasts)."""
    if len(layout) != 2 or layout[0] not in "NT" or layout[1] not in "NT":
        raise ValueError("layout must be two letters from N/T")
    _need(A, "A", torch.uint8)
    _need(B, "B", torch.uint8)
    _need(sA, "sA", torch.float32)
    _need(sB, "sB", torch.float32)
    strideA = M * K if strideA is None else strideA
    strideB = N * K if strideB is None else strideB
    strideC = M * N if strideC is None else strideC
    if A.numel() < (batch - 1) * strideA + M * K or B.numel() < (batch - 1) * strideB + N * K:
        raise ValueError("operand buffers too small for the batch strides")
    out = (torch.empty((batch, M, N), dtype=torch.bfloat16, device=A.device)
           if out is None else out)
    _need(out, "out", torch.bfloat16)
    if out.numel() < (batch - 1) * strideC + M * N:
        raise ValueError("output buffer too small")
    _check_bias(bias, bias_scale, N)
    lib = _lib_for_call()
    if workspace is not None:
        wp, wn = _ws(workspace)
        st = lib.fp8_tensor_gemm_ws(layout[0].encode(), layout[1].encode(), batch, _ptr(A),
                                    strideA, _ptr(sA), _ptr(B), strideB, _ptr(sB), _ptr(bias),
                                    _ptr(bias_scale), _ptr(out), strideC, M, N, K, wp, wn,
                                    _stream(A))
    elif bias is None:
        st = lib.fp8_tensor_gemm(layout[0].encode(), layout[1].encode(), batch, _ptr(A), strideA,
                                 _ptr(sA), _ptr(B), strideB, _ptr(sB), _ptr(out), strideC, M, N,
                                 K, _stream(A))
    else:
        st = lib.fp8_tensor_gemm_bias(layout[0].encode(), layout[1].encode(), batch, _ptr(A),
                                      strideA, _ptr(sA), _ptr(B), strideB, _ptr(sB), _ptr(bias),
                                      _ptr(bias_scale), _ptr(out), strideC, M, N, K, _stream(A))
    _check(st, "fp8_tensor_gemm")
    return out
