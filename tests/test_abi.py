"""The C-ABI library loads, exports every declared symbol, and its host-only
logic (status strings, scale-layout arithmetic, route selector, argument
validation that returns before any launch) behaves as the header states.
No kernel is launched here."""
import ctypes
import os
import re

import numpy as np
import pytest

import scaled_precision_gemm_gb300 as spg
from tests.helpers import sf_blocked_to_rowmajor, sf_rowmajor_to_blocked

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from scaled_precision_gemm_gb300 import build
    build.build()
    return spg.load_library()


def declared_symbols():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"^SPG_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, re.M)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert spg.status_string(0) == "SPG_OK"
    assert spg.status_string(5) == "SPG_ERR_TIMEOUT"
    assert spg.status_string(99) == "SPG_ERR_UNKNOWN"
    assert lib.spg_version() >= 200  # spg_route with swap_ab
    assert ctypes.sizeof(spg.Route) == 72  # the C struct's size (static_assert in host.cu)


@pytest.mark.parametrize("rows,K", [(1, 64), (128, 256), (129, 17408), (300, 5120), (64, 320)])
def test_sf_layout_matches_definition(lib, rows, K):
    assert spg.nvfp4_sf_bytes(rows, K) == ((rows + 127) // 128 * 128) * ((K + 63) // 64 * 4)
    rng = np.random.default_rng(rows + K)
    sf = rng.integers(0, 0x7F, size=(rows, K // 16), dtype=np.uint8)
    blocked = sf_rowmajor_to_blocked(sf, rows, K)
    assert blocked.size == spg.nvfp4_sf_bytes(rows, K)
    for r in {0, rows - 1, rows // 2, min(rows - 1, 37)}:
        for kb in {0, K // 16 - 1, (K // 16) // 2}:
            assert blocked[spg.nvfp4_sf_offset(r, kb, K)] == sf[r, kb]
    assert np.array_equal(sf_blocked_to_rowmajor(blocked, rows, K), sf)
    # every (row, kb) maps to a distinct byte
    offs = {spg.nvfp4_sf_offset(r, kb, K) for r in range(min(rows, 130)) for kb in range(K // 16)}
    assert len(offs) == min(rows, 130) * (K // 16)
    assert spg.nvfp4_sf_offset(-1, 0, K) == -1 and spg.nvfp4_sf_offset(0, K // 16, K) == -1


def test_route_selector(lib):
    r = spg.select_route("fp8_rowscaled", 4096, 5120, 17408, "add")
    assert r["block_m"] in (128, 256) and r["block_n"] in (128, 256)
    assert r["tiles"] == (4096 // r["block_m"]) * (5120 // r["block_n"])
    per_unit = 2 if r["block_m"] == 256 else 1          # two-SM tiles run on CTA pairs
    assert r["grid"] % per_unit == 0 and 1 <= r["grid"] // per_unit <= r["tiles"]
    assert r["grid"] <= 152
    assert r["smem_bytes"] <= 232448
    small = spg.select_route("fp8_rowscaled", 64, 128, 256, "linear")
    # one tile; a lone two-SM tile is split along N over up to 4 CTA pairs
    assert small["tiles"] == 1 and small["grid"] in (1, 2, 4, 8)
    nv = spg.select_route("nvfp4", 4096, 5120, 17408, "add")
    assert (nv["block_m"], nv["block_n"]) == (256, 256) and nv["tiles"] == 320
    assert nv["grid"] == 152 and nv["acc_buffers"] == 1
    # narrow T: the one-CTA 128x128 tile spreads the weight stream wider
    nv = spg.select_route("nvfp4", 256, 5120, 17408, "add")
    assert (nv["block_m"], nv["block_n"], nv["tiles"], nv["grid"]) == (128, 128, 80, 80)
    b = spg.select_route("fp8_tensor", 512, 512, 512, "linear", batch=64)
    assert b["tiles"] % 64 == 0
    with pytest.raises(spg.SpgError):
        spg.select_route(7, 1, 1, 1)


def test_route_selector_forced_variants(lib, monkeypatch):
    for v, (bm, bn) in {"2sm": (256, 256), "2sm192": (256, 192), "2sm160": (256, 160),
                        "2sm128": (256, 128), "1sm256": (128, 256), "1sm128": (128, 128)}.items():
        monkeypatch.setenv("SPG_FORCE_VARIANT", v)
        r = spg.select_route("fp8_rowscaled", 1000, 5120, 6144, "linear")
        assert (r["block_m"], r["block_n"]) == (bm, bn)
    monkeypatch.delenv("SPG_FORCE_VARIANT")
    # large square problems take the two-SM pair tile; one tiny tile takes one CTA
    assert spg.select_route("fp8_tensor", 8192, 8192, 8192)["block_m"] == 256
    assert spg.select_route("fp8_rowscaled", 64, 128, 256)["tiles"] == 1
    # T=1024 x N=5120: a pair tile narrower than 256 fills the 76 pairs better
    # than the 80 tiles of the 256-wide one (one full wave + 4 tiles)
    r = spg.select_route("fp8_rowscaled", 1024, 5120, 17408, "add")
    assert r["block_m"] == 256 and r["grid"] == 152
    assert r["tiles"] == 4 * ((5120 + r["block_n"] - 1) // r["block_n"])


def test_route_selector_gemv(lib, monkeypatch):
    """NVFP4 at T <= 4 takes the CUDA-core GEMV (variant 4: two weight rows
    per warp, four warps per CTA, no workspace) for N up to 16384 and T = 1
    or K <= 8192; a forced tile variant, wider N or T > 4 does not."""
    monkeypatch.delenv("SPG_FORCE_TAIL", raising=False)
    monkeypatch.delenv("SPG_FORCE_VARIANT", raising=False)
    for T, K in [(1, 17408), (1, 6144), (2, 6144), (3, 6144), (4, 6144)]:
        for epi in ("linear", "add", "swiglu"):
            r = spg.select_route("nvfp4", T, 5120, K, epi, workspace=True)
            assert r["variant"] == 4 and r["block_n"] == 2 and r["grid"] == 640
            assert r["split_k"] == 1 and r["workspace_bytes"] == 0
            assert r["smem_bytes"] == T * (K // 32) * 34  # decoded activations
    assert spg.gemm_workspace_bytes("nvfp4", 1, 5120, 17408, "add") == 0
    for T in (2, 3, 4):
        assert spg.select_route("nvfp4", T, 5120, 17408, "add")["variant"] == 7
    assert spg.select_route("nvfp4", 2, 16384, 17408, "add")["variant"] != 4
    assert spg.select_route("nvfp4", 1, 34816, 5120, "swiglu")["variant"] != 4
    assert spg.select_route("fp8_rowscaled", 1, 5120, 17408, "add")["variant"] != 4
    monkeypatch.setenv("SPG_FORCE_VARIANT", "2sm_st")
    assert spg.select_route("nvfp4", 1, 5120, 17408, "add")["variant"] == 3
    monkeypatch.setenv("SPG_FORCE_VARIANT", "gemv")
    assert spg.select_route("nvfp4", 4, 5120, 17408, "add")["variant"] == 4
    assert spg.select_route("nvfp4", 1, 34816, 5120, "swiglu")["variant"] == 4
    # the decoded activations must fit the CTA's shared memory
    assert spg.select_route("nvfp4", 4, 256, 48128, "add")["variant"] == 4
    assert spg.select_route("nvfp4", 4, 256, 48384, "add")["variant"] != 4
    assert spg.select_route("nvfp4", 5, 5120, 17408, "add")["variant"] != 4


def test_act_workspace_sizes(lib, monkeypatch):
    """The activation operators' workspace: none for the fused NVFP4 decode
    kernel; otherwise the activation codes and scales (256-byte aligned
    pieces) followed by the GEMM's own K-split workspace."""
    for v in ("SPG_FORCE_VARIANT", "SPG_FORCE_TAIL", "SPG_FORCE_GROUP_M"):
        monkeypatch.delenv(v, raising=False)
    up = lambda v: (v + 255) // 256 * 256
    # the fused decode kernel only where pinned (T <= 4, its shared memory)
    monkeypatch.setenv("SPG_FORCE_VARIANT", "gemv_fused")
    for T in (1, 2, 3, 4):
        assert spg.act_workspace_bytes("nvfp4", T, 34816, 5120, "swiglu") == 0
    assert spg.act_workspace_bytes("nvfp4", 5, 5120, 6144, "add") > 0
    monkeypatch.delenv("SPG_FORCE_VARIANT")
    for T, N, K, epi in [(1, 5120, 17408, "add"), (2, 5120, 6144, "add"), (1, 5120, 6144, "add"),
                         (1, 34816, 5120, "swiglu"), (4, 34816, 5120, "swiglu"),
                         (5, 5120, 17408, "add"), (64, 5120, 6144, "add"),
                         (8192, 34816, 5120, "swiglu")]:
        need = 256 + up(T * K // 2) + up(spg.nvfp4_sf_bytes(T, K))
        assert spg.act_workspace_bytes("nvfp4", T, N, K, epi) == \
            need + spg.gemm_workspace_bytes("nvfp4", T, N, K, epi)
    for T, N, K, epi in [(1, 5120, 17408, "add"), (1024, 5120, 17408, "add"),
                         (4096, 34816, 5120, "swiglu")]:
        need = up(T * K) + up(4 * T)
        assert spg.act_workspace_bytes("fp8_rowscaled", T, N, K, epi) == \
            need + spg.gemm_workspace_bytes("fp8_rowscaled", T, N, K, epi)
    assert lib.spg_act_workspace_bytes(2, 64, 64, 64, 0) == 0      # per-tensor: no operator
    assert lib.spg_act_workspace_bytes(1, 64, 64, 96, 0) == 0      # NVFP4 K % 64
    assert lib.spg_act_workspace_bytes(0, 0, 64, 64, 0) == 0


def test_route_selector_swap(lib, monkeypatch):
    """The swapped narrow-T tile: FP8 row-scaled, one problem, linear or
    linear_add, T <= 128; token tile 64 or 128 wide, weights in 256-row tiles.
    With fewer weight tiles than pairs every tile is split along K and its
    pieces run as the pairs of one cluster (variant 8, no workspace, with or
    without one); SPG_FORCE_TAIL=none keeps the whole tiles."""
    monkeypatch.delenv("SPG_FORCE_TAIL", raising=False)
    monkeypatch.setenv("SPG_FORCE_VARIANT", "swap")
    for T, bn in [(1, 64), (64, 64), (65, 128), (128, 128)]:
        for epi in ["linear", "add"]:
            for ws in (False, True):
                r = spg.select_route("fp8_rowscaled", T, 5120, 17408, epi, workspace=ws)
                assert r["swap_ab"] == 1 and r["block_m"] == 256 and r["block_n"] == bn, (T, r)
                assert r["variant"] == 8 and r["tiles"] == 20 and r["split_k"] == 3, r
                assert r["split_n"] == 1 and r["workspace_bytes"] == 0, r
                assert r["grid"] == 2 * 60
                assert r["smem_bytes"] <= 232448
            assert spg.gemm_workspace_bytes("fp8_rowscaled", T, 5120, 17408, epi) == 0
    monkeypatch.setenv("SPG_FORCE_TAIL", "none")
    plain = spg.select_route("fp8_rowscaled", 64, 5120, 17408, "add")
    assert plain["swap_ab"] == 1 and plain["variant"] == 6 and plain["split_k"] == 1
    assert plain["grid"] == 40
    monkeypatch.delenv("SPG_FORCE_TAIL")
    # more weight tiles than pairs (forced): the last partial wave splits
    # through a workspace, without one the tiles stay whole
    r = spg.select_route("fp8_rowscaled", 64, 40960, 17408, "add", workspace=True)
    assert r["variant"] == 6 and r["tiles"] == 160 and r["split_k"] > 1 and r["workspace_bytes"] > 0
    r = spg.select_route("fp8_rowscaled", 64, 40960, 17408, "add")
    assert r["variant"] == 6 and r["split_k"] == 1 and r["workspace_bytes"] == 0
    # the default: swapped while the weight tiles leave half of the pairs
    # free (or T <= 16 and one wave of tiles)
    monkeypatch.delenv("SPG_FORCE_VARIANT")
    for T, N, swapped in [(1, 5120, 1), (64, 6144, 1), (128, 9728, 1), (128, 9984, 0),
                          (16, 17408, 1), (17, 17408, 0), (16, 19712, 0), (129, 5120, 0)]:
        r = spg.select_route("fp8_rowscaled", T, N, 17408, "add", workspace=True)
        assert r["swap_ab"] == swapped, (T, N, r)
    # a short K is not split when the finish costs more than it saves
    r = spg.select_route("fp8_rowscaled", 64, 2048, 1024, "add", workspace=True)
    assert r["swap_ab"] == 1 and r["split_k"] == 1
    # not swapped: wider T, SwiGLU, batches, other GEMM kinds
    assert spg.select_route("fp8_rowscaled", 129, 5120, 17408, "add")["swap_ab"] == 0
    assert spg.select_route("fp8_rowscaled", 64, 5120, 17408, "swiglu")["swap_ab"] == 0
    assert spg.select_route("fp8_tensor", 64, 5120, 17408, "linear", 2)["swap_ab"] == 0
    assert spg.select_route("nvfp4", 64, 5120, 17408, "add")["swap_ab"] == 0


def test_route_selector_cluster_split(lib, monkeypatch):
    """NVFP4 with few tiles: one-CTA 128 x 128 tiles whose K is split over
    the CTAs of a cluster (variant 7) wherever every tile gets two to four
    pieces of at least 8 K blocks in one wave, with or without a workspace
    (it needs none); the GEMV keeps decode widths, wide problems keep the
    pair tiles."""
    monkeypatch.delenv("SPG_FORCE_VARIANT", raising=False)
    monkeypatch.delenv("SPG_FORCE_TAIL", raising=False)
    for T, N, K, epi, S in [(3, 5120, 17408, "add", 3), (128, 5120, 17408, "linear", 3),
                            (64, 5120, 6144, "swiglu", 3), (512, 512, 4096, "add", 2),
                            (200, 1024, 8192, "add", 4)]:
        for ws in (False, True):
            r = spg.select_route("nvfp4", T, N, K, epi, workspace=ws)
            tiles = -(-T // 128) * -(-N // 128)
            assert (r["variant"], r["block_m"], r["block_n"], r["split_k"]) == (7, 128, 128, S), r
            assert r["grid"] == tiles * S <= 152 and r["workspace_bytes"] == 0, r
            nkb = K // 256
            kbps = -(-nkb // S)
            assert kbps >= 8 and (S - 1) * kbps < nkb  # no empty piece
        assert spg.gemm_workspace_bytes("nvfp4", T, N, K, epi) == 0
    assert spg.select_route("nvfp4", 1, 5120, 17408, "add")["variant"] == 4   # GEMV
    assert spg.select_route("nvfp4", 256, 5120, 17408, "add")["variant"] == 2  # 80 tiles
    assert spg.select_route("nvfp4", 1024, 5120, 17408, "add")["variant"] == 3
    assert spg.select_route("nvfp4", 64, 5120, 2048, "add")["variant"] != 7   # 8 K blocks
    monkeypatch.setenv("SPG_FORCE_VARIANT", "1sm256_cks")
    r = spg.select_route("nvfp4", 256, 5120, 17408, "add")
    assert (r["variant"], r["block_n"], r["split_k"], r["grid"]) == (7, 256, 3, 120), r
    monkeypatch.setenv("SPG_FORCE_VARIANT", "2sm_st")
    assert spg.select_route("nvfp4", 128, 5120, 17408, "add")["variant"] == 3


def test_route_selector_k_split(lib, monkeypatch):
    """Workspace routes split the last partial wave along K; the plain routes never do."""
    monkeypatch.delenv("SPG_FORCE_VARIANT", raising=False)
    monkeypatch.delenv("SPG_FORCE_TAIL", raising=False)
    for kind, T, N, K, epi in [("fp8_rowscaled", 256, 5120, 17408, "add"),
                               ("fp8_rowscaled", 64, 6144, 17408, "linear"),
                               ("nvfp4", 128, 5120, 17408, "add"),
                               ("fp8_tensor", 128, 4096, 16384, "linear")]:
        # narrow T splits inside clusters by default; pin the unswapped pair tile
        pin = {"nvfp4": "2sm_st", "fp8_rowscaled": "2sm", "fp8_tensor": "2sm"}[kind]
        monkeypatch.setenv("SPG_FORCE_VARIANT", pin)
        plain = spg.select_route(kind, T, N, K, epi)
        assert plain["split_k"] == 1 and plain["workspace_bytes"] == 0
        r = spg.select_route(kind, T, N, K, epi, workspace=True)
        assert r["block_m"] == 256 and 2 <= r["split_k"] <= 4, (kind, T, r)
        tail = r["tiles"] % 76 if r["tiles"] % 76 else 76
        assert r["tiles"] < 76 and tail == r["tiles"]
        # slices (piece x CTA x 128 rows x block_n fp32), then one 8-byte
        # counter per (CTA, lane quarter, 32-column chunk)
        cw = 64 if epi == "swiglu" else 32
        per_tile = r["split_k"] * 2 * 128 * r["block_n"] * 4 + 2 * 4 * (r["block_n"] // cw) * 8
        assert r["workspace_bytes"] == tail * per_tile
        ws = spg.gemm_workspace_bytes(kind, T, N, K, epi)
        # the per-tensor size covers both B layouts
        assert ws == r["workspace_bytes"] if kind != "fp8_tensor" else ws >= r["workspace_bytes"]
        items = r["tiles"] * r["split_k"]
        assert r["grid"] == 2 * min(items, 76)
        nkb = (K // 2 if kind == "nvfp4" else K + 127) // 128
        kbps = -(-nkb // r["split_k"])
        assert kbps >= 4 and (r["split_k"] - 1) * kbps < nkb  # no empty piece
    monkeypatch.delenv("SPG_FORCE_VARIANT", raising=False)
    # NVFP4 at T = 256: the one-CTA 128 x 128 tile (measured faster there)
    assert spg.select_route("nvfp4", 256, 5120, 17408, "add", workspace=True)["block_m"] == 128
    # short K: the finish costs more than the split saves
    assert spg.gemm_workspace_bytes("fp8_rowscaled", 256, 6144, 5120, "add") == 0
    # whole waves (19 x 4 pair tiles on 76 pairs): nothing to split
    assert spg.gemm_workspace_bytes("fp8_rowscaled", 19 * 256, 1024, 17408, "add") == 0
    # the tail pin
    monkeypatch.setenv("SPG_FORCE_TAIL", "none")
    assert spg.select_route("fp8_rowscaled", 256, 5120, 17408, "add", workspace=True)[
        "split_k"] == 1
    monkeypatch.setenv("SPG_FORCE_TAIL", "k")
    r = spg.select_route("fp8_rowscaled", 1024, 5120, 17408, "add", workspace=True)
    assert r["split_k"] > 1 and r["split_n"] == 1


def _vp(x):
    return ctypes.c_void_p(x)


def test_argument_validation_before_launch(lib):
    A, Wt, Y = _vp(0x10000), _vp(0x20000), _vp(0x30000)
    sa, sw = _vp(0x40000), _vp(0x50000)
    f = lib.fp8_rowscaled_gemm
    assert f(A, sa, Wt, sw, None, Y, -1, 8, 16, 0, None) == 1
    assert f(A, sa, Wt, sw, None, Y, 4, 8, 16, 3, None) == 1
    assert f(A, sa, Wt, sw, None, Y, 0, 8, 16, 0, None) == 0          # empty: no-op
    assert f(None, sa, Wt, sw, None, Y, 4, 8, 16, 0, None) == 1
    assert f(A, sa, Wt, sw, None, Y, 4, 8, 24, 0, None) == 2          # K % 16
    assert f(A, sa, Wt, sw, None, Y, 4, 12, 16, 0, None) == 2         # N % 8
    assert f(A, sa, Wt, sw, None, Y, 4, 24, 16, 2, None) == 2         # SwiGLU N % 16
    assert f(A, sa, Wt, sw, None, Y, 4, 8, 16, 1, None) == 1          # ADD without residual
    assert f(_vp(0x10008), sa, Wt, sw, None, Y, 4, 8, 16, 0, None) == 3
    g = lib.nvfp4_gemm
    assert g(A, A, sa, Wt, Wt, sw, None, Y, 4, 8, 128, 0, None) == 2   # K % 256
    t = lib.fp8_tensor_gemm
    assert t(b"X", b"T", 1, A, 0, sa, Wt, 0, sw, Y, 0, 4, 8, 16, None) == 1
    assert t(b"T", b"N", 1, A, 0, sa, Wt, 0, sw, Y, 0, 8, 8, 16, None) == 2   # M % 16 for 'T'
    assert t(b"N", b"T", 0, A, 0, sa, Wt, 0, sw, Y, 0, 4, 8, 16, None) == 0   # empty batch
    q = lib.spg_quantize_fp8_rows
    assert q(A, 4, 12, Y, sa, None) == 2
    assert q(A, 0, 16, Y, sa, None) == 0
    qn = lib.spg_quantize_nvfp4
    assert qn(A, 4, 96, sa, Y, Wt, None) == 2


def test_oracle_is_not_imported_by_the_package():
    import sys
    src = open(os.path.join(ROOT, "scaled_precision_gemm_gb300", "__init__.py")).read()
    assert "oracle" not in re.sub(r'""".*?"""', "", src, flags=re.S)
    assert all("oracle" not in open(os.path.join(ROOT, "scaled_precision_gemm_gb300", "csrc", f)).read()
               for f in os.listdir(os.path.join(ROOT, "scaled_precision_gemm_gb300", "csrc")))


def test_forced_route_is_read_once_until_reload(lib, monkeypatch):
    """The selector reads SPG_FORCE_VARIANT once; a later change of the
    variable takes effect only after spg_debug_reload_env (the binding calls
    it when it sees the variable change)."""
    def route():
        r = spg.Route()
        assert lib.spg_select_route(0, 1000, 5120, 6144, 0, 1, ctypes.byref(r)) == 0
        return r.block_m, r.block_n

    monkeypatch.setenv("SPG_FORCE_VARIANT", "2sm128")
    lib.spg_debug_reload_env()
    assert route() == (256, 128)
    monkeypatch.setenv("SPG_FORCE_VARIANT", "1sm256")
    assert route() == (256, 128)          # not re-read yet
    lib.spg_debug_reload_env()
    assert route() == (128, 256)
    # through the binding, the change is noticed without an explicit reload
    monkeypatch.setenv("SPG_FORCE_VARIANT", "2sm160")
    assert spg.select_route("fp8_rowscaled", 1000, 5120, 6144)["block_n"] == 160
    monkeypatch.delenv("SPG_FORCE_VARIANT")
    lib.spg_debug_reload_env()
