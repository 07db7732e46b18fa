"""Route-selector invariants over a sweep of shapes (host only): what the
kernels rely on when the route is launched.

* a pair route launches an even grid of at most 2 x 76 CTAs, a one-CTA route
  at most 152, the GEMV one CTA per 4 weight-row pairs;
* dynamic shared memory stays within the 232,448-byte opt-in limit (the
  GEMV within its 200 KB bound);
* a K split has 2-4 pieces, none empty, each at least 4 K blocks, and the
  workspace query returns exactly the plan's bytes (the per-tensor GEMM:
  at least, it covers both B layouts); plain routes never split K;
* the swapped tile is FP8 (row-scaled linear / linear_add, or per-tensor),
  T <= 128, one problem; the GEMV is NVFP4 with T <= 4.
"""
import itertools

import pytest

import scaled_precision_gemm_gb300 as spg

SMEM_MAX = 232448
PAIRS = 76


def nkb(kind, K):
    return (K // 2 + 127) // 128 if kind == "nvfp4" else (K + 127) // 128


SHAPES = list(itertools.product([1, 3, 16, 64, 100, 128, 129, 256, 1000, 1024, 4096, 8192],
                                [128, 5120, 6144, 17408, 34816],
                                [256, 1024, 5120, 6144, 17408]))


@pytest.fixture(autouse=True)
def _no_pins(monkeypatch):
    monkeypatch.delenv("SPG_FORCE_VARIANT", raising=False)
    monkeypatch.delenv("SPG_FORCE_TAIL", raising=False)


@pytest.mark.parametrize("kind", ["fp8_rowscaled", "nvfp4", "fp8_tensor"])
@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
def test_route_invariants(kind, epi):
    if kind == "fp8_tensor" and epi != "linear":
        pytest.skip("the per-tensor GEMM has the linear epilogue only")
    for T, N, K in SHAPES:
        if kind == "nvfp4" and K % 256:
            continue
        for ws in (False, True):
            r = spg.select_route(kind, T, N, K, epi, workspace=ws)
            tag = (kind, epi, T, N, K, ws, r)
            assert r["grid"] >= 1, tag
            if r["variant"] == 4 and kind == "nvfp4":
                assert T <= 4 and r["grid"] == (N // 2 + 3) // 4, tag
                assert r["smem_bytes"] <= 200 * 1024 and r["split_k"] == 1, tag
                continue
            assert r["smem_bytes"] <= SMEM_MAX, tag
            if r["block_m"] == 256:
                assert r["grid"] % 2 == 0 and r["grid"] <= 2 * PAIRS, tag
            else:
                assert r["grid"] <= 2 * PAIRS, tag
            if r["swap_ab"]:
                assert kind in ("fp8_rowscaled", "fp8_tensor") and epi != "swiglu" and T <= 128, tag
                assert r["block_n"] == (64 if T <= 64 else 128), tag
            if r["variant"] == 8:
                # swapped tile, every tile split inside clusters of 2 x split_k CTAs
                s, n = r["split_k"], nkb(kind, K)
                kbps = -(-n // s)
                assert r["swap_ab"] == 1 and kind != "nvfp4", tag
                assert 2 <= s <= 4 and kbps >= 4 and (s - 1) * kbps < n, tag
                assert r["tiles"] * s <= PAIRS and r["grid"] == 2 * r["tiles"] * s, tag
                assert r["workspace_bytes"] == 0 and r["split_n"] == 1, tag
                continue
            if r["variant"] == 7 and kind == "nvfp4":
                # K split inside clusters: one piece per CTA, one wave, no workspace
                s, n = r["split_k"], nkb(kind, K)
                kbps = -(-n // s)
                tiles = -(-T // 128) * -(-N // r["block_n"])
                assert 2 <= s <= 4 and kbps >= 8 and (s - 1) * kbps < n, tag
                assert r["block_m"] == 128 and r["grid"] == tiles * s <= 2 * PAIRS, tag
                assert r["workspace_bytes"] == 0 and r["split_n"] == 1, tag
                continue
            if not ws:
                assert r["split_k"] == 1 and r["workspace_bytes"] == 0, tag
            if r["split_k"] > 1:
                s, n = r["split_k"], nkb(kind, K)
                kbps = -(-n // s)
                assert 2 <= s <= 4 and kbps >= 4 and (s - 1) * kbps < n, tag
                assert r["split_n"] == 1 and r["workspace_bytes"] > 0, tag
            if ws:
                need = spg.gemm_workspace_bytes(kind, T, N, K, epi)
                if kind == "fp8_tensor":
                    assert need >= r["workspace_bytes"], tag
                else:
                    assert need == r["workspace_bytes"], tag


def recv_bytes(bn, cw, s):
    """Partial sums one CTA of a cluster K split receives: per owned chunk,
    32-column sub-block, source piece and TMEM lane quarter a 4 KB block."""
    return -(-(bn // cw) // s) * (cw // 32) * s * 4 * 4096


@pytest.mark.parametrize("pin", [None, "1sm_cks", "1sm256_cks", "swap"])
@pytest.mark.parametrize("epi", ["linear", "add", "swiglu"])
def test_cluster_split_plans(pin, epi, monkeypatch):
    """Every K split inside clusters (variants 7 and 8, default or pinned):
    one wave with one piece per CTA (pair), 2-4 pieces, none empty, clusters
    of at most 8 CTAs, and the partial sums each CTA receives fit its
    operand ring, which is where they land."""
    if pin:
        monkeypatch.setenv("SPG_FORCE_VARIANT", pin)
    seen = 0
    for T, N, K in SHAPES:
        for kind in ("nvfp4", "fp8_rowscaled"):
            if kind == "nvfp4" and K % 256:
                continue
            r = spg.select_route(kind, T, N, K, epi)
            tag = (pin, kind, epi, T, N, K, r)
            if r["variant"] == 7 and kind == "nvfp4":
                s, n, bn = r["split_k"], nkb(kind, K), r["block_n"]
                kbps = -(-n // s)
                tiles = -(-T // 128) * -(-N // bn)
                assert 2 <= s <= 4 and kbps >= 8 and (s - 1) * kbps < n, tag
                assert r["grid"] == tiles * s <= 2 * PAIRS, tag
                stage = 128 * 128 + bn * 128 + 2048 + (bn // 128) * 2048
                assert r["stages"] * stage + 1024 + 4 * 2 * 2048 + 256 <= SMEM_MAX, tag
                cw = 64 if epi == "swiglu" else 32
                assert recv_bytes(bn, cw, s) <= r["stages"] * stage, tag
                seen += 1
            elif r["variant"] == 8:
                s, n, bn = r["split_k"], nkb(kind, K), r["block_n"]
                assert kind != "nvfp4" and epi != "swiglu" and r["swap_ab"] == 1, tag
                assert 2 <= s <= 4 and 2 * s <= 8 and (s - 1) * (-(-n // s)) < n, tag
                assert r["tiles"] * s <= PAIRS and r["grid"] == 2 * r["tiles"] * s, tag
                stage = 128 * 128 + bn // 2 * 128
                assert recv_bytes(bn, 32, s) <= r["stages"] * stage, tag
                seen += 1
    if pin != "swap" or epi != "swiglu":
        assert seen > 0
