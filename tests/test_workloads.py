"""The seeded input generators against their stated recipe: shapes, the BF16 storage
of every BF16 tensor, reproducibility, and the distributions (standard deviations,
unit-rms Student-t rows, outlier channels, alpha = 2 r).  The generators hold none of
the method's arithmetic; these checks pin what both the CUDA path and the oracle are
fed."""
import numpy as np
import pytest

from nvfp4_frozen_projection_gb300 import workloads as wl


def _is_bf16(a):
    return np.array_equal(wl.bf16_round(a), a)


def _std_close(a, std, rel=0.02):
    s = float(np.std(a.astype(np.float64)))
    assert s == pytest.approx(std, rel=rel), (s, std)


def test_reproducible():
    a, b = wl.tiny(), wl.tiny()
    for k in ("x", "dy"):
        assert np.array_equal(a[k], b[k])
    for k in ("W", "A", "B"):
        assert np.array_equal(getattr(a["proj"], k), getattr(b["proj"], k))


def test_tiny_recipe():
    d = wl.tiny()
    p = d["proj"]
    assert d["x"].shape == (64, 256) and d["dy"].shape == (64, 256)
    assert (p.d_in, p.d_out, p.r, p.alpha) == (256, 256, 8, 16.0) and p.scale == 2.0
    assert p.W.shape == (256, 256) and p.A.shape == (256, 8) and p.B.shape == (8, 256)
    assert _is_bf16(d["x"]) and _is_bf16(d["dy"]) and _is_bf16(p.A) and _is_bf16(p.B)
    assert p.W.dtype == np.float32


def test_q3b_outlier_channels_and_scales():
    d = wl.q3b()
    x, p = d["x"], d["proj"]
    assert x.shape == (4096, 3072) and _is_bf16(x)
    col_rms = np.sqrt(np.mean(x.astype(np.float64) ** 2, axis=0))
    # round(0.001 * 3072) = 3 channels scaled by 20; every other channel N(0, 1)
    outliers = np.flatnonzero(col_rms > 5.0)
    assert outliers.size == 3
    assert np.all(np.abs(col_rms[outliers] - 20.0) < 1.5)
    assert np.all(np.abs(np.delete(col_rms, outliers) - 1.0) < 0.1)
    _std_close(p.W, 0.02)
    _std_close(p.A, 1.0 / np.sqrt(3072), rel=0.05)
    _std_close(p.B, 0.1, rel=0.05)
    _std_close(d["dy"], 1e-2)
    assert (p.r, p.alpha) == (16, 32.0)


def test_layer3b_recipe():
    d = wl.layer3b()
    x = d["x"]
    assert x.shape == (8192, 3072) and _is_bf16(x)
    # Student-t (nu = 3) scaled to unit global rms: heavy tails, rms 1
    assert float(np.sqrt(np.mean(x.astype(np.float64) ** 2))) == pytest.approx(1.0, rel=0.01)
    assert float(np.max(np.abs(x))) > 20.0
    for g in ("gamma1", "gamma2"):
        assert d[g].shape == (3072,) and _is_bf16(d[g])
        assert float(np.mean(d[g])) == pytest.approx(1.0, abs=0.01)
        _std_close(d[g] - 1.0, 0.1, rel=0.1)
    shapes = {"q": (3072, 3072), "k": (1024, 3072), "v": (1024, 3072), "o": (3072, 3072),
              "gate_up": (16384, 3072), "down": (3072, 8192)}
    for k, shp in shapes.items():
        assert d[k].W.shape == shp, k
        assert d[k].alpha == 2 * d[k].r, k
    # q, k and v are separate tensors; gate|up is one weight, adapters side by side
    # and B block-diagonal
    gu = d["gate_up"]
    assert gu.r == 32 and gu.scale == 2.0
    assert not np.any(gu.B[:16, 8192:]) and not np.any(gu.B[16:, :8192])
    _std_close(d["attn"], 1.0)
    for k in ("dy", "dq", "dk", "dv"):
        assert _is_bf16(d[k])
        _std_close(d[k], 1e-2)
    assert d["dk"].shape == (8192, 1024) and d["dv"].shape == (8192, 1024)
    assert not np.array_equal(d["dk"], d["dv"])
