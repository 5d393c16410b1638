"""Pins of the oracle's normalize-from-partials (``oracle.partials``), the
consumer side of the GEMM-epilogue statistics of NVIDIA/cutlass discussion
874 (example 37's gemm_with_layernorm).

Pinned against: a hand-worked H = 4 example (tests/golden), the two-pass
statistics of ``norm_fwd`` when the partials are exact, independence of the
tile width, and closed forms for one tile and for single-column tiles. A
plausible slip in the combination (a dropped or unweighted tile-mean term,
the wrong width of the ragged last tile, the variance without the mean
subtracted) fails one of them, as the last test shows by planting each.
"""

import json
import os

import numpy as np
import pytest

import oracle
from oracle import partials as P

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "ln_fwd_from_partials_h4.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("tile", ["2", "3"])
@pytest.mark.parametrize("kind", [P.SUM_SQ, P.SUM_M2])
def test_hand_worked_example(tile, kind):
    g = _golden()
    x = np.array(g["x"], dtype=np.float64)
    t = g["tiles"][tile]
    psum, psq = P.row_tile_partials(x, int(tile), kind, fmt="f64")
    np.testing.assert_array_equal(psum, t["psum"])
    np.testing.assert_array_equal(psq, t[kind])
    ones = np.ones(4)
    for mode in (P.LAYERNORM, P.RMSNORM):
        e = g[mode]
        mean, v = P.combine_partials(psum, psq, int(tile), 4, kind, mode)
        np.testing.assert_array_equal(v, e["var"] if mode == P.LAYERNORM else e["ms"])
        o = P.norm_fwd_from_partials(x, psum, psq, int(tile), kind, ones,
                                     None, e["eps"], mode, False, "f64")
        np.testing.assert_array_equal(o["rstd_exact"], e["rstd"])
        np.testing.assert_array_equal(o["y_exact"], e["y"])
        if mode == P.LAYERNORM:
            np.testing.assert_array_equal(o["mean_exact"], e["mean"])


def _rows(rng, rows, H, offset=0.0):
    x = oracle.round_to_format(offset + rng.standard_normal((rows, H)), "bf16")
    return x


@pytest.mark.parametrize("kind", [P.SUM_SQ, P.SUM_M2])
@pytest.mark.parametrize("mode", [P.LAYERNORM, P.RMSNORM])
@pytest.mark.parametrize("H,tile", [(384, 128), (384, 100), (384, 384), (384, 1000),
                                    (320, 64), (1000, 7), (8, 1)])
@pytest.mark.parametrize("zc", [False, True])
def test_exact_partials_give_the_two_pass_statistics(kind, mode, H, tile, zc):
    """With partials kept exact (fp64), the combination reproduces the
    two-pass statistics and output of norm_fwd on the same stored rows."""
    rng = np.random.default_rng(H * 7 + tile)
    x = _rows(rng, 33, H, offset=0.3)
    gamma = 0.1 * rng.standard_normal(H) + (0.0 if zc else 1.0)
    beta = 0.1 * rng.standard_normal(H) if mode == P.LAYERNORM else None
    ref = oracle.norm_fwd(x, None, None, gamma, beta, 1e-5, mode, zc, "bf16")
    psum, psq = P.row_tile_partials(x, tile, kind, fmt="f64")
    got = P.norm_fwd_from_partials(x, psum, psq, tile, kind, gamma, beta, 1e-5, mode, zc, "bf16")
    np.testing.assert_allclose(got["rstd_exact"], ref["rstd_exact"], rtol=1e-12)
    if mode == P.LAYERNORM:
        np.testing.assert_allclose(got["mean_exact"], ref["mean_exact"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(got["y_exact"], ref["y_exact"], rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("kind", [P.SUM_SQ, P.SUM_M2])
def test_independent_of_tile_width(kind):
    rng = np.random.default_rng(5)
    x = _rows(rng, 17, 384)
    stats = []
    for tile in (1, 3, 16, 100, 128, 383, 384, 4096):
        psum, psq = P.row_tile_partials(x, tile, kind, fmt="f64")
        stats.append(P.combine_partials(psum, psq, tile, 384, kind, P.LAYERNORM))
    for m, v in stats[1:]:
        np.testing.assert_allclose(m, stats[0][0], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(v, stats[0][1], rtol=1e-12)


def test_closed_forms_one_tile_and_single_columns():
    rng = np.random.default_rng(9)
    x = _rows(rng, 5, 64)
    # one tile: M2 is the row's own centred sum of squares, the sum form
    # reads E[s^2] - E[s]^2 straight off
    psum, psq = P.row_tile_partials(x, 64, P.SUM_M2, fmt="f64")
    m, v = P.combine_partials(psum, psq, 64, 64, P.SUM_M2, P.LAYERNORM)
    np.testing.assert_allclose(v, psq[:, 0] / 64, rtol=1e-14)
    np.testing.assert_allclose(v, x.var(axis=1), rtol=1e-12)
    # single-column tiles: every tile's M2 is 0 and its mean is the value
    psum, psq = P.row_tile_partials(x, 1, P.SUM_M2, fmt="f64")
    assert (psq == 0).all()
    np.testing.assert_array_equal(psum, x)
    m, v = P.combine_partials(psum, psq, 1, 64, P.SUM_M2, P.LAYERNORM)
    np.testing.assert_allclose(v, x.var(axis=1), rtol=1e-12)
    assert list(P.tile_widths(10, 4)) == [4, 4, 2]
    assert list(P.tile_widths(8, 4)) == [4, 4]


def test_fp32_partials_stay_within_fp32_bounds():
    """Partials rounded to fp32, as an epilogue stores them, move the
    statistics by no more than fp32 rounding of the sums allows."""
    rng = np.random.default_rng(11)
    x = _rows(rng, 64, 384)
    ref = oracle.norm_fwd(x, None, None, np.ones(384), None, 1e-5, P.LAYERNORM, False, "bf16")
    for kind in (P.SUM_SQ, P.SUM_M2):
        psum, psq = P.row_tile_partials(x, 128, kind, fmt="f32")
        o = P.norm_fwd_from_partials(x, psum, psq, 128, kind, np.ones(384), None, 1e-5,
                                     P.LAYERNORM, False, "bf16")
        np.testing.assert_allclose(o["rstd_exact"], ref["rstd_exact"], rtol=1e-6)
        scale = np.abs(x).mean(axis=1)
        assert (np.abs(o["mean_exact"] - ref["mean_exact"]) <= 1e-6 * scale).all()


def test_planted_mistakes_fail_the_pins(monkeypatch):
    """Each plausible slip in the combination, planted in the oracle, fails
    at least one of the pins above."""
    g = _golden()
    x = np.array(g["x"], dtype=np.float64)
    rng = np.random.default_rng(3)
    xr = _rows(rng, 9, 384, offset=0.5)
    ref = oracle.norm_fwd(xr, None, None, np.ones(384), None, 1e-5, P.LAYERNORM, False, "bf16")

    def caught(fn):
        monkeypatch.setattr(P, "combine_partials", fn)
        try:
            ok_hand = True
            for tile in (2, 3):
                psum, psq = P.row_tile_partials(x, tile, P.SUM_M2, fmt="f64")
                _, v = P.combine_partials(psum, psq, tile, 4, P.SUM_M2, P.LAYERNORM)
                ok_hand &= bool(np.allclose(v, 3.5))
            psum, psq = P.row_tile_partials(xr, 100, P.SUM_M2, fmt="f64")
            o = P.norm_fwd_from_partials(xr, psum, psq, 100, P.SUM_M2, np.ones(384), None,
                                         1e-5, P.LAYERNORM, False, "bf16")
            ok_two_pass = bool(np.allclose(o["rstd_exact"], ref["rstd_exact"], rtol=1e-12))
            return not (ok_hand and ok_two_pass)
        finally:
            monkeypatch.undo()

    real = P.combine_partials
    n_of = P.tile_widths

    def drop_tile_mean_term(psum, psq, tile, H, kind, mode):
        mean = psum.sum(axis=1) / H
        return mean, psq.sum(axis=1) / H

    def unweighted_tile_term(psum, psq, tile, H, kind, mode):
        n = n_of(H, tile).astype(float)
        mean = psum.sum(axis=1) / H
        return mean, (psq.sum(axis=1) + ((psum / n - mean[:, None]) ** 2).sum(axis=1)) / H

    def full_width_last_tile(psum, psq, tile, H, kind, mode):
        n = np.full(psum.shape[1], float(tile))
        mean = psum.sum(axis=1) / H
        m_t = psum / n
        return mean, (psq.sum(axis=1) + (n * (m_t - mean[:, None]) ** 2).sum(axis=1)) / H

    def mean_not_subtracted(psum, psq, tile, H, kind, mode):
        n = n_of(H, tile).astype(float)
        mean = psum.sum(axis=1) / H
        return mean, (psq + n * (psum / n) ** 2).sum(axis=1) / H

    for bad in (drop_tile_mean_term, unweighted_tile_term, full_width_last_tile,
                mean_not_subtracted):
        assert caught(bad), bad.__name__
    assert not caught(real)
