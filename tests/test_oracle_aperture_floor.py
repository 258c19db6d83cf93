"""Pins of the oracle's aperture floor, decided in exact arithmetic.

Reading R17: a soft-aperture amplitude below 2^-16 transmits nothing.  On a scan grid
commensurate with the detector (no rotation) the shifted apertures a(alpha_k -+ lambda Q')
fall exactly on the aperture's outer edge at many grid points; float64 rounding then
leaves some of them a rounding-level positive amplitude, which the unit-modulus
normalisation of the transfer would turn into a full-size corrected term.  The pages'
zero-transfer rule (both shifted apertures exactly zero, "SSB performance notes", MPS
zero-transfer q-space checkpoint) is read with this floor.

The workloads' geometry is exact in rational numbers: with the detector sampling
d = alpha_c / R_BF and the scan step lambda / (N_d d), the shifted aperture argument in
units of d is (dx, dy) -+ (N_d / N) R_theta (mx, my) for BF offset (dx, dy) and signed scan
frequency indices (mx, my), and the outer edge is R_BF + 1/2.  So every amplitude below is
decided exactly: with fractions at rotation 0 and with 50-digit arithmetic otherwise.  Points
farther than 2^-5 (in units of d) from the edge are decided by the float64 values
themselves (their rounding is below 1e-13 there), the rest exactly.  The pins:

* every amplitude that is exactly zero is zero in the oracle (the floor is needed: at
  rotation 0 hundreds of them come out positive in float64 without it);
* every exact amplitude of at least 2^-16 is the oracle's within 1e-12 (on the rotated
  grids some lie in [2^-16, 2^-8), so a floor of 2^-8 fails this);
* the oracle's two-sideband transfer is exactly zero wherever both shifted apertures are
  exactly zero (a floor applied to a(alpha_k) alone fails this);
* the genuinely positive amplitudes that the floor zeroes (exact value in (0, 2^-16)) are
  counted: none on the unrotated grids, 8 at the small workload's 5 degrees, and their
  effect on the loss (1.05e-6 relative) is a tenth of the 1e-5 parity tolerance.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import ssb_oracle as _core  # the module whose aperture() reads the floor
import ssb_synth

mpmath = pytest.importorskip("mpmath")

FLOOR = 2.0 ** -16
BAND = 2.0 ** -5  # points closer than this to the edge (units of d) are decided exactly


def _ideal(w):
    R = Fraction(str(w.bf_radius_px))
    return R + Fraction(1, 2), Fraction(w.det_n, w.scan_n)


def _exact_amplitude(w, dy, dx, sgn, my, mx, rot):
    """Exact a(alpha_k + sgn lambda R_rot Q) of the ideal geometry (float of the exact value)."""
    edge, r = _ideal(w)
    if rot == 0.0:
        ex = dx + sgn * mx * r
        ey = dy + sgn * my * r
        d2 = ex * ex + ey * ey
        if d2 >= edge * edge:
            return 0.0
        with mpmath.workdps(50):
            v = mpmath.mpf(edge.numerator) / edge.denominator - mpmath.sqrt(
                mpmath.mpf(d2.numerator) / d2.denominator)
            return float(min(v, 1))
    with mpmath.workdps(50):
        c, s = mpmath.cos(mpmath.mpf(rot)), mpmath.sin(mpmath.mpf(rot))
        rr = mpmath.mpf(r.numerator) / r.denominator
        ex = dx + sgn * rr * (mx * c - my * s)
        ey = dy + sgn * rr * (mx * s + my * c)
        v = mpmath.mpf(edge.numerator) / edge.denominator - mpmath.sqrt(ex * ex + ey * ey)
        return float(min(max(v, 0), 1))


def _shifted(g, k, sgn, rot):
    """The float64 arguments alpha_k + sgn lambda Q' exactly as the oracle's transfer forms them."""
    lqx, lqy = oracle.rotated_frequencies(g, rot)
    return g.alpha_x[k] + sgn * (g.lam * lqx), g.alpha_y[k] + sgn * (g.lam * lqy)


def _edge_census(name, rot):
    """Per (k, sign): the oracle's amplitudes, the exact ones on the points near the edge,
    and the tallies the pins need."""
    w = ssb_synth.WORKLOADS[name]
    geom = ssb_synth.make_geometry(w)
    g = oracle.Geom.from_obj(geom)
    n = g.n
    m = np.fft.fftfreq(n, d=1.0 / n).astype(int)
    edge = float(_ideal(w)[0])
    out = {"exact_zero_raw_positive": 0, "floored_positive": 0, "band_2m16_2m8": 0,
           "max_err_above_floor": 0.0, "exact_zero_nonzero": 0, "both_zero": []}
    for k in range(g.n_bf):
        dy, dx = int(geom.bf_det_yx[k][0]), int(geom.bf_det_yx[k][1])
        zero_masks = []
        for sgn in (-1, 1):
            bx, by = _shifted(g, k, sgn, rot)
            a = oracle.aperture(bx, by, g.semi, g.dalpha)
            floor, _core.APERTURE_FLOOR = _core.APERTURE_FLOOR, 0.0
            try:
                raw = oracle.aperture(bx, by, g.semi, g.dalpha)  # the same without the floor
            finally:
                _core.APERTURE_FLOOR = floor
            d = np.sqrt(bx * bx + by * by) / g.dalpha
            zero = d >= edge  # exact outside the band
            near = np.argwhere(np.abs(d - edge) < BAND)
            for iy, ix in near:
                ae = _exact_amplitude(w, dy, dx, sgn, int(m[iy]), int(m[ix]), rot)
                zero[iy, ix] = ae == 0.0
                if ae == 0.0:
                    if a[iy, ix] != 0.0:
                        out["exact_zero_nonzero"] += 1
                    out["exact_zero_raw_positive"] += int(raw[iy, ix] > 0.0)
                elif ae < FLOOR * (1.0 - 1e-9):
                    out["floored_positive"] += 1
                    assert a[iy, ix] == 0.0
                else:
                    out["max_err_above_floor"] = max(out["max_err_above_floor"], abs(a[iy, ix] - ae))
                    out["band_2m16_2m8"] += int(ae < 2.0 ** -8)
            # away from the edge the float64 amplitude is either exactly 0 or well above it
            far = np.abs(d - edge) >= BAND
            assert np.all(a[far & (d >= edge)] == 0.0)
            assert np.all(a[far & (d < edge)] >= BAND)
            zero_masks.append(zero)
        out["both_zero"].append(zero_masks[0] & zero_masks[1])
    return g, out


@pytest.mark.parametrize("name,rot", [("tiny", 0.0), ("small", 0.0)])
def test_floor_zeroes_exactly_the_edge_points_on_unrotated_grids(name, rot):
    _, s = _edge_census(name, rot)
    print(name, rot, {k: v for k, v in s.items() if k != "both_zero"})
    assert s["exact_zero_nonzero"] == 0
    assert s["max_err_above_floor"] <= 1e-12
    assert s["floored_positive"] == 0  # no genuinely positive amplitude is zeroed
    # the floor is needed: float64 leaves rounding-level amplitudes on the exact edge
    assert s["exact_zero_raw_positive"] > 0


@pytest.mark.parametrize("name,rot,max_floored", [("tiny", 0.2, 0), ("small", math.radians(5.0), 16)])
def test_floor_keeps_every_amplitude_above_it_on_rotated_grids(name, rot, max_floored):
    _, s = _edge_census(name, rot)
    print(name, rot, {k: v for k, v in s.items() if k != "both_zero"})
    assert s["exact_zero_nonzero"] == 0
    assert s["max_err_above_floor"] <= 1e-12
    # amplitudes between 2^-16 and 2^-8 exist here, so a higher floor would fail above
    assert s["band_2m16_2m8"] > 0
    # genuinely positive amplitudes below the floor (zeroed by the reading), counted
    assert s["floored_positive"] <= max_floored


def test_transfer_is_exactly_zero_where_both_shifted_apertures_are(tiny_data):
    w, geom, _, _ = tiny_data
    g, s = _edge_census("tiny", 0.0)
    theta = w.truth  # rotation 0: the grid is commensurate with the detector
    hits = 0
    for k in range(g.n_bf):
        gam = oracle.transfer(g, k, theta)
        both = s["both_zero"][k]
        assert np.all(gam[both] == 0.0), k
        hits += int(both.sum())
    assert hits > 0
    # without the floor some of those points would carry a rounding-level transfer
    assert s["exact_zero_raw_positive"] > 0


def test_loss_effect_of_the_floor_is_below_the_tolerance(monkeypatch):
    """At the small workload's truth (5 degrees) the floor zeroes 8 genuinely positive
    amplitudes below 2^-16 (exact values near 6e-6).  The normalised transfer is
    discontinuous at the aperture edge, so each of them is a full-size term either way; the
    loss moves by 1.05e-6 relative against a floor that zeroes rounding-level amplitudes only
    (2^-40), a tenth of the 1e-5 parity tolerance.  A float32 evaluation cannot place such
    points reliably (its amplitude rounding near the edge is a few 1e-6), which is why the
    floor sits at 2^-16, some five times above it."""
    w = ssb_synth.WORKLOADS["small"]
    geom, counts, _ = ssb_synth.simulate_counts_numpy(w)
    base = oracle.objective(geom, w.truth, counts=counts)["loss"]
    monkeypatch.setattr(_core, "APERTURE_FLOOR", 2.0 ** -40)  # rounding-level zeros only
    low = oracle.objective(geom, w.truth, counts=counts)["loss"]
    rel = abs(base - low) / base
    print("relative loss change, floor 2^-16 against 2^-40:", rel)
    assert rel < 2e-6
