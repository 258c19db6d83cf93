"""Pure-Python brute-force evaluation of the SSB objective for tiny inputs.

Written independently of the vectorised oracle: direct double sums for both
transforms on the full grid (no half-plane, no mirror rule, no FFT), per-point
transfer evaluation with cmath, and explicit moment loops.  The aperture amplitudes come
from 50-digit arithmetic on the exact input values, so an amplitude is zero only when it
is zero exactly (the oracle reaches the same zeros through its 2^-16 floor; where the two
could differ, genuine amplitudes below 2^-16, the floor's own pins count them).  Only
usable for N <= 8 and a handful of BF pixels.
"""
import cmath
import math

import mpmath


def _signed(q, n):
    # fftfreq ordering: 0..n/2-1 positive, n/2..n-1 negative (Nyquist negative)
    return q if q < n // 2 else q - n


def _amplitude(ax, ay, semi, da):
    """Soft aperture clip((semi - |alpha|)/da + 1/2, 0, 1) evaluated in 50-digit arithmetic
    from the arguments' exact values (mpmath numbers or floats), so that zero means exactly
    zero: no floor, no float64 rounding at the edge."""
    with mpmath.workdps(50):
        a = (mpmath.mpf(semi) - mpmath.sqrt(ax * ax + ay * ay)) / mpmath.mpf(da) + mpmath.mpf(1) / 2
        return float(min(max(a, 0), 1))


def _probe(ax, ay, lam, semi, da, c10, c12, phi12, amp=None):
    if amp is None:
        amp = _amplitude(ax, ay, semi, da)
    ax, ay = float(ax), float(ay)
    ph = (math.pi / lam) * (c10 * (ax * ax + ay * ay)
                            + c12 * ((ax * ax - ay * ay) * math.cos(2 * phi12)
                                     + 2 * ax * ay * math.sin(2 * phi12)))
    return amp, ph


def objective_loops(counts, geom, theta, mode="ssb2"):
    n = int(geom.scan_n)
    p = n * n
    lam = geom.wavelength_A
    semi = geom.semiangle_mrad * 1e-3
    da = geom.det_sampling_mrad * 1e-3
    c10, c12, phi12, rot = theta[0] * 10.0, theta[1] * 10.0, theta[2], theta[3]
    cr, sr = math.cos(rot), math.sin(rot)
    with mpmath.workdps(50):
        mcr, msr = mpmath.cos(mpmath.mpf(rot)), mpmath.sin(mpmath.mpf(rot))
    nb = len(geom.bf_det_yx)
    s1 = [[0.0] * n for _ in range(n)]
    s2 = [[0.0] * n for _ in range(n)]
    phases = []
    for k in range(nb):
        ay_k = float(geom.bf_det_yx[k][0]) * da
        ax_k = float(geom.bf_det_yx[k][1]) * da
        with mpmath.workdps(50):
            may_k = mpmath.mpf(float(geom.bf_det_yx[k][0])) * mpmath.mpf(da)
            max_k = mpmath.mpf(float(geom.bf_det_yx[k][1])) * mpmath.mpf(da)
        img = [[float(counts[k][y][x]) for x in range(n)] for y in range(n)]
        # forward DFT on the full grid
        spec = [[0j] * n for _ in range(n)]
        for qy in range(n):
            for qx in range(n):
                acc = 0j
                for y in range(n):
                    for x in range(n):
                        acc += img[y][x] * cmath.exp(-2j * math.pi * (qy * y + qx * x) / n)
                spec[qy][qx] = acc
        # correction at each signed frequency
        ak_amp, ak_ph = _probe(ax_k, ay_k, lam, semi, da, c10, c12, phi12)
        corr = [[0j] * n for _ in range(n)]
        for qy in range(n):
            for qx in range(n):
                if qx == 0 and qy == 0:
                    corr[qy][qx] = spec[0][0]
                    continue
                fx = _signed(qx, n) / (n * geom.scan_step_A)
                fy = _signed(qy, n) / (n * geom.scan_step_A)
                lx = lam * (cr * fx - sr * fy)
                ly = lam * (sr * fx + cr * fy)
                # the shifted apertures' amplitudes from the exact shifted arguments
                with mpmath.workdps(50):
                    mfx = mpmath.mpf(_signed(qx, n)) / (n * mpmath.mpf(geom.scan_step_A))
                    mfy = mpmath.mpf(_signed(qy, n)) / (n * mpmath.mpf(geom.scan_step_A))
                    mlx = mpmath.mpf(lam) * (mcr * mfx - msr * mfy)
                    mly = mpmath.mpf(lam) * (msr * mfx + mcr * mfy)
                    amp_m = _amplitude(max_k - mlx, may_k - mly, semi, da)
                    amp_p = _amplitude(max_k + mlx, may_k + mly, semi, da)
                am, pm = _probe(ax_k - lx, ay_k - ly, lam, semi, da, c10, c12, phi12, amp_m)
                ap, pp = _probe(ax_k + lx, ay_k + ly, lam, semi, da, c10, c12, phi12, amp_p)
                if mode == "ssb2":
                    term1 = ak_amp * am * cmath.exp(1j * (pm - ak_ph))
                    term2 = ak_amp * ap * cmath.exp(1j * (ak_ph - pp))
                    gam = term1 - term2
                    corr[qy][qx] = 0j if abs(gam) == 0.0 else spec[qy][qx] * gam.conjugate() / abs(gam)
                elif mode == "ssb1":
                    corr[qy][qx] = (spec[qy][qx] * cmath.exp(1j * (ak_ph - pm))
                                    if ak_amp * am > 0.0 else 0j)
                else:
                    corr[qy][qx] = spec[qy][qx]
        # inverse DFT and phase
        ph = [[0.0] * n for _ in range(n)]
        for y in range(n):
            for x in range(n):
                acc = 0j
                for qy in range(n):
                    for qx in range(n):
                        acc += corr[qy][qx] * cmath.exp(2j * math.pi * (qy * y + qx * x) / n)
                acc /= p
                v = math.atan2(acc.imag, acc.real)
                ph[y][x] = v
                s1[y][x] += v
                s2[y][x] += v * v
        phases.append(ph)
    loss = 0.0
    for y in range(n):
        for x in range(n):
            m = s1[y][x] / nb
            loss += s2[y][x] / nb - m * m
    return loss / p, phases


def upsample_loops(obj, factor):
    """Band-limited interpolation by direct double sums (forward DFT over the N x N grid at
    signed frequencies, then the inverse sum evaluated on the (factor N)^2 grid), per-point
    cmath; tiny inputs only."""
    n = len(obj)
    fn = factor * n
    ks = [_signed(q, n) for q in range(n)]
    spec = {}
    for ky in ks:
        for kx in ks:
            acc = 0j
            for ny in range(n):
                for nx in range(n):
                    acc += obj[ny][nx] * cmath.exp(-2j * math.pi * (ky * ny + kx * nx) / n)
            spec[(ky, kx)] = acc
    out = [[0j] * fn for _ in range(fn)]
    for my in range(fn):
        for mx in range(fn):
            acc = 0j
            for (ky, kx), v in spec.items():
                acc += v * cmath.exp(2j * math.pi * (ky * my + kx * mx) / fn)
            out[my][mx] = acc / (n * n)
    return out
