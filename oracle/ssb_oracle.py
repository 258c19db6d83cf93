"""Float64 CPU oracle for the single-sideband (SSB) phase-variance objective.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module.  It shares no code with the CUDA library and
the library never calls it.

What it computes (the plain definition; no blocking, fusion or reordering):

For every bright-field (BF) detector pixel k, in row-major detector order,
  1. I_k(r)   = counts[k][ry][rx] as float64;
  2. G_k(Q)   = sum_r I_k(r) exp(-2 pi i Q.r), kept as the Hermitian half-plane
                (rfft2), the "complex64 Hermitian G cache" of the pages ("SSB
                performance notes", BF-major G_qk layout entry; "Later SSB performance
                checkpoints", fftA section);
  3. on the full N x N fftfreq grid, Q' = R_theta Q and
        A(alpha)  = a(alpha) exp(i chi(alpha)),
        Gamma_k(Q) = conj(A(alpha_k)) A(alpha_k - lambda Q')
                     - A(alpha_k) conj(A(alpha_k + lambda Q')),
     the two-sideband transfer with "both shifted apertures" and "two shifted-phase
     sincos calls" ("SSB performance notes", MPS zero-transfer q-space checkpoint and
     the v8 follow-ups);
  4. C_k(Q)   = G_k(Q) conj(Gamma_k)/|Gamma_k| (the "gamma normalization"), exactly 0
                where Gamma_k = 0 (zero transfer, same checkpoint), and C_k(0) = G_k(0),
                the positive DC term ("MPS zero-aperture elimination checkpoint");
  5. c_k(r)   = IFFT2[C_k](r) (inverse transforms, column pass then row pass);
  6. phi_k(r) = atan2(Im c_k, Re c_k);
  7. S1(r) = sum_k phi_k(r), S2(r) = sum_k phi_k(r)^2, in ascending k.

Outputs: loss L = (1/P) sum_r [S2/n_bf - (S1/n_bf)^2] (population variance over the
BF terms averaged over all scan pixels; every BF pixel stays in the normalisation,
"SSB performance notes", automatic 8,937-BF checkpoint), mean phase S1/n_bf, and
the object redraw O(r) = (1/n_bf) sum_k c_k(r) with its phase ("phase-of-mean"), and its
band-limited interpolation onto a finer scan grid (upsample_object).

Readings where the pages are silent (each listed in the design notes):
  * transfer "ssb2" (default) is Gamma above; "ssb1" is the single-sideband factor
    exp(i(chi(alpha_k) - chi(alpha_k - lambda Q'))) masked by a(alpha_k) a(alpha_k -
    lambda Q') > 0; "identity" (C = G) is a test mode only;
  * chi(alpha) = (pi/lambda)[C10 |alpha|^2 + C12((ax^2 - ay^2) cos 2phi12
    + 2 ax ay sin 2phi12)], C in Angstrom (nm x 10), alpha in rad;
  * a(alpha) = clip((alpha_c - |alpha|)/d_alpha + 1/2, 0, 1), taken as exactly 0 when
    that value is below APERTURE_FLOOR = 2^-16.  A scan grid commensurate with the
    detector (e.g. no rotation) places shifted apertures exactly on the outer edge, where
    unit-modulus normalisation turns "zero transfer" into a full-magnitude term; without
    the floor, rounding alone would decide between the two.  The pages' zero-transfer
    rule ("both shifted apertures are exactly zero") is read with this floor;
  * Q' = R_theta Q with Q'x = cos Qx - sin Qy, Q'y = sin Qx + cos Qy; the detector
    angles are not rotated;
  * the Nyquist bin of fftfreq is negative and the correction is evaluated at the
    signed frequency of each grid point (no anti-Hermitian shortcut here);
  * atan2 follows the C/numpy convention (atan2(0, 0) = 0).
"""
from __future__ import annotations

import math
import os
from typing import Optional, Sequence

import numpy as np

MODES = ("ssb2", "ssb1", "identity")
APERTURE_FLOOR = 2.0 ** -16


# ----------------------------------------------------------------------------
# geometry and probe
# ----------------------------------------------------------------------------

class Geom:
    """Plain float64 view of the acquisition geometry."""

    def __init__(self, scan_n, scan_step_A, wavelength_A, semiangle_mrad,
                 det_sampling_mrad, bf_det_yx):
        self.n = int(scan_n)
        self.step = float(scan_step_A)
        self.lam = float(wavelength_A)
        self.semi = float(semiangle_mrad) * 1e-3
        self.dalpha = float(det_sampling_mrad) * 1e-3
        yx = np.asarray(bf_det_yx, dtype=np.float64).reshape(-1, 2)
        self.alpha_y = yx[:, 0] * self.dalpha
        self.alpha_x = yx[:, 1] * self.dalpha
        self.n_bf = yx.shape[0]

    @classmethod
    def from_obj(cls, g):
        return cls(g.scan_n, g.scan_step_A, g.wavelength_A, g.semiangle_mrad,
                   g.det_sampling_mrad, g.bf_det_yx)


def aperture(ax, ay, semi, dalpha):
    """Soft probe aperture a(alpha) = clip((alpha_c - |alpha|)/d_alpha + 1/2, 0, 1),
    with values below APERTURE_FLOOR taken as exactly zero."""
    r = np.sqrt(ax * ax + ay * ay)
    a = np.clip((semi - r) / dalpha + 0.5, 0.0, 1.0)
    return np.where(a < APERTURE_FLOOR, 0.0, a)


def chi(ax, ay, lam, c10_A, c12_A, phi12):
    """Aberration phase (rad) for defocus C10 and twofold astigmatism |C12| at phi12."""
    return (np.pi / lam) * (c10_A * (ax * ax + ay * ay)
                            + c12_A * ((ax * ax - ay * ay) * np.cos(2.0 * phi12)
                                       + 2.0 * ax * ay * np.sin(2.0 * phi12)))


def probe(ax, ay, g: Geom, theta):
    """A(alpha) = a(alpha) exp(i chi(alpha))."""
    c10, c12, phi12 = theta[0] * 10.0, theta[1] * 10.0, theta[2]
    return aperture(ax, ay, g.semi, g.dalpha) * np.exp(1j * chi(ax, ay, g.lam, c10, c12, phi12))


def scan_frequencies(g: Geom):
    """(Qx, Qy) broadcastable grids: Qx varies along columns, Qy along rows."""
    f = np.fft.fftfreq(g.n, d=g.step)
    return f[None, :], f[:, None]


def rotated_frequencies(g: Geom, rotation):
    qx, qy = scan_frequencies(g)
    c, s = math.cos(rotation), math.sin(rotation)
    return c * qx - s * qy, s * qx + c * qy


# ----------------------------------------------------------------------------
# transforms
# ----------------------------------------------------------------------------

def dft_matrix(n: int, sign: int) -> np.ndarray:
    """Direct DFT matrix exp(sign 2 pi i j m / n) (brute force, small n only)."""
    j = np.arange(n)
    return np.exp(sign * 2j * np.pi * np.outer(j, j) / n)


def fft2_forward(x, direct=False):
    if direct:
        f = dft_matrix(x.shape[0], -1)
        return f @ x @ f.T
    return np.fft.fft2(x)


def ifft2_inverse(x, direct=False):
    if direct:
        f = dft_matrix(x.shape[0], +1)
        return (f @ x @ f.T) / x.size
    return np.fft.ifft2(x)


def g_plane(counts_k, direct=False) -> np.ndarray:
    """Hermitian half-plane G_k[Qy][Qx], Qx = 0..N/2 (float64 rfft2 of the counts)."""
    i_k = np.asarray(counts_k, dtype=np.float64)
    n = i_k.shape[0]
    if direct:
        return fft2_forward(i_k.astype(np.complex128), direct=True)[:, : n // 2 + 1]
    return np.fft.rfft2(i_k)


def full_plane(gh: np.ndarray) -> np.ndarray:
    """Full N x N spectrum from the half-plane: G(Qy, Qx) = conj(G(-Qy, N - Qx))."""
    n = gh.shape[0]
    out = np.empty((n, n), dtype=np.complex128)
    out[:, : n // 2 + 1] = gh
    ny = (-np.arange(n)) % n
    nx = n - np.arange(n // 2 + 1, n)
    out[:, n // 2 + 1:] = np.conj(gh[ny][:, nx])
    return out


# ----------------------------------------------------------------------------
# correction
# ----------------------------------------------------------------------------

def transfer(g: Geom, k: int, theta) -> np.ndarray:
    """Gamma_k(Q) on the full grid (two-sideband transfer)."""
    lqx, lqy = rotated_frequencies(g, theta[3])
    lqx = g.lam * lqx
    lqy = g.lam * lqy
    ax, ay = g.alpha_x[k], g.alpha_y[k]
    a_k = probe(np.float64(ax), np.float64(ay), g, theta)
    a_m = probe(ax - lqx, ay - lqy, g, theta)
    a_p = probe(ax + lqx, ay + lqy, g, theta)
    return np.conj(a_k) * a_m - a_k * np.conj(a_p)


def corrected_spectrum(g: Geom, k: int, gfull: np.ndarray, theta, mode="ssb2") -> np.ndarray:
    """C_k(Q) for the chosen transfer reading; C_k(0) = G_k(0) in every mode."""
    if mode == "identity":
        return gfull.copy()
    if mode == "ssb2":
        gam = transfer(g, k, theta)
        mag = np.abs(gam)
        safe = np.where(mag > 0.0, mag, 1.0)
        c = np.where(mag > 0.0, gfull * np.conj(gam) / safe, 0.0 + 0.0j)
    elif mode == "ssb1":
        lqx, lqy = rotated_frequencies(g, theta[3])
        lqx = g.lam * lqx
        lqy = g.lam * lqy
        ax, ay = g.alpha_x[k], g.alpha_y[k]
        c10, c12, phi12 = theta[0] * 10.0, theta[1] * 10.0, theta[2]
        dchi = (chi(ax, ay, g.lam, c10, c12, phi12)
                - chi(ax - lqx, ay - lqy, g.lam, c10, c12, phi12))
        mask = (aperture(ax, ay, g.semi, g.dalpha)
                * aperture(ax - lqx, ay - lqy, g.semi, g.dalpha)) > 0.0
        c = np.where(mask, gfull * np.exp(1j * dchi), 0.0 + 0.0j)
    else:
        raise ValueError(mode)
    c[0, 0] = gfull[0, 0]
    return c


# ----------------------------------------------------------------------------
# objective
# ----------------------------------------------------------------------------

def bf_phase(c_spec: np.ndarray, direct=False):
    """(phi_k, c_k): the inverse 2-D transform and its phase."""
    c = ifft2_inverse(c_spec, direct=direct)
    return np.arctan2(c.imag, c.real), c


def _partial(args):
    """Moments and object sum over a contiguous range of BF pixels, ascending k."""
    (geom_args, k0, k1, data, data_is_g, theta, mode, direct, want_object,
     want_phases, branch_tol) = args
    g = Geom(*geom_args)
    n = g.n
    s1 = np.zeros((n, n))
    s2 = np.zeros((n, n))
    osum = np.zeros((n, n), dtype=np.complex128) if want_object else None
    phases = [] if want_phases else None
    near_pi = np.zeros((n, n), dtype=bool)
    for i, k in enumerate(range(k0, k1)):
        gh = data[i] if data_is_g else g_plane(data[i], direct=direct)
        cs = corrected_spectrum(g, k, full_plane(gh), theta, mode)
        phi, c = bf_phase(cs, direct=direct)
        s1 += phi
        s2 += phi * phi
        near_pi |= np.abs(np.abs(phi) - np.pi) < branch_tol
        if want_object:
            osum += c
        if want_phases:
            phases.append(phi)
    return s1, s2, osum, phases, near_pi


def _geom_args(g: Geom):
    yx = np.stack([g.alpha_y / g.dalpha, g.alpha_x / g.dalpha], axis=1)
    return (g.n, g.step, g.lam, g.semi * 1e3, g.dalpha * 1e3, yx)


def objective(geom, theta, counts=None, g_half=None, mode="ssb2", direct=False,
              want_object=False, want_phases=False, workers: int = 1,
              bf_range: Optional[Sequence[int]] = None, branch_tol: float = 1e-4):
    """Evaluate the SSB phase-variance objective in float64.

    geom:   ssb_synth.Geometry-like object or Geom
    counts: [n_bf][N][N] integer counts (or g_half: [n_bf][N][N/2+1] complex)
    workers: >1 splits the BF range into contiguous chunks processed in spawned
             processes; chunk partials are added in ascending chunk order.
    bf_range: optional (k0, k1) restricting the sum (the normalisation then uses
             the restricted count).
    branch_tol: pixels where some BF phase lies within this distance of +-pi are
             flagged in "branch_cut" (a float32 evaluation may land on the other side
             of the atan2 branch cut there).
    Returns a dict with loss, mean_phase, s1, s2, n_bf, branch_cut and optionally
    object / phases.
    """
    g = geom if isinstance(geom, Geom) else Geom.from_obj(geom)
    theta = tuple(float(x) for x in theta)
    data = counts if counts is not None else g_half
    data_is_g = counts is None
    k0, k1 = (0, g.n_bf) if bf_range is None else (int(bf_range[0]), int(bf_range[1]))
    ga = _geom_args(g)
    if workers <= 1 or k1 - k0 < 2 * workers:
        parts = [_partial((ga, k0, k1, data[k0:k1], data_is_g, theta, mode, direct,
                           want_object, want_phases, branch_tol))]
    else:
        import multiprocessing as mp
        bounds = np.linspace(k0, k1, workers + 1).astype(int)
        jobs = [(ga, int(a), int(b), data[a:b], data_is_g, theta, mode, direct,
                 want_object, want_phases, branch_tol)
                for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
        with mp.get_context("spawn").Pool(len(jobs)) as pool:
            parts = pool.map(_partial, jobs)
    n = g.n
    s1 = np.zeros((n, n))
    s2 = np.zeros((n, n))
    osum = np.zeros((n, n), dtype=np.complex128) if want_object else None
    phases = [] if want_phases else None
    near_pi = np.zeros((n, n), dtype=bool)
    for p in parts:
        near_pi |= p[4]
        s1 += p[0]
        s2 += p[1]
        if want_object:
            osum += p[2]
        if want_phases:
            phases.extend(p[3])
    nb = k1 - k0
    loss = float(np.mean(s2 / nb - (s1 / nb) ** 2))
    out = {"loss": loss, "mean_phase": s1 / nb, "s1": s1, "s2": s2, "n_bf": nb,
           "branch_cut": near_pi}
    if want_object:
        out["object"] = osum / nb
        out["object_phase"] = np.angle(osum / nb)
    if want_phases:
        out["phases"] = np.stack(phases)
    return out


def loss_batch(geom, thetas, counts=None, g_half=None, mode="ssb2", workers=1):
    """Loss for each trial in `thetas` (shape [T][4])."""
    return np.array([objective(geom, th, counts=counts, g_half=g_half, mode=mode,
                               workers=workers)["loss"] for th in np.asarray(thetas)])


def object_from_spectrum_sum(geom, theta, counts, mode="ssb2"):
    """Object redraw written as IFFT2 of the BF-summed corrected spectrum,
    (1/n_bf) IFFT2[sum_k C_k]; equal to (1/n_bf) sum_k c_k by linearity."""
    g = geom if isinstance(geom, Geom) else Geom.from_obj(geom)
    csum = np.zeros((g.n, g.n), dtype=np.complex128)
    for k in range(g.n_bf):
        csum += corrected_spectrum(g, k, full_plane(g_plane(counts[k])), theta, mode)
    return np.fft.ifft2(csum) / g.n_bf


def upsample_object(obj: np.ndarray, factor: int) -> np.ndarray:
    """Band-limited interpolation of the object redraw onto a scan grid `factor` times
    finer, the plainest reading of the pages' reconstruct(result, upsample=factor)
    ("Later SSB performance checkpoints", joint CUDA calibration, output reconstruction
    at factors 1-4): the N x N spectrum of the object keeps its fftfreq (signed, Nyquist
    negative) frequencies on the (factor N)^2 grid, every other frequency is zero, and
    the inverse transform is scaled so that the samples at multiples of `factor` are the
    original ones:
        O_up(m) = (1/N^2) sum_k O^(k) exp(2 pi i k.m / (factor N)).
    """
    n = obj.shape[0]
    assert obj.shape == (n, n) and factor >= 1
    fn = factor * n
    spec = np.fft.fft2(np.asarray(obj, dtype=np.complex128))
    k = np.fft.fftfreq(n, d=1.0 / n).astype(np.int64)  # signed integer frequencies
    big = np.zeros((fn, fn), dtype=np.complex128)
    big[np.ix_(k % fn, k % fn)] = spec
    return np.fft.ifft2(big) * factor * factor


def branch_cut_pixels(phases: np.ndarray, tol: float = 1e-4) -> np.ndarray:
    """Mask of scan pixels where some BF phase lies within `tol` of +-pi; a float32
    evaluation may legitimately land on the other side of the atan2 branch cut there."""
    return np.any(np.abs(np.abs(phases) - np.pi) < tol, axis=0)


def default_workers() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)
