"""Seeded synthetic 4D-STEM inputs for the SSB phase-variance objective.

This module only makes *inputs*: detector geometry, bright-field (BF) pixel lists,
integer detector counts and trial aberration draws.  It holds none of the SSB method
(no correction, no inverse transform, no phase, no variance).  Both the float64 CPU
oracle and the CUDA library consume what it produces; neither imports the other.

The counts come from a forward-scattering simulation with its own probe function:
a periodic weak-phase object t(r) = exp(i phi(r)) on the N x N scan grid, illuminated
by a probe whose angular spectrum is a(alpha) exp(i chi(alpha)), recorded at point
detector pixels alpha_k.  For detector pixel k the exit intensity over the scan is

    psi_k(r) = IFFT2[ FFT2[t](Q) * A_true(alpha_k - lambda R_theta Q) ](r),
    I_k(r)   = |psi_k(r)|^2,

scaled so that the mean over BF pixels and scan positions equals the configured dose,
then Poisson-sampled.  The dataset sizes, dose, dtypes and true aberrations follow the
five workloads listed for this objective (tiny 32^2 scan / 113 BF up to the full
512^2 scan / 8,937 BF that the "Later SSB performance checkpoints" page measures in
"2026-09-11 full-aperture Apple M5 floor checkpoint").

Conventions (shared by construction with any consumer, stated here once):
  * scan pixel (ry, rx), row y, column x; scan frequencies Q = fftfreq(N, d=step)
    on both axes (Nyquist bin negative);
  * Q' = R_theta Q:  Q'x = cos(t) Qx - sin(t) Qy,  Q'y = sin(t) Qx + cos(t) Qy;
  * detector angles alpha_k = (dx, dy) * det_sampling, with (dy, dx) the BF pixel
    offsets from the detector centre (N_d/2, N_d/2), in row-major detector order;
  * the 300 kV relativistic electron wavelength, 0.0196875 Angstrom;
  * scan step = lambda / (N_d * det_sampling), so the scan Nyquist frequency maps to
    the detector half-width.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

WAVELENGTH_300KV_A = 0.0196875  # Angstrom, relativistic, 300 kV


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic dataset recipe."""
    name: str
    scan_n: int            # N: N x N scan
    det_n: int             # N_d: N_d x N_d detector
    bf_radius_px: float    # BF disk radius on the detector, pixels
    dtype: str             # "u16" or "u32" counts
    mean_count: float      # mean counts per BF pixel per scan position
    object_rms_rad: float  # rms of the object phase
    truth: tuple           # (C10_nm, C12_nm, phi12_rad, rotation_rad)
    seed: int              # generator seed (object noise + Poisson)
    trial_seed: int        # seed for random trial draws
    n_trials: int          # trials in the workload's batch
    semiangle_mrad: float = 20.0
    object_sigma_px: float = 2.0


def _deg(x):
    return math.radians(x)


WORKLOADS = {
    "tiny": Workload("tiny", 32, 24, 6.0, "u16", 200.0, 0.1,
                     (50.0, 0.0, 0.0, 0.0), seed=0, trial_seed=100, n_trials=1),
    "small": Workload("small", 128, 64, 15.0, "u16", 200.0, 0.2,
                      (-80.0, 10.0, _deg(30.0), _deg(5.0)), seed=1, trial_seed=101, n_trials=16),
    "medium": Workload("medium", 256, 96, 27.0, "u32", 500.0, 0.2,
                       (-80.0, 10.0, _deg(30.0), _deg(5.0)), seed=2, trial_seed=102, n_trials=200),
    "full": Workload("full", 512, 192, 53.3, "u32", 1000.0, 0.2,
                     (120.0, 25.0, _deg(60.0), _deg(-12.0)), seed=3, trial_seed=103, n_trials=1),
}


@dataclasses.dataclass
class Geometry:
    """Acquisition geometry; mirrors the C struct ssb_geometry."""
    scan_n: int
    scan_step_A: float
    wavelength_A: float
    semiangle_mrad: float
    det_sampling_mrad: float
    det_n: int
    bf_det_yx: np.ndarray  # float32 [n_bf][2], (dy, dx) px from the detector centre

    @property
    def n_bf(self) -> int:
        return int(self.bf_det_yx.shape[0])


def bf_pixels(det_n: int, radius_px: float) -> np.ndarray:
    """Detector pixels inside the BF disk, row-major, as (dy, dx) offsets from the
    centre (det_n/2, det_n/2): (row - c)^2 + (col - c)^2 <= R^2."""
    c = det_n / 2.0
    rows, cols = np.meshgrid(np.arange(det_n), np.arange(det_n), indexing="ij")
    dy = rows - c
    dx = cols - c
    inside = dy * dy + dx * dx <= radius_px * radius_px
    return np.stack([dy[inside], dx[inside]], axis=1).astype(np.float32)


def make_geometry(w: Workload, bf_subset: Optional[np.ndarray] = None) -> Geometry:
    det_sampling = w.semiangle_mrad / w.bf_radius_px
    step = WAVELENGTH_300KV_A / (w.det_n * det_sampling * 1e-3)
    yx = bf_pixels(w.det_n, w.bf_radius_px)
    if bf_subset is not None:
        yx = yx[bf_subset]
    return Geometry(w.scan_n, float(step), WAVELENGTH_300KV_A, w.semiangle_mrad,
                    float(det_sampling), w.det_n, np.ascontiguousarray(yx))


# ----------------------------------------------------------------------------
# forward model (input synthesis only)
# ----------------------------------------------------------------------------

def _probe_numpy(ax, ay, lam, semi, dalpha, c10_A, c12_A, phi12):
    """Probe angular spectrum used to *simulate* data: soft aperture times exp(i chi)."""
    r = np.sqrt(ax * ax + ay * ay)
    amp = np.clip((semi - r) / dalpha + 0.5, 0.0, 1.0)
    ph = (np.pi / lam) * (c10_A * (ax * ax + ay * ay)
                          + c12_A * ((ax * ax - ay * ay) * np.cos(2 * phi12)
                                     + 2.0 * ax * ay * np.sin(2 * phi12)))
    return amp * np.exp(1j * ph)


def object_phase(n: int, sigma_px: float, rms: float, rng: np.random.Generator) -> np.ndarray:
    """Periodic Gaussian-filtered white noise, renormalised to the requested rms."""
    z = rng.standard_normal((n, n))
    f = np.fft.fftfreq(n)
    f2 = f[:, None] ** 2 + f[None, :] ** 2
    zf = np.fft.ifft2(np.fft.fft2(z) * np.exp(-2.0 * np.pi ** 2 * sigma_px ** 2 * f2)).real
    zf -= zf.mean()
    return rms * zf / zf.std()


def _scan_q(geom: Geometry):
    f = np.fft.fftfreq(geom.scan_n, d=geom.scan_step_A)
    return f[None, :], f[:, None]  # Qx (columns), Qy (rows)


def simulate_counts_numpy(w: Workload, geom: Optional[Geometry] = None,
                          truth: Optional[tuple] = None) -> tuple:
    """Return (geometry, counts [n_bf][N][N] uint16/uint32, object phase [N][N])."""
    geom = geom or make_geometry(w)
    truth = truth if truth is not None else w.truth
    rng = np.random.Generator(np.random.PCG64(w.seed))
    n = geom.scan_n
    phi = object_phase(n, w.object_sigma_px, w.object_rms_rad, rng)
    tf = np.fft.fft2(np.exp(1j * phi))
    qx, qy = _scan_q(geom)
    c, s = math.cos(truth[3]), math.sin(truth[3])
    lqx = geom.wavelength_A * (c * qx - s * qy)
    lqy = geom.wavelength_A * (s * qx + c * qy)
    semi = geom.semiangle_mrad * 1e-3
    da = geom.det_sampling_mrad * 1e-3
    c10, c12, phi12 = truth[0] * 10.0, truth[1] * 10.0, truth[2]
    ak = geom.bf_det_yx.astype(np.float64) * da  # (ay, ax)
    tf2 = np.abs(tf) ** 2
    # dose normalisation from Parseval: mean_r |psi_k|^2 = sum_Q |F_k|^2 / P^2
    p2 = float(n) ** 4
    means = np.empty(geom.n_bf)
    for k in range(geom.n_bf):
        amp = _probe_numpy(ak[k, 1] - lqx, ak[k, 0] - lqy, geom.wavelength_A, semi, da,
                           c10, c12, phi12)
        means[k] = float(np.sum(tf2 * np.abs(amp) ** 2)) / p2
    scale = w.mean_count / means.mean()
    dt = np.uint16 if w.dtype == "u16" else np.uint32
    counts = np.empty((geom.n_bf, n, n), dtype=dt)
    for k in range(geom.n_bf):
        pk = _probe_numpy(ak[k, 1] - lqx, ak[k, 0] - lqy, geom.wavelength_A, semi, da,
                          c10, c12, phi12)
        inten = np.abs(np.fft.ifft2(tf * pk)) ** 2
        lamk = inten * scale
        counts[k] = np.minimum(rng.poisson(lamk), np.iinfo(dt).max).astype(dt)
    return geom, counts, phi


def simulate_counts_torch(w: Workload, device, geom: Optional[Geometry] = None,
                          truth: Optional[tuple] = None, chunk: int = 128):
    """Same recipe on a torch device (complex64), for workloads too large for numpy.

    Returns (geometry, counts tensor [n_bf][N][N] on `device`, object phase numpy)."""
    import torch
    geom = geom or make_geometry(w)
    truth = truth if truth is not None else w.truth
    rng = np.random.Generator(np.random.PCG64(w.seed))
    n = geom.scan_n
    phi = object_phase(n, w.object_sigma_px, w.object_rms_rad, rng)
    dev = torch.device(device)
    tf = torch.fft.fft2(torch.exp(1j * torch.from_numpy(phi).to(dev)))  # complex128
    tf2 = (tf.abs() ** 2).to(torch.float32)[None]
    tf = tf.to(torch.complex64)
    f = np.fft.fftfreq(n, d=geom.scan_step_A)
    qx, qy = f[None, :], f[:, None]
    c, s = math.cos(truth[3]), math.sin(truth[3])
    lam = geom.wavelength_A
    lqx = torch.from_numpy(lam * (c * qx - s * qy)).to(dev, torch.float32)
    lqy = torch.from_numpy(lam * (s * qx + c * qy)).to(dev, torch.float32)
    semi = geom.semiangle_mrad * 1e-3
    da = geom.det_sampling_mrad * 1e-3
    c10, c12, phi12 = truth[0] * 10.0, truth[1] * 10.0, truth[2]
    ak = torch.from_numpy(geom.bf_det_yx.astype(np.float64) * da).to(dev, torch.float32)
    k_pi = math.pi / lam
    c2, s2 = math.cos(2 * phi12), math.sin(2 * phi12)

    def probe(kk):
        # float32 is ample for synthesising inputs; phases are reduced mod 2 pi
        ax = ak[kk, 1][:, None, None] - lqx[None]
        ay = ak[kk, 0][:, None, None] - lqy[None]
        r = torch.sqrt(ax * ax + ay * ay)
        amp = torch.clamp((semi - r) / da + 0.5, 0.0, 1.0)
        ph = k_pi * (c10 * (ax * ax + ay * ay) + c12 * ((ax * ax - ay * ay) * c2 + 2.0 * ax * ay * s2))
        return amp, torch.remainder(ph, 2 * math.pi)

    means = []
    for k0 in range(0, geom.n_bf, chunk):
        kk = torch.arange(k0, min(geom.n_bf, k0 + chunk), device=dev)
        amp, _ = probe(kk)
        means.append(((tf2 * amp * amp).sum(dim=(1, 2), dtype=torch.float64) / float(n) ** 4))
    scale = w.mean_count / float(torch.cat(means).mean())
    tdt = torch.int32 if w.dtype == "u32" else torch.int16
    counts = torch.empty((geom.n_bf, n, n), dtype=tdt, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    for k0 in range(0, geom.n_bf, chunk):
        kk = torch.arange(k0, min(geom.n_bf, k0 + chunk), device=dev)
        amp, ph = probe(kk)
        psi = torch.fft.ifft2(tf[None] * torch.polar(amp, ph))
        rate = (psi.real ** 2 + psi.imag ** 2) * scale
        draw = torch.poisson(rate, generator=gen)
        if w.dtype == "u32":
            counts[k0:k0 + kk.numel()] = draw.clamp_(max=2 ** 31 - 1).to(torch.int32)
        else:
            # uint16 bit pattern stored in an int16 tensor
            counts[k0:k0 + kk.numel()] = draw.clamp_(max=2 ** 16 - 1).to(torch.int32).to(torch.int16)
    return geom, counts, phi


def draw_trials(w: Workload, t: int, seed: Optional[int] = None) -> np.ndarray:
    """Random trial aberrations: C10 ~ U[-200, 200] nm, |C12| ~ U[0, 30] nm,
    phi12 ~ U[0, pi), rotation fixed at the workload's truth.  Returns float64 [t][4]."""
    rng = np.random.Generator(np.random.PCG64(w.trial_seed if seed is None else seed))
    out = np.empty((t, 4))
    out[:, 0] = rng.uniform(-200.0, 200.0, t)
    out[:, 1] = rng.uniform(0.0, 30.0, t)
    out[:, 2] = rng.uniform(0.0, np.pi, t)
    out[:, 3] = w.truth[3]
    return out
