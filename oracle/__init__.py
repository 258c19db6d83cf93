"""Float64 CPU oracle of the SSB phase-variance objective.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the benchmark's
CPU-baseline leg, never by the library.  See ssb_oracle for the definition it follows.
"""
from .ssb_oracle import (  # noqa: F401
    MODES, Geom, aperture, chi, probe, scan_frequencies, rotated_frequencies,
    dft_matrix, fft2_forward, ifft2_inverse, g_plane, full_plane, transfer,
    corrected_spectrum, bf_phase, objective, loss_batch, object_from_spectrum_sum,
    upsample_object, branch_cut_pixels, default_workers,
)
