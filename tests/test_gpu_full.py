"""Parity at the full size the benchmark times (and the SSB1 transfer at the same size): 512 x 512 scan, 192 x 192 detector, all
8,937 BF pixels, uint32 counts (mean 1,000), generated on the GPU exactly as bench.py
does, evaluated through the C ABI in the benchmark's launch configuration, and compared
with the float64 oracle run over every BF pixel in spawned processes on the host cores.

Tolerances as for the other parity tests: loss within 1e-5 relative, mean phase within
1e-4 rad off the atan2 branch cut."""
import numpy as np
import pytest

import oracle
import ssb_synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def full_case():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from stem_ssb_phase_gb300 import build
    build.build()
    import stem_ssb_phase_gb300 as m
    w = ssb_synth.WORKLOADS["full"]
    geom, counts, _ = ssb_synth.simulate_counts_torch(w, "cuda")
    host = counts.cpu().numpy().view(np.uint32)
    ctx = m.SSB(geom, counts)
    del counts
    torch.cuda.empty_cache()
    yield w, geom, host, ctx
    ctx.close()


@pytest.fixture(scope="module")
def full_ref(full_case):
    """The oracle at the trial the benchmark times, over every BF pixel, with the object."""
    w, geom, host, _ = full_case
    theta = ssb_synth.draw_trials(w, 1)[0]
    return theta, oracle.objective(geom, theta, counts=host, want_object=True,
                                   workers=min(32, oracle.default_workers()))


def _check_mean_phase(mp, ref):
    mask = ~ref["branch_cut"]
    err = np.abs(mp.cpu().numpy().astype(np.float64) - ref["mean_phase"])[mask]
    assert mask.mean() > 0.9
    assert err.max() <= 1e-4, (err.max(), int((err > 1e-4).sum()))


def _check_object(gpu_obj, want, tol=1e-5, elem=1e-4):
    """Relative L2 error and, element by element, the error against the largest modulus
    (float32 rounding on these DC-dominated objects reaches 1.6e-5 of it)."""
    o = gpu_obj.astype(np.complex128)
    assert np.linalg.norm(o - want) <= tol * np.linalg.norm(want)
    err = np.abs(o - want)
    assert err.max() <= elem * np.abs(want).max(), err.max() / np.abs(want).max()


def test_full_size_loss_and_mean_phase_match_the_oracle(full_case, full_ref):
    w, geom, host, ctx = full_case
    theta, ref = full_ref  # the trial the benchmark times
    mp, obj, loss = ctx.reconstruct(theta, want_object=True)
    assert abs(loss - ref["loss"]) <= 1e-5 * ref["loss"], (loss, ref["loss"])
    _check_mean_phase(mp, ref)
    _check_object(obj.cpu().numpy(), ref["object"])


def test_full_size_at_the_generating_aberrations(full_case):
    """A second full-size trial: the truth (small loss, phases concentrated near zero)."""
    w, geom, host, ctx = full_case
    mp, _, loss = ctx.reconstruct(w.truth, want_object=False)
    ref = oracle.objective(geom, w.truth, counts=host, workers=min(32, oracle.default_workers()))
    assert abs(loss - ref["loss"]) <= 1e-5 * ref["loss"], (loss, ref["loss"])
    _check_mean_phase(mp, ref)


def test_full_size_batch_equals_scalar_calls(full_case):
    w, geom, host, ctx = full_case
    thetas = np.vstack([np.array(w.truth)[None], ssb_synth.draw_trials(w, 2, seed=9)])
    batch = ctx.loss_batch(thetas)
    singles = np.array([ctx.loss(t) for t in thetas])
    assert np.array_equal(batch, singles)
    assert np.array_equal(ctx.loss_batch(thetas), batch)  # run to run
    # the generating aberrations give the smallest loss of the three
    assert int(np.argmin(batch)) == 0


def test_full_size_ssb1_matches_the_oracle(full_case):
    """The SSB1 transfer at full size: all 512 columns and full complex row transforms."""
    w, geom, host, _ = full_case
    import stem_ssb_phase_gb300 as m
    theta = ssb_synth.draw_trials(w, 1)[0]
    ctx = m.SSB(geom, host, transfer="ssb1")
    try:
        mp, _, loss = ctx.reconstruct(theta, want_object=False)
        batch = ctx.loss_batch(np.array(theta)[None])
    finally:
        ctx.close()
    assert batch[0] == loss
    ref = oracle.objective(geom, theta, counts=host, mode="ssb1",
                           workers=min(32, oracle.default_workers()))
    assert abs(loss - ref["loss"]) <= 1e-5 * ref["loss"], (loss, ref["loss"])
    mask = ~ref["branch_cut"]
    err = np.abs(mp.cpu().numpy().astype(np.float64) - ref["mean_phase"])[mask]
    assert mask.mean() > 0.9
    assert err.max() <= 1e-4, (err.max(), int((err > 1e-4).sum()))


def test_full_size_upsampled_redraw_matches_the_oracle(full_case, full_ref):
    """The 4x redraw the upsampled bench times (2048 x 2048 output) against the oracle's
    full-size object interpolated by the oracle: object within 1e-5 relative L2, phase
    within 1e-4 rad (modulo 2 pi) where the modulus is at least 5 % of its RMS."""
    _, _, _, ctx = full_case
    theta, ref = full_ref
    ph, obj, _ = ctx.reconstruct_upsampled(theta, 4)
    up = oracle.upsample_object(ref["object"], 4)
    _check_object(obj.cpu().numpy(), up)
    mask = np.abs(up) >= 0.05 * np.sqrt(np.mean(np.abs(up) ** 2))
    assert mask.mean() > 0.5
    d = np.angle(np.exp(1j * (ph.cpu().numpy().astype(np.float64) - np.angle(up))))[mask]
    assert np.abs(d).max() <= 1e-4, np.abs(d).max()


def test_full_size_redraw_without_loss_matches_the_oracle(full_case, full_ref):
    """The phase-of-mean redraw the redraw bench times (spectral sum over all 8,937 BF
    pixels, one 2-D inverse transform), at factor 1 and 4, against the oracle's object."""
    _, _, _, ctx = full_case
    theta, ref = full_ref
    for f in (1, 4):
        ph, obj = ctx.redraw(theta, f)
        want = ref["object"] if f == 1 else oracle.upsample_object(ref["object"], f)
        _check_object(obj.cpu().numpy(), want)
        mask = np.abs(want) >= 0.05 * np.sqrt(np.mean(np.abs(want) ** 2))
        assert mask.mean() > 0.5
        d = np.angle(np.exp(1j * (ph.cpu().numpy().astype(np.float64) - np.angle(want))))[mask]
        assert np.abs(d).max() <= 1e-4, (f, np.abs(d).max())
