"""Upsampled object redraw (band-limited interpolation onto a scan grid `factor` times
finer) through the C ABI, against the float64 oracle's object interpolated by
oracle.upsample_object on the same seeded inputs.

Tolerances: the object within 1e-5 relative L2 (two float32 products of length N after
the objective's own float32 path); the phase within 1e-4 rad, compared modulo 2 pi, on
pixels whose modulus is at least 5 % of the object's RMS modulus (the phase of a near-zero
value is not determined by the float32 object); the samples on the original grid equal the
object of ssb_reconstruct within 1e-5 relative L2."""
import numpy as np
import pytest

import oracle
import ssb_synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

OBJ_RTOL = 1e-5
ELEM_RTOL = 1e-4  # element-wise error against the object's largest modulus
PHASE_ATOL = 1e-4


@pytest.fixture(scope="module")
def ssbgpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from stem_ssb_phase_gb300 import build
    build.build()
    import stem_ssb_phase_gb300 as m
    m.load_library()
    return m


def _data(name):
    w = ssb_synth.WORKLOADS[name]
    geom, counts, _ = ssb_synth.simulate_counts_numpy(w)
    return w, geom, counts


@pytest.fixture(scope="module")
def tiny_data():
    return _data("tiny")


@pytest.fixture(scope="module")
def small_data():
    return _data("small")


def _workers():
    return min(16, oracle.default_workers())


def check_upsampled(ph, obj, ref_obj, factor):
    """ph, obj: GPU outputs (numpy); ref_obj: the oracle's N x N object."""
    up = oracle.upsample_object(ref_obj, factor)
    assert obj.shape == up.shape and ph.shape == up.shape
    o = obj.astype(np.complex128)
    rel = np.linalg.norm(o - up) / np.linalg.norm(up)
    assert rel <= OBJ_RTOL, rel
    # element by element, against the largest modulus: a localised error fails here (float32
    # rounding on these DC-dominated objects reaches 1.6e-5 of the largest modulus)
    assert np.abs(o - up).max() <= ELEM_RTOL * np.abs(up).max()
    rms = np.sqrt(np.mean(np.abs(up) ** 2))
    mask = np.abs(up) >= 0.05 * rms
    assert mask.mean() > 0.5
    d = np.angle(np.exp(1j * (ph.astype(np.float64) - np.angle(up))))[mask]
    assert np.abs(d).max() <= PHASE_ATOL, (np.abs(d).max(), int((np.abs(d) > PHASE_ATOL).sum()))
    # the phase output is the argument of the object output, pixel by pixel
    d2 = np.angle(np.exp(1j * (ph.astype(np.float64) - np.angle(o))))
    assert np.abs(d2).max() <= 1e-5


@pytest.mark.parametrize("factor", [1, 2, 3, 4])
@pytest.mark.parametrize("name", ["tiny", "small"])
def test_upsampled_object_matches_the_oracle(ssbgpu, tiny_data, small_data, name, factor):
    w, geom, counts = tiny_data if name == "tiny" else small_data
    ctx = ssbgpu.SSB(geom, counts)
    ph, obj, loss = ctx.reconstruct_upsampled(w.truth, factor)
    ref = oracle.objective(geom, w.truth, counts=counts, want_object=True, workers=_workers())
    assert abs(loss - ref["loss"]) <= 1e-5 * ref["loss"]
    check_upsampled(ph.cpu().numpy(), obj.cpu().numpy(), ref["object"], factor)
    # the original scan positions keep the object of the plain redraw
    _, obj1, loss1 = ctx.reconstruct(w.truth)
    assert loss1 == loss
    o1 = obj1.cpu().numpy().astype(np.complex128)
    sub = obj.cpu().numpy()[::factor, ::factor].astype(np.complex128)
    assert np.linalg.norm(sub - o1) <= 1e-5 * np.linalg.norm(o1)


@pytest.mark.parametrize("factor", [5, 8])
def test_large_factors(ssbgpu, tiny_data, factor):
    """Factors past the pages' 1-4, up to the largest accepted (an odd one and 8)."""
    w, geom, counts = tiny_data
    ctx = ssbgpu.SSB(geom, counts)
    ph, obj, _ = ctx.reconstruct_upsampled(w.truth, factor)
    ref = oracle.objective(geom, w.truth, counts=counts, want_object=True)
    check_upsampled(ph.cpu().numpy(), obj.cpu().numpy(), ref["object"], factor)
    ph2, obj2 = ctx.redraw(w.truth, factor)
    check_upsampled(ph2.cpu().numpy(), obj2.cpu().numpy(), ref["object"], factor)


def test_ssb1_upsampled_object(ssbgpu, small_data):
    w, geom, counts = small_data
    ctx = ssbgpu.SSB(geom, counts, transfer="ssb1")
    ph, obj, _ = ctx.reconstruct_upsampled(w.truth, 2)
    ref = oracle.objective(geom, w.truth, counts=counts, mode="ssb1", want_object=True,
                           workers=_workers())
    check_upsampled(ph.cpu().numpy(), obj.cpu().numpy(), ref["object"], 2)


def test_factor_changes_and_phase_only_output(ssbgpu, tiny_data):
    """Alternating factors reuse or regrow the context's scratch; the phase alone (no
    object, no loss) is the same as with the object."""
    w, geom, counts = tiny_data
    ctx = ssbgpu.SSB(geom, counts)
    first = {f: ctx.reconstruct_upsampled(w.truth, f) for f in (3, 1, 4, 2)}
    for f in (2, 4, 3):
        ph, obj, loss = ctx.reconstruct_upsampled(w.truth, f, want_object=False, want_loss=False)
        assert obj is None and loss is None
        assert torch.equal(ph, first[f][0])


def test_bad_factor_is_rejected(ssbgpu, tiny_data):
    """Out-of-range factors fail on the host with SSB_ERR_ARG before any device work (the
    one-element output buffer is never written)."""
    w, geom, counts = tiny_data
    ctx = ssbgpu.SSB(geom, counts)
    buf = torch.zeros(1, device="cuda")
    for f in (0, -1, 9):
        st = ctx._lib.ssb_reconstruct_upsampled(ctx._ctx, ssbgpu._params([w.truth]), f,
                                                buf.data_ptr(), None, None, None)
        assert st == 1
        assert b"factor" in ctx._lib.ssb_last_error()
    assert float(buf[0]) == 0.0
