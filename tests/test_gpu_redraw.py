"""Phase-of-mean redraw without the loss (ssb_redraw: spectral sum over the BF pixels and one
2-D inverse transform) through the C ABI, against the float64 oracle's object, the mean
over BF pixels of the per-BF inverse transforms, on the same seeded inputs.

Tolerances: the object within 1e-5 relative L2; the phase arg O within 1e-4 rad, compared
modulo 2 pi, on pixels whose modulus is at least 5 % of the object's RMS modulus; at
factor > 1 the same against the oracle's interpolation of its object."""
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


def check_object(ph, obj, ref):
    """ph, obj: GPU outputs (numpy); ref: the oracle's complex object on the same grid."""
    assert obj.shape == ref.shape and ph.shape == ref.shape
    o = obj.astype(np.complex128)
    rel = np.linalg.norm(o - ref) / np.linalg.norm(ref)
    assert rel <= OBJ_RTOL, rel
    # element by element, against the largest modulus: a localised error fails here (float32
    # rounding on these DC-dominated objects reaches 1.6e-5 of the largest modulus)
    assert np.abs(o - ref).max() <= ELEM_RTOL * np.abs(ref).max()
    mask = np.abs(ref) >= 0.05 * np.sqrt(np.mean(np.abs(ref) ** 2))
    assert mask.mean() > 0.5
    d = np.abs(np.angle(np.exp(1j * (ph.astype(np.float64) - np.angle(ref)))))[mask]
    assert d.max() <= PHASE_ATOL, (d.max(), int((d > PHASE_ATOL).sum()))


@pytest.mark.parametrize("transfer", ["ssb2", "ssb1"])
@pytest.mark.parametrize("name", ["tiny", "small"])
def test_redraw_matches_the_oracle_object(ssbgpu, tiny_data, small_data, name, transfer):
    w, geom, counts = tiny_data if name == "tiny" else small_data
    ctx = ssbgpu.SSB(geom, counts, transfer=transfer)
    th = ssb_synth.draw_trials(w, 1, seed=5)[0]
    ph, obj = ctx.redraw(th)
    ref = oracle.objective(geom, th, counts=counts, mode=transfer, want_object=True,
                           workers=_workers())
    check_object(ph.cpu().numpy(), obj.cpu().numpy(), ref["object"])
    # the same object as the per-BF path of ssb_reconstruct
    _, obj_b, _ = ctx.reconstruct(th)
    a, b = obj.cpu().numpy().astype(np.complex128), obj_b.cpu().numpy().astype(np.complex128)
    assert np.linalg.norm(a - b) <= 1e-5 * np.linalg.norm(b)
    # run to run identical
    ph2, obj2 = ctx.redraw(th)
    assert torch.equal(ph, ph2) and torch.equal(obj, obj2)


@pytest.mark.parametrize("factor", [2, 3])
@pytest.mark.parametrize("transfer", ["ssb2", "ssb1"])
def test_upsampled_redraw_matches_the_oracle(ssbgpu, tiny_data, transfer, factor):
    w, geom, counts = tiny_data
    ctx = ssbgpu.SSB(geom, counts, transfer=transfer)
    ph, obj = ctx.redraw(w.truth, factor)
    ref = oracle.objective(geom, w.truth, counts=counts, mode=transfer, want_object=True)
    check_object(ph.cpu().numpy(), obj.cpu().numpy(), oracle.upsample_object(ref["object"], factor))
    # the phase alone is the same
    ph_only, none = ctx.redraw(w.truth, factor, want_object=False)
    assert none is None and torch.equal(ph_only, ph)


@pytest.mark.parametrize("transfer", ["ssb2", "ssb1"])
@pytest.mark.parametrize("scan_n,det_n,radius,n_sub", [(64, 32, 8.0, None), (256, 96, 27.0, 40),
                                                      (512, 192, 53.3, 24)])
def test_redraw_other_scan_sizes(ssbgpu, scan_n, det_n, radius, n_sub, transfer):
    w = ssb_synth.Workload("edge", scan_n, det_n, radius, "u32", 300.0, 0.2,
                           (-40.0, 12.0, 0.6, 0.2), seed=21, trial_seed=22, n_trials=1)
    sub = None
    if n_sub is not None:
        n_all = ssb_synth.make_geometry(w).n_bf
        sub = np.linspace(0, n_all - 1, n_sub).astype(int)
    geom = ssb_synth.make_geometry(w, bf_subset=sub)
    _, counts, _ = ssb_synth.simulate_counts_numpy(w, geom=geom)
    ctx = ssbgpu.SSB(geom, counts, transfer=transfer)
    th = (-30.0, 10.0, 0.5, 0.2)
    ph, obj = ctx.redraw(th)
    ref = oracle.objective(geom, th, counts=counts, mode=transfer, want_object=True,
                           workers=_workers())
    check_object(ph.cpu().numpy(), obj.cpu().numpy(), ref["object"])


def test_redraw_single_bf_pixel(ssbgpu, tiny_data):
    w, geom, counts = tiny_data
    g1 = ssb_synth.make_geometry(w, bf_subset=np.array([40]))
    ctx = ssbgpu.SSB(g1, counts[40:41])
    th = (30.0, 4.0, 0.3, 0.1)
    ph, obj = ctx.redraw(th)
    ref = oracle.objective(g1, th, counts=counts[40:41], want_object=True)
    check_object(ph.cpu().numpy(), obj.cpu().numpy(), ref["object"])


@pytest.mark.parametrize("transfer", ["ssb2", "ssb1"])
def test_redraw_of_inactive_bf_pixels_is_flat(ssbgpu, tiny_data, transfer):
    """a(alpha_k) = 0 for every BF pixel: only the DC terms survive, the object is the
    constant mean count and its phase is exactly zero."""
    w, geom, counts = tiny_data
    r = np.hypot(geom.bf_det_yx[:, 0], geom.bf_det_yx[:, 1])
    sub = np.nonzero(r >= 2.0)[0]
    g2 = ssb_synth.make_geometry(w, bf_subset=sub)
    g2.semiangle_mrad = 1.0
    ctx = ssbgpu.SSB(g2, counts[sub], transfer=transfer)
    th = (50.0, 3.0, 0.2, 0.1)
    ph, obj = ctx.redraw(th)
    assert float(ph.abs().max()) == 0.0
    ref = oracle.objective(g2, th, counts=counts[sub], mode=transfer, want_object=True)
    o = obj.cpu().numpy().astype(np.complex128)
    assert np.linalg.norm(o - ref["object"]) <= OBJ_RTOL * np.linalg.norm(ref["object"])


def test_profiling_session_times_the_redraw(ssbgpu, tiny_data):
    w, geom, counts = tiny_data
    ctx = ssbgpu.SSB(geom, counts)
    ssbgpu.profile_begin()
    with pytest.raises(ssbgpu.SSBError):
        ssbgpu.profile_begin()  # one session per thread
    ctx.redraw(w.truth, 2)
    prof = ssbgpu.profile_end()
    for k in ("k_redraw_sum", "k_redraw_combine", "k_redraw_fft", "k_up_fwd", "k_up_cols", "k_up_rows"):
        assert k in prof and prof[k][1] > 0.0, (k, prof)
    assert prof["k_redraw_fft"][0] == 2
    with pytest.raises(ssbgpu.SSBError):
        ssbgpu.profile_end()  # no session open


def test_redraw_bad_arguments(ssbgpu, tiny_data):
    w, geom, counts = tiny_data
    ctx = ssbgpu.SSB(geom, counts)
    buf = torch.zeros(1, device="cuda")
    for f in (0, 9):
        st = ctx._lib.ssb_redraw(ctx._ctx, ssbgpu._params([w.truth]), f, buf.data_ptr(), None, None)
        assert st == 1
    st = ctx._lib.ssb_redraw(ctx._ctx, ssbgpu._params([(float("nan"), 0.0, 0.0, 0.0)]), 1,
                             buf.data_ptr(), None, None)
    assert st == 1
    assert float(buf[0]) == 0.0
