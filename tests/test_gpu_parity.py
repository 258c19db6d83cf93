"""GPU path (through the C ABI) against the float64 oracle on the same seeded inputs.

Tolerances (stated for the objective): loss within 1e-5 relative; mean phase within
1e-4 rad on pixels where no BF phase lies within 1e-4 of +-pi (atan2 branch cut); the
float32 counts bit-exact; the G cache within a float32 FFT bound (relative L2 2e-6)."""
import math

import numpy as np
import pytest

import oracle
import ssb_synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

LOSS_RTOL = 1e-5
PHASE_ATOL = 1e-4
OBJ_RTOL = 1e-5
ELEM_RTOL = 1e-4  # element-wise error against the object's largest modulus


@pytest.fixture(scope="module")
def ssbgpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from stem_ssb_phase_gb300 import build
    build.build()
    import stem_ssb_phase_gb300 as m
    m.load_library()
    return m


def _workers():
    return min(16, oracle.default_workers())


@pytest.fixture(scope="module")
def small_data():
    w = ssb_synth.WORKLOADS["small"]
    geom, counts, phi = ssb_synth.simulate_counts_numpy(w)
    return w, geom, counts, phi


def _check_object(gpu_obj, want, tol=OBJ_RTOL, elem=ELEM_RTOL):
    """Object redraw: relative L2 error and, element by element, the error against the
    object's largest modulus (a localised error in a few pixels fails the second; float32
    rounding on these DC-dominated objects reaches 1.6e-5 of the largest modulus)."""
    o = gpu_obj.astype(np.complex128)
    scale = np.abs(want).max()
    assert np.linalg.norm(o - want) <= tol * np.linalg.norm(want)
    err = np.abs(o - want)
    assert err.max() <= elem * scale, (err.max() / scale, np.unravel_index(int(err.argmax()), err.shape))


def _check_phase(gpu_mp, ref, tol=PHASE_ATOL):
    mask = ~ref["branch_cut"]
    err = np.abs(gpu_mp.astype(np.float64) - ref["mean_phase"])[mask]
    assert mask.mean() > 0.9
    assert err.max() <= tol, (err.max(), int((err > tol).sum()))


# ---------------------------------------------------------------- unpack and G cache

def test_unpack_counts_bit_exact(ssbgpu):
    rng = np.random.default_rng(0)
    u16 = rng.integers(0, 65536, size=(3, 64, 64), dtype=np.uint16)
    t16 = torch.from_numpy(u16.view(np.int16)).cuda()
    out = ssbgpu.unpack_counts(t16).cpu().numpy()
    assert np.array_equal(out, u16.astype(np.float32))
    u32 = rng.integers(0, 2 ** 24 + 1, size=(2, 64, 64), dtype=np.uint32)
    u32.flat[:3] = [0, 2 ** 24, 2 ** 24 - 1]
    t32 = torch.from_numpy(u32.view(np.int32)).cuda()
    out = ssbgpu.unpack_counts(t32).cpu().numpy()
    assert np.array_equal(out.astype(np.uint32), u32)
    assert np.array_equal(out, u32.astype(np.float32))


def test_unpack_rejects_counts_beyond_float32_exact_range(ssbgpu):
    bad = torch.tensor([1, 2 ** 24 + 1, 3], dtype=torch.int32, device="cuda")
    with pytest.raises(ssbgpu.SSBError) as ei:
        ssbgpu.unpack_counts(bad)
    assert ei.value.status == 1


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_g_cache_matches_oracle(ssbgpu, name, tiny_data, small_data):
    w, geom, counts, _ = tiny_data if name == "tiny" else small_data
    ctx = ssbgpu.SSB(geom, counts)
    g = ctx.export_g().cpu().numpy()  # [k][Qx][Qy]
    ks = range(geom.n_bf) if name == "tiny" else range(0, geom.n_bf, 37)
    for k in ks:
        ref = oracle.g_plane(counts[k]).T  # -> [Qx][Qy]
        rel = np.linalg.norm(g[k] - ref) / np.linalg.norm(ref)
        assert rel < 2e-6, (k, rel)
    gb, sb = ctx.info()
    assert gb == geom.n_bf * (w.scan_n // 2 + 1) * w.scan_n * 8
    ctx.close()


def test_device_counts_give_the_same_cache(ssbgpu, tiny_data):
    _, geom, counts, _ = tiny_data
    a = ssbgpu.SSB(geom, counts).export_g()
    b = ssbgpu.SSB(geom, torch.from_numpy(counts.view(np.int16)).cuda()).export_g()
    assert torch.equal(a, b)


# ---------------------------------------------------------------- loss / phase / object

@pytest.mark.parametrize("transfer", ["ssb2", "ssb1"])
def test_tiny_objective(ssbgpu, tiny_data, transfer):
    w, geom, counts, _ = tiny_data
    ctx = ssbgpu.SSB(geom, counts, transfer=transfer)
    thetas = np.vstack([np.array(w.truth)[None], ssb_synth.draw_trials(w, 5, seed=5)])
    gpu = ctx.loss_batch(thetas)
    for th, lg in zip(thetas, gpu):
        ref = oracle.objective(geom, th, counts=counts, mode=transfer)
        assert abs(lg - ref["loss"]) <= LOSS_RTOL * ref["loss"], (th, lg, ref["loss"])
    mp, obj, loss = ctx.reconstruct(w.truth)
    ref = oracle.objective(geom, w.truth, counts=counts, mode=transfer, want_object=True)
    _check_phase(mp.cpu().numpy(), ref)
    _check_object(obj.cpu().numpy(), ref["object"])
    assert abs(loss - ref["loss"]) <= LOSS_RTOL * ref["loss"]


@pytest.mark.parametrize("transfer", ["ssb2", "ssb1"])
def test_small_batch_of_trials(ssbgpu, small_data, transfer):
    w, geom, counts, _ = small_data
    ctx = ssbgpu.SSB(geom, counts, transfer=transfer)
    thetas = ssb_synth.draw_trials(w, w.n_trials)
    gpu = ctx.loss_batch(thetas)
    for th, lg in zip(thetas[:4], gpu[:4]):
        ref = oracle.objective(geom, th, counts=counts, mode=transfer, workers=_workers())
        assert abs(lg - ref["loss"]) <= LOSS_RTOL * ref["loss"], (th, lg, ref["loss"])
    # batch entries equal single-trial calls bit for bit
    singles = np.array([ctx.loss(th) for th in thetas])
    assert np.array_equal(singles, gpu)
    # and repeated calls are deterministic
    assert np.array_equal(ctx.loss_batch(thetas), gpu)


@pytest.mark.parametrize("transfer", ["ssb2", "ssb1"])
def test_small_truth_phase_and_object(ssbgpu, small_data, transfer):
    w, geom, counts, _ = small_data
    ctx = ssbgpu.SSB(geom, counts, transfer=transfer)
    mp, obj, loss = ctx.reconstruct(w.truth)
    ref = oracle.objective(geom, w.truth, counts=counts, mode=transfer, want_object=True,
                           workers=_workers())
    assert abs(loss - ref["loss"]) <= LOSS_RTOL * ref["loss"]
    _check_phase(mp.cpu().numpy(), ref)
    _check_object(obj.cpu().numpy(), ref["object"])


@pytest.fixture(scope="module")
def medium_data():
    w = ssb_synth.WORKLOADS["medium"]
    geom, counts, _ = ssb_synth.simulate_counts_numpy(w)
    return w, geom, counts


@pytest.mark.slow
@pytest.mark.parametrize("transfer", ["ssb2", "ssb1"])
def test_medium_objective(ssbgpu, medium_data, transfer):
    w, geom, counts = medium_data
    ctx = ssbgpu.SSB(geom, counts, transfer=transfer)
    thetas = np.vstack([np.array(w.truth)[None], ssb_synth.draw_trials(w, w.n_trials)])
    gpu = ctx.loss_batch(thetas)
    assert np.all(np.isfinite(gpu))
    # the truth, the first trials and trials spread over the batch (both buffer sets)
    for j in (0, 1, 2, 67, 134, 200):
        ref = oracle.objective(geom, thetas[j], counts=counts, mode=transfer, workers=_workers())
        assert abs(gpu[j] - ref["loss"]) <= LOSS_RTOL * ref["loss"], (j, gpu[j], ref["loss"])
    # object redraw at the best trial
    best = thetas[int(np.argmin(gpu))]
    mp, obj, loss = ctx.reconstruct(best)
    assert loss == gpu[int(np.argmin(gpu))]
    ref = oracle.objective(geom, best, counts=counts, mode=transfer, want_object=True,
                           workers=_workers())
    _check_phase(mp.cpu().numpy(), ref)
    _check_object(obj.cpu().numpy(), ref["object"])


# ---------------------------------------------------------------- edge cases

def test_single_bf_pixel(ssbgpu, tiny_data):
    w, geom, counts, _ = tiny_data
    g1 = ssb_synth.make_geometry(w, bf_subset=np.array([40]))
    ctx = ssbgpu.SSB(g1, counts[40:41])
    th = (30.0, 4.0, 0.3, 0.1)
    ref = oracle.objective(g1, th, counts=counts[40:41])
    # one BF term: zero variance; the float32 phi^2 against the float64 S1^2 leaves a
    # rounding-level residue, bounded relative to the second moment of the phase
    assert ref["loss"] == 0.0
    assert abs(ctx.loss(th)) <= 1e-6 * float(np.mean(ref["s2"]))
    mp, _, _ = ctx.reconstruct(th, want_object=False)
    refp = oracle.objective(g1, th, counts=counts[40:41])
    _check_phase(mp.cpu().numpy(), refp)


@pytest.mark.parametrize("transfer", ["ssb2", "ssb1"])
def test_inactive_bf_pixels_give_zero_phase(ssbgpu, tiny_data, transfer):
    w, geom, counts, _ = tiny_data
    # BF pixels at least 2 px off axis with a 1 mrad probe aperture: a(alpha_k) = 0
    r = np.hypot(geom.bf_det_yx[:, 0], geom.bf_det_yx[:, 1])
    sub = np.nonzero(r >= 2.0)[0]
    g2 = ssb_synth.make_geometry(w, bf_subset=sub)
    g2.semiangle_mrad = 1.0
    ctx = ssbgpu.SSB(g2, counts[sub], transfer=transfer)
    th = (50.0, 3.0, 0.2, 0.1)
    assert oracle.objective(g2, th, counts=counts[sub], mode=transfer)["loss"] == 0.0
    assert ctx.loss(th) == 0.0
    mp, _, _ = ctx.reconstruct(th, want_object=False)
    assert float(mp.abs().max()) == 0.0
    # mixed: the inactive pixels stay in the normalisation
    g3 = ssb_synth.make_geometry(w)
    g3.semiangle_mrad = 4.0
    ctx3 = ssbgpu.SSB(g3, counts, transfer=transfer)
    ref = oracle.objective(g3, th, counts=counts, mode=transfer)
    assert abs(ctx3.loss(th) - ref["loss"]) <= LOSS_RTOL * ref["loss"]


@pytest.mark.parametrize("transfer", ["ssb2", "ssb1"])
@pytest.mark.parametrize("scan_n,det_n,radius,n_sub", [(64, 32, 8.0, None), (512, 192, 53.3, 24),
                                                      (256, 96, 27.0, 40)])
def test_other_scan_sizes(ssbgpu, scan_n, det_n, radius, n_sub, transfer):
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
    ref = oracle.objective(geom, th, counts=counts, mode=transfer, workers=_workers())
    assert abs(ctx.loss(th) - ref["loss"]) <= LOSS_RTOL * ref["loss"]
    mp, _, _ = ctx.reconstruct(th, want_object=False)
    _check_phase(mp.cpu().numpy(), ref)


def test_bad_arguments_raise(ssbgpu, tiny_data):
    _, geom, counts, _ = tiny_data
    ctx = ssbgpu.SSB(geom, counts)
    with pytest.raises(ssbgpu.SSBError) as ei:
        ctx.loss((float("nan"), 0.0, 0.0, 0.0))
    assert ei.value.status == 1
    bad = counts.astype(np.uint32)
    bad[0, 0, 0] = 2 ** 24 + 5
    with pytest.raises(ssbgpu.SSBError) as ei:
        ssbgpu.SSB(geom, bad)
    assert ei.value.status == 1
