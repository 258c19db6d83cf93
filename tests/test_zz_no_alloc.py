"""ssb_loss_noalloc, the entry point for callers that cannot allocate device memory
(allocation-free real-time pipelines, plug-ins whose host application owns the GPU
memory): through the C ABI, its loss must match
ssb_loss_batch's on the same G cache within the tests' loss tolerance, on two calls in a
row, and oversized problems must be refused before any device work.

This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest

import ssb_synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

LOSS_RTOL = 1e-5


@pytest.fixture(scope="module")
def ssbgpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from stem_ssb_phase_gb300 import build
    build.build()
    import stem_ssb_phase_gb300 as m
    m.load_library()
    return m


def _geometry_struct(m, geom):
    yx = np.ascontiguousarray(np.asarray(geom.bf_det_yx, dtype=np.float32).reshape(-1, 2))
    g = m._Geometry(int(geom.scan_n), float(geom.scan_step_A), float(geom.wavelength_A),
                    float(geom.semiangle_mrad), float(geom.det_sampling_mrad), int(yx.shape[0]),
                    yx.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    return g, yx


def _noalloc_loss(m, g, gcache, theta):
    out = ctypes.c_double(float("nan"))
    p = m._params([theta])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = m.load_library().ssb_loss_noalloc(ctypes.byref(g), ctypes.c_void_p(gcache.data_ptr()),
                                           p, ctypes.byref(out), stream)
    return st, out.value


def _cases():
    small = ssb_synth.WORKLOADS["small"]
    full = ssb_synth.WORKLOADS["full"]
    sub = np.linspace(0, ssb_synth.make_geometry(full).n_bf - 1, 40).astype(int)
    return [(small, None), (full, sub)]


@pytest.mark.parametrize("case", [0, 1])
def test_noalloc_matches_loss_batch_on_two_calls(ssbgpu, case):
    w, sub = _cases()[case]
    geom = ssb_synth.make_geometry(w, bf_subset=sub)
    _, counts, _ = ssb_synth.simulate_counts_numpy(w, geom=geom)
    ctx = ssbgpu.SSB(geom, counts)
    thetas = np.vstack([np.array(w.truth)[None], ssb_synth.draw_trials(w, 1, seed=77)])
    ref = ctx.loss_batch(thetas)
    gcache = ctx.export_g()
    g, keep = _geometry_struct(ssbgpu, geom)
    for th, lr in zip(thetas, ref):
        first = _noalloc_loss(ssbgpu, g, gcache, th)
        second = _noalloc_loss(ssbgpu, g, gcache, th)
        for st, val in (first, second):
            assert st == 0, ssbgpu.load_library().ssb_last_error()
            assert abs(val - lr) <= LOSS_RTOL * lr, (val, lr)
        assert first[1] == second[1]  # the shared scratch is fully re-initialised
    ctx.close()


def test_noalloc_rejects_problems_beyond_its_scratch(ssbgpu):
    w = ssb_synth.WORKLOADS["small"]
    geom = ssb_synth.make_geometry(w)
    big = np.zeros((20000, 2), np.float32)
    g = ssbgpu._Geometry(geom.scan_n, geom.scan_step_A, geom.wavelength_A, geom.semiangle_mrad,
                         geom.det_sampling_mrad, big.shape[0],
                         big.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    dummy = torch.zeros(16, dtype=torch.complex64, device="cuda")
    st, _ = _noalloc_loss(ssbgpu, g, dummy, w.truth)
    assert st == 1
    assert b"no-allocation" in ssbgpu.load_library().ssb_last_error()
