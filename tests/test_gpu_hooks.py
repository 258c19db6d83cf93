"""Device paths that ordinary inputs do not reach, through the test hooks of
include/ssb_debug.h (C ABI):

* a bounded scheduler wait that runs out: the kernel raises its error word, every wait
  stops, the call returns SSB_ERR_TIMEOUT whichever trial of a batch it happened in, the
  losses from that trial on are NaN, and the GPU keeps answering (nothing traps);
* a batch equals its trials evaluated one by one, bit for bit, although consecutive trials
  run on two streams with their own buffers;
* scratch poisoned with 0xFF bytes (NaN) before a call: every result equals the
  unpoisoned one bit for bit, so nothing the objective reads is left over from an earlier
  call (the pages' phase-only against phase-plus-loss bit-identity check, "SSB performance
  notes", MPS wider exact-simplex checkpoint, made stronger);
* the float32 phase function against float64 atan2 on a dense grid over all quadrants,
  the axes, |y| = |x|, signed zeros and values next to +-pi.
"""
import ctypes
import math

import numpy as np
import pytest

import ssb_synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SSB_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def ssbgpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from stem_ssb_phase_gb300 import build
    build.build()
    import stem_ssb_phase_gb300 as m
    m.load_library()
    return m


def _raw_loss_batch(m, ctx, thetas):
    """ssb_loss_batch through ctypes, returning (status, losses) even on failure."""
    p = m._params(thetas)
    out = (ctypes.c_double * len(p))(*([-1.0] * len(p)))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = m.load_library().ssb_loss_batch(ctx._ctx, p, len(p), out, stream)
    return st, np.frombuffer(out, dtype=np.float64).copy()


# ---------------------------------------------------------------- bounded waits

@pytest.fixture(scope="module")
def tiny_ctx(ssbgpu, tiny_data):
    w, geom, counts, _ = tiny_data
    ctx = ssbgpu.SSB(geom, counts)
    thetas = np.vstack([np.array(w.truth)[None], ssb_synth.draw_trials(w, 5, seed=5)])
    yield ctx, thetas, ctx.loss_batch(thetas)
    ctx.close()


@pytest.mark.parametrize("stalled", [0, 1, 2, 4])
def test_a_wait_that_runs_out_in_any_trial_is_reported(ssbgpu, tiny_ctx, stalled):
    ctx, thetas, ref = tiny_ctx
    ctx.debug_stall_next(stalled, 64)
    st, out = _raw_loss_batch(ssbgpu, ctx, thetas)
    assert st == SSB_ERR_TIMEOUT, ssbgpu.load_library().ssb_last_error()
    assert b"ran out" in ssbgpu.load_library().ssb_last_error()
    # from the stalled trial on the losses are NaN; the trials before it are exact, except
    # that the one just before it overlaps it on the GPU and may have stopped too
    before = max(stalled - 1, 0)
    assert np.array_equal(out[:before], ref[:before])
    if stalled >= 1:
        assert out[stalled - 1] == ref[stalled - 1] or np.isnan(out[stalled - 1])
    assert np.isnan(out[stalled:]).all()
    # the hook is consumed and the GPU still answers: the next call is exact again
    assert np.array_equal(ctx.loss_batch(thetas), ref)


def test_a_timeout_in_one_chunk_of_a_long_batch(ssbgpu, tiny_ctx):
    """ssb_loss_batch evaluates long batches in chunks of 4,096 trials and checks the error
    word after each: a wait that runs out leaves NaN for the rest of its chunk (set by the
    loss kernel) and for the chunks not evaluated after it (set by the host)."""
    ctx, thetas, ref = tiny_ctx
    chunk = 4096
    T = chunk + 5
    big = np.resize(thetas, (T, thetas.shape[1]))
    want = np.resize(ref, T)
    ctx.debug_stall_next(10, 64)  # in the first chunk
    st, out = _raw_loss_batch(ssbgpu, ctx, big)
    assert st == SSB_ERR_TIMEOUT
    assert np.array_equal(out[:9], want[:9])
    assert out[9] == want[9] or np.isnan(out[9])  # overlaps the stalled launch
    assert np.isnan(out[10:]).all()
    ctx.debug_stall_next(chunk + 2, 64)  # in the second chunk
    st, out = _raw_loss_batch(ssbgpu, ctx, big)
    assert st == SSB_ERR_TIMEOUT
    assert np.array_equal(out[:chunk + 1], want[:chunk + 1])
    assert out[chunk + 1] == want[chunk + 1] or np.isnan(out[chunk + 1])
    assert np.isnan(out[chunk + 2:]).all()
    assert np.array_equal(ctx.loss_batch(thetas), ref)


def test_the_hook_is_consumed_by_the_next_call_even_if_it_does_not_reach_it(ssbgpu, tiny_ctx):
    ctx, thetas, ref = tiny_ctx
    ctx.debug_stall_next(len(thetas) - 1, 64)
    # a two-trial call evaluates neither that trial index nor beyond: it succeeds
    assert np.array_equal(ctx.loss_batch(thetas[:2]), ref[:2])
    # and has consumed the hook, so a call that does reach that index is exact too
    st, out = _raw_loss_batch(ssbgpu, ctx, thetas)
    assert st == 0
    assert np.array_equal(out, ref)


def test_a_wait_that_runs_out_in_reconstruct_is_reported(ssbgpu, tiny_ctx):
    ctx, thetas, ref = tiny_ctx
    ctx.debug_stall_next(0, 64)
    with pytest.raises(ssbgpu.SSBError) as ei:
        ctx.reconstruct(thetas[0])
    assert ei.value.status == SSB_ERR_TIMEOUT
    mp, obj, loss = ctx.reconstruct(thetas[0])
    assert loss == ref[0]
    assert torch.isfinite(mp).all() and torch.isfinite(torch.view_as_real(obj)).all()


def test_batch_equals_single_trial_calls(ssbgpu, tiny_ctx):
    ctx, thetas, ref = tiny_ctx
    singles = np.array([ctx.loss(th) for th in thetas])
    assert np.array_equal(singles, ref)
    # odd-length and repeated batches alternate the buffer sets differently
    assert np.array_equal(ctx.loss_batch(thetas[1:]), ref[1:])
    assert np.array_equal(ctx.loss_batch(np.vstack([thetas, thetas])), np.concatenate([ref, ref]))


# ---------------------------------------------------------------- poisoned scratch

def _all_results(ctx, thetas):
    losses = ctx.loss_batch(thetas)
    mp, obj, loss = ctx.reconstruct(thetas[0])
    return losses, mp.cpu().numpy(), obj.cpu().numpy(), loss


@pytest.mark.parametrize("workload", ["tiny", "small"])
@pytest.mark.parametrize("transfer", ["ssb2", "ssb1"])
def test_results_do_not_depend_on_scratch_contents(ssbgpu, workload, transfer):
    w = ssb_synth.WORKLOADS[workload]
    geom, counts, _ = ssb_synth.simulate_counts_numpy(w)
    ctx = ssbgpu.SSB(geom, counts, transfer=transfer)
    thetas = np.vstack([np.array(w.truth)[None], ssb_synth.draw_trials(w, 2, seed=9)])
    clean = _all_results(ctx, thetas)
    ctx.debug_poison_scratch()
    poisoned = _all_results(ctx, thetas)
    ctx.close()
    assert np.array_equal(clean[0], poisoned[0])
    assert np.all(np.isfinite(poisoned[0]))
    assert np.array_equal(clean[1], poisoned[1])
    assert np.array_equal(clean[2], poisoned[2])
    assert clean[3] == poisoned[3]


# ---------------------------------------------------------------- phase function

# Accuracy of the float32 phase function (its polynomial is fitted to atan on [0, 1] by
# iteratively reweighted least squares; float32 Horner error 1.35e-7 rad there).  The
# ratio min/max carries at most 2 ulp of division error (__fdividef), which the slope
# (at most 1) passes on, and the unfolding pi/2 - r, pi - r rounds once more (half an ulp
# of the result, up to 1.2e-7 next to pi), so the whole function stays within
# 1.4e-7 + 2 ulp(a) + ulp(result)/2 <= 4e-7 rad.
ATAN2_BOUND = 4e-7
POLY_BOUND = 1.4e-7


def _phase(ssbgpu, y, x):
    yt = torch.from_numpy(np.ascontiguousarray(y, np.float32)).cuda()
    xt = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    return ssbgpu.debug_atan2(yt, xt).cpu().numpy()


def _err(got, y, x):
    ref = np.arctan2(y.astype(np.float64), x.astype(np.float64))
    d = np.abs(got.astype(np.float64) - ref)
    return np.minimum(d, 2 * np.pi - d)  # +pi and -pi are the same phase


def test_phase_function_on_a_dense_grid(ssbgpu):
    g = np.linspace(-1.0, 1.0, 4096, dtype=np.float32)
    y, x = np.meshgrid(g, g, indexing="ij")
    e = _err(_phase(ssbgpu, y, x), y, x)
    assert e.max() <= ATAN2_BOUND, e.max()
    # the first octant (0 <= y <= x) has no unfolding: the polynomial and the division only
    oct1 = (y >= 0) & (y <= x)
    assert e[oct1].max() <= POLY_BOUND + 2.0 ** -23, e[oct1].max()  # + 2 ulp of a < 1


def test_phase_function_over_magnitudes_and_special_lines(ssbgpu):
    rng = np.random.default_rng(3)
    n = 1 << 20
    ang = rng.uniform(-np.pi, np.pi, n)
    mag = np.exp2(rng.uniform(-60.0, 60.0, n))
    y = (mag * np.sin(ang)).astype(np.float32)
    x = (mag * np.cos(ang)).astype(np.float32)
    t = np.exp2(np.arange(-40, 41, dtype=np.float64)).astype(np.float32)
    one = np.ones_like(t)
    lines_y = np.concatenate([t, -t, t, -t, one * 1e-30, -one * 1e-30, t * 1e-7, -t * 1e-7])
    lines_x = np.concatenate([t, t, -t, -t, -one, -one, -t, -t])  # |y| = |x| and next to +-pi
    y = np.concatenate([y, lines_y])
    x = np.concatenate([x, lines_x])
    e = _err(_phase(ssbgpu, y, x), y, x)
    assert e.max() <= ATAN2_BOUND, e.max()


def test_phase_function_signed_zeros_and_axes(ssbgpu):
    pi32 = float(np.float32(math.pi))
    hp32 = float(np.float32(math.pi / 2))
    y = np.array([0.0, -0.0, 0.0, -0.0, 3.0, -3.0, 3.0, -3.0, 0.0], np.float32)
    x = np.array([2.0, 2.0, -2.0, -2.0, 0.0, 0.0, -0.0, -0.0, 0.0], np.float32)
    got = _phase(ssbgpu, y, x)
    want = [0.0, -0.0, pi32, -pi32, hp32, -hp32, hp32, -hp32, 0.0]
    assert got.tolist() == want
    assert np.signbit(got[1]) and not np.signbit(got[0])  # atan2(-0, +x) = -0
