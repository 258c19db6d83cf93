"""The C-ABI library builds for sm_103a, loads without a GPU and exports every symbol the
public header declares; the binding rejects bad arguments before reaching a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

import stem_ssb_phase_gb300 as ssbgpu
from stem_ssb_phase_gb300 import build as ssbbuild

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")
HEADER = os.path.join(INCLUDE, "ssb.h")
DEBUG_HEADER = os.path.join(INCLUDE, "ssb_debug.h")


@pytest.fixture(scope="module")
def lib():
    ssbbuild.build()
    return ssbgpu.load_library()


def declared_functions(path=HEADER):
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssb_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert set(declared_functions()) == set(ssbgpu.EXPORTS)
    assert set(declared_functions(DEBUG_HEADER)) == set(ssbgpu.DEBUG_EXPORTS)


def test_every_header_is_covered():
    assert sorted(os.listdir(INCLUDE)) == ["ssb.h", "ssb_debug.h"]


@pytest.mark.parametrize("header", [HEADER, DEBUG_HEADER])
def test_every_declared_symbol_is_exported(lib, header):
    for name in declared_functions(header):
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_test_hooks_reject_bad_arguments_on_the_host(lib):
    assert lib.ssb_debug_stall_next(None, 0, 4) == 1
    assert lib.ssb_debug_poison_scratch(None, None) == 1
    assert lib.ssb_debug_atan2(None, None, 4, None, None) == 1
    assert lib.ssb_debug_atan2(None, None, 0, None, None) == 0  # n = 0 is a no-op


def test_status_strings(lib):
    for code, name in ssbgpu.STATUS.items():
        assert ssbgpu.status_string(code) == name


def test_null_arguments_fail_before_any_device_work(lib):
    out = ctypes.c_void_p()
    assert lib.ssb_prepare(None, None, 0, 0, 0, None, ctypes.byref(out)) == 1
    assert out.value is None
    assert lib.ssb_loss_batch(None, None, 1, None, None) == 1
    assert lib.ssb_reconstruct(None, None, None, None, None, None) == 1
    assert lib.ssb_reconstruct_upsampled(None, None, 2, None, None, None, None) == 1
    assert lib.ssb_redraw(None, None, 1, None, None, None) == 1
    assert lib.ssb_profile_end(None, 0, None) == 1  # no session open
    assert lib.ssb_info(None, None, None) == 1
    assert lib.ssb_export_g(None, None, 0, None) == 1


def test_unsupported_scan_size_is_rejected_on_the_host(lib):
    yx = np.zeros((1, 2), np.float32)
    g = ssbgpu._Geometry(48, 0.25, 0.0197, 20.0, 3.3, 1,
                         yx.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    counts = np.zeros((1, 48, 48), np.uint16)
    out = ctypes.c_void_p()
    st = lib.ssb_prepare(ctypes.byref(g), counts.ctypes.data, 0, 0, 0, None, ctypes.byref(out))
    assert st == 2  # SSB_ERR_UNSUPPORTED
    assert b"scan_n" in lib.ssb_last_error()


@pytest.mark.parametrize("field,value", [("scan_step_A", float("nan")), ("wavelength_A", -1.0),
                                         ("n_bf", 0)])
def test_invalid_geometry_is_rejected(lib, field, value):
    yx = np.zeros((1, 2), np.float32)
    vals = dict(scan_n=32, scan_step_A=0.25, wavelength_A=0.0197, semiangle_mrad=20.0,
                det_sampling_mrad=3.3, n_bf=1)
    vals[field] = value
    g = ssbgpu._Geometry(vals["scan_n"], vals["scan_step_A"], vals["wavelength_A"],
                         vals["semiangle_mrad"], vals["det_sampling_mrad"], vals["n_bf"],
                         yx.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    counts = np.zeros((1, 32, 32), np.uint16)
    out = ctypes.c_void_p()
    assert lib.ssb_prepare(ctypes.byref(g), counts.ctypes.data, 0, 0, 0, None,
                           ctypes.byref(out)) == 1


def test_profiling_session_bookkeeping_on_the_host(lib):
    """A session with no launches needs no device: it opens once per thread, closes with
    an empty report, and a second close is refused."""
    ssbgpu.profile_begin()
    with pytest.raises(ssbgpu.SSBError) as ei:
        ssbgpu.profile_begin()
    assert ei.value.status == 1
    assert lib.ssb_profile_objective(None, None, None, 0, None, None) == 1
    assert ssbgpu.profile_end() == {}
    with pytest.raises(ssbgpu.SSBError) as ei:
        ssbgpu.profile_end()
    assert ei.value.status == 1
