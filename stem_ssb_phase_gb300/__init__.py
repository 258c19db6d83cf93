"""Python binding of libssb (SSB phase-variance objective on GB300, sm_103a).

Argument marshalling only: every step of the objective runs in the library's CUDA
kernels.  PyTorch is used for device memory and streams.  There is no CPU fallback:
if libssb.so is missing or cannot be loaded, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssb.so")

SSB_U16, SSB_U32 = 0, 1
TRANSFERS = {"ssb2": 0, "ssb1": 1}
STATUS = {0: "SSB_OK", 1: "SSB_ERR_ARG", 2: "SSB_ERR_UNSUPPORTED", 3: "SSB_ERR_OOM",
          4: "SSB_ERR_CUDA", 5: "SSB_ERR_TIMEOUT", 6: "SSB_ERR_DEVICE_FLAG"}

# every symbol include/ssb.h declares
EXPORTS = ("ssb_prepare", "ssb_loss_batch", "ssb_reconstruct", "ssb_reconstruct_upsampled",
           "ssb_info", "ssb_export_g",
           "ssb_unpack_counts", "ssb_profile_objective", "ssb_profile_begin", "ssb_profile_end",
           "ssb_redraw", "ssb_loss_noalloc", "ssb_status_string",
           "ssb_last_error", "ssb_kernel_launches", "ssb_destroy")
# the test hooks include/ssb_debug.h declares
DEBUG_EXPORTS = ("ssb_debug_stall_next", "ssb_debug_poison_scratch", "ssb_debug_atan2")


class SSBError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__("%s failed: %s (%s)" % (where, STATUS.get(status, status), detail))


class _Geometry(ctypes.Structure):
    _fields_ = [("scan_n", ctypes.c_int), ("scan_step_A", ctypes.c_double),
                ("wavelength_A", ctypes.c_double), ("semiangle_mrad", ctypes.c_double),
                ("det_sampling_mrad", ctypes.c_double), ("n_bf", ctypes.c_int),
                ("bf_det_yx", ctypes.POINTER(ctypes.c_float))]


class _KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int), ("ms", ctypes.c_double)]


class _Params(ctypes.Structure):
    _fields_ = [("C10_nm", ctypes.c_double), ("C12_nm", ctypes.c_double),
                ("phi12_rad", ctypes.c_double), ("rotation_rad", ctypes.c_double)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libssb.so (built by stem_ssb_phase_gb300.build.build()); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError("libssb.so is not built (%s); run stem_ssb_phase_gb300.build.build()" % path)
    lib = ctypes.CDLL(path)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.ssb_prepare.argtypes = [ctypes.POINTER(_Geometry), vp, i, i, i, vp, ctypes.POINTER(vp)]
    lib.ssb_loss_batch.argtypes = [vp, ctypes.POINTER(_Params), i, ctypes.POINTER(ctypes.c_double), vp]
    lib.ssb_reconstruct.argtypes = [vp, ctypes.POINTER(_Params), vp, vp,
                                    ctypes.POINTER(ctypes.c_double), vp]
    lib.ssb_reconstruct_upsampled.argtypes = [vp, ctypes.POINTER(_Params), i, vp, vp,
                                              ctypes.POINTER(ctypes.c_double), vp]
    lib.ssb_info.argtypes = [vp, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    lib.ssb_export_g.argtypes = [vp, vp, i, vp]
    lib.ssb_unpack_counts.argtypes = [vp, i, sz, vp, vp]
    lib.ssb_profile_objective.argtypes = [vp, ctypes.POINTER(_Params), ctypes.POINTER(_KernelTime),
                                          i, ctypes.POINTER(i), vp]
    lib.ssb_profile_begin.argtypes = []
    lib.ssb_profile_end.argtypes = [ctypes.POINTER(_KernelTime), i, ctypes.POINTER(i)]
    lib.ssb_redraw.argtypes = [vp, ctypes.POINTER(_Params), i, vp, vp, vp]
    lib.ssb_loss_noalloc.argtypes = [ctypes.POINTER(_Geometry), vp, ctypes.POINTER(_Params),
                                     ctypes.POINTER(ctypes.c_double), vp]
    lib.ssb_status_string.argtypes = [i]
    lib.ssb_status_string.restype = ctypes.c_char_p
    lib.ssb_last_error.argtypes = []
    lib.ssb_last_error.restype = ctypes.c_char_p
    lib.ssb_kernel_launches.argtypes = []
    lib.ssb_kernel_launches.restype = ctypes.c_uint64
    lib.ssb_destroy.argtypes = [vp]
    lib.ssb_destroy.restype = None
    lib.ssb_debug_stall_next.argtypes = [vp, i, ctypes.c_uint]
    lib.ssb_debug_poison_scratch.argtypes = [vp, vp]
    lib.ssb_debug_atan2.argtypes = [vp, vp, sz, vp, vp]
    for name in ("ssb_prepare", "ssb_loss_batch", "ssb_reconstruct", "ssb_reconstruct_upsampled", "ssb_info",
                 "ssb_export_g", "ssb_unpack_counts", "ssb_profile_objective",
                 "ssb_profile_begin", "ssb_profile_end", "ssb_redraw", "ssb_loss_noalloc") + DEBUG_EXPORTS:
        getattr(lib, name).restype = i
    _lib = lib
    return lib


def _check(st: int, where: str):
    if st != 0:
        raise SSBError(st, where, load_library().ssb_last_error().decode())


def _stream_handle(stream) -> ctypes.c_void_p:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _params(thetas) -> ctypes.Array:
    th = np.asarray(thetas, dtype=np.float64).reshape(-1, 4)
    arr = (_Params * len(th))()
    for j, t in enumerate(th):
        arr[j] = _Params(*map(float, t))
    return arr


def kernel_launches() -> int:
    return int(load_library().ssb_kernel_launches())


class SSB:
    """A prepared dataset: the G cache of one 4D-STEM acquisition on the current GPU.

    geometry: an object with scan_n, scan_step_A, wavelength_A, semiangle_mrad,
              det_sampling_mrad and bf_det_yx ([n_bf][2] float32), e.g.
              ssb_synth.Geometry.
    counts:   [n_bf][N][N] counts, either a numpy uint16/uint32 array (host) or a CUDA
              torch tensor (uint16/int16 as uint16 bits, uint32/int32 as uint32 bits).
    transfer: "ssb2" (two-sideband transfer, default) or "ssb1".
    """

    def __init__(self, geometry, counts, transfer: str = "ssb2", stream=None):
        import torch
        lib = load_library()
        self._lib = lib
        self._ctx = ctypes.c_void_p()
        yx = np.ascontiguousarray(np.asarray(geometry.bf_det_yx, dtype=np.float32).reshape(-1, 2))
        self.n_bf = int(yx.shape[0])
        self.N = int(geometry.scan_n)
        self._yx = yx
        g = _Geometry(self.N, float(geometry.scan_step_A), float(geometry.wavelength_A),
                      float(geometry.semiangle_mrad), float(geometry.det_sampling_mrad), self.n_bf,
                      yx.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
        if isinstance(counts, torch.Tensor):
            if not counts.is_cuda:
                counts = counts.cpu().numpy()
        if isinstance(counts, np.ndarray):
            if counts.dtype == np.uint16:
                dt = SSB_U16
            elif counts.dtype == np.uint32:
                dt = SSB_U32
            else:
                raise TypeError("counts must be uint16 or uint32, got %s" % counts.dtype)
            if counts.shape != (self.n_bf, self.N, self.N):
                raise ValueError("counts shape %s != (%d, %d, %d)" % (counts.shape, self.n_bf, self.N, self.N))
            host = np.ascontiguousarray(counts)
            ptr, on_dev = host.ctypes.data, 0
            keep = host
        else:
            if counts.element_size() == 2:
                dt = SSB_U16
            elif counts.element_size() == 4 and not counts.is_floating_point():
                dt = SSB_U32
            else:
                raise TypeError("device counts must be a 16- or 32-bit integer tensor")
            if tuple(counts.shape) != (self.n_bf, self.N, self.N):
                raise ValueError("counts shape mismatch")
            keep = counts.contiguous()
            ptr, on_dev = keep.data_ptr(), 1
        st = lib.ssb_prepare(ctypes.byref(g), ctypes.c_void_p(ptr), dt, on_dev,
                             TRANSFERS[transfer], _stream_handle(stream), ctypes.byref(self._ctx))
        del keep
        _check(st, "ssb_prepare")

    # ------------------------------------------------------------------ queries
    def info(self):
        gb, sb = ctypes.c_size_t(), ctypes.c_size_t()
        _check(self._lib.ssb_info(self._ctx, ctypes.byref(gb), ctypes.byref(sb)), "ssb_info")
        return int(gb.value), int(sb.value)

    # ------------------------------------------------------------------ objective
    def loss_batch(self, thetas: Sequence, stream=None) -> np.ndarray:
        """Losses (float64) for a [T][4] array of (C10 nm, |C12| nm, phi12 rad, rotation rad)."""
        p = _params(thetas)
        out = (ctypes.c_double * len(p))()
        _check(self._lib.ssb_loss_batch(self._ctx, p, len(p), out, _stream_handle(stream)),
               "ssb_loss_batch")
        return np.frombuffer(out, dtype=np.float64).copy()

    def loss(self, theta, stream=None) -> float:
        return float(self.loss_batch([theta], stream=stream)[0])

    def reconstruct(self, theta, want_object: bool = True, want_loss: bool = True, stream=None):
        """(mean phase [N][N] float32, object [N][N] complex64 or None, loss or None)."""
        import torch
        mp = torch.empty((self.N, self.N), dtype=torch.float32, device="cuda")
        obj = torch.empty((self.N, self.N), dtype=torch.complex64, device="cuda") if want_object else None
        loss = ctypes.c_double(float("nan"))
        p = _params([theta])
        _check(self._lib.ssb_reconstruct(self._ctx, p, ctypes.c_void_p(mp.data_ptr()),
                                         ctypes.c_void_p(obj.data_ptr()) if obj is not None else None,
                                         ctypes.byref(loss) if want_loss else None,
                                         _stream_handle(stream)), "ssb_reconstruct")
        return mp, obj, (float(loss.value) if want_loss else None)

    def reconstruct_upsampled(self, theta, factor: int, want_object: bool = True,
                              want_loss: bool = True, stream=None):
        """(phase [fN][fN] float32, object [fN][fN] complex64 or None, loss or None) of the
        object redrawn band-limited on a scan grid `factor` times finer."""
        import torch
        fn = int(factor) * self.N
        ph = torch.empty((fn, fn), dtype=torch.float32, device="cuda")
        obj = torch.empty((fn, fn), dtype=torch.complex64, device="cuda") if want_object else None
        loss = ctypes.c_double(float("nan"))
        p = _params([theta])
        _check(self._lib.ssb_reconstruct_upsampled(
            self._ctx, p, int(factor), ctypes.c_void_p(ph.data_ptr()),
            ctypes.c_void_p(obj.data_ptr()) if obj is not None else None,
            ctypes.byref(loss) if want_loss else None, _stream_handle(stream)),
            "ssb_reconstruct_upsampled")
        return ph, obj, (float(loss.value) if want_loss else None)

    def profile(self, theta, stream=None) -> dict:
        """{kernel name: (launches, total device ms)} for one objective at theta."""
        cap = 64
        out = (_KernelTime * cap)()
        n = ctypes.c_int(0)
        _check(self._lib.ssb_profile_objective(self._ctx, _params([theta]), out, cap,
                                               ctypes.byref(n), _stream_handle(stream)),
               "ssb_profile_objective")
        return {out[j].name.decode(): (int(out[j].launches), float(out[j].ms))
                for j in range(min(cap, n.value))}

    def redraw(self, theta, factor: int = 1, want_object: bool = True, stream=None):
        """(phase arg O [fN][fN] float32, object O [fN][fN] complex64 or None): the
        phase-of-mean redraw from the spectral sum, without the loss."""
        import torch
        fn = int(factor) * self.N
        ph = torch.empty((fn, fn), dtype=torch.float32, device="cuda")
        obj = torch.empty((fn, fn), dtype=torch.complex64, device="cuda") if want_object else None
        p = _params([theta])
        _check(self._lib.ssb_redraw(self._ctx, p, int(factor), ctypes.c_void_p(ph.data_ptr()),
                                    ctypes.c_void_p(obj.data_ptr()) if obj is not None else None,
                                    _stream_handle(stream)), "ssb_redraw")
        return ph, obj

    # ------------------------------------------------------------------ test hooks
    def debug_stall_next(self, evaluation: int, polls: int):
        """Make evaluation `evaluation` of the next objective call stall its row tasks on a
        count nothing reaches, giving up after `polls` polls (ssb_debug.h)."""
        _check(self._lib.ssb_debug_stall_next(self._ctx, int(evaluation), int(polls)),
               "ssb_debug_stall_next")

    def debug_poison_scratch(self, stream=None):
        """Fill every per-evaluation scratch buffer with 0xFF bytes (NaN) (ssb_debug.h)."""
        _check(self._lib.ssb_debug_poison_scratch(self._ctx, _stream_handle(stream)),
               "ssb_debug_poison_scratch")

    def export_g(self, stream=None):
        """The G cache as a CUDA complex64 tensor [n_bf][N/2+1][N] (Qx-major, Qy contiguous)."""
        import torch
        out = torch.empty((self.n_bf, self.N // 2 + 1, self.N), dtype=torch.complex64, device="cuda")
        _check(self._lib.ssb_export_g(self._ctx, ctypes.c_void_p(out.data_ptr()), 1,
                                      _stream_handle(stream)), "ssb_export_g")
        return out

    def close(self):
        if getattr(self, "_ctx", None) is not None and self._ctx.value:
            self._lib.ssb_destroy(self._ctx)
            self._ctx = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def profile_begin():
    """Start timing every library launch this thread makes (see profile_end)."""
    _check(load_library().ssb_profile_begin(), "ssb_profile_begin")


def profile_end() -> dict:
    """{kernel name: (launches, total device ms)} since profile_begin on this thread."""
    lib = load_library()
    cap = 64
    out = (_KernelTime * cap)()
    n = ctypes.c_int(0)
    _check(lib.ssb_profile_end(out, cap, ctypes.byref(n)), "ssb_profile_end")
    return {out[j].name.decode(): (int(out[j].launches), float(out[j].ms))
            for j in range(min(cap, n.value))}


def unpack_counts(counts, stream=None):
    """float32 copy of a CUDA integer count tensor through the library's unpack kernel."""
    import torch
    lib = load_library()
    if counts.element_size() == 2:
        dt = SSB_U16
    elif counts.element_size() == 4 and not counts.is_floating_point():
        dt = SSB_U32
    else:
        raise TypeError("counts must be a 16- or 32-bit integer CUDA tensor")
    src = counts.contiguous()
    out = torch.empty(src.shape, dtype=torch.float32, device=src.device)
    _check(lib.ssb_unpack_counts(ctypes.c_void_p(src.data_ptr()), dt, src.numel(),
                                 ctypes.c_void_p(out.data_ptr()), _stream_handle(stream)),
           "ssb_unpack_counts")
    return out


def debug_atan2(y, x, stream=None):
    """The objective's float32 phase function atan2(y, x) on CUDA float32 tensors."""
    import torch
    yc, xc = y.contiguous(), x.contiguous()
    if yc.dtype != torch.float32 or xc.dtype != torch.float32 or yc.shape != xc.shape:
        raise TypeError("y and x must be float32 CUDA tensors of one shape")
    out = torch.empty_like(yc)
    _check(load_library().ssb_debug_atan2(ctypes.c_void_p(yc.data_ptr()), ctypes.c_void_p(xc.data_ptr()),
                                          yc.numel(), ctypes.c_void_p(out.data_ptr()),
                                          _stream_handle(stream)), "ssb_debug_atan2")
    return out


def status_string(code: int) -> str:
    return load_library().ssb_status_string(code).decode()
