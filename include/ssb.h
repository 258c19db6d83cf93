/*
 * ssb.h -- C ABI of the GB300 (sm_103a) single-sideband (SSB) phase-variance library.
 *
 * The library evaluates, on one GPU, the exact SSB phase-variance objective used to fit
 * probe aberrations in 4D-STEM, and batches of it over trial aberrations.  The objective
 * and its measured workloads are the subject of the quantem.gpu pages "Later SSB
 * performance checkpoints" (section "2026-09-11 full-aperture Apple M5 floor checkpoint":
 * all 8,937 BF terms, 512x512 scan, packed counts, "one exact phase-variance evaluation")
 * and "SSB performance notes" (Hermitian G_qk evidence, gamma correction, zero transfer,
 * ordered phase / phase^2 reductions, object redraw).
 *
 * For BF detector pixel k with detector angle alpha_k and scan frequency Q (fftfreq grid,
 * rotated Q' = R_theta Q):
 *   G_k(Q)     = rfft2 over the scan of the counts of pixel k         (ssb_prepare)
 *   A(alpha)   = a(alpha) exp(i chi(alpha))
 *   Gamma_k(Q) = conj(A(alpha_k)) A(alpha_k - lambda Q') - A(alpha_k) conj(A(alpha_k + lambda Q'))
 *   C_k(Q)     = G_k(Q) conj(Gamma_k)/|Gamma_k|  (0 where Gamma_k = 0),  C_k(0) = G_k(0)
 *   c_k(r)     = IFFT2[C_k](r),  phi_k(r) = atan2(Im c_k, Re c_k)
 *   loss       = (1/P) sum_r [ S2(r)/n_bf - (S1(r)/n_bf)^2 ],  S1 = sum_k phi_k, S2 = sum_k phi_k^2
 *   chi(alpha) = (pi/lambda) [C10 |alpha|^2 + C12 ((ax^2 - ay^2) cos 2phi12 + 2 ax ay sin 2phi12)]
 *   a(alpha)   = clip((alpha_c - |alpha|)/d_alpha + 1/2, 0, 1), taken as 0 below 2^-16
 *                (an aperture edge that a scan grid commensurate with the detector hits
 *                exactly transmits nothing, whatever the rounding)
 * C10, C12 in nm; angles in rad; lambda and the scan step in Angstrom.
 *
 * Conventions for every entry point:
 *   - Status codes only; no exception crosses the ABI and no kernel traps.
 *   - "host" pointers are ordinary CPU memory; "device" pointers are CUDA global memory
 *     of the current device.  The caller owns every buffer it passes.
 *   - cuda_stream is a cudaStream_t (NULL = the legacy default stream).  Work is ordered
 *     on that stream; entry points that return host results synchronise it first.
 *   - A context is bound to the device that was current at ssb_prepare, owns its G cache
 *     and scratch, is used by one stream at a time and is not thread-safe.
 */
#ifndef SSB_H
#define SSB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ssb_ctx ssb_ctx;

/* Acquisition geometry.  bf_det_yx is host memory, [n_bf][2] float32 (dy, dx) detector
 * pixel offsets from the optical axis, in row-major detector order; it is copied. */
typedef struct {
    int          scan_n;            /* N: 32, 64, 128, 256 or 512 (square N x N scan)  */
    double       scan_step_A;       /* scan step (Angstrom), > 0                        */
    double       wavelength_A;      /* electron wavelength (Angstrom), > 0              */
    double       semiangle_mrad;    /* probe aperture semiangle alpha_c, > 0            */
    double       det_sampling_mrad; /* detector angular sampling d_alpha (mrad/px) > 0  */
    int          n_bf;              /* number of BF pixels, >= 1                        */
    const float *bf_det_yx;         /* host [n_bf][2]                                   */
} ssb_geometry;

/* One trial aberration set theta. */
typedef struct {
    double C10_nm;       /* defocus                                   */
    double C12_nm;       /* twofold astigmatism magnitude |C12|       */
    double phi12_rad;    /* astigmatism azimuth                        */
    double rotation_rad; /* scan rotation: Q'x = cos Qx - sin Qy, Q'y = sin Qx + cos Qy */
} ssb_params;

typedef enum {
    SSB_OK = 0,
    SSB_ERR_ARG = 1,          /* invalid argument (null pointer, size, non-finite value) */
    SSB_ERR_UNSUPPORTED = 2,  /* valid but unsupported (scan size, device)               */
    SSB_ERR_OOM = 3,          /* device allocation failed                                */
    SSB_ERR_CUDA = 4,         /* a CUDA runtime call failed (see ssb_last_error)         */
    SSB_ERR_TIMEOUT = 5,      /* a bounded device wait ran out                           */
    SSB_ERR_DEVICE_FLAG = 6   /* a kernel raised its error flag (see ssb_last_error)     */
} ssb_status;

typedef enum { SSB_U16 = 0, SSB_U32 = 1 } ssb_dtype;

/* Reading of the correction.  SSB2 (default) is Gamma above, normalised to unit modulus.
 * SSB1 is the single-sideband factor exp(i(chi(alpha_k) - chi(alpha_k - lambda Q')))
 * masked by a(alpha_k) a(alpha_k - lambda Q') > 0 (the aberration factor as first stated
 * for this objective); both keep C_k(0) = G_k(0). */
typedef enum { SSB_TRANSFER_SSB2 = 0, SSB_TRANSFER_SSB1 = 1 } ssb_transfer;

/* Build the scan-Fourier G cache from packed integer counts (page "SSB performance notes",
 * BF-major G_qk; page "Later SSB performance checkpoints": packed uint32 counts).
 *   counts: [n_bf][N][N] uint16 or uint32 (dtype), row-major, host or device memory
 *           (counts_on_device = 0 / 1).  Read during the call only, not retained.
 *           Every count must be <= 2^24 so that the float32 conversion is exact;
 *           larger counts fail with SSB_ERR_ARG.
 *   out:    receives a new context on success (NULL on failure).
 * G is stored complex64 [n_bf][N/2+1][N]: half-plane column Qx, then Qy contiguous. */
ssb_status ssb_prepare(const ssb_geometry *g, const void *counts, ssb_dtype dtype,
                       int counts_on_device, ssb_transfer transfer, void *cuda_stream,
                       ssb_ctx **out);

/* Exact objective for T trials (page "SSB performance notes", multi-candidate
 * evaluation: each trial keeps its own correction, FFTs, phase and loss).  Here each
 * trial is one launch of the persistent kernel, which reads the G cache once; the G read
 * is not what bounds the kernel, so trials do not share it.  Consecutive trials alternate
 * between cuda_stream and a second stream of the context (each with its own buffers), so
 * that one launch's last tasks overlap the next launch's start; the call is still ordered
 * after earlier work on cuda_stream, and later work on cuda_stream after it.  theta: host
 * [T]; loss_out: host [T] (float64).  T >= 1.  Each entry equals the loss of a
 * single-trial call with the same theta, bit for bit; the transfer is the context's.
 * SSB_ERR_TIMEOUT: a bounded wait of the kernel ran out; the losses of that trial and of
 * every later one are NaN, and so may be the loss of the trial that overlapped it. */
ssb_status ssb_loss_batch(ssb_ctx *c, const ssb_params *theta, int T, double *loss_out,
                          void *cuda_stream);

/* Mean phase and object redraw at one theta (page "Later SSB performance checkpoints":
 * "object redraw"; page "SSB performance notes": phase-of-mean output).
 *   mean_phase_out: device [N][N] float32, S1/n_bf            (required)
 *   object_c64_out: device [N][N] complex64 interleaved, (1/n_bf) sum_k c_k   (nullable)
 *   loss_out:       host, one float64                          (nullable)
 * SSB_ERR_TIMEOUT as for ssb_loss_batch (the outputs are then unspecified). */
ssb_status ssb_reconstruct(ssb_ctx *c, const ssb_params *theta, float *mean_phase_out,
                           float *object_c64_out, double *loss_out, void *cuda_stream);

/* Largest factor ssb_reconstruct_upsampled accepts. */
#define SSB_MAX_UPSAMPLE 8

/* Object redraw on a scan grid `factor` times finer (page "Later SSB performance
 * checkpoints", joint CUDA calibration: reconstruction with an upsampling factor of 1 to 4).
 * The BF-summed object of ssb_reconstruct is interpolated band-limited: its N x N discrete
 * spectrum is kept at the signed frequencies -N/2 .. N/2-1 of the (factor N)^2 grid, every
 * other frequency is zero, and the grid's inverse transform is scaled by factor^2 so that
 * the original samples are kept (O_up[factor m][factor n] = O[m][n]).
 *   factor:         1 .. SSB_MAX_UPSAMPLE (1 gives the object of ssb_reconstruct)
 *   phase_out:      device [factor N][factor N] float32, arg of the object  (required)
 *   object_c64_out: device [factor N][factor N] complex64 interleaved        (nullable)
 *   loss_out:       host, one float64                                        (nullable)
 * The interpolation runs as factor^2 twisted N x N inverse transforms of the object's
 * spectrum, so any integer factor is exact up to float32 rounding.  The context allocates
 * a twist table (factor N complex64) and (factor + 2) N^2 complex64 of transform scratch
 * on the first call with a larger factor (not counted by ssb_info); SSB_ERR_OOM if that
 * fails. */
ssb_status ssb_reconstruct_upsampled(ssb_ctx *c, const ssb_params *theta, int factor,
                                     float *phase_out, float *object_c64_out, double *loss_out,
                                     void *cuda_stream);

/* Phase-of-mean redraw without the loss (page "Later SSB performance checkpoints", joint
 * calibration section: output reconstruction "phase only", factors 1 to 4).  The object
 * O = (1/n_bf) sum_k c_k is computed through its spectrum, O = (1/n_bf) IFFT2[sum_k C_k]
 * (equal by linearity): one sum of the corrected spectra over the BF pixels and a single
 * 2-D inverse transform, with no per-BF transform, phase or moment.  The correction and the
 * transfer are the objective's; the BF sum runs in 32 fixed slices (float32 within runs of
 * 32 BF pixels, float64 across), so results are run-to-run identical.  factor > 1 then
 * interpolates as ssb_reconstruct_upsampled does.
 *   factor:         1 .. SSB_MAX_UPSAMPLE
 *   phase_out:      device [factor N][factor N] float32, arg O              (required)
 *   object_c64_out: device [factor N][factor N] complex64 interleaved, O     (nullable)
 * The context allocates the slice sums (32 N^2 complex128) and two N^2 complex64 buffers
 * on the first call (not counted by ssb_info); SSB_ERR_OOM if that fails. */
ssb_status ssb_redraw(ssb_ctx *c, const ssb_params *theta, int factor, float *phase_out,
                      float *object_c64_out, void *cuda_stream);

/* Sizes of the G cache and of the scratch the context holds (either pointer nullable). */
ssb_status ssb_info(const ssb_ctx *c, size_t *g_bytes, size_t *scratch_bytes);

/* Copy the G cache, complex64 [n_bf][N/2+1][N], to dst (device or host, dst_on_device).
 * dst must hold g_bytes (ssb_info).  Synchronises the stream. */
ssb_status ssb_export_g(const ssb_ctx *c, void *dst, int dst_on_device, void *cuda_stream);

/* The count-unpacking step of ssb_prepare on its own: out[i] = (float)in[i] for n device
 * elements of dtype.  Counts above 2^24 give SSB_ERR_ARG (out is then unspecified). */
ssb_status ssb_unpack_counts(const void *in_device, ssb_dtype dtype, size_t n,
                             float *out_device, void *cuda_stream);

/* Per-kernel timing of one objective evaluation (tracing aid, as the pages' stage
 * profiles): the call runs one exact objective at theta with a CUDA event pair around
 * every launch on cuda_stream, then reports, per kernel name, the launch count and the
 * summed device time in milliseconds.  out: host [cap]; *n_out receives the number of
 * distinct kernels (entries beyond cap are dropped).  Synchronises the stream. */
typedef struct {
    char   name[48];
    int    launches;
    double ms;
} ssb_kernel_time;

ssb_status ssb_profile_objective(ssb_ctx *c, const ssb_params *theta, ssb_kernel_time *out,
                                 int cap, int *n_out, void *cuda_stream);

/* Per-kernel timing of every library call this thread makes between ssb_profile_begin
 * and ssb_profile_end (tracing aid): each launch gets a CUDA event pair on the stream it
 * runs on.  ssb_profile_end waits for those events and reports, per kernel name, the
 * launch count and the summed device time in milliseconds, as ssb_profile_objective does
 * (out: host [cap]; *n_out: distinct kernels).  One session per thread at a time;
 * ssb_profile_begin with a session (or ssb_profile_objective) already open on the thread,
 * or ssb_profile_end without one, gives SSB_ERR_ARG. */
ssb_status ssb_profile_begin(void);
ssb_status ssb_profile_end(ssb_kernel_time *out, int cap, int *n_out);

/* Loss of one trial without any device allocation.  (The pages have no counterpart: this
 * entry point exists for callers of this library that cannot allocate device memory when
 * they need a loss -- real-time pipelines that forbid allocation after set-up, because an
 * allocation can block on the driver and break their timing, and plug-ins whose host
 * application owns all GPU memory through its own allocator.)
 *   g:              geometry, as for ssb_prepare (host); transfer is SSB2.
 *   g_cache_device: the G cache on the current device, complex64 [n_bf][N/2+1][N], the
 *                   layout ssb_export_g writes; read only.
 *   theta:          host, one trial.     loss_out: host, one float64.
 * All scratch lives in one static 24 MiB device array that every GPU using the library
 * holds until the process exits; problems that do not fit (n_bf > 16384, or a layout
 * beyond 24 MiB) fail with SSB_ERR_ARG before any device work.  Set-up: the first call on
 * a device (and the first after that device's context was reset) looks up the array's
 * device address.  *loss_out is written only when the call returns SSB_OK.
 * Calls share the array and its contents persist between calls (what must start at zero
 * is cleared by each call), so calls that overlap on the GPU -- concurrent streams,
 * threads or devices sharing a call in flight -- race and must be serialised by the
 * caller.  Synchronises the stream.  Same loss as ssb_loss_batch up to float rounding
 * (its BF batches are smaller). */
ssb_status ssb_loss_noalloc(const ssb_geometry *g, const void *g_cache_device,
                            const ssb_params *theta, double *loss_out, void *cuda_stream);

/* Human-readable name of a status. */
const char *ssb_status_string(ssb_status s);

/* Detail of the most recent failure on the calling thread ("" if none). */
const char *ssb_last_error(void);

/* Number of kernels the library has launched in this process. */
uint64_t ssb_kernel_launches(void);

/* Release a context and its device memory (NULL is a no-op). */
void ssb_destroy(ssb_ctx *c);

#ifdef __cplusplus
}
#endif
#endif /* SSB_H */
