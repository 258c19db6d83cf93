// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "../../include/ssb.h"
#include "ssb_device.cuh"

namespace ssb {

// Records the detail that ssb_last_error() reports on this thread.
void set_last_error(const char *msg);

// Launch-count bookkeeping (every kernel launch of the library goes through this).
void count_launch(uint64_t n = 1);

// Optional per-launch timing: when a profiling call is active on this thread,
// prof_begin/prof_end bracket a launch with CUDA events; otherwise they do nothing.
void prof_begin(const char *name, cudaStream_t s);
void prof_end(cudaStream_t s);

// Per-trial float64 constants derived on the host from theta and the geometry.
struct TrialHost {
    double cr, sr;        // rotation cos / sin
    double m00, m01, m11; // aberration matrix M (Angstrom): chi(u) = (pi/lambda) u^T M u
};

// ---- G-cache builder (ssb_prep.cu) ----
// counts [kc][N][N] raw (dtype) -> float32 F [kc][N][N]; sets *flag bit 1 on counts > 2^24
cudaError_t launch_unpack(const void *raw, ssb_dtype dtype, size_t n, float *out, int *flag,
                          cudaStream_t s);
// F [kc][N][N] float32 -> G [kc][N/2+1][N] complex64 using tmp [kc][N/2+1][N]
cudaError_t launch_rfft2(int N, const float *F, float2 *tmp, float2 *G, int kc,
                         const float2 *tw, cudaStream_t s);

// ---- objective (ssb_objective.cu) ----
struct ObjectiveArgs {
    int N;
    int n_bf;
    const float2 *G;        // [n_bf][N/2+1][N]
    const float4 *kgeo;     // [n_bf] (alpha_x, alpha_y, a_k, 0), float32
    const double2 *kalpha;  // [n_bf] (alpha_x, alpha_y), float64
    uint2 *kturn;           // [n_bf] per-trial B slopes (32-bit turn fractions)
    float2 *E;              // [N][N] per-trial e^{i chi(lambda Q')}
    const float2 *tw;       // [N] twiddles exp(+2 pi i m/N)
    double *S1;             // [N][N] float64 sum of phases
    double2 *Osum;          // [N][N] float64 object accumulator (nullable)
    double *loss;           // device float64, one per trial slot
    // fused (persistent) path
    float2 *Zring;          // column-pass intermediate ring
    float2 *hring;          // Nyquist-row Hermitian parts ring
    float2 *rring;          // Nyquist-row transforms ring
    double *S2g;            // per row task sums of phi^2
    unsigned *sync;         // scheduler counters
    unsigned *err;          // error word (raised by a wait that ran out)
    int Bk;                 // BF planes per batch
    int D;                  // ring slots
    int mode;               // 0 SSB2, 1 SSB1
    double step, lam, semi, dalpha;  // geometry (Angstrom, rad)
    unsigned wait_limit;    // polls before a scheduler wait gives up (0: the default)
    int stall;              // test hook: row tasks wait for a count never reached
};

TrialHost trial_host(const ssb_params &t);
// float32 per-trial constants for the correction factor
TrialConst make_trial_const(const ObjectiveArgs &a, const TrialHost &th, int N);
// per-trial tables E and kturn
cudaError_t launch_theta_tables(const ObjectiveArgs &a, const TrialHost &th, cudaStream_t s);

// persistent fused path (SSB2): sizes of its buffers and the evaluation itself
size_t fused_sync_words(int N, int n_bf, int Bk);
size_t fused_ring_elems(int N, int Bk, int D, bool ssb1 = false);  // ssb1: all N columns
size_t fused_hring_elems(int N, int Bk, int D);
size_t fused_rring_elems(int N, int Bk, int D);
int fused_row_tasks(int N);
size_t fused_s2g_elems(int N);  // per row task S2 sums, then the loss kernel's block partials
// One full objective evaluation on the persistent fused kernel (accumulators and
// scheduler words cleared first), loss written to *loss_slot.  The error word (a.err) is
// not cleared here: the caller clears it once per library call and reads it at the end, so
// a wait that ran out in any evaluation of the call is reported (and every later loss of
// the call is NaN).
cudaError_t run_objective_fused(const ObjectiveArgs &a, const ssb_params &theta, double *loss_slot,
                                bool want_object, cudaStream_t s);

// mean phase = S1/n_bf (float32), object = Osum * scale (complex64) if out_obj != nullptr
cudaError_t launch_finalize(const ObjectiveArgs &a, float *mean_phase, float *out_obj,
                            cudaStream_t s);

// ---- upsampled redraw (ssb_upsample.cu) ----
// Twist table exp(2 pi i m / (factor N)), m < factor N (complex64), and the size of the
// transform scratch (factor + 2 planes of N x N complex64).
size_t upsample_table_elems(int N, int factor);
size_t upsample_scratch_elems(int N, int factor);
void upsample_table(int N, int factor, std::vector<float2> &tab);
// From Osum (filled by an evaluation with want_object): phase [fN][fN] float32 and, if
// obj_out != nullptr, the object [fN][fN] complex64 on the factor-times finer grid.
cudaError_t launch_upsample(const ObjectiveArgs &a, int factor, const float2 *tab, float2 *T,
                            float *phase_out, float2 *obj_out, cudaStream_t s);

}  // namespace ssb
