// Per-trial tables and outputs of the exact SSB phase-variance objective (the objective
// itself runs in the persistent fused kernel).
//
//   k_theta_E, k_theta_k  per-trial tables: E(Q) = e^{i chi(lambda Q')} and the per-BF
//                         slopes of the bilinear phase B (32-bit turn fractions), from
//                         float64.
//   k_finalize            mean phase S1 / n_bf and the BF-summed object, for the redraw.
#include <cmath>

#include "ssb_device.cuh"
#include "ssb_internal.h"

namespace ssb {

// ---------------------------------------------------------------- per-trial tables

__global__ void k_theta_E(float2 *__restrict__ Et, int N, double inv_nstep, double lam,
                          double cr, double sr, double m00, double m01, double m11) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N * N) return;
    const int nx = i / N, ny = i - nx * N;  // stored [nx][ny]
    const int sx = nx < N / 2 ? nx : nx - N, sy = ny < N / 2 ? ny : ny - N;
    const double fx = sx * inv_nstep, fy = sy * inv_nstep;
    const double qx = cr * fx - sr * fy, qy = sr * fx + cr * fy;
    // chi(lambda Q') / 2 pi = (lambda/2) Q'^T M Q'   (turns)
    const double t = 0.5 * lam * (m00 * qx * qx + 2.0 * m01 * qx * qy + m11 * qy * qy);
    const double fr = t - rint(t);  // exact range reduction in float64, |fr| <= 1/2
    // the table is complex64: the float32 function of the reduced angle is as accurate as
    // rounding a float64 one, at a fraction of the float64 cost
    float s, c;
    sincospif((float)(2.0 * fr), &s, &c);
    Et[i] = make_float2(c, s);
}

__device__ __forceinline__ uint32_t turn_fraction_u32(double turns) {
    const double f = turns - floor(turns);  // [0, 1)
    const long long v = llrint(f * 4294967296.0);
    return (uint32_t)(v & 0xffffffffLL);
}

__global__ void k_theta_k(uint2 *__restrict__ kturn, const double2 *__restrict__ kalpha,
                          int n_bf, double inv_nstep, double cr, double sr, double m00,
                          double m01, double m11) {
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= n_bf) return;
    const double2 a = kalpha[k];
    // B / 2 pi = alpha_k^T M Q' = (R^T M alpha_k) . Q,  Q = (sx, sy) / (N step)
    const double ux = m00 * a.x + m01 * a.y, uy = m01 * a.x + m11 * a.y;
    const double vx = cr * ux + sr * uy, vy = -sr * ux + cr * uy;
    kturn[k] = make_uint2(turn_fraction_u32(vx * inv_nstep), turn_fraction_u32(vy * inv_nstep));
}


// ---------------------------------------------------------------- outputs

__global__ void k_finalize(const double *__restrict__ S1, const double2 *__restrict__ Osum,
                           int P, double inv_n, double obj_scale, float *__restrict__ mean_phase,
                           float2 *__restrict__ obj) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= P) return;
    mean_phase[i] = (float)(s1_value(S1, i) * inv_n);
    if (obj) {
        const double2 o = Osum[i];
        obj[i] = make_float2((float)(o.x * obj_scale), (float)(o.y * obj_scale));
    }
}

// ---------------------------------------------------------------- host orchestration

TrialHost trial_host(const ssb_params &t) {
    TrialHost th;
    th.cr = std::cos(t.rotation_rad);
    th.sr = std::sin(t.rotation_rad);
    const double c10 = t.C10_nm * 10.0, c12 = t.C12_nm * 10.0;
    th.m00 = c10 + c12 * std::cos(2.0 * t.phi12_rad);
    th.m11 = c10 - c12 * std::cos(2.0 * t.phi12_rad);
    th.m01 = c12 * std::sin(2.0 * t.phi12_rad);
    return th;
}

TrialConst make_trial_const(const ObjectiveArgs &a, const TrialHost &th, int N) {
    TrialConst tc;
    tc.cr = (float)th.cr;
    tc.sr = (float)th.sr;
    tc.semi = (float)a.semi;
    tc.inv_dalpha = (float)(1.0 / a.dalpha);
    const double q = a.lam / (N * a.step);
    const double inner = a.semi - 0.5 * a.dalpha, outer = a.semi + 0.5 * a.dalpha;
    tc.inner2 = inner > 0.0 ? (float)(inner * inner) * (1.0f - 4e-7f) : -1.0f;
    tc.outer2 = (float)(outer * outer) * (1.0f + 4e-7f);
    tc.lam_q = (float)q;
    tc.zero_r = (float)(outer * (1.0 + 1e-4));
    return tc;
}

cudaError_t launch_theta_tables(const ObjectiveArgs &a, const TrialHost &th, cudaStream_t s) {
    const int N = a.N, P = N * N;
    const double inv_nstep = 1.0 / (N * a.step);
    prof_begin("k_theta_E", s);
    k_theta_E<<<(P + 255) / 256, 256, 0, s>>>(a.E, N, inv_nstep, a.lam, th.cr, th.sr, th.m00,
                                             th.m01, th.m11);
    prof_end(s);
    count_launch();
    prof_begin("k_theta_k", s);
    k_theta_k<<<(a.n_bf + 127) / 128, 128, 0, s>>>(a.kturn, a.kalpha, a.n_bf, inv_nstep, th.cr,
                                                  th.sr, th.m00, th.m01, th.m11);
    prof_end(s);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_finalize(const ObjectiveArgs &a, float *mean_phase, float *out_obj,
                            cudaStream_t s) {
    const int P = a.N * a.N;
    const double scale = 1.0 / ((double)P * (double)a.n_bf);
    k_finalize<<<(P + 255) / 256, 256, 0, s>>>(a.S1, a.Osum, P, 1.0 / a.n_bf, scale, mean_phase,
                                               (float2 *)out_obj);
    count_launch();
    return cudaGetLastError();
}

}  // namespace ssb
