// The exact SSB phase-variance objective, batched over BF pixels.
//
//   k_theta_tables   per-trial tables: E(Q) = e^{i chi(lambda Q')} and the per-BF slopes
//                    of the bilinear phase B (32-bit turn fractions), from float64.
//   k_correct_cols   correction ("gamma", page "SSB performance notes") fused with the
//                    column inverse FFT over Qy; each half-plane column of G feeds the
//                    two output columns Qx and N-Qx (mirror rule G(-Q) = conj G(Q)).
//   k_rows_moments   row inverse FFT over Qx, phi = atan2, per-pixel sum of phi and phi^2
//                    in ascending BF order (page "Later SSB performance checkpoints",
//                    pass 2 "row IFFT + atan moments").
//   k_loss           fixed-order float64 reduction to the scalar loss.
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
    const double fr = t - rint(t);
    double s, c;
    sincospi(2.0 * fr, &s, &c);
    Et[i] = make_float2((float)c, (float)s);
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

// ---------------------------------------------------------------- correction + column IFFT

constexpr int kColsPerBlock = 4;

template <int N>
__global__ void __launch_bounds__(256) k_correct_cols(
    const float2 *__restrict__ G, float2 *__restrict__ X, const float2 *__restrict__ Et,
    const float4 *__restrict__ kgeo, const uint2 *__restrict__ kturn,
    const float2 *__restrict__ twg, TrialConst tc, int k0) {
    constexpr int CW = kColsPerBlock;
    constexpr int H = N / 2 + 1;
    extern __shared__ float2 sm[];
    float2 *tw = sm, *b0 = sm + N, *b1 = b0 + 2 * CW * N;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int kb = blockIdx.y, k = k0 + kb, g0 = blockIdx.x * CW;
    for (int i = tid; i < N; i += nt) tw[i] = twg[i];
    const float4 geo = kgeo[k];
    const uint2 bt = kturn[k];
    const float2 *Gk = G + (size_t)k * H * N;
    for (int idx = tid; idx < CW * N; idx += nt) {
        const int c = idx / N, ny = idx & (N - 1), g = g0 + c;
        const int ny2 = (N - ny) & (N - 1);
        float2 ca = make_float2(0.f, 0.f), cb = make_float2(0.f, 0.f);
        if (g < H) {
            const float2 v = Gk[(size_t)g * N + ny];
            ca = cmul(v, correction_factor<N>(ny, g, geo, bt, Et[(size_t)g * N + ny], tc));
            if (g > 0 && g < N / 2)  // G(ny2, N-g) = conj(G(ny, g))
                cb = cmul(cconj(v), correction_factor<N>(ny2, N - g, geo, bt,
                                                         Et[(size_t)(N - g) * N + ny2], tc));
        }
        b0[c * N + ny] = ca;
        b0[(CW + c) * N + ny2] = cb;
    }
    __syncthreads();
    const float2 *res = fft_batch_smem<N, +1>(b0, b1, 2 * CW, N, tw, tid, nt) ? b1 : b0;
    float2 *Xk = X + (size_t)kb * N * N;
    for (int idx = tid; idx < 2 * CW * N; idx += nt) {
        const int c = idx % (2 * CW), ry = idx / (2 * CW);
        if (c < CW) {
            const int g = g0 + c;
            if (g < H) Xk[(size_t)ry * N + g] = res[c * N + ry];
        } else {
            const int g = g0 + c - CW;
            if (g > 0 && g < N / 2) Xk[(size_t)ry * N + (N - g)] = res[c * N + ry];
        }
    }
}

// ---------------------------------------------------------------- row IFFT + atan2 + moments

template <int N, bool OBJ>
__global__ void __launch_bounds__(256) k_rows_moments(const float2 *__restrict__ X, int nb,
                                                      double *__restrict__ S1,
                                                      double *__restrict__ S2,
                                                      double2 *__restrict__ Osum,
                                                      const float2 *__restrict__ twg) {
    constexpr int RW = 1024 / N;
    constexpr int EPT = RW * N / 256;
    extern __shared__ float2 sm[];
    float2 *tw = sm, *b0 = sm + N, *b1 = b0 + RW * N;
    const int tid = threadIdx.x;
    const int ry0 = blockIdx.x * RW;
    for (int i = tid; i < N; i += 256) tw[i] = twg[i];
    float a1[EPT], a2[EPT];
    float2 ao[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        a1[e] = 0.f;
        a2[e] = 0.f;
        ao[e] = make_float2(0.f, 0.f);
    }
    for (int kb = 0; kb < nb; ++kb) {
        const float2 *src = X + ((size_t)kb * N + ry0) * N;
#pragma unroll
        for (int e = 0; e < EPT; ++e) b0[tid + e * 256] = src[tid + e * 256];
        __syncthreads();
        const float2 *res = fft_batch_smem<N, +1>(b0, b1, RW, N, tw, tid, 256) ? b1 : b0;
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
            const float2 v = res[tid + e * 256];
            const float phi = atan2f(v.y, v.x);
            a1[e] += phi;
            a2[e] = fmaf(phi, phi, a2[e]);
            if (OBJ) ao[e] = cadd(ao[e], v);
        }
        __syncthreads();
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        const size_t i = (size_t)ry0 * N + tid + e * 256;
        S1[i] += (double)a1[e];
        S2[i] += (double)a2[e];
        if (OBJ) Osum[i] = make_double2(Osum[i].x + ao[e].x, Osum[i].y + ao[e].y);
    }
}

// ---------------------------------------------------------------- loss and outputs

__global__ void __launch_bounds__(1024) k_loss(const double *__restrict__ S1,
                                               const double *__restrict__ S2, int P,
                                               double inv_n, double *__restrict__ out) {
    __shared__ double red[1024];
    const int tid = threadIdx.x;
    double acc = 0.0;
    for (int i = tid; i < P; i += 1024) {
        const double m = S1[i] * inv_n;
        acc += S2[i] * inv_n - m * m;
    }
    red[tid] = acc;
    __syncthreads();
    for (int s = 512; s > 0; s >>= 1) {
        if (tid < s) red[tid] += red[tid + s];
        __syncthreads();
    }
    if (tid == 0) *out = red[0] / (double)P;
}

__global__ void k_finalize(const double *__restrict__ S1, const double2 *__restrict__ Osum,
                           int P, double inv_n, double obj_scale, float *__restrict__ mean_phase,
                           float2 *__restrict__ obj) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= P) return;
    mean_phase[i] = (float)(S1[i] * inv_n);
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
    tc.lam = (float)a.lam;
    tc.inv_nstep = (float)(1.0 / (N * a.step));
    tc.semi = (float)a.semi;
    tc.inv_dalpha = (float)(1.0 / a.dalpha);
    tc.mode = a.mode;
    const double q = a.lam / (N * a.step);
    tc.lxs = (float)(q * th.cr);
    tc.lxy = (float)(-q * th.sr);
    tc.lys = (float)(q * th.sr);
    tc.lyy = (float)(q * th.cr);
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

template <int N>
static cudaError_t objective_n(const ObjectiveArgs &a, const TrialHost &th, double *loss_slot,
                               bool want_object, cudaStream_t s) {
    constexpr int P = N * N;
    cudaError_t e;
    if ((e = launch_theta_tables(a, th, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.S1, 0, sizeof(double) * P, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.S2, 0, sizeof(double) * P, s)) != cudaSuccess) return e;
    if (want_object && (e = cudaMemsetAsync(a.Osum, 0, sizeof(double2) * P, s)) != cudaSuccess)
        return e;
    const TrialConst tc = make_trial_const(a, th, N);
    constexpr int CW = kColsPerBlock;
    constexpr int H = N / 2 + 1;
    const size_t smem1 = (size_t)(N + 4 * CW * N) * sizeof(float2);
    const size_t smem2 = (size_t)(N + 2 * 1024) * sizeof(float2);
    if ((e = cudaFuncSetAttribute(k_correct_cols<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem1)) != cudaSuccess)
        return e;
    for (int k0 = 0; k0 < a.n_bf; k0 += a.B) {
        const int nb = a.n_bf - k0 < a.B ? a.n_bf - k0 : a.B;
        prof_begin("k_correct_cols", s);
        k_correct_cols<N><<<dim3((H + CW - 1) / CW, nb), 256, smem1, s>>>(
            a.G, a.X, a.E, a.kgeo, a.kturn, a.tw, tc, k0);
        prof_end(s);
        count_launch();
        prof_begin("k_rows_moments", s);
        if (want_object)
            k_rows_moments<N, true><<<N / (1024 / N), 256, smem2, s>>>(a.X, nb, a.S1, a.S2,
                                                                        a.Osum, a.tw);
        else
            k_rows_moments<N, false><<<N / (1024 / N), 256, smem2, s>>>(a.X, nb, a.S1, a.S2,
                                                                         a.Osum, a.tw);
        prof_end(s);
        count_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    prof_begin("k_loss", s);
    k_loss<<<1, 1024, 0, s>>>(a.S1, a.S2, P, 1.0 / a.n_bf, loss_slot);
    prof_end(s);
    count_launch();
    return cudaGetLastError();
}

cudaError_t run_objective(const ObjectiveArgs &a, const ssb_params &theta, double *loss_slot,
                          bool want_object, cudaStream_t s) {
    const TrialHost th = trial_host(theta);
    switch (a.N) {
        case 32: return objective_n<32>(a, th, loss_slot, want_object, s);
        case 64: return objective_n<64>(a, th, loss_slot, want_object, s);
        case 128: return objective_n<128>(a, th, loss_slot, want_object, s);
        case 256: return objective_n<256>(a, th, loss_slot, want_object, s);
        case 512: return objective_n<512>(a, th, loss_slot, want_object, s);
        default: return cudaErrorInvalidValue;
    }
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
