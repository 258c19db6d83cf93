// Object redraw without the loss: the phase-of-mean output (page "Later SSB performance
// checkpoints", joint calibration section, "phase only" output times; page "SSB
// performance notes", object redraw), computed from its definition through linearity,
//     O(r) = (1/n_bf) sum_k c_k(r) = (1/n_bf) IFFT2[ sum_k C_k ](r),
// so the per-BF inverse transforms, phases and moments of the objective are not needed:
//   k_redraw_sum      sum over the BF pixels of the corrected spectra C_k (the same
//                     correction as the objective), in fixed slices of the BF range;
//                     float32 within runs of 32 BF, float64 across them (a float pair by
//                     exact two-sums instead measured slower here)
//   k_redraw_combine  the slices added in slice order; for SSB2 the other half plane from
//                     the anti-Hermitian symmetry of the corrected spectrum
//   k_redraw_fft      one 2-D inverse transform of the N x N sum (register FFTs over
//                     the columns, then the rows), the unnormalised result written to
//                     the object accumulator, and on request the phase arg O and the
//                     object O / (N^2 n_bf)
// SSB2: C_k(-Q) = -conj C_k(Q) off the DC bin and the Nyquist row, so the half-plane
// columns 0..N/2 are summed directly, plus the Nyquist-row bins of the other half (the
// mirror bin of (nx, N/2) is evaluated at signed (-nx, -N/2), not at the negation of
// (nx, -N/2)); every other bin follows from the symmetry.  SSB1 has no symmetry: all N
// columns are summed, the other half reading the cache through G(-Q) = conj G(Q).
#include <algorithm>

#include "ssb_device.cuh"
#include "ssb_internal.h"
#include "ssb_redraw.h"
#include "ssb_regfft.cuh"

namespace ssb {

namespace {

constexpr int kRdThreads = 128;  // threads per block of the spectral sum
constexpr int kRdBins = 4;       // bins per thread, rows ny = jj + (N / kRdBins) r
constexpr int kRdRun = 32;       // BF planes summed in float32 before the float64 update
constexpr int kRdSlices = 32;    // BF slices of the spectral sum (fixed: the result is
                                 // the same on every device)
constexpr int kRdFftThreads = 128;
constexpr int kRdPts = 16;       // points per thread of the redraw transforms

struct RedrawArgs {
    const float2 *G;        // [n_bf][N/2+1][N]
    const float4 *kgeo;     // [n_bf]
    const uint2 *kturn;     // [n_bf]
    const float2 *E;        // [N][N]
    TrialConst tc;
    int n_bf, kps;          // BF pixels, BF pixels per slice
    double2 *part;          // [slices][N][N] slice sums
    int slices;
    float2 *S;              // [N][N] full-plane spectral sum, [nx][ny]
    float2 *T;              // [N][N] after the column transforms, [nx][ry]
    const float2 *tw;       // [N] exp(+2 pi i m / N)
    double2 *Osum;          // [N][N] unnormalised inverse transform, [ry][rx]
    float *phase;           // [N][N] or null
    float2 *obj;            // [N][N] or null
    double obj_scale;       // 1 / (N^2 n_bf)
};

__device__ __forceinline__ void cadd_to(float2 &a, float2 b) {
    a.x += b.x;
    a.y += b.y;
}
__device__ __forceinline__ void flush(double2 &t, float2 &a) {
    t.x += (double)a.x;
    t.y += (double)a.y;
    a = make_float2(0.f, 0.f);
}

// The column's G values of plane k (none when the column carries no transfer there).
template <int N, bool SSB1>
__device__ __forceinline__ void rd_load(const float2 *__restrict__ G, int k, int nx, int jj, bool zero,
                                        float2 (&gv)[kRdBins]) {
    constexpr int TPC = N / kRdBins, HG = N / 2 + 1;
    if (zero) return;
    if (!SSB1 || nx <= N / 2) {
        const float2 *g = G + ((size_t)k * HG + nx) * N + jj;
#pragma unroll
        for (int r = 0; r < kRdBins; ++r) gv[r] = __ldcs(g + TPC * r);
    } else {  // G(nx, ny) = conj G(N - nx, N - ny), row index mod N
        const float2 *g = G + ((size_t)k * HG + (N - nx)) * N;
#pragma unroll
        for (int r = 0; r < kRdBins; ++r) gv[r] = cconj(__ldcs(g + ((N - jj - TPC * r) & (N - 1))));
    }
}

// Block (x: column group, y: BF slice).  Thread jj of a column holds rows jj + TPC r.  The
// slice's per-BF geometry is staged in shared memory in the form the column terms need --
// u = alpha_k . (cos, sin) of the scan rotation, q u, q w and |alpha_k|^2 (q = lam_q), the
// very float expressions of column_zero and col_geom, evaluated once per BF pixel instead of
// once per column and BF pixel -- and the G values of the next plane are loaded while the
// current plane is corrected.
template <int N, bool SSB1>
__global__ void __launch_bounds__(kRdThreads) k_redraw_sum(RedrawArgs p) {
    constexpr int TPC = N / kRdBins;                      // threads per column
    constexpr int CPB = TPC >= kRdThreads ? 1 : kRdThreads / TPC;  // columns per block
    constexpr int NCOL = SSB1 ? N : N / 2 + 1;
    static_assert(TPC <= kRdThreads && kRdThreads % TPC == 0, "column split");
    extern __shared__ float4 rd_geo[];  // [kps] (u, q u, q w, |alpha|^2), uint2 [kps], float [kps] a_k
    uint2 *rd_bt = (uint2 *)(rd_geo + p.kps);
    float *rd_a = (float *)(rd_bt + p.kps);
    const int k0 = blockIdx.y * p.kps, k1 = min(p.n_bf, k0 + p.kps);
    const int nk = max(0, k1 - k0);
    const TrialConst &tc = p.tc;
    for (int i = threadIdx.x; i < nk; i += kRdThreads) {
        const float4 g = __ldg(p.kgeo + k0 + i);
        const float q = tc.lam_q;
        const float u = fmaf(g.x, tc.cr, g.y * tc.sr), w = fmaf(g.y, tc.cr, -g.x * tc.sr);
        rd_geo[i] = make_float4(u, q * u, q * w, fmaf(g.x, g.x, g.y * g.y));
        rd_bt[i] = __ldg(p.kturn + k0 + i);
        rd_a[i] = g.z;
    }
    __syncthreads();
    const int jj = threadIdx.x % TPC;
    const int nx = blockIdx.x * CPB + threadIdx.x / TPC;
    if (nx >= NCOL) return;  // no block-level synchronisation below
    const int sx = nx < N / 2 ? nx : nx - N;
    const float fsx = (float)sx;
    const float osx = tc.lam_q * fsx;           // the column's offset along the rotated axis
    const float q2 = tc.lam_q * tc.lam_q, sx2 = fsx * fsx;
    float2 e[kRdBins];
#pragma unroll
    for (int r = 0; r < kRdBins; ++r) e[r] = __ldg(p.E + (size_t)nx * N + jj + TPC * r);
    // SSB2: the thread holding row N/2 (jj = 0, r = kRdBins / 2) of a column 1..N/2-1 also
    // sums the mirror Nyquist bin (N - nx, N/2)
    const bool nyq = !SSB1 && jj == 0 && nx >= 1 && nx < N / 2;
    const float2 em = nyq ? __ldg(p.E + (size_t)(N - nx) * N + N / 2) : make_float2(0.f, 0.f);
    double2 tot[kRdBins];
    float2 acc[kRdBins];
#pragma unroll
    for (int r = 0; r < kRdBins; ++r) {
        tot[r] = make_double2(0.0, 0.0);
        acc[r] = make_float2(0.f, 0.f);
    }
    double2 totm = make_double2(0.0, 0.0);
    float2 accm = make_float2(0.f, 0.f);
    // column_zero / column_zero1 of BF pixel i of the slice, from its staged u
    auto is_zero = [&](int i) {
        const float u = rd_geo[i].x;
        return nx > 0 && (!(rd_a[i] > 0.0f) ||
                          (fabsf(u - osx) >= tc.zero_r && (SSB1 || fabsf(u + osx) >= tc.zero_r)));
    };
    float2 gv[kRdBins], gn[kRdBins];
    bool zero = nk > 0 ? is_zero(0) : true;
    rd_load<N, SSB1>(p.G, k0, nx, jj, zero, gv);
    for (int it = 0; it < nk; ++it) {
        const float4 geo = rd_geo[it];
        const uint2 bt = rd_bt[it];
        const bool zn = it + 1 < nk ? is_zero(it + 1) : true;
        rd_load<N, SSB1>(p.G, k0 + it + 1, nx, jj, zn, gn);
        if (!zero) {
            const bool active = rd_a[it] > 0.0f;
            // col_geom's terms: base = q^2 sx^2 + |alpha|^2, p0 = (q u) sx, qw = q w
            ColGeom cg;
            cg.q2 = q2;
            cg.base = fmaf(q2, sx2, geo.w);
            cg.p0 = geo.y * fsx;
            cg.qw = geo.z;
            const uint32_t phx = bt.x * (uint32_t)sx;
#pragma unroll
            for (int r = 0; r < kRdBins; ++r) {
                const int ny = jj + TPC * r;
                const int sy = ny < N / 2 ? ny : ny - N;
                float2 cv = make_float2(0.f, 0.f);
                if (active)
                    cv = SSB1 ? correct_ssb1(gv[r], (float)sy, sy, e[r], cg, phx, bt.y, tc)
                              : correct_ssb2(gv[r], (float)sy, sy, e[r], cg, phx, bt.y, tc);
                if ((nx | ny) == 0) cv = gv[r];  // C(0) = G(0)
                cadd_to(acc[r], cv);
            }
            if (nyq && active) {
                // bin (N - nx, N/2): G = conj G(nx, N/2), signed bins (-nx, -N/2), where the
                // column geometry has p0 negated and the x part of B is negated
                ColGeom cm = cg;
                cm.p0 = -cg.p0;
                cadd_to(accm, correct_ssb2(cconj(gv[kRdBins / 2]), -(float)(N / 2), -N / 2, em, cm,
                                           0u - phx, bt.y, tc));
            }
        }
        if ((it % kRdRun) == kRdRun - 1) {
#pragma unroll
            for (int r = 0; r < kRdBins; ++r) flush(tot[r], acc[r]);
            flush(totm, accm);
        }
        zero = zn;
#pragma unroll
        for (int r = 0; r < kRdBins; ++r) gv[r] = gn[r];
    }
#pragma unroll
    for (int r = 0; r < kRdBins; ++r) flush(tot[r], acc[r]);
    flush(totm, accm);
    double2 *out = p.part + (size_t)blockIdx.y * N * N;
#pragma unroll
    for (int r = 0; r < kRdBins; ++r) out[(size_t)nx * N + jj + TPC * r] = tot[r];
    if (nyq) out[(size_t)(N - nx) * N + N / 2] = totm;
}

// Slice sums added in slice order; SSB2 bins outside the summed set from -conj of their
// mirror bin.
template <int N, bool SSB1>
__global__ void k_redraw_combine(RedrawArgs p) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N * N) return;
    const int nx = i / N, ny = i - nx * N;
    const bool direct = SSB1 || nx <= N / 2 || ny == N / 2;
    const int src = direct ? i : (N - nx) * N + ((N - ny) & (N - 1));
    double sx = 0.0, sy = 0.0;
    for (int s = 0; s < p.slices; ++s) {
        const double2 d = p.part[(size_t)s * N * N + src];
        sx += d.x;
        sy += d.y;
    }
    p.S[i] = direct ? make_float2((float)sx, (float)sy) : make_float2((float)-sx, (float)sy);
}

}  // namespace

namespace {

__device__ __forceinline__ void redraw_warp_bar() { __syncwarp(); }

// One inverse transform of length N per group of N/16 threads (16 points each); ROWS = false
// transforms the columns of S (over ny, contiguous) into T, ROWS = true the rows of T (over
// nx, stride N) into the object accumulator [ry][rx].  Groups past the last line run on a
// clamped line (every lane of a warp takes part in its synchronisation) and store nothing.
template <int N, bool ROWS>
__global__ void __launch_bounds__(kRdFftThreads) k_redraw_fft(RedrawArgs p) {
    constexpr int T = N / kRdPts;
    constexpr int GROUPS = kRdFftThreads / T;
    constexpr int PAD = PadLen<N>::value;
    __shared__ float2 tws[PAD];
    __shared__ float2 scratch[GROUPS * PAD];
    for (int i = threadIdx.x; i < N; i += kRdFftThreads) tws[lay(i)] = p.tw[i];
    __syncthreads();
    const int grp = threadIdx.x / T, j = threadIdx.x % T;
    const int line = blockIdx.x * GROUPS + grp;
    const bool valid = line < N;
    const int ld = valid ? line : N - 1;
    float2 v[kRdPts];
#pragma unroll
    for (int r = 0; r < kRdPts; ++r)
        v[r] = ROWS ? p.T[(size_t)(j + T * r) * N + ld] : p.S[(size_t)ld * N + j + T * r];
    reg_fft<N, kRdPts, +1>(v, scratch + grp * PAD, tws, j, redraw_warp_bar);
    if (!valid) return;
#pragma unroll
    for (int r = 0; r < kRdPts; ++r) {
        const size_t o = (size_t)ld * N + j + T * r;
        if (!ROWS) {
            p.T[o] = v[r];
        } else {
            p.Osum[o] = make_double2((double)v[r].x, (double)v[r].y);
            if (p.phase) p.phase[o] = atan2f(v[r].y, v[r].x);
            if (p.obj)
                p.obj[o] = make_float2((float)(v[r].x * p.obj_scale), (float)(v[r].y * p.obj_scale));
        }
    }
}

template <int N, bool SSB1>
cudaError_t redraw_n(RedrawArgs &r, cudaStream_t s) {
    constexpr int TPC = N / kRdBins;
    constexpr int CPB = TPC >= kRdThreads ? 1 : kRdThreads / TPC;
    constexpr int NCOL = SSB1 ? N : N / 2 + 1;
    const size_t smem = (sizeof(float4) + sizeof(uint2) + sizeof(float)) * (size_t)r.kps;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_redraw_sum<N, SSB1>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    prof_begin("k_redraw_sum", s);
    k_redraw_sum<N, SSB1><<<dim3((NCOL + CPB - 1) / CPB, r.slices), kRdThreads, smem, s>>>(r);
    prof_end(s);
    count_launch();
    prof_begin("k_redraw_combine", s);
    k_redraw_combine<N, SSB1><<<(N * N + 255) / 256, 256, 0, s>>>(r);
    prof_end(s);
    count_launch();
    constexpr int GROUPS = kRdFftThreads / (N / kRdPts);
    const int blocks = (N + GROUPS - 1) / GROUPS;
    prof_begin("k_redraw_fft", s);
    k_redraw_fft<N, false><<<blocks, kRdFftThreads, 0, s>>>(r);
    prof_end(s);
    count_launch();
    prof_begin("k_redraw_fft", s);
    k_redraw_fft<N, true><<<blocks, kRdFftThreads, 0, s>>>(r);
    prof_end(s);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

int redraw_slices(int n_bf) { return std::min(n_bf, kRdSlices); }
size_t redraw_part_elems(int N, int n_bf) { return (size_t)redraw_slices(n_bf) * N * N; }

cudaError_t launch_redraw(const ObjectiveArgs &a, const ssb_params &theta, double2 *part, float2 *S,
                          float2 *T, float *phase_out, float2 *obj_out, cudaStream_t s) {
    const TrialHost th = trial_host(theta);
    cudaError_t e = launch_theta_tables(a, th, s);
    if (e != cudaSuccess) return e;
    RedrawArgs r;
    r.G = a.G;
    r.kgeo = a.kgeo;
    r.kturn = a.kturn;
    r.E = a.E;
    r.tc = make_trial_const(a, th, a.N);
    r.n_bf = a.n_bf;
    r.slices = redraw_slices(a.n_bf);
    r.kps = (a.n_bf + r.slices - 1) / r.slices;
    r.part = part;
    r.S = S;
    r.T = T;
    r.tw = a.tw;
    r.Osum = a.Osum;
    r.phase = phase_out;
    r.obj = obj_out;
    r.obj_scale = 1.0 / ((double)a.N * a.N * (double)a.n_bf);
    const bool s1 = a.mode == 1;
    switch (a.N) {
        case 32: return s1 ? redraw_n<32, true>(r, s) : redraw_n<32, false>(r, s);
        case 64: return s1 ? redraw_n<64, true>(r, s) : redraw_n<64, false>(r, s);
        case 128: return s1 ? redraw_n<128, true>(r, s) : redraw_n<128, false>(r, s);
        case 256: return s1 ? redraw_n<256, true>(r, s) : redraw_n<256, false>(r, s);
        case 512: return s1 ? redraw_n<512, true>(r, s) : redraw_n<512, false>(r, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssb
