// Upsampled object redraw: band-limited interpolation of the BF-summed object onto a scan
// grid `factor` times finer (page "Later SSB performance checkpoints", joint CUDA
// calibration: reconstruct(result, upsample=factor) for factors 1-4; read as Fourier
// interpolation, the object's N x N spectrum kept at its signed fftfreq frequencies on the
// (factor N)^2 grid and every other frequency zero).
//
// In real space this is O_up = A O A^T with the (fN x N) interpolation matrix
//     A[m][n] = a(m - f n),   a(d) = (1/N) sum_{k=-N/2}^{N/2-1} exp(2 pi i k d / (f N)),
// evaluated on the host in float64 through the stable form
//     a(d) = (1/N) sin(N phi/2) / sin(phi/2) exp(-i phi/2),   phi = 2 pi d / (f N),
// with a(0) = 1 (a vanishes at the other multiples of f, so the original samples are
// kept).  The two products run as tiled complex GEMMs in float32 on the CUDA cores:
// T = O A^T (N x fN), then O_up = A T (fN x fN) with the phase (and optionally the
// object) written in the epilogue.  It is a small dense contraction (2.1e9 complex
// multiply-adds at f = 4, N = 512) next to the objective, and needs float32 accuracy,
// which the bf16/tf32 tensor-core formats do not give.
#include <cmath>
#include <vector>

#include "ssb_device.cuh"
#include "ssb_internal.h"

namespace ssb {

namespace {

constexpr int kBM = 64, kBQ = 64, kBK = 16;  // block tile (rows x columns), K step
constexpr int kUpThreads = 256;              // 16 x 16 threads, 4 x 4 outputs each

struct UpArgs {
    int N, f, off;             // off: index of a(0) in the table
    const float2 *tab;         // a(d), d = -off .. f N - 1
    const double2 *osum;       // [N][N] BF sum of the corrected images (pass 1)
    double scale;              // object = osum * scale
    float2 *T;                 // [N][f N] (pass 1 output, pass 2 input)
    float *phase;              // [f N][f N] (pass 2)
    float2 *obj;               // [f N][f N] or null (pass 2)
};

// Element (m, k) of the left operand and (k, q) of the right operand of each pass.
template <int PASS>
__device__ __forceinline__ float2 left_at(const UpArgs &u, int m, int k) {
    if (PASS == 0) {
        const double2 o = u.osum[(size_t)m * u.N + k];
        return make_float2((float)(o.x * u.scale), (float)(o.y * u.scale));
    }
    return u.tab[m - u.f * k + u.off];  // A[m][k]
}

template <int PASS>
__device__ __forceinline__ float2 right_at(const UpArgs &u, int k, int q) {
    if (PASS == 0) return u.tab[q - u.f * k + u.off];  // A^T[k][q] = A[q][k]
    return u.T[(size_t)k * u.f * u.N + q];
}

// C[M][Q] = sum_k L(m, k) R(k, q), K = N.  Pass 0: M = N, Q = f N, C -> T.  Pass 1:
// M = Q = f N, C -> phase (and object).  Thread (ty, tx) owns rows ty + 16 i and columns
// tx + 16 j of the block tile (i, j < 4), so its shared-memory reads are broadcasts or
// consecutive.
template <int PASS>
__global__ void __launch_bounds__(kUpThreads, 2) k_upsample(UpArgs u) {
    __shared__ float2 Ls[kBK][kBM];
    __shared__ float2 Rs[kBK][kBQ];
    const int M = PASS == 0 ? u.N : u.f * u.N, Q = u.f * u.N, K = u.N;
    const int m0 = blockIdx.y * kBM, q0 = blockIdx.x * kBQ;
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    float2 acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.f, 0.f);
    for (int k0 = 0; k0 < K; k0 += kBK) {
        // stage the tiles: 1024 elements each, 4 per thread (zero outside the matrices)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int e = tid + t * kUpThreads;
            const int lk = e / kBM, lm = e % kBM;  // L tile, stored k-major
            const int m = m0 + lm, k = k0 + lk;
            Ls[lk][lm] = (m < M && k < K) ? left_at<PASS>(u, m, k) : make_float2(0.f, 0.f);
            const int rk = e / kBQ, rq = e % kBQ;
            const int q = q0 + rq, kr = k0 + rk;
            Rs[rk][rq] = (q < Q && kr < K) ? right_at<PASS>(u, kr, q) : make_float2(0.f, 0.f);
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
            float2 l[4], r[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) l[i] = Ls[kk][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) r[j] = Rs[kk][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j].x = fmaf(l[i].x, r[j].x, fmaf(-l[i].y, r[j].y, acc[i][j].x));
                    acc[i][j].y = fmaf(l[i].x, r[j].y, fmaf(l[i].y, r[j].x, acc[i][j].y));
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty + 16 * i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = q0 + tx + 16 * j;
            if (q >= Q) continue;
            const size_t o = (size_t)m * Q + q;
            if (PASS == 0) {
                u.T[o] = acc[i][j];
            } else {
                u.phase[o] = atan2f(acc[i][j].y, acc[i][j].x);
                if (u.obj) u.obj[o] = acc[i][j];
            }
        }
    }
}

}  // namespace

size_t upsample_table_elems(int N, int factor) { return (size_t)factor * N + (size_t)factor * (N - 1); }
size_t upsample_scratch_elems(int N, int factor) { return (size_t)N * factor * N; }

void upsample_table(int N, int factor, std::vector<float2> &tab) {
    const int off = factor * (N - 1), fn = factor * N;
    tab.assign(upsample_table_elems(N, factor), make_float2(0.f, 0.f));
    const double pi = 3.14159265358979323846;
    for (int d = -off; d < fn; ++d) {
        double re = 1.0, im = 0.0;
        if (d != 0) {
            const double phi = 2.0 * pi * d / fn;
            const double ratio = std::sin(0.5 * N * phi) / (N * std::sin(0.5 * phi));
            re = ratio * std::cos(-0.5 * phi);
            im = ratio * std::sin(-0.5 * phi);
        }
        tab[d + off] = make_float2((float)re, (float)im);
    }
}

cudaError_t launch_upsample(const ObjectiveArgs &a, int factor, const float2 *tab, float2 *T,
                            float *phase_out, float2 *obj_out, cudaStream_t s) {
    UpArgs u;
    u.N = a.N;
    u.f = factor;
    u.off = factor * (a.N - 1);
    u.tab = tab;
    u.osum = a.Osum;
    u.scale = 1.0 / ((double)a.N * a.N * (double)a.n_bf);  // (1/P) inverse transform, 1/n_bf
    u.T = T;
    u.phase = phase_out;
    u.obj = obj_out;
    const int fn = factor * a.N;
    prof_begin("k_upsample_rows", s);
    k_upsample<0><<<dim3((fn + kBQ - 1) / kBQ, (a.N + kBM - 1) / kBM), kUpThreads, 0, s>>>(u);
    prof_end(s);
    count_launch();
    prof_begin("k_upsample_cols", s);
    k_upsample<1><<<dim3((fn + kBQ - 1) / kBQ, (fn + kBM - 1) / kBM), kUpThreads, 0, s>>>(u);
    prof_end(s);
    count_launch();
    return cudaGetLastError();
}

}  // namespace ssb
