// Upsampled object redraw: band-limited interpolation of the BF-summed object onto a scan
// grid `factor` times finer (page "Later SSB performance checkpoints", joint CUDA
// calibration: reconstruct(result, upsample=factor) for factors 1-4; read as Fourier
// interpolation, the object's N x N spectrum kept at its signed fftfreq frequencies on the
// (factor N)^2 grid and every other frequency zero):
//     O_up(m) = (1/N^2) sum_{k in [-N/2, N/2)^2} O^(k) exp(2 pi i k.m / (f N)),  O^ = FFT2(O).
// Splitting each output index as m = f q + p (q < N, p < f) turns this into f^2 ordinary
// N x N inverse transforms of twisted spectra:
//     O_up(f qy + py, f qx + px) = (1/N^2) IFFT2_N[ O^(k) w^(ky py + kx px) ](qy, qx),
//     w = exp(2 pi i / (f N)),
// so every factor, power of two or not, runs on the library's N-point register FFTs:
//   k_up_fwd    O^ = FFT2 of the object accumulator (rows, then columns)
//   k_up_cols   for each py and column kx: twist by w^(ky py), inverse over ky
//   k_up_rows   for each (py, px) and row qy: twist by w^(kx px), inverse over kx, and the
//               phase (and the object) written at (f qy + py, f qx + px)
// About 5 f^2 N^2 log2 N flops (0.19 GFLOP at f = 4, N = 512) instead of the 21 GFLOP of
// the interpolation written as two dense products; the work is bound by memory latency and
// L2 traffic, not by arithmetic.  The twist table w^m (m < f N) is evaluated on the host in
// float64.
#include <cmath>
#include <vector>

#include "ssb_device.cuh"
#include "ssb_internal.h"
#include "ssb_regfft.cuh"

namespace ssb {

namespace {

constexpr int kUpThreads = 128;
constexpr int kUpPts = 16;  // points per thread of the N-point transforms

struct UpArgs {
    int f;                      // factor
    const double2 *osum;        // [N][N] object accumulator, [y][x]
    const float2 *tw;           // [N] exp(+2 pi i m / N)
    const float2 *twf;          // [f N] exp(+2 pi i m / (f N))
    float2 *W;                  // [N][N] rows transformed, [y][kx]
    float2 *spec;               // [N][N] spectrum, [kx][ky]
    float2 *U;                  // [f][N][N] columns inverse-transformed, [py][kx][qy]
    float *phase;               // [f N][f N]
    float2 *obj;                // [f N][f N] or null
    float scale;                // 1 / (N^4 n_bf): object = IFFT2(FFT2(Osum) twist) * scale
};

__device__ __forceinline__ void up_warp_bar() { __syncwarp(); }

// Twist factor w^(s p) for a signed frequency s, from the table of w^m, m < f N.
__device__ __forceinline__ float2 twist(const float2 *twf, int fn, int s, int pp) {
    int m = (s * pp) % fn;
    if (m < 0) m += fn;
    return __ldg(twf + m);
}

// One N-point transform per group of N/16 threads.  Lines past `lines` run on a clamped
// line (every lane of a warp takes part in the exchanges) and store nothing.  MODE:
//   0  forward over x of Osum row y          -> W[y][kx]
//   1  forward over y of W column kx         -> spec[kx][ky]
//   2  inverse over ky of column kx, twisted -> U[py][kx][qy]      (line = py N + kx)
//   3  inverse over kx of row qy, twisted    -> out (f qy + py, f qx + px)
//                                               (line = (py N + qy) f + px: the groups of a
//                                               block share the U values they read and fill
//                                               neighbouring outputs)
template <int N, int MODE>
__global__ void __launch_bounds__(kUpThreads) k_up_line(UpArgs u, int lines) {
    constexpr int T = N / kUpPts;
    constexpr int GROUPS = kUpThreads / T;
    constexpr int PAD = PadLen<N>::value;
    __shared__ float2 tws[PAD];
    __shared__ float2 scratch[GROUPS * PAD];
    for (int i = threadIdx.x; i < N; i += kUpThreads) tws[lay(i)] = u.tw[i];
    __syncthreads();
    const int grp = threadIdx.x / T, j = threadIdx.x % T;
    const int line = blockIdx.x * GROUPS + grp;
    const bool valid = line < lines;
    const int ld = valid ? line : lines - 1;
    const int fn = u.f * N;
    float2 v[kUpPts];
    if (MODE == 0) {
#pragma unroll
        for (int r = 0; r < kUpPts; ++r) {
            const double2 o = u.osum[(size_t)ld * N + j + T * r];
            v[r] = make_float2((float)o.x, (float)o.y);
        }
    } else if (MODE == 1) {
#pragma unroll
        for (int r = 0; r < kUpPts; ++r) v[r] = u.W[(size_t)(j + T * r) * N + ld];
    } else if (MODE == 2) {
        const int py = ld / N, kx = ld - py * N;
#pragma unroll
        for (int r = 0; r < kUpPts; ++r) {
            const int ky = j + T * r;
            const int sy = ky < N / 2 ? ky : ky - N;
            v[r] = cmul(u.spec[(size_t)kx * N + ky], twist(u.twf, fn, sy, py));
        }
    } else {
        const int t = ld / u.f, px = ld - t * u.f;
        const int py = t / N, qy = t - py * N;
#pragma unroll
        for (int r = 0; r < kUpPts; ++r) {
            const int kx = j + T * r;
            const int sx = kx < N / 2 ? kx : kx - N;
            v[r] = cmul(u.U[((size_t)py * N + kx) * N + qy], twist(u.twf, fn, sx, px));
        }
    }
    if (MODE <= 1)
        reg_fft<N, kUpPts, -1>(v, scratch + grp * PAD, tws, j, up_warp_bar);
    else
        reg_fft<N, kUpPts, +1>(v, scratch + grp * PAD, tws, j, up_warp_bar);
    if (!valid) return;
    if (MODE == 0) {
#pragma unroll
        for (int r = 0; r < kUpPts; ++r) u.W[(size_t)ld * N + j + T * r] = v[r];
    } else if (MODE == 1) {
#pragma unroll
        for (int r = 0; r < kUpPts; ++r) u.spec[(size_t)ld * N + j + T * r] = v[r];
    } else if (MODE == 2) {
#pragma unroll
        for (int r = 0; r < kUpPts; ++r) u.U[(size_t)ld * N + j + T * r] = v[r];
    } else {
        const int t = ld / u.f, px = ld - t * u.f;
        const int py = t / N, qy = t - py * N;
        const size_t row = (size_t)(u.f * qy + py) * fn + px;
#pragma unroll
        for (int r = 0; r < kUpPts; ++r) {
            const size_t o = row + (size_t)u.f * (j + T * r);
            u.phase[o] = atan2f(v[r].y, v[r].x);
            if (u.obj) u.obj[o] = make_float2(v[r].x * u.scale, v[r].y * u.scale);
        }
    }
}

template <int N, int MODE>
void up_launch(const UpArgs &u, int lines, const char *name, cudaStream_t s) {
    constexpr int GROUPS = kUpThreads / (N / kUpPts);
    prof_begin(name, s);
    k_up_line<N, MODE><<<(lines + GROUPS - 1) / GROUPS, kUpThreads, 0, s>>>(u, lines);
    prof_end(s);
    count_launch();
}

template <int N>
cudaError_t upsample_n(const UpArgs &u, cudaStream_t s) {
    up_launch<N, 0>(u, N, "k_up_fwd", s);
    up_launch<N, 1>(u, N, "k_up_fwd", s);
    up_launch<N, 2>(u, u.f * N, "k_up_cols", s);
    up_launch<N, 3>(u, u.f * u.f * N, "k_up_rows", s);
    return cudaGetLastError();
}

}  // namespace

size_t upsample_table_elems(int N, int factor) { return (size_t)factor * N; }
// U (factor planes of N x N), then W and the spectrum
size_t upsample_scratch_elems(int N, int factor) { return (size_t)(factor + 2) * N * N; }

void upsample_table(int N, int factor, std::vector<float2> &tab) {
    const int fn = factor * N;
    tab.resize(fn);
    const double pi = 3.14159265358979323846;
    for (int m = 0; m < fn; ++m) {
        const double a = 2.0 * pi * m / fn;
        tab[m] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
}

cudaError_t launch_upsample(const ObjectiveArgs &a, int factor, const float2 *tab, float2 *T,
                            float *phase_out, float2 *obj_out, cudaStream_t s) {
    const size_t P = (size_t)a.N * a.N;
    UpArgs u;
    u.f = factor;
    u.osum = a.Osum;
    u.tw = a.tw;
    u.twf = tab;
    u.U = T;
    u.W = T + (size_t)factor * P;
    u.spec = u.W + P;
    u.phase = phase_out;
    u.obj = obj_out;
    // FFT2(Osum) = N^2 sum_k C_k and Osum = N^2 n_bf O, so O_up = IFFT2(...) / (N^4 n_bf)
    u.scale = (float)(1.0 / ((double)P * (double)P * (double)a.n_bf));
    switch (a.N) {
        case 32: return upsample_n<32>(u, s);
        case 64: return upsample_n<64>(u, s);
        case 128: return upsample_n<128>(u, s);
        case 256: return upsample_n<256>(u, s);
        case 512: return upsample_n<512>(u, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssb
