// Register-resident FFT of length N by a group of T = N/E threads, each holding E points
// (E = 8 or 16; with E = 16 one warp holds a 512-point transform and only warp-level
// synchronisation is needed).
//
// Thread j of the group holds x[j + T r] (r = 0..E-1) on entry and X[j + T r] on exit
// (natural order on both sides).  Passes follow Stockham's self-sorting schedule (radix 8,
// then a final radix 4 or 2 when log2 N is not a multiple of 3); between passes the
// points go through a padded shared-memory buffer of N + N/8 complex values per group.
// A radix-R pass has N/R butterflies: butterfly b reads x[b + (N/R) q], twists it by
// exp(S 2 pi i q (b mod Ns) / (Ns R)), takes the R-point DFT and writes
// y[(b - b mod Ns) R + b mod Ns + Ns q].  Thread j runs butterflies b = j + T m,
// m < E/R, whose inputs are exactly its registers m + (E/R) q, so no shuffle is needed,
// and the last pass leaves its outputs in registers in natural order.
#pragma once

#include "ssb_device.cuh"

namespace ssb {

// Padded shared-memory index: one spare slot every 8 complex values keeps the pass
// exchanges (and twiddle reads) free of most bank conflicts for 64-bit accesses.
__device__ __forceinline__ int padx(int i) { return i + (i >> 3); }

template <int N, int E>
struct RegFFT {
    static constexpr int T = N / E;
    static constexpr int SMEM = N + N / 8;  // complex values per group
    static constexpr int LOG2N = N == 16 ? 4 : N == 32 ? 5 : N == 64 ? 6 : N == 128 ? 7 : N == 256 ? 8 : 9;
    static constexpr int N8 = LOG2N / 3;        // radix-8 passes
    static constexpr int TAIL = LOG2N - 3 * N8; // 0, 1 (radix 2) or 2 (radix 4)
};

// 8-point DFT in registers with exponent sign S, by one radix-2 split into two 4-point DFTs.
template <int S>
__device__ __forceinline__ void dft8(float2 (&v)[8]) {
    constexpr float R2 = 0.70710678118654752f;
    float2 a[4], b[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        a[q] = cadd(v[q], v[q + 4]);
        b[q] = csub(v[q], v[q + 4]);
    }
    // b_q *= exp(S 2 pi i q / 8)
    b[1] = make_float2(R2 * (b[1].x - S * b[1].y), R2 * (b[1].y + S * b[1].x));
    b[2] = S > 0 ? make_float2(-b[2].y, b[2].x) : make_float2(b[2].y, -b[2].x);
    b[3] = make_float2(R2 * (-b[3].x - S * b[3].y), R2 * (-b[3].y + S * b[3].x));
    dft4<S>(a[0], a[1], a[2], a[3]);
    dft4<S>(b[0], b[1], b[2], b[3]);
    v[0] = a[0]; v[1] = b[0]; v[2] = a[1]; v[3] = b[1];
    v[4] = a[2]; v[5] = b[2]; v[6] = a[3]; v[7] = b[3];
}

// One Stockham pass of radix R (8, 4 or 2) over the group's registers, span Ns.
// twp is the padded twiddle table: twp[padx(m)] = exp(+2 pi i m / N).
template <int N, int E, int R, int S, bool LAST, typename Bar>
__device__ __forceinline__ void stockham_pass(float2 (&v)[E], float2 *sm, const float2 *twp,
                                              int j, int Ns, Bar bar) {
    constexpr int T = N / E;
    constexpr int PER = E / R;  // butterflies per thread
#pragma unroll
    for (int m = 0; m < PER; ++m) {
        const int b = j + T * m;
        const int k = b & (Ns - 1);
        float2 u[R];
#pragma unroll
        for (int q = 0; q < R; ++q) u[q] = v[m + PER * q];
        if (Ns > 1) {
            // one table read, the other twiddles as products of it (depth 3 for radix 8)
            const float2 w1 = twid<S>(twp, padx(k * (N / (Ns * R))));
            if (R == 2) {
                u[1] = cmul(u[1], w1);
            } else {
                const float2 w2 = cmul(w1, w1);
                const float2 w3 = cmul(w2, w1);
                u[1] = cmul(u[1], w1);
                u[2] = cmul(u[2], w2);
                u[3] = cmul(u[3], w3);
                if (R == 8) {
                    const float2 w4 = cmul(w2, w2);
                    const float2 w5 = cmul(w4, w1);
                    const float2 w6 = cmul(w3, w3);
                    const float2 w7 = cmul(w4, w3);
                    u[4] = cmul(u[4], w4);
                    u[5] = cmul(u[5], w5);
                    u[6] = cmul(u[6], w6);
                    u[7] = cmul(u[7], w7);
                }
            }
        }
        if (R == 8) {
            float2 w[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) w[q] = u[q];
            dft8<S>(w);
#pragma unroll
            for (int q = 0; q < 8; ++q) u[q] = w[q];
        } else if (R == 4) {
            dft4<S>(u[0], u[1], u[2], u[3]);
        } else {
            const float2 t = u[1];
            u[1] = csub(u[0], t);
            u[0] = cadd(u[0], t);
        }
        if (LAST) {
            // final pass: Ns = N/R, output index b + Ns q = j + T (m + PER q)
#pragma unroll
            for (int q = 0; q < R; ++q) v[m + PER * q] = u[q];
        } else {
            const int o = (b - k) * R + k;
#pragma unroll
            for (int q = 0; q < R; ++q) sm[padx(o + Ns * q)] = u[q];
        }
    }
    if (!LAST) {
        bar();
#pragma unroll
        for (int r = 0; r < E; ++r) v[r] = sm[padx(j + T * r)];
        bar();
    }
}

// Full transform.  sm: this group's N + N/8 complex scratch; twp: padded twiddle table.
template <int N, int E, int S, typename Bar>
__device__ __forceinline__ void reg_fft(float2 (&v)[E], float2 *sm, const float2 *twp, int j,
                                        Bar bar) {
    using F = RegFFT<N, E>;
    int Ns = 1;
    if (F::TAIL == 0) {
#pragma unroll
        for (int p = 0; p < F::N8 - 1; ++p) {
            stockham_pass<N, E, 8, S, false>(v, sm, twp, j, Ns, bar);
            Ns *= 8;
        }
        stockham_pass<N, E, 8, S, true>(v, sm, twp, j, Ns, bar);
    } else {
#pragma unroll
        for (int p = 0; p < F::N8; ++p) {
            stockham_pass<N, E, 8, S, false>(v, sm, twp, j, Ns, bar);
            Ns *= 8;
        }
        if (F::TAIL == 2)
            stockham_pass<N, E, 4, S, true>(v, sm, twp, j, Ns, bar);
        else
            stockham_pass<N, E, 2, S, true>(v, sm, twp, j, Ns, bar);
    }
}

}  // namespace ssb
