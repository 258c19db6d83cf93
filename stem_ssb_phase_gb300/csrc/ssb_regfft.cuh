// Register-resident FFT of length N by a group of T = N/E threads, each holding E points
// (E = 8 or 16; with E = 16 one warp holds a 512-point transform and only warp-level
// synchronisation is needed).
//
// Thread j of the group holds x[j + T r] (r = 0..E-1) on entry and X[j + T r] on exit
// (natural order on both sides).  Passes follow Stockham's self-sorting schedule (radix 8,
// then a final radix 4 or 2 when log2 N is not a multiple of 3); between passes the
// points go through a shared-memory buffer of PadLen<N> complex values per group.
// A radix-R pass has N/R butterflies: butterfly b reads x[b + (N/R) q], twists it by
// exp(S 2 pi i q (b mod Ns) / (Ns R)), takes the R-point DFT and writes
// y[(b - b mod Ns) R + b mod Ns + Ns q].  Thread j runs butterflies b = j + T m,
// m < E/R, whose inputs are exactly its registers m + (E/R) q, so no shuffle is needed,
// and the last pass leaves its outputs in registers in natural order.
#pragma once

#include "ssb_device.cuh"

namespace ssb {

// Padded shared-memory slot of complex value i: one spare slot every 16.  For 64-bit
// accesses (16 lanes per 128-byte wavefront) this keeps the exchange reads, the first
// pass's writes and the twiddle reads free of bank conflicts; the second pass's writes
// (span 8) take two-way conflicts.  Among paddings i + sum c_s (i >> s) none does better
// for the 512- and 256-point transforms, and a padding keeps every access of a pass at a
// constant offset from one per-thread base.  (An XOR swizzle that removes the remaining
// conflicts too measured no faster: its offsets cost instructions.)
constexpr int kPadShift = 4;
__device__ __forceinline__ int lay(int i) { return i + (i >> kPadShift); }
template <int N>
struct PadLen {
    static constexpr int value = N + (N >> kPadShift);
};
// lay(j + T r) from base = lay(j), for j < T and T a multiple of 16
template <int T>
__device__ __forceinline__ int lay_seq(int base, int r) { return base + lay(T * r); }
// lay(o + Ns q) from base = lay(o): o a multiple of 8 when Ns = 1, o mod 16 < 8 when Ns = 8
__device__ __forceinline__ int lay_out(int base, int Ns, int q) { return base + lay(Ns * q); }
// lay(i + c) = lay(i) + lay_shift(c) for c a multiple of 16
__device__ __forceinline__ int lay_shift(int c) { return lay(c); }

template <int N, int E>
struct RegFFT {
    static constexpr int T = N / E;
    static constexpr int SMEM = PadLen<N>::value;  // complex values per group
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
// twp is the twiddle table in the same layout: twp[lay(m)] = exp(+2 pi i m / N).
// Non-final passes are radix 8 with Ns = 1 or 8; with T a multiple of 16 every slot a
// thread touches is a constant offset from one per-thread base (lay_seq, lay_out and
// lay_shift), otherwise each slot is computed in full.
template <int N, int E, int R, int S, bool LAST, typename Bar>
__device__ __forceinline__ void stockham_pass(float2 (&v)[E], float2 *sm, const float2 *twp,
                                              int j, int Ns, Bar bar) {
    constexpr int T = N / E;
    constexpr int PER = E / R;  // butterflies per thread
    constexpr bool kSeq = T % 16 == 0;
    // outputs of butterfly m start at (b - k) R + k = o0 + R T m (k = j mod Ns for Ns <= T)
    const int k0 = j & (Ns - 1);
    const int wbase = lay((j - k0) * R + k0);
#pragma unroll
    for (int m = 0; m < PER; ++m) {
        const int b = j + T * m;
        const int k = b & (Ns - 1);
        float2 u[R];
#pragma unroll
        for (int q = 0; q < R; ++q) u[q] = v[m + PER * q];
        if (Ns > 1) {
            // one table read, the other twiddles as products of it (depth 3 for radix 8)
            const float2 w1 = twid<S>(twp, lay(k * (N / (Ns * R))));
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
#pragma unroll
            for (int q = 0; q < R; ++q) {
                const int a = kSeq ? lay_out(wbase, Ns, q) + lay_shift(R * T * m)
                                   : lay((b - k) * R + k + Ns * q);
                sm[a] = u[q];
            }
        }
    }
    if (!LAST) {
        bar();
        const int rbase = lay(j);
#pragma unroll
        for (int r = 0; r < E; ++r) v[r] = sm[kSeq ? lay_seq<T>(rbase, r) : lay(j + T * r)];
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
