// Device building blocks shared by the SSB kernels: complex helpers, a batched
// shared-memory Stockham FFT (G-cache builder), the soft aperture, the per-element SSB2
// and SSB1 corrections, the zero-transfer column tests and the atan2 used for phases.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ssb {

// Per-pixel phase sums S1 (8 bytes per pixel) are kept as a pair of floats hi + lo updated
// by an exact two-sum: about 48 significant bits without float64 arithmetic (the float64
// pipe of this GPU is narrow; float64 additions measured 0.9 % slower per objective).

// s = (hi, lo) += v: hi takes the float32 sum, lo the exact rounding error of that sum
// (Knuth's two-sum, six additions, valid for any magnitudes).
__device__ __forceinline__ float2 df_add(float2 s, float v) {
    const float hi = s.x + v;
    const float bv = hi - s.x;
    const float err = (s.x - (hi - bv)) + (v - bv);
    return make_float2(hi, s.y + err);
}

// S1 of pixel i (stored as float2 hi, lo) as a float64 value
__device__ __forceinline__ double s1_value(const double *S1, int i) {
    const float2 e = reinterpret_cast<const float2 *>(S1)[i];
    return (double)e.x + (double)e.y;
}

__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cconj(float2 a) { return make_float2(a.x, -a.y); }

// Twiddle exp(S * 2 pi i m / N) from a table tw[m] = exp(+2 pi i m / N), 0 <= m < N.
template <int S>
__device__ __forceinline__ float2 twid(const float2 *tw, int m) {
    float2 w = tw[m];
    return S > 0 ? w : cconj(w);
}

// In-place 4-point DFT with exponent sign S (+1 inverse, -1 forward).
template <int S>
__device__ __forceinline__ void dft4(float2 &a0, float2 &a1, float2 &a2, float2 &a3) {
    float2 t0 = cadd(a0, a2), t1 = csub(a0, a2), t2 = cadd(a1, a3), d = csub(a1, a3);
    float2 t3 = S > 0 ? make_float2(-d.y, d.x) : make_float2(d.y, -d.x);  // (i S) d
    a0 = cadd(t0, t2);
    a2 = csub(t0, t2);
    a1 = cadd(t1, t3);
    a3 = csub(t1, t3);
}

// NF length-N transforms held in shared memory at buf0 + f * LD (f < NF), computed by
// all nthr threads of the block with a Stockham autosort schedule: radix-4 passes, then
// one radix-2 pass when log2 N is odd.  Pass with span Ns and radix R: butterfly j
// reads x[j + r N/R], applies exp(S 2 pi i r (j mod Ns)/(Ns R)), takes the R-point DFT
// and writes y[(j - j mod Ns) R + j mod Ns + r Ns] (Stockham's self-sorting FFT, as in
// Govindaraju et al., "High performance discrete Fourier transforms on graphics
// processors", SC 2008).  Unnormalised.  Returns 0 if the result is in buf0, 1 if in buf1.
// Every thread of the block must call it (it synchronises the block after each pass).
template <int N, int S>
__device__ int fft_batch_smem(float2 *buf0, float2 *buf1, int NF, int LD, const float2 *tw,
                              int tid, int nthr) {
    float2 *src = buf0, *dst = buf1;
    int which = 0;
    int Ns = 1;
#pragma unroll 1
    for (; Ns * 4 <= N; Ns *= 4) {
        constexpr int nb = N / 4;
        const int step = N / (Ns * 4);
        for (int idx = tid; idx < NF * nb; idx += nthr) {
            const int f = idx / nb, j = idx - f * nb;
            const float2 *s = src + f * LD;
            float2 *d = dst + f * LD;
            const int k = j & (Ns - 1);
            float2 v0 = s[j], v1 = s[j + nb], v2 = s[j + 2 * nb], v3 = s[j + 3 * nb];
            if (Ns > 1) {
                const int m = k * step;
                v1 = cmul(v1, twid<S>(tw, m));
                v2 = cmul(v2, twid<S>(tw, 2 * m));
                v3 = cmul(v3, twid<S>(tw, 3 * m));
            }
            dft4<S>(v0, v1, v2, v3);
            const int o = (j - k) * 4 + k;
            d[o] = v0;
            d[o + Ns] = v1;
            d[o + 2 * Ns] = v2;
            d[o + 3 * Ns] = v3;
        }
        __syncthreads();
        float2 *t = src; src = dst; dst = t;
        which ^= 1;
    }
    if (Ns < N) {  // radix-2 pass, Ns == N/2
        constexpr int nb = N / 2;
        for (int idx = tid; idx < NF * nb; idx += nthr) {
            const int f = idx / nb, j = idx - f * nb;
            const float2 *s = src + f * LD;
            float2 *d = dst + f * LD;
            float2 v0 = s[j], v1 = cmul(s[j + nb], twid<S>(tw, j));
            d[j] = cadd(v0, v1);
            d[j + nb] = csub(v0, v1);
        }
        __syncthreads();
        which ^= 1;
    }
    return which;
}

// Per-trial constants of the correction (float32 copies of host float64 values).
struct TrialConst {
    float cr, sr;       // cos, sin of the scan rotation
    float semi;         // aperture semiangle (rad)
    float inv_dalpha;   // 1 / detector sampling (1/rad)
    float inner2;       // |alpha|^2 at or below which a(alpha) = 1 (negative: never)
    float outer2;       // |alpha|^2 at or above which a(alpha) = 0
    float lam_q;        // lambda / (N * scan step): |lambda Q'| per frequency bin (rad)
    float zero_r;       // outer aperture radius with a 1e-4 margin (rad), see column_zero
};

// True when both shifted apertures vanish on the whole scan-frequency column sx of BF
// pixel alpha_k = (ax, ay), so that the column's SSB2 transfer is exactly zero.  As sy
// runs, lambda Q'(sx, sy) traces the line sx lam_q (cos, sin) + t (-sin, cos); its
// distance from alpha_k is |u - sx lam_q| and from -alpha_k |u + sx lam_q|, with
// u = ax cos + ay sin.  Both distances at least zero_r (the outer radius plus a 1e-4
// margin, far above float32 rounding) put every element outside both apertures.
__device__ __forceinline__ bool column_zero(int sx, float ax, float ay, const TrialConst &tc) {
    const float u = fmaf(ax, tc.cr, ay * tc.sr);
    const float o = tc.lam_q * (float)sx;
    return fabsf(u - o) >= tc.zero_r && fabsf(u + o) >= tc.zero_r;
}
// The SSB1 transfer needs only the aperture at alpha_k - lambda Q': the column is zero when
// its line passes at least zero_r from alpha_k.
__device__ __forceinline__ bool column_zero1(int sx, float ax, float ay, const TrialConst &tc) {
    const float u = fmaf(ax, tc.cr, ay * tc.sr);
    return fabsf(u - tc.lam_q * (float)sx) >= tc.zero_r;
}

// Amplitudes below this are exactly zero transfer: a scan grid commensurate with the
// detector can put a shifted aperture exactly on its outer edge, where the unit-modulus
// normalisation would otherwise let rounding choose between zero and a full-size term.
constexpr float kApertureFloor = 1.0f / 65536.0f;

// Soft aperture a(alpha) = clip((alpha_c - |alpha|)/d_alpha + 1/2, 0, 1), from |alpha|^2,
// with exact inside/outside shortcuts: a = 1 for
// |alpha| <= alpha_c - d_alpha/2 and a = 0 for |alpha| >= alpha_c + d_alpha/2 need no
// square root; the rim between them takes the full expression and the zero floor.
__device__ __forceinline__ float aperture_r2(float r2, const TrialConst &tc) {
    if (r2 >= tc.outer2) return 0.0f;
    if (r2 <= tc.inner2) return 1.0f;
    const float r = r2 > 0.0f ? r2 * rsqrtf(r2) : 0.0f;
    const float a = fminf(fmaxf(fmaf(tc.semi - r, tc.inv_dalpha, 0.5f), 0.0f), 1.0f);
    return a < kApertureFloor ? 0.0f : a;
}


// Squared distances |alpha_k -+ lambda Q'|^2 along one scan-frequency column sx, without
// forming lambda Q': with (u, w) = alpha_k in the frame rotated by the scan rotation and
// q = lam_q, |alpha_k -+ lambda Q'|^2 = |alpha_k|^2 + q^2 (sx^2 + sy^2) -+ 2 q (u sx + w sy).
// The caller fills base = |alpha_k|^2 + q^2 sx^2, p0 = q u sx, qw = q w and q2 = q^2 once
// per column; each element then costs five float operations.
struct ColGeom {
    float base, p0, qw, q2;
};

__device__ __forceinline__ ColGeom col_geom(int sx, float ax, float ay, const TrialConst &tc) {
    const float q = tc.lam_q, fsx = (float)sx;
    const float u = fmaf(ax, tc.cr, ay * tc.sr), w = fmaf(ay, tc.cr, -ax * tc.sr);
    ColGeom cg;
    cg.q2 = q * q;
    cg.base = fmaf(cg.q2, fsx * fsx, fmaf(ax, ax, ay * ay));
    cg.p0 = q * u * fsx;
    cg.qw = q * w;
    return cg;
}

// SSB2 correction of one G value at signed bins (sx, sy): C = G conj(Gamma)/|Gamma|, 0 where
// Gamma = 0.  With chi quadratic, chi(alpha_k -+ lambda Q') = chi(alpha_k) + chi(lambda Q')
// -+ B with B = 2 pi alpha_k^T M Q' linear in Q (M the aberration matrix), so
//   Gamma_k = a_k e^{-iB} [a_- e^{i chiQ} - a_+ e^{-i chiQ}] = a_k e^{-iB} D,
//   D = (a_- - a_+) cos chiQ + i (a_- + a_+) sin chiQ,
// and conj(Gamma)/|Gamma| = e^{iB} conj(D)/|D| (an exact rewriting).  chiQ comes from the
// per-trial table E = e^{i chiQ}; B is carried exactly as a 32-bit fixed-point fraction of
// a turn, b_x sx + b_y sy mod 2^32, so its range reduction is exact.  The per-column terms
// come from the caller: the column geometry cg and phx = b_x sx; fsy is the signed bin sy
// as a float, sy itself enters the exact turn-fraction phase; DC (C(0) = G(0)) and
// a_k = 0 are handled there too.
__device__ __forceinline__ float2 correct_ssb2(float2 g, float fsy, int sy, float2 e,
                                                const ColGeom &cg, uint32_t phx, uint32_t by,
                                                const TrialConst &tc) {
    const float b = fmaf(cg.q2, fsy * fsy, cg.base);
    const float pq = fmaf(cg.qw, fsy, cg.p0);
    const float am = aperture_r2(fmaf(-2.0f, pq, b), tc);
    const float ap = aperture_r2(fmaf(2.0f, pq, b), tc);
    const float dx = (am - ap) * e.x, dy = (am + ap) * e.y;
    const float d2 = fmaf(dx, dx, dy * dy);
    if (!(d2 > 0.0f)) return make_float2(0.0f, 0.0f);  // zero transfer
    const uint32_t ph = phx + by * (uint32_t)sy;
    float sb, cb;
    __sincosf((float)(int32_t)ph * 1.4629180792671596e-09f, &sb, &cb);  // 2 pi ph / 2^32
    const float inv = rsqrtf(d2);
    return cmul(g, cmul(make_float2(dx * inv, -dy * inv), make_float2(cb, sb)));
}

// SSB1 correction of one G value, F = e^{iB} conj(E) where a(alpha_k - lambda Q') > 0 and 0
// elsewhere (the caller handles DC and a_k = 0): chi(alpha_k) - chi(alpha_k - lambda Q') =
// B - chi(lambda Q'), the same separable terms as the SSB2 correction.
__device__ __forceinline__ float2 correct_ssb1(float2 g, float fsy, int sy, float2 e,
                                                const ColGeom &cg, uint32_t phx, uint32_t by,
                                                const TrialConst &tc) {
    const float b = fmaf(cg.q2, fsy * fsy, cg.base);
    const float pq = fmaf(cg.qw, fsy, cg.p0);
    if (!(aperture_r2(fmaf(-2.0f, pq, b), tc) > 0.0f)) return make_float2(0.0f, 0.0f);
    const uint32_t ph = phx + by * (uint32_t)sy;
    float sb, cb;
    __sincosf((float)(int32_t)ph * 1.4629180792671596e-09f, &sb, &cb);  // 2 pi ph / 2^32
    return cmul(g, cmul(make_float2(cb, sb), cconj(e)));
}


// Phase atan2(y, x) in (-pi, pi]: octant reduction to a = min/max in [0, 1], an odd
// degree-15 polynomial in a fitted to atan on [0, 1] for this library by iteratively
// reweighted least squares (float32 Horner error 1.35e-7 rad), then the unfolding
// pi/2 - p, pi - p and the sign of y.  With the approximate division (2 ulp) and the
// unfolding's rounding the whole function is within 4e-7 rad of atan2 for |x|, |y| normal
// floats below 2^126 or zero (checked on the GPU against float64 atan2).
__device__ __forceinline__ float fast_atan2(float y, float x) {
    const float ax = fabsf(x), ay = fabsf(y);
    const float mx = fmaxf(ax, ay), mn = fminf(ax, ay);
    // 0/0 -> 0 without a branch (mx below the smallest normal float is taken as that value)
    const float a = __fdividef(mn, fmaxf(mx, 1.17549435e-38f));
    const float s = a * a;
    float p = -4.054552875e-03f;
    p = fmaf(p, s, 2.186291292e-02f);
    p = fmaf(p, s, -5.591227114e-02f);
    p = fmaf(p, s, 9.642194211e-02f);
    p = fmaf(p, s, -1.390862912e-01f);
    p = fmaf(p, s, 1.994656622e-01f);
    p = fmaf(p, s, -3.332985938e-01f);
    p = fmaf(p, s, 9.999993443e-01f);
    float r = p * a;
    if (ay > ax) r = 1.57079632679489662f - r;
    if (x < 0.0f) r = 3.14159265358979324f - r;
    return copysignf(r, y);
}

}  // namespace ssb
