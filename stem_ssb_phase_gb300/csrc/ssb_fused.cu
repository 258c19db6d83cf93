// Persistent, ticket-scheduled evaluation of the exact SSB objective, for both transfers.
//
// The pages locate the cost of the exact objective in the column -> row intermediate that
// is written and re-read through global memory ("Later SSB performance checkpoints",
// 2026-09-11 checkpoints: about 18.8 GB per evaluation).  Here that intermediate stays in
// L2: BF planes are processed in batches of Bk planes through a ring of D batch slots
// (tens of MB), by one persistent kernel on every SM.
//
// SSB2 (the normalised two-sideband transfer) does half the work, exactly.  Off DC and
// the Nyquist lines its corrected spectrum is anti-Hermitian, C(-Q) = -conj C(Q) (the
// relation of "SSB performance notes", 257-row intermediate prototype).  So only the
// N/2+1 half-plane columns are corrected and column-transformed; each row is rebuilt from
// them as
//     Zfull(ry, N - nx) = -conj Z(ry, nx) + 2 (-1)^ry conj h(nx),   1 <= nx < N/2,
// where h(nx) = (C(N/2, nx) + conj C(N/2, N - nx)) / 2 is the Hermitian part of the
// Nyquist row, whose bins have no negative-frequency partner (the violation the pages
// isolate).  Columns 0 and N/2 are transformed in full.  The result equals the plain
// two-dimensional inverse transform in exact arithmetic.  SSB1 (the literal
// single-sideband factor) has no such symmetry: all N columns, full complex rows.
//
// Tasks (ticket order, phase p = [columns of batch p, rows of batch p-1]):
//   column task (batch b, plane, CW columns, kColsPerWarp per warp): G load, correction,
//       column IFFT, store to the ring slot, one column contiguous, Z[slot][plane][nx][ry]
//       (SSB2 columns 0 < nx < N/2 as Z - (-1)^ry h(nx), the form the row rebuild uses);
//       columns with exactly zero transfer store zeros without the work; for SSB2 the
//       task that completes a plane's column pass also transforms its Nyquist-row term;
//   row task (batch b, RT rows): for each plane of the batch, rebuild the full rows (SSB2)
//       or take them as they are (SSB1), row IFFT, phi = atan2, accumulate; then add the
//       batch's per-pixel sums into S1 (a float pair per pixel, exact two-sum; S2 and the
//       object in float64) in batch order.
// A block takes its next ticket when its current task has finished its work, just before
// the task's completion fence (the two round trips overlap).  (Taking a column ticket any
// earlier, even just before the task's ring writes, measured about 14 % slower overall.)  A task waits only for tasks holding smaller
// tickets, so the schedule cannot deadlock whatever the number of resident blocks.
// Every wait is bounded; on timeout the kernel raises an error flag, all waits stop and
// the host reports SSB_ERR_TIMEOUT.
#include <algorithm>
#include <cstring>
#include <mutex>

#include <cuda.h>           // CUtensorMap (the encode call is resolved at run time)
#include <cudaTypedefs.h>

#include "ssb_device.cuh"
#include "ssb_internal.h"
#include "ssb_regfft.cuh"

namespace ssb {

#ifndef SSB_FUSED_THREADS
#define SSB_FUSED_THREADS 256
#endif
constexpr int kFusedThreads = SSB_FUSED_THREADS;  // threads per block (4 or 8 warps)
constexpr int kFusedBlocksPerSM = 512 / kFusedThreads;
constexpr int kPts = 16;                    // points per thread in every transform
#ifndef SSB_COLS_PER_WARP
#define SSB_COLS_PER_WARP 2
#endif
constexpr int kColsPerWarp = SSB_COLS_PER_WARP;  // columns each transform group takes per task
constexpr unsigned kWaitLimit = 1u << 24;  // polls of ~0.1-1 us each before giving up

struct FusedParams {
    const float2 *G;      // [n_bf][H][N]
    const float2 *Et;     // [N (nx)][N (ny)] e^{i chi(lambda Q')}
    const float4 *kgeo;   // per BF (alpha_x, alpha_y, a_k, 0)
    const uint2 *kturn;   // per BF bilinear phase slopes
    const float2 *tw;     // [N] exp(+2 pi i m/N)
    float2 *Z;            // ring [D][Bk][H][N]: column-pass output, one column contiguous
    float2 *hrow;         // ring [D][Bk][LDZ], Nyquist-row Hermitian parts
    float2 *rrow;         // ring [D][Bk][N/2]: Rp(2j) + i Rp(2j+1), Rp the Nyquist-row term
    double *S1;           // [P] 8 bytes per pixel, stored as float2 (hi, lo): see df_add
    double *S2g;          // [row tasks]
    double2 *Osum;        // [P] (object redraw only)
    unsigned *sync;       // ticket, col_done[nbatch], plane_free[nbatch][Bk],
                          // h_cnt[nbatch][Bk], chain[row tasks]
    unsigned *err;        // error word, cleared once per library call (shared by the
                          // evaluations of a call, so a timeout stays raised)
    int n_bf, Bk, nbatch;
    int D;                // ring slots (batches in flight)
    unsigned wait_limit;  // polls before a wait gives up (kWaitLimit unless a test lowers it)
    int stall;            // test hook: row tasks wait for a count that is never reached
    TrialConst tc;
};

// Shapes of the fused kernel.  SSB2 (anti-Hermitian spectrum): the N/2 + 1 half-plane
// columns, rows rebuilt by the C2R split into N/2-point transforms.  SSB1 (no symmetry):
// all N columns and full N-point complex row transforms.
template <int N, bool SSB1 = false>
struct FusedShape {
    static constexpr int T = N / kPts;              // threads per transform (rows and columns)
    static constexpr int GROUPS = kFusedThreads / T;  // transforms per block
    static constexpr int H = SSB1 ? N : N / 2 + 1;  // columns corrected and column-transformed
    static constexpr int M = SSB1 ? N : N / 2;      // row transform length
    static constexpr int RE = SSB1 ? kPts : 8;      // row transform points per thread (M / T)
    static constexpr int CW = GROUPS * kColsPerWarp;  // columns per column task
    // rows per row task (multiple of 4), one per transform group.  (Two rows per warp --
    // 16-row tasks with 128-bit tile reads and interleaved row transforms -- measured slower
    // in every form tried: whole-batch tasks release ring planes too late for the column
    // tasks, half-batch tasks pay a second ordered update per batch, and the shared reads
    // save only about 5 % of a row's instructions.)
    static constexpr int RT = GROUPS < N ? GROUPS : N;
    // Column tasks per plane.  (For SSB2 at N = 512 the last of the 17 takes column N/2
    // alone; moving that column into the task that completes the plane, beside the
    // Nyquist-row term, measured slower: it lengthens each plane's critical path.)
    static constexpr int CT = (H + CW - 1) / CW;
    static constexpr int NR = N / RT;               // row tasks per trial
    static constexpr int SMF = RegFFT<N, kPts>::SMEM;  // FFT scratch per group
    static constexpr int LDZ = (N / 2 + 1 + 7) / 8 * 8;  // h row stride (64 B multiple)
    static constexpr int RC = RT / 2;               // 16-byte chunks per column segment
    // staged column-segment stride: SSB2 pads by one chunk; SSB1 (twice the columns) keeps
    // segments dense and places chunk c of column nx at c xor ((nx >> SWS) mod RC) instead.
    // With 8-row segments two columns share a 128-byte bank row, so the xor follows nx / 2:
    // 16 consecutive columns then cover 8 bank pairs (two-way conflicts, the least 16-byte
    // chunks allow).
    static constexpr int LDC = SSB1 ? RT : RT + 2;
    static constexpr int SWS = RT == 8 ? 1 : 0;
    // SSB1 with 8- or 16-row segments stages each plane with 2D tensor copies whose 64- or
    // 128-byte swizzle is exactly the chunk xor above (16-byte chunk bits 4.. of the shared
    // address xor bits 7..); boxes of BOXN columns.  Other shapes use cp.async.
    static constexpr bool TMA = SSB1 && (RT == 8 || RT == 16);
    static constexpr int BOXN = H < 256 ? H : 256;
    static constexpr int NBOX = (H + BOXN - 1) / BOXN;
    // dynamic shared memory layout, in float2 units.  A block runs one task at a time, so
    // the column task's FFT scratch and the row task's scratch + staged planes share OFF_U.
    static constexpr int SMR = RegFFT<M, RE>::SMEM;                 // row FFT scratch per group
    static constexpr int OFF_TW = 0;                                // padded twiddles
    static constexpr int OFF_TW2 = OFF_TW + (PadLen<N>::value + 1) / 2 * 2;  // N/2-point table
    static constexpr int OFF_RED = OFF_TW2 + (PadLen<N / 2>::value + 1) / 2 * 2;  // partials
    static constexpr int OFF_U = OFF_RED + 16;
    static constexpr int OFF_FFT = OFF_U;                           // column task: [GROUPS][SMF]
    static constexpr int OFF_RFFT = OFF_U;                          // row task: [GROUPS][SMR]
    // [2][TILEBUF]; tensor-copy destinations start on a 1024-byte boundary (128 float2)
    static constexpr int OFF_TILE = TMA ? (OFF_RFFT + GROUPS * SMR + 127) / 128 * 128
                                        : OFF_RFFT + (GROUPS * SMR + 1) / 2 * 2;
    static constexpr int TILEBUF = SSB1 ? H * LDC : H * LDC + M;  // segments (, Rp)
    static constexpr int U_COL = GROUPS * SMF;
    // cp.async tiles are triple-buffered (one block barrier per plane), tensor-copy tiles
    // double-buffered
    static constexpr int U_ROW = OFF_TILE - OFF_U + (TMA ? 2 : 3) * TILEBUF;
    // + 128 float2 so that the tiles can be placed on a 1024-byte boundary at run time
    static constexpr int TOTAL = OFF_U + (U_COL > U_ROW ? U_COL : U_ROW) + (TMA ? 128 : 0);
    static constexpr size_t BYTES = (size_t)TOTAL * sizeof(float2);
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int K>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(K) : "memory"); }

// mbarrier and tensor-copy helpers (shared addresses from __cvta_generic_to_shared).
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
    asm volatile("mbarrier.init.shared.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    return done != 0u;
}
// One 2D box of the tensor map into shared memory, completing on bar.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(bar) : "memory");
}

__device__ __forceinline__ void red_relaxed_add(unsigned *p, unsigned v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Release by one thread after a block barrier: the block's earlier writes become visible
// to any thread that observes the following relaxed write or reduction with an acquire.
__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ unsigned atom_add_relaxed(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_relaxed(unsigned *p, unsigned v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Called by one thread: wait until *addr >= target.  Returns false if the wait gave up
// (error flag already raised elsewhere, or the poll budget ran out, which raises it).
__device__ bool wait_at_least(const unsigned *addr, unsigned target, unsigned *err,
                              unsigned limit) {
    unsigned polls = 0;
    while (ld_acquire(addr) < target) {
        if (ld_acquire(err) != 0u) return false;
        if (++polls > limit) {
            atomicOr(err, 2u);
            return false;
        }
        __nanosleep(128);
    }
    return true;
}

// Wait until the barrier's phase with the given parity has completed.  Bounded: it gives
// up when the error flag is raised elsewhere, or raises it when the poll budget runs out.
__device__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned *err) {
    for (unsigned polls = 0; polls < kWaitLimit; ++polls) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((polls & 255u) == 255u && ld_acquire(err) != 0u) return false;
    }
    atomicOr(err, 4u);
    return false;
}

// Transforms never span warps (T <= 32), so their exchanges need only warp sync.
__device__ __forceinline__ void warp_bar() { __syncwarp(); }

// ---------------------------------------------------------------- column task

// Rp(rx) = 2 Re sum_{0 < nx < N/2} h(nx) e^{2 pi i nx rx / N}, the Nyquist-row contribution
// to Re c (times (-1)^ry), as one N/2-point complex IFFT of the packed real-output form;
// stored as Rp(2j) + i Rp(2j+1).  Run by one group of T threads.
// Every lane of the calling warp must call it (the transform synchronises the warp);
// only the group with store = true writes the result.
template <int N>
__device__ void nyquist_transform(const FusedParams &p, float2 *fsm, const float2 *twN,
                                  const float2 *twM, int slot, int kk, int j, bool store) {
    using S = FusedShape<N>;
    const float2 *h = p.hrow + ((size_t)slot * p.Bk + kk) * S::LDZ;
    float2 v[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int m = j + S::T * r, mc = S::M - m;
        const float2 hm = (m >= 1) ? __ldcg(h + m) : make_float2(0.f, 0.f);
        const float2 hc = (mc >= 1 && mc < S::M) ? __ldcg(h + mc) : make_float2(0.f, 0.f);
        const float2 a = make_float2(hm.x + hc.x, hm.y - hc.y);
        const float2 bb = cmul(make_float2(hm.x - hc.x, hm.y + hc.y), twid<+1>(twN, lay(m)));
        v[r] = make_float2(a.x - bb.y, a.y + bb.x);
    }
    reg_fft<S::M, 8, +1>(v, fsm, twM, j, warp_bar);
    if (store) {
        float2 *out = p.rrow + ((size_t)slot * p.Bk + kk) * S::M + j;
#pragma unroll
        for (int r = 0; r < 8; ++r) __stcg(out + S::T * r, v[r]);
    }
}

// One transformed column: column nx of BF plane k (plane kk of ring slot `slot`), by the
// calling thread's transform group (thread j of T).  Loads G and E, applies the correction,
// runs the column IFFT and leaves the result in v; for SSB2 also the Nyquist-row Hermitian
// part h(nx) of the mirror bin (hstore: this thread stores hval).  Groups with valid =
// false transform zeros.  Columns with exactly zero transfer (SSB2: both shifted
// apertures miss the whole column; SSB1: the aperture at alpha_k - lambda Q' does; every
// column but DC for an inactive BF pixel) skip the loads, the correction and the
// transform: the decision is uniform over the warp, and v is then zero.  Every lane of the
// warp must call it (the transform synchronises the warp).
// SSB1 column nx > N/2 reads the cache's column N - nx at the mirrored rows, conjugated
// (G(-Q) = conj G(Q)).
// For SSB2 columns 0 < nx < N/2 the Nyquist bin enters the transform as C(N/2, nx) - h(nx),
// so that the column comes out as Z(ry, nx) - (-1)^ry h(nx), the form the row rebuild
// uses (a constant added at bin N/2 adds (-1)^ry times it to output ry).  (Subtracting
// (-1)^ry h from the 512 outputs instead, after the transform, measured 0.9 % slower.)
// column_correct does the loads and the correction (returning the warp-uniform skip
// decision); column_compute adds the transform.
template <int N, bool SSB1>
__device__ __forceinline__ bool column_correct(const FusedParams &p, int k, int nx, bool valid,
                                               const float4 &geo, const uint2 &bt,
                                               float2 (&v)[kPts], float2 &hval, bool &hstore) {
    using S = FusedShape<N, SSB1>;
    constexpr int HG = N / 2 + 1;  // columns of the half-plane G cache
    const int j = threadIdx.x % S::T;
    const int sx = nx < N / 2 ? nx : nx - N;
    const bool zero = nx > 0 && (!(geo.z > 0.0f) || (SSB1 ? column_zero1(sx, geo.x, geo.y, p.tc)
                                                           : column_zero(sx, geo.x, geo.y, p.tc)));
    const bool skip = __all_sync(0xffffffffu, zero || !valid);
    hval = make_float2(0.f, 0.f);
    hstore = !SSB1 && valid && skip && j == 0 && nx >= 1 && nx < N / 2;  // h = 0 there
    if (valid && !skip) {
        const float2 *e = p.Et + (size_t)nx * N + j;
        float2 ev[kPts];
        if (!SSB1 || nx <= N / 2) {
            const float2 *g = p.G + ((size_t)k * HG + nx) * N + j;
#pragma unroll
            for (int r = 0; r < kPts; ++r) v[r] = __ldcs(g + S::T * r);
        } else {  // G(ny, nx) = conj G(N - ny, N - nx), row indices mod N
            const float2 *g = p.G + ((size_t)k * HG + (N - nx)) * N;
#pragma unroll
            for (int r = 0; r < kPts; ++r) v[r] = cconj(__ldcs(g + ((N - j - S::T * r) & (N - 1))));
        }
#pragma unroll
        for (int r = 0; r < kPts; ++r) ev[r] = __ldcg(e + S::T * r);  // L2 only: 0.2 % faster than via L1
        const ColGeom cg = col_geom(sx, geo.x, geo.y, p.tc);
        const float fj = (float)j;
        const uint32_t phx = bt.x * (uint32_t)sx;
        const bool active = geo.z > 0.0f;  // a(alpha_k) = 0: only the DC term survives
#pragma unroll
        for (int r = 0; r < kPts; ++r) {
            const int ny = j + S::T * r;
            // signed bin: ny for r < kPts/2 (ny < N/2), ny - N above
            const int off = S::T * r - (r >= kPts / 2 ? N : 0);
            const int sy = j + off;
            const float fsy = fj + (float)off;
            const float2 gv = v[r];
            float2 cv = make_float2(0.f, 0.f);
            if (active)
                cv = SSB1 ? correct_ssb1(gv, fsy, sy, ev[r], cg, phx, bt.y, p.tc)
                          : correct_ssb2(gv, fsy, sy, ev[r], cg, phx, bt.y, p.tc);
            if ((nx | ny) == 0) cv = gv;  // C(0) = G(0)
            if (!SSB1 && r == kPts / 2 && j == 0 && nx >= 1 && nx < N / 2) {
                // Nyquist row (ny = N/2): the mirror bin N - nx has no partner and
                // carries its own correction, at signed bins (-nx, -N/2), where the
                // column geometry has p0 negated
                const float2 em = __ldcg(p.Et + (size_t)(N - nx) * N + N / 2);
                ColGeom cm = cg;
                cm.p0 = -cg.p0;
                const float2 c2 = active ? correct_ssb2(cconj(gv), -(float)(N / 2), -N / 2, em, cm,
                                                         0u - phx, bt.y, p.tc)
                                         : make_float2(0.f, 0.f);
                hval = make_float2(0.5f * (cv.x + c2.x), 0.5f * (cv.y - c2.y));
                hstore = true;
                cv = csub(cv, hval);  // the Nyquist bin's anti-Hermitian part
            }
            v[r] = cv;
        }
    } else {
#pragma unroll
        for (int r = 0; r < kPts; ++r) v[r] = make_float2(0.f, 0.f);
    }
    return skip;
}

template <int N, bool SSB1>
__device__ __forceinline__ void column_compute(const FusedParams &p, float2 *smem, int k, int nx,
                                               bool valid, const float4 &geo, const uint2 &bt,
                                               float2 (&v)[kPts], float2 &hval, bool &hstore) {
    using S = FusedShape<N, SSB1>;
    const int grp = threadIdx.x / S::T, j = threadIdx.x % S::T;
    if (!column_correct<N, SSB1>(p, k, nx, valid, geo, bt, v, hval, hstore)) {
        reg_fft<N, kPts, +1>(v, smem + S::OFF_FFT + grp * S::SMF, smem + S::OFF_TW, j, warp_bar);
    }
}

// Store a transformed column into its ring plane (and h(nx), SSB2).  The ring lines carry
// an L2 evict-last hint: fewer of them leave L2 between their row task and the column
// task that overwrites them a few batches later, so fewer dead lines are written back
// (472 against 594 kB of DRAM writes per plane on the 2048-plane case, same time).
template <int N, bool SSB1>
__device__ __forceinline__ void column_store(const FusedParams &p, int slot, int kk, int nx,
                                             const float2 (&v)[kPts], float2 hval, bool hstore) {
    using S = FusedShape<N, SSB1>;
    const int j = threadIdx.x % S::T;
    float2 *z = p.Z + (((size_t)slot * p.Bk + kk) * S::H + nx) * N + j;
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
#pragma unroll
    for (int r = 0; r < kPts; ++r)
        asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(z + S::T * r), "f"(v[r].x),
                     "f"(v[r].y), "l"(pol) : "memory");
    if (hstore) __stcg(p.hrow + ((size_t)slot * p.Bk + kk) * S::LDZ + nx, hval);
}

// One column task: CW of the plane's H transformed columns, kColsPerWarp per transform
// group in turn.  free_word (NULL on the slot's first use) counts the row tasks of batch
// b - D that have released this plane of the ring slot; the task overwrites the plane only
// once all of them have.  Each warp reads the count when the task starts and checks it
// before its first ring write, so the load's latency hides behind the column work.
// Returns, uniform over the warp, whether the warp could write the slot.
template <int N, bool SSB1>
__device__ int column_task(const FusedParams &p, float2 *smem, int b, int idx,
                           const unsigned *free_word, unsigned *err) {
    using S = FusedShape<N, SSB1>;
    const int tid = threadIdx.x, grp = tid / S::T, lane = tid & 31;
    const int kk = idx / S::CT, ct = idx - kk * S::CT;
    const int k = b * p.Bk + kk;
    const int slot = b % p.D;
    unsigned freed = (unsigned)S::NR;
    if (lane == 0 && free_word) freed = ld_acquire(free_word);
    const float4 geo = __ldg(p.kgeo + k);
    const uint2 bt = __ldg(p.kturn + k);
    int ok = 1;
#pragma unroll 1
    for (int c = 0; c < kColsPerWarp; ++c) {
        const int nx = ct * S::CW + c * S::GROUPS + grp;
        const bool valid = nx < S::H;
        float2 v[kPts];
        float2 hval;
        bool hstore;
        column_compute<N, SSB1>(p, smem, k, nx, valid, geo, bt, v, hval, hstore);
        if (c == 0) {
            if (lane == 0 && freed < (unsigned)S::NR)
                ok = wait_at_least(free_word, (unsigned)S::NR, err, p.wait_limit);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();  // the warp's ring writes follow lane 0's acquire
        }
        if (valid && ok) column_store<N, SSB1>(p, slot, kk, nx, v, hval, hstore);
    }
    return ok;
}

// ---------------------------------------------------------------- row task

// Start the asynchronous copy of one plane's RT-row segment of every transformed column
// (RT consecutive values, contiguous in the column-major ring) and, for SSB2, of its
// Nyquist terms h and of its Nyquist-row transform Rp.  SSB1 places 16-byte chunk c of
// column nx at chunk c xor ((nx >> SWS) mod RC) of the column's dense segment.
template <int N, bool SSB1>
__device__ __forceinline__ void row_issue(const FusedParams &p, int slot, int kk, int ry0,
                                          float2 *buf) {
    using S = FusedShape<N, SSB1>;
    const float2 *zsrc = p.Z + ((size_t)slot * p.Bk + kk) * S::H * N + ry0;
    for (int e = threadIdx.x; e < S::H * S::RC; e += kFusedThreads) {
        const int nx = e / S::RC, c = e - nx * S::RC;
        const int cd = SSB1 ? (c ^ ((nx >> S::SWS) & (S::RC - 1))) : c;
        cp_async16(buf + nx * S::LDC + 2 * cd, zsrc + (size_t)nx * N + 2 * c);
    }
    if (SSB1) {
        cp_async_commit();
        return;
    }
    const float2 *rsrc = p.rrow + ((size_t)slot * p.Bk + kk) * S::M;
    for (int e = threadIdx.x; e < S::M / 2; e += kFusedThreads)
        cp_async16(buf + S::H * S::LDC + 2 * e, rsrc + 2 * e);
    cp_async_commit();
}

// Tensor-copy staging of one SSB1 plane (one thread): NBOX boxes of BOXN columns x RT rows
// of the ring, swizzled by the copy itself, completing on bar.
template <int N, bool SSB1>
__device__ __forceinline__ void row_issue_tma(const FusedParams &p, const CUtensorMap *map,
                                              int slot, int kk, int ry0, float2 *buf,
                                              uint32_t bar) {
    using S = FusedShape<N, SSB1>;
    // the buffer was last used through ordinary loads and stores
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_expect_tx(bar, (unsigned)(S::TILEBUF * sizeof(float2)));
    const int row0 = (slot * p.Bk + kk) * S::H;
#pragma unroll
    for (int bx = 0; bx < S::NBOX; ++bx)
        tma_load_2d(smem_u32(buf + bx * S::BOXN * S::RT), map, ry0, row0 + bx * S::BOXN, bar);
}

// Row ry of the corrected image, split by symmetry (exact):
//   Im c = real IFFT of Y(m) = -i (Z(m) - s h(m)) (0 < m < N/2; the ring already holds
//          Z(m) - s h(m) for these columns, see column_correct), Y(0) = Im Z(0),
//          Y(N/2) = Im Z(N/2), done as one N/2-point complex IFFT of
//          V(m) = Y(m) + conj Y(N/2-m) + i (Y(m) - conj Y(N/2-m)) e^{2 pi i m/N},
//          whose output holds Im c at pixels 2j (real part) and 2j+1 (imaginary part);
//   Re c = Re Z(0) + (-1)^rx Re Z(N/2) + s Rp(rx),   s = (-1)^ry.
// SSB1 row ry: one N-point complex IFFT of the staged row, c at pixels j + T r.
// With tensor-copy staging (S::TMA), bars holds the two tile buffers' barriers and tphase
// their completed-phase parities (bit i for buffer i), the same in every thread.
template <int N, bool OBJ, bool SSB1>
__device__ void row_task(const FusedParams &p, float2 *smem, int b, int rt, int planes,
                         unsigned *plane_free, unsigned *chain, unsigned *err, int *s_ok,
                         const CUtensorMap *map, uint32_t bars, unsigned &tphase) {
    using S = FusedShape<N, SSB1>;
    const int tid = threadIdx.x, grp = tid / S::T, j = tid % S::T;
    const int slot = b % p.D;
    const int ry0 = rt * S::RT;
    const bool active = S::RT >= S::GROUPS || grp < S::RT;  // N = 32 leaves some groups idle
    const int lr = active ? grp : 0;
    const int ry = ry0 + lr;
    const float sg = (ry & 1) ? -1.0f : 1.0f;       // (-1)^ry
    const float2 *twN = smem + S::OFF_TW;
    float2 *tiles = smem + S::OFF_TILE;
    if (S::TMA)  // tensor-copy destinations on a 1024-byte boundary (slack reserved in TOTAL)
        tiles = reinterpret_cast<float2 *>((reinterpret_cast<uintptr_t>(tiles) + 1023) &
                                           ~(uintptr_t)1023);
    float acc1[2 * 8];
    float2 acco[2 * 8];
    float acc2 = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        acc1[r] = 0.f;
        acco[r] = make_float2(0.f, 0.f);
    }
    if (S::TMA) {
        if (tid == 0) row_issue_tma<N, SSB1>(p, map, slot, 0, ry0, tiles, bars);
    } else {
        row_issue<N, SSB1>(p, slot, 0, ry0, tiles);
        if (planes > 1) row_issue<N, SSB1>(p, slot, 1, ry0, tiles + S::TILEBUF);
    }
    for (int kk = 0; kk < planes; ++kk) {
        const int buf = S::TMA ? (kk & 1) : kk % 3;
        float2 *cur = tiles + buf * S::TILEBUF;
        if (S::TMA) {
            __syncthreads();  // everyone is done with the other buffer (plane kk - 1)
            if (tid == 0 && kk + 1 < planes)
                row_issue_tma<N, SSB1>(p, map, slot, kk + 1, ry0, tiles + (buf ^ 1) * S::TILEBUF,
                                       bars + 8u * (buf ^ 1));
            mbar_wait(bars + 8u * buf, (tphase >> buf) & 1u, err);  // plane kk has landed
            tphase ^= 1u << buf;
        } else {
            // planes kk and kk + 1 are in flight; the barrier publishes plane kk to the block
            // and frees the buffer of plane kk - 1, which then receives plane kk + 2
            if (kk + 1 < planes)
                cp_async_wait<1>();
            else
                cp_async_wait<0>();
            __syncthreads();
            if (kk + 2 < planes)
                row_issue<N, SSB1>(p, slot, kk + 2, ry0, tiles + ((kk + 2) % 3) * S::TILEBUF);
        }
        if (tid == 0) {
            // This task no longer needs plane kk of the slot: columns of batch b + D may
            // overwrite it once every row task has passed it.  The plane's reads have all
            // completed (their data is in shared memory), so no fence is needed here.
            red_relaxed_add(plane_free + (size_t)b * p.Bk + kk, 1u);
        }
        if constexpr (SSB1) {
            float2 v[kPts];
#pragma unroll
            for (int r = 0; r < kPts; ++r) {
                const int nx = j + S::T * r;  // element (nx, lr): chunk lr / 2 of column nx, swizzled
                v[r] = active ? cur[nx * S::LDC + 2 * ((lr >> 1) ^ ((nx >> S::SWS) & (S::RC - 1))) +
                                    (lr & 1)]
                              : make_float2(0.f, 0.f);
            }
            reg_fft<N, kPts, +1>(v, smem + S::OFF_RFFT + grp * S::SMR, twN, j, warp_bar);
#pragma unroll
            for (int r = 0; r < kPts; ++r) {
                const float ph = fast_atan2(v[r].y, v[r].x);
                acc1[r] += ph;
                acc2 = fmaf(ph, ph, acc2);
                if (OBJ) acco[r] = cadd(acco[r], v[r]);
            }
        } else {
            const float2 *seg = cur + lr;               // element (nx, lr) at seg[nx * LDC]
            const float2 *rp = cur + S::H * S::LDC;
            const float2 z0 = seg[0], zm = seg[S::M * S::LDC];
            float2 v[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int m = j + S::T * r, mc = S::M - m;
                float2 ym, yc;
                if (m == 0) {
                    ym = make_float2(z0.y, 0.f);
                    yc = make_float2(zm.y, 0.f);
                } else {  // the ring holds Z - s h for these columns
                    const float2 za = seg[m * S::LDC], zb = seg[mc * S::LDC];
                    ym = make_float2(za.y, -za.x);
                    yc = make_float2(zb.y, -zb.x);
                }
                const float2 a = make_float2(ym.x + yc.x, ym.y - yc.y);
                const float2 bb = cmul(make_float2(ym.x - yc.x, ym.y + yc.y), twid<+1>(twN, lay(m)));
                v[r] = active ? make_float2(a.x - bb.y, a.y + bb.x) : make_float2(0.f, 0.f);
            }
            reg_fft<S::M, 8, +1>(v, smem + S::OFF_RFFT + grp * S::SMR, smem + S::OFF_TW2, j, warp_bar);
            const float re_even = z0.x + zm.x, re_odd = z0.x - zm.x;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float2 rpv = rp[j + S::T * r];
                const float re0 = fmaf(sg, rpv.x, re_even), re1 = fmaf(sg, rpv.y, re_odd);
                const float p0 = fast_atan2(v[r].x, re0), p1 = fast_atan2(v[r].y, re1);
                acc1[2 * r] += p0;
                acc1[2 * r + 1] += p1;
                acc2 = fmaf(p0, p0, acc2);
                acc2 = fmaf(p1, p1, acc2);
                if (OBJ) {
                    acco[2 * r] = cadd(acco[2 * r], make_float2(re0, v[r].x));
                    acco[2 * r + 1] = cadd(acco[2 * r + 1], make_float2(re1, v[r].y));
                }
            }
        }
    }
    // Add this batch into the accumulators (S1 by exact two-sums into its float pair, the
    // object sums in float64).  Only this update is ordered: it
    // waits until the previous batch's task for the same rows has made its own update,
    // which keeps the per-pixel summation order fixed while the tasks themselves overlap.
    if (tid == 0) *s_ok = wait_at_least(chain + rt, (unsigned)b, err, p.wait_limit);
    __syncthreads();
    if (SSB1 && active && *s_ok) {
        // pixel j + T r of row ry holds acc1[r]; loads are issued in groups ahead of their
        // stores (a store through the same pointer would hold back each following load)
        // (the first batch writes its sums: the accumulators need no clearing)
        constexpr int GS = OBJ ? 4 : 16;
        float2 *s1 = reinterpret_cast<float2 *>(p.S1 + (size_t)ry * N) + j;
#pragma unroll
        for (int g0 = 0; g0 < 16; g0 += GS) {
            float2 old[GS];
#pragma unroll
            for (int r = 0; r < GS; ++r)
                old[r] = b == 0 ? make_float2(0.f, 0.f) : __ldcg(s1 + S::T * (g0 + r));
#pragma unroll
            for (int r = 0; r < GS; ++r) s1[S::T * (g0 + r)] = df_add(old[r], acc1[g0 + r]);
        }
        if (OBJ) {
            double2 *os = p.Osum + (size_t)ry * N + j;
#pragma unroll
            for (int g0 = 0; g0 < 16; g0 += 4) {
                double2 o[4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    o[r] = b == 0 ? make_double2(0.0, 0.0) : __ldcg(os + S::T * (g0 + r));
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    os[S::T * (g0 + r)] = make_double2(o[r].x + acco[g0 + r].x, o[r].y + acco[g0 + r].y);
            }
        }
    }
    if (!SSB1 && active && *s_ok) {
        // Loads are issued in groups ahead of their stores: a store through the same
        // pointer would otherwise hold back each following load for a full round trip.
        // A thread owns pixel pairs (2 (j + T r), 2 (j + T r) + 1).  With the object sums
        // live, smaller groups keep the registers within the launch bound.
        // (the first batch writes its sums: the accumulators need no clearing)
        constexpr int GS = OBJ ? 2 : 8;  // S1 pixel pairs per group
        float4 *s1 = reinterpret_cast<float4 *>(p.S1 + (size_t)ry * N) + j;
#pragma unroll
        for (int g0 = 0; g0 < 8; g0 += GS) {
            float4 old[GS];
#pragma unroll
            for (int r = 0; r < GS; ++r)
                old[r] = b == 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : __ldcg(s1 + S::T * (g0 + r));
#pragma unroll
            for (int r = 0; r < GS; ++r) {
                const float2 a = df_add(make_float2(old[r].x, old[r].y), acc1[2 * (g0 + r)]);
                const float2 c = df_add(make_float2(old[r].z, old[r].w), acc1[2 * (g0 + r) + 1]);
                s1[S::T * (g0 + r)] = make_float4(a.x, a.y, c.x, c.y);
            }
        }
        if (OBJ) {
            double2 *os = p.Osum + (size_t)ry * N + 2 * j;  // pixel 2 (j + T r) + e at 2 T r + e
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const double2 z = make_double2(0.0, 0.0);
                const double2 o0 = b == 0 ? z : __ldcg(os + 2 * S::T * r);
                const double2 o1 = b == 0 ? z : __ldcg(os + 2 * S::T * r + 1);
                const float2 a0 = acco[2 * r], a1 = acco[2 * r + 1];
                os[2 * S::T * r] = make_double2(o0.x + a0.x, o0.y + a0.y);
                os[2 * S::T * r + 1] = make_double2(o1.x + a1.x, o1.y + a1.y);
            }
        }
    }
    // sum of phi^2: warp shuffles, then the warp partials in a fixed order
    double w2 = active ? (double)acc2 : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w2 += __shfl_down_sync(0xffffffffu, w2, o);
    double *red = reinterpret_cast<double *>(smem + S::OFF_RED);
    if ((tid & 31) == 0) red[tid >> 5] = w2;
    __syncthreads();
    if (tid == 0) {
        double t = 0.0;
#pragma unroll
        for (int w = 0; w < kFusedThreads / 32; ++w) t += red[w];
        if (*s_ok) p.S2g[rt] = (b == 0 ? 0.0 : __ldcg(p.S2g + rt)) + t;
    }
}

// ---------------------------------------------------------------- scheduler

struct Task {
    int kind;  // 0 column, 1 row, 2 none
    int b, idx;
};

__device__ __forceinline__ int planes_in(const FusedParams &p, int b) {
    return b < p.nbatch - 1 ? p.Bk : p.n_bf - p.Bk * (p.nbatch - 1);
}

// Ticket t -> task.  Phase 0 = columns of batch 0; phase q (1 <= q < nbatch) = columns
// of batch q then rows of batch q-1; phase nbatch = rows of the last batch.
template <int N, bool SSB1>
__device__ Task decode_ticket(const FusedParams &p, unsigned t) {
    using S = FusedShape<N, SSB1>;
    const unsigned nc_full = (unsigned)p.Bk * S::CT;
    const unsigned nc_last = (unsigned)planes_in(p, p.nbatch - 1) * S::CT;
    const unsigned nr = S::NR;
    const unsigned nc0 = p.nbatch == 1 ? nc_last : nc_full;
    if (t < nc0) return Task{0, 0, (int)t};
    t -= nc0;
    if (p.nbatch >= 2) {
        const unsigned phase = nc_full + nr;
        const unsigned nfull = (unsigned)(p.nbatch - 2);
        if (t < nfull * phase) {
            const unsigned q = 1 + t / phase, r = t % phase;
            if (r < nc_full) return Task{0, (int)q, (int)r};
            return Task{1, (int)q - 1, (int)(r - nc_full)};
        }
        t -= nfull * phase;
        if (t < nc_last) return Task{0, p.nbatch - 1, (int)t};
        t -= nc_last;
        if (t < nr) return Task{1, p.nbatch - 2, (int)t};
        t -= nr;
    }
    if (t < nr) return Task{1, p.nbatch - 1, (int)t};
    return Task{2, 0, 0};
}

template <int N, bool OBJ, bool SSB1>
__global__ void __launch_bounds__(kFusedThreads, kFusedBlocksPerSM)
    k_fused(FusedParams p, const __grid_constant__ CUtensorMap ring_map) {
    using S = FusedShape<N, SSB1>;
    extern __shared__ __align__(16) float2 smem[];
    __shared__ unsigned s_ticket;
    __shared__ int s_ok;
    __shared__ int s_nyq;
    __shared__ __align__(8) unsigned long long s_tile_bar[2];  // tensor-copy tile barriers
    const int tid = threadIdx.x;
    const uint32_t tile_bars = smem_u32(s_tile_bar);
    unsigned tile_phase = 0u;
    if (S::TMA && tid == 0) {
        mbar_init(tile_bars, 1u);
        mbar_init(tile_bars + 8u, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = tid; i < N; i += kFusedThreads) smem[S::OFF_TW + lay(i)] = p.tw[i];
    for (int i = tid; i < S::M; i += kFusedThreads) smem[S::OFF_TW2 + lay(i)] = p.tw[2 * i];
    unsigned *err = p.err;
    unsigned *ticket = p.sync;
    unsigned *col_done = p.sync + 1;
    unsigned *plane_free = col_done + p.nbatch;
    unsigned *h_cnt = plane_free + (size_t)p.nbatch * p.Bk;
    unsigned *chain = h_cnt + (size_t)p.nbatch * p.Bk;
    __syncthreads();
    // The ticket in s_ticket is read after the barrier at the top of the loop; thread 0
    // takes the next one only after the task's last barrier and its completion signals.
    if (tid == 0) s_ticket = atomicAdd(ticket, 1u);
    __syncthreads();
    // Each task ends with a block barrier that publishes the next ticket in s_ticket (tid 0
    // writes it again only after the next task's first barrier, which every warp reaches
    // after reading it).
    while (true) {
        const Task task = decode_ticket<N, SSB1>(p, s_ticket);
        if (task.kind == 2) break;
        if (task.kind == 0) {
            const int kk = task.idx / S::CT;
            // this plane of the ring slot was last read by the row tasks of batch b - D
            const unsigned *free_word =
                task.b >= p.D ? plane_free + (size_t)(task.b - p.D) * p.Bk + kk : nullptr;
            const int ok = column_task<N, SSB1>(p, smem, task.b, task.idx, free_word, err);
            __syncthreads();
            if (tid == 0) {
                // the next ticket's round trip overlaps the fence
                const unsigned next = atomicAdd(ticket, 1u);
                fence_acq_rel();  // publishes the task's ring columns and Nyquist terms
                // SSB2: the task that completes the plane's column pass also transforms the
                // plane's Nyquist terms.  The count is a relaxed atomic after the fence (a
                // release); only the completing task then fences again to acquire the other
                // tasks' h.  (An acq_rel atomic, which fences on both sides in every task,
                // measured 0.7 % slower overall.)
                if (SSB1) {
                    s_nyq = 0;
                } else {
                    const unsigned done = atom_add_relaxed(h_cnt + (size_t)task.b * p.Bk + kk, 1u) + 1u;
                    s_nyq = done == (unsigned)S::CT;
                    if (s_nyq) fence_acq_rel();
                }
                if (!s_nyq) red_relaxed_add(col_done + task.b, 1u);
                s_ticket = next;
            }
            __syncthreads();  // publishes s_ticket and s_nyq
            if (!SSB1 && s_nyq && tid < 32) {
                // Warp 0 alone transforms the plane's Nyquist terms and signals it, while the
                // other warps go on to the next task.  Its scratch (the first N/2 + N/32 slots
                // of the FFT region) is group 0's in either kind of task, so nothing the next
                // task's other warps touch overlaps it.
                if (ok)  // whole warp: the transform synchronises the warp
                    nyquist_transform<N>(p, smem + S::OFF_FFT + (tid / S::T) * S::SMF,
                                         smem + S::OFF_TW, smem + S::OFF_TW2, task.b % p.D, kk,
                                         tid % S::T, tid < S::T);
                __syncwarp();
                if (tid == 0) {
                    fence_acq_rel();  // publishes Rp
                    red_relaxed_add(col_done + task.b, 1u);
                }
            }
        } else {
            if (tid == 0)
                s_ok = wait_at_least(col_done + task.b,
                                     p.stall ? 0xffffffffu : (unsigned)(planes_in(p, task.b) * S::CT),
                                     err, p.wait_limit);
            __syncthreads();
            if (s_ok) {
                row_task<N, OBJ, SSB1>(p, smem, task.b, task.idx, planes_in(p, task.b), plane_free,
                                       chain, err, &s_ok, &ring_map, tile_bars, tile_phase);
            } else if (tid == 0) {  // release the planes anyway so that no wait is left behind
                for (int kk = 0; kk < planes_in(p, task.b); ++kk)
                    atomicAdd(plane_free + (size_t)task.b * p.Bk + kk, 1u);
            }
            __syncthreads();
            if (tid == 0) {
                const unsigned next = atomicAdd(ticket, 1u);  // its round trip overlaps the fence
                fence_acq_rel();  // publishes the task's S1, S2 (and object) updates
                st_relaxed(chain + task.idx, (unsigned)task.b + 1u);
                s_ticket = next;
            }
            __syncthreads();  // publishes s_ticket
        }
    }
}

// ---------------------------------------------------------------- loss

// L = (1/P) sum_r [S2(r)/n - (S1(r)/n)^2], with S2 summed per row task (NaN when the
// error word is raised).  Each block reduces
// one contiguous range of pixels in a fixed order (strided per thread, then a shared-memory
// tree) into part[block]; the block that finishes last (counted in *cnt, cleared with the
// scheduler words before every evaluation) adds the partials in block order and the row
// task sums in task order.  The result does not depend on which block finishes last.
constexpr int kLossBlocks = 128, kLossThreads = 256;

__global__ void __launch_bounds__(kLossThreads) k_loss_fused(const double *__restrict__ S1,
                                                             const double *__restrict__ S2g, int nr,
                                                             int P, double inv_n, double *part,
                                                             unsigned *cnt, const unsigned *err,
                                                             double *__restrict__ out) {
    __shared__ double red[kLossThreads];
    __shared__ unsigned s_rank;
    const int tid = threadIdx.x;
    const int per = (P + kLossBlocks - 1) / kLossBlocks;
    const int i0 = blockIdx.x * per, i1 = min(P, i0 + per);
    double acc = 0.0;
    for (int i = i0 + tid; i < i1; i += kLossThreads) {
        const double m = s1_value(S1, i) * inv_n;
        acc -= m * m;
    }
    red[tid] = acc;
    __syncthreads();
    for (int h = kLossThreads / 2; h > 0; h >>= 1) {
        if (tid < h) red[tid] += red[tid + h];
        __syncthreads();
    }
    if (tid == 0) {
        part[blockIdx.x] = red[0];
        __threadfence();
        s_rank = atomicAdd(cnt, 1u);
    }
    __syncthreads();
    if (s_rank != kLossBlocks - 1 || tid != 0) return;
    __threadfence();
    double sm = 0.0, s2 = 0.0;
    for (int b = 0; b < kLossBlocks; ++b) sm += __ldcg(part + b);
    for (int r = 0; r < nr; ++r) s2 += S2g[r] * inv_n;
    // a wait of this library call gave up (here or in an earlier trial): no valid loss
    *out = *err != 0u ? __longlong_as_double(0x7ff8000000000000LL) : (s2 + sm) / (double)P;
}

// ---------------------------------------------------------------- host side

static int row_tasks_for(int N) {
    const int groups = kFusedThreads / (N / kPts);
    return N / std::min(groups, N);
}

// scheduler words, then the loss kernel's block counter (the last word)
size_t fused_sync_words(int N, int n_bf, int Bk) {
    const int nbatch = (n_bf + Bk - 1) / Bk;
    return 1 + (size_t)nbatch * (1 + 2 * (size_t)Bk) + (size_t)row_tasks_for(N) + 1;
}

static size_t ldz_for(int N) { return (size_t)((N / 2 + 1 + 7) / 8 * 8); }
size_t fused_ring_elems(int N, int Bk, int D, bool ssb1) {
    return (size_t)D * Bk * (size_t)N * (ssb1 ? N : N / 2 + 1);
}
size_t fused_hring_elems(int N, int Bk, int D) { return (size_t)D * Bk * ldz_for(N); }
size_t fused_rring_elems(int N, int Bk, int D) { return (size_t)D * Bk * (size_t)(N / 2); }
int fused_row_tasks(int N) { return row_tasks_for(N); }
size_t fused_s2g_elems(int N) { return (size_t)row_tasks_for(N) + kLossBlocks; }

// cuTensorMapEncodeTiled, resolved once through the runtime (no link against the driver
// library); null if the driver does not provide it.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// The ring as a 2D tensor of 8-byte elements: x = row ry (N, contiguous), y = transformed
// column of every slot and plane (D Bk H).  Boxes of RT rows x BOXN columns, swizzled to
// match the row task's reads.
template <int N, bool SSB1>
static cudaError_t ring_tensor_map(const FusedParams &fp, CUtensorMap *map) {
    using S = FusedShape<N, SSB1>;
    std::memset(map, 0, sizeof(*map));
    if (!S::TMA) return cudaSuccess;  // not used
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)fp.D * fp.Bk * S::H};
    const cuuint64_t strides[1] = {(cuuint64_t)N * sizeof(float2)};
    const cuuint32_t box[2] = {(cuuint32_t)S::RT, (cuuint32_t)S::BOXN};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT64, 2, fp.Z, dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              S::RT == 8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int N, bool OBJ, bool SSB1>
static cudaError_t fused_launch(const FusedParams &fp, cudaStream_t s) {
    using S = FusedShape<N, SSB1>;
    cudaError_t e;
    CUtensorMap ring_map;
    if ((e = ring_tensor_map<N, SSB1>(fp, &ring_map)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(k_fused<N, OBJ, SSB1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)S::BYTES)) != cudaSuccess)
        return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_fused<N, OBJ, SSB1>, kFusedThreads,
                                                           S::BYTES)) != cudaSuccess)
        return e;
    const long tickets = (long)fp.nbatch * (fp.Bk * S::CT + S::NR);
    const int grid = (int)std::max(1L, std::min((long)sms * std::max(per_sm, 1), tickets));
    prof_begin("k_fused", s);
    k_fused<N, OBJ, SSB1><<<grid, kFusedThreads, S::BYTES, s>>>(fp, ring_map);
    prof_end(s);
    count_launch();
    return cudaGetLastError();
}

template <int N, bool SSB1>
static cudaError_t fused_objective_n(const ObjectiveArgs &a, const TrialHost &th, double *loss_slot,
                                     bool want_object, cudaStream_t s) {
    constexpr int NR = FusedShape<N, SSB1>::NR;  // row tasks per trial
    cudaError_t e;
    if ((e = launch_theta_tables(a, th, s)) != cudaSuccess) return e;
    const size_t P = (size_t)N * N;
    const int nbatch = (a.n_bf + a.Bk - 1) / a.Bk;
    // (S1, the object sums and the per-row-task S2 are written, not added, by the first
    // batch's row tasks, so they need no clearing here)
    // the scheduler words (the error word is the caller's, cleared once per library call so
    // that a wait that ran out in any trial of a batch is still reported)
    if ((e = cudaMemsetAsync(a.sync, 0, sizeof(unsigned) * fused_sync_words(N, a.n_bf, a.Bk), s)) !=
        cudaSuccess)
        return e;
    FusedParams fp;
    fp.G = a.G;
    fp.Et = a.E;
    fp.kgeo = a.kgeo;
    fp.kturn = a.kturn;
    fp.tw = a.tw;
    fp.Z = a.Zring;
    fp.hrow = a.hring;
    fp.rrow = a.rring;
    fp.S1 = a.S1;
    fp.S2g = a.S2g;
    fp.Osum = a.Osum;
    fp.sync = a.sync;
    fp.err = a.err;
    fp.n_bf = a.n_bf;
    fp.Bk = a.Bk;
    fp.nbatch = nbatch;
    fp.D = a.D;
    fp.wait_limit = a.wait_limit ? a.wait_limit : kWaitLimit;
    fp.stall = a.stall;
    fp.tc = make_trial_const(a, th, N);
    e = want_object ? fused_launch<N, true, SSB1>(fp, s) : fused_launch<N, false, SSB1>(fp, s);
    if (e != cudaSuccess) return e;
    prof_begin("k_loss", s);
    k_loss_fused<<<kLossBlocks, kLossThreads, 0, s>>>(
        a.S1, a.S2g, NR, (int)P, 1.0 / a.n_bf, a.S2g + NR,
        a.sync + fused_sync_words(N, a.n_bf, a.Bk) - 1, a.err, loss_slot);
    prof_end(s);
    count_launch();
    return cudaGetLastError();
}

cudaError_t run_objective_fused(const ObjectiveArgs &a, const ssb_params &theta, double *loss_slot,
                                bool want_object, cudaStream_t s) {
    const TrialHost th = trial_host(theta);
    const bool s1 = a.mode == 1;
    switch (a.N) {
        case 32: return s1 ? fused_objective_n<32, true>(a, th, loss_slot, want_object, s)
                           : fused_objective_n<32, false>(a, th, loss_slot, want_object, s);
        case 64: return s1 ? fused_objective_n<64, true>(a, th, loss_slot, want_object, s)
                           : fused_objective_n<64, false>(a, th, loss_slot, want_object, s);
        case 128: return s1 ? fused_objective_n<128, true>(a, th, loss_slot, want_object, s)
                            : fused_objective_n<128, false>(a, th, loss_slot, want_object, s);
        case 256: return s1 ? fused_objective_n<256, true>(a, th, loss_slot, want_object, s)
                            : fused_objective_n<256, false>(a, th, loss_slot, want_object, s);
        case 512: return s1 ? fused_objective_n<512, true>(a, th, loss_slot, want_object, s)
                            : fused_objective_n<512, false>(a, th, loss_slot, want_object, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssb
