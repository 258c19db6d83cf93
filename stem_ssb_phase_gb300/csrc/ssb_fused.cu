// Persistent, ticket-scheduled evaluation of the exact SSB objective (SSB2 transfer).
//
// The pages locate the cost of the exact objective in the column -> row intermediate that
// is written and re-read through global memory ("Later SSB performance checkpoints",
// 2026-09-11 checkpoints: about 18.8 GB per evaluation).  Here that intermediate never
// leaves L2: BF planes are processed in batches of Bk planes through a ring of D batch
// slots (tens of MB, L2-resident), by one persistent kernel on every SM.
//
// Work is cut in half exactly.  Off DC and the Nyquist lines the corrected spectrum is
// anti-Hermitian, C(-Q) = -conj C(Q) (the relation of "SSB performance notes", 257-row
// intermediate prototype).  So only the N/2+1 half-plane columns are corrected and
// column-transformed; each row is rebuilt from them as
//     Zfull(ry, N - nx) = -conj Z(ry, nx) + 2 (-1)^ry conj h(nx),   1 <= nx < N/2,
// where h(nx) = (C(N/2, nx) + conj C(N/2, N - nx)) / 2 is the Hermitian part of the
// Nyquist row, whose bins have no negative-frequency partner (the violation the pages
// isolate).  Columns 0 and N/2 are transformed in full.  The result equals the plain
// two-dimensional inverse transform in exact arithmetic.
//
// Tasks (ticket order, phase p = [columns of batch p, rows of batch p-1]):
//   column task (batch b, plane, CW half-plane columns): G load, correction, column IFFT,
//       store to the ring slot in 4-row tiles Z[slot][plane][ry/4][nx][ry%4];
//   row task (batch b, RT rows): for each plane of the batch, rebuild the full rows,
//       row IFFT, phi = atan2, accumulate; then add the batch's per-pixel sums into the
//       float64 S1 (and S2, object) in batch order.
// A task waits only for tasks holding smaller tickets, so the schedule cannot deadlock
// whatever the number of resident blocks.  Every wait is bounded; on timeout the kernel
// raises an error flag, all waits stop and the host reports SSB_ERR_TIMEOUT.
#include <algorithm>

#include "ssb_device.cuh"
#include "ssb_internal.h"
#include "ssb_regfft.cuh"

namespace ssb {

constexpr int kFusedThreads = 256;
constexpr int kRingSlots = 3;
constexpr unsigned kWaitLimit = 1u << 24;  // polls of ~0.1-1 us each before giving up

struct FusedParams {
    const float2 *G;      // [n_bf][H][N]
    const float2 *Et;     // [N (nx)][N (ny)] e^{i chi(lambda Q')}
    const float4 *kgeo;   // per BF (alpha_x, alpha_y, a_k, 0)
    const uint2 *kturn;   // per BF bilinear phase slopes
    const float2 *tw;     // [N] exp(+2 pi i m/N)
    float2 *Z;            // ring [D][Bk][N/4][H][4]
    float2 *hrow;         // ring [D][Bk][H]
    double *S1;           // [P]
    double *S2g;          // [row tasks]
    double2 *Osum;        // [P] (object redraw only)
    unsigned *sync;       // ticket, error, col_done[nbatch], row_done[nbatch], chain[row tasks]
    int n_bf, Bk, nbatch;
    TrialConst tc;
};

template <int N>
struct FusedShape {
    static constexpr int T = N / 8;                 // threads per transform
    static constexpr int H = N / 2 + 1;             // half-plane columns
    static constexpr int CW = kFusedThreads / T;    // columns per column task
    static constexpr int RT = CW < N ? CW : N;      // rows per row task (multiple of 4)
    static constexpr int CT = (H + CW - 1) / CW;    // column tasks per plane
    static constexpr int NR = N / RT;               // row tasks per trial
    static constexpr int SMF = RegFFT<N>::SMEM;     // FFT scratch per group
    // dynamic shared memory layout, in float2 units
    static constexpr int OFF_TW = 0;
    static constexpr int OFF_FFT = OFF_TW + N;
    static constexpr int OFF_TILE = OFF_FFT + CW * SMF;
    static constexpr int OFF_H = OFF_TILE + RT * H;
    static constexpr int OFF_RED = OFF_H + ((H + 1) & ~1);
    static constexpr int TOTAL = OFF_RED + kFusedThreads;  // reduction uses 8 bytes each
    static constexpr size_t BYTES = (size_t)TOTAL * sizeof(float2);
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Called by one thread: wait until *addr >= target.  Returns false if the wait gave up
// (error flag already raised elsewhere, or the poll budget ran out, which raises it).
__device__ bool wait_at_least(const unsigned *addr, unsigned target, unsigned *err) {
    unsigned polls = 0;
    while (ld_acquire(addr) < target) {
        if (ld_acquire(err) != 0u) return false;
        if (++polls > kWaitLimit) {
            atomicOr(err, 2u);
            return false;
        }
        __nanosleep(128);
    }
    return true;
}

__device__ __forceinline__ void block_bar() { __syncthreads(); }

// ---------------------------------------------------------------- column task

template <int N>
__device__ void column_task(const FusedParams &p, float2 *smem, int b, int idx) {
    using S = FusedShape<N>;
    const int tid = threadIdx.x, grp = tid / S::T, j = tid % S::T;
    const int kk = idx / S::CT, ct = idx - kk * S::CT;
    const int k = b * p.Bk + kk;
    const int slot = b % kRingSlots;
    const int nx = ct * S::CW + grp;
    const bool valid = nx < S::H;
    const float4 geo = p.kgeo[k];
    const uint2 bt = p.kturn[k];
    float2 v[8];
    if (valid) {
        const float2 *g = p.G + ((size_t)k * S::H + nx) * N;
        const float2 *e = p.Et + (size_t)nx * N;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int ny = j + S::T * r;
            const float2 gv = __ldcs(g + ny);
            v[r] = cmul(gv, correction_factor<N>(ny, nx, geo, bt, __ldg(e + ny), p.tc));
            if (r == 4 && j == 0 && nx >= 1 && nx < N / 2) {
                // Nyquist row: its mirror bin carries its own correction (no partner)
                const float2 f2 = correction_factor<N>(N / 2, N - nx, geo, bt,
                                                       __ldg(p.Et + (size_t)(N - nx) * N + N / 2), p.tc);
                const float2 c2 = cmul(cconj(gv), f2);
                const float2 h = make_float2(0.5f * (v[r].x + c2.x), 0.5f * (v[r].y - c2.y));
                __stcg(p.hrow + ((size_t)slot * p.Bk + kk) * S::H + nx, h);
            }
        }
    } else {
#pragma unroll
        for (int r = 0; r < 8; ++r) v[r] = make_float2(0.f, 0.f);
    }
    reg_fft<N, +1>(v, smem + S::OFF_FFT + grp * S::SMF, smem + S::OFF_TW, j, block_bar);
    if (valid) {
        float2 *z = p.Z + ((size_t)slot * p.Bk + kk) * (size_t)(N / 4) * S::H * 4;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int ry = j + S::T * r;
            __stcg(z + ((size_t)(ry >> 2) * S::H + nx) * 4 + (ry & 3), v[r]);
        }
    }
}

// ---------------------------------------------------------------- row task

template <int N, bool OBJ>
__device__ void row_task(const FusedParams &p, float2 *smem, int b, int rt, int planes) {
    using S = FusedShape<N>;
    const int tid = threadIdx.x, grp = tid / S::T, j = tid % S::T;
    const int slot = b % kRingSlots;
    const int ry0 = rt * S::RT;
    const bool active = grp < S::RT;                // N = 32 leaves some groups idle
    const int ry = ry0 + (active ? grp : 0);        // this group's row
    const int lt = grp >> 2, lb = grp & 3;          // tile within the task, row within tile
    const float sgn2 = (ry & 1) ? -2.0f : 2.0f;     // 2 (-1)^ry
    float2 *tile = smem + S::OFF_TILE;
    float2 *hs = smem + S::OFF_H;
    float acc1[8];
    float2 acco[8];
    float acc2 = 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        acc1[r] = 0.f;
        acco[r] = make_float2(0.f, 0.f);
    }
    for (int kk = 0; kk < planes; ++kk) {
        // stage this task's RT/4 row tiles (contiguous) and the plane's Nyquist terms
        const float4 *zsrc = reinterpret_cast<const float4 *>(
            p.Z + (((size_t)slot * p.Bk + kk) * (size_t)(N / 4) + ry0 / 4) * S::H * 4);
        float4 *tdst = reinterpret_cast<float4 *>(tile);
        for (int i = tid; i < S::RT * S::H / 2; i += kFusedThreads) tdst[i] = __ldcg(zsrc + i);
        const float2 *hsrc = p.hrow + ((size_t)slot * p.Bk + kk) * S::H;
        for (int i = tid; i < S::H; i += kFusedThreads) hs[i] = __ldcg(hsrc + i);
        __syncthreads();
        float2 v[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int nx = j + S::T * r;
            if (!active) {
                v[r] = make_float2(0.f, 0.f);
            } else if (nx <= N / 2) {
                v[r] = tile[((size_t)lt * S::H + nx) * 4 + lb];
            } else {
                const int m = N - nx;
                const float2 z = tile[((size_t)lt * S::H + m) * 4 + lb];
                const float2 h = hs[m];
                v[r] = make_float2(fmaf(sgn2, h.x, -z.x), fmaf(-sgn2, h.y, z.y));
            }
        }
        reg_fft<N, +1>(v, smem + S::OFF_FFT + grp * S::SMF, smem + S::OFF_TW, j, block_bar);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const float phi = atan2f(v[r].y, v[r].x);
            acc1[r] += phi;
            acc2 = fmaf(phi, phi, acc2);
            if (OBJ) acco[r] = cadd(acco[r], v[r]);
        }
        __syncthreads();  // tile and hs are reloaded for the next plane
    }
    // add this batch into the float64 accumulators (batches arrive in order per task)
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        if (!active) break;
        const size_t i = (size_t)ry * N + j + S::T * r;
        p.S1[i] = __ldcg(p.S1 + i) + (double)acc1[r];
        if (OBJ) {
            const double2 o = __ldcg(p.Osum + i);
            p.Osum[i] = make_double2(o.x + acco[r].x, o.y + acco[r].y);
        }
    }
    double *red = reinterpret_cast<double *>(smem + S::OFF_RED);
    red[tid] = active ? (double)acc2 : 0.0;
    __syncthreads();
#pragma unroll
    for (int s = kFusedThreads / 2; s > 0; s >>= 1) {
        if (tid < s) red[tid] += red[tid + s];
        __syncthreads();
    }
    if (tid == 0) p.S2g[rt] = __ldcg(p.S2g + rt) + red[0];
}

// ---------------------------------------------------------------- scheduler

struct Task {
    int kind;  // 0 column, 1 row, 2 none
    int b, idx;
};

template <int N>
__device__ __forceinline__ int planes_in(const FusedParams &p, int b) {
    return b < p.nbatch - 1 ? p.Bk : p.n_bf - p.Bk * (p.nbatch - 1);
}

// Ticket t -> task.  Phase 0 = columns of batch 0; phase q (1 <= q < nbatch) = columns
// of batch q then rows of batch q-1; phase nbatch = rows of the last batch.
template <int N>
__device__ Task decode_ticket(const FusedParams &p, unsigned t) {
    using S = FusedShape<N>;
    const unsigned nc_full = (unsigned)p.Bk * S::CT;
    const unsigned nc_last = (unsigned)planes_in<N>(p, p.nbatch - 1) * S::CT;
    const unsigned nr = S::NR;
    Task task{2, 0, 0};
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
    return task;
}

template <int N, bool OBJ>
__global__ void __launch_bounds__(kFusedThreads) k_fused(FusedParams p) {
    using S = FusedShape<N>;
    extern __shared__ float2 smem[];
    __shared__ unsigned s_ticket;
    __shared__ int s_ok;
    const int tid = threadIdx.x;
    for (int i = tid; i < N; i += kFusedThreads) smem[S::OFF_TW + i] = p.tw[i];
    unsigned *ticket = p.sync;
    unsigned *err = p.sync + 1;
    unsigned *col_done = p.sync + 2;
    unsigned *row_done = col_done + p.nbatch;
    unsigned *chain = row_done + p.nbatch;
    __syncthreads();
    while (true) {
        if (tid == 0) s_ticket = atomicAdd(ticket, 1u);
        __syncthreads();
        const Task task = decode_ticket<N>(p, s_ticket);
        if (task.kind == 2) break;
        if (tid == 0) {
            bool ok = true;
            if (task.kind == 0) {
                if (task.b >= kRingSlots)  // ring slot still being read by rows of b - D
                    ok = wait_at_least(row_done + task.b - kRingSlots, (unsigned)S::NR, err);
            } else {
                ok = wait_at_least(col_done + task.b, (unsigned)(planes_in<N>(p, task.b) * S::CT), err);
                ok = ok && wait_at_least(chain + task.idx, (unsigned)task.b, err);
            }
            s_ok = ok;
        }
        __syncthreads();
        if (task.kind == 0) {
            if (s_ok) column_task<N>(p, smem, task.b, task.idx);
            __syncthreads();
            if (tid == 0) {
                __threadfence();
                atomicAdd(col_done + task.b, 1u);
            }
        } else {
            if (s_ok) row_task<N, OBJ>(p, smem, task.b, task.idx, planes_in<N>(p, task.b));
            __syncthreads();
            if (tid == 0) {
                __threadfence();
                st_release(chain + task.idx, (unsigned)task.b + 1u);
                atomicAdd(row_done + task.b, 1u);
            }
        }
    }
}

// ---------------------------------------------------------------- loss

__global__ void __launch_bounds__(1024) k_loss_fused(const double *__restrict__ S1,
                                                     const double *__restrict__ S2g, int nr,
                                                     int P, double inv_n, double *__restrict__ out) {
    __shared__ double red[1024];
    const int tid = threadIdx.x;
    double acc = 0.0;
    for (int i = tid; i < P; i += 1024) {
        const double m = S1[i] * inv_n;
        acc -= m * m;
    }
    for (int i = tid; i < nr; i += 1024) acc += S2g[i] * inv_n;
    red[tid] = acc;
    __syncthreads();
    for (int s = 512; s > 0; s >>= 1) {
        if (tid < s) red[tid] += red[tid + s];
        __syncthreads();
    }
    if (tid == 0) *out = red[0] / (double)P;
}

// ---------------------------------------------------------------- host side

size_t fused_sync_words(int N, int n_bf, int Bk) {
    const int nbatch = (n_bf + Bk - 1) / Bk;
    const int rt = std::min(kFusedThreads / (N / 8), N);
    return 2 + 2 * (size_t)nbatch + (size_t)(N / rt);
}

size_t fused_ring_elems(int N, int Bk) { return (size_t)kRingSlots * Bk * (size_t)N * (N / 2 + 1); }
size_t fused_hring_elems(int N, int Bk) { return (size_t)kRingSlots * Bk * (size_t)(N / 2 + 1); }
int fused_row_tasks(int N) { return N / std::min(kFusedThreads / (N / 8), N); }

template <int N, bool OBJ>
static cudaError_t fused_launch(const FusedParams &fp, cudaStream_t s) {
    using S = FusedShape<N>;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k_fused<N, OBJ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)S::BYTES)) != cudaSuccess)
        return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_fused<N, OBJ>, kFusedThreads,
                                                           S::BYTES)) != cudaSuccess)
        return e;
    const long tickets = (long)fp.nbatch * (fp.Bk * S::CT + S::NR);
    const int grid = (int)std::max(1L, std::min((long)sms * std::max(per_sm, 1), tickets));
    prof_begin("k_fused", s);
    k_fused<N, OBJ><<<grid, kFusedThreads, S::BYTES, s>>>(fp);
    prof_end(s);
    count_launch();
    return cudaGetLastError();
}

template <int N>
static cudaError_t fused_objective_n(const ObjectiveArgs &a, const TrialHost &th, double *loss_slot,
                                     bool want_object, cudaStream_t s) {
    using S = FusedShape<N>;
    cudaError_t e;
    if ((e = launch_theta_tables(a, th, s)) != cudaSuccess) return e;
    const size_t P = (size_t)N * N;
    const int nbatch = (a.n_bf + a.Bk - 1) / a.Bk;
    if ((e = cudaMemsetAsync(a.S1, 0, sizeof(double) * P, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.S2g, 0, sizeof(double) * S::NR, s)) != cudaSuccess) return e;
    if (want_object && (e = cudaMemsetAsync(a.Osum, 0, sizeof(double2) * P, s)) != cudaSuccess)
        return e;
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
    fp.S1 = a.S1;
    fp.S2g = a.S2g;
    fp.Osum = a.Osum;
    fp.sync = a.sync;
    fp.n_bf = a.n_bf;
    fp.Bk = a.Bk;
    fp.nbatch = nbatch;
    fp.tc = make_trial_const(a, th, N);
    e = want_object ? fused_launch<N, true>(fp, s) : fused_launch<N, false>(fp, s);
    if (e != cudaSuccess) return e;
    prof_begin("k_loss", s);
    k_loss_fused<<<1, 1024, 0, s>>>(a.S1, a.S2g, S::NR, (int)P, 1.0 / a.n_bf, loss_slot);
    prof_end(s);
    count_launch();
    return cudaGetLastError();
}

cudaError_t run_objective_fused(const ObjectiveArgs &a, const ssb_params &theta, double *loss_slot,
                                bool want_object, cudaStream_t s) {
    const TrialHost th = trial_host(theta);
    switch (a.N) {
        case 32: return fused_objective_n<32>(a, th, loss_slot, want_object, s);
        case 64: return fused_objective_n<64>(a, th, loss_slot, want_object, s);
        case 128: return fused_objective_n<128>(a, th, loss_slot, want_object, s);
        case 256: return fused_objective_n<256>(a, th, loss_slot, want_object, s);
        case 512: return fused_objective_n<512>(a, th, loss_slot, want_object, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssb
