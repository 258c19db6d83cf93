// C ABI of the SSB library: argument validation, context ownership, orchestration.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <limits>
#include <new>
#include <string>
#include <vector>

#include "../../include/ssb_debug.h"
#include "ssb_device.cuh"
#include "ssb_internal.h"
#include "ssb_redraw.h"

#ifndef SSB_FUSED_BK
#define SSB_FUSED_BK 16
#endif
#ifndef SSB_FUSED_RING
#define SSB_FUSED_RING 4
#endif
// SSB1 (all N columns, twice the ring per plane): 10-plane batches in 3 slots, 60 MB at
// N = 512 (8 planes in 4 slots measured 0.5 % slower, 6 in 4 slots 4 % slower, 16 in 2
// slots 60 % slower)
#ifndef SSB_FUSED_BK1
#define SSB_FUSED_BK1 10
#endif
#ifndef SSB_FUSED_RING1
#define SSB_FUSED_RING1 3
#endif

namespace ssb {

static std::atomic<uint64_t> g_launches{0};
void count_launch(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

static thread_local std::string g_last_error;

void set_last_error(const char *msg) { g_last_error = msg ? msg : ""; }

// ---- per-launch profiler (active only inside ssb_profile_objective) ----
struct ProfRecord {
    std::string name;
    cudaEvent_t a, b;
};
struct Profiler {
    std::vector<ProfRecord> recs;
    bool open = false;
};
static thread_local Profiler *g_prof = nullptr;

void prof_begin(const char *name, cudaStream_t s) {
    if (!g_prof) return;
    ProfRecord r;
    r.name = name;
    cudaEventCreate(&r.a);
    cudaEventCreate(&r.b);
    cudaEventRecord(r.a, s);
    g_prof->recs.push_back(r);
    g_prof->open = true;
}

void prof_end(cudaStream_t s) {
    if (!g_prof || !g_prof->open) return;
    cudaEventRecord(g_prof->recs.back().b, s);
    g_prof->open = false;
}

static ssb_status fail(ssb_status st, const std::string &msg) {
    g_last_error = msg;
    return st;
}

static ssb_status cuda_fail(cudaError_t e, const char *what) {
    g_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    (void)cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? SSB_ERR_OOM : SSB_ERR_CUDA;
}

#define SSB_CK(call)                                         \
    do {                                                     \
        cudaError_t _e = (call);                             \
        if (_e != cudaSuccess) return cuda_fail(_e, #call);  \
    } while (0)

// Makes the context's device current for the duration of a call.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace ssb

using namespace ssb;

// The buffers one evaluation in flight works in: per-trial tables, the column-to-row ring,
// the accumulators and the scheduler words.  A context holds two sets, so that consecutive
// trials of a batch can overlap on the GPU.
struct TrialSet {
    uint2 *kturn = nullptr;
    float2 *E = nullptr;
    double *S1 = nullptr;
    float2 *Zring = nullptr, *hring = nullptr, *rring = nullptr;
    double *S2g = nullptr;
    unsigned *sync = nullptr;
};

struct ssb_ctx {
    int dev = 0;
    int N = 0, n_bf = 0;
    double step = 0, lam = 0, semi = 0, dalpha = 0;
    ssb_transfer transfer = SSB_TRANSFER_SSB2;
    float2 *G = nullptr;
    float4 *kgeo = nullptr;
    double2 *kalpha = nullptr;
    float2 *tw = nullptr;
    TrialSet set[2];
    double2 *Osum = nullptr;  // object sums (set 0 only: ssb_reconstruct)
    double *loss = nullptr;
    int loss_cap = 0;
    unsigned *err = nullptr;  // error word of the current library call
    int Bk = 0, D = 0;
    // second stream of a batch (odd trials) and the events that fork and join it
    cudaStream_t aux = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    int *flag = nullptr;
    size_t g_bytes = 0, scratch_bytes = 0;
    // upsampled redraw scratch, allocated on first use for the largest factor seen
    float2 *up_T = nullptr, *up_tab = nullptr;
    int up_factor = 0;
    // redraw-without-loss scratch, allocated on first use
    double2 *rd_part = nullptr;
    float2 *rd_S = nullptr, *rd_T = nullptr;
    // test hook (ssb_debug_stall_next): the evaluation with this index in the next call
    // stalls its row tasks on a count that is never reached, with this poll limit; the
    // call_* copies are the hook as the current call took it over
    int dbg_stall_eval = -1;
    unsigned dbg_wait_limit = 0;
    int call_stall_eval = -1;
    unsigned call_wait_limit = 0;

    ObjectiveArgs args(int si = 0) const {
        const TrialSet &t = set[si];
        ObjectiveArgs a;
        a.N = N;
        a.n_bf = n_bf;
        a.G = G;
        a.kgeo = kgeo;
        a.kalpha = kalpha;
        a.kturn = t.kturn;
        a.E = t.E;
        a.tw = tw;
        a.S1 = t.S1;
        a.Osum = si == 0 ? Osum : nullptr;
        a.loss = loss;
        a.Zring = t.Zring;
        a.hring = t.hring;
        a.rring = t.rring;
        a.S2g = t.S2g;
        a.sync = t.sync;
        a.err = err;
        a.Bk = Bk;
        a.D = D;
        a.mode = transfer == SSB_TRANSFER_SSB1 ? 1 : 0;
        a.step = step;
        a.lam = lam;
        a.semi = semi;
        a.dalpha = dalpha;
        a.wait_limit = 0;
        a.stall = 0;
        return a;
    }
};

static void free_ctx(ssb_ctx *c) {
    if (!c) return;
    void *ptrs[] = {c->G, c->kgeo, c->kalpha, c->tw, c->Osum, c->loss, c->err, c->flag,
                    c->up_T,  c->up_tab, c->rd_part, c->rd_S, c->rd_T};
    for (void *p : ptrs)
        if (p) cudaFree(p);
    for (const TrialSet &t : c->set) {
        void *tp[] = {t.kturn, t.E, t.S1, t.Zring, t.hring, t.rring, t.S2g, t.sync};
        for (void *p : tp)
            if (p) cudaFree(p);
    }
    if (c->ev_fork) cudaEventDestroy(c->ev_fork);
    if (c->ev_join) cudaEventDestroy(c->ev_join);
    if (c->aux) cudaStreamDestroy(c->aux);
    delete c;
}

static bool finite_pos(double v) { return std::isfinite(v) && v > 0.0; }

// Evaluation number `index` of the current library call (the stall test hook applies to
// one), in buffer set `si`.
static cudaError_t evaluate(const ssb_ctx *c, const ssb_params &theta, double *loss_slot,
                            bool want_object, cudaStream_t s, int index = 0, int si = 0) {
    ObjectiveArgs a = c->args(si);
    if (index == c->call_stall_eval) {
        a.stall = 1;
        a.wait_limit = c->call_wait_limit;
    }
    return run_objective_fused(a, theta, loss_slot, want_object, s);
}

// Start of a library call that evaluates the objective: take over (and so consume) the
// stall test hook, whatever the call's outcome, and clear the scheduler's error word (it
// stays raised for the rest of the call once a wait has run out).
static ssb_status begin_call(ssb_ctx *c, cudaStream_t s) {
    c->call_stall_eval = c->dbg_stall_eval;
    c->call_wait_limit = c->dbg_wait_limit;
    c->dbg_stall_eval = -1;
    c->dbg_wait_limit = 0;
    SSB_CK(cudaMemsetAsync(c->err, 0, sizeof(unsigned), s));
    return SSB_OK;
}

// End of such a call, or of one chunk of it: the scheduler's error word (a bounded wait
// that ran out in any of the call's evaluations so far).
static ssb_status check_sync(ssb_ctx *c, cudaStream_t s) {
    unsigned h = 0;
    SSB_CK(cudaMemcpyAsync(&h, c->err, sizeof(unsigned), cudaMemcpyDeviceToHost, s));
    SSB_CK(cudaStreamSynchronize(s));
    if (h) return fail(SSB_ERR_TIMEOUT, "a scheduler wait in the fused objective kernel ran out");
    return SSB_OK;
}

static bool valid_theta(const ssb_params &t) {
    return std::isfinite(t.C10_nm) && std::isfinite(t.C12_nm) && std::isfinite(t.phi12_rad) &&
           std::isfinite(t.rotation_rad);
}

template <typename T>
static cudaError_t dev_alloc(T **p, size_t count, size_t *acc) {
    *acc += count * sizeof(T);
    return cudaMalloc((void **)p, count * sizeof(T));
}

static ssb_status check_flag(ssb_ctx *c, cudaStream_t s) {
    int h = 0;
    SSB_CK(cudaMemcpyAsync(&h, c->flag, sizeof(int), cudaMemcpyDeviceToHost, s));
    SSB_CK(cudaStreamSynchronize(s));
    if (h & 1) {
        SSB_CK(cudaMemsetAsync(c->flag, 0, sizeof(int), s));
        return fail(SSB_ERR_ARG, "a count exceeds 2^24 and cannot be converted to float32 exactly");
    }
    if (h) {
        SSB_CK(cudaMemsetAsync(c->flag, 0, sizeof(int), s));
        return fail(SSB_ERR_DEVICE_FLAG, "kernel error flag " + std::to_string(h));
    }
    return SSB_OK;
}

extern "C" {

const char *ssb_status_string(ssb_status s) {
    switch (s) {
        case SSB_OK: return "SSB_OK";
        case SSB_ERR_ARG: return "SSB_ERR_ARG";
        case SSB_ERR_UNSUPPORTED: return "SSB_ERR_UNSUPPORTED";
        case SSB_ERR_OOM: return "SSB_ERR_OOM";
        case SSB_ERR_CUDA: return "SSB_ERR_CUDA";
        case SSB_ERR_TIMEOUT: return "SSB_ERR_TIMEOUT";
        case SSB_ERR_DEVICE_FLAG: return "SSB_ERR_DEVICE_FLAG";
    }
    return "SSB_ERR_UNKNOWN";
}

const char *ssb_last_error(void) { return g_last_error.c_str(); }

uint64_t ssb_kernel_launches(void) { return g_launches.load(); }

ssb_status ssb_prepare(const ssb_geometry *g, const void *counts, ssb_dtype dtype,
                       int counts_on_device, ssb_transfer transfer, void *cuda_stream,
                       ssb_ctx **out) {
    g_last_error.clear();
    if (!out) return fail(SSB_ERR_ARG, "out is NULL");
    *out = nullptr;
    if (!g || !counts) return fail(SSB_ERR_ARG, "geometry or counts is NULL");
    const int N = g->scan_n;
    if (N != 32 && N != 64 && N != 128 && N != 256 && N != 512)
        return fail(SSB_ERR_UNSUPPORTED, "scan_n must be 32, 64, 128, 256 or 512");
    if (g->n_bf < 1) return fail(SSB_ERR_ARG, "n_bf must be >= 1");
    if (!g->bf_det_yx) return fail(SSB_ERR_ARG, "bf_det_yx is NULL");
    if (!finite_pos(g->scan_step_A) || !finite_pos(g->wavelength_A) ||
        !finite_pos(g->semiangle_mrad) || !finite_pos(g->det_sampling_mrad))
        return fail(SSB_ERR_ARG, "geometry scalars must be finite and positive");
    if (dtype != SSB_U16 && dtype != SSB_U32) return fail(SSB_ERR_ARG, "unknown dtype");
    if (transfer != SSB_TRANSFER_SSB2 && transfer != SSB_TRANSFER_SSB1)
        return fail(SSB_ERR_ARG, "unknown transfer");
    for (int k = 0; k < 2 * g->n_bf; ++k)
        if (!std::isfinite(g->bf_det_yx[k])) return fail(SSB_ERR_ARG, "bf_det_yx has a non-finite entry");
    cudaStream_t s = (cudaStream_t)cuda_stream;

    ssb_ctx *c = new (std::nothrow) ssb_ctx();
    if (!c) return fail(SSB_ERR_OOM, "host allocation failed");
    SSB_CK(cudaGetDevice(&c->dev));
    c->N = N;
    c->n_bf = g->n_bf;
    c->step = g->scan_step_A;
    c->lam = g->wavelength_A;
    c->semi = g->semiangle_mrad * 1e-3;
    c->dalpha = g->det_sampling_mrad * 1e-3;
    c->transfer = transfer;
    const int H = N / 2 + 1;
    const size_t P = (size_t)N * N;

    ssb_status st = SSB_OK;
    auto bail = [&](ssb_status code) {
        free_ctx(c);
        return code;
    };
    cudaError_t e;
    size_t gb = 0, sb = 0;
#define SSB_ALLOC(ptr, count, acc)                                       \
    if ((e = dev_alloc(&(ptr), (count), &(acc))) != cudaSuccess) {       \
        st = cuda_fail(e, "cudaMalloc " #ptr);                           \
        return bail(st);                                                 \
    }
    SSB_ALLOC(c->G, (size_t)c->n_bf * H * N, gb);
    SSB_ALLOC(c->kgeo, (size_t)c->n_bf, sb);
    SSB_ALLOC(c->kalpha, (size_t)c->n_bf, sb);
    SSB_ALLOC(c->tw, (size_t)N, sb);
    // Both transfers run on the persistent fused kernel.  Batch size and ring depth: four
    // batches in flight keep the column work flowing while row tasks drain the oldest
    // slot, and the ring stays within L2 (67 MB at N = 512; SSB1 transforms all N columns,
    // so its ring holds 30 planes in 3 slots, 60 MB).  Larger batches amortise each row task's fixed
    // costs further but push the ring out of L2: at 24 planes and more the whole
    // intermediate round-trips HBM (about 3x the G bytes of DRAM traffic).
    const bool ssb1 = transfer == SSB_TRANSFER_SSB1;
    c->Bk = std::min(ssb1 ? SSB_FUSED_BK1 : SSB_FUSED_BK, c->n_bf);
    c->D = ssb1 ? SSB_FUSED_RING1 : SSB_FUSED_RING;
    for (TrialSet &t : c->set) {
        SSB_ALLOC(t.kturn, (size_t)c->n_bf, sb);
        SSB_ALLOC(t.E, P, sb);
        SSB_ALLOC(t.Zring, fused_ring_elems(N, c->Bk, c->D, ssb1), sb);
        SSB_ALLOC(t.hring, fused_hring_elems(N, c->Bk, c->D), sb);
        SSB_ALLOC(t.rring, fused_rring_elems(N, c->Bk, c->D), sb);
        SSB_ALLOC(t.S2g, fused_s2g_elems(N), sb);
        SSB_ALLOC(t.sync, fused_sync_words(N, c->n_bf, c->Bk), sb);
        SSB_ALLOC(t.S1, P, sb);
    }
    SSB_ALLOC(c->Osum, P, sb);
    SSB_ALLOC(c->err, (size_t)1, sb);
    c->loss_cap = 4096;
    SSB_ALLOC(c->loss, (size_t)c->loss_cap, sb);
    SSB_ALLOC(c->flag, (size_t)1, sb);
    c->g_bytes = gb;
    c->scratch_bytes = sb;
    if ((e = cudaStreamCreateWithFlags(&c->aux, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming)) != cudaSuccess) {
        st = cuda_fail(e, "stream or event creation");
        return bail(st);
    }

    // per-BF geometry (float64 on the host)
    std::vector<float4> kgeo(c->n_bf);
    std::vector<double2> kal(c->n_bf);
    for (int k = 0; k < c->n_bf; ++k) {
        const double ay = (double)g->bf_det_yx[2 * k] * c->dalpha;
        const double ax = (double)g->bf_det_yx[2 * k + 1] * c->dalpha;
        const double r = std::sqrt(ax * ax + ay * ay);
        double amp = std::min(1.0, std::max(0.0, (c->semi - r) / c->dalpha + 0.5));
        if (amp < 1.0 / 65536.0) amp = 0.0;  // zero-transfer floor of the aperture
        kgeo[k] = make_float4((float)ax, (float)ay, (float)amp, 0.f);
        kal[k] = make_double2(ax, ay);
    }
    std::vector<float2> tw(N);
    for (int m = 0; m < N; ++m) {
        const double a = 2.0 * M_PI * (double)m / (double)N;
        tw[m] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
#define SSB_CK_BAIL(call)                                  \
    if ((e = (call)) != cudaSuccess) {                     \
        st = cuda_fail(e, #call);                          \
        return bail(st);                                   \
    }
    SSB_CK_BAIL(cudaMemcpyAsync(c->kgeo, kgeo.data(), sizeof(float4) * c->n_bf, cudaMemcpyHostToDevice, s));
    SSB_CK_BAIL(cudaMemcpyAsync(c->kalpha, kal.data(), sizeof(double2) * c->n_bf, cudaMemcpyHostToDevice, s));
    SSB_CK_BAIL(cudaMemcpyAsync(c->tw, tw.data(), sizeof(float2) * N, cudaMemcpyHostToDevice, s));
    SSB_CK_BAIL(cudaMemsetAsync(c->flag, 0, sizeof(int), s));

    // counts -> float32 -> G, in chunks of BF planes
    const size_t esz = dtype == SSB_U16 ? 2 : 4;
    const size_t per_bf = P * esz + P * sizeof(float) + (size_t)H * N * sizeof(float2);
    const int KC = (int)std::max<size_t>(1, std::min<size_t>((size_t)c->n_bf, (256u << 20) / per_bf));
    void *raw = nullptr;
    float *F = nullptr;
    float2 *tmp = nullptr;
    auto free_stage = [&]() {
        if (raw) cudaFree(raw);
        if (F) cudaFree(F);
        if (tmp) cudaFree(tmp);
        raw = nullptr;
        F = nullptr;
        tmp = nullptr;
    };
    if (!counts_on_device && (e = cudaMalloc(&raw, (size_t)KC * P * esz)) != cudaSuccess) {
        free_stage();
        return bail(cuda_fail(e, "cudaMalloc counts staging"));
    }
    if ((e = cudaMalloc((void **)&F, (size_t)KC * P * sizeof(float))) != cudaSuccess ||
        (e = cudaMalloc((void **)&tmp, (size_t)KC * H * N * sizeof(float2))) != cudaSuccess) {
        free_stage();
        return bail(cuda_fail(e, "cudaMalloc prepare staging"));
    }
    for (int k0 = 0; k0 < c->n_bf; k0 += KC) {
        const int kc = std::min(KC, c->n_bf - k0);
        const char *src = (const char *)counts + (size_t)k0 * P * esz;
        const void *dsrc = src;
        if (!counts_on_device) {
            if ((e = cudaMemcpyAsync(raw, src, (size_t)kc * P * esz, cudaMemcpyHostToDevice, s)) !=
                cudaSuccess) {
                free_stage();
                return bail(cuda_fail(e, "counts host-to-device copy"));
            }
            dsrc = raw;
        }
        if ((e = launch_unpack(dsrc, dtype, (size_t)kc * P, F, c->flag, s)) != cudaSuccess ||
            (e = launch_rfft2(N, F, tmp, c->G + (size_t)k0 * H * N, kc, c->tw, s)) != cudaSuccess) {
            free_stage();
            return bail(cuda_fail(e, "G cache build"));
        }
    }
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) {
        free_stage();
        return bail(cuda_fail(e, "prepare synchronise"));
    }
    free_stage();
    if ((st = check_flag(c, s)) != SSB_OK) return bail(st);
    *out = c;
    return SSB_OK;
#undef SSB_ALLOC
#undef SSB_CK_BAIL
}

ssb_status ssb_loss_batch(ssb_ctx *c, const ssb_params *theta, int T, double *loss_out,
                          void *cuda_stream) {
    g_last_error.clear();
    if (!c || !theta || !loss_out) return fail(SSB_ERR_ARG, "NULL argument");
    if (T < 1) return fail(SSB_ERR_ARG, "T must be >= 1");
    for (int t = 0; t < T; ++t)
        if (!valid_theta(theta[t])) return fail(SSB_ERR_ARG, "non-finite theta");
    DeviceGuard dg(c->dev);
    if (!dg.ok) return fail(SSB_ERR_CUDA, "cannot select the context's device");
    cudaStream_t s = (cudaStream_t)cuda_stream;
    ssb_status st = begin_call(c, s);
    if (st != SSB_OK) return st;
    // Consecutive trials alternate between the caller's stream (buffer set 0) and the
    // context's second stream (set 1), so that the end of one persistent launch, where its
    // last row tasks leave most SMs idle, overlaps the per-trial tables and the first
    // column tasks of the next.  Each trial's arithmetic is the same as a scalar call's.
    for (int t0 = 0; t0 < T; t0 += c->loss_cap) {
        const int tn = std::min(c->loss_cap, T - t0);
        const bool overlap = tn >= 2;
        if (overlap) {
            SSB_CK(cudaEventRecord(c->ev_fork, s));
            SSB_CK(cudaStreamWaitEvent(c->aux, c->ev_fork, 0));
        }
        for (int t = 0; t < tn; ++t) {
            const int si = overlap ? (t & 1) : 0;
            cudaError_t e = evaluate(c, theta[t0 + t], c->loss + t, false, si ? c->aux : s, t0 + t, si);
            if (e != cudaSuccess) return cuda_fail(e, "objective launch");
        }
        if (overlap) {
            SSB_CK(cudaEventRecord(c->ev_join, c->aux));
            SSB_CK(cudaStreamWaitEvent(s, c->ev_join, 0));
        }
        SSB_CK(cudaMemcpyAsync(loss_out + t0, c->loss, sizeof(double) * tn, cudaMemcpyDeviceToHost, s));
        // the error word is cleared once per call, so this sees a wait that ran out in any
        // trial so far (those trials and all later ones of the chunk have NaN losses); the
        // chunks after it are not evaluated and their losses are NaN too
        if ((st = check_sync(c, s)) != SSB_OK) {
            for (int t = t0 + tn; t < T; ++t) loss_out[t] = std::numeric_limits<double>::quiet_NaN();
            return st;
        }
    }
    return SSB_OK;
}

ssb_status ssb_reconstruct(ssb_ctx *c, const ssb_params *theta, float *mean_phase_out,
                           float *object_c64_out, double *loss_out, void *cuda_stream) {
    g_last_error.clear();
    if (!c || !theta || !mean_phase_out) return fail(SSB_ERR_ARG, "NULL argument");
    if (!valid_theta(*theta)) return fail(SSB_ERR_ARG, "non-finite theta");
    DeviceGuard dg(c->dev);
    if (!dg.ok) return fail(SSB_ERR_CUDA, "cannot select the context's device");
    cudaStream_t s = (cudaStream_t)cuda_stream;
    const ObjectiveArgs a = c->args();
    ssb_status st = begin_call(c, s);
    if (st != SSB_OK) return st;
    cudaError_t e = evaluate(c, *theta, c->loss, object_c64_out != nullptr, s);
    if (e != cudaSuccess) return cuda_fail(e, "objective launch");
    if ((e = launch_finalize(a, mean_phase_out, object_c64_out, s)) != cudaSuccess)
        return cuda_fail(e, "finalize launch");
    if (loss_out) {
        SSB_CK(cudaMemcpyAsync(loss_out, c->loss, sizeof(double), cudaMemcpyDeviceToHost, s));
    }
    SSB_CK(cudaStreamSynchronize(s));
    return check_sync(c, s);
}

// Interpolation table and intermediate for `factor` (regrown for a larger factor).
static ssb_status ensure_upsample(ssb_ctx *c, int factor, cudaStream_t s) {
    if (factor == c->up_factor && c->up_T && c->up_tab) return SSB_OK;
    SSB_CK(cudaStreamSynchronize(s));
    if (factor > c->up_factor || !c->up_T) {
        if (c->up_T) cudaFree(c->up_T);
        c->up_T = nullptr;
        if (cudaMalloc((void **)&c->up_T, sizeof(float2) * upsample_scratch_elems(c->N, factor)) !=
            cudaSuccess) {
            cudaGetLastError();
            c->up_factor = 0;
            return fail(SSB_ERR_OOM, "cannot allocate the upsampling scratch");
        }
    }
    if (c->up_tab) cudaFree(c->up_tab);
    c->up_tab = nullptr;
    std::vector<float2> tab;
    upsample_table(c->N, factor, tab);
    if (cudaMalloc((void **)&c->up_tab, sizeof(float2) * tab.size()) != cudaSuccess) {
        cudaGetLastError();
        c->up_factor = 0;
        return fail(SSB_ERR_OOM, "cannot allocate the interpolation table");
    }
    SSB_CK(cudaMemcpy(c->up_tab, tab.data(), sizeof(float2) * tab.size(), cudaMemcpyHostToDevice));
    c->up_factor = factor;
    return SSB_OK;
}

// Slice sums, spectral sum and transform buffers of the redraw without the loss.
static ssb_status ensure_redraw(ssb_ctx *c) {
    if (c->rd_part && c->rd_S && c->rd_T) return SSB_OK;
    const size_t P = (size_t)c->N * c->N;
    if (cudaMalloc((void **)&c->rd_part, sizeof(double2) * redraw_part_elems(c->N, c->n_bf)) != cudaSuccess ||
        cudaMalloc((void **)&c->rd_S, sizeof(float2) * P) != cudaSuccess ||
        cudaMalloc((void **)&c->rd_T, sizeof(float2) * P) != cudaSuccess) {
        cudaGetLastError();
        void *ptrs[] = {c->rd_part, c->rd_S, c->rd_T};
        for (void *q : ptrs)
            if (q) cudaFree(q);
        c->rd_part = nullptr;
        c->rd_S = c->rd_T = nullptr;
        return fail(SSB_ERR_OOM, "cannot allocate the redraw scratch");
    }
    return SSB_OK;
}

ssb_status ssb_reconstruct_upsampled(ssb_ctx *c, const ssb_params *theta, int factor,
                                     float *phase_out, float *object_c64_out, double *loss_out,
                                     void *cuda_stream) {
    g_last_error.clear();
    if (!c || !theta || !phase_out) return fail(SSB_ERR_ARG, "NULL argument");
    if (factor < 1 || factor > SSB_MAX_UPSAMPLE)
        return fail(SSB_ERR_ARG, "upsampling factor must be in 1.." + std::to_string(SSB_MAX_UPSAMPLE));
    if (!valid_theta(*theta)) return fail(SSB_ERR_ARG, "non-finite theta");
    DeviceGuard dg(c->dev);
    if (!dg.ok) return fail(SSB_ERR_CUDA, "cannot select the context's device");
    cudaStream_t s = (cudaStream_t)cuda_stream;
    ssb_status st = ensure_upsample(c, factor, s);
    if (st != SSB_OK) return st;
    if ((st = begin_call(c, s)) != SSB_OK) return st;
    const ObjectiveArgs a = c->args();
    cudaError_t e = evaluate(c, *theta, c->loss, true, s);
    if (e != cudaSuccess) return cuda_fail(e, "objective launch");
    if ((e = launch_upsample(a, factor, c->up_tab, c->up_T, phase_out, (float2 *)object_c64_out, s)) !=
        cudaSuccess)
        return cuda_fail(e, "upsampling launch");
    if (loss_out) {
        SSB_CK(cudaMemcpyAsync(loss_out, c->loss, sizeof(double), cudaMemcpyDeviceToHost, s));
    }
    SSB_CK(cudaStreamSynchronize(s));
    return check_sync(c, s);
}

ssb_status ssb_redraw(ssb_ctx *c, const ssb_params *theta, int factor, float *phase_out,
                      float *object_c64_out, void *cuda_stream) {
    g_last_error.clear();
    if (!c || !theta || !phase_out) return fail(SSB_ERR_ARG, "NULL argument");
    if (factor < 1 || factor > SSB_MAX_UPSAMPLE)
        return fail(SSB_ERR_ARG, "upsampling factor must be in 1.." + std::to_string(SSB_MAX_UPSAMPLE));
    if (!valid_theta(*theta)) return fail(SSB_ERR_ARG, "non-finite theta");
    DeviceGuard dg(c->dev);
    if (!dg.ok) return fail(SSB_ERR_CUDA, "cannot select the context's device");
    cudaStream_t s = (cudaStream_t)cuda_stream;
    ssb_status st = ensure_redraw(c);
    if (st != SSB_OK) return st;
    if (factor > 1 && (st = ensure_upsample(c, factor, s)) != SSB_OK) return st;
    const ObjectiveArgs a = c->args();
    cudaError_t e = launch_redraw(a, *theta, c->rd_part, c->rd_S, c->rd_T,
                                  factor == 1 ? phase_out : nullptr,
                                  factor == 1 ? (float2 *)object_c64_out : nullptr, s);
    if (e != cudaSuccess) return cuda_fail(e, "redraw launch");
    if (factor > 1 &&
        (e = launch_upsample(a, factor, c->up_tab, c->up_T, phase_out, (float2 *)object_c64_out, s)) !=
            cudaSuccess)
        return cuda_fail(e, "upsampling launch");
    SSB_CK(cudaStreamSynchronize(s));
    return SSB_OK;
}

// Reads back the events a profiled call recorded: per kernel name, launches and summed ms.
static ssb_status collect_profile(Profiler &prof, cudaError_t e, ssb_kernel_time *out, int cap,
                                  int *n_out, const char *what) {
    std::vector<ssb_kernel_time> agg;
    for (auto &r : prof.recs) {
        float ms = 0.f;
        if (e == cudaSuccess) e = cudaEventSynchronize(r.b);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.a, r.b);
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
        size_t j = 0;
        while (j < agg.size() && r.name != agg[j].name) ++j;
        if (j == agg.size()) {
            ssb_kernel_time t;
            std::memset(&t, 0, sizeof(t));
            std::strncpy(t.name, r.name.c_str(), sizeof(t.name) - 1);
            agg.push_back(t);
        }
        agg[j].launches += 1;
        agg[j].ms += ms;
    }
    if (e != cudaSuccess) return cuda_fail(e, what);
    *n_out = (int)agg.size();
    for (int j = 0; j < (int)agg.size() && j < cap; ++j) out[j] = agg[j];
    return SSB_OK;
}

ssb_status ssb_profile_objective(ssb_ctx *c, const ssb_params *theta, ssb_kernel_time *out,
                                 int cap, int *n_out, void *cuda_stream) {
    g_last_error.clear();
    if (!c || !theta || !n_out || (cap > 0 && !out) || cap < 0) return fail(SSB_ERR_ARG, "bad argument");
    if (!valid_theta(*theta)) return fail(SSB_ERR_ARG, "non-finite theta");
    DeviceGuard dg(c->dev);
    if (!dg.ok) return fail(SSB_ERR_CUDA, "cannot select the context's device");
    cudaStream_t s = (cudaStream_t)cuda_stream;
    if (g_prof) return fail(SSB_ERR_ARG, "a profiling session is open on this thread");
    ssb_status st = begin_call(c, s);
    if (st != SSB_OK) return st;
    Profiler prof;
    g_prof = &prof;
    cudaError_t e = evaluate(c, *theta, c->loss, false, s);
    g_prof = nullptr;
    if ((st = collect_profile(prof, e, out, cap, n_out, "profiled objective")) != SSB_OK) return st;
    return check_sync(c, s);
}

static thread_local Profiler *g_session = nullptr;

ssb_status ssb_profile_begin(void) {
    g_last_error.clear();
    if (g_prof) return fail(SSB_ERR_ARG, "a profiling session is already open on this thread");
    g_session = new (std::nothrow) Profiler;
    if (!g_session) return fail(SSB_ERR_OOM, "cannot allocate the profiler");
    g_prof = g_session;
    return SSB_OK;
}

ssb_status ssb_profile_end(ssb_kernel_time *out, int cap, int *n_out) {
    g_last_error.clear();
    if (!g_session || g_prof != g_session) return fail(SSB_ERR_ARG, "no profiling session is open on this thread");
    g_prof = nullptr;
    Profiler *prof = g_session;
    g_session = nullptr;
    ssb_status st;
    if (!n_out || cap < 0 || (cap > 0 && !out)) {
        for (auto &r : prof->recs) {
            cudaEventSynchronize(r.b);
            cudaEventDestroy(r.a);
            cudaEventDestroy(r.b);
        }
        st = fail(SSB_ERR_ARG, "bad argument");
    } else {
        st = collect_profile(*prof, cudaSuccess, out, cap, n_out, "profiling session");
    }
    delete prof;
    return st;
}

ssb_status ssb_info(const ssb_ctx *c, size_t *g_bytes, size_t *scratch_bytes) {
    if (!c) return fail(SSB_ERR_ARG, "NULL context");
    if (g_bytes) *g_bytes = c->g_bytes;
    if (scratch_bytes) *scratch_bytes = c->scratch_bytes;
    return SSB_OK;
}

ssb_status ssb_export_g(const ssb_ctx *c, void *dst, int dst_on_device, void *cuda_stream) {
    g_last_error.clear();
    if (!c || !dst) return fail(SSB_ERR_ARG, "NULL argument");
    DeviceGuard dg(c->dev);
    if (!dg.ok) return fail(SSB_ERR_CUDA, "cannot select the context's device");
    cudaStream_t s = (cudaStream_t)cuda_stream;
    SSB_CK(cudaMemcpyAsync(dst, c->G, c->g_bytes,
                           dst_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost, s));
    SSB_CK(cudaStreamSynchronize(s));
    return SSB_OK;
}

ssb_status ssb_unpack_counts(const void *in_device, ssb_dtype dtype, size_t n, float *out_device,
                             void *cuda_stream) {
    g_last_error.clear();
    if ((!in_device || !out_device) && n > 0) return fail(SSB_ERR_ARG, "NULL argument");
    if (dtype != SSB_U16 && dtype != SSB_U32) return fail(SSB_ERR_ARG, "unknown dtype");
    if (n == 0) return SSB_OK;
    cudaStream_t s = (cudaStream_t)cuda_stream;
    int *flag = nullptr;
    SSB_CK(cudaMalloc((void **)&flag, sizeof(int)));
    cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(int), s);
    if (e == cudaSuccess) e = launch_unpack(in_device, dtype, n, out_device, flag, s);
    int h = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h, flag, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaFree(flag);
    if (e != cudaSuccess) return cuda_fail(e, "unpack");
    if (h & 1) return fail(SSB_ERR_ARG, "a count exceeds 2^24 and cannot be converted to float32 exactly");
    return SSB_OK;
}

ssb_status ssb_debug_stall_next(ssb_ctx *c, int evaluation, unsigned polls) {
    g_last_error.clear();
    if (!c) return fail(SSB_ERR_ARG, "NULL context");
    if (evaluation < 0) return fail(SSB_ERR_ARG, "evaluation must be >= 0");
    c->dbg_stall_eval = evaluation;
    c->dbg_wait_limit = polls ? polls : 1u;
    return SSB_OK;
}

ssb_status ssb_debug_poison_scratch(ssb_ctx *c, void *cuda_stream) {
    g_last_error.clear();
    if (!c) return fail(SSB_ERR_ARG, "NULL context");
    DeviceGuard dg(c->dev);
    if (!dg.ok) return fail(SSB_ERR_CUDA, "cannot select the context's device");
    cudaStream_t s = (cudaStream_t)cuda_stream;
    const size_t P = (size_t)c->N * c->N;
    const bool ssb1 = c->transfer == SSB_TRANSFER_SSB1;
    struct Buf {
        void *p;
        size_t bytes;
    };
    std::vector<Buf> bufs = {
        {c->Osum, P * sizeof(double2)},
        {c->loss, (size_t)c->loss_cap * sizeof(double)},
        {c->err, sizeof(unsigned)},
    };
    for (const TrialSet &t : c->set) {
        bufs.push_back({t.Zring, fused_ring_elems(c->N, c->Bk, c->D, ssb1) * sizeof(float2)});
        bufs.push_back({t.hring, fused_hring_elems(c->N, c->Bk, c->D) * sizeof(float2)});
        bufs.push_back({t.rring, fused_rring_elems(c->N, c->Bk, c->D) * sizeof(float2)});
        bufs.push_back({t.S2g, fused_s2g_elems(c->N) * sizeof(double)});
        bufs.push_back({t.sync, fused_sync_words(c->N, c->n_bf, c->Bk) * sizeof(unsigned)});
        bufs.push_back({t.S1, P * sizeof(double)});
        bufs.push_back({t.E, P * sizeof(float2)});
        bufs.push_back({t.kturn, (size_t)c->n_bf * sizeof(uint2)});
    }
    for (const Buf &b : bufs) SSB_CK(cudaMemsetAsync(b.p, 0xff, b.bytes, s));
    SSB_CK(cudaStreamSynchronize(s));
    return SSB_OK;
}

void ssb_destroy(ssb_ctx *c) {
    if (!c) return;
    DeviceGuard dg(c->dev);
    cudaDeviceSynchronize();
    free_ctx(c);
}

}  // extern "C"
