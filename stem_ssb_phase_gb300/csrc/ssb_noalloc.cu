// ssb_loss_noalloc: the SSB2 objective for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they need a loss: real-time
// pipelines that plan all device memory up front and forbid allocation afterwards (an
// allocation can block on the driver and break their timing), and plug-ins that live
// inside a host application which owns the GPU memory through its own allocator (memory
// taken behind its back can make the host's own allocations fail).  This entry point
// serves them: every byte of
// scratch it needs (per-trial tables, per-BF geometry, the column-to-row ring, the
// accumulators and the scheduler words) lives in one file-scope device array of fixed
// size, reserved when the library's device code is loaded on a GPU and kept until the
// process exits.  It runs the same persistent kernel as ssb_loss_batch, with a smaller
// batch and ring so that the whole scratch stays modest.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "ssb_internal.h"

namespace ssb {

constexpr size_t kNoallocScratchBytes = 24u << 20;  // 24 MiB
constexpr int kNoallocMaxBF = 16384;
constexpr int kNoallocBk = 4;    // BF planes per batch
constexpr int kNoallocRing = 3;  // ring slots
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a stand-in for the symbol, never a device
// address: host code obtains the address with cudaGetSymbolAddress (below).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Per device: the scratch's device address and the id of the context it was looked up in.
static void *g_scratch_addr[kMaxDevices];
static unsigned long long g_scratch_ctx[kMaxDevices];
static std::mutex g_scratch_mu;

// Unique id of the current context (0 if the driver cannot say); a device whose context was
// destroyed (cudaDeviceReset) and created again gets a new id, and its module a new address.
static unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

// Device address of the scratch on the current device.  Set-up: looked up with
// cudaGetSymbolAddress on the first call on each device (with that device current), and
// again whenever the device's context has changed since (after cudaDeviceReset).
static cudaError_t scratch_base(unsigned char **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const unsigned long long ctx = current_context_id();  // 0 before the context exists
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // creates the context if needed
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx ? ctx : current_context_id();
    }
    *out = (unsigned char *)g_scratch_addr[dev];
    return cudaSuccess;
}

struct NoallocLayout {
    size_t E, S1, Z, h, rp, S2g, kgeo, kalpha, kturn, yx, tw, loss, err, sync, total;
};

static size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

static NoallocLayout noalloc_layout(int N, int n_bf) {
    NoallocLayout L;
    const size_t P = (size_t)N * N;
    const int bk = n_bf < kNoallocBk ? n_bf : kNoallocBk;
    size_t o = 0;
    L.E = o;      o = up256(o + P * sizeof(float2));
    L.S1 = o;     o = up256(o + P * sizeof(double));
    L.Z = o;      o = up256(o + fused_ring_elems(N, bk, kNoallocRing) * sizeof(float2));
    L.h = o;      o = up256(o + fused_hring_elems(N, bk, kNoallocRing) * sizeof(float2));
    L.rp = o;     o = up256(o + fused_rring_elems(N, bk, kNoallocRing) * sizeof(float2));
    L.S2g = o;    o = up256(o + fused_s2g_elems(N) * sizeof(double));
    L.kgeo = o;   o = up256(o + (size_t)n_bf * sizeof(float4));
    L.kalpha = o; o = up256(o + (size_t)n_bf * sizeof(double2));
    L.kturn = o;  o = up256(o + (size_t)n_bf * sizeof(uint2));
    L.yx = o;     o = up256(o + (size_t)n_bf * 2 * sizeof(float));
    L.tw = o;     o = up256(o + (size_t)N * sizeof(float2));
    L.loss = o;   o = up256(o + sizeof(double));
    L.err = o;    o = up256(o + sizeof(unsigned));
    L.sync = o;   o = up256(o + fused_sync_words(N, n_bf, bk) * sizeof(unsigned));
    L.total = o;
    return L;
}

// Per-BF angles and aperture amplitude (the same float64 arithmetic as ssb_prepare).
__global__ void k_noalloc_geometry(const float *__restrict__ yx, int n_bf, double dalpha,
                                   double semi, float4 *__restrict__ kgeo,
                                   double2 *__restrict__ kalpha) {
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= n_bf) return;
    const double ay = (double)yx[2 * k] * dalpha;
    const double ax = (double)yx[2 * k + 1] * dalpha;
    const double r = sqrt(ax * ax + ay * ay);
    double amp = fmin(1.0, fmax(0.0, (semi - r) / dalpha + 0.5));
    if (amp < 1.0 / 65536.0) amp = 0.0;
    kgeo[k] = make_float4((float)ax, (float)ay, (float)amp, 0.f);
    kalpha[k] = make_double2(ax, ay);
}

__global__ void k_noalloc_twiddles(float2 *__restrict__ tw, int N) {
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    if (m >= N) return;
    double s, c;
    sincospi(2.0 * m / N, &s, &c);
    tw[m] = make_float2((float)c, (float)s);
}

}  // namespace ssb

using namespace ssb;

extern "C" ssb_status ssb_loss_noalloc(const ssb_geometry *g, const void *g_cache_device,
                                       const ssb_params *theta, double *loss_out,
                                       void *cuda_stream) {
    auto fail = [](ssb_status st, const char *msg) {
        set_last_error(msg);
        return st;
    };
    set_last_error("");
    if (!g || !g_cache_device || !theta || !loss_out) return fail(SSB_ERR_ARG, "NULL argument");
    const int N = g->scan_n;
    if (N != 32 && N != 64 && N != 128 && N != 256 && N != 512)
        return fail(SSB_ERR_UNSUPPORTED, "scan_n must be 32, 64, 128, 256 or 512");
    if (g->n_bf < 1 || !g->bf_det_yx) return fail(SSB_ERR_ARG, "n_bf must be >= 1 with bf_det_yx");
    if (g->n_bf > kNoallocMaxBF)
        return fail(SSB_ERR_ARG, "n_bf exceeds the no-allocation limit of 16384 BF pixels");
    auto pos = [](double v) { return v > 0.0 && v < 1e300; };
    if (!pos(g->scan_step_A) || !pos(g->wavelength_A) || !pos(g->semiangle_mrad) ||
        !pos(g->det_sampling_mrad))
        return fail(SSB_ERR_ARG, "geometry scalars must be finite and positive");
    for (int k = 0; k < 2 * g->n_bf; ++k)
        if (!(g->bf_det_yx[k] == g->bf_det_yx[k]) || g->bf_det_yx[k] > 1e30f || g->bf_det_yx[k] < -1e30f)
            return fail(SSB_ERR_ARG, "bf_det_yx has a non-finite entry");
    const double tv[4] = {theta->C10_nm, theta->C12_nm, theta->phi12_rad, theta->rotation_rad};
    for (double v : tv)
        if (!(v == v) || v > 1e300 || v < -1e300) return fail(SSB_ERR_ARG, "non-finite theta");
    const NoallocLayout L = noalloc_layout(N, g->n_bf);
    if (L.total > kNoallocScratchBytes)
        return fail(SSB_ERR_ARG, "problem exceeds the 24 MiB no-allocation scratch");

    cudaStream_t s = (cudaStream_t)cuda_stream;
    unsigned char *base = nullptr;
    cudaError_t e = scratch_base(&base);
    if (e != cudaSuccess) return fail(SSB_ERR_CUDA, "cudaGetSymbolAddress of the scratch failed");

    ObjectiveArgs a;
    std::memset(&a, 0, sizeof(a));
    a.N = N;
    a.n_bf = g->n_bf;
    a.G = (const float2 *)g_cache_device;
    a.kgeo = (const float4 *)(base + L.kgeo);
    a.kalpha = (const double2 *)(base + L.kalpha);
    a.kturn = (uint2 *)(base + L.kturn);
    a.E = (float2 *)(base + L.E);
    a.tw = (const float2 *)(base + L.tw);
    a.S1 = (double *)(base + L.S1);
    a.loss = (double *)(base + L.loss);
    a.Zring = (float2 *)(base + L.Z);
    a.hring = (float2 *)(base + L.h);
    a.rring = (float2 *)(base + L.rp);
    a.S2g = (double *)(base + L.S2g);
    a.sync = (unsigned *)(base + L.sync);
    a.err = (unsigned *)(base + L.err);
    a.Bk = g->n_bf < kNoallocBk ? g->n_bf : kNoallocBk;
    a.D = kNoallocRing;
    a.mode = 0;
    a.step = g->scan_step_A;
    a.lam = g->wavelength_A;
    a.semi = g->semiangle_mrad * 1e-3;
    a.dalpha = g->det_sampling_mrad * 1e-3;

    // per-BF geometry and twiddles into the scratch, and the error word cleared (the
    // accumulators and the other scheduler words are cleared by the objective itself)
    e = cudaMemcpyAsync(base + L.yx, g->bf_det_yx, sizeof(float) * 2 * (size_t)g->n_bf,
                        cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.err, 0, sizeof(unsigned), s);
    if (e == cudaSuccess) {
        k_noalloc_geometry<<<(g->n_bf + 127) / 128, 128, 0, s>>>(
            (const float *)(base + L.yx), g->n_bf, a.dalpha, a.semi, (float4 *)(base + L.kgeo),
            (double2 *)(base + L.kalpha));
        count_launch();
        k_noalloc_twiddles<<<(N + 127) / 128, 128, 0, s>>>((float2 *)(base + L.tw), N);
        count_launch();
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = run_objective_fused(a, *theta, a.loss, false, s);
    // the loss and the error word land in host locals; *loss_out is written only on success
    unsigned err_word = 0;
    double loss = 0.0;
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&loss, a.loss, sizeof(double), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&err_word, a.err, sizeof(unsigned), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return fail(SSB_ERR_CUDA, cudaGetErrorString(e));
    }
    if (err_word) return fail(SSB_ERR_TIMEOUT, "a scheduler wait in the fused objective kernel ran out");
    *loss_out = loss;
    return SSB_OK;
}
