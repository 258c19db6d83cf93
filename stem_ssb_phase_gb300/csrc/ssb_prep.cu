// G-cache builder: integer counts -> float32 -> Hermitian half-plane rfft2 over the scan.
//
// Page "SSB performance notes" (BF-major G_qk materialisation): one rfft2 over the scan
// per BF column gives the Hermitian (N, N/2+1) complex64 evidence, made BF-major once.
// This build stores it [k][Qx = 0..N/2][Qy = 0..N-1] with Qy contiguous so that the
// objective's column pass reads each half-plane column as one contiguous run.
#include <algorithm>

#include "ssb_device.cuh"
#include "ssb_internal.h"

namespace ssb {

template <typename T>
__global__ void k_unpack(const T *__restrict__ in, float *__restrict__ out, size_t n,
                         int *__restrict__ flag) {
    bool bad = false;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const uint32_t v = (uint32_t)in[i];
        bad |= v > (1u << 24);
        out[i] = (float)v;  // exact for v <= 2^24
    }
    if (bad) atomicOr(flag, 1);
}

cudaError_t launch_unpack(const void *raw, ssb_dtype dtype, size_t n, float *out, int *flag,
                          cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const size_t want = (n + threads - 1) / threads;
    const int blocks = (int)std::min<size_t>(want, 152 * 16);
    if (dtype == SSB_U16)
        k_unpack<uint16_t><<<blocks, threads, 0, s>>>((const uint16_t *)raw, out, n, flag);
    else
        k_unpack<uint32_t><<<blocks, threads, 0, s>>>((const uint32_t *)raw, out, n, flag);
    count_launch();
    return cudaGetLastError();
}

template <int N>
constexpr int prep_rows() { return N >= 512 ? 8 : (N >= 256 ? 16 : (N >= 128 ? 32 : N)); }

// Forward FFT along x of RW scan rows of one BF plane; keeps Qx = 0..N/2 and writes them
// transposed, tmp[kc][Qx][ry], so the column pass reads contiguous runs.
template <int N>
__global__ void __launch_bounds__(256) k_prep_rows(const float *__restrict__ F,
                                                   float2 *__restrict__ tmp,
                                                   const float2 *__restrict__ twg) {
    constexpr int RW = prep_rows<N>();
    constexpr int H = N / 2 + 1;
    extern __shared__ float2 sm[];
    float2 *tw = sm, *b0 = sm + N, *b1 = b0 + RW * N;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int kc = blockIdx.y, ry0 = blockIdx.x * RW;
    for (int i = tid; i < N; i += nt) tw[i] = twg[i];
    const float *src = F + ((size_t)kc * N + ry0) * N;
    for (int i = tid; i < RW * N; i += nt) b0[i] = make_float2(src[i], 0.0f);
    __syncthreads();
    const float2 *res = fft_batch_smem<N, -1>(b0, b1, RW, N, tw, tid, nt) ? b1 : b0;
    float2 *dst = tmp + (size_t)kc * H * N;
    for (int i = tid; i < RW * H; i += nt) {
        const int r = i % RW, qx = i / RW;
        dst[(size_t)qx * N + ry0 + r] = res[r * N + qx];
    }
}

// Forward FFT along y of RW half-plane columns: G[k][Qx][Qy].
template <int N>
__global__ void __launch_bounds__(256) k_prep_cols(const float2 *__restrict__ tmp,
                                                   float2 *__restrict__ G,
                                                   const float2 *__restrict__ twg) {
    constexpr int RW = prep_rows<N>();
    constexpr int H = N / 2 + 1;
    extern __shared__ float2 sm[];
    float2 *tw = sm, *b0 = sm + N, *b1 = b0 + RW * N;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int kc = blockIdx.y, q0 = blockIdx.x * RW;
    const int nq = min(RW, H - q0);
    for (int i = tid; i < N; i += nt) tw[i] = twg[i];
    const float2 *src = tmp + ((size_t)kc * H + q0) * N;
    for (int i = tid; i < RW * N; i += nt) b0[i] = i < nq * N ? src[i] : make_float2(0.f, 0.f);
    __syncthreads();
    const float2 *res = fft_batch_smem<N, -1>(b0, b1, RW, N, tw, tid, nt) ? b1 : b0;
    float2 *dst = G + ((size_t)kc * H + q0) * N;
    for (int i = tid; i < nq * N; i += nt) dst[i] = res[i];
}

template <int N>
static cudaError_t rfft2_n(const float *F, float2 *tmp, float2 *G, int kc, const float2 *tw,
                           cudaStream_t s) {
    constexpr int RW = prep_rows<N>();
    constexpr int H = N / 2 + 1;
    const size_t smem = (size_t)(N + 2 * RW * N) * sizeof(float2);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k_prep_rows<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(k_prep_cols<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
        return e;
    k_prep_rows<N><<<dim3(N / RW, kc), 256, smem, s>>>(F, tmp, tw);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k_prep_cols<N><<<dim3((H + RW - 1) / RW, kc), 256, smem, s>>>(tmp, G, tw);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_rfft2(int N, const float *F, float2 *tmp, float2 *G, int kc,
                         const float2 *tw, cudaStream_t s) {
    switch (N) {
        case 32: return rfft2_n<32>(F, tmp, G, kc, tw, s);
        case 64: return rfft2_n<64>(F, tmp, G, kc, tw, s);
        case 128: return rfft2_n<128>(F, tmp, G, kc, tw, s);
        case 256: return rfft2_n<256>(F, tmp, G, kc, tw, s);
        case 512: return rfft2_n<512>(F, tmp, G, kc, tw, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssb
