// CUDA-core local GEMM: the per-rank product C_r = A_r . B_r over the rank's
// slice of the contracted dim ("Sharded matrix multiplication and result
// ownership", step 3; "Row Parallelism", Z_i = X_i A_i), with fp32 FMA
// accumulation.  It serves fp32 inputs and bf16 shapes whose rows TMA cannot
// address (a row pitch that is not a multiple of 16 bytes); every other bf16
// product runs on the tensor cores (gemm_tcgen05.cu).
//
// Fused mode sums the G products of a reduction group in ascending rank
// order (each rank's product finished in its own fp32 accumulator first),
// which equals the standalone reduction of the unfused partials bit for bit.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "checked.cuh"
#include "gelu.cuh"
#include "pdl.cuh"
#include "shmm_internal.h"

namespace {

using shmm_dev::in_bounds;

constexpr int BM = 64, BN = 64, BK = 16, TM = 4, TN = 4;

struct SimtK {
    const void *A[SHMM_MAX_RANKS];
    const void *B[SHMM_MAX_RANKS];
    void *out[SHMM_MAX_RANKS];
    int G, mode;
    bool fused, gelu;
    int64_t M, N, Kd;
    int *status;               // device status word (bounds-checked build)
    int64_t a_n, b_n, out_n;   // elements per A, B and output buffer
};

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ void put(T *p, float v);
template <> __device__ __forceinline__ void put<float>(float *p, float v) { *p = v; }
template <> __device__ __forceinline__ void put<__nv_bfloat16>(__nv_bfloat16 *p, float v) {
    *p = __float2bfloat16_rn(v);
}


// One 64x64 output tile of one rank's product into acc (fp32, ascending k).
// The k-tiles are software-pipelined: all of a tile's global loads are
// issued at once into registers, and the next tile's loads are in flight
// while the current one is multiplied from shared memory.  (Loading element
// by element into shared memory put one memory latency per element on the
// critical path: 32 us for a single 64x64x64 tile.)  256 threads.
template <typename IT>
__device__ __forceinline__ void tile_product(const SimtK &k, const IT *__restrict__ A, const IT *__restrict__ B,
                                             int64_t M, int64_t N, int64_t Kd, int64_t m0, int64_t n0,
                                             float (*As)[BM], float (*Bs)[BN], float acc[TM][TN]) {
    constexpr int LA = BM * BK / 256, LB = BK * BN / 256;  // elements per thread
    const int tid = threadIdx.x;
    const int tr = tid / (BN / TN), tc = tid % (BN / TN);
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;
    float ra[LA], rb[LB];
    // A tile: BM x BK (stored transposed); B tile: BK x BN; zero-filled
    // outside the matrices
    auto load = [&](int64_t k0) {
#pragma unroll
        for (int i = 0; i < LA; ++i) {
            const int idx = tid + i * 256, r = idx / BK, c = idx % BK;
            const int64_t gr = m0 + r, gc = k0 + c;
            ra[i] = (gr < M && gc < Kd && in_bounds(k.status, gr * Kd + gc, 1, k.a_n)) ? to_f(A[gr * Kd + gc]) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < LB; ++i) {
            const int idx = tid + i * 256, r = idx / BN, c = idx % BN;
            const int64_t gr = k0 + r, gc = n0 + c;
            rb[i] = (gr < Kd && gc < N && in_bounds(k.status, gr * N + gc, 1, k.b_n)) ? to_f(B[gr * N + gc]) : 0.0f;
        }
    };
    load(0);
    for (int64_t k0 = 0; k0 < Kd; k0 += BK) {
#pragma unroll
        for (int i = 0; i < LA; ++i) {
            const int idx = tid + i * 256;
            As[idx % BK][idx / BK] = ra[i];
        }
#pragma unroll
        for (int i = 0; i < LB; ++i) {
            const int idx = tid + i * 256;
            Bs[idx / BN][idx % BN] = rb[i];
        }
        __syncthreads();
        if (k0 + BK < Kd) load(k0 + BK);  // next tile's loads in flight during the FMAs
#pragma unroll 4
        for (int kk = 0; kk < BK; ++kk) {
            float a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = As[kk][tr * TM + i];
#pragma unroll
            for (int j = 0; j < TN; ++j) b[j] = Bs[kk][tc * TN + j];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
}

template <typename IT, typename OT>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const __grid_constant__ SimtK k) {
    shmm_pdl::pdl_enter();
    __shared__ float As[BK][BM];
    __shared__ float Bs[BK][BN];
    const int unit = blockIdx.z;
    const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
    const int tr = threadIdx.x / (BN / TN), tc = threadIdx.x % (BN / TN);
    const int G = k.fused ? k.G : 1;
    float sum[TM][TN];
    for (int q = 0; q < G; ++q) {
        float acc[TM][TN];
        tile_product<IT>(k, (const IT *)k.A[unit * G + q], (const IT *)k.B[unit * G + q], k.M, k.N,
                         k.Kd, m0, n0, As, Bs, acc);
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) sum[i][j] = (q == 0) ? acc[i][j] : sum[i][j] + acc[i][j];
    }
    // the epilogue runs once per tile: kept rolled, since a launch of a few
    // tiles waits mostly on fetching its code
#pragma unroll 1
    for (int i = 0; i < TM; ++i) {
        const int64_t row = m0 + tr * TM + i;
        if (row >= k.M) continue;
#pragma unroll 1
        for (int j = 0; j < TN; ++j) {
            const int64_t col = n0 + tc * TN + j;
            if (col >= k.N) continue;
            const float v = k.gelu ? gelu_tanh(sum[i][j]) : sum[i][j];
            if (!k.fused) {
                if (in_bounds(k.status, row * k.N + col, 1, k.out_n)) put<OT>((OT *)k.out[unit] + row * k.N + col, v);
            } else if (k.mode == 0) {  // 32-bit owner arithmetic: M, N < 2^31
                const uint32_t per = (uint32_t)(k.M / G), b = (uint32_t)row / per;
                const int64_t off = (int64_t)((uint32_t)row - b * per) * k.N + col;
                if (in_bounds(k.status, off, 1, k.out_n)) put<OT>((OT *)k.out[unit * G + b] + off, v);
            } else if (k.mode == 1) {
                const uint32_t per = (uint32_t)(k.N / G), b = (uint32_t)col / per;
                const int64_t off = row * per + ((uint32_t)col - b * per);
                if (in_bounds(k.status, off, 1, k.out_n)) put<OT>((OT *)k.out[unit * G + b] + off, v);
            } else if (in_bounds(k.status, row * k.N + col, 1, k.out_n)) {
                for (int b = 0; b < G; ++b) put<OT>((OT *)k.out[unit * G + b] + row * k.N + col, v);
            }
        }
    }
}

}  // namespace

namespace shmm {

int launch_gemm_simt(const GemmArgs &a, int *status, void *stream) {
    const int G = a.fused ? a.G : 1;
    if (a.units * G > SHMM_MAX_RANKS) return (int)cudaErrorInvalidValue;
    if (a.M == 0 || a.N == 0 || a.units == 0) return 0;
    SimtK k;
    for (int i = 0; i < a.units * G; ++i) {
        k.A[i] = a.A[i];
        k.B[i] = a.B[i];
    }
    for (int i = 0; i < (a.fused ? a.units * G : a.units); ++i) k.out[i] = a.out[i];
    k.G = G;
    k.mode = a.mode;
    k.fused = a.fused;
    k.gelu = a.gelu;
    k.M = a.M;
    k.N = a.N;
    k.Kd = a.Kd;
    k.status = status;
    k.a_n = a.M * a.Kd;
    k.b_n = a.Kd * a.N;
    k.out_n = a.fused && a.mode != 2 ? a.M * a.N / G : a.M * a.N;  // an owner's block, or a whole copy
    const int64_t gy = (a.M + BM - 1) / BM, gx = (a.N + BN - 1) / BN;
    if (gy > 65535 || a.M >= ((int64_t)1 << 31) || a.N >= ((int64_t)1 << 31))
        return (int)cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)a.units);
    cudaStream_t s = (cudaStream_t)stream;
    count_launch();
    using shmm_pdl::launch_pdl;
    cudaError_t e;
    if (a.in_dt == SHMM_F32 && a.out_dt == SHMM_F32) e = launch_pdl(gemm_simt_kernel<float, float>, grid, dim3(256), 0, s, k);
    else if (a.in_dt == SHMM_F32) e = launch_pdl(gemm_simt_kernel<float, __nv_bfloat16>, grid, dim3(256), 0, s, k);
    else if (a.out_dt == SHMM_F32) e = launch_pdl(gemm_simt_kernel<__nv_bfloat16, float>, grid, dim3(256), 0, s, k);
    else e = launch_pdl(gemm_simt_kernel<__nv_bfloat16, __nv_bfloat16>, grid, dim3(256), 0, s, k);
    return (int)e;
}

}  // namespace shmm
