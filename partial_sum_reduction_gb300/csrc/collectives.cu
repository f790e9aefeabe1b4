// On-device collectives between virtual ranks held on one GPU: the
// partial-sum reduce-scatter / all-reduce and the all-gather copy.
//
// Reduce-scatter sums partial results across an axis and leaves the output
// sharded; all-reduce gives every rank the full sum; all-gather reassembles a
// sharded array on every rank ("Sharding Matrix Multiply", Communication
// primitives; "Sharded matmuls and collectives on a torus", The four
// collectives).  On one GPU every rank's buffer is in the same HBM, so a
// collective is one HBM-bound pass: each thread reads the G ranks' 16-byte
// vectors at one position, adds them in fp32 and writes the result to the
// owner(s).  No ring schedule is needed.
//
// Summation order: ascending rank id, one fp32 rounding per addition (the
// canonical order), or a balanced pairwise tree over the ranks built from
// warp shuffles (lane q of a W-lane subgroup holds rank q; absent leaves are
// -0.0).  Both are fixed orders, so results are reproducible bit for bit.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>

#include "checked.cuh"
#include "device_wait.cuh"
#include "gelu.cuh"
#include "pdl.cuh"
#include "shmm_internal.h"

namespace {

using shmm_pdl::pdl_enter;
// Every collective kernel runs 256 threads and is a programmatic dependent
// launch (pdl.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, size_t smem, cudaStream_t s, Args... args) {
    return shmm_pdl::launch_pdl(kern, grid, dim3(256), smem, s, args...);
}

using shmm_dev::in_bounds;

constexpr int kMaxPtrs = SHMM_MAX_RANKS;

struct ReduceK {
    const void *src[kMaxPtrs];  // group-major: [g*G + q], q ascending rank
    void *dst[kMaxPtrs];        // [g*G + b]: owner of block b (RS) / member b (AR)
    int G, ngroups, mode;       // mode: 0 RS rows, 1 RS cols, 2 AR
    int64_t rows, cols, n;      // per-rank partial shape, n = rows*cols
    int64_t nvec;               // vectors per group (per rank's partial)
    int *status;                // device status word (bounds-checked build)
    int64_t src_n, dst_n;       // elements per source / destination buffer
};

struct GatherK {
    const void *src[kMaxPtrs];  // [g*G + p]: block at grid position p
    void *dst[kMaxPtrs];        // [g*G + m]: every member m
    int G, ngroups, blocks1;
    int64_t brows, bvecs;       // block rows, 16-byte vectors per block row
    int64_t full_vecs;          // vectors per row of the gathered box
    int64_t nvec;               // vectors per group = G * brows * bvecs
    int *status;                // device status word (bounds-checked build)
    int64_t src_n, dst_n;       // vectors (or elements) per shard / gathered box
};

// ---- 16-byte vectors of 4 fp32 or 8 bf16 values, widened to fp32 -------

template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void load(const void *p, float *v) {
        const float4 x = __ldcs(reinterpret_cast<const float4 *>(p));
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    }
    __device__ static void store(void *p, const float *v) {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(v[0], v[1], v[2], v[3]));
    }
    __device__ static float load1(const void *p) { return __ldcs(reinterpret_cast<const float *>(p)); }
    __device__ static void store1(void *p, float v) { *reinterpret_cast<float *>(p) = v; }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const void *p, float *v) {
        const uint4 x = __ldcs(reinterpret_cast<const uint4 *>(p));
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static void store(void *p, const float *v) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
        __stcs(reinterpret_cast<uint4 *>(p), make_uint4(w[0], w[1], w[2], w[3]));
    }
    __device__ static float load1(const void *p) {
        return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
    }
    __device__ static void store1(void *p, float v) {
        *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(v);
    }
};

// Stores NV consecutive fp32 values as OT with one or two vector stores
// (NV * sizeof(OT) is 8, 16 or 32 bytes; the address is aligned to it).
template <typename OT, int NV>
__device__ __forceinline__ void store_n(void *p, const float *v) {
    if constexpr (sizeof(OT) == 4) {
#pragma unroll
        for (int i = 0; i < NV; i += 4)
            __stcs(reinterpret_cast<float4 *>(p) + i / 4, make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
    } else {
        uint32_t w[NV / 2];
#pragma unroll
        for (int i = 0; i < NV / 2; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
        if constexpr (NV == 8) __stcs(reinterpret_cast<uint4 *>(p), make_uint4(w[0], w[1], w[2], w[3]));
        else __stcs(reinterpret_cast<uint2 *>(p), make_uint2(w[0], w[1]));
    }
}

// Destination owner b and element offset for element e of a partial.  IT is
// the index type: 32-bit whenever every index of the launch fits, since
// 64-bit integer division costs many times more instructions.
template <typename IT>
__device__ __forceinline__ void route(const ReduceK &k, IT e, int *b, IT *off) {
    if (k.mode == 0) {
        const IT per = (IT)(k.n / k.G);
        *b = (int)(e / per);
        *off = e - (IT)(*b) * per;
    } else if (k.mode == 1) {
        const IT cols = (IT)k.cols, per = (IT)(k.cols / k.G);
        const IT row = e / cols, col = e - row * cols;
        *b = (int)(col / per);
        *off = row * per + (col - (IT)(*b) * per);
    } else {
        *b = -1;
        *off = e;
    }
}

template <typename OT, int NV, typename IT>
__device__ __forceinline__ void write_out(const ReduceK &k, int g, IT e, float *s, bool gelu) {
    if (gelu)
#pragma unroll
        for (int i = 0; i < NV; ++i) s[i] = gelu_tanh(s[i]);
    int b;
    IT off;
    route<IT>(k, e, &b, &off);
    if (!in_bounds(k.status, (int64_t)off, NV, k.dst_n)) return;
    const int q0 = b >= 0 ? b : 0, q1 = b >= 0 ? b + 1 : k.G;
    for (int q = q0; q < q1; ++q) {
        OT *d = (OT *)k.dst[g * k.G + q] + off;
        if constexpr (NV == 1) Vec<OT>::store1(d, s[0]);
        else store_n<OT, NV>(d, s);
    }
}

// Rank sum over 16-byte vectors; group g = blockIdx.y.  GT > 0: group size
// known at compile time (all G loads issued before the adds); GT == 0:
// runtime G.  TREE (GT a power of two only): the G vectors held in registers
// are added as a balanced pairwise tree over the ranks in ascending order --
// the same tree, and the same bits, as the warp-shuffle kernel below, at the
// memory rate of the sequential order.
template <typename PT, typename OT, int GT, int UNROLL, typename IT, bool TREE = false>
__global__ void __launch_bounds__(256) reduce_seq_kernel(const __grid_constant__ ReduceK k, bool gelu) {
    pdl_enter();
    static_assert(!TREE || (GT > 0 && (GT & (GT - 1)) == 0), "register tree needs a power-of-two G");
    constexpr int V = Vec<PT>::N;
    const int G = GT > 0 ? GT : k.G;
    const int g = blockIdx.y;
    const IT total = (IT)k.nvec;
    const IT stride = (IT)gridDim.x * blockDim.x * UNROLL;
    const void *const *src = k.src + g * G;
    for (IT base = (IT)blockIdx.x * blockDim.x * UNROLL + threadIdx.x; base < total; base += stride) {
        float acc[UNROLL][V];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const IT v = base + (IT)u * blockDim.x;
            if (v >= total) continue;
            const IT e = v * V;
            if (!in_bounds(k.status, (int64_t)e, V, k.src_n)) {
#pragma unroll
                for (int i = 0; i < V; ++i) acc[u][i] = 0.0f;
                continue;
            }
            if constexpr (GT > 0) {
                float x[GT][V];
#pragma unroll
                for (int q = 0; q < GT; ++q) Vec<PT>::load((const PT *)src[q] + e, x[q]);
                if constexpr (TREE) {
#pragma unroll
                    for (int w = GT; w > 1; w >>= 1)
#pragma unroll
                        for (int r = 0; r < w / 2; ++r)
#pragma unroll
                            for (int i = 0; i < V; ++i) x[r][i] = x[2 * r][i] + x[2 * r + 1][i];
#pragma unroll
                    for (int i = 0; i < V; ++i) acc[u][i] = x[0][i];
                } else {
#pragma unroll
                    for (int i = 0; i < V; ++i) {
                        float s = x[0][i];
#pragma unroll
                        for (int q = 1; q < GT; ++q) s = s + x[q][i];
                        acc[u][i] = s;
                    }
                }
            } else {
                Vec<PT>::load((const PT *)src[0] + e, acc[u]);
                for (int q = 1; q < G; q += 4) {
                    float x[4][V];
                    const int m = min(4, G - q);
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        if (t < m) Vec<PT>::load((const PT *)src[q + t] + e, x[t]);
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        if (t < m)
#pragma unroll
                            for (int i = 0; i < V; ++i) acc[u][i] = acc[u][i] + x[t][i];
                }
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const IT v = base + (IT)u * blockDim.x;
            if (v >= total) continue;
            write_out<OT, V, IT>(k, g, v * V, acc[u], gelu);
        }
    }
}

// Scalar fallback for shapes whose owner blocks are not whole vectors.
template <typename PT, typename OT, bool TREE, typename IT>
__global__ void __launch_bounds__(256) reduce_scalar_kernel(const __grid_constant__ ReduceK k, bool gelu) {
    pdl_enter();
    const int g = blockIdx.y;
    const IT total = (IT)k.n;
    for (IT e = (IT)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (IT)gridDim.x * blockDim.x) {
        if (!in_bounds(k.status, (int64_t)e, 1, k.src_n)) continue;
        float s;
        if (!TREE) {
            s = Vec<PT>::load1((const PT *)k.src[g * k.G] + e);
            for (int q = 1; q < k.G; ++q) s = s + Vec<PT>::load1((const PT *)k.src[g * k.G + q] + e);
        } else {
            float lv[32];  // the launcher admits the tree for G <= 32 only
            int W = 1;
            while (W < k.G) W <<= 1;
            if (W > 32) W = 32;
            for (int q = 0; q < W; ++q)
                lv[q] = q < k.G ? Vec<PT>::load1((const PT *)k.src[g * k.G + q] + e) : -0.0f;
            for (int w = W; w > 1; w >>= 1)
                for (int q = 0; q < w / 2; ++q) lv[q] = lv[2 * q] + lv[2 * q + 1];
            s = lv[0];
        }
        write_out<OT, 1, IT>(k, g, e, &s, gelu);
    }
}

// Pairwise tree with warp shuffles: a W-lane subgroup (W = next power of two
// >= G) reduces one vector position; lane q loads rank q (q < G) or -0.0.
// After log2(W) xor-shuffle levels every lane holds the same total (fp32
// addition is commutative bit for bit), so lane q writes destination q.
template <typename PT, typename OT, int W, int UNROLL, typename IT>
__global__ void __launch_bounds__(256) reduce_tree_kernel(const __grid_constant__ ReduceK k, bool gelu) {
    pdl_enter();
    constexpr int V = Vec<PT>::N;
    constexpr int PER_WARP = 32 / W;  // vector positions per warp per step
    const int lane = threadIdx.x & 31;
    const int q = lane % W;
    const int sub = lane / W;
    const int g = blockIdx.y;
    const IT warps = (IT)gridDim.x * (blockDim.x / 32);
    const IT warp = (IT)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const IT total = (IT)k.nvec;
    const PT *src = q < k.G ? (const PT *)k.src[g * k.G + q] : nullptr;
    for (IT base = warp * PER_WARP * UNROLL; base < total; base += warps * PER_WARP * UNROLL) {
        float x[UNROLL][V];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const IT v = base + (IT)u * PER_WARP + sub;
            if (v < total && src && in_bounds(k.status, (int64_t)v * V, V, k.src_n)) {
                Vec<PT>::load(src + v * V, x[u]);
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i) x[u][i] = -0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
#pragma unroll
            for (int off = 1; off < W; off <<= 1)
#pragma unroll
                for (int i = 0; i < V; ++i) x[u][i] = x[u][i] + __shfl_xor_sync(0xffffffffu, x[u][i], off);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const IT v = base + (IT)u * PER_WARP + sub;
            if (v >= total || q >= k.G) continue;
            float s[V];
#pragma unroll
            for (int i = 0; i < V; ++i) s[i] = gelu ? gelu_tanh(x[u][i]) : x[u][i];
            int b;
            IT off;
            route<IT>(k, v * V, &b, &off);
            if (b >= 0 && b != q) continue;  // RS: only the owner's lane writes
            if (!in_bounds(k.status, (int64_t)off, V, k.dst_n)) continue;
            store_n<OT, V>((OT *)k.dst[g * k.G + q] + off, s);
        }
    }
}

int sm_count() {
    static shmm::PerDevice<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= shmm::kMaxDevices) return 148;
    int n = cache.get(dev);
    if (n) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache.set(dev, n);
    return n;
}

// Grid for `work` items per group, `per_block` items per CTA and `groups`
// groups along y: about 8 resident CTAs per SM in total.
dim3 grid_for(int64_t work, int per_block, int groups) {
    const int64_t want = (work + per_block - 1) / per_block;
    int64_t cap = (int64_t)sm_count() * 8 / (groups > 0 ? groups : 1);
    if (cap < 1) cap = 1;
    return dim3((unsigned)(want < 1 ? 1 : (want > cap ? cap : want)), (unsigned)groups, 1);
}

// CTAs of 256 threads that one SM holds at once for `kernel` (cached).
template <typename... P>
int resident_per_sm(void (*kernel)(P...)) {
    static std::mutex mu;
    static std::map<const void *, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    const void *key = reinterpret_cast<const void *>(kernel);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 256, 0) != cudaSuccess || n < 1) n = 1;
    cache[key] = n;
    return n;
}
template <typename... P>
dim3 grid_resident(void (*kernel)(P...), int64_t work, int per_block, int groups) {
    const int64_t want = (work + per_block - 1) / per_block;
    int64_t cap = (int64_t)sm_count() * resident_per_sm(kernel) / (groups > 0 ? groups : 1);
    if (cap < 1) cap = 1;
    return dim3((unsigned)(want < 1 ? 1 : (want > cap ? cap : want)), (unsigned)groups, 1);
}

template <typename PT, typename OT, typename IT>
cudaError_t reduce_dispatch(const ReduceK &k, bool vec_ok, bool tree, bool gelu, cudaStream_t s) {
    if (!vec_ok) {
        const dim3 grid = grid_for(k.n, 256, k.ngroups);
        if (tree) (void)launch_k(reduce_scalar_kernel<PT, OT, true, IT>, grid, 0, s, k, gelu);
        else (void)launch_k(reduce_scalar_kernel<PT, OT, false, IT>, grid, 0, s, k, gelu);
        return cudaGetLastError();
    }
    if (tree && (k.G == 2 || k.G == 4 || k.G == 8 || k.G == 16)) {
        // power-of-two groups fit in registers: pairwise tree per thread
        switch (k.G) {
            case 2: {  // as the sequential two-rank case below
                constexpr int U2 = sizeof(PT) == 2 ? 2 : 4;
                auto kern = reduce_seq_kernel<PT, OT, 2, U2, IT, true>;
                const bool resident = sizeof(PT) == 2 || k.mode != 2;
                const dim3 grid = resident ? grid_resident(kern, k.nvec, 256 * U2, k.ngroups)
                                           : grid_for(k.nvec, 256 * U2, k.ngroups);
                (void)launch_k(kern, grid, 0, s, k, gelu);
                break;
            }
            case 4: (void)launch_k(reduce_seq_kernel<PT, OT, 4, 2, IT, true>, grid_for(k.nvec, 256 * 2, k.ngroups), 0, s, k, gelu); break;
            case 8:  // as the sequential eight-rank case below
                if (sizeof(PT) == 4 && k.mode == 2)
                    (void)launch_k(reduce_seq_kernel<PT, OT, 8, 1, IT, true>, grid_for(k.nvec, 256, k.ngroups), 0, s, k, gelu);
                else
                    (void)launch_k(reduce_seq_kernel<PT, OT, 8, 2, IT, true>, grid_for(k.nvec, 512, k.ngroups), 0, s, k, gelu);
                break;
            default: (void)launch_k(reduce_seq_kernel<PT, OT, 16, 1, IT, true>, grid_for(k.nvec, 256, k.ngroups), 0, s, k, gelu); break;
        }
        return cudaGetLastError();
    }
    if (tree) {
        // other group sizes: one rank per lane, shuffles pad to a power of two
        int W = 1;
        while (W < k.G) W <<= 1;
        constexpr int U = 4;  // vector positions per lane in flight
        const dim3 grid = grid_for(k.nvec, 8 * (32 / W) * U, k.ngroups);  // 8 warps per CTA
        switch (W) {
            case 1: (void)launch_k(reduce_tree_kernel<PT, OT, 1, U, IT>, grid, 0, s, k, gelu); break;
            case 2: (void)launch_k(reduce_tree_kernel<PT, OT, 2, U, IT>, grid, 0, s, k, gelu); break;
            case 4: (void)launch_k(reduce_tree_kernel<PT, OT, 4, U, IT>, grid, 0, s, k, gelu); break;
            case 8: (void)launch_k(reduce_tree_kernel<PT, OT, 8, U, IT>, grid, 0, s, k, gelu); break;
            case 16: (void)launch_k(reduce_tree_kernel<PT, OT, 16, U, IT>, grid, 0, s, k, gelu); break;
            default: (void)launch_k(reduce_tree_kernel<PT, OT, 32, U, IT>, grid, 0, s, k, gelu); break;
        }
        return cudaGetLastError();
    }
    switch (k.G) {
        case 1: (void)launch_k(reduce_seq_kernel<PT, OT, 1, 4, IT>, grid_for(k.nvec, 256 * 4, k.ngroups), 0, s, k, gelu); break;
        case 2: {
            // Two ranks (measured at 64 and 256 MiB per rank): bf16 partials
            // with 2 vectors per thread and a grid of resident CTAs only,
            // 0.75-0.93 -> 0.95 of the copy rate; fp32 keeps 4 vectors, and
            // the resident grid lifts its reduce-scatter 0.89-0.93 -> 0.95-0.99
            // but slows its all-reduce 0.98 -> 0.94, which keeps 8 CTAs/SM.
            constexpr int U2 = sizeof(PT) == 2 ? 2 : 4;
            auto kern = reduce_seq_kernel<PT, OT, 2, U2, IT>;
            const bool resident = sizeof(PT) == 2 || k.mode != 2;
            const dim3 grid = resident ? grid_resident(kern, k.nvec, 256 * U2, k.ngroups)
                                       : grid_for(k.nvec, 256 * U2, k.ngroups);
            (void)launch_k(kern, grid, 0, s, k, gelu);
            break;
        }
        case 4: (void)launch_k(reduce_seq_kernel<PT, OT, 4, 2, IT>, grid_for(k.nvec, 256 * 2, k.ngroups), 0, s, k, gelu); break;
        case 8:
            // Eight ranks (256 MiB per rank): two vectors per thread, 16 loads
            // in flight, took the reduce-scatter from 0.965 to 0.973-0.976 of
            // the copy rate (fp32) and 0.965 -> 0.987 (bf16), the bf16
            // all-reduce 0.948 -> 0.978; the fp32 all-reduce lost (0.972 ->
            // 0.945) and keeps one.
            if (sizeof(PT) == 4 && k.mode == 2)
                (void)launch_k(reduce_seq_kernel<PT, OT, 8, 1, IT>, grid_for(k.nvec, 256, k.ngroups), 0, s, k, gelu);
            else
                (void)launch_k(reduce_seq_kernel<PT, OT, 8, 2, IT>, grid_for(k.nvec, 512, k.ngroups), 0, s, k, gelu);
            break;
        case 16: (void)launch_k(reduce_seq_kernel<PT, OT, 16, 1, IT>, grid_for(k.nvec, 256, k.ngroups), 0, s, k, gelu); break;
        default: (void)launch_k(reduce_seq_kernel<PT, OT, 0, 1, IT>, grid_for(k.nvec, 256, k.ngroups), 0, s, k, gelu); break;
    }
    return cudaGetLastError();
}

template <typename PT, typename OT>
cudaError_t reduce_dispatch_idx(const ReduceK &k, bool vec_ok, bool tree, bool gelu, cudaStream_t s) {
    // every element index of one rank's partial fits in 32 bits?
    if (k.n < ((int64_t)1 << 32) - 64) return reduce_dispatch<PT, OT, uint32_t>(k, vec_ok, tree, gelu, s);
    return reduce_dispatch<PT, OT, uint64_t>(k, vec_ok, tree, gelu, s);
}

// All-gather: one read of each source vector, G writes; group g = blockIdx.y.
// 16-byte vectors: four loads per thread issued before their stores (one
// load in flight per thread left the gather at 0.88 of the copy rate).
template <bool VEC16, typename IT>
__global__ void __launch_bounds__(256) gather_kernel(const __grid_constant__ GatherK k, int elem) {
    pdl_enter();
    const int g = blockIdx.y;
    const IT total = (IT)k.nvec;
    const IT bvecs = (IT)k.bvecs, brows = (IT)k.brows, per_block = brows * bvecs;
    const IT full_vecs = (IT)k.full_vecs;
    if constexpr (VEC16) {
        // four independent loads per thread in flight before the stores
        constexpr int U = 4;
        for (IT base = (IT)blockIdx.x * blockDim.x * U + threadIdx.x; base < total;
             base += (IT)gridDim.x * blockDim.x * U) {
            uint4 x[U];
            IT dst_off[U];
            bool ok[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const IT v = base + (IT)u * blockDim.x;
                if (v >= total) continue;
                const int p = (int)(v / per_block);
                const IT w = v - (IT)p * per_block;
                const IT r = w / bvecs, c = w - r * bvecs;
                const int p0 = p / k.blocks1, p1 = p - p0 * k.blocks1;
                dst_off[u] = ((IT)p0 * brows + r) * full_vecs + (IT)p1 * bvecs + c;
                ok[u] = in_bounds(k.status, (int64_t)w, 1, k.src_n) &&
                        in_bounds(k.status, (int64_t)dst_off[u], 1, k.dst_n);
                if (ok[u]) x[u] = __ldcs(reinterpret_cast<const uint4 *>(k.src[g * k.G + p]) + w);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const IT v = base + (IT)u * blockDim.x;
                if (v >= total || !ok[u]) continue;
                for (int m = 0; m < k.G; ++m) __stcs(reinterpret_cast<uint4 *>(k.dst[g * k.G + m]) + dst_off[u], x[u]);
            }
        }
    } else {
        for (IT v = (IT)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += (IT)gridDim.x * blockDim.x) {
            const int p = (int)(v / per_block);
            const IT w = v - (IT)p * per_block;
            const IT r = w / bvecs, c = w - r * bvecs;
            const int p0 = p / k.blocks1, p1 = p - p0 * k.blocks1;
            const IT src_off = w;
            const IT dst_off = ((IT)p0 * brows + r) * full_vecs + (IT)p1 * bvecs + c;
            if (!in_bounds(k.status, (int64_t)src_off, 1, k.src_n) ||
                !in_bounds(k.status, (int64_t)dst_off, 1, k.dst_n))
                continue;
            if (elem == 4) {  // element-wise: "vectors" are single elements
                const uint32_t x = reinterpret_cast<const uint32_t *>(k.src[g * k.G + p])[src_off];
                for (int m = 0; m < k.G; ++m) reinterpret_cast<uint32_t *>(k.dst[g * k.G + m])[dst_off] = x;
            } else {
                const uint16_t x = reinterpret_cast<const uint16_t *>(k.src[g * k.G + p])[src_off];
                for (int m = 0; m < k.G; ++m) reinterpret_cast<uint16_t *>(k.dst[g * k.G + m])[dst_off] = x;
            }
        }
    }
}

// ---- layer normalisation fused with the all-gather of row blocks ---------

struct LnK {
    const void *src[kMaxPtrs];  // [g*G + p]: block p of group g
    void *dst[kMaxPtrs];        // [g*G + m]: every member's gathered buffer
    const float *gamma, *beta;
    float eps;
    int G;
    int64_t brows, cols;
    int *status;                // device status word (bounds-checked build)
    int64_t src_n, dst_n, gb_n;  // elements per block / gathered buffer / gamma and beta
};

// Deterministic block-wide sum (fixed shuffle tree, then warps in order).
__device__ __forceinline__ float block_sum(float v, float *scratch) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x / 32, nw = blockDim.x / 32;
    __syncthreads();  // scratch is reused between calls
    if ((threadIdx.x & 31) == 0) scratch[w] = v;
    __syncthreads();
    float t = 0.0f;
    for (int i = 0; i < nw; ++i) t += scratch[i];
    return t;
}

// One CTA per row (grid-stride over the group's G*brows rows; group =
// blockIdx.y): mean, then the biased variance of the deviations, then
// y = (x - mean) / sqrt(var + eps) * gamma + beta in fp32, written to every
// member.  This path re-reads the row element by element (any cols); rows of
// whole 16-byte vectors, cols <= 8192, take the register path below.
template <typename T>
__global__ void __launch_bounds__(256) ln_gather_scalar_kernel(const __grid_constant__ LnK k) {
    pdl_enter();
    __shared__ float scratch[32];
    const int g = blockIdx.y;
    const int64_t rows = (int64_t)k.G * k.brows;
    const float inv_n = 1.0f / (float)k.cols;
    for (int64_t t = blockIdx.x; t < rows; t += gridDim.x) {
        const int p = (int)(t / k.brows);
        const int64_t rr = t - (int64_t)p * k.brows;
        const int64_t drow = ((int64_t)p * k.brows + rr) * k.cols;
        if (!in_bounds(k.status, rr * k.cols, k.cols, k.src_n) || !in_bounds(k.status, drow, k.cols, k.dst_n) ||
            !in_bounds(k.status, 0, k.cols, k.gb_n))
            continue;  // the same for every thread of the CTA: block_sum stays collective
        const T *x = (const T *)k.src[g * k.G + p] + rr * k.cols;
        float sum = 0.0f, mean, rstd;
        for (int64_t c = threadIdx.x; c < k.cols; c += blockDim.x) sum += Vec<T>::load1(x + c);
        mean = block_sum(sum, scratch) * inv_n;
        float sq = 0.0f;
        for (int64_t c = threadIdx.x; c < k.cols; c += blockDim.x) {
            const float d = Vec<T>::load1(x + c) - mean;
            sq += d * d;
        }
        rstd = 1.0f / sqrtf(block_sum(sq, scratch) * inv_n + k.eps);
        for (int64_t c = threadIdx.x; c < k.cols; c += blockDim.x) {
            const float y = (Vec<T>::load1(x + c) - mean) * rstd * k.gamma[c] + k.beta[c];
            for (int m = 0; m < k.G; ++m) Vec<T>::store1((T *)k.dst[g * k.G + m] + drow + c, y);
        }
    }
}

// Register path, same arithmetic: each thread holds NVT 16-byte vectors of
// the row.  They are the same columns in every row, so the thread reads its
// gamma and beta once, not per row (reading them per element per row left
// LayerNorm + all-gather at 0.76 of the copy rate; now 0.865, within 4 % of
// the plain all-gather).
template <typename T, int NVT>
__global__ void __launch_bounds__(256) ln_gather_reg_kernel(const __grid_constant__ LnK k) {
    pdl_enter();
    constexpr int V = 16 / sizeof(T);
    __shared__ float scratch[32];
    const int g = blockIdx.y;
    const int64_t rows = (int64_t)k.G * k.brows;
    const float inv_n = 1.0f / (float)k.cols;
    const int nvec = (int)(k.cols / V);
    float ga[NVT][V], be[NVT][V];
#pragma unroll
    for (int j = 0; j < NVT; ++j) {
        const int vi = threadIdx.x + j * blockDim.x;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const bool in = vi < nvec && in_bounds(k.status, (int64_t)vi * V + i, 1, k.gb_n);
            ga[j][i] = in ? k.gamma[(int64_t)vi * V + i] : 0.0f;
            be[j][i] = in ? k.beta[(int64_t)vi * V + i] : 0.0f;
        }
    }
    auto load_row = [&](int64_t t, float (*v)[V]) {
        const int p = (int)(t / k.brows);
        const int64_t rr = t - (int64_t)p * k.brows;
        const T *x = (const T *)k.src[g * k.G + p] + rr * k.cols;
#pragma unroll
        for (int j = 0; j < NVT; ++j) {
            const int vi = threadIdx.x + j * blockDim.x;
            if (vi < nvec && in_bounds(k.status, rr * k.cols + (int64_t)vi * V, V, k.src_n))
                Vec<T>::load(x + (int64_t)vi * V, v[j]);
            else
#pragma unroll
                for (int i = 0; i < V; ++i) v[j][i] = 0.0f;
        }
    };
    float v[NVT][V];
    if ((int64_t)blockIdx.x < rows) load_row(blockIdx.x, v);
    for (int64_t t = blockIdx.x; t < rows; t += gridDim.x) {
        const int p = (int)(t / k.brows);
        const int64_t rr = t - (int64_t)p * k.brows;
        float sum = 0.0f;
#pragma unroll
        for (int j = 0; j < NVT; ++j)
#pragma unroll
            for (int i = 0; i < V; ++i) sum += v[j][i];
        const float mean = block_sum(sum, scratch) * inv_n;
        float sq = 0.0f;
#pragma unroll
        for (int j = 0; j < NVT; ++j) {
            const int vi = threadIdx.x + j * blockDim.x;
            if (vi < nvec)
#pragma unroll
                for (int i = 0; i < V; ++i) sq += (v[j][i] - mean) * (v[j][i] - mean);
        }
        const float rstd = 1.0f / sqrtf(block_sum(sq, scratch) * inv_n + k.eps);
#pragma unroll
        for (int j = 0; j < NVT; ++j) {
            const int vi = threadIdx.x + j * blockDim.x;
            if (vi >= nvec) continue;
            float y[V];
#pragma unroll
            for (int i = 0; i < V; ++i) y[i] = (v[j][i] - mean) * rstd * ga[j][i] + be[j][i];
            const int64_t d0 = ((int64_t)p * k.brows + rr) * k.cols + (int64_t)vi * V;
            if (!in_bounds(k.status, d0, V, k.dst_n)) continue;
            for (int m = 0; m < k.G; ++m) store_n<T, V>((T *)k.dst[g * k.G + m] + d0, y);
        }
        if (t + gridDim.x < rows) load_row(t + gridDim.x, v);
    }
}

// Bulk-copy path, same arithmetic per row as the register path (the same
// vectors per thread, the same block sums): thread 0 keeps `stages` (2 to
// kLnMaxStages, as many as kLnSmemBudget holds) rows of the
// CTA's walk in flight through the bulk-copy engine (cp.async.bulk into
// shared memory, completion counted on one mbarrier per stage), so the row a
// CTA normalises has landed while the next ones stream in.  The register
// path has one row in flight per CTA, which leaves a two- or four-rank
// gather latency-bound (few stores per row to hide the load behind).
// Thread 0 alone waits on a stage, bounded, and the CTA follows it through
// __syncthreads, so every thread leaves the loop at the same row; before
// exit thread 0 waits (bounded) for every copy it issued.
constexpr int kLnMaxStages = 4;
template <typename T, int NVT>
__device__ __forceinline__ void ln_gather_bulk(const LnK &k, int stages) {
    constexpr int V = 16 / sizeof(T);
    extern __shared__ __align__(128) uint8_t ln_rows[];  // `stages` rows of cols elements
    __shared__ __align__(8) uint64_t bars[kLnMaxStages];
    __shared__ float scratch[32];
    __shared__ int abort_flag, go;
    const int g = blockIdx.y;
    const int64_t rows = (int64_t)k.G * k.brows;
    const uint32_t row_bytes = (uint32_t)(k.cols * (int64_t)sizeof(T));
    const float inv_n = 1.0f / (float)k.cols;
    const int nvec = (int)(k.cols / V);
    float ga[NVT][V], be[NVT][V];
#pragma unroll
    for (int j = 0; j < NVT; ++j) {
        const int vi = threadIdx.x + j * blockDim.x;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const bool in = vi < nvec && in_bounds(k.status, (int64_t)vi * V + i, 1, k.gb_n);
            ga[j][i] = in ? k.gamma[(int64_t)vi * V + i] : 0.0f;
            be[j][i] = in ? k.beta[(int64_t)vi * V + i] : 0.0f;
        }
    }
    auto bar = [&](int st) { return shmm_dev::smem_u32(&bars[st]); };
    // Thread 0: start the copy of row t into stage st (a plain arrival when
    // the bounds-checked build finds the row outside its block).
    auto issue = [&](int st, int64_t t) {
        const int p = (int)(t / k.brows);
        const int64_t rr = t - (int64_t)p * k.brows;
        if (!in_bounds(k.status, rr * k.cols, k.cols, k.src_n)) {
            shmm_dev::mbar_arrive(bar(st));
            return;
        }
        const char *src = (const char *)k.src[g * k.G + p] + rr * (int64_t)row_bytes;
        shmm_dev::mbar_expect_tx(bar(st), row_bytes);
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                shmm_dev::smem_u32(ln_rows + (size_t)st * row_bytes)),
            "l"(src), "r"(row_bytes), "r"(bar(st))
            : "memory");
    };
    if (threadIdx.x == 0) {
        for (int st = 0; st < stages; ++st) shmm_dev::mbar_init(bar(st), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int st = 0; st < stages; ++st) {
            const int64_t t = (int64_t)blockIdx.x + (int64_t)st * gridDim.x;
            if (t < rows) issue(st, t);
        }
    }
    __syncthreads();
    int it = 0;  // rows this CTA has taken
    for (int64_t t = blockIdx.x; t < rows; t += gridDim.x, ++it) {
        const int st = it % stages;
        if (threadIdx.x == 0) go = shmm_dev::mbar_wait(bar(st), (uint32_t)(it / stages) & 1, &abort_flag, k.status);
        __syncthreads();
        if (!go) break;
        const T *x = reinterpret_cast<const T *>(ln_rows + (size_t)st * row_bytes);
        float v[NVT][V];
#pragma unroll
        for (int j = 0; j < NVT; ++j) {
            const int vi = threadIdx.x + j * blockDim.x;
            if (vi < nvec) {
                const uint4 w = *reinterpret_cast<const uint4 *>(x + (int64_t)vi * V);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                if constexpr (sizeof(T) == 4) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[j][i] = __uint_as_float(ws[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        v[j][2 * i] = __uint_as_float(ws[i] << 16);
                        v[j][2 * i + 1] = __uint_as_float(ws[i] & 0xffff0000u);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i) v[j][i] = 0.0f;
            }
        }
        const int p = (int)(t / k.brows);
        const int64_t rr = t - (int64_t)p * k.brows;
        float sum = 0.0f;
#pragma unroll
        for (int j = 0; j < NVT; ++j)
#pragma unroll
            for (int i = 0; i < V; ++i) sum += v[j][i];
        const float mean = block_sum(sum, scratch) * inv_n;
        float sq = 0.0f;
#pragma unroll
        for (int j = 0; j < NVT; ++j) {
            const int vi = threadIdx.x + j * blockDim.x;
            if (vi < nvec)
#pragma unroll
                for (int i = 0; i < V; ++i) sq += (v[j][i] - mean) * (v[j][i] - mean);
        }
        // block_sum's barriers also order every thread's reads of this stage
        // before thread 0 refills it below
        const float rstd = 1.0f / sqrtf(block_sum(sq, scratch) * inv_n + k.eps);
        if (threadIdx.x == 0) {
            const int64_t next = t + (int64_t)stages * gridDim.x;
            if (next < rows) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(st, next);
            }
        }
#pragma unroll
        for (int j = 0; j < NVT; ++j) {
            const int vi = threadIdx.x + j * blockDim.x;
            if (vi >= nvec) continue;
            float y[V];
#pragma unroll
            for (int i = 0; i < V; ++i) y[i] = (v[j][i] - mean) * rstd * ga[j][i] + be[j][i];
            const int64_t d0 = ((int64_t)p * k.brows + rr) * k.cols + (int64_t)vi * V;
            if (!in_bounds(k.status, d0, V, k.dst_n)) continue;
            for (int m = 0; m < k.G; ++m) store_n<T, V>((T *)k.dst[g * k.G + m] + d0, y);
        }
    }
    // Never leave a copy into shared memory in flight at exit.  Row u of this
    // CTA's walk was issued for u < it + stages and consumed for u < it;
    // after an abort, wait (bounded) for the issued rows not consumed.
    if (threadIdx.x == 0) {
        const int64_t n = rows > (int64_t)blockIdx.x ? (rows - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        for (int64_t u = it; u < n && u < (int64_t)it + stages; ++u)
            shmm_dev::mbar_wait(bar((int)(u % stages)), (uint32_t)(u / stages) & 1, &abort_flag, k.status, false);
    }
}

// The bulk path's kernels: the compiler's own register budget (three CTAs
// per SM for rows of up to 4096 bf16 columns), and a 64-register cap for
// four CTAs per SM.  With two members a row has few stores to hide its two
// block reductions behind, so more rows in flight pay: four CTAs took bf16
// rows of 4096 from 0.76 to 0.81 of the copy rate at 256 MiB; with 8
// members, and for fp32, the cap cost more than the extra rows gave.
template <typename T, int NVT>
__global__ void __launch_bounds__(256) ln_gather_bulk_kernel(const __grid_constant__ LnK k, int stages) {
    pdl_enter();
    ln_gather_bulk<T, NVT>(k, stages);
}
template <typename T, int NVT>
__global__ void __launch_bounds__(256, 4) ln_gather_bulk4_kernel(const __grid_constant__ LnK k, int stages) {
    pdl_enter();
    ln_gather_bulk<T, NVT>(k, stages);
}

// Dynamic shared memory the bulk-copy LayerNorm may take per CTA (above the
// 48 KB default, so each instantiation opts in once per device).
constexpr int kLnSmemBudget = 64 * 1024;
template <typename T, int NVT, bool FOUR = false>
cudaError_t launch_ln_bulk(const LnK &k, dim3 grid, int stages, size_t smem, cudaStream_t s) {
    void (*kern)(LnK, int);
    if constexpr (FOUR)
        kern = ln_gather_bulk4_kernel<T, NVT>;
    else
        kern = ln_gather_bulk_kernel<T, NVT>;
    static shmm::PerDevice<int> attr_set;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= shmm::kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set.get(dev)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kLnSmemBudget);
        if (e != cudaSuccess) return e;
        attr_set.set(dev, 1);
    }
    (void)launch_k(kern, grid, smem, s, k, stages);
    return cudaGetLastError();
}

// ---- reshard: rectangles between rank buffers ------------------------------

constexpr int kMaxRects = 256;  // one launch for a 16-rank all-to-all (16 x 16 rectangles)

struct CopyK {
    shmm::CopyRect r[kMaxRects];
    int *status;  // device status word (bounds-checked build)
};

// Rectangle blockIdx.y; the CTAs along x stride over its rows x units, a unit
// being a 16-byte vector (VEC) or one element of `elem` bytes.  Vectors: four
// independent loads per thread in flight before their stores (one in flight
// left a 16 MiB all-to-all at 0.47 of the copy rate, latency-bound).
template <bool VEC, typename IT>
__global__ void __launch_bounds__(256) copy_rects_kernel(const __grid_constant__ CopyK k, int elem) {
    pdl_enter();
    const shmm::CopyRect &R = k.r[blockIdx.y];
    const IT per_row = VEC ? (IT)(R.w * elem / 16) : (IT)R.w;
    const IT total = per_row * (IT)R.h;
    const IT sld = VEC ? (IT)(R.src_ld * elem / 16) : (IT)R.src_ld;
    const IT dld = VEC ? (IT)(R.dst_ld * elem / 16) : (IT)R.dst_ld;
    const int64_t sroom = VEC ? R.src_room * elem / 16 : R.src_room;
    const int64_t droom = VEC ? R.dst_room * elem / 16 : R.dst_room;
    if constexpr (VEC) {
        constexpr int U = 4;
        for (IT base = (IT)blockIdx.x * blockDim.x * U + threadIdx.x; base < total;
             base += (IT)gridDim.x * blockDim.x * U) {
            uint4 x[U];
            IT doff[U];
            bool ok[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const IT v = base + (IT)u * blockDim.x;
                ok[u] = v < total;
                if (!ok[u]) continue;
                const IT row = v / per_row, c = v - row * per_row;
                doff[u] = row * dld + c;
                ok[u] = in_bounds(k.status, (int64_t)(row * sld + c), 1, sroom) &&
                        in_bounds(k.status, (int64_t)doff[u], 1, droom);
                if (ok[u]) x[u] = __ldcs(reinterpret_cast<const uint4 *>(R.src) + row * sld + c);
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (ok[u]) __stcs(reinterpret_cast<uint4 *>(R.dst) + doff[u], x[u]);
        }
    } else {
        for (IT v = (IT)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += (IT)gridDim.x * blockDim.x) {
            const IT row = v / per_row, c = v - row * per_row;
            if (!in_bounds(k.status, (int64_t)(row * sld + c), 1, sroom) ||
                !in_bounds(k.status, (int64_t)(row * dld + c), 1, droom))
                continue;
            if (elem == 4) {
                reinterpret_cast<uint32_t *>(R.dst)[row * dld + c] =
                    reinterpret_cast<const uint32_t *>(R.src)[row * sld + c];
            } else {
                reinterpret_cast<uint16_t *>(R.dst)[row * dld + c] =
                    reinterpret_cast<const uint16_t *>(R.src)[row * sld + c];
            }
        }
    }
}

}  // namespace

namespace shmm {

int launch_layernorm_gather(const LayerNormArgs &a, int *status, void *stream) {
    if (a.ngroups * a.G > kMaxPtrs) return (int)cudaErrorInvalidValue;
    if (a.brows == 0 || a.cols == 0 || a.ngroups == 0) return 0;
    LnK k;
    for (int i = 0; i < a.ngroups * a.G; ++i) {
        k.src[i] = a.src[i];
        k.dst[i] = a.dst[i];
    }
    k.gamma = a.gamma;
    k.beta = a.beta;
    k.eps = a.eps;
    k.G = a.G;
    k.brows = a.brows;
    k.cols = a.cols;
    k.status = status;
    k.src_n = a.brows * a.cols;
    k.dst_n = (int64_t)a.G * a.brows * a.cols;
    k.gb_n = a.cols;
    const int V = a.dt == SHMM_F32 ? 4 : 8;
    const bool reg = a.cols % V == 0 && a.cols <= (int64_t)V * 4 * 256;
    const int64_t rows = (int64_t)a.G * a.brows;
    int64_t want = rows, cap = (int64_t)sm_count() * 8 / a.ngroups;
    if (cap < 1) cap = 1;
    const dim3 grid((unsigned)(want < cap ? want : cap), (unsigned)a.ngroups, 1);
    cudaStream_t s = (cudaStream_t)stream;
    count_launch();
    const int nvt = (int)((a.cols / V + 255) / 256);  // vectors per thread
    // Rows staged through shared memory by the bulk-copy engine, up to 4 in
    // flight per CTA within kLnSmemBudget, when at least two fit.
    const int64_t row_bytes = a.cols * (a.dt == SHMM_F32 ? 4 : 2);
    int64_t stages = kLnSmemBudget / (row_bytes > 0 ? row_bytes : 1);
    if (stages > kLnMaxStages) stages = kLnMaxStages;
    const char *env = getenv("SHMM_LN_BULK");
    const bool bulk = env ? env[0] != '0' : true;
    if (reg && bulk && stages >= 2) {
        const size_t sm = (size_t)stages * (size_t)row_bytes;
        const int st = (int)stages;
        cudaError_t e;
        if (a.dt == SHMM_F32)
            e = nvt <= 1 ? launch_ln_bulk<float, 1>(k, grid, st, sm, s)
                         : nvt == 2 ? launch_ln_bulk<float, 2>(k, grid, st, sm, s) : launch_ln_bulk<float, 4>(k, grid, st, sm, s);
        else if (a.G <= 2 && nvt <= 2)  // four CTAs per SM (see the kernels)
            e = nvt <= 1 ? launch_ln_bulk<__nv_bfloat16, 1, true>(k, grid, st, sm, s)
                         : launch_ln_bulk<__nv_bfloat16, 2, true>(k, grid, st, sm, s);
        else
            e = nvt <= 1 ? launch_ln_bulk<__nv_bfloat16, 1>(k, grid, st, sm, s)
                         : nvt == 2 ? launch_ln_bulk<__nv_bfloat16, 2>(k, grid, st, sm, s)
                                    : launch_ln_bulk<__nv_bfloat16, 4>(k, grid, st, sm, s);
        return (int)e;
    }
    if (reg && a.dt == SHMM_F32) {
        if (nvt <= 1) (void)launch_k(ln_gather_reg_kernel<float, 1>, grid, 0, s, k);
        else if (nvt == 2) (void)launch_k(ln_gather_reg_kernel<float, 2>, grid, 0, s, k);
        else (void)launch_k(ln_gather_reg_kernel<float, 4>, grid, 0, s, k);
    } else if (reg) {
        if (nvt <= 1) (void)launch_k(ln_gather_reg_kernel<__nv_bfloat16, 1>, grid, 0, s, k);
        else if (nvt == 2) (void)launch_k(ln_gather_reg_kernel<__nv_bfloat16, 2>, grid, 0, s, k);
        else (void)launch_k(ln_gather_reg_kernel<__nv_bfloat16, 4>, grid, 0, s, k);
    } else if (a.dt == SHMM_F32) {
        (void)launch_k(ln_gather_scalar_kernel<float>, grid, 0, s, k);
    } else {
        (void)launch_k(ln_gather_scalar_kernel<__nv_bfloat16>, grid, 0, s, k);
    }
    return (int)cudaGetLastError();
}

int launch_copy_rects(const CopyRect *rects, int n, int elem, int *status, void *stream) {
    cudaStream_t s = (cudaStream_t)stream;
    for (int i0 = 0; i0 < n; i0 += kMaxRects) {
        const int m = (n - i0) < kMaxRects ? (n - i0) : kMaxRects;
        CopyK k;
        k.status = status;
        bool vec = true, small = true;
        int64_t most = 0;
        for (int i = 0; i < m; ++i) {
            const CopyRect &r = rects[i0 + i];
            k.r[i] = r;
            vec = vec && (r.w * elem) % 16 == 0 && (r.src_ld * elem) % 16 == 0 && (r.dst_ld * elem) % 16 == 0 &&
                  reinterpret_cast<uintptr_t>(r.src) % 16 == 0 && reinterpret_cast<uintptr_t>(r.dst) % 16 == 0;
            const int64_t items = r.h * r.w;
            most = items > most ? items : most;
            small = small && r.h * (r.src_ld > r.dst_ld ? r.src_ld : r.dst_ld) < ((int64_t)1 << 32) - 64;
        }
        if (most == 0) continue;
        const int64_t units = vec ? most * elem / 16 : most;
        int64_t want = (units + 1023) / 1024;
        const int64_t cap = (int64_t)sm_count() * 8 / m > 0 ? (int64_t)sm_count() * 8 / m : 1;
        if (want > cap) want = cap;
        if (want < 1) want = 1;
        const dim3 grid((unsigned)want, (unsigned)m, 1);
        count_launch();
        if (vec) {
            if (small) (void)launch_k(copy_rects_kernel<true, uint32_t>, grid, 0, s, k, elem);
            else (void)launch_k(copy_rects_kernel<true, uint64_t>, grid, 0, s, k, elem);
        } else {
            if (small) (void)launch_k(copy_rects_kernel<false, uint32_t>, grid, 0, s, k, elem);
            else (void)launch_k(copy_rects_kernel<false, uint64_t>, grid, 0, s, k, elem);
        }
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return (int)e;
    }
    return 0;
}


int launch_reduce(const ReduceArgs &a, int *status, void *stream) {
    if (a.ngroups * a.G > kMaxPtrs) return (int)cudaErrorInvalidValue;
    const int64_t n = a.rows * a.cols;
    if (n == 0 || a.ngroups == 0) return 0;
    ReduceK k;
    for (int i = 0; i < a.ngroups * a.G; ++i) {
        k.src[i] = a.src[i];
        k.dst[i] = a.dst[i];
    }
    k.G = a.G;
    k.ngroups = a.ngroups;
    k.mode = a.mode;
    k.rows = a.rows;
    k.cols = a.cols;
    k.n = n;
    k.status = status;
    k.src_n = n;
    k.dst_n = a.mode == 2 ? n : n / a.G;  // a reduce-scatter owner holds 1/G of the partial
    if (a.tree && a.G > 32) return (int)cudaErrorInvalidValue;
    const int V = a.pt == SHMM_F32 ? 4 : 8;
    // A 16-byte vector of partials (V elements) must not straddle an owner
    // boundary or a row of a column-scattered block.
    bool vec_ok = n % V == 0;
    if (a.mode == 0) vec_ok = vec_ok && ((n / a.G) % V == 0);
    if (a.mode == 1) vec_ok = vec_ok && ((a.cols / a.G) % V == 0);
    k.nvec = vec_ok ? n / V : n;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    count_launch();
    if (a.pt == SHMM_F32 && a.ot == SHMM_F32) e = reduce_dispatch_idx<float, float>(k, vec_ok, a.tree, a.gelu, s);
    else if (a.pt == SHMM_F32) e = reduce_dispatch_idx<float, __nv_bfloat16>(k, vec_ok, a.tree, a.gelu, s);
    else if (a.ot == SHMM_BF16) e = reduce_dispatch_idx<__nv_bfloat16, __nv_bfloat16>(k, vec_ok, a.tree, a.gelu, s);
    else e = reduce_dispatch_idx<__nv_bfloat16, float>(k, vec_ok, a.tree, a.gelu, s);
    return (int)e;
}

int launch_gather(const GatherArgs &a, int *status, void *stream) {
    if (a.ngroups * a.G > kMaxPtrs) return (int)cudaErrorInvalidValue;
    if (a.brows == 0 || a.bcols == 0 || a.ngroups == 0) return 0;
    GatherK k;
    for (int i = 0; i < a.ngroups * a.G; ++i) {
        k.src[i] = a.src[i];
        k.dst[i] = a.dst[i];
    }
    k.G = a.G;
    k.ngroups = a.ngroups;
    k.blocks1 = a.blocks1;
    k.brows = a.brows;
    const bool vec = (a.bcols * a.elem) % 16 == 0;
    const int64_t per = vec ? 16 / a.elem : 1;
    k.bvecs = a.bcols / per;
    k.full_vecs = (int64_t)a.blocks1 * k.bvecs;
    k.nvec = (int64_t)a.G * a.brows * k.bvecs;
    k.status = status;
    const int64_t unit = vec ? 16 : a.elem;  // bytes per vector or element
    k.src_n = a.brows * a.bcols * a.elem / unit;
    k.dst_n = (int64_t)a.blocks0 * a.brows * a.blocks1 * a.bcols * a.elem / unit;
    cudaStream_t s = (cudaStream_t)stream;
    const dim3 grid = grid_for(k.nvec, vec ? 256 * 4 : 256, k.ngroups);
    const int elem = (int)a.elem;
    const bool small = k.nvec < ((int64_t)1 << 32) - 64 &&
                       (int64_t)a.blocks0 * a.brows * k.full_vecs < ((int64_t)1 << 32) - 64;
    count_launch();
    if (vec) {
        if (small) (void)launch_k(gather_kernel<true, uint32_t>, grid, 0, s, k, elem);
        else (void)launch_k(gather_kernel<true, uint64_t>, grid, 0, s, k, elem);
    } else {
        if (small) (void)launch_k(gather_kernel<false, uint32_t>, grid, 0, s, k, elem);
        else (void)launch_k(gather_kernel<false, uint64_t>, grid, 0, s, k, elem);
    }
    return (int)cudaGetLastError();
}

}  // namespace shmm
