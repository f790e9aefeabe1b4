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

#include "shmm_internal.h"

namespace {

constexpr int kMaxPtrs = SHMM_MAX_RANKS;

struct ReduceK {
    const void *src[kMaxPtrs];  // group-major: [g*G + q], q ascending rank
    void *dst[kMaxPtrs];        // [g*G + b]: owner of block b (RS) / member b (AR)
    int G, ngroups, mode;       // mode: 0 RS rows, 1 RS cols, 2 AR
    int64_t rows, cols, n;      // per-rank partial shape, n = rows*cols
    int64_t nvec;               // vectors per group
};

struct GatherK {
    const void *src[kMaxPtrs];  // [g*G + p]: block at grid position p
    void *dst[kMaxPtrs];        // [g*G + m]: every member m
    int G, ngroups, blocks1;
    int64_t brows, bvecs;       // block rows, 16-byte vectors per block row
    int64_t full_vecs;          // vectors per row of the gathered box
    int64_t nvec;               // vectors per group = G * brows * bvecs
};

__device__ __forceinline__ float gelu_tanh(float x) {
    // tanh-form GeLU (Hendrycks & Gimpel 2016); sqrt(2/pi) = 0.7978845608...
    const float inner = 0.7978845608028654f * (x + 0.044715f * x * x * x);
    return 0.5f * x * (1.0f + tanhf(inner));
}

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

// Destination element index and owner for element e of the partial.
__device__ __forceinline__ void route(const ReduceK &k, int64_t e, int *b, int64_t *off) {
    if (k.mode == 0) {
        const int64_t per = k.n / k.G;
        *b = (int)(e / per);
        *off = e - (int64_t)(*b) * per;
    } else if (k.mode == 1) {
        const int64_t row = e / k.cols, col = e - row * k.cols, per = k.cols / k.G;
        *b = (int)(col / per);
        *off = row * per + (col - (int64_t)(*b) * per);
    } else {
        *b = -1;
        *off = e;
    }
}

template <typename OT, int NV>
__device__ __forceinline__ void write_out(const ReduceK &k, int g, int64_t e, float *s, bool gelu) {
    if (gelu)
#pragma unroll
        for (int i = 0; i < NV; ++i) s[i] = gelu_tanh(s[i]);
    int b;
    int64_t off;
    route(k, e, &b, &off);
    const int q0 = b >= 0 ? b : 0, q1 = b >= 0 ? b + 1 : k.G;
    for (int q = q0; q < q1; ++q) {
        OT *d = (OT *)k.dst[g * k.G + q] + off;
        if constexpr (NV == 1) Vec<OT>::store1(d, s[0]);
        else store_n<OT, NV>(d, s);
    }
}

// Sequential rank-order sum, 16-byte vectors.  GT > 0: group size known at
// compile time (all G loads issued before the adds); GT == 0: runtime G.
template <typename PT, typename OT, int GT, int UNROLL>
__global__ void __launch_bounds__(256) reduce_seq_kernel(const __grid_constant__ ReduceK k, bool gelu) {
    constexpr int V = Vec<PT>::N;
    const int G = GT > 0 ? GT : k.G;
    const int64_t total = k.nvec * k.ngroups;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * UNROLL;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x * UNROLL + threadIdx.x; base < total;
         base += stride) {
        float acc[UNROLL][V];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t v = base + (int64_t)u * blockDim.x;
            if (v >= total) continue;
            const int g = (int)(v / k.nvec);
            const int64_t e = (v - (int64_t)g * k.nvec) * V;
            if constexpr (GT > 0) {
                float x[GT][V];
#pragma unroll
                for (int q = 0; q < GT; ++q)
                    Vec<PT>::load((const PT *)k.src[g * GT + q] + e, x[q]);
#pragma unroll
                for (int i = 0; i < V; ++i) {
                    float s = x[0][i];
#pragma unroll
                    for (int q = 1; q < GT; ++q) s = s + x[q][i];
                    acc[u][i] = s;
                }
            } else {
                Vec<PT>::load((const PT *)k.src[g * G] + e, acc[u]);
                for (int q = 1; q < G; q += 4) {
                    float x[4][V];
                    const int m = min(4, G - q);
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        if (t < m) Vec<PT>::load((const PT *)k.src[g * G + q + t] + e, x[t]);
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
            const int64_t v = base + (int64_t)u * blockDim.x;
            if (v >= total) continue;
            const int g = (int)(v / k.nvec);
            const int64_t e = (v - (int64_t)g * k.nvec) * V;
            write_out<OT, V>(k, g, e, acc[u], gelu);
        }
    }
}

// Scalar fallback for shapes whose rows/owner blocks are not whole vectors.
template <typename PT, typename OT, bool TREE>
__global__ void __launch_bounds__(256) reduce_scalar_kernel(const __grid_constant__ ReduceK k, bool gelu) {
    const int64_t total = k.n * k.ngroups;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int g = (int)(v / k.n);
        const int64_t e = v - (int64_t)g * k.n;
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
        write_out<OT, 1>(k, g, e, &s, gelu);
    }
}

// Pairwise tree with warp shuffles: a W-lane subgroup (W = next power of two
// >= G) reduces one vector position; lane q loads rank q (q < G) or -0.0.
// After log2(W) xor-shuffle levels every lane holds the same total (fp32
// addition is commutative bit for bit), so lane q writes destination q.
template <typename PT, typename OT, int W, int UNROLL>
__global__ void __launch_bounds__(256) reduce_tree_kernel(const __grid_constant__ ReduceK k, bool gelu) {
    constexpr int V = Vec<PT>::N;
    constexpr int PER_WARP = 32 / W;  // vector positions per warp per step
    const int lane = threadIdx.x & 31;
    const int q = lane % W;
    const int sub = lane / W;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int64_t total = k.nvec * k.ngroups;
    for (int64_t base = warp * PER_WARP * UNROLL; base < total; base += warps * PER_WARP * UNROLL) {
        float x[UNROLL][V];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t v = base + (int64_t)u * PER_WARP + sub;
            if (v < total && q < k.G) {
                const int g = (int)(v / k.nvec);
                const int64_t e = (v - (int64_t)g * k.nvec) * V;
                Vec<PT>::load((const PT *)k.src[g * k.G + q] + e, x[u]);
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
            const int64_t v = base + (int64_t)u * PER_WARP + sub;
            if (v >= total || q >= k.G) continue;
            const int g = (int)(v / k.nvec);
            const int64_t e = (v - (int64_t)g * k.nvec) * V;
            float s[V];
#pragma unroll
            for (int i = 0; i < V; ++i) s[i] = gelu ? gelu_tanh(x[u][i]) : x[u][i];
            int b;
            int64_t off;
            route(k, e, &b, &off);
            if (b >= 0 && b != q) continue;  // RS: only the owner's lane writes
            store_n<OT, V>((OT *)k.dst[g * k.G + q] + off, s);
        }
    }
}

int sm_count() {
    static int cached[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

unsigned grid_for(int64_t work, int per_block) {
    const int64_t want = (work + per_block - 1) / per_block;
    const int64_t cap = (int64_t)sm_count() * 8;
    return (unsigned)(want < 1 ? 1 : (want > cap ? cap : want));
}

template <typename PT, typename OT>
cudaError_t reduce_dispatch(const ReduceK &k, bool vec_ok, bool tree, bool gelu, cudaStream_t s) {
    const int64_t total_vec = k.nvec * k.ngroups;
    if (!vec_ok) {
        const unsigned grid = grid_for(k.n * k.ngroups, 256);
        if (tree) reduce_scalar_kernel<PT, OT, true><<<grid, 256, 0, s>>>(k, gelu);
        else reduce_scalar_kernel<PT, OT, false><<<grid, 256, 0, s>>>(k, gelu);
        return cudaGetLastError();
    }
    if (tree) {
        int W = 1;
        while (W < k.G) W <<= 1;
        const unsigned grid = grid_for(total_vec, 8 * (32 / W) * 2);  // 8 warps, UNROLL 2
        switch (W) {
            case 1: reduce_tree_kernel<PT, OT, 1, 2><<<grid, 256, 0, s>>>(k, gelu); break;
            case 2: reduce_tree_kernel<PT, OT, 2, 2><<<grid, 256, 0, s>>>(k, gelu); break;
            case 4: reduce_tree_kernel<PT, OT, 4, 2><<<grid, 256, 0, s>>>(k, gelu); break;
            case 8: reduce_tree_kernel<PT, OT, 8, 2><<<grid, 256, 0, s>>>(k, gelu); break;
            case 16: reduce_tree_kernel<PT, OT, 16, 2><<<grid, 256, 0, s>>>(k, gelu); break;
            default: reduce_tree_kernel<PT, OT, 32, 2><<<grid, 256, 0, s>>>(k, gelu); break;
        }
        return cudaGetLastError();
    }
    switch (k.G) {
        case 1: reduce_seq_kernel<PT, OT, 1, 4><<<grid_for(total_vec, 256 * 4), 256, 0, s>>>(k, gelu); break;
        case 2: reduce_seq_kernel<PT, OT, 2, 4><<<grid_for(total_vec, 256 * 4), 256, 0, s>>>(k, gelu); break;
        case 4: reduce_seq_kernel<PT, OT, 4, 2><<<grid_for(total_vec, 256 * 2), 256, 0, s>>>(k, gelu); break;
        case 8: reduce_seq_kernel<PT, OT, 8, 1><<<grid_for(total_vec, 256), 256, 0, s>>>(k, gelu); break;
        case 16: reduce_seq_kernel<PT, OT, 16, 1><<<grid_for(total_vec, 256), 256, 0, s>>>(k, gelu); break;
        default: reduce_seq_kernel<PT, OT, 0, 1><<<grid_for(total_vec, 256), 256, 0, s>>>(k, gelu); break;
    }
    return cudaGetLastError();
}

// All-gather: one read of each source vector, G writes.
template <bool VEC16>
__global__ void __launch_bounds__(256) gather_kernel(const __grid_constant__ GatherK k, int64_t elem) {
    const int64_t total = k.nvec * k.ngroups;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int g = (int)(v / k.nvec);
        int64_t w = v - (int64_t)g * k.nvec;
        const int64_t per_block = k.brows * k.bvecs;
        const int p = (int)(w / per_block);
        w -= (int64_t)p * per_block;
        const int64_t r = w / k.bvecs, c = w - r * k.bvecs;
        const int p0 = p / k.blocks1, p1 = p - p0 * k.blocks1;
        const int64_t src_off = r * k.bvecs + c;
        const int64_t dst_off = ((int64_t)p0 * k.brows + r) * k.full_vecs + (int64_t)p1 * k.bvecs + c;
        if (VEC16) {
            const uint4 x = __ldcs(reinterpret_cast<const uint4 *>(k.src[g * k.G + p]) + src_off);
            for (int m = 0; m < k.G; ++m) __stcs(reinterpret_cast<uint4 *>(k.dst[g * k.G + m]) + dst_off, x);
        } else {
            // element-wise: "vectors" are single elements of `elem` bytes
            if (elem == 4) {
                const uint32_t x = reinterpret_cast<const uint32_t *>(k.src[g * k.G + p])[src_off];
                for (int m = 0; m < k.G; ++m) reinterpret_cast<uint32_t *>(k.dst[g * k.G + m])[dst_off] = x;
            } else {
                const uint16_t x = reinterpret_cast<const uint16_t *>(k.src[g * k.G + p])[src_off];
                for (int m = 0; m < k.G; ++m) reinterpret_cast<uint16_t *>(k.dst[g * k.G + m])[dst_off] = x;
            }
        }
    }
}

}  // namespace

namespace shmm {

int launch_reduce(const ReduceArgs &a, int *status, void *stream) {
    (void)status;
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
    if (a.pt == SHMM_F32 && a.ot == SHMM_F32) e = reduce_dispatch<float, float>(k, vec_ok, a.tree, a.gelu, s);
    else if (a.pt == SHMM_F32) e = reduce_dispatch<float, __nv_bfloat16>(k, vec_ok, a.tree, a.gelu, s);
    else if (a.ot == SHMM_BF16) e = reduce_dispatch<__nv_bfloat16, __nv_bfloat16>(k, vec_ok, a.tree, a.gelu, s);
    else e = reduce_dispatch<__nv_bfloat16, float>(k, vec_ok, a.tree, a.gelu, s);
    return (int)e;
}

int launch_gather(const GatherArgs &a, int *status, void *stream) {
    (void)status;
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
    cudaStream_t s = (cudaStream_t)stream;
    const unsigned grid = grid_for(k.nvec * k.ngroups, 256 * 2);
    count_launch();
    if (vec) gather_kernel<true><<<grid, 256, 0, s>>>(k, a.elem);
    else gather_kernel<false><<<grid, 256, 0, s>>>(k, a.elem);
    return (int)cudaGetLastError();
}

}  // namespace shmm
