// Tensor-core local GEMM for sm_103a: every virtual rank's product
// P_r = A_r . B_r over its slice of the contracted dim ("Sharded matrix
// multiplication and result ownership", step 3; "Row Parallelism",
// Z_i = X_i A_i), bf16 inputs, fp32 accumulation, optionally with the
// partial-sum reduction fused into the epilogue (same page, step 4).
//
// Two persistent kernels, one CTA per SM, with the same warp roles:
//   warp 0      TMA producer: per k-block of 64, the CTA's rows of A (K-major,
//               128-byte swizzle) and its columns of B in 64x64 boxes (B is
//               row-major [J,K], i.e. MN-major for the MMA: no transpose)
//               into a shared-memory ring of stages guarded by mbarriers;
//   warp 1      allocates the 512 TMEM columns and issues tcgen05.mma from
//               one thread, committing each stage back to the producer and
//               each finished accumulator to the epilogue;
//   warps 2..   epilogue: tcgen05.ld of the fp32 accumulator (warp w reads
//               TMEM lanes 32*(w%4)..+31, one output row per thread), GeLU,
//               rounding, and bulk tensor stores through shared memory.
// gemm_tc2_kernel<NH> runs on CTA pairs (cta_group::2, M = 256) with
// 256 x 256 (NH = 1) or 256 x 512 (NH = 2) tiles; gemm_tc_kernel<256> on
// single CTAs with 128 x 256 tiles, for local M <= 128.
// Work units are (rank, m-tile, n-tile) or, fused, (group, m-tile, n-tile).
// A launch may carry several independent products (segments: their tiles
// follow one another in one persistent walk), each with its own shapes,
// group size and output mode; operands and outputs are reached through
// per-launch tensor-map tables.
// Fused, the G ranks' products of a reduction group accumulate in one fp32
// TMEM accumulator, rank after rank in ascending order (one contraction over
// the group's concatenated J); with the rank-order option each rank's
// product is its own accumulator and the epilogue adds them in ascending
// rank order in fp32, equal to the standalone reduction bit for bit.  Each
// output tile is written once, to its owner (reduce-scatter) or to every
// member (all-reduce).
//
// Every mbarrier wait is bounded (~2 s of SM clock); on expiry the kernel
// raises an abort flag, records SHMM_ERR_TIMEOUT in the device status word,
// drains its own TMA loads and MMAs, frees TMEM and returns.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "checked.cuh"
#include "device_wait.cuh"
#include "gelu.cuh"
#include "shmm_internal.h"

namespace {

constexpr int BM = 128;          // rows per tile (TMEM lanes)
constexpr int BK = 64;           // bf16 per k-block: one 128-byte swizzle row
constexpr int UMMA_K = 16;       // K of one tcgen05.mma kind::f16
constexpr int kMaxMaps = 16;     // rank operand pairs per launch
constexpr int kThreads = 192;

constexpr int kMaxSegs = 4;      // products (sharded matmuls) per launch

// One product of a launch: its units' local GEMMs (ranks, or reduction
// groups when fused), shapes and output mode.  A launch runs the work items
// of its segments one after another in one persistent tile walk.
struct TcSeg {
    int tile_base;   // first work item of the segment
    int units, G, mode;
    int fused, gelu, out_f32;
    int accum;  // fused: the group's products accumulate in one TMEM buffer
    int64_t M, N, Kd;
    int m_tiles, n_tiles, k_blocks;
    int slot_base;   // operand slots slot_base + unit * Gq + q
    int out_base;    // outputs out_base + unit (unfused) or + unit * G + b
    // each operand slot is a b0 x b1 grid of brows x bcols shards (1 x 1
    // when the operand is read whole)
    int a_b0, a_b1, b_b0, b_b1;
    int64_t a_brows, a_bcols, b_brows, b_bcols;
    int tma_store;  // 1: the epilogue stores through tmC, else per-thread stores
    int64_t out_n;  // elements per output buffer (per-thread stores, bounds-checked build)
};

struct TcK {
    CUtensorMap tmA[kMaxMaps];   // one map per distinct A buffer or shard of the launch
    CUtensorMap tmB[kMaxMaps];
    void *out[kMaxMaps];
    CUtensorMap tmC[kMaxMaps];  // output i as the epilogue's TMA stores see it
    int *status;
    // operand slot i's block p (row-major over its segment's b0 x b1 grid) is
    // map a_idx[i][p]
    uint8_t a_idx[kMaxMaps][kMaxMaps];
    uint8_t b_idx[kMaxMaps][kMaxMaps];
    int n_maps_a, n_maps_b;
    int nseg, total;  // segments; work items of all segments
    // Work items from half_from on are half tiles: item half_from + 2 i + h
    // is 256-column half h of tile half_from + i (half_from = total: none).
    int half_from;
    TcSeg seg[kMaxSegs];
};

// The segment holding work item t.
__device__ __forceinline__ int seg_of(const TcK &k, int t) {
    int si = 0;
    for (int i = 1; i < k.nseg; ++i)
        if (t >= k.seg[i].tile_base) si = i;
    return si;
}

// Operands read in place from an all-gather group's shards: which shard of
// the b0 x b1 grid holds coordinate `x` along one dim, and the coordinate
// inside it.  Boxes never straddle a shard (the planner only fuses when shard
// edges fall on box edges); coordinates past the operand's end stay past the
// last shard's end, where TMA fills zeros.  Grids of one block cost nothing.
__device__ __forceinline__ int shard_split(int blocks, int64_t extent, int64_t x, int32_t *local) {
    if (blocks == 1) {
        *local = (int32_t)x;
        return 0;
    }
    int p = (int)((uint32_t)x / (uint32_t)extent);
    if (p > blocks - 1) p = blocks - 1;
    *local = (int32_t)(x - (int64_t)p * extent);
    return p;
}

// An operand's walk along the contracted dim: the shard holding k-block kb
// and the coordinate inside it (an operand read whole is one shard), advanced
// one k-block at a time (an in-place gather's shard edges along K fall on
// k-block edges), so the producer divides only once per tile.  Past the last
// shard the coordinate keeps growing, as in shard_split.
struct KWalk {
    int p;
    int32_t local;
    __device__ __forceinline__ void start(int blocks, int64_t extent) { p = shard_split(blocks, extent, 0, &local); }
    // true when the walk entered the next shard
    __device__ __forceinline__ bool advance(int blocks, int64_t extent, int step) {
        local += step;
        if (p < blocks - 1 && local >= extent) {
            local -= (int32_t)extent;
            ++p;
            return true;
        }
        return false;
    }
};

// ---- PTX wrappers ------------------------------------------------------

using namespace shmm_dev;

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

// Bulk tensor store of a staged shared-memory box to global memory; bulk
// groups are per-thread state, so one lane issues, commits and waits.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int32_t c0, int32_t c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// At most `keep` (0, 1 or 3) committed store groups may still be reading
// shared memory.
__device__ __forceinline__ void bulk_wait_read(int keep) {
    if (keep >= 3) asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory");
    else if (keep == 1) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
    else asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Every committed store has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Generic-proxy shared-memory writes become visible to the async proxy.
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch.  wait: until the grids this one depends on
// have completed and their memory is visible (returns at once for a grid
// launched without the dependency).  launch_dependents: the next grid in
// the stream may be scheduled, onto SMs this one leaves free, once every
// CTA here has issued it; it runs up to its own wait.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2),
// descriptor version 1, base offset 0 (tiles are 1024-byte aligned).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A
// K-major, B MN-major, N = bn, M = 128.
__host__ __device__ constexpr uint32_t instr_desc(int bn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
           ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
        " [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
        " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
        " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}


// ---- CTA-pair (cluster of 2) helpers for the cta_group::2 kernel ---------

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Arrivals without release semantics, for the epilogue's hand-back of a
// TMEM buffer: it publishes no memory writes.  Its TMEM reads have
// finished (tcgen05.wait::ld) and are ordered before the MMAs that reuse
// the buffer by the tcgen05 fences on both sides of the barrier.  Measured
// at a tile boundary, right after a warp's last bulk store: about 1000
// cycles for a release arrive at cluster scope, about 190 at CTA scope,
// 11 relaxed; the MMA waits for the slowest of them.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait whose success makes the releasing side's earlier writes
// (from any CTA of the cluster) visible: for hand-offs between the pair.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, int *status) {
    const long long t0 = clock64();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if (clock64() - t0 > kWaitLimit) {
            atomicExch(status, (int)SHMM_ERR_TIMEOUT);
            return false;
        }
    }
}

// Counts `bytes` as arrived on a barrier of this CTA without a copy.
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (here: the leader's).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                 int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void umma2_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the mbarrier at this shared offset in both CTAs of the pair once
// every cta_group::2 MMA issued so far by this thread has completed.
__device__ __forceinline__ void umma2_commit_both(uint32_t bar) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar), "h"(mask)
        : "memory");
}

// Instruction descriptor for the pair MMA: M = 256 (128 rows per CTA).
__host__ __device__ constexpr uint32_t instr_desc_pair(int bn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
           ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
}

// Stores n (<= 32) consecutive values of one row starting at `p` (element
// pointer of type fp32 or bf16).  vec: whole 16-byte vectors are legal.
__device__ __forceinline__ void store_run(void *p, const float *v, int n, bool f32, bool vec) {
    if (f32) {
        float *d = static_cast<float *>(p);
        if (vec && n == 32) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4 *>(d + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else {
            for (int i = 0; i < n; ++i) d[i] = v[i];
        }
    } else {
        __nv_bfloat16 *d = static_cast<__nv_bfloat16 *>(p);
        if (vec && n == 32) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
                uint32_t w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(v[i + 2 * j], v[i + 2 * j + 1]);
                    w[j] = *reinterpret_cast<const uint32_t *>(&h);
                }
                *reinterpret_cast<uint4 *>(d + i) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        } else {
            for (int i = 0; i < n; ++i) d[i] = __float2bfloat16_rn(v[i]);
        }
    }
}

// Writes n (<= 32) finished values of output row `row`, columns col0.., of
// unit `unit`: the rank's own block (unfused), the owner's block of a
// reduce-scatter along rows (mode 0) or columns (mode 1), or every group
// member's copy (mode 2).
__device__ __forceinline__ void store_tile_row(const TcK &k, const TcSeg &g, int unit, int Gq, int64_t row,
                                               int64_t col0, const float *v, int n, bool f32, int64_t es) {
    void *const *out = k.out + g.out_base;
    if (!g.fused) {
        const int64_t off = row * g.N + col0;
        if (!in_bounds(k.status, off, n, g.out_n)) return;
        store_run((char *)out[unit] + off * es, v, n, f32, true);
    } else if (g.mode == 0) {
        const int64_t per = g.M / Gq;
        const int b = (int)(row / per);
        const int64_t off = (row - b * per) * g.N + col0;
        if (!in_bounds(k.status, off, n, g.out_n)) return;
        store_run((char *)out[unit * Gq + b] + off * es, v, n, f32, true);
    } else if (g.mode == 1) {
        const int64_t per = g.N / Gq;
        if ((per % 32) == 0) {
            const int b = (int)(col0 / per);
            const int64_t off = row * per + (col0 - b * per);
            if (!in_bounds(k.status, off, n, g.out_n)) return;
            store_run((char *)out[unit * Gq + b] + off * es, v, n, f32, true);
        } else {
            for (int i = 0; i < n; ++i) {
                const int64_t col = col0 + i;
                const int b = (int)(col / per);
                const int64_t off = row * per + (col - b * per);
                if (!in_bounds(k.status, off, 1, g.out_n)) continue;
                store_run((char *)out[unit * Gq + b] + off * es, v + i, 1, f32, false);
            }
        }
    } else {
        const int64_t off = row * g.N + col0;
        if (!in_bounds(k.status, off, n, g.out_n)) return;
        for (int b = 0; b < Gq; ++b) store_run((char *)out[unit * Gq + b] + off * es, v, n, f32, true);
    }
}

// Work item t -> (segment, unit, m-tile, n-tile).  Within a unit the tiles run in
// bands of kBandM m-tiles: m fastest inside a band, then n, then the next
// band.  The CTAs working at one time then cover a roughly square block of
// the output (about 8 x 9.5 tiles for 76 CTA pairs) instead of a few whole
// columns, so each wave streams fewer A row panels and B column panels from
// DRAM.
constexpr int kBandM = 8;
__device__ __forceinline__ void tile_coords(const TcK &k, int t, int *si, int *unit, int *mt, int *nt) {
    *si = seg_of(k, t);
    const TcSeg &g = k.seg[*si];
    t -= g.tile_base;
    const int per_unit = g.m_tiles * g.n_tiles;
    *unit = t / per_unit;
    const int r = t - *unit * per_unit;
    const int band_tiles = kBandM * g.n_tiles;
    const int band = r / band_tiles;
    const int m0 = band * kBandM;
    const int bm = g.m_tiles - m0 < kBandM ? g.m_tiles - m0 : kBandM;  // the last band may be short
    const int q = r - band * band_tiles;
    *mt = m0 + q % bm;
    *nt = q / bm;
}

// Work item t -> its tile's coordinates, and *hh: which 256-column half a
// half-tile item covers (0 or 1), or -1 for a whole tile.
__device__ __forceinline__ void item_coords(const TcK &k, int t, int *si, int *unit, int *mt, int *nt, int *hh) {
    if (t < k.half_from) {
        *hh = -1;
        tile_coords(k, t, si, unit, mt, nt);
        return;
    }
    const int i = t - k.half_from;
    *hh = i & 1;
    tile_coords(k, k.half_from + (i >> 1), si, unit, mt, nt);
}

// Epilogue output staging: 32 KB per CTA, shared evenly by the epilogue
// warps (8 KB each with four warps, 4 KB with eight).  A warp cycles
// through its share in 32 x 32 boxes (4 KB at fp32, 2 KB at bf16), so it
// fills the next box while earlier boxes' stores still read theirs.
constexpr int kStagingBytes = 32 * 1024;

// Row r of a 32 x 32 output box into its staging buffer, in the swizzled
// layout the output tensor maps declare: bf16 rows are 64 bytes and 16-byte
// unit j lands at unit j ^ ((r >> 1) & 3) (64-byte swizzle); fp32 rows are
// 128 bytes and unit j lands at j ^ (r & 7) (128-byte swizzle).  A warp's 32
// rows then spread over all banks: four shared-memory wavefronts per 16-byte
// store, the minimum for 512 bytes.
__device__ __forceinline__ void stage_row(uint32_t buf, int r, const float *v, bool f32) {
    if (f32) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t a = buf + (uint32_t)(r * 128 + ((j ^ (r & 7)) * 16));
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v[4 * j]), "f"(v[4 * j + 1]),
                         "f"(v[4 * j + 2]), "f"(v[4 * j + 3])
                         : "memory");
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
                w[i] = *reinterpret_cast<const uint32_t *>(&h);
            }
            const uint32_t a = buf + (uint32_t)(r * 64 + ((j ^ ((r >> 1) & 3)) * 16));
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                         "r"(w[3])
                         : "memory");
        }
    }
}

// Final pass over one finished 256-column sub-tile for one epilogue warp:
// output rows row0..row0+31 (row0 < M), the 32-column chunks c0..c1-1 of
// the sub-tile starting at column col_base, TMEM lanes from lane_s.  Each
// chunk is loaded from TMEM, passed through GeLU if asked, rounded into the
// next box of the warp's staging share (`share` bytes at cbuf) and written
// by one bulk tensor store per destination: the unit's block, the owner's
// block of a reduce-scatter, or every member's copy of an all-reduce.
// Stores clip at the output's edges.  `staged` counts the warp's boxes (it
// picks the box).
__device__ __forceinline__ void store_tile_tma(const TcK &k, const TcSeg &g, int unit, int Gq, int row0,
                                               int col_base, int c0, int c1, uint32_t lane_s, uint32_t cbuf,
                                               uint32_t share, uint32_t *staged, int lane) {
    const bool f32 = g.out_f32 != 0;
    const CUtensorMap *tmC = k.tmC + g.out_base;
    const uint32_t box = f32 ? 4096u : 2048u;
    const uint32_t nbuf = share / box;  // 1, 2 or 4
#pragma unroll 1
    for (int c = c0; c < c1; ++c) {
        const int col0 = col_base + c * 32;
        if (col0 >= g.N) break;
        float v[32];
        tmem_ld32(lane_s + (uint32_t)(c * 32), v);
        if (g.gelu) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = gelu_tanh(v[i]);
        }
        const uint32_t buf = cbuf + (*staged % nbuf) * box;
        if (lane == 0) bulk_wait_read((int)nbuf - 1);  // the store nbuf boxes back has read this box
        __syncwarp();
        stage_row(buf, lane, v, f32);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (!g.fused) {
                tma_store_2d(&tmC[unit], buf, col0, row0);
            } else if (g.mode == 0) {
                const int per = (int)(g.M / Gq), b = row0 / per;
                tma_store_2d(&tmC[unit * Gq + b], buf, col0, row0 - b * per);
            } else if (g.mode == 1) {
                const int per = (int)(g.N / Gq), b = col0 / per;
                tma_store_2d(&tmC[unit * Gq + b], buf, col0 - b * per, row0);
            } else {
                for (int b = 0; b < Gq; ++b) tma_store_2d(&tmC[unit * Gq + b], buf, col0, row0);
            }
            bulk_commit();
        }
        ++*staged;
    }
}

// Epilogue of one warp (warps 2..5) over the tiles its CTA (or CTA pair)
// owns: work items first, first + stride, ... < total; output rows
// mt * tile_rows + row_base + [0, 32) of each tile, TMEM lanes from
// lane_base.  A tile is NH sub-tiles of 256 columns.  With NH = 1, tile i's
// sum S sits in TMEM buffer i % 2; in rank order the group's later products
// arrive in the other buffer W and are folded into S (fp32, ascending rank
// order), W handed back after each; accumulating, S already holds the sum.
// With NH = 2 (accumulating or unfused only), sub-tile h sits in buffer h.
// Then GeLU if asked, one rounding and the stores (bulk tensor stores
// through the staging buffers at cbuf, or per thread), and S is handed back.
// full_bar(b): the barrier on which the MMA thread reports a finished
// product in buffer b; release(b): hands buffer b back (every lane calls
// it after its last TMEM read of the buffer; one arrival per warp).
template <int NH, typename FullBar, typename Release>
__device__ __forceinline__ void drain_tiles(const TcK &k, int first, int stride, int tile_rows, int row_base,
                                            uint32_t lane_base, int c0, int c1, uint32_t cbuf, uint32_t share,
                                            int lane, volatile int *abort_flag, FullBar full_bar, Release release) {
    constexpr int BN = 256;
    uint32_t staged = 0;
    uint32_t used0 = 0, used1 = 0;  // finished products consumed per buffer
    // One lane waits; the warp reconverges before the .sync.aligned TMEM
    // instructions.
    auto warp_wait_full = [&](int b) -> bool {
        const uint32_t n = b ? used1 : used0;
        int ok = 1;
        if (lane == 0) ok = mbar_wait(full_bar(b), n & 1, abort_flag, k.status) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (b) ++used1;
        else ++used0;
        if (ok) fence_after();
        return ok != 0;
    };
    int tile_iter = 0;
    bool ok = true;
    for (int t = first; t < k.total && ok; t += stride, ++tile_iter) {
        int si, unit, mt, nt, hh;
        item_coords(k, t, &si, &unit, &mt, &nt, &hh);
        const TcSeg &g = k.seg[si];
        const int Gq = g.fused ? g.G : 1;
        const bool f32 = g.out_f32 != 0;
        const int64_t es = f32 ? 4 : 2;
        const int nh = hh >= 0 ? 1 : NH;  // a half tile fills buffer 0 only
        for (int h = 0; h < nh && ok; ++h) {
            const int bS = NH == 2 ? h : (tile_iter & 1), bW = bS ^ 1;
            const uint32_t s_base = lane_base + (uint32_t)(bS * BN);
            const uint32_t w_base = lane_base + (uint32_t)(bW * BN);
            if (!warp_wait_full(bS)) {  // S = product of the group's first rank
                ok = false;
                break;
            }
            const int folds = g.accum || NH == 2 ? 1 : Gq;  // accum: S already holds the sum
            for (int q = 1; q < folds; ++q) {
                // S = S + P_q in fp32: the ascending-rank sequential sum
                if (!warp_wait_full(bW)) {
                    ok = false;
                    break;
                }
#pragma unroll 1
                for (int c = c0; c < c1; ++c) {
                    float a[32], w[32];
                    tmem_ld32(s_base + (uint32_t)(c * 32), a);
                    tmem_ld32(w_base + (uint32_t)(c * 32), w);
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = a[i] + w[i];
                    tmem_st32(s_base + (uint32_t)(c * 32), a);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                release(bW);  // W may take the next product
            }
            if (!ok) break;
            const int row0 = mt * tile_rows + row_base;
            const int col_base = (nt * NH + (hh >= 0 ? hh : h)) * BN;
            if (g.tma_store) {
                if (row0 < g.M)
                    store_tile_tma(k, g, unit, Gq, row0, col_base, c0, c1, s_base, cbuf, share, &staged, lane);
            } else {
                const int64_t row = (int64_t)row0 + lane;
                const bool row_ok = row < g.M;
#pragma unroll 1
                for (int c = c0; c < c1; ++c) {
                    float v[32];
                    tmem_ld32(s_base + (uint32_t)(c * 32), v);
                    if (g.gelu) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = gelu_tanh(v[i]);
                    }
                    const int64_t col0 = (int64_t)col_base + c * 32;
                    if (!row_ok || col0 >= g.N) continue;
                    const int n = (int)((g.N - col0) < 32 ? (g.N - col0) : 32);
                    store_tile_row(k, g, unit, Gq, row, col0, v, n, f32, es);
                }
            }
            release(bS);  // S may take the next tile's products
        }
    }
    if (lane == 0) bulk_wait_all();  // no store still reads staging at exit
    __syncwarp();
}

template <int BN>
struct Cfg {
    static constexpr int A_BYTES = BM * BK * 2;           // 16 KB
    static constexpr int B_BYTES = BK * BN * 2;           // BN * 128
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int STAGES = (200 * 1024) / STAGE > 8 ? 8 : (200 * 1024) / STAGE;
    static constexpr int SMEM = STAGES * STAGE + kStagingBytes + 1024 /*align*/ + 1024 /*barriers, tables*/;
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ TcK k) {
    using C = Cfg<BN>;
    constexpr int S = C::STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *tiles = smem;
    uint8_t *staging = smem + S * C::STAGE;  // 1024-byte aligned: the swizzle needs it
    uint64_t *bars = reinterpret_cast<uint64_t *>(staging + kStagingBytes);
    // bars: full[S], empty[S], acc_full[2], acc_empty[2], drain
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * S + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    // Operand slot -> map tables, copied once from the parameters into the
    // shared-memory tail (the producer looks a tile's maps up there).
    uint8_t *s_aidx = reinterpret_cast<uint8_t *>(tmem_holder + 16);
    uint8_t *s_bidx = s_aidx + kMaxMaps * kMaxMaps;
    for (int i = threadIdx.x; i < kMaxMaps * kMaxMaps; i += blockDim.x) {
        s_aidx[i] = k.a_idx[i / kMaxMaps][i % kMaxMaps];
        s_bidx[i] = k.b_idx[i / kMaxMaps][i % kMaxMaps];
    }

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int total = k.total;

    auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
    auto empty_bar = [&](int s) { return smem_u32(&bars[S + s]); };
    auto accf_bar = [&](int s) { return smem_u32(&bars[2 * S + s]); };
    auto acce_bar = [&](int s) { return smem_u32(&bars[2 * S + 2 + s]); };
    const uint32_t drain_bar = smem_u32(&bars[2 * S + 4]);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(accf_bar(s), 1);
            mbar_init(acce_bar(s), 4);  // one arrival per epilogue warp
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_u32(tmem_holder))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // The prologue above (no global memory) may overlap the end of the
    // previous kernel in the stream; the tiles wait for it.
    grid_dependency_wait();
    grid_launch_dependents();

    auto decode = [&](int t, int *si, int *unit, int *mt, int *nt) { tile_coords(k, t, si, unit, mt, nt); };

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            for (int i = 0; i < k.n_maps_a; ++i) prefetch_map(&k.tmA[i]);
            for (int i = 0; i < k.n_maps_b; ++i) prefetch_map(&k.tmB[i]);
            uint32_t it = 0;
            int last_parity[8];
            for (int s = 0; s < 8; ++s) last_parity[s] = -1;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                int si, unit, mt, nt;
                decode(t, &si, &unit, &mt, &nt);
                const TcSeg &g = k.seg[si];
                const int Gq = g.fused ? g.G : 1;
                for (int q = 0; q < Gq && ok; ++q) {
                    const int ri = g.slot_base + unit * Gq + q;
                    // The slot's maps are looked up once per tile: the row of A
                    // and each B box's column shard are fixed for it; the K
                    // shards (in-place gathers split K) advance.
                    constexpr int NB = BN / 64;
                    int32_t a_r, bx[NB];
                    int bp1[NB];
                    const int a_p0 = shard_split(g.a_b0, g.a_brows, (int64_t)mt * BM, &a_r);
                    KWalk wa, wb;
                    wa.start(g.a_b1, g.a_bcols);
                    wb.start(g.b_b0, g.b_brows);
                    const CUtensorMap *map_a = &k.tmA[s_aidx[ri * kMaxMaps + a_p0 * g.a_b1 + wa.p]];
                    const CUtensorMap *map_b[NB];
#pragma unroll
                    for (int c = 0; c < NB; ++c) {
                        bp1[c] = shard_split(g.b_b1, g.b_bcols, (int64_t)nt * BN + c * 64, &bx[c]);
                        map_b[c] = &k.tmB[s_bidx[ri * kMaxMaps + wb.p * g.b_b1 + bp1[c]]];
                    }
                    for (int kb = 0; kb < g.k_blocks; ++kb, ++it) {
                        const int s = it % S;
                        const uint32_t ph = (it / S) & 1;
                        if (!mbar_wait(empty_bar(s), ph ^ 1, abort_flag, k.status)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(full_bar(s), C::STAGE);
                        const uint32_t a_dst = smem_u32(tiles + s * C::STAGE);
                        const uint32_t b_dst = a_dst + C::A_BYTES;
                        tma_load_2d(a_dst, map_a, full_bar(s), wa.local, a_r);
#pragma unroll
                        for (int c = 0; c < NB; ++c) tma_load_2d(b_dst + c * 8192, map_b[c], full_bar(s), bx[c], wb.local);
                        if (wa.advance(g.a_b1, g.a_bcols, BK))
                            map_a = &k.tmA[s_aidx[ri * kMaxMaps + a_p0 * g.a_b1 + wa.p]];
                        if (wb.advance(g.b_b0, g.b_brows, BK))
#pragma unroll
                            for (int c = 0; c < NB; ++c) map_b[c] = &k.tmB[s_bidx[ri * kMaxMaps + wb.p * g.b_b1 + bp1[c]]];
                        last_parity[s] = (int)ph;
                    }
                }
            }
            // Never leave a TMA write to shared memory in flight at exit.
            for (int s = 0; s < S; ++s)
                if (last_parity[s] >= 0)
                    mbar_wait(full_bar(s), (uint32_t)last_parity[s], abort_flag, k.status, false);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        // Two TMEM buffers of BN columns.  Tile i (this CTA's i-th) keeps its
        // running sum S in buffer i%2.  Rank order: ranks 1..G-1 of the tile
        // are computed in the other buffer W and folded into S by the
        // epilogue.  Accumulating (k.accum): every rank's k-blocks continue
        // the same accumulation in S, one contraction over the group's
        // concatenated K.  A buffer is refilled only after the epilogue
        // released its previous contents.
        if (lane == 0) {
            constexpr uint32_t idesc = instr_desc(BN);
            uint32_t it = 0;
            uint32_t fills0 = 0, fills1 = 0;
            int tile_iter = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tile_iter) {
                const TcSeg &g = k.seg[seg_of(k, t)];
                const int Gq = g.fused ? g.G : 1;
                const bool accum = g.accum != 0;
                const int k_blocks = g.k_blocks;
                const int bS = tile_iter & 1;
                for (int q = 0; q < Gq && ok; ++q) {
                    // accum: every rank's product continues the sum in S
                    const bool into_s = q == 0 || accum;
                    const int b = into_s ? bS : (bS ^ 1);
                    const uint32_t nf = b ? fills1 : fills0;
                    if ((q == 0 || !accum) && !mbar_wait(acce_bar(b), (nf & 1) ^ 1, abort_flag, k.status)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(b * BN);
                    for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                        const int s = it % S;
                        const uint32_t ph = (it / S) & 1;
                        if (!mbar_wait(full_bar(s), ph, abort_flag, k.status)) {
                            ok = false;
                            break;
                        }
                        fence_after();
                        const uint32_t a_addr = smem_u32(tiles + s * C::STAGE);
                        const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                            // A: K-major, advance 32 bytes per 16 k inside the
                            // swizzle row.  B: MN-major, 16 k rows = 2 atoms.
                            const uint64_t ad = smem_desc(a_addr + kk * 32, 16, 1024);
                            const uint64_t bd = smem_desc(b_addr + kk * 2048, 8192, 1024);
                            umma_f16(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0 || (q > 0 && accum)) ? 1u : 0u);
                        }
                        umma_commit(empty_bar(s));
                    }
                    if (!ok) break;
                    if (accum && q < Gq - 1) continue;  // S is not finished
                    umma_commit(accf_bar(b));
                    if (b) ++fills1;
                    else ++fills0;
                }
            }
            // Drain: every MMA issued by this thread has completed.
            umma_commit(drain_bar);
            mbar_wait(drain_bar, 0, abort_flag, k.status, false);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int quad = warp % 4;
        drain_tiles<1>(k, blockIdx.x, gridDim.x, BM, quad * 32, tmem_base + ((uint32_t)(quad * 32) << 16),
                       0, BN / 32, smem_u32(staging) + (uint32_t)((warp - 2) * (kStagingBytes / 4)),
                       kStagingBytes / 4, lane, abort_flag,
                    [&](int b) { return accf_bar(b); },
                    [&](int b) {
                        fence_before();
                        __syncwarp();
                        if (lane == 31) mbar_arrive_relaxed(acce_bar(b));
                    });
    }

    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem_base)
                     : "memory");
    }
}


// ---- CTA-pair kernel: 256 x (256 NH) output tiles on two SMs --------------
//
// A cluster of two CTAs computes one tile with tcgen05.mma cta_group::2
// (M = 256, N = 256, K = 16): each CTA stages its own 128 rows of A and its
// 128 of each 256-column half's columns of B, and the pair's accumulator is
// split by rows over the two TMEMs.  The even CTA (the leader) issues the
// MMAs; both CTAs' TMA loads complete on the leader's full barrier; the
// leader's commits reach both CTAs' barriers.  Each CTA's epilogue drains
// its own 128 rows exactly as in the single-CTA kernel.
//
// NH = 1: 256x256 tiles, 32 KB per CTA per k-block (6 stages), TMEM holds two
// tiles so one tile's epilogue overlaps the next tile's MMAs.  NH = 2:
// 256x512 tiles, two MMAs per K step sharing the A operand, 48 KB per CTA
// per k-block (4 stages): a quarter fewer operand bytes per FLOP, for
// products whose operand loads (not the tensor pipe) set the pace.  The
// tile's two halves fill all of TMEM, so the next tile's MMAs into half h
// wait until the epilogue has drained half h.  NH = 2 serves accumulating
// or unfused launches only (no rank-order fold needs a spare buffer).

template <int NH>
struct Cfg2 {
    static constexpr int A_BYTES = BM * BK * 2;        // 16 KB: this CTA's 128 rows
    static constexpr int B_BYTES = NH * BK * 128 * 2;  // 16 KB per half: this CTA's 128 columns of it
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int STAGES = NH == 1 ? 6 : 4;
    static constexpr int SMEM = STAGES * STAGE + kStagingBytes + 1024 /*align*/ + 1024 /*barriers, tables*/;
    // Epilogue warps: with a tile's drain exposed (NH = 2), two per TMEM lane
    // quadrant, each draining half of the columns, so the drain takes half
    // as long.
    static constexpr int EPI_WARPS = NH == 2 ? 8 : 4;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
};

template <int NH>
__global__ void __launch_bounds__(Cfg2<NH>::THREADS, 1) gemm_tc2_kernel(const __grid_constant__ TcK k) {
    using C = Cfg2<NH>;
    constexpr int S = C::STAGES;
    constexpr int BN = 256;           // N of one MMA, and of one TMEM buffer
    constexpr int TW = BN * NH;       // tile width
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *tiles = smem;
    uint8_t *staging = smem + S * C::STAGE;  // 1024-byte aligned: the swizzle needs it
    uint64_t *bars = reinterpret_cast<uint64_t *>(staging + kStagingBytes);
    // bars: full[S], empty[S], acc_full[2], acc_empty[2], drain
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * S + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    // The peer producer's final load count, handed to the leader through
    // handoff_bar (both used in the leader CTA only).
    volatile uint32_t *peer_issued = tmem_holder + 2;
    uint64_t *handoff = reinterpret_cast<uint64_t *>(tmem_holder + 4);
    // ... and its bytes of each of its last S stages (slots 6 .. 6 + S - 1)
    volatile uint32_t *peer_bytes = tmem_holder + 6;
    static_assert(S <= 8, "the peer's stage bytes take slots 6..13 before the map tables at slot 16");
    // Operand slot -> map tables, copied once from the parameters into the
    // shared-memory tail (the producer looks a tile's maps up there).
    uint8_t *s_aidx = reinterpret_cast<uint8_t *>(tmem_holder + 16);
    uint8_t *s_bidx = s_aidx + kMaxMaps * kMaxMaps;
    for (int i = threadIdx.x; i < kMaxMaps * kMaxMaps; i += blockDim.x) {
        s_aidx[i] = k.a_idx[i / kMaxMaps][i % kMaxMaps];
        s_bidx[i] = k.b_idx[i / kMaxMaps][i % kMaxMaps];
    }

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t cr = cluster_ctarank();  // 0: leader, 1: peer
    const uint32_t handoff_bar = smem_u32(handoff);
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int total = k.total;  // 256 x TW tiles of every segment

    auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
    auto empty_bar = [&](int s) { return smem_u32(&bars[S + s]); };
    auto accf_bar = [&](int s) { return smem_u32(&bars[2 * S + s]); };
    auto acce_bar = [&](int s) { return smem_u32(&bars[2 * S + 2 + s]); };
    const uint32_t drain_bar = smem_u32(&bars[2 * S + 4]);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(accf_bar(s), 1);
            mbar_init(acce_bar(s), 2 * C::EPI_WARPS);  // both CTAs' epilogue warps
        }
        mbar_init(drain_bar, 1);
        mbar_init(handoff_bar, 1);
        *abort_flag = 0;
        *peer_issued = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        // collective over the pair: the same columns in both TMEMs
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_u32(tmem_holder))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any remote use
    fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // The prologue above (no global memory) may overlap the end of the
    // previous kernel in the stream; the tiles wait for it.
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        if (lane == 0) {
            for (int i = 0; i < k.n_maps_a; ++i) prefetch_map(&k.tmA[i]);
            for (int i = 0; i < k.n_maps_b; ++i) prefetch_map(&k.tmB[i]);
            uint32_t it = 0;  // stages loaded
            uint32_t stage_bytes[S];  // this CTA's bytes of each stage it loaded last
            bool ok = true;
            for (int t = pair; t < total && ok; t += npairs) {
                int si, unit, mt, nt, hh;
                item_coords(k, t, &si, &unit, &mt, &nt, &hh);
                const TcSeg &g = k.seg[si];
                const int Gq = g.fused ? g.G : 1;
                // A half tile loads A and the two B boxes of its half, into the
                // first half's slots.
                const int nb = hh >= 0 ? 2 : 2 * NH;
                const uint32_t bytes = hh >= 0 ? (uint32_t)(C::A_BYTES + C::B_BYTES / NH) : (uint32_t)C::STAGE;
                for (int q = 0; q < Gq && ok; ++q) {
                    const int ri = g.slot_base + unit * Gq + q;
                    // The slot's maps are looked up once per tile: the row of A
                    // and each B box's column shard are fixed for it; the K
                    // shards (in-place gathers split K) advance.
                    constexpr int NB = 2 * NH;
                    int32_t a_r, bx[NB];
                    int bp1[NB];
                    const int a_p0 = shard_split(g.a_b0, g.a_brows, (int64_t)mt * 256 + (int)cr * BM, &a_r);
                    KWalk wa, wb;
                    wa.start(g.a_b1, g.a_bcols);
                    wb.start(g.b_b0, g.b_brows);
                    const CUtensorMap *map_a = &k.tmA[s_aidx[ri * kMaxMaps + a_p0 * g.a_b1 + wa.p]];
                    const CUtensorMap *map_b[NB];
#pragma unroll
                    for (int j = 0; j < NB; ++j) {
                        const int jj = hh >= 0 ? 2 * hh + (j & 1) : j;  // the box's place in the whole tile
                        bp1[j] = shard_split(g.b_b1, g.b_bcols,
                                             (int64_t)nt * TW + (jj / 2) * BN + (int)cr * 128 + (jj % 2) * 64, &bx[j]);
                        map_b[j] = &k.tmB[s_bidx[ri * kMaxMaps + wb.p * g.b_b1 + bp1[j]]];
                    }
                    for (int kb = 0; kb < g.k_blocks; ++kb, ++it) {
                        const int s = it % S;
                        const uint32_t ph = (it / S) & 1;
                        if (!mbar_wait(empty_bar(s), ph ^ 1, abort_flag, k.status)) {
                            ok = false;
                            break;
                        }
                        if (cr == 0) mbar_expect_tx(full_bar(s), 2 * bytes);
                        stage_bytes[s] = bytes;
                        const uint32_t bar = mapa_shared(full_bar(s), 0);
                        const uint32_t a_dst = smem_u32(tiles + s * C::STAGE);
                        const uint32_t b_dst = a_dst + C::A_BYTES;
                        tma_load_2d_pair(a_dst, map_a, bar, wa.local, a_r);
#pragma unroll
                        for (int j = 0; j < NB; ++j)
                            if (j < nb) tma_load_2d_pair(b_dst + j * 8192, map_b[j], bar, bx[j], wb.local);
                        if (wa.advance(g.a_b1, g.a_bcols, BK))
                            map_a = &k.tmA[s_aidx[ri * kMaxMaps + a_p0 * g.a_b1 + wa.p]];
                        if (wb.advance(g.b_b0, g.b_brows, BK))
#pragma unroll
                            for (int j = 0; j < NB; ++j) map_b[j] = &k.tmB[s_bidx[ri * kMaxMaps + wb.p * g.b_b1 + bp1[j]]];
                    }
                }
            }
            // Both CTAs' loads of a stage complete on the leader's barrier, so
            // the leader alone can tell when every load of the pair has
            // landed; the peer cannot leave before it does (the cluster
            // barrier at the end).  The peer hands over how many stages it
            // loaded.  Without an abort both CTAs loaded the same stages; after
            // one they may differ by up to S stages (each loads stage i only
            // after the MMAs freed stage i - S, which needed the leader to
            // have armed it): the leader arms the peer's extra stages for the
            // peer's half, and stands in for the half the peer never loaded,
            // so every stage's last phase completes once the loads that were
            // issued have landed.
            // A stage's bytes depend on its work item (whole or half tile), so
            // the peer hands over its bytes of its last S stages as well.
            if (cr == 1) {
                for (int s = 0; s < S; ++s)
                    if ((uint32_t)s < it)
                        st_cluster_u32(mapa_shared(smem_u32((const void *)(peer_bytes + s)), 0), stage_bytes[s]);
                st_cluster_u32(mapa_shared(smem_u32((const void *)peer_issued), 0), it);
                mbar_arrive_cluster(mapa_shared(handoff_bar, 0));
            } else {
                uint32_t it_peer = it;
                if (mbar_wait_cluster(handoff_bar, 0, k.status)) it_peer = *peer_issued;
                const uint32_t it_max = it_peer > it ? it_peer : it;
                for (uint32_t i = it_peer < it ? it_peer : it; i < it_max; ++i) {
                    const int s = (int)(i % S);
                    if (i >= it) mbar_expect_tx(full_bar(s), peer_bytes[s]);  // the peer's half only
                    else mbar_complete_tx(full_bar(s), stage_bytes[s]);       // the half never loaded
                }
                for (uint32_t i = it_max > (uint32_t)S ? it_max - S : 0; i < it_max; ++i)
                    mbar_wait(full_bar((int)(i % S)), (i / S) & 1, abort_flag, k.status, false);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (leader CTA only) ----------------
        if (lane == 0 && cr == 0) {
            constexpr uint32_t idesc = instr_desc_pair(BN);
            uint32_t it = 0;
            uint32_t fills[2] = {0, 0};  // products finished per TMEM buffer
            int tile_iter = 0;
            bool ok = true;
            for (int t = pair; t < total && ok; t += npairs, ++tile_iter) {
                const bool half = t >= k.half_from;  // a half tile: buffer 0 only
                const int nh = half ? 1 : NH;
                const TcSeg &g = k.seg[seg_of(k, half ? k.half_from + ((t - k.half_from) >> 1) : t)];
                const int Gq = g.fused ? g.G : 1;
                const bool accum = g.accum != 0;
                const int k_blocks = g.k_blocks;
                // NH = 1: the tile's sum S in buffer tile_iter % 2 (rank order:
                // later products in the other); NH = 2: half h in buffer h
                const int bS = NH == 2 ? 0 : (tile_iter & 1);
                for (int q = 0; q < Gq && ok; ++q) {
                    // accum: every rank's product continues the sum in S
                    const bool into_s = q == 0 || accum;
                    const int b = into_s ? bS : (bS ^ 1);
                    const bool fresh = q == 0 || !accum;  // this product starts its buffers
                    // The four K=16 MMAs of the k-block in stage st into buffer
                    // buf, half h of the stage's B; `first` starts the buffer's
                    // sum instead of adding to it.
                    auto issue = [&](int st, int buf, int h, bool first) {
                        const uint32_t a_addr = smem_u32(tiles + st * C::STAGE);
                        const uint32_t b_addr = a_addr + C::A_BYTES + (uint32_t)(h * 16384);
                        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                            const uint64_t ad = smem_desc(a_addr + kk * 32, 16, 1024);
                            const uint64_t bd = smem_desc(b_addr + kk * 2048, 8192, 1024);
                            umma2_f16(d_tmem, ad, bd, idesc, (!first || kk > 0) ? 1u : 0u);
                        }
                    };
                    // A fresh buffer waits until the epilogue has handed back
                    // its previous fill.
                    auto wait_free = [&](int buf) -> bool {
                        if (!mbar_wait(acce_bar(buf), (fills[buf] & 1) ^ 1, abort_flag, k.status)) return false;
                        fence_after();
                        return true;
                    };
                    int kb = 0;
                    if (NH == 2 && fresh) {
                        // Half 0 runs ahead over the first R loaded stages while the
                        // epilogue still drains half 1 of the previous tile, then half 1
                        // catches up on the same stages; each half still adds its
                        // k-blocks in ascending order.
                        const int R = k_blocks < S ? k_blocks : S;
                        if (!wait_free(b)) {
                            ok = false;
                            break;
                        }
                        for (kb = 0; kb < R; ++kb) {
                            const uint32_t u = it + (uint32_t)kb;
                            if (!mbar_wait(full_bar((int)(u % S)), (u / S) & 1, abort_flag, k.status)) {
                                ok = false;
                                break;
                            }
                            fence_after();
                            issue((int)(u % S), b, 0, kb == 0);
                            if (half) umma2_commit_both(empty_bar((int)(u % S)));
                        }
                        if (!ok) break;
                        if (!half) {
                            if (!wait_free(b + 1)) {
                                ok = false;
                                break;
                            }
                            for (kb = 0; kb < R; ++kb) {
                                const int st = (int)((it + (uint32_t)kb) % S);
                                issue(st, b + 1, 1, kb == 0);
                                umma2_commit_both(empty_bar(st));
                            }
                        }
                        it += (uint32_t)R;
                    }
                    for (; kb < k_blocks && ok; ++kb, ++it) {
                        const int s = it % S;
                        const uint32_t ph = (it / S) & 1;
                        if (!mbar_wait(full_bar(s), ph, abort_flag, k.status)) {
                            ok = false;
                            break;
                        }
                        fence_after();
#pragma unroll
                        for (int h = 0; h < NH; ++h) {
                            if (h >= nh) break;
                            if (kb == 0 && fresh && !wait_free(b + h)) {  // 256x256 tiles only
                                ok = false;
                                break;
                            }
                            issue(s, b + h, h, kb == 0 && !(q > 0 && accum));
                        }
                        if (!ok) break;
                        umma2_commit_both(empty_bar(s));
                    }
                    if (!ok) break;
                    if (accum && q < Gq - 1) continue;  // S is not finished
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        if (h >= nh) break;
                        umma2_commit_both(accf_bar(b + h));
                        ++fills[b + h];
                    }
                }
            }
            umma2_commit_both(drain_bar);
            mbar_wait(drain_bar, 0, abort_flag, k.status, false);
        }
    } else {
        // ---------------- epilogue (warps 2.., both CTAs) ----------------
        // A warp reaches only its own TMEM lane quadrant (warp % 4); with
        // eight epilogue warps, two share a quadrant and split the columns.
        const int ew = warp - 2;
        const int quad = warp % 4;
        constexpr int CH = (BN / 32) / (C::EPI_WARPS / 4);  // 32-column chunks per warp
        const int c0 = (ew / 4) * CH;
        constexpr uint32_t share = kStagingBytes / C::EPI_WARPS;
        drain_tiles<NH>(k, pair, npairs, 256, (int)cr * BM + quad * 32,
                    tmem_base + ((uint32_t)(quad * 32) << 16), c0, c0 + CH,
                    smem_u32(staging) + (uint32_t)ew * share, share, lane, abort_flag,
                    [&](int b) { return accf_bar(b); },
                    [&](int b) {
                        fence_before();
                        __syncwarp();
                        if (lane == 31) mbar_arrive_cluster_relaxed(mapa_shared(acce_bar(b), 0));  // the leader's barrier
                    });
    }

    fence_before();
    __syncthreads();
    cluster_sync_all();  // no CTA leaves while its peer may still signal it
    fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 512;" ::"r"(tmem_base)
                     : "memory");
    }
}

// ---- host side ----------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(std::string *msg) {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    static std::string err;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e =
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p)
            err = "cuTensorMapEncodeTiled not available from the driver";
        else
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!fn && msg) *msg = err;
    return fn;
}

// 2-D tensor map over a row-major rows x cols matrix, box (bx inner, by):
// bf16 operands with 128-byte swizzle by default; the epilogue's output maps
// pass their own element type and swizzle.
bool make_map(EncodeTiledFn fn, CUtensorMap *m, const void *base, int64_t rows, int64_t cols, uint32_t bx,
              uint32_t by, bool f32 = false, CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(cols * (f32 ? 4 : 2))};
    const cuuint32_t box[2] = {bx, by};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoded tensor maps, reused across calls: a map holds nothing but the
// address, shape, strides and box it was encoded with, so an entry matching
// all of them is valid whatever allocation now lives at that address.
struct MapCacheEntry {
    const void *ptr;
    int64_t rows, cols;
    uint32_t bx, by;
    bool f32;
    CUtensorMapSwizzle sw;
    bool valid;
    CUtensorMap map;
};

bool cached_map(EncodeTiledFn fn, CUtensorMap *m, const void *base, int64_t rows, int64_t cols, uint32_t bx,
                uint32_t by, bool f32 = false, CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B) {
    constexpr int kEntries = 64;
    thread_local MapCacheEntry cache[kEntries] = {};
    thread_local int next = 0;
    for (int i = 0; i < kEntries; ++i) {
        const MapCacheEntry &e = cache[i];
        if (e.valid && e.ptr == base && e.rows == rows && e.cols == cols && e.bx == bx && e.by == by &&
            e.f32 == f32 && e.sw == sw) {
            *m = e.map;
            return true;
        }
    }
    MapCacheEntry &e = cache[next];
    next = (next + 1) % kEntries;
    e.valid = false;
    if (!make_map(fn, &e.map, base, rows, cols, bx, by, f32, sw)) return false;
    e.ptr = base;
    e.f32 = f32;
    e.sw = sw;
    e.rows = rows;
    e.cols = cols;
    e.bx = bx;
    e.by = by;
    e.valid = true;
    *m = e.map;
    return true;
}

int num_sms() {
    static shmm::PerDevice<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= shmm::kMaxDevices) return 148;
    int n = cache.get(dev);
    if (n) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache.set(dev, n);
    return n;
}

// Tile grid of every segment for tiles of tile_rows x tile_cols: the
// segments' work items follow one another in segment order.
void set_tiles(TcK &k, int tile_rows, int tile_cols) {
    int base = 0;
    for (int i = 0; i < k.nseg; ++i) {
        TcSeg &g = k.seg[i];
        g.m_tiles = (int)((g.M + tile_rows - 1) / tile_rows);
        g.n_tiles = (int)((g.N + tile_cols - 1) / tile_cols);
        g.tile_base = base;
        base += g.units * g.m_tiles * g.n_tiles;
    }
    k.total = base;
    k.half_from = base;
}

// Tiles of a partial last wave of 256 x 512 tiles that run as 256-column
// halves: when the wave would leave at least half the pairs idle, its r
// tiles become 2 r half tiles, one round on 2 r pairs.  A half tile has
// half the MMAs of a whole one for two thirds of its loads (A, and B of its
// half), so it runs at the 256 x 256 kernel's load-bound rate: about 0.6
// of a whole tile's time.  The halves add every output element's products
// in the same order as the whole tile.  Returns r, or 0 for no split;
// SHMM_TC_HALF_TAIL=0 turns it off.
int tail_halves(int64_t tiles, int pairs) {
    const char *e = getenv("SHMM_TC_HALF_TAIL");
    if (e && e[0] == '0') return 0;
    if (pairs < 1 || tiles < pairs) return 0;
    const int64_t r = tiles % pairs;
    return (r > 0 && 2 * r <= pairs) ? (int)r : 0;
}

template <int BN>
cudaError_t launch_bn(TcK &k, cudaStream_t s, int max_sms) {
    using C = Cfg<BN>;
    static shmm::PerDevice<int> attr_set;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= shmm::kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set.get(dev)) {
        e = cudaFuncSetAttribute(gemm_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set.set(dev, 1);
    }
    set_tiles(k, BM, BN);
    const int64_t total = k.total;
    int ctas = num_sms();
    if (max_sms > 0 && max_sms < ctas) ctas = max_sms;
    const int grid = (int)(total < ctas ? total : ctas);
    // a programmatic dependent of the kernel before it, as the pair kernel
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    const char *pdl = getenv("SHMM_PDL");
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = (pdl && pdl[0] == '0') ? 0 : 1;
    shmm::count_launch();
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN>, k);
}

// CTA pairs of gemm_tc2_kernel<NH> that can be resident at once (one CTA
// per SM); 0 if none.  Sets the kernel's shared-memory attribute on first use
// per device.
template <int NH>
cudaError_t pair_capacity(int *pairs) {
    using C = Cfg2<NH>;
    static std::mutex mu;
    static bool attr_set[64] = {};
    static int max_pairs[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(gemm_tc2_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t q = {};
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = 2;
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        q.gridDim = dim3((unsigned)(num_sms() & ~1));
        q.blockDim = dim3(C::THREADS);
        q.dynamicSmemBytes = C::SMEM;
        q.attrs = qa;
        q.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, gemm_tc2_kernel<NH>, &q);
        if (e != cudaSuccess) return e;
        max_pairs[dev] = n < 0 ? 0 : n;
        attr_set[dev] = true;
    }
    *pairs = max_pairs[dev];
    return cudaSuccess;
}

// Pairs a launch may use: the resident capacity, capped by the plan's SM
// limit (two SMs per pair; at least one pair).
int limit_pairs(int cap, int max_sms) {
    if (max_sms > 0 && cap > 0) {
        const int lim = max_sms / 2 > 0 ? max_sms / 2 : 1;
        if (lim < cap) return lim;
    }
    return cap;
}

// Launches the CTA-pair kernel: clusters of two, at most as many pairs as can
// be resident at once (and as the plan's SM limit allows).
template <int NH>
cudaError_t launch_pair(TcK &k, cudaStream_t s, int max_sms) {
    using C = Cfg2<NH>;
    int cap = 0;
    const cudaError_t ce = pair_capacity<NH>(&cap);
    if (ce != cudaSuccess) return ce;
    if (cap < 1) return cudaErrorNotSupported;  // no pair can be resident: the caller falls back
    cap = limit_pairs(cap, max_sms);
    set_tiles(k, 256, 256 * NH);
    const int64_t total = k.total;
    const int npairs = (int)(total < cap ? total : cap);
    if (NH == 2) {
        const int r = tail_halves(total, npairs);
        if (r) {
            k.half_from = (int)(total - r);
            k.total = (int)(total + r);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // A programmatic dependent of the previous kernel in the stream: the
    // prologue (barriers, TMEM, cluster sync) overlaps that kernel's last
    // wave, and a pair GEMM launched next may start its own on the SMs this
    // one frees.  SHMM_PDL=0 launches in plain stream order.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    const char *pdl = getenv("SHMM_PDL");
    cfg.gridDim = dim3((unsigned)(2 * npairs));
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = (pdl && pdl[0] == '0') ? 1 : 2;
    shmm::count_launch();
    return cudaLaunchKernelEx(&cfg, gemm_tc2_kernel<NH>, k);
}

bool pair_kernel_enabled() {
    const char *e = getenv("SHMM_TC_PAIR");
    return !(e && e[0] == '0');
}

// Tile width of the pair kernel for this launch.  256 x 512 tiles (NH = 2)
// move a quarter fewer operand bytes per FLOP; the 256 x 256 kernel's loads
// hold its MMAs back (its tensor pipe alone, fed from stale shared memory,
// runs 1.13x faster; with a quarter of its loads removed, 1.12x).  But a
// wide tile fills TMEM, so each tile boundary idles the tensor pipe while
// the epilogue drains half 0 (half 0 of the next tile then runs ahead over
// the loaded stages while half 1 drains); and wide tiles halve the tile
// count, so a launch of few tiles can lose more to its last partial wave.
// Measured on 8192^2 x K products (same wave counts), wide / narrow time =
// 0.88 (1 + 4 / k-blocks per tile): 0.99 at K = 2048, 0.93 at 4096, 0.91 at
// 16384 (the MLP's GeLU matmul, 64 k-blocks: 0.98 across 27 and 14 waves).
// Pick the smaller estimate: waves x work per tile x that factor, where a
// last wave split into half tiles (tail_halves) counts 0.6.
// SHMM_TC_WIDE=0 / 1 forces 256- / 512-column tiles (tests compare them).
int pair_halves(const TcK &k, int max_sms) {
    bool wide_ok = false;
    for (int i = 0; i < k.nseg; ++i) {
        const TcSeg &g = k.seg[i];
        if (g.fused && !g.accum && g.G > 1) return 1;  // the rank-order fold needs TMEM's second buffer
        if (g.N > 256) wide_ok = true;
    }
    const char *env = getenv("SHMM_TC_WIDE");
    if (env && env[0] == '0') return 1;
    if (env && env[0] == '1') return 2;
    if (!wide_ok) return 1;
    int cap1 = 0, cap2 = 0;
    if (pair_capacity<1>(&cap1) != cudaSuccess || pair_capacity<2>(&cap2) != cudaSuccess || cap1 < 1 || cap2 < 1)
        return 1;
    cap1 = limit_pairs(cap1, max_sms);
    cap2 = limit_pairs(cap2, max_sms);
    int64_t t1 = 0, t2 = 0;
    double kb_sum = 0.0;  // k-blocks over the wide tiles (weights the per-tile estimate)
    for (int i = 0; i < k.nseg; ++i) {
        const TcSeg &g = k.seg[i];
        const int64_t m_t = (g.M + 255) / 256;
        const int64_t w = (int64_t)g.units * m_t * ((g.N + 511) / 512);
        t1 += (int64_t)g.units * m_t * ((g.N + 255) / 256);
        t2 += w;
        kb_sum += (double)w * g.k_blocks * (g.fused && g.accum ? g.G : 1);
    }
    const double kb = t2 > 0 ? kb_sum / (double)t2 : 1.0;  // k-blocks per tile
    const double narrow = (double)((t1 + cap1 - 1) / cap1);
    // a partial last wave split into half tiles takes about 0.6 of a round
    const double rounds2 = (double)(t2 / cap2) + (t2 % cap2 == 0 ? 0.0 : tail_halves(t2, cap2) ? 0.6 : 1.0);
    const double wide = rounds2 * 2.0 * 0.88 * (1.0 + 4.0 / kb);
    return wide < narrow ? 2 : 1;
}

}  // namespace

namespace shmm {

bool tcgen05_supported(const GemmArgs &a) {
    const int G = a.fused ? a.G : 1;
    return a.in_dt == SHMM_BF16 && a.M > 0 && a.N > 0 && a.Kd > 0 && a.Kd % 8 == 0 &&
           a.N % 8 == 0 && G <= kMaxMaps && a.M <= ((int64_t)1 << 31) && a.N <= ((int64_t)1 << 31) &&
           a.Kd <= ((int64_t)1 << 31);
}

int launch_gemm_tcgen05(const GemmArgs *args, int nargs, int *status, void *stream, std::string *msg) {
    EncodeTiledFn fn = encode_fn(msg);
    if (!fn) return (int)cudaErrorNotSupported;
    cudaStream_t s = (cudaStream_t)stream;
    // Chunks of units (at most kMaxMaps operand slots each), grouped by the
    // kernel they need: CTA pairs (local M above one 128-row tile) or single
    // CTAs.  Each launch packs consecutive chunks of one group as segments.
    struct Chunk {
        const GemmArgs *a;
        int u0, nu;
    };
    std::vector<Chunk> groups[2];  // [0] pair kernel, [1] single-CTA kernel
    for (int i = 0; i < nargs; ++i) {
        const GemmArgs &a = args[i];
        const int G = a.fused ? a.G : 1;
        const int a_nb = a.A_src ? a.a_b0 * a.a_b1 : 1;
        const int b_nb = a.B_src ? a.b_b0 * a.b_b1 : 1;
        if (a_nb > kMaxMaps || b_nb > kMaxMaps) {
            if (msg) *msg = "all-gather group larger than one launch's operand maps";
            return (int)cudaErrorInvalidValue;
        }
        const int per_launch = kMaxMaps / G;  // units per launch
        const int grp = (a.M > BM && pair_kernel_enabled()) ? 0 : 1;
        for (int u0 = 0; u0 < a.units; u0 += per_launch)
            groups[grp].push_back({&a, u0, (a.units - u0) < per_launch ? (a.units - u0) : per_launch});
    }
    for (int grp = 0; grp < 2; ++grp) {
        const std::vector<Chunk> &chunks = groups[grp];
        size_t ci = 0;
        while (ci < chunks.size()) {
            TcK k;
            memset(&k, 0, sizeof k);
            // One tensor map per distinct operand buffer (a shard may serve
            // several slots, and plans may share buffers); per slot, a block
            // table.
            const void *ptrs_a[kMaxMaps], *ptrs_b[kMaxMaps];
            int64_t dims_a[kMaxMaps][2], dims_b[kMaxMaps][2];
            int na = 0, nb = 0, slots = 0, outs = 0;
            bool limited = true;  // every segment carries an SM limit
            int max_sms = 0;
            auto map_of = [&](const void *ptr, const void **ptrs, int64_t (*dims)[2], int *n, CUtensorMap *maps,
                              int64_t rows, int64_t cols, uint32_t bx, uint32_t by) -> int {
                for (int j = 0; j < *n; ++j)
                    if (ptrs[j] == ptr && dims[j][0] == rows && dims[j][1] == cols) return j;
                if (*n >= kMaxMaps) return -1;
                if (!cached_map(fn, &maps[*n], ptr, rows, cols, bx, by)) return -2;
                ptrs[*n] = ptr;
                dims[*n][0] = rows;
                dims[*n][1] = cols;
                return (*n)++;
            };
            while (ci < chunks.size() && k.nseg < kMaxSegs) {
                const Chunk &c = chunks[ci];
                const GemmArgs &a = *c.a;
                const int G = a.fused ? a.G : 1;
                const int nout = a.fused ? c.nu * G : c.nu;
                if (slots + c.nu * G > kMaxMaps || outs + nout > kMaxMaps) break;
                const int a_nb = a.A_src ? a.a_b0 * a.a_b1 : 1;
                const int b_nb = a.B_src ? a.b_b0 * a.b_b1 : 1;
                const int64_t a_rows = a.A_src ? a.a_brows : a.M, a_cols = a.A_src ? a.a_bcols : a.Kd;
                const int64_t b_rows = a.B_src ? a.b_brows : a.Kd, b_cols = a.B_src ? a.b_bcols : a.N;
                const int na0 = na, nb0 = nb;
                int m = 0;
                for (int i = 0; i < c.nu * G && m >= 0; ++i) {
                    const int gi = c.u0 * G + i;
                    for (int p = 0; p < a_nb && m >= 0; ++p) {
                        const void *ptr = a.A_src ? a.A_src[(size_t)gi * a_nb + p] : a.A[gi];
                        m = map_of(ptr, ptrs_a, dims_a, &na, k.tmA, a_rows, a_cols, BK, BM);
                        if (m >= 0) k.a_idx[slots + i][p] = (uint8_t)m;
                    }
                    for (int p = 0; p < b_nb && m >= 0; ++p) {
                        const void *ptr = a.B_src ? a.B_src[(size_t)gi * b_nb + p] : a.B[gi];
                        m = map_of(ptr, ptrs_b, dims_b, &nb, k.tmB, b_rows, b_cols, 64, BK);
                        if (m >= 0) k.b_idx[slots + i][p] = (uint8_t)m;
                    }
                }
                if (m == -2) {
                    if (msg) *msg = "cuTensorMapEncodeTiled rejected an operand";
                    return (int)cudaErrorInvalidValue;
                }
                if (m == -1) {  // out of maps: this chunk starts the next launch
                    na = na0;
                    nb = nb0;
                    if (k.nseg == 0) {
                        if (msg) *msg = "more than 16 distinct operand buffers in one chunk";
                        return (int)cudaErrorInvalidValue;
                    }
                    break;
                }
                TcSeg &g = k.seg[k.nseg++];
                g.units = c.nu;
                g.G = G;
                g.mode = a.mode;
                g.fused = a.fused ? 1 : 0;
                g.accum = a.fused && !a.rank_order ? 1 : 0;
                g.gelu = a.gelu ? 1 : 0;
                g.out_f32 = a.out_dt == SHMM_F32 ? 1 : 0;
                g.M = a.M;
                g.N = a.N;
                g.Kd = a.Kd;
                g.k_blocks = (int)((a.Kd + BK - 1) / BK);
                g.slot_base = slots;
                g.out_base = outs;
                g.a_b0 = a.A_src ? a.a_b0 : 1;
                g.a_b1 = a.A_src ? a.a_b1 : 1;
                g.b_b0 = a.B_src ? a.b_b0 : 1;
                g.b_b1 = a.B_src ? a.b_b1 : 1;
                g.a_brows = a_rows;
                g.a_bcols = a_cols;
                g.b_brows = b_rows;
                g.b_bcols = b_cols;
                for (int i = 0; i < nout; ++i) k.out[outs + i] = a.out[(a.fused ? c.u0 * G : c.u0) + i];
                // Output maps for the TMA-store epilogue: each destination block
                // as rows x cols, 32 x 32 boxes.  A reduce-scatter's owner
                // blocks must hold whole 32-row (32-column) boxes, else
                // per-thread stores.
                const bool out_f32 = a.out_dt == SHMM_F32;
                int64_t c_rows = a.M, c_cols = a.N;
                bool tma_store = true;
                if (a.fused && a.mode == 0) {
                    c_rows = a.M / G;
                    tma_store = c_rows % 32 == 0;
                } else if (a.fused && a.mode == 1) {
                    c_cols = a.N / G;
                    tma_store = c_cols % 32 == 0;
                }
                if ((c_cols * (out_f32 ? 4 : 2)) % 16) tma_store = false;
                for (int i = 0; i < nout && tma_store; ++i)
                    tma_store = cached_map(fn, &k.tmC[outs + i], k.out[outs + i], c_rows, c_cols, 32, 32, out_f32,
                                           out_f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
                g.tma_store = tma_store ? 1 : 0;
                g.out_n = c_rows * c_cols;  // an owner's block, or a whole copy
                slots += c.nu * G;
                outs += nout;
                if (a.max_sms <= 0) limited = false;
                else if (a.max_sms > max_sms) max_sms = a.max_sms;
                ++ci;
            }
            k.n_maps_a = na;
            k.n_maps_b = nb;
            k.status = status;
            if (!limited) max_sms = 0;
            // 256-row tiles on CTA pairs unless the local M fits one 128-row tile
            cudaError_t e = cudaErrorNotSupported;
            if (grp == 0)
                e = pair_halves(k, max_sms) == 2 ? launch_pair<2>(k, s, max_sms) : launch_pair<1>(k, s, max_sms);
            if (e == cudaErrorNotSupported) e = launch_bn<256>(k, s, max_sms);  // single CTAs when no pair fits
            if (e != cudaSuccess) return (int)e;
        }
    }
    return 0;
}

}  // namespace shmm
