// Internal declarations shared by the host planner, the C-ABI glue and the
// kernel launchers of libshmm.  Not part of the public interface.
#pragma once

#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cstdint>
#include <string>
#include <vector>

#include "shmm.h"

namespace shmm {

// A value per CUDA device, looked up once with that device current and kept
// for the life of the process.  Host threads may make their first calls on a
// device at the same time: each may look the value up, and every one stores
// the same value, through atomics.  Devices 0 .. kMaxDevices-1 only.
constexpr int kMaxDevices = 64;
template <typename T>
struct PerDevice {
    std::atomic<T> slot[kMaxDevices];
    T get(int dev) const { return slot[dev].load(std::memory_order_acquire); }
    void set(int dev, T v) { slot[dev].store(v, std::memory_order_release); }
};

// Ordered list of mesh axis indices splitting one array dim (first = major).
struct AxisList {
    int n = 0;
    int ax[SHMM_MAX_AXES] = {};
    bool contains(int a) const {
        for (int i = 0; i < n; ++i)
            if (ax[i] == a) return true;
        return false;
    }
    void push(int a) { ax[n++] = a; }
    bool operator==(const AxisList &o) const {
        if (n != o.n) return false;
        for (int i = 0; i < n; ++i)
            if (ax[i] != o.ax[i]) return false;
        return true;
    }
};

struct Spec2 {
    AxisList d[2];
};

// A box: offsets and extents of a rank's block in a global 2-D array.
struct Box {
    int64_t off[2];
    int64_t ext[2];
    int64_t numel() const { return ext[0] * ext[1]; }
};

// Ranks that exchange data in one collective, grouped.  Group g's members
// are members[g*size .. g*size+size) in ascending rank id.
struct Groups {
    int size = 1;
    int count = 0;
    std::vector<int> members;
    // Reduction: owner[g*size + b] = rank owning block b of the scattered dim.
    // Gather: src_at[g*size + p] = rank whose block sits at grid position p
    // (row-major over a blocks0 x blocks1 grid) of the gathered box.
    std::vector<int> by_block;
    int blocks0 = 1, blocks1 = 1;
};

}  // namespace shmm

struct shmm_plan {
    int naxes = 0;
    int size[SHMM_MAX_AXES] = {};
    int nranks = 1;
    int64_t I = 0, J = 0, K = 0;
    shmm_dtype_t in_dt = SHMM_BF16, out_dt = SHMM_BF16, part_dt = SHMM_F32;
    uint32_t flags = 0;
    shmm::Spec2 A, B, C;                      // as given
    shmm::Spec2 A_loc, B_loc, nat, red, out;  // derived
    shmm::AxisList U, gA, gB, gC;             // unreduced / gathered axes
    int case_id = 1;
    int collective = SHMM_COLL_NONE;
    int scatter_dim = -1;
    bool tensor_core = false;
    // Case 2/4 operands are read from their owners' shards by the GEMM's TMA
    // producer (SHMM_FLAG_FUSED, tensor cores, every TMA box inside one shard,
    // at most 16 ranks) instead of being all-gathered into the workspace.
    bool fused_gather = false;
    // Reduction runs in the GEMM epilogue: SHMM_FLAG_FUSED, partial sums to
    // reduce, and (on tensor cores) at most 16 ranks per group, the operand
    // descriptors one launch carries.
    bool fused = false;
    int max_sms = 0;  // SMs the plan's tensor-core GEMM launches may occupy (0: all)
    std::vector<shmm::Box> boxes[7];          // [shmm_tensor_t][rank]
    shmm::Groups red_groups, gA_groups, gB_groups, gC_groups;
};

namespace shmm {

int64_t elem_bytes(shmm_dtype_t t);
// Sets the calling thread's last-error message and returns `st`.
shmm_status_t fail(shmm_status_t st, const std::string &msg);
void clear_error();
// SHMM_INJECT_FAIL="name1,name2": those entry points fail before enqueuing.
bool injected(const char *fn);

// ---- kernel launchers (device code in the .cu files) -------------------

// Partial-sum reduction over groups of `G` ranks.  src[g*G+q]: group g's
// q-th rank in ascending rank order, a rows x cols row-major buffer of
// dtype `pt`.  mode 0 = reduce-scatter along dim 0, 1 = along dim 1, 2 =
// all-reduce.  dst[g*G+b]: owner of block b (RS) or any member (AR), dtype
// `ot`.  Returns a cudaError_t value (0 = success).
struct ReduceArgs {
    int G = 1, ngroups = 0;
    int64_t rows = 0, cols = 0;
    int mode = 2;
    bool tree = false, gelu = false;
    shmm_dtype_t pt = SHMM_F32, ot = SHMM_F32;
    const void *const *src = nullptr;
    void *const *dst = nullptr;
};
int launch_reduce(const ReduceArgs &a, int *status, void *stream);

// All-gather over groups of G ranks: each member's dst buffer (full box,
// blocks0*brows x blocks1*bcols) receives block p from src[g*G+p] (a brows x
// bcols buffer).  dst[g*G+m] for every member m.
struct GatherArgs {
    int G = 1, ngroups = 0;
    int blocks0 = 1, blocks1 = 1;
    int64_t brows = 0, bcols = 0;
    int64_t elem = 2;
    const void *const *src = nullptr;
    void *const *dst = nullptr;
};
int launch_gather(const GatherArgs &a, int *status, void *stream);

// Layer normalisation of rows, fused with an all-gather of row blocks: group
// g's block p (src[g*G+p], brows x cols) is normalised row by row and
// written as rows [p*brows, (p+1)*brows) of every member's gathered buffer
// dst[g*G+m] (G*brows x cols).  G = 1 is plain layer normalisation.
struct LayerNormArgs {
    int G = 1, ngroups = 1;
    int64_t brows = 0, cols = 0;
    shmm_dtype_t dt = SHMM_BF16;
    const float *gamma = nullptr, *beta = nullptr;
    float eps = 1e-5f;
    const void *const *src = nullptr;
    void *const *dst = nullptr;
};
int launch_layernorm_gather(const LayerNormArgs &a, int *status, void *stream);

// Copies rectangles between row-major buffers: rectangle i moves h[i] rows of
// w[i] elements of `elem` bytes from src[i] (row pitch src_ld[i] elements) to
// dst[i] (pitch dst_ld[i]).  The reshard (all-to-all) collective.
// src_room / dst_room: elements from src[i] / dst[i] to the end of their
// buffers (the extents the bounds-checked build compares indices with).
struct CopyRect {
    const void *src;
    void *dst;
    int64_t src_ld, dst_ld, h, w;
    int64_t src_room, dst_room;
};
int launch_copy_rects(const CopyRect *rects, int n, int elem, int *status, void *stream);

// Local GEMMs.  For unit u (a rank, or a reduction group when fused), the
// G operand pairs A[u*G+q] (M x Kd, row-major) and B[u*G+q] (Kd x N,
// row-major) are multiplied.  Unfused (G == 1 per unit): out[u] = A.B.
// Fused: the G products are summed, by default in one fp32 accumulator over
// the group's concatenated K (tensor cores), with rank_order (and always on
// CUDA cores) each formed on its own and added in ascending q order; mode
// 0/1 scatter along dim 0/1 to out[u*G+b], mode 2 writes every out[u*G+b].
struct GemmArgs {
    int units = 0;          // ranks (unfused) or groups (fused)
    int G = 1;              // ranks per unit
    bool fused = false;
    bool rank_order = false;  // fused: per-rank partials added in q order
    int mode = 2;           // fused write mode (0/1 RS dim, 2 AR)
    bool gelu = false;
    int max_sms = 0;        // tensor cores: SMs a launch may occupy (0: all)
    int64_t M = 0, N = 0, Kd = 0;
    shmm_dtype_t in_dt = SHMM_BF16, out_dt = SHMM_F32;
    const void *const *A = nullptr;
    const void *const *B = nullptr;
    void *const *out = nullptr;
    // Operands read in place from the shards of their all-gather group
    // (tensor cores only): the local operand of slot i is a b0 x b1 grid of
    // brows x bcols shards, shard p at A_src[i * b0 * b1 + p] (row-major
    // grid).  NULL: the operand is A[i] (B[i]) itself.
    const void *const *A_src = nullptr;
    int a_b0 = 1, a_b1 = 1;
    int64_t a_brows = 0, a_bcols = 0;
    const void *const *B_src = nullptr;
    int b_b0 = 1, b_b1 = 1;
    int64_t b_brows = 0, b_bcols = 0;
};
int launch_gemm_simt(const GemmArgs &a, int *status, void *stream);
bool tcgen05_supported(const GemmArgs &a);
// Local GEMMs of `n` independent products in as few launches as the
// kernels' tables allow (several products share one persistent tile walk).
// Returns a cudaError_t value; sets *msg on a failure outside CUDA.
int launch_gemm_tcgen05(const GemmArgs *a, int n, int *status, void *stream, std::string *msg);

// Count of kernels enqueued by this library since it was loaded.
void count_launch(int n = 1);

// An NVTX range around the enqueueing of one entry point or phase: a
// profiler (ncu --nvtx, Nsight Systems) files the kernels launched inside it
// under its name.  With no profiler attached, push and pop cost a call each.
class Range {
  public:
    explicit Range(const char *name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range &) = delete;
    Range &operator=(const Range &) = delete;
};

// Device address of the status word that kernels set when a bounded wait
// expires or (bounds-checked build) an index falls outside its buffer, on
// the current device.  Returns a cudaError_t value.
int device_status_ptr(int **ptr);

}  // namespace shmm
