// C-ABI entry points of libshmm that enqueue device work: argument checks,
// workspace carving and dispatch to the kernels.  The plan itself is built
// by planner.cpp.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "device_wait.cuh"
#include "shmm_internal.h"

using shmm::fail;

// Status word written by kernels whose bounded waits expire (0 = fine).
__device__ int g_shmm_status_word;

// Fixed workspace for shmm_run_static_workspace, for callers that cannot
// allocate device memory themselves.  Every device that loads this library
// holds these SHMM_STATIC_WORKSPACE_BYTES until the process exits, and every
// call on a device shares them.
static __device__ __align__(256) unsigned char g_shmm_static_workspace[SHMM_STATIC_WORKSPACE_BYTES];

namespace {

// The current device, or -1 with a message in *err.
int current_device(std::string *err) {
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return -1;
    }
    if (dev < 0 || dev >= shmm::kMaxDevices) {
        *err = "device " + std::to_string(dev) + " is beyond the " + std::to_string(shmm::kMaxDevices) +
               " devices this library supports";
        return -1;
    }
    return dev;
}

// Device address of a __device__ variable on the current device.  Host code
// cannot use the variable's name as a device pointer, so the address is
// looked up once per device (with that device current) and cached; after a
// cudaDeviceReset the cached address is stale, so reset no device while
// this library is in use.
template <typename T>
void *symbol_ptr(shmm::PerDevice<void *> &cache, const T &symbol, std::string *err) {
    const int dev = current_device(err);
    if (dev < 0) return nullptr;
    void *p = cache.get(dev);
    if (p) return p;
    const cudaError_t e = cudaGetSymbolAddress(&p, symbol);
    if (e != cudaSuccess) {
        *err = std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e);
        return nullptr;
    }
    cache.set(dev, p);
    return p;
}

int *status_ptr(std::string *err) {
    static shmm::PerDevice<void *> cache;
    return static_cast<int *>(symbol_ptr(cache, g_shmm_status_word, err));
}

// Address of g_shmm_static_workspace on the current device.
void *static_workspace_ptr(std::string *err) {
    static shmm::PerDevice<void *> cache;
    return symbol_ptr(cache, g_shmm_static_workspace, err);
}

// A wait on an mbarrier that nothing ever arrives at, through the same
// bounded wait the pipelines use: it gives up after `limit` cycles and
// records SHMM_ERR_TIMEOUT.
__global__ void selftest_wait_kernel(int *status, long long limit) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        shmm_dev::mbar_init(shmm_dev::smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        shmm_dev::mbar_wait(shmm_dev::smem_u32(&bar), 0, &abort_flag, status, true, limit);
    }
}

using shmm::injected;

}  // namespace

int shmm::device_status_ptr(int **ptr) {
    std::string err;
    *ptr = status_ptr(&err);
    return *ptr ? 0 : (int)cudaErrorNoDevice;
}

namespace {

shmm_status_t cuda_fail(const char *fn, int e, const std::string &extra = "") {
    std::string m = std::string(fn) + ": " + cudaGetErrorString((cudaError_t)e);
    if (!extra.empty()) m += " (" + extra + ")";
    return fail(SHMM_ERR_CUDA, m);
}

// Per-rank pointer array: non-NULL, 16-byte aligned (NULL allowed for empty
// boxes).
shmm_status_t check_ptrs(const shmm_plan_t *p, const void *const *arr, int tensor, const char *fn,
                         const char *what) {
    if (!arr) return fail(SHMM_ERR_NULL, std::string(fn) + ": " + what + " array is NULL");
    for (int r = 0; r < p->nranks; ++r) {
        if (p->boxes[tensor][r].numel() == 0) continue;
        if (!arr[r])
            return fail(SHMM_ERR_NULL, std::string(fn) + ": " + what + "[" + std::to_string(r) + "] is NULL");
        if (reinterpret_cast<uintptr_t>(arr[r]) % 16)
            return fail(SHMM_ERR_ALIGN, std::string(fn) + ": " + what + "[" + std::to_string(r) +
                                            "] is not 16-byte aligned");
    }
    return SHMM_OK;
}

shmm_status_t check_workspace(const shmm_plan_t *p, const void *workspace, size_t workspace_bytes,
                              const char *fn) {
    size_t need = 0;
    shmm_workspace_size(p, &need);
    if (workspace_bytes < need)
        return fail(SHMM_ERR_NOMEM, std::string(fn) + ": workspace of " + std::to_string(workspace_bytes) +
                                        " bytes, " + std::to_string(need) + " needed");
    if (need && !workspace) return fail(SHMM_ERR_NULL, std::string(fn) + ": workspace is NULL");
    if (need && reinterpret_cast<uintptr_t>(workspace) % 256)
        return fail(SHMM_ERR_ALIGN, std::string(fn) + ": workspace is not 256-byte aligned");
    return SHMM_OK;
}

shmm::GemmArgs gemm_args(const shmm_plan_t *p) {
    shmm::GemmArgs g;
    const shmm::Box &al = p->boxes[SHMM_TENSOR_A_LOCAL][0];
    const shmm::Box &bl = p->boxes[SHMM_TENSOR_B_LOCAL][0];
    g.M = al.ext[0];
    g.Kd = al.ext[1];
    g.N = bl.ext[1];
    g.in_dt = p->in_dt;
    g.max_sms = p->max_sms;
    return g;
}

int run_gemm(const shmm_plan_t *p, const shmm::GemmArgs &g, int *status, void *stream, std::string *msg) {
    if (p->tensor_core && shmm::tcgen05_supported(g)) return shmm::launch_gemm_tcgen05(&g, 1, status, stream, msg);
    if (g.A_src || g.B_src) {  // in-place gathers exist only on the tensor-core path
        *msg = "in-place operand gather needs the tensor-core GEMM";
        return (int)cudaErrorNotSupported;
    }
    return shmm::launch_gemm_simt(g, status, stream);
}

// Unfused local GEMMs of all ranks: out[r] = A[r] . B[r].
int gemm_unfused(const shmm_plan_t *p, const void *const *A, const void *const *B, void *const *out,
                 shmm_dtype_t out_dt, bool gelu, int *status, void *stream, std::string *msg) {
    shmm::GemmArgs g = gemm_args(p);
    g.units = p->nranks;
    g.G = 1;
    g.out_dt = out_dt;
    g.gelu = gelu;
    g.A = A;
    g.B = B;
    g.out = out;
    return run_gemm(p, g, status, stream, msg);
}

// Reduction (standalone) from partial buffers to destinations.
int reduce(const shmm_plan_t *p, const void *const *P, void *const *dst, int mode, int *status,
           void *stream) {
    const shmm::Groups &g = p->red_groups;
    std::vector<const void *> src(g.members.size());
    std::vector<void *> out(g.members.size());
    for (size_t i = 0; i < g.members.size(); ++i) {
        src[i] = P[g.members[i]];
        out[i] = (mode == 2 || p->scatter_dim < 0) ? dst[g.members[i]] : dst[g.by_block[i]];
    }
    shmm::ReduceArgs a;
    a.G = g.size;
    a.ngroups = g.count;
    a.rows = p->boxes[SHMM_TENSOR_P][0].ext[0];
    a.cols = p->boxes[SHMM_TENSOR_P][0].ext[1];
    a.mode = mode;
    a.tree = (p->flags & SHMM_FLAG_TREE) != 0;
    a.gelu = (p->flags & SHMM_FLAG_GELU) != 0;
    a.pt = p->part_dt;
    a.ot = p->out_dt;
    a.src = src.data();
    a.dst = out.data();
    return shmm::launch_reduce(a, status, stream);
}

// GEMM arguments for units [u0, u1) of the local GEMM: ranks when nothing
// is reduced, reduction groups when the reduction is fused.  Operands come
// from A[r], B[r]; results go to dst[r] (a group's owner blocks for a
// reduce-scatter, every member for an all-reduce).  The pointer arrays live
// in `ptrs`; slot_rank[i] is the rank of operand slot i.
struct UnitPtrs {
    std::vector<const void *> a, b;
    std::vector<void *> out;
    std::vector<int> slot_rank;
};
shmm::GemmArgs unit_args(const shmm_plan_t *p, const void *const *A, const void *const *B, void *const *dst,
                         int u0, int u1, UnitPtrs *ptrs) {
    shmm::GemmArgs ga = gemm_args(p);
    ga.out_dt = p->out_dt;
    ga.gelu = (p->flags & SHMM_FLAG_GELU) != 0;
    ptrs->a.clear();
    ptrs->b.clear();
    ptrs->out.clear();
    ptrs->slot_rank.clear();
    if (!p->U.n) {
        ga.units = u1 - u0;
        ga.G = 1;
        for (int r = u0; r < u1; ++r) {
            ptrs->a.push_back(A[r]);
            ptrs->b.push_back(B[r]);
            ptrs->out.push_back(dst[r]);
            ptrs->slot_rank.push_back(r);
        }
    } else {
        const shmm::Groups &g = p->red_groups;
        const bool rs = p->collective == SHMM_COLL_REDUCE_SCATTER;
        for (int i = u0 * g.size; i < u1 * g.size; ++i) {
            const int r = g.members[i];
            ptrs->a.push_back(A[r]);
            ptrs->b.push_back(B[r]);
            ptrs->out.push_back(rs ? dst[g.by_block[i]] : dst[r]);
            ptrs->slot_rank.push_back(r);
        }
        ga.units = u1 - u0;
        ga.G = g.size;
        ga.fused = true;
        ga.rank_order = (p->flags & SHMM_FLAG_RANK_ORDER) != 0;
        ga.mode = rs ? p->scatter_dim : 2;
    }
    ga.A = ptrs->a.data();
    ga.B = ptrs->b.data();
    ga.out = ptrs->out.data();
    return ga;
}

// In-place gather (the plan's fused_gather): per GEMM operand slot (a rank),
// the shard of each block of its all-gather group, in grid order, into
// a_src / b_src, which must outlive the launch.
void attach_gather(const shmm_plan_t *p, const void *const *A_r, const void *const *B_r,
                   const std::vector<int> &slot_rank, shmm::GemmArgs *ga, std::vector<const void *> *a_src,
                   std::vector<const void *> *b_src) {
    if (!p->fused_gather) return;
    auto shard_table = [&](const shmm::Groups &g, const void *const *shards, std::vector<const void *> *out) {
        out->assign(slot_rank.size() * g.size, nullptr);
        for (size_t i = 0; i < slot_rank.size(); ++i) {
            int gi = 0;
            for (size_t j = 0; j < g.members.size(); ++j)
                if (g.members[j] == slot_rank[i]) gi = (int)j / g.size;
            for (int q = 0; q < g.size; ++q) (*out)[i * g.size + q] = shards[g.by_block[gi * g.size + q]];
        }
    };
    if (p->gA.n) {
        shard_table(p->gA_groups, A_r, a_src);
        ga->A_src = a_src->data();
        ga->a_b0 = p->gA_groups.blocks0;
        ga->a_b1 = p->gA_groups.blocks1;
        ga->a_brows = p->boxes[SHMM_TENSOR_A][0].ext[0];
        ga->a_bcols = p->boxes[SHMM_TENSOR_A][0].ext[1];
    }
    if (p->gB.n) {
        shard_table(p->gB_groups, B_r, b_src);
        ga->B_src = b_src->data();
        ga->b_b0 = p->gB_groups.blocks0;
        ga->b_b1 = p->gB_groups.blocks1;
        ga->b_brows = p->boxes[SHMM_TENSOR_B][0].ext[0];
        ga->b_bcols = p->boxes[SHMM_TENSOR_B][0].ext[1];
    }
}

// Streams shmm_run_host copies on, created once per device and kept for the
// life of the process: host-to-device uploads, device-to-device replica
// copies (kept off the upload stream, which the host link limits) and
// device-to-host downloads, each ordered against the others by events.
// Per device, created once: uploads, replica copies, downloads, and a
// second compute stream on which every other stage's GEMM runs.
struct SideStreams {
    cudaStream_t up = nullptr, rep = nullptr, down = nullptr, alt = nullptr;
};
cudaError_t side_streams(SideStreams *out) {
    static std::mutex mu;
    static SideStreams cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev].up) {
        cudaStream_t st[4] = {};
        for (int i = 0; i < 4; ++i) {
            e = cudaStreamCreateWithFlags(&st[i], cudaStreamNonBlocking);
            if (e != cudaSuccess) {
                for (int j = 0; j < i; ++j) cudaStreamDestroy(st[j]);
                return e;
            }
        }
        cache[dev].up = st[0];
        cache[dev].rep = st[1];
        cache[dev].down = st[2];
        cache[dev].alt = st[3];
    }
    *out = cache[dev];
    return cudaSuccess;
}

// Box b of a row-major global host array with `cols` columns <-> a dense
// device buffer holding exactly that box.  Whole rows are one linear copy.
cudaError_t upload_box(void *dev, const void *host, const shmm::Box &b, int64_t cols, int64_t es,
                       cudaStream_t s) {
    const char *src = static_cast<const char *>(host) + (b.off[0] * cols + b.off[1]) * es;
    const size_t w = (size_t)(b.ext[1] * es);
    if (b.ext[1] == cols) return cudaMemcpyAsync(dev, src, w * (size_t)b.ext[0], cudaMemcpyHostToDevice, s);
    return cudaMemcpy2DAsync(dev, w, src, (size_t)(cols * es), w, (size_t)b.ext[0], cudaMemcpyHostToDevice, s);
}
cudaError_t download_box(void *host, const void *dev, const shmm::Box &b, int64_t cols, int64_t es,
                         cudaStream_t s) {
    char *dst = static_cast<char *>(host) + (b.off[0] * cols + b.off[1]) * es;
    const size_t w = (size_t)(b.ext[1] * es);
    if (b.ext[1] == cols) return cudaMemcpyAsync(dst, dev, w * (size_t)b.ext[0], cudaMemcpyDeviceToHost, s);
    return cudaMemcpy2DAsync(dst, (size_t)(cols * es), dev, w, w, (size_t)b.ext[0], cudaMemcpyDeviceToHost, s);
}

int gather(const shmm_plan_t *p, const shmm::Groups &g, int src_tensor, int64_t elem,
           const void *const *shard, void *const *full, int *status, void *stream) {
    std::vector<const void *> src(g.members.size());
    std::vector<void *> dst(g.members.size());
    for (size_t i = 0; i < g.members.size(); ++i) {
        src[i] = shard[g.by_block[i]];
        dst[i] = full[g.members[i]];
    }
    shmm::GatherArgs a;
    a.G = g.size;
    a.ngroups = g.count;
    a.blocks0 = g.blocks0;
    a.blocks1 = g.blocks1;
    a.brows = p->boxes[src_tensor][0].ext[0];
    a.bcols = p->boxes[src_tensor][0].ext[1];
    a.elem = elem;
    a.src = src.data();
    a.dst = dst.data();
    return shmm::launch_gather(a, status, stream);
}

}  // namespace

extern "C" {

shmm_status_t shmm_local_matmul(const shmm_plan_t *p, const void *const *A_r, const void *const *B_r,
                                void *const *P_r, void *stream) {
    static const char *fn = "shmm_local_matmul";
    shmm::clear_error();
    shmm::Range range(fn);
    if (!p) return fail(SHMM_ERR_NULL, std::string(fn) + ": plan is NULL");
    if (injected(fn)) return fail(SHMM_ERR_INJECTED, std::string(fn) + ": injected failure");
    shmm_status_t st;
    if ((st = check_ptrs(p, A_r, SHMM_TENSOR_A_LOCAL, fn, "A_r")) != SHMM_OK) return st;
    if ((st = check_ptrs(p, B_r, SHMM_TENSOR_B_LOCAL, fn, "B_r")) != SHMM_OK) return st;
    if ((st = check_ptrs(p, (const void *const *)P_r, SHMM_TENSOR_P, fn, "P_r")) != SHMM_OK) return st;
    std::string err;
    int *status = status_ptr(&err);
    if (!status) return fail(SHMM_ERR_CUDA, std::string(fn) + ": " + err);
    const bool reduces = p->U.n > 0;
    const shmm_dtype_t odt = reduces ? p->part_dt : p->out_dt;
    const bool gelu = !reduces && (p->flags & SHMM_FLAG_GELU);
    const int e = gemm_unfused(p, A_r, B_r, P_r, odt, gelu, status, stream, &err);
    if (e) return cuda_fail(fn, e, err);
    return SHMM_OK;
}

static shmm_status_t reduce_entry(const char *fn, const shmm_plan_t *p, const void *const *P_r,
                                  void *const *C_r, void *stream, bool all_reduce) {
    shmm::clear_error();
    shmm::Range range(fn);
    if (!p) return fail(SHMM_ERR_NULL, std::string(fn) + ": plan is NULL");
    if (injected(fn)) return fail(SHMM_ERR_INJECTED, std::string(fn) + ": injected failure");
    if (p->U.n == 0)
        return fail(SHMM_ERR_UNSUPPORTED, std::string(fn) + ": the plan has no partial sums to reduce");
    if (p->flags & SHMM_FLAG_TREE && p->red_groups.size > 32)
        return fail(SHMM_ERR_UNSUPPORTED, std::string(fn) + ": tree order supports groups of <= 32 ranks");
    shmm_status_t st;
    if ((st = check_ptrs(p, P_r, SHMM_TENSOR_P, fn, "P_r")) != SHMM_OK) return st;
    int mode = 2;
    int out_tensor = SHMM_TENSOR_P;
    if (!all_reduce) {
        if (p->scatter_dim >= 0) {
            mode = p->scatter_dim;
            out_tensor = SHMM_TENSOR_C_REDUCED;
        } else {
            mode = 0;  // all-reduce plan: rank q of the group takes row block q
            if (p->boxes[SHMM_TENSOR_P][0].ext[0] % p->red_groups.size)
                return fail(SHMM_ERR_SHAPE, std::string(fn) + ": rows do not split over the group");
        }
    }
    if (!C_r) return fail(SHMM_ERR_NULL, std::string(fn) + ": C_r array is NULL");
    for (int r = 0; r < p->nranks; ++r) {
        if (p->boxes[out_tensor][r].numel() == 0) continue;
        if (!C_r[r]) return fail(SHMM_ERR_NULL, std::string(fn) + ": C_r[" + std::to_string(r) + "] is NULL");
        if (reinterpret_cast<uintptr_t>(C_r[r]) % 16)
            return fail(SHMM_ERR_ALIGN, std::string(fn) + ": C_r[" + std::to_string(r) + "] is not 16-byte aligned");
    }
    std::string err;
    int *status = status_ptr(&err);
    if (!status) return fail(SHMM_ERR_CUDA, std::string(fn) + ": " + err);
    // An all-reduce plan reduce-scattered by rows (mode 0, no scatter dim):
    // reduce() gives row block q to the group's q-th member.
    const int e = reduce(p, P_r, C_r, mode, status, stream);
    if (e) return cuda_fail(fn, e);
    return SHMM_OK;
}

shmm_status_t shmm_reduce_scatter(const shmm_plan_t *p, const void *const *P_r, void *const *C_r,
                                  void *stream) {
    return reduce_entry("shmm_reduce_scatter", p, P_r, C_r, stream, false);
}

shmm_status_t shmm_all_reduce(const shmm_plan_t *p, const void *const *P_r, void *const *C_r,
                              void *stream) {
    return reduce_entry("shmm_all_reduce", p, P_r, C_r, stream, true);
}

shmm_status_t shmm_all_gather(const shmm_plan_t *p, int tensor, const void *const *shard_r,
                              void *const *full_r, void *stream) {
    static const char *fn = "shmm_all_gather";
    shmm::clear_error();
    shmm::Range range(fn);
    if (!p) return fail(SHMM_ERR_NULL, std::string(fn) + ": plan is NULL");
    if (injected(fn)) return fail(SHMM_ERR_INJECTED, std::string(fn) + ": injected failure");
    const shmm::Groups *g;
    int src_t, dst_t;
    int64_t elem;
    if (tensor == SHMM_TENSOR_A) {
        g = &p->gA_groups; src_t = SHMM_TENSOR_A; dst_t = SHMM_TENSOR_A_LOCAL;
        elem = shmm::elem_bytes(p->in_dt);
    } else if (tensor == SHMM_TENSOR_B) {
        g = &p->gB_groups; src_t = SHMM_TENSOR_B; dst_t = SHMM_TENSOR_B_LOCAL;
        elem = shmm::elem_bytes(p->in_dt);
    } else if (tensor == SHMM_TENSOR_C) {
        g = &p->gC_groups; src_t = SHMM_TENSOR_C_REDUCED; dst_t = SHMM_TENSOR_C;
        elem = shmm::elem_bytes(p->out_dt);
    } else {
        return fail(SHMM_ERR_UNSUPPORTED, std::string(fn) + ": tensor must be A, B or C");
    }
    if (g->size == 1)
        return fail(SHMM_ERR_UNSUPPORTED, std::string(fn) + ": the plan gathers nothing for this tensor");
    shmm_status_t st;
    if ((st = check_ptrs(p, shard_r, src_t, fn, "shard_r")) != SHMM_OK) return st;
    if ((st = check_ptrs(p, (const void *const *)full_r, dst_t, fn, "full_r")) != SHMM_OK) return st;
    std::string err;
    int *status = status_ptr(&err);
    if (!status) return fail(SHMM_ERR_CUDA, std::string(fn) + ": " + err);
    const int e = gather(p, *g, src_t, elem, shard_r, full_r, status, stream);
    if (e) return cuda_fail(fn, e);
    return SHMM_OK;
}

shmm_status_t shmm_run(const shmm_plan_t *p, const void *const *A_r, const void *const *B_r,
                       void *const *C_r, void *workspace, size_t workspace_bytes, void *stream) {
    static const char *fn = "shmm_run";
    shmm::clear_error();
    shmm::Range range(fn);
    if (!p) return fail(SHMM_ERR_NULL, std::string(fn) + ": plan is NULL");
    if (injected(fn)) return fail(SHMM_ERR_INJECTED, std::string(fn) + ": injected failure");
    shmm_status_t st;
    if ((st = check_ptrs(p, A_r, SHMM_TENSOR_A, fn, "A_r")) != SHMM_OK) return st;
    if ((st = check_ptrs(p, B_r, SHMM_TENSOR_B, fn, "B_r")) != SHMM_OK) return st;
    if ((st = check_ptrs(p, (const void *const *)C_r, SHMM_TENSOR_C, fn, "C_r")) != SHMM_OK) return st;
    if ((st = check_workspace(p, workspace, workspace_bytes, fn)) != SHMM_OK) return st;
    std::string err;
    int *status = status_ptr(&err);
    if (!status) return fail(SHMM_ERR_CUDA, std::string(fn) + ": " + err);

    // Carve the workspace: per-rank 256-byte-aligned slots.
    char *ws = static_cast<char *>(workspace);
    auto carve = [&](int tensor, int64_t elem, std::vector<void *> *slots) {
        const size_t slot = (size_t)((p->boxes[tensor][0].numel() * elem + 255) / 256 * 256);
        slots->resize(p->nranks);
        for (int r = 0; r < p->nranks; ++r) {
            (*slots)[r] = ws;
            ws += slot;
        }
    };
    const int64_t in_b = shmm::elem_bytes(p->in_dt), out_b = shmm::elem_bytes(p->out_dt);
    std::vector<const void *> A_loc(A_r, A_r + p->nranks), B_loc(B_r, B_r + p->nranks);
    std::vector<void *> wa, wb, wp, wc;
    int e = 0;
    if (p->gA.n && !p->fused_gather) {
        shmm::Range phase("gather A");
        carve(SHMM_TENSOR_A_LOCAL, in_b, &wa);
        e = gather(p, p->gA_groups, SHMM_TENSOR_A, in_b, A_r, wa.data(), status, stream);
        if (e) return cuda_fail(fn, e, "gather A");
        for (int r = 0; r < p->nranks; ++r) A_loc[r] = wa[r];
    }
    if (p->gB.n && !p->fused_gather) {
        shmm::Range phase("gather B");
        carve(SHMM_TENSOR_B_LOCAL, in_b, &wb);
        e = gather(p, p->gB_groups, SHMM_TENSOR_B, in_b, B_r, wb.data(), status, stream);
        if (e) return cuda_fail(fn, e, "gather B");
        for (int r = 0; r < p->nranks; ++r) B_loc[r] = wb[r];
    }
    std::vector<const void *> a_src, b_src;
    const bool fused = p->fused;
    if (p->U.n && !fused) carve(SHMM_TENSOR_P, shmm::elem_bytes(p->part_dt), &wp);
    std::vector<void *> dst(C_r, C_r + p->nranks);
    if (p->gC.n) {
        carve(SHMM_TENSOR_C_REDUCED, out_b, &wc);
        dst = wc;
    }
    UnitPtrs up;
    if (!p->U.n) {
        shmm::Range phase("local matmul");
        shmm::GemmArgs ga = unit_args(p, A_loc.data(), B_loc.data(), dst.data(), 0, p->nranks, &up);
        attach_gather(p, A_r, B_r, up.slot_rank, &ga, &a_src, &b_src);
        e = run_gemm(p, ga, status, stream, &err);
        if (e) return cuda_fail(fn, e, err);
    } else if (fused) {
        shmm::Range phase("local matmul + fused reduction");
        shmm::GemmArgs ga = unit_args(p, A_loc.data(), B_loc.data(), dst.data(), 0, p->red_groups.count, &up);
        attach_gather(p, A_r, B_r, up.slot_rank, &ga, &a_src, &b_src);
        e = run_gemm(p, ga, status, stream, &err);
        if (e) return cuda_fail(fn, e, err);
    } else {
        shmm::GemmArgs ga = gemm_args(p);
        ga.units = p->nranks;
        ga.G = 1;
        ga.out_dt = p->part_dt;
        ga.A = A_loc.data();
        ga.B = B_loc.data();
        ga.out = wp.data();
        std::vector<int> by_rank(p->nranks);
        for (int r = 0; r < p->nranks; ++r) by_rank[r] = r;
        attach_gather(p, A_r, B_r, by_rank, &ga, &a_src, &b_src);
        {
            shmm::Range phase("local matmul");
            e = run_gemm(p, ga, status, stream, &err);
        }
        if (e) return cuda_fail(fn, e, err);
        const int mode = p->collective == SHMM_COLL_REDUCE_SCATTER ? p->scatter_dim : 2;
        {
            shmm::Range phase(mode == 2 ? "all-reduce" : "reduce-scatter");
            e = reduce(p, (const void *const *)wp.data(), dst.data(), mode, status, stream);
        }
        if (e) return cuda_fail(fn, e, "reduce");
    }
    if (p->gC.n) {
        shmm::Range phase("gather C");
        e = gather(p, p->gC_groups, SHMM_TENSOR_C_REDUCED, out_b, (const void *const *)wc.data(), C_r,
                   status, stream);
        if (e) return cuda_fail(fn, e, "gather C");
    }
    return SHMM_OK;
}

shmm_status_t shmm_layernorm(int64_t rows, int64_t cols, shmm_dtype_t dtype, const void *x,
                             const float *gamma, const float *beta, float eps, void *y, void *stream) {
    static const char *fn = "shmm_layernorm";
    shmm::clear_error();
    shmm::Range range(fn);
    if (injected(fn)) return fail(SHMM_ERR_INJECTED, std::string(fn) + ": injected failure");
    if (dtype != SHMM_F32 && dtype != SHMM_BF16) return fail(SHMM_ERR_DTYPE, std::string(fn) + ": bad dtype");
    if (rows < 0 || cols < 0) return fail(SHMM_ERR_SHAPE, std::string(fn) + ": negative size");
    if (rows == 0 || cols == 0) return SHMM_OK;
    if (!x || !y || !gamma || !beta) return fail(SHMM_ERR_NULL, std::string(fn) + ": NULL argument");
    if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(y) % 16)
        return fail(SHMM_ERR_ALIGN, std::string(fn) + ": x and y must be 16-byte aligned");
    if (!(eps >= 0.0f)) return fail(SHMM_ERR_SHAPE, std::string(fn) + ": eps must be >= 0");
    shmm::LayerNormArgs a;
    a.G = 1;
    a.ngroups = 1;
    a.brows = rows;
    a.cols = cols;
    a.dt = dtype;
    a.gamma = gamma;
    a.beta = beta;
    a.eps = eps;
    a.src = &x;
    a.dst = &y;
    std::string err;
    int *status = status_ptr(&err);
    if (!status) return fail(SHMM_ERR_CUDA, std::string(fn) + ": " + err);
    const int e = shmm::launch_layernorm_gather(a, status, stream);
    if (e) return cuda_fail(fn, e);
    return SHMM_OK;
}

shmm_status_t shmm_layernorm_all_gather(const shmm_plan_t *p, const void *const *shard_r, const float *gamma,
                                        const float *beta, float eps, void *const *full_r, void *stream) {
    static const char *fn = "shmm_layernorm_all_gather";
    shmm::clear_error();
    shmm::Range range(fn);
    if (!p) return fail(SHMM_ERR_NULL, std::string(fn) + ": plan is NULL");
    if (injected(fn)) return fail(SHMM_ERR_INJECTED, std::string(fn) + ": injected failure");
    const shmm::Groups &g = p->gC_groups;
    if (g.size == 1 || g.blocks1 != 1)
        return fail(SHMM_ERR_UNSUPPORTED, std::string(fn) + ": the plan must all-gather its result along rows");
    if (!gamma || !beta) return fail(SHMM_ERR_NULL, std::string(fn) + ": gamma/beta NULL");
    if (!(eps >= 0.0f)) return fail(SHMM_ERR_SHAPE, std::string(fn) + ": eps must be >= 0");
    shmm_status_t st;
    if ((st = check_ptrs(p, shard_r, SHMM_TENSOR_C_REDUCED, fn, "shard_r")) != SHMM_OK) return st;
    if ((st = check_ptrs(p, (const void *const *)full_r, SHMM_TENSOR_C, fn, "full_r")) != SHMM_OK) return st;
    std::vector<const void *> src(g.members.size());
    std::vector<void *> dst(g.members.size());
    for (size_t i = 0; i < g.members.size(); ++i) {
        src[i] = shard_r[g.by_block[i]];
        dst[i] = full_r[g.members[i]];
    }
    shmm::LayerNormArgs a;
    a.G = g.size;
    a.ngroups = g.count;
    a.brows = p->boxes[SHMM_TENSOR_C_REDUCED][0].ext[0];
    a.cols = p->boxes[SHMM_TENSOR_C_REDUCED][0].ext[1];
    a.dt = p->out_dt;
    a.gamma = gamma;
    a.beta = beta;
    a.eps = eps;
    a.src = src.data();
    a.dst = dst.data();
    std::string err;
    int *status = status_ptr(&err);
    if (!status) return fail(SHMM_ERR_CUDA, std::string(fn) + ": " + err);
    const int e = shmm::launch_layernorm_gather(a, status, stream);
    if (e) return cuda_fail(fn, e);
    return SHMM_OK;
}

shmm_status_t shmm_run_static_workspace(const shmm_plan_t *p, const void *const *A_r,
                                        const void *const *B_r, void *const *C_r, void *stream) {
    static const char *fn = "shmm_run_static_workspace";
    shmm::clear_error();
    shmm::Range range(fn);
    if (!p) return fail(SHMM_ERR_NULL, std::string(fn) + ": plan is NULL");
    if (injected(fn)) return fail(SHMM_ERR_INJECTED, std::string(fn) + ": injected failure");
    size_t need = 0;
    shmm_workspace_size(p, &need);
    if (need > (size_t)SHMM_STATIC_WORKSPACE_BYTES)
        return fail(SHMM_ERR_NOMEM, std::string(fn) + ": the plan needs " + std::to_string(need) +
                                        " bytes of workspace, more than the " +
                                        std::to_string((size_t)SHMM_STATIC_WORKSPACE_BYTES) +
                                        " of the static workspace; use shmm_run with a workspace you allocate");
    void *ws = nullptr;
    if (need) {
        std::string err;
        ws = static_workspace_ptr(&err);
        if (!ws) return fail(SHMM_ERR_CUDA, std::string(fn) + ": " + err);
    }
    return shmm_run(p, A_r, B_r, C_r, ws, need, stream);
}

shmm_status_t shmm_run_batch(int n, const shmm_plan_t *const *plans, const void *const *const *A_r,
                             const void *const *const *B_r, void *const *const *C_r, void *const *workspaces,
                             const size_t *workspace_bytes, void *stream) {
    static const char *fn = "shmm_run_batch";
    shmm::clear_error();
    shmm::Range range(fn);
    if (n < 0) return fail(SHMM_ERR_SHAPE, std::string(fn) + ": n < 0");
    if (n == 0) return SHMM_OK;
    if (!plans || !A_r || !B_r || !C_r) return fail(SHMM_ERR_NULL, std::string(fn) + ": NULL array");
    if (injected(fn)) return fail(SHMM_ERR_INJECTED, std::string(fn) + ": injected failure");
    // Everything is checked before anything is enqueued.
    for (int i = 0; i < n; ++i) {
        const shmm_plan_t *p = plans[i];
        const std::string at = std::string(fn) + " (plan " + std::to_string(i) + ")";
        if (!p) return fail(SHMM_ERR_NULL, at + ": plan is NULL");
        shmm_status_t st;
        if ((st = check_ptrs(p, A_r[i], SHMM_TENSOR_A, at.c_str(), "A_r")) != SHMM_OK) return st;
        if ((st = check_ptrs(p, B_r[i], SHMM_TENSOR_B, at.c_str(), "B_r")) != SHMM_OK) return st;
        if ((st = check_ptrs(p, (const void *const *)C_r[i], SHMM_TENSOR_C, at.c_str(), "C_r")) != SHMM_OK)
            return st;
        if ((st = check_workspace(p, workspaces ? workspaces[i] : nullptr, workspace_bytes ? workspace_bytes[i] : 0,
                                  at.c_str())) != SHMM_OK)
            return st;
    }
    std::string err;
    int *status = status_ptr(&err);
    if (!status) return fail(SHMM_ERR_CUDA, std::string(fn) + ": " + err);
    // A plan whose shmm_run is one tensor-core GEMM launch (operands read in
    // place or whole, a fused reduction or none, the result where the GEMM
    // writes it) joins the shared launch; any other plan runs as shmm_run.
    std::vector<int> joined;
    for (int i = 0; i < n; ++i) {
        const shmm_plan_t *p = plans[i];
        const bool one_launch = p->tensor_core && (!p->gA.n || p->fused_gather) &&
                                (!p->gB.n || p->fused_gather) && (!p->U.n || p->fused) && !p->gC.n &&
                                shmm::tcgen05_supported(gemm_args(p));
        if (one_launch) {
            joined.push_back(i);
            continue;
        }
        const shmm_status_t st = shmm_run(p, A_r[i], B_r[i], C_r[i], workspaces ? workspaces[i] : nullptr,
                                          workspace_bytes ? workspace_bytes[i] : 0, stream);
        if (st != SHMM_OK) return st;
    }
    if (joined.empty()) return SHMM_OK;
    // Per joined plan: its GEMM arguments and the pointer tables they refer
    // to (kept alive until the launch is enqueued).
    std::vector<UnitPtrs> up(joined.size());
    std::vector<std::vector<const void *>> a_src(joined.size()), b_src(joined.size());
    std::vector<shmm::GemmArgs> ga(joined.size());
    for (size_t j = 0; j < joined.size(); ++j) {
        const int i = joined[j];
        const shmm_plan_t *p = plans[i];
        ga[j] = unit_args(p, A_r[i], B_r[i], C_r[i], 0, p->U.n ? p->red_groups.count : p->nranks, &up[j]);
        attach_gather(p, A_r[i], B_r[i], up[j].slot_rank, &ga[j], &a_src[j], &b_src[j]);
    }
    int e;
    {
        shmm::Range phase("local matmuls of the batch");
        e = shmm::launch_gemm_tcgen05(ga.data(), (int)ga.size(), status, stream, &err);
    }
    if (e) return cuda_fail(fn, e, err);
    return SHMM_OK;
}

shmm_status_t shmm_run_host(const shmm_plan_t *p, const void *A_host, const void *B_host, void *C_host,
                            void *const *A_r, void *const *B_r, void *const *C_r, void *workspace,
                            size_t workspace_bytes, void *stream) {
    static const char *fn = "shmm_run_host";
    constexpr int kStages = 16;
    shmm::clear_error();
    shmm::Range range(fn);
    if (!p) return fail(SHMM_ERR_NULL, std::string(fn) + ": plan is NULL");
    if (injected(fn)) return fail(SHMM_ERR_INJECTED, std::string(fn) + ": injected failure");
    shmm_status_t st;
    if ((st = check_ptrs(p, (const void *const *)A_r, SHMM_TENSOR_A, fn, "A_r")) != SHMM_OK) return st;
    if ((st = check_ptrs(p, (const void *const *)B_r, SHMM_TENSOR_B, fn, "B_r")) != SHMM_OK) return st;
    if ((st = check_ptrs(p, (const void *const *)C_r, SHMM_TENSOR_C, fn, "C_r")) != SHMM_OK) return st;
    if ((st = check_workspace(p, workspace, workspace_bytes, fn)) != SHMM_OK) return st;
    std::string err;
    int *status = status_ptr(&err);
    if (!status) return fail(SHMM_ERR_CUDA, std::string(fn) + ": " + err);
    SideStreams ss;
    cudaError_t e = side_streams(&ss);
    if (e != cudaSuccess) return cuda_fail(fn, e, "side streams");

    // Units whose GEMMs read only their own ranks' shards and write only
    // their own ranks' results (no operand or result gather; a reduction
    // only if fused): uploads of later stages overlap earlier stages' GEMMs,
    // and downloads overlap later GEMMs.  Otherwise one stage runs shmm_run.
    // With few units, a unit's stage is further split into blocks of output
    // rows (multiples of the 256-row tile) wherever a block of C rows needs
    // only the same rows of A: no reduction, an all-reduce, or a
    // reduce-scatter over columns.
    const bool staged = !p->gA.n && !p->gB.n && !p->gC.n && (!p->U.n || p->fused);
    const int units = p->U.n ? p->red_groups.count : p->nranks;
    const int64_t M = p->boxes[SHMM_TENSOR_A_LOCAL][0].ext[0];
    const int64_t Kd = p->boxes[SHMM_TENSOR_A_LOCAL][0].ext[1];
    const int64_t c_cols = p->boxes[SHMM_TENSOR_C][0].ext[1];
    // At most one stage per 16 MB of host operands: a stage costs a launch
    // and a few events, ~10-20 us, against ~76 us to upload 16 MB.
    const int64_t in_b = shmm::elem_bytes(p->in_dt), out_b = shmm::elem_bytes(p->out_dt);
    const int64_t host_bytes = ((A_host ? p->I * p->J : 0) + (B_host ? p->J * p->K : 0)) * in_b;
    const int want_stages = (int)std::max<int64_t>(1, std::min<int64_t>(kStages, host_bytes >> 24));
    const bool row_blocks = staged && units < want_stages &&
                            !(p->U.n && p->collective == SHMM_COLL_REDUCE_SCATTER && p->scatter_dim == 0);
    struct Stage {
        int u0, u1;
        bool block;      // a block of rows: [r0, r1) of the units' A and C boxes
        int64_t r0, r1;  // (otherwise whole boxes)
    };
    std::vector<Stage> plan_stages;
    if (!staged) {
        plan_stages.push_back({0, units, false, 0, M});
    } else if (row_blocks) {
        const int64_t want = std::min<int64_t>((want_stages + units - 1) / units, (M + 255) / 256);
        const int64_t rows = ((M + want - 1) / want + 255) / 256 * 256;
        for (int u = 0; u < units; ++u)
            for (int64_t r0 = 0; r0 < M; r0 += rows)
                plan_stages.push_back({u, u + 1, true, r0, std::min(M, r0 + rows)});
    } else {
        const int n = std::min(units, want_stages);
        for (int i = 0; i < n; ++i) plan_stages.push_back({i * units / n, (i + 1) * units / n, false, 0, M});
    }
    cudaStream_t cs = (cudaStream_t)stream;

    std::vector<cudaEvent_t> events;
    auto recorded = [&](cudaStream_t on, cudaEvent_t *ev) -> cudaError_t {
        cudaError_t r = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (r != cudaSuccess) return r;
        events.push_back(*ev);
        return cudaEventRecord(*ev, on);
    };
    auto record = [&](cudaStream_t on, cudaStream_t waiter) -> cudaError_t {
        cudaEvent_t ev;
        const cudaError_t r = recorded(on, &ev);
        return r == cudaSuccess ? cudaStreamWaitEvent(waiter, ev, 0) : r;
    };
    // Every exit joins the side streams back into the caller's stream, so
    // nothing this call enqueued outlives what the caller orders after it.
    auto finish = [&](shmm_status_t result) -> shmm_status_t {
        record(ss.up, cs);
        record(ss.rep, cs);
        record(ss.down, cs);
        record(ss.alt, cs);
        for (cudaEvent_t ev : events) cudaEventDestroy(ev);  // released once complete
        return result;
    };
    if ((e = record(cs, ss.up)) != cudaSuccess || (e = record(cs, ss.rep)) != cudaSuccess ||
        (e = record(cs, ss.down)) != cudaSuccess || (e = record(cs, ss.alt)) != cudaSuccess)
        return finish(cuda_fail(fn, e, "events"));

    // Each distinct shard (A: each row block of it) crosses the host link
    // once; a replica is a device copy of the first rank's upload, on the
    // replica stream after an event that follows the stage's uploads.
    typedef std::pair<std::pair<int64_t, int64_t>, int64_t> Key;  // box offset, first row
    std::map<Key, int> first_a, first_b, done_c;
    struct Replica {
        void *dst;
        const void *src;
        size_t bytes;
    };
    std::vector<Replica> replicas;
    // B crosses the link whole at its first use.  The ranks holding replicas
    // of that box get their device copies right after it, on the replica
    // stream, whatever stage they belong to.  Staged GEMMs read the uploaded
    // box itself (b_read), so they never wait for a replica; one shmm_run
    // over every rank waits for the copies.  (Copying a replica in its own
    // rank's stage held that stage's GEMM behind 0.47 GB of device copies.)
    std::map<std::pair<int64_t, int64_t>, std::vector<int>> b_holders;
    if (B_host)
        for (int r = 0; r < p->nranks; ++r) {
            const shmm::Box &b = p->boxes[SHMM_TENSOR_B][r];
            if (b.numel()) b_holders[std::make_pair(b.off[0], b.off[1])].push_back(r);
        }
    struct EarlyCopy {
        int rank;
        Replica c;
    };
    std::vector<EarlyCopy> early;
    std::vector<cudaEvent_t> b_ready(p->nranks, nullptr);
    std::vector<const void *> b_read(B_r, B_r + p->nranks);  // the B buffer each rank's GEMM reads
    // Rows [r0, r1) of box b, and where they start in its dense buffer.
    auto rows_of = [](const shmm::Box &b, int64_t r0, int64_t r1) {
        shmm::Box s = b;
        s.off[0] += r0;
        s.ext[0] = r1 - r0;
        return s;
    };
    std::vector<char> b_done(p->nranks, 0);
    auto upload = [&](int r, const Stage &stg) -> cudaError_t {
        struct Op {
            const void *host;
            int tensor;
            int64_t cols;
            void *const *dev;
            std::map<Key, int> *first;
            bool whole;  // B: the whole box at its first use
        } ops[2] = {{A_host, SHMM_TENSOR_A, p->J, A_r, &first_a, false},
                    {B_host, SHMM_TENSOR_B, p->K, B_r, &first_b, true}};
        for (const Op &o : ops) {
            const shmm::Box &whole = p->boxes[o.tensor][r];
            if (!o.host || whole.numel() == 0) continue;
            if (o.whole) {
                if (b_done[r]) continue;  // an earlier row block brought it
                b_done[r] = 1;
            }
            const bool part = stg.block && !o.whole;
            const int64_t q0 = part ? stg.r0 : 0, q1 = part ? stg.r1 : whole.ext[0];
            const Key key(std::make_pair(whole.off[0], whole.off[1]), q0);
            const shmm::Box b = rows_of(whole, q0, q1);
            const size_t at = (size_t)(q0 * whole.ext[1] * in_b), bytes = (size_t)(b.numel() * in_b);
            char *dst = static_cast<char *>(o.dev[r]) + at;
            const auto it = o.first->find(key);
            cudaError_t r2;
            if (it == o.first->end()) {
                (*o.first)[key] = r;
                r2 = upload_box(dst, o.host, b, o.cols, in_b, ss.up);
                if (o.whole)
                    for (int h : b_holders[std::make_pair(whole.off[0], whole.off[1])])
                        if (!b_done[h]) {
                            b_done[h] = 1;
                            early.push_back({h, {static_cast<char *>(o.dev[h]) + at, dst, bytes}});
                            b_read[h] = dst;
                        }
            } else {
                replicas.push_back({dst, static_cast<const char *>(o.dev[it->second]) + at, bytes});
                r2 = cudaSuccess;
            }
            if (r2 != cudaSuccess) return r2;
        }
        return cudaSuccess;
    };
    auto download = [&](int r, const Stage &stg) -> cudaError_t {
        const shmm::Box &whole = p->boxes[SHMM_TENSOR_C][r];
        if (!C_host || whole.numel() == 0) return cudaSuccess;
        const int64_t r0 = stg.block ? stg.r0 : 0, r1 = stg.block ? stg.r1 : whole.ext[0];
        const Key key(std::make_pair(whole.off[0], whole.off[1]), r0);
        if (done_c.count(key)) return cudaSuccess;  // a replica: written once
        done_c[key] = r;
        const char *src = static_cast<const char *>(C_r[r]) + (size_t)(r0 * whole.ext[1] * out_b);
        return download_box(C_host, src, rows_of(whole, r0, r1), p->K, out_b, ss.down);
    };

    int si = 0;
    for (const Stage &stg : plan_stages) {
        shmm::Range phase("stage");
        const int u0 = stg.u0, u1 = stg.u1;
        // Consecutive stages' GEMMs alternate between the caller's stream
        // and a second one, so one stage's last partial wave of tiles
        // overlaps the next stage's first.
        cudaStream_t gs = staged && (si++ & 1) ? ss.alt : cs;
        std::vector<int> ranks;
        if (!staged) {
            for (int r = 0; r < p->nranks; ++r) ranks.push_back(r);
        } else if (!p->U.n) {
            for (int r = u0; r < u1; ++r) ranks.push_back(r);
        } else {
            const shmm::Groups &g = p->red_groups;
            for (int i = u0 * g.size; i < u1 * g.size; ++i) ranks.push_back(g.members[i]);
        }
        replicas.clear();
        for (int r : ranks)
            if ((e = upload(r, stg)) != cudaSuccess) return finish(cuda_fail(fn, e, "upload"));
        if ((e = record(ss.up, gs)) != cudaSuccess) return finish(cuda_fail(fn, e, "events"));
        if (!replicas.empty() || !early.empty())
            if ((e = record(ss.up, ss.rep)) != cudaSuccess) return finish(cuda_fail(fn, e, "events"));
        if (!replicas.empty()) {
            for (const Replica &c : replicas)
                if ((e = cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyDeviceToDevice, ss.rep)) != cudaSuccess)
                    return finish(cuda_fail(fn, e, "replica copy"));
            if ((e = record(ss.rep, gs)) != cudaSuccess) return finish(cuda_fail(fn, e, "events"));
        }
        for (const EarlyCopy &c : early) {
            if ((e = cudaMemcpyAsync(c.c.dst, c.c.src, c.c.bytes, cudaMemcpyDeviceToDevice, ss.rep)) != cudaSuccess ||
                (e = recorded(ss.rep, &b_ready[c.rank])) != cudaSuccess)
                return finish(cuda_fail(fn, e, "replica copy"));
        }
        early.clear();
        if (!staged)  // shmm_run reads every rank's own B
            for (int r : ranks)
                if (b_ready[r] && (e = cudaStreamWaitEvent(gs, b_ready[r], 0)) != cudaSuccess)
                    return finish(cuda_fail(fn, e, "events"));
        if (staged) {
            UnitPtrs up;
            shmm::GemmArgs ga = unit_args(p, (const void *const *)A_r, b_read.data(), C_r, u0, u1, &up);
            if (stg.block) {  // a block of rows: the same rows of every slot's A and C
                ga.M = stg.r1 - stg.r0;
                for (auto &a : up.a) a = static_cast<const char *>(a) + stg.r0 * Kd * in_b;
                for (auto &o : up.out) o = static_cast<char *>(o) + stg.r0 * c_cols * out_b;
            }
            const int ge = run_gemm(p, ga, status, gs, &err);
            if (ge) return finish(cuda_fail(fn, ge, err));
        } else {
            st = shmm_run(p, (const void *const *)A_r, (const void *const *)B_r, C_r, workspace,
                          workspace_bytes, stream);
            if (st != SHMM_OK) {
                const std::string m = shmm_last_error();
                return finish(fail(st, std::string(fn) + ": " + m));
            }
        }
        if ((e = record(gs, ss.down)) != cudaSuccess) return finish(cuda_fail(fn, e, "events"));
        for (int r : ranks)
            if ((e = download(r, stg)) != cudaSuccess) return finish(cuda_fail(fn, e, "download"));
    }
    return finish(SHMM_OK);
}

shmm_status_t shmm_selftest_wait_timeout(uint64_t limit_cycles, void *stream) {
    static const char *fn = "shmm_selftest_wait_timeout";
    shmm::clear_error();
    if (limit_cycles < 1000 || limit_cycles > 4000000000ull)
        return fail(SHMM_ERR_SHAPE, std::string(fn) + ": limit must be in [1e3, 4e9] cycles");
    std::string err;
    int *status = status_ptr(&err);
    if (!status) return fail(SHMM_ERR_CUDA, std::string(fn) + ": " + err);
    shmm::count_launch();
    selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status, (long long)limit_cycles);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(fn, e);
    return SHMM_OK;
}

shmm_status_t shmm_sync_status(void *stream) {
    shmm::clear_error();
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail("shmm_sync_status", e);
    std::string err;
    if (!status_ptr(&err)) return fail(SHMM_ERR_CUDA, "shmm_sync_status: " + err);
    int v = 0;
    e = cudaMemcpyFromSymbolAsync(&v, g_shmm_status_word, sizeof v, 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail("shmm_sync_status", e);
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_shmm_status_word, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail("shmm_sync_status", e);
        return fail((shmm_status_t)v, "shmm_sync_status: a kernel reported " +
                                          std::string(shmm_status_string((shmm_status_t)v)));
    }
    return SHMM_OK;
}

}  // extern "C"
