// Host planner of libshmm: mesh and sharding validation, classification into
// the four cases of a sharded matmul, per-rank boxes, reduction and gather
// groups, owners, byte and FLOP counts.  No device code.
//
// Case rules follow "Sharding Matrix Multiply" (Cases 1-4, Summary) and
// "Sharded matmuls and collectives on a torus" (The four cases); the choice
// of collective follows the consumer ownership of "Sharded matrix
// multiplication and result ownership" (The mechanism, steps 1-5).

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "shmm_internal.h"

using shmm::AxisList;
using shmm::Box;
using shmm::Groups;
using shmm::Spec2;

namespace shmm {

static thread_local std::string g_last_error;

shmm_status_t fail(shmm_status_t st, const std::string &msg) {
    g_last_error = msg;
    return st;
}
void clear_error() { g_last_error.clear(); }

bool injected(const char *fn) {
    const char *env = getenv("SHMM_INJECT_FAIL");
    if (!env || !*env) return false;
    const std::string list = std::string(",") + env + ",";
    return list.find(std::string(",") + fn + ",") != std::string::npos;
}

int64_t elem_bytes(shmm_dtype_t t) { return t == SHMM_F32 ? 4 : 2; }

static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

}  // namespace shmm

namespace {

// Rank id -> coordinate on axis `a` (row-major, first axis major).
int coord(const shmm_plan_t &p, int rank, int a) {
    int stride = 1;
    for (int i = p.naxes - 1; i > a; --i) stride *= p.size[i];
    return (rank / stride) % p.size[a];
}

int64_t ways(const shmm_plan_t &p, const AxisList &l) {
    int64_t n = 1;
    for (int i = 0; i < l.n; ++i) n *= p.size[l.ax[i]];
    return n;
}

// Block index of `rank` along a dim split by `l` (first listed axis major).
int64_t block_index(const shmm_plan_t &p, const AxisList &l, int rank) {
    int64_t idx = 0;
    for (int i = 0; i < l.n; ++i) idx = idx * p.size[l.ax[i]] + coord(p, rank, l.ax[i]);
    return idx;
}

Box box_of(const shmm_plan_t &p, const Spec2 &s, int64_t d0, int64_t d1, int rank) {
    Box b;
    const int64_t dims[2] = {d0, d1};
    for (int d = 0; d < 2; ++d) {
        const int64_t n = ways(p, s.d[d]);
        b.ext[d] = dims[d] / n;
        b.off[d] = block_index(p, s.d[d], rank) * b.ext[d];
    }
    return b;
}

bool divides(const shmm_plan_t &p, const Spec2 &s, int64_t d0, int64_t d1) {
    return d0 % ways(p, s.d[0]) == 0 && d1 % ways(p, s.d[1]) == 0;
}

// Converts and validates one public spec: known axes, each axis at most once.
bool read_spec(const shmm_plan_t &p, const shmm_spec_t *in, Spec2 *out, std::string *why) {
    bool used[SHMM_MAX_AXES] = {};
    for (int d = 0; d < 2; ++d) {
        if (in->naxes[d] < 0 || in->naxes[d] > SHMM_MAX_AXES) {
            *why = "axis count out of range";
            return false;
        }
        out->d[d].n = 0;
        for (int i = 0; i < in->naxes[d]; ++i) {
            const int a = in->axes[d][i];
            if (a < 0 || a >= p.naxes) {
                *why = "unknown mesh axis index " + std::to_string(a);
                return false;
            }
            if (used[a]) {
                *why = std::string("mesh axis '") + std::to_string(a) +
                       "' splits more than one dim of the array";
                return false;
            }
            used[a] = true;
            out->d[d].push(a);
        }
    }
    return true;
}

bool is_prefix(const AxisList &pre, const AxisList &l) {
    if (pre.n > l.n) return false;
    for (int i = 0; i < pre.n; ++i)
        if (pre.ax[i] != l.ax[i]) return false;
    return true;
}

// Ranks that agree with every coordinate outside `free` form a group; the
// leader is the member with all `free` coordinates zero.
void make_groups(const shmm_plan_t &p, const AxisList &free, Groups *g) {
    g->size = (int)ways(p, free);
    g->count = p.nranks / g->size;
    g->members.clear();
    for (int r = 0; r < p.nranks; ++r) {
        bool leader = true;
        for (int i = 0; i < free.n; ++i)
            if (coord(p, r, free.ax[i]) != 0) leader = false;
        if (!leader) continue;
        for (int q = 0; q < p.nranks; ++q) {
            bool same = true;
            for (int a = 0; a < p.naxes; ++a)
                if (!free.contains(a) && coord(p, q, a) != coord(p, r, a)) same = false;
            if (same) g->members.push_back(q);  // ascending q
        }
    }
}

// For gather groups: the grid position of each member's source box inside
// the destination box of the group's leader.
void place_blocks(const shmm_plan_t &p, Groups *g, int src_tensor, int dst_tensor) {
    g->by_block.assign(g->members.size(), -1);
    if (g->members.empty()) return;
    const Box &s0 = p.boxes[src_tensor][g->members[0]];
    const Box &d0 = p.boxes[dst_tensor][g->members[0]];
    g->blocks0 = (int)(d0.ext[0] / s0.ext[0]);
    g->blocks1 = (int)(d0.ext[1] / s0.ext[1]);
    for (int gi = 0; gi < g->count; ++gi) {
        const int lead = g->members[gi * g->size];
        const Box &d = p.boxes[dst_tensor][lead];
        for (int m = 0; m < g->size; ++m) {
            const int r = g->members[gi * g->size + m];
            const Box &s = p.boxes[src_tensor][r];
            const int64_t b0 = (s.off[0] - d.off[0]) / s.ext[0];
            const int64_t b1 = (s.off[1] - d.off[1]) / s.ext[1];
            g->by_block[gi * g->size + b0 * g->blocks1 + b1] = r;
        }
    }
}

}  // namespace

extern "C" {

shmm_status_t shmm_plan(const shmm_mesh_t *mesh, const shmm_spec_t *spec_A,
                        const shmm_spec_t *spec_B, const shmm_spec_t *spec_C, int64_t I,
                        int64_t J, int64_t K, shmm_dtype_t in_dtype, shmm_dtype_t out_dtype,
                        uint32_t flags, shmm_plan_t **plan_out) {
    using shmm::fail;
    shmm::clear_error();
    if (!mesh || !spec_A || !spec_B || !spec_C || !plan_out)
        return fail(SHMM_ERR_NULL, "shmm_plan: NULL argument");
    *plan_out = nullptr;
    if (mesh->naxes < 0 || mesh->naxes > SHMM_MAX_AXES)
        return fail(SHMM_ERR_SHAPE, "shmm_plan: mesh axis count out of range");
    if (in_dtype != SHMM_F32 && in_dtype != SHMM_BF16)
        return fail(SHMM_ERR_DTYPE, "shmm_plan: input dtype must be F32 or BF16");
    if (out_dtype != SHMM_F32 && out_dtype != SHMM_BF16)
        return fail(SHMM_ERR_DTYPE, "shmm_plan: output dtype must be F32 or BF16");
    if (I < 0 || J < 0 || K < 0)
        return fail(SHMM_ERR_SHAPE, "shmm_plan: negative size");
    const int64_t lim = (int64_t)1 << 40;
    if (I > lim || J > lim || K > lim || (I && K && I > ((int64_t)1 << 62) / 4 / K) ||
        (I && J && I > ((int64_t)1 << 62) / 4 / J) || (J && K && J > ((int64_t)1 << 62) / 4 / K))
        return fail(SHMM_ERR_SHAPE, "shmm_plan: array larger than 2^62 bytes");

    shmm_plan_t *p = new (std::nothrow) shmm_plan_t();
    if (!p) return fail(SHMM_ERR_NOMEM, "shmm_plan: out of host memory");
    struct Guard {
        shmm_plan_t *owned;
        ~Guard() { delete owned; }
    } guard{p};

    p->naxes = mesh->naxes;
    int64_t n = 1;
    for (int a = 0; a < mesh->naxes; ++a) {
        if (mesh->size[a] < 1) return fail(SHMM_ERR_SHAPE, "shmm_plan: mesh axis size < 1");
        p->size[a] = mesh->size[a];
        n *= mesh->size[a];
        if (n > SHMM_MAX_RANKS)
            return fail(SHMM_ERR_SHAPE, "shmm_plan: more than SHMM_MAX_RANKS ranks");
        for (int b = 0; b < a; ++b)
            if (strncmp(mesh->name[a], mesh->name[b], SHMM_AXIS_NAME_LEN) == 0)
                return fail(SHMM_ERR_INVALID_SPEC, "shmm_plan: duplicate mesh axis name");
    }
    p->nranks = (int)n;
    p->I = I;
    p->J = J;
    p->K = K;
    p->in_dt = in_dtype;
    p->out_dt = out_dtype;
    p->flags = flags;
    p->part_dt = (flags & SHMM_FLAG_PARTIAL_OUT_DTYPE) ? out_dtype : SHMM_F32;

    std::string why;
    if (!read_spec(*p, spec_A, &p->A, &why)) return fail(SHMM_ERR_INVALID_SPEC, "A: " + why);
    if (!read_spec(*p, spec_B, &p->B, &why)) return fail(SHMM_ERR_INVALID_SPEC, "B: " + why);
    if (!read_spec(*p, spec_C, &p->C, &why)) return fail(SHMM_ERR_ILLEGAL_OUTPUT, "C: " + why);

    // Case classification.
    const AxisList &aI = p->A.d[0], &aJ = p->A.d[1], &bJ = p->B.d[0], &bK = p->B.d[1];
    p->A_loc = p->A;
    p->B_loc = p->B;
    if (aJ.n > 0 && aJ == bJ) {
        p->case_id = 3;  // partial sums C{U}
        p->U = aJ;
    } else if (aJ.n > 0 || bJ.n > 0) {
        p->case_id = 2;  // all-gather the J-sharded operand(s) along J
        p->gA = aJ;
        p->gB = bJ;
        p->A_loc.d[1].n = 0;
        p->B_loc.d[0].n = 0;
    } else {
        p->case_id = 1;
    }
    bool shared = false;
    for (int i = 0; i < aI.n; ++i)
        if (bK.contains(aI.ax[i])) shared = true;
    if (shared) {  // only diagonal blocks would exist: gather B along K
        if (p->case_id == 1) p->case_id = 4;
        for (int i = 0; i < bK.n; ++i) p->gB.push(bK.ax[i]);
        p->B_loc.d[1].n = 0;
    }
    p->nat.d[0] = p->A_loc.d[0];
    p->nat.d[1] = p->B_loc.d[1];

    // Collective required by the consumer's ownership.
    const AxisList &cI = p->C.d[0], &cK = p->C.d[1];
    p->red = p->nat;
    if (p->U.n > 0) {
        bool inI = false, inK = false;
        for (int i = 0; i < p->U.n; ++i) {
            inI |= cI.contains(p->U.ax[i]);
            inK |= cK.contains(p->U.ax[i]);
        }
        if (inI && inK)
            return fail(SHMM_ERR_INVALID_SPEC, "C: reduced axes may scatter over one dim only");
        if (inI || inK) {
            const int d = inI ? 0 : 1;
            for (int i = 0; i < p->U.n; ++i) p->red.d[d].push(p->U.ax[i]);
            p->collective = SHMM_COLL_REDUCE_SCATTER;
            p->scatter_dim = d;
        } else {
            p->collective = SHMM_COLL_ALL_REDUCE;
        }
    }
    for (int d = 0; d < 2; ++d) {
        if (!is_prefix(p->C.d[d], p->red.d[d]))
            return fail(SHMM_ERR_INVALID_SPEC,
                        "C: requested ownership is not reachable by reduction and all-gather");
        for (int i = p->C.d[d].n; i < p->red.d[d].n; ++i) p->gC.push(p->red.d[d].ax[i]);
    }
    p->out = p->C;

    // Every split must be even.
    if (!divides(*p, p->A, I, J) || !divides(*p, p->B, J, K) || !divides(*p, p->red, I, K) ||
        !divides(*p, p->out, I, K))
        return fail(SHMM_ERR_SHAPE, "shmm_plan: a dim does not split evenly over its axes");

    // Per-rank boxes.
    const Spec2 *specs[7] = {&p->A, &p->B, &p->out, &p->nat, &p->A_loc, &p->B_loc, &p->red};
    const int64_t dims[7][2] = {{I, J}, {J, K}, {I, K}, {I, K}, {I, J}, {J, K}, {I, K}};
    for (int t = 0; t < 7; ++t) {
        p->boxes[t].resize(p->nranks);
        for (int r = 0; r < p->nranks; ++r)
            p->boxes[t][r] = box_of(*p, *specs[t], dims[t][0], dims[t][1], r);
    }

    // Reduction groups and owners.
    make_groups(*p, p->U, &p->red_groups);
    {
        Groups &g = p->red_groups;
        g.by_block.assign(g.members.size(), -1);
        for (int gi = 0; gi < g.count; ++gi)
            for (int m = 0; m < g.size; ++m) {
                const int r = g.members[gi * g.size + m];
                int b = 0;
                if (p->scatter_dim >= 0) {
                    const Box &nb = p->boxes[SHMM_TENSOR_P][r];
                    const Box &rb = p->boxes[SHMM_TENSOR_C_REDUCED][r];
                    const int d = p->scatter_dim;
                    b = (int)((rb.off[d] - nb.off[d]) / rb.ext[d]);
                } else {
                    b = m;
                }
                g.by_block[gi * g.size + b] = r;
            }
    }
    make_groups(*p, p->gA, &p->gA_groups);
    place_blocks(*p, &p->gA_groups, SHMM_TENSOR_A, SHMM_TENSOR_A_LOCAL);
    make_groups(*p, p->gB, &p->gB_groups);
    place_blocks(*p, &p->gB_groups, SHMM_TENSOR_B, SHMM_TENSOR_B_LOCAL);
    make_groups(*p, p->gC, &p->gC_groups);
    place_blocks(*p, &p->gC_groups, SHMM_TENSOR_C_REDUCED, SHMM_TENSOR_C);

    // Engine of the local GEMM.
    const Box &al = p->boxes[SHMM_TENSOR_A_LOCAL][0];
    const Box &bl = p->boxes[SHMM_TENSOR_B_LOCAL][0];
    p->tensor_core = in_dtype == SHMM_BF16 && !(flags & SHMM_FLAG_SIMT) && al.ext[0] > 0 &&
                     al.ext[1] > 0 && bl.ext[1] > 0 && al.ext[1] % 8 == 0 && bl.ext[1] % 8 == 0;

    p->fused = p->U.n > 0 && (flags & SHMM_FLAG_FUSED) &&
               (!p->tensor_core || p->red_groups.size <= 16);
    // The operand all-gathers fuse into the GEMM's loads when every TMA box
    // (64 columns, 64 or 128 rows) lies inside one shard.
    {
        const Box &a = p->boxes[SHMM_TENSOR_A][0], &b = p->boxes[SHMM_TENSOR_B][0];
        const Groups &ga = p->gA_groups, &gb = p->gB_groups;
        const bool a_ok = (ga.blocks1 == 1 || a.ext[1] % 64 == 0) && (ga.blocks0 == 1 || a.ext[0] % 128 == 0) &&
                          a.ext[1] % 8 == 0;
        const bool b_ok = (gb.blocks0 == 1 || b.ext[0] % 64 == 0) && (gb.blocks1 == 1 || b.ext[1] % 64 == 0) &&
                          b.ext[1] % 8 == 0;
        p->fused_gather = (flags & SHMM_FLAG_FUSED) && p->tensor_core && (p->gA.n || p->gB.n) &&
                          p->nranks <= 16 && (p->gA.n == 0 || a_ok) && (p->gB.n == 0 || b_ok) &&
                          a.numel() > 0 && b.numel() > 0;
    }

    guard.owned = nullptr;
    *plan_out = p;
    return SHMM_OK;
}

shmm_status_t shmm_plan_destroy(shmm_plan_t *plan) {
    delete plan;
    return SHMM_OK;
}

shmm_status_t shmm_plan_set_sm_limit(shmm_plan_t *plan, int max_sms) {
    shmm::clear_error();
    if (!plan) return shmm::fail(SHMM_ERR_NULL, "shmm_plan_set_sm_limit: plan is NULL");
    if (max_sms < 0) return shmm::fail(SHMM_ERR_SHAPE, "shmm_plan_set_sm_limit: max_sms < 0");
    plan->max_sms = max_sms;
    return SHMM_OK;
}

shmm_status_t shmm_workspace_size(const shmm_plan_t *p, size_t *bytes) {
    if (!p || !bytes) return shmm::fail(SHMM_ERR_NULL, "shmm_workspace_size: NULL argument");
    auto slot = [](int64_t b) { return (size_t)((b + 255) / 256 * 256); };
    size_t ws = 0;
    const int64_t in_b = shmm::elem_bytes(p->in_dt), out_b = shmm::elem_bytes(p->out_dt);
    if (p->gA.n && !p->fused_gather) ws += p->nranks * slot(p->boxes[SHMM_TENSOR_A_LOCAL][0].numel() * in_b);
    if (p->gB.n && !p->fused_gather) ws += p->nranks * slot(p->boxes[SHMM_TENSOR_B_LOCAL][0].numel() * in_b);
    if (p->U.n && !p->fused)
        ws += p->nranks *
              slot(p->boxes[SHMM_TENSOR_P][0].numel() * shmm::elem_bytes(p->part_dt));
    if (p->gC.n) ws += p->nranks * slot(p->boxes[SHMM_TENSOR_C_REDUCED][0].numel() * out_b);
    *bytes = ws;
    return SHMM_OK;
}

shmm_status_t shmm_plan_query(const shmm_plan_t *p, shmm_plan_info_t *info) {
    if (!p || !info) return shmm::fail(SHMM_ERR_NULL, "shmm_plan_query: NULL argument");
    memset(info, 0, sizeof *info);
    info->case_id = p->case_id;
    info->collective = p->collective;
    info->scatter_dim = p->scatter_dim;
    info->nranks = p->nranks;
    info->group_size = p->red_groups.size;
    info->ngroups = p->red_groups.count;
    info->gather_A_size = p->gA_groups.size;
    info->gather_B_size = p->gB_groups.size;
    info->gather_C_size = p->gC_groups.size;
    info->in_dtype = p->in_dt;
    info->out_dtype = p->out_dt;
    info->partial_dtype = p->part_dt;
    info->flags = p->flags;
    info->tensor_core = p->tensor_core ? 1 : 0;
    info->fused = p->fused ? 1 : 0;
    info->fused_gather = p->fused_gather ? 1 : 0;
    const Box &al = p->boxes[SHMM_TENSOR_A_LOCAL][0];
    const Box &bl = p->boxes[SHMM_TENSOR_B_LOCAL][0];
    info->local_I = al.ext[0];
    info->local_J = al.ext[1];
    info->local_K = bl.ext[1];
    info->flops_per_rank = 2 * al.ext[0] * al.ext[1] * bl.ext[1];
    // Payload counted once at the sender: (G-1) blocks of V/G per rank.
    const int64_t in_b = shmm::elem_bytes(p->in_dt), out_b = shmm::elem_bytes(p->out_dt);
    const int64_t gA = p->gA_groups.size, gB = p->gB_groups.size, gC = p->gC_groups.size;
    info->payload_operand_ag = (gA - 1) * p->boxes[SHMM_TENSOR_A][0].numel() * in_b +
                               (gB - 1) * p->boxes[SHMM_TENSOR_B][0].numel() * in_b;
    const int64_t G = p->red_groups.size;
    const int64_t V = p->boxes[SHMM_TENSOR_P][0].numel();
    info->payload_reduce_scatter = G > 1 ? (G - 1) * (V / G) * shmm::elem_bytes(p->part_dt) : 0;
    info->payload_result_ag = (gC - 1) * p->boxes[SHMM_TENSOR_C_REDUCED][0].numel() * out_b;
    if (p->collective == SHMM_COLL_ALL_REDUCE) info->payload_result_ag += (G - 1) * (V / G) * out_b;
    shmm_workspace_size(p, &info->workspace_bytes);
    return SHMM_OK;
}

shmm_status_t shmm_plan_rank_box(const shmm_plan_t *p, int tensor, int rank, int64_t off[2],
                                 int64_t ext[2]) {
    if (!p || !off || !ext) return shmm::fail(SHMM_ERR_NULL, "shmm_plan_rank_box: NULL argument");
    if (tensor < 0 || tensor > SHMM_TENSOR_C_REDUCED)
        return shmm::fail(SHMM_ERR_UNSUPPORTED, "shmm_plan_rank_box: unknown tensor");
    if (rank < 0 || rank >= p->nranks)
        return shmm::fail(SHMM_ERR_SHAPE, "shmm_plan_rank_box: rank out of range");
    const Box &b = p->boxes[tensor][rank];
    off[0] = b.off[0];
    off[1] = b.off[1];
    ext[0] = b.ext[0];
    ext[1] = b.ext[1];
    return SHMM_OK;
}

shmm_status_t shmm_plan_group(const shmm_plan_t *p, int rank, int *ranks) {
    if (!p || !ranks) return shmm::fail(SHMM_ERR_NULL, "shmm_plan_group: NULL argument");
    if (rank < 0 || rank >= p->nranks)
        return shmm::fail(SHMM_ERR_SHAPE, "shmm_plan_group: rank out of range");
    const shmm::Groups &g = p->red_groups;
    for (int gi = 0; gi < g.count; ++gi)
        for (int m = 0; m < g.size; ++m)
            if (g.members[gi * g.size + m] == rank) {
                for (int q = 0; q < g.size; ++q) ranks[q] = g.members[gi * g.size + q];
                return SHMM_OK;
            }
    return shmm::fail(SHMM_ERR_SHAPE, "shmm_plan_group: rank in no group");
}

shmm_status_t shmm_reshard(const shmm_mesh_t *mesh, const shmm_spec_t *spec_from,
                           const shmm_spec_t *spec_to, int64_t rows, int64_t cols, shmm_dtype_t dtype,
                           const void *const *src_r, void *const *dst_r, void *stream) {
    using shmm::fail;
    shmm::clear_error();
    shmm::Range range("shmm_reshard");
    static const char *fn = "shmm_reshard: ";
    if (!mesh || !spec_from || !spec_to || !src_r || !dst_r) return fail(SHMM_ERR_NULL, std::string(fn) + "NULL argument");
    if (dtype != SHMM_F32 && dtype != SHMM_BF16) return fail(SHMM_ERR_DTYPE, std::string(fn) + "dtype must be F32 or BF16");
    if (rows < 0 || cols < 0 || rows > ((int64_t)1 << 40) || cols > ((int64_t)1 << 40))
        return fail(SHMM_ERR_SHAPE, std::string(fn) + "bad array shape");
    if (mesh->naxes < 0 || mesh->naxes > SHMM_MAX_AXES) return fail(SHMM_ERR_SHAPE, std::string(fn) + "bad mesh");
    shmm_plan_t p;
    p.naxes = mesh->naxes;
    int64_t n = 1;
    for (int a = 0; a < mesh->naxes; ++a) {
        if (mesh->size[a] < 1) return fail(SHMM_ERR_SHAPE, std::string(fn) + "mesh axis size < 1");
        p.size[a] = mesh->size[a];
        n *= mesh->size[a];
        if (n > SHMM_MAX_RANKS) return fail(SHMM_ERR_SHAPE, std::string(fn) + "more than SHMM_MAX_RANKS ranks");
    }
    p.nranks = (int)n;
    Spec2 from, to;
    std::string why;
    if (!read_spec(p, spec_from, &from, &why)) return fail(SHMM_ERR_INVALID_SPEC, std::string(fn) + "from: " + why);
    if (!read_spec(p, spec_to, &to, &why)) return fail(SHMM_ERR_INVALID_SPEC, std::string(fn) + "to: " + why);
    if (!divides(p, from, rows, cols) || !divides(p, to, rows, cols))
        return fail(SHMM_ERR_SHAPE, std::string(fn) + "a dim does not split evenly over its axes");
    const int64_t nb0 = ways(p, from.d[0]), nb1 = ways(p, from.d[1]);
    const int64_t bh = rows / nb0, bw = cols / nb1;
    const int64_t eb = shmm::elem_bytes(dtype);
    for (int r = 0; r < p.nranks; ++r) {
        const Box sb = box_of(p, from, rows, cols, r), db = box_of(p, to, rows, cols, r);
        if (sb.numel() && (!src_r[r] || reinterpret_cast<uintptr_t>(src_r[r]) % 16))
            return fail(src_r[r] ? SHMM_ERR_ALIGN : SHMM_ERR_NULL, std::string(fn) + "src_r[" + std::to_string(r) + "]");
        if (db.numel() && (!dst_r[r] || reinterpret_cast<uintptr_t>(dst_r[r]) % 16))
            return fail(dst_r[r] ? SHMM_ERR_ALIGN : SHMM_ERR_NULL, std::string(fn) + "dst_r[" + std::to_string(r) + "]");
    }
    if (rows == 0 || cols == 0) return SHMM_OK;
    // The source sharding cuts the array into nb0 x nb1 blocks; destination
    // box D of rank r is covered by the blocks it overlaps.  Each overlap is
    // read from the block's holder that shares r's coordinates on every axis
    // the source sharding leaves replicated.
    std::vector<shmm::CopyRect> rects;
    for (int r = 0; r < p.nranks; ++r) {
        const Box D = box_of(p, to, rows, cols, r);
        if (D.numel() == 0) continue;
        for (int64_t i = D.off[0] / bh; i * bh < D.off[0] + D.ext[0]; ++i)
            for (int64_t j = D.off[1] / bw; j * bw < D.off[1] + D.ext[1]; ++j) {
                int c[SHMM_MAX_AXES];
                for (int a = 0; a < p.naxes; ++a) c[a] = coord(p, r, a);
                int64_t q = i;
                for (int t = from.d[0].n - 1; t >= 0; --t) {  // first listed axis major
                    const int a = from.d[0].ax[t];
                    c[a] = (int)(q % p.size[a]);
                    q /= p.size[a];
                }
                q = j;
                for (int t = from.d[1].n - 1; t >= 0; --t) {
                    const int a = from.d[1].ax[t];
                    c[a] = (int)(q % p.size[a]);
                    q /= p.size[a];
                }
                int s = 0;
                for (int a = 0; a < p.naxes; ++a) s = s * p.size[a] + c[a];
                const int64_t r0 = std::max(D.off[0], i * bh), r1 = std::min(D.off[0] + D.ext[0], (i + 1) * bh);
                const int64_t c0 = std::max(D.off[1], j * bw), c1 = std::min(D.off[1] + D.ext[1], (j + 1) * bw);
                shmm::CopyRect cr;
                const int64_t so = (r0 - i * bh) * bw + (c0 - j * bw);
                const int64_t dof = (r0 - D.off[0]) * D.ext[1] + (c0 - D.off[1]);
                cr.src = static_cast<const char *>(src_r[s]) + so * eb;
                cr.dst = static_cast<char *>(dst_r[r]) + dof * eb;
                cr.src_room = bh * bw - so;
                cr.dst_room = D.numel() - dof;
                cr.src_ld = bw;
                cr.dst_ld = D.ext[1];
                cr.h = r1 - r0;
                cr.w = c1 - c0;
                rects.push_back(cr);
            }
    }
    if (shmm::injected("shmm_reshard")) return fail(SHMM_ERR_INJECTED, std::string(fn) + "injected failure");
    int *status = nullptr;
    if (const int se = shmm::device_status_ptr(&status))
        return fail(SHMM_ERR_CUDA, std::string(fn) + "device status word (" + std::to_string(se) + ")");
    const int e = shmm::launch_copy_rects(rects.data(), (int)rects.size(), (int)eb, status, stream);
    if (e) return fail(SHMM_ERR_CUDA, std::string(fn) + "kernel launch failed (" + std::to_string(e) + ")");
    return SHMM_OK;
}

shmm_status_t shmm_choose_operand(int64_t B, int64_t D, int64_t F, int axis_size, int elem_bytes,
                                  const shmm_device_model_t *dev, shmm_operand_choice_t *out) {
    shmm::clear_error();
    if (!dev || !out) return shmm::fail(SHMM_ERR_NULL, "shmm_choose_operand: NULL argument");
    if (B <= 0 || D <= 0 || F <= 0 || axis_size < 1 || elem_bytes <= 0 || !(dev->flops_per_s > 0) ||
        !(dev->bytes_per_s > 0))
        return shmm::fail(SHMM_ERR_SHAPE, "shmm_choose_operand: sizes and rates must be positive");
    const double C = dev->flops_per_s, W = dev->bytes_per_s, e = (double)elem_bytes;
    const double b = (double)B, d = (double)D, f = (double)F, n = (double)axis_size;
    const double flops = 2.0 * b * d * f;
    // strategy 1: all-gather the weight (V = e*D*F, time V/W), whole product
    out->bytes_gather = e * d * f;
    const double comm1 = out->bytes_gather / W, comp1 = flops / C;
    // strategy 2: all-reduce the [B,F] partials (2V/W with V = e*B*F), 1/n of it
    out->bytes_reduce = 2.0 * e * b * f;
    const double comm2 = out->bytes_reduce / W, comp2 = flops / (n * C);
    out->t_gather = comm1 > comp1 ? comm1 : comp1;
    out->t_reduce = comm2 > comp2 ? comm2 : comp2;
    out->gather_compute_bound = comp1 > comm1 ? 1 : 0;
    out->choice = out->t_reduce < out->t_gather ? 2 : 1;
    return SHMM_OK;
}

const char *shmm_status_string(shmm_status_t s) {
    switch (s) {
        case SHMM_OK: return "SHMM_OK";
        case SHMM_ERR_INVALID_SPEC: return "SHMM_ERR_INVALID_SPEC";
        case SHMM_ERR_ILLEGAL_OUTPUT: return "SHMM_ERR_ILLEGAL_OUTPUT";
        case SHMM_ERR_SHAPE: return "SHMM_ERR_SHAPE";
        case SHMM_ERR_DTYPE: return "SHMM_ERR_DTYPE";
        case SHMM_ERR_NULL: return "SHMM_ERR_NULL";
        case SHMM_ERR_ALIGN: return "SHMM_ERR_ALIGN";
        case SHMM_ERR_CUDA: return "SHMM_ERR_CUDA";
        case SHMM_ERR_TIMEOUT: return "SHMM_ERR_TIMEOUT";
        case SHMM_ERR_NOMEM: return "SHMM_ERR_NOMEM";
        case SHMM_ERR_UNSUPPORTED: return "SHMM_ERR_UNSUPPORTED";
        case SHMM_ERR_INJECTED: return "SHMM_ERR_INJECTED";
        case SHMM_ERR_BOUNDS: return "SHMM_ERR_BOUNDS";
    }
    return "SHMM_ERR_UNKNOWN";
}

const char *shmm_last_error(void) { return shmm::g_last_error.c_str(); }

int shmm_version(void) { return 100; }

#ifdef SHMM_CHECKED
int shmm_bounds_checked(void) { return 1; }
#else
int shmm_bounds_checked(void) { return 0; }
#endif

uint64_t shmm_kernel_launches(void) { return shmm::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
