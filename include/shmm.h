/*
 * shmm.h -- C-ABI of libshmm: the sharded matmul A[I,J] . B[J,K] -> C[I,K]
 * with partial-sum reduction, for virtual ranks held on one GPU.
 *
 * The operation.  A mesh is a grid of ranks with named axes, e.g. {X:4,Y:2}
 * for 8 ranks; a sharding says which mesh axes split which array dims
 * ("Sharded matmuls and collectives on a torus", Notation).  A sharded matmul
 * is a local GEMM per rank plus the collectives the sharding implies
 * ("Sharding Matrix Multiply", Cases 1-4 and Summary):
 *   case 1  no operand sharded on J: local GEMM only;
 *   case 2  one operand sharded on J: all-gather it along J, then GEMM;
 *   case 3  both sharded on J along the same axes: each rank's GEMM yields a
 *           partial sum C{U}; a reduce-scatter (disjoint output shards) or an
 *           all-reduce (replicated output) finishes it;
 *   case 4  a mesh axis shards both A's I and B's K: all-gather B along K,
 *           then case 1.
 * Which collective runs is fixed by the ownership the consumer asks for
 * ("Sharded matrix multiplication and result ownership", The mechanism,
 * steps 1-5): all-reduce for a replicated C, reduce-scatter for row- (or
 * column-) owned C, all-gather only when the consumer needs the whole tensor.
 *
 * Virtual ranks.  Rank r's data lives in device buffers of its own; every
 * call takes a host array of N device pointers, one per rank, indexed by rank
 * id.  Rank ids are row-major over the mesh axes, first axis major; a dim
 * split by several axes (I_XY) flattens them with the first listed major.
 * Each buffer holds exactly that rank's box (shmm_plan_rank_box) as a dense
 * row-major matrix (leading dimension = box width).  Buffers of different
 * ranks must not overlap.  They may be slices of one allocation.
 *
 * Ownership of memory.  The caller allocates and frees every device buffer
 * (operands, results, partials, workspace).  The library allocates no device
 * memory; it owns only shmm_plan_t objects (host memory), freed by
 * shmm_plan_destroy.
 *
 * Execution.  Device work is enqueued asynchronously on `stream` (a
 * cudaStream_t; NULL = the legacy default stream) and the call returns once
 * it is enqueued.  Arguments are validated before anything is enqueued; a
 * call that returns an error has enqueued nothing, except SHMM_ERR_CUDA from
 * a launch in a multi-kernel call, after which the outputs are undefined.
 *
 * Errors.  Every entry point returns shmm_status_t (SHMM_OK = 0).  Errors are
 * not sticky: each call validates its own arguments.  shmm_last_error()
 * returns a human-readable message for the calling thread's last failure.
 * Device-side faults that kernels detect without trapping (a pipeline wait
 * that exceeded its time limit) are recorded in a device status word read by
 * shmm_sync_status().
 *
 * Numerics.  Inputs are bf16 or fp32.  Products accumulate in fp32; partial
 * sums are stored in fp32 (unless SHMM_FLAG_PARTIAL_OUT_DTYPE); the sum over a
 * reduction group is formed in fp32 in ascending rank order, one rounding per
 * addition, then rounded once to the output type (bf16: round to nearest
 * even).  SHMM_FLAG_TREE sums with a balanced pairwise tree over the ranks in
 * ascending order instead.  The fused path (SHMM_FLAG_FUSED) on tensor cores
 * accumulates the group's products in one fp32 accumulator, as one
 * contraction over the group's concatenated K in ascending rank order: the
 * same sum, rounded in a different order (no per-rank partial is formed).
 * With SHMM_FLAG_RANK_ORDER it keeps each rank's partial in its own fp32
 * accumulator and adds them in ascending rank order, so it matches the
 * standalone sequential reduction bit for bit; the CUDA-core path always
 * does this.  Every path is deterministic: one input gives one result.
 *
 * Environment (read at each call; none is needed in normal use).
 *   SHMM_TC_PAIR=0     tensor-core GEMMs on single CTAs (128-row tiles)
 *                      instead of CTA pairs (256-row tiles).
 *   SHMM_TC_WIDE=0|1   CTA-pair tiles 256 columns wide (0) or 512 (1)
 *                      instead of the launcher's choice.  Both widths give
 *                      the same bits.
 *   SHMM_TC_HALF_TAIL=0  no half tiles: by default, when the last wave of
 *                      256 x 512 tiles would leave at least half the CTA
 *                      pairs idle, its tiles run as 256-column halves, one
 *                      round on twice as many pairs.  Both give the same
 *                      bits.
 *   SHMM_PDL=0         the GEMMs and the collective kernels launch in
 *                      plain stream order.  By default each is a
 *                      programmatic dependent of the kernel before it in
 *                      the stream: its set-up may run while that kernel
 *                      finishes, and it touches no global memory until
 *                      that kernel has completed.
 *   SHMM_LN_BULK=0     LayerNorm (+ all-gather) reads each row with
 *                      per-thread loads instead of staging several rows
 *                      in shared memory through the bulk-copy engine.
 *                      Both give the same bits.
 *   SHMM_INJECT_FAIL=name[,name...]  the named entry points fail with
 *                      SHMM_ERR_INJECTED before enqueuing anything (tests
 *                      of error propagation).
 */
#ifndef SHMM_H
#define SHMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SHMM_OK = 0,
    SHMM_ERR_INVALID_SPEC = 1,   /* unknown axis, an axis splitting two dims of
                                    one array, or an ownership change that is
                                    neither a reduction nor an all-gather */
    SHMM_ERR_ILLEGAL_OUTPUT = 2, /* the requested C sharding is itself illegal,
                                    e.g. C[I_X,K_X] (cheat-sheet, Case 4) */
    SHMM_ERR_SHAPE = 3,          /* a dim does not split evenly, a size is
                                    <= 0, a buffer would exceed 2^62 bytes, or
                                    too many ranks/axes */
    SHMM_ERR_DTYPE = 4,          /* unsupported dtype combination */
    SHMM_ERR_NULL = 5,           /* a required pointer is NULL */
    SHMM_ERR_ALIGN = 6,          /* a device pointer is not 16-byte aligned */
    SHMM_ERR_CUDA = 7,           /* a CUDA runtime/driver call failed */
    SHMM_ERR_TIMEOUT = 8,        /* a kernel's bounded wait expired (device
                                    status word; see shmm_sync_status) */
    SHMM_ERR_NOMEM = 9,          /* host allocation failed, or the workspace
                                    passed is smaller than required */
    SHMM_ERR_UNSUPPORTED = 10,   /* valid request the plan does not need or
                                    this operation cannot serve (e.g. a
                                    reduce-scatter on a plan with no
                                    contracted-axis split) */
    SHMM_ERR_INJECTED = 11,      /* failure forced by SHMM_INJECT_FAIL (tests) */
    SHMM_ERR_BOUNDS = 12         /* bounds-checked build only: a kernel computed
                                    a global index outside its buffer and
                                    skipped the access (device status word;
                                    see shmm_bounds_checked) */
} shmm_status_t;

typedef enum { SHMM_F32 = 0, SHMM_BF16 = 1 } shmm_dtype_t;

#define SHMM_MAX_AXES 8
#define SHMM_AXIS_NAME_LEN 8
#define SHMM_MAX_RANKS 256

/* A device mesh: `naxes` named axes, rank count = product of sizes. */
typedef struct {
    int naxes;
    char name[SHMM_MAX_AXES][SHMM_AXIS_NAME_LEN]; /* NUL-terminated */
    int size[SHMM_MAX_AXES];                      /* each >= 1 */
} shmm_mesh_t;

/* A sharding of a 2-D array: for dim d (0 = rows, 1 = cols), the mesh axis
 * indices that split it, first = major.  naxes[d] == 0 means the dim is not
 * split (replicated over every axis not named anywhere). */
typedef struct {
    int naxes[2];
    int axes[2][SHMM_MAX_AXES];
} shmm_spec_t;

/* Plan flags */
#define SHMM_FLAG_FUSED 0x1u   /* shmm_run: fuse the collectives into the GEMM.
                                  Partial sums are reduced inside the GEMM:
                                  each output tile is summed over its
                                  reduction group (in its accumulator, or in
                                  the epilogue with SHMM_FLAG_RANK_ORDER) and
                                  written once to its owner(s).  Operand
                                  all-gathers (cases 2, 4) become in-place
                                  reads of the owners' shards by the GEMM's
                                  loads, where shard edges allow
                                  (info.fused_gather) */
#define SHMM_FLAG_GELU 0x2u    /* apply GeLU (tanh form) to the finished result
                                  before the output rounding (the column-
                                  parallel first matmul of an MLP pair) */
#define SHMM_FLAG_TREE 0x4u    /* standalone reduction: warp-shuffle pairwise
                                  tree over the ranks instead of the sequential
                                  rank-order sum */
#define SHMM_FLAG_PARTIAL_OUT_DTYPE 0x8u /* partial buffers are stored in the
                                  output dtype instead of fp32 */
#define SHMM_FLAG_RANK_ORDER 0x20u /* with SHMM_FLAG_FUSED: form every rank's
                                  partial on its own and add the partials in
                                  ascending rank order in the epilogue (bit
                                  for bit the standalone reduction), instead
                                  of accumulating the group's products in one
                                  accumulator; slower when the group is large
                                  (each rank's product drains the MMA
                                  pipeline before the epilogue can add it) */
#define SHMM_FLAG_SIMT 0x10u   /* local GEMM on CUDA cores even for bf16 (the
                                  tensor-core path is used otherwise whenever
                                  the shapes allow TMA: J_r, K_r multiples of
                                  8) */

/* Boxes a plan defines for each rank (shmm_plan_rank_box `tensor`). */
typedef enum {
    SHMM_TENSOR_A = 0,         /* rank's shard of A, as given */
    SHMM_TENSOR_B = 1,         /* rank's shard of B, as given */
    SHMM_TENSOR_C = 2,         /* rank's block of C, as requested */
    SHMM_TENSOR_P = 3,         /* rank's local product / partial C{U} */
    SHMM_TENSOR_A_LOCAL = 4,   /* A as the local GEMM reads it (after the
                                  case 2/4 all-gather) */
    SHMM_TENSOR_B_LOCAL = 5,
    SHMM_TENSOR_C_REDUCED = 6  /* rank's block after the reduction (the owner
                                  block of a reduce-scatter), before any
                                  all-gather of the result */
} shmm_tensor_t;

typedef enum {
    SHMM_COLL_NONE = 0,
    SHMM_COLL_REDUCE_SCATTER = 1,
    SHMM_COLL_ALL_REDUCE = 2
} shmm_collective_t;

typedef struct {
    int case_id;           /* 1..4 (cheat-sheet numbering) */
    int collective;        /* shmm_collective_t of the partial-sum reduction */
    int scatter_dim;       /* reduce-scatter dim: 0 = I, 1 = K; -1 if none */
    int nranks;
    int group_size;        /* ranks per reduction group (1 = none) */
    int ngroups;           /* number of reduction groups */
    int gather_A_size;     /* ranks per all-gather group of A (1 = none) */
    int gather_B_size;
    int gather_C_size;     /* ranks per all-gather group of the result */
    int in_dtype, out_dtype, partial_dtype;
    uint32_t flags;
    int tensor_core;       /* 1 if the local GEMM runs on tcgen05 */
    int fused;             /* 1 if shmm_run reduces inside the GEMM
                              (SHMM_FLAG_FUSED honoured: on tensor cores, at
                              most 16 ranks per group; otherwise shmm_run
                              reduces with the standalone kernel) */
    int64_t local_I, local_J, local_K;   /* per-rank GEMM M, K, N */
    int64_t flops_per_rank;              /* 2 * local_I * local_J * local_K */
    int64_t payload_operand_ag;          /* bytes each rank sends, counted once
                                            at the sender (ownership page,
                                            step 6) */
    int64_t payload_reduce_scatter;
    int64_t payload_result_ag;
    size_t workspace_bytes;              /* shmm_run's workspace requirement */
    int fused_gather;      /* 1 if shmm_run reads the case 2/4 operands in
                              place from their owners' shards inside the GEMM
                              (SHMM_FLAG_FUSED, tensor cores, shard edges on
                              64-column / 128-row boundaries, <= 16 ranks)
                              instead of all-gathering them first */
} shmm_plan_info_t;

typedef struct shmm_plan shmm_plan_t;

/* Builds a plan: validates the shardings (a mesh axis splits at most one dim
 * of an array: cheat-sheet Notation, Rule), classifies the case, derives the
 * operand gathers, the reduction groups (ranks that differ only on the
 * contracted axes), the owner of every output block and the collective the
 * requested C sharding needs (ownership page, steps 1-5).  Host only.
 *   mesh, spec_A, spec_B, spec_C  in: the mesh and the three shardings
 *                                     (spec_C = the consumer's ownership)
 *   I, J, K                       in: global sizes; every split must be even
 *   in_dtype                      in: dtype of A and B
 *   out_dtype                     in: dtype of C
 *   flags                         in: SHMM_FLAG_*
 *   plan                          out: new plan, owned by the caller
 * Errors: NULL, SHAPE, INVALID_SPEC, ILLEGAL_OUTPUT, DTYPE, NOMEM. */
shmm_status_t shmm_plan(const shmm_mesh_t *mesh, const shmm_spec_t *spec_A,
                        const shmm_spec_t *spec_B, const shmm_spec_t *spec_C,
                        int64_t I, int64_t J, int64_t K, shmm_dtype_t in_dtype,
                        shmm_dtype_t out_dtype, uint32_t flags, shmm_plan_t **plan);

/* Frees a plan (NULL is accepted). */
shmm_status_t shmm_plan_destroy(shmm_plan_t *plan);

/* Caps how many SMs the plan's tensor-core GEMM launches occupy: at most
 * max_sms / 2 CTA pairs (or max_sms single CTAs) take the plan's tiles, in
 * the same tile order.  0 (the default) lets a launch take every SM.  The
 * cap lets independent plans run side by side on separate streams, each on
 * its own share of the SMs, instead of queueing whole-GPU launches with a
 * partial last wave each; results do not depend on it.  It has no effect on
 * the CUDA-core GEMM or the collective kernels.  Not thread-safe against a
 * concurrent shmm_run on the same plan.  Errors: NULL, SHAPE (max_sms < 0). */
shmm_status_t shmm_plan_set_sm_limit(shmm_plan_t *plan, int max_sms);

/* Fills `info` with the plan's classification, shapes and byte counts. */
shmm_status_t shmm_plan_query(const shmm_plan_t *plan, shmm_plan_info_t *info);

/* Offsets and extents (rows, cols) of `rank`'s box of `tensor` in the global
 * array: the "completed values with explicit per-rank coordinates" of the
 * ownership page (Interfaces).  Errors: NULL, SHAPE (rank out of range),
 * UNSUPPORTED (unknown tensor). */
shmm_status_t shmm_plan_rank_box(const shmm_plan_t *plan, int tensor, int rank,
                                 int64_t off[2], int64_t ext[2]);

/* Ranks of `rank`'s reduction group in ascending order (the summation
 * order); `ranks` must hold info.group_size entries. */
shmm_status_t shmm_plan_group(const shmm_plan_t *plan, int rank, int *ranks);

/* shmm_run's workspace requirement in bytes (0 if none). */
shmm_status_t shmm_workspace_size(const shmm_plan_t *plan, size_t *bytes);

/* Local GEMM of every rank (ownership page, step 3; Row Parallelism,
 * Z_i = X_i A_i): P_r = A_r . B_r over the rank's slice of J.
 *   A_r[N]  in: box SHMM_TENSOR_A_LOCAL, in_dtype
 *   B_r[N]  in: box SHMM_TENSOR_B_LOCAL, in_dtype
 *   P_r[N]  out: box SHMM_TENSOR_P; fp32 partials if the plan reduces (or
 *           out_dtype with SHMM_FLAG_PARTIAL_OUT_DTYPE), else out_dtype with
 *           GeLU applied if SHMM_FLAG_GELU.
 * Errors: NULL, ALIGN, CUDA. */
shmm_status_t shmm_local_matmul(const shmm_plan_t *plan, const void *const *A_r,
                                const void *const *B_r, void *const *P_r, void *stream);

/* Reduce-scatter of the partials over each reduction group ("Sharding Matrix
 * Multiply", Communication primitives; ownership page, step 4): for each
 * element, the fp32 sum over the group's partials in ascending rank order
 * (pairwise tree with SHMM_FLAG_TREE), GeLU if flagged, rounded to out_dtype,
 * written only to the rank that owns it.
 *   P_r[N]  in: box SHMM_TENSOR_P, partial dtype
 *   C_r[N]  out: box SHMM_TENSOR_C_REDUCED of a reduce-scatter plan; for an
 *           all-reduce plan, row block q (rows / group_size rows, dim 0) of
 *           the partial goes to the group's q-th rank in ascending rank id
 * Errors: NULL, ALIGN, UNSUPPORTED (plan has no contracted-axis split), CUDA. */
shmm_status_t shmm_reduce_scatter(const shmm_plan_t *plan, const void *const *P_r,
                                  void *const *C_r, void *stream);

/* All-reduce of the partials: every rank of a group receives the whole sum
 * (same arithmetic as shmm_reduce_scatter).
 *   P_r[N]  in: box SHMM_TENSOR_P
 *   C_r[N]  out: box SHMM_TENSOR_P, out_dtype
 * Errors: NULL, ALIGN, UNSUPPORTED, CUDA. */
shmm_status_t shmm_all_reduce(const shmm_plan_t *plan, const void *const *P_r,
                              void *const *C_r, void *stream);

/* All-gather ("Sharding Matrix Multiply", AllGather): every rank of a gather
 * group receives the concatenation of the group's blocks.
 *   tensor = SHMM_TENSOR_A: shards (box A) -> full (box A_LOCAL), in_dtype
 *   tensor = SHMM_TENSOR_B: shards (box B) -> full (box B_LOCAL), in_dtype
 *   tensor = SHMM_TENSOR_C: owner blocks (box C_REDUCED) -> requested blocks
 *                           (box C), out_dtype
 * Errors: NULL, ALIGN, UNSUPPORTED (the plan gathers nothing for `tensor`),
 * CUDA. */
shmm_status_t shmm_all_gather(const shmm_plan_t *plan, int tensor, const void *const *shard_r,
                              void *const *full_r, void *stream);

/* The whole sharded matmul: operand all-gathers (cases 2, 4), local GEMMs,
 * the reduction (fused into the GEMM with SHMM_FLAG_FUSED, else a
 * standalone kernel over fp32 partials in the workspace) and the result
 * all-gather the requested ownership needs.
 *   A_r[N], B_r[N]  in: boxes SHMM_TENSOR_A / SHMM_TENSOR_B
 *   C_r[N]          out: box SHMM_TENSOR_C
 *   workspace       device memory of >= shmm_workspace_size() bytes, 256-byte
 *                   aligned (may be NULL when the size is 0)
 * Errors: NULL, ALIGN, NOMEM (workspace too small), CUDA. */
shmm_status_t shmm_run(const shmm_plan_t *plan, const void *const *A_r, const void *const *B_r,
                       void *const *C_r, void *workspace, size_t workspace_bytes, void *stream);

/* The sharded matmul end to end from host memory: the pages' input is the
 * global operands plus their sharding, the output the completed values with
 * explicit per-rank coordinates ("Sharded matmuls and collectives on a
 * torus", interface of the sharded matmul).  This call scatters global A and
 * B onto the ranks' device buffers, runs shmm_run's arithmetic, and writes
 * the global C back to host memory.
 *   A_host  in: global A [I, J], row-major, in_dtype, host memory; NULL when
 *           A_r already holds every rank's shard (nothing is uploaded)
 *   B_host  in: global B [J, K], likewise
 *   C_host  out: global C [I, K], row-major, out_dtype, host memory; every
 *           element written once, from the lowest rank holding it; NULL to
 *           leave the result on the device only
 *   A_r[N], B_r[N]  out (or in, for a NULL host operand): device buffers of
 *           boxes SHMM_TENSOR_A / SHMM_TENSOR_B; each distinct shard crosses
 *           the host link once, and ranks holding the same box (replicas)
 *           receive device-to-device copies of it
 *   C_r[N]  out: box SHMM_TENSOR_C, as for shmm_run
 *   workspace, workspace_bytes: as for shmm_run
 * Results are bit for bit those of uploading the shards and calling
 * shmm_run.  When every unit of work reads only its own ranks' shards (no
 * operand or result all-gather; a reduction only if fused), the work runs
 * in stages, at most one per 16 MB of host operands and at most 16:
 * reduction groups or ranks, each split into blocks of 256-row multiples
 * when there are fewer units than stages and a block of C rows needs only
 * the same rows of A.  A stage's uploads overlap the previous stage's GEMM
 * and its downloads overlap the next; consecutive stages' GEMMs alternate
 * between `stream` and a second compute stream, so they may overlap too.
 * A B box goes up whole at its first use, and its replicas are copied
 * right after it (the staged GEMMs read the uploaded box itself).
 * Copies and those GEMMs run on four library-owned streams of the current
 * device (uploads, replica copies, downloads, compute; created on first
 * use, kept until exit), ordered against `stream` by events: they start
 * after the work already enqueued on `stream`, and work enqueued on `stream`
 * after this call sees every copy complete.  Host buffers must stay valid
 * until then; page-locked host memory is needed for copies that overlap
 * compute (pageable memory works, serialised).
 * Errors: NULL, ALIGN, NOMEM (workspace), CUDA; the shmm_run errors. */
shmm_status_t shmm_run_host(const shmm_plan_t *plan, const void *A_host, const void *B_host, void *C_host,
                            void *const *A_r, void *const *B_r, void *const *C_r, void *workspace,
                            size_t workspace_bytes, void *stream);

/* Reshard a 2-D array [rows, cols] between two shardings on one mesh:
 * every rank's block under `spec_to` is assembled from the blocks holding it
 * under `spec_from` (one read and one write of each element).  This is the
 * AllToAll of "Sharding Matrix Multiply" (Communication primitives) and of
 * the torus page (The four collectives): A[I, J_X] -> A[I_X, J] moves which
 * dim is sharded; it also covers all-gathers (axes dropped) and slicing
 * (axes added).  Where the source replicates a block, rank r reads the copy
 * held by the rank that shares its coordinates on the replicated axes.
 *   src_r[N]  in: box of each rank under spec_from (row-major, dense)
 *   dst_r[N]  out: box of each rank under spec_to
 * No plan: host work is O(ranks x source blocks) per call.
 * Errors: NULL, SHAPE, INVALID_SPEC, DTYPE, ALIGN, CUDA. */
shmm_status_t shmm_reshard(const shmm_mesh_t *mesh, const shmm_spec_t *spec_from,
                           const shmm_spec_t *spec_to, int64_t rows, int64_t cols, shmm_dtype_t dtype,
                           const void *const *src_r, void *const *dst_r, void *stream);

/* Layer normalisation of every row of x [rows, cols] (a token over its
 * features): y = (x - mean) / sqrt(var + eps) * gamma[c] + beta[c], mean and
 * biased variance over the row, computed in fp32 and rounded once to dtype.
 * The per-token normalisation the sequence-parallel block applies locally
 * ("The simple maths behind parallel training", Sequence parallelism).
 *   x, y       device buffers (may be the same), 16-byte aligned
 *   gamma, beta  device fp32 arrays of `cols`
 * Errors: NULL, ALIGN, SHAPE, DTYPE, CUDA. */
shmm_status_t shmm_layernorm(int64_t rows, int64_t cols, shmm_dtype_t dtype, const void *x,
                             const float *gamma, const float *beta, float eps, void *y, void *stream);

/* Sequence parallelism's normalise-then-gather in one pass: for a plan whose
 * result is row-owned and requested whole (its all-gather runs along rows:
 * e.g. a reduce-scatter over tokens, Y[T_X, D], gathered to Y[T, D]), every
 * owner block (box SHMM_TENSOR_C_REDUCED) is layer-normalised row by row and
 * written to every member's gathered block (box SHMM_TENSOR_C).  Each row
 * is read once.  gamma, beta: fp32 arrays of the row length shared by all
 * ranks.  Errors: NULL, ALIGN, UNSUPPORTED (no row all-gather), CUDA. */
shmm_status_t shmm_layernorm_all_gather(const shmm_plan_t *plan, const void *const *shard_r,
                                        const float *gamma, const float *beta, float eps,
                                        void *const *full_r, void *stream);

/* ---- planner: which operand to move ("Sharded matmuls and collectives on
 * a torus", Which operand to move: the ICI roofline) ---------------------- */

/* Per-device rates of the model: C (dense matmul FLOP/s) and W (bytes/s one
 * device moves on the mesh axis, e.g. the ICI link rate of an axis, or HBM
 * bandwidth for virtual ranks sharing one GPU). */
typedef struct {
    double flops_per_s;
    double bytes_per_s;
} shmm_device_model_t;

typedef struct {
    int choice;              /* 1: all-gather W; 2: keep W sharded, reshard X
                                to X[B,D_X], all-reduce the [B,F] partials */
    int gather_compute_bound;/* strategy 1's matmul outlasts its all-gather
                                (B > C/W) */
    double bytes_gather;     /* bytes strategy 1 moves per device: e*D*F */
    double bytes_reduce;     /* bytes strategy 2 moves per device: 2*e*B*F */
    double t_gather;         /* modelled seconds, max(communication, compute) */
    double t_reduce;
} shmm_operand_choice_t;

/* For X[B,D] . W[D_X,F] on a mesh axis of `axis_size` devices with element
 * size `elem_bytes`: strategy 1 all-gathers W (e*D*F bytes at W, eq. 5.1)
 * and computes the whole 2*B*D*F product per device; strategy 2 moves the
 * activations (an all-reduce of e*B*F bytes, 2V/W, eq. 5.2) and computes
 * 2*B*D*F/axis_size.  Each strategy costs max(communication, compute)
 * (communication overlaps the matmul); the cheaper one is returned.  At
 * large B this picks strategy 2 exactly when D > 2C/W, the page's threshold.
 * Host only.  Errors: NULL, SHAPE (a size <= 0, rates <= 0). */
shmm_status_t shmm_choose_operand(int64_t B, int64_t D, int64_t F, int axis_size, int elem_bytes,
                                  const shmm_device_model_t *device, shmm_operand_choice_t *out);

/* Runs n independent sharded matmuls, as n calls of shmm_run would, with
 * their local GEMMs sharing launches: every plan whose shmm_run is a single
 * tensor-core GEMM launch (operands read whole or gathered in place, a
 * fused reduction or none, no all-gather of the result) joins one
 * persistent tile walk over all their tiles (up to 4 plans and 16 operand
 * slots and outputs per launch; more take further launches). Sharing a
 * launch pays its fixed cost once and fills the last wave of tiles with
 * other plans' work. Plans that do not qualify run through shmm_run first,
 * on the same stream. Each plan's results are bit for bit those of its own
 * shmm_run. The plans must be independent: no output buffer of one may be
 * an input or output of another. SM limits (shmm_plan_set_sm_limit) apply
 * only when every joined plan has one; the launch then takes the largest.
 *   n                 in: number of plans (0: nothing to do)
 *   plans             in: n plans
 *   A_r, B_r, C_r     in: per plan, its per-rank pointer array, as shmm_run
 *   workspaces        in: per plan, its workspace (NULL entries, or a NULL
 *                         array, where no plan needs one)
 *   workspace_bytes   in: per plan, the workspace sizes (or NULL)
 *   stream            in: cudaStream_t
 * Every plan and pointer is checked before anything is enqueued.
 * Errors: those of shmm_run (the message names the plan's index), and
 * SHAPE (n < 0), NULL (NULL arrays). */
shmm_status_t shmm_run_batch(int n, const shmm_plan_t *const *plans, const void *const *const *A_r,
                             const void *const *const *B_r, void *const *const *C_r,
                             void *const *workspaces, const size_t *workspace_bytes, void *stream);

/* Size of the fixed device workspace behind shmm_run_static_workspace. *//* Size of the fixed device workspace behind shmm_run_static_workspace. */
#define SHMM_STATIC_WORKSPACE_BYTES (64u << 20)

/* shmm_run for callers that cannot allocate device memory: a plugin or host
 * framework that hands over only input and output buffers and offers no
 * allocator, or a latency-critical caller that must not call cudaMalloc
 * (which can synchronise the device) once it is running.  The pages have no
 * counterpart: this is an interface convenience of this library.
 * Same arguments and results as shmm_run, without the workspace: the
 * workspace is a file-scope device array of SHMM_STATIC_WORKSPACE_BYTES
 * (64 MiB) that every device loading the library holds until the process
 * exits.  This call allocates nothing.
 *   - Plans whose shmm_workspace_size() exceeds SHMM_STATIC_WORKSPACE_BYTES
 *     are rejected with SHMM_ERR_NOMEM before anything is enqueued.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  Host threads may make first calls at the
 *     same time.  The address stays cached for the process, so reset no
 *     device (cudaDeviceReset) while the library is in use; devices with an
 *     index of 64 or more are rejected with SHMM_ERR_CUDA.
 *   - Every call on a device shares the one array and it keeps the last
 *     call's contents; nothing in it needs to start at zero (each use
 *     writes every byte it later reads).  Calls that overlap on the GPU
 *     (different streams, or host threads without ordering) race on it:
 *     order them on one stream.
 * Errors: those of shmm_run, and NOMEM (workspace need above the limit). */
shmm_status_t shmm_run_static_workspace(const shmm_plan_t *plan, const void *const *A_r,
                                        const void *const *B_r, void *const *C_r, void *stream);

/* Synchronises `stream`, then reads and clears the device status word that
 * kernels set when a bounded wait expires (or, in the bounds-checked build,
 * when an index falls outside its buffer).  Returns SHMM_OK,
 * SHMM_ERR_TIMEOUT, SHMM_ERR_BOUNDS or SHMM_ERR_CUDA. */
shmm_status_t shmm_sync_status(void *stream);

/* Failure-detection self-test: enqueues one kernel that waits on a barrier
 * nothing arrives at, through the same bounded wait every pipeline wait of
 * this library uses, with a limit of `limit_cycles` SM clock cycles
 * (1e3..4e9; the pipelines use ~4e9, about 2 s).  The wait gives up, records
 * SHMM_ERR_TIMEOUT in the device status word and the kernel returns: the next
 * shmm_sync_status() reports SHMM_ERR_TIMEOUT and clears it, and the context
 * stays usable.  No counterpart on the pages: a test of this library's own
 * fault handling.  Errors: SHAPE (limit out of range), CUDA. */
shmm_status_t shmm_selftest_wait_timeout(uint64_t limit_cycles, void *stream);

/* Message for the calling thread's last failed call ("" if none). */
const char *shmm_last_error(void);

/* Static name of a status code. */
const char *shmm_status_string(shmm_status_t status);

/* Library version, major * 10000 + minor * 100 + patch. */
int shmm_version(void);

/* 1 if this library is the bounds-checked build (libshmm_checked.so,
 * compiled with SHMM_CHECKED), else 0.  That build compares every global
 * index its kernels compute with the extent of the buffer it addresses,
 * derived from the buffer sizes this header documents; an index outside it
 * is not accessed and shmm_sync_status() then reports SHMM_ERR_BOUNDS.  The
 * tensor-core GEMM's operand loads and bulk result stores go through tensor
 * maps whose extents are those buffer sizes, so the TMA unit clips them; its
 * per-thread store path is checked like the other kernels.  A debugging aid
 * with no counterpart on the pages; the checks cost time, so the ordinary
 * build leaves them out. */
int shmm_bounds_checked(void);

/* Number of kernels this library has enqueued since it was loaded, over all
 * threads and devices (a diagnostic for benchmarks and tests). */
uint64_t shmm_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* SHMM_H */
