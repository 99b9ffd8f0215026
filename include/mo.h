/*
 * mo.h -- C ABI of the GB300 (sm_103a) owner-local optimizer step.
 *
 * The library implements the optimizer step that owner placement makes local
 * ("MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter
 * sharding", section 3 and section 4.4: the owner of a whole 2D matrix runs
 * Muon on it; the tail owner runs AdamW on the packed non-matrix tensors), and
 * the row-normalised alternative RMNP ("Optimizers In A Sharded World: Muon's
 * O(mn) Vs RMNP's Zero", sections 1 and 5).
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers on the current CUDA device, owned
 *    by the caller. Tables (mo_matrix, mo_tail_seg) and parameter structs are
 *    HOST memory, read during the call and not retained.
 *  - Matrices are dense row-major [rows, cols] ([out, in]) with no padding.
 *    Every base pointer must be 16-byte aligned.
 *  - Work is enqueued on `stream` and is asynchronous; no call synchronises
 *    the stream except mo_last_device_error. State (W, V, m, v) is updated
 *    in place.
 *  - Return value: MO_OK (0) or a negative MO_ERR_* code. Every argument is
 *    validated before anything is enqueued, so a rejected call has no effect.
 *    A failing CUDA runtime call yields MO_ERR_CUDA; mo_last_cuda_error()
 *    returns its cudaError_t.
 *  - A table with n == 0 is a no-op returning MO_OK.
 *  - NaN/Inf in gradients propagate; they are not checked.
 *  - Not thread-safe for concurrent calls that share a workspace.
 */
#ifndef MO_H_
#define MO_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MO_ABI_VERSION 4

enum mo_status {
  MO_OK = 0,
  MO_ERR_NULL_POINTER = -1,      /* a required pointer is NULL */
  MO_ERR_BAD_SHAPE = -2,         /* rows/cols/numel <= 0, n < 0, or a size over the supported maximum */
  MO_ERR_MISALIGNED = -3,        /* a device pointer is not 16-byte aligned */
  MO_ERR_BAD_PARAM = -4,         /* a hyperparameter is NaN/Inf or out of range */
  MO_ERR_WORKSPACE_TOO_SMALL = -5,
  MO_ERR_OVERLAP = -6,           /* W, V (or p, m, v) of one entry overlap */
  MO_ERR_CUDA = -7,              /* a CUDA runtime call failed; see mo_last_cuda_error() */
  MO_ERR_DEVICE_TIMEOUT = -8,    /* a bounded device-side wait expired (see mo_last_device_error) */
  MO_ERR_UNSUPPORTED_DEVICE = -9, /* the current device is not sm_103 */
  MO_ERR_SCRATCH_LIMIT = -10      /* muon_owner_step_noalloc: table too large for the built-in scratch */
};

/* One 2D matrix of an owner's shape table ("MatrixFSDP", section 4.1: one
 * full segment per matrix on its owner).
 *   W    fp32 [rows, cols] master weight, updated in place
 *   G    bf16 [rows, cols] gradient (bit pattern of bfloat16), read only
 *   V    fp32 [rows, cols] momentum, updated in place
 * W and V must not overlap; G may alias nothing that is written. */
typedef struct {
  float* W;
  const void* G;
  float* V;
  int64_t rows;
  int64_t cols;
} mo_matrix;

/* Muon hyperparameters ("Optimizers In A Sharded World", section 1 and the
 * appendix benchmark script; "MatrixFSDP", section 5.1 for weight decay).
 *   V <- mu V + G;  U = V (or G + mu V with nesterov);
 *   X0 = U / (||U||_F + eps), transposed if rows > cols;
 *   ns_steps x { A = X X^T;  B = b A + c A A;  X = a X + B X }   (MO_NS_GRAM)
 *   ns_steps x { A = X X^T;  B = A X;  X = a X + b B + c A B }   (MO_NS_APPENDIX)
 *   W <- W (1 - lr wd) - lr s X (transposed back), with
 *   s = sqrt(max(1, rows/cols)) (MO_LR_ORIGINAL) or 0.2 sqrt(max(rows, cols))
 *   (MO_LR_MATCH_RMS_ADAMW).
 * Defaults: lr 0.02, wd 0.01, mu 0.95, (a,b,c) = (3.4445, -4.7750, 2.0315),
 * eps 1e-7, ns_steps 5, ns_form MO_NS_GRAM, lr_adjust MO_LR_ORIGINAL,
 * nesterov 0. ns_steps must be in [1, 100]; nesterov 0 or 1.
 *  - MO_NS_GRAM is the fast form (5 (3 m^2 n + m^3) flops for m <= n). The
 *    appendix script's form costs 25 m^2 n and needs a larger workspace
 *    (mo_muon_workspace_bytes depends on ns_form); the two agree in exact
 *    arithmetic and differ by bf16 rounding.
 *  - nesterov and MO_LR_MATCH_RMS_ADAMW are the update of torch.optim.Muon,
 *    which "MatrixFSDP" section 5.1 runs (with match_rms_adamw, momentum 0.5
 *    and 2 Newton-Schulz steps for its convergence runs). */
enum mo_ns_form { MO_NS_GRAM = 0, MO_NS_APPENDIX = 1 };
enum mo_lr_adjust { MO_LR_ORIGINAL = 0, MO_LR_MATCH_RMS_ADAMW = 1 };
typedef struct {
  float lr, wd, mu, a, b, c, eps;
  int32_t ns_steps;
  int32_t ns_form;     /* enum mo_ns_form */
  int32_t lr_adjust;   /* enum mo_lr_adjust */
  int32_t nesterov;    /* 0: orthogonalise V; 1: orthogonalise G + mu V */
} mo_muon_params;

/* RMNP hyperparameters ("Optimizers In A Sharded World", section 1 and the
 * appendix rmnp_local): V <- mu V + G; D_i = V_i / max(||V_i||_2, eps) per
 * stored row; W <- W (1 - lr wd) - lr sqrt(max(1, rows/cols)) D.
 * eps defaults to 1e-12. */
typedef struct {
  float lr, wd, mu, eps;
} mo_rmnp_params;

/* One packed segment of the non-matrix AdamW tail ("MatrixFSDP", section 3).
 * p, g, m, v: fp32 [numel]; p, m, v updated in place, g read only. */
typedef struct {
  float* p;
  const float* g;
  float* m;
  float* v;
  int64_t numel;
} mo_tail_seg;

/* AdamW hyperparameters ("MatrixFSDP", section 5.1: decoupled weight decay).
 * step is t AFTER the increment (t >= 1):
 *   m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2;
 *   p <- p (1 - lr wd) - lr (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps). */
typedef struct {
  float lr, wd, beta1, beta2, eps;
  int64_t step;
} mo_adamw_params;

/* Bytes of device workspace muon_owner_step needs for this table. Host-only
 * computation (no CUDA call). Returns 0 if the table or params are invalid. */
size_t mo_muon_workspace_bytes(const mo_matrix* tbl, int32_t n, const mo_muon_params* params);

/* The Muon step over every matrix of the table, on `stream`.
 * ws: device workspace of at least mo_muon_workspace_bytes() bytes, 256-byte
 * aligned, owned by the caller; its contents are scratch, overwritten by every
 * call (two calls in flight on different streams must not share it).
 * Launches: one fused momentum + norm + bf16-cast prologue, then for each of
 * the ns_steps iterations three grouped tcgen05 GEMM launches (Gram, A.A with
 * the b A + c A A epilogue, B.X with the a X + epilogue; with MO_NS_APPENDIX:
 * Gram, A.X, A.B with the a X + b B + epilogue); the last launch applies the
 * weight update in its epilogue. Matrices are independent. Tables with a
 * matrix of max(rows, cols) > 32768 add, after each Gram launch, one launch
 * that sums the Gram slice partials (see mo_muon_tile_schedule); their
 * workspace includes m x m fp32 per slice. */
int muon_owner_step(const mo_matrix* tbl, int32_t n, const mo_muon_params* params,
                    void* ws, size_t ws_bytes, cudaStream_t stream);

/* As muon_owner_step, and additionally records `ev_ns_begin` on the stream
 * after the prologue (before the first GEMM launch) and `ev_ns_end` after the
 * last GEMM launch, so the caller can time the Newton-Schulz part alone.
 * Either event may be NULL. */
int muon_owner_step_timed(const mo_matrix* tbl, int32_t n, const mo_muon_params* params,
                          void* ws, size_t ws_bytes, cudaStream_t stream,
                          cudaEvent_t ev_ns_begin, cudaEvent_t ev_ns_end);

/* The same Muon step for callers that cannot allocate device memory (no
 * counterpart on the pages; it exists for the library's users). Processes
 * whose device memory is owned by another allocator, and contexts where
 * cudaMalloc is not allowed, cannot provide the `ws` buffer muon_owner_step
 * needs. This entry point allocates nothing: its scratch is a file-scope
 * device array of mo_static_scratch_bytes() bytes (64 MiB), which every device
 * that runs this code holds until the process exits.
 *  - Tables whose mo_muon_workspace_bytes() exceeds that size are rejected
 *    with MO_ERR_SCRATCH_LIMIT before anything is enqueued.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress with that device current) and keeps it for the
 *    life of the process; make that first call before any stream capture.
 *    A cudaDeviceReset recreates the device's context and may move the
 *    array, so calls after one are not supported.
 *  - All calls share the one array and it keeps the last call's contents;
 *    each call rewrites everything the step needs zeroed. Calls that overlap
 *    on the GPU (different streams, or concurrent host threads) race on it.
 * Arguments, layout, results and the other status codes are those of
 * muon_owner_step. */
int muon_owner_step_noalloc(const mo_matrix* tbl, int32_t n, const mo_muon_params* params, cudaStream_t stream);

/* Size in bytes of the scratch array muon_owner_step_noalloc uses. */
size_t mo_static_scratch_bytes(void);

/* A Muon step planned once for a fixed table, hyperparameters and workspace
 * (no counterpart on the pages; for callers that capture their training step
 * in a CUDA graph). muon_owner_step uploads its workspace header from host
 * memory on every call, which a graph cannot replay safely; a plan uploads it
 * once, and each step then enqueues only device work.
 *  - mo_muon_plan_create: validates and plans like muon_owner_step, binds the
 *    plan to `ws` (same size and alignment rules) and enqueues the header
 *    upload on `stream` (from pageable memory: call it outside any stream
 *    capture). Steps on other streams must be ordered after that upload.
 *    *out is set only on MO_OK; n must be >= 1.
 *  - mo_muon_plan_step: enqueues one Muon step on `stream`: a memset of the
 *    step's counters and flags, then the launches of muon_owner_step. No
 *    host-to-device copy and no planning, so it may be captured in a CUDA
 *    graph and the graph replayed. It returns MO_ERR_BAD_PARAM if the current
 *    device is not the plan's. Results are bit-identical to muon_owner_step
 *    with the same learning rate.
 *  - Learning rate: every step reads lr from the device fp32 at
 *    mo_muon_plan_lr_ptr(plan), initialised to params->lr by the create call,
 *    so a schedule can write it between steps or graph replays (stream
 *    ordered); decay = 1 - lr wd is formed on the device in double. The other
 *    hyperparameters are fixed at creation.
 *  - While a plan exists, `ws` belongs to it; two steps of one plan must not
 *    be in flight at once. W, G and V are accessed through the table's
 *    pointers, which must stay valid while steps or captured graphs run.
 *  - mo_muon_plan_destroy frees host memory only; a graph captured from the
 *    plan stays valid as long as `ws` and the tensors do. NULL is a no-op. */
typedef struct mo_muon_plan_s* mo_muon_plan;
int mo_muon_plan_create(const mo_matrix* tbl, int32_t n, const mo_muon_params* params,
                        void* ws, size_t ws_bytes, cudaStream_t stream, mo_muon_plan* out);
int mo_muon_plan_step(mo_muon_plan plan, cudaStream_t stream);
float* mo_muon_plan_lr_ptr(mo_muon_plan plan);   /* device address; NULL for a NULL plan */
int mo_muon_plan_destroy(mo_muon_plan plan);

/* AdamW over every tail segment, on `stream` (one grouped launch per 256
 * segments). */
int adamw_tail_step(const mo_tail_seg* segs, int32_t n, const mo_adamw_params* params,
                    cudaStream_t stream);

/* RMNP over every matrix of the table, on `stream` (one grouped launch per 512
 * matrices; no workspace). The shape scale is sqrt(max(1, rows/cols)) of each
 * entry's own rows and cols. Rows are independent, so an entry may also be a
 * contiguous row block of a larger matrix; use rmnp_step_scaled to give such
 * blocks the whole matrix's scale. */
int rmnp_step(const mo_matrix* tbl, int32_t n, const mo_rmnp_params* params, cudaStream_t stream);

/* RMNP with an explicit per-entry shape scale (scales[i] replaces
 * sqrt(max(1, rows/cols)) for entry i), so that row blocks of one matrix can
 * be updated with the whole matrix's scale ("Optimizers In A Sharded World",
 * appendix rmnp_local: the scale uses the full matrix's rows). */
int rmnp_step_scaled(const mo_matrix* tbl, const float* scales, int32_t n,
                     const mo_rmnp_params* params, cudaStream_t stream);

/* HTRMNP: RMNP whose row direction keeps a power of the row norm.
 * "Optimizers In A Sharded World" section 7 says HTRMNP scales the row
 * direction with a power of the row norm, p = 0.125 by default, and prints no
 * formula; this library takes the reading
 *   V <- mu V + G;  D_i = V_i / max(||V_i||_2, eps)^(1 - power);
 *   W <- W (1 - lr wd) - lr sqrt(max(1, rows/cols)) D,
 * so power = 0 is rmnp_step and power = 1 applies the momentum itself.
 * Arguments and layout as rmnp_step; power must be in [0, 1]
 * (MO_ERR_BAD_PARAM otherwise). */
int htrmnp_step(const mo_matrix* tbl, int32_t n, const mo_rmnp_params* params, float power, cudaStream_t stream);

/* Device-resident hyperparameters, for steps captured in a CUDA graph (no
 * counterpart on the pages). A captured launch keeps the arguments it was
 * captured with; these entry points read the values that change from step to
 * step from device memory when the kernels run, so a schedule can update them
 * between replays (stream ordered).
 *  - adamw_tail_step_dev: as adamw_tail_step, with t (after the increment,
 *    >= 1) read from the device int64 *d_step (8-byte aligned), and lr from
 *    the device float *d_lr when d_lr is not NULL (4-byte aligned). The
 *    caller advances *d_step between steps (for example inside the captured
 *    graph); params->step, and params->lr when d_lr is set, are ignored (and
 *    not validated). The device values are used as found.
 *  - rmnp_step_dev: rmnp_step (power 0) or htrmnp_step (power in (0, 1]),
 *    with lr read from the device float *d_lr (not NULL); params->lr is
 *    ignored.
 * Every AdamW and RMNP kernel forms its per-step factors (1 - lr wd, the
 * bias corrections) on the device from lr, wd and t, so these entry points
 * give results bit-identical to the by-value ones for the same values. */
int adamw_tail_step_dev(const mo_tail_seg* segs, int32_t n, const mo_adamw_params* params,
                        const int64_t* d_step, const float* d_lr, cudaStream_t stream);
int rmnp_step_dev(const mo_matrix* tbl, int32_t n, const mo_rmnp_params* params, float power,
                  const float* d_lr, cudaStream_t stream);

/* RMNP with rows cut into column shards ("Optimizers In A Sharded World",
 * section 3, column-cut tensor parallelism, and the appendix's column-cut
 * scheme), evaluated on one GPU: each table entry is one dense column shard
 * [rows, cols_i] of a logical matrix; entries with equal group[i] are shards
 * of the same matrix, must be consecutive in the table and have equal rows.
 * Per shard: V <- mu V + G and the sum of squares of each of its rows; per
 * row of a matrix, the shard partials are added in table order (the page's
 * all-reduce); then every shard updates
 *   W <- W (1 - lr wd) - lr scales[i] V / max(sqrt(total), eps).
 * params->eps is the clamp (the page's scheme uses 1e-7). scales[i] is
 * normally sqrt(max(1, rows / total_cols)) of the whole matrix.
 * ws: device buffer of mo_rmnp_colcut_workspace_bytes() bytes (the per-row
 * partial sums), 16-byte aligned. At most 512 entries per call. */
size_t mo_rmnp_colcut_workspace_bytes(const mo_matrix* shards, int32_t n);
int rmnp_colcut_step(const mo_matrix* shards, const int32_t* group, const float* scales, int32_t n,
                     const mo_rmnp_params* params, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Synchronises `stream`, then returns and clears the device-side status word:
 * MO_OK, or MO_ERR_DEVICE_TIMEOUT if a bounded wait inside a kernel expired
 * (the kernel then skipped its remaining work and released its resources). */
int mo_last_device_error(cudaStream_t stream);

/* cudaError_t of the most recent MO_ERR_CUDA on this thread (0 if none). */
int mo_last_cuda_error(void);

/* Static description of a status code (never NULL). */
const char* mo_status_string(int status);

/* MO_ABI_VERSION of the loaded library. */
int mo_abi_version(void);

/* ---- host-side planning, exposed for inspection and testing (no CUDA) ---- */

/* One output tile of a grouped Newton-Schulz GEMM launch. */
typedef struct {
  uint32_t mat;   /* index into the shape table */
  uint16_t tm;    /* tile row (units of 256 rows: one CTA pair) */
  uint16_t tn;    /* tile column (units of 256 columns) */
} mo_tile;

enum mo_ns_phase { MO_PHASE_GRAM = 0, MO_PHASE_POLY = 1, MO_PHASE_UPDATE = 2 };

/* Writes the tile schedule of one phase (in launch order) into out[0..cap)
 * and the tile count into *count. A launch with at least 256 tiles per CTA
 * pair (128 for the last launch, which applies the weight update) hands them
 * out in this order from one device counter, each pair taking the next as it
 * frees up; a shorter launch assigns them statically (pair c of P runs tiles
 * c, c + P, c + 2P, ...). Returns MO_OK, or MO_ERR_BAD_SHAPE if cap is
 * too small (then *count holds the required size). Tiles are sorted by
 * decreasing reduction length K (n for the Gram, m otherwise), ties broken by
 * table index, then tile row and tile column (Gram, A.A) or tile column and
 * tile row (B.X). Gram and A.A tiles cover only tiles that touch the upper
 * triangle (col_end > row_begin). A Gram with n > 32768 is split along its
 * reduction into slices of 32768 columns (the last one shorter), each
 * accumulated separately in fp32 and summed by a reduction launch: its tiles
 * appear once per slice, with K = the slice length, after the whole
 * matrices of equal K in (matrix, slice) order, reported with the matrix's
 * index. */
int mo_muon_tile_schedule(const mo_matrix* tbl, int32_t n, int32_t phase,
                          mo_tile* out, int64_t cap, int64_t* count);

/* Tile schedule of the Newton-Schulz launches (muon_owner_step_coverage). */
enum mo_ns_schedule {
  MO_SCHED_AUTO = 0,     /* as muon_owner_step: by tiles per CTA pair */
  MO_SCHED_STATIC = 1,   /* every launch assigns its tiles statically */
  MO_SCHED_COUNTER = 2   /* every launch hands out its tiles from its counter */
};

/* Test support (no counterpart on the pages): muon_owner_step that also
 * counts on the device how often each Newton-Schulz output tile was executed,
 * under the tile schedule `schedule` (mo_ns_schedule; MO_ERR_BAD_PARAM for
 * another value). Every tile's arithmetic is the same under either schedule,
 * so the results are too, bit for bit.
 *  - *needed (must not be NULL) receives the number of uint32 counters: two
 *    per tile (the even and the odd CTA of the pair that computes it) for
 *    every GEMM launch of the step, in launch order (per iteration: Gram,
 *    then A.A (appendix form: A.X), then B.X), each launch's tiles in its
 *    launch order (mo_muon_tile_schedule; a long Gram's slices are separate
 *    tiles there).
 *  - coverage NULL: nothing runs (size query, host only). Otherwise
 *    `coverage` is a caller-zeroed device buffer of coverage_len counters
 *    (MO_ERR_BAD_SHAPE if fewer than *needed) and the step runs as
 *    muon_owner_step would, with the same results; every counter reads 1
 *    afterwards when each tile ran exactly once on each CTA of its pair.
 * Other arguments and status codes as muon_owner_step. */
int muon_owner_step_coverage(const mo_matrix* tbl, int32_t n, const mo_muon_params* params,
                             void* ws, size_t ws_bytes, uint32_t* coverage, int64_t coverage_len,
                             int32_t schedule, int64_t* needed, cudaStream_t stream);

/* ---- owner planning ("MatrixFSDP", section 4.1, Algorithm 1) ----
 * A role is one 2D matrix or the packed non-matrix tail of one block. The
 * planner assigns every role whole to one of `world` owner ranks, balancing
 * the owner-resident element count (the load). Host only; no CUDA call.
 *   MO_PLAN_ROLE_GREEDY   blocks in increasing block id; within a block the
 *                         roles in decreasing numel (ties: table order), each
 *                         to the currently lightest rank (ties: lowest rank);
 *                         loads carry across blocks.
 *   MO_PLAN_SCOPE_GREEDY  all roles pooled in decreasing numel (ties: table
 *                         order), each to the lightest rank.
 *   MO_PLAN_COST_AWARE    ScopeGreedy if its max/avg load ratio is strictly
 *                         lower than RoleGreedy's and no rank owns more than
 *                         `block_cap` elements within one block (block_cap <= 0:
 *                         no cap); RoleGreedy otherwise.
 * owner_out[nroles] receives the owner of each role, load_out[world] (may be
 * NULL) the per-rank loads, chosen_out (may be NULL) the strategy applied.
 * Returns MO_ERR_BAD_PARAM for an unknown strategy or world < 1,
 * MO_ERR_BAD_SHAPE for negative numel or block ids, MO_ERR_NULL_POINTER for
 * missing arrays. */
typedef struct {
  int64_t numel;   /* elements of the role (>= 0) */
  int32_t block;   /* FSDP block (wrap unit) the role belongs to (>= 0) */
  int32_t is_tail; /* 1 for a block's packed non-matrix tail, 0 for a matrix */
} mo_role;

enum mo_plan_strategy { MO_PLAN_ROLE_GREEDY = 0, MO_PLAN_SCOPE_GREEDY = 1, MO_PLAN_COST_AWARE = 2 };

int mo_plan_owners(const mo_role* roles, int32_t nroles, int32_t world, int32_t strategy, int64_t block_cap,
                   int32_t* owner_out, int64_t* load_out, int32_t* chosen_out);

/* ---- diagnostics ---- */

/* Launches one CTA that waits on a barrier nothing will complete, with a
 * bounded wait of `timeout_ns` nanoseconds (clamped to [1e3, 1e10]); on
 * expiry it records MO_ERR_DEVICE_TIMEOUT in the device status word and
 * returns. Used to test the bounded-wait error path without hanging. */
int mo_selftest_bounded_wait(int64_t timeout_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MO_H_ */
