/*
 * nf.h -- C ABI of the GB300 (sm_103a) inner-persistent row-normalization
 * library (libnf.so).
 *
 * What the library computes, and where the operations come from:
 *   - Fused residual add + RMSNorm forward, in place: the RMSNormAdd
 *     benchmark with in-place update semantics in "optimize inner persistent
 *     scheduler for static fusion" (NVIDIA/Fuser PR #5281), changes
 *     walkthrough, test_rmsnorm_add_fwd.py entry.
 *   - RMSNorm forward and LayerNorm forward: "TMA inner persistent
 *     scheduler" (NVIDIA/Fuser PR #5587), description (RMS norm and layer
 *     norm, with a workspace).
 *   - LayerNorm backward as a combined per-row (inner) and across-rows
 *     (outer) reduction: "Llu/ln bwd" (NVIDIA/Fuser PR #207), title and the
 *     discussion, which names the layer norm backward as the special case of
 *     a grid-parallel normalization reducing both within and across rows.
 *   - The other variants that discussion lists: grid-parallel inner
 *     normalization (rows longer than one CTA: the cluster and split
 *     families) and outer normalization (nf_outer_norm_*); and the
 *     backward passes of RMSNorm and of the fused residual add.
 * The pages name the operations but print no formulas; each function below
 * states the textbook definition it implements.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout.   Activations are row-major, contiguous [rows, hidden] arrays of
 *           bf16 (IEEE binary32 with the low 16 mantissa bits dropped),
 *           row stride = hidden.  Weight, gamma and beta are [hidden] bf16.
 *           mean/rstd are [rows] fp32; dgamma/dbeta are [hidden] fp32.
 * Pointers. Every data pointer is a DEVICE pointer on the current CUDA
 *           device (or managed memory).  bf16 pointers, dgamma, dbeta and
 *           the workspace must be 16-byte aligned; mean/rstd 4-byte
 *           aligned.  Null pointers are accepted only when rows == 0.
 * hidden.   The compiled sizes 1024, 2048, 4096, 5120, 8192, 12288 get
 *           kernels specialized per size.  Any other multiple of 8 up to
 *           32768 (forward ops) or 16384 (backward ops) runs on the
 *           runtime-hidden kernels (NF_PATH_DYNAMIC); longer rows, up to
 *           262144 (forward) or 131072 (backward), run on the grid-parallel
 *           cluster kernels (NF_PATH_CLUSTER), which split one row over a
 *           cluster of 2, 4 or 8 CTAs; longer still, up to
 *           NF_SPLIT_MAX_HIDDEN, on the split kernels (NF_PATH_SPLIT), which
 *           spread a row over any number of CTAs, or, for up to 8 rows that
 *           fit on chip, the grid kernels (NF_PATH_GRID), which hold the
 *           rows in shared memory across one grid barrier; both need a
 *           workspace (the forward ops then take the _ws entry points).
 *           Other values (not a positive multiple of 8, or longer) return
 *           NF_ERR_UNSUPPORTED_HIDDEN.
 * rows.     Any value >= 0; rows == 0 returns NF_OK without launching.
 * eps.      Finite and > 0.
 * Stream.   Work is enqueued on `stream` (NULL = the legacy default
 *           stream) and the call returns without synchronizing.
 * Ownership.The caller owns every buffer (workspaces included); the
 *           library allocates no device memory.  It caches, per device, the
 *           SM count and the address of its device status word.
 * Launches. Kernels are launched as programmatic dependents of the work
 *           ahead of them on the stream; each waits for that work to
 *           complete before it touches memory, so stream order holds for
 *           every caller, and the calls can be captured into CUDA graphs.
 *           The first call of an entry point on a device sets kernel
 *           attributes (cudaFuncSetAttribute) and caches device state, so
 *           make that first call outside a stream capture.
 * Errors.   Argument checks happen before any launch and return a status;
 *           a failed launch returns NF_ERR_CUDA.  Nothing is thrown across
 *           the ABI.  A kernel that gives up on a bounded wait records
 *           NF_ERR_TIMEOUT in the device status word (read it with
 *           nf_get_device_status) and returns without trapping.
 * Aliasing. Outputs may not partially overlap inputs or each other; the
 *           only aliasing allowed is stated per function.
 * Results.  Accumulation is fp32; results are bit-identical from run to
 *           run on the same device (every reduction has a fixed order).
 */
#ifndef NF_H_
#define NF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NF_OK = 0,
    NF_ERR_INVALID_ARG = 1,         /* null pointer, rows < 0, bad eps, bad overlap */
    NF_ERR_UNSUPPORTED_HIDDEN = 2,  /* hidden not in the compiled set */
    NF_ERR_MISALIGNED = 3,          /* pointer alignment rule broken */
    NF_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace_bytes below the queried size */
    NF_ERR_CUDA = 5,                /* a CUDA runtime call or launch failed */
    NF_ERR_TIMEOUT = 6,             /* a kernel gave up on a bounded wait */
    NF_ERR_UNSUPPORTED_PATH = 7     /* forced path not built for this op/size */
} nf_status;

/* = cudaStream_t.  NULL is the legacy default stream. */
typedef struct CUstream_st* nf_stream;

/* Kernel families.  NF_PATH_AUTO lets the library choose from rows, hidden
 * and the SM count; the others force one family (for tests and ablations).
 *   REG     -- row resident in registers, 128-bit loads, one row per group
 *              of threads ("optimize inner persistent scheduler for static
 *              fusion": static hidden size, warp-multiple block size).
 *   CLUSTER -- one row split across a thread-block cluster, partial sums
 *              exchanged through distributed shared memory: the small-batch
 *              idea of the same page (more SMs per row), and the
 *              grid-parallel inner normalization "Llu/ln bwd" lists as
 *              missing (rows longer than one CTA holds; any hidden, forward
 *              and backward).
 *   BULK    -- a producer warp stages rows into a shared-memory ring with
 *              bulk asynchronous copies; consumer warps read 128-bit vectors
 *              from shared memory; registers move from producer to
 *              consumers ("TMA inner persistent scheduler").
 *   DYNAMIC -- the hidden size is a runtime argument (any multiple of 8 up
 *              to 32768 forward, 16384 backward); a thread owns at most
 *              four 16-byte vectors of a row, a compile-time bound ("TMA
 *              inner persistent scheduler": dynamic block dimensions).  The
 *              backward, and the RMSNorm / LayerNorm forward on rows of one
 *              warp, stream the next row through a per-thread copy ring in
 *              shared memory (nf_plan_query reports its bytes).  The only
 *              family for hidden sizes outside the compiled set.
 *   SPLIT   -- one row cut into 8192-element chunks, one CTA per (chunk,
 *              row), the row statistics passed through a caller workspace
 *              in global memory: grid-parallel inner normalization across
 *              any number of CTAs ("Llu/ln bwd"), for rows longer than a
 *              cluster holds (any multiple of 8 up to NF_SPLIT_MAX_HIDDEN).
 *              Forward calls on this family need a workspace: use the _ws
 *              entry points and nf_workspace_size.
 *   GRID    -- the split family's rows held on chip: one cooperative launch
 *              of one 512-thread CTA per SM; CTA c keeps its slice of
 *              ceil(hidden / 8 / SMs) vectors of EVERY row in shared memory,
 *              the CTAs exchange the per-row partial sums through the
 *              workspace across one grid barrier (a bounded wait: if it runs
 *              out the kernel records NF_ERR_TIMEOUT in the device status
 *              word and returns), and every CTA adds them in the same fixed
 *              order.  Each input row is read from memory once (the
 *              backward reads dy a second time, from L2), and a column's
 *              every row is in one CTA, so the backward writes
 *              dgamma / dbeta (dw) directly.  For 1 to 8 rows whose slices
 *              fit (rows * ceil(hidden / 8 / SMs) * 16 bytes within about
 *              226 KB): on GB300 up to 4 rows of 4194304 or 8 of 2097152.
 *              The automatic choice takes it wherever the split family
 *              would run and the rows fit, except for the RMSNorm backward
 *              (the split family's apply pass measured faster there).
 *              Forward calls need a workspace, as for SPLIT.  The fused op normalizes the residual as
 *              stored (bf16), the literal reading of the in-place update;
 *              the other families normalize the fp32 sum (both are within
 *              the stated tolerance of the exact result).                   */
typedef enum {
    NF_PATH_AUTO = 0,
    NF_PATH_REG = 1,
    NF_PATH_CLUSTER = 2,
    NF_PATH_BULK = 3,
    NF_PATH_DYNAMIC = 4,
    NF_PATH_SPLIT = 5,
    NF_PATH_GRID = 6
} nf_path;

/* Longest row any family handles (the split family). */
#define NF_SPLIT_MAX_HIDDEN (1LL << 26)

/* Operation ids for nf_plan_query. */
typedef enum {
    NF_OP_FUSED_ADD_RMSNORM = 0,
    NF_OP_RMSNORM_FWD = 1,
    NF_OP_LAYERNORM_FWD = 2,
    NF_OP_LAYERNORM_BWD = 3,
    NF_OP_RMSNORM_BWD = 4
} nf_op;

/* A launch plan, as chosen for (op, rows, hidden) on the current device. */
typedef struct {
    int32_t path;            /* nf_path actually used (never AUTO) */
    int32_t grid;            /* CTAs in the main launch */
    int32_t block;           /* threads per CTA */
    int32_t cluster;         /* CTAs per cluster (1 = none) */
    int32_t rows_per_cta;    /* rows a CTA computes at once (bulk: consumer row groups) */
    int32_t smem_bytes;      /* dynamic shared memory per CTA */
    int32_t launches;        /* kernel launches per call */
    int32_t partials;        /* column-partial slots (backward ops), else 0 */
} nf_plan;

/* Fused residual add + RMSNorm forward, in place.  For each row r:
 *     s_j          = x[r][j] + residual[r][j]          (fp32)
 *     residual[r][j] <- bf16(s_j)
 *     x[r][j]       <- bf16( s_j * rsqrt(mean_k(s_k^2) + eps) * weight[j] )
 * The normalization reads the unrounded fp32 sum s.  x and residual are
 * both read and written; they must not overlap each other, and weight must
 * not overlap either. */
nf_status nf_fused_add_rmsnorm(void* x, void* residual, const void* weight,
                               int64_t rows, int64_t hidden, float eps, nf_stream stream);

/* Bytes of workspace `op` needs for (rows, hidden) on the current device,
 * enough under every kernel family (so nf_set_path cannot make it short).
 * For the forward ops it is nonzero only because the split family (rows
 * longer than a cluster holds, or forced) keeps per-row partial statistics
 * there: rows * (8 * chunks + 8) bytes, chunks = ceil(hidden / 8192).  For
 * the backward ops it equals nf_layernorm_bwd_workspace_size /
 * nf_rmsnorm_bwd_workspace_size.  0 when rows == 0, hidden is unsupported,
 * op is unknown or the device cannot be queried. */
size_t nf_workspace_size(nf_op op, int64_t rows, int64_t hidden);

/* The forward entry points with a caller workspace (16-byte aligned, at
 * least nf_workspace_size(op, rows, hidden) bytes, contents irrelevant, not
 * overlapping any argument).  They behave exactly as the plain calls; the
 * workspace is used only when the plan is the split family (automatic
 * beyond the runtime-hidden limits, or forced).  Without a workspace (the
 * plain calls, or NULL here) an automatic split plan runs on the cluster
 * family instead where that holds the row (hidden <= 262144); longer rows,
 * or a forced split, return NF_ERR_WORKSPACE_TOO_SMALL. */
nf_status nf_fused_add_rmsnorm_ws(void* x, void* residual, const void* weight, int64_t rows,
                                  int64_t hidden, float eps, void* workspace,
                                  size_t workspace_bytes, nf_stream stream);

/* RMSNorm forward:  y[r][j] = bf16( x[r][j] * rsqrt(mean_k(x[r][k]^2) + eps) * weight[j] ).
 * y may be x itself (in place); any other overlap is rejected. */
nf_status nf_rmsnorm_fwd(void* y, const void* x, const void* weight,
                         int64_t rows, int64_t hidden, float eps, nf_stream stream);
nf_status nf_rmsnorm_fwd_ws(void* y, const void* x, const void* weight, int64_t rows,
                            int64_t hidden, float eps, void* workspace, size_t workspace_bytes,
                            nf_stream stream);

/* LayerNorm forward with biased variance:
 *     mean[r] = (1/H) sum_j x[r][j]
 *     var     = (1/H) sum_j (x[r][j] - mean[r])^2        (two passes over the resident row)
 *     rstd[r] = rsqrt(var + eps)
 *     y[r][j] = bf16( (x[r][j] - mean[r]) * rstd[r] * gamma[j] + beta[j] )
 * mean and rstd (fp32, [rows]) are the values a backward pass needs; either
 * may be NULL to skip it.  y may be x itself. */
nf_status nf_layernorm_fwd(void* y, float* mean, float* rstd, const void* x,
                           const void* gamma, const void* beta,
                           int64_t rows, int64_t hidden, float eps, nf_stream stream);
nf_status nf_layernorm_fwd_ws(void* y, float* mean, float* rstd, const void* x,
                              const void* gamma, const void* beta, int64_t rows, int64_t hidden,
                              float eps, void* workspace, size_t workspace_bytes,
                              nf_stream stream);

/* Bytes of workspace nf_layernorm_bwd needs for (rows, hidden) on the
 * current device, under any kernel family (0 when rows == 0 or hidden is
 * unsupported).  The value depends on the device's SM count, so query it
 * on the device that runs the call.  Returns 0 also if the device cannot
 * be queried. */
size_t nf_layernorm_bwd_workspace_size(int64_t rows, int64_t hidden);

/* LayerNorm backward.  With xhat = (x - mean) * rstd and g = dy * gamma:
 *   inner (per row):   dx[r][j] = bf16( rstd[r] * ( g_j - mean_k(g_k) - xhat_j * mean_k(g_k * xhat_k) ) )
 *   outer (per column): dgamma[j] = sum_r dy[r][j] * xhat[r][j],  dbeta[j] = sum_r dy[r][j]
 * mean/rstd are the forward's saved values (eps is folded into rstd, so
 * none is passed).  dgamma/dbeta are overwritten, not accumulated.  The
 * column sums go through `workspace` in two stages -- per-CTA partials,
 * then a fixed-order sum -- so they are deterministic.  workspace is a
 * caller-owned device buffer, 16-byte aligned, of at least
 * nf_layernorm_bwd_workspace_size(rows, hidden) bytes; its contents on
 * entry do not matter.  dx may be dy or x itself (exact alias).  With
 * rows == 0 nothing is read and dgamma/dbeta, where not NULL, are set to 0
 * (an empty column sum). */
nf_status nf_layernorm_bwd(void* dx, float* dgamma, float* dbeta,
                           const void* dy, const void* x, const float* mean, const float* rstd,
                           const void* gamma, int64_t rows, int64_t hidden,
                           void* workspace, size_t workspace_bytes, nf_stream stream);

/* Bytes of workspace nf_rmsnorm_bwd needs for (rows, hidden) on the current
 * device, under any kernel family (same rules as the LayerNorm query). */
size_t nf_rmsnorm_bwd_workspace_size(int64_t rows, int64_t hidden);

/* RMSNorm backward (the RMS counterpart of the combined inner + outer
 * reduction of "Llu/ln bwd"; "TMA inner persistent scheduler": RMS norm
 * with a workspace).  For y = x * rstd * w with
 * rstd = rsqrt(mean_k(x_k^2) + eps), g = dy * w and xhat = x * rstd:
 *   inner (per row):    dx[r][j] = bf16( rstd * ( g_j - xhat_j * mean_k(g_k * xhat_k) ) )
 *   outer (per column): dw[j]    = sum_r dy[r][j] * xhat[r][j]          (fp32, overwritten)
 * rstd is recomputed from x inside the kernel (one more sum in the same
 * row reduction, no extra memory traffic), so the forward need not save
 * it; pass the forward's eps.  The column sums go through `workspace` in
 * two fixed-order stages (deterministic).  dx may be dy or x itself.
 * rows == 0 sets dw (if not NULL) to 0.  Same pointer, alignment and
 * workspace rules as nf_layernorm_bwd. */
nf_status nf_rmsnorm_bwd(void* dx, float* dw, const void* dy, const void* x, const void* weight,
                         int64_t rows, int64_t hidden, float eps, void* workspace,
                         size_t workspace_bytes, nf_stream stream);

/* Fused residual-add + RMSNorm backward ("optimize inner persistent
 * scheduler for static fusion" pairs the fused add + RMSNorm forward with
 * in-place residual semantics; this is its gradient).  The forward left
 * s = x + residual in `residual` and y = s * rstd(s) * w in x.  Given the
 * gradient dy of y and, optionally, dres of the residual stream s:
 *   rstd   = rsqrt(mean_j(s_j^2) + eps)     (recomputed from the saved s)
 *   dx     = bf16( rstd * (g - s * rstd^2 * mean_j(g * s)) + dres ),  g = dy * w
 *   dw[j]  = sum_r dy[r][j] * s[r][j] * rstd[r]                      (fp32)
 * dx is the gradient of both forward inputs (x and residual).  dres may be
 * NULL (no residual-stream gradient); dx may be exactly dy, dres or
 * residual (in place).  Same hidden sizes, workspace (see
 * nf_rmsnorm_bwd_workspace_size), alignment and error rules as
 * nf_rmsnorm_bwd; dres, if given, must be 16-byte aligned. */
nf_status nf_fused_add_rmsnorm_bwd(void* dx, float* dw, const void* dy, const void* dres,
                                   const void* residual, const void* weight, int64_t rows,
                                   int64_t hidden, float eps, void* workspace,
                                   size_t workspace_bytes, nf_stream stream);

/* Size of the fixed scratch area nf_layernorm_bwd_noalloc uses. */
#define NF_LAYERNORM_BWD_NOALLOC_SCRATCH_BYTES (16u << 20)

/* LayerNorm backward that allocates nothing and takes no workspace.  The
 * source pages have no counterpart to this call; it is an addition of this
 * library for callers that cannot call cudaMalloc where they run the
 * backward pass (code inside a region where the framework's caching
 * allocator must not be entered, plugins that only receive pre-allocated
 * buffers, latency-critical paths that cannot take cudaMalloc's implicit
 * synchronization).  Same arguments, results and rules as nf_layernorm_bwd
 * minus the workspace: the column partials go to a fixed
 * NF_LAYERNORM_BWD_NOALLOC_SCRATCH_BYTES area of static device memory
 * inside the library (held by every GPU that loads the library until the
 * process exits).  Argument errors return what nf_layernorm_bwd returns, in
 * the same order, before the area is looked at.  A size whose partials need
 * more than the area under the plan the call runs returns
 * NF_ERR_WORKSPACE_TOO_SMALL before anything is launched.  At the compiled
 * sizes the largest need is hidden 12288 (one slot of 2 * 12288 fp32 per
 * SM: 14.25 MiB on a 152-SM GPU, so a part with more than 170 SMs refuses
 * it); the runtime-hidden sizes near 16384 and the split family's very long
 * rows can need more and are refused.  The first call on each device looks
 * up the area's device address (cudaGetSymbolAddress, with that device
 * current) and caches it; make that first call before any stream capture.
 * cudaDeviceReset ends the context that owns the area, so a process that
 * resets a device must not call this entry point on that device again.
 * Every call shares the one area, which keeps the last call's contents
 * (nothing needs clearing: every partial is written before it is read);
 * calls that overlap on the GPU -- on different streams or from different
 * host threads -- race on it, so serialize them. */
nf_status nf_layernorm_bwd_noalloc(void* dx, float* dgamma, float* dbeta, const void* dy,
                                   const void* x, const float* mean, const float* rstd,
                                   const void* gamma, int64_t rows, int64_t hidden,
                                   nf_stream stream);

/* Outer normalization: the statistics run down the columns, over the rows
 * (batch normalization of a [rows, hidden] matrix in training mode; the
 * "Llu/ln bwd" discussion lists block- and grid-parallel outer
 * normalization among the normalization variants).  For each column j:
 *     mean[j] = (1/R) sum_r x[r][j]
 *     var_j   = (1/R) sum_r (x[r][j] - mean[j])^2          (biased)
 *     rstd[j] = rsqrt(var_j + eps)
 *     y[r][j] = bf16( (x[r][j] - mean[j]) * rstd[j] * gamma[j] + beta[j] )
 * hidden: any multiple of 8 (no compiled-size restriction); rows >= 0
 * (rows == 0 writes nothing).  mean/rstd ([hidden] fp32) may be NULL.  The
 * per-column statistics are merged from row stripes in a fixed order
 * (Chan's pairwise formula), so results are deterministic.  workspace:
 * caller-owned, 16-byte aligned, at least
 * nf_outer_norm_workspace_size(rows, hidden) bytes, contents irrelevant.
 * y may be x itself.  Two forms: three streaming launches (statistics per
 * row stripe, a merge per column, the apply pass), the default; and, with
 * nf_set_path(NF_PATH_GRID), one cooperative launch that keeps each CTA's
 * row stripe on chip band of columns by band and merges across bounded grid
 * barriers (reads x once, but measured slower; NF_ERR_UNSUPPORTED_PATH when
 * a stripe of rows / SMs rows does not fit two band buffers of 16 vectors). */
size_t nf_outer_norm_workspace_size(int64_t rows, int64_t hidden);
nf_status nf_outer_norm_fwd(void* y, float* mean, float* rstd, const void* x, const void* gamma,
                            const void* beta, int64_t rows, int64_t hidden, float eps,
                            void* workspace, size_t workspace_bytes, nf_stream stream);

/* Outer normalization backward (saved per-column mean/rstd).  With
 * xhat = (x - mean[j]) * rstd[j] and g = dy * gamma[j]:
 *   dx[r][j]  = bf16( rstd[j] * ( g - (1/R) sum_s g[s][j] - xhat * (1/R) sum_s g[s][j] xhat[s][j] ) )
 *   dgamma[j] = sum_r dy[r][j] * xhat[r][j],  dbeta[j] = sum_r dy[r][j]   (fp32, overwritten)
 * The column sums go through `workspace` and the fixed-order column
 * reduction.  dx may be dy or x itself.  rows == 0 sets dgamma/dbeta (if
 * not NULL) to 0.  Same pointer and workspace rules as the forward. */
nf_status nf_outer_norm_bwd(void* dx, float* dgamma, float* dbeta, const void* dy, const void* x,
                            const float* mean, const float* rstd, const void* gamma, int64_t rows,
                            int64_t hidden, void* workspace, size_t workspace_bytes,
                            nf_stream stream);

/* Force a kernel family for every later call in this process (NF_PATH_AUTO
 * restores the library's choice).  A call whose op/size has no kernel of the
 * forced family returns NF_ERR_UNSUPPORTED_PATH.  Not thread-safe with
 * respect to calls in flight on other host threads; meant for tests and
 * ablations. */
nf_status nf_set_path(nf_path path);

/* The plan a call of `op` with (rows, hidden) would use now on the current
 * device, without launching anything. */
nf_status nf_plan_query(nf_op op, int64_t rows, int64_t hidden, nf_plan* out);

/* Pure host planning, no CUDA call: the plan for (op, rows, hidden) on a
 * device with `sm_count` SMs under the kernel-family choice `path`
 * (NF_PATH_AUTO = the library's own rule).  nf_plan_query and every entry
 * point use exactly this function with the device's SM count and the
 * nf_set_path setting.  Returns NF_ERR_UNSUPPORTED_HIDDEN,
 * NF_ERR_UNSUPPORTED_PATH or NF_ERR_INVALID_ARG (rows < 0, sm_count < 1,
 * unknown op or path, out == NULL) without touching *out. */
nf_status nf_plan_compute(nf_op op, int64_t rows, int64_t hidden, int32_t sm_count,
                          nf_path path, nf_plan* out);

/* Copy the device status word of the current device to the host after the
 * work queued on `stream` finishes (this synchronizes `stream`), reset it to
 * NF_OK, and return the copied value (NF_OK or NF_ERR_TIMEOUT), or
 * NF_ERR_CUDA if the copy itself fails. */
nf_status nf_get_device_status(nf_stream stream);

/* Test hook for the bounded-wait machinery: launch one CTA that waits on a
 * shared-memory barrier which nothing completes, giving up after
 * `timeout_ns` nanoseconds (clamped to [1e3, 1e9]).  The kernel records
 * NF_ERR_TIMEOUT in the device status word and returns normally; the
 * context stays usable. */
nf_status nf_selftest_wait_timeout(int64_t timeout_ns, nf_stream stream);

/* Test hook for the grid family's barrier: launch two cooperative CTAs that
 * wait at the grid barrier for a third CTA that does not exist, giving up
 * after `timeout_ns` nanoseconds (clamped to [1e3, 1e9]).  `workspace`: 16
 * bytes of device memory, 16-byte aligned, for the arrival counter (zeroed
 * on `stream` first).  The kernel records NF_ERR_TIMEOUT in the device
 * status word and returns normally.  NF_ERR_INVALID_ARG (null) or
 * NF_ERR_MISALIGNED before launching anything. */
nf_status nf_selftest_grid_timeout(void* workspace, int64_t timeout_ns, nf_stream stream);

/* Measurement hook: the launch floor set beside small-batch timings.
 * kind 0 launches one 32-thread CTA that only waits for the previous
 * kernel in the stream and exits (launched as a programmatic dependent,
 * like every operation's kernels); dst, src and bytes are ignored.  kind 1
 * copies `bytes` bytes (a positive multiple of 16) from src to dst
 * (16-byte aligned device pointers, not overlapping) with 256-thread CTAs
 * holding 4 16-byte vectors per thread, launched the same way: the
 * simplest kernel that moves a small-batch call's bytes.  Returns
 * NF_ERR_INVALID_ARG (unknown kind, bad size, null or overlapping
 * buffers) or NF_ERR_MISALIGNED before launching anything. */
nf_status nf_selftest_floor(int32_t kind, void* dst, const void* src, int64_t bytes,
                            nf_stream stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* nf_status_string(nf_status status);

/* Library version string (static). */
const char* nf_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NF_H_ */
