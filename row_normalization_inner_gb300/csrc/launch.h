// Host-side launchers, one per kernel family.  Internal to libnf.so: the
// C ABI in include/nf.h validates arguments, picks a plan and calls these.
// Every launcher takes an already validated hidden size from the compiled
// set and returns the launch's cudaError_t.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace nf {

// Row-group shape of the register path for `hidden`: threads per row,
// rows per CTA.  False if `hidden` is not compiled.
bool reg_shape(int64_t hidden, int* tpr, int* rpc);
// Register-path forward calls of at most this many rows load their
// parameters before the first row and run one row per CTA, with twice the
// threads per row of larger calls.
constexpr int64_t kSmallCallRows = 256;
// Cluster path: CTAs per row (the cluster size) and threads per CTA.
bool cluster_shape(int64_t hidden, int* ctas_per_row, int* threads);
// Bulk path: threads per CTA (one producer warp group + consumer row
// groups), ring stages, dynamic shared memory and consumer row groups for
// `op` (0 fused, 1 rms, 2 ln fwd, 3 ln bwd, 4 rms bwd).  False if no bulk kernel
// exists for (op, hidden).
bool bulk_shape(int op, int64_t hidden, int* threads, int* stages, int* smem_bytes, int* groups);

// Register path (rows resident in registers).
// `sms` bounds the first wave of CTAs, which warm L2 with their first row
// before waiting for the kernel ahead in the stream.
cudaError_t launch_fused_reg(int64_t hidden, void* x, void* res, const void* w, int64_t rows,
                             float eps, int grid, int sms, cudaStream_t st);
cudaError_t launch_rms_reg(int64_t hidden, void* y, const void* x, const void* w, int64_t rows,
                           float eps, int grid, int sms, cudaStream_t st);
cudaError_t launch_ln_fwd_reg(int64_t hidden, void* y, float* mean, float* rstd, const void* x,
                              const void* gamma, const void* beta, int64_t rows, float eps,
                              int grid, int sms, cudaStream_t st);

// Cluster path (one row split across a cluster of CTAs).
cudaError_t launch_fused_cluster(int64_t hidden, void* x, void* res, const void* w, int64_t rows,
                                 float eps, int grid, cudaStream_t st);
cudaError_t launch_rms_cluster(int64_t hidden, void* y, const void* x, const void* w, int64_t rows,
                               float eps, int grid, cudaStream_t st);
cudaError_t launch_ln_fwd_cluster(int64_t hidden, void* y, float* mean, float* rstd, const void* x,
                                  const void* gamma, const void* beta, int64_t rows, float eps,
                                  int grid, cudaStream_t st);

// LayerNorm backward, stage 1 (register path): `grid` persistent CTAs,
// RPC row groups each, one column-partial slot per group.
cudaError_t launch_ln_bwd_reg(int64_t hidden, void* dx, float* ws, const void* dy, const void* x,
                              const float* mean, const float* rstd, const void* gamma,
                              int64_t rows, int grid, cudaStream_t st);
// Stage 2: dgamma/dbeta = fixed-order sum over the slots of ws[slot][2][hidden].
cudaError_t launch_column_reduce(const float* ws, float* dgamma, float* dbeta, int nslots,
                                 int64_t hidden, cudaStream_t st);

// One-plane variant: out[j] = fixed-order sum over the slots of ws[slot][hidden].
cudaError_t launch_column_reduce1(const float* ws, float* out, int nslots, int64_t hidden,
                                  cudaStream_t st);
// RMSNorm backward, stage 1 (register path): RPC slots per CTA, ws[slot][hidden].
cudaError_t launch_rms_bwd_reg(int64_t hidden, void* dx, float* ws, const void* dy, const void* x,
                               const void* dres, const void* w, int64_t rows, float eps, int grid,
                               cudaStream_t st);

// Bulk-copy staged path: `grid` persistent CTAs (one per SM), each over a
// contiguous row stripe; `status` is the device status word.
cudaError_t launch_fused_bulk(int64_t hidden, void* x, void* res, const void* w, int64_t rows,
                              float eps, int grid, int* status, cudaStream_t st);
cudaError_t launch_rms_bulk(int64_t hidden, void* y, const void* x, const void* w, int64_t rows,
                            float eps, int grid, int* status, cudaStream_t st);
cudaError_t launch_ln_fwd_bulk(int64_t hidden, void* y, float* mean, float* rstd, const void* x,
                               const void* gamma, const void* beta, int64_t rows, float eps,
                               int grid, int* status, cudaStream_t st);
// Stage 1 of LayerNorm backward on the bulk path: one column-partial slot
// per CTA (the row groups fold theirs inside the CTA).
cudaError_t launch_ln_bwd_bulk(int64_t hidden, void* dx, float* ws, const void* dy, const void* x,
                               const float* mean, const float* rstd, const void* gamma,
                               int64_t rows, int grid, int* status, cudaStream_t st);

// RMSNorm backward, stage 1 on the bulk path (one slot of ws[slot][hidden] per CTA).
cudaError_t launch_rms_bwd_bulk(int64_t hidden, void* dx, float* ws, const void* dy, const void* x,
                                const void* dres, const void* w, int64_t rows, float eps, int grid,
                                int* status, cudaStream_t st);

// Row-block backward kernels for hidden 1024 and 2048 (the bulk path's
// backward there): blocks of consecutive rows per bulk copy, a whole row per
// thread group, one column-partial slot per CTA, grid_per_sm x SMs CTAs.
// op: 3 LayerNorm backward, 4 RMSNorm backward.
bool rows_bwd_shape(int op, int64_t hidden, int* threads, int* stages, int* smem_bytes, int* groups,
                    int* grid_per_sm);
cudaError_t launch_ln_bwd_rows(int64_t hidden, void* dx, float* ws, const void* dy, const void* x,
                               const float* mean, const float* rstd, const void* gamma,
                               int64_t rows, int grid, int* status, cudaStream_t st);
cudaError_t launch_rms_bwd_rows(int64_t hidden, void* dx, float* ws, const void* dy, const void* x,
                                const void* dres, const void* w, int64_t rows, float eps, int grid,
                                int* status, cudaStream_t st);

// Runtime-hidden path (any hidden that is a multiple of 8 up to
// dyn_max_hidden(op)).  op: 0 fused, 1 rms fwd, 2 ln fwd, 3 ln bwd, 4 rms bwd.
// [kernel-span grid_norm] (the argument block the grid kernels read)
struct DynArgs {
    uint16_t* out0;          // fused: x; rms/ln fwd: y; bwd: dx
    uint16_t* out1;          // fused: residual
    const uint16_t* in0;     // x
    const uint16_t* in1;     // fused: residual; bwd: dy
    const uint16_t* p0;      // weight / gamma
    const uint16_t* p1;      // beta
    const uint16_t* add;     // rms bwd: gradient added to dx (fused-add backward), or null
    float* mean;             // ln fwd out / ln bwd in
    float* rstd;
    float* ws;               // bwd partials [grid][planes][hidden]
    float* cols0;            // split bwd with one row block: dgamma / dw written directly
    float* cols1;            //   and dbeta (the column reduction is then skipped), else null
    int64_t rows;
    int hidden;
    float eps;
};
// [end kernel-span grid_norm]
bool dyn_shape(int op, int64_t hidden, int* threads);
// Backward: resident CTAs per SM and the copy ring's shared memory; `add`:
// the ring also carries the fused-add backward's residual-stream gradient.
int dyn_bwd_per_sm(int64_t hidden, bool add);
size_t dyn_bwd_smem(int64_t hidden, bool add);
// Forward: the same for the forward's copy ring, used for rows of one warp
// (0 bytes: one CTA per row, no ring).
int dyn_fwd_per_sm(int op, int64_t hidden);
size_t dyn_fwd_smem(int op, int64_t hidden);
int64_t dyn_max_hidden(int op);
cudaError_t launch_dyn(int op, const DynArgs& a, int grid, cudaStream_t st);

// Grid-parallel inner normalization for long rows (runtime hidden, one row
// per cluster of `ctas` CTAs).  Forward up to long_max_hidden(op) = 262144,
// backward up to 131072.  op numbering as for the runtime-hidden path.
bool long_shape(int op, int64_t hidden, int* ctas, int* threads, int* slice);
int64_t long_max_hidden(int op);
cudaError_t launch_long(int op, const DynArgs& a, int grid, cudaStream_t st);

// Split rows (grid-parallel inner normalization across any number of CTAs):
// chunks of 8192 elements, partial statistics through the workspace.
constexpr int64_t kSplitMaxHidden = 1LL << 26;
// Backward row blocks of at most this many rows merge their rows' statistics
// inside the apply pass instead of in a separate launch.
constexpr int kSplitMergeRows = 16;
bool split_shape(int op, int64_t rows, int64_t hidden, int sms, int* nchunks, int* rblocks);
size_t split_workspace_bytes(int op, int64_t rows, int64_t hidden, int sms);
cudaError_t launch_split(int op, const DynArgs& a, void* workspace, int sms, cudaStream_t st);

// Grid-resident rows (one cooperative launch, one CTA per SM, each holding
// its column slice of every row in shared memory across a bounded grid
// barrier): calls of at most kGridMaxRows rows whose slices fit.  *vc:
// 8-element vectors per CTA per row; *smem: dynamic shared memory per CTA.
constexpr int kGridMaxRows = 8;
bool grid_shape(int op, int64_t rows, int64_t hidden, int sms, int* vc, size_t* smem);
size_t grid_workspace_bytes(int op, int64_t rows, int64_t hidden, int sms);
cudaError_t launch_grid(int op, const DynArgs& a, void* workspace, int sms, int* status, cudaStream_t st);
// Test hook: two cooperative CTAs wait at the grid barrier for a third that
// never comes; the bounded wait runs out and records NF_ERR_TIMEOUT.
cudaError_t launch_grid_selftest(void* counter16, uint64_t limit_ns, int* status, cudaStream_t st);

// Workspace bytes the plan `pl` of (op, rows, hidden) needs on a device of
// `sms` SMs (0 for forward plans that need none).
size_t plan_workspace_bytes(int op, int64_t rows, int64_t hidden, int sms, int path, int partials);

// Outer (per-column) normalization: row stripes, workspace bytes covering
// both directions, and the launch sequences.
int outer_stripes(int64_t rows, int64_t hidden, int sms);
size_t outer_workspace_bytes(int64_t rows, int64_t hidden, int sms);
cudaError_t launch_outer_fwd(void* y, float* mean, float* rstd, const void* x, const void* gamma,
                             const void* beta, int64_t rows, int64_t hidden, float eps,
                             void* workspace, int sms, cudaStream_t st);
cudaError_t launch_outer_bwd(void* dx, float* dgamma, float* dbeta, const void* dy, const void* x,
                             const float* mean, const float* rstd, const void* gamma, int64_t rows,
                             int64_t hidden, void* workspace, int sms, cudaStream_t st);
// The same on chip (the grid family): one cooperative launch, the row
// stripes held in shared memory band of columns by band, two bounded grid
// barriers per band.  For shapes where outer_grid_shape holds.
bool outer_grid_shape(int64_t rows, int64_t hidden, int sms, int* bvec, size_t* smem);
size_t outer_grid_workspace_bytes(int64_t rows, int64_t hidden, int sms);
cudaError_t launch_outer_grid_fwd(void* y, float* mean, float* rstd, const void* x, const void* gamma,
                                  const void* beta, int64_t rows, int64_t hidden, float eps,
                                  void* workspace, int sms, int* status, cudaStream_t st);

// Bounded-wait self test (see nf_selftest_wait_timeout).
cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t st);

}  // namespace nf
