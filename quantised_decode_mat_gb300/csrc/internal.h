// internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qmd.h"

namespace qmd {

// Error bits in the device error word.
enum : unsigned {
    ERRBIT_QMV_WAIT = 1u,     // a mat-vec pipeline wait gave up
    ERRBIT_DEBUG_WAIT = 2u,   // the test-only wait kernel gave up (as intended)
    ERRBIT_DRAIN_WAIT = 4u,   // draining copies after a give-up also gave up
    ERRBIT_PLAN = 8u,         // a launch whose geometry its plan does not allow (rows per CTA, threads)
};

struct DeviceInfo {
    int device;
    int sm_count;
    int smem_optin;   // max dynamic shared memory per block (opt-in)
    int smem_per_sm;  // shared memory per multiprocessor
    int cc_major, cc_minor;
};

// Device properties of the current device (cached); QMD_ERR_DEVICE if there is none.
qmd_status current_device(DeviceInfo *out);

// Address of the error word on the current device (set up once per device).
unsigned *device_error_word();

uint64_t wait_limit_ns();

// Test-only launch flags (bit 0: launch without programmatic dependent launch; bit 1: compute
// batches of 5..8 vectors with the dp4a kernel even where the tensor-core kernel applies; bit 2:
// the tensor-core kernel for every batch of 3..8; bit 3: the dp4a slice kernel instead of the
// row-lane kernel; bit 4: the row-lane kernel for batches of 3 and 4 as well).
unsigned launch_flags();
enum : unsigned {
    LAUNCH_NO_PDL = 1u,
    LAUNCH_DP4A_ONLY = 2u,
    LAUNCH_TC_ALL = 4u,
    LAUNCH_SLICE = 8u,
    LAUNCH_RL = 16u,
    LAUNCH_RL_DEEP = 32u,  // row-lane plan: rings up to 4 deep for one vector and one-step rows too
};

#ifdef QMD_TRACE
// Traced build: the stamp records for the next launch of `ctas` CTAs (QMD_TRACE_FIELDS each), or
// NULL when no trace buffer is set or it is full.
unsigned long long *trace_reserve(int ctas);
#endif

// Record a CUDA error for qmd_last_error_detail and map it to a status.
qmd_status fail(qmd_status st, const char *what, cudaError_t e);

// ---- mat-vec -------------------------------------------------------------------------------
struct QmvArgs {
    int fmt;  // QMD_Q4_K, QMD_Q5_K or QMD_Q6_K_SPLIT
    const uint8_t *W;
    const uint8_t *Wpre;
    const int8_t *xqs;
    const float *xd;
    const int16_t *xbs;
    float *y;
    int64_t rows;
    int nb;
    int batch;
    int32_t *dbg_dots;  // non-NULL selects the recording variant
    int32_t *dbg_sm;
    const float *x;      // non-NULL selects the fused form (packs x itself)
    int8_t *xq_qs_out;   // fused form: optional copy of the packed activations
    float *xq_d_out;
    int16_t *xq_bs_out;
    const float *r = nullptr;  // RMSNorm form: optional residual
    const float *g = nullptr;  // non-NULL selects the RMSNorm form (packs RMSNorm(x + r) * g)
    float *h_out = nullptr;    // RMSNorm form: optional h = x + r, written by CTA 0
    float eps = 0.0f;
    unsigned *ws = nullptr;    // optional scheduling workspace (row-lane kernel)
};

// Row-lane kernel with a workspace: how many of `tiles` 4-row tiles are handed out by claims.
int64_t dynamic_tiles(int64_t tiles);

struct QmvPlan {
    int layout;  // 0: dp4a slice kernel (qmv.cuh); 1: tensor-core kernel (qmv_tc.cuh); 2: row-lane kernel (qmv_rl.cuh);
                 // 3: split-K kernel (qmv_splitk.cuh)
    int grid, threads, smem, stages;
    int WR, RG, PR;  // warps per row group, row groups per CTA, rows per group per stage
    int row_bytes, pre_bytes, stage_bytes, row_stride;
    int tc_rows;  // tensor-core kernel: rows per CTA rounded up to its tile rows (sizes the run sums)
    int pre_steps = 0;  // row-lane, tensor-core, split-K kernels: ring slots per warp requested before the dependency wait
    int ksplit = 0;     // split-K kernel: CTAs per cluster, each with a slice of every row's blocks
    int tiles_c = 0;    // split-K kernel: the most 8-row tiles a cluster's range has
};

// Launch shape for these sizes on this device; QMD_ERR_SHAPE if K is above the batch's limit.
// mode: 0 plain, 1 recording, 2 fused pack (the kernel variants)
qmd_status qmv_plan(int fmt, int64_t rows, int nb, int batch, const DeviceInfo &dev, QmvPlan *plan,
                    int mode = 0);

qmd_status launch_qmv_q4k(const QmvArgs &a, const QmvPlan &plan, cudaStream_t s);
qmd_status launch_qmv_q5k(const QmvArgs &a, const QmvPlan &plan, cudaStream_t s);
qmd_status launch_qmv_q6k(const QmvArgs &a, const QmvPlan &plan, cudaStream_t s);
// Registers per thread of the dp4a kernel instance (batch, rows per stage, mode); 0 if unknown.
int qmv_regs_q4k(int batch, int PR, int mode);
int qmv_regs_q5k(int batch, int PR, int mode);
int qmv_regs_q6k(int batch, int PR, int mode);

// ---- pack, bind, debug ---------------------------------------------------------------------
qmd_status launch_rmsnorm_q8k_pack(const float *x, const float *r, const float *g, float eps, float *h_out,
                                   int8_t *qs, float *d, int16_t *bsums, int64_t K, int batch, cudaStream_t s);
qmd_status launch_q8k_pack(const float *x, int8_t *qs, float *d, int16_t *bsums, int64_t nblocks,
                           cudaStream_t s);
qmd_status launch_q6k_split(const uint8_t *gguf, uint8_t *body, uint16_t *prefix, int64_t rows,
                            int nb, int64_t prefix_stride, cudaStream_t s);

}  // namespace qmd
