/*
 * qmd.h -- C ABI of libqmd: decode-time Q4_K / Q6_K x q8_K matrix-vector products on one
 * NVIDIA GB300 (sm_103a).
 *
 * The operation ("Language models on the device: the cajeta-llm kernels", §1 and §2.1-2.2):
 * activations are quantised on the device to q8_K (256 values a block, one scale and eight
 * sub-block sums); each output row is an integer dot product of the row's GGUF K-quant weight
 * blocks against those bytes, with the per-sub-block scales and mins folded in through a
 * rank-one epilogue; batched decode dots one pass over a weight row against up to 8
 * activation columns.  At bind, a Q6_K weight is split into a scale prefix plus 208-byte
 * bodies and a Q4_K slab is read in place as 32-bit words (§1).
 *
 * Conventions for every call
 *  - All pointers to tensors are DEVICE pointers, owned by the caller, who also owns the
 *    stream.  The library allocates no device or host memory on any compute call (only the
 *    measurement helper qmd_measure_alu creates and frees its own scratch), keeps no per-call
 *    state, and never synchronises the stream (except qmd_get_device_error, which says so).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Calls
 *    are asynchronous; buffers must stay live until the stream has passed the work.
 *  - Arguments are validated on the host before anything is launched.  A call that returns
 *    anything but QMD_OK has launched nothing and written nothing.  There is no fallback:
 *    a refused call returns its named reason ("One kernel, any device", §1, the seven named
 *    launch refusals; "Kernel SPI and the selection algorithm", "Why a kernel declines").
 *  - Layouts are batch-major and row-major; K is the reduction length (columns of W), a
 *    multiple of 256; nb = K / 256.
 *  - Launch order: qmd_q8k_pack, qmd_rmsnorm_q8k_pack and qmd_qmatvec are launched as
 *    programmatic dependents of the preceding kernel in the stream.  Before waiting for that
 *    kernel to finish they read only weight buffers (W, W_aux; the norm gain g); everything
 *    else is read and written after it has finished.  Weights therefore must not be written
 *    by the kernel launched immediately before them in the same stream unless that kernel
 *    signals completion only by exiting (every kernel not written for programmatic launch
 *    does; so do this library's bind calls).
 */
#ifndef QMD_H
#define QMD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QMD_QK 256        /* values per K-quant and q8_K block */
#define QMD_MAX_BATCH 8   /* activation columns per weight pass */
#define QMD_Q4K_BLOCK_BYTES 144
#define QMD_Q5K_BLOCK_BYTES 176
#define QMD_Q6K_BLOCK_BYTES 210
#define QMD_Q6K_BODY_BYTES 208
#define QMD_WORKSPACE_BYTES 4096 /* scheduling workspace of qmd_qmatvec_ws / qmd_qmatvec_x_ws */

typedef enum qmd_status {
    QMD_OK = 0,
    QMD_ERR_NULL = 1,                  /* a required pointer is NULL */
    QMD_ERR_FORMAT = 2,                /* unknown weight format */
    QMD_ERR_K_NOT_MULTIPLE_OF_256 = 3, /* K % 256 != 0 */
    QMD_ERR_BATCH = 4,                 /* batch outside [1, QMD_MAX_BATCH] */
    QMD_ERR_MISALIGNED = 5,            /* a pointer is not aligned as the call requires */
    QMD_ERR_SHAPE = 6,                 /* rows < 1, K < 256, K above the call's limit, or a size overflow */
    QMD_ERR_LAUNCH = 7,                /* the CUDA runtime refused the launch (see qmd_last_error_detail) */
    QMD_ERR_DEVICE_TIMEOUT = 8,        /* a bounded wait inside a kernel gave up (qmd_get_device_error) */
    QMD_ERR_DEVICE = 9,                /* no usable CUDA device, or it is not an sm_103 part */
    QMD_ERR_VALUE = 10                 /* a scalar argument is out of its range (e.g. eps < 0 or not finite),
                                          or buffers that must not overlap do */
} qmd_status;

/* Weight formats, named by their GGUF type ids. */
typedef enum qmd_fmt {
    QMD_Q4_K = 12,       /* canonical GGUF Q4_K blocks, used in place (viewed as 32-bit words) */
    QMD_Q5_K = 13,       /* canonical GGUF Q5_K blocks, used in place */
    QMD_Q6_K_SPLIT = 14  /* GGUF Q6_K after qmd_bind_q6k: 208-byte bodies + f16 scale prefix */
} qmd_fmt;

/* A batch of q8_K-packed activation vectors, all device pointers, batch-major:
 *   qs    int8  [batch][K]       the codes, x ~= d * q, q in [-127, 127]
 *   d     f32   [batch][nb]      one scale per 256-value block
 *   bsums int16 [batch][nb][8]   sum of the 32 codes of each sub-block                   */
typedef struct qmd_q8k {
    int8_t *qs;
    float *d;
    int16_t *bsums;
} qmd_q8k;

typedef struct qmd_q8k_const {
    const int8_t *qs;
    const float *d;
    const int16_t *bsums;
} qmd_q8k_const;

/*
 * qmd_q8k_pack -- quantise `batch` f32 vectors of length K to q8_K
 * ("Language models on the device: the cajeta-llm kernels", §1: q8kPackKernel, 256 values a
 * block, one scale and eight sub-block sums).
 *
 * Per 256-value block, all in f32: amax = max |x|; if amax == 0 then d = 0 and every code and
 * sum is 0; otherwise q = clamp(round_to_nearest_even(x * (127 / amax)), -127, 127) (the
 * quotient and the product each rounded to f32) and d = amax / 127; bsums[j] is the sum of
 * codes 32j .. 32j+31.  In a block so small that 127/amax overflows to infinity, nonzero
 * values get +-127 and zeros get 0 (their product 0 * inf is NaN, whose code is 0).
 * Non-finite inputs are outside the contract (no fault, result unspecified).
 *
 *   x   f32 [batch][K], 16-byte aligned          (read)
 *   xq  qs and bsums 16-byte aligned, d 4-byte    (written)
 * Errors: NULL, K_NOT_MULTIPLE_OF_256, SHAPE (K < 256 or batch*K overflows), BATCH,
 * MISALIGNED, DEVICE, LAUNCH.
 */
qmd_status qmd_q8k_pack(const float *x, qmd_q8k xq, int64_t K, int batch, void *stream);

/*
 * qmd_rmsnorm_q8k_pack -- RMSNorm with an optional residual add, then the q8_K pack, in one
 * launch ("Language models on the device: the cajeta-llm kernels", §2.6: the normalisation and
 * residual kernels that produce the activation the device q8_K quantiser of §1 packs):
 *     h = x + r                     (r NULL: h = x)
 *     n = (h * (1 / sqrt(sum(h * h) / K + eps))) * g
 *     xq = qmd_q8k_pack(n)
 * per vector, each f32 operation rounded on its own (sqrt and the divisions correctly
 * rounded).  The sum of squares is taken in this order, so that results are reproducible
 * bit for bit: partial sum t (t < 256) adds the squares of elements t, t + 256, t + 512, ...
 * left to right; each group of 32 partials (32w .. 32w+31) is added as a pairwise tree,
 * p[l] += p[l + s] for s = 16, 8, 4, 2, 1 and l < s; the eight group totals left to right.
 *
 *   x      f32 [batch][K], 16-byte aligned                               (read)
 *   r      f32 [batch][K] residual stream, 16-byte aligned, or NULL        (read)
 *   g      f32 [K] gain, shared by every vector, 16-byte aligned           (read)
 *   eps    added to the mean square; finite and >= 0
 *   h_out  f32 [batch][K], 16-byte aligned, receives h; or NULL.  It may be the same buffer
 *          as x or r (an in-place residual update); it must not overlap g or xq.
 *   xq     as qmd_q8k_pack (written)
 * Errors: NULL (x, g or xq), K_NOT_MULTIPLE_OF_256, SHAPE (K < 256 or batch*K overflows),
 * BATCH, MISALIGNED, VALUE (eps), DEVICE, LAUNCH.
 */
qmd_status qmd_rmsnorm_q8k_pack(const float *x, const float *r, const float *g, float eps, float *h_out,
                                qmd_q8k xq, int64_t K, int batch, void *stream);

/*
 * qmd_qmatvec -- y[v][r] = sum over the row's blocks of the rank-one epilogue of integer
 * sub-block dots, for v < batch, r < rows
 * ("Language models on the device: the cajeta-llm kernels", §1, §2.1 one row finished by a
 * reduction; §2.2 the batched "Cols" form: one pass over a weight row serves all columns;
 * §2.3 Q5_K is Q4_K with a fifth-bit plane OR-ed into bit four of each code).
 *
 * Per 256-value block b of row r against vector v (exact int32 S and M, f32 elsewhere, each
 * operation rounded on its own):
 *   Q4_K, Q5_K:  S = sum_j sc_j * dot_j,  M = sum_j m_j * bsums[v][b][j]   (j = 0..7, 32 values;
 *                Q4_K codes 0..15, Q5_K codes 0..31)
 *                term = d_x * ( f32(d) * (float)S - f32(dmin) * (float)M )
 *   Q6_K_SPLIT:  S = sum_s sc_s * dot'_s, dot'_s over 16 values of (q - 32) * q8   (s = 0..15)
 *                term = d_x * ( f32(d) * (float)S )
 * and the row's terms are summed in f32 in this order: blocks in groups of four, each group
 * (t0 + t1) + (t2 + t3) with absent blocks past the row's end counted as +0; groups in runs
 * of four (16 blocks), each run ((G0 + G1) + G2) + G3 with absent groups counted as +0; then
 * the run sums left to right.  y is overwritten, not accumulated.
 *
 *   fmt    QMD_Q4_K, QMD_Q5_K or QMD_Q6_K_SPLIT
 *   W      Q4_K: GGUF blocks u8 [rows][nb][144] (16-byte aligned; read in place as u32 words)
 *          Q5_K: GGUF blocks u8 [rows][nb][176] (16-byte aligned; read in place)
 *          Q6_K_SPLIT: bodies u8 [rows][nb][208] from qmd_bind_q6k (16-byte aligned)
 *   W_aux  Q4_K, Q5_K: ignored (may be NULL).  Q6_K_SPLIT: the f16 scale prefix from qmd_bind_q6k,
 *          [rows][qmd_q6k_prefix_stride(K)] (16-byte aligned)
 *   xq     packed activations for `batch` vectors of length K (qs, bsums 16-byte aligned,
 *          d 4-byte aligned; bsums may be NULL for Q6_K_SPLIT, which does not read them)
 *   y      f32 [batch][rows], 4-byte aligned (written)
 * Limits: 1 <= batch <= 8; any K up to 32768 for batch <= 2 and up to 16384 above; longer
 * rows go to the tensor-core kernel, which takes them run by run when its per-run row sums
 * (32 x (ceil(K / 4096) - 1) bytes for each row a multiprocessor handles) fit in shared memory
 * (K = 32768: about 50,000 rows); QMD_ERR_SHAPE otherwise.
 * y must not overlap the packed input (other CTAs may still read it while one writes y).
 * Errors: NULL, FORMAT, K_NOT_MULTIPLE_OF_256, BATCH, MISALIGNED, SHAPE, VALUE (overlap), DEVICE,
 * LAUNCH.
 * Device-side bounded waits that give up, and a CTA that finds its launch geometry does not match
 * its plan (it then returns without touching memory), set a flag read by qmd_get_device_error.
 */
qmd_status qmd_qmatvec(qmd_fmt fmt, const void *W, const void *W_aux, qmd_q8k_const xq, float *y,
                       int64_t rows, int64_t K, int batch, void *stream);

/*
 * qmd_qmatvec_x -- the q8_K pack and the mat-vec in one launch: y is exactly
 * qmd_qmatvec(fmt, W, W_aux, qmd_q8k_pack(x), ...), with the same bits, but each CTA packs
 * the f32 activations itself into shared memory instead of reading a packed copy, which
 * removes a dependent launch from the stream ("Language models on the device: the cajeta-llm
 * kernels", §1 q8kPackKernel and the decode mat-vecs, here fused).
 *   x       f32 [batch][K], 16-byte aligned (read)
 *   xq_out  optional: if its three pointers are non-NULL, the packed activations are also
 *           written there (qs and bsums 16-byte aligned, d 4-byte aligned), the same bytes
 *           qmd_q8k_pack writes; all three NULL writes nothing.
 * Other arguments, limits and errors as qmd_qmatvec; in addition the batch's packed codes
 * (batch x K bytes) must fit in shared memory beside the weight stages (QMD_ERR_SHAPE
 * otherwise; every K <= 16384 at batch <= 4 and K <= 32768 at batch 1 fit), and neither y nor
 * xq_out may overlap x (every CTA reads x while others write): QMD_ERR_VALUE.
 */
qmd_status qmd_qmatvec_x(qmd_fmt fmt, const void *W, const void *W_aux, const float *x, qmd_q8k xq_out,
                         float *y, int64_t rows, int64_t K, int batch, void *stream);

/*
 * qmd_qmatvec_ws, qmd_qmatvec_x_ws -- qmd_qmatvec and qmd_qmatvec_x with a scheduling workspace:
 * the same results, bit for bit.  With one vector and enough rows that every warp of the
 * row-lane kernel has two 2-row tiles of its own (e.g. 28672 rows), the first three quarters of
 * the rows are split evenly over the multiprocessors as usual, and the last quarter is handed to
 * warps two rows at a time, in the order they ask for more work, so that a multiprocessor that
 * runs slow does not set the end of the launch.  Other launches ignore the workspace.  This is a scheduling choice of this implementation; the pages
 * have no counterpart.
 *   workspace  device, QMD_WORKSPACE_BYTES bytes, 16-byte aligned, owned by the caller.  Zero it
 *              once; every call that completes leaves it zeroed again.  Calls ordered in one stream
 *              may share one workspace; calls that may run at the same time on the GPU (other
 *              streams, concurrent graphs) need their own.  After a call reports
 *              QMD_ERR_DEVICE_TIMEOUT (qmd_get_device_error) zero the workspace again.
 * Other arguments, limits and errors as qmd_qmatvec / qmd_qmatvec_x; in addition NULL (no
 * workspace) and MISALIGNED (workspace).
 */
qmd_status qmd_qmatvec_ws(qmd_fmt fmt, const void *W, const void *W_aux, qmd_q8k_const xq, float *y,
                          int64_t rows, int64_t K, int batch, void *workspace, void *stream);
qmd_status qmd_qmatvec_x_ws(qmd_fmt fmt, const void *W, const void *W_aux, const float *x, qmd_q8k xq_out,
                            float *y, int64_t rows, int64_t K, int batch, void *workspace, void *stream);

/*
 * qmd_qmatvec_x_static -- qmd_qmatvec_x_ws without a caller-supplied workspace, for callers that
 * cannot allocate device memory: a plug-in whose host framework owns all device memory and hands
 * it only its inputs and outputs, or code that must not allocate on its inference path.  The
 * pages have no counterpart; this is a convenience of this library.
 *
 * The same results as qmd_qmatvec_x, bit for bit, scheduled as qmd_qmatvec_x_ws schedules them.
 * The workspace is the library's own: one QMD_WORKSPACE_BYTES array in device memory, defined at
 * file scope, which every GPU that loads the library holds until the process exits.  The call
 * allocates nothing (no cudaMalloc, no allocating library routine); it clears that array with
 * cudaMemsetAsync on `stream` and then launches the mat-vec.
 *  - The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 *    with that device current) and keeps it; make that first call before any stream capture.
 *  - Every call uses the same array, which keeps what the last call left: calls that may overlap
 *    on the GPU (other streams, concurrent graphs) race on it and give wrong results.  Issue them
 *    in one stream, or use qmd_qmatvec_x_ws with a workspace per stream.
 *  - Size limit: the array is one workspace, which schedules every shape the call accepts (its
 *    counters do not grow with the problem); shapes beyond qmd_qmatvec_x's limits are refused
 *    with the same statuses, before anything is launched.
 * Arguments, limits and errors as qmd_qmatvec_x; in addition DEVICE if the array's address cannot
 * be found on the current device.
 */
qmd_status qmd_qmatvec_x_static(qmd_fmt fmt, const void *W, const void *W_aux, const float *x, qmd_q8k xq_out,
                                float *y, int64_t rows, int64_t K, int batch, void *stream);

/*
 * qmd_qmatvec_rmsnorm_x -- the residual add, the RMSNorm, the q8_K pack and the mat-vec in one
 * launch: y is exactly qmd_qmatvec(fmt, W, W_aux, qmd_rmsnorm_q8k_pack(x, r, g, eps), ...),
 * with the same bits -- the same h, the same sum-of-squares order, the same codes ("Language
 * models on the device: the cajeta-llm kernels", §2.6 the normalisation and residual kernels
 * ahead of the device quantiser of §1 and the decode mat-vecs, here one launch).  Each CTA
 * forms h and its sum of squares itself, so the normalised vector never goes to memory and a
 * dependent launch leaves the stream.
 *   x, r, g, eps  as qmd_rmsnorm_q8k_pack (r may be NULL)
 *   h_out   f32 [batch][K], 16-byte aligned, receives h (written by one CTA); or NULL.  Unlike
 *           qmd_rmsnorm_q8k_pack it must NOT overlap x, r or g, since every CTA still reads x
 *           and r while it is written (QMD_ERR_VALUE); nor may y or xq_out overlap x or r.
 *   xq_out  optional, as qmd_qmatvec_x: the packed codes of the normalised vector
 * Other arguments as qmd_qmatvec.  Limits: at one or two vectors, any K whose packed codes fit
 * in shared memory beside the weight stages (about 180,000 at one vector); at three to eight,
 * the dp4a kernel's (K up to 16384); longer rows give QMD_ERR_SHAPE (pack with
 * qmd_rmsnorm_q8k_pack and call qmd_qmatvec instead).
 * Errors: NULL (W, x, g, y, a partial xq_out, or W_aux for Q6_K_SPLIT), FORMAT,
 * K_NOT_MULTIPLE_OF_256, BATCH, MISALIGNED, VALUE (eps, or h_out overlapping x, r or g),
 * SHAPE, DEVICE, LAUNCH.
 */
qmd_status qmd_qmatvec_rmsnorm_x(qmd_fmt fmt, const void *W, const void *W_aux, const float *x, const float *r,
                                 const float *g, float eps, float *h_out, qmd_q8k xq_out, float *y, int64_t rows,
                                 int64_t K, int batch, void *stream);

/*
 * qmd_q6k_prefix_stride -- entries (f16) per row of the Q6_K scale prefix: nb rounded up to
 * a multiple of 8, so that every prefix row starts on a 16-byte boundary.  0 if K is not a
 * positive multiple of 256.
 */
int64_t qmd_q6k_prefix_stride(int64_t K);

/*
 * qmd_q6k_split_bytes -- sizes of the two buffers qmd_bind_q6k writes:
 *   body   rows * nb * 208 bytes,  prefix   rows * qmd_q6k_prefix_stride(K) * 2 bytes.
 * ("Language models on the device: the cajeta-llm kernels", §1: scale prefix plus 208-byte
 * bodies.)  Errors: NULL, K_NOT_MULTIPLE_OF_256, SHAPE.
 */
qmd_status qmd_q6k_split_bytes(int64_t rows, int64_t K, size_t *body_bytes, size_t *prefix_bytes);

/*
 * qmd_bind_q6k -- bind-time relayout of a canonical GGUF Q6_K slab ("Language models on the
 * device: the cajeta-llm kernels", §1 and §2.6 split relayouts).  Each 210-byte block
 * (ql 128 B, qh 64 B, 16 int8 scales, f16 d) becomes a 208-byte body holding the first 208
 * bytes unchanged, and its f16 d goes to prefix[r][b]; prefix padding entries are zero.
 * Run once at load ("Kernel SPI and the selection algorithm": relayout once at load, never
 * per call).
 *   gguf    u8 [rows][nb][210], 2-byte aligned (read)
 *   body    u8 [rows][nb][208], 16-byte aligned (written)
 *   prefix  f16 [rows][qmd_q6k_prefix_stride(K)], 16-byte aligned (written)
 * The three buffers must not overlap.
 * Errors: NULL, K_NOT_MULTIPLE_OF_256, SHAPE, MISALIGNED, DEVICE, LAUNCH.
 */
qmd_status qmd_bind_q6k(const void *gguf, void *body, void *prefix, int64_t rows, int64_t K,
                        void *stream);

/*
 * qmd_bind_q4k -- the Q4_K bind is a view: the GGUF slab u8 [rows][nb][144] is read in place
 * as u32 [rows][nb][36] ("Language models on the device: the cajeta-llm kernels", §1: a Q4_K
 * slab is viewed as 32-bit words).  This call copies nothing; it checks that the slab can be
 * so viewed (16-byte aligned, K a multiple of 256, size without overflow).
 * Errors: NULL, K_NOT_MULTIPLE_OF_256, SHAPE, MISALIGNED.
 */
qmd_status qmd_bind_q4k(const void *gguf, int64_t rows, int64_t K);

/*
 * qmd_bind_q5k -- the Q5_K bind is a view as well: the GGUF slab u8 [rows][nb][176] (176 =
 * 11 x 16 bytes) is read in place.  Copies nothing; checks that the slab can be (16-byte
 * aligned, K a multiple of 256, size without overflow).
 * Errors: NULL, K_NOT_MULTIPLE_OF_256, SHAPE, MISALIGNED.
 */
qmd_status qmd_bind_q5k(const void *gguf, int64_t rows, int64_t K);

/* Name of a status code (static string). */
const char *qmd_status_str(qmd_status s);

/* Detail of the last QMD_ERR_LAUNCH / QMD_ERR_DEVICE on the calling thread (static or
 * thread-local string; empty if none). */
const char *qmd_last_error_detail(void);

/*
 * qmd_get_device_error -- synchronises `stream`, then reads and clears the current device's
 * error word, which kernels set when a bounded wait (on an asynchronous copy) gives up instead
 * of hanging.  Returns QMD_ERR_DEVICE_TIMEOUT if it was set, QMD_ERR_LAUNCH if the stream
 * reported a CUDA error, else QMD_OK.  ("One kernel, any device", §1: a refused launch is
 * returned with its reason, never dropped.)
 */
qmd_status qmd_get_device_error(void *stream);

/*
 * qmd_set_wait_limit_ns -- the time after which a bounded wait inside a kernel gives up
 * (default 1e9 ns).  Process-wide; applies to launches made after the call.
 */
void qmd_set_wait_limit_ns(uint64_t ns);

/*
 * qmd_qmatvec_launch_info -- the launch qmd_qmatvec would make for these sizes on the current
 * device: grid (CTAs), threads per CTA, dynamic shared bytes, pipeline stages, rows per
 * stage.  Any output pointer may be NULL.  Errors as qmd_qmatvec's shape checks.
 */
qmd_status qmd_qmatvec_launch_info(qmd_fmt fmt, int64_t rows, int64_t K, int batch, int *grid,
                                   int *threads, int *smem_bytes, int *stages, int *rows_per_stage);

/*
 * qmd_qmatvec_launch_kernel -- which kernel qmd_qmatvec would run for these sizes on the current
 * device: 0 the dp4a slice kernel, 1 the tensor-core kernel, 2 the row-lane kernel, 3 the split-K
 * kernel; a negative
 * qmd_status if the call would be refused.  (Debug launch flags and forced plans apply.)
 */
int qmd_qmatvec_launch_kernel(qmd_fmt fmt, int64_t rows, int64_t K, int batch);

/* ---- test-only entry points (same kernels, extra outputs) --------------------------------- */

/*
 * qmd_debug_qmatvec_dump -- qmd_qmatvec plus a record of its integer arithmetic, from the
 * same kernel code with extra stores.
 *   dots  int32 [batch][rows][nb][16], zeroed by the caller:
 *         Q4_K, Q5_K: entry j < 8 is dot_j of sub-block j (entries 8..15 stay 0);
 *         Q6_K_SPLIT: entry s is dot'_s of group s.
 *   sm    int32 [batch][rows][nb][2]: the block's S and (Q4_K, Q5_K) M; M = 0 for Q6_K_SPLIT.
 * Both 16-byte aligned.  Errors as qmd_qmatvec, plus NULL for dots/sm; at batches of 1..4
 * this entry also refuses K > 16384 (QMD_ERR_SHAPE).
 */
qmd_status qmd_debug_qmatvec_dump(qmd_fmt fmt, const void *W, const void *W_aux, qmd_q8k_const xq,
                                  float *y, int64_t rows, int64_t K, int batch, int32_t *dots,
                                  int32_t *sm, void *stream);

/*
 * qmd_measure_alu -- this device's issue rates for the two exact multiply-add paths of the
 * mat-vec, for an ALU roofline beside the HBM one: dp4a instructions per second (each sums
 * four int8 x int8 products into an int32; counted per thread) and f16 tensor FLOP/s through
 * mma.sync.m16n8k16 with f32 accumulation.  Two register-only kernels of a few milliseconds
 * on a private stream; the call waits for them.  Errors: NULL (either pointer), DEVICE, LAUNCH.
 */
qmd_status qmd_measure_alu(double *dp4a_per_s, double *mma_flop_per_s);

/*
 * qmd_measure_read_bw -- this device's read-only streaming rate, the ceiling for a kernel that
 * only reads its large operand: one CTA per multiprocessor streams its share of `buf` into shared
 * memory by 1-D bulk asynchronous copies (the path the mat-vecs read weights by) and discards it,
 * five times after a warm-up; bytes_per_s = 5 x bytes / elapsed.  `buf` is the caller's (device,
 * 16-byte aligned, bytes a multiple of 16 and at least 12288; make it several times the L2 so
 * that the reads come from HBM); only its contents' placement matters.  The call creates and
 * destroys a stream and two events and waits for its kernels.  Errors: NULL, MISALIGNED, SHAPE,
 * DEVICE, LAUNCH; a bounded wait that gives up sets the device error word.
 */
qmd_status qmd_measure_read_bw(const void *buf, size_t bytes, double *bytes_per_s);

/*
 * qmd_debug_wait_timeout -- launches one CTA that waits, with the given limit, on a
 * shared-memory barrier that nothing completes; the wait gives up, sets the device error
 * word and the kernel returns.  Used to test the bounded-wait path without hanging a GPU.
 */
qmd_status qmd_debug_wait_timeout(uint64_t limit_ns, void *stream);

/*
 * qmd_debug_set_plan -- override the mat-vec launch plan for launches made after the call:
 * row groups per CTA (each ceil(K/1024) warps; capped by the thread limit), rows per row group
 * per stage (1..8, rounded down to 1, 2, 4 or 8, then halved until rows x batch <= 16), a
 * cap on pipeline stages (a cap below 3 keeps batches of 5..8 off the tensor-core kernel), and
 * CTAs per multiprocessor (1..8); 0 keeps the default of each.
 * For the row-lane kernel, row groups are its warps with a ring and stages the slots of each ring.
 * Results do not depend on the plan; tests use this to drive the stage ring through many
 * wrap-arounds on small inputs.  Process-wide.
 */
void qmd_debug_set_plan(int row_groups, int rows_per_stage, int max_stages, int ctas_per_sm);

/*
 * qmd_debug_set_launch_flags -- test-only launch options for later launches: bit 0 launches
 * qmd_q8k_pack and qmd_qmatvec without programmatic dependent launch (plain stream order);
 * bit 1 computes batches of 5..8 vectors with the dp4a kernel even where the tensor-core
 * kernel would be chosen; bit 2 computes every batch of 3..8 vectors with the tensor-core
 * kernel where it fits (rows of more than 16 blocks run by run); bit 3 keeps one and two vectors
 * off the row-lane kernel (the dp4a slice kernel, or the tensor-core kernel for rows the slice
 * kernel cannot take); bit 4 puts three and four vectors on the row-lane kernel as well; bit 5
 * gives the row-lane kernel rings up to 4 deep for one vector and rows of at most 16 blocks too
 * (its plan keeps them at 2 there).  Results are the same either way.  Process-wide.
 */
void qmd_debug_set_launch_flags(unsigned flags);

/*
 * qmd_debug_set_dynamic_tiles -- test-only: the share, per mille (0..1000), of a row-lane launch's
 * 2-row tiles that qmd_qmatvec_ws hands out by claims (the rest split evenly); any other value
 * restores the default.  Results do not depend on it.  Process-wide.
 */
void qmd_debug_set_dynamic_tiles(int per_mille);

/*
 * qmd_debug_set_split_k -- split-K for later launches of one or two vectors (plain and fused
 * forms; "Language models on the device: the cajeta-llm kernels", §2.3: partial sums along K
 * and a fixup that adds them): each row's groups of four blocks are split over `ctas` CTAs
 * (2..8) of a thread-block cluster, each packing and multiplying only its slice, and the cluster
 * adds the slices' group sums in the declared row order through distributed shared memory.
 * Applies where a row has at least `ctas` groups; any other value restores the default plan.
 * Results are the same bits either way.  Process-wide.
 */
void qmd_debug_set_split_k(int ctas);

/* Library version, MAJOR*10000 + MINOR*100 + PATCH. */
int qmd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QMD_H */
