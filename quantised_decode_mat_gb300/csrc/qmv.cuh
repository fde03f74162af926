// qmv.cuh -- the Q4_K / Q5_K / Q6_K x q8_K decode mat-vec kernel (templated on format, batch,
// rows per stage).
//
// What it computes ("Language models on the device: the cajeta-llm kernels"):
//   §1   integer dot products of weight codes against q8_K activation bytes, with the
//        per-sub-block scales (and Q4_K's mins, through the q8_K sub-block sums) folded in by a
//        rank-one epilogue per 256-value block;
//   §2.1 a reduction over the row's blocks finishes each output row;
//   §2.2 batched decode: one pass over a weight row is dotted against up to 8 vectors;
//   §2.3 a Q5_K member differs from the Q4_K one only in staging, the fifth-bit plane OR-ed
//        into bit four of each code (here: in registers, before the dot products).
//
// How, on sm_103a.  The pages' design has one wave own a row, each lane loading its own words
// from global memory, with "prefetch twins" issuing the next block's loads early.  Here:
//   * Persistent CTAs own contiguous row ranges.  A CTA's rows stream through a ring of
//     shared-memory stages (each RG x PR whole rows) by 1-D bulk async copies (cp.async.bulk,
//     mbarrier completion, L2 evict-first): kilobytes in flight per SM without registers.
//   * A CTA is RG row groups of WR = ceil(nb / 4) warps.  Warp w of a group covers blocks
//     4w .. 4w+3 of each of its PR rows; lane (g, k) = (lane / 8, lane % 8) takes 16-byte slice
//     k of block 4w+g.  A thread's slice is the same for every row, so its activation bytes
//     (2 x 16 B per vector) stay in registers for the whole kernel.  Per row it reads 16 B of
//     codes (plus the block header) from shared memory, widens nibbles / 6-bit codes in
//     registers and runs 8 dp4a per vector.
//   * The 8 lanes of a block combine their integers exactly by a reduce-scatter over the
//     PR x B (row, vector) slots, so each lane holds one slot's block total and evaluates
//     that block's f32 epilogue; the warp then sums its four blocks as (t0 + t1) + (t2 + t3).
//   * No CTA-wide barrier in the main loop.  Each warp posts its per-row partials in shared
//     memory and bumps the stage's arrival counter; the warp that arrives last adds the WR
//     partials of each row left to right, writes y, and re-issues the stage's copy.  Warps
//     never wait for one another, only for data.
//   * Programmatic dependent launch: the first stages are requested before waiting for the
//     previous kernel in the stream (which produces the activations).
//   * Every barrier wait is bounded; on give-up a warp flags the device error word, waits
//     (bounded) for the CTA's copies in flight, and exits.
#pragma once

#include <mutex>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "q8k.cuh"

namespace qmd {

struct QmvKParams {
    const uint8_t *W;     // Q4_K blocks or Q6_K bodies, [rows][row_bytes]
    const uint8_t *Wpre;  // Q6_K f16 prefix, [rows][pre_bytes]
    const int8_t *xqs;
    const float *xd;
    const int16_t *xbs;
    float *y;
    int64_t rows;
    int nb, WR, RG, stages, row_bytes, pre_bytes, stage_bytes, row_stride;
    int batch;
    int tc_rows;          // tensor-core kernel: rows per CTA rounded up to its tile rows
    int32_t *dbg_dots;
    int32_t *dbg_sm;
    const float *x;       // fused form: f32 activations [B][K], packed inside the kernel
    int8_t *xq_qs_out;    // fused form, optional: the packed activations, written by CTA 0
    float *xq_d_out;
    int16_t *xq_bs_out;
    const float *r;       // RMSNorm form: optional residual [B][K] (h = x + r, else h = x)
    const float *g;       // RMSNorm form: gain [K]
    float *h_out;         // RMSNorm form, optional: h, written by CTA 0
    float eps;            // RMSNorm form
    unsigned *err;
    unsigned long long wait_ns;
    unsigned *ws;         // row-lane kernel: the scheduling workspace (two counters), or NULL
    int64_t dyn_tiles;    // row-lane kernel with a workspace: the last tiles, handed out by claims
    int pre_steps;        // row-lane, tensor-core kernels: ring slots per warp requested before the dependency wait
#ifdef QMD_TRACE
    unsigned long long *trace;  // traced build: QMD_TRACE_FIELDS time stamps per CTA, or NULL
#endif
};

// Traced build only (compiled with -DQMD_TRACE): per-CTA global-timer stamps of the phases of a
// launch, for the per-phase breakdown of a decode step.  Fields: 0 entry, 1 first weight copies
// requested, 2 dependency wait released, 3 activations ready, 4 first stage landed, 5 the last
// stage's rows written, 6 exit (the latest warp), 7 SM id | CTA << 16 | grid << 32 | kind << 48.
constexpr int QMD_TRACE_FIELDS = 8;
#ifdef QMD_TRACE
#define QMD_STAMP(P, I)                                                                            \
    do {                                                                                           \
        if ((P).trace)                                                                             \
            (P).trace[(size_t)blockIdx.x * QMD_TRACE_FIELDS + (I)] = globaltimer_ns();             \
    } while (0)
#else
#define QMD_STAMP(P, I) \
    do {                \
    } while (0)
#endif

// Kernel variants: plain; recording the integer arithmetic; packing f32 activations itself;
// packing the RMSNorm of x (+ a residual) itself.
enum QmvMode { QMV_PLAIN = 0, QMV_DUMP = 1, QMV_PACK = 2, QMV_NORM = 3 };

__host__ __device__ inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

struct SmemLayout {
    int red_off, cnt_off, bar_off, dx_off, bs_off, acts_off, norm_off, total;
};

// Shared memory: ring [stages][stage_bytes] | red f32 [stages][RG][WR][slots] | counters u32
// [stages] | mbarriers u64 [stages] | dx f32 [B][nb] | Q4_K bsums i16 [B][nb][8] | fused form:
// the packed codes i8 [B][K] | RMSNorm form: warp sums of squares f32 [B][8] and 1/rms f32 [B].
// slots: 8, or 16 when a stage has more than 8 (row, vector) pairs per warp.
__host__ __device__ inline SmemLayout qmv_smem_layout(int stages, int stage_bytes, int RG, int WR,
                                                      int B, int nb, bool q6, bool pack = false,
                                                      int slots = 8, bool norm = false)
{
    SmemLayout L;
    int o = stages * stage_bytes;
    L.red_off = o;
    o += stages * RG * WR * slots * 4;
    L.cnt_off = o;
    o = align_up(o + stages * 4, 8);
    L.bar_off = o;
    o += stages * 8;
    L.dx_off = o;
    o = align_up(o + B * nb * 4, 16);
    L.bs_off = o;
    if (!q6)
        o += B * nb * 16;
    o = align_up(o, 16);
    L.acts_off = o;
    if (pack)
        o += B * nb * 256;
    L.norm_off = o;
    if (norm)
        o += B * 9 * 4;
    L.total = align_up(o, 16);
    return L;
}

// Reduce-scatter over the 8 lanes of a block (lane bits 0..2): v[0..P) are this lane's partial
// sums for P slots (P a power of two); on return the lane holds the 8-lane total of slot
// k >> (3 - log2 P).  Integer adds, so the order is immaterial.
template <int P>
__device__ __forceinline__ int reduce_scatter(int (&v)[P], int k)
{
    constexpr int LP = P >= 8 ? 3 : P >= 4 ? 2 : P >= 2 ? 1 : 0;
#pragma unroll
    for (int st = 0; st < LP; ++st) {
        const int half = P >> (st + 1);
        const int m = 4 >> st;
        const bool up = k & m;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const int send = up ? v[i] : v[i + half];
            const int keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
    int s = v[0];
#pragma unroll
    for (int st = LP; st < 3; ++st)
        s += __shfl_xor_sync(0xffffffffu, s, 4 >> st);
    return s;
}

// The same for 16 slots: after the three halving steps lane k holds the 8-lane totals of slots
// 2k and 2k+1 in v[0], v[1].
__device__ __forceinline__ void reduce_scatter16(int (&v)[16], int k)
{
#pragma unroll
    for (int st = 0; st < 3; ++st) {
        const int half = 16 >> (st + 1);
        const int m = 4 >> st;
        const bool up = k & m;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const int send = up ? v[i] : v[i + half];
            const int keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
}

__device__ __forceinline__ int dp4a_chain(const uint4 &w, const uint4 &a)
{
    int s = __dp4a((int)w.x, (int)a.x, 0);
    s = __dp4a((int)w.y, (int)a.y, s);
    s = __dp4a((int)w.z, (int)a.z, s);
    return __dp4a((int)w.w, (int)a.w, s);
}

// Four-way byte dot product with unsigned bytes in a and signed bytes in b.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Dot of the high nibbles of w (left in place, i.e. 16 x code) with a: 16 x the nibble dot.
__device__ __forceinline__ int dp4a_chain_hi16(const uint4 &w, const uint4 &a)
{
    int s = dp4a_us(w.x & 0xF0F0F0F0u, a.x, 0);
    s = dp4a_us(w.y & 0xF0F0F0F0u, a.y, s);
    s = dp4a_us(w.z & 0xF0F0F0F0u, a.z, s);
    return dp4a_us(w.w & 0xF0F0F0F0u, a.w, s);
}

__device__ __forceinline__ int dp4a_chain_lo(const uint4 &w, const uint4 &a)
{
    int s = __dp4a((int)(w.x & 0x0F0F0F0Fu), (int)a.x, 0);
    s = __dp4a((int)(w.y & 0x0F0F0F0Fu), (int)a.y, s);
    s = __dp4a((int)(w.z & 0x0F0F0F0Fu), (int)a.z, s);
    return __dp4a((int)(w.w & 0x0F0F0F0Fu), (int)a.w, s);
}

// Threads a CTA may have: 1024 for one or two vectors with at most 8 (row, vector) slots per
// warp (32 warps cover K = 32768), else 512.  The recording variant keeps the lower bound so
// that it never spills.
__host__ __device__ constexpr int qmv_max_threads(int B, int PR, int mode)
{
    return (B <= 2 && PR * B <= 8 && mode != QMV_DUMP) ? 1024 : 512;
}

// F is the format: QMD_Q4_K, QMD_Q5_K or QMD_Q6_K_SPLIT.
template <int F, int B, int PR, int MODE>
__global__ void __launch_bounds__(qmv_max_threads(B, PR, MODE), 1) qmv_kernel(const QmvKParams p)
{
    constexpr bool Q6 = F == QMD_Q6_K_SPLIT;
    constexpr bool Q5 = F == QMD_Q5_K;
    constexpr bool DUMP = MODE == QMV_DUMP;
    constexpr bool NORM = MODE == QMV_NORM;
    constexpr bool PACK = MODE == QMV_PACK || NORM;  // both pack their activations themselves
    constexpr int P = PR * B;                                               // (row, vector) slots
    static_assert(P >= 1 && P <= 16, "PR x B must be at most 16");
    constexpr int PP = P > 8 ? 16 : P > 4 ? 8 : P > 2 ? 4 : P > 1 ? 2 : 1;  // padded to a power of two
    constexpr int NS = PP > 8 ? 2 : 1;                                      // slots per lane
    constexpr int LP = PP >= 8 ? 3 : PP == 4 ? 2 : PP == 2 ? 1 : 0;
    constexpr int DUP = 8 >> LP;  // lanes of a block holding the same slot
    constexpr int SL = 8 * NS;    // block-group sums per warp per stage
    constexpr int BLOCK_BYTES = Q6 ? 208 : Q5 ? 176 : 144;
    extern __shared__ __align__(128) uint8_t smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int WR = p.WR, RG = p.RG, nb = p.nb;
    const int NWT = WR * RG;  // warps in the CTA
    const int rg = warp / WR, wr = warp - rg * WR;
    const int g = lane >> 3, k = lane & 7;
    const int blk = 4 * wr + g;
    const bool blk_ok = blk < nb;
    const int TR = RG * PR;
    const int64_t r0 = p.rows * (int64_t)blockIdx.x / gridDim.x;
    const int64_t r1 = p.rows * (int64_t)(blockIdx.x + 1) / gridDim.x;
    const int nch = (int)((r1 - r0 + TR - 1) / TR);
    const SmemLayout L = qmv_smem_layout(p.stages, p.stage_bytes, RG, WR, B, nb, Q6, PACK, SL, NORM);
    float *s_red = reinterpret_cast<float *>(smem + L.red_off);
    unsigned *s_cnt = reinterpret_cast<unsigned *>(smem + L.cnt_off);
    const float *s_dx = reinterpret_cast<const float *>(smem + L.dx_off);
    const int16_t *s_bs = reinterpret_cast<const int16_t *>(smem + L.bs_off);
    const uint32_t bar0 = smem_addr(smem + L.bar_off);
    const uint32_t ring0 = smem_addr(smem);
#ifdef QMD_TRACE
    if (tid == 0 && p.trace) {
        p.trace[(size_t)blockIdx.x * QMD_TRACE_FIELDS] = globaltimer_ns();
        p.trace[(size_t)blockIdx.x * QMD_TRACE_FIELDS + 7] =
            (unsigned long long)smid() | ((unsigned long long)blockIdx.x << 16) |
            ((unsigned long long)gridDim.x << 32) | ((unsigned long long)(PACK ? 1 : 2) << 48);
    }
#endif
    // A launch whose plan does not fit the kernel: the RMSNorm form's sum of squares takes 256
    // threads, and the layout must lie inside the dynamic shared memory the launch was given.
    if ((NORM && NWT < 8) || (uint32_t)L.total > dynamic_smem_bytes()) {
        pdl_wait();  // so that a kernel launched after this one still finds its predecessor done
        if (tid == 0)
            atomicOr(p.err, ERRBIT_PLAN);
        return;
    }

    // Stream chunk c (rows r0 + c*TR ..) into stage st = c % stages.  The chunk's rows are one
    // contiguous span of W, copied by as few bulk copies as possible (each issue costs the
    // issuing thread tens of nanoseconds), plus one copy of the rows' Q6_K prefix.
    auto issue = [&](int c, int st) {
        const int64_t rs = r0 + (int64_t)c * TR;
        const int nr = (int)min((int64_t)TR, r1 - rs);
        const uint32_t bar = bar0 + 8u * st;
        const uint32_t body = (uint32_t)(nr * p.row_bytes);
        const uint32_t pre = Q6 ? (uint32_t)(nr * p.pre_bytes) : 0u;
        mbar_arrive_expect_tx(bar, body + pre);
        const uint64_t pol = policy_evict_first();
        const uint32_t dst = ring0 + (uint32_t)(st * p.stage_bytes);
        const uint8_t *src = p.W + rs * p.row_bytes;
        for (uint32_t off = 0; off < body; off += 65536u)
            bulk_copy_g2s(dst + off, src + off, min(65536u, body - off), bar, pol);
        if (Q6)
            bulk_copy_g2s(dst + (uint32_t)(TR * p.row_stride), p.Wpre + rs * p.pre_bytes, pre, bar, pol);
    };

    if (tid == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(bar0 + 8u * i, 1);
            s_cnt[i] = 0;
        }
        fence_barrier_init();
    }
    __syncthreads();
    // the first stages, one per warp (issuing a bulk copy costs its thread tens of ns)
    for (int c = warp; c < min(p.stages, nch); c += NWT)
        if (lane == 0)
            issue(c, c);
    if (tid == 0)
        QMD_STAMP(p, 1);

    pdl_launch_dependents();
    pdl_wait();  // activations come from earlier work in the stream
    if (tid == 0)
        QMD_STAMP(p, 2);

    // ---- this thread's activation slice, for all B vectors (fixed for every row) ----------
    const int64_t K = (int64_t)nb * 256;
    int off_lo;
    if (Q6)
        off_lo = 128 * (k >> 2) + 32 * ((k >> 1) & 1) + 16 * (k & 1);  // group 8hh + 2tl + half
    else
        off_lo = 64 * (k >> 1) + 16 * (k & 1);  // sub-block 2c, half k&1
    constexpr int HI = Q6 ? 64 : 32;            // the high-nibble run sits this far further on
    if (PACK) {
        // Fused form: quantise the B x nb activation blocks into shared memory, one warp per
        // block, with the same arithmetic as the stand-alone pack kernel.
        int8_t *acts = reinterpret_cast<int8_t *>(smem + L.acts_off);
        float *dx = reinterpret_cast<float *>(smem + L.dx_off);
        int16_t *bs = reinterpret_cast<int16_t *>(smem + L.bs_off);
        const bool out = blockIdx.x == 0 && p.xq_qs_out != nullptr;
        float *s_inv = reinterpret_cast<float *>(smem + L.norm_off) + B * 8;  // RMSNorm form: 1/rms
        if (NORM) {
            // RMSNorm of h = x (+ r), each f32 operation rounded alone, the sum of squares in
            // the order the stand-alone RMSNorm pack declares (so the codes are the same): thread
            // t of the first 256 adds the squares of elements t, t + 256, ... left to right; each
            // warp combines its partials by xor-shuffles 16, 8, 4, 2, 1; the eight warp totals
            // are added left to right.  CTA 0 writes h when asked.
            float *s_part = reinterpret_cast<float *>(smem + L.norm_off);
            for (int v = 0; v < B; ++v) {
                if (tid < 256) {
                    const float *xv = p.x + v * K;
                    const float *rv = p.r ? p.r + v * K : nullptr;
                    float *hv = (p.h_out && blockIdx.x == 0) ? p.h_out + v * K : nullptr;
                    float acc = 0.0f;
                    constexpr int U = 8;  // loads in flight per thread per round (registers: 1024-thread bound)
                    for (int64_t i0 = tid; i0 < K; i0 += (int64_t)U * 256) {
                        float xu[U], ru[U];
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            const int64_t i = i0 + (int64_t)u * 256;
                            xu[u] = i < K ? xv[i] : 0.0f;
                            ru[u] = (rv && i < K) ? rv[i] : 0.0f;
                        }
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            const int64_t i = i0 + (int64_t)u * 256;
                            if (i < K) {
                                const float h = rv ? __fadd_rn(xu[u], ru[u]) : xu[u];
                                if (hv)
                                    hv[i] = h;
                                acc = __fadd_rn(acc, __fmul_rn(h, h));
                            }
                        }
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
                    if (lane == 0)
                        s_part[v * 8 + warp] = acc;
                }
            }
            __syncthreads();
            if (tid < B) {
                float total = s_part[tid * 8];
                for (int w = 1; w < 8; ++w)
                    total = __fadd_rn(total, s_part[tid * 8 + w]);
                const float ms = __fdiv_rn(total, (float)K);
                s_inv[tid] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, p.eps)));
            }
            __syncthreads();
        }
        constexpr int QB = NORM ? 1 : 4;  // blocks per warp whose loads are in flight together
        for (int b0 = warp; b0 < B * nb; b0 += QB * NWT) {
            float4 xa[QB], xb[QB];
#pragma unroll
            for (int u = 0; u < QB; ++u) {
                const int b = b0 + u * NWT;
                if (b < B * nb) {
                    const float4 *src = reinterpret_cast<const float4 *>(p.x + (int64_t)b * 256 + 8 * lane);
                    xa[u] = src[0];
                    xb[u] = src[1];
                    if (NORM) {  // n = (h * (1/rms)) * g with h = x (+ r), as the RMSNorm pack does
                        const int v = b / nb, blk_g = b - v * nb;
                        float4 ra = make_float4(0.f, 0.f, 0.f, 0.f), rb = ra;
                        if (p.r) {
                            const float4 *rsrc = reinterpret_cast<const float4 *>(p.r + (int64_t)b * 256 + 8 * lane);
                            ra = rsrc[0];
                            rb = rsrc[1];
                        }
                        const float4 *gsrc = reinterpret_cast<const float4 *>(p.g + blk_g * 256 + 8 * lane);
                        const float4 ga = gsrc[0], gb = gsrc[1];
                        const float inv = s_inv[v];
                        auto nrm = [&](float x, float r, float gg) {
                            const float h = p.r ? __fadd_rn(x, r) : x;
                            return __fmul_rn(__fmul_rn(h, inv), gg);
                        };
                        xa[u] = make_float4(nrm(xa[u].x, ra.x, ga.x), nrm(xa[u].y, ra.y, ga.y), nrm(xa[u].z, ra.z, ga.z),
                                            nrm(xa[u].w, ra.w, ga.w));
                        xb[u] = make_float4(nrm(xb[u].x, rb.x, gb.x), nrm(xb[u].y, rb.y, gb.y), nrm(xb[u].z, rb.z, gb.z),
                                            nrm(xb[u].w, rb.w, gb.w));
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < QB; ++u) {
                const int b = b0 + u * NWT;  // the same for every lane of the warp
                if (b < B * nb) {
                    const float v8[8] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w, xb[u].x, xb[u].y, xb[u].z, xb[u].w};
                    const Q8Block r = q8k_quantise_block(v8);
                    *reinterpret_cast<uint2 *>(acts + b * 256 + 8 * lane) = r.codes;
                    if (!Q6 && (lane & 3) == 0)
                        bs[b * 8 + (lane >> 2)] = (int16_t)r.sum4;
                    if (lane == 0)
                        dx[b] = r.d;
                    if (out) {
                        *reinterpret_cast<uint2 *>(p.xq_qs_out + (int64_t)b * 256 + 8 * lane) = r.codes;
                        if ((lane & 3) == 0)
                            p.xq_bs_out[b * 8 + (lane >> 2)] = (int16_t)r.sum4;
                        if (lane == 0)
                            p.xq_d_out[b] = r.d;
                    }
                }
            }
        }
        __syncthreads();
    }
    const int8_t *act_src = PACK ? reinterpret_cast<const int8_t *>(smem + L.acts_off) : p.xqs;
    uint4 alo[B], ahi[B];
    int xs_lo[B], xs_hi[B];
#pragma unroll
    for (int v = 0; v < B; ++v) {
        if (blk_ok) {
            const int8_t *base = act_src + v * K + 256 * blk + off_lo;
            alo[v] = *reinterpret_cast<const uint4 *>(base);
            ahi[v] = *reinterpret_cast<const uint4 *>(base + HI);
        } else {
            alo[v] = make_uint4(0, 0, 0, 0);
            ahi[v] = make_uint4(0, 0, 0, 0);
        }
        if (Q6) {  // sums of the 16 activation codes, for the -32 offset of Q6_K codes
            const uint4 ones = make_uint4(0x01010101u, 0x01010101u, 0x01010101u, 0x01010101u);
            xs_lo[v] = dp4a_chain(ones, alo[v]);
            xs_hi[v] = dp4a_chain(ones, ahi[v]);
        }
    }
    if (!PACK) {
        float *dx = reinterpret_cast<float *>(smem + L.dx_off);
        for (int i = tid; i < B * nb; i += blockDim.x)
            dx[i] = p.xd[i];
        if (!Q6) {
            int4 *bs = reinterpret_cast<int4 *>(smem + L.bs_off);
            const int4 *src = reinterpret_cast<const int4 *>(p.xbs);
            for (int i = tid; i < B * nb; i += blockDim.x)
                bs[i] = src[i];
        }
    }
    __syncthreads();
    if (tid == 0)
        QMD_STAMP(p, 3);

    // lane constants for reading a block's scales and codes
    const bool hiw = (k >> 1) >= 2;  // Q4_K: sub-blocks 4..7 use the split 6-bit fields
    const uint32_t sel_lo = Q6 ? (uint32_t)(0x4440 | (2 * ((k >> 1) & 1) + (k & 1)))
                               : (uint32_t)(0x4440 | (((k >> 1) & 1) << 1));
    const uint32_t sel_hi = sel_lo + 1;  // Q4_K: the next byte (sub-block 2c+1)
    const int q6_qh_off = 128 + 32 * (k >> 2) + 16 * (k & 1);
    const int q6_sc_off = 192 + 8 * (k >> 2);
    const int q6_sl = 4 - 2 * ((k >> 1) & 1);  // low run: 2-bit field t=tl moved to bits 4..5
    const int q6_sh = 2 * ((k >> 1) & 1);      // high run: field t=tl+2 moved to bits 4..5
    // Q5_K: this lane's fifth bits are bits 2c (low run) and 2c+1 (high run) of the 16 qh
    // bytes 16 (k & 1) ..; a rotation right by these amounts brings each to bit 4 of its byte
    const int q5_rl = (2 * (k >> 1) - 4) & 31, q5_rh = (2 * (k >> 1) - 3) & 31;

    // this lane's slot(s) after the reduce-scatter: k >> (3 - LP), or 2k and 2k+1 for 16
    int slot[NS], spr[NS], sv[NS], srow[NS];
    bool slot_ok[NS];
#pragma unroll
    for (int e = 0; e < NS; ++e) {
        slot[e] = NS == 2 ? 2 * k + e : k >> (3 - LP);
        slot_ok[e] = slot[e] < P;
        spr[e] = slot_ok[e] ? slot[e] / B : PR;
        sv[e] = slot_ok[e] ? slot[e] - (slot[e] / B) * B : 0;
        srow[e] = rg * PR + spr[e];  // the slot's row within the stage
    }

    const unsigned long long wait_ns = p.wait_ns;
    // this chunk's stage (c % stages) and barrier phase ((c / stages) & 1), stepped without a
    // division: an integer division by the runtime ring depth on every chunk cost 4 % of the
    // batch-1 kernel's instructions
    int st = 0;
    uint32_t parity = 0u;
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
        if (!mbar_wait_bounded(bar0 + 8u * st, parity, wait_ns)) {
            // A copy did not land in time: flag it, wait (bounded) for the copies that may
            // still be in flight so that none writes shared memory after the CTA exits, leave.
            if (lane == 0) {
                atomicOr(p.err, ERRBIT_QMV_WAIT);
                for (int cc = c; cc < min(nch, c + p.stages); ++cc)
                    if (!mbar_wait_bounded(bar0 + 8u * (cc % p.stages), (uint32_t)(cc / p.stages) & 1u,
                                           wait_ns)) {
                        atomicOr(p.err, ERRBIT_DRAIN_WAIT);
                        break;
                    }
            }
            __syncwarp();
            return;
        }
        if (c == 0 && tid == 0)
            QMD_STAMP(p, 4);
        const uint8_t *stage = smem + (size_t)st * p.stage_bytes;
        const int64_t rs = r0 + (int64_t)c * TR;
        const int nr = (int)min((int64_t)TR, r1 - rs);

        // ---- integer slice dots, folded with the sub-block scales -------------------------
        // Q4_K partials are carried as 16 x S (the high-nibble dots come out scaled by 16);
        // Q5_K and Q6_K partials are S itself.
        int S[PP];
#pragma unroll
        for (int i = 0; i < PP; ++i)
            S[i] = 0;
        auto row_dots = [&](int i, int pr) {
            const uint8_t *bp = stage + i * p.row_stride + blk * BLOCK_BYTES;
            if (Q5) {
                const uint4 h = lds128(bp);
                const uint4 q = lds128(bp + 48 + 16 * k);
                const uint4 qh = lds128(bp + 16 + 16 * (k & 1));
                const uint32_t scw = hiw ? ((h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u))
                                         : (h.y & 0x3F3F3F3Fu);
                const int sc_lo = (int)__byte_perm(scw, 0u, sel_lo);
                const int sc_hi = (int)__byte_perm(scw, 0u, sel_hi);
                // 5-bit codes, one per byte: the nibble, with the fifth bit OR-ed into bit 4
                uint4 wlo, whi;
                wlo.x = (q.x & 0x0F0F0F0Fu) | (__funnelshift_r(qh.x, qh.x, q5_rl) & 0x10101010u);
                wlo.y = (q.y & 0x0F0F0F0Fu) | (__funnelshift_r(qh.y, qh.y, q5_rl) & 0x10101010u);
                wlo.z = (q.z & 0x0F0F0F0Fu) | (__funnelshift_r(qh.z, qh.z, q5_rl) & 0x10101010u);
                wlo.w = (q.w & 0x0F0F0F0Fu) | (__funnelshift_r(qh.w, qh.w, q5_rl) & 0x10101010u);
                whi.x = ((q.x >> 4) & 0x0F0F0F0Fu) | (__funnelshift_r(qh.x, qh.x, q5_rh) & 0x10101010u);
                whi.y = ((q.y >> 4) & 0x0F0F0F0Fu) | (__funnelshift_r(qh.y, qh.y, q5_rh) & 0x10101010u);
                whi.z = ((q.z >> 4) & 0x0F0F0F0Fu) | (__funnelshift_r(qh.z, qh.z, q5_rh) & 0x10101010u);
                whi.w = ((q.w >> 4) & 0x0F0F0F0Fu) | (__funnelshift_r(qh.w, qh.w, q5_rh) & 0x10101010u);
#pragma unroll
                for (int v = 0; v < B; ++v) {
                    const int dl = dp4a_chain(wlo, alo[v]);
                    const int dh = dp4a_chain(whi, ahi[v]);
                    S[pr * B + v] = sc_lo * dl + sc_hi * dh;
                    if (DUMP) {  // sub-blocks 2c, 2c+1: this lane holds half of each
                        int32_t *dd = p.dbg_dots + ((v * p.rows + rs + i) * nb + blk) * 16;
                        atomicAdd(dd + 2 * (k >> 1), dl);
                        atomicAdd(dd + 2 * (k >> 1) + 1, dh);
                    }
                }
            } else if (!Q6) {
                const uint4 h = lds128(bp);
                const uint4 q = lds128(bp + 16 + 16 * k);
                // this lane's sub-blocks' 6-bit scales (bytes of scw), then the two it needs
                const uint32_t scw = hiw ? ((h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u))
                                         : (h.y & 0x3F3F3F3Fu);
                const int sc_lo = (int)__byte_perm(scw, 0u, sel_lo);
                const int sc_hi = (int)__byte_perm(scw, 0u, sel_hi);
#pragma unroll
                for (int v = 0; v < B; ++v) {
                    const int dl = dp4a_chain_lo(q, alo[v]);
                    const int dh16 = dp4a_chain_hi16(q, ahi[v]);
                    S[pr * B + v] = sc_lo * (dl << 4) + sc_hi * dh16;
                    if (DUMP) {  // sub-blocks 2c, 2c+1: this lane holds half of each
                        int32_t *dd = p.dbg_dots + ((v * p.rows + rs + i) * nb + blk) * 16;
                        atomicAdd(dd + 2 * (k >> 1), dl);
                        atomicAdd(dd + 2 * (k >> 1) + 1, dh16 >> 4);
                    }
                }
            } else {
                const uint4 ql = lds128(bp + 16 * k);
                const uint4 qh = lds128(bp + q6_qh_off);
                const uint2 scw = *reinterpret_cast<const uint2 *>(bp + q6_sc_off);
                const int sc_lo = (int)(int8_t)__byte_perm(scw.x, 0u, sel_lo);
                const int sc_hi = (int)(int8_t)__byte_perm(scw.y, 0u, sel_lo);
                uint4 wlo, whi;  // 6-bit codes of the low / high element runs, one per byte
                wlo.x = (ql.x & 0x0F0F0F0Fu) | ((qh.x << q6_sl) & 0x30303030u);
                wlo.y = (ql.y & 0x0F0F0F0Fu) | ((qh.y << q6_sl) & 0x30303030u);
                wlo.z = (ql.z & 0x0F0F0F0Fu) | ((qh.z << q6_sl) & 0x30303030u);
                wlo.w = (ql.w & 0x0F0F0F0Fu) | ((qh.w << q6_sl) & 0x30303030u);
                whi.x = ((ql.x >> 4) & 0x0F0F0F0Fu) | ((qh.x >> q6_sh) & 0x30303030u);
                whi.y = ((ql.y >> 4) & 0x0F0F0F0Fu) | ((qh.y >> q6_sh) & 0x30303030u);
                whi.z = ((ql.z >> 4) & 0x0F0F0F0Fu) | ((qh.z >> q6_sh) & 0x30303030u);
                whi.w = ((ql.w >> 4) & 0x0F0F0F0Fu) | ((qh.w >> q6_sh) & 0x30303030u);
#pragma unroll
                for (int v = 0; v < B; ++v) {
                    const int dl = dp4a_chain(wlo, alo[v]) - 32 * xs_lo[v];
                    const int dh = dp4a_chain(whi, ahi[v]) - 32 * xs_hi[v];
                    S[pr * B + v] = sc_lo * dl + sc_hi * dh;
                    if (DUMP) {
                        int32_t *dd = p.dbg_dots + ((v * p.rows + rs + i) * nb + blk) * 16;
                        const int s_lo = 8 * (k >> 2) + (k & 3);
                        dd[s_lo] = dl;
                        dd[s_lo + 4] = dh;
                    }
                }
            }
        };
        if (blk_ok) {
            if (nr == TR) {  // full chunk: no per-row predicates
#pragma unroll
                for (int pr = 0; pr < PR; ++pr)
                    row_dots(rg * PR + pr, pr);
            } else {
#pragma unroll
                for (int pr = 0; pr < PR; ++pr)
                    if (rg * PR + pr < nr)
                        row_dots(rg * PR + pr, pr);
            }
        }

        // ---- exact block totals, then this lane's slot epilogue(s) -------------------------
        int Sv[NS];
        if constexpr (NS == 2) {
            reduce_scatter16(S, k);
            Sv[0] = S[0];
            Sv[NS - 1] = S[1];
        } else {
            Sv[0] = reduce_scatter<PP>(S, k);
        }
        float t[NS];
#pragma unroll
        for (int e = 0; e < NS; ++e) {
        t[e] = 0.0f;
        if (blk_ok && slot_ok[e] && srow[e] < nr) {
            const uint8_t *bp = stage + srow[e] * p.row_stride + blk * BLOCK_BYTES;
            const float dx = s_dx[sv[e] * nb + blk];
            const int Sb = (Q6 || Q5) ? Sv[e] : (Sv[e] >> 4);  // exact: Q4_K carried 16 x S
            const float fS = __int2float_rn(Sb);
            int M = 0;
            if (!Q6) {
                const uint4 h = lds128(bp);
                const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xffffu)));
                const float dmin = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
                const uint32_t m0 = h.z & 0x3F3F3F3Fu;
                const uint32_t m1 = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
                const int4 bs = *reinterpret_cast<const int4 *>(s_bs + (sv[e] * nb + blk) * 8);
                M = __dp2a_lo(bs.x, (int)m0, 0);
                M = __dp2a_hi(bs.y, (int)m0, M);
                M = __dp2a_lo(bs.z, (int)m1, M);
                M = __dp2a_hi(bs.w, (int)m1, M);
                const float fM = __int2float_rn(M);
                t[e] = __fmul_rn(dx, __fsub_rn(__fmul_rn(d, fS), __fmul_rn(dmin, fM)));
            } else {
                const unsigned short dbits = *reinterpret_cast<const unsigned short *>(
                    stage + TR * p.row_stride + srow[e] * p.pre_bytes + 2 * blk);
                const float d = __half2float(__ushort_as_half(dbits));
                t[e] = __fmul_rn(dx, __fmul_rn(d, fS));
            }
            if (DUMP && (k & (DUP - 1)) == 0) {
                int32_t *sm = p.dbg_sm + ((sv[e] * p.rows + rs + srow[e]) * nb + blk) * 2;
                sm[0] = Sb;
                sm[1] = M;
            }
        }
        }
        // blocks 4wr .. 4wr+3 of this warp: (t0 + t1) + (t2 + t3)
        float *red = s_red + (size_t)st * RG * WR * SL;
#pragma unroll
        for (int e = 0; e < NS; ++e) {
            float te = __fadd_rn(t[e], __shfl_xor_sync(0xffffffffu, t[e], 8));
            te = __fadd_rn(te, __shfl_xor_sync(0xffffffffu, te, 16));
            if (g == 0)
                red[(rg * WR + wr) * SL + NS * k + e] = te;
        }
        __syncwarp();

        // ---- arrive; the last warp of the stage finishes its rows and refills it -----------
        unsigned last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&s_cnt[st], 1u) == (unsigned)(NWT - 1);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence_block();
            // entry (row group frg, ri) of the warps' group sums: slot ri (16 slots) or
            // ri >> (3 - LP) (kept by DUP lanes, the first one counts).  The group sums (four
            // blocks each) are added in runs of four groups, ((G0 + G1) + G2) + G3 with absent
            // groups as +0, then the runs left to right.
            for (int idx = lane; idx < RG * SL; idx += 32) {
                const int frg = idx / SL, ri = idx - (idx / SL) * SL;
                const int fslot = NS == 2 ? ri : ri >> (3 - LP);
                const int frow = frg * PR + (fslot < P ? fslot / B : PR);
                if ((NS == 2 || (ri & (DUP - 1)) == 0) && fslot < P && frow < nr) {
                    const float *rr = red + (frg * WR) * SL + ri;
                    float acc = 0.0f;
                    for (int w0 = 0; w0 < WR; w0 += 4) {
                        float run = rr[w0 * SL];
                        for (int w = w0 + 1; w < w0 + 4; ++w)
                            run = __fadd_rn(run, w < WR ? rr[w * SL] : 0.0f);
                        acc = w0 == 0 ? run : __fadd_rn(acc, run);
                    }
                    p.y[(fslot - (fslot / B) * B) * p.rows + rs + frow] = acc;
                }
            }
            __syncwarp();
            if (lane == 0) {
                s_cnt[st] = 0;
                if (c + p.stages < nch)
                    issue(c + p.stages, st);  // every warp of the CTA is done with this stage
                if (c == nch - 1)
                    QMD_STAMP(p, 5);
            }
        }
        if (++st == p.stages) {
            st = 0;
            parity ^= 1u;
        }
    }
#ifdef QMD_TRACE
    if (lane == 0 && p.trace)
        atomicMax(p.trace + (size_t)blockIdx.x * QMD_TRACE_FIELDS + 6, globaltimer_ns());
#endif
}

// Launch one kernel instance with the plan's shape: opt in to its shared memory, cap the grid
// at what is resident at once (a persistent grid; rows are split by gridDim), and launch it as
// a programmatic dependent of the previous kernel in the stream.
template <auto Kern, typename Params>
qmd_status launch_kernel(const Params &kp, const QmvPlan &plan, cudaStream_t s)
{
    auto kern = Kern;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return QMD_ERR_DEVICE;
    // Per instance: the shared memory opted in per device, and the resident-CTA count per
    // (device, threads, shared bytes).  Filled on first use; callers may launch from several
    // host threads, so the tables sit behind a lock (launches themselves do not).
    struct Occ {
        int dev, threads, smem, max_ctas;
    };
    static std::mutex mu;
    static int set_bytes[64] = {0};
    static Occ occ[16] = {};
    static int n_occ = 0;
    int cap = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (set_bytes[dev] < plan.smem) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem);
            if (e != cudaSuccess)
                return fail(QMD_ERR_LAUNCH, "qmv smem attribute", e);
            set_bytes[dev] = plan.smem;
        }
        for (int i = 0; i < n_occ && i < 16; ++i)
            if (occ[i].dev == dev && occ[i].threads == plan.threads && occ[i].smem == plan.smem)
                cap = occ[i].max_ctas;
        if (cap == 0) {
            int per_sm = 0, sms = 0;
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, plan.threads, plan.smem);
            if (e != cudaSuccess)
                return fail(QMD_ERR_LAUNCH, "qmv occupancy", e);
            if (per_sm < 1)
                return QMD_ERR_SHAPE;
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            cap = per_sm * sms;
            occ[n_occ % 16] = Occ{dev, plan.threads, plan.smem, cap};
            ++n_occ;
        }
    }
    // Persistent grid: no more CTAs than can be resident at once (rows are split by gridDim).
    // The tensor-core kernel keeps its planned grid, which sized its per-CTA run sums; its
    // CTAs never wait for one another, so any that do not fit at once run later.
    int grid = (plan.grid < cap || plan.tc_rows > 0) ? plan.grid : cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)plan.threads);
    cfg.dynamicSmemBytes = (size_t)plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & LAUNCH_NO_PDL) ? 0 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, kp);
    if (e != cudaSuccess)
        return fail(QMD_ERR_LAUNCH, "qmv launch", e);
    return QMD_OK;
}

template <int F, int B, int PR, int MODE>
qmd_status launch_one(const QmvKParams &kp, const QmvPlan &plan, cudaStream_t s)
{
    return launch_kernel<qmv_kernel<F, B, PR, MODE>>(kp, plan, s);
}

// Rows per stage and row group (PR x B <= 16); the plan picks one.
template <int F, int B, int MODE>
qmd_status launch_rows(const QmvKParams &kp, const QmvPlan &plan, cudaStream_t s)
{
    switch (plan.PR) {
    case 1:
        return launch_one<F, B, 1, MODE>(kp, plan, s);
    case 2:
        if constexpr (2 * B <= 16)
            return launch_one<F, B, 2, MODE>(kp, plan, s);
        break;
    case 4:
        if constexpr (4 * B <= 16)
            return launch_one<F, B, 4, MODE>(kp, plan, s);
        break;
    case 8:
        if constexpr (8 * B <= 16)
            return launch_one<F, B, 8, MODE>(kp, plan, s);
        break;
    }
    return QMD_ERR_SHAPE;
}

// Registers per thread of one instance (the plan sizes CTAs per SM by them); 0 if unknown.
template <int F, int B, int MODE>
int instance_regs(int PR)
{
    cudaFuncAttributes fa{};
    cudaError_t e = cudaErrorInvalidValue;
    switch (PR) {
    case 1:
        e = cudaFuncGetAttributes(&fa, qmv_kernel<F, B, 1, MODE>);
        break;
    case 2:
        if constexpr (2 * B <= 16)
            e = cudaFuncGetAttributes(&fa, qmv_kernel<F, B, 2, MODE>);
        break;
    case 4:
        if constexpr (4 * B <= 16)
            e = cudaFuncGetAttributes(&fa, qmv_kernel<F, B, 4, MODE>);
        break;
    case 8:
        if constexpr (8 * B <= 16)
            e = cudaFuncGetAttributes(&fa, qmv_kernel<F, B, 8, MODE>);
        break;
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return fa.numRegs;
}

template <int F>
int qmv_slice_regs(int batch, int PR, int mode)
{
#define QMD_CASE(BB)                                                                                 \
    case BB:                                                                                         \
        return mode == QMV_PACK   ? instance_regs<F, BB, QMV_PACK>(PR)                               \
               : mode == QMV_NORM ? instance_regs<F, BB, QMV_NORM>(PR)                               \
               : mode == QMV_DUMP ? instance_regs<F, BB, QMV_DUMP>(PR)                               \
                                  : instance_regs<F, BB, QMV_PLAIN>(PR);
    switch (batch) {
        QMD_CASE(1)
        QMD_CASE(2)
        QMD_CASE(3)
        QMD_CASE(4)
        QMD_CASE(5)
        QMD_CASE(6)
        QMD_CASE(7)
        QMD_CASE(8)
    default:
        return 0;
    }
#undef QMD_CASE
}

// Kernel parameters from the call's arguments and the plan; mode is the kernel variant.
inline qmd_status make_params(const QmvArgs &a, const QmvPlan &plan, QmvKParams &kp, int &mode)
{
    kp.W = a.W;
    kp.Wpre = a.Wpre;
    kp.xqs = a.xqs;
    kp.xd = a.xd;
    kp.xbs = a.xbs;
    kp.y = a.y;
    kp.rows = a.rows;
    kp.nb = a.nb;
    kp.batch = a.batch;
    kp.WR = plan.WR;
    kp.RG = plan.RG;
    kp.stages = plan.stages;
    kp.row_bytes = plan.row_bytes;
    kp.pre_bytes = plan.pre_bytes;
    kp.stage_bytes = plan.stage_bytes;
    kp.row_stride = plan.row_stride;
    kp.tc_rows = plan.tc_rows;
    kp.dbg_dots = a.dbg_dots;
    kp.dbg_sm = a.dbg_sm;
    kp.x = a.x;
    kp.xq_qs_out = a.xq_qs_out;
    kp.xq_d_out = a.xq_d_out;
    kp.xq_bs_out = a.xq_bs_out;
    kp.r = a.r;
    kp.g = a.g;
    kp.h_out = a.h_out;
    kp.eps = a.eps;
    kp.err = device_error_word();
    kp.wait_ns = wait_limit_ns();
    // Only the row-lane kernel schedules through the workspace, only for one vector and only
    // where each warp has at least two tiles of its own: a claimed tile costs a round trip to the
    // counter, which pays back only by evening out warps that run several tiles in sequence
    // (measured on the 7B shapes at one vector: gate|up 13.5 -> 12.6 us; q|k|v, o and down, one
    // tile per warp, slower; at two vectors the 8-layer step took 41.9 against 39.4 us a layer).
    const int64_t tiles = (a.rows + 3) / 4;
    const bool deep = plan.layout == 2 && a.batch == 1 && tiles >= 2 * (int64_t)plan.WR * plan.grid;
    kp.ws = deep ? a.ws : nullptr;
    kp.pre_steps = plan.pre_steps;
    kp.dyn_tiles = kp.ws ? dynamic_tiles(tiles) : 0;
    if (kp.dyn_tiles == 0)
        kp.ws = nullptr;
#ifdef QMD_TRACE
    kp.trace = trace_reserve(plan.grid);
#endif
    if (kp.err == nullptr)
        return QMD_ERR_DEVICE;
    mode = a.g != nullptr ? QMV_NORM : a.x != nullptr ? QMV_PACK : a.dbg_dots != nullptr ? QMV_DUMP : QMV_PLAIN;
    return QMD_OK;
}

template <int F>
qmd_status launch_qmv_slice(const QmvKParams &kp, const QmvPlan &plan, int batch, int mode, cudaStream_t s)
{
#define QMD_CASE(BB)                                                                                 \
    case BB:                                                                                         \
        return mode == QMV_PACK   ? launch_rows<F, BB, QMV_PACK>(kp, plan, s)                        \
               : mode == QMV_NORM ? launch_rows<F, BB, QMV_NORM>(kp, plan, s)                        \
               : mode == QMV_DUMP ? launch_rows<F, BB, QMV_DUMP>(kp, plan, s)                        \
                                  : launch_rows<F, BB, QMV_PLAIN>(kp, plan, s);
    switch (batch) {
        QMD_CASE(1)
        QMD_CASE(2)
        QMD_CASE(3)
        QMD_CASE(4)
        QMD_CASE(5)
        QMD_CASE(6)
        QMD_CASE(7)
        QMD_CASE(8)
    default:
        return QMD_ERR_BATCH;
    }
#undef QMD_CASE
}

}  // namespace qmd
