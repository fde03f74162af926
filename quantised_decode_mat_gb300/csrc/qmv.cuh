// qmv.cuh -- the Q4_K / Q6_K x q8_K decode mat-vec kernel (templated on format and batch).
//
// What it computes ("Language models on the device: the cajeta-llm kernels"):
//   §1   integer dot products of weight codes against q8_K activation bytes, with the
//        per-sub-block scales (and Q4_K's mins, through the q8_K sub-block sums) folded in by a
//        rank-one epilogue per 256-value block;
//   §2.1 a reduction over the row's blocks finishes each output row;
//   §2.2 batched decode: one pass over a weight row is dotted against up to 8 vectors.
//
// How, on sm_103a (differs from the pages' wave-per-row design, which had one wave own a row
// and each lane load its own words):
//   * Persistent CTAs, each owning a contiguous range of rows.  A row range is one contiguous
//     span of weight bytes, so it is streamed into a ring of shared-memory stages by 1-D bulk
//     async copies (cp.async.bulk, one elected thread, mbarrier completion), evict-first in
//     L2.  Nothing else is read from HBM in the main loop.
//   * A CTA is RG row groups of WR warps; warp w of a group covers blocks 4w .. 4w+3 of a
//     row and lane (g, k) = (lane/8, lane%8) one 16-byte slice k of block 4w+g.  A thread's
//     slice is the same for every row, so its activation bytes (2 x 16 B per vector) are
//     loaded once into registers and reused across all rows; per row a thread reads 16 B of
//     codes (plus the block header) from shared memory, widens nibbles / 6-bit codes in
//     registers and runs 8 dp4a per vector.
//   * Integer partial sums S of a block (8 lanes) are combined exactly by an 8-lane
//     reduce-scatter over PR rows x B vectors, so each lane ends with one (row, vector)
//     block total and computes that block's f32 epilogue exactly as the oracle states it.
//   * Block terms are summed in f32 by a declared tree: the four blocks of a warp as
//     (t0 + t1) + (t2 + t3) (xor-shuffles 8, 16), then the warps' group sums left to right.
//   * Programmatic dependent launch: the weight stream is started before waiting for the
//     previous kernel in the stream (which produced the activations); everything that reads
//     activations or writes y comes after the wait.
//   * Every pipeline wait is bounded; on give-up the CTA sets the device error word, waits
//     (bounded) for its own copies in flight, and exits.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace qmd {

struct QmvKParams {
    const uint8_t *W;     // Q4_K blocks or Q6_K bodies, [rows][row_bytes]
    const uint8_t *Wpre;  // Q6_K f16 prefix, [rows][pre_bytes]
    const int8_t *xqs;
    const float *xd;
    const int16_t *xbs;
    float *y;
    int64_t rows;
    int nb, WR, RG, stages, row_bytes, pre_bytes, stage_bytes;
    int32_t *dbg_dots;
    int32_t *dbg_sm;
    unsigned *err;
    unsigned long long wait_ns;
};

template <int B>
struct Tiling {
    static constexpr int PR = (8 / B) > 0 ? (8 / B) : 1;  // rows per row group per stage
    static constexpr int P = PR * B;                      // (row, vector) totals per 8 lanes
};

__host__ __device__ inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

struct SmemLayout {
    int dx_off, bs_off, red_off, bar_off, total;
};

// Shared memory: [stages][stage_bytes] ring | dx f32 [B][nb] | bsums i16 [B][nb][8] (Q4_K)
//                | red f32 [2][RG][WR][8] | mbarriers u64 [stages]
__host__ __device__ inline SmemLayout qmv_smem_layout(int stages, int stage_bytes, int B, int nb,
                                                      bool q4k, int RG, int WR)
{
    SmemLayout L;
    int o = stages * stage_bytes;
    L.dx_off = o;
    o = align_up(o + B * nb * 4, 16);
    L.bs_off = o;
    if (q4k)
        o += B * nb * 16;
    L.red_off = o;
    o += 2 * RG * WR * 8 * 4;
    o = align_up(o, 8);
    L.bar_off = o;
    o += stages * 8;
    L.total = align_up(o, 16);
    return L;
}

// 8-lane reduce-scatter (lanes differing in bits 0..2): on return lane k holds the sum over
// the 8 lanes of value index k.  Integer adds, so the order is immaterial.
__device__ __forceinline__ int reduce_scatter8(int (&v)[8], int k)
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool up = k & 4;
        const int send = up ? v[i] : v[i + 4];
        const int keep = up ? v[i + 4] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool up = k & 2;
        const int send = up ? v[i] : v[i + 2];
        const int keep = up ? v[i + 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    const bool up = k & 1;
    const int send = up ? v[0] : v[1];
    const int keep = up ? v[1] : v[0];
    return keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

__device__ __forceinline__ int dp4a_chain(const uint4 &w, const uint4 &a)
{
    int s = __dp4a((int)w.x, (int)a.x, 0);
    s = __dp4a((int)w.y, (int)a.y, s);
    s = __dp4a((int)w.z, (int)a.z, s);
    return __dp4a((int)w.w, (int)a.w, s);
}

template <bool Q6, int B, bool DUMP>
__global__ void __launch_bounds__(B <= 2 ? 1024 : 512, 1) qmv_kernel(const QmvKParams p)
{
    constexpr int PR = Tiling<B>::PR;
    constexpr int P = Tiling<B>::P;
    constexpr int BLOCK_BYTES = Q6 ? 208 : 144;
    extern __shared__ __align__(128) uint8_t smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int WR = p.WR, RG = p.RG, nb = p.nb;
    const int rg = warp / WR, wr = warp - rg * WR;
    const int g = lane >> 3, k = lane & 7;
    const int blk = 4 * wr + g;
    const bool blk_ok = blk < nb;
    const int TR = RG * PR;
    const int64_t r0 = p.rows * (int64_t)blockIdx.x / gridDim.x;
    const int64_t r1 = p.rows * (int64_t)(blockIdx.x + 1) / gridDim.x;
    const int nch = (int)((r1 - r0 + TR - 1) / TR);
    const SmemLayout L = qmv_smem_layout(p.stages, p.stage_bytes, B, nb, !Q6, RG, WR);
    const float *s_dx = reinterpret_cast<const float *>(smem + L.dx_off);
    const int16_t *s_bs = reinterpret_cast<const int16_t *>(smem + L.bs_off);
    float *s_red = reinterpret_cast<float *>(smem + L.red_off);
    const uint32_t bar0 = smem_addr(smem + L.bar_off);
    const uint32_t ring0 = smem_addr(smem);

    // Stream chunk c (rows r0 + c*TR ..) into stage c % stages.
    auto issue = [&](int c) {
        const int st = c % p.stages;
        const int64_t rs = r0 + (int64_t)c * TR;
        const int nr = (int)min((int64_t)TR, r1 - rs);
        const uint32_t bar = bar0 + 8u * st;
        const uint32_t body = (uint32_t)nr * (uint32_t)p.row_bytes;
        const uint32_t pre = Q6 ? (uint32_t)nr * (uint32_t)p.pre_bytes : 0u;
        mbar_arrive_expect_tx(bar, body + pre);
        const uint64_t pol = policy_evict_first();
        const uint8_t *src = p.W + rs * p.row_bytes;
        const uint32_t dst = ring0 + (uint32_t)st * (uint32_t)p.stage_bytes;
#pragma unroll 1
        for (uint32_t off = 0; off < body; off += 16384u)
            bulk_copy_g2s(dst + off, src + off, min(16384u, body - off), bar, pol);
        if (Q6)
            bulk_copy_g2s(dst + (uint32_t)TR * (uint32_t)p.row_bytes, p.Wpre + rs * p.pre_bytes, pre,
                          bar, pol);
    };

    if (tid == 0) {
        for (int i = 0; i < p.stages; ++i)
            mbar_init(bar0 + 8u * i, 1);
        fence_barrier_init();
        const int first = min(p.stages, nch);
        for (int c = 0; c < first; ++c)
            issue(c);
    }
    __syncthreads();

    pdl_launch_dependents();
    pdl_wait();  // activations come from earlier work in the stream

    // ---- this thread's activation slice, for all B vectors (fixed for every row) ----------
    const int64_t K = (int64_t)nb * 256;
    int off_lo;
    if (Q6) {
        const int hh = k >> 2, tl = (k >> 1) & 1, half = k & 1;
        off_lo = 128 * hh + 32 * tl + 16 * half;  // elements of group 8hh + 2tl + half
    } else {
        off_lo = 64 * (k >> 1) + 16 * (k & 1);  // elements of sub-block 2c, half k&1
    }
    constexpr int HI = Q6 ? 64 : 32;  // the high-nibble elements sit this far further on
    uint4 alo[B], ahi[B];
    int xs_lo[B], xs_hi[B];
#pragma unroll
    for (int v = 0; v < B; ++v) {
        if (blk_ok) {
            const int8_t *base = p.xqs + v * K + 256 * blk + off_lo;
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
    {
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

    const unsigned long long wait_ns = p.wait_ns;
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
        const int st = c % p.stages;
        const uint32_t parity = (uint32_t)(c / p.stages) & 1u;
        const bool ok = mbar_wait_bounded(bar0 + 8u * st, parity, wait_ns);
        const uint8_t *stage = smem + (size_t)st * p.stage_bytes;
        const int64_t rs = r0 + (int64_t)c * TR;
        const int nr = (int)min((int64_t)TR, r1 - rs);

        // ---- integer slice dots, folded with the sub-block scales -------------------------
        int S[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            S[i] = 0;
#pragma unroll
        for (int pr = 0; pr < PR; ++pr) {
            const int i = rg * PR + pr;
            if (blk_ok && i < nr) {
                const uint8_t *bp = stage + i * p.row_bytes + blk * BLOCK_BYTES;
                int sc_lo, sc_hi;
                uint4 wlo, whi;  // codes of the low / high element runs, one byte each
                if (!Q6) {
                    const uint4 h = lds128(bp);
                    const uint4 q = lds128(bp + 16 + 16 * k);
                    const int c2 = k >> 1;
                    const uint32_t scw = c2 < 2 ? (h.y & 0x3F3F3F3Fu)
                                                : ((h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u));
                    const int sh = (c2 & 1) << 4;
                    sc_lo = (scw >> sh) & 0xff;
                    sc_hi = (scw >> (sh + 8)) & 0xff;
                    wlo = make_uint4(q.x & 0x0F0F0F0Fu, q.y & 0x0F0F0F0Fu, q.z & 0x0F0F0F0Fu,
                                     q.w & 0x0F0F0F0Fu);
                    whi = make_uint4((q.x >> 4) & 0x0F0F0F0Fu, (q.y >> 4) & 0x0F0F0F0Fu,
                                     (q.z >> 4) & 0x0F0F0F0Fu, (q.w >> 4) & 0x0F0F0F0Fu);
                } else {
                    const int hh = k >> 2, tl = (k >> 1) & 1, half = k & 1;
                    const uint4 ql = lds128(bp + 16 * k);
                    const uint4 qh = lds128(bp + 128 + 32 * hh + 16 * half);
                    const uint2 scw = *reinterpret_cast<const uint2 *>(bp + 192 + 8 * hh);
                    const int sb = 8 * (2 * tl + half);
                    sc_lo = (int)(int8_t)(scw.x >> sb);
                    sc_hi = (int)(int8_t)(scw.y >> sb);
                    const int slo = 2 * tl, shi = 2 * tl + 4;
                    wlo = make_uint4((ql.x & 0x0F0F0F0Fu) | (((qh.x >> slo) & 0x03030303u) << 4),
                                     (ql.y & 0x0F0F0F0Fu) | (((qh.y >> slo) & 0x03030303u) << 4),
                                     (ql.z & 0x0F0F0F0Fu) | (((qh.z >> slo) & 0x03030303u) << 4),
                                     (ql.w & 0x0F0F0F0Fu) | (((qh.w >> slo) & 0x03030303u) << 4));
                    whi = make_uint4(((ql.x >> 4) & 0x0F0F0F0Fu) | (((qh.x >> shi) & 0x03030303u) << 4),
                                     ((ql.y >> 4) & 0x0F0F0F0Fu) | (((qh.y >> shi) & 0x03030303u) << 4),
                                     ((ql.z >> 4) & 0x0F0F0F0Fu) | (((qh.z >> shi) & 0x03030303u) << 4),
                                     ((ql.w >> 4) & 0x0F0F0F0Fu) | (((qh.w >> shi) & 0x03030303u) << 4));
                }
#pragma unroll
                for (int v = 0; v < B; ++v) {
                    int dl = dp4a_chain(wlo, alo[v]);
                    int dh = dp4a_chain(whi, ahi[v]);
                    if (Q6) {
                        dl -= 32 * xs_lo[v];
                        dh -= 32 * xs_hi[v];
                    }
                    S[pr * B + v] = sc_lo * dl + sc_hi * dh;
                    if (DUMP) {
                        int32_t *dd = p.dbg_dots + ((v * p.rows + rs + i) * nb + blk) * 16;
                        if (Q6) {
                            const int s_lo = 8 * (k >> 2) + (k & 3);
                            dd[s_lo] = dl;
                            dd[s_lo + 4] = dh;
                        } else {
                            dd[2 * k] = dl;
                            dd[2 * k + 1] = dh;
                        }
                    }
                }
            }
        }

        // ---- exact block totals, then this lane's block epilogue --------------------------
        const int Sv = reduce_scatter8(S, k);
        float t = 0.0f;
        if (k < P) {
            const int pr = k / B, v = k - pr * B;
            const int i = rg * PR + pr;
            if (blk_ok && i < nr) {
                const uint8_t *bp = stage + i * p.row_bytes + blk * BLOCK_BYTES;
                const float dx = s_dx[v * nb + blk];
                const float fS = __int2float_rn(Sv);
                int M = 0;
                if (!Q6) {
                    const uint4 h = lds128(bp);
                    const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xffffu)));
                    const float dmin = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
                    const uint32_t m0 = h.z & 0x3F3F3F3Fu;
                    const uint32_t m1 = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
                    const int4 bs = *reinterpret_cast<const int4 *>(s_bs + (v * nb + blk) * 8);
                    M = __dp2a_lo(bs.x, (int)m0, 0);
                    M = __dp2a_hi(bs.y, (int)m0, M);
                    M = __dp2a_lo(bs.z, (int)m1, M);
                    M = __dp2a_hi(bs.w, (int)m1, M);
                    const float fM = __int2float_rn(M);
                    t = __fmul_rn(dx, __fsub_rn(__fmul_rn(d, fS), __fmul_rn(dmin, fM)));
                } else {
                    const unsigned short dbits = *reinterpret_cast<const unsigned short *>(
                        stage + TR * p.row_bytes + i * p.pre_bytes + 2 * blk);
                    const float d = __half2float(__ushort_as_half(dbits));
                    t = __fmul_rn(dx, __fmul_rn(d, fS));
                }
                if (DUMP) {
                    int32_t *sm = p.dbg_sm + ((v * p.rows + rs + i) * nb + blk) * 2;
                    sm[0] = Sv;
                    sm[1] = M;
                }
            }
        }
        // blocks 4wr .. 4wr+3 of this warp: (t0 + t1) + (t2 + t3)
        t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 8));
        t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 16));
        const int buf = c & 1;
        if (g == 0 && k < P)
            s_red[((buf * RG + rg) * WR + wr) * 8 + k] = t;

        if (__syncthreads_or(!ok)) {
            // A copy did not land in time: flag it, wait (bounded) for this CTA's copies still
            // in flight so none writes shared memory after exit, and leave.
            if (tid == 0) {
                atomicOr(p.err, ERRBIT_QMV_WAIT);
                const int last = min(nch, c + p.stages);
                for (int cc = c; cc < last; ++cc) {
                    if (!mbar_wait_bounded(bar0 + 8u * (cc % p.stages), (uint32_t)(cc / p.stages) & 1u,
                                           wait_ns)) {
                        atomicOr(p.err, ERRBIT_DRAIN_WAIT);
                        break;
                    }
                }
            }
            return;
        }
        if (tid == 0 && c + p.stages < nch)
            issue(c + p.stages);  // every thread is done with this stage

        // ---- row totals: the warps' group sums, left to right ------------------------------
        if (wr == 0 && g == 0 && k < P) {
            const int pr = k / B, v = k - pr * B;
            const int i = rg * PR + pr;
            if (i < nr) {
                const float *red = s_red + ((buf * RG + rg) * WR) * 8 + k;
                float acc = red[0];
                for (int w = 1; w < WR; ++w)
                    acc = __fadd_rn(acc, red[w * 8]);
                p.y[v * p.rows + rs + i] = acc;
            }
        }
    }
}

template <bool Q6, int B, bool DUMP>
qmd_status launch_one(const QmvKParams &kp, const QmvPlan &plan, cudaStream_t s)
{
    auto kern = qmv_kernel<Q6, B, DUMP>;
    // opt in to the shared memory this launch needs (cached per device)
    static int set_bytes[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64)
        return QMD_ERR_DEVICE;
    if (set_bytes[dev] < plan.smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem);
        if (e != cudaSuccess)
            return fail(QMD_ERR_LAUNCH, "qmv smem attribute", e);
        set_bytes[dev] = plan.smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid);
    cfg.blockDim = dim3((unsigned)plan.threads);
    cfg.dynamicSmemBytes = (size_t)plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, kp);
    if (e != cudaSuccess)
        return fail(QMD_ERR_LAUNCH, "qmv launch", e);
    return QMD_OK;
}

template <bool Q6>
qmd_status launch_qmv(const QmvArgs &a, const QmvPlan &plan, cudaStream_t s)
{
    QmvKParams kp;
    kp.W = a.W;
    kp.Wpre = a.Wpre;
    kp.xqs = a.xqs;
    kp.xd = a.xd;
    kp.xbs = a.xbs;
    kp.y = a.y;
    kp.rows = a.rows;
    kp.nb = a.nb;
    kp.WR = plan.WR;
    kp.RG = plan.RG;
    kp.stages = plan.stages;
    kp.row_bytes = plan.row_bytes;
    kp.pre_bytes = plan.pre_bytes;
    kp.stage_bytes = plan.stage_bytes;
    kp.dbg_dots = a.dbg_dots;
    kp.dbg_sm = a.dbg_sm;
    kp.err = device_error_word();
    kp.wait_ns = wait_limit_ns();
    if (kp.err == nullptr)
        return QMD_ERR_DEVICE;
    const bool dump = a.dbg_dots != nullptr;
#define QMD_CASE(BB)                                                                   \
    case BB:                                                                           \
        return dump ? launch_one<Q6, BB, true>(kp, plan, s) : launch_one<Q6, BB, false>(kp, plan, s);
    switch (a.batch) {
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
