// qmv_tc.cuh -- the decode mat-vec on the tensor cores, for Q4_K, Q5_K and Q6_K (split) rows
// of any length: batches of 5..8 vectors, and rows too long for the dp4a kernel at any batch.
//
// Same computation and the same bits as qmv_kernel (qmv.cuh): integer sub-block dots, the
// per-block rank-one epilogue, the declared row order ("Language models on the device: the
// cajeta-llm kernels", §1, §2.1, §2.2; §2.3 for Q5_K's fifth bit).  What differs is who does
// the multiply-adds.  With several vectors the dp4a form spends most of its instructions on
// per-vector dots, cross-lane reductions and per-slot epilogues; here a warp-wide
// mma.sync.m16n8k16 (f16 inputs, f32 accumulate) multiplies a 16-row x 16-value slice of
// weight codes by the same 16 values of all eight (zero-padded) vectors at once, and the
// cross-lane sum over those 16 values happens inside the instruction.
//
// Exactness.  Every operand is a small integer held exactly in f16: a weight code n (0..15, 0..31
// with Q5_K's fifth bit, 0..63 for Q6_K) enters as 1024 + n (the code's bits in the mantissa of
// 1024; a Q4_K / Q5_K high-nibble code as 1024 + 16 n), an activation code as itself
// (|q| <= 127).  The accumulator starts at -1024 x (the sum of the activation codes the step
// covers) -- for Q6_K at -1056 x that sum, which also takes the codes' -32 offset -- so the step
// leaves the exact integer dot (16 times it for a high nibble): every partial sum is an integer
// below 2^24 in magnitude, whatever order the unit adds in.  The dots leave as exact integers
// and everything after (S, M, the f32 epilogue, the row sum) is the dp4a kernel's arithmetic.
//
// Value order inside a step.  The MMA's k index can be any permutation of the step's 16 values,
// as long as both operands use the same one.  Q4_K / Q5_K (32-value sub-blocks, two steps
// each): lane (g, t) = (lane / 4, lane % 4) takes, of each 32-byte code chunk, the eight bytes
// 8t .. 8t+7 (one 8-byte shared load per row), so step u in {0, 1} covers bytes 8t + 4u + i,
// i = 0, 2 as the MMA's k = 2t, 2t+1 and i = 1, 3 as k = 2t+8, 2t+9.  That order lets one
// masked OR turn two codes of a word into an f16 pair (bytes 0 and 2 of the word, then of the
// word shifted by a byte); a high nibble enters in place, as 16 n, and its sub-block's scale
// carries the 1/16.  Q6_K (16-value sub-blocks, one step
// each): lane t takes values 4t .. 4t+3 of the sub-block, whose low nibbles and high bit pairs
// sit in one 4-byte word of ql and one of qh.
//
// Work split and staging.  A CTA has one warp per block of a run of 16 blocks (fewer for shorter
// rows); warp w owns block 16r + w of every row in run r, and the CTA walks its rows' tiles of
// 16 or 32 rows run by run.  At the start of a run a warp loads, for the whole run, the B
// fragments of vector g over its block's 256 values (32 registers) and the block's per-vector
// constants, and per 16-row MMA sub-tile computes the block term of rows g and g+8 for vectors
// 2t and 2t+1.  Each warp streams its own column (the tile's rows x one block, plus the rows'
// f16 scales for Q6_K) through a private ring of STAGES slots: one tensor copy (TMA) per tile
// and operand, issued by lane 0 and completing on the slot's mbarrier (p.pre_steps slots before
// the dependency wait, the rest once the warp's activation fragments are loaded).  The rows land dense
// (144, 176 or 208 bytes apart), which keeps every fragment load at its minimum number of
// shared-memory wavefronts: the eight rows g of a load start 4, 12 or 20 banks apart.  CTAs take
// whole tiles.
// Warps never wait for each other to refill; they meet only to sum a tile: each posts its block
// terms, and the last to arrive adds the run's terms of every (row, vector) in the declared
// order (groups of four blocks, runs of four groups).  A run that is not the row's last leaves
// its sums in shared memory; the last run's finisher adds the runs left to right and writes y.
#pragma once

#include <cstring>
#include <mutex>

#include <cuda.h>

#include "qmv.cuh"

namespace qmd {

constexpr int TC_ROWS = 16;      // rows per MMA sub-tile (the MMA's M)
constexpr int TC_RED = 3;        // tiles whose block terms can be pending at once
constexpr int TC_RUN = 16;       // blocks per run (warps per CTA at most)
constexpr int TC_MIN_BATCH = 5;  // smallest batch the plan gives to this kernel for rows the dp4a kernel can take,
constexpr int TC_MIN_BATCH_TALL = 3;  // and for many rows a CTA in 32-row tiles (at least TC_TALL_ROWS)
constexpr int TC_TALL_ROWS = 64;

__host__ __device__ constexpr int tc_block_bytes(int fmt)
{
    return fmt == QMD_Q6_K_SPLIT ? 208 : fmt == QMD_Q5_K ? 176 : 144;
}
// Rows per tile: 16, one MMA sub-tile, with rings of 3 or 4 slots per warp; 32, two sub-tiles
// under one copy, one term post and one finisher, with rings of 2 slots (a ring depth of 2 selects
// it).  The taller tile halves the per-tile bookkeeping (the copy's issue, the barrier waits, the
// term post and its arrival count) where it does not give a CTA more rows.
__host__ __device__ constexpr int tc_tile_rows(int stages) { return stages == 2 ? 2 * TC_ROWS : TC_ROWS; }
// a ring slot: the tile's rows of one block, dense as the tensor copy writes them, and for Q6_K
// the rows' 16-byte prefix chunks (eight f16 scales, the block's among them); a multiple of 128
// bytes
__host__ __device__ constexpr int tc_slot_bytes(int fmt, int th = TC_ROWS)
{
    return th * tc_block_bytes(fmt) + (fmt == QMD_Q6_K_SPLIT ? th * 16 : 0);
}
__host__ __device__ constexpr int tc_steps(int fmt) { return fmt == QMD_Q6_K_SPLIT ? 16 : 8; }

struct TcLayout {
    int bar_off, red_off, bias_off, cnt_off, fin_off, done_off, run_off, acts_off, dx_off, bs_off, total;
};

// Shared memory: warp rings [RW][stages][slot] | ring barriers u64 [RW][stages] | block terms f32
// [TC_RED][RW][tile rows][8 vectors]
// | accumulator starts f32 [RW][steps][4 lane columns t][b(2t), b(2t+1), b(2t), b(2t+1)] (each
// lane's C operand as one 16-byte load) | arrival counters u32 [TC_RED] | finished
// tile i32 [TC_RED] | finished runs per row tile i32 [rows_pad / 16] | earlier runs' sums f32
// [runs - 1][rows_pad][8] | fused form only: codes i8 [B][K], d f32 [B][nb], sums i16
// [B][nb][8].  RW = min(nb, 16) warps; rows_pad = the CTA's rows rounded up to the tile rows.
__host__ __device__ inline TcLayout qmv_tc_layout(int stages, int fmt, int nb, int B, bool pack, int rows_pad)
{
    const int RW = nb < TC_RUN ? nb : TC_RUN;
    const int runs = (nb + TC_RUN - 1) / TC_RUN;
    const int th = tc_tile_rows(stages);
    TcLayout L;
    int o = RW * stages * tc_slot_bytes(fmt, th);
    L.bar_off = o;
    o = align_up(o + RW * stages * 8, 16);
    L.red_off = o;
    o += TC_RED * RW * th * 8 * 4;
    L.bias_off = o;
    o += RW * tc_steps(fmt) * 16 * 4;
    L.cnt_off = o;
    o += TC_RED * 4;
    L.fin_off = o;
    o += TC_RED * 4;
    L.done_off = o;
    o = align_up(o + (rows_pad / th) * 4, 16);
    L.run_off = o;
    o += (runs - 1) * rows_pad * 8 * 4;
    L.acts_off = o;
    if (pack)
        o += B * nb * 256;
    L.dx_off = o;
    if (pack)
        o = align_up(o + B * nb * 4, 16);
    L.bs_off = o;
    if (pack && fmt != QMD_Q6_K_SPLIT)
        o += B * nb * 16;
    L.total = align_up(o, 16);
    return L;
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d = a * b + c with c separate (the first step of a sub-block starts from the bias registers)
__device__ __forceinline__ void mma_16816_c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                            float c0, float c1, float c2, float c3)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

// Byte b (0..3) of w as an exact float: the byte under the exponent of 2^23, minus 2^23.
__device__ __forceinline__ float byte_as_float(uint32_t w, uint32_t b)
{
    return __fsub_rn(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | b)), 8388608.0f);
}

// Byte b (0..3) of w over 16 as an exact float: the byte under the exponent of 2^19, whose
// mantissa unit is 1/16, minus 2^19.
__device__ __forceinline__ float byte16th_as_float(uint32_t w, uint32_t b)
{
    return __fsub_rn(__uint_as_float(__byte_perm(w, 0x49000000u, 0x7440u | b)), 524288.0f);
}

// The bits of w under mask M in bytes 0 and 2 (M = 0x000F000F: low nibbles n; 0x00F000F0: high
// nibbles, 16 n) as the f16 pair 1024 + those bits: they sit in the mantissa of 0x6400 (1024,
// unit 1).  One three-input logic operation, (w & M) | k, with k = 0x64006400 held in a register
// (k6400()): written out, the compiler splits it in two.
template <uint32_t M>
__device__ __forceinline__ uint32_t nib_f16x2(uint32_t w, uint32_t k)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "n"(M), "r"(k));
    return r;
}
__device__ __forceinline__ uint32_t k6400()
{
    uint32_t k;
    asm("mov.b32 %0, 0x64006400;" : "=r"(k));
    return k;
}

// Signed byte b (0..3) of w as an exact float: (byte ^ 0x80) is byte + 128 in 0..255 under the
// exponent of 2^23, minus 2^23 + 128.
__device__ __forceinline__ float sbyte_as_float(uint32_t w, uint32_t b)
{
    return __fsub_rn(__uint_as_float(__byte_perm(w ^ 0x80808080u, 0x4B000000u, 0x7440u | b)), 8388736.0f);
}

// Two signed bytes (bytes lo, lo+1 of w) as an exact f16 pair: (byte ^ 0x80) under a 0x64
// exponent byte is 1024 + 128 + q, minus 1152.
__device__ __forceinline__ uint32_t s8x2_to_f16x2(uint32_t w, uint32_t sel)
{
    const uint32_t biased = __byte_perm(w ^ 0x80808080u, 0x64u, sel);
    const __half2 h = __hsub2(*reinterpret_cast<const __half2 *>(&biased), __halves2half2(__ushort_as_half(0x6480u),
                                                                                           __ushort_as_half(0x6480u)));
    return *reinterpret_cast<const uint32_t *>(&h);
}

// An integer-valued float of magnitude below 2^22 as an int: adding 1.5 * 2^23 leaves the
// integer in the low mantissa bits exactly (full-rate add and integer subtract, no conversion).
__device__ __forceinline__ int exact_small_int(float v)
{
    return __float_as_int(__fadd_rn(v, 12582912.0f)) - 0x4B400000;
}

__device__ __forceinline__ uint32_t lds32(const void *p) { return *reinterpret_cast<const uint32_t *>(p); }

// component-wise f32 addition, each rounded alone
__device__ __forceinline__ float4 add4(float4 a, float4 b)
{
    return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}
// A warp that finds its term slot still unsummed sleeps this long between polls, leaving the
// issue slots to the warps doing dot products (measured: polling without a sleep took a fifth
// of the kernel's instructions at batch 8).
constexpr unsigned SPIN_NS = 32;

// The kernel's parameters: the common ones and the tensor maps its copies read through.
struct TcParams {
    QmvKParams k;
    CUtensorMap wmap;    // W as u8 [rows][row_bytes], box: one block's bytes x the tile's rows
    CUtensorMap premap;  // Q6_K prefix as u16 [rows][prefix stride], box: 8 scales x the tile's rows
};

// F is QMD_Q4_K, QMD_Q5_K or QMD_Q6_K_SPLIT; STAGES is the depth of each warp's ring (2: tiles of
// 32 rows, else 16); MULTI walks rows of more than 16 blocks run by run (without it the row is a
// single run and the run bookkeeping compiles away).
template <int F, int MODE, int STAGES, bool MULTI>
__global__ void __launch_bounds__(512, 1) qmv_tc_kernel(const __grid_constant__ TcParams tp)
{
    const QmvKParams &p = tp.k;
    constexpr bool Q6 = F == QMD_Q6_K_SPLIT;
    constexpr bool Q5 = F == QMD_Q5_K;
    constexpr bool DUMP = MODE == QMV_DUMP;
    constexpr bool PACK = MODE == QMV_PACK;
    constexpr int BLOCK_BYTES = tc_block_bytes(F);
    constexpr int RSTRIDE = BLOCK_BYTES;  // rows of a slot
    constexpr int TH = tc_tile_rows(STAGES);  // rows per tile
    constexpr int SUB = TH / TC_ROWS;         // MMA sub-tiles per tile
    constexpr int SLOT = tc_slot_bytes(F, TH);
    constexpr int NSTEP = tc_steps(F);     // accumulator starts per block and vector
    constexpr int QS_OFF = Q5 ? 48 : 16;
    extern __shared__ __align__(128) uint8_t smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nb = p.nb, B = p.batch;
    const int RW = blockDim.x >> 5;  // warps: min(nb, 16)
    const int runs = MULTI ? (nb + TC_RUN - 1) / TC_RUN : 1;
    const int g = lane >> 2, t = lane & 3;
    // rows are split in whole tiles, so only the matrix's last tile is partial (its missing rows
    // arrive as zeros from the tensor copy) and no tile is read by two CTAs
    const int64_t tiles = (p.rows + TH - 1) / TH;
    const int64_t tb0 = tiles * blockIdx.x / gridDim.x, tb1 = tiles * (blockIdx.x + 1) / gridDim.x;
    const int64_t r0 = tb0 * TH, r1 = min(p.rows, tb1 * TH);
    const int nt = (int)(tb1 - tb0);  // row tiles of this CTA
    const int ntot = runs * nt;       // tiles, run by run
    const TcLayout L = qmv_tc_layout(STAGES, F, nb, B, PACK, p.tc_rows);
    uint8_t *ring = smem + (size_t)warp * STAGES * SLOT;
    float *s_red = reinterpret_cast<float *>(smem + L.red_off);
    unsigned *s_cnt = reinterpret_cast<unsigned *>(smem + L.cnt_off);
    volatile int *s_fin = reinterpret_cast<volatile int *>(smem + L.fin_off);
    volatile int *s_done = reinterpret_cast<volatile int *>(smem + L.done_off);
    float *s_run = reinterpret_cast<float *>(smem + L.run_off);
    const uint64_t pol = policy_evict_first();
#ifdef QMD_TRACE
    if (tid == 0 && p.trace) {
        p.trace[(size_t)blockIdx.x * QMD_TRACE_FIELDS] = globaltimer_ns();
        p.trace[(size_t)blockIdx.x * QMD_TRACE_FIELDS + 7] =
            (unsigned long long)smid() | ((unsigned long long)blockIdx.x << 16) |
            ((unsigned long long)gridDim.x << 32) | ((unsigned long long)(PACK ? 1 : 2) << 48);
    }
#endif
    if (runs > 1 && nt * TH > p.tc_rows) {  // more rows than the run-sum buffer was sized for
        pdl_wait();  // so that a kernel launched after this one still finds its predecessor done
        if (tid == 0)
            atomicOr(p.err, ERRBIT_PLAN);
        return;
    }

    // this warp's column of tile T (run T / nt, rows r0 + TH (T % nt) ..) into ring slot
    // T % STAGES: one tensor copy of the tile's rows' block and, for Q6_K, one of the rows' 16-byte
    // prefix chunks holding the block's scale, both completing on the slot's barrier.  Issued
    // by lane 0; a warp copies only the tiles of runs in which it has a block.
    const uint32_t ring0 = smem_addr(ring);
    const uint32_t bar0 = smem_addr(smem + L.bar_off) + 8u * (uint32_t)(warp * STAGES);
    auto copies = [&](int T) { return T < ntot && (MULTI ? T / nt : 0) * TC_RUN + warp < nb; };
    auto issue = [&](int T) {
        if (copies(T)) {
            const int r = MULTI ? T / nt : 0, c = MULTI ? T - r * nt : T;
            const int b = r * TC_RUN + warp;
            const uint32_t st = (uint32_t)(T % STAGES);
            const uint32_t bar = bar0 + 8u * st, dst = ring0 + st * SLOT;
            const int y = (int)(r0 + (int64_t)c * TH);
            mbar_arrive_expect_tx(bar, SLOT);
            tma_load_2d(dst, &tp.wmap, b * BLOCK_BYTES, y, bar, pol);
            if (Q6)
                tma_load_2d(dst + TH * BLOCK_BYTES, &tp.premap, b & ~7, y, bar, pol);
        }
    };
    const unsigned long long wait_ns = p.wait_ns;
    // wait (bounded) for this warp's copies of tiles T0 .. T0 + STAGES - 1 still in flight, so
    // that none lands after the warp has gone
    auto drain = [&](int T0) {
        for (int u = T0; u < T0 + STAGES; ++u)
            if (copies(u))
                (void)mbar_wait_bounded(bar0 + 8u * (uint32_t)(u % STAGES), (uint32_t)(u / STAGES) & 1u, wait_ns);
    };

    if (tid < TC_RED) {
        s_cnt[tid] = 0;
        s_fin[tid] = tid - TC_RED;  // slot tid is free for tile tid
    }
    if (runs > 1)
        for (int i = tid; i < nt; i += blockDim.x)
            s_done[i] = 0;
    if (lane == 0) {
        for (int i = 0; i < STAGES; ++i)
            mbar_init(bar0 + 8u * i, 1);
        fence_barrier_init();
#pragma unroll
        for (int T = 0; T < STAGES; ++T)
            if (T < p.pre_steps)
                issue(T);
    }
    __syncthreads();

    pdl_launch_dependents();
    if (tid == 0)
        QMD_STAMP(p, 1);
    pdl_wait();  // activations come from earlier work in the stream
    if (tid == 0)
        QMD_STAMP(p, 2);

    const int64_t K = (int64_t)nb * 256;
    const int8_t *a_src = p.xqs;
    const float *d_src = p.xd;
    const int16_t *b_src = p.xbs;
    if (PACK) {
        // Fused form: quantise the B x nb activation blocks into shared memory, one warp per
        // block, with the block quantiser of the stand-alone pack kernel.
        int8_t *acts = reinterpret_cast<int8_t *>(smem + L.acts_off);
        float *dx = reinterpret_cast<float *>(smem + L.dx_off);
        int16_t *bs = reinterpret_cast<int16_t *>(smem + L.bs_off);
        const bool out = blockIdx.x == 0 && p.xq_qs_out != nullptr;
        // four blocks' loads in flight per warp, then their four quantisations (a warp packs
        // B x nb / RW blocks: one round trip to L2 per four instead of per block)
        constexpr int PK = 4;
        for (int b0 = warp; b0 < B * nb; b0 += PK * RW) {
            float4 xa[PK], xb[PK];
#pragma unroll
            for (int u = 0; u < PK; ++u) {
                const int b = b0 + u * RW;
                if (b < B * nb) {
                    const float4 *src = reinterpret_cast<const float4 *>(p.x + (int64_t)b * 256 + 8 * lane);
                    xa[u] = src[0];
                    xb[u] = src[1];
                }
            }
#pragma unroll
            for (int u = 0; u < PK; ++u) {
                const int b = b0 + u * RW;  // the same for every lane of the warp
                if (b < B * nb) {
                    const float v8[8] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w, xb[u].x, xb[u].y, xb[u].z, xb[u].w};
                    const Q8Block q = q8k_quantise_block(v8);
                    *reinterpret_cast<uint2 *>(acts + b * 256 + 8 * lane) = q.codes;
                    if (!Q6 && (lane & 3) == 0)
                        bs[b * 8 + (lane >> 2)] = (int16_t)q.sum4;
                    if (lane == 0)
                        dx[b] = q.d;
                    if (out) {
                        *reinterpret_cast<uint2 *>(p.xq_qs_out + (int64_t)b * 256 + 8 * lane) = q.codes;
                        if ((lane & 3) == 0)
                            p.xq_bs_out[b * 8 + (lane >> 2)] = (int16_t)q.sum4;
                        if (lane == 0)
                            p.xq_d_out[b] = q.d;
                    }
                }
            }
        }
        __syncthreads();
        a_src = acts;
        d_src = dx;
        b_src = bs;
    }

    // this lane's operands for the current run, loaded at the run's first tile: B fragments of
    // vector g over the warp's block, and for vectors 2t, 2t+1 the block's scale (and, Q4_K /
    // Q5_K, its eight sub-block sums); the accumulator starts go to the warp's bias table
    uint32_t bfr[32];
    float dxv[2];
    int4 bsv[2];
    float *bias = reinterpret_cast<float *>(smem + L.bias_off) + warp * NSTEP * 16;
    auto load_run = [&](int blk) {
        const bool have = g < B;
        if (Q6) {
            // step s = sub-block s: the lane's values 4t .. 4t+3, one word; the start is
            // -1056 x the sub-block's 16 codes (the 1024 of the code encoding and the -32 offset)
            const int8_t *xv = a_src + (int64_t)g * K + 256 * blk + 4 * t;
#pragma unroll
            for (int s = 0; s < 16; ++s) {
                const uint32_t w = have ? *reinterpret_cast<const uint32_t *>(xv + 16 * s) : 0u;
                bfr[2 * s] = s8x2_to_f16x2(w, 0x4140u);
                bfr[2 * s + 1] = s8x2_to_f16x2(w, 0x4342u);
                int ps = __dp4a((int)w, 0x01010101, 0);
                ps += __shfl_xor_sync(0xffffffffu, ps, 1);
                ps += __shfl_xor_sync(0xffffffffu, ps, 2);
                if (t == 0) {  // vector g's start, in lane column g / 2 of step s
                    float *bq = bias + (s * 4 + (g >> 1)) * 4 + (g & 1);
                    bq[0] = bq[2] = -1056.0f * (float)ps;
                }
            }
        } else {
            // k-step (j, u): the lane's four values of sub-block j are 32j + 8t + 4u + i, i = 0, 2
            // as the MMA's k = 2t, 2t+1 and i = 1, 3 as k = 2t+8, 2t+9, matching the A fragments
            // built below (codes of bytes 0, 2 of a word, then of its bytes 1, 3)
            const int8_t *xv = a_src + (int64_t)g * K + 256 * blk + 8 * t;
            uint2 xw[8];  // the lane's eight bytes of each 32-value sub-block, all loads first
#pragma unroll
            for (int j = 0; j < 8; ++j)
                xw[j] = have ? *reinterpret_cast<const uint2 *>(xv + 32 * j) : make_uint2(0u, 0u);
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint32_t w = u ? xw[j].y : xw[j].x;
                    bfr[4 * j + 2 * u] = s8x2_to_f16x2(w, 0x4240u);      // values 8t + 4u, +2
                    bfr[4 * j + 2 * u + 1] = s8x2_to_f16x2(w, 0x4341u);  // values +1, +3
                }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int v = 2 * t + e;
            if (v < B) {
                dxv[e] = d_src[v * nb + blk];
                bsv[e] = Q6 ? make_int4(0, 0, 0, 0) : *reinterpret_cast<const int4 *>(b_src + (v * nb + blk) * 8);
            } else {
                dxv[e] = 0.0f;
                bsv[e] = make_int4(0, 0, 0, 0);
            }
            if (!Q6) {  // -1024 x the q8_K sub-block sums
                const int s8[8] = {(int)(int16_t)(bsv[e].x & 0xffff), bsv[e].x >> 16, (int)(int16_t)(bsv[e].y & 0xffff),
                                   bsv[e].y >> 16, (int)(int16_t)(bsv[e].z & 0xffff), bsv[e].z >> 16,
                                   (int)(int16_t)(bsv[e].w & 0xffff), bsv[e].w >> 16};
                if (g == 0) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float *bq = bias + (j * 4 + t) * 4 + e;
                        bq[0] = bq[2] = -1024.0f * (float)s8[j];
                    }
                }
            }
        }
        __syncwarp();
    };

    int run_nb = MULTI ? 0 : nb, blk = warp;
    if (!MULTI)
        load_run(warp);
    if (lane == 0)  // the rest of the ring, after the activations are in registers
        for (int T = p.pre_steps; T < STAGES; ++T)
            issue(T);
    if (tid == 0)
        QMD_STAMP(p, 3);
#pragma unroll 1
    for (int T = 0; T < ntot; ++T) {
        const int r = MULTI ? T / nt : 0, c = MULTI ? T - r * nt : T;
        if (MULTI && c == 0) {
            run_nb = min(TC_RUN, nb - r * TC_RUN);
            if (warp >= run_nb)
                break;  // only the last run can be short; this warp has no block in it
            blk = r * TC_RUN + warp;
            load_run(blk);
        }
        // tile T's copies have landed (bounded; the decision is the warp's)
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8u * (uint32_t)(T % STAGES), (uint32_t)(T / STAGES) & 1u,
                                                       wait_ns))) {
            if (lane == 0)
                atomicOr(p.err, ERRBIT_QMV_WAIT);
            drain(T);
            return;
        }
        const int64_t rs0 = r0 + (int64_t)c * TH;  // the tile's first row
        if (T == 0 && tid == 0)
            QMD_STAMP(p, 4);

        // the tile's term slot must have been summed for tile T - TC_RED (bounded wait; the clock
        // is read every 16th poll)
        const int rslot = T % TC_RED;
        int ok = 1;
        if (lane == 0 && s_fin[rslot] != T - TC_RED) {
            const uint64_t t0 = globaltimer_ns();
            for (unsigned n = 1; s_fin[rslot] != T - TC_RED; ++n) {
                __nanosleep(SPIN_NS);
                if ((n & 15) == 0 && globaltimer_ns() - t0 > wait_ns) {
                    ok = 0;
                    atomicOr(p.err, ERRBIT_QMV_WAIT);
                    break;
                }
            }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
            drain(T);  // no copy may land after the warp is gone
            return;
        }
        float *red = s_red + ((size_t)rslot * RW + warp) * TH * 8;
        const uint8_t *slot = ring + (T % STAGES) * SLOT;

#pragma unroll 1
        for (int sub = 0; sub < SUB; ++sub) {
            // rows g and g+8 of MMA sub-tile `sub` (rows past nr hold zeros: computed, never stored)
            const int64_t rs = rs0 + TC_ROWS * sub;
            const int nr = (int)min((int64_t)TC_ROWS, r1 - rs);
            const uint8_t *rowA = slot + (TC_ROWS * sub + g) * RSTRIDE;
            const uint8_t *rowB = rowA + 8 * RSTRIDE;
            int S[2][2] = {{0, 0}, {0, 0}};  // [row A/B][vector 2t / 2t+1]
            float term[2][2];
            if constexpr (Q6) {
                // 16 sub-blocks of 16 values; sum_s sc_s * dot_s in f32 banked to int32 every two
                // sub-blocks: |sc| <= 128 and |dot| <= 16 * 32 * 127, so each partial is an integer
                // below 2^24 and the fused multiply-adds are exact
                const uint4 scA = lds128(rowA + 192), scB = lds128(rowB + 192);
                float Sf[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // [row g v0, v1, g+8 v0, v1]
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // ql words (t6 & 1, half) at 64h + 16 (2 (t6 & 1) + half) + 4t; qh words (half)
                    uint32_t qlA[4], qlB[4], qhA[2], qhB[2];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        qlA[i] = lds32(rowA + 64 * h + 16 * i + 4 * t);
                        qlB[i] = lds32(rowB + 64 * h + 16 * i + 4 * t);
                    }
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        qhA[i] = lds32(rowA + 128 + 32 * h + 16 * i + 4 * t);
                        qhB[i] = lds32(rowB + 128 + 32 * h + 16 * i + 4 * t);
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int s = 8 * h + j, t6 = j >> 1, half = j & 1;
                        const int qi = 2 * (t6 & 1) + half, nsh = 4 * (t6 >> 1), hsh = 2 * t6;
                        // six-bit codes of the lane's four values, one per byte
                        const uint32_t wA = ((qlA[qi] >> nsh) & 0x0F0F0F0Fu) | (((qhA[half] >> hsh) & 0x03030303u) << 4);
                        const uint32_t wB = ((qlB[qi] >> nsh) & 0x0F0F0F0Fu) | (((qhB[half] >> hsh) & 0x03030303u) << 4);
                        const uint32_t a[4] = {__byte_perm(wA, 0x64u, 0x4140u), __byte_perm(wB, 0x64u, 0x4140u),
                                               __byte_perm(wA, 0x64u, 0x4342u), __byte_perm(wB, 0x64u, 0x4342u)};
                        const float4 bb = *reinterpret_cast<const float4 *>(bias + (s * 4 + t) * 4);
                        float d[4];
                        mma_16816_c(d, a, bfr[2 * s], bfr[2 * s + 1], bb.x, bb.y, bb.z, bb.w);
                        // d holds the exact dots [row g: v 2t, 2t+1 | row g+8: v 2t, 2t+1]
                        const uint32_t wsA = s < 4 ? scA.x : s < 8 ? scA.y : s < 12 ? scA.z : scA.w;
                        const uint32_t wsB = s < 4 ? scB.x : s < 8 ? scB.y : s < 12 ? scB.z : scB.w;
                        const float fA = sbyte_as_float(wsA, (uint32_t)(s & 3));
                        const float fB = sbyte_as_float(wsB, (uint32_t)(s & 3));
                        Sf[0] = __fmaf_rn(fA, d[0], Sf[0]);
                        Sf[1] = __fmaf_rn(fA, d[1], Sf[1]);
                        Sf[2] = __fmaf_rn(fB, d[2], Sf[2]);
                        Sf[3] = __fmaf_rn(fB, d[3], Sf[3]);
                        if (j & 1) {  // bank two sub-blocks as int32 (exact)
                            S[0][0] += __float2int_rn(Sf[0]);
                            S[0][1] += __float2int_rn(Sf[1]);
                            S[1][0] += __float2int_rn(Sf[2]);
                            S[1][1] += __float2int_rn(Sf[3]);
                            Sf[0] = Sf[1] = Sf[2] = Sf[3] = 0.0f;
                        }
                        if (DUMP) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int row = g + 8 * (i >> 1), v = 2 * t + (i & 1);
                                if (row < nr && v < B)
                                    p.dbg_dots[((v * p.rows + rs + row) * nb + blk) * 16 + s] = exact_small_int(d[i]);
                            }
                        }
                    }
                }
                // the block's f32 terms: dx * (d * S), d the row's f16 scale from its prefix chunk
                const uint8_t *pre = slot + TH * BLOCK_BYTES;
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int row = g + 8 * rr;
                    const unsigned short hb =
                        *reinterpret_cast<const unsigned short *>(pre + 16 * (TC_ROWS * sub + row) + 2 * (blk & 7));
                    const float d = __half2float(__ushort_as_half(hb));
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        term[rr][e] = __fmul_rn(dxv[e], __fmul_rn(d, __int2float_rn(S[rr][e])));
                        if (DUMP && row < nr && 2 * t + e < B) {
                            int32_t *sm = p.dbg_sm + (((2 * t + e) * p.rows + rs + row) * nb + blk) * 2;
                            sm[0] = S[rr][e];
                            sm[1] = 0;
                        }
                    }
                }
            } else {
                const uint4 hA = lds128(rowA), hB = lds128(rowB);
                // six-bit scales of sub-blocks 0..3 and 4..7, one per byte
                const uint32_t scA0 = hA.y & 0x3F3F3F3Fu, scA1 = (hA.w & 0x0F0F0F0Fu) | ((hA.y >> 2) & 0x30303030u);
                const uint32_t scB0 = hB.y & 0x3F3F3F3Fu, scB1 = (hB.w & 0x0F0F0F0Fu) | ((hB.y >> 2) & 0x30303030u);
                // Q5_K: the fifth bits of this lane's bytes 8t .. 8t+7 of every chunk (bit 2cq, 2cq+1)
                uint2 qhA = make_uint2(0, 0), qhB = make_uint2(0, 0);
                if (Q5) {
                    qhA = *reinterpret_cast<const uint2 *>(rowA + 16 + 8 * t);
                    qhB = *reinterpret_cast<const uint2 *>(rowB + 16 + 8 * t);
                }
                // Q4_K: sum_j sc_j * dot_j in f32 over each half block (sub-blocks 0..3, 4..7): every
                // product and partial sum is an integer of magnitude at most 4 * 63 * 15 * 127 * 32
                // < 2^24, so the f32 fused multiply-adds are exact, and the f32 sum of the two halves
                // is S rounded to f32 once -- the value the epilogue converts S to.  Q5_K (codes up to
                // 31) sums in int32.
                float Sf[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};  // [half][g v0, v1, g+8 v0, v1]
                const uint32_t k64 = k6400();
#pragma unroll
                for (int cq = 0; cq < 4; ++cq) {  // 32-byte code chunk cq: sub-blocks 2cq (low), 2cq+1 (high)
                    float dlo[4], dhi[4];
                    const float4 blo = *reinterpret_cast<const float4 *>(bias + ((2 * cq) * 4 + t) * 4);
                    const float4 bhi = *reinterpret_cast<const float4 *>(bias + ((2 * cq + 1) * 4 + t) * 4);
                    const uint2 cA = *reinterpret_cast<const uint2 *>(rowA + QS_OFF + 32 * cq + 8 * t);
                    const uint2 cB = *reinterpret_cast<const uint2 *>(rowB + QS_OFF + 32 * cq + 8 * t);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        // bytes 8t + 4u + i: values +0, +2 from the word itself, +1, +3 from it shifted
                        // by a byte; low nibbles as 1024 + n, high nibbles as 1024 + 16 n (their dots
                        // come out 16-fold, which the high scale's 1/16 takes back)
                        const uint32_t wA = u ? cA.y : cA.x, wB = u ? cB.y : cB.x;
                        const uint32_t sA = wA >> 8, sB = wB >> 8;
                        uint32_t alo[4] = {nib_f16x2<0x000F000Fu>(wA, k64), nib_f16x2<0x000F000Fu>(wB, k64),
                                           nib_f16x2<0x000F000Fu>(sA, k64), nib_f16x2<0x000F000Fu>(sB, k64)};
                        uint32_t ahi[4] = {nib_f16x2<0x00F000F0u>(wA, k64), nib_f16x2<0x00F000F0u>(wB, k64),
                                           nib_f16x2<0x00F000F0u>(sA, k64), nib_f16x2<0x00F000F0u>(sB, k64)};
                        if (Q5) {
                            // bit 4 of byte i of the rotated fifth-bit words is value +i's fifth bit:
                            // 16 in a low code (f16 bit 4), 256 in a 16-fold high code (f16 bit 8)
                            const uint32_t qA = u ? qhA.y : qhA.x, qB = u ? qhB.y : qhB.x;
                            const int rl = (2 * cq - 4) & 31, rh = (2 * cq - 3) & 31;
                            const uint32_t lA = __funnelshift_r(qA, qA, rl), lB = __funnelshift_r(qB, qB, rl);
                            const uint32_t xA = __funnelshift_r(qA, qA, rh), xB = __funnelshift_r(qB, qB, rh);
                            alo[0] |= lA & 0x00100010u;
                            alo[1] |= lB & 0x00100010u;
                            alo[2] |= (lA >> 8) & 0x00100010u;
                            alo[3] |= (lB >> 8) & 0x00100010u;
                            ahi[0] |= (xA << 4) & 0x01000100u;
                            ahi[1] |= (xB << 4) & 0x01000100u;
                            ahi[2] |= (xA >> 4) & 0x01000100u;
                            ahi[3] |= (xB >> 4) & 0x01000100u;
                        }
                        if (u == 0) {
                            mma_16816_c(dlo, alo, bfr[8 * cq], bfr[8 * cq + 1], blo.x, blo.y, blo.z, blo.w);
                            mma_16816_c(dhi, ahi, bfr[8 * cq + 4], bfr[8 * cq + 5], bhi.x, bhi.y, bhi.z, bhi.w);
                        } else {
                            mma_16816(dlo, alo, bfr[8 * cq + 2], bfr[8 * cq + 3]);
                            mma_16816(dhi, ahi, bfr[8 * cq + 6], bfr[8 * cq + 7]);
                        }
                    }
                    // dlo holds the exact dots, dhi 16 x the exact dots [row g: v 2t, 2t+1 | row g+8: v 2t, 2t+1]
                    const uint32_t wsA = cq < 2 ? scA0 : scA1, wsB = cq < 2 ? scB0 : scB1;
                    const uint32_t bl = 2 * (cq & 1), bh = bl + 1;
                    if (!Q5) {
                        const float fAl = byte_as_float(wsA, bl), fAh = byte16th_as_float(wsA, bh);
                        const float fBl = byte_as_float(wsB, bl), fBh = byte16th_as_float(wsB, bh);
                        float *Sh = Sf[cq >> 1];
                        Sh[0] = __fmaf_rn(fAh, dhi[0], __fmaf_rn(fAl, dlo[0], Sh[0]));
                        Sh[1] = __fmaf_rn(fAh, dhi[1], __fmaf_rn(fAl, dlo[1], Sh[1]));
                        Sh[2] = __fmaf_rn(fBh, dhi[2], __fmaf_rn(fBl, dlo[2], Sh[2]));
                        Sh[3] = __fmaf_rn(fBh, dhi[3], __fmaf_rn(fBl, dlo[3], Sh[3]));
                    } else {
                        const uint32_t sl = 0x4440u | bl, sh = 0x4440u | bh;
                        const int sAl = (int)__byte_perm(wsA, 0u, sl), sAh = (int)__byte_perm(wsA, 0u, sh);
                        const int sBl = (int)__byte_perm(wsB, 0u, sl), sBh = (int)__byte_perm(wsB, 0u, sh);
                        S[0][0] += sAl * exact_small_int(dlo[0]) + sAh * (exact_small_int(dhi[0]) >> 4);
                        S[0][1] += sAl * exact_small_int(dlo[1]) + sAh * (exact_small_int(dhi[1]) >> 4);
                        S[1][0] += sBl * exact_small_int(dlo[2]) + sBh * (exact_small_int(dhi[2]) >> 4);
                        S[1][1] += sBl * exact_small_int(dlo[3]) + sBh * (exact_small_int(dhi[3]) >> 4);
                    }
                    if (DUMP) {
                        int il[4], ih[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            il[i] = exact_small_int(dlo[i]);
                            ih[i] = exact_small_int(dhi[i]) >> 4;
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int row = g + 8 * (i >> 1), v = 2 * t + (i & 1);
                            if (row < nr && v < B) {
                                int32_t *dd = p.dbg_dots + ((v * p.rows + rs + row) * nb + blk) * 16;
                                dd[2 * cq] = il[i];
                                dd[2 * cq + 1] = ih[i];
                            }
                        }
                    }
                }

                // ---- the block's f32 terms for (rows g, g+8) x (vectors 2t, 2t+1) ------------
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const uint4 h = rr ? hB : hA;
                    const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xffffu)));
                    const float dmin = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
                    const uint32_t m0 = h.z & 0x3F3F3F3Fu;
                    const uint32_t m1 = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
                    const int row = g + 8 * rr;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        int M = __dp2a_lo(bsv[e].x, (int)m0, 0);
                        M = __dp2a_hi(bsv[e].y, (int)m0, M);
                        M = __dp2a_lo(bsv[e].z, (int)m1, M);
                        M = __dp2a_hi(bsv[e].w, (int)m1, M);
                        const float fS = Q5 ? __int2float_rn(S[rr][e]) : __fadd_rn(Sf[0][2 * rr + e], Sf[1][2 * rr + e]);
                        term[rr][e] = __fmul_rn(dxv[e], __fsub_rn(__fmul_rn(d, fS), __fmul_rn(dmin, __int2float_rn(M))));
                        if (DUMP && row < nr && 2 * t + e < B) {
                            int32_t *sm = p.dbg_sm + (((2 * t + e) * p.rows + rs + row) * nb + blk) * 2;
                            sm[0] = Q5 ? S[rr][e] : __float2int_rn(Sf[0][2 * rr + e]) + __float2int_rn(Sf[1][2 * rr + e]);
                            sm[1] = M;
                        }
                    }
                }
            }
            // ---- post the sub-tile's terms ----
            float *rsub = red + TC_ROWS * sub * 8;
            *reinterpret_cast<float2 *>(rsub + g * 8 + 2 * t) = make_float2(term[0][0], term[0][1]);
            *reinterpret_cast<float2 *>(rsub + (g + 8) * 8 + 2 * t) = make_float2(term[1][0], term[1][1]);
        }  // sub-tiles
        __syncwarp();  // every lane is done with this ring slot and has posted its terms
        if (lane == 0) {
            fence_proxy_async_smem();  // the warp's reads of the slot before the copy's writes
            issue(T + STAGES);         // refill it with this warp's column of tile T + STAGES
        }

        // ---- the last warp to arrive adds the run's terms of every (row, vector) ----------------
        unsigned last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&s_cnt[rslot], 1u) == (unsigned)(run_nb - 1);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence_block();
            const bool final_run = !MULTI || r == runs - 1;
            if (MULTI && final_run && runs > 1) {  // the tile's earlier runs must have been summed (bounded)
                int ok2 = 1;
                if (lane == 0) {
                    const uint64_t t0 = globaltimer_ns();
                    while (s_done[c] != runs - 1) {
                        if (globaltimer_ns() - t0 > wait_ns) {
                            ok2 = 0;
                            atomicOr(p.err, ERRBIT_QMV_WAIT);
                            break;
                        }
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok2, 0)) {
                    drain(T + 1);
                    return;
                }
                __threadfence_block();
            }
            // declared order: groups of four blocks (t0 + t1) + (t2 + t3), absent blocks +0; a
            // run is ((G0 + G1) + G2) + G3, absent groups +0; the row adds its runs left to right
            const float *base = s_red + (size_t)rslot * RW * TH * 8;
            const int nrt = (int)min((int64_t)TH, r1 - rs0);  // the tile's rows in the matrix
#pragma unroll 1
            for (int sub = 0; sub < SUB; ++sub) {  // lane: row 16 sub + lane / 2, vectors 4 (lane % 2) .. +3
                const int row = TC_ROWS * sub + (lane >> 1), v0 = 4 * (lane & 1);
                if (row < nrt && v0 < B) {
                    const int o = row * 8 + v0;
                    float4 run = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        float4 x4[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            x4[i] = 4 * q4 + i < run_nb ? *reinterpret_cast<const float4 *>(base + (4 * q4 + i) * TH * 8 + o)
                                                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        const float4 G = add4(add4(x4[0], x4[1]), add4(x4[2], x4[3]));
                        run = q4 == 0 ? G : add4(run, G);
                    }
                    const int prow = c * TH + row;  // the row within this CTA
                    if (!final_run) {
                        *reinterpret_cast<float4 *>(s_run + ((size_t)r * p.tc_rows + prow) * 8 + v0) = run;
                    } else {
                        float4 acc = run;
                        if (MULTI && runs > 1) {
                            acc = *reinterpret_cast<const float4 *>(s_run + (size_t)prow * 8 + v0);
                            for (int rp = 1; rp < runs - 1; ++rp)
                                acc = add4(acc, *reinterpret_cast<const float4 *>(s_run + ((size_t)rp * p.tc_rows + prow) * 8 + v0));
                            acc = add4(acc, run);
                        }
                        float *yv = p.y + (int64_t)v0 * p.rows + rs0 + row;
                        const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (v0 + i < B)
                                yv[(int64_t)i * p.rows] = a4[i];
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                s_cnt[rslot] = 0;
                __threadfence_block();
                if (MULTI && !final_run)  // finishers of one row tile's runs may overlap
                    atomicAdd(const_cast<int *>(&s_done[c]), 1);
                s_fin[rslot] = T;
#ifdef QMD_TRACE
                if (final_run && p.trace)
                    atomicMax(p.trace + (size_t)blockIdx.x * QMD_TRACE_FIELDS + 5, globaltimer_ns());
#endif
            }
        }
    }
#ifdef QMD_TRACE
    if (lane == 0 && p.trace)
        atomicMax(p.trace + (size_t)blockIdx.x * QMD_TRACE_FIELDS + 6, globaltimer_ns());
#endif
    // every tile a warp copies it also consumes, so no copy is in flight here
}

template <int F, int STAGES, bool MULTI>
qmd_status launch_tc_stages(const TcParams &tp, const QmvPlan &plan, int mode, cudaStream_t s)
{
    return mode == QMV_PACK   ? launch_kernel<qmv_tc_kernel<F, QMV_PACK, STAGES, MULTI>>(tp, plan, s)
           : mode == QMV_DUMP ? launch_kernel<qmv_tc_kernel<F, QMV_DUMP, STAGES, MULTI>>(tp, plan, s)
                              : launch_kernel<qmv_tc_kernel<F, QMV_PLAIN, STAGES, MULTI>>(tp, plan, s);
}

// The driver's tensor-map encoder, looked up once through the runtime (no link to the driver
// library); NULL if this driver does not provide it.
using TensorMapEncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                       const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                       CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                       CUtensorMapFloatOOBfill);
inline TensorMapEncodeFn tensor_map_encoder()
{
    static TensorMapEncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<TensorMapEncodeFn>(f);
    });
    return fn;
}

// Tensor maps of one call: W as bytes [rows][row_bytes] in boxes of one block x th rows (rows
// past the end read as zeros), and for Q6_K the prefix as u16 [rows][prefix stride] in boxes of
// 8 entries x th rows.  Row pitches are multiples of 16 bytes (144, 176 and 208 are; the prefix
// stride is a multiple of 8 entries), bases 16-byte aligned (checked by the caller).
template <int F>
qmd_status tc_tensor_maps(const QmvKParams &kp, TcParams &tp, int th)
{
    const TensorMapEncodeFn enc = tensor_map_encoder();
    if (!enc)
        return fail(QMD_ERR_LAUNCH, "cuTensorMapEncodeTiled entry point", cudaErrorNotSupported);
    std::memset(&tp.wmap, 0, sizeof tp.wmap);
    std::memset(&tp.premap, 0, sizeof tp.premap);
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t wdim[2] = {(cuuint64_t)kp.row_bytes, (cuuint64_t)kp.rows};
    const cuuint64_t wstr[1] = {(cuuint64_t)kp.row_bytes};
    const cuuint32_t wbox[2] = {(cuuint32_t)tc_block_bytes(F), (cuuint32_t)th};
    if (enc(&tp.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(kp.W), wdim, wstr, wbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return fail(QMD_ERR_LAUNCH, "tensor map of the weights", cudaErrorInvalidValue);
    if (F == QMD_Q6_K_SPLIT) {
        const cuuint64_t pdim[2] = {(cuuint64_t)(kp.pre_bytes / 2), (cuuint64_t)kp.rows};
        const cuuint64_t pstr[1] = {(cuuint64_t)kp.pre_bytes};
        const cuuint32_t pbox[2] = {8, (cuuint32_t)th};
        if (enc(&tp.premap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint8_t *>(kp.Wpre), pdim, pstr, pbox, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return fail(QMD_ERR_LAUNCH, "tensor map of the Q6_K prefix", cudaErrorInvalidValue);
    }
    return QMD_OK;
}

template <int F>
qmd_status launch_qmv_tc(const QmvKParams &kp, const QmvPlan &plan, int mode, cudaStream_t s)
{
    const bool multi = kp.nb > TC_RUN;
    if (mode == QMV_NORM)  // the RMSNorm form is not built in this kernel
        return QMD_ERR_SHAPE;
    TcParams tp;
    tp.k = kp;
    const qmd_status st = tc_tensor_maps<F>(kp, tp, tc_tile_rows(plan.stages));
    if (st != QMD_OK)
        return st;
    switch (plan.stages) {
    case 2:  // 32-row tiles, rows of one run (Q6_K's two-slot rings of them do not fit beside 16 warps)
        if constexpr (F != QMD_Q6_K_SPLIT)
            if (!multi)
                return launch_tc_stages<F, 2, false>(tp, plan, mode, s);
        break;
    case 3:
        return multi ? launch_tc_stages<F, 3, true>(tp, plan, mode, s) : launch_tc_stages<F, 3, false>(tp, plan, mode, s);
    case 4:
        return multi ? launch_tc_stages<F, 4, true>(tp, plan, mode, s) : launch_tc_stages<F, 4, false>(tp, plan, mode, s);
    }
    return QMD_ERR_SHAPE;
}

}  // namespace qmd
