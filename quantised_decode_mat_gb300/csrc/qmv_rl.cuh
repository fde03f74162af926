// qmv_rl.cuh -- the decode mat-vec with one lane per whole block-row, for Q4_K, Q5_K and Q6_K
// (split) weights and one to four activation vectors.
//
// Same computation and the same bits as qmv_kernel (qmv.cuh) and qmv_tc_kernel: integer
// sub-block dots against q8_K codes, the per-block rank-one epilogue, the declared row order
// ("Language models on the device: the cajeta-llm kernels", §1, §2.1, §2.2; §2.3 for Q5_K's
// fifth bit).  What differs is the work split, chosen to spend as few instructions as possible
// on each weight byte.
//
// At one vector the other kernels give each block-row to several lanes (8 lanes of 16 bytes, or
// a warp-wide MMA), so every lane decodes the block header again, the lanes' integers must be
// combined by shuffles and each (block, row) needs its own epilogue slot: about 20 warp
// instructions per 144-byte block-row, which left the batch-1 mat-vec bound by instruction
// issue almost as much as by HBM.  Here a lane owns a whole block-row: it reads the header once,
// runs the 64 dp4a of the block against activation codes broadcast from shared memory, and
// evaluates the block's epilogue itself -- about 6 warp instructions per block-row.
//
// Work split.  Lane (r, g) = (lane / 16, lane % 16) takes row r of a 2-row tile and block 16s + g
// of step s, so one warp step covers 2 rows x 16 blocks: one run of the declared row order.  A
// warp owns whole rows: it walks all steps of each of its tiles and sums the row's terms in
// registers in the declared order -- blocks in groups of four, (t0 + t1) + (t2 + t3) by two
// xor-shuffles inside each quarter of the 16 lanes of a row; the run's four groups, ((G0 + G1) +
// G2) + G3; runs left to right -- so warps never wait for each other after the activations are
// in place.  CTAs (one per SM) take contiguous ranges of tiles, and warps take every W-th tile
// of it.  (Tiles of 4 rows x 8 blocks gave the short 4096-row projections only ~7 warps per SM,
// whose compute then set their time.)
//
// Staging.  Each warp streams its own steps through a private ring of S slots: lane 0 issues one
// 3-D tensor copy (TMA) per step -- the box is (block bytes, 8 blocks, 4 rows) of the weight
// tensor viewed as [rows][nb][block bytes] -- plus, for Q6_K, a 2-D copy of the 2 rows' 32-byte
// chunks of the scale prefix; both complete on the slot's mbarrier.  The box lands as [2 rows]
// [16 blocks][block bytes]: with 144, 176 or 208-byte blocks a 16-byte load by the 32 lanes hits
// each group of four banks exactly four times, the minimum for 512 bytes.  Blocks and rows past
// the tensor's end read as zeros (their lanes skip the work and add +0).  A producer warp
// requests the first ring fills around the programmatic-launch wait (weights only).  Activation
// codes sit in shared memory 272 bytes apart per block, so the 16 blocks a warp reads at once
// spread evenly over the bank groups and each 16-byte load takes the minimum two wavefronts.
#pragma once

#include "qmv_tc.cuh"

namespace qmd {

constexpr int RL_ROWS = 2;        // rows per tile (lane bit 4)
constexpr int RL_BLOCKS = 16;     // blocks per step, one run of the row order (lane bits 0..3)
constexpr int RL_ACT = 272;       // shared-memory bytes per activation block: 256 codes + 16 pad
constexpr int RL_MAX_WARPS = 16;  // warps that own rings, and warps that pack
// Ring / packing warps a CTA may have for B vectors: 16 for one or two, 8 above (so that the
// larger per-lane state of three and four vectors fits in registers), plus the warp that
// requests the first ring fills.
__host__ __device__ constexpr int rl_max_warps(int B) { return B <= 2 ? RL_MAX_WARPS : 12; }
__host__ __device__ constexpr int rl_max_threads(int B) { return 32 * (rl_max_warps(B) + 1); }
constexpr int RL_MAX_BATCH = 4;   // vectors per launch
constexpr int RL_DEFAULT_BATCH = 2;  // the plan's default for at most this many vectors
constexpr int RL_POOLS = 8;          // claim pools of the scheduling workspace (CTA b draws from pool b % 8)
constexpr int RL_WS_STRIDE = 64;     // words between the workspace's counters (256 bytes: separate L2 lines)
static_assert(RL_WS_STRIDE * (RL_POOLS + 1) * 4 <= QMD_WORKSPACE_BYTES, "the pools' counters and the done word");
constexpr int RL_PRE_STEPS = 2;   // default ring slots per warp requested before the dependency wait
constexpr int RL_FEW_TILES = 32;  // a one-vector launch with at most this many tiles per CTA requests one

__host__ __device__ constexpr int rl_block_bytes(int f) { return f == QMD_Q6_K_SPLIT ? 208 : f == QMD_Q5_K ? 176 : 144; }
__host__ __device__ constexpr int rl_box_bytes(int f) { return RL_ROWS * RL_BLOCKS * rl_block_bytes(f); }
// bytes one step's copies complete on its barrier: the box, and the Q6_K prefix chunks
__host__ __device__ constexpr int rl_tx_bytes(int f) { return rl_box_bytes(f) + (f == QMD_Q6_K_SPLIT ? RL_ROWS * RL_BLOCKS * 2 : 0); }
// a ring slot, a multiple of 128 bytes: the box, then (Q6_K) the prefix chunks
__host__ __device__ constexpr int rl_slot_bytes(int f) { return rl_box_bytes(f) + (f == QMD_Q6_K_SPLIT ? 128 : 0); }

struct RlLayout {
    int bar_off, tile_off, sched_off, act_off, dx_off, aux_off, norm_off, total;
};

// Shared memory: rings [W][S][slot] | mbarriers u64 [W][S] | the tile of each slot's step i32
// [W][S] | activation codes i8 [B][nb][272] | block scales f32 [B][nb] | Q4_K, Q5_K: sums i16
// [B][nb][8] of each 32 codes; Q6_K: sums i16 [B][nb][16] of each 16 codes (for the -32 offset
// of the weight codes) | RMSNorm form: warp sums of squares f32 [B][8] and 1/rms f32 [B].
__host__ __device__ inline RlLayout qmv_rl_layout(int f, int W, int S, int B, int nb, bool norm = false)
{
    RlLayout L;
    int o = W * S * rl_slot_bytes(f);
    L.bar_off = o;
    o += W * S * 8;
    L.tile_off = o;
    o += W * S * 4;
    L.sched_off = o;  // two words: the CTA's pool is empty; warps done claiming
    o = align_up(o + 8, 16);
    L.act_off = o;
    o += B * nb * RL_ACT;
    L.dx_off = o;
    o = align_up(o + B * nb * 4, 16);
    L.aux_off = o;
    o += B * nb * (f == QMD_Q6_K_SPLIT ? 32 : 16);
    L.norm_off = o;
    if (norm)
        o += B * 9 * 4;
    L.total = align_up(o, 16);
    return L;
}

struct RlParams {
    QmvKParams k;        // k.WR: warps with a ring (the others only pack); k.stages: ring slots per warp
    CUtensorMap wmap;    // W as u8 [rows][nb][block bytes], box: block bytes x 16 blocks x 2 rows
    CUtensorMap premap;  // Q6_K prefix as u16 [rows][prefix stride], box: 16 scales x 2 rows
};

// Byte b of w, sign-extended (a signed bit-field extract).
__device__ __forceinline__ int sbyte(uint32_t w, int b)
{
    int r;
    asm("bfe.s32 %0, %1, %2, 8;" : "=r"(r) : "r"(w), "r"(8 * b));
    return r;
}

__device__ __forceinline__ int dp4a4(const uint4 &w, const uint4 &a, int c)
{
    c = __dp4a((int)w.x, (int)a.x, c);
    c = __dp4a((int)w.y, (int)a.y, c);
    c = __dp4a((int)w.z, (int)a.z, c);
    return __dp4a((int)w.w, (int)a.w, c);
}

__device__ __forceinline__ int dp4a4_us(const uint4 &w, const uint4 &a, int c)
{
    c = dp4a_us(w.x, a.x, c);
    c = dp4a_us(w.y, a.y, c);
    c = dp4a_us(w.z, a.z, c);
    return dp4a_us(w.w, a.w, c);
}

__device__ __forceinline__ uint4 and4(const uint4 &w, uint32_t m)
{
    return make_uint4(w.x & m, w.y & m, w.z & m, w.w & m);
}

// The block terms of one block-row for the B vectors: this lane's row `row` (< rows when
// `live`), block blk, weight bytes at bp (in the box), activation codes of block blk at act
// (vector v at act + v * nb * RL_ACT), the block scales sdx [B][nb] and code sums saux, the
// Q6_K scale d as f16 bits.
template <int F, int B, bool DUMP>
__device__ __forceinline__ void rl_block_terms(const uint8_t *bp, const int8_t *act, const float *sdx,
                                               const int16_t *saux, int nb, int blk, unsigned short q6_d,
                                               const QmvKParams &p, int64_t row, bool live, float (&t)[B])
{
    constexpr bool Q6 = F == QMD_Q6_K_SPLIT;
    constexpr bool Q5 = F == QMD_Q5_K;
    const size_t vstride = (size_t)nb * RL_ACT;
    if constexpr (!Q6) {
        const uint4 h = lds128(bp);
        const uint32_t sc03 = h.y & 0x3F3F3F3Fu, m03 = h.z & 0x3F3F3F3Fu;
        const uint32_t sc47 = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
        const uint32_t m47 = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
        uint4 qh0, qh1;  // Q5_K: fifth bits of values t and 32 + t of each 64, t < 16 / t >= 16
        if (Q5) {
            qh0 = lds128(bp + 16);
            qh1 = lds128(bp + 32);
        }
        constexpr int CODES = Q5 ? 48 : 16;
        int Slo[B], Shi[B];
#pragma unroll
        for (int v = 0; v < B; ++v)
            Slo[v] = Shi[v] = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            // code bytes 32c .. 32c+31: low nibbles are values 64c + t, high nibbles 64c + 32 + t
            const uint4 qa = lds128(bp + CODES + 32 * c), qb = lds128(bp + CODES + 16 + 32 * c);
            uint4 la, lb, ha, hb;
            if (Q5) {
                // bit 2c (low run) or 2c + 1 (high run) of each fifth-bit byte, rotated to bit 4
                constexpr uint32_t M4 = 0x0F0F0F0Fu, M5 = 0x10101010u;
                const int rl = (2 * c - 4) & 31, rh = (2 * c - 3) & 31;
                la = make_uint4((qa.x & M4) | (__funnelshift_r(qh0.x, qh0.x, rl) & M5),
                                (qa.y & M4) | (__funnelshift_r(qh0.y, qh0.y, rl) & M5),
                                (qa.z & M4) | (__funnelshift_r(qh0.z, qh0.z, rl) & M5),
                                (qa.w & M4) | (__funnelshift_r(qh0.w, qh0.w, rl) & M5));
                lb = make_uint4((qb.x & M4) | (__funnelshift_r(qh1.x, qh1.x, rl) & M5),
                                (qb.y & M4) | (__funnelshift_r(qh1.y, qh1.y, rl) & M5),
                                (qb.z & M4) | (__funnelshift_r(qh1.z, qh1.z, rl) & M5),
                                (qb.w & M4) | (__funnelshift_r(qh1.w, qh1.w, rl) & M5));
                ha = make_uint4(((qa.x >> 4) & M4) | (__funnelshift_r(qh0.x, qh0.x, rh) & M5),
                                ((qa.y >> 4) & M4) | (__funnelshift_r(qh0.y, qh0.y, rh) & M5),
                                ((qa.z >> 4) & M4) | (__funnelshift_r(qh0.z, qh0.z, rh) & M5),
                                ((qa.w >> 4) & M4) | (__funnelshift_r(qh0.w, qh0.w, rh) & M5));
                hb = make_uint4(((qb.x >> 4) & M4) | (__funnelshift_r(qh1.x, qh1.x, rh) & M5),
                                ((qb.y >> 4) & M4) | (__funnelshift_r(qh1.y, qh1.y, rh) & M5),
                                ((qb.z >> 4) & M4) | (__funnelshift_r(qh1.z, qh1.z, rh) & M5),
                                ((qb.w >> 4) & M4) | (__funnelshift_r(qh1.w, qh1.w, rh) & M5));
            } else {
                // high nibbles masked in place: an unsigned x signed dp4a then gives 16 x the dot
                la = and4(qa, 0x0F0F0F0Fu);
                lb = and4(qb, 0x0F0F0F0Fu);
                ha = and4(qa, 0xF0F0F0F0u);
                hb = and4(qb, 0xF0F0F0F0u);
            }
            const uint32_t scw = c < 2 ? sc03 : sc47;
            const int sl = (int)__byte_perm(scw, 0u, 0x4440u | (uint32_t)((2 * c) & 3));
            const int sh = (int)__byte_perm(scw, 0u, 0x4440u | (uint32_t)((2 * c + 1) & 3));
#pragma unroll
            for (int v = 0; v < B; ++v) {
                const int8_t *av = act + v * vstride + 64 * c;
                const uint4 a0 = lds128(av), a1 = lds128(av + 16), a2 = lds128(av + 32), a3 = lds128(av + 48);
                const int dl = dp4a4(lb, a1, dp4a4(la, a0, 0));
                const int dh = Q5 ? dp4a4(hb, a3, dp4a4(ha, a2, 0)) : dp4a4_us(hb, a3, dp4a4_us(ha, a2, 0));
                Slo[v] += sl * dl;
                Shi[v] += sh * dh;
                if (DUMP && live) {
                    int32_t *dd = p.dbg_dots + (((int64_t)v * p.rows + row) * nb + blk) * 16;
                    dd[2 * c] = dl;
                    dd[2 * c + 1] = Q5 ? dh : dh >> 4;
                }
            }
        }
        const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xffffu)));
        const float dmin = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
#pragma unroll
        for (int v = 0; v < B; ++v) {
            const int S = Q5 ? Slo[v] + Shi[v] : Slo[v] + (Shi[v] >> 4);  // exact: Shi carries 16 x
            const int4 bs = *reinterpret_cast<const int4 *>(saux + ((size_t)v * nb + blk) * 8);
            int M = __dp2a_lo(bs.x, (int)m03, 0);
            M = __dp2a_hi(bs.y, (int)m03, M);
            M = __dp2a_lo(bs.z, (int)m47, M);
            M = __dp2a_hi(bs.w, (int)m47, M);
            const float dx = sdx[(size_t)v * nb + blk];
            t[v] = __fmul_rn(dx, __fsub_rn(__fmul_rn(d, __int2float_rn(S)), __fmul_rn(dmin, __int2float_rn(M))));
            if (DUMP && live) {
                int32_t *sm = p.dbg_sm + (((int64_t)v * p.rows + row) * nb + blk) * 2;
                sm[0] = S;
                sm[1] = M;
            }
        }
    } else {
        // Q6_K body: ql [0, 128), qh [128, 192), int8 scales [192, 208).  Value 128hh + 32q + l
        // (quarter q, l < 32) takes the low (q < 2) or high nibble of ql[64hh + 32 (q & 1) + l]
        // and bits 2q, 2q + 1 of qh[32hh + l]; its 16-value sub-block is 8hh + 2q + l / 16.
        const uint4 sc = lds128(bp + 192);
        const uint32_t scw[4] = {sc.x, sc.y, sc.z, sc.w};
        int Sd[B];
#pragma unroll
        for (int v = 0; v < B; ++v)
            Sd[v] = 0;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint4 qh = lds128(bp + 128 + 32 * hh + 16 * j);
                const uint4 l0 = lds128(bp + 64 * hh + 16 * j), l1 = lds128(bp + 64 * hh + 32 + 16 * j);
                constexpr uint32_t M4 = 0x0F0F0F0Fu, M6 = 0x30303030u;
                uint4 q[4];
                q[0] = make_uint4((l0.x & M4) | ((qh.x << 4) & M6), (l0.y & M4) | ((qh.y << 4) & M6),
                                  (l0.z & M4) | ((qh.z << 4) & M6), (l0.w & M4) | ((qh.w << 4) & M6));
                q[1] = make_uint4((l1.x & M4) | ((qh.x << 2) & M6), (l1.y & M4) | ((qh.y << 2) & M6),
                                  (l1.z & M4) | ((qh.z << 2) & M6), (l1.w & M4) | ((qh.w << 2) & M6));
                q[2] = make_uint4(((l0.x >> 4) & M4) | (qh.x & M6), ((l0.y >> 4) & M4) | (qh.y & M6),
                                  ((l0.z >> 4) & M4) | (qh.z & M6), ((l0.w >> 4) & M4) | (qh.w & M6));
                q[3] = make_uint4(((l1.x >> 4) & M4) | ((qh.x >> 2) & M6), ((l1.y >> 4) & M4) | ((qh.y >> 2) & M6),
                                  ((l1.z >> 4) & M4) | ((qh.z >> 2) & M6), ((l1.w >> 4) & M4) | ((qh.w >> 2) & M6));
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const int s = 8 * hh + 2 * qq + j;
                    const int scs = sbyte(scw[s >> 2], s & 3);
#pragma unroll
                    for (int v = 0; v < B; ++v) {
                        const uint4 a = lds128(act + v * vstride + 16 * s);
                        const int dot = dp4a4(q[qq], a, 0);  // codes 0..63: signed bytes
                        Sd[v] += scs * dot;
                        if (DUMP && live) {
                            const int xs = saux[((size_t)v * nb + blk) * 16 + s];
                            p.dbg_dots[(((int64_t)v * p.rows + row) * nb + blk) * 16 + s] = dot - 32 * xs;
                        }
                    }
                }
            }
        }
        const float d = __half2float(__ushort_as_half(q6_d));
#pragma unroll
        for (int v = 0; v < B; ++v) {
            // S = sum_s sc_s (dot_s - 32 xs_s): the -32 offset through the 16-code sums
            const uint4 x0 = lds128(saux + ((size_t)v * nb + blk) * 16);
            const uint4 x1 = lds128(saux + ((size_t)v * nb + blk) * 16 + 8);
            int C = __dp2a_lo((int)x0.x, (int)sc.x, 0);
            C = __dp2a_hi((int)x0.y, (int)sc.x, C);
            C = __dp2a_lo((int)x0.z, (int)sc.y, C);
            C = __dp2a_hi((int)x0.w, (int)sc.y, C);
            C = __dp2a_lo((int)x1.x, (int)sc.z, C);
            C = __dp2a_hi((int)x1.y, (int)sc.z, C);
            C = __dp2a_lo((int)x1.z, (int)sc.w, C);
            C = __dp2a_hi((int)x1.w, (int)sc.w, C);
            const int S = Sd[v] - 32 * C;
            const float dx = sdx[(size_t)v * nb + blk];
            t[v] = __fmul_rn(dx, __fmul_rn(d, __int2float_rn(S)));
            if (DUMP && live) {
                int32_t *sm = p.dbg_sm + (((int64_t)v * p.rows + row) * nb + blk) * 2;
                sm[0] = S;
                sm[1] = 0;
            }
        }
    }
}

// F is QMD_Q4_K, QMD_Q5_K or QMD_Q6_K_SPLIT; B the vectors; MODE plain, recording or packing.
template <int F, int B, int MODE>
__global__ void __launch_bounds__(rl_max_threads(B), 1) qmv_rl_kernel(const __grid_constant__ RlParams rp)
{
    constexpr bool Q6 = F == QMD_Q6_K_SPLIT;
    constexpr bool NORM = MODE == QMV_NORM;
    constexpr bool PACK = MODE == QMV_PACK || NORM;  // both pack f32 activations themselves
    constexpr bool DUMP = MODE == QMV_DUMP;
    constexpr int BB = rl_block_bytes(F);
    constexpr int SLOT = rl_slot_bytes(F);
    constexpr int BOX = rl_box_bytes(F);
    static_assert(B >= 1 && B <= RL_MAX_BATCH, "one to four vectors");
    const QmvKParams &p = rp.k;
    extern __shared__ __align__(128) uint8_t smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int W = p.WR, S = p.stages, nb = p.nb;  // warps 0 .. W-1 own rings and tiles
    const int NW = blockDim.x >> 5;                // warp NW-1 requests the first ring fills,
    const int NP = NW - 1;                         // warps 0 .. NP-1 pack the activations
    const int r = lane >> 4, g = lane & 15;
    const int nsteps = (nb + RL_BLOCKS - 1) / RL_BLOCKS;
    // The tiles: without a workspace, CTA b owns q or q + 1 consecutive tiles of an even split
    // [ts0, ts1) and its warp w takes ts0 + w, ts0 + w + W, ...  With one, only the first `nstat`
    // tiles are split so; the last p.dyn_tiles go to warps one at a time, in the order their
    // claims reach the workspace's counters (after the dependency wait), so that CTAs which run
    // slow do not set the end.  (Tile counts are below 2^29: 32-bit arithmetic.)
    unsigned *const ws = p.ws;
    const unsigned ntiles = (unsigned)((p.rows + RL_ROWS - 1) / RL_ROWS);
    const unsigned ndyn = ws ? (unsigned)p.dyn_tiles : 0u;
    const unsigned nstat = ntiles - ndyn;
    const unsigned bx = blockIdx.x, G = gridDim.x;
    const unsigned st_q = nstat / G, st_rem = nstat - st_q * G;
    const int64_t ts0 = (int64_t)bx * st_q + min(bx, st_rem), ts1 = ts0 + st_q + (bx < st_rem ? 1 : 0);
    const RlLayout L = qmv_rl_layout(F, W, S, B, nb, NORM);
#ifdef QMD_TRACE
    if (tid == 0 && p.trace) {
        p.trace[(size_t)blockIdx.x * QMD_TRACE_FIELDS] = globaltimer_ns();
        p.trace[(size_t)blockIdx.x * QMD_TRACE_FIELDS + 7] =
            (unsigned long long)smid() | ((unsigned long long)blockIdx.x << 16) |
            ((unsigned long long)gridDim.x << 32) | ((unsigned long long)(PACK ? 1 : 2) << 48);
    }
#endif
    // A launch whose geometry is not the plan's: flag it and leave without touching memory (after
    // the dependency wait, so that kernels launched after this one still see its predecessor done).
    if (NW < W + 1 || (NORM && NW - 1 < 8) || (uint32_t)L.total > dynamic_smem_bytes()) {
        pdl_wait();
        if (tid == 0)
            atomicOr(p.err, ERRBIT_PLAN);
        return;
    }

    const uint64_t pol = policy_evict_first();
    const uint32_t bars = smem_addr(smem + L.bar_off);
    int *const s_tiles = reinterpret_cast<int *>(smem + L.tile_off);
    // the copies of step s of `tile` into slot `slot` of warp w's ring (one thread)
    auto issue_w = [&](int w, int64_t tile, int s, int slot) {
        const uint32_t bar = bars + 8u * (uint32_t)(w * S + slot);
        s_tiles[w * S + slot] = (int)tile;
        mbar_arrive_expect_tx(bar, (uint32_t)rl_tx_bytes(F));
        const uint32_t dst = smem_addr(smem + (size_t)(w * S + slot) * SLOT);
        tma_load_3d(dst, &rp.wmap, 0, RL_BLOCKS * s, (int)(RL_ROWS * tile), bar, pol);
        if (Q6)
            tma_load_2d(dst + BOX, &rp.premap, RL_BLOCKS * s, (int)(RL_ROWS * tile), bar, pol);
    };
    volatile int *s_sched = reinterpret_cast<volatile int *>(smem + L.sched_off);  // [0] pool empty, [1] warps done
    if (tid == 0) {
        s_sched[0] = 0;
        s_sched[1] = 0;
    }
    if (warp == NP && lane == 0) {
        for (int i = 0; i < W * S; ++i)
            mbar_init(bars + 8u * (uint32_t)i, 1);
        fence_barrier_init();
    }
    __syncthreads();  // barriers initialised before any warp waits on them
    pdl_launch_dependents();

    // The first S steps of every ring's static tiles, requested by the one warp that does
    // nothing else (a tensor copy takes the unit tens of nanoseconds, so a few dozen of them would
    // hold up the packing warps), slot by slot across the warps so that every warp's first steps
    // come first: p.pre_steps slots (2) before the dependency wait -- they read weights only --
    // and the rest once the activations are packed, since the pack's loads from L2 share the
    // SM's path with these copies (measured on the 8-layer step: 1, 2, 3, 4 slots before the wait
    // with the rest after the pack 33.4, 31.4, 31.6, 31.7 us a layer; the rest right after the
    // wait instead 31.8-32.0).
    if (warp == NP) {
        int64_t tk = 0;  // the static tile (of each warp's sequence) of slot k's step
        int sk = 0;      // and the step within it
        auto issue_slot = [&](int k) {
            for (int w = 0; w < W; ++w) {
                const int64_t t = ts0 + w + tk * W;
                if (t < ts1)
                    issue_w(w, t, sk, k);
            }
            if (++sk == nsteps) {
                sk = 0;
                ++tk;
            }
        };
        const int pre = p.pre_steps < S ? p.pre_steps : S;
        if (lane == 0) {
            for (int k = 0; k < pre; ++k)
                issue_slot(k);
            QMD_STAMP(p, 1);
        }
        if (pre < S) {
            // the rest once the activations are packed: the pack's loads share the SM's path
            // from L2 with these copies (the whole warp meets the packing warps' barrier)
            __syncwarp();
            asm volatile("bar.sync 1, %0;" ::"r"(32 * NW) : "memory");
            if (lane == 0)
                for (int k = pre; k < S; ++k)
                    issue_slot(k);
        }
        return;  // the copies complete on the barriers by themselves
    }

    const int wr = warp < W ? warp : 0;  // packing warps past W have no ring (and no steps)
    const uint32_t bar0 = bars + 8u * (uint32_t)(wr * S);
    auto issue = [&](int64_t tile, int s, int slot) { issue_w(wr, tile, s, slot); };
    // Lane 0's schedule: the next static tile, then claimed ones.  The dynamic tiles are cut into
    // RL_POOLS pools, one per group of CTAs (b % RL_POOLS), each with its own counter, so that
    // claims spread over several addresses.  A claim is sent one tile ahead, so that its answer
    // is back when the tile's first copy is issued; every answer is used (a tile of the pool) or
    // marks the pool empty for the whole CTA (a shared-memory flag, so that the CTA's other warps
    // stop asking).  The last warp of a CTA to finish claiming counts the CTA on the workspace's
    // done word; the CTA that completes that count resets every word to 0, so the next call that
    // uses the workspace finds it zeroed.
    const unsigned npools = G < (unsigned)RL_POOLS ? G : (unsigned)RL_POOLS;
    const unsigned pool = bx % npools;
    const unsigned pq = ndyn / npools, prem = ndyn - pq * npools;
    const int64_t pool0 = (int64_t)nstat + (int64_t)pool * pq + min(pool, prem);
    const int64_t pool_n = pq + (pool < prem ? 1 : 0);
    unsigned *const cnt = ws ? ws + RL_WS_STRIDE * pool : nullptr;
    // the cursor after the steps the first warp requested: n0 of this warp's static steps
    const int64_t nstw = (warp < W && ts1 - ts0 > warp) ? (ts1 - ts0 - warp + W - 1) / W : 0;
    const int64_t n0 = nstw * nsteps < S ? nstw * nsteps : S;
    int64_t issued = n0;
    int is = (int)(n0 % nsteps);
    int64_t itile = ts0 + warp + (n0 / nsteps) * W;  // mid-tile (is > 0): the tile being requested
    int64_t st_next = is ? itile + W : itile;        // the next static tile to start
    unsigned pending = 0u;
    bool have_pending = false, claims_done = (ws == nullptr);
    auto finish_claims = [&]() {
        claims_done = true;
        if (atomicAdd(const_cast<int *>(s_sched) + 1, 1) == W - 1 &&
            atomicAdd(ws + RL_WS_STRIDE * RL_POOLS, 1u) == gridDim.x - 1u) {
            for (int k = 0; k < RL_POOLS; ++k)
                atomicExch(ws + RL_WS_STRIDE * k, 0u);
            atomicExch(ws + RL_WS_STRIDE * RL_POOLS, 0u);
        }
    };
    auto next_tile = [&](bool dyn_ok) -> int64_t {
        if (st_next < ts1) {
            const int64_t t = st_next;
            st_next += W;
            if (st_next >= ts1 && dyn_ok && !claims_done && !have_pending && !s_sched[0]) {
                pending = atomicAdd(cnt, 1u);  // the first claim, sent early
                have_pending = true;
            }
            return t;
        }
        if (!dyn_ok || claims_done)
            return -1;
        unsigned c;
        if (have_pending) {
            c = pending;
            have_pending = false;
        } else if (s_sched[0]) {
            finish_claims();
            return -1;
        } else {
            c = atomicAdd(cnt, 1u);
        }
        if ((int64_t)c >= pool_n) {
            s_sched[0] = 1;
            finish_claims();
            return -1;
        }
        if (!s_sched[0]) {
            pending = atomicAdd(cnt, 1u);  // the next claim, sent early
            have_pending = true;
        }
        return pool0 + c;
    };
    auto issue_next = [&](bool dyn_ok, int slot) -> bool {  // lane 0: request the next step into `slot`
        if (is == 0) {
            itile = next_tile(dyn_ok);
            if (itile < 0)
                return false;
        }
        issue(itile, is, slot);
        if (++is == nsteps)
            is = 0;
        ++issued;
        return true;
    };

    pdl_wait();  // activations come from earlier work in the stream
    if (tid == 0)
        QMD_STAMP(p, 2);

    // ---- activations into shared memory: codes (padded blocks), scales, sums ---------------
    int8_t *acts = reinterpret_cast<int8_t *>(smem + L.act_off);
    float *sdx = reinterpret_cast<float *>(smem + L.dx_off);
    int16_t *saux = reinterpret_cast<int16_t *>(smem + L.aux_off);
    const int NBv = B * nb;  // activation blocks
    if (PACK) {
        const int64_t K = (int64_t)nb * 256;
        float *s_part = reinterpret_cast<float *>(smem + L.norm_off);  // RMSNorm form: [B][8] and 1/rms [B]
        float *s_inv = s_part + B * 8;
        if (NORM) {
            // RMSNorm of h = x (+ r), each f32 operation rounded alone, the sum of squares in the
            // order the stand-alone RMSNorm pack declares (so the codes are the same): thread t
            // of the first 256 adds the squares of elements t, t + 256, ... left to right; each
            // warp combines its partials by xor-shuffles 16, 8, 4, 2, 1; the eight warp totals
            // are added left to right.  CTA 0 writes h when asked.
            for (int v = 0; v < B; ++v) {
                if (tid < 256) {
                    const float *xv = p.x + v * K;
                    const float *rv = p.r ? p.r + v * K : nullptr;
                    float *hv = (p.h_out && blockIdx.x == 0) ? p.h_out + v * K : nullptr;
                    float acc = 0.0f;
                    constexpr int U = 8;  // loads in flight per thread per round
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
            asm volatile("bar.sync 2, %0;" ::"r"(32 * NP) : "memory");
            if (tid < B) {
                float total = s_part[tid * 8];
                for (int w = 1; w < 8; ++w)
                    total = __fadd_rn(total, s_part[tid * 8 + w]);
                const float ms = __fdiv_rn(total, (float)K);
                s_inv[tid] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, p.eps)));
            }
            asm volatile("bar.sync 2, %0;" ::"r"(32 * NP) : "memory");
        }
        // quantise the f32 activations (RMSNorm form: n = (h * (1/rms)) * g), one warp per
        // block, the stand-alone pack's arithmetic
        const bool out = blockIdx.x == 0 && p.xq_qs_out != nullptr;
        for (int b0 = warp; b0 < NBv; b0 += 4 * NP) {
            float4 xa[4], xb[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int b = b0 + u * NP;
                if (b < NBv) {
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
            for (int u = 0; u < 4; ++u) {
                const int b = b0 + u * NP;  // the same for every lane of the warp
                if (b < NBv) {
                    const float v8[8] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w, xb[u].x, xb[u].y, xb[u].z, xb[u].w};
                    const Q8Block qb = q8k_quantise_block(v8);
                    *reinterpret_cast<uint2 *>(acts + (size_t)b * RL_ACT + 8 * lane) = qb.codes;
                    if (Q6) {
                        if ((lane & 1) == 0)
                            saux[b * 16 + (lane >> 1)] = (int16_t)qb.sum2;
                    } else if ((lane & 3) == 0) {
                        saux[b * 8 + (lane >> 2)] = (int16_t)qb.sum4;
                    }
                    if (lane == 0)
                        sdx[b] = qb.d;
                    if (out) {
                        *reinterpret_cast<uint2 *>(p.xq_qs_out + (int64_t)b * 256 + 8 * lane) = qb.codes;
                        if ((lane & 3) == 0)
                            p.xq_bs_out[b * 8 + (lane >> 2)] = (int16_t)qb.sum4;
                        if (lane == 0)
                            p.xq_d_out[b] = qb.d;
                    }
                }
            }
        }
    } else {
        // packed input: the codes 16 bytes at a time into the padded blocks; Q6_K also sums each
        // 16 codes; the scales and (Q4_K, Q5_K) the 32-code sums
        for (int i = tid; i < NBv * 16; i += 32 * NP) {
            const int b = i >> 4, c = i & 15;
            const uint4 q = *reinterpret_cast<const uint4 *>(p.xqs + (int64_t)b * 256 + 16 * c);
            *reinterpret_cast<uint4 *>(acts + (size_t)b * RL_ACT + 16 * c) = q;
            if (Q6)
                saux[b * 16 + c] = (int16_t)dp4a4(q, make_uint4(0x01010101u, 0x01010101u, 0x01010101u, 0x01010101u), 0);
        }
        for (int i = tid; i < NBv; i += 32 * NP) {
            sdx[i] = p.xd[i];
            if (!Q6)
                *reinterpret_cast<int4 *>(saux + i * 8) = reinterpret_cast<const int4 *>(p.xbs)[i];
        }
    }
    // the packing warps, and the requesting warp if it still has copies to request after the pack
    asm volatile("bar.sync 1, %0;" ::"r"(32 * (p.pre_steps < S ? NW : NP)) : "memory");
    if (tid == 0)
        QMD_STAMP(p, 3);
    // the rest of the ring (claims may start now)
    if (lane == 0 && warp < W)
        while (issued < S && issue_next(true, (int)issued)) {
        }

    // ---- the warp's steps --------------------------------------------------------------------
    const unsigned long long wait_ns = p.wait_ns;
    float T[B];
#pragma unroll
    for (int v = 0; v < B; ++v)
        T[v] = 0.0f;
    int64_t tile = -1;
    int s = 0, slot = 0;
    uint32_t par = 0u;
#pragma unroll 1
    for (int64_t i = 0; warp < W; ++i) {
        if (!__shfl_sync(0xffffffffu, (int)(issued > i), 0))  // lane 0 knows whether step i exists
            break;
        // (the whole warp takes the same branch: a lane that gave up makes every lane leave)
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8u * (uint32_t)slot, par, wait_ns))) {
            // A copy did not land in time: flag it, wait (bounded) for this warp's copies that
            // may still be in flight (steps i .. issued - 1), settle its claims, leave.
            if (lane == 0) {
                atomicOr(p.err, ERRBIT_QMV_WAIT);
                int sl = slot;
                uint32_t pa = par;
                for (int64_t j = i; j < issued; ++j) {
                    if (!mbar_wait_bounded(bar0 + 8u * (uint32_t)sl, pa, wait_ns)) {
                        atomicOr(p.err, ERRBIT_DRAIN_WAIT);
                        break;
                    }
                    if (++sl == S) {
                        sl = 0;
                        pa ^= 1u;
                    }
                }
                if (!claims_done)
                    finish_claims();
            }
            __syncwarp();
            return;
        }
        if (i == 0 && warp == 0 && lane == 0)
            QMD_STAMP(p, 4);
        if (s == 0)
            tile = s_tiles[wr * S + slot];
        const uint8_t *box = smem + (size_t)(wr * S + slot) * SLOT;
        const int blk = RL_BLOCKS * s + g;
        const int64_t row = RL_ROWS * tile + r;
        float t[B];
        if (blk < nb) {
            const unsigned short q6d =
                Q6 ? *reinterpret_cast<const unsigned short *>(box + BOX + 2 * (RL_BLOCKS * r + g)) : (unsigned short)0;
            rl_block_terms<F, B, DUMP>(box + (r * RL_BLOCKS + g) * BB, acts + (size_t)blk * RL_ACT, sdx, saux, nb,
                                       blk, q6d, p, row, row < p.rows, t);
        } else {
#pragma unroll
            for (int v = 0; v < B; ++v)
                t[v] = 0.0f;  // a block past the row's end adds +0
        }
        // the slot is consumed: refill it with the step S ahead
        __syncwarp();
        if (lane == 0) {
            fence_proxy_async_smem();
            issue_next(true, slot);
        }
        // The step is run s of the row: groups of four blocks, (t0 + t1) + (t2 + t3) by two
        // xor-shuffles inside each quarter of the row's 16 lanes (absent blocks add +0); then the
        // run, ((G0 + G1) + G2) + G3, from the four quarters (absent groups are +0 the same way);
        // the runs left to right.  Every lane of the row ends with the same bits.
        const int q0 = lane & 16;  // the row's first lane
#pragma unroll
        for (int v = 0; v < B; ++v) {
            float gs = __fadd_rn(t[v], __shfl_xor_sync(0xffffffffu, t[v], 1));
            gs = __fadd_rn(gs, __shfl_xor_sync(0xffffffffu, gs, 2));
            const float G0 = __shfl_sync(0xffffffffu, gs, q0), G1 = __shfl_sync(0xffffffffu, gs, q0 + 4);
            const float G2 = __shfl_sync(0xffffffffu, gs, q0 + 8), G3 = __shfl_sync(0xffffffffu, gs, q0 + 12);
            const float Rv = __fadd_rn(__fadd_rn(__fadd_rn(G0, G1), G2), G3);
            T[v] = s == 0 ? Rv : __fadd_rn(T[v], Rv);
        }
        if (s == nsteps - 1) {
            if (row < p.rows) {
#pragma unroll
                for (int v = 0; v < B; ++v)
                    if (g == v)
                        p.y[(int64_t)v * p.rows + row] = T[v];
            }
            s = 0;
        } else {
            ++s;
        }
        if (++slot == S) {
            slot = 0;
            par ^= 1u;
        }
    }
#ifdef QMD_TRACE
    if (lane == 0 && p.trace) {
        atomicMax(p.trace + (size_t)blockIdx.x * QMD_TRACE_FIELDS + 5, globaltimer_ns());
        atomicMax(p.trace + (size_t)blockIdx.x * QMD_TRACE_FIELDS + 6, globaltimer_ns());
    }
#endif
    // every step this warp requested it also consumed, so no copy is in flight here
}

// Tensor maps of one call: W as bytes [rows][nb][block bytes] in boxes of (block bytes, 16
// blocks, 2 rows) -- blocks and rows past the end read as zeros -- and for Q6_K the prefix as
// u16 [rows][prefix stride] in boxes of 16 entries x 2 rows.  Strides are multiples of 16 bytes
// (block bytes 144, 176, 208; the prefix stride a multiple of 8 entries), bases 16-byte aligned
// (checked by the caller).
template <int F>
qmd_status rl_tensor_maps(const QmvKParams &kp, RlParams &rp)
{
    const TensorMapEncodeFn enc = tensor_map_encoder();
    if (!enc)
        return fail(QMD_ERR_LAUNCH, "cuTensorMapEncodeTiled entry point", cudaErrorNotSupported);
    std::memset(&rp.wmap, 0, sizeof rp.wmap);
    std::memset(&rp.premap, 0, sizeof rp.premap);
    const cuuint32_t estr[3] = {1, 1, 1};
    const cuuint64_t wdim[3] = {(cuuint64_t)rl_block_bytes(F), (cuuint64_t)kp.nb, (cuuint64_t)kp.rows};
    const cuuint64_t wstr[2] = {(cuuint64_t)rl_block_bytes(F), (cuuint64_t)kp.row_bytes};
    const cuuint32_t wbox[3] = {(cuuint32_t)rl_block_bytes(F), (cuuint32_t)RL_BLOCKS, (cuuint32_t)RL_ROWS};
    if (enc(&rp.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(kp.W), wdim, wstr, wbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return fail(QMD_ERR_LAUNCH, "tensor map of the weights", cudaErrorInvalidValue);
    if (F == QMD_Q6_K_SPLIT) {
        const cuuint64_t pdim[2] = {(cuuint64_t)(kp.pre_bytes / 2), (cuuint64_t)kp.rows};
        const cuuint64_t pstr[1] = {(cuuint64_t)kp.pre_bytes};
        const cuuint32_t pbox[2] = {(cuuint32_t)RL_BLOCKS, (cuuint32_t)RL_ROWS};
        if (enc(&rp.premap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint8_t *>(kp.Wpre), pdim, pstr, pbox,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return fail(QMD_ERR_LAUNCH, "tensor map of the Q6_K prefix", cudaErrorInvalidValue);
    }
    return QMD_OK;
}

template <int F, int B>
qmd_status launch_rl_batch(const RlParams &rp, const QmvPlan &plan, int mode, cudaStream_t s)
{
    return mode == QMV_PACK   ? launch_kernel<qmv_rl_kernel<F, B, QMV_PACK>>(rp, plan, s)
           : mode == QMV_NORM ? launch_kernel<qmv_rl_kernel<F, B, QMV_NORM>>(rp, plan, s)
           : mode == QMV_DUMP ? launch_kernel<qmv_rl_kernel<F, B, QMV_DUMP>>(rp, plan, s)
                              : launch_kernel<qmv_rl_kernel<F, B, QMV_PLAIN>>(rp, plan, s);
}

template <int F>
qmd_status launch_qmv_rl(const QmvKParams &kp, const QmvPlan &plan, int mode, int batch, cudaStream_t s)
{
    RlParams rp;
    rp.k = kp;
    const qmd_status st = rl_tensor_maps<F>(kp, rp);
    if (st != QMD_OK)
        return st;
    switch (batch) {
    case 1:
        return launch_rl_batch<F, 1>(rp, plan, mode, s);
    case 2:
        return launch_rl_batch<F, 2>(rp, plan, mode, s);
    case 3:
        return launch_rl_batch<F, 3>(rp, plan, mode, s);
    case 4:
        return launch_rl_batch<F, 4>(rp, plan, mode, s);
    }
    return QMD_ERR_BATCH;
}

}  // namespace qmd
