// qmv_splitk.cuh -- the split-K form of the one- and two-vector mat-vec, for launches whose rows
// alone give the SMs little to do: the CTAs of a thread-block cluster share a range of rows and
// each takes a slice of every row's blocks (a slice of K), so each packs only its slice of the
// activations; the slices' group sums meet in distributed shared memory, where the cluster adds
// them in the declared row order.
//
// "Language models on the device: the cajeta-llm kernels", §2.3 (split-K partial sums along K
// and a fixup that combines them, for grids the rows alone underfill).  The block terms are the
// row-lane kernel's (rl_block_terms, §1, §2.1, §2.2), and the sums follow the declared row
// order, so y has the same bits as every other kernel and the oracle: blocks in groups of four,
// (t0 + t1) + (t2 + t3), absent blocks +0; the four groups of a run of sixteen blocks,
// ((G0 + G1) + G2) + G3, absent groups +0; the runs left to right.
//
// Work split.  Lane (r, j) = (lane / 4, lane % 4) takes row r of an 8-row tile and block j of a
// group of four blocks: a warp step is 8 rows x one group, and two xor-shuffles leave the group
// sum G of row r in lane 4r.  A cluster of KS CTAs owns a contiguous range of tiles; its CTA of
// rank k owns groups [floor(k gq / KS), floor((k + 1) gq / KS)) of every row (gq groups a row),
// and its ring warps take the range's tiles in turn (warp w: tiles w, w + W, ...), each walking
// its slice group by group.  (Handing the (tile, group) steps to the warps one by one instead,
// so that more warps have work, was slower: 4096 x 4096 at two slices 5.3 against 4.2 us.)
// Every G is kept in the CTA's shared memory at [vector][row][group].
// After a cluster barrier each CTA finishes 1/KS of the range's rows: it reads each group sum
// from the CTA that owns it (ld.shared::cluster) and adds them in the declared order.  A second
// cluster barrier keeps every CTA's shared memory in place until its peers have read it.
//
// Staging as in the row-lane kernel: a private ring of S slots per warp, one 3-D tensor copy per
// step (box: block bytes x 4 blocks x 8 rows of W viewed as [rows][nb][block bytes], landing as
// [8 rows][4 blocks][block bytes]; blocks and rows past the end read as zeros), plus for Q6_K a
// 2-D copy of the 8 rows' f16 scales of the eight blocks around the group (16 bytes a row, the
// narrowest copy allowed); p.pre_steps slots per warp are requested before the dependency wait,
// the rest once the activations are in shared memory.
//
// Waits.  Every ring wait is bounded: a warp that gives up sets the device error word, waits
// (bounded again) for its copies in flight and skips its remaining steps.  Both cluster barriers
// are met by every thread of every CTA of the cluster on every path past the launch check (whose
// outcome is the same for every CTA of a launch), so they complete once the bounded waits before
// them have.
#pragma once

#include "qmv_rl.cuh"

namespace qmd {

constexpr int SK_ROWS = 8;       // rows per tile (lane bits 2..4)
constexpr int SK_BLOCKS = 4;     // blocks per step: one group of the row order (lane bits 0..1)
constexpr int SK_MAX_WARPS = 16;
constexpr int SK_MAX_SPLIT = 8;  // CTAs per cluster: the portable cluster size
constexpr int SK_MAX_BATCH = 2;

__host__ __device__ constexpr int sk_box_bytes(int f) { return SK_ROWS * SK_BLOCKS * rl_block_bytes(f); }
// a ring slot (a multiple of 128 bytes): the box, then (Q6_K) the 8 rows' 16-byte scale chunks
__host__ __device__ constexpr int sk_slot_bytes(int f) { return sk_box_bytes(f) + (f == QMD_Q6_K_SPLIT ? SK_ROWS * 16 : 0); }
// the first group of rank k's slice, for gq groups a row over KS ranks
__host__ __device__ constexpr int sk_g0(int k, int gq, int KS) { return (k * gq) / KS; }
// the rank whose slice holds group g: the largest k with sk_g0(k) <= g
__host__ __device__ constexpr int sk_owner(int g, int gq, int KS) { return ((g + 1) * KS - 1) / gq; }
// the 8-row tiles [c0, c1) of cluster cid of NC: an even split of ntiles, the first
// ntiles % NC clusters one tile more
__host__ __device__ inline void sk_cluster_tiles(int64_t cid, int64_t NC, int64_t ntiles, int64_t *c0, int64_t *c1)
{
    const int64_t tq = ntiles / NC, trem = ntiles - tq * NC;
    *c0 = cid * tq + (cid < trem ? cid : trem);
    *c1 = *c0 + tq + (cid < trem ? 1 : 0);
}

struct SkLayout {
    int bar_off, act_off, dx_off, aux_off, part_off, total;
};

// Shared memory: rings [W][S][slot] | mbarriers u64 [W][S] | activation codes i8 [B][nbs][272] |
// block scales f32 [B][nbs] | Q4_K, Q5_K: sums i16 [B][nbs][8] of each 32 codes; Q6_K: sums i16
// [B][nbs][16] of each 16 codes | group sums f32 [B][rows_c][gq].  nbs: the most blocks a slice
// has (4 x its groups); rows_c: the most rows a cluster's range has.
__host__ __device__ inline SkLayout qmv_sk_layout(int f, int W, int S, int B, int nbs, int rows_c, int gq)
{
    SkLayout L;
    int o = W * S * sk_slot_bytes(f);
    L.bar_off = o;
    o += W * S * 8;
    L.act_off = align_up(o, 16);
    o = L.act_off + B * nbs * RL_ACT;
    L.dx_off = o;
    o = align_up(o + B * nbs * 4, 16);
    L.aux_off = o;
    o += B * nbs * (f == QMD_Q6_K_SPLIT ? 32 : 16);
    L.part_off = align_up(o, 16);
    o = L.part_off + B * rows_c * gq * 4;
    L.total = align_up(o, 16);
    return L;
}

struct SkParams {
    QmvKParams k;        // k.WR: ring warps; k.stages: slots a ring; k.pre_steps: slots before the wait
    CUtensorMap wmap;    // W as u8 [rows][nb][block bytes], box: block bytes x 4 blocks x 8 rows
    CUtensorMap premap;  // Q6_K prefix as u16 [rows][prefix stride], box: 8 scales x 8 rows
    int ks;              // CTAs per cluster: K slices
    int tiles_c;         // the most 8-row tiles a cluster's range has (sizes the group sums)
};

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t clusters_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster: earlier shared-memory writes are visible to the
// cluster's reads after it.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// An f32 in the shared memory of cluster rank `rank`, at this CTA's shared address `addr`.
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr, uint32_t rank)
{
    uint32_t a;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(addr), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}

// F is QMD_Q4_K, QMD_Q5_K or QMD_Q6_K_SPLIT; B the vectors; PACK: quantise f32 activations in
// the kernel (the fused form) rather than read packed ones.
template <int F, int B, bool PACK>
__global__ void __launch_bounds__(32 * SK_MAX_WARPS, 1) qmv_sk_kernel(const __grid_constant__ SkParams sp)
{
    constexpr bool Q6 = F == QMD_Q6_K_SPLIT;
    constexpr int BB = rl_block_bytes(F);
    constexpr int SLOT = sk_slot_bytes(F);
    constexpr int BOX = sk_box_bytes(F);
    static_assert(B >= 1 && B <= SK_MAX_BATCH, "one or two vectors");
    const QmvKParams &p = sp.k;
    extern __shared__ __align__(128) uint8_t smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NW = blockDim.x >> 5, W = p.WR, S = p.stages, nb = p.nb;
    const int KS = sp.ks >= 1 ? sp.ks : 1, gq = (nb + SK_BLOCKS - 1) / SK_BLOCKS;
    const int rank = (int)cluster_ctarank();
    const unsigned cid = cluster_id_x(), NC = clusters_x();
    const int g0 = sk_g0(rank, gq, KS), g1 = sk_g0(rank + 1, gq, KS);
    const int nbs = SK_BLOCKS * ((gq + KS - 1) / KS);   // activation blocks per vector in shared memory
    const int blk0 = SK_BLOCKS * g0;                     // this slice's first block
    const int nbl = min(nb, SK_BLOCKS * g1) - blk0;      // and its block count
    // the cluster's tiles: an even split of the 8-row tiles over the clusters
    const int64_t ntiles = (p.rows + SK_ROWS - 1) / SK_ROWS;
    int64_t c0, c1;
    sk_cluster_tiles(cid, NC, ntiles, &c0, &c1);
    const int rows_c = SK_ROWS * sp.tiles_c;
    const SkLayout L = qmv_sk_layout(F, W, S, B, nbs, rows_c, gq);
    // A launch whose geometry is not the plan's: flag it and leave without touching memory.  Every
    // term is the same for all CTAs of a cluster, so either all of them leave or none does.
    if ((int)cluster_nctarank() != sp.ks || KS > gq || NW < W || W < 1 || S < 1 || c1 - c0 > sp.tiles_c ||
        (uint32_t)L.total > dynamic_smem_bytes()) {
        pdl_wait();
        if (tid == 0)
            atomicOr(p.err, ERRBIT_PLAN);
        return;
    }

    const uint64_t pol = policy_evict_first();
    const uint32_t bars = smem_addr(smem + L.bar_off);
    if (tid == 0) {
        for (int i = 0; i < W * S; ++i)
            mbar_init(bars + 8u * (uint32_t)i, 1);
        fence_barrier_init();
    }
    __syncthreads();  // barriers initialised before any warp waits on them
    pdl_launch_dependents();

    // This warp's steps: tiles c0 + warp, c0 + warp + W, ... each over groups g0 .. g1 - 1.
    // Lane 0 requests them in order into slots 0, 1, ..., S - 1, 0, ...
    const int ns = g1 - g0;
    const int64_t ntw = (warp < W && c1 - c0 > warp) ? (c1 - c0 - warp + W - 1) / W : 0;
    const int64_t nst = ntw * ns;
    const uint32_t bar0 = bars + 8u * (uint32_t)((warp < W ? warp : 0) * S);
    int64_t issued = 0, it_tile = c0 + warp;
    int it_grp = g0, it_slot = 0;
    auto issue_next = [&]() {  // lane 0
        const uint32_t bar = bar0 + 8u * (uint32_t)it_slot;
        mbar_arrive_expect_tx(bar, (uint32_t)(Q6 ? BOX + SK_ROWS * 16 : BOX));
        const uint32_t dst = smem_addr(smem + (size_t)(warp * S + it_slot) * SLOT);
        tma_load_3d(dst, &sp.wmap, 0, SK_BLOCKS * it_grp, (int)(SK_ROWS * it_tile), bar, pol);
        if (Q6)
            tma_load_2d(dst + BOX, &sp.premap, (SK_BLOCKS * it_grp) & ~7, (int)(SK_ROWS * it_tile), bar, pol);
        ++issued;
        if (++it_grp == g1) {
            it_grp = g0;
            it_tile += W;
        }
        if (++it_slot == S)
            it_slot = 0;
    };
    const int pre = p.pre_steps < S ? p.pre_steps : S;
    if (lane == 0)
        while (issued < nst && issued < pre)
            issue_next();

    pdl_wait();  // activations come from earlier work in the stream

    // ---- this slice's activations into shared memory: codes, scales, sums ---------------------
    int8_t *acts = reinterpret_cast<int8_t *>(smem + L.act_off);
    float *sdx = reinterpret_cast<float *>(smem + L.dx_off);
    int16_t *saux = reinterpret_cast<int16_t *>(smem + L.aux_off);
    const int NBv = B * nbl;  // (vector v, slice block b) is item v * nbl + b, stored at v * nbs + b
    if (PACK) {
        // one warp per block, two blocks in flight; cluster 0 writes the packed activations when asked
        const bool out = cid == 0 && p.xq_qs_out != nullptr;
        for (int i0 = warp; i0 < NBv; i0 += 2 * NW) {
            float4 xa[2], xb[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * NW;
                if (i < NBv) {
                    const int v = i / nbl, b = i - v * nbl;
                    const float4 *src = reinterpret_cast<const float4 *>(p.x + ((int64_t)v * nb + blk0 + b) * 256 + 8 * lane);
                    xa[u] = src[0];
                    xb[u] = src[1];
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * NW;  // the same for every lane of the warp
                if (i < NBv) {
                    const int v = i / nbl, b = i - v * nbl, li = v * nbs + b;
                    const int64_t gb = (int64_t)v * nb + blk0 + b;
                    const float v8[8] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w, xb[u].x, xb[u].y, xb[u].z, xb[u].w};
                    const Q8Block qb = q8k_quantise_block(v8);
                    *reinterpret_cast<uint2 *>(acts + (size_t)li * RL_ACT + 8 * lane) = qb.codes;
                    if (Q6) {
                        if ((lane & 1) == 0)
                            saux[li * 16 + (lane >> 1)] = (int16_t)qb.sum2;
                    } else if ((lane & 3) == 0) {
                        saux[li * 8 + (lane >> 2)] = (int16_t)qb.sum4;
                    }
                    if (lane == 0)
                        sdx[li] = qb.d;
                    if (out) {
                        *reinterpret_cast<uint2 *>(p.xq_qs_out + gb * 256 + 8 * lane) = qb.codes;
                        if ((lane & 3) == 0)
                            p.xq_bs_out[gb * 8 + (lane >> 2)] = (int16_t)qb.sum4;
                        if (lane == 0)
                            p.xq_d_out[gb] = qb.d;
                    }
                }
            }
        }
    } else {
        // packed input: the codes 16 bytes at a time; Q6_K also sums each 16 codes; the scales and
        // (Q4_K, Q5_K) the 32-code sums
        for (int i = tid; i < NBv * 16; i += blockDim.x) {
            const int it = i >> 4, c = i & 15;
            const int v = it / nbl, b = it - v * nbl, li = v * nbs + b;
            const int64_t gb = (int64_t)v * nb + blk0 + b;
            const uint4 q = *reinterpret_cast<const uint4 *>(p.xqs + gb * 256 + 16 * c);
            *reinterpret_cast<uint4 *>(acts + (size_t)li * RL_ACT + 16 * c) = q;
            if (Q6)
                saux[li * 16 + c] = (int16_t)dp4a4(q, make_uint4(0x01010101u, 0x01010101u, 0x01010101u, 0x01010101u), 0);
        }
        for (int it = tid; it < NBv; it += blockDim.x) {
            const int v = it / nbl, b = it - v * nbl, li = v * nbs + b;
            const int64_t gb = (int64_t)v * nb + blk0 + b;
            sdx[li] = p.xd[gb];
            if (!Q6)
                *reinterpret_cast<int4 *>(saux + li * 8) = reinterpret_cast<const int4 *>(p.xbs)[gb];
        }
    }
    __syncthreads();
    if (lane == 0)  // the rest of the ring
        while (issued < nst && issued < S)
            issue_next();

    // ---- the warp's steps: group sums into shared memory --------------------------------------
    float *part = reinterpret_cast<float *>(smem + L.part_off);  // [B][rows_c][gq]
    const int r = lane >> 2, j = lane & 3;
    const int64_t crow0 = SK_ROWS * c0;  // the range's first row
    const unsigned long long wait_ns = p.wait_ns;
    int slot = 0, grp = g0;
    uint32_t par = 0u;
    int64_t tile = c0 + warp;
#pragma unroll 1
    for (int64_t i = 0; i < nst; ++i) {
        // (the whole warp takes the same branch)
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8u * (uint32_t)slot, par, wait_ns))) {
            // A copy did not land in time: flag it, wait (bounded) for this warp's copies that may
            // still be in flight (steps i .. issued - 1) and skip the remaining steps.
            if (lane == 0) {
                atomicOr(p.err, ERRBIT_QMV_WAIT);
                int sl = slot;
                uint32_t pa = par;
                for (int64_t k = i; k < issued; ++k) {
                    if (!mbar_wait_bounded(bar0 + 8u * (uint32_t)sl, pa, wait_ns)) {
                        atomicOr(p.err, ERRBIT_DRAIN_WAIT);
                        break;
                    }
                    if (++sl == S) {
                        sl = 0;
                        pa ^= 1u;
                    }
                }
            }
            break;
        }
        const uint8_t *box = smem + (size_t)(warp * S + slot) * SLOT;
        const int blk = SK_BLOCKS * grp + j;  // this lane's block of the row
        const int64_t row = SK_ROWS * tile + r;
        float t[B];
        if (blk < nb) {
            const unsigned short q6d =
                Q6 ? *reinterpret_cast<const unsigned short *>(box + BOX + 2 * (8 * r + blk - ((SK_BLOCKS * grp) & ~7)))
                   : (unsigned short)0;
            rl_block_terms<F, B, false>(box + (r * SK_BLOCKS + j) * BB, acts + (size_t)(blk - blk0) * RL_ACT, sdx, saux,
                                        nbs, blk - blk0, q6d, p, row, row < p.rows, t);
        } else {
#pragma unroll
            for (int v = 0; v < B; ++v)
                t[v] = 0.0f;  // a block past the row's end adds +0
        }
        // the slot is consumed: refill it with the step S ahead
        __syncwarp();
        if (lane == 0 && issued < nst) {
            fence_proxy_async_smem();
            issue_next();
        }
        // the group: (t0 + t1) + (t2 + t3), every lane of the quarter with the same bits
#pragma unroll
        for (int v = 0; v < B; ++v) {
            float gs = __fadd_rn(t[v], __shfl_xor_sync(0xffffffffu, t[v], 1));
            gs = __fadd_rn(gs, __shfl_xor_sync(0xffffffffu, gs, 2));
            if (j == 0 && row < p.rows)
                part[((size_t)v * rows_c + (size_t)(row - crow0)) * gq + grp] = gs;
        }
        if (++grp == g1) {
            grp = g0;
            tile += W;
        }
        if (++slot == S) {
            slot = 0;
            par ^= 1u;
        }
    }
    __syncwarp();

    // ---- the fixup: this rank's share of the range's rows, every group from its owner ---------
    cluster_sync();
    {
        const int64_t nrow = min(p.rows, SK_ROWS * c1) - crow0;
        const uint32_t part_a = smem_addr(part);
        for (int64_t i = (int64_t)rank * blockDim.x + tid; i < B * nrow; i += (int64_t)KS * blockDim.x) {
            const int v = (int)(i / nrow);
            const int64_t lr = i - v * nrow;
            const uint32_t rowa = part_a + 4u * (uint32_t)(((size_t)v * rows_c + (size_t)lr) * gq);
            float T = 0.0f;
            for (int run = 0; SK_BLOCKS * run < gq; ++run) {
                float G[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int gg = 4 * run + q;
                    G[q] = gg < gq ? ld_cluster_f32(rowa + 4u * (uint32_t)gg, (uint32_t)sk_owner(gg, gq, KS)) : 0.0f;
                }
                const float R = __fadd_rn(__fadd_rn(__fadd_rn(G[0], G[1]), G[2]), G[3]);
                T = run == 0 ? R : __fadd_rn(T, R);
            }
            p.y[(int64_t)v * p.rows + crow0 + lr] = T;
        }
    }
    __syncwarp();
    cluster_sync();  // peers are done reading this CTA's group sums
}

// Tensor maps of one call: W as bytes [rows][nb][block bytes] in boxes of (block bytes, 4 blocks,
// 8 rows) -- blocks and rows past the end read as zeros -- and for Q6_K the prefix as u16 [rows]
// [prefix stride] in boxes of 8 entries x 8 rows.  Strides are multiples of 16 bytes (block bytes
// 144, 176, 208; the prefix stride a multiple of 8 entries), bases 16-byte aligned (checked by
// the caller); every copy starts at x = 0 (weights) or at a multiple of 8 entries (prefix).
template <int F>
qmd_status sk_tensor_maps(const QmvKParams &kp, SkParams &sp)
{
    const TensorMapEncodeFn enc = tensor_map_encoder();
    if (!enc)
        return fail(QMD_ERR_LAUNCH, "cuTensorMapEncodeTiled entry point", cudaErrorNotSupported);
    std::memset(&sp.wmap, 0, sizeof sp.wmap);
    std::memset(&sp.premap, 0, sizeof sp.premap);
    const cuuint32_t estr[3] = {1, 1, 1};
    const cuuint64_t wdim[3] = {(cuuint64_t)rl_block_bytes(F), (cuuint64_t)kp.nb, (cuuint64_t)kp.rows};
    const cuuint64_t wstr[2] = {(cuuint64_t)rl_block_bytes(F), (cuuint64_t)kp.row_bytes};
    const cuuint32_t wbox[3] = {(cuuint32_t)rl_block_bytes(F), (cuuint32_t)SK_BLOCKS, (cuuint32_t)SK_ROWS};
    if (enc(&sp.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(kp.W), wdim, wstr, wbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return fail(QMD_ERR_LAUNCH, "tensor map of the weights", cudaErrorInvalidValue);
    if (F == QMD_Q6_K_SPLIT) {
        const cuuint64_t pdim[2] = {(cuuint64_t)(kp.pre_bytes / 2), (cuuint64_t)kp.rows};
        const cuuint64_t pstr[1] = {(cuuint64_t)kp.pre_bytes};
        const cuuint32_t pbox[2] = {8u, (cuuint32_t)SK_ROWS};
        if (enc(&sp.premap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint8_t *>(kp.Wpre), pdim, pstr, pbox,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return fail(QMD_ERR_LAUNCH, "tensor map of the Q6_K prefix", cudaErrorInvalidValue);
    }
    return QMD_OK;
}

// Launch with the plan's cluster size as a programmatic dependent of the previous kernel.  The
// plan's grid (a whole number of clusters) was sized for one CTA per SM; where fewer clusters
// of this shape can be resident at once (a cluster's CTAs share one GPU processing cluster),
// the grid shrinks to those and each cluster's range grows, so the group-sum buffer grows with
// it and the ring gives up slots where both no longer fit.
template <int F, auto Kern>
qmd_status launch_sk_kernel(SkParams sp, const QmvPlan &plan, int batch, cudaStream_t s)
{
    auto kern = Kern;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return QMD_ERR_DEVICE;
    const int KS = plan.ksplit;
    const int gq = (sp.k.nb + SK_BLOCKS - 1) / SK_BLOCKS;
    const int nbs = SK_BLOCKS * ((gq + KS - 1) / KS);
    const int64_t ntiles = (sp.k.rows + SK_ROWS - 1) / SK_ROWS;
    struct Fit {
        int dev, ks, threads, smem, clusters;
    };
    static std::mutex mu;
    static int set_bytes[64] = {0};
    static Fit fits[16] = {};
    static int n_fit = 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)KS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3((unsigned)plan.threads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & LAUNCH_NO_PDL) ? 1 : 2;
    int64_t nc = plan.grid / KS;
    int tiles_c = plan.tiles_c, smem = plan.smem, stages = plan.stages;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int pass = 0; pass < 3; ++pass) {
            if (set_bytes[dev] < smem) {
                cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                if (e != cudaSuccess)
                    return fail(QMD_ERR_LAUNCH, "split-K smem attribute", e);
                set_bytes[dev] = smem;
            }
            int fit = 0;
            for (int i = 0; i < n_fit && i < 16; ++i)
                if (fits[i].dev == dev && fits[i].ks == KS && fits[i].threads == plan.threads && fits[i].smem == smem)
                    fit = fits[i].clusters;
            if (fit == 0) {
                cfg.gridDim = dim3((unsigned)(nc * KS));
                cfg.dynamicSmemBytes = (size_t)smem;
                cudaError_t e = cudaOccupancyMaxActiveClusters(&fit, kern, &cfg);
                if (e != cudaSuccess)
                    return fail(QMD_ERR_LAUNCH, "split-K cluster occupancy", e);
                if (fit < 1)
                    return QMD_ERR_SHAPE;
                fits[n_fit % 16] = Fit{dev, KS, plan.threads, smem, fit};
                ++n_fit;
            }
            if (nc <= fit)
                break;
            // fewer clusters at once than the plan assumed: longer ranges, more group sums, and
            // a shallower ring where the deeper one no longer fits
            nc = fit;
            tiles_c = (int)((ntiles + nc - 1) / nc);
            DeviceInfo di;
            if (current_device(&di) != QMD_OK)
                return QMD_ERR_DEVICE;
            int budget = di.smem_per_sm - 1024;
            if (budget > di.smem_optin)
                budget = di.smem_optin;
            for (; stages >= 1; --stages)
                if (qmv_sk_layout(F, plan.WR, stages, batch, nbs, SK_ROWS * tiles_c, gq).total <= budget)
                    break;
            if (stages < 1)
                return QMD_ERR_SHAPE;
            smem = qmv_sk_layout(F, plan.WR, stages, batch, nbs, SK_ROWS * tiles_c, gq).total;
        }
        if (set_bytes[dev] < smem) {  // (a range grown on the last pass)
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess)
                return fail(QMD_ERR_LAUNCH, "split-K smem attribute", e);
            set_bytes[dev] = smem;
        }
    }
    sp.k.stages = stages;
    if (sp.k.pre_steps > stages)
        sp.k.pre_steps = stages;
    sp.tiles_c = tiles_c;
    sp.ks = KS;
    cfg.gridDim = dim3((unsigned)(nc * KS));
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, sp);
    if (e != cudaSuccess)
        return fail(QMD_ERR_LAUNCH, "split-K launch", e);
    return QMD_OK;
}

template <int F>
qmd_status launch_qmv_sk(const QmvKParams &kp, const QmvPlan &plan, int mode, int batch, cudaStream_t s)
{
    SkParams sp;
    sp.k = kp;
    sp.ks = plan.ksplit;
    sp.tiles_c = plan.tiles_c;
    const qmd_status st = sk_tensor_maps<F>(kp, sp);
    if (st != QMD_OK)
        return st;
    const bool pack = mode == QMV_PACK;
    if (mode != QMV_PACK && mode != QMV_PLAIN)
        return QMD_ERR_SHAPE;
    switch (batch) {
    case 1:
        return pack ? launch_sk_kernel<F, qmv_sk_kernel<F, 1, true>>(sp, plan, 1, s)
                    : launch_sk_kernel<F, qmv_sk_kernel<F, 1, false>>(sp, plan, 1, s);
    case 2:
        return pack ? launch_sk_kernel<F, qmv_sk_kernel<F, 2, true>>(sp, plan, 2, s)
                    : launch_sk_kernel<F, qmv_sk_kernel<F, 2, false>>(sp, plan, 2, s);
    }
    return QMD_ERR_BATCH;
}

}  // namespace qmd
