// Host-only check of the split-K kernel's partition and shared-memory layout arithmetic, from the
// kernel's own header: the K slices of a row (sk_g0, sk_owner), the clusters' tile ranges
// (sk_cluster_tiles) and the layout (qmv_sk_layout).  Prints "ok" and exits 0, or names the first
// case that fails and exits 1.  No device code runs.
#include <cstdio>
#include <cstdlib>

#include "qmv_splitk.cuh"

using namespace qmd;

static int fail(const char *what, long a, long b, long c)
{
    std::printf("FAIL %s (%ld, %ld, %ld)\n", what, a, b, c);
    return 1;
}

int main()
{
    // Every row's gq groups split over KS ranks: contiguous, in order, none empty, none longer
    // than ceil(gq / KS) (the activation space each CTA reserves), every group owned by the rank
    // whose slice holds it.
    for (int nb = 1; nb <= 256; ++nb) {
        const int gq = (nb + SK_BLOCKS - 1) / SK_BLOCKS;
        for (int KS = 2; KS <= SK_MAX_SPLIT && KS <= gq; ++KS) {
            if (sk_g0(0, gq, KS) != 0 || sk_g0(KS, gq, KS) != gq)
                return fail("slices do not span the row", nb, KS, gq);
            for (int k = 0; k < KS; ++k) {
                const int n = sk_g0(k + 1, gq, KS) - sk_g0(k, gq, KS);
                if (n < 1 || n > (gq + KS - 1) / KS)
                    return fail("slice size", nb, KS, k);
            }
            for (int g = 0; g < gq; ++g) {
                const int o = sk_owner(g, gq, KS);
                if (o < 0 || o >= KS || sk_g0(o, gq, KS) > g || g >= sk_g0(o + 1, gq, KS))
                    return fail("owner", nb, KS, g);
            }
        }
    }
    // The clusters' tile ranges: contiguous, in order, covering every tile once, none longer than
    // ceil(ntiles / NC) (what the plan sizes the group sums by).
    for (long ntiles = 1; ntiles <= 3000; ntiles += (ntiles < 300 ? 1 : 37)) {
        for (long NC = 1; NC <= 152 && NC <= ntiles; ++NC) {
            int64_t prev = 0;
            for (long cid = 0; cid < NC; ++cid) {
                int64_t c0, c1;
                sk_cluster_tiles(cid, NC, ntiles, &c0, &c1);
                if (c0 != prev || c1 <= c0 || c1 - c0 > (ntiles + NC - 1) / NC)
                    return fail("cluster tiles", ntiles, NC, cid);
                prev = c1;
            }
            if (prev != ntiles)
                return fail("cluster tiles do not cover", ntiles, NC, prev);
        }
    }
    // The layout: regions in order and aligned (ring slots on 128 bytes, barriers on 8, the rest
    // on 16), each region holding what the kernel indexes in it, the total covering the last.
    const int fmts[3] = {QMD_Q4_K, QMD_Q5_K, QMD_Q6_K_SPLIT};
    for (int f : fmts) {
        if (sk_slot_bytes(f) % 128 != 0 || sk_box_bytes(f) != SK_ROWS * SK_BLOCKS * rl_block_bytes(f))
            return fail("slot", f, sk_slot_bytes(f), 0);
        for (int W = 1; W <= SK_MAX_WARPS; ++W)
            for (int S = 1; S <= 4; ++S)
                for (int B = 1; B <= SK_MAX_BATCH; ++B)
                    for (int gq = 1; gq <= 64; gq += 3)
                        for (int rows_c = 8; rows_c <= 512; rows_c *= 2) {
                            const int nbs = SK_BLOCKS * gq;
                            const SkLayout L = qmv_sk_layout(f, W, S, B, nbs, rows_c, gq);
                            if (L.bar_off != W * S * sk_slot_bytes(f) || L.bar_off % 8 != 0)
                                return fail("barriers", f, W, S);
                            if (L.act_off < L.bar_off + W * S * 8 || L.act_off % 16 != 0)
                                return fail("codes", f, W, S);
                            if (L.dx_off < L.act_off + B * nbs * RL_ACT || L.dx_off % 16 != 0)
                                return fail("scales", f, B, nbs);
                            if (L.aux_off < L.dx_off + B * nbs * 4 || L.aux_off % 16 != 0)
                                return fail("sums", f, B, nbs);
                            const int aux = B * nbs * (f == QMD_Q6_K_SPLIT ? 16 : 8) * 2;
                            if (L.part_off < L.aux_off + aux || L.part_off % 16 != 0)
                                return fail("group sums", f, B, nbs);
                            if (L.total < L.part_off + B * rows_c * gq * 4 || L.total % 16 != 0)
                                return fail("total", f, rows_c, gq);
                        }
    }
    std::printf("ok\n");
    return 0;
}
