// api.cu -- the C ABI of libqmd: argument validation, launch planning, the device error word.
//
// Every entry point validates its arguments on the host and returns a named status before
// anything is launched ("One kernel, any device", §1: a refused launch carries one of seven
// named reasons; "Kernel SPI and the selection algorithm", "Why a kernel declines": a K-quant
// tensor whose last dimension is not a multiple of 256 is rejected).  There is no fallback
// path: a refused call does nothing.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "qmv_splitk.cuh"

namespace qmd {

// One word per device, set by kernels whose bounded waits give up.  A file-scope device
// variable: the library never allocates.
static __device__ unsigned int g_error_word;

// The scheduling workspace of qmd_qmatvec_x_static: one QMD_WORKSPACE_BYTES workspace per device,
// a file-scope device array that every device loading the library holds until the process ends.
// Host code must not pass its name to a kernel (on the host it stands in for the array, it is not
// a device address): the address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned int g_static_ws[QMD_WORKSPACE_BYTES / 4];

static thread_local char g_detail[320];
static std::atomic<unsigned long long> g_wait_ns{1000000000ull};
static std::atomic<int> g_force_rg{0}, g_force_rows{0}, g_force_stages{0}, g_force_cps{0};
static std::atomic<int> g_force_split{0};  // split-K: CTAs per cluster (0: the default plan)
// Per mille of a row-lane launch's tiles handed out by claims when a workspace is given
// (measured on the 7B shapes; qmd_debug_set_dynamic_tiles overrides it).
static constexpr int DYN_PERMILLE = 250;
static std::atomic<int> g_dyn_permille{-1};

int64_t dynamic_tiles(int64_t tiles)
{
    const int pm = g_dyn_permille.load() >= 0 ? g_dyn_permille.load() : DYN_PERMILLE;
    return tiles * pm / 1000;
}

qmd_status fail(qmd_status st, const char *what, cudaError_t e)
{
    snprintf(g_detail, sizeof g_detail, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    (void)cudaGetLastError();  // clear a non-sticky launch error
    return st;
}

uint64_t wait_limit_ns() { return g_wait_ns.load(); }

static std::atomic<unsigned> g_launch_flags{0};
unsigned launch_flags() { return g_launch_flags.load(); }

qmd_status current_device(DeviceInfo *out)
{
    static DeviceInfo cache[64];
    static std::atomic<bool> have[64];
    static std::mutex fill;  // the first call per device fills its entry
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(QMD_ERR_DEVICE, "cudaGetDevice", e);
    if (dev < 0 || dev >= 64)
        return QMD_ERR_DEVICE;
    if (!have[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(fill);
        if (have[dev].load(std::memory_order_acquire)) {
            *out = cache[dev];
            return QMD_OK;
        }
        DeviceInfo d = {};
        d.device = dev;
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return fail(QMD_ERR_DEVICE, "cudaDeviceGetAttribute", e);
        if (d.cc_major != 10 || d.cc_minor != 3) {
            snprintf(g_detail, sizeof g_detail, "device %d is sm_%d%d; libqmd is built for sm_103a only", dev,
                     d.cc_major, d.cc_minor);
            return QMD_ERR_DEVICE;
        }
        cache[dev] = d;
        have[dev].store(true, std::memory_order_release);
    }
    *out = cache[dev];
    return QMD_OK;
}

unsigned *device_error_word()
{
    static std::atomic<unsigned *> addr[64];
    static std::mutex fill;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    if (addr[dev].load(std::memory_order_acquire) == nullptr) {
        std::lock_guard<std::mutex> lock(fill);
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_error_word);
        if (e != cudaSuccess) {
            fail(QMD_ERR_DEVICE, "cudaGetSymbolAddress(error word)", e);
            return nullptr;
        }
        addr[dev].store(static_cast<unsigned *>(p), std::memory_order_release);
    }
    return addr[dev].load(std::memory_order_acquire);
}

#ifdef QMD_TRACE
// Traced build: one caller-owned device buffer of stamp records; each launch takes the next
// `ctas` records and logs (first record, CTAs) on the host, in launch (or capture) order.
static std::mutex g_trace_mu;
static unsigned long long *g_trace_buf = nullptr;
static int64_t g_trace_cap = 0, g_trace_used = 0;
static std::vector<int64_t> g_trace_log;

unsigned long long *trace_reserve(int ctas)
{
    std::lock_guard<std::mutex> lock(g_trace_mu);
    if (!g_trace_buf || ctas < 1 || g_trace_used + ctas > g_trace_cap)
        return nullptr;
    unsigned long long *p = g_trace_buf + g_trace_used * QMD_TRACE_FIELDS;
    g_trace_log.push_back(g_trace_used);
    g_trace_log.push_back(ctas);
    g_trace_used += ctas;
    return p;
}
#endif

// Device address of g_static_ws on the current device, looked up on the first call there (with
// that device current) and kept; NULL, with the reason recorded, if the lookup fails.
static unsigned *static_workspace()
{
    static std::atomic<unsigned *> addr[64];
    static std::mutex fill;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    if (addr[dev].load(std::memory_order_acquire) == nullptr) {
        std::lock_guard<std::mutex> lock(fill);
        if (addr[dev].load(std::memory_order_acquire) == nullptr) {
            void *p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
            if (e != cudaSuccess || p == nullptr) {
                fail(QMD_ERR_DEVICE, "cudaGetSymbolAddress(static workspace)", e);
                return nullptr;
            }
            addr[dev].store(static_cast<unsigned *>(p), std::memory_order_release);
        }
    }
    return addr[dev].load(std::memory_order_acquire);
}

// Rows per row group per stage: 8 at one or two vectors, 4 at three or four, 2 above (16 (row,
// vector) slots per warp from two vectors up; measured on the 7B shapes with the CTA counts
// chosen below).
static int default_rows_per_stage(bool q6, int batch)
{
    (void)q6;
    if (batch <= 2)
        return 8;
    if (batch <= 4)
        return 4;
    return 2;
}

// Registers per thread of a dp4a kernel instance, looked up once per (format, batch, rows per
// stage, mode); if the lookup fails, the launch bound's worst case.
static int kernel_regs(int fmt, int batch, int PR, int mode)
{
    static std::atomic<int> cache[3][QMD_MAX_BATCH + 1][4][4];
    const int fi = fmt == QMD_Q6_K_SPLIT ? 2 : fmt == QMD_Q5_K ? 1 : 0;
    const int pi = PR >= 8 ? 3 : PR >= 4 ? 2 : PR >= 2 ? 1 : 0;
    if (batch < 1 || batch > QMD_MAX_BATCH || mode < 0 || mode > 3)
        return 65536 / qmv_max_threads(batch, PR, mode);
    std::atomic<int> &slot = cache[fi][batch][pi][mode];
    int r = slot.load();
    if (r == 0) {
        r = fi == 2 ? qmv_regs_q6k(batch, PR, mode) : fi == 1 ? qmv_regs_q5k(batch, PR, mode)
                                                     : qmv_regs_q4k(batch, PR, mode);
        if (r <= 0)
            r = 65536 / qmv_max_threads(batch, PR, mode);
        slot.store(r);
    }
    return r;
}

// CTAs of `threads` threads that fit on an SM by registers (allocated per thread in units of 8)
// and by threads.
static int reg_cap_ctas(int regs, int threads)
{
    const int r = (regs + 7) & ~7;
    int cap = 65536 / (r * threads);
    if (cap > 2048 / threads)
        cap = 2048 / threads;
    return cap < 1 ? 1 : cap;
}

// Ring depth and CTAs per SM for a stage geometry; false if nothing fits.
static bool fit_stages(const DeviceInfo &dev, int64_t rows, int TR, int stage_bytes, int per_stage_extra,
                       int fixed, int cps, int max_stages, QmvPlan *pl)
{
    for (; cps >= 1; --cps) {
        int budget = dev.smem_per_sm / cps - 1024;
        if (budget > dev.smem_optin)
            budget = dev.smem_optin;
        int64_t grid = (int64_t)dev.sm_count * cps;
        if (grid > rows)
            grid = rows;
        const int64_t rows_per_cta = (rows + grid - 1) / grid;
        const int64_t chunks = (rows_per_cta + TR - 1) / TR;
        int64_t stages = (budget - fixed) / (stage_bytes + per_stage_extra);
        if (stages > max_stages)
            stages = max_stages;
        if (stages > chunks)
            stages = chunks;
        if (g_force_stages.load() > 0 && stages > g_force_stages.load())
            stages = g_force_stages.load();
        if (stages < 1)
            continue;
        pl->grid = (int)grid;
        pl->stages = (int)stages;
        return true;
    }
    return false;
}

// Row-lane kernel (qmv_rl.cuh): one CTA per SM (more when forced), a ring for as many warps as
// the CTA has 2-row tiles up to 16, the deepest ring (up to 4 steps per warp -- 2 for one vector
// and rows of one step -- no more than a warp has steps) that fits beside the activations, up to
// 16 warps to pack them, and one more warp that requests the rings' first fills.  false if
// nothing fits (very long rows).
static bool rl_plan(int fmt, int64_t rows, int nb, int batch, const DeviceInfo &dev, QmvPlan *pl, bool norm)
{
    const int64_t tiles = (rows + RL_ROWS - 1) / RL_ROWS;
    const int nsteps = (nb + RL_BLOCKS - 1) / RL_BLOCKS;
    const int cps = g_force_cps.load() > 0 ? g_force_cps.load() : 1;
    int64_t grid = (int64_t)dev.sm_count * cps;
    if (grid > tiles)
        grid = tiles;
    const int64_t per_cta = (tiles + grid - 1) / grid;
    const int wmax = rl_max_warps(batch);
    // One vector and rows of one step (at most 16 blocks): rings of 2.  Measured on the 32-layer
    // step (gate|up is the projection it changes; q|k|v and o have 1-2 steps a warp): 4357 ->
    // 4553 GB/s; rings of 1 4331.  (An 8-warp CTA for q|k|v and o with every slot requested
    // before the wait, faster in chains of one projection, lost in the step: 4430-4542.)
    const bool forced = g_force_rg.load() > 0 || g_force_stages.load() > 0 || g_force_rows.load() > 0;
    const bool ring2 = batch == 1 && nsteps == 1 && !norm && !forced && !(launch_flags() & LAUNCH_RL_DEEP);
    int W = g_force_rg.load() > 0 ? g_force_rg.load() : (int)(per_cta < wmax ? per_cta : wmax);
    if (W > wmax)
        W = wmax;
    if (W < 1)
        W = 1;
    int budget = dev.smem_per_sm / cps - 1024;
    if (budget > dev.smem_optin)
        budget = dev.smem_optin;
    const int64_t steps = (per_cta + W - 1) / W * nsteps;  // most steps a warp has
    int S = g_force_stages.load() > 0 ? g_force_stages.load() : ring2 ? 2 : 4;
    if (S > steps)
        S = (int)steps;
    for (; S >= 1; --S)
        if (qmv_rl_layout(fmt, W, S, batch, nb, norm).total <= budget)
            break;
    if (S < 1)
        return false;
    // every warp of the CTA packs (or loads) the activations: at least as many warps as blocks to
    // pack, up to 16, even where fewer warps have tiles
    int NW = W;
    const int64_t blocks = (int64_t)batch * nb;
    const int want = (int)(blocks < wmax ? blocks : wmax);
    if (g_force_rg.load() <= 0 && NW < want)
        NW = want;
    if (norm && NW < 8)  // the RMSNorm form sums the squares with 256 threads
        NW = 8;
    pl->layout = 2;
    pl->grid = (int)grid;
    pl->threads = 32 * (NW + 1);  // plus the warp that requests the first ring fills
    pl->smem = qmv_rl_layout(fmt, W, S, batch, nb, norm).total;
    pl->stages = S;
    pl->WR = W;
    pl->RG = 1;
    pl->PR = RL_ROWS;
    pl->stage_bytes = rl_slot_bytes(fmt);
    // ring slots per warp requested before the dependency wait (the rest after the pack); a
    // forced rows-per-stage value stands for this count here
    // ...and of those, launches with few tiles per CTA (q|k|v) request one slot per warp before
    // the wait instead of two: measured inside the 32-layer step, 4547 -> 4572 GB/s (gate|up, with
    // many tiles, lost: 4547 -> 4457); the requests then compete less with the previous launch's
    // last reads.
    const int pre = g_force_rows.load() > 0                  ? g_force_rows.load()
                    : (ring2 && per_cta <= RL_FEW_TILES) ? 1
                                                             : RL_PRE_STEPS;
    pl->pre_steps = pre < S ? pre : S;
    return true;
}

// Split-K kernel (qmv_splitk.cuh): clusters of KS CTAs, one CTA per SM, each cluster a range of
// 8-row tiles and each CTA one of KS slices of every row's groups of four blocks; a ring for as
// many warps as the range has tiles up to 16 (or the forced row-group count), the deepest ring up to 4 steps (no more than a warp
// has) that fits beside the activations and the group sums, and up to 16 warps to pack the
// slice's activations.  false where it does not apply: more than two vectors, fewer groups than
// slices, or nothing fits.
static bool sk_plan(int fmt, int64_t rows, int nb, int batch, int KS, const DeviceInfo &dev, QmvPlan *pl)
{
    const int gq = (nb + SK_BLOCKS - 1) / SK_BLOCKS;
    if (batch > SK_MAX_BATCH || KS < 2 || KS > SK_MAX_SPLIT || KS > gq)
        return false;
    const int64_t ntiles = (rows + SK_ROWS - 1) / SK_ROWS;
    int64_t nc = dev.sm_count / KS;
    if (nc > ntiles)
        nc = ntiles;
    if (nc < 1)
        return false;
    const int64_t tiles_c = (ntiles + nc - 1) / nc;
    if (tiles_c > (1 << 20))
        return false;
    int W = (int)(tiles_c < SK_MAX_WARPS ? tiles_c : SK_MAX_WARPS);
    if (g_force_rg.load() > 0)
        W = g_force_rg.load() < SK_MAX_WARPS ? g_force_rg.load() : SK_MAX_WARPS;
    const int gs = (gq + KS - 1) / KS;  // the most groups a slice has
    const int nbs = SK_BLOCKS * gs;
    int budget = dev.smem_per_sm - 1024;
    if (budget > dev.smem_optin)
        budget = dev.smem_optin;
    const int64_t steps = (tiles_c + W - 1) / W * gs;  // most steps a warp has
    int S = g_force_stages.load() > 0 ? g_force_stages.load() : 4;
    if (S > steps)
        S = (int)steps;
    for (; S >= 1; --S)
        if (qmv_sk_layout(fmt, W, S, batch, nbs, (int)(SK_ROWS * tiles_c), gq).total <= budget)
            break;
    if (S < 1)
        return false;
    const int want = batch * nbs < SK_MAX_WARPS ? batch * nbs : SK_MAX_WARPS;
    const int NW = W > want ? W : want;
    pl->layout = 3;
    pl->grid = (int)(nc * KS);
    pl->threads = 32 * NW;
    pl->smem = qmv_sk_layout(fmt, W, S, batch, nbs, (int)(SK_ROWS * tiles_c), gq).total;
    pl->stages = S;
    pl->WR = W;
    pl->RG = 1;
    pl->PR = SK_ROWS;
    pl->stage_bytes = sk_slot_bytes(fmt);
    pl->ksplit = KS;
    pl->tiles_c = (int)tiles_c;
    // ring slots per warp requested before the dependency wait (a forced rows-per-stage value
    // stands for this count here)
    const int pre = g_force_rows.load() > 0 ? g_force_rows.load() : RL_PRE_STEPS;
    pl->pre_steps = pre < S ? pre : S;
    return true;
}

qmd_status qmv_plan(int fmt, int64_t rows, int nb, int batch, const DeviceInfo &dev, QmvPlan *pl, int mode)
{
    const bool q6 = fmt == QMD_Q6_K_SPLIT;
    const bool norm = mode == QMV_NORM;
    const bool fused = mode == QMV_PACK || norm;  // the CTAs pack the activations themselves
    const int row_bytes = nb * (q6 ? 208 : fmt == QMD_Q5_K ? 176 : 144);
    const int pre_bytes = q6 ? align_up(nb, 8) * 2 : 0;
    pl->row_bytes = row_bytes;
    pl->pre_bytes = pre_bytes;
    pl->row_stride = row_bytes;
    // Tensor-core kernel.  Chosen where it was measured faster -- Q4_K / Q5_K rows of at most 16
    // blocks at 5..8 vectors, and at 3..4 where its 32-row tiles give every CTA many rows (Q6_K's
    // 14336-wide down projection: 24.4 us against 24.9 on dp4a at 8 vectors, kept on dp4a) --
    // and for rows the dp4a kernel cannot take (more than 128 blocks at one or two vectors, 64
    // above), which it walks run by run.  One warp per block of a run of 16 blocks, each with its own ring of tiles;
    // about 16 warps per SM.  Tiles of 32 rows (rings of 2) where that gives no CTA more rows
    // than tiles of 16 do and the rings fit (rows of one run, not Q6_K), else tiles of 16 rows with the deepest
    // ring (3 or 4 tiles per warp) that fits beside the run sums (and, fused, the packed
    // activations).  A forced ring cap of 2 asks for 32-row tiles, of 3 or more caps the 16-row
    // ring, of 1 selects the dp4a kernel, and so does a shape that does not fit.  The RMSNorm
    // form exists in the row-lane and dp4a kernels, not in this one.
    const int fst = g_force_stages.load();
    pl->tc_rows = 0;
    // One or two vectors: the row-lane kernel, unless a test flag asks for another kernel (three
    // and four on it too when a flag asks).
    // Split-K where asked (plain and fused forms, one or two vectors, rows of at least as many
    // groups of four blocks as slices).
    pl->ksplit = 0;
    pl->tiles_c = 0;
    if ((mode == QMV_PLAIN || mode == QMV_PACK) && g_force_split.load() >= 2 &&
        sk_plan(fmt, rows, nb, batch, g_force_split.load(), dev, pl))
        return QMD_OK;
    const bool rl_batch = batch <= RL_DEFAULT_BATCH || ((launch_flags() & LAUNCH_RL) && batch <= RL_MAX_BATCH);
    if (rl_batch && !(launch_flags() & (LAUNCH_SLICE | LAUNCH_TC_ALL)) &&
        rl_plan(fmt, rows, nb, batch, dev, pl, mode == QMV_NORM))
        return QMD_OK;
    // Three and four vectors: the tensor cores only where 32-row tiles give every CTA many rows
    // (measured on the 7B shapes: gate|up 18.5 against 20.3 us on dp4a at four vectors; q|k|v
    // 7.7 against 6.8 and o 5.3 against 5.3, whose CTAs have 27-40 rows)
    bool tall = false;
    if (batch >= TC_MIN_BATCH_TALL && batch < TC_MIN_BATCH && nb <= TC_RUN && fmt != QMD_Q6_K_SPLIT) {
        const int rw = nb < TC_RUN ? nb : TC_RUN;
        const int64_t cta = (int64_t)dev.sm_count * (16 / rw > 0 ? 16 / rw : 1);
        const int64_t t16 = (rows + TC_ROWS - 1) / TC_ROWS, t32 = (rows + 2 * TC_ROWS - 1) / (2 * TC_ROWS);
        const int64_t g16 = cta < t16 ? cta : t16, g32 = cta < t32 ? cta : t32;
        const int64_t rp16 = (t16 + g16 - 1) / g16 * TC_ROWS, rp32 = (t32 + g32 - 1) / g32 * 2 * TC_ROWS;
        tall = rp32 <= rp16 && rp32 >= TC_TALL_ROWS;
    }
    const bool tc_faster = (batch >= TC_MIN_BATCH || tall) && nb <= TC_RUN && fmt != QMD_Q6_K_SPLIT;
    const bool dp4a_cannot = nb > (batch <= 2 ? 128 : 64);
    const bool tc_forced = (launch_flags() & LAUNCH_TC_ALL) && batch >= 3;
    if (!norm && (tc_faster || dp4a_cannot || tc_forced) && !(launch_flags() & LAUNCH_DP4A_ONLY) &&
        (fst <= 0 || fst >= 2)) {
        const int RW = nb < TC_RUN ? nb : TC_RUN;
        int cps = g_force_cps.load() > 0 ? g_force_cps.load() : (16 / RW > 0 ? 16 / RW : 1);
        if (cps > 8)
            cps = 8;
        int st = 0;
        int64_t grid = 0, rows_pad = 0;
        for (; cps >= 1; --cps) {
            int budget = dev.smem_per_sm / cps - 1024;
            if (budget > dev.smem_optin)
                budget = dev.smem_optin;
            // CTAs and rows per CTA for tiles of th rows: every CTA takes whole tiles
            auto split = [&](int th, int64_t *g, int64_t *rp) {
                const int64_t nt = (rows + th - 1) / th;
                *g = (int64_t)dev.sm_count * cps < nt ? (int64_t)dev.sm_count * cps : nt;
                *rp = (rows + th * *g - 1) / (th * *g) * th;
            };
            int64_t g16, rp16, g32, rp32;
            split(TC_ROWS, &g16, &rp16);
            split(2 * TC_ROWS, &g32, &rp32);
            st = 0;
            const bool try32 = fmt != QMD_Q6_K_SPLIT && nb <= TC_RUN && (fst == 2 || (fst <= 0 && rp32 <= rp16));
            if (try32 && rp32 <= (1 << 16) && qmv_tc_layout(2, fmt, nb, batch, fused, (int)rp32).total <= budget) {
                st = 2;
                grid = g32;
                rows_pad = rp32;
                break;
            }
            if (fst != 2 && rp16 <= (1 << 16))
                for (st = 4; st >= 3; --st)
                    if ((fst <= 0 || st <= fst) && qmv_tc_layout(st, fmt, nb, batch, fused, (int)rp16).total <= budget)
                        break;
            if (st >= 3) {
                grid = g16;
                rows_pad = rp16;
                break;
            }
        }
        if (cps >= 1 && st >= 2) {  // otherwise the dp4a kernel below takes the call
            pl->layout = 1;
            pl->grid = (int)grid;
            pl->stages = st;
            pl->threads = 32 * RW;
            pl->smem = qmv_tc_layout(st, fmt, nb, batch, fused, (int)rows_pad).total;
            pl->WR = RW;
            pl->RG = 1;
            pl->PR = tc_tile_rows(st);
            pl->stage_bytes = tc_slot_bytes(fmt, tc_tile_rows(st));
            pl->tc_rows = (int)rows_pad;
            // one ring slot per warp requested before the dependency wait, the rest once the
            // warp's activation fragments are loaded (the fragments' loads otherwise arrive behind
            // every SM's pre-wait copies): 32-layer step at 8 / 4 vectors 2137 / 2774 GB/s with
            // the whole ring before the wait, 2159 / 2851 with one slot, 2018 / 2705 with none
            pl->pre_steps = 1;
            return QMD_OK;
        }
    }
    // A warp covers 4 blocks of a row, 8 lanes per block; a row takes ceil(nb / 4) warps.
    const int WR = (nb + 3) / 4;
    int PR = g_force_rows.load() > 0 ? g_force_rows.load() : default_rows_per_stage(q6, batch);
    while (PR & (PR - 1))  // the slice kernel is built for 1, 2, 4 or 8 rows
        PR &= PR - 1;
    while (PR > 1 && PR * batch > 16)
        PR >>= 1;
    // more than 8 (row, vector) slots per warp lower the launch bound to 512 threads; long rows
    // keep 8 slots and the 1024-thread bound
    while (PR > 1 && PR * batch > 8 && WR * 32 > qmv_max_threads(batch, PR, mode))
        PR >>= 1;
    const int max_threads = qmv_max_threads(batch, PR, mode);  // the kernel's launch bound
    if (WR * 32 > max_threads)
        return QMD_ERR_SHAPE;
    const int slots = PR * batch > 8 ? 16 : 8;
    // Row groups per CTA: 1, except in the fused form at batch 1 (below).
    int RG = g_force_rg.load() > 0 ? g_force_rg.load() : 1;
    // CTAs per SM: about 32 warps per SM (the kernel is bound by instruction latency, so warps
    // matter more than stage depth); capped at launch by the occupancy calculator.
    int cps = g_force_cps.load() > 0 ? g_force_cps.load() : 0;
    const int64_t per_sm = (rows + dev.sm_count - 1) / dev.sm_count;
    if (fused && batch == 1) {
        // Every CTA packs the whole f32 vector for itself, after the dependency wait, so the
        // pack's latency is on the critical path of every launch.  Measured on the 7B shapes:
        //  * few rows per SM (up to two 8-row stages per row group): wide CTAs of at least 16
        //    warps (two row groups at least), each streaming its rows as one chunk, one or two
        //    CTAs per SM -- the pack then costs one block per warp;
        //  * many rows per SM: 8-warp CTAs, about 32 warps per SM, several chunks each;
        //  * a stage of at most 96 KB, so that two fit in an SM's shared memory.
        int rg_small = 16 / WR > 2 ? 16 / WR : 2;
        if (rg_small * WR * 32 > max_threads)
            rg_small = max_threads / (WR * 32);
        if (rg_small < 1)
            rg_small = 1;
        const bool small = per_sm <= 2 * rg_small * 8;
        if (g_force_rg.load() <= 0)
            RG = small ? rg_small : (8 / WR > 1 ? 8 / WR : 1);
        if (g_force_rows.load() <= 0)
            while (PR > 1 && (int64_t)RG * PR * (row_bytes + pre_bytes) > 96 * 1024)
                PR >>= 1;
        if (cps <= 0) {
            const int rgc = RG < max_threads / (WR * 32) ? RG : max_threads / (WR * 32);
            const int tr = rgc * PR;
            cps = small ? (int)((per_sm + tr - 1) / (tr > 0 ? tr : 1)) : 32 / (rgc * WR);
            const int cap = reg_cap_ctas(kernel_regs(fmt, batch, PR, mode), rgc * WR * 32);
            if (cps > cap)
                cps = cap;
            if (cps < 1)
                cps = 1;
        }
    } else if (batch <= 4) {
        // Packed input, one to four vectors: 8-warp CTAs (one row group per 8 warps of a row), as
        // many per SM as the registers allow but no more than it takes for each CTA to stream
        // its rows as one chunk (measured on the 7B shapes at batches 1, 2 and 4).
        if (g_force_rg.load() <= 0)
            RG = 8 / WR > 1 ? 8 / WR : 1;
        if (cps <= 0) {
            const int rgc = RG < max_threads / (WR * 32) ? RG : max_threads / (WR * 32);
            const int tr = (rgc > 0 ? rgc : 1) * PR;
            const int64_t want = (per_sm + tr - 1) / tr;
            const int cap = reg_cap_ctas(kernel_regs(fmt, batch, PR, mode), (rgc > 0 ? rgc : 1) * WR * 32);
            cps = want < cap ? (int)want : cap;
            if (cps < 1)
                cps = 1;
        }
    }
    if (RG * WR * 32 > max_threads)
        RG = max_threads / (WR * 32);
    if (RG < 1)
        RG = 1;
    // The RMSNorm form sums the squares with the first 256 threads of each CTA.
    if (norm && RG * WR < 8)
        RG = (8 + WR - 1) / WR;
    if (norm && RG * WR * 32 > max_threads)
        return QMD_ERR_SHAPE;
    const int TR = RG * PR;
    const int64_t sb64 = (int64_t)TR * (row_bytes + pre_bytes);
    if (sb64 > dev.smem_optin)
        return QMD_ERR_SHAPE;
    const int stage_bytes = align_up((int)sb64, 128);
    const int extra = RG * WR * slots * 4 + 16;  // partials + counter + barrier per stage
    if (cps <= 0)
        cps = 32 / (RG * WR) > 0 ? 32 / (RG * WR) : 1;
    if (cps > 8)
        cps = 8;
    const int fixed = qmv_smem_layout(0, stage_bytes, RG, WR, batch, nb, q6, fused, slots, norm).total + 64;
    // Ring depth: up to 8 stages, but 2 for two to four vectors -- bulk copies in flight together
    // share the SM's bandwidth, so a deeper ring delays its first stage, and the dot products,
    // with little headroom over the copies, never catch up (measured on the 7B shapes).
    const int max_stages = (g_force_stages.load() <= 0 && batch >= 2 && batch <= 4) ? 2 : 8;
    if (!fit_stages(dev, rows, TR, stage_bytes, extra, fixed, cps, max_stages, pl))
        return QMD_ERR_SHAPE;
    pl->layout = 0;
    pl->threads = RG * WR * 32;
    pl->smem = qmv_smem_layout(pl->stages, stage_bytes, RG, WR, batch, nb, q6, fused, slots, norm).total;
    pl->WR = WR;
    pl->RG = RG;
    pl->PR = PR;
    pl->stage_bytes = stage_bytes;
    return QMD_OK;
}

// Test-only: one CTA waits on a barrier nothing completes, gives up after limit_ns, flags it.
__global__ void debug_wait_kernel(unsigned *err, unsigned long long limit_ns)
{
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(b, 0, limit_ns);
    if (__syncthreads_or(!ok) && threadIdx.x == 0)
        atomicOr(err, ERRBIT_DEBUG_WAIT);
}

}  // namespace qmd

using namespace qmd;

namespace {

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qmd_status check_k(int64_t K)
{
    if (K < QMD_QK)
        return K > 0 && K % QMD_QK != 0 ? QMD_ERR_K_NOT_MULTIPLE_OF_256 : QMD_ERR_SHAPE;
    if (K % QMD_QK != 0)
        return QMD_ERR_K_NOT_MULTIPLE_OF_256;
    if (K / QMD_QK > (1 << 20))
        return QMD_ERR_SHAPE;
    return QMD_OK;
}

// Do [a, a + na) and [b, b + nb) bytes overlap?
inline bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return a && b && pa < pb + nb && pb < pa + na;
}

// Outputs a mat-vec writes while other CTAs may still read its inputs must not share bytes with
// them: y (every form) and the fused forms' packed copy xq_out against x, r and the packed input.
qmd_status outputs_apart(const float *y, int64_t rows, int batch, int64_t K, const float *x, const float *r,
                         qmd_q8k_const xq, qmd_q8k xq_out)
{
    const size_t nb = (size_t)(K / QMD_QK);
    const size_t yb = (size_t)batch * (size_t)rows * 4, vb = (size_t)batch * (size_t)K * 4;
    const size_t qsb = (size_t)batch * (size_t)K, db = (size_t)batch * nb * 4, bsb = (size_t)batch * nb * 16;
    const void *outs[4] = {y, xq_out.qs, xq_out.d, xq_out.bsums};
    const size_t outb[4] = {yb, qsb, db, bsb};
    const void *ins[5] = {x, r, xq.qs, xq.d, xq.bsums};
    const size_t inb[5] = {vb, vb, qsb, db, bsb};
    for (int o = 0; o < 4; ++o)
        for (int i = 0; i < 5; ++i)
            if (overlaps(outs[o], outb[o], ins[i], inb[i]))
                return QMD_ERR_VALUE;
    return QMD_OK;
}

// The RMSNorm form's extra arguments; g == NULL selects the other forms.
struct NormArgs {
    const float *r = nullptr;
    const float *g = nullptr;
    float eps = 0.0f;
    float *h_out = nullptr;
};

qmd_status qmatvec_common(qmd_fmt fmt, const void *W, const void *W_aux, qmd_q8k_const xq, float *y,
                          int64_t rows, int64_t K, int batch, int32_t *dots, int32_t *sm, bool dump,
                          const float *x, qmd_q8k xq_out, void *stream, const NormArgs &na = NormArgs(),
                          void *workspace = nullptr)
{
    if (fmt != QMD_Q4_K && fmt != QMD_Q5_K && fmt != QMD_Q6_K_SPLIT)
        return QMD_ERR_FORMAT;
    const bool q6 = fmt == QMD_Q6_K_SPLIT;
    const bool fused = x != nullptr;
    const bool want_out = xq_out.qs || xq_out.d || xq_out.bsums;
    if (!W || !y || (q6 && !W_aux) || (dump && (!dots || !sm)))
        return QMD_ERR_NULL;
    if (!fused && (!xq.qs || !xq.d || (!q6 && !xq.bsums)))
        return QMD_ERR_NULL;
    if (fused && want_out && (!xq_out.qs || !xq_out.d || !xq_out.bsums))
        return QMD_ERR_NULL;
    qmd_status st = check_k(K);
    if (st != QMD_OK)
        return st;
    if (batch < 1 || batch > QMD_MAX_BATCH)
        return QMD_ERR_BATCH;
    if (rows < 1 || rows > (int64_t)1 << 31)
        return QMD_ERR_SHAPE;
    const int nb = (int)(K / QMD_QK);
    if (!aligned(W, 16) || (q6 && !aligned(W_aux, 16)) || !aligned(y, 4) ||
        (!fused && (!aligned(xq.qs, 16) || (!q6 && !aligned(xq.bsums, 16)) || !aligned(xq.d, 4))) ||
        (fused && !aligned(x, 16)) ||
        (fused && want_out && (!aligned(xq_out.qs, 16) || !aligned(xq_out.bsums, 16) || !aligned(xq_out.d, 4))) ||
        (dump && (!aligned(dots, 16) || !aligned(sm, 16))) ||
        (na.g && (!aligned(na.g, 16) || (na.r && !aligned(na.r, 16)) || (na.h_out && !aligned(na.h_out, 16)))) ||
        (workspace && !aligned(workspace, 16)))
        return QMD_ERR_MISALIGNED;
    if (na.g) {
        if (!(na.eps >= 0.0f) || !(na.eps <= 3.4028234663852886e38f))  // rejects NaN, negatives and +inf
            return QMD_ERR_VALUE;
        // h is written by one CTA while every CTA still reads x and r: they must not share bytes
        const size_t vb = (size_t)batch * (size_t)K * sizeof(float);
        if (overlaps(na.h_out, vb, x, vb) || overlaps(na.h_out, vb, na.r, vb) ||
            overlaps(na.h_out, vb, na.g, (size_t)K * sizeof(float)))
            return QMD_ERR_VALUE;
    }
    if ((st = outputs_apart(y, rows, batch, K, x, na.r, xq, fused ? xq_out : qmd_q8k{nullptr, nullptr, nullptr})) !=
        QMD_OK)
        return st;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != QMD_OK)
        return st;
    QmvPlan plan;
    const int mode = na.g ? QMV_NORM : fused ? QMV_PACK : dump ? QMV_DUMP : QMV_PLAIN;
    if ((st = qmv_plan(fmt, rows, nb, batch, dev, &plan, mode)) != QMD_OK)
        return st;
    QmvArgs a;
    a.fmt = fmt;
    a.W = static_cast<const uint8_t *>(W);
    a.Wpre = static_cast<const uint8_t *>(W_aux);
    a.xqs = xq.qs;
    a.xd = xq.d;
    a.xbs = xq.bsums;
    a.y = y;
    a.rows = rows;
    a.nb = nb;
    a.batch = batch;
    a.dbg_dots = dump ? dots : nullptr;
    a.dbg_sm = dump ? sm : nullptr;
    a.x = x;
    a.xq_qs_out = fused && want_out ? xq_out.qs : nullptr;
    a.xq_d_out = fused && want_out ? xq_out.d : nullptr;
    a.xq_bs_out = fused && want_out ? xq_out.bsums : nullptr;
    a.r = na.r;
    a.g = na.g;
    a.eps = na.eps;
    a.h_out = na.h_out;
    a.ws = static_cast<unsigned *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return q6 ? launch_qmv_q6k(a, plan, s) : fmt == QMD_Q5_K ? launch_qmv_q5k(a, plan, s) : launch_qmv_q4k(a, plan, s);
}

}  // namespace

extern "C" {

qmd_status qmd_q8k_pack(const float *x, qmd_q8k xq, int64_t K, int batch, void *stream)
{
    if (!x || !xq.qs || !xq.d || !xq.bsums)
        return QMD_ERR_NULL;
    qmd_status st = check_k(K);
    if (st != QMD_OK)
        return st;
    if (batch < 1 || batch > QMD_MAX_BATCH)
        return QMD_ERR_BATCH;
    if (!aligned(x, 16) || !aligned(xq.qs, 16) || !aligned(xq.bsums, 16) || !aligned(xq.d, 4))
        return QMD_ERR_MISALIGNED;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != QMD_OK)
        return st;
    return launch_q8k_pack(x, xq.qs, xq.d, xq.bsums, (int64_t)batch * (K / QMD_QK),
                           static_cast<cudaStream_t>(stream));
}

qmd_status qmd_rmsnorm_q8k_pack(const float *x, const float *r, const float *g, float eps, float *h_out,
                                qmd_q8k xq, int64_t K, int batch, void *stream)
{
    if (!x || !g || !xq.qs || !xq.d || !xq.bsums)
        return QMD_ERR_NULL;
    qmd_status st = check_k(K);
    if (st != QMD_OK)
        return st;
    if (batch < 1 || batch > QMD_MAX_BATCH)
        return QMD_ERR_BATCH;
    if (!aligned(x, 16) || (r && !aligned(r, 16)) || !aligned(g, 16) || (h_out && !aligned(h_out, 16)) ||
        !aligned(xq.qs, 16) || !aligned(xq.bsums, 16) || !aligned(xq.d, 4))
        return QMD_ERR_MISALIGNED;
    if (!(eps >= 0.0f) || !(eps <= 3.4028234663852886e38f))  // rejects NaN, negatives and +inf
        return QMD_ERR_VALUE;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != QMD_OK)
        return st;
    return launch_rmsnorm_q8k_pack(x, r, g, eps, h_out, xq.qs, xq.d, xq.bsums, K, batch,
                                   static_cast<cudaStream_t>(stream));
}

qmd_status qmd_qmatvec(qmd_fmt fmt, const void *W, const void *W_aux, qmd_q8k_const xq, float *y,
                       int64_t rows, int64_t K, int batch, void *stream)
{
    const qmd_q8k none = {nullptr, nullptr, nullptr};
    return qmatvec_common(fmt, W, W_aux, xq, y, rows, K, batch, nullptr, nullptr, false, nullptr, none, stream);
}

qmd_status qmd_qmatvec_x(qmd_fmt fmt, const void *W, const void *W_aux, const float *x, qmd_q8k xq_out,
                         float *y, int64_t rows, int64_t K, int batch, void *stream)
{
    if (!x)
        return QMD_ERR_NULL;
    const qmd_q8k_const unused = {nullptr, nullptr, nullptr};
    return qmatvec_common(fmt, W, W_aux, unused, y, rows, K, batch, nullptr, nullptr, false, x, xq_out, stream);
}

qmd_status qmd_qmatvec_ws(qmd_fmt fmt, const void *W, const void *W_aux, qmd_q8k_const xq, float *y, int64_t rows,
                          int64_t K, int batch, void *workspace, void *stream)
{
    if (!workspace)
        return QMD_ERR_NULL;
    const qmd_q8k none = {nullptr, nullptr, nullptr};
    return qmatvec_common(fmt, W, W_aux, xq, y, rows, K, batch, nullptr, nullptr, false, nullptr, none, stream,
                          NormArgs(), workspace);
}

qmd_status qmd_qmatvec_x_ws(qmd_fmt fmt, const void *W, const void *W_aux, const float *x, qmd_q8k xq_out,
                            float *y, int64_t rows, int64_t K, int batch, void *workspace, void *stream)
{
    if (!x || !workspace)
        return QMD_ERR_NULL;
    const qmd_q8k_const unused = {nullptr, nullptr, nullptr};
    return qmatvec_common(fmt, W, W_aux, unused, y, rows, K, batch, nullptr, nullptr, false, x, xq_out, stream,
                          NormArgs(), workspace);
}

qmd_status qmd_qmatvec_x_static(qmd_fmt fmt, const void *W, const void *W_aux, const float *x, qmd_q8k xq_out,
                                float *y, int64_t rows, int64_t K, int batch, void *stream)
{
    if (!x)
        return QMD_ERR_NULL;
    // The static array holds one workspace, and one workspace schedules every shape the call
    // accepts (the counters do not grow with the problem); a larger need is refused.
    static_assert(sizeof(g_static_ws) >= QMD_WORKSPACE_BYTES, "the static workspace holds one workspace");
    DeviceInfo dev;
    qmd_status st = current_device(&dev);
    if (st != QMD_OK)
        return st;
    unsigned *ws = static_workspace();
    if (!ws)
        return QMD_ERR_DEVICE;
    // The checks qmd_qmatvec_x makes, first, so that a refused call launches nothing (not even
    // the clearing of the workspace).
    const qmd_q8k_const unused = {nullptr, nullptr, nullptr};
    if (fmt != QMD_Q4_K && fmt != QMD_Q5_K && fmt != QMD_Q6_K_SPLIT)
        return QMD_ERR_FORMAT;
    const bool q6 = fmt == QMD_Q6_K_SPLIT;
    const bool want_out = xq_out.qs || xq_out.d || xq_out.bsums;
    if (!W || !y || (q6 && !W_aux) || (want_out && (!xq_out.qs || !xq_out.d || !xq_out.bsums)))
        return QMD_ERR_NULL;
    if ((st = check_k(K)) != QMD_OK)
        return st;
    if (batch < 1 || batch > QMD_MAX_BATCH)
        return QMD_ERR_BATCH;
    if (rows < 1 || rows > (int64_t)1 << 31)
        return QMD_ERR_SHAPE;
    if (!aligned(W, 16) || (q6 && !aligned(W_aux, 16)) || !aligned(y, 4) || !aligned(x, 16) ||
        (want_out && (!aligned(xq_out.qs, 16) || !aligned(xq_out.bsums, 16) || !aligned(xq_out.d, 4))))
        return QMD_ERR_MISALIGNED;
    if ((st = outputs_apart(y, rows, batch, K, x, nullptr, unused, xq_out)) != QMD_OK)
        return st;
    QmvPlan plan;
    if ((st = qmv_plan(fmt, rows, (int)(K / QMD_QK), batch, dev, &plan, QMV_PACK)) != QMD_OK)
        return st;
    // Every call starts from a cleared workspace: the array keeps whatever the last call left.
    const cudaError_t e = cudaMemsetAsync(ws, 0, QMD_WORKSPACE_BYTES, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return fail(QMD_ERR_LAUNCH, "clear the static workspace", e);
    return qmatvec_common(fmt, W, W_aux, unused, y, rows, K, batch, nullptr, nullptr, false, x, xq_out, stream,
                          NormArgs(), ws);
}

qmd_status qmd_qmatvec_rmsnorm_x(qmd_fmt fmt, const void *W, const void *W_aux, const float *x, const float *r,
                                 const float *g, float eps, float *h_out, qmd_q8k xq_out, float *y, int64_t rows,
                                 int64_t K, int batch, void *stream)
{
    if (!x || !g)
        return QMD_ERR_NULL;
    const qmd_q8k_const unused = {nullptr, nullptr, nullptr};
    NormArgs na;
    na.r = r;
    na.g = g;
    na.eps = eps;
    na.h_out = h_out;
    return qmatvec_common(fmt, W, W_aux, unused, y, rows, K, batch, nullptr, nullptr, false, x, xq_out, stream, na);
}

qmd_status qmd_debug_qmatvec_dump(qmd_fmt fmt, const void *W, const void *W_aux, qmd_q8k_const xq,
                                  float *y, int64_t rows, int64_t K, int batch, int32_t *dots,
                                  int32_t *sm, void *stream)
{
    const qmd_q8k none = {nullptr, nullptr, nullptr};
    return qmatvec_common(fmt, W, W_aux, xq, y, rows, K, batch, dots, sm, true, nullptr, none, stream);
}

int64_t qmd_q6k_prefix_stride(int64_t K)
{
    if (K <= 0 || K % QMD_QK != 0)
        return 0;
    return (K / QMD_QK + 7) / 8 * 8;
}

qmd_status qmd_q6k_split_bytes(int64_t rows, int64_t K, size_t *body_bytes, size_t *prefix_bytes)
{
    if (!body_bytes || !prefix_bytes)
        return QMD_ERR_NULL;
    qmd_status st = check_k(K);
    if (st != QMD_OK)
        return st;
    if (rows < 1 || rows > (int64_t)1 << 31)
        return QMD_ERR_SHAPE;
    const int64_t nb = K / QMD_QK;
    *body_bytes = (size_t)(rows * nb * QMD_Q6K_BODY_BYTES);
    *prefix_bytes = (size_t)(rows * qmd_q6k_prefix_stride(K) * 2);
    return QMD_OK;
}

qmd_status qmd_bind_q6k(const void *gguf, void *body, void *prefix, int64_t rows, int64_t K, void *stream)
{
    if (!gguf || !body || !prefix)
        return QMD_ERR_NULL;
    qmd_status st = check_k(K);
    if (st != QMD_OK)
        return st;
    if (rows < 1 || rows > (int64_t)1 << 31)
        return QMD_ERR_SHAPE;
    if (!aligned(gguf, 2) || !aligned(body, 16) || !aligned(prefix, 16))
        return QMD_ERR_MISALIGNED;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != QMD_OK)
        return st;
    return launch_q6k_split(static_cast<const uint8_t *>(gguf), static_cast<uint8_t *>(body),
                            static_cast<uint16_t *>(prefix), rows, (int)(K / QMD_QK),
                            qmd_q6k_prefix_stride(K), static_cast<cudaStream_t>(stream));
}

qmd_status qmd_bind_q4k(const void *gguf, int64_t rows, int64_t K)
{
    if (!gguf)
        return QMD_ERR_NULL;
    qmd_status st = check_k(K);
    if (st != QMD_OK)
        return st;
    if (rows < 1 || rows > (int64_t)1 << 31)
        return QMD_ERR_SHAPE;
    if (!aligned(gguf, 16))
        return QMD_ERR_MISALIGNED;
    return QMD_OK;
}

qmd_status qmd_bind_q5k(const void *gguf, int64_t rows, int64_t K) { return qmd_bind_q4k(gguf, rows, K); }

const char *qmd_status_str(qmd_status s)
{
    switch (s) {
    case QMD_OK: return "QMD_OK";
    case QMD_ERR_NULL: return "QMD_ERR_NULL";
    case QMD_ERR_FORMAT: return "QMD_ERR_FORMAT";
    case QMD_ERR_K_NOT_MULTIPLE_OF_256: return "QMD_ERR_K_NOT_MULTIPLE_OF_256";
    case QMD_ERR_BATCH: return "QMD_ERR_BATCH";
    case QMD_ERR_MISALIGNED: return "QMD_ERR_MISALIGNED";
    case QMD_ERR_SHAPE: return "QMD_ERR_SHAPE";
    case QMD_ERR_LAUNCH: return "QMD_ERR_LAUNCH";
    case QMD_ERR_DEVICE_TIMEOUT: return "QMD_ERR_DEVICE_TIMEOUT";
    case QMD_ERR_DEVICE: return "QMD_ERR_DEVICE";
    case QMD_ERR_VALUE: return "QMD_ERR_VALUE";
    }
    return "QMD_ERR_UNKNOWN";
}

const char *qmd_last_error_detail(void) { return g_detail; }

qmd_status qmd_get_device_error(void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return fail(QMD_ERR_LAUNCH, "stream", e);
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_error_word, sizeof v);
    if (e != cudaSuccess)
        return fail(QMD_ERR_LAUNCH, "read error word", e);
    if (v != 0) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof zero);
        if (e != cudaSuccess)
            return fail(QMD_ERR_LAUNCH, "clear error word", e);
        snprintf(g_detail, sizeof g_detail, "device error word 0x%x", v);
        return QMD_ERR_DEVICE_TIMEOUT;
    }
    return QMD_OK;
}

void qmd_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns); }

void qmd_debug_set_plan(int row_groups, int rows_per_stage, int max_stages, int ctas_per_sm)
{
    g_force_rg.store(row_groups > 0 && row_groups <= 32 ? row_groups : 0);
    g_force_rows.store(rows_per_stage >= 1 && rows_per_stage <= 8 ? rows_per_stage : 0);
    g_force_stages.store(max_stages > 0 ? max_stages : 0);
    g_force_cps.store(ctas_per_sm > 0 && ctas_per_sm <= 8 ? ctas_per_sm : 0);
}

qmd_status qmd_qmatvec_launch_info(qmd_fmt fmt, int64_t rows, int64_t K, int batch, int *grid,
                                   int *threads, int *smem_bytes, int *stages, int *rows_per_stage)
{
    if (fmt != QMD_Q4_K && fmt != QMD_Q5_K && fmt != QMD_Q6_K_SPLIT)
        return QMD_ERR_FORMAT;
    qmd_status st = check_k(K);
    if (st != QMD_OK)
        return st;
    if (batch < 1 || batch > QMD_MAX_BATCH)
        return QMD_ERR_BATCH;
    if (rows < 1 || rows > (int64_t)1 << 31)
        return QMD_ERR_SHAPE;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != QMD_OK)
        return st;
    QmvPlan p;
    if ((st = qmv_plan(fmt, rows, (int)(K / QMD_QK), batch, dev, &p)) != QMD_OK)
        return st;
    if (grid) *grid = p.grid;
    if (threads) *threads = p.threads;
    if (smem_bytes) *smem_bytes = p.smem;
    if (stages) *stages = p.stages;
    if (rows_per_stage) *rows_per_stage = p.RG * p.PR;
    return QMD_OK;
}

int qmd_qmatvec_launch_kernel(qmd_fmt fmt, int64_t rows, int64_t K, int batch)
{
    if (fmt != QMD_Q4_K && fmt != QMD_Q5_K && fmt != QMD_Q6_K_SPLIT)
        return -(int)QMD_ERR_FORMAT;
    qmd_status st = check_k(K);
    if (st != QMD_OK)
        return -(int)st;
    if (batch < 1 || batch > QMD_MAX_BATCH)
        return -(int)QMD_ERR_BATCH;
    if (rows < 1 || rows > (int64_t)1 << 31)
        return -(int)QMD_ERR_SHAPE;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != QMD_OK)
        return -(int)st;
    QmvPlan p;
    if ((st = qmv_plan(fmt, rows, (int)(K / QMD_QK), batch, dev, &p)) != QMD_OK)
        return -(int)st;
    return p.layout;
}

qmd_status qmd_debug_wait_timeout(uint64_t limit_ns, void *stream)
{
    DeviceInfo dev;
    qmd_status st = current_device(&dev);
    if (st != QMD_OK)
        return st;
    unsigned *err = device_error_word();
    if (!err)
        return QMD_ERR_DEVICE;
    debug_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, (unsigned long long)limit_ns);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(QMD_ERR_LAUNCH, "debug wait launch", e);
    return QMD_OK;
}

void qmd_debug_set_launch_flags(unsigned flags) { g_launch_flags.store(flags); }

void qmd_debug_set_split_k(int ctas) { g_force_split.store(ctas >= 2 && ctas <= SK_MAX_SPLIT ? ctas : 0); }

void qmd_debug_set_dynamic_tiles(int per_mille)
{
    g_dyn_permille.store(per_mille >= 0 && per_mille <= 1000 ? per_mille : -1);
}

#ifdef QMD_TRACE
qmd_status qmd_debug_trace(void *buf, int64_t records)
{
    std::lock_guard<std::mutex> lock(g_trace_mu);
    if (buf && (!aligned(buf, 8) || records < 0))
        return QMD_ERR_VALUE;
    g_trace_buf = static_cast<unsigned long long *>(buf);
    g_trace_cap = buf ? records : 0;
    g_trace_used = 0;
    g_trace_log.clear();
    return QMD_OK;
}

int64_t qmd_debug_trace_launches(int64_t *first, int32_t *ctas, int64_t max)
{
    std::lock_guard<std::mutex> lock(g_trace_mu);
    const int64_t n = (int64_t)g_trace_log.size() / 2;
    for (int64_t i = 0; i < n && i < max; ++i) {
        if (first)
            first[i] = g_trace_log[2 * i];
        if (ctas)
            ctas[i] = (int32_t)g_trace_log[2 * i + 1];
    }
    return n;
}
#endif

int qmd_version(void) { return 100; }

}  // extern "C"
