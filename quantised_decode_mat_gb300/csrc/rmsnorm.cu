// rmsnorm.cu -- RMSNorm with a residual add, fused into the q8_K pack.
//
// "Language models on the device: the cajeta-llm kernels", §2.6 lists the normalisation and
// residual kernels (rmsnorm*, add*) that sit beside the device q8_K quantiser (§1,
// q8kPackKernel); in a decode step they produce the activation the quantiser packs.  Here the
// three are one launch, so the normalised f32 vector never goes to memory:
//     h = x + r                          (r absent: h = x; h is the new residual stream)
//     n = (h * (1 / sqrt(sum(h * h) / K + eps))) * g
//     xq = q8_K pack of n                 (the block arithmetic of q8k.cuh)
// Every f32 operation is rounded on its own (explicit _rn intrinsics, so nothing is contracted
// into a fused multiply-add); sqrt and the divisions are correctly rounded.  The packed codes
// depend on the bits of n, so the sum of squares has a declared order: thread t of the
// 256-thread CTA adds the squares of elements t, t + 256, t + 512, ... left to right; each
// warp combines its 32 partials by xor-shuffles 16, 8, 4, 2, 1 (a pairwise tree); the eight
// warp totals are added left to right.
//
// One CTA per vector.  Phase 1 streams x (and r) -- all of a thread's loads of a round in flight
// before any store, since h may be the same buffer as x or r -- writes h when asked, keeps it
// in shared memory when it fits, and sums the squares; phase 2 normalises and quantises one
// 256-value block per warp from that copy (or re-reads h / recomputes x + r with the same
// addition for rows too long for shared memory).
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "q8k.cuh"

namespace qmd {

constexpr int RMS_THREADS = 256;
constexpr int RMS_SMEM_MAX_K = 16384;  // h kept in shared memory up to this width (64 KB)

template <bool HS>
__global__ void __launch_bounds__(RMS_THREADS)
    rmsnorm_q8k_pack_kernel(const float *x, const float *r, const float *__restrict__ g, float eps, float *h_out,
                            int8_t *__restrict__ qs, float *__restrict__ d, int16_t *__restrict__ bsums, int64_t K)
{
    __shared__ float s_part[RMS_THREADS / 32];
    __shared__ float s_inv;
    extern __shared__ __align__(16) float s_h[];  // HS: h of this vector

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t nb = K / 256;
    // The gain is a weight: this lane's slice of it for the warp's first GP blocks is fetched
    // before waiting on the preceding kernel, so its latency overlaps that wait and phase 1.
    constexpr int GP = 2;
    float4 gpre[GP][2];
#pragma unroll
    for (int j = 0; j < GP; ++j) {
        const int64_t b = warp + (int64_t)j * (RMS_THREADS / 32);
        if (b < nb) {
            gpre[j][0] = *reinterpret_cast<const float4 *>(g + b * 256 + 8 * lane);
            gpre[j][1] = *reinterpret_cast<const float4 *>(g + b * 256 + 8 * lane + 4);
        }
    }

    pdl_launch_dependents();
    pdl_wait();  // x and r are produced by earlier work in the stream

    const int64_t base = (int64_t)blockIdx.x * K;
    const float *xv = x + base;
    const float *rv = r ? r + base : nullptr;
    float *hv = h_out ? h_out + base : nullptr;

    // ---- phase 1: h, and this thread's sum of squares (elements tid + 256 j, j ascending) ----
    float p = 0.0f;
    constexpr int U = 16;  // loads in flight per thread per round; the adds stay in ascending j
    for (int64_t i0 = tid; i0 < K; i0 += (int64_t)U * RMS_THREADS) {
        float xu[U], ru[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + (int64_t)u * RMS_THREADS;
            xu[u] = i < K ? xv[i] : 0.0f;
            ru[u] = (rv && i < K) ? rv[i] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + (int64_t)u * RMS_THREADS;
            if (i < K) {
                const float hu = rv ? __fadd_rn(xu[u], ru[u]) : xu[u];
                if (hv)
                    hv[i] = hu;
                if (HS)
                    s_h[i] = hu;
                p = __fadd_rn(p, __fmul_rn(hu, hu));
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, o));
    if (lane == 0)
        s_part[warp] = p;
    __syncthreads();
    if (tid == 0) {
        float total = s_part[0];
        for (int w = 1; w < RMS_THREADS / 32; ++w)
            total = __fadd_rn(total, s_part[w]);
        const float ms = __fdiv_rn(total, (float)K);
        s_inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    }
    __syncthreads();  // also orders phase 1's stores of h before phase 2's loads
    const float inv = s_inv;

    // ---- phase 2: normalise and quantise, one warp per 256-value block ---------------------
    for (int64_t b = warp, j = 0; b < nb; b += RMS_THREADS / 32, ++j) {
        const int64_t e = b * 256 + 8 * lane;
        float h8[8];
        if (HS) {
            const float4 a0 = *reinterpret_cast<const float4 *>(s_h + e);
            const float4 a1 = *reinterpret_cast<const float4 *>(s_h + e + 4);
            h8[0] = a0.x; h8[1] = a0.y; h8[2] = a0.z; h8[3] = a0.w;
            h8[4] = a1.x; h8[5] = a1.y; h8[6] = a1.z; h8[7] = a1.w;
        } else if (hv) {
            const float4 a0 = *reinterpret_cast<const float4 *>(hv + e);
            const float4 a1 = *reinterpret_cast<const float4 *>(hv + e + 4);
            h8[0] = a0.x; h8[1] = a0.y; h8[2] = a0.z; h8[3] = a0.w;
            h8[4] = a1.x; h8[5] = a1.y; h8[6] = a1.z; h8[7] = a1.w;
        } else {
            const float4 a0 = *reinterpret_cast<const float4 *>(xv + e);
            const float4 a1 = *reinterpret_cast<const float4 *>(xv + e + 4);
            h8[0] = a0.x; h8[1] = a0.y; h8[2] = a0.z; h8[3] = a0.w;
            h8[4] = a1.x; h8[5] = a1.y; h8[6] = a1.z; h8[7] = a1.w;
            if (rv) {
                const float4 c0 = *reinterpret_cast<const float4 *>(rv + e);
                const float4 c1 = *reinterpret_cast<const float4 *>(rv + e + 4);
                const float c8[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    h8[i] = __fadd_rn(h8[i], c8[i]);
            }
        }
        float4 g0, g1;
        if (j < GP) {
            g0 = j == 0 ? gpre[0][0] : gpre[1][0];
            g1 = j == 0 ? gpre[0][1] : gpre[1][1];
        } else {
            g0 = *reinterpret_cast<const float4 *>(g + e);
            g1 = *reinterpret_cast<const float4 *>(g + e + 4);
        }
        const float g8[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        float n8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            n8[i] = __fmul_rn(__fmul_rn(h8[i], inv), g8[i]);
        const Q8Block q = q8k_quantise_block(n8);
        const int64_t blk = (int64_t)blockIdx.x * nb + b;
        *reinterpret_cast<uint2 *>(qs + blk * 256 + 8 * lane) = q.codes;
        if ((lane & 3) == 0)
            bsums[blk * 8 + (lane >> 2)] = (int16_t)q.sum4;
        if (lane == 0)
            d[blk] = q.d;
    }
}

qmd_status launch_rmsnorm_q8k_pack(const float *x, const float *r, const float *g, float eps, float *h_out,
                                   int8_t *qs, float *d, int16_t *bsums, int64_t K, int batch, cudaStream_t s)
{
    const bool hs = K <= RMS_SMEM_MAX_K;
    if (hs) {
        // Opt in to 64 KB of dynamic shared memory once per device; host threads may race here.
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
            return QMD_ERR_DEVICE;
        static std::mutex mu;
        static bool opted[64] = {false};
        std::lock_guard<std::mutex> lock(mu);
        if (!opted[dev]) {
            cudaError_t e = cudaFuncSetAttribute(rmsnorm_q8k_pack_kernel<true>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)(RMS_SMEM_MAX_K * sizeof(float)));
            if (e != cudaSuccess)
                return fail(QMD_ERR_LAUNCH, "rmsnorm_q8k_pack smem attribute", e);
            opted[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)batch);
    cfg.blockDim = dim3(RMS_THREADS);
    cfg.dynamicSmemBytes = hs ? (size_t)K * sizeof(float) : 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & LAUNCH_NO_PDL) ? 0 : 1;
    cudaError_t e = hs ? cudaLaunchKernelEx(&cfg, rmsnorm_q8k_pack_kernel<true>, x, r, g, eps, h_out, qs, d, bsums, K)
                       : cudaLaunchKernelEx(&cfg, rmsnorm_q8k_pack_kernel<false>, x, r, g, eps, h_out, qs, d, bsums, K);
    if (e != cudaSuccess)
        return fail(QMD_ERR_LAUNCH, "rmsnorm_q8k_pack launch", e);
    return QMD_OK;
}

}  // namespace qmd
