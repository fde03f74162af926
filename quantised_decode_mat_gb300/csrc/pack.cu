// pack.cu -- q8_K quantisation of f32 activations on the device.
//
// "Language models on the device: the cajeta-llm kernels", §1: activations are quantised on
// the device to q8_K (q8kPackKernel), 256 values a block, one scale and eight sub-block sums,
// so that the mat-vec's arithmetic is an integer dot product.
//
// One warp per 256-value block; lane l owns values 8l .. 8l+7 (two 16-byte loads).  The block
// arithmetic is in q8k.cuh, shared with the fused pack + mat-vec kernel.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "q8k.cuh"
#include "qmv.cuh"

namespace qmd {

constexpr int PACK_WARPS = 8;

__global__ void __launch_bounds__(PACK_WARPS * 32)
    q8k_pack_kernel(const float *__restrict__ x, int8_t *__restrict__ qs, float *__restrict__ d,
                    int16_t *__restrict__ bsums, int64_t nblocks
#ifdef QMD_TRACE
                    , unsigned long long *trace
#endif
    )
{
#ifdef QMD_TRACE
    // traced build: entry, wait released and exit (fields 0, 2, 6), as the mat-vec records them
    unsigned long long *rec = trace ? trace + (size_t)blockIdx.x * QMD_TRACE_FIELDS : nullptr;
    if (rec && threadIdx.x == 0) {
        rec[0] = globaltimer_ns();
        rec[7] = (unsigned long long)smid() | ((unsigned long long)blockIdx.x << 16) |
                 ((unsigned long long)gridDim.x << 32) | (3ull << 48);
    }
#endif
    pdl_launch_dependents();
    pdl_wait();  // x is produced by earlier work in the stream
#ifdef QMD_TRACE
    if (rec && threadIdx.x == 0)
        rec[2] = globaltimer_ns();
    if (rec && (threadIdx.x & 31) == 0) {
        // every warp, even one past the last block, stamps its exit
        const int64_t b = (int64_t)blockIdx.x * PACK_WARPS + (threadIdx.x >> 5);
        if (b >= nblocks)
            atomicMax(rec + 6, globaltimer_ns());
    }
#endif

    const int lane = threadIdx.x & 31;
    const int64_t blk = (int64_t)blockIdx.x * PACK_WARPS + (threadIdx.x >> 5);
    if (blk >= nblocks)
        return;

    const float4 *src = reinterpret_cast<const float4 *>(x + blk * 256 + 8 * lane);
    const float4 a = src[0], b = src[1];
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const Q8Block r = q8k_quantise_block(v);
    *reinterpret_cast<uint2 *>(qs + blk * 256 + 8 * lane) = r.codes;
    if ((lane & 3) == 0)
        bsums[blk * 8 + (lane >> 2)] = (int16_t)r.sum4;
    if (lane == 0)
        d[blk] = r.d;
#ifdef QMD_TRACE
    if (rec && lane == 0)
        atomicMax(rec + 6, globaltimer_ns());
#endif
}

qmd_status launch_q8k_pack(const float *x, int8_t *qs, float *d, int16_t *bsums, int64_t nblocks,
                           cudaStream_t s)
{
    const int64_t grid = (nblocks + PACK_WARPS - 1) / PACK_WARPS;
    if (grid > 0x7fffffff)
        return QMD_ERR_SHAPE;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(PACK_WARPS * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_flags() & LAUNCH_NO_PDL) ? 0 : 1;
#ifdef QMD_TRACE
    cudaError_t e = cudaLaunchKernelEx(&cfg, q8k_pack_kernel, x, qs, d, bsums, nblocks, trace_reserve((int)grid));
#else
    cudaError_t e = cudaLaunchKernelEx(&cfg, q8k_pack_kernel, x, qs, d, bsums, nblocks);
#endif
    if (e != cudaSuccess)
        return fail(QMD_ERR_LAUNCH, "q8k_pack launch", e);
    return QMD_OK;
}

}  // namespace qmd
