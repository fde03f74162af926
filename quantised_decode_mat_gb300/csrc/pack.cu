// pack.cu -- q8_K quantisation of f32 activations on the device.
//
// "Language models on the device: the cajeta-llm kernels", §1: activations are quantised on
// the device to q8_K (q8kPackKernel), 256 values a block, one scale and eight sub-block sums,
// so that the mat-vec's arithmetic is an integer dot product.
//
// One warp per 256-value block; lane l owns values 8l .. 8l+7 (two 16-byte loads).  Every
// decision that produces a code is taken in f32 with the rounding spelled out: the scale is
// 127/amax rounded once, the product x*iscale rounded once, then rounded to nearest-even.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace qmd {

constexpr int PACK_WARPS = 8;

__global__ void __launch_bounds__(PACK_WARPS * 32)
    q8k_pack_kernel(const float *__restrict__ x, int8_t *__restrict__ qs, float *__restrict__ d,
                    int16_t *__restrict__ bsums, int64_t nblocks)
{
    pdl_launch_dependents();
    pdl_wait();  // x is produced by earlier work in the stream

    const int lane = threadIdx.x & 31;
    const int64_t blk = (int64_t)blockIdx.x * PACK_WARPS + (threadIdx.x >> 5);
    if (blk >= nblocks)
        return;

    const float4 *src = reinterpret_cast<const float4 *>(x + blk * 256 + 8 * lane);
    const float4 a = src[0], b = src[1];
    float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};

    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));

    const float iscale = amax == 0.0f ? 0.0f : __fdiv_rn(127.0f, amax);
    int q[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float pr = __fmul_rn(v[i], iscale);
        // 127/amax is +inf when amax < 127/FLT_MAX; then 0 * inf is NaN, whose code is 0
        int r = pr != pr ? 0 : __float2int_rn(pr);
        r = min(127, max(-127, r));
        q[i] = r;
        sum += r;
    }
    uint2 packed;
    packed.x = (q[0] & 255) | ((q[1] & 255) << 8) | ((q[2] & 255) << 16) | ((uint32_t)(q[3] & 255) << 24);
    packed.y = (q[4] & 255) | ((q[5] & 255) << 8) | ((q[6] & 255) << 16) | ((uint32_t)(q[7] & 255) << 24);
    *reinterpret_cast<uint2 *>(qs + blk * 256 + 8 * lane) = packed;

    // sub-block j = lanes 4j .. 4j+3
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    if ((lane & 3) == 0)
        bsums[blk * 8 + (lane >> 2)] = (int16_t)sum;
    if (lane == 0)
        d[blk] = amax == 0.0f ? 0.0f : __fdiv_rn(amax, 127.0f);
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
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, q8k_pack_kernel, x, qs, d, bsums, nblocks);
    if (e != cudaSuccess)
        return fail(QMD_ERR_LAUNCH, "q8k_pack launch", e);
    return QMD_OK;
}

}  // namespace qmd
