// q8k.cuh -- the q8_K block quantiser shared by the stand-alone pack kernel and the fused
// pack + mat-vec kernel, so that both produce the same bytes.
//
// "Language models on the device: the cajeta-llm kernels", §1: activations are quantised on
// the device to q8_K, 256 values a block, one scale and eight sub-block sums.  Per block, all
// in f32: amax = max |x|; iscale = 127 / amax (rounded once); code = clamp(round-to-nearest-
// even(x * iscale), -127, 127) with the product rounded once; d = amax / 127; the sum of each
// run of 32 codes.  If amax is 0 every output is 0.  If 127 / amax overflows to infinity, a
// zero value's product is NaN and its code is 0.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qmd {

struct Q8Block {
    uint2 codes;  // this lane's 8 codes, packed little-endian
    int sum2;     // the sum of the 16 codes of lanes 2s, 2s+1 (valid in both)
    int sum4;     // the lane's sub-block sum (valid in lanes 4j, for sub-block j)
    float d;      // the block scale (valid in every lane)
};

// One warp quantises one 256-value block; lane l owns values 8l .. 8l+7 (v[0..8)).
__device__ __forceinline__ Q8Block q8k_quantise_block(const float (&v)[8])
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));

    const float iscale = amax == 0.0f ? 0.0f : __fdiv_rn(127.0f, amax);
    Q8Block out;
    int sum;
    if (iscale <= 3.402823466e38f) {  // finite (the same for every lane)
        // |x * iscale| <= 127 (1 + 2^-23) < 127.5 for every finite x, so round-to-nearest-even
        // needs no clamp: adding 1.5 * 2^23 (unit 1, an even integer) rounds the product to the
        // nearest integer, ties to even, and leaves it in the low mantissa bits -- the low byte
        // of the sum's bits is the code in two's complement.  A NaN product (a NaN value, or an
        // infinite one against a zero scale) gives code 0.
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float pr = __fmul_rn(v[i], iscale);
            w[i] = pr != pr ? 0x4B400000u : __float_as_uint(__fadd_rn(pr, 12582912.0f));
        }
        out.codes.x = __byte_perm(__byte_perm(w[0], w[1], 0x5140u), __byte_perm(w[2], w[3], 0x5140u), 0x5410u);
        out.codes.y = __byte_perm(__byte_perm(w[4], w[5], 0x5140u), __byte_perm(w[6], w[7], 0x5140u), 0x5410u);
        sum = __dp4a((int)out.codes.y, 0x01010101, __dp4a((int)out.codes.x, 0x01010101, 0));
    } else {
        // 127 / amax overflowed (amax below about 3.7e-37): products are infinite or NaN;
        // clamp after the rounding, NaN to 0
        int q[8];
        sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float pr = __fmul_rn(v[i], iscale);
            int r = pr != pr ? 0 : __float2int_rn(pr);
            r = min(127, max(-127, r));
            q[i] = r;
            sum += r;
        }
        out.codes.x = (q[0] & 255) | ((q[1] & 255) << 8) | ((q[2] & 255) << 16) | ((uint32_t)(q[3] & 255) << 24);
        out.codes.y = (q[4] & 255) | ((q[5] & 255) << 8) | ((q[6] & 255) << 16) | ((uint32_t)(q[7] & 255) << 24);
    }
    // sub-block j = lanes 4j .. 4j+3
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    out.sum2 = sum;
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    out.sum4 = sum;
    out.d = amax == 0.0f ? 0.0f : __fdiv_rn(amax, 127.0f);
    return out;
}

}  // namespace qmd
