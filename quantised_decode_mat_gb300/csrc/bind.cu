// bind.cu -- bind-time relayout of a canonical GGUF Q6_K slab into the split layout.
//
// "Language models on the device: the cajeta-llm kernels", §1: at bind the Q6_K blocks are
// split into a scale prefix and 208-byte bodies so that kernels read them with aligned 16-byte
// loads.  The 210-byte GGUF block is ql (128 B), qh (64 B), 16 int8 scales, f16 d: the body is
// the first 208 bytes unchanged and d moves to prefix[row][block].  Prefix rows are padded to
// a multiple of 8 entries (16 bytes) with zeros so that each row starts 16-byte aligned.
// Runs once at load; not on the decode path.
#include <cuda_runtime.h>

#include "internal.h"

namespace qmd {

__global__ void q6k_split_kernel(const uint16_t *__restrict__ gguf, uint16_t *__restrict__ body,
                                 uint16_t *__restrict__ prefix, int64_t rows, int nb,
                                 int64_t pstride)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nblk = rows * nb;
    // 105 half-words per 210-byte block: 104 of body, then d
    for (int64_t t = first; t < nblk * 105; t += stride) {
        const int64_t blk = t / 105;
        const int hw = (int)(t - blk * 105);
        const uint16_t v = gguf[t];
        if (hw < 104) {
            body[blk * 104 + hw] = v;
        } else {
            const int64_t r = blk / nb, b = blk - r * nb;
            prefix[r * pstride + b] = v;
        }
    }
    const int64_t pad = pstride - nb;
    for (int64_t t = first; t < rows * pad; t += stride) {
        const int64_t r = t / pad;
        prefix[r * pstride + nb + (t - r * pad)] = 0;
    }
}

qmd_status launch_q6k_split(const uint8_t *gguf, uint8_t *body, uint16_t *prefix, int64_t rows,
                            int nb, int64_t prefix_stride, cudaStream_t s)
{
    const int64_t work = rows * nb * 105;
    int64_t grid = (work + 255) / 256;
    if (grid > 65535LL * 16)
        grid = 65535LL * 16;
    if (grid < 1)
        grid = 1;
    q6k_split_kernel<<<(unsigned)grid, 256, 0, s>>>(reinterpret_cast<const uint16_t *>(gguf),
                                                    reinterpret_cast<uint16_t *>(body), prefix, rows,
                                                    nb, prefix_stride);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(QMD_ERR_LAUNCH, "q6k split launch", e);
    return QMD_OK;
}

}  // namespace qmd
