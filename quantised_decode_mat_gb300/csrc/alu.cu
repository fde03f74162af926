// alu.cu -- measured issue rates of the two integer-exact multiply-add paths the mat-vec uses,
// for an ALU roofline beside the HBM one: dp4a (four int8 x int8 products and their sum into
// an int32, one instruction per thread) and the warp-wide mma.sync.m16n8k16 with f16 inputs
// and f32 accumulation.  Both kernels keep every operand in registers (no memory traffic but
// one conditional store), run independent dependency chains so that issue, not latency, is the
// limit, and end after a fixed iteration count.
#include <cuda_runtime.h>

#include "internal.h"
#include "qmv_tc.cuh"

namespace qmd {

constexpr int ALU_CHAINS = 8;

__global__ void __launch_bounds__(256) dp4a_rate_kernel(int iters, int *sink)
{
    int acc[ALU_CHAINS];
    const int b = 0x01020304 ^ (int)(threadIdx.x * 2654435761u);
#pragma unroll
    for (int c = 0; c < ALU_CHAINS; ++c)
        acc[c] = (int)threadIdx.x + c;
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < ALU_CHAINS; ++c)
            acc[c] = __dp4a(acc[c], b, acc[c]);
    }
    int s = 0;
#pragma unroll
    for (int c = 0; c < ALU_CHAINS; ++c)
        s ^= acc[c];
    if (s == 0x7eadbeef)  // practically never; keeps the chains live
        sink[0] = s;
}

__global__ void __launch_bounds__(256) mma_rate_kernel(int iters, float *sink)
{
    float d[4][4];
    uint32_t a[4];
    const uint32_t x = 0x3c003c00u ^ (threadIdx.x & 1u);  // f16 pairs near 1.0
#pragma unroll
    for (int i = 0; i < 4; ++i)
        a[i] = x + i;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            d[c][i] = 0.0f;
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
            mma_16816(d[c], a, x, x + c);
    }
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            s += d[c][i];
    if (s == 1234.5f)
        sink[0] = s;
}

// Read-only streaming: every CTA (one per SM) walks its share of a buffer in 12 KB chunks, each
// of 8 warps keeping two chunks in flight with 1-D bulk copies into shared memory (the path the
// mat-vecs read their weights by), and discards them.  Bounded waits flag `err`.
constexpr int RD_WARPS = 8, RD_STAGES = 2, RD_CHUNK = 12288;

__global__ void __launch_bounds__(RD_WARPS * 32, 1)
    read_rate_kernel(const uint8_t *buf, int64_t bytes, unsigned *err, unsigned long long wait_ns)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) unsigned long long bars[RD_WARPS * RD_STAGES];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nchunks = (bytes + RD_CHUNK - 1) / RD_CHUNK;
    const int64_t c0 = nchunks * blockIdx.x / gridDim.x, c1 = nchunks * (blockIdx.x + 1) / gridDim.x;
    if (lane != 0)
        return;
    const uint32_t bar0 = smem_addr(&bars[warp * RD_STAGES]);
    const uint32_t dst0 = smem_addr(smem + (size_t)warp * RD_STAGES * RD_CHUNK);
    for (int i = 0; i < RD_STAGES; ++i)
        mbar_init(bar0 + 8u * i, 1);
    fence_barrier_init();
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int64_t c, int st) {
        const int64_t off = c * RD_CHUNK;
        const uint32_t n = (uint32_t)min((int64_t)RD_CHUNK, bytes - off);
        mbar_arrive_expect_tx(bar0 + 8u * st, n);
        bulk_copy_g2s(dst0 + (uint32_t)(st * RD_CHUNK), buf + off, n, bar0 + 8u * st, pol);
    };
    int64_t c = c0 + warp;
    for (int st = 0; st < RD_STAGES && c + (int64_t)st * RD_WARPS < c1; ++st)
        issue(c + (int64_t)st * RD_WARPS, st);
    int st = 0;
    uint32_t par = 0u;
    for (; c < c1; c += RD_WARPS) {
        if (!mbar_wait_bounded(bar0 + 8u * st, par, wait_ns)) {
            // flag it, wait (bounded) for the other stage's copy if one was issued, leave
            atomicOr(err, ERRBIT_QMV_WAIT);
            const int64_t other = c + RD_WARPS;
            if (other < c1 && !mbar_wait_bounded(bar0 + 8u * (st ^ 1), par ^ (st == RD_STAGES - 1 ? 1u : 0u), wait_ns))
                atomicOr(err, ERRBIT_DRAIN_WAIT);
            return;
        }
        const int64_t next = c + (int64_t)RD_STAGES * RD_WARPS;
        if (next < c1)
            issue(next, st);
        if (++st == RD_STAGES) {
            st = 0;
            par ^= 1u;
        }
    }
}

}  // namespace qmd

extern "C" qmd_status qmd_measure_read_bw(const void *buf, size_t bytes, double *bytes_per_s)
{
    using namespace qmd;
    if (!buf || !bytes_per_s)
        return QMD_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(buf) % 16 != 0)
        return QMD_ERR_MISALIGNED;
    if (bytes < (size_t)RD_CHUNK || bytes % 16 != 0)
        return QMD_ERR_SHAPE;
    DeviceInfo dev;
    qmd_status st = current_device(&dev);
    if (st != QMD_OK)
        return st;
    unsigned *err = device_error_word();
    if (!err)
        return QMD_ERR_DEVICE;
    const int smem = RD_WARPS * RD_STAGES * RD_CHUNK;
    cudaError_t e = cudaFuncSetAttribute(read_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaStream_t s = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (e == cudaSuccess)
        e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e == cudaSuccess)
        e = cudaEventCreate(&e0);
    if (e == cudaSuccess)
        e = cudaEventCreate(&e1);
    const int reps = 5;
    float ms = 0.0f;
    const unsigned long long wait_ns = wait_limit_ns();
    const uint8_t *b = static_cast<const uint8_t *>(buf);
    if (e == cudaSuccess) {
        read_rate_kernel<<<dev.sm_count, RD_WARPS * 32, smem, s>>>(b, (int64_t)bytes, err, wait_ns);  // warm up
        e = cudaEventRecord(e0, s);
    }
    for (int i = 0; i < reps && e == cudaSuccess; ++i)
        read_rate_kernel<<<dev.sm_count, RD_WARPS * 32, smem, s>>>(b, (int64_t)bytes, err, wait_ns);
    if (e == cudaSuccess)
        e = cudaEventRecord(e1, s);
    if (e == cudaSuccess)
        e = cudaEventSynchronize(e1);
    if (e == cudaSuccess)
        e = cudaEventElapsedTime(&ms, e0, e1);
    if (e == cudaSuccess)
        e = cudaGetLastError();
    if (e0)
        cudaEventDestroy(e0);
    if (e1)
        cudaEventDestroy(e1);
    if (s)
        cudaStreamDestroy(s);
    if (e != cudaSuccess)
        return fail(QMD_ERR_LAUNCH, "read rate kernel", e);
    *bytes_per_s = (double)bytes * reps / (ms * 1e-3);
    return QMD_OK;
}

extern "C" qmd_status qmd_measure_alu(double *dp4a_per_s, double *mma_flop_per_s)
{
    using namespace qmd;
    if (!dp4a_per_s || !mma_flop_per_s)
        return QMD_ERR_NULL;
    DeviceInfo dev;
    qmd_status st = current_device(&dev);
    if (st != QMD_OK)
        return st;
    int *sink = nullptr;
    cudaStream_t s = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e = cudaMalloc(&sink, 16);
    if (e == cudaSuccess)
        e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e == cudaSuccess)
        e = cudaEventCreate(&e0);
    if (e == cudaSuccess)
        e = cudaEventCreate(&e1);
    const int blocks = dev.sm_count * 8, threads = 256;
    const int it_dp4a = 1 << 14, it_mma = 1 << 12;
    float ms_dp4a = 0.0f, ms_mma = 0.0f;
    for (int pass = 0; pass < 2 && e == cudaSuccess; ++pass) {  // pass 0 warms up
        dp4a_rate_kernel<<<blocks, threads, 0, s>>>(pass ? it_dp4a : 64, sink);
        e = cudaEventRecord(e0, s);
        dp4a_rate_kernel<<<blocks, threads, 0, s>>>(it_dp4a, sink);
        if (e == cudaSuccess)
            e = cudaEventRecord(e1, s);
        if (e == cudaSuccess)
            e = cudaEventSynchronize(e1);
        if (e == cudaSuccess)
            e = cudaEventElapsedTime(&ms_dp4a, e0, e1);
        if (e == cudaSuccess)
            mma_rate_kernel<<<blocks, threads, 0, s>>>(pass ? it_mma : 16, reinterpret_cast<float *>(sink));
        if (e == cudaSuccess)
            e = cudaEventRecord(e0, s);
        if (e == cudaSuccess)
            mma_rate_kernel<<<blocks, threads, 0, s>>>(it_mma, reinterpret_cast<float *>(sink));
        if (e == cudaSuccess)
            e = cudaEventRecord(e1, s);
        if (e == cudaSuccess)
            e = cudaEventSynchronize(e1);
        if (e == cudaSuccess)
            e = cudaEventElapsedTime(&ms_mma, e0, e1);
        if (e == cudaSuccess)
            e = cudaGetLastError();
    }
    if (e0)
        cudaEventDestroy(e0);
    if (e1)
        cudaEventDestroy(e1);
    if (s)
        cudaStreamDestroy(s);
    if (sink)
        cudaFree(sink);
    if (e != cudaSuccess)
        return fail(QMD_ERR_LAUNCH, "alu rate kernels", e);
    const double threads_total = (double)blocks * threads;
    *dp4a_per_s = threads_total * it_dp4a * ALU_CHAINS / (ms_dp4a * 1e-3);
    const double warps_total = threads_total / 32.0;
    *mma_flop_per_s = warps_total * it_mma * 4 * (16.0 * 8.0 * 16.0 * 2.0) / (ms_mma * 1e-3);
    return QMD_OK;
}
