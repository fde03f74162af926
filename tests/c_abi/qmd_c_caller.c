/*
 * qmd_c_caller.c -- a plain C99 caller of libqmd, for the ABI test: it includes only qmd.h and the
 * CUDA runtime's C header, allocates device memory itself, and calls the library through its C
 * entry points as a C program would.
 *
 *   qmd_c_caller IN OUT
 * IN:  int64 rows, int64 K, int32 batch, then the Q4_K weights (rows x K/256 x 144 bytes) and the
 *      activations (batch x K f32), all little-endian.
 * OUT: y from qmd_q8k_pack + qmd_qmatvec, then y from qmd_qmatvec_x (each batch x rows f32).
 * Exit status: 0 on success, 2 on bad input, 3 on a CUDA error, 10 + the qmd status of a call
 * that was refused.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "qmd.h"

static int cuda_ok(cudaError_t e, const char *what)
{
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        return 0;
    }
    return 1;
}

int main(int argc, char **argv)
{
    FILE *in, *out;
    int64_t rows, K;
    int32_t batch;
    size_t wbytes, xbytes, ybytes, nb;
    void *hw, *hx, *hy;
    void *dw = NULL, *dx = NULL, *dy = NULL, *dqs = NULL, *dd = NULL, *dbs = NULL;
    qmd_q8k xq;
    qmd_q8k_const xqc;
    qmd_q8k none = {NULL, NULL, NULL};
    qmd_status st;
    int rc = 0;

    if (argc != 3 || !(in = fopen(argv[1], "rb")))
        return 2;
    if (fread(&rows, 8, 1, in) != 1 || fread(&K, 8, 1, in) != 1 || fread(&batch, 4, 1, in) != 1 || rows < 1 ||
        K < QMD_QK || batch < 1 || batch > QMD_MAX_BATCH)
        return 2;
    nb = (size_t)(K / QMD_QK);
    wbytes = (size_t)rows * nb * QMD_Q4K_BLOCK_BYTES;
    xbytes = (size_t)batch * (size_t)K * sizeof(float);
    ybytes = (size_t)batch * (size_t)rows * sizeof(float);
    hw = malloc(wbytes);
    hx = malloc(xbytes);
    hy = malloc(2 * ybytes);
    if (!hw || !hx || !hy || fread(hw, 1, wbytes, in) != wbytes || fread(hx, 1, xbytes, in) != xbytes)
        return 2;
    fclose(in);

    if (!cuda_ok(cudaMalloc(&dw, wbytes), "cudaMalloc W") || !cuda_ok(cudaMalloc(&dx, xbytes), "cudaMalloc x") ||
        !cuda_ok(cudaMalloc(&dy, 2 * ybytes), "cudaMalloc y") ||
        !cuda_ok(cudaMalloc(&dqs, (size_t)batch * (size_t)K), "cudaMalloc qs") ||
        !cuda_ok(cudaMalloc(&dd, (size_t)batch * nb * sizeof(float)), "cudaMalloc d") ||
        !cuda_ok(cudaMalloc(&dbs, (size_t)batch * nb * 8 * sizeof(int16_t)), "cudaMalloc bsums") ||
        !cuda_ok(cudaMemcpy(dw, hw, wbytes, cudaMemcpyHostToDevice), "copy W") ||
        !cuda_ok(cudaMemcpy(dx, hx, xbytes, cudaMemcpyHostToDevice), "copy x"))
        return 3;

    st = qmd_bind_q4k(dw, rows, K);
    if (st != QMD_OK)
        return 10 + (int)st;
    xq.qs = (int8_t *)dqs;
    xq.d = (float *)dd;
    xq.bsums = (int16_t *)dbs;
    st = qmd_q8k_pack((const float *)dx, xq, K, batch, NULL);
    if (st != QMD_OK)
        return 10 + (int)st;
    xqc.qs = xq.qs;
    xqc.d = xq.d;
    xqc.bsums = xq.bsums;
    st = qmd_qmatvec(QMD_Q4_K, dw, NULL, xqc, (float *)dy, rows, K, batch, NULL);
    if (st != QMD_OK)
        return 10 + (int)st;
    st = qmd_qmatvec_x(QMD_Q4_K, dw, NULL, (const float *)dx, none, (float *)dy + (size_t)batch * (size_t)rows,
                       rows, K, batch, NULL);
    if (st != QMD_OK)
        return 10 + (int)st;
    st = qmd_get_device_error(NULL);
    if (st != QMD_OK) {
        fprintf(stderr, "%s: %s\n", qmd_status_str(st), qmd_last_error_detail());
        return 10 + (int)st;
    }
    if (!cuda_ok(cudaMemcpy(hy, dy, 2 * ybytes, cudaMemcpyDeviceToHost), "copy y"))
        return 3;
    out = fopen(argv[2], "wb");
    if (!out || fwrite(hy, 1, 2 * ybytes, out) != 2 * ybytes)
        rc = 2;
    if (out)
        fclose(out);
    cudaFree(dw);
    cudaFree(dx);
    cudaFree(dy);
    cudaFree(dqs);
    cudaFree(dd);
    cudaFree(dbs);
    free(hw);
    free(hx);
    free(hy);
    printf("ok: libqmd %d, %s\n", qmd_version(), qmd_status_str(QMD_OK));
    return rc;
}
