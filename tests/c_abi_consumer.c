/*
 * c_abi_consumer.c -- a plain C99 program that uses libq4mm through include/q4mm.h only:
 * no Python, no PyTorch.  It reads seeded inputs from raw files, runs the decode GEMV, the
 * prefill GEMM, the LUT4 matmul and the routed Q4_0 mat-vec on a CUDA stream of its own,
 * and writes the outputs to raw files for the test to compare with the oracle.
 *
 * usage: c_abi_consumer DIR
 *   DIR/int4_x.bin   bf16 [M, K]            DIR/int4_w.bin  uint32 [N, K/8]
 *   DIR/int4_s.bin   bf16 [N, K/32]         DIR/int4_b.bin  bf16 [N, K/32]
 *   DIR/lut4_x.bin   bf16 [ML, KL]          DIR/lut4_p.bin  uint8 [NL*KL/2]
 *   DIR/lut4_s.bin   f32 [NL*KL/64]         DIR/lut4_book.bin f32 [16]
 *   DIR/moe_x.bin    f32 [T, KQ]            DIR/moe_w.bin   Q4_0 experts
 *   DIR/moe_ids.bin  uint32 [T*TOPK]
 *   DIR/dims.txt     "M N K ML NL KL T TOPK NQ KQ E STRIDE"
 * writes DIR/gemv_y.bin, DIR/gemm_y.bin (bf16 [M, N]), DIR/lut4_y.bin (bf16 [ML, NL]),
 * DIR/moe_out.bin (f32 [T*TOPK, NQ]).  Exit status 0 on success.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "q4mm.h"

static char path_buf[4096];

static const char *path(const char *dir, const char *name)
{
    snprintf(path_buf, sizeof path_buf, "%s/%s", dir, name);
    return path_buf;
}

static void *read_file(const char *dir, const char *name, size_t bytes)
{
    FILE *f = fopen(path(dir, name), "rb");
    void *buf = malloc(bytes ? bytes : 1);
    if (!f || !buf || fread(buf, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot read %s (%zu bytes)\n", name, bytes);
        exit(2);
    }
    fclose(f);
    return buf;
}

static void write_file(const char *dir, const char *name, const void *buf, size_t bytes)
{
    FILE *f = fopen(path(dir, name), "wb");
    if (!f || fwrite(buf, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot write %s\n", name);
        exit(2);
    }
    fclose(f);
}

static void cuda_ok(cudaError_t e, const char *what)
{
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        exit(3);
    }
}

static void q4mm_ok(q4mm_status s, const char *what)
{
    if (s != Q4MM_OK) {
        fprintf(stderr, "%s: %s\n", what, q4mm_status_string(s));
        exit(4);
    }
}

/* Device copy of a host buffer (the caller owns and frees it). */
static void *to_device(const void *host, size_t bytes)
{
    void *d = NULL;
    cuda_ok(cudaMalloc(&d, bytes ? bytes : 16), "cudaMalloc");
    cuda_ok(cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice), "cudaMemcpy H2D");
    return d;
}

int main(int argc, char **argv)
{
    if (argc != 2) {
        fprintf(stderr, "usage: %s DIR\n", argv[0]);
        return 1;
    }
    const char *dir = argv[1];
    long long M, N, K, ML, NL, KL, T, TOPK, NQ, KQ, E;
    unsigned long long STRIDE;
    FILE *df = fopen(path(dir, "dims.txt"), "r");
    if (!df || fscanf(df, "%lld %lld %lld %lld %lld %lld %lld %lld %lld %lld %lld %llu", &M, &N, &K, &ML, &NL,
                      &KL, &T, &TOPK, &NQ, &KQ, &E, &STRIDE) != 12) {
        fprintf(stderr, "cannot read dims.txt\n");
        return 2;
    }
    fclose(df);

    cudaStream_t stream;
    cuda_ok(cudaStreamCreate(&stream), "cudaStreamCreate");
    q4mm_stream_t st = (q4mm_stream_t)stream;

    /* INT4 group-32 affine: decode GEMV and prefill GEMM on the same operands. */
    size_t bx = (size_t)M * K * 2, bw = (size_t)N * (K / 8) * 4, bs = (size_t)N * (K / 32) * 2, by = (size_t)M * N * 2;
    void *hx = read_file(dir, "int4_x.bin", bx), *hw = read_file(dir, "int4_w.bin", bw);
    void *hs = read_file(dir, "int4_s.bin", bs), *hb = read_file(dir, "int4_b.bin", bs);
    void *dx = to_device(hx, bx), *dw = to_device(hw, bw), *ds = to_device(hs, bs), *db = to_device(hb, bs);
    void *dy1 = NULL, *dy2 = NULL;
    cuda_ok(cudaMalloc(&dy1, by), "cudaMalloc y");
    cuda_ok(cudaMalloc(&dy2, by), "cudaMalloc y");
    q4mm_ok(q4_gemv((const uint16_t *)dx, (const uint32_t *)dw, (const uint16_t *)ds, (const uint16_t *)db,
                    (uint16_t *)dy1, M, N, K, st), "q4_gemv");
    q4mm_ok(q4_gemm((const uint16_t *)dx, (const uint32_t *)dw, (const uint16_t *)ds, (const uint16_t *)db,
                    (uint16_t *)dy2, M, N, K, st), "q4_gemm");

    /* LUT4 (transpose = 1, block 64); the codebook is a host array. */
    size_t blx = (size_t)ML * KL * 2, blp = (size_t)NL * KL / 2, bls = (size_t)NL * KL / 64 * 4, bly = (size_t)ML * NL * 2;
    void *hlx = read_file(dir, "lut4_x.bin", blx), *hlp = read_file(dir, "lut4_p.bin", blp);
    void *hls = read_file(dir, "lut4_s.bin", bls);
    float *book = (float *)read_file(dir, "lut4_book.bin", 16 * sizeof(float));
    void *dlx = to_device(hlx, blx), *dlp = to_device(hlp, blp), *dls = to_device(hls, bls), *dly = NULL;
    cuda_ok(cudaMalloc(&dly, bly), "cudaMalloc lut4 y");
    q4mm_ok(lut4_matmul((const uint16_t *)dlx, (const uint8_t *)dlp, (const float *)dls, book, (uint16_t *)dly, ML,
                        NL, KL, 64, 1, st), "lut4_matmul");

    /* GGML Q4_0 routed mat-vec (mode 1: no workspace). */
    size_t bmx = (size_t)T * KQ * 4, bmw = (size_t)E * STRIDE, bmi = (size_t)T * TOPK * 4;
    size_t bmo = (size_t)T * TOPK * NQ * 4;
    void *hmx = read_file(dir, "moe_x.bin", bmx), *hmw = read_file(dir, "moe_w.bin", bmw);
    void *hmi = read_file(dir, "moe_ids.bin", bmi);
    void *dmx = to_device(hmx, bmx), *dmw = to_device(hmw, bmw), *dmi = to_device(hmi, bmi), *dmo = NULL;
    cuda_ok(cudaMalloc(&dmo, bmo), "cudaMalloc moe out");
    q4mm_ok(q4_0_matmul_id((const float *)dmx, dmw, (const uint32_t *)dmi, (float *)dmo, T, TOPK, NQ, KQ, E, STRIDE, 1,
                           NULL, 0, st), "q4_0_matmul_id");

    cuda_ok(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
    uint32_t flags = 0;
    q4mm_ok(q4mm_device_errors(&flags, 1), "q4mm_device_errors");
    if (flags != 0) {
        fprintf(stderr, "device error flags 0x%x\n", flags);
        return 5;
    }

    void *out = malloc(by > bly ? (by > bmo ? by : bmo) : (bly > bmo ? bly : bmo));
    cuda_ok(cudaMemcpy(out, dy1, by, cudaMemcpyDeviceToHost), "D2H");
    write_file(dir, "gemv_y.bin", out, by);
    cuda_ok(cudaMemcpy(out, dy2, by, cudaMemcpyDeviceToHost), "D2H");
    write_file(dir, "gemm_y.bin", out, by);
    cuda_ok(cudaMemcpy(out, dly, bly, cudaMemcpyDeviceToHost), "D2H");
    write_file(dir, "lut4_y.bin", out, bly);
    cuda_ok(cudaMemcpy(out, dmo, bmo, cudaMemcpyDeviceToHost), "D2H");
    write_file(dir, "moe_out.bin", out, bmo);

    void *dev_bufs[] = {dx, dw, ds, db, dy1, dy2, dlx, dlp, dls, dly, dmx, dmw, dmi, dmo};
    for (size_t i = 0; i < sizeof dev_bufs / sizeof dev_bufs[0]; ++i) cudaFree(dev_bufs[i]);
    void *host_bufs[] = {hx, hw, hs, hb, hlx, hlp, hls, book, hmx, hmw, hmi, out};
    for (size_t i = 0; i < sizeof host_bufs / sizeof host_bufs[0]; ++i) free(host_bufs[i]);
    cudaStreamDestroy(stream);
    printf("c_abi_consumer ok\n");
    return 0;
}
