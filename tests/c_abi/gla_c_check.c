/*
 * gla_c_check.c -- drives libgla through its C ABI from plain C: no Python,
 * no torch. Reads a case written by tests/test_gpu_c_abi.py (raw
 * little-endian files in a directory), runs gla_chunk_fwd (bf16) and
 * gla_decode_step (bf16) on a stream it creates, and writes the outputs back
 * for the test to compare against the oracle.
 *
 *   gla_c_check <dir> B T H
 * Files in <dir>: q.bin k.bin v.bin (bf16 bits, [B,T,H,96] / [B,T,H,192]),
 * ll.bin (fp32 [H]), scale.bin (fp32), dq.bin dk.bin dv.bin (bf16, decode
 * step [B,H,96] / [B,H,192]). Written: o.bin (bf16), hT.bin (fp32),
 * od.bin (bf16), S.bin (fp32, the state after the decode step, which starts
 * from hT).
 */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gla.h"

static void *read_file(const char *dir, const char *name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) { fprintf(stderr, "cannot open %s\n", path); exit(2); }
    void *p = malloc(bytes);
    if (fread(p, 1, bytes, f) != bytes) { fprintf(stderr, "short read %s\n", path); exit(2); }
    fclose(f);
    return p;
}

static void write_file(const char *dir, const char *name, const void *p, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (!f || fwrite(p, 1, bytes, f) != bytes) { fprintf(stderr, "cannot write %s\n", path); exit(2); }
    fclose(f);
}

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
    fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_)); return 3; } } while (0)
#define GK(x) do { gla_status s_ = (x); if (s_ != GLA_OK) { \
    fprintf(stderr, "%s: %s (%s)\n", #x, gla_status_string(s_), gla_last_error()); return 4; } } while (0)

static void *to_device(const void *h, size_t bytes) {
    void *d = NULL;
    if (cudaMalloc(&d, bytes) != cudaSuccess || cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        fprintf(stderr, "device copy failed\n");
        exit(3);
    }
    return d;
}

int main(int argc, char **argv) {
    if (argc != 5) { fprintf(stderr, "usage: %s dir B T H\n", argv[0]); return 1; }
    const char *dir = argv[1];
    const int B = atoi(argv[2]), T = atoi(argv[3]), H = atoi(argv[4]);
    const int dk = 96, dv = 192, C = 128;
    const size_t nq = (size_t)B * T * H * dk, nv = (size_t)B * T * H * dv, ns = (size_t)B * H * dk * dv;
    float scale;
    float *sp = read_file(dir, "scale.bin", sizeof(float));
    scale = *sp;
    void *hq = read_file(dir, "q.bin", nq * 2), *hk = read_file(dir, "k.bin", nq * 2);
    void *hv = read_file(dir, "v.bin", nv * 2), *hll = read_file(dir, "ll.bin", (size_t)H * 4);
    void *hdq = read_file(dir, "dq.bin", (size_t)B * H * dk * 2), *hdk = read_file(dir, "dk.bin", (size_t)B * H * dk * 2);
    void *hdv = read_file(dir, "dv.bin", (size_t)B * H * dv * 2);

    cudaStream_t st;
    CK(cudaStreamCreate(&st));
    void *q = to_device(hq, nq * 2), *k = to_device(hk, nq * 2), *v = to_device(hv, nv * 2);
    float *ll = to_device(hll, (size_t)H * 4);
    void *o = NULL, *od = NULL;
    float *hT = NULL;
    CK(cudaMalloc(&o, nv * 2));
    CK(cudaMalloc((void **)&hT, ns * 4));
    CK(cudaMalloc(&od, (size_t)B * H * dv * 2));
    size_t ws_bytes = gla_chunk_fwd_workspace_size(B, T, H, dk, dv, C, GLA_BF16);
    void *ws = NULL;
    if (ws_bytes) CK(cudaMalloc(&ws, ws_bytes));

    GK(gla_chunk_fwd(q, k, v, ll, NULL, scale, B, T, H, dk, dv, C, GLA_BF16, o, hT, ws, ws_bytes, st));
    /* one serving step from the prefill's final state (the state page is hT) */
    void *dq = to_device(hdq, (size_t)B * H * dk * 2), *dkk = to_device(hdk, (size_t)B * H * dk * 2);
    void *dvv = to_device(hdv, (size_t)B * H * dv * 2);
    float *S = NULL;
    CK(cudaMalloc((void **)&S, ns * 4));
    CK(cudaMemcpyAsync(S, hT, ns * 4, cudaMemcpyDeviceToDevice, st));
    GK(gla_decode_step(dq, dkk, dvv, ll, S, scale, B, H, dk, dv, GLA_BF16, od, st));
    GK(gla_check(st));

    void *out = malloc(nv * 2 > ns * 4 ? nv * 2 : ns * 4);
    CK(cudaMemcpy(out, o, nv * 2, cudaMemcpyDeviceToHost));
    write_file(dir, "o.bin", out, nv * 2);
    CK(cudaMemcpy(out, hT, ns * 4, cudaMemcpyDeviceToHost));
    write_file(dir, "hT.bin", out, ns * 4);
    CK(cudaMemcpy(out, od, (size_t)B * H * dv * 2, cudaMemcpyDeviceToHost));
    write_file(dir, "od.bin", out, (size_t)B * H * dv * 2);
    CK(cudaMemcpy(out, S, ns * 4, cudaMemcpyDeviceToHost));
    write_file(dir, "S.bin", out, ns * 4);
    printf("launches in the last call: %d\n", gla_last_launch_count());
    return 0;
}
