/*
 * A plain C caller of the paged decode-attention library: no Python, no
 * torch, only include/pa.h and the CUDA runtime for device memory.
 *
 * Usage: pa_c_client DIR
 * DIR/sizes.txt holds "S Hq Hkv hd bs num_blocks max_blocks dtype partition
 * num_pairs scale" (dtype 0 = fp32, 1 = bf16); DIR/{q,k_cache,v_cache,k_new,v_new}.bin
 * hold the tensors in the layouts include/pa.h states, DIR/{tables,lens}.bin
 * int32, DIR/{slots,pairs}.bin int64.  The client runs one decode step the way
 * a serving loop would: the copy-on-write block copies, the new tokens' cache
 * write, then decode attention, and writes DIR/{out,k_cache_out,v_cache_out}.bin.
 * Exit status 0 on success; any library or CUDA error is printed.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "pa.h"

static void *read_file(const char *dir, const char *name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) { fprintf(stderr, "cannot open %s\n", path); exit(2); }
    void *buf = malloc(bytes ? bytes : 1);
    if (!buf || fread(buf, 1, bytes, f) != bytes) { fprintf(stderr, "short read %s\n", path); exit(2); }
    fclose(f);
    return buf;
}

static void write_file(const char *dir, const char *name, const void *buf, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (!f || fwrite(buf, 1, bytes, f) != bytes) { fprintf(stderr, "cannot write %s\n", path); exit(2); }
    fclose(f);
}

static void *to_device(const void *host, size_t bytes) {
    void *d = NULL;
    if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess) { fprintf(stderr, "cudaMalloc failed\n"); exit(3); }
    if (bytes && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        fprintf(stderr, "cudaMemcpy failed\n");
        exit(3);
    }
    return d;
}

static void check(int rc, const char *what) {
    if (rc != PA_OK) {
        fprintf(stderr, "%s failed: %d (%s)\n", what, rc, pa_last_error_string());
        exit(4);
    }
}

int main(int argc, char **argv) {
    if (argc != 2) { fprintf(stderr, "usage: %s DIR\n", argv[0]); return 1; }
    const char *dir = argv[1];
    char path[4096];
    snprintf(path, sizeof path, "%s/sizes.txt", dir);
    FILE *f = fopen(path, "r");
    int S, Hq, Hkv, hd, bs, nb, mb, dtype, P, npairs;
    float scale;
    if (!f || fscanf(f, "%d %d %d %d %d %d %d %d %d %d %f", &S, &Hq, &Hkv, &hd, &bs, &nb, &mb, &dtype, &P,
                     &npairs, &scale) != 11) {
        fprintf(stderr, "bad sizes.txt\n");
        return 2;
    }
    fclose(f);
    const size_t e = dtype == PA_F32 ? 4 : 2;
    const size_t qb = (size_t)S * Hq * hd * e, cb = (size_t)nb * Hkv * bs * hd * e, nbytes = (size_t)S * Hkv * hd * e;
    void *hq = read_file(dir, "q.bin", qb), *hk = read_file(dir, "k_cache.bin", cb);
    void *hv = read_file(dir, "v_cache.bin", cb), *hkn = read_file(dir, "k_new.bin", nbytes);
    void *hvn = read_file(dir, "v_new.bin", nbytes);
    int32_t *ht = read_file(dir, "tables.bin", (size_t)S * mb * 4), *hl = read_file(dir, "lens.bin", (size_t)S * 4);
    int64_t *hs = read_file(dir, "slots.bin", (size_t)S * 8), *hp = read_file(dir, "pairs.bin", (size_t)npairs * 16);
    int max_len = 0;
    for (int i = 0; i < S; ++i) max_len = hl[i] > max_len ? hl[i] : max_len;

    void *q = to_device(hq, qb), *kc = to_device(hk, cb), *vc = to_device(hv, cb);
    void *kn = to_device(hkn, nbytes), *vn = to_device(hvn, nbytes);
    void *t = to_device(ht, (size_t)S * mb * 4), *l = to_device(hl, (size_t)S * 4);
    void *slots = to_device(hs, (size_t)S * 8), *pairs = to_device(hp, (size_t)npairs * 16);
    void *out = NULL;
    if (cudaMalloc(&out, qb) != cudaSuccess) return 3;
    int32_t *status = NULL;
    if (cudaMalloc((void **)&status, 4) != cudaSuccess || cudaMemset(status, 0, 4) != cudaSuccess) return 3;

    /* workspace for the split-K partials, sized by the library */
    const size_t ws_bytes = pa_decode_workspace_size(S, Hq, hd, max_len, P);
    void *ws = NULL;
    if (ws_bytes && (cudaMalloc(&ws, ws_bytes) != cudaSuccess || cudaMemset(ws, 0, ws_bytes) != cudaSuccess))
        return 3;

    check(pa_copy_blocks(kc, vc, pairs, npairs, Hkv, hd, bs, nb, dtype, status, NULL), "pa_copy_blocks");
    check(pa_reshape_and_cache(kn, vn, kc, vc, slots, S, Hkv, hd, bs, nb, dtype, status, NULL),
          "pa_reshape_and_cache");
    pa_decode_args a;
    memset(&a, 0, sizeof a);
    a.num_seqs = S;
    a.max_blocks_per_seq = mb;
    a.num_blocks = nb;
    a.dtype = dtype;
    a.partition_size = P;
    a.max_context_len = max_len;
    a.workspace = ws;
    a.workspace_bytes = ws_bytes;
    a.dev_status = status;
    a.stream = NULL;
    a.phase = PA_PHASE_ALL;
    check(pa_decode(out, q, kc, vc, t, l, Hq, Hkv, hd, bs, scale, &a), "pa_decode");
    if (cudaDeviceSynchronize() != cudaSuccess) { fprintf(stderr, "device error\n"); return 3; }

    int32_t st = -1;
    void *hout = malloc(qb), *hk2 = malloc(cb), *hv2 = malloc(cb);
    if (cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(hout, out, qb, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(hk2, kc, cb, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(hv2, vc, cb, cudaMemcpyDeviceToHost) != cudaSuccess)
        return 3;
    if (st != 0) { fprintf(stderr, "device status %d\n", st); return 5; }
    write_file(dir, "out.bin", hout, qb);
    write_file(dir, "k_cache_out.bin", hk2, cb);
    write_file(dir, "v_cache_out.bin", hv2, cb);
    printf("pa_c_client: %d sequences decoded, library version %x\n", S, pa_version());
    return 0;
}
