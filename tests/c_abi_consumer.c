/* A plain C (C11) consumer of libropekv: includes include/ropekv.h, links the
 * shared library and the CUDA runtime, and calls the C ABI with raw pointers
 * and sizes -- no Python, no torch.
 *
 *   c_abi_consumer host
 *       host-only calls: rope_check_capacity, ropekv_status_string and
 *       ropekv_set_residency_cap; prints one line per result.
 *   c_abi_consumer packed B S Hq Hkv D r cap style cos_sin.bin qkv.bin out_qkv.bin out_cache.bin
 *       reads the FP32 cos/sin table [1, cap, r] and the FP16 qkv bits
 *       [B, S, Hq+2Hkv, D], runs rope_write_kv_packed on the device with a
 *       zeroed cache [B, 2, Hkv, cap, D], and writes the rotated qkv and the
 *       cache back as raw bits.
 * Exit status 0 on success; any CUDA or library error is printed and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ropekv.h"

static int fail_cuda(const char* what, cudaError_t e)
{
    fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
    return 1;
}

static void* read_file(const char* path, size_t bytes)
{
    FILE* f = fopen(path, "rb");
    void* p = malloc(bytes ? bytes : 1);
    if (!f || !p || fread(p, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot read %zu bytes from %s\n", bytes, path);
        exit(1);
    }
    fclose(f);
    return p;
}

static void write_file(const char* path, const void* p, size_t bytes)
{
    FILE* f = fopen(path, "wb");
    if (!f || fwrite(p, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot write %s\n", path);
        exit(1);
    }
    fclose(f);
}

static int run_host(void)
{
    printf("capacity(4096, 4096) = %d\n", rope_check_capacity(4096, 4096));
    printf("capacity(4097, 4096) = %d\n", rope_check_capacity(4097, 4096));
    for (int s = 0; s >= -10; --s)
        printf("status %d: %s\n", s, ropekv_status_string(s));
    /* the residency-cap switch returns its previous setting (on by default) */
    const int was = ropekv_set_residency_cap(0);
    const int now = ropekv_set_residency_cap(was);
    printf("residency cap: default %d, after switching off %d\n", was, now);
    return 0;
}

static int run_packed(char** v)
{
    ropekv_dims d;
    memset(&d, 0, sizeof d);
    d.batch = atoi(v[0]);
    d.seqLen = atoi(v[1]);
    d.numQHeads = atoi(v[2]);
    d.numKVHeads = atoi(v[3]);
    d.headDim = atoi(v[4]);
    d.rotaryDim = atoi(v[5]);
    d.kvCapacity = atoi(v[6]);
    d.style = atoi(v[7]);
    d.cosSinBatch = 1;
    d.cosSinSeqLen = d.kvCapacity;
    const size_t H = (size_t)d.numQHeads + 2 * (size_t)d.numKVHeads;
    const size_t csBytes = (size_t)d.kvCapacity * d.rotaryDim * sizeof(float);
    const size_t qkvBytes = (size_t)d.batch * d.seqLen * H * d.headDim * sizeof(uint16_t);
    const size_t cacheBytes =
        (size_t)d.batch * 2 * d.numKVHeads * d.kvCapacity * d.headDim * sizeof(uint16_t);

    float* hCs = (float*)read_file(v[8], csBytes);
    uint16_t* hQkv = (uint16_t*)read_file(v[9], qkvBytes);
    uint16_t* hCache = (uint16_t*)malloc(cacheBytes);
    float* dCs = NULL;
    uint16_t *dQkv = NULL, *dCache = NULL;
    cudaError_t e;
    if ((e = cudaMalloc((void**)&dCs, csBytes)) != cudaSuccess) return fail_cuda("cudaMalloc", e);
    if ((e = cudaMalloc((void**)&dQkv, qkvBytes)) != cudaSuccess) return fail_cuda("cudaMalloc", e);
    if ((e = cudaMalloc((void**)&dCache, cacheBytes)) != cudaSuccess)
        return fail_cuda("cudaMalloc", e);
    if ((e = cudaMemcpy(dCs, hCs, csBytes, cudaMemcpyHostToDevice)) != cudaSuccess ||
        (e = cudaMemcpy(dQkv, hQkv, qkvBytes, cudaMemcpyHostToDevice)) != cudaSuccess ||
        (e = cudaMemset(dCache, 0, cacheBytes)) != cudaSuccess)
        return fail_cuda("upload", e);

    const int rc = rope_write_kv_packed(dCs, dQkv, dCache, &d, NULL);
    if (rc != ROPEKV_OK) {
        fprintf(stderr, "rope_write_kv_packed: %s\n", ropekv_status_string(rc));
        return 1;
    }
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return fail_cuda("kernel", e);
    if ((e = cudaMemcpy(hQkv, dQkv, qkvBytes, cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemcpy(hCache, dCache, cacheBytes, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return fail_cuda("download", e);
    write_file(v[10], hQkv, qkvBytes);
    write_file(v[11], hCache, cacheBytes);
    cudaFree(dCs);
    cudaFree(dQkv);
    cudaFree(dCache);
    free(hCs);
    free(hQkv);
    free(hCache);
    printf("ok\n");
    return 0;
}

int main(int argc, char** argv)
{
    if (argc == 2 && strcmp(argv[1], "host") == 0)
        return run_host();
    if (argc == 14 && strcmp(argv[1], "packed") == 0)
        return run_packed(argv + 2);
    fprintf(stderr, "usage: %s host | packed B S Hq Hkv D r cap style cs qkv out_qkv out_cache\n",
            argv[0]);
    return 2;
}
