/*
 * abi_consumer.c -- a plain C program that uses the library only through
 * include/rope3d.h and the CUDA runtime: it reads Q and K from files, rotates
 * them with rope3d_apply_pair (device buffers) and rope3d_apply_pair_host
 * (host buffers), checks that the two agree, and writes Q_out and K_out.
 * tests/test_gpu_c_abi.py builds and runs it and compares the outputs with the
 * CPU oracle.
 *
 * usage: abi_consumer q.bin k.bin q_out.bin k_out.bin B T H W heads head_dim d_T d_H d_W dtype
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "rope3d.h"

static int fail(const char *what, int rc)
{
    fprintf(stderr, "%s failed: %d (%s)\n", what, rc, rope3d_status_string(rc));
    return 1;
}

static void *read_file(const char *path, size_t bytes)
{
    FILE *f = fopen(path, "rb");
    if (!f)
        return NULL;
    void *buf = malloc(bytes);
    if (buf && fread(buf, 1, bytes, f) != bytes) {
        free(buf);
        buf = NULL;
    }
    fclose(f);
    return buf;
}

static int write_file(const char *path, const void *buf, size_t bytes)
{
    FILE *f = fopen(path, "wb");
    if (!f)
        return -1;
    size_t n = fwrite(buf, 1, bytes, f);
    fclose(f);
    return n == bytes ? 0 : -1;
}

int main(int argc, char **argv)
{
    if (argc != 15) {
        fprintf(stderr, "usage: %s q k q_out k_out B T H W heads head_dim dT dH dW dtype\n", argv[0]);
        return 2;
    }
    const int64_t B = atoll(argv[5]), T = atoll(argv[6]), H = atoll(argv[7]), W = atoll(argv[8]);
    const int64_t heads = atoll(argv[9]), head_dim = atoll(argv[10]);
    const int32_t split[3] = {atoi(argv[11]), atoi(argv[12]), atoi(argv[13])};
    const int32_t dtype = atoi(argv[14]);
    const size_t esize = dtype == ROPE3D_F32 ? 4 : 2;
    const size_t bytes = (size_t)(B * T * H * W * heads * head_dim) * esize;

    void *hq = read_file(argv[1], bytes), *hk = read_file(argv[2], bytes);
    if (!hq || !hk) {
        fprintf(stderr, "cannot read the inputs\n");
        return 1;
    }
    void *dq, *dk, *dqo, *dko;
    if (cudaMalloc(&dq, bytes) || cudaMalloc(&dk, bytes) || cudaMalloc(&dqo, bytes) ||
        cudaMalloc(&dko, bytes))
        return fail("cudaMalloc", ROPE3D_ERR_NOMEM);
    cudaMemcpy(dq, hq, bytes, cudaMemcpyHostToDevice);
    cudaMemcpy(dk, hk, bytes, cudaMemcpyHostToDevice);

    rope3d_tables *tables = NULL;
    int rc = rope3d_build_tables(T, H, W, split, 10000.0, NULL, &tables);
    if (rc != ROPE3D_OK)
        return fail("rope3d_build_tables", rc);
    rc = rope3d_apply_pair(dq, dk, dqo, dko, tables, B, T, H, W, heads, head_dim, split, dtype, NULL);
    if (rc != ROPE3D_OK)
        return fail("rope3d_apply_pair", rc);
    if (cudaDeviceSynchronize() != cudaSuccess)
        return fail("cudaDeviceSynchronize", ROPE3D_ERR_CUDA);

    void *oq = malloc(bytes), *ok = malloc(bytes), *hoq = malloc(bytes), *hok = malloc(bytes);
    cudaMemcpy(oq, dqo, bytes, cudaMemcpyDeviceToHost);
    cudaMemcpy(ok, dko, bytes, cudaMemcpyDeviceToHost);

    /* the host-buffer entry point gives the same bytes */
    rc = rope3d_apply_pair_host(hq, hk, hoq, hok, tables, B, T, H, W, heads, head_dim, split, dtype, NULL);
    if (rc != ROPE3D_OK)
        return fail("rope3d_apply_pair_host", rc);
    if (memcmp(oq, hoq, bytes) != 0 || memcmp(ok, hok, bytes) != 0) {
        fprintf(stderr, "device and host entry points disagree\n");
        return 1;
    }
    /* a preflight rejection comes back as a status, not a crash */
    rc = rope3d_apply_pair(dq, dk, dq, dko, tables, B, T, H, W, heads, head_dim, split, dtype, NULL);
    if (rc != ROPE3D_ERR_ALIAS)
        return fail("aliased call (expected ROPE3D_ERR_ALIAS)", rc);

    if (write_file(argv[3], oq, bytes) || write_file(argv[4], ok, bytes)) {
        fprintf(stderr, "cannot write the outputs\n");
        return 1;
    }
    rope3d_release_tables(tables);
    rope3d_release_scratch();
    cudaFree(dq);
    cudaFree(dk);
    cudaFree(dqo);
    cudaFree(dko);
    free(hq);
    free(hk);
    free(oq);
    free(ok);
    free(hoq);
    free(hok);
    printf("ok\n");
    return 0;
}
