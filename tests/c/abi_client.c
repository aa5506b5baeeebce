/* A plain C client of libew.so: compiled by the tests with a C compiler
 * against include/ew.h only (no CUDA headers), to show the ABI is usable from
 * C.  Mode "host": argument validation and planning, which never reach the
 * GPU.  Mode "gpu": allocates device memory through the CUDA runtime,
 * runs ew_add / ew_relu / ew_add_relu on the inputs read from argv[2], argv[3]
 * (raw binary32 files) and writes the results to argv[4]-argv[6]. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ew.h"

#define EXPECT(cond)                                                        \
    do {                                                                    \
        if (!(cond)) {                                                      \
            fprintf(stderr, "%s:%d: check failed: %s\n", __FILE__, __LINE__, #cond); \
            return 1;                                                       \
        }                                                                   \
    } while (0)

static int host_mode(void) {
    void *p = (void *)(uintptr_t)0x10000000u; /* never dereferenced */
    char *q = (char *)p;
    EXPECT(ew_version() >= 100);
    EXPECT(ew_add(EW_F32, p, q + 4096, q + 8192, 0, NULL) == EW_OK);
    EXPECT(ew_add(EW_F32, NULL, q + 4096, q + 8192, 10, NULL) == EW_ERR_NULL_POINTER);
    EXPECT(ew_add((ew_dtype)9, p, q + 4096, q + 8192, 10, NULL) == EW_ERR_UNSUPPORTED_DTYPE);
    EXPECT(ew_add(EW_F32, p, q + 4096, q + 4, 10, NULL) == EW_ERR_OVERLAP);
    EXPECT(ew_relu(EW_BF16, q + 1, q + 4096, 10, NULL) == EW_ERR_INVALID_VALUE);
    EXPECT(ew_gather_stride(EW_F16, p, q + 4096, 10, 0, NULL) == EW_ERR_INVALID_VALUE);
    EXPECT(ew_set_path((ew_path)7) == EW_ERR_INVALID_VALUE);
    EXPECT(ew_set_schedule((ew_schedule)7) == EW_ERR_INVALID_VALUE);
    EXPECT(strncmp(ew_status_string(EW_ERR_OVERLAP), "EW_ERR_OVERLAP", 14) == 0);

    const void *ptrs[3] = {q + 2, q + 2 + 4096, q + 2 + 8192};
    ew_plan pl;
    EXPECT(ew_plan_query(EW_BF16, ptrs, 3, 1000, &pl) == EW_OK);
    EXPECT(pl.vec_bytes == 32 && pl.head == 15);
    EXPECT(pl.head + pl.nvec * 16 + pl.tail == 1000);
    EXPECT(ew_set_path(EW_PATH_V128) == EW_OK);
    EXPECT(ew_plan_query(EW_BF16, ptrs, 3, 1000, &pl) == EW_OK);
    EXPECT(pl.vec_bytes == 16 && pl.head == 7);
    EXPECT(pl.head + pl.nvec * 8 + pl.tail == 1000);
    EXPECT(ew_set_path(EW_PATH_AUTO) == EW_OK);

    ew_launch_record rec;
    EXPECT(ew_last_launch(&rec) == EW_OK && rec.launches == 0);
    /* a gather plan, host only: stride 12 on 2^20 fp32 elements runs the
       fixed-stride tiled kernel, 192 threads, 320 lap positions per block */
    EXPECT(ew_gather_plan_query(EW_F32, q, q + (1 << 22), 1 << 20, 12, &rec) == EW_OK);
    EXPECT(rec.launches == 1 && rec.schedule == EW_SCHED_TILED && rec.block == 192);
    EXPECT(rec.grid == ((1 << 20) / 12 + 1 + 319) / 320 && rec.vec_bytes == 16);
    EXPECT(ew_gather_plan_query(EW_F32, q, q + (1 << 22), 1 << 20, 12, NULL) == EW_ERR_NULL_POINTER);
    printf("host ok\n");
    return 0;
}

/* The few CUDA runtime entry points the GPU mode needs, declared by hand so
 * that this file includes no CUDA header. */
extern int cudaMalloc(void **p, size_t bytes);
extern int cudaFree(void *p);
extern int cudaMemcpy(void *dst, const void *src, size_t bytes, int kind);
extern int cudaDeviceSynchronize(void);

static float *read_f32(const char *path, int64_t *n) {
    FILE *f = fopen(path, "rb");
    if (!f) return NULL;
    fseek(f, 0, SEEK_END);
    long bytes = ftell(f);
    fseek(f, 0, SEEK_SET);
    float *buf = (float *)malloc((size_t)bytes);
    if (buf && fread(buf, 1, (size_t)bytes, f) != (size_t)bytes) { free(buf); buf = NULL; }
    fclose(f);
    *n = bytes / 4;
    return buf;
}

static int write_f32(const char *path, const float *buf, int64_t n) {
    FILE *f = fopen(path, "wb");
    if (!f) return 1;
    size_t w = fwrite(buf, 4, (size_t)n, f);
    fclose(f);
    return w == (size_t)n ? 0 : 1;
}

static int gpu_mode(char **argv) {
    int64_t n = 0, nb = 0;
    float *a = read_f32(argv[2], &n), *b = read_f32(argv[3], &nb);
    EXPECT(a && b && n == nb && n > 0);
    float *out = (float *)malloc((size_t)n * 4);
    void *da, *db, *dc;
    EXPECT(cudaMalloc(&da, (size_t)n * 4) == 0);
    EXPECT(cudaMalloc(&db, (size_t)n * 4) == 0);
    EXPECT(cudaMalloc(&dc, (size_t)n * 4) == 0);
    EXPECT(cudaMemcpy(da, a, (size_t)n * 4, 1) == 0); /* host to device */
    EXPECT(cudaMemcpy(db, b, (size_t)n * 4, 1) == 0);

    EXPECT(ew_add(EW_F32, da, db, dc, n, NULL) == EW_OK);
    EXPECT(cudaMemcpy(out, dc, (size_t)n * 4, 2) == 0); /* device to host */
    EXPECT(write_f32(argv[4], out, n) == 0);

    EXPECT(ew_relu(EW_F32, da, dc, n, NULL) == EW_OK);
    EXPECT(cudaMemcpy(out, dc, (size_t)n * 4, 2) == 0);
    EXPECT(write_f32(argv[5], out, n) == 0);

    EXPECT(ew_add_relu(EW_F32, da, db, dc, n, NULL) == EW_OK);
    EXPECT(cudaMemcpy(out, dc, (size_t)n * 4, 2) == 0);
    EXPECT(write_f32(argv[6], out, n) == 0);

    int32_t code = -1;
    EXPECT(ew_device_error(NULL, &code) == EW_OK && code == 0);
    EXPECT(cudaDeviceSynchronize() == 0);
    cudaFree(da);
    cudaFree(db);
    cudaFree(dc);
    free(a);
    free(b);
    free(out);
    printf("gpu ok\n");
    return 0;
}

int main(int argc, char **argv) {
    if (argc >= 2 && strcmp(argv[1], "host") == 0) return host_mode();
    if (argc >= 7 && strcmp(argv[1], "gpu") == 0) return gpu_mode(argv);
    fprintf(stderr, "usage: abi_client host | gpu a.bin b.bin add.bin relu.bin add_relu.bin\n");
    return 2;
}
