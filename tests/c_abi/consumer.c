/*
 * A plain C consumer of libtrfn.so: the C ABI used without Python or C++.
 * It normalises a seeded 8 x 32 x 48 x 3 batch (ImageNet preset, flip and
 * erase records from tr_sample_aug_params) to binary16 NHWC on the GPU and
 * writes the input, the records and the output to files for the test to
 * check against the oracle.
 *
 * usage: consumer <out_dir>      exit status 0 on success
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "tr_fused_norm.h"

enum { N = 8, H = 32, W = 48, C = 3 };

static int write_file(const char* dir, const char* name, const void* p, size_t n) {
    char path[1024];
    FILE* f;
    snprintf(path, sizeof path, "%s/%s", dir, name);
    f = fopen(path, "wb");
    if (!f) return 1;
    if (fwrite(p, 1, n, f) != n) {
        fclose(f);
        return 1;
    }
    return fclose(f) != 0;
}

#define CHECK_TR(call)                                                             \
    do {                                                                           \
        int rc_ = (call);                                                          \
        if (rc_ != TR_OK) {                                                        \
            fprintf(stderr, "%s: %s (%s)\n", #call, tr_status_string(rc_),         \
                    tr_last_error_message());                                      \
            return 1;                                                              \
        }                                                                          \
    } while (0)

#define CHECK_CUDA(call)                                                           \
    do {                                                                           \
        cudaError_t e_ = (call);                                                   \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));            \
            return 1;                                                              \
        }                                                                          \
    } while (0)

int main(int argc, char** argv) {
    const size_t in_bytes = (size_t)N * H * W * C;
    const size_t out_bytes = in_bytes * 2;
    float mean[3], std[3];
    int channels = 0, flags = -1;
    uint64_t next = 0;
    tr_aug_param rec[N];
    uint8_t* src = (uint8_t*)malloc(in_bytes);
    uint16_t* out = (uint16_t*)malloc(out_bytes);
    uint8_t *d_src = NULL, *d_dst = NULL;
    tr_aug_param* d_rec = NULL;
    uint32_t state = 12345u;
    size_t i;
    if (argc < 2 || !src || !out) return 2;

    for (i = 0; i < in_bytes; ++i) {   /* a fixed xorshift stream */
        state ^= state << 13;
        state ^= state >> 17;
        state ^= state << 5;
        src[i] = (uint8_t)(state >> 24);
    }
    CHECK_TR(tr_norm_preset(TR_PRESET_IMAGENET, mean, std, &channels));
    if (channels != C) return 3;
    CHECK_TR(tr_sample_aug_params(77u, 0u, N, H, W, 1, 0.5f, 1, 0.5f, 0.02f, 0.33f, 0.3f, 3.3f, rec, &next));

    CHECK_CUDA(cudaMalloc((void**)&d_src, in_bytes));
    CHECK_CUDA(cudaMalloc((void**)&d_dst, out_bytes));
    CHECK_CUDA(cudaMalloc((void**)&d_rec, sizeof rec));
    CHECK_CUDA(cudaMemcpy(d_src, src, in_bytes, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_rec, rec, sizeof rec, cudaMemcpyHostToDevice));
    /* the tiled kernel, forced (AUTO would pick the per-element kernel for so small a batch) */
    CHECK_TR(tr_fused_norm_variant(d_src, d_dst, N, H, W, C, mean, std, d_rec, TR_OUT_F16, TR_LAYOUT_NHWC,
                                   NULL, TR_VARIANT_TILED));
    CHECK_CUDA(cudaDeviceSynchronize());
    CHECK_CUDA(cudaMemcpy(out, d_dst, out_bytes, cudaMemcpyDeviceToHost));
    CHECK_TR(tr_device_status(&flags, 0));
    if (flags != 0) return 4;

    if (write_file(argv[1], "src.u8", src, in_bytes) || write_file(argv[1], "rec.i32", rec, sizeof rec) ||
        write_file(argv[1], "out.f16", out, out_bytes))
        return 5;
    cudaFree(d_src);
    cudaFree(d_dst);
    cudaFree(d_rec);
    free(src);
    free(out);
    printf("consumer ok, next offset %llu\n", (unsigned long long)next);
    return 0;
}
