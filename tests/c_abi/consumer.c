/* A plain C consumer of libfp8q.so: the C ABI used without Python or torch.
 *
 *   consumer check              argument checks only (no GPU work: every call
 *                               fails validation or is an empty no-op)
 *   consumer quantize IN OUT F  reads n bf16 values (uint16 bit patterns) from
 *                               file IN, quantizes them on the GPU with
 *                               fp8q_quantize_blockwise in format F (0 = e4m3,
 *                               1 = e5m2), and writes the n codes followed by
 *                               the ceil(n/128) float scales to file OUT.
 * The caller compares OUT with the oracle; this program holds none of the
 * codec's arithmetic.  Exit status 0 on success. */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fp8q.h"

static int expect(const char* what, fp8q_status_t got, fp8q_status_t want) {
    if (got != want) {
        fprintf(stderr, "%s: status %d (%s), expected %d\n", what, (int)got, fp8q_status_string(got), (int)want);
        return 1;
    }
    return 0;
}

static int check(void) {
    void* a = (void*)(uintptr_t)0x7F0000000000ull;      /* aligned fake device addresses, never touched */
    uint8_t* c = (uint8_t*)(uintptr_t)0x7F0001000000ull;
    float* s = (float*)(uintptr_t)0x7F0002000000ull;
    int bad = 0;
    bad |= expect("empty input", fp8q_quantize_blockwise(NULL, 0, FP8Q_E4M3, NULL, NULL, NULL), FP8Q_OK);
    bad |= expect("null input", fp8q_quantize_blockwise(NULL, 1024, FP8Q_E4M3, c, s, NULL), FP8Q_ERR_NULL);
    bad |= expect("bad format", fp8q_quantize_blockwise(a, 1024, (fp8q_format_t)7, c, s, NULL), FP8Q_ERR_FORMAT);
    bad |= expect("misaligned", fp8q_quantize_blockwise((char*)a + 2, 1024, FP8Q_E4M3, c, s, NULL), FP8Q_ERR_ALIGN);
    bad |= expect("too large", fp8q_quantize_blockwise(a, FP8Q_MAX_ELEMENTS + 1, FP8Q_E4M3, c, s, NULL),
                  FP8Q_ERR_SIZE);
    bad |= expect("mxfp8 K", mxfp8_quantize_swizzled(a, 1, 128, 48, c, (uint8_t*)s, NULL), FP8Q_ERR_K);
    if (fp8q_num_scales(129) != 2 || fp8q_num_scales(0) != 0) bad |= 1;
    if (mxfp8_swizzled_scale_bytes(1, 256, 256) != 2048) bad |= 1;
    if (strcmp(fp8q_status_string(FP8Q_OK), "ok") != 0) bad |= 1;
    printf(bad ? "check: FAILED\n" : "check: ok\n");
    return bad;
}

static int quantize(const char* in, const char* out, int fmt) {
    FILE* f = fopen(in, "rb");
    if (!f) return 2;
    fseek(f, 0, SEEK_END);
    const size_t n = (size_t)ftell(f) / 2;
    fseek(f, 0, SEEK_SET);
    uint16_t* x = (uint16_t*)malloc(2 * n + 16);
    if (!x || fread(x, 2, n, f) != n) return 2;
    fclose(f);
    const size_t nb = fp8q_num_scales(n);
    void *dx = NULL, *dc = NULL, *ds = NULL;
    if (cudaMalloc(&dx, 2 * n + 16) != cudaSuccess || cudaMalloc(&dc, n + 16) != cudaSuccess ||
        cudaMalloc(&ds, 4 * nb + 16) != cudaSuccess)
        return 3;
    if (cudaMemcpy(dx, x, 2 * n, cudaMemcpyHostToDevice) != cudaSuccess) return 3;
    const fp8q_status_t st = fp8q_quantize_blockwise(dx, n, (fp8q_format_t)fmt, (uint8_t*)dc, (float*)ds, NULL);
    if (st != FP8Q_OK) {
        fprintf(stderr, "quantize: %s\n", fp8q_status_string(st));
        return 4;
    }
    unsigned flags = 0;
    if (fp8q_device_errors(&flags, 1) != FP8Q_OK || flags != 0) return 5;     /* also synchronizes */
    uint8_t* codes = (uint8_t*)malloc(n + 1);
    float* scales = (float*)malloc(4 * nb + 4);
    if (cudaMemcpy(codes, dc, n, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(scales, ds, 4 * nb, cudaMemcpyDeviceToHost) != cudaSuccess)
        return 3;
    FILE* g = fopen(out, "wb");
    if (!g || fwrite(codes, 1, n, g) != n || fwrite(scales, 4, nb, g) != nb) return 2;
    fclose(g);
    cudaFree(dx);
    cudaFree(dc);
    cudaFree(ds);
    free(x);
    free(codes);
    free(scales);
    printf("quantize: ok (%zu elements)\n", n);
    return 0;
}

int main(int argc, char** argv) {
    if (argc >= 2 && strcmp(argv[1], "check") == 0) return check();
    if (argc >= 5 && strcmp(argv[1], "quantize") == 0) return quantize(argv[2], argv[3], atoi(argv[4]));
    fprintf(stderr, "usage: consumer check | consumer quantize IN OUT FORMAT\n");
    return 64;
}
