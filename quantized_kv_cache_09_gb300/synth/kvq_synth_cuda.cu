/*
 * kvq_synth_cuda.cu -- device build of the seeded synthetic-input generator
 * (definitions in kvq_synth.h).  Produces the same bits as kvq_synth_host.c
 * for every element, so full-size workloads can be generated in HBM while the
 * oracle regenerates any slice of them on the host.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_synth.h"

__global__ void kvq_synth_fill_f16_kernel(uint16_t *__restrict__ out, int64_t n, uint64_t key,
                                          int64_t index0, float sigma,
                                          const uint8_t *__restrict__ mask, int64_t period,
                                          float outlier_mult)
{
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        int64_t g = index0 + i;
        float mult = (mask && mask[g % period]) ? outlier_mult : 1.0f;
        out[i] = kvq_synth_normal_f16(key, (uint64_t)g, sigma, mult);
    }
}

extern "C" int kvq_synth_fill_f16_cuda(uint16_t *out, int64_t n, uint64_t seed, uint64_t stream,
                                       int64_t index0, float sigma, const uint8_t *mask,
                                       int64_t period, float outlier_mult, cudaStream_t s)
{
    if (n <= 0) return 0;
    if (!out || (mask && period <= 0)) return 1;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (n + 255) / 256;
    int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 16;
    if (blocks > cap) blocks = cap;
    kvq_synth_fill_f16_kernel<<<(unsigned)blocks, 256, 0, s>>>(out, n, kvq_synth_key(seed, stream),
                                                               index0, sigma, mask, period, outlier_mult);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
