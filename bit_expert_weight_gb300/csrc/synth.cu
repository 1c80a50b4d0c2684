// synth.cu -- on-device twin of the benchmark's seeded input generator
// (bit_expert_weight_gb300/synth.py): counter-based SplitMix64 (Steele, Lea
// & Flood, OOPSLA 2014; Stafford "Mix13" finaliser), twelve 16-bit uniforms
// summed into an Irwin-Hall(12) normal that is exact in fp32, one fp32
// multiply by the scale, optional outlier / zero marks, bf16 round to nearest
// even.  It holds none of the MoE method's arithmetic; the host twin regenerates
// any slice bit for bit (a test checks the two agree).
#include <stdint.h>

#include <cuda_runtime.h>

#include "smoe_synth.h"

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__global__ void synth_kernel(uint16_t *out, int64_t n, int64_t start, uint64_t key, float s_norm,
                             float s_out, uint32_t t_out, uint64_t t_out_full, uint32_t t_zero,
                             uint64_t t_zero_full)
{
    const uint64_t gamma = 0x9E3779B97F4A7C15ull;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t e = static_cast<uint64_t>(start + i);
        int64_t acc = 0;
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            const uint64_t wv = mix64(key + (4 * e + q + 1) * gamma);
#pragma unroll
            for (int h = 0; h < 4; ++h)
                acc += static_cast<int64_t>((wv >> (16 * h)) & 0xFFFFull);
        }
        const uint64_t fl = mix64(key + (4 * e + 3 + 1) * gamma);
        const int64_t C = 2 * acc - 12 * 65535;
        const float z = __fmul_rn(static_cast<float>(C), 7.62939453125e-06f);  // 2^-17
        const bool is_out = t_out_full ? true : (fl & 0xFFFFFFFFull) < t_out;
        const bool is_zero = t_zero_full ? true : (fl >> 32) < t_zero;
        float v = __fmul_rn(z, is_out ? s_out : s_norm);
        if (is_zero)
            v = 0.0f;
        const uint32_t u = __float_as_uint(v);
        out[i] = static_cast<uint16_t>((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
    }
}

}  // namespace

extern "C" int smoe_synth_bf16(uint16_t *out, int64_t n, int64_t start, uint64_t key, float s_norm,
                               float s_out, uint64_t t_out, uint64_t t_zero, void *cuda_stream)
{
    if (n < 0 || start < 0 || (n > 0 && !out))
        return -1;
    if (n == 0)
        return 0;
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (n + 255) / 256;
    if (blocks > (int64_t)sms * 32)
        blocks = (int64_t)sms * 32;
    synth_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
        out, n, start, key, s_norm, s_out, static_cast<uint32_t>(t_out > 0xFFFFFFFFull ? 0 : t_out),
        t_out > 0xFFFFFFFFull ? 1ull : 0ull,
        static_cast<uint32_t>(t_zero > 0xFFFFFFFFull ? 0 : t_zero),
        t_zero > 0xFFFFFFFFull ? 1ull : 0ull);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
