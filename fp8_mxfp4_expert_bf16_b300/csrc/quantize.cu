// MXFP4 quantisation of fp32 weight rows on the GPU (OCP Microscaling v1.0
// rule): the expert format of "MiMo V2.6 Pro and Flash architecture
// teardown", section "Why Are the V2.6 Files Half the Size of V2.5?" (two
// 4-bit values per byte, one 8-bit scale per 32 values).  The same page
// notes that the experts were rounded to MXFP4 after every RL update; this
// kernel is that rounding step, producing exactly the input format of
// moe_load_weights.
//
// Per 32 consecutive values of a row: shared exponent X = floor(log2(amax))
// - 2 (2 = the largest E2M1 exponent), clamped to [-127, 127], stored as the
// E8M0 byte X + 127 (an all-zero block stores 127 and zero codes); each
// value's code is the E2M1 value of v / 2^X nearest to it, ties to the even
// code, saturating at 6.  Two codes per byte, first value in the low nibble.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe_mx.h"

namespace moe {

// E2M1 code of a value already divided by its block scale: the number of
// decision points (midpoints .25 .75 1.25 1.75 2.5 3.5 5 between the
// magnitudes 0 .5 1 1.5 2 3 4 6) it lies beyond; a value on a midpoint
// rounds to the even code.
__device__ __forceinline__ uint32_t e2m1_code(float v)
{
    const float a = fabsf(v);
    const uint32_t c = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
                       (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) + (uint32_t)(a > 5.0f);
    return (signbit(v) ? 8u : 0u) | c;
}

// One thread per 32-value block.
__global__ void k_mxfp4_quantize(const float* __restrict__ w, size_t nblocks, uint8_t* __restrict__ packed,
                                 uint8_t* __restrict__ scales)
{
    for (size_t b = blockIdx.x * (size_t)blockDim.x + threadIdx.x; b < nblocks; b += (size_t)gridDim.x * blockDim.x) {
        const float4* src = reinterpret_cast<const float4*>(w + b * 32);
        float v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 f = src[i];
            v[4 * i] = f.x, v[4 * i + 1] = f.y, v[4 * i + 2] = f.z, v[4 * i + 3] = f.w;
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
        int X = 0;
        if (amax > 0.f) {
            int p;
            frexpf(amax, &p);                 // amax = m * 2^p, m in [0.5, 1): floor(log2 amax) = p - 1
            X = max(-127, min(127, p - 3));
        }
        scales[b] = (uint8_t)(X + 127);
        // 2^-X is a normal fp32 number for every X an fp32 amax can produce,
        // and multiplying by it is exact for the magnitudes that matter
        const float inv = __int_as_float((127 - X) << 23);
        uint32_t word[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t acc = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t code = amax > 0.f ? e2m1_code(v[8 * q + i] * inv) : 0u;
                acc |= code << (4 * i);
            }
            word[q] = acc;
        }
        reinterpret_cast<uint4*>(packed)[b] = make_uint4(word[0], word[1], word[2], word[3]);
    }
}

}  // namespace moe

// defined in api.cu: the message moe_last_error(NULL) returns
void moe_set_handle_free_error(const char* msg);

extern "C" moe_status moe_mxfp4_quantize(const float* w, size_t rows, int K, uint8_t* packed, uint8_t* scales,
                                         void* stream)
{
    if (K <= 0 || K % 32 != 0) {
        moe_set_handle_free_error("moe_mxfp4_quantize: K must be a positive multiple of 32");
        return MOE_ERR_SHAPE;
    }
    if (rows == 0) return MOE_OK;
    if (!w || !packed || !scales) {
        moe_set_handle_free_error("moe_mxfp4_quantize: NULL pointer");
        return MOE_ERR_INVALID_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(packed)) & 15u) {
        moe_set_handle_free_error("moe_mxfp4_quantize: w and packed must be 16-byte aligned");
        return MOE_ERR_INVALID_ARG;
    }
    const size_t nblocks = rows * (size_t)(K / 32);
    size_t grid = (nblocks + 255) / 256;
    if (grid > 65535 * 16) grid = 65535 * 16;
    moe::k_mxfp4_quantize<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(w, nblocks, packed, scales);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        moe_set_handle_free_error(cudaGetErrorString(e));
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}
