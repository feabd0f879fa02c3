// Throughput probe of the tensor-core instruction the grouped GEMMs are built
// on: tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale, M = 128, N = 256,
// K = 32, e4m3 activations (A) against E2M1 weights (B) with one E8M0 scale
// per 32 values.  It measures the dense rate the prefill roofline divides by.
// The same kernel times other N and the operand order of the light m-tiles
// in the promotion modes (E2M1 weights as the 128-row A operand, N e4m3
// token rows as B): the instruction's cost in cycles for each shape.
//
// One CTA per SM (the shared-memory request leaves room for one), four
// warps: warp 1 allocates TMEM, copies the two scale chunks into it and then
// runs the issue loop the GEMMs use (the whole warp in the loop, one lane
// chosen by elect.sync issues each MMA), four MMAs per 128-wide K step over
// operands that stay resident in shared memory, the accumulator restarting
// every 32 K steps as at the start of a GEMM tile.  The operands hold
// pseudo-random valid codes (no e4m3 NaN), so the tensor pipe switches as it
// does on real data.  Thread 0 of warp 1 reads the SM cycle counter and the
// global timer around the loop, so the host learns the SM clock during the
// run.  The closing wait is bounded like every other wait of the library.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "../../include/moe_mx.h"
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kPeakABytes = 128 * 128;         // 128 rows x 128 e4m3 (one K step)
constexpr int kPeakBBytes = 256 * 128;         // 256 rows x 128 B: E2M1 in 16-byte slots
constexpr int kPeakSFOff = kPeakABytes + kPeakBBytes;
constexpr int kPeakSmem = 160 * 1024;          // more than half of an SM's shared memory: one CTA per SM

struct PeakOut {
    long long cycles;
    long long ns;
    int err;
    int pad;
};

__device__ __forceinline__ uint32_t hash32(uint32_t x)
{
    x ^= x >> 16;
    x *= 0x7FEB352Du;
    x ^= x >> 15;
    x *= 0x846CA68Bu;
    x ^= x >> 16;
    return x;
}

__global__ void __launch_bounds__(128, 1) k_mma_peak(int n_steps, int N, int tokens_on_n, PeakOut* out)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t done_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5;

    // operands: random e4m3 codes without NaN (A), random E2M1 nibbles (B);
    // scale chunks: E8M0 1.0 in every byte
    uint32_t* w = reinterpret_cast<uint32_t*>(smem);
    for (int i = threadIdx.x; i < kPeakSFOff / 4; i += blockDim.x) {
        uint32_t v = hash32(i * 2654435761u + blockIdx.x);
        if (i < kPeakABytes / 4) v &= 0xF7F7F7F7u;   // exponent field at most 1110: never 0x7F / 0xFF
        w[i] = v;
    }
    for (int i = threadIdx.x; i < (512 + 1024) / 4; i += blockDim.x) w[kPeakSFOff / 4 + i] = 0x7F7F7F7Fu;
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&done_bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 1) {
        const uint32_t s0 = smem_u32(smem);
        // activation rows (e4m3) at s0, weight rows (E2M1 in 16-byte slots) after them
        const uint64_t xd = desc_kmajor_sw128(s0), wd = desc_kmajor_sw128(s0 + kPeakABytes);
        const uint64_t ad = tokens_on_n ? wd : xd, bd = tokens_on_n ? xd : wd;
        const uint32_t sfa = tmem + 256, sfb = tmem + 264;
        tmem_cp_32x128b_warpx4_elect(sfa, desc_sf_chunk(s0 + kPeakSFOff));
        tmem_cp_32x128b_warpx4_elect(sfb, desc_sf_chunk(s0 + kPeakSFOff + 512));
        tmem_cp_32x128b_warpx4_elect(sfb + 4u, desc_sf_chunk(s0 + kPeakSFOff + 1024));
        const uint32_t id0 = tokens_on_n ? idesc_mxf8f6f4(128, (uint32_t)N, kTypeE2M1, kTypeE4M3)
                                         : idesc_mxf8f6f4(128, (uint32_t)N, kTypeE4M3, kTypeE2M1);
        const uint32_t id1 = idesc_with_sf_id(id0, 1, 1), id2 = idesc_with_sf_id(id0, 2, 2),
                       id3 = idesc_with_sf_id(id0, 3, 3);
        __syncwarp();
        long long c0 = 0, t0 = 0;
        if ((threadIdx.x & 31) == 0) {
            c0 = clock64();
            t0 = (long long)globaltimer_ns();
        }
        for (int st = 0; st < n_steps; ++st) {
            mma_mxf8f6f4_elect(tmem, ad, bd, id0, sfa, sfb, (st & 31) != 0 ? 1u : 0u);
            mma_mxf8f6f4_elect(tmem, ad + 2, bd + 2, id1, sfa, sfb, 1u);
            mma_mxf8f6f4_elect(tmem, ad + 4, bd + 4, id2, sfa, sfb, 1u);
            mma_mxf8f6f4_elect(tmem, ad + 6, bd + 6, id3, sfa, sfb, 1u);
        }
        tc_commit_elect(smem_u32(&done_bar));
        const bool ok = mbar_wait(smem_u32(&done_bar), 0u, &abort_flag);
        if ((threadIdx.x & 31) == 0) {
            PeakOut& o = out[blockIdx.x];
            o.cycles = clock64() - c0;
            o.ns = (long long)globaltimer_ns() - t0;
            o.err = ok ? 0 : 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace moe

void moe_set_handle_free_error(const char* msg);

// Runs `launches` probe launches; cycles / ns / CUDA-event ms of the last launch's CTAs.
static moe_status run_probe(const char* who, int device, int steps_per_cta, int launches, int N, int tokens_on_n,
                            double* cyc_per_sm, double* ns_per_sm, float* ms_all, int* nsm_out)
{
    char buf[256];
    auto fail = [&](moe_status st, const char* what, cudaError_t e) {
        snprintf(buf, sizeof buf, "%s: %s%s%s", who, what, e != cudaSuccess ? ": " : "",
                 e != cudaSuccess ? cudaGetErrorString(e) : "");
        moe_set_handle_free_error(buf);
        return st;
    };
    cudaError_t e = cudaSetDevice(device);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaSetDevice", e);
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, device);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaGetDeviceProperties", e);
    if (prop.major != 10 || prop.minor != 3) return fail(MOE_ERR_UNSUPPORTED, "the device is not sm_103", cudaSuccess);
    const int nsm = prop.multiProcessorCount;
    e = cudaFuncSetAttribute(moe::k_mma_peak, cudaFuncAttributeMaxDynamicSharedMemorySize, moe::kPeakSmem + 1024);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaFuncSetAttribute", e);
    moe::PeakOut* d_out = nullptr;
    e = cudaMalloc(&d_out, sizeof(moe::PeakOut) * nsm);
    if (e != cudaSuccess) return fail(MOE_ERR_OOM, "cudaMalloc", e);
    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    cudaEventCreate(&ev0);
    cudaEventCreate(&ev1);
    double cyc = 0, ns = 0;
    int errs = 0;
    float ms = 0.f;
    e = cudaEventRecord(ev0, 0);
    for (int i = 0; i < launches && e == cudaSuccess; ++i) {
        moe::k_mma_peak<<<nsm, 128, moe::kPeakSmem + 1024>>>(steps_per_cta, N, tokens_on_n, d_out);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaEventRecord(ev1, 0);
    if (e == cudaSuccess) e = cudaEventSynchronize(ev1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, ev0, ev1);
    moe::PeakOut* h_out = new moe::PeakOut[nsm];
    if (e == cudaSuccess) e = cudaMemcpy(h_out, d_out, sizeof(moe::PeakOut) * nsm, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess)
        for (int i = 0; i < nsm; ++i) {
            cyc += (double)h_out[i].cycles;
            ns += (double)h_out[i].ns;
            errs += h_out[i].err;
        }
    delete[] h_out;
    cudaFree(d_out);
    cudaEventDestroy(ev0);
    cudaEventDestroy(ev1);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "launch or readback", e);
    if (errs) return fail(MOE_ERR_TIMEOUT, "a CTA's closing wait timed out", cudaSuccess);
    *cyc_per_sm = cyc / nsm;
    *ns_per_sm = ns / nsm;
    *ms_all = ms;
    *nsm_out = nsm;
    return MOE_OK;
}

static moe_status probe_arg_error(const char* msg)
{
    moe_set_handle_free_error(msg);
    return MOE_ERR_INVALID_ARG;
}

extern "C" moe_status moe_selftest_mma_peak(int device, int steps_per_cta, int launches, float* result)
{
    if (!result) return probe_arg_error("moe_selftest_mma_peak: result is NULL");
    if (steps_per_cta < 1 || steps_per_cta > (1 << 22) || launches < 1 || launches > 100000)
        return probe_arg_error("moe_selftest_mma_peak: steps_per_cta must be in [1, 2^22] and launches in [1, 10^5]");
    double cyc = 0, ns = 0;
    float ms = 0.f;
    int nsm = 0;
    const moe_status st = run_probe("moe_selftest_mma_peak", device, steps_per_cta, launches, 256, 0, &cyc, &ns, &ms, &nsm);
    if (st != MOE_OK) return st;
    const double flop = 2.0 * 128 * 256 * 32 * 4.0 * steps_per_cta * nsm * launches;
    result[0] = (float)(flop / (ms * 1e-3) / 1e12);             // TFLOP/s over all launches (CUDA events)
    result[1] = (float)(cyc / ns * 1e3);                         // mean SM clock (MHz) of the last launch
    result[2] = (float)(cyc / (4.0 * steps_per_cta));            // SM cycles per MMA (last launch)
    result[3] = ms;
    return MOE_OK;
}

extern "C" moe_status moe_selftest_mma_shape(int device, int n, int tokens_on_n, int steps_per_cta, float* result)
{
    if (!result) return probe_arg_error("moe_selftest_mma_shape: result is NULL");
    if (steps_per_cta < 1 || steps_per_cta > (1 << 22))
        return probe_arg_error("moe_selftest_mma_shape: steps_per_cta must be in [1, 2^22]");
    if (n < 16 || n % 16 != 0 || n > (tokens_on_n ? 128 : 256) || (tokens_on_n != 0 && tokens_on_n != 1))
        return probe_arg_error("moe_selftest_mma_shape: n must be a multiple of 16 in [16, 256] (tokens_on_n = 0) "
                               "or [16, 128] (tokens_on_n = 1)");
    double cyc = 0, ns = 0;
    float ms = 0.f;
    int nsm = 0;
    const moe_status st = run_probe("moe_selftest_mma_shape", device, steps_per_cta, 1, n, tokens_on_n, &cyc, &ns, &ms, &nsm);
    if (st != MOE_OK) return st;
    result[0] = (float)(cyc / (4.0 * steps_per_cta));            // SM cycles per MMA
    result[1] = (float)(cyc / ns * 1e3);                         // mean SM clock (MHz)
    result[2] = (float)(2.0 * 128 * n * 32 * 4.0 * steps_per_cta * nsm / (ms * 1e-3) / 1e12);   // TFLOP/s
    return MOE_OK;
}
