// Router logits on the tensor cores: logits[t][e] = sum_h x[t][h] * Wr[e][h]
// + logit_bias[e], bf16 inputs (products exact), fp32 accumulation in TMEM.
//
// Router definition: "MiMo V2.6 Pro and Flash architecture teardown", section
// "How Big Is Each Expert?" (the router scores every expert of the layer) and
// section "Why Are the V2.6 Files Half the Size of V2.5?" (router weights in
// BF16).
//
// One CTA per (N-expert tile, 128-token tile), N = 64 or 128.  Warp 0 lane 0
// streams 64-wide K slices of x and Wr with TMA (128-byte swizzle) through a
// 4-stage ring; warp 1 lane 0 issues tcgen05.mma kind::f16 (128 x N x 16)
// into TMEM; then all four warps read their 32 TMEM lanes (tokens) and write
// the logits.  Waits are bounded in time as in the grouped GEMMs.
#include <cuda_runtime.h>

#include <cstdint>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kRStages = 4;
constexpr int kRABytes = 128 * 128;   // 128 tokens x 64 bf16
constexpr int kRBBytes = 128 * 128;   // up to 128 experts x 64 bf16
constexpr int kRStageStride = kRABytes + kRBBytes;
constexpr int kRBarOff = kRStages * kRStageStride;
constexpr int kRSmemBytes = kRBarOff + 256 + 1024;

struct RouterCtl {
    uint64_t full[kRStages];
    uint64_t empty[kRStages];
    uint64_t acc_full;
    uint32_t tmem_base;
    int abort;
};

// kind::f16 instruction descriptor: D f32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 and 10-12 = 1), both K-major, N>>3 at 17-22, M>>4 at 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void router_fail(RouterCtl* ctl, int32_t* err, int where)
{
    if (atomicCAS(err, 0, kDevErrTimeout) == 0) {
        err[1] = where;
        err[2] = blockIdx.x;
    }
    *(volatile int*)&ctl->abort = 1;
}

// Split-K (blockIdx.z, small batches): each CTA sums `KB` of the K-steps
// starting at z * KB and stores raw partial products to part[z][t][e]; the
// top-k kernel adds the partials in split order plus the logit bias.
__global__ void __launch_bounds__(128, 1)
    k_router_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const float* __restrict__ lb, float* __restrict__ logits, float* __restrict__ part, int T, int E,
                int KB, int N, int32_t* err)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    RouterCtl* ctl = reinterpret_cast<RouterCtl*>(smem + kRBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the expert tile is the fastest grid dimension: the CTAs that share a
    // 128-token tile of x run side by side, so x comes from HBM about once
    const int nt = blockIdx.x, mt = blockIdx.y;
    const int kb0 = blockIdx.z * KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRStages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        mbar_init(smem_u32(&ctl->acc_full), 1);
        ctl->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), (uint32_t)N);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // x (and the logit buffers) belong to the previous kernel on the stream
    // until it has completed
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t tmem = ctl->tmem_base;
    const volatile int* abrt = &ctl->abort;

    if (warp == 0 && lane == 0) {
        const uint32_t tx = (uint32_t)kRABytes + (uint32_t)N * 128u;
        int last = -1;
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % kRStages;
            const uint32_t ph = (uint32_t)(kb / kRStages) & 1u;
            if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abrt)) {
                router_fail(ctl, err, 11);
                break;
            }
            uint8_t* st = smem + s * kRStageStride;
            const uint32_t fb = smem_u32(&ctl->full[s]);
            mbar_arrive_expect_tx(fb, tx);
            tma_load_2d(smem_u32(st), &tmX, fb, (kb0 + kb) * 64, mt * 128);
            tma_load_2d(smem_u32(st + kRABytes), &tmW, fb, (kb0 + kb) * 64, nt * N);
            last = kb;
        }
        // every copy started here has landed before the CTA may exit
        int zero = 0;
        for (int kb = last - kRStages + 1; kb <= last; ++kb)
            if (kb >= 0 && !mbar_wait(smem_u32(&ctl->full[kb % kRStages]), (uint32_t)(kb / kRStages) & 1u, &zero))
                router_fail(ctl, err, 12);
    } else if (warp == 1 && lane == 0) {
        const uint32_t idesc = idesc_bf16(128, (uint32_t)N);
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % kRStages;
            const uint32_t ph = (uint32_t)(kb / kRStages) & 1u;
            if (!mbar_wait(smem_u32(&ctl->full[s]), ph, abrt)) {
                router_fail(ctl, err, 13);
                break;
            }
            tc_fence_after();
            const uint32_t st = smem_u32(smem + s * kRStageStride);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem, desc_kmajor_sw128(st + 32u * k), desc_kmajor_sw128(st + kRABytes + 32u * k), idesc,
                         (kb | k) != 0 ? 1u : 0u);
            tc_commit(smem_u32(&ctl->empty[s]));
        }
        // acc_full also serves as the drain: it completes once every MMA above has completed
        tc_commit(smem_u32(&ctl->acc_full));
    }
    __syncwarp();

    // epilogue: all four warps
    int zero = 0;
    if (mbar_wait(smem_u32(&ctl->acc_full), 0u, &zero)) {
        tc_fence_after();
        const int row = warp * 32 + lane;
        const int t = mt * 128 + row;
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        for (int c = 0; c < N / 16; ++c) {
            uint32_t v[16];
            tmem_ld16(tl + 16u * c, v);
            tmem_ld_wait();
            if (t < T && !ctl->abort) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int e = nt * N + 16 * c + j;
                    if (e < E) {
                        if (part) part[((size_t)blockIdx.z * T + t) * E + e] = __uint_as_float(v[j]);
                        else logits[(size_t)t * E + e] = __uint_as_float(v[j]) + lb[e];
                    }
                }
            }
        }
    } else {
        router_fail(ctl, err, 14);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)N);
    }
}

cudaError_t router_set_attributes()
{
    return cudaFuncSetAttribute(k_router_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmemBytes);
}

int router_tile_n(int T) { return T <= 512 ? 64 : 128; }

// Split factor for a batch of T tokens: up to kRouterMaxSplit, at least 4
// K-steps (of 64) per split, dividing the K-steps evenly; 1 for large T.
int router_split(int T, int H)
{
    if (T > kRouterSplitMaxT) return 1;
    const int KB = H / 64;
    int S = kRouterMaxSplit;
    while (S > 1 && (KB % S != 0 || KB / S < 4)) S >>= 1;
    return S;
}

cudaError_t launch_router_tc(const DevState& s, const CUtensorMap& tmX, int T, cudaStream_t st, int ksplit)
{
    const int N = router_tile_n(T);
    dim3 grid((s.E + N - 1) / N, (T + 127) / 128, ksplit);
    return launch_kernel(k_router_tc, grid, dim3(128), kRSmemBytes, st, s.pdl, tmX, N == 64 ? s.tm_wr64 : s.tm_wr128,
                         s.lb, s.logits, ksplit > 1 ? s.logit_part : nullptr, T, s.E, s.H / 64 / ksplit, N, s.err);
}

}  // namespace moe
