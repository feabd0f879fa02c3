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

#include <climits>
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

// ---------------------------------------------------------------------------
// Prefill-sized batches: the router and the top-k gate in one kernel.  One
// CTA per 128 tokens computes the logits of all E experts (E <= 512 fp32
// TMEM columns, MMAs of at most 256 columns per expert chunk) from 64-wide K
// slices of x and of every router row, so x is read once and the logits do
// not make a round trip through memory before the selection.  Then 16
// warps read the logits out of TMEM, warp (q, g) the rows of lane quarter q
// (32 tokens, one per thread) in column group g (every fourth 16-column
// chunk): logits (+ logit bias, also stored for the getters), scores
// (sigmoid, or softmax over the experts, its row maximum and sum combined
// across the groups through shared memory), keys = scores + correction
// bias, and each thread's partial top 8 under the order key descending,
// ties to the lower expert index, a NaN key ranking last (a chunk's
// candidates enter best first).  One thread per token then merges its four
// sorted partial lists by their heads (the ring's shared memory is free once
// the MMAs are done) -- the selection of the separate top-k kernel; gates =
// the selected scores / their sum, summed in selection order.
constexpr int kRTMaxStages = 4;
constexpr int kRTGroups = 4;                             // epilogue warps per TMEM lane quarter (column groups)
constexpr int kRTThreads = 32 * 4 * kRTGroups;
constexpr int kRTXBytes = 128 * 128;                     // 128 tokens x 64 bf16
// the epilogue's scratch (row maxima / sums, partial lists) reuses the ring,
// whose smallest form (E <= 128: four 32 KB stages) it must fit
static_assert(4 * (kRTGroups * 128 + 3 * 128 * kRTGroups * kMaxTopK) <= 4 * (kRTXBytes + 128 * 128),
              "router epilogue scratch");
constexpr int kRTSmemBytes = 232448;                      // the opt-in maximum; the ring takes what fits

struct RouterTopkCtl {
    uint64_t full[kRTMaxStages];
    uint64_t empty[kRTMaxStages];
    uint64_t acc_full;
    uint32_t tmem_base;
    int abort;
    float lb[kMaxExperts];
    float cb[kMaxExperts];
};

__device__ __forceinline__ void router_fail(RouterTopkCtl* ctl, int32_t* err, int where)
{
    if (atomicCAS(err, 0, kDevErrTimeout) == 0) {
        err[1] = where;
        err[2] = blockIdx.x;
    }
    *(volatile int*)&ctl->abort = 1;
}

// stage layout: the x tile, then Epad = E rounded up to 128 router rows (128-row TMA boxes)
__host__ __device__ __forceinline__ int rt_epad(int E) { return (E + 127) / 128 * 128; }
__host__ __device__ __forceinline__ int rt_stage_bytes(int E) { return kRTXBytes + rt_epad(E) * 128; }
__host__ __device__ __forceinline__ int rt_stages(int E)
{
    const int n = (kRTSmemBytes - 1024 - (int)sizeof(RouterTopkCtl)) / rt_stage_bytes(E);
    return n < kRTMaxStages ? n : kRTMaxStages;
}
__host__ __device__ __forceinline__ uint32_t rt_tmem_cols(int E16)
{
    uint32_t c = 32;
    while ((int)c < E16) c <<= 1;
    return c;
}

__device__ __forceinline__ void mma_bf16_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__global__ void __launch_bounds__(kRTThreads, 1)
    k_router_topk(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                  const float* __restrict__ lb, const float* __restrict__ cb, float* __restrict__ logits,
                  int32_t* __restrict__ ids, float* __restrict__ gates, int T, int E, int K, int KB, int score_func,
                  int32_t* err)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int nst = rt_stages(E), stride = rt_stage_bytes(E), epad = rt_epad(E);
    RouterTopkCtl* ctl = reinterpret_cast<RouterTopkCtl*>(smem + nst * stride);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = blockIdx.x;
    const int E16 = (E + 15) / 16 * 16;
    const uint32_t ncols = rt_tmem_cols(E16);
    const int n0 = E16 < 256 ? E16 : 256, n1 = E16 - n0;   // the two expert chunks' MMA widths

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        mbar_init(smem_u32(&ctl->acc_full), 1);
        ctl->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        ctl->lb[e] = lb[e];
        ctl->cb[e] = cb[e];
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // x and the routing outputs belong to the previous kernel on the stream until it has completed
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t tmem = ctl->tmem_base;
    const volatile int* abrt = &ctl->abort;

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t tx = (uint32_t)stride;
            int last = -1;
            for (int kb = 0; kb < KB; ++kb) {
                const int s = kb % nst;
                const uint32_t ph = (uint32_t)(kb / nst) & 1u;
                if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abrt)) {
                    router_fail(ctl, err, 21);
                    break;
                }
                uint8_t* st = smem + s * stride;
                const uint32_t fb = smem_u32(&ctl->full[s]);
                mbar_arrive_expect_tx(fb, tx);
                tma_load_2d(smem_u32(st), &tmX, fb, kb * 64, mt * 128);
                for (int r = 0; r < epad; r += 128) tma_load_2d(smem_u32(st + kRTXBytes + r * 128), &tmW, fb, kb * 64, r);
                last = kb;
            }
            // every copy started here has landed before the ring is read again or the CTA exits
            int zero = 0;
            for (int kb = last - nst + 1; kb <= last; ++kb)
                if (kb >= 0 && !mbar_wait(smem_u32(&ctl->full[kb % nst]), (uint32_t)(kb / nst) & 1u, &zero))
                    router_fail(ctl, err, 22);
        }
    } else if (warp == 1) {
        // the whole warp runs the loop, one elected lane issues
        const uint32_t id0 = idesc_bf16(128, (uint32_t)n0), id1 = idesc_bf16(128, (uint32_t)(n1 > 0 ? n1 : 16));
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % nst;
            const uint32_t ph = (uint32_t)(kb / nst) & 1u;
            if (!__all_sync(~0u, mbar_wait(smem_u32(&ctl->full[s]), ph, abrt))) {
                if (lane == 0) router_fail(ctl, err, 23);
                break;
            }
            tc_fence_after();
            const uint32_t st = smem_u32(smem + s * stride);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint64_t ad = desc_kmajor_sw128(st + 32u * k);
                const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
                mma_bf16_elect(tmem, ad, desc_kmajor_sw128(st + kRTXBytes + 32u * k), id0, acc);
                if (n1 > 0)
                    mma_bf16_elect(tmem + 256u, ad, desc_kmajor_sw128(st + kRTXBytes + 256u * 128u + 32u * k), id1,
                                   acc);
            }
            tc_commit_elect(smem_u32(&ctl->empty[s]));
        }
        // acc_full also serves as the drain: it completes once every MMA above has completed
        tc_commit_elect(smem_u32(&ctl->acc_full));
    }
    __syncwarp();

    // epilogue: warp (q, g) = lane quarter q, column group g; thread = token row
    int zero = 0;
    const bool acc_ok = mbar_wait(smem_u32(&ctl->acc_full), 0u, &zero);
    if (!acc_ok && lane == 0) router_fail(ctl, err, 24);
    const int q = warp & 3, g = warp >> 2;
    const int row = q * 32 + lane;
    const int t = mt * 128 + row;
    const bool live = acc_ok && t < T && !ctl->abort;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    const int nc = (E + 15) / 16;
    // the ring's shared memory, free once every MMA has completed: the groups'
    // row maxima / sums, then their partial lists
    float* red = reinterpret_cast<float*>(smem);                               // [kRTGroups][128]
    float* pk = red + kRTGroups * 128;                                          // [128][kRTGroups][kMaxTopK]
    float* ps = pk + 128 * kRTGroups * kMaxTopK;
    int* pi = reinterpret_cast<int*>(ps + 128 * kRTGroups * kMaxTopK);
    if (acc_ok) tc_fence_after();
    // softmax: the row's maximum and the sum of exp(l - max) (each group in
    // expert order, the groups added in group order)
    float m = 0.f, sum = 1.f;
    if (score_func != 0) {
        float pm = -INFINITY;
        for (int c = g; c < nc && acc_ok; c += kRTGroups) {
            uint32_t v[16];
            tmem_ld16(tl + 16u * c, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (16 * c + j < E) pm = fmaxf(pm, __uint_as_float(v[j]) + ctl->lb[16 * c + j]);
        }
        red[g * 128 + row] = pm;
        __syncthreads();
        m = red[row];
        for (int gg = 1; gg < kRTGroups; ++gg) m = fmaxf(m, red[gg * 128 + row]);
        __syncthreads();
        float psum = 0.f;
        for (int c = g; c < nc && acc_ok; c += kRTGroups) {
            uint32_t v[16];
            tmem_ld16(tl + 16u * c, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (16 * c + j < E) psum += expf(__uint_as_float(v[j]) + ctl->lb[16 * c + j] - m);
        }
        red[g * 128 + row] = psum;
        __syncthreads();
        sum = 0.f;
        for (int gg = 0; gg < kRTGroups; ++gg) sum += red[gg * 128 + row];
    }
    // the top kMaxTopK under (key descending, index ascending); a fixed length
    // keeps the list in registers, the first K entries are the top K
    float lk[kMaxTopK], ls[kMaxTopK];
    int li[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        lk[j] = -INFINITY;
        ls[j] = 0.f;
        li[j] = INT_MAX;
    }
    float thr_k = -INFINITY;   // the list's last entry: a candidate must beat it
    int thr_i = INT_MAX;
    auto insert = [&](float key, int e, float sc) {
        if (key > thr_k || (key == thr_k && e < thr_i)) {
            // carry the candidate down the sorted list: each entry it beats
            // moves one place down
            float ck = key, cs = sc;
            int ci = e;
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
                const bool b = ck > lk[j] || (ck == lk[j] && ci < li[j]);
                const float tk = b ? lk[j] : ck, ts = b ? ls[j] : cs;
                const int ti = b ? li[j] : ci;
                lk[j] = b ? ck : lk[j];
                ls[j] = b ? cs : ls[j];
                li[j] = b ? ci : li[j];
                ck = tk;
                cs = ts;
                ci = ti;
            }
            thr_k = lk[kMaxTopK - 1];
            thr_i = li[kMaxTopK - 1];
        }
    };
    if (acc_ok) {
#pragma unroll 1
        for (int c = g; c < nc; c += kRTGroups) {
            uint32_t v[16];
            tmem_ld16(tl + 16u * c, v);
            tmem_ld_wait();
            // the chunk's keys first; then its candidates that beat the list's
            // last entry go in best first, so a lane loops only as often as it
            // inserts (the lanes are different tokens: inserting element by
            // element would run the insertion for almost every element)
            float kk[16], ss[16];
            uint32_t pend = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int e = 16 * c + j;
                const float l = __uint_as_float(v[j]) + (e < E ? ctl->lb[e] : 0.f);
                if (live && e < E) logits[(size_t)t * E + e] = l;
                const float sc = score_func == 0 ? 1.0f / (1.0f + expf(-l)) : expf(l - m) / sum;
                const float kv = sc + (e < E ? ctl->cb[e] : 0.f);
                kk[j] = isnan(kv) ? -INFINITY : kv;
                ss[j] = sc;
                pend |= (e < E ? 1u : 0u) << j;
            }
            while (pend) {
                // the best pending candidate (key descending, index ascending)
                float ck = -INFINITY, cs = 0.f;
                int cj = -1;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (((pend >> j) & 1u) && (cj < 0 || kk[j] > ck)) {
                        ck = kk[j];
                        cs = ss[j];
                        cj = j;
                    }
                const int ce = 16 * c + cj;
                if (!(ck > thr_k || (ck == thr_k && ce < thr_i))) break;   // nothing left beats the list
                pend &= ~(1u << cj);
                insert(ck, ce, cs);
            }
        }
    }
    __syncthreads();   // every group has read its maxima / sums
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        const int o = (row * kRTGroups + g) * kMaxTopK + j;
        pk[o] = lk[j];
        ps[o] = ls[j];
        pi[o] = li[j];
    }
    __syncthreads();
    if (g == 0) {
        // merge the four partial lists of this thread's token: each is sorted
        // under the same order and they hold distinct experts, so the list
        // takes the best of the four heads kMaxTopK times
        int hd[kRTGroups];
#pragma unroll
        for (int gg = 0; gg < kRTGroups; ++gg) hd[gg] = 0;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            float bk = -INFINITY, bs = 0.f;
            int bi = INT_MAX, bg = 0;
#pragma unroll
            for (int gg = 0; gg < kRTGroups; ++gg) {
                if (hd[gg] < kMaxTopK) {
                    const int o = (row * kRTGroups + gg) * kMaxTopK + hd[gg];
                    const float k2 = pk[o];
                    const int i2 = pi[o];
                    if (k2 > bk || (k2 == bk && i2 < bi)) {
                        bk = k2;
                        bi = i2;
                        bs = ps[o];
                        bg = gg;
                    }
                }
            }
#pragma unroll
            for (int gg = 0; gg < kRTGroups; ++gg) hd[gg] += gg == bg ? 1 : 0;
            lk[j] = bk;
            ls[j] = bs;
            li[j] = bi;
        }
        if (live) {
            float ssum = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j)
                if (j < K) ssum += ls[j];
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j)
                if (j < K) {
                    ids[(size_t)t * K + j] = li[j];
                    gates[(size_t)t * K + j] = ls[j] / ssum;
                }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

cudaError_t router_set_attributes()
{
    cudaError_t e = cudaFuncSetAttribute(k_router_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_router_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, kRTSmemBytes);
    return e;
}

bool router_fused(int T, int E) { return T >= kRouterFusedMinT && E <= kMaxExperts; }

cudaError_t launch_router_topk(const DevState& s, const CUtensorMap& tmX, int T, cudaStream_t st)
{
    const int smem = rt_stages(s.E) * rt_stage_bytes(s.E) + (int)sizeof(RouterTopkCtl) + 1024;
    return launch_kernel(k_router_topk, dim3((T + 127) / 128), dim3(kRTThreads), smem, st, s.pdl, tmX, s.tm_wr128, s.lb,
                         s.cb, s.logits, s.ids, s.gates, T, s.E, s.K, s.H / 64, s.score_func, s.err);
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
