// Router, top-k gate, token->expert dispatch with activation quantisation,
// gate-weighted combine, and the small load-time / debug kernels.
//
// The layer follows the web pages on MiMo-V2.6: "MiMo V2.6 Pro and Flash
// architecture teardown", section "How Big Is Each Expert?" (sigmoid router
// with a per-expert correction bias, 8 experts per token) and section "Why
// Are the V2.6 Files Half the Size of V2.5?" (bf16 router); vLLM recipe
// "XiaomiMiMo/MiMo-V2.6-Pro-RL", "Overview" (block-wise e4m3 compute).
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cstdint>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------------ top-k
// Router logits of token t for this lane's experts (e = lane + 32 i): either
// the finished logits, or the sum of the split-K partial products in split
// order plus the logit bias (then also stored as the token's logits).
constexpr int kMaxV = kMaxExperts / 32;

__device__ __forceinline__ void token_logits(const float* __restrict__ logits, const float* __restrict__ part,
                                             int ksplit, const float* __restrict__ lb, float* __restrict__ logits_out,
                                             int t, int T, int E, int lane, float (&l)[kMaxV])
{
#pragma unroll
    for (int i = 0; i < kMaxV; ++i) {
        const int e = lane + 32 * i;
        if (e >= E) {
            l[i] = -INFINITY;
        } else if (ksplit > 1) {
            // all partial loads are issued before the (ordered) additions
            float p[kRouterMaxSplit];
#pragma unroll
            for (int z = 0; z < kRouterMaxSplit; ++z) p[z] = z < ksplit ? part[((size_t)z * T + t) * E + e] : 0.f;
            float v = 0.f;
#pragma unroll
            for (int z = 0; z < kRouterMaxSplit; ++z) v += p[z];
            v += lb[e];
            logits_out[(size_t)t * E + e] = v;
            l[i] = v;
        } else {
            l[i] = logits[(size_t)t * E + e];
        }
    }
}

// Scores s = sigmoid(l) (or softmax over experts), keys = s + correction
// bias; k rounds of a warp arg-max over (key desc, index asc); gates =
// selected scores / their sum (summed in selection order).  Lane j < k ends
// with slot j's expert and gate.
__device__ __forceinline__ void warp_topk(float (&sc)[kMaxV], const float* __restrict__ cb, int E, int K,
                                          int score_func, int lane, int& my_id, float& my_gate)
{
    float key[kMaxV];
    if (score_func == 0) {
#pragma unroll
        for (int i = 0; i < kMaxV; ++i) sc[i] = 1.0f / (1.0f + expf(-sc[i]));
    } else {
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < kMaxV; ++i) m = fmaxf(m, sc[i]);
        m = warp_max(m);
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxV; ++i) {
            sc[i] = (lane + 32 * i < E) ? expf(sc[i] - m) : 0.f;
            sum += sc[i];
        }
        sum = warp_sum(sum);
#pragma unroll
        for (int i = 0; i < kMaxV; ++i) sc[i] = sc[i] / sum;
    }
#pragma unroll
    for (int i = 0; i < kMaxV; ++i) {
        const int e = lane + 32 * i;
        const float kv = (e < E) ? sc[i] + cb[e] : -INFINITY;
        key[i] = isnan(kv) ? -INFINITY : kv;   // a NaN score ranks last, so every slot gets a valid expert
    }
    uint32_t taken = 0;
    float my_s = 0.f, ssum = 0.f;
    my_id = 0;
    for (int j = 0; j < K; ++j) {
        float bk = -INFINITY, bs = 0.f;
        int be = INT_MAX;
#pragma unroll
        for (int i = 0; i < kMaxV; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && (key[i] > bk || (key[i] == bk && e < be))) {
                bk = key[i];
                be = e;
                bs = sc[i];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            const float os = __shfl_xor_sync(0xffffffffu, bs, o);
            if (ok > bk || (ok == bk && oe < be)) {
                bk = ok;
                be = oe;
                bs = os;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == j) {
            my_id = be;
            my_s = bs;
        }
        ssum += bs;
    }
    my_gate = my_s / ssum;
}

// One warp per token.
__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ logits, const float* __restrict__ part,
                                              int ksplit, const float* __restrict__ lb, float* __restrict__ logits_out,
                                              const float* __restrict__ cb, int32_t* __restrict__ ids,
                                              float* __restrict__ gates, int T, int E, int K, int score_func)
{
    griddep_wait();
    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    float sc[kMaxV];
    token_logits(logits, part, ksplit, lb, logits_out, t, T, E, lane, sc);
    int id;
    float g;
    warp_topk(sc, cb, E, K, score_func, lane, id, g);
    if (lane < K) {
        ids[(size_t)t * K + lane] = id;
        gates[(size_t)t * K + lane] = g;
    }
}

// Small batches (split-K router): one block per token.  Each thread adds the
// split partials of up to kMaxExperts / kTopkSplitThreads experts in split
// order, then the logit bias, and stores the token's logits; warp 0 then
// selects from the logits in shared memory.  All partial loads of a thread
// are issued before its additions.
constexpr int kTopkSplitThreads = 128;
constexpr int kTopkSplitPer = kMaxExperts / kTopkSplitThreads;

__global__ void __launch_bounds__(kTopkSplitThreads) k_topk_split(const float* __restrict__ part, int ksplit,
                                                                  const float* __restrict__ lb,
                                                                  float* __restrict__ logits_out,
                                                                  const float* __restrict__ cb, int32_t* __restrict__ ids,
                                                                  float* __restrict__ gates, int T, int E, int K,
                                                                  int score_func)
{
    griddep_wait();
    griddep_launch_dependents();
    __shared__ float l_s[kMaxExperts];
    const int t = blockIdx.x;
    float p[kTopkSplitPer][kRouterMaxSplit];
#pragma unroll
    for (int i = 0; i < kTopkSplitPer; ++i) {
        const int e = threadIdx.x + kTopkSplitThreads * i;
#pragma unroll
        for (int z = 0; z < kRouterMaxSplit; ++z)
            p[i][z] = (e < E && z < ksplit) ? part[((size_t)z * T + t) * E + e] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kTopkSplitPer; ++i) {
        const int e = threadIdx.x + kTopkSplitThreads * i;
        if (e < E) {
            float v = 0.f;
#pragma unroll
            for (int z = 0; z < kRouterMaxSplit; ++z) v += p[i][z];
            v += lb[e];
            logits_out[(size_t)t * E + e] = v;
            l_s[e] = v;
        }
    }
    __syncthreads();
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    float sc[kMaxV];
#pragma unroll
    for (int i = 0; i < kMaxV; ++i) {
        const int e = lane + 32 * i;
        sc[i] = e < E ? l_s[e] : -INFINITY;
    }
    int id;
    float g;
    warp_topk(sc, cb, E, K, score_func, lane, id, g);
    if (lane < K) {
        ids[(size_t)t * K + lane] = id;
        gates[(size_t)t * K + lane] = g;
    }
}

cudaError_t launch_topk(const DevState& s, int T, cudaStream_t st, int ksplit)
{
    if (ksplit > 1)
        return launch_kernel(k_topk_split, dim3(T), dim3(kTopkSplitThreads), 0, st, s.pdl, (const float*)s.logit_part,
                             ksplit, s.lb, s.logits, s.cb, s.ids, s.gates, T, s.E, s.K, s.score_func);
    return launch_kernel(k_topk, dim3((T + 7) / 8), dim3(256), 0, st, s.pdl, (const float*)s.logits,
                         (const float*)s.logit_part, ksplit, s.lb, s.logits, s.cb, s.ids, s.gates, T, s.E, s.K,
                         s.score_func);
}

// ------------------------------------------------------------------ dispatch
// (1) per 256-token chunk, the expert histogram of its (token, slot) pairs.
__global__ void __launch_bounds__(kChunk) k_chunk_hist(const int32_t* __restrict__ ids, int32_t* __restrict__ chunk_hist,
                                                       int T, int E, int K, int32_t* err)
{
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int hist[kMaxExperts];
    for (int e = threadIdx.x; e < E; e += kChunk) hist[e] = 0;
    __syncthreads();
    const int t = blockIdx.x * kChunk + threadIdx.x;
    if (t < T) {
        for (int j = 0; j < K; ++j) {
            int e = ids[(size_t)t * K + j];
            if (e < 0 || e >= E) {   // cannot happen for ids from k_topk; keep every index in bounds anyway
                atomicCAS(err, 0, kDevErrBounds);
                e = min(max(e, 0), E - 1);
            }
            atomicAdd(&hist[e], 1);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kChunk) chunk_hist[(size_t)blockIdx.x * E + e] = hist[e];
}

template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < NT / 32) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        if (lane < NT / 32) warp_tot[lane] = w;
    }
    __syncthreads();
    const int base = (warp > 0) ? warp_tot[warp - 1] : 0;
    __syncthreads();
    return base + inc - v;
}

// (2) one block: per-expert running sums over chunks (chunk base offsets),
// expert counts, exclusive scans (offsets, m-tile offsets) and the m-tile
// lists: every 128-row m-tile with its expert and valid rows, and the split
// into light m-tiles (at most kLightRows valid rows: only an expert's last
// m-tile can be one) and heavy m-tiles, each list in m-tile order.
__global__ void __launch_bounds__(kMaxExperts) k_scan(const int32_t* __restrict__ chunk_hist,
                                                      int32_t* __restrict__ chunk_base, int32_t* __restrict__ counts,
                                                      int32_t* __restrict__ offsets, int32_t* __restrict__ mtile_off,
                                                      int32_t* __restrict__ mtile_expert,
                                                      int32_t* __restrict__ mtile_rows, int32_t* __restrict__ n_mtiles,
                                                      int32_t* __restrict__ light_list,
                                                      int32_t* __restrict__ heavy_list, int nchunk, int E,
                                                      int light_rows)
{
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int warp_tot[32];
    const int e = threadIdx.x;
    int run = 0;
    if (e < E) {
        for (int c = 0; c < nchunk; ++c) {
            const int v = chunk_hist[(size_t)c * E + e];
            chunk_base[(size_t)c * E + e] = run;
            run += v;
        }
        counts[e] = run;
    }
    const int mt = (run + kBM - 1) / kBM;
    const int rem = run - (mt - 1) * kBM;                 // rows of the last m-tile
    const int light = (mt > 0 && rem <= light_rows) ? 1 : 0;
    const int heavy = mt - light;
    const int ex_cnt = block_exclusive_scan<kMaxExperts>(run, warp_tot);
    const int ex_mt = block_exclusive_scan<kMaxExperts>(mt, warp_tot);
    const int ex_light = block_exclusive_scan<kMaxExperts>(light, warp_tot);
    const int ex_heavy = block_exclusive_scan<kMaxExperts>(heavy, warp_tot);
    if (e < E) {
        offsets[e] = ex_cnt;
        mtile_off[e] = ex_mt;
        for (int m = 0; m < mt; ++m) {
            mtile_expert[ex_mt + m] = e;
            mtile_rows[ex_mt + m] = min(kBM, run - kBM * m);
        }
        for (int m = 0; m < heavy; ++m) heavy_list[ex_heavy + m] = ex_mt + m;
        if (light) light_list[ex_light] = ex_mt + mt - 1;
        if (e == E - 1) {
            offsets[E] = ex_cnt + run;
            mtile_off[E] = ex_mt + mt;
            n_mtiles[0] = ex_mt + mt;
            n_mtiles[1] = ex_light + light;
            n_mtiles[2] = ex_heavy + heavy;
        }
    }
}

// (3) per chunk: stable rank of every (token, slot) among the chunk's tokens
// routed to the same expert (popcount of a per-expert token bitmask); its
// padded row = 128 * mtile_off[e] + chunk base + rank.
__global__ void __launch_bounds__(kChunk) k_scatter_rows(const int32_t* __restrict__ ids,
                                                         const int32_t* __restrict__ chunk_base,
                                                         const int32_t* __restrict__ mtile_off,
                                                         int32_t* __restrict__ prow, int T, int E, int K)
{
    griddep_wait();
    griddep_launch_dependents();
    __shared__ uint32_t mask[kMaxExperts][kChunk / 32];
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = tid; i < E * (kChunk / 32); i += kChunk) (&mask[0][0])[i] = 0u;
    __syncthreads();
    const int t = blockIdx.x * kChunk + tid;
    if (t < T)
        for (int j = 0; j < K; ++j) atomicOr(&mask[min(max(ids[(size_t)t * K + j], 0), E - 1)][tid >> 5], 1u << lane);
    __syncthreads();
    if (t < T) {
        for (int j = 0; j < K; ++j) {
            const int e = min(max(ids[(size_t)t * K + j], 0), E - 1);
            int rank = __popc(mask[e][tid >> 5] & ((1u << lane) - 1u));
            for (int w = 0; w < (tid >> 5); ++w) rank += __popc(mask[e][w]);
            prow[(size_t)t * K + j] = mtile_off[e] * kBM + chunk_base[(size_t)blockIdx.x * E + e] + rank;
        }
    }
}

// (4) 1 x 128 e4m3 quantisation of every token's activations, written to all
// k of its rows.  One warp per (token, 128-wide block).
//
// Quantisation of one block of 128 values: amax; the smallest integer e with
// amax <= 448 * 2^e (from amax = f * 2^p, f in [0.5,1): e = p-9 if f <= 0.875
// else p-8), clamped to [-127, 127], zero block -> 0; codes e4m3(v * 2^-e)
// with round-to-nearest-even and saturation; the scale byte e + 127.
__device__ __forceinline__ int act_block_exponent(float amax)
{
    if (!(amax > 0.f)) return 0;
    int p;
    const float f = frexpf(amax, &p);
    int e = (f <= 0.875f) ? p - 9 : p - 8;
    return max(-127, min(127, e));
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d)
{
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

__device__ __forceinline__ float pow2_neg(int e) { return __int_as_float((127 - e) << 23); }

// One warp per token and group of kQBlocks 1 x 128 blocks: the token's k
// destination rows are read once, the group's loads are all in flight before
// the first block is quantised, and each block's codes go to every
// destination row (each store fills 128 contiguous bytes).
constexpr int kQBlocks = 4;

__global__ void __launch_bounds__(256) k_quant_scatter(const uint16_t* __restrict__ x, const int32_t* __restrict__ prow,
                                                       uint8_t* __restrict__ aq, uint32_t* __restrict__ asf, int T,
                                                       int H, int K)
{
    griddep_wait();
    griddep_launch_dependents();
    const int KB = H / 128, NG = (KB + kQBlocks - 1) / kQBlocks, lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (gw >= (long long)T * NG) return;
    const int t = (int)(gw / NG), b0 = (int)(gw - (long long)t * NG) * kQBlocks;
    const int my_row = lane < K ? prow[(size_t)t * K + lane] : 0;
    uint2 v[kQBlocks];
#pragma unroll
    for (int i = 0; i < kQBlocks; ++i)
        if (b0 + i < KB) v[i] = *reinterpret_cast<const uint2*>(x + (size_t)t * H + (b0 + i) * 128 + lane * 4);
    int rows[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) rows[j] = __shfl_sync(0xffffffffu, my_row, j);
#pragma unroll
    for (int i = 0; i < kQBlocks; ++i) {
        const int b = b0 + i;
        if (b >= KB) break;
        const float f0 = bf16_lo(v[i].x), f1 = bf16_hi(v[i].x), f2 = bf16_lo(v[i].y), f3 = bf16_hi(v[i].y);
        const float amax = warp_max(fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3))));
        const int ex = act_block_exponent(amax);
        const float inv = pow2_neg(ex);
        const uint32_t word = e4m3x4(f0 * inv, f1 * inv, f2 * inv, f3 * inv);
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
            if (j < K) *reinterpret_cast<uint32_t*>(aq + (size_t)rows[j] * H + b * 128 + lane * 4) = word;
        if (lane < K) asf[sf_word_index(my_row >> 7, b, KB, my_row & 127)] = (uint32_t)(ex + 127) * 0x01010101u;
    }
}

// The fp32-scale variant: s = amax / 448 and codes e4m3(v / s), both fp32
// divisions rounded to nearest (an all-zero block: s = 0, zero codes); s goes
// to the fp32 scale table of every destination row.
__global__ void __launch_bounds__(256) k_quant_scatter_f32s(const uint16_t* __restrict__ x,
                                                            const int32_t* __restrict__ prow, uint8_t* __restrict__ aq,
                                                            float* __restrict__ asf32, int T, int H, int K)
{
    griddep_wait();
    griddep_launch_dependents();
    const int KB = H / 128, NG = (KB + kQBlocks - 1) / kQBlocks, lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (gw >= (long long)T * NG) return;
    const int t = (int)(gw / NG), b0 = (int)(gw - (long long)t * NG) * kQBlocks;
    const int my_row = lane < K ? prow[(size_t)t * K + lane] : 0;
    uint2 v[kQBlocks];
#pragma unroll
    for (int i = 0; i < kQBlocks; ++i)
        if (b0 + i < KB) v[i] = *reinterpret_cast<const uint2*>(x + (size_t)t * H + (b0 + i) * 128 + lane * 4);
    int rows[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) rows[j] = __shfl_sync(0xffffffffu, my_row, j);
#pragma unroll
    for (int i = 0; i < kQBlocks; ++i) {
        const int b = b0 + i;
        if (b >= KB) break;
        const float f0 = bf16_lo(v[i].x), f1 = bf16_hi(v[i].x), f2 = bf16_lo(v[i].y), f3 = bf16_hi(v[i].y);
        const float amax = warp_max(fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3))));
        const float sc = __fdiv_rn(amax, 448.0f);
        const uint32_t word = amax > 0.0f ? e4m3x4(__fdiv_rn(f0, sc), __fdiv_rn(f1, sc), __fdiv_rn(f2, sc),
                                                   __fdiv_rn(f3, sc))
                                          : 0u;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
            if (j < K) *reinterpret_cast<uint32_t*>(aq + (size_t)rows[j] * H + b * 128 + lane * 4) = word;
        if (lane < K) asf32[(size_t)my_row * KB + b] = sc;
    }
}

// Small batches (T <= 256, one dispatch chunk): one block builds the expert
// histogram and token bit-masks, the scan and m-tile lists, and the stable
// ranks - the work of k_chunk_hist, k_scan and k_scatter_rows in a single
// launch.
constexpr int kSmallT = kChunk;

__global__ void __launch_bounds__(kMaxExperts) k_dispatch_small(
    const int32_t* __restrict__ ids, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ mtile_off, int32_t* __restrict__ mtile_expert, int32_t* __restrict__ mtile_rows,
    int32_t* __restrict__ n_mtiles, int32_t* __restrict__ light_list, int32_t* __restrict__ heavy_list,
    int32_t* __restrict__ prow, int T, int E, int K, int light_rows)
{
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int hist[kMaxExperts];
    __shared__ int mt_off_s[kMaxExperts];
    __shared__ uint32_t mask[kMaxExperts][kSmallT / 32];
    __shared__ int warp_tot[32];
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = tid; i < kMaxExperts; i += blockDim.x) hist[i] = 0;
    for (int i = tid; i < kMaxExperts * (kSmallT / 32); i += blockDim.x) (&mask[0][0])[i] = 0u;
    __syncthreads();
    int my_ids[kMaxTopK];
    if (tid < T) {
        for (int j = 0; j < K; ++j) {
            const int ex = min(max(ids[(size_t)tid * K + j], 0), E - 1);
            my_ids[j] = ex;
            atomicAdd(&hist[ex], 1);
            atomicOr(&mask[ex][tid >> 5], 1u << lane);
        }
    }
    __syncthreads();
    // counts, scans, m-tile lists (thread = expert)
    const int e = tid;
    const int run = e < E ? hist[e] : 0;
    const int mt = (run + kBM - 1) / kBM;
    const int rem = run - (mt - 1) * kBM;
    const int light = (mt > 0 && rem <= light_rows) ? 1 : 0;
    const int heavy = mt - light;
    const int ex_cnt = block_exclusive_scan<kMaxExperts>(run, warp_tot);
    const int ex_mt = block_exclusive_scan<kMaxExperts>(mt, warp_tot);
    const int ex_light = block_exclusive_scan<kMaxExperts>(light, warp_tot);
    const int ex_heavy = block_exclusive_scan<kMaxExperts>(heavy, warp_tot);
    if (e < E) {
        counts[e] = run;
        offsets[e] = ex_cnt;
        mtile_off[e] = ex_mt;
        mt_off_s[e] = ex_mt;
        for (int m = 0; m < mt; ++m) {
            mtile_expert[ex_mt + m] = e;
            mtile_rows[ex_mt + m] = min(kBM, run - kBM * m);
        }
        for (int m = 0; m < heavy; ++m) heavy_list[ex_heavy + m] = ex_mt + m;
        if (light) light_list[ex_light] = ex_mt + mt - 1;
        if (e == E - 1) {
            offsets[E] = ex_cnt + run;
            mtile_off[E] = ex_mt + mt;
            n_mtiles[0] = ex_mt + mt;
            n_mtiles[1] = ex_light + light;
            n_mtiles[2] = ex_heavy + heavy;
        }
    }
    __syncthreads();
    // stable ranks (thread = token)
    if (tid < T) {
        for (int j = 0; j < K; ++j) {
            const int ex = my_ids[j];
            int rank = __popc(mask[ex][tid >> 5] & ((1u << lane) - 1u));
            for (int w = 0; w < (tid >> 5); ++w) rank += __popc(mask[ex][w]);
            prow[(size_t)tid * K + j] = mt_off_s[ex] * kBM + rank;
        }
    }
}

// m-tiles with at most kLightRows valid rows run in the GEMMs' light phase at
// every batch size: with the tokens on the MMA's N side they cost a fraction
// of a full 128-row tile's multiply-adds (with skewed routing many experts'
// last m-tiles hold a few rows: Pro prefill 2.5% faster, at higher clocks
// under the power cap; Flash prefill unchanged).

cudaError_t launch_dispatch_small(const DevState& s, int T, cudaStream_t st)
{
    return launch_kernel(k_dispatch_small, dim3(1), dim3(kMaxExperts), 0, st, s.pdl, (const int32_t*)s.ids, s.counts,
                         s.offsets, s.mtile_off, s.mtile_expert, s.mtile_rows, s.n_mtiles, s.light_list, s.heavy_list,
                         s.prow, T, s.E, s.K, kLightRows);
}

cudaError_t launch_quant_scatter(const DevState& s, const uint16_t* x, int T, cudaStream_t st)
{
    const long long warps = (long long)T * ((s.H / 128 + kQBlocks - 1) / kQBlocks);
    if (s.act_f32)
        return launch_kernel(k_quant_scatter_f32s, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, st, s.pdl, x,
                             (const int32_t*)s.prow, s.aq, s.asf32, T, s.H, s.K);
    return launch_kernel(k_quant_scatter, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, st, s.pdl, x,
                         (const int32_t*)s.prow, s.aq, s.asf, T, s.H, s.K);
}

cudaError_t launch_dispatch(const DevState& s, const uint16_t* x, int T, cudaStream_t st, int* nlaunch)
{
    const int nchunk = (T + kChunk - 1) / kChunk;
    cudaError_t e = launch_kernel(k_chunk_hist, dim3(nchunk), dim3(kChunk), 0, st, s.pdl, (const int32_t*)s.ids,
                                  s.chunk_hist, T, s.E, s.K, s.err);
    if (e == cudaSuccess)
        e = launch_kernel(k_scan, dim3(1), dim3(kMaxExperts), 0, st, s.pdl, (const int32_t*)s.chunk_hist, s.chunk_base,
                          s.counts, s.offsets, s.mtile_off, s.mtile_expert, s.mtile_rows, s.n_mtiles, s.light_list,
                          s.heavy_list, nchunk, s.E, kLightRows);
    if (e == cudaSuccess)
        e = launch_kernel(k_scatter_rows, dim3(nchunk), dim3(kChunk), 0, st, s.pdl, (const int32_t*)s.ids,
                          (const int32_t*)s.chunk_base, (const int32_t*)s.mtile_off, s.prow, T, s.E, s.K);
    if (e == cudaSuccess) e = launch_quant_scatter(s, x, T, st);
    *nlaunch += 4;
    return e;
}

// ------------------------------------------------------------------ combine
// y[t] = bf16_rne( sum_j gate[t][j] * o[row(t, j)] ), fp32 fused multiply-adds
// in slot order.  Block (t, c): 1024 columns of token t, one float4 per
// thread; the k expert-output loads are all issued before the additions.
// With kF32Out the fp32 sum is stored unrounded (a tensor-parallel shard's
// partial output, rounded once after the partials are added up).
constexpr int kCombineCols = 1024;

template <bool kF32Out>
__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ obuf, const int32_t* __restrict__ prow,
                                                 const float* __restrict__ gates, void* __restrict__ y, int H, int K)
{
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int rows[kMaxTopK];
    __shared__ float g[kMaxTopK];
    const int t = blockIdx.x;
    if (threadIdx.x < K) {
        rows[threadIdx.x] = prow[(size_t)t * K + threadIdx.x];
        g[threadIdx.x] = gates[(size_t)t * K + threadIdx.x];
    }
    __syncthreads();
    const int h4 = blockIdx.y * (kCombineCols / 4) + threadIdx.x;
    if (h4 >= H / 4) return;
    float4 o[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
        if (j < K) o[j] = reinterpret_cast<const float4*>(obuf + (size_t)rows[j] * H)[h4];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        if (j < K) {
            acc.x = fmaf(g[j], o[j].x, acc.x);
            acc.y = fmaf(g[j], o[j].y, acc.y);
            acc.z = fmaf(g[j], o[j].z, acc.z);
            acc.w = fmaf(g[j], o[j].w, acc.w);
        }
    }
    if constexpr (kF32Out) {
        reinterpret_cast<float4*>(static_cast<float*>(y) + (size_t)t * H)[h4] = acc;
    } else {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 out;
        out.x = *reinterpret_cast<const uint32_t*>(&lo);
        out.y = *reinterpret_cast<const uint32_t*>(&hi);
        reinterpret_cast<uint2*>(static_cast<uint16_t*>(y) + (size_t)t * H)[h4] = out;
    }
}

cudaError_t launch_combine(const DevState& s, uint16_t* y, int T, cudaStream_t st)
{
    const dim3 grid(T, (s.H + kCombineCols - 1) / kCombineCols);
    return launch_kernel(k_combine<false>, grid, dim3(256), 0, st, s.pdl, (const float*)s.obuf, (const int32_t*)s.prow,
                         (const float*)s.gates, (void*)y, s.H, s.K);
}

cudaError_t launch_combine_f32(const DevState& s, float* y32, int T, cudaStream_t st)
{
    const dim3 grid(T, (s.H + kCombineCols - 1) / kCombineCols);
    return launch_kernel(k_combine<true>, grid, dim3(256), 0, st, s.pdl, (const float*)s.obuf, (const int32_t*)s.prow,
                         (const float*)s.gates, (void*)y32, s.H, s.K);
}

// The tensor-parallel shards' partial outputs added up in shard order (fp32)
// and rounded once to bf16: y[i] = bf16_rne(p0[i] + p1[i] + ...).
struct Partials {
    const float* p[kMaxTp];
};

__global__ void __launch_bounds__(256) k_sum_partials(Partials parts, int n_parts, size_t n, uint16_t* __restrict__ y)
{
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        float v = parts.p[0][i];
        for (int r = 1; r < n_parts; ++r) v += parts.p[r][i];
        const __nv_bfloat16 b = __float2bfloat16_rn(v);
        y[i] = *reinterpret_cast<const uint16_t*>(&b);
    }
}

cudaError_t launch_sum_partials(const float* const* parts, int n_parts, size_t n, uint16_t* y, cudaStream_t st)
{
    Partials p{};
    for (int r = 0; r < n_parts; ++r) p.p[r] = parts[r];
    const size_t blocks = (n + 255) / 256;
    k_sum_partials<<<(unsigned)(blocks < 4736 ? blocks : 4736), 256, 0, st>>>(p, n_parts, n, y);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ load time
// Weight rows of one expert are grouped into tiles of 128 * halves rows (a
// GEMM n-tile) and K into 128-wide steps.  mode 0 (fused gate/up, R = 2I):
// tile nt holds gate rows [128 nt, 128 nt + 128) as half 0 and the matching
// up rows (I + same) as half 1.  mode 1 (down, R = H): tile nt holds rows
// [128 halves nt, 128 halves (nt + 1)), half = which 128-row part.
__device__ __forceinline__ void tile_of_row(int r, int mode, int halves, int I128, int& nt, int& half, int& rr)
{
    rr = r & 127;
    const int blk = r >> 7;                 // 128-row block index within the expert
    if (mode == 0) {
        half = blk / I128;
        nt = blk - half * I128;
    } else {
        nt = blk / halves;
        half = blk - nt * halves;
    }
}

// Both projections are stored as one interleaved, tile-major buffer: for
// every (expert e, n-tile nt, K-step kb) a block of halves * 136 rows of 64
// bytes - the halves * 128 weight rows of that GEMM stage (E2M1 codes, 128
// per row) followed by halves * 8 rows holding the stage's scale chunks
// (512 bytes per 128 weight rows, in tcgen05.cp order: row rr's word at
// (rr % 32) * 4 + rr / 32 holds the E8M0 bytes of the four 32-wide K
// sub-blocks).  One stage then reads one contiguous run of memory.
__host__ __device__ __forceinline__ size_t wblock_row(int e, int nt, int kb, int NT, int KB, int halves)
{
    return ((((size_t)e * NT + nt) * KB + kb) * halves) * kWBlockRowsPerHalf;
}

__global__ void k_repack_sf(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int E, int KB, int NT,
                            int halves, int rows_total, int K32, int mode, int I128)
{
    const size_t n = (size_t)E * rows_total * KB;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int kb = (int)(i % KB);
        const size_t er = i / KB;
        const int r = (int)(er % rows_total);
        const int e = (int)(er / rows_total);
        int nt, half, rr;
        tile_of_row(r, mode, halves, I128, nt, half, rr);
        const uint8_t* s = src + er * K32 + kb * 4;
        const uint32_t w = (uint32_t)s[0] | ((uint32_t)s[1] << 8) | ((uint32_t)s[2] << 16) | ((uint32_t)s[3] << 24);
        const size_t sf_row = wblock_row(e, nt, kb, NT, KB, halves) + (size_t)halves * 128;
        uint32_t* chunk = reinterpret_cast<uint32_t*>(dst + sf_row * 64 + (size_t)half * 512);
        chunk[(rr & 31) * 4 + (rr >> 5)] = w;
    }
}

cudaError_t launch_repack_sf(const uint8_t* src, uint8_t* dst, int E, int KB, int NT, int halves, int rows_total,
                             int K32, int mode, int I128, cudaStream_t st)
{
    k_repack_sf<<<2368, 256, 0, st>>>(src, dst, E, KB, NT, halves, rows_total, K32, mode, I128);
    return cudaGetLastError();
}

// Canonical packed E2M1 [E][R][K/2] -> the weight rows of the interleaved
// tile-major buffer.  One thread per 16 bytes.
__global__ void k_repack_w(const uint4* __restrict__ src, uint4* __restrict__ dst, int E, int KB, int NT, int halves,
                           int rows_total, int mode, int I128)
{
    const size_t n = (size_t)E * rows_total * KB * 4;   // 16-byte pieces
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int q = (int)(i & 3);                 // 16-byte piece within the 64-byte row slice
        const int kb = (int)((i >> 2) % KB);
        const size_t er = (i >> 2) / KB;
        const int r = (int)(er % rows_total);
        const int e = (int)(er / rows_total);
        int nt, half, rr;
        tile_of_row(r, mode, halves, I128, nt, half, rr);
        const size_t row_t = wblock_row(e, nt, kb, NT, KB, halves) + (size_t)half * 128 + rr;
        dst[row_t * 4 + q] = src[i];
    }
}

cudaError_t launch_repack_w(const uint8_t* src, uint8_t* dst, int E, int KB, int NT, int halves, int rows_total,
                            int mode, int I128, cudaStream_t st)
{
    k_repack_w<<<4736, 256, 0, st>>>(reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), E, KB, NT,
                                     halves, rows_total, mode, I128);
    return cudaGetLastError();
}

// fp8 expert format: canonical e4m3 [E][R][K] -> tile-major blocks
// [E][NT][KB] of halves * 128 rows x 128 bytes (one GEMM stage's weight
// rows, the same n-tile grouping as above; no scale rows: the fp32 block
// scales stay in their own table).  One thread per 16 bytes.
__global__ void k_repack_w8(const uint4* __restrict__ src, uint4* __restrict__ dst, int E, int KB, int NT, int halves,
                            int rows_total, int mode, int I128)
{
    const size_t n = (size_t)E * rows_total * KB * 8;   // 16-byte pieces
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int q = (int)(i & 7);                 // 16-byte piece within the 128-byte row slice
        const int kb = (int)((i >> 3) % KB);
        const size_t er = (i >> 3) / KB;
        const int r = (int)(er % rows_total);
        const int e = (int)(er / rows_total);
        int nt, half, rr;
        tile_of_row(r, mode, halves, I128, nt, half, rr);
        const size_t row_t = ((((size_t)e * NT + nt) * KB + kb) * halves + half) * 128 + rr;
        dst[row_t * 8 + q] = src[i];
    }
}

cudaError_t launch_repack_w8(const uint8_t* src, uint8_t* dst, int E, int KB, int NT, int halves, int rows_total,
                             int mode, int I128, cudaStream_t st)
{
    k_repack_w8<<<4736, 256, 0, st>>>(reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), E, KB, NT,
                                      halves, rows_total, mode, I128);
    return cudaGetLastError();
}

// Invalid fp8 expert input: an e4m3 NaN code (0x7F / 0xFF), or a block scale
// that is negative, infinite or NaN.
__global__ void k_check_fp8(const uint8_t* __restrict__ q, size_t n, const float* __restrict__ s, size_t ns,
                            int32_t* flag)
{
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        if ((q[i] & 0x7Fu) == 0x7Fu) {
            atomicOr(flag, 1);
            break;
        }
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < ns; i += (size_t)gridDim.x * blockDim.x)
        if (!(s[i] >= 0.0f) || isinf(s[i])) {
            atomicOr(flag, 1);
            break;
        }
}

cudaError_t launch_check_fp8(const uint8_t* q, size_t n, const float* s, size_t ns, int32_t* flag, cudaStream_t st)
{
    k_check_fp8<<<1184, 256, 0, st>>>(q, n, s, ns, flag);
    return cudaGetLastError();
}

__global__ void k_check_e8m0(const uint8_t* __restrict__ p, size_t n, int32_t* flag)
{
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        if (p[i] == 0xFFu) {
            atomicOr(flag, 1);
            return;
        }
}

cudaError_t launch_check_e8m0(const uint8_t* p, size_t n, int32_t* flag, cudaStream_t st)
{
    k_check_e8m0<<<1184, 256, 0, st>>>(p, n, flag);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ getters
__global__ void k_unpad_perm(const int32_t* __restrict__ prow, const int32_t* __restrict__ ids,
                             const int32_t* __restrict__ offsets, const int32_t* __restrict__ mtile_off,
                             int32_t* __restrict__ out, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int e = ids[i];
    out[i] = offsets[e] + (prow[i] - mtile_off[e] * kBM);
}

cudaError_t launch_unpad_perm(const DevState& s, int T, int32_t* out, cudaStream_t st)
{
    const int n = T * s.K;
    k_unpad_perm<<<(n + 255) / 256, 256, 0, st>>>(s.prow, s.ids, s.offsets, s.mtile_off, out, n);
    return cudaGetLastError();
}

__device__ __forceinline__ int padded_row_of(const int32_t* offsets, const int32_t* mtile_off, int E, int r)
{
    int lo = 0, hi = E - 1;   // last e with offsets[e] <= r and a non-empty range
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offsets[mid] <= r) lo = mid;
        else hi = mid - 1;
    }
    return mtile_off[lo] * kBM + (r - offsets[lo]);
}

// which = 0: activation codes of token t (its slot-0 row); which = 1: SwiGLU
// codes of canonical row r.  One block per output row.
__global__ void k_gather_q(const uint8_t* __restrict__ src, const uint32_t* __restrict__ sf, const int32_t* prow,
                           const int32_t* offsets, const int32_t* mtile_off, int E, int K, int width, int which,
                           uint8_t* __restrict__ q, uint8_t* __restrict__ sc)
{
    const int r = blockIdx.x;
    const int prw = (which == 0) ? prow[(size_t)r * K] : padded_row_of(offsets, mtile_off, E, r);
    const int KB = width / 128;
    for (int i = threadIdx.x; i < width; i += blockDim.x)
        if (q) q[(size_t)r * width + i] = src[(size_t)prw * width + i];
    for (int kb = threadIdx.x; kb < KB; kb += blockDim.x)
        if (sc) sc[(size_t)r * KB + kb] = (uint8_t)(sf[sf_word_index(prw >> 7, kb, KB, prw & 127)] & 0xFFu);
}

// Block scales of the rows of a getter as fp32 values: E8M0 bytes decoded
// (2^(b-127)), or the fp32-scale table as stored.
__global__ void k_gather_scales_f32(const uint32_t* __restrict__ sf, const float* __restrict__ sf32, const int32_t* prow,
                                    const int32_t* offsets, const int32_t* mtile_off, int E, int K, int KB, int which,
                                    float* __restrict__ out)
{
    const int r = blockIdx.x;
    const int prw = (which == 0) ? prow[(size_t)r * K] : padded_row_of(offsets, mtile_off, E, r);
    for (int kb = threadIdx.x; kb < KB; kb += blockDim.x) {
        float v;
        if (sf32) {
            v = sf32[(size_t)prw * KB + kb];
        } else {
            const int b = (int)(sf[sf_word_index(prw >> 7, kb, KB, prw & 127)] & 0xFFu);
            v = b == 0 ? 0x1p-127f : __int_as_float(b << 23);   // 2^(b - 127); byte 0 is 2^-127 (subnormal)
        }
        out[(size_t)r * KB + kb] = v;
    }
}

cudaError_t launch_gather_scales_f32(const DevState& s, int T, int which, float* out, cudaStream_t st)
{
    const int rows = (which == 0) ? T : T * s.K;
    if (rows == 0) return cudaSuccess;
    if (which == 0)
        k_gather_scales_f32<<<rows, 128, 0, st>>>(s.asf, s.act_f32 ? s.asf32 : nullptr, s.prow, s.offsets,
                                                  s.mtile_off, s.E, s.K, s.H / 128, 0, out);
    else
        k_gather_scales_f32<<<rows, 128, 0, st>>>(s.hsf, s.act_f32 ? s.hsf32 : nullptr, s.prow, s.offsets,
                                                  s.mtile_off, s.E, s.K, s.I / 128, 1, out);
    return cudaGetLastError();
}

cudaError_t launch_gather_rows_u8(const DevState& s, int T, int which, uint8_t* q, uint8_t* sc, cudaStream_t st)
{
    const int rows = (which == 0) ? T : T * s.K;
    if (rows == 0) return cudaSuccess;
    if (which == 0)
        k_gather_q<<<rows, 256, 0, st>>>(s.aq, s.asf, s.prow, s.offsets, s.mtile_off, s.E, s.K, s.H, 0, q, sc);
    else
        k_gather_q<<<rows, 256, 0, st>>>(s.hq, s.hsf, s.prow, s.offsets, s.mtile_off, s.E, s.K, s.I, 1, q, sc);
    return cudaGetLastError();
}

__global__ void k_gather_obuf(const float* __restrict__ obuf, const int32_t* offsets, const int32_t* mtile_off, int E,
                              int H, float* __restrict__ out)
{
    const int r = blockIdx.x;
    const int prw = padded_row_of(offsets, mtile_off, E, r);
    for (int i = threadIdx.x; i < H; i += blockDim.x) out[(size_t)r * H + i] = obuf[(size_t)prw * H + i];
}

cudaError_t launch_gather_obuf(const DevState& s, int T, float* out, cudaStream_t st)
{
    const int rows = T * s.K;
    if (rows == 0) return cudaSuccess;
    k_gather_obuf<<<rows, 256, 0, st>>>(s.obuf, s.offsets, s.mtile_off, s.E, s.H, out);
    return cudaGetLastError();
}

}  // namespace moe
