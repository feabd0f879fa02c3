// C ABI of the routed MXFP4 MoE layer: argument checks, device workspace,
// TMA tensor maps, weight loading, the stream-ordered forward and the debug
// getters.  See include/moe_mx.h for the contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/moe_mx.h"
#include "moe_internal.cuh"
#include "ptx.cuh"

using namespace moe;

static const char* kStageNames[] = {"router", "topk", "dispatch", "gemm1_gate_up", "gemm2_down", "combine"};
constexpr int kNumStages = 6;
constexpr int kProfSlots = 64;   // forwards whose stage events are kept

struct moe_handle {
    moe_config cfg{};
    DevState s{};
    bool loaded = false;
    int last_T = -1;
    int last_launches = 0;
    bool profiling = false;
    cudaEvent_t ev[kProfSlots][kNumStages + 1] = {};
    bool ev_valid = false;
    int prof_count = 0;      // forwards recorded since profiling was enabled / last read
    std::vector<void*> allocs;
    // staging for the host-buffer entry points: two slots, so that one call's
    // copies overlap the neighbouring calls' forwards
    uint16_t* xbuf[2] = {nullptr, nullptr};
    uint16_t* ybuf[2] = {nullptr, nullptr};
    cudaStream_t s_in = nullptr, s_out = nullptr;   // copy streams (host -> device, device -> host)
    cudaEvent_t ev_in[2] = {}, ev_fwd[2] = {}, ev_out[2] = {};
    bool host_ready = false;      // streams and events created
    bool slot_used[2] = {false, false};
    int host_calls = 0;           // host-buffer calls so far (slot = calls % 2)
    // owned weight buffers
    void* w_alloc[8] = {};      // [7]: staging of whole tensors while a shard loads its slice
    // tensor-parallel shard of the expert middle dimension (1 / 0: the whole layer)
    int tp_size = 1, tp_rank = 0, I_full = 0;
    std::string err;
};

static thread_local std::string g_err;

// Set the message moe_last_error(NULL) returns (for entry points without a handle).
void moe_set_handle_free_error(const char* msg) { g_err = msg; }

// noalloc.cu: the error record of the allocation-free routing on the current device
moe_status noalloc_error_record(int32_t** out);

static moe_status fail(moe_handle* h, moe_status st, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (h) h->err = buf;
    else g_err = buf;
    return st;
}

#define CUDA_TRY(h, call)                                                                            \
    do {                                                                                             \
        cudaError_t e_ = (call);                                                                     \
        if (e_ != cudaSuccess)                                                                       \
            return fail((h), e_ == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA, "%s: %s (%s:%d)", \
                        #call, cudaGetErrorString(e_), __FILE__, __LINE__);                          \
    } while (0)

static PFN_cuTensorMapEncodeTiled_v12000 get_encode()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D tensor map over a row-major [rows][inner] tensor, 128-byte swizzle.
static bool make_map(CUtensorMap* m, CUtensorMapDataType dt, void* base, uint64_t inner, uint64_t rows,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows)
{
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(m, dt, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <typename T>
static moe_status dalloc(moe_handle* h, T** p, size_t bytes)
{
    void* q = nullptr;
    cudaError_t e = cudaMalloc(&q, bytes < 256 ? 256 : bytes);
    if (e != cudaSuccess)
        return fail(h, MOE_ERR_OOM, "cudaMalloc(%zu bytes): %s", bytes, cudaGetErrorString(e));
    h->allocs.push_back(q);
    *p = static_cast<T*>(q);
    return MOE_OK;
}

static moe_status getter_prologue(moe_handle* h)
{
    if (!h) return fail(nullptr, MOE_ERR_INVALID_ARG, "handle is NULL");
    if (h->last_T < 0) return fail(h, MOE_ERR_NOT_LOADED, "no forward has run since the weights were loaded");
    return moe_check_device_error(h);
}

template <typename Fn>
static moe_status with_tmp(moe_handle* h, size_t bytes, void* host_out, Fn&& fill)
{
    if (!host_out || bytes == 0) return MOE_OK;
    void* d = nullptr;
    CUDA_TRY(h, cudaMalloc(&d, bytes));
    cudaError_t e = fill(d);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(host_out, d, bytes, cudaMemcpyDeviceToHost);
    cudaFree(d);
    if (e != cudaSuccess) return fail(h, MOE_ERR_CUDA, "getter: %s", cudaGetErrorString(e));
    return MOE_OK;
}

// Tensor-parallel shards keep a slice of the expert middle dimension I: rank
// r of G holds middle columns [r Il, (r + 1) Il), Il = I / G, of every
// expert.  The canonical tensors are first copied whole into `full` (device)
// and the slice is then gathered into `dst`:
//  * W13-like tensors [E][2 If][row bytes] (gate rows, then up rows): rows
//    [r Il, (r+1) Il) of each half -> [E][2 Il][row bytes];
//  * W2-like tensors [rows][If-dependent bytes]: the byte range
//    [r * loc_bytes, (r + 1) * loc_bytes) of every row -> [rows][loc_bytes].
// With G = 1 the tensor is copied as it is.
static cudaError_t stage_w13(void* dst, const void* src, void* full, size_t E, size_t If, size_t Il, size_t r,
                             size_t row_bytes)
{
    if (If == Il) return cudaMemcpy(dst, src, E * 2 * If * row_bytes, cudaMemcpyDefault);
    cudaError_t e = cudaMemcpy(full, src, E * 2 * If * row_bytes, cudaMemcpyDefault);
    for (size_t half = 0; half < 2 && e == cudaSuccess; ++half)
        e = cudaMemcpy2D(static_cast<uint8_t*>(dst) + half * Il * row_bytes, 2 * Il * row_bytes,
                         static_cast<const uint8_t*>(full) + (half * If + r * Il) * row_bytes, 2 * If * row_bytes,
                         Il * row_bytes, E, cudaMemcpyDeviceToDevice);
    return e;
}

static cudaError_t stage_w2(void* dst, const void* src, void* full, size_t rows, size_t full_bytes, size_t loc_bytes,
                            size_t r)
{
    if (full_bytes == loc_bytes) return cudaMemcpy(dst, src, rows * full_bytes, cudaMemcpyDefault);
    cudaError_t e = cudaMemcpy(full, src, rows * full_bytes, cudaMemcpyDefault);
    if (e == cudaSuccess)
        e = cudaMemcpy2D(dst, loc_bytes, static_cast<const uint8_t*>(full) + r * loc_bytes, full_bytes, loc_bytes, rows,
                         cudaMemcpyDeviceToDevice);
    return e;
}

extern "C" {

const char* moe_status_string(moe_status s)
{
    switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_SHAPE: return "unsupported shape";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_OOM: return "out of device memory";
    case MOE_ERR_NOT_LOADED: return "weights not loaded / no forward yet";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_UNSUPPORTED: return "unsupported device";
    case MOE_ERR_DEVICE: return "device-side error";
    }
    return "unknown status";
}

const char* moe_last_error(moe_handle* h) { return h ? h->err.c_str() : g_err.c_str(); }

int moe_stage_count(void) { return kNumStages; }
const char* moe_stage_name(int i) { return (i >= 0 && i < kNumStages) ? kStageNames[i] : ""; }

moe_status moe_destroy(moe_handle* h)
{
    if (!h) return MOE_OK;
    cudaSetDevice(h->cfg.device);
    for (void* p : h->allocs) cudaFree(p);
    for (void* p : h->w_alloc)
        if (p) cudaFree(p);
    if (h->ev_valid)
        for (auto& slot : h->ev)
            for (auto& e : slot) cudaEventDestroy(e);
    if (h->host_ready) {
        cudaStreamSynchronize(h->s_out);
        for (int b = 0; b < 2; ++b) {
            cudaEventDestroy(h->ev_in[b]);
            cudaEventDestroy(h->ev_fwd[b]);
            cudaEventDestroy(h->ev_out[b]);
        }
        cudaStreamDestroy(h->s_in);
        cudaStreamDestroy(h->s_out);
    }
    delete h;
    return MOE_OK;
}

moe_status moe_init(const moe_config* cfg, moe_handle** out)
{
    if (!out) return fail(nullptr, MOE_ERR_INVALID_ARG, "moe_init: out is NULL");
    *out = nullptr;
    if (!cfg) return fail(nullptr, MOE_ERR_INVALID_ARG, "moe_init: cfg is NULL");
    const moe_config c = *cfg;
    if (c.hidden < 128 || c.hidden > 16384 || c.hidden % 128)
        return fail(nullptr, MOE_ERR_SHAPE, "hidden=%d: must be a multiple of 128 in [128, 16384]", c.hidden);
    if (c.inter < 128 || c.inter > 16384 || c.inter % 128)
        return fail(nullptr, MOE_ERR_SHAPE, "inter=%d: must be a multiple of 128 in [128, 16384]", c.inter);
    if (c.num_experts < 1 || c.num_experts > kMaxExperts)
        return fail(nullptr, MOE_ERR_SHAPE, "num_experts=%d: must be in [1, %d]", c.num_experts, kMaxExperts);
    if (c.top_k < 1 || c.top_k > kMaxTopK || c.top_k > c.num_experts)
        return fail(nullptr, MOE_ERR_SHAPE, "top_k=%d: must be in [1, min(E, 8)]", c.top_k);
    if (c.max_tokens < 1 || c.max_tokens > (1 << 20))
        return fail(nullptr, MOE_ERR_SHAPE, "max_tokens=%d: must be in [1, 2^20]", c.max_tokens);
    if (c.score_func != MOE_SCORE_SIGMOID && c.score_func != MOE_SCORE_SOFTMAX)
        return fail(nullptr, MOE_ERR_INVALID_ARG, "score_func=%d", c.score_func);
    if (c.act_scale_mode != MOE_ACT_SCALE_E8M0 && c.act_scale_mode != MOE_ACT_SCALE_F32)
        return fail(nullptr, MOE_ERR_INVALID_ARG, "act_scale_mode=%d", c.act_scale_mode);
    const int G = c.tp_size == 0 ? 1 : c.tp_size;
    if (G < 1 || G > kMaxTp || c.tp_rank < 0 || c.tp_rank >= G)
        return fail(nullptr, MOE_ERR_INVALID_ARG, "tp_size=%d tp_rank=%d: need 1 <= tp_size <= %d, 0 <= tp_rank < tp_size",
                    c.tp_size, c.tp_rank, kMaxTp);
    if (c.inter % (128 * G))
        return fail(nullptr, MOE_ERR_SHAPE, "inter=%d is not a multiple of 128 * tp_size=%d", c.inter, 128 * G);
    if (cudaSetDevice(c.device) != cudaSuccess)
        return fail(nullptr, MOE_ERR_CUDA, "cudaSetDevice(%d) failed", c.device);
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, c.device) != cudaSuccess)
        return fail(nullptr, MOE_ERR_CUDA, "cudaGetDeviceProperties failed");
    if (prop.major != 10 || prop.minor != 3)
        return fail(nullptr, MOE_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                    c.device, prop.major, prop.minor);
    if (!get_encode()) return fail(nullptr, MOE_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");

    moe_handle* h = new moe_handle;
    h->cfg = c;
    h->tp_size = G;
    h->tp_rank = c.tp_rank;
    h->I_full = c.inter;
    DevState& s = h->s;
    s.H = c.hidden;
    s.I = c.inter / G;   // this shard's slice of the expert middle dimension
    s.E = c.num_experts;
    s.K = c.top_k;
    s.Tm = c.max_tokens;
    s.score_func = c.score_func;
    s.act_f32 = c.act_scale_mode == MOE_ACT_SCALE_F32;
    s.KB1 = s.H / 128;
    s.KB2 = s.I / 128;
    s.NT1 = s.I / 128;
    s.BN2 = (s.H % 256 == 0) ? 256 : 128;
    s.NT2 = s.H / s.BN2;
    s.MTmax = (s.Tm * s.K + kBM - 1) / kBM + s.E;
    s.Rmax = s.MTmax * kBM;
    s.nchunk_max = (s.Tm + kChunk - 1) / kChunk;
    s.num_sms = prop.multiProcessorCount;

    moe_status st;
#define ALLOC(ptr, bytes)                                      \
    if ((st = dalloc(h, &(ptr), (bytes))) != MOE_OK) {         \
        std::string m = h->err;                                \
        moe_destroy(h);                                        \
        return fail(nullptr, st, "%s", m.c_str());             \
    }
    ALLOC(s.logits, sizeof(float) * s.Tm * s.E);
    ALLOC(s.logit_part, sizeof(float) * kRouterMaxSplit * (s.Tm < kRouterSplitMaxT ? s.Tm : kRouterSplitMaxT) * s.E);
    ALLOC(s.ids, sizeof(int32_t) * s.Tm * s.K);
    ALLOC(s.gates, sizeof(float) * s.Tm * s.K);
    ALLOC(s.chunk_hist, sizeof(int32_t) * s.nchunk_max * s.E);
    ALLOC(s.chunk_base, sizeof(int32_t) * s.nchunk_max * s.E);
    ALLOC(s.counts, sizeof(int32_t) * s.E);
    ALLOC(s.offsets, sizeof(int32_t) * (s.E + 1));
    ALLOC(s.mtile_off, sizeof(int32_t) * (s.E + 1));
    ALLOC(s.mtile_expert, sizeof(int32_t) * s.MTmax);
    ALLOC(s.mtile_rows, sizeof(int32_t) * s.MTmax);
    ALLOC(s.n_mtiles, sizeof(int32_t) * 4);
    ALLOC(s.light_list, sizeof(int32_t) * s.MTmax);
    ALLOC(s.heavy_list, sizeof(int32_t) * s.MTmax);
    ALLOC(s.prow, sizeof(int32_t) * s.Tm * s.K);
    ALLOC(s.aq, (size_t)s.Rmax * s.H);
    ALLOC(s.asf, sizeof(uint32_t) * (size_t)s.MTmax * s.KB1 * 128);
    ALLOC(s.hq, (size_t)s.Rmax * s.I);
    ALLOC(s.hsf, sizeof(uint32_t) * (size_t)s.MTmax * s.KB2 * 128);
    ALLOC(s.obuf, sizeof(float) * (size_t)s.Rmax * s.H);
    if (s.act_f32) {
        ALLOC(s.asf32, sizeof(float) * (size_t)s.Rmax * s.KB1);
        ALLOC(s.hsf32, sizeof(float) * (size_t)s.Rmax * s.KB2);
    }
    ALLOC(s.err, sizeof(int32_t) * 4);
    for (int b = 0; b < 2; ++b) {
        ALLOC(h->xbuf[b], sizeof(uint16_t) * (size_t)s.Tm * s.H);
        ALLOC(h->ybuf[b], sizeof(uint16_t) * (size_t)s.Tm * s.H);
    }
#undef ALLOC
    // padding rows of the activation / SwiGLU buffers are never written by a
    // forward; zero them once so every tile reads finite values
    bool ok = cudaMemset(s.aq, 0, (size_t)s.Rmax * s.H) == cudaSuccess &&
              cudaMemset(s.asf, 0, sizeof(uint32_t) * (size_t)s.MTmax * s.KB1 * 128) == cudaSuccess &&
              cudaMemset(s.hq, 0, (size_t)s.Rmax * s.I) == cudaSuccess &&
              cudaMemset(s.hsf, 0, sizeof(uint32_t) * (size_t)s.MTmax * s.KB2 * 128) == cudaSuccess &&
              cudaMemset(s.err, 0, sizeof(int32_t) * 4) == cudaSuccess &&
              cudaMemset(s.n_mtiles, 0, sizeof(int32_t) * 4) == cudaSuccess;
    if (ok && s.act_f32)
        ok = cudaMemset(s.asf32, 0, sizeof(float) * (size_t)s.Rmax * s.KB1) == cudaSuccess &&
             cudaMemset(s.hsf32, 0, sizeof(float) * (size_t)s.Rmax * s.KB2) == cudaSuccess;
    const uint32_t boxes[kNumABox] = {8, 16, 32, 64, 128};
    for (int i = 0; ok && i < kNumABox; ++i) {
        ok = make_map(&s.tm_aq[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, s.aq, s.H, s.Rmax, s.H, 128, boxes[i]) &&
             make_map(&s.tm_hq[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, s.hq, s.I, s.Rmax, s.I, 128, boxes[i]);
    }
    if (ok)
        ok = gemm_set_attributes() == cudaSuccess && router_set_attributes() == cudaSuccess;

    if (ok) ok = cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) {
        moe_destroy(h);
        return fail(nullptr, MOE_ERR_CUDA, "moe_init: workspace setup failed: %s",
                    cudaGetErrorString(cudaGetLastError()));
    }
    *out = h;
    return MOE_OK;
}

moe_status moe_load_weights(moe_handle* h, const uint16_t* router_w, const float* logit_bias, const float* sel_bias,
                            const uint8_t* w13_q, const uint8_t* w13_s, const uint8_t* w2_q, const uint8_t* w2_s)
{
    if (!h) return fail(nullptr, MOE_ERR_INVALID_ARG, "moe_load_weights: handle is NULL");
    if (!router_w || !w13_q || !w13_s || !w2_q || !w2_s)
        return fail(h, MOE_ERR_INVALID_ARG, "moe_load_weights: a required weight pointer is NULL");
    DevState& s = h->s;
    CUDA_TRY(h, cudaSetDevice(h->cfg.device));
    h->loaded = false;
    for (void*& p : h->w_alloc)
        if (p) {
            cudaFree(p);
            p = nullptr;
        }
    const size_t E = s.E, H = s.H, I = s.I;   // I: this shard's middle width
    const size_t If = h->I_full, r = h->tp_rank;
    const size_t n_wr = E * H * 2, n_13q = E * 2 * I * H / 2, n_13s = E * 2 * I * H / 32, n_2q = E * H * I / 2,
                 n_2s = E * H * I / 32;
    const int halves2 = s.BN2 / 128;
    const uint64_t rows13 = (uint64_t)E * s.NT1 * s.KB1 * 2 * kWBlockRowsPerHalf;
    const uint64_t rows2 = (uint64_t)E * s.NT2 * s.KB2 * halves2 * kWBlockRowsPerHalf;
    void *d_wr, *d_b, *d_13, *d_2, *d_tmp, *d_full = nullptr;
    size_t n_tmp = n_13q;
    if (n_2q > n_tmp) n_tmp = n_2q;
    if (If != I) {   // a shard: the canonical tensors are staged whole, then sliced
        CUDA_TRY(h, cudaMalloc(&d_full, E * 2 * If * H / 2 > E * H * If / 2 ? E * 2 * If * H / 2 : E * H * If / 2));
        h->w_alloc[7] = d_full;
    }
    CUDA_TRY(h, cudaMalloc(&d_wr, n_wr));
    h->w_alloc[0] = d_wr;
    CUDA_TRY(h, cudaMalloc(&d_b, 2 * E * sizeof(float)));
    h->w_alloc[1] = d_b;
    CUDA_TRY(h, cudaMalloc(&d_13, rows13 * 64));
    h->w_alloc[2] = d_13;
    CUDA_TRY(h, cudaMalloc(&d_2, rows2 * 64));
    h->w_alloc[3] = d_2;
    CUDA_TRY(h, cudaMalloc(&d_tmp, n_tmp + 256));
    h->w_alloc[6] = d_tmp;
    float* d_lb = static_cast<float*>(d_b);
    float* d_cb = d_lb + E;
    uint8_t* tmp = static_cast<uint8_t*>(d_tmp);
    CUDA_TRY(h, cudaMemcpy(d_wr, router_w, n_wr, cudaMemcpyDefault));
    CUDA_TRY(h, cudaMemset(d_b, 0, 2 * E * sizeof(float)));
    if (logit_bias) CUDA_TRY(h, cudaMemcpy(d_lb, logit_bias, E * sizeof(float), cudaMemcpyDefault));
    if (sel_bias) CUDA_TRY(h, cudaMemcpy(d_cb, sel_bias, E * sizeof(float), cudaMemcpyDefault));
    // expert values: canonical [E][R][K/2] (this shard's slice) -> interleaved
    // tile-major blocks (one contiguous run per GEMM stage)
    CUDA_TRY(h, stage_w13(tmp, w13_q, d_full, E, If, I, r, H / 2));
    CUDA_TRY(h, launch_repack_w(tmp, static_cast<uint8_t*>(d_13), s.E, s.KB1, s.NT1, 2, 2 * s.I, 0, s.I / 128, 0));
    CUDA_TRY(h, cudaDeviceSynchronize());
    CUDA_TRY(h, stage_w2(tmp, w2_q, d_full, E * H, If / 2, I / 2, r));
    CUDA_TRY(h, launch_repack_w(tmp, static_cast<uint8_t*>(d_2), s.E, s.KB2, s.NT2, halves2, s.H, 1, s.I / 128, 0));
    CUDA_TRY(h, cudaDeviceSynchronize());

    int32_t* flag = s.err + 3;
    CUDA_TRY(h, cudaMemset(flag, 0, sizeof(int32_t)));
    // scales: canonical [E][R][K/32] -> the scale rows of the same blocks
    CUDA_TRY(h, stage_w13(tmp, w13_s, d_full, E, If, I, r, H / 32));
    CUDA_TRY(h, launch_check_e8m0(tmp, n_13s, flag, 0));
    CUDA_TRY(h, launch_repack_sf(tmp, static_cast<uint8_t*>(d_13), s.E, s.KB1, s.NT1, 2, 2 * s.I, s.H / 32, 0,
                                 s.I / 128, 0));
    CUDA_TRY(h, cudaDeviceSynchronize());
    CUDA_TRY(h, stage_w2(tmp, w2_s, d_full, E * H, If / 32, I / 32, r));
    CUDA_TRY(h, launch_check_e8m0(tmp, n_2s, flag, 0));
    CUDA_TRY(h, launch_repack_sf(tmp, static_cast<uint8_t*>(d_2), s.E, s.KB2, s.NT2, halves2, s.H, s.I / 32, 1,
                                 s.I / 128, 0));
    CUDA_TRY(h, cudaDeviceSynchronize());
    int32_t nan_found = 0;
    CUDA_TRY(h, cudaMemcpy(&nan_found, flag, sizeof(int32_t), cudaMemcpyDeviceToHost));
    cudaFree(d_tmp);
    h->w_alloc[6] = nullptr;
    if (d_full) {
        cudaFree(d_full);
        h->w_alloc[7] = nullptr;
    }
    if (nan_found) {
        CUDA_TRY(h, cudaMemset(flag, 0, sizeof(int32_t)));
        return fail(h, MOE_ERR_INVALID_ARG, "moe_load_weights: an expert scale byte is 0xFF (E8M0 NaN)");
    }
    // interleaved blocks as 2-D tensors of 64-byte rows; a box covers one stage's weight rows
    if (!make_map(&s.tm_w13, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, d_13, 128, rows13, 64, 128, 256) ||
        !make_map(&s.tm_w2, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, d_2, 128, rows2, 64, 128, 128 * halves2) ||
        !make_map(&s.tm_wr64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d_wr, H, E, H * 2, 64, 64) ||
        !make_map(&s.tm_wr128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d_wr, H, E, H * 2, 64, 128))
        return fail(h, MOE_ERR_CUDA, "moe_load_weights: cuTensorMapEncodeTiled failed for the weights");
    s.wr = static_cast<const uint16_t*>(d_wr);
    s.lb = d_lb;
    s.cb = d_cb;
    s.w13q = static_cast<const uint8_t*>(d_13);
    s.w2q = static_cast<const uint8_t*>(d_2);
    s.w_fp8 = 0;
    s.ws13 = s.ws2 = nullptr;
    h->loaded = true;
    h->last_T = -1;
    return MOE_OK;
}

moe_status moe_load_weights_fp8(moe_handle* h, const uint16_t* router_w, const float* logit_bias,
                                const float* sel_bias, const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                                const float* w2_scale)
{
    if (!h) return fail(nullptr, MOE_ERR_INVALID_ARG, "moe_load_weights_fp8: handle is NULL");
    if (!router_w || !w13 || !w13_scale || !w2 || !w2_scale)
        return fail(h, MOE_ERR_INVALID_ARG, "moe_load_weights_fp8: a required weight pointer is NULL");
    DevState& s = h->s;
    CUDA_TRY(h, cudaSetDevice(h->cfg.device));
    h->loaded = false;
    for (void*& p : h->w_alloc)
        if (p) {
            cudaFree(p);
            p = nullptr;
        }
    const size_t E = s.E, H = s.H, I = s.I;   // I: this shard's middle width
    const size_t If = h->I_full, r = h->tp_rank;
    const size_t n_wr = E * H * 2, n_13 = E * 2 * I * H, n_2 = E * H * I;
    const size_t n_13s = E * (2 * I / 128) * (H / 128), n_2s = E * (H / 128) * (I / 128);
    const int halves2 = s.BN2 / 128;
    // tile-major blocks of 128-byte rows (e4m3, K = 128 per row)
    const uint64_t rows13 = (uint64_t)E * s.NT1 * s.KB1 * 2 * 128;
    const uint64_t rows2 = (uint64_t)E * s.NT2 * s.KB2 * halves2 * 128;
    void *d_wr, *d_b, *d_13, *d_2, *d_s13, *d_s2, *d_tmp;
    CUDA_TRY(h, cudaMalloc(&d_wr, n_wr));
    h->w_alloc[0] = d_wr;
    CUDA_TRY(h, cudaMalloc(&d_b, 2 * E * sizeof(float)));
    h->w_alloc[1] = d_b;
    CUDA_TRY(h, cudaMalloc(&d_13, rows13 * 128));
    h->w_alloc[2] = d_13;
    CUDA_TRY(h, cudaMalloc(&d_2, rows2 * 128));
    h->w_alloc[3] = d_2;
    CUDA_TRY(h, cudaMalloc(&d_s13, n_13s * sizeof(float)));
    h->w_alloc[4] = d_s13;
    CUDA_TRY(h, cudaMalloc(&d_s2, n_2s * sizeof(float)));
    h->w_alloc[5] = d_s2;
    CUDA_TRY(h, cudaMalloc(&d_tmp, (n_13 > n_2 ? n_13 : n_2) + 256));
    h->w_alloc[6] = d_tmp;
    void* d_full = nullptr;
    if (If != I) {   // a shard: the canonical tensors are staged whole, then sliced
        CUDA_TRY(h, cudaMalloc(&d_full, E * 2 * If * H));
        h->w_alloc[7] = d_full;
    }
    float* d_lb = static_cast<float*>(d_b);
    float* d_cb = d_lb + E;
    uint8_t* tmp = static_cast<uint8_t*>(d_tmp);
    CUDA_TRY(h, cudaMemcpy(d_wr, router_w, n_wr, cudaMemcpyDefault));
    CUDA_TRY(h, cudaMemset(d_b, 0, 2 * E * sizeof(float)));
    if (logit_bias) CUDA_TRY(h, cudaMemcpy(d_lb, logit_bias, E * sizeof(float), cudaMemcpyDefault));
    if (sel_bias) CUDA_TRY(h, cudaMemcpy(d_cb, sel_bias, E * sizeof(float), cudaMemcpyDefault));
    int32_t* flag = s.err + 3;
    CUDA_TRY(h, cudaMemset(flag, 0, sizeof(int32_t)));
    CUDA_TRY(h, stage_w13(tmp, w13, d_full, E, If, I, r, H));
    CUDA_TRY(h, launch_check_fp8(tmp, n_13, nullptr, 0, flag, 0));
    CUDA_TRY(h, launch_repack_w8(tmp, static_cast<uint8_t*>(d_13), s.E, s.KB1, s.NT1, 2, 2 * s.I, 0, s.I / 128, 0));
    CUDA_TRY(h, cudaDeviceSynchronize());
    CUDA_TRY(h, stage_w2(tmp, w2, d_full, E * H, If, I, r));
    CUDA_TRY(h, launch_check_fp8(tmp, n_2, nullptr, 0, flag, 0));
    CUDA_TRY(h, launch_repack_w8(tmp, static_cast<uint8_t*>(d_2), s.E, s.KB2, s.NT2, halves2, s.H, 1, s.I / 128, 0));
    CUDA_TRY(h, cudaDeviceSynchronize());
    // block scales: [E][2I/128][H/128] (gate block rows, then up) and [E][H/128][I/128]
    CUDA_TRY(h, stage_w13(d_s13, w13_scale, d_full, E, If / 128, I / 128, r, 4 * (H / 128)));
    CUDA_TRY(h, stage_w2(d_s2, w2_scale, d_full, E * (H / 128), 4 * (If / 128), 4 * (I / 128), r));
    CUDA_TRY(h, launch_check_fp8(nullptr, 0, static_cast<const float*>(d_s13), n_13s, flag, 0));
    CUDA_TRY(h, launch_check_fp8(nullptr, 0, static_cast<const float*>(d_s2), n_2s, flag, 0));
    int32_t bad = 0;
    CUDA_TRY(h, cudaMemcpy(&bad, flag, sizeof(int32_t), cudaMemcpyDeviceToHost));
    cudaFree(d_tmp);
    h->w_alloc[6] = nullptr;
    cudaFree(d_full);
    h->w_alloc[7] = nullptr;
    if (bad) {
        CUDA_TRY(h, cudaMemset(flag, 0, sizeof(int32_t)));
        return fail(h, MOE_ERR_INVALID_ARG,
                    "moe_load_weights_fp8: an e4m3 NaN code or a negative / non-finite block scale");
    }
    if (!make_map(&s.tm_w13, CU_TENSOR_MAP_DATA_TYPE_UINT8, d_13, 128, rows13, 128, 128, 256) ||
        !make_map(&s.tm_w2, CU_TENSOR_MAP_DATA_TYPE_UINT8, d_2, 128, rows2, 128, 128, 128 * halves2) ||
        !make_map(&s.tm_wr64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d_wr, H, E, H * 2, 64, 64) ||
        !make_map(&s.tm_wr128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d_wr, H, E, H * 2, 64, 128))
        return fail(h, MOE_ERR_CUDA, "moe_load_weights_fp8: cuTensorMapEncodeTiled failed for the weights");
    s.wr = static_cast<const uint16_t*>(d_wr);
    s.lb = d_lb;
    s.cb = d_cb;
    s.w13q = static_cast<const uint8_t*>(d_13);
    s.w2q = static_cast<const uint8_t*>(d_2);
    s.ws13 = static_cast<const float*>(d_s13);
    s.ws2 = static_cast<const float*>(d_s2);
    s.w_fp8 = 1;
    h->loaded = true;
    h->last_T = -1;
    return MOE_OK;
}

moe_status moe_set_profiling(moe_handle* h, int enable)
{
    if (!h) return fail(nullptr, MOE_ERR_INVALID_ARG, "handle is NULL");
    CUDA_TRY(h, cudaSetDevice(h->cfg.device));
    if (enable && !h->ev_valid) {
        for (auto& slot : h->ev)
            for (auto& e : slot) CUDA_TRY(h, cudaEventCreate(&e));
        h->ev_valid = true;
    }
    h->profiling = enable != 0;
    h->prof_count = 0;
    return MOE_OK;
}

// The forward of moe_forward (y bf16) and moe_forward_partial (y fp32, not rounded).
static moe_status forward_impl(moe_handle* h, const uint16_t* x, int T, void* y, bool f32_out, void* stream,
                               const char* who)
{
    if (!h) return fail(nullptr, MOE_ERR_INVALID_ARG, "%s: handle is NULL", who);
    if (!h->loaded) return fail(h, MOE_ERR_NOT_LOADED, "%s: weights not loaded", who);
    if (T < 0 || T > h->s.Tm) return fail(h, MOE_ERR_SHAPE, "%s: T=%d outside [0, max_tokens=%d]", who, T, h->s.Tm);
    if (T == 0) return MOE_OK;
    if (!x || !y) return fail(h, MOE_ERR_INVALID_ARG, "%s: x or y is NULL", who);
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u)
        return fail(h, MOE_ERR_INVALID_ARG, "%s: x and y must be 16-byte aligned", who);
    const size_t xbytes = (size_t)T * h->s.H * 2, ybytes = (size_t)T * h->s.H * (f32_out ? 4 : 2);
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x), ya = reinterpret_cast<uintptr_t>(y);
    if (xa < ya + ybytes && ya < xa + xbytes) return fail(h, MOE_ERR_INVALID_ARG, "%s: x and y overlap", who);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const DevState& s = h->s;
    CUDA_TRY(h, cudaSetDevice(h->cfg.device));
    const bool prof = h->profiling && h->ev_valid;
    cudaEvent_t* ev = h->ev[h->prof_count % kProfSlots];
    int n = 0;
    CUtensorMap tmX;
    if (!make_map(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<uint16_t*>(x), s.H, (uint64_t)T, (uint64_t)s.H * 2,
                  64, 128))
        return fail(h, MOE_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed for x", who);
    const int ksplit = router_split(T, s.H);
    if (prof) CUDA_TRY(h, cudaEventRecord(ev[0], st));
    if (router_fused(T, s.E)) {
        // prefill-sized batch: the top-k runs in the router's epilogue (the
        // "topk" stage then times nothing)
        CUDA_TRY(h, launch_router_topk(s, tmX, T, st));
        ++n;
        if (prof) CUDA_TRY(h, cudaEventRecord(ev[1], st));
    } else {
        CUDA_TRY(h, launch_router_tc(s, tmX, T, st, ksplit));
        ++n;
        if (prof) CUDA_TRY(h, cudaEventRecord(ev[1], st));
        CUDA_TRY(h, launch_topk(s, T, st, ksplit));
        ++n;
    }
    if (prof) CUDA_TRY(h, cudaEventRecord(ev[2], st));
    if (T <= kChunk) {
        // small batch: histogram, scan and ranks in one single-block kernel
        CUDA_TRY(h, launch_dispatch_small(s, T, st));
        CUDA_TRY(h, launch_quant_scatter(s, x, T, st));
        n += 2;
    } else {
        CUDA_TRY(h, launch_dispatch(s, x, T, st, &n));
    }
    if (prof) CUDA_TRY(h, cudaEventRecord(ev[3], st));
    CUDA_TRY(h, launch_gemm1(s, st, T));   // light then heavy m-tiles, one launch
    ++n;
    if (prof) CUDA_TRY(h, cudaEventRecord(ev[4], st));
    CUDA_TRY(h, launch_gemm2(s, st, T));
    ++n;
    if (prof) CUDA_TRY(h, cudaEventRecord(ev[5], st));
    CUDA_TRY(h, f32_out ? launch_combine_f32(s, static_cast<float*>(y), T, st)
                        : launch_combine(s, static_cast<uint16_t*>(y), T, st));
    ++n;
    if (prof) CUDA_TRY(h, cudaEventRecord(ev[6], st));
    h->last_T = T;
    h->last_launches = n;
    if (prof) ++h->prof_count;
    return MOE_OK;
}

moe_status moe_forward(moe_handle* h, const uint16_t* x, int T, uint16_t* y, void* stream)
{
    return forward_impl(h, x, T, y, false, stream, "moe_forward");
}

moe_status moe_forward_partial(moe_handle* h, const uint16_t* x, int T, float* y32, void* stream)
{
    return forward_impl(h, x, T, y32, true, stream, "moe_forward_partial");
}

moe_status moe_sum_partials_bf16(const float* const* parts, int n_parts, size_t n, uint16_t* y, void* stream)
{
    if (!parts || !y || n_parts < 1 || n_parts > kMaxTp)
        return fail(nullptr, MOE_ERR_INVALID_ARG, "moe_sum_partials_bf16: need 1..%d partials and an output", kMaxTp);
    for (int i = 0; i < n_parts; ++i)
        if (!parts[i]) return fail(nullptr, MOE_ERR_INVALID_ARG, "moe_sum_partials_bf16: partial %d is NULL", i);
    if (n == 0) return MOE_OK;
    cudaError_t e = launch_sum_partials(parts, n_parts, n, y, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return fail(nullptr, MOE_ERR_CUDA, "moe_sum_partials_bf16: %s", cudaGetErrorString(e));
    return MOE_OK;
}

// One host-buffer forward in staging slot b = calls % 2, on three streams:
// the input copy on s_in (after the forward that last read slot b's input
// buffer), the forward on `stream` (after the input copy, and after the
// output copy that last read slot b's output buffer), the output copy on
// s_out (after the forward).  So call i's input copy overlaps call i-1's
// forward and call i-1's output copy overlaps call i's forward.
static moe_status forward_host_enqueue(moe_handle* h, const uint16_t* x_host, int T, uint16_t* y_host, void* stream,
                                       const char* who)
{
    if (!h) return fail(nullptr, MOE_ERR_INVALID_ARG, "%s: handle is NULL", who);
    if (!h->loaded) return fail(h, MOE_ERR_NOT_LOADED, "%s: weights not loaded", who);
    if (T < 0 || T > h->s.Tm) return fail(h, MOE_ERR_SHAPE, "%s: T=%d outside [0, max_tokens=%d]", who, T, h->s.Tm);
    if (T == 0) return MOE_OK;
    if (!x_host || !y_host) return fail(h, MOE_ERR_INVALID_ARG, "%s: x or y is NULL", who);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)T * h->s.H * 2;
    CUDA_TRY(h, cudaSetDevice(h->cfg.device));
    if (!h->host_ready) {
        CUDA_TRY(h, cudaStreamCreateWithFlags(&h->s_in, cudaStreamNonBlocking));
        CUDA_TRY(h, cudaStreamCreateWithFlags(&h->s_out, cudaStreamNonBlocking));
        for (int b = 0; b < 2; ++b) {
            CUDA_TRY(h, cudaEventCreateWithFlags(&h->ev_in[b], cudaEventDisableTiming));
            CUDA_TRY(h, cudaEventCreateWithFlags(&h->ev_fwd[b], cudaEventDisableTiming));
            CUDA_TRY(h, cudaEventCreateWithFlags(&h->ev_out[b], cudaEventDisableTiming));
        }
        h->host_ready = true;
    }
    const int b = h->host_calls & 1;
    if (h->slot_used[b]) CUDA_TRY(h, cudaStreamWaitEvent(h->s_in, h->ev_fwd[b], 0));
    CUDA_TRY(h, cudaMemcpyAsync(h->xbuf[b], x_host, bytes, cudaMemcpyHostToDevice, h->s_in));
    CUDA_TRY(h, cudaEventRecord(h->ev_in[b], h->s_in));
    CUDA_TRY(h, cudaStreamWaitEvent(st, h->ev_in[b], 0));
    if (h->slot_used[b]) CUDA_TRY(h, cudaStreamWaitEvent(st, h->ev_out[b], 0));
    moe_status r = moe_forward(h, h->xbuf[b], T, h->ybuf[b], stream);
    if (r != MOE_OK) return r;
    CUDA_TRY(h, cudaEventRecord(h->ev_fwd[b], st));
    CUDA_TRY(h, cudaStreamWaitEvent(h->s_out, h->ev_fwd[b], 0));
    CUDA_TRY(h, cudaMemcpyAsync(y_host, h->ybuf[b], bytes, cudaMemcpyDeviceToHost, h->s_out));
    CUDA_TRY(h, cudaEventRecord(h->ev_out[b], h->s_out));
    h->slot_used[b] = true;
    ++h->host_calls;
    return MOE_OK;
}

moe_status moe_forward_host(moe_handle* h, const uint16_t* x_host, int T, uint16_t* y_host, void* stream)
{
    moe_status r = forward_host_enqueue(h, x_host, T, y_host, stream, "moe_forward_host");
    if (r != MOE_OK || T == 0) return r;
    return moe_host_sync(h);
}

moe_status moe_forward_host_async(moe_handle* h, const uint16_t* x_host, int T, uint16_t* y_host, void* stream)
{
    return forward_host_enqueue(h, x_host, T, y_host, stream, "moe_forward_host_async");
}

moe_status moe_host_sync(moe_handle* h)
{
    if (!h) return fail(nullptr, MOE_ERR_INVALID_ARG, "moe_host_sync: handle is NULL");
    if (!h->host_ready) return MOE_OK;
    CUDA_TRY(h, cudaSetDevice(h->cfg.device));
    CUDA_TRY(h, cudaStreamSynchronize(h->s_out));
    return MOE_OK;
}

int moe_last_launch_count(moe_handle* h) { return h ? h->last_launches : 0; }

moe_status moe_debug_fill_workspace(moe_handle* h, int byte)
{
    if (!h) return fail(nullptr, MOE_ERR_INVALID_ARG, "moe_debug_fill_workspace: handle is NULL");
    if (byte < 0 || byte > 255) return fail(h, MOE_ERR_INVALID_ARG, "moe_debug_fill_workspace: byte=%d", byte);
    DevState& s = h->s;
    CUDA_TRY(h, cudaSetDevice(h->cfg.device));
    CUDA_TRY(h, cudaDeviceSynchronize());
    const size_t Tm = s.Tm, E = s.E, K = s.K, R = s.Rmax, MT = s.MTmax;
    const size_t Ts = Tm < (size_t)kRouterSplitMaxT ? Tm : (size_t)kRouterSplitMaxT;
    struct Buf { void* p; size_t n; } bufs[] = {
        {s.logits, 4 * Tm * E}, {s.logit_part, 4 * kRouterMaxSplit * Ts * E}, {s.ids, 4 * Tm * K},
        {s.gates, 4 * Tm * K}, {s.chunk_hist, 4 * (size_t)s.nchunk_max * E},
        {s.chunk_base, 4 * (size_t)s.nchunk_max * E}, {s.counts, 4 * E}, {s.offsets, 4 * (E + 1)},
        {s.mtile_off, 4 * (E + 1)}, {s.mtile_expert, 4 * MT}, {s.mtile_rows, 4 * MT}, {s.n_mtiles, 4 * 4},
        {s.light_list, 4 * MT}, {s.heavy_list, 4 * MT}, {s.prow, 4 * Tm * K}, {s.aq, R * s.H},
        {s.asf, 4 * MT * s.KB1 * 128}, {s.hq, R * s.I}, {s.hsf, 4 * MT * s.KB2 * 128},
        {s.asf32, s.act_f32 ? 4 * R * s.KB1 : 0}, {s.hsf32, s.act_f32 ? 4 * R * s.KB2 : 0},
        {s.obuf, 4 * R * s.H}, {h->xbuf[0], 2 * Tm * s.H}, {h->ybuf[0], 2 * Tm * s.H},
        {h->xbuf[1], 2 * Tm * s.H}, {h->ybuf[1], 2 * Tm * s.H}};
    for (const Buf& b : bufs)
        if (b.p && b.n) CUDA_TRY(h, cudaMemset(b.p, byte, b.n));
    CUDA_TRY(h, cudaDeviceSynchronize());
    h->last_T = -1;
    return MOE_OK;
}

}   // extern "C"

namespace moe {
// The kernels' timeout path, on purpose: one thread waits on a barrier that
// nothing completes, gives up after limit_ns, and records the timeout in the
// error word exactly as a GEMM or router wait would (site 99).
__global__ void k_wait_probe(int32_t* err, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_for(smem_u32(&bar), 0u, &abort_flag, limit_ns)) {
        if (atomicCAS(err, 0, kDevErrTimeout) == 0) {
            err[1] = 99;
            err[2] = blockIdx.x;
        }
    }
}
}  // namespace moe

extern "C" {

moe_status moe_selftest_wait_timeout(moe_handle* h, unsigned int limit_us)
{
    if (limit_us < 1 || limit_us > 1000000)
        return fail(h, MOE_ERR_INVALID_ARG, "moe_selftest_wait_timeout: limit_us=%u outside [1, 10^6]", limit_us);
    int32_t* err = nullptr;
    if (h) {
        CUDA_TRY(h, cudaSetDevice(h->cfg.device));
        err = h->s.err;
    } else {
        moe_status st = noalloc_error_record(&err);   // the allocation-free routing's error record
        if (st != MOE_OK) return st;
    }
    moe::k_wait_probe<<<1, 32>>>(err, (uint64_t)limit_us * 1000ull);
    CUDA_TRY(h, cudaGetLastError());
    return MOE_OK;
}

moe_status moe_check_device_error(moe_handle* h)
{
    if (!h) return fail(nullptr, MOE_ERR_INVALID_ARG, "handle is NULL");
    CUDA_TRY(h, cudaSetDevice(h->cfg.device));
    CUDA_TRY(h, cudaDeviceSynchronize());
    int32_t w[3] = {0, 0, 0};
    CUDA_TRY(h, cudaMemcpy(w, h->s.err, sizeof w, cudaMemcpyDeviceToHost));
    if (w[0] == 0) return MOE_OK;
    CUDA_TRY(h, cudaMemset(h->s.err, 0, 3 * sizeof(int32_t)));
    if (w[0] == kDevErrTimeout)
        return fail(h, MOE_ERR_TIMEOUT, "a kernel wait timed out (site %d, block %d)", w[1], w[2]);
    return fail(h, MOE_ERR_DEVICE, "device error code %d (site %d)", w[0], w[1]);
}

moe_status moe_get_logits(moe_handle* h, float* logits)
{
    moe_status r = getter_prologue(h);
    if (r != MOE_OK) return r;
    if (logits)
        CUDA_TRY(h, cudaMemcpy(logits, h->s.logits, sizeof(float) * h->last_T * h->s.E, cudaMemcpyDeviceToHost));
    return MOE_OK;
}

moe_status moe_get_routing(moe_handle* h, int32_t* ids, float* gates)
{
    moe_status r = getter_prologue(h);
    if (r != MOE_OK) return r;
    const size_t n = (size_t)h->last_T * h->s.K;
    if (ids) CUDA_TRY(h, cudaMemcpy(ids, h->s.ids, sizeof(int32_t) * n, cudaMemcpyDeviceToHost));
    if (gates) CUDA_TRY(h, cudaMemcpy(gates, h->s.gates, sizeof(float) * n, cudaMemcpyDeviceToHost));
    return MOE_OK;
}

moe_status moe_get_expert_counts(moe_handle* h, int32_t* counts, int32_t* offsets)
{
    moe_status r = getter_prologue(h);
    if (r != MOE_OK) return r;
    if (counts) CUDA_TRY(h, cudaMemcpy(counts, h->s.counts, sizeof(int32_t) * h->s.E, cudaMemcpyDeviceToHost));
    if (offsets)
        CUDA_TRY(h, cudaMemcpy(offsets, h->s.offsets, sizeof(int32_t) * (h->s.E + 1), cudaMemcpyDeviceToHost));
    return MOE_OK;
}

moe_status moe_get_permutation(moe_handle* h, int32_t* perm)
{
    moe_status r = getter_prologue(h);
    if (r != MOE_OK) return r;
    const int T = h->last_T;
    return with_tmp(h, sizeof(int32_t) * T * h->s.K, perm,
                    [&](void* d) { return launch_unpad_perm(h->s, T, static_cast<int32_t*>(d), 0); });
}

static moe_status get_quant(moe_handle* h, int which, uint8_t* q, uint8_t* sc)
{
    moe_status r = getter_prologue(h);
    if (r != MOE_OK) return r;
    if (sc && h->s.act_f32)
        return fail(h, MOE_ERR_INVALID_ARG,
                    "the handle keeps fp32 activation scales: pass scale = NULL and use the *_scales_f32 getter");
    const int T = h->last_T;
    const size_t rows = which == 0 ? (size_t)T : (size_t)T * h->s.K;
    const size_t width = which == 0 ? h->s.H : h->s.I;
    const size_t qb = rows * width, sb = rows * (width / 128);
    uint8_t *dq = nullptr, *ds = nullptr;
    CUDA_TRY(h, cudaMalloc(&dq, qb + sb + 256));
    ds = dq + qb;
    cudaError_t e = launch_gather_rows_u8(h->s, T, which, dq, ds, 0);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess && q) e = cudaMemcpy(q, dq, qb, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && sc) e = cudaMemcpy(sc, ds, sb, cudaMemcpyDeviceToHost);
    cudaFree(dq);
    if (e != cudaSuccess) return fail(h, MOE_ERR_CUDA, "getter: %s", cudaGetErrorString(e));
    return MOE_OK;
}

moe_status moe_get_act_quant(moe_handle* h, uint8_t* q, uint8_t* scale) { return get_quant(h, 0, q, scale); }

static moe_status get_scales_f32(moe_handle* h, int which, float* out)
{
    moe_status r = getter_prologue(h);
    if (r != MOE_OK) return r;
    const int T = h->last_T;
    const size_t rows = which == 0 ? (size_t)T : (size_t)T * h->s.K;
    const size_t width = which == 0 ? h->s.H : h->s.I;
    return with_tmp(h, sizeof(float) * rows * (width / 128), out,
                    [&](void* d) { return launch_gather_scales_f32(h->s, T, which, static_cast<float*>(d), 0); });
}

moe_status moe_get_act_scales_f32(moe_handle* h, float* scale) { return get_scales_f32(h, 0, scale); }
moe_status moe_get_inter_scales_f32(moe_handle* h, float* scale) { return get_scales_f32(h, 1, scale); }
moe_status moe_get_inter_quant(moe_handle* h, uint8_t* q, uint8_t* scale) { return get_quant(h, 1, q, scale); }

moe_status moe_get_expert_out(moe_handle* h, float* out)
{
    moe_status r = getter_prologue(h);
    if (r != MOE_OK) return r;
    const int T = h->last_T;
    return with_tmp(h, sizeof(float) * (size_t)T * h->s.K * h->s.H, out,
                    [&](void* d) { return launch_gather_obuf(h->s, T, static_cast<float*>(d), 0); });
}

moe_status moe_get_stage_times(moe_handle* h, float* ms, int n)
{
    if (!h || !ms) return fail(h, MOE_ERR_INVALID_ARG, "moe_get_stage_times: NULL argument");
    if (!h->profiling || !h->ev_valid || h->prof_count == 0)
        return fail(h, MOE_ERR_NOT_LOADED, "moe_get_stage_times: profiling off or no forward recorded");
    const int cnt = h->prof_count < kProfSlots ? h->prof_count : kProfSlots;
    const int last = (h->prof_count - 1) % kProfSlots;
    CUDA_TRY(h, cudaEventSynchronize(h->ev[last][kNumStages]));
    for (int i = 0; i < n && i < kNumStages; ++i) {
        double sum = 0.0;
        for (int k = 0; k < cnt; ++k) {
            const int slot = (h->prof_count - 1 - k) % kProfSlots;
            float t = 0.f;
            CUDA_TRY(h, cudaEventElapsedTime(&t, h->ev[slot][i], h->ev[slot][i + 1]));
            sum += t;
        }
        ms[i] = (float)(sum / cnt);
    }
    h->prof_count = 0;
    return MOE_OK;
}

}  // extern "C"
