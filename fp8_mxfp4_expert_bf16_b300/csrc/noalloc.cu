// Routing without any device allocation: the router logits live in a
// fixed-size array compiled into this library instead of a workspace from
// cudaMalloc.  Some callers cannot allocate device memory on the call path:
// code whose device memory is owned by its own allocator or budget, and
// latency-critical serving loops, where cudaMalloc / cudaFree may
// synchronise the device and stall work that is already in flight.  They
// pass every input and output buffer themselves and this entry point adds
// nothing to the device's allocations.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/moe_mx.h"
#include "moe_internal.cuh"

using namespace moe;

// Largest T * E the fixed scratch holds (router logits, fp32): 4 MiB.
constexpr size_t kNoAllocMaxLogits = size_t(1) << 20;
// Layout of the scratch (in floats): logits, then two zero bias vectors
// (used when a bias pointer is NULL), then a 4-word error record.
constexpr size_t kNoAllocZeroOff = kNoAllocMaxLogits;
constexpr size_t kNoAllocErrOff = kNoAllocZeroOff + 2 * kMaxExperts;
constexpr size_t kNoAllocWords = kNoAllocErrOff + 4;

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocWords];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
float* g_scratch_ptr[kMaxDevices] = {};   // device address of the scratch, per device

void set_error(const char* msg);

// Once per device, with that device current: look up the scratch's device
// address (host code cannot use the symbol itself) and set the router
// kernel's shared-memory limit.
moe_status setup_device(int dev, float** out)
{
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_ptr[dev]) {
        *out = g_scratch_ptr[dev];
        return MOE_OK;
    }
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
        char buf[256];
        snprintf(buf, sizeof buf, "moe_route_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
        set_error(buf);
        return MOE_ERR_CUDA;
    }
    e = router_set_attributes();
    if (e != cudaSuccess) {
        char buf[256];
        snprintf(buf, sizeof buf, "moe_route_noalloc: cudaFuncSetAttribute failed: %s", cudaGetErrorString(e));
        set_error(buf);
        return MOE_ERR_CUDA;
    }
    g_scratch_ptr[dev] = static_cast<float*>(p);
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
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

bool bf16_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// defined in api.cu: the message moe_last_error(NULL) returns
void moe_set_handle_free_error(const char* msg);

namespace {
void set_error(const char* msg) { moe_set_handle_free_error(msg); }
}

extern "C" moe_status moe_route_noalloc(const uint16_t* x, int T, int H, const uint16_t* router_w,
                                        const float* logit_bias, const float* sel_bias, int E, int k,
                                        int score_func, int32_t* ids, float* gates, void* stream)
{
    char buf[256];
    if (T < 0 || E < 1 || E > kMaxExperts || k < 1 || k > kMaxTopK || k > E || H < 64 || H % 64 ||
        (score_func != MOE_SCORE_SIGMOID && score_func != MOE_SCORE_SOFTMAX)) {
        snprintf(buf, sizeof buf, "moe_route_noalloc: bad shape T=%d H=%d E=%d k=%d score_func=%d", T, H, E, k,
                 score_func);
        set_error(buf);
        return MOE_ERR_SHAPE;
    }
    if ((size_t)T * (size_t)E > kNoAllocMaxLogits) {
        snprintf(buf, sizeof buf,
                 "moe_route_noalloc: T*E = %zu exceeds the fixed scratch of %zu router logits", (size_t)T * E,
                 kNoAllocMaxLogits);
        set_error(buf);
        return MOE_ERR_SHAPE;
    }
    if (T == 0) return MOE_OK;
    if (!x || !router_w || !ids || !gates) {
        set_error("moe_route_noalloc: x, router_w, ids and gates must not be NULL");
        return MOE_ERR_INVALID_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(router_w)) & 15u) {
        set_error("moe_route_noalloc: x and router_w must be 16-byte aligned");
        return MOE_ERR_INVALID_ARG;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        set_error("moe_route_noalloc: no current CUDA device");
        return MOE_ERR_CUDA;
    }
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) {
        set_error("moe_route_noalloc: the current device is not sm_103");
        return MOE_ERR_UNSUPPORTED;
    }
    float* scratch = nullptr;
    moe_status st = setup_device(dev, &scratch);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // the zero bias vectors must be zero (nothing writes them; cleared anyway);
    // the logits are fully overwritten by the router before top-k reads them.
    // The error record is left alone: a timeout of an earlier call stays
    // recorded until moe_route_noalloc_check_error reads and clears it.
    cudaError_t e = cudaMemsetAsync(scratch + kNoAllocZeroOff, 0, 2 * kMaxExperts * sizeof(float), s);

    DevState ds{};
    ds.pdl = false;   // plain stream order, as for any other library call on the caller's stream
    ds.H = H;
    ds.E = E;
    ds.K = k;
    ds.score_func = score_func;
    ds.wr = router_w;
    ds.lb = logit_bias ? logit_bias : scratch + kNoAllocZeroOff;
    ds.cb = sel_bias ? sel_bias : scratch + kNoAllocZeroOff + kMaxExperts;
    ds.logits = scratch;
    ds.ids = ids;
    ds.gates = gates;
    ds.err = reinterpret_cast<int32_t*>(scratch + kNoAllocErrOff);
    CUtensorMap tmX;
    if (!bf16_map(&tmX, x, (uint64_t)H, (uint64_t)T, 128) || !bf16_map(&ds.tm_wr64, router_w, H, E, 64) ||
        !bf16_map(&ds.tm_wr128, router_w, H, E, 128)) {
        set_error("moe_route_noalloc: cuTensorMapEncodeTiled failed");
        return MOE_ERR_CUDA;
    }
    if (e == cudaSuccess) e = launch_router_tc(ds, tmX, T, s);
    if (e == cudaSuccess) e = launch_topk(ds, T, s);
    if (e != cudaSuccess) {
        snprintf(buf, sizeof buf, "moe_route_noalloc: launch failed: %s", cudaGetErrorString(e));
        set_error(buf);
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

// The error record of the scratch on the current device (for the library's
// wait-timeout self-test, which can target it instead of a handle's).
moe_status noalloc_error_record(int32_t** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        set_error("no current CUDA device");
        return MOE_ERR_CUDA;
    }
    float* scratch = nullptr;
    moe_status st = setup_device(dev, &scratch);
    if (st == MOE_OK) *out = reinterpret_cast<int32_t*>(scratch + kNoAllocErrOff);
    return st;
}

extern "C" moe_status moe_route_noalloc_check_error(void* stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        set_error("moe_route_noalloc_check_error: no current CUDA device");
        return MOE_ERR_CUDA;
    }
    char buf[256];
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    int32_t w[3] = {0, 0, 0};
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(w, g_noalloc_scratch, sizeof w, kNoAllocErrOff * sizeof(float));
    if (e == cudaSuccess && w[0] != 0) {
        const int32_t zero[3] = {0, 0, 0};
        e = cudaMemcpyToSymbol(g_noalloc_scratch, zero, sizeof zero, kNoAllocErrOff * sizeof(float));
    }
    if (e != cudaSuccess) {
        snprintf(buf, sizeof buf, "moe_route_noalloc_check_error: %s", cudaGetErrorString(e));
        set_error(buf);
        return MOE_ERR_CUDA;
    }
    if (w[0] == 0) return MOE_OK;
    snprintf(buf, sizeof buf, "moe_route_noalloc: a kernel wait %s (site %d, block %d)",
             w[0] == kDevErrTimeout ? "timed out" : "reported an error", w[1], w[2]);
    set_error(buf);
    return w[0] == kDevErrTimeout ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE;
}
