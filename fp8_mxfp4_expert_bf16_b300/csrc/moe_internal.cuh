// Internal state shared by the host orchestration and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

constexpr int kBM = 128;            // rows per grouped-GEMM tile (tokens of one expert)
constexpr int kBK = 128;            // K elements per pipeline stage
constexpr int kChunk = 256;         // tokens per dispatch chunk
constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 8;
constexpr int kNumABox = 5;         // activation tile maps with 8 / 16 / 32 / 64 / 128 rows
constexpr int kWBlockRowsPerHalf = 136;   // interleaved weight block: 128 weight rows + 8 scale rows of 64 B
constexpr int kRouterMaxSplit = 16;       // split-K factor of the router for small batches
constexpr int kRouterSplitMaxT = 512;     // batches up to this size use the split-K router
constexpr int kRouterFusedMinT = 4096;    // batches from this size use the router with the top-k in its epilogue
constexpr int kLightRows = 16;      // m-tiles with at most this many rows use the light GEMM shape
constexpr int kMaxTp = 8;           // tensor-parallel shards of the expert middle dimension

// Error word codes written by kernels (first writer wins).
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrBounds = 2;

struct DevState {
    int H, I, E, K, Tm, score_func;
    int act_f32;         // activation blocks carry fp32 scales (amax / 448) instead of E8M0 ones
    int w_fp8 = 0;       // experts in the fp8 block format (e4m3 + fp32 scale per 128 x 128) instead of MXFP4
    int KB1, KB2;        // H/128, I/128: K-blocks of the two grouped GEMMs
    int NT1, NT2, BN2;   // n-tiles: G1 (I/128, 256 columns = gate 128 + up 128), G2 (H/BN2)
    int MTmax;           // max 128-row m-tiles: ceil(Tm*K/128) + E
    int Rmax;            // MTmax * 128 padded rows
    int nchunk_max;      // ceil(Tm / kChunk)

    // weights (owned)
    const uint16_t* wr = nullptr;   // [E][H] bf16
    const float* lb = nullptr;      // [E]
    const float* cb = nullptr;      // [E]
    // interleaved tile-major blocks [E][NT][KB] of halves * 136 rows x 64 B:
    // the stage's E2M1 weight rows (gate half, up half for w13), then its
    // scale chunks in tcgen05.cp order
    const uint8_t* w13q = nullptr;
    const uint8_t* w2q = nullptr;
    // fp8 block format: the fp32 block scales [E][R/128][K/128] of each projection
    const float* ws13 = nullptr;
    const float* ws2 = nullptr;

    // workspace
    float* logits;        // [Tm][E]
    float* logit_part;    // [kRouterMaxSplit][min(Tm, kRouterSplitMaxT)][E] split-K partial logits (small T)
    int32_t* ids;         // [Tm][K]
    float* gates;         // [Tm][K]
    int32_t* chunk_hist;  // [nchunk_max][E]
    int32_t* chunk_base;  // [nchunk_max][E]
    int32_t* counts;      // [E]
    int32_t* offsets;     // [E+1] unpadded exclusive scan
    int32_t* mtile_off;   // [E+1] exclusive scan of ceil(count/128)
    int32_t* mtile_expert;// [MTmax]
    int32_t* mtile_rows;  // [MTmax] valid rows of each m-tile (1..128)
    int32_t* n_mtiles;    // [4]: all m-tiles, light m-tiles (<= kLightRows valid rows), heavy m-tiles
    int32_t* light_list;  // [MTmax] m-tiles with at most kLightRows valid rows (light GEMM shape)
    int32_t* heavy_list;  // [MTmax] the other m-tiles (128-row GEMMs)
    int32_t* prow;        // [Tm*K] padded row of each (token, slot)
    uint8_t* aq;          // [Rmax][H]   e4m3 activations, expert-contiguous padded rows
    uint32_t* asf;        // [MTmax][KB1][128] scale words in tcgen05.cp order
    uint8_t* hq;          // [Rmax][I]   e4m3 SwiGLU output
    uint32_t* hsf;        // [MTmax][KB2][128]
    float* asf32;         // [Rmax][KB1] fp32 activation scales (fp32-scale mode only)
    float* hsf32;         // [Rmax][KB2] fp32 SwiGLU-output scales (fp32-scale mode only)
    float* obuf;          // [Rmax][H]   expert outputs (fp32)
    int32_t* err;         // [4] error word, where, aux

    // tensor maps (host copies, passed by value to the GEMM kernels)
    CUtensorMap tm_aq[kNumABox], tm_hq[kNumABox], tm_w13, tm_w2;
    CUtensorMap tm_wr64, tm_wr128;   // router weights, 64 / 128-row boxes
    int num_sms;
    bool pdl = true;     // launch the forward's kernels with programmatic stream serialisation
};

// Launch `kernel` on `st`; with `pdl` the launch may begin while the previous
// kernel on the stream is still running (the kernel itself waits, with
// griddep_wait, before it touches what that kernel writes).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                          Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Prefill-sized batches (on average at least 32 rows per expert): every heavy
// m-tile of the grouped GEMMs is loaded as a full 128-row activation box (its
// padding rows are zero in HBM, so the MMAs on them spend little energy; the
// GEMMs are bound by the power cap there).
__host__ __forceinline__ bool prefill_mode(const DevState& s, int T) { return (long long)T * s.K >= 32LL * s.E; }

// Word index of row r of m-tile mt, K-block kb, in a scale-factor buffer laid
// out for tcgen05.cp .32x128b.warpx4: per (mt, kb) 128 words, row r at word
// (r % 32) * 4 + r / 32; each word holds the 4 E8M0 bytes of the four
// 32-wide K sub-blocks.
__host__ __device__ __forceinline__ size_t sf_word_index(int mt, int kb, int KB, int r)
{
    return ((size_t)mt * KB + kb) * 128 + (size_t)(r & 31) * 4 + (r >> 5);
}

// launchers (route.cu)
cudaError_t launch_topk(const DevState& s, int T, cudaStream_t st, int ksplit = 1);
cudaError_t launch_dispatch_small(const DevState& s, int T, cudaStream_t st);
cudaError_t launch_quant_scatter(const DevState& s, const uint16_t* x, int T, cudaStream_t st);
cudaError_t launch_dispatch(const DevState& s, const uint16_t* x, int T, cudaStream_t st, int* nlaunch);
cudaError_t launch_combine(const DevState& s, uint16_t* y, int T, cudaStream_t st);
cudaError_t launch_combine_f32(const DevState& s, float* y32, int T, cudaStream_t st);
cudaError_t launch_sum_partials(const float* const* parts, int n_parts, size_t n, uint16_t* y, cudaStream_t st);
// load-time helpers (route.cu)
cudaError_t launch_repack_sf(const uint8_t* src, uint8_t* dst, int E, int KB, int NT, int halves, int rows_total,
                             int K32, int mode, int I128, cudaStream_t st);
cudaError_t launch_repack_w(const uint8_t* src, uint8_t* dst, int E, int KB, int NT, int halves, int rows_total,
                            int mode, int I128, cudaStream_t st);
cudaError_t launch_check_e8m0(const uint8_t* p, size_t n, int32_t* flag, cudaStream_t st);
cudaError_t launch_repack_w8(const uint8_t* src, uint8_t* dst, int E, int KB, int NT, int halves, int rows_total,
                             int mode, int I128, cudaStream_t st);
cudaError_t launch_check_fp8(const uint8_t* q, size_t n, const float* s, size_t ns, int32_t* flag, cudaStream_t st);
// getter helpers (route.cu)
cudaError_t launch_unpad_perm(const DevState& s, int T, int32_t* out, cudaStream_t st);
cudaError_t launch_gather_rows_u8(const DevState& s, int T, int which, uint8_t* q, uint8_t* sc, cudaStream_t st);
cudaError_t launch_gather_obuf(const DevState& s, int T, float* out, cudaStream_t st);
cudaError_t launch_gather_scales_f32(const DevState& s, int T, int which, float* out, cudaStream_t st);
// router on the tensor cores (router_gemm.cu)
cudaError_t launch_router_tc(const DevState& s, const CUtensorMap& tmX, int T, cudaStream_t st, int ksplit = 1);
int router_split(int T, int H);
cudaError_t router_set_attributes();
bool router_fused(int T, int E);
cudaError_t launch_router_topk(const DevState& s, const CUtensorMap& tmX, int T, cudaStream_t st);
// grouped GEMMs (mx_gemm.cu)
cudaError_t launch_gemm1(const DevState& s, cudaStream_t st, int T);
cudaError_t launch_gemm2(const DevState& s, cudaStream_t st, int T);
cudaError_t gemm_set_attributes();

}  // namespace moe
