// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05), with
// MXFP4 weights consumed natively by the block-scaled MMA and e4m3
// activations with power-of-two (E8M0) block scales.
//
// Layer definition: "MiMo V2.6 Pro and Flash architecture teardown", section
// "How Big Is Each Expert?" (gate, up and down projections around a
// 2,048-wide middle) and section "Why Are the V2.6 Files Half the Size of
// V2.5?" (MXFP4: E2M1 pairs per byte, one E8M0 scale per 32 values); vLLM
// recipe "XiaomiMiMo/MiMo-V2.6-Pro-RL", "Overview" (computed as block-wise
// FP8 e4m3).
//
// One persistent CTA per SM walks two static lists of (m-tile, n-tile)
// tiles: first the light m-tiles (at most 16 valid rows), then the heavy
// ones, each phase with the shared-memory ring shape that suits it.  An
// m-tile is 128 consecutive padded rows of one expert; an n-tile is 256
// weight rows (gate 128 + up 128 of one 128-wide slice of the expert's
// middle for the gate/up GEMM; 256 output features for the down GEMM).
// Warp roles:
//   warp 0      TMA producer: per 128-wide K step, the activation tile
//               (128 B rows, 128-byte swizzle), the weight tile (one
//               contiguous block of the tile-major weight layout; E2M1 codes
//               expanded by TMA into 16-byte groups, the operand format of
//               kind::mxf8f6f4) and both scale-factor chunks;
//   warp 1      TMEM owner and MMA issuer: copies the scale chunks into
//               TMEM (tcgen05.cp) and issues 4 block-scaled 128x256x32 MMAs
//               per stage into one fp32 accumulator in TMEM; the whole warp
//               runs the loop and one elected lane issues each operation;
//   warps 2-9   epilogue (two warps per TMEM lane quarter, each half of the
//               columns): TMEM -> registers; gate/up: h = silu(g) * u and
//               re-quantisation of h to e4m3 per 1 x 128 block (the two
//               warps of a row combine their amax through shared memory);
//               down: fp32 rows to the expert-output buffer.  The single
//               accumulator (TMEM also holds the scale chunks, so it cannot
//               be double-buffered) is released early by parking columns in
//               the TMEM columns the phase leaves free: the up half (gate/up)
//               or three of each warp's four column blocks (down, heavy).
// The promotion modes (fp32 activation scales, or fp8 experts with fp32
// block scales) cannot fold their scales into the MMA: each K-step's product
// lands in TMEM as a separate partial that the epilogue scales and adds in
// registers.  Heavy m-tiles use a ring of three 128-column partials (one per
// K-step and weight half); light m-tiles swap the operands, weights as the
// 128-row A operand and the 16 token rows as B, so that a partial is only 16
// columns wide and a ring unit carries four K-steps of both halves (see
// kSwN).
// Programmatic dependent launch: the kernel may start while the previous
// kernel of the forward (which writes the activations) is still running.
// Before waiting for it, the producer streams what does not depend on it:
// the weight tiles of the first ring stages.  Only then does it wait and
// load the activation tiles.
// All waits are bounded in time; a wait that gives up writes an error word,
// raises a CTA-wide abort flag, and the CTA drains its copies / MMAs and
// frees TMEM before exiting.
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

// The two ring shapes (one kernel runs both phases in turn):
//  heavy (m-tiles with more than kLightRows = 16 valid rows): 128-row
//    activation slot, 4-stage ring;
//  light (at most 16 valid rows: decode, and an expert's last m-tile): the
//    activation slot holds only the 16-row box (2 KB), which buys 6 stages;
//    these m-tiles put the token rows on the MMA's N side (see kSwN).
// With six stages in flight per SM (about 100 KB of weights) the weight
// stream needs no separate L2 prefetch; one measured on top of the ring
// slowed both GEMMs.
template <bool kLight>
struct Shape {
    static_assert(kLightRows == 16, "light ring shape");
    static constexpr int kStages = kLight ? 6 : 4;
    static constexpr int kABytes = kLight ? 16 * 128 : kBM * 128;
    static constexpr int kBOff = kABytes;
    static constexpr int kSFAOff = kBOff + 2 * 128 * 128;     // weight tile: 256 rows x 128 B (16-byte slots)
    static constexpr int kSFBOff = kSFAOff + 512;
    static constexpr int kStageStride = ((kSFBOff + 1024 + 1023) / 1024) * 1024;
    static constexpr int kRingBytes = kStages * kStageStride;
    // activation box heights of the phase's activation maps (light: two)
    static constexpr int kBox0 = kLight ? 8 : 32, kBox1 = kLight ? 16 : 64, kBox2 = kLight ? 16 : 128;
};
constexpr int kRingBytes =
    Shape<true>::kRingBytes > Shape<false>::kRingBytes ? Shape<true>::kRingBytes : Shape<false>::kRingBytes;

// A 128 x 128 E2M1 box occupies 16 KB of shared memory (each 8 bytes of
// packed codes followed by an 8-byte gap) but completes only the 8 KB it
// reads from global memory on the barrier's transaction count.
constexpr uint32_t kBHalfTxBytes = 128 * 64;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;      // accumulator: 256 fp32 columns
constexpr uint32_t kSFCol = 256;     // stage s: SFA at kSFCol + 16 s (4 cols), SFB at +8 (8 cols)
constexpr uint32_t kStashHeavyCol = 320;  // down epilogue, heavy phase: 3 x 32 columns per warp parked here
constexpr uint32_t kStashCol = 384;  // gate/up epilogue: the tile's up columns parked here (128 cols)
static_assert(kSFCol + 16 * Shape<false>::kStages <= kStashHeavyCol && kStashHeavyCol + 2 * 96 <= kTmemCols,
              "heavy-phase down stash overlaps the heavy ring's scale chunks");
static_assert(kSFCol + 16 * Shape<true>::kStages <= kStashCol && kStashCol + 128 <= kTmemCols,
              "gate/up stash overlaps the light ring's scale chunks");
// The promotion modes (fp32 activation scales, or fp8 experts with fp32
// block scales) lay TMEM out differently: a ring of kPBufs partial products
// of one 128-row half of a tile's weight rows and one K-step (128 fp32
// columns each), so that the MMAs of the next half-steps run while the
// epilogue folds the previous ones into its registers; then the stages'
// scale chunks and a constant unit chunk.
constexpr int kPBufs = 3;
constexpr uint32_t kPBufCol = 0;
constexpr uint32_t kPSFCol = kPBufCol + 128 * kPBufs;   // stage s: SFA at + 16 s (4 cols), SFB at + 8 (8 cols)
constexpr uint32_t kPUnitCol = kPSFCol + 16 * 6;        // E8M0 1.0 chunk, twice (8 cols)
static_assert(Shape<true>::kStages <= 6 && Shape<false>::kStages <= 6, "promotion-mode scale chunks");
static_assert(kPUnitCol + 8 <= kTmemCols, "promotion-mode TMEM layout");
// Light m-tiles (at most 16 valid rows) put the tokens on the MMA's N side:
// the weights are the 128-row A operand (one MMA group per 128-row half of
// the tile) and the 16 activation rows the B operand, so an MMA computes the
// 128 x 16 outputs that are used instead of 128 x 256 (a 128 x 16 x 32 MMA
// costs 39 cycles against 128 for 128 x 256 x 32, and 1/16 of the
// multiply-adds: in decode the 128 x 256 form kept the tensor pipe busy on
// rows it discarded and drove the chip to its power cap).  An accumulator is
// then 16 TMEM columns (tokens) by 128 lanes (weight rows):
//   E8M0 activations: one 32-column pair (both halves) per tile, a ring of
//     kSwTBufs tiles, read once at the tile's end;
//   promotion modes: one 16-column partial per (K-step, half), kSwG K-steps
//     of both halves per unit of a ring of kSwPBufs units, each partial
//     folded into registers with its fp32 scale(s).
constexpr int kSwN = 16;                 // MMA N: the light m-tile's rows
constexpr int kSwRingCols = 384;         // TMEM columns of the accumulator ring
constexpr int kSwTBufs = 8;
constexpr int kSwG = 4;                  // promotion: K-steps per ring unit (both halves, 32 columns each)
constexpr int kSwPBufs = kSwRingCols / (32 * kSwG);
constexpr uint32_t kSwBufCol = 0;
constexpr uint32_t kSwSFCol = kSwRingCols;   // stage s: weight scales (half 0, half 1) at + 16 s, + 4; activation scales at + 8
constexpr uint32_t kSwUnitCol = kSwSFCol + 16 * 6;   // E8M0 1.0 chunk (4 cols)
constexpr int kMaxPBufs = 8;            // barriers of the accumulator rings (all three kinds)
static_assert(kLightRows == kSwN, "light m-tile rows");
static_assert(kSwTBufs * 2 * kSwN <= (int)kSwSFCol && kSwPBufs * kSwG * 2 * kSwN <= (int)kSwSFCol,
              "light accumulator ring");
static_assert(kSwSFCol + 16 * Shape<true>::kStages <= kSwUnitCol && kSwUnitCol + 4 <= kTmemCols, "light TMEM layout");
static_assert(kPBufs <= kMaxPBufs && kSwPBufs <= kMaxPBufs && kSwTBufs <= kMaxPBufs, "accumulator ring barriers");
constexpr int kEpiWarps = 8;                       // two per TMEM lane quarter
constexpr int kThreads = 32 * (2 + kEpiWarps);     // TMA warp, MMA warp, epilogue warps

struct GemmArgs {
    const uint32_t* sfa;         // activation scale words [MT][KB][128]
    const int32_t* mtile_expert;
    const int32_t* mtile_rows;
    const int32_t* light_list;   // m-tiles of the light phase, and their number
    const int32_t* light_count;
    const int32_t* heavy_list;   // m-tiles of the heavy phase, and their number
    const int32_t* heavy_count;
    const uint8_t* wq;           // interleaved tile-major blocks [E][NT][KB]: halves*128 weight rows, halves*8 scale rows
    int KB;                      // K / 128
    int NT;                      // n-tiles per m-tile
    int halves;                  // n-tile width / 128 (2, or 1 for a 128-wide down GEMM tile)
    // gate/up epilogue
    uint8_t* hq;                 // [R][I] e4m3
    uint32_t* hsf;               // [MT][I/128][128]
    int I;
    // down epilogue
    float* obuf;                 // [R][H]
    int H;
    // fp32-scale mode: the activation rows' fp32 block scales [R][KB], and
    // (gate/up) the output table for the SwiGLU rows' scales [R][I/128]
    const float* as32;
    float* hs32;
    // fp8 expert format: the projection's fp32 block scales [E][R/128][KB]
    const float* ws;
    int early_trigger;           // let the next kernel be scheduled right after the wait (else at the end)
    int full_box;                // heavy phase: always the 128-row activation box (prefill-sized batches)
    int32_t* err;
};

template <int kStages>
struct PhaseCtl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full;
    uint64_t acc_empty;
    uint64_t drain;
    uint64_t red_full[2];
    uint64_t pfull[kMaxPBufs];    // accumulator ring (promotion partials, light tiles): buffer b is in TMEM
    uint64_t pempty[kMaxPBufs];   // every epilogue warp has read buffer b
    float red[2][8][32];          // per-warp row amax halves, double-buffered by tile parity
};

struct GemmCtl {
    uint32_t unit_sf[128];        // promotion modes: E8M0 1.0 in every byte (a tcgen05.cp chunk)
    PhaseCtl<Shape<true>::kStages> light;
    PhaseCtl<Shape<false>::kStages> heavy;
    uint32_t tmem_base;
    int abort;
};
constexpr int kSmemBytes = kRingBytes + (int)sizeof(GemmCtl) + 1024;   // + alignment of the ring to 1 KB
static_assert(kSmemBytes <= 232448, "shared memory");

__device__ __forceinline__ void raise_error(GemmCtl* g, int32_t* err, int where)
{
    if (atomicCAS(err, 0, kDevErrTimeout) == 0) {
        err[1] = where;
        err[2] = blockIdx.x;
    }
    *(volatile int*)&g->abort = 1;
}

template <int kStages>
__device__ __forceinline__ void init_phase(PhaseCtl<kStages>& pc)
{
    for (int s = 0; s < kStages; ++s) {
        mbar_init(smem_u32(&pc.full[s]), 1);
        mbar_init(smem_u32(&pc.empty[s]), 1);
    }
    mbar_init(smem_u32(&pc.acc_full), 1);
    mbar_init(smem_u32(&pc.acc_empty), kEpiWarps);
    mbar_init(smem_u32(&pc.red_full[0]), kEpiWarps);
    mbar_init(smem_u32(&pc.red_full[1]), kEpiWarps);
    mbar_init(smem_u32(&pc.drain), 1);
    for (int b = 0; b < kMaxPBufs; ++b) {
        mbar_init(smem_u32(&pc.pfull[b]), 1);
        mbar_init(smem_u32(&pc.pempty[b]), kEpiWarps);
    }
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d)
{
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

// smallest integer e with amax <= 448 * 2^e (clamped to [-127, 127]; 0 for
// an all-zero block), exactly from the binary exponent of amax
__device__ __forceinline__ int act_block_exponent(float amax)
{
    if (!(amax > 0.f)) return 0;
    int p;
    const float f = frexpf(amax, &p);
    const int e = (f <= 0.875f) ? p - 9 : p - 8;
    return max(-127, min(127, e));
}

// The producer's wait for the previous kernel of the forward (done once per
// CTA, before the first activation load).  Tile lists and weights are read
// before it: the lists come from the dispatch kernel, which had completed
// before the previous kernel passed its own wait and allowed this one to
// start.  A GEMM followed by another GEMM then lets it be scheduled at
// once (early_trigger), so that its CTAs take over SMs as this kernel's CTAs
// finish and stream their first weights meanwhile; the last GEMM lets its
// successor (the combine, which has nothing to do before its own wait) be
// scheduled only near the end of each CTA's work, so that waiting combine
// blocks do not sit beside running GEMM CTAs.
__device__ __forceinline__ void producer_wait_once(bool& waited, int early_trigger)
{
    if (!waited) {
        griddep_wait();
        if (early_trigger) griddep_launch_dependents();
        waited = true;
    }
}

// Down-GEMM epilogue of one warp, heavy m-tiles: kCols (64 or 128) fp32
// accumulator columns of its 32 TMEM lanes (rows), in blocks of 32 columns.
// Blocks 1.. are first copied to `stash` (TMEM columns outside the
// accumulator, through registers), block 0 is read, and the accumulator is
// released (arrive on `acc_empty`).  Each block is read with the 16-lane x
// 256-bit shape, which gives four neighbouring threads 8 consecutive columns
// of one row: every thread then stores 8-byte pieces, and each store
// instruction of the warp fills whole 32-byte sectors of 8 rows (no
// transposes across the warp).  dst0 is row 0 of the warp's 32 rows,
// `live_rows` how many of them are valid, rows `row_stride` floats apart.
template <int kCols>
__device__ __forceinline__ void store_rows_sectors(uint32_t taddr, uint32_t stash, int live_rows, float* dst0,
                                                   size_t row_stride, uint32_t acc_empty, int lane)
{
    if (live_rows > 0) {
#pragma unroll 1
        for (int b = 1; b < kCols / 32; ++b) {
            uint32_t a[32];
            tmem_ld32(taddr + 32u * b, a);
            tmem_ld_wait();
            tmem_st32(stash + 32u * (b - 1), a);
            tmem_st_wait();
        }
    }
    const int r0 = lane >> 2, c0 = 2 * (lane & 3);
#pragma unroll 1
    for (int b = 0; b < kCols / 32; ++b) {
        uint32_t lo[16], hi[16];   // rows 0..15, rows 16..31 of the block
        const uint32_t src = b == 0 ? taddr : stash + 32u * (b - 1);
        if (live_rows > 0) {
            tmem_ld_16x256b_x4(src, lo);
            tmem_ld_16x256b_x4(src + (16u << 16), hi);
            tmem_ld_wait();
        }
        if (b == 0) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
        }
        if (live_rows <= 0) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = 32 * b + 8 * j + c0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {   // rows r0, r0 + 8, r0 + 16, r0 + 24
                const int r = r0 + 8 * q;
                const uint32_t* v = q < 2 ? lo : hi;
                const int k = 4 * j + 2 * (q & 1);
                if (r < live_rows)
                    *reinterpret_cast<float2*>(dst0 + (size_t)r * row_stride + col) =
                        make_float2(__uint_as_float(v[k]), __uint_as_float(v[k + 1]));
            }
        }
    }
}

// The tiles one CTA works on in a phase: tiles blockIdx.x, + gridDim.x, ...
// of the phase's count * NT (m-tile, n-tile) tiles, m-tile-major.
struct TileSeq {
    int first, step, total, per_mt;
    __device__ __forceinline__ TileSeq(int count, int NT)
        : first((int)blockIdx.x), step((int)gridDim.x), total(count * NT), per_mt(NT)
    {
    }
    __device__ __forceinline__ int mt_index(int t) const { return t / per_mt; }
    __device__ __forceinline__ int nt_of(int t) const { return t - (t / per_mt) * per_mt; }
};

// 8-bit e4m3 code of one value (round to nearest even, saturating)
__device__ __forceinline__ uint32_t e4m3x1(float v)
{
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(v, 0.0f), __NV_SATFINITE, __NV_E4M3) & 0xFFu;
}

// v[sel] for a warp-uniform or per-lane index, without local memory
__device__ __forceinline__ float pick8(const float (&v)[8], int sel)
{
    float r = v[0];
#pragma unroll
    for (int j = 1; j < 8; ++j) r = sel == j ? v[j] : r;
    return r;
}

// MMA issuer of a light phase with the tokens on the N side (see kSwN).
template <int kMode, bool kF32S, bool kW8>
__device__ __forceinline__ void light_mma(uint8_t* smem, GemmCtl* g, PhaseCtl<Shape<true>::kStages>& pc,
                                          uint32_t tmem, const GemmArgs& args, const TileSeq& ts, int lane)
{
    using S = Shape<true>;
    constexpr int kStages = S::kStages, kStageStride = S::kStageStride;
    constexpr bool kPromo = kF32S || kW8;
    const volatile int* abrt = &g->abort;
    const int KB = args.KB, halves = args.halves;
    const uint32_t idesc = idesc_mxf8f6f4(128, kSwN, kW8 ? kTypeE4M3 : kTypeE2M1, kTypeE4M3);
    const uint32_t id1 = idesc_with_sf_id(idesc, 1, 1), id2 = idesc_with_sf_id(idesc, 2, 2),
                   id3 = idesc_with_sf_id(idesc, 3, 3);
    const uint32_t s0 = smem_u32(smem);
    const uint64_t wd0 = desc_kmajor_sw128(s0 + S::kBOff);   // weight rows: the A operand
    const uint64_t xd0 = desc_kmajor_sw128(s0);              // activation rows: the B operand
    const uint64_t sfw0 = desc_sf_chunk(s0 + S::kSFBOff), sfx0 = desc_sf_chunk(s0 + S::kSFAOff);
    const uint32_t full0 = smem_u32(&pc.full[0]), empty0 = smem_u32(&pc.empty[0]);
    if constexpr (kPromo) tmem_cp_32x128b_warpx4_elect(tmem + kSwUnitCol, desc_sf_chunk(smem_u32(g->unit_sf)));
    int s = 0;
    uint32_t ph = 0, doff = 0;
    int b = 0;             // accumulator ring position: partial (promotion) or tile (E8M0)
    uint32_t pph = 0;      // its fill count's parity
    bool wrapped = false;  // every buffer of the ring has been filled once
    bool ok = true;
    // take the ring's next buffer once the epilogue has read its previous contents
    auto acquire = [&](int nbufs, int where, int& idx) {
        if (wrapped && !__all_sync(~0u, mbar_wait(smem_u32(&pc.pempty[b]), pph ^ 1u, abrt))) {
            if (lane == 0) raise_error(g, args.err, where);
            return false;
        }
        idx = b;
        if (++b == nbufs) {
            b = 0;
            pph ^= 1u;
            wrapped = true;
        }
        return true;
    };
    for (int tile = ts.first; tile < ts.total && ok; tile += ts.step) {
        int ub = 0;   // this tile's (E8M0) or this unit's (promotion) accumulator buffer
        if constexpr (!kPromo) {
            if (!acquire(kSwTBufs, 13, ub)) break;
            tc_fence_after();
        }
        for (int kb = 0; kb < KB && ok; ++kb) {
            const int g_in = kPromo ? kb % kSwG : 0;   // K-step within the unit
            if (kPromo && g_in == 0) {
                if (!acquire(kSwPBufs, 15, ub)) {
                    ok = false;
                    break;
                }
            }
            if (!__all_sync(~0u, mbar_wait(full0 + 8u * s, ph, abrt))) {
                if (lane == 0) raise_error(g, args.err, 14);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sfw_t = tmem + kSwSFCol + 16u * s, sfx_t = sfw_t + 8u;
            if constexpr (!kW8) {
                tmem_cp_32x128b_warpx4_elect(sfw_t, sfw0 + doff);
                if (halves == 2) tmem_cp_32x128b_warpx4_elect(sfw_t + 4u, sfw0 + doff + (512 >> 4));
            }
            if constexpr (!kF32S) tmem_cp_32x128b_warpx4_elect(sfx_t, sfx0 + doff);
            const uint32_t sfb = kF32S ? tmem + kSwUnitCol : sfx_t;
            // promotion: the K-step's partials (one per half) in slot g_in of the
            // unit; E8M0: the tile's accumulator pair
            const uint32_t d0 = kPromo ? tmem + kSwBufCol + 2u * kSwN * (uint32_t)(kSwG * ub + g_in)
                                       : tmem + kSwBufCol + 2u * kSwN * (uint32_t)ub;
            for (int h = 0; h < halves; ++h) {
                // the half's 128 weight rows start 16 KB into the stage's weight tile
                const uint32_t d = d0 + (uint32_t)kSwN * (uint32_t)h;
                const uint32_t sfa = kW8 ? tmem + kSwUnitCol : sfw_t + 4u * (uint32_t)h;
                const uint64_t ad = wd0 + doff + (uint64_t)h * (16384 >> 4), bd = xd0 + doff;
                mma_mxf8f6f4_elect(d, ad, bd, idesc, sfa, sfb, (!kPromo && kb != 0) ? 1u : 0u);
                mma_mxf8f6f4_elect(d, ad + 2, bd + 2, id1, sfa, sfb, 1u);
                mma_mxf8f6f4_elect(d, ad + 4, bd + 4, id2, sfa, sfb, 1u);
                mma_mxf8f6f4_elect(d, ad + 6, bd + 6, id3, sfa, sfb, 1u);
            }
            if (kPromo && (g_in == kSwG - 1 || kb == KB - 1)) tc_commit_elect(smem_u32(&pc.pfull[ub]));
            tc_commit_elect(empty0 + 8u * s);
            if (++s == kStages) {
                s = 0;
                ph ^= 1u;
                doff = 0;
            } else {
                doff += kStageStride >> 4;
            }
        }
        if constexpr (!kPromo) {
            if (ok) tc_commit_elect(smem_u32(&pc.pfull[ub]));
        }
    }
    // all MMAs of this warp complete before the ring or TMEM is reused
    int zero = 0;
    tc_commit_elect(smem_u32(&pc.drain));
    if (!mbar_wait(smem_u32(&pc.drain), 0u, &zero) && lane == 0) raise_error(g, args.err, 5);
}

// Epilogue of a light phase with the tokens on the N side.  Warp (q, hw):
// weight rows 32q .. 32q+31 of each half (its TMEM lane quarter), tokens
// 8hw .. 8hw+7 (TMEM columns); acc[h][j] = output of weight row 32q + lane of
// half h for token 8hw + j.  Tokens at or past the m-tile's valid rows hold
// padding or stale shared memory (any bit pattern) and are never used.
template <int kMode, bool kF32S, bool kW8>
__device__ __forceinline__ void light_epilogue(GemmCtl* g, PhaseCtl<Shape<true>::kStages>& pc, uint32_t tmem,
                                               const GemmArgs& args, const int32_t* list, const TileSeq& ts,
                                               int warp, int lane)
{
    constexpr bool kPromo = kF32S || kW8;
    const volatile int* abrt = &g->abort;
    const int ew = warp - 2, q = warp & 3, hw = ew >> 2;
    const int KB = args.KB, halves = args.halves;
    const int tok0 = 8 * hw;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + kSwBufCol + (uint32_t)tok0;
    int b = 0;
    uint32_t pph = 0;
    auto ring_take = [&](int where) {
        if (!mbar_wait(smem_u32(&pc.pfull[b]), pph, abrt)) {
            raise_error(g, args.err, where);
            return false;
        }
        tc_fence_after();
        return true;
    };
    auto ring_release = [&](int nbufs) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&pc.pempty[b]));
        if (++b == nbufs) {
            b = 0;
            pph ^= 1u;
        }
    };
    // activation scales come from the previous kernel (quantisation, or the
    // gate/up GEMM): wait for it before the first read
    if (kF32S) griddep_wait();
    int tcount = 0;
    for (int tile = ts.first; tile < ts.total; tile += ts.step, ++tcount) {
        const int mt = list[ts.mt_index(tile)], nt = ts.nt_of(tile);
        const int rows = args.mtile_rows[mt];
        const bool warp_live = tok0 < rows;
        float acc[2][8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[0][j] = acc[1][j] = 0.0f;
        bool ok = true;
        if constexpr (kPromo) {
            // acc += s_token * s_weight_block * partial, in K order
            const float* wsa = nullptr;
            const float* wsb = nullptr;
            if constexpr (kW8) {
                const int e = args.mtile_expert[mt];
                const int RB = kMode == 0 ? 2 * (args.I / 128) : args.H / 128;
                const int rba = kMode == 0 ? nt : nt * halves;
                const int rbb = kMode == 0 ? args.I / 128 + nt : rba + (halves == 2 ? 1 : 0);
                wsa = args.ws + ((size_t)e * RB + rba) * KB;
                wsb = args.ws + ((size_t)e * RB + rbb) * KB;
            }
            const float* xs = kF32S ? args.as32 + (size_t)(mt * kBM + tok0) * KB : nullptr;
            for (int kb0 = 0; kb0 < KB && ok; kb0 += kSwG) {
                const int n_in = min(kSwG, KB - kb0);   // K-steps in this unit
                // the unit's scales: the tokens' fp32 activation scales and the
                // weight blocks' scales of its K-steps (loading them a unit ahead
                // measured no faster)
                float sx[kSwG][8], wa[kSwG], wb[kSwG];
#pragma unroll
                for (int gg = 0; gg < kSwG; ++gg) {
                    const int kb = kb0 + gg;
                    const bool in = gg < n_in;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        sx[gg][j] = (kF32S && in && tok0 + j < rows) ? xs[(size_t)j * KB + kb] : 1.0f;
                    wa[gg] = (kW8 && in) ? wsa[kb] : 1.0f;
                    wb[gg] = (kW8 && in) ? wsb[kb] : 1.0f;
                }
                if (!ring_take(16)) {
                    ok = false;
                    break;
                }
                if (warp_live) {
                    uint32_t pv[kSwG][2][8];
                    const uint32_t src = tl + 2u * kSwN * (uint32_t)(kSwG * b);
#pragma unroll
                    for (int gg = 0; gg < kSwG; ++gg) {
                        if (gg < n_in) {
                            tmem_ld8(src + 2u * kSwN * gg, pv[gg][0]);
                            if (halves == 2) tmem_ld8(src + 2u * kSwN * gg + kSwN, pv[gg][1]);
                        }
                    }
                    tmem_ld_wait();
                    // K order: K-step kb0 + gg, then the next
#pragma unroll
                    for (int gg = 0; gg < kSwG; ++gg) {
                        if (gg < n_in) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                acc[0][j] = fmaf(sx[gg][j] * wa[gg], __uint_as_float(pv[gg][0][j]), acc[0][j]);
                                if (halves == 2)
                                    acc[1][j] = fmaf(sx[gg][j] * wb[gg], __uint_as_float(pv[gg][1][j]), acc[1][j]);
                            }
                        }
                    }
                }
                ring_release(kSwPBufs);
            }
        } else {
            if (!ring_take(16)) break;
            if (warp_live) {
                uint32_t p0[8], p1[8];
                tmem_ld8(tl + 2u * kSwN * (uint32_t)b, p0);
                if (halves == 2) tmem_ld8(tl + 2u * kSwN * (uint32_t)b + kSwN, p1);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    acc[0][j] = __uint_as_float(p0[j]);
                    acc[1][j] = halves == 2 ? __uint_as_float(p1[j]) : 0.0f;
                }
            }
            ring_release(kSwTBufs);
        }
        if (!ok) break;
        const int i = 32 * q + lane;   // weight row within each half
        if constexpr (kMode == 0) {
            // h = silu(g) * u per token, then the token's 1 x 128 block of h
            // (this n-tile's 128 middle columns: 4 lane quarters x 32 lanes)
            // re-quantised to e4m3
            float hv[8], am[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const bool live = tok0 + j < rows;
                const float gf = live ? acc[0][j] : 0.0f;
                const float uf = live ? acc[1][j] : 0.0f;
                hv[j] = __fdividef(gf, 1.0f + __expf(-gf)) * uf;
                float m = fabsf(hv[j]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(~0u, m, o));
                am[j] = m;
            }
            const int p = tcount & 1;
            if (lane < 8) pc.red[p][ew][lane] = pick8(am, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&pc.red_full[p]));
            if (!mbar_wait(smem_u32(&pc.red_full[p]), (uint32_t)(tcount >> 1) & 1u, abrt)) {
                raise_error(g, args.err, 17);
                break;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                am[j] = fmaxf(fmaxf(pc.red[p][4 * hw][j], pc.red[p][4 * hw + 1][j]),
                              fmaxf(pc.red[p][4 * hw + 2][j], pc.red[p][4 * hw + 3][j]));
            uint8_t* hcol = args.hq + (size_t)(mt * kBM + tok0) * args.I + nt * 128 + i;
            if constexpr (!kF32S) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int ex = act_block_exponent(am[j]);
                    if (tok0 + j < rows) hcol[(size_t)j * args.I] = (uint8_t)e4m3x1(hv[j] * __int_as_float((127 - ex) << 23));
                }
                if (q == 0 && lane < 8 && tok0 + lane < rows)
                    args.hsf[sf_word_index(mt, nt, args.I / 128, tok0 + lane)] =
                        (uint32_t)(act_block_exponent(pick8(am, lane)) + 127) * 0x01010101u;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float s2 = __fdiv_rn(am[j], 448.0f);
                    if (tok0 + j < rows) hcol[(size_t)j * args.I] = (uint8_t)(am[j] > 0.0f ? e4m3x1(__fdiv_rn(hv[j], s2)) : 0u);
                }
                if (q == 0 && lane < 8 && tok0 + lane < rows)
                    args.hs32[(size_t)(mt * kBM + tok0 + lane) * (args.I / 128) + nt] = __fdiv_rn(pick8(am, lane), 448.0f);
            }
        } else {
            // fp32 expert-output rows: for each token, the warp's 32 lanes
            // store 32 consecutive features
            float* ocol = args.obuf + (size_t)(mt * kBM + tok0) * args.H + (size_t)nt * (128 * halves) + i;
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (h < halves) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (tok0 + j < rows) ocol[(size_t)j * args.H + 128 * h] = acc[h][j];
                }
        }
    }
}

// One phase (the light or the heavy m-tile list) of the grouped GEMM.  Every
// role drains its own work before returning: the producer waits until its
// copies have landed, the MMA issuer until its MMAs have completed, the
// epilogue has read its last accumulator.
template <int kMode, bool kLight, bool kF32S, bool kW8>
__device__ __forceinline__ void gemm_phase(uint8_t* smem, GemmCtl* g, PhaseCtl<Shape<kLight>::kStages>& pc,
                                           uint32_t tmem, const CUtensorMap* tmA0, const CUtensorMap* tmA1,
                                           const CUtensorMap* tmA2, const CUtensorMap* tmW, const GemmArgs& args,
                                           const int32_t* list, int count, bool& waited)
{
    using S = Shape<kLight>;
    constexpr int kStages = S::kStages, kStageStride = S::kStageStride;
    constexpr int kSFAOff = S::kSFAOff, kSFBOff = S::kSFBOff;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const volatile int* abrt = &g->abort;
    const int NT = args.NT, KB = args.KB;
    const TileSeq ts(count, NT);

    if (warp == 0) {
        if (lane == 0 && ts.first < ts.total) {
            // ------------------------------------------------ TMA producer
            uint32_t last_phase[kStages];
            bool issued[kStages];
            for (int s = 0; s < kStages; ++s) issued[s] = false, last_phase[s] = 0;
            // Tile metadata (m-tile, expert, valid rows) is loaded ahead so the
            // global-load latency never sits between two TMA issues.
            const int stride = ts.step;
            auto load_mt = [&](int tile) { return tile < ts.total ? list[ts.mt_index(tile)] : 0; };
            int it = 0, pre = 0;
            bool ok = true;
            int cur_mt = load_mt(ts.first);
            int cur_e = args.mtile_expert[cur_mt], cur_rows = args.mtile_rows[cur_mt];
            int nxt_mt = load_mt(ts.first + stride);
            for (int tile = ts.first; tile < ts.total && ok; tile += stride) {
                const int mt = cur_mt, nt = ts.nt_of(tile);
                const int e = cur_e;
                const int rows = cur_rows;
                cur_mt = nxt_mt;
                cur_e = args.mtile_expert[cur_mt];
                cur_rows = args.mtile_rows[cur_mt];
                nxt_mt = load_mt(tile + 2 * stride);
                // activation box: the smallest of the three heights that covers the
                // valid rows (prefill-sized batches: always the full 128-row box)
                const int sel = (!kLight && args.full_box) ? 2 : (rows <= S::kBox0 ? 0 : (rows <= S::kBox1 ? 1 : 2));
                const CUtensorMap* tA = sel == 0 ? tmA0 : (sel == 1 ? tmA1 : tmA2);
                const uint32_t a_bytes = (uint32_t)(sel == 0 ? S::kBox0 : (sel == 1 ? S::kBox1 : S::kBox2)) * 128u;
                auto load_a = [&](uint8_t* st, uint32_t fb, int kb) { tma_load_2d(smem_u32(st), tA, fb, kb * kBK, mt * kBM); };
                // weight bytes of a stage: E2M1 rows (8 KB per 128 rows) + their scale chunks,
                // or e4m3 rows (16 KB per 128 rows, block scales applied in the epilogue)
                const uint32_t tx = a_bytes +
                                    (kW8 ? (uint32_t)args.halves * 16384u : args.halves * (kBHalfTxBytes + 512)) +
                                    (kF32S ? 0u : 512u);
                constexpr int kRowsHalf = kW8 ? 128 : kWBlockRowsPerHalf;
                // first row of this tile's interleaved weight blocks
                const size_t wrow0 = ((size_t)(e * NT + nt) * KB) * args.halves * kRowsHalf;
                const uint32_t* sfa = args.sfa + (size_t)mt * KB * 128;
                if (!waited) {
                    // Before the wait: the weight tile and its scales for the
                    // first ring stages (free at the start of a phase), each
                    // barrier armed with the stage's full byte count.
                    pre = KB < kStages ? KB : kStages;
                    for (int kb = 0; kb < pre; ++kb) {
                        uint8_t* st = smem + kb * kStageStride;
                        const uint32_t fb = smem_u32(&pc.full[kb]);
                        mbar_arrive_expect_tx(fb, tx);
                        const size_t wrow = wrow0 + (size_t)kb * args.halves * kRowsHalf;
                        tma_load_2d(smem_u32(st + S::kBOff), tmW, fb, 0, (int)wrow);
                        if constexpr (!kW8)
                            bulk_load(smem_u32(st + kSFBOff), args.wq + (wrow + (size_t)args.halves * 128) * 64,
                                      args.halves * 512, fb);
                        issued[kb] = true;
                        last_phase[kb] = 0;
                    }
                    producer_wait_once(waited, args.early_trigger);
                    for (int kb = 0; kb < pre; ++kb) {
                        uint8_t* st = smem + kb * kStageStride;
                        const uint32_t fb = smem_u32(&pc.full[kb]);
                        load_a(st, fb, kb);
                        if constexpr (!kF32S) bulk_load(smem_u32(st + kSFAOff), sfa + (size_t)kb * 128, 512, fb);
                    }
                }
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    if (it < pre) continue;   // issued before the wait
                    const int s = it % kStages;
                    const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                    if (!mbar_wait(smem_u32(&pc.empty[s]), ph ^ 1u, abrt)) {
                        raise_error(g, args.err, 1);
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + s * kStageStride;
                    const uint32_t fb = smem_u32(&pc.full[s]);
                    mbar_arrive_expect_tx(fb, tx);
                    load_a(st, fb, kb);
                    // the stage's weight rows (both halves) are one box; its scale chunks follow them
                    const size_t wrow = wrow0 + (size_t)kb * args.halves * kRowsHalf;
                    tma_load_2d(smem_u32(st + S::kBOff), tmW, fb, 0, (int)wrow);
                    if constexpr (!kF32S) bulk_load(smem_u32(st + kSFAOff), sfa + (size_t)kb * 128, 512, fb);
                    if constexpr (!kW8)
                        bulk_load(smem_u32(st + kSFBOff), args.wq + (wrow + (size_t)args.halves * 128) * 64,
                                  args.halves * 512, fb);
                    issued[s] = true;
                    last_phase[s] = ph;
                }
            }
            // wait for every copy this thread started before the ring is reused
            int zero = 0;
            for (int s = 0; s < kStages; ++s)
                if (issued[s] && !mbar_wait(smem_u32(&pc.full[s]), last_phase[s], &zero))
                    raise_error(g, args.err, 2);
        }
    } else if (warp == 1 && kLight) {
        // light m-tiles: tokens on the MMA's N side
        if constexpr (kLight) light_mma<kMode, kF32S, kW8>(smem, g, pc, tmem, args, ts, lane);
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // The loops run on the whole warp (one elected lane issues each
        // tcgen05 operation), which keeps their control flow and descriptors
        // warp-uniform.  The tensor pipe holds only a few MMAs ahead, so the
        // issue path between two MMAs is kept to a handful of instructions
        // (the warp shares its SM sub-partition with two epilogue warps):
        // all descriptors of stage 0 are built once, a stage's are those
        // plus a fixed offset (the start-address field counts 16-byte units
        // and never carries: shared addresses stay below 2^18 bytes), and
        // the ring position is stepped, not divided out of a counter.
        {
            const uint32_t idesc = idesc_mxf8f6f4(128, 128 * args.halves, kTypeE4M3, kW8 ? kTypeE4M3 : kTypeE2M1);
            const uint32_t s0 = smem_u32(smem);
            const uint64_t ad0 = desc_kmajor_sw128(s0), bd0 = desc_kmajor_sw128(s0 + S::kBOff);
            const uint64_t sfad0 = desc_sf_chunk(s0 + kSFAOff), sfbd0 = desc_sf_chunk(s0 + kSFBOff);
            const uint32_t id1 = idesc_with_sf_id(idesc, 1, 1), id2 = idesc_with_sf_id(idesc, 2, 2),
                           id3 = idesc_with_sf_id(idesc, 3, 3);
            const uint32_t full0 = smem_u32(&pc.full[0]), empty0 = smem_u32(&pc.empty[0]);
            const uint32_t acc = tmem + kAccCol;
            const bool two = args.halves == 2;
            int s = 0, tcount = 0;
            uint32_t ph = 0, doff = 0;
            bool ok = true;
            auto advance = [&]() {
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                    doff = 0;
                } else {
                    doff += kStageStride >> 4;
                }
            };
            if constexpr (kF32S || kW8) {
                // One partial product per K-step and 128-row half of the
                // weight tile, into the next buffer of the partial ring, handed
                // to the epilogue, which folds the fp32 scales in (the rows'
                // activation scales and / or the weights' block scales; in the
                // MMA those are unit E8M0 chunks).  A buffer is refilled once
                // every epilogue warp has read its previous partial.
                const uint32_t idh = idesc_mxf8f6f4(128, 128, kTypeE4M3, kW8 ? kTypeE4M3 : kTypeE2M1);
                const uint32_t idh1 = idesc_with_sf_id(idh, 1, 1), idh2 = idesc_with_sf_id(idh, 2, 2),
                               idh3 = idesc_with_sf_id(idh, 3, 3);
                const uint64_t unit = desc_sf_chunk(smem_u32(g->unit_sf));
                tmem_cp_32x128b_warpx4_elect(tmem + kPUnitCol, unit);
                tmem_cp_32x128b_warpx4_elect(tmem + kPUnitCol + 4u, unit);
                int b = 0;            // partial buffer of the next half-step
                uint32_t pph = 0;     // its fill count's parity
                bool wrapped = false; // every buffer has been filled once
                for (int tile = ts.first; tile < ts.total && ok; tile += ts.step) {
                    for (int kb = 0; kb < KB && ok; ++kb) {
                        if (!__all_sync(~0u, mbar_wait(full0 + 8u * s, ph, abrt))) {
                            if (lane == 0) raise_error(g, args.err, 8);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        uint32_t sfa_t = tmem + kPUnitCol, sfb_t = tmem + kPUnitCol;
                        if constexpr (!kF32S) {
                            sfa_t = tmem + kPSFCol + 16u * s;
                            tmem_cp_32x128b_warpx4_elect(sfa_t, sfad0 + doff);
                        }
                        if constexpr (!kW8) {
                            sfb_t = tmem + kPSFCol + 16u * s + 8u;
                            tmem_cp_32x128b_warpx4_elect(sfb_t, sfbd0 + doff);
                            if (two) tmem_cp_32x128b_warpx4_elect(sfb_t + 4u, sfbd0 + doff + (512 >> 4));
                        }
                        for (int h = 0; h < args.halves; ++h) {
                            if (wrapped &&
                                !__all_sync(~0u, mbar_wait(smem_u32(&pc.pempty[b]), pph ^ 1u, abrt))) {
                                if (lane == 0) raise_error(g, args.err, 9);
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t pacc = tmem + kPBufCol + 128u * (uint32_t)b;
                            // the half's 128 weight rows start 16 KB into the stage's weight tile;
                            // its scale chunk is the half's 4 columns of the stage's SFB
                            const uint64_t ad = ad0 + doff, bd = bd0 + doff + (uint64_t)h * (16384 >> 4);
                            const uint32_t sfb_h = kW8 ? sfb_t : sfb_t + 4u * (uint32_t)h;
                            mma_mxf8f6f4_elect(pacc, ad, bd, idh, sfa_t, sfb_h, 0u);
                            mma_mxf8f6f4_elect(pacc, ad + 2, bd + 2, idh1, sfa_t, sfb_h, 1u);
                            mma_mxf8f6f4_elect(pacc, ad + 4, bd + 4, idh2, sfa_t, sfb_h, 1u);
                            mma_mxf8f6f4_elect(pacc, ad + 6, bd + 6, idh3, sfa_t, sfb_h, 1u);
                            tc_commit_elect(smem_u32(&pc.pfull[b]));
                            if (++b == kPBufs) {
                                b = 0;
                                pph ^= 1u;
                                wrapped = true;
                            }
                        }
                        if (!ok) break;
                        tc_commit_elect(empty0 + 8u * s);
                        advance();
                    }
                }
            } else {
                for (int tile = ts.first; tile < ts.total && ok; tile += ts.step, ++tcount) {
                    if (tcount > 0 &&
                        !__all_sync(~0u, mbar_wait(smem_u32(&pc.acc_empty), (uint32_t)(tcount - 1) & 1u, abrt))) {
                        if (lane == 0) raise_error(g, args.err, 3);
                        break;
                    }
                    tc_fence_after();
                    for (int kb = 0; kb < KB; ++kb) {
                        if (!__all_sync(~0u, mbar_wait(full0 + 8u * s, ph, abrt))) {
                            if (lane == 0) raise_error(g, args.err, 4);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sfa_t = tmem + kSFCol + 16u * s;
                        const uint64_t ad = ad0 + doff, bd = bd0 + doff;
                        tmem_cp_32x128b_warpx4_elect(sfa_t, sfad0 + doff);
                        tmem_cp_32x128b_warpx4_elect(sfa_t + 8u, sfbd0 + doff);
                        if (two) tmem_cp_32x128b_warpx4_elect(sfa_t + 12u, sfbd0 + doff + (512 >> 4));
                        mma_mxf8f6f4_elect(acc, ad, bd, idesc, sfa_t, sfa_t + 8u, kb != 0 ? 1u : 0u);
                        mma_mxf8f6f4_elect(acc, ad + 2, bd + 2, id1, sfa_t, sfa_t + 8u, 1u);
                        mma_mxf8f6f4_elect(acc, ad + 4, bd + 4, id2, sfa_t, sfa_t + 8u, 1u);
                        mma_mxf8f6f4_elect(acc, ad + 6, bd + 6, id3, sfa_t, sfa_t + 8u, 1u);
                        tc_commit_elect(empty0 + 8u * s);
                        advance();
                    }
                    if (ok) tc_commit_elect(smem_u32(&pc.acc_full));
                }
            }
            // all MMAs of this warp complete before the ring or TMEM is reused
            int zero = 0;
            tc_commit_elect(smem_u32(&pc.drain));
            if (!mbar_wait(smem_u32(&pc.drain), 0u, &zero) && lane == 0) raise_error(g, args.err, 5);
        }
    } else if (kLight) {
        if constexpr (kLight) light_epilogue<kMode, kF32S, kW8>(g, pc, tmem, args, list, ts, warp, lane);
    } else {
        // ---------------------------------------------------- epilogue
        // Eight warps, two per TMEM lane quarter: warp pair (q, q + 4) shares
        // rows 32q .. 32q+31 and splits the columns, which halves the time the
        // accumulator is held before the next tile's MMAs may start.
        const int ew = warp - 2;                      // 0..7
        const int q = warp & 3;                       // this warp's TMEM lane quarter
        const int hw = ew >> 2;                       // which half of the columns
        const int row = q * 32 + lane;
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
        int tcount = 0;
        if constexpr (kF32S || kW8) {
            // promotion modes: per K-step and weight half, this warp's 64
            // partial columns of that half are read from TMEM and folded into
            // fp32 registers, acc += s * partial in K order, s = the row's
            // fp32 activation scale and / or the fp32 scale of the weight
            // block the half belongs to; warps without live rows still take
            // part in each hand-off.  Gate/up: acc[0, 64) = gate columns
            // [64 hw, +64) of the n-tile, acc[64, 128) the same up columns;
            // down: acc[64 h + j] = output feature 128 h + 64 hw + j of the
            // tile.
            constexpr int kW = 128;
            int b = 0;            // partial buffer of the next half-step
            uint32_t pph = 0;     // its fill count's parity
            // activation scales come from the previous kernel (quantisation,
            // or the gate/up GEMM): wait for it before the first read
            if (kF32S) griddep_wait();
            for (int tile = ts.first; tile < ts.total; tile += ts.step, ++tcount) {
                const int mt = list[ts.mt_index(tile)], nt = ts.nt_of(tile);
                const int rows = args.mtile_rows[mt];
                const bool warp_live = q * 32 < rows;
                const bool row_live = row < rows;
                const int halves = args.halves;
                const uint32_t c0 = 64u * (uint32_t)hw;   // this warp's columns within each half
                const float* srow = kF32S ? args.as32 + (size_t)(mt * kBM + row) * KB : nullptr;
                // weight blocks of the two halves: gate / up rows of the n-tile
                // (gate/up), or the tile's 128-feature blocks (down)
                const float* wsa = nullptr;
                const float* wsb = nullptr;
                if constexpr (kW8) {
                    const int e = args.mtile_expert[mt];
                    const int RB = kMode == 0 ? 2 * (args.I / 128) : args.H / 128;
                    const int rba = kMode == 0 ? nt : nt * halves;
                    const int rbb = kMode == 0 ? args.I / 128 + nt : rba + (halves == 2 ? 1 : 0);
                    wsa = args.ws + ((size_t)e * RB + rba) * KB;
                    wsb = args.ws + ((size_t)e * RB + rbb) * KB;
                }
                float acc[kW];
#pragma unroll
                for (int j = 0; j < kW; ++j) acc[j] = 0.0f;
                float s_next = kF32S ? (row_live ? srow[0] : 0.0f) : 1.0f;
                float wa_next = kW8 ? wsa[0] : 1.0f, wb_next = kW8 ? wsb[0] : 1.0f;
                bool ok = true;
                for (int kb = 0; kb < KB && ok; ++kb) {
                    const float sc_a = s_next * wa_next, sc_b = s_next * wb_next;
                    if (kb + 1 < KB) {
                        if constexpr (kF32S) s_next = row_live ? srow[kb + 1] : 0.0f;
                        if constexpr (kW8) {
                            wa_next = wsa[kb + 1];
                            wb_next = wsb[kb + 1];
                        }
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h < halves) {
                            if (!mbar_wait(smem_u32(&pc.pfull[b]), pph, abrt)) {
                                raise_error(g, args.err, 10);
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            if (warp_live) {
                                const float sc = h == 0 ? sc_a : sc_b;
                                const uint32_t src = tl + kPBufCol + 128u * (uint32_t)b + c0;
#pragma unroll
                                for (int c = 0; c < 2; ++c) {
                                    uint32_t pv[32];
                                    tmem_ld32(src + 32u * c, pv);
                                    tmem_ld_wait();
#pragma unroll
                                    for (int j = 0; j < 32; ++j)
                                        acc[64 * h + 32 * c + j] = fmaf(sc, __uint_as_float(pv[j]), acc[64 * h + 32 * c + j]);
                                }
                            }
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(smem_u32(&pc.pempty[b]));
                            if (++b == kPBufs) {
                                b = 0;
                                pph ^= 1u;
                            }
                        }
                    }
                }
                if (!ok) break;
                if (kMode == 0 && !kF32S) {
                    // h = silu(g) * u on the promoted sums, then the power-of-two
                    // re-quantisation of the row's 128-wide block
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        const float gf = row_live ? acc[j] : 0.0f;
                        const float uf = row_live ? acc[64 + j] : 0.0f;
                        acc[j] = __fdividef(gf, 1.0f + __expf(-gf)) * uf;
                    }
                    float amax = 0.f;
#pragma unroll
                    for (int j = 0; j < 64; ++j) amax = fmaxf(amax, fabsf(acc[j]));
                    const int p = tcount & 1;
                    pc.red[p][ew][lane] = amax;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&pc.red_full[p]));
                    if (!mbar_wait(smem_u32(&pc.red_full[p]), (uint32_t)(tcount >> 1) & 1u, abrt)) {
                        raise_error(g, args.err, 12);
                        break;
                    }
                    amax = fmaxf(amax, pc.red[p][ew ^ 4][lane]);
                    if (row_live) {
                        const int ex = act_block_exponent(amax);
                        const float inv = __int_as_float((127 - ex) << 23);
                        uint4* dst =
                            reinterpret_cast<uint4*>(args.hq + (size_t)(mt * kBM + row) * args.I + nt * 128 + 64 * hw);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const float* hv = acc + 16 * v;
                            uint4 w;
                            w.x = e4m3x4(hv[0] * inv, hv[1] * inv, hv[2] * inv, hv[3] * inv);
                            w.y = e4m3x4(hv[4] * inv, hv[5] * inv, hv[6] * inv, hv[7] * inv);
                            w.z = e4m3x4(hv[8] * inv, hv[9] * inv, hv[10] * inv, hv[11] * inv);
                            w.w = e4m3x4(hv[12] * inv, hv[13] * inv, hv[14] * inv, hv[15] * inv);
                            dst[v] = w;
                        }
                        if (hw == 0)
                            args.hsf[sf_word_index(mt, nt, args.I / 128, row)] = (uint32_t)(ex + 127) * 0x01010101u;
                    }
                } else if (kMode == 0) {
                    // h = silu(g) * u on the promoted sums, then the fp32-scale
                    // re-quantisation of the row's 128-wide block
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        const float gf = row_live ? acc[j] : 0.0f;
                        const float uf = row_live ? acc[64 + j] : 0.0f;
                        acc[j] = __fdividef(gf, 1.0f + __expf(-gf)) * uf;
                    }
                    float amax = 0.f;
#pragma unroll
                    for (int j = 0; j < 64; ++j) amax = fmaxf(amax, fabsf(acc[j]));
                    const int p = tcount & 1;
                    pc.red[p][ew][lane] = amax;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&pc.red_full[p]));
                    if (!mbar_wait(smem_u32(&pc.red_full[p]), (uint32_t)(tcount >> 1) & 1u, abrt)) {
                        raise_error(g, args.err, 11);
                        break;
                    }
                    amax = fmaxf(amax, pc.red[p][ew ^ 4][lane]);
                    if (row_live) {
                        const float s2 = __fdiv_rn(amax, 448.0f);
                        uint4* dst =
                            reinterpret_cast<uint4*>(args.hq + (size_t)(mt * kBM + row) * args.I + nt * 128 + 64 * hw);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint32_t w4[4];
#pragma unroll
                            for (int w = 0; w < 4; ++w) {
                                const float* hv = acc + 16 * v + 4 * w;
                                w4[w] = amax > 0.0f ? e4m3x4(__fdiv_rn(hv[0], s2), __fdiv_rn(hv[1], s2),
                                                             __fdiv_rn(hv[2], s2), __fdiv_rn(hv[3], s2))
                                                    : 0u;
                            }
                            dst[v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                        if (hw == 0) args.hs32[(size_t)(mt * kBM + row) * (args.I / 128) + nt] = s2;
                    }
                } else if (row_live) {
                    float* orow = args.obuf + (size_t)(mt * kBM + row) * args.H + (size_t)nt * (128 * halves) + c0;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h < halves) {
                            float4* d4 = reinterpret_cast<float4*>(orow + 128 * h);
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                d4[j] = make_float4(acc[64 * h + 4 * j], acc[64 * h + 4 * j + 1],
                                                    acc[64 * h + 4 * j + 2], acc[64 * h + 4 * j + 3]);
                        }
                    }
                }
            }
        } else
        for (int tile = ts.first; tile < ts.total; tile += ts.step, ++tcount) {
            const int mt = list[ts.mt_index(tile)], nt = ts.nt_of(tile);
            const int rows = args.mtile_rows[mt];
            if (!mbar_wait(smem_u32(&pc.acc_full), (uint32_t)tcount & 1u, abrt)) {
                raise_error(g, args.err, 6);
                break;
            }
            tc_fence_after();
            // Rows at or past `rows` hold padding or stale shared memory (any bit
            // pattern): no arithmetic touches them, and a warp whose 32 rows are
            // all invalid skips its TMEM loads entirely.
            const bool warp_live = q * 32 < rows;
            const bool row_live = row < rows;
            if (kMode == 0) {
                static_assert(!(kF32S || kW8), "the gate/up stash is for the E8M0 epilogue only");
                // this warp: middle columns [64 hw, 64 hw + 64) of the tile's 128
                float h[64];
                const uint32_t stash = tl + kStashCol + 64u * hw;
                if (warp_live) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t gg[16], u[16];
                        tmem_ld16(tl + kAccCol + 64u * hw + 16u * c, gg);
                        tmem_ld16(tl + kAccCol + 128u + 64u * hw + 16u * c, u);
                        tmem_ld_wait();
                        tmem_st16(stash + 16u * c, u);
#pragma unroll
                        for (int j = 0; j < 16; ++j) h[16 * c + j] = __uint_as_float(gg[j]);
                        tmem_st_wait();
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&pc.acc_empty));
                if (warp_live) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t u[16];
                        tmem_ld16(stash + 16u * c, u);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float gf = row_live ? h[16 * c + j] : 0.0f;
                            const float uf = row_live ? __uint_as_float(u[j]) : 0.0f;
                            h[16 * c + j] = __fdividef(gf, 1.0f + __expf(-gf)) * uf;
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) h[j] = 0.0f;
                }
                // the row's amax over all 128 columns: combine with the partner warp
                float amax = 0.f;
#pragma unroll
                for (int j = 0; j < 64; ++j) amax = fmaxf(amax, fabsf(h[j]));
                const int p = tcount & 1;
                pc.red[p][ew][lane] = amax;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&pc.red_full[p]));
                if (!mbar_wait(smem_u32(&pc.red_full[p]), (uint32_t)(tcount >> 1) & 1u, abrt)) {
                    raise_error(g, args.err, 7);
                    break;
                }
                amax = fmaxf(amax, pc.red[p][ew ^ 4][lane]);
                if (row_live) {
                    const int ex = act_block_exponent(amax);
                    const float inv = __int_as_float((127 - ex) << 23);
                    uint4* dst =
                        reinterpret_cast<uint4*>(args.hq + (size_t)(mt * kBM + row) * args.I + nt * 128 + 64 * hw);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = e4m3x4(h[16 * v + 0] * inv, h[16 * v + 1] * inv, h[16 * v + 2] * inv, h[16 * v + 3] * inv);
                        w.y = e4m3x4(h[16 * v + 4] * inv, h[16 * v + 5] * inv, h[16 * v + 6] * inv, h[16 * v + 7] * inv);
                        w.z = e4m3x4(h[16 * v + 8] * inv, h[16 * v + 9] * inv, h[16 * v + 10] * inv, h[16 * v + 11] * inv);
                        w.w = e4m3x4(h[16 * v + 12] * inv, h[16 * v + 13] * inv, h[16 * v + 14] * inv, h[16 * v + 15] * inv);
                        dst[v] = w;
                    }
                    if (hw == 0)
                        args.hsf[sf_word_index(mt, nt, args.I / 128, row)] = (uint32_t)(ex + 127) * 0x01010101u;
                }
            } else {
                static_assert(!(kF32S || kW8), "the heavy down stash is for the E8M0 epilogue only");
                // this warp: output columns [hw * ncols / 2, (hw + 1) * ncols / 2).  The
                // whole slice is read into registers first and the accumulator released,
                // so the next tile's MMAs run while the rows are stored.
                const int ncols = 128 * args.halves, half_cols = ncols / 2;
                float* dst0 =
                    args.obuf + (size_t)(mt * kBM + q * 32) * args.H + (size_t)nt * ncols + hw * half_cols;
                const int live = warp_live ? min(32, rows - q * 32) : 0;
                const uint32_t taddr = tl + kAccCol + (uint32_t)(hw * half_cols);
                if (half_cols == 128)
                    store_rows_sectors<128>(taddr, tl + kStashHeavyCol + 96u * hw, live, dst0, (size_t)args.H,
                                            smem_u32(&pc.acc_empty), lane);
                else
                    store_rows_sectors<64>(taddr, tl + kStashHeavyCol + 96u * hw, live, dst0, (size_t)args.H,
                                           smem_u32(&pc.acc_empty), lane);
            }
        }
    }
}

// mode 0: gate/up + SwiGLU + e4m3 requant, 1: down -> fp32 rows; kF32S: the
// activation blocks carry fp32 scales, kW8: the experts are e4m3 with fp32
// 128 x 128 block scales (either one: promotion in the epilogue)
template <int kMode, bool kF32S, bool kW8>
__global__ void __launch_bounds__(kThreads, 1)
    k_mx_gemm(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
              const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmA3,
              const __grid_constant__ CUtensorMap tmA4, const __grid_constant__ CUtensorMap tmW, const GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    GemmCtl* g = reinterpret_cast<GemmCtl*>(smem + kRingBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (kF32S || kW8) {
        for (int i = threadIdx.x; i < 128; i += blockDim.x) g->unit_sf[i] = 0x7F7F7F7Fu;   // E8M0 1.0
        fence_proxy_async_smem();   // generic-proxy writes above, read by tcgen05.cp
    }
    if (threadIdx.x == 0) {
        init_phase(g->light);
        init_phase(g->heavy);
        g->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA0);
        tma_prefetch_desc(&tmA1);
        tma_prefetch_desc(&tmA2);
        tma_prefetch_desc(&tmA3);
        tma_prefetch_desc(&tmA4);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&g->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = g->tmem_base;
    bool waited = false;   // the producer's wait for the previous kernel (producer thread only)

    gemm_phase<kMode, true, kF32S, kW8>(smem, g, g->light, tmem, &tmA0, &tmA1, &tmA1, &tmW, args, args.light_list,
                                        *args.light_count, waited);
    // the heavy phase reuses the ring and the accumulator: every role of the
    // light phase has drained its own work
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!*(volatile int*)&g->abort)
        gemm_phase<kMode, false, kF32S, kW8>(smem, g, g->heavy, tmem, &tmA2, &tmA3, &tmA4, &tmW, args,
                                             args.heavy_list, *args.heavy_count, waited);
    // a CTA without tiles still waits before it lets the next kernel start
    if (warp == 0 && lane == 0) {
        producer_wait_once(waited, args.early_trigger);
        griddep_launch_dependents();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

cudaError_t gemm_set_attributes()
{
    const void* ks[] = {(const void*)k_mx_gemm<0, false, false>, (const void*)k_mx_gemm<1, false, false>,
                        (const void*)k_mx_gemm<0, true, false>,  (const void*)k_mx_gemm<1, true, false>,
                        (const void*)k_mx_gemm<0, false, true>,  (const void*)k_mx_gemm<1, false, true>,
                        (const void*)k_mx_gemm<0, true, true>,   (const void*)k_mx_gemm<1, true, true>};
    cudaError_t e = cudaSuccess;
    for (const void* k : ks)
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    return e;
}

static GemmArgs common_args(const DevState& s)
{
    GemmArgs a{};
    a.mtile_expert = s.mtile_expert;
    a.mtile_rows = s.mtile_rows;
    a.light_list = s.light_list;
    a.light_count = s.n_mtiles + 1;
    a.heavy_list = s.heavy_list;
    a.heavy_count = s.n_mtiles + 2;
    a.err = s.err;
    return a;
}

static GemmArgs gemm1_args(const DevState& s)
{
    GemmArgs a = common_args(s);
    a.sfa = s.asf;
    a.wq = s.w13q;
    a.KB = s.KB1;
    a.NT = s.NT1;
    a.halves = 2;
    a.hq = s.hq;
    a.hsf = s.hsf;
    a.I = s.I;
    return a;
}

static GemmArgs gemm2_args(const DevState& s)
{
    GemmArgs a = common_args(s);
    a.sfa = s.hsf;
    a.wq = s.w2q;
    a.KB = s.KB2;
    a.NT = s.NT2;
    a.halves = s.BN2 / 128;
    a.obuf = s.obuf;
    a.H = s.H;
    return a;
}

template <int kMode, bool kF32S, bool kW8>
static cudaError_t launch_variant(const DevState& s, cudaStream_t st, const GemmArgs& a, const CUtensorMap* tA,
                                  const CUtensorMap& tW)
{
    return launch_kernel(k_mx_gemm<kMode, kF32S, kW8>, dim3(s.num_sms), dim3(kThreads), kSmemBytes, st, s.pdl, tA[0],
                         tA[1], tA[2], tA[3], tA[4], tW, a);
}

template <int kMode>
static cudaError_t launch_mode(const DevState& s, cudaStream_t st, const GemmArgs& a, const CUtensorMap* tA,
                               const CUtensorMap& tW)
{
    if (s.w_fp8) {
        return s.act_f32 ? launch_variant<kMode, true, true>(s, st, a, tA, tW)
                         : launch_variant<kMode, false, true>(s, st, a, tA, tW);
    }
    return s.act_f32 ? launch_variant<kMode, true, false>(s, st, a, tA, tW)
                     : launch_variant<kMode, false, false>(s, st, a, tA, tW);
}

// Light m-tiles (activation boxes of 8 / 16 rows: maps 0, 1), then heavy
// m-tiles (32 / 64 / 128 rows: maps 2..4), in one launch.
cudaError_t launch_gemm1(const DevState& s, cudaStream_t st, int T)
{
    GemmArgs a = gemm1_args(s);
    a.early_trigger = 1;   // the down GEMM follows
    a.full_box = prefill_mode(s, T) ? 1 : 0;
    a.as32 = s.asf32;
    a.hs32 = s.hsf32;
    a.ws = s.ws13;
    return launch_mode<0>(s, st, a, s.tm_aq, s.tm_w13);
}

cudaError_t launch_gemm2(const DevState& s, cudaStream_t st, int T)
{
    GemmArgs a = gemm2_args(s);
    a.early_trigger = 0;   // the combine follows
    a.full_box = prefill_mode(s, T) ? 1 : 0;
    a.as32 = s.hsf32;
    a.ws = s.ws2;
    return launch_mode<1>(s, st, a, s.tm_hq, s.tm_w2);
}

}  // namespace moe
