/*
 * moe_mx.h — C ABI of a single-GPU (sm_103a) routed Mixture-of-Experts
 * feed-forward layer whose expert weights are stored as MXFP4 and computed
 * against block-scaled FP8 (e4m3) activations.
 *
 * What the layer computes (web pages on MiMo-V2.6):
 *  - "MiMo V2.6 Pro and Flash architecture teardown" (kgptalkie), section
 *    "How Big Is Each Expert?": a router scores the experts with a sigmoid
 *    plus a per-expert correction bias, 8 experts per token, each expert a
 *    gate / up / down projection around a 2,048-wide middle; section "How Is
 *    the Backbone Built?": no shared expert; section "Why Are the V2.6 Files
 *    Half the Size of V2.5?": experts in MXFP4 (two E2M1 values per byte, one
 *    E8M0 scale per 32 values), router weights in BF16.
 *  - vLLM recipe "XiaomiMiMo/MiMo-V2.6-Pro-RL", section "Overview": 384
 *    routed experts, top-8; weights stored as mxfp4 and computed as
 *    block-wise FP8 e4m3.
 *  - devupai "MiMo-V2.6-Flash", section "Self-Hosting": a dynamic
 *    activation scheme.
 *
 * Per token t (H = hidden, I = expert width, E = experts, k = top-k):
 *   logits = x[t] . Wr^T + logit_bias                      (fp32)
 *   s = sigmoid(logits) (or softmax),  key = s + sel_bias
 *   ids = top-k of key (descending, ties to the lower index)
 *   gates = s[ids] / sum(s[ids])
 *   a = e4m3 quantisation of x[t], one power-of-two scale per 1 x 128 block
 *   for each selected expert e:
 *       [g | u] = a . W13[e]^T      (W13 [2I][H]: gate rows, then up rows)
 *       h = silu(g) * u,  re-quantised to e4m3 per 1 x 128 block
 *       o = h . W2[e]^T             (W2 [H][I])
 *   y[t] = bf16( sum_j gates[j] * o_j )   (fp32 accumulation)
 *
 * Conventions for every entry point:
 *  - Returns a moe_status; MOE_OK is 0.  On failure moe_last_error() gives a
 *    one-line reason (a handle-less failure is reported through the NULL
 *    handle, moe_last_error(NULL)).
 *  - "device" pointers are CUDA device memory of the handle's device;
 *    "host" pointers are ordinary (pageable or pinned) host memory.  Where
 *    either is accepted this is said.
 *  - The caller keeps ownership of every buffer it passes; the library keeps
 *    ownership of its weights copy and its workspace until moe_destroy.
 *  - bf16 values are passed as 16-bit patterns (uint16_t).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *  - A handle is not thread-safe: calls on one handle must not overlap.
 */
#ifndef MOE_MX_H
#define MOE_MX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* NULL pointer, bad enum, bad value (e.g. a NaN E8M0 byte) */
    MOE_ERR_SHAPE = 2,        /* a dimension outside the supported set */
    MOE_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
    MOE_ERR_OOM = 4,          /* device allocation failed */
    MOE_ERR_NOT_LOADED = 5,   /* forward before moe_load_weights, or getter before forward */
    MOE_ERR_TIMEOUT = 6,      /* a kernel's bounded wait gave up (reported by a later call) */
    MOE_ERR_UNSUPPORTED = 7,  /* device is not sm_103 / feature not built */
    MOE_ERR_DEVICE = 8        /* a kernel reported an internal consistency error */
} moe_status;

typedef struct moe_handle moe_handle;

enum { MOE_SCORE_SIGMOID = 0, MOE_SCORE_SOFTMAX = 1 };

/* Activation scale of the 1 x 128 e4m3 blocks (both the layer input and the
 * SwiGLU output).  The pages say only "block-wise e4m3" (vLLM recipe
 * "XiaomiMiMo/MiMo-V2.6-Pro-RL", "Overview") and "dynamic activation
 * scheme" (devupai "MiMo-V2.6-Flash", "Self-Hosting"):
 *   MOE_ACT_SCALE_E8M0: a power-of-two scale per block, the smallest that
 *     keeps the block's amax within 448 (the scale the block-scaled tensor
 *     cores take directly; the default);
 *   MOE_ACT_SCALE_F32: s = amax / 448 per block in fp32, codes e4m3 of the
 *     fp32 quotient v / s (an all-zero block: s = 0, zero codes); the GEMMs
 *     then fold s into fp32 partial sums per 128-wide K block. */
enum { MOE_ACT_SCALE_E8M0 = 0, MOE_ACT_SCALE_F32 = 1 };

typedef struct {
    int hidden;       /* H: multiple of 128, 128..16384 */
    int inter;        /* I: multiple of 128, 128..16384 */
    int num_experts;  /* E: 1..512 */
    int top_k;        /* k: 1..min(E, 8) */
    int max_tokens;   /* workspace is sized for 0 <= T <= max_tokens (>= 1) */
    int score_func;   /* MOE_SCORE_SIGMOID (the pages' router) or MOE_SCORE_SOFTMAX */
    int device;       /* CUDA device ordinal; the device must be sm_103 */
    int act_scale_mode; /* MOE_ACT_SCALE_E8M0 (0, default) or MOE_ACT_SCALE_F32 */
    /* Tensor-parallel shard of the expert middle dimension (the pages' TP8 /
     * TP4 deployments: vLLM recipe "XiaomiMiMo/MiMo-V2.6-Pro-RL", "Overview"
     * hardware line and the TP8 (H200) / TP4 (MI355X) launch recipes).
     * tp_size G in 1..8 (0 means 1), 0 <= tp_rank < G, inter a multiple of
     * 128 * G.  Shard r keeps, for every expert, gate and up rows
     * [r I/G, (r+1) I/G) of W13 and the same columns of W2, so its SwiGLU
     * blocks of 128 are exactly the whole layer's; routing, dispatch and the
     * input quantisation are the same on every shard.  Its output is a
     * partial sum (moe_forward_partial); the layer output is the sum of the
     * G partials rounded once to bf16 (an all-reduce, then
     * moe_sum_partials_bf16).  inter stays the whole layer's I. */
    int tp_size;
    int tp_rank;
} moe_config;

/* Create a handle: checks the configuration and the device, allocates the
 * workspace for max_tokens tokens on cfg->device.  *out receives the handle
 * (NULL on failure). */
moe_status moe_init(const moe_config* cfg, moe_handle** out);

/* Free everything the handle owns.  NULL is accepted (no-op). */
moe_status moe_destroy(moe_handle* h);

/* Copy the layer's weights into the handle (host or device pointers; the
 * copy is synchronous and the caller's buffers may be freed afterwards).
 * The tensors are always the whole layer's; a tensor-parallel shard keeps
 * its slice (and checks only the scales it keeps).
 *   router_w   bf16 [E][H]
 *   logit_bias fp32 [E], added to the router logits; NULL = zeros
 *   sel_bias   fp32 [E], the correction bias added to the scores for
 *              selection only; NULL = zeros
 *   w13_q      u8 [E][2I][H/2]  packed E2M1, element 2i in the low nibble;
 *              rows [0, I) are the gate projection, [I, 2I) the up projection
 *   w13_s      u8 [E][2I][H/32] E8M0 scale per 32 consecutive inputs
 *   w2_q       u8 [E][H][I/2]   down projection, packed E2M1
 *   w2_s       u8 [E][H][I/32]
 * A scale byte 0xFF (E8M0 NaN) fails with MOE_ERR_INVALID_ARG and leaves the
 * handle without weights. */
moe_status moe_load_weights(moe_handle* h, const uint16_t* router_w, const float* logit_bias,
                            const float* sel_bias, const uint8_t* w13_q, const uint8_t* w13_s,
                            const uint8_t* w2_q, const uint8_t* w2_s);

/* The same with the experts in the fp8 block format of the V2.5 files
 * ("MiMo V2.6 Pro and Flash architecture teardown", section "Why Are the
 * V2.6 Files Half the Size of V2.5?", the V2.5 / V2.6 table, row "Routed
 * experts": FP8 E4M3 with one F32 scale per 128 x 128 block): the weight is
 * e4m3(q) * scale of its block (exactly, no requantisation).
 *   w13        u8 e4m3 [E][2I][H] (gate rows [0, I), up rows [I, 2I))
 *   w13_scale  fp32 [E][2I/128][H/128]
 *   w2         u8 e4m3 [E][H][I]
 *   w2_scale   fp32 [E][H/128][I/128]
 * An e4m3 NaN code (0x7F, 0xFF) or a negative / non-finite scale fails with
 * MOE_ERR_INVALID_ARG and leaves the handle without weights.  The GEMMs then
 * fold the block scales into fp32 partial sums per 128-wide K block. */
moe_status moe_load_weights_fp8(moe_handle* h, const uint16_t* router_w, const float* logit_bias,
                                const float* sel_bias, const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                                const float* w2_scale);

/* y = layer(x) for T tokens: x bf16 [T][H] and y bf16 [T][H] are device
 * pointers (x and y must not overlap).  Enqueued on `stream`; returns without
 * waiting for the GPU and without reading anything back, so it can be
 * captured in a CUDA graph.  T = 0 is a no-op.  T > max_tokens fails with
 * MOE_ERR_SHAPE.  A device-side timeout of an earlier call is reported by
 * the next call that synchronises (moe_check_device_error or a getter). */
moe_status moe_forward(moe_handle* h, const uint16_t* x, int T, uint16_t* y, void* stream);

/* The same forward with the gate-weighted sum left in fp32 and not rounded:
 * y32 fp32 [T][H] device.  For a tensor-parallel shard this is its partial
 * output (sum over the shard's slice of the expert middle dimension); for
 * tp_size 1 it is the layer output before the bf16 rounding. */
moe_status moe_forward_partial(moe_handle* h, const uint16_t* x, int T, float* y32, void* stream);

/* y[i] = bf16( parts[0][i] + parts[1][i] + ... ), the n_parts (1..8) fp32
 * device arrays of n elements added in index order in fp32, rounded once to
 * nearest even: the layer output from the shards' partials (or from one
 * all-reduced sum, n_parts = 1).  `parts` is a host array of device
 * pointers; y bf16 device.  Enqueued on `stream` (current device); errors
 * through moe_last_error(NULL). */
moe_status moe_sum_partials_bf16(const float* const* parts, int n_parts, size_t n, uint16_t* y, void* stream);

/* Same layer with host buffers: copies x (host, [T][H] bf16) to the device,
 * runs moe_forward on `stream`, copies y back to y_host and waits until y_host
 * holds the output.  Pinned host memory gives the fastest copies. */
moe_status moe_forward_host(moe_handle* h, const uint16_t* x_host, int T, uint16_t* y_host, void* stream);

/* The same without waiting: enqueues the input copy, the forward (on
 * `stream`) and the output copy, and returns.  The handle keeps two device
 * staging slots and two copy streams of its own, so the copies of one call
 * overlap the forwards of the previous and next calls (a stream of batches
 * runs at about the rate of its slowest engine: copy in, compute, copy out).
 * x_host must stay unchanged and y_host untouched until the call's output has
 * arrived: moe_host_sync waits for every call issued so far.  x_host and
 * y_host must be pinned (page-locked) for the copies to run asynchronously.
 * Issue the forwards of one handle on one stream (they share its
 * workspace).  Errors of the enqueue are returned; device-side errors as for
 * moe_forward. */
moe_status moe_forward_host_async(moe_handle* h, const uint16_t* x_host, int T, uint16_t* y_host, void* stream);
moe_status moe_host_sync(moe_handle* h);

/* Debug getters for the last forward (they synchronise the device and copy
 * to HOST memory; T and k are those of that forward):
 *   logits   fp32 [T][E]
 *   ids      int32 [T][k] selected experts in selection order
 *   gates    fp32 [T][k]
 *   counts   int32 [E], offsets int32 [E+1] (exclusive scan of counts)
 *   perm     int32 [T*k]: perm[t*k+j] = row of (token t, slot j) in the
 *            expert-contiguous order, token-ascending within an expert
 *   act q    u8 [T][H] e4m3 codes of x, scale u8 [T][H/128] E8M0 bytes
 *   inter q  u8 [T*k][I] e4m3 codes of silu(g)*u in perm order,
 *            scale u8 [T*k][I/128] (a tensor-parallel shard: its I/G
 *            columns, [T*k][I/G] and [T*k][I/(128 G)])
 *   (with MOE_ACT_SCALE_F32 the u8 scale outputs must be NULL: the scales
 *   are fp32 and come from the two *_scales_f32 getters, which in either
 *   mode return every block scale as its fp32 value, [T][H/128] and
 *   [T*k][I/128])
 *   expert_out fp32 [T*k][H]: o of every (token, slot) row in perm order
 *            (a shard: the partial over its slice)
 * Any output pointer may be NULL to skip it. */
moe_status moe_get_logits(moe_handle* h, float* logits);
moe_status moe_get_routing(moe_handle* h, int32_t* ids, float* gates);
moe_status moe_get_expert_counts(moe_handle* h, int32_t* counts, int32_t* offsets);
moe_status moe_get_permutation(moe_handle* h, int32_t* perm);
moe_status moe_get_act_quant(moe_handle* h, uint8_t* q, uint8_t* scale);
moe_status moe_get_inter_quant(moe_handle* h, uint8_t* q, uint8_t* scale);
moe_status moe_get_act_scales_f32(moe_handle* h, float* scale);
moe_status moe_get_inter_scales_f32(moe_handle* h, float* scale);
moe_status moe_get_expert_out(moe_handle* h, float* out);

/* Per-stage timing of subsequent forwards: CUDA events recorded between the
 * stages on the forward's stream, kept for the 64 most recent forwards.
 * moe_get_stage_times waits for the last recorded forward and writes, for
 * each of min(n, moe_stage_count()) stages, its average milliseconds over
 * the forwards recorded since profiling was enabled or the times were last
 * read (at most the last 64); then it starts a new recording window.  The
 * stages (moe_stage_name): router, topk, dispatch, gemm1_gate_up,
 * gemm2_down, combine.  For batches of at least 4,096 tokens the top-k runs
 * in the router kernel's epilogue and the topk stage times nothing. */
moe_status moe_set_profiling(moe_handle* h, int enable);
moe_status moe_get_stage_times(moe_handle* h, float* ms, int n);
int moe_stage_count(void);
const char* moe_stage_name(int i);

/* Synchronise the device and report (then clear) an error word written by a
 * kernel (MOE_ERR_TIMEOUT from a bounded wait, MOE_ERR_DEVICE otherwise). */
moe_status moe_check_device_error(moe_handle* h);

/* Self-test of the kernels' bounded waits (the pages have no counterpart;
 * it checks the library's own failure detection without harming the GPU):
 * launches one small kernel on the legacy default stream whose thread waits
 * on a barrier that nothing completes; after limit_us microseconds
 * (1 .. 1,000,000) the wait gives up, records MOE_ERR_TIMEOUT in the
 * handle's device error word (site 99) as any kernel wait would, and the
 * kernel exits normally.  The next moe_check_device_error (or getter)
 * reports MOE_ERR_TIMEOUT and clears the word; the context stays usable.
 * With h = NULL the timeout is recorded in the error record of the
 * allocation-free routing (moe_route_noalloc) on the current device, which
 * moe_route_noalloc_check_error reports. */
moe_status moe_selftest_wait_timeout(moe_handle* h, unsigned int limit_us);

/* Throughput probe of the block-scaled tensor-core instruction the grouped
 * GEMMs issue (the pages have no counterpart: it measures the denominator of
 * the prefill roofline): tcgen05.mma kind::mxf8f6f4 .block_scale, M = 128,
 * N = 256, K = 32, e4m3 x E2M1 with E8M0 scales, operands resident in shared
 * memory, accumulation in TMEM.  One CTA per SM of `device` issues
 * 4 * steps_per_cta MMAs (1 .. 2^22 steps) with the GEMMs' issue loop;
 * `launches` (1 .. 10^5) launches run back to back on the legacy default
 * stream and the call waits for them.  result (host, float[4]):
 *   [0] dense TFLOP/s over all launches (2*128*256*32 per MMA, CUDA events),
 *   [1] mean SM clock in MHz during the last launch (cycle counter against
 *       the global timer), [2] SM cycles per MMA in the last launch,
 *   [3] elapsed milliseconds of all launches.
 * Allocates a small result buffer; errors through moe_last_error(NULL). */
moe_status moe_selftest_mma_peak(int device, int steps_per_cta, int launches, float* result);

/* The same probe for other shapes of the instruction (no counterpart in the
 * pages either): M = 128, K = 32, N = n columns, in the order the heavy
 * m-tiles use (tokens_on_n = 0: 128 e4m3 token rows as A, n E2M1 weight rows
 * as B; n a multiple of 16 in [16, 256]) or the order of the light m-tiles
 * in the promotion modes (tokens_on_n = 1: 128 E2M1 weight rows as A, n
 * e4m3 token rows as B; n a multiple of 16 in [16, 128]).  One launch of
 * 4 * steps_per_cta MMAs per SM (1 .. 2^22 steps), waited for.  result
 * (host, float[3]): [0] SM cycles per MMA, [1] mean SM clock in MHz, [2]
 * dense TFLOP/s (2*128*n*32 per MMA).  Errors through moe_last_error(NULL). */
moe_status moe_selftest_mma_shape(int device, int n, int tokens_on_n, int steps_per_cta, float* result);

/* Debug: fill every workspace buffer of the handle (routing and dispatch
 * tables, the quantised activation and SwiGLU rows with their scales, the
 * expert outputs, the host-entry staging buffers; not the device error word)
 * with `byte` (0 .. 255), synchronously.  A forward writes everything it
 * reads, so its output does not depend on what was there before; the tests
 * check this with 0xFF (NaN as e4m3, E8M0, bf16 and fp32).  The getters
 * report MOE_ERR_NOT_LOADED until the next forward. */
moe_status moe_debug_fill_workspace(moe_handle* h, int byte);

/* Number of kernels the last forward launched. */
int moe_last_launch_count(moe_handle* h);


const char* moe_last_error(moe_handle* h);
const char* moe_status_string(moe_status s);

/* MXFP4 quantisation of fp32 weights on the device: the weight format of
 * "MiMo V2.6 Pro and Flash architecture teardown", section "Why Are the
 * V2.6 Files Half the Size of V2.5?" (two E2M1 values per byte, one E8M0
 * scale per 32 values), which the page says the experts were re-rounded to
 * after every RL update.  OCP Microscaling v1.0 rule per 32 consecutive
 * values of a row: X = floor(log2(amax)) - 2 clamped to [-127, 127], scale
 * byte X + 127 (127 for an all-zero block), code = nearest E2M1 value of
 * v / 2^X with ties to the even code, saturating at 6.
 *   w       fp32 [rows][K] device, finite values, 16-byte aligned
 *   packed  u8 [rows][K/2] device output, element 2i in the low nibble
 *   scales  u8 [rows][K/32] device output
 * K must be a positive multiple of 32.  Enqueued on `stream` (current
 * device); errors through moe_last_error(NULL).  The output is the
 * w13_q / w13_s (or w2_q / w2_s) input of moe_load_weights. */
moe_status moe_mxfp4_quantize(const float* w, size_t rows, int K, uint8_t* packed, uint8_t* scales, void* stream);

/* Routing that allocates no device memory (the pages have no counterpart of
 * this entry point; it serves callers that cannot allocate on their call
 * path: code whose device memory belongs to its own allocator or budget, and
 * latency-critical loops in which cudaMalloc / cudaFree could synchronise
 * the device and stall work already in flight).
 *
 * Computes the router and top-k gate of the layer (the router and top-k
 * kernels of moe_forward) for T tokens, without a handle.  The logits are
 * accumulated over all of H in one pass, whereas moe_forward splits H into
 * up to 16 partial sums for T <= 512: the fp32 rounding differs, so where a
 * token's k-th and (k+1)-th keys lie within that rounding the two entry
 * points may select differently (both selections are valid top-k sets).
 *   x          bf16 [T][H] device, 16-byte aligned
 *   router_w   bf16 [E][H] device, 16-byte aligned
 *   logit_bias fp32 [E] device or NULL (zeros); sel_bias fp32 [E] device or NULL
 *   ids        int32 [T][k] device output (selection order)
 *   gates      fp32 [T][k] device output
 * on `stream`, on the current CUDA device (which must be sm_103).  H must be
 * a multiple of 64, 1 <= E <= 512, 1 <= k <= min(E, 8).
 *
 * Scratch: the router logits go to a fixed array compiled into the library,
 * T * E <= 1,048,576 floats (4 MiB); every GPU that loads the library holds
 * it until the process exits.  Larger T * E fails with MOE_ERR_SHAPE.  The
 * first call on a device also looks up that array's device address and sets
 * a kernel attribute on that device; make that first call before any stream
 * capture.  All calls share the one array and it keeps the last call's
 * contents, so calls that overlap on the GPU (different streams, or several
 * threads) race and must be serialised by the caller.  The call does not
 * wait for the GPU, so a kernel wait that gives up is recorded in the
 * array's error record (kept until read) and reported by
 * moe_route_noalloc_check_error.  Errors are reported through
 * moe_last_error(NULL). */
moe_status moe_route_noalloc(const uint16_t* x, int T, int H, const uint16_t* router_w, const float* logit_bias,
                             const float* sel_bias, int E, int k, int score_func, int32_t* ids, float* gates,
                             void* stream);

/* Waits for `stream`, then reports and clears the error record of the
 * allocation-free routing on the current device: MOE_ERR_TIMEOUT if a kernel
 * wait of an earlier moe_route_noalloc call gave up since the last check
 * (MOE_ERR_DEVICE for another kernel error), MOE_OK otherwise.  Reads and
 * clears the record with cudaMemcpyFromSymbol / cudaMemcpyToSymbol, so it
 * allocates nothing either; it synchronises, so keep it out of stream
 * capture.  Errors through moe_last_error(NULL). */
moe_status moe_route_noalloc_check_error(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_MX_H */
