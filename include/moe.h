/*
 * moe.h -- C ABI of the GB300-native single-GPU Mixture-of-Experts layer
 * forward: router -> align -> expert GEMM1 + SwiGLU -> expert GEMM2 ->
 * weighted finalize.
 *
 * Pages the operations follow (cited per entry point below):
 *   [P1] "How an MoE Model Picks Its Experts During LLM Inference"
 *   [P2] "Mixture of Experts"
 *   [P3] "MoE Kernels, in depth"
 *   [P4] "How GPUs Fuse Communication and Computation During LLM Inference"
 *
 * Common rules
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *     the argument says "host".  The library never allocates, frees or
 *     synchronises; every call only enqueues kernels on `stream` (a
 *     cudaStream_t; NULL = the legacy default stream) and returns.
 *   - Matrices are dense, row-major, contiguous.  bf16 is IEEE bfloat16;
 *     E4M3 is OCP FP8 e4m3 (one byte); E2M1 is OCP FP4 e2m1 packed two per
 *     byte, low nibble first.  Block scales are UE8M0 bytes (value
 *     2^(s-127)), one per 32 consecutive values of a row along the
 *     contraction dimension.
 *   - Arguments are checked on the host before anything is launched; a
 *     violation returns MOE_ERR_ARG (bad value) or MOE_ERR_UNSUPPORTED (a
 *     valid but unimplemented combination) and launches nothing.  T = 0 is a
 *     valid no-op.
 *   - Errors found on the device (an expert id outside [0,E), a bounded wait
 *     that expired) never trap: the kernel skips the offending access and ORs
 *     a code into the sticky error word at the start of the workspace; read
 *     it with moe_read_device_error.
 *   - Workspace: `ws` is caller-owned device memory of at least the size the
 *     matching *_workspace_bytes function returns, 256-byte aligned.  It must
 *     be zeroed once before its first use (moe_workspace_init); the library
 *     leaves it in a reusable state after every successful call.  Two calls
 *     that overlap in time must not share a workspace.
 */
#ifndef ROUTER_EXPERTS_GB300_MOE_H
#define ROUTER_EXPERTS_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_ARG = 1,          /* invalid argument (nothing launched)              */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but unimplemented combination              */
  MOE_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed                */
  MOE_ERR_DEVICE = 4        /* returned by moe_read_device_error when set       */
} moe_status;

typedef enum {
  MOE_SCORING_SOFTMAX = 0,
  MOE_SCORING_SIGMOID = 1,
  MOE_SCORING_SQRT_SOFTPLUS = 2
} moe_scoring;

typedef enum { MOE_DT_BF16 = 0, MOE_DT_F32 = 1, MOE_DT_E4M3 = 2, MOE_DT_E2M1 = 3 } moe_dtype;

/* Workspace header words a test may set (byte offsets from the workspace
 * start; everything else in the header is the library's own):
 *   MOE_WS_ALIGN_BARRIER_OFFSET  int32[2]: arrival counter and generation of
 *                                the align kernel's grid barrier (0 at rest)
 *   MOE_WS_WAIT_LIMIT_OFFSET     int64: when > 0, the align kernel's grid
 *                                barrier gives up after this many SM clock
 *                                cycles instead of about 2^32 (~2 s); a test
 *                                hook that makes the bounded-wait expiry
 *                                path cheap to exercise.  0 after
 *                                moe_workspace_init. */
#define MOE_WS_ALIGN_BARRIER_OFFSET 5120
#define MOE_WS_WAIT_LIMIT_OFFSET 5376

/* Bits of the device error word. */
#define MOE_DEVERR_BAD_EXPERT_ID 1 /* an expert id outside [0,E) was skipped          */
#define MOE_DEVERR_WAIT_TIMEOUT 2  /* a bounded in-kernel wait expired; outputs invalid */
#define MOE_DEVERR_BAD_TABLE 4     /* a block table entry was out of range (clamped)  */

/* ---------------------------------------------------------------------------
 * Router.  [P1] §1.1 (three steps: gate GEMM, scores, top-k + rescale),
 * §1.3 (rank key = score + bias used only for selection; the weight is the
 * unbiased score, Figure 3), §2.4 (bf16 inputs, fp32 logits and bias), §4
 * (reference router: weights / (sum + 1e-20)), §5.3 (one warp per token row,
 * k rounds, lowest expert id wins ties).  [P2] "Mixture of Experts", the gate
 * (a d x E linear without bias) and DeepSeek's grouped, bias-corrected
 * routing: group score = sum of the two largest rank keys of the group, keep
 * topk_group groups, mask the rest, top-k, weights from the original scores,
 * renormalise, multiply by the routed scaling factor.
 *
 *   hidden       [T,H] in hidden_dt: BF16, F32, or E4M3 with hidden_scale
 *                [T,H/32] (the router then sees the exact dequantised value)
 *   gate         [E,H] in gate_dt: BF16 or F32
 *   bias         [E] fp32 selection bias, or NULL for none
 *   scoring      MOE_SCORING_SOFTMAX (over all E logits), _SIGMOID, or
 *                _SQRT_SOFTPLUS: sqrt(ln(1 + e^l)) per expert ([P1] §1.3:
 *                DeepSeek-V4 takes the square root of a softplus in place
 *                of the sigmoid; the rank key and weights follow as for the
 *                sigmoid)
 *   n_group      1 = plain top-k; else E % n_group == 0, E/n_group >= 2,
 *                1 <= topk_group <= n_group, topk_group*E/n_group >= k
 *   renormalize  nonzero: w_j /= (sum_j w_j + 1e-20); then w_j *= scaling
 *   topk_ids     [T,k] int32 out, selection order (best first)
 *   topk_weights [T,k] fp32 out
 * Limits: 1 <= k <= min(E,16), E <= 512, H % 32 == 0.  Logits are fp32 sums
 * of exact products (fp32 inputs are split into three bf16 parts).
 *
 * Execution.  When H % 64 == 0, E % 16 == 0 with E <= 256 (or E % 32 == 0
 * with E <= 512), hidden is BF16 or E4M3 and the gate is BF16 (or F32 with at
 * least 8 tokens): the gate GEMM runs on the tensor cores in 128-token tiles
 * with the K range split over CTAs; up to 4 tokens the CTA that finishes its
 * token tile's splits last sums each token's partials in split order and
 * selects (one launch), above that a second launch does (plus one conversion
 * launch first when hidden is E4M3 or the gate is F32).  Otherwise ([P1]
 * §5.1's one-kernel router): one fused launch whose CTAs split the gate read
 * with mma.sync and whose last CTA per token tile selects.  On GB300 the
 * tensor-core path was measured faster from the first token.  Both paths
 * give the same ids except where two rank keys are within fp32
 * summation-order noise of each other.
 * moe_router_kernel_count returns how many kernels moe_router enqueues for
 * these shapes and types (0 when T == 0).
 * ------------------------------------------------------------------------- */
size_t moe_router_workspace_bytes(int T, int H, int E);
int moe_router_kernel_count(int T, int H, int E, int hidden_dt, int gate_dt);
int moe_router(const void* hidden, int hidden_dt, const uint8_t* hidden_scale, const void* gate,
               int gate_dt, const float* bias, int T, int H, int E, int k, int scoring,
               int n_group, int topk_group, int renormalize, float scaling, int32_t* topk_ids,
               float* topk_weights, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * moe_router_cast_e4m3 -- the router on a bf16 hidden state that also writes
 * the hidden rows' FP8 cast for low-bit experts.  [P4] §1.1: a small kernel
 * converts the layer input to FP8, computes the scales and writes both
 * together with the router's output.  Same arguments, rules, workspace and
 * kernels as moe_router with hidden_dt BF16; the warp that selects token t
 * also writes row t of
 *   codes  [T,H] e4m3 (16-byte aligned) and scales [T,H/32] UE8M0,
 * exactly the bytes moe_cast_e4m3 writes.  moe_layer uses this path for a
 * bf16 hidden with e2m1 experts.
 * ------------------------------------------------------------------------- */
int moe_router_cast_e4m3(const void* hidden, const void* gate, int gate_dt, const float* bias,
                         int T, int H, int E, int k, int scoring, int n_group, int topk_group,
                         int renormalize, float scaling, int32_t* topk_ids, float* topk_weights,
                         uint8_t* codes, uint8_t* scales, void* ws, size_t ws_bytes,
                         void* stream);

/* ---------------------------------------------------------------------------
 * moe_router_noalloc -- the router for callers that cannot allocate device
 * memory.  (No counterpart on the pages: it exists for this library's users.)
 *
 * Some callers cannot call cudaMalloc or any other allocator: code embedded
 * in a host framework that owns all device memory, plugins whose process
 * memory pool must not grow, or hosts that forbid allocation after start-up.
 * moe_router needs a caller-allocated workspace; this variant instead keeps
 * its scratch (partial logits and tickets) in one fixed array of device
 * memory that belongs to the library (a file-scope static __device__ array),
 * so the caller passes only the inputs and the outputs, exactly as for
 * moe_router, and nothing is allocated or freed.
 *
 *   - Same arguments and rules as moe_router, without ws/ws_bytes; always
 *     the one-launch kernel, so its ids can differ from moe_router's tiled
 *     path only on near-ties (see Execution above).
 *   - Limit: the partial logits of one call, KS * T * E * 4 bytes with the
 *     K-split count KS the router picks (16 for a few tokens, 1 for thousands),
 *     must fit in MOE_ROUTER_NOALLOC_MAX_LOGIT_BYTES (8 MiB), and
 *     T <= 262,144.  Larger problems are rejected with MOE_ERR_ARG before
 *     anything is launched (e.g. T = 4,096 fits for every E <= 512;
 *     T = 8,192 with E = 512 does not).
 *   - The array (8 MiB of partial logits and 64 KiB of tickets) exists on
 *     every GPU that loads the library, until the process exits.
 *   - The array's device address is looked up (cudaGetSymbolAddress, with
 *     the device current) by the first call in each CUDA context and cached
 *     per device with the id of that context; a call made in another context
 *     of the device (after cudaDeviceReset, or with a context of the
 *     caller's own made current) looks it up again.  Make the first call in
 *     a context before any stream capture.
 *   - Every call shares the one array and leaves its contents behind; each
 *     call clears the tickets it uses before launching.  Calls that overlap in
 *     time on the GPU (different streams, or several host threads) race on
 *     the array and produce wrong results: serialise them.
 *   - No device-side errors are reported: the one-launch router kernel has
 *     no waits and no input value it could flag, so there is no error word
 *     to read (moe_read_device_error applies to caller workspaces only).
 * ------------------------------------------------------------------------- */
#define MOE_ROUTER_NOALLOC_MAX_LOGIT_BYTES (8u << 20)
int moe_router_noalloc(const void* hidden, int hidden_dt, const uint8_t* hidden_scale,
                       const void* gate, int gate_dt, const float* bias, int T, int H, int E,
                       int k, int scoring, int n_group, int topk_group, int renormalize,
                       float scaling, int32_t* topk_ids, float* topk_weights, void* stream);

/* ---------------------------------------------------------------------------
 * Align (moe_align_block_size).  [P3] "Alignment: making ragged routing
 * tileable" (count per expert, round up to block_m, exclusive prefix sum,
 * sorted assignment ids with the sentinel T*k for padding, expert of every
 * block, padded length; no host sync; buffers sized for the worst case
 * T*k + E*(block_m-1)).  [P2] "vLLM's Triton path: align, then index" (worked
 * example; unused block entries are -1).
 *
 *   topk_ids        [T,k] int32; assignment a = t*k + j
 *   sorted_ids      [cap_rows] int32 out: assignments grouped by expert in
 *                   ascending expert id, within an expert in ascending a
 *                   (deterministic); pads and the tail hold T*k
 *   cap_rows        >= T*k + E*(block_m-1)
 *   block_expert    [ceil(cap_rows/block_m)] int32 out; -1 past the end
 *   num_post_padded [1] int32 out: sum over experts of ceil(count/block_m)*block_m
 * Limits: block_m in {16, 64, 128}; E <= 1024.  An id outside [0,E) is
 * skipped (not placed) and sets MOE_DEVERR_BAD_EXPERT_ID.
 * ------------------------------------------------------------------------- */
size_t moe_align_workspace_bytes(void);
int moe_align(const int32_t* topk_ids, int T, int k, int E, int block_m, int32_t* sorted_ids,
              int64_t cap_rows, int32_t* block_expert, int32_t* num_post_padded, void* ws,
              size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Expert GEMMs.  [P3] "The fused expert GEMM" (each tile looks up its expert
 * in block_expert and its rows in sorted_ids; the activation gather is folded
 * into the operand load; padding rows masked; gate and up are one 2F x H
 * matrix with SwiGLU silu(g) * u in the epilogue; the routing weight is
 * applied in the down GEMM's epilogue so the combine is a plain sum).
 * [P2] w13 [E, 2F, H] (gate rows 0..F-1, up rows F..2F-1), w2 [E, H, F].
 * [P4] §3.5: SwiGLU and FP8 re-quantisation (a power-of-two scale per 32
 * values, the smallest with amax/scale <= 448) fused into one epilogue.
 *
 * moe_expert_gemm1: inter[p, f] = silu(g) * u for every padded row p <
 *   num_post_padded, where g/u are row (sorted_ids[p] / k) of x times the
 *   gate/up rows of w13[block_expert[p / block_m]]; pad rows are written 0.
 *   act_dt BF16: x [T,H] bf16, inter [cap_rows, F] bf16.
 * moe_expert_gemm2: stage[a, h] = bf16(weight[a] * sum_f inter[p, f] * w2[e, h, f])
 *   for every real row p (a = sorted_ids[p] < T*k).
 * moe_grouped_ffn: both, with inter held in the workspace.
 * Low-bit GEMM1 with a workspace of moe_ffn_workspace_bytes (and in
 * moe_layer for an e4m3 hidden): one extra launch first copies x's rows (codes
 * and scale bytes) into the blocks' padded order in the workspace, so the
 * GEMM reads its token tiles by TMA; with a smaller workspace
 * (moe_expert_gemm1 needs only the header) the GEMM gathers the rows itself.
 * w_dt must equal act_dt (BF16) or be E2M1 with act_dt E4M3 (low-bit).
 * Limits: H % 64 == 0, F % 32 == 0 (low-bit: H % 128 == 0, F % 128 == 0 and
 * every scale array 4-byte aligned), block_m in {16, 64, 128} (MOE_ERR_ARG
 * otherwise); any other dtype pair returns MOE_ERR_UNSUPPORTED.
 *
 * Low-bit layouts ([P4] §1.1: FP4 weights, FP8 tokens, one power-of-two
 * scale byte 2^(s-127) per 32 values along the contraction):
 *   x [T,H] e4m3 codes, x_scale [T,H/32]; w13 [E,2F,H/2] e2m1 packed (low
 *   nibble = even column), w13_scale [E,2F,H/32]; inter [cap_rows,F] e4m3
 *   codes, inter_scale [cap_rows,F/32] (written by gemm1: [P4] §3.5 scale =
 *   smallest power of two with amax/scale <= 448, codes rounded to nearest
 *   even and saturated at 448); w2 [E,H,F/2] e2m1, w2_scale [E,H,F/32].
 *   w13 and w2 must be 32-byte aligned, the other low-bit arrays 16-byte
 *   (codes) or 4-byte (scales) aligned (MOE_ERR_ARG otherwise).
 *   The tensor core applies every scale byte as an exact power of two and
 *   accumulates in fp32, so the result is the dequantised product up to fp32
 *   accumulation rounding while the scaled values stay in the fp32 normal
 *   range.
 * ------------------------------------------------------------------------- */
size_t moe_ffn_workspace_bytes(int T, int H, int F, int E, int k, int block_m, int act_dt);
int moe_expert_gemm1(const void* x, int act_dt, const uint8_t* x_scale, const void* w13,
                     const uint8_t* w13_scale, int w_dt, int T, int H, int F, int E, int k,
                     int block_m, const int32_t* sorted_ids, const int32_t* block_expert,
                     const int32_t* num_post_padded, int64_t cap_rows, void* inter,
                     uint8_t* inter_scale, void* ws, size_t ws_bytes, void* stream);
int moe_expert_gemm2(const void* inter, const uint8_t* inter_scale, int act_dt, const void* w2,
                     const uint8_t* w2_scale, int w_dt, int T, int H, int F, int E, int k,
                     int block_m, const int32_t* sorted_ids, const int32_t* block_expert,
                     const int32_t* num_post_padded, int64_t cap_rows,
                     const float* topk_weights, void* stage, void* ws, size_t ws_bytes,
                     void* stream);
int moe_grouped_ffn(const void* x, const uint8_t* x_scale, int act_dt, const void* w13,
                    const uint8_t* w13_scale, const void* w2, const uint8_t* w2_scale, int w_dt,
                    int T, int H, int F, int E, int k, int block_m, const int32_t* sorted_ids,
                    const int32_t* block_expert, const int32_t* num_post_padded,
                    int64_t cap_rows, const float* topk_weights, void* stage, void* ws,
                    size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Finalize.  [P3] "Combine" (a gather per token summing its k rows in a fixed
 * order is deterministic); [P2] ops.moe_sum reduces the top-k axis of the
 * [T, k, H] cache; [P4] §3.7 (add the slots as 32-bit floats in slot order,
 * round once to 16 bits).
 *   stage [T*k, H] bf16 (weights already applied), out [T, H] bf16:
 *   out[t, h] = bf16(sum_{j=0..k-1} stage[t*k + j, h]) summed in fp32.
 *   The staged rows themselves are bf16 (moe_expert_gemm2 rounds each
 *   weighted slot row once), so a layer output is rounded once per slot row
 *   and once more after the fp32 sum.
 * ------------------------------------------------------------------------- */
int moe_finalize(const void* stage, int T, int k, int H, void* out, void* stream);

/* ---------------------------------------------------------------------------
 * FP8 cast of a layer input.  [P4] §1.1 (a small kernel converts the layer
 * input to FP8 and writes the scales) with §3.5's scale rule; [P3] "Low
 * precision" (quantise activations in a pass that moves the rows anyway).
 *   x      [T,H] bf16, 16-byte aligned, H % 32 == 0
 *   codes  [T,H] e4m3 out, 16-byte aligned
 *   scales [T,H/32] UE8M0 out: per 32 values the smallest 2^s (s in
 *          [-127, 127], 0 for an all-zero group) with amax / 2^s <= 448
 *   codes = e4m3(x / 2^s), nearest, ties to even, saturating at 448.
 * MOE_ERR_ARG for invalid shapes or alignment; T == 0 is a no-op.
 * ------------------------------------------------------------------------- */
int moe_cast_e4m3(const void* x, int T, int H, uint8_t* codes, uint8_t* scales, void* stream);

/* ---------------------------------------------------------------------------
 * The whole layer: router, align, GEMM1 + SwiGLU, GEMM2 + weight, finalize,
 * enqueued back to back with no host synchronisation.  block_m = 0 picks the
 * tile height from the mean rows per expert T*k/E: 16 below 8, 64 below 64,
 * else 128 ([P3] "Tile shape is the main tuning knob ... depends on tokens
 * per expert").  act_dt/w_dt as for the expert GEMMs; the router reads
 * `hidden` (dequantised when E4M3).  out [T,H] bf16.
 * act_dt BF16 with w_dt E2M1 (hidden_scale ignored): the router reads the
 * bf16 rows and the experts read their FP8 cast, the codes and scales of
 * moe_cast_e4m3, which the router's selecting warps write next to each
 * token's ids and weights ([P4] §1.1: the cast in front of the fused expert
 * kernel writes them together with the router's output); hidden must be
 * 16-byte aligned.
 * One token (T == 1) skips the align launch: its k experts are distinct, so
 * every block holds one assignment and the GEMMs read topk_ids as the block
 * table ([P2] "vLLM's Triton path": the naive block assignment of small
 * batches).
 * moe_layer_kernel_count returns how many kernels moe_layer enqueues for
 * these shapes and types (0 when T == 0 or the arguments are invalid).
 * ------------------------------------------------------------------------- */
size_t moe_layer_workspace_bytes(int T, int H, int F, int E, int k, int block_m, int act_dt);
int moe_layer_kernel_count(int T, int H, int F, int E, int k, int act_dt, int gate_dt,
                           int w_dt);
int moe_layer(const void* hidden, int act_dt, const uint8_t* hidden_scale, const void* gate,
              int gate_dt, const float* bias, const void* w13, const uint8_t* w13_scale,
              const void* w2, const uint8_t* w2_scale, int w_dt, int T, int H, int F, int E,
              int k, int scoring, int n_group, int topk_group, int renormalize, float scaling,
              int block_m, void* out, void* ws, size_t ws_bytes, void* stream);
/* Tile height moe_layer uses for block_m = 0. */
int moe_pick_block_m(int T, int k, int E);

/* ---------------------------------------------------------------------------
 * The whole layer in ONE persistent kernel, for small batches.  [P4] §3.3
 * (GEMM 1 of an expert starts once its tokens are there, signalled by
 * readiness counters), §3.4 (the fused kernel on a single GPU), §3.6 (GEMM 2
 * tasks start before GEMM 1 has finished, waiting only for the rows they
 * read).  The steps are the separate entry points': the one-launch router
 * ([P1] §5.1, §5.3), the align with block_m 16 ([P3] Alignment), GEMM1 +
 * SwiGLU and GEMM2 + routing weight ([P3] The fused expert GEMM) and the
 * fixed-order combine ([P3] Combine), so the output equals moe_layer's up to
 * the router's fp32 summation order.
 *   Same arguments as moe_layer with every tensor bf16 (hidden [T,H], gate
 *   [E,H], w13 [E,2F,H], w2 [E,H,F]; bias fp32 or NULL).  Limits: 1 <= T*k
 *   <= 512, E <= 512, k <= 16, H % 64 == 0, F % 64 == 0, and the router's
 *   expert tiles of 8 times its token tiles of 16 (ceil(E/8)*ceil(T/16)) at
 *   most the GPU's SM count; MOE_ERR_ARG otherwise (nothing launched).
 *   topk_ids [T,k] int32 / topk_weights [T,k] fp32: where the router's
 *   selection goes (the caller may keep it, e.g. for expert-load statistics),
 *   or both NULL to keep it in the workspace.
 *   w13, w2, out 16-byte aligned; ws of moe_layer_persistent_workspace_bytes
 *   (0 for shapes outside the limits), zeroed once before first use.
 * One cooperative launch of one CTA per SM; every in-kernel wait (routing
 * done, a block's GEMM1 rows ready) is bounded and sets
 * MOE_DEVERR_WAIT_TIMEOUT on expiry.
 * ------------------------------------------------------------------------- */
size_t moe_layer_persistent_workspace_bytes(int T, int H, int F, int E, int k);
int moe_layer_persistent(const void* hidden, const void* gate, const float* bias, const void* w13,
                         const void* w2, int T, int H, int F, int E, int k, int scoring,
                         int n_group, int topk_group, int renormalize, float scaling, void* out,
                         int32_t* topk_ids, float* topk_weights, void* ws, size_t ws_bytes,
                         void* stream);

/* ---------------------------------------------------------------------------
 * Floor probes (measurement only; they compute nothing of the method).
 * [P1] §3.3 "The Floor": the least a router can cost is one kernel launch and
 * one cold read of the gate weight, measured with kernels that do no useful
 * work.
 * moe_probe_empty: an empty kernel of `blocks` blocks of `threads` threads
 *   (1 <= blocks <= 2^20, 1 <= threads <= 512).
 * moe_probe_read: every thread of ceil(bytes/16/512) blocks of 512 threads
 *   loads 16 bytes of p (device, 16-byte aligned; bytes a multiple of 16), so
 *   the kernel reads the buffer once.  sink is one device int32 that is
 *   written only if a loaded 16-byte word XORs to 0x9E3779B9 (it keeps the
 *   loads from being removed; its value means nothing).
 * MOE_ERR_ARG for invalid arguments.
 * ------------------------------------------------------------------------- */
int moe_probe_empty(int blocks, int threads, void* stream);
int moe_probe_read(const void* p, size_t bytes, int32_t* sink, void* stream);

/* ---------------------------------------------------------------------------
 * Utilities.
 * ------------------------------------------------------------------------- */
/* Zero `ws_bytes` bytes of a workspace (asynchronous on `stream`). */
int moe_workspace_init(void* ws, size_t ws_bytes, void* stream);
/* SYNCHRONISING: waits for `stream`, copies the device error word into *code
 * (host), clears it when `clear` is nonzero.  Returns MOE_OK when the word is
 * 0, MOE_ERR_DEVICE when it is not, MOE_ERR_CUDA on a CUDA failure. */
int moe_read_device_error(void* ws, int32_t* code, int clear, void* stream);
/* Human-readable status. */
const char* moe_status_string(int status);
/* Text of the last CUDA error seen by any entry point of this thread ("" if none). */
const char* moe_last_cuda_error_string(void);

#ifdef __cplusplus
}
#endif
#endif /* ROUTER_EXPERTS_GB300_MOE_H */
