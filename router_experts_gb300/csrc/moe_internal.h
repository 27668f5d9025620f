// moe_internal.h -- host-side declarations shared by the translation units of
// the CUDA library (kernel launchers, workspace layout).  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace moe {

// ---- fixed workspace header (offsets independent of shapes, so a workspace
// zeroed once stays valid across calls of any shape) --------------------------
constexpr size_t kWsErrOffset = 0;                  // int32 sticky error word
constexpr size_t kWsFfnTicketOffset = 1024;         // int32[kFfnMaxTickets]
constexpr int kFfnMaxTickets = 1024;
constexpr size_t kWsAlignBarrierOffset = 5120;      // int32[2] grid barrier of the align kernel
constexpr size_t kWsAlignTicketOffset = 5128;       // int32 align: CTAs done reading the counts
constexpr size_t kWsWaitLimitOffset = 5376;         // int64 test hook: align barrier limit (cycles)
constexpr size_t kWsDecodeCounterOffset = 6144;     // int32[3] persistent layer: routed, zeroed, done
constexpr size_t kWsRouterTicketOffset = 8192;      // int32[kRouterMaxTiles]
constexpr int kRouterMaxTiles = 65536;              // token tiles of 16 -> T <= 1,048,576
constexpr size_t kWsAlignHistOffset = kWsRouterTicketOffset + 4ull * kRouterMaxTiles;
constexpr int kAlignMaxCtas = 64;                   // int32[kAlignMaxCtas][kAlignMaxE]
constexpr int kAlignMaxE = 1024;
constexpr size_t kWsHeaderBytes = kWsAlignHistOffset + 4ull * kAlignMaxCtas * kAlignMaxE;

constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Raise a kernel's dynamic shared-memory limit on the current device, once per
// device (the limit is an attribute of the function on each device, so a
// process that drives several GPUs sets it on every one).  `done` is the
// caller's per-kernel record of the devices already set (devices 0..63;
// higher ones are set on every call).
inline bool ensure_smem_limit(const void* kernel, int bytes,
                              std::atomic<unsigned long long>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  done.fetch_or(bit, std::memory_order_release);
  return true;
}

// ---- router -----------------------------------------------------------------
struct RouterPlan {
  // fused one-launch kernel (any T)
  int nb8;        // n8 tiles of experts per CTA (1 or 8)
  int et;         // experts per CTA
  int ne;         // expert tiles
  int nt;         // token tiles of 16
  int ks;         // K splits across CTAs
  // tiled tensor-core path (bf16 or e4m3 hidden, bf16 or fp32 gate)
  int T;
  bool tiled;
  int tnt;        // token tiles of 128
  int tks;        // K splits across CTAs
  bool fused_select;  // T <= kRouterFusedSelectMaxT: the GEMM's last CTA selects
  size_t xb_off, gp_off;  // offsets in the scratch of the bf16 x and the gate planes
  size_t scratch_bytes;
};
// Up to this many tokens the tensor-core router selects in the last CTA of
// its gate GEMM (one launch; its six warps select one token each); above it
// a selection kernel follows (measured on GB300: one launch saves 2 µs at
// T = 1 for Qwen3, none for DeepSeek-V3, and costs 2-6 µs at T = 8, where
// the last CTA's warps select twice in turn).
constexpr int kRouterFusedSelectMaxT = 4;
// allow_tiled = false keeps every T on the fused kernel.
RouterPlan plan_router(int T, int H, int E, bool allow_tiled = true);
// Argument rules shared by every router entry point: MOE_OK, MOE_ERR_ARG or
// MOE_ERR_UNSUPPORTED (the codes of include/moe.h).
int check_router(const void* hidden, int hidden_dt, const uint8_t* hidden_scale, const void* gate,
                 int gate_dt, int T, int H, int E, int k, int scoring, int n_group,
                 int topk_group);
// hidden_dt: 0 bf16, 1 f32, 2 e4m3; gate_dt: 0 bf16, 1 f32
bool router_uses_tiled(const RouterPlan& plan, int hidden_dt, int gate_dt);
int launch_router(const void* hidden, int hidden_dt, const uint8_t* hidden_scale,
                  const void* gate, int gate_dt, const float* bias, int T, int H, int E, int k,
                  int scoring, int n_group, int topk_group, int renormalize, float scaling,
                  int32_t* topk_ids, float* topk_weights, float* scratch, int* tickets, int* err,
                  const RouterPlan& plan, cudaStream_t stream, uint8_t* cast_codes = nullptr,
                  uint8_t* cast_scales = nullptr, int* align_hist = nullptr, int align_seg = 0);
// cast_codes / cast_scales (bf16 hidden only, 16-byte aligned rows): the
// selecting warp of every token also writes the token's FP8 cast ([T, H]
// e4m3 codes, [T, H/32] UE8M0 scales), as moe_cast_e4m3 would.
// align_hist / align_seg: the selecting warp also adds each selected
// assignment a = t*k + j to align_hist[(a / align_seg) * E + id] (the counts
// launch_align takes with precounted = true).

// ---- align ------------------------------------------------------------------
// The align kernel's split of the n = T*k assignments: G CTAs (one per 512
// assignments, 1..16), CTA c owning [c*seg, (c+1)*seg), seg a multiple of 32.
inline void align_partition(int n, int* G, int* seg) {
  int g = (n + 511) / 512;
  g = g < 1 ? 1 : (g > 16 ? 16 : g);
  *G = g;
  *seg = ((n + g - 1) / g + 31) / 32 * 32;
}
// hist: int32[kAlignMaxCtas * kAlignMaxE] scratch; bar: int32[2], zero before
// the first call (self-resetting afterwards); wait_limit: the workspace's
// barrier-limit word (nullptr or 0: the default limit).
// precounted: the router's selection already added every assignment to hist
// ([G][E] of align_partition's segments), so the kernel skips publishing its
// counts and the grid barrier.  Either way, with more than one CTA the last
// CTA to have read hist zeroes it again (ticket: an int32, zero before the
// first call, self-resetting), so hist is all zeros between calls.
int launch_align(const int32_t* topk_ids, int T, int k, int E, int block_m, int32_t* sorted_ids,
                 int64_t cap_rows, int32_t* block_expert, int32_t* num_post_padded, int* hist,
                 int* bar, int* err, const long long* wait_limit, cudaStream_t stream,
                 bool precounted = false, int* ticket = nullptr);

// ---- expert GEMMs -------------------------------------------------------------
struct FfnParams {
  const int32_t* sorted_ids;
  const int32_t* block_expert;
  const int32_t* num_post_padded;
  const void* x;               // GEMM1 activations [T, H]
  void* inter;                 // GEMM1 output / GEMM2 input [cap, F]
  const float* topk_weights;   // GEMM2 row weights [T*k]
  void* stage;                 // GEMM2 output [T*k, H]
  float* partial;              // split-K partial sums
  int* tickets;                // split-K tickets (self-resetting)
  int* err;
  int T, H, F, E, k;
  int cap_rows;
  int max_slots;               // capacity of `partial`, in units
  int naive;                   // single-assignment blocks (see padded_rows)
};
int ffn_max_slots(int block_m);
size_t ffn_partial_bytes(int block_m);
// kind 0: GEMM1 + SwiGLU, kind 1: GEMM2 + routing weight.
int launch_ffn_gemm(int kind, int block_m, const void* w, const FfnParams& p, int num_sms,
                    cudaStream_t stream, const char** why);

// ---- low-bit expert GEMMs (e4m3 activations x e2m1 weights, UE8M0 per 32) ------
struct LowbitParams {
  const int32_t* sorted_ids;
  const int32_t* block_expert;
  const int32_t* num_post_padded;
  const uint8_t* act;          // GEMM1: x codes [T, H]; GEMM2: inter codes [cap, F]
  const uint8_t* act_scale;    // GEMM1: [T, H/32]; GEMM2: [cap, F/32]
  const uint8_t* w;            // GEMM1: w13 [E*2F, H/2]; GEMM2: w2 [E*H, F/2]
  const uint8_t* w_scale;      // GEMM1: [E*2F, H/32]; GEMM2: [E*H, F/32]
  uint8_t* inter_q;            // GEMM1 output codes [cap, F]
  uint8_t* inter_scale;        // GEMM1 output scales [cap, F/32]
  const float* topk_weights;   // GEMM2 row weights [T*k]
  __nv_bfloat16* stage;        // GEMM2 output [T*k, H]
  int* err;
  int T, H, F, E, k, BM;
  int cap_rows;
  int naive;                   // single-assignment blocks (see padded_rows)
};
// xperm / xperm_scale (GEMM1 only; nullptr: gather the rows instead): room
// for cap_rows x H codes and cap_rows x H/32 scale bytes, 256-byte aligned;
// GEMM1 then launches a permutation of its token rows into the blocks'
// padded order first and loads them by TMA.
int launch_lowbit_gemm(int kind, const LowbitParams& p, int num_sms, cudaStream_t stream,
                       uint8_t* xperm = nullptr, uint8_t* xperm_scale = nullptr);
// bf16 x [T, H] (16-byte aligned, H % 32 == 0) -> e4m3 codes [T, H] (16-byte
// aligned) and UE8M0 scale bytes [T, H/32].
int launch_cast_e4m3(const void* x, int T, int H, uint8_t* codes, uint8_t* scales,
                     cudaStream_t stream);

// ---- finalize -----------------------------------------------------------------
int launch_finalize(const void* stage, int T, int k, int H, void* out, cudaStream_t stream);

// ---- persistent decode layer (decode.cu) ----------------------------------------
constexpr int kDecodeMaxAssignments = 512;  // T*k
constexpr int kDecodeMaxSlots = 1024;       // split-K partial slots per GEMM (as ffn.cu, BM 16)
struct DecodePlan {
  bool ok;
  int ne, nt, ks;  // router items: expert tiles of 8, token tiles of 16, K slices
  size_t logits, ids, wts, ready, tokcnt, tick1, tick2, part1, part2, inter, stage, bytes;
};
// Shapes the persistent layer takes (bf16), the router's item split and the
// layout of its workspace region (offsets from the region start).
DecodePlan plan_decode(int T, int H, int F, int E, int k, int num_sms);
// topk_ids / topk_weights: where the router writes (both nullptr: the
// workspace region); region: d.bytes of workspace (zeroed once, left
// reusable); router_tickets:
// the header's router tickets; counters: int32[3] of the header (zeroed once).
int launch_decode_layer(const void* hidden, const void* gate, const float* bias, const void* w13,
                        const void* w2, int T, int H, int F, int E, int k, int scoring,
                        int n_group, int topk_group, int renormalize, float scaling, void* out,
                        int32_t* topk_ids, float* topk_weights, char* region,
                        int* router_tickets, int* counters, int* err, const DecodePlan& d,
                        int num_sms, cudaStream_t stream);

// ---- floor probes (measurement) -------------------------------------------------
int launch_probe_empty(int blocks, int threads, cudaStream_t stream);
int launch_probe_read(const void* p, size_t bytes, int* sink, cudaStream_t stream);

int device_num_sms();

// 2-D bf16 tensor map of a row-major [rows, cols] matrix: 128-byte swizzle,
// box = 64 columns x box_rows rows, zero fill out of bounds.
bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_rows);
// 2-D byte tensor map of a row-major [rows, cols] byte matrix: 128-byte
// swizzle, box = 128 bytes x box_rows rows, zero fill out of bounds.
bool make_map_u8_sw128(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_rows);
// 2-D map of a row-major [rows, cols] matrix of e2m1 codes packed two per
// byte (low nibble first): each 16 codes land in shared memory as their 8
// packed bytes followed by an 8-byte gap that the copy leaves untouched (the
// operand layout of the block-scaled MMA for 4-bit types); 128-byte swizzle,
// box = 128 codes x box_rows rows.  base must be 32-byte aligned and cols a
// multiple of 128.  A load completes cols/2 * rows bytes of transactions
// (the packed size), not the shared-memory footprint.
bool make_map_e2m1(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_rows);

}  // namespace moe
