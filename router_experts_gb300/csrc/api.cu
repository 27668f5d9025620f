// api.cu -- the C ABI declared in include/moe.h: host-side argument checks,
// workspace layout and the stream-ordered launches of the kernels.
#include <stdio.h>
#include <string.h>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace moe {

static thread_local char g_last_cuda_error[256] = "";

static int cuda_fail(const char* what, cudaError_t e) {
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", what, cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}
static int launch_fail(const char* what) {
  const cudaError_t e = cudaGetLastError();
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", what,
           e == cudaSuccess ? "launch rejected" : cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

int device_num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---- layouts ------------------------------------------------------------------
struct FfnLayout {
  size_t inter, partial, xperm, xperm_scale, total;  // offsets from the region start
};
// The intermediate: bf16 [cap, F]; low-bit: e4m3 codes [cap, F] then UE8M0
// scales [cap, F/32].
static size_t inter_bytes(size_t cap, int F, int act_dt) {
  if (act_dt == MOE_DT_E4M3) return align_up(cap * F, 256) + align_up(cap * (F / 32), 256);
  return align_up(cap * F * 2, 256);
}
// Low-bit: GEMM1's token rows permuted into the padded order (e4m3 codes
// [cap, H] and scale bytes [cap, H/32]) follow the split-K partials.
static FfnLayout ffn_layout(int T, int H, int F, int E, int k, int block_m, bool with_inter,
                            int act_dt = MOE_DT_BF16) {
  FfnLayout L{};
  size_t off = 0;
  const size_t cap = static_cast<size_t>(T) * k + static_cast<size_t>(E) * (block_m - 1);
  if (with_inter) {
    L.inter = off;
    off += inter_bytes(cap, F, act_dt);
  }
  L.partial = off;
  off += ffn_partial_bytes(block_m);
  L.xperm = L.xperm_scale = 0;
  if (act_dt == MOE_DT_E4M3) {
    L.xperm = off;
    off += align_up(cap * H, 256);
    L.xperm_scale = off;
    off += align_up(cap * (H / 32), 256);
  }
  L.total = off;
  return L;
}

struct LayerLayout {
  size_t ids, wts, sorted, blk, npp, stage, router, ffn, xq, xs, total;
  int64_t cap;
};
static LayerLayout layer_layout(int T, int H, int F, int E, int k, int block_m,
                                int act_dt = MOE_DT_BF16) {
  LayerLayout L{};
  size_t off = kWsHeaderBytes;
  const size_t nk = static_cast<size_t>(T) * k;
  L.cap = static_cast<int64_t>(nk) + static_cast<int64_t>(E) * (block_m - 1);
  L.ids = off;
  off += align_up(nk * 4, 256);
  L.wts = off;
  off += align_up(nk * 4, 256);
  L.sorted = off;
  off += align_up(static_cast<size_t>(L.cap) * 4, 256);
  L.blk = off;
  off += align_up(static_cast<size_t>((L.cap + block_m - 1) / block_m) * 4, 256);
  L.npp = off;
  off += 256;
  L.stage = off;
  off += align_up(nk * H * 2, 256);
  L.router = off;
  off += plan_router(T, H, E).scratch_bytes;
  L.ffn = off;
  off += ffn_layout(T, H, F, E, k, block_m, true, act_dt).total;
  // a bf16 hidden may feed low-bit experts: room for its FP8 cast (the
  // low-bit intermediate is smaller than the bf16 one reserved above)
  L.xq = L.xs = 0;
  if (act_dt == MOE_DT_BF16) {
    L.xq = off;
    off += align_up(static_cast<size_t>(T) * H, 256);
    L.xs = off;
    off += align_up(static_cast<size_t>(T) * (H / 32), 256);
  }
  L.total = off;
  return L;
}

static int* err_word(void* ws) { return reinterpret_cast<int*>(static_cast<char*>(ws) + kWsErrOffset); }
static int* align_hist(void* ws) {
  return reinterpret_cast<int*>(static_cast<char*>(ws) + kWsAlignHistOffset);
}
static int* align_bar(void* ws) {
  return reinterpret_cast<int*>(static_cast<char*>(ws) + kWsAlignBarrierOffset);
}
static int* align_ticket(void* ws) {
  return reinterpret_cast<int*>(static_cast<char*>(ws) + kWsAlignTicketOffset);
}
static const long long* wait_limit_word(void* ws) {
  return reinterpret_cast<const long long*>(static_cast<char*>(ws) + kWsWaitLimitOffset);
}
static_assert(kWsAlignBarrierOffset == MOE_WS_ALIGN_BARRIER_OFFSET, "header layout");
static_assert(kWsWaitLimitOffset == MOE_WS_WAIT_LIMIT_OFFSET, "header layout");

// ---- checks -------------------------------------------------------------------
// Host-side argument rules of the router (moe_router, moe_router_noalloc and
// the router step of moe_layer).
int check_router(const void* hidden, int hidden_dt, const uint8_t* hidden_scale,
                 const void* gate, int gate_dt, int T, int H, int E, int k, int scoring,
                 int n_group, int topk_group) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0) return MOE_ERR_ARG;
  if (k > E || k > 16 || E > 512 || H % 32 != 0) return MOE_ERR_ARG;
  if (T > 16 * kRouterMaxTiles) return MOE_ERR_ARG;
  if (scoring != MOE_SCORING_SOFTMAX && scoring != MOE_SCORING_SIGMOID &&
      scoring != MOE_SCORING_SQRT_SOFTPLUS)
    return MOE_ERR_ARG;
  if (n_group < 1 || n_group > 32) return MOE_ERR_ARG;
  if (n_group > 1) {
    if (E % n_group != 0 || E / n_group < 2) return MOE_ERR_ARG;
    if (topk_group < 1 || topk_group > n_group) return MOE_ERR_ARG;
    if (topk_group * (E / n_group) < k) return MOE_ERR_ARG;
  }
  if (hidden_dt != MOE_DT_BF16 && hidden_dt != MOE_DT_F32 && hidden_dt != MOE_DT_E4M3)
    return MOE_ERR_UNSUPPORTED;
  if (gate_dt != MOE_DT_BF16 && gate_dt != MOE_DT_F32) return MOE_ERR_UNSUPPORTED;
  if (T > 0) {
    if (!hidden || !gate) return MOE_ERR_ARG;
    if (hidden_dt == MOE_DT_E4M3 && !hidden_scale) return MOE_ERR_ARG;
    if (!aligned(hidden, 16) || !aligned(gate, 16)) return MOE_ERR_ARG;
  }
  return MOE_OK;
}

static int check_block_m(int block_m) {
  return (block_m == 16 || block_m == 64 || block_m == 128) ? MOE_OK : MOE_ERR_ARG;
}

static int check_ffn(int act_dt, int w_dt, int T, int H, int F, int E, int k, int block_m,
                     int64_t cap_rows) {
  if (T < 0 || H <= 0 || F <= 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_ARG;
  if (H % 64 != 0 || F % 32 != 0) return MOE_ERR_ARG;
  if (check_block_m(block_m) != MOE_OK) return MOE_ERR_ARG;
  if (cap_rows < static_cast<int64_t>(T) * k + static_cast<int64_t>(E) * (block_m - 1))
    return MOE_ERR_ARG;
  if (cap_rows > 0x7fffffffll || static_cast<int64_t>(E) * 2 * F > 0x7fffffffll ||
      static_cast<int64_t>(E) * H > 0x7fffffffll)
    return MOE_ERR_ARG;
  if (act_dt == MOE_DT_BF16 && w_dt == MOE_DT_BF16) return MOE_OK;
  if (act_dt == MOE_DT_E4M3 && w_dt == MOE_DT_E2M1)
    // both contractions in whole 128-value steps: every scale row is a whole
    // number of 4-byte words
    return (F % 128 == 0 && H % 128 == 0) ? MOE_OK : MOE_ERR_ARG;
  return MOE_ERR_UNSUPPORTED;
}

static FfnParams ffn_params(int T, int H, int F, int E, int k, int block_m,
                            const int32_t* sorted_ids, const int32_t* block_expert,
                            const int32_t* npp, int64_t cap_rows, void* ws, size_t region_off,
                            const FfnLayout& L) {
  FfnParams p{};
  p.sorted_ids = sorted_ids;
  p.block_expert = block_expert;
  p.num_post_padded = npp;
  p.partial = reinterpret_cast<float*>(static_cast<char*>(ws) + region_off + L.partial);
  p.tickets = reinterpret_cast<int*>(static_cast<char*>(ws) + kWsFfnTicketOffset);
  p.err = err_word(ws);
  p.T = T;
  p.H = H;
  p.F = F;
  p.E = E;
  p.k = k;
  p.cap_rows = static_cast<int>(cap_rows);
  p.max_slots = ffn_max_slots(block_m) < kFfnMaxTickets ? ffn_max_slots(block_m) : kFfnMaxTickets;
  return p;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported combination";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE: return "device error word set";
  }
  return "unknown status";
}

const char* moe_last_cuda_error_string(void) { return g_last_cuda_error; }

int moe_pick_block_m(int T, int k, int E) {
  if (E <= 0) return 16;
  const long long tk = static_cast<long long>(T) * k;
  if (tk < 8ll * E) return 16;
  if (tk < 64ll * E) return 64;
  return 128;
}

int moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < kWsHeaderBytes) return MOE_ERR_ARG;
  const cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail("cudaMemsetAsync", e);
}

int moe_read_device_error(void* ws, int32_t* code, int clear, void* stream) {
  if (!ws || !code) return MOE_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
  int32_t v = 0;
  e = cudaMemcpy(&v, err_word(ws), sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail("cudaMemcpy", e);
  *code = v;
  if (clear && v) {
    e = cudaMemset(err_word(ws), 0, sizeof(int32_t));
    if (e != cudaSuccess) return cuda_fail("cudaMemset", e);
  }
  return v ? MOE_ERR_DEVICE : MOE_OK;
}

// ---- router -------------------------------------------------------------------
size_t moe_router_workspace_bytes(int T, int H, int E) {
  if (T < 0 || H <= 0 || E <= 0) return 0;
  return kWsHeaderBytes + plan_router(T, H, E).scratch_bytes;
}

int moe_router_kernel_count(int T, int H, int E, int hidden_dt, int gate_dt) {
  if (T <= 0 || H <= 0 || E <= 0) return 0;
  const RouterPlan p = plan_router(T, H, E);
  if (!router_uses_tiled(p, hidden_dt, gate_dt)) return 1;
  return (p.fused_select ? 1 : 2) + ((hidden_dt == MOE_DT_E4M3 || gate_dt == MOE_DT_F32) ? 1 : 0);
}

int moe_router(const void* hidden, int hidden_dt, const uint8_t* hidden_scale, const void* gate,
               int gate_dt, const float* bias, int T, int H, int E, int k, int scoring,
               int n_group, int topk_group, int renormalize, float scaling, int32_t* topk_ids,
               float* topk_weights, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_router(hidden, hidden_dt, hidden_scale, gate, gate_dt, T, H, E, k, scoring,
                        n_group, topk_group);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!topk_ids || !topk_weights || !ws) return MOE_ERR_ARG;
  if (ws_bytes < moe_router_workspace_bytes(T, H, E) || !aligned(ws, 256)) return MOE_ERR_ARG;
  const RouterPlan plan = plan_router(T, H, E);
  char* base = static_cast<char*>(ws);
  if (launch_router(hidden, hidden_dt, hidden_scale, gate, gate_dt, bias, T, H, E, k, scoring,
                    n_group, topk_group, renormalize, scaling, topk_ids, topk_weights,
                    reinterpret_cast<float*>(base + kWsHeaderBytes),
                    reinterpret_cast<int*>(base + kWsRouterTicketOffset), err_word(ws), plan,
                    static_cast<cudaStream_t>(stream)) != 0)
    return launch_fail("router kernel");
  return MOE_OK;
}

int moe_router_cast_e4m3(const void* hidden, const void* gate, int gate_dt, const float* bias,
                         int T, int H, int E, int k, int scoring, int n_group, int topk_group,
                         int renormalize, float scaling, int32_t* topk_ids, float* topk_weights,
                         uint8_t* codes, uint8_t* scales, void* ws, size_t ws_bytes,
                         void* stream) {
  int rc = check_router(hidden, MOE_DT_BF16, nullptr, gate, gate_dt, T, H, E, k, scoring,
                        n_group, topk_group);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!topk_ids || !topk_weights || !codes || !scales || !ws || !aligned(codes, 16))
    return MOE_ERR_ARG;
  if (ws_bytes < moe_router_workspace_bytes(T, H, E) || !aligned(ws, 256)) return MOE_ERR_ARG;
  const RouterPlan plan = plan_router(T, H, E);
  char* base = static_cast<char*>(ws);
  if (launch_router(hidden, MOE_DT_BF16, nullptr, gate, gate_dt, bias, T, H, E, k, scoring,
                    n_group, topk_group, renormalize, scaling, topk_ids, topk_weights,
                    reinterpret_cast<float*>(base + kWsHeaderBytes),
                    reinterpret_cast<int*>(base + kWsRouterTicketOffset), err_word(ws), plan,
                    static_cast<cudaStream_t>(stream), codes, scales) != 0)
    return launch_fail("router kernel");
  return MOE_OK;
}

// ---- align --------------------------------------------------------------------
size_t moe_align_workspace_bytes(void) { return kWsHeaderBytes; }

int moe_align(const int32_t* topk_ids, int T, int k, int E, int block_m, int32_t* sorted_ids,
              int64_t cap_rows, int32_t* block_expert, int32_t* num_post_padded, void* ws,
              size_t ws_bytes, void* stream) {
  if (T < 0 || k <= 0 || E <= 0 || E > 1024) return MOE_ERR_ARG;
  if (check_block_m(block_m) != MOE_OK) return MOE_ERR_ARG;
  if (cap_rows < static_cast<int64_t>(T) * k + static_cast<int64_t>(E) * (block_m - 1) ||
      cap_rows > 0x7fffffffll)
    return MOE_ERR_ARG;
  if ((T > 0 && !topk_ids) || !sorted_ids || !block_expert || !num_post_padded || !ws)
    return MOE_ERR_ARG;
  if (ws_bytes < kWsHeaderBytes || !aligned(ws, 256)) return MOE_ERR_ARG;
  if (launch_align(topk_ids, T, k, E, block_m, sorted_ids, cap_rows, block_expert,
                   num_post_padded, align_hist(ws), align_bar(ws), err_word(ws),
                   wait_limit_word(ws), static_cast<cudaStream_t>(stream), false,
                   align_ticket(ws)) != 0)
    return launch_fail("align kernel");
  return MOE_OK;
}

// ---- expert GEMMs --------------------------------------------------------------
size_t moe_ffn_workspace_bytes(int T, int H, int F, int E, int k, int block_m, int act_dt) {
  (void)H;
  if (T < 0 || F <= 0 || E <= 0 || k <= 0 || check_block_m(block_m) != MOE_OK) return 0;
  return kWsHeaderBytes + ffn_layout(T, H, F, E, k, block_m, true, act_dt).total;
}

// Low-bit path: kind 0 reads x codes/scales and writes the e4m3 intermediate
// (codes + scales); kind 1 reads it and writes the bf16 stage.
static int expert_gemm_lowbit(int kind, const void* act, const uint8_t* act_scale,
                              const void* w, const uint8_t* w_scale, int T, int H, int F, int E,
                              int k, int block_m, const int32_t* sorted_ids,
                              const int32_t* block_expert, const int32_t* npp, int64_t cap_rows,
                              uint8_t* inter_q, uint8_t* inter_scale, const float* topk_weights,
                              void* stage, void* ws, cudaStream_t stream, int naive = 0,
                              uint8_t* xperm = nullptr, uint8_t* xperm_scale = nullptr) {
  if (!act || !act_scale || !w || !w_scale || !sorted_ids || !block_expert || !npp || !ws)
    return MOE_ERR_ARG;
  if (kind == 0 && (!inter_q || !inter_scale)) return MOE_ERR_ARG;
  if (kind == 1 && (!topk_weights || !stage)) return MOE_ERR_ARG;
  if (!aligned(act, 16) || !aligned(w, 32) || !aligned(act_scale, 4) || !aligned(w_scale, 4) ||
      (inter_q && !aligned(inter_q, 32)) || (inter_scale && !aligned(inter_scale, 4)) ||
      (stage && !aligned(stage, 32)))
    return MOE_ERR_ARG;
  LowbitParams p{};
  p.sorted_ids = sorted_ids;
  p.block_expert = block_expert;
  p.num_post_padded = npp;
  p.act = static_cast<const uint8_t*>(act);
  p.act_scale = act_scale;
  p.w = static_cast<const uint8_t*>(w);
  p.w_scale = w_scale;
  p.inter_q = inter_q;
  p.inter_scale = inter_scale;
  p.topk_weights = topk_weights;
  p.stage = static_cast<__nv_bfloat16*>(stage);
  p.err = err_word(ws);
  p.T = T;
  p.H = H;
  p.F = F;
  p.E = E;
  p.k = k;
  p.BM = block_m;
  p.cap_rows = static_cast<int>(cap_rows);
  p.naive = naive;
  const int sms = device_num_sms();
  if (sms <= 0) return cuda_fail("cudaDeviceGetAttribute", cudaGetLastError());
  if (launch_lowbit_gemm(kind, p, sms, stream, xperm, xperm_scale) != 0)
    return launch_fail("low-bit GEMM kernel");
  return MOE_OK;
}

static int expert_gemm(int kind, const void* act, int act_dt, const void* w, int w_dt, int T,
                       int H, int F, int E, int k, int block_m, const int32_t* sorted_ids,
                       const int32_t* block_expert, const int32_t* npp, int64_t cap_rows,
                       void* inter, const float* topk_weights, void* stage, void* ws,
                       size_t ws_bytes, bool inter_in_ws, cudaStream_t stream) {
  int rc = check_ffn(act_dt, w_dt, T, H, F, E, k, block_m, cap_rows);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!act || !w || !sorted_ids || !block_expert || !npp || !ws) return MOE_ERR_ARG;
  if (kind == 0 && !inter) return MOE_ERR_ARG;
  if (kind == 1 && (!topk_weights || !stage)) return MOE_ERR_ARG;
  // the intermediate and the stage are written with 32-byte stores
  if (!aligned(ws, 256) || !aligned(act, 16) || !aligned(w, 16) || (inter && !aligned(inter, 32)) ||
      (stage && !aligned(stage, 32)))
    return MOE_ERR_ARG;
  const FfnLayout L = ffn_layout(T, H, F, E, k, block_m, inter_in_ws);
  if (ws_bytes < kWsHeaderBytes + L.total) return MOE_ERR_ARG;
  FfnParams p = ffn_params(T, H, F, E, k, block_m, sorted_ids, block_expert, npp, cap_rows, ws,
                           kWsHeaderBytes, L);
  if (kind == 0) {
    p.x = act;
    p.inter = inter;
  } else {
    p.inter = const_cast<void*>(act);
    p.topk_weights = topk_weights;
    p.stage = stage;
  }
  const int sms = device_num_sms();
  if (sms <= 0) return cuda_fail("cudaDeviceGetAttribute", cudaGetLastError());
  const char* why = "";
  if (launch_ffn_gemm(kind, block_m, w, p, sms, stream, &why) != 0) return launch_fail(why);
  return MOE_OK;
}

int moe_expert_gemm1(const void* x, int act_dt, const uint8_t* x_scale, const void* w13,
                     const uint8_t* w13_scale, int w_dt, int T, int H, int F, int E, int k,
                     int block_m, const int32_t* sorted_ids, const int32_t* block_expert,
                     const int32_t* num_post_padded, int64_t cap_rows, void* inter,
                     uint8_t* inter_scale, void* ws, size_t ws_bytes, void* stream) {
  if (act_dt == MOE_DT_E4M3) {
    const int rc = check_ffn(act_dt, w_dt, T, H, F, E, k, block_m, cap_rows);
    if (rc != MOE_OK) return rc;
    if (T == 0) return MOE_OK;
    if (ws_bytes < kWsHeaderBytes || !aligned(ws, 256)) return MOE_ERR_ARG;
    // a workspace of moe_ffn_workspace_bytes holds the permuted token rows
    // (read by TMA); a smaller one gets the gathering kernel
    const FfnLayout L = ffn_layout(T, H, F, E, k, block_m, false, MOE_DT_E4M3);
    const bool room = ws_bytes >= kWsHeaderBytes + L.total &&
                      cap_rows <= static_cast<int64_t>(T) * k + static_cast<int64_t>(E) * (block_m - 1);
    char* base = static_cast<char*>(ws) + kWsHeaderBytes;
    return expert_gemm_lowbit(0, x, x_scale, w13, w13_scale, T, H, F, E, k, block_m, sorted_ids,
                              block_expert, num_post_padded, cap_rows,
                              static_cast<uint8_t*>(inter), inter_scale, nullptr, nullptr, ws,
                              static_cast<cudaStream_t>(stream), 0,
                              room ? reinterpret_cast<uint8_t*>(base + L.xperm) : nullptr,
                              room ? reinterpret_cast<uint8_t*>(base + L.xperm_scale) : nullptr);
  }
  return expert_gemm(0, x, act_dt, w13, w_dt, T, H, F, E, k, block_m, sorted_ids, block_expert,
                     num_post_padded, cap_rows, inter, nullptr, nullptr, ws, ws_bytes, false,
                     static_cast<cudaStream_t>(stream));
}

int moe_expert_gemm2(const void* inter, const uint8_t* inter_scale, int act_dt, const void* w2,
                     const uint8_t* w2_scale, int w_dt, int T, int H, int F, int E, int k,
                     int block_m, const int32_t* sorted_ids, const int32_t* block_expert,
                     const int32_t* num_post_padded, int64_t cap_rows,
                     const float* topk_weights, void* stage, void* ws, size_t ws_bytes,
                     void* stream) {
  if (act_dt == MOE_DT_E4M3) {
    const int rc = check_ffn(act_dt, w_dt, T, H, F, E, k, block_m, cap_rows);
    if (rc != MOE_OK) return rc;
    if (T == 0) return MOE_OK;
    if (ws_bytes < kWsHeaderBytes || !aligned(ws, 256)) return MOE_ERR_ARG;
    return expert_gemm_lowbit(1, inter, inter_scale, w2, w2_scale, T, H, F, E, k, block_m,
                              sorted_ids, block_expert, num_post_padded, cap_rows, nullptr,
                              nullptr, topk_weights, stage, ws, static_cast<cudaStream_t>(stream));
  }
  return expert_gemm(1, inter, act_dt, w2, w_dt, T, H, F, E, k, block_m, sorted_ids,
                     block_expert, num_post_padded, cap_rows, nullptr, topk_weights, stage, ws,
                     ws_bytes, false, static_cast<cudaStream_t>(stream));
}

int moe_grouped_ffn(const void* x, const uint8_t* x_scale, int act_dt, const void* w13,
                    const uint8_t* w13_scale, const void* w2, const uint8_t* w2_scale, int w_dt,
                    int T, int H, int F, int E, int k, int block_m, const int32_t* sorted_ids,
                    const int32_t* block_expert, const int32_t* num_post_padded,
                    int64_t cap_rows, const float* topk_weights, void* stage, void* ws,
                    size_t ws_bytes, void* stream) {
  int rc = check_ffn(act_dt, w_dt, T, H, F, E, k, block_m, cap_rows);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!ws || !aligned(ws, 256)) return MOE_ERR_ARG;
  if (ws_bytes < moe_ffn_workspace_bytes(T, H, F, E, k, block_m, act_dt)) return MOE_ERR_ARG;
  if (cap_rows != static_cast<int64_t>(T) * k + static_cast<int64_t>(E) * (block_m - 1))
    return MOE_ERR_ARG;  // the workspace holds exactly the worst-case intermediate
  const FfnLayout L = ffn_layout(T, H, F, E, k, block_m, true, act_dt);
  void* inter = static_cast<char*>(ws) + kWsHeaderBytes + L.inter;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (act_dt == MOE_DT_E4M3) {
    uint8_t* iq = static_cast<uint8_t*>(inter);
    uint8_t* isc = iq + align_up(static_cast<size_t>(cap_rows) * F, 256);
    char* region = static_cast<char*>(ws) + kWsHeaderBytes;
    rc = expert_gemm_lowbit(0, x, x_scale, w13, w13_scale, T, H, F, E, k, block_m, sorted_ids,
                            block_expert, num_post_padded, cap_rows, iq, isc, nullptr, nullptr,
                            ws, s, 0, reinterpret_cast<uint8_t*>(region + L.xperm),
                            reinterpret_cast<uint8_t*>(region + L.xperm_scale));
    if (rc != MOE_OK) return rc;
    return expert_gemm_lowbit(1, iq, isc, w2, w2_scale, T, H, F, E, k, block_m, sorted_ids,
                              block_expert, num_post_padded, cap_rows, nullptr, nullptr,
                              topk_weights, stage, ws, s);
  }
  rc = expert_gemm(0, x, act_dt, w13, w_dt, T, H, F, E, k, block_m, sorted_ids, block_expert,
                   num_post_padded, cap_rows, inter, nullptr, nullptr, ws, ws_bytes, true, s);
  if (rc != MOE_OK) return rc;
  return expert_gemm(1, inter, act_dt, w2, w_dt, T, H, F, E, k, block_m, sorted_ids,
                     block_expert, num_post_padded, cap_rows, nullptr, topk_weights, stage, ws,
                     ws_bytes, true, s);
}

// ---- finalize -------------------------------------------------------------------
int moe_finalize(const void* stage, int T, int k, int H, void* out, void* stream) {
  if (T < 0 || k <= 0 || H <= 0 || H % 8 != 0) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!stage || !out || !aligned(stage, 16) || !aligned(out, 16)) return MOE_ERR_ARG;
  if (launch_finalize(stage, T, k, H, out, static_cast<cudaStream_t>(stream)) != 0)
    return launch_fail("finalize kernel");
  return MOE_OK;
}

// One token skips the alignment: every block holds one assignment ("Mixture
// of Experts": vLLM's naive block assignment, there for T*k*4 <= E).  A
// token's k experts are distinct, so these are exactly align's blocks; with
// more tokens two assignments may share an expert, and separate blocks would
// stream that expert's weights twice (measured: DeepSeek-V3, 8 tokens, 836 us
// instead of 388), so the shortcut stops at one token.  The intermediate
// needs k*BLOCK_M rows, within the capacity k + E*(BLOCK_M-1) as k <= E.
static bool layer_skips_align(int T, int k, int E) {
  (void)k;
  (void)E;
  return T == 1;
}

// ---- persistent layer for small batches ------------------------------------------
size_t moe_layer_persistent_workspace_bytes(int T, int H, int F, int E, int k) {
  if (T < 1 || H <= 0 || F <= 0 || E <= 0 || k <= 0) return 0;
  const DecodePlan d = plan_decode(T, H, F, E, k, device_num_sms() > 0 ? device_num_sms() : 152);
  return d.ok ? kWsHeaderBytes + d.bytes : 0;
}

int moe_layer_persistent(const void* hidden, const void* gate, const float* bias, const void* w13,
                         const void* w2, int T, int H, int F, int E, int k, int scoring,
                         int n_group, int topk_group, int renormalize, float scaling, void* out,
                         int32_t* topk_ids, float* topk_weights, void* ws, size_t ws_bytes,
                         void* stream) {
  int rc = check_router(hidden, MOE_DT_BF16, nullptr, gate, MOE_DT_BF16, T, H, E, k, scoring,
                        n_group, topk_group);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (F <= 0) return MOE_ERR_ARG;
  // shape limits first (any SM count), then the plan for this GPU
  if (!plan_decode(T, H, F, E, k, 1 << 20).ok) return MOE_ERR_ARG;
  if (!w13 || !w2 || !out || !ws) return MOE_ERR_ARG;
  if (!aligned(w13, 16) || !aligned(w2, 16) || !aligned(out, 16) || !aligned(ws, 256))
    return MOE_ERR_ARG;
  if ((topk_ids == nullptr) != (topk_weights == nullptr)) return MOE_ERR_ARG;
  const int sms = device_num_sms();
  if (sms <= 0) return cuda_fail("cudaDeviceGetAttribute", cudaGetLastError());
  const DecodePlan d = plan_decode(T, H, F, E, k, sms);
  if (!d.ok) return MOE_ERR_ARG;
  if (ws_bytes < kWsHeaderBytes + d.bytes) return MOE_ERR_ARG;
  char* base = static_cast<char*>(ws);
  if (launch_decode_layer(hidden, gate, bias, w13, w2, T, H, F, E, k, scoring, n_group,
                          topk_group, renormalize, scaling, out, topk_ids, topk_weights,
                          base + kWsHeaderBytes,
                          reinterpret_cast<int*>(base + kWsRouterTicketOffset),
                          reinterpret_cast<int*>(base + kWsDecodeCounterOffset), err_word(ws),
                          d, sms, static_cast<cudaStream_t>(stream)) != 0)
    return launch_fail("persistent layer kernel");
  return MOE_OK;
}

// ---- floor probes -----------------------------------------------------------------
int moe_probe_empty(int blocks, int threads, void* stream) {
  if (blocks < 1 || blocks > (1 << 20) || threads < 1 || threads > 512) return MOE_ERR_ARG;
  if (launch_probe_empty(blocks, threads, static_cast<cudaStream_t>(stream)) != 0)
    return launch_fail("probe kernel");
  return MOE_OK;
}

int moe_probe_read(const void* p, size_t bytes, int32_t* sink, void* stream) {
  if (!p || !sink || bytes < 16 || bytes % 16 != 0 || !aligned(p, 16) ||
      bytes / 16 > (static_cast<size_t>(1) << 40))
    return MOE_ERR_ARG;
  if (launch_probe_read(p, bytes, sink, static_cast<cudaStream_t>(stream)) != 0)
    return launch_fail("probe kernel");
  return MOE_OK;
}

// ---- FP8 cast -------------------------------------------------------------------
int moe_cast_e4m3(const void* x, int T, int H, uint8_t* codes, uint8_t* scales, void* stream) {
  if (T < 0 || H <= 0 || H % 32 != 0) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 16)) return MOE_ERR_ARG;
  if (launch_cast_e4m3(x, T, H, codes, scales, static_cast<cudaStream_t>(stream)) != 0)
    return launch_fail("cast kernel");
  return MOE_OK;
}

// ---- layer ------------------------------------------------------------------------
size_t moe_layer_workspace_bytes(int T, int H, int F, int E, int k, int block_m, int act_dt) {
  if (T < 0 || H <= 0 || F <= 0 || E <= 0 || k <= 0) return 0;
  if (block_m == 0) block_m = moe_pick_block_m(T, k, E);
  if (check_block_m(block_m) != MOE_OK) return 0;
  return layer_layout(T, H, F, E, k, block_m, act_dt).total;
}

int moe_layer_kernel_count(int T, int H, int F, int E, int k, int act_dt, int gate_dt,
                           int w_dt) {
  if (T <= 0 || H <= 0 || F <= 0 || E <= 0 || k <= 0) return 0;
  // router + align (none for single-assignment blocks), GEMM1, GEMM2,
  // finalize (the FP8 cast of a bf16 hidden for e2m1 experts rides in the
  // router's selection launch; an e4m3 hidden's rows are permuted into the
  // blocks' padded order by one more launch in front of GEMM1)
  const int align = layer_skips_align(T, k, E) ? 0 : 1;
  const int perm = (act_dt == MOE_DT_E4M3 && w_dt == MOE_DT_E2M1) ? 1 : 0;
  return moe_router_kernel_count(T, H, E, act_dt, gate_dt) + align + 3 + perm;
}

int moe_layer(const void* hidden, int act_dt, const uint8_t* hidden_scale, const void* gate,
              int gate_dt, const float* bias, const void* w13, const uint8_t* w13_scale,
              const void* w2, const uint8_t* w2_scale, int w_dt, int T, int H, int F, int E,
              int k, int scoring, int n_group, int topk_group, int renormalize, float scaling,
              int block_m, void* out, void* ws, size_t ws_bytes, void* stream) {
  if (block_m == 0) block_m = moe_pick_block_m(T, k, E);
  int rc = check_router(hidden, act_dt, hidden_scale, gate, gate_dt, T, H, E, k, scoring,
                        n_group, topk_group);
  if (rc != MOE_OK) return rc;
  const LayerLayout L = layer_layout(T, H, F, E, k, block_m, act_dt);
  // a bf16 hidden with e2m1 experts: the router reads the bf16 rows, the
  // experts their FP8 cast (made here, in front of the expert GEMMs)
  const bool cast_input = act_dt == MOE_DT_BF16 && w_dt == MOE_DT_E2M1;
  const int ffn_dt = cast_input ? MOE_DT_E4M3 : act_dt;
  rc = check_ffn(ffn_dt, w_dt, T, H, F, E, k, block_m, L.cap);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!out || !ws || !w13 || !w2) return MOE_ERR_ARG;
  if (cast_input && !aligned(hidden, 16)) return MOE_ERR_ARG;
  if (ws_bytes < L.total || !aligned(ws, 256)) return MOE_ERR_ARG;
  char* base = static_cast<char*>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* ids = reinterpret_cast<int32_t*>(base + L.ids);
  float* wts = reinterpret_cast<float*>(base + L.wts);
  int32_t* sorted = reinterpret_cast<int32_t*>(base + L.sorted);
  int32_t* blk = reinterpret_cast<int32_t*>(base + L.blk);
  int32_t* npp = reinterpret_cast<int32_t*>(base + L.npp);
  void* stage = base + L.stage;
  const RouterPlan plan = plan_router(T, H, E);
  // a bf16 hidden for e2m1 experts: the router's selecting warps also write
  // the rows' FP8 cast ("How GPUs Fuse ..." §1.1), so no separate cast launch
  uint8_t* cq = cast_input ? reinterpret_cast<uint8_t*>(base + L.xq) : nullptr;
  uint8_t* cs = cast_input ? reinterpret_cast<uint8_t*>(base + L.xs) : nullptr;
  // with more than one align CTA, the router's selecting warps count the
  // assignments of every align segment as they select ("How an MoE Model
  // Picks Its Experts ..." §6.1), so the align launch needs no grid barrier
  const int naive = layer_skips_align(T, k, E) ? 1 : 0;
  int align_g = 1, align_seg = 0;
  align_partition(T * k, &align_g, &align_seg);
  const bool precount = !naive && align_g > 1 && T * k > 32;
  if (launch_router(hidden, act_dt, hidden_scale, gate, gate_dt, bias, T, H, E, k, scoring,
                    n_group, topk_group, renormalize, scaling, ids, wts,
                    reinterpret_cast<float*>(base + L.router),
                    reinterpret_cast<int*>(base + kWsRouterTicketOffset), err_word(ws), plan,
                    s, cq, cs, precount ? align_hist(ws) : nullptr, align_seg) != 0)
    return launch_fail("router kernel");
  if (naive) {
    // the GEMMs read the router's ids as the block table and need no other
    // align output (the pointers below are never dereferenced)
    blk = ids;
    sorted = ids;
    npp = ids;
  } else if (launch_align(ids, T, k, E, block_m, sorted, L.cap, blk, npp, align_hist(ws),
                          align_bar(ws), err_word(ws), wait_limit_word(ws), s, precount,
                          align_ticket(ws)) != 0) {
    return launch_fail("align kernel");
  }
  const FfnLayout FL = ffn_layout(T, H, F, E, k, block_m, true, ffn_dt);
  void* inter = base + L.ffn + FL.inter;
  if (ffn_dt == MOE_DT_E4M3) {
    const void* xq = cast_input ? static_cast<const void*>(cq) : hidden;
    const uint8_t* xs = cast_input ? cs : hidden_scale;
    if (!xs || !w13_scale || !w2_scale) return MOE_ERR_ARG;
    uint8_t* iq = static_cast<uint8_t*>(inter);
    uint8_t* isc = iq + align_up(static_cast<size_t>(L.cap) * F, 256);
    // an e4m3 hidden: its rows are permuted into the padded order in the
    // workspace (room reserved by the layout), so GEMM1 reads them by TMA; a
    // bf16 hidden's cast (whose workspace holds no permuted copy) is gathered
    uint8_t* xp = cast_input ? nullptr : reinterpret_cast<uint8_t*>(base + L.ffn + FL.xperm);
    uint8_t* xps =
        cast_input ? nullptr : reinterpret_cast<uint8_t*>(base + L.ffn + FL.xperm_scale);
    rc = expert_gemm_lowbit(0, xq, xs, w13, w13_scale, T, H, F, E, k, block_m,
                            sorted, blk, npp, L.cap, iq, isc, nullptr, nullptr, ws, s, naive,
                            xp, xps);
    if (rc != MOE_OK) return rc;
    rc = expert_gemm_lowbit(1, iq, isc, w2, w2_scale, T, H, F, E, k, block_m, sorted, blk, npp,
                            L.cap, nullptr, nullptr, wts, stage, ws, s, naive);
    if (rc != MOE_OK) return rc;
    if (launch_finalize(stage, T, k, H, out, s) != 0) return launch_fail("finalize kernel");
    return MOE_OK;
  }
  FfnParams p = ffn_params(T, H, F, E, k, block_m, sorted, blk, npp, L.cap, ws, L.ffn, FL);
  p.naive = naive;
  const int sms = device_num_sms();
  if (sms <= 0) return cuda_fail("cudaDeviceGetAttribute", cudaGetLastError());
  const char* why = "";
  p.x = hidden;
  p.inter = inter;
  if (launch_ffn_gemm(0, block_m, w13, p, sms, s, &why) != 0) return launch_fail(why);
  p.topk_weights = wts;
  p.stage = stage;
  if (launch_ffn_gemm(1, block_m, w2, p, sms, s, &why) != 0) return launch_fail(why);
  if (launch_finalize(stage, T, k, H, out, s) != 0) return launch_fail("finalize kernel");
  return MOE_OK;
}

}  // extern "C"
