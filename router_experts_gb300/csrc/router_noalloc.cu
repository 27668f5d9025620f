// router_noalloc.cu -- moe_router_noalloc: the router for callers that cannot
// allocate device memory.
//
// Some callers of this library cannot call cudaMalloc or any allocator: code
// running inside a host framework that owns all device memory and hands out
// only its own tensors, plugins loaded into a process whose memory pool must
// not grow, or hosts that forbid allocation after start-up.  moe_router needs
// a caller-provided workspace for its partial logits and tickets; this entry
// point instead uses one fixed array in device memory that is part of the
// library itself (a file-scope static __device__ array below).  Every GPU
// that loads the library holds that array until the process exits.
//
// The scratch array is shared by every call: a call leaves its partial logits
// and tickets in it, and the next call clears the tickets it needs before
// launching.  Two calls that run at the same time on the GPU (on different
// streams, or overlapping) race on the array and give wrong results.
#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace {

constexpr size_t kErrBytes = 256;                        // error word, padded
constexpr int kMaxTokenTiles = 16384;                    // tickets: T <= 262,144
constexpr size_t kTicketBytes = 4ull * kMaxTokenTiles;   // 64 KiB
constexpr size_t kLogitBytes = MOE_ROUTER_NOALLOC_MAX_LOGIT_BYTES;  // 8 MiB
constexpr size_t kScratchBytes = kErrBytes + kTicketBytes + kLogitBytes;

static __device__ __align__(256) unsigned char g_router_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[64] = {};

// Device address of the scratch array on the current device, looked up once
// per device (host code only ever holds a host-side stand-in for the symbol,
// so the address must come from the runtime).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_router_noalloc_scratch) != cudaSuccess || p == nullptr)
      return -1;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int moe_router_noalloc(const void* hidden, int hidden_dt, const uint8_t* hidden_scale,
                                  const void* gate, int gate_dt, const float* bias, int T, int H,
                                  int E, int k, int scoring, int n_group, int topk_group,
                                  int renormalize, float scaling, int32_t* topk_ids,
                                  float* topk_weights, void* stream) {
  // the same argument rules as moe_router
  if (T < 0 || H <= 0 || E <= 0 || k <= 0) return MOE_ERR_ARG;
  if (k > E || k > 16 || E > 512 || H % 32 != 0) return MOE_ERR_ARG;
  if (scoring != MOE_SCORING_SOFTMAX && scoring != MOE_SCORING_SIGMOID &&
      scoring != MOE_SCORING_SQRT_SOFTPLUS)
    return MOE_ERR_ARG;
  if (n_group < 1 || n_group > 32) return MOE_ERR_ARG;
  if (n_group > 1 && (E % n_group != 0 || E / n_group < 2 || topk_group < 1 ||
                      topk_group > n_group || topk_group * (E / n_group) < k))
    return MOE_ERR_ARG;
  if (hidden_dt != MOE_DT_BF16 && hidden_dt != MOE_DT_F32 && hidden_dt != MOE_DT_E4M3)
    return MOE_ERR_UNSUPPORTED;
  if (gate_dt != MOE_DT_BF16 && gate_dt != MOE_DT_F32) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!hidden || !gate || !topk_ids || !topk_weights) return MOE_ERR_ARG;
  if (hidden_dt == MOE_DT_E4M3 && !hidden_scale) return MOE_ERR_ARG;
  if (!aligned16(hidden) || !aligned16(gate)) return MOE_ERR_ARG;

  // the static array bounds the problem size
  const moe::RouterPlan plan = moe::plan_router(T, H, E, false);
  if (plan.nt > kMaxTokenTiles || plan.scratch_bytes > kLogitBytes) return MOE_ERR_ARG;

  void* base = nullptr;
  if (scratch_address(&base) != 0) return MOE_ERR_CUDA;
  char* b = static_cast<char*>(base);
  int* err = reinterpret_cast<int*>(b);
  int* tickets = reinterpret_cast<int*>(b + kErrBytes);
  float* logits = reinterpret_cast<float*>(b + kErrBytes + kTicketBytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // the array keeps the previous call's contents: the tickets must start at 0
  if (cudaMemsetAsync(tickets, 0, sizeof(int) * plan.nt, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_router(hidden, hidden_dt, hidden_scale, gate, gate_dt, bias, T, H, E, k, scoring,
                         n_group, topk_group, renormalize, scaling, topk_ids, topk_weights, logits,
                         tickets, err, plan, s) != 0)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
