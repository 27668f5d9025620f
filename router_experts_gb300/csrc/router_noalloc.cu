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

constexpr int kMaxTokenTiles = 16384;                    // tickets: T <= 262,144
constexpr size_t kTicketBytes = 4ull * kMaxTokenTiles;   // 64 KiB
constexpr size_t kLogitBytes = MOE_ROUTER_NOALLOC_MAX_LOGIT_BYTES;  // 8 MiB
constexpr size_t kScratchBytes = kTicketBytes + kLogitBytes;

static __device__ __align__(256) unsigned char g_router_noalloc_scratch[kScratchBytes];

// The array's device address belongs to one CUDA context: after
// cudaDeviceReset (or when the caller makes another context current) the
// module is loaded again and the array may sit elsewhere.  The address is
// therefore cached per device together with the unique id of the context it
// was looked up in, and looked up again whenever the current context differs.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct CachedAddress {
  unsigned long long ctx_id;
  void* addr;
};

std::mutex g_mu;
CachedAddress g_cache[64] = {};
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Unique id of the calling thread's current context (false if none is
// current yet).  Called with g_mu held.
bool current_context_id(unsigned long long* id) {
  if (!g_ctx_get_current || !g_ctx_get_id) {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) !=
            cudaSuccess ||
        qa != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
            cudaSuccess ||
        qb != cudaDriverEntryPointSuccess)
      return false;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(a);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(b);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current device's current
// context (host code only ever holds a host-side stand-in for the symbol, so
// the address must come from the runtime).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long id = 0;
  const bool have_ctx = current_context_id(&id);
  if (!have_ctx || g_cache[dev].addr == nullptr || g_cache[dev].ctx_id != id) {
    void* p = nullptr;
    // (the lookup also makes the device's primary context current if no
    // context was current yet)
    if (cudaGetSymbolAddress(&p, g_router_noalloc_scratch) != cudaSuccess || p == nullptr)
      return -1;
    if (!current_context_id(&id)) return -1;
    g_cache[dev].ctx_id = id;
    g_cache[dev].addr = p;
  }
  *out = g_cache[dev].addr;
  return 0;
}

}  // namespace

extern "C" int moe_router_noalloc(const void* hidden, int hidden_dt, const uint8_t* hidden_scale,
                                  const void* gate, int gate_dt, const float* bias, int T, int H,
                                  int E, int k, int scoring, int n_group, int topk_group,
                                  int renormalize, float scaling, int32_t* topk_ids,
                                  float* topk_weights, void* stream) {
  // the same argument rules as moe_router
  const int rc = moe::check_router(hidden, hidden_dt, hidden_scale, gate, gate_dt, T, H, E, k,
                                   scoring, n_group, topk_group);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!topk_ids || !topk_weights) return MOE_ERR_ARG;

  // the static array bounds the problem size
  const moe::RouterPlan plan = moe::plan_router(T, H, E, false);
  if (plan.nt > kMaxTokenTiles || plan.scratch_bytes > kLogitBytes) return MOE_ERR_ARG;

  void* base = nullptr;
  if (scratch_address(&base) != 0) return MOE_ERR_CUDA;
  char* b = static_cast<char*>(base);
  int* tickets = reinterpret_cast<int*>(b);
  float* logits = reinterpret_cast<float*>(b + kTicketBytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // the array keeps the previous call's contents: the tickets must start at 0
  if (cudaMemsetAsync(tickets, 0, sizeof(int) * plan.nt, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_router(hidden, hidden_dt, hidden_scale, gate, gate_dt, bias, T, H, E, k, scoring,
                         n_group, topk_group, renormalize, scaling, topk_ids, topk_weights, logits,
                         tickets, /*err=*/nullptr, plan, s) != 0)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
