// finalize.cu -- weighted combine back to token order.
//
// Follows "MoE Kernels, in depth", Combine (a gather in which each program
// owns a token and sums its k rows in a fixed order is deterministic),
// "Mixture of Experts" (ops.moe_sum reduces the top-k axis of the [T, k, H]
// cache; the routing weight was applied by the down GEMM) and "How GPUs Fuse
// Communication and Computation During LLM Inference" §3.7 (add the k slots
// as 32-bit floats in slot order, round once to 16 bits).  The staged rows
// are already bf16 (the down GEMM rounds each weighted slot row once), so an
// output is rounded twice in all: once per slot row in the stage and once
// here, after the fp32 sum.
//
// Memory-bound: one thread per 8 consecutive outputs (16-byte loads of each
// of the token's k staged rows, all issued before the first add when k <= 8,
// one 16-byte store).
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

// KMAX > 0: the k rows are loaded before any is added (k <= KMAX), so each
// thread keeps k 16-byte loads in flight; KMAX = 0: any k, one row at a time.
// Both add the rows in slot order, so their results are identical.
template <int KMAX>
__global__ void __launch_bounds__(256) finalize_kernel(const uint4* __restrict__ stage, int T,
                                                       int k, int H8, uint4* __restrict__ out) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(T) * H8) return;
  const long long t = idx / H8;
  const int c = static_cast<int>(idx % H8);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  auto add_row = [&](const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
      const float2 f = __bfloat1622float2(b);
      acc[2 * i] += f.x;
      acc[2 * i + 1] += f.y;
    }
  };
  const uint4* row = stage + t * k * H8 + c;
  if constexpr (KMAX > 0) {
    uint4 v[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k) v[j] = __ldg(row + static_cast<long long>(j) * H8);
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k) add_row(v[j]);
  } else {
    for (int j = 0; j < k; ++j) add_row(__ldg(row + static_cast<long long>(j) * H8));
  }
  out[t * H8 + c] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                               pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
}

}  // namespace

int launch_finalize(const void* stage, int T, int k, int H, void* out, cudaStream_t stream) {
  const int H8 = H / 8;
  const long long n = static_cast<long long>(T) * H8;
  const int blocks = static_cast<int>((n + 255) / 256);
  const uint4* st = reinterpret_cast<const uint4*>(stage);
  uint4* o = reinterpret_cast<uint4*>(out);
  if (k <= 8)
    finalize_kernel<8><<<blocks, 256, 0, stream>>>(st, T, k, H8, o);
  else
    finalize_kernel<0><<<blocks, 256, 0, stream>>>(st, T, k, H8, o);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace moe
