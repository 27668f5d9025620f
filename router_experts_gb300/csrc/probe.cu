// probe.cu -- the two kernels that measure a router's floor on this GPU.
//
// Follows "How an MoE Model Picks Its Experts During LLM Inference" §3.3, The
// Floor: the least a router can cost is one launch plus one cold read of the
// gate weight.  The page measures it with kernels that do no useful work: an
// empty kernel (one block, or as many blocks as the read below), and a kernel
// whose every thread loads 16 bytes of the gate so that the whole matrix is
// read once.  The loaded bytes feed a comparison whose store almost never
// happens, so the loads cannot be removed; the sink is written only if the
// 16 bytes XOR to one particular word.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kProbeThreads = 512;

__global__ void __launch_bounds__(kProbeThreads) probe_empty_kernel() {}

__global__ void __launch_bounds__(kProbeThreads)
    probe_read_kernel(const uint4* __restrict__ p, long long n16, int* sink) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n16) return;
  const uint4 v = p[i];
  if ((v.x ^ v.y ^ v.z ^ v.w) == 0x9E3779B9u) *sink = static_cast<int>(i);
}

}  // namespace

int launch_probe_empty(int blocks, int threads, cudaStream_t stream) {
  probe_empty_kernel<<<blocks, threads, 0, stream>>>();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_probe_read(const void* p, size_t bytes, int* sink, cudaStream_t stream) {
  const long long n16 = static_cast<long long>(bytes / 16);
  const long long blocks = (n16 + kProbeThreads - 1) / kProbeThreads;
  probe_read_kernel<<<static_cast<unsigned>(blocks), kProbeThreads, 0, stream>>>(
      static_cast<const uint4*>(p), n16, sink);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace moe
