// align.cu -- moe_align_block_size in one launch, deterministic, no host sync.
//
// Follows "MoE Kernels, in depth", Alignment (count per expert, round each
// count up to BLOCK_M, exclusive prefix sum, expert-sorted block-padded order,
// sentinel T*k for padding, expert of every block, padded length read by the
// GEMMs from device memory; buffers sized for T*k + E*(BLOCK_M-1)) and
// "Mixture of Experts", vLLM's Triton path (the worked example; block entries
// past the padded length are -1).  Where the pages' CUDA kernel places rows
// with atomics (order within an expert varies run to run), this kernel places
// them in ascending assignment id, so its output is unique.
//
// One CTA of 1024 threads.  Warp w owns a contiguous segment of assignments.
// Pass 1: per 32-assignment chunk, __match_any_sync groups lanes with the same
// expert and the group leader adds the group size to the warp's shared-memory
// histogram row.  Then, per expert, an exclusive scan over the 32 warp rows
// gives each warp its base inside the expert, and a block-wide exclusive scan
// of the padded counts gives the experts' starts.  Pass 2 re-walks the segment
// in order: position = start[e] + warp base + rank among equal lanes to the
// left; the leader advances the warp's running base.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kAlignThreads = 1024;

MOE_DEV int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

__global__ void __launch_bounds__(kAlignThreads) align_kernel(const int32_t* __restrict__ ids,
                                                              int n, int E, int BM,
                                                              int32_t* __restrict__ sorted_ids,
                                                              long long cap,
                                                              int32_t* __restrict__ block_expert,
                                                              long long nblocks_cap,
                                                              int32_t* __restrict__ npp, int* err) {
  extern __shared__ int sm[];
  int* cnt = sm;              // [32][E]: warp histogram, then running positions
  int* tot = cnt + 32 * E;    // [E] assignments per expert
  int* start = tot + E;       // [E] padded start of each expert
  int* wsum = start + E;      // [32]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned lt_mask = (1u << lane) - 1u;

  for (int i = tid; i < 32 * E; i += kAlignThreads) cnt[i] = 0;
  __syncthreads();

  const int per_warp = ((n + 31) / 32 + 31) / 32 * 32;
  const int a0 = warp * per_warp;
  const int a1 = min(n, a0 + per_warp);

  bool bad = false;
  for (int base = a0; base < a1; base += 32) {
    const int a = base + lane;
    const bool act = a < a1;
    const int e = act ? __ldg(ids + a) : -1;
    const bool ok = act && e >= 0 && e < E;
    bad |= act && !ok;
    const int key = ok ? e : (0x40000000 | lane);  // invalid lanes match nobody
    const unsigned m = __match_any_sync(0xffffffffu, key);
    if (ok && lane == __ffs(m) - 1) cnt[warp * E + e] += __popc(m);
  }
  if (bad) raise_error(err, kErrBadExpert);
  __syncthreads();

  for (int e = tid; e < E; e += kAlignThreads) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += c;
    }
    tot[e] = run;
  }
  __syncthreads();

  // exclusive scan of the padded counts (E <= 1024: one expert per thread)
  const int pad = (tid < E) ? (tot[tid] + BM - 1) / BM * BM : 0;
  const int incl = warp_incl_scan(pad);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) wsum[lane] = warp_incl_scan(wsum[lane]);
  __syncthreads();
  const int excl = incl - pad + (warp > 0 ? wsum[warp - 1] : 0);
  if (tid < E) start[tid] = excl;
  const int total = wsum[31];
  __syncthreads();
  for (int i = tid; i < 32 * E; i += kAlignThreads) cnt[i] += start[i % E];
  __syncthreads();

  for (int base = a0; base < a1; base += 32) {
    const int a = base + lane;
    const bool act = a < a1;
    const int e = act ? __ldg(ids + a) : -1;
    const bool ok = act && e >= 0 && e < E;
    const int key = ok ? e : (0x40000000 | lane);
    const unsigned m = __match_any_sync(0xffffffffu, key);
    const int pos0 = ok ? cnt[warp * E + e] : 0;
    __syncwarp();
    if (ok) {
      sorted_ids[pos0 + __popc(m & lt_mask)] = a;
      if (lane == __ffs(m) - 1) cnt[warp * E + e] = pos0 + __popc(m);
    }
    __syncwarp();
  }

  // padding rows of every expert and the block table
  for (int e = tid; e < E; e += kAlignThreads) {
    const int s = start[e], c = tot[e], p = (c + BM - 1) / BM * BM;
    for (int pos = s + c; pos < s + p; ++pos) sorted_ids[pos] = n;
    for (int b = s / BM; b < (s + p) / BM; ++b) block_expert[b] = e;
  }
  // tail up to the capacity
  for (long long pos = total + tid; pos < cap; pos += kAlignThreads) sorted_ids[pos] = n;
  for (long long b = total / BM + tid; b < nblocks_cap; b += kAlignThreads) block_expert[b] = -1;
  if (tid == 0) *npp = total;
}

}  // namespace

int launch_align(const int32_t* topk_ids, int T, int k, int E, int block_m, int32_t* sorted_ids,
                 int64_t cap_rows, int32_t* block_expert, int32_t* num_post_padded, int* err,
                 cudaStream_t stream) {
  const int n = T * k;
  const size_t smem = (32 * static_cast<size_t>(E) + 2 * E + 32) * sizeof(int);
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             32 * 1024 * 4 + 2 * 1024 * 4 + 128) != cudaSuccess)
      return -1;
    attr_set = true;
  }
  const long long nbc = (cap_rows + block_m - 1) / block_m;
  align_kernel<<<1, kAlignThreads, smem, stream>>>(topk_ids, n, E, block_m, sorted_ids, cap_rows,
                                                    block_expert, nbc, num_post_padded, err);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace moe
