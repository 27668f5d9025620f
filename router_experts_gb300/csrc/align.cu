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
// Pass 1 counts the segment into the warp's shared-memory histogram row.  Then, per expert, an exclusive scan over the 32 warp rows
// gives each warp its base inside the expert, and a block-wide exclusive scan
// of the padded counts gives the experts' starts.  Pass 2 re-walks the segment
// in 32-assignment chunks: one ballot per id bit finds the lanes holding the
// same expert, position = start[e] + warp base + rank among those lanes to the
// left, and the group leader advances the warp's running base.  When the
// problem fits in shared memory, pass 2 places into a compact shared-memory
// array and a final sweep writes sorted_ids (pads and tail included) and the
// block table with coalesced stores; a single SM issuing tens of thousands of
// scattered 4-byte stores is otherwise the bottleneck.
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

// Mask of the lanes holding the same expert id as this lane (0 for an invalid
// lane), from one ballot per id bit: the lanes that agree with this lane on
// every bit.
MOE_DEV unsigned match_lanes(int e, bool valid, int nbits) {
  unsigned m = __ballot_sync(0xffffffffu, valid);
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (e >> b) & 1;
    const unsigned v = __ballot_sync(0xffffffffu, bit);
    m &= bit ? v : ~v;
  }
  return valid ? m : 0u;
}

// Expert id of assignment a: from the shared-memory copy when the ids were
// staged (STAGED), else from global memory.  Invalid ids read as -1.
template <bool STAGED>
MOE_DEV int load_id(const int32_t* __restrict__ ids, const uint16_t* sid, int a, int E) {
  if constexpr (STAGED) {
    const int v = sid[a];
    return v == 0xFFFF ? -1 : v;
  } else {
    const int v = __ldg(ids + a);
    return (v >= 0 && v < E) ? v : -1;
  }
}

// Shared-memory layout of the compact (STAGED) variant, in 32-bit words:
//   cnt[32][E] | tot[E] | start[E] | cstart[E] | wsum[32] | blk[nbc]
//   | sid[n] (uint16) | out[n] (uint16)
struct AlignSmem {
  size_t words, bytes;
};
inline AlignSmem align_smem(int n, int E, long long nbc) {
  AlignSmem m;
  m.words = 32 * static_cast<size_t>(E) + 3 * static_cast<size_t>(E) + 32 + nbc;
  m.bytes = m.words * 4 + align_up(static_cast<size_t>(n) * 2, 16) * 2;
  return m;
}

// STAGED: ids staged in shared memory (16-bit) and the sorted assignment ids
// built in shared memory first, so every global store is coalesced.
// Otherwise (problems too large for shared memory): ids read from global
// memory and placed with scattered stores.
template <bool STAGED>
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
  int* cstart = start + E;    // [E] start of each expert among the real assignments
  int* wsum = cstart + E;     // [32]
  int* blk = wsum + 32;       // [nblocks_cap] (STAGED) expert of each block
  uint16_t* sid = reinterpret_cast<uint16_t*>(blk + (STAGED ? nblocks_cap : 0));
  uint16_t* out = sid + align_up(static_cast<size_t>(n), 8);  // [n] (STAGED)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int nbits = 32 - __clz(max(E - 1, 1));

  for (int i = tid; i < 32 * E; i += kAlignThreads) cnt[i] = 0;
  bool bad = false;
  if constexpr (STAGED) {
    // coalesced copy of the ids into shared memory as 16-bit values; each
    // thread issues several independent loads before it stores
    constexpr int kU = 8;
    for (int a0s = tid; a0s < n; a0s += kAlignThreads * kU) {
      int v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int a = a0s + u * kAlignThreads;
        v[u] = (a < n) ? __ldg(ids + a) : 0;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int a = a0s + u * kAlignThreads;
        if (a < n) {
          const bool ok = v[u] >= 0 && v[u] < E;
          bad |= !ok;
          sid[a] = ok ? static_cast<uint16_t>(v[u]) : static_cast<uint16_t>(0xFFFF);
        }
      }
    }
  }
  __syncthreads();

  const int per_warp = ((n + 31) / 32 + 31) / 32 * 32;
  const int a0 = warp * per_warp;
  const int a1 = min(n, a0 + per_warp);

  // pass 1: per-warp histogram (shared-memory atomics on the warp's own row)
  for (int a = a0 + lane; a < a1; a += 32) {
    const int e = load_id<STAGED>(ids, sid, a, E);
    if (e >= 0) atomicAdd(&cnt[warp * E + e], 1);
    else if constexpr (!STAGED) bad = true;
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

  // exclusive scans over experts (E <= 1024: one expert per thread) of the
  // padded counts (starts in sorted_ids) and of the real counts (compact starts)
  const int cnt_e = (tid < E) ? tot[tid] : 0;
  const int pad = (cnt_e + BM - 1) / BM * BM;
  const int incl = warp_incl_scan(pad);
  const int cincl = warp_incl_scan(cnt_e);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) wsum[lane] = warp_incl_scan(wsum[lane]);
  __syncthreads();
  const int excl = incl - pad + (warp > 0 ? wsum[warp - 1] : 0);
  const int total = wsum[31];
  __syncthreads();
  if (lane == 31) wsum[warp] = cincl;
  __syncthreads();
  if (warp == 0) wsum[lane] = warp_incl_scan(wsum[lane]);
  __syncthreads();
  const int cexcl = cincl - cnt_e + (warp > 0 ? wsum[warp - 1] : 0);
  if (tid < E) {
    start[tid] = excl;
    cstart[tid] = cexcl;
  }
  __syncthreads();
  // warp bases: compact positions (STAGED) or positions in sorted_ids
  for (int i = tid; i < 32 * E; i += kAlignThreads)
    cnt[i] += STAGED ? cstart[i % E] : start[i % E];
  if constexpr (STAGED) {
    for (int e = tid; e < E; e += kAlignThreads) {
      const int s = start[e], p = (tot[e] + BM - 1) / BM * BM;
      for (int b = s / BM; b < (s + p) / BM; ++b) blk[b] = e;
    }
  }
  __syncthreads();

  // pass 2: place in order.  The lane masks of a group of chunks do not depend
  // on each other, so they are computed first; the running positions are then
  // advanced chunk by chunk.
  constexpr int kGroup = 8;
  for (int g0 = a0; g0 < a1; g0 += 32 * kGroup) {
    const int nch = min(kGroup, (a1 - g0 + 31) / 32);
    int ev[kGroup];
    unsigned mv[kGroup];
#pragma unroll
    for (int c = 0; c < kGroup; ++c) {
      if (c < nch) {
        const int a = g0 + 32 * c + lane;
        ev[c] = (a < a1) ? load_id<STAGED>(ids, sid, a, E) : -1;
        mv[c] = match_lanes(ev[c], ev[c] >= 0, nbits);
      }
    }
#pragma unroll
    for (int c = 0; c < kGroup; ++c) {
      if (c < nch) {
        const int a = g0 + 32 * c + lane;
        const int e = ev[c];
        const unsigned m = mv[c];
        const int pos0 = (e >= 0) ? cnt[warp * E + e] : 0;
        __syncwarp();
        if (e >= 0) {
          const int pos = pos0 + __popc(m & lt_mask);
          if constexpr (STAGED) out[pos] = static_cast<uint16_t>(a);
          else sorted_ids[pos] = a;
          if (lane == __ffs(m) - 1) cnt[warp * E + e] = pos0 + __popc(m);
        }
        __syncwarp();
      }
    }
  }

  if constexpr (STAGED) {
    __syncthreads();
    // coalesced write-out: every padded position looks up its block's expert
    const long long nb_used = total / BM;
    for (long long p = tid; p < cap; p += kAlignThreads) {
      int v = n;
      if (p < total) {
        const int e = blk[p / BM];
        const int r = static_cast<int>(p) - start[e];
        if (r < tot[e]) v = out[cstart[e] + r];
      }
      sorted_ids[p] = v;
    }
    for (long long b = tid; b < nblocks_cap; b += kAlignThreads)
      block_expert[b] = (b < nb_used) ? blk[b] : -1;
  } else {
    // padding rows of every expert and the block table
    for (int e = tid; e < E; e += kAlignThreads) {
      const int s = start[e], c = tot[e], p = (c + BM - 1) / BM * BM;
      for (int pos = s + c; pos < s + p; ++pos) sorted_ids[pos] = n;
      for (int b = s / BM; b < (s + p) / BM; ++b) block_expert[b] = e;
    }
    // tail up to the capacity
    for (long long pos = total + tid; pos < cap; pos += kAlignThreads) sorted_ids[pos] = n;
    for (long long b = total / BM + tid; b < nblocks_cap; b += kAlignThreads) block_expert[b] = -1;
  }
  if (tid == 0) *npp = total;
}

}  // namespace

int launch_align(const int32_t* topk_ids, int T, int k, int E, int block_m, int32_t* sorted_ids,
                 int64_t cap_rows, int32_t* block_expert, int32_t* num_post_padded, int* err,
                 cudaStream_t stream) {
  const int n = T * k;
  const long long nbc = (cap_rows + block_m - 1) / block_m;
  const AlignSmem staged = align_smem(n, E, nbc);
  const size_t plain = (32 * static_cast<size_t>(E) + 3 * static_cast<size_t>(E) + 32) * 4;
  constexpr size_t kMaxSmem = 227 * 1024;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(align_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kMaxSmem)) != cudaSuccess ||
        cudaFuncSetAttribute(align_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kMaxSmem)) != cudaSuccess)
      return -1;
    attr_set = true;
  }
  // 16-bit staging holds assignment ids below 65,535 and expert ids below 65,535
  if (staged.bytes <= kMaxSmem && n < 65535)
    align_kernel<true><<<1, kAlignThreads, staged.bytes, stream>>>(
        topk_ids, n, E, block_m, sorted_ids, cap_rows, block_expert, nbc, num_post_padded, err);
  else
    align_kernel<false><<<1, kAlignThreads, plain, stream>>>(
        topk_ids, n, E, block_m, sorted_ids, cap_rows, block_expert, nbc, num_post_padded, err);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace moe
