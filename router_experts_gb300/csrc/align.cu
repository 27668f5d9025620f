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
// One cooperative launch of G CTAs (G grows with T*k, one CTA per 512
// assignments, at most 16), 16 warps each.  CTA c owns a contiguous segment
// of the assignments and warp w a contiguous piece of it.
//   1. Count: each warp counts its piece into its shared-memory histogram row;
//      a scan over the 16 rows gives each warp its base inside the CTA and the
//      CTA's count per expert, published to a [G][E] table in the workspace.
//   2. One grid barrier.  Every CTA then reads the table's E columns: the
//      total per expert and the CTA's base = the counts of the CTAs before it.
//      A block-wide scan of the padded totals gives the experts' starts.
//   3. Place: each warp re-walks its piece in 32-assignment chunks; one ballot
//      per id bit finds the lanes holding the same expert; position = start +
//      CTA base + warp base + rank among those lanes to the left; the group
//      leader advances the running base.  Positions are disjoint across CTAs.
//   4. Fill: the pads of every expert, the tail up to the capacity, and the
//      block table are split over all warps of the grid.
// With G = 1 (small T*k) step 2 reads the CTA's own counts and skips the
// barrier; with at most 32 assignments one warp does the counting and placing
// (align_few).
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kAlignThreads = 512;
constexpr int kAlignWarps = kAlignThreads / 32;
// one CTA per 512 assignments, at most 16 (more spend longer in the grid
// barrier): align_partition in moe_internal.h
static_assert(16 <= kAlignMaxCtas, "per-CTA histogram rows of the workspace");

struct AlignArgs {
  const int32_t* ids;
  int32_t* sorted;
  int32_t* blk;
  int32_t* npp;
  int* hist;  // [G][E]
  int* bar;
  int* err;
  const long long* wait_limit;  // workspace test hook: barrier limit in cycles, 0 = default
  int* ticket;                  // precounted: CTAs done reading hist
  long long cap, nbc;
  int n, E, BM, G, seg;
  int precounted;               // hist already holds every CTA's counts (the router's)
};

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

MOE_DEV int load_id(const int32_t* __restrict__ ids, int a, int E) {
  const int v = __ldg(ids + a);
  return (v >= 0 && v < E) ? v : -1;
}

// Few assignments (n <= 32, decode): warp 0 handles them all with warp
// intrinsics -- the lanes with the same expert (one ballot per id bit), each
// group's start = the padded counts of the groups with smaller expert ids,
// each assignment's slot = start + its rank in its group -- and records the
// groups in expert order; then every thread fills its share of the pads, the
// tail and the block table.  Same output as the general path.
MOE_DEV void align_few(const AlignArgs& a, int* sm) {
  int* ge = sm;        // [32] expert of group g (expert order)
  int* gs = sm + 32;   // [32] padded start
  int* gc = sm + 64;   // [32] assignments
  int* gt = sm + 96;   // [2] groups, padded total
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, BM = a.BM;
  if (warp == 0) {
    int e = -1;
    if (lane < a.n) {
      e = load_id(a.ids, lane, E);
      if (e < 0) raise_error(a.err, kErrBadExpert);
    }
    const unsigned m = match_lanes(e, e >= 0, 32 - __clz(max(E - 1, 1)));
    const bool leader = e >= 0 && lane == __ffs(m) - 1;
    const int cnt = __popc(m);
    const int pad = (cnt + BM - 1) / BM * BM;
    int start = 0, g = 0;
    for (int j = 0; j < 32; ++j) {
      const int ej = __shfl_sync(0xffffffffu, e, j);
      const int lj = __shfl_sync(0xffffffffu, leader ? 1 : 0, j);
      const int pj = __shfl_sync(0xffffffffu, pad, j);
      if (lj && ej < e) {
        start += pj;
        ++g;
      }
    }
    if (e >= 0) {
      const int pos = start + __popc(m & ((1u << lane) - 1u));
      if (pos < a.cap) a.sorted[pos] = lane;
    }
    if (leader) {
      ge[g] = e;
      gs[g] = start;
      gc[g] = cnt;
    }
    const int total = __reduce_add_sync(0xffffffffu, leader ? pad : 0);
    const int ng = __popc(__ballot_sync(0xffffffffu, leader));
    if (lane == 0) {
      gt[0] = ng;
      gt[1] = total;
      *a.npp = total;
    }
  }
  __syncthreads();
  const int ng = gt[0], total = gt[1];
  // pads inside the groups and the tail: n; data slots were written above
  for (long long p = tid; p < a.cap; p += kAlignThreads) {
    bool pad_slot = p >= total;
    for (int g = 0; !pad_slot && g < ng; ++g)
      if (p >= gs[g] + gc[g] && p < gs[g] + (gc[g] + BM - 1) / BM * BM) pad_slot = true;
    if (pad_slot) a.sorted[p] = a.n;
  }
  for (long long b = tid; b < a.nbc; b += kAlignThreads) {
    const long long p0 = b * BM;
    int e = -1;
    for (int g = 0; g < ng; ++g)
      if (p0 >= gs[g] && p0 < gs[g] + (gc[g] + BM - 1) / BM * BM) e = ge[g];
    a.blk[b] = e;
  }
}

// Shared memory, 32-bit words: cnt[16][E] | tot[E] | start[E] | base[E] | wsum[32]
inline size_t align_smem_bytes(int E) {
  return (static_cast<size_t>(kAlignWarps) * E + 3 * static_cast<size_t>(E) + 32) * 4;
}

__global__ void __launch_bounds__(kAlignThreads) align_kernel(const AlignArgs a) {
  extern __shared__ int sm[];
  if (a.n <= 32) {
    align_few(a, sm);
    return;
  }
  const int E = a.E, BM = a.BM;
  int* cnt = sm;                      // [16][E]: warp histogram, then running positions
  int* tot = cnt + kAlignWarps * E;   // [E] assignments per expert (whole problem)
  int* start = tot + E;               // [E] padded start of each expert
  int* base = start + E;              // [E] this CTA's count, then its base per expert
  int* wsum = base + E;               // [32]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int nbits = 32 - __clz(max(E - 1, 1));

  // this CTA's segment and this warp's piece of it
  const int s0 = min(a.n, c * a.seg), s1 = min(a.n, s0 + a.seg);
  const int per_warp = ((s1 - s0 + kAlignWarps - 1) / kAlignWarps + 31) / 32 * 32;
  const int w0 = min(s1, s0 + warp * per_warp), w1 = min(s1, w0 + per_warp);

  for (int i = tid; i < kAlignWarps * E; i += kAlignThreads) cnt[i] = 0;
  __syncthreads();

  // 1. count (shared-memory atomics on the warp's own row)
  bool bad = false;
  for (int p = w0 + lane; p < w1; p += 32) {
    const int e = load_id(a.ids, p, E);
    if (e >= 0) atomicAdd(&cnt[warp * E + e], 1);
    else bad = true;
  }
  if (bad) raise_error(a.err, kErrBadExpert);
  __syncthreads();
  for (int e = tid; e < E; e += kAlignThreads) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kAlignWarps; ++w) {
      const int v = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += v;
    }
    base[e] = run;
    if (a.G > 1 && !a.precounted) a.hist[static_cast<size_t>(c) * E + e] = run;
  }

  // 2. totals and this CTA's base per expert
  if (a.G > 1) {
    // on a timed-out barrier the table is incomplete: write nothing.  With
    // the router's counts the table is complete before the launch: no barrier
    if (!a.precounted &&
        !grid_barrier(a.bar, a.G, a.err, a.wait_limit ? __ldcg(a.wait_limit) : 0))
      return;
    for (int e = tid; e < E; e += kAlignThreads) {
      int t = 0, b = 0;
      for (int c0 = 0; c0 < a.G; c0 += 8) {
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          v[u] = (c0 + u < a.G) ? __ldcg(a.hist + static_cast<size_t>(c0 + u) * E + e) : 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          t += v[u];
          b += (c0 + u < c) ? v[u] : 0;
        }
      }
      tot[e] = t;
      base[e] = b;
    }
    {
      // the last CTA to have read the table zeroes it, so it is all zeros
      // between calls (the router of the next layer call adds its counts to
      // it)
      __syncthreads();
      if (tid == 0) {
        const int old = ticket_add_acq_rel(a.ticket, 1);
        const int last = old == a.G - 1;
        if (last) store_relaxed_gpu(a.ticket, 0);
        wsum[0] = last;
      }
      __syncthreads();
      if (wsum[0]) {
        for (int i = tid; i < a.G * E; i += kAlignThreads) a.hist[i] = 0;
      }
      __syncthreads();
    }
  } else {
    for (int e = tid; e < E; e += kAlignThreads) {
      tot[e] = base[e];
      base[e] = 0;
    }
  }
  __syncthreads();

  // exclusive scan over experts of the padded counts (two experts per thread,
  // E <= 1024)
  const int ea = 2 * tid, eb = 2 * tid + 1;
  const int pa = (ea < E) ? (tot[ea] + BM - 1) / BM * BM : 0;
  const int pb = (eb < E) ? (tot[eb] + BM - 1) / BM * BM : 0;
  const int incl = warp_incl_scan(pa + pb);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = (lane < kAlignWarps) ? wsum[lane] : 0;
    const int s = warp_incl_scan(v);
    if (lane < kAlignWarps) wsum[lane] = s;
  }
  __syncthreads();
  const int excl = incl - pa - pb + (warp > 0 ? wsum[warp - 1] : 0);
  const int total = wsum[kAlignWarps - 1];
  if (ea < E) start[ea] = excl;
  if (eb < E) start[eb] = excl + pa;
  __syncthreads();
  // running positions: expert start + CTA base + warp base
  for (int i = tid; i < kAlignWarps * E; i += kAlignThreads) {
    const int e = i % E;
    cnt[i] += start[e] + base[e];
  }
  __syncthreads();

  // 3. place in ascending assignment order.  The lane masks of a group of
  // chunks do not depend on each other, so they are computed first; the
  // running positions are then advanced chunk by chunk.
  constexpr int kGroup = 4;
  for (int g0 = w0; g0 < w1; g0 += 32 * kGroup) {
    int ev[kGroup];
    unsigned mv[kGroup];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const int p = g0 + 32 * u + lane;
      ev[u] = (p < w1) ? load_id(a.ids, p, E) : -1;
    }
#pragma unroll
    for (int u = 0; u < kGroup; ++u) mv[u] = match_lanes(ev[u], ev[u] >= 0, nbits);
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const int p = g0 + 32 * u + lane;
      const int e = ev[u];
      const unsigned m = mv[u];
      const int pos0 = (e >= 0) ? cnt[warp * E + e] : 0;
      __syncwarp();
      if (e >= 0) {
        const int pos = pos0 + __popc(m & lt_mask);
        if (pos >= 0 && pos < a.cap) a.sorted[pos] = p;
        if (lane == __ffs(m) - 1) cnt[warp * E + e] = pos0 + __popc(m);
      }
      __syncwarp();
    }
  }

  // 4. fill, split over every warp of the grid: each expert's pad rows and
  // blocks, then the tail of sorted_ids and of the block table
  const int gw = c * kAlignWarps + warp, nw = a.G * kAlignWarps;
  // (every write is bounded by the buffer sizes, so a table corrupted
  // outside this kernel cannot send a write out of range)
  for (int e = gw; e < E; e += nw) {
    const int s = start[e], t = tot[e], pd = (t + BM - 1) / BM * BM;
    for (int p = s + t + lane; p < s + pd; p += 32)
      if (p >= 0 && p < a.cap) a.sorted[p] = a.n;
    for (int b = s / BM + lane; b < (s + pd) / BM; b += 32)
      if (b >= 0 && b < a.nbc) a.blk[b] = e;
  }
  const long long gt = static_cast<long long>(c) * kAlignThreads + tid;
  const long long nt = static_cast<long long>(a.G) * kAlignThreads;
  const long long tail = total < 0 ? 0 : total;
  for (long long p = tail + gt; p < a.cap; p += nt) a.sorted[p] = a.n;
  for (long long b = tail / BM + gt; b < a.nbc; b += nt) a.blk[b] = -1;
  if (c == 0 && tid == 0) *a.npp = total;
}

}  // namespace

int launch_align(const int32_t* topk_ids, int T, int k, int E, int block_m, int32_t* sorted_ids,
                 int64_t cap_rows, int32_t* block_expert, int32_t* num_post_padded, int* hist,
                 int* bar, int* err, const long long* wait_limit, cudaStream_t stream,
                 bool precounted, int* ticket) {
  if (E > kAlignMaxE) return -1;
  AlignArgs a;
  a.wait_limit = wait_limit;
  a.ticket = ticket;
  a.ids = topk_ids;
  a.sorted = sorted_ids;
  a.blk = block_expert;
  a.npp = num_post_padded;
  a.hist = hist;
  a.bar = bar;
  a.err = err;
  a.cap = cap_rows;
  a.nbc = (cap_rows + block_m - 1) / block_m;
  a.n = T * k;
  a.E = E;
  a.BM = block_m;
  align_partition(a.n, &a.G, &a.seg);
  a.precounted = (precounted && a.G > 1 && a.n > 32) ? 1 : 0;
  if (a.G > 1 && ticket == nullptr) return -1;
  // (align_few uses 98 words whatever E is)
  const size_t smem = align_smem_bytes(E) > 512 ? align_smem_bytes(E) : 512;
  static std::atomic<unsigned long long> smem_set{0};
  if (!ensure_smem_limit(reinterpret_cast<const void*>(align_kernel),
                         static_cast<int>(align_smem_bytes(kAlignMaxE)), smem_set))
    return -1;
  // the CTAs meet at a grid barrier: a cooperative launch guarantees that
  // all of them are resident at once (or fails to launch)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(a.G);
  cfg.blockDim = dim3(kAlignThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = (a.G > 1) ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, align_kernel, a) != cudaSuccess) return -1;
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace moe
