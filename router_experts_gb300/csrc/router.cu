// router.cu -- the fused router: gate GEMM to fp32 logits, softmax or sigmoid,
// fp32 selection bias, group-limited top-k (lowest expert id wins ties),
// renormalisation and routed scaling, in ONE launch.
//
// Follows "How an MoE Model Picks Its Experts During LLM Inference": §1.1
// (three steps), §1.3 (rank key = score + bias, weight = unbiased score),
// §2.4 (bf16 inputs, fp32 logits and bias), §4 (weights / (sum + 1e-20)),
// §5.1 (many CTAs each own a slice of experts so the cold gate read runs at
// memory speed), §5.3 (a warp owns a token row, k rounds, lowest id wins);
// and "Mixture of Experts" (DeepSeek's grouped, bias-corrected routing: group
// score = sum of the top-2 rank keys, keep topk_group groups, routed scaling).
//
// Layout of the work.  CTA (x, y, z) owns experts [x*ET, x*ET+ET), tokens
// [y*16, y*16+16) and the K slice z of KS.  Its 8 warps take 32-wide steps of
// the slice round-robin and multiply with mma.sync m16n8k16 (bf16 x bf16 ->
// fp32; fp32 sources are split into three bf16 parts so every product is
// exact).  A fixed-order shared-memory sum over warps gives the CTA's partial
// logits, stored to an L2-resident scratch.  The last CTA of a token tile to
// finish (atomic ticket, no spinning) sums the KS partials in order and runs
// the selection with one warp per token, the token's E logits in registers
// (E/32 per lane), and writes only the k ids and weights.
#include <cuda_fp8.h>

#include <algorithm>
#include <climits>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "router_device.cuh"

namespace moe {

namespace {

constexpr int kTargetCtas = 304;      // two CTAs per SM of a 152-SM part
// The tiled tensor-core path is used from the first token for bf16 gates and
// from 8 tokens for fp32 gates (whose three-plane conversion launch costs more
// than it saves on fewer tokens); measured on GB300 against the one-launch
// kernel at T = 1 .. 255 with L2 flushed.
constexpr int kTiledMinTokensF32Gate = 8;

template <int XDT, int GDT, int NB8>
__global__ void __launch_bounds__(kRouterThreads) router_kernel(const RouterArgs a) {
  __shared__ __align__(16) float sbuf[router_item_smem_floats<NB8>()];
  __shared__ int s_last;
  router_item<XDT, GDT, NB8>(a, blockIdx.x, blockIdx.y, blockIdx.z, gridDim.x * gridDim.z, sbuf,
                             &s_last);
}

// ---------------------------------------------------------------------------
// Tiled path for many tokens.  The fused kernel reads the gate once per
// 16-token tile, which at thousands of tokens turns the gate GEMM into T/16
// gate-sized L2 streams.  Here the gate GEMM runs on the 5th-generation tensor
// cores in 128-token tiles (operands staged by TMA, one thread issuing
// tcgen05.mma, fp32 logits accumulated in TMEM), with the K range split over
// CTAs so that one wave covers the GPU; a second kernel sums every token's
// split partials in split order and runs the same per-token selection as the
// fused kernel (one warp per token).  Operands that are not bf16 are first
// made exact bf16 operands: e4m3 x dequantised (an e4m3 value times a power
// of two is a bf16 number), an fp32 gate split into three bf16 planes that sum
// to the fp32 value, each plane multiplied and accumulated in turn.
// ---------------------------------------------------------------------------
constexpr int kRgThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM, warps 2-5 epilogue
constexpr int kRouterMaxSplits = 32;  // K splits of the tensor-core router (plan_router)
constexpr int kRgBK = 64;        // K elements per stage (128 bytes of bf16)
constexpr int kRgSmemBudget = 200 * 1024;
constexpr int kRgBarBytes = 256;

struct RgParams {
  float* part;   // [KS][T][E] fp32 partial logits
  int* err;
  int T, H, E, KS;
  int planes;    // B planes (1: bf16 gate, 3: fp32 gate split)
  int nb;        // N of one MMA (E, or E/2 when E > 256)
  int nmma;      // MMAs per K step (1 or 2)
  int stages, stage_bytes;
  uint32_t idesc;
};

// Every token's split partials summed in split order into the warp's row
// buffer, then the selection; one warp per token.
template <int S>
MOE_DEV void select_from_partials(const RouterArgs& a, const float* part, int t, float* row,
                                  const float* sbias) {
  const int lane = threadIdx.x & 31;
  const size_t slice = static_cast<size_t>(a.T) * a.E;
  const float* src = part + static_cast<size_t>(t) * a.E;
  float acc[S];
#pragma unroll
  for (int i = 0; i < S; ++i) acc[i] = 0.f;
  // every load of a group of four splits is issued before any of them is summed
  for (int s0 = 0; s0 < a.KS; s0 += 4) {
    float v[4][S];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int i = 0; i < S; ++i) {
        const int e = lane + 32 * i;
        v[u][i] = (s0 + u < a.KS && e < a.E) ? __ldcg(src + (s0 + u) * slice + e) : 0.f;
      }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int i = 0; i < S; ++i) acc[i] += v[u][i];
  }
#pragma unroll
  for (int i = 0; i < S; ++i)
    if (lane + 32 * i < a.E) row[lane + 32 * i] = acc[i];
  __syncwarp();
  select_token<S>(a, t, row, sbias);
  cast_token_row(a, t);
}

// S > 0 (few tokens): the CTA that finishes a token tile's K splits last
// (acquire-release ticket per token tile, no spinning) also sums the
// partials and selects the tile's tokens, one warp per token, so the router
// is one launch; S = ceil(E / 32).  S = 0: partials only (the selection is
// its own launch).
template <int S>
__global__ void __launch_bounds__(kRgThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ CUtensorMap tm_g, const RgParams p,
                       const RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int NS = p.stages;  // ring stages
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + NS * p.stage_bytes);
  uint64_t* empty_bar = full_bar + NS;
  uint64_t* acc_bar = empty_bar + NS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * 128, z = blockIdx.y;
  const int KB = p.H / kRgBK;
  const int kb0 = z * KB / p.KS, kb1 = (z + 1) * KB / p.KS;
  const int nit = (kb1 - kb0) * p.planes;
  constexpr int kABytes = 128 * 128;
  const uint32_t tcols = p.E <= 256 ? 256u : 512u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    mbar_init(acc_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, tcols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_g);
      for (int it = 0; it < nit; ++it) {
        const int st = it % NS;
        const uint32_t ph = (it / NS) & 1u;
        if (!mbar_wait(&empty_bar[st], ph ^ 1u, abort_flag, p.err)) break;
        const int kb = kb0 + it / p.planes, pl = it % p.planes;
        uint8_t* sa = smem + st * p.stage_bytes;
        uint8_t* sb = sa + kABytes;
        mbar_arrive_expect_tx(&full_bar[st], p.stage_bytes);
        tma_load_2d(sa, &tm_x, &full_bar[st], kb * kRgBK, t0);
        for (int h = 0; h < p.nmma; ++h)
          tma_load_2d(sb + h * p.nb * 128, &tm_g, &full_bar[st], kb * kRgBK, pl * p.E + h * p.nb);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool alive = true;
      for (int it = 0; it < nit; ++it) {
        const int st = it % NS;
        const uint32_t ph = (it / NS) & 1u;
        if (!mbar_wait(&full_bar[st], ph, abort_flag, p.err)) {
          alive = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + st * p.stage_bytes);
        const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
        for (int kk = 0; kk < kRgBK / 16; ++kk) {
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          const uint64_t adesc = sw128_desc(a_addr + kk * 32);
          for (int h = 0; h < p.nmma; ++h)
            umma_f16(tmem_base + h * p.nb, adesc,
                     sw128_desc(b_addr + h * p.nb * 128 + kk * 32), p.idesc, acc);
        }
        umma_commit(&empty_bar[st]);
      }
      if (alive) umma_commit(acc_bar);
    }
  } else {
    // ---------------- epilogue: TMEM lane quarter warp % 4 ----------------
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const bool ok = mbar_wait(acc_bar, 0, abort_flag, p.err);
    if (!named_bar_any(1, 128, !ok || *abort_flag)) {
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int t = t0 + r;
      float* dst = p.part + (static_cast<size_t>(z) * p.T + t) * p.E;
      for (int c = 0; c < p.E; c += 16) {
        uint32_t v[16];
        tmem_ld16(tb + c, v);
        tmem_ld_wait();
        reg_fence16(v);
        if (t < p.T) {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            __stcg(reinterpret_cast<float4*>(dst + c + i),
                   make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                               __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3])));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tcols);
  }
  if constexpr (S > 0) {
    // one thread draws the ticket: release of this CTA's partials (stored
    // before the barrier above), acquire of the other splits'
    __shared__ int s_last;
    if (threadIdx.x == 0) {
      const int old = ticket_add_acq_rel(a.tickets + blockIdx.x, 1);
      const int last = old == p.KS - 1;
      if (last) store_relaxed_gpu(a.tickets + blockIdx.x, 0);  // ready for the next launch
      s_last = last;
    }
    __syncthreads();
    if (!s_last || *abort_flag) return;
    // the ring is idle now (every stage was consumed before the accumulator
    // was complete): it holds the bias and the tile's summed logits
    float* sbias = reinterpret_cast<float*>(smem);
    float* rows = sbias + 32 * S;  // [tokens of the tile][E]
    for (int e = threadIdx.x; e < a.E; e += kRgThreads) sbias[e] = a.bias ? __ldg(a.bias + e) : 0.f;
    const int t_end = min(p.T, t0 + 128);
    const int nt = t_end - t0;
    // every thread sums (token, expert) pairs over the splits in split
    // order, all of a pair's split loads in flight at once
    const size_t slice = static_cast<size_t>(p.T) * a.E;
    for (int pr = threadIdx.x; pr < nt * a.E; pr += kRgThreads) {
      const int tt = pr / a.E, e = pr - tt * a.E;
      const float* src = p.part + static_cast<size_t>(t0 + tt) * a.E + e;
      float v[kRouterMaxSplits];
#pragma unroll
      for (int z2 = 0; z2 < kRouterMaxSplits; ++z2) v[z2] = z2 < p.KS ? __ldcg(src + z2 * slice) : 0.f;
      float acc = 0.f;
#pragma unroll
      for (int z2 = 0; z2 < kRouterMaxSplits; ++z2) acc += v[z2];
      rows[tt * a.E + e] = acc;
    }
    __syncthreads();
    for (int t = t0 + warp; t < t_end; t += kRgThreads / 32) {
      select_token<S>(a, t, rows + (t - t0) * a.E, sbias);
      cast_token_row(a, t);
    }
  }
}

// Sum of each token's split partials (split order) and the selection; one
// warp per token, eight tokens per CTA.  Compiled per slot count S (E <= 32*S)
// so each instance keeps only the registers its selection needs.
template <int S>
__global__ void __launch_bounds__(kRouterThreads) router_select_kernel(const RouterArgs a,
                                                                       const float* part) {
  __shared__ __align__(16) float rows[8][32 * S];
  __shared__ float sbias[32 * S];
  const int warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < a.E; e += kRouterThreads)
    sbias[e] = a.bias ? __ldg(a.bias + e) : 0.f;
  __syncthreads();
  const int t = blockIdx.x * 8 + warp;
  if (t >= a.T) return;
  select_from_partials<S>(a, part, t, rows[warp], sbias);
}

// Exact bf16 operands for the tiled gate GEMM: x e4m3 codes times their
// power-of-two scale (one per 32 along H), and the fp32 gate as three bf16
// planes [3][E*H].  Eight elements per thread step.
__global__ void __launch_bounds__(256) router_prep_kernel(const uint8_t* x8, const uint8_t* xs,
                                                          __nv_bfloat16* xb, long long nx, int H,
                                                          const float* g32, __nv_bfloat16* gp,
                                                          long long ng) {
  const long long ux = x8 ? nx / 8 : 0, ug = g32 ? ng / 8 : 0;
  for (long long u = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; u < ux + ug;
       u += static_cast<long long>(gridDim.x) * blockDim.x) {
    if (u < ux) {
      const long long j = u * 8;
      const long long row = j / H;
      const int col = static_cast<int>(j - row * H);
      const float s = exp2f(static_cast<float>(static_cast<int>(xs[row * (H / 32) + col / 32]) - 127));
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(x8 + j));
      const uint32_t w[2] = {v.x, v.y};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_fp8x2_storage_t pr =
            static_cast<__nv_fp8x2_storage_t>((w[i / 2] >> (16 * (i % 2))) & 0xFFFFu);
        __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
        const float2 f2 = __half22float2(*reinterpret_cast<__half2*>(&hr));
        o[i] = pack_bf16x2(f2.x * s, f2.y * s);
      }
      *reinterpret_cast<uint4*>(xb + j) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      const long long j = (u - ux) * 8;
      const float4* gsrc = reinterpret_cast<const float4*>(g32 + j);
      const float4 a0 = __ldg(gsrc), a1 = __ldg(gsrc + 1);
      const float f[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      Pieces<3> pc;
      split8(f, pc);
#pragma unroll
      for (int pl = 0; pl < 3; ++pl)
        *reinterpret_cast<uint4*>(gp + pl * ng + j) =
            make_uint4(pc.r[pl][0], pc.r[pl][1], pc.r[pl][2], pc.r[pl][3]);
    }
  }
}

template <int XDT, int GDT>
int launch_typed(const RouterArgs& a, const RouterPlan& plan, cudaStream_t stream) {
  dim3 grid(plan.ne, plan.nt, plan.ks);
  if (plan.nb8 == 1)
    router_kernel<XDT, GDT, 1><<<grid, kRouterThreads, 0, stream>>>(a);
  else
    router_kernel<XDT, GDT, 8><<<grid, kRouterThreads, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <int S>
int launch_gemm(dim3 grid, int smem, cudaStream_t stream, const CUtensorMap& tm_x,
                const CUtensorMap& tm_g, const RgParams& p, const RouterArgs& a) {
  static std::atomic<unsigned long long> smem_set{0};
  if (!ensure_smem_limit(reinterpret_cast<const void*>(router_gemm_kernel<S>),
                         kRgSmemBudget + 1024 + kRgBarBytes, smem_set))
    return -1;
  router_gemm_kernel<S><<<grid, kRgThreads, smem, stream>>>(tm_x, tm_g, p, a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_tiled(RouterArgs a, int hidden_dt, int gate_dt, const RouterPlan& plan,
                 cudaStream_t stream) {
  const int T = a.T, H = a.H, E = a.E;
  char* sc = reinterpret_cast<char*>(a.scratch);
  float* part = a.scratch;
  __nv_bfloat16* xb = reinterpret_cast<__nv_bfloat16*>(sc + plan.xb_off);
  __nv_bfloat16* gp = reinterpret_cast<__nv_bfloat16*>(sc + plan.gp_off);
  const bool conv_x = hidden_dt == 2, conv_g = gate_dt == 1;
  if (conv_x || conv_g) {
    const long long nx = static_cast<long long>(T) * H, ng = static_cast<long long>(E) * H;
    const long long units = (conv_x ? nx / 8 : 0) + (conv_g ? ng / 8 : 0);
    const int blocks = static_cast<int>(std::min<long long>((units + 255) / 256, 4 * kTargetCtas));
    router_prep_kernel<<<blocks, 256, 0, stream>>>(
        conv_x ? static_cast<const uint8_t*>(a.x) : nullptr, a.x_scale, xb, nx, H,
        conv_g ? static_cast<const float*>(a.gate) : nullptr, gp, ng);
    if (cudaGetLastError() != cudaSuccess) return -1;
  }
  RgParams p{};
  p.part = part;
  p.err = a.err;
  p.T = T;
  p.H = H;
  p.E = E;
  p.KS = plan.tks;
  p.planes = conv_g ? 3 : 1;
  p.nmma = E <= 256 ? 1 : 2;
  p.nb = E / p.nmma;
  p.stage_bytes = 128 * 128 + E * 128;
  p.stages = std::min(6, kRgSmemBudget / p.stage_bytes);
  p.idesc = idesc_bf16_f32(128, p.nb);
  CUtensorMap tm_x, tm_g;
  if (!make_map_bf16(&tm_x, conv_x ? static_cast<const void*>(xb) : a.x, T, H, 128)) return -1;
  if (!make_map_bf16(&tm_g, conv_g ? static_cast<const void*>(gp) : a.gate,
                     static_cast<uint64_t>(p.planes) * E, H, p.nb))
    return -1;
  const int smem = p.stages * p.stage_bytes + 1024 + kRgBarBytes;
  a.KS = plan.tks;
  const int sl = (E + 31) / 32, blocks = (T + 7) / 8;
  const dim3 grid(plan.tnt, plan.tks);
  if (plan.fused_select) {
    // the last CTA of the token tile selects: one launch
    if (sl <= 1) return launch_gemm<1>(grid, smem, stream, tm_x, tm_g, p, a);
    if (sl <= 2) return launch_gemm<2>(grid, smem, stream, tm_x, tm_g, p, a);
    if (sl <= 4) return launch_gemm<4>(grid, smem, stream, tm_x, tm_g, p, a);
    if (sl <= 8) return launch_gemm<8>(grid, smem, stream, tm_x, tm_g, p, a);
    if (sl <= 9) return launch_gemm<9>(grid, smem, stream, tm_x, tm_g, p, a);
    return launch_gemm<16>(grid, smem, stream, tm_x, tm_g, p, a);
  }
  if (launch_gemm<0>(grid, smem, stream, tm_x, tm_g, p, a) != 0) return -1;
  if (sl <= 1) router_select_kernel<1><<<blocks, kRouterThreads, 0, stream>>>(a, part);
  else if (sl <= 2) router_select_kernel<2><<<blocks, kRouterThreads, 0, stream>>>(a, part);
  else if (sl <= 4) router_select_kernel<4><<<blocks, kRouterThreads, 0, stream>>>(a, part);
  else if (sl <= 8) router_select_kernel<8><<<blocks, kRouterThreads, 0, stream>>>(a, part);
  else if (sl <= 9) router_select_kernel<9><<<blocks, kRouterThreads, 0, stream>>>(a, part);
  else router_select_kernel<16><<<blocks, kRouterThreads, 0, stream>>>(a, part);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

RouterPlan plan_router(int T, int H, int E, bool allow_tiled) {
  RouterPlan p{};
  p.nb8 = (T >= 128) ? 8 : 1;
  p.et = 8 * p.nb8;
  p.ne = (E + p.et - 1) / p.et;
  p.nt = (T + 15) / 16;
  p.ks = 1;
  const int steps = H / 32;
  // grow the K split while the grid stays within one wave (two CTAs per SM)
  while (p.ks < 16 && (long long)p.ne * p.nt * p.ks * 2 <= kTargetCtas && steps % (2 * p.ks) == 0)
    p.ks *= 2;
  p.scratch_bytes = align_up(static_cast<size_t>(p.ks) * T * E * sizeof(float), 256);
  // tiled path: T >= 256, E a multiple of 16 that one or two MMAs cover
  p.T = T;
  p.tiled = allow_tiled && T >= 1 && H % kRgBK == 0 && E >= 16 && E % 16 == 0 &&
            (E <= 256 || (E <= 512 && E % 32 == 0));
  if (p.tiled) {
    p.tnt = (T + 127) / 128;
    const int KB = H / kRgBK;
    p.tks = 1;
    while (p.tks < 16 && p.tnt * p.tks * 2 <= kTargetCtas / 2 && KB / (2 * p.tks) >= 2) p.tks *= 2;
    const size_t part = align_up(static_cast<size_t>(p.tks) * T * E * sizeof(float), 256);
    p.xb_off = part;
    p.gp_off = p.xb_off + align_up(static_cast<size_t>(T) * H * 2, 256);
    const size_t total = p.gp_off + align_up(static_cast<size_t>(3) * E * H * 2, 256);
    if (total > p.scratch_bytes) p.scratch_bytes = total;
    p.fused_select = T <= kRouterFusedSelectMaxT;
    if (p.fused_select) {
      // a few tokens: the gate read is the whole cost, so split K further
      // (up to 32 CTAs, at least two K steps each) until each CTA's share is
      // in flight at once
      while (p.tks < 32 && KB / (2 * p.tks) >= 2) p.tks *= 2;
      const size_t part2 = align_up(static_cast<size_t>(p.tks) * T * E * sizeof(float), 256);
      if (part2 > p.xb_off) {
        p.xb_off = part2;
        p.gp_off = p.xb_off + align_up(static_cast<size_t>(T) * H * 2, 256);
        const size_t total2 = p.gp_off + align_up(static_cast<size_t>(3) * E * H * 2, 256);
        if (total2 > p.scratch_bytes) p.scratch_bytes = total2;
      }
    }
  }
  return p;
}

bool router_uses_tiled(const RouterPlan& plan, int hidden_dt, int gate_dt) {
  return plan.tiled && (hidden_dt == 0 || hidden_dt == 2) &&
         (gate_dt == 0 || (gate_dt == 1 && plan.T >= kTiledMinTokensF32Gate));
}

int launch_router(const void* hidden, int hidden_dt, const uint8_t* hidden_scale,
                  const void* gate, int gate_dt, const float* bias, int T, int H, int E, int k,
                  int scoring, int n_group, int topk_group, int renormalize, float scaling,
                  int32_t* topk_ids, float* topk_weights, float* scratch, int* tickets, int* err,
                  const RouterPlan& plan, cudaStream_t stream, uint8_t* cast_codes,
                  uint8_t* cast_scales, int* align_hist, int align_seg) {
  if (cast_codes != nullptr && (hidden_dt != 0 || cast_scales == nullptr)) return -2;
  if (align_hist != nullptr && align_seg <= 0) return -2;
  RouterArgs a;
  a.cast_codes = cast_codes;
  a.cast_scales = cast_scales;
  a.align_hist = align_hist;
  a.align_seg = align_seg;
  a.x = hidden;
  a.x_scale = hidden_scale;
  a.gate = gate;
  a.bias = bias;
  a.scratch = scratch;
  a.tickets = tickets;
  a.ids = topk_ids;
  a.wts = topk_weights;
  a.err = err;
  a.T = T;
  a.H = H;
  a.E = E;
  a.k = k;
  a.scoring = scoring;
  a.n_group = n_group;
  a.topk_group = topk_group;
  a.renorm = renormalize;
  a.KS = plan.ks;
  a.scaling = scaling;
  // hidden: 0 bf16, 1 f32, 2 e4m3; gate: 0 bf16, 1 f32
  if (router_uses_tiled(plan, hidden_dt, gate_dt))
    return launch_tiled(a, hidden_dt, gate_dt, plan, stream);
  if (hidden_dt == 0 && gate_dt == 0) return launch_typed<0, 0>(a, plan, stream);
  if (hidden_dt == 0 && gate_dt == 1) return launch_typed<0, 1>(a, plan, stream);
  if (hidden_dt == 1 && gate_dt == 0) return launch_typed<1, 0>(a, plan, stream);
  if (hidden_dt == 1 && gate_dt == 1) return launch_typed<1, 1>(a, plan, stream);
  if (hidden_dt == 2 && gate_dt == 0) return launch_typed<2, 0>(a, plan, stream);
  if (hidden_dt == 2 && gate_dt == 1) return launch_typed<2, 1>(a, plan, stream);
  return -2;
}

}  // namespace moe
