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

#include <climits>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kRouterThreads = 256;
constexpr int kMaxSlotsPerLane = 16;  // E <= 512
constexpr int kTargetCtas = 304;      // two CTAs per SM of a 152-SM part

struct RouterArgs {
  const void* x;
  const uint8_t* x_scale;
  const void* gate;
  const float* bias;
  float* scratch;   // [KS][T][E]
  int* tickets;     // [ceil(T/16)]
  int32_t* ids;
  float* wts;
  int* err;
  int T, H, E, k, scoring, n_group, topk_group, renorm, KS;
  float scaling;
};

// Eight consecutive source values -> up to three bf16 parts, as four packed
// bf16x2 registers per part (pairs (0,1), (2,3), (4,5), (6,7)).
template <int P>
struct Pieces {
  uint32_t r[P][4];
};

MOE_DEV void split8(const float (&f)[8], Pieces<3>& out) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a = f[2 * i], b = f[2 * i + 1];
    __nv_bfloat16 ah = __float2bfloat16_rn(a), bh = __float2bfloat16_rn(b);
    float ar = a - __bfloat162float(ah), br = b - __bfloat162float(bh);
    __nv_bfloat16 am = __float2bfloat16_rn(ar), bm = __float2bfloat16_rn(br);
    float ar2 = ar - __bfloat162float(am), br2 = br - __bfloat162float(bm);
    __nv_bfloat16 al = __float2bfloat16_rn(ar2), bl = __float2bfloat16_rn(br2);
    __nv_bfloat162 h2, m2, l2;
    h2.x = ah; h2.y = bh;
    m2.x = am; m2.y = bm;
    l2.x = al; l2.y = bl;
    out.r[0][i] = *reinterpret_cast<uint32_t*>(&h2);
    out.r[1][i] = *reinterpret_cast<uint32_t*>(&m2);
    out.r[2][i] = *reinterpret_cast<uint32_t*>(&l2);
  }
}

// dtype codes: 0 bf16, 1 f32, 2 e4m3 (+ scale per 32)
template <int DT>
struct SrcPieces {
  static constexpr int P = (DT == 1) ? 3 : 1;
};

// Load elements [h, h+8) of row `row` (row < rows, else zeros).
template <int DT>
MOE_DEV void load8(const void* base, const uint8_t* scale, int row, int rows, int H, int h,
                   Pieces<SrcPieces<DT>::P>& out) {
  if (row >= rows) {
#pragma unroll
    for (int p = 0; p < SrcPieces<DT>::P; ++p)
#pragma unroll
      for (int i = 0; i < 4; ++i) out.r[p][i] = 0u;
    return;
  }
  const size_t off = static_cast<size_t>(row) * H + h;
  if constexpr (DT == 0) {
    uint4 v = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(base) + off));
    out.r[0][0] = v.x; out.r[0][1] = v.y; out.r[0][2] = v.z; out.r[0][3] = v.w;
  } else if constexpr (DT == 1) {
    const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + off);
    float4 a = __ldg(p), b = __ldg(p + 1);
    float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    split8(f, out);
  } else {
    uint2 v = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(base) + off));
    const float s = exp2f(static_cast<float>(static_cast<int>(scale[static_cast<size_t>(row) * (H / 32) + h / 32]) - 127));
    uint32_t w[2] = {v.x, v.y};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_fp8x2_storage_t pr = static_cast<__nv_fp8x2_storage_t>((w[i / 2] >> (16 * (i % 2))) & 0xFFFFu);
      __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
      __half2 hh = *reinterpret_cast<__half2*>(&hr);
      float2 f2 = __half22float2(hh);
      out.r[0][i] = pack_bf16x2(f2.x * s, f2.y * s);  // exact: e4m3 * 2^u fits bf16
    }
  }
}

MOE_DEV void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                            uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

MOE_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Selection for one token by one warp; E <= 32 * S (S slots per lane, expert
// lane + 32 i in slot i).  `row` holds the token's E fp32 logits (shared
// memory).  Every warp-wide argmax is two redux operations: the largest
// order-mapped key, then the lowest expert id holding it.
template <int S>
MOE_DEV void select_token(const RouterArgs& a, int t, const float* row, const float* sbias) {
  const int lane = threadIdx.x & 31;
  const int E = a.E;
  float sc[S], key[S];
  bool ok[S];
#pragma unroll
  for (int i = 0; i < S; ++i) {
    const int e = lane + 32 * i;
    ok[i] = e < E;
    sc[i] = ok[i] ? row[e] : -INFINITY;  // logits for now
  }
  if (a.scoring == 0) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < S; ++i) m = fmaxf(m, sc[i]);
    m = ord2f(__reduce_max_sync(0xffffffffu, f2ord(m)));
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < S; ++i) {
      sc[i] = ok[i] ? expf(sc[i] - m) : 0.f;
      sum += sc[i];
    }
    sum = warp_sum(sum);
    const float inv = 1.0f / sum;
#pragma unroll
    for (int i = 0; i < S; ++i) sc[i] *= inv;
  } else {
#pragma unroll
    for (int i = 0; i < S; ++i) sc[i] = ok[i] ? 1.0f / (1.0f + expf(-sc[i])) : 0.f;
  }
#pragma unroll
  for (int i = 0; i < S; ++i) {
    const int e = lane + 32 * i;
    key[i] = ok[i] ? sc[i] + sbias[e] : -INFINITY;
  }
  // group-limited selection: keep the topk_group groups with the largest sum
  // of their two best rank keys (lowest group id on ties)
  if (a.n_group > 1) {
    const int gs = E / a.n_group;
    int grp[S];
#pragma unroll
    for (int i = 0; i < S; ++i) grp[i] = ok[i] ? (lane + 32 * i) / gs : -1;
    uint32_t my_g = 0;  // lane g: order-mapped score of group g
    for (int g = 0; g < a.n_group; ++g) {
      float t1 = -INFINITY, t2 = -INFINITY;
#pragma unroll
      for (int i = 0; i < S; ++i) {
        if (grp[i] == g) {
          const float v = key[i];
          if (v > t1) {
            t2 = t1;
            t1 = v;
          } else if (v > t2) {
            t2 = v;
          }
        }
      }
      const uint32_t o1 = f2ord(t1);
      const uint32_t b1 = __reduce_max_sync(0xffffffffu, o1);
      const unsigned holders = __ballot_sync(0xffffffffu, o1 == b1);
      uint32_t b2 = b1;
      if (__popc(holders) < 2) b2 = __reduce_max_sync(0xffffffffu, o1 == b1 ? f2ord(t2) : o1);
      if (lane == g) my_g = f2ord(ord2f(b1) + ord2f(b2));
    }
    uint32_t kept = 0;
    for (int r = 0; r < a.topk_group; ++r) {
      const bool cand = lane < a.n_group && !((kept >> lane) & 1u);
      const uint32_t gmax = __reduce_max_sync(0xffffffffu, cand ? my_g : 0u);
      const int sel = __reduce_min_sync(0xffffffffu, (cand && my_g == gmax) ? lane : 32);
      if (sel < 32) kept |= 1u << sel;
    }
#pragma unroll
    for (int i = 0; i < S; ++i)
      if (ok[i] && !((kept >> grp[i]) & 1u)) ok[i] = false;
  }
  // k rounds of a warp argmax (largest key, lowest id on ties); lane j keeps
  // the j-th winner
  int my_id = -1;
  float my_s = 0.f;
  for (int j = 0; j < a.k; ++j) {
    uint32_t bk = 0;
    int be = INT_MAX;
    float bs = 0.f;
#pragma unroll
    for (int i = 0; i < S; ++i) {
      const uint32_t o = f2ord(key[i]);
      if (ok[i] && (o > bk || (o == bk && lane + 32 * i < be))) {
        bk = o;
        be = lane + 32 * i;
        bs = sc[i];
      }
    }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
    const int win = __reduce_min_sync(0xffffffffu, (be != INT_MAX && bk == kmax) ? be : INT_MAX);
    const int owner = (win == INT_MAX) ? 0 : (win & 31);
    const float ws = __shfl_sync(0xffffffffu, bs, owner);
    if (lane == owner && win != INT_MAX) {
#pragma unroll
      for (int i = 0; i < S; ++i)
        if (lane + 32 * i == win) ok[i] = false;
    }
    if (lane == j) {
      my_id = (win == INT_MAX) ? -1 : win;
      my_s = ws;
    }
  }
  const float sum = warp_sum(lane < a.k ? my_s : 0.f);
  const float denom = a.renorm ? (sum + 1e-20f) : 1.0f;
  if (lane < a.k) {
    a.ids[static_cast<size_t>(t) * a.k + lane] = my_id;
    a.wts[static_cast<size_t>(t) * a.k + lane] = my_s / denom * a.scaling;
  }
}

MOE_DEV void select_dispatch(const RouterArgs& a, int t, const float* row, const float* sbias) {
  const int s = (a.E + 31) / 32;
  if (s <= 1) select_token<1>(a, t, row, sbias);
  else if (s <= 2) select_token<2>(a, t, row, sbias);
  else if (s <= 4) select_token<4>(a, t, row, sbias);
  else if (s <= 8) select_token<8>(a, t, row, sbias);
  else if (s <= 9) select_token<9>(a, t, row, sbias);
  else select_token<16>(a, t, row, sbias);
}

template <int XDT, int GDT, int NB8>
__global__ void __launch_bounds__(kRouterThreads) router_kernel(const RouterArgs a) {
  constexpr int ET = 8 * NB8;
  constexpr int XP = SrcPieces<XDT>::P, GP = SrcPieces<GDT>::P;
  // per-warp partial logits, later reused for the token tile's full logits
  constexpr int kRedFloats = 8 * 16 * ET;
  constexpr int kTileFloats = (16 + 1) * 32 * kMaxSlotsPerLane;  // 16 logit rows + bias
  __shared__ __align__(16) float sbuf[kRedFloats > kTileFloats ? kRedFloats : kTileFloats];
  float(*red)[16][ET] = reinterpret_cast<float(*)[16][ET]>(sbuf);
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int e0 = blockIdx.x * ET, t0 = blockIdx.y * 16, ks = blockIdx.z;
  const int HK = a.H / a.KS;
  const int step0 = ks * HK / 32, nsteps = HK / 32;

  float acc[NB8][4];
#pragma unroll
  for (int j = 0; j < NB8; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[j][c] = 0.f;

  for (int st = warp; st < nsteps; st += 8) {
    const int h = (step0 + st) * 32 + 8 * q;
    Pieces<XP> xa, xb;  // rows g and g + 8 of the token tile
    load8<XDT>(a.x, a.x_scale, t0 + g, a.T, a.H, h, xa);
    load8<XDT>(a.x, a.x_scale, t0 + g + 8, a.T, a.H, h, xb);
#pragma unroll
    for (int j = 0; j < NB8; ++j) {
      Pieces<GP> gb;
      load8<GDT>(a.gate, nullptr, e0 + 8 * j + g, a.E, a.H, h, gb);
      // product pieces (px, pg) with px + pg <= 2; each 32-wide step is two
      // k16 MMAs over a permutation of the step's K indices shared by A and B
#pragma unroll
      for (int px = 0; px < XP; ++px) {
#pragma unroll
        for (int pg = 0; pg < GP; ++pg) {
          if (px + pg > 2) continue;
          mma_bf16_16816(acc[j], xa.r[px][0], xb.r[px][0], xa.r[px][1], xb.r[px][1],
                         gb.r[pg][0], gb.r[pg][1]);
          mma_bf16_16816(acc[j], xa.r[px][2], xb.r[px][2], xa.r[px][3], xb.r[px][3],
                         gb.r[pg][2], gb.r[pg][3]);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NB8; ++j) {
    red[warp][g][8 * j + 2 * q] = acc[j][0];
    red[warp][g][8 * j + 2 * q + 1] = acc[j][1];
    red[warp][g + 8][8 * j + 2 * q] = acc[j][2];
    red[warp][g + 8][8 * j + 2 * q + 1] = acc[j][3];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < 16 * ET; idx += kRouterThreads) {
    const int r = idx / ET, c = idx % ET;
    float v = red[0][r][c];
#pragma unroll
    for (int w = 1; w < 8; ++w) v += red[w][r][c];
    const int t = t0 + r, e = e0 + c;
    if (t < a.T && e < a.E) a.scratch[(static_cast<size_t>(ks) * a.T + t) * a.E + e] = v;
  }
  // last CTA of this token tile does the selection: one thread draws a
  // ticket (release of this CTA's partials, acquire of the others')
  __syncthreads();
  if (threadIdx.x == 0) {
    const int total = gridDim.x * gridDim.z;
    const int old = ticket_add_acq_rel(a.tickets + blockIdx.y, 1);
    const int last = (old == total - 1);
    if (last) store_relaxed_gpu(a.tickets + blockIdx.y, 0);  // ready for the next launch
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;
  // sum the K-slice partials of the tile's logits in slice order.  Each thread
  // owns up to kPer logits and issues all their loads (every slice) before
  // summing, so the reduction costs one L2 round trip; the bias rides along.
  const int rows = min(16, a.T - t0);
  float* tile = sbuf;                                   // [16][E]
  float* sbias = sbuf + 16 * 32 * kMaxSlotsPerLane;    // [E], after the 16 logit rows
  const size_t slice = static_cast<size_t>(a.T) * a.E;
  const int nlog = rows * a.E;
  constexpr int kPer = 8;
  for (int base = threadIdx.x; base < nlog; base += kRouterThreads * kPer) {
    float acc[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int idx = base + u * kRouterThreads;
      acc[u] = 0.f;
      if (idx < nlog) {
        const int r = idx / a.E, e = idx - r * a.E;
        acc[u] = __ldcg(a.scratch + static_cast<size_t>(t0 + r) * a.E + e);
      }
    }
    for (int s = 1; s < a.KS; ++s) {
      float part[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int idx = base + u * kRouterThreads;
        part[u] = 0.f;
        if (idx < nlog) {
          const int r = idx / a.E, e = idx - r * a.E;
          part[u] = __ldcg(a.scratch + s * slice + static_cast<size_t>(t0 + r) * a.E + e);
        }
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) acc[u] += part[u];
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int idx = base + u * kRouterThreads;
      if (idx < nlog) tile[idx] = acc[u];
    }
  }
  for (int e = threadIdx.x; e < a.E; e += kRouterThreads)
    sbias[e] = a.bias ? __ldg(a.bias + e) : 0.f;
  __syncthreads();
  for (int r = warp; r < rows; r += 8) select_dispatch(a, t0 + r, tile + r * a.E, sbias);
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

}  // namespace

RouterPlan plan_router(int T, int H, int E) {
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
  return p;
}

int launch_router(const void* hidden, int hidden_dt, const uint8_t* hidden_scale,
                  const void* gate, int gate_dt, const float* bias, int T, int H, int E, int k,
                  int scoring, int n_group, int topk_group, int renormalize, float scaling,
                  int32_t* topk_ids, float* topk_weights, float* scratch, int* tickets, int* err,
                  const RouterPlan& plan, cudaStream_t stream) {
  RouterArgs a;
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
  if (hidden_dt == 0 && gate_dt == 0) return launch_typed<0, 0>(a, plan, stream);
  if (hidden_dt == 0 && gate_dt == 1) return launch_typed<0, 1>(a, plan, stream);
  if (hidden_dt == 1 && gate_dt == 0) return launch_typed<1, 0>(a, plan, stream);
  if (hidden_dt == 1 && gate_dt == 1) return launch_typed<1, 1>(a, plan, stream);
  if (hidden_dt == 2 && gate_dt == 0) return launch_typed<2, 0>(a, plan, stream);
  if (hidden_dt == 2 && gate_dt == 1) return launch_typed<2, 1>(a, plan, stream);
  return -2;
}

}  // namespace moe
