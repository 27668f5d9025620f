// router_device.cuh -- device code of the one-launch router, shared by the
// router kernels (router.cu) and the persistent decode layer (decode.cu).
//
// Follows "How an MoE Model Picks Its Experts During LLM Inference": §1.1
// (three steps), §1.3 (rank key = score + bias, weight = unbiased score),
// §2.4 (bf16 inputs, fp32 logits and bias), §4 (weights / (sum + 1e-20)),
// §5.1 (many CTAs each own a slice of experts so the cold gate read runs at
// memory speed), §5.3 (a warp owns a token row, k rounds, lowest id wins);
// and "Mixture of Experts" (DeepSeek's grouped, bias-corrected routing: group
// score = sum of the top-2 rank keys, keep topk_group groups, routed scaling).
#pragma once

#include <cuda_fp8.h>

#include <climits>

#include "moe_common.cuh"

namespace moe {

constexpr int kRouterThreads = 256;
constexpr int kMaxSlotsPerLane = 16;  // E <= 512

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
  // optional FP8 cast of the bf16 hidden rows, written by the selecting warp
  // of each token next to its ids and weights (nullptr: none)
  uint8_t* cast_codes;   // [T, H] e4m3
  uint8_t* cast_scales;  // [T, H/32] UE8M0
  // optional per-segment expert counts for the align that follows ("How an
  // MoE Model Picks Its Experts ..." §6.1: the routing stage counts as it
  // selects): assignment a adds 1 to align_hist[(a / align_seg) * E + id]
  int* align_hist;
  int align_seg;
  int T, H, E, k, scoring, n_group, topk_group, renorm, KS;
  float scaling;
};

// "How GPUs Fuse Communication and Computation During LLM Inference" §1.1:
// the layer input's FP8 codes and scales are written together with the
// router's outputs.  The warp that selected token t also casts its bf16 row
// (one group of 32 values per lane at a time; cast_e4m3_group32).
MOE_DEV void cast_token_row(const RouterArgs& a, int t) {
  if (a.cast_codes == nullptr) return;
  const int lane = threadIdx.x & 31;
  const int G = a.H / 32;
  const uint4* src = reinterpret_cast<const uint4*>(
      reinterpret_cast<const __nv_bfloat16*>(a.x) + static_cast<size_t>(t) * a.H);
  uint4* dst = reinterpret_cast<uint4*>(a.cast_codes + static_cast<size_t>(t) * a.H);
  uint8_t* sc = a.cast_scales + static_cast<size_t>(t) * G;
  for (int g = lane; g < G; g += 32) cast_e4m3_group32(src + 4 * g, dst + 2 * g, sc + g);
}

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
  } else if (a.scoring == 1) {
#pragma unroll
    for (int i = 0; i < S; ++i) sc[i] = ok[i] ? 1.0f / (1.0f + expf(-sc[i])) : 0.f;
  } else {
    // sqrt(softplus(l)), softplus(l) = max(l, 0) + ln(1 + e^-|l|) (no overflow)
#pragma unroll
    for (int i = 0; i < S; ++i)
      sc[i] = ok[i] ? sqrtf(fmaxf(sc[i], 0.f) + log1pf(expf(-fabsf(sc[i])))) : 0.f;
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
    // group g is slot g when a group holds 32 experts (one per lane): the
    // groups' top-2 sums then reduce side by side rather than one group after
    // another (compiled up to 8 slots: the unrolled code in the 9-slot
    // instance slowed its gate without groups, E = 288, by about 1 us)
    const bool by_slot = S <= 8 && gs == 32;
    if constexpr (S <= 8) {
#pragma unroll
      for (int i = 0; i < S; ++i) {
        if (by_slot && i < a.n_group) {
          float t1 = -INFINITY;
          if (grp[i] == i && key[i] > t1) t1 = key[i];
          const uint32_t o1 = f2ord(t1);
          const uint32_t b1 = __reduce_max_sync(0xffffffffu, o1);
          const unsigned holders = __ballot_sync(0xffffffffu, o1 == b1);
          uint32_t b2 = b1;
          if (__popc(holders) < 2)
            b2 = __reduce_max_sync(0xffffffffu, o1 == b1 ? f2ord(-INFINITY) : o1);
          if (lane == i) my_g = f2ord(ord2f(b1) + ord2f(b2));
        }
      }
    }
    for (int g = 0; !by_slot && g < a.n_group; ++g) {
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
    if (a.align_hist != nullptr && my_id >= 0) {
      const long long asg = static_cast<long long>(t) * a.k + lane;
      atomicAdd(a.align_hist + (asg / a.align_seg) * a.E + my_id, 1);
    }
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

// Shared-memory floats router_item needs (its caller provides them).
template <int NB8>
constexpr int router_item_smem_floats() {
  return (8 * 16 * 8 * NB8 > (16 + 1) * 32 * kMaxSlotsPerLane) ? 8 * 16 * 8 * NB8
                                                                : (16 + 1) * 32 * kMaxSlotsPerLane;
}

// One work item of the one-launch router, run by the 256 threads of a CTA:
// experts [bx*ET, bx*ET+ET), tokens [by*16, by*16+16), K slice bz of a.KS.
// tile_items = the number of items of the token tile (expert tiles x K
// slices); the item that finishes last sums the tile's partials and selects.
// sbuf: router_item_smem_floats<NB8>() floats of shared memory (16-byte
// aligned); s_flag: one shared int.  Returns true in the CTA that selected.
template <int XDT, int GDT, int NB8>
MOE_DEV bool router_item(const RouterArgs& a, int bx, int by, int bz, int tile_items, float* sbuf,
                         int* s_flag) {
  constexpr int ET = 8 * NB8;
  constexpr int XP = SrcPieces<XDT>::P, GP = SrcPieces<GDT>::P;
  // sbuf: per-warp partial logits, later reused for the token tile's full
  // logits (16 rows) and the bias
  float(*red)[16][ET] = reinterpret_cast<float(*)[16][ET]>(sbuf);
  int& s_last = *s_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int e0 = bx * ET, t0 = by * 16, ks = bz;
  const int HK = a.H / a.KS;
  const int step0 = ks * HK / 32, nsteps = HK / 32;

  float acc[NB8][4];
#pragma unroll
  for (int j = 0; j < NB8; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[j][c] = 0.f;

  // U of the warp's K steps are loaded before any of them is multiplied, so
  // their global round trips overlap (U from the registers the fragments take)
  constexpr int kFragRegs = (2 * XP + GP * NB8) * 4;
  constexpr int U = (NB8 > 1) ? 1 : (kFragRegs * 4 <= 64 ? 4 : (kFragRegs * 2 <= 64 ? 2 : 1));
  for (int st0 = warp; st0 < nsteps; st0 += 8 * U) {
    Pieces<XP> xa[U], xb[U];  // rows g and g + 8 of the token tile
    Pieces<GP> gb[U][NB8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int st = st0 + 8 * u;
      if (st < nsteps) {
        const int h = (step0 + st) * 32 + 8 * q;
        load8<XDT>(a.x, a.x_scale, t0 + g, a.T, a.H, h, xa[u]);
        load8<XDT>(a.x, a.x_scale, t0 + g + 8, a.T, a.H, h, xb[u]);
#pragma unroll
        for (int j = 0; j < NB8; ++j) load8<GDT>(a.gate, nullptr, e0 + 8 * j + g, a.E, a.H, h, gb[u][j]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (st0 + 8 * u >= nsteps) break;
#pragma unroll
      for (int j = 0; j < NB8; ++j) {
        // product pieces (px, pg) with px + pg <= 2; each 32-wide step is two
        // k16 MMAs over a permutation of the step's K indices shared by A and B
#pragma unroll
        for (int px = 0; px < XP; ++px) {
#pragma unroll
          for (int pg = 0; pg < GP; ++pg) {
            if (px + pg > 2) continue;
            mma_bf16_16816(acc[j], xa[u].r[px][0], xb[u].r[px][0], xa[u].r[px][1],
                           xb[u].r[px][1], gb[u][j].r[pg][0], gb[u][j].r[pg][1]);
            mma_bf16_16816(acc[j], xa[u].r[px][2], xb[u].r[px][2], xa[u].r[px][3],
                           xb[u].r[px][3], gb[u][j].r[pg][2], gb[u][j].r[pg][3]);
          }
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
    const int old = ticket_add_acq_rel(a.tickets + by, 1);
    const int last = (old == tile_items - 1);
    if (last) store_relaxed_gpu(a.tickets + by, 0);  // ready for the next launch
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return false;
  // sum the K-slice partials of the tile's logits in slice order.  Each thread
  // owns up to kPer logits and issues the loads of four slices for all of them
  // before adding any, so the reduction costs ceil(KS/4) L2 round trips; the
  // bias rides along.
  const int rows = min(16, a.T - t0);
  float* tile = sbuf;                                   // [16][E]
  float* sbias = sbuf + 16 * 32 * kMaxSlotsPerLane;    // [E], after the 16 logit rows
  const size_t slice = static_cast<size_t>(a.T) * a.E;
  const int nlog = rows * a.E;
  constexpr int kPer = 8;
  for (int base = threadIdx.x; base < nlog; base += kRouterThreads * kPer) {
    float acc[kPer];
    size_t off[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int idx = base + u * kRouterThreads;
      const int r = idx / a.E, e = idx - r * a.E;
      off[u] = static_cast<size_t>(t0 + r) * a.E + e;
      acc[u] = 0.f;
    }
    for (int s0 = 0; s0 < a.KS; s0 += 4) {
      float part[4][kPer];
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int idx = base + u * kRouterThreads;
          part[q][u] = (s0 + q < a.KS && idx < nlog) ? __ldcg(a.scratch + (s0 + q) * slice + off[u])
                                                     : 0.f;
        }
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int u = 0; u < kPer; ++u)
          if (s0 + q < a.KS) acc[u] = (s0 + q == 0) ? part[q][u] : acc[u] + part[q][u];
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
  for (int r = warp; r < rows; r += 8) {
    select_dispatch(a, t0 + r, tile + r * a.E, sbias);
    cast_token_row(a, t0 + r);
  }
  return true;
}

}  // namespace moe
