// ffn.cu -- the grouped expert GEMMs on the 5th-generation tensor cores.
//
// Follows "MoE Kernels, in depth", The fused expert GEMM (every tile looks up
// its expert in block_expert and its rows in sorted_ids, the activation gather
// is folded into the operand load, padding rows are masked, gate and up form
// one 2F x H matrix with SwiGLU in the epilogue, the routing weight is applied
// in the down GEMM's epilogue) and "Mixture of Experts" (w13 [E, 2F, H] with
// the gate rows first, w2 [E, H, F]; row = sorted id // top_k).
//
// One persistent kernel per GEMM, one CTA per SM, 8 warps:
//   warp 0      TMA producer: expert weight tiles (and, for GEMM2, the
//               intermediate rows) into a ring of shared-memory stages
//   warp 1      TMEM allocator and the single thread issuing tcgen05.mma
//   warps 2-3   GEMM1 only: gather of the token rows x[sorted_id / k] with
//               16-byte cp.async straight into the 128-byte-swizzled operand
//               layout (zero-filled for padding rows)
//   warps 4-7   epilogue: TMEM -> registers -> SwiGLU / routing weight ->
//               global memory; two TMEM accumulators so the epilogue of one
//               tile overlaps the MMAs of the next
//
// Tile orientation depends on the tile height BM (rows per expert block):
//   BM = 128: A = 128 token rows (M = 128), B = 256 weight rows (N = 256);
//             GEMM1 loads the 128 gate rows and the matching 128 up rows as
//             two boxes so the epilogue pairs column c with column c + 128.
//   BM = 16/64 ("swap"): A = 128 weight rows (M = 128), B = the BM token rows
//             (N = BM); GEMM1 issues two MMAs per K step (gate rows, up rows)
//             into two accumulators.  Few tokens per expert is the decode
//             regime, which streams weights: when the tiles are too few to
//             fill the GPU the K range is split (chosen on the device from the
//             padded length) and the last split to finish (atomic ticket, no
//             spinning) sums the fp32 partials in split order and runs the
//             epilogue.
// Above H = 4096 the row tiles run on CTA pairs (ffn_pair_kernel): two blocks
// of one expert share the 256-row weight tile, each CTA loading one half and
// multicasting it to both.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

// Warps: 0 TMA producer, 1 MMA issuer (+ TMEM), 2 .. 1+GW token-row gather
// (GEMM1; idle in GEMM2), then four epilogue warps.
constexpr int kBK = 64;                 // K elements per stage (128 bytes of bf16)
constexpr int kStageBudget = 220 * 1024;

// Tile geometry.
//   Swap tiles (BLOCK_M 16 / 64): A = 128 weight rows (GEMM1: 128 gate rows
//   and the matching 128 up rows, two MMAs per K step), B = the block's BM
//   token rows; double-buffered TMEM accumulators; optional split-K.
//   Row tiles (BLOCK_M 128): A = the block's 128 token rows, B = 256 weight
//   rows (GEMM1: 128 gate rows + the matching 128 up rows, two TMA boxes, so
//   the epilogue pairs column c with column c + 128); one 128x256 MMA per K
//   step; two 256-column accumulators, double-buffered.
template <int KIND, int BM, int GW = 2>
struct Cfg {
  static constexpr bool SWAP = BM < 128;
  static constexpr bool GATHER = KIND == 0;
  static constexpr int NT = (KIND == 0) ? 128 : (SWAP ? 128 : 256);  // output tile width
  static constexpr int A_BYTES = (SWAP && KIND == 0) ? 2 * 128 * 128 : 128 * 128;
  static constexpr int B_BYTES = SWAP ? BM * 128 : 256 * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES_RAW = kStageBudget / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
  static constexpr int ACC_COLS = SWAP ? ((KIND == 0) ? 2 * BM : BM) : 256;
  static constexpr int TMEM_COLS = !SWAP                   ? 512
                                   : (2 * ACC_COLS <= 32)  ? 32
                                   : (2 * ACC_COLS <= 64)  ? 64
                                   : (2 * ACC_COLS <= 128) ? 128
                                   : (2 * ACC_COLS <= 256) ? 256
                                                           : 512;
  static constexpr uint32_t IDESC = SWAP ? idesc_bf16_f32(128, BM) : idesc_bf16_f32(128, 256);
  // gather: 16-byte chunks per gather thread per stage (32*GW threads, 8
  // chunks per 128-byte token row)
  static constexpr int G_THREADS = 32 * GW;
  static constexpr int G_ROWS = SWAP ? BM : 128;
  static constexpr int G_PER_THREAD = G_ROWS * 8 / G_THREADS;
  static constexpr int THREADS = 64 + G_THREADS + 128;
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + BAR_BYTES;
  static_assert(G_PER_THREAD >= 2 && (G_ROWS * 8) % G_THREADS == 0, "gather split");
  static_assert(STAGE_BYTES % 1024 == 0, "stage tiles must keep 1024-byte alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Split count for the swap tiles: minimise waves x (k-blocks per unit + a
// per-unit overhead), within the partial-sum capacity.  The overhead is
// kSplitUnitCost k-blocks: a unit refills the operand pipeline from HBM and,
// split, writes fp32 partials that the last split reads back, about 7 us
// against about 0.5 us per k-block (fitted to GEMM1 times of the Qwen3 layer
// at 1, 4 and 5 tokens; 14, 20 and 28 time alike).  Lane l of the calling warp
// evaluates s = l + 1 (every lane must call); ties go to the fewest splits.
// 32-bit arithmetic: every product stays below 2^31.
constexpr int kSplitUnitCost = 14;
MOE_DEV int choose_splits(int ug, int KB, int ctas, int max_slots) {
  const int lane = threadIdx.x & 31;
  const int s = lane + 1;
  uint32_t key = 0xFFFFFFFFu;
  if (ug > 0 && s <= KB && (s == 1 || ug * s <= max_slots)) {
    const int waves = (ug * s + ctas - 1) / ctas;
    const int cost = waves * ((KB + s - 1) / s + kSplitUnitCost);
    key = (static_cast<uint32_t>(min(cost, (1 << 26) - 1)) << 5) | static_cast<uint32_t>(lane);
  }
  key = __reduce_min_sync(0xffffffffu, key);
  return (key == 0xFFFFFFFFu) ? 1 : static_cast<int>(key & 31u) + 1;
}

struct Sched {
  int nblk, ntiles, KB, S, num_units;
};

// Work decomposition, identical in every CTA: unit = (block, output tile,
// K split); blocks major, so the units of one block (and the blocks of one
// expert) run side by side and share their operand tiles through L2.
template <int KIND, int BM>
MOE_DEV Sched make_sched(const FfnParams& p) {
  using C = Cfg<KIND, BM>;
  Sched s;
  s.nblk = padded_rows(p, BM) / BM;
  s.ntiles = (KIND == 0) ? (p.F + C::NT - 1) / C::NT : (p.H + C::NT - 1) / C::NT;
  const int K = (KIND == 0) ? p.H : p.F;
  s.KB = (K + kBK - 1) / kBK;
  s.S = C::SWAP ? choose_splits(s.nblk * s.ntiles, s.KB, gridDim.x, p.max_slots) : 1;
  s.num_units = s.nblk * s.ntiles * s.S;
  return s;
}

struct Unit {
  int b, n, s, ug, kb0, kb1, e;
};

template <int KIND, int BM>
MOE_DEV Unit decode_unit(const FfnParams& p, const Sched& sc, int u) {
  Unit x;
  x.s = u % sc.S;
  x.ug = u / sc.S;
  x.b = x.ug / sc.ntiles;
  x.n = x.ug % sc.ntiles;
  x.kb0 = x.s * sc.KB / sc.S;  // KB <= 2^16 and s <= 32: no overflow
  x.kb1 = (x.s + 1) * sc.KB / sc.S;
  int e = __ldg(p.block_expert + x.b);
  if (e < 0 || e >= p.E) {
    if (threadIdx.x == 0) raise_error(p.err, kErrBadTable);
    e = min(max(e, 0), p.E - 1);
  }
  x.e = e;
  return x;
}

// 16 fp32 accumulator columns of this thread's TMEM lane.
MOE_DEV void load_cols(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  tmem_ld16(taddr, r);
  tmem_ld_wait();
  reg_fence16(r);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 summed split-K partial columns of one row (split order 0..S-1).
MOE_DEV void load_partial_cols(const float* base, size_t slot_stride, int S, float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 16; i += 4) {
    float4 t = __ldcg(reinterpret_cast<const float4*>(base + i));
    v[i] = t.x;
    v[i + 1] = t.y;
    v[i + 2] = t.z;
    v[i + 3] = t.w;
  }
  for (int s = 1; s < S; ++s) {
    const float* b = base + s * slot_stride;
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      float4 t = __ldcg(reinterpret_cast<const float4*>(b + i));
      v[i] += t.x;
      v[i + 1] += t.y;
      v[i + 2] += t.z;
      v[i + 3] += t.w;
    }
  }
}

// Epilogue of one swap tile (BLOCK_M 16/64) for the thread owning TMEM lane
// `row` (a feature of GEMM1, an output column of GEMM2).  `fetch(col, v)`
// returns 16 accumulator columns (tokens of the block) starting at `col`.
template <int KIND, int BM, class Fetch>
MOE_DEV void epilogue_tile(const FfnParams& p, const Unit& u, int row, Fetch&& fetch) {
  using C = Cfg<KIND, BM>;
  const int nk = p.T * p.k;
  if constexpr (KIND == 0 && C::SWAP) {
    // row = feature f0 + row; columns: gate tokens [0, BM), up tokens [BM, 2BM)
    const int f = u.n * C::NT + row;
    __nv_bfloat16* inter = reinterpret_cast<__nv_bfloat16*>(p.inter);
#pragma unroll 1
    for (int c0 = 0; c0 < BM; c0 += 16) {
      float g[16], v[16];
      fetch(c0, g);
      fetch(BM + c0, v);
      if (f < p.F) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const size_t prow = static_cast<size_t>(u.b) * BM + c0 + c;
          inter[prow * p.F + f] = __float2bfloat16_rn(swiglu_f(g[c], v[c]));
        }
      }
    }
  } else {
    // row = output column h of the layer; columns: the block's tokens
    const int h = u.n * C::NT + row;
    __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(p.stage);
#pragma unroll 1
    for (int c0 = 0; c0 < BM; c0 += 16) {
      float v[16];
      fetch(c0, v);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int a = row_assignment(p, u.b, BM, c0 + c);
        if (a >= 0 && a < nk && h < p.H) {
          const float w = __ldg(p.topk_weights + a);
          stage[static_cast<size_t>(a) * p.H + h] = __float2bfloat16_rn(v[c] * w);
        }
      }
    }
  }
}

// Epilogue of a 128-token tile (BLOCK_M 128) straight from TMEM, with the
// TMEM load of chunk c+1 in flight while chunk c is computed and stored.
template <int KIND>
MOE_DEV void epilogue_rows128(const FfnParams& p, const Unit& u, int row, uint32_t tb) {
  constexpr int NCH = (KIND == 0) ? 8 : 16;  // 16-column chunks of the tile
  constexpr int NT = (KIND == 0) ? 128 : 256;
  const size_t prow = static_cast<size_t>(u.b) * 128 + row;
  int a = 0;
  bool valid = true;
  float w = 1.f;
  if constexpr (KIND == 1) {
    a = row_assignment(p, u.b, 128, row);
    valid = a >= 0 && a < p.T * p.k;
    w = valid ? __ldg(p.topk_weights + a) : 0.f;
  }
  uint32_t ra[2][16], rb[2][16];
  tmem_ld16(tb, ra[0]);
  if constexpr (KIND == 0) tmem_ld16(tb + 128, rb[0]);
  tmem_ld_wait();
  reg_fence16(ra[0]);
  if constexpr (KIND == 0) reg_fence16(rb[0]);
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const int cur = c & 1, nxt = cur ^ 1;
    if (c + 1 < NCH) {
      tmem_ld16(tb + 16 * (c + 1), ra[nxt]);
      if constexpr (KIND == 0) tmem_ld16(tb + 128 + 16 * (c + 1), rb[nxt]);
    }
    const int col = u.n * NT + 16 * c;
    uint32_t o[8];
    if constexpr (KIND == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        o[i] = pack_bf16x2(swiglu_f(__uint_as_float(ra[cur][2 * i]), __uint_as_float(rb[cur][2 * i])),
                           swiglu_f(__uint_as_float(ra[cur][2 * i + 1]),
                                    __uint_as_float(rb[cur][2 * i + 1])));
      if (col + 16 <= p.F)
        st_global_v8(reinterpret_cast<__nv_bfloat16*>(p.inter) + prow * p.F + col, o);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        o[i] = pack_bf16x2(__uint_as_float(ra[cur][2 * i]) * w,
                           __uint_as_float(ra[cur][2 * i + 1]) * w);
      if (valid && col + 16 <= p.H)
        st_global_v8(reinterpret_cast<__nv_bfloat16*>(p.stage) + static_cast<size_t>(a) * p.H + col, o);
    }
    if (c + 1 < NCH) {
      tmem_ld_wait();
      reg_fence16(ra[nxt]);
      if constexpr (KIND == 0) reg_fence16(rb[nxt]);
    }
  }
}

template <int KIND, int BM, int GW>
__global__ void __launch_bounds__(Cfg<KIND, BM, GW>::THREADS, 1)
    ffn_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                    const __grid_constant__ CUtensorMap tm_in, const FfnParams p) {
  using C = Cfg<KIND, BM, GW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty_bar = full_bar + C::STAGES;
  uint64_t* tfull_bar = empty_bar + C::STAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty_bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Sched sc = make_sched<KIND, BM>(p);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full_bar[i], 1 + (C::GATHER ? C::G_THREADS : 0));
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], 4);
    }
    *abort_flag = 0;
    *last_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      if (KIND == 1) tma_prefetch_desc(&tm_in);
      uint32_t it = 0;
      bool alive = true;
      for (int uu = blockIdx.x; alive && uu < sc.num_units; uu += gridDim.x) {
        const Unit u = decode_unit<KIND, BM>(p, sc, uu);
        // row tiles: the CTA's next unit, so the L2 warm-up of weight tiles
        // runs across the unit boundary (decode tiles stream each weight once
        // and gain nothing from it)
        const bool has_next = uu + static_cast<int>(gridDim.x) < sc.num_units;
        const Unit nu =
            has_next ? decode_unit<KIND, BM>(p, sc, uu + gridDim.x) : u;
        for (int kb = u.kb0; kb < u.kb1; ++kb, ++it) {
          if constexpr (!C::SWAP) {
            int tkb = kb + C::STAGES;
            const Unit* tu = &u;
            if (tkb >= u.kb1 && has_next) {
              tkb = nu.kb0 + (tkb - u.kb1);
              tu = &nu;
            }
            if (tkb < tu->kb1) {
              if constexpr (KIND == 0) {
                const int grow = tu->e * 2 * p.F + tu->n * C::NT;
                tma_prefetch_l2_2d(&tm_w, tkb * kBK, grow);
                tma_prefetch_l2_2d(&tm_w, tkb * kBK, grow + p.F);
              } else {
                tma_prefetch_l2_2d(&tm_w, tkb * kBK, tu->e * p.H + tu->n * C::NT);
              }
            }
          }
          const int st = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&empty_bar[st], ph ^ 1u, abort_flag, p.err)) {
            alive = false;
            break;
          }
          uint8_t* sa = smem + st * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          const int kc = kb * kBK;
          if constexpr (KIND == 0) {
            const int grow = u.e * 2 * p.F + u.n * C::NT;
            uint8_t* dst = C::SWAP ? sa : sb;
            mbar_arrive_expect_tx(&full_bar[st], 2 * 128 * 128);
            tma_load_2d(dst, &tm_w, &full_bar[st], kc, grow);
            tma_load_2d(dst + 128 * 128, &tm_w, &full_bar[st], kc, grow + p.F);
          } else {
            const int wrow = u.e * p.H + u.n * C::NT;
            if constexpr (C::SWAP) {
              mbar_arrive_expect_tx(&full_bar[st], C::STAGE_BYTES);
              tma_load_2d(sa, &tm_w, &full_bar[st], kc, wrow);
              tma_load_2d(sb, &tm_in, &full_bar[st], kc, u.b * BM);
            } else {
              mbar_arrive_expect_tx(&full_bar[st], C::STAGE_BYTES);
              tma_load_2d(sa, &tm_in, &full_bar[st], kc, u.b * BM);
              tma_load_2d(sb, &tm_w, &full_bar[st], kc, wrow);
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, acc_it = 0;
      bool alive = true;
      for (int uu = blockIdx.x; alive && uu < sc.num_units; uu += gridDim.x, ++acc_it) {
        const Unit u = decode_unit<KIND, BM>(p, sc, uu);
        const int buf = acc_it & 1;
        const uint32_t aph = (acc_it >> 1) & 1u;
        if (!mbar_wait(&tempty_bar[buf], aph ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * C::ACC_COLS;
        for (int kb = u.kb0; kb < u.kb1; ++kb, ++it) {
          const int st = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&full_bar[st], ph, abort_flag, p.err)) {
            alive = false;
            break;
          }
          if constexpr (C::GATHER) fence_proxy_async_smem();  // cp.async rows -> tensor core
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + st * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t acc = (kb > u.kb0 || kk > 0) ? 1u : 0u;
            const uint64_t bdesc = sw128_desc(b_addr + kk * 32);
            umma_f16(d, sw128_desc(a_addr + kk * 32), bdesc, C::IDESC, acc);
            if constexpr (KIND == 0 && C::SWAP)
              umma_f16(d + BM, sw128_desc(a_addr + 128 * 128 + kk * 32), bdesc, C::IDESC, acc);
          }
          umma_commit(&empty_bar[st]);
        }
        if (!alive) break;
        umma_commit(&tfull_bar[buf]);
      }
    }
  } else if (warp < 2 + GW) {
    // ---------------- token-row gather (GEMM1) ----------------
    if constexpr (C::GATHER) {
      const int gt = threadIdx.x - 64;  // 0 .. G_THREADS-1
      const int chunk = gt & 7;
      const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(p.x);
      const int nk = p.T * p.k;
      uint32_t it = 0;
      bool alive = true;
      for (int uu = blockIdx.x; alive && uu < sc.num_units; uu += gridDim.x) {
        const Unit u = decode_unit<KIND, BM>(p, sc, uu);
        const __nv_bfloat16* src[C::G_PER_THREAD];
        uint32_t nbytes[C::G_PER_THREAD];
#pragma unroll
        for (int i = 0; i < C::G_PER_THREAD; ++i) {
          const int r = (gt >> 3) + (C::G_THREADS / 8) * i;
          const int a = row_assignment(p, u.b, BM, r);
          const bool valid = a >= 0 && a < nk;
          src[i] = valid ? x + static_cast<size_t>(a / p.k) * p.H + chunk * 8 : x;
          nbytes[i] = valid ? 16u : 0u;
        }
        for (int kb = u.kb0; kb < u.kb1; ++kb, ++it) {
          const int st = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&empty_bar[st], ph ^ 1u, abort_flag, p.err)) {
            alive = false;
            break;
          }
          const uint32_t tile = smem_u32(smem + st * C::STAGE_BYTES) + (C::SWAP ? C::A_BYTES : 0);
#pragma unroll
          for (int i = 0; i < C::G_PER_THREAD; ++i) {
            const int r = (gt >> 3) + (C::G_THREADS / 8) * i;
            const uint32_t dst = tile + r * 128 + ((chunk ^ (r & 7)) << 4);
            cp_async_16(dst, nbytes[i] ? src[i] + kb * kBK : src[i], nbytes[i]);
          }
          // the stage barrier counts this thread's arrival when its copies land;
          // the MMA issuer orders them before its tensor-core reads (proxy fence)
          cp_async_mbar_arrive_noinc(&full_bar[st]);
        }
      }
      cp_async_wait_all();
    }
  } else {
    // ---------------- epilogue ----------------
    const int ew = warp & 3;  // a warp reads the TMEM lane quarter warp % 4
    const int row = ew * 32 + lane;
    const int et = row;
    uint32_t acc_it = 0;
    for (int uu = blockIdx.x; uu < sc.num_units; uu += gridDim.x, ++acc_it) {
      const Unit u = decode_unit<KIND, BM>(p, sc, uu);
      const int buf = acc_it & 1;
      const uint32_t aph = (acc_it >> 1) & 1u;
      // every epilogue thread takes the same decision to stop
      const bool ok = mbar_wait(&tfull_bar[buf], aph, abort_flag, p.err);
      if (named_bar_any(1, 128, !ok || *abort_flag)) break;
      tc_fence_after();
      const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(ew * 32) << 16);
      const uint32_t tb = lane_base + buf * C::ACC_COLS;
      if (sc.S == 1) {
        if constexpr (!C::SWAP)
          epilogue_rows128<KIND>(p, u, row, tb);
        else
          epilogue_tile<KIND, BM>(p, u, row,
                                  [&](int col, float (&v)[16]) { load_cols(tb + col, v); });
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar[buf]);
      } else {
        // split-K: publish this split's partial, the last split finishes
        const size_t slot_stride = static_cast<size_t>(128) * C::ACC_COLS;
        float* mine = p.partial + (static_cast<size_t>(u.ug) * sc.S + u.s) * slot_stride +
                      static_cast<size_t>(row) * C::ACC_COLS;
#pragma unroll 1
        for (int c0 = 0; c0 < C::ACC_COLS; c0 += 16) {
          float v[16];
          load_cols(tb + c0, v);
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            __stcg(reinterpret_cast<float4*>(mine + c0 + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar[buf]);
        // one thread draws the ticket: release of the 128 rows just written,
        // acquire of the other splits' rows
        named_bar_sync(1, 128);
        if (et == 0) {
          const int old = ticket_add_acq_rel(p.tickets + u.ug, 1);
          const int last = (old == sc.S - 1);
          if (last) store_relaxed_gpu(p.tickets + u.ug, 0);  // ready for the next launch
          *last_flag = last;
        }
        named_bar_sync(1, 128);
        if (*last_flag) {
          const float* base0 = p.partial + static_cast<size_t>(u.ug) * sc.S * slot_stride +
                               static_cast<size_t>(row) * C::ACC_COLS;
          epilogue_tile<KIND, BM>(p, u, row, [&](int col, float (&v)[16]) {
            load_partial_cols(base0 + col, slot_stride, sc.S, v);
          });
        }
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Row tiles (BLOCK_M 128) on CTA pairs: the two CTAs of a cluster share the
// 256-row weight tile of a K step when they compute two blocks of the same
// expert ("paired" task): each loads one 128-row half and multicasts it to
// both, so each fetches 32 KB per step (its 16 KB token tile and one weight
// half) instead of 48 KB.  A block without a partner (the odd last block of
// an expert) runs as a "solo" task next to another solo block in the other
// CTA, each loading its whole weight tile; the two CTAs still step through
// the same number of K steps, and every stage is released only when both
// CTAs' MMAs are done with it (each MMA commit arrives on the stage's empty
// barrier in both CTAs), so a multicast never overwrites a stage that the
// other CTA still reads.
// ---------------------------------------------------------------------------
constexpr int kPairMaxBlocks = 4096;
constexpr uint16_t kNoBlock = 0xFFFF;

template <int KIND, int GW>
struct PairCfg {
  using C = Cfg<KIND, 128, GW>;
  static constexpr int TASK_BYTES = kPairMaxBlocks * 5;  // tb0, tb1 (u16), paired flag (u8)
  static constexpr int SMEM_BYTES = C::SMEM_BYTES + TASK_BYTES;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// The task list, identical in every CTA, in block order: paired tasks
// (blocks b, b+1 of one expert) and the solo blocks (the odd last block of
// an expert) two per task (the second slot kNoBlock when their number is
// odd), a solo task placed where its first block is -- so an expert's last
// block runs next to its pairs and finds its weight tiles in L2 (queued
// after all pairs, it fetched them again: DeepSeek-V3 layer T = 4096
// 3,694 -> 3,446 us).  All threads; scratch: nblk + 2,112 ints of shared
// memory the ring lends before its first load.
template <int NTHREADS>
MOE_DEV int build_pair_tasks(const int32_t* block_expert, int nblk, uint16_t* tb0, uint16_t* tb1,
                             uint8_t* tpair, int* scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = NTHREADS / 32;
  int* be = scratch;            // [nblk] block -> expert
  int* wsum = scratch + kPairMaxBlocks;  // [NW]
  for (int b = tid; b < nblk; b += NTHREADS) be[b] = __ldg(block_expert + b);
  __syncthreads();
  const int per = (nblk + NTHREADS - 1) / NTHREADS;
  const int b0 = min(nblk, tid * per), b1 = min(nblk, b0 + per);
  // role of each block: paired-first (even position in its expert's run with
  // a successor in the run) or solo (odd run, last block); counts packed as
  // solo << 16 | paired
  int mine = 0;
  for (int b = b0; b < b1; ++b) {
    const int e = be[b];
    int st = b;
    while (st > 0 && be[st - 1] == e) --st;
    int en = b;
    while (en + 1 < nblk && be[en + 1] == e) ++en;
    const int L = en - st + 1, j = b - st;
    if ((j & 1) == 0 && j + 1 < L) mine += 1;
    else if ((L & 1) && j == L - 1) mine += 1 << 16;
  }
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < NW ? wsum[lane] : 0;
    int sc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, sc, o);
      if (lane >= o) sc += u;
    }
    if (lane < NW) wsum[lane] = sc;
  }
  __syncthreads();
  const int total = wsum[NW - 1];
  const int NP = total & 0xFFFF, NS = total >> 16;
  const int before0 = incl - mine + (warp > 0 ? wsum[warp - 1] : 0);
  // tasks in block order: a paired task where its first block is, a solo
  // task where the first of its two solo blocks is; solo_pos[j]: the task
  // of solo pair j, which its second block joins after the barrier
  int* solo_pos = wsum + 64;
  int before = before0;
  for (int b = b0; b < b1; ++b) {
    const int e = be[b];
    int st = b;
    while (st > 0 && be[st - 1] == e) --st;
    int en = b;
    while (en + 1 < nblk && be[en + 1] == e) ++en;
    const int L = en - st + 1, j = b - st;
    const int np = before & 0xFFFF, ns = before >> 16;
    if ((j & 1) == 0 && j + 1 < L) {
      const int t = np + (ns + 1) / 2;
      tb0[t] = static_cast<uint16_t>(b);
      tb1[t] = static_cast<uint16_t>(b + 1);
      tpair[t] = 1;
      before += 1;
    } else if ((L & 1) && j == L - 1) {
      if ((ns & 1) == 0) {
        const int t = np + ns / 2;
        tb0[t] = static_cast<uint16_t>(b);
        tb1[t] = kNoBlock;
        tpair[t] = 0;
        solo_pos[ns / 2] = t;
      }
      before += 1 << 16;
    }
  }
  __syncthreads();
  before = before0;
  for (int b = b0; b < b1; ++b) {
    const int e = be[b];
    int st = b;
    while (st > 0 && be[st - 1] == e) --st;
    int en = b;
    while (en + 1 < nblk && be[en + 1] == e) ++en;
    const int L = en - st + 1, j = b - st;
    if ((j & 1) == 0 && j + 1 < L) {
      before += 1;
    } else if ((L & 1) && j == L - 1) {
      const int ns = before >> 16;
      if (ns & 1) tb1[solo_pos[ns / 2]] = static_cast<uint16_t>(b);
      before += 1 << 16;
    }
  }
  __syncthreads();
  return NP + (NS + 1) / 2;
}

template <int KIND, int GW>
__global__ void __launch_bounds__(Cfg<KIND, 128, GW>::THREADS, 1)
    ffn_pair_kernel(const __grid_constant__ CUtensorMap tm_w,
                    const __grid_constant__ CUtensorMap tm_in, const FfnParams p) {
  using C = Cfg<KIND, 128, GW>;
  constexpr int HALF = 128 * 128;  // one 128-row half of the weight tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty_bar = full_bar + C::STAGES;
  uint64_t* tfull_bar = empty_bar + C::STAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty_bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint16_t* tb0 = reinterpret_cast<uint16_t*>(smem + C::STAGES * C::STAGE_BYTES + C::BAR_BYTES);
  uint16_t* tb1 = tb0 + kPairMaxBlocks;
  uint8_t* tpair = reinterpret_cast<uint8_t*>(tb1 + kPairMaxBlocks);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const int nblk = min(padded_rows(p, 128) / 128, kPairMaxBlocks);
  const int ntasks = build_pair_tasks<C::THREADS>(p.block_expert, nblk, tb0, tb1, tpair,
                                                  reinterpret_cast<int*>(smem));
  fence_proxy_async_smem();  // the ring lent scratch: TMA writes it next
  const int ntiles = (KIND == 0) ? (p.F + 127) / 128 : (p.H + 255) / 256;
  // K steps (GEMM2: F % 64 may be 32; the copy zero-fills past F)
  const int KB = (((KIND == 0) ? p.H : p.F) + kBK - 1) / kBK;
  const int num_units = ntasks * ntiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full_bar[i], 1 + (C::GATHER ? C::G_THREADS : 0));
      mbar_init(&empty_bar[i], 2);  // both CTAs' MMA commits
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], 4);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  // the other CTA's barriers exist before any multicast or remote commit
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  struct PU {
    int b, n, e, eb;
    bool paired;
  };
  auto task_expert = [&](int t) { return __ldg(p.block_expert + tb0[t]); };
  auto unit_of = [&](int uu) {
    PU x;
    int t = uu / ntiles;
    x.n = uu % ntiles;
    if (tpair[t]) {
      // a run of paired tasks of one expert walks its output tiles n-major:
      // the clusters on the run share each weight tile at about the same
      // time (fetched about once instead of once per wave of the run), while
      // the run's token rows stay in L2 across its output tiles (DeepSeek-V3
      // layer T = 4096 3,485 -> 3,420 us)
      const int e0 = task_expert(t);
      int t0 = t, t1 = t + 1;
      while (t0 > 0 && tpair[t0 - 1] && task_expert(t0 - 1) == e0) --t0;
      while (t1 < ntasks && tpair[t1] && task_expert(t1) == e0) ++t1;
      const int L = t1 - t0;
      if (L > 1) {
        const int v = uu - t0 * ntiles;
        x.n = v / L;
        t = t0 + v % L;
      }
    }
    x.paired = tpair[t] != 0;
    const uint16_t bb = rank == 0 ? tb0[t] : tb1[t];
    x.b = bb == kNoBlock ? -1 : static_cast<int>(bb);
    x.eb = x.b >= 0 ? x.b : static_cast<int>(tb0[t]);  // a null slot loads its partner's tiles
    int e = __ldg(p.block_expert + x.eb);
    if (e < 0 || e >= p.E) {
      if (threadIdx.x == 0) raise_error(p.err, kErrBadTable);
      e = min(max(e, 0), p.E - 1);
    }
    x.e = e;
    return x;
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      if (KIND == 1) tma_prefetch_desc(&tm_in);
      uint32_t it = 0;
      bool alive = true;
      for (int uu = cid; alive && uu < num_units; uu += ncl) {
        const PU u = unit_of(uu);
        // weight rows of the two halves of this unit's tile
        const int h0 = (KIND == 0) ? u.e * 2 * p.F + u.n * 128 : u.e * p.H + u.n * 256;
        const int h1 = (KIND == 0) ? h0 + p.F : h0 + 128;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          // warm L2 with this CTA's halves a ring ahead
          if (kb + C::STAGES < KB) {
            const int pk = (kb + C::STAGES) * kBK;
            if (!u.paired || rank == 0) tma_prefetch_l2_2d(&tm_w, pk, h0);
            if (!u.paired || rank == 1) tma_prefetch_l2_2d(&tm_w, pk, h1);
          }
          const int st = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&empty_bar[st], ph ^ 1u, abort_flag, p.err)) {
            alive = false;
            break;
          }
          uint8_t* sa = smem + st * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          const int kc = kb * kBK;
          mbar_arrive_expect_tx(&full_bar[st], KIND == 0 ? C::B_BYTES : C::STAGE_BYTES);
          if constexpr (KIND == 1) tma_load_2d(sa, &tm_in, &full_bar[st], kc, u.eb * 128);
          if (u.paired) {
            tma_load_2d_mc(sb + rank * HALF, &tm_w, &full_bar[st], kc, rank == 0 ? h0 : h1, 0x3);
          } else {
            tma_load_2d(sb, &tm_w, &full_bar[st], kc, h0);
            tma_load_2d(sb + HALF, &tm_w, &full_bar[st], kc, h1);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, acc_it = 0;
      bool alive = true;
      for (int uu = cid; alive && uu < num_units; uu += ncl, ++acc_it) {
        const int buf = acc_it & 1;
        const uint32_t aph = (acc_it >> 1) & 1u;
        if (!mbar_wait(&tempty_bar[buf], aph ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * C::ACC_COLS;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int st = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&full_bar[st], ph, abort_flag, p.err)) {
            alive = false;
            break;
          }
          if constexpr (C::GATHER) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + st * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_f16(d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32), C::IDESC,
                     (kb > 0 || kk > 0) ? 1u : 0u);
          umma_commit_mc(&empty_bar[st], 0x3);  // the stage is free once both CTAs are done
        }
        if (!alive) break;
        umma_commit(&tfull_bar[buf]);
      }
    }
  } else if (warp < 2 + GW) {
    // ---------------- token-row gather (GEMM1) ----------------
    if constexpr (C::GATHER) {
      const int gt = threadIdx.x - 64;
      const int chunk = gt & 7;
      const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(p.x);
      const int nk = p.T * p.k;
      uint32_t it = 0;
      bool alive = true;
      for (int uu = cid; alive && uu < num_units; uu += ncl) {
        const PU u = unit_of(uu);
        const __nv_bfloat16* src[C::G_PER_THREAD];
        uint32_t nbytes[C::G_PER_THREAD];
#pragma unroll
        for (int i = 0; i < C::G_PER_THREAD; ++i) {
          const int r = (gt >> 3) + (C::G_THREADS / 8) * i;
          const int a = u.b >= 0 ? row_assignment(p, u.b, 128, r) : nk;
          const bool valid = a >= 0 && a < nk;
          src[i] = valid ? x + static_cast<size_t>(a / p.k) * p.H + chunk * 8 : x;
          nbytes[i] = valid ? 16u : 0u;
        }
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int st = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1u;
          if (!mbar_wait(&empty_bar[st], ph ^ 1u, abort_flag, p.err)) {
            alive = false;
            break;
          }
          const uint32_t tile = smem_u32(smem + st * C::STAGE_BYTES);
#pragma unroll
          for (int i = 0; i < C::G_PER_THREAD; ++i) {
            const int r = (gt >> 3) + (C::G_THREADS / 8) * i;
            const uint32_t dst = tile + r * 128 + ((chunk ^ (r & 7)) << 4);
            cp_async_16(dst, nbytes[i] ? src[i] + kb * kBK : src[i], nbytes[i]);
          }
          cp_async_mbar_arrive_noinc(&full_bar[st]);
        }
      }
      cp_async_wait_all();
    }
  } else {
    // ---------------- epilogue ----------------
    const int ew = warp & 3;
    const int row = ew * 32 + lane;
    uint32_t acc_it = 0;
    for (int uu = cid; uu < num_units; uu += ncl, ++acc_it) {
      const PU pu = unit_of(uu);
      const int buf = acc_it & 1;
      const uint32_t aph = (acc_it >> 1) & 1u;
      const bool ok = mbar_wait(&tfull_bar[buf], aph, abort_flag, p.err);
      if (named_bar_any(1, 128, !ok || *abort_flag)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + buf * C::ACC_COLS;
      if (pu.b >= 0) {
        Unit u{};
        u.b = pu.b;
        u.n = pu.n;
        u.e = pu.e;
        epilogue_rows128<KIND>(p, u, row, tb);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[buf]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  // neither CTA leaves while the other may still multicast into it or
  // commit onto its barriers
  cluster_sync_all();
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D bf16 map of a row-major [rows, cols] matrix; box = 64 columns x box_rows.
bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_rows) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte map of a row-major [rows, cols] byte matrix; box = 128 bytes x
// box_rows rows, 128-byte swizzle, zero fill out of bounds.
bool make_map_u8_sw128(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_rows) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map of packed e2m1 codes [rows, cols codes], cols/2 bytes per row;
// box = 128 codes x box_rows rows, each 16 codes widened to a 16-byte slot
// in shared memory, 128-byte swizzle.
bool make_map_e2m1(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_rows) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 31u) != 0 || cols % 128 != 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols / 2};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <int KIND, int BM, int GW = 2>
int launch_kind(const CUtensorMap& tw, const CUtensorMap& tin, const FfnParams& p, int num_sms,
                cudaStream_t stream) {
  using C = Cfg<KIND, BM, GW>;
  static std::atomic<unsigned long long> smem_set{0};
  if (!ensure_smem_limit(reinterpret_cast<const void*>(ffn_gemm_kernel<KIND, BM, GW>),
                         C::SMEM_BYTES, smem_set))
    return -1;
  ffn_gemm_kernel<KIND, BM, GW><<<num_sms, C::THREADS, C::SMEM_BYTES, stream>>>(tw, tin, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

template <int KIND, int GW>
int launch_pair(const CUtensorMap& tw, const CUtensorMap& tin, const FfnParams& p, int num_sms,
                cudaStream_t stream, const char** why) {
  using PC = PairCfg<KIND, GW>;
  using C = Cfg<KIND, 128, GW>;
  static std::atomic<unsigned long long> smem_set{0};
  if (!ensure_smem_limit(reinterpret_cast<const void*>(ffn_pair_kernel<KIND, GW>),
                         PC::SMEM_BYTES, smem_set)) {
    *why = "CTA-pair kernel: shared-memory limit not accepted";
    return -1;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(num_sms & ~1);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = PC::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // as many CTA pairs as fit at once (a GPC with an odd number of free SMs
  // leaves one out): the kernel is persistent, every pair must be resident
  // (co-residency is for speed only: no CTA waits on another cluster, so
  // when the query gives nothing, one pair per two SMs is launched and a
  // pair that cannot be placed at once runs when one leaves)
  int nclusters = 0;
  if (cudaOccupancyMaxActiveClusters(&nclusters, ffn_pair_kernel<KIND, GW>, &cfg) != cudaSuccess ||
      nclusters < 1) {
    (void)cudaGetLastError();
    nclusters = num_sms / 2;
  }
  cfg.gridDim = dim3(2 * (nclusters < num_sms / 2 ? nclusters : num_sms / 2));
  if (cudaLaunchKernelEx(&cfg, ffn_pair_kernel<KIND, GW>, tw, tin, p) != cudaSuccess) {
    *why = "CTA-pair kernel: launch failed";
    return -1;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// GEMM1 row tiles gather with four warps; up to this H one CTA runs a tile,
// above it CTA pairs do (with four warps each), and the single-CTA kernel
// that remains above it (task lists past kPairMaxBlocks) keeps two (measured
// per shape on GB300).
constexpr int kGather4MaxH = 4096;

int ffn_max_slots(int block_m) { return block_m == 16 ? 1024 : (block_m == 64 ? 256 : 0); }

size_t ffn_partial_bytes(int block_m) {
  // GEMM1 (two accumulators of block_m columns) needs the most per slot
  return align_up(static_cast<size_t>(ffn_max_slots(block_m)) * 128 * 2 * block_m * 4, 256);
}

int launch_ffn_gemm(int kind, int block_m, const void* w, const FfnParams& p, int num_sms,
                    cudaStream_t stream, const char** why) {
  CUtensorMap tw, tin;
  const bool swap = block_m < 128;
  // row tiles above H = kGather4MaxH run on CTA pairs that share the weight
  // tile (measured: DeepSeek-V3 shape, H = 7168, layer 5-7.5 % faster;
  // Qwen3 shape, H = 2048, up to 21 % slower), when the task list fits
  const bool pair = block_m == 128 && p.H > kGather4MaxH &&
                    static_cast<long long>(p.cap_rows) / 128 <= kPairMaxBlocks;
  if (kind == 0) {
    // w13 [E*2F, H], box 64 x 128
    if (!make_map_bf16(&tw, w, static_cast<uint64_t>(p.E) * 2 * p.F, p.H, 128)) {
      *why = "cuTensorMapEncodeTiled failed for w13";
      return -1;
    }
    tin = tw;
  } else {
    // (row tiles on CTA pairs load the weight tile as two 128-row halves)
    if (!make_map_bf16(&tw, w, static_cast<uint64_t>(p.E) * p.H, p.F,
                       (swap || pair) ? 128 : 256)) {
      *why = "cuTensorMapEncodeTiled failed for w2";
      return -1;
    }
    if (!make_map_bf16(&tin, p.inter, static_cast<uint64_t>(p.cap_rows), p.F, block_m)) {
      *why = "cuTensorMapEncodeTiled failed for the intermediate";
      return -1;
    }
  }
  int rc = -1;
  if (kind == 0) {
    if (block_m == 16) rc = launch_kind<0, 16>(tw, tin, p, num_sms, stream);
    else if (block_m == 64) rc = launch_kind<0, 64>(tw, tin, p, num_sms, stream);
    else if (p.H <= kGather4MaxH) rc = launch_kind<0, 128, 4>(tw, tin, p, num_sms, stream);
    else if (pair) rc = launch_pair<0, 4>(tw, tin, p, num_sms, stream, why);
    else rc = launch_kind<0, 128>(tw, tin, p, num_sms, stream);
  } else {
    if (block_m == 16) rc = launch_kind<1, 16>(tw, tin, p, num_sms, stream);
    else if (block_m == 64) rc = launch_kind<1, 64>(tw, tin, p, num_sms, stream);
    else if (pair) rc = launch_pair<1, 2>(tw, tin, p, num_sms, stream, why);
    else rc = launch_kind<1, 128>(tw, tin, p, num_sms, stream);
  }
  if (rc != 0 && **why == '\0') *why = "kernel launch failed";
  return rc;
}

}  // namespace moe
