// decode.cu -- the whole MoE layer in ONE persistent kernel for small batches
// (T*k <= 512: the decode regime, where five dependent launches and their
// metadata reads, not bandwidth, set the layer's time).
//
// Follows "How GPUs Fuse Communication and Computation During LLM Inference":
// §3.3 (an expert's GEMM 1 starts as soon as its tokens are there, signalled
// by readiness counters), §3.4 (the fused kernel on one GPU), §3.6 (GEMM 2
// tasks start before GEMM 1 is finished, each waiting only for the rows it
// reads, so the SMs keep streaming expert weights across the boundary); the
// steps themselves are those of the separate kernels: the one-launch router
// ("How an MoE Model Picks Its Experts During LLM Inference" §5.1, §5.3),
// moe_align_block_size ("MoE Kernels, in depth", Alignment), the grouped
// GEMMs with SwiGLU and the routing weight in their epilogues ("MoE Kernels,
// in depth", The fused expert GEMM) and the fixed-order combine ("MoE
// Kernels, in depth", Combine).
//
// One cooperative launch of one CTA per SM (all CTAs resident, so they may
// wait on one another; every wait is bounded), 8 warps:
//   R. Router: CTA i < (expert tiles x token tiles x K slices) runs one item
//      of the one-launch router (router_device.cuh); the last item of a token
//      tile selects and publishes the tile (release counter).  Every CTA then
//      waits until all token tiles are routed.
//   A. Align, in every CTA's shared memory: the T*k assignments sorted by
//      expert (ascending expert id, within an expert ascending assignment
//      id), cut into blocks of 16 rows: block b = (expert, first row, rows).
//   G. Units, handed out round-robin over the CTAs, all GEMM1 units first:
//      GEMM1 unit (block, 128 features, K split) and GEMM2 unit (block, 128
//      output columns, K split); warp-specialised like the separate GEMMs
//      (warp 0 TMA of the weight tiles, warp 1 TMEM + the tcgen05.mma thread,
//      warps 2-3 the 16 token rows by cp.async, warps 4-7 the epilogue).
//      The weights are the MMA's M = 128 and the block's 16 tokens its N.
//      A GEMM1 unit's finishing epilogue writes SwiGLU rows of the
//      intermediate and bumps its block's readiness counter; the loads of a
//      GEMM2 unit's intermediate rows wait for that counter to reach the
//      block's feature-tile count, while its weight tiles stream in
//      meanwhile.  A GEMM2 unit's finishing epilogue writes the weighted
//      slot rows and bumps a counter per (token, column tile); the epilogue
//      that brings it to k sums the token's k slot rows in slot order (fp32)
//      and writes the output.
//   The counters of the workspace region (block readiness, token tiles,
//   split tickets) are zeroed by the CTAs at the start of every launch (the
//   GEMM phase waits for all of them), so the region may hold anything other
//   entry points left there; the last CTA to finish resets the three header
//   counters (routed, zeroed, done) for the next launch.
// No wait depends on a later unit: every CTA runs its GEMM1 units before its
// GEMM2 units, and GEMM1 units wait on nothing but the routing.
#include "moe_common.cuh"
#include "moe_internal.h"
#include "router_device.cuh"

namespace moe {

namespace {

constexpr int kDThreads = 256;
constexpr int kDBM = 16;                          // rows per block (MMA N)
constexpr int kDBK = 64;                          // K elements per stage
constexpr int kDA1 = 2 * 128 * 128;               // GEMM1 A: 128 gate + 128 up rows
constexpr int kDA2 = 128 * 128;                   // GEMM2 A: 128 rows of w2
constexpr int kDBOff = kDA1;                      // B (16 token rows) after A
constexpr int kDStage = kDA1 + kDBM * 128;        // 34 KB
constexpr int kDStages = 6;
constexpr int kDRing = kDStages * kDStage;
constexpr int kDAcc = 32;                         // accumulator columns (gate 16 + up 16)
constexpr int kDTmemCols = 64;                    // two accumulators
constexpr int kDMaxAsg = kDecodeMaxAssignments;   // T*k
constexpr int kDMaxE = 512;
constexpr int kDGatherThreads = 64;
constexpr uint32_t kDIdesc = idesc_bf16_f32(128, kDBM);
// split-K: a unit costs this many k-blocks beyond its own (see ffn.cu)
constexpr int kDSplitUnitCost = 14;

static_assert(kDStage % 1024 == 0, "stage alignment");

struct DecParams {
  RouterArgs r;           // router: hidden, gate, bias, partial logits, tickets, ids, weights
  int r_ne, r_nt;         // router items: expert tiles x token tiles (x r.KS K slices)
  const __nv_bfloat16* x;
  __nv_bfloat16* inter;   // [T*k*16, F]
  __nv_bfloat16* stage;   // [T*k, H]
  __nv_bfloat16* out;     // [T, H]
  float* part1;           // GEMM1 split partials [slots][128][32]
  float* part2;           // GEMM2 split partials [slots][128][16]
  int* tick1;             // [max_slots]
  int* tick2;
  int* ready;             // [T*k] per block: finished GEMM1 feature tiles
  int* tokcnt;            // [T * ceil(H/128)]
  int* routed;            // routed token tiles
  int* zeroed;            // CTAs that have zeroed their share of the region's counters
  int* done;              // finished CTAs
  int nzero;              // ints from `ready` on that every launch zeroes first
  int* err;
  int T, H, F, E, k;
  int max_slots;
};

struct DSmem {
  uint64_t full[kDStages], empty[kDStages], tfull[2], tempty[2];
  uint32_t tmem_slot;
  int abort_flag, last_flag, s_flag;
  int nblk, S1, S2;
  int fin[kDBM];
  int sa[kDMaxAsg];       // assignments sorted by expert
  int blk_e[kDMaxAsg];    // block -> expert
  int blk_s[kDMaxAsg];    // block -> index of its first row in sa
  int blk_n[kDMaxAsg];    // block -> rows (1..16)
};

constexpr int kDSmemBytes = kDRing + 1024 + static_cast<int>(sizeof(DSmem));
static_assert(kDSmemBytes <= 232448, "shared memory budget");

MOE_DEV void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded spin (one thread) until *p >= target; false on timeout or abort.
MOE_DEV bool wait_at_least(const int* p, int target, volatile int* abort_flag, int* err) {
  const long long t0 = clock64();
  while (load_acquire_gpu(p) < target) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      *abort_flag = 1;
      raise_error(err, kErrTimeout);
      return false;
    }
    __nanosleep(32);
  }
  return true;
}

MOE_DEV int choose_splits_d(int ug, int KB, int ctas, int max_slots) {
  const int lane = threadIdx.x & 31;
  const int s = lane + 1;
  uint32_t key = 0xFFFFFFFFu;
  if (ug > 0 && s <= KB && (s == 1 || ug * s <= max_slots)) {
    const int waves = (ug * s + ctas - 1) / ctas;
    const int cost = waves * ((KB + s - 1) / s + kDSplitUnitCost);
    key = (static_cast<uint32_t>(min(cost, (1 << 26) - 1)) << 5) | static_cast<uint32_t>(lane);
  }
  key = __reduce_min_sync(0xffffffffu, key);
  return (key == 0xFFFFFFFFu) ? 1 : static_cast<int>(key & 31u) + 1;
}

struct DUnit {
  int kind, b, n, s, ug, kb0, kb1, e, S;
};

struct DSched {
  int nblk, nt1, nt2, KB1, KB2, S1, S2, nu1, nu;
};

MOE_DEV DUnit decode_unit(const DSched& sc, const DSmem& sm, int u) {
  DUnit x;
  int uu = u, nt = sc.nt1, KB = sc.KB1;
  x.kind = 0;
  x.S = sc.S1;
  if (u >= sc.nu1) {
    uu = u - sc.nu1;
    nt = sc.nt2;
    KB = sc.KB2;
    x.kind = 1;
    x.S = sc.S2;
  }
  x.s = uu % x.S;
  x.ug = uu / x.S;
  x.b = x.ug / nt;
  x.n = x.ug % nt;
  x.kb0 = x.s * KB / x.S;
  x.kb1 = (x.s + 1) * KB / x.S;
  x.e = sm.blk_e[x.b];
  return x;
}

// assignment held by row r of block b, or -1 for a padding row
MOE_DEV int row_asg(const DSmem& sm, int b, int r) {
  return r < sm.blk_n[b] ? sm.sa[sm.blk_s[b] + r] : -1;
}

MOE_DEV void load_cols16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  tmem_ld16(taddr, r);
  tmem_ld_wait();
  reg_fence16(r);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

MOE_DEV void load_part16(const float* base, size_t slot_stride, int S, float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 16; i += 4) {
    const float4 t = __ldcg(reinterpret_cast<const float4*>(base + i));
    v[i] = t.x;
    v[i + 1] = t.y;
    v[i + 2] = t.z;
    v[i + 3] = t.w;
  }
  for (int s = 1; s < S; ++s) {
    const float* b = base + s * slot_stride;
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const float4 t = __ldcg(reinterpret_cast<const float4*>(b + i));
      v[i] += t.x;
      v[i + 1] += t.y;
      v[i + 2] += t.z;
      v[i + 3] += t.w;
    }
  }
}

// Step A: the block table of the routed assignments, in shared memory.
// Same blocks as moe_align with BLOCK_M 16: experts in ascending id, within
// an expert the assignments in ascending id, ceil(count/16) blocks each.
MOE_DEV void build_blocks(const DecParams& p, DSmem& sm, int* cnt, int* off, int* bstart,
                          int* sid) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = p.T * p.k, E = p.E;
  for (int e = tid; e < E; e += kDThreads) {
    cnt[e] = 0;
    off[e] = 0;
  }
  __syncthreads();
  // the router's ids, read once (one L2 round trip) into shared memory
  for (int a = tid; a < n; a += kDThreads) {
    int e = __ldcg(p.r.ids + a);
    if (e >= 0 && e < E) {
      atomicAdd(&cnt[e], 1);
    } else {
      raise_error(p.err, kErrBadExpert);
      e = -1;
    }
    sid[a] = e;
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive scans of the counts (row starts) and of the block counts;
    // lane l owns experts [l*per, (l+1)*per)
    const int per = (E + 31) / 32;
    int rs = 0, bs = 0;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        rs += cnt[e];
        bs += (cnt[e] + kDBM - 1) / kDBM;
      }
    }
    int ri = rs, bi = bs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int r2 = __shfl_up_sync(0xffffffffu, ri, o);
      const int b2 = __shfl_up_sync(0xffffffffu, bi, o);
      if (lane >= o) {
        ri += r2;
        bi += b2;
      }
    }
    int r0 = ri - rs, b0 = bi - bs;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        off[e] = r0;  // row start of expert e in sa (a running position below)
        bstart[e] = b0;
        r0 += cnt[e];
        b0 += (cnt[e] + kDBM - 1) / kDBM;
      }
    }
    if (lane == 31) sm.nblk = bi;
    __syncwarp();
    // place in ascending assignment order, 32 at a time: lanes holding the
    // same expert (one ballot per id bit) take consecutive positions
    const int nbits = 32 - __clz(max(E - 1, 1));
    for (int c0 = 0; c0 < n; c0 += 32) {
      const int a = c0 + lane;
      const int e = (a < n) ? sid[a] : -1;
      unsigned m = __ballot_sync(0xffffffffu, e >= 0);
      for (int bit = 0; bit < nbits; ++bit) {
        const bool v = (e >> bit) & 1;
        const unsigned bal = __ballot_sync(0xffffffffu, v);
        m &= v ? bal : ~bal;
      }
      const int pos0 = (e >= 0) ? off[e] : 0;
      __syncwarp();
      if (e >= 0) {
        sm.sa[pos0 + __popc(m & ((1u << lane) - 1u))] = a;
        if (lane == __ffs(m) - 1) off[e] = pos0 + __popc(m);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // block table: expert e's blocks start at bstart[e]; its rows end at off[e]
  for (int e = tid; e < E; e += kDThreads) {
    const int c = cnt[e];
    if (c == 0) continue;
    const int r0 = off[e] - c;
    for (int j = 0; j * kDBM < c; ++j) {
      const int b = bstart[e] + j;
      sm.blk_e[b] = e;
      sm.blk_s[b] = r0 + j * kDBM;
      sm.blk_n[b] = min(kDBM, c - j * kDBM);
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kDThreads, 1)
    decode_layer_kernel(const __grid_constant__ CUtensorMap tm_w13,
                        const __grid_constant__ CUtensorMap tm_w2, const DecParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  DSmem& sm = *reinterpret_cast<DSmem*>(ring + kDRing);
  volatile int* abort_flag = &sm.abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;

  if (tid == 0) {
    for (int i = 0; i < kDStages; ++i) {
      mbar_init(&sm.full[i], 1 + kDGatherThreads);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.tfull[i], 1);
      mbar_init(&sm.tempty[i], 4);
    }
    sm.abort_flag = 0;
    sm.last_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(&sm.tmem_slot, kDTmemCols);

  // ---- zero this CTA's share of the counters in the region (ready,
  // tokcnt, split tickets: contiguous ints from p.ready), whatever another
  // entry point left in the workspace; the GEMM phase waits for all shares
  {
    const int per = (p.nzero + G - 1) / G;
    const int z0 = blockIdx.x * per, z1 = min(p.nzero, z0 + per);
    for (int i = z0 + tid; i < z1; i += kDThreads) p.ready[i] = 0;
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      red_release_add(p.zeroed, 1);
    }
  }

  // ---- R: router items; the last item of each token tile selects ----
  const int items = p.r_ne * p.r_nt * p.r.KS;
  if (static_cast<int>(blockIdx.x) < items) {
    const int it = blockIdx.x;
    const int bx = it % p.r_ne, by = (it / p.r_ne) % p.r_nt, bz = it / (p.r_ne * p.r_nt);
    // the ring's memory is free until the GEMM phase
    const bool sel = router_item<0, 0, 1>(p.r, bx, by, bz, p.r_ne * p.r.KS,
                                          reinterpret_cast<float*>(ring), &sm.s_flag);
    __syncthreads();
    if (sel && tid == 0) {
      __threadfence();
      red_release_add(p.routed, 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem_slot;
  if (tid == 0 && wait_at_least(p.routed, p.r_nt, abort_flag, p.err))
    wait_at_least(p.zeroed, G, abort_flag, p.err);
  __syncthreads();

  // ---- A: block table; G: schedule ----
  DSched sc{};
  if (!*abort_flag) {
    int* scratch = reinterpret_cast<int*>(ring);  // free until the GEMM phase
    build_blocks(p, sm, scratch, scratch + kDMaxE, scratch + 2 * kDMaxE, scratch + 3 * kDMaxE);
    if (warp == 0) {
      const int nb = sm.nblk;
      const int s1 = choose_splits_d(nb * ((p.F + 127) / 128), p.H / kDBK, G, p.max_slots);
      const int s2 = choose_splits_d(nb * ((p.H + 127) / 128), p.F / kDBK, G, p.max_slots);
      if (lane == 0) {
        sm.S1 = s1;
        sm.S2 = s2;
      }
    }
    // the ring held generic-proxy data (router, tables); TMA writes it next
    fence_proxy_async_smem();
    __syncthreads();
    sc.nblk = sm.nblk;
    sc.nt1 = (p.F + 127) / 128;
    sc.nt2 = (p.H + 127) / 128;
    sc.KB1 = p.H / kDBK;
    sc.KB2 = p.F / kDBK;
    sc.S1 = sm.S1;
    sc.S2 = sm.S2;
    sc.nu1 = sc.nblk * sc.nt1 * sc.S1;
    sc.nu = sc.nu1 + sc.nblk * sc.nt2 * sc.S2;
  }

  if (warp == 0) {
    // ---------------- TMA producer: weight tiles ----------------
    if (lane == 0 && !*abort_flag) {
      tma_prefetch_desc(&tm_w13);
      tma_prefetch_desc(&tm_w2);
      uint32_t it = 0;
      bool alive = true;
      for (int u = blockIdx.x; alive && u < sc.nu; u += G) {
        const DUnit U = decode_unit(sc, sm, u);
        for (int kb = U.kb0; kb < U.kb1; ++kb, ++it) {
          const int st = it % kDStages;
          const uint32_t ph = (it / kDStages) & 1u;
          if (!mbar_wait(&sm.empty[st], ph ^ 1u, abort_flag, p.err)) {
            alive = false;
            break;
          }
          uint8_t* sa = ring + st * kDStage;
          const int kc = kb * kDBK;
          if (U.kind == 0) {
            const int grow = U.e * 2 * p.F + U.n * 128;
            mbar_arrive_expect_tx(&sm.full[st], kDA1);
            tma_load_2d(sa, &tm_w13, &sm.full[st], kc, grow);
            tma_load_2d(sa + 128 * 128, &tm_w13, &sm.full[st], kc, grow + p.F);
          } else {
            mbar_arrive_expect_tx(&sm.full[st], kDA2);
            tma_load_2d(sa, &tm_w2, &sm.full[st], kc, U.e * p.H + U.n * 128);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && !*abort_flag) {
      uint32_t it = 0, acc_it = 0;
      bool alive = true;
      for (int u = blockIdx.x; alive && u < sc.nu; u += G, ++acc_it) {
        const DUnit U = decode_unit(sc, sm, u);
        const int buf = acc_it & 1;
        const uint32_t aph = (acc_it >> 1) & 1u;
        if (!mbar_wait(&sm.tempty[buf], aph ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * kDAcc;
        for (int kb = U.kb0; kb < U.kb1; ++kb, ++it) {
          const int st = it % kDStages;
          const uint32_t ph = (it / kDStages) & 1u;
          if (!mbar_wait(&sm.full[st], ph, abort_flag, p.err)) {
            alive = false;
            break;
          }
          fence_proxy_async_smem();  // cp.async token rows -> tensor core
          tc_fence_after();
          const uint32_t a_addr = smem_u32(ring + st * kDStage);
          const uint32_t b_addr = a_addr + kDBOff;
#pragma unroll
          for (int kk = 0; kk < kDBK / 16; ++kk) {
            const uint32_t acc = (kb > U.kb0 || kk > 0) ? 1u : 0u;
            const uint64_t bdesc = sw128_desc(b_addr + kk * 32);
            umma_f16(d, sw128_desc(a_addr + kk * 32), bdesc, kDIdesc, acc);
            if (U.kind == 0)
              umma_f16(d + kDBM, sw128_desc(a_addr + 128 * 128 + kk * 32), bdesc, kDIdesc, acc);
          }
          umma_commit(&sm.empty[st]);
        }
        if (!alive) break;
        umma_commit(&sm.tfull[buf]);
      }
    }
  } else if (warp < 4) {
    // ---------------- token rows (B operand) ----------------
    // GEMM1: x[a / k] for the block's assignments (zeros for padding rows);
    // GEMM2: the block's 16 intermediate rows, once the block is ready
    const int gt = tid - 64;  // 0 .. 63
    const int chunk = gt & 7;
    const int nk = p.T * p.k;
    uint32_t it = 0;
    bool alive = !*abort_flag;
    for (int u = blockIdx.x; alive && u < sc.nu; u += G) {
      const DUnit U = decode_unit(sc, sm, u);
      const __nv_bfloat16* src[2];
      uint32_t nbytes[2];
      // lane 0 of each gather warp waits (and acquires) for the block's rows;
      // the two warps take no barrier together, so one of them giving up
      // cannot strand the other
      if (U.kind == 1) {
        int ok = 1;
        if (lane == 0) ok = wait_at_least(p.ready + U.b, sc.nt1, abort_flag, p.err) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = (gt >> 3) + 8 * i;
        if (U.kind == 0) {
          const int a = row_asg(sm, U.b, r);
          const bool valid = a >= 0 && a < nk;
          src[i] = valid ? p.x + static_cast<size_t>(a / p.k) * p.H + chunk * 8 : p.x;
          nbytes[i] = valid ? 16u : 0u;
        } else {
          src[i] = p.inter + (static_cast<size_t>(U.b) * kDBM + r) * p.F + chunk * 8;
          nbytes[i] = 16u;
        }
      }
      for (int kb = U.kb0; kb < U.kb1; ++kb, ++it) {
        const int st = it % kDStages;
        const uint32_t ph = (it / kDStages) & 1u;
        if (!mbar_wait(&sm.empty[st], ph ^ 1u, abort_flag, p.err)) {
          alive = false;
          break;
        }
        const uint32_t tile = smem_u32(ring + st * kDStage) + kDBOff;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = (gt >> 3) + 8 * i;
          const uint32_t dst = tile + r * 128 + ((chunk ^ (r & 7)) << 4);
          cp_async_16(dst, nbytes[i] ? src[i] + kb * kDBK : src[i], nbytes[i]);
        }
        cp_async_mbar_arrive_noinc(&sm.full[st]);
      }
    }
    cp_async_wait_all();
  } else {
    // ---------------- epilogue ----------------
    const int ew = warp & 3;
    const int row = ew * 32 + lane;
    const int nk = p.T * p.k;
    uint32_t acc_it = 0;
    for (int u = blockIdx.x; u < sc.nu; u += G, ++acc_it) {
      const DUnit U = decode_unit(sc, sm, u);
      const int buf = acc_it & 1;
      const uint32_t aph = (acc_it >> 1) & 1u;
      const bool ok = mbar_wait(&sm.tfull[buf], aph, abort_flag, p.err);
      if (named_bar_any(1, 128, !ok || *abort_flag)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + buf * kDAcc;
      const int ncols = U.kind == 0 ? 2 * kDBM : kDBM;
      float* part = U.kind == 0 ? p.part1 : p.part2;
      int* tick = U.kind == 0 ? p.tick1 : p.tick2;
      const size_t slot_stride = static_cast<size_t>(128) * ncols;
      float g[16], v[16];
      bool finish = true;
      if (U.S == 1) {
        load_cols16(tb, g);
        if (U.kind == 0) load_cols16(tb + kDBM, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.tempty[buf]);
      } else {
        // split-K: publish this split's partial; the last split finishes
        float* mine = part + (static_cast<size_t>(U.ug) * U.S + U.s) * slot_stride +
                      static_cast<size_t>(row) * ncols;
        for (int c0 = 0; c0 < ncols; c0 += 16) {
          float t[16];
          load_cols16(tb + c0, t);
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            __stcg(reinterpret_cast<float4*>(mine + c0 + i),
                   make_float4(t[i], t[i + 1], t[i + 2], t[i + 3]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.tempty[buf]);
        named_bar_sync(1, 128);
        if (row == 0) {
          const int old = ticket_add_acq_rel(tick + U.ug, 1);
          const int last = (old == U.S - 1);
          if (last) store_relaxed_gpu(tick + U.ug, 0);
          sm.last_flag = last;
        }
        named_bar_sync(1, 128);
        finish = sm.last_flag != 0;
        if (finish) {
          const float* base0 = part + static_cast<size_t>(U.ug) * U.S * slot_stride +
                               static_cast<size_t>(row) * ncols;
          load_part16(base0, slot_stride, U.S, g);
          if (U.kind == 0) load_part16(base0 + kDBM, slot_stride, U.S, v);
        }
      }
      if (!finish) continue;
      if (U.kind == 0) {
        // SwiGLU rows of the intermediate (padding rows too: zeros), then
        // the block's readiness counter
        const int f = U.n * 128 + row;
        if (f < p.F) {
#pragma unroll
          for (int c = 0; c < kDBM; ++c)
            p.inter[(static_cast<size_t>(U.b) * kDBM + c) * p.F + f] =
                __float2bfloat16_rn(swiglu_f(g[c], v[c]));
        }
        named_bar_sync(1, 128);
        if (row == 0) {
          __threadfence();
          red_release_add(p.ready + U.b, 1);
        }
      } else {
        // weighted slot rows, then the combine of every token whose k slot
        // rows of this column tile are all written
        const int h = U.n * 128 + row;
#pragma unroll
        for (int c = 0; c < kDBM; ++c) {
          const int a = row_asg(sm, U.b, c);
          if (a >= 0 && a < nk && h < p.H) {
            const float w = __ldcg(p.r.wts + a);
            p.stage[static_cast<size_t>(a) * p.H + h] = __float2bfloat16_rn(g[c] * w);
          }
        }
        named_bar_sync(1, 128);
        if (row < kDBM) {
          const int a = row_asg(sm, U.b, row);
          int t = -1;
          if (a >= 0 && a < nk) {
            __threadfence();
            const int old = ticket_add_acq_rel(p.tokcnt + (a / p.k) * sc.nt2 + U.n, 1);
            if (old == p.k - 1) t = a / p.k;
          }
          sm.fin[row] = t;
        }
        named_bar_sync(1, 128);
        if (h < p.H) {
          for (int c = 0; c < kDBM; ++c) {
            const int t = sm.fin[c];
            if (t < 0) continue;
            const __nv_bfloat16* srow = p.stage + static_cast<size_t>(t) * p.k * p.H + h;
            float acc = 0.f;
            for (int j = 0; j < p.k; ++j)
              acc += __bfloat162float(__ldcg(srow + static_cast<size_t>(j) * p.H));
            p.out[static_cast<size_t>(t) * p.H + h] = __float2bfloat16_rn(acc);
          }
        }
        named_bar_sync(1, 128);  // sm.fin is rewritten by the next unit
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kDTmemCols);
  }
  // the last CTA to finish resets the header counters for the next launch
  // (every other CTA has finished all its reads and writes of them)
  if (tid == 0) {
    __threadfence();
    const int old = ticket_add_acq_rel(p.done, 1);
    sm.last_flag = (old == G - 1);
  }
  __syncthreads();
  if (sm.last_flag && tid == 0) {
    *p.routed = 0;
    *p.zeroed = 0;
    store_relaxed_gpu(p.done, 0);
  }
}

}  // namespace

DecodePlan plan_decode(int T, int H, int F, int E, int k, int num_sms) {
  DecodePlan d{};
  d.ok = T >= 1 && static_cast<long long>(T) * k <= kDMaxAsg && E >= 1 && E <= kDMaxE &&
         k <= 16 && k <= E && H % kDBK == 0 && F % kDBK == 0 && H >= kDBK && F >= kDBK &&
         num_sms >= 1;
  d.ne = (E + 7) / 8;
  d.nt = (T + 15) / 16;
  d.ks = 1;
  const int steps = H / 32;
  while (d.ks < 16 && d.ne * d.nt * (2 * d.ks) <= num_sms && steps % (2 * d.ks) == 0) d.ks *= 2;
  if (d.ne * d.nt * d.ks > num_sms) d.ok = false;  // every router item needs its own CTA
  const size_t nk = static_cast<size_t>(T) * k;
  size_t off = 0;
  d.logits = off;
  off += align_up(static_cast<size_t>(d.ks) * T * E * 4, 256);
  d.ids = off;
  off += align_up(nk * 4, 256);
  d.wts = off;
  off += align_up(nk * 4, 256);
  d.ready = off;
  off += align_up(nk * 4, 256);
  d.tokcnt = off;
  off += align_up(static_cast<size_t>(T) * ((H + 127) / 128) * 4, 256);
  d.tick1 = off;
  off += align_up(static_cast<size_t>(kDecodeMaxSlots) * 4, 256);
  d.tick2 = off;
  off += align_up(static_cast<size_t>(kDecodeMaxSlots) * 4, 256);
  d.part1 = off;
  off += static_cast<size_t>(kDecodeMaxSlots) * 128 * 2 * kDBM * 4;
  d.part2 = off;
  off += static_cast<size_t>(kDecodeMaxSlots) * 128 * kDBM * 4;
  d.inter = off;
  off += align_up(nk * kDBM * F * 2, 256);
  d.stage = off;
  off += align_up(nk * H * 2, 256);
  d.bytes = off;
  return d;
}

int launch_decode_layer(const void* hidden, const void* gate, const float* bias, const void* w13,
                        const void* w2, int T, int H, int F, int E, int k, int scoring,
                        int n_group, int topk_group, int renormalize, float scaling, void* out,
                        int32_t* topk_ids, float* topk_weights, char* region,
                        int* router_tickets, int* counters, int* err, const DecodePlan& d,
                        int num_sms, cudaStream_t stream) {
  CUtensorMap tm13, tm2;
  if (!make_map_bf16(&tm13, w13, static_cast<uint64_t>(E) * 2 * F, H, 128)) return -1;
  if (!make_map_bf16(&tm2, w2, static_cast<uint64_t>(E) * H, F, 128)) return -1;
  DecParams p{};
  RouterArgs& r = p.r;
  r.x = hidden;
  r.x_scale = nullptr;
  r.gate = gate;
  r.bias = bias;
  r.scratch = reinterpret_cast<float*>(region + d.logits);
  r.tickets = router_tickets;
  r.ids = topk_ids ? topk_ids : reinterpret_cast<int32_t*>(region + d.ids);
  r.wts = topk_weights ? topk_weights : reinterpret_cast<float*>(region + d.wts);
  r.err = err;
  r.cast_codes = nullptr;
  r.cast_scales = nullptr;
  r.align_hist = nullptr;
  r.align_seg = 0;
  r.T = T;
  r.H = H;
  r.E = E;
  r.k = k;
  r.scoring = scoring;
  r.n_group = n_group;
  r.topk_group = topk_group;
  r.renorm = renormalize;
  r.KS = d.ks;
  r.scaling = scaling;
  p.r_ne = d.ne;
  p.r_nt = d.nt;
  p.x = static_cast<const __nv_bfloat16*>(hidden);
  p.inter = reinterpret_cast<__nv_bfloat16*>(region + d.inter);
  p.stage = reinterpret_cast<__nv_bfloat16*>(region + d.stage);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.part1 = reinterpret_cast<float*>(region + d.part1);
  p.part2 = reinterpret_cast<float*>(region + d.part2);
  p.tick1 = reinterpret_cast<int*>(region + d.tick1);
  p.tick2 = reinterpret_cast<int*>(region + d.tick2);
  p.ready = reinterpret_cast<int*>(region + d.ready);
  p.tokcnt = reinterpret_cast<int*>(region + d.tokcnt);
  p.routed = counters;
  p.zeroed = counters + 1;
  p.done = counters + 2;
  p.nzero = static_cast<int>((d.part1 - d.ready) / 4);
  p.err = err;
  p.T = T;
  p.H = H;
  p.F = F;
  p.E = E;
  p.k = k;
  p.max_slots = kDecodeMaxSlots;
  static std::atomic<unsigned long long> smem_set{0};
  if (!ensure_smem_limit(reinterpret_cast<const void*>(decode_layer_kernel), kDSmemBytes,
                         smem_set))
    return -1;
  // the CTAs wait on one another: a cooperative launch guarantees that all
  // of them are resident at once (or fails to launch)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kDThreads);
  cfg.dynamicSmemBytes = kDSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_layer_kernel, tm13, tm2, p) != cudaSuccess) return -1;
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace moe
