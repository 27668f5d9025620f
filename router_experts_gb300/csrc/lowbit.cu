// lowbit.cu -- the expert GEMMs of the low-bit layer: FP8 e4m3 activations x
// FP4 e2m1 weights, each with one UE8M0 scale per 32 values along K.
//
// Follows "How GPUs Fuse Communication and Computation During LLM Inference"
// §1.1 (FP4 expert weights, FP8 token values, a scale per group of 32 values;
// the output of GEMM 1 is re-quantised before GEMM 2 reads it) and §3.5 (the
// GEMM 1 epilogue does SwiGLU and the re-quantisation: scale = the smallest
// power of two with amax / scale <= 448, codes = fp8(act / scale)); the tile
// scheme of "MoE Kernels, in depth" (expert from block_expert, rows from
// sorted_ids, gather folded into the load, weight in the down GEMM's
// epilogue).
//
// The products run on the block-scaled tensor-core MMA (tcgen05.mma
// kind::mxf8f6f4, A = e4m3, B = e2m1, one UE8M0 scale per 32 values of each
// operand row, fp32 accumulation in TMEM).  Nothing is converted on the SMs,
// and the one thread that issues the MMAs does little else per K step than
// wait on one barrier, issue four MMAs and one commit (every tcgen05
// instruction costs that thread tens of nanoseconds):
//   B = 256 weight rows, loaded by TMA straight from the packed e2m1 codes
//       with the 16 x 4-bit / 16-byte tensor-map type: each 16 codes land as
//       their 8 packed bytes plus an 8-byte gap, the MMA's 4-bit operand
//       layout (the copy counts the packed bytes in its transactions);
//   A = 128 token rows of e4m3 codes: GEMM1 gathers them by sorted_ids with
//       cp.async (the MMA thread fences the generic-proxy writes before the
//       tensor core reads them); GEMM2 reads its contiguous intermediate rows
//       with one 2-D TMA copy;
//   scale words (4 K-blocks of one row) are written to TMEM by four warps,
//       one per TMEM lane quarter, with tcgen05.st: row m of A at lane m,
//       column base + m/32; row n of B at lane n mod 32 of every quarter,
//       column base + 4 + n/32; byte j scales K-block j of the step.  The
//       words are staged in groups of 4 steps (one 16-byte copy per row and
//       operand) a few groups ahead.
// Tile: M = 128 token rows of one block (BLOCK_M rows valid), N = 256 weight
// rows (GEMM1: 128 gate rows + the matching 128 up rows), K steps of 128
// (four K = 32 MMAs).  One ring of K steps (token tile + weight tile + a
// 16-column TMEM scale slot) with one full and one empty barrier per step.
// The 256-column accumulator and the scale slots fill the 512 TMEM columns
// but for one accumulator, so the next tile's MMAs start once the epilogue
// has read the accumulator (its loads run ahead meanwhile); against 128-row
// weight tiles with two accumulators, each token tile feeds twice the MMA
// work and the MMA thread issues half the instructions per FLOP, which is
// what bounded the step (operand latency over the ring's depth, and about
// 40 ns per MMA instruction).
// 14 warps:
//   warp 0      TMA of the weight tiles
//   warp 1      TMEM allocation and the single thread issuing the MMAs
//   warps 2-5   token tiles (GEMM1 cp.async gather; GEMM2 one TMA copy)
//   warps 6-9   scale words -> TMEM (lane quarter = warp % 4)
//   warps 10-13 epilogue (lane quarter = warp % 4)
#include <cuda_fp8.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kMxThreads = 448;
constexpr int kMxBK = 128;                  // K values per stage (4 MMAs of K = 32)
constexpr int kMxNT = 256;                  // weight rows per tile (MMA N)
constexpr int kMxStages = 4;                // ring of K steps
constexpr int kMxSfSlots = 3;               // scale staging slots, 4 K steps each
constexpr int kMxATile = 128 * kMxBK;       // 16 KB token tile (one byte per code)
constexpr int kMxBTile = kMxNT * kMxBK;     // 32 KB weight tile (one byte per 4-bit code in smem)
constexpr int kMxStageBytes = kMxATile + kMxBTile;
// scale staging: [kMxSfSlots][token rows 0..127 | weight rows 0..255][4 steps x 4 bytes]
constexpr int kMxSfSlotBytes = (128 + kMxNT) * 16;
constexpr int kMxSfStageBytes = kMxSfSlots * kMxSfSlotBytes;
constexpr int kMxBarBytes = 256;
constexpr int kMxSmem = kMxStages * kMxStageBytes + kMxSfStageBytes + kMxBarBytes + 1024;
static_assert(kMxSmem <= 232448, "shared memory budget");
static_assert(kMxStageBytes % 1024 == 0, "stage tiles must keep 1024-byte alignment");
constexpr uint32_t kMxAccCols = kMxNT;      // one accumulator
constexpr uint32_t kMxSfCol0 = kMxAccCols;  // scale slots after it
constexpr uint32_t kMxSfCols = 16;          // per ring stage: A at +0..3, B at +4..11
constexpr uint32_t kMxTmemCols = 512;
static_assert(kMxSfCol0 + kMxSfCols * kMxStages <= kMxTmemCols, "TMEM columns");
static_assert(2 * (kMxStages + 1) * 8 + 8 <= kMxBarBytes, "barrier space");

// Instruction descriptor of the block-scaled MMA: e4m3 A, e2m1 B (both
// K-major), UE8M0 scales, fp32 D; sf_id picks the scale byte of the 32-bit
// TMEM word for both operands.
__host__ __device__ constexpr uint32_t idesc_mxf8f4(int M, int N, int sf_id) {
  return (static_cast<uint32_t>(sf_id) << 4) | (5u << 10) |
         (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(M >> 4) << 24) | (static_cast<uint32_t>(sf_id) << 29);
}

// D[tmem] (+)= (A * sa)[smem] * (B * sb)[smem]^T with per-32 UE8M0 scales in TMEM.
MOE_DEV void umma_mxf8f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Warp-wide TMEM stores (lane i of the warp -> TMEM lane (address lane field + i)).
MOE_DEV void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
MOE_DEV void tmem_st4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(v0), "r"(v1), "r"(v2), "r"(v3)
               : "memory");
}
MOE_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
MOE_DEV uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// e4m3 codes of 32 activations with their UE8M0 exponent byte: scale = the
// smallest power of two 2^s with amax <= 448 * 2^s (2^0 when all are zero).
MOE_DEV uint32_t requant32(const float (&v)[32], uint32_t (&codes)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  int s = 0;
  if (amax > 0.f) {
    // ceil(log2(amax / 448)) from the bits of the fp32 quotient
    const float q = amax / 448.0f;
    const uint32_t bits = __float_as_uint(q);
    s = static_cast<int>((bits >> 23) & 0xFFu) - 127 + ((bits & 0x7FFFFFu) ? 1 : 0);
    s = max(-127, min(127, s));
  }
  const float inv = exp2f(static_cast<float>(-s));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i] * inv, v[4 * i + 1] * inv), __NV_SATFINITE,
                                 __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i + 2] * inv, v[4 * i + 3] * inv),
                                 __NV_SATFINITE, __NV_E4M3);
    codes[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return static_cast<uint32_t>(s + 127);
}

struct MxUnit {
  int b, n, e;
};

// Weight row r (0..255) of the tile of unit u: GEMM1 gate rows n*128 + r for
// r < 128 and the matching up rows for r >= 128 (F % 128 == 0); GEMM2 rows
// n*256 + r, held inside the expert's H rows: when H % 256 == 128 the last
// tile's second half repeats rows of the expert, whose columns no epilogue
// stores.
template <int KIND>
MOE_DEV int mx_wrow(const LowbitParams& p, const MxUnit& u, int r) {
  if constexpr (KIND == 0) {
    const int f = u.n * (kMxNT / 2) + (r & 127);
    return u.e * 2 * p.F + ((r < 128) ? 0 : p.F) + f;
  } else {
    return u.e * p.H + min(u.n * kMxNT + r, p.H - 1);
  }
}
// First weight row of the 128-row box h (0, 1) of unit u's tile.
template <int KIND>
MOE_DEV int mx_wbox(const LowbitParams& p, const MxUnit& u, int h) {
  if constexpr (KIND == 0) return u.e * 2 * p.F + h * p.F + u.n * (kMxNT / 2);
  else return u.e * p.H + min(u.n * kMxNT + 128 * h, p.H - 128);
}

// GATHER: GEMM1's token rows are gathered from x by sorted_ids (cp.async);
// otherwise the A rows are already in the block's padded order (GEMM2's
// intermediate, or GEMM1's rows permuted by permute_rows_kernel) and one 2-D
// TMA copy per step loads them.
template <int KIND, bool GATHER>
__global__ void __launch_bounds__(kMxThreads, 1)
    lowbit_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_a, const LowbitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // ring stage s: token tile at s * kMxStageBytes, weight tile kMxATile after it
  uint32_t* sfstage = reinterpret_cast<uint32_t*>(smem + kMxStages * kMxStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kMxStages * kMxStageBytes + kMxSfStageBytes);
  uint64_t* empty = full + kMxStages;
  uint64_t* tfull = empty + kMxStages;
  uint64_t* tempty = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = (KIND == 0) ? p.H : p.F;
  const int KS = K / kMxBK;
  const int nblk = padded_rows(p, p.BM) / p.BM;
  const int ntiles = (KIND == 0) ? p.F / (kMxNT / 2) : (p.H + kMxNT - 1) / kMxNT;
  const int num_units = nblk * ntiles;
  const int bmr = min(p.BM, 128);  // token rows of a tile that hold data

  if (threadIdx.x == 0) {
    for (int i = 0; i < kMxStages; ++i) {
      // weight TMA expect-tx arrival + tokens (GEMM1: 128 cp.async arrivals,
      // GEMM2: one TMA expect-tx arrival) + the four scale warps
      mbar_init(&full[i], 1 + (GATHER ? 128 : 1) + 4);
      mbar_init(&empty[i], 1);  // MMA commit
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 4);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kMxTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto decode = [&](int uu) {
    MxUnit u;
    u.b = uu / ntiles;
    u.n = uu % ntiles;
    int e = __ldg(p.block_expert + u.b);
    if (e < 0 || e >= p.E) {
      if (threadIdx.x == 0) raise_error(p.err, kErrBadTable);
      e = min(max(e, 0), p.E - 1);
    }
    u.e = e;
    return u;
  };
  // token row of tile row r (GEMM1), or -1 for a padding row
  auto token_of = [&](const MxUnit& u, int r) -> int {
    if (r >= p.BM) return -1;
    const int a = row_assignment(p, u.b, p.BM, r);
    return (a >= 0 && a < p.T * p.k) ? a / p.k : -1;
  };

  if (warp == 0) {
    // ---------------- weight tiles (TMA) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      uint32_t it = 0;
      bool alive = true;
      for (int uu = blockIdx.x; alive && uu < num_units; uu += gridDim.x) {
        const MxUnit u = decode(uu);
        const int r0 = mx_wbox<KIND>(p, u, 0), r1 = mx_wbox<KIND>(p, u, 1);
        for (int ks = 0; ks < KS; ++ks, ++it) {
          const int s = it % kMxStages;
          if (!mbar_wait(&empty[s], ((it / kMxStages) & 1u) ^ 1u, abort_flag, p.err)) {
            alive = false;
            break;
          }
          uint8_t* dst = smem + s * kMxStageBytes + kMxATile;
          // two 128-row boxes of 128 codes: 2 x 128 x 64 packed bytes
          mbar_arrive_expect_tx(&full[s], kMxNT * kMxBK / 2);
          tma_load_2d(dst, &tm_w, &full[s], ks * kMxBK, r0);
          tma_load_2d(dst + 128 * 128, &tm_w, &full[s], ks * kMxBK, r1);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, acc_it = 0;
      bool alive = true;
      for (int uu = blockIdx.x; alive && uu < num_units; uu += gridDim.x, ++acc_it) {
        if (!mbar_wait(tempty, (acc_it & 1u) ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base;
        for (int ks = 0; ks < KS; ++ks, ++it) {
          const int s = it % kMxStages;
          if (!mbar_wait(&full[s], (it / kMxStages) & 1u, abort_flag, p.err)) {
            alive = false;
            break;
          }
          if constexpr (GATHER) fence_proxy_async_smem();  // cp.async rows -> tensor core
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + s * kMxStageBytes);
          const uint32_t b_addr = a_addr + kMxATile;
          const uint32_t sf_t = tmem_base + kMxSfCol0 + kMxSfCols * s;
#pragma unroll
          for (int kk = 0; kk < kMxBK / 32; ++kk)
            umma_mxf8f4(d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32),
                        idesc_mxf8f4(128, kMxNT, kk), sf_t, sf_t + 4,
                        (ks > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        if (!alive) break;
        umma_commit(tfull);
      }
    }
  } else if (warp < 6) {
    // ---------------- token tiles ----------------
    if constexpr (GATHER) {
      // cp.async gather: thread gt copies 16-byte chunk gt % 8 of tile rows
      // gt/8 + 16i; its arrival counts when its copies have landed (the MMA
      // thread fences before the tensor core reads them)
      const int gt = threadIdx.x - 64;  // 0..127
      const int chunk = gt & 7;
      uint32_t it = 0;
      bool alive = true;
      for (int uu = blockIdx.x; alive && uu < num_units; uu += gridDim.x) {
        const MxUnit u = decode(uu);
        const uint8_t* src[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int tr = token_of(u, (gt >> 3) + 16 * i);
          src[i] = tr >= 0 ? p.act + static_cast<size_t>(tr) * K + chunk * 16 : nullptr;
        }
        for (int ks = 0; ks < KS; ++ks, ++it) {
          const int s = it % kMxStages;
          if (!mbar_wait(&empty[s], ((it / kMxStages) & 1u) ^ 1u, abort_flag, p.err)) {
            alive = false;
            break;
          }
          const uint32_t tile = smem_u32(smem + s * kMxStageBytes);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = (gt >> 3) + 16 * i;
            cp_async_16(tile + r * 128 + ((chunk ^ (r & 7)) << 4),
                        src[i] ? static_cast<const void*>(src[i] + ks * kMxBK) : p.act,
                        src[i] ? 16u : 0u);
          }
          cp_async_mbar_arrive_noinc(&full[s]);
        }
      }
      cp_async_wait_all();
    } else if (warp == 2 && lane == 0) {
      // the block's rows are contiguous: one 2-D box of bmr rows per step
      tma_prefetch_desc(&tm_a);
      uint32_t it = 0;
      bool alive = true;
      for (int uu = blockIdx.x; alive && uu < num_units; uu += gridDim.x) {
        const MxUnit u = decode(uu);
        for (int ks = 0; ks < KS; ++ks, ++it) {
          const int s = it % kMxStages;
          if (!mbar_wait(&empty[s], ((it / kMxStages) & 1u) ^ 1u, abort_flag, p.err)) {
            alive = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(bmr) * kMxBK);
          tma_load_2d(smem + s * kMxStageBytes, &tm_a, &full[s], ks * kMxBK, u.b * p.BM);
        }
      }
    }
  } else if (warp < 10) {
    // ---------------- scale words -> TMEM ----------------
    // The four warps (lane quarter q = warp % 4) stage the scale words of
    // groups of 4 K steps in a ring of kMxSfSlots slots; thread (q, l) copies
    // those of token row 32q + l and of weight rows 32q + l and 128 + 32q + l
    // (16 bytes = 4 steps when a scale row is a multiple of 16 bytes, else
    // one word per step), kMxSfSlots - 1 groups ahead.  After a named barrier
    // of the four warps every thread reads the word of its token row and the
    // words of weight rows 32c + l (c = 0..7), and stores them into the
    // step's TMEM slot once the MMAs that last read that slot are done.
    const int q = warp & 3;
    const int r = 32 * q + lane;  // staged row of this thread
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t stage_base = smem_u32(sfstage);  // [slot][A 128 | B 256 rows][16 bytes]
    const int my_units = num_units > static_cast<int>(blockIdx.x)
                             ? (num_units - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x
                             : 0;
    const int gpu = (KS + 3) / 4;  // groups per unit
    const int n_g = my_units * gpu;
    // 16-byte copies need 16-byte aligned scale rows (row length and base)
    const bool wide = (K / 32) % 16 == 0 &&
                      (reinterpret_cast<uintptr_t>(p.act_scale) & 15u) == 0 &&
                      (reinterpret_cast<uintptr_t>(p.w_scale) & 15u) == 0;
    int pf_unit = -1;
    const uint8_t* pa = nullptr;
    const uint8_t* pb = nullptr;
    const uint8_t* pb2 = nullptr;
    auto issue = [&](int g) {
      const int un = g / gpu, gi = g % gpu;
      if (un != pf_unit) {
        pf_unit = un;
        const MxUnit u = decode(static_cast<int>(blockIdx.x) + un * static_cast<int>(gridDim.x));
        pa = nullptr;
        if constexpr (GATHER) {
          const int t = token_of(u, r);
          if (t >= 0) pa = p.act_scale + static_cast<size_t>(t) * (K / 32);
        } else {
          if (r < p.BM) pa = p.act_scale + (static_cast<size_t>(u.b) * p.BM + r) * (K / 32);
        }
        pb = p.w_scale + static_cast<size_t>(mx_wrow<KIND>(p, u, r)) * (K / 32);
        pb2 = p.w_scale + static_cast<size_t>(mx_wrow<KIND>(p, u, r + 128)) * (K / 32);
      }
      const uint32_t dst = stage_base + (g % kMxSfSlots) * kMxSfSlotBytes + r * 16;
      const uint32_t dstb = stage_base + (g % kMxSfSlots) * kMxSfSlotBytes + 2048 + r * 16;
      if (wide) {
        cp_async_16(dst, pa ? static_cast<const void*>(pa + 16 * gi) : p.act_scale, pa ? 16u : 0u);
        cp_async_16(dstb, pb + 16 * gi, 16u);
        cp_async_16(dstb + 2048, pb2 + 16 * gi, 16u);
      } else {
        const int nw = min(4, KS - 4 * gi);
        for (int w = 0; w < nw; ++w) {
          cp_async_4(dst + 4 * w, pa ? static_cast<const void*>(pa + 16 * gi + 4 * w) : p.act_scale,
                     pa ? 4u : 0u);
          cp_async_4(dstb + 4 * w, pb + 16 * gi + 4 * w, 4u);
          cp_async_4(dstb + 2048 + 4 * w, pb2 + 16 * gi + 4 * w, 4u);
        }
      }
    };
    for (int g = 0; g < kMxSfSlots - 1; ++g) {
      if (g < n_g) issue(g);
      cp_async_commit();
    }
    bool alive = true;
    for (int g = 0; alive && g < n_g; ++g) {
      cp_async_wait<kMxSfSlots - 2>();  // this thread's copies of group g have landed
      // every thread's copies of group g have landed, and every thread has
      // read group g - 1, whose slot the next copies reuse
      named_bar_sync(2, 128);
      if (g + kMxSfSlots - 1 < n_g) issue(g + kMxSfSlots - 1);
      cp_async_commit();  // one group per iteration (empty past the end)
      const uint32_t slot = stage_base + (g % kMxSfSlots) * kMxSfSlotBytes;
      const int gi = g % gpu;
      const int j0 = (g / gpu) * KS + 4 * gi;
      const int nst = min(4, KS - 4 * gi);
      for (int t = 0; t < nst; ++t) {
        const uint32_t wa = ld_shared_u32(slot + r * 16 + 4 * t);
        uint32_t wb[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) wb[c] = ld_shared_u32(slot + 2048 + (32 * c + lane) * 16 + 4 * t);
        const int j = j0 + t;
        const int s = j % kMxStages;
        // the slot's previous scales were read by the MMAs of step j - kMxStages
        const bool ok = mbar_wait(&empty[s], ((j / kMxStages) & 1u) ^ 1u, abort_flag, p.err);
        if (__any_sync(0xffffffffu, !ok)) {
          alive = false;
          break;
        }
        const uint32_t col = kMxSfCol0 + kMxSfCols * s;
        tmem_st1(lane_base + col + q, wa);
        tmem_st4(lane_base + col + 4, wb[0], wb[1], wb[2], wb[3]);
        tmem_st4(lane_base + col + 8, wb[4], wb[5], wb[6], wb[7]);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
      }
      // the four warps stop together (they meet at the named barrier)
      if (named_bar_any(3, 128, !alive)) alive = false;
    }
    cp_async_wait_all();
  } else {
    // ---------------- epilogue ----------------
    const int ew = warp & 3;
    const int row = ew * 32 + lane;
    uint32_t acc_it = 0;
    // the accumulator is handed back to the MMA thread as soon as the last
    // columns are in registers
    auto release = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
    };
    for (int uu = blockIdx.x; uu < num_units; uu += gridDim.x, ++acc_it) {
      const MxUnit u = decode(uu);
      const bool ok = mbar_wait(tfull, acc_it & 1u, abort_flag, p.err);
      if (named_bar_any(1, 128, !ok || *abort_flag)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(ew * 32) << 16);
      const bool rvalid = row < p.BM;
      const size_t prow = static_cast<size_t>(u.b) * p.BM + row;
      if constexpr (KIND == 0) {
        // a padding row is written as zero codes with scale 2^0 (its token
        // tile row may hold anything when the rows come permuted)
        int a0 = p.T * p.k;
        if (rvalid) a0 = row_assignment(p, u.b, p.BM, row);
        const bool pad = a0 < 0 || a0 >= p.T * p.k;
        // SwiGLU of gate column c and up column 128 + c, re-quantised per 32
        constexpr int NJ = kMxNT / 64;
#pragma unroll 1
        for (int j = 0; j < NJ; ++j) {
          uint32_t g0[16], g1[16], u0[16], u1[16];
          tmem_ld16(tb + 32 * j, g0);
          tmem_ld16(tb + 32 * j + 16, g1);
          tmem_ld16(tb + kMxNT / 2 + 32 * j, u0);
          tmem_ld16(tb + kMxNT / 2 + 32 * j + 16, u1);
          tmem_ld_wait();
          reg_fence16(g0);
          reg_fence16(g1);
          reg_fence16(u0);
          reg_fence16(u1);
          if (j == NJ - 1) release();
          float act[32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            act[i] = swiglu_f(__uint_as_float(g0[i]), __uint_as_float(u0[i]));
            act[16 + i] = swiglu_f(__uint_as_float(g1[i]), __uint_as_float(u1[i]));
          }
          uint32_t codes[8];
          uint32_t sbyte = requant32(act, codes);
          if (pad) {
#pragma unroll
            for (int i = 0; i < 8; ++i) codes[i] = 0u;
            sbyte = 127u;
          }
          const int f = u.n * (kMxNT / 2) + 32 * j;
          if (rvalid && f + 32 <= p.F) {
            st_global_v8(p.inter_q + prow * p.F + f, codes);
            p.inter_scale[prow * (p.F / 32) + f / 32] = static_cast<uint8_t>(sbyte);
          }
        }
      } else {
        int a = p.T * p.k;
        if (rvalid) a = row_assignment(p, u.b, p.BM, row);
        const bool valid = rvalid && a >= 0 && a < p.T * p.k;
        const float w = valid ? __ldg(p.topk_weights + a) : 0.f;
        // 16-column chunks, the TMEM load of chunk c + 1 in flight while
        // chunk c is scaled and stored
        constexpr int NCH = kMxNT / 16;
        uint32_t r[2][16];
        tmem_ld16(tb, r[0]);
        tmem_ld_wait();
        reg_fence16(r[0]);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const int cur = c & 1, nxt = cur ^ 1;
          if (c + 1 < NCH) tmem_ld16(tb + 16 * (c + 1), r[nxt]);
          const int h = u.n * kMxNT + 16 * c;
          if (valid && h + 16 <= p.H) {
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              o[i] = pack_bf16x2(__uint_as_float(r[cur][2 * i]) * w,
                                 __uint_as_float(r[cur][2 * i + 1]) * w);
            st_global_v8(p.stage + static_cast<size_t>(a) * p.H + h, o);
          }
          if (c + 1 < NCH) {
            tmem_ld_wait();
            reg_fence16(r[nxt]);
            if (c + 1 == NCH - 1) release();
          }
        }
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kMxTmemCols);
  }
}

// GEMM1's token rows in the blocks' padded order: position q below the
// padded length holds row a / k of x (codes and scale bytes) for its
// assignment a = sorted_ids[q], so GEMM1 loads its A tiles with one 2-D TMA
// copy per step as GEMM2 does.  Padding positions are not written: their
// products reach only padding rows of the accumulators, for which the
// epilogue writes zeros.  One warp per position: H bytes of codes in 16-byte pieces, H/32
// scale bytes in 4-byte words (H % 128 == 0).
__global__ void __launch_bounds__(256) permute_rows_kernel(const LowbitParams p, uint8_t* xq,
                                                           uint8_t* xs) {
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * 8;
  const int npp = padded_rows(p, p.BM);
  const int nk = p.T * p.k;
  const int H16 = p.H / 16, H128 = p.H / 128;
  for (long long q = blockIdx.x * 8ll + (threadIdx.x >> 5); q < npp; q += warps) {
    const int a = row_assignment(p, static_cast<int>(q / p.BM), p.BM, static_cast<int>(q % p.BM));
    if (a < 0 || a >= nk) continue;
    const uint4* src = reinterpret_cast<const uint4*>(p.act + static_cast<size_t>(a / p.k) * p.H);
    uint4* dst = reinterpret_cast<uint4*>(xq + static_cast<size_t>(q) * p.H);
    // eight 16-byte loads in flight per lane before the stores
    for (int i0 = lane; i0 < H16; i0 += 32 * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + 32 * u < H16) v[u] = __ldg(src + i0 + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + 32 * u < H16) dst[i0 + 32 * u] = v[u];
    }
    const uint32_t* ss =
        reinterpret_cast<const uint32_t*>(p.act_scale + static_cast<size_t>(a / p.k) * (p.H / 32));
    uint32_t* sd = reinterpret_cast<uint32_t*>(xs + static_cast<size_t>(q) * (p.H / 32));
    for (int i = lane; i < H128; i += 32) sd[i] = __ldg(ss + i);
  }
}

// FP8 cast of the layer input ("How GPUs Fuse ..." §1.1: a small kernel turns
// the layer input into FP8 codes and writes the scales; the scale rule of
// §3.5): bf16 x [T, H] -> e4m3 codes [T, H] and one UE8M0 byte per 32 values
// (cast_e4m3_group32).  One thread per group of 32: 64 bytes in, 33 out.
__global__ void __launch_bounds__(256) cast_e4m3_kernel(const uint4* __restrict__ x,
                                                        long long groups, uint4* __restrict__ codes,
                                                        uint8_t* __restrict__ scales) {
  for (long long g = blockIdx.x * 256ll + threadIdx.x; g < groups;
       g += static_cast<long long>(gridDim.x) * 256)
    cast_e4m3_group32(x + 4 * g, codes + 2 * g, scales + g);
}

}  // namespace

int launch_cast_e4m3(const void* x, int T, int H, uint8_t* codes, uint8_t* scales,
                     cudaStream_t stream) {
  const long long groups = static_cast<long long>(T) * (H / 32);
  if (groups == 0) return 0;
  const long long want = (groups + 255) / 256;
  const int blocks = static_cast<int>(want < 152 * 16 ? want : 152 * 16);
  cast_e4m3_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4*>(x), groups,
                                               reinterpret_cast<uint4*>(codes), scales);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_lowbit_gemm(int kind, const LowbitParams& p, int num_sms, cudaStream_t stream,
                       uint8_t* xperm, uint8_t* xperm_scale) {
  static std::atomic<unsigned long long> smem_set0{0}, smem_set0p{0}, smem_set1{0};
  if (!ensure_smem_limit(reinterpret_cast<const void*>(lowbit_gemm_kernel<0, true>), kMxSmem,
                         smem_set0) ||
      !ensure_smem_limit(reinterpret_cast<const void*>(lowbit_gemm_kernel<0, false>), kMxSmem,
                         smem_set0p) ||
      !ensure_smem_limit(reinterpret_cast<const void*>(lowbit_gemm_kernel<1, false>), kMxSmem,
                         smem_set1))
    return -1;
  // packed weight codes [E*2F or E*H rows, K codes], box 128 codes x 128 rows
  const int K = (kind == 0) ? p.H : p.F;
  const uint64_t rows = (kind == 0) ? static_cast<uint64_t>(p.E) * 2 * p.F
                                    : static_cast<uint64_t>(p.E) * p.H;
  CUtensorMap tm_w, tm_a;
  if (!make_map_e2m1(&tm_w, p.w, rows, static_cast<uint64_t>(K), 128)) return -1;
  // token rows by TMA: one box = the data rows of a block
  const uint32_t bmr = static_cast<uint32_t>(p.BM < 128 ? p.BM : 128);
  if (kind == 0 && xperm == nullptr) {
    tm_a = tm_w;  // unused: GEMM1 gathers its token rows with cp.async
    lowbit_gemm_kernel<0, true><<<num_sms, kMxThreads, kMxSmem, stream>>>(tm_w, tm_a, p);
  } else if (kind == 0) {
    // GEMM1's rows permuted into the padded order first, then read like
    // GEMM2 reads the intermediate
    // one warp per position of the capacity (eight per block), so every row
    // copy is in flight at once
    const long long pblocks = (static_cast<long long>(p.cap_rows) + 7) / 8;
    permute_rows_kernel<<<static_cast<unsigned>(pblocks > 0 ? pblocks : 1), 256, 0, stream>>>(
        p, xperm, xperm_scale);
    if (cudaGetLastError() != cudaSuccess) return -1;
    if (!make_map_u8_sw128(&tm_a, xperm, static_cast<uint64_t>(p.cap_rows),
                           static_cast<uint64_t>(p.H), bmr))
      return -1;
    LowbitParams q = p;
    q.act = xperm;
    q.act_scale = xperm_scale;
    lowbit_gemm_kernel<0, false><<<num_sms, kMxThreads, kMxSmem, stream>>>(tm_w, tm_a, q);
  } else {
    // intermediate codes [cap_rows, F]
    if (!make_map_u8_sw128(&tm_a, p.act, static_cast<uint64_t>(p.cap_rows),
                           static_cast<uint64_t>(p.F), bmr))
      return -1;
    lowbit_gemm_kernel<1, false><<<num_sms, kMxThreads, kMxSmem, stream>>>(tm_w, tm_a, p);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace moe
