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
// The products run on the block-scaled tensor-core MMA
// (tcgen05.mma kind::mxf8f6f4 with one UE8M0 scale per 32 values of each
// operand row, fp32 accumulation in TMEM), so the scales are applied by the
// tensor core and the operands stay one byte wide in shared memory:
//   A = 128 token rows of e4m3 codes, gathered as they are (no conversion);
//   B = 128 weight rows, e2m1 codes widened to e4m3 (exact: every e2m1 value
//       is an e4m3 value) by converter warps;
//   scale factors are written to TMEM with tcgen05.st: for row m of A, lane m
//   and column base + m/32; for row n of B, lane n mod 32 (in every lane
//   quarter) and column base + n/32; byte j of the word scales the j-th
//   32-value block of a 128-value K step.
// Tile: M = 128 token rows of one block (BLOCK_M rows valid), N = 128 weight
// rows (GEMM1: 64 gate rows + the matching 64 up rows), K steps of 128 (four
// K=32 MMAs).  Two 128-column accumulators, double-buffered.
// 16 warps:
//   warp 0      TMA of the packed weight codes (ring of 6 raw stages, L2
//               warmed one ring ahead) and,
//               one row per lane, cp.async of their scale words
//   warp 1      TMEM allocation and the single thread issuing the MMAs
//   warps 2-3   cp.async gather of the token codes and scale words straight
//               into the token-tile ring (6 deep: it covers the gather latency)
//   warps 4-11  widen the weight codes into the weight-tile ring (4 deep); warps 4-7
//               write the token scale factors to TMEM, warps 8-11 the weight
//               scale factors
//   warps 12-15 epilogue (TMEM lane quarter = warp % 4)
#include <cuda_fp8.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kMxThreads = 512;
constexpr int kMxBK = 128;                  // K values per stage (4 MMAs of K = 32)
constexpr int kMxNT = 128;                  // weight rows per tile (MMA N)
// Token tiles wait on gather latency, so their ring is deep; the widened
// weight tiles are written just ahead of their MMAs, so theirs is short.
constexpr int kMxAStages = 6;               // token-code tiles
constexpr int kMxBStages = 4;               // widened weight tiles (and scale-factor slots)
constexpr int kMxRawStages = 6;             // packed weight-code stages (streamed from HBM)
constexpr int kMxA = 128 * kMxBK;           // 16 KB of token codes
constexpr int kMxB = kMxNT * kMxBK;         // 16 KB of widened weight codes
constexpr int kMxRawW = kMxNT * (kMxBK / 2);  // 8 KB of packed weight codes
constexpr int kMxABytes = kMxAStages * kMxA;
constexpr int kMxBBytes = kMxBStages * kMxB;
constexpr int kMxRawBytes = kMxRawStages * kMxRawW;
constexpr int kMxSfaBytes = kMxAStages * 128 * 4;      // token scale words per token tile
constexpr int kMxSfbBytes = kMxRawStages * kMxNT * 4;  // weight scale words per raw stage
constexpr int kMxBarBytes = 512;
constexpr int kMxSmem =
    kMxABytes + kMxBBytes + kMxRawBytes + kMxSfaBytes + kMxSfbBytes + kMxBarBytes + 1024;
static_assert(kMxSmem <= 232448, "shared memory budget");
constexpr uint32_t kMxAccCols = 128;        // per accumulator buffer
constexpr uint32_t kMxSfCol0 = 256;         // scale-factor columns: 8 per weight-tile slot
constexpr uint32_t kMxTmemCols = 512;

// Instruction descriptor of the block-scaled MMA: e4m3 A and B (K-major),
// UE8M0 scales, fp32 D; sf_id picks the scale byte of the 32-bit TMEM word.
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, int sf_id) {
  return (static_cast<uint32_t>(sf_id) << 4) | (static_cast<uint32_t>(N >> 3) << 17) |
         (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) | (static_cast<uint32_t>(sf_id) << 29);
}

// D[tmem] (+)= (A * sa)[smem] * (B * sb)[smem]^T with per-32 UE8M0 scales in TMEM.
MOE_DEV void umma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
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

// 4 bytes = 8 e2m1 codes (low nibble first) -> 8 e4m3 codes (two words, in
// order): hardware e2m1x2 -> f16x2 and f16x2 -> e4m3x2 conversions, both
// exact on these values.
MOE_DEV uint2 e2m1x8_to_e4m3x8(uint32_t w) {
  uint32_t h[4];
  asm("{\n"
      " .reg .b8 q0, q1, q2, q3;\n"
      " mov.b32 {q0, q1, q2, q3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, q0;\n"
      " cvt.rn.f16x2.e2m1x2 %1, q1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, q2;\n"
      " cvt.rn.f16x2.e2m1x2 %3, q3;\n"
      "}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint16_t b;
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(b) : "r"(h[i]));
    o[i] = b;
  }
  return make_uint2(o[0] | (o[1] << 16), o[2] | (o[3] << 16));
}

MOE_DEV void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
MOE_DEV uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
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

// Weight row r (0..127) of the tile of unit u: GEMM1 gate rows n*64 + r for
// r < 64 and the matching up rows for r >= 64; GEMM2 rows n*128 + r.
template <int KIND>
MOE_DEV int mx_wrow(const LowbitParams& p, const MxUnit& u, int r) {
  if constexpr (KIND == 0) {
    const int f = u.n * (kMxNT / 2) + (r & 63);
    return u.e * 2 * p.F + ((r < 64) ? 0 : p.F) + f;
  } else {
    return u.e * p.H + u.n * kMxNT + r;
  }
}

template <int KIND>
__global__ void __launch_bounds__(kMxThreads, 1)
    lowbit_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const LowbitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* atile = smem;                  // [kMxAStages][128 token rows x 128 codes]
  uint8_t* btile = atile + kMxABytes;     // [kMxBStages][128 weight rows x 128 codes]
  uint8_t* raw = btile + kMxBBytes;       // [kMxRawStages][128 rows x 64 bytes]
  uint32_t* sfa = reinterpret_cast<uint32_t*>(raw + kMxRawBytes);  // [kMxAStages][128]
  uint32_t* sfb = sfa + kMxAStages * 128;                          // [kMxRawStages][128]
  uint64_t* wfull = reinterpret_cast<uint64_t*>(sfb + kMxRawStages * kMxNT);
  uint64_t* wempty = wfull + kMxRawStages;
  uint64_t* afull = wempty + kMxRawStages;
  uint64_t* aempty = afull + kMxAStages;
  uint64_t* ready = aempty + kMxAStages;
  uint64_t* bempty = ready + kMxBStages;
  uint64_t* tfull = bempty + kMxBStages;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = (KIND == 0) ? p.H : p.F;
  const int KS = K / kMxBK;
  int npp = __ldg(p.num_post_padded);
  npp = max(0, min(npp, p.cap_rows));
  const int nblk = npp / p.BM;
  const int ntiles = (KIND == 0) ? p.F / (kMxNT / 2) : p.H / kMxNT;
  const int num_units = nblk * ntiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kMxRawStages; ++i) {
      mbar_init(&wfull[i], 1 + 32);  // TMA bytes + the scale-word copies of warp 0
      mbar_init(&wempty[i], 8);      // converter warps
    }
    for (int i = 0; i < kMxAStages; ++i) {
      mbar_init(&afull[i], 64);      // gather threads
      mbar_init(&aempty[i], 1);      // MMA commit
    }
    for (int i = 0; i < kMxBStages; ++i) {
      mbar_init(&ready[i], 8);       // converter warps
      mbar_init(&bempty[i], 1);      // MMA commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
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

  if (warp == 0) {
    // ---------------- packed weight codes (TMA) + their scale words ----------------
    if (lane == 0) tma_prefetch_desc(&tm_w);
    uint32_t it = 0;
    bool alive = true;
    for (int uu = blockIdx.x; alive && uu < num_units; uu += gridDim.x) {
      const MxUnit u = decode(uu);
      const uint8_t* srow[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        srow[i] = p.w_scale + static_cast<size_t>(mx_wrow<KIND>(p, u, lane + 32 * i)) * (K / 32);
      const int r0 = mx_wrow<KIND>(p, u, 0), r64 = mx_wrow<KIND>(p, u, 64);
      // the next unit of this CTA, for warming L2 one raw ring ahead
      const bool has_next = uu + static_cast<int>(gridDim.x) < num_units;
      const MxUnit nu = has_next ? decode(uu + gridDim.x) : u;
      const int n0 = mx_wrow<KIND>(p, nu, 0), n64 = mx_wrow<KIND>(p, nu, 64);
      for (int ks = 0; ks < KS; ++ks, ++it) {
        if (lane == 0) {
          int pk = ks + kMxRawStages, p0 = r0, p64 = r64;
          if (pk >= KS && has_next) {
            pk -= KS;
            p0 = n0;
            p64 = n64;
          }
          if (pk < KS) {
            tma_prefetch_l2_2d(&tm_w, pk * (kMxBK / 2), p0);
            tma_prefetch_l2_2d(&tm_w, pk * (kMxBK / 2), p64);
          }
        }
        const int ws = it % kMxRawStages;
        const uint32_t ph = (it / kMxRawStages) & 1u;
        const bool ok = mbar_wait(&wempty[ws], ph ^ 1u, abort_flag, p.err);
        if (__any_sync(0xffffffffu, !ok)) {
          alive = false;
          break;
        }
        if (lane == 0) {
          uint8_t* dst = raw + ws * kMxRawW;
          mbar_arrive_expect_tx(&wfull[ws], kMxRawW);
          tma_load_2d(dst, &tm_w, &wfull[ws], ks * (kMxBK / 2), r0);
          tma_load_2d(dst + 64 * 64, &tm_w, &wfull[ws], ks * (kMxBK / 2), r64);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
          cp_async_4(smem_u32(sfb + ws * kMxNT + lane + 32 * i), srow[i] + ks * 4, 4u);
        cp_async_mbar_arrive_noinc(&wfull[ws]);
      }
    }
    cp_async_wait_all();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, acc_it = 0;
      bool alive = true;
      for (int uu = blockIdx.x; alive && uu < num_units; uu += gridDim.x, ++acc_it) {
        const int buf = acc_it & 1;
        const uint32_t aph = (acc_it >> 1) & 1u;
        if (!mbar_wait(&tempty[buf], aph ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * kMxAccCols;
        for (int ks = 0; ks < KS; ++ks, ++it) {
          const int sa = it % kMxAStages, sb = it % kMxBStages;
          const uint32_t bph = (it / kMxBStages) & 1u;
          // the converters signal after the token tile of this step has landed
          if (!mbar_wait(&ready[sb], bph, abort_flag, p.err)) {
            alive = false;
            break;
          }
          fence_proxy_async_smem();  // cp.async token rows -> tensor core
          tc_fence_after();
          const uint32_t a_addr = smem_u32(atile + sa * kMxA);
          const uint32_t b_addr = smem_u32(btile + sb * kMxB);
          const uint32_t sfa_t = tmem_base + kMxSfCol0 + 8 * sb;
#pragma unroll
          for (int kk = 0; kk < kMxBK / 32; ++kk)
            umma_mxf8(d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32),
                      idesc_mxf8(128, kMxNT, kk), sfa_t, sfa_t + 4, (ks > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&aempty[sa]);
          umma_commit(&bempty[sb]);
        }
        if (!alive) break;
        umma_commit(&tfull[buf]);
      }
    }
  } else if (warp < 4) {
    // ---------------- token codes + scale words (cp.async gather) ----------------
    const int gt = threadIdx.x - 64;  // 0..63
    const int chunk = gt & 7;
    uint32_t it = 0;
    bool alive = true;
    auto row_src = [&](const MxUnit& u, int r, const uint8_t*& codes, const uint8_t*& scales) {
      codes = nullptr;
      scales = nullptr;
      if (r >= p.BM) return;
      const size_t prow = static_cast<size_t>(u.b) * p.BM + r;
      if constexpr (KIND == 0) {
        const int a = __ldg(p.sorted_ids + prow);
        if (a < 0 || a >= p.T * p.k) return;
        const size_t tok = static_cast<size_t>(a / p.k);
        codes = p.act + tok * K;
        scales = p.act_scale + tok * (K / 32);
      } else {
        codes = p.act + prow * K;
        scales = p.act_scale + prow * (K / 32);
      }
    };
    for (int uu = blockIdx.x; alive && uu < num_units; uu += gridDim.x) {
      const MxUnit u = decode(uu);
      const uint8_t* src[16];
      const uint8_t* ssrc[2];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint8_t* sc;
        row_src(u, (gt >> 3) + 8 * i, src[i], sc);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint8_t* cd;
        row_src(u, gt + 64 * j, cd, ssrc[j]);
      }
      for (int ks = 0; ks < KS; ++ks, ++it) {
        const int s = it % kMxAStages;
        const uint32_t ph = (it / kMxAStages) & 1u;
        if (!mbar_wait(&aempty[s], ph ^ 1u, abort_flag, p.err)) {
          alive = false;
          break;
        }
        const uint32_t tile = smem_u32(atile + s * kMxA);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = (gt >> 3) + 8 * i;
          const uint32_t dst = tile + r * 128 + ((chunk ^ (r & 7)) << 4);
          cp_async_16(dst, src[i] ? static_cast<const void*>(src[i] + ks * kMxBK + chunk * 16) : p.act,
                      src[i] ? 16u : 0u);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
          cp_async_4(smem_u32(sfa + s * 128 + gt + 64 * j),
                     ssrc[j] ? static_cast<const void*>(ssrc[j] + ks * 4) : p.act_scale,
                     ssrc[j] ? 4u : 0u);
        // the stage barrier counts this thread's arrival when its copies land
        cp_async_mbar_arrive_noinc(&afull[s]);
      }
    }
    cp_async_wait_all();
  } else if (warp < 12) {
    // ---------------- weight codes -> e4m3 operand, scale factors -> TMEM ----------------
    const int ct = threadIdx.x - 128;  // 0..255: half (ct & 1) of weight row ct >> 1
    const int row = ct >> 1, half = ct & 1;
    const int q = warp & 3;            // this warp's TMEM lane quarter
    const bool token_sf = warp < 8;    // warps 4-7: token scales, warps 8-11: weight scales
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t it = 0;
    bool alive = true;
    for (int uu = blockIdx.x; alive && uu < num_units; uu += gridDim.x) {
      for (int ks = 0; ks < KS; ++ks, ++it) {
        const int sa = it % kMxAStages, sb = it % kMxBStages, ws = it % kMxRawStages;
        const uint32_t aph = (it / kMxAStages) & 1u, bph = (it / kMxBStages) & 1u,
                       wph = (it / kMxRawStages) & 1u;
        bool ok = mbar_wait(&bempty[sb], bph ^ 1u, abort_flag, p.err);
        ok = ok && mbar_wait(&wfull[ws], wph, abort_flag, p.err);
        if (token_sf) ok = ok && mbar_wait(&afull[sa], aph, abort_flag, p.err);
        // the warp stops as one (its lanes meet in the warp-wide TMEM stores)
        if (__any_sync(0xffffffffu, !ok)) {
          alive = false;
          break;
        }
        // 32 packed bytes (64 codes) of the row -> 64 e4m3 bytes, 128-byte swizzle
        const uint32_t rsrc = smem_u32(raw + ws * kMxRawW) + row * 64 + half * 32;
        const uint4 w0 = ld_shared_v4(rsrc), w1 = ld_shared_v4(rsrc + 16);
        const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        const uint32_t bt = smem_u32(btile + sb * kMxB) + row * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint2 lo = e2m1x8_to_e4m3x8(words[2 * j]);
          const uint2 hi = e2m1x8_to_e4m3x8(words[2 * j + 1]);
          const int c = 4 * half + j;
          st_shared_v4(bt + ((c ^ (row & 7)) << 4), lo.x, lo.y, hi.x, hi.y);
        }
        const uint32_t sf_col = kMxSfCol0 + 8 * sb;
        if (token_sf) {
          // token row 32q + lane: lane 32q + lane, column sf_col + q
          tmem_st1(lane_base + sf_col + q,
                   ld_shared_u32(smem_u32(sfa + sa * 128 + q * 32 + lane)));
        } else {
          // weight row 32c + lane: lane (mod 32) of every quarter, column sf_col + 4 + c
          const uint32_t* w = sfb + ws * kMxNT;
          tmem_st4(lane_base + sf_col + 4, w[lane], w[32 + lane], w[64 + lane], w[96 + lane]);
        }
        tmem_st_wait();
        fence_proxy_async_smem();  // generic-proxy tile writes -> tensor core reads
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&ready[sb]);
          mbar_arrive(&wempty[ws]);
        }
      }
    }
  } else if (warp >= 12) {
    // ---------------- epilogue ----------------
    const int ew = warp & 3;
    const int row = ew * 32 + lane;
    uint32_t acc_it = 0;
    for (int uu = blockIdx.x; uu < num_units; uu += gridDim.x, ++acc_it) {
      const MxUnit u = decode(uu);
      const int buf = acc_it & 1;
      const uint32_t aph = (acc_it >> 1) & 1u;
      const bool ok = mbar_wait(&tfull[buf], aph, abort_flag, p.err);
      if (named_bar_any(1, 128, !ok || *abort_flag)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + buf * kMxAccCols;
      const bool rvalid = row < p.BM;
      const size_t prow = static_cast<size_t>(u.b) * p.BM + row;
      if constexpr (KIND == 0) {
        // SwiGLU of gate column c and up column 64 + c, re-quantised per 32
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
          uint32_t g0[16], g1[16], u0[16], u1[16];
          tmem_ld16(tb + 32 * j, g0);
          tmem_ld16(tb + 32 * j + 16, g1);
          tmem_ld16(tb + 64 + 32 * j, u0);
          tmem_ld16(tb + 64 + 32 * j + 16, u1);
          tmem_ld_wait();
          reg_fence16(g0);
          reg_fence16(g1);
          reg_fence16(u0);
          reg_fence16(u1);
          float act[32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            act[i] = swiglu_f(__uint_as_float(g0[i]), __uint_as_float(u0[i]));
            act[16 + i] = swiglu_f(__uint_as_float(g1[i]), __uint_as_float(u1[i]));
          }
          uint32_t codes[8];
          const uint32_t sbyte = requant32(act, codes);
          const int f = u.n * (kMxNT / 2) + 32 * j;
          if (rvalid && f + 32 <= p.F) {
            st_global_v8(p.inter_q + prow * p.F + f, codes);
            p.inter_scale[prow * (p.F / 32) + f / 32] = static_cast<uint8_t>(sbyte);
          }
        }
      } else {
        int a = p.T * p.k;
        if (rvalid) a = __ldg(p.sorted_ids + prow);
        const bool valid = rvalid && a >= 0 && a < p.T * p.k;
        const float w = valid ? __ldg(p.topk_weights + a) : 0.f;
#pragma unroll 1
        for (int c = 0; c < kMxNT / 16; ++c) {
          uint32_t r[16];
          tmem_ld16(tb + 16 * c, r);
          tmem_ld_wait();
          reg_fence16(r);
          const int h = u.n * kMxNT + 16 * c;
          if (valid && h + 16 <= p.H) {
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              o[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * w, __uint_as_float(r[2 * i + 1]) * w);
            st_global_v8(p.stage + static_cast<size_t>(a) * p.H + h, o);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kMxTmemCols);
  }
}

}  // namespace

int launch_lowbit_gemm(int kind, const LowbitParams& p, int num_sms, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(lowbit_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMxSmem) != cudaSuccess ||
        cudaFuncSetAttribute(lowbit_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMxSmem) != cudaSuccess)
      return -1;
    attr_set = true;
  }
  // packed weight codes [E*2F or E*H rows, K/2 bytes], box 64 bytes x 64 rows
  const int K = (kind == 0) ? p.H : p.F;
  const uint64_t rows = (kind == 0) ? static_cast<uint64_t>(p.E) * 2 * p.F
                                    : static_cast<uint64_t>(p.E) * p.H;
  CUtensorMap tm_w;
  if (!make_map_u8(&tm_w, p.w, rows, static_cast<uint64_t>(K) / 2, 64, 64)) return -1;
  if (kind == 0)
    lowbit_gemm_kernel<0><<<num_sms, kMxThreads, kMxSmem, stream>>>(tm_w, p);
  else
    lowbit_gemm_kernel<1><<<num_sms, kMxThreads, kMxSmem, stream>>>(tm_w, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace moe
