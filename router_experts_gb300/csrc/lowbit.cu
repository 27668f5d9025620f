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
// operand row, fp32 accumulation in TMEM).  Nothing is converted on the SMs:
//   B = 128 weight rows, loaded by TMA straight from the packed e2m1 codes
//       with the 16 x 4-bit / 16-byte tensor-map type: each 16 codes land as
//       their 8 packed bytes plus an 8-byte gap, the MMA's 4-bit operand
//       layout (the copy counts the packed bytes in its transactions);
//   A = 128 token rows of e4m3 codes: GEMM1 gathers them by sorted_ids with
//       cp.async, GEMM2 reads its contiguous intermediate rows by TMA;
//   scale words (4 K-blocks of one row) are copied into a [32][4]-word image
//       per operand (word c of image row l = operand row 32c + l) and moved
//       to TMEM by the MMA thread with tcgen05.cp 32x128b.warpx4, which puts
//       image row l in lane l of every lane quarter: row m of A reads lane m,
//       column base + m/32; row n of B reads lane n mod 32, column base + 4 +
//       n/32; byte j of the word scales K-block j of the step.
// Tile: M = 128 token rows of one block (BLOCK_M rows valid), N = 128 weight
// rows (GEMM1: 64 gate rows + the matching 64 up rows), K steps of 128 (four
// K = 32 MMAs).  Two 128-column accumulators, double-buffered; the scale
// words of a step sit in an 8-column TMEM slot tied to its weight stage.
// 10 warps:
//   warp 0      TMA of the weight tiles (L2 warmed kMxL2Ahead steps ahead
//               through a plain byte map of the same codes)
//               and, one row per lane, cp.async of their scale words
//   warp 1      TMEM allocation and the single thread issuing tcgen05.cp and
//               the MMAs
//   warps 2-5   token tiles: GEMM1 cp.async gather of the codes and scale
//               words; GEMM2 TMA of the codes, cp.async of the scale words
//   warps 6-9   epilogue (TMEM lane quarter = warp % 4)
#include <cuda_fp8.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kMxThreads = 320;
constexpr int kMxBK = 128;                  // K values per stage (4 MMAs of K = 32)
constexpr int kMxNT = 128;                  // weight rows per tile (MMA N)
constexpr int kMxAStages = 7;               // token tiles
constexpr int kMxBStages = 6;               // weight tiles (and TMEM scale slots)
constexpr int kMxL2Ahead = 12;              // weight steps warmed in L2 ahead of their load
constexpr int kMxTile = 128 * kMxBK;        // 16 KB per tile (one byte per code in smem)
constexpr int kMxSfImg = 128 * 4;           // 512 B: one operand's scale words of a step
constexpr int kMxBarBytes = 512;
constexpr int kMxSmem =
    (kMxAStages + kMxBStages) * (kMxTile + kMxSfImg) + kMxBarBytes + 1024;
static_assert(kMxSmem <= 232448, "shared memory budget");
constexpr uint32_t kMxAccCols = 128;        // per accumulator buffer
constexpr uint32_t kMxSfCol0 = 256;         // scale slots: 8 columns per weight stage
constexpr uint32_t kMxTmemCols = 512;
static_assert(kMxSfCol0 + 8 * kMxBStages <= kMxTmemCols, "TMEM columns");

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

// Shared-memory descriptor of a [32 rows x 16 bytes] image, no swizzle: one
// 16-byte core-matrix column, row groups of 8 every 128 bytes.
MOE_DEV uint64_t sf_image_desc(uint32_t smem_byte_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_byte_addr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                           // leading byte offset (unused)
  d |= static_cast<uint64_t>(128 >> 4) << 32;                    // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                           // descriptor version
  return d;
}

// Copy a [32 x 128-bit] shared-memory image into 4 TMEM columns of every lane
// quarter (image row l -> lanes l, 32 + l, 64 + l, 96 + l).  Ordered before
// the MMAs the same thread issues after it.
MOE_DEV void tmem_cp_32x128_x4(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
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
    lowbit_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_wpf,
                       const __grid_constant__ CUtensorMap tm_a, const LowbitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* atile = smem;                              // [kMxAStages][128 rows x 128 codes]
  uint8_t* btile = atile + kMxAStages * kMxTile;      // [kMxBStages][128 rows x 128 slots]
  uint32_t* sfa = reinterpret_cast<uint32_t*>(btile + kMxBStages * kMxTile);  // [kMxAStages][128]
  uint32_t* sfb = sfa + kMxAStages * 128;                                     // [kMxBStages][128]
  uint64_t* afull = reinterpret_cast<uint64_t*>(sfb + kMxBStages * 128);
  uint64_t* aempty = afull + kMxAStages;
  uint64_t* bfull = aempty + kMxAStages;
  uint64_t* bempty = bfull + kMxBStages;
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
  const int bmr = min(p.BM, 128);  // token rows of a tile that hold data

  if (threadIdx.x == 0) {
    for (int i = 0; i < kMxAStages; ++i) {
      // gather threads (cp.async arrivals); GEMM2 adds the TMA's expect-tx arrival
      mbar_init(&afull[i], 128 + (KIND == 1 ? 1 : 0));
      mbar_init(&aempty[i], 1);  // MMA commit
    }
    for (int i = 0; i < kMxBStages; ++i) {
      mbar_init(&bfull[i], 1 + 32);  // TMA bytes + the scale-word copies of warp 0
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
    // ---------------- weight tiles (TMA) + their scale words ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      tma_prefetch_desc(&tm_wpf);
    }
    uint32_t it = 0;
    bool alive = true;
    for (int uu = blockIdx.x; alive && uu < num_units; uu += gridDim.x) {
      const MxUnit u = decode(uu);
      // lane l copies the scale words of rows l, 32 + l, 64 + l, 96 + l: image
      // row l, words 0..3
      const uint8_t* srow[4];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        srow[c] = p.w_scale + static_cast<size_t>(mx_wrow<KIND>(p, u, lane + 32 * c)) * (K / 32);
      const int r0 = mx_wrow<KIND>(p, u, 0), r64 = mx_wrow<KIND>(p, u, 64);
      // the next unit of this CTA, for warming L2 across the unit boundary
      const bool has_next = uu + static_cast<int>(gridDim.x) < num_units;
      const MxUnit nu = has_next ? decode(uu + gridDim.x) : u;
      const int n0 = mx_wrow<KIND>(p, nu, 0), n64 = mx_wrow<KIND>(p, nu, 64);
      for (int ks = 0; ks < KS; ++ks, ++it) {
        if (lane == 0) {
          int pk = ks + kMxL2Ahead, p0 = r0, p64 = r64;
          if (pk >= KS && has_next) {
            pk -= KS;
            p0 = n0;
            p64 = n64;
          }
          if (pk < KS) {  // byte map of the packed codes: x in bytes
            tma_prefetch_l2_2d(&tm_wpf, pk * (kMxBK / 2), p0);
            tma_prefetch_l2_2d(&tm_wpf, pk * (kMxBK / 2), p64);
          }
        }
        const int ws = it % kMxBStages;
        const uint32_t ph = (it / kMxBStages) & 1u;
        const bool ok = mbar_wait(&bempty[ws], ph ^ 1u, abort_flag, p.err);
        if (__any_sync(0xffffffffu, !ok)) {
          alive = false;
          break;
        }
        if (lane == 0) {
          uint8_t* dst = btile + ws * kMxTile;
          // two 64-row boxes of 128 codes: 2 x 64 x 64 packed bytes
          mbar_arrive_expect_tx(&bfull[ws], kMxNT * kMxBK / 2);
          tma_load_2d(dst, &tm_w, &bfull[ws], ks * kMxBK, r0);
          tma_load_2d(dst + 64 * 128, &tm_w, &bfull[ws], ks * kMxBK, r64);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
          cp_async_4(smem_u32(sfb + ws * 128 + 4 * lane + c), srow[c] + ks * 4, 4u);
        cp_async_mbar_arrive_noinc(&bfull[ws]);
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
          if (!mbar_wait(&afull[sa], (it / kMxAStages) & 1u, abort_flag, p.err) ||
              !mbar_wait(&bfull[sb], (it / kMxBStages) & 1u, abort_flag, p.err)) {
            alive = false;
            break;
          }
          fence_proxy_async_smem();  // cp.async rows and scale words -> tensor core
          tc_fence_after();
          // The scale slot of weight stage sb was last read by the MMAs of step
          // it - kMxBStages, complete before that stage was refilled.
          const uint32_t sf_t = tmem_base + kMxSfCol0 + 8 * sb;
          tmem_cp_32x128_x4(sf_t, sf_image_desc(smem_u32(sfa + sa * 128)));
          tmem_cp_32x128_x4(sf_t + 4, sf_image_desc(smem_u32(sfb + sb * 128)));
          const uint32_t a_addr = smem_u32(atile + sa * kMxTile);
          const uint32_t b_addr = smem_u32(btile + sb * kMxTile);
#pragma unroll
          for (int kk = 0; kk < kMxBK / 32; ++kk)
            umma_mxf8f4(d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32),
                        idesc_mxf8f4(128, kMxNT, kk), sf_t, sf_t + 4,
                        (ks > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&aempty[sa]);
          umma_commit(&bempty[sb]);
        }
        if (!alive) break;
        umma_commit(&tfull[buf]);
      }
    }
  } else if (warp < 6) {
    // ---------------- token tiles + their scale words ----------------
    const int gt = threadIdx.x - 64;  // 0..127
    const int chunk = gt & 7;
    // image slot of row gt's scale word: image row gt % 32, word gt / 32
    const int sf_word = 4 * (gt & 31) + (gt >> 5);
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
    if (KIND == 1 && gt == 0) tma_prefetch_desc(&tm_a);
    for (int uu = blockIdx.x; alive && uu < num_units; uu += gridDim.x) {
      const MxUnit u = decode(uu);
      const uint8_t* src[8];
      const uint8_t* ssrc;
      {
        const uint8_t* cd;
        row_src(u, gt, cd, ssrc);
      }
      if constexpr (KIND == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint8_t* sc;
          row_src(u, (gt >> 3) + 16 * i, src[i], sc);
        }
      }
      for (int ks = 0; ks < KS; ++ks, ++it) {
        const int s = it % kMxAStages;
        const uint32_t ph = (it / kMxAStages) & 1u;
        if (!mbar_wait(&aempty[s], ph ^ 1u, abort_flag, p.err)) {
          alive = false;
          break;
        }
        if constexpr (KIND == 0) {
          const uint32_t tile = smem_u32(atile + s * kMxTile);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = (gt >> 3) + 16 * i;
            const uint32_t dst = tile + r * 128 + ((chunk ^ (r & 7)) << 4);
            cp_async_16(dst,
                        src[i] ? static_cast<const void*>(src[i] + ks * kMxBK + chunk * 16) : p.act,
                        src[i] ? 16u : 0u);
          }
        } else {
          // the block's rows are contiguous: one box of bmr rows
          if (gt == 0) {
            mbar_arrive_expect_tx(&afull[s], static_cast<uint32_t>(bmr) * kMxBK);
            tma_load_2d(atile + s * kMxTile, &tm_a, &afull[s], ks * kMxBK, u.b * p.BM);
          }
        }
        cp_async_4(smem_u32(sfa + s * 128 + sf_word),
                   ssrc ? static_cast<const void*>(ssrc + ks * 4) : p.act_scale, ssrc ? 4u : 0u);
        // the stage barrier counts this thread's arrival when its copies land
        cp_async_mbar_arrive_noinc(&afull[s]);
      }
    }
    cp_async_wait_all();
  } else {
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
  // packed weight codes [E*2F or E*H rows, K codes], box 128 codes x 64 rows
  const int K = (kind == 0) ? p.H : p.F;
  const uint64_t rows = (kind == 0) ? static_cast<uint64_t>(p.E) * 2 * p.F
                                    : static_cast<uint64_t>(p.E) * p.H;
  // the same bytes as a plain byte map (box 64 bytes x 64 rows) for the L2 warm-up
  CUtensorMap tm_w, tm_wpf, tm_a;
  if (!make_map_e2m1(&tm_w, p.w, rows, static_cast<uint64_t>(K), 64)) return -1;
  if (!make_map_u8(&tm_wpf, p.w, rows, static_cast<uint64_t>(K) / 2, 64, 64)) return -1;
  if (kind == 0) {
    tm_a = tm_w;  // unused: GEMM1 gathers its token rows
    lowbit_gemm_kernel<0><<<num_sms, kMxThreads, kMxSmem, stream>>>(tm_w, tm_wpf, tm_a, p);
  } else {
    // intermediate codes [cap_rows, F], one box = the data rows of a block
    const uint32_t bmr = static_cast<uint32_t>(p.BM < 128 ? p.BM : 128);
    if (!make_map_u8_sw128(&tm_a, p.act, static_cast<uint64_t>(p.cap_rows),
                           static_cast<uint64_t>(p.F), bmr))
      return -1;
    lowbit_gemm_kernel<1><<<num_sms, kMxThreads, kMxSmem, stream>>>(tm_w, tm_wpf, tm_a, p);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace moe
