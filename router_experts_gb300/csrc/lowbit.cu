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
// HBM traffic stays low-bit: converter warps read the packed codes and the
// scale bytes, dequantise them into f16 in registers (exact while the value
// fits: e2m1 x 2^u for u in [-14, 13], e4m3 x 2^u for u in [-14, 7]; the
// exponent is clamped to [-14, 15] before the multiply), and write the
// 128-byte-swizzled operand tiles that a single thread feeds to
// tcgen05.mma kind::f16 (f16 x f16 -> fp32 in TMEM; every product is exact).
// 16 warps: warp 1 allocates TMEM and issues the MMAs, warps 2-9 convert
// (one weight row and half a token row each per stage), warps 12-15 run the
// epilogue; the others idle.  Tile: M = 128 token rows of one block (BLOCK_M
// rows valid), N = 256 weight rows, K steps of 64, four stages, two
// double-buffered 256-column accumulators.
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kLbThreads = 512;
constexpr int kLbStages = 2;                // f16 operand stages
constexpr int kLbA = 128 * 128;             // 128 token rows x 64 f16
constexpr int kLbB = 256 * 128;             // 256 weight rows x 64 f16
constexpr int kLbStage = kLbA + kLbB;       // 48 KB
constexpr int kLbConv = 256;                // converter threads (warps 2-9)
// Raw codes are staged per converter thread: each K step's 32 weight-code
// bytes, 32 token-code bytes and the aligned words holding their scale bytes
// land in the thread's own shared-memory slot by cp.async, kLbDepth steps
// ahead of their conversion.
constexpr int kLbDepth = 6;
constexpr int kLbSlot = 80;                 // 32 W | 32 X | 4 W scales | 4 X scale | pad
constexpr int kLbRawBytes = kLbDepth * kLbConv * kLbSlot;
constexpr int kLbSmem = kLbStages * kLbStage + kLbRawBytes + 1024 + 512;
static_assert(kLbSmem <= 232448, "shared memory budget");
constexpr uint32_t kLbIdesc = (1u << 4) | (static_cast<uint32_t>(256 >> 3) << 17) |
                              (static_cast<uint32_t>(128 >> 4) << 24);  // f16 x f16 -> f32

// f16x2 holding 2^(code-127) twice (exponent clamped to the normal f16 range).
MOE_DEV uint32_t scale_f16x2(uint32_t code) {
  int e = static_cast<int>(code) - 127;
  e = max(-14, min(15, e));
  const uint32_t h = static_cast<uint32_t>(e + 15) << 10;
  return h | (h << 16);
}

MOE_DEV uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 x = *reinterpret_cast<__half2*>(&a), y = *reinterpret_cast<__half2*>(&b);
  __half2 r = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&r);
}

// 4 bytes = 8 e2m1 codes (low nibble first) -> 8 f16 (4 registers), scaled.
// One hardware conversion per byte (two codes; the low nibble becomes the low
// half of the f16 pair), then one f16x2 multiply by the power-of-two scale.
MOE_DEV void fp4x8_to_f16(uint32_t w, uint32_t s2, uint32_t (&o)[4]) {
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
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = hmul2_u32(h[i], s2);
}
// 8 bytes = 8 e4m3 codes -> 8 f16 (4 registers), scaled: one hardware
// conversion per code pair (low byte -> low half), one f16x2 multiply.
MOE_DEV void fp8x8_to_f16(uint32_t lo, uint32_t hi, uint32_t s2, uint32_t (&o)[4]) {
  uint32_t h[4];
  asm("{\n"
      " .reg .b16 p0, p1, p2, p3;\n"
      " mov.b32 {p0, p1}, %4;\n"
      " mov.b32 {p2, p3}, %5;\n"
      " cvt.rn.f16x2.e4m3x2 %0, p0;\n"
      " cvt.rn.f16x2.e4m3x2 %1, p1;\n"
      " cvt.rn.f16x2.e4m3x2 %2, p2;\n"
      " cvt.rn.f16x2.e4m3x2 %3, p3;\n"
      "}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(lo), "r"(hi));
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = hmul2_u32(h[i], s2);
}

MOE_DEV void st_shared_v4(uint32_t addr, const uint32_t (&v)[4]) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3])
               : "memory");
}

struct LbUnit {
  int b, n, e;
};

// Source rows of one converter thread for one unit: weight row ct of the
// tile and half (ct & 1) of token row ct >> 1.  Null pointers stand for
// padding (their copies zero-fill the slot).
struct LbRows {
  const uint8_t* w;    // weight codes of the row (K/2 bytes)
  const uint8_t* wsc;  // its scale bytes (K/32)
  const uint8_t* x;    // token codes of the row (K bytes)
  const uint8_t* xsc;  // its scale bytes (K/32)
};

template <int KIND>
MOE_DEV LbRows lb_rows(const LowbitParams& p, const LbUnit& u, int ct, int K) {
  LbRows r{};
  int wrow;
  bool wv;
  if constexpr (KIND == 0) {
    const int fr = u.n * 128 + (ct & 127);
    wv = fr < p.F;
    wrow = u.e * 2 * p.F + ((ct < 128) ? 0 : p.F) + fr;
  } else {
    const int hr = u.n * 256 + ct;
    wv = hr < p.H;
    wrow = u.e * p.H + hr;
  }
  if (wv) {
    r.w = p.w + static_cast<size_t>(wrow) * (K / 2);
    r.wsc = p.w_scale + static_cast<size_t>(wrow) * (K / 32);
  }
  const int tr = ct >> 1;
  if (tr < p.BM) {
    const size_t prow = static_cast<size_t>(u.b) * p.BM + tr;
    if constexpr (KIND == 0) {
      const int a = __ldg(p.sorted_ids + prow);
      if (a >= 0 && a < p.T * p.k) {
        const size_t tok = static_cast<size_t>(a / p.k);
        r.x = p.act + tok * K;
        r.xsc = p.act_scale + tok * (K / 32);
      }
    } else {
      r.x = p.act + prow * K;
      r.xsc = p.act_scale + prow * (K / 32);
    }
  }
  return r;
}

// cp.async of K step kb into a slot: 32 weight-code bytes, the 32 token-code
// bytes of this thread's half row, and the 4-byte words holding the scale
// bytes (every scale row starts 4-byte aligned and spans a multiple of 4
// bytes, so a word never leaves its row).
MOE_DEV void lb_issue(const LbRows& r, int kb, int half, uint32_t slot, const void* dummy) {
  const uint8_t* w = r.w ? r.w + static_cast<size_t>(kb) * 32 : nullptr;
  const uint8_t* x = r.x ? r.x + static_cast<size_t>(kb) * 64 + half * 32 : nullptr;
  cp_async_16(slot, w ? static_cast<const void*>(w) : dummy, w ? 16u : 0u);
  cp_async_16(slot + 16, w ? static_cast<const void*>(w + 16) : dummy, w ? 16u : 0u);
  cp_async_16(slot + 32, x ? static_cast<const void*>(x) : dummy, x ? 16u : 0u);
  cp_async_16(slot + 48, x ? static_cast<const void*>(x + 16) : dummy, x ? 16u : 0u);
  cp_async_4(slot + 64, r.wsc ? static_cast<const void*>(r.wsc + ((2 * kb) & ~3)) : dummy,
             r.wsc ? 4u : 0u);
  cp_async_4(slot + 68, r.xsc ? static_cast<const void*>(r.xsc + ((2 * kb + half) & ~3)) : dummy,
             r.xsc ? 4u : 0u);
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

// Dequantise K step kb from a slot into the swizzled f16 operand tiles: the
// weight row ct into B, and (rows present in the block) half a token row into
// A.  Zero-filled codes of padding give zeros whatever their scale.
MOE_DEV void lb_convert(uint32_t slot, int kb, int ct, int BM, uint32_t a_tile, uint32_t b_tile) {
  const uint4 w0 = ld_shared_v4(slot), w1 = ld_shared_v4(slot + 16);
  const uint32_t wsw = ld_shared_u32(slot + 64);
  {
    const int b0 = (2 * kb) & 3;
    const uint32_t s_lo = scale_f16x2((wsw >> (8 * b0)) & 0xFFu);
    const uint32_t s_hi = scale_f16x2((wsw >> (8 * (b0 + 1))) & 0xFFu);
    const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const uint32_t row = ct;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t o[4];
      fp4x8_to_f16(words[j], j < 4 ? s_lo : s_hi, o);
      st_shared_v4(b_tile + row * 128 + ((j ^ (row & 7)) << 4), o);
    }
  }
  const int tr = ct >> 1, half = ct & 1;
  if (tr < BM) {
    const uint4 x0 = ld_shared_v4(slot + 32), x1 = ld_shared_v4(slot + 48);
    const uint32_t xsw = ld_shared_u32(slot + 68);
    const uint32_t s2 = scale_f16x2((xsw >> (8 * ((2 * kb + half) & 3))) & 0xFFu);
    const uint32_t words[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t o[4];
      fp8x8_to_f16(words[2 * j], words[2 * j + 1], s2, o);
      const int chunk = half * 4 + j;
      st_shared_v4(a_tile + tr * 128 + ((chunk ^ (tr & 7)) << 4), o);
    }
  }
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

template <int KIND>
__global__ void __launch_bounds__(kLbThreads, 1) lowbit_gemm_kernel(const LowbitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kLbStages * kLbStage + kLbRawBytes);
  uint64_t* empty_bar = full_bar + kLbStages;
  uint64_t* tfull_bar = empty_bar + kLbStages;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty_bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = (KIND == 0) ? p.H : p.F;
  const int KB = K / 64;
  int npp = __ldg(p.num_post_padded);
  npp = max(0, min(npp, p.cap_rows));
  const int nblk = npp / p.BM;
  const int ntiles = (KIND == 0) ? (p.F + 127) / 128 : (p.H + 255) / 256;
  const int num_units = nblk * ntiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kLbStages; ++i) {
      mbar_init(&full_bar[i], kLbConv / 32);  // one arrival per converter warp
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], 4);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto decode = [&](int uu) {
    LbUnit u;
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

  if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, acc_it = 0;
      bool alive = true;
      for (int uu = blockIdx.x; alive && uu < num_units; uu += gridDim.x, ++acc_it) {
        const int buf = acc_it & 1;
        const uint32_t aph = (acc_it >> 1) & 1u;
        if (!mbar_wait(&tempty_bar[buf], aph ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * 256;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int st = it % kLbStages;
          const uint32_t ph = (it / kLbStages) & 1u;
          if (!mbar_wait(&full_bar[st], ph, abort_flag, p.err)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + st * kLbStage);
          const uint32_t b_addr = a_addr + kLbA;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_f16(d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32), kLbIdesc,
                     (kb > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty_bar[st]);
        }
        if (!alive) break;
        umma_commit(&tfull_bar[buf]);
      }
    }
  } else if (warp >= 2 && warp < 10) {
    // ---------------- converters ----------------
    // Each thread runs its own cp.async pipeline kLbDepth K steps deep over
    // the flat sequence (unit, K step) of this CTA; it reads back only its own
    // slots, so cp.async.wait_group alone orders copy and use.
    const int ct = threadIdx.x - 64;  // 0..255
    const int half = ct & 1;
    const uint32_t raw0 = smem_u32(smem + kLbStages * kLbStage) + ct * kLbSlot;
    constexpr uint32_t kRawStride = kLbConv * kLbSlot;
    int iu = blockIdx.x, ikb = 0;
    LbRows ir{};
    if (iu < num_units) ir = lb_rows<KIND>(p, decode(iu), ct, K);
    uint32_t q_issue = 0;
    auto issue_next = [&]() {
      if (iu < num_units) {
        lb_issue(ir, ikb, half, raw0 + (q_issue % kLbDepth) * kRawStride, p.w);
        if (++ikb == KB) {
          ikb = 0;
          iu += gridDim.x;
          if (iu < num_units) ir = lb_rows<KIND>(p, decode(iu), ct, K);
        }
      }
      cp_async_commit();  // empty groups past the end keep the group count uniform
      ++q_issue;
    };
    for (int d = 0; d < kLbDepth - 1; ++d) issue_next();
    uint32_t it = 0;
    bool alive = true;
    for (int uu = blockIdx.x; alive && uu < num_units; uu += gridDim.x) {
      for (int kb = 0; kb < KB; ++kb, ++it) {
        issue_next();
        cp_async_wait<kLbDepth - 1>();  // this thread's copies of step `it` have landed
        const int st = it % kLbStages;
        const uint32_t ph = (it / kLbStages) & 1u;
        // the warp stops as one (its lanes meet at __syncwarp below)
        const bool ok = mbar_wait(&empty_bar[st], ph ^ 1u, abort_flag, p.err);
        if (__any_sync(0xffffffffu, !ok)) {
          alive = false;
          break;
        }
        const uint32_t a_tile = smem_u32(smem + st * kLbStage);
        lb_convert(raw0 + (it % kLbDepth) * kRawStride, kb, ct, p.BM, a_tile, a_tile + kLbA);
        fence_proxy_async_smem();  // generic-proxy tile writes -> tensor core reads
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_bar[st]);
      }
    }
    cp_async_wait_all();
  } else if (warp >= 12) {
    // ---------------- epilogue ----------------
    const int ew = warp - 12;
    const int row = ew * 32 + lane;
    uint32_t acc_it = 0;
    for (int uu = blockIdx.x; uu < num_units; uu += gridDim.x, ++acc_it) {
      const LbUnit u = decode(uu);
      const int buf = acc_it & 1;
      const uint32_t aph = (acc_it >> 1) & 1u;
      const bool ok = mbar_wait(&tfull_bar[buf], aph, abort_flag, p.err);
      if (named_bar_any(1, 128, !ok || *abort_flag)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + buf * 256;
      const bool rvalid = row < p.BM;
      const size_t prow = static_cast<size_t>(u.b) * p.BM + row;
      if constexpr (KIND == 0) {
        // SwiGLU of gate column c and up column 128 + c, re-quantised per 32
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          uint32_t g0[16], g1[16], u0[16], u1[16];
          tmem_ld16(tb + 32 * j, g0);
          tmem_ld16(tb + 32 * j + 16, g1);
          tmem_ld16(tb + 128 + 32 * j, u0);
          tmem_ld16(tb + 128 + 32 * j + 16, u1);
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
          const int f = u.n * 128 + 32 * j;
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
        for (int c = 0; c < 16; ++c) {
          uint32_t r[16];
          tmem_ld16(tb + 16 * c, r);
          tmem_ld_wait();
          reg_fence16(r);
          const int h = u.n * 256 + 16 * c;
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
      if (lane == 0) mbar_arrive(&tempty_bar[buf]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace

int launch_lowbit_gemm(int kind, const LowbitParams& p, int num_sms, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(lowbit_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kLbSmem) != cudaSuccess ||
        cudaFuncSetAttribute(lowbit_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kLbSmem) != cudaSuccess)
      return -1;
    attr_set = true;
  }
  if (kind == 0)
    lowbit_gemm_kernel<0><<<num_sms, kLbThreads, kLbSmem, stream>>>(p);
  else
    lowbit_gemm_kernel<1><<<num_sms, kLbThreads, kLbSmem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace moe
