// moe_common.cuh -- device helpers shared by the kernels of the CUDA library:
// error word, bounded mbarrier waits, TMA, cp.async and tcgen05 (UMMA / TMEM)
// wrappers written as inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MOE_DEV __device__ __forceinline__

namespace moe {

// ---------------------------------------------------------------------------
// Device error word (sticky, OR-ed) -- bits mirror include/moe.h.
// ---------------------------------------------------------------------------
enum : int { kErrBadExpert = 1, kErrTimeout = 2, kErrBadTable = 4 };

MOE_DEV void raise_error(int* err, int code) {
  if (err) atomicOr(err, code);
}

// A bounded wait gives up after this many SM clock cycles (~2 s at 2 GHz).
constexpr long long kWaitLimitCycles = 1ll << 32;

MOE_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
MOE_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
MOE_DEV void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

MOE_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n}\n" ::"r"(
          smem_u32(bar))
      : "memory");
}
MOE_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], "
      "%1;\n}\n" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
MOE_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, "
      "1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait until the phase with parity `parity` of `bar` has completed.  Gives up
// (sets the CTA abort flag and the device error word) after kWaitLimitCycles or
// as soon as another role of the CTA has given up.  Returns false on give-up.
MOE_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      *abort_flag = 1;
      raise_error(err, kErrTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (tiled bulk tensor copies, global -> shared)
// ---------------------------------------------------------------------------
MOE_DEV void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2-D tile load: c0 = innermost (element) coordinate, c1 = row.
MOE_DEV void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// 2-D tile load delivered to the same shared-memory offset of every CTA of
// the cluster in cta_mask, each CTA's barrier (same offset) counting the
// bytes that reach it.
MOE_DEV void tma_load_2d_mc(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                            uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "h"(cta_mask)
      : "memory");
}
MOE_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster (release / acquire).
MOE_DEV void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Warm L2 with a tile (no shared memory, no barrier) ahead of its load.
MOE_DEV void tma_prefetch_l2_2d(const CUtensorMap* map, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}

// ---------------------------------------------------------------------------
// Block tables of the expert GEMMs.  Normally the align outputs: padded
// length, block_expert, sorted_ids.  With `naive` set (one token: "Mixture
// of Experts", vLLM's path that skips the alignment), every block holds one
// assignment: block b is assignment b in row 0 (padding in the other rows),
// block_expert is topk_ids itself, and the padded length is T*k*BLOCK_M.
// ---------------------------------------------------------------------------
template <class P>
MOE_DEV int padded_rows(const P& p, int bm) {
  const int npp = p.naive ? p.T * p.k * bm : __ldg(p.num_post_padded);
  return max(0, min(npp, p.cap_rows));
}
template <class P>
MOE_DEV int row_assignment(const P& p, int b, int bm, int r) {
  if (p.naive) return r == 0 ? b : p.T * p.k;
  return __ldg(p.sorted_ids + static_cast<size_t>(b) * bm + r);
}

// ---------------------------------------------------------------------------
// cp.async (16-byte global -> shared, zero-filled when src_bytes == 0)
// ---------------------------------------------------------------------------
MOE_DEV void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
MOE_DEV void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
MOE_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Arrive on `bar` (counted in its expected arrivals) once all cp.async copies
// issued so far by this thread have landed; the thread does not wait.
MOE_DEV void cp_async_mbar_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
MOE_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
template <int N>
MOE_DEV void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Make generic-proxy writes to shared memory visible to the async proxy
// (tensor core operand reads).
MOE_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

MOE_DEV void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Named barrier that also returns, to every participating thread, whether any
// of them passed pred = true.
MOE_DEV bool named_bar_any(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 "
      "%0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation tensor core (cta_group::1)
// ---------------------------------------------------------------------------
// Warp-wide: allocate `ncols` TMEM columns (power of two, 32..512); the base
// address is written to *slot (shared memory).
MOE_DEV void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
MOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
MOE_DEV void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                      uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, "
      "%2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on the barrier at the same offset in every CTA of the
// cluster in cta_mask when all tcgen05 operations issued so far by this
// thread have completed.
MOE_DEV void umma_commit_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}
// Arrive (once) on `bar` when all tcgen05 operations issued so far by this
// thread have completed.
MOE_DEV void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Warp-wide TMEM load: lane i of the warp receives 16 consecutive 32-bit
// columns of TMEM lane (address lane field + i).
MOE_DEV void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
MOE_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// After tmem_ld_wait: ties the loaded registers to a point after the wait so
// no use of them can be scheduled before the asynchronous load completed.
MOE_DEV void reg_fence16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes (64 bf16 of K), 8-row groups 1024 bytes
// apart, tile base 1024-byte aligned.  Advancing along K inside the 128-byte
// row is done by adding the byte offset to the start address.
MOE_DEV uint64_t sw128_desc(uint32_t smem_byte_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_byte_addr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                           // leading byte offset (16 B, unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                   // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                           // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                           // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// cross-CTA hand-off without spinning: the threads of a CTA (or of a named
// barrier group) write their results, synchronise, and one thread bumps a
// ticket with acquire-release semantics at GPU scope; the CTA that draws the
// last ticket reads the others' results with L2 (ld.global.cg) loads.
// ---------------------------------------------------------------------------
MOE_DEV int ticket_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}
MOE_DEV void store_relaxed_gpu(int* p, int v) {
  asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
MOE_DEV int load_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
MOE_DEV void store_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Barrier over the CTAs of a cooperative launch (all co-resident).  bar[0]
// counts arrivals and is reset by the last CTA, bar[1] is a generation that
// the last CTA advances; both start at zero.  The wait is bounded: after
// `limit` SM clock cycles (kWaitLimitCycles when limit <= 0) it records
// kErrTimeout and returns false to every thread of the CTA (the caller must
// then skip whatever depends on the other CTAs).
MOE_DEV bool grid_barrier(int* bar, int nctas, int* err, long long limit = 0) {
  if (limit <= 0) limit = kWaitLimitCycles;
  __shared__ int gb_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const int gen = load_acquire_gpu(bar + 1);
    __threadfence();
    const int old = ticket_add_acq_rel(bar, 1);
    if (old == nctas - 1) {
      store_relaxed_gpu(bar, 0);
      store_release_gpu(bar + 1, gen + 1);
    } else {
      const long long t0 = clock64();
      while (load_acquire_gpu(bar + 1) == gen) {
        if (clock64() - t0 > limit) {
          raise_error(err, kErrTimeout);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    gb_ok = ok;
  }
  __syncthreads();
  return gb_ok != 0;
}

// Order-preserving map of fp32 onto uint32 (for warp max/min reductions).
MOE_DEV uint32_t f2ord(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
MOE_DEV float ord2f(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// ---------------------------------------------------------------------------
// small numeric helpers
// ---------------------------------------------------------------------------
// silu(g) * u with silu(g) = g * sigmoid(g) = (g/2) * (1 + tanh(g/2)): one
// hardware tanh instead of an exponential and a reciprocal.  Relative error
// about 2^-11, below the bf16 rounding of the result.
MOE_DEV float swiglu_f(float g, float u) {
  const float hg = 0.5f * g;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(hg));
  return fmaf(hg, t, hg) * u;
}
// 32-byte store (one full sector); the address must be 32-byte aligned.
MOE_DEV void st_global_v8(void* p, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

MOE_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// FP8 cast of 32 consecutive bf16 values ("How GPUs Fuse Communication and
// Computation During LLM Inference" §1.1 and the scale rule of §3.5): 2^s is
// the smallest power of two with amax / 2^s <= 448 (s in [-127, 127]; 0 for
// an all-zero group), codes = e4m3(v / 2^s), nearest, ties to even,
// saturating; the scale byte is s + 127 (UE8M0).  s comes from amax's binary
// exponent, not from a rounded quotient: amax = m * 2^e with m in [0.5, 1)
// and 448 = 0.875 * 2^9, so amax <= 448 * 2^s exactly when s >= e - 9
// (m <= 0.875) or s >= e - 8 (m > 0.875).  src: four 16-byte words (64
// bytes), dst: two 16-byte words of codes.
MOE_DEV void cast_e4m3_group32(const uint4* __restrict__ src, uint4* __restrict__ dst,
                               uint8_t* __restrict__ scale) {
  uint4 raw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) raw[i] = __ldg(src + i);
  float v[32];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);  // bf16 -> fp32, exact
      v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  int s = 0;
  if (amax > 0.f) {
    int e;
    const float m = frexpf(amax, &e);
    s = (m <= 0.875f) ? e - 9 : e - 8;
    s = max(-127, min(127, s));
  }
  // 2^-s exactly (2^127 at most; 2^-127 is the subnormal 0x00400000)
  const float mul = (s <= 126) ? __int_as_float((127 - s) << 23) : __int_as_float(0x00400000);
  uint32_t c[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(v[4 * i] * mul, v[4 * i + 1] * mul), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(v[4 * i + 2] * mul, v[4 * i + 3] * mul), __NV_SATFINITE, __NV_E4M3);
    c[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
  dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
  *scale = static_cast<uint8_t>(s + 127);
}

}  // namespace moe
