// Device-side building blocks of the sm_103a FP8 pipeline: numeric helpers
// (bf16, FP8 conversion, exp_ref, absmax bit tricks), reductions, and inline
// PTX wrappers for mbarriers, TMA and the tcgen05 tensor-core instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8q {

constexpr unsigned kStatusNonfinite = 0x1u;
constexpr unsigned kStatusTimeout = 0x2u;

// --------------------------------------------------------------------------
// Numerics
// --------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// |value| of two packed bf16 as fp32 bit patterns; non-negative floats order like
// unsigned integers, and NaN patterns sort above +inf, so an integer max is an
// exact, order-independent absmax that propagates NaN.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t w) {
  return max((w & 0x7FFFu) << 16, w & 0x7FFF0000u);
}
__device__ __forceinline__ uint32_t abs_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }

// Two fp32 -> two FP8 codes (lo in the low byte), round-to-nearest-even, saturating.
template <int FMT>
__device__ __forceinline__ uint16_t cvt_fp8x2(float lo, float hi) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE,
                                            FMT == 0 ? __NV_E4M3 : __NV_E5M2);
}
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x4(float a, float b, float c, float d) {
  return (uint32_t)cvt_fp8x2<FMT>(a, b) | ((uint32_t)cvt_fp8x2<FMT>(c, d) << 16);
}

__device__ __forceinline__ float fmt_max(int fmt) { return fmt == 0 ? 448.0f : 57344.0f; }

// scale = fmax / amax (correctly rounded), scale_inv = 1 / scale; amax == 0 -> 1, 1.
__device__ __forceinline__ void scale_from_amax(float amax, int fmt, float& s, float& si) {
  if (amax == 0.0f) { s = 1.0f; si = 1.0f; return; }
  s = __fdiv_rn(fmt_max(fmt), amax);
  si = __fdiv_rn(1.0f, s);
}

// e^x as a fixed sequence of single-rounding fp32 operations: Cody-Waite
// reduction x = k*ln2 + r (ln2 split into a 9-bit high part, so k*hi is exact,
// plus a low correction) and the degree-8 Taylor polynomial of e^r in Horner
// form, both as fused multiply-adds, then multiplication by 2^k assembled
// from exponent bits (two steps when the result is subnormal).  Same answer
// on every run and every GPU.
__device__ __forceinline__ float exp_ref(float x) {
  if (x != x) return x;
  if (x > 88.72283935546875f) return __int_as_float(0x7F800000);
  if (x < -103.972084045410156f) return 0.0f;
  const float kf = rintf(__fmul_rn(x, 1.44269502162933349609375f));
  const float r = __fmaf_rn(-kf, -2.12194440e-4f, __fmaf_rn(-kf, 0.693359375f, x));
  float p = 1.0f / 40320.0f;
  p = __fmaf_rn(p, r, 1.0f / 5040.0f);
  p = __fmaf_rn(p, r, 1.0f / 720.0f);
  p = __fmaf_rn(p, r, 1.0f / 120.0f);
  p = __fmaf_rn(p, r, 1.0f / 24.0f);
  p = __fmaf_rn(p, r, 1.0f / 6.0f);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const int k = (int)kf;
  if (k > 127) return __fmul_rn(__fmul_rn(p, 2.0f), __uint_as_float((uint32_t)(127 + 127) << 23));
  if (k >= -126) return __fmul_rn(p, __uint_as_float((uint32_t)(k + 127) << 23));
  return __fmul_rn(__fmul_rn(p, __uint_as_float((uint32_t)(k + 64 + 127) << 23)),
                   __uint_as_float((uint32_t)(127 - 64) << 23));
}

// a = silu(h) * u = (h / (1 + e^-h)) * u, one rounding per operation.
__device__ __forceinline__ float swiglu_ref(float h, float u) {
  const float e = exp_ref(-h);
  const float den = __fadd_rn(1.0f, e);
  return __fmul_rn(__fdiv_rn(h, den), u);
}

// a = silu(h) * u with the hardware exponential and reciprocal: a few fp32 ulp
// from the exactly rounded sequence (swiglu_ref), at a sixth of its instructions.
// The fused forward's a only feeds the per-tensor E4M3 quantizer, whose codes
// can differ only where a lies within those ulps of a rounding midpoint (about
// 2^-18 of the codes, each by one step); the standalone swiglu_quant keeps the
// exact form.  The gate/up GEMM's epilogue (absmax of a) and the cast pass that
// recomputes a from the stored H use this one function, so both see the same a.
// Large negative h: e^-h overflows to inf (or den > 2^126) and the reciprocal
// flushes to 0, so a = -0 * u, as the exact form rounds to.
__device__ __forceinline__ float swiglu_fast(float h, float u) {
  return __fmul_rn(__fdividef(h, __fadd_rn(1.0f, __expf(-h))), u);
}

// --------------------------------------------------------------------------
// Reductions
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) { return __reduce_max_sync(0xFFFFFFFFu, v); }

// Max over the block; result valid in every thread.  blockDim.x multiple of 32, <= 1024.
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* smem32) {
  v = warp_max_u32(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) smem32[warp] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  uint32_t r = lane < nw ? smem32[lane] : 0u;
  r = warp_max_u32(r);
  __syncthreads();
  return r;
}

// Max of P per-block partials (fp32 bit patterns of |v|), read by one warp.
__device__ __forceinline__ float reduce_partials_warp(const uint32_t* __restrict__ partial, int P) {
  uint32_t m = 0;
  for (int i = threadIdx.x & 31; i < P; i += 32) m = max(m, partial[i]);
  return __uint_as_float(warp_max_u32(m));
}

// --------------------------------------------------------------------------
// Global memory access
// --------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ld_v4(const void* p) { return *reinterpret_cast<const uint4*>(p); }
// Requests the L2 lines of the `bytes` bytes at p (bytes > 0, all inside one allocation).
__device__ __forceinline__ void prefetch_l2_span(const void* p, int bytes) {
  const char* c = static_cast<const char*>(p);
  for (int b = 0; b < bytes; b += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(c + b));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(c + bytes - 1));
}
__device__ __forceinline__ void st_v4(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// --------------------------------------------------------------------------
// Timing for bounded waits
// --------------------------------------------------------------------------
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

// --------------------------------------------------------------------------
// mbarrier
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits until the phase with the given parity has completed.  Gives up (returns
// false) after limit_ns or as soon as *abort is set by another role.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
}

// The same wait through the non-suspending probe (mbarrier.test_wait): try_wait may hold the
// thread in the hardware for a system-dependent time before it reports an incomplete phase, so a
// limit shorter than that is honoured only this way (the self-tests that make short waits run out).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_poll(uint64_t* bar, uint32_t parity, volatile int* abort, uint64_t limit_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_test_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// --------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), 2D tiles into shared memory
// --------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_addr(dst)), "l"(tm), "r"(smem_addr(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// --------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads
// --------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem], kind::f8f6f4, one CTA.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same MMA with 16-bit operands (kind::f16; bf16 per the instruction
// descriptor), K = 16 per instruction.  Used by the BF16 baseline and the
// attention core.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Block-scaled MXFP8 MMA (kind::mxf8f6f4.block_scale, one E8M0 scale per 32 elements of K):
// D[tmem] (+)= (A * 2^sfA) (B * 2^sfB) with the scales read from tensor memory at sfa / sfb; the
// instruction descriptor's scale-factor ids pick the byte of each 32-bit scale word (the K block).
__device__ __forceinline__ void umma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}\n"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Scale-factor ids of the instruction descriptor for the kk-th 32-element K block of a 128-byte
// stage: the byte of B's scale word (bits 4-5) and of A's (bits 29-30).
__device__ __forceinline__ uint32_t mx_sf_ids(int kk) { return ((uint32_t)kk << 4) | ((uint32_t)kk << 29); }
// Copy of a 512-byte scale chunk (32 rows of 16 bytes in shared memory) into tensor memory: 4
// columns of 32-bit words at taddr, the same 32 rows in each of the four 32-lane quarters, so that
// quarter q's lane l, column j holds the codes of chunk row 32 j + l.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// Shared-memory descriptor of a scale chunk: no swizzle, 8-row core matrices of 16-byte rows, 128
// bytes apart (the stride between core matrices; one core matrix wide, so the leading offset is
// never stepped).
__device__ __forceinline__ uint64_t smem_desc_sf(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(128 >> 4) << 32) |
         (1ull << 46);
}
// 1D bulk copy global -> shared completing on an mbarrier (both addresses 16-byte aligned, bytes a
// multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}
// Arrive on `bar` once every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}
// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2), sm_100 version bits.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

#define FP8Q_TMEM_LD32_REGS(r)                                                                          \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),       \
      "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),          \
      "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),        \
      "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),        \
      "=r"(r[29]), "=r"(r[30]), "=r"(r[31])

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes
// 32*(w%4)..+31), followed by the wait in the same asm statement so that no use
// of the registers can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FP8Q_TMEM_LD32_REGS(r)
      : "r"(taddr)
      : "memory");
}
// Two 32-column loads (e.g. matching gate and up columns) and one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, uint32_t (&r)[32], uint32_t (&s)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FP8Q_TMEM_LD32_REGS(r), FP8Q_TMEM_LD32_REGS(s)
      : "r"(ta), "r"(tb)
      : "memory");
}

}  // namespace fp8q
