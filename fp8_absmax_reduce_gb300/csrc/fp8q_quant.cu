// HBM-bound kernels of the FP8 block pipeline: per-tensor absmax quantization,
// RMSNorm + quantization, SwiGLU + requantization, RMSNorm backward.
//
// Every quantizer is two passes over its input (LLMQ §4: "dynamic quantization
// adds overhead"; the per-tensor scale needs the whole tensor's absmax before
// the first code can be written):
//   pass 1: 16-byte vector loads, |v| max as fp32 bit patterns (exact and
//           order-independent), warp shuffle + block reduction, one partial
//           per block;
//   pass 2: every block reduces the partials itself (a few KB from L2), derives
//           scale = fmax/amax, and casts with cvt.rn.satfinite to E4M3/E5M2.
// No atomics on floating point, no counters to reset: deterministic and
// re-entrant on one stream.
#include <algorithm>
#include <climits>

#include "fp8q_common.cuh"
#include "fp8q_internal.h"

namespace fp8q {

namespace {

constexpr int kThreads = 256;

inline int grid_for(int64_t items, int cap) {
  int64_t b = (items + kThreads - 1) / kThreads;
  if (b < 1) b = 1;
  return (int)(b < cap ? b : cap);
}

// The grid-stride items i = first, first + stride, ... of a [rows, per_row] item grid as (row, col)
// pairs, without a 64-bit division per item: the stride is split once into whole rows and a
// remainder column step.
struct RowWalk {
  int64_t row, drow;
  int col, dcol, per_row;
  __device__ RowWalk(int64_t first, int64_t stride, int per_row_) : per_row(per_row_) {
    row = first / per_row;
    col = (int)(first - row * per_row);
    drow = stride / per_row;
    dcol = (int)(stride - drow * per_row);
  }
  __device__ void next() {
    row += drow;
    col += dcol;
    if (col >= per_row) {
      col -= per_row;
      ++row;
    }
  }
};

inline cudaError_t post_launch(const Launch& L) {
  if (L.launches) ++*L.launches;
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Pass 1: absmax partials
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ uint32_t vec_absmax(uint4 v) {
  if (DT == 0) {
    return max(max(absmax_bf16x2(v.x), absmax_bf16x2(v.y)), max(absmax_bf16x2(v.z), absmax_bf16x2(v.w)));
  } else {
    return max(max(v.x & 0x7FFFFFFFu, v.y & 0x7FFFFFFFu), max(v.z & 0x7FFFFFFFu, v.w & 0x7FFFFFFFu));
  }
}

template <int DT>
__device__ __forceinline__ uint32_t elem_absbits(const uint8_t* x, int64_t e) {
  if (DT == 0) return ((uint32_t)(reinterpret_cast<const uint16_t*>(x)[e]) & 0x7FFFu) << 16;
  return reinterpret_cast<const uint32_t*>(x)[e] & 0x7FFFFFFFu;
}

// Block `bid` of `nblk` (the kernel's own grid, or a range of blocks of a combined launch).
template <int DT>
__device__ __forceinline__ void absmax_body(const uint8_t* __restrict__ x, int64_t n, uint32_t* __restrict__ partial,
                                            int bid, int nblk, uint32_t* red) {
  constexpr int per = DT == 0 ? 8 : 4;  // elements per 16-byte vector
  const int64_t nvec = n / per;
  const int64_t stride = (int64_t)nblk * blockDim.x;
  int64_t i = (int64_t)bid * blockDim.x + threadIdx.x;
  uint32_t m = 0;
  for (; i + 3 * stride < nvec; i += 4 * stride) {
    const uint4 v0 = ld_nc_v4(x + 16 * i);
    const uint4 v1 = ld_nc_v4(x + 16 * (i + stride));
    const uint4 v2 = ld_nc_v4(x + 16 * (i + 2 * stride));
    const uint4 v3 = ld_nc_v4(x + 16 * (i + 3 * stride));
    m = max(m, max(max(vec_absmax<DT>(v0), vec_absmax<DT>(v1)), max(vec_absmax<DT>(v2), vec_absmax<DT>(v3))));
  }
  for (; i < nvec; i += stride) m = max(m, vec_absmax<DT>(ld_nc_v4(x + 16 * i)));
  if (bid == 0)
    for (int64_t e = nvec * per + threadIdx.x; e < n; e += blockDim.x) m = max(m, elem_absbits<DT>(x, e));
  m = block_max_u32(m, red);
  if (threadIdx.x == 0) partial[bid] = m;
}

template <int DT>
__global__ void __launch_bounds__(kThreads) k_absmax_partial(const uint8_t* __restrict__ x, int64_t n,
                                                             uint32_t* __restrict__ partial) {
  __shared__ uint32_t red[32];
  absmax_body<DT>(x, n, partial, blockIdx.x, gridDim.x, red);
}

// ---------------------------------------------------------------------------
// Pass 2: finalize the scale (every block) and cast
// ---------------------------------------------------------------------------
// Reduces the partials in warp 0 and publishes the scale in shared memory; block 0
// also writes {amax, scale, scale_inv} and flags a non-finite amax.
__device__ __forceinline__ float finalize_scale(const uint32_t* partial, int P, int fmt, float* scal,
                                                unsigned* status, float* s_shared, bool first) {
  if (threadIdx.x < 32) {
    const float amax = reduce_partials_warp(partial, P);
    if (threadIdx.x == 0) {
      float s, si;
      scale_from_amax(amax, fmt, s, si);
      *s_shared = s;
      if (first) {
        scal[0] = amax;
        scal[1] = s;
        scal[2] = si;
        if (!(__float_as_uint(amax) < 0x7F800000u)) atomicOr(status, kStatusNonfinite);
      }
    }
  }
  __syncthreads();
  return *s_shared;
}

template <int DT>
__device__ __forceinline__ void load16(const uint8_t* x, int64_t item, float (&v)[16]) {
  if (DT == 0) {
    const uint4 a = ld_nc_v4(x + 32 * item), b = ld_nc_v4(x + 32 * item + 16);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) { v[2 * k] = bf16_lo(w[k]); v[2 * k + 1] = bf16_hi(w[k]); }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 a = ld_nc_v4(x + 64 * item + 16 * k);
      v[4 * k] = __uint_as_float(a.x); v[4 * k + 1] = __uint_as_float(a.y);
      v[4 * k + 2] = __uint_as_float(a.z); v[4 * k + 3] = __uint_as_float(a.w);
    }
  }
}

template <int FMT>
__device__ __forceinline__ uint4 cast16(const float (&v)[16], float s) {
  uint4 o;
  o.x = cvt_fp8x4<FMT>(__fmul_rn(v[0], s), __fmul_rn(v[1], s), __fmul_rn(v[2], s), __fmul_rn(v[3], s));
  o.y = cvt_fp8x4<FMT>(__fmul_rn(v[4], s), __fmul_rn(v[5], s), __fmul_rn(v[6], s), __fmul_rn(v[7], s));
  o.z = cvt_fp8x4<FMT>(__fmul_rn(v[8], s), __fmul_rn(v[9], s), __fmul_rn(v[10], s), __fmul_rn(v[11], s));
  o.w = cvt_fp8x4<FMT>(__fmul_rn(v[12], s), __fmul_rn(v[13], s), __fmul_rn(v[14], s), __fmul_rn(v[15], s));
  return o;
}

template <int FMT>
__device__ __forceinline__ uint8_t cvt_fp8(float v) {
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, FMT == 0 ? __NV_E4M3 : __NV_E5M2);
}

template <int DT, int FMT>
__device__ __forceinline__ void quant_cast_body(const uint8_t* __restrict__ x, int64_t n,
                                                const uint32_t* __restrict__ partial, int P, uint8_t* __restrict__ q,
                                                float* __restrict__ scal, unsigned* status, int bid, int nblk,
                                                float* s_sh) {
  const float s = finalize_scale(partial, P, FMT, scal, status, s_sh, bid == 0);
  const int64_t items = n / 16;
  const int64_t stride = (int64_t)nblk * blockDim.x;
  for (int64_t i = (int64_t)bid * blockDim.x + threadIdx.x; i < items; i += stride) {
    float v[16];
    load16<DT>(x, i, v);
    st_v4(q + 16 * i, cast16<FMT>(v, s));
  }
  if (bid == 0)
    for (int64_t e = items * 16 + threadIdx.x; e < n; e += blockDim.x) {
      const float v = DT == 0 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(x)[e] << 16)
                              : reinterpret_cast<const float*>(x)[e];
      q[e] = cvt_fp8<FMT>(__fmul_rn(v, s));
    }
}

template <int DT, int FMT>
__global__ void __launch_bounds__(kThreads) k_quant_cast(const uint8_t* __restrict__ x, int64_t n,
                                                         const uint32_t* __restrict__ partial, int P,
                                                         uint8_t* __restrict__ q, float* __restrict__ scal,
                                                         unsigned* status) {
  __shared__ float s_sh;
  quant_cast_body<DT, FMT>(x, n, partial, P, q, scal, status, blockIdx.x, gridDim.x, &s_sh);
}

// ---------------------------------------------------------------------------
// RMSNorm
// ---------------------------------------------------------------------------
// One warp per row.  Lane l holds the squares of x[256c + 8l .. +8) of chunk c.
// The fp32 sum of squares is the pairwise sum of the row (zero-padded to 8192
// terms, which adds exact zeros only): an 8-leaf tree per lane, a butterfly
// across lanes (each level adds adjacent subtrees), then a tree over the 32
// chunk sums.  NC (even, >= the row's 256-element chunks) bounds the chunks:
// the chunks from NC to 32 are all zero, so the tree's additions of a chunk at
// or beyond NC add exact zeros and are left out.
// The kernel is latency-bound (a row's work is one dependent chain per warp),
// so it runs many warps (64 registers a thread) and does two chunks per
// instruction with the packed fp32 operations (__fmul2_rn / __fadd2_rn: each
// half rounds exactly like __fmul_rn / __fadd_rn, so the sums are unchanged).
// The second half of the pass re-reads the row (from L1).
// OUT16 (the BF16 baseline): instead of the absmax partials, the same pass
// writes n = bf16((x rstd) g) -- there is no scale to wait for.
constexpr int kStatsWarps = 8;
// resident blocks per SM: 64 registers a thread up to 16 chunks, more for longer rows
constexpr int stats_blocks_per_sm(int nc) { return nc <= 16 ? 4 : nc <= 24 ? 3 : 2; }

template <bool OUT16, int NC>
__device__ __forceinline__ void rmsnorm_stats_body(const uint16_t* __restrict__ x, const uint16_t* __restrict__ g,
                                                   int64_t T, int d, float eps, float* __restrict__ rstd,
                                                   uint32_t* __restrict__ partial, uint16_t* __restrict__ n16,
                                                   int bid, int nblk, uint32_t* red) {
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)nblk * kStatsWarps;
  uint32_t m = 0;
  for (int64_t row = (int64_t)bid * kStatsWarps + (threadIdx.x >> 5); row < T; row += nw) {
    const uint16_t* xr = x + row * d;
    float cs[NC];
#pragma unroll
    for (int c = 0; c < NC; c += 2) {
      // chunk c in the .x halves, chunk c + 1 in the .y halves
      const int j0 = c * 256 + lane * 8, j1 = j0 + 256;
      const uint4 a = j0 < d ? ld_v4(xr + j0) : make_uint4(0u, 0u, 0u, 0u);
      const uint4 b = j1 < d ? ld_v4(xr + j1) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
      float2 q[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 lo = make_float2(bf16_lo(aw[k]), bf16_lo(bw[k]));
        const float2 hi = make_float2(bf16_hi(aw[k]), bf16_hi(bw[k]));
        q[2 * k] = __fmul2_rn(lo, lo);
        q[2 * k + 1] = __fmul2_rn(hi, hi);
      }
      const float2 t = __fadd2_rn(__fadd2_rn(__fadd2_rn(q[0], q[1]), __fadd2_rn(q[2], q[3])),
                                  __fadd2_rn(__fadd2_rn(q[4], q[5]), __fadd2_rn(q[6], q[7])));
      cs[c] = t.x;
      cs[c + 1] = t.y;
    }
    // (a chunk past the row's end holds zeros, and zero + zero is exact)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1)
#pragma unroll
      for (int c = 0; c < NC; c += 2)
        if (c * 256 < d) {
          const float2 sh = make_float2(__shfl_xor_sync(0xFFFFFFFFu, cs[c], o),
                                        __shfl_xor_sync(0xFFFFFFFFu, cs[c + 1], o));
          const float2 t = __fadd2_rn(make_float2(cs[c], cs[c + 1]), sh);
          cs[c] = t.x;
          cs[c + 1] = t.y;
        }
#pragma unroll
    for (int v = 1; v < 32; v <<= 1)
#pragma unroll
      for (int k = 0; k < 32; k += 2 * v)
        if (k + v < NC) cs[k] = __fadd_rn(cs[k], cs[k + v]);
    const float rs = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(cs[0], (float)d), eps)));
    if (lane == 0) rstd[row] = rs;
    const float2 rs2 = make_float2(rs, rs);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int j0 = c * 256 + lane * 8;
      if (j0 >= d) continue;
      const uint4 gw = ld_v4(g + j0), xv = ld_v4(xr + j0);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, gg[4] = {gw.x, gw.y, gw.z, gw.w};
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 n = __fmul2_rn(__fmul2_rn(make_float2(bf16_lo(xw[k]), bf16_hi(xw[k])), rs2),
                                    make_float2(bf16_lo(gg[k]), bf16_hi(gg[k])));
        if (OUT16) o[k] = pack_bf16x2(n.x, n.y);
        else m = max(m, max(abs_bits(n.x), abs_bits(n.y)));
      }
      if (OUT16) st_v4(n16 + row * d + j0, make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
  if (!OUT16) {
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) partial[bid] = m;
  }
}

template <bool OUT16, int NC>
__global__ void __launch_bounds__(kStatsWarps * 32, stats_blocks_per_sm(NC))
    k_rmsnorm_stats(const uint16_t* __restrict__ x, const uint16_t* __restrict__ g, int64_t T, int d, float eps,
                    float* __restrict__ rstd, uint32_t* __restrict__ partial, uint16_t* __restrict__ n16) {
  __shared__ uint32_t red[32];
  rmsnorm_stats_body<OUT16, NC>(x, g, T, d, eps, rstd, partial, n16, blockIdx.x, gridDim.x, red);
}

// Launches k_rmsnorm_stats with the smallest chunk bound that holds a row of d elements, on a
// grid of at most one wave of resident blocks and at most `cap`; returns the grid size.
template <bool OUT16>
int rmsnorm_stats_dispatch(int64_t T, int d, int64_t cap, const Launch& L, const uint16_t* x, const uint16_t* g,
                           float eps, float* rstd, uint32_t* partial, uint16_t* n16) {
  const int nc = d <= 1024 ? 4 : d <= 2048 ? 8 : d <= 4096 ? 16 : d <= 6144 ? 24 : 32;
  const int64_t blocks = (T + kStatsWarps - 1) / kStatsWarps;
  const int64_t fit = (int64_t)L.num_sms * stats_blocks_per_sm(nc);
  const int grid = (int)std::min<int64_t>(blocks, std::min<int64_t>(fit, cap));
  const int th = kStatsWarps * 32;
  switch (nc) {
    case 4: k_rmsnorm_stats<OUT16, 4><<<grid, th, 0, L.stream>>>(x, g, T, d, eps, rstd, partial, n16); break;
    case 8: k_rmsnorm_stats<OUT16, 8><<<grid, th, 0, L.stream>>>(x, g, T, d, eps, rstd, partial, n16); break;
    case 16: k_rmsnorm_stats<OUT16, 16><<<grid, th, 0, L.stream>>>(x, g, T, d, eps, rstd, partial, n16); break;
    case 24: k_rmsnorm_stats<OUT16, 24><<<grid, th, 0, L.stream>>>(x, g, T, d, eps, rstd, partial, n16); break;
    default: k_rmsnorm_stats<OUT16, 32><<<grid, th, 0, L.stream>>>(x, g, T, d, eps, rstd, partial, n16); break;
  }
  return grid;
}

__device__ __forceinline__ void rmsnorm_cast_body(const uint16_t* __restrict__ x, const uint16_t* __restrict__ g,
                                                  const float* __restrict__ rstd, int64_t T, int d,
                                                  const uint32_t* __restrict__ partial, int P, uint8_t* __restrict__ q,
                                                  float* __restrict__ scal, unsigned* status, int bid, int nblk,
                                                  float* s_sh) {
  const float s = finalize_scale(partial, P, 0, scal, status, s_sh, bid == 0);
  for (RowWalk w((int64_t)bid * blockDim.x + threadIdx.x, (int64_t)nblk * blockDim.x, d / 16); w.row < T;
       w.next()) {
    const int64_t row = w.row;
    const int j0 = w.col * 16;
    const float rs = rstd[row];
    const uint16_t* xr = x + row * d + j0;
    const uint4 a = ld_nc_v4(xr), b = ld_nc_v4(xr + 8), ga = ld_v4(g + j0), gb = ld_v4(g + j0 + 8);
    const uint32_t xw[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const uint32_t gw[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
    float v[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[2 * k] = __fmul_rn(__fmul_rn(bf16_lo(xw[k]), rs), bf16_lo(gw[k]));
      v[2 * k + 1] = __fmul_rn(__fmul_rn(bf16_hi(xw[k]), rs), bf16_hi(gw[k]));
    }
    st_v4(q + row * d + j0, cast16<0>(v, s));
  }
}

__global__ void __launch_bounds__(kThreads) k_rmsnorm_cast(const uint16_t* __restrict__ x,
                                                           const uint16_t* __restrict__ g,
                                                           const float* __restrict__ rstd, int64_t T, int d,
                                                           const uint32_t* __restrict__ partial, int P,
                                                           uint8_t* __restrict__ q, float* __restrict__ scal,
                                                           unsigned* status) {
  __shared__ float s_sh;
  rmsnorm_cast_body(x, g, rstd, T, d, partial, P, q, scal, status, blockIdx.x, gridDim.x, &s_sh);
}

// ---------------------------------------------------------------------------
// The forward's quantizer prologue in two launches instead of six: pass 1 runs the RMSNorm
// statistics of x (its first blocks, one per SM: latency-bound rows) beside the absmax reductions
// of W_gu and W_d (bandwidth-bound), pass 2 the three casts.  The work of every block range is
// exactly that of the separate kernels (the same bodies), so the results are identical.
// ---------------------------------------------------------------------------
struct Prologue {
  const uint16_t* x; const uint16_t* g; int64_t T; int d; float eps; float* rstd;
  uint32_t* part_n; int P_n;            // RMSNorm statistics blocks and partials
  const uint8_t* wgu; int64_t n_wgu; uint32_t* part_wgu; int P_wgu;
  const uint8_t* wd; int64_t n_wd; uint32_t* part_wd; int P_wd;
  uint8_t* n8; float* s_n; int G_n;     // pass 2: casts and their block counts
  uint8_t* wgu8; float* s_wgu; int G_wgu;
  uint8_t* wd8; float* s_wd; int G_wd;
  unsigned* status;
};

template <int NC>
__global__ void __launch_bounds__(kStatsWarps * 32, stats_blocks_per_sm(NC)) k_prologue_stats(const Prologue a) {
  __shared__ uint32_t red[32];
  int b = blockIdx.x;
  if (b < a.P_n) {
    rmsnorm_stats_body<false, NC>(a.x, a.g, a.T, a.d, a.eps, a.rstd, a.part_n, nullptr, b, a.P_n, red);
    return;
  }
  b -= a.P_n;
  if (b < a.P_wgu) {
    absmax_body<0>(a.wgu, a.n_wgu, a.part_wgu, b, a.P_wgu, red);
    return;
  }
  absmax_body<0>(a.wd, a.n_wd, a.part_wd, b - a.P_wgu, a.P_wd, red);
}

__global__ void __launch_bounds__(kThreads) k_prologue_cast(const Prologue a) {
  __shared__ float s_sh;
  int b = blockIdx.x;
  if (b < a.G_wgu) {
    quant_cast_body<0, 0>(a.wgu, a.n_wgu, a.part_wgu, a.P_wgu, a.wgu8, a.s_wgu, a.status, b, a.G_wgu, &s_sh);
    return;
  }
  b -= a.G_wgu;
  if (b < a.G_wd) {
    quant_cast_body<0, 0>(a.wd, a.n_wd, a.part_wd, a.P_wd, a.wd8, a.s_wd, a.status, b, a.G_wd, &s_sh);
    return;
  }
  rmsnorm_cast_body(a.x, a.g, a.rstd, a.T, a.d, a.part_n, a.P_n, a.n8, a.s_n, a.status, b - a.G_wd, a.G_n, &s_sh);
}

// ---------------------------------------------------------------------------
// SwiGLU: a = silu(gate) * up over H [T, 2f]
// ---------------------------------------------------------------------------
// FAST: swiglu_fast (the fused forward), else the exactly rounded swiglu_ref.
template <bool FAST = false>
__device__ __forceinline__ void swiglu8(const uint16_t* H, int64_t row, int f, int j0, float (&a)[8]) {
  const uint16_t* hr = H + row * 2 * (int64_t)f + j0;
  const uint4 gv = ld_nc_v4(hr), uv = ld_nc_v4(hr + f);
  const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (FAST) {
      a[2 * k] = swiglu_fast(bf16_lo(gw[k]), bf16_lo(uw[k]));
      a[2 * k + 1] = swiglu_fast(bf16_hi(gw[k]), bf16_hi(uw[k]));
    } else {
      a[2 * k] = swiglu_ref(bf16_lo(gw[k]), bf16_lo(uw[k]));
      a[2 * k + 1] = swiglu_ref(bf16_hi(gw[k]), bf16_hi(uw[k]));
    }
  }
}

__global__ void __launch_bounds__(kThreads) k_swiglu_amax(const uint16_t* __restrict__ H, int64_t T, int f,
                                                          uint32_t* __restrict__ partial) {
  __shared__ uint32_t red[32];
  uint32_t m = 0;
  for (RowWalk w((int64_t)blockIdx.x * blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x, f / 8); w.row < T;
       w.next()) {
    float a[8];
    swiglu8(H, w.row, f, w.col * 8, a);
#pragma unroll
    for (int k = 0; k < 8; ++k) m = max(m, abs_bits(a[k]));
  }
  m = block_max_u32(m, red);
  if (threadIdx.x == 0) partial[blockIdx.x] = m;
}

template <int FMT, bool FAST>
__global__ void __launch_bounds__(kThreads) k_swiglu_cast(const uint16_t* __restrict__ H, int64_t T, int f,
                                                          const uint32_t* __restrict__ partial, int P,
                                                          uint8_t* __restrict__ q, float* __restrict__ scal,
                                                          unsigned* status) {
  __shared__ float s_sh;
  const float s = finalize_scale(partial, P, FMT, scal, status, &s_sh, blockIdx.x == 0);
  for (RowWalk w((int64_t)blockIdx.x * blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x, f / 8); w.row < T;
       w.next()) {
    const int64_t row = w.row;
    const int j0 = w.col * 8;
    float a[8];
    swiglu8<FAST>(H, row, f, j0, a);
    uint2 o;
    o.x = cvt_fp8x4<FMT>(__fmul_rn(a[0], s), __fmul_rn(a[1], s), __fmul_rn(a[2], s), __fmul_rn(a[3], s));
    o.y = cvt_fp8x4<FMT>(__fmul_rn(a[4], s), __fmul_rn(a[5], s), __fmul_rn(a[6], s), __fmul_rn(a[7], s));
    *reinterpret_cast<uint2*>(q + row * (int64_t)f + j0) = o;
  }
}

// ---------------------------------------------------------------------------
// RMSNorm backward + residual.  A block owns `rows` consecutive rows (one wave
// of resident blocks covers all T rows).  Per row: nh = x rstd, u = dN g,
// dot = sum_j u nh (block reduction, fixed order), dX = dY + rstd (u - nh dot/d).
// dg partials accumulate per block in registers (fixed row order) and are
// reduced over blocks in a fixed order by k_dg_finalize.
// ---------------------------------------------------------------------------
// Rows staged whole in shared memory by the bulk-copy engine: thread t owns the one 8-column group
// j0 = 8 t (the block is ceil(d / 8) threads rounded up to whole warps, at most 1024 for d <= 8192).
// A ring of S row slots, each [dN row (4d B) | x row (2d B) | dY row (2d B)], is filled by
// cp.async.bulk copies that one thread issues up to S rows ahead, completing on the slot's
// mbarrier: the bytes in flight per SM are set by the ring, not by registers, and the block's
// threads issue no load instructions for their inputs.  A thread takes its 8 values of each piece
// into registers before the row's block barrier, so once every thread has passed that barrier the
// slot is free and the issuing thread refills it with row rr + S.
// Every wait is bounded; a thread whose wait expires flags its warp's entry of the row's reduction,
// every thread sees the flag after the same barrier and leaves the loop, and the issuing thread
// waits (again bounded) for the copies it still has in flight before the block exits.
constexpr int kBwdSlotsMax = 8;
constexpr int kBwdSmemBudget = 200 * 1024;  // per SM, shared by its resident blocks

inline int bwd_tma_threads(int d) { return ((d / 8 + 31) / 32) * 32; }
// Two blocks per SM (two independent row chains) where their threads' registers (at most 64
// each) and two rings of three row slots fit, else one.
inline int bwd_tma_blocks_per_sm(int d) {
  return bwd_tma_threads(d) <= 512 && 2 * 3 * (size_t)8 * d <= (size_t)kBwdSmemBudget ? 2 : 1;
}

// POLL: the waits probe without suspending (mbar_poll), for the self-test of the abort sequence.
template <bool POLL>
__global__ void __launch_bounds__(1024, 1) k_rmsnorm_bwd_tma(const float* __restrict__ dN,
                                                              const uint16_t* __restrict__ x,
                                                              const uint16_t* __restrict__ dY,
                                                              const uint16_t* __restrict__ g,
                                                              const float* __restrict__ rstd, int64_t T, int d,
                                                              int rows, int S, uint16_t* __restrict__ dX,
                                                              float* __restrict__ dg_partial, unsigned* status,
                                                              uint64_t wait_ns) {
  extern __shared__ __align__(128) uint8_t bwd_rows[];  // S slots of 8 d bytes
  __shared__ uint64_t full[kBwdSlotsMax];
  __shared__ float red[2][32];
  __shared__ int bad[2][32];
  __shared__ volatile int give_up;  // lets the other waiting threads stop early once one wait has expired
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nwarps = blockDim.x >> 5;
  const int j0 = 8 * t;
  const bool mine = j0 < d;
  const int64_t r0 = (int64_t)blockIdx.x * rows;
  const int nrows = (int)((T - r0) < rows ? (T - r0) : rows);
  const uint32_t slot_bytes = 8u * (uint32_t)d;
  if (t == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    give_up = 0;
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int rr) {  // thread 0 only
    const int s = rr % S;
    const int64_t row = r0 + rr;
    uint8_t* slot = bwd_rows + (size_t)s * slot_bytes;
    mbar_arrive_expect_tx(&full[s], slot_bytes);
    bulk_load(slot, dN + row * d, 4u * d, &full[s]);
    bulk_load(slot + 4 * d, x + row * d, 2u * d, &full[s]);
    bulk_load(slot + 6 * d, dY + row * d, 2u * d, &full[s]);
  };
  if (t == 0)
    for (int k = 0; k < S && k < nrows; ++k) issue(k);
  float gv[8], dga[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) { gv[k] = 0.0f; dga[k] = 0.0f; }
  if (mine) {
    const uint4 w = ld_v4(g + j0);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) { gv[2 * k] = bf16_lo(ww[k]); gv[2 * k + 1] = bf16_hi(ww[k]); }
  }
  const float inv_d = 1.0f / (float)d;
  int rr = 0;
  bool aborted = false;
  float rs_next = rstd[r0];  // a row's rstd is requested one row ahead, off the row's critical path
  for (; rr < nrows; ++rr) {
    const int s = rr % S;
    const float rs = rs_next;
    if (rr + 1 < nrows) rs_next = rstd[r0 + rr + 1];
    const uint32_t par = (uint32_t)(rr / S) & 1u;
    const bool ok = POLL ? mbar_poll(&full[s], par, &give_up, wait_ns) : mbar_wait(&full[s], par, &give_up, wait_ns);
    if (!ok) give_up = 1;
    const uint8_t* slot = bwd_rows + (size_t)s * slot_bytes;
    const int64_t row = r0 + rr;
    float dnv[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    uint32_t xw[4] = {0u, 0u, 0u, 0u}, yw[4] = {0u, 0u, 0u, 0u};
    float dot = 0.0f;
    if (mine) {
      const uint4 d0 = *reinterpret_cast<const uint4*>(slot + 4 * j0);
      const uint4 d1 = *reinterpret_cast<const uint4*>(slot + 4 * j0 + 16);
      const uint4 xv = *reinterpret_cast<const uint4*>(slot + 4 * d + 2 * j0);
      const uint4 yv = *reinterpret_cast<const uint4*>(slot + 6 * d + 2 * j0);
      dnv[0] = __uint_as_float(d0.x); dnv[1] = __uint_as_float(d0.y);
      dnv[2] = __uint_as_float(d0.z); dnv[3] = __uint_as_float(d0.w);
      dnv[4] = __uint_as_float(d1.x); dnv[5] = __uint_as_float(d1.y);
      dnv[6] = __uint_as_float(d1.z); dnv[7] = __uint_as_float(d1.w);
      xw[0] = xv.x; xw[1] = xv.y; xw[2] = xv.z; xw[3] = xv.w;
      yw[0] = yv.x; yw[1] = yv.y; yw[2] = yv.z; yw[3] = yv.w;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float nh = ((k & 1) ? bf16_hi(xw[k >> 1]) : bf16_lo(xw[k >> 1])) * rs;
        dot += (dnv[k] * gv[k]) * nh;
        dga[k] += dnv[k] * nh;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, o);
    const int warp_bad = __any_sync(0xFFFFFFFFu, !ok);
    if (lane == 0) {
      red[rr & 1][warp] = dot;
      bad[rr & 1][warp] = warp_bad;
    }
    __syncthreads();
    // every warp sums the per-warp partials itself: lane w takes warp w's, then a butterfly (the
    // same tree in every warp, so every thread holds the same total)
    float tot = lane < nwarps ? red[rr & 1][lane] : 0.0f;
    const int any_bad = __any_sync(0xFFFFFFFFu, lane < nwarps && bad[rr & 1][lane] != 0);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
    if (any_bad) {
      aborted = true;
      break;
    }
    // every thread has its values of row rr in registers: the slot takes row rr + S
    if (t == 0 && rr + S < nrows) issue(rr + S);
    const float mean = tot * inv_d;
    if (mine) {
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float nlo = bf16_lo(xw[k]) * rs, nhi = bf16_hi(xw[k]) * rs;
        const float a = bf16_lo(yw[k]) + rs * (dnv[2 * k] * gv[2 * k] - nlo * mean);
        const float b = bf16_hi(yw[k]) + rs * (dnv[2 * k + 1] * gv[2 * k + 1] - nhi * mean);
        o[k] = pack_bf16x2(a, b);
      }
      st_v4(dX + row * d + j0, make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
  if (aborted) {
    if (t == 0) {
      atomicOr(status, kStatusTimeout);
      // rows rr .. rr + S - 1 may still have copies in flight into this block's ring
      volatile int never = 0;
      for (int k = rr; k < rr + S && k < nrows; ++k)
        mbar_wait(&full[k % S], (uint32_t)(k / S) & 1u, &never);
    }
    return;
  }
  if (mine) {
    float* dst = dg_partial + (int64_t)blockIdx.x * d + j0;
    st_v4(dst, make_uint4(__float_as_uint(dga[0]), __float_as_uint(dga[1]), __float_as_uint(dga[2]),
                          __float_as_uint(dga[3])));
    st_v4(dst + 4, make_uint4(__float_as_uint(dga[4]), __float_as_uint(dga[5]), __float_as_uint(dga[6]),
                              __float_as_uint(dga[7])));
  }
}

// dg[j] = sum over the nblk partial rows, in a fixed order: a block owns 32 columns; thread
// (ty, tx) sums rows ty, ty + 32, ... of column j0 + tx (independent loads, several in flight per
// thread), then the 32 partial sums of a column are added in a fixed tree over ty.
constexpr int kFinRows = 32;

__global__ void __launch_bounds__(32 * kFinRows) k_dg_finalize(const float* __restrict__ dg_partial, int nblk,
                                                               int d, float* __restrict__ dg) {
  __shared__ float part[kFinRows][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int j = blockIdx.x * 32 + tx;
  float s = 0.0f;
  if (j < d) {
#pragma unroll 4
    for (int b = ty; b < nblk; b += kFinRows) s += dg_partial[(int64_t)b * d + j];
  }
  part[ty][tx] = s;
  __syncthreads();
#pragma unroll
  for (int w = kFinRows / 2; w > 0; w >>= 1) {
    if (ty < w) part[ty][tx] += part[ty + w][tx];
    __syncthreads();
  }
  if (ty == 0 && j < d) dg[j] = part[0][tx];
}

// One thread waits on an mbarrier that nothing ever arrives at, through the
// same bounded wait the GEMM uses, and reports the expiry in the status word.
__global__ void k_selftest_bounded_wait(unsigned* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int never;
  mbar_init(&bar, 1);
  never = 0;
  fence_mbar_init();
  if (!mbar_wait(&bar, 0, &never, limit_ns)) atomicOr(status, kStatusTimeout);
}

}  // namespace

cudaError_t launch_selftest_bounded_wait(uint64_t limit_ns, const Launch& L) {
  k_selftest_bounded_wait<<<1, 1, 0, L.stream>>>(L.status, limit_ns);
  return post_launch(L);
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
int absmax_partial_blocks(int dtype, int64_t n) {
  const int64_t nvec = dtype == 0 ? n / 8 : n / 4;
  return grid_for(nvec / 4 > 0 ? nvec / 4 : 1, kMaxPartials);
}

cudaError_t launch_absmax_partial(const void* x, int dtype, int64_t n, uint32_t* partial, int* P,
                                  const Launch& L) {
  const int grid = absmax_partial_blocks(dtype, n);
  *P = grid;
  if (dtype == 0)
    k_absmax_partial<0><<<grid, kThreads, 0, L.stream>>>((const uint8_t*)x, n, partial);
  else
    k_absmax_partial<1><<<grid, kThreads, 0, L.stream>>>((const uint8_t*)x, n, partial);
  return post_launch(L);
}

cudaError_t launch_quant_cast(const void* x, int dtype, int64_t n, int fmt, const uint32_t* partial, int P,
                              uint8_t* q, float* scal, const Launch& L) {
  const int grid = grid_for(n / 16 > 0 ? n / 16 : 1, L.num_sms * 8);
  const uint8_t* xb = (const uint8_t*)x;
  if (dtype == 0 && fmt == 0)
    k_quant_cast<0, 0><<<grid, kThreads, 0, L.stream>>>(xb, n, partial, P, q, scal, L.status);
  else if (dtype == 0)
    k_quant_cast<0, 1><<<grid, kThreads, 0, L.stream>>>(xb, n, partial, P, q, scal, L.status);
  else if (fmt == 0)
    k_quant_cast<1, 0><<<grid, kThreads, 0, L.stream>>>(xb, n, partial, P, q, scal, L.status);
  else
    k_quant_cast<1, 1><<<grid, kThreads, 0, L.stream>>>(xb, n, partial, P, q, scal, L.status);
  return post_launch(L);
}

cudaError_t launch_rmsnorm_stats(const uint16_t* x, const uint16_t* g, int64_t T, int d, float eps, float* rstd,
                                 uint32_t* partial, int* P, const Launch& L) {
  // one wave of resident blocks, each warp looping over rows; one absmax partial per block
  const int grid = rmsnorm_stats_dispatch<false>(T, d, kMaxPartials, L, x, g, eps, rstd, partial, nullptr);
  if (grid < 1) return cudaErrorInvalidConfiguration;
  *P = grid;
  return post_launch(L);
}

cudaError_t launch_prologue(int pass, const uint16_t* x, const uint16_t* g, int64_t T, int d, float eps, float* rstd,
                            const uint16_t* W_gu, int64_t n_wgu, const uint16_t* W_d, int64_t n_wd,
                            uint32_t* part_n, uint32_t* part_wgu, uint32_t* part_wd, uint8_t* n8, float* s_n,
                            uint8_t* W_gu8, float* s_wgu, uint8_t* W_d8, float* s_wd, const Launch& L) {
  Prologue a{};
  a.x = x; a.g = g; a.T = T; a.d = d; a.eps = eps; a.rstd = rstd;
  a.part_n = part_n;
  // The statistics blocks are latency-bound (a warp's row is one long dependent chain) while the
  // weight reductions stream: one statistics block per SM leaves the other slots to the weights,
  // unless x is at least a third of the launch's bytes, when the statistics take every slot
  // (measured on the 32B block: the attention side's prologue 143 -> 83 us, the MLP side's and the
  // 7B block's slower with more than one).
  const int nc = d <= 1024 ? 4 : d <= 2048 ? 8 : d <= 4096 ? 16 : d <= 6144 ? 24 : 32;
  const bool x_heavy = 3 * T * (int64_t)d >= T * (int64_t)d + n_wgu + n_wd;
  const int64_t stats_slots = (int64_t)L.num_sms * (x_heavy ? stats_blocks_per_sm(nc) : 1);
  a.P_n = (int)std::min<int64_t>(std::min<int64_t>(stats_slots, kMaxPartials), (T + kStatsWarps - 1) / kStatsWarps);
  a.wgu = (const uint8_t*)W_gu; a.n_wgu = n_wgu; a.part_wgu = part_wgu; a.P_wgu = absmax_partial_blocks(0, n_wgu);
  a.wd = (const uint8_t*)W_d; a.n_wd = n_wd; a.part_wd = part_wd; a.P_wd = absmax_partial_blocks(0, n_wd);
  a.n8 = n8; a.s_n = s_n; a.G_n = grid_for(T * (d / 16), L.num_sms * 8);
  a.wgu8 = W_gu8; a.s_wgu = s_wgu; a.G_wgu = grid_for(n_wgu / 16 > 0 ? n_wgu / 16 : 1, L.num_sms * 8);
  a.wd8 = W_d8; a.s_wd = s_wd; a.G_wd = grid_for(n_wd / 16 > 0 ? n_wd / 16 : 1, L.num_sms * 8);
  a.status = L.status;
  if (pass == 2) {
    k_prologue_cast<<<a.G_wgu + a.G_wd + a.G_n, kThreads, 0, L.stream>>>(a);
    return post_launch(L);
  }
  const int g1 = a.P_n + a.P_wgu + a.P_wd, th = kStatsWarps * 32;
  switch (nc) {
    case 4: k_prologue_stats<4><<<g1, th, 0, L.stream>>>(a); break;
    case 8: k_prologue_stats<8><<<g1, th, 0, L.stream>>>(a); break;
    case 16: k_prologue_stats<16><<<g1, th, 0, L.stream>>>(a); break;
    case 24: k_prologue_stats<24><<<g1, th, 0, L.stream>>>(a); break;
    default: k_prologue_stats<32><<<g1, th, 0, L.stream>>>(a); break;
  }
  return post_launch(L);
}

cudaError_t launch_rmsnorm_bf16(const uint16_t* x, const uint16_t* g, int64_t T, int d, float eps, float* rstd,
                                uint16_t* n16, const Launch& L) {
  if (rmsnorm_stats_dispatch<true>(T, d, INT32_MAX, L, x, g, eps, rstd, nullptr, n16) < 1)
    return cudaErrorInvalidConfiguration;
  return post_launch(L);
}

cudaError_t launch_rmsnorm_cast(const uint16_t* x, const uint16_t* g, const float* rstd, int64_t T, int d,
                                const uint32_t* partial, int P, uint8_t* q, float* scal, const Launch& L) {
  const int grid = grid_for(T * (d / 16), L.num_sms * 8);
  k_rmsnorm_cast<<<grid, kThreads, 0, L.stream>>>(x, g, rstd, T, d, partial, P, q, scal, L.status);
  return post_launch(L);
}

cudaError_t launch_swiglu_amax(const uint16_t* H, int64_t T, int f, uint32_t* partial, int* P, const Launch& L) {
  const int grid = grid_for(T * (f / 8), kMaxPartials);
  *P = grid;
  k_swiglu_amax<<<grid, kThreads, 0, L.stream>>>(H, T, f, partial);
  return post_launch(L);
}

cudaError_t launch_swiglu_cast(const uint16_t* H, int64_t T, int f, int fmt, const uint32_t* partial, int P,
                               uint8_t* q, float* scal, const Launch& L, bool fast) {
  const int grid = grid_for(T * (f / 8), L.num_sms * 8);
  if (fast)
    k_swiglu_cast<0, true><<<grid, kThreads, 0, L.stream>>>(H, T, f, partial, P, q, scal, L.status);
  else if (fmt == 0)
    k_swiglu_cast<0, false><<<grid, kThreads, 0, L.stream>>>(H, T, f, partial, P, q, scal, L.status);
  else
    k_swiglu_cast<1, false><<<grid, kThreads, 0, L.stream>>>(H, T, f, partial, P, q, scal, L.status);
  return post_launch(L);
}

cudaError_t launch_rmsnorm_bwd(const float* dN, const uint16_t* x, const uint16_t* dY, const uint16_t* g,
                               const float* rstd, int64_t T, int d, uint16_t* dX, float* dg_partial, float* dg,
                               const Launch& L, uint64_t wait_ns) {
  // one wave of resident blocks, consecutive rows each (at least kBwdRows: the dg partials'
  // workspace holds ceil(T / kBwdRows) rows); a block's ring takes as many row slots as its share
  // of the budget holds
  const size_t slot = (size_t)8 * d;
  const int bps = bwd_tma_blocks_per_sm(d);
  const int S = (int)std::min<size_t>(kBwdSlotsMax, kBwdSmemBudget / bps / slot);
  if (S < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)S * slot;
  const int64_t wave = (int64_t)L.num_sms * bps;
  const int rows = (int)std::max<int64_t>(kBwdRows, (T + wave - 1) / wave);
  const int nblk = (int)((T + rows - 1) / rows);
  static int configured_device[2] = {-1, -1};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool poll = wait_ns != 0;  // the self-test's short limits
  const void* fn = poll ? (const void*)k_rmsnorm_bwd_tma<true> : (const void*)k_rmsnorm_bwd_tma<false>;
  if (configured_device[poll] != dev) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmemBudget);
    if (e != cudaSuccess) return e;
    configured_device[poll] = dev;
  }
  if (poll)
    k_rmsnorm_bwd_tma<true><<<nblk, bwd_tma_threads(d), smem, L.stream>>>(dN, x, dY, g, rstd, T, d, rows, S, dX,
                                                                          dg_partial, L.status, wait_ns);
  else
    k_rmsnorm_bwd_tma<false><<<nblk, bwd_tma_threads(d), smem, L.stream>>>(dN, x, dY, g, rstd, T, d, rows, S, dX,
                                                                           dg_partial, L.status, kWaitLimitNs);
  cudaError_t e = post_launch(L);
  if (e != cudaSuccess) return e;
  k_dg_finalize<<<(d + 31) / 32, 32 * kFinRows, 0, L.stream>>>(dg_partial, nblk, d, dg);
  return post_launch(L);
}

}  // namespace fp8q
