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
// of resident blocks covers all T rows); thread t owns the 8-column groups
// j = 8 (t + 256 c), c < NG.  Per row: nh = x rstd, u = dN g,
// dot = sum_j u nh (block reduction, fixed order), dX = dY + rstd (u - nh dot/d).
// A row's dN, x and dY reach shared memory through a ring of kBwdRing slots
// filled by asynchronous 16-byte copies, kBwdRing - 1 rows ahead of their use
// (one row of prefetch cannot cover the DRAM latency behind a row's short
// dependent chain); each thread copies and reads back only its own pieces, so
// the ring needs no barrier beyond the thread's cp.async.wait_group.
// dg partials accumulate per block in registers (fixed row order) and are
// reduced over blocks in a fixed order by k_dg_finalize.
// ---------------------------------------------------------------------------
// Rows of up to 4096 columns (at most two 8-column groups per thread): the next row's dN and x
// in registers while the current one is reduced, two blocks per SM -- at these sizes this
// measured faster than the shared-memory ring below, which wins for longer rows.
template <int NG>
struct BwdRow {
  uint4 d0[NG], d1[NG], xv[NG], yv[NG];
};

template <int NG>
__device__ __forceinline__ void bwd_load_row(BwdRow<NG>& r, const float* __restrict__ dN,
                                             const uint16_t* __restrict__ x, const uint16_t* __restrict__ dY,
                                             int64_t row, int d, int t) {
#pragma unroll
  for (int c = 0; c < NG; ++c) {
    const int j0 = 8 * (t + kThreads * c);
    if (j0 < d) {
      const float* dn = dN + row * d + j0;
      r.d0[c] = ld_nc_v4(dn);
      r.d1[c] = ld_nc_v4(dn + 4);
      r.xv[c] = ld_nc_v4(x + row * d + j0);
      r.yv[c] = ld_nc_v4(dY + row * d + j0);
    } else {
      r.d0[c] = r.d1[c] = r.xv[c] = r.yv[c] = make_uint4(0, 0, 0, 0);
    }
  }
}

template <int NG>
__global__ void __launch_bounds__(kThreads) k_rmsnorm_bwd_reg(const float* __restrict__ dN,
                                                          const uint16_t* __restrict__ x,
                                                          const uint16_t* __restrict__ dY,
                                                          const uint16_t* __restrict__ g,
                                                          const float* __restrict__ rstd, int64_t T, int d,
                                                          int rows, uint16_t* __restrict__ dX,
                                                          float* __restrict__ dg_partial) {
  __shared__ float red[2][kThreads / 32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  float gv[NG][8], dga[NG][8];
#pragma unroll
  for (int c = 0; c < NG; ++c) {
    const int j0 = 8 * (t + kThreads * c);
#pragma unroll
    for (int k = 0; k < 8; ++k) { gv[c][k] = 0.0f; dga[c][k] = 0.0f; }
    if (j0 < d) {
      const uint4 w = ld_v4(g + j0);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) { gv[c][2 * k] = bf16_lo(ww[k]); gv[c][2 * k + 1] = bf16_hi(ww[k]); }
    }
  }
  const float inv_d = 1.0f / (float)d;
  const int64_t r0 = (int64_t)blockIdx.x * rows;
  const int nrows = (int)((T - r0) < rows ? (T - r0) : rows);
  BwdRow<NG> cur;
  bwd_load_row<NG>(cur, dN, x, dY, r0, d, t);
  for (int rr = 0; rr < nrows; ++rr) {
    const int64_t row = r0 + rr;
    BwdRow<NG> nxt;
    if (rr + 1 < nrows) bwd_load_row<NG>(nxt, dN, x, dY, row + 1, d, t);
    const uint4* yv = cur.yv;
    const float rs = rstd[row];
    float nh[NG][8], u[NG][8];
    float dot = 0.0f;
#pragma unroll
    for (int c = 0; c < NG; ++c) {
      const float dnv[8] = {__uint_as_float(cur.d0[c].x), __uint_as_float(cur.d0[c].y),
                            __uint_as_float(cur.d0[c].z), __uint_as_float(cur.d0[c].w),
                            __uint_as_float(cur.d1[c].x), __uint_as_float(cur.d1[c].y),
                            __uint_as_float(cur.d1[c].z), __uint_as_float(cur.d1[c].w)};
      const uint32_t xw[4] = {cur.xv[c].x, cur.xv[c].y, cur.xv[c].z, cur.xv[c].w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float xk = (k & 1) ? bf16_hi(xw[k >> 1]) : bf16_lo(xw[k >> 1]);
        nh[c][k] = xk * rs;
        u[c][k] = dnv[k] * gv[c][k];
        dot += u[c][k] * nh[c][k];
        dga[c][k] += dnv[k] * nh[c][k];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, o);
    if (lane == 0) red[rr & 1][warp] = dot;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) tot += red[rr & 1][w];
    const float mean = tot * inv_d;
#pragma unroll
    for (int c = 0; c < NG; ++c) {
      const int j0 = 8 * (t + kThreads * c);
      if (j0 < d) {
        const uint32_t yw[4] = {yv[c].x, yv[c].y, yv[c].z, yv[c].w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float a = bf16_lo(yw[k]) + rs * (u[c][2 * k] - nh[c][2 * k] * mean);
          const float b = bf16_hi(yw[k]) + rs * (u[c][2 * k + 1] - nh[c][2 * k + 1] * mean);
          o[k] = pack_bf16x2(a, b);
        }
        st_v4(dX + row * d + j0, make_uint4(o[0], o[1], o[2], o[3]));
      }
    }
    if (rr + 1 < nrows) cur = nxt;
  }
#pragma unroll
  for (int c = 0; c < NG; ++c) {
    const int j0 = 8 * (t + kThreads * c);
    if (j0 < d) {
      float* dst = dg_partial + (int64_t)blockIdx.x * d + j0;
      st_v4(dst, make_uint4(__float_as_uint(dga[c][0]), __float_as_uint(dga[c][1]), __float_as_uint(dga[c][2]),
                            __float_as_uint(dga[c][3])));
      st_v4(dst + 4, make_uint4(__float_as_uint(dga[c][4]), __float_as_uint(dga[c][5]),
                                __float_as_uint(dga[c][6]), __float_as_uint(dga[c][7])));
    }
  }
}

constexpr int kBwdRing = 3;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Shared memory of one k_rmsnorm_bwd block: kBwdRing slots of NG x 4 pieces (dN lo, dN hi, x, dY)
// of 16 bytes per thread.
inline size_t rmsnorm_bwd_smem(int ng) { return (size_t)kBwdRing * ng * 4 * kThreads * 16; }

template <int NG>
__global__ void __launch_bounds__(kThreads, 2) k_rmsnorm_bwd(const float* __restrict__ dN,
                                                             const uint16_t* __restrict__ x,
                                                             const uint16_t* __restrict__ dY,
                                                             const uint16_t* __restrict__ g,
                                                             const float* __restrict__ rstd, int64_t T, int d,
                                                             int rows, uint16_t* __restrict__ dX,
                                                             float* __restrict__ dg_partial) {
  extern __shared__ uint4 bwd_ring[];  // [slot][group][piece][thread]
  __shared__ float red[2][kThreads / 32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  float gv[NG][8], dga[NG][8];
#pragma unroll
  for (int c = 0; c < NG; ++c) {
    const int j0 = 8 * (t + kThreads * c);
#pragma unroll
    for (int k = 0; k < 8; ++k) { gv[c][k] = 0.0f; dga[c][k] = 0.0f; }
    if (j0 < d) {
      const uint4 w = ld_v4(g + j0);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) { gv[c][2 * k] = bf16_lo(ww[k]); gv[c][2 * k + 1] = bf16_hi(ww[k]); }
    }
  }
  const float inv_d = 1.0f / (float)d;
  const int64_t r0 = (int64_t)blockIdx.x * rows;
  const int nrows = (int)((T - r0) < rows ? (T - r0) : rows);
  const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(bwd_ring);
  // piece q of group c of slot sl, this thread's 16 bytes
  auto piece = [&](int sl, int c, int q) { return ((sl * NG + c) * 4 + q) * kThreads + t; };
  auto issue = [&](int rr) {
    if (rr < nrows) {
      const int64_t row = r0 + rr;
      const int sl = rr % kBwdRing;
#pragma unroll
      for (int c = 0; c < NG; ++c) {
        const int j0 = 8 * (t + kThreads * c);
        if (j0 < d) {
          const float* dn = dN + row * d + j0;
          cp_async16(ring_s + 16u * piece(sl, c, 0), dn);
          cp_async16(ring_s + 16u * piece(sl, c, 1), dn + 4);
          cp_async16(ring_s + 16u * piece(sl, c, 2), x + row * d + j0);
          cp_async16(ring_s + 16u * piece(sl, c, 3), dY + row * d + j0);
        }
      }
    }
    cp_async_commit();  // an empty group keeps the group count uniform
  };
#pragma unroll
  for (int k = 0; k < kBwdRing - 1; ++k) issue(k);
  for (int rr = 0; rr < nrows; ++rr) {
    const int64_t row = r0 + rr;
    issue(rr + kBwdRing - 1);
    cp_async_wait<kBwdRing - 1>();  // this thread's pieces of row rr have landed
    const int sl = rr % kBwdRing;
    const float rs = rstd[row];
    float dot = 0.0f;
#pragma unroll
    for (int c = 0; c < NG; ++c) {
      const int j0 = 8 * (t + kThreads * c);
      if (j0 >= d) continue;
      const uint4 d0 = bwd_ring[piece(sl, c, 0)], d1 = bwd_ring[piece(sl, c, 1)], xv = bwd_ring[piece(sl, c, 2)];
      const float dnv[8] = {__uint_as_float(d0.x), __uint_as_float(d0.y), __uint_as_float(d0.z), __uint_as_float(d0.w),
                            __uint_as_float(d1.x), __uint_as_float(d1.y), __uint_as_float(d1.z), __uint_as_float(d1.w)};
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float xk = (k & 1) ? bf16_hi(xw[k >> 1]) : bf16_lo(xw[k >> 1]);
        const float nh = xk * rs;
        dot += (dnv[k] * gv[c][k]) * nh;
        dga[c][k] += dnv[k] * nh;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, o);
    if (lane == 0) red[rr & 1][warp] = dot;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) tot += red[rr & 1][w];
    const float mean = tot * inv_d;
#pragma unroll
    for (int c = 0; c < NG; ++c) {
      const int j0 = 8 * (t + kThreads * c);
      if (j0 >= d) continue;
      const uint4 d0 = bwd_ring[piece(sl, c, 0)], d1 = bwd_ring[piece(sl, c, 1)], xv = bwd_ring[piece(sl, c, 2)],
                  yv = bwd_ring[piece(sl, c, 3)];
      const float dnv[8] = {__uint_as_float(d0.x), __uint_as_float(d0.y), __uint_as_float(d0.z), __uint_as_float(d0.w),
                            __uint_as_float(d1.x), __uint_as_float(d1.y), __uint_as_float(d1.z), __uint_as_float(d1.w)};
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, yw[4] = {yv.x, yv.y, yv.z, yv.w};
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float nlo = bf16_lo(xw[k]) * rs, nhi = bf16_hi(xw[k]) * rs;
        const float a = bf16_lo(yw[k]) + rs * (dnv[2 * k] * gv[c][2 * k] - nlo * mean);
        const float bb = bf16_hi(yw[k]) + rs * (dnv[2 * k + 1] * gv[c][2 * k + 1] - nhi * mean);
        o[k] = pack_bf16x2(a, bb);
      }
      st_v4(dX + row * d + j0, make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
  cp_async_wait<0>();
#pragma unroll
  for (int c = 0; c < NG; ++c) {
    const int j0 = 8 * (t + kThreads * c);
    if (j0 < d) {
      float* dst = dg_partial + (int64_t)blockIdx.x * d + j0;
      st_v4(dst, make_uint4(__float_as_uint(dga[c][0]), __float_as_uint(dga[c][1]), __float_as_uint(dga[c][2]),
                            __float_as_uint(dga[c][3])));
      st_v4(dst + 4, make_uint4(__float_as_uint(dga[c][4]), __float_as_uint(dga[c][5]),
                                __float_as_uint(dga[c][6]), __float_as_uint(dga[c][7])));
    }
  }
}

// dg[j] = sum over the nblk partial rows, in a fixed order: a block owns 32 columns;
// thread (ty, tx) sums rows ty, ty+8, ... of column j0+tx, then the 8 partial sums
// are added in ty order.
__global__ void __launch_bounds__(kThreads) k_dg_finalize(const float* __restrict__ dg_partial, int nblk, int d,
                                                          float* __restrict__ dg) {
  __shared__ float part[8][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int j = blockIdx.x * 32 + tx;
  float s = 0.0f;
  if (j < d)
    for (int b = ty; b < nblk; b += 8) s += dg_partial[(int64_t)b * d + j];
  part[ty][tx] = s;
  __syncthreads();
  if (ty == 0 && j < d) {
    float tot = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) tot += part[k][tx];
    dg[j] = tot;
  }
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
  a.P_n = (int)std::min<int64_t>(L.num_sms, (T + kStatsWarps - 1) / kStatsWarps);
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
  const int nc = d <= 1024 ? 4 : d <= 2048 ? 8 : d <= 4096 ? 16 : d <= 6144 ? 24 : 32;
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
                               const Launch& L) {
  const int ng = (d + 8 * kThreads - 1) / (8 * kThreads);
  if (ng <= 2) {
    int per_sm = 0;
    const void* fn = ng == 1 ? (const void*)k_rmsnorm_bwd_reg<1> : (const void*)k_rmsnorm_bwd_reg<2>;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, 0) != cudaSuccess || per_sm < 1)
      per_sm = 1;
    const int64_t wave = (int64_t)L.num_sms * per_sm;
    const int rows = (int)std::max<int64_t>(kBwdRows, (T + wave - 1) / wave);
    const int nblk = (int)((T + rows - 1) / rows);
    if (ng == 1) k_rmsnorm_bwd_reg<1><<<nblk, kThreads, 0, L.stream>>>(dN, x, dY, g, rstd, T, d, rows, dX, dg_partial);
    else k_rmsnorm_bwd_reg<2><<<nblk, kThreads, 0, L.stream>>>(dN, x, dY, g, rstd, T, d, rows, dX, dg_partial);
    cudaError_t e = post_launch(L);
    if (e != cudaSuccess) return e;
    k_dg_finalize<<<(d + 31) / 32, kThreads, 0, L.stream>>>(dg_partial, nblk, d, dg);
    return post_launch(L);
  }
  const size_t smem = rmsnorm_bwd_smem(ng <= 4 ? ng : 4);
  // one wave of resident blocks (two per SM when their rings fit), consecutive rows each (at least
  // kBwdRows: the dg partials' workspace holds ceil(T / kBwdRows) rows)
  const int64_t wave = (int64_t)L.num_sms * (smem <= 110 * 1024 ? 2 : 1);
  const int rows = (int)std::max<int64_t>(kBwdRows, (T + wave - 1) / wave);
  const int nblk = (int)((T + rows - 1) / rows);
  static int configured_device[5] = {-1, -1, -1, -1, -1};
  int dev = 0;
  cudaGetDevice(&dev);
  auto go = [&](auto kernel, int which) -> cudaError_t {
    if (configured_device[which] != dev) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      configured_device[which] = dev;
    }
    kernel<<<nblk, kThreads, smem, L.stream>>>(dN, x, dY, g, rstd, T, d, rows, dX, dg_partial);
    return cudaSuccess;
  };
  cudaError_t le;
  switch (ng) {
    case 3: le = go(k_rmsnorm_bwd<3>, 3); break;
    default: le = go(k_rmsnorm_bwd<4>, 4); break;
  }
  if (le != cudaSuccess) return le;
  cudaError_t e = post_launch(L);
  if (e != cudaSuccess) return e;
  k_dg_finalize<<<(d + 31) / 32, kThreads, 0, L.stream>>>(dg_partial, nblk, d, dg);
  return post_launch(L);
}

}  // namespace fp8q
