// Block-scaled (MXFP8) quantization for sm_103a.
//
// LLMQ §2 ("LLMQ: Efficient Lower-Precision Pretraining for Consumer GPUs")
// names inner-dimension block scaling as the scaling Blackwell tensor cores
// support natively.  Format (OCP Microscaling): 32 consecutive elements along
// a GEMM's contraction dimension share one power-of-two scale 2^X, stored as
// the E8M0 code X + 127; the elements are E4M3 or E5M2 codes.  Scale rule
// (the per-tensor "no clipping" rule applied per block): X is the smallest
// integer with amax_block <= fmax * 2^X, clamped to [-127, 127]; an all-zero
// block has X = -127; a block holding NaN or Inf gets the NaN code 0xFF, NaN
// element codes and the NONFINITE status bit.  Element code =
// cvt.rn.satfinite(fl32(v * 2^-X)).
//
// One pass over the input writes both directions a training step needs: the
// blocks along each row (32 consecutive columns: the tensor as a K-major GEMM
// operand, K = its columns) and the blocks down each column (32 consecutive
// rows: the tensor as an MN-major operand, K = its rows).  There is no global
// reduction, so unlike the per-tensor quantizer no second pass is needed.
//
// Scale-factor layout (what the block-scaled GEMM loads into tensor memory):
// an operand with `rows` rows along M (or N) and contraction length K keeps
// its E8M0 codes in 512-byte chunks, one per 128 rows x 128 K (4 blocks), in
// row-chunk-major order; inside a chunk, row r and block b of the chunk sit at
// byte (r % 32) * 16 + (r / 32) * 4 + b.
//
// CTA tile: 32 rows x 128 columns, 256 threads; thread t holds row t / 8 and
// the 16 columns 16 (t % 8) ..; a row block is a lane pair, a column block the
// 32 rows of the tile (warp shuffles over the warp's 4 rows, then shared
// memory over the 8 warps).
#include "fp8q_common.cuh"
#include "fp8q_internal.h"

namespace fp8q {

namespace {

constexpr int kThreads = 256;
constexpr int kTileRows = 32, kTileCols = 128;

inline cudaError_t post_launch(const Launch& L) {
  if (L.launches) ++*L.launches;
  return cudaGetLastError();
}

// The smallest X in [-127, 127] with a <= fmax * 2^X for a finite, non-negative a given by its
// fp32 bits.  fmax = 1.75 * 2^EMAX (E4M3: 448, EMAX 8; E5M2: 57344, EMAX 15).  With a = M * 2^e,
// M in [1, 2): a <= 1.75 * 2^(X + EMAX) exactly when X >= e - EMAX + (M > 1.75).
template <int FMT>
__device__ __forceinline__ int mx_exponent(uint32_t abits) {
  constexpr int EMAX = FMT == 0 ? 8 : 15;
  if (abits == 0) return -127;
  int e;
  bool above;
  const uint32_t E = abits >> 23, m = abits & 0x7FFFFFu;
  if (E != 0) {
    e = (int)E - 127;
    above = m > 0x600000u;  // M = 1 + m / 2^23 > 1.75
  } else {                  // subnormal: a = m * 2^-149
    const int p = 31 - __clz((int)m);
    e = p - 149;
    above = 4ull * m > 7ull << p;  // m / 2^p > 1.75
  }
  int X = e - EMAX + (above ? 1 : 0);
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}

// 2^-X as fp32 (X in [-127, 127]; 2^-127 is subnormal).
__device__ __forceinline__ float pow2_neg(int X) {
  return X == 127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(127 - X) << 23);
}

// Byte offset of (operand row r, contraction index k) in the chunked scale layout.
__device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t k, int64_t n_kchunks) {
  return ((r >> 7) * n_kchunks + (k >> 7)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + ((k >> 5) & 3);
}

// 16 codes of v * s (s = 2^-X) packed in a uint4.
template <int FMT>
__device__ __forceinline__ uint4 codes16(const float (&v)[16], float s) {
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    w[q] = cvt_fp8x4<FMT>(__fmul_rn(v[4 * q], s), __fmul_rn(v[4 * q + 1], s), __fmul_rn(v[4 * q + 2], s),
                          __fmul_rn(v[4 * q + 3], s));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

struct MxArgs {
  const void* x;        // IN 0: bf16 [R, C]; 1: fp32 [R, C]; 2: bf16 H [R, 2C]; 3: bf16 x [R, C]
  const uint16_t* g;    // IN 3: RMSNorm gain [C]
  const float* rstd;    // IN 3: [R]
  int64_t R, C;
  uint8_t* q_r; uint8_t* sf_r;  // blocks along rows (K = C), or null
  uint8_t* q_c; uint8_t* sf_c;  // blocks down columns (K = R), or null
  unsigned* status;
};

// The 16 input values of (row, columns c .. c + 15): the tensor itself, SwiGLU of [gate | up]
// (swiglu_fast, as the fused forward's a), or the RMSNorm output fl32(fl32(x rstd) g).
template <int IN>
__device__ __forceinline__ void load16(const MxArgs& p, int64_t row, int64_t c, float (&v)[16]) {
  if (IN == 1) {
    const float* xr = static_cast<const float*>(p.x) + row * p.C + c;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = ld_nc_v4(xr + 4 * q);
      v[4 * q] = __uint_as_float(w.x); v[4 * q + 1] = __uint_as_float(w.y);
      v[4 * q + 2] = __uint_as_float(w.z); v[4 * q + 3] = __uint_as_float(w.w);
    }
    return;
  }
  const int64_t ld = IN == 2 ? 2 * p.C : p.C;
  const uint16_t* xr = static_cast<const uint16_t*>(p.x) + row * ld + c;
  uint32_t xw[8];
  {
    const uint4 a = ld_nc_v4(xr), b = ld_nc_v4(xr + 8);
    xw[0] = a.x; xw[1] = a.y; xw[2] = a.z; xw[3] = a.w; xw[4] = b.x; xw[5] = b.y; xw[6] = b.z; xw[7] = b.w;
  }
  if (IN == 0) {
#pragma unroll
    for (int k = 0; k < 8; ++k) { v[2 * k] = bf16_lo(xw[k]); v[2 * k + 1] = bf16_hi(xw[k]); }
  } else if (IN == 2) {
    const uint4 a = ld_nc_v4(xr + p.C), b = ld_nc_v4(xr + p.C + 8);
    const uint32_t uw[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[2 * k] = swiglu_fast(bf16_lo(xw[k]), bf16_lo(uw[k]));
      v[2 * k + 1] = swiglu_fast(bf16_hi(xw[k]), bf16_hi(uw[k]));
    }
  } else {
    const float rs = p.rstd[row];
    const uint4 ga = ld_v4(p.g + c), gb = ld_v4(p.g + c + 8);
    const uint32_t gw[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[2 * k] = __fmul_rn(__fmul_rn(bf16_lo(xw[k]), rs), bf16_lo(gw[k]));
      v[2 * k + 1] = __fmul_rn(__fmul_rn(bf16_hi(xw[k]), rs), bf16_hi(gw[k]));
    }
  }
}

constexpr uint32_t kInfBits = 0x7F800000u;
constexpr uint32_t kNanCodes4 = 0x7F7F7F7Fu;  // four NaN codes (0x7F in both formats)

template <int IN, int FMT>
__global__ void __launch_bounds__(kThreads) k_mx_quant(const MxArgs p) {
  __shared__ uint32_t colmax[kThreads / 32][kTileCols];
  __shared__ int colx[kTileCols];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int tr = t >> 3, seg = t & 7;
  const int64_t tiles_c = p.C / kTileCols;
  const int64_t tiles = (p.R / kTileRows) * tiles_c;
  bool nonfinite = false;
  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t r0 = (tile / tiles_c) * kTileRows, c0 = (tile % tiles_c) * kTileCols;
    const int64_t row = r0 + tr, col = c0 + seg * 16;
    float v[16];
    load16<IN>(p, row, col, v);
    uint32_t am[16];
    uint32_t rmax = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      am[j] = abs_bits(v[j]);
      rmax = max(rmax, am[j]);
    }
    // ---- blocks along the row: 32 columns = this lane and its pair
    if (p.q_r) {
      rmax = max(rmax, __shfl_xor_sync(0xFFFFFFFFu, rmax, 1));
      uint4 out;
      uint8_t sfc;
      if (rmax >= kInfBits) {
        out = make_uint4(kNanCodes4, kNanCodes4, kNanCodes4, kNanCodes4);
        sfc = 0xFF;
        nonfinite = true;
      } else {
        const int X = mx_exponent<FMT>(rmax);
        out = codes16<FMT>(v, pow2_neg(X));
        sfc = (uint8_t)(X + 127);
      }
      st_v4(p.q_r + row * p.C + col, out);
      if ((seg & 1) == 0) p.sf_r[sf_offset(row, col, p.C >> 7)] = sfc;
    }
    // ---- blocks down the column: the tile's 32 rows
    if (p.q_c) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        uint32_t m = max(am[j], __shfl_xor_sync(0xFFFFFFFFu, am[j], 8));
        am[j] = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
      }
      if (lane < 8) {
#pragma unroll
        for (int j = 0; j < 16; ++j) colmax[warp][lane * 16 + j] = am[j];
      }
      __syncthreads();
      if (t < kTileCols) {
        uint32_t m = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) m = max(m, colmax[w][t]);
        int X;
        uint8_t sfc;
        if (m >= kInfBits) {
          X = 1000;  // marks a non-finite column block
          sfc = 0xFF;
          nonfinite = true;
        } else {
          X = mx_exponent<FMT>(m);
          sfc = (uint8_t)(X + 127);
        }
        colx[t] = X;
        p.sf_c[sf_offset(c0 + t, r0, p.R >> 7)] = sfc;
      }
      __syncthreads();
      float s[16];
      bool bad = false;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int X = colx[seg * 16 + j];
        bad |= X == 1000;
        s[j] = X == 1000 ? 1.0f : pow2_neg(X);
      }
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w[q] = cvt_fp8x4<FMT>(__fmul_rn(v[4 * q], s[4 * q]), __fmul_rn(v[4 * q + 1], s[4 * q + 1]),
                              __fmul_rn(v[4 * q + 2], s[4 * q + 2]), __fmul_rn(v[4 * q + 3], s[4 * q + 3]));
      if (bad) {  // every element of a non-finite column block is the NaN code
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (colx[seg * 16 + j] == 1000) w[j >> 2] = (w[j >> 2] & ~(0xFFu << (8 * (j & 3)))) | (0x7Fu << (8 * (j & 3)));
      }
      st_v4(p.q_c + row * p.C + col, make_uint4(w[0], w[1], w[2], w[3]));
      __syncthreads();  // colmax / colx are rewritten by the next tile
    }
  }
  if (nonfinite) atomicOr(p.status, kStatusNonfinite);
}

template <int IN>
cudaError_t launch_in(const MxArgs& a, int fmt, const Launch& L) {
  const int64_t tiles = (a.R / kTileRows) * (a.C / kTileCols);
  const int64_t cap = (int64_t)L.num_sms * 8;
  const int grid = (int)(tiles < cap ? (tiles > 0 ? tiles : 1) : cap);
  if (fmt == 0) k_mx_quant<IN, 0><<<grid, kThreads, 0, L.stream>>>(a);
  else k_mx_quant<IN, 1><<<grid, kThreads, 0, L.stream>>>(a);
  return post_launch(L);
}

}  // namespace

size_t mx_scale_bytes(int64_t rows, int64_t K) { return (size_t)(((rows + 127) / 128) * ((K + 127) / 128) * 512); }

cudaError_t launch_mx_quant(int in_kind, const void* x, const uint16_t* g, const float* rstd, int64_t R, int64_t C,
                            int fmt, uint8_t* q_r, uint8_t* sf_r, uint8_t* q_c, uint8_t* sf_c, const Launch& L) {
  MxArgs a{x, g, rstd, R, C, q_r, sf_r, q_c, sf_c, L.status};
  switch (in_kind) {
    case kMxInBf16: return launch_in<0>(a, fmt, L);
    case kMxInF32: return launch_in<1>(a, fmt, L);
    case kMxInSwiglu: return launch_in<2>(a, fmt, L);
    default: return launch_in<3>(a, fmt, L);
  }
}

}  // namespace fp8q
