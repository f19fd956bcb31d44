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
// CTA tile: 32 rows x 128 columns, 256 threads; each thread holds 8 columns of
// two rows, and a warp's load reads two whole 128-column row segments
// (coalesced); a row block is 4 consecutive lanes, a column block the tile's 32
// rows (a warp shuffle over its 4 rows, then shared memory over the 8 warps).
// Each thread loads its next tile's inputs before it reduces and writes the
// current one, so the loads stay in flight across the tile's barriers.
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

struct MxArgs {
  const void* x;        // IN 0: bf16 [R, C]; 1: fp32 [R, C]; 2: bf16 H [R, 2C]; 3: bf16 x [R, C]
  const uint16_t* g;    // IN 3: RMSNorm gain [C]
  const float* rstd;    // IN 3: [R]
  int64_t R, C;
  uint8_t* q_r; uint8_t* sf_r;  // blocks along rows (K = C), or null
  uint8_t* q_c; uint8_t* sf_c;  // blocks down columns (K = R), or null
  unsigned* status;
};

// Thread layout of a 32 x 128 tile: warp w, lane l holds rows 2 (w + 8 k) + (l / 16), k = 0, 1, and
// the 8 columns 8 (l % 16) ..; a warp's load instruction reads two whole 128-column row segments.
__device__ __forceinline__ int tile_row(int warp, int lane, int k) { return 2 * (warp + 8 * k) + (lane >> 4); }

// The raw words of one thread's inputs (8 columns of one row), loaded one tile ahead of their use:
// bf16 x (1 vector), fp32 x (2), bf16 gate and up of H (1 + 1), bf16 x of the RMSNorm (1).
struct Raw {
  uint4 w[2][2];  // [row k][vector]
};

template <int IN>
__device__ __forceinline__ uint4 raw_vec(const MxArgs& p, int64_t row, int64_t c, int i) {
  if (IN == 1) return ld_nc_v4(static_cast<const float*>(p.x) + row * p.C + c + 4 * i);
  const int64_t ld = IN == 2 ? 2 * p.C : p.C;
  return ld_nc_v4(static_cast<const uint16_t*>(p.x) + row * ld + c + (i ? p.C : 0));
}

template <int IN>
__device__ __forceinline__ Raw load_raw(const MxArgs& p, int64_t r0, int64_t c, int warp, int lane) {
  Raw r;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int64_t row = r0 + tile_row(warp, lane, k);
    r.w[k][0] = raw_vec<IN>(p, row, c, 0);
    if (IN == 1 || IN == 2) r.w[k][1] = raw_vec<IN>(p, row, c, 1);
  }
  return r;
}

// The 8 input values of one row: the tensor itself, SwiGLU of [gate | up] (swiglu_fast, as the
// fused forward's a), or the RMSNorm output fl32(fl32(x rstd) g).
template <int IN>
__device__ __forceinline__ void decode8(const uint4 (&w)[2], const MxArgs& p, int64_t row, int64_t c, float (&v)[8]) {
  if (IN == 1) {
    v[0] = __uint_as_float(w[0].x); v[1] = __uint_as_float(w[0].y);
    v[2] = __uint_as_float(w[0].z); v[3] = __uint_as_float(w[0].w);
    v[4] = __uint_as_float(w[1].x); v[5] = __uint_as_float(w[1].y);
    v[6] = __uint_as_float(w[1].z); v[7] = __uint_as_float(w[1].w);
    return;
  }
  const uint32_t xw[4] = {w[0].x, w[0].y, w[0].z, w[0].w};
  if (IN == 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k) { v[2 * k] = bf16_lo(xw[k]); v[2 * k + 1] = bf16_hi(xw[k]); }
  } else if (IN == 2) {
    const uint32_t uw[4] = {w[1].x, w[1].y, w[1].z, w[1].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = swiglu_fast(bf16_lo(xw[k]), bf16_lo(uw[k]));
      v[2 * k + 1] = swiglu_fast(bf16_hi(xw[k]), bf16_hi(uw[k]));
    }
  } else {
    const float rs = p.rstd[row];
    const uint4 gv = ld_v4(p.g + c);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __fmul_rn(__fmul_rn(bf16_lo(xw[k]), rs), bf16_lo(gw[k]));
      v[2 * k + 1] = __fmul_rn(__fmul_rn(bf16_hi(xw[k]), rs), bf16_hi(gw[k]));
    }
  }
}

// 8 codes of v[j] * s[j] packed in a uint2.
template <int FMT>
__device__ __forceinline__ uint2 codes8(const float (&v)[8], const float (&s)[8]) {
  return make_uint2(cvt_fp8x4<FMT>(__fmul_rn(v[0], s[0]), __fmul_rn(v[1], s[1]), __fmul_rn(v[2], s[2]),
                                   __fmul_rn(v[3], s[3])),
                    cvt_fp8x4<FMT>(__fmul_rn(v[4], s[4]), __fmul_rn(v[5], s[5]), __fmul_rn(v[6], s[6]),
                                   __fmul_rn(v[7], s[7])));
}
__device__ __forceinline__ void st_v2(void* p, uint2 v) { *reinterpret_cast<uint2*>(p) = v; }

constexpr uint32_t kInfBits = 0x7F800000u;
constexpr uint32_t kNanCodes4 = 0x7F7F7F7Fu;  // four NaN codes (0x7F in both formats)
constexpr int kNonfiniteX = 1000;             // marks a non-finite column block in colx

template <int IN, int FMT>
__global__ void __launch_bounds__(kThreads) k_mx_quant(const MxArgs p) {
  // the column-block reduction's buffers, double-buffered by tile parity so that one barrier per
  // phase suffices (a tile's reads of buffer b finish before the next tile but one rewrites it)
  __shared__ __align__(16) uint32_t colmax[2][kThreads / 32][kTileCols];
  __shared__ int colx[2][kTileCols];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int cseg = (lane & 15) * 8;  // this thread's first column in the tile
  const int64_t tiles_c = p.C / kTileCols;
  const int64_t tiles = (p.R / kTileRows) * tiles_c;
  bool nonfinite = false;
  int64_t tile = blockIdx.x;
  Raw raw;
  if (tile < tiles) raw = load_raw<IN>(p, (tile / tiles_c) * kTileRows, (tile % tiles_c) * kTileCols + cseg, warp, lane);
  for (int par = 0; tile < tiles; tile += gridDim.x, par ^= 1) {
    const int64_t r0 = (tile / tiles_c) * kTileRows, c0 = (tile % tiles_c) * kTileCols;
    const int64_t col = c0 + cseg;
    float v[2][8];
#pragma unroll
    for (int k = 0; k < 2; ++k) decode8<IN>(raw.w[k], p, r0 + tile_row(warp, lane, k), col, v[k]);
    // the next tile's inputs are in flight while this one is reduced and written
    const int64_t nt = tile + gridDim.x;
    if (nt < tiles) raw = load_raw<IN>(p, (nt / tiles_c) * kTileRows, (nt % tiles_c) * kTileCols + cseg, warp, lane);
    // ---- blocks along the row: 32 columns = 4 consecutive lanes
    if (p.q_r) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) m = max(m, abs_bits(v[k][j]));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        const int64_t row = r0 + tile_row(warp, lane, k);
        uint2 out;
        uint8_t sfc;
        if (m >= kInfBits) {
          out = make_uint2(kNanCodes4, kNanCodes4);
          sfc = 0xFF;
          nonfinite = true;
        } else {
          const int X = mx_exponent<FMT>(m);
          const float sc = pow2_neg(X);
          const float s8[8] = {sc, sc, sc, sc, sc, sc, sc, sc};
          out = codes8<FMT>(v[k], s8);
          sfc = (uint8_t)(X + 127);
        }
        st_v2(p.q_r + row * p.C + col, out);
        if ((lane & 3) == 0) p.sf_r[sf_offset(row, col, p.C >> 7)] = sfc;
      }
    }
    // ---- blocks down the column: the tile's 32 rows (2 per thread, 2 lanes per warp, 8 warps)
    if (p.q_c) {
      uint32_t cm[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t m = max(abs_bits(v[0][j]), abs_bits(v[1][j]));
        cm[j] = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
      }
      if (lane < 16) {
        st_v4(&colmax[par][warp][cseg], make_uint4(cm[0], cm[1], cm[2], cm[3]));
        st_v4(&colmax[par][warp][cseg + 4], make_uint4(cm[4], cm[5], cm[6], cm[7]));
      }
      __syncthreads();
      if (t < kTileCols) {
        uint32_t m = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) m = max(m, colmax[par][w][t]);
        int X;
        uint8_t sfc;
        if (m >= kInfBits) {
          X = kNonfiniteX;
          sfc = 0xFF;
          nonfinite = true;
        } else {
          X = mx_exponent<FMT>(m);
          sfc = (uint8_t)(X + 127);
        }
        colx[par][t] = X;
        p.sf_c[sf_offset(c0 + t, r0, p.R >> 7)] = sfc;
      }
      __syncthreads();
      float s[8];
      bool bad = false;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int X = colx[par][cseg + j];
        bad |= X == kNonfiniteX;
        s[j] = X == kNonfiniteX ? 1.0f : pow2_neg(X);
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        uint2 out = codes8<FMT>(v[k], s);
        if (bad) {  // every element of a non-finite column block is the NaN code
          uint32_t w2[2] = {out.x, out.y};
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (colx[par][cseg + j] == kNonfiniteX)
              w2[j >> 2] = (w2[j >> 2] & ~(0xFFu << (8 * (j & 3)))) | (0x7Fu << (8 * (j & 3)));
          out = make_uint2(w2[0], w2[1]);
        }
        st_v2(p.q_c + (r0 + tile_row(warp, lane, k)) * p.C + col, out);
      }
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
