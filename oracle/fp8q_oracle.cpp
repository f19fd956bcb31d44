// CPU oracle for the FP8 per-tensor-absmax transformer-block pipeline.
//
// TEST INFRASTRUCTURE ONLY.  This library is loaded by the test-suite, by the
// package's smoke() check and by the benchmark's CPU-baseline leg, nothing
// else.  The CUDA library never links, includes or calls it, and it shares no
// code, header, table or constant generator with the CUDA library.
//
// What it states, and where the statement comes from:
//   * "LLMQ: Efficient Lower-Precision Pretraining for Consumer GPUs"
//     (paperlayer.ai summary of arXiv 2512.15306), §1: FP8 training with
//     dynamic tensor-level scaling.
//   * "Periodic Reporting for period 1 - FastML" (CORDIS), paragraph "FP8
//     training without delayed scaling": just-in-time tensor-level absmax
//     scaling that guarantees no value clipping.
//   * LLMQ §3.1 (activation checkpointing): absmax statistics are retained
//     per tensor; quantization follows the nonlinearity (SwiGLU).
//   * LLMQ §5, Figure 2: E4M3 for activations/weights, E5M2 for activation
//     gradients.
//   * LLMQ §3 / §3.1 / §3.2: non-matmul ops (RMSNorm, SwiGLU, residual) are
//     fused around the GEMMs; kernels are deterministic.
//   * FP8 encodings follow the OCP 8-bit floating point specification
//     (E4M3 "FN": no infinities, max 448; E5M2: IEEE-like, max 57344).
//   * LLMQ §2: inner-dimension (block) scaling, native on Blackwell; the block
//     format is the OCP Microscaling one (32 elements, E8M0 scale).
// The pages give no formula beyond these sentences; every concrete choice
// below (scale = fmax/amax, fp32 product before the cast, RNE with
// saturation, RMSNorm epsilon and pairwise fp32 sum of squares, SwiGLU in
// fp32 with exp_ref, bf16 storage points) is a stated reading of them.
//
// Two arithmetic modes share one code path:
//   quantized (exact == 0): the FP8 pipeline.  Every rounding point is an
//     explicit call (to_bf16, fp32 expression, fp8 encode).  GEMMs accumulate
//     in fp64 (exact for E4M3 x E4M3 at every size used here).
//   exact (exact == 1): the same block with every rounding point removed and
//     all arithmetic in fp64.  Used to pin the backward formulas against
//     finite differences of the forward.
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -fno-fast-math -fPIC -shared
// (-ffp-contract=off keeps every fp32 expression at one rounding per
// operation on both x86-64 and aarch64).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ----------------------------------------------------------------------------
// Bit helpers, bf16
// ----------------------------------------------------------------------------
float f32_from_bits(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }
uint32_t bits_from_f32(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }

double bf16_value(uint16_t h) { return (double)f32_from_bits((uint32_t)h << 16); }

// Round v to the nearest number with `frac` fraction bits whose exponent is at
// least `emin` (so values below 2^emin land on the subnormal grid), ties to
// even.  No overflow handling: callers saturate or overflow themselves.
double round_binary(double v, int frac, int emin) {
  if (v == 0.0 || !std::isfinite(v)) return v;
  int e;
  std::frexp(std::fabs(v), &e);            // |v| in [2^(e-1), 2^e)
  int ex = std::max(e - 1, emin);
  double quantum = std::ldexp(1.0, ex - frac);
  return std::nearbyint(v / quantum) * quantum;   // default mode: ties-to-even
}

// One rounding from a real (given as double) to bf16, IEEE round-to-nearest-even,
// overflow to infinity.
uint16_t to_bf16_bits(double v) {
  if (std::isnan(v)) return (uint16_t)(0x7FC0 | (std::signbit(v) ? 0x8000 : 0));
  double r = round_binary(v, 7, -126);
  float rf = (float)r;                      // exact, or +-inf when r = +-2^128
  return (uint16_t)(bits_from_f32(rf) >> 16);
}
double to_bf16(double v) { return bf16_value(to_bf16_bits(v)); }

// ----------------------------------------------------------------------------
// FP8 codec (OCP E4M3 "FN" and E5M2), round-to-nearest-even, saturating
// ----------------------------------------------------------------------------
enum { FMT_E4M3 = 0, FMT_E5M2 = 1 };

struct Fp8Format {
  int frac;        // fraction bits
  int emin;        // exponent of the smallest normal
  int bias;
  double maxv;     // largest finite magnitude
  uint8_t nan_code;
};

const Fp8Format& fp8_format(int fmt) {
  static const Fp8Format e4m3 = {3, -6, 7, 448.0, 0x7F};
  static const Fp8Format e5m2 = {2, -14, 15, 57344.0, 0x7F};
  return fmt == FMT_E5M2 ? e5m2 : e4m3;
}

double fp8_decode(uint8_t c, int fmt) {
  const Fp8Format& F = fp8_format(fmt);
  const int ebits = 7 - F.frac;
  const int emask = (1 << ebits) - 1;
  const int mmask = (1 << F.frac) - 1;
  const double sign = (c & 0x80) ? -1.0 : 1.0;
  const int e = (c >> F.frac) & emask;
  const int m = c & mmask;
  if (fmt == FMT_E4M3 && e == emask && m == mmask) return std::nan("");
  if (fmt == FMT_E5M2 && e == emask) return m == 0 ? sign * HUGE_VAL : std::nan("");
  if (e == 0) return sign * std::ldexp((double)m, F.emin - F.frac);
  return sign * std::ldexp(1.0 + std::ldexp((double)m, -F.frac), e - F.bias);
}

// fp32 -> fp8 with round-to-nearest-even and saturation to +-max (so +-inf
// saturates too); NaN -> the format's NaN code; the sign of zero is kept.
uint8_t fp8_encode(float v, int fmt) {
  const Fp8Format& F = fp8_format(fmt);
  if (std::isnan(v)) return F.nan_code;
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  double a = round_binary(std::fabs((double)v), F.frac, F.emin);
  if (a > F.maxv) a = F.maxv;
  if (a == 0.0) return sign;
  int e;
  std::frexp(a, &e);
  const int ex = e - 1;
  if (ex < F.emin) {                               // subnormal grid
    int m = (int)(a / std::ldexp(1.0, F.emin - F.frac));
    return (uint8_t)(sign | m);
  }
  int m = (int)(a / std::ldexp(1.0, ex - F.frac)) - (1 << F.frac);
  return (uint8_t)(sign | ((ex + F.bias) << F.frac) | m);
}

// ----------------------------------------------------------------------------
// exp_ref: fp32 exponential with a fixed operation sequence so that SwiGLU has
// one bit-exact answer.  Method: Cody & Waite argument reduction
// x = k ln2 + r with ln2 split in a short high part (exact k*hi) and a low
// correction, |r| <= ln2/2, then the Taylor polynomial of e^r to degree 8 in
// Horner form, then multiplication by 2^k built from exponent bits.  The
// reduction and every Horner step are IEEE-754 fused multiply-adds (one
// rounding each, std::fma); every other operation is a single IEEE fp32
// operation.
// ----------------------------------------------------------------------------
float exp_ref(float x) {
  if (std::isnan(x)) return x;
  if (x > 88.72283935546875f) return HUGE_VALF;     // e^x > FLT_MAX
  if (x < -103.972084045410156f) return 0.0f;       // e^x < half the smallest subnormal
  const float log2e = 1.44269502162933349609375f;   // fp32(1/ln 2)
  const float ln2_hi = 0.693359375f;                // 355/512, 9 significant bits
  const float ln2_lo = -2.12194440e-4f;             // fp32(ln 2 - 355/512)
  const float kf = std::nearbyint(x * log2e);
  const float r = std::fma(-kf, ln2_lo, std::fma(-kf, ln2_hi, x));
  float p = 1.0f / 40320.0f;                        // 1/8!
  p = std::fma(p, r, 1.0f / 5040.0f);
  p = std::fma(p, r, 1.0f / 720.0f);
  p = std::fma(p, r, 1.0f / 120.0f);
  p = std::fma(p, r, 1.0f / 24.0f);
  p = std::fma(p, r, 1.0f / 6.0f);
  p = std::fma(p, r, 0.5f);
  p = std::fma(p, r, 1.0f);
  p = std::fma(p, r, 1.0f);
  const int k = (int)kf;                            // -150 <= k <= 128
  if (k > 127) return (p * 2.0f) * f32_from_bits((uint32_t)(127 + 127) << 23);
  if (k >= -126) return p * f32_from_bits((uint32_t)(k + 127) << 23);
  // subnormal result: scale into the normal range first, then one rounding
  return (p * f32_from_bits((uint32_t)(k + 64 + 127) << 23)) * f32_from_bits((uint32_t)(127 - 64) << 23);
}

// ----------------------------------------------------------------------------
// Per-tensor absmax scaling
// ----------------------------------------------------------------------------
struct Scal { float amax, scale, scale_inv; };

// s = fl32(fmax / amax): the tensor's absmax element lands exactly on +-fmax,
// nothing is clipped.  amax == 0 gives s = 1.  Non-finite amax follows IEEE.
Scal scale_from_amax(float amax, int fmt) {
  Scal r;
  r.amax = amax;
  if (amax == 0.0f) { r.scale = 1.0f; r.scale_inv = 1.0f; return r; }
  const float fmax = (float)fp8_format(fmt).maxv;
  r.scale = fmax / amax;
  r.scale_inv = 1.0f / r.scale;
  return r;
}

float abs_max(const std::vector<double>& v) {
  float m = 0.0f;
  bool nan = false;
  for (double x : v) {
    if (std::isnan(x)) nan = true;
    m = std::max(m, (float)std::fabs(x));
  }
  return nan ? std::nanf("") : m;
}

bool finite_scal(const Scal& s) { return std::isfinite(s.amax); }

// A quantized operand: codes, the tensor's scalars, and the decoded codes as
// doubles (unscaled; the GEMM applies scale_inv of both operands once).
struct QTensor {
  std::vector<uint8_t> code;
  std::vector<double> deq;
  Scal s;
};

// In quantized mode: amax -> s -> code = fp8(fl32(v * s)).  Every v must be an
// fp32 value.  In exact mode the operand passes through with scale_inv = 1.
QTensor quantize(const std::vector<double>& v, int fmt, bool exact) {
  QTensor q;
  if (exact) {
    q.deq = v;
    q.s = {abs_max(v), 1.0f, 1.0f};
    return q;
  }
  q.s = scale_from_amax(abs_max(v), fmt);
  q.code.resize(v.size());
  q.deq.resize(v.size());
  for (size_t i = 0; i < v.size(); ++i) {
    const float p = (float)v[i] * q.s.scale;
    q.code[i] = fp8_encode(p, fmt);
    q.deq[i] = fp8_decode(q.code[i], fmt);
  }
  return q;
}

// ----------------------------------------------------------------------------
// Block scaling (MXFP8).  LLMQ §2 names inner-dimension (block) scaling as the
// scaling Blackwell tensor cores support natively.  Its formats are those of
// the OCP Microscaling (MX) specification: a block of 32 consecutive elements
// along a GEMM's contraction dimension shares one scale 2^X stored as an
// 8-bit E8M0 code X + 127 (0xFF is NaN); the elements are E4M3 or E5M2 codes.
// Reading of the scale choice (the pages fix none; the FastML report's
// "no clipping" rule carried from the tensor to the block): X is the smallest
// integer with amax_block <= fmax * 2^X, clamped to the code range
// [-127, 127]; an all-zero block takes X = -127 (code 0); a block holding NaN
// or Inf takes code 0xFF and sets the status bit.  Element code =
// fp8(fl32(v * 2^-X)), round to nearest even with saturation; its value is
// decode(code) * 2^X.
// ----------------------------------------------------------------------------
constexpr int kMxBlock = 32;

// The smallest X in [-127, 127] with amax <= fmax * 2^X (amax finite, >= 0).
int mx_exponent(double amax, int fmt) {
  const double fmax = fp8_format(fmt).maxv;
  if (amax == 0.0) return -127;
  int X = (int)std::ceil(std::log2(amax / fmax));  // an estimate; the loops make it exact
  X = std::max(-127, std::min(127, X));
  while (X > -127 && amax <= std::ldexp(fmax, X - 1)) --X;
  while (X < 127 && amax > std::ldexp(fmax, X)) ++X;
  return X;
}

// A block-scaled operand: element codes (same layout as the input), one E8M0
// code per block, and each element's value decode(code) * 2^X as a double.
struct MxTensor {
  std::vector<uint8_t> code;
  std::vector<uint8_t> sf;   // along_rows == 0: [R][ceil(C/32)]; along_rows == 1: [ceil(R/32)][C]
  std::vector<double> deq;
  int status = 0;
};

// Blocks of 32 consecutive elements of a row (along_rows == 0: the contraction
// runs along the columns) or of a column (along_rows == 1: it runs along the
// rows) of the R x C matrix v; a last partial block holds the remainder.
MxTensor mx_quantize(const std::vector<double>& v, int64_t R, int64_t C, int fmt, bool along_rows) {
  MxTensor q;
  q.code.assign((size_t)(R * C), 0);
  q.deq.assign((size_t)(R * C), 0.0);
  const int64_t nb_r = along_rows ? (R + kMxBlock - 1) / kMxBlock : R;
  const int64_t nb_c = along_rows ? C : (C + kMxBlock - 1) / kMxBlock;
  q.sf.assign((size_t)(nb_r * nb_c), 0);
  for (int64_t br = 0; br < nb_r; ++br)
    for (int64_t bc = 0; bc < nb_c; ++bc) {
      // the block's elements
      std::vector<int64_t> idx;
      if (along_rows) {
        for (int64_t r = br * kMxBlock; r < std::min(R, (br + 1) * kMxBlock); ++r) idx.push_back(r * C + bc);
      } else {
        for (int64_t c = bc * kMxBlock; c < std::min(C, (bc + 1) * kMxBlock); ++c) idx.push_back(br * C + c);
      }
      double amax = 0.0;
      bool finite = true;
      for (int64_t i : idx) {
        if (!std::isfinite(v[i])) finite = false;
        else amax = std::max(amax, std::fabs(v[i]));
      }
      if (!finite) {
        q.sf[br * nb_c + bc] = 0xFF;
        q.status |= 1;
        for (int64_t i : idx) { q.code[i] = fp8_format(fmt).nan_code; q.deq[i] = std::nan(""); }
        continue;
      }
      const int X = mx_exponent(amax, fmt);
      q.sf[br * nb_c + bc] = (uint8_t)(X + 127);
      const float inv = (float)std::ldexp(1.0, -X);
      for (int64_t i : idx) {
        q.code[i] = fp8_encode((float)v[i] * inv, fmt);
        q.deq[i] = std::ldexp(fp8_decode(q.code[i], fmt), X);
      }
    }
  return q;
}

// ----------------------------------------------------------------------------
// GEMM: C[M,N] = A[M,K] B[K,N] in fp64, row-major operands.  Rows of C may be
// split over threads; every element's arithmetic and order is the same for
// any thread count.
// ----------------------------------------------------------------------------
void matmul_rows(const double* A, const double* B, double* C, int64_t N, int64_t K,
                 int64_t r0, int64_t r1) {
  for (int64_t i = r0; i < r1; ++i) {
    double* c = C + i * N;
    std::fill(c, c + N, 0.0);
    for (int64_t k = 0; k < K; ++k) {
      const double a = A[i * K + k];
      const double* b = B + k * N;
      for (int64_t j = 0; j < N; ++j) c[j] += a * b[j];
    }
  }
}

std::vector<double> matmul(const std::vector<double>& A, const std::vector<double>& B,
                           int64_t M, int64_t N, int64_t K, int nthreads) {
  std::vector<double> C((size_t)(M * N));
  nthreads = std::max(1, std::min<int>(nthreads, (int)std::max<int64_t>(M, 1)));
  if (nthreads == 1) {
    matmul_rows(A.data(), B.data(), C.data(), N, K, 0, M);
    return C;
  }
  std::vector<std::thread> pool;
  for (int t = 0; t < nthreads; ++t) {
    int64_t r0 = M * t / nthreads, r1 = M * (t + 1) / nthreads;
    pool.emplace_back(matmul_rows, A.data(), B.data(), C.data(), N, K, r0, r1);
  }
  for (auto& th : pool) th.join();
  return C;
}

std::vector<double> transpose(const std::vector<double>& X, int64_t R, int64_t Cn) {
  std::vector<double> Y((size_t)(R * Cn));
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < Cn; ++c) Y[c * R + r] = X[r * Cn + c];
  return Y;
}

// ----------------------------------------------------------------------------
// RMSNorm forward
// ----------------------------------------------------------------------------
// Pairwise (recursive halving) sum in fp32: a range of length n > 1 is split
// at the largest power of two below n and the two halves are added.
float pairwise_sum(const float* v, int64_t n) {
  if (n == 0) return 0.0f;
  if (n == 1) return v[0];
  int64_t m = 1;
  while (m * 2 < n) m *= 2;
  return pairwise_sum(v, m) + pairwise_sum(v + m, n - m);
}

// n = (x * rstd) * g with rstd = 1/sqrt(mean(x^2) + eps).
// Quantized mode (all fp32, one rounding per op): sum of squares by pairwise
// summation, mean = S/d, rstd = 1/sqrt(mean + eps).  Exact mode: fp64.
void rmsnorm_fwd(const std::vector<double>& x, const std::vector<double>& g, int64_t T, int64_t d,
                 float eps, bool exact, std::vector<double>& n, std::vector<double>& rstd) {
  n.assign((size_t)(T * d), 0.0);
  rstd.assign((size_t)T, 0.0);
  std::vector<float> sq((size_t)d);
  for (int64_t t = 0; t < T; ++t) {
    const double* xr = &x[t * d];
    if (!exact) {
      for (int64_t j = 0; j < d; ++j) sq[j] = (float)xr[j] * (float)xr[j];
      const float S = pairwise_sum(sq.data(), d);
      const float mean = S / (float)d;
      const float ms = mean + eps;
      const float rs = 1.0f / std::sqrt(ms);
      rstd[t] = rs;
      for (int64_t j = 0; j < d; ++j) n[t * d + j] = ((float)xr[j] * rs) * (float)g[j];
    } else {
      double S = 0.0;
      for (int64_t j = 0; j < d; ++j) S += xr[j] * xr[j];
      const double rs = 1.0 / std::sqrt(S / (double)d + (double)eps);
      rstd[t] = rs;
      for (int64_t j = 0; j < d; ++j) n[t * d + j] = xr[j] * rs * g[j];
    }
  }
}

// ----------------------------------------------------------------------------
// SwiGLU forward: a = silu(gate) * up, silu(h) = h / (1 + e^-h).
// H is [T, 2f] with the gate half in columns [0, f) and the up half in [f, 2f).
// Quantized mode: fp32, e = exp_ref(-h), den = 1 + e, sil = h / den, a = sil*u.
// ----------------------------------------------------------------------------
std::vector<double> swiglu_fwd(const std::vector<double>& H, int64_t T, int64_t f, bool exact) {
  std::vector<double> a((size_t)(T * f));
  for (int64_t t = 0; t < T; ++t)
    for (int64_t j = 0; j < f; ++j) {
      const double h = H[t * 2 * f + j], u = H[t * 2 * f + f + j];
      if (!exact) {
        const float hf = (float)h, uf = (float)u;
        const float e = exp_ref(-hf);
        const float den = 1.0f + e;
        const float sil = hf / den;
        a[t * f + j] = sil * uf;
      } else {
        a[t * f + j] = h / (1.0 + std::exp(-h)) * u;
      }
    }
  return a;
}

// ----------------------------------------------------------------------------
// The MLP block.  Forward (LLMQ §1, §3, §3.1; FastML report):
//   Wgu8 = q(W_gu), Wd8 = q(W_d)                         E4M3, per tensor
//   n = RMSNorm(x) * g ; n8 = q(n)                       E4M3
//   H = bf16(alpha1 * n8 @ Wgu8)                         [T, 2f] gate | up
//   a = silu(H_gate) * H_up ; a8 = q(a)                  E4M3
//   y = bf16(x + alpha2 * a8 @ Wd8)                      residual
// Backward (straight-through quantizers; gradients E5M2 per LLMQ §5 Fig. 2, or
// E4M3 -- the recipe that figure shows tracking BF16 -- when grad_fmt says so):
//   dY8 = q5(dY)
//   dA  = alpha3 * dY8 @ Wd8^T                           (fp32 in registers on a GPU)
//   dH_gate = dA * up * s * (1 + h (1 - s)), dH_up = dA * silu(h), s = sigmoid(h)
//   dH = bf16(dH) ; dH8 = q5(dH)
//   dW_d  = alpha4 * a8^T @ dY8                          fp32
//   dN    = alpha5 * dH8 @ Wgu8^T                        fp32
//   dW_gu = alpha6 * n8^T @ dH8                          fp32
//   nh = x * rstd ; u = dN * g
//   dX = bf16(dY + rstd * (u - nh * mean_j(u * nh))) ; dg = sum_t dN * nh
// ----------------------------------------------------------------------------
struct BlockIO {
  int64_t T, d, f;
  float eps;
  int exact;
  int nthreads;
  int grad_fmt;  // format of the quantized gradients (E5M2 by default, E4M3 for LLMQ's E4M3-everywhere recipe)
  // inputs, [T,d] [d] [d,2f] [f,d] (and dY [T,d] for backward), as doubles
  const double* x; const double* g; const double* Wgu; const double* Wd; const double* dY;
  // forward outputs (doubles hold the stored value: bf16 / fp32 / decoded code)
  double* y; double* H; double* rstd;
  uint8_t* Wgu8; uint8_t* Wd8; uint8_t* n8; uint8_t* a8;
  float* scal_fwd;   // 4 x (amax, scale, scale_inv): W_gu, W_d, n, a
  // backward outputs
  double* dX; double* dWgu; double* dWd; double* dg; double* dN; double* dH;
  uint8_t* dY8; uint8_t* dH8;
  float* scal_bwd;   // 2 x (amax, scale, scale_inv): dY, dH
  // BF16 baseline (LLMQ §4/§5 measure FP8 training against BF16 training):
  // every operand the FP8 block casts is instead stored as bf16, scale 1
  int bf16;
  double* n16;       // [T,d] the stored bf16 n (bf16 mode)
  double* a16;       // [T,f] the stored bf16 a (bf16 mode)
  // Block-scaled MXFP8 (mx != 0; LLMQ §2): every GEMM operand is block-scaled
  // along that GEMM's contraction dimension instead of per tensor, so a tensor
  // that two GEMMs contract along different dimensions is quantized twice.
  // Slots (kMx*): codes [same shape as the tensor] in mxq, E8M0 codes in mxs
  // ([R][C/32] for blocks along a row, [R/32][C] for blocks along a column).
  int mx;
  uint8_t* mxq[12];
  uint8_t* mxs[12];
};

// MX operand slots: tensor, then the direction of its blocks ("_r": 32
// consecutive columns of a row, "_c": 32 consecutive rows of a column).
enum MxSlot {
  kMxWgu_r = 0,  // W_gu [d,2f] along 2f: the gate/up dgrad dN = dH W_gu^T
  kMxWgu_c,      // along d: the gate/up GEMM H = n W_gu
  kMxWd_r,       // W_d [f,d] along d: the down dgrad dA = dY W_d^T
  kMxWd_c,       // along f: the down GEMM y = x + a W_d
  kMxN_r,        // n [T,d] along d: the gate/up GEMM
  kMxN_c,        // along T: the gate/up wgrad dW_gu = n^T dH
  kMxA_r,        // a [T,f] along f: the down GEMM
  kMxA_c,        // along T: the down wgrad dW_d = a^T dY
  kMxDY_r,       // dY [T,d] along d: the down dgrad
  kMxDY_c,       // along T: the down wgrad
  kMxDH_r,       // dH [T,2f] along 2f: the gate/up dgrad
  kMxDH_c,       // along T: the gate/up wgrad
  kMxSlots
};

void put_scal(float* dst, const Scal& s) { dst[0] = s.amax; dst[1] = s.scale; dst[2] = s.scale_inv; }

template <class T> void put(T* dst, const std::vector<T>& v) {
  if (dst) std::copy(v.begin(), v.end(), dst);
}

// An operand of the block's GEMMs: in the FP8 block the per-tensor absmax
// quantization; in the BF16 baseline one round-to-nearest-even to bf16 with
// scale 1 (a no-op for tensors that already are bf16: weights, dY, dH).
QTensor operand(const std::vector<double>& v, int fmt, const BlockIO& io) {
  if (!io.bf16) return quantize(v, fmt, io.exact != 0);
  QTensor q;
  q.s = {abs_max(v), 1.0f, 1.0f};
  q.deq.resize(v.size());
  for (size_t i = 0; i < v.size(); ++i) q.deq[i] = to_bf16(v[i]);
  return q;
}

struct FwdState {
  QTensor Wgu, Wd, n, a;
  std::vector<double> nval, rstd, H, y;
  MxTensor mx[kMxSlots];  // MX mode: the forward's slots (W_gu, W_d, n, a)
  int status = 0;
};

void put_mx(const BlockIO& io, int slot, const MxTensor& t) {
  if (io.mxq[slot]) std::copy(t.code.begin(), t.code.end(), io.mxq[slot]);
  if (io.mxs[slot]) std::copy(t.sf.begin(), t.sf.end(), io.mxs[slot]);
}

// The MX forward: the same steps as block_forward with every per-tensor
// quantization replaced by the block quantization along the GEMM's contraction
// dimension (no alpha: the block scales are part of each operand's value).
FwdState block_forward_mx(const BlockIO& io) {
  const int64_t T = io.T, d = io.d, f = io.f;
  FwdState S;
  std::vector<double> x(io.x, io.x + T * d), g(io.g, io.g + d);
  std::vector<double> Wgu(io.Wgu, io.Wgu + d * 2 * f), Wd(io.Wd, io.Wd + f * d);
  S.mx[kMxWgu_c] = mx_quantize(Wgu, d, 2 * f, FMT_E4M3, true);
  S.mx[kMxWgu_r] = mx_quantize(Wgu, d, 2 * f, FMT_E4M3, false);
  S.mx[kMxWd_c] = mx_quantize(Wd, f, d, FMT_E4M3, true);
  S.mx[kMxWd_r] = mx_quantize(Wd, f, d, FMT_E4M3, false);
  rmsnorm_fwd(x, g, T, d, io.eps, false, S.nval, S.rstd);
  S.mx[kMxN_r] = mx_quantize(S.nval, T, d, FMT_E4M3, false);
  S.mx[kMxN_c] = mx_quantize(S.nval, T, d, FMT_E4M3, true);

  std::vector<double> acc1 = matmul(S.mx[kMxN_r].deq, S.mx[kMxWgu_c].deq, T, 2 * f, d, io.nthreads);
  S.H.resize(acc1.size());
  for (size_t i = 0; i < acc1.size(); ++i) S.H[i] = to_bf16(acc1[i]);

  std::vector<double> a = swiglu_fwd(S.H, T, f, false);
  S.mx[kMxA_r] = mx_quantize(a, T, f, FMT_E4M3, false);
  S.mx[kMxA_c] = mx_quantize(a, T, f, FMT_E4M3, true);

  std::vector<double> acc2 = matmul(S.mx[kMxA_r].deq, S.mx[kMxWd_c].deq, T, d, f, io.nthreads);
  S.y.resize(acc2.size());
  for (size_t i = 0; i < acc2.size(); ++i) S.y[i] = to_bf16(x[i] + acc2[i]);
  for (int k = kMxWgu_r; k <= kMxA_c; ++k) S.status |= S.mx[k].status;
  return S;
}

// status bit 1: a tensor's absmax was not finite
FwdState block_forward(const BlockIO& io) {
  if (io.mx) return block_forward_mx(io);
  const int64_t T = io.T, d = io.d, f = io.f;
  const bool ex = io.exact != 0;
  FwdState S;
  std::vector<double> x(io.x, io.x + T * d), g(io.g, io.g + d);
  std::vector<double> Wgu(io.Wgu, io.Wgu + d * 2 * f), Wd(io.Wd, io.Wd + f * d);

  S.Wgu = operand(Wgu, FMT_E4M3, io);
  S.Wd = operand(Wd, FMT_E4M3, io);
  rmsnorm_fwd(x, g, T, d, io.eps, ex, S.nval, S.rstd);
  S.n = operand(S.nval, FMT_E4M3, io);

  const double alpha1 = ex ? 1.0 : (double)(S.n.s.scale_inv * S.Wgu.s.scale_inv);
  std::vector<double> acc1 = matmul(S.n.deq, S.Wgu.deq, T, 2 * f, d, io.nthreads);
  S.H.resize(acc1.size());
  for (size_t i = 0; i < acc1.size(); ++i) S.H[i] = ex ? acc1[i] : to_bf16(alpha1 * acc1[i]);

  S.a = operand(swiglu_fwd(S.H, T, f, ex), FMT_E4M3, io);

  const double alpha2 = ex ? 1.0 : (double)(S.a.s.scale_inv * S.Wd.s.scale_inv);
  std::vector<double> acc2 = matmul(S.a.deq, S.Wd.deq, T, d, f, io.nthreads);
  S.y.resize(acc2.size());
  for (size_t i = 0; i < acc2.size(); ++i)
    S.y[i] = ex ? x[i] + acc2[i] : to_bf16(x[i] + alpha2 * acc2[i]);

  for (const Scal* s : {&S.Wgu.s, &S.Wd.s, &S.n.s, &S.a.s})
    if (!finite_scal(*s)) S.status |= 1;
  return S;
}

void write_forward(const BlockIO& io, const FwdState& S) {
  put(io.y, S.y);
  put(io.H, S.H);
  put(io.rstd, S.rstd);
  if (io.mx) {
    for (int k = kMxWgu_r; k <= kMxA_c; ++k) put_mx(io, k, S.mx[k]);
    return;
  }
  if (!io.exact) {
    put(io.Wgu8, S.Wgu.code); put(io.Wd8, S.Wd.code);
    put(io.n8, S.n.code); put(io.a8, S.a.code);
  }
  if (io.bf16) { put(io.n16, S.n.deq); put(io.a16, S.a.deq); }
  if (io.scal_fwd) {
    put_scal(io.scal_fwd + 0, S.Wgu.s); put_scal(io.scal_fwd + 3, S.Wd.s);
    put_scal(io.scal_fwd + 6, S.n.s); put_scal(io.scal_fwd + 9, S.a.s);
  }
}

// SwiGLU backward at the bf16 storage point: dH from dA and the stored H.
std::vector<double> swiglu_bwd(const std::vector<double>& H, const std::vector<double>& dA, int64_t T, int64_t f,
                               bool ex) {
  std::vector<double> dH((size_t)(T * 2 * f));
  for (int64_t t = 0; t < T; ++t)
    for (int64_t j = 0; j < f; ++j) {
      const double h = H[t * 2 * f + j], u = H[t * 2 * f + f + j];
      const double da = dA[t * f + j];
      const double sg = 1.0 / (1.0 + std::exp(-h));
      const double dg_ = da * u * sg * (1.0 + h * (1.0 - sg));
      const double du_ = da * h * sg;
      dH[t * 2 * f + j] = ex ? dg_ : to_bf16(dg_);
      dH[t * 2 * f + f + j] = ex ? du_ : to_bf16(du_);
    }
  return dH;
}

void rmsnorm_bwd(const std::vector<double>& x, const std::vector<double>& g, const std::vector<double>& rstd,
                 const std::vector<double>& dN, const std::vector<double>& dres, int64_t T, int64_t d, bool ex,
                 std::vector<double>& dX, std::vector<double>& dg);

// The MX backward: the block_backward steps with block-scaled operands; each
// GEMM takes the quantization of its operands along its own contraction
// dimension (the wgrad GEMMs contract over tokens).
int block_backward_mx(const BlockIO& io, const FwdState& S) {
  const int64_t T = io.T, d = io.d, f = io.f;
  int status = S.status;
  std::vector<double> x(io.x, io.x + T * d), g(io.g, io.g + d), dY(io.dY, io.dY + T * d);
  const int gf = io.grad_fmt;
  MxTensor dY_r = mx_quantize(dY, T, d, gf, false), dY_c = mx_quantize(dY, T, d, gf, true);

  std::vector<double> dA = matmul(dY_r.deq, transpose(S.mx[kMxWd_r].deq, f, d), T, f, d, io.nthreads);
  std::vector<double> dH = swiglu_bwd(S.H, dA, T, f, false);
  MxTensor dH_r = mx_quantize(dH, T, 2 * f, gf, false), dH_c = mx_quantize(dH, T, 2 * f, gf, true);

  std::vector<double> dWd = matmul(transpose(S.mx[kMxA_c].deq, T, f), dY_c.deq, f, d, T, io.nthreads);
  for (double& v : dWd) v = (double)(float)v;
  std::vector<double> dN = matmul(dH_r.deq, transpose(S.mx[kMxWgu_r].deq, d, 2 * f), T, d, 2 * f, io.nthreads);
  for (double& v : dN) v = (double)(float)v;
  std::vector<double> dWgu = matmul(transpose(S.mx[kMxN_c].deq, T, d), dH_c.deq, d, 2 * f, T, io.nthreads);
  for (double& v : dWgu) v = (double)(float)v;

  std::vector<double> dX, dgv;
  rmsnorm_bwd(x, g, S.rstd, dN, dY, T, d, false, dX, dgv);
  for (const MxTensor* t : {&dY_r, &dY_c, &dH_r, &dH_c}) status |= t->status;

  put(io.dX, dX); put(io.dWgu, dWgu); put(io.dWd, dWd); put(io.dg, dgv);
  put(io.dN, dN); put(io.dH, dH);
  put_mx(io, kMxDY_r, dY_r); put_mx(io, kMxDY_c, dY_c); put_mx(io, kMxDH_r, dH_r); put_mx(io, kMxDH_c, dH_c);
  return status;
}

int block_backward(const BlockIO& io, const FwdState& S) {
  if (io.mx) return block_backward_mx(io, S);
  const int64_t T = io.T, d = io.d, f = io.f;
  const bool ex = io.exact != 0;
  int status = S.status;
  std::vector<double> x(io.x, io.x + T * d), g(io.g, io.g + d), dY(io.dY, io.dY + T * d);

  const int gf = io.grad_fmt;
  QTensor dY8 = operand(dY, gf, io);

  // dA = alpha3 * dY8 @ Wd8^T   ([T,d] x [d,f])
  const double alpha3 = ex ? 1.0 : (double)(dY8.s.scale_inv * S.Wd.s.scale_inv);
  std::vector<double> WdT = transpose(S.Wd.deq, f, d);
  std::vector<double> dA = matmul(dY8.deq, WdT, T, f, d, io.nthreads);
  for (double& v : dA) v *= alpha3;

  std::vector<double> dH((size_t)(T * 2 * f));
  for (int64_t t = 0; t < T; ++t)
    for (int64_t j = 0; j < f; ++j) {
      const double h = S.H[t * 2 * f + j], u = S.H[t * 2 * f + f + j];
      const double da = dA[t * f + j];
      const double sg = 1.0 / (1.0 + std::exp(-h));
      double dg_ = da * u * sg * (1.0 + h * (1.0 - sg));
      double du_ = da * h * sg;
      dH[t * 2 * f + j] = ex ? dg_ : to_bf16(dg_);
      dH[t * 2 * f + f + j] = ex ? du_ : to_bf16(du_);
    }
  QTensor dH8 = operand(dH, gf, io);

  auto out32 = [&](double v) { return ex ? v : (double)(float)v; };

  // dW_d = alpha4 * a8^T @ dY8   ([f,T] x [T,d])
  const double alpha4 = ex ? 1.0 : (double)(S.a.s.scale_inv * dY8.s.scale_inv);
  std::vector<double> dWd = matmul(transpose(S.a.deq, T, f), dY8.deq, f, d, T, io.nthreads);
  for (double& v : dWd) v = out32(alpha4 * v);

  // dN = alpha5 * dH8 @ Wgu8^T   ([T,2f] x [2f,d])
  const double alpha5 = ex ? 1.0 : (double)(dH8.s.scale_inv * S.Wgu.s.scale_inv);
  std::vector<double> dN = matmul(dH8.deq, transpose(S.Wgu.deq, d, 2 * f), T, d, 2 * f, io.nthreads);
  for (double& v : dN) v = out32(alpha5 * v);

  // dW_gu = alpha6 * n8^T @ dH8  ([d,T] x [T,2f])
  const double alpha6 = ex ? 1.0 : (double)(S.n.s.scale_inv * dH8.s.scale_inv);
  std::vector<double> dWgu = matmul(transpose(S.n.deq, T, d), dH8.deq, d, 2 * f, T, io.nthreads);
  for (double& v : dWgu) v = out32(alpha6 * v);

  // RMSNorm backward + residual
  std::vector<double> dX((size_t)(T * d)), dgv((size_t)d, 0.0);
  for (int64_t t = 0; t < T; ++t) {
    const double rs = S.rstd[t];
    double dot = 0.0;
    for (int64_t j = 0; j < d; ++j) {
      const double nh = x[t * d + j] * rs;
      dot += dN[t * d + j] * g[j] * nh;
    }
    dot /= (double)d;
    for (int64_t j = 0; j < d; ++j) {
      const double nh = x[t * d + j] * rs;
      const double u = dN[t * d + j] * g[j];
      const double v = dY[t * d + j] + rs * (u - nh * dot);
      dX[t * d + j] = ex ? v : to_bf16(v);
      dgv[j] += dN[t * d + j] * nh;
    }
  }
  if (!ex) for (double& v : dgv) v = (double)(float)v;

  for (const Scal* s : {&dY8.s, &dH8.s})
    if (!finite_scal(*s)) status |= 1;

  put(io.dX, dX); put(io.dWgu, dWgu); put(io.dWd, dWd); put(io.dg, dgv);
  put(io.dN, dN); put(io.dH, dH);
  if (!ex) { put(io.dY8, dY8.code); put(io.dH8, dH8.code); }
  if (io.scal_bwd) { put_scal(io.scal_bwd + 0, dY8.s); put_scal(io.scal_bwd + 3, dH8.s); }
  return status;
}

// ----------------------------------------------------------------------------
// The attention core between the QKV and O projections (LLMQ §2/§3 name the
// transformer block's attention; the pages fix no attention arithmetic, so this
// is plain causal softmax attention with grouped K/V heads, in fp64):
//   qkv row of token t = [q_0 .. q_{Hq-1} | k_0 .. k_{Hkv-1} | v_0 .. v_{Hkv-1}], dh each
//   tokens form B sequences of S consecutive tokens; query position i sees keys 0..i
//   of its own sequence; q head h reads kv head h / (Hq / Hkv)
//   s_ik = (q_i . k_k) / sqrt(dh);  P = softmax over k;  att_i = sum_k P_ik v_k
//   att = bf16(att) (exact mode: unrounded);  lse_i = m_i + log(sum_k e^(s_ik - m_i))
// Backward (d_att = dO given; the plain gradient of the definition above):
//   dP_ik = dO_i . v_k;  D_i = sum_k P_ik dP_ik;  dS_ik = P_ik (dP_ik - D_i)
//   dq_i = sum_k dS_ik k_k / sqrt(dh);  dk_k = sum over the group's heads and i of
//   dS_ik q_i / sqrt(dh);  dv_k = sum over the group's heads and i of P_ik dO_i
//   dqkv = bf16 (exact mode: unrounded)
// ----------------------------------------------------------------------------
struct AttnIO {
  int64_t B, S, Hq, Hkv, dh;
  int exact;
  int nthreads;
  const double* qkv;    // [B*S, (Hq + 2 Hkv) dh]
  double* att;          // [B*S, Hq dh]
  double* lse;          // [Hq, B*S]
  const double* d_att;  // [B*S, Hq dh] (backward)
  double* dqkv;         // [B*S, (Hq + 2 Hkv) dh] (backward)
  double* att_abs;      // optional [B*S, Hq dh]: sum_k P_ik |v_k| (the size of the terms of att_i)
  // optional [B*S, (Hq + 2 Hkv) dh], the size of the terms of each gradient when P, dS and att
  // carry relative errors (Dabs_i = sum_c |dO_ic| (att_abs_ic + |att_ic|) bounds D's error scale):
  //   dq: sum_k |k_k| (|dS_ik| + P_ik Dabs_i) / sqrt(dh); dk: the same over i with |q_i|;
  //   dv: sum_i P_ik |dO_i|
  double* dqkv_abs;
};

// P row of (sequence b, head h, query i): probabilities of keys 0..i (fp64).
void attn_probs(const AttnIO& io, int64_t b, int64_t h, int64_t i, std::vector<double>& p, double* lse) {
  const int64_t nq = (io.Hq + 2 * io.Hkv) * io.dh, kvh = h / (io.Hq / io.Hkv);
  const double sc = 1.0 / std::sqrt((double)io.dh);
  const double* q = io.qkv + (b * io.S + i) * nq + h * io.dh;
  p.assign((size_t)(i + 1), 0.0);
  double m = -INFINITY;
  for (int64_t k = 0; k <= i; ++k) {
    const double* kr = io.qkv + (b * io.S + k) * nq + (io.Hq + kvh) * io.dh;
    double dot = 0.0;
    for (int64_t c = 0; c < io.dh; ++c) dot += q[c] * kr[c];
    p[k] = dot * sc;
    m = std::max(m, p[k]);
  }
  double l = 0.0;
  for (int64_t k = 0; k <= i; ++k) { p[k] = std::exp(p[k] - m); l += p[k]; }
  for (int64_t k = 0; k <= i; ++k) p[k] /= l;
  if (lse) *lse = m + std::log(l);
}

void attn_fwd_heads(const AttnIO* io, int64_t w0, int64_t w1) {
  const int64_t nq = (io->Hq + 2 * io->Hkv) * io->dh, da = io->Hq * io->dh, T = io->B * io->S;
  std::vector<double> p;
  for (int64_t w = w0; w < w1; ++w) {   // w = b * Hq + h
    const int64_t b = w / io->Hq, h = w % io->Hq, kvh = h / (io->Hq / io->Hkv);
    for (int64_t i = 0; i < io->S; ++i) {
      double lse = 0.0;
      attn_probs(*io, b, h, i, p, &lse);
      double* o = io->att + (b * io->S + i) * da + h * io->dh;
      for (int64_t c = 0; c < io->dh; ++c) {
        double acc = 0.0, aabs = 0.0;
        for (int64_t k = 0; k <= i; ++k) {
          const double v = io->qkv[(b * io->S + k) * nq + (io->Hq + io->Hkv + kvh) * io->dh + c];
          acc += p[k] * v;
          aabs += p[k] * std::fabs(v);
        }
        o[c] = io->exact ? acc : to_bf16(acc);
        if (io->att_abs) io->att_abs[(b * io->S + i) * da + h * io->dh + c] = aabs;
      }
      if (io->lse) io->lse[h * T + b * io->S + i] = lse;
    }
  }
}

// One (sequence, kv head) group per work item: every dq of the group's heads and the
// group's dk, dv (sums over its heads in a fixed order).
void attn_bwd_groups(const AttnIO* io, int64_t w0, int64_t w1) {
  const int64_t nq = (io->Hq + 2 * io->Hkv) * io->dh, da = io->Hq * io->dh, dh = io->dh;
  const int64_t rep = io->Hq / io->Hkv;
  const double sc = 1.0 / std::sqrt((double)dh);
  std::vector<double> p, dp;
  for (int64_t w = w0; w < w1; ++w) {   // w = b * Hkv + kvh
    const int64_t b = w / io->Hkv, kvh = w % io->Hkv;
    std::vector<double> dk((size_t)(io->S * dh), 0.0), dv((size_t)(io->S * dh), 0.0);
    std::vector<double> dka(io->dqkv_abs ? (size_t)(io->S * dh) : 0, 0.0), dva(dka.size(), 0.0);
    auto krow = [&](int64_t k) { return io->qkv + (b * io->S + k) * nq + (io->Hq + kvh) * dh; };
    auto vrow = [&](int64_t k) { return io->qkv + (b * io->S + k) * nq + (io->Hq + io->Hkv + kvh) * dh; };
    for (int64_t h = kvh * rep; h < (kvh + 1) * rep; ++h)
      for (int64_t i = 0; i < io->S; ++i) {
        attn_probs(*io, b, h, i, p, nullptr);
        const double* q = io->qkv + (b * io->S + i) * nq + h * dh;
        const double* dO = io->d_att + (b * io->S + i) * da + h * dh;
        dp.assign((size_t)(i + 1), 0.0);
        double D = 0.0;
        for (int64_t k = 0; k <= i; ++k) {
          const double* v = vrow(k);
          double acc = 0.0;
          for (int64_t c = 0; c < dh; ++c) acc += dO[c] * v[c];
          dp[k] = acc;
          D += p[k] * acc;
        }
        double Dabs = 0.0;
        if (io->dqkv_abs) {
          for (int64_t c = 0; c < dh; ++c) {
            double o = 0.0, oa = 0.0;
            for (int64_t k = 0; k <= i; ++k) {
              o += p[k] * vrow(k)[c];
              oa += p[k] * std::fabs(vrow(k)[c]);
            }
            Dabs += std::fabs(dO[c]) * (oa + std::fabs(o));
          }
          double* dqa = io->dqkv_abs + (b * io->S + i) * nq + h * dh;
          for (int64_t c = 0; c < dh; ++c) dqa[c] = 0.0;
          for (int64_t k = 0; k <= i; ++k) {
            const double w = std::fabs(p[k] * (dp[k] - D)) + p[k] * Dabs;
            const double* kr = krow(k);
            for (int64_t c = 0; c < dh; ++c) {
              dqa[c] += w * std::fabs(kr[c]) * sc;
              dka[k * dh + c] += w * std::fabs(q[c]) * sc;
              dva[k * dh + c] += p[k] * std::fabs(dO[c]);
            }
          }
        }
        double* dq = io->dqkv + (b * io->S + i) * nq + h * dh;
        for (int64_t c = 0; c < dh; ++c) dq[c] = 0.0;
        for (int64_t k = 0; k <= i; ++k) {
          const double ds = p[k] * (dp[k] - D);
          const double* kr = krow(k);
          for (int64_t c = 0; c < dh; ++c) {
            dq[c] += ds * kr[c] * sc;
            dk[k * dh + c] += ds * q[c] * sc;
            dv[k * dh + c] += p[k] * dO[c];
          }
        }
        if (!io->exact) for (int64_t c = 0; c < dh; ++c) dq[c] = to_bf16(dq[c]);
      }
    for (int64_t k = 0; k < io->S; ++k)
      for (int64_t c = 0; c < dh; ++c) {
        double* row = io->dqkv + (b * io->S + k) * nq;
        row[(io->Hq + kvh) * dh + c] = io->exact ? dk[k * dh + c] : to_bf16(dk[k * dh + c]);
        row[(io->Hq + io->Hkv + kvh) * dh + c] = io->exact ? dv[k * dh + c] : to_bf16(dv[k * dh + c]);
        if (io->dqkv_abs) {
          double* ra = io->dqkv_abs + (b * io->S + k) * nq;
          ra[(io->Hq + kvh) * dh + c] = dka[k * dh + c];
          ra[(io->Hq + io->Hkv + kvh) * dh + c] = dva[k * dh + c];
        }
      }
  }
}

template <class F>
void parallel_items(int64_t n, int nthreads, F fn) {
  nthreads = std::max(1, std::min<int>(nthreads, (int)std::max<int64_t>(n, 1)));
  if (nthreads == 1) { fn(0, n); return; }
  std::vector<std::thread> pool;
  for (int t = 0; t < nthreads; ++t) pool.emplace_back(fn, n * t / nthreads, n * (t + 1) / nthreads);
  for (auto& th : pool) th.join();
}

int attention(const AttnIO& io, bool backward) {
  if (io.B < 1 || io.S < 1 || io.Hq < 1 || io.Hkv < 1 || io.dh < 1 || io.Hq % io.Hkv) return 2;
  parallel_items(io.B * io.Hq, io.nthreads, [&](int64_t a, int64_t b) { attn_fwd_heads(&io, a, b); });
  if (backward)
    parallel_items(io.B * io.Hkv, io.nthreads, [&](int64_t a, int64_t b) { attn_bwd_groups(&io, a, b); });
  return 0;
}

// ----------------------------------------------------------------------------
// The full transformer block's matmuls (the 32B-class workload).  The attention
// core itself is not part of this path: its output `att` [T,d] and the gradient
// arriving at its input `dQKV` [T,nq] are given tensors.  Reading of the block:
//   forward   W_qkv8 = q(W_qkv), W_o8 = q(W_o)                     E4M3
//             n1 = RMSNorm(x) * g1, n1_8 = q(n1)
//             qkv = bf16(alpha n1_8 @ W_qkv8)                      [T, nq], feeds the core
//             att8 = q(att);  h = bf16(x + alpha att8 @ W_o8)      attention residual
//             y = MLP block on h (gain g2)
//   backward  dh = the MLP block's input gradient
//             dh8 = q5(dh);  d_att = bf16(alpha dh8 @ W_o8^T);  dW_o = alpha att8^T @ dh8
//             dQKV8 = q5(dQKV); dN1 = alpha dQKV8 @ W_qkv8^T;  dW_qkv = alpha n1_8^T @ dQKV8
//             dX = bf16(dh + RMSNorm'(dN1));  dg1 = sum_t dN1 * x * rstd1
// ----------------------------------------------------------------------------
struct FullIO {
  int64_t T, d, f, nq;
  float eps;
  int exact;
  int nthreads;
  const double* att;    // [T,d]
  const double* g1;     // [d]
  const double* Wqkv;   // [d,nq]
  const double* Wo;     // [d,d]
  const double* dQKV;   // [T,nq] (backward)
  double* qkv;          // [T,nq]
  double* h;            // [T,d]  (the MLP's input; io_mlp.x must point here)
  double* rstd1;        // [T]
  uint8_t* Wqkv8; uint8_t* Wo8; uint8_t* n1_8; uint8_t* att8;
  float* scal_attn;     // 6 x 3: W_qkv, W_o, n1, att, dh, dQKV
  double* dX; double* dWqkv; double* dWo; double* dg1; double* d_att; double* dh;
  uint8_t* dh8; uint8_t* dqkv8;
  BlockIO mlp;          // x = h (set by the caller), g, Wgu, Wd, dY and all MLP outputs
  const double* x;      // [T,d] block input
  // attention core (nonzero n_heads): att and dQKV are computed from qkv and d_att by the
  // core above instead of being given; d = n_heads * head_dim, T = n_seq * seq_len
  int64_t n_heads, n_kv_heads, head_dim, seq_len;
  double* att_out;      // [T,d] the core's output (bf16 values)
  double* lse;          // [n_heads, T]
  double* dqkv_out;     // [T,nq] the core's input gradient (bf16 values)
  double* n1_16;        // [T,d] the stored bf16 n1 (BF16 baseline, mlp.bf16)
};

// RMSNorm backward with a residual gradient: dx = dres + rstd (u - nh mean(u nh)), u = dN g.
void rmsnorm_bwd(const std::vector<double>& x, const std::vector<double>& g, const std::vector<double>& rstd,
                 const std::vector<double>& dN, const std::vector<double>& dres, int64_t T, int64_t d, bool ex,
                 std::vector<double>& dX, std::vector<double>& dg) {
  dX.assign((size_t)(T * d), 0.0);
  dg.assign((size_t)d, 0.0);
  for (int64_t t = 0; t < T; ++t) {
    const double rs = rstd[t];
    double dot = 0.0;
    for (int64_t j = 0; j < d; ++j) dot += dN[t * d + j] * g[j] * (x[t * d + j] * rs);
    dot /= (double)d;
    for (int64_t j = 0; j < d; ++j) {
      const double nh = x[t * d + j] * rs;
      const double u = dN[t * d + j] * g[j];
      const double v = dres[t * d + j] + rs * (u - nh * dot);
      dX[t * d + j] = ex ? v : to_bf16(v);
      dg[j] += dN[t * d + j] * nh;
    }
  }
  if (!ex) for (double& v : dg) v = (double)(float)v;
}

int full_block(FullIO& io, bool backward) {
  const int64_t T = io.T, d = io.d, nq = io.nq;
  const bool ex = io.exact != 0;
  const bool core = io.n_heads > 0;
  int status = 0;
  std::vector<double> x(io.x, io.x + T * d), g1(io.g1, io.g1 + d);
  // every operand goes through the MLP block's codec: per-tensor FP8, or bf16 in the BF16 baseline
  QTensor Wqkv = operand(std::vector<double>(io.Wqkv, io.Wqkv + d * nq), FMT_E4M3, io.mlp);
  QTensor Wo = operand(std::vector<double>(io.Wo, io.Wo + d * d), FMT_E4M3, io.mlp);
  std::vector<double> n1, rstd1;
  rmsnorm_fwd(x, g1, T, d, io.eps, ex, n1, rstd1);
  QTensor n1q = operand(n1, FMT_E4M3, io.mlp);

  const double a_qkv = ex ? 1.0 : (double)(n1q.s.scale_inv * Wqkv.s.scale_inv);
  std::vector<double> qkv = matmul(n1q.deq, Wqkv.deq, T, nq, d, io.nthreads);
  for (double& v : qkv) v = ex ? a_qkv * v : to_bf16(a_qkv * v);

  std::vector<double> att, lse;
  AttnIO aio{};
  if (core) {
    if (io.n_heads * io.head_dim != d || (io.n_heads + 2 * io.n_kv_heads) * io.head_dim != nq ||
        io.seq_len < 1 || T % io.seq_len)
      return 2;
    att.assign((size_t)(T * d), 0.0);
    lse.assign((size_t)(io.n_heads * T), 0.0);
    aio = AttnIO{T / io.seq_len, io.seq_len, io.n_heads, io.n_kv_heads, io.head_dim, io.exact, io.nthreads,
                 qkv.data(), att.data(), lse.data(), nullptr, nullptr, nullptr, nullptr};
    if (attention(aio, false)) return 2;
    put(io.att_out, att);
    put(io.lse, lse);
  } else {
    att.assign(io.att, io.att + T * d);
  }
  QTensor attq = operand(att, FMT_E4M3, io.mlp);
  const double a_o = ex ? 1.0 : (double)(attq.s.scale_inv * Wo.s.scale_inv);
  std::vector<double> h = matmul(attq.deq, Wo.deq, T, d, d, io.nthreads);
  for (size_t i = 0; i < h.size(); ++i) h[i] = ex ? x[i] + a_o * h[i] : to_bf16(x[i] + a_o * h[i]);

  put(io.qkv, qkv);
  put(io.h, h);
  put(io.rstd1, rstd1);
  if (io.mlp.bf16) put(io.n1_16, n1q.deq);
  if (!ex) { put(io.Wqkv8, Wqkv.code); put(io.Wo8, Wo.code); put(io.n1_8, n1q.code); put(io.att8, attq.code); }
  if (io.scal_attn) {
    put_scal(io.scal_attn + 0, Wqkv.s); put_scal(io.scal_attn + 3, Wo.s);
    put_scal(io.scal_attn + 6, n1q.s); put_scal(io.scal_attn + 9, attq.s);
  }
  for (const Scal* sc : {&Wqkv.s, &Wo.s, &n1q.s, &attq.s})
    if (!finite_scal(*sc)) status |= 1;

  // the MLP block on h
  BlockIO m = io.mlp;
  m.x = h.data();
  FwdState S = block_forward(m);
  write_forward(m, S);
  status |= S.status;
  if (!backward) return status;
  std::vector<double> dh((size_t)(T * d));
  m.dX = dh.data();
  status |= block_backward(m, S);
  put(io.dh, dh);

  // O projection backward
  QTensor dhq = operand(dh, io.mlp.grad_fmt, io.mlp);
  const double a_od = ex ? 1.0 : (double)(dhq.s.scale_inv * Wo.s.scale_inv);
  std::vector<double> datt = matmul(dhq.deq, transpose(Wo.deq, d, d), T, d, d, io.nthreads);
  for (double& v : datt) v = ex ? a_od * v : to_bf16(a_od * v);
  const double a_ow = ex ? 1.0 : (double)(attq.s.scale_inv * dhq.s.scale_inv);
  std::vector<double> dWo = matmul(transpose(attq.deq, T, d), dhq.deq, d, d, T, io.nthreads);
  for (double& v : dWo) v = ex ? a_ow * v : (double)(float)(a_ow * v);

  // the attention core's backward: dQKV from d_att (else dQKV is given)
  std::vector<double> dqkv;
  if (core) {
    dqkv.assign((size_t)(T * nq), 0.0);
    aio.d_att = datt.data();
    aio.dqkv = dqkv.data();
    parallel_items(aio.B * aio.Hkv, aio.nthreads, [&](int64_t a, int64_t b) { attn_bwd_groups(&aio, a, b); });
    put(io.dqkv_out, dqkv);
  } else {
    dqkv.assign(io.dQKV, io.dQKV + T * nq);
  }

  // QKV projection backward
  QTensor dqq = operand(dqkv, io.mlp.grad_fmt, io.mlp);
  const double a_qd = ex ? 1.0 : (double)(dqq.s.scale_inv * Wqkv.s.scale_inv);
  std::vector<double> dN1 = matmul(dqq.deq, transpose(Wqkv.deq, d, nq), T, d, nq, io.nthreads);
  for (double& v : dN1) v = ex ? a_qd * v : (double)(float)(a_qd * v);
  const double a_qw = ex ? 1.0 : (double)(n1q.s.scale_inv * dqq.s.scale_inv);
  std::vector<double> dWqkv = matmul(transpose(n1q.deq, T, d), dqq.deq, d, nq, T, io.nthreads);
  for (double& v : dWqkv) v = ex ? a_qw * v : (double)(float)(a_qw * v);

  std::vector<double> dX, dg1;
  rmsnorm_bwd(x, g1, rstd1, dN1, dh, T, d, ex, dX, dg1);

  put(io.d_att, datt); put(io.dWo, dWo); put(io.dWqkv, dWqkv); put(io.dX, dX); put(io.dg1, dg1);
  if (!ex) { put(io.dh8, dhq.code); put(io.dqkv8, dqq.code); }
  if (io.scal_attn) { put_scal(io.scal_attn + 12, dhq.s); put_scal(io.scal_attn + 15, dqq.s); }
  for (const Scal* sc : {&dhq.s, &dqq.s})
    if (!finite_scal(*sc)) status |= 1;
  return status;
}

std::vector<double> load_input(const void* x, int dtype, int64_t n) {
  // dtype 0: bf16 bits, 1: fp32
  std::vector<double> v((size_t)n);
  if (dtype == 0) {
    const uint16_t* p = (const uint16_t*)x;
    for (int64_t i = 0; i < n; ++i) v[i] = bf16_value(p[i]);
  } else {
    const float* p = (const float*)x;
    for (int64_t i = 0; i < n; ++i) v[i] = (double)p[i];
  }
  return v;
}

}  // namespace

// ============================================================================
// C entry points (ctypes).  Status: 0 ok, bit 1 = non-finite absmax.
// ============================================================================
extern "C" {

int fo_abi_version() { return 1; }

uint8_t fo_fp8_encode(float v, int fmt) { return fp8_encode(v, fmt); }
double fo_fp8_decode(uint8_t c, int fmt) { return fp8_decode(c, fmt); }

void fo_fp8_encode_n(const float* v, int64_t n, int fmt, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = fp8_encode(v[i], fmt);
}
void fo_fp8_decode_n(const uint8_t* c, int64_t n, int fmt, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = fp8_decode(c[i], fmt);
}
void fo_bf16_round_n(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = to_bf16_bits(v[i]);
}

float fo_exp_ref(float x) { return exp_ref(x); }
void fo_exp_ref_n(const float* x, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = exp_ref(x[i]);
}

float fo_pairwise_sum(const float* v, int64_t n) { return pairwise_sum(v, n); }

// Per-tensor absmax quantization of n values (dtype 0 bf16 bits, 1 fp32).
// scal3 = (amax, scale, scale_inv).
int fo_quantize_absmax(const void* x, int dtype, int64_t n, int fmt, uint8_t* q, float* scal3) {
  QTensor t = quantize(load_input(x, dtype, n), fmt, false);
  std::copy(t.code.begin(), t.code.end(), q);
  put_scal(scal3, t.s);
  return finite_scal(t.s) ? 0 : 1;
}

// RMSNorm (gain g, epsilon eps) followed by per-tensor E4M3 quantization.
int fo_rmsnorm_quant(const uint16_t* x, const uint16_t* g, int64_t T, int64_t d, float eps,
                     uint8_t* q, float* scal3, float* rstd) {
  std::vector<double> n, rs;
  rmsnorm_fwd(load_input(x, 0, T * d), load_input(g, 0, d), T, d, eps, false, n, rs);
  QTensor t = quantize(n, FMT_E4M3, false);
  std::copy(t.code.begin(), t.code.end(), q);
  put_scal(scal3, t.s);
  for (int64_t i = 0; i < T; ++i) rstd[i] = (float)rs[i];
  return finite_scal(t.s) ? 0 : 1;
}

// RMSNorm backward with the residual gradient on given values: dX = dres + rstd (u - nh mean(u nh)),
// u = dN g, nh = x rstd; dg = sum over rows of dN nh.  dX is rounded to bf16 and dg to fp32 unless
// `exact` (then both are the fp64 values).
int fo_rmsnorm_bwd(const double* dN, const double* x, const double* g, const double* rstd, const double* dres,
                   int64_t T, int64_t d, int exact, double* dX, double* dg) {
  std::vector<double> X, G;
  rmsnorm_bwd(std::vector<double>(x, x + T * d), std::vector<double>(g, g + d), std::vector<double>(rstd, rstd + T),
              std::vector<double>(dN, dN + T * d), std::vector<double>(dres, dres + T * d), T, d, exact != 0, X, G);
  put(dX, X);
  put(dg, G);
  return 0;
}

// SwiGLU of H [T, 2f] (gate | up, bf16 bits) followed by per-tensor quantization.
int fo_swiglu_quant(const uint16_t* H, int64_t T, int64_t f, int fmt, uint8_t* q, float* scal3) {
  QTensor t = quantize(swiglu_fwd(load_input(H, 0, T * 2 * f), T, f, false), fmt, false);
  std::copy(t.code.begin(), t.code.end(), q);
  put_scal(scal3, t.s);
  return finite_scal(t.s) ? 0 : 1;
}

// C = alpha * op(A) op(B) (+ residual), alpha = fl32(sinvA * sinvB).
//   layout 0 NN: A [M,K], B [K,N];  1 NT: A [M,K], B [N,K];  2 TN: A [K,M], B [K,N]
// out_dtype 0: bf16 bits (with optional bf16 residual [M,N]), 1: fp32, 2: fp64
// (the unrounded alpha * acc, for tests).
int fo_gemm_scaled(int layout, int64_t M, int64_t N, int64_t K, const uint8_t* A, int fmtA,
                   const uint8_t* B, int fmtB, float sinvA, float sinvB, const uint16_t* residual,
                   int out_dtype, void* C, int nthreads) {
  std::vector<double> a((size_t)(M * K)), b((size_t)(K * N));
  for (int64_t i = 0; i < M; ++i)
    for (int64_t k = 0; k < K; ++k)
      a[i * K + k] = fp8_decode(layout == 2 ? A[k * M + i] : A[i * K + k], fmtA);
  for (int64_t k = 0; k < K; ++k)
    for (int64_t j = 0; j < N; ++j)
      b[k * N + j] = fp8_decode(layout == 1 ? B[j * K + k] : B[k * N + j], fmtB);
  std::vector<double> acc = matmul(a, b, M, N, K, nthreads);
  const double alpha = (double)(sinvA * sinvB);
  for (int64_t i = 0; i < M * N; ++i) {
    double v = alpha * acc[i];
    if (out_dtype == 0) {
      if (residual) v += bf16_value(residual[i]);
      ((uint16_t*)C)[i] = to_bf16_bits(v);
    } else if (out_dtype == 1) {
      ((float*)C)[i] = (float)v;
    } else {
      ((double*)C)[i] = v;
    }
  }
  return 0;
}

// Block quantization (MXFP8) of an R x C tensor (dtype 0 bf16 bits, 1 fp32):
// along_rows 0 = blocks of 32 consecutive columns of a row, sf [R][ceil(C/32)];
// 1 = blocks of 32 consecutive rows of a column, sf [ceil(R/32)][C].
int fo_mx_quantize(const void* x, int dtype, int64_t R, int64_t C, int fmt, int along_rows, uint8_t* q,
                   uint8_t* sf) {
  MxTensor t = mx_quantize(load_input(x, dtype, R * C), R, C, fmt, along_rows != 0);
  std::copy(t.code.begin(), t.code.end(), q);
  std::copy(t.sf.begin(), t.sf.end(), sf);
  return t.status;
}

// Block-scaled GEMM: C = op(A) op(B) (+ residual) with every element of A and B
// worth decode(code) * 2^(sf - 127) of its K-block of 32 (layouts as
// fo_gemm_scaled).  sfA is [M][ceil(K/32)] (block m, k), sfB [N][ceil(K/32)]
// (block n, k), whatever the operands' storage layout.
int fo_gemm_mx(int layout, int64_t M, int64_t N, int64_t K, const uint8_t* A, int fmtA, const uint8_t* sfA,
               const uint8_t* B, int fmtB, const uint8_t* sfB, const uint16_t* residual, int out_dtype, void* C,
               int nthreads) {
  const int64_t KB = (K + kMxBlock - 1) / kMxBlock;
  auto sfval = [](uint8_t c) { return c == 0xFF ? std::nan("") : std::ldexp(1.0, (int)c - 127); };
  std::vector<double> a((size_t)(M * K)), b((size_t)(K * N));
  for (int64_t i = 0; i < M; ++i)
    for (int64_t k = 0; k < K; ++k)
      a[i * K + k] = fp8_decode(layout == 2 ? A[k * M + i] : A[i * K + k], fmtA) * sfval(sfA[i * KB + k / kMxBlock]);
  for (int64_t k = 0; k < K; ++k)
    for (int64_t j = 0; j < N; ++j)
      b[k * N + j] = fp8_decode(layout == 1 ? B[j * K + k] : B[k * N + j], fmtB) * sfval(sfB[j * KB + k / kMxBlock]);
  std::vector<double> acc = matmul(a, b, M, N, K, nthreads);
  for (int64_t i = 0; i < M * N; ++i) {
    double v = acc[i];
    if (out_dtype == 0) {
      if (residual) v += bf16_value(residual[i]);
      ((uint16_t*)C)[i] = to_bf16_bits(v);
    } else if (out_dtype == 1) {
      ((float*)C)[i] = (float)v;
    } else {
      ((double*)C)[i] = v;
    }
  }
  return 0;
}

// Block forward / backward.  The struct layout is mirrored by oracle/__init__.py.
int fo_block_forward(const BlockIO* io) {
  FwdState S = block_forward(*io);
  write_forward(*io, S);
  return S.status;
}

// The full block's matmuls (attention core given as att / dQKV); the struct is
// mirrored by oracle/__init__.py.
int fo_full_block(FullIO* io, int backward) { return full_block(*io, backward != 0); }
int fo_attention(const AttnIO* io, int backward) { return attention(*io, backward != 0); }

int fo_block_forward_backward(const BlockIO* io) {
  FwdState S = block_forward(*io);
  write_forward(*io, S);
  return block_backward(*io, S);
}

}  // extern "C"
