// Internal launch interface between the C ABI (fp8q_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fp8q {

// Upper bound on the number of per-block absmax partials any reduction pass writes.
constexpr int kMaxPartials = 1024;
// Rows per block of the RMSNorm backward (one fp32 dg partial row per block).
constexpr int kBwdRows = 16;

struct Launch {
  cudaStream_t stream;
  unsigned* status;  // device status word (FP8Q_STATUS_* bits)
  int num_sms;
  int* launches;     // incremented once per kernel launch
};

// Device address of the library's status word and the SM count of the current
// device (resolved once per device).  Returns 0 on success.
int device_status_and_sms(unsigned** status, int* num_sms);

// Per-tensor absmax quantization: pass 1 writes *P partials, pass 2 casts.
// absmax_partial_blocks: the number of partials pass 1 writes for n elements (its grid size;
// never more than kMaxPartials).
int absmax_partial_blocks(int dtype, int64_t n);
cudaError_t launch_absmax_partial(const void* x, int dtype, int64_t n, uint32_t* partial, int* P,
                                  const Launch& L);
cudaError_t launch_quant_cast(const void* x, int dtype, int64_t n, int fmt, const uint32_t* partial, int P,
                              uint8_t* q, float* scal, const Launch& L);

// RMSNorm: pass 1 (rstd + absmax partials), pass 2 (cast to E4M3).
cudaError_t launch_rmsnorm_stats(const uint16_t* x, const uint16_t* g, int64_t T, int d, float eps, float* rstd,
                                 uint32_t* partial, int* P, const Launch& L);
// The forward's quantizer prologue in two launches: pass 1 (RMSNorm statistics of x | absmax
// partials of W_gu | of W_d), pass 2 (cast W_gu | cast W_d | cast n): the same results as the six
// separate launches (bf16 weights of n_wgu / n_wd elements -> E4M3; n8 from x, g, rstd).  Each
// partial array holds up to kMaxPartials.  Both passes take the same arguments.
cudaError_t launch_prologue(int pass, const uint16_t* x, const uint16_t* g, int64_t T, int d, float eps, float* rstd,
                            const uint16_t* W_gu, int64_t n_wgu, const uint16_t* W_d, int64_t n_wd,
                            uint32_t* part_n, uint32_t* part_wgu, uint32_t* part_wd, uint8_t* n8, float* s_n,
                            uint8_t* W_gu8, float* s_wgu, uint8_t* W_d8, float* s_wd, const Launch& L);
// BF16 baseline: one pass, rstd and n = bf16((x rstd) g) (no absmax, no cast).
cudaError_t launch_rmsnorm_bf16(const uint16_t* x, const uint16_t* g, int64_t T, int d, float eps, float* rstd,
                                uint16_t* n16, const Launch& L);
cudaError_t launch_rmsnorm_cast(const uint16_t* x, const uint16_t* g, const float* rstd, int64_t T, int d,
                                const uint32_t* partial, int P, uint8_t* q, float* scal, const Launch& L);

// SwiGLU of H [T,2f]: pass 1 (absmax partials of a), pass 2 (cast).
cudaError_t launch_swiglu_amax(const uint16_t* H, int64_t T, int f, uint32_t* partial, int* P, const Launch& L);
// fast: the fused forward's E4M3 cast, with a = swiglu_fast (as the gate/up GEMM's absmax saw it).
cudaError_t launch_swiglu_cast(const uint16_t* H, int64_t T, int f, int fmt, const uint32_t* partial, int P,
                               uint8_t* q, float* scal, const Launch& L, bool fast = false);

// RMSNorm backward + residual: dX = dY + rstd (u - nh mean(u nh)), dg = sum_t dN nh.
// dg_partial: ceil(T / kBwdRows) x d floats of workspace.  wait_ns: the limit of every wait on a
// row's copies (0: the default 2 s; otherwise the self-test of the abort sequence, whose waits
// probe without suspending so that a limit of nanoseconds is honoured).
cudaError_t launch_rmsnorm_bwd(const float* dN, const uint16_t* x, const uint16_t* dY, const uint16_t* g,
                               const float* rstd, int64_t T, int d, uint16_t* dX, float* dg_partial, float* dg,
                               const Launch& L, uint64_t wait_ns = 0);

// Attention core (bf16, causal, grouped K/V heads, head dim 128, S a multiple of 128).
cudaError_t launch_attn_fwd(const uint16_t* qkv, int64_t T, int S, int Hq, int Hkv, uint16_t* att, float* lse,
                            const Launch& L);
// Backward: D = rowsum(dO * att) and lse2 = lse log2(e) ([Hq, T] each), then dK/dV and dQ into dqkv.
cudaError_t launch_attn_bwd_delta(const uint16_t* att, const uint16_t* datt, const float* lse, int64_t T, int Hq,
                                  float* delta, float* lse2, const Launch& L);
cudaError_t launch_attn_bwd_dkdv(const uint16_t* qkv, const uint16_t* datt, int64_t T, int S, int Hq, int Hkv,
                                 const float* delta, const float* lse2, uint16_t* dqkv, const Launch& L);
cudaError_t launch_attn_bwd_dq(const uint16_t* qkv, const uint16_t* datt, int64_t T, int S, int Hq, int Hkv,
                               const float* delta, const float* lse2, uint16_t* dqkv, const Launch& L);

// Diagnostics: a bounded wait that is made to run out (see fp8q_selftest_bounded_wait).
cudaError_t launch_selftest_bounded_wait(uint64_t limit_ns, const Launch& L);

// Block-scaled (MXFP8) quantization of a [R, C] tensor, R and C multiples of 128, in one pass:
// q_r/sf_r (blocks of 32 along each row; the operand of a GEMM contracting over C) and/or
// q_c/sf_c (blocks of 32 down each column; contracting over R); either pair may be null.  Inputs:
// kMxInBf16 / kMxInF32 x [R, C]; kMxInSwiglu: bf16 H [R, 2C] (gate | up) -> a = SwiGLU(H);
// kMxInRmsnorm: bf16 x [R, C] with gain g [C] and rstd [R] -> n = fl32(fl32(x rstd) g).
// Scale codes go to the chunked layout the block-scaled GEMM reads (mx_scale_bytes bytes).
enum MxIn { kMxInBf16 = 0, kMxInF32 = 1, kMxInSwiglu = 2, kMxInRmsnorm = 3 };
size_t mx_scale_bytes(int64_t rows, int64_t K);
cudaError_t launch_mx_quant(int in_kind, const void* x, const uint16_t* g, const float* rstd, int64_t R, int64_t C,
                            int fmt, uint8_t* q_r, uint8_t* sf_r, uint8_t* q_c, uint8_t* sf_c, const Launch& L);

// Bookkeeping of the C ABI for entry points implemented outside fp8q_api.cu: the trace bracket
// of one kernel step (an NVTX range, and CUDA events while the kernel trace is on) and the count
// that fp8q_last_launch_count() reports.
enum TraceKind { kTraceAbsmaxPartial = 0, kTraceQuantCast = 1 };
bool trace_step_begin(cudaStream_t s, int kind);  // returns whether events were recorded
void trace_step_end(cudaStream_t s, bool active);
void set_last_launch_count(int n);

// ---------------------------------------------------------------------------
// GEMM
// ---------------------------------------------------------------------------
enum GemmEpilogue {
  kEpiStore = 0,      // C = alpha * acc (bf16 or fp32)
  kEpiResidual = 1,   // C = bf16(R + alpha * acc)
  kEpiSwiglu = 2,     // H = bf16(alpha * acc) for paired gate/up columns, absmax of a = SwiGLU(H)
  kEpiSwigluBwd = 3,  // dH = bf16(SwiGLU'(H) * alpha * acc) + absmax of dH
};

struct GemmProblem {
  int a_mn, b_mn;        // operand is MN-major (1) or K-major (0)
  int M, N, K;           // output rows/cols (kEpiSwiglu: N = f gate columns), reduction length
  const uint8_t* A; int64_t lda; int fmtA;
  const uint8_t* B; int64_t ldb; int fmtB;
  int64_t b_cols;        // extent of B's N dimension in storage (2f for the paired gate/up layout)
  const float* sinvA; const float* sinvB;
  int epi; int out_f32;
  void* C; int64_t ldc;  // kEpiSwiglu/kEpiSwigluBwd: [M, 2f] gate | up
  const uint16_t* R; int64_t ldr;  // residual (kEpiResidual) or H (kEpiSwigluBwd)
  const float* qscale;             // kEpiSwiglu: optional scale of a; a is written as E4M3 codes to q8
  uint8_t* q8;                     //   [M, N] E4M3
  uint32_t* amax_partial;          // per-CTA partials for the two SwiGLU epilogues
  int op16;                        // 1: bf16 operands (lda/ldb in elements), no scales (alpha = 1)
  uint16_t* a16;                   // op16 with kEpiSwiglu: bf16 SwiGLU output a [M, N]
  // Block-scaled MXFP8 (mx = 1): sinvA/sinvB unused (alpha = 1); sfA / sfB hold the E8M0 codes of
  // A (rows M) and B (rows b_cols) in the chunked layout of launch_mx_quant; K a multiple of 128.
  int mx;
  const uint8_t* sfA; const uint8_t* sfB;
  // Limit of the kernel's pipeline waits in ns (0: the default 2 s).  Only the GEMM self test sets
  // it, to a few microseconds, so that ordinary waits give up and the abort sequence runs.
  uint64_t wait_ns;
};
// Launches the persistent tcgen05 GEMM; *P receives the number of partials written.
cudaError_t launch_gemm(const GemmProblem& g, int* P, const Launch& L);

}  // namespace fp8q
