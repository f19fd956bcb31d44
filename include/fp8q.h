/*
 * fp8q.h -- C ABI of the GB300 (sm_103a) FP8 transformer-block pipeline with
 * just-in-time per-tensor absmax scaling.
 *
 * The operations follow the LLMQ pages:
 *   "LLMQ: Efficient Lower-Precision Pretraining for Consumer GPUs"
 *   (paperlayer.ai summary of arXiv 2512.15306), §1: FP8 training with dynamic
 *   tensor-level scaling; §3/§3.1/§3.2: fused non-matmul ops, retained absmax
 *   statistics for requantization, deterministic kernels; §4: dynamic
 *   quantization and backward transposes are the FP8 overheads; §5 Figure 2:
 *   E4M3 forward, E5M2 activation gradients.
 *   "Periodic Reporting for period 1 - FastML" (CORDIS), "FP8 training
 *   without delayed scaling": just-in-time tensor-level absmax scaling,
 *   guaranteeing no value clipping.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Memory: every pointer is a DEVICE pointer unless stated otherwise.  The
 *    caller owns all memory (inputs, outputs, workspace); the library never
 *    allocates or frees device memory.  Tensors are dense and row-major.
 *    bf16 tensors are passed as raw 16-bit storage.
 *  - Alignment: tensor base pointers must be 16-byte aligned.
 *  - Streams: every call only enqueues kernels on `stream` (a cudaStream_t;
 *    NULL is the legacy default stream) and never synchronizes with the host.
 *  - Scales: a "scal" argument points to 3 device floats
 *    {amax, scale, scale_inv}: amax = max |v| over the whole tensor,
 *    scale = fl32(fmt_max / amax) (1 when amax == 0), scale_inv = fl32(1/scale).
 *    A tensor is quantized as code = fp8_rne_satfinite(fl32(v * scale)), so
 *    the absmax element maps to +-fmt_max and nothing is clipped.
 *    fmt_max: E4M3 448, E5M2 57344.
 *  - Workspace: `ws`/`ws_bytes` is caller-provided device scratch of at least
 *    the size the matching *_workspace_size() function returns, 256-byte
 *    aligned; its contents need no initialisation and are garbage afterwards.
 *    Two calls that are in flight at the same time need distinct workspaces.
 *  - Synchronous errors (bad arguments) are returned before anything is
 *    enqueued.  Kernel launch failures return FP8Q_ERR_CUDA.  Conditions that
 *    are only known on the device (a non-finite amax; a bounded wait that ran
 *    out) are recorded in a per-device status word that fp8q_get_status()
 *    reads after the caller has synchronized the stream.
 *  - Determinism: the same inputs give the same output bits on the same GPU
 *    model (no floating-point atomics; fixed reduction orders).
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FP8Q_API __attribute__((visibility("default")))
#else
#define FP8Q_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP8Q_OK = 0,
  FP8Q_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or leading dimension   */
  FP8Q_ERR_UNSUPPORTED = 2,  /* valid request the library does not implement            */
  FP8Q_ERR_CUDA = 3,         /* a CUDA runtime/driver call or a kernel launch failed      */
  FP8Q_ERR_TIMEOUT = 4,      /* device status only: a bounded wait in a kernel ran out    */
  FP8Q_ERR_NONFINITE = 5,    /* device status only: a tensor's amax was Inf or NaN        */
  FP8Q_ERR_WORKSPACE = 6     /* workspace pointer null/misaligned or ws_bytes too small   */
} fp8q_status;

typedef enum { FP8Q_E4M3 = 0, FP8Q_E5M2 = 1 } fp8q_fmt;
typedef enum { FP8Q_BF16 = 0, FP8Q_F32 = 1 } fp8q_dtype;
/* Operand storage of fp8_gemm_scaled (C[M,N] = op(A) op(B), all row-major):
 *   NN: A [M,K], B [K,N]      NT: A [M,K], B [N,K]      TN: A [K,M], B [K,N]   */
typedef enum { FP8Q_NN = 0, FP8Q_NT = 1, FP8Q_TN = 2 } fp8q_layout;

typedef void* fp8q_stream; /* cudaStream_t */

/* Device status bits returned by fp8q_get_status. */
#define FP8Q_STATUS_NONFINITE 0x1u
#define FP8Q_STATUS_TIMEOUT 0x2u

/* ------------------------------------------------------------------------ */
/* Per-tensor absmax quantization (LLMQ §1 dynamic tensor-level scaling;    */
/* FastML report: just-in-time absmax scaling, no clipping).                */
/* ------------------------------------------------------------------------ */
/* x: n elements of x_dtype (bf16 or fp32); q: n codes of fmt; scal: 3 floats.
 * Two passes: a vectorised absmax reduction (warp shuffles, block reduction,
 * one partial per block in ws), then a cast pass that finalises the scale
 * from the partials and writes the codes.  Returns FP8Q_OK or a sync error. */
FP8Q_API size_t fp8_quantize_absmax_workspace_size(int64_t n);
FP8Q_API int fp8_quantize_absmax(const void* x, fp8q_dtype x_dtype, int64_t n, fp8q_fmt fmt, uint8_t* q,
                        float* scal, void* ws, size_t ws_bytes, fp8q_stream stream);

/* The same quantization for callers that cannot allocate device memory, so
 * cannot provide the workspace above: code inside a framework that owns every
 * allocation through its own pool and gives none to plug-ins, and
 * latency-critical loops that must avoid cudaMalloc/cudaFree because those
 * synchronize the device.  The paper has no counterpart; this is an interface
 * convenience.
 *
 * The scratch (1024 absmax partials, 4 KiB) is a fixed array in the library's
 * own device memory: one copy per GPU that loads the library, held until the
 * process exits.  Every call on a device shares it and it keeps the last
 * call's contents; nothing needs clearing (each call overwrites the partials
 * it reads).  Two calls whose kernels overlap on the GPU (different streams
 * without ordering) race on the array and give wrong results.  The first call
 * on each device looks up the array's device address (cudaGetSymbolAddress);
 * make that first call before any stream capture.  No cudaMalloc, cudaFree or
 * other allocating routine is called.  Inputs and outputs are the caller's, as
 * for fp8_quantize_absmax, with the same results bit for bit.  Returns
 * FP8Q_ERR_INVALID_ARG for bad arguments or a tensor that would need more
 * than the 1024 partials (the first pass is capped at 1024 blocks, so every
 * n >= 1 fits); a non-finite amax sets FP8Q_STATUS_NONFINITE as usual. */
FP8Q_API int fp8_quantize_absmax_noalloc(const void* x, fp8q_dtype x_dtype, int64_t n, fp8q_fmt fmt, uint8_t* q,
                                         float* scal, fp8q_stream stream);

/* ------------------------------------------------------------------------ */
/* Scaled FP8 GEMM (LLMQ §4: FP8 matmuls dominate; backward dgrad/wgrad use  */
/* the transposed layouts without separate transpose buffers).              */
/* ------------------------------------------------------------------------ */
/* C = alpha * op(A) op(B) (+ residual), alpha = fl32(sinvA[0] * sinvB[0]),
 * accumulated in fp32 on the tcgen05 tensor cores (kind::f8f6f4).
 *   A, B: FP8 codes (formats fmtA/fmtB may differ), stored per `layout`, with
 *         leading dimensions lda/ldb in elements (= bytes).
 *   sinvA, sinvB: device pointers to one float each (a tensor's scale_inv).
 *   C: [M,N] of out_dtype, leading dimension ldc elements.
 *   residual: optional bf16 [M,N] (ldr elements) added in fp32 before the
 *             bf16 rounding; requires out_dtype == FP8Q_BF16.
 * Requirements: M,N,K >= 1; the contiguous dimension of each operand (K for a
 * K-major operand, M or N for an MN-major one) and its leading dimension are
 * multiples of 16; ldc, ldr multiples of 8.  */
FP8Q_API int fp8_gemm_scaled(fp8q_layout layout, int64_t M, int64_t N, int64_t K, const uint8_t* A,
                    fp8q_fmt fmtA, int64_t lda, const uint8_t* B, fp8q_fmt fmtB, int64_t ldb,
                    const float* sinvA, const float* sinvB, void* C, fp8q_dtype out_dtype,
                    int64_t ldc, const void* residual, int64_t ldr, fp8q_stream stream);

/* ------------------------------------------------------------------------ */
/* RMSNorm fused with the absmax reduction and the E4M3 cast (LLMQ §3).     */
/* ------------------------------------------------------------------------ */
/* x [T,d] bf16, g [d] bf16 -> q [T,d] E4M3, scal, rstd [T] fp32.
 * rstd_t = fl32(1 / fl32(sqrt(fl32(fl32(S_t / d) + eps)))), S_t the fp32
 * pairwise sum of x^2 over the row; n = fl32(fl32(x * rstd) * g).
 * Requirements: T >= 1, d multiple of 16, 16 <= d <= 8192. */
FP8Q_API size_t rmsnorm_quant_workspace_size(int64_t T, int64_t d);
FP8Q_API int rmsnorm_quant(const void* x, const void* g, int64_t T, int64_t d, float eps, uint8_t* q,
                  float* scal, float* rstd, void* ws, size_t ws_bytes, fp8q_stream stream);

/* ------------------------------------------------------------------------ */
/* SwiGLU fused with requantization (LLMQ §3.1: quantization fused with the */
/* nonlinearity).                                                           */
/* ------------------------------------------------------------------------ */
/* H [T,2f] bf16 (gate in columns [0,f), up in [f,2f)) -> q [T,f] of fmt.
 * a = fl32(fl32(h / fl32(1 + exp_ref(-h))) * u) in fp32; exp_ref is a fixed
 * fp32 sequence (Cody-Waite reduction and a degree-8 Taylor polynomial in
 * fused multiply-adds), so the result is bit-reproducible.  Requirements: T >= 1, f multiple of 16. */
FP8Q_API size_t swiglu_quant_workspace_size(int64_t T, int64_t f);
FP8Q_API int swiglu_quant(const void* H, int64_t T, int64_t f, fp8q_fmt fmt, uint8_t* q, float* scal,
                 void* ws, size_t ws_bytes, fp8q_stream stream);

/* ------------------------------------------------------------------------ */
/* RMSNorm backward with the residual gradient: the last step of the        */
/* block's backward (LLMQ §3: the non-matmul ops around the matmuls).       */
/* ------------------------------------------------------------------------ */
/* dN [T,d] fp32 (the gradient at the normalized output n = x rstd g), x [T,d]
 * bf16 (the block input), dY [T,d] bf16 (the residual branch's gradient),
 * g [d] bf16, rstd [T] fp32 (the forward's, as rmsnorm_quant writes it)
 * -> dX [T,d] bf16 and dg [d] fp32, with nh = x rstd and u = dN g:
 *   m_t  = (1/d) sum_j u_tj nh_tj,
 *   dX   = bf16(dY + rstd (u - nh m_t)),
 *   dg_j = sum_t dN_tj nh_tj.
 * The sums are fp32 in a fixed order (a row: 8 columns per thread, a warp
 * butterfly, a butterfly over the warps; dg: per-block partials over runs of
 * consecutive rows, then over blocks in block order), so a result repeats bit
 * for bit on one device and differs from the exact value by fp32 rounding.
 * Requirements: 1 <= T <= 2^28, d a multiple of 16, 16 <= d <= 8192; dN, x,
 * dY, g and dX 16-byte aligned; rstd and dg 4-byte aligned.  Workspace:
 * rmsnorm_bwd_workspace_size(T, d) bytes, 256-byte aligned (the per-block dg
 * partials; FP8Q_ERR_WORKSPACE when missing, misaligned or too small).  The
 * caller owns every buffer; the call only enqueues work on `stream`. */
FP8Q_API size_t rmsnorm_bwd_workspace_size(int64_t T, int64_t d);
FP8Q_API int rmsnorm_bwd(const float* dN, const void* x, const void* dY, const void* g, const float* rstd,
                         int64_t T, int64_t d, void* dX, float* dg, void* ws, size_t ws_bytes,
                         fp8q_stream stream);

/* ------------------------------------------------------------------------ */
/* Block-scaled MXFP8 (LLMQ §2: inner-dimension block scaling, which the    */
/* Blackwell tensor cores support natively).                                */
/* ------------------------------------------------------------------------ */
/* Format (OCP Microscaling): 32 consecutive elements along a GEMM's
 * contraction dimension share one scale 2^X, stored as the E8M0 code X + 127
 * (0xFF = NaN); the elements are E4M3 or E5M2 codes worth decode(code) * 2^X.
 * Scale rule (the per-tensor rule's "no clipping", per block): X is the
 * smallest integer with amax_block <= fmt_max * 2^X, clamped to [-127, 127];
 * an all-zero block has X = -127 (code 0); code = fp8_rne_satfinite(fl32(v *
 * 2^-X)).  A block holding NaN or Inf gets scale code 0xFF, element codes 0x7F
 * and sets FP8Q_STATUS_NONFINITE.
 *
 * Scale layout ("chunked"): an operand with `rows` rows along M (or N) and
 * contraction length K keeps its codes in 512-byte chunks, one per 128 rows x
 * 128 K (4 blocks), chunk (i, j) at byte (i * ceil(K/128) + j) * 512; row r,
 * block b of a chunk at byte (r % 32) * 16 + (r / 32) * 4 + b.  This is the
 * order in which the GEMM copies scales into tensor memory.  mx_scale_bytes
 * returns the size. */
FP8Q_API size_t mx_scale_bytes(int64_t rows, int64_t K);

/* x [R,C] (bf16 or fp32) -> in one pass, either or both of
 *   q_r [R,C] codes + sf_r: blocks of 32 consecutive columns of a row -- x as
 *     a GEMM operand contracted over its columns (K = C, rows = R);
 *   q_c [R,C] codes + sf_c: blocks of 32 consecutive rows of a column -- x as
 *     an operand contracted over its rows (K = R, rows = C).
 * Either pair may be NULL (not both).  Requirements: R, C multiples of 128;
 * 16-byte aligned pointers; sf_r holds mx_scale_bytes(R, C) bytes, sf_c
 * mx_scale_bytes(C, R).  Deterministic, no workspace. */
FP8Q_API int mx_quantize(const void* x, fp8q_dtype x_dtype, int64_t R, int64_t C, fp8q_fmt fmt, uint8_t* q_r,
                         uint8_t* sf_r, uint8_t* q_c, uint8_t* sf_c, fp8q_stream stream);

/* Block-scaled GEMM C = op(A) op(B) (+ residual) on the tcgen05 tensor cores
 * (kind::mxf8f6f4.block_scale, fp32 accumulation; no per-tensor alpha).
 * Layouts and leading dimensions as fp8_gemm_scaled.  sfA: the chunked
 * scales of A as an operand with M rows and contraction K (for NN / NT that is
 * mx_quantize's sf_r of A [M,K]; for TN, sf_c of A [K,M]); sfB likewise with N
 * rows (NN / TN: sf_c of B [K,N]; NT: sf_r of B [N,K]).  Requirements: K a
 * multiple of 128; M, N >= 1 as fp8_gemm_scaled; scales of rows past M (N) in
 * the last chunk are read but do not reach C. */
FP8Q_API int fp8_gemm_mx(fp8q_layout layout, int64_t M, int64_t N, int64_t K, const uint8_t* A, fp8q_fmt fmtA,
                         int64_t lda, const uint8_t* sfA, const uint8_t* B, fp8q_fmt fmtB, int64_t ldb,
                         const uint8_t* sfB, void* C, fp8q_dtype out_dtype, int64_t ldc, const void* residual,
                         int64_t ldr, fp8q_stream stream);

/* One block-scaled operand: codes and chunked scales. */
typedef struct fp8q_mx_tensor {
  uint8_t* q;
  uint8_t* sf;
} fp8q_mx_tensor;

/* ------------------------------------------------------------------------ */
/* The MLP block, forward and backward (bias-free SwiGLU MLP with RMSNorm   */
/* and bf16 residual; E4M3 activations/weights, E5M2 gradients).            */
/* ------------------------------------------------------------------------ */
/* Forward:  W_gu8 = q(W_gu), W_d8 = q(W_d), n8 = q(RMSNorm(x) * g),
 *           H = bf16(alpha * n8 @ W_gu8)  [T,2f],  a8 = q(silu(H_gate) * H_up),
 *           y = bf16(x + alpha * a8 @ W_d8).
 * Backward: dY8 = q5(dY),  dA = alpha * dY8 @ W_d8^T   (q5: E5M2, or E4M3 with grad_e4m3),
 *           dH = bf16(SwiGLU'(H) * dA), dH8 = q5(dH),
 *           dW_d = alpha * a8^T @ dY8,  dN = alpha * dH8 @ W_gu8^T,
 *           dW_gu = alpha * n8^T @ dH8  (fp32),
 *           dX = bf16(dY + RMSNorm'(dN)),  dg = sum_t dN * x * rstd.
 * Every alpha is the product of the two operands' scale_inv.
 * W_gu holds [W_gate | W_up] as one tensor with one scale. */
typedef struct fp8q_mlp {
  int64_t T, d, f; /* tokens, model width, FFN width: d, f multiples of 16, d <= 8192 */
  float eps;       /* RMSNorm epsilon */
  /* inputs */
  const void* x;    /* [T,d]  bf16 */
  const void* g;    /* [d]    bf16 RMSNorm gain */
  const void* W_gu; /* [d,2f] bf16 */
  const void* W_d;  /* [f,d]  bf16 */
  /* forward outputs, kept for the backward */
  void* y;          /* [T,d]  bf16 */
  uint8_t* W_gu8;   /* [d,2f] E4M3 */
  uint8_t* W_d8;    /* [f,d]  E4M3 */
  uint8_t* n8;      /* [T,d]  E4M3 */
  float* rstd;      /* [T]    fp32 */
  void* H;          /* [T,2f] bf16 */
  uint8_t* a8;      /* [T,f]  E4M3 */
  float* scal;      /* [6][3] {amax, scale, scale_inv} of W_gu, W_d, n, a, dY, dH */
  /* backward input/outputs */
  const void* dY;   /* [T,d]  bf16 */
  void* dX;         /* [T,d]  bf16 */
  float* dW_gu;     /* [d,2f] fp32 */
  float* dW_d;      /* [f,d]  fp32 */
  float* dg;        /* [d]    fp32 */
  /* optional views of backward intermediates; NULL = kept in the workspace */
  uint8_t* dY8;     /* [T,d]  E5M2 */
  void* dH;         /* [T,2f] bf16 */
  uint8_t* dH8;     /* [T,2f] E5M2 */
  float* dN;        /* [T,d]  fp32 */
  /* Recompute mode (LLMQ §3.1: activations are recomputed in the backward from
   * what was retained, here n8 and the scales; the retained absmax scale of a
   * lets SwiGLU and its E4M3 cast fuse into the recomputing GEMM's epilogue).
   * Nonzero: mlp_block_bwd does not read the forward's H and a8; it recomputes
   * H = bf16(alpha n8 @ W_gu8) into H and a8 = q(SwiGLU(H)) with scal's
   * retained scale of a into a8, bit-identical to the forward's, so the
   * caller need not keep H and a8 alive between the forward and backward. */
  int recompute;
  /* Nonzero: every gradient the backward quantizes (dY, dH; in fp8q_block also
   * dh and dQKV) is E4M3 instead of E5M2 -- LLMQ §5 Figure 2's recipe with E4M3
   * forward and backward.  Zero (default): E5M2 gradients. */
  int grad_e4m3;
  /* Nonzero: the BF16 baseline the FP8 path is measured against (LLMQ §4 and
   * §5 compare FP8 training with BF16 training).  The same block with no
   * quantization: the GEMMs (tcgen05 kind::f16) read bf16 operands -- W_gu,
   * W_d, n16, a16, dY and dH -- with no scale factors; n16 = bf16((x rstd) g),
   * H = bf16(n16 @ W_gu), a16 = bf16(SwiGLU(H)), y = bf16(x + a16 @ W_d) and
   * the backward as above with every q() the identity.  W_gu8, W_d8, n8, a8,
   * dY8, dH8 and scal are neither read nor written (may be NULL); n16 and a16
   * are required.  Not combinable with recompute or grad_e4m3 (returns
   * FP8Q_ERR_UNSUPPORTED); fp8q_block rejects it too. */
  int bf16;
  void* n16;        /* [T,d]  bf16 normalized input (bf16 != 0) */
  void* a16;        /* [T,f]  bf16 SwiGLU output (bf16 != 0) */
  /* Non-null: the block-scaled MXFP8 block (LLMQ §2: inner-dimension block
   * scaling, native on Blackwell); see fp8q_mlp_mx below.  W_gu8, W_d8, n8,
   * a8, dY8, dH8 and scal are then neither read nor written (may be NULL). */
  const struct fp8q_mlp_mx* mx;
} fp8q_mlp;

/* The MXFP8 block (fp8q_mlp.mx).  The same steps as the per-tensor block with
 * every quantization block-scaled along the contraction dimension of the GEMM
 * that reads it, so a tensor two GEMMs contract differently is quantized both
 * ways (one mx_quantize pass each; "_r" = blocks along a row, "_c" = down a
 * column); the GEMMs take no alpha:
 *   H = bf16(n_r @ W_gu_c),  a = SwiGLU(H),  y = bf16(x + a_r @ W_d_c);
 *   dA = dY_r @ W_d_r^T,  dH = bf16(SwiGLU'(H) dA),  dW_d = a_c^T @ dY_c,
 *   dN = dH_r @ W_gu_r^T,  dW_gu = n_c^T @ dH_c,  dX, dg as before.
 * n = fl32(fl32(x rstd) g) with the per-tensor block's rstd.  Gradients
 * (dY, dH) are E5M2 (E4M3 with grad_e4m3).  Every tensor here is caller
 * memory: codes like the tensor they encode, scales in the chunked layout
 * (sf of an "_r" tensor [R,C]: mx_scale_bytes(R, C); "_c": mx_scale_bytes(C, R)).
 * The forward writes W_gu_*, W_d_*, n_*, a_*, which the backward reads; the
 * backward writes dY_*, dH_*.  Requirements: T, d, f multiples of 128; not
 * combinable with recompute or bf16 (FP8Q_ERR_UNSUPPORTED); the workspace is
 * mlp_block_workspace_size's. */
typedef struct fp8q_mlp_mx {
  fp8q_mx_tensor W_gu_r, W_gu_c; /* [d,2f] E4M3 */
  fp8q_mx_tensor W_d_r, W_d_c;   /* [f,d]  E4M3 */
  fp8q_mx_tensor n_r, n_c;       /* [T,d]  E4M3 */
  fp8q_mx_tensor a_r, a_c;       /* [T,f]  E4M3 */
  fp8q_mx_tensor dY_r, dY_c;     /* [T,d]  E5M2 (E4M3 with grad_e4m3) */
  fp8q_mx_tensor dH_r, dH_c;     /* [T,2f] E5M2 (E4M3 with grad_e4m3) */
} fp8q_mlp_mx;

/* backward != 0 sizes the workspace for mlp_block_bwd (which also suffices for mlp_block_fwd). */
FP8Q_API size_t mlp_block_workspace_size(int64_t T, int64_t d, int64_t f, int backward);
FP8Q_API int mlp_block_fwd(const fp8q_mlp* m, void* ws, size_t ws_bytes, fp8q_stream stream);
/* Reads the forward's saved tensors (W_gu8, W_d8, n8, rstd, H, a8, scal[0..3]). */
FP8Q_API int mlp_block_bwd(const fp8q_mlp* m, void* ws, size_t ws_bytes, fp8q_stream stream);

/* Training steps from and to host memory, pipelined.  Step i copies its inputs (x, g, W_gu, W_d,
 * dY) from host[i] into device set i % 2 (dev0 or dev1), runs mlp_block_fwd + mlp_block_bwd on
 * `stream`, and copies the outputs (y, dX, dW_gu, dW_d, dg) back into host[i].  The copies run on
 * two streams of the library's own, ordered by events, so step i+1's inputs arrive and step
 * i-1's outputs leave while step i computes; the kernels stay in order on `stream`, so one
 * workspace serves both sets (mlp_block_workspace_size(T, d, f, 1) bytes).  A null host pointer
 * means that tensor does not cross the host link in that step: an input already resident on the
 * device (the weights and gain of a model kept in HBM), an output left there (weight gradients
 * for an optimizer on the device).  dev0 and dev1 must have the same sizes and switches; a buffer
 * they share must have a null host pointer in every step (their intermediates may be shared
 * freely).  Host buffers should be pinned (pageable memory makes the copies synchronous).
 * Returns once everything is enqueued; `stream` is ordered after the last copy, so a
 * synchronisation of `stream` (or an event recorded on it) covers the whole run.  The pages
 * describe no such runtime; this is the executor a trainer feeding the block from the host uses. */
typedef struct fp8q_mlp_host_io {
  const void* x;    /* [T,d]  bf16 */
  const void* g;    /* [d]    bf16 */
  const void* W_gu; /* [d,2f] bf16 */
  const void* W_d;  /* [f,d]  bf16 */
  const void* dY;   /* [T,d]  bf16 */
  void* y;          /* [T,d]  bf16 */
  void* dX;         /* [T,d]  bf16 */
  float* dW_gu;     /* [d,2f] fp32 */
  float* dW_d;      /* [f,d]  fp32 */
  float* dg;        /* [d]    fp32 */
} fp8q_mlp_host_io;
FP8Q_API int mlp_block_run_steps(const fp8q_mlp* dev0, const fp8q_mlp* dev1, const fp8q_mlp_host_io* host,
                                 int n_steps, void* ws, size_t ws_bytes, fp8q_stream stream);
/* The same for forward-only steps (mlp_block_fwd alone): x, g, W_gu, W_d in, y out; the host
 * pointers of the backward's tensors (dY, dX, dW_gu, dW_d, dg) must be null; workspace
 * mlp_block_workspace_size(T, d, f, 0) bytes. */
FP8Q_API int mlp_block_fwd_run_steps(const fp8q_mlp* dev0, const fp8q_mlp* dev1, const fp8q_mlp_host_io* host,
                                     int n_steps, void* ws, size_t ws_bytes, fp8q_stream stream);

/* ------------------------------------------------------------------------ */
/* The full transformer block's matmuls around an attention core computed   */
/* elsewhere (the 32B-class workload): attention-side RMSNorm + QKV         */
/* projection, O projection + residual, then the MLP block.                 */
/* ------------------------------------------------------------------------ */
/* Forward:  n1_8 = q(RMSNorm(x) * g1), qkv = bf16(alpha n1_8 @ W_qkv8) (the
 *           core's input), att8 = q(att) (the core's output, given),
 *           h = bf16(x + alpha att8 @ W_o8), then mlp_block_fwd on h
 *           (mlp.x must be h; mlp.y is the block output).
 * Backward: mlp_block_bwd with mlp.dY = the block's dY gives dh in mlp.dX;
 *           dh8 = q5(dh), d_att = bf16(alpha dh8 @ W_o8^T) (to the core),
 *           dW_o = alpha att8^T @ dh8; dQKV8 = q5(dQKV) (dQKV: the gradient
 *           arriving at qkv from the core), dN1 = alpha dQKV8 @ W_qkv8^T,
 *           dW_qkv = alpha n1_8^T @ dQKV8, dX = bf16(dh + RMSNorm'(dN1)), dg1.
 * Requirements as for fp8q_mlp, plus n_qkv a multiple of 16. */
typedef struct fp8q_block {
  int64_t T, d, f, n_qkv;
  float eps;
  const void* x;      /* [T,d]     bf16 block input */
  const void* g1;     /* [d]       bf16 attention-side RMSNorm gain */
  const void* W_qkv;  /* [d,n_qkv] bf16 */
  const void* W_o;    /* [d,d]     bf16 */
  void* att;          /* [T,d]     bf16 attention core output (input; written by block_fwd when n_heads != 0) */
  void* qkv;          /* [T,n_qkv] bf16 attention core input (forward output) */
  void* h;            /* [T,d]     bf16 attention residual output = the MLP input */
  uint8_t* W_qkv8;    /* [d,n_qkv] E4M3 */
  uint8_t* W_o8;      /* [d,d]     E4M3 */
  uint8_t* n1_8;      /* [T,d]     E4M3 */
  float* rstd1;       /* [T]       fp32 */
  uint8_t* att8;      /* [T,d]     E4M3 */
  float* scal;        /* [6][3] {amax, scale, scale_inv} of W_qkv, W_o, n1, att, dh, dQKV */
  fp8q_mlp mlp;       /* the MLP sub-block: mlp.x == h, mlp.dX receives dh */
  void* dQKV;         /* [T,n_qkv] bf16 gradient from the attention core (input; written by block_bwd
                       * when n_heads != 0) */
  void* d_att;        /* [T,d]     bf16 gradient to the attention core */
  void* dX;           /* [T,d]     bf16 */
  float* dW_qkv;      /* [d,n_qkv] fp32 */
  float* dW_o;        /* [d,d]     fp32 */
  float* dg1;         /* [d]       fp32 */
  /* optional views of backward intermediates; NULL = kept in the workspace */
  uint8_t* dh8;       /* [T,d]     E5M2 */
  uint8_t* dQKV8;     /* [T,n_qkv] E5M2 */
  float* dN1;         /* [T,d]     fp32 */
  /* The attention core inside the block (nonzero n_heads): block_fwd computes att = attention_fwd(qkv)
   * (and lse) right after the QKV projection, block_bwd computes dQKV = attention_bwd(qkv, att, lse,
   * d_att) right after the O projection's dgrad; att and dQKV are then outputs.  Requires
   * n_heads * 128 = d, (n_heads + 2 n_kv_heads) * 128 = n_qkv and attention_fwd's conditions on
   * seq_len.  Zero: att and dQKV are given (an attention core computed elsewhere). */
  int n_heads, n_kv_heads;
  int64_t seq_len;
  float* lse;         /* [n_heads,T] fp32, written by block_fwd, read by block_bwd (n_heads != 0) */
  /* BF16 baseline of the whole block (mlp.bf16 != 0; see fp8q_mlp.bf16): every GEMM reads bf16
   * operands with no scale factors -- W_qkv, W_o, att, dh, dQKV and n1_16 = bf16((x rstd1) g1);
   * W_qkv8, W_o8, n1_8, att8, scal, dh8 and dQKV8 are neither read nor written (may be NULL). */
  void* n1_16;        /* [T,d] bf16 (mlp.bf16 != 0) */
} fp8q_block;

FP8Q_API size_t block_workspace_size(int64_t T, int64_t d, int64_t f, int64_t n_qkv, int backward);
FP8Q_API int block_fwd(const fp8q_block* b, void* ws, size_t ws_bytes, fp8q_stream stream);
FP8Q_API int block_bwd(const fp8q_block* b, void* ws, size_t ws_bytes, fp8q_stream stream);

/* Pipelined steps of the full block from and to host memory, as mlp_block_run_steps: step i
 * copies its inputs from host[i] into device set i % 2, runs block_fwd (and block_bwd when
 * backward != 0) on `stream`, and copies its outputs back into host[i], step i + 1's inputs and
 * step i - 1's outputs moving while step i computes.  A null host pointer keeps that tensor on
 * the device in that step; a buffer both sets share must be null in every step.  Without
 * backward, the backward's host pointers (dY, dQKV, dX, d_att and the gradients) must be null;
 * with the attention core inside (n_heads != 0), att and dQKV are the block's own results and
 * their host pointers must be null.  Host tensors have the device tensors' shapes and types (y
 * is mlp.y; g, W_gu, W_d, dY, dW_gu, dW_d, dg those of mlp).  Workspace
 * block_workspace_size(T, d, f, n_qkv, backward) bytes. */
typedef struct fp8q_block_host_io {
  const void* x;
  const void* g1;
  const void* W_qkv;
  const void* W_o;
  const void* att;
  const void* g;
  const void* W_gu;
  const void* W_d;
  const void* dY;
  const void* dQKV;
  void* y;
  void* dX;
  void* d_att;
  float* dW_qkv;
  float* dW_o;
  float* dg1;
  float* dW_gu;
  float* dW_d;
  float* dg;
} fp8q_block_host_io;
FP8Q_API int block_run_steps(const fp8q_block* dev0, const fp8q_block* dev1, const fp8q_block_host_io* host,
                             int n_steps, int backward, void* ws, size_t ws_bytes, fp8q_stream stream);

/* ------------------------------------------------------------------------ */
/* The attention core between the QKV and O projections.  LLMQ §2/§3 name    */
/* the transformer block's attention and custom kernels for it; the pages    */
/* fix no attention arithmetic, so this is plain causal softmax attention    */
/* with grouped K/V heads, bf16 in and out, fp32 softmax and accumulation.  */
/* ------------------------------------------------------------------------ */
/* qkv [T, (n_heads + 2 n_kv_heads) head_dim] bf16, row t = [q heads | k heads | v heads]
 * (the QKV projection's output); the T tokens form T / seq_len sequences of seq_len
 * consecutive tokens; query position i sees keys 0..i of its own sequence; query head h
 * reads K/V head h / (n_heads / n_kv_heads); scale 1 / sqrt(head_dim).
 *   att [T, n_heads head_dim] bf16: att_i = sum_k softmax_k(q_i . k_k / sqrt(head_dim)) v_k
 *   lse [n_heads, T] fp32: natural log of each row's softmax denominator (kept for the backward)
 * P is rounded to bf16 before it multiplies V (the tensor-core operand), its row sum is not.
 * Requirements: head_dim = 128 and seq_len a positive multiple of 128 (else
 * FP8Q_ERR_UNSUPPORTED); n_heads a multiple of n_kv_heads, T a multiple of seq_len, T and
 * (T / 128) n_heads below 2^31, pointers 16-byte aligned (else FP8Q_ERR_INVALID_ARG).
 * Asynchronous; no workspace. */
FP8Q_API int attention_fwd(const void* qkv, int64_t T, int64_t seq_len, int n_heads, int n_kv_heads, int head_dim,
                           void* att, float* lse, fp8q_stream stream);
/* Backward of attention_fwd: the plain gradient of the definition above, with d_att = dO
 * [T, n_heads head_dim] bf16 given, att and lse as attention_fwd wrote them:
 *   dP = dO V^T, D = rowsum(dO * att), dS = P (dP - D);  dq = dS K / sqrt(head_dim),
 *   dk = dS^T Q / sqrt(head_dim) and dv = P^T dO summed over the query heads of each K/V head.
 * dqkv [T, (n_heads + 2 n_kv_heads) head_dim] bf16 (same layout as qkv) is overwritten in full.
 * P and dS are rounded to bf16 as tensor-core operands.  Deterministic (no atomics: a K/V
 * head's gradient is summed over its query heads inside one CTA).  Workspace:
 * attention_bwd_workspace_size(T, n_heads) bytes (D and lse in the log2 domain), 256-byte
 * aligned.  Requirements and errors as attention_fwd. */
FP8Q_API size_t attention_bwd_workspace_size(int64_t T, int n_heads);
FP8Q_API int attention_bwd(const void* qkv, const void* att, const float* lse, const void* d_att, int64_t T,
                           int64_t seq_len, int n_heads, int n_kv_heads, int head_dim, void* dqkv, void* ws,
                           size_t ws_bytes, fp8q_stream stream);

/* ------------------------------------------------------------------------ */
/* Status and introspection                                                 */
/* ------------------------------------------------------------------------ */
/* Reads (and with clear != 0 resets) the current device's status word
 * (FP8Q_STATUS_* bits).  Call after synchronizing the streams that ran the
 * library's kernels.  Returns the bits, or -1 if the read itself failed. */
FP8Q_API int fp8q_get_status(int clear);
/* Short description of an fp8q_status value (static storage). */
FP8Q_API const char* fp8q_status_string(int status);
/* Number of kernel launches the most recent successful call on this host
 * thread enqueued. */
FP8Q_API int fp8q_last_launch_count(void);

/* Diagnostics for the failure-detection path (no page counterpart): enqueues
 * one thread that waits on an mbarrier nothing ever arrives at, through the
 * same bounded wait every pipelined kernel of the library uses, with the given
 * limit (1 ms .. 10 s) instead of the production 2 s.  When the limit runs out
 * the kernel sets FP8Q_STATUS_TIMEOUT and returns; the context stays usable.
 * Returns FP8Q_OK once enqueued. */
FP8Q_API int fp8q_selftest_bounded_wait(int64_t limit_ns, fp8q_stream stream);

/* Diagnostics for the GEMM's abort sequence (no page counterpart): the same
 * launch as fp8_gemm_scaled (mx == 0) or fp8_gemm_mx (mx != 0; sfA, sfB as
 * there, sinvA, sinvB unused), except that every pipeline wait of the kernel
 * (stage ring, accumulator hand-off) gives up after limit_ns (1 us .. 10 s)
 * instead of 2 s.  With a limit of a few microseconds ordinary waits run out:
 * the CTA records FP8Q_STATUS_TIMEOUT, stops issuing, waits (with the full
 * 2 s limit) for the copies and MMAs it issued, frees its tensor memory and
 * exits; C is then incomplete and the context stays usable.  Returns FP8Q_OK
 * once enqueued (synchronous errors as the GEMM entry points). */
FP8Q_API int fp8q_selftest_gemm_wait_limit(fp8q_layout layout, int64_t M, int64_t N, int64_t K, const uint8_t* A,
                                           fp8q_fmt fmtA, int64_t lda, const uint8_t* B, fp8q_fmt fmtB, int64_t ldb,
                                           const float* sinvA, const float* sinvB, int mx, const uint8_t* sfA,
                                           const uint8_t* sfB, void* C, fp8q_dtype out_dtype, int64_t ldc,
                                           int64_t limit_ns, fp8q_stream stream);

/* Diagnostics for the RMSNorm backward's abort sequence (no page counterpart):
 * rmsnorm_bwd, except that every wait of a block on the bulk copies of its
 * rows probes the barrier without suspending and gives up after limit_ns
 * (1 ns .. 10 s) instead of 2 s.  With a limit of a few nanoseconds the first
 * waits run out: the block records
 * FP8Q_STATUS_TIMEOUT, stops, waits (with the full 2 s limit) for the copies
 * still in flight into its shared memory and exits; dX and dg are then
 * incomplete and the context stays usable.  Returns FP8Q_OK once enqueued
 * (synchronous errors as rmsnorm_bwd). */
FP8Q_API int fp8q_selftest_rmsnorm_bwd_wait_limit(const float* dN, const void* x, const void* dY, const void* g,
                                                  const float* rstd, int64_t T, int64_t d, void* dX, float* dg,
                                                  void* ws, size_t ws_bytes, int64_t limit_ns,
                                                  fp8q_stream stream);

/* Kernel-level timing for benchmarks.  While tracing is on for the calling
 * host thread, each kernel step the library enqueues is bracketed by two CUDA
 * events recorded on the stream it is launched on (host-side CUDA objects; no
 * device memory).  fp8q_trace_start(capacity) creates 2*capacity events and
 * turns tracing on (FP8Q_ERR_CUDA if event creation fails); steps beyond
 * capacity are not traced.  fp8q_trace_stop() turns it off;
 * fp8q_trace_resume() turns it back on, keeping the steps recorded so far
 * (FP8Q_ERR_INVALID_ARG before the first fp8q_trace_start), so that a
 * caller can trace a sample of its steps.  Steps enqueued
 * while the stream is being captured into a CUDA graph record their events as
 * event-record nodes of the graph: each run of the graph records them again,
 * and fp8q_trace_read() then reports the latest run.
 * fp8q_trace_read() waits for the recorded events, writes each step's
 * duration in milliseconds and its kernel kind, and returns the count.
 * fp8q_kernel_name(kind) names a kind (static storage). */
FP8Q_API int fp8q_trace_start(int capacity);
FP8Q_API int fp8q_trace_stop(void);
FP8Q_API int fp8q_trace_resume(void);
FP8Q_API int fp8q_trace_read(float* ms, int* kinds, int capacity);
FP8Q_API const char* fp8q_kernel_name(int kind);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */
