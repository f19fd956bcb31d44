// C ABI of the FP8 block pipeline (declared in include/fp8q.h): argument
// validation, workspace carving and the forward/backward orchestration of the
// MLP block.  Every call only enqueues kernels on the caller's stream.
#include "fp8q.h"
#include "fp8q_internal.h"

#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

namespace {

using namespace fp8q;

__device__ unsigned g_status_word;

thread_local int t_last_launches = 0;
// Pipeline-wait limit of the GEMMs enqueued by the next fp8_gemm_scaled / fp8_gemm_mx call on this
// thread (0: the default); set only for the duration of fp8q_selftest_gemm_wait_limit.
thread_local uint64_t t_gemm_wait_ns = 0;

// ---- kernel-level trace (benchmarks) ------------------------------------------
enum Kind {
  kKAbsmaxPartial = 0, kKQuantCast, kKRmsnormStats, kKRmsnormCast, kKSwigluAmax, kKSwigluCast, kKRmsnormBwd,
  kKGemmGateUp, kKGemmDown, kKGemmDownDgrad, kKGemmDownWgrad, kKGemmGateUpDgrad, kKGemmGateUpWgrad, kKGemm,
  kKGemmQkv, kKGemmOResidual, kKGemmODgrad, kKGemmOWgrad, kKGemmQkvDgrad, kKGemmQkvWgrad,
  kKGemmGateUpRecompute, kKRmsnormBf16, kKAttnFwd, kKAttnBwdDelta, kKAttnBwdDkdv, kKAttnBwdDq,
  kKMxQuant, kKPrologueStats, kKPrologueCast,
  kKCount
};
const char* const kKindNames[kKCount] = {
    "absmax_partial", "quant_cast", "rmsnorm_stats", "rmsnorm_cast", "swiglu_amax", "swiglu_cast",
    "rmsnorm_bwd", "gemm_gate_up_swiglu", "gemm_down_residual", "gemm_down_dgrad_swiglu_bwd",
    "gemm_down_wgrad", "gemm_gate_up_dgrad", "gemm_gate_up_wgrad", "gemm",
    "gemm_qkv", "gemm_o_residual", "gemm_o_dgrad", "gemm_o_wgrad", "gemm_qkv_dgrad", "gemm_qkv_wgrad",
    "gemm_gate_up_recompute", "rmsnorm_bf16", "attn_fwd", "attn_bwd_delta", "attn_bwd_dkdv", "attn_bwd_dq",
    "mx_quant", "prologue_stats", "prologue_cast"};

struct Trace {
  bool on = false;
  std::vector<cudaEvent_t> ev;
  std::vector<int> kinds;
  int n = 0;
};
thread_local Trace t_trace;

}  // namespace

namespace fp8q {

// Under stream capture an event is recorded as an external record: it becomes an event-record node
// of the graph, recorded each time the graph runs (a plain record would only order the capture's
// own streams, and the external flag is refused outside a capture).
static void trace_record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

bool trace_step_begin(cudaStream_t s, int kind) {
  nvtxRangePushA(kKindNames[kind]);
  Trace& t = t_trace;
  if (!t.on || t.n >= (int)t.kinds.size()) return false;
  t.kinds[t.n] = kind;
  trace_record(t.ev[2 * t.n], s);
  return true;
}

void trace_step_end(cudaStream_t s, bool active) {
  if (active) {
    trace_record(t_trace.ev[2 * t_trace.n + 1], s);
    ++t_trace.n;
  }
  nvtxRangePop();
}

void set_last_launch_count(int n) { t_last_launches = n; }

}  // namespace fp8q

namespace {

static_assert((int)kKAbsmaxPartial == (int)kTraceAbsmaxPartial && (int)kKQuantCast == (int)kTraceQuantCast,
              "trace kinds");

// One kernel step: an NVTX range named for the kernel kind (seen by profilers, free otherwise)
// and, while the trace is on, a pair of CUDA events around its launches.
struct TraceScope {
  cudaStream_t s;
  bool active;
  TraceScope(cudaStream_t st, int kind) : s(st), active(trace_step_begin(st, kind)) {}
  ~TraceScope() { trace_step_end(s, active); }
};

struct DevInfo {
  int num_sms = 0;
  unsigned* status = nullptr;
};

int device_info(DevInfo* out) {
  static std::mutex mu;
  static DevInfo cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8Q_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  DevInfo& d = cache[dev];
  if (!d.status) {
    int sms = 0;
    void* st = nullptr;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FP8Q_ERR_CUDA;
    if (cudaGetSymbolAddress(&st, g_status_word) != cudaSuccess) return FP8Q_ERR_CUDA;
    d.num_sms = sms;
    d.status = static_cast<unsigned*>(st);
  }
  *out = d;
  return FP8Q_OK;
}

struct Ctx {
  Launch L;
  int launches = 0;
};

int make_ctx(Ctx* c, fp8q_stream stream) {
  DevInfo d;
  int e = device_info(&d);
  if (e) return e;
  c->L.stream = static_cast<cudaStream_t>(stream);
  c->L.status = d.status;
  c->L.num_sms = d.num_sms;
  c->L.launches = &c->launches;
  return FP8Q_OK;
}

inline bool al16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }
inline size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

// Sequential carve-out of 256-byte aligned pieces from the caller's workspace.
struct Carver {
  uint8_t* base;
  size_t cap, off = 0;
  bool ok = true;
  void* take(size_t bytes) {
    void* p = base + off;
    off += round256(bytes);
    if (off > cap) ok = false;
    return p;
  }
};

constexpr size_t kPartialBytes = sizeof(uint32_t) * kMaxPartials;

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA; }

// One traced kernel step: enqueue `expr` on c.L.stream, return FP8Q_ERR_CUDA on failure.
#define FP8Q_STEP(kind, expr)                   \
  do {                                          \
    TraceScope _ts(c.L.stream, (kind));         \
    int _st = cuda_status(expr);                \
    if (_st != FP8Q_OK) return _st;             \
  } while (0)

int finish(const Ctx& c) {
  t_last_launches = c.launches;
  return FP8Q_OK;
}

int check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (need == 0) return FP8Q_OK;
  if (!ws || ((uintptr_t)ws & 255u) != 0 || ws_bytes < need) return FP8Q_ERR_WORKSPACE;
  return FP8Q_OK;
}

// ---- workspace layouts -------------------------------------------------------
struct MlpWs {
  uint32_t* part_q;    // quantizer partials
  uint32_t* part_g;    // GEMM epilogue partials
  uint32_t* part_w;    // the forward prologue's third partial array
  uint8_t* dY8;
  uint16_t* dH;
  uint8_t* dH8;
  float* dN;
  float* dg_part;
};

size_t mlp_ws_layout(int64_t T, int64_t d, int64_t f, int backward, uint8_t* base, MlpWs* w) {
  Carver c{base, ~size_t(0)};
  MlpWs tmp{};
  tmp.part_q = (uint32_t*)c.take(kPartialBytes);
  tmp.part_g = (uint32_t*)c.take(kPartialBytes);
  tmp.part_w = (uint32_t*)c.take(kPartialBytes);
  if (backward) {
    tmp.dY8 = (uint8_t*)c.take((size_t)(T * d));
    tmp.dH = (uint16_t*)c.take((size_t)(T * 2 * f) * 2);
    tmp.dH8 = (uint8_t*)c.take((size_t)(T * 2 * f));
    tmp.dN = (float*)c.take((size_t)(T * d) * 4);
    tmp.dg_part = (float*)c.take((size_t)((T + kBwdRows - 1) / kBwdRows) * (size_t)d * 4);
  }
  if (w) *w = tmp;
  return c.off;
}

bool mx_ok(const fp8q_mx_tensor& t) { return al16(t.q) && al16(t.sf); }

int validate_mlp(const fp8q_mlp* m, bool backward) {
  if (!m) return FP8Q_ERR_INVALID_ARG;
  if (m->T < 1 || m->d < 16 || m->f < 16 || m->d % 16 || m->f % 16 || m->d > 8192) return FP8Q_ERR_INVALID_ARG;
  if (m->T > (int64_t)1 << 24 || m->f > (int64_t)1 << 20) return FP8Q_ERR_INVALID_ARG;
  if (m->mx) {
    if (m->recompute || m->bf16) return FP8Q_ERR_UNSUPPORTED;
    if (m->T % 128 || m->d % 128 || m->f % 128) return FP8Q_ERR_INVALID_ARG;
    const fp8q_mlp_mx& x = *m->mx;
    const void* must[] = {m->x, m->g, m->W_gu, m->W_d, m->rstd, m->H};
    for (const void* p : must)
      if (!al16(p)) return FP8Q_ERR_INVALID_ARG;
    for (const fp8q_mx_tensor* t : {&x.W_gu_r, &x.W_gu_c, &x.W_d_r, &x.W_d_c, &x.n_r, &x.n_c, &x.a_r, &x.a_c})
      if (!mx_ok(*t)) return FP8Q_ERR_INVALID_ARG;
    if (!backward) return al16(m->y) ? FP8Q_OK : FP8Q_ERR_INVALID_ARG;
    const void* must_b[] = {m->dY, m->dX, m->dW_gu, m->dW_d, m->dg};
    for (const void* p : must_b)
      if (!al16(p)) return FP8Q_ERR_INVALID_ARG;
    for (const fp8q_mx_tensor* t : {&x.dY_r, &x.dY_c, &x.dH_r, &x.dH_c})
      if (!mx_ok(*t)) return FP8Q_ERR_INVALID_ARG;
    return ((m->dH && !al16(m->dH)) || (m->dN && !al16(m->dN))) ? FP8Q_ERR_INVALID_ARG : FP8Q_OK;
  }
  if (m->bf16) {
    if (m->recompute || m->grad_e4m3) return FP8Q_ERR_UNSUPPORTED;
    const void* must16[] = {m->x, m->g, m->W_gu, m->W_d, m->n16, m->rstd, m->H, m->a16};
    for (const void* p : must16)
      if (!al16(p)) return FP8Q_ERR_INVALID_ARG;
    if (!backward) return al16(m->y) ? FP8Q_OK : FP8Q_ERR_INVALID_ARG;
    const void* must16_b[] = {m->dY, m->dX, m->dW_gu, m->dW_d, m->dg};
    for (const void* p : must16_b)
      if (!al16(p)) return FP8Q_ERR_INVALID_ARG;
    return ((m->dH && !al16(m->dH)) || (m->dN && !al16(m->dN))) ? FP8Q_ERR_INVALID_ARG : FP8Q_OK;
  }
  const void* must[] = {m->x, m->g, m->W_gu, m->W_d, m->W_gu8, m->W_d8, m->n8, m->rstd, m->H, m->a8, m->scal};
  for (const void* p : must)
    if (!al16(p)) return FP8Q_ERR_INVALID_ARG;
  if (!backward) return al16(m->y) ? FP8Q_OK : FP8Q_ERR_INVALID_ARG;
  const void* must_b[] = {m->dY, m->dX, m->dW_gu, m->dW_d, m->dg};
  for (const void* p : must_b)
    if (!al16(p)) return FP8Q_ERR_INVALID_ARG;
  const void* opt[] = {m->dY8, m->dH, m->dH8, m->dN};
  for (const void* p : opt)
    if (p && !al16(p)) return FP8Q_ERR_INVALID_ARG;
  return FP8Q_OK;
}

// A GEMM of the BF16 baseline: bf16 operands, alpha = 1.
GemmProblem bf16_gemm(int a_mn, int b_mn, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                      const void* B, int64_t ldb, int64_t b_cols, int epi, int out_f32, void* C, int64_t ldc) {
  GemmProblem g{};
  g.op16 = 1;
  g.a_mn = a_mn;
  g.b_mn = b_mn;
  g.M = (int)M;
  g.N = (int)N;
  g.K = (int)K;
  g.A = static_cast<const uint8_t*>(A);
  g.lda = lda;
  g.B = static_cast<const uint8_t*>(B);
  g.ldb = ldb;
  g.b_cols = b_cols;
  g.epi = epi;
  g.out_f32 = out_f32;
  g.C = C;
  g.ldc = ldc;
  return g;
}

// The BF16 baseline's forward: the FP8 sequence with every cast removed.
int mlp_fwd_run_bf16(const fp8q_mlp* m, Ctx& c) {
  const int64_t T = m->T, d = m->d, f = m->f;
  int P = 0;
  FP8Q_STEP(kKRmsnormBf16, launch_rmsnorm_bf16((const uint16_t*)m->x, (const uint16_t*)m->g, T, (int)d, m->eps, m->rstd,
                                (uint16_t*)m->n16, c.L));
  // G1: H = bf16(n16 @ W_gu), a16 = bf16(SwiGLU(H)) in the epilogue
  GemmProblem g1 = bf16_gemm(0, 1, T, f, d, m->n16, d, m->W_gu, 2 * f, 2 * f, kEpiSwiglu, 0, m->H, 2 * f);
  g1.a16 = (uint16_t*)m->a16;
  FP8Q_STEP(kKGemmGateUp, launch_gemm(g1, &P, c.L));
  // G2: y = bf16(x + a16 @ W_d)
  GemmProblem g2 = bf16_gemm(0, 1, T, d, f, m->a16, f, m->W_d, d, d, kEpiResidual, 0, m->y, d);
  g2.R = (const uint16_t*)m->x;
  g2.ldr = d;
  FP8Q_STEP(kKGemmDown, launch_gemm(g2, &P, c.L));
  return FP8Q_OK;
}

// The BF16 baseline's backward (same layouts as the FP8 backward, no casts).
int mlp_bwd_run_bf16(const fp8q_mlp* m, const MlpWs& w, Ctx& c) {
  const int64_t T = m->T, d = m->d, f = m->f;
  uint16_t* dH = m->dH ? (uint16_t*)m->dH : w.dH;
  float* dN = m->dN ? m->dN : w.dN;
  int P = 0;
  // G3 (NT): dA = dY @ W_d^T, SwiGLU backward fused -> dH
  GemmProblem g3 = bf16_gemm(0, 0, T, f, d, m->dY, d, m->W_d, d, f, kEpiSwigluBwd, 0, dH, 2 * f);
  g3.R = (const uint16_t*)m->H;
  g3.ldr = 2 * f;
  FP8Q_STEP(kKGemmDownDgrad, launch_gemm(g3, &P, c.L));
  // G4 (TN): dW_d = a16^T @ dY
  FP8Q_STEP(kKGemmDownWgrad,
            launch_gemm(bf16_gemm(1, 1, f, d, T, m->a16, f, m->dY, d, d, kEpiStore, 1, m->dW_d, d), &P, c.L));
  // G5 (NT): dN = dH @ W_gu^T
  FP8Q_STEP(kKGemmGateUpDgrad,
            launch_gemm(bf16_gemm(0, 0, T, d, 2 * f, dH, 2 * f, m->W_gu, 2 * f, d, kEpiStore, 1, dN, d), &P, c.L));
  // G6 (TN): dW_gu = n16^T @ dH
  FP8Q_STEP(kKGemmGateUpWgrad, launch_gemm(bf16_gemm(1, 1, d, 2 * f, T, m->n16, d, dH, 2 * f, 2 * f, kEpiStore, 1,
                                                     m->dW_gu, 2 * f),
                                           &P, c.L));
  FP8Q_STEP(kKRmsnormBwd, launch_rmsnorm_bwd(dN, (const uint16_t*)m->x, (const uint16_t*)m->dY, (const uint16_t*)m->g,
                                             m->rstd, T, (int)d, (uint16_t*)m->dX, w.dg_part, m->dg, c.L));
  return FP8Q_OK;
}

// The MLP block's kernel sequences, enqueued on c.L.stream (shared by
// mlp_block_* and block_*).
// A GEMM of the MXFP8 block: codes and chunked scales of both operands, no alpha.
GemmProblem mx_gemm(int a_mn, int b_mn, int64_t M, int64_t N, int64_t K, const fp8q_mx_tensor& A, int fmtA,
                    int64_t lda, const fp8q_mx_tensor& B, int fmtB, int64_t ldb, int64_t b_cols, int epi, int out_f32,
                    void* C, int64_t ldc) {
  GemmProblem g{};
  g.mx = 1;
  g.a_mn = a_mn;
  g.b_mn = b_mn;
  g.M = (int)M;
  g.N = (int)N;
  g.K = (int)K;
  g.A = A.q;
  g.sfA = A.sf;
  g.lda = lda;
  g.fmtA = fmtA;
  g.B = B.q;
  g.sfB = B.sf;
  g.ldb = ldb;
  g.fmtB = fmtB;
  g.b_cols = b_cols;
  g.epi = epi;
  g.out_f32 = out_f32;
  g.C = C;
  g.ldc = ldc;
  return g;
}

// The MXFP8 block's forward: weights and n quantized both ways (one pass each), the gate/up GEMM
// with the SwiGLU epilogue writing H, a = SwiGLU(H) quantized both ways, the down GEMM + residual.
int mlp_fwd_run_mx(const fp8q_mlp* m, const MlpWs& w, Ctx& c) {
  const int64_t T = m->T, d = m->d, f = m->f;
  const fp8q_mlp_mx& x = *m->mx;
  int P = 0;
  FP8Q_STEP(kKMxQuant, launch_mx_quant(kMxInBf16, m->W_gu, nullptr, nullptr, d, 2 * f, 0, x.W_gu_r.q, x.W_gu_r.sf,
                                       x.W_gu_c.q, x.W_gu_c.sf, c.L));
  FP8Q_STEP(kKMxQuant, launch_mx_quant(kMxInBf16, m->W_d, nullptr, nullptr, f, d, 0, x.W_d_r.q, x.W_d_r.sf, x.W_d_c.q,
                                       x.W_d_c.sf, c.L));
  FP8Q_STEP(kKRmsnormStats, launch_rmsnorm_stats((const uint16_t*)m->x, (const uint16_t*)m->g, T, (int)d, m->eps,
                                                 m->rstd, w.part_q, &P, c.L));
  FP8Q_STEP(kKMxQuant, launch_mx_quant(kMxInRmsnorm, m->x, (const uint16_t*)m->g, m->rstd, T, d, 0, x.n_r.q, x.n_r.sf,
                                       x.n_c.q, x.n_c.sf, c.L));
  GemmProblem g1 = mx_gemm(0, 1, T, f, d, x.n_r, 0, d, x.W_gu_c, 0, 2 * f, 2 * f, kEpiSwiglu, 0, m->H, 2 * f);
  FP8Q_STEP(kKGemmGateUp, launch_gemm(g1, &P, c.L));
  FP8Q_STEP(kKMxQuant, launch_mx_quant(kMxInSwiglu, m->H, nullptr, nullptr, T, f, 0, x.a_r.q, x.a_r.sf, x.a_c.q,
                                       x.a_c.sf, c.L));
  GemmProblem g2 = mx_gemm(0, 1, T, d, f, x.a_r, 0, f, x.W_d_c, 0, d, d, kEpiResidual, 0, m->y, d);
  g2.R = (const uint16_t*)m->x;
  g2.ldr = d;
  FP8Q_STEP(kKGemmDown, launch_gemm(g2, &P, c.L));
  return FP8Q_OK;
}

// The MXFP8 block's backward: each GEMM reads its operands quantized along its own contraction
// dimension (the wgrads contract over tokens: the "_c" tensors).
int mlp_bwd_run_mx(const fp8q_mlp* m, const MlpWs& w, Ctx& c) {
  const int64_t T = m->T, d = m->d, f = m->f;
  const fp8q_mlp_mx& x = *m->mx;
  uint16_t* dH = m->dH ? (uint16_t*)m->dH : w.dH;
  float* dN = m->dN ? m->dN : w.dN;
  const int gf = m->grad_e4m3 ? 0 : 1;
  int P = 0;
  FP8Q_STEP(kKMxQuant, launch_mx_quant(kMxInBf16, m->dY, nullptr, nullptr, T, d, gf, x.dY_r.q, x.dY_r.sf, x.dY_c.q,
                                       x.dY_c.sf, c.L));
  GemmProblem g3 = mx_gemm(0, 0, T, f, d, x.dY_r, gf, d, x.W_d_r, 0, d, f, kEpiSwigluBwd, 0, dH, 2 * f);
  g3.R = (const uint16_t*)m->H;
  g3.ldr = 2 * f;
  FP8Q_STEP(kKGemmDownDgrad, launch_gemm(g3, &P, c.L));
  FP8Q_STEP(kKMxQuant, launch_mx_quant(kMxInBf16, dH, nullptr, nullptr, T, 2 * f, gf, x.dH_r.q, x.dH_r.sf, x.dH_c.q,
                                       x.dH_c.sf, c.L));
  GemmProblem g4 = mx_gemm(1, 1, f, d, T, x.a_c, 0, f, x.dY_c, gf, d, d, kEpiStore, 1, m->dW_d, d);
  FP8Q_STEP(kKGemmDownWgrad, launch_gemm(g4, &P, c.L));
  GemmProblem g5 = mx_gemm(0, 0, T, d, 2 * f, x.dH_r, gf, 2 * f, x.W_gu_r, 0, 2 * f, d, kEpiStore, 1, dN, d);
  FP8Q_STEP(kKGemmGateUpDgrad, launch_gemm(g5, &P, c.L));
  GemmProblem g6 = mx_gemm(1, 1, d, 2 * f, T, x.n_c, 0, d, x.dH_c, gf, 2 * f, 2 * f, kEpiStore, 1, m->dW_gu, 2 * f);
  FP8Q_STEP(kKGemmGateUpWgrad, launch_gemm(g6, &P, c.L));
  FP8Q_STEP(kKRmsnormBwd, launch_rmsnorm_bwd(dN, (const uint16_t*)m->x, (const uint16_t*)m->dY, (const uint16_t*)m->g,
                                             m->rstd, T, (int)d, (uint16_t*)m->dX, w.dg_part, m->dg, c.L));
  return FP8Q_OK;
}

int mlp_fwd_run(const fp8q_mlp* m, const MlpWs& w, Ctx& c) {
  if (m->bf16) return mlp_fwd_run_bf16(m, c);
  if (m->mx) return mlp_fwd_run_mx(m, w, c);
  const int64_t T = m->T, d = m->d, f = m->f;
  float* s_wgu = m->scal + 0;
  float* s_wd = m->scal + 3;
  float* s_n = m->scal + 6;
  float* s_a = m->scal + 9;
  int P = 0;
  // weights (re-quantized every step: weights change every step) and RMSNorm, per-tensor E4M3: the
  // RMSNorm statistics beside the two weight absmax reductions, then the three casts
  for (int pass = 1; pass <= 2; ++pass)
    FP8Q_STEP(pass == 1 ? kKPrologueStats : kKPrologueCast,
              launch_prologue(pass, (const uint16_t*)m->x, (const uint16_t*)m->g, T, (int)d, m->eps, m->rstd,
                              (const uint16_t*)m->W_gu, d * 2 * f, (const uint16_t*)m->W_d, f * d, w.part_q, w.part_g,
                              w.part_w, m->n8, s_n, m->W_gu8, s_wgu, m->W_d8, s_wd, c.L));
  // G1: H = bf16(alpha n8 @ W_gu8) with the absmax of a = SwiGLU(H) fused in the epilogue
  GemmProblem g1{};
  g1.a_mn = 0;
  g1.b_mn = 1;
  g1.M = (int)T;
  g1.N = (int)f;
  g1.K = (int)d;
  g1.A = m->n8;
  g1.lda = d;
  g1.fmtA = 0;
  g1.B = m->W_gu8;
  g1.ldb = 2 * f;
  g1.fmtB = 0;
  g1.b_cols = 2 * f;
  g1.sinvA = s_n + 2;
  g1.sinvB = s_wgu + 2;
  g1.epi = kEpiSwiglu;
  g1.C = m->H;
  g1.ldc = 2 * f;
  g1.amax_partial = w.part_g;
  FP8Q_STEP(kKGemmGateUp, launch_gemm(g1, &P, c.L));
  // a8 = q(a): a recomputed from the stored H by the epilogue's own SwiGLU (reading H costs the
  // same bytes as reading an fp32 copy of a would), scale from the epilogue's partials
  FP8Q_STEP(kKSwigluCast, launch_swiglu_cast((const uint16_t*)m->H, T, (int)f, 0, w.part_g, P, m->a8, s_a, c.L, true));
  // G2: y = bf16(x + alpha a8 @ W_d8)
  GemmProblem g2{};
  g2.a_mn = 0;
  g2.b_mn = 1;
  g2.M = (int)T;
  g2.N = (int)d;
  g2.K = (int)f;
  g2.A = m->a8;
  g2.lda = f;
  g2.fmtA = 0;
  g2.B = m->W_d8;
  g2.ldb = d;
  g2.fmtB = 0;
  g2.b_cols = d;
  g2.sinvA = s_a + 2;
  g2.sinvB = s_wd + 2;
  g2.epi = kEpiResidual;
  g2.C = m->y;
  g2.ldc = d;
  g2.R = (const uint16_t*)m->x;
  g2.ldr = d;
  FP8Q_STEP(kKGemmDown, launch_gemm(g2, &P, c.L));
  return FP8Q_OK;
}

int mlp_bwd_run(const fp8q_mlp* m, const MlpWs& w, Ctx& c) {
  if (m->bf16) return mlp_bwd_run_bf16(m, w, c);
  if (m->mx) return mlp_bwd_run_mx(m, w, c);
  const int64_t T = m->T, d = m->d, f = m->f;
  const float* s_wgu = m->scal + 0;
  const float* s_wd = m->scal + 3;
  const float* s_n = m->scal + 6;
  const float* s_a = m->scal + 9;
  float* s_dy = m->scal + 12;
  float* s_dh = m->scal + 15;
  if (m->recompute) {
    // H and a8 again from the retained n8, W_gu8 and scales; SwiGLU + E4M3 cast fused
    GemmProblem g1{};
    g1.a_mn = 0;
    g1.b_mn = 1;
    g1.M = (int)T;
    g1.N = (int)f;
    g1.K = (int)d;
    g1.A = m->n8;
    g1.lda = d;
    g1.fmtA = 0;
    g1.B = m->W_gu8;
    g1.ldb = 2 * f;
    g1.fmtB = 0;
    g1.b_cols = 2 * f;
    g1.sinvA = s_n + 2;
    g1.sinvB = s_wgu + 2;
    g1.epi = kEpiSwiglu;
    g1.C = m->H;
    g1.ldc = 2 * f;
    g1.qscale = s_a + 1;
    g1.q8 = m->a8;
    int Pr = 0;
    FP8Q_STEP(kKGemmGateUpRecompute, launch_gemm(g1, &Pr, c.L));
  }
  uint8_t* dY8 = m->dY8 ? m->dY8 : w.dY8;
  uint16_t* dH = m->dH ? (uint16_t*)m->dH : w.dH;
  uint8_t* dH8 = m->dH8 ? m->dH8 : w.dH8;
  float* dN = m->dN ? m->dN : w.dN;
  const int gf = m->grad_e4m3 ? 0 : 1;  // gradient format: E5M2 unless the E4M3 recipe is asked for
  int P = 0;
  // dY8 = q5(dY)
  FP8Q_STEP(kKAbsmaxPartial, launch_absmax_partial(m->dY, 0, T * d, w.part_q, &P, c.L));
  FP8Q_STEP(kKQuantCast, launch_quant_cast(m->dY, 0, T * d, gf, w.part_q, P, dY8, s_dy, c.L));
  // G3 (NT): dA = alpha dY8 @ W_d8^T, SwiGLU backward fused -> dH + absmax partials
  GemmProblem g3{};
  g3.a_mn = 0;
  g3.b_mn = 0;
  g3.M = (int)T;
  g3.N = (int)f;
  g3.K = (int)d;
  g3.A = dY8;
  g3.lda = d;
  g3.fmtA = gf;
  g3.B = m->W_d8;
  g3.ldb = d;
  g3.fmtB = 0;
  g3.b_cols = f;
  g3.sinvA = s_dy + 2;
  g3.sinvB = s_wd + 2;
  g3.epi = kEpiSwigluBwd;
  g3.C = dH;
  g3.ldc = 2 * f;
  g3.R = (const uint16_t*)m->H;
  g3.ldr = 2 * f;
  g3.amax_partial = w.part_g;
  FP8Q_STEP(kKGemmDownDgrad, launch_gemm(g3, &P, c.L));
  // dH8 = q5(dH)
  FP8Q_STEP(kKQuantCast, launch_quant_cast(dH, 0, T * 2 * f, gf, w.part_g, P, dH8, s_dh, c.L));
  // G4 (TN): dW_d = alpha a8^T @ dY8
  GemmProblem g4{};
  g4.a_mn = 1;
  g4.b_mn = 1;
  g4.M = (int)f;
  g4.N = (int)d;
  g4.K = (int)T;
  g4.A = m->a8;
  g4.lda = f;
  g4.fmtA = 0;
  g4.B = dY8;
  g4.ldb = d;
  g4.fmtB = gf;
  g4.b_cols = d;
  g4.sinvA = s_a + 2;
  g4.sinvB = s_dy + 2;
  g4.epi = kEpiStore;
  g4.out_f32 = 1;
  g4.C = m->dW_d;
  g4.ldc = d;
  FP8Q_STEP(kKGemmDownWgrad, launch_gemm(g4, &P, c.L));
  // G5 (NT): dN = alpha dH8 @ W_gu8^T
  GemmProblem g5{};
  g5.a_mn = 0;
  g5.b_mn = 0;
  g5.M = (int)T;
  g5.N = (int)d;
  g5.K = (int)(2 * f);
  g5.A = dH8;
  g5.lda = 2 * f;
  g5.fmtA = gf;
  g5.B = m->W_gu8;
  g5.ldb = 2 * f;
  g5.fmtB = 0;
  g5.b_cols = d;
  g5.sinvA = s_dh + 2;
  g5.sinvB = s_wgu + 2;
  g5.epi = kEpiStore;
  g5.out_f32 = 1;
  g5.C = dN;
  g5.ldc = d;
  FP8Q_STEP(kKGemmGateUpDgrad, launch_gemm(g5, &P, c.L));
  // G6 (TN): dW_gu = alpha n8^T @ dH8
  GemmProblem g6{};
  g6.a_mn = 1;
  g6.b_mn = 1;
  g6.M = (int)d;
  g6.N = (int)(2 * f);
  g6.K = (int)T;
  g6.A = m->n8;
  g6.lda = d;
  g6.fmtA = 0;
  g6.B = dH8;
  g6.ldb = 2 * f;
  g6.fmtB = gf;
  g6.b_cols = 2 * f;
  g6.sinvA = s_n + 2;
  g6.sinvB = s_dh + 2;
  g6.epi = kEpiStore;
  g6.out_f32 = 1;
  g6.C = m->dW_gu;
  g6.ldc = 2 * f;
  FP8Q_STEP(kKGemmGateUpWgrad, launch_gemm(g6, &P, c.L));
  // RMSNorm backward + residual
  FP8Q_STEP(kKRmsnormBwd, launch_rmsnorm_bwd(dN, (const uint16_t*)m->x, (const uint16_t*)m->dY, (const uint16_t*)m->g, m->rstd,
                              T, (int)d, (uint16_t*)m->dX, w.dg_part, m->dg, c.L));
  return FP8Q_OK;
}

// ---- the full block ---------------------------------------------------------
struct BlockWs {
  MlpWs mlp;
  uint8_t* mlp_base;
  uint32_t* part;   // attention-side quantizer partials
  uint8_t* dh8;     // [T,d] E5M2
  uint8_t* dqkv8;   // [T,nq] E5M2
  float* dN1;       // [T,d]
  float* dg1_part;  // dg partials of the attention-side RMSNorm backward
  float* attn_delta;  // [d/128, T] the attention core backward's D (core mode)
  float* attn_lse2;   // [d/128, T] its lse in the log2 domain
};

size_t block_ws_layout(int64_t T, int64_t d, int64_t f, int64_t nq, int backward, uint8_t* base, BlockWs* w) {
  const size_t mlp_bytes = round256(mlp_ws_layout(T, d, f, backward, nullptr, nullptr));
  Carver c{base, ~size_t(0)};
  BlockWs tmp{};
  tmp.mlp_base = (uint8_t*)c.take(mlp_bytes);
  tmp.part = (uint32_t*)c.take(kPartialBytes);
  if (backward) {
    tmp.dh8 = (uint8_t*)c.take((size_t)(T * d));
    tmp.dqkv8 = (uint8_t*)c.take((size_t)(T * nq));
    tmp.dN1 = (float*)c.take((size_t)(T * d) * 4);
    tmp.dg1_part = (float*)c.take((size_t)((T + kBwdRows - 1) / kBwdRows) * (size_t)d * 4);
    tmp.attn_delta = (float*)c.take((size_t)T * (size_t)(d / 128) * 4);
    tmp.attn_lse2 = (float*)c.take((size_t)T * (size_t)(d / 128) * 4);
  }
  if (base) mlp_ws_layout(T, d, f, backward, tmp.mlp_base, &tmp.mlp);
  if (w) *w = tmp;
  return c.off;
}

// The attention core's shape conditions (see attention_fwd in fp8q.h).
int validate_attention(const void* qkv, int64_t T, int64_t S, int Hq, int Hkv, int dh) {
  if (!al16(qkv) || T < 1 || S < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || T % S) return FP8Q_ERR_INVALID_ARG;
  if (dh != 128 || S % 128) return FP8Q_ERR_UNSUPPORTED;
  // the kernels' one-dimensional grids count (T / 128) x n_heads CTAs in an int
  if (T > ((int64_t)1 << 31) - 1 || T / 128 * Hq > ((int64_t)1 << 31) - 1) return FP8Q_ERR_INVALID_ARG;
  return FP8Q_OK;
}

int validate_block(const fp8q_block* b, bool backward) {
  if (!b) return FP8Q_ERR_INVALID_ARG;
  const fp8q_mlp& m = b->mlp;
  if (m.T != b->T || m.d != b->d || m.f != b->f || m.x != b->h) return FP8Q_ERR_INVALID_ARG;
  if (m.mx) return FP8Q_ERR_UNSUPPORTED;  // the MXFP8 mode is built for the MLP block
  if (b->n_qkv < 16 || b->n_qkv % 16 || b->n_qkv > (int64_t)1 << 20) return FP8Q_ERR_INVALID_ARG;
  int e = validate_mlp(&m, backward);
  if (e) return e;
  if (b->n_heads) {
    if (b->n_kv_heads < 1 || (int64_t)b->n_heads * 128 != b->d ||
        (int64_t)(b->n_heads + 2 * b->n_kv_heads) * 128 != b->n_qkv || !al16(b->lse))
      return FP8Q_ERR_INVALID_ARG;
    if ((e = validate_attention(b->qkv, b->T, b->seq_len, b->n_heads, b->n_kv_heads, 128))) return e;
  }
  if (m.bf16) {
    const void* must16[] = {b->x, b->g1, b->W_qkv, b->W_o, b->att, b->qkv, b->h, b->rstd1, b->n1_16};
    for (const void* p : must16)
      if (!al16(p)) return FP8Q_ERR_INVALID_ARG;
  } else {
    const void* must[] = {b->x, b->g1, b->W_qkv, b->W_o, b->att, b->qkv, b->h, b->W_qkv8, b->W_o8, b->n1_8,
                          b->rstd1, b->att8, b->scal};
    for (const void* p : must)
      if (!al16(p)) return FP8Q_ERR_INVALID_ARG;
  }
  if (!backward) return FP8Q_OK;
  const void* must_b[] = {b->dQKV, b->d_att, b->dX, b->dW_qkv, b->dW_o, b->dg1};
  for (const void* p : must_b)
    if (!al16(p)) return FP8Q_ERR_INVALID_ARG;
  const void* opt[] = {b->dh8, b->dQKV8, b->dN1};
  for (const void* p : opt)
    if (p && !al16(p)) return FP8Q_ERR_INVALID_ARG;
  return FP8Q_OK;
}

GemmProblem gemm_problem(int a_mn, int b_mn, int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                         int fmtA, const uint8_t* B, int64_t ldb, int fmtB, int64_t b_cols, const float* sinvA,
                         const float* sinvB, int epi, int out_f32, void* C, int64_t ldc) {
  GemmProblem g{};
  g.a_mn = a_mn;
  g.b_mn = b_mn;
  g.M = (int)M;
  g.N = (int)N;
  g.K = (int)K;
  g.A = A;
  g.lda = lda;
  g.fmtA = fmtA;
  g.B = B;
  g.ldb = ldb;
  g.fmtB = fmtB;
  g.b_cols = b_cols;
  g.sinvA = sinvA;
  g.sinvB = sinvB;
  g.epi = epi;
  g.out_f32 = out_f32;
  g.C = C;
  g.ldc = ldc;
  return g;
}

// The block's BF16 baseline: the FP8 sequences with every cast removed (bf16 operands, alpha = 1).
int block_fwd_run_bf16(const fp8q_block* b, const BlockWs& w, Ctx& c) {
  const int64_t T = b->T, d = b->d, nq = b->n_qkv;
  int P = 0;
  FP8Q_STEP(kKRmsnormBf16, launch_rmsnorm_bf16((const uint16_t*)b->x, (const uint16_t*)b->g1, T, (int)d, b->eps,
                                               b->rstd1, (uint16_t*)b->n1_16, c.L));
  FP8Q_STEP(kKGemmQkv,
            launch_gemm(bf16_gemm(0, 1, T, nq, d, b->n1_16, d, b->W_qkv, nq, nq, kEpiStore, 0, b->qkv, nq), &P, c.L));
  if (b->n_heads)
    FP8Q_STEP(kKAttnFwd, launch_attn_fwd((const uint16_t*)b->qkv, T, (int)b->seq_len, b->n_heads, b->n_kv_heads,
                                         (uint16_t*)b->att, b->lse, c.L));
  GemmProblem go = bf16_gemm(0, 1, T, d, d, b->att, d, b->W_o, d, d, kEpiResidual, 0, b->h, d);
  go.R = (const uint16_t*)b->x;
  go.ldr = d;
  FP8Q_STEP(kKGemmOResidual, launch_gemm(go, &P, c.L));
  return mlp_fwd_run(&b->mlp, w.mlp, c);
}

int block_bwd_run_bf16(const fp8q_block* b, const BlockWs& w, Ctx& c) {
  const int64_t T = b->T, d = b->d, nq = b->n_qkv;
  int e = mlp_bwd_run(&b->mlp, w.mlp, c);
  if (e) return e;
  const void* dh = b->mlp.dX;
  float* dN1 = b->dN1 ? b->dN1 : w.dN1;
  int P = 0;
  FP8Q_STEP(kKGemmODgrad,
            launch_gemm(bf16_gemm(0, 0, T, d, d, dh, d, b->W_o, d, d, kEpiStore, 0, b->d_att, d), &P, c.L));
  FP8Q_STEP(kKGemmOWgrad,
            launch_gemm(bf16_gemm(1, 1, d, d, T, b->att, d, dh, d, d, kEpiStore, 1, b->dW_o, d), &P, c.L));
  if (b->n_heads) {
    const uint16_t* q16 = (const uint16_t*)b->qkv;
    const uint16_t* do16 = (const uint16_t*)b->d_att;
    const int S = (int)b->seq_len;
    FP8Q_STEP(kKAttnBwdDelta, launch_attn_bwd_delta((const uint16_t*)b->att, do16, b->lse, T, b->n_heads,
                                                    w.attn_delta, w.attn_lse2, c.L));
    FP8Q_STEP(kKAttnBwdDkdv, launch_attn_bwd_dkdv(q16, do16, T, S, b->n_heads, b->n_kv_heads, w.attn_delta,
                                                  w.attn_lse2, (uint16_t*)b->dQKV, c.L));
    FP8Q_STEP(kKAttnBwdDq, launch_attn_bwd_dq(q16, do16, T, S, b->n_heads, b->n_kv_heads, w.attn_delta, w.attn_lse2,
                                              (uint16_t*)b->dQKV, c.L));
  }
  FP8Q_STEP(kKGemmQkvDgrad,
            launch_gemm(bf16_gemm(0, 0, T, d, nq, b->dQKV, nq, b->W_qkv, nq, d, kEpiStore, 1, dN1, d), &P, c.L));
  FP8Q_STEP(kKGemmQkvWgrad, launch_gemm(bf16_gemm(1, 1, d, nq, T, b->n1_16, d, b->dQKV, nq, nq, kEpiStore, 1,
                                                  b->dW_qkv, nq),
                                        &P, c.L));
  FP8Q_STEP(kKRmsnormBwd, launch_rmsnorm_bwd(dN1, (const uint16_t*)b->x, (const uint16_t*)dh,
                                             (const uint16_t*)b->g1, b->rstd1, T, (int)d, (uint16_t*)b->dX,
                                             w.dg1_part, b->dg1, c.L));
  return FP8Q_OK;
}

int block_fwd_run(const fp8q_block* b, const BlockWs& w, Ctx& c) {
  if (b->mlp.bf16) return block_fwd_run_bf16(b, w, c);
  const int64_t T = b->T, d = b->d, nq = b->n_qkv;
  float* s_qkv = b->scal + 0;
  float* s_o = b->scal + 3;
  float* s_n1 = b->scal + 6;
  float* s_att = b->scal + 9;
  int P = 0;
  // W_qkv, W_o and the attention-side RMSNorm, per-tensor E4M3, through the two-launch prologue (the
  // MLP's partial arrays are free until the MLP runs)
  for (int pass = 1; pass <= 2; ++pass)
    FP8Q_STEP(pass == 1 ? kKPrologueStats : kKPrologueCast,
              launch_prologue(pass, (const uint16_t*)b->x, (const uint16_t*)b->g1, T, (int)d, b->eps, b->rstd1,
                              (const uint16_t*)b->W_qkv, d * nq, (const uint16_t*)b->W_o, d * d, w.part,
                              w.mlp.part_q, w.mlp.part_g, b->n1_8, s_n1, b->W_qkv8, s_qkv, b->W_o8, s_o, c.L));
  // qkv = bf16(alpha n1_8 @ W_qkv8)
  GemmProblem gq = gemm_problem(0, 1, T, nq, d, b->n1_8, d, 0, b->W_qkv8, nq, 0, nq, s_n1 + 2, s_qkv + 2, kEpiStore,
                                0, b->qkv, nq);
  FP8Q_STEP(kKGemmQkv, launch_gemm(gq, &P, c.L));
  // the attention core: att (and lse) from qkv
  if (b->n_heads)
    FP8Q_STEP(kKAttnFwd, launch_attn_fwd((const uint16_t*)b->qkv, T, (int)b->seq_len, b->n_heads, b->n_kv_heads,
                                         (uint16_t*)b->att, b->lse, c.L));
  // h = bf16(x + alpha q(att) @ W_o8)
  FP8Q_STEP(kKAbsmaxPartial, launch_absmax_partial(b->att, 0, T * d, w.part, &P, c.L));
  FP8Q_STEP(kKQuantCast, launch_quant_cast(b->att, 0, T * d, 0, w.part, P, b->att8, s_att, c.L));
  GemmProblem go = gemm_problem(0, 1, T, d, d, b->att8, d, 0, b->W_o8, d, 0, d, s_att + 2, s_o + 2, kEpiResidual, 0,
                                b->h, d);
  go.R = (const uint16_t*)b->x;
  go.ldr = d;
  FP8Q_STEP(kKGemmOResidual, launch_gemm(go, &P, c.L));
  return mlp_fwd_run(&b->mlp, w.mlp, c);
}

int block_bwd_run(const fp8q_block* b, const BlockWs& w, Ctx& c) {
  if (b->mlp.bf16) return block_bwd_run_bf16(b, w, c);
  const int64_t T = b->T, d = b->d, nq = b->n_qkv;
  const float* s_qkv = b->scal + 0;
  const float* s_o = b->scal + 3;
  const float* s_n1 = b->scal + 6;
  const float* s_att = b->scal + 9;
  float* s_dh = b->scal + 12;
  float* s_dq = b->scal + 15;
  int e = mlp_bwd_run(&b->mlp, w.mlp, c);
  if (e) return e;
  const void* dh = b->mlp.dX;
  uint8_t* dh8 = b->dh8 ? b->dh8 : w.dh8;
  uint8_t* dqkv8 = b->dQKV8 ? b->dQKV8 : w.dqkv8;
  float* dN1 = b->dN1 ? b->dN1 : w.dN1;
  const int gf = b->mlp.grad_e4m3 ? 0 : 1;
  int P = 0;
  FP8Q_STEP(kKAbsmaxPartial, launch_absmax_partial(dh, 0, T * d, w.part, &P, c.L));
  FP8Q_STEP(kKQuantCast, launch_quant_cast(dh, 0, T * d, gf, w.part, P, dh8, s_dh, c.L));
  // d_att = bf16(alpha dh8 @ W_o8^T): B = W_o8 [d_in, d_out] is K-major for this product
  GemmProblem god = gemm_problem(0, 0, T, d, d, dh8, d, gf, b->W_o8, d, 0, d, s_dh + 2, s_o + 2, kEpiStore, 0,
                                 b->d_att, d);
  FP8Q_STEP(kKGemmODgrad, launch_gemm(god, &P, c.L));
  // dW_o = alpha att8^T @ dh8
  GemmProblem gow = gemm_problem(1, 1, d, d, T, b->att8, d, 0, dh8, d, gf, d, s_att + 2, s_dh + 2, kEpiStore, 1,
                                 b->dW_o, d);
  FP8Q_STEP(kKGemmOWgrad, launch_gemm(gow, &P, c.L));
  // the attention core's backward: dQKV from d_att
  if (b->n_heads) {
    const uint16_t* q16 = (const uint16_t*)b->qkv;
    const uint16_t* do16 = (const uint16_t*)b->d_att;
    const int S = (int)b->seq_len;
    FP8Q_STEP(kKAttnBwdDelta, launch_attn_bwd_delta((const uint16_t*)b->att, do16, b->lse, T, b->n_heads,
                                                    w.attn_delta, w.attn_lse2, c.L));
    FP8Q_STEP(kKAttnBwdDkdv, launch_attn_bwd_dkdv(q16, do16, T, S, b->n_heads, b->n_kv_heads, w.attn_delta,
                                                  w.attn_lse2, (uint16_t*)b->dQKV, c.L));
    FP8Q_STEP(kKAttnBwdDq, launch_attn_bwd_dq(q16, do16, T, S, b->n_heads, b->n_kv_heads, w.attn_delta, w.attn_lse2,
                                              (uint16_t*)b->dQKV, c.L));
  }
  // dQKV8 = q5(dQKV); dN1 = alpha dQKV8 @ W_qkv8^T; dW_qkv = alpha n1_8^T @ dQKV8
  FP8Q_STEP(kKAbsmaxPartial, launch_absmax_partial(b->dQKV, 0, T * nq, w.part, &P, c.L));
  FP8Q_STEP(kKQuantCast, launch_quant_cast(b->dQKV, 0, T * nq, gf, w.part, P, dqkv8, s_dq, c.L));
  GemmProblem gqd = gemm_problem(0, 0, T, d, nq, dqkv8, nq, gf, b->W_qkv8, nq, 0, d, s_dq + 2, s_qkv + 2, kEpiStore,
                                 1, dN1, d);
  FP8Q_STEP(kKGemmQkvDgrad, launch_gemm(gqd, &P, c.L));
  GemmProblem gqw = gemm_problem(1, 1, d, nq, T, b->n1_8, d, 0, dqkv8, nq, gf, nq, s_n1 + 2, s_dq + 2, kEpiStore, 1,
                                 b->dW_qkv, nq);
  FP8Q_STEP(kKGemmQkvWgrad, launch_gemm(gqw, &P, c.L));
  // dX = bf16(dh + RMSNorm_1'(dN1)), dg1
  FP8Q_STEP(kKRmsnormBwd, launch_rmsnorm_bwd(dN1, (const uint16_t*)b->x, (const uint16_t*)dh,
                                             (const uint16_t*)b->g1, b->rstd1, T, (int)d, (uint16_t*)b->dX,
                                             w.dg1_part, b->dg1, c.L));
  return FP8Q_OK;
}

}  // namespace

int fp8q::device_status_and_sms(unsigned** status, int* num_sms) {
  DevInfo d;
  if (device_info(&d)) return FP8Q_ERR_CUDA;
  *status = d.status;
  *num_sms = d.num_sms;
  return FP8Q_OK;
}

extern "C" {

// ---------------------------------------------------------------------------
size_t fp8_quantize_absmax_workspace_size(int64_t n) {
  (void)n;
  return round256(kPartialBytes);
}

int fp8_quantize_absmax(const void* x, fp8q_dtype x_dtype, int64_t n, fp8q_fmt fmt, uint8_t* q, float* scal,
                        void* ws, size_t ws_bytes, fp8q_stream stream) {
  if (n < 1 || !al16(x) || !al16(q) || !scal || ((uintptr_t)scal & 3u)) return FP8Q_ERR_INVALID_ARG;
  if ((x_dtype != FP8Q_BF16 && x_dtype != FP8Q_F32) || (fmt != FP8Q_E4M3 && fmt != FP8Q_E5M2))
    return FP8Q_ERR_INVALID_ARG;
  int e = check_ws(ws, ws_bytes, fp8_quantize_absmax_workspace_size(n));
  if (e) return e;
  Ctx c;
  if ((e = make_ctx(&c, stream))) return e;
  uint32_t* part = static_cast<uint32_t*>(ws);
  int P = 0;
  FP8Q_STEP(kKAbsmaxPartial, launch_absmax_partial(x, (int)x_dtype, n, part, &P, c.L));
  FP8Q_STEP(kKQuantCast, launch_quant_cast(x, (int)x_dtype, n, (int)fmt, part, P, q, scal, c.L));
  return finish(c);
}

// ---------------------------------------------------------------------------
int fp8_gemm_scaled(fp8q_layout layout, int64_t M, int64_t N, int64_t K, const uint8_t* A, fp8q_fmt fmtA,
                    int64_t lda, const uint8_t* B, fp8q_fmt fmtB, int64_t ldb, const float* sinvA,
                    const float* sinvB, void* C, fp8q_dtype out_dtype, int64_t ldc, const void* residual,
                    int64_t ldr, fp8q_stream stream) {
  if (M < 1 || N < 1 || K < 1 || M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return FP8Q_ERR_INVALID_ARG;
  if (!al16(A) || !al16(B) || !al16(C) || !sinvA || !sinvB) return FP8Q_ERR_INVALID_ARG;
  if ((fmtA != FP8Q_E4M3 && fmtA != FP8Q_E5M2) || (fmtB != FP8Q_E4M3 && fmtB != FP8Q_E5M2))
    return FP8Q_ERR_INVALID_ARG;
  if (out_dtype != FP8Q_BF16 && out_dtype != FP8Q_F32) return FP8Q_ERR_INVALID_ARG;
  if (layout != FP8Q_NN && layout != FP8Q_NT && layout != FP8Q_TN) return FP8Q_ERR_INVALID_ARG;
  GemmProblem g{};
  g.a_mn = layout == FP8Q_TN;
  g.b_mn = layout != FP8Q_NT;
  const int64_t a_inner = g.a_mn ? M : K, b_inner = g.b_mn ? N : K;
  if (a_inner % 16 || b_inner % 16 || lda < a_inner || ldb < b_inner || lda % 16 || ldb % 16)
    return FP8Q_ERR_INVALID_ARG;
  if (ldc < N || ldc % 8) return FP8Q_ERR_INVALID_ARG;
  if (residual) {
    if (out_dtype != FP8Q_BF16 || !al16(residual) || ldr < N || ldr % 8) return FP8Q_ERR_INVALID_ARG;
  }
  Ctx c;
  int e = make_ctx(&c, stream);
  if (e) return e;
  g.M = (int)M;
  g.N = (int)N;
  g.K = (int)K;
  g.A = A;
  g.lda = lda;
  g.fmtA = (int)fmtA;
  g.B = B;
  g.ldb = ldb;
  g.fmtB = (int)fmtB;
  g.b_cols = N;
  g.sinvA = sinvA;
  g.sinvB = sinvB;
  g.epi = residual ? kEpiResidual : kEpiStore;
  g.out_f32 = out_dtype == FP8Q_F32;
  g.C = C;
  g.ldc = ldc;
  g.R = static_cast<const uint16_t*>(residual);
  g.ldr = ldr;
  g.wait_ns = t_gemm_wait_ns;
  int P = 0;
  FP8Q_STEP(kKGemm, launch_gemm(g, &P, c.L));
  return finish(c);
}

// ---------------------------------------------------------------------------
int fp8q_selftest_gemm_wait_limit(fp8q_layout layout, int64_t M, int64_t N, int64_t K, const uint8_t* A,
                                  fp8q_fmt fmtA, int64_t lda, const uint8_t* B, fp8q_fmt fmtB, int64_t ldb,
                                  const float* sinvA, const float* sinvB, int mx, const uint8_t* sfA,
                                  const uint8_t* sfB, void* C, fp8q_dtype out_dtype, int64_t ldc, int64_t limit_ns,
                                  fp8q_stream stream) {
  if (limit_ns < 1000 || limit_ns > 10000000000ll) return FP8Q_ERR_INVALID_ARG;
  t_gemm_wait_ns = (uint64_t)limit_ns;
  const int rc = mx ? fp8_gemm_mx(layout, M, N, K, A, fmtA, lda, sfA, B, fmtB, ldb, sfB, C, out_dtype, ldc, nullptr,
                                  0, stream)
                    : fp8_gemm_scaled(layout, M, N, K, A, fmtA, lda, B, fmtB, ldb, sinvA, sinvB, C, out_dtype, ldc,
                                      nullptr, 0, stream);
  t_gemm_wait_ns = 0;
  return rc;
}

// ---------------------------------------------------------------------------
size_t mx_scale_bytes(int64_t rows, int64_t K) { return fp8q::mx_scale_bytes(rows, K); }

int mx_quantize(const void* x, fp8q_dtype x_dtype, int64_t R, int64_t C, fp8q_fmt fmt, uint8_t* q_r, uint8_t* sf_r,
                uint8_t* q_c, uint8_t* sf_c, fp8q_stream stream) {
  if (!al16(x) || R < 128 || C < 128 || R % 128 || C % 128 || R > ((int64_t)1 << 30) || C > ((int64_t)1 << 30))
    return FP8Q_ERR_INVALID_ARG;
  if ((x_dtype != FP8Q_BF16 && x_dtype != FP8Q_F32) || (fmt != FP8Q_E4M3 && fmt != FP8Q_E5M2))
    return FP8Q_ERR_INVALID_ARG;
  if (!q_r && !q_c) return FP8Q_ERR_INVALID_ARG;
  if ((q_r && (!al16(q_r) || !al16(sf_r))) || (q_c && (!al16(q_c) || !al16(sf_c)))) return FP8Q_ERR_INVALID_ARG;
  Ctx c;
  int e = make_ctx(&c, stream);
  if (e) return e;
  FP8Q_STEP(kKMxQuant, launch_mx_quant(x_dtype == FP8Q_BF16 ? kMxInBf16 : kMxInF32, x, nullptr, nullptr, R, C,
                                       (int)fmt, q_r, q_r ? sf_r : nullptr, q_c, q_c ? sf_c : nullptr, c.L));
  return finish(c);
}

int fp8_gemm_mx(fp8q_layout layout, int64_t M, int64_t N, int64_t K, const uint8_t* A, fp8q_fmt fmtA, int64_t lda,
                const uint8_t* sfA, const uint8_t* B, fp8q_fmt fmtB, int64_t ldb, const uint8_t* sfB, void* C,
                fp8q_dtype out_dtype, int64_t ldc, const void* residual, int64_t ldr, fp8q_stream stream) {
  if (M < 1 || N < 1 || K < 128 || K % 128 || M > (1 << 30) || N > (1 << 30) || K > (1 << 30))
    return FP8Q_ERR_INVALID_ARG;
  if (!al16(A) || !al16(B) || !al16(C) || !al16(sfA) || !al16(sfB)) return FP8Q_ERR_INVALID_ARG;
  if ((fmtA != FP8Q_E4M3 && fmtA != FP8Q_E5M2) || (fmtB != FP8Q_E4M3 && fmtB != FP8Q_E5M2))
    return FP8Q_ERR_INVALID_ARG;
  if (out_dtype != FP8Q_BF16 && out_dtype != FP8Q_F32) return FP8Q_ERR_INVALID_ARG;
  if (layout != FP8Q_NN && layout != FP8Q_NT && layout != FP8Q_TN) return FP8Q_ERR_INVALID_ARG;
  const int a_mn = layout == FP8Q_TN, b_mn = layout != FP8Q_NT;
  const int64_t a_inner = a_mn ? M : K, b_inner = b_mn ? N : K;
  if (a_inner % 16 || b_inner % 16 || lda < a_inner || ldb < b_inner || lda % 16 || ldb % 16)
    return FP8Q_ERR_INVALID_ARG;
  if (ldc < N || ldc % 8) return FP8Q_ERR_INVALID_ARG;
  if (residual && (out_dtype != FP8Q_BF16 || !al16(residual) || ldr < N || ldr % 8)) return FP8Q_ERR_INVALID_ARG;
  Ctx c;
  int e = make_ctx(&c, stream);
  if (e) return e;
  GemmProblem g = mx_gemm(a_mn, b_mn, M, N, K, fp8q_mx_tensor{const_cast<uint8_t*>(A), const_cast<uint8_t*>(sfA)},
                          (int)fmtA, lda, fp8q_mx_tensor{const_cast<uint8_t*>(B), const_cast<uint8_t*>(sfB)}, (int)fmtB,
                          ldb, N, residual ? kEpiResidual : kEpiStore, out_dtype == FP8Q_F32, C, ldc);
  g.R = static_cast<const uint16_t*>(residual);
  g.ldr = ldr;
  g.wait_ns = t_gemm_wait_ns;
  int P = 0;
  FP8Q_STEP(kKGemm, launch_gemm(g, &P, c.L));
  return finish(c);
}

// ---------------------------------------------------------------------------
size_t rmsnorm_quant_workspace_size(int64_t T, int64_t d) {
  (void)T;
  (void)d;
  return round256(kPartialBytes);
}

int rmsnorm_quant(const void* x, const void* g, int64_t T, int64_t d, float eps, uint8_t* q, float* scal,
                  float* rstd, void* ws, size_t ws_bytes, fp8q_stream stream) {
  if (T < 1 || d < 16 || d % 16 || d > 8192 || T > ((int64_t)1 << 28)) return FP8Q_ERR_INVALID_ARG;
  if (!al16(x) || !al16(g) || !al16(q) || !scal || !rstd || !(eps >= 0.0f)) return FP8Q_ERR_INVALID_ARG;
  int e = check_ws(ws, ws_bytes, rmsnorm_quant_workspace_size(T, d));
  if (e) return e;
  Ctx c;
  if ((e = make_ctx(&c, stream))) return e;
  uint32_t* part = static_cast<uint32_t*>(ws);
  int P = 0;
  FP8Q_STEP(kKRmsnormStats, launch_rmsnorm_stats((const uint16_t*)x, (const uint16_t*)g, T, (int)d, eps, rstd, part, &P, c.L));
  FP8Q_STEP(kKRmsnormCast, launch_rmsnorm_cast((const uint16_t*)x, (const uint16_t*)g, rstd, T, (int)d, part, P, q, scal, c.L));
  return finish(c);
}

// ---------------------------------------------------------------------------
size_t rmsnorm_bwd_workspace_size(int64_t T, int64_t d) {
  if (T < 1 || d < 1) return 0;
  return round256((size_t)((T + kBwdRows - 1) / kBwdRows) * (size_t)d * 4);
}

namespace {
int rmsnorm_bwd_run(const float* dN, const void* x, const void* dY, const void* g, const float* rstd, int64_t T,
                    int64_t d, void* dX, float* dg, void* ws, size_t ws_bytes, fp8q_stream stream, uint64_t wait_ns) {
  if (T < 1 || d < 16 || d % 16 || d > 8192 || T > ((int64_t)1 << 28)) return FP8Q_ERR_INVALID_ARG;
  if (!al16(dN) || !al16(x) || !al16(dY) || !al16(g) || !al16(dX)) return FP8Q_ERR_INVALID_ARG;
  if (!rstd || ((uintptr_t)rstd & 3u) || !dg || ((uintptr_t)dg & 3u)) return FP8Q_ERR_INVALID_ARG;
  int e = check_ws(ws, ws_bytes, rmsnorm_bwd_workspace_size(T, d));
  if (e) return e;
  Ctx c;
  if ((e = make_ctx(&c, stream))) return e;
  FP8Q_STEP(kKRmsnormBwd, launch_rmsnorm_bwd(dN, (const uint16_t*)x, (const uint16_t*)dY, (const uint16_t*)g, rstd,
                                             T, (int)d, (uint16_t*)dX, static_cast<float*>(ws), dg, c.L, wait_ns));
  return finish(c);
}
}  // namespace

int rmsnorm_bwd(const float* dN, const void* x, const void* dY, const void* g, const float* rstd, int64_t T,
                int64_t d, void* dX, float* dg, void* ws, size_t ws_bytes, fp8q_stream stream) {
  return rmsnorm_bwd_run(dN, x, dY, g, rstd, T, d, dX, dg, ws, ws_bytes, stream, 0);
}

int fp8q_selftest_rmsnorm_bwd_wait_limit(const float* dN, const void* x, const void* dY, const void* g,
                                         const float* rstd, int64_t T, int64_t d, void* dX, float* dg, void* ws,
                                         size_t ws_bytes, int64_t limit_ns, fp8q_stream stream) {
  if (limit_ns < 1 || limit_ns > 10000000000LL) return FP8Q_ERR_INVALID_ARG;
  return rmsnorm_bwd_run(dN, x, dY, g, rstd, T, d, dX, dg, ws, ws_bytes, stream, (uint64_t)limit_ns);
}

// ---------------------------------------------------------------------------
size_t swiglu_quant_workspace_size(int64_t T, int64_t f) {
  (void)T;
  (void)f;
  return round256(kPartialBytes);
}

int swiglu_quant(const void* H, int64_t T, int64_t f, fp8q_fmt fmt, uint8_t* q, float* scal, void* ws,
                 size_t ws_bytes, fp8q_stream stream) {
  if (T < 1 || f < 16 || f % 16 || f > (1 << 24) || T > ((int64_t)1 << 28)) return FP8Q_ERR_INVALID_ARG;
  if (!al16(H) || !al16(q) || !scal || (fmt != FP8Q_E4M3 && fmt != FP8Q_E5M2)) return FP8Q_ERR_INVALID_ARG;
  int e = check_ws(ws, ws_bytes, swiglu_quant_workspace_size(T, f));
  if (e) return e;
  Ctx c;
  if ((e = make_ctx(&c, stream))) return e;
  uint32_t* part = static_cast<uint32_t*>(ws);
  int P = 0;
  FP8Q_STEP(kKSwigluAmax, launch_swiglu_amax((const uint16_t*)H, T, (int)f, part, &P, c.L));
  FP8Q_STEP(kKSwigluCast, launch_swiglu_cast((const uint16_t*)H, T, (int)f, (int)fmt, part, P, q, scal, c.L));
  return finish(c);
}

// ---------------------------------------------------------------------------
size_t mlp_block_workspace_size(int64_t T, int64_t d, int64_t f, int backward) {
  return mlp_ws_layout(T, d, f, backward, nullptr, nullptr);
}

int mlp_block_fwd(const fp8q_mlp* m, void* ws, size_t ws_bytes, fp8q_stream stream) {
  int e = validate_mlp(m, false);
  if (e) return e;
  if ((e = check_ws(ws, ws_bytes, mlp_block_workspace_size(m->T, m->d, m->f, 0)))) return e;
  Ctx c;
  if ((e = make_ctx(&c, stream))) return e;
  MlpWs w;
  mlp_ws_layout(m->T, m->d, m->f, 0, static_cast<uint8_t*>(ws), &w);
  if ((e = mlp_fwd_run(m, w, c))) return e;
  return finish(c);
}

int mlp_block_bwd(const fp8q_mlp* m, void* ws, size_t ws_bytes, fp8q_stream stream) {
  int e = validate_mlp(m, true);
  if (e) return e;
  if ((e = check_ws(ws, ws_bytes, mlp_block_workspace_size(m->T, m->d, m->f, 1)))) return e;
  Ctx c;
  if ((e = make_ctx(&c, stream))) return e;
  MlpWs w;
  mlp_ws_layout(m->T, m->d, m->f, 1, static_cast<uint8_t*>(ws), &w);
  if ((e = mlp_bwd_run(m, w, c))) return e;
  return finish(c);
}

// ---------------------------------------------------------------------------
size_t block_workspace_size(int64_t T, int64_t d, int64_t f, int64_t n_qkv, int backward) {
  return block_ws_layout(T, d, f, n_qkv, backward, nullptr, nullptr);
}

int block_fwd(const fp8q_block* b, void* ws, size_t ws_bytes, fp8q_stream stream) {
  int e = validate_block(b, false);
  if (e) return e;
  if ((e = check_ws(ws, ws_bytes, block_workspace_size(b->T, b->d, b->f, b->n_qkv, 0)))) return e;
  Ctx c;
  if ((e = make_ctx(&c, stream))) return e;
  BlockWs w;
  block_ws_layout(b->T, b->d, b->f, b->n_qkv, 0, static_cast<uint8_t*>(ws), &w);
  if ((e = block_fwd_run(b, w, c))) return e;
  return finish(c);
}

int block_bwd(const fp8q_block* b, void* ws, size_t ws_bytes, fp8q_stream stream) {
  int e = validate_block(b, true);
  if (e) return e;
  if ((e = check_ws(ws, ws_bytes, block_workspace_size(b->T, b->d, b->f, b->n_qkv, 1)))) return e;
  Ctx c;
  if ((e = make_ctx(&c, stream))) return e;
  BlockWs w;
  block_ws_layout(b->T, b->d, b->f, b->n_qkv, 1, static_cast<uint8_t*>(ws), &w);
  if ((e = block_bwd_run(b, w, c))) return e;
  return finish(c);
}

// ---------------------------------------------------------------------------
// Pipelined steps from and to host memory
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {

// Two copy streams and the events that order the pipeline, created once per device.
struct CopyEngines {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t in_done[2], compute_done[2], out_done[2];
  bool ready = false;
};

int copy_engines(CopyEngines** out) {
  static std::mutex mu;
  static CopyEngines cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8Q_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  CopyEngines& c = cache[dev];
  if (!c.ready) {
    if (cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking) != cudaSuccess)
      return FP8Q_ERR_CUDA;
    for (int s = 0; s < 2; ++s)
      if (cudaEventCreateWithFlags(&c.in_done[s], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&c.compute_done[s], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&c.out_done[s], cudaEventDisableTiming) != cudaSuccess)
        return FP8Q_ERR_CUDA;
    c.ready = true;
  }
  *out = &c;
  return FP8Q_OK;
}

// The tensors a step exchanges with the host: n_in inputs, then n_out outputs, each with its
// size and its device buffer in set 0 and set 1.
constexpr int kMaxIo = 20;
struct IoList {
  int n_in = 0, n_out = 0;
  size_t bytes[kMaxIo] = {};
  const void* dev[2][kMaxIo] = {};
  void add(const void* d0, const void* d1, size_t n) {
    dev[0][n_in + n_out] = d0;
    dev[1][n_in + n_out] = d1;
    bytes[n_in + n_out] = n;
  }
  void in(const void* d0, const void* d1, size_t n) { add(d0, d1, n), ++n_in; }
  void out(const void* d0, const void* d1, size_t n) { add(d0, d1, n), ++n_out; }
};

// A device buffer both sets share must never move: host(i, k), step i's host pointer of tensor k,
// is null in every step for such a buffer (and a tensor that moves needs both device buffers).
template <class Host>
int check_io(const IoList& io, int n_steps, Host host) {
  for (int k = 0; k < io.n_in + io.n_out; ++k) {
    bool moved = false;
    for (int i = 0; i < n_steps; ++i) moved = moved || host(i, k) != nullptr;
    if (moved && (!io.dev[0][k] || !io.dev[1][k] || io.dev[0][k] == io.dev[1][k])) return FP8Q_ERR_INVALID_ARG;
  }
  return FP8Q_OK;
}

// Step i runs on set i % 2: its inputs are copied in on the h2d stream once step i - 2 (the set's
// last user) has computed, compute(set) runs on the caller's stream once they are in and step
// i - 2's outputs have left, and the outputs go out on the d2h stream.  host(i, k) is step i's
// host pointer of tensor k (null: the tensor stays on the device).  check_io has passed.
template <class Host, class Compute>
int run_pipelined(const IoList& io, int n_steps, Host host, Compute compute, const Ctx& c) {
  const int n = io.n_in + io.n_out;
  CopyEngines* ce = nullptr;
  int e;
  if ((e = copy_engines(&ce))) return e;
  cudaStream_t cs = c.L.stream;
#define FP8Q_CUDA(expr)                              \
  do {                                               \
    if ((expr) != cudaSuccess) return FP8Q_ERR_CUDA; \
  } while (0)
  for (int i = 0; i < n_steps; ++i) {
    const int s = i & 1;
    if (i >= 2) FP8Q_CUDA(cudaStreamWaitEvent(ce->h2d, ce->compute_done[s], 0));
    for (int k = 0; k < io.n_in; ++k)
      if (const void* h = host(i, k))
        FP8Q_CUDA(cudaMemcpyAsync(const_cast<void*>(io.dev[s][k]), h, io.bytes[k], cudaMemcpyHostToDevice, ce->h2d));
    FP8Q_CUDA(cudaEventRecord(ce->in_done[s], ce->h2d));
    FP8Q_CUDA(cudaStreamWaitEvent(cs, ce->in_done[s], 0));
    if (i >= 2) FP8Q_CUDA(cudaStreamWaitEvent(cs, ce->out_done[s], 0));
    if ((e = compute(s))) return e;
    FP8Q_CUDA(cudaEventRecord(ce->compute_done[s], cs));
    FP8Q_CUDA(cudaStreamWaitEvent(ce->d2h, ce->compute_done[s], 0));
    for (int k = io.n_in; k < n; ++k)
      if (const void* h = host(i, k))
        FP8Q_CUDA(cudaMemcpyAsync(const_cast<void*>(h), io.dev[s][k], io.bytes[k], cudaMemcpyDeviceToHost, ce->d2h));
    FP8Q_CUDA(cudaEventRecord(ce->out_done[s], ce->d2h));
  }
  // the caller's stream ends after the last outputs (and every earlier copy) have landed
  FP8Q_CUDA(cudaStreamWaitEvent(cs, ce->out_done[(n_steps - 1) & 1], 0));
  if (n_steps >= 2) FP8Q_CUDA(cudaStreamWaitEvent(cs, ce->out_done[n_steps & 1], 0));
#undef FP8Q_CUDA
  return FP8Q_OK;
}

bool same_shape(const fp8q_mlp* a, const fp8q_mlp* b) {
  return a->T == b->T && a->d == b->d && a->f == b->f && a->recompute == b->recompute &&
         a->grad_e4m3 == b->grad_e4m3 && a->bf16 == b->bf16;
}

bool same_shape(const fp8q_block* a, const fp8q_block* b) {
  return a->T == b->T && a->d == b->d && a->f == b->f && a->n_qkv == b->n_qkv && a->n_heads == b->n_heads &&
         a->n_kv_heads == b->n_kv_heads && a->seq_len == b->seq_len && same_shape(&a->mlp, &b->mlp);
}

// The MLP block's host tensors in fp8q_mlp_host_io order: x, g, W_gu, W_d, dY in; y, dX, dW_gu,
// dW_d, dg out.
IoList mlp_io(const fp8q_mlp* m0, const fp8q_mlp* m1) {
  const size_t T = (size_t)m0->T, d = (size_t)m0->d, f = (size_t)m0->f;
  IoList io;
  io.in(m0->x, m1->x, T * d * 2);
  io.in(m0->g, m1->g, d * 2);
  io.in(m0->W_gu, m1->W_gu, d * 2 * f * 2);
  io.in(m0->W_d, m1->W_d, f * d * 2);
  io.in(m0->dY, m1->dY, T * d * 2);
  io.out(m0->y, m1->y, T * d * 2);
  io.out(m0->dX, m1->dX, T * d * 2);
  io.out(m0->dW_gu, m1->dW_gu, d * 2 * f * 4);
  io.out(m0->dW_d, m1->dW_d, f * d * 4);
  io.out(m0->dg, m1->dg, d * 4);
  return io;
}

const void* mlp_host(const fp8q_mlp_host_io& h, int k) {
  const void* p[10] = {h.x, h.g, h.W_gu, h.W_d, h.dY, h.y, h.dX, h.dW_gu, h.dW_d, h.dg};
  return p[k];
}

int mlp_run_steps(const fp8q_mlp* dev0, const fp8q_mlp* dev1, const fp8q_mlp_host_io* host, int n_steps,
                  bool backward, void* ws, size_t ws_bytes, fp8q_stream stream) {
  const fp8q_mlp* dev[2] = {dev0, dev1};
  int e;
  if (!dev0 || !dev1 || !host || n_steps < 1) return FP8Q_ERR_INVALID_ARG;
  for (const fp8q_mlp* m : dev)
    if ((e = validate_mlp(m, backward))) return e;
  if (!same_shape(dev0, dev1)) return FP8Q_ERR_INVALID_ARG;
  if (!backward)
    for (int i = 0; i < n_steps; ++i)
      for (int k : {4, 6, 7, 8, 9})  // dY, dX, dW_gu, dW_d, dg
        if (mlp_host(host[i], k)) return FP8Q_ERR_INVALID_ARG;
  if ((e = check_ws(ws, ws_bytes, mlp_block_workspace_size(dev0->T, dev0->d, dev0->f, backward ? 1 : 0)))) return e;
  const IoList io = mlp_io(dev0, dev1);
  auto host_at = [&](int i, int k) { return mlp_host(host[i], k); };
  if ((e = check_io(io, n_steps, host_at))) return e;
  Ctx c;
  if ((e = make_ctx(&c, stream))) return e;
  MlpWs w;
  mlp_ws_layout(dev0->T, dev0->d, dev0->f, backward ? 1 : 0, static_cast<uint8_t*>(ws), &w);
  if ((e = run_pipelined(
           io, n_steps, host_at,
           [&](int s) {
             int r = mlp_fwd_run(dev[s], w, c);
             return r || !backward ? r : mlp_bwd_run(dev[s], w, c);
           },
           c)))
    return e;
  return finish(c);
}

// The full block's host tensors in fp8q_block_host_io order.
IoList block_io(const fp8q_block* b0, const fp8q_block* b1) {
  const size_t T = (size_t)b0->T, d = (size_t)b0->d, f = (size_t)b0->f, nq = (size_t)b0->n_qkv;
  IoList io;
  io.in(b0->x, b1->x, T * d * 2);
  io.in(b0->g1, b1->g1, d * 2);
  io.in(b0->W_qkv, b1->W_qkv, d * nq * 2);
  io.in(b0->W_o, b1->W_o, d * d * 2);
  io.in(b0->att, b1->att, T * d * 2);
  io.in(b0->mlp.g, b1->mlp.g, d * 2);
  io.in(b0->mlp.W_gu, b1->mlp.W_gu, d * 2 * f * 2);
  io.in(b0->mlp.W_d, b1->mlp.W_d, f * d * 2);
  io.in(b0->mlp.dY, b1->mlp.dY, T * d * 2);
  io.in(b0->dQKV, b1->dQKV, T * nq * 2);
  io.out(b0->mlp.y, b1->mlp.y, T * d * 2);
  io.out(b0->dX, b1->dX, T * d * 2);
  io.out(b0->d_att, b1->d_att, T * d * 2);
  io.out(b0->dW_qkv, b1->dW_qkv, d * nq * 4);
  io.out(b0->dW_o, b1->dW_o, d * d * 4);
  io.out(b0->dg1, b1->dg1, d * 4);
  io.out(b0->mlp.dW_gu, b1->mlp.dW_gu, d * 2 * f * 4);
  io.out(b0->mlp.dW_d, b1->mlp.dW_d, f * d * 4);
  io.out(b0->mlp.dg, b1->mlp.dg, d * 4);
  return io;
}

const void* block_host(const fp8q_block_host_io& h, int k) {
  const void* p[19] = {h.x,  h.g1, h.W_qkv, h.W_o,   h.att,  h.g,   h.W_gu,   h.W_d,  h.dY, h.dQKV,
                       h.y,  h.dX, h.d_att, h.dW_qkv, h.dW_o, h.dg1, h.dW_gu, h.dW_d, h.dg};
  return p[k];
}

}  // namespace

extern "C" {

int mlp_block_run_steps(const fp8q_mlp* dev0, const fp8q_mlp* dev1, const fp8q_mlp_host_io* host, int n_steps,
                        void* ws, size_t ws_bytes, fp8q_stream stream) {
  return mlp_run_steps(dev0, dev1, host, n_steps, true, ws, ws_bytes, stream);
}

int mlp_block_fwd_run_steps(const fp8q_mlp* dev0, const fp8q_mlp* dev1, const fp8q_mlp_host_io* host, int n_steps,
                            void* ws, size_t ws_bytes, fp8q_stream stream) {
  return mlp_run_steps(dev0, dev1, host, n_steps, false, ws, ws_bytes, stream);
}

int block_run_steps(const fp8q_block* dev0, const fp8q_block* dev1, const fp8q_block_host_io* host, int n_steps,
                    int backward, void* ws, size_t ws_bytes, fp8q_stream stream) {
  const fp8q_block* dev[2] = {dev0, dev1};
  int e;
  if (!dev0 || !dev1 || !host || n_steps < 1) return FP8Q_ERR_INVALID_ARG;
  for (const fp8q_block* b : dev)
    if ((e = validate_block(b, backward != 0))) return e;
  if (!same_shape(dev0, dev1)) return FP8Q_ERR_INVALID_ARG;
  for (int i = 0; i < n_steps; ++i) {
    // with the attention core inside, att and dQKV are the block's own results, not inputs
    if (dev0->n_heads && (host[i].att || host[i].dQKV)) return FP8Q_ERR_INVALID_ARG;
    if (!backward)
      for (int k : {8, 9, 11, 12, 13, 14, 15, 16, 17, 18})  // the backward's inputs and outputs
        if (block_host(host[i], k)) return FP8Q_ERR_INVALID_ARG;
  }
  const int bw = backward ? 1 : 0;
  if ((e = check_ws(ws, ws_bytes, block_workspace_size(dev0->T, dev0->d, dev0->f, dev0->n_qkv, bw)))) return e;
  const IoList io = block_io(dev0, dev1);
  auto host_at = [&](int i, int k) { return block_host(host[i], k); };
  if ((e = check_io(io, n_steps, host_at))) return e;
  Ctx c;
  if ((e = make_ctx(&c, stream))) return e;
  BlockWs w;
  block_ws_layout(dev0->T, dev0->d, dev0->f, dev0->n_qkv, bw, static_cast<uint8_t*>(ws), &w);
  if ((e = run_pipelined(
           io, n_steps, host_at,
           [&](int s) {
             int r = block_fwd_run(dev[s], w, c);
             return r || !backward ? r : block_bwd_run(dev[s], w, c);
           },
           c)))
    return e;
  return finish(c);
}

// ---------------------------------------------------------------------------
// The attention core
// ---------------------------------------------------------------------------
int attention_fwd(const void* qkv, int64_t T, int64_t seq_len, int n_heads, int n_kv_heads, int head_dim,
                  void* att, float* lse, fp8q_stream stream) {
  int e = validate_attention(qkv, T, seq_len, n_heads, n_kv_heads, head_dim);
  if (e) return e;
  if (!al16(att) || !al16(lse)) return FP8Q_ERR_INVALID_ARG;
  Ctx c;
  if ((e = make_ctx(&c, stream))) return e;
  FP8Q_STEP(kKAttnFwd, launch_attn_fwd(static_cast<const uint16_t*>(qkv), T, (int)seq_len, n_heads, n_kv_heads,
                                       static_cast<uint16_t*>(att), lse, c.L));
  return finish(c);
}

size_t attention_bwd_workspace_size(int64_t T, int n_heads) {
  if (T < 1 || n_heads < 1) return 0;
  return 2 * round256((size_t)T * (size_t)n_heads * 4);
}

int attention_bwd(const void* qkv, const void* att, const float* lse, const void* d_att, int64_t T, int64_t seq_len,
                  int n_heads, int n_kv_heads, int head_dim, void* dqkv, void* ws, size_t ws_bytes,
                  fp8q_stream stream) {
  int e = validate_attention(qkv, T, seq_len, n_heads, n_kv_heads, head_dim);
  if (e) return e;
  if (!al16(att) || !al16(lse) || !al16(d_att) || !al16(dqkv)) return FP8Q_ERR_INVALID_ARG;
  if ((e = check_ws(ws, ws_bytes, attention_bwd_workspace_size(T, n_heads)))) return e;
  Ctx c;
  if ((e = make_ctx(&c, stream))) return e;
  float* delta = static_cast<float*>(ws);
  float* lse2 = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + round256((size_t)T * (size_t)n_heads * 4));
  const uint16_t* q16 = static_cast<const uint16_t*>(qkv);
  const uint16_t* do16 = static_cast<const uint16_t*>(d_att);
  uint16_t* dq16 = static_cast<uint16_t*>(dqkv);
  const int S = (int)seq_len;
  FP8Q_STEP(kKAttnBwdDelta, launch_attn_bwd_delta(static_cast<const uint16_t*>(att), do16, lse, T, n_heads, delta,
                                                  lse2, c.L));
  FP8Q_STEP(kKAttnBwdDkdv, launch_attn_bwd_dkdv(q16, do16, T, S, n_heads, n_kv_heads, delta, lse2, dq16, c.L));
  FP8Q_STEP(kKAttnBwdDq, launch_attn_bwd_dq(q16, do16, T, S, n_heads, n_kv_heads, delta, lse2, dq16, c.L));
  return finish(c);
}

// ---------------------------------------------------------------------------
int fp8q_get_status(int clear) {
  DevInfo d;
  if (device_info(&d)) return -1;
  unsigned v = 0;
  if (cudaMemcpy(&v, d.status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  if (clear) {
    const unsigned z = 0;
    if (cudaMemcpy(d.status, &z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return -1;
  }
  return (int)v;
}

const char* fp8q_status_string(int status) {
  switch (status) {
    case FP8Q_OK: return "ok";
    case FP8Q_ERR_INVALID_ARG: return "invalid argument";
    case FP8Q_ERR_UNSUPPORTED: return "unsupported";
    case FP8Q_ERR_CUDA: return "CUDA error";
    case FP8Q_ERR_TIMEOUT: return "device wait timed out";
    case FP8Q_ERR_NONFINITE: return "non-finite absmax";
    case FP8Q_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

int fp8q_last_launch_count(void) { return t_last_launches; }

int fp8q_selftest_bounded_wait(int64_t limit_ns, fp8q_stream stream) {
  if (limit_ns < 1000000 || limit_ns > 10000000000LL) return FP8Q_ERR_INVALID_ARG;
  Ctx c;
  int e = make_ctx(&c, stream);
  if (e) return e;
  if (launch_selftest_bounded_wait((uint64_t)limit_ns, c.L) != cudaSuccess) return FP8Q_ERR_CUDA;
  return finish(c);
}

int fp8q_trace_start(int capacity) {
  Trace& t = t_trace;
  if (capacity < 1) return FP8Q_ERR_INVALID_ARG;
  for (cudaEvent_t e : t.ev) cudaEventDestroy(e);
  t.ev.assign(2 * (size_t)capacity, nullptr);
  for (auto& e : t.ev)
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      t.on = false;
      return FP8Q_ERR_CUDA;
    }
  t.kinds.assign((size_t)capacity, -1);
  t.n = 0;
  t.on = true;
  return FP8Q_OK;
}

int fp8q_trace_stop(void) {
  t_trace.on = false;
  return FP8Q_OK;
}

int fp8q_trace_resume(void) {
  if (t_trace.ev.empty()) return FP8Q_ERR_INVALID_ARG;
  t_trace.on = true;
  return FP8Q_OK;
}

int fp8q_trace_read(float* ms, int* kinds, int capacity) {
  Trace& t = t_trace;
  const int n = t.n < capacity ? t.n : capacity;
  for (int i = 0; i < n; ++i) {
    if (cudaEventSynchronize(t.ev[2 * i + 1]) != cudaSuccess) return -1;
    float v = 0.0f;
    if (cudaEventElapsedTime(&v, t.ev[2 * i], t.ev[2 * i + 1]) != cudaSuccess) return -1;
    ms[i] = v;
    kinds[i] = t.kinds[i];
  }
  return n;
}

const char* fp8q_kernel_name(int kind) { return kind >= 0 && kind < kKCount ? kKindNames[kind] : "unknown"; }

}  // extern "C"
