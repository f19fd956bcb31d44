// The attention core between the QKV and O projections of the transformer
// block (LLMQ §2/§3 name the block's attention and its custom kernels; the
// pages fix no attention arithmetic): causal softmax attention with grouped
// K/V heads, bf16 in and out, on the 5th-generation tensor cores
// (tcgen05.mma kind::f16, bf16 operands, fp32 accumulation in TMEM).
//
// qkv row of token t = [q_0 .. q_{Hq-1} | k_0 .. k_{Hkv-1} | v_0 .. v_{Hkv-1}],
// 128 elements per head; the T tokens form T / S sequences of S consecutive
// tokens; query head h reads K/V head h / (Hq / Hkv); scale 1 / sqrt(128).
//
// Forward, one CTA per (128-query tile, query head, sequence), 256 threads:
//   warp 0      TMA producer: the Q tile once, K and V tiles of 128 keys into a
//               2-stage ring (128 x 128 bf16 tiles as two 64-element-wide
//               128-byte-swizzled boxes);
//   warp 1      MMA issuer: S_j = Q K_j^T into one of two TMEM buffers, then
//               O_j = P_j V_j into a third (V is the MN-major operand);
//   warp 2      TMEM allocation (512 columns);
//   warps 4..7  softmax, one thread per query row (TMEM lane): row max of S_j
//               (scores pre-multiplied by log2(e)/sqrt(128)), p = 2^(s - m),
//               P_j as bf16 into a swizzled shared tile for the second MMA,
//               the running sum, and O in registers, O = O 2^(m_old - m) + O_j;
//               at the end O / l goes out through the Q tile with TMA stores
//               and lse = ln 2 (m + log2 l).
// Every mbarrier wait is bounded; on expiry the CTA records FP8Q_STATUS_TIMEOUT,
// stops issuing work, drains what it issued, frees TMEM and exits.
#include "fp8q_common.cuh"
#include "fp8q_internal.h"

#include <mutex>

namespace fp8q {

namespace {

constexpr int kDh = 128;                 // head dimension
constexpr int kAtom = 16384;             // 128 rows x 128 bytes: one 64-element-wide swizzle atom column
constexpr int kTile = 2 * kAtom;         // a 128 x 128 bf16 operand tile
constexpr int kAttnThreads = 256;
constexpr int kTmemCols = 512;

// forward shared-memory layout (bytes from the 1024-aligned base)
constexpr int kFQ = 0;
constexpr int kFK = kFQ + kTile;         // [2] stages
constexpr int kFV = kFK + 2 * kTile;     // [2] stages
constexpr int kFP = kFV + 2 * kTile;
constexpr int kFBar = kFP + kTile;
constexpr int kFwdSmem = kFBar + 256 + 1024;
static_assert(kFwdSmem <= 232448, "shared memory per CTA");

struct AttnArgs {
  int T, S, Hq, Hkv;
  int n_qt;            // query tiles per sequence
  float scale_log2;    // log2(e) / sqrt(128)
  float* lse;          // [Hq, T]
  unsigned* status;
};

// Instruction descriptor: kind::f16 with bf16 A and B, fp32 accumulator, M = N = 128,
// A K-major, B K-major (b_mn = 0) or MN-major (1).
__host__ __device__ constexpr uint32_t idesc_bf16_128(int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
}

// D (+)= A B^T over K = 128 with A and B both K-major 128 x 128 tiles.
__device__ __forceinline__ void mma_tile_kk(uint32_t d, uint32_t a, uint32_t b, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = (uint32_t)((kk >> 2) * kAtom + (kk & 3) * 32);
    umma_bf16(d, smem_desc_sw128(a + off, 16, 1024), smem_desc_sw128(b + off, 16, 1024), idesc_bf16_128(0),
              (accumulate || kk) ? 1u : 0u);
  }
}
// D (+)= A B over K = 128 with A K-major and B MN-major (rows = K, two 64-wide N atoms).
__device__ __forceinline__ void mma_tile_kmn(uint32_t d, uint32_t a, uint32_t b, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t aoff = (uint32_t)((kk >> 2) * kAtom + (kk & 3) * 32);
    umma_bf16(d, smem_desc_sw128(a + aoff, 16, 1024), smem_desc_sw128(b + kk * 2048, kAtom, 1024),
              idesc_bf16_128(1), (accumulate || kk) ? 1u : 0u);
  }
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
// 32 bf16 values (16 packed words) of row r, columns 32c .. 32c+31, into a K-major
// 128 x 128 swizzled tile (16-byte chunk j of a 128-byte row sits at j ^ (r % 8)).
__device__ __forceinline__ void tile_put32(uint32_t tile, int r, int c, const uint32_t (&w)[16]) {
  const uint32_t row = tile + (uint32_t)((c >> 1) * kAtom + r * 128);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int chunk = (c & 1) * 4 + q;
    st_shared_v4(row + (uint32_t)((chunk ^ (r & 7)) << 4),
                 make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
  }
}
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tm), "r"(src),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_and_wait() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Forward
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kAttnThreads, 1)
    k_attn_fwd(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmAtt,
               const AttnArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kFBar);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;    // [2]
  uint64_t* kv_empty = bars + 3;   // [2]
  uint64_t* s_full = bars + 5;     // [2]
  uint64_t* s_free = bars + 7;     // [2]
  uint64_t* p_full = bars + 9;
  uint64_t* p_free = bars + 10;
  uint64_t* o_full = bars + 11;
  uint64_t* o_free = bars + 12;
  uint64_t* drain = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int qt = p.n_qt - 1 - (int)blockIdx.x;  // the longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (p.Hq / p.Hkv);
  const int t0 = b * p.S + qt * 128;
  const int n = qt + 1;  // key tiles 0 .. qt (causal)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(p_free, 1);
    mbar_init(o_full, 1);
    mbar_init(o_free, 128);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQKV);
    tma_prefetch_desc(&tmAtt);
  }
  if (warp == 2) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_addr(smem);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      bool ok = true;
      uint32_t issued = 0, issued_par = 0;  // kv stages with a load in flight, and its phase parity
      mbar_arrive_expect_tx(q_full, kTile);
      tma_load_2d(smem + kFQ, &tmQKV, q_full, h * kDh, t0);
      tma_load_2d(smem + kFQ + kAtom, &tmQKV, q_full, h * kDh + 64, t0);
      const int xk = (p.Hq + g) * kDh, xv = (p.Hq + p.Hkv + g) * kDh;
      for (int j = 0; j < n; ++j) {
        const int st = j & 1;
        const uint32_t u = (uint32_t)(j >> 1) & 1u;
        if (!mbar_wait(&kv_empty[st], u ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sk = smem + kFK + st * kTile;
        uint8_t* sv = smem + kFV + st * kTile;
        const int y = b * p.S + j * 128;
        mbar_arrive_expect_tx(&kv_full[st], 2 * kTile);
        tma_load_2d(sk, &tmQKV, &kv_full[st], xk, y);
        tma_load_2d(sk + kAtom, &tmQKV, &kv_full[st], xk + 64, y);
        tma_load_2d(sv, &tmQKV, &kv_full[st], xv, y);
        tma_load_2d(sv + kAtom, &tmQKV, &kv_full[st], xv + 64, y);
        issued |= 1u << st;
        issued_par = (issued_par & ~(1u << st)) | (u << st);
      }
      if (!ok) {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
        int dummy = 0;
        mbar_wait(q_full, 0, &dummy);
        for (int s = 0; s < 2; ++s)
          if (issued & (1u << s)) mbar_wait(&kv_full[s], (issued_par >> s) & 1u, &dummy);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t tS = tmem, tO = tmem + 256;
      bool ok = mbar_wait(q_full, 0, abort_flag);
      for (int j = 0; j <= n && ok; ++j) {
        if (j < n) {
          const int st = j & 1;
          const uint32_t u = (uint32_t)(j >> 1) & 1u;
          if (!mbar_wait(&kv_full[st], u, abort_flag) || !mbar_wait(&s_free[st], u ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tile_kk(tS + st * 128, sbase + kFQ, sbase + kFK + st * kTile, false);
          umma_commit(&s_full[st]);
        }
        if (j >= 1) {
          const int i = j - 1, st = i & 1;
          const uint32_t par = (uint32_t)i & 1u;
          if (!mbar_wait(p_full, par, abort_flag) || !mbar_wait(o_free, par ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tile_kmn(tO, sbase + kFP, sbase + kFV + st * kTile, false);
          umma_commit(o_full);
          umma_commit(p_free);
          umma_commit(&kv_empty[st]);
        }
      }
      if (!ok) {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      umma_commit(drain);
      int dummy = 0;
      mbar_wait(drain, 0, &dummy);
    }
  } else if (warp >= 4) {
    // ---------------- softmax + O ----------------
    const int r = threadIdx.x - 128;  // query row of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off, tO = tmem + 256 + lane_off;
    float o[kDh];
#pragma unroll
    for (int c = 0; c < kDh; ++c) o[c] = 0.0f;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int st = j & 1;
      const uint32_t u = (uint32_t)(j >> 1) & 1u;
      const bool diag = j == qt;
      if (!mbar_wait(&s_full[st], u, abort_flag)) { ok = false; break; }
      tc_fence_after();
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t sv[32];
        tmem_ld32(tS + st * 128 + c * 32, sv);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float s = __uint_as_float(sv[k]) * p.scale_log2;
          if (!(diag && c * 32 + k > r)) mx = fmaxf(mx, s);
        }
      }
      const float m_new = fmaxf(m, mx);
      const float alpha = ex2_approx(m - m_new);
      if (!mbar_wait(p_free, ((uint32_t)j & 1u) ^ 1u, abort_flag)) { ok = false; break; }
      float rs = 0.0f;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t sv[32], w[16];
        tmem_ld32(tS + st * 128 + c * 32, sv);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int c0 = c * 32 + 2 * k;
          const float p0 = (diag && c0 > r) ? 0.0f : ex2_approx(__uint_as_float(sv[2 * k]) * p.scale_log2 - m_new);
          const float p1 =
              (diag && c0 + 1 > r) ? 0.0f : ex2_approx(__uint_as_float(sv[2 * k + 1]) * p.scale_log2 - m_new);
          rs += p0 + p1;
          w[k] = pack_bf16x2(p0, p1);
        }
        tile_put32(sbase + kFP, r, c, w);
      }
      tc_fence_before();
      mbar_arrive(&s_free[st]);
      fence_async_shared();
      mbar_arrive(p_full);
      l = l * alpha + rs;
      m = m_new;
      if (!mbar_wait(o_full, (uint32_t)j & 1u, abort_flag)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t ov[32];
        tmem_ld32(tO + c * 32, ov);
#pragma unroll
        for (int k = 0; k < 32; ++k) o[c * 32 + k] = fmaf(o[c * 32 + k], alpha, __uint_as_float(ov[k]));
      }
      tc_fence_before();
      mbar_arrive(o_free);
    }
    if (!ok) {
      atomicOr(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // O / l goes out through the Q tile: every S MMA (the tile's readers) has completed once
    // the last s_full was seen.  Each of the 128 threads reaches the named barrier once.
    if (ok) {
      const float inv = 1.0f / l;  // l >= 1: the row maximum contributes 2^0
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(o[c * 32 + 2 * k] * inv, o[c * 32 + 2 * k + 1] * inv);
        tile_put32(sbase + kFQ, r, c, w);
      }
      p.lse[(int64_t)h * p.T + t0 + r] = (m + log2f(l)) * 0.693147180559945309f;
    }
    fence_async_shared();
    named_bar_sync(1, 128);
    if (r == 0 && !*abort_flag) {
      tma_store_2d(&tmAtt, sbase + kFQ, h * kDh, t0);
      tma_store_2d(&tmAtt, sbase + kFQ + kAtom, h * kDh + 64, t0);
      bulk_commit_and_wait();
    }
  }
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// bf16 matrix [rows, cols] (row stride ld elements) in 64 x 128 boxes (128-byte rows, 128-byte swizzle).
bool make_tile_map(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t ld) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class K>
cudaError_t set_smem(K kernel, int bytes) {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device == dev) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) configured_device = dev;
  return e;
}

}  // namespace

cudaError_t launch_attn_fwd(const uint16_t* qkv, int64_t T, int S, int Hq, int Hkv, uint16_t* att, float* lse,
                            const Launch& L) {
  const int64_t nq = (int64_t)(Hq + 2 * Hkv) * kDh;
  CUtensorMap tq, ta;
  if (!make_tile_map(&tq, qkv, nq, T, nq) || !make_tile_map(&ta, att, (int64_t)Hq * kDh, T, (int64_t)Hq * kDh))
    return cudaErrorInvalidValue;
  AttnArgs a{};
  a.T = (int)T;
  a.S = S;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.n_qt = S / 128;
  a.scale_log2 = 1.44269504088896341f / 11.3137084989847604f;  // log2(e) / sqrt(128)
  a.lse = lse;
  a.status = L.status;
  cudaError_t e = set_smem(k_attn_fwd, kFwdSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)a.n_qt, (unsigned)Hq, (unsigned)(T / S));
  k_attn_fwd<<<grid, kAttnThreads, kFwdSmem, L.stream>>>(tq, ta, a);
  if (L.launches) ++*L.launches;
  return cudaGetLastError();
}

}  // namespace fp8q
