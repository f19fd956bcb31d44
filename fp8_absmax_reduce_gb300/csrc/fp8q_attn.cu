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
//   warp 1      MMA issuer: S_j = Q K_j^T into one of two TMEM buffers, and one
//               step behind O += P_{j-1} V_{j-1} into a third (V MN-major);
//   warp 2      TMEM allocation (512 columns);
//   warps 4..7  softmax, one thread per query row (TMEM lane): S_j read once into
//               registers (scores times log2(e)/sqrt(128)), p = 2^(s - m_ref) as bf16
//               into one of two swizzled shared P tiles, the running sum l; the
//               reference max m_ref moves (and O in TMEM is rescaled) only when a
//               tile's max exceeds it by more than 8, so most steps touch only S;
//               at the end O / l goes out through the Q tile with TMA stores and
//               lse = ln 2 (m_ref + log2 l).
// Backward (dO = d_att), three kernels:
//   k_attn_bwd_delta  D = rowsum(dO * O) over the stored att, and lse in the
//                     log2 domain, per (token, head);
//   k_attn_bwd_dkdv   one CTA per (128-key tile, K/V head, sequence): with its K
//                     and V tiles in shared memory it walks the group's query
//                     heads and the query tiles at or after it; S^T = K Q^T and
//                     dP^T = V dO^T into TMEM, one thread per key row forms
//                     P^T = 2^(s - lse) and dS^T = P^T (dP^T - D) as bf16 operand
//                     tiles, and dV += P^T dO, dK += dS^T Q accumulate in TMEM
//                     (the group's sum stays inside the CTA: deterministic);
//   k_attn_bwd_dq     one CTA per (128-query tile, query head, sequence): S and
//                     dP, then dS, then dQ += dS K over the key tiles 0 .. i, with dS
//                     double-buffered in TMEM as the MMA's A operand.
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
// The backward kernels run two element-wise warpgroups (warps 4-7 and 8-11) that split every
// tile's columns: their passes need no row reductions, and two warps per SM sub-partition hide
// each other's latencies.
constexpr int kAttnBwdThreads = 384;
constexpr int kTmemCols = 512;

// forward shared-memory layout (bytes from the 1024-aligned base)
constexpr int kFQ = 0;
constexpr int kFK = kFQ + kTile;         // [2] stages
constexpr int kFV = kFK + 2 * kTile;     // [2] stages
constexpr int kFP = kFV + 2 * kTile;     // [2] P buffers
constexpr int kFBar = kFP + 2 * kTile;
constexpr int kFwdSmem = kFBar + 256 + 1024;  // 19 barriers, the TMEM slot and the abort flag fit in 256 B
static_assert(kFwdSmem <= 232448, "shared memory per CTA");

struct AttnArgs {
  int T, S, Hq, Hkv;
  int n_qt;            // query tiles per sequence
  float scale_log2;    // log2(e) / sqrt(128)
  float* lse;          // [Hq, T]
  unsigned* status;
};

// CTA order.  A CTA's work depends on its tile's place on the causal diagonal, so a grid walked
// tile by tile inside each (head, sequence) pair leaves the longest CTAs of the last pairs to run
// alone at the end (in a greedy schedule of 32 tiles per pair on 152 SMs: 17 % over the ideal for
// dK/dV, 3 % for dQ, 7 % for the paired forward).  The grids are one-dimensional instead and hand
// the tiles out in bands of BAND, the longest band first, every (head, sequence) pair of a band
// before the next band, each pair's tiles of the band together: the longest CTAs start first and
// the last ones dispatched are short, while the CTAs of a band that share a pair run at the same
// time and share its re-read tiles in L2.  Wider bands keep more of that sharing, narrower ones
// balance better.  rank 0 is the longest tile of a pair; the last band may be narrower.
template <int BAND>
__device__ __forceinline__ void cta_order(int n_tiles, int heads, int n_seq, int& rank, int& h, int& b) {
  const int pairs = heads * n_seq;
  const int band = (int)blockIdx.x / (BAND * pairs);
  const int k0 = band * BAND;
  const int width = min(BAND, n_tiles - k0);
  const int rem = (int)blockIdx.x - band * BAND * pairs;
  const int pair = rem / width;
  rank = k0 + rem % width;
  h = pair % heads;
  b = pair / heads;
}
// Band widths, measured on 32 tiles per pair (32B block: 40 query / 8 K/V heads, 4 sequences of
// 4096), as each kernel's time over the forward's in the same step (the clocks move with the power
// cap): the forward re-reads only K and V (67 MB in all, L2-resident whatever the order) and takes
// bands of one tile (~1 % faster than pairs walked in order); dK/dV, which re-reads the group's Q
// and dO (335 MB), 2.49 with one band of all -> 2.18 with bands of 2 (2.19 with 4, 2.24 with 8);
// dQ, which re-reads K and V, 1.65 with one band of all, 1.72 / 1.67 / 1.64 with bands of 4 / 8 / 16.
constexpr int kFwdBand = 1, kDkdvBand = 2, kDqBand = 16;

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

// A wait in the warps that use warp-collective tcgen05.ld/st: every lane waits, and the whole
// warp goes on only if every lane's wait succeeded (so a time-out leaves the warp together).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort)) != 0;
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
// 32 consecutive fp32 columns of this thread's TMEM lane from registers, then the wait.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// A row's reference maximum (log2 domain) moves only when a tile's maximum exceeds it by more
// than this: the probabilities 2^(s - m_ref) then stay below 2^8 (exact in fp32, in bf16's range)
// and O, accumulated by the tensor core in TMEM, is rescaled only on those rare steps.
constexpr float kRescaleSlack = 8.0f;

// S row of this thread (128 raw scores) into registers and the maximum of the scaled scores
// (times log2(e)/sqrt(128); the scale is positive, so it is applied once to the raw maximum).
// MASK (the diagonal tile): keys after the query row r become -inf.  Eight partial maxima keep
// the reduction's dependency chain short.
template <bool MASK>
__device__ __forceinline__ float load_scores(uint32_t tS, int r, float scale_log2, float (&sv)[128]) {
  float mp[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mp[i] = -INFINITY;
#pragma unroll
  for (int c2 = 0; c2 < 4; c2 += 2) {
    uint32_t w[2][32];
    tmem_ld32x2(tS + c2 * 32, tS + c2 * 32 + 32, w[0], w[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int col = (c2 + h) * 32 + k;
        const float x = (MASK && col > r) ? -INFINITY : __uint_as_float(w[h][k]);
        sv[col] = x;
        mp[k & 7] = fmaxf(mp[k & 7], x);
      }
  }
  const float m = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])), fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
  return m * scale_log2;
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    k_attn_fwd(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmAtt,
               const AttnArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kFBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;     // [2]
  uint64_t* k_empty = bars + 3;    // [2] K_j is free once S_j is computed
  uint64_t* s_full = bars + 5;     // [2]
  uint64_t* s_free = bars + 7;     // [2]
  uint64_t* p_full = bars + 9;     // [2]
  uint64_t* p_free = bars + 11;    // [2]
  uint64_t* o_full = bars + 13;    // one phase per P V product
  uint64_t* drain = bars + 14;
  uint64_t* v_full = bars + 15;    // [2]
  uint64_t* v_empty = bars + 17;   // [2] V_j is free once P_j V_j is computed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 19);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  int rank, h, b;
  cta_order<kFwdBand>(p.n_qt, p.Hq, p.T / p.S, rank, h, b);
  const int qt = p.n_qt - 1 - rank;
  const int g = h / (p.Hq / p.Hkv);
  const int t0 = b * p.S + qt * 128;
  const int n = qt + 1;  // key tiles 0 .. qt (causal)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 128);
      mbar_init(&p_full[s], 128);
      mbar_init(&p_free[s], 1);
    }
    mbar_init(o_full, 1);
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
      // K and V stages with a load in flight, and its phase parity (bits 0-1: K, 2-3: V)
      uint32_t issued = 0, issued_par = 0;
      mbar_arrive_expect_tx(q_full, kTile);
      tma_load_2d(smem + kFQ, &tmQKV, q_full, h * kDh, t0);
      tma_load_2d(smem + kFQ + kAtom, &tmQKV, q_full, h * kDh + 64, t0);
      const int xk = (p.Hq + g) * kDh, xv = (p.Hq + p.Hkv + g) * kDh;
      for (int j = 0; j < n; ++j) {
        const int st = j & 1;
        const uint32_t u = (uint32_t)(j >> 1) & 1u;
        const int y = b * p.S + j * 128;
        if (!mbar_wait(&k_empty[st], u ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sk = smem + kFK + st * kTile;
        mbar_arrive_expect_tx(&k_full[st], kTile);
        tma_load_2d(sk, &tmQKV, &k_full[st], xk, y);
        tma_load_2d(sk + kAtom, &tmQKV, &k_full[st], xk + 64, y);
        issued |= 1u << st;
        issued_par = (issued_par & ~(1u << st)) | (u << st);
        if (!mbar_wait(&v_empty[st], u ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sv = smem + kFV + st * kTile;
        mbar_arrive_expect_tx(&v_full[st], kTile);
        tma_load_2d(sv, &tmQKV, &v_full[st], xv, y);
        tma_load_2d(sv + kAtom, &tmQKV, &v_full[st], xv + 64, y);
        issued |= 4u << st;
        issued_par = (issued_par & ~(4u << st)) | (u << (st + 2));
      }
      if (!ok) {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
        int dummy = 0;
        mbar_wait(q_full, 0, &dummy);
        for (int s = 0; s < 2; ++s) {
          if (issued & (1u << s)) mbar_wait(&k_full[s], (issued_par >> s) & 1u, &dummy);
          if (issued & (4u << s)) mbar_wait(&v_full[s], (issued_par >> (s + 2)) & 1u, &dummy);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: S_j, then (one step behind) O += P_{j-1} V_{j-1} ----------------
      const uint32_t tS = tmem, tO = tmem + 256;
      bool ok = mbar_wait(q_full, 0, abort_flag);
      for (int j = 0; j <= n && ok; ++j) {
        if (j < n) {
          const int st = j & 1;
          const uint32_t u = (uint32_t)(j >> 1) & 1u;
          if (!mbar_wait(&k_full[st], u, abort_flag) || !mbar_wait(&s_free[st], u ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tile_kk(tS + st * 128, sbase + kFQ, sbase + kFK + st * kTile, false);
          umma_commit(&s_full[st]);
          umma_commit(&k_empty[st]);
        }
        if (j >= 1) {
          const int i = j - 1, pb = i & 1;
          const uint32_t ui = (uint32_t)(i >> 1) & 1u;
          if (!mbar_wait(&p_full[pb], ui, abort_flag) || !mbar_wait(&v_full[i & 1], ui, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tile_kmn(tO, sbase + kFP + pb * kTile, sbase + kFV + (i & 1) * kTile, i > 0);
          umma_commit(o_full);
          umma_commit(&p_free[pb]);
          umma_commit(&v_empty[i & 1]);
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
    // ---------------- softmax (one query row per thread) ----------------
    const int r = threadIdx.x - 128;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off, tO = tmem + 256 + lane_off;
    float m_ref = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < n && ok; ++j) {
      const int st = j & 1, pb = j & 1;
      const uint32_t u = (uint32_t)(j >> 1) & 1u;
      const bool diag = j == qt;
      if (!warp_wait(&s_full[st], u, abort_flag)) { ok = false; break; }
      tc_fence_after();
      float sv[128];
      const float mx = diag ? load_scores<true>(tS + st * 128, r, p.scale_log2, sv)
                            : load_scores<false>(tS + st * 128, r, p.scale_log2, sv);
      // S_j is in registers: the MMA may overwrite this buffer with S_{j+2}
      tc_fence_before();
      mbar_arrive(&s_free[st]);
      if (__any_sync(0xFFFFFFFFu, mx > m_ref + kRescaleSlack)) {
        const float m_new = fmaxf(m_ref, mx);
        const float alpha = ex2_approx(m_ref - m_new);  // 0 on the first tile, 1 where nothing moves
        if (j > 0) {
          // O holds the products up to j-1: wait for the last one, then rescale this lane's row
          if (!warp_wait(o_full, (uint32_t)(j - 1) & 1u, abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t w[32];
            tmem_ld32(tO + c * 32, w);
#pragma unroll
            for (int k = 0; k < 32; ++k) w[k] = __float_as_uint(__uint_as_float(w[k]) * alpha);
            tmem_st32(tO + c * 32, w);
          }
        }
        l *= alpha;
        m_ref = m_new;
      }
      if (!warp_wait(&p_free[pb], u ^ 1u, abort_flag)) { ok = false; break; }
      float2 rp[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) rp[i] = make_float2(0.0f, 0.0f);
      const float2 sc = make_float2(p.scale_log2, p.scale_log2), nm = make_float2(-m_ref, -m_ref);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          // 2^(s scale - m_ref), two scores per packed fused multiply-add; 2^-inf = 0 for masked keys
          const float2 x = __ffma2_rn(make_float2(sv[c * 32 + 2 * k], sv[c * 32 + 2 * k + 1]), sc, nm);
          const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
          rp[k & 3] = __fadd2_rn(rp[k & 3], make_float2(p0, p1));
          w[k] = pack_bf16x2(p0, p1);
        }
        tile_put32(sbase + kFP + pb * kTile, r, c, w);
      }
      {
        const float2 t = __fadd2_rn(__fadd2_rn(rp[0], rp[1]), __fadd2_rn(rp[2], rp[3]));
        l += t.x + t.y;
      }
      tc_fence_before();
      fence_async_shared();
      mbar_arrive(&p_full[pb]);
    }
    if (ok && !warp_wait(o_full, (uint32_t)(n - 1) & 1u, abort_flag)) ok = false;
    if (!ok) {
      atomicOr(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // O / l goes out through the Q tile: every MMA (the tile's readers) has completed once the
    // last product was seen.  Each of the 128 threads reaches the named barrier once.
    if (ok) {
      tc_fence_after();
      const float inv = 1.0f / l;  // l >= 1: the row's maximum M contributes 2^(M - m_ref) >= 1
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t ov[32], w[16];
        tmem_ld32(tO + c * 32, ov);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          w[k] = pack_bf16x2(__uint_as_float(ov[2 * k]) * inv, __uint_as_float(ov[2 * k + 1]) * inv);
        tile_put32(sbase + kFQ, r, c, w);
      }
      p.lse[(int64_t)h * p.T + t0 + r] = (m_ref + log2f(l)) * 0.693147180559945309f;
    }
    fence_async_shared();
    named_bar_sync(1, 128);
    if (r == 0 && !*abort_flag) {
      tma_store_2d(&tmAtt, sbase + kFQ, h * kDh, t0);
      tma_store_2d(&tmAtt, sbase + kFQ + kAtom, h * kDh + 64, t0);
      bulk_commit_and_wait();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Forward, two query tiles per CTA
// ---------------------------------------------------------------------------
// One CTA per (pair of query tiles 2i, 2i+1, query head, sequence), 384 threads.  The two tiles
// (A = 2i, B = 2i + 1) share every K/V tile (B needs one more, its diagonal), and each has its
// own S and O in TMEM (S_A, S_B, O_A, O_B: all 512 columns) and its own softmax warpgroup
// (warps 4-7 for A, 8-11 for B), so one tile's softmax runs while the tensor core works on the
// other's products:
//   warp 0      lane 0: both Q tiles once, K tiles into a 2-stage ring; lane 1: V tiles into a
//               single stage (each lane waits only on its own ring);
//   warp 1      MMA issuer, per key tile j: S_A(j), O_A += P_A(j-1) V_{j-1}, S_B(j),
//               O_B += P_B(j-1) V_{j-1} (K_j released after both S, V_{j-1} after both P V);
//   warp 2      TMEM allocation;
//   warps 4-11  softmax as in k_attn_fwd (scores in the log2 domain, lazy rescale of O with
//               slack kRescaleSlack), but S is read from TMEM twice -- once for the row maximum,
//               once for the probabilities -- so a thread holds 32-64 scores at a time, not 128.
// Shared memory: Q_A, Q_B, two K stages, one V stage, P_A, P_B (7 x 32 KB).
constexpr int kPQA = 0;
constexpr int kPQB = kPQA + kTile;
constexpr int kPK = kPQB + kTile;        // [2] stages
constexpr int kPV = kPK + 2 * kTile;     // [1] stage
constexpr int kPPA = kPV + kTile;
constexpr int kPPB = kPPA + kTile;
constexpr int kPBar = kPPB + kTile;
constexpr int kPairSmem = kPBar + 256 + 1024;
static_assert(kPairSmem <= 232448, "shared memory per CTA");
constexpr int kPairThreads = 384;

// Maximum of this thread's row of S times log2(e)/sqrt(128); MASK: keys after row r are -inf.
// The scale is positive, so the maximum of the raw scores times the scale is the maximum of the
// scaled scores (rounding is monotonic): one multiply per row, not per score.
template <bool MASK>
__device__ __forceinline__ float row_max(uint32_t tS, int r, float scale_log2) {
  float mp[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mp[i] = -INFINITY;
#pragma unroll
  for (int c2 = 0; c2 < 4; c2 += 2) {
    uint32_t w[2][32];
    tmem_ld32x2(tS + c2 * 32, tS + c2 * 32 + 32, w[0], w[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int col = (c2 + h) * 32 + k;
        const float x = (MASK && col > r) ? -INFINITY : __uint_as_float(w[h][k]);
        mp[k & 7] = fmaxf(mp[k & 7], x);
      }
  }
  const float m = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])), fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
  return m * scale_log2;
}

// p = 2^(s scale - m_ref) of this thread's row of S as bf16 into the K-major P tile (two scores
// per packed fused multiply-add); returns the row sum of the unrounded probabilities.  The thread
// arrives on s_free right after its last TMEM load, so the next S product can start while the
// last chunk's probabilities are formed.
template <bool MASK>
__device__ __forceinline__ float row_probs(uint32_t tS, int r, float scale_log2, float m_ref, uint32_t ptile,
                                           uint64_t* s_free) {
  float2 rp[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) rp[i] = make_float2(0.0f, 0.0f);
  const float2 sc = make_float2(scale_log2, scale_log2), nm = make_float2(-m_ref, -m_ref);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t sw[32], w[16];
    tmem_ld32(tS + c * 32, sw);
    if (c == 3) {
      tc_fence_before();
      mbar_arrive(s_free);
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int col = c * 32 + 2 * k;
      const float2 x = __ffma2_rn(make_float2(__uint_as_float(sw[2 * k]), __uint_as_float(sw[2 * k + 1])), sc, nm);
      const float p0 = (MASK && col > r) ? 0.0f : ex2_approx(x.x);
      const float p1 = (MASK && col + 1 > r) ? 0.0f : ex2_approx(x.y);
      rp[k & 3] = __fadd2_rn(rp[k & 3], make_float2(p0, p1));
      w[k] = pack_bf16x2(p0, p1);
    }
    tile_put32(ptile, r, c, w);
  }
  const float2 t = __fadd2_rn(__fadd2_rn(rp[0], rp[1]), __fadd2_rn(rp[2], rp[3]));
  return t.x + t.y;
}

__global__ void __launch_bounds__(kPairThreads, 1)
    k_attn_fwd_pair(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmAtt,
                    const AttnArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [2]
  uint64_t* k_empty = bars + 3;  // [2] K_j is free once S_A(j), S_B(j) are computed
  uint64_t* v_full = bars + 5;
  uint64_t* v_empty = bars + 6;  // V_j is free once both P V_j products are computed
  uint64_t* s_full = bars + 7;   // [2] per tile (A, B)
  uint64_t* s_free = bars + 9;   // [2] the softmax has read S
  uint64_t* p_full = bars + 11;  // [2] P written
  uint64_t* p_free = bars + 13;  // [2] P V read P (and O holds every product so far)
  uint64_t* o_full = bars + 15;  // [2] one phase per P V product
  uint64_t* drain = bars + 17;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  int rank, h, b;
  cta_order<kFwdBand>(p.n_qt / 2, p.Hq, p.T / p.S, rank, h, b);
  const int pr = p.n_qt / 2 - 1 - rank;
  const int g = h / (p.Hq / p.Hkv);
  const int qa = 2 * pr;
  const int na = qa + 1, nb = qa + 2;  // key tiles of A (0 .. qa) and of B (0 .. qa + 1)
  const int t0a = b * p.S + qa * 128, t0b = t0a + 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s2 = 0; s2 < 2; ++s2) {
      mbar_init(&k_full[s2], 1);
      mbar_init(&k_empty[s2], 1);
      mbar_init(&s_full[s2], 1);
      mbar_init(&s_free[s2], 128);
      mbar_init(&p_full[s2], 128);
      mbar_init(&p_free[s2], 1);
      mbar_init(&o_full[s2], 1);
    }
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
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
  const int xk = (p.Hq + g) * kDh, xv = (p.Hq + p.Hkv + g) * kDh;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- Q tiles, then the K ring ----------------
      bool ok = true;
      uint32_t issued = 0, issued_par = 0;
      mbar_arrive_expect_tx(q_full, 2 * kTile);
      tma_load_2d(smem + kPQA, &tmQKV, q_full, h * kDh, t0a);
      tma_load_2d(smem + kPQA + kAtom, &tmQKV, q_full, h * kDh + 64, t0a);
      tma_load_2d(smem + kPQB, &tmQKV, q_full, h * kDh, t0b);
      tma_load_2d(smem + kPQB + kAtom, &tmQKV, q_full, h * kDh + 64, t0b);
      for (int j = 0; j < nb; ++j) {
        const int st = j & 1;
        const uint32_t u = (uint32_t)(j >> 1) & 1u;
        if (!mbar_wait(&k_empty[st], u ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sk = smem + kPK + st * kTile;
        const int y = b * p.S + j * 128;
        mbar_arrive_expect_tx(&k_full[st], kTile);
        tma_load_2d(sk, &tmQKV, &k_full[st], xk, y);
        tma_load_2d(sk + kAtom, &tmQKV, &k_full[st], xk + 64, y);
        issued |= 1u << st;
        issued_par = (issued_par & ~(1u << st)) | (u << st);
      }
      if (!ok) {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
        int dummy = 0;
        mbar_wait(q_full, 0, &dummy);
        for (int s2 = 0; s2 < 2; ++s2)
          if (issued & (1u << s2)) mbar_wait(&k_full[s2], (issued_par >> s2) & 1u, &dummy);
      }
    } else if (lane == 1) {
      // ---------------- the V stage ----------------
      bool ok = true;
      int last = -1;  // the last V load issued
      for (int j = 0; j < nb; ++j) {
        if (!mbar_wait(v_empty, ((uint32_t)j & 1u) ^ 1u, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(v_full, kTile);
        const int y = b * p.S + j * 128;
        tma_load_2d(smem + kPV, &tmQKV, v_full, xv, y);
        tma_load_2d(smem + kPV + kAtom, &tmQKV, v_full, xv + 64, y);
        last = j;
      }
      if (!ok) {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
        int dummy = 0;
        if (last >= 0) mbar_wait(v_full, (uint32_t)last & 1u, &dummy);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t tSa = tmem, tSb = tmem + 128, tOa = tmem + 256, tOb = tmem + 384;
      bool ok = mbar_wait(q_full, 0, abort_flag);
      // per key tile j: S_A(j), then O_A += P_A(j-1) V_{j-1} (both wait only on tile A's softmax),
      // then S_B(j) and O_B += P_B(j-1) V_{j-1} -- each tile's chain is independent of the other's
      for (int j = 0; j <= nb && ok; ++j) {
        const int st = j & 1, i = j - 1;
        const uint32_t u = (uint32_t)(j >> 1) & 1u, par = (uint32_t)j & 1u, pi = (uint32_t)i & 1u;
        if (j < nb && !mbar_wait(&k_full[st], u, abort_flag)) { ok = false; break; }
        if (j < na) {
          if (!mbar_wait(&s_free[0], par ^ 1u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          mma_tile_kk(tSa, sbase + kPQA, sbase + kPK + st * kTile, false);  // S_A = Q_A K_j^T
          umma_commit(&s_full[0]);
        }
        if (j >= 1 && i < na) {
          if (!mbar_wait(v_full, pi, abort_flag) || !mbar_wait(&p_full[0], pi, abort_flag)) { ok = false; break; }
          tc_fence_after();
          mma_tile_kmn(tOa, sbase + kPPA, sbase + kPV, i > 0);  // O_A += P_A V_i
          umma_commit(&o_full[0]);
          umma_commit(&p_free[0]);
        }
        if (j < nb) {
          if (!mbar_wait(&s_free[1], par ^ 1u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          mma_tile_kk(tSb, sbase + kPQB, sbase + kPK + st * kTile, false);    // S_B = Q_B K_j^T
          umma_commit(&s_full[1]);
          umma_commit(&k_empty[st]);
        }
        if (j >= 1) {
          if (!mbar_wait(v_full, pi, abort_flag) || !mbar_wait(&p_full[1], pi, abort_flag)) { ok = false; break; }
          tc_fence_after();
          mma_tile_kmn(tOb, sbase + kPPB, sbase + kPV, i > 0);    // O_B += P_B V_i
          umma_commit(&o_full[1]);
          umma_commit(&p_free[1]);
          umma_commit(v_empty);
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
    // ---------------- softmax: warps 4-7 tile A, warps 8-11 tile B ----------------
    const int side = (warp - 4) >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + (uint32_t)(side * 128) + lane_off, tO = tmem + 256 + (uint32_t)(side * 128) + lane_off;
    const uint32_t ptile = sbase + (side ? kPPB : kPPA);
    const int nx = side ? nb : na;
    const int diag = nx - 1;
    float m_ref = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nx && ok; ++j) {
      const uint32_t par = (uint32_t)j & 1u;
      if (!warp_wait(&s_full[side], par, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const bool dg = j == diag;
      const float mx = dg ? row_max<true>(tS, r, p.scale_log2) : row_max<false>(tS, r, p.scale_log2);
      // P V_{j-1} has read P and O holds every product up to j - 1
      if (!warp_wait(&p_free[side], par ^ 1u, abort_flag)) { ok = false; break; }
      tc_fence_after();
      if (__any_sync(0xFFFFFFFFu, mx > m_ref + kRescaleSlack)) {
        const float m_new = fmaxf(m_ref, mx);
        const float alpha = ex2_approx(m_ref - m_new);  // 0 on the first tile, 1 where nothing moves
        if (j > 0) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t w[32];
            tmem_ld32(tO + c * 32, w);
#pragma unroll
            for (int k = 0; k < 32; ++k) w[k] = __float_as_uint(__uint_as_float(w[k]) * alpha);
            tmem_st32(tO + c * 32, w);
          }
        }
        l *= alpha;
        m_ref = m_new;
      }
      l += dg ? row_probs<true>(tS, r, p.scale_log2, m_ref, ptile, &s_free[side])
              : row_probs<false>(tS, r, p.scale_log2, m_ref, ptile, &s_free[side]);
      fence_async_shared();
      mbar_arrive(&p_full[side]);
    }
    if (ok && !warp_wait(&o_full[side], (uint32_t)(nx - 1) & 1u, abort_flag)) ok = false;
    if (!ok) {
      atomicOr(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // O / l goes out through this tile's Q buffer (its last reader, S(nx - 1), has completed)
    const uint32_t qtile = sbase + (side ? kPQB : kPQA);
    const int t0 = side ? t0b : t0a;
    if (ok) {
      tc_fence_after();
      const float inv = 1.0f / l;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t ov[32], w[16];
        tmem_ld32(tO + c * 32, ov);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          w[k] = pack_bf16x2(__uint_as_float(ov[2 * k]) * inv, __uint_as_float(ov[2 * k + 1]) * inv);
        tile_put32(qtile, r, c, w);
      }
      p.lse[(int64_t)h * p.T + t0 + r] = (m_ref + log2f(l)) * 0.693147180559945309f;
    }
    fence_async_shared();
    named_bar_sync(1 + side, 128);
    if (r == 0 && !*abort_flag) {
      tma_store_2d(&tmAtt, qtile, h * kDh, t0);
      tma_store_2d(&tmAtt, qtile + kAtom, h * kDh + 64, t0);
      bulk_commit_and_wait();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Backward
// ---------------------------------------------------------------------------
struct AttnBwdArgs {
  int T, S, Hq, Hkv;
  int n_qt;
  float scale_log2;   // log2(e) / sqrt(128)
  float scale;        // 1 / sqrt(128)
  const float* lse2;  // [Hq, T] lse in the log2 domain
  const float* delta; // [Hq, T] D = rowsum(dO * O)
  unsigned* status;
};

__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// D[h, t] = sum_c dO[t, h*128 + c] * O[t, h*128 + c] (fp32, fixed order), lse2 = lse * log2(e).
// Lane l of a half-warp takes columns 8l .. 8l+7 of its head.
__global__ void __launch_bounds__(256) k_attn_bwd_delta(const uint16_t* __restrict__ att,
                                                        const uint16_t* __restrict__ datt,
                                                        const float* __restrict__ lse, int T, int Hq,
                                                        float* __restrict__ delta, float* __restrict__ lse2) {
  // one warp per (token, pair of heads): each half-warp reads one head's 128 elements of O and dO
  // as 16-byte pieces and reduces over its 16 lanes; consecutive warps take consecutive tokens of
  // the same head pair, so the per-head outputs (head-major) are written in runs
  const int hp_count = (Hq + 1) >> 1;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (int64_t)T * hp_count) return;
  const int hp = (int)(wid / T), t = (int)(wid - (int64_t)hp * T);
  const int h = 2 * hp + (lane >> 4);
  const bool live = h < Hq;
  float v = 0.0f;
  if (live) {
    const int64_t off = (int64_t)t * Hq * kDh + h * kDh + (lane & 15) * 8;
    const uint4 o = *reinterpret_cast<const uint4*>(att + off);
    const uint4 gd = *reinterpret_cast<const uint4*>(datt + off);
    const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, gw[4] = {gd.x, gd.y, gd.z, gd.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v = fmaf(bf16_lo(ow[k]), bf16_lo(gw[k]), v);
      v = fmaf(bf16_hi(ow[k]), bf16_hi(gw[k]), v);
    }
  }
#pragma unroll
  for (int k = 8; k >= 1; k >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, k);
  if (live && (lane & 15) == 0) {
    delta[(int64_t)h * T + t] = v;
    lse2[(int64_t)h * T + t] = lse[(int64_t)h * T + t] * 1.44269504088896341f;
  }
}

// 32 columns of a dS row (bf16 pairs) from the S and dP columns: P = 2^(s scale - lse2),
// dS = P (dP - D).  dQ (per row lse2, D): MASK drops keys after the query row r.  dK/dV
// (per column lse2, D from shared memory): MASK drops the columns before r, which the caller
// sets to the key row minus the query sub-tile's offset from the key tile.
// dS row chunk of the dQ pass: p = 2^(s scale - lse2), dS = p (dP - D), two columns per packed
// fused multiply-add / add / multiply.
template <bool MASK>
__device__ __forceinline__ void ds_row_chunk(const uint32_t (&sv)[32], const uint32_t (&dv)[32], int c, int r,
                                             float scale_log2, float lse2, float dlt, uint32_t (&w)[16]) {
  const float2 sc = make_float2(scale_log2, scale_log2), nl = make_float2(-lse2, -lse2), nd = make_float2(-dlt, -dlt);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int col = c * 32 + 2 * k;
    const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1])), sc, nl);
    const float2 pp = make_float2((MASK && col > r) ? 0.0f : ex2_approx(x.x), (MASK && col + 1 > r) ? 0.0f : ex2_approx(x.y));
    const float2 dd =
        __fmul2_rn(pp, __fadd2_rn(make_float2(__uint_as_float(dv[2 * k]), __uint_as_float(dv[2 * k + 1])), nd));
    w[k] = pack_bf16x2(dd.x, dd.y);
  }
}
// P^T and dS^T column chunk of the dK/dV pass (one key row per thread, query columns): lse2 and D
// per column from shared memory.
template <bool MASK>
__device__ __forceinline__ void pds_col_chunk(const uint32_t (&sv)[32], const uint32_t (&dv)[32], int c, int r,
                                              float scale_log2, const float* lse2, const float* dlt,
                                              uint32_t (&wp)[16], uint32_t (&ws)[16]) {
  const float2 sc = make_float2(scale_log2, scale_log2);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int col = c * 32 + 2 * k;
    const float2 l2 = *reinterpret_cast<const float2*>(lse2 + col), d2 = *reinterpret_cast<const float2*>(dlt + col);
    const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1])), sc,
                                make_float2(-l2.x, -l2.y));
    const float2 pt = make_float2((MASK && col < r) ? 0.0f : ex2_approx(x.x), (MASK && col + 1 < r) ? 0.0f : ex2_approx(x.y));
    const float2 dd = __fmul2_rn(
        pt, __fadd2_rn(make_float2(__uint_as_float(dv[2 * k]), __uint_as_float(dv[2 * k + 1])), make_float2(-d2.x, -d2.y)));
    wp[k] = pack_bf16x2(pt.x, pt.y);
    ws[k] = pack_bf16x2(dd.x, dd.y);
  }
}

// dK, dV: 64-query sub-tiles, so that two S^T / dP^T buffers (128 x 64 fp32 each) fit in TMEM
// beside the dV and dK accumulators and the Q / dO sub-tiles and the P^T / dS^T operand tiles are
// double-buffered: the next sub-tile's MMAs run while the current one's element-wise pass does.
constexpr int kSubAtom = 8192;            // 64 rows x 128 bytes
constexpr int kSubTile = 2 * kSubAtom;    // 64 x 128 bf16 (Q or dO sub-tile)
constexpr int kOpTile = 16384;            // 128 x 64 bf16 (P^T or dS^T): one 128-row swizzle atom column
constexpr int kKK = 0;                    // K tile (128 x 128)
constexpr int kKV = kKK + kTile;          // V tile
constexpr int kQdoStages = 3;             // a sub-tile's load starts three items ahead of its use
constexpr int kKQ = kKV + kTile;          // [3] Q sub-tiles
constexpr int kKO = kKQ + kQdoStages * kSubTile;  // [3] dO sub-tiles
constexpr int kKPT = kKO + kQdoStages * kSubTile; // [2] P^T tiles (contiguous: 32 KB staging for dV at the end)
constexpr int kKDST = kKPT + 2 * kOpTile; // [2] dS^T tiles (the same for dK)
constexpr int kKVec = kKDST + 2 * kOpTile; // [3] x (lse2[64], delta[64])
constexpr int kKBar = kKVec + kQdoStages * 512;
constexpr int kDkdvSmem = kKBar + 256 + 1024;
static_assert(kDkdvSmem <= 232448, "shared memory per CTA");

__host__ __device__ constexpr uint32_t idesc_bf16_n(int n, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | (((uint32_t)n >> 3) << 17) | ((128u >> 4) << 24);
}
// D (+)= A B^T, K = 128: A a K-major 128-row tile (16 KB atoms), B a K-major 64-row sub-tile (8 KB atoms).
__device__ __forceinline__ void mma_sub_kk(uint32_t d, uint32_t a, uint32_t b) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    umma_bf16(d, smem_desc_sw128(a + (kk >> 2) * kAtom + (kk & 3) * 32, 16, 1024),
              smem_desc_sw128(b + (kk >> 2) * kSubAtom + (kk & 3) * 32, 16, 1024), idesc_bf16_n(64, 0),
              kk ? 1u : 0u);
}
// D (+)= A B, K = 64: A a K-major 128 x 64 tile (one atom), B an MN-major 64-row sub-tile (N = 128).
__device__ __forceinline__ void mma_sub_kmn(uint32_t d, uint32_t a, uint32_t b, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    umma_bf16(d, smem_desc_sw128(a + kk * 32, 16, 1024), smem_desc_sw128(b + kk * 2048, kSubAtom, 1024),
              idesc_bf16_n(128, 1), (accumulate || kk) ? 1u : 0u);
}

__global__ void __launch_bounds__(kAttnBwdThreads, 1)
    k_attn_bwd_dkdv(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmQ64,
                    const __grid_constant__ CUtensorMap tmDO64, const __grid_constant__ CUtensorMap tmDQKV,
                    const AttnBwdArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kKBar);
  uint64_t* kv_full = bars + 0;
  uint64_t* qdo_full = bars + 1;   // [3]
  uint64_t* qdo_empty = bars + 4;  // [3]
  uint64_t* s_full = bars + 7;     // [2]
  uint64_t* s_free = bars + 9;     // [2]
  uint64_t* p_full = bars + 11;    // [2]
  uint64_t* p_free = bars + 13;    // [2]
  uint64_t* acc_full = bars + 15;
  uint64_t* drain = bars + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  int jt, g, b;  // key tile jt sees the query sub-tiles at or after it: jt = 0 is the longest
  cta_order<kDkdvBand>(p.n_qt, p.Hkv, p.T / p.S, jt, g, b);
  const int rep = p.Hq / p.Hkv;
  const int n_sub = 2 * (p.n_qt - jt);  // 64-query sub-tiles at or after this key tile
  const int n_items = rep * n_sub;      // item u: head g*rep + u / n_sub, sub-tile u % n_sub
  const int k0 = b * p.S + jt * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < kQdoStages; ++s) {
      mbar_init(&qdo_full[s], 1);
      mbar_init(&qdo_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 256);
      mbar_init(&p_full[s], 256);
      mbar_init(&p_free[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQKV);
    tma_prefetch_desc(&tmQ64);
    tma_prefetch_desc(&tmDO64);
    tma_prefetch_desc(&tmDQKV);
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
      uint32_t issued = 0, issued_par = 0;  // sub-tile stages with a load in flight, and its parity
      const int xk = (p.Hq + g) * kDh, xv = (p.Hq + p.Hkv + g) * kDh;
      mbar_arrive_expect_tx(kv_full, 2 * kTile);
      tma_load_2d(smem + kKK, &tmQKV, kv_full, xk, k0);
      tma_load_2d(smem + kKK + kAtom, &tmQKV, kv_full, xk + 64, k0);
      tma_load_2d(smem + kKV, &tmQKV, kv_full, xv, k0);
      tma_load_2d(smem + kKV + kAtom, &tmQKV, kv_full, xv + 64, k0);
      for (int u = 0; u < n_items; ++u) {
        const int st = u % kQdoStages;
        const uint32_t par = (uint32_t)(u / kQdoStages) & 1u;
        if (!mbar_wait(&qdo_empty[st], par ^ 1u, abort_flag)) { ok = false; break; }
        const int h = g * rep + u / n_sub;
        const int q0 = k0 + (u % n_sub) * 64;
        uint8_t* sq = smem + kKQ + st * kSubTile;
        uint8_t* so = smem + kKO + st * kSubTile;
        float* vec = reinterpret_cast<float*>(smem + kKVec + st * 512);  // st: the Q/dO stage
        mbar_arrive_expect_tx(&qdo_full[st], 2 * kSubTile + 512);
        tma_load_2d(sq, &tmQ64, &qdo_full[st], h * kDh, q0);
        tma_load_2d(sq + kSubAtom, &tmQ64, &qdo_full[st], h * kDh + 64, q0);
        tma_load_2d(so, &tmDO64, &qdo_full[st], h * kDh, q0);
        tma_load_2d(so + kSubAtom, &tmDO64, &qdo_full[st], h * kDh + 64, q0);
        bulk_load_1d(vec, p.lse2 + (int64_t)h * p.T + q0, 256, &qdo_full[st]);
        bulk_load_1d(vec + 64, p.delta + (int64_t)h * p.T + q0, 256, &qdo_full[st]);
        issued |= 1u << st;
        issued_par = (issued_par & ~(1u << st)) | (par << st);
      }
      if (!ok) {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
        int dummy = 0;
        mbar_wait(kv_full, 0, &dummy);
        for (int s = 0; s < kQdoStages; ++s)
          if (issued & (1u << s)) mbar_wait(&qdo_full[s], (issued_par >> s) & 1u, &dummy);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: S^T, dP^T of item u; dV, dK of item u-1 ----------------
      const uint32_t tdV = tmem + 256, tdK = tmem + 384;
      bool ok = mbar_wait(kv_full, 0, abort_flag);
      for (int u = 0; u <= n_items && ok; ++u) {
        if (u < n_items) {
          const int qs = u % kQdoStages, sb = u & 1;
          if (!mbar_wait(&qdo_full[qs], (uint32_t)(u / kQdoStages) & 1u, abort_flag) ||
              !mbar_wait(&s_free[sb], ((uint32_t)(u >> 1) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_sub_kk(tmem + sb * 64, sbase + kKK, sbase + kKQ + qs * kSubTile);        // S^T = K Q^T
          mma_sub_kk(tmem + 128 + sb * 64, sbase + kKV, sbase + kKO + qs * kSubTile);  // dP^T = V dO^T
          umma_commit(&s_full[sb]);
        }
        if (u >= 1) {
          const int i = u - 1, pb = i & 1, qs = i % kQdoStages;
          if (!mbar_wait(&p_full[pb], (uint32_t)(i >> 1) & 1u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          mma_sub_kmn(tdV, sbase + kKPT + pb * kOpTile, sbase + kKO + qs * kSubTile, i > 0);   // dV += P^T dO
          mma_sub_kmn(tdK, sbase + kKDST + pb * kOpTile, sbase + kKQ + qs * kSubTile, i > 0);  // dK += dS^T Q
          umma_commit(&qdo_empty[qs]);
          umma_commit(&p_free[pb]);
        }
      }
      if (ok) umma_commit(acc_full);
      else {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      umma_commit(drain);
      int dummy = 0;
      mbar_wait(drain, 0, &dummy);
    }
  } else if (warp >= 4) {
    // ---------------- P^T, dS^T (one key row per thread; warpgroup wg takes 32 of the 64 query columns) ----------------
    const int wg = (warp - 4) >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = true;
    for (int u = 0; u < n_items; ++u) {
      const int st = u & 1, qs = u % kQdoStages, v = u % n_sub;
      const uint32_t par = (uint32_t)(u >> 1) & 1u;
      // qdo_full: this thread reads the lse2 / delta vectors that arrived with the sub-tiles
      if (!warp_wait(&qdo_full[qs], (uint32_t)(u / kQdoStages) & 1u, abort_flag) ||
          !warp_wait(&s_full[st], par, abort_flag) || !warp_wait(&p_free[st], par ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* vec = reinterpret_cast<const float*>(smem + kKVec + qs * 512);
      {
        const int c = wg;
        uint32_t sv[32], dv[32], wp[16], ws[16];
        tmem_ld32x2(tmem + lane_off + st * 64 + c * 32, tmem + lane_off + 128 + st * 64 + c * 32, sv, dv);
        // sub-tiles 0 and 1 overlap the key tile: query q0 + col sees key k0 + r iff col >= r - 64 v
        if (v < 2) pds_col_chunk<true>(sv, dv, c, r - 64 * v, p.scale_log2, vec, vec + 64, wp, ws);
        else pds_col_chunk<false>(sv, dv, c, 0, p.scale_log2, vec, vec + 64, wp, ws);
        tile_put32(sbase + kKPT + st * kOpTile, r, c, wp);
        tile_put32(sbase + kKDST + st * kOpTile, r, c, ws);
      }
      tc_fence_before();
      mbar_arrive(&s_free[st]);
      fence_async_shared();
      mbar_arrive(&p_full[st]);
    }
    if (ok && !warp_wait(acc_full, 0, abort_flag)) ok = false;
    if (!ok) {
      atomicOr(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // dV and dK rows (dK scaled by 1/sqrt(128)) out through the P^T and dS^T regions (32 KB each,
    // the two 64-column halves of a 128 x 128 tile); every MMA has completed
    if (ok) {
      tc_fence_after();
#pragma unroll 1
      for (int c = 2 * wg; c < 2 * wg + 2; ++c) {
        uint32_t vv[32], kv[32], wv[16], wk[16];
        tmem_ld32(tmem + lane_off + 256 + c * 32, vv);
        tmem_ld32(tmem + lane_off + 384 + c * 32, kv);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          wv[k] = pack_bf16x2(__uint_as_float(vv[2 * k]), __uint_as_float(vv[2 * k + 1]));
          wk[k] = pack_bf16x2(__uint_as_float(kv[2 * k]) * p.scale, __uint_as_float(kv[2 * k + 1]) * p.scale);
        }
        tile_put32(sbase + kKPT, r, c, wv);
        tile_put32(sbase + kKDST, r, c, wk);
      }
    }
    fence_async_shared();
    named_bar_sync(1, 256);
    if (wg == 0 && r == 0 && !*abort_flag) {
      const int xk = (p.Hq + g) * kDh, xv = (p.Hq + p.Hkv + g) * kDh;
      tma_store_2d(&tmDQKV, sbase + kKDST, xk, k0);
      tma_store_2d(&tmDQKV, sbase + kKDST + kAtom, xk + 64, k0);
      tma_store_2d(&tmDQKV, sbase + kKPT, xv, k0);
      tma_store_2d(&tmDQKV, sbase + kKPT + kAtom, xv + 64, k0);
      bulk_commit_and_wait();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, kTmemCols);
}

// dQ shared-memory layout
// K_j feeds S_j and, a step later, dQ += dS_j K_j, so its stage is held the longest: three K
// stages let K_{j+3} load while the tensor core works on tiles j+1 and j+2.  V_j feeds only dP_j and
// its stage is released as soon as that product completes: two V stages.  (With one ring of two
// K/V stages released by dQ += dS_j K_j, the MMA that follows it, S_{j+2}, waited for the ring's
// reload on every tile.)
constexpr int kDqKStages = 3;
constexpr int kQQ = 0;
constexpr int kQO = kQQ + kTile;
constexpr int kQK = kQO + kTile;                // [3] stages
constexpr int kQV = kQK + kDqKStages * kTile;  // [2] stages
constexpr int kQBar = kQV + 2 * kTile;
constexpr int kDqSmem = kQBar + 256 + 1024;
static_assert(kDqSmem <= 232448, "shared memory per CTA");

// dQ TMEM columns: S, dP and the dQ accumulator (128 fp32 columns each), then two dS buffers of
// 128 x 128 bf16 (64 columns each, two keys per 32-bit column, the lower key in the low half):
// dQ += dS K takes dS as its A operand straight from TMEM, so the element-wise warps write it with
// tcgen05.st and no shared-memory tile or proxy fence sits between them and the MMA, and with two
// buffers dS_j is written while dQ += dS_{j-1} K_{j-1} still reads the other.
constexpr uint32_t kDqColS = 0, kDqColDP = 128, kDqColDQ = 256, kDqColDS = 384;

// 16 consecutive 32-bit columns of this thread's TMEM lane from registers (no wait).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// D (+)= A B, kind::f16 with A (bf16, K-major: row i in TMEM lane i, K along the columns) in TMEM
// at a_tmem and B (bf16) described in shared memory.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n"
      ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D (+)= A B over K = 128: A a 128 x 128 bf16 tile in TMEM (64 columns), B MN-major in shared
// memory (rows = K, two 64-wide N atoms).  K step kk: A columns 8 kk .. 8 kk + 7, B rows 16 kk ..
__device__ __forceinline__ void mma_tile_tmn(uint32_t d, uint32_t a_tmem, uint32_t b, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    umma_bf16_ts(d, a_tmem + (uint32_t)(kk * 8), smem_desc_sw128(b + kk * 2048, kAtom, 1024), idesc_bf16_128(1),
                 (accumulate || kk) ? 1u : 0u);
}

__global__ void __launch_bounds__(kAttnBwdThreads, 1)
    k_attn_bwd_dq(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmDO,
                  const __grid_constant__ CUtensorMap tmDQKV, const AttnBwdArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kQBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [3]
  uint64_t* k_empty = bars + 4;   // [3]
  uint64_t* v_full = bars + 7;    // [2]
  uint64_t* v_empty = bars + 9;   // [2]
  uint64_t* s_full = bars + 11;
  uint64_t* s_free = bars + 12;
  uint64_t* ds_full = bars + 13;  // [2]
  uint64_t* ds_free = bars + 15;  // [2]
  uint64_t* acc_full = bars + 17;
  uint64_t* drain = bars + 18;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 19);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  int rank, h, b;
  cta_order<kDqBand>(p.n_qt, p.Hq, p.T / p.S, rank, h, b);
  const int qt = p.n_qt - 1 - rank;
  const int g = h / (p.Hq / p.Hkv);
  const int t0 = b * p.S + qt * 128;
  const int n = qt + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kDqKStages; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
    mbar_init(s_full, 1);
    mbar_init(s_free, 256);
    for (int s = 0; s < 2; ++s) { mbar_init(&ds_full[s], 256); mbar_init(&ds_free[s], 1); }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQKV);
    tma_prefetch_desc(&tmDO);
    tma_prefetch_desc(&tmDQKV);
  }
  if (warp == 2) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_addr(smem);

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      // loads in flight, and the parity of their full[] phase: K stages in bits 0..2, V in 3..4
      uint32_t issued = 0, issued_par = 0;
      mbar_arrive_expect_tx(q_full, 2 * kTile);
      tma_load_2d(smem + kQQ, &tmQKV, q_full, h * kDh, t0);
      tma_load_2d(smem + kQQ + kAtom, &tmQKV, q_full, h * kDh + 64, t0);
      tma_load_2d(smem + kQO, &tmDO, q_full, h * kDh, t0);
      tma_load_2d(smem + kQO + kAtom, &tmDO, q_full, h * kDh + 64, t0);
      const int xk = (p.Hq + g) * kDh, xv = (p.Hq + p.Hkv + g) * kDh;
      for (int j = 0; j < n; ++j) {
        const int y = b * p.S + j * 128;
        const int ks = j % kDqKStages, vs = j & 1;
        const uint32_t ku = (uint32_t)(j / kDqKStages) & 1u, vu = (uint32_t)(j >> 1) & 1u;
        if (!mbar_wait(&k_empty[ks], ku ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sk = smem + kQK + ks * kTile;
        mbar_arrive_expect_tx(&k_full[ks], kTile);
        tma_load_2d(sk, &tmQKV, &k_full[ks], xk, y);
        tma_load_2d(sk + kAtom, &tmQKV, &k_full[ks], xk + 64, y);
        issued |= 1u << ks;
        issued_par = (issued_par & ~(1u << ks)) | (ku << ks);
        if (!mbar_wait(&v_empty[vs], vu ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sv = smem + kQV + vs * kTile;
        mbar_arrive_expect_tx(&v_full[vs], kTile);
        tma_load_2d(sv, &tmQKV, &v_full[vs], xv, y);
        tma_load_2d(sv + kAtom, &tmQKV, &v_full[vs], xv + 64, y);
        issued |= 1u << (3 + vs);
        issued_par = (issued_par & ~(1u << (3 + vs))) | (vu << (3 + vs));
      }
      if (!ok) {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
        int dummy = 0;
        mbar_wait(q_full, 0, &dummy);
        for (int s = 0; s < kDqKStages; ++s)
          if (issued & (1u << s)) mbar_wait(&k_full[s], (issued_par >> s) & 1u, &dummy);
        for (int s = 0; s < 2; ++s)
          if (issued & (1u << (3 + s))) mbar_wait(&v_full[s], (issued_par >> (3 + s)) & 1u, &dummy);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t tS = tmem + kDqColS, tdP = tmem + kDqColDP, tdQ = tmem + kDqColDQ;
      // S_j and dP_j are issued as soon as the element-wise warps have taken S_{j-1} and dP_{j-1}
      // into registers, ahead of dQ += dS_{j-1} K_{j-1}: the tensor core works on tile j while the
      // element-wise pass forms dS_{j-1}
      bool ok = mbar_wait(q_full, 0, abort_flag);
      for (int j = 0; j <= n && ok; ++j) {
        if (j < n) {
          const int ks = j % kDqKStages, vs = j & 1;
          const uint32_t ku = (uint32_t)(j / kDqKStages) & 1u, vu = (uint32_t)(j >> 1) & 1u, par = (uint32_t)j & 1u;
          if (!mbar_wait(&k_full[ks], ku, abort_flag) || !mbar_wait(&v_full[vs], vu, abort_flag) ||
              !mbar_wait(s_free, par ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tile_kk(tS, sbase + kQQ, sbase + kQK + ks * kTile, false);   // S = Q K^T
          mma_tile_kk(tdP, sbase + kQO, sbase + kQV + vs * kTile, false);  // dP = dO V^T
          umma_commit(s_full);
          umma_commit(&v_empty[vs]);
        }
        if (j > 0) {
          const int jj = j - 1, ks = jj % kDqKStages, sb = jj & 1;
          if (!mbar_wait(&ds_full[sb], (uint32_t)(jj >> 1) & 1u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          mma_tile_tmn(tdQ, tmem + kDqColDS + (uint32_t)(sb * 64), sbase + kQK + ks * kTile, jj > 0);  // dQ += dS K
          umma_commit(&k_empty[ks]);
          umma_commit(&ds_free[sb]);
        }
      }
      if (ok) umma_commit(acc_full);
      else {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      umma_commit(drain);
      int dummy = 0;
      mbar_wait(drain, 0, &dummy);
    }
  } else if (warp >= 4) {
    // one query row per thread; warpgroup wg takes the key columns 64 wg .. 64 wg + 63
    const int wg = (warp - 4) >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + kDqColS + lane_off, tdP = tmem + kDqColDP + lane_off;
    const float lse2 = p.lse2[(int64_t)h * p.T + t0 + r];
    const float dlt = p.delta[(int64_t)h * p.T + t0 + r];
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const uint32_t par = (uint32_t)j & 1u;
      const bool diag = j == qt;
      if (!warp_wait(s_full, par, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // this warpgroup's 64 columns of S_j and dP_j into registers, then TMEM is free for S_{j+1}
      const int c0 = 2 * wg, c1 = c0 + 1;
      uint32_t s0[32], d0[32], s1[32], d1[32];
      tmem_ld32x2(tS + c0 * 32, tdP + c0 * 32, s0, d0);
      tmem_ld32x2(tS + c1 * 32, tdP + c1 * 32, s1, d1);
      tc_fence_before();
      mbar_arrive(s_free);
      // dS buffer j & 1 is rewritten once dQ += dS_{j-2} K_{j-2} has read it
      const int sb = j & 1;
      if (!warp_wait(&ds_free[sb], ((uint32_t)(j >> 1) & 1u) ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      const uint32_t tdS = tmem + kDqColDS + (uint32_t)(sb * 64) + lane_off;
      uint32_t w[16];
      if (diag) ds_row_chunk<true>(s0, d0, c0, r, p.scale_log2, lse2, dlt, w);
      else ds_row_chunk<false>(s0, d0, c0, r, p.scale_log2, lse2, dlt, w);
      tmem_st16(tdS + (uint32_t)(c0 * 16), w);
      if (diag) ds_row_chunk<true>(s1, d1, c1, r, p.scale_log2, lse2, dlt, w);
      else ds_row_chunk<false>(s1, d1, c1, r, p.scale_log2, lse2, dlt, w);
      tmem_st16(tdS + (uint32_t)(c1 * 16), w);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&ds_full[sb]);
    }
    if (ok && !warp_wait(acc_full, 0, abort_flag)) ok = false;
    if (!ok) {
      atomicOr(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // dQ row (scaled by 1/sqrt(128)) out through the Q tile (every MMA has completed)
    if (ok) {
      tc_fence_after();
      const uint32_t tdQ = tmem + kDqColDQ + lane_off;
#pragma unroll 1
      for (int c = 2 * wg; c < 2 * wg + 2; ++c) {
        uint32_t qv[32], w[16];
        tmem_ld32(tdQ + c * 32, qv);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          w[k] = pack_bf16x2(__uint_as_float(qv[2 * k]) * p.scale, __uint_as_float(qv[2 * k + 1]) * p.scale);
        tile_put32(sbase + kQQ, r, c, w);
      }
    }
    fence_async_shared();
    named_bar_sync(1, 256);
    if (wg == 0 && r == 0 && !*abort_flag) {
      tma_store_2d(&tmDQKV, sbase + kQQ, h * kDh, t0);
      tma_store_2d(&tmDQKV, sbase + kQQ + kAtom, h * kDh + 64, t0);
      bulk_commit_and_wait();
    }
  }
  tc_fence_before();
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

// bf16 matrix [rows, cols] (row stride ld elements) in boxes 64 elements (128 bytes) wide and
// box_rows high, 128-byte swizzle.
bool make_tile_map(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t ld, int box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Opt a kernel into its dynamic shared memory once per device; `configured` is that kernel's own flag.
template <class K>
cudaError_t set_smem(K kernel, int bytes, int& configured) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured == dev) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) configured = dev;
  return e;
}
int g_cfg_fwd = -1, g_cfg_fwd_pair = -1, g_cfg_dkdv = -1, g_cfg_dq = -1;

AttnBwdArgs bwd_args(int64_t T, int S, int Hq, int Hkv, const float* delta, const float* lse2, const Launch& L) {
  AttnBwdArgs a{};
  a.T = (int)T;
  a.S = S;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.n_qt = S / 128;
  a.scale_log2 = 1.44269504088896341f / 11.3137084989847604f;  // log2(e) / sqrt(128)
  a.scale = 1.0f / 11.3137084989847604f;
  a.lse2 = lse2;
  a.delta = delta;
  a.status = L.status;
  return a;
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
  if (a.n_qt % 2 == 0) {
    // pairs of query tiles share their K/V tiles and overlap each other's softmax
    cudaError_t e = set_smem(k_attn_fwd_pair, kPairSmem, g_cfg_fwd_pair);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(a.n_qt / 2) * (unsigned)Hq * (unsigned)(T / S);
    k_attn_fwd_pair<<<grid, kPairThreads, kPairSmem, L.stream>>>(tq, ta, a);
  } else {
    cudaError_t e = set_smem(k_attn_fwd, kFwdSmem, g_cfg_fwd);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)a.n_qt * (unsigned)Hq * (unsigned)(T / S);
    k_attn_fwd<<<grid, kAttnThreads, kFwdSmem, L.stream>>>(tq, ta, a);
  }
  if (L.launches) ++*L.launches;
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_delta(const uint16_t* att, const uint16_t* datt, const float* lse, int64_t T, int Hq,
                                  float* delta, float* lse2, const Launch& L) {
  const int64_t warps = T * ((Hq + 1) / 2);
  k_attn_bwd_delta<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, L.stream>>>(att, datt, lse, (int)T, Hq, delta, lse2);
  if (L.launches) ++*L.launches;
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dkdv(const uint16_t* qkv, const uint16_t* datt, int64_t T, int S, int Hq, int Hkv,
                                 const float* delta, const float* lse2, uint16_t* dqkv, const Launch& L) {
  const int64_t nq = (int64_t)(Hq + 2 * Hkv) * kDh, da = (int64_t)Hq * kDh;
  CUtensorMap tq, tq64, tdo64, tdq;
  if (!make_tile_map(&tq, qkv, nq, T, nq) || !make_tile_map(&tq64, qkv, nq, T, nq, 64) ||
      !make_tile_map(&tdo64, datt, da, T, da, 64) || !make_tile_map(&tdq, dqkv, nq, T, nq))
    return cudaErrorInvalidValue;
  const AttnBwdArgs a = bwd_args(T, S, Hq, Hkv, delta, lse2, L);
  cudaError_t e = set_smem(k_attn_bwd_dkdv, kDkdvSmem, g_cfg_dkdv);
  if (e != cudaSuccess) return e;
  k_attn_bwd_dkdv<<<(unsigned)a.n_qt * (unsigned)Hkv * (unsigned)(T / S), kAttnBwdThreads, kDkdvSmem, L.stream>>>(
      tq, tq64, tdo64, tdq, a);
  if (L.launches) ++*L.launches;
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dq(const uint16_t* qkv, const uint16_t* datt, int64_t T, int S, int Hq, int Hkv,
                               const float* delta, const float* lse2, uint16_t* dqkv, const Launch& L) {
  const int64_t nq = (int64_t)(Hq + 2 * Hkv) * kDh, da = (int64_t)Hq * kDh;
  CUtensorMap tq, tdo, tdq;
  if (!make_tile_map(&tq, qkv, nq, T, nq) || !make_tile_map(&tdo, datt, da, T, da) ||
      !make_tile_map(&tdq, dqkv, nq, T, nq))
    return cudaErrorInvalidValue;
  const AttnBwdArgs a = bwd_args(T, S, Hq, Hkv, delta, lse2, L);
  cudaError_t e = set_smem(k_attn_bwd_dq, kDqSmem, g_cfg_dq);
  if (e != cudaSuccess) return e;
  k_attn_bwd_dq<<<(unsigned)a.n_qt * (unsigned)Hq * (unsigned)(T / S), kAttnBwdThreads, kDqSmem, L.stream>>>(
      tq, tdo, tdq, a);
  if (L.launches) ++*L.launches;
  return cudaGetLastError();
}

}  // namespace fp8q
