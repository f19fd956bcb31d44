// Persistent, warp-specialised FP8 GEMM for sm_103a on the 5th-generation
// tensor cores (tcgen05.mma kind::f8f6f4), with the block pipeline's
// epilogues fused in (LLMQ §3: non-matmul ops fused around the matmuls;
// §3.1: quantization fused with the nonlinearity; §4: FP8 matmuls dominate).
//
// Tile 128 x 256 x 128 (M x N x K bytes), one CTA per SM, 4-stage TMA ring:
//   warp 0      TMA producer: A tile 128x128 B and B tile as two 128x128 B
//               halves (the halves let the gate/up GEMM pair column j of the
//               gate with column f+j of the up projection inside one tile);
//   warp 1      MMA issuer: 4 x tcgen05.mma 128x256x32 per stage into one of
//               two TMEM accumulators (2 x 256 fp32 columns), tcgen05.commit
//               frees the smem stage / hands the accumulator to the epilogue;
//   warp 2      TMEM allocation (512 columns) and release;
//   warps 4..11 epilogue, two warpgroups: warp w reads TMEM lanes
//               32*(w%4)..+31 (= 32 rows); warpgroup 0 takes the first half
//               of the accumulator columns, warpgroup 1 the second half;
//               scale by alpha = sinvA * sinvB, fused op, then each warp
//               writes its 32x32 output block into a swizzled 4 KB shared
//               staging buffer and stores it with one TMA tensor store
//               (coalesced, clipped at the tensor edges).
// Operands may be K-major or MN-major in global memory (NN/NT/TN layouts
// without transpose copies): TMA boxes are 128 B wide along the contiguous
// dimension with the 128-byte swizzle, and the UMMA shared-memory descriptors
// declare the matching major-ness.
// The same kernel with 16-bit operands (OP16: bf16, tcgen05.mma kind::f16,
// K = 16 per instruction) is the BF16 baseline the FP8 path is compared with:
// a stage still holds 128 bytes of K per row (64 bf16), so the ring, the
// swizzle and the epilogues are unchanged; the scale factor alpha is 1.
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA records
// FP8Q_STATUS_TIMEOUT, stops issuing work, drains what it issued, frees TMEM
// and exits.
#include "fp8q_common.cuh"
#include "fp8q_internal.h"

#include <mutex>

namespace fp8q {

namespace {

constexpr int BM = 128, BN = 256, BK = 128;  // BK: bytes of K per stage
constexpr int kATile = BM * BK;   // 16 KB
constexpr int kBHalf = 128 * BK;  // 16 KB
constexpr int kStage = kATile + 2 * kBHalf;
constexpr int kThreads = 384;   // warps 0-3: TMA / MMA / TMEM / idle; warps 4-11: epilogue
constexpr int kEpiThreads = 256;
constexpr int kTmemCols = 512;
constexpr int kStagingBytes = 4096;                  // per epilogue warp
constexpr int kSfChunk = 512;                        // E8M0 codes of 128 rows x 4 blocks of 32

// Shared-memory and tensor-memory plan of the 128 x 256 kernel.  Per-tensor FP8 and bf16: a 4-stage
// operand ring and two TMEM accumulators (the epilogue of one tile overlaps the next tile's MMAs).
// Block-scaled MXFP8 (MX): each stage also carries the stage's scale chunks (A: 128 rows, B: two
// 128-column halves, 4 blocks of 32 each), which the MMA thread copies into tensor memory next to
// the accumulator; a 3-stage ring leaves room for them, and one accumulator (TMEM columns 0-255)
// leaves the columns from 256 for the per-stage scale slots (32 columns each, A and B 16 apart).
template <int MX>
struct Plan {
  static constexpr int kStages = MX ? 3 : 4;
  static constexpr int kAcc = MX ? 1 : 2;
  static constexpr int kSfStage = MX ? 3 * kSfChunk : 0;
  static constexpr int kSfOffset = kStages * kStage;
  static constexpr int kStagingOffset = kSfOffset + ((kStages * kSfStage + 1023) & ~1023);
  static constexpr int kBarOffset = kStagingOffset + 8 * kStagingBytes;
  static constexpr int kSmemBytes = kBarOffset + 256 + 1024;  // + barriers + alignment slack
  static constexpr int kSfTmemCol = 256;                     // first scale column (MX)
  static constexpr int kSfTmemStage = 32;                    // A: 4 columns at +0, B: 2 x 4 at +16
  static constexpr int kSfTmemB = 16;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(!MX || kSfTmemCol + kStages * kSfTmemStage <= kTmemCols, "tensor memory");
};
constexpr int kGroupRows = 2048;                     // rows of A per rasterisation group (the default)

struct Args {
  int M, N, K;
  int m_tiles, n_tiles, k_blocks;
  int m_units, num_tiles;  // scheduling units: M tiles; num_tiles = m_units x n_tiles
  int group;               // M units per rasterisation group
  int b_step, b_half1;  // B's N coordinate of a tile = nb * b_step (+ b_half1 for the second half)
  int epi, out_f32;
  uint32_t idesc;
  const float* sinvA;
  const float* sinvB;
  void* C;
  int64_t ldc;
  const uint16_t* R;
  int64_t ldr;
  uint16_t* aux16;  // kEpiSwiglu: the bf16 SwiGLU output a [M, N] (ld = N), or null
  const uint8_t* sfA;  // MX: E8M0 scale chunks of A (rows M) and B (rows b_cols), sf_kc chunks per row chunk
  const uint8_t* sfB;
  int sf_kc;
  int b_cols;
  uint64_t wait_ns;  // limit of every pipeline wait (the drains after a time-out keep kWaitLimitNs)
  const float* qscale;  // kEpiSwiglu: with it, a is written as E4M3 codes fp8(fl32(a * *qscale)) instead
  uint32_t* amax_partial;
  unsigned* status;
};

// Unit -> (M unit, N tile), rasterised in groups of p.group M units: all N tiles of a group before
// the next group, M fastest inside it, so that the group's A rows stay in L2 while B streams.
__device__ __forceinline__ void tile_coords(int tile, const Args& p, int& mb, int& nb) {
  const int G = p.group;
  const int span = G * p.n_tiles;
  const int grp = tile / span;
  const int first_m = grp * G;
  const int gm = min(G, p.m_units - first_m);
  const int local = tile - grp * span;
  mb = first_m + local % gm;
  nb = local / gm;
}

// ---------------------------------------------------------------------------
// Epilogue helpers.  One thread = one output row of its warp's 32-row slice;
// a chunk is 32 consecutive columns.  Outputs go through the warp's staging
// buffer: 32 x 32 bf16 in the 64-byte-swizzle layout (64 B rows) or 32 x 32
// fp32 in the 128-byte-swizzle layout (128 B rows), matching the tensor maps.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// bf16 round-to-nearest-even of the exact value s + e, where s is an fp32
// rounding of it and e the rounding error (|e| <= half an fp32 ulp).  Only an
// s exactly on a bf16 midpoint can round differently from the exact value;
// there the sign of e decides.  This makes each bf16 storage point one rounding
// of the exact result instead of two (fp32, then bf16).
__device__ __forceinline__ float round_bf16_exact(float s, float e) {
  const uint32_t u = __float_as_uint(s);
  if ((u & 0xFFFFu) == 0x8000u && e != 0.0f && (u & 0x7F800000u) != 0x7F800000u) {
    const bool away = (e > 0.0f) == ((u >> 31) == 0u);  // e pushes the magnitude up
    return __uint_as_float((away ? u + 0x8000u : u - 0x8000u) & 0xFFFF0000u);
  }
  return round_bf16(s);
}
// bf16 of alpha * acc, one rounding of the exact product.
__device__ __forceinline__ float bf16_of_product(float alpha, float acc) {
  const float v = __fmul_rn(alpha, acc);
  return round_bf16_exact(v, __fmaf_rn(alpha, acc, -v));
}
// bf16 of r + alpha * acc (r a bf16 value), one rounding of the exact sum.
__device__ __forceinline__ float bf16_of_residual(float r, float alpha, float acc) {
  const float v = __fmul_rn(alpha, acc);
  const float ev = __fmaf_rn(alpha, acc, -v);  // alpha * acc = v + ev exactly
  const float s = __fadd_rn(r, v);
  const float bb = __fsub_rn(s, r);            // TwoSum: r + v = s + es exactly
  const float es = __fadd_rn(__fsub_rn(r, __fsub_rn(s, bb)), __fsub_rn(v, bb));
  return round_bf16_exact(s, __fadd_rn(es, ev));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void stage_bf16(uint32_t buf, int r, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    st_shared_v4(buf + r * 64 + ((q ^ ((r >> 1) & 3)) << 4),
                 make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                            pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7])));
}
// 32 rows x 32 bytes of FP8 codes (32-byte rows, 32-byte swizzle).
__device__ __forceinline__ void stage_u8(uint32_t buf, int r, const uint32_t (&w)[8]) {
#pragma unroll
  for (int q = 0; q < 2; ++q)
    st_shared_v4(buf + r * 32 + ((q ^ ((r >> 2) & 1)) << 4), make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
}
__device__ __forceinline__ void stage_f32(uint32_t buf, int r, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    st_shared_v4(buf + r * 128 + ((q ^ (r & 7)) << 4),
                 make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]), __float_as_uint(v[4 * q + 2]),
                            __float_as_uint(v[4 * q + 3])));
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tm), "r"(src),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// The staging buffer may be rewritten once the warp's previous stores have read it.
__device__ __forceinline__ void staging_acquire(int lane) {
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
}
// Make this warp's shared-memory writes visible to the TMA engine.
__device__ __forceinline__ void staging_publish() {
  fence_async_shared();
  __syncwarp();
}

__device__ __forceinline__ void load_bf16x32(const uint16_t* src, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = ld_v4(src + 8 * q);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) { v[8 * q + 2 * k] = bf16_lo(ww[k]); v[8 * q + 2 * k + 1] = bf16_hi(ww[k]); }
  }
}

// dA = alpha * acc; with h = H_gate, u = H_up, s = sigmoid(h):
// dH_gate = dA u s (1 + h (1 - s)), dH_up = dA h s, both rounded to bf16.
// dH is a GEMM output checked against the oracle with a tolerance, so the
// sigmoid may use the fast hardware exponential and reciprocal.
__device__ __forceinline__ void swiglu_bwd1(float da, float h, float u, float& dg, float& du) {
  const float s = __fdividef(1.0f, 1.0f + __expf(-h));
  const float hs = h * s;
  dg = round_bf16(da * u * (s + hs * (1.0f - s)));
  du = round_bf16(da * hs);
}

// H words of one 32-column chunk of a row: gate in h[0..3], up in h[4..7]
// (8 bf16 each); columns at or beyond ncol read as zero.
__device__ __forceinline__ void load_h_chunk(const Args& p, int row, int col, int ncol, uint4 (&h)[8]) {
  const uint16_t* hrow = p.R + (int64_t)row * p.ldr;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (8 * q < ncol) {
      h[q] = ld_v4(hrow + col + 8 * q);
      h[4 + q] = ld_v4(hrow + p.N + col + 8 * q);
    } else {
      h[q] = h[4 + q] = make_uint4(0, 0, 0, 0);
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// Output maps: tmC (C, or the gate half of H / dH), tmC2 (the up half), tmAux
// (the SwiGLU output a); unused ones are copies of tmC.
// MX: block-scaled MXFP8 operands (tcgen05.mma kind::mxf8f6f4.block_scale), alpha = 1.
template <int A_MN, int B_MN, int OP16, int MX>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_f8(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2,
              const __grid_constant__ CUtensorMap tmAux, const Args p) {
  static_assert(!(MX && OP16), "block scaling takes FP8 operands");
  using PL = Plan<MX>;
  constexpr int STAGES = PL::kStages;
  constexpr int NACC = PL::kAcc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + PL::kBarOffset);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;   // [NACC]
  uint64_t* tempty = tfull + NACC;    // [NACC]
  uint64_t* drain = tempty + NACC;    // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* cta_amax = reinterpret_cast<uint32_t*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's tiles: first, first + step, ...
  const int u_first = (int)blockIdx.x;
  const int u_step = (int)gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < NACC; ++a) { mbar_init(&tfull[a], 1); mbar_init(&tempty[a], kEpiThreads); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *cta_amax = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 2) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;      // bit s: stage s has a load in flight or consumed
      uint32_t issued_par = 0;  // bit s: parity of the full[] phase of that load
      bool ok = true;
      for (int tile = u_first; tile < p.num_tiles && ok; tile += u_step) {
        int mb, nb;
        tile_coords(tile, p, mb, nb);
        const int m0 = mb * BM;
        const int n0 = nb * p.b_step, n1 = n0 + p.b_half1;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.wait_ns)) { ok = false; break; }
          uint8_t* sA = smem + stage * kStage;
          uint8_t* sB = sA + kATile;
          // the whole stage lands here: the A tile and both B halves (and their scale chunks)
          mbar_arrive_expect_tx(&full[stage], kStage + PL::kSfStage);
          const int k0 = kb * (OP16 ? BK / 2 : BK);  // in elements
          if (MX) {
            // chunk (row chunk, kb) of each operand: A's 128 rows, B's two 128-column halves (a
            // half past B's columns -- a ragged last tile -- repeats the first: its columns are
            // zero-filled and never stored)
            uint8_t* sSF = smem + PL::kSfOffset + stage * PL::kSfStage;
            const int n1c = n1 < p.b_cols ? n1 : n0;
            bulk_load(sSF, p.sfA + ((int64_t)(m0 >> 7) * p.sf_kc + kb) * kSfChunk, kSfChunk, &full[stage]);
            bulk_load(sSF + kSfChunk, p.sfB + ((int64_t)(n0 >> 7) * p.sf_kc + kb) * kSfChunk, kSfChunk, &full[stage]);
            bulk_load(sSF + 2 * kSfChunk, p.sfB + ((int64_t)(n1c >> 7) * p.sf_kc + kb) * kSfChunk, kSfChunk,
                      &full[stage]);
          }
          if (A_MN) {
            if (OP16) {  // two 64-element-wide MN boxes of 64 K rows
              tma_load_2d(sA, &tmA, &full[stage], m0, k0);
              tma_load_2d(sA + kATile / 2, &tmA, &full[stage], m0 + 64, k0);
            } else {
              tma_load_2d(sA, &tmA, &full[stage], m0, k0);
            }
          } else {
            tma_load_2d(sA, &tmA, &full[stage], k0, m0);
          }
          if (B_MN) {
            if (OP16) {
              tma_load_2d(sB, &tmB, &full[stage], n0, k0);
              tma_load_2d(sB + kBHalf / 2, &tmB, &full[stage], n0 + 64, k0);
              tma_load_2d(sB + kBHalf, &tmB, &full[stage], n1, k0);
              tma_load_2d(sB + kBHalf + kBHalf / 2, &tmB, &full[stage], n1 + 64, k0);
            } else {
              tma_load_2d(sB, &tmB, &full[stage], n0, k0);
              tma_load_2d(sB + kBHalf, &tmB, &full[stage], n1, k0);
            }
          } else {
            tma_load_2d(sB, &tmB, &full[stage], k0, n0);
            tma_load_2d(sB + kBHalf, &tmB, &full[stage], k0, n1);
          }
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
        // let every copy this thread started land before the CTA can exit
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s)) {
            int dummy = 0;
            mbar_wait(&full[s], (issued_par >> s) & 1u, &dummy);
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = u_first; tile < p.num_tiles && ok; tile += u_step) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sA = smem_addr(smem + stage * kStage);
          const uint32_t sB = sA + kATile;
          // MX: the stage's scale chunks into its tensor-memory slot (A: 4 columns, B: 2 x 4 from
          // column 16 of the slot, the second half's chunk 4 columns after the first); a
          // tcgen05.cp and the MMAs issued after it by this thread execute in order.  The slot was
          // last read by the MMAs of this stage's previous fill, whose commit released the stage
          // before its refill could complete.
          const uint32_t t_sfa = tmem_base + (uint32_t)(PL::kSfTmemCol + stage * PL::kSfTmemStage);
          const uint32_t t_sfb = t_sfa + PL::kSfTmemB;
          if (MX) {
            const uint32_t sSF = smem_addr(smem + PL::kSfOffset + stage * PL::kSfStage);
            tc_cp_sf(t_sfa, smem_desc_sf(sSF));
            tc_cp_sf(t_sfb, smem_desc_sf(sSF + kSfChunk));
            tc_cp_sf(t_sfb + 4, smem_desc_sf(sSF + 2 * kSfChunk));
          }
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            // One MMA consumes 32 bytes of K (32 FP8 or 16 bf16 elements).  K-major: advance
            // 32 bytes inside the 128-byte swizzle row.  MN-major: advance 32 (FP8) or 16 (bf16)
            // K rows of 128 B; consecutive 128-byte-wide MN blocks lie one block (all K rows of
            // the stage) apart.
            constexpr uint32_t kMnStep = OP16 ? 2048 : 4096, kMnLbo = OP16 ? kBHalf / 2 : kBHalf;
            const uint64_t ad = A_MN ? smem_desc_sw128(sA + kk * kMnStep, kMnLbo, 1024) : smem_desc_sw128(sA + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(sB + kk * kMnStep, kMnLbo, 1024) : smem_desc_sw128(sB + kk * 32, 16, 1024);
            if (OP16) umma_bf16(d_tmem, ad, bd, p.idesc, (kb | kk) != 0 ? 1u : 0u);
            else if (MX) umma_mx(d_tmem, ad, bd, p.idesc | mx_sf_ids(kk), t_sfa, t_sfb, (kb | kk) != 0 ? 1u : 0u);
            else umma_f8(d_tmem, ad, bd, p.idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok) {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // wait for every MMA this thread issued before TMEM can be released
      umma_commit(drain);
      int dummy = 0;
      mbar_wait(drain, 0, &dummy);
    }
  } else if (warp >= 4) {
    // ---------------- epilogue ----------------
    const int sub = warp & 3;
    const int half = (warp - 4) >> 2;  // which half of the accumulator columns
    const uint32_t buf = smem_addr(smem + PL::kStagingOffset + (warp - 4) * kStagingBytes);
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t amax = 0;
    const float alpha = p.sinvA ? __fmul_rn(*p.sinvA, *p.sinvB) : 1.0f;  // 1: unscaled (bf16) operands
    for (int tile = u_first; tile < p.num_tiles; tile += u_step) {
      int mb, nb;
      tile_coords(tile, p, mb, nb);
      const int row0 = mb * BM + sub * 32;
      const int row = row0 + lane;
      const bool row_ok = row < p.M;
      const bool warp_ok = row0 < p.M;  // any row of this warp's slice in range
      // The SwiGLU backward's first H chunk is requested before the accumulator is ready.  (An
      // L2 prefetch of the warp's whole part of the tile measured slower: one request per lane
      // and line through the same load path as the chunks themselves.)
      uint4 hn[8];
      if (p.epi == kEpiSwigluBwd) {
        const int cs = nb * BN + 128 * half;
        if (row_ok && cs < p.N) load_h_chunk(p, row, cs, min(32, p.N - cs), hn);
      }
      // lane 0 waits and the warp follows its result: the tcgen05.ld below is warp-collective,
      // so a time-out must take the whole warp out together
      int full_ok = 0;
      if (lane == 0) full_ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, p.wait_ns) ? 1 : 0;
      if (!__shfl_sync(0xFFFFFFFFu, full_ok, 0)) {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(sub * 32) << 16);
      if (p.epi == kEpiSwiglu) {
        const int col0 = nb * 128;
#pragma unroll 1
        for (int c = 2 * half; c < 2 * half + 2; ++c) {
          uint32_t ag[32], au[32];
          tmem_ld32x2(tbase + c * 32, tbase + 128 + c * 32, ag, au);
          const int col = col0 + c * 32;
          const int ncol = min(32, p.N - col);
          float hg[32], hu[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            // H = bf16 of the fp32 product (two roundings: its cost in this epilogue-bound
            // GEMM outweighs the rare last-bit difference from one rounding)
            hg[j] = round_bf16(__fmul_rn(alpha, __uint_as_float(ag[j])));
            hu[j] = round_bf16(__fmul_rn(alpha, __uint_as_float(au[j])));
          }
          if (warp_ok && ncol > 0) {
            staging_acquire(lane);
            stage_bf16(buf, lane, hg);
            stage_bf16(buf + 2048, lane, hu);
            staging_publish();
            if (lane == 0) {
              tma_store_2d(&tmC, buf, col, row0);
              tma_store_2d(&tmC2, buf + 2048, col, row0);
              bulk_commit();
            }
          }
          if (p.aux16 || p.qscale) {
            // a = SwiGLU(H) is written too: bf16 (the BF16 baseline) or, recomputing with the
            // retained scale, as E4M3 codes (SwiGLU fused with the cast)
            float a[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              a[j] = swiglu_fast(hg[j], hu[j]);
              if (row_ok && j < ncol) amax = max(amax, abs_bits(a[j]));
            }
            if (warp_ok && ncol > 0) {
              staging_acquire(lane);
              if (p.aux16) {
                stage_bf16(buf, lane, a);
              } else {
                const float sq = *p.qscale;
                uint32_t w[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  w[q] = cvt_fp8x4<0>(__fmul_rn(a[4 * q], sq), __fmul_rn(a[4 * q + 1], sq),
                                      __fmul_rn(a[4 * q + 2], sq), __fmul_rn(a[4 * q + 3], sq));
                stage_u8(buf, lane, w);
              }
              staging_publish();
              if (lane == 0) {
                tma_store_2d(&tmAux, buf, col, row0);
                bulk_commit();
              }
            }
          } else if (p.amax_partial) {
            // only the absmax of a (the cast pass recomputes a from the stored H); the block-scaled
            // path has no per-tensor scale and skips it
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (row_ok && j < ncol) amax = max(amax, abs_bits(swiglu_fast(hg[j], hu[j])));
          }
        }
      } else if (p.epi == kEpiSwigluBwd) {
        // the next chunk's H words are in flight while the current chunk is computed (the
        // first chunk's were requested before the accumulator wait)
        const int col0 = nb * BN;
#pragma unroll 1
        for (int c = 4 * half; c < 4 * half + 4; ++c) {
          uint4 hc[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) hc[q] = hn[q];
          const int col = col0 + c * 32;
          if (c + 1 < 4 * half + 4 && row_ok && col + 32 < p.N) load_h_chunk(p, row, col + 32, min(32, p.N - col - 32), hn);
          uint32_t acc32[32];
          tmem_ld32(tbase + c * 32, acc32);
          const int ncol = min(32, p.N - col);
          if (!warp_ok || ncol <= 0) continue;
          float dg[32], du[32];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t gw[4] = {hc[q].x, hc[q].y, hc[q].z, hc[q].w};
            const uint32_t uw[4] = {hc[4 + q].x, hc[4 + q].y, hc[4 + q].z, hc[4 + q].w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int j = 8 * q + k;
              const float h = (k & 1) ? bf16_hi(gw[k >> 1]) : bf16_lo(gw[k >> 1]);
              const float u = (k & 1) ? bf16_hi(uw[k >> 1]) : bf16_lo(uw[k >> 1]);
              swiglu_bwd1(__fmul_rn(alpha, __uint_as_float(acc32[j])), h, u, dg[j], du[j]);
              if (row_ok && j < ncol) amax = max(amax, max(abs_bits(dg[j]), abs_bits(du[j])));
            }
          }
          staging_acquire(lane);
          stage_bf16(buf, lane, dg);
          stage_bf16(buf + 2048, lane, du);
          staging_publish();
          if (lane == 0) {
            tma_store_2d(&tmC, buf, col, row0);
            tma_store_2d(&tmC2, buf + 2048, col, row0);
            bulk_commit();
          }
        }
      } else {
        const int col0 = nb * BN;
#pragma unroll 1
        for (int c = 4 * half; c < 4 * half + 4; ++c) {
          uint32_t acc32[32];
          tmem_ld32(tbase + c * 32, acc32);
          const int col = col0 + c * 32;
          const int ncol = min(32, p.N - col);
          if (!warp_ok || ncol <= 0) continue;
          float v[32];
          if (p.out_f32) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(alpha, __uint_as_float(acc32[j]));
          } else if (p.epi == kEpiResidual) {
            // bf16(r + alpha * acc) as one rounding of the exact sum
            float rv[32];
            const uint16_t* r = p.R + (int64_t)row * p.ldr + col;
            if (row_ok && ncol == 32) {
              load_bf16x32(r, rv);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) rv[j] = (row_ok && j < ncol) ? __uint_as_float((uint32_t)r[j] << 16) : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = bf16_of_residual(rv[j], alpha, __uint_as_float(acc32[j]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = bf16_of_product(alpha, __uint_as_float(acc32[j]));
          }
          staging_acquire(lane);
          if (p.out_f32) stage_f32(buf, lane, v);
          else stage_bf16(buf, lane, v);
          staging_publish();
          if (lane == 0) {
            tma_store_2d(&tmC, buf, col, row0);
            bulk_commit();
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0) bulk_wait_all();  // every TMA store of this warp has completed
    amax = warp_max_u32(amax);
    if (lane == 0) atomicMax(cta_amax, amax);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0 && p.amax_partial) p.amax_partial[blockIdx.x] = *cta_amax;
  if (warp == 2) tmem_dealloc(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------
// The wide variant for the long-K GEMMs with plain epilogues (store, residual):
// a 256 x 256 CTA tile made of two 128-row halves that share the B tile (two
// tcgen05.mma per k-step into two accumulators, all 512 TMEM columns), so a
// stage moves 64 KB for twice the MMA work of a 48 KB 128 x 256 stage -- a
// third fewer operand bytes per FLOP reaching the SM, which is what bounds the
// 128 x 256 mainloop.  The price: no second accumulator, so the epilogue of a
// tile does not overlap the next tile's MMAs; with K >= kWideMinK the MMAs of
// a tile take 10x or more the epilogue's time.  launch_gemm picks it per GEMM
// by the estimate in wide_pays (wave quantization included).
// ---------------------------------------------------------------------------
constexpr int kWideStages = 3;
constexpr int kWideStage = 2 * kATile + 2 * kBHalf;  // 64 KB
constexpr int kWideStagingOffset = kWideStages * kWideStage;
constexpr int kWideBarOffset = kWideStagingOffset + 8 * kStagingBytes;
constexpr int kWideSmemBytes = kWideBarOffset + 256 + 1024;
static_assert(kWideSmemBytes <= 232448, "shared memory per CTA");
constexpr int kWideMinK = 8192;

// Whether the wide tile is expected to finish first.  A wide tile does the work of two 128 x 256
// tiles in ~0.86 of their time (measured on the 7B-class GEMMs: a third fewer operand bytes per
// FLOP) plus its exposed epilogue (~5 us against 2 * 256 * 256 * K flops at ~23 TFLOP/s per SM);
// both variants run in waves of one tile per SM, so the last, partial wave decides as much as the
// per-tile speed.
bool wide_pays(int64_t M, int n_tiles, int64_t K, int num_sms) {
  const int64_t tiles_w = (M + 255) / 256 * n_tiles, tiles_n = (M + 127) / 128 * n_tiles;
  const double waves_w = (double)((tiles_w + num_sms - 1) / num_sms);
  const double waves_n = (double)((tiles_n + num_sms - 1) / num_sms);
  const double epi = 5e-6 * 23e12 / (2.0 * 256 * 256 * (double)K);
  return waves_w * 2.0 * 0.86 * (1.0 + epi) < waves_n;
}

template <int A_MN, int B_MN>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_f8_wide(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const Args p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kWideBarOffset);
  uint64_t* empty = full + kWideStages;
  uint64_t* tfull = empty + kWideStages;  // [1]
  uint64_t* tempty = tfull + 1;           // [1]
  uint64_t* drain = tempty + 1;           // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kWideStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    mbar_init(tfull, 1);
    mbar_init(tempty, kEpiThreads);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 2) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, p, mb, nb);
        const int m0 = mb * 256;
        const int n0 = nb * p.b_step, n1 = n0 + p.b_half1;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.wait_ns)) { ok = false; break; }
          uint8_t* sA = smem + stage * kWideStage;
          uint8_t* sB = sA + 2 * kATile;
          mbar_arrive_expect_tx(&full[stage], kWideStage);
          const int k0 = kb * BK;
          if (A_MN) {
            tma_load_2d(sA, &tmA, &full[stage], m0, k0);
            tma_load_2d(sA + kATile, &tmA, &full[stage], m0 + 128, k0);
          } else {
            tma_load_2d(sA, &tmA, &full[stage], k0, m0);
            tma_load_2d(sA + kATile, &tmA, &full[stage], k0, m0 + 128);
          }
          if (B_MN) {
            tma_load_2d(sB, &tmB, &full[stage], n0, k0);
            tma_load_2d(sB + kBHalf, &tmB, &full[stage], n1, k0);
          } else {
            tma_load_2d(sB, &tmB, &full[stage], k0, n0);
            tma_load_2d(sB + kBHalf, &tmB, &full[stage], k0, n1);
          }
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kWideStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
        for (int s = 0; s < kWideStages; ++s)
          if (issued & (1u << s)) {
            int dummy = 0;
            mbar_wait(&full[s], (issued_par >> s) & 1u, &dummy);
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: two 128 x 256 x 32 MMAs per k-step ----------------
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
        if (!mbar_wait(tempty, acc_phase ^ 1u, abort_flag, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sA = smem_addr(smem + stage * kWideStage);
          const uint32_t sB = sA + 2 * kATile;
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            const uint64_t bd = B_MN ? smem_desc_sw128(sB + kk * 4096, kBHalf, 1024) : smem_desc_sw128(sB + kk * 32, 16, 1024);
#pragma unroll
            for (int hm = 0; hm < 2; ++hm) {
              const uint32_t a = sA + hm * kATile;
              const uint64_t ad = A_MN ? smem_desc_sw128(a + kk * 4096, kBHalf, 1024) : smem_desc_sw128(a + kk * 32, 16, 1024);
              umma_f8(tmem_base + hm * BN, ad, bd, p.idesc, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          umma_commit(&empty[stage]);
          if (++stage == kWideStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(tfull);
        acc_phase ^= 1u;
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
    // ---------------- epilogue: warpgroup hm drains accumulator hm (rows 128 hm ..) ----------------
    const int sub = warp & 3;
    const int hm = (warp - 4) >> 2;
    const uint32_t buf = smem_addr(smem + kWideStagingOffset + (warp - 4) * kStagingBytes);
    uint32_t acc_phase = 0;
    const float alpha = __fmul_rn(*p.sinvA, *p.sinvB);
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      int mb, nb;
      tile_coords(tile, p, mb, nb);
      const int row0 = mb * 256 + hm * 128 + sub * 32;
      const int row = row0 + lane;
      const bool row_ok = row < p.M;
      const bool warp_ok = row0 < p.M;
      const int col0 = nb * BN;
      // The residual is requested before the accumulator is ready (this epilogue does not overlap
      // the next tile's MMAs, so its read latency would be exposed): the L2 lines of the lane's
      // row segment, and the first chunk's words into registers; chunk c + 1's words are then in
      // flight while chunk c is computed.
      const bool res = !p.out_f32 && p.epi == kEpiResidual;
      uint4 rn[4];
      if (res && row_ok && col0 < p.N) {
        const uint16_t* r = p.R + (int64_t)row * p.ldr + col0;
        prefetch_l2_span(r, 2 * min(BN, p.N - col0));
        if (p.N - col0 >= 32)
#pragma unroll
          for (int q = 0; q < 4; ++q) rn[q] = ld_v4(r + 8 * q);
      }
      int full_ok = 0;
      if (lane == 0) full_ok = mbar_wait(tfull, acc_phase, abort_flag, p.wait_ns) ? 1 : 0;
      if (!__shfl_sync(0xFFFFFFFFu, full_ok, 0)) {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + (uint32_t)(hm * BN) + ((uint32_t)(sub * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t acc32[32];
        tmem_ld32(tbase + c * 32, acc32);
        const int col = col0 + c * 32;
        const int ncol = min(32, p.N - col);
        uint4 rc[4];
        if (res) {
#pragma unroll
          for (int q = 0; q < 4; ++q) rc[q] = rn[q];
          if (c + 1 < BN / 32 && row_ok && p.N - (col + 32) >= 32) {
            const uint16_t* r = p.R + (int64_t)row * p.ldr + col + 32;
#pragma unroll
            for (int q = 0; q < 4; ++q) rn[q] = ld_v4(r + 8 * q);
          }
        }
        if (!warp_ok || ncol <= 0) continue;
        float v[32];
        if (p.out_f32) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(alpha, __uint_as_float(acc32[j]));
        } else if (p.epi == kEpiResidual) {
          float rv[32];
          const uint16_t* r = p.R + (int64_t)row * p.ldr + col;
          if (row_ok && ncol == 32) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t ww[4] = {rc[q].x, rc[q].y, rc[q].z, rc[q].w};
#pragma unroll
              for (int k = 0; k < 4; ++k) { rv[8 * q + 2 * k] = bf16_lo(ww[k]); rv[8 * q + 2 * k + 1] = bf16_hi(ww[k]); }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) rv[j] = (row_ok && j < ncol) ? __uint_as_float((uint32_t)r[j] << 16) : 0.0f;
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = bf16_of_residual(rv[j], alpha, __uint_as_float(acc32[j]));
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = bf16_of_product(alpha, __uint_as_float(acc32[j]));
        }
        staging_acquire(lane);
        if (p.out_f32) stage_f32(buf, lane, v);
        else stage_bf16(buf, lane, v);
        staging_publish();
        if (lane == 0) {
          tma_store_2d(&tmC, buf, col, row0);
          bulk_commit();
        }
      }
      tc_fence_before();
      mbar_arrive(tempty);
      acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_all();  // every TMA store of this warp has completed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
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

// 2D operand [outer, inner] with row stride `ld` elements, 128-byte-swizzled boxes 128 bytes
// wide: FP8 (es = 1) 128 x 128 elements; bf16 (es = 2) 64 elements x `box_outer` rows
// (128 for a K-major operand, 64 = the K rows of one stage for an MN-major one).
bool make_tmap(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int64_t ld, int es = 1,
               int box_outer = 128) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  const cuuint64_t strides[1] = {(cuuint64_t)(ld * es)};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / es), (cuuint32_t)box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
             const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output tensor [rows, cols] (row stride ld elements) stored in 32 x 32 element
// boxes: bf16 boxes are 64 B wide (64-byte swizzle), fp32 boxes 128 B wide
// (128-byte swizzle), uint8 boxes 32 B wide (32-byte swizzle), matching
// stage_bf16 / stage_f32 / stage_u8.
enum OutKind { kOutBf16, kOutF32, kOutU8 };
bool make_out_tmap(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t ld, OutKind kind) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const int64_t es = kind == kOutF32 ? 4 : (kind == kOutBf16 ? 2 : 1);
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(ld * es)};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = kind == kOutF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : kind == kOutBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle sw = kind == kOutF32 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : kind == kOutBf16 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                   : CU_TENSOR_MAP_SWIZZLE_32B;
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Instruction descriptor for kind::f8f6f4 and kind::f16: fp32 accumulator, A/B
// formats (f8f6f4: E4M3 = 0, E5M2 = 1; f16: bf16 = 1), operand major-ness
// (bit 15 A, bit 16 B; 1 = MN-major), N >> 3 at bit 17, M >> 4 at bit 24.
uint32_t make_idesc(int fmtA, int fmtB, int a_mn, int b_mn) {
  return (1u << 4) | ((uint32_t)fmtA << 7) | ((uint32_t)fmtB << 10) | ((uint32_t)a_mn << 15) |
         ((uint32_t)b_mn << 16) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}
// Instruction descriptor for kind::mxf8f6f4.block_scale: A/B formats, major-ness, N >> 3, M >> 4 as
// above; bit 23 = the scale type E8M0; the accumulator is fp32 by definition, and bits 4-5 / 29-30
// are the per-MMA scale-factor ids (mx_sf_ids), left zero here.
uint32_t make_idesc_mx(int fmtA, int fmtB, int a_mn, int b_mn) {
  return ((uint32_t)fmtA << 7) | ((uint32_t)fmtB << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(BN >> 3) << 17) | (1u << 23) | ((uint32_t)(BM >> 4) << 24);
}

template <int A_MN, int B_MN, int OP16, int MX>
cudaError_t configure_t() {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_f8<A_MN, B_MN, OP16, MX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Plan<MX>::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return cudaSuccess;
}

template <int A_MN, int B_MN, int OP16, int MX = 0>
cudaError_t launch_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tc2,
                     const CUtensorMap& taux, const Args& a, int grid, cudaStream_t s) {
  cudaError_t e = configure_t<A_MN, B_MN, OP16, MX>();
  if (e != cudaSuccess) return e;
  k_gemm_f8<A_MN, B_MN, OP16, MX><<<grid, kThreads, Plan<MX>::kSmemBytes, s>>>(ta, tb, tc, tc2, taux, a);
  return cudaGetLastError();
}

template <int A_MN, int B_MN>
cudaError_t launch_wide_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const Args& a, int grid,
                          cudaStream_t s) {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_f8_wide<A_MN, B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kWideSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  k_gemm_f8_wide<A_MN, B_MN><<<grid, kThreads, kWideSmemBytes, s>>>(ta, tb, tc, a);
  return cudaGetLastError();
}

// The rasterisation group of a GEMM, in M units of unit_rows rows.  A group walks its M units for
// each N tile in turn, so its A rows are re-read from L2 while B passes once per group.  When all of
// A fits comfortably in L2 (and is the smaller operand), one group spanning every M unit reads each
// operand byte from DRAM once; when B does instead, groups of one M unit walk N fastest and keep B
// resident; otherwise groups of kGroupRows rows bound A's share of L2.  "Comfortably": 48 MB or
// less (a 96 MB A measured slower: the streamed B and the output evict it), and no epilogue
// side input as large as the output streaming through L2 beside it (the SwiGLU backward reads H,
// 2 x 2 bytes per output element: with a resident 29 MB A its DRAM reads grew by 92 MB per launch).
int raster_group(int64_t a_bytes, int64_t b_bytes, int m_units, int unit_rows, bool side_stream) {
  constexpr int64_t kResident = 48ll << 20;
  if (!side_stream && a_bytes <= b_bytes && a_bytes <= kResident) return m_units;
  if (!side_stream && b_bytes < a_bytes && b_bytes <= kResident) return 1;
  const int g = kGroupRows / unit_rows;
  return g < 1 ? 1 : g;
}

}  // namespace

cudaError_t launch_gemm(const GemmProblem& g, int* P, const Launch& L) {
  Args a{};
  a.M = g.M;
  a.N = g.N;
  a.K = g.K;
  a.epi = g.epi;
  a.out_f32 = g.out_f32;
  a.sinvA = g.sinvA;
  a.sinvB = g.sinvB;
  a.C = g.C;
  a.ldc = g.ldc;
  a.R = g.R;
  a.ldr = g.ldr;
  a.aux16 = g.op16 ? g.a16 : nullptr;
  a.qscale = g.op16 ? nullptr : g.qscale;
  a.amax_partial = g.amax_partial;
  a.status = L.status;
  a.idesc = g.op16 ? make_idesc(1, 1, g.a_mn, g.b_mn)
                   : (g.mx ? make_idesc_mx(g.fmtA, g.fmtB, g.a_mn, g.b_mn) : make_idesc(g.fmtA, g.fmtB, g.a_mn, g.b_mn));
  if (g.mx) {
    if (g.op16 || g.K % 128 != 0 || !g.sfA || !g.sfB) return cudaErrorInvalidValue;
    a.sinvA = a.sinvB = nullptr;  // alpha = 1: the block scales are part of the operands
    a.sfA = g.sfA;
    a.sfB = g.sfB;
    a.sf_kc = g.K / 128;
  }
  a.b_cols = (int)g.b_cols;
  a.wait_ns = g.wait_ns ? g.wait_ns : kWaitLimitNs;
  a.m_tiles = (g.M + BM - 1) / BM;
  if (g.epi == kEpiSwiglu) {
    a.n_tiles = (g.N + 127) / 128;  // 128 gate + the matching 128 up columns per tile
    a.b_step = 128;
    a.b_half1 = g.N;
  } else {
    a.n_tiles = (g.N + BN - 1) / BN;
    a.b_step = BN;
    a.b_half1 = 128;
  }
  const int bk = g.op16 ? BK / 2 : BK;  // K elements per stage
  a.k_blocks = (g.K + bk - 1) / bk;
  a.num_tiles = a.m_tiles * a.n_tiles;

  CUtensorMap ta, tb, tc, tc2, taux;
  const int es = g.op16 ? 2 : 1;
  const int mn_rows = g.op16 ? 64 : 128;  // K rows of an MN-major box
  const bool ok_a = g.a_mn ? make_tmap(&ta, g.A, g.M, g.K, g.lda, es, mn_rows) : make_tmap(&ta, g.A, g.K, g.M, g.lda, es);
  const bool ok_b = g.b_mn ? make_tmap(&tb, g.B, g.b_cols, g.K, g.ldb, es, mn_rows)
                           : make_tmap(&tb, g.B, g.K, g.b_cols, g.ldb, es);
  bool ok_c;
  if (g.epi == kEpiSwiglu || g.epi == kEpiSwigluBwd) {
    // gate half [M, f] and up half [M, f] of the [M, 2f] output, each clipped at f
    const uint16_t* c = static_cast<const uint16_t*>(g.C);
    ok_c = make_out_tmap(&tc, c, g.N, g.M, g.ldc, kOutBf16) && make_out_tmap(&tc2, c + g.N, g.N, g.M, g.ldc, kOutBf16);
    taux = tc;
    if (ok_c && g.op16 && g.a16) ok_c = make_out_tmap(&taux, g.a16, g.N, g.M, g.N, kOutBf16);
    else if (ok_c && g.qscale && g.q8) ok_c = make_out_tmap(&taux, g.q8, g.N, g.M, g.N, kOutU8);
  } else {
    ok_c = make_out_tmap(&tc, g.C, g.N, g.M, g.ldc, g.out_f32 ? kOutF32 : kOutBf16);
    tc2 = taux = tc;
  }
  if (!ok_a || !ok_b || !ok_c) return cudaErrorInvalidValue;

  // long-K FP8 GEMMs with plain epilogues take the 256 x 256 tile
  const bool wide = !g.op16 && !g.mx && (g.epi == kEpiStore || g.epi == kEpiResidual) && g.K >= kWideMinK && g.M >= 256 &&
                    wide_pays(g.M, a.n_tiles, g.K, L.num_sms);
  if (wide) {
    a.m_tiles = (g.M + 255) / 256;
    a.num_tiles = a.m_tiles * a.n_tiles;
  }
  a.m_units = a.m_tiles;
  a.num_tiles = a.m_units * a.n_tiles;
  const int grid = a.num_tiles < L.num_sms ? a.num_tiles : L.num_sms;
  const int64_t es_bytes = g.op16 ? 2 : 1;
  a.group = raster_group((int64_t)g.M * g.K * es_bytes, (int64_t)g.b_cols * g.K * es_bytes, a.m_units,
                         wide ? 256 : BM, g.epi == kEpiSwigluBwd);
  *P = grid;
  cudaError_t e;
  if (wide) {
    if (g.a_mn == 0 && g.b_mn == 1) e = launch_wide_t<0, 1>(ta, tb, tc, a, grid, L.stream);
    else if (g.a_mn == 0 && g.b_mn == 0) e = launch_wide_t<0, 0>(ta, tb, tc, a, grid, L.stream);
    else if (g.a_mn == 1 && g.b_mn == 1) e = launch_wide_t<1, 1>(ta, tb, tc, a, grid, L.stream);
    else return cudaErrorInvalidValue;
    if (L.launches) ++*L.launches;
    return e;
  }
  if (g.mx) {  // the three layouts of the block (NN, NT, TN)
    if (g.a_mn == 0 && g.b_mn == 1) e = launch_t<0, 1, 0, 1>(ta, tb, tc, tc2, taux, a, grid, L.stream);
    else if (g.a_mn == 0 && g.b_mn == 0) e = launch_t<0, 0, 0, 1>(ta, tb, tc, tc2, taux, a, grid, L.stream);
    else if (g.a_mn == 1 && g.b_mn == 1) e = launch_t<1, 1, 0, 1>(ta, tb, tc, tc2, taux, a, grid, L.stream);
    else return cudaErrorInvalidValue;
  } else if (g.op16) {  // the three layouts of the block (NN, NT, TN)
    if (g.a_mn == 0 && g.b_mn == 1) e = launch_t<0, 1, 1>(ta, tb, tc, tc2, taux, a, grid, L.stream);
    else if (g.a_mn == 0 && g.b_mn == 0) e = launch_t<0, 0, 1>(ta, tb, tc, tc2, taux, a, grid, L.stream);
    else if (g.a_mn == 1 && g.b_mn == 1) e = launch_t<1, 1, 1>(ta, tb, tc, tc2, taux, a, grid, L.stream);
    else return cudaErrorInvalidValue;
  } else {
    if (g.a_mn == 0 && g.b_mn == 1) e = launch_t<0, 1, 0>(ta, tb, tc, tc2, taux, a, grid, L.stream);
    else if (g.a_mn == 0 && g.b_mn == 0) e = launch_t<0, 0, 0>(ta, tb, tc, tc2, taux, a, grid, L.stream);
    else if (g.a_mn == 1 && g.b_mn == 1) e = launch_t<1, 1, 0>(ta, tb, tc, tc2, taux, a, grid, L.stream);
    else e = launch_t<1, 0, 0>(ta, tb, tc, tc2, taux, a, grid, L.stream);
  }
  if (L.launches) ++*L.launches;
  return e;
}

}  // namespace fp8q
