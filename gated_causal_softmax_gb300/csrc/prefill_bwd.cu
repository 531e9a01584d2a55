// Prefill backward, single pass: dQ is folded into the dK/dV pass
// (fla-org/flash-linear-attention #1322 "Gluon attention backend with large head
// dimensions": Oct 5 comment -- each score and dP tile is computed once, dQ partials
// accumulate into a zero-initialised fp32 buffer that is converted afterwards, gate and
// sink partials use fp32 reductions; Oct 3 comment -- probabilities recomputed in fp32).
//
// One CTA per (128-key tile, kv head); it loops over the query heads of its GQA group and
// over 64-row query tiles in the causal / window range.  Per query tile:
//     S^T  = K Q^T            (TMEM, fp32)        P^T  = 2^(S^T*scale*log2e + G_i - G_j - LSE_i)
//     dP^T = V dO^T           (TMEM, fp32)        dS^T = P^T o (dP^T - delta_i)
//     dV  += P^T dO           (A operand = P^T in TMEM, bf16)
//     dK  += dS^T Q           (A operand = dS^T in TMEM, bf16)
//     dQ^T = K^T dS^T         (dS^T staged in shared memory, bf16) -> fp32 bulk reduce-add
// plus fp32 row / column sums of dS for the gate and sink gradients.
//
// Warp roles (192 threads): warp 0 TMA producer (K/V once, Q/dO tiles double-buffered,
// per-column LSE / delta / gate vectors), warp 1 tcgen05 issuer, warps 2..5 one thread
// per key row (TMEM lane).
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace gcs {
namespace {

constexpr int kBN = 128;  // keys per CTA (TMEM lanes)
constexpr int kBM = 64;   // query rows per step
constexpr int kThreads = 192;
constexpr int kKVChunk = 128 * 128;  // 128 rows x 64 bf16
constexpr int kQChunk = 64 * 128;    // 64 rows x 64 bf16
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

template <int DQK, int DV>
struct BwdCfg {
  static constexpr int KCH = DQK / 64;
  static constexpr int VCH = DV / 64;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KCH * kKVChunk;
  static constexpr int OFF_Q = OFF_V + VCH * kKVChunk;          // [2][KCH] q chunks
  static constexpr int OFF_DO = OFF_Q + 2 * KCH * kQChunk;      // [2][VCH] dO chunks
  static constexpr int OFF_DS = OFF_DO + 2 * VCH * kQChunk;     // 128 rows x 64 bf16
  static constexpr int STG_BYTES = kBM * DQK * 4;               // fp32 dQ staging tile
  static constexpr int OFF_STG = OFF_DS + kKVChunk;             // [2] staging tiles
  static constexpr int OFF_VEC = OFF_STG + 2 * STG_BYTES;       // [2][3][64] floats
  static constexpr int OFF_BAR = OFF_VEC + 2 * 3 * kBM * 4;
  static constexpr int NBAR = 16;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  // TMEM columns
  static constexpr int T_S = 0, T_DP = 64, T_DQ = 128, T_DV = 192, T_DK = 192 + DV;
  static_assert(T_DK + DQK <= 512, "TMEM budget");
};

__device__ __forceinline__ bool find_kv_tile(const int32_t* cu, int num_seqs, int t, int& start, int& len, int& jt) {
  for (int s = 0; s < num_seqs; ++s) {
    const int a = __ldg(cu + s), b = __ldg(cu + s + 1);
    const int n = (b - a + kBN - 1) / kBN;
    if (t < n) {
      start = a;
      len = b - a;
      jt = t;  // early key tiles see the most queries: hand them out first
      return true;
    }
    t -= n;
  }
  return false;
}

__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

template <int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const BwdParams p) {
  using C = BwdCfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  int seq_start, len, jt;
  if (!find_kv_tile(p.cu_seqlens, p.num_seqs, blockIdx.x, seq_start, len, jt)) return;
  const int kvh = blockIdx.y;
  const int group = p.hq / p.hkv;
  const int j0 = jt * kBN;
  // query tiles that see any key of this tile: i >= j0 (causal), i < j0 + 127 + W (window)
  const int it_lo = j0 / kBM;
  int i_hi = len - 1;
  if (p.window > 0) i_hi = min(i_hi, j0 + kBN - 1 + p.window - 1);
  const int it_hi = i_hi / kBM;
  const int n_it = it_hi - it_lo + 1;
  const int nsteps = n_it * group;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;    // [2]
  uint64_t* q_empty = bars + 3;   // [2]
  uint64_t* s_full = bars + 5;
  uint64_t* p_full = bars + 6;
  uint64_t* mma_done = bars + 7;
  uint64_t* dq_free = bars + 8;
  uint64_t* stg_full = bars + 9;  // [2]
  uint64_t* stg_free = bars + 11; // [2]
  uint64_t* drain = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const Abort ab{abort_flag, p.status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&q_full[b], 2);
      mbar_init(&q_empty[b], 1);
      mbar_init(&stg_full[b], 128);
      mbar_init(&stg_free[b], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 4);
    mbar_init(mma_done, 1);
    mbar_init(dq_free, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmDO);
      mbar_expect_tx(kv_full, (C::KCH + C::VCH) * kKVChunk);
      for (int c = 0; c < C::KCH; ++c)
        tma_load_2d(smem + C::OFF_K + c * kKVChunk, &tmK, kv_full, kvh * DQK + c * 64, seq_start + j0);
      for (int c = 0; c < C::VCH; ++c)
        tma_load_2d(smem + C::OFF_V + c * kKVChunk, &tmV, kv_full, kvh * DV + c * 64, seq_start + j0);
    }
    const uint64_t pol = l2_policy_evict_last();
    for (int s = 0; s < nsteps && ok; ++s) {
      const int b = s & 1;
      const int h = kvh * group + s / n_it;
      const int i0 = (it_lo + s % n_it) * kBM;
      if (lane == 0) {
        ok = wait_bar(&q_empty[b], ((s >> 1) & 1) ^ 1, ab);
        if (ok) {
          mbar_expect_tx(&q_full[b], (C::KCH + C::VCH) * kQChunk);
          for (int c = 0; c < C::KCH; ++c)
            tma_load_2d_hint(smem + C::OFF_Q + (b * C::KCH + c) * kQChunk, &tmQ, &q_full[b], h * DQK + c * 64,
                             seq_start + i0, pol);
          for (int c = 0; c < C::VCH; ++c)
            tma_load_2d_hint(smem + C::OFF_DO + (b * C::VCH + c) * kQChunk, &tmDO, &q_full[b], h * DV + c * 64,
                             seq_start + i0, pol);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      // per-column vectors: [0] G_i - LSE_i (log2 units), [1] delta_i, both for i0 .. i0+63
      float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC) + b * 3 * kBM;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = lane * 2 + u;
        const int i = i0 + c;
        float colterm = 0.f, dl = 0.f;
        if (i < len) {
          const size_t idx = (size_t)h * p.total + seq_start + i;
          colterm = -__ldg(p.lse + idx) * kLog2e;
          if (p.gT) colterm += __ldg(p.gT + idx);
          dl = __ldg(p.delta + idx);
        }
        vec[c] = colterm;
        vec[kBM + c] = dl;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full[b]);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16(128, kBM, false, false);   // S^T, dP^T
      const uint32_t idDV = idesc_bf16(128, DV, false, true);    // dV += P^T dO
      const uint32_t idDK = idesc_bf16(128, DQK, false, true);   // dK += dS^T Q
      const uint32_t idDQ = idesc_bf16(128, kBM, true, true);    // dQ^T = K^T dS^T
      const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q), sDO = smem_u32(smem + C::OFF_DO);
      const uint32_t sDS = smem_u32(smem + C::OFF_DS);
      bool ok = wait_bar(kv_full, 0, ab);
      for (int s = 0; s < nsteps && ok; ++s) {
        const int b = s & 1;
        ok = wait_bar(&q_full[b], (s >> 1) & 1, ab);
        if (!ok) break;
        if (s > 0) {
          // S^T / dP^T columns still hold the previous step's P^T / dS^T operands
          ok = wait_bar(mma_done, (s - 1) & 1, ab);
          if (!ok) break;
        }
        tc_fence_after();
        const uint32_t qb = sQ + b * C::KCH * kQChunk, dob = sDO + b * C::VCH * kQChunk;
        for (int c = 0; c < C::KCH; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + C::T_S, sdesc_sw128(sK + c * kKVChunk + k * 32, 16, 1024),
                   sdesc_sw128(qb + c * kQChunk + k * 32, 16, 1024), idS, (c | k) != 0);
        for (int c = 0; c < C::VCH; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + C::T_DP, sdesc_sw128(sV + c * kKVChunk + k * 32, 16, 1024),
                   sdesc_sw128(dob + c * kQChunk + k * 32, 16, 1024), idS, (c | k) != 0);
        mma_commit(s_full);
        ok = wait_bar(p_full, s & 1, ab);
        if (!ok) break;
        tc_fence_after();
        // K dimension = 64 query rows = 4 steps of 16 rows (2048 B in the MN-major views)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts(tmem + C::T_DV, tmem + C::T_S + k * 8, sdesc_sw128(dob + k * 2048, kQChunk, 1024), idDV,
                 (s > 0 || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts(tmem + C::T_DK, tmem + C::T_DP + k * 8, sdesc_sw128(qb + k * 2048, kQChunk, 1024), idDK,
                 (s > 0 || k > 0) ? 1u : 0u);
        if (s > 0) {
          ok = wait_bar(dq_free, (s - 1) & 1, ab);
          if (!ok) break;
          tc_fence_after();
        }
        // dQ^T: M = 128 rows of K^T (DQK = 64 pads rows 64..127 with the V tile; ignored)
        const uint32_t lboK = (DQK >= 128) ? kKVChunk : (C::OFF_V - C::OFF_K);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss(tmem + C::T_DQ, sdesc_sw128(sK + k * 2048, lboK, 1024), sdesc_sw128(sDS + k * 2048, kKVChunk, 1024),
                 idDQ, k > 0);
        mma_commit(mma_done);
        mma_commit(&q_empty[b]);
      }
      if (!ok) {
        mma_commit(drain);
        mbar_wait(drain, 0, nullptr);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ key rows
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int jl = j0 + r;
    const bool has_gate = p.gT != nullptr;
    const bool want_row = p.dg_row != nullptr;
    const float gj = (has_gate && jl < len) ? __ldg(p.gT + (size_t)(kvh * group) * p.total + seq_start + jl) : 0.f;
    float rowterm = -gj;
    float dgcol = 0.f;
    bool ok = true;
    uint8_t* sDS = smem + C::OFF_DS;
    for (int s = 0; s < nsteps; ++s) {
      const int b = s & 1;
      const int hi = s / n_it;
      const int h = kvh * group + hi;
      const int i0 = (it_lo + s % n_it) * kBM;
      if (s % n_it == 0 && s > 0) {
        // new query head: flush the column sums of dS of the previous head, reload G_j
        if (has_gate && jl < len) p.dg_col[(size_t)(h - 1) * p.total + seq_start + jl] = dgcol;
        dgcol = 0.f;
        rowterm = (has_gate && jl < len) ? -__ldg(p.gT + (size_t)h * p.total + seq_start + jl) : 0.f;
      }
      ok = wait_bar(&q_full[b], (s >> 1) & 1, ab);
      if (!ok) break;
      ok = wait_bar(s_full, s & 1, ab);
      if (!ok) break;
      tc_fence_after();
      uint32_t sv[64], dp[64];
      tmem_ld32(tmem + lane_off + C::T_S, sv);
      tmem_ld32(tmem + lane_off + C::T_S + 32, sv + 32);
      tmem_ld32(tmem + lane_off + C::T_DP, dp);
      tmem_ld32(tmem + lane_off + C::T_DP + 32, dp + 32);
      tmem_ld_wait();
      const float* vec = reinterpret_cast<const float*>(smem + C::OFF_VEC) + b * 3 * kBM;
      const bool need_mask = (i0 < j0 + kBN - 1) || (p.window > 0 && i0 + kBM - 1 - j0 >= p.window) ||
                             (i0 + kBM > len);
      // P (fp32) and dS (fp32) for this key row against 64 query columns
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        float t = fmaf(__uint_as_float(sv[c]), p.scale_log2, vec[c]) + rowterm;
        if (need_mask) {
          const int i = i0 + c;
          const bool vis = (i < len) && (jl <= i) && (p.window == 0 || i - jl < p.window);
          t = vis ? t : neg_inf();
        }
        const float pr = ex2(t);
        const float ds = pr * (__uint_as_float(dp[c]) - vec[kBM + c]);
        sv[c] = __float_as_uint(pr);
        dp[c] = __float_as_uint(ds);
      }
      // P^T and dS^T as bf16 MMA operands in TMEM (over the consumed score columns)
      {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1]));
        tmem_st32(tmem + lane_off + C::T_S, pk);
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(__uint_as_float(dp[2 * c]), __uint_as_float(dp[2 * c + 1]));
        tmem_st32(tmem + lane_off + C::T_DP, pk);
        // dS^T row r (64 bf16 = 128 B) into the 128-B-swizzled operand tile for dQ^T; the
        // previous step's dQ^T MMA finished reading it (mma_done was waited in its drain)
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(sDS + sw128_offset(r, q)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
      // fp32 sums of dS: over this row's query columns (column sum of dS for key j) ...
      if (has_gate) {
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) acc += __uint_as_float(dp[c]);
        dgcol += acc;
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      // ... and over the 128 key rows for each query column (row sum of dS for query i):
      // transpose-reduce within the warp, lane l ends with columns 2l, 2l+1
      if (want_row) {
        float v[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) v[c] = __uint_as_float(dp[c]);
#pragma unroll
        for (int half = 32; half >= 2; half >>= 1) {
          const bool upper = (lane & (half >> 1)) != 0;
#pragma unroll
          for (int c = 0; c < half; ++c) {
            const float send = upper ? v[c] : v[c + half];
            const float keep = upper ? v[c + half] : v[c];
            v[c] = keep + __shfl_xor_sync(0xffffffffu, send, half >> 1);
          }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = i0 + 2 * lane + e;
          if (i < len) atomicAdd(p.dg_row + (size_t)h * p.total + seq_start + i, v[e]);
        }
      }
      // ---- drain dQ^T of this step: TMEM -> registers -> fp32 staging tile -> bulk reduce-add
      ok = wait_bar(mma_done, s & 1, ab);
      if (!ok) break;
      tc_fence_after();
      uint32_t dq[64];
      tmem_ld32(tmem + lane_off + C::T_DQ, dq);
      tmem_ld32(tmem + lane_off + C::T_DQ + 32, dq + 32);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free);
      ok = wait_bar(&stg_free[b], ((s >> 1) & 1) ^ 1, ab);
      if (!ok) break;
      float* stg = reinterpret_cast<float*>(smem + C::OFF_STG + b * C::STG_BYTES);
      if (r < DQK) {
#pragma unroll
        for (int c = 0; c < 64; ++c) stg[c * DQK + r] = __uint_as_float(dq[c]) * p.scale;
      }
      fence_proxy_async_smem();
      mbar_arrive(&stg_full[b]);
      if (threadIdx.x == 64) {
        // one thread issues the reduce-adds of the valid query rows of this step
        ok = wait_bar(&stg_full[b], (s >> 1) & 1, ab);
        if (ok) {
          const int nrows = min(kBM, len - i0);
          for (int c = 0; c < nrows; ++c)
            bulk_reduce_add_f32(p.dq_acc + ((size_t)(seq_start + i0 + c) * p.hq + h) * DQK, stg + c * DQK, DQK * 4);
          bulk_commit();
          // the other buffer's reduce-adds (previous step) have read their source by now
          bulk_wait_read<1>();
          if (s > 0) mbar_arrive(&stg_free[b ^ 1]);
        }
      }
      if (!ok) break;
    }
    if (threadIdx.x == 64) bulk_wait<0>();
    if (ok && nsteps > 0 && has_gate && jl < len)
      p.dg_col[(size_t)(kvh * group + group - 1) * p.total + seq_start + jl] = dgcol;
    // ---- epilogue: dV and scale * dK for this key row (TMEM loads are warp-collective,
    // only the stores depend on the row being inside the sequence)
    if (ok) {
      tc_fence_after();
      const bool row_ok = jl < len;
      uint16_t* dvrow = p.grad_v + ((size_t)(seq_start + (row_ok ? jl : 0)) * p.hkv + kvh) * DV;
      uint16_t* dkrow = p.grad_k + ((size_t)(seq_start + (row_ok ? jl : 0)) * p.hkv + kvh) * DQK;
#pragma unroll 1
      for (int c = 0; c < (DV + DQK) / 32; ++c) {
        const bool is_v = c < DV / 32;
        const uint32_t col = is_v ? C::T_DV + c * 32 : C::T_DK + (c - DV / 32) * 32;
        const float sc = is_v ? 1.f : p.scale;
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + col, v);
        tmem_ld_wait();
        if (row_ok) {
          uint4* d = reinterpret_cast<uint4*>(is_v ? dvrow + c * 32 : dkrow + (c - DV / 32) * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            d[q] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * q]) * sc, __uint_as_float(v[8 * q + 1]) * sc),
                              pack_bf16x2(__uint_as_float(v[8 * q + 2]) * sc, __uint_as_float(v[8 * q + 3]) * sc),
                              pack_bf16x2(__uint_as_float(v[8 * q + 4]) * sc, __uint_as_float(v[8 * q + 5]) * sc),
                              pack_bf16x2(__uint_as_float(v[8 * q + 6]) * sc, __uint_as_float(v[8 * q + 7]) * sc));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DQK, int DV>
cudaError_t launch_t(const BwdParams& p, const BwdMaps& maps, int num_tiles, cudaStream_t s) {
  using C = BwdCfg<DQK, DV>;
  auto kern = prefill_bwd_kernel<DQK, DV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<dim3(num_tiles, p.hkv), kThreads, C::SMEM, s>>>(maps.q, maps.k, maps.v, maps.dout, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_bwd(const BwdParams& p, const BwdMaps& maps, int num_kv_tiles, cudaStream_t s) {
  if (p.dqk == 64 && p.dv == 64) return launch_t<64, 64>(p, maps, num_kv_tiles, s);
  if (p.dqk == 128 && p.dv == 128) return launch_t<128, 128>(p, maps, num_kv_tiles, s);
  return cudaErrorInvalidValue;
}

}  // namespace gcs
