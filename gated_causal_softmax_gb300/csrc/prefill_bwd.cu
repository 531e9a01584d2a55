// Prefill backward, dK / dV pass of the two-pass backward (fla-org/flash-linear-attention
// #1322 "Gluon attention backend with large head dimensions": Oct 5 comment keeps the
// two-pass route beside the fused-dQ experiment; Oct 3 comment -- probabilities
// recomputed in fp32).  dQ and the row sums of dS come from the dQ pass
// (prefill_bwd_dq.cu), so this kernel has no reduce-adds on its hot path.
//
// One CTA per (128-key tile, kv head); it loops over the query heads of its GQA group and
// over 64-row query tiles in the causal / window range ("steps").  Per step:
//     S^T  = K Q^T            (TMEM, fp32)        P^T  = 2^(S^T*scale*log2e + G_i - G_j - LSE_i)
//     dP^T = V dO^T           (TMEM, fp32)        dS^T = P^T o (dP^T - delta_i)
//     dV  += P^T dO           (A operand = P^T, bf16, written over the consumed S^T)
//     dK  += dS^T Q           (A operand = dS^T, bf16, written over the consumed dP^T)
// plus the fp32 column sums of dS (gate gradient), one thread per key row.
//
// Warp roles (320 threads): warp 0 TMA producer (K/V once; Q, dO and the packed
// per-column LSE / delta / gate vectors in rotating buffers), warp 1 tcgen05 issuer,
// warps 2..5 and 6..9 two ping-pong softmax warpgroups: warpgroup w owns TMEM buffers
// S^T[w], dP^T[w] and handles the steps s with s % 2 == w, so one warpgroup's
// exponentials overlap the other warpgroup's MMAs.  P^T and dS^T are signalled
// separately (dV starts as soon as P^T is in TMEM).  tcgen05.mma operations issued by
// one thread execute in issue order, so an MMA may overwrite TMEM columns that an
// earlier MMA reads as its A operand.
#include "kernels.h"
#include "sm103_ptx.cuh"
#include "tiles.cuh"

namespace gcs {
namespace {

constexpr int kBN = 128;  // keys per CTA (TMEM lanes)
constexpr int kBM = 64;   // query rows per step
constexpr int kThreads = 320;
constexpr int kNQB = 4;   // query-side buffers
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
  static constexpr int OFF_Q = OFF_V + VCH * kKVChunk;            // [kNQB][KCH] chunks
  static constexpr int OFF_DO = OFF_Q + kNQB * KCH * kQChunk;     // [kNQB][VCH] chunks
  static constexpr int OFF_VEC = OFF_DO + kNQB * VCH * kQChunk;   // [kNQB][2][64] floats
  static constexpr int OFF_BAR = OFF_VEC + kNQB * 2 * kBM * 4;
  static constexpr int NBAR = 24;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  // TMEM columns: score buffers S^T[b] at 64b, dP^T[b] at 128 + 64b, dV, dK
  static constexpr int T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + DV;
  static_assert(T_DK + DQK <= 512, "TMEM budget");
};

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// P for 32 query columns of a key row: pr = 2^(S scale log2e + colterm_i + rowterm),
// MASK keeps columns cmin..cmax (compile-time variant: unmasked steps carry no mask work).
template <bool MASK>
__device__ __forceinline__ void p_chunk(float* pr, const uint32_t* sv, const float4* ct4, float rowterm,
                                        float scale_log2, int cb, int cmin, int cmax) {
#pragma unroll
  for (int c4 = 0; c4 < 8; ++c4) {
    const float4 ct = ct4[c4];
    const float cts[4] = {ct.x + rowterm, ct.y + rowterm, ct.z + rowterm, ct.w + rowterm};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = 4 * c4 + e;
      float t = fmaf(__uint_as_float(sv[c]), scale_log2, cts[e]);
      if (MASK) t = (cb + c >= cmin && cb + c <= cmax) ? t : neg_inf();
      pr[c] = ex2(t);
    }
  }
}

template <int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const BwdParams p) {
  using C = BwdCfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  // heaviest key tiles (most query tiles after them) first
  TileRef tr;
  if (!lpt_tile(p.cu_seqlens, p.num_seqs, kBN, blockIdx.y, tr)) return;
  const int seq_start = tr.start, len = tr.len, jt = tr.n - 1 - tr.u;
  int qoff = 0;  // first 64-row query tile of this sequence in the packed vectors
  for (int q = 0; q < tr.seq; ++q) qoff += (__ldg(p.cu_seqlens + q + 1) - __ldg(p.cu_seqlens + q) + kBM - 1) / kBM;
  const int kvh = blockIdx.x;
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
  uint64_t* q_full = bars + 1;     // [kNQB]
  uint64_t* q_empty = bars + 5;    // [kNQB]
  uint64_t* s_full = bars + 9;     // [2] S^T[b] written
  uint64_t* dp_full = bars + 11;   // [2] dP^T[b] written
  uint64_t* pv_ready = bars + 13;  // [2] P^T[b] stored (A operand of dV)
  uint64_t* ds_ready = bars + 15;  // [2] dS^T[b] stored (A operand of dK)
  uint64_t* drain = bars + 19;
  uint64_t* all_done = bars + 20;  // every MMA of the CTA retired (epilogue)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const Abort ab{abort_flag, p.status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int b = 0; b < kNQB; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&dp_full[b], 1);
      mbar_init(&pv_ready[b], 4);
      mbar_init(&ds_ready[b], 4);
    }
    mbar_init(drain, 1);
    mbar_init(all_done, 1);
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
    if (lane == 0) {
      for (int s = 0; s < nsteps && ok; ++s) {
        const int qb = s % kNQB;
        const int h = kvh * group + s / n_it;
        const int it = it_lo + s % n_it;
        ok = wait_bar(&q_empty[qb], ((s / kNQB) & 1) ^ 1, ab);
        if (!ok) break;
        mbar_expect_tx(&q_full[qb], (C::KCH + C::VCH) * kQChunk + 2 * kBM * 4);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_2d_hint(smem + C::OFF_Q + (qb * C::KCH + c) * kQChunk, &tmQ, &q_full[qb], h * DQK + c * 64,
                           seq_start + it * kBM, pol);
        for (int c = 0; c < C::VCH; ++c)
          tma_load_2d_hint(smem + C::OFF_DO + (qb * C::VCH + c) * kQChunk, &tmDO, &q_full[qb], h * DV + c * 64,
                           seq_start + it * kBM, pol);
        // per-column vectors: [0..63] (G_i - LSE_i) log2 e, [64..127] delta_i
        bulk_load(smem + C::OFF_VEC + qb * 2 * kBM * 4, p.vecp + ((size_t)h * p.n_qtiles + qoff + it) * 2 * kBM,
                  2 * kBM * 4, &q_full[qb]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16(128, kBM, false, false);   // S^T, dP^T
      const uint32_t idDV = idesc_bf16(128, DV, false, true);    // dV += P^T dO
      const uint32_t idDK = idesc_bf16(128, DQK, false, true);   // dK += dS^T Q
      // descriptors built once; offsets are added to the address field (shared-memory
      // addresses stay below 2^18, so the 14-bit field never carries)
      const uint64_t dK0 = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
      const uint64_t dDO0 = sdesc_sw128(smem_u32(smem + C::OFF_DO), 16, 1024);
      const uint64_t dQmn0 = sdesc_sw128(smem_u32(smem + C::OFF_Q), kQChunk, 1024);
      const uint64_t dDOmn0 = sdesc_sw128(smem_u32(smem + C::OFF_DO), kQChunk, 1024);
      constexpr uint32_t kKV16 = kKVChunk >> 4, kQ16 = kQChunk >> 4;
      bool ok = wait_bar(kv_full, 0, ab);
      auto issue_s = [&](int t) -> bool {  // S^T(t) = K Q(t)^T -> S^T[t & 1]
        const int qb = t % kNQB, b = t & 1;
        if (!wait_bar(&q_full[qb], (t / kNQB) & 1, ab)) return false;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < C::KCH; ++c) {
          const uint64_t a = dK0 + c * kKV16, bq = dQ0 + (qb * C::KCH + c) * kQ16;
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ss(tmem + C::T_S + 64 * b, a + 2 * k, bq + 2 * k, idS, (c | k) != 0);
        }
        mma_commit(&s_full[b]);
        return true;
      };
      auto issue_dp = [&](int t) {  // dP^T(t) = V dO(t)^T -> dP^T[t & 1] (Q/dO(t) already landed)
        const int qb = t % kNQB, b = t & 1;
#pragma unroll
        for (int c = 0; c < C::VCH; ++c) {
          const uint64_t a = dV0 + c * kKV16, bd = dDO0 + (qb * C::VCH + c) * kQ16;
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ss(tmem + C::T_DP + 64 * b, a + 2 * k, bd + 2 * k, idS, (c | k) != 0);
        }
        mma_commit(&dp_full[b]);
      };
      for (int t = 0; t < 2 && t < nsteps && ok; ++t) {
        ok = issue_s(t);
        if (ok) issue_dp(t);
      }
      for (int s = 0; s < nsteps && ok; ++s) {
        const int b = s & 1, qb = s % kNQB;
        const uint64_t qa = dQmn0 + qb * C::KCH * kQ16, da = dDOmn0 + qb * C::VCH * kQ16;
        ok = wait_bar(&pv_ready[b], (s >> 1) & 1, ab);
        if (!ok) break;
        tc_fence_after();
        // K dimension = 64 query rows = 4 steps of 16 rows (2048 B in the MN-major views)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts(tmem + C::T_DV, tmem + C::T_S + 64 * b + k * 8, da + 128 * k, idDV, (s > 0 || k > 0) ? 1u : 0u);
        ok = wait_bar(&ds_ready[b], (s >> 1) & 1, ab);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts(tmem + C::T_DK, tmem + C::T_DP + 64 * b + k * 8, qa + 128 * k, idDK, (s > 0 || k > 0) ? 1u : 0u);
        mma_commit(&q_empty[qb]);
        // next scores of this buffer pair (P^T / dS^T were read by the MMAs above)
        if (s + 2 < nsteps) {
          ok = issue_s(s + 2);
          if (ok) issue_dp(s + 2);
        }
      }
      if (ok) mma_commit(all_done);
      if (!ok) {
        mma_commit(drain);
        mbar_wait(drain, 0, nullptr);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ key rows (two warpgroups)
    const int wg = (warp - 2) >> 2;     // steps s with s % 2 == wg, TMEM buffer wg
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::T_S + 64 * wg;
    const uint32_t tDP = tmem + lane_off + C::T_DP + 64 * wg;
    const int jl = j0 + r;
    const bool has_gate = p.gT != nullptr;
    float dgcol = 0.f;
    int cur_h = -1;
    float rowterm = 0.f;
    bool ok = true;
    for (int s = wg; s < nsteps; s += 2) {
      const int qb = s % kNQB;
      const int h = kvh * group + s / n_it;
      const int i0 = (it_lo + s % n_it) * kBM;
      if (h != cur_h) {
        // new query head: flush the column sums of dS of the previous head, reload G_j
        if (cur_h >= 0 && has_gate && jl < len) red_add_f32(p.dg_col + (size_t)cur_h * p.total + seq_start + jl, dgcol);
        dgcol = 0.f;
        cur_h = h;
        rowterm = (has_gate && jl < len) ? -__ldg(p.gT + (size_t)h * p.total + seq_start + jl) : 0.f;
      }
      ok = wait_bar(&q_full[qb], (s / kNQB) & 1, ab);
      if (!ok) break;
      const float4* vec4 = reinterpret_cast<const float4*>(smem + C::OFF_VEC + qb * 2 * kBM * 4);
      const bool need_mask = (i0 < j0 + kBN - 1) || (p.window > 0 && i0 + kBM - 1 - j0 >= p.window) ||
                             (i0 + kBM > len);
      // ---- P = 2^(S scale log2e + G_i - LSE_i - G_j) in fp32, P^T (bf16) over S^T
      ok = wait_bar(&s_full[wg], (s >> 1) & 1, ab);
      if (!ok) break;
      tc_fence_after();
      // visible query columns of this key row: causal i >= j, window i - j < W, i < len
      const int cmin = jl - i0;
      const int cmax = min(p.window > 0 ? jl + p.window - 1 - i0 : (1 << 30), len - 1 - i0);
      float pr[64];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t sv[32];
        tmem_ld32(tS + 32 * ch, sv);
        tmem_ld_wait();
        if (need_mask)
          p_chunk<true>(pr + 32 * ch, sv, vec4 + 8 * ch, rowterm, p.scale_log2, 32 * ch, cmin, cmax);
        else
          p_chunk<false>(pr + 32 * ch, sv, vec4 + 8 * ch, rowterm, p.scale_log2, 32 * ch, cmin, cmax);
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(pr[32 * ch + 2 * c], pr[32 * ch + 2 * c + 1]);
        tmem_st16(tS + 16 * ch, pk);  // over S^T columns already loaded
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pv_ready[wg]);
      // ---- dS = P (dP - delta_i) in fp32, dS^T (bf16) over dP^T
      ok = wait_bar(&dp_full[wg], (s >> 1) & 1, ab);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t dp[32];
        tmem_ld32(tDP + 32 * ch, dp);
        tmem_ld_wait();
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 dl = vec4[16 + 8 * ch + c4];
          const float dls[4] = {dl.x, dl.y, dl.z, dl.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 4 * c4 + e, col = 32 * ch + c;
            pr[col] = pr[col] * (__uint_as_float(dp[c]) - dls[e]);
          }
        }
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(pr[32 * ch + 2 * c], pr[32 * ch + 2 * c + 1]);
        tmem_st16(tDP + 16 * ch, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ds_ready[wg]);
      // fp32 column sum of dS for this key row (gate gradient)
      if (has_gate) {
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) acc[c & 7] += pr[c];
        dgcol += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      }
    }
    if (ok && cur_h >= 0 && has_gate && jl < len)
      red_add_f32(p.dg_col + (size_t)cur_h * p.total + seq_start + jl, dgcol);
    // ---- epilogue (warpgroup 0): dV and scale * dK for this key row.  TMEM loads are
    // warp-collective; only the stores depend on the row being inside the sequence.
    if (ok && wg == 0 && nsteps > 0) {
      // a single-use barrier: the per-buffer mma_done barriers may be more than one phase
      // ahead of this warpgroup, where a parity wait could alias
      ok = wait_bar(all_done, 0, ab);
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
  kern<<<dim3(p.hkv, num_tiles), kThreads, C::SMEM, s>>>(maps.q, maps.k, maps.v, maps.dout, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_bwd(const BwdParams& p, const BwdMaps& maps, int num_kv_tiles, cudaStream_t s) {
  if (p.dqk == 64 && p.dv == 64) return launch_t<64, 64>(p, maps, num_kv_tiles, s);
  if (p.dqk == 128 && p.dv == 128) return launch_t<128, 128>(p, maps, num_kv_tiles, s);
  return cudaErrorInvalidValue;
}

}  // namespace gcs
