// Prefill backward, dQ pass (the two-pass backward that fla-org/flash-linear-attention
// #1322 "Gluon attention backend with large head dimensions" keeps beside its fused-dQ
// experiment, Oct 5 comment): one CTA per (128-row query tile, query head) recomputes
// the scores and dP for every key tile it sees and accumulates dQ in TMEM, so dQ is
// written once, in bf16, with no fp32 buffer and no reduce-adds.  The fp32 row sums of
// dS (gate and sink gradients, Oct 3 comment) are thread-local here: one thread per row.
//
// Per key tile (visited from the diagonal backwards):
//     S  = Q K^T                 (TMEM, two buffers)   P  = 2^(S scale log2e + G_i - LSE_i - G_j)
//     dP = dO V^T                (TMEM)                dS = P o (dP - delta_i)
//     dQ += dS K                 (A operand = dS, bf16, written over the consumed S)
// Warp roles (192 threads): warp 0 TMA producer (Q and dO once; K and V tiles through two
// stages each), warp 1 tcgen05 issuer, warps 2..5 one thread per query row.
#include "kernels.h"
#include "sm103_ptx.cuh"
#include "tiles.cuh"

namespace gcs {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kChunk = 128 * 128;  // 128 rows x 64 bf16
constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

template <int D>
struct DqCfg {
  static constexpr int CH = D / 64;
  static constexpr int TILE = CH * kChunk;  // one 128-row tile of a D-wide operand
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + TILE;
  static constexpr int OFF_K = OFF_DO + TILE;   // [2] stages
  static constexpr int OFF_V = OFF_K + 2 * TILE;  // [2] stages
  static constexpr int OFF_G = OFF_V + 2 * TILE;  // [4 warps][2][128] floats
  static constexpr int OFF_BAR = OFF_G + 4 * 2 * kBN * 4;
  static constexpr int OFF_MISC = OFF_BAR + 16 * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  // TMEM: S[b] at 128 b, dP at 256, dQ at 384
  static constexpr int T_S = 0, T_DP = 256, T_DQ = 384;
};

// One 32-column chunk of a query row: dS = 2^(S scale log2e + rowterm - G_j) (dP - delta)
// in place (fp32), returning its sum.  MASK keeps columns jmin..jmax only; the mask is a
// compile-time variant so that unmasked tiles carry no per-element mask work.
template <bool MASK>
__device__ __forceinline__ float dq_chunk(uint32_t* sv, const uint32_t* dp, const float* gj, int jb, float rowterm,
                                          float scale_log2, float dl, int jmin, int jmax) {
  float acc[4] = {0.f, 0.f, 0.f, 0.f};  // independent partial sums (latency)
  // -G_j as 16-B broadcast loads: shared-memory loads compete with running MMAs' operand reads
  const float4* gj4 = reinterpret_cast<const float4*>(gj + jb);
#pragma unroll
  for (int c4 = 0; c4 < 8; ++c4) {
    const float4 g4 = gj4[c4];
    const float gs[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = 4 * c4 + e;
      float t = fmaf(__uint_as_float(sv[c]), scale_log2, rowterm) + gs[e];
      if (MASK) t = (jb + c >= jmin && jb + c <= jmax) ? t : neg_inf();
      const float ds = ex2(t) * (__uint_as_float(dp[c]) - dl);
      acc[c & 3] += ds;
      sv[c] = __float_as_uint(ds);
    }
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                          const BwdParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align_1k(smem_raw);

  // heaviest query tiles (most key tiles to visit) first
  TileRef tr;
  if (!lpt_tile(p.cu_seqlens, p.num_seqs, kBM, blockIdx.y, tr)) return;
  const int seq_start = tr.start, len = tr.len, qt = tr.u;
  const int h = blockIdx.x;
  const int kvh = h / (p.hq / p.hkv);
  const int q0 = qt * kBM;
  const int hi_t = qt;
  int lo_t = 0;
  if (p.window > 0) {
    const int lo_j = q0 - p.window + 1;
    lo_t = lo_j > 0 ? lo_j / kBN : 0;
  }
  const int nt = hi_t - lo_t + 1;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* qd_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [2]
  uint64_t* k_empty = bars + 3;  // [2]
  uint64_t* v_full = bars + 5;   // [2]
  uint64_t* v_empty = bars + 7;  // [2]
  uint64_t* s_full = bars + 9;   // [2]
  uint64_t* dp_full = bars + 11;
  uint64_t* ds_ready = bars + 12;
  uint64_t* dq_done = bars + 13;
  uint64_t* drain = bars + 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  float* sG = reinterpret_cast<float*>(smem + C::OFF_G);
  const Abort ab{abort_flag, p.status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(qd_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
    }
    mbar_init(dp_full, 1);
    mbar_init(ds_ready, 4);
    mbar_init(dq_done, 1);
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
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmDO);
      const uint64_t pol_kv = l2_policy_evict_last();
      mbar_expect_tx(qd_full, 2 * C::TILE);
      for (int c = 0; c < C::CH; ++c) {
        tma_load_3d(smem + C::OFF_Q + c * kChunk, &tmQ, qd_full, c * 64, h, seq_start + q0);
        tma_load_3d(smem + C::OFF_DO + c * kChunk, &tmDO, qd_full, c * 64, h, seq_start + q0);
      }
      bool ok = true;
      for (int n = 0; n < nt && ok; ++n) {
        const int kb = n & 1;
        const int y = seq_start + (hi_t - n) * kBN;
        ok = wait_bar(&k_empty[kb], ((n >> 1) & 1) ^ 1, ab);
        if (!ok) break;
        mbar_expect_tx(&k_full[kb], C::TILE);
        for (int c = 0; c < C::CH; ++c)
          tma_load_3d_hint(smem + C::OFF_K + kb * C::TILE + c * kChunk, &tmK, &k_full[kb], c * 64, kvh, y,
                           pol_kv);
        ok = wait_bar(&v_empty[kb], ((n >> 1) & 1) ^ 1, ab);
        if (!ok) break;
        mbar_expect_tx(&v_full[kb], C::TILE);
        for (int c = 0; c < C::CH; ++c)
          tma_load_3d_hint(smem + C::OFF_V + kb * C::TILE + c * kChunk, &tmV, &v_full[kb], c * 64, kvh, y,
                           pol_kv);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idSS = idesc_bf16(128, kBN, false, false);  // S, dP
      const uint32_t idDQ = idesc_bf16(128, D, false, true);     // dQ += dS K (K as MN-major B)
      // descriptors built once; offsets are added to the address field (shared-memory
      // addresses stay below 2^18, so the 14-bit field never carries)
      const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
      const uint64_t dDO0 = sdesc_sw128(smem_u32(smem + C::OFF_DO), 16, 1024);
      const uint64_t dK0 = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024);
      const uint64_t dKmn0 = sdesc_sw128(smem_u32(smem + C::OFF_K), kChunk, 1024);
      constexpr uint32_t kChunk16 = kChunk >> 4, kTile16 = C::TILE >> 4;
      // Waits are batched ahead of runs of back-to-back MMAs: the tensor pipe has almost no
      // issue queue, so each stall of this thread on a barrier leaves it idle.
      auto mma_s = [&](int n) {  // S(n) = Q K(n)^T into S[n & 1] (K(n) landed)
        const int kb = n & 1;
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          const uint64_t a = dQ0 + c * kChunk16, b = dK0 + kb * kTile16 + c * kChunk16;
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ss(tmem + C::T_S + 128 * (n & 1), a + 2 * k, b + 2 * k, idSS, (c | k) != 0);
        }
        mma_commit(&s_full[n & 1]);
      };
      auto mma_dp = [&](int n) {  // dP(n) = dO V(n)^T (V(n) landed)
        const int kb = n & 1;
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          const uint64_t a = dDO0 + c * kChunk16, b = dV0 + kb * kTile16 + c * kChunk16;
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ss(tmem + C::T_DP, a + 2 * k, b + 2 * k, idSS, (c | k) != 0);
        }
        mma_commit(dp_full);
        mma_commit(&v_empty[kb]);
      };
      bool ok = wait_bars(ab, qd_full, 0, &k_full[0], 0, &v_full[0], 0);
      if (ok) {
        tc_fence_after();
        mma_s(0);
        mma_dp(0);
      }
      if (ok && nt > 1) {
        ok = wait_bars(ab, &k_full[1], 0);
        if (ok) {
          tc_fence_after();
          mma_s(1);
        }
      }
      for (int n = 0; n < nt && ok; ++n) {
        const int b = n & 1, kb = n & 1;
        const bool more = n + 1 < nt;
        // dS(n) stored (the warps consumed dP(n) before signalling), V(n+1) landed
        ok = more ? wait_bars(ab, ds_ready, n & 1, &v_full[(n + 1) & 1], ((n + 1) >> 1) & 1)
                  : wait_bars(ab, ds_ready, n & 1);
        if (!ok) break;
        tc_fence_after();
        if (more) mma_dp(n + 1);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts(tmem + C::T_DQ, tmem + C::T_S + 128 * b + k * 8, dKmn0 + kb * kTile16 + 128 * k, idDQ,
                 (n > 0 || k > 0) ? 1u : 0u);
        mma_commit(&k_empty[kb]);
        // scores of tile n + 2 over buffer b (its dS was read by the dQ MMAs above); its K
        // stage was freed by those MMAs, so this wait covers the load
        if (n + 2 < nt) {
          ok = wait_bars(ab, &k_full[kb], ((n + 2) >> 1) & 1);
          if (!ok) break;
          tc_fence_after();
          mma_s(n + 2);
        }
      }
      if (ok) mma_commit(dq_done);
      if (!ok) {
        mma_commit(drain);
        mbar_wait(drain, 0, nullptr);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ query rows
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int il = q0 + r;
    const bool row_valid = il < len;
    const size_t rix = (size_t)h * p.total + seq_start + (row_valid ? il : 0);
    const bool has_gate = p.gT != nullptr;
    // invalid rows get -inf: every probability of theirs is 0
    const float rowterm = row_valid ? (-__ldg(p.lse + rix) * kLog2e + (has_gate ? __ldg(p.gT + rix) : 0.f))
                                    : neg_inf();
    const float dl = row_valid ? __ldg(p.delta + rix) : 0.f;
    float dgrow = 0.f;
    bool ok = true;
    if (!has_gate) {
      // no gate: the G_j buffers stay zero
      for (int u = lane; u < 2 * kBN; u += 32) sG[quarter * 2 * kBN + u] = 0.f;
      __syncwarp();
    }
    for (int n = 0; n < nt; ++n) {
      const int jt = hi_t - n, j0 = jt * kBN, b = n & 1;
      float* gj = sG + (quarter * 2 + b) * kBN;  // this warp's copy of -G_j for the tile
      if (has_gate) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int jl = j0 + lane * 4 + u;
          gj[lane * 4 + u] = (jl < len) ? -__ldg(p.gT + (size_t)h * p.total + seq_start + jl) : 0.f;
        }
        __syncwarp();
      }
      ok = wait_bar(&s_full[b], (n >> 1) & 1, ab);
      if (!ok) break;
      ok = wait_bar(dp_full, n & 1, ab);
      if (!ok) break;
      tc_fence_after();
      const bool need_mask = (jt == hi_t) || (p.window > 0 && j0 < q0 + kBM - p.window);
      // visible key columns of this row within the tile: causal j <= i, window i - j < W
      const int jmax = il - j0;
      const int jmin = p.window > 0 ? il - p.window + 1 - j0 : -(1 << 30);
      const uint32_t tS = tmem + lane_off + C::T_S + 128 * b, tDP = tmem + lane_off + C::T_DP;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t sv[32], dp[32];
        tmem_ld32(tS + 32 * ch, sv);
        tmem_ld32(tDP + 32 * ch, dp);
        tmem_ld_wait();
        dgrow += need_mask ? dq_chunk<true>(sv, dp, gj, 32 * ch, rowterm, p.scale_log2, dl, jmin, jmax)
                           : dq_chunk<false>(sv, dp, gj, 32 * ch, rowterm, p.scale_log2, dl, jmin, jmax);
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1]));
        tmem_st16(tS + 16 * ch, pk);  // dS (bf16) over S columns already loaded
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_ready);
    }
    if (ok) ok = wait_bar(dq_done, 0, ab);
    if (ok) {
      tc_fence_after();
      uint16_t* dqrow = p.grad_q + (size_t)(seq_start + (row_valid ? il : 0)) * p.dq_ts + (size_t)h * p.dq_hs;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + C::T_DQ + c * 32, v);
        tmem_ld_wait();
        if (row_valid) {
          uint4* d = reinterpret_cast<uint4*>(dqrow + c * 32);
          const float sc = p.scale;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            d[q] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * q]) * sc, __uint_as_float(v[8 * q + 1]) * sc),
                              pack_bf16x2(__uint_as_float(v[8 * q + 2]) * sc, __uint_as_float(v[8 * q + 3]) * sc),
                              pack_bf16x2(__uint_as_float(v[8 * q + 4]) * sc, __uint_as_float(v[8 * q + 5]) * sc),
                              pack_bf16x2(__uint_as_float(v[8 * q + 6]) * sc, __uint_as_float(v[8 * q + 7]) * sc));
        }
      }
      if (row_valid && p.dg_row) p.dg_row[rix] = dgrow;
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

template <int D>
cudaError_t launch_t(const BwdParams& p, const BwdMaps& maps, int num_tiles, cudaStream_t s) {
  using C = DqCfg<D>;
  auto kern = prefill_bwd_dq_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<dim3(p.hq, num_tiles), kThreads, C::SMEM, s>>>(maps.q, maps.k, maps.v, maps.dout, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_bwd_dq(const BwdParams& p, const BwdMaps& maps, int num_q_tiles, cudaStream_t s) {
  if (p.dqk == 64 && p.dv == 64) return launch_t<64>(p, maps, num_q_tiles, s);
  if (p.dqk == 128 && p.dv == 128) return launch_t<128>(p, maps, num_q_tiles, s);
  return cudaErrorInvalidValue;
}

}  // namespace gcs
