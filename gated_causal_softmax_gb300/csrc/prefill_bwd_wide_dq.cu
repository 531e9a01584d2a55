// dQ pass of the backward for head dims above 128 (fla-org/flash-linear-attention #1322
// "Gluon attention backend with large head dimensions": Description, gradients for head dims
// through 512; the two-pass backward, a separate dQ kernel with no fp32 reduce-add).
//
// One CTA per (64 query rows, query head).  Q and dO of the 64 rows stay in shared memory; K
// and V tiles of 128 keys stream through a ring of 32 KB stages (two 64-column chunks each).
// Per key tile, in a fixed order, with the key dimension on the TMEM lanes:
//     S^T  = K Q^T           (M = 128 keys, N = 64 queries, K = DQK)
//     dP^T = V dO^T          (K = DV)
//     P^T = exp(S^T scale + G_i - G_j - LSE_i), dS^T = P^T (dP^T - delta_i) -> bf16 in smem
//     dQ^T += K^T dS^T       (M = 128 dims per half, N = 64 queries, K = 128 keys; the K tile
//                             streams a second time for it)
// dQ^T accumulates in TMEM over every visible key tile and is written once, in bf16; the dS
// row sums (gate and sink gradients) accumulate in registers and are summed over the four
// key-row warps in a fixed order.  Nothing is reduce-added, so dQ and the row sums do not
// depend on scheduling.  The key-stationary role kernel computes dK, dV and the dS column
// sums.
#include "kernels.h"
#include "sm103_ptx.cuh"
#include "tiles.cuh"

namespace gcs {
namespace {

constexpr int kBN = 128;      // keys per tile
constexpr int kBM = 64;       // query rows per CTA
constexpr int kThreads = 192;
constexpr int kStage = 16384; // one 128-row x 64-column bf16 chunk
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

template <int DQK, int DV>
struct WdqCfg {
  static constexpr int QCH = DQK / 64, VCH = DV / 64;  // 64-column chunks
  static constexpr int KP = DQK / 128, VP = DV / 128;  // pairs of chunks
  static constexpr int PAIR = 2 * kStage;
  static constexpr int OFF_Q = 0;                              // [QCH] x 8 KB (64 rows x 64 cols)
  static constexpr int OFF_DO = OFF_Q + QCH * (kStage / 2);    // [VCH] x 8 KB
  static constexpr int OFF_DS = OFF_DO + VCH * (kStage / 2);   // dS^T: 128 keys x 64 queries bf16
  static constexpr int OFF_RING = OFF_DS + kStage;
  static constexpr int NST_FIT = (227 * 1024 - 4096 - OFF_RING) / PAIR;
  static constexpr int NST = NST_FIT < 4 ? NST_FIT : 4;
  static constexpr int OFF_VEC = OFF_RING + NST * PAIR;        // colterm[64], delta[64], row sums [4][64]
  static constexpr int OFF_BAR = OFF_VEC + 6 * kBM * 4;
  static constexpr int OFF_MISC = OFF_BAR + (2 * NST + 16) * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static_assert(NST >= 2, "ring depth");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  // TMEM: S^T 0..63, dP^T 64..127, dQ^T half p at 128 + 64 p
  static constexpr int T_S = 0, T_DP = 64, T_DQ = 128;
  static constexpr uint32_t TCOLS = (T_DQ + 64 * KP) <= 256 ? 256 : 512;
};

template <int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_bwd_wide_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                               const BwdParams p) {
  using C = WdqCfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align_1k(smem_raw);

  TileRef tr;
  if (!lpt_tile(p.cu_seqlens, p.num_seqs, kBM, blockIdx.y, tr)) return;
  const int seq_start = tr.start, len = tr.len;
  const int h = blockIdx.x;
  const int kvh = h / (p.hq / p.hkv);
  const int i0 = tr.u * kBM;
  const int i_last = min(i0 + kBM, len) - 1;
  // key tiles seen by rows i0 .. i_last: causal up to i_last, window from i0 - W + 1
  const int jt_hi = i_last / kBN;
  const int jt_lo = p.window > 0 ? max(0, i0 - p.window + 1) / kBN : 0;
  const int nt = jt_hi - jt_lo + 1;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;             // [NST]
  uint64_t* empty = bars + C::NST;   // [NST]
  uint64_t* q_full = bars + 2 * C::NST;
  uint64_t* s_full = q_full + 1;
  uint64_t* p_full = q_full + 2;
  uint64_t* ds_free = q_full + 3;
  uint64_t* dq_done = q_full + 4;
  uint64_t* drain = q_full + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const Abort ab{abort_flag, p.status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 4);
    mbar_init(ds_free, 1);
    mbar_init(dq_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TCOLS);
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
      const int yq = seq_start + i0;
      mbar_expect_tx(q_full, (C::QCH + C::VCH) * (kStage / 2));
      for (int c = 0; c < C::QCH; ++c)
        tma_load_3d(smem + C::OFF_Q + c * (kStage / 2), &tmQ, q_full, c * 64, h, yq);
      for (int c = 0; c < C::VCH; ++c)
        tma_load_3d(smem + C::OFF_DO + c * (kStage / 2), &tmDO, q_full, c * 64, h, yq);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      // one 32 KB stage = columns x0 .. x0 + 127 of the tile's 128 key rows
      auto issue = [&](const CUtensorMap* m, int x0, int y) -> bool {
        if (!wait_bar(&empty[stage], phase ^ 1, ab)) return false;
        mbar_expect_tx(&full[stage], C::PAIR);
        uint8_t* dst = smem + C::OFF_RING + stage * C::PAIR;
        tma_load_3d(dst, m, &full[stage], x0, kvh, y);
        tma_load_3d(dst + kStage, m, &full[stage], x0 + 64, kvh, y);
        if (++stage == C::NST) {
          stage = 0;
          phase ^= 1;
        }
        return true;
      };
      for (int t = 0; t < nt && ok; ++t) {
        const int yk = seq_start + (jt_lo + t) * kBN;
        for (int q = 0; q < C::KP && ok; ++q) ok = issue(&tmK, q * 128, yk);  // S^T
        for (int q = 0; q < C::VP && ok; ++q) ok = issue(&tmV, q * 128, yk);   // dP^T
        for (int q = 0; q < C::KP && ok; ++q) ok = issue(&tmK, q * 128, yk);  // dQ^T
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16(128, kBM, false, false);  // S^T, dP^T
      const uint32_t idDQ = idesc_bf16(128, kBM, true, true);   // dQ^T half
      const uint32_t sQ = smem_u32(smem + C::OFF_Q), sDO = smem_u32(smem + C::OFF_DO);
      const uint32_t sDS = smem_u32(smem + C::OFF_DS), sRing = smem_u32(smem + C::OFF_RING);
      uint32_t stage = 0, phase = 0;
      auto take = [&](uint32_t& addr) -> bool {
        if (!wait_bar(&full[stage], phase, ab)) return false;
        tc_fence_after();
        addr = sRing + stage * C::PAIR;
        return true;
      };
      auto give = [&]() {
        mma_commit(&empty[stage]);
        if (++stage == C::NST) {
          stage = 0;
          phase ^= 1;
        }
      };
      bool ok = wait_bar(q_full, 0, ab);
      for (int t = 0; t < nt && ok; ++t) {
        // S^T = K Q^T over all DQK columns
        for (int q = 0; q < C::KP && ok; ++q) {
          uint32_t a = 0;
          ok = take(a);
          if (!ok) break;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = 2 * q + e;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(tmem + C::T_S, sdesc_sw128(a + e * kStage + k * 32, 16, 1024),
                     sdesc_sw128(sQ + c * (kStage / 2) + k * 32, 16, 1024), idS, (c | k) != 0);
          }
          give();
        }
        // dP^T = V dO^T over all DV columns
        for (int q = 0; q < C::VP && ok; ++q) {
          uint32_t a = 0;
          ok = take(a);
          if (!ok) break;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = 2 * q + e;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(tmem + C::T_DP, sdesc_sw128(a + e * kStage + k * 32, 16, 1024),
                     sdesc_sw128(sDO + c * (kStage / 2) + k * 32, 16, 1024), idS, (c | k) != 0);
          }
          give();
        }
        if (!ok) break;
        mma_commit(s_full);
        // dQ^T += K^T dS^T once the key rows have written dS^T
        ok = wait_bar(p_full, t & 1, ab);
        if (!ok) break;
        tc_fence_after();
        for (int q = 0; q < C::KP && ok; ++q) {
          uint32_t a = 0;
          ok = take(a);
          if (!ok) break;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ss(tmem + C::T_DQ + 64 * q, sdesc_sw128(a + k * 2048, kStage, 1024),
                   sdesc_sw128(sDS + k * 2048, kStage, 1024), idDQ, (t > 0 || k > 0) ? 1u : 0u);
          give();
        }
        if (!ok) break;
        mma_commit(ds_free);
      }
      if (ok) mma_commit(dq_done);
      if (!ok) {
        mma_commit(drain);
        mbar_wait(drain, 0, nullptr);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ key rows (4 warps)
    const int quarter = warp & 3;       // warps 2..5 reach TMEM lanes 64..127, 0..63
    const int r = quarter * 32 + lane;  // key row of the tile, TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::T_S, tDP = tmem + lane_off + C::T_DP;
    const bool has_gate = p.gT != nullptr;
    const bool want_row = p.dg_row != nullptr;
    uint8_t* sDS = smem + C::OFF_DS;
    float* colterm = reinterpret_cast<float*>(smem + C::OFF_VEC);
    float* dlt = colterm + kBM;
    float* rsum = colterm + 2 * kBM;  // [4 warps][64]
    // per-query terms of the 64 rows: -LSE_i log2 e + G_i, and delta_i
    if (r < kBM) {
      const int i = i0 + r;
      float ct = 0.f;
      if (i < len) {
        const size_t idx = (size_t)h * p.total + seq_start + i;
        ct = -__ldg(p.lse + idx) * kLog2e;
        if (has_gate) ct += __ldg(p.gT + idx);
      }
      colterm[r] = ct;
    } else {
      const int i = i0 + r - kBM;
      dlt[r - kBM] = (i < len) ? __ldg(p.delta + (size_t)h * p.total + seq_start + i) : 0.f;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    float rs0 = 0.f, rs1 = 0.f;  // sum over this warp's keys of dS for queries lane and 32 + lane
    bool ok = true;
    for (int t = 0; t < nt; ++t) {
      const int j0 = (jt_lo + t) * kBN;
      const int jl = j0 + r;
      const float rowterm = (has_gate && jl < len) ? -__ldg(p.gT + (size_t)h * p.total + seq_start + jl) : 0.f;
      ok = wait_bar(s_full, t & 1, ab);
      if (!ok) break;
      tc_fence_after();
      // dS^T of the previous tile must have been read by its dQ MMAs
      if (t > 0) {
        ok = wait_bar(ds_free, (t - 1) & 1, ab);
        if (!ok) break;
      }
      const bool need_mask =
          (i0 < j0 + kBN - 1) || (p.window > 0 && i0 + kBM - 1 - j0 >= p.window) || (i0 + kBM > len);
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t sv[32], dp[32];
        tmem_ld32(tS + 32 * ch, sv);
        tmem_ld32(tDP + 32 * ch, dp);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int col = 32 * ch + c;
          float tt = fmaf(__uint_as_float(sv[c]), p.scale_log2, colterm[col]) + rowterm;
          if (need_mask) {
            const int i = i0 + col;
            const bool vis = (i < len) && (jl <= i) && (p.window == 0 || i - jl < p.window);
            tt = vis ? tt : neg_inf();
          }
          const float pr = ex2(tt);
          dp[c] = __float_as_uint(pr * (__uint_as_float(dp[c]) - dlt[col]));
        }
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(__uint_as_float(dp[2 * c]), __uint_as_float(dp[2 * c + 1]));
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(sDS + sw128_offset(r, 4 * ch + q)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        if (want_row) {
          // column sums over this warp's 32 keys: lane l ends with query 32 ch + l
          float v[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = __uint_as_float(dp[c]);
#pragma unroll
          for (int half = 16; half >= 1; half >>= 1) {
            const bool upper = (lane & half) != 0;
#pragma unroll
            for (int c = 0; c < half; ++c) {
              const float send = upper ? v[c] : v[c + half];
              const float keep = upper ? v[c + half] : v[c];
              v[c] = keep + __shfl_xor_sync(0xffffffffu, send, half);
            }
          }
          if (ch == 0)
            rs0 += v[0];
          else
            rs1 += v[0];
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok) ok = wait_bar(dq_done, 0, ab);
    if (ok) {
      tc_fence_after();
      // dQ^T halves: lane r holds dims 128 q + r for the 64 queries
      const int nrows = min(kBM, len - i0);
      const size_t row_stride = (size_t)p.dq_ts;
#pragma unroll 1
      for (int q = 0; q < C::KP; ++q) {
        uint32_t dq[64];
        tmem_ld32(tmem + lane_off + C::T_DQ + 64 * q, dq);
        tmem_ld32(tmem + lane_off + C::T_DQ + 64 * q + 32, dq + 32);
        tmem_ld_wait();
        uint16_t* base = p.grad_q + (size_t)(seq_start + i0) * p.dq_ts + (size_t)h * p.dq_hs + 128 * q + r;
#pragma unroll
        for (int c = 0; c < kBM; ++c)
          if (c < nrows) {
            const uint32_t b = pack_bf16x2(__uint_as_float(dq[c]) * p.scale, 0.f);
            base[c * row_stride] = static_cast<uint16_t>(b & 0xffffu);
          }
      }
      if (want_row) {
        rsum[quarter * kBM + lane] = rs0;
        rsum[quarter * kBM + 32 + lane] = rs1;
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (ok && want_row && quarter == 0) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = 32 * u + lane;
        const float v = ((rsum[c] + rsum[kBM + c]) + rsum[2 * kBM + c]) + rsum[3 * kBM + c];
        if (i0 + c < len) p.dg_row[(size_t)h * p.total + seq_start + i0 + c] = v;
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
    tmem_dealloc(tmem, C::TCOLS);
  }
}

template <int DQK, int DV>
cudaError_t launch_t(const BwdParams& p, const BwdMaps& maps, int num_q_tiles, cudaStream_t s) {
  using C = WdqCfg<DQK, DV>;
  auto kern = prefill_bwd_wide_dq_kernel<DQK, DV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<dim3(p.hq, num_q_tiles), kThreads, C::SMEM, s>>>(maps.q, maps.k, maps.v, maps.dout, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_bwd_wide_dq(const BwdParams& p, const BwdMaps& maps, int num_q_tiles, cudaStream_t s) {
  if (p.dqk == 256 && p.dv == 256) return launch_t<256, 256>(p, maps, num_q_tiles, s);
  if (p.dqk == 256 && p.dv == 512) return launch_t<256, 512>(p, maps, num_q_tiles, s);
  if (p.dqk == 512 && p.dv == 512) return launch_t<512, 512>(p, maps, num_q_tiles, s);
  return cudaErrorInvalidValue;
}

}  // namespace gcs
