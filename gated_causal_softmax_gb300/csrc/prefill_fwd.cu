// Prefill forward: gated causal softmax attention, one CTA per (128-row query tile,
// query head, value-column chunk).
//
// Computes, for every visible (i, j) pair of a sequence (fla-org/flash-linear-attention
// #1322 "Gluon attention backend with large head dimensions", Description):
//     s_ij = scale * q_i . k_j + G_i - G_j      (G: cumulative log gates)
//     O_i  = sum_j e^{s_ij} v_j / (sum_j e^{s_ij} + e^{sigma_h}),   LSE_i = ln(denominator)
//
// Warp roles (192 threads):
//   warp 0      TMA producer: the Q tile once, then K and V tiles as 128 x 64 bf16
//               chunks (128-B swizzle) through a ring of shared-memory stages.
//   warp 1      tcgen05 issuer: S = Q K^T into one of two TMEM score buffers, then
//               O += P V with P read from TMEM (bf16, written over the scores).
//   warps 2..5  softmax: one thread per query row (TMEM lane); gate, causal / window
//               masks and the sink are folded into the score row; online softmax in
//               log2 units with a lazy rescale of O (only when the running max grows by
//               more than 2^8); epilogue O / l -> bf16, LSE.
// Key tiles are visited from the diagonal backwards: with decaying gates the largest
// scores come first, so the running max rarely moves and O is rarely rescaled.
#include "kernels.h"
#include "sm103_ptx.cuh"
#include "tiles.cuh"

namespace gcs {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kChunk = 128 * 128;  // bytes of one 128-row x 64-col bf16 tile
constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.0f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// Three-input maximum (one instruction on this architecture).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <int DQK, int DVC>
struct FwdCfg {
  static constexpr int QCH = DQK / 64;
  static constexpr int KCH = DQK / 64;
  static constexpr int VCH = DVC / 64;
  static constexpr int NST = DQK >= 512 ? 5 : 8;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = QCH * kChunk;
  static constexpr int OFF_G = OFF_RING + NST * kChunk;
  static constexpr int OFF_BAR = OFF_G + 4 * 2 * kBN * 4;  // per softmax warp, double-buffered
  static constexpr int NBAR = 1 + 2 * NST + 6 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(256 + DVC <= 512, "TMEM budget");
};

template <int DQK, int DVC>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<DQK, DVC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align_1k(smem_raw);

  // heaviest query tiles (most key tiles to visit) first
  TileRef tr;
  if (!lpt_tile(p.cu_seqlens, p.num_seqs, kBM, blockIdx.y, tr)) return;
  const int seq_start = tr.start, len = tr.len, qt = tr.u;
  const int h = blockIdx.x;
  const int kvh = h / (p.hq / p.hkv);
  const int dv0 = blockIdx.z * DVC;
  const int q0 = qt * kBM;
  const int hi_t = qt;
  int lo_t = 0;
  if (p.window > 0) {
    const int lo_j = q0 - p.window + 1;
    lo_t = lo_j > 0 ? lo_j / kBN : 0;
  }
  const int nt = hi_t - lo_t + 1;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = bars + 1 + C::NST;
  uint64_t* s_full = bars + 1 + 2 * C::NST;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = s_full + 4;
  uint64_t* drain = s_full + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  float* sG = reinterpret_cast<float*>(smem + C::OFF_G);
  const Abort ab{abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
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
  const uint32_t tO = tmem + 256;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const uint64_t pol_kv = l2_policy_evict_last();
      const uint64_t pol_q = l2_policy_evict_first();
      mbar_expect_tx(q_full, C::QCH * kChunk);
      for (int c = 0; c < C::QCH; ++c)
        tma_load_3d_hint(smem + C::OFF_Q + c * kChunk, &tmQ, q_full, c * 64, h, seq_start + q0, pol_q);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int n = 0; n <= nt && ok; ++n) {
        if (n < nt) {
          const int y = seq_start + (hi_t - n) * kBN;
          for (int c = 0; c < C::KCH && ok; ++c) {
            ok = wait_bar(&kv_empty[stage], phase ^ 1, ab);
            if (!ok) break;
            mbar_expect_tx(&kv_full[stage], kChunk);
            tma_load_3d_hint(smem + C::OFF_RING + stage * kChunk, &tmK, &kv_full[stage], c * 64, kvh, y,
                             pol_kv);
            if (++stage == C::NST) { stage = 0; phase ^= 1; }
          }
        }
        if (n >= 1 && ok) {
          const int y = seq_start + (hi_t - (n - 1)) * kBN;
          for (int c = 0; c < C::VCH && ok; ++c) {
            ok = wait_bar(&kv_empty[stage], phase ^ 1, ab);
            if (!ok) break;
            mbar_expect_tx(&kv_full[stage], kChunk);
            tma_load_3d_hint(smem + C::OFF_RING + stage * kChunk, &tmV, &kv_full[stage], dv0 + c * 64, kvh, y,
                             pol_kv);
            if (++stage == C::NST) { stage = 0; phase ^= 1; }
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16(128, kBN, false, false);
      // P V per pair of 64-column value chunks in adjacent ring stages as one N = 128 MMA (LBO =
      // one stage; an N = 64 MMA costs nearly as much as an N = 128 one), a lone chunk with N = 64
      const uint32_t idPV = idesc_bf16(128, 64, false, true);
      const uint32_t idPV2 = idesc_bf16(128, 128, false, true);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q);
      const uint32_t sRing = smem_u32(smem + C::OFF_RING);
      uint32_t stage = 0, phase = 0;
      bool ok = wait_bar(q_full, 0, ab);
      for (int n = 0; n <= nt && ok; ++n) {
        if (n < nt) {
          const int b = n & 1;
          if (n >= 2) ok = wait_bar(&pv_done[b], ((n - 2) >> 1) & 1, ab);
          if (!ok) break;
          tc_fence_after();
          const uint32_t dS = tmem + b * 128;
          for (int c = 0; c < C::KCH && ok; ++c) {
            ok = wait_bar(&kv_full[stage], phase, ab);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = sdesc_sw128(sQ + c * kChunk + k * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(sRing + stage * kChunk + k * 32, 16, 1024);
              mma_ss(dS, ad, bd, idS, (c | k) != 0);
            }
            mma_commit(&kv_empty[stage]);
            if (++stage == C::NST) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          mma_commit(&s_full[b]);
        }
        if (n >= 1) {
          const int m = n - 1, bm = m & 1;
          ok = wait_bar(&p_full[bm], (m >> 1) & 1, ab);
          if (!ok) break;
          tc_fence_after();
          const uint32_t aP = tmem + bm * 128;
          for (int c = 0; c < C::VCH && ok;) {
            const bool pair = c + 1 < C::VCH && stage + 1 < C::NST;
            ok = wait_bar(&kv_full[stage], phase, ab);
            if (ok && pair) ok = wait_bar(&kv_full[stage + 1], phase, ab);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t bd = sdesc_sw128(sRing + stage * kChunk + k * 2048, kChunk, 1024);
              mma_ts(tO + c * 64, aP + k * 8, bd, pair ? idPV2 : idPV, (m > 0 || k > 0) ? 1u : 0u);
            }
            for (int u = 0; u < (pair ? 2 : 1); ++u) {
              mma_commit(&kv_empty[stage]);
              if (++stage == C::NST) { stage = 0; phase ^= 1; }
            }
            c += pair ? 2 : 1;
          }
          if (!ok) break;
          mma_commit(&pv_done[bm]);
        }
      }
      if (!ok) {
        // let every issued MMA retire before TMEM is released
        mma_commit(drain);
        mbar_wait(drain, 0, nullptr);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int il = q0 + r;
    const bool row_valid = il < len;
    const int tok = seq_start + (row_valid ? il : len - 1);
    const bool has_gate = p.gT != nullptr;
    // G_i is the same for every key of the row: the scores are kept without it (the softmax
    // does not change), the sink logit is shifted by -G_i, and G_i returns in the LSE
    float m = p.sink ? __ldg(p.sink + h) * kLog2e - (has_gate ? __ldg(p.gT + (size_t)h * p.total + tok) : 0.f)
                     : neg_inf();
    float l = p.sink ? 1.f : 0.f;
    bool ok = true;
    if (!has_gate) {
      // no gate: the G_j buffers stay zero
      for (int u = lane; u < 2 * kBN; u += 32) sG[quarter * 2 * kBN + u] = 0.f;
      __syncwarp();
    }
    for (int n = 0; n < nt; ++n) {
      const int jt = hi_t - n;
      const int j0 = jt * kBN;
      const int b = n & 1;
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
      tc_fence_after();
      uint32_t sv[128];
      tmem_ld32(tmem + lane_off + b * 128 + 0, sv);
      tmem_ld32(tmem + lane_off + b * 128 + 32, sv + 32);
      tmem_ld32(tmem + lane_off + b * 128 + 64, sv + 64);
      tmem_ld32(tmem + lane_off + b * 128 + 96, sv + 96);
      tmem_ld_wait();
      const bool need_mask = (jt == hi_t) || (p.window > 0 && j0 < q0 + kBM - p.window);
      // visible key columns of this row within the tile: causal j <= i, window i - j < W
      const int jmax = il - j0;
      const int jmin = p.window > 0 ? il - p.window + 1 - j0 : -(1 << 30);
      // row max with 8 independent partial maxima (a single 128-long chain is latency-bound)
      float mxp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mxp[e] = neg_inf();
      if (need_mask) {
#pragma unroll
        for (int j = 0; j < 128; j += 2) {
          float t0 = fmaf(__uint_as_float(sv[j]), p.scale_log2, gj[j]);
          float t1 = fmaf(__uint_as_float(sv[j + 1]), p.scale_log2, gj[j + 1]);
          t0 = (j >= jmin && j <= jmax) ? t0 : neg_inf();
          t1 = (j + 1 >= jmin && j + 1 <= jmax) ? t1 : neg_inf();
          sv[j] = __float_as_uint(t0);
          sv[j + 1] = __float_as_uint(t1);
          mxp[(j >> 1) & 7] = fmax3(mxp[(j >> 1) & 7], t0, t1);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 128; j += 2) {
          const float t0 = fmaf(__uint_as_float(sv[j]), p.scale_log2, gj[j]);
          const float t1 = fmaf(__uint_as_float(sv[j + 1]), p.scale_log2, gj[j + 1]);
          sv[j] = __float_as_uint(t0);
          sv[j + 1] = __float_as_uint(t1);
          mxp[(j >> 1) & 7] = fmax3(mxp[(j >> 1) & 7], t0, t1);
        }
      }
      const float mx = fmax3(fmax3(mxp[0], mxp[1], mxp[2]), fmax3(mxp[3], mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7]));
      const float m_new = fmaxf(m, mx);
      const bool need = m_new > m + kRescale;
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? ex2(m - m_new) : 1.f;
        if (n > 0) {
          ok = wait_bar(&pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, ab);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < DVC / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + lane_off + c * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
            tmem_st32(tO + lane_off + c * 32, ov);
          }
          tmem_st_wait();
        }
        l *= alpha;
        if (need) m = m_new;
      }
      const float mu = (m == neg_inf()) ? 0.f : m;
      float lsp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) lsp[e] = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const float p0 = ex2(__uint_as_float(sv[half * 64 + 2 * jj]) - mu);
          const float p1 = ex2(__uint_as_float(sv[half * 64 + 2 * jj + 1]) - mu);
          lsp[jj & 7] += p0 + p1;
          pk[jj] = pack_bf16x2(p0, p1);
        }
        tmem_st32(tmem + lane_off + b * 128 + half * 32, pk);
      }
      l += ((lsp[0] + lsp[1]) + (lsp[2] + lsp[3])) + ((lsp[4] + lsp[5]) + (lsp[6] + lsp[7]));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[b]);
    }
    if (ok) ok = wait_bar(&pv_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1, ab);
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      uint16_t* orow = p.o + (size_t)(seq_start + (row_valid ? il : 0)) * p.o_ts + (size_t)h * p.o_hs + dv0;
#pragma unroll 1
      for (int c = 0; c < DVC / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tO + lane_off + c * 32, ov);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          pk[j] = pack_bf16x2(__uint_as_float(ov[2 * j]) * inv_l, __uint_as_float(ov[2 * j + 1]) * inv_l);
        if (row_valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
      }
      if (row_valid && blockIdx.z == 0) {
        const float gi = has_gate ? __ldg(p.gT + (size_t)h * p.total + tok) : 0.f;
        p.lse[(size_t)h * p.total + seq_start + il] = (m + gi + log2f(l)) * kLn2;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // give copies already in flight time to land before the CTA's shared memory goes away
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DQK, int DVC>
cudaError_t launch_t(const FwdParams& p, const FwdMaps& maps, int num_tiles, cudaStream_t s) {
  using C = FwdCfg<DQK, DVC>;
  auto kern = prefill_fwd_kernel<DQK, DVC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.hq, num_tiles, p.dv / DVC);  // heads fastest, so every head's heavy tiles go first
  kern<<<grid, kThreads, C::SMEM, s>>>(maps.q, maps.k, maps.v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_fwd(const FwdParams& p, const FwdMaps& maps, int num_tiles, cudaStream_t s) {
  if (p.dqk == 64 && p.dv_chunk == 64) return launch_t<64, 64>(p, maps, num_tiles, s);
  if (p.dqk == 128 && p.dv_chunk == 128) return launch_t<128, 128>(p, maps, num_tiles, s);
  if (p.dqk == 256 && p.dv_chunk == 256) return launch_t<256, 256>(p, maps, num_tiles, s);
  if (p.dqk == 512 && p.dv_chunk == 256) return launch_t<512, 256>(p, maps, num_tiles, s);
  return cudaErrorInvalidValue;
}

}  // namespace gcs
