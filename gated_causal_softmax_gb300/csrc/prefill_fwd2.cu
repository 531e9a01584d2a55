// Prefill forward for head dims <= 128: two 128-row query tiles per CTA (fla-org/
// flash-linear-attention #1322 "Gluon attention backend with large head dimensions",
// Description: causal attention with log gates, sliding windows and a sink bias).
//
// Same arithmetic as prefill_fwd.cu; the difference is the schedule.  One CTA takes two
// 128-row query tiles A and B: with a GQA group of even size, the same rows of two query heads
// of the group (same causal range, so both tiles take part in every key tile); otherwise 256
// query rows of one head (rows q0..q0+127 and q0+128..q0+255).  Each tile has
// its own TMEM score buffer and accumulator (S_A, S_B, O_A, O_B: 4 x 128 columns) and its
// own softmax warpgroup, and the MMA issuer interleaves them
//     PV_A(n), S_A(n+1), PV_B(n), S_B(n+1), ...
// so one warpgroup's exponentials overlap the other tile's MMAs, and both tiles share every
// K / V tile loaded into shared memory.
//
// Warp roles (384 threads): warp 0 TMA producer (Q_A, Q_B once; K and V chunks through a
// ring), warp 1 tcgen05 issuer, warps 2-3 idle; warps 4-7 softmax of tile A, warps 8-11
// softmax of tile B (one thread per row).  setmaxnreg moves registers from the first
// warpgroup to the softmax warpgroups, which keep a 128-column score row in registers.
#include "kernels.h"
#include "sm103_ptx.cuh"
#include "tiles.cuh"

namespace gcs {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kChunk = 128 * 128;
constexpr int kThreads = 384;
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

template <int D>
struct Fwd2Cfg {
  static constexpr int CH = D / 64;
  static constexpr int TILE = CH * kChunk;                 // one K or V tile (128 keys)
  static constexpr int NST = 8 / CH;                       // ring stages, one tile each
  static constexpr int OFF_Q = 0;                           // [2 tiles][CH] chunks
  static constexpr int OFF_RING = 2 * CH * kChunk;
  static constexpr int OFF_G = OFF_RING + NST * TILE;      // [2 tiles][4 warps][2][128] floats
  static constexpr int OFF_BAR = OFF_G + 2 * 4 * 2 * kBN * 4;
  static constexpr int OFF_MISC = OFF_BAR + (2 * NST + 16) * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// Register split (per thread): warpgroup 0 (producer, MMA, 2 idle warps) 112, the two softmax
// warpgroups 192 each: 128 x 112 + 256 x 192 = 63488 <= 384 threads x 168 at launch (both
// tile pairings compile without spills at this split; at 120 / 184 the softmax spills).
__device__ __forceinline__ void reg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 112;\n" ::: "memory"); }
__device__ __forceinline__ void reg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 192;\n" ::: "memory"); }

// HP (head pairs, GQA groups of even size): tiles A and B are the same 128 query rows of two
// query heads of one group, so they share every key tile over the same causal range.
// Otherwise they are 256 consecutive query rows of one head.
template <int D, bool HP>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_fwd2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = Fwd2Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align_1k(smem_raw);

  // heaviest query tiles (or 256-row pairs) first
  TileRef tr;
  if (!lpt_tile(p.cu_seqlens, p.num_seqs, HP ? kBM : 2 * kBM, blockIdx.y, tr)) return;
  const int seq_start = tr.start, len = tr.len;
  // tile x: query head h0 + (HP ? x : 0), first query row q0 + (HP ? 0 : 128 x)
  const int h0 = HP ? 2 * (int)blockIdx.x : (int)blockIdx.x;
  const int kvh = h0 / (p.hq / p.hkv);
  const int q0 = HP ? tr.u * kBM : tr.u * 2 * kBM;
  const int qt[2] = {q0 / kBM, HP ? q0 / kBM : q0 / kBM + 1};
  const bool valid_b = HP || q0 + kBM < len;
  int lo[2];
  for (int x = 0; x < 2; ++x) {
    const int lo_j = qt[x] * kBM - p.window + 1;
    lo[x] = (p.window > 0 && lo_j > 0) ? lo_j / kBN : 0;
  }
  const int hi_t = valid_b ? qt[1] : qt[0];
  const int lo_t = lo[0];
  const int nt = hi_t - lo_t + 1;
  // tile x takes part in key tile n (jt = hi_t - n) when jt lies in [lo[x], qt[x]], i.e. when
  // n lies in [hi_t - qt[x], hi_t - lo[x]] (an empty range for an invalid tile B)
  const int n_first[2] = {hi_t - qt[0], valid_b ? hi_t - qt[1] : nt};
  const int n_last[2] = {hi_t - lo[0], valid_b ? hi_t - lo[1] : -1};
  auto part = [&](int x, int n) -> bool { return n >= n_first[x] && n <= n_last[x]; };

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;              // [NST]
  uint64_t* empty = bars + C::NST;    // [NST]
  uint64_t* q_full = bars + 2 * C::NST;
  uint64_t* s_full = q_full + 1;      // [2 tiles]
  uint64_t* p_full = q_full + 3;      // [2 tiles]
  uint64_t* pv_done = q_full + 5;     // [2 tiles]
  uint64_t* drain = q_full + 7;
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
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 4);
      mbar_init(&pv_done[x], 1);
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

  if (warp < 4) {
    reg_dec();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const uint64_t pol_kv = l2_policy_evict_last();
      const uint64_t pol_q = l2_policy_evict_first();
      mbar_expect_tx(q_full, 2 * C::CH * kChunk);
      for (int x = 0; x < 2; ++x)
        for (int c = 0; c < C::CH; ++c)
          tma_load_3d_hint(smem + C::OFF_Q + (x * C::CH + c) * kChunk, &tmQ, q_full, c * 64, HP ? h0 + x : h0,
                           seq_start + q0 + (HP ? 0 : x * kBM), pol_q);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int n = 0; n < nt && ok; ++n) {
        const int y = seq_start + (hi_t - n) * kBN;
        for (int kv = 0; kv < 2 && ok; ++kv) {
          ok = wait_bar(&empty[stage], phase ^ 1, ab);
          if (!ok) break;
          mbar_expect_tx(&full[stage], C::TILE);
          for (int c = 0; c < C::CH; ++c)
            tma_load_3d_hint(smem + C::OFF_RING + stage * C::TILE + c * kChunk, kv ? &tmV : &tmK, &full[stage],
                             c * 64, kvh, y, pol_kv);
          if (++stage == C::NST) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      // One MMA with N < 128 takes nearly as long as one with N = 128, so P V is issued with
      // N = D across the D/64 value chunks of a ring stage (LBO = one chunk).  Descriptors are built once; an operand offset is added to the address field
      // (shared-memory addresses stay below 2^18, so the 14-bit field never carries).
      const uint32_t idS = idesc_bf16(128, kBN, false, false);
      const uint32_t idPV = idesc_bf16(128, D, false, true);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
      const uint64_t dK0 = sdesc_sw128(smem_u32(smem + C::OFF_RING), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + C::OFF_RING), kChunk, 1024);
      constexpr uint32_t kChunk16 = kChunk >> 4;
      constexpr uint32_t kTile16 = C::TILE >> 4;
      // Waits are batched ahead of runs of back-to-back MMAs: the tensor pipe has almost no
      // issue queue, so each stall of this thread on a barrier leaves it idle.
      uint32_t stage = 0, phase = 0;  // ring position of the next tile (K, V, K, V, ...)
      auto next = [&](uint32_t& st, uint32_t& ph) {
        st = stage;
        ph = phase;
        if (++stage == C::NST) {
          stage = 0;
          phase ^= 1;
        }
      };
      auto mma_s = [&](int x, uint32_t st) {  // S_x = Q_x K^T over ring stage st
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          const uint64_t a = dQ0 + (x * C::CH + c) * kChunk16, b = dK0 + st * kTile16 + c * kChunk16;
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ss(tmem + 128 * x, a + 2 * k, b + 2 * k, idS, (c | k) != 0);
        }
        mma_commit(&s_full[x]);
      };
      int kp[2] = {0, 0};  // PV issued per tile (accumulate flag and p_full parity)
      uint32_t sk = 0, pk = 0;
      next(sk, pk);  // K of key tile 0
      bool ok = wait_bars(ab, q_full, 0, &full[sk], pk);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (part(x, 0)) mma_s(x, sk);
        mma_commit(&empty[sk]);
      }
      for (int n = 0; n < nt && ok; ++n) {
        const bool more = n + 1 < nt;
        uint32_t sv, pv, sk1 = 0, pk1 = 0;
        next(sv, pv);  // V of key tile n
        if (more) next(sk1, pk1);  // K of key tile n + 1
        bool first = true;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!ok) break;
          const bool do_pv = part(x, n), do_s = more && part(x, n + 1);
          if (!do_pv && !do_s) continue;
          // the first batch also waits for this key tile's V and the next one's K
          if (first)
            ok = wait_bars(ab, &full[sv], pv, more ? &full[sk1] : nullptr, pk1, do_pv ? &p_full[x] : nullptr,
                           kp[x] & 1);
          else if (do_pv)
            ok = wait_bars(ab, &p_full[x], kp[x] & 1);
          first = false;
          if (!ok) break;
          tc_fence_after();
          if (do_pv) {
            const uint64_t b = dV0 + sv * kTile16;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ts(tmem + 256 + 128 * x, tmem + 128 * x + k * 8, b + 128 * k, idPV, (kp[x] > 0 || k > 0) ? 1u : 0u);
            mma_commit(&pv_done[x]);
            ++kp[x];
          }
          // next scores of this tile over its buffer (P was read by the PV above)
          if (do_s) mma_s(x, sk1);
        }
        if (!ok) break;
        mma_commit(&empty[sv]);
        if (more) mma_commit(&empty[sk1]);
      }
      if (!ok) {
        mma_commit(drain);
        mbar_wait(drain, 0, nullptr);
      }
    }
    __syncwarp();
  } else {
    reg_inc();
    // ------------------------------------------------------------ softmax, tile x
    const int x = (warp - 4) >> 2;
    const int my_first = x ? n_first[1] : n_first[0], my_last = x ? n_last[1] : n_last[0];
    const int my_qt = x ? qt[1] : qt[0];
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + 128 * x, tO = tmem + lane_off + 256 + 128 * x;
    const int h = HP ? h0 + x : h0;
    const int xq0 = q0 + (HP ? 0 : x * kBM);
    const int il = xq0 + r;
    const bool row_valid = il < len;
    const int tok = seq_start + (row_valid ? il : len - 1);
    const bool has_gate = p.gT != nullptr;
    // The row's own G_i is the same for every key, so the scores are kept without it (the
    // softmax does not change) and it returns in the LSE; the sink logit, which carries no
    // G_i, is shifted by -G_i instead.
    float m = p.sink ? __ldg(p.sink + h) * kLog2e - (has_gate ? __ldg(p.gT + (size_t)h * p.total + tok) : 0.f)
                     : neg_inf();
    float l = p.sink ? 1.f : 0.f;
    float* sG = reinterpret_cast<float*>(smem + C::OFF_G) + (x * 4 + quarter) * 2 * kBN;
    if (!has_gate) {
      for (int u = lane; u < 2 * kBN; u += 32) sG[u] = 0.f;
      __syncwarp();
    }
    bool ok = true;
    int kx = 0;  // key tiles processed by this tile
    for (int n = 0; n < nt; ++n) {
      if (n < my_first || n > my_last) continue;
      const int jt = hi_t - n, j0 = jt * kBN;
      float* gj = sG + (kx & 1) * kBN;  // this warp's copy of -G_j for the key tile
      if (has_gate) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int jl = j0 + lane * 4 + u;
          gj[lane * 4 + u] = (jl < len) ? -__ldg(p.gT + (size_t)h * p.total + seq_start + jl) : 0.f;
        }
        __syncwarp();
      }
      ok = wait_bar(&s_full[x], kx & 1, ab);
      if (!ok) break;
      tc_fence_after();
      uint32_t sv[128];
      tmem_ld32(tS + 0, sv);
      tmem_ld32(tS + 32, sv + 32);
      tmem_ld32(tS + 64, sv + 64);
      tmem_ld32(tS + 96, sv + 96);
      tmem_ld_wait();
      const bool need_mask = (jt == my_qt) || (p.window > 0 && j0 < xq0 + kBM - p.window);
      const int jmax = il - j0;
      const int jmin = p.window > 0 ? il - p.window + 1 - j0 : -(1 << 30);
      float mxp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mxp[e] = neg_inf();
      // t = s scale log2e - G_j (one FMA), maxima three at a time; -G_j read as 16-B broadcast
      // loads: shared-memory loads compete with the operand reads of running MMAs, so fewer,
      // wider ones
      const float4* gj4 = reinterpret_cast<const float4*>(gj);
      if (need_mask) {
#pragma unroll
        for (int j4 = 0; j4 < 32; ++j4) {
          const float4 g4 = gj4[j4];
          const float gs[4] = {g4.x, g4.y, g4.z, g4.w};
          float t[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * j4 + e;
            t[e] = fmaf(__uint_as_float(sv[j]), p.scale_log2, gs[e]);
            t[e] = (j >= jmin && j <= jmax) ? t[e] : neg_inf();
            sv[j] = __float_as_uint(t[e]);
          }
          mxp[(2 * j4) & 7] = fmax3(mxp[(2 * j4) & 7], t[0], t[1]);
          mxp[(2 * j4 + 1) & 7] = fmax3(mxp[(2 * j4 + 1) & 7], t[2], t[3]);
        }
      } else {
#pragma unroll
        for (int j4 = 0; j4 < 32; ++j4) {
          const float4 g4 = gj4[j4];
          const float gs[4] = {g4.x, g4.y, g4.z, g4.w};
          float t[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * j4 + e;
            t[e] = fmaf(__uint_as_float(sv[j]), p.scale_log2, gs[e]);
            sv[j] = __float_as_uint(t[e]);
          }
          mxp[(2 * j4) & 7] = fmax3(mxp[(2 * j4) & 7], t[0], t[1]);
          mxp[(2 * j4 + 1) & 7] = fmax3(mxp[(2 * j4 + 1) & 7], t[2], t[3]);
        }
      }
      const float mx = fmax3(fmax3(mxp[0], mxp[1], mxp[2]), fmax3(mxp[3], mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7]));
      const float m_new = fmaxf(m, mx);
      const bool need = m_new > m + kRescale;
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? ex2(m - m_new) : 1.f;
        if (kx > 0) {
          // O holds the previous key tiles: wait for their PV before scaling it
          ok = wait_bar(&pv_done[x], (kx - 1) & 1, ab);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + c * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
            tmem_st32(tO + c * 32, ov);
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
        tmem_st32(tS + half * 32, pk);
      }
      l += ((lsp[0] + lsp[1]) + (lsp[2] + lsp[3])) + ((lsp[4] + lsp[5]) + (lsp[6] + lsp[7]));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[x]);
      ++kx;
    }
    if (ok && kx > 0) ok = wait_bar(&pv_done[x], (kx - 1) & 1, ab);
    if (ok && kx > 0) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      uint16_t* orow = p.o + (size_t)(seq_start + (row_valid ? il : 0)) * p.o_ts + (size_t)h * p.o_hs;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tO + c * 32, ov);
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
      // G_i read again here rather than kept live through the loop
      const float gi = has_gate ? __ldg(p.gT + (size_t)h * p.total + tok) : 0.f;
      if (row_valid) p.lse[(size_t)h * p.total + seq_start + il] = (m + gi + log2f(l)) * kLn2;
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

template <int D, bool HP>
cudaError_t launch_t(const FwdParams& p, const FwdMaps& maps, int num_units, cudaStream_t s) {
  using C = Fwd2Cfg<D>;
  auto kern = prefill_fwd2_kernel<D, HP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<dim3(HP ? p.hq / 2 : p.hq, num_units), kThreads, C::SMEM, s>>>(maps.q, maps.k, maps.v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_fwd2(const FwdParams& p, const FwdMaps& maps, cudaStream_t s) {
  // GQA groups of even size pair two query heads per CTA over 128-row tiles; otherwise two
  // consecutive 128-row tiles of one head (an upper bound on the tiles of the packed batch:
  // the CTAs past the last tile return at once)
  const bool hp = (p.hq / p.hkv) % 2 == 0;
  const int units = hp ? (p.total + kBM - 1) / kBM + p.num_seqs : (p.total + 2 * kBM - 1) / (2 * kBM) + p.num_seqs;
  if (p.dqk == 64 && p.dv == 64) return hp ? launch_t<64, true>(p, maps, units, s) : launch_t<64, false>(p, maps, units, s);
  if (p.dqk == 128 && p.dv == 128)
    return hp ? launch_t<128, true>(p, maps, units, s) : launch_t<128, false>(p, maps, units, s);
  return cudaErrorInvalidValue;
}

}  // namespace gcs
