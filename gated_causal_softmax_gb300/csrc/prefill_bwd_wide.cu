// Prefill backward for head dims above 128 (fla-org/flash-linear-attention #1322
// "Gluon attention backend with large head dimensions": Description, head dims through
// 512; Oct 3 / Oct 5 comments for the fp32 sink / gate reductions and the fp32 dQ buffer).
//
// At 128 key rows per tile the fp32 dK and dV accumulators of a 256/512-wide head need
// 768-1024 TMEM columns (512 exist), and the K / V tiles alone exceed shared memory.  The
// work of one (128-key tile, kv head) is therefore split over CTAs by output columns:
//   role V   (kind 0):  dV[:, v0 : v0+256)                 needs P  -> recomputes S
//   role KQ  (kind 1):  dK[:, k0 : k0+256), dQ[:, k0 : k0+256)  needs dS -> recomputes S, dP
//   role K   (kind 2):  dK[:, k0 : k0+256) only, for the deterministic backward, whose dQ and
//                       dS row sums come from the query-stationary pass (prefill_bwd_wide_dq.cu)
// Every role recomputes the full-width contractions it needs; the extra work is the price
// of fitting the accumulators in TMEM.  The K-side and dV roles of a call run in one launch.  Operands stream through a ring of 16 KB stages
// (128 x 64 or 64 x 64 bf16 chunks, 128-B swizzle); the K columns a role keeps using
// (its own 256 dims) stay resident.  One softmax warpgroup, one thread per key row.
// Per query step of BM rows (s = step; the pipeline is sequential per step, except that role V at
// Dqk = 256 computes step s + 1's S^T into a second TMEM buffer while step s's P^T is formed):
//     S^T = K Q^T (TMEM)   [dP^T = V dO^T (TMEM)]   P^T / dS^T in fp32, bf16 operands
//     role V:  dV  += P^T dO[:, v0..]
//     role KQ: dK  += dS^T Q[:, k0..];  dQ^T[k0..] = K[:, k0..]^T dS^T -> fp32 reduce-adds
//     role K:  dK  += dS^T Q[:, k0..]
// Row / column sums of dS (gate and sink gradients) are taken by the KQ role with k0 = 0; the
// K role takes the column sums only (thread-local per key row and head, added once to a
// zeroed entry, so they do not depend on scheduling).
#include "kernels.h"
#include "sm103_ptx.cuh"
#include "tiles.cuh"

namespace gcs {
namespace {

constexpr int kBN = 128;
constexpr int kThreads = 192;
constexpr int kStage = 16384;
constexpr int kW = 256;  // output columns per role
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// BM = query rows per step: 128 for the dV and dK-only roles (N = 128 MMAs), 64 for the
// dK + dQ role, whose dQ^T halves need the TMEM columns that 128-row steps would take.
template <int DQK, int DV, int KIND, int BM>
struct WideCfg {
  static_assert(BM == 64 || BM == 128, "query step");
  static_assert(KIND != 1 || BM == 64, "the dQ role keeps 64-row steps");
  static constexpr int KCH = DQK / 64, VCH = DV / 64, WCH = kW / 64;
  static constexpr int NRES = (KIND >= 1 ? kW : (DQK < kW ? DQK : kW)) / 64;  // resident K chunks
  static constexpr int NST = 8;
  static constexpr int OFF_KRES = 0;
  static constexpr int OFF_RING = OFF_KRES + NRES * kStage;
  static constexpr int OFF_DS = OFF_RING + NST * kStage;
  static constexpr int OFF_VEC = OFF_DS + (KIND == 1 ? kStage : 0);  // [2][2][64] floats
  static constexpr int OFF_BAR = OFF_VEC + 2 * 2 * BM * 4;
  static constexpr int OFF_MISC = OFF_BAR + (2 * NST + 16) * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  // TMEM: S^T 0..BM-1, dP^T BM..2BM-1, accumulator (dV or dK) 2BM..2BM+255, dQ^T halves 384..511
  static constexpr int T_S = 0, T_DP = BM, T_ACC = 2 * BM, T_DQ = 384;
  static_assert(T_ACC + 256 <= 512, "TMEM columns");
};

// One role of one (128-key tile, kv head): role index `role` of its kind (output columns
// 256 role ..), tile blockIdx.y, kv head blockIdx.x.
template <int DQK, int DV, int KIND, int BM>
__device__ __forceinline__ void wide_role(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                          const CUtensorMap& tmDO, const BwdParams& p, int role) {
  using C = WideCfg<DQK, DV, KIND, BM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align_1k(smem_raw);

  TileRef tr;
  if (!lpt_tile(p.cu_seqlens, p.num_seqs, kBN, blockIdx.y, tr)) return;
  const int seq_start = tr.start, len = tr.len, jt = tr.n - 1 - tr.u;
  const int kvh = blockIdx.x;
  const int w0 = role * kW;               // v0 (role V) or k0 (roles KQ, K)
  const int res0 = (KIND >= 1) ? w0 / 64 : 0;  // first resident K chunk
  const int group = p.hq / p.hkv;
  const int j0 = jt * kBN;
  const int it_lo = j0 / BM;
  int i_hi = len - 1;
  if (p.window > 0) i_hi = min(i_hi, j0 + kBN - 1 + p.window - 1);
  const int n_it = i_hi / BM - it_lo + 1;
  const int nsteps = n_it * group;
  const bool sums = (KIND >= 1) && (w0 == 0);  // this role takes the dS column (and row) sums
  // Role V double-buffers S^T (its dP^T columns are free) when the next step's score operands and
  // this step's dO chunks fit in the ring together (Dqk = 256: K resident, 4 + 4 chunks of 8), so
  // that the producer can stage this step's dO while the next scores stream.  At Dqk = 512 the 12
  // score chunks would push the dO loads behind them and expose their latency (a double buffer
  // there measured slower), so that shape keeps the single buffer.
  constexpr bool DB = KIND == 0 && (2 * C::KCH - C::NRES) + C::WCH <= C::NST;
  static_assert(C::KCH > 0 && C::VCH > 0 && C::WCH > 0, "head-dim chunks");

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;                 // [NST]
  uint64_t* empty = bars + C::NST;       // [NST]
  uint64_t* kv_full = bars + 2 * C::NST;
  uint64_t* vec_full = kv_full + 1;      // [2]
  uint64_t* vec_empty = kv_full + 3;     // [2]
  uint64_t* s_full = kv_full + 5;
  uint64_t* p_full = kv_full + 6;
  uint64_t* mma_done = kv_full + 7;
  uint64_t* dq_free = kv_full + 8;
  uint64_t* drain = kv_full + 9;
  // role V with DB (below): S^T is double-buffered, so the scores of step s + 1
  // are computed while the key-row warps turn step s into P^T; per buffer b = s & 1 a scores-ready
  // and a P^T-ready barrier, and one barrier for the accumulator after the last step
  uint64_t* s_full2 = kv_full + 10;  // [2]
  uint64_t* p_full2 = kv_full + 12;  // [2]
  uint64_t* acc_done = kv_full + 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const Abort ab{abort_flag, p.status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(kv_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&vec_full[b], 1);
      mbar_init(&vec_empty[b], 4);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 4);
    mbar_init(mma_done, 1);
    mbar_init(dq_free, 4);
    mbar_init(drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full2[b], 1);
      mbar_init(&p_full2[b], 4);
    }
    mbar_init(acc_done, 1);
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
    uint32_t stage = 0, phase = 0;
    // (x, hd, y) = (column within the head, head, token)
    auto issue = [&](const CUtensorMap* m, int x, int hd, int y, uint32_t bytes) -> bool {
      if (!wait_bar(&empty[stage], phase ^ 1, ab)) return false;
      mbar_expect_tx(&full[stage], bytes);
      tma_load_3d(smem + C::OFF_RING + stage * kStage, m, &full[stage], x, hd, y);
      if (++stage == C::NST) {
        stage = 0;
        phase ^= 1;
      }
      return true;
    };
    if (lane == 0) {
      mbar_expect_tx(kv_full, C::NRES * kStage);
      for (int c = 0; c < C::NRES; ++c)
        tma_load_3d(smem + C::OFF_KRES + c * kStage, &tmK, kv_full, (res0 + c) * 64, kvh, seq_start + j0);
    }
    if constexpr (DB) {
      // the per-column vectors of step s: (G_i - LSE_i) log2 e and delta_i, into buffer s & 1
      auto put_vectors = [&](int s) -> bool {
        const int h = kvh * group + s / n_it;
        const int i0 = (it_lo + s % n_it) * BM;
        bool okv = true;
        if (lane == 0) okv = wait_bar(&vec_empty[s & 1], ((s >> 1) & 1) ^ 1, ab);
        okv = __shfl_sync(0xffffffffu, okv ? 1 : 0, 0) != 0;
        if (!okv) return false;
        float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC) + (s & 1) * 2 * BM;
  #pragma unroll
        for (int u = 0; u < BM / 32; ++u) {
          const int c = lane * (BM / 32) + u;
          const int i = i0 + c;
          float colterm = 0.f, dl = 0.f;
          if (i < len) {
            const size_t idx = (size_t)h * p.total + seq_start + i;
            colterm = -__ldg(p.lse + idx) * kLog2e;
            if (p.gT) colterm += __ldg(p.gT + idx);
            dl = __ldg(p.delta + idx);
          }
          vec[c] = colterm;
          vec[BM + c] = dl;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&vec_full[s & 1]);
        return true;
      };
      // operands of step s's score MMAs: streamed K chunks and the Q chunks (lane 0)
      auto put_score_operands = [&](int s) -> bool {
        const int h = kvh * group + s / n_it;
        const int yq = seq_start + (it_lo + s % n_it) * BM, yk = seq_start + j0;
        bool okl = true;
        if (lane == 0) {
          for (int c = 0; c < C::KCH && okl; ++c) {
            if (c < res0 || c >= res0 + C::NRES) okl = issue(&tmK, c * 64, kvh, yk, kStage);
            if (okl) okl = issue(&tmQ, c * 64, h, yq, BM * 128);
          }
        }
        return __shfl_sync(0xffffffffu, okl ? 1 : 0, 0) != 0;
      };
      // consumption order of the MMA warp: S(0), then per step s: S(s + 1), dV(s)
      if (nsteps > 0) ok = put_score_operands(0) && put_vectors(0);
      for (int s = 0; s < nsteps && ok; ++s) {
        if (s + 1 < nsteps) ok = put_score_operands(s + 1) && put_vectors(s + 1);
        if (!ok) break;
        const int h = kvh * group + s / n_it;
        const int yq = seq_start + (it_lo + s % n_it) * BM;
        if (lane == 0)
          for (int c = 0; c < C::WCH && ok; ++c) ok = issue(&tmDO, w0 + c * 64, h, yq, BM * 128);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      }
    } else {
      for (int s = 0; s < nsteps && ok; ++s) {
        const int h = kvh * group + s / n_it;
        const int i0 = (it_lo + s % n_it) * BM;
        const int yq = seq_start + i0, yk = seq_start + j0;
        if (lane == 0) {
          for (int c = 0; c < C::KCH && ok; ++c) {
            if (c < res0 || c >= res0 + C::NRES) ok = issue(&tmK, c * 64, kvh, yk, kStage);
            if (ok) ok = issue(&tmQ, c * 64, h, yq, BM * 128);
          }
          if (KIND >= 1) {
            for (int c = 0; c < C::VCH && ok; ++c) {
              ok = issue(&tmV, c * 64, kvh, yk, kStage);
              if (ok) ok = issue(&tmDO, c * 64, h, yq, BM * 128);
            }
            for (int c = 0; c < C::WCH && ok; ++c) ok = issue(&tmQ, w0 + c * 64, h, yq, BM * 128);
          } else {
            for (int c = 0; c < C::WCH && ok; ++c) ok = issue(&tmDO, w0 + c * 64, h, yq, BM * 128);
          }
          if (ok) ok = wait_bar(&vec_empty[s & 1], ((s >> 1) & 1) ^ 1, ab);
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC) + (s & 1) * 2 * BM;
  #pragma unroll
        for (int u = 0; u < BM / 32; ++u) {
          const int c = lane * (BM / 32) + u;
          const int i = i0 + c;
          float colterm = 0.f, dl = 0.f;
          if (i < len) {
            const size_t idx = (size_t)h * p.total + seq_start + i;
            colterm = -__ldg(p.lse + idx) * kLog2e;
            if (p.gT) colterm += __ldg(p.gT + idx);
            dl = __ldg(p.delta + idx);
          }
          vec[c] = colterm;
          vec[BM + c] = dl;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&vec_full[s & 1]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16(128, BM, false, false);  // S^T, dP^T
      const uint32_t idAcc = idesc_bf16(128, 64, false, true);   // dV / dK, one 64-column chunk
      const uint32_t idAcc2 = idesc_bf16(128, 128, false, true); // two chunks in adjacent stages
      const uint32_t idDQ = idesc_bf16(128, BM, true, true);    // dQ^T half
      const uint32_t sRes = smem_u32(smem + C::OFF_KRES), sRing = smem_u32(smem + C::OFF_RING);
      const uint32_t sDS = smem_u32(smem + C::OFF_DS);
      uint32_t stage = 0, phase = 0;
      auto take = [&](uint32_t& addr) -> bool {  // wait for the current ring stage
        if (!wait_bar(&full[stage], phase, ab)) return false;
        tc_fence_after();
        addr = sRing + stage * kStage;
        return true;
      };
      auto advance = [&]() {
        if (++stage == C::NST) {
          stage = 0;
          phase ^= 1;
        }
      };
      auto give = [&]() {  // release the current stage once the MMAs issued so far retire
        mma_commit(&empty[stage]);
        advance();
      };
      bool ok = wait_bar(kv_full, 0, ab);
      if constexpr (DB) {
        // S^T = K Q^T over all of DQK (K chunk resident or streamed, Q chunk streamed) into the
        // columns at t_s
        auto scores = [&](uint32_t t_s) -> bool {
          for (int c = 0; c < C::KCH; ++c) {
            uint32_t a = 0, bq = 0;
            int kst = -1;
            if (c >= res0 && c < res0 + C::NRES) {
              a = sRes + (c - res0) * kStage;
            } else {
              if (!take(a)) return false;
              kst = stage;
              advance();
            }
            if (!take(bq)) return false;
  #pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(tmem + t_s, sdesc_sw128(a + k * 32, 16, 1024), sdesc_sw128(bq + k * 32, 16, 1024), idS,
                     (c | k) != 0);
            if (kst >= 0) mma_commit(&empty[kst]);
            give();
          }
          return true;
        };
        // accumulator += A x (dO or Q chunks): a pair of 64-column chunks in adjacent ring stages as
        // one N = 128 MMA (LBO = one stage; an N = 64 MMA costs nearly as much as an N = 128 one), a
        // lone chunk with N = 64
        auto accumulate = [&](uint32_t aT, bool first) -> bool {
          for (int c = 0; c < C::WCH;) {
            const bool pair = c + 1 < C::WCH && stage + 1 < C::NST;
            uint32_t bq = 0;
            if (!take(bq)) return false;
            if (pair && !wait_bar(&full[stage + 1], phase, ab)) return false;
            tc_fence_after();
  #pragma unroll
            for (int k = 0; k < BM / 16; ++k)
              mma_ts(tmem + C::T_ACC + c * 64, aT + k * 8, sdesc_sw128(bq + k * 2048, kStage, 1024),
                     pair ? idAcc2 : idAcc, (!first || k > 0) ? 1u : 0u);
            give();
            if (pair) give();
            c += pair ? 2 : 1;
          }
          return true;
        };
        // S(0); then per step s: S(s + 1) into the other buffer, wait for P^T(s), dV(s).  MMAs run
        // in issue order, so S(s + 2) (issued after dV(s)) overwrites buffer s & 1 only after dV(s)
        // has read P^T(s) there.
        if (ok && nsteps > 0) {
          ok = scores(C::T_S);
          if (ok) mma_commit(&s_full2[0]);
        }
        for (int s = 0; s < nsteps && ok; ++s) {
          if (s + 1 < nsteps) {
            ok = scores(C::T_S + ((s + 1) & 1) * BM);
            if (!ok) break;
            mma_commit(&s_full2[(s + 1) & 1]);
          }
          ok = wait_bar(&p_full2[s & 1], (s >> 1) & 1, ab);
          if (!ok) break;
          tc_fence_after();
          ok = accumulate(tmem + C::T_S + (s & 1) * BM, s == 0);
        }
        if (ok && nsteps > 0) mma_commit(acc_done);
      } else {
        for (int s = 0; s < nsteps && ok; ++s) {
          // S^T = K Q^T over all of DQK (K chunk resident or streamed, Q chunk streamed)
          for (int c = 0; c < C::KCH && ok; ++c) {
            uint32_t a = 0, bq = 0;
            int kst = -1;
            if (c >= res0 && c < res0 + C::NRES) {
              a = sRes + (c - res0) * kStage;
            } else {
              ok = take(a);
              if (!ok) break;
              kst = stage;
              advance();
            }
            ok = take(bq);
            if (!ok) break;
  #pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(tmem + C::T_S, sdesc_sw128(a + k * 32, 16, 1024), sdesc_sw128(bq + k * 32, 16, 1024), idS,
                     (c | k) != 0);
            if (kst >= 0) mma_commit(&empty[kst]);
            give();
          }
          if (!ok) break;
          if (KIND >= 1) {
            // dP^T = V dO^T over all of DV
            for (int c = 0; c < C::VCH && ok; ++c) {
              uint32_t a = 0, bq = 0;
              ok = take(a);
              if (!ok) break;
              const int vst = stage;
              advance();
              ok = take(bq);
              if (!ok) break;
  #pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_ss(tmem + C::T_DP, sdesc_sw128(a + k * 32, 16, 1024), sdesc_sw128(bq + k * 32, 16, 1024), idS,
                       (c | k) != 0);
              mma_commit(&empty[vst]);
              give();
            }
            if (!ok) break;
          }
          mma_commit(s_full);
          ok = wait_bar(p_full, s & 1, ab);
          if (!ok) break;
          tc_fence_after();
          // accumulator += (P^T or dS^T) x (dO or Q): a pair of 64-column chunks in adjacent ring
          // stages as one N = 128 MMA (LBO = one stage; an N = 64 MMA costs nearly as much as an
          // N = 128 one), a lone chunk with N = 64
          const uint32_t aT = tmem + (KIND >= 1 ? C::T_DP : C::T_S);
          for (int c = 0; c < C::WCH && ok;) {
            const bool pair = c + 1 < C::WCH && stage + 1 < C::NST;
            uint32_t bq = 0;
            ok = take(bq);
            if (ok && pair) ok = wait_bar(&full[stage + 1], phase, ab);
            if (!ok) break;
            tc_fence_after();
  #pragma unroll
            for (int k = 0; k < BM / 16; ++k)
              mma_ts(tmem + C::T_ACC + c * 64, aT + k * 8, sdesc_sw128(bq + k * 2048, kStage, 1024),
                     pair ? idAcc2 : idAcc, (s > 0 || k > 0) ? 1u : 0u);
            give();
            if (pair) give();
            c += pair ? 2 : 1;
          }
          if (!ok) break;
          if (KIND == 1) {
            if (s > 0) {
              ok = wait_bar(dq_free, (s - 1) & 1, ab);
              if (!ok) break;
              tc_fence_after();
            }
            // dQ^T for dims w0 .. w0+255: two M=128 halves from the resident K chunks
  #pragma unroll
            for (int hf = 0; hf < 2; ++hf)
  #pragma unroll
              for (int k = 0; k < 8; ++k)
                mma_ss(tmem + C::T_DQ + hf * 64, sdesc_sw128(sRes + 2 * hf * kStage + k * 2048, kStage, 1024),
                       sdesc_sw128(sDS + k * 2048, kStage, 1024), idDQ, k > 0);
          }
          mma_commit(mma_done);
        }
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
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::T_S, tDP = tmem + lane_off + C::T_DP;
    const int jl = j0 + r;
    const bool has_gate = p.gT != nullptr;
    const bool want_row = KIND == 1 && sums && p.dg_row != nullptr;
    uint8_t* sDS = smem + C::OFF_DS;
    float dgcol = 0.f, rowterm = 0.f;
    int cur_h = -1;
    bool ok = true;
    for (int s = 0; s < nsteps; ++s) {
      const int h = kvh * group + s / n_it;
      const int i0 = (it_lo + s % n_it) * BM;
      if (h != cur_h) {
        if (sums && cur_h >= 0 && has_gate && jl < len)
          red_add_f32(p.dg_col + (size_t)cur_h * p.total + seq_start + jl, dgcol);
        dgcol = 0.f;
        cur_h = h;
        rowterm = (has_gate && jl < len) ? -__ldg(p.gT + (size_t)h * p.total + seq_start + jl) : 0.f;
      }
      ok = wait_bar(&vec_full[s & 1], (s >> 1) & 1, ab);
      if (!ok) break;
      ok = DB ? wait_bar(&s_full2[s & 1], (s >> 1) & 1, ab) : wait_bar(s_full, s & 1, ab);
      if (!ok) break;
      tc_fence_after();
      // role V with DB: this step's score buffer
      const uint32_t tSs = tS + (DB ? (s & 1) * BM : 0);
      const float* vec = reinterpret_cast<const float*>(smem + C::OFF_VEC) + (s & 1) * 2 * BM;
      const bool need_mask = (i0 < j0 + kBN - 1) || (p.window > 0 && i0 + BM - 1 - j0 >= p.window) ||
                             (i0 + BM > len);
#pragma unroll
      for (int ch = 0; ch < BM / 32; ++ch) {
        uint32_t sv[32], dp[32];
        tmem_ld32(tSs + 32 * ch, sv);
        if (KIND >= 1) tmem_ld32(tDP + 32 * ch, dp);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int col = 32 * ch + c;
          float t = fmaf(__uint_as_float(sv[c]), p.scale_log2, vec[col]) + rowterm;
          if (need_mask) {
            const int i = i0 + col;
            const bool vis = (i < len) && (jl <= i) && (p.window == 0 || i - jl < p.window);
            t = vis ? t : neg_inf();
          }
          const float pr = ex2(t);
          sv[c] = __float_as_uint(pr);
          if (KIND >= 1) dp[c] = __float_as_uint(pr * (__uint_as_float(dp[c]) - vec[BM + col]));
        }
        uint32_t pk[16];
        if (KIND == 0) {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[c] = pack_bf16x2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1]));
          tmem_st16(tSs + 16 * ch, pk);
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[c] = pack_bf16x2(__uint_as_float(dp[2 * c]), __uint_as_float(dp[2 * c + 1]));
          tmem_st16(tDP + 16 * ch, pk);
          if (KIND == 1) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(sDS + sw128_offset(r, 4 * ch + q)) =
                  make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
          if (sums && has_gate) {
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) acc += __uint_as_float(dp[c]);
            dgcol += acc;
          }
          if (want_row) {
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
            const int i = i0 + 32 * ch + lane;
            if (i < len) red_add_f32(p.dg_row + (size_t)h * p.total + seq_start + i, v[0]);
          }
        }
      }
      tmem_st_wait();
      if (KIND == 1) fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&vec_empty[s & 1]);
        mbar_arrive(DB ? &p_full2[s & 1] : p_full);
      }
      if (DB) continue;  // the next step's scores are already under way
      ok = wait_bar(mma_done, s & 1, ab);
      if (!ok) break;
      if (KIND == 1) {
        // dQ^T halves: lane r holds dims w0 + r (half 0) and w0 + 128 + r (half 1)
        tc_fence_after();
        uint32_t dq[64];
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          tmem_ld32(tmem + lane_off + C::T_DQ + hf * 64, dq);
          tmem_ld32(tmem + lane_off + C::T_DQ + hf * 64 + 32, dq + 32);
          tmem_ld_wait();
          if (hf == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dq_free);
          }
          const int nrows = min(BM, len - i0);
          float* base = p.dq_acc + ((size_t)(seq_start + i0) * p.hq + h) * DQK + w0 + hf * 128 + r;
          const size_t row_stride = (size_t)p.hq * DQK;
#pragma unroll
          for (int c = 0; c < BM; ++c)
            if (c < nrows) red_add_f32(base + c * row_stride, __uint_as_float(dq[c]) * p.scale);
        }
      }
    }
    if (ok && sums && cur_h >= 0 && has_gate && jl < len)
      red_add_f32(p.dg_col + (size_t)cur_h * p.total + seq_start + jl, dgcol);
    // ---- epilogue: dV (role V) or scale * dK (role KQ), columns w0 .. w0+255
    if (ok && nsteps > 0 && DB) ok = wait_bar(acc_done, 0, ab);
    if (ok && nsteps > 0) {
      tc_fence_after();
      const bool row_ok = jl < len;
      const size_t tok = (size_t)(seq_start + (row_ok ? jl : 0));
      uint16_t* dst = (KIND >= 1) ? p.grad_k + tok * p.dk_ts + (size_t)kvh * p.dk_hs + w0
                                  : p.grad_v + tok * p.dv_ts + (size_t)kvh * p.dv_hs + w0;
      const float sc = (KIND >= 1) ? p.scale : 1.f;
#pragma unroll 1
      for (int c = 0; c < kW / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + C::T_ACC + c * 32, v);
        tmem_ld_wait();
        if (row_ok) {
          uint4* d = reinterpret_cast<uint4*>(dst + c * 32);
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

// Both kinds of role in one launch, so that the dV roles fill the SMs the heavier dK roles'
// last wave leaves idle: blockIdx.z < DQK / 256 selects a dK role (KQ_KIND: 1 with dQ, 2 without),
// the rest the dV roles.  The K-side roles come first (they are dispatched first).
template <int DQK, int DV, int KQ_KIND>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_bwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ64, const __grid_constant__ CUtensorMap tmQ128,
                            const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ CUtensorMap tmDO64, const __grid_constant__ CUtensorMap tmDO128,
                            const BwdParams p) {
  constexpr int nk = DQK / kW;
  constexpr int bk = KQ_KIND == 1 ? 64 : 128;  // query rows per step of the K-side role
  if ((int)blockIdx.z < nk)
    wide_role<DQK, DV, KQ_KIND, bk>(bk == 64 ? tmQ64 : tmQ128, tmK, tmV, bk == 64 ? tmDO64 : tmDO128, p, blockIdx.z);
  else
    wide_role<DQK, DV, 0, 128>(tmQ128, tmK, tmV, tmDO128, p, blockIdx.z - nk);
}

template <int DQK, int DV, int KQ_KIND>
cudaError_t launch_roles(const BwdParams& p, const BwdMaps& maps, int num_tiles, cudaStream_t s) {
  constexpr int bk = KQ_KIND == 1 ? 64 : 128;
  constexpr int smem = WideCfg<DQK, DV, KQ_KIND, bk>::SMEM > WideCfg<DQK, DV, 0, 128>::SMEM
                           ? WideCfg<DQK, DV, KQ_KIND, bk>::SMEM
                           : WideCfg<DQK, DV, 0, 128>::SMEM;
  auto kern = prefill_bwd_wide_kernel<DQK, DV, KQ_KIND>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int roles = DQK / kW + DV / kW;
  kern<<<dim3(p.hkv, num_tiles, roles), kThreads, smem, s>>>(maps.q, maps.q128, maps.k, maps.v, maps.dout,
                                                             maps.dout128, p);
  return cudaGetLastError();
}

template <int DQK, int DV>
cudaError_t launch_both(const BwdParams& p, const BwdMaps& maps, int num_tiles, bool with_dq, cudaStream_t s) {
  return with_dq ? launch_roles<DQK, DV, 1>(p, maps, num_tiles, s) : launch_roles<DQK, DV, 2>(p, maps, num_tiles, s);
}

}  // namespace

cudaError_t launch_prefill_bwd_wide(const BwdParams& p, const BwdMaps& maps, int num_kv_tiles, bool with_dq,
                                    cudaStream_t s) {
  if (p.dqk == 256 && p.dv == 256) return launch_both<256, 256>(p, maps, num_kv_tiles, with_dq, s);
  if (p.dqk == 256 && p.dv == 512) return launch_both<256, 512>(p, maps, num_kv_tiles, with_dq, s);
  if (p.dqk == 512 && p.dv == 512) return launch_both<512, 512>(p, maps, num_kv_tiles, with_dq, s);
  return cudaErrorInvalidValue;
}

}  // namespace gcs
