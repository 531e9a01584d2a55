// Prefill backward, single pass with dQ fused into the dK / dV pass (fla-org/flash-linear-
// attention #1322 "Gluon attention backend with large head dimensions": the comment of Oct 5
// sends dQ partials into a zero-initialised fp32 buffer that is converted after the kernel;
// the comment of Oct 3 recomputes the probabilities in fp32).  Head dim 128.
//
// One CTA per (128-key tile, kv head); it loops over the query heads of its GQA group and
// over 128-row query tiles in the causal / window range ("steps").  Per step:
//     S^T  = K Q^T       (TMEM, fp32)     P^T  = 2^(S^T scale log2e + G_i - G_j - LSE_i)
//     dP^T = V dO^T      (TMEM, fp32)     dS^T = P^T o (dP^T - delta_i)
//     dV  += P^T dO      (A = P^T, bf16 over the consumed S^T in TMEM)
//     dK  += dS^T Q      (A = dS^T, bf16 over the consumed dP^T in TMEM)
//     dQ   = dS K        (A = dS^T in shared memory read MN-major, B = the resident K tile MN-major)
// and dQ is reduce-added in fp32 into a zeroed buffer, plus the fp32 row and column sums of dS
// (gate and sink gradients).
//
// TMEM (512 columns): S^T | dP^T, then dQ of the same step | dV | dK.  The issue order
//     dV(s), S^T(s+1), dK(s), dQ(s), [dQ(s) read out], dP^T(s+1), dV(s+1), ...
// keeps every overwrite behind the MMA that reads the old contents: tcgen05.mma operations
// issued by one thread execute in issue order, so S^T(s+1) may replace the P^T that dV(s)
// reads and dQ(s) the dS^T that dK(s) reads; dP^T(s+1) waits until the softmax warps have
// loaded dQ(s).  dS^T reaches shared memory in the dO tile of its own step, which dV(s) and
// dP^T(s) have finished reading by then (dv_done), so the kernel needs no extra tile.
//
// dQ leaves through shared memory: once dQ(s) is in TMEM (lane = query row) the two softmax
// warpgroups each load their 64 head dims and write them as two 128-row x 32-dim fp32 boxes
// with the 128-byte swizzle (16-byte stores, 32 KB) into a tile no MMA reads any more --
// warpgroup 0 into the dO(s) tile, warpgroup 1 into the Q(s) tile -- and tiled bulk
// reduce-adds (fp32 add in L2) send the boxes to the dQ accumulator.  The bulk operations are issued and awaited by warps 2 and 3, which then
// hand the tile back to the producer, so the softmax warps never wait for them.  Query rows of
// a block that lie past the sequence hold exact zeros (their probabilities are 0), so adding
// them to the next sequence's rows changes nothing; rows past the tensor are clipped.
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 tcgen05 issuer, warps 2-3 the dQ bulk
// reduce-adds of warpgroups 0 and 1, warps 4-7 and 8-11 the two halves (query columns 0-63,
// 64-127) of every step.
#include "kernels.h"
#include "sm103_ptx.cuh"
#include "tiles.cuh"

namespace gcs {
namespace {

constexpr int kD = 128;
constexpr int kBN = 128;  // keys per CTA (TMEM lanes)
constexpr int kBM = 128;  // query rows per step (MMA N)
constexpr int kThreads = 384;
constexpr int kChunk = 128 * 128;  // 128 rows x 64 bf16: one swizzled operand chunk
constexpr int kCH = kD / 64;
constexpr int kTile = kCH * kChunk;
constexpr int kVecBytes = 2 * kBM * 4;  // per step: two packed 64-row tiles of (colterm, delta)
constexpr int kSmemOptinMax = 232448;
constexpr int kNQ = 3;   // Q buffers
constexpr int kNDO = 2;  // dO (then dS^T) + vector buffers

constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + kTile;
constexpr int OFF_Q = OFF_V + kTile;            // [kNQ]
constexpr int OFF_DO = OFF_Q + kNQ * kTile;     // [kNDO]
constexpr int OFF_VEC = OFF_DO + kNDO * kTile;  // [kNDO] x kVecBytes
constexpr int OFF_BAR = OFF_VEC + kNDO * kVecBytes;
constexpr int NBAR = 24;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM = OFF_MISC + 16;
static_assert(SMEM <= kSmemOptinMax, "shared memory budget");
constexpr int T_S = 0, T_DP = 128, T_DV = 256, T_DK = 384;  // T_DP also holds dQ

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// Register split: warpgroup 0 (producer, MMA issuer with its extra descriptors, the two
// reduce-add warps) 104, the softmax warpgroups 200: 128 x 104 + 256 x 200 = 64512 = 384 threads
// x 168 at launch.
__device__ __forceinline__ void reg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 104;\n" ::: "memory"); }
__device__ __forceinline__ void reg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 200;\n" ::: "memory"); }

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

template <bool MASK>
__device__ __forceinline__ void p_row(float* pr, const uint32_t* sv, const float4* ct4, float rowterm,
                                      float scale_log2, int cmin, int cmax) {
#pragma unroll
  for (int c4 = 0; c4 < 16; ++c4) {
    const float4 ct = ct4[c4];
    const float cts[4] = {ct.x + rowterm, ct.y + rowterm, ct.z + rowterm, ct.w + rowterm};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = 4 * c4 + e;
      float t = fmaf(__uint_as_float(sv[c]), scale_log2, cts[e]);
      if (MASK) t = (c >= cmin && c <= cmax) ? t : neg_inf();
      pr[c] = ex2(t);
    }
  }
}

// Sum over the warp's 32 lanes of v[0..31] (lane l's row): on return lane l holds the sum of
// column l.  Each halving step exchanges the half of the columns the partner keeps.
__device__ __forceinline__ float warp_column_sums(float* v, int lane) {
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
  return v[0];
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_bwd_fused_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                             const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];

  TileRef tr;
  if (!lpt_tile(p.cu_seqlens, p.num_seqs, kBN, blockIdx.y, tr)) return;
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicCAS(p.status, kDevOk, kDevUnsupported);
    return;
  }
  const int seq_start = tr.start, len = tr.len, jt = tr.n - 1 - tr.u;
  int qoff = 0;  // first 64-row query tile of this sequence in the packed vectors
  for (int q = 0; q < tr.seq; ++q) qoff += (__ldg(p.cu_seqlens + q + 1) - __ldg(p.cu_seqlens + q) + 63) / 64;
  const int kvh = blockIdx.x;
  const int group = p.hq / p.hkv;
  const int j0 = jt * kBN;
  const int it_lo = jt;
  int i_hi = len - 1;
  if (p.window > 0) i_hi = min(i_hi, j0 + kBN - 1 + p.window - 1);
  const int it_hi = i_hi / kBM;
  const int n_it = it_hi - it_lo + 1;
  const int nsteps = n_it * group;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;      // [kNQ] Q tile landed
  uint64_t* q_empty = bars + 4;     // [kNQ] dK of its step retired and the dQ block staged there sent
  uint64_t* do_full = bars + 7;     // [kNDO] dO tile and vectors landed
  uint64_t* do_empty = bars + 9;    // [kNDO] the dQ block staged in it sent (after dS^T and dO uses)
  uint64_t* s_full = bars + 11;     // S^T written
  uint64_t* dp_full = bars + 12;    // dP^T written
  uint64_t* p_ready = bars + 13;    // P^T stored in TMEM (8 warps)
  uint64_t* ds_ready = bars + 14;   // dS^T stored in TMEM (8 warps)
  uint64_t* ds_smem = bars + 15;    // dS^T stored in shared memory (8 warps)
  uint64_t* dv_done = bars + 16;    // dV of the step retired: its dO tile may take dS^T
  uint64_t* dq_full = bars + 17;    // dQ written
  uint64_t* dq_read = bars + 18;    // dQ loaded by the 8 softmax warps
  uint64_t* all_done = bars + 19;   // every MMA of the CTA retired (epilogue)
  uint64_t* drain = bars + 20;
  uint64_t* stage_full = bars + 21;  // [2] a warpgroup's dQ block written to shared memory (4 warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  const Abort ab{abort_flag, p.status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int b = 0; b < kNQ; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 1);
    }
    for (int b = 0; b < kNDO; ++b) {
      mbar_init(&do_full[b], 1);
      mbar_init(&do_empty[b], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, 8);
    mbar_init(ds_ready, 8);
    mbar_init(ds_smem, 8);
    mbar_init(dv_done, 1);
    mbar_init(dq_full, 1);
    mbar_init(dq_read, 8);
    mbar_init(all_done, 1);
    mbar_init(drain, 1);
    mbar_init(&stage_full[0], 4);
    mbar_init(&stage_full[1], 4);
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
      prefetch_tmap(&tmDO);
      mbar_expect_tx(kv_full, 2 * kTile);
      for (int c = 0; c < kCH; ++c)
        tma_load_3d(smem + OFF_K + c * kChunk, &tmK, kv_full, c * 64, kvh, seq_start + j0);
      for (int c = 0; c < kCH; ++c)
        tma_load_3d(smem + OFF_V + c * kChunk, &tmV, kv_full, c * 64, kvh, seq_start + j0);
      const uint64_t pol = l2_policy_evict_last();
      for (int s = 0; s < nsteps; ++s) {
        const int qb = s % kNQ, db = s % kNDO;
        const int h = kvh * group + s / n_it;
        const int it = it_lo + s % n_it;
        if (!wait_bar(&q_empty[qb], ((s / kNQ) & 1) ^ 1, ab)) break;
        mbar_expect_tx(&q_full[qb], kTile);
        for (int c = 0; c < kCH; ++c)
          tma_load_3d_hint(smem + OFF_Q + qb * kTile + c * kChunk, &tmQ, &q_full[qb], c * 64, h,
                           seq_start + it * kBM, pol);
        if (!wait_bar(&do_empty[db], ((s / kNDO) & 1) ^ 1, ab)) break;
        mbar_expect_tx(&do_full[db], kTile + kVecBytes);
        for (int c = 0; c < kCH; ++c)
          tma_load_3d_hint(smem + OFF_DO + db * kTile + c * kChunk, &tmDO, &do_full[db], c * 64, h,
                           seq_start + it * kBM, pol);
        bulk_load(smem + OFF_VEC + db * kVecBytes, p.vecp + ((size_t)h * p.n_qtiles + qoff + 2 * it) * 128,
                  kVecBytes, &do_full[db]);
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t idS = idesc_bf16(128, kBM, false, false);  // S^T, dP^T: N = 128 query rows
      const uint32_t idAcc = idesc_bf16(128, kD, false, true);  // dV, dK: B = dO / Q, MN-major
      const uint32_t idDQ = idesc_bf16(kBM, kD, true, true);    // dQ: A = dS (the dS^T tile), B = K, both MN-major
      const uint64_t dK0 = sdesc_sw128(smem_u32(smem + OFF_K), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + OFF_V), 16, 1024);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + OFF_Q), 16, 1024);
      const uint64_t dDO0 = sdesc_sw128(smem_u32(smem + OFF_DO), 16, 1024);
      const uint64_t dKmn0 = sdesc_sw128(smem_u32(smem + OFF_K), kChunk, 1024);
      const uint64_t dQmn0 = sdesc_sw128(smem_u32(smem + OFF_Q), kChunk, 1024);
      const uint64_t dDOmn0 = sdesc_sw128(smem_u32(smem + OFF_DO), kChunk, 1024);
      constexpr uint32_t kChunk16 = kChunk >> 4, kTile16 = kTile >> 4;
      auto mma_s = [&](int t) {  // S^T(t) = K Q(t)^T
        const int qb = t % kNQ;
#pragma unroll
        for (int c = 0; c < kCH; ++c) {
          const uint64_t a = dK0 + c * kChunk16, b = dQ0 + qb * kTile16 + c * kChunk16;
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ss(tmem + T_S, a + 2 * k, b + 2 * k, idS, (c | k) != 0);
        }
        mma_commit(s_full);
      };
      auto mma_dp = [&](int t) {  // dP^T(t) = V dO(t)^T
        const int db = t % kNDO;
#pragma unroll
        for (int c = 0; c < kCH; ++c) {
          const uint64_t a = dV0 + c * kChunk16, b = dDO0 + db * kTile16 + c * kChunk16;
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ss(tmem + T_DP, a + 2 * k, b + 2 * k, idS, (c | k) != 0);
        }
        mma_commit(dp_full);
      };
      bool ok = wait_bars(ab, kv_full, 0, &q_full[0], 0, &do_full[0], 0);
      if (ok) {
        tc_fence_after();
        mma_s(0);
        mma_dp(0);
      }
      for (int s = 0; s < nsteps && ok; ++s) {
        const int qb = s % kNQ, db = s % kNDO;
        const bool more = s + 1 < nsteps;
        // P^T(s) stored, Q(s+1) landed
        ok = more ? wait_bars(ab, p_ready, s & 1, &q_full[(s + 1) % kNQ], ((s + 1) / kNQ) & 1)
                  : wait_bars(ab, p_ready, s & 1);
        if (!ok) break;
        tc_fence_after();
        // dV += P^T dO (P^T of query columns 0-63 at T_S + 0..31, of 64-127 at T_S + 64..95)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts(tmem + T_DV, tmem + T_S + (k >> 2) * 64 + 8 * (k & 3), dDOmn0 + db * kTile16 + 128 * k, idAcc,
                 (s > 0 || k > 0) ? 1u : 0u);
        mma_commit(dv_done);
        if (more) mma_s(s + 1);
        // dS^T(s) in TMEM: dK += dS^T Q
        ok = wait_bar(ds_ready, s & 1, ab);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts(tmem + T_DK, tmem + T_DP + (k >> 2) * 64 + 8 * (k & 3), dQmn0 + qb * kTile16 + 128 * k, idAcc,
                 (s > 0 || k > 0) ? 1u : 0u);
        // dS^T(s) in shared memory (the dO(s) tile): dQ = dS K over the dP^T columns (TMEM lane =
        // query row, column = head dim)
        ok = wait_bar(ds_smem, s & 1, ab);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss(tmem + T_DP, dDOmn0 + db * kTile16 + 128 * k, dKmn0 + 128 * k, idDQ, k > 0 ? 1u : 0u);
        mma_commit(dq_full);
        if (more) {
          // dQ(s) loaded by the softmax warps, dO(s+1) landed
          ok = wait_bars(ab, dq_read, s & 1, &do_full[(s + 1) % kNDO], ((s + 1) / kNDO) & 1);
          if (!ok) break;
          tc_fence_after();
          mma_dp(s + 1);
        }
      }
      if (ok) mma_commit(all_done);
      if (!ok) {
        mma_commit(drain);
        mbar_wait(drain, 0, nullptr);
      }
    } else if (warp >= 2 && lane == 0) {
      // ---------------------------------------------------------- dQ bulk reduce-adds
      // warp 2: warpgroup 0's blocks (dO tiles), warp 3: warpgroup 1's blocks (Q tiles)
      const int wg = warp - 2;
      prefetch_tmap(&tmDQ);
      for (int s = 0; s < nsteps; ++s) {
        const int qb = s % kNQ, db = s % kNDO;
        const int h = kvh * group + s / n_it;
        const int i0 = (it_lo + s % n_it) * kBM;
        if (!wait_bar(&stage_full[wg], s & 1, ab)) break;
        const uint8_t* src = smem + (wg == 0 ? OFF_DO + db * kTile : OFF_Q + qb * kTile);
        // this warpgroup's head dims 64 wg .. 64 wg + 63 as two 32-dim x 128-row boxes
        for (int b = 0; b < 2; ++b) tma_reduce_add_3d(&tmDQ, src + b * kChunk, 64 * wg + 32 * b, h, seq_start + i0);
        bulk_commit_group();
        bulk_wait_group_read0();
        mbar_arrive(wg == 0 ? &do_empty[db] : &q_empty[qb]);
      }
      bulk_wait_group0();
    }
    __syncwarp();
  } else {
    reg_inc();
    // ------------------------------------------------------------ key rows, 64 query columns
    const int wg = (warp - 4) >> 2;     // query columns 64 wg .. 64 wg + 63 of every step
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row within the tile = TMEM lane (dQ: query row)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + T_S + 64 * wg;
    const uint32_t tDP = tmem + lane_off + T_DP + 64 * wg;
    const int jl = j0 + r;
    const bool has_gate = p.gT != nullptr;
    const bool want_row = p.dg_row != nullptr;
    float dgcol = 0.f;
    int cur_h = -1;
    float rowterm = 0.f;
    bool ok = true;
    for (int s = 0; s < nsteps; ++s) {
      const int db = s % kNDO;
      const int h = kvh * group + s / n_it;
      const int i0 = (it_lo + s % n_it) * kBM;
      if (h != cur_h) {
        // new query head: flush the column sums of dS of the previous head, reload G_j
        if (cur_h >= 0 && has_gate && jl < len) red_add_f32(p.dg_col + (size_t)cur_h * p.total + seq_start + jl, dgcol);
        dgcol = 0.f;
        cur_h = h;
        rowterm = (has_gate && jl < len) ? -__ldg(p.gT + (size_t)h * p.total + seq_start + jl) : 0.f;
      }
      ok = wait_bar(&do_full[db], (s / kNDO) & 1, ab);
      if (!ok) break;
      const float4* vec4 = reinterpret_cast<const float4*>(smem + OFF_VEC + db * kVecBytes + wg * (kVecBytes / 2));
      const bool need_mask = (i0 < j0 + kBN - 1) || (p.window > 0 && i0 + kBM - 1 - j0 >= p.window) ||
                             (i0 + kBM > len);
      const int cb = i0 + 64 * wg;
      const int cmin = jl - cb;
      const int cmax = min(p.window > 0 ? jl + p.window - 1 - cb : (1 << 30), len - 1 - cb);
      // ---- P in fp32, P^T (bf16) over S^T
      ok = wait_bar(s_full, s & 1, ab);
      if (!ok) break;
      tc_fence_after();
      float pr[64];
      {
        uint32_t sv[64];
        tmem_ld32(tS, sv);
        tmem_ld32(tS + 32, sv + 32);
        tmem_ld_wait();
        if (need_mask)
          p_row<true>(pr, sv, vec4, rowterm, p.scale_log2, cmin, cmax);
        else
          p_row<false>(pr, sv, vec4, rowterm, p.scale_log2, cmin, cmax);
      }
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(pr[32 * ch + 2 * c], pr[32 * ch + 2 * c + 1]);
        tmem_st16(tS + 16 * ch, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready);
      // ---- dS = P (dP - delta_i) in fp32; dS^T (bf16) over this warpgroup's dP^T columns
      ok = wait_bar(dp_full, s & 1, ab);
      if (!ok) break;
      tc_fence_after();
      uint32_t dsk[32];  // dS^T row, bf16 pairs
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
            const int col = 32 * ch + 4 * c4 + e;
            pr[col] = pr[col] * (__uint_as_float(dp[4 * c4 + e]) - dls[e]);
          }
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) dsk[16 * ch + c] = pack_bf16x2(pr[32 * ch + 2 * c], pr[32 * ch + 2 * c + 1]);
        tmem_st16(tDP + 16 * ch, dsk + 16 * ch);  // over dP^T columns already loaded
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_ready);
      // ---- dS^T into the dO(s) tile (chunk wg, key row r), once dV(s) has read dO(s)
      ok = wait_bar(dv_done, s & 1, ab);
      if (!ok) break;
      {
        uint8_t* tile = smem + OFF_DO + db * kTile + wg * kChunk;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(tile + sw128_offset(r, u)) =
              make_uint4(dsk[4 * u], dsk[4 * u + 1], dsk[4 * u + 2], dsk[4 * u + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_smem);
      // fp32 column sums of dS for this key row (gate gradient)
      if (has_gate) {
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) acc[c & 7] += pr[c];
        dgcol += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      }
      // fp32 row sums of dS over this warp's 32 key rows, per query column (gate and sink)
      if (want_row) {
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const float sum = warp_column_sums(pr + 32 * ch, lane);
          const int i = cb + 32 * ch + lane;
          if (i < len) red_add_f32(p.dg_row + (size_t)h * p.total + seq_start + i, sum);
        }
      }
      // ---- dQ(s): lane r = query row i0 + r, this warpgroup's 64 head dims, staged as two
      // [128 query rows][32 dims] fp32 boxes with the 128-byte swizzle for the bulk
      // reduce-adds (warp 2 + wg sends them)
      ok = wait_bar(dq_full, s & 1, ab);
      if (!ok) break;
      tc_fence_after();
      uint32_t dq[64];
      tmem_ld32(tDP, dq);
      tmem_ld32(tDP + 32, dq + 32);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_read);
      {
        uint8_t* stage = smem + (wg == 0 ? OFF_DO + db * kTile : OFF_Q + (s % kNQ) * kTile);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float4 v = make_float4(__uint_as_float(dq[4 * u]) * p.scale, __uint_as_float(dq[4 * u + 1]) * p.scale,
                                       __uint_as_float(dq[4 * u + 2]) * p.scale,
                                       __uint_as_float(dq[4 * u + 3]) * p.scale);
          *reinterpret_cast<float4*>(stage + (u >> 3) * kChunk + sw128_offset(r, u & 7)) = v;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&stage_full[wg]);
    }
    if (ok && cur_h >= 0 && has_gate && jl < len)
      red_add_f32(p.dg_col + (size_t)cur_h * p.total + seq_start + jl, dgcol);
    // ---- epilogue: warpgroup 0 writes dV, warpgroup 1 scale * dK for its key rows
    if (ok && nsteps > 0) {
      ok = wait_bar(all_done, 0, ab);
      if (ok) {
        tc_fence_after();
        const bool row_ok = jl < len;
        const size_t tok = (size_t)(seq_start + (row_ok ? jl : 0));
        uint16_t* dst = wg == 0 ? p.grad_v + tok * p.dv_ts + (size_t)kvh * p.dv_hs
                                : p.grad_k + tok * p.dk_ts + (size_t)kvh * p.dk_hs;
        const uint32_t col0 = wg == 0 ? T_DV : T_DK;
        const float sc = wg == 0 ? 1.f : p.scale;
#pragma unroll 1
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + col0 + c * 32, v);
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
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // a role gave up: let copies and MMAs already in flight land before TMEM is released
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_prefill_bwd_fused(const BwdParams& p, const BwdMaps& maps, int num_kv_tiles, cudaStream_t s) {
  if (p.dqk != kD || p.dv != kD || p.dq_acc == nullptr) return cudaErrorInvalidValue;
  auto kern = prefill_bwd_fused_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  kern<<<dim3(p.hkv, num_kv_tiles), kThreads, SMEM, s>>>(maps.q128, maps.k, maps.v, maps.dout128, maps.dq_acc, p);
  return cudaGetLastError();
}

}  // namespace gcs
