// Paged chunked prefill over an fp8 e4m3 KV cache: the query rows of a request are the last
// q_len positions of its cached context, any q_len (ROCm/aiter PR #6660, commit messages:
// every batch that is not all-decode takes the 2d unified-attention route, one program per
// (KV head, query block); "Technical details": per-token K and V scales laid out like the
// cache pages, K scales on the score columns, V scales on the probability columns after the
// row sum, slots past seq_len unused).  The decoding features of fla-org/flash-linear-
// attention #1322 (Description: log gates, sliding windows, a sink) apply as in decode.
//
// Row t of a request sits at position L - q_len + t and sees keys 0 .. L - q_len + t
// (bottom-right causal alignment).  A 128-row query tile is 128 / G positions x the G query
// heads of one kv head (G = 16 or 8; row = G * position + head); one CTA takes two tiles and one
// segment of the context.  A "page" is 16 tokens; a cache block of block_size = 16 k tokens
// holds k of them at consecutive slots.  With one segment per request the CTA writes the bf16 output (the
// sink in its denominator); with several it writes split-K partials (unnormalised
// accumulator, running max in log2 units and row sum) that the decode combine merges.
//
// Warp roles (384 threads):
//   warp 0      producer: per 128-key tile, the 8 pages' K (2 KB each, tensor copy with the
//               128-byte swizzle) with their K and V scales (64 B each) and the group's gates
//               (1 KB) by plain bulk copy, then the 8 V pages (swizzled), one copy per lane
//   warp 1      tcgen05 issuer: S_x = Q_x K^T (both operands in shared memory) and
//               O_x += P_x V (P in TMEM), interleaved PV_A(n), S_A(n+1), PV_B(n), S_B(n+1)
//   warps 2-3   converters: e4m3 -> f16 (exact) into 128-byte-swizzled operand stages, slots
//               at or past seq_len zeroed (their bytes may be NaN); per-key vectors for the
//               softmax: K scale x softmax scale x log2 e, V scale x 2^4, -G x log2 e
//   warps 4-7   softmax of tile A, warps 8-11 softmax of tile B, one thread per row
// Q, K, V and P enter the tensor cores as f16 (Q rounded from bf16; e4m3 -> f16 is exact),
// with fp32 accumulation.  P * vscale is carried scaled by 2^4; with the lazy rescale
// threshold of 2^4 every P * vscale * 2^4 stays below 256 * vscale.
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace gcs {
namespace {

constexpr int kPage = 16;
constexpr int kD = 128;
constexpr int kRows = 16;         // partial rows per (unit, query position), as in decode
constexpr int kTileKeys = 128;    // 8 pages
constexpr int kThreads = 384;
constexpr int kStage = 16384;     // one f16 operand stage: 128 rows x 64 dims or 64 keys x 128 dims
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kPScale = 16.f;   // P * vscale carried x 2^4
constexpr float kRescale = 4.f;   // lazy rescale threshold (log2 units): P <= 2^4

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// Three-input maximum (one instruction on this architecture).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <bool FEAT>
struct PpCfg {
  static constexpr int NST = FEAT ? 6 : 7;                 // f16 operand stages
  static constexpr int OFF_Q = 0;                          // [2 tiles][2 dim chunks] x 16 KB
  static constexpr int OFF_RING = 4 * kStage;
  static constexpr int OFF_KRAW = OFF_RING + NST * kStage; // K pages | K scales | V scales | gates
  static constexpr int KR_KS = 8 * 2048, KR_VS = KR_KS + 512, KR_G = KR_VS + 512;
  static constexpr int KRAW = KR_G + (FEAT ? 8 * 1024 : 0);
  static constexpr int OFF_VRAW = OFF_KRAW + KRAW;         // V pages
  static constexpr int OFF_AUX = OFF_VRAW + 8 * 2048;      // [2] x {ks'[128], vs'[128], G'[16][128]}
  static constexpr int AUX = 1024 + (FEAT ? 8192 : 0);
  static constexpr int OFF_BAR = OFF_AUX + 2 * AUX;
  static constexpr int OFF_MISC = OFF_BAR + (2 * NST + 24) * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// Register split: warpgroup 0 (producer, MMA, converters) 88, the softmax warpgroups 208:
// 128 x 88 + 256 x 208 = 64512 = 384 threads x 168 at launch.  The converters spill a few
// words at 88; 96 / 200 removes that but measured slower (the softmax wants the registers).
__device__ __forceinline__ void reg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 88;\n" ::: "memory"); }
__device__ __forceinline__ void reg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 208;\n" ::: "memory"); }

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void sts128(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// four e4m3 bytes (lowest byte first) -> two f16x2 words (lowest element in the low half)
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <bool FEAT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_paged_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const DecodeParams p) {
  using C = PpCfg<FEAT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align_1k(smem_raw);

  const int nseg = p.max_segs;
  const int seg = blockIdx.x % nseg, qp = blockIdx.x / nseg;
  const int kvh = blockIdx.y;
  // Requests in order of decreasing context (ties by index) when there are at most 32, so
  // the last CTAs to start are the lightest; every warp ranks them with shuffles.
  int r = blockIdx.z;
  if (p.num_reqs <= 32) {
    const int ln = threadIdx.x & 31;
    const int li = ln < p.num_reqs ? __ldg(p.seq_lens + ln) : -1;
    int rank = 0;
    for (int s2 = 0; s2 < p.num_reqs; ++s2) {
      const int ls = __shfl_sync(0xffffffffu, li, s2);
      rank += (ls > li) || (ls == li && s2 < ln);
    }
    r = __ffs(__ballot_sync(0xffffffffu, ln < p.num_reqs && rank == static_cast<int>(blockIdx.z))) - 1;
  }
  const int q_begin = __ldg(p.cu_q + r);
  const int ql = __ldg(p.cu_q + r + 1) - q_begin;
  const int L = __ldg(p.seq_lens + r);
  const int G = p.group, lgG = G == 16 ? 4 : 3;  // query heads per kv head (16 or 8)
  const int pos_tile = 128 / G;                 // positions of a 128-row query tile
  const int lbp = p.log2_block_pages;              // cache blocks hold 2^lbp 16-token pages
  const int pos0 = qp * 2 * pos_tile;
  if (pos0 >= ql) return;
  const int npages = (L + kPage - 1) / kPage;
  const int pb = seg * p.seg_pages;
  if (pb >= npages) return;  // past the request's last segment (the combine stops before it)
  const int pend = min(pb + p.seg_pages, npages);
  const int key_seg0 = pb * kPage;
  const int ntile_seg = (pend - pb + 7) / 8;
  const bool direct = p.part_acc == nullptr;
  const int W = FEAT ? p.window : 0;

  // key tiles of the segment (index jt, keys key_seg0 + 128 jt ..) that each query tile sees
  int lo[2], hi[2];
  for (int x = 0; x < 2; ++x) {
    const int px = pos0 + x * pos_tile;
    lo[x] = 0;
    hi[x] = -1;
    if (px >= ql) continue;
    const int lk_min = L - ql + px, lk_max = L - ql + min(px + pos_tile - 1, ql - 1);
    if (lk_max >= key_seg0) hi[x] = min(ntile_seg - 1, (lk_max - key_seg0) / kTileKeys);
    const int fk = W > 0 ? max(0, lk_min - W + 1) : 0;
    if (fk > key_seg0) lo[x] = (fk - key_seg0) / kTileKeys;
  }
  int hi_t = -1, lo_t = 1 << 30;
  for (int x = 0; x < 2; ++x)
    if (lo[x] <= hi[x]) {
      hi_t = max(hi_t, hi[x]);
      lo_t = min(lo_t, lo[x]);
    }
  const size_t rows_per_unit = (size_t)p.max_q_len * kRows;
  const size_t unit = ((size_t)r * p.max_segs + seg) * p.hkv + kvh;
  if (hi_t < 0) {
    // nothing of this segment is visible to these 16 positions: empty partials (weight 0)
    if (!direct) {
      const int npos = min(2 * pos_tile, ql - pos0);
      const size_t row0 = unit * rows_per_unit + (size_t)pos0 * G;
      float4* acc = reinterpret_cast<float4*>(p.part_acc + row0 * kD);
      for (int i = threadIdx.x; i < npos * G * (kD / 4); i += blockDim.x) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      float2* ml = reinterpret_cast<float2*>(p.part_ml) + row0;
      for (int i = threadIdx.x; i < npos * G; i += blockDim.x) ml[i] = make_float2(neg_inf(), 0.f);
    }
    return;
  }
  const int nt = hi_t - lo_t + 1;  // processed as jt = hi_t - n, n = 0 .. nt - 1
  int n_first[2], n_last[2];
  for (int x = 0; x < 2; ++x) {
    const bool any = lo[x] <= hi[x];
    n_first[x] = any ? hi_t - hi[x] : nt;
    n_last[x] = any ? hi_t - lo[x] : -1;
  }
  auto part = [&](int x, int n) -> bool { return n >= n_first[x] && n <= n_last[x]; };

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;               // [NST] f16 stages written
  uint64_t* empty = bars + C::NST;     // [NST] f16 stages consumed
  uint64_t* kr_full = bars + 2 * C::NST;
  uint64_t* kr_empty = kr_full + 1;
  uint64_t* vr_full = kr_full + 2;
  uint64_t* vr_empty = kr_full + 3;
  uint64_t* aux_full = kr_full + 4;    // [2]
  uint64_t* aux_empty = kr_full + 6;   // [2]
  uint64_t* q_full = kr_full + 8;      // [2 tiles]
  uint64_t* s_full = kr_full + 10;     // [2 tiles]
  uint64_t* p_full = kr_full + 12;     // [2 tiles]
  uint64_t* pv_done = kr_full + 14;    // [2 tiles]
  uint64_t* drain = kr_full + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const Abort ab{abort_flag, p.status};
  uint8_t* kraw = smem + C::OFF_KRAW;
  uint8_t* vraw = smem + C::OFF_VRAW;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 2);
      mbar_init(&empty[i], 1);
    }
    mbar_init(kr_full, 1);
    mbar_init(kr_empty, 2);
    mbar_init(vr_full, 1);
    mbar_init(vr_empty, 2);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&aux_full[i], 2);
      mbar_init(&aux_empty[i], 8);
      mbar_init(&q_full[i], 4);
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

  if (warp < 4) {
    reg_dec();
    if (warp == 0) {
      // ---------------------------------------------------------- page producer
      const int32_t* trow = p.block_table + (size_t)r * p.max_blocks;
      const bool per_token = p.scale_mode == 0;
      const bool has_gate = FEAT && p.g_cache != nullptr;
      const int pl = lane & 7, kind = lane >> 3;  // 0: K page, 1: K scales, 2: V scales, 3: gates
      if (lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
      }
      for (int n = 0; n < nt; ++n) {
        const int pg0 = pb + (hi_t - n) * 8;
        const int nv = min(8, pend - pg0);  // pages of the tile that exist
        const uint32_t par = (n & 1) ^ 1;
        bool okl = wait_bar(kr_empty, par, ab);
        if (!__all_sync(0xffffffffu, okl)) break;
        if (lane == 0)
          mbar_expect_tx(kr_full, nv * (2048 + (per_token ? 128 : 0) + (has_gate ? G * kPage * 4 : 0)));
        __syncwarp();
        const int pg = pg0 + pl;
        const int blk = pl < nv ? __ldg(trow + (pg >> lbp)) : 0;
        const int sub = (pg & ((1 << lbp) - 1)) * kPage;  // first slot of the page in its block
        const size_t slot0 = ((size_t)blk * p.hkv + kvh) * p.block_size + sub;
        if (pl < nv) {
          if (kind == 0) {
            tma_load_4d(kraw + pl * 2048, &tmK, kr_full, 0, p.kv_head_inner ? kvh : sub, p.kv_head_inner ? sub : kvh,
                        blk);
          } else if (kind == 1 && per_token) {
            bulk_load(kraw + C::KR_KS + pl * 64, p.k_scale + slot0, 64, kr_full);
          } else if (kind == 2 && per_token) {
            bulk_load(kraw + C::KR_VS + pl * 64, p.v_scale + slot0, 64, kr_full);
          } else if (kind == 3 && has_gate) {
            // the group's G heads x 16 slots: adjacent when a block is one page
            const float* src = p.g_cache + ((size_t)blk * p.hq + kvh * G) * p.block_size + sub;
            if (lbp == 0) {
              bulk_load(kraw + C::KR_G + pl * 1024, src, G * kPage * 4, kr_full);
            } else {
              for (int hh = 0; hh < G; ++hh)
                bulk_load(kraw + C::KR_G + pl * 1024 + hh * kPage * 4, src + (size_t)hh * p.block_size, kPage * 4,
                          kr_full);
            }
          }
        }
        okl = wait_bar(vr_empty, par, ab);
        if (!__all_sync(0xffffffffu, okl)) break;
        if (lane == 0) mbar_expect_tx(vr_full, nv * 2048);
        __syncwarp();
        if (kind == 0 && pl < nv)
          tma_load_4d(vraw + pl * 2048, &tmV, vr_full, 0, p.kv_head_inner ? kvh : sub, p.kv_head_inner ? sub : kvh,
                      blk);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // -------------------------------------------------------- MMA issuer
        const uint32_t idS = idesc_f16(128, kTileKeys, false, false);
        const uint32_t idPV = idesc_f16(128, kD, false, true);
        const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
        const uint64_t dK0 = sdesc_sw128(smem_u32(smem + C::OFF_RING), 16, 1024);
        const uint64_t dV0 = sdesc_sw128(smem_u32(smem + C::OFF_RING), kStage / 2, 1024);
        constexpr uint32_t kSt16 = kStage >> 4;
        uint32_t stage = 0, phase = 0;  // ring position of the next stage (K0 K1 V0 V1 per tile)
        auto next = [&](uint32_t& st, uint32_t& ph) {
          st = stage;
          ph = phase;
          if (++stage == C::NST) {
            stage = 0;
            phase ^= 1;
          }
        };
        auto mma_s = [&](int x, uint32_t k0, uint32_t k1) {  // S_x = Q_x K^T
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint64_t a = dQ0 + (x * 2 + c) * kSt16, b = dK0 + (c ? k1 : k0) * kSt16;
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_ss(tmem + 128 * x, a + 2 * k, b + 2 * k, idS, (c | k) != 0);
          }
          mma_commit(&s_full[x]);
        };
        auto mma_pv = [&](int x, uint32_t v0, uint32_t v1, bool acc) {  // O_x += P_x V
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint64_t b = dV0 + (h ? v1 : v0) * kSt16;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ts(tmem + 256 + 128 * x, tmem + 128 * x + (4 * h + k) * 8, b + 128 * k, idPV,
                     (acc || h || k) ? 1u : 0u);
          }
          mma_commit(&pv_done[x]);
        };
        bool qr[2] = {false, false};
        int kp[2] = {0, 0};
        uint32_t k0, pk0, k1, pk1;
        next(k0, pk0);
        next(k1, pk1);
        bool ok = wait_bars(ab, &full[k0], pk0, &full[k1], pk1);
        for (int x = 0; x < 2 && ok; ++x) {
          if (!part(x, 0)) continue;
          ok = wait_bar(&q_full[x], 0, ab);
          qr[x] = true;
          if (!ok) break;
          tc_fence_after();
          mma_s(x, k0, k1);
        }
        if (ok) {
          mma_commit(&empty[k0]);
          mma_commit(&empty[k1]);
        }
        for (int n = 0; n < nt && ok; ++n) {
          const bool more = n + 1 < nt;
          uint32_t v0, pv0, v1, pv1, n0 = 0, pn0 = 0, n1 = 0, pn1 = 0;
          next(v0, pv0);
          next(v1, pv1);
          if (more) {
            next(n0, pn0);
            next(n1, pn1);
          }
          bool waited = false;
          for (int x = 0; x < 2 && ok; ++x) {
            const bool do_pv = part(x, n), do_s = more && part(x, n + 1);
            if (!do_pv && !do_s) continue;
            if (!waited) {
              ok = wait_bars(ab, &full[v0], pv0, &full[v1], pv1, do_pv ? &p_full[x] : nullptr, kp[x] & 1);
              if (ok && more) ok = wait_bars(ab, &full[n0], pn0, &full[n1], pn1);
              waited = true;
            } else if (do_pv) {
              ok = wait_bar(&p_full[x], kp[x] & 1, ab);
            }
            if (ok && do_s && !qr[x]) {
              ok = wait_bar(&q_full[x], 0, ab);
              qr[x] = true;
            }
            if (!ok) break;
            tc_fence_after();
            if (do_pv) {
              mma_pv(x, v0, v1, kp[x] > 0);
              ++kp[x];
            }
            if (do_s) mma_s(x, n0, n1);
          }
          // a stage is released only after its data was waited for, so the converter never
          // runs two phases ahead of this thread
          if (ok && !waited) {
            ok = wait_bars(ab, &full[v0], pv0, &full[v1], pv1);
            if (ok && more) ok = wait_bars(ab, &full[n0], pn0, &full[n1], pn1);
          }
          if (!ok) break;
          mma_commit(&empty[v0]);
          mma_commit(&empty[v1]);
          if (more) {
            mma_commit(&empty[n0]);
            mma_commit(&empty[n1]);
          }
        }
        if (!ok) {
          mma_commit(drain);
          mbar_wait(drain, 0, nullptr);
        }
      }
      __syncwarp();
    } else {
      // ---------------------------------------------------------- converters (warps 2-3)
      const int c = threadIdx.x - 64;  // 0 .. 63
      const bool per_token = p.scale_mode == 0;
      const bool has_gate = FEAT && p.g_cache != nullptr;
      const float kst = per_token ? 0.f : __ldg(p.k_scale), vst = per_token ? 0.f : __ldg(p.v_scale);
      const float sl2 = p.scale * kLog2e;
      uint8_t* ring = smem + C::OFF_RING;
      uint32_t stage = 0, phase = 0;
      auto next = [&](uint32_t& st, uint32_t& ph) {
        st = stage;
        ph = phase;
        if (++stage == C::NST) {
          stage = 0;
          phase ^= 1;
        }
      };
      // 8 pages of fp8 rows (128 B, 128-byte swizzled) -> f16 operand rows.  Thread c takes the
      // keys 8 i + (c & 7), i = 0..15, and the 16-dim group q = c / 8 of each: a quarter warp
      // reads one group of eight consecutive keys and writes the two 16-B halves of each result
      // to units (2 (q & 3), 2 (q & 3) + 1) of their swizzled rows, all in different bank groups.
      //   K (is_v false): stage sa holds dims 0..63, sb dims 64..127; row = key (K-major).
      //   V (is_v true):  stage sa holds keys 0..63, sb keys 64..127; inside a stage, dims
      //                   0..63 then 64..127 (8 KB apart), row = key (MN-major).
      const int cq = c >> 3, ck = c & 7;
      const uint32_t su0 = ((2 * (cq & 3)) ^ ck) << 4, su1 = ((2 * (cq & 3) + 1) ^ ck) << 4;
      auto convert = [&](const uint8_t* raw, int key0, bool is_v, uint32_t sa, uint32_t sb) {
        const uint8_t* src = raw + ck * 128 + ((cq ^ ck) << 4);
        uint8_t* dst_a;
        uint8_t* dst_b;
        if (!is_v) {
          dst_a = dst_b = ring + ((cq >> 2) ? sb : sa) * kStage + ck * 128;
        } else {
          dst_a = ring + sa * kStage + (cq >> 2) * (kStage / 2) + ck * 128;
          dst_b = ring + sb * kStage + (cq >> 2) * (kStage / 2) + ck * 128;
        }
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
          uint4 xv = make_uint4(0u, 0u, 0u, 0u);
          if (key0 + 8 * i + ck < L) xv = lds128(src + i * 1024);
          uint32_t w[8];
          e4m3x4_to_f16(xv.x, w[0], w[1]);
          e4m3x4_to_f16(xv.y, w[2], w[3]);
          e4m3x4_to_f16(xv.z, w[4], w[5]);
          e4m3x4_to_f16(xv.w, w[6], w[7]);
          uint8_t* row = !is_v ? dst_a + i * 1024 : (i < 8 ? dst_a + i * 1024 : dst_b + (i - 8) * 1024);
          sts128(row + su0, make_uint4(w[0], w[1], w[2], w[3]));
          sts128(row + su1, make_uint4(w[4], w[5], w[6], w[7]));
        }
      };
      for (int n = 0; n < nt; ++n) {
        const int key0 = key_seg0 + (hi_t - n) * kTileKeys;
        const int a = n & 1;
        bool ok = wait_bar(kr_full, n & 1, ab) && wait_bar(&aux_empty[a], ((n >> 1) & 1) ^ 1, ab);
        if (!ok) break;
        // per-key vectors of this tile (zero at or past seq_len)
        float* ax = reinterpret_cast<float*>(smem + C::OFF_AUX + a * C::AUX);
        for (int k = c; k < kTileKeys; k += 64) {
          const bool valid = key0 + k < L;
          const float ks = per_token ? reinterpret_cast<const float*>(kraw + C::KR_KS)[k] : kst;
          const float vs = per_token ? reinterpret_cast<const float*>(kraw + C::KR_VS)[k] : vst;
          ax[k] = valid ? ks * sl2 : 0.f;
          ax[kTileKeys + k] = valid ? vs * kPScale : 0.f;
        }
        if (FEAT) {
          // -G_j in log2 units for the group's G heads: raw pages hold [head][slot], 1 KB apart
          const float* gr = reinterpret_cast<const float*>(kraw + C::KR_G);
          for (int i = c; i < p.group * kTileKeys; i += 64) {
            const int h = i >> 7, k = i & 127;
            ax[2 * kTileKeys + i] =
                (has_gate && key0 + k < L) ? -gr[(k >> 4) * 256 + h * kPage + (k & 15)] * kLog2e : 0.f;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&aux_full[a]);
        uint32_t s0, p0, s1, p1;
        next(s0, p0);
        next(s1, p1);
        ok = wait_bar(&empty[s0], p0 ^ 1, ab) && wait_bar(&empty[s1], p1 ^ 1, ab);
        if (!ok) break;
        convert(kraw, key0, false, s0, s1);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full[s0]);
          mbar_arrive(&full[s1]);
          mbar_arrive(kr_empty);
        }
        uint32_t s2, p2, s3, p3;
        next(s2, p2);
        next(s3, p3);
        ok = wait_bar(vr_full, n & 1, ab) && wait_bar(&empty[s2], p2 ^ 1, ab) && wait_bar(&empty[s3], p3 ^ 1, ab);
        if (!ok) break;
        convert(vraw, key0, true, s2, s3);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full[s2]);
          mbar_arrive(&full[s3]);
          mbar_arrive(vr_empty);
        }
      }
    }
    __syncwarp();
  } else {
    reg_inc();
    // ------------------------------------------------------------ softmax, tile x
    const int x = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int rr = quarter * 32 + lane;  // row of the tile
    const int head = rr & (G - 1);
    const int pos = pos0 + x * pos_tile + (rr >> lgG);
    const bool row_valid = pos < ql;
    const int posc = min(pos, ql - 1);
    const int lastk = L - ql + posc;  // last key this row sees
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + 128 * x, tO = tmem + lane_off + 256 + 128 * x;
    {
      // this row of Q: bf16 -> f16 into the 128-B-swizzled K-major tile (two 64-dim chunks)
      const uint4* src =
          reinterpret_cast<const uint4*>(p.q + (size_t)(q_begin + posc) * p.q_ts + (size_t)(kvh * G + head) * p.q_hs);
      uint8_t* qs = smem + C::OFF_Q + x * 2 * kStage;
#pragma unroll 4
      for (int u = 0; u < 16; ++u) {
        const uint4 v = row_valid ? __ldg(src + u) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 f = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                                   bf16x2_to_f16x2(v.w));
        sts128(qs + (u >> 3) * kStage + rr * 128 + (((u & 7) ^ (rr & 7)) << 4), f);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full[x]);
    }
    const bool has_gate = FEAT && p.g_cache != nullptr;
    float gi = 0.f;  // the row's own G (log2 units)
    if (has_gate) {
      const int blk = __ldg(p.block_table + (size_t)r * p.max_blocks + lastk / p.block_size);
      gi = __ldg(p.g_cache + ((size_t)blk * p.hq + kvh * G + head) * p.block_size + lastk % p.block_size) * kLog2e;
    }
    const bool sink_here = direct && p.sink != nullptr;
    float m = sink_here ? __ldg(p.sink + kvh * G + head) * kLog2e : neg_inf();
    float l = sink_here ? 1.f : 0.f;
    const int my_first = x ? n_first[1] : n_first[0], my_last = x ? n_last[1] : n_last[0];
    const int t_lk_min = L - ql + pos0 + x * pos_tile;
    const int t_lk_max = L - ql + min(pos0 + x * pos_tile + pos_tile - 1, ql - 1);
    bool ok = true;
    int kx = 0;  // key tiles processed by this query tile
    for (int n = 0; n < nt; ++n) {
      const int a = n & 1;
      ok = wait_bar(&aux_full[a], (n >> 1) & 1, ab);
      if (!ok) break;
      if (n >= my_first && n <= my_last) {
        const int j0 = key_seg0 + (hi_t - n) * kTileKeys;
        ok = wait_bar(&s_full[x], kx & 1, ab);
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[128];
        tmem_ld32(tS + 0, sv);
        tmem_ld32(tS + 32, sv + 32);
        tmem_ld32(tS + 64, sv + 64);
        tmem_ld32(tS + 96, sv + 96);
        tmem_ld_wait();
        const float* ax = reinterpret_cast<const float*>(smem + C::OFF_AUX + a * C::AUX);
        const float4* ks4 = reinterpret_cast<const float4*>(ax);
        const float4* vs4 = reinterpret_cast<const float4*>(ax + kTileKeys);
        const float4* g4 = reinterpret_cast<const float4*>(ax + 2 * kTileKeys + head * kTileKeys);
        const bool need_mask = (j0 + kTileKeys - 1 > t_lk_min) || (W > 0 && j0 < t_lk_max - W + 1);
        const int jmax = lastk - j0;
        const int jmin = W > 0 ? lastk - W + 1 - j0 : -(1 << 30);
        float mxp[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mxp[e] = neg_inf();
#pragma unroll
        for (int j4 = 0; j4 < 32; ++j4) {
          const float4 k4 = ks4[j4];
          const float ks[4] = {k4.x, k4.y, k4.z, k4.w};
          float gs[4] = {gi, gi, gi, gi};
          if (FEAT) {
            const float4 g = g4[j4];
            gs[0] += g.x;
            gs[1] += g.y;
            gs[2] += g.z;
            gs[3] += g.w;
          }
          float t[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * j4 + e;
            t[e] = FEAT ? fmaf(__uint_as_float(sv[j]), ks[e], gs[e]) : __uint_as_float(sv[j]) * ks[e];
            if (need_mask) t[e] = (j >= jmin && j <= jmax) ? t[e] : neg_inf();
            sv[j] = __float_as_uint(t[e]);
          }
          mxp[(2 * j4) & 7] = fmax3(mxp[(2 * j4) & 7], t[0], t[1]);
          mxp[(2 * j4 + 1) & 7] = fmax3(mxp[(2 * j4 + 1) & 7], t[2], t[3]);
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
            for (int cc = 0; cc < kD / 32; ++cc) {
              uint32_t ov[32];
              tmem_ld32(tO + cc * 32, ov);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
              tmem_st32(tO + cc * 32, ov);
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
          for (int jj = 0; jj < 16; ++jj) {
            const int j = half * 64 + 4 * jj;
            const float4 v4 = vs4[j >> 2];
            const float p0 = ex2(__uint_as_float(sv[j]) - mu), p1 = ex2(__uint_as_float(sv[j + 1]) - mu);
            const float p2 = ex2(__uint_as_float(sv[j + 2]) - mu), p3 = ex2(__uint_as_float(sv[j + 3]) - mu);
            lsp[(2 * jj) & 7] += p0 + p1;
            lsp[(2 * jj + 1) & 7] += p2 + p3;
            // V scales multiply the probabilities after the row sum
            pk[2 * jj] = pack_f16x2(p0 * v4.x, p1 * v4.y);
            pk[2 * jj + 1] = pack_f16x2(p2 * v4.z, p3 * v4.w);
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
      __syncwarp();
      if (lane == 0) mbar_arrive(&aux_empty[a]);
    }
    if (ok && kx > 0) ok = wait_bar(&pv_done[x], (kx - 1) & 1, ab);
    if (ok) {
      if (kx > 0) tc_fence_after();
      if (direct) {
        if (kx > 0) {
          const float inv = 1.f / (kPScale * l);
          uint16_t* orow = p.out + (size_t)(q_begin + posc) * p.out_ts + (size_t)(kvh * G + head) * p.out_hs;
#pragma unroll 1
          for (int cc = 0; cc < kD / 32; ++cc) {
            uint32_t ov[32];
            tmem_ld32(tO + cc * 32, ov);
            tmem_ld_wait();
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[j] = pack_bf16x2(__uint_as_float(ov[2 * j]) * inv, __uint_as_float(ov[2 * j + 1]) * inv);
            if (row_valid) {
              uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
              for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            }
          }
        }
      } else {
        const size_t row = unit * rows_per_unit + (size_t)posc * G + head;
        float4* arow = reinterpret_cast<float4*>(p.part_acc + row * kD);
        if (kx > 0) {
          constexpr float kInv = 1.f / kPScale;
#pragma unroll 1
          for (int cc = 0; cc < kD / 32; ++cc) {
            uint32_t ov[32];
            tmem_ld32(tO + cc * 32, ov);
            tmem_ld_wait();
            if (row_valid) {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                arow[cc * 8 + j] = make_float4(__uint_as_float(ov[4 * j]) * kInv, __uint_as_float(ov[4 * j + 1]) * kInv,
                                               __uint_as_float(ov[4 * j + 2]) * kInv,
                                               __uint_as_float(ov[4 * j + 3]) * kInv);
            }
          }
        } else if (row_valid) {
          for (int j = 0; j < kD / 4; ++j) arow[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (row_valid)
          reinterpret_cast<float2*>(p.part_ml)[row] = kx > 0 ? make_float2(m, l) : make_float2(neg_inf(), 0.f);
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

template <bool FEAT>
cudaError_t launch_t(const DecodeParams& p, const DecodeMaps& maps, int qpairs, cudaStream_t s) {
  using C = PpCfg<FEAT>;
  auto kern = prefill_paged_kernel<FEAT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<dim3(qpairs * p.max_segs, p.hkv, p.num_reqs), kThreads, C::SMEM, s>>>(maps.k, maps.v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_paged(const DecodeParams& p, const DecodeMaps& maps, cudaStream_t s,
                                 const cudaEvent_t* ev_before, const cudaEvent_t* ev_after) {
  const int pos_pair = 2 * (128 / p.group);  // query positions of one CTA
  const int qpairs = (p.max_q_len + pos_pair - 1) / pos_pair;
  if (ev_before && *ev_before) cudaEventRecord(*ev_before, s);
  const bool feat = p.g_cache != nullptr || p.window > 0;
  cudaError_t e = feat ? launch_t<true>(p, maps, qpairs, s) : launch_t<false>(p, maps, qpairs, s);
  if (ev_after && *ev_after) cudaEventRecord(*ev_after, s);
  if (e != cudaSuccess) return e;
  if (p.part_acc == nullptr) return cudaSuccess;
  return launch_decode_combine(p, s);
}

}  // namespace gcs
