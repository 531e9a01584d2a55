// Paged decode / short-query attention over an fp8 e4m3 KV cache with per-token scales.
//
// ROCm/aiter PR #6660 (gfx1250 unified attention), commit messages and "Technical
// details": one fp32 K and V scale per cached token and KV head, laid out [num_blocks,
// num_kv_heads, block_size]; each tile is one page; K scales multiply the QK columns; V
// scales multiply the P columns after the row sum; slots past seq_len get scale 0; the
// context is split into segments (split-K) whose partials are merged by an LSE-weighted
// reduce in which an empty partial (M = -inf) weighs 0.
//
// decode_split_kernel: one CTA per (segment, kv head, request).  Warp 0 streams pages
// (K 2 KB, V 2 KB, 16 K scales, 16 V scales) into a 16-stage shared-memory ring, eight pages
// per round: each of its 32 lanes issues one of the round's 32 copies (a copy is a
// per-thread instruction, and one lane issuing them all serially was the bottleneck).  A
// "page" here is 16 tokens: a cache block of block_size = 16 k tokens holds k of them at
// consecutive slots.  The
// fp8 K and V pages come by tensor copy with the 128-byte swizzle, so the consumers' 16-B
// reads of four rows at one column, or of two columns of two rows, hit eight different bank
// groups; the scales (and gates) come by plain bulk copy.  Warps 1..4 each own one m16 MMA
// tile of query rows -- the 16 query heads of a GQA group of 16 at one query position, or the
// 8 heads of a group of 8 at two consecutive positions (rows 0-7 and 8-15) -- and a share of
// the pages (the query's MMA fragments are kept in
// shared memory, one copy per query position, so the loop runs without register spills);
// fp8 -> f16 conversion is exact,
// QK^T and PV run on mma.sync m16n8k16 with fp32 accumulation, softmax in fp32 (log2
// units).  A row's reference max moves only when its max grows by more than 2^3, so P <= 8
// and most pages skip the accumulator rescale; P * vscale is scaled by 2^5 before the f16
// rounding (round-to-nearest, no truncation bias) and the factor is removed in fp32 afterwards.
// decode_combine_kernel: LSE-weighted merge of the segments of each (query row, head).
#include <mutex>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace gcs {
namespace {

// Fixed scratch for the allocation-free decode entry point: the split-K partials live
// here instead of in a caller-provided workspace.  Every GPU that loads the library
// holds this array until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
constexpr int kMaxScratchDevices = 64;
void* g_noalloc_ptr[kMaxScratchDevices] = {nullptr};
std::mutex g_noalloc_mu;

constexpr int kPage = 16;
constexpr int kD = 128;
constexpr int kRows = 16;  // rows of an m16 tile; partial rows per (unit, query position)
// Ring layout: a K | V ring of NST pages (fp8: 2 KB + 2 KB, rows of 128 B stored with the
// 128-byte swizzle of the tensor copy; bf16: 4 KB + 4 KB, linear) and, beside it, a ring of
// the pages' small vectors: K and V scales (per-token fp8, 64 B each) and, with the decoding
// features, the cumulative gates of the group's 16 query heads (16 x 16 fp32 = 1 KB).
// Stages fill ~72 KB (three CTAs per SM); the producer issues BATCH pages per round, one
// copy per lane.
template <int KVF, bool PT, bool FEAT, bool SQ>
struct DecCfg {
  static constexpr int KB = KVF == 0 ? 2048 : 4096;  // bytes of one page of K (or V) for one kv head
  static constexpr bool SCALES = KVF == 0 && !PT;    // per-token scale copies
  static constexpr int KV = 2 * KB;                  // K | V of one page (a multiple of 1 KB)
  static constexpr int G_OFF = SCALES ? 128 : 0;     // gates inside a small-vector stage
  static constexpr int AUX = G_OFF + (FEAT ? 1024 : 0);
  // Ring budget: ~72 KB, three CTAs per SM with the query fragments of one position (4 KB).
  // SQ (3 or 4 query positions, 16 KB of fragments) trims the ring so that three CTAs still
  // fit: short-query calls are latency-bound, and 12 consumer warps per SM beat 8 with a
  // deeper ring.
  static constexpr int BUDGET = SQ ? 57 * 1024 : 72 * 1024;
  // NST is a multiple of 4: the page groups of a CTA are 4 / (query tiles) warps (4, 2 or 1),
  // so the previous page of every stage belongs to the warp that waits for the stage's next
  // page.  That warp has therefore seen the previous phase complete, and a full-barrier parity
  // wait cannot match the phase before it (which a stage consumed by another warp could, while
  // the previous page's copy is still in flight).
  static constexpr int NST = ((BUDGET / (KV + AUX)) < 16 ? (BUDGET / (KV + AUX)) : 16) & ~3;
  static constexpr int OFF_AUX = NST * KV;
  static constexpr int SMEM = OFF_AUX + NST * AUX + 1024;  // + alignment of the base to 1 KB
  static constexpr int KINDS = 2 + (SCALES ? 2 : 0) + (FEAT ? 1 : 0);  // K, V (, K/V scales) (, gates)
  // pages per producer round: a power of two, one copy per lane, at most half the ring
  static constexpr int BATCH = (KINDS * 8 <= 32 && NST >= 16) ? 8 : (NST >= 8 ? 4 : 2);
  static_assert(NST % 4 == 0 && NST >= 4, "stages per page-group warp");
  static_assert(KINDS * BATCH <= 32 && NST >= 2 * BATCH, "producer round");
};
constexpr int kThreads = 160;
constexpr float kLog2e = 1.4426950408889634f;
// Each row's reference max moves only when the row max grows by more than 2^kLazy (log2 units),
// so P <= 2^3; the fp8 path rounds P * vscale to f16 after a 2^5 pre-scale, which keeps
// 2^3 * 255 * 2^5 = 65280 below the f16 maximum for every V scale below 255.
constexpr float kLazy = 3.f;
constexpr float kPScale = 32.f;
constexpr float kInvPScale = 1.f / 32.f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

// two e4m3 bytes (low byte = first element) -> f16x2 (low half = first element)
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t bf16pair_to_f16x2(uint32_t w) {
  const float lo = __uint_as_float(w << 16);
  const float hi = __uint_as_float(w & 0xffff0000u);
  return pack_f16x2(lo, hi);
}

// KVF: 0 fp8 e4m3 codes, 1 bf16 values.  PT: one K and one V scale for the whole cache (fp8).
// FEAT: the decoding features (gates from g_cache when given, the window; the sink is the
// combine's).  G: query heads per kv head, 16 or 8.  SQ: 3 or 4 query positions (a smaller
// ring).  PG1: cache blocks of one 16-token page (the page index is the block-table index,
// which keeps the producer's first copies of a CTA a few instructions shorter).
template <int KVF, bool PT, bool FEAT, int G, bool SQ, bool PG1>
__global__ void __launch_bounds__(kThreads, 3)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const DecodeParams p) {
  using C = DecCfg<KVF, PT, FEAT, SQ>;
  constexpr int kNST = C::NST, kBatch = C::BATCH;
  constexpr int kKinds = C::KINDS;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the swizzled tensor copies want 1 KB-aligned pages
  uint8_t* kv = smem_align_1k(smem_raw);
  uint8_t* aux = kv + C::OFF_AUX;
  __shared__ uint64_t full[kNST], empty[kNST];
  __shared__ int abort_flag_s;
  const int seg = blockIdx.x, kvh = blockIdx.y, r = blockIdx.z;
  const int L = __ldg(p.seq_lens + r);
  const int q_begin = __ldg(p.cu_q + r);
  const int ql = __ldg(p.cu_q + r + 1) - q_begin;
  const int npages = (L + kPage - 1) / kPage;
  int pb = seg * p.seg_pages;
  if (pb >= npages || ql < 1 || ql > 4) return;
  constexpr int ppt = kRows / G;  // query positions per m16 tile: 1 or 2
  const int ntile = (ql + ppt - 1) / ppt;
  const int lbp = p.log2_block_pages;  // cache blocks hold 2^lbp 16-token pages
  const int pend = min(pb + p.seg_pages, npages);
  if (FEAT && p.window > 0) {
    // pages before the earliest key any query row of the request sees are skipped; a segment
    // that lies wholly before them writes nothing (the combine starts after it)
    const int first_page = max(0, L - ql - p.window + 1) / kPage;
    if (pend <= first_page) return;
    pb = max(pb, first_page);
  }
  const int np = pend - pb;
  const bool has_gate = FEAT && p.g_cache != nullptr;
  const int ng = 4 / ntile;  // page groups

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], ntile);
    }
    abort_flag_s = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Abort ab{&abort_flag_s, p.status};

  if (warp == 0) {
    // ------------------------------------------------------------ page producer
    // lane = kBatch * kind + page within the round; kind 0: K, 1: V, then (per-token fp8)
    // 2: K scales, 3: V scales, then (features) the gates of the group's query heads
    const int32_t* trow = p.block_table + (size_t)r * p.max_blocks;
    const int pl = lane & (kBatch - 1), kind = lane / kBatch;
    const int g_kind = C::SCALES ? 4 : 2;
    const bool is_g = FEAT && kind == g_kind;
    const uint32_t bytes = kind < 2 ? C::KB : is_g ? G * kPage * 4 : kPage * 4;
    const uint32_t dst_off = kind < 2 ? kind * C::KB : is_g ? C::G_OFF : (kind - 2) * 64;
    if (KVF == 0 && lane == 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
    }
    const uint32_t tx = 2 * C::KB + (C::SCALES ? 2 * kPage * 4 : 0) + (has_gate ? G * kPage * 4 : 0);
    // each lane's block-table entry for its page of the next round is read one round ahead, so
    // the read's latency overlaps this round's waits and copies
    const bool lane_kind = kind < kKinds && (!is_g || has_gate);
    auto table_entry = [&](int i) -> int {
      const int pg = pb + i;
      return (lane_kind && i < np) ? (PG1 ? __ldg(trow + pg) : __ldg(trow + (pg >> lbp))) : 0;
    };
    int blk_next = table_entry(pl);
    for (int base = 0; base < np; base += kBatch) {
      const int i = base + pl;
      const bool act = i < np && lane_kind;
      const int stage = i % kNST;
      const int blk = blk_next;  // block of this lane's page
      blk_next = table_entry(i + kBatch);
      bool okl = true;
      if (act) okl = wait_bar(&empty[stage], ((i / kNST) & 1) ^ 1, ab);
      if (!__all_sync(0xffffffffu, okl)) break;
      if (act && kind == 0) mbar_expect_tx(&full[stage], tx);
      __syncwarp();
      if (act) {
        const int pg = pb + i;
        const int sub = PG1 ? 0 : (pg & ((1 << lbp) - 1)) * kPage;           // first slot of the page
        const size_t slot0 = ((size_t)blk * p.hkv + kvh) * p.block_size + sub;
        if (KVF == 0 && kind < 2) {
          // fp8 K or V page: one 16-slot x 128-B box of the cache's 4-D map (dims in stride order)
          tma_load_4d(kv + stage * C::KV + dst_off, kind ? &tmV : &tmK, &full[stage], 0, p.kv_head_inner ? kvh : sub,
                      p.kv_head_inner ? sub : kvh, blk);
        } else if (kind < 2) {
          // bf16 K or V page: one 4 KB copy when its 16 rows are adjacent, else one per row
          const uint8_t* src = (kind == 0 ? p.k_cache : p.v_cache) + (size_t)blk * p.kv_bs + (size_t)kvh * p.kv_hs +
                               (size_t)sub * p.kv_ss;
          uint8_t* dst = kv + stage * C::KV + dst_off;
          if (p.kv_ss == C::KB / kPage) {
            bulk_load(dst, src, bytes, &full[stage]);
          } else {
            for (int rr = 0; rr < kPage; ++rr)
              bulk_load(dst + rr * (C::KB / kPage), src + rr * p.kv_ss, C::KB / kPage, &full[stage]);
          }
        } else if (is_g) {
          // the group's G heads x 16 slots of gates: adjacent when a block is one page
          const float* src = p.g_cache + ((size_t)blk * p.hq + kvh * G) * p.block_size + sub;
          if (lbp == 0) {
            bulk_load(aux + stage * C::AUX + dst_off, src, bytes, &full[stage]);
          } else {
            for (int hh = 0; hh < G; ++hh)
              bulk_load(aux + stage * C::AUX + dst_off + hh * kPage * 4, src + (size_t)hh * p.block_size, kPage * 4,
                        &full[stage]);
          }
        } else {
          bulk_load(aux + stage * C::AUX + dst_off, (kind == 2 ? p.k_scale : p.v_scale) + slot0, bytes, &full[stage]);
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int mt = cw % ntile, grp = cw / ntile;
  const bool active = grp < ng;
  const int g = lane >> 2, tq = lane & 3;
  // tile rows g (A) and g + 8 (B): (query position, head of the group) = (mt, g) and (mt, g + 8)
  // for a group of 16; (2 mt, g) and (2 mt + 1, g) for a group of 8 (row B unused past q_len)
  const int posA = mt * ppt, posB = mt * ppt + ppt - 1;
  const int headA = g, headB = ppt == 2 ? g : g + 8;
  const bool validB = posB < ql;
  const int lastkA = L - ql + posA;                  // last key visible to row A
  const int lastkB = ppt == 1 ? lastkA : validB ? L - ql + posB : -1;  // and to row B (none past q_len)
  // a page whose slots all lie at or below both rows' last keys (and, with a window, above
  // both windows' starts) needs no per-slot masks; with row B past q_len no page qualifies
  const int lastk_min = min(lastkA, lastkB), lastk_max = max(lastkA, lastkB);
  const float sl2 = p.scale * kLog2e;
  float o[16][4];
#pragma unroll
  for (int u = 0; u < 16; ++u) o[u][0] = o[u][1] = o[u][2] = o[u][3] = 0.f;
  float m0 = neg_inf(), m1 = neg_inf(), l0 = 0.f, l1 = 0.f;
  bool ok = true;

  // query fragments in shared memory, one copy per query position: [8 k-steps][32 lanes]
  uint4* qf = reinterpret_cast<uint4*>(aux + C::NST * C::AUX) + mt * (8 * 32);
  if (active && grp == 0) {
    uint32_t qa[8][4];
    {
      const uint16_t* q0p = p.q + (size_t)(q_begin + posA) * p.q_ts + (size_t)(kvh * G + headA) * p.q_hs + 32 * tq;
      const uint16_t* q1p =
          p.q + (size_t)(q_begin + min(posB, ql - 1)) * p.q_ts + (size_t)(kvh * G + headB) * p.q_hs + 32 * tq;
      uint32_t w0[16], w1[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(q0p) + j);
        const uint4 b = validB ? __ldg(reinterpret_cast<const uint4*>(q1p) + j) : make_uint4(0u, 0u, 0u, 0u);
        w0[4 * j] = a.x; w0[4 * j + 1] = a.y; w0[4 * j + 2] = a.z; w0[4 * j + 3] = a.w;
        w1[4 * j] = b.x; w1[4 * j + 1] = b.y; w1[4 * j + 2] = b.z; w1[4 * j + 3] = b.w;
      }
      // k-step s covers physical dims 32tq + 4s .. 32tq + 4s + 3 of this thread; the fp8
      // path multiplies in f16 (exact e4m3 -> f16), the bf16 path in bf16
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        qa[s][0] = KVF == 0 ? bf16pair_to_f16x2(w0[2 * s]) : w0[2 * s];
        qa[s][1] = KVF == 0 ? bf16pair_to_f16x2(w1[2 * s]) : w1[2 * s];
        qa[s][2] = KVF == 0 ? bf16pair_to_f16x2(w0[2 * s + 1]) : w0[2 * s + 1];
        qa[s][3] = KVF == 0 ? bf16pair_to_f16x2(w1[2 * s + 1]) : w1[2 * s + 1];
      }
    }
#pragma unroll
    for (int s = 0; s < 8; ++s) qf[s * 32 + lane] = make_uint4(qa[s][0], qa[s][1], qa[s][2], qa[s][3]);
  }
  named_bar_sync(1, 128);
  if (active) {
    // one K and one V scale for the whole cache (fp8 per-tensor)
    const float kst = PT ? __ldg(p.k_scale) : 1.f, vst = PT ? __ldg(p.v_scale) : 1.f;
    // each row's own cumulative gate (log2 units) at its position
    float gq0 = 0.f, gq1 = 0.f;
    if (has_gate) {
      const int32_t* trow = p.block_table + (size_t)r * p.max_blocks;
      const int kB = validB ? lastkB : lastkA;  // row B past q_len reads row A's entry (unused)
      const int bA = __ldg(trow + lastkA / p.block_size), bB = __ldg(trow + kB / p.block_size);
      gq0 = __ldg(p.g_cache + ((size_t)bA * p.hq + kvh * G + headA) * p.block_size + lastkA % p.block_size) * kLog2e;
      gq1 = __ldg(p.g_cache + ((size_t)bB * p.hq + kvh * G + headB) * p.block_size + kB % p.block_size) * kLog2e;
    }
    for (int i = grp; i < np; i += ng) {
      const int stage = i % kNST;
      ok = wait_bar(&full[stage], (i / kNST) & 1, ab);
      if (!ok) break;
      const uint8_t* st = kv + stage * C::KV;    // K page | V page
      const uint8_t* sa = aux + stage * C::AUX;  // K scales | V scales | gates
      // gates of this thread's four keys for heads g and g + 8 (read before the stage is freed)
      float gk[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if (has_gate) {
        const float* gs = reinterpret_cast<const float*>(sa + C::G_OFF);
#pragma unroll
        for (int rw2 = 0; rw2 < 2; ++rw2) {
          const int hd = rw2 ? headB : headA;
          const float2 a = *reinterpret_cast<const float2*>(gs + hd * kPage + 2 * tq);
          const float2 b = *reinterpret_cast<const float2*>(gs + hd * kPage + 8 + 2 * tq);
          gk[rw2][0] = a.x; gk[rw2][1] = a.y; gk[rw2][2] = b.x; gk[rw2][3] = b.y;
        }
      }
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
      float ks[4], vs[4];  // K / V scale of this thread's four columns
      if constexpr (KVF == 0) {
        // dims 32tq .. 32tq + 31 of keys g and g + 8: 16-B units 2tq and 2tq + 1 of those rows,
        // at unit ^ (row & 7) in the swizzled page (conflict-free across each quarter warp)
        const uint32_t u0 = ((2 * tq) ^ (g & 7)) << 4, u1 = ((2 * tq + 1) ^ (g & 7)) << 4;
        const uint4 ka0 = lds128(st + g * kD + u0);
        const uint4 ka1 = lds128(st + g * kD + u1);
        const uint4 kb0 = lds128(st + (8 + g) * kD + u0);
        const uint4 kb1 = lds128(st + (8 + g) * kD + u1);
        if constexpr (PT) {
          ks[0] = ks[1] = ks[2] = ks[3] = kst;
          vs[0] = vs[1] = vs[2] = vs[3] = vst;
        } else {
          const float2 ksA = *reinterpret_cast<const float2*>(sa + 8 * tq);
          const float2 ksB = *reinterpret_cast<const float2*>(sa + 32 + 8 * tq);
          const float2 vsA = *reinterpret_cast<const float2*>(sa + 64 + 8 * tq);
          const float2 vsB = *reinterpret_cast<const float2*>(sa + 64 + 32 + 8 * tq);
          ks[0] = ksA.x; ks[1] = ksA.y; ks[2] = ksB.x; ks[3] = ksB.y;
          vs[0] = vsA.x; vs[1] = vsA.y; vs[2] = vsB.x; vs[3] = vsB.y;
        }
        // (values are read after the softmax and the stage is released then: fewer live registers)
        // S = q . k8 over the page: n-tile 0 = slots 0..7, n-tile 1 = slots 8..15
        const uint32_t kw0[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
        const uint32_t kw1[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          uint32_t b0, b1;
          const uint4 qv = qf[s * 32 + lane];
          const uint32_t qa[4] = {qv.x, qv.y, qv.z, qv.w};
          e4m3x4_to_f16x2x2(kw0[s], b0, b1);
          mma_f16(s0, qa, b0, b1);
          e4m3x4_to_f16x2x2(kw1[s], b0, b1);
          mma_f16(s1, qa, b0, b1);
        }
      } else {
        // bf16 page: 16 keys x 256 B; this thread's 32 dims of keys g and g + 8 (64 B each)
        uint32_t kw0[16], kw1[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 a = lds128(st + g * 256 + 64 * tq + 16 * c);
          const uint4 b = lds128(st + (8 + g) * 256 + 64 * tq + 16 * c);
          kw0[4 * c] = a.x; kw0[4 * c + 1] = a.y; kw0[4 * c + 2] = a.z; kw0[4 * c + 3] = a.w;
          kw1[4 * c] = b.x; kw1[4 * c + 1] = b.y; kw1[4 * c + 2] = b.z; kw1[4 * c + 3] = b.w;
        }
        ks[0] = ks[1] = ks[2] = ks[3] = 1.f;
        vs[0] = vs[1] = vs[2] = vs[3] = 1.f;
        // (values are read after the softmax and the stage is released then: fewer live registers)
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint4 qv = qf[s * 32 + lane];
          const uint32_t qa[4] = {qv.x, qv.y, qv.z, qv.w};
          mma_bf16(s0, qa, kw0[2 * s], kw0[2 * s + 1]);
          mma_bf16(s1, qa, kw1[2 * s], kw1[2 * s + 1]);
        }
      }
      // this thread's columns: slots 2tq, 2tq+1 (n-tile 0) and 8+2tq, 9+2tq (n-tile 1)
      const int tok0 = (pb + i) * kPage + 2 * tq;
      const int tk[4] = {tok0, tok0 + 1, tok0 + 8, tok0 + 9};
      const int pfirst = (pb + i) * kPage;
      const bool inner = pfirst + kPage - 1 <= lastk_min &&
                         !(FEAT && p.window > 0 && pfirst <= lastk_max - p.window);  // uniform per warp
      float x[2][4];  // [row g / g+8][column]
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float sa = (c < 2) ? s0[c] : s1[c - 2];
        const float sb = (c < 2) ? s0[c + 2] : s1[c];
        if (FEAT) {  // + G_i - G_j
          x[0][c] = fmaf(sa, sl2 * ks[c], fmaf(-gk[0][c], kLog2e, gq0));
          x[1][c] = fmaf(sb, sl2 * ks[c], fmaf(-gk[1][c], kLog2e, gq1));
        } else {
          x[0][c] = sa * sl2 * ks[c];
          x[1][c] = sb * sl2 * ks[c];
        }
      }
      if (!inner) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          bool visA = tk[c] <= lastkA, visB = tk[c] <= lastkB;
          if (FEAT && p.window > 0) {
            visA = visA && tk[c] > lastkA - p.window;
            visB = visB && tk[c] > lastkB - p.window;
          }
          if (!visA) x[0][c] = neg_inf();
          if (!visB) x[1][c] = neg_inf();
        }
      }
      float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[0][2], x[0][3]));
      float mx1 = fmaxf(fmaxf(x[1][0], x[1][1]), fmaxf(x[1][2], x[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      // a row's reference max moves (and its accumulators are rescaled) only when the row max
      // grows by more than 2^kLazy; a first finite max always moves it (-inf + kLazy = -inf)
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      const bool up0 = n0 > m0 + kLazy, up1 = n1 > m1 + kLazy;
      const float a0 = up0 ? ex2(m0 - n0) : 1.f;
      const float a1 = up1 ? ex2(m1 - n1) : 1.f;
      if (up0) m0 = n0;
      if (up1) m1 = n1;
      const float u0 = (m0 == neg_inf()) ? 0.f : m0;
      const float u1 = (m1 == neg_inf()) ? 0.f : m1;
      float pr[2][4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        pr[0][c] = ex2(x[0][c] - u0);
        pr[1][c] = ex2(x[1][c] - u1);
      }
      l0 = l0 * a0 + (pr[0][0] + pr[0][1]) + (pr[0][2] + pr[0][3]);
      l1 = l1 * a1 + (pr[1][0] + pr[1][1]) + (pr[1][2] + pr[1][3]);
      // the accumulators change only where a row's reference moved (the factor is 1 elsewhere)
      if (__any_sync(0xffffffffu, up0 || up1)) {
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          o[u][0] *= a0;
          o[u][1] *= a0;
          o[u][2] *= a1;
          o[u][3] *= a1;
        }
      }
      // V scales multiply the probabilities after the row sum; slots >= L get scale 0, and
      // their value bytes are never multiplied (NaN allowed there)
#pragma unroll
      for (int c = 0; c < 4; ++c) vs[c] *= KVF == 0 ? kPScale : 1.f;
      if (!inner) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (tk[c] >= L) vs[c] = 0.f;
      }
      if constexpr (KVF == 0) {
        uint32_t pa[4];
        pa[0] = pack_f16x2(pr[0][0] * vs[0], pr[0][1] * vs[1]);
        pa[1] = pack_f16x2(pr[1][0] * vs[0], pr[1][1] * vs[1]);
        pa[2] = pack_f16x2(pr[0][2] * vs[2], pr[0][3] * vs[3]);
        pa[3] = pack_f16x2(pr[1][2] * vs[2], pr[1][3] * vs[3]);
        // value fragments: dims 16g .. 16g + 15 (16-B unit g) of slots 2tq, 2tq+1, 2tq+8, 2tq+9;
        // slots at or past seq_len are zero (NaN allowed in their bytes)
        uint4 vr[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int row = 2 * tq + (c & 1) + 8 * (c >> 1);
          vr[c] = lds128(st + C::KB + row * kD + ((g ^ (row & 7)) << 4));
        }
        if (!inner) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (tk[c] >= L) vr[c] = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        const uint32_t va[4] = {vr[0].x, vr[0].y, vr[0].z, vr[0].w}, vb[4] = {vr[1].x, vr[1].y, vr[1].z, vr[1].w};
        const uint32_t vc[4] = {vr[2].x, vr[2].y, vr[2].z, vr[2].w}, vd[4] = {vr[3].x, vr[3].y, vr[3].z, vr[3].w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t lo01, hi01, lo23, hi23;
          // bytes (4w, 4w+1) of slots (2tq, 2tq+1) interleaved, then bytes (4w+2, 4w+3)
          const uint32_t ab01 = prmt(va[w], vb[w], 0x5140);
          const uint32_t ab23 = prmt(va[w], vb[w], 0x7362);
          const uint32_t cd01 = prmt(vc[w], vd[w], 0x5140);
          const uint32_t cd23 = prmt(vc[w], vd[w], 0x7362);
          uint32_t b0, b1;
          e4m3x4_to_f16x2x2(ab01, lo01, hi01);
          e4m3x4_to_f16x2x2(cd01, b0, b1);
          mma_f16(o[4 * w + 0], pa, lo01, b0);
          mma_f16(o[4 * w + 1], pa, hi01, b1);
          e4m3x4_to_f16x2x2(ab23, lo23, hi23);
          e4m3x4_to_f16x2x2(cd23, b0, b1);
          mma_f16(o[4 * w + 2], pa, lo23, b0);
          mma_f16(o[4 * w + 3], pa, hi23, b1);
        }
      } else {
        uint32_t pa[4];
        pa[0] = pack_bf16x2(pr[0][0] * vs[0], pr[0][1] * vs[1]);
        pa[1] = pack_bf16x2(pr[1][0] * vs[0], pr[1][1] * vs[1]);
        pa[2] = pack_bf16x2(pr[0][2] * vs[2], pr[0][3] * vs[3]);
        pa[3] = pack_bf16x2(pr[1][2] * vs[2], pr[1][3] * vs[3]);
        // values of rows 2tq, 2tq+1, 2tq+8, 2tq+9 (tk[0..3]), dims 16g .. 16g + 15 (32 B each);
        // rows at or past seq_len are zero (NaN allowed in their bytes)
        uint32_t rw[4][8];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const int row = 2 * tq + (rr & 1) + 8 * (rr >> 1);
          uint4 a = lds128(st + C::KB + row * 256 + 32 * g), b = lds128(st + C::KB + row * 256 + 32 * g + 16);
          if (!inner && tk[rr] >= L) a = b = make_uint4(0, 0, 0, 0);
          rw[rr][0] = a.x; rw[rr][1] = a.y; rw[rr][2] = a.z; rw[rr][3] = a.w;
          rw[rr][4] = b.x; rw[rr][5] = b.y; rw[rr][6] = b.z; rw[rr][7] = b.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const uint32_t sel = (u & 1) ? 0x7632 : 0x5410;
          const uint32_t b0 = prmt(rw[0][u >> 1], rw[1][u >> 1], sel);  // keys 2tq, 2tq + 1
          const uint32_t b1 = prmt(rw[2][u >> 1], rw[3][u >> 1], sel);  // keys 2tq + 8, 2tq + 9
          mma_bf16(o[u], pa, b0, b1);
        }
      }
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }

  // ------------------------------------------------ merge page groups, write the partial
  // thread (g, tq) holds dims 32tq + u (o[u][0], o[u][2]) and 32tq + 16 + u (o[u][1], o[u][3])
  float* red = reinterpret_cast<float*>(kv);  // reuses the ring: [4 warps][16 rows][130]
  if (ng > 1) {
    named_bar_sync(1, 128);  // every consumer is done with the ring
    if (active) {
      float* mine = red + cw * (16 * 130);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        mine[g * 130 + 32 * tq + u] = o[u][0];
        mine[g * 130 + 32 * tq + 16 + u] = o[u][1];
        mine[(g + 8) * 130 + 32 * tq + u] = o[u][2];
        mine[(g + 8) * 130 + 32 * tq + 16 + u] = o[u][3];
      }
      if (tq == 0) {
        mine[g * 130 + 128] = m0;
        mine[g * 130 + 129] = l0;
        mine[(g + 8) * 130 + 128] = m1;
        mine[(g + 8) * 130 + 129] = l1;
      }
    }
    named_bar_sync(1, 128);
    if (active && grp == 0) {
      for (int gg = 1; gg < ng; ++gg) {
        const float* other = red + (gg * ntile + mt) * (16 * 130);
        const float om0 = other[g * 130 + 128], ol0 = other[g * 130 + 129];
        const float om1 = other[(g + 8) * 130 + 128], ol1 = other[(g + 8) * 130 + 129];
        const float n0 = fmaxf(m0, om0), n1 = fmaxf(m1, om1);
        const float wa0 = (m0 == neg_inf()) ? 0.f : ex2(m0 - n0);
        const float wb0 = (om0 == neg_inf()) ? 0.f : ex2(om0 - n0);
        const float wa1 = (m1 == neg_inf()) ? 0.f : ex2(m1 - n1);
        const float wb1 = (om1 == neg_inf()) ? 0.f : ex2(om1 - n1);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          o[u][0] = o[u][0] * wa0 + other[g * 130 + 32 * tq + u] * wb0;
          o[u][1] = o[u][1] * wa0 + other[g * 130 + 32 * tq + 16 + u] * wb0;
          o[u][2] = o[u][2] * wa1 + other[(g + 8) * 130 + 32 * tq + u] * wb1;
          o[u][3] = o[u][3] * wa1 + other[(g + 8) * 130 + 32 * tq + 16 + u] * wb1;
        }
        l0 = l0 * wa0 + ol0 * wb0;
        l1 = l1 * wa1 + ol1 * wb1;
        m0 = n0;
        m1 = n1;
      }
    }
  }
  if (active && grp == 0) {
    constexpr float kOut = KVF == 0 ? kInvPScale : 1.f;  // the fp8 path carries P scaled by 2^5
    const size_t unit = ((size_t)r * p.max_segs + seg) * p.hkv + kvh;
    const int rows = p.max_q_len * kRows;
    const size_t row0 = unit * rows + posA * G + headA;
    // row B past q_len (group of 8, odd q_len) writes its all-empty result into its own slot,
    // which the combine never reads
    const size_t row1 = unit * rows + posB * G + headB;
    float4* d0 = reinterpret_cast<float4*>(p.part_acc + row0 * kD + 32 * tq);
    float4* d1 = reinterpret_cast<float4*>(p.part_acc + row1 * kD + 32 * tq);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      d0[k] = make_float4(o[4 * k][0] * kOut, o[4 * k + 1][0] * kOut, o[4 * k + 2][0] * kOut,
                          o[4 * k + 3][0] * kOut);
      d0[4 + k] = make_float4(o[4 * k][1] * kOut, o[4 * k + 1][1] * kOut, o[4 * k + 2][1] * kOut,
                              o[4 * k + 3][1] * kOut);
      d1[k] = make_float4(o[4 * k][2] * kOut, o[4 * k + 1][2] * kOut, o[4 * k + 2][2] * kOut,
                          o[4 * k + 3][2] * kOut);
      d1[4 + k] = make_float4(o[4 * k][3] * kOut, o[4 * k + 1][3] * kOut,
                              o[4 * k + 2][3] * kOut, o[4 * k + 3][3] * kOut);
    }
    if (tq == 0) {
      reinterpret_cast<float2*>(p.part_ml)[row0] = make_float2(m0, l0);
      reinterpret_cast<float2*>(p.part_ml)[row1] = make_float2(m1, l1);
    }
  }
}

// Online merge of a partial (m2, l2, a2) into (m, l, a): both are relative to their own
// reference max (log2 units); an empty partial has m = -inf and weighs 0.
__device__ __forceinline__ void merge_partial(float& m, float& l, float (&a)[8], float m2, float l2,
                                              const float (&a2)[8]) {
  const float M = fmaxf(m, m2);
  const float w1 = (m == neg_inf()) ? 0.f : ex2(m - M);
  const float w2 = (m2 == neg_inf()) ? 0.f : ex2(m2 - M);
  l = w1 * l + w2 * l2;
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = w1 * a[j] + w2 * a2[j];
  m = M;
}

// One CTA per (request x query position, kv head, 16 / SL query heads); 256 threads = 16 / SL
// heads x 16 groups of 8 value dims x SL segment lanes.  The SL lanes of a (head, dims) pair are
// adjacent: each merges every SL-th segment online (their loads are independent), then log2 SL
// shuffle rounds merge them.  SL = 4 for short contexts, 8 from 32 segments on (fewer serial
// merges per lane: 3 x 4 queries at 227K, 114 segments, 20.1 -> 17.5 us per combine; 16 lanes
// measured no better than 4 there, and 16 lanes on 16 segments cost the 64 x 1 call 8 us).
template <int SL>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeParams p) {
  constexpr int kHeads = 16 / SL;  // query heads per CTA
  const int r = blockIdx.x / p.max_q_len, t = blockIdx.x % p.max_q_len;
  const int kvh = blockIdx.y;
  const int q_begin = __ldg(p.cu_q + r);
  const int ql = __ldg(p.cu_q + r + 1) - q_begin;
  if (t >= ql) return;
  const int L = __ldg(p.seq_lens + r);
  const int npages = (L + kPage - 1) / kPage;
  const int nseg = (npages + p.seg_pages - 1) / p.seg_pages;
  const int G = p.group;
  const int sl = threadIdx.x & (SL - 1), dg = (threadIdx.x / SL) & 15;
  const int hh = blockIdx.z * kHeads + threadIdx.x / (16 * SL);
  const int d0 = dg * 8;
  const int rows = p.max_q_len * kRows;
  const int row = t * G + hh;
  auto unit_row = [&](int s) { return ((((size_t)r * p.max_segs + s) * p.hkv + kvh) * rows + row); };
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  // segments wholly before every window of the request were not written (see the split kernel)
  const int s_begin = p.window > 0 ? (max(0, L - ql - p.window + 1) / kPage) / p.seg_pages : 0;
  float m = neg_inf(), l = 0.f;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (hh < G) {
#pragma unroll 2
    for (int s = s_begin + sl; s < nseg; s += SL) {
      const float2 v = ml[unit_row(s)];
      const float4* a = reinterpret_cast<const float4*>(p.part_acc + unit_row(s) * kD + d0);
      const float4 x0 = a[0], x1 = a[1];
      const float a2[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      merge_partial(m, l, acc, v.x, v.y, a2);
    }
  }
#pragma unroll
  for (int off = 1; off < SL; off <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    float a2[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) a2[j] = __shfl_xor_sync(0xffffffffu, acc[j], off);
    merge_partial(m, l, acc, m2, l2, a2);
  }
  if (sl != 0 || hh >= G) return;
  // the sink logit (log2 units) joins the max and, once, the denominator
  float den = l;
  if (p.sink) {
    const float sg = __ldg(p.sink + kvh * G + hh) * kLog2e;
    const float M = fmaxf(m, sg);
    const float w = (m == neg_inf()) ? 0.f : ex2(m - M);
    den = w * l + ex2(sg - M);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] *= w;
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint4 outv;
  outv.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  outv.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
  outv.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
  outv.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
  *reinterpret_cast<uint4*>(p.out + (size_t)(q_begin + t) * p.out_ts + (size_t)(kvh * G + hh) * p.out_hs + d0) = outv;
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, const DecodeMaps& maps, cudaStream_t s,
                          const cudaEvent_t* ev_before, const cudaEvent_t* ev_after) {
  dim3 g1(p.max_segs, p.hkv, p.num_reqs);
  auto run = [&](auto kern, int smem) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem + 4096 * 4);
    if (e != cudaSuccess) return e;
    if (ev_before && *ev_before) cudaEventRecord(*ev_before, s);
    // + the query fragments: 4 KB per query position
    kern<<<g1, kThreads, smem + 4096 * p.max_q_len, s>>>(maps.k, maps.v, p);
    return cudaGetLastError();
  };
  cudaError_t e;
  // the sink alone needs no change in the split kernel (it is the combine's)
  const bool feat = p.g_cache != nullptr || p.window > 0;
#define GCS_RUN3(KVF, PT, F, SQ, P1)                                                                 \
  (p.group == 8 ? run(decode_split_kernel<KVF, PT, F, 8, SQ, P1>, DecCfg<KVF, PT, F, SQ>::SMEM)       \
                : run(decode_split_kernel<KVF, PT, F, 16, SQ, P1>, DecCfg<KVF, PT, F, SQ>::SMEM))
#define GCS_RUN2(KVF, PT, F, SQ) \
  (p.log2_block_pages == 0 ? GCS_RUN3(KVF, PT, F, SQ, true) : GCS_RUN3(KVF, PT, F, SQ, false))
#define GCS_RUN(KVF, PT, F) (p.max_q_len > 2 ? GCS_RUN2(KVF, PT, F, true) : GCS_RUN2(KVF, PT, F, false))
  if (p.kv_format == 1)
    e = feat ? GCS_RUN(1, false, true) : GCS_RUN(1, false, false);
  else if (p.scale_mode == 1)
    e = feat ? GCS_RUN(0, true, true) : GCS_RUN(0, true, false);
  else
    e = feat ? GCS_RUN(0, false, true) : GCS_RUN(0, false, false);
#undef GCS_RUN
#undef GCS_RUN2
#undef GCS_RUN3
  if (ev_after && *ev_after) cudaEventRecord(*ev_after, s);
  if (e != cudaSuccess) return e;
  return launch_decode_combine(p, s);
}

cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t s) {
  if (p.max_segs >= 32) {
    dim3 g2(p.num_reqs * p.max_q_len, p.hkv, p.group / 2);
    decode_combine_kernel<8><<<g2, 256, 0, s>>>(p);
  } else {
    dim3 g2(p.num_reqs * p.max_q_len, p.hkv, (p.group + 3) / 4);
    decode_combine_kernel<4><<<g2, 256, 0, s>>>(p);
  }
  return cudaGetLastError();
}

// Device address of the static scratch on the current device.  The first call on a
// device looks the address up (cudaGetSymbolAddress, with that device current); later
// calls reuse it.
cudaError_t decode_noalloc_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace gcs
