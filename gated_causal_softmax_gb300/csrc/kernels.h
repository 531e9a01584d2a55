// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace gcs {

// Per-device status word (GCS_OK / GCS_ERR_DEVICE_TIMEOUT), written by kernels.
int* device_status_ptr();

struct FwdParams {
  const int32_t* cu_seqlens;
  int num_seqs;
  int total;
  int hq, hkv, dqk, dv;
  int dv_chunk;          // value columns handled by one CTA
  float scale_log2;      // scale * log2(e)
  int window;            // 0 = none
  const float* gT;       // G^T [hq, total] in log2 units (gate cumsum * log2 e), or null
  const float* sink;     // [hq] natural-log sink logits, or null
  uint16_t* o;           // bf16 [total, hq, dv] at token * o_ts + head * o_hs
  long long o_ts, o_hs;  // element strides of o
  float* lse;            // [hq, total]
  int* status;
};

struct FwdMaps {
  CUtensorMap q, k, v;  // 3-D bf16 maps {dim, heads, tokens}, box 64 x 1 x 128, 128-B swizzle
};

cudaError_t launch_prefill_fwd(const FwdParams& p, const FwdMaps& maps, int num_tiles, cudaStream_t s);
// Head dims 64 / 128: two 128-row query tiles per CTA (two query heads of a GQA group over the
// same rows when the group size is even, else 256 rows of one head).
cudaError_t launch_prefill_fwd2(const FwdParams& p, const FwdMaps& maps, cudaStream_t s);

struct BwdParams {
  const int32_t* cu_seqlens;
  int num_seqs;
  int total;
  int hq, hkv, dqk, dv;
  float scale;           // softmax scale
  float scale_log2;      // scale * log2(e)
  int window;
  const float* gT;       // G^T [hq, total] (log2 units) or null
  const float* lse;      // [hq, total] natural log
  const float* delta;    // [hq, total] rowsum(dO * O)
  uint16_t* grad_q;      // bf16 [total, hq, dqk] (written directly by the dQ pass)
  uint16_t* grad_k;      // bf16 [total, hkv, dqk]
  uint16_t* grad_v;      // bf16 [total, hkv, dv]
  long long dq_ts, dq_hs, dk_ts, dk_hs, dv_ts, dv_hs;  // element strides (token, head) of the three
  float* dq_acc;         // fp32 [total, hq, dqk] (zeroed; single pass and wide reduce-add route)
  float* dg_row;         // fp32 [hq, total] sum_j dS_ij; null if not needed
  float* dg_col;         // fp32 [hq, total] sum_i dS_ij (zeroed); null if no gate
  const float* vecp;     // packed per-(head, 64-row query tile) vectors (see launch_bwd_pack)
  int n_qtiles;          // query tiles per head in vecp
  int* status;
};

struct BwdMaps {
  CUtensorMap q, k, v, dout;   // 3-D bf16 maps {dim, heads, tokens}, 128-B swizzle (q, dout: 64-row boxes)
  CUtensorMap q128, dout128;   // q, dout with 128-row boxes (dQ pass)
  CUtensorMap dq_acc;          // fp32 dQ accumulator {dqk, heads, tokens}, box 32 x 1 x 128, 128-B swizzle
                               // (single-pass route only)
};

cudaError_t launch_prefill_bwd(const BwdParams& p, const BwdMaps& maps, int num_kv_tiles, cudaStream_t s);
// Single-pass backward at head dim 128: dK, dV written, dQ and the dS row sums reduce-added
// into the zeroed fp32 buffers p.dq_acc and p.dg_row (q / dout maps with 128-row boxes).
cudaError_t launch_prefill_bwd_fused(const BwdParams& p, const BwdMaps& maps, int num_kv_tiles, cudaStream_t s);
// dQ pass of the two-pass backward (head dims <= 128): writes dQ (bf16) and dS row sums.
cudaError_t launch_prefill_bwd_dq(const BwdParams& p, const BwdMaps& maps, int num_q_tiles, cudaStream_t s);
// Head dims above 128, key-stationary output-column roles: dV chunks, and dK chunks that
// also reduce-add dQ and the dS row sums into fp32 buffers (with_dq) or leave them to the
// query-stationary dQ pass (deterministic route; it writes dQ in bf16 and the row sums).
cudaError_t launch_prefill_bwd_wide_dq(const BwdParams& p, const BwdMaps& maps, int num_q_tiles, cudaStream_t s);
cudaError_t launch_prefill_bwd_wide(const BwdParams& p, const BwdMaps& maps, int num_kv_tiles, bool with_dq,
                                    cudaStream_t s);

// Small HBM-bound helpers.
cudaError_t launch_gate_cumsum(const float* g, const int32_t* cu, int num_seqs, int total, int hq, float* gT,
                               cudaStream_t s);
// Before the backward attention kernels, one launch: G (when gT is set; the gate cumsum of
// the log gates g) beside delta_i = dO_i . O_i and the zeroing of the fp32 dQ accumulator and
// the dS row / column sums (each where set).  n_scan is set by the launcher.
struct PreArgs {
  const uint16_t* o;
  const uint16_t* dout;
  int total, hq, dv, dqk;
  long long o_ts, o_hs, do_ts, do_hs;  // element strides (token, head)
  float* delta;                        // [hq, total]
  float* dq_acc;                       // [total, hq, dqk] or null
  float* dg_row;                       // [hq, total] or null
  float* dg_col;                       // [hq, total] or null
  const float* g;                      // log gates [total, hq] (with gT)
  const int32_t* cu;
  int num_seqs;
  float* gT;                           // [hq, total] or null
  int n_scan;
};
cudaError_t launch_bwd_pre(const PreArgs& a, cudaStream_t s);
// Packs (G_i - LSE_i) * log2 e and delta_i per (head, 64-row query tile): vecp
// [hq][n_qtiles][128] with n_qtiles = ceil(total / 64) + num_seqs.
cudaError_t launch_bwd_pack(const int32_t* cu, int num_seqs, int total, int hq, int n_qtiles, const float* lse,
                            const float* gT, const float* delta, float* vecp, cudaStream_t s);
// After the backward attention kernels, one launch: the dQ conversion (when dq_acc is set),
// d log_gate (when dlog_gate is set) and d sink (when dsink is set).  n4, n_gate and n_sink are
// set by the launcher.
struct PostArgs {
  const float* dq_acc;  // [total, hq, dqk] fp32 or null
  uint16_t* dq;
  int total, hq, dqk;
  long long dq_ts, dq_hs;
  const int32_t* cu;
  int num_seqs;
  const float* dg_row;  // [hq, total]
  const float* dg_col;  // [hq, total]
  float* dlog_gate;     // [total, hq] or null
  const float* lse;     // [hq, total]
  const float* delta;   // [hq, total]
  const float* sink;    // [hq]
  float* dsink;         // [hq] or null
  size_t n4;
  int n_gate, n_sink;
};
cudaError_t launch_bwd_post(const PostArgs& a, cudaStream_t s);

struct DecodeParams {
  const int32_t* cu_q;
  const int32_t* seq_lens;
  const int32_t* block_table;
  int max_blocks;
  const uint8_t* k_cache;  // fp8 e4m3 codes or bf16 values (kv_format)
  const uint8_t* v_cache;
  const float* k_scale;    // per token [num_blocks, hkv, 16], per tensor [1], or null (bf16)
  const float* v_scale;
  int kv_format;           // 0: fp8 e4m3, 1: bf16
  int scale_mode;          // 0: per token, 1: per tensor
  const float* g_cache;    // cumulative log gates [num_blocks, hq, 16] (natural log), or null
  const float* sink;       // [hq] sink logits, or null
  int window;              // 0 = none
  int num_reqs, hq, hkv;
  int max_q_len;
  int max_segs;          // segments per request slot in the partial buffers
  int seg_pages;         // pages per segment
  float scale;
  const uint16_t* q;     // bf16 [total_q, hq, 128] at token * q_ts + head * q_hs
  uint16_t* out;         // bf16 [total_q, hq, 128] at token * out_ts + head * out_hs
  long long q_ts, q_hs, out_ts, out_hs;  // element strides
  long long kv_bs, kv_hs, kv_ss;         // byte strides (block, kv head, slot) of both caches
  int kv_head_inner;     // 1: the kv head stride is below the slot stride (fp8 maps order dims so)
  int block_size;        // tokens per cache block: 16-token pages times a power of two
  int log2_block_pages;  // log2(block_size / 16)
  int group;             // query heads per kv head: 16 or 8
  float* part_acc;       // [units, 4*16, 128]
  float* part_ml;        // [units, 4*16, 2]
  int* status;
};

// fp8 K and V caches as 4-D maps {128 B, slot, kv head, block} (slot and kv head swapped when
// kv_head_inner), box one page of 16 slots x 128 B, 128-byte swizzle; unused for a bf16 cache.
struct DecodeMaps {
  CUtensorMap k, v;
};

// ev_before / ev_after (may point to null events) are recorded around the split-K kernel.
cudaError_t launch_decode(const DecodeParams& p, const DecodeMaps& maps, cudaStream_t s,
                          const cudaEvent_t* ev_before, const cudaEvent_t* ev_after);

// LSE-weighted merge of the split-K partials of every (query row, query head) into p.out.
cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t s);

// Paged chunked prefill (any q_len) over an fp8 cache.  p.part_acc == nullptr: one segment
// per request, the kernel writes p.out; otherwise split-K partials and the combine.
cudaError_t launch_prefill_paged(const DecodeParams& p, const DecodeMaps& maps, cudaStream_t s,
                                 const cudaEvent_t* ev_before, const cudaEvent_t* ev_after);

// One CTA that waits on a barrier phase nothing completes; its bounded wait records a
// timeout in *status and the kernel exits.
cudaError_t launch_bounded_wait_selftest(int* status, cudaStream_t s);

// Device-content checks (one CTA, before the call's kernels): record kDevInvalidArg in *status
// when a precondition on the index arrays fails, and write to cu_out (if not null) a copy of
// cu_seqlens / cu_q, or all zeros (an empty batch) on a failure.
cudaError_t launch_check_prefill(const int32_t* cu, int num_seqs, int total, int max_seqlen, int32_t* cu_out,
                                 int* status, cudaStream_t s);
// The f16 operand limits of an fp8 cache (hkv = 0: nothing to check, a bf16 cache).
struct PagedOperandCheck {
  const uint16_t* q;      // bf16 [total_q, hq, d] at token * q_ts + head * q_hs
  long long q_ts, q_hs;
  int hq, d, hkv;
  const float* v_scale;   // per token [num_blocks, hkv, block_size] or per tensor [1]
  int per_tensor;
};
cudaError_t launch_check_paged(const int32_t* cu_q, const int32_t* seq_lens, const int32_t* table, int num_reqs,
                               int total_q, int max_q_len, int max_seq_len, int max_blocks, int num_blocks,
                               int block_size, int window, const PagedOperandCheck& fp8, int32_t* cu_out,
                               int* status, cudaStream_t s);

// Size of the static scratch behind attn_decode_paged_noalloc (64 MiB).
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

// Device address of that scratch on the current device (set up on first use per device).
cudaError_t decode_noalloc_scratch(void** ptr);

}  // namespace gcs
