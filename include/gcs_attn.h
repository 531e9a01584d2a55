/*
 * gcs_attn.h -- C ABI of the GB300 (sm_103a) gated causal softmax attention library.
 *
 * Four calls make up the hot path:
 *   attn_fwd           prefill forward  (O, LSE)
 *   attn_bwd           prefill backward (dQ, dK, dV, d log_gate, d sink)
 *   attn_decode_paged  paged single-query / short-query decode over an fp8 e4m3 KV cache
 *   attn_prefill_paged paged chunked prefill (query chunks of any length) over the same cache
 *
 * Sources for what each call computes (page title, section):
 *   [FLA] fla-org/flash-linear-attention issue #1322 "[Perf] Gluon attention backend with
 *         large head dimensions" -- Description: the causal attention contract (dense and
 *         packed variable-length inputs, MHA/GQA/MQA, unequal query/key and value head
 *         dims up to 512, logarithmic gates, sliding windows, sink bias, gradients);
 *         comment of Oct 3: the sink gradient is accumulated in fp32 from the backward
 *         probabilities, not from the rounded output; comment of Oct 5: dQ partials
 *         accumulate into a zero-initialised fp32 buffer and are converted afterwards.
 *   [AIT] ROCm/aiter PR #6660 (gfx1250 unified attention) -- commit messages and
 *         "Technical details": per-token fp32 K/V scales laid out [num_blocks,
 *         num_kv_heads, block_size]; K scales multiply QK columns; V scales multiply P
 *         columns after the row sum; slots past seq_len get scale 0; split-K over context
 *         segments with an LSE-weighted reduce in which an empty partial (M = -inf)
 *         weighs 0; per-token scales on a prefill shape are rejected.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller (inputs, outputs and
 *     workspace).  The library never allocates, frees or synchronises.
 *   - Every call is asynchronous on the given stream.  Arguments are validated on the
 *     host first; on any error the call returns a nonzero gcs_status and launches
 *     nothing, so outputs are untouched.
 *   - Tensors are row-major with the last dimension contiguous and base addresses 16-byte
 *     aligned.  The [tokens, heads, head_dim] tensors of the prefill and paged calls (q, k,
 *     v, o, dout, the gradients, the paged q and out) take element strides (token, head)
 *     given as gcs_strides, and the paged caches take element strides (block, kv head, slot);
 *     all-zero strides mean contiguous.  Everything else (gates, sinks, LSE, scales, index
 *     arrays) is contiguous.
 *   - No output may share a byte with an input or with another output (the kernels read
 *     and write concurrently); such a call returns GCS_ERR_INVALID_ARG.  Inputs may share
 *     memory with each other.
 *   - bf16 = bfloat16 stored as uint16; fp8 = OCP e4m3 ("fn") stored as uint8.
 *   - Device-side contents (cu_seqlens monotone and ending at total_tokens, page-table
 *     entries in [0, num_blocks), seq_lens >= q_len) are preconditions; they are not
 *     checked on the host because reading them would synchronise.  gcs_set_device_checks
 *     makes every call check them on the device first (see "device-content checks").
 *   - Every wait inside a kernel is bounded (2 s).  A kernel that gives up records
 *     GCS_ERR_DEVICE_TIMEOUT in a per-device status word, releases its resources and
 *     returns; read it with gcs_get_device_status().
 *   - The library caches, per device, the device addresses of its own status word and of
 *     the scratch of attn_decode_paged_noalloc.  cudaDeviceReset unloads the library's
 *     device code and those addresses go stale: do not call the library on a device after
 *     cudaDeviceReset of that device in the same process.
 */
#ifndef GCS_ATTN_H_
#define GCS_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gcs_stream_t; /* same type as cudaStream_t; NULL = legacy default stream */

/* Element strides of a [tokens, heads, head_dim] tensor whose head_dim is contiguous: element
 * (t, h, d) sits at base[t * token + h * head + d].  {0, 0} means the contiguous layout
 * {heads * head_dim, head_dim}.  Otherwise the layout must be token-major without overlap,
 * head >= head_dim and token >= heads * head, with both multiples of 8 elements (16 bytes, the
 * granule of the tensor copies and vector stores); any other layout returns
 * GCS_ERR_UNSUPPORTED.  A slice of a fused projection, e.g. q, k and v as views of one
 * [tokens, (hq + 2 hkv) * d] buffer, is such a layout. */
typedef struct {
  int64_t token;
  int64_t head;
} gcs_strides;

typedef enum {
  GCS_OK = 0,
  GCS_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned base, inconsistent shape */
  GCS_ERR_UNSUPPORTED = 2,   /* a shape / dtype / layout this library does not implement   */
  GCS_ERR_WORKSPACE = 3,     /* workspace pointer NULL or smaller than the *_workspace size */
  GCS_ERR_CUDA = 4,          /* a CUDA launch or runtime call failed                       */
  GCS_ERR_DEVICE_TIMEOUT = 5 /* a kernel gave up on a bounded wait (device status word)    */
} gcs_status;

const char* gcs_status_str(int status);

/* ------------------------------------------------------------------ prefill
 * Causal softmax attention over packed sequences ([FLA] Description).
 * Sequence s occupies tokens cu_seqlens[s] .. cu_seqlens[s+1]-1 of the packed tensors;
 * dense [B, T] inputs are the special case cu_seqlens = {0, T, 2T, ..., B*T}.
 * Query head h reads kv head h / (hq / hkv) (MHA: hq == hkv; MQA: hkv == 1).
 * Score of query token i and key token j of the same sequence:
 *     s_ij = scale * (q_i . k_j) + G_i - G_j,   G = per-sequence inclusive cumsum of log_gate
 * visible iff j <= i and (window == 0 or i - j < window).  The per-head sink logit sigma_h
 * joins the softmax denominator only:  P_ij = e^{s_ij} / (sum_j e^{s_ij} + e^{sigma_h}).
 * Supported (dqk, dv): (64, 64), (128, 128), (256, 256), (256, 512), (512, 512).
 */
typedef struct {
  int num_seqs;               /* >= 1                                                    */
  const int32_t* cu_seqlens;  /* device int32 [num_seqs + 1]                            */
  int total_tokens;           /* host copy of cu_seqlens[num_seqs]; >= 1                */
  int max_seqlen;             /* host upper bound on any sequence length                */
  int hq, hkv;                /* query heads, kv heads; hq % hkv == 0                    */
  int dqk, dv;                /* head dims of q/k and of v                               */
  float scale;                /* softmax scale (usually 1/sqrt(dqk))                     */
  int window;                 /* 0 = none, else number of visible keys including self    */
  const void* q;              /* bf16 [total_tokens, hq, dqk]                            */
  const void* k;              /* bf16 [total_tokens, hkv, dqk]                           */
  const void* v;              /* bf16 [total_tokens, hkv, dv]                            */
  const float* log_gate;      /* fp32 [total_tokens, hq] per-token log forget gates, or NULL */
  const float* sink;          /* fp32 [hq] sink logits, or NULL                          */
  int deterministic;          /* attn_bwd: 1 = a separate query-stationary dQ pass, every
                                 gradient written once or summed in a fixed order; 0 = the
                                 faster route for the shape: a single pass with fp32
                                 reduce-adds of dQ and the dS row sums at head dim 128 and at
                                 dqk = 256, the separate dQ pass at 64 (the only route there)
                                 and at dqk = 512. */
  gcs_strides q_stride, k_stride, v_stride;  /* layouts of q, k, v ({0, 0} = contiguous)      */
  gcs_strides o_stride;       /* attn_fwd's output o and attn_bwd's input o                    */
  gcs_strides do_stride;      /* attn_bwd's dout                                               */
  gcs_strides dq_stride, dk_stride, dv_stride;  /* attn_bwd's outputs dq, dk, dv              */
} gcs_prefill_args;

/* Workspace bytes attn_fwd needs (0 when there is no gate). */
size_t attn_fwd_workspace(const gcs_prefill_args* a);

/* Forward.  o: bf16 [total_tokens, hq, dv] (layout a->o_stride); lse: fp32 [hq, total_tokens]
 * contiguous, natural-log logsumexp of each row's scores including the sink term (needed by
 * attn_bwd).  Outputs that share bytes with an input or with each other are rejected; two
 * strided tensors with the same token stride whose per-token byte ranges interleave without
 * meeting (e.g. heads of one fused buffer) do not share bytes. */
int attn_fwd(const gcs_prefill_args* a, void* o, float* lse, void* workspace, size_t workspace_bytes,
             gcs_stream_t stream);

/* Workspace bytes attn_bwd needs. */
size_t attn_bwd_workspace(const gcs_prefill_args* a);

/* Backward of L = sum(O * dO) ([FLA] Description, the gradient list; Oct 3 / Oct 5 comments).
 * o, lse: the forward's outputs (o in layout a->o_stride); dout: bf16 [total_tokens, hq, dv]
 * (a->do_stride).  Outputs: dq bf16 [total_tokens, hq, dqk] (a->dq_stride), dk bf16
 * [total_tokens, hkv, dqk] (a->dk_stride), dv bf16 [total_tokens, hkv, dv] (a->dv_stride),
 * dlog_gate fp32 [total_tokens, hq] contiguous (must be NULL iff
 * log_gate is NULL), dsink fp32 [hq] (must be NULL iff sink is NULL).
 * The sink gradient is -sum_i p_sink,i * sum_j P_ij (dO_i . v_j), accumulated in fp32.
 * With a->deterministic = 1 (and always at head dim 64, and at dqk = 512) dQ is accumulated per
 * query tile in a separate pass and every gradient is written once or summed in a fixed order,
 * so repeated calls give the same bits.  Otherwise (head dim 128, dqk = 256) dQ, d log_gate and
 * d sink come from fp32 reduce-adds into zero-initialised buffers (the [FLA] comment of Oct 5),
 * and their low bits may vary from run to run. */
int attn_bwd(const gcs_prefill_args* a, const void* o, const float* lse, const void* dout, void* dq, void* dk,
             void* dv, float* dlog_gate, float* dsink, void* workspace, size_t workspace_bytes,
             gcs_stream_t stream);

/* ------------------------------------------------------------------ paged decode
 * Decode / short-query attention over a paged KV cache ([AIT] commits 1-3, Technical
 * details): fp8 e4m3 with per-token fp32 scales (the default), fp8 e4m3 with one K and one
 * V scale for the whole cache (per-tensor, which the page leaves on its earlier code path),
 * or bf16 with no scales (the bf16-KV route of commit 3).  Request r has
 * q_len = cu_q[r+1] - cu_q[r] query rows (1..4) and seq_len = seq_lens[r] cached tokens (the
 * query tokens are the last q_len of them); query row t sits at position seq_len - q_len + t
 * and sees keys 0 .. seq_len - q_len + t.  Key j of request r lives in block
 * block_table[r][j / block_size],
 * slot j % block_size.  Dequantised key = e4m3(k) * k_scale[block][kv_head][slot], same for
 * values.  s_j = scale * k_scale_j * (q . k8_j); the row sum uses the unscaled e^{s_j - m};
 * the V scales multiply the probabilities after the row sum.  Slots at or past seq_len are
 * never used (scale 0, probability 0), whatever their bytes or scales hold (NaN allowed).
 * The context is split into segments of segment_len tokens; each (request, kv head,
 * segment) yields a partial (acc, M, L) and a combine kernel merges them with weights
 * e^{M_s - max M}; a partial with no visible key (M = -inf) weighs 0.
 * With per-tensor scales, k_scale and v_scale each point to one fp32 used for every token;
 * with a bf16 cache, k_cache / v_cache hold bf16 values and k_scale, v_scale must be NULL.
 * Decoding features (the [FLA] Description asks for the prefill features on the packed
 * single-query decode too), each optional: g_cache holds the cumulative log gates G of the
 * cached tokens, paged like the scales but per query head, fp32 [num_blocks, hq, block_size]
 * (natural-log units); the score becomes scale*q.k_j + G_i - G_j with G_i the entry at the query row's
 * own position.  window W > 0 keeps keys with position_i - j < W.  sink fp32 [hq] adds
 * e^sink_h to the softmax denominator (once, in the combine).
 * Supported: d == 128; hq / hkv == 16 or 8 (GQA groups of 16 or 8 query heads); block_size
 * 16 x 2^k tokens (16, 32, 64, 128, ..., 4096); 1 <= q_len <= 4; segment_len a positive multiple
 * of 16.
 * Operand precision of an fp8 cache: the tensor cores see f16.  q is rounded from bf16 to f16,
 * so no |q| may exceed 65504 (the f16 maximum); K and V codes convert to f16 exactly;
 * P * vscale is rounded to nearest f16 after a 2^5 pre-scale (P <= 2^3: a row's reference max
 * moves only when the row max grows by more than 2^3), so every V scale of a slot below
 * seq_len must stay below 255.  Outside these limits the output holds inf or NaN.
 * The host cannot read device values; checked mode (gcs_set_device_checks) checks both on the
 * device and records GCS_ERR_INVALID_ARG when one fails.
 */
enum { GCS_KV_FP8_E4M3 = 0, GCS_KV_BF16 = 1 };
enum { GCS_SCALE_PER_TOKEN = 0, GCS_SCALE_PER_TENSOR = 1 };
typedef struct {
  int num_reqs;                /* >= 1                                                   */
  const int32_t* cu_q;         /* device int32 [num_reqs + 1]                           */
  int total_q;                 /* host copy of cu_q[num_reqs]                           */
  int max_q_len;               /* host upper bound on q_len, 1..4                        */
  const int32_t* seq_lens;     /* device int32 [num_reqs], each >= its q_len             */
  int max_seq_len;             /* host upper bound on seq_lens                           */
  const int32_t* block_table;  /* device int32 [num_reqs, max_blocks_per_req]           */
  int max_blocks_per_req;      /* row stride of block_table                             */
  const void* k_cache;         /* fp8 e4m3 or bf16 [num_blocks, hkv, block_size, d]     */
  const void* v_cache;         /* same format as k_cache                                 */
  const float* k_scale;        /* fp32 [num_blocks, hkv, block_size], or [1], or NULL   */
  const float* v_scale;        /* same layout as k_scale                                 */
  int num_blocks, block_size;  /* cache blocks, tokens per block                        */
  int hq, hkv, d;              /* query heads, kv heads, head dim                       */
  float scale;                 /* softmax scale                                         */
  int segment_len;             /* split-K segment length in tokens                      */
  const void* q;               /* bf16 [total_q, hq, d]                                 */
  int kv_format;               /* GCS_KV_FP8_E4M3 or GCS_KV_BF16                         */
  int scale_mode;              /* GCS_SCALE_PER_TOKEN or GCS_SCALE_PER_TENSOR (fp8 only) */
  const float* g_cache;        /* fp32 [num_blocks, hq, block_size] cumulative log gates, or NULL */
  const float* sink;           /* fp32 [hq] sink logits, or NULL                          */
  int window;                  /* sliding window in keys, 0 = none                        */
  gcs_strides q_stride;        /* layout of q ({0, 0} = contiguous)                       */
  gcs_strides out_stride;      /* layout of out ({0, 0} = contiguous)                     */
  int64_t kv_stride_block, kv_stride_head, kv_stride_slot;
                               /* element strides of both caches (block, kv head, slot); all 0 =
                                  contiguous [num_blocks, hkv, block_size, d].  The d elements of
                                  a slot are contiguous; every stride is a multiple of 16 bytes;
                                  the slots and kv heads of a block nest without overlap (slot
                                  >= d and head >= block_size * slot, or head >= d and slot >=
                                  hkv * head: the [num_blocks, block_size, hkv, d] cache layout of
                                  vLLM-style engines) and block covers both.  Scales and gates
                                  stay contiguous [num_blocks, ..., block_size]. */
} gcs_decode_args;

/* Workspace bytes attn_decode_paged needs (split-K partials). */
size_t attn_decode_workspace(const gcs_decode_args* a);

/* out: bf16 [total_q, hq, d]. */
int attn_decode_paged(const gcs_decode_args* a, void* out, void* workspace, size_t workspace_bytes,
                      gcs_stream_t stream);

/* Allocation-free variant of attn_decode_paged (no counterpart in the pages: this is a
 * library convenience).  Some callers cannot allocate device memory for a workspace: a
 * host runtime with a fixed, pre-planned memory budget, a C program without a device
 * allocator of its own, or a latency-critical decode loop in which a cudaMalloc (which
 * may synchronise the device) is not acceptable.  This entry point takes the same
 * arguments minus the workspace and keeps the split-K partials in a fixed scratch array
 * compiled into the library (64 MiB, held on every GPU that loads the library until the
 * process exits).  It calls no allocator.
 *   - Sizes whose partials exceed the scratch (attn_decode_workspace(a) > 64 MiB) are
 *     rejected with GCS_ERR_WORKSPACE before anything is launched.
 *   - The first call on a device looks up the scratch's device address (with that device
 *     current); make that first call before any stream capture on that device.
 *   - All calls share the one scratch array and it keeps the previous call's contents;
 *     nothing needs clearing because every partial a call reads it first writes.  Calls
 *     that overlap on the GPU (e.g. on two concurrent streams) race on the scratch and
 *     give wrong results: serialise them.
 * out: bf16 [total_q, hq, d]; returns the same statuses as attn_decode_paged. */
int attn_decode_paged_noalloc(const gcs_decode_args* a, void* out, gcs_stream_t stream);

/* ------------------------------------------------------------------ paged chunked prefill
 * Attention of query chunks of any length over the same paged fp8 KV cache ([AIT] commit
 * messages: a batch that is not all-decode takes the 2d unified-attention route, one
 * program per (kv head, query block)).  Arguments and semantics are those of
 * attn_decode_paged (gcs_decode_args, the decoding features included), except:
 *   - q_len = cu_q[r+1] - cu_q[r] may be any value in 1 .. seq_lens[r]; max_q_len >= 1 is
 *     its host upper bound.  Query row t of request r still sits at position
 *     seq_len - q_len + t and sees keys 0 .. seq_len - q_len + t (and the window).
 *   - fp8 e4m3 with per-token or per-tensor scales; a bf16 cache is GCS_ERR_UNSUPPORTED.
 *     (The pages' 2d route rejects per-token scales; here they are applied as in decode.)
 *   - segment_len == 0 lets the library split the context: one segment per request when
 *     the query blocks alone give about two CTAs per SM (the kernel then writes out
 *     directly and needs no workspace), otherwise segments sized for that many CTAs whose
 *     split-K partials the decode combine merges.  A positive segment_len must be a
 *     multiple of 128 tokens.  attn_prefill_paged_workspace(a) gives the bytes needed
 *     (0 when nothing is split; the choice depends on the current device's SM count).
 *   - The tensor cores see Q rounded from bf16 to f16 (|q| < 65504), K and V as exact f16
 *     from e4m3, and P * vscale rounded to f16 (vscale < 255), with fp32 accumulation.
 * out: bf16 [total_q, hq, d].  Preconditions: q_len <= seq_len per request. */
size_t attn_prefill_paged_workspace(const gcs_decode_args* a);
int attn_prefill_paged(const gcs_decode_args* a, void* out, void* workspace, size_t workspace_bytes,
                       gcs_stream_t stream);

/* ------------------------------------------------------------------ status
 * Per-device status word written by kernels that gave up on a bounded wait.
 * Copies the word for the current device into *status (synchronous) and, if clear != 0,
 * resets it to GCS_OK.  Returns GCS_OK or GCS_ERR_CUDA. */
int gcs_get_device_status(int* status, int clear);

/* Self-test of the bounded waits (a library diagnostic with no counterpart in the pages).
 * Launches one small kernel on the stream that waits, through the same bounded wait every
 * kernel uses, on a barrier phase that nothing completes.  After the 2 s wait limit it
 * records GCS_ERR_DEVICE_TIMEOUT in the current device's status word and exits; the context
 * stays usable.  Read (and clear) the word with gcs_get_device_status.
 * Returns GCS_OK once the kernel is launched, or GCS_ERR_CUDA. */
int gcs_selftest_bounded_wait(gcs_stream_t stream);

/* ------------------------------------------------------------------ device-content checks
 * A library diagnostic with no counterpart in the pages.  The preconditions checked:
 *   prefill: cu_seqlens[0] == 0, cu_seqlens[num_seqs] == total_tokens, and every length
 *            cu_seqlens[s+1] - cu_seqlens[s] in 0 .. max_seqlen;
 *   paged:   cu_q[0] == 0, cu_q[num_reqs] == total_q; for every request
 *            0 <= q_len <= max_q_len and q_len <= seq_len <= max_seq_len; and, for a request
 *            with q_len >= 1, every block_table entry in [0, num_blocks) from the 128-key tile
 *            that holds the earliest key one of its query rows sees (key 0 without a window)
 *            up to the page of its last cached token (the pages the paged calls can read);
 *            with an fp8 cache, the f16 operand limits: every |q| <= 65504 and every V scale
 *            of those pages' slots below seq_len (or the per-tensor V scale) < 255.
 * A failed check records GCS_ERR_INVALID_ARG in the current device's status word (first
 * writer wins, like a timeout); read it with gcs_get_device_status.
 *
 * gcs_set_device_checks(1) turns on checked mode for every later call of this process (0
 * turns it off; other values return GCS_ERR_INVALID_ARG).  In checked mode each attn_* call
 * first launches one single-CTA kernel on its stream that checks its arrays and writes a copy
 * of cu_seqlens (or cu_q) to the end of the call's workspace; the call's kernels read that
 * copy.  When a check fails the copy is all zeros, an empty batch: no kernel then reads
 * through an index taken from these arrays, so a broken array cannot send a kernel outside a
 * buffer.
 * The outputs of such a call are unspecified.  The copy takes ((num_seqs or num_reqs) + 1)
 * x 4 bytes, rounded up to 256, more workspace: the *_workspace queries include it while
 * checked mode is on (query them after switching the mode), so attn_fwd and
 * attn_prefill_paged then need a workspace even where they otherwise take none;
 * attn_decode_paged_noalloc keeps it in its scratch.  gcs_get_device_checks returns the mode.
 *
 * gcs_check_prefill_inputs / gcs_check_paged_inputs run the same checks on their own (no
 * copy, nothing else launched) on the stream, after the host validation of attn_fwd (or
 * attn_bwd) and of attn_decode_paged or attn_prefill_paged, whose errors they return.
 * Return GCS_OK once the kernel is launched, or the host validation's error, or
 * GCS_ERR_CUDA. */
int gcs_set_device_checks(int enable);
int gcs_get_device_checks(void);
int gcs_check_prefill_inputs(const gcs_prefill_args* a, gcs_stream_t stream);
int gcs_check_paged_inputs(const gcs_decode_args* a, gcs_stream_t stream);

/* ------------------------------------------------------------------ instrumentation
 * Arms two caller-created CUDA events (cudaEvent_t, passed as void*) for the next attn_fwd,
 * attn_bwd, attn_decode_paged or attn_prefill_paged call made by this host thread: `before`
 * is recorded on the call's stream immediately before its main attention kernels (the
 * prefill forward kernel; the backward's attention kernels -- dQ pass + dK/dV pass, or the
 * wide-head role kernels; the split-K decode kernel; the paged prefill kernel) and `after`
 * immediately after them, so
 * cudaEventElapsedTime(before, after) is their device time.  The events are
 * disarmed once used; passing NULL, NULL disarms them.  Returns GCS_OK. */
int gcs_set_kernel_events(void* before, void* after);

/* Library version string. */
const char* gcs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GCS_ATTN_H_ */
