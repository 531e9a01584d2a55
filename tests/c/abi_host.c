/* Host-only checks of the C ABI from plain C99: a C program sees every call through
 * include/gcs_attn.h alone, invalid arguments return their documented status before any
 * CUDA call, and the workspace queries return the sizes the header documents.  No device
 * memory is addressed and nothing is launched: every call below is refused on the host or
 * is a size query. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "gcs_attn.h"

#define FAKE ((const void*)(uintptr_t)0x10000)          /* aligned, never dereferenced */
#define OUT ((void*)(uintptr_t)((uint64_t)1 << 36))      /* fake outputs far from FAKE */
#define OUT2 ((void*)(uintptr_t)(((uint64_t)1 << 36) + ((uint64_t)1 << 30)))

static int failures = 0;
#define EXPECT(cond)                                                    \
  do {                                                                  \
    if (!(cond)) {                                                      \
      fprintf(stderr, "%s:%d: failed: %s\n", __FILE__, __LINE__, #cond); \
      ++failures;                                                       \
    }                                                                   \
  } while (0)

static gcs_prefill_args prefill(void) {
  gcs_prefill_args a;
  memset(&a, 0, sizeof a);
  a.num_seqs = 1;
  a.cu_seqlens = (const int32_t*)FAKE;
  a.total_tokens = 256;
  a.max_seqlen = 256;
  a.hq = 4;
  a.hkv = 2;
  a.dqk = 128;
  a.dv = 128;
  a.scale = 0.088f;
  a.q = FAKE;
  a.k = FAKE;
  a.v = FAKE;
  return a;
}

static gcs_decode_args decode(void) {
  gcs_decode_args a;
  memset(&a, 0, sizeof a);
  a.num_reqs = 2;
  a.cu_q = (const int32_t*)FAKE;
  a.total_q = 2;
  a.max_q_len = 1;
  a.seq_lens = (const int32_t*)FAKE;
  a.max_seq_len = 4096;
  a.block_table = (const int32_t*)FAKE;
  a.max_blocks_per_req = 256;
  a.k_cache = FAKE;
  a.v_cache = FAKE;
  a.k_scale = (const float*)FAKE;
  a.v_scale = (const float*)FAKE;
  a.num_blocks = 600;
  a.block_size = 16;
  a.hq = 64;
  a.hkv = 4;
  a.d = 128;
  a.scale = 0.088f;
  a.segment_len = 2048;
  a.q = FAKE;
  a.kv_format = GCS_KV_FP8_E4M3;
  a.scale_mode = GCS_SCALE_PER_TOKEN;
  return a;
}

int main(void) {
  gcs_prefill_args a = prefill(), b;
  gcs_decode_args d = decode(), e;

  EXPECT(strncmp(gcs_version(), "gcs_attn", 8) == 0);
  EXPECT(strcmp(gcs_status_str(GCS_ERR_WORKSPACE), "workspace missing or too small") == 0);

  /* prefill: workspace sizes, then refusals before any launch */
  EXPECT(attn_fwd_workspace(&a) == 0);
  a.log_gate = (const float*)FAKE;
  EXPECT(attn_fwd_workspace(&a) == 4u * 4u * 256u); /* G^T [hq, tot] fp32 */
  EXPECT(attn_bwd_workspace(&a) > attn_fwd_workspace(&a));
  b = a;
  b.hq = 3;
  EXPECT(attn_fwd(&b, OUT, OUT2, NULL, 0, NULL) == GCS_ERR_INVALID_ARG);
  EXPECT(attn_fwd_workspace(&b) == 0);
  b = a;
  b.dqk = 96;
  b.dv = 96;
  EXPECT(attn_fwd(&b, OUT, OUT2, NULL, 0, NULL) == GCS_ERR_UNSUPPORTED);
  b = a;
  b.window = -1;
  EXPECT(attn_fwd(&b, OUT, OUT2, NULL, 0, NULL) == GCS_ERR_INVALID_ARG);
  EXPECT(attn_fwd(&a, OUT, OUT2, NULL, 0, NULL) == GCS_ERR_WORKSPACE); /* gated: needs G^T */
  EXPECT(attn_fwd(&a, (void*)FAKE, OUT2, NULL, 0, NULL) == GCS_ERR_INVALID_ARG); /* o on q */
  EXPECT(attn_bwd(&a, OUT, (const float*)OUT2, FAKE, OUT, OUT2, OUT, NULL, NULL, NULL, 0, NULL) ==
         GCS_ERR_INVALID_ARG); /* gated backward without dlog_gate */

  /* strides: a q slice of a fused [tokens, (hq + 2 hkv) * d] projection is accepted; heads
   * that overlap, a token stride below the heads' span, or a stride off the 16-byte granule
   * are refused before any launch */
  b = a;
  b.q_stride.token = (4 + 2 * 2) * 128;
  b.q_stride.head = 128;
  EXPECT(attn_fwd(&b, OUT, OUT2, NULL, 0, NULL) == GCS_ERR_WORKSPACE);
  b.q_stride.head = 100;
  EXPECT(attn_fwd(&b, OUT, OUT2, NULL, 0, NULL) == GCS_ERR_UNSUPPORTED);
  b.q_stride.head = 128;
  b.q_stride.token = 3 * 128;
  EXPECT(attn_fwd(&b, OUT, OUT2, NULL, 0, NULL) == GCS_ERR_UNSUPPORTED);
  b.q_stride.token = 4 * 128 + 4;
  EXPECT(attn_fwd(&b, OUT, OUT2, NULL, 0, NULL) == GCS_ERR_UNSUPPORTED);
  b = a;
  b.o_stride.token = -8;
  EXPECT(attn_fwd(&b, OUT, OUT2, NULL, 0, NULL) == GCS_ERR_INVALID_ARG);
  b = a;
  b.dk_stride.head = 64; /* the output store needs head >= dqk */
  b.dk_stride.token = 256;
  EXPECT(attn_bwd_workspace(&b) == 0);

  /* decode: split-K partials of 2 requests x 2 segments x 4 kv heads x 16 rows */
  {
    const size_t units = 2 * 2 * 4, rows = 16;
    EXPECT(attn_decode_workspace(&d) == units * rows * 128 * 4 + units * rows * 2 * 4);
  }
  e = d;
  e.max_q_len = 5; /* per-token scales on a prefill shape */
  EXPECT(attn_decode_paged(&e, OUT, NULL, 0, NULL) == GCS_ERR_UNSUPPORTED);
  EXPECT(attn_decode_workspace(&e) == 0);
  e = d;
  e.kv_format = GCS_KV_BF16; /* a bf16 cache takes no scales */
  EXPECT(attn_decode_paged(&e, OUT, NULL, 0, NULL) == GCS_ERR_INVALID_ARG);
  e.k_scale = NULL;
  e.v_scale = NULL;
  EXPECT(attn_decode_workspace(&e) == attn_decode_workspace(&d));
  EXPECT(attn_decode_paged(&d, OUT, NULL, 0, NULL) == GCS_ERR_WORKSPACE);
  EXPECT(attn_decode_paged(&d, (void*)FAKE, NULL, 0, NULL) == GCS_ERR_INVALID_ARG); /* out on q */
  e = d;
  e.num_reqs = 256;
  e.max_seq_len = 1 << 20;
  e.max_blocks_per_req = (1 << 20) / 16;
  EXPECT(attn_decode_workspace(&e) > ((size_t)64 << 20));
  EXPECT(attn_decode_paged_noalloc(&e, OUT, NULL) == GCS_ERR_WORKSPACE); /* partials exceed the scratch */

  /* cache strides: the [num_blocks, block_size, hkv, d] layout is accepted, slots that
   * overlap a kv head's rows are not */
  e = d;
  e.kv_stride_block = 16 * 4 * 128;
  e.kv_stride_head = 128;
  e.kv_stride_slot = 4 * 128;
  EXPECT(attn_decode_workspace(&e) == attn_decode_workspace(&d));
  EXPECT(attn_decode_paged(&e, OUT, NULL, 0, NULL) == GCS_ERR_WORKSPACE);
  e.kv_stride_slot = 2 * 128;
  EXPECT(attn_decode_paged(&e, OUT, NULL, 0, NULL) == GCS_ERR_UNSUPPORTED);
  e.kv_stride_slot = 4 * 128 + 8;
  EXPECT(attn_decode_paged(&e, OUT, NULL, 0, NULL) == GCS_ERR_UNSUPPORTED);

  /* paged prefill: any q_len, segments of whole 128-key tiles */
  e = d;
  e.max_q_len = 64;
  e.segment_len = 256;
  EXPECT(attn_prefill_paged_workspace(&e) > 0);
  EXPECT(attn_prefill_paged(&e, OUT, NULL, 0, NULL) == GCS_ERR_WORKSPACE);
  e.segment_len = 200;
  EXPECT(attn_prefill_paged(&e, OUT, NULL, 0, NULL) == GCS_ERR_UNSUPPORTED);

  /* checked mode: the switch, and the copy of cu_seqlens at the end of every workspace */
  EXPECT(gcs_set_device_checks(2) == GCS_ERR_INVALID_ARG);
  EXPECT(gcs_get_device_checks() == 0);
  {
    const size_t before = attn_fwd_workspace(&a);
    EXPECT(gcs_set_device_checks(1) == GCS_OK);
    EXPECT(gcs_get_device_checks() == 1);
    EXPECT(attn_fwd_workspace(&a) == before + 256);
    EXPECT(gcs_set_device_checks(0) == GCS_OK);
    EXPECT(attn_fwd_workspace(&a) == before);
  }
  EXPECT(gcs_get_device_status(NULL, 0) == GCS_ERR_INVALID_ARG);

  if (failures) {
    fprintf(stderr, "%d check(s) failed\n", failures);
    return 1;
  }
  printf("ok\n");
  return 0;
}
