// C ABI: host-side validation, workspace carving, TMA descriptor encoding and launches.
// Nothing here allocates device memory or synchronises (except gcs_get_device_status,
// which is a synchronous query by design).
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/gcs_attn.h"
#include "kernels.h"

namespace gcs {

__device__ int g_device_status = 0;

namespace {

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {nullptr};
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// gcs_set_device_checks: every call first checks its index arrays on the device
std::atomic<int> g_device_checks{0};
bool device_checks_on() { return g_device_checks.load(std::memory_order_relaxed) != 0; }

// events armed by gcs_set_kernel_events for the next call of this thread
thread_local cudaEvent_t t_ev_before = nullptr, t_ev_after = nullptr;

struct KernelTimer {
  cudaStream_t s;
  cudaEvent_t b, a;
  explicit KernelTimer(cudaStream_t st) : s(st), b(t_ev_before), a(t_ev_after) {
    t_ev_before = t_ev_after = nullptr;
  }
  void before() const {
    if (b) cudaEventRecord(b, s);
  }
  void after() const {
    if (a) cudaEventRecord(a, s);
  }
};
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// 2-D bf16 view [rows, width] with a 64 x box_rows box and 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t width, uint64_t rows, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {width, rows};
  cuuint64_t strides[1] = {width * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte view [rows, 128] of a paged fp8 cache, one page (16 rows x 128 B) per box, 128-byte
// swizzle.
bool make_page_map_u8(CUtensorMap* m, const void* base, uint64_t rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {128, rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, 16};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x) { return (x + 255) & ~size_t(255); }

// Byte range [a, b) of a caller buffer; a null pointer is an empty range.
struct Span {
  uintptr_t a, b;
};
Span span(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Span{a, p ? a + bytes : a};
}
bool overlap(const Span& x, const Span& y) { return x.a < x.b && y.a < y.b && x.a < y.b && y.a < x.b; }

// True when an output range overlaps an input range or another output range (kernels read
// their inputs and write their outputs concurrently, so any overlap is a race).
template <size_t NO, size_t NI>
bool outputs_overlap(const Span (&outs)[NO], const Span (&ins)[NI]) {
  for (size_t i = 0; i < NO; ++i) {
    for (size_t j = 0; j < NI; ++j)
      if (overlap(outs[i], ins[j])) return true;
    for (size_t j = i + 1; j < NO; ++j)
      if (overlap(outs[i], outs[j])) return true;
  }
  return false;
}

// Carves consecutive 256-B aligned regions out of a workspace.
struct Carver {
  uint8_t* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += round_up(count * sizeof(T));
    return p;
  }
};

bool supported_dims(int dqk, int dv) {
  return (dqk == 64 && dv == 64) || (dqk == 128 && dv == 128) || (dqk == 256 && dv == 256) ||
         (dqk == 256 && dv == 512) || (dqk == 512 && dv == 512);
}

int check_prefill(const gcs_prefill_args* a) {
  if (!a) return GCS_ERR_INVALID_ARG;
  if (a->num_seqs < 1 || a->total_tokens < 1 || a->max_seqlen < 1 || a->hq < 1 || a->hkv < 1)
    return GCS_ERR_INVALID_ARG;
  if (a->hq % a->hkv != 0) return GCS_ERR_INVALID_ARG;
  if (a->window < 0) return GCS_ERR_INVALID_ARG;
  if (a->deterministic != 0 && a->deterministic != 1) return GCS_ERR_INVALID_ARG;
  if (!std::isfinite(a->scale)) return GCS_ERR_INVALID_ARG;
  if (!a->cu_seqlens || !a->q || !a->k || !a->v) return GCS_ERR_INVALID_ARG;
  if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v)) return GCS_ERR_INVALID_ARG;
  if ((a->log_gate && !aligned16(a->log_gate)) || (a->sink && (reinterpret_cast<uintptr_t>(a->sink) & 3u)))
    return GCS_ERR_INVALID_ARG;
  if (!supported_dims(a->dqk, a->dv)) return GCS_ERR_UNSUPPORTED;
  // TMA coordinates and element offsets are 32-bit; keep every tensor below 2^31 elements
  const double big = 2147483647.0;
  if ((double)a->total_tokens * a->hq * (a->dqk > a->dv ? a->dqk : a->dv) > big) return GCS_ERR_UNSUPPORTED;
  return GCS_OK;
}

// Byte ranges of a prefill call's inputs: q, k, v, log_gate, sink, cu_seqlens.
struct PrefillSpans {
  Span q, k, v, g, s, cu;
};
PrefillSpans prefill_spans(const gcs_prefill_args* a) {
  const size_t t = (size_t)a->total_tokens;
  return PrefillSpans{span(a->q, t * a->hq * a->dqk * 2),     span(a->k, t * a->hkv * a->dqk * 2),
                      span(a->v, t * a->hkv * a->dv * 2),     span(a->log_gate, t * a->hq * 4),
                      span(a->sink, (size_t)a->hq * 4),       span(a->cu_seqlens, ((size_t)a->num_seqs + 1) * 4)};
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? GCS_OK : GCS_ERR_CUDA; }

int* status_ptr_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

// With device checks on, every workspace ends with the checked copy of cu_seqlens / cu_q.
size_t fwd_ws(const gcs_prefill_args* a, bool chk) {
  Carver c{nullptr};
  if (a->log_gate) c.take<float>((size_t)a->hq * a->total_tokens);
  if (chk) c.take<int32_t>((size_t)a->num_seqs + 1);
  return c.off;
}

// Head dims <= 128 take the two-pass backward (dQ pass + dK/dV pass, no fp32 dQ buffer);
// wider heads take the output-column roles with an fp32 dQ accumulator.
bool two_pass(const gcs_prefill_args* a) { return a->dqk <= 128 && a->dv <= 128; }

// Head dims above 128 take the query-stationary dQ pass when asked for a deterministic result,
// and where it is also the faster route (Dqk = 512, where the reduce-add role's 64-row steps
// cost more than the dQ pass's recompute); otherwise the dK role reduce-adds dQ in fp32.
bool wide_two_pass(const gcs_prefill_args* a) { return a->deterministic != 0 || a->dqk == 512; }

size_t bwd_ws(const gcs_prefill_args* a, bool chk) {
  Carver c{nullptr};
  const size_t ht = (size_t)a->hq * a->total_tokens;
  if (a->log_gate) c.take<float>(ht);                         // G^T
  c.take<float>(ht);                                           // delta
  if (!two_pass(a) && !wide_two_pass(a)) c.take<float>((size_t)a->total_tokens * a->hq * a->dqk);  // dQ accumulator
  if (a->log_gate || a->sink) c.take<float>(ht);               // row sums of dS
  if (a->log_gate) c.take<float>(ht);                          // column sums of dS
  c.take<float>((size_t)a->hq * ((a->total_tokens + 63) / 64 + a->num_seqs) * 128);  // packed vectors
  if (chk) c.take<int32_t>((size_t)a->num_seqs + 1);
  return c.off;
}

}  // namespace

int* device_status_ptr() { return status_ptr_for_current_device(); }

}  // namespace gcs

using namespace gcs;

extern "C" {

const char* gcs_status_str(int s) {
  switch (s) {
    case GCS_OK: return "ok";
    case GCS_ERR_INVALID_ARG: return "invalid argument";
    case GCS_ERR_UNSUPPORTED: return "unsupported shape, dtype or layout";
    case GCS_ERR_WORKSPACE: return "workspace missing or too small";
    case GCS_ERR_CUDA: return "CUDA error";
    case GCS_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a bounded wait";
    default: return "unknown status";
  }
}

const char* gcs_version(void) { return "gcs_attn 0.1 (sm_103a)"; }

size_t attn_fwd_workspace(const gcs_prefill_args* a) {
  return (a && check_prefill(a) == GCS_OK) ? fwd_ws(a, device_checks_on()) : 0;
}

size_t attn_bwd_workspace(const gcs_prefill_args* a) {
  return (a && check_prefill(a) == GCS_OK) ? bwd_ws(a, device_checks_on()) : 0;
}

int attn_fwd(const gcs_prefill_args* a, void* o, float* lse, void* workspace, size_t workspace_bytes,
             gcs_stream_t stream) {
  int st = check_prefill(a);
  if (st != GCS_OK) return st;
  if (!o || !lse || !aligned16(o) || !aligned16(lse)) return GCS_ERR_INVALID_ARG;
  {
    const size_t t = (size_t)a->total_tokens;
    const PrefillSpans in = prefill_spans(a);
    const Span outs[] = {span(o, t * a->hq * a->dv * 2), span(lse, t * a->hq * 4)};
    const Span ins[] = {in.q, in.k, in.v, in.g, in.s, in.cu};
    if (outputs_overlap(outs, ins)) return GCS_ERR_INVALID_ARG;
  }
  const bool chk = device_checks_on();
  const size_t need = fwd_ws(a, chk);
  if (need > 0 && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return GCS_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* status = device_status_ptr();
  if (!status) return GCS_ERR_CUDA;

  Carver c{static_cast<uint8_t*>(workspace)};
  float* gT = a->log_gate ? c.take<float>((size_t)a->hq * a->total_tokens) : nullptr;
  int32_t* cu_chk = chk ? c.take<int32_t>((size_t)a->num_seqs + 1) : nullptr;

  FwdMaps maps;
  if (!make_map(&maps.q, a->q, (uint64_t)a->hq * a->dqk, a->total_tokens, 128) ||
      !make_map(&maps.k, a->k, (uint64_t)a->hkv * a->dqk, a->total_tokens, 128) ||
      !make_map(&maps.v, a->v, (uint64_t)a->hkv * a->dv, a->total_tokens, 128))
    return GCS_ERR_CUDA;

  // the kernels read the checked copy of cu_seqlens when device checks are on
  const int32_t* cu = a->cu_seqlens;
  if (cu_chk) {
    st = cuda_status(launch_check_prefill(a->cu_seqlens, a->num_seqs, a->total_tokens, a->max_seqlen, cu_chk, status, s));
    if (st != GCS_OK) return st;
    cu = cu_chk;
  }
  if (gT) {
    st = cuda_status(launch_gate_cumsum(a->log_gate, cu, a->num_seqs, a->total_tokens, a->hq, gT, s));
    if (st != GCS_OK) return st;
  }
  FwdParams p;
  p.cu_seqlens = cu;
  p.num_seqs = a->num_seqs;
  p.total = a->total_tokens;
  p.hq = a->hq;
  p.hkv = a->hkv;
  p.dqk = a->dqk;
  p.dv = a->dv;
  p.dv_chunk = a->dv > 256 ? 256 : a->dv;
  p.scale_log2 = a->scale * 1.4426950408889634f;
  p.window = a->window;
  p.gT = gT;
  p.sink = a->sink;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.status = status;
  KernelTimer timer(s);
  timer.before();
  if (a->dqk == a->dv && a->dqk <= 128) {
    const int num_pairs = (a->total_tokens + 255) / 256 + a->num_seqs;
    st = cuda_status(launch_prefill_fwd2(p, maps, num_pairs, s));
  } else {
    const int num_tiles = (a->total_tokens + 127) / 128 + a->num_seqs;
    st = cuda_status(launch_prefill_fwd(p, maps, num_tiles, s));
  }
  timer.after();
  return st;
}

int attn_bwd(const gcs_prefill_args* a, const void* o, const float* lse, const void* dout, void* dq, void* dk, void* dv,
             float* dlog_gate, float* dsink, void* workspace, size_t workspace_bytes, gcs_stream_t stream) {
  int st = check_prefill(a);
  if (st != GCS_OK) return st;
  if (!o || !lse || !dout || !dq || !dk || !dv) return GCS_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(lse) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return GCS_ERR_INVALID_ARG;
  if ((dlog_gate == nullptr) != (a->log_gate == nullptr)) return GCS_ERR_INVALID_ARG;
  if ((dsink == nullptr) != (a->sink == nullptr)) return GCS_ERR_INVALID_ARG;
  {
    const size_t t = (size_t)a->total_tokens;
    const PrefillSpans in = prefill_spans(a);
    const Span outs[] = {span(dq, t * a->hq * a->dqk * 2), span(dk, t * a->hkv * a->dqk * 2),
                         span(dv, t * a->hkv * a->dv * 2), span(dlog_gate, t * a->hq * 4),
                         span(dsink, (size_t)a->hq * 4)};
    const Span ins[] = {in.q,  in.k, in.v, in.g, in.s, in.cu, span(o, t * a->hq * a->dv * 2), span(lse, t * a->hq * 4),
                        span(dout, t * a->hq * a->dv * 2)};
    if (outputs_overlap(outs, ins)) return GCS_ERR_INVALID_ARG;
  }
  const bool chk = device_checks_on();
  const size_t need = bwd_ws(a, chk);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return GCS_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* status = device_status_ptr();
  if (!status) return GCS_ERR_CUDA;

  const size_t ht = (size_t)a->hq * a->total_tokens;
  Carver c{static_cast<uint8_t*>(workspace)};
  float* gT = a->log_gate ? c.take<float>(ht) : nullptr;
  float* delta = c.take<float>(ht);
  const bool tp = two_pass(a);
  const bool wide_det = !tp && wide_two_pass(a);
  // fp32 dQ accumulator: wide heads on the reduce-add route only
  float* dq_acc = (tp || wide_det) ? nullptr : c.take<float>((size_t)a->total_tokens * a->hq * a->dqk);
  float* dg_row = (a->log_gate || a->sink) ? c.take<float>(ht) : nullptr;
  float* dg_col = a->log_gate ? c.take<float>(ht) : nullptr;
  const int n_qtiles = (a->total_tokens + 63) / 64 + a->num_seqs;
  float* vecp = c.take<float>((size_t)a->hq * n_qtiles * 128);
  int32_t* cu_chk = chk ? c.take<int32_t>((size_t)a->num_seqs + 1) : nullptr;

  BwdMaps maps;
  if (!make_map(&maps.q, a->q, (uint64_t)a->hq * a->dqk, a->total_tokens, 64) ||
      !make_map(&maps.k, a->k, (uint64_t)a->hkv * a->dqk, a->total_tokens, 128) ||
      !make_map(&maps.v, a->v, (uint64_t)a->hkv * a->dv, a->total_tokens, 128) ||
      !make_map(&maps.dout, dout, (uint64_t)a->hq * a->dv, a->total_tokens, 64) ||
      !make_map(&maps.q128, a->q, (uint64_t)a->hq * a->dqk, a->total_tokens, 128) ||
      !make_map(&maps.dout128, dout, (uint64_t)a->hq * a->dv, a->total_tokens, 128))
    return GCS_ERR_CUDA;

  const int32_t* cu = a->cu_seqlens;
  if (cu_chk) {
    st = cuda_status(launch_check_prefill(a->cu_seqlens, a->num_seqs, a->total_tokens, a->max_seqlen, cu_chk, status, s));
    if (st != GCS_OK) return st;
    cu = cu_chk;
  }
  if (gT) {
    st = cuda_status(launch_gate_cumsum(a->log_gate, cu, a->num_seqs, a->total_tokens, a->hq, gT, s));
    if (st != GCS_OK) return st;
  }
  st = cuda_status(launch_bwd_pre(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout),
                                  a->total_tokens, a->hq, a->dv, a->dqk, delta, dq_acc, dg_row, dg_col, s));
  if (st != GCS_OK) return st;

  st = cuda_status(launch_bwd_pack(cu, a->num_seqs, a->total_tokens, a->hq, n_qtiles, lse, gT, delta,
                                   vecp, s));
  if (st != GCS_OK) return st;

  BwdParams p;
  p.cu_seqlens = cu;
  p.num_seqs = a->num_seqs;
  p.total = a->total_tokens;
  p.hq = a->hq;
  p.hkv = a->hkv;
  p.dqk = a->dqk;
  p.dv = a->dv;
  p.scale = a->scale;
  p.scale_log2 = a->scale * 1.4426950408889634f;
  p.window = a->window;
  p.gT = gT;
  p.lse = lse;
  p.delta = delta;
  p.grad_q = static_cast<uint16_t*>(dq);
  p.grad_k = static_cast<uint16_t*>(dk);
  p.grad_v = static_cast<uint16_t*>(dv);
  p.dq_acc = dq_acc;
  p.dg_row = dg_row;
  p.dg_col = dg_col;
  p.vecp = vecp;
  p.n_qtiles = n_qtiles;
  p.status = status;
  const int num_tiles = (a->total_tokens + 127) / 128 + a->num_seqs;
  KernelTimer timer(s);
  if (tp) {
    // dQ pass (query tiles of 128 rows), then the dK/dV pass; the timer brackets both
    BwdMaps dqmaps = maps;
    dqmaps.q = maps.q128;
    dqmaps.dout = maps.dout128;
    timer.before();
    st = cuda_status(launch_prefill_bwd_dq(p, dqmaps, num_tiles, s));
    if (st != GCS_OK) return st;
    st = cuda_status(launch_prefill_bwd(p, maps, num_tiles, s));
    timer.after();
  } else if (wide_det) {
    // dQ pass (query tiles of 64 rows), then the dK / dV roles; the timer brackets both
    timer.before();
    st = cuda_status(launch_prefill_bwd_wide_dq(p, maps, n_qtiles, s));
    if (st != GCS_OK) return st;
    st = cuda_status(launch_prefill_bwd_wide(p, maps, num_tiles, false, s));
    timer.after();
  } else {
    timer.before();
    st = cuda_status(launch_prefill_bwd_wide(p, maps, num_tiles, true, s));
    timer.after();
  }
  if (st != GCS_OK) return st;
  return cuda_status(launch_bwd_post(dq_acc, static_cast<uint16_t*>(dq), a->total_tokens, a->hq, a->dqk,
                                     cu, a->num_seqs, dg_row, dg_col, dlog_gate, lse, delta, a->sink,
                                     dsink, s));
}

static int check_decode(const gcs_decode_args* a) {
  if (!a) return GCS_ERR_INVALID_ARG;
  if (a->num_reqs < 1 || a->total_q < 1 || a->max_q_len < 1 || a->max_seq_len < 1 || a->max_blocks_per_req < 1 ||
      a->num_blocks < 1 || a->hq < 1 || a->hkv < 1 || a->segment_len < 1)
    return GCS_ERR_INVALID_ARG;
  if (!a->cu_q || !a->seq_lens || !a->block_table || !a->k_cache || !a->v_cache || !a->q)
    return GCS_ERR_INVALID_ARG;
  if (!std::isfinite(a->scale)) return GCS_ERR_INVALID_ARG;
  if (a->kv_format == GCS_KV_BF16) {
    // a bf16 cache carries no scales
    if (a->k_scale || a->v_scale || a->scale_mode != GCS_SCALE_PER_TOKEN) return GCS_ERR_INVALID_ARG;
  } else if (a->kv_format == GCS_KV_FP8_E4M3) {
    if (!a->k_scale || !a->v_scale) return GCS_ERR_INVALID_ARG;
    if (a->scale_mode == GCS_SCALE_PER_TOKEN) {
      if (!aligned16(a->k_scale) || !aligned16(a->v_scale)) return GCS_ERR_INVALID_ARG;
    } else if (a->scale_mode == GCS_SCALE_PER_TENSOR) {
      if ((reinterpret_cast<uintptr_t>(a->k_scale) | reinterpret_cast<uintptr_t>(a->v_scale)) & 3u)
        return GCS_ERR_INVALID_ARG;
    } else {
      return GCS_ERR_INVALID_ARG;
    }
  } else {
    return GCS_ERR_INVALID_ARG;
  }
  // per-token scales are only read on decode / short-query shapes (a prefill shape is rejected)
  if (a->max_q_len > 4) return GCS_ERR_UNSUPPORTED;
  if (a->d != 128 || a->block_size != 16 || a->hq != 16 * a->hkv) return GCS_ERR_UNSUPPORTED;
  if (a->segment_len % a->block_size != 0) return GCS_ERR_UNSUPPORTED;
  if ((long long)a->max_blocks_per_req * a->block_size < a->max_seq_len) return GCS_ERR_INVALID_ARG;
  if (!aligned16(a->k_cache) || !aligned16(a->v_cache) || !aligned16(a->q)) return GCS_ERR_INVALID_ARG;
  if (a->window < 0) return GCS_ERR_INVALID_ARG;
  if (a->g_cache && !aligned16(a->g_cache)) return GCS_ERR_INVALID_ARG;
  if (a->sink && (reinterpret_cast<uintptr_t>(a->sink) & 3u)) return GCS_ERR_INVALID_ARG;
  if ((double)a->num_blocks * a->hkv * a->block_size * a->d > 9.0e15) return GCS_ERR_UNSUPPORTED;
  // the fp8 pages are fetched by tensor copies whose row coordinate is a 32-bit integer
  if (a->kv_format == GCS_KV_FP8_E4M3 && (double)a->num_blocks * a->hkv * a->block_size > 2147483647.0)
    return GCS_ERR_UNSUPPORTED;
  return GCS_OK;
}

// True when the output of a paged call overlaps one of its inputs.
static bool paged_out_overlaps(const gcs_decode_args* a, const void* out) {
  const size_t rows = (size_t)a->num_blocks * a->hkv * a->block_size;
  const size_t elt = a->kv_format == GCS_KV_BF16 ? 2 : 1;
  const size_t sc = a->scale_mode == GCS_SCALE_PER_TENSOR ? 4 : rows * 4;
  const Span outs[] = {span(out, (size_t)a->total_q * a->hq * a->d * 2)};
  const Span ins[] = {span(a->q, (size_t)a->total_q * a->hq * a->d * 2),
                      span(a->k_cache, rows * a->d * elt),
                      span(a->v_cache, rows * a->d * elt),
                      span(a->k_scale, sc),
                      span(a->v_scale, sc),
                      span(a->block_table, (size_t)a->num_reqs * a->max_blocks_per_req * 4),
                      span(a->seq_lens, (size_t)a->num_reqs * 4),
                      span(a->cu_q, ((size_t)a->num_reqs + 1) * 4),
                      span(a->g_cache, (size_t)a->num_blocks * a->hq * a->block_size * 4),
                      span(a->sink, (size_t)a->hq * 4)};
  return outputs_overlap(outs, ins);
}

// Kernel parameters common to the paged calls (segments and partial buffers set by the caller).
static void fill_paged_params(const gcs_decode_args* a, void* out, int* status, DecodeParams& p) {
  p.cu_q = a->cu_q;
  p.seq_lens = a->seq_lens;
  p.block_table = a->block_table;
  p.max_blocks = a->max_blocks_per_req;
  p.k_cache = static_cast<const uint8_t*>(a->k_cache);
  p.v_cache = static_cast<const uint8_t*>(a->v_cache);
  p.k_scale = a->k_scale;
  p.v_scale = a->v_scale;
  p.kv_format = a->kv_format;
  p.scale_mode = a->scale_mode;
  p.g_cache = a->g_cache;
  p.sink = a->sink;
  p.window = a->window;
  p.num_reqs = a->num_reqs;
  p.hq = a->hq;
  p.hkv = a->hkv;
  p.max_q_len = a->max_q_len;
  p.max_segs = 1;
  p.seg_pages = 0;
  p.scale = a->scale;
  p.q = static_cast<const uint16_t*>(a->q);
  p.out = static_cast<uint16_t*>(out);
  p.part_acc = nullptr;
  p.part_ml = nullptr;
  p.status = status;
}

// Bytes of the split-K partials (acc, then (m, l)) of num_reqs x max_segs x hkv units.
static size_t partials_ws(const gcs_decode_args* a, int max_segs) {
  const size_t units = (size_t)a->num_reqs * max_segs * a->hkv;
  const size_t rows = (size_t)a->max_q_len * 16;
  return round_up(units * rows * 128 * sizeof(float)) + round_up(units * rows * 2 * sizeof(float));
}

// Bytes of the checked copy of cu_q that ends the workspace when device checks are on.
static size_t cu_q_copy_ws(const gcs_decode_args* a, bool chk) {
  return chk ? round_up(((size_t)a->num_reqs + 1) * sizeof(int32_t)) : 0;
}

static size_t decode_ws(const gcs_decode_args* a, bool chk, int* max_segs_out) {
  const int max_segs = (a->max_seq_len + a->segment_len - 1) / a->segment_len;
  if (max_segs_out) *max_segs_out = max_segs;
  return partials_ws(a, max_segs) + cu_q_copy_ws(a, chk);
}

// Runs the device-content checks of a paged call when they are on: p.cu_q then points to the
// checked copy at byte offset `off` of the workspace.
static int paged_checks(const gcs_decode_args* a, void* workspace, size_t off, DecodeParams& p, cudaStream_t s) {
  int32_t* cu_chk = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + off);
  const int st = cuda_status(launch_check_paged(a->cu_q, a->seq_lens, a->block_table, a->num_reqs, a->total_q,
                                                a->max_q_len, a->max_seq_len, a->max_blocks_per_req, a->num_blocks,
                                                a->block_size, a->window, cu_chk, p.status, s));
  if (st == GCS_OK) p.cu_q = cu_chk;
  return st;
}

size_t attn_decode_workspace(const gcs_decode_args* a) {
  return (a && check_decode(a) == GCS_OK) ? decode_ws(a, device_checks_on(), nullptr) : 0;
}

int attn_decode_paged(const gcs_decode_args* a, void* out, void* workspace, size_t workspace_bytes,
                      gcs_stream_t stream) {
  int st = check_decode(a);
  if (st != GCS_OK) return st;
  if (!out || !aligned16(out)) return GCS_ERR_INVALID_ARG;
  if (paged_out_overlaps(a, out)) return GCS_ERR_INVALID_ARG;
  int max_segs = 0;
  const bool chk = device_checks_on();
  const size_t need = decode_ws(a, chk, &max_segs);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return GCS_ERR_WORKSPACE;
  int* status = device_status_ptr();
  if (!status) return GCS_ERR_CUDA;
  const size_t units = (size_t)a->num_reqs * max_segs * a->hkv;
  const size_t rows = (size_t)a->max_q_len * 16;
  DecodeParams p;
  fill_paged_params(a, out, status, p);
  p.max_segs = max_segs;
  p.seg_pages = a->segment_len / a->block_size;
  p.part_acc = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + round_up(units * rows * 128 * sizeof(float)));
  DecodeMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (a->kv_format == GCS_KV_FP8_E4M3) {
    const uint64_t cache_rows = (uint64_t)a->num_blocks * a->hkv * a->block_size;
    if (!make_page_map_u8(&maps.k, a->k_cache, cache_rows) || !make_page_map_u8(&maps.v, a->v_cache, cache_rows))
      return GCS_ERR_CUDA;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (chk) {
    const int st2 = paged_checks(a, workspace, partials_ws(a, max_segs), p, s);
    if (st2 != GCS_OK) return st2;
  }
  KernelTimer timer(s);
  return cuda_status(launch_decode(p, maps, s, &timer.b, &timer.a));
}

int attn_decode_paged_noalloc(const gcs_decode_args* a, void* out, gcs_stream_t stream) {
  int st = check_decode(a);
  if (st != GCS_OK) return st;
  // the split-K partials must fit the library's fixed scratch
  if (decode_ws(a, device_checks_on(), nullptr) > kNoAllocScratchBytes) return GCS_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (decode_noalloc_scratch(&scratch) != cudaSuccess) return GCS_ERR_CUDA;
  return attn_decode_paged(a, out, scratch, kNoAllocScratchBytes, stream);
}

// Paged chunked prefill: the decode checks with the q_len limit lifted, fp8 only, and
// segment_len 0 (automatic) or a multiple of 128 tokens (one key tile of 8 pages).
static int check_prefill_paged(const gcs_decode_args* a) {
  if (!a) return GCS_ERR_INVALID_ARG;
  if (a->max_q_len < 1 || a->segment_len < 0) return GCS_ERR_INVALID_ARG;
  gcs_decode_args b = *a;
  b.max_q_len = a->max_q_len < 4 ? a->max_q_len : 4;
  b.segment_len = a->segment_len > 0 ? a->segment_len : 128;
  const int st = check_decode(&b);
  if (st != GCS_OK) return st;
  if (a->kv_format != GCS_KV_FP8_E4M3) return GCS_ERR_UNSUPPORTED;
  if (a->segment_len % 128 != 0) return GCS_ERR_UNSUPPORTED;
  if (a->max_q_len > a->max_seq_len) return GCS_ERR_INVALID_ARG;
  return GCS_OK;
}

struct PagedPlan {
  int seg_pages = 0, max_segs = 1;  // max_segs 1: one segment per request, the kernel writes out directly
  size_t part_ws = 0;               // split-K partials (none with one segment)
  size_t ws = 0;                    // + the checked copy of cu_q with device checks on
};

// Segments of the paged prefill: the caller's, or (segment_len 0) the fewest that give
// about two CTAs per SM with the query blocks of 16 positions x kv heads x requests.
static bool plan_prefill_paged(const gcs_decode_args* a, bool chk, PagedPlan* pl) {
  const int max_pages = (a->max_seq_len + 15) / 16;
  int sp;
  if (a->segment_len > 0) {
    sp = a->segment_len / 16;
  } else {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return false;
    const long long ctas = (long long)((a->max_q_len + 15) / 16) * a->hkv * a->num_reqs;
    long long want = (2LL * nsm + ctas - 1) / ctas;
    if (want < 1) want = 1;
    sp = (int)((max_pages + want - 1) / want);
    sp = ((sp + 7) / 8) * 8;
  }
  pl->seg_pages = sp;
  pl->max_segs = (max_pages + sp - 1) / sp;
  pl->part_ws = pl->max_segs > 1 ? partials_ws(a, pl->max_segs) : 0;
  pl->ws = pl->part_ws + cu_q_copy_ws(a, chk);
  return true;
}

size_t attn_prefill_paged_workspace(const gcs_decode_args* a) {
  PagedPlan pl;
  if (!a || check_prefill_paged(a) != GCS_OK || !plan_prefill_paged(a, device_checks_on(), &pl)) return 0;
  return pl.ws;
}

int attn_prefill_paged(const gcs_decode_args* a, void* out, void* workspace, size_t workspace_bytes,
                       gcs_stream_t stream) {
  int st = check_prefill_paged(a);
  if (st != GCS_OK) return st;
  if (!out || !aligned16(out)) return GCS_ERR_INVALID_ARG;
  if (paged_out_overlaps(a, out)) return GCS_ERR_INVALID_ARG;
  PagedPlan pl;
  const bool chk = device_checks_on();
  if (!plan_prefill_paged(a, chk, &pl)) return GCS_ERR_CUDA;
  if (pl.ws > 0 && (!workspace || workspace_bytes < pl.ws || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return GCS_ERR_WORKSPACE;
  int* status = device_status_ptr();
  if (!status) return GCS_ERR_CUDA;
  DecodeParams p;
  fill_paged_params(a, out, status, p);
  p.max_segs = pl.max_segs;
  p.seg_pages = pl.seg_pages;
  if (pl.max_segs > 1) {
    const size_t units = (size_t)a->num_reqs * pl.max_segs * a->hkv;
    const size_t rows = (size_t)a->max_q_len * 16;
    p.part_acc = static_cast<float*>(workspace);
    p.part_ml =
        reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + round_up(units * rows * 128 * sizeof(float)));
  }
  DecodeMaps maps;
  const uint64_t cache_rows = (uint64_t)a->num_blocks * a->hkv * a->block_size;
  if (!make_page_map_u8(&maps.k, a->k_cache, cache_rows) || !make_page_map_u8(&maps.v, a->v_cache, cache_rows))
    return GCS_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (chk) {
    const int st2 = paged_checks(a, workspace, pl.part_ws, p, s);
    if (st2 != GCS_OK) return st2;
  }
  KernelTimer timer(s);
  return cuda_status(launch_prefill_paged(p, maps, s, &timer.b, &timer.a));
}

int gcs_set_device_checks(int enable) {
  if (enable != 0 && enable != 1) return GCS_ERR_INVALID_ARG;
  g_device_checks.store(enable, std::memory_order_relaxed);
  return GCS_OK;
}

int gcs_get_device_checks(void) { return device_checks_on() ? 1 : 0; }

int gcs_check_prefill_inputs(const gcs_prefill_args* a, gcs_stream_t stream) {
  const int st = check_prefill(a);
  if (st != GCS_OK) return st;
  int* status = device_status_ptr();
  if (!status) return GCS_ERR_CUDA;
  return cuda_status(launch_check_prefill(a->cu_seqlens, a->num_seqs, a->total_tokens, a->max_seqlen, nullptr, status,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int gcs_check_paged_inputs(const gcs_decode_args* a, gcs_stream_t stream) {
  // the arguments of either paged call
  if (check_decode(a) != GCS_OK) {
    const int st = check_prefill_paged(a);
    if (st != GCS_OK) return st;
  }
  int* status = device_status_ptr();
  if (!status) return GCS_ERR_CUDA;
  return cuda_status(launch_check_paged(a->cu_q, a->seq_lens, a->block_table, a->num_reqs, a->total_q, a->max_q_len,
                                        a->max_seq_len, a->max_blocks_per_req, a->num_blocks, a->block_size,
                                        a->window, nullptr, status, reinterpret_cast<cudaStream_t>(stream)));
}

int gcs_set_kernel_events(void* before, void* after) {
  t_ev_before = static_cast<cudaEvent_t>(before);
  t_ev_after = static_cast<cudaEvent_t>(after);
  return GCS_OK;
}

int gcs_selftest_bounded_wait(gcs_stream_t stream) {
  int* d = device_status_ptr();
  if (!d) return GCS_ERR_CUDA;
  return cuda_status(launch_bounded_wait_selftest(d, reinterpret_cast<cudaStream_t>(stream)));
}

int gcs_get_device_status(int* status, int clear) {
  if (!status) return GCS_ERR_INVALID_ARG;
  int* d = device_status_ptr();
  if (!d) return GCS_ERR_CUDA;
  if (cudaMemcpy(status, d, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GCS_ERR_CUDA;
  if (clear && cudaMemset(d, 0, sizeof(int)) != cudaSuccess) return GCS_ERR_CUDA;
  return GCS_OK;
}

}  // extern "C"
