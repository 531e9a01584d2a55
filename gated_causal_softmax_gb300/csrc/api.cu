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

// Element strides (token, head) of a [tokens, heads, dim] tensor with dim contiguous.
struct Layout {
  long long ts, hs;
};

// 3-D bf16 map {dim, heads, tokens} with a 64 x 1 x box_rows box and 128-byte swizzle: one
// box is 64 columns of one head for box_rows tokens, the same shared-memory tile as a 2-D box.
bool make_map(CUtensorMap* m, const void* base, int dim, int heads, int tokens, const Layout& l, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)l.hs * 2, (cuuint64_t)l.ts * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D fp32 map {dim, heads, tokens} of a contiguous [tokens, heads, dim] accumulator with a
// 32 x 1 x box_rows box and the 128-byte swizzle: the target of tiled reduce-adds.
bool make_map_f32(CUtensorMap* m, void* base, int dim, int heads, int tokens, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)dim * 4, (cuuint64_t)dim * heads * 4};
  cuuint32_t box[3] = {32, 1, box_rows};  // 32 fp32 = one 128-byte swizzle row
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Byte strides (block, kv head, slot) of a paged cache.
struct CacheLayout {
  long long bs, hs, ss;
  bool head_inner() const { return hs < ss; }
};

// 4-D byte map of a paged fp8 cache, dims in increasing stride order: {128 B, slot, kv head,
// block}, or {128 B, kv head, slot, block} when the kv head is the inner one.  One box is one
// 16-slot page of one kv head (16 x 128 B, 128-byte swizzle), the same tile either way.
bool make_page_map_u8(CUtensorMap* m, const void* base, int num_blocks, int hkv, int block_size,
                      const CacheLayout& l) {
  auto enc = encode_fn();
  if (!enc) return false;
  const bool hi = l.head_inner();
  cuuint64_t dims[4] = {128, (cuuint64_t)(hi ? hkv : block_size), (cuuint64_t)(hi ? block_size : hkv),
                        (cuuint64_t)num_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)(hi ? l.hs : l.ss), (cuuint64_t)(hi ? l.ss : l.hs), (cuuint64_t)l.bs};
  cuuint32_t box[4] = {128, hi ? 1u : 16u, hi ? 16u : 1u, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, es,
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
// A strided token-major tensor: byte range plus the period (token stride in bytes) and the
// bytes one token covers; period 0 = one dense range.
struct TSpan {
  uintptr_t a, b;
  unsigned long long period, width;
};
TSpan tspan(const void* p, int tokens, int heads, int dim, const Layout& l, int elt) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  if (!p || tokens <= 0) return TSpan{a, a, 0, 0};
  const unsigned long long w = ((unsigned long long)(heads - 1) * l.hs + dim) * elt;
  return TSpan{a, a + (unsigned long long)(tokens - 1) * l.ts * elt + w, (unsigned long long)l.ts * elt, w};
}
TSpan tspan(const Span& s) { return TSpan{s.a, s.b, 0, 0}; }
// True when two byte sets meet.  Two tensors with the same token period whose per-token ranges
// sit side by side within every period (heads of one fused buffer) do not.
bool overlap(const TSpan& x, const TSpan& y) {
  if (!(x.a < x.b && y.a < y.b && x.a < y.b && y.a < x.b)) return false;
  if (x.period != 0 && x.period == y.period && x.width <= x.period && y.width <= y.period) {
    const unsigned long long P = x.period;
    const unsigned long long d = (unsigned long long)((y.a >= x.a ? y.a - x.a : P - (x.a - y.a) % P) % P);
    return !(d >= x.width && d + y.width <= P);
  }
  return true;
}

// True when an output range overlaps an input range or another output range (kernels read
// their inputs and write their outputs concurrently, so any overlap is a race).
template <size_t NO, size_t NI>
bool outputs_overlap(const TSpan (&outs)[NO], const TSpan (&ins)[NI]) {
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

// {0, 0} = contiguous; otherwise token-major without overlap, 16-byte granules.
int resolve_layout(const gcs_strides& st, int heads, int dim, Layout* out) {
  if (st.token == 0 && st.head == 0) {
    *out = Layout{(long long)heads * dim, dim};
    return GCS_OK;
  }
  if (st.token < 0 || st.head < 0) return GCS_ERR_INVALID_ARG;
  if (st.head < dim || st.token < (long long)heads * st.head) return GCS_ERR_UNSUPPORTED;
  if ((st.head % 8) != 0 || (st.token % 8) != 0) return GCS_ERR_UNSUPPORTED;
  if (st.token > (1LL << 38)) return GCS_ERR_UNSUPPORTED;  // tensor-copy strides stay below 2^40 bytes
  *out = Layout{st.token, st.head};
  return GCS_OK;
}

struct PrefillLayouts {
  Layout q, k, v, o, dout, dq, dk, dv;
};

int prefill_layouts(const gcs_prefill_args* a, PrefillLayouts* l) {
  int st;
  if ((st = resolve_layout(a->q_stride, a->hq, a->dqk, &l->q)) != GCS_OK) return st;
  if ((st = resolve_layout(a->k_stride, a->hkv, a->dqk, &l->k)) != GCS_OK) return st;
  if ((st = resolve_layout(a->v_stride, a->hkv, a->dv, &l->v)) != GCS_OK) return st;
  if ((st = resolve_layout(a->o_stride, a->hq, a->dv, &l->o)) != GCS_OK) return st;
  if ((st = resolve_layout(a->do_stride, a->hq, a->dv, &l->dout)) != GCS_OK) return st;
  if ((st = resolve_layout(a->dq_stride, a->hq, a->dqk, &l->dq)) != GCS_OK) return st;
  if ((st = resolve_layout(a->dk_stride, a->hkv, a->dqk, &l->dk)) != GCS_OK) return st;
  return resolve_layout(a->dv_stride, a->hkv, a->dv, &l->dv);
}

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
  // 32-bit element counts of the contiguous fp32 workspaces and in-kernel indices: keep every
  // tensor below 2^31 elements
  const double big = 2147483647.0;
  if ((double)a->total_tokens * a->hq * (a->dqk > a->dv ? a->dqk : a->dv) > big) return GCS_ERR_UNSUPPORTED;
  PrefillLayouts l;
  return prefill_layouts(a, &l);
}

// Byte ranges of a prefill call's inputs: q, k, v, log_gate, sink, cu_seqlens.
struct PrefillSpans {
  TSpan q, k, v, g, s, cu;
};
PrefillSpans prefill_spans(const gcs_prefill_args* a, const PrefillLayouts& l) {
  const size_t t = (size_t)a->total_tokens;
  const int T = a->total_tokens;
  return PrefillSpans{tspan(a->q, T, a->hq, a->dqk, l.q, 2),         tspan(a->k, T, a->hkv, a->dqk, l.k, 2),
                      tspan(a->v, T, a->hkv, a->dv, l.v, 2),         tspan(span(a->log_gate, t * a->hq * 4)),
                      tspan(span(a->sink, (size_t)a->hq * 4)), tspan(span(a->cu_seqlens, ((size_t)a->num_seqs + 1) * 4))};
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

// Head dim 128 without `deterministic` takes the single-pass backward (dQ reduce-added into an
// fp32 buffer); head dim 64, and 128 with `deterministic`, the two-pass backward (dQ pass +
// dK/dV pass, no fp32 dQ buffer); wider heads the output-column roles below.
bool fused(const gcs_prefill_args* a) { return a->dqk == 128 && a->dv == 128 && a->deterministic == 0; }
bool two_pass(const gcs_prefill_args* a) { return a->dqk <= 128 && a->dv <= 128 && !fused(a); }

// Head dims above 128 take the query-stationary dQ pass when asked for a deterministic result,
// and where it is also the faster route (Dqk = 512, where the reduce-add role's 64-row steps
// cost more than the dQ pass's recompute); otherwise the dK role reduce-adds dQ in fp32.
bool wide_two_pass(const gcs_prefill_args* a) { return a->deterministic != 0 || a->dqk == 512; }

size_t bwd_ws(const gcs_prefill_args* a, bool chk) {
  Carver c{nullptr};
  const size_t ht = (size_t)a->hq * a->total_tokens;
  if (a->log_gate) c.take<float>(ht);                         // G^T
  c.take<float>(ht);                                           // delta
  if (fused(a) || (a->dqk > 128 && !wide_two_pass(a)))
    c.take<float>((size_t)a->total_tokens * a->hq * a->dqk);  // dQ accumulator
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
  PrefillLayouts lay;
  prefill_layouts(a, &lay);
  {
    const size_t t = (size_t)a->total_tokens;
    const PrefillSpans in = prefill_spans(a, lay);
    const TSpan outs[] = {tspan(o, a->total_tokens, a->hq, a->dv, lay.o, 2), tspan(span(lse, t * a->hq * 4))};
    const TSpan ins[] = {in.q, in.k, in.v, in.g, in.s, in.cu};
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
  if (!make_map(&maps.q, a->q, a->dqk, a->hq, a->total_tokens, lay.q, 128) ||
      !make_map(&maps.k, a->k, a->dqk, a->hkv, a->total_tokens, lay.k, 128) ||
      !make_map(&maps.v, a->v, a->dv, a->hkv, a->total_tokens, lay.v, 128))
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
  p.o_ts = lay.o.ts;
  p.o_hs = lay.o.hs;
  p.lse = lse;
  p.status = status;
  KernelTimer timer(s);
  timer.before();
  if (a->dqk == a->dv && a->dqk <= 128) {
    st = cuda_status(launch_prefill_fwd2(p, maps, s));
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
  PrefillLayouts lay;
  prefill_layouts(a, &lay);
  {
    const size_t t = (size_t)a->total_tokens;
    const int T = a->total_tokens;
    const PrefillSpans in = prefill_spans(a, lay);
    const TSpan outs[] = {tspan(dq, T, a->hq, a->dqk, lay.dq, 2), tspan(dk, T, a->hkv, a->dqk, lay.dk, 2),
                          tspan(dv, T, a->hkv, a->dv, lay.dv, 2), tspan(span(dlog_gate, t * a->hq * 4)),
                          tspan(span(dsink, (size_t)a->hq * 4))};
    const TSpan ins[] = {in.q, in.k, in.v, in.g, in.s, in.cu, tspan(o, T, a->hq, a->dv, lay.o, 2),
                         tspan(span(lse, t * a->hq * 4)), tspan(dout, T, a->hq, a->dv, lay.dout, 2)};
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
  const bool fu = fused(a);
  const bool tp = two_pass(a);
  const bool wide_det = !tp && !fu && wide_two_pass(a);
  // fp32 dQ accumulator: the single-pass route and wide heads on the reduce-add route
  float* dq_acc = (tp || wide_det) ? nullptr : c.take<float>((size_t)a->total_tokens * a->hq * a->dqk);
  float* dg_row = (a->log_gate || a->sink) ? c.take<float>(ht) : nullptr;
  float* dg_col = a->log_gate ? c.take<float>(ht) : nullptr;
  const int n_qtiles = (a->total_tokens + 63) / 64 + a->num_seqs;
  float* vecp = c.take<float>((size_t)a->hq * n_qtiles * 128);
  int32_t* cu_chk = chk ? c.take<int32_t>((size_t)a->num_seqs + 1) : nullptr;

  BwdMaps maps;
  const int T = a->total_tokens;
  if (!make_map(&maps.q, a->q, a->dqk, a->hq, T, lay.q, 64) ||
      !make_map(&maps.k, a->k, a->dqk, a->hkv, T, lay.k, 128) ||
      !make_map(&maps.v, a->v, a->dv, a->hkv, T, lay.v, 128) ||
      !make_map(&maps.dout, dout, a->dv, a->hq, T, lay.dout, 64) ||
      !make_map(&maps.q128, a->q, a->dqk, a->hq, T, lay.q, 128) ||
      !make_map(&maps.dout128, dout, a->dv, a->hq, T, lay.dout, 128))
    return GCS_ERR_CUDA;
  std::memset(&maps.dq_acc, 0, sizeof(maps.dq_acc));
  if (fu && !make_map_f32(&maps.dq_acc, dq_acc, a->dqk, a->hq, T, 128)) return GCS_ERR_CUDA;

  const int32_t* cu = a->cu_seqlens;
  if (cu_chk) {
    st = cuda_status(launch_check_prefill(a->cu_seqlens, a->num_seqs, a->total_tokens, a->max_seqlen, cu_chk, status, s));
    if (st != GCS_OK) return st;
    cu = cu_chk;
  }
  PreArgs pre{};
  pre.o = static_cast<const uint16_t*>(o);
  pre.dout = static_cast<const uint16_t*>(dout);
  pre.total = a->total_tokens;
  pre.hq = a->hq;
  pre.dv = a->dv;
  pre.dqk = a->dqk;
  pre.o_ts = lay.o.ts;
  pre.o_hs = lay.o.hs;
  pre.do_ts = lay.dout.ts;
  pre.do_hs = lay.dout.hs;
  pre.delta = delta;
  pre.dq_acc = dq_acc;
  pre.dg_row = dg_row;
  pre.dg_col = dg_col;
  pre.g = a->log_gate;
  pre.cu = cu;
  pre.num_seqs = a->num_seqs;
  pre.gT = gT;
  st = cuda_status(launch_bwd_pre(pre, s));
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
  p.dq_ts = lay.dq.ts;
  p.dq_hs = lay.dq.hs;
  p.dk_ts = lay.dk.ts;
  p.dk_hs = lay.dk.hs;
  p.dv_ts = lay.dv.ts;
  p.dv_hs = lay.dv.hs;
  p.dq_acc = dq_acc;
  p.dg_row = dg_row;
  p.dg_col = dg_col;
  p.vecp = vecp;
  p.n_qtiles = n_qtiles;
  p.status = status;
  const int num_tiles = (a->total_tokens + 127) / 128 + a->num_seqs;
  KernelTimer timer(s);
  if (fu) {
    timer.before();
    st = cuda_status(launch_prefill_bwd_fused(p, maps, num_tiles, s));
    timer.after();
  } else if (tp) {
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
  PostArgs post{};
  post.dq_acc = dq_acc;
  post.dq = static_cast<uint16_t*>(dq);
  post.total = a->total_tokens;
  post.hq = a->hq;
  post.dqk = a->dqk;
  post.dq_ts = lay.dq.ts;
  post.dq_hs = lay.dq.hs;
  post.cu = cu;
  post.num_seqs = a->num_seqs;
  post.dg_row = dg_row;
  post.dg_col = dg_col;
  post.dlog_gate = dlog_gate;
  post.lse = lse;
  post.delta = delta;
  post.sink = a->sink;
  post.dsink = dsink;
  return cuda_status(launch_bwd_post(post, s));
}

// Byte strides of the paged caches; all-zero element strides = contiguous
// [num_blocks, hkv, block_size, d].
static int cache_layout(const gcs_decode_args* a, CacheLayout* l) {
  const long long elt = a->kv_format == GCS_KV_BF16 ? 2 : 1;
  const long long row = (long long)a->d * elt;
  if (a->kv_stride_block == 0 && a->kv_stride_head == 0 && a->kv_stride_slot == 0) {
    *l = CacheLayout{(long long)a->hkv * a->block_size * row, (long long)a->block_size * row, row};
    return GCS_OK;
  }
  if (a->kv_stride_block < 0 || a->kv_stride_head < 0 || a->kv_stride_slot < 0) return GCS_ERR_INVALID_ARG;
  const long long b = a->kv_stride_block * elt, h = a->kv_stride_head * elt, sl = a->kv_stride_slot * elt;
  if ((b % 16) || (h % 16) || (sl % 16) || b >= (1LL << 40)) return GCS_ERR_UNSUPPORTED;
  const bool slot_inner = sl >= row && h >= (long long)a->block_size * sl;
  const bool head_inner = h >= row && sl >= (long long)a->hkv * h;
  if (!slot_inner && !head_inner) return GCS_ERR_UNSUPPORTED;
  if (b < (long long)(a->hkv - 1) * h + (long long)(a->block_size - 1) * sl + row) return GCS_ERR_UNSUPPORTED;
  *l = CacheLayout{b, h, sl};
  return GCS_OK;
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
  // head dim 128; GQA groups of 16 or 8 query heads; blocks of whole 16-token pages
  if (a->d != 128 || (a->hq != 16 * a->hkv && a->hq != 8 * a->hkv)) return GCS_ERR_UNSUPPORTED;
  // cache blocks of 16 x 2^k tokens (16, 32, 64, 128, ...)
  if (a->block_size < 16 || a->block_size > 4096 || (a->block_size & (a->block_size - 1)) != 0)
    return GCS_ERR_UNSUPPORTED;
  if (a->segment_len % 16 != 0) return GCS_ERR_UNSUPPORTED;
  if ((long long)a->max_blocks_per_req * a->block_size < a->max_seq_len) return GCS_ERR_INVALID_ARG;
  if (!aligned16(a->k_cache) || !aligned16(a->v_cache) || !aligned16(a->q)) return GCS_ERR_INVALID_ARG;
  if (a->window < 0) return GCS_ERR_INVALID_ARG;
  if (a->g_cache && !aligned16(a->g_cache)) return GCS_ERR_INVALID_ARG;
  if (a->sink && (reinterpret_cast<uintptr_t>(a->sink) & 3u)) return GCS_ERR_INVALID_ARG;
  if ((double)a->num_blocks * a->hkv * a->block_size * a->d > 9.0e15) return GCS_ERR_UNSUPPORTED;
  CacheLayout cl;
  int st = cache_layout(a, &cl);
  if (st != GCS_OK) return st;
  Layout lq, lo;
  if ((st = resolve_layout(a->q_stride, a->hq, a->d, &lq)) != GCS_OK) return st;
  return resolve_layout(a->out_stride, a->hq, a->d, &lo);
}

// True when the output of a paged call overlaps one of its inputs.
static bool paged_out_overlaps(const gcs_decode_args* a, const void* out) {
  const size_t rows = (size_t)a->num_blocks * a->hkv * a->block_size;
  const size_t elt = a->kv_format == GCS_KV_BF16 ? 2 : 1;
  const size_t sc = a->scale_mode == GCS_SCALE_PER_TENSOR ? 4 : rows * 4;
  CacheLayout cl;
  Layout lq, lo;
  cache_layout(a, &cl);
  resolve_layout(a->q_stride, a->hq, a->d, &lq);
  resolve_layout(a->out_stride, a->hq, a->d, &lo);
  const size_t cache_bytes = (size_t)(a->num_blocks - 1) * cl.bs + (size_t)(a->hkv - 1) * cl.hs +
                             (size_t)(a->block_size - 1) * cl.ss + (size_t)a->d * elt;
  const TSpan outs[] = {tspan(out, a->total_q, a->hq, a->d, lo, 2)};
  const TSpan ins[] = {tspan(a->q, a->total_q, a->hq, a->d, lq, 2),
                       tspan(span(a->k_cache, cache_bytes)),
                       tspan(span(a->v_cache, cache_bytes)),
                       tspan(span(a->k_scale, sc)),
                       tspan(span(a->v_scale, sc)),
                       tspan(span(a->block_table, (size_t)a->num_reqs * a->max_blocks_per_req * 4)),
                       tspan(span(a->seq_lens, (size_t)a->num_reqs * 4)),
                       tspan(span(a->cu_q, ((size_t)a->num_reqs + 1) * 4)),
                       tspan(span(a->g_cache, (size_t)a->num_blocks * a->hq * a->block_size * 4)),
                       tspan(span(a->sink, (size_t)a->hq * 4))};
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
  CacheLayout cl;
  Layout lq, lo;
  cache_layout(a, &cl);
  resolve_layout(a->q_stride, a->hq, a->d, &lq);
  resolve_layout(a->out_stride, a->hq, a->d, &lo);
  p.q_ts = lq.ts;
  p.q_hs = lq.hs;
  p.out_ts = lo.ts;
  p.out_hs = lo.hs;
  p.kv_bs = cl.bs;
  p.kv_hs = cl.hs;
  p.kv_ss = cl.ss;
  p.kv_head_inner = cl.head_inner() ? 1 : 0;
  p.block_size = a->block_size;
  p.log2_block_pages = 0;
  while ((16 << p.log2_block_pages) < a->block_size) ++p.log2_block_pages;
  p.group = a->hq / a->hkv;
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
static PagedOperandCheck operand_check(const gcs_decode_args* a) {
  PagedOperandCheck c{};
  if (a->kv_format != GCS_KV_FP8_E4M3) return c;  // hkv 0: nothing to check
  Layout lq;
  resolve_layout(a->q_stride, a->hq, a->d, &lq);
  c.q = static_cast<const uint16_t*>(a->q);
  c.q_ts = lq.ts;
  c.q_hs = lq.hs;
  c.hq = a->hq;
  c.d = a->d;
  c.hkv = a->hkv;
  c.v_scale = a->v_scale;
  c.per_tensor = a->scale_mode == GCS_SCALE_PER_TENSOR ? 1 : 0;
  return c;
}

static int paged_checks(const gcs_decode_args* a, void* workspace, size_t off, DecodeParams& p, cudaStream_t s) {
  int32_t* cu_chk = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + off);
  const int st = cuda_status(launch_check_paged(a->cu_q, a->seq_lens, a->block_table, a->num_reqs, a->total_q,
                                                a->max_q_len, a->max_seq_len, a->max_blocks_per_req, a->num_blocks,
                                                a->block_size, a->window, operand_check(a), cu_chk, p.status, s));
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
  p.seg_pages = a->segment_len / 16;
  p.part_acc = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + round_up(units * rows * 128 * sizeof(float)));
  DecodeMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (a->kv_format == GCS_KV_FP8_E4M3) {
    CacheLayout cl;
    cache_layout(a, &cl);
    if (!make_page_map_u8(&maps.k, a->k_cache, a->num_blocks, a->hkv, a->block_size, cl) ||
        !make_page_map_u8(&maps.v, a->v_cache, a->num_blocks, a->hkv, a->block_size, cl))
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
  CacheLayout cl;
  cache_layout(a, &cl);
  if (!make_page_map_u8(&maps.k, a->k_cache, a->num_blocks, a->hkv, a->block_size, cl) ||
      !make_page_map_u8(&maps.v, a->v_cache, a->num_blocks, a->hkv, a->block_size, cl))
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
                                        a->window, operand_check(a), nullptr, status,
                                        reinterpret_cast<cudaStream_t>(stream)));
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
