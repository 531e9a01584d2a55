// Small bandwidth-bound kernels around the prefill attention kernels.
//
//   gate_cumsum   G_t = sum of log gates from the sequence start to t (inclusive), per
//                 query head; written transposed [hq, total] and pre-multiplied by
//                 log2(e) for the exp2-based softmax.  (fla-org/flash-linear-attention
//                 #1322, Description: logarithmic gates.)
//   bwd_pre       delta_i = sum_d dO_id * O_id in fp32 from the stored bf16 output;
//                 zeroes the fp32 dQ accumulator and the dS row / column sums.
//   bwd_post      dQ = bf16(dQ_acc) (Oct 5 comment: fp32 buffer converted after the
//                 kernel); d log_gate = reverse cumsum of (rowsum dS - colsum dS);
//                 d sink_h = -sum_i p_sink,i * sum_j P_ij dP_ij (Oct 3 comment), where the
//                 fp32 row sum sum_j P_ij dP_ij is recovered exactly from the fp32 row sum
//                 of dS:  sum_j P_ij dP_ij = sum_j dS_ij + delta_i * (1 - p_sink,i).
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace gcs {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kScanThreads = 256;
constexpr int kScanPer = 4;

// Block-wide inclusive scan of one value per thread; returns the inclusive prefix and
// writes the block total into *total.
__device__ __forceinline__ float block_scan(float x, float* warp_sums, float* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  float before = 0.f, all = 0.f;
  for (int w = 0; w < kScanThreads / 32; ++w) {
    const float s = warp_sums[w];
    if (w < warp) before += s;
    all += s;
  }
  __syncthreads();
  *total = all;
  return x + before;
}

// grid (num_seqs, hq)
__global__ void __launch_bounds__(kScanThreads) gate_cumsum_kernel(const float* __restrict__ g,
                                                                   const int32_t* __restrict__ cu, int total, int hq,
                                                                   float* __restrict__ gT) {
  __shared__ float warp_sums[kScanThreads / 32];
  const int s = blockIdx.x, h = blockIdx.y;
  const int a = __ldg(cu + s), b = __ldg(cu + s + 1);
  float carry = 0.f;
  for (int base = a; base < b; base += kScanThreads * kScanPer) {
    float v[kScanPer];
    float local = 0.f;
#pragma unroll
    for (int u = 0; u < kScanPer; ++u) {
      const int t = base + threadIdx.x * kScanPer + u;
      local += (t < b) ? __ldg(g + (size_t)t * hq + h) : 0.f;
      v[u] = local;
    }
    float chunk_total;
    const float incl = block_scan(local, warp_sums, &chunk_total);
    const float excl = carry + incl - local;
#pragma unroll
    for (int u = 0; u < kScanPer; ++u) {
      const int t = base + threadIdx.x * kScanPer + u;
      if (t < b) gT[(size_t)h * total + t] = (excl + v[u]) * kLog2e;
    }
    carry += chunk_total;
  }
}

// one warp per (token, head) row
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t* __restrict__ o,
                                                      const uint16_t* __restrict__ dout, int total, int hq, int dv,
                                                      float* __restrict__ delta) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= total * hq) return;
  const uint4* po = reinterpret_cast<const uint4*>(o + (size_t)row * dv);
  const uint4* pd = reinterpret_cast<const uint4*>(dout + (size_t)row * dv);
  float acc = 0.f;
  for (int c = lane; c < dv / 8; c += 32) {
    const uint4 a = __ldg(po + c), b = __ldg(pd + c);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc = fmaf(__uint_as_float(aw[k] << 16), __uint_as_float(bw[k] << 16), acc);
      acc = fmaf(__uint_as_float(aw[k] & 0xffff0000u), __uint_as_float(bw[k] & 0xffff0000u), acc);
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    const int t = row / hq, h = row % hq;
    delta[(size_t)h * total + t] = acc;
  }
}

__global__ void __launch_bounds__(256) dq_convert_kernel(const float4* __restrict__ src, uint2* __restrict__ dst,
                                                         size_t n4) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const float4 v = src[i];
    dst[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}

// grid (num_seqs, hq): dg_t = sum_{u >= t} (row_u - col_u), scanned from the sequence end.
__global__ void __launch_bounds__(kScanThreads) dgate_kernel(const float* __restrict__ row,
                                                             const float* __restrict__ col,
                                                             const int32_t* __restrict__ cu, int total, int hq,
                                                             float* __restrict__ dg) {
  __shared__ float warp_sums[kScanThreads / 32];
  const int s = blockIdx.x, h = blockIdx.y;
  const int a = __ldg(cu + s), b = __ldg(cu + s + 1);
  const float* rr = row + (size_t)h * total;
  const float* cc = col + (size_t)h * total;
  float carry = 0.f;
  // walk backwards: element k of the reversed sequence is token b - 1 - k
  for (int base = 0; base < b - a; base += kScanThreads * kScanPer) {
    float v[kScanPer];
    float local = 0.f;
#pragma unroll
    for (int u = 0; u < kScanPer; ++u) {
      const int k = base + threadIdx.x * kScanPer + u;
      const int t = b - 1 - k;
      local += (t >= a) ? (rr[t] - cc[t]) : 0.f;
      v[u] = local;
    }
    float chunk_total;
    const float incl = block_scan(local, warp_sums, &chunk_total);
    const float excl = carry + incl - local;
#pragma unroll
    for (int u = 0; u < kScanPer; ++u) {
      const int k = base + threadIdx.x * kScanPer + u;
      const int t = b - 1 - k;
      if (t >= a) dg[(size_t)t * hq + h] = excl + v[u];
    }
    carry += chunk_total;
  }
}

// grid (hq): dsink_h = -sum_i p_i (rowsum_i + delta_i (1 - p_i)), p_i = e^{sigma_h - lse_i}
__global__ void __launch_bounds__(256) dsink_kernel(const float* __restrict__ row, const float* __restrict__ lse,
                                                    const float* __restrict__ delta, const float* __restrict__ sink,
                                                    int total, float* __restrict__ dsink) {
  __shared__ float red[8];
  const int h = blockIdx.x;
  const float sig = __ldg(sink + h);
  float acc = 0.f;
  for (int t = threadIdx.x; t < total; t += blockDim.x) {
    const size_t i = (size_t)h * total + t;
    const float ps = __expf(sig - lse[i]);
    acc += ps * (row[i] + delta[i] * (1.f - ps));
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += red[w];
    dsink[h] = -s;
  }
}

// grid (query tiles of 64 rows over all sequences, hq), 64 threads: packs the per-column
// vectors the fused backward reads per step, [h][tile][0..63] = (G_i - LSE_i) * log2 e,
// [64..127] = delta_i, so one aligned 512-B bulk copy fetches them.
__global__ void __launch_bounds__(64) bwd_pack_kernel(const int32_t* __restrict__ cu, int num_seqs, int total,
                                                      const float* __restrict__ lse, const float* __restrict__ gT,
                                                      const float* __restrict__ delta, float* __restrict__ vecp) {
  int t = blockIdx.x;
  int start = -1, len = 0, local = 0;
  for (int s = 0; s < num_seqs; ++s) {
    const int a = __ldg(cu + s), b = __ldg(cu + s + 1);
    const int n = (b - a + 63) / 64;
    if (t < n) {
      start = a;
      len = b - a;
      local = t;
      break;
    }
    t -= n;
  }
  // tiles past the last sequence are zero-filled: a 128-row consumer step may read one
  const int h = blockIdx.y;
  const int i = local * 64 + threadIdx.x;
  float colterm = 0.f, dl = 0.f;
  if (start >= 0 && i < len) {
    const size_t idx = (size_t)h * total + start + i;
    colterm = -__ldg(lse + idx) * kLog2e;
    if (gT) colterm += __ldg(gT + idx);
    dl = __ldg(delta + idx);
  }
  float* dst = vecp + ((size_t)h * gridDim.x + blockIdx.x) * 128;
  dst[threadIdx.x] = colterm;
  dst[64 + threadIdx.x] = dl;
}

}  // namespace

cudaError_t launch_bwd_pack(const int32_t* cu, int num_seqs, int total, int hq, int n_qtiles, const float* lse,
                            const float* gT, const float* delta, float* vecp, cudaStream_t s) {
  bwd_pack_kernel<<<dim3(n_qtiles, hq), 64, 0, s>>>(cu, num_seqs, total, lse, gT, delta, vecp);
  return cudaGetLastError();
}

cudaError_t launch_gate_cumsum(const float* g, const int32_t* cu, int num_seqs, int total, int hq, float* gT,
                               cudaStream_t s) {
  gate_cumsum_kernel<<<dim3(num_seqs, hq), kScanThreads, 0, s>>>(g, cu, total, hq, gT);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const uint16_t* o, const uint16_t* dout, int total, int hq, int dv, int dqk, float* delta,
                           float* dq_acc, float* dg_row, float* dg_col, cudaStream_t s) {
  const int rows = total * hq;
  bwd_pre_kernel<<<(rows + 7) / 8, 256, 0, s>>>(o, dout, total, hq, dv, delta);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (dq_acc) e = cudaMemsetAsync(dq_acc, 0, (size_t)total * hq * dqk * sizeof(float), s);
  if (e != cudaSuccess) return e;
  if (dg_row) e = cudaMemsetAsync(dg_row, 0, (size_t)total * hq * sizeof(float), s);
  if (e != cudaSuccess) return e;
  if (dg_col) e = cudaMemsetAsync(dg_col, 0, (size_t)total * hq * sizeof(float), s);
  return e;
}

cudaError_t launch_bwd_post(const float* dq_acc, uint16_t* dq, int total, int hq, int dqk, const int32_t* cu,
                            int num_seqs, const float* dg_row, const float* dg_col, float* dlog_gate,
                            const float* lse, const float* delta, const float* sink, float* dsink, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if (dq_acc) {
    const size_t n4 = (size_t)total * hq * dqk / 4;
    const int blocks = (int)((n4 + 255) / 256 < 152 * 16 ? (n4 + 255) / 256 : 152 * 16);
    dq_convert_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(dq_acc), reinterpret_cast<uint2*>(dq),
                                             n4);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (dlog_gate) {
    dgate_kernel<<<dim3(num_seqs, hq), kScanThreads, 0, s>>>(dg_row, dg_col, cu, total, hq, dlog_gate);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (dsink) {
    dsink_kernel<<<hq, 256, 0, s>>>(dg_row, lse, delta, sink, total, dsink);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace gcs
