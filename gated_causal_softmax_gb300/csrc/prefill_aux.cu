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
#include <algorithm>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace gcs {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
// One block per (sequence, head) scans 8192 tokens per pass: sequences up to that length take
// one pass of independent loads (the scans are latency-bound), longer ones carry the running
// total between passes.
constexpr int kScanThreads = 1024;
constexpr int kScanPer = 8;

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

// L = min(32, dv / 8) lanes per (token, head) row, 8 elements (16 B of O and of dO) per lane
// and chunk; each warp takes 32 / L consecutive rows at a time, grid-stride.  The loop is
// uniform across the warp (rows past the end load nothing), so the shuffles see every lane.
// O and dO rows sit at token * ts + head * hs (element strides; dims contiguous).
template <int L>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t* __restrict__ o,
                                                      const uint16_t* __restrict__ dout, int total, int hq, int dv,
                                                      long long o_ts, long long o_hs, long long do_ts,
                                                      long long do_hs, float* __restrict__ delta) {
  constexpr int kRowsPerWarp = 32 / L;
  const int lane = threadIdx.x & (L - 1);
  const int group = (threadIdx.x & 31) / L;
  const int rows = total * hq;
  const int chunks = dv / (8 * L);
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int row0 = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kRowsPerWarp; row0 < rows;
       row0 += warps * kRowsPerWarp) {
    const int row = row0 + group;
    const bool valid = row < rows;
    float acc0 = 0.f, acc1 = 0.f;
    if (valid) {
      const long long t = row / hq, h = row % hq;
      const uint4* po = reinterpret_cast<const uint4*>(o + t * o_ts + h * o_hs);
      const uint4* pd = reinterpret_cast<const uint4*>(dout + t * do_ts + h * do_hs);
      for (int c = 0; c < chunks; ++c) {
        const uint4 a = __ldg(po + c * L + lane), b = __ldg(pd + c * L + lane);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc0 = fmaf(__uint_as_float(aw[k] << 16), __uint_as_float(bw[k] << 16), acc0);
          acc1 = fmaf(__uint_as_float(aw[k] & 0xffff0000u), __uint_as_float(bw[k] & 0xffff0000u), acc1);
        }
      }
    }
    float acc = acc0 + acc1;
#pragma unroll
    for (int off = L / 2; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, L);
    if (valid && lane == 0) {
      const int t = row / hq, h = row % hq;
      delta[(size_t)h * total + t] = acc;
    }
  }
}

// fp32 dQ accumulator [total, hq, dqk] (contiguous) -> bf16 dQ at token * ts + head * hs.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float4* __restrict__ src, uint16_t* __restrict__ dst,
                                                         size_t n4, int hq, int dqk, long long ts, long long hs) {
  const int q4 = dqk / 4;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const float4 v = src[i];
    const size_t rh = i / q4;
    const long long d = (long long)(i % q4) * 4, h = (long long)(rh % hq), t = (long long)(rh / hq);
    *reinterpret_cast<uint2*>(dst + t * ts + h * hs + d) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
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

// grid (hq), 1024 threads: dsink_h = -sum_i p_i (rowsum_i + delta_i (1 - p_i)), p_i = e^{sigma_h - lse_i};
// four independent rows per thread and iteration keep loads in flight.  One block per head
// sums in a fixed order, so the result does not depend on scheduling.
__global__ void __launch_bounds__(1024) dsink_kernel(const float* __restrict__ row, const float* __restrict__ lse,
                                                     const float* __restrict__ delta, const float* __restrict__ sink,
                                                     int total, float* __restrict__ dsink) {
  __shared__ float red[32];
  const int h = blockIdx.x;
  const float sig = __ldg(sink + h);
  const float* rr = row + (size_t)h * total;
  const float* ll = lse + (size_t)h * total;
  const float* dd = delta + (size_t)h * total;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int base = 0; base < total; base += 4 * 1024) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = base + u * 1024 + threadIdx.x;
      if (t < total) {
        const float ps = __expf(sig - __ldg(ll + t));
        acc[u] += ps * (__ldg(rr + t) + __ldg(dd + t) * (1.f - ps));
      }
    }
  }
  float a = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
  for (int off = 16; off; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x < 32) {
    a = red[threadIdx.x];
#pragma unroll
    for (int off = 16; off; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
    if (threadIdx.x == 0) dsink[h] = -a;
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

cudaError_t launch_bwd_pre(const uint16_t* o, const uint16_t* dout, int total, int hq, int dv, int dqk,
                           long long o_ts, long long o_hs, long long do_ts, long long do_hs, float* delta,
                           float* dq_acc, float* dg_row, float* dg_col, cudaStream_t s) {
  // enough blocks to fill the GPU several times over; rows are grid-stride
  const int L = dv >= 256 ? 32 : dv / 8;
  const long long lanes = (long long)total * hq * L;
  const int blocks = (int)std::min<long long>((lanes + 255) / 256, 152 * 16);
  if (L == 8) bwd_pre_kernel<8><<<blocks, 256, 0, s>>>(o, dout, total, hq, dv, o_ts, o_hs, do_ts, do_hs, delta);
  else if (L == 16) bwd_pre_kernel<16><<<blocks, 256, 0, s>>>(o, dout, total, hq, dv, o_ts, o_hs, do_ts, do_hs, delta);
  else bwd_pre_kernel<32><<<blocks, 256, 0, s>>>(o, dout, total, hq, dv, o_ts, o_hs, do_ts, do_hs, delta);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (dq_acc) e = cudaMemsetAsync(dq_acc, 0, (size_t)total * hq * dqk * sizeof(float), s);
  if (e != cudaSuccess) return e;
  if (dg_row) e = cudaMemsetAsync(dg_row, 0, (size_t)total * hq * sizeof(float), s);
  if (e != cudaSuccess) return e;
  if (dg_col) e = cudaMemsetAsync(dg_col, 0, (size_t)total * hq * sizeof(float), s);
  return e;
}

cudaError_t launch_bwd_post(const float* dq_acc, uint16_t* dq, int total, int hq, int dqk, long long dq_ts,
                            long long dq_hs, const int32_t* cu, int num_seqs, const float* dg_row,
                            const float* dg_col, float* dlog_gate, const float* lse, const float* delta,
                            const float* sink, float* dsink, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if (dq_acc) {
    const size_t n4 = (size_t)total * hq * dqk / 4;
    const int blocks = (int)((n4 + 255) / 256 < 152 * 16 ? (n4 + 255) / 256 : 152 * 16);
    dq_convert_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(dq_acc), dq, n4, hq, dqk, dq_ts,
                                             dq_hs);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (dlog_gate) {
    dgate_kernel<<<dim3(num_seqs, hq), kScanThreads, 0, s>>>(dg_row, dg_col, cu, total, hq, dlog_gate);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (dsink) {
    dsink_kernel<<<hq, 1024, 0, s>>>(dg_row, lse, delta, sink, total, dsink);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace gcs
