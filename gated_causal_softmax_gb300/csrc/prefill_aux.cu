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

// G of sequence s, head h by one kScanThreads-thread block.
__device__ __forceinline__ void gate_cumsum_block(const float* __restrict__ g, const int32_t* __restrict__ cu,
                                                  int total, int hq, float* __restrict__ gT, int s, int h,
                                                  float* warp_sums) {
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

// grid (num_seqs, hq)
__global__ void __launch_bounds__(kScanThreads) gate_cumsum_kernel(const float* __restrict__ g,
                                                                   const int32_t* __restrict__ cu, int total, int hq,
                                                                   float* __restrict__ gT) {
  __shared__ float warp_sums[kScanThreads / 32];
  gate_cumsum_block(g, cu, total, hq, gT, blockIdx.x, blockIdx.y, warp_sums);
}

// L = min(32, dv / 8) lanes per (token, head) row, 8 elements (16 B of O and of dO) per lane
// and chunk; each warp takes 32 / L consecutive rows at a time, grid-stride over the role's
// blocks.  The loop is uniform across the warp (rows past the end load nothing), so the
// shuffles see every lane.  O and dO rows sit at token * ts + head * hs (element strides;
// dims contiguous).  The same lanes zero the row's fp32 dQ accumulator ([total, hq, dqk],
// contiguous) and its entries of the dS row and column sums ([hq, total]).
template <int L>
__device__ __forceinline__ void pre_rows(const PreArgs& a, int blk, int nblk) {
  constexpr int kRowsPerWarp = 32 / L;
  const int lane = threadIdx.x & (L - 1);
  const int group = (threadIdx.x & 31) / L;
  const int rows = a.total * a.hq;
  const int chunks = a.dv / (8 * L);
  const int warps = nblk * (blockDim.x >> 5);
  for (int row0 = (blk * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kRowsPerWarp; row0 < rows;
       row0 += warps * kRowsPerWarp) {
    const int row = row0 + group;
    const bool valid = row < rows;
    const int t = valid ? row / a.hq : 0, h = valid ? row % a.hq : 0;
    float acc0 = 0.f, acc1 = 0.f;
    if (valid) {
      const uint4* po = reinterpret_cast<const uint4*>(a.o + (long long)t * a.o_ts + (long long)h * a.o_hs);
      const uint4* pd = reinterpret_cast<const uint4*>(a.dout + (long long)t * a.do_ts + (long long)h * a.do_hs);
      for (int c = 0; c < chunks; ++c) {
        const uint4 x = __ldg(po + c * L + lane), y = __ldg(pd + c * L + lane);
        const uint32_t aw[4] = {x.x, x.y, x.z, x.w}, bw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc0 = fmaf(__uint_as_float(aw[k] << 16), __uint_as_float(bw[k] << 16), acc0);
          acc1 = fmaf(__uint_as_float(aw[k] & 0xffff0000u), __uint_as_float(bw[k] & 0xffff0000u), acc1);
        }
      }
      if (a.dq_acc) {
        float4* z = reinterpret_cast<float4*>(a.dq_acc + (size_t)row * a.dqk);
        for (int c = lane; c < a.dqk / 4; c += L) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float acc = acc0 + acc1;
#pragma unroll
    for (int off = L / 2; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, L);
    if (valid && lane == 0) {
      const size_t idx = (size_t)h * a.total + t;
      a.delta[idx] = acc;
      if (a.dg_row) a.dg_row[idx] = 0.f;
      if (a.dg_col) a.dg_col[idx] = 0.f;
    }
  }
}

// Blocks [0, n_scan): the gate cumsum of (sequence b / hq, head b % hq); the rest: delta and
// the zeroing above.  The two roles touch disjoint data, so one launch runs them side by side.
template <int L>
__global__ void __launch_bounds__(kScanThreads) bwd_pre_kernel(const PreArgs a) {
  __shared__ float warp_sums[kScanThreads / 32];
  if ((int)blockIdx.x < a.n_scan) {
    gate_cumsum_block(a.g, a.cu, a.total, a.hq, a.gT, blockIdx.x / a.hq, blockIdx.x % a.hq, warp_sums);
    return;
  }
  pre_rows<L>(a, blockIdx.x - a.n_scan, gridDim.x - a.n_scan);
}

// fp32 dQ accumulator [total, hq, dqk] (contiguous) -> bf16 dQ at token * ts + head * hs,
// grid-stride over the role's blocks.  Every prefill tensor holds fewer than 2^31 elements (a
// host check), so the element index fits 32 bits; head dims are powers of two, so the head-dim
// offset is a mask and one 32-bit division per float4 splits the row into (token, head).
__device__ __forceinline__ void dq_convert_range(const PostArgs& a, int blk, int nblk) {
  const float4* src = reinterpret_cast<const float4*>(a.dq_acc);
  const int lq4 = __ffs(a.dqk >> 2) - 1;  // log2(dqk / 4)
  const int n4 = static_cast<int>(a.n4);
  for (int i = blk * blockDim.x + threadIdx.x; i < n4; i += nblk * blockDim.x) {
    const float4 v = src[i];
    const int rh = i >> lq4;
    const int t = rh / a.hq, h = rh - t * a.hq;
    const int d = (i & ((1 << lq4) - 1)) * 4;
    *reinterpret_cast<uint2*>(a.dq + (long long)t * a.dq_ts + (long long)h * a.dq_hs + d) =
        make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}

// d log_gate of sequence s, head h: dg_t = sum_{u >= t} (row_u - col_u), scanned from the
// sequence end by one kScanThreads-thread block.
__device__ __forceinline__ void dgate_block(const PostArgs& a, int s, int h, float* warp_sums) {
  const int lo = __ldg(a.cu + s), hi = __ldg(a.cu + s + 1);
  const float* rr = a.dg_row + (size_t)h * a.total;
  const float* cc = a.dg_col + (size_t)h * a.total;
  float carry = 0.f;
  // walk backwards: element k of the reversed sequence is token hi - 1 - k
  for (int base = 0; base < hi - lo; base += kScanThreads * kScanPer) {
    float v[kScanPer];
    float local = 0.f;
#pragma unroll
    for (int u = 0; u < kScanPer; ++u) {
      const int k = base + threadIdx.x * kScanPer + u;
      const int t = hi - 1 - k;
      local += (t >= lo) ? (rr[t] - cc[t]) : 0.f;
      v[u] = local;
    }
    float chunk_total;
    const float incl = block_scan(local, warp_sums, &chunk_total);
    const float excl = carry + incl - local;
#pragma unroll
    for (int u = 0; u < kScanPer; ++u) {
      const int k = base + threadIdx.x * kScanPer + u;
      const int t = hi - 1 - k;
      if (t >= lo) a.dlog_gate[(size_t)t * a.hq + h] = excl + v[u];
    }
    carry += chunk_total;
  }
}

// dsink_h = -sum_i p_i (rowsum_i + delta_i (1 - p_i)), p_i = e^{sigma_h - lse_i}, by one
// 1024-thread block; four independent rows per thread and iteration keep loads in flight.
// One block per head sums in a fixed order, so the result does not depend on scheduling.
__device__ __forceinline__ void dsink_block(const PostArgs& a, int h, float* red) {
  const float sig = __ldg(a.sink + h);
  const float* rr = a.dg_row + (size_t)h * a.total;
  const float* ll = a.lse + (size_t)h * a.total;
  const float* dd = a.delta + (size_t)h * a.total;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int base = 0; base < a.total; base += 4 * 1024) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = base + u * 1024 + threadIdx.x;
      if (t < a.total) {
        const float ps = __expf(sig - __ldg(ll + t));
        acc[u] += ps * (__ldg(rr + t) + __ldg(dd + t) * (1.f - ps));
      }
    }
  }
  float x = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
  for (int off = 16; off; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  __syncthreads();
  if (threadIdx.x < 32) {
    x = red[threadIdx.x];
#pragma unroll
    for (int off = 16; off; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    if (threadIdx.x == 0) a.dsink[h] = -x;
  }
}

// Blocks [0, n_gate): d log_gate of (sequence b / hq, head b % hq); [n_gate, n_gate + n_sink):
// d sink of head b - n_gate; the rest: the dQ conversion.  The roles write disjoint outputs, so
// one launch runs the latency-bound scans beside the bandwidth-bound conversion.
__global__ void __launch_bounds__(1024) bwd_post_kernel(const PostArgs a) {
  __shared__ float sm[32];
  int b = blockIdx.x;
  if (b < a.n_gate) {
    dgate_block(a, b / a.hq, b % a.hq, sm);
    return;
  }
  b -= a.n_gate;
  if (b < a.n_sink) {
    dsink_block(a, b, sm);
    return;
  }
  dq_convert_range(a, b - a.n_sink, gridDim.x - a.n_gate - a.n_sink);
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

cudaError_t launch_bwd_pre(const PreArgs& args, cudaStream_t s) {
  PreArgs a = args;
  a.n_scan = a.gT ? a.num_seqs * a.hq : 0;
  // enough row blocks to fill the GPU several times over; rows are grid-stride
  const int L = a.dv >= 256 ? 32 : a.dv / 8;
  const long long lanes = (long long)a.total * a.hq * L;
  const int blocks = a.n_scan + (int)std::min<long long>((lanes + kScanThreads - 1) / kScanThreads, 152 * 4);
  if (L == 8) bwd_pre_kernel<8><<<blocks, kScanThreads, 0, s>>>(a);
  else if (L == 16) bwd_pre_kernel<16><<<blocks, kScanThreads, 0, s>>>(a);
  else bwd_pre_kernel<32><<<blocks, kScanThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_post(const PostArgs& args, cudaStream_t s) {
  PostArgs a = args;
  a.n4 = a.dq_acc ? (size_t)a.total * a.hq * a.dqk / 4 : 0;
  a.n_gate = a.dlog_gate ? a.num_seqs * a.hq : 0;
  a.n_sink = a.dsink ? a.hq : 0;
  const int n_conv = (int)std::min<size_t>((a.n4 + 1023) / 1024, 152 * 4);
  const int blocks = a.n_gate + a.n_sink + n_conv;
  if (blocks == 0) return cudaSuccess;
  bwd_post_kernel<<<blocks, 1024, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace gcs
