// Device-content checks of the index arrays a call reads (a library diagnostic with no
// counterpart in the pages).  The host cannot read cu_seqlens, cu_q, seq_lens or the page
// table without synchronising, so one CTA reads them on the call's stream, before the call's
// kernels, and checks the preconditions the public header states for them.
//
// The CTA also writes the array of cumulative lengths (cu_seqlens or cu_q) that the call's
// kernels then read in place of the caller's: a copy when every check holds, and all zeros
// (an empty batch) when one fails, in which case it records kDevInvalidArg in the device
// status word.  In an empty batch every prefill tile and every paged request has no rows, so
// no kernel reads through an index taken from these arrays (the kernels that sweep every
// token, such as the backward's delta, stay within total_tokens, which the host checked).
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace gcs {
namespace {

constexpr int kCheckThreads = 1024;

// Combines the threads' verdicts, records a failure and writes the copy (cu_out may be null).
__device__ __forceinline__ void finish_check(bool bad_here, int* bad_s, const int32_t* cu, int n1,
                                             int32_t* cu_out, int* status) {
  if (bad_here) atomicOr(bad_s, 1);
  __syncthreads();
  const bool bad = *bad_s != 0;
  if (bad && threadIdx.x == 0) atomicCAS(status, kDevOk, kDevInvalidArg);
  if (cu_out)
    for (int i = threadIdx.x; i < n1; i += blockDim.x) cu_out[i] = bad ? 0 : __ldg(cu + i);
}

// cu_seqlens: starts at 0, ends at total, and every length lies in 0 .. max_seqlen.
__global__ void __launch_bounds__(kCheckThreads) check_prefill_kernel(const int32_t* __restrict__ cu, int num_seqs,
                                                                      int total, int max_seqlen,
                                                                      int32_t* __restrict__ cu_out, int* status) {
  __shared__ int bad_s;
  if (threadIdx.x == 0) bad_s = 0;
  __syncthreads();
  bool bad = false;
  if (threadIdx.x == 0) bad = __ldg(cu) != 0 || __ldg(cu + num_seqs) != total;
  for (int s = threadIdx.x; s < num_seqs; s += blockDim.x) {
    const long long len = (long long)__ldg(cu + s + 1) - __ldg(cu + s);
    bad = bad || len < 0 || len > max_seqlen;
  }
  finish_check(bad, &bad_s, cu, num_seqs + 1, cu_out, status);
}

// cu_q starts at 0 and ends at total_q; request r has 0 <= q_len <= max_q_len query rows and
// q_len <= seq_len <= max_seq_len cached tokens; the page-table entries of the pages the
// paged calls can read for it lie in [0, num_blocks).  Those pages run from the 128-key tile
// that holds the earliest key any of its query rows sees (key 0 without a window) to the
// page of its last cached token; a request with no query rows reads none.  One warp per
// request, one lane per page.
//
// With an fp8 cache (f16 operands, fp8.hkv > 0) it also checks the operand limits: every |q| at
// most 65504 (q, strided, is read in 16-byte units) and every V scale of the slots below
// seq_len in those pages below 255 in magnitude (per tensor: the one scale).
__global__ void __launch_bounds__(kCheckThreads) check_paged_kernel(
    const int32_t* __restrict__ cu_q, const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ table,
    int num_reqs, int total_q, int max_q_len, int max_seq_len, int max_blocks, int num_blocks, int block_size,
    int window, PagedOperandCheck fp8, int32_t* __restrict__ cu_out, int* status) {
  __shared__ int bad_s;
  if (threadIdx.x == 0) bad_s = 0;
  __syncthreads();
  bool bad = false;
  if (threadIdx.x == 0) bad = __ldg(cu_q) != 0 || __ldg(cu_q + num_reqs) != total_q;
  if (fp8.hkv > 0) {
    // q: total_q x hq rows of d / 8 16-byte units
    const int units = fp8.d / 8;
    const long long n = (long long)total_q * fp8.hq * units;
    for (long long i = threadIdx.x; i < n; i += blockDim.x) {
      const long long row = i / units, t = row / fp8.hq, h = row % fp8.hq;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(fp8.q + t * fp8.q_ts + h * fp8.q_hs) + i % units);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // bf16 magnitude bits above 65504 (0x477fe0), NaN included
        bad = bad || (w[k] & 0x7fffu) > 0x477fu || (w[k] >> 16 & 0x7fffu) > 0x477fu;
      }
    }
    if (fp8.per_tensor && threadIdx.x == 0) bad = bad || !(fabsf(__ldg(fp8.v_scale)) < 255.f);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int r = warp; r < num_reqs; r += nwarps) {
    const long long ql = (long long)__ldg(cu_q + r + 1) - __ldg(cu_q + r);
    const int L = __ldg(seq_lens + r);
    if (ql < 0 || ql > max_q_len || L < ql || L > max_seq_len) {
      bad = true;
      continue;
    }
    if (ql == 0) continue;
    const int first_key = window > 0 ? max(0, L - static_cast<int>(ql) - window + 1) : 0;
    const int p0 = (first_key / 128) * 128 / block_size;  // block holding the first key of that tile
    const int np = (L + block_size - 1) / block_size;  // <= max_blocks: L <= max_seq_len
    for (int pg = p0 + lane; pg < np; pg += 32) {
      const int blk = __ldg(table + (size_t)r * max_blocks + pg);
      bad = bad || blk < 0 || blk >= num_blocks;
      if (fp8.hkv > 0 && !fp8.per_tensor && blk >= 0 && blk < num_blocks) {
        const int nslot = min(block_size, L - pg * block_size);
        for (int h = 0; h < fp8.hkv; ++h)
          for (int sl = 0; sl < nslot; ++sl)
            bad = bad || !(fabsf(__ldg(fp8.v_scale + ((size_t)blk * fp8.hkv + h) * block_size + sl)) < 255.f);
      }
    }
  }
  finish_check(bad, &bad_s, cu_q, num_reqs + 1, cu_out, status);
}

}  // namespace

cudaError_t launch_check_prefill(const int32_t* cu, int num_seqs, int total, int max_seqlen, int32_t* cu_out,
                                 int* status, cudaStream_t s) {
  check_prefill_kernel<<<1, kCheckThreads, 0, s>>>(cu, num_seqs, total, max_seqlen, cu_out, status);
  return cudaGetLastError();
}

cudaError_t launch_check_paged(const int32_t* cu_q, const int32_t* seq_lens, const int32_t* table, int num_reqs,
                               int total_q, int max_q_len, int max_seq_len, int max_blocks, int num_blocks,
                               int block_size, int window, const PagedOperandCheck& fp8, int32_t* cu_out,
                               int* status, cudaStream_t s) {
  check_paged_kernel<<<1, kCheckThreads, 0, s>>>(cu_q, seq_lens, table, num_reqs, total_q, max_q_len, max_seq_len,
                                                 max_blocks, num_blocks, block_size, window, fp8, cu_out, status);
  return cudaGetLastError();
}

}  // namespace gcs
