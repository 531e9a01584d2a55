// Work ordering for the causal prefill kernels.
//
// A causal tile's cost grows with its distance from the sequence start (forward: query
// tile q sees q + 1 key tiles) or from the sequence end (backward: key tile j is seen by
// the query tiles after it).  CTAs are dispatched in blockIdx order as SMs free up, so
// handing out tiles heaviest-first (longest-processing-time order) keeps the last wave
// short.  Tile "weight" u: 0 for the lightest tile of a sequence, n_s - 1 for the
// heaviest, where n_s = ceil(len_s / rows).  Rank r (blockIdx.x) maps to the r-th tile in
// order of u descending, ties by sequence index.
#pragma once

#include <cstdint>

namespace gcs {

constexpr int kLptMaxSeqs = 64;  // beyond this, plain sequence order (the search is O(num_seqs))

struct TileRef {
  int start;  // first token of the sequence
  int len;    // sequence length
  int u;      // weight rank inside the sequence (0 = lightest)
  int n;      // tiles in the sequence
  int seq;    // sequence index
};

__device__ __forceinline__ int lpt_count_ge(const int32_t* cu, int num_seqs, int rows, int q) {
  int c = 0;
  for (int s = 0; s < num_seqs; ++s) {
    const int n = (__ldg(cu + s + 1) - __ldg(cu + s) + rows - 1) / rows;
    c += n > q ? n - q : 0;
  }
  return c;
}

// Returns false when r is past the last tile.
__device__ __forceinline__ bool lpt_tile(const int32_t* cu, int num_seqs, int rows, int r, TileRef& t) {
  if (num_seqs > kLptMaxSeqs) {
    // plain order: sequences in turn, heaviest tile of each first
    for (int s = 0; s < num_seqs; ++s) {
      const int a = __ldg(cu + s), b = __ldg(cu + s + 1);
      const int n = (b - a + rows - 1) / rows;
      if (r < n) {
        t = TileRef{a, b - a, n - 1 - r, n, s};
        return true;
      }
      r -= n;
    }
    return false;
  }
  int max_n = 0, total = 0;
  for (int s = 0; s < num_seqs; ++s) {
    const int n = (__ldg(cu + s + 1) - __ldg(cu + s) + rows - 1) / rows;
    max_n = n > max_n ? n : max_n;
    total += n;
  }
  if (r >= total) return false;
  // largest q with count_ge(q) > r (count_ge(0) = total > r)
  int lo = 0, hi = max_n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (lpt_count_ge(cu, num_seqs, rows, mid) > r)
      lo = mid;
    else
      hi = mid - 1;
  }
  int k = r - lpt_count_ge(cu, num_seqs, rows, lo + 1);  // index among sequences with n_s > lo
  for (int s = 0; s < num_seqs; ++s) {
    const int a = __ldg(cu + s), b = __ldg(cu + s + 1);
    const int n = (b - a + rows - 1) / rows;
    if (n > lo) {
      if (k == 0) {
        t = TileRef{a, b - a, lo, n, s};
        return true;
      }
      --k;
    }
  }
  return false;
}

}  // namespace gcs
