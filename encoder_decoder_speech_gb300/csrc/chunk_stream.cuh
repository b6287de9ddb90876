// The chunk numbering shared by the persistent split-T decode kernels: the valid
// key chunks of every (slot, row) are numbered densely, slot-major, then row, then
// key order; each CTA takes one equal contiguous range of the numbers; a row cut by
// a range boundary is merged from per-segment (max, sum, accumulator) states.
#pragma once

#include <cmath>
#include <cstdint>

namespace cxa {

// Position in the dense chunk numbering: slot b, row-in-slot lh, chunk c.
struct Cursor {
  int b, lh, c;
};

// s_first[b] = number of slot b's first chunk (s_first[B] = total), s_nch[b] =
// chunks per row of slot b; both live in shared memory.
__device__ __forceinline__ Cursor locate(long long g, const long long* s_first, const int* s_nch, int B) {
  int lo = 0, hi = B - 1;   // last b with s_first[b] <= g
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_first[mid] <= g) lo = mid; else hi = mid - 1;
  }
  const long long local = g - s_first[lo];
  Cursor cur;
  cur.b = lo;
  cur.lh = static_cast<int>(local / s_nch[lo]);
  cur.c = static_cast<int>(local - static_cast<long long>(cur.lh) * s_nch[lo]);
  return cur;
}

// The next chunk in the numbering (slots without chunks are skipped).
__device__ __forceinline__ void advance(Cursor& cur, const int* s_nch, int B, int LH) {
  if (++cur.c < s_nch[cur.b]) return;
  cur.c = 0;
  if (++cur.lh < LH) return;
  cur.lh = 0;
  do {
    ++cur.b;
  } while (cur.b < B && s_nch[cur.b] == 0);
}

// The CTA that owns dense chunk g when total chunks are split into `ranges`
// equal ranges [j*total/ranges, (j+1)*total/ranges).
__device__ __forceinline__ long long owner_of(long long g, long long total, long long ranges) {
  return ((g + 1) * ranges + total - 1) / total - 1;
}

// Weight of a softmax state with running max m (base 2) against a merged max M
// (0 for an empty state, m == -inf).
__device__ __forceinline__ float rescale(float m, float M) { return m == -INFINITY ? 0.f : exp2f(m - M); }

__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace cxa
