// The decode stream schedule shared by the bf16 and the W8A8 weight streams.
//
// The listed experts' matrices are cut into NSR stages each; the n_list * NSR
// stages are dealt out as contiguous, equal ranges of L stages, one range per
// CTA.  A CTA's range meets an expert in one contiguous part; the part index
// j = CTA index - the first CTA of that expert addresses its partial sums.
#pragma once

#include "internal.cuh"

namespace moe {

// Stages per CTA range: equal ranges covering all stages with at most G CTAs,
// and no expert spanning more than jcap ranges.
__device__ __forceinline__ int stream_len(int n_list, int NSR, int G, int jcap) {
  const int total = n_list * NSR;
  int L = (total + G - 1) / G;
  if ((NSR + L - 1) / L + 1 > jcap) L = (NSR + jcap - 2) / (jcap - 1);
  return L;
}

__device__ __forceinline__ bool stream_slot(const FfnArgs& a, int li, int& e, int& slot) {
  e = a.list_e[li];
  if (e < 0 || e >= a.E) return false;
  slot = a.list_s ? a.list_s[li] : a.e2s ? a.e2s[e] : e;
  return slot >= 0 && slot < a.S;
}

struct StreamSeg {
  int e, slot, s_lo, s_hi, j, p0, nb;
};

// Calls f(seg) for each (expert part, token batch of at most RB rows) of the
// range [beg, end) in order; stops early when f returns false.  Every role of
// a CTA walks the same list.
template <int RB, class F>
__device__ __forceinline__ void stream_segments(const FfnArgs& a, int NSR, int L, int beg, int end, F&& f) {
  for (int li = beg / NSR; li * NSR < end; ++li) {
    StreamSeg g;
    if (!stream_slot(a, li, g.e, g.slot)) continue;
    g.s_lo = max(beg, li * NSR) - li * NSR;
    g.s_hi = min(end, (li + 1) * NSR) - li * NSR;
    g.j = (int)blockIdx.x - (li * NSR) / L;
    const int pb = a.offset[g.e], pe = a.offset[g.e + 1];
    for (g.p0 = pb; g.p0 < pe; g.p0 += RB) {
      g.nb = min(RB, pe - g.p0);
      if (!f(g)) return;
    }
  }
}

// Parts an expert spans for list index li: J = last CTA - first CTA + 1.
__device__ __forceinline__ int stream_parts(int li, int NSR, int L) {
  return ((li + 1) * NSR - 1) / L - (li * NSR) / L + 1;
}

// Batched schedule: every listed expert contributes ceil(rows / RB) token
// batches, and the stage sequence runs over batches ("virtual experts"), so an
// expert whose tokens need several passes over its weights also gets several
// stage ranges and no CTA carries more work than another.
// vpre[li] = batches before list index li; vpre[n_list] = all batches.  Every
// thread of the block calls this (block scan); vpre holds n_list + 1 ints.
template <int RB>
__device__ __forceinline__ void stream_batch_prefix(const FfnArgs& a, int n_list, int* vpre, int* tmp) {
  int base = 0;
  for (int l0 = 0; l0 < n_list; l0 += blockDim.x) {
    const int li = l0 + threadIdx.x;
    int nbat = 0;
    if (li < n_list) {
      int e, slot;
      if (stream_slot(a, li, e, slot)) nbat = (a.offset[e + 1] - a.offset[e] + RB - 1) / RB;
    }
    int tot = 0;
    const int ex = block_exclusive_scan(nbat, tmp, &tot);
    if (li < n_list) vpre[li] = base + ex;
    base += tot;
  }
  if (threadIdx.x == 0) vpre[n_list] = base;
  __syncthreads();
}

// The list index whose batches contain batch vi: the largest li with vpre[li] <= vi < vpre[li + 1].
__device__ __forceinline__ int stream_batch_owner(const int* vpre, int n_list, int vi) {
  int lo = 0, hi = n_list;  // vpre[lo] <= vi < vpre[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (vpre[mid] <= vi) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Calls f(seg) for each batch part of the stage range [beg, end) over batches.
template <int RB, class F>
__device__ __forceinline__ void stream_segments_batched(const FfnArgs& a, const int* vpre, int n_list, int NSR, int L,
                                                        int beg, int end, F&& f) {
  for (int vi = beg / NSR; vi * NSR < end; ++vi) {
    StreamSeg g;
    const int li = stream_batch_owner(vpre, n_list, vi);
    if (!stream_slot(a, li, g.e, g.slot)) continue;
    g.s_lo = max(beg, vi * NSR) - vi * NSR;
    g.s_hi = min(end, (vi + 1) * NSR) - vi * NSR;
    g.j = (int)blockIdx.x - (vi * NSR) / L;
    g.p0 = a.offset[g.e] + (vi - vpre[li]) * RB;
    g.nb = min(RB, a.offset[g.e + 1] - g.p0);
    if (!f(g)) return;
  }
}

}  // namespace moe
