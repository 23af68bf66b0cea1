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
  slot = a.e2s ? a.e2s[e] : e;
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

}  // namespace moe
