// Top-k selection of key blocks for one query block: the k largest scores,
// ties to the lower block index, written in ascending block order.
//
// Runs on a group of `nthreads` threads (a multiple of 32, at most 1024)
// synchronised with named barrier `bar_id`.  Method: MSB-first radix select
// (4 passes of 8 bits) over order-preserving 32-bit keys finds the k-th largest
// key tau and how many of the tied keys are needed; an ordered compaction over
// the row then emits every key > tau and the lowest-index keys == tau.
#pragma once

#include "common.cuh"

namespace sda {

struct TopkScratch {
  unsigned hist[256];
  unsigned warp_a[32];
  unsigned warp_b[32];
  unsigned prefix;
  unsigned remaining;
};

__device__ __forceinline__ unsigned order_key(float f) {
  unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ inline void topk_select(const float* scores, int n, int k, int32_t* out, int tid, int nthreads,
                                   int bar_id, TopkScratch* s) {
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  unsigned prefix = 0, mask = 0;
  unsigned remaining = (unsigned)k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += nthreads) s->hist[i] = 0;
    named_bar(bar_id, nthreads);
    for (int j = tid; j < n; j += nthreads) {
      unsigned key = order_key(scores[j]);
      if ((key & mask) == prefix) atomicAdd(&s->hist[(key >> shift) & 255u], 1u);
    }
    named_bar(bar_id, nthreads);
    if (tid == 0) {
      unsigned above = 0;
      int b = 255;
      for (; b > 0; --b) {
        unsigned h = s->hist[b];
        if (above + h >= remaining) break;
        above += h;
      }
      s->prefix = prefix | ((unsigned)b << shift);
      s->remaining = remaining - above;
    }
    named_bar(bar_id, nthreads);
    prefix = s->prefix;
    remaining = s->remaining;
    mask |= 0xFFu << shift;
    named_bar(bar_id, nthreads);
  }
  const unsigned tau = prefix;  // key of the k-th largest score
  // Ordered compaction: keys > tau, plus the first `remaining` keys == tau.
  unsigned base_sel = 0, base_eq = 0;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int c0 = 0; c0 < n; c0 += nthreads) {
    const int j = c0 + tid;
    unsigned key = j < n ? order_key(scores[j]) : 0u;
    bool gt = j < n && key > tau;
    bool eq = j < n && key == tau;
    unsigned meq = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) s->warp_b[warp] = __popc(meq);
    named_bar(bar_id, nthreads);
    unsigned eq_before = base_eq + __popc(meq & lt_mask);
    for (int w = 0; w < warp; ++w) eq_before += s->warp_b[w];
    bool sel = gt || (eq && eq_before < remaining);
    unsigned msel = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) s->warp_a[warp] = __popc(msel);
    named_bar(bar_id, nthreads);
    unsigned pos = base_sel + __popc(msel & lt_mask);
    for (int w = 0; w < warp; ++w) pos += s->warp_a[w];
    if (sel && pos < (unsigned)k) out[pos] = j;
    unsigned tot_sel = 0, tot_eq = 0;
    for (int w = 0; w < nwarps; ++w) {
      tot_sel += s->warp_a[w];
      tot_eq += s->warp_b[w];
    }
    base_sel += tot_sel;
    base_eq += tot_eq;
    named_bar(bar_id, nthreads);
  }
}

}  // namespace sda
