// Streaming top-k helpers over candidate lists kept in ascending position
// order, for the fused prefill indexer.
//
// A candidate is (key, position) with key = float_key(score): a larger key is
// a larger score, equal keys are equal scores, and between equal scores the
// lower position is preferred.  Because a list is in ascending position
// order, "lower position" is "earlier in the list".
//
// cut_list keeps every candidate whose key is at least a threshold thr chosen
// with histograms of 256 equal-width bins over the key range still open
// (starting from the caller's bounds [lo, hi]), such that at least k
// candidates are kept.  It stops refining as soon as the kept count is at most `limit`;
// with limit == k it is an exact top-k (remaining ties at thr are broken by
// list order).  Either way, a later candidate whose key is <= thr is beaten
// by k kept candidates, so thr is a valid insertion threshold afterwards.
#pragma once
#include "topk_select.cuh"

namespace ic {

// Keep, in order, the entries with key > thr and the first eq_keep entries
// (in list order) with key == thr.  Returns the kept count.  Every write
// lands at or below the index it came from, and each half of the list is
// read into registers before any of its writes.
template <int NTHREADS, int SEG, class Sync>
__device__ int compact_keys(uint32_t* key, int* pos, int n, uint32_t thr, int eq_keep, SelectScratch* scr, int tid,
                            Sync sync) {
  constexpr int HS = (SEG + 1) / 2;
  const bool ties = eq_keep < n;   // otherwise every key == thr is kept
  int written = 0, eq_seen = 0;
  const int half_n = (n + 1) / 2;
#pragma unroll 1
  for (int part = 0; part < 2; ++part) {
    const int p0 = part ? half_n : 0;
    const int pn = part ? n - half_n : half_n;
    uint32_t vk[HS];
    int vp[HS];
    unsigned gt = 0, eq = 0;
    int n_eq = 0;
    const int seg = (pn + NTHREADS - 1) / NTHREADS;
    const int b0 = p0 + tid * seg;
#pragma unroll
    for (int j = 0; j < HS; ++j) {
      const int i = b0 + j;
      if (j < seg && i < p0 + pn) {
        vk[j] = key[i];
        vp[j] = pos[i];
        if (vk[j] > thr) gt |= 1u << j;
        else if (vk[j] == thr) { eq |= 1u << j; ++n_eq; }
      }
    }
    int eq_before = 0;
    if (ties) {
      int eq_total;
      eq_before = eq_seen + block_exclusive_scan(n_eq, scr->warp_sums, NTHREADS, eq_total, tid, sync);
      eq_seen += eq_total;
    }
    unsigned keepm = gt;
#pragma unroll
    for (int j = 0; j < HS; ++j) {
      if (eq & (1u << j)) {
        if (!ties || eq_before < eq_keep) keepm |= 1u << j;
        ++eq_before;
      }
    }
    int total;
    int off = written + block_exclusive_scan(__popc(keepm), scr->warp_sums, NTHREADS, total, tid, sync);
#pragma unroll
    for (int j = 0; j < HS; ++j) {
      if (keepm & (1u << j)) {
        key[off] = vk[j];
        pos[off] = vp[j];
        ++off;
      }
    }
    written += total;
    sync();
  }
  return written;
}

// See the file comment.  n > k >= 1, n <= NTHREADS * SEG.  Every entry has
// lo <= key <= hi except exactly above0 (< k) entries with key > hi, which
// are all kept.  Returns the kept count; *thr_out = thr.
template <int NTHREADS, int SEG, class Sync>
__device__ int cut_list(uint32_t* key, int* pos, int n, int k, int limit, uint32_t lo, uint32_t hi,
                        SelectScratch* scr, int tid, Sync sync, uint32_t* thr_out, int above0 = 0) {
  const int lane = tid & 31, wid = tid >> 5;
  uint32_t rlo = lo, rhi = hi;   // the entries still to decide have rlo <= key <= rhi
  int need = k - above0;         // still to take from them
  int above = above0;            // entries above the range (all kept)
  int match = n - above0;        // entries in the range
  while (rlo < rhi && above + match > limit && match != need) {
    // up to 256 bins of 2^shift keys each, from rlo: the bins follow the
    // range, not the bit boundaries of the keys, so that keys crowded just
    // above the threshold still spread over many bins
    const uint32_t span = rhi - rlo;
    const int shift = max(0, 24 - __clz(span));   // span >> shift <= 255
    for (int i = tid; i < 256; i += NTHREADS) scr->hist[i] = 0;
    sync();
    for (int i = tid; i < n; i += NTHREADS) {
      const uint32_t h = key[i];
      if (h >= rlo && h <= rhi) atomicAdd(&scr->hist[(h - rlo) >> shift], 1);
    }
    sync();
    if (wid == 0) {
      int c[8];
      int s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { c[j] = scr->hist[255 - 8 * lane - j]; s += c[j]; }
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const int excl = incl - s;
      if (excl < need && need <= incl) {
        int cum = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (cum + c[j] >= need) {
            scr->sel_digit = 255 - 8 * lane - j;
            scr->sel_need = need - cum;
            scr->sel_done = c[j];            // entries in the chosen bin
            break;
          }
          cum += c[j];
        }
      }
    }
    sync();
    const uint32_t dsel = static_cast<uint32_t>(scr->sel_digit);
    const int nneed = scr->sel_need;
    match = scr->sel_done;
    above += need - nneed;
    need = nneed;
    const uint32_t blo = rlo + (dsel << shift);
    const uint32_t width = (1u << shift) - 1u;   // the chosen bin is [blo, blo + width] (shift <= 24)
    rhi = (rhi - blo <= width) ? rhi : blo + width;
    rlo = blo;
    sync();
  }
  // kept: everything above the range, then from the range's entries either
  // all of them (a key >= rlo) or, when the range is one value, the first
  // `need` in list order
  const int eq_keep = (rlo == rhi && above + match > limit) ? need : n;
  *thr_out = rlo;
  return compact_keys<NTHREADS, SEG>(key, pos, n, rlo, eq_keep, scr, tid, sync);
}

}  // namespace ic
