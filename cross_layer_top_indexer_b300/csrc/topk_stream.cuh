// Streaming top-k helpers over candidate lists kept in ascending position
// order, for the fused prefill indexer.
//
// A candidate is (key, position) with key = float_key(score): a larger key is
// a larger score, equal keys are equal scores, and between equal scores the
// lower position is preferred.  Because a list is in ascending position
// order, "lower position" is "earlier in the list".
//
// cut_list keeps every candidate whose key is at least a threshold thr chosen
// with a most-significant-digit histogram (8-bit digits below the bits that
// the caller's bounds [lo, hi] share), such that at least k candidates are
// kept.  It stops refining as soon as the kept count is at most `limit`;
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

// See the file comment.  n > k >= 1, n <= NTHREADS * SEG, lo <= key[i] <= hi
// for every i.  Returns the kept count; *thr_out = thr.
template <int NTHREADS, int SEG, class Sync>
__device__ int cut_list(uint32_t* key, int* pos, int n, int k, int limit, uint32_t lo, uint32_t hi,
                        SelectScratch* scr, int tid, Sync sync, uint32_t* thr_out) {
  const int lane = tid & 31, wid = tid >> 5;
  int kb = lo == hi ? 32 : __clz(lo ^ hi);     // leading bits shared by every key
  uint32_t msk = top_mask(kb), pre = hi & msk;
  int need = k;        // still to take from the entries matching the prefix
  int above = 0;       // entries strictly above the prefix (all kept)
  int match = n;       // entries matching the prefix
  while (kb < 32 && above + match > limit && match != need) {
    const int w = min(8, 32 - kb);
    const int shift = 32 - kb - w;
    const uint32_t dmask = (1u << w) - 1u;
    for (int i = tid; i < 256; i += NTHREADS) scr->hist[i] = 0;
    sync();
    for (int i = tid; i < n; i += NTHREADS) {
      const uint32_t h = key[i];
      if ((h & msk) == pre) atomicAdd(&scr->hist[(h >> shift) & dmask], 1);
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
    pre |= dsel << shift;
    msk |= dmask << shift;
    kb += w;
    sync();
  }
  // kept: everything above the prefix, then from the prefix's entries either
  // all of them (a key >= pre) or, when the keys are fully resolved (all equal
  // to pre), the first `need` in list order
  const int eq_keep = (kb >= 32 && above + match > limit) ? need : n;
  *thr_out = pre;
  return compact_keys<NTHREADS, SEG>(key, pos, n, pre, eq_keep, scr, tid, sync);
}

}  // namespace ic
