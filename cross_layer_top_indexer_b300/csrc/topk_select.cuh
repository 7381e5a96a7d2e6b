// Block-wide exact selection helpers shared by the indexer kernels.
//
// A candidate is (score, position).  Preference: higher score, then lower
// position.  The 64-bit composite (float_key(score) << 32) | ~position is
// therefore strictly larger for every preferred candidate, and all
// composites are distinct.  Selection keeps the k largest composites with a
// most-significant-digit radix select (up to 8-bit digits), and compaction
// keeps the survivors in their original (ascending position) order.
//
// The caller passes bounds that every candidate satisfies (its score key
// lies in [lo_key, hi_key], its position in [0, max_pos]); the leading bits
// those bounds share are common to all candidates and are not histogrammed.
#pragma once
#include "ic_common.cuh"

namespace ic {

struct SelectScratch {
  int hist[256];
  int warp_sums[32];
  int sel_digit;
  int sel_need;
  int sel_done;
  uint32_t tau;
};

// Threads of the group are tid = 0 .. nthreads-1 (whole warps); `sync`
// synchronises exactly that group.
struct BlockSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

template <class Sync>
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int nthreads, int& total, int tid,
                                                    Sync sync) {
  const int lane = tid & 31, wid = tid >> 5, nw = nthreads >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_sums[wid] = incl;
  sync();
  // every warp scans the warp totals itself (no second round through
  // shared memory); the barrier after lets the next scan reuse warp_sums
  const int s = lane < nw ? warp_sums[lane] : 0;
  int si = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, si, o);
    if (lane >= o) si += t;
  }
  total = __shfl_sync(0xffffffffu, si, 31);
  const int before = __shfl_sync(0xffffffffu, si - s, wid);
  sync();
  return before + incl - v;
}

// Mask of the top `bits` bits of a word (0 <= bits <= 32).
__device__ __forceinline__ uint32_t top_mask(int bits) { return bits <= 0 ? 0u : (0xFFFFFFFFu << (32 - bits)); }

// Keep the k best of the n candidates (sc[0..n), pos[0..n)), in place and in
// order; returns through scr->tau the smallest kept float_key.  n > k >= 1.
// All threads of the group must call it.  SEG = max entries per thread
// (n <= NTHREADS * SEG).  Bounds: lo_key <= float_key(sc[i]) <= hi_key and
// 0 <= pos[i] <= max_pos for every i.
template <int NTHREADS, int SEG, class Sync = BlockSync>
__device__ void select_keep_topk(float* sc, int* pos, int n, int k, SelectScratch* scr, int tid, Sync sync,
                                 uint32_t lo_key, uint32_t hi_key, uint32_t max_pos) {
  const int lane = tid & 31, wid = tid >> 5;
  // bits shared by every candidate: the common prefix of the bounds
  int kh = lo_key == hi_key ? 32 : __clz(lo_key ^ hi_key);
  int kl = max_pos == 0 ? 32 : __clz(max_pos);     // ~pos lies in [~max_pos, 0xFFFFFFFF]
  uint32_t msk_hi = top_mask(kh), pre_hi = hi_key & msk_hi;
  uint32_t msk_lo = top_mask(kl), pre_lo = 0xFFFFFFFFu & msk_lo;
  int need = k;
  while (kh < 32 || kl < 32) {
    const bool hw = kh < 32;
    const int known = hw ? kh : kl;
    const int w = min(8, 32 - known);
    const int shift = 32 - known - w;
    const uint32_t dmask = (1u << w) - 1u;
    for (int i = tid; i < 256; i += NTHREADS) scr->hist[i] = 0;
    sync();
    for (int i = tid; i < n; i += NTHREADS) {
      const uint32_t h = float_key(sc[i]);
      const uint32_t l = ~static_cast<uint32_t>(pos[i]);
      if ((h & msk_hi) == pre_hi && (l & msk_lo) == pre_lo) atomicAdd(&scr->hist[((hw ? h : l) >> shift) & dmask], 1);
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
        int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      int excl = incl - s;
      if (excl < need && need <= incl) {
        int cum = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (cum + c[j] >= need) {
            scr->sel_digit = 255 - 8 * lane - j;
            scr->sel_need = need - cum;
            scr->sel_done = (c[j] == need - cum);
            break;
          }
          cum += c[j];
        }
      }
    }
    sync();
    const uint32_t dsel = static_cast<uint32_t>(scr->sel_digit);
    need = scr->sel_need;
    const int done = scr->sel_done;
    if (hw) { pre_hi |= dsel << shift; msk_hi |= dmask << shift; kh += w; }
    else    { pre_lo |= dsel << shift; msk_lo |= dmask << shift; kl += w; }
    sync();
    if (done) break;
  }
  // Ordered compaction in two halves (fewer registers): contiguous segment
  // per thread, block scan of the counts.  Every write lands at or below the
  // index it came from, and each half is read into registers before any of
  // its writes.
  if (tid == 0) scr->tau = 0xffffffffu;
  uint32_t local_min = 0xffffffffu;
  constexpr int HS = (SEG + 1) / 2;
  int written = 0;
  const int half_n = (n + 1) / 2;
#pragma unroll 1
  for (int part = 0; part < 2; ++part) {
    const int p0 = part ? half_n : 0;
    const int pn = part ? n - half_n : half_n;
    float vs[HS];
    int vp[HS];
    int keep = 0;
    unsigned flags = 0;
    const int seg = (pn + NTHREADS - 1) / NTHREADS;
    const int b0 = p0 + tid * seg;
#pragma unroll
    for (int j = 0; j < HS; ++j) {
      const int i = b0 + j;
      if (j < seg && i < p0 + pn) {
        vs[j] = sc[i];
        vp[j] = pos[i];
        const uint32_t mh = float_key(vs[j]) & msk_hi;
        const uint32_t ml = ~static_cast<uint32_t>(vp[j]) & msk_lo;
        const bool take = (mh > pre_hi) || (mh == pre_hi && ml >= pre_lo);
        if (take) { flags |= 1u << j; ++keep; }
      }
    }
    int total;
    int off = written + block_exclusive_scan(keep, scr->warp_sums, NTHREADS, total, tid, sync);
#pragma unroll
    for (int j = 0; j < HS; ++j) {
      if (flags & (1u << j)) {
        sc[off] = vs[j];
        pos[off] = vp[j];
        ++off;
        const uint32_t h = float_key(vs[j]);
        local_min = h < local_min ? h : local_min;
      }
    }
    written += total;
    sync();
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    uint32_t t = __shfl_xor_sync(0xffffffffu, local_min, o);
    local_min = t < local_min ? t : local_min;
  }
  if (lane == 0 && local_min != 0xffffffffu) atomicMin(&scr->tau, local_min);
  sync();
}

}  // namespace ic
