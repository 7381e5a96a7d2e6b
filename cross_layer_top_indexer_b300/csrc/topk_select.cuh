// Block-wide exact selection helpers shared by the indexer kernels.
//
// A candidate is (score, position).  Preference: higher score, then lower
// position.  The 64-bit composite (float_key(score) << 32) | ~position is
// therefore strictly larger for every preferred candidate, and all
// composites are distinct.  Selection keeps the k largest composites with a
// most-significant-digit radix select (8-bit digits), and compaction keeps
// the survivors in their original (ascending position) order.
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
  if (wid == 0) {
    int s = lane < nw ? warp_sums[lane] : 0;
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += t;
    }
    if (lane < nw) warp_sums[lane] = si - s;   // exclusive prefix of warps
    if (lane == 31) warp_sums[31] = si;        // grand total (nw <= 31)
  }
  sync();
  total = warp_sums[31];
  int r = warp_sums[wid] + incl - v;
  sync();
  return r;
}

// Keep the k best of the n candidates (sc[0..n), pos[0..n)), in place and in
// order; returns through scr->tau the smallest kept float_key.  n > k >= 1.
// All threads of the block must call it.  SEG = max entries per thread.
template <int NTHREADS, int SEG, class Sync = BlockSync>
__device__ void select_keep_topk(float* sc, int* pos, int n, int k, SelectScratch* scr, int tid = -1,
                                 Sync sync = Sync()) {
  if (tid < 0) tid = threadIdx.x;
  const int lane = tid & 31, wid = tid >> 5;
  uint32_t pre_hi = 0, msk_hi = 0, pre_lo = 0, msk_lo = 0;
  int need = k;
  for (int pass = 0; pass < 8; ++pass) {
    const bool hi_word = pass < 4;
    const int shift = 24 - 8 * (pass & 3);
    for (int i = tid; i < 256; i += NTHREADS) scr->hist[i] = 0;
    sync();
    for (int i = tid; i < n; i += NTHREADS) {
      uint32_t h = float_key(sc[i]);
      uint32_t l = ~(uint32_t)pos[i];
      if ((h & msk_hi) == pre_hi && (l & msk_lo) == pre_lo) {
        uint32_t d = ((hi_word ? h : l) >> shift) & 255u;
        atomicAdd(&scr->hist[d], 1);
      }
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
    const uint32_t dsel = (uint32_t)scr->sel_digit;
    need = scr->sel_need;
    const int done = scr->sel_done;
    if (hi_word) { pre_hi |= dsel << shift; msk_hi |= 255u << shift; }
    else         { pre_lo |= dsel << shift; msk_lo |= 255u << shift; }
    sync();
    if (done) break;
  }
  // Ordered compaction: contiguous segment per thread, block scan of counts.
  if (tid == 0) scr->tau = 0xffffffffu;
  float vs[SEG];
  int vp[SEG];
  int keep = 0;
  unsigned flags = 0;
  const int seg = (n + NTHREADS - 1) / NTHREADS;
  const int b0 = tid * seg;
#pragma unroll
  for (int j = 0; j < SEG; ++j) {
    const int i = b0 + j;
    if (j < seg && i < n) {
      vs[j] = sc[i];
      vp[j] = pos[i];
      uint32_t h = float_key(vs[j]);
      uint32_t l = ~(uint32_t)vp[j];
      uint32_t mh = h & msk_hi, ml = l & msk_lo;
      bool take = (mh > pre_hi) || (mh == pre_hi && ml >= pre_lo);
      if (take) { flags |= 1u << j; ++keep; }
    }
  }
  int total;
  int off = block_exclusive_scan(keep, scr->warp_sums, NTHREADS, total, tid, sync);
  uint32_t local_min = 0xffffffffu;
#pragma unroll
  for (int j = 0; j < SEG; ++j) {
    if (flags & (1u << j)) {
      sc[off] = vs[j];
      pos[off] = vp[j];
      ++off;
      uint32_t h = float_key(vs[j]);
      local_min = h < local_min ? h : local_min;
    }
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
