// Decode indexer: few query rows per sequence against a long key cache.
//
// Same score as the prefill kernel (DSA lightning-indexer score used by
// IndexCache's Full layers; notes page "NLP--IndexCache", "背景 & 问题提出"),
// but the work is spread over the KEYS, so a handful of query rows still
// fills the GPU.  Each query row's causal scores are staged in the workspace
// (one fp32 row per query, O(L), never an L x L matrix), then the exact
// top-k is selected and written in ascending position order.
//
// Scores: the tensor-core kernel (indexer_decode_tc.cu) for one row per
// sequence with H = 64, d = 128; otherwise decode_scores_kernel below (one
// CTA per (tile of keys, query row), mma.sync).
// Select: with the tensor-core scorer and a workspace that holds the
// histogram, the clustered select (select_cluster_kernel, a cluster of CTAs
// per row); otherwise decode_select_kernel, one CTA per row.
#include <cooperative_groups.h>

#include "ic_common.cuh"
#include "ic_kernels.h"
#include "tc_utils.cuh"
#include "topk_stream.cuh"

namespace ic {
namespace {

namespace cg = cooperative_groups;

constexpr int DKT = 256;          // keys per scoring CTA (8 warps x 32)
constexpr int DTHREADS = 256;
constexpr int HMAX = 64;

template <int D>
struct DecodeSmem {
  static constexpr int P = D + 8;
  __nv_bfloat16 qs[HMAX][P];
  __nv_bfloat16 ks[DKT][P];
  float wsm[HMAX];
  float ksc[DKT];
};

size_t row_pitch(int S) { return (size_t)((S + 3) / 4) * 4; }

template <int D>
__global__ void __launch_bounds__(DTHREADS)
decode_scores_kernel(IndexerArgs a, float* scores, int h_pad, size_t pitch) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<DecodeSmem<D>*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int row = blockIdx.y;                 // b * T + t
  const int b = row / a.T, t = row - b * a.T;
  const int pos = a.q_pos0 + t;
  const int s0 = blockIdx.x * DKT;
  if (s0 > pos) return;                       // tile entirely past this row's position
  const int n_keys = pos + 1;

  {
    const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(a.q) + (size_t)row * a.H * D;
    constexpr int CH = D / 8;
    for (int i = tid; i < h_pad * CH; i += DTHREADS) {
      const int h = i / CH, c = i % CH;
      const bool ok = h < a.H;
      cp_async16(&sm.qs[h][c * 8], ok ? qg + (size_t)h * D + c * 8 : qg, ok);
    }
    for (int h = tid; h < HMAX; h += DTHREADS) sm.wsm[h] = h < a.H ? a.w[(size_t)row * a.H + h] : 0.0f;
  }
  if (!a.e4m3) {
    const __nv_bfloat16* kg_ = reinterpret_cast<const __nv_bfloat16*>(a.kI) + (size_t)b * a.S_cap * D;
    constexpr int CH = D / 8;
    for (int i = tid; i < DKT * CH; i += DTHREADS) {
      const int r = i / CH, c = i % CH, s = s0 + r;
      const bool ok = s < n_keys;
      cp_async16(&sm.ks[r][c * 8], ok ? kg_ + (size_t)s * D + c * 8 : kg_, ok);
    }
    for (int r = tid; r < DKT; r += DTHREADS) sm.ksc[r] = 1.0f;
  } else {
    const uint8_t* kg8 = reinterpret_cast<const uint8_t*>(a.kI) + (size_t)b * a.S_cap * D;
    constexpr int CH = D / 16;
    for (int i = tid; i < DKT * CH; i += DTHREADS) {
      const int r = i / CH, c = i % CH, s = s0 + r;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (s < n_keys) v = *reinterpret_cast<const uint4*>(kg8 + (size_t)s * D + c * 16);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t x = wv[j];
        o[2 * j] = e4m3_to_bf16_bits(x & 0xFF) | (e4m3_to_bf16_bits((x >> 8) & 0xFF) << 16);
        o[2 * j + 1] = e4m3_to_bf16_bits((x >> 16) & 0xFF) | (e4m3_to_bf16_bits(x >> 24) << 16);
      }
      uint4* dst = reinterpret_cast<uint4*>(&sm.ks[r][c * 16]);
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
    for (int r = tid; r < DKT; r += DTHREADS) {
      const int s = s0 + r;
      sm.ksc[r] = s < n_keys ? a.kscale[(size_t)b * a.S_cap + s] : 0.0f;
    }
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();

  const int n_tiles_h = h_pad / 8;
  float acc[2][8][4];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[m][n][j] = 0.0f;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    uint32_t af[2][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
      ldmatrix_x4(af[m][0], af[m][1], af[m][2], af[m][3],
                  &sm.ks[wid * 32 + m * 16 + (lane & 15)][kk * 16 + (lane >> 4) * 8]);
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      if (2 * np < n_tiles_h) {
        const int mat = lane >> 3;
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(b0, b1, b2, b3, &sm.qs[np * 16 + (mat >> 1) * 8 + (lane & 7)][kk * 16 + (mat & 1) * 8]);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          mma_bf16_16816(acc[m][2 * np], af[m][0], af[m][1], af[m][2], af[m][3], b0, b1);
          mma_bf16_16816(acc[m][2 * np + 1], af[m][0], af[m][1], af[m][2], af[m][3], b2, b3);
        }
      }
    }
  }
  float* out = scores + (size_t)row * pitch;
#pragma unroll
  for (int m = 0; m < 2; ++m) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float part = 0.0f;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        if (n < n_tiles_h) {
          const int h = n * 8 + 2 * (lane & 3);
          part = fmaf(sm.wsm[h], fmaxf(acc[m][n][2 * half], 0.0f), part);
          part = fmaf(sm.wsm[h + 1], fmaxf(acc[m][n][2 * half + 1], 0.0f), part);
        }
      }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      const int r = wid * 32 + m * 16 + half * 8 + (lane >> 2);
      const int s = s0 + r;
      if ((lane & 3) == 0 && s < n_keys) out[s] = part * sm.ksc[r];
    }
  }
}

// ---------------------------------------------------------------------------
// Exact top-k of one staged score row (one CTA per row).
// ---------------------------------------------------------------------------

constexpr int STHREADS = 512;
constexpr int SWARPS = STHREADS / 32;

// General path: most-significant-digit radix select over the composite
// (score key, ~position), one pass over the row per 8-bit digit, then an
// ordered write.  Used when the fast path's candidate set does not fit.
__device__ void radix_select_row(const float* sc, int n, int k, int32_t* out) {
  __shared__ int whist[SWARPS][256];
  __shared__ int hist[256];
  __shared__ int wsum[33];
  __shared__ int sel_digit, sel_need, sel_done;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  uint32_t pre_hi = 0, msk_hi = 0, pre_lo = 0, msk_lo = 0;
  int need = k;
  for (int pass = 0; pass < 8; ++pass) {
    const bool hi_word = pass < 4;
    const int shift = 24 - 8 * (pass & 3);
    for (int i = lane; i < 256; i += 32) whist[wid][i] = 0;
    __syncwarp();
    for (int i = tid; i < n; i += STHREADS) {
      const uint32_t h = float_key(sc[i]);
      const uint32_t l = ~(uint32_t)i;
      if ((h & msk_hi) == pre_hi && (l & msk_lo) == pre_lo)
        atomicAdd(&whist[wid][((hi_word ? h : l) >> shift) & 255u], 1);
    }
    __syncthreads();
    for (int d = tid; d < 256; d += STHREADS) {
      int s = 0;
      for (int w = 0; w < SWARPS; ++w) s += whist[w][d];
      hist[d] = s;
    }
    __syncthreads();
    if (wid == 0) {
      int c[8];
      int s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { c[j] = hist[255 - 8 * lane - j]; s += c[j]; }
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int excl = incl - s;
      if (excl < need && need <= incl) {
        int cum = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (cum + c[j] >= need) {
            sel_digit = 255 - 8 * lane - j;
            sel_need = need - cum;
            sel_done = (c[j] == need - cum);
            break;
          }
          cum += c[j];
        }
      }
    }
    __syncthreads();
    const uint32_t d = (uint32_t)sel_digit;
    need = sel_need;
    const int done = sel_done;
    if (hi_word) { pre_hi |= d << shift; msk_hi |= 255u << shift; }
    else         { pre_lo |= d << shift; msk_lo |= 255u << shift; }
    __syncthreads();
    if (done) break;
  }
  // Ordered write of the k survivors: chunks of STHREADS * 4 positions.
  int written = 0;
  for (int c0 = 0; c0 < n; c0 += STHREADS * 4) {
    int cnt = 0;
    unsigned f = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = c0 + tid * 4 + j;
      if (i < n) {
        const uint32_t mh = float_key(sc[i]) & msk_hi;
        const uint32_t ml = (~(uint32_t)i) & msk_lo;
        if (mh > pre_hi || (mh == pre_hi && ml >= pre_lo)) { f |= 1u << j; ++cnt; }
      }
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      const int s = lane < SWARPS ? wsum[lane] : 0;
      int si = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, si, o);
        if (lane >= o) si += v;
      }
      wsum[lane] = si - s;
      if (lane == 31) wsum[32] = si;
    }
    __syncthreads();
    int off = written + wsum[wid] + incl - cnt;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (f & (1u << j)) {
        if (off < k) out[off] = c0 + tid * 4 + j;
        ++off;
      }
    written += wsum[32];
    __syncthreads();
  }
}

// Fast path.  Pass 1 histograms the top 12 bits of every score key; the bin
// holding the k-th largest key is the threshold bin.  Pass 2 copies, in
// position order, every entry whose key is in or above that bin into shared
// memory (each warp takes a contiguous segment: it counts its entries, the
// warps' offsets are scanned, and a second sweep writes them with warp
// prefix sums).  If more than k were copied, cut_list keeps exactly the k
// best, ties to the earlier (lower) position.  The row is read three times,
// from L2, where the scoring kernel just wrote it.
constexpr int FBITS = 12;
constexpr int FBINS = 1 << FBITS;
constexpr int FSEG = 16;
constexpr int FCAP = STHREADS * FSEG;    // candidates held in shared memory

struct FastSelSmem {
  int hist[FBINS];
  uint32_t key[FCAP];
  int pos[FCAP];
  int woff[SWARPS];
  SelectScratch scr;
  int bsel, ncand;
};

__device__ __forceinline__ float4 load_row4(const float* sc, int i, int n) {
  if (i + 3 < n) return __ldcg(reinterpret_cast<const float4*>(sc + i));
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (i < n) v.x = sc[i];
  if (i + 1 < n) v.y = sc[i + 1];
  if (i + 2 < n) v.z = sc[i + 2];
  return v;
}

__global__ void __launch_bounds__(STHREADS)
decode_select_kernel(const float* scores, size_t pitch, int32_t* idx, int T, int q_pos0, int k) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  FastSelSmem& sm = *reinterpret_cast<FastSelSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int row = blockIdx.x;
  const int t = row % T;
  const int n = q_pos0 + t + 1;
  const float* sc = scores + (size_t)row * pitch;    // 16-byte aligned rows
  int32_t* out = idx + (size_t)row * k;

  if (n <= k) {
    for (int j = tid; j < k; j += STHREADS) out[j] = j < n ? j : -1;
    return;
  }
  // ---- pass 1: histogram of key >> 20
  for (int i = tid; i < FBINS; i += STHREADS) sm.hist[i] = 0;
  __syncthreads();
  constexpr int UNR = 8;
  for (int base = 4 * tid; base < n; base += 4 * STHREADS * UNR) {
    float4 v[UNR];
#pragma unroll
    for (int j = 0; j < UNR; ++j) v[j] = load_row4(sc, base + 4 * STHREADS * j, n);
#pragma unroll
    for (int j = 0; j < UNR; ++j) {
      const int i = base + 4 * STHREADS * j;
      if (i < n) atomicAdd(&sm.hist[float_key(v[j].x) >> 20], 1);
      if (i + 1 < n) atomicAdd(&sm.hist[float_key(v[j].y) >> 20], 1);
      if (i + 2 < n) atomicAdd(&sm.hist[float_key(v[j].z) >> 20], 1);
      if (i + 3 < n) atomicAdd(&sm.hist[float_key(v[j].w) >> 20], 1);
    }
  }
  __syncthreads();
  // ---- threshold bin: thread t holds bins FBINS-1-8t .. FBINS-8-8t (descending)
  {
    constexpr int BPT = FBINS / STHREADS;
    int c[BPT];
    int s = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) { c[j] = sm.hist[FBINS - 1 - BPT * tid - j]; s += c[j]; }
    int total;
    const int excl = block_exclusive_scan(s, sm.scr.warp_sums, STHREADS, total, tid, BlockSync());
    if (excl < k && k <= excl + s) {
      int cum = excl;
#pragma unroll
      for (int j = 0; j < BPT; ++j) {
        if (cum + c[j] >= k) { sm.bsel = FBINS - 1 - BPT * tid - j; sm.ncand = cum + c[j]; break; }
        cum += c[j];
      }
    }
  }
  __syncthreads();
  const int ncand = sm.ncand;
  if (ncand > FCAP) {
    radix_select_row(sc, n, k, out);
    return;
  }
  const uint32_t lo = static_cast<uint32_t>(sm.bsel) << 20;
  // ---- pass 2: ordered copy of the keys >= lo; warp wid takes [seg0, seg1)
  const int segE = ((n + SWARPS - 1) / SWARPS + 127) & ~127;
  const int seg0 = min(n, wid * segE), seg1 = min(n, seg0 + segE);
  int cnt = 0;
  for (int c0 = seg0; c0 < seg1; c0 += 128 * 4) {
    float4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = load_row4(sc, c0 + 128 * j + 4 * lane, seg1);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = c0 + 128 * j + 4 * lane;
      cnt += (i < seg1 && float_key(v[j].x) >= lo) + (i + 1 < seg1 && float_key(v[j].y) >= lo) +
             (i + 2 < seg1 && float_key(v[j].z) >= lo) + (i + 3 < seg1 && float_key(v[j].w) >= lo);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if (lane == 0) sm.woff[wid] = cnt;
  __syncthreads();
  if (wid == 0) {
    const int v = lane < SWARPS ? sm.woff[lane] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane < SWARPS) sm.woff[lane] = incl - v;
  }
  __syncthreads();
  int off = sm.woff[wid];
  for (int c0 = seg0; c0 < seg1; c0 += 128) {
    const int i = c0 + 4 * lane;
    const float4 v = load_row4(sc, i, seg1);
    const uint32_t kk[4] = {float_key(v.x), float_key(v.y), float_key(v.z), float_key(v.w)};
    unsigned f = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (i + j < seg1 && kk[j] >= lo) f |= 1u << j;
    const int c = __popc(f);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    int o2 = off + incl - c;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (f & (1u << j)) { sm.key[o2] = kk[j]; sm.pos[o2] = i + j; ++o2; }
    off += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncthreads();
  if (ncand > k) {
    uint32_t thr;
    cut_list<STHREADS, FSEG>(sm.key, sm.pos, ncand, k, k, lo, 0xFFFFFFFFu, &sm.scr, tid, BlockSync(), &thr);
  }
  for (int j = tid; j < k; j += STHREADS) out[j] = sm.pos[j];
}

cudaError_t launch_select(float* scores, size_t pitch, const IndexerArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(FastSelSmem);
  cudaError_t e = cudaFuncSetAttribute(decode_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  decode_select_kernel<<<a.B * a.T, STHREADS, smem, st>>>(scores, pitch, a.idx, a.T, a.q_pos0, a.k);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Clustered select (one query row per sequence, after the tensor-core
// scorer, which leaves a histogram of each row's score keys by their top
// kDecHistBits bits).  The threshold bin is the bin of the k-th largest key;
// the entries in and above it are the row's ncand candidates.  A cluster of
// SCL CTAs takes one row: CTA r copies the r-th part of the score row into
// its shared memory with bulk copies (one thread issues them; its 128 KB
// land in about 1.6 us) and lists its candidates (key, position), in
// position order; after the
// cluster barrier every CTA stores its list into CTA 0's, after the lists of
// the CTAs before it, through distributed shared memory; CTA 0 then cuts the
// threshold bin's entries to exactly k (the candidates above the bin are all
// kept) and writes the positions, which are already ascending.  Rows with
// more than FCAP candidates, or whose lists disagree with the histogram,
// take the general radix path.
// ---------------------------------------------------------------------------
constexpr int HBINS = 1 << kDecHistBits;
constexpr int SCL = 4;                   // CTAs per row (one cluster)
constexpr int SUNR = 17;                 // 16-byte reads per thread per pass
constexpr int SPASS = STHREADS * 4 * SUNR;   // scores per pass: a quarter of a 131K-key row in one
constexpr int SPIECE = 16384;            // bytes per bulk copy

struct DecWs {
  float* scores;
  int* hist;    // [rows][HBINS]
  size_t pitch;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

DecWs carve_ws(void* ws, int rows, int S, size_t* total) {
  DecWs d;
  d.pitch = row_pitch(S);
  unsigned char* p = static_cast<unsigned char*>(ws);
  size_t off = 0;
  d.scores = reinterpret_cast<float*>(p + off);
  off += align256(static_cast<size_t>(rows) * d.pitch * sizeof(float));
  d.hist = reinterpret_cast<int*>(p + off);
  off += align256(static_cast<size_t>(rows) * HBINS * sizeof(int));
  *total = off;
  return d;
}

// Threshold bin of a row from its histogram: the bin b* with
// count(bins > b*) < k <= count(bins >= b*); *ncand = count(bins >= b*).
// All NT threads call it; NT * BPT == HBINS.
template <int NT>
__device__ void threshold_bin(const int* h, int k, int* warp_sums, int* s_bsel, int* s_ncand) {
  constexpr int BPT = HBINS / NT;
  const int tid = threadIdx.x;
  if (tid == 0) { *s_bsel = 0; *s_ncand = 0x7FFFFFFF; }   // a histogram short of k sends the row to the radix path
  int c[BPT];
  int s = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) { c[j] = h[HBINS - 1 - BPT * tid - j]; s += c[j]; }
  int total;
  const int excl = block_exclusive_scan(s, warp_sums, NT, total, tid, BlockSync());
  if (excl < k && k <= excl + s) {
    int cum = excl;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
      if (cum + c[j] >= k) { *s_bsel = HBINS - 1 - BPT * tid - j; *s_ncand = cum + c[j]; break; }
      cum += c[j];
    }
  }
  __syncthreads();
}

// The bin b of h[0 .. NB) (NB / STHREADS consecutive bins per thread) where
// the count from the top reaches `need`: count(bins > b) < need <= count(bins
// >= b); *rem = need - count(bins > b).  All STHREADS threads call it.
template <int NB>
__device__ void top_down_bin(const int* h, int need, SelectScratch* scr, int* bin, int* rem) {
  constexpr int BPT = NB / STHREADS;
  const int tid = threadIdx.x;
  int c[BPT];
  int sum = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) { c[j] = h[NB - 1 - BPT * tid - j]; sum += c[j]; }
  int total;
  const int excl = block_exclusive_scan(sum, scr->warp_sums, STHREADS, total, tid, BlockSync());
  if (excl < need && need <= excl + sum) {
    int cum = excl;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
      if (cum + c[j] >= need) { scr->sel_digit = NB - 1 - BPT * tid - j; scr->sel_need = need - cum; break; }
      cum += c[j];
    }
  }
  __syncthreads();
  *bin = scr->sel_digit;
  *rem = scr->sel_need;
  __syncthreads();
}

// Exactly k of the n candidates (key[i], pos[i]), i in position order, to
// out in that order: the `above` entries over the threshold bin [lo, lo +
// 2^21) (fewer than k) and the best k - above of the bin's own entries, ties
// to the lower position.  Two histograms of the 21 bits under the bin's
// (2048 bins of the upper 11, then 1024 of the lower 10 within the chosen
// one) give the exact threshold key; one ordered pass writes the
// positions.  h: scratch of 2048 ints.  All STHREADS threads call it.
__device__ void cut_bin_to_out(const uint32_t* key, const int* pos, int n, int k, uint32_t lo, int above, int* h,
                               SelectScratch* scr, int32_t* out) {
  constexpr int LOW = 32 - kDecHistBits;
  constexpr int BB = 10, NA = 1 << (LOW - BB), NB = 1 << BB;
  static_assert(NA % STHREADS == 0 && NB % STHREADS == 0, "bins per thread");
  const int tid = threadIdx.x;
  const uint32_t hi = lo | ((1u << LOW) - 1u);
  const int seg = (n + STHREADS - 1) / STHREADS;
  const int i0 = min(n, tid * seg), i1 = min(n, i0 + seg);
  // the upper 11 bits
  for (int b = tid; b < NA; b += STHREADS) h[b] = 0;
  __syncthreads();
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = key[i];
    if (kk <= hi) atomicAdd(&h[(kk - lo) >> BB], 1);   // every candidate has kk >= lo
  }
  __syncthreads();
  int ba, need_a;
  top_down_bin<NA>(h, k - above, scr, &ba, &need_a);
  // the lower 10 bits, within bin ba
  const uint32_t lo_a = lo + (static_cast<uint32_t>(ba) << BB), hi_a = lo_a + (NB - 1);
  for (int b = tid; b < NB; b += STHREADS) h[b] = 0;
  __syncthreads();
  for (int i = i0; i < i1; ++i) {
    const uint32_t kk = key[i];
    if (kk >= lo_a && kk <= hi_a) atomicAdd(&h[kk - lo_a], 1);
  }
  __syncthreads();
  int bb, eq_keep;
  top_down_bin<NB>(h, need_a, scr, &bb, &eq_keep);
  const uint32_t thr = lo_a + static_cast<uint32_t>(bb);
  // keep key > thr, and the first eq_keep entries with key == thr
  int n_eq = 0;
  for (int i = i0; i < i1; ++i) n_eq += key[i] == thr;
  int eq_total;
  int eq_rank = block_exclusive_scan(n_eq, scr->warp_sums, STHREADS, eq_total, tid, BlockSync());
  int n_keep = 0;
  for (int i = i0, e = eq_rank; i < i1; ++i) {
    const uint32_t kk = key[i];
    n_keep += kk > thr || (kk == thr && e++ < eq_keep);
  }
  int tot;
  int off = block_exclusive_scan(n_keep, scr->warp_sums, STHREADS, tot, tid, BlockSync());
  for (int i = i0, e = eq_rank; i < i1; ++i) {
    const uint32_t kk = key[i];
    if (kk > thr || (kk == thr && e++ < eq_keep)) {
      if (off < k) out[off] = pos[i];
      ++off;
    }
  }
  // (tot == k whenever the lists agree with the histogram, as the caller checked)
  for (int j = tot + tid; j < k; j += STHREADS) out[j] = -1;
}

struct __align__(16) ClusterSelSmem {
  float buf[SPASS];                      // a pass of this CTA's part of the score row
  uint32_t key[FCAP];
  int pos[FCAP];
  SelectScratch scr;
  uint64_t bar;
  int bsel, ncand, count, good;
};

__global__ void __cluster_dims__(SCL, 1, 1) __launch_bounds__(STHREADS)
select_cluster_kernel(const float* scores, size_t pitch, const int* hist, int32_t* idx, int n, int k, int* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ClusterSelSmem& sm = *reinterpret_cast<ClusterSelSmem*>(smem_raw);   // bulk copies need 16-byte alignment
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int row = blockIdx.y, tid = threadIdx.x;
  if (tid == 0) {
    tc::mbar_init(&sm.bar, 1);
    tc::fence_mbar_init();
  }
  grid_dep_wait();                               // the scores and the histogram of the scorer just before
  grid_dep_trigger();
  const float* sc = scores + static_cast<size_t>(row) * pitch;
  int32_t* out = idx + static_cast<size_t>(row) * k;
  // the branches below depend only on (n, k, the row's histogram): every CTA
  // of the cluster takes the same one
  if (n <= k) {
    if (rank == 0)
      for (int j = tid; j < k; j += STHREADS) out[j] = j < n ? j : -1;
    return;
  }
  // this CTA's part of the row (a multiple of 4 scores, so copies stay 16-byte aligned)
  const int part = ((n + SCL - 1) / SCL + 3) & ~3;
  const int p0 = min(n, rank * part), p1 = min(n, p0 + part);
  // a pass's scores into buf, by bulk copies (thread 0)
  auto issue = [&](int base) {
    if (tid == 0) {
      // up to the row's pitch, which holds n rounded up to 4 scores
      const uint32_t bytes = static_cast<uint32_t>(((min(p1 - base, SPASS) + 3) & ~3) * sizeof(float));
      tc::fence_proxy_async_smem();              // the last pass's reads of buf come before these writes
      tc::mbar_arrive_expect_tx(&sm.bar, bytes);
      for (uint32_t off = 0; off < bytes; off += SPIECE)
        tc::bulk_g2s(reinterpret_cast<char*>(sm.buf) + off, reinterpret_cast<const char*>(sc + base) + off,
                     min(static_cast<uint32_t>(SPIECE), bytes - off), &sm.bar);
    }
  };
  if (p0 < p1) issue(p0);                        // the first pass lands while the threshold is found
  const int* hrow = hist + static_cast<size_t>(row) * HBINS;
  threshold_bin<STHREADS>(hrow, k, sm.scr.warp_sums, &sm.bsel, &sm.ncand);   // ends with a CTA barrier
  const int ncand = sm.ncand;
  if (ncand > FCAP) {
    if (p0 < p1 && tid == 0) tc::mbar_wait(&sm.bar, 0, nullptr);   // no copy may land after the exit
    if (rank == 0) radix_select_row(sc, n, k, out);
    return;
  }
  // key(x) >= lo  <=>  x >= lo_f for every score that is not a NaN (a NaN
  // key would make the lists disagree with the histogram: radix path)
  const uint32_t lo = static_cast<uint32_t>(sm.bsel) << (32 - kDecHistBits);
  const float lo_f = key_float(lo);
  // Thread t lists the scores [4 SUNR t, 4 SUNR (t + 1)) of each pass, so
  // the pass's position order is the thread order.  A thread marks its
  // candidates in a bit mask as it reads them (independent 16-byte reads,
  // 272 bytes apart: distinct banks within each 8-thread phase) and then
  // visits only the marked ones, about 2 of its 68 scores on average.
  int run = 0;
  bool ok = true;
  uint32_t phase = 0;
  for (int base = p0; base < p1; base += SPASS, phase ^= 1u) {
    if (base != p0) issue(base);
    if (!tc::mbar_wait(&sm.bar, phase, nullptr)) {
      ok = false;                                // a copy may still land: waited for again before the exit
      if (status) atomicExch(status, kDevTimeout);
    }
    const int t0 = 4 * SUNR * tid;               // this thread's first entry of the pass
    const int nmine = max(0, min(4 * SUNR, p1 - base - t0));
    const float4* mine = reinterpret_cast<const float4*>(&sm.buf[t0]);
    uint32_t m[(SUNR + 7) / 8] = {};             // bit 4 j + c: entry 4 j + c is a candidate
#pragma unroll
    for (int j = 0; j < SUNR; ++j) {
      const float4 x = mine[j];
      const uint32_t f = (x.x >= lo_f ? 1u : 0u) | (x.y >= lo_f ? 2u : 0u) | (x.z >= lo_f ? 4u : 0u) |
                         (x.w >= lo_f ? 8u : 0u);
      m[j >> 3] |= f << (4 * (j & 7));
    }
    // entries past the part (the last thread of the row's end) are dropped
#pragma unroll
    for (int w = 0; w < (SUNR + 7) / 8; ++w) {
      const int keep = nmine - 32 * w;
      m[w] &= keep >= 32 ? 0xFFFFFFFFu : (keep <= 0 ? 0u : (1u << keep) - 1u);
    }
    int cl = 0;
#pragma unroll
    for (int w = 0; w < (SUNR + 7) / 8; ++w) cl += __popc(m[w]);
    int tot;
    // (its barriers also keep every thread's reads of buf ahead of the next pass's copies)
    int off = run + block_exclusive_scan(cl, sm.scr.warp_sums, STHREADS, tot, tid, BlockSync());
#pragma unroll
    for (int w = 0; w < (SUNR + 7) / 8; ++w) {
      for (uint32_t mw = m[w]; mw != 0u; mw &= mw - 1u, ++off) {
        const int i = 32 * w + __ffs(mw) - 1;
        if (off < FCAP) {
          sm.key[off] = float_key(sm.buf[t0 + i]);
          sm.pos[off] = base + t0 + i;
        }
      }
    }
    run += tot;
    ok = __syncthreads_and(ok);                  // one decision for the CTA
    if (!ok) break;
  }
  if (tid == 0) sm.count = ok ? run : -1;        // a CTA whose copy gave up sends the row to the radix path
  cluster.sync();                                // every CTA's list and count are complete
  // this CTA's list goes to CTA 0's, after the lists of the CTAs before it
  int before = 0, total = 0;
#pragma unroll
  for (int r = 0; r < SCL; ++r) {
    const int c = r == rank ? sm.count : *cluster.map_shared_rank(&sm.count, r);
    if (c < 0) total = -1 << 30;
    if (r < rank) before += c;
    total += c;
  }
  const bool good = total == ncand;              // then every count is within FCAP too
  if (good && rank > 0) {
    uint32_t* dk = cluster.map_shared_rank(sm.key, 0);
    int* dp = cluster.map_shared_rank(sm.pos, 0);
    for (int i = tid; i < sm.count; i += STHREADS) {
      dk[before + i] = sm.key[i];
      dp[before + i] = sm.pos[i];
    }
  }
  cluster.sync();                                // CTA 0 holds every list
  if (!ok && tid == 0) tc::mbar_wait(&sm.bar, phase, nullptr);
  if (rank != 0) return;
  if (!good) {                                   // lists disagree with the histogram: the general path
    radix_select_row(sc, n, k, out);
    return;
  }
  if (ncand > k)
    cut_bin_to_out(sm.key, sm.pos, ncand, k, lo, ncand - hrow[sm.bsel], reinterpret_cast<int*>(sm.buf), &sm.scr, out);
  else
    for (int j = tid; j < k; j += STHREADS) out[j] = sm.pos[j];
}

// Clears the score histograms before the scorer adds into them.  A kernel
// (not a memset) so that the launches around it keep their programmatic
// dependent launch edges; it waits for the kernel before it, which may
// still read the previous call's histograms.
__global__ void __launch_bounds__(256) zero_words_kernel(uint4* p, size_t n16) {
  grid_dep_wait();
  grid_dep_trigger();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Whether clusters of SCL CTAs with the clustered select's shared memory fit
// the device (asked once per process; otherwise the one-CTA select runs).
bool cluster_select_ok() {
  static int ok = -1;
  if (ok < 0) {
    int v = 0, n = 0;
    const size_t smem = sizeof(ClusterSelSmem);
    cudaError_t q = cudaFuncSetAttribute(select_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (q == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(SCL, 1);
      cfg.blockDim = dim3(STHREADS);
      cfg.dynamicSmemBytes = smem;
      q = cudaOccupancyMaxActiveClusters(&n, select_cluster_kernel, &cfg);
      if (q == cudaSuccess && n > 0) v = 1;
    }
    if (q != cudaSuccess) cudaGetLastError();    // a refused query leaves no error behind
    ok = v;
  }
  return ok == 1;
}

cudaError_t launch_cluster_select(const DecWs& d, const IndexerArgs& a, int* dev_status, cudaStream_t st) {
  const int n = a.q_pos0 + 1;                    // one row per sequence (T = 1)
  const size_t smem = sizeof(ClusterSelSmem);
  const cudaError_t e = cudaFuncSetAttribute(select_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(select_cluster_kernel, dim3(SCL, a.B), dim3(STHREADS), smem, st,
                    static_cast<const float*>(d.scores), d.pitch, static_cast<const int*>(d.hist), a.idx, n, a.k,
                    dev_status);
}

template <int D>
cudaError_t launch_scores(const IndexerArgs& a, float* scores, size_t pitch, cudaStream_t st) {
  const int h_pad = ((a.H + 15) / 16) * 16;
  const size_t smem = sizeof(DecodeSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(decode_scores_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int max_keys = a.q_pos0 + a.T;          // the last row's causal count
  dim3 grid((max_keys + DKT - 1) / DKT, a.B * a.T);
  decode_scores_kernel<D><<<grid, DTHREADS, smem, st>>>(a, scores, h_pad, pitch);
  return cudaGetLastError();
}

}  // namespace

size_t indexer_decode_ws_bytes(int B, int T, int S) { return (size_t)B * T * row_pitch(S) * sizeof(float); }

size_t indexer_decode_ws_fast_bytes(int B, int T, int S) {
  size_t total = 0;
  carve_ws(nullptr, B * T, S, &total);
  return total;
}

cudaError_t launch_indexer_decode(const IndexerArgs& a, void* ws, size_t ws_bytes, int* dev_status,
                                  cudaStream_t st) {
  if (ws_bytes < indexer_decode_ws_bytes(a.B, a.T, a.S)) return cudaErrorInvalidValue;
  float* scores = reinterpret_cast<float*>(ws);
  const size_t pitch = row_pitch(a.S);
  cudaError_t e;
  if (indexer_decode_tc_supported(a)) {
    size_t need = 0;
    const DecWs d = carve_ws(ws, a.B * a.T, a.S, &need);
    if (ws_bytes >= need && cluster_select_ok()) {
      // histogram built by the scorer, then the clustered select
      // rows * HBINS ints: a whole number of 16-byte words (HBINS is a multiple of 4)
      const size_t n16 = static_cast<size_t>(a.B) * a.T * HBINS / 4;
      e = launch_pdl(zero_words_kernel, dim3(static_cast<unsigned>((n16 + 255) / 256 < 148 ? (n16 + 255) / 256 : 148)),
                     dim3(256), 0, st, reinterpret_cast<uint4*>(d.hist), n16);
      if (e != cudaSuccess) return e;
      e = launch_indexer_decode_tc(a, scores, pitch, d.hist, dev_status, st);
      if (e != cudaSuccess) return e;
      return launch_cluster_select(d, a, dev_status, st);
    }
    e = launch_indexer_decode_tc(a, scores, pitch, nullptr, dev_status, st);
    if (e != cudaSuccess) return e;
    return launch_select(scores, pitch, a, st);
  }
  switch (a.D) {
    case 32: e = launch_scores<32>(a, scores, pitch, st); break;
    case 64: e = launch_scores<64>(a, scores, pitch, st); break;
    case 128: e = launch_scores<128>(a, scores, pitch, st); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return launch_select(scores, pitch, a, st);
}

}  // namespace ic
