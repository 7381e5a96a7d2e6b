// Sparse core attention over the selected key/value rows.
//
// IndexCache leaves core attention as in DeepSeek Sparse Attention: each
// query attends only to its k selected tokens, cutting the cost from O(L^2)
// to O(Lk) (notes page "NLP--IndexCache", section "背景 & 问题提出").  All
// query heads read the one shared K/V head.
//
// One CTA per (query row, split).  The CTA loads its share of the index row
// into shared memory once, walks it in chunks of KC positions, gathers those
// K and V rows into shared memory through registers (double buffered: the
// next chunk's loads are in flight during the current chunk's math, and
// depend on no global load of their own index), and runs a
// flash-style online softmax on the tensor cores with the heads on the MMA
// M axis.  Four warps: two head tiles of 16 x two halves of every chunk; the
// halves are merged at the end.  With one split the CTA writes bf16 O;
// with several it writes fp32 partial (max, sum, unnormalised O) to the
// workspace and a second kernel merges the splits.
#include <math.h>

#include "ic_common.cuh"
#include "ic_kernels.h"

namespace ic {
namespace {

constexpr int KC = 64;          // index positions per chunk
constexpr int ATHREADS = 128;   // 4 warps
constexpr int HQMAX = 32;
constexpr int DHMAX = 128;      // the tcgen05 kernel's head dim (its partials use this layout)
constexpr float kLog2e = 1.4426950408889634f;

template <int DH>
struct AttnSmem {
  static constexpr int P = DH + 8;
  __nv_bfloat16 q[HQMAX][P];
  __nv_bfloat16 k[2][KC][P];
  __nv_bfloat16 v[2][KC][P];
  int idx[2][KC];
  int32_t sidx[kMaxK];         // this split's index positions, loaded once
  float m_x[HQMAX];            // merge buffers for the second key half
  float l_x[HQMAX];
  float o_x[HQMAX][DH + 4];
};

struct Partial {               // per (row, split): m[HQMAX], l[HQMAX], o[HQMAX][DH]
  __host__ __device__ static size_t floats(int dh) { return (size_t)2 * HQMAX + (size_t)HQMAX * dh; }
};

// Chunk gathers go through registers: each thread loads its 16-byte pieces
// of the chunk's K and V rows with plain global loads (the next chunk's are
// in flight while the current one is computed), then stores them into the
// shared-memory buffer.  Plain loads sustain several times the random-row
// gather rate of cp.async on this GPU.
template <int DH>
struct ChunkRegs {
  static constexpr int CH = DH / 8;                 // 16-byte pieces per row
  static constexpr int N = KC * CH / ATHREADS;      // pieces per thread per tensor
  uint4 k[N], v[N];
  int s[N];                                         // source row of each piece (-1: empty slot)
};

// sidx: the split's index positions in shared memory, from position jb on.
template <int DH>
__device__ __forceinline__ void gather_load(ChunkRegs<DH>& g, const int32_t* sidx, int jb, int j0, int k,
                                            const __nv_bfloat16* Kb, const __nv_bfloat16* Vb, int S, int tid) {
  constexpr int CH = ChunkRegs<DH>::CH;
#pragma unroll
  for (int u = 0; u < ChunkRegs<DH>::N; ++u) {
    const int i = tid + ATHREADS * u;
    const int r = i / CH, c = i % CH;
    const int j = j0 + r;
    const int src = j < k ? sidx[j - jb] : -1;
    const bool ok = src >= 0 && src < S;   // an index outside [0, S) is an empty slot: never read
    g.s[u] = ok ? src : -1;
    g.k[u] = ok ? __ldcg(reinterpret_cast<const uint4*>(Kb + (size_t)src * DH) + c) : make_uint4(0u, 0u, 0u, 0u);
    g.v[u] = ok ? __ldcg(reinterpret_cast<const uint4*>(Vb + (size_t)src * DH) + c) : make_uint4(0u, 0u, 0u, 0u);
  }
}

template <int DH>
__device__ __forceinline__ void gather_store(AttnSmem<DH>& sm, int buf, const ChunkRegs<DH>& g, int tid) {
  constexpr int CH = ChunkRegs<DH>::CH;
#pragma unroll
  for (int u = 0; u < ChunkRegs<DH>::N; ++u) {
    const int i = tid + ATHREADS * u;
    const int r = i / CH, c = i % CH;
    *reinterpret_cast<uint4*>(&sm.k[buf][r][c * 8]) = g.k[u];
    *reinterpret_cast<uint4*>(&sm.v[buf][r][c * 8]) = g.v[u];
    if (c == 0) sm.idx[buf][r] = g.s[u];
  }
}

template <int DH>
__global__ void __launch_bounds__(ATHREADS)
sparse_attn_kernel(AttnArgs a, int nsplit, int chunks_per_split, float* partials) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<AttnSmem<DH>*>(smem_raw);
  constexpr int NT = DH / 8;       // n-tiles of the output

  grid_dep_wait();                 // Q, the index row and K/V may come from the kernels just before
  grid_dep_trigger();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int row = blockIdx.x;      // b * T + t
  const int split = blockIdx.y;
  const int b = row / a.T;
  const int mh = wid & 1, kh = wid >> 1;
  const int hq_tiles = (a.Hq + 15) / 16;
  const int32_t* irow = a.idx + (size_t)row * a.k;
  const __nv_bfloat16* Kb = reinterpret_cast<const __nv_bfloat16*>(a.K) + (size_t)b * a.S_cap * DH;
  const __nv_bfloat16* Vb = reinterpret_cast<const __nv_bfloat16*>(a.V) + (size_t)b * a.S_cap * DH;

  // stage Q (zero rows past Hq)
  {
    const __nv_bfloat16* Qg = reinterpret_cast<const __nv_bfloat16*>(a.Q) + (size_t)row * a.Hq * DH;
    constexpr int CH = DH / 8;
    for (int i = tid; i < HQMAX * CH; i += ATHREADS) {
      const int h = i / CH, c = i % CH;
      const bool ok = h < a.Hq;
      cp_async16(&sm.q[h][c * 8], ok ? Qg + (size_t)h * DH + c * 8 : Qg, ok);
    }
    cp_async_commit();
  }
  const int n_chunks_total = (a.k + KC - 1) / KC;
  const int c_begin = split * chunks_per_split;
  const int c_end = min(n_chunks_total, c_begin + chunks_per_split);

  // the split's index positions, in one round trip
  const int jb = c_begin * KC, je = min(a.k, c_end * KC);
  for (int j = jb + tid; j < je; j += ATHREADS) sm.sidx[j - jb] = __ldg(irow + j);
  __syncthreads();
  ChunkRegs<DH> gr;
  if (c_begin < c_end) {
    gather_load<DH>(gr, sm.sidx, jb, c_begin * KC, a.k, Kb, Vb, a.S, tid);
    gather_store<DH>(sm, 0, gr, tid);
  }
  cp_async_wait<0>();
  __syncthreads();

  const bool active = mh < hq_tiles;
  // Q fragments of this warp's 16 heads, all of DH
  uint32_t qf[DH / 16][4];
  if (active) {
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk)
      ldmatrix_x4(qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3],
                  &sm.q[mh * 16 + (lane & 15)][kk * 16 + (lane >> 4) * 8]);
  }
  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int j = 0; j < 4; ++j) o[n][j] = 0.0f;
  float m_r[2] = {-INFINITY, -INFINITY};   // running max (log2 domain), rows g and g+8
  float l_r[2] = {0.0f, 0.0f};
  const float sl2 = a.scale * kLog2e;

  for (int c = c_begin; c < c_end; ++c) {
    const int buf = (c - c_begin) & 1;
    // the next chunk's loads are in flight while this one is computed
    if (c + 1 < c_end) gather_load<DH>(gr, sm.sidx, jb, (c + 1) * KC, a.k, Kb, Vb, a.S, tid);
    if (active) {
      // scores for this warp's 32 keys of the chunk: 4 n-tiles of 8 keys
      float s[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[n][j] = 0.0f;
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const int mat = lane >> 3;
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(b0, b1, b2, b3,
                      &sm.k[buf][kh * 32 + np * 16 + (mat >> 1) * 8 + (lane & 7)][kk * 16 + (mat & 1) * 8]);
          mma_bf16_16816(s[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
          mma_bf16_16816(s[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
        }
      }
      // mask empty slots, scale into the log2 domain, row max
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < 4; ++n) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int key = kh * 32 + n * 8 + 2 * (lane & 3) + (j & 1);
          const float v = sm.idx[buf][key] >= 0 ? s[n][j] * sl2 : -INFINITY;
          s[n][j] = v;
          mx[j >> 1] = fmaxf(mx[j >> 1], v);
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      }
      float alpha[2], mref[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float mnew = fmaxf(m_r[r], mx[r]);
        mref[r] = mnew == -INFINITY ? 0.0f : mnew;
        alpha[r] = exp2f(m_r[r] - mref[r]);     // 0 when m_r is -inf
        m_r[r] = mnew;
      }
      float rs[2] = {0.0f, 0.0f};
#pragma unroll
      for (int n = 0; n < 4; ++n) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float p = exp2f(s[n][j] - mref[j >> 1]);
          s[n][j] = p;
          rs[j >> 1] += p;
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
        rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
        l_r[r] = l_r[r] * alpha[r] + rs[r];
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][0] *= alpha[0]; o[n][1] *= alpha[0];
        o[n][2] *= alpha[1]; o[n][3] *= alpha[1];
      }
      // O += P V : two k-steps of 16 keys
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const uint32_t p0 = pack_bf16x2(s[2 * ks][0], s[2 * ks][1]);
        const uint32_t p1 = pack_bf16x2(s[2 * ks][2], s[2 * ks][3]);
        const uint32_t p2 = pack_bf16x2(s[2 * ks + 1][0], s[2 * ks + 1][1]);
        const uint32_t p3 = pack_bf16x2(s[2 * ks + 1][2], s[2 * ks + 1][3]);
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          const int mat = lane >> 3;
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(b0, b1, b2, b3,
                            &sm.v[buf][kh * 32 + ks * 16 + (mat & 1) * 8 + (lane & 7)][np * 16 + (mat >> 1) * 8]);
          mma_bf16_16816(o[2 * np], p0, p1, p2, p3, b0, b1);
          mma_bf16_16816(o[2 * np + 1], p0, p1, p2, p3, b2, b3);
        }
      }
    }
    if (c + 1 < c_end) gather_store<DH>(sm, buf ^ 1, gr, tid);
    __syncthreads();
  }

  // merge the two key halves: warps kh=1 publish, warps kh=0 combine
  const int g = lane >> 2, cq = lane & 3;
  if (active && kh == 1) {
    if (cq == 0) {
      sm.m_x[mh * 16 + g] = m_r[0]; sm.l_x[mh * 16 + g] = l_r[0];
      sm.m_x[mh * 16 + g + 8] = m_r[1]; sm.l_x[mh * 16 + g + 8] = l_r[1];
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      sm.o_x[mh * 16 + g][n * 8 + 2 * cq] = o[n][0];
      sm.o_x[mh * 16 + g][n * 8 + 2 * cq + 1] = o[n][1];
      sm.o_x[mh * 16 + g + 8][n * 8 + 2 * cq] = o[n][2];
      sm.o_x[mh * 16 + g + 8][n * 8 + 2 * cq + 1] = o[n][3];
    }
  }
  __syncthreads();
  if (!(active && kh == 0)) return;
  float fa[2], fb[2], mm[2], ll[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int h = mh * 16 + g + 8 * r;
    const float m1 = sm.m_x[h], l1 = sm.l_x[h];
    const float M = fmaxf(m_r[r], m1);
    const float Mr = M == -INFINITY ? 0.0f : M;
    fa[r] = exp2f(m_r[r] - Mr);
    fb[r] = exp2f(m1 - Mr);
    mm[r] = M;
    ll[r] = l_r[r] * fa[r] + l1 * fb[r];
  }
  if (nsplit == 1) {
    __nv_bfloat16* Ob = reinterpret_cast<__nv_bfloat16*>(a.O) + (size_t)row * a.Hq * DH;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int h = mh * 16 + g + 8 * r;
      if (h >= a.Hq) continue;
      const float inv = ll[r] > 0.0f ? 1.0f / ll[r] : 0.0f;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int d = n * 8 + 2 * cq;
        const float v0 = (o[n][2 * r] * fa[r] + sm.o_x[h][d] * fb[r]) * inv;
        const float v1 = (o[n][2 * r + 1] * fa[r] + sm.o_x[h][d + 1] * fb[r]) * inv;
        *reinterpret_cast<uint32_t*>(Ob + (size_t)h * DH + d) = pack_bf16x2(v0, v1);
      }
    }
  } else {
    float* pbase = partials + ((size_t)row * nsplit + split) * Partial::floats(DH);
    float* pm = pbase;
    float* pl = pbase + HQMAX;
    float* po = pbase + 2 * HQMAX;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int h = mh * 16 + g + 8 * r;
      if (cq == 0) { pm[h] = mm[r]; pl[h] = ll[r]; }
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int d = n * 8 + 2 * cq;
        po[(size_t)h * DH + d] = o[n][2 * r] * fa[r] + sm.o_x[h][d] * fb[r];
        po[(size_t)h * DH + d + 1] = o[n][2 * r + 1] * fa[r] + sm.o_x[h][d + 1] * fb[r];
      }
    }
  }
}

// Merge the splits of one (row, head): block = DH threads, grid = (rows, Hq).
// Every split's values are loaded before the first is used, so the loads
// overlap (one round trip instead of one per split).
constexpr int MAX_SPLITS = (kMaxK + KC - 1) / KC;

template <int DH>
__global__ void attn_combine_kernel(const float* partials, int nsplit, int Hq, void* O) {
  grid_dep_wait();
  grid_dep_trigger();
  const int row = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const size_t stride = Partial::floats(DH);
  const float* base = partials + (size_t)row * nsplit * stride;
  float mv[MAX_SPLITS], lv[MAX_SPLITS], ov[MAX_SPLITS];
#pragma unroll
  for (int s = 0; s < MAX_SPLITS; ++s) {
    if (s < nsplit) {
      const float* p = base + s * stride;
      mv[s] = p[h];
      lv[s] = p[HQMAX + h];
      ov[s] = p[2 * HQMAX + (size_t)h * DH + d];
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int s = 0; s < MAX_SPLITS; ++s)
    if (s < nsplit) M = fmaxf(M, mv[s]);
  const float Mr = M == -INFINITY ? 0.0f : M;
  float l = 0.0f, acc = 0.0f;
#pragma unroll
  for (int s = 0; s < MAX_SPLITS; ++s) {
    if (s < nsplit) {
      const float f = exp2f(mv[s] - Mr);
      l += lv[s] * f;
      acc += ov[s] * f;
    }
  }
  const float v = l > 0.0f ? acc / l : 0.0f;
  reinterpret_cast<__nv_bfloat16*>(O)[((size_t)row * Hq + h) * DH + d] = __float2bfloat16_rn(v);
}

// Splits of the k positions of a row: about four chunks per CTA (fewer
// partial states to write and merge), but at least one CTA per SM in all.
// Measured at the decode workload (32 rows, k = 2048, 32 chunks): 1, 2, 4, 8
// and 16 chunks per CTA take 28.0, 21.7, 19.7, 24.9 and 39.8 us.
int pick_splits(int rows, int k) {
  const int n_chunks = (k + KC - 1) / KC;
  if (rows >= 2 * 148) return 1;
  const int by_work = (n_chunks + 3) / 4;
  const int by_sms = (148 + rows - 1) / rows;
  const int want = by_work > by_sms ? by_work : by_sms;
  return want < n_chunks ? want : n_chunks;
}

template <int DH>
cudaError_t launch_dh(const AttnArgs& a, void* ws, size_t ws_bytes, cudaStream_t st) {
  const int rows = a.B * a.T;
  int nsplit = pick_splits(rows, a.k);
  const int n_chunks = (a.k + KC - 1) / KC;
  const int cps = (n_chunks + nsplit - 1) / nsplit;
  nsplit = (n_chunks + cps - 1) / cps;
  const size_t need = nsplit > 1 ? (size_t)rows * nsplit * Partial::floats(DH) * sizeof(float) : 0;
  if (need > ws_bytes || nsplit > MAX_SPLITS) return cudaErrorInvalidValue;
  const size_t smem = sizeof(AttnSmem<DH>);
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(rows, nsplit);
  e = launch_pdl(sparse_attn_kernel<DH>, grid, dim3(ATHREADS), smem, st, a, nsplit, cps, reinterpret_cast<float*>(ws));
  if (e != cudaSuccess || nsplit == 1) return e;
  return launch_pdl(attn_combine_kernel<DH>, dim3(rows, a.Hq), dim3(DH), 0, st, reinterpret_cast<const float*>(ws),
                    nsplit, a.Hq, a.O);
}

}  // namespace

size_t attn_ws_bytes(int B, int T, int Hq, int Dh, int k) {
  const int rows = B * T;
  const int n_chunks = (k + KC - 1) / KC;
  int nsplit = pick_splits(rows, k);
  const int cps = (n_chunks + nsplit - 1) / nsplit;
  nsplit = (n_chunks + cps - 1) / cps;
  // the tcgen05 kernel's shares, when it takes the shapes (the key-cache
  // size does not change the count, so the workspace covers either path)
  AttnArgs t{};
  t.B = B;
  t.T = T;
  t.Hq = Hq;
  t.Dh = Dh;
  t.k = k;
  const int tsplit = sparse_attn_tc_splits(t);
  const int most = tsplit > nsplit ? tsplit : nsplit;
  return most > 1 ? (size_t)rows * most * Partial::floats(Dh) * sizeof(float) : 0;
}

cudaError_t launch_sparse_attn(const AttnArgs& a, void* ws, size_t ws_bytes, int* dev_status, cudaStream_t st) {
  const int tsplit = sparse_attn_tc_splits(a);
  if (tsplit == 1) return launch_sparse_attn_tc(a, 1, nullptr, dev_status, st);
  if (tsplit > 1) {
    // each row shared among tsplit CTAs of the tcgen05 kernel, then merged:
    // inside the launch (one cluster per row) when the shares fit one per
    // CTA, else by the combine kernel
    if (sparse_attn_tc_cluster_merge(a, tsplit)) return launch_sparse_attn_tc(a, tsplit, nullptr, dev_status, st);
    const int rows = a.B * a.T;
    if ((size_t)rows * tsplit * Partial::floats(DHMAX) * sizeof(float) > ws_bytes) return cudaErrorInvalidValue;
    cudaError_t e = launch_sparse_attn_tc(a, tsplit, reinterpret_cast<float*>(ws), dev_status, st);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_combine_kernel<DHMAX>, dim3(rows, a.Hq), dim3(DHMAX), 0, st,
                      reinterpret_cast<const float*>(ws), tsplit, a.Hq, a.O);
  }
  switch (a.Dh) {
    case 64: return launch_dh<64>(a, ws, ws_bytes, st);
    case 128: return launch_dh<128>(a, ws, ws_bytes, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ic
