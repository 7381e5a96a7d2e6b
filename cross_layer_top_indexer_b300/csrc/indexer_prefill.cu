// Fused lightning indexer + streaming top-k for prefill (many query rows).
//
// Score (DeepSeek-Sparse-Attention indexer, used by IndexCache's Full
// layers; notes page "NLP--IndexCache", section "背景 & 问题提出"):
//     I[t,s] = sum_h w[t,h] * ReLU(q[t,h,:] . kI[s,:])   for s <= pos(t)
// (times k_scale[s] for e4m3 keys: a positive factor commutes with ReLU).
//
// One CTA owns QPB consecutive query rows of one sequence and streams the
// causal key rows in tiles of KT.  Per tile the tensor cores produce the
// [keys x (query, head)] dot products (keys on the MMA M axis, so a thread
// ends up holding whole head rows of one key and the head sum is a register
// reduction plus two quad shuffles); the weighted ReLU sum is formed in
// registers and the score row of the tile goes to shared memory only.
//
// Streaming top-k per query: a candidate list in shared memory, kept in
// ascending position order, and a threshold tau = smallest kept score after
// the last compaction.  A key enters iff its score is strictly above tau:
// keys arrive in ascending position, so a key that only ties tau loses to
// the kept entry (lower position).  When the list could overflow during the
// next tile it is cut back to the k best by an exact radix select.  After
// the last tile the list holds the answer in ascending order.
#include "ic_common.cuh"
#include "ic_kernels.h"
#include "topk_select.cuh"

namespace ic {
namespace {

constexpr int QPB = 4;                 // query rows per CTA
constexpr int KT = 128;                // key rows per tile
constexpr int NTHREADS = 256;          // 8 warps: 4 key groups x 2 query pairs
constexpr int CAP = kMaxK + 512;       // candidate slots per query row
constexpr int SEG = CAP / NTHREADS;    // entries per thread in a compaction
constexpr int HMAX = 64;

template <int D>
struct PrefillSmem {
  static constexpr int P = D + 8;      // padded row pitch (bf16) against bank conflicts
  __nv_bfloat16 qs[QPB][HMAX][P];
  __nv_bfloat16 ks[KT][P];
  float wsm[QPB][HMAX];
  float tsc[QPB][KT];
  float ksc[KT];
  float cand_s[QPB][CAP];
  int cand_p[QPB][CAP];
  int cnt[QPB];
  uint32_t tau[QPB];
  int wc[2][4];
  SelectScratch scr;
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
indexer_prefill_kernel(IndexerArgs a, int n_groups, int h_pad) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<PrefillSmem<D>*>(smem_raw);

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int g = n_groups - 1 - (int)blockIdx.x;   // longest causal range first
  const int b = blockIdx.y;
  const int t0 = g * QPB;
  const int nq = min(QPB, a.T - t0);
  const int pos0 = a.q_pos0 + t0;                 // position of the CTA's first row
  const int n_keys = pos0 + nq;                   // keys 0 .. last row's position
  int32_t* out = a.idx + ((size_t)b * a.T + t0) * a.k;

  if (n_keys <= a.k) {
    // Every causal position of every row is selected.
    for (int i = tid; i < nq * a.k; i += NTHREADS) {
      const int qi = i / a.k, j = i - qi * a.k;
      out[i] = (j <= pos0 + qi) ? j : -1;
    }
    return;
  }

  // ---- stage the CTA's queries and head weights ----
  {
    const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(a.q);
    constexpr int CH = D / 8;                       // 16-byte chunks per row
    for (int i = tid; i < QPB * h_pad * CH; i += NTHREADS) {
      const int c = i % CH, h = (i / CH) % h_pad, qi = i / (CH * h_pad);
      const bool ok = qi < nq && h < a.H;
      const __nv_bfloat16* src = ok ? qg + (((size_t)b * a.T + t0 + qi) * a.H + h) * D + c * 8 : qg;
      cp_async16(&sm.qs[qi][h][c * 8], src, ok);
    }
    cp_async_commit();
    for (int i = tid; i < QPB * HMAX; i += NTHREADS) {
      const int qi = i / HMAX, h = i % HMAX;
      sm.wsm[qi][h] = (qi < nq && h < a.H) ? a.w[((size_t)b * a.T + t0 + qi) * a.H + h] : 0.0f;
    }
    if (tid < QPB) { sm.cnt[tid] = 0; sm.tau[tid] = 0u; }
  }

  const int kg = wid & 3;            // key group: rows kg*32 .. kg*32+31 of the tile
  const int qh = wid >> 2;           // query pair: rows 2qh, 2qh+1
  const int n_tiles_h = h_pad / 8;   // n-tiles of 8 heads

  for (int s0 = 0; s0 < n_keys; s0 += KT) {
    // ---- key tile -> shared (bf16) ----
    if (!a.e4m3) {
      const __nv_bfloat16* kg_ = reinterpret_cast<const __nv_bfloat16*>(a.kI) + (size_t)b * a.S_cap * D;
      constexpr int CH = D / 8;
      for (int i = tid; i < KT * CH; i += NTHREADS) {
        const int r = i / CH, c = i % CH;
        const int s = s0 + r;
        const bool ok = s < n_keys;
        cp_async16(&sm.ks[r][c * 8], ok ? kg_ + (size_t)s * D + c * 8 : kg_, ok);
      }
      cp_async_commit();
      if (tid < KT) sm.ksc[tid] = 1.0f;
    } else {
      const uint8_t* kg8 = reinterpret_cast<const uint8_t*>(a.kI) + (size_t)b * a.S_cap * D;
      constexpr int CH = D / 16;                    // 16 e4m3 per load
      for (int i = tid; i < KT * CH; i += NTHREADS) {
        const int r = i / CH, c = i % CH;
        const int s = s0 + r;
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
      if (tid < KT) {
        const int s = s0 + tid;
        sm.ksc[tid] = s < n_keys ? a.kscale[(size_t)b * a.S_cap + s] : 0.0f;
      }
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- tensor-core scores of this tile -> sm.tsc ----
#pragma unroll 1
    for (int qq = 0; qq < 2; ++qq) {
      const int qi = 2 * qh + qq;
      if (qi >= nq) break;
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
                      &sm.ks[kg * 32 + m * 16 + (lane & 15)][kk * 16 + (lane >> 4) * 8]);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          if (2 * np < n_tiles_h) {
            const int mat = lane >> 3;
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(b0, b1, b2, b3,
                        &sm.qs[qi][np * 16 + (mat >> 1) * 8 + (lane & 7)][kk * 16 + (mat & 1) * 8]);
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              mma_bf16_16816(acc[m][2 * np], af[m][0], af[m][1], af[m][2], af[m][3], b0, b1);
              mma_bf16_16816(acc[m][2 * np + 1], af[m][0], af[m][1], af[m][2], af[m][3], b2, b3);
            }
          }
        }
      }
      // weighted ReLU over this lane's heads, then over the quad
#pragma unroll
      for (int m = 0; m < 2; ++m) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float part = 0.0f;
#pragma unroll
          for (int n = 0; n < 8; ++n) {
            if (n < n_tiles_h) {
              const int h = n * 8 + 2 * (lane & 3);
              part = fmaf(sm.wsm[qi][h], fmaxf(acc[m][n][2 * half], 0.0f), part);
              part = fmaf(sm.wsm[qi][h + 1], fmaxf(acc[m][n][2 * half + 1], 0.0f), part);
            }
          }
          part += __shfl_xor_sync(0xffffffffu, part, 1);
          part += __shfl_xor_sync(0xffffffffu, part, 2);
          if ((lane & 3) == 0) {
            const int r = kg * 32 + m * 16 + half * 8 + (lane >> 2);
            sm.tsc[qi][r] = part * sm.ksc[r];
          }
        }
      }
    }
    __syncthreads();

    // ---- cut back any list that could overflow during this tile ----
#pragma unroll 1
    for (int qi = 0; qi < nq; ++qi) {
      const int c = sm.cnt[qi];
      if (c > CAP - KT) {
        select_keep_topk<NTHREADS, SEG>(sm.cand_s[qi], sm.cand_p[qi], c, a.k, &sm.scr, tid, BlockSync(),
                                        sm.tau[qi], 0xFFFFFFFFu, static_cast<uint32_t>(pos0 + qi));
        if (tid == 0) { sm.cnt[qi] = a.k; sm.tau[qi] = sm.scr.tau; }
        __syncthreads();
      }
    }

    // ---- ordered insertion of the keys above tau ----
    {
      const int key = tid & (KT - 1), half = tid >> 7, w4 = key >> 5;
      const int s = s0 + key;
#pragma unroll 1
      for (int r = 0; r < 2; ++r) {
        const int qi = half + 2 * r;
        bool take = false;
        float sc = 0.0f;
        if (qi < nq) {
          sc = sm.tsc[qi][key];
          take = (s <= pos0 + qi) && (float_key(sc) > sm.tau[qi]);
        }
        const unsigned bal = __ballot_sync(0xffffffffu, take);
        if (lane == 0) sm.wc[half][w4] = __popc(bal);
        __syncthreads();
        if (qi < nq) {
          int off = __popc(bal & ((1u << lane) - 1u));
          for (int j = 0; j < w4; ++j) off += sm.wc[half][j];
          const int base = sm.cnt[qi];
          if (take) { sm.cand_s[qi][base + off] = sc; sm.cand_p[qi][base + off] = s; }
        }
        __syncthreads();
        if (key == 0 && qi < nq)
          sm.cnt[qi] += sm.wc[half][0] + sm.wc[half][1] + sm.wc[half][2] + sm.wc[half][3];
        __syncthreads();
      }
    }
  }

  // ---- final cut to k and write-out (already in ascending position order) ----
#pragma unroll 1
  for (int qi = 0; qi < nq; ++qi) {
    const int c = sm.cnt[qi];
    if (c > a.k) {
      select_keep_topk<NTHREADS, SEG>(sm.cand_s[qi], sm.cand_p[qi], c, a.k, &sm.scr, tid, BlockSync(),
                                      sm.tau[qi], 0xFFFFFFFFu, static_cast<uint32_t>(pos0 + qi));
      if (tid == 0) sm.cnt[qi] = a.k;
      __syncthreads();
    }
    const int n = min(c, a.k);
    int32_t* row = out + (size_t)qi * a.k;
    for (int j = tid; j < a.k; j += NTHREADS) row[j] = j < n ? sm.cand_p[qi][j] : -1;
  }
}

template <int D>
cudaError_t launch_d(const IndexerArgs& a, cudaStream_t st) {
  const int n_groups = (a.T + QPB - 1) / QPB;
  const int h_pad = ((a.H + 15) / 16) * 16;
  const size_t smem = sizeof(PrefillSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(indexer_prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(n_groups, a.B);
  indexer_prefill_kernel<D><<<grid, NTHREADS, smem, st>>>(a, n_groups, h_pad);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_prefill(const IndexerArgs& a, int* /*dev_status*/, cudaStream_t st) {
  switch (a.D) {
    case 32: return launch_d<32>(a, st);
    case 64: return launch_d<64>(a, st);
    case 128: return launch_d<128>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ic
