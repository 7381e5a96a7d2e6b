// Sparse core attention on the 5th-generation tensor cores (tcgen05 +
// tensor memory), for the production head shape: 32 query heads sharing one
// K/V head of dim 128, bf16.
//
// IndexCache keeps DeepSeek-Sparse-Attention's core attention: each query
// attends only to its k selected tokens, O(L^2) -> O(Lk) (notes page
// "NLP--IndexCache", section "背景 & 问题提出").
//
//   O[t,h,:] = sum_j softmax_j(scale * Q[t,h,:] . K[idx_j,:]) V[idx_j,:]
//
// Every query row gathers its own k K rows and k V rows, so the work per row
// is a pair of skinny products over gathered operands; the bound is the
// gather out of L2, and the design keeps as many gathered bytes in flight as
// shared memory allows.  Keys go on the MMA M axis (128 per tile, TMEM lanes):
//
//   S^T[key, h]  = K_tile (M=128 keys, K-major) x Q^T (N=32 heads, K-major)
//   O^T[d, h]   += V_tile^T (M=128 d, MN-major) x P^T (N=32 heads, MN-major)
//
// so the softmax thread that owns key lane j holds that key's 32 head
// scores, and the output accumulates in TMEM with d on the lanes.
//
// Persistent CTAs (one per SM) walk work items item = blockIdx.x + i*gridDim.x:
// whole query rows, or, with few rows (decode), a range of a row's tiles.  A
// share of a row ends with its reference max, sum and unnormalised O.  When
// the shares fit one per CTA, the CTAs of a row are launched as one thread
// block cluster: each stages its share in shared memory and, after the
// cluster barrier, CTA r merges heads [r HQ/n, (r+1) HQ/n) of the row from
// all the shares through distributed shared memory and writes O.  Otherwise
// the shares go to a workspace and a combine kernel merges them.
// Warp roles (14 warps):
//   warps 0-7  softmax + epilogue in two head groups: warps 0-3 own heads
//              0-15, warps 4-7 heads 16-31 (warp w reads TMEM lane quarter
//              w % 4); thread = key lane for P, = d lane for O.  Thread 0
//              also loads Q (TMA tile) and the index row (bulk copy) two
//              rows ahead into a double buffer.
//   warp 8     MMA issuer of QK^T, over the CTA's tiles in one flat sequence
//   warp 13    MMA issuer of PV (tile g after its P is written); QK^T and PV
//              have an issuing warp each, because the issue of a tcgen05.mma
//              holds its thread about as long as one of these N = 32 MMAs runs
//   warps 9-12 producers: the K rows and the V rows of every tile, gathered
//              with 16-byte asynchronous copies into a ring of 32 KB slots
//              (order K0 V0 K1 V1 ...) in the 128-byte-swizzled operand layout.
//              Every producer thread copies one 16-byte chunk of an eighth of
//              the rows of every slot, then registers an arrival on the slot's
//              mbarrier that fires once its copies have landed
//              (cp.async.mbarrier.arrive.noinc), so the producers never wait
//              for their own copies and run ahead as far as the ring allows;
//              the MMA issuers fence the landed rows into the async proxy
//              after their wait.  Measured on B300 at L = 32768: 3.44 ms per
//              layer, against 3.97 when each slot was published by the
//              producers two slots later (cp.async.wait_group), which tied a
//              slot's publication to the ring's release two tiles back; four
//              producer warps instead of two took 4.17 to 3.94 ms before that.
//
// Empty slots (index -1 or outside [0, S)) are masked in the softmax, so
// their rows may hold anything; they are copied from row (slot position &
// smask), a readable row that differs from slot to slot.  Copying all of
// them from one row made every CTA hit the same L2 lines during the
// early rows (fewer than k causal keys) and slowed the whole launch: 5.02
// against 4.17 ms per layer at L = 32768.  A zero-filling copy, or an integer
// modulo per slot, cost more than it saved.
//
// Softmax (per head group, the groups never wait on each other): the
// reference max m_h of a head is raised only when some score of a tile
// exceeds it by more than kTau (log2 units), so p = 2^(x - m) <= 2^kTau.  The
// common tile therefore needs no cross-lane reduction at all: one vote says
// whether any score crossed the threshold.  Only then (and on a row's first
// tile) is the exact tile maximum reduced across the 128 key lanes, m_h
// moved, and the group's O columns in TMEM rescaled (after the previous PV
// finished).  The sum l_h is kept per thread (one partial per key lane) and
// reduced across the lanes once per row; the row's output (O / l_h, bf16) is
// written at the next row's first tile, from the other O buffer.
//
// Every wait is bounded; a wait that gives up sets the CTA's abort flag and
// the device status word, every role winds down, in-flight MMAs and copies
// are waited for (bounded), and tensor memory is released before returning.
#include <cooperative_groups.h>
#include <math.h>

#include "ic_common.cuh"
#include "ic_kernels.h"
#include "tc_utils.cuh"

namespace ic {
namespace {

// An arrival on bar that fires once every cp.async this thread has issued so
// far has landed (the barrier's count includes it: .noinc).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

constexpr int HQ = 32;                       // query heads (MMA N)
constexpr int DH = 128;                      // head dim
constexpr int KT = 128;                      // keys per tile (MMA M of QK^T)
constexpr int NSLOT = 5;                     // ring slots of 32 KB (a K or a V tile)
constexpr int SLOT_BYTES = KT * DH * 2;      // 32 KB: two 64-column halves, 128-byte swizzle
constexpr int HALF_BYTES = SLOT_BYTES / 2;
constexpr int Q_BYTES = HQ * DH * 2;         // 8 KB
constexpr int P_BYTES = KT * HQ * 2;         // 8 KB: [key][head] bf16, 64-byte swizzle
constexpr int HG = 16;                       // heads per softmax group
constexpr int SOFT_THREADS = 256;            // two groups of 128
constexpr int GROUP_THREADS = 128;
constexpr int MMA_WARP = 8;
constexpr int PROD_WARP0 = 9;
constexpr int PROD_WARPS = 4;
constexpr int PROD_THREADS = PROD_WARPS * 32;
constexpr int PROD_ROWS = KT * 16 / PROD_THREADS;   // rows of a slot each producer thread copies (one chunk each)
constexpr int PV_WARP = PROD_WARP0 + PROD_WARPS;   // 11
constexpr int NTHREADS = (PV_WARP + 1) * 32;
constexpr uint32_t TMEM_COLS = 128;          // S: 2 x 32 columns, O: 2 x 32 columns
// Waiting threads stay suspended in try_wait for up to this long instead of
// polling: 3.34 against 3.37 ms per layer at L = 32768 (fewer issue slots
// taken from the softmax warps by polling producers and MMA issuers).
constexpr uint32_t kWaitHintNs = 20000;
constexpr float kTau = 8.0f;
constexpr float kMInit = -1.0e30f;           // reference max before any valid key (finite: no inf - inf)
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t IDESC_QK = tc::idesc_bf16_f32(KT, HQ);
constexpr uint32_t IDESC_PV = tc::idesc_bf16_f32(DH, HQ) | (1u << 15) | (1u << 16);   // A and B MN-major

struct __align__(1024) AttnTcSmem {
  uint8_t ring[NSLOT][SLOT_BYTES];
  uint8_t qs[2][Q_BYTES];                    // per row buffer: two 64-column halves of 32 x 128 B
  uint8_t ps[2][P_BYTES];
  int32_t idx[2][kMaxK];
  float red[8][HG];                          // per-warp partial max / sum (warp w: group w / 4)
  float m_ref[HQ];
  float alpha[HQ];
  float inv_l[2][HQ];                        // per O buffer
  float m_fin[2][HQ];                        // per O buffer: the reference max at the item's end (log2 units)
  float l_fin[2][HQ];                        //   and the sum of its p
  uint64_t full[NSLOT], empty[NSLOT];
  uint64_t qfull[2];
  uint64_t sfull[2], sempty[2];
  uint64_t pfull[2], pempty[2];
  uint64_t ofull[2], oempty[2];
  uint64_t rowfree[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void set_abort(AttnTcSmem& sm, int* status) {
  sm.abort = 1;
  if (status) atomicExch(status, kDevTimeout);
}

// Lanes i and i + 16 of the warp end with the maximum (or sum) over all 32
// lanes of v[i % 16]: exchange steps of 8, 4, 2, 1 values, then one more
// across the two half-warps.
template <bool kMax>
__device__ __forceinline__ float warp_reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float keep = upper ? v[i + w] : v[i];
      const float send = upper ? v[i] : v[i + w];
      const float got = __shfl_xor_sync(0xffffffffu, send, w);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  const float got = __shfl_xor_sync(0xffffffffu, v[0], 16);
  return kMax ? fmaxf(v[0], got) : v[0] + got;
}

// Q rows and the index row of `row` into buffer qb (completion on qfull[qb]).
__device__ __forceinline__ void load_row_inputs(AttnTcSmem& sm, const CUtensorMap* tm_q, const AttnArgs& a, int row,
                                                int qb) {
  tc::mbar_arrive_expect_tx(&sm.qfull[qb], Q_BYTES + a.k * 4);
  tc::tma_load_2d(sm.qs[qb], tm_q, &sm.qfull[qb], 0, row * HQ);
  tc::tma_load_2d(sm.qs[qb] + Q_BYTES / 2, tm_q, &sm.qfull[qb], 64, row * HQ);
  tc::bulk_g2s(sm.idx[qb], a.idx + static_cast<size_t>(row) * a.k, a.k * 4, &sm.qfull[qb]);
}

// kSplit: each row shared among nsplit CTAs (partials out); otherwise whole
// rows (bf16 O out), with none of the share arithmetic in the loops.
template <bool kSplit>
__global__ void __launch_bounds__(NTHREADS, 1)
sparse_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, AttnArgs a, int nsplit, float* partials,
                      int* status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  AttnTcSmem& sm = *reinterpret_cast<AttnTcSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rows = a.B * a.T;
  const int k = a.k;
  const int nt = (k + KT - 1) / KT;
  // Work items: item i is tiles [j0, j0 + jn) of query row i / nsplit (whole
  // rows when nsplit == 1; every item has at least one tile).  This CTA
  // takes items blockIdx.x, blockIdx.x + gridDim.x, ...; n_rows counts them.
  if constexpr (!kSplit) nsplit = 1;
  const int tps = (nt + nsplit - 1) / nsplit;
  const int n_items = rows * nsplit;
  const int n_rows = n_items > static_cast<int>(blockIdx.x)
                         ? (n_items - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                         : 0;
  auto item_of = [&](int n) { return static_cast<int>(blockIdx.x) + n * static_cast<int>(gridDim.x); };
  auto item_row = [&](int n) { return kSplit ? item_of(n) / nsplit : item_of(n); };
  auto item_j0 = [&](int n) { return kSplit ? (item_of(n) % nsplit) * tps : 0; };
  auto item_jn = [&](int n) {
    if constexpr (!kSplit) return nt;
    const int j0 = item_j0(n);
    return min(nt, j0 + tps) - j0;
  };
  // rows 0 .. smask are readable (smask + 1 is the largest power of two <= S)
  const int smask = static_cast<int>((0x80000000u >> __clz(static_cast<uint32_t>(a.S))) - 1u);

  if (tid == 0) {
    for (int s = 0; s < NSLOT; ++s) {
      tc::mbar_init(&sm.full[s], PROD_THREADS);
      tc::mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&sm.qfull[s], 1);
      tc::mbar_init(&sm.sfull[s], 1);
      // one arrival per softmax warp (lane 0, after the warp's own accesses)
      tc::mbar_init(&sm.sempty[s], SOFT_THREADS / 32);
      tc::mbar_init(&sm.pfull[s], SOFT_THREADS / 32);
      tc::mbar_init(&sm.pempty[s], 1);
      tc::mbar_init(&sm.ofull[s], 1);
      tc::mbar_init(&sm.oempty[s], SOFT_THREADS / 32);
      tc::mbar_init(&sm.rowfree[s], SOFT_THREADS / 32);
    }
    tc::mbar_init(&sm.drain, 2);            // both MMA issuers
    sm.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tc::tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  // The set-up above may overlap the kernel before.  Q, the index rows and
  // K/V are read once it has completed, or at once when the caller knows
  // that kernel does not write them (inputs_ready); O is written only after
  // it has completed either way.
  const bool early = a.inputs_ready != 0;
  if (!early) grid_dep_wait();
  grid_dep_trigger();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t tS = tmem;          // columns 0..63: S buffers
  const uint32_t tO = tmem + 64;     // columns 64..127: O buffers

  if (warp == PV_WARP) {
    // ================= MMA issuer: O^T += V^T P^T =================
    if (lane == 0) {
      bool ok = true;
      uint32_t gp = 0;
      // the V tile of tile g is ring item 2g + 1: its slot and phase advance
      // by two items per tile; descriptors are built once and only their
      // start address moves (by 16-byte units, within the 256 KB window)
      int slot = 1;
      uint32_t phase = 0;
      const uint64_t dv0 = tc::sdesc(tc::smem_u32(sm.ring[0]), HALF_BYTES, 1024, 2);
      const uint64_t dp0 = tc::sdesc(tc::smem_u32(sm.ps[0]), 0, 512, 4);
      for (int n = 0; ok && n < n_rows; ++n) {
      const int j0 = item_j0(n), j1 = j0 + item_jn(n);
      for (int j = j0; j < j1; ++j, ++gp) {
        const int ob = n & 1;
        const int pb = gp & 1;
        if (j == j0 && !tc::mbar_wait<kWaitHintNs>(&sm.oempty[ob], ((n >> 1) & 1) ^ 1, &sm.abort)) { ok = false; break; }
        if (!tc::mbar_wait<kWaitHintNs>(&sm.full[slot], phase, &sm.abort)) { ok = false; break; }
        if (!tc::mbar_wait<kWaitHintNs>(&sm.pfull[pb], (gp >> 1) & 1, &sm.abort)) { ok = false; break; }
        tc::tc_fence_after();
        tc::fence_proxy_async_smem();   // the gathered rows (generic-proxy copies) before the MMA reads them
        const uint64_t dv = dv0 + static_cast<uint64_t>(slot * (SLOT_BYTES >> 4));
        const uint64_t dp = dp0 + static_cast<uint64_t>(pb * (P_BYTES >> 4));
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk)
          tc::mma_f16(tO + ob * HQ, dv + kk * (2048 >> 4), dp + kk * (1024 >> 4), IDESC_PV,
                      (j > j0 || kk != 0) ? 1u : 0u);
        tc::mma_commit(&sm.empty[slot]);
        tc::mma_commit(&sm.pempty[pb]);
        if (j == j1 - 1) tc::mma_commit(&sm.ofull[ob]);
        slot += 2;
        if (slot >= NSLOT) { slot -= NSLOT; phase ^= 1u; }
      }
      }
      if (!ok) set_abort(sm, status);
      // every MMA issued so far is complete before tensor memory is released
      tc::mma_commit(&sm.drain);
      if (!tc::mbar_wait<kWaitHintNs>(&sm.drain, 0, nullptr, 4000000000ull)) set_abort(sm, status);
    }
    __syncwarp();
  } else if (warp >= PROD_WARP0) {
    // ================= producers =================
    constexpr int RSTEP = PROD_THREADS / 16;
    const int pt = tid - PROD_WARP0 * 32;            // 0 .. PROD_THREADS-1
    const int c = pt & 15;                           // 16-byte chunk of a 256-byte row
    const int half = c >> 3, cc = c & 7;
    const int r0 = pt >> 4;                          // rows r0, r0 + RSTEP, ...
    const __nv_bfloat16* Kg = reinterpret_cast<const __nv_bfloat16*>(a.K) + c * 8;
    const __nv_bfloat16* Vg = reinterpret_cast<const __nv_bfloat16*>(a.V) + c * 8;
    int slot = 0;                                    // ring item: K0 V0 K1 V1 ...
    uint32_t phase = 0;
    bool ok = true;
    for (int n = 0; ok && n < n_rows; ++n) {
      const int row = item_row(n);
      const int j0 = item_j0(n), j1 = j0 + item_jn(n);
      const int qb = n & 1;
      // a wait that gave up in any lane ends the whole warp's loop
      if (!__all_sync(0xffffffffu, tc::mbar_wait<kWaitHintNs>(&sm.qfull[qb], (n >> 1) & 1, &sm.abort))) { ok = false; break; }
      const size_t base_row = static_cast<size_t>(row / a.T) * a.S_cap;
      for (int j = j0; ok && j < j1; ++j) {
        int src[PROD_ROWS];
        const int32_t* irow = sm.idx[qb] + j * KT;
        const int lim = k - j * KT;                  // positions past k are empty slots
#pragma unroll
        for (int i = 0; i < PROD_ROWS; ++i) {
          const int r = r0 + RSTEP * i;
          const int s = r < lim ? irow[r] : -1;
          src[i] = (s >= 0 && s < a.S) ? s : ((j * KT + r) & smask);   // empty slot: a spread, readable row
        }
#pragma unroll 1
        for (int kv = 0; kv < 2; ++kv) {
          const bool w_ok = tc::mbar_wait<kWaitHintNs>(&sm.empty[slot], phase ^ 1u, &sm.abort);
          if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
          const __nv_bfloat16* base = (kv ? Vg : Kg) + base_row * DH;
          uint8_t* dst = sm.ring[slot] + half * HALF_BYTES;
#pragma unroll
          for (int i = 0; i < PROD_ROWS; ++i) {
            const int r = r0 + RSTEP * i;
            cp_async16(dst + r * 128 + ((cc ^ (r & 7)) << 4), base + static_cast<size_t>(src[i]) * DH, true);
          }
          cp_async_arrive_noinc(&sm.full[slot]);
          if (++slot == NSLOT) { slot = 0; phase ^= 1u; }
        }
      }
    }
    // no copy of ours may still be landing when the CTA exits
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    if (!ok) set_abort(sm, status);
  } else if (warp == MMA_WARP) {
    // ================= MMA issuer: S^T = K Q^T =================
    if (lane == 0) {
      bool ok = true;
      uint32_t g = 0;
      // the K tile of tile g is ring item 2g (slot and phase advance by two
      // items per tile); descriptors as in the PV issuer
      int slot = 0;
      uint32_t phase = 0;
      const uint64_t dk0 = tc::sdesc_k_sw128(tc::smem_u32(sm.ring[0]));
      const uint64_t dq0 = tc::sdesc_k_sw128(tc::smem_u32(sm.qs[0]));
      for (int n = 0; ok && n < n_rows; ++n) {
      const int j0 = item_j0(n), j1 = j0 + item_jn(n);
      for (int j = j0; j < j1; ++j, ++g) {
        const int qb = n & 1;
        const int sb = g & 1;
        if (j == j0 && !tc::mbar_wait<kWaitHintNs>(&sm.qfull[qb], (n >> 1) & 1, &sm.abort)) { ok = false; break; }
        if (!tc::mbar_wait<kWaitHintNs>(&sm.sempty[sb], ((g >> 1) & 1) ^ 1, &sm.abort)) { ok = false; break; }
        if (!tc::mbar_wait<kWaitHintNs>(&sm.full[slot], phase, &sm.abort)) { ok = false; break; }
        tc::tc_fence_after();
        tc::fence_proxy_async_smem();
        const uint64_t dk = dk0 + static_cast<uint64_t>(slot * (SLOT_BYTES >> 4));
        const uint64_t dq = dq0 + static_cast<uint64_t>(qb * (Q_BYTES >> 4));
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint32_t off = (kk >> 2) * HALF_BYTES + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * (Q_BYTES / 2) + (kk & 3) * 32;
          tc::mma_f16(tS + sb * HQ, dk + (off >> 4), dq + (qoff >> 4), IDESC_QK, kk != 0);
        }
        tc::mma_commit(&sm.empty[slot]);
        tc::mma_commit(&sm.sfull[sb]);
        slot += 2;
        if (slot >= NSLOT) { slot -= NSLOT; phase ^= 1u; }
      }
      }
      if (!ok) set_abort(sm, status);
      // every MMA issued so far is complete before tensor memory is released
      tc::mma_commit(&sm.drain);
      if (!tc::mbar_wait<kWaitHintNs>(&sm.drain, 0, nullptr, 4000000000ull)) set_abort(sm, status);
    }
    __syncwarp();
  } else {
    // ================= softmax + epilogue (warps 0-7, two head groups) =================
    const int grp = warp >> 2;                     // heads 16*grp .. 16*grp + 15
    const int gw = warp & 3;                       // warp within the group = TMEM lane quarter
    const int bar_id = 1 + grp;
    const int my_lane = gw * 32 + lane;            // key lane (S, P) and d lane (O)
    const uint32_t lane_field = static_cast<uint32_t>(gw * 32) << 16;
    const int h0 = grp * HG;
    const float sl2 = a.scale * kLog2e;
    int rows_loaded = 0;                           // thread 0: rows whose inputs were requested
    if (tid == 0) {
      tc::tma_prefetch_map(&tm_q);
      for (int n = 0; n < 2 && n < n_rows; ++n) load_row_inputs(sm, &tm_q, a, item_row(n), n);
      rows_loaded = n_rows < 2 ? n_rows : 2;
    }
    // Row m's output, O / l_h as bf16, once its last PV is complete.  It runs
    // at the next row's first tile (after that tile's P is handed over), so
    // the softmax never waits for the PV pipeline to drain at a row boundary.
    auto finish_row = [&](int m) -> bool {
      if (early) grid_dep_wait();
      const int mb = m & 1;
      const bool w_ok = tc::mbar_wait<kWaitHintNs>(&sm.ofull[mb], (m >> 1) & 1, &sm.abort);
      if (tc::named_sync_or(bar_id, GROUP_THREADS, !w_ok || sm.abort)) return false;
      tc::tc_fence_after();
      uint32_t o[HG];
      tc::tmem_ld_x16(tO + mb * HQ + h0 + lane_field, o);
      tc::tmem_wait_ld();
      tc::tc_fence_before();
      __syncwarp();
      // Q and the index row of row m are no longer read by anyone either (both
      // groups passed its last tile, the MMA's last QK^T of it is complete)
      if (lane == 0) {
        tc::mbar_arrive(&sm.oempty[mb]);
        tc::mbar_arrive(&sm.rowfree[mb]);
      }
      const int mrow = item_row(m);
      if (tid == 0 && m + 2 < n_rows) {
        // load row m + 2 into the buffer
        if (tc::mbar_wait<kWaitHintNs>(&sm.rowfree[mb], (m >> 1) & 1, &sm.abort)) {
          load_row_inputs(sm, &tm_q, a, item_row(m + 2), mb);
          rows_loaded = m + 3;
        }
      }
      if constexpr (!kSplit) {
        __nv_bfloat16* Ob = reinterpret_cast<__nv_bfloat16*>(a.O) + static_cast<size_t>(mrow) * HQ * DH +
                            static_cast<size_t>(h0) * DH + my_lane;
#pragma unroll
        for (int h = 0; h < HG; ++h) Ob[h * DH] = __float2bfloat16_rn(__uint_as_float(o[h]) * sm.inv_l[mb][h0 + h]);
      } else {
        // a share of a row: (reference max, sum, unnormalised O) per head,
        // merged with the row's other shares in the cluster (O staged in
        // the ring, free once the last PV is complete; the max and the sum
        // stay in m_fin / l_fin) or by the combine kernel
        if (partials == nullptr) {
          float* so = reinterpret_cast<float*>(sm.ring[0]) + static_cast<size_t>(h0) * DH + my_lane;
#pragma unroll
          for (int h = 0; h < HG; ++h) so[h * DH] = __uint_as_float(o[h]);
          return true;
        }
        float* pb = partials + static_cast<size_t>(item_of(m)) * (2 * HQ + HQ * DH);
        if (gw == 0 && lane < HG) {
          pb[h0 + lane] = sm.m_fin[mb][h0 + lane];
          pb[HQ + h0 + lane] = sm.l_fin[mb][h0 + lane];
        }
        float* po = pb + 2 * HQ + static_cast<size_t>(h0) * DH + my_lane;
#pragma unroll
        for (int h = 0; h < HG; ++h) po[h * DH] = __uint_as_float(o[h]);
      }
      return true;
    };
    uint32_t g = 0;
    bool ok = true;
    for (int n = 0; ok && n < n_rows; ++n) {
      const int qb = n & 1;
      const int j0 = item_j0(n), j1 = j0 + item_jn(n);
      if (!tc::mbar_wait<kWaitHintNs>(&sm.qfull[qb], (n >> 1) & 1, &sm.abort)) ok = false;
      if (tc::named_sync_or(bar_id, GROUP_THREADS, !ok || sm.abort)) { ok = false; break; }
      float lp[HG], mr[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) { lp[h] = 0.0f; mr[h] = kMInit; }
      for (int j = j0; j < j1; ++j, ++g) {
        const int sb = g & 1;
        const int pb = g & 1;
        // S(g) ready and the P buffer free (PV(g-2) done); a wait that gave up
        // is agreed on at the group's next barrier
        bool w_ok = tc::mbar_wait<kWaitHintNs>(&sm.sfull[sb], (g >> 1) & 1, &sm.abort);
        w_ok = w_ok && tc::mbar_wait<kWaitHintNs>(&sm.pempty[pb], ((g >> 1) & 1) ^ 1, &sm.abort);
        tc::tc_fence_after();
        uint32_t r[HG];
        tc::tmem_ld_x16(tS + sb * HQ + h0 + lane_field, r);
        tc::tmem_wait_ld();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.sempty[sb]);
        const int kj = j * KT + my_lane;
        const int sidx = kj < k ? sm.idx[qb][kj] : -1;
        const bool valid = sidx >= 0 && sidx < a.S;
        const float sv = valid ? sl2 : 0.0f;       // an empty slot scores -inf: 0 * s - inf
        const float ov = valid ? 0.0f : -INFINITY;
        // exponent t = s * scale * log2(e) - m for every head; a tile whose t
        // stays <= kTau everywhere needs no change of the reference max
        float t[HG];
        float tmax = -INFINITY;
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          t[h] = fmaf(__uint_as_float(r[h]), sv, ov - mr[h]);
          tmax = fmaxf(tmax, t[h]);
        }
        const bool slow = tc::named_sync_or(bar_id, GROUP_THREADS, j == j0 || tmax > kTau || !w_ok || sm.abort);
        if (slow) {
          if (tc::named_sync_or(bar_id, GROUP_THREADS, !w_ok || sm.abort)) { ok = false; break; }
          // exact tile maximum per head of the group, across the 128 key lanes
          {
            float y[HG];
#pragma unroll
            for (int h = 0; h < HG; ++h) y[h] = fmaf(__uint_as_float(r[h]), sv, ov);   // s*scale*log2(e) or -inf
            sm.red[warp][lane & 15] = warp_reduce_scatter16<true>(y, lane);
          }
          tc::named_sync(bar_id, GROUP_THREADS);
          if (gw == 0 && lane < HG) {
            const float* rd = &sm.red[grp * 4][0];
            const float mt = fmaxf(fmaxf(rd[lane], rd[HG + lane]), fmaxf(rd[2 * HG + lane], rd[3 * HG + lane]));
            const float mo = j == j0 ? kMInit : sm.m_ref[h0 + lane];
            const float mn = fmaxf(mo, mt);
            sm.alpha[h0 + lane] = exp2f(mo - mn);
            sm.m_ref[h0 + lane] = mn;
          }
          tc::named_sync(bar_id, GROUP_THREADS);
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            const float mn = sm.m_ref[h0 + h];
            t[h] = fmaf(__uint_as_float(r[h]), sv, ov) - mn;
            mr[h] = mn;
            lp[h] *= sm.alpha[h0 + h];
          }
          if (j > j0) {
            // this group's O columns hold tiles 0 .. j-1 once PV(g-1) is done: scale them in place
            const uint32_t gp = g - 1;
            w_ok = tc::mbar_wait<kWaitHintNs>(&sm.pempty[gp & 1], (gp >> 1) & 1, &sm.abort);
            if (tc::named_sync_or(bar_id, GROUP_THREADS, !w_ok || sm.abort)) { ok = false; break; }
            tc::tc_fence_after();
            uint32_t o[HG];
            const uint32_t taddr = tO + qb * HQ + h0 + lane_field;
            tc::tmem_ld_x16(taddr, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < HG; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * sm.alpha[h0 + h]);
            tc::tmem_st_x16(taddr, o);
            tc::tmem_wait_st();
          }
        }
        uint32_t pk[HG / 2];
#pragma unroll
        for (int h = 0; h < HG; h += 2) {
          const float p0 = tc::ex2_approx(t[h]);
          const float p1 = tc::ex2_approx(t[h + 1]);
          lp[h] += p0;
          lp[h + 1] += p1;
          pk[h / 2] = pack_bf16x2(p0, p1);
        }
        // row my_lane of P: 64 bytes, 16-byte chunk c at (c ^ ((row >> 1) & 3)) (64-byte swizzle);
        // this group writes chunks 2*grp and 2*grp + 1
        uint8_t* prow = sm.ps[pb] + my_lane * 64;
        const int sx = (my_lane >> 1) & 3;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c = 2 * grp + c2;
          *reinterpret_cast<uint4*>(prow + ((c ^ sx) << 4)) =
              make_uint4(pk[4 * c2], pk[4 * c2 + 1], pk[4 * c2 + 2], pk[4 * c2 + 3]);
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.pfull[pb]);
        if (j == j0 && n > 0 && !finish_row(n - 1)) { ok = false; break; }
      }
      if (!ok) break;
      // ---- row end: l_h (the output is written by finish_row) ----
      sm.red[warp][lane & 15] = warp_reduce_scatter16<false>(lp, lane);
      tc::named_sync(bar_id, GROUP_THREADS);
      if (gw == 0 && lane < HG) {
        const float* rd = &sm.red[grp * 4][0];
        const float l = rd[lane] + rd[HG + lane] + rd[2 * HG + lane] + rd[3 * HG + lane];
        sm.inv_l[qb][h0 + lane] = l > 0.0f ? 1.0f / l : 0.0f;
        sm.l_fin[qb][h0 + lane] = l;
        sm.m_fin[qb][h0 + lane] = sm.m_ref[h0 + lane];
      }
    }
    if (ok && n_rows > 0 && !finish_row(n_rows - 1)) ok = false;
    if (!ok) set_abort(sm, status);
    // no row-input copy of ours may still be landing when the CTA exits
    // (the last two rows requested; earlier ones were waited for before their
    // buffer was reused)
    if (tid == 0) {
      for (int r = rows_loaded > 2 ? rows_loaded - 2 : 0; r < rows_loaded; ++r)
        tc::mbar_wait<kWaitHintNs>(&sm.qfull[r & 1], (r >> 1) & 1, nullptr);
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == MMA_WARP) tc::tmem_dealloc(tmem, TMEM_COLS);
  if constexpr (kSplit) {
    if (partials == nullptr) {
      // one item per CTA, the row's nsplit CTAs are this cluster (rank = share)
      namespace cg = cooperative_groups;
      cg::cluster_group cluster = cg::this_cluster();
      cluster.sync();                            // every share is staged
      if (early) grid_dep_wait();
      const int rank = static_cast<int>(cluster.block_rank());
      const int row = item_row(0);
      const int hpc = (HQ + nsplit - 1) / nsplit;
      const int hb = min(HQ, rank * hpc), he = min(HQ, hb + hpc);
      __nv_bfloat16* Ob = reinterpret_cast<__nv_bfloat16*>(a.O) + static_cast<size_t>(row) * HQ * DH;
      for (int e = hb * DH + tid; e < he * DH; e += NTHREADS) {
        const int h = e / DH;
        // every share's values are requested before any is used (one round
        // trip through the cluster instead of one per share)
        float mv[kTcMaxClusterSplit], lv[kTcMaxClusterSplit], ov[kTcMaxClusterSplit];
#pragma unroll
        for (int r = 0; r < kTcMaxClusterSplit; ++r) {
          if (r < nsplit) {
            mv[r] = *cluster.map_shared_rank(&sm.m_fin[0][h], r);
            lv[r] = *cluster.map_shared_rank(&sm.l_fin[0][h], r);
            ov[r] = *cluster.map_shared_rank(reinterpret_cast<float*>(sm.ring[0]) + e, r);
          }
        }
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < kTcMaxClusterSplit; ++r)
          if (r < nsplit) M = fmaxf(M, mv[r]);
        float l = 0.0f, acc = 0.0f;
#pragma unroll
        for (int r = 0; r < kTcMaxClusterSplit; ++r) {
          if (r < nsplit) {
            const float f = exp2f(mv[r] - M);
            l += lv[r] * f;
            acc += ov[r] * f;
          }
        }
        Ob[e] = __float2bfloat16_rn(l > 0.0f ? acc / l : 0.0f);
      }
      cluster.sync();                            // no other CTA reads this one's shares any more
    }
  }
}

}  // namespace

int sparse_attn_tc_splits(const AttnArgs& a) {
  const long long rows = static_cast<long long>(a.B) * a.T;
  if (a.Hq != HQ || a.Dh != DH || (a.k % 4) != 0 || a.k <= KT || rows * HQ >= (1ll << 31) ||
      static_cast<long long>(a.B) * a.S_cap >= (1ll << 31))
    return 0;
  if (rows >= 2 * kTcTargetCtas) return 1;   // whole rows, at least two per CTA
  // few rows (decode): each row's tiles are shared among up to
  // kTcTargetCtas / rows CTAs, at least two tiles each
  const int nt = (a.k + KT - 1) / KT;
  int ns = static_cast<int>(kTcTargetCtas / rows);
  ns = ns < nt / 2 ? ns : nt / 2;
  if (ns < 2) return 0;
  const int tps = (nt + ns - 1) / ns;
  return (nt + tps - 1) / tps;                 // every share non-empty
}

cudaError_t launch_sparse_attn_tc(const AttnArgs& a, int nsplit, float* partials, int* dev_status, cudaStream_t st) {
  CUtensorMap tm_q, tm_k, tm_v;
  const uint64_t rows = static_cast<uint64_t>(a.B) * a.T;
  if (nsplit < 1) return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tm_q, a.Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows * HQ, DH, HQ, 64))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tm_k, a.K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(a.B) * a.S_cap, DH, 1,
                      64))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tm_v, a.V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(a.B) * a.S_cap, DH, 1,
                      64))
    return cudaErrorInvalidValue;
  int dev = 0, n_sm = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  const size_t smem = sizeof(AttnTcSmem) + 1024;
  auto kern = nsplit > 1 ? sparse_attn_tc_kernel<true> : sparse_attn_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const uint64_t items = rows * static_cast<uint64_t>(nsplit);
  const int grid = static_cast<int>(items < static_cast<uint64_t>(n_sm) ? items : n_sm);
  if (nsplit > 1 && partials == nullptr) {
    // one share per CTA, the shares of a row as one cluster, merged in it
    if (items > static_cast<uint64_t>(n_sm) || nsplit > kTcMaxClusterSplit) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(items));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(nsplit);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, sparse_attn_tc_kernel<true>, tm_q, tm_k, tm_v, a, nsplit, partials, dev_status);
  }
  return launch_pdl(kern, dim3(grid), dim3(NTHREADS), smem, st, tm_q, tm_k, tm_v, a, nsplit, partials, dev_status);
}

bool sparse_attn_tc_cluster_merge(const AttnArgs& a, int nsplit) {
  int dev = 0, n_sm = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  const long long items = static_cast<long long>(a.B) * a.T * nsplit;
  if (nsplit < 2 || nsplit > kTcMaxClusterSplit || items > n_sm) return false;
  // clusters of nsplit CTAs with this shared memory must fit the device
  // (asked once per size and process)
  static int fits[kTcMaxClusterSplit + 1] = {-1, -1, -1, -1, -1, -1, -1, -1, -1};
  if (fits[nsplit] < 0) {
    int v = 0, n = 0;
    const size_t smem = sizeof(AttnTcSmem) + 1024;
    cudaError_t q = cudaFuncSetAttribute(sparse_attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (q == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(nsplit));
      cfg.blockDim = dim3(NTHREADS);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(nsplit);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      q = cudaOccupancyMaxActiveClusters(&n, sparse_attn_tc_kernel<true>, &cfg);
      if (q == cudaSuccess && n > 0) v = 1;
    }
    if (q != cudaSuccess) cudaGetLastError();    // a refused query leaves no error behind
    fits[nsplit] = v;
  }
  return fits[nsplit] == 1;
}

}  // namespace ic
