// Fused lightning indexer + streaming top-k on the 5th-generation tensor
// cores (tcgen05 + TMA + tensor memory), for the production indexer shape
// H_I = 64 heads, d_I = 128, bf16 keys or e4m3 keys with a per-key scale.
//
// Score (DSA lightning-indexer score, the Full layers of IndexCache; notes
// page "NLP--IndexCache", section "背景 & 问题提出"):
//     I[t,s] = sum_h w[t,h] * ReLU(q[t,h,:] . kI[s,:]),   s <= pos(t).
//
// One CTA owns QPB = 4 consecutive query rows.  Their q rows form the MMA's
// B operand (N = 4 x 64 = 256 columns, loaded once by TMA); key tiles of
// 128 rows form the A operand (M = 128, keys on the TMEM lanes), streamed by
// TMA in K-halves of 64 features through a 4-deep ring.  One thread issues
// the MMAs into two TMEM accumulators of 128 x 256 fp32 (all 512 columns),
// so the tensor core fills one while the epilogue drains the other.
//
// Warp roles (18 warps):
//   warp 0     TMA producer (q once, then key half-tiles)
//   warp 1     TMEM allocator + MMA issuer
//   warps 2-17 epilogue: four warpgroups; warpgroup g owns query row g.
//              Thread = one key (its TMEM lane); it reads the 64 head dot
//              products of its row in quarters of 16 (each quarter's load
//              in flight while the previous one is summed), forms the
//              weighted ReLU sum in registers, and runs the streaming top-k.
//
// e4m3 keys: every e4m3 value (subnormals included) is a bf16 value, so a
// small kernel first widens the keys the call reads into a bf16 copy in the
// workspace, exactly; the same TMA-fed kernel then runs on bf16 q and keys,
// and the key's scale multiplies its head sum (a positive factor commutes
// with ReLU).  No operand is rounded.
//
// Streaming top-k (per row, in shared memory): a candidate list of (key,
// position), key = an order-preserving integer image of the score, kept in
// ascending position order.  A key enters iff it is above the row's
// threshold tau; keys arrive in ascending position, so a key that only ties
// tau loses to k kept candidates with lower positions.  The four warps of a
// warpgroup each own a quarter of a tile's keys; they exchange their
// per-row insert counts at the one barrier of each tile and append in order,
// so no other synchronisation is needed.  When a tile would overflow the
// list, the list is cut: every candidate below a threshold found with a
// most-significant-digit histogram (at least k kept) is dropped, in order,
// and tau rises to that threshold.  After the last tile an exact cut to k
// (ties to the lower position) leaves the answer, already ascending.  The
// L x L scores never leave the SM.
//
// Every wait is bounded: a wait that gives up sets the CTA's abort flag and
// the device status word; all roles then wind down, wait (bounded) for the
// MMAs already issued, and release tensor memory before returning.
#include "ic_common.cuh"
#include "ic_kernels.h"
#include "tc_utils.cuh"
#include "topk_stream.cuh"

#include <algorithm>

namespace ic {
namespace {

constexpr int QPB = 4;                   // query rows per CTA
constexpr int HH = 64;                   // indexer heads
constexpr int DD = 128;                  // indexer feature dim
constexpr int NCOL = QPB * HH;           // MMA N = 256
constexpr int KT = 128;                  // keys per tile (MMA M)
constexpr int KSTAGES = 4;               // ring of K-half tiles (16 KB each)
constexpr int CAP = kMaxK + 896;         // candidate slots per row (what shared memory leaves: 227 KB in all)
constexpr int WG_THREADS = 128;
constexpr int SEG = CAP / WG_THREADS;    // entries per thread in a cut
// A cut keeps at most this many: close to k, so that the threshold it leaves
// is nearly the k-th best key and few later keys are listed only to be cut
// again (10.07 ms per F layer at L = 32768 against 10.27 with k + 128 and
// 10.85 with CAP - 2 KT; an exact cut, k, 10.68: its extra passes cost more
// than they save).  At most CAP - 2 KT, so every cut frees at least two tiles.
constexpr int CUT_LIMIT = kMaxK + 64;
static_assert(CUT_LIMIT <= CAP - 2 * KT, "a cut must free two tiles");

// Epilogue layout: four warpgroups of one row each (four epilogue warps per
// SM sub-partition hide the tensor-memory and barrier latencies).
struct Layout {
  static constexpr int RPW = 1;                              // rows per epilogue warpgroup
  static constexpr int NWG = QPB / RPW;                      // epilogue warpgroups
  static constexpr int EPI_THREADS = NWG * WG_THREADS;
  static constexpr int NTHREADS = EPI_THREADS + 64;
};

// Operand kinds of the kernel.
enum Kind : int {
  KEYS_BF16 = 0,   // bf16 q and keys (kind::f16)
  KEYS_E4M3 = 1,   // bf16 q, e4m3 keys widened to bf16 in the workspace, per-key scale in the epilogue
  QK_E4M3 = 2,     // e4m3 q and keys as stored (kind::f8f6f4), per-(row, head) q scale folded into w,
                   // per-key scale in the epilogue
};
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = tc::idesc_bf16_f32(KT, NCOL);
constexpr uint32_t IDESC_E4M3 = tc::idesc_e4m3_f32(KT, NCOL);

struct __align__(1024) TcSmem {
  uint8_t qb[2][NCOL * 128];             // B operand: two K-halves, 256 rows x 128 B (SW128)
  uint8_t kst[KSTAGES][KT * 128];        // A operand ring: K-half tiles, 128 rows x 128 B (SW128)
  float wsm[QPB][HH];
  uint32_t cand_k[QPB][CAP];             // float_key of the score
  int cand_p[QPB][CAP];
  uint64_t full[KSTAGES];
  uint64_t empty[KSTAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t qfull;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  // per tile parity, row and key quarter: insert count
  alignas(16) int xc[2][QPB][4];
  SelectScratch scr[QPB];
};

struct WgSync {
  int id;
  __device__ __forceinline__ void operator()() const { tc::named_sync(id, WG_THREADS); }
};

// Largest of the warpgroup's per-thread values (all 128 threads call it).
__device__ __forceinline__ uint32_t list_max(uint32_t v, SelectScratch* scr, int wtid, const WgSync& sync) {
  v = __reduce_max_sync(0xffffffffu, v);
  if ((wtid & 31) == 0) scr->warp_sums[wtid >> 5] = static_cast<int>(v);
  sync();
  const uint32_t m = max(max(static_cast<uint32_t>(scr->warp_sums[0]), static_cast<uint32_t>(scr->warp_sums[1])),
                         max(static_cast<uint32_t>(scr->warp_sums[2]), static_cast<uint32_t>(scr->warp_sums[3])));
  sync();
  return m;
}

__device__ __forceinline__ void set_abort(TcSmem& sm, int* status) {
  sm.abort = 1;
  if (status) atomicExch(status, kDevTimeout);
}

// e4m3 byte pairs -> bf16 pairs, exactly: every e4m3 value (subnormals
// included) is a bf16 value.  Normal codes move the exponent from bias 7 to
// bias 127 and the 3 mantissa bits to the top of bf16's 7; subnormal codes
// (exponent field 0) are m * 2^-9.
__device__ __forceinline__ uint32_t e4m3_pair_to_bf16_pair(uint32_t v) {
  return e4m3_to_bf16_bits(v & 0xFFu) | (e4m3_to_bf16_bits((v >> 8) & 0xFFu) << 16);
}

// e4m3 keys [B, S_cap, 128] (rows 0 .. S-1 of each sequence) -> bf16 keys
// [B, S, 128], one 16-byte chunk of 16 codes per thread.
__global__ void __launch_bounds__(256) widen_e4m3_keys_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                              int B, int S, int S_cap) {
  const size_t per_seq = static_cast<size_t>(S) * (DD / 16);
  const size_t n_chunks = per_seq * B;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_chunks;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t b = i / per_seq, r = i - b * per_seq;
    const uint4 x = __ldcs(src + b * static_cast<size_t>(S_cap) * (DD / 16) + r);
    uint4 lo, hi;
    lo.x = e4m3_pair_to_bf16_pair(x.x);       lo.y = e4m3_pair_to_bf16_pair(x.x >> 16);
    lo.z = e4m3_pair_to_bf16_pair(x.y);       lo.w = e4m3_pair_to_bf16_pair(x.y >> 16);
    hi.x = e4m3_pair_to_bf16_pair(x.z);       hi.y = e4m3_pair_to_bf16_pair(x.z >> 16);
    hi.z = e4m3_pair_to_bf16_pair(x.w);       hi.w = e4m3_pair_to_bf16_pair(x.w >> 16);
    dst[2 * i] = lo;
    dst[2 * i + 1] = hi;
  }
}

template <int KIND>
__global__ void __launch_bounds__(Layout::NTHREADS, 1)
indexer_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          IndexerArgs a, int n_groups, int key_rows, int* status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the dynamic shared window is 1024-aligned for the swizzled operands
  TcSmem& sm = *reinterpret_cast<TcSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // limit of every wait on another role's progress (the wind-down waits for
  // this CTA's own copies and MMAs keep their fixed limits)
  const uint64_t lim = a.wait_ns ? a.wait_ns : kWaitLimitNs;
  const int g = n_groups - 1 - static_cast<int>(blockIdx.x);   // longest causal range first
  const int b = blockIdx.y;
  const int t0 = g * QPB;
  const int nq = min(QPB, a.T - t0);
  const int pos0 = a.q_pos0 + t0;
  const int n_keys = pos0 + nq;
  int32_t* out = a.idx + (static_cast<size_t>(b) * a.T + t0) * a.k;

  using LY = Layout;
  constexpr bool E4M3 = KIND != KEYS_BF16;      // a per-key scale multiplies the head sum
  constexpr bool FP8 = KIND == QK_E4M3;         // 8-bit operands: one 16 KB stage per 128-key tile
  constexpr int kThreads = LY::NTHREADS;
  constexpr int RPW = LY::RPW;
  if (n_keys <= a.k) {   // every causal position of every row is selected
    for (int i = tid; i < nq * a.k; i += kThreads) {
      const int qi = i / a.k, j = i - qi * a.k;
      out[i] = (j <= pos0 + qi) ? j : -1;
    }
    return;
  }
  const int nt = (n_keys + KT - 1) / KT;

  // ---- set-up ----
  if (tid == 0) {
    for (int s = 0; s < KSTAGES; ++s) {
      tc::mbar_init(&sm.full[s], 1);
      tc::mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) { tc::mbar_init(&sm.tfull[s], 1); tc::mbar_init(&sm.tempty[s], LY::EPI_THREADS); }
    tc::mbar_init(&sm.qfull, 1);
    tc::mbar_init(&sm.drain, 1);
    sm.abort = 0;
    tc::fence_mbar_init();
  }
  for (int i = tid; i < QPB * HH; i += kThreads) {
    const int qi = i / HH, h = i % HH;
    const size_t wi = (static_cast<size_t>(b) * a.T + t0 + qi) * HH + h;
    // e4m3 q: its positive per-(row, head) scale moves through the ReLU into w
    sm.wsm[qi][h] = qi < nq ? (FP8 ? a.w[wi] * a.qscale[wi] : a.w[wi]) : 0.0f;
  }
  if (warp == 1) {
    tc::tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      tc::tma_prefetch_map(&tm_q);
      tc::tma_prefetch_map(&tm_k);
      const int qrow = (b * a.T + t0) * HH;
      // q rows are read by this CTA only; key tiles by every CTA of the sequence
      const uint64_t once = tc::l2_evict_first(), keep = tc::l2_evict_last();
      if (FP8) {
        // 256 q rows of 128 e4m3 bytes: one 128-byte-swizzled box
        tc::mbar_arrive_expect_tx(&sm.qfull, NCOL * 128);
        tc::tma_load_2d_hint(sm.qb[0], &tm_q, &sm.qfull, 0, qrow, once);
      } else {
        tc::mbar_arrive_expect_tx(&sm.qfull, 2 * NCOL * 128);
        tc::tma_load_2d_hint(sm.qb[0], &tm_q, &sm.qfull, 0, qrow, once);
        tc::tma_load_2d_hint(sm.qb[1], &tm_q, &sm.qfull, 64, qrow, once);
      }
      const int krow0 = b * key_rows;
      // stages: bf16 keys two K-halves of 64 features per tile, e4m3 keys the whole tile
      constexpr int kPerTile = FP8 ? 1 : 2;
      int issued = 0;
      for (int it = 0; it < kPerTile * nt; ++it) {
        const int s = it % KSTAGES;
        const uint32_t ph = (it / KSTAGES) & 1;
        if (!tc::mbar_wait(&sm.empty[s], ph ^ 1, &sm.abort, lim)) { set_abort(sm, status); break; }
        tc::mbar_arrive_expect_tx(&sm.full[s], KT * 128);
        if (FP8) tc::tma_load_2d_hint(sm.kst[s], &tm_k, &sm.full[s], 0, krow0 + it * KT, keep);
        else tc::tma_load_2d_hint(sm.kst[s], &tm_k, &sm.full[s], (it & 1) * 64, krow0 + (it >> 1) * KT, keep);
        issued = it + 1;
      }
      // no copy of ours may still be landing in shared memory when the CTA exits
      tc::mbar_wait(&sm.qfull, 0, nullptr);
      for (int it = (issued > KSTAGES ? issued - KSTAGES : 0); it < issued; ++it)
        tc::mbar_wait(&sm.full[it % KSTAGES], (it / KSTAGES) & 1, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      bool ok = tc::mbar_wait(&sm.qfull, 0, &sm.abort, lim);
      if (!ok) set_abort(sm, status);
      const uint32_t qb0 = tc::smem_u32(sm.qb[0]);
      const uint32_t qb1 = tc::smem_u32(sm.qb[1]);
      for (int j = 0; ok && j < nt; ++j) {
        const int acc = j & 1;
        if (!tc::mbar_wait(&sm.tempty[acc], ((j >> 1) & 1) ^ 1, &sm.abort, lim)) { set_abort(sm, status); break; }
        tc::tc_fence_after();
        const uint32_t d_tmem = tmem + acc * NCOL;
        for (int h = 0; h < (FP8 ? 1 : 2); ++h) {
          const int it = FP8 ? j : 2 * j + h;
          const int s = it % KSTAGES;
          if (!tc::mbar_wait(&sm.full[s], (it / KSTAGES) & 1, &sm.abort, lim)) { set_abort(sm, status); ok = false; break; }
          tc::tc_fence_after();
          const uint32_t a_base = tc::smem_u32(sm.kst[s]);
          const uint32_t b_base = h ? qb1 : qb0;
          // each MMA takes 32 bytes of every 128-byte row: 16 bf16 or 32 e4m3 features
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            if (FP8)
              tc::mma_f8f6f4(d_tmem, tc::sdesc_k_sw128(a_base + kk * 32), tc::sdesc_k_sw128(b_base + kk * 32),
                             IDESC_E4M3, kk != 0);
            else
              tc::mma_f16(d_tmem, tc::sdesc_k_sw128(a_base + kk * 32), tc::sdesc_k_sw128(b_base + kk * 32),
                          IDESC, (h | kk) != 0);
          }
          tc::mma_commit(&sm.empty[s]);   // frees the stage once these MMAs are done
        }
        if (!ok) break;
        tc::mma_commit(&sm.tfull[acc]);   // accumulator ready for the epilogue
      }
      // every MMA issued so far is complete before tensor memory is released
      tc::mma_commit(&sm.drain);
      if (!tc::mbar_wait(&sm.drain, 0, nullptr, 4000000000ull)) set_abort(sm, status);
    }
    __syncwarp();
  } else {
    // ================= epilogue: scores + streaming top-k =================
    const int wg = (warp - 2) >> 2;               // epilogue warpgroup
    const int quarter = warp & 3;                 // TMEM lane quarter this warp may read
    const int key_local = quarter * 32 + lane;
    const int wtid = tid - 64 - wg * WG_THREADS;  // 0..127 within the warpgroup
    const WgSync wsync{1 + wg};
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    const int q0 = RPW * wg;                      // this warpgroup's rows q0 .. q0 + RPW - 1
    const unsigned lanes_below = (1u << lane) - 1u;
    // per-row state, identical in every thread of the warpgroup
    int cnt[RPW];
    uint32_t tau[RPW];                              // a key enters iff key > tau (every listed key is)
    uint32_t kmax[RPW];                             // largest key this thread listed (bounds the list at a cut)
#pragma unroll
    for (int qq = 0; qq < RPW; ++qq) { cnt[qq] = 0; tau[qq] = 0u; kmax[qq] = 0u; }

    // e4m3: the key scales of the next tile are loaded one tile ahead
    const float* ksrow = E4M3 ? a.kscale + static_cast<size_t>(b) * a.S_cap : nullptr;
    float ks_next = (E4M3 && key_local < n_keys) ? __ldg(ksrow + key_local) : 1.0f;

    bool aborted = false;
    for (int j = 0; j < nt; ++j) {
      const int acc = j & 1;
      const int par = j & 1;
      const float ks = ks_next;
      if (E4M3) {
        const int sn = (j + 1) * KT + key_local;
        ks_next = sn < n_keys ? __ldg(ksrow + sn) : 1.0f;
      }
      const bool ok = tc::mbar_wait(&sm.tfull[acc], (j >> 1) & 1, &sm.abort, lim);
      if (!ok) set_abort(sm, status);
      tc::tc_fence_after();
      uint32_t key[RPW];
#pragma unroll
      for (int qq = 0; qq < RPW; ++qq) {
        const uint32_t col = tmem + lane_field + acc * NCOL + (q0 + qq) * HH;
        const float* wq = sm.wsm[q0 + qq];
        float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;   // four chains: the FMA latencies overlap
        auto accumulate = [&](const uint32_t (&r)[32], const float* wh) {
#pragma unroll
          for (int h = 0; h < 32; h += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(wh + h);
            s0 = fmaf(w4.x, fmaxf(__uint_as_float(r[h + 0]), 0.0f), s0);
            s1 = fmaf(w4.y, fmaxf(__uint_as_float(r[h + 1]), 0.0f), s1);
            s2 = fmaf(w4.z, fmaxf(__uint_as_float(r[h + 2]), 0.0f), s2);
            s3 = fmaf(w4.w, fmaxf(__uint_as_float(r[h + 3]), 0.0f), s3);
          }
        };
        if constexpr (RPW == 1) {
          // quarters of 16 heads, each quarter's load in flight while the one
          // before is summed (two 16-register buffers, as many live registers
          // as one 32-column load)
          auto acc16 = [&](const uint32_t (&r)[16], const float* wh) {
#pragma unroll
            for (int h = 0; h < 16; h += 4) {
              const float4 w4 = *reinterpret_cast<const float4*>(wh + h);
              s0 = fmaf(w4.x, fmaxf(__uint_as_float(r[h + 0]), 0.0f), s0);
              s1 = fmaf(w4.y, fmaxf(__uint_as_float(r[h + 1]), 0.0f), s1);
              s2 = fmaf(w4.z, fmaxf(__uint_as_float(r[h + 2]), 0.0f), s2);
              s3 = fmaf(w4.w, fmaxf(__uint_as_float(r[h + 3]), 0.0f), s3);
            }
          };
          // the values of a load are used only after its wait
          auto fence16 = [](uint32_t (&r)[16]) {
            asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                         "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                         "+r"(r[14]), "+r"(r[15]));
          };
          uint32_t ra[16], rb[16];
          tc::tmem_ld_x16(col, ra);
          tc::tmem_wait_ld();
          fence16(ra);
          tc::tmem_ld_x16(col + 16, rb);
          acc16(ra, wq);
          tc::tmem_wait_ld();
          fence16(rb);
          tc::tmem_ld_x16(col + 32, ra);
          acc16(rb, wq + 16);
          tc::tmem_wait_ld();
          fence16(ra);
          tc::tmem_ld_x16(col + 48, rb);
          acc16(ra, wq + 32);
          tc::tmem_wait_ld();
          fence16(rb);
          acc16(rb, wq + 48);
        } else {
          uint32_t r0[32], r1[32];
          tc::tmem_ld_x32(col, r0);
          tc::tmem_ld_x32(col + 32, r1);
          tc::tmem_wait_ld();
          accumulate(r0, wq);
          accumulate(r1, wq + 32);
        }
        key[qq] = float_key(E4M3 ? ((s0 + s1) + (s2 + s3)) * ks : (s0 + s1) + (s2 + s3));
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&sm.tempty[acc]);           // accumulator may be overwritten

      // this warp's candidates of the tile; counts and key bounds go to the other warps
      const int s_pos = j * KT + key_local;
      bool valid[RPW], take[RPW];
      unsigned bal[RPW];
#pragma unroll
      for (int qq = 0; qq < RPW; ++qq) {
        const int qi = q0 + qq;
        valid[qq] = qi < nq && s_pos <= pos0 + qi;
        take[qq] = valid[qq] && key[qq] > tau[qq];
        bal[qq] = __ballot_sync(0xffffffffu, take[qq]);
        if (take[qq]) kmax[qq] = max(kmax[qq], key[qq]);
        if (lane == 0) sm.xc[par][qi][quarter] = __popc(bal[qq]);
      }
      // the tile's one barrier: the exchange, and one abort decision for the warpgroup
      if (tc::named_sync_or(1 + wg, WG_THREADS, !ok || sm.abort)) { aborted = true; break; }
#pragma unroll
      for (int qq = 0; qq < RPW; ++qq) {
        const int qi = q0 + qq;
        int4 cv = *reinterpret_cast<const int4*>(&sm.xc[par][qi][0]);   // the four warps' counts, one load
        int tot = (cv.x + cv.y) + (cv.z + cv.w);
        if (cnt[qq] + tot > CAP) {
          // the list would overflow: cut it, raise tau, recount this tile's keys
          uint32_t thr;
          cnt[qq] = cut_list<WG_THREADS, SEG>(sm.cand_k[qi], sm.cand_p[qi], cnt[qq], a.k, CUT_LIMIT, tau[qq],
                                              list_max(kmax[qq], &sm.scr[wg], wtid, wsync), &sm.scr[wg], wtid, wsync,
                                              &thr);
          tau[qq] = thr;
          take[qq] = valid[qq] && key[qq] > tau[qq];
          bal[qq] = __ballot_sync(0xffffffffu, take[qq]);
          if (lane == 0) sm.xc[par][qi][quarter] = __popc(bal[qq]);
          wsync();
          cv = *reinterpret_cast<const int4*>(&sm.xc[par][qi][0]);
          tot = (cv.x + cv.y) + (cv.z + cv.w);
        }
        if (tot == 0) continue;
        int off = cnt[qq];
        off += (quarter > 0 ? cv.x : 0) + (quarter > 1 ? cv.y : 0) + (quarter > 2 ? cv.z : 0);
        if (take[qq]) {
          const int slot = off + __popc(bal[qq] & lanes_below);
          sm.cand_k[qi][slot] = key[qq];
          sm.cand_p[qi][slot] = s_pos;
        }
        cnt[qq] += tot;
      }
    }
    if (!aborted) aborted = tc::named_sync_or(1 + wg, WG_THREADS, sm.abort != 0);
    // exact cut to k and write-out (ascending already)
    if (!aborted) {
#pragma unroll
      for (int qq = 0; qq < RPW; ++qq) {
        const int qi = q0 + qq;
        if (qi >= nq) break;
        int c = cnt[qq];
        if (c > a.k) {
          uint32_t thr;
          c = cut_list<WG_THREADS, SEG>(sm.cand_k[qi], sm.cand_p[qi], c, a.k, a.k, tau[qq],
                                        list_max(kmax[qq], &sm.scr[wg], wtid, wsync), &sm.scr[wg], wtid, wsync, &thr);
        }
        int32_t* row = out + static_cast<size_t>(qi) * a.k;
        for (int x = wtid; x < a.k; x += WG_THREADS) row[x] = x < c ? sm.cand_p[qi][x] : -1;
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

bool indexer_prefill_tc_supported(const IndexerArgs& a) {
  return a.H == HH && a.D == DD && a.T > kDecodeMaxT && (!a.e4m3 || a.kscale != nullptr);
}

size_t indexer_prefill_tc_ws_bytes(int B, int T, int S, int H, int D, bool e4m3) {
  // e4m3 keys (with bf16 q) on this kernel's shape: their exact bf16
  // widening, [B, S, 128]; e4m3 q with e4m3 keys needs none
  if (!e4m3 || H != HH || D != DD || T <= kDecodeMaxT) return 0;
  return (static_cast<size_t>(B) * S * DD * 2 + 255) / 256 * 256;
}

cudaError_t launch_indexer_prefill_tc(const IndexerArgs& a, void* ws, size_t ws_bytes, int* dev_status,
                                      cudaStream_t st) {
  CUtensorMap tm_q, tm_k;
  if (a.qscale) {
    // e4m3 q and keys as stored: q as [B*T*H, 128] bytes, box 256 rows; keys
    // as [B*S_cap, 128] bytes, box 128 rows (128-byte rows, 128-byte swizzle)
    if (!a.e4m3 || !encode_tmap_2d(&tm_q, a.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                                   static_cast<uint64_t>(a.B) * a.T * HH, DD, NCOL, DD))
      return cudaErrorInvalidValue;
    if (!encode_tmap_2d(&tm_k, a.kI, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, static_cast<uint64_t>(a.B) * a.S_cap, DD, KT,
                        DD))
      return cudaErrorInvalidValue;
    const int n_groups = (a.T + QPB - 1) / QPB;
    const size_t smem = sizeof(TcSmem) + 1024;
    auto kern = indexer_prefill_tc_kernel<QK_E4M3>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<dim3(n_groups, a.B), Layout::NTHREADS, smem, st>>>(tm_q, tm_k, a, n_groups, a.S_cap, dev_status);
    return cudaGetLastError();
  }
  // q as [B*T*H, 128] bf16 rows, box 256 rows; keys as [B*key_rows, 128], box 128 rows
  if (!encode_tmap_2d(&tm_q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(a.B) * a.T * HH, DD,
                      NCOL, 64))
    return cudaErrorInvalidValue;
  const void* keys = a.kI;
  int key_rows = a.S_cap;
  if (a.e4m3) {
    // e4m3 keys are widened to bf16 once per call (exact; the scale stays a
    // per-key factor applied after the head sum), then fed by TMA like bf16 keys
    if (ws_bytes < indexer_prefill_tc_ws_bytes(a.B, a.T, a.S, a.H, a.D, true) || ws == nullptr)
      return cudaErrorInvalidValue;
    const size_t chunks = static_cast<size_t>(a.B) * a.S * (DD / 16);
    const int blocks = static_cast<int>(std::min<size_t>((chunks + 255) / 256, 148 * 16));
    widen_e4m3_keys_kernel<<<blocks, 256, 0, st>>>(static_cast<const uint4*>(a.kI), static_cast<uint4*>(ws), a.B,
                                                   a.S, a.S_cap);
    keys = ws;
    key_rows = a.S;
  }
  if (!encode_tmap_2d(&tm_k, keys, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(a.B) * key_rows, DD,
                      KT, 64))
    return cudaErrorInvalidValue;
  const int n_groups = (a.T + QPB - 1) / QPB;
  const size_t smem = sizeof(TcSmem) + 1024;
  auto kern = a.e4m3 ? indexer_prefill_tc_kernel<KEYS_E4M3> : indexer_prefill_tc_kernel<KEYS_BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(n_groups, a.B);
  kern<<<grid, Layout::NTHREADS, smem, st>>>(tm_q, tm_k, a, n_groups, key_rows, dev_status);
  return cudaGetLastError();
}

}  // namespace ic
