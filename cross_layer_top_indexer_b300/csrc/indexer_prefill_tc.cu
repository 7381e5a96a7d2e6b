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
// TMA in K-halves of 64 features through a 3-deep ring.  One thread issues
// the MMAs into two TMEM accumulators of 128 x 256 fp32 (all 512 columns),
// so the tensor core fills one while the epilogue drains the other.
//
// Warp roles (10 warps; 12 for e4m3 keys):
//   warp 0     TMA producer (q once, then key half-tiles; for e4m3 keys only q)
//   warp 1     TMEM allocator + MMA issuer
//   warps 2-9  epilogue: two warpgroups; warpgroup g owns query rows 2g and
//              2g+1.  Thread = one key (its TMEM lane); it reads the 64 head
//              dot products of each of its two rows, forms the weighted ReLU
//              sum in registers, and runs the streaming top-k.
//   warps 10-11 (e4m3 keys) widen each key tile from global memory into the
//              ring as f16, exactly (every e4m3 value is an f16), with the
//              hardware conversion.
//
// e4m3 keys: the MMA runs on f16 operands (kind::f16).  Each bf16 q row is
// rewritten in place as f16 times a power of two 2^e_h that brings its
// largest magnitude into [2^14, 2^15); f16 has 11 significant bits against
// bf16's 8, so every element not below 2^-17 after scaling (a relative
// 2^-31 of the row's largest) is carried exactly.  The weight w_h is
// multiplied by 2^-e_h, so the epilogue is unchanged, and the key's scale
// multiplies the score (a positive factor commutes with ReLU).
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

namespace ic {
namespace {

constexpr int QPB = 4;                   // query rows per CTA
constexpr int HH = 64;                   // indexer heads
constexpr int DD = 128;                  // indexer feature dim
constexpr int NCOL = QPB * HH;           // MMA N = 256
constexpr int KT = 128;                  // keys per tile (MMA M)
constexpr int KSTAGES = 4;               // ring of K-half tiles (16 KB each)
constexpr int CAP = kMaxK + 768;         // candidate slots per row
constexpr int WG_THREADS = 128;
constexpr int SEG = CAP / WG_THREADS;    // entries per thread in a cut
constexpr int CUT_LIMIT = CAP - 2 * KT;  // a cut leaves room for at least two tiles
constexpr int CONV_THREADS = 64;         // e4m3 keys: two converter warps

// Epilogue layout: bf16 keys run four warpgroups of one row each (four
// epilogue warps per SM sub-partition hide the tensor-memory and barrier
// latencies); e4m3 keys, whose converter warps need the registers, run two
// warpgroups of two rows each.
template <bool E4M3> struct Layout {
  static constexpr int RPW = E4M3 ? 2 : 1;                   // rows per epilogue warpgroup
  static constexpr int NWG = QPB / RPW;                      // epilogue warpgroups
  static constexpr int EPI_THREADS = NWG * WG_THREADS;
  static constexpr int CONV_WARP0 = 2 + NWG * 4;             // first converter warp (e4m3)
  static constexpr int NTHREADS = EPI_THREADS + 64 + (E4M3 ? CONV_THREADS : 0);
};
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = tc::idesc_bf16_f32(KT, NCOL);
constexpr uint32_t IDESC_F16 = tc::idesc_f16_f32(KT, NCOL);

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
  uint64_t qconv;                        // e4m3 keys: q rewritten as scaled f16
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  // per tile parity, row and key quarter: insert count, largest and smallest inserted key
  int xc[2][QPB][4];
  uint32_t xmax[2][QPB][4];
  uint32_t xmin[2][QPB][4];
  SelectScratch scr[QPB];
};

struct WgSync {
  int id;
  __device__ __forceinline__ void operator()() const { tc::named_sync(id, WG_THREADS); }
};

__device__ __forceinline__ void set_abort(TcSmem& sm, int* status) {
  sm.abort = 1;
  if (status) atomicExch(status, kDevTimeout);
}

// Eight bf16 (one 16-byte chunk) -> eight floats.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& c, float* f) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

// Two e4m3 bytes (the low 16 bits, low byte first) -> two f16, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(v)));
  return h2;
}

// Two floats -> packed f16x2 (round to nearest), `lo` in the low half.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <bool E4M3>
__global__ void __launch_bounds__(Layout<E4M3>::NTHREADS, 1)
indexer_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          IndexerArgs a, int n_groups, int* status) {
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

  using LY = Layout<E4M3>;
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
      tc::mbar_init(&sm.full[s], E4M3 ? CONV_THREADS : 1);
      tc::mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) { tc::mbar_init(&sm.tfull[s], 1); tc::mbar_init(&sm.tempty[s], LY::EPI_THREADS); }
    tc::mbar_init(&sm.qfull, 1);
    tc::mbar_init(&sm.qconv, LY::EPI_THREADS);
    tc::mbar_init(&sm.drain, 1);
    sm.abort = 0;
    tc::fence_mbar_init();
  }
  for (int i = tid; i < QPB * HH; i += kThreads) {
    const int qi = i / HH, h = i % HH;
    sm.wsm[qi][h] = qi < nq ? a.w[(static_cast<size_t>(b) * a.T + t0 + qi) * HH + h] : 0.0f;
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
      tc::mbar_arrive_expect_tx(&sm.qfull, 2 * NCOL * 128);
      tc::tma_load_2d_hint(sm.qb[0], &tm_q, &sm.qfull, 0, qrow, once);
      tc::tma_load_2d_hint(sm.qb[1], &tm_q, &sm.qfull, 64, qrow, once);
      const int krow0 = b * a.S_cap;
      int issued = 0;
      for (int it = 0; !E4M3 && it < 2 * nt; ++it) {
        const int s = it % KSTAGES;
        const uint32_t ph = (it / KSTAGES) & 1;
        if (!tc::mbar_wait(&sm.empty[s], ph ^ 1, &sm.abort, lim)) { set_abort(sm, status); break; }
        tc::mbar_arrive_expect_tx(&sm.full[s], KT * 128);
        tc::tma_load_2d_hint(sm.kst[s], &tm_k, &sm.full[s], (it & 1) * 64, krow0 + (it >> 1) * KT, keep);
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
      bool ok = tc::mbar_wait(E4M3 ? &sm.qconv : &sm.qfull, 0, &sm.abort, lim);
      if (!ok) set_abort(sm, status);
      const uint32_t qb0 = tc::smem_u32(sm.qb[0]);
      const uint32_t qb1 = tc::smem_u32(sm.qb[1]);
      for (int j = 0; ok && j < nt; ++j) {
        const int acc = j & 1;
        if (!tc::mbar_wait(&sm.tempty[acc], ((j >> 1) & 1) ^ 1, &sm.abort, lim)) { set_abort(sm, status); break; }
        tc::tc_fence_after();
        const uint32_t d_tmem = tmem + acc * NCOL;
        for (int h = 0; h < 2; ++h) {
          const int it = 2 * j + h;
          const int s = it % KSTAGES;
          if (!tc::mbar_wait(&sm.full[s], (it / KSTAGES) & 1, &sm.abort, lim)) { set_abort(sm, status); ok = false; break; }
          tc::tc_fence_after();
          const uint32_t a_base = tc::smem_u32(sm.kst[s]);
          const uint32_t b_base = h ? qb1 : qb0;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_f16(d_tmem, tc::sdesc_k_sw128(a_base + kk * 32), tc::sdesc_k_sw128(b_base + kk * 32),
                        E4M3 ? IDESC_F16 : IDESC, (h | kk) != 0);
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
  } else if (warp >= LY::CONV_WARP0) {
    // ================= e4m3 keys -> f16 operand tiles =================
    if constexpr (E4M3) {
      const int ct = tid - LY::CONV_WARP0 * 32;     // 0..63
      const uint8_t* kbase = static_cast<const uint8_t*>(a.kI);
      const long long krow0 = static_cast<long long>(b) * a.S_cap;
      const long long nrows = static_cast<long long>(a.B) * a.S_cap;
      // a tile is 128 rows x 128 B = 1024 pieces of 16 B; piece c = ct + 64u:
      // row c >> 3, features 16 (c & 7) .. +15 (a warp reads 4 whole rows)
      auto load_tile = [&](int j, uint4 (&raw)[16]) {
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int c = ct + 64 * u;
          const long long row = krow0 + static_cast<long long>(j) * KT + (c >> 3);
          raw[u] = row < nrows ? __ldg(reinterpret_cast<const uint4*>(kbase + row * DD + 16 * (c & 7)))
                               : make_uint4(0u, 0u, 0u, 0u);
        }
      };
      // both K-halves of tile j go to ring stages 2j, 2j+1
      auto store_tile = [&](int j, const uint4 (&raw)[16]) -> bool {
        const int it0 = 2 * j;
        const int s0 = it0 % KSTAGES, s1 = (it0 + 1) % KSTAGES;
        if (!tc::mbar_wait(&sm.empty[s0], ((it0 / KSTAGES) & 1) ^ 1, &sm.abort, lim)) return false;
        if (!tc::mbar_wait(&sm.empty[s1], (((it0 + 1) / KSTAGES) & 1) ^ 1, &sm.abort, lim)) return false;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int c = ct + 64 * u;
          const int r = c >> 3, pc = c & 7;
          uint8_t* dst = sm.kst[pc < 4 ? s0 : s1] + r * 128;
          const int c0 = 2 * (pc & 3);                // f16 chunks c0, c0+1 of the 64-feature half
          const uint4 x = raw[u];
          const uint4 o0 = make_uint4(e4m3x2_to_f16x2(x.x), e4m3x2_to_f16x2(x.x >> 16), e4m3x2_to_f16x2(x.y),
                                      e4m3x2_to_f16x2(x.y >> 16));
          const uint4 o1 = make_uint4(e4m3x2_to_f16x2(x.z), e4m3x2_to_f16x2(x.z >> 16), e4m3x2_to_f16x2(x.w),
                                      e4m3x2_to_f16x2(x.w >> 16));
          *reinterpret_cast<uint4*>(dst + ((c0 ^ (r & 7)) << 4)) = o0;
          *reinterpret_cast<uint4*>(dst + (((c0 + 1) ^ (r & 7)) << 4)) = o1;
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&sm.full[s0]);
        tc::mbar_arrive(&sm.full[s1]);
        return true;
      };
      // one tile's loads stay in flight while the previous one is converted
      uint4 ra[16], rb[16];
      bool ok = true;
      load_tile(0, ra);
      for (int j = 0; j < nt; j += 2) {
        if (j + 1 < nt) load_tile(j + 1, rb);
        if (!(ok = store_tile(j, ra))) break;
        if (j + 1 >= nt) break;
        if (j + 2 < nt) load_tile(j + 2, ra);
        if (!(ok = store_tile(j + 1, rb))) break;
      }
      if (!ok) set_abort(sm, status);
    }
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
    uint32_t tau[RPW];                              // a key enters iff key > tau
    uint32_t rmin[RPW], rmax[RPW];                  // bounds of the keys in the list
#pragma unroll
    for (int qq = 0; qq < RPW; ++qq) { cnt[qq] = 0; tau[qq] = 0u; rmin[qq] = 0xFFFFFFFFu; rmax[qq] = 0u; }

    if constexpr (E4M3) {
      // this warpgroup's two q rows: thread = (row q0 + wtid / 64, head wtid % 64)
      const bool okq = tc::mbar_wait(&sm.qfull, 0, &sm.abort, lim);
      if (!okq) set_abort(sm, status);
      const int qi = q0 + (wtid >> 6), hd = wtid & 63;
      const int qr = qi * HH + hd;                  // row of the 256-row B operand
      const int sw = qr & 7;
      float amax = 0.0f;
      if (okq) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float f[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(sm.qb[hh] + qr * 128 + ((c ^ sw) << 4)), f);
#pragma unroll
            for (int x = 0; x < 8; ++x) amax = fmaxf(amax, fabsf(f[x]));
          }
      }
      const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
      const int e = amax > 0.0f ? max(-120, min(126, 141 - ex)) : 0;
      const float scale = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
      const float inv_scale = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
      if (okq) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4* p = reinterpret_cast<uint4*>(sm.qb[hh] + qr * 128 + ((c ^ sw) << 4));
            float f[8];
            bf16x8_to_f32(*p, f);
            *p = make_uint4(f32x2_to_f16x2(f[0] * scale, f[1] * scale), f32x2_to_f16x2(f[2] * scale, f[3] * scale),
                            f32x2_to_f16x2(f[4] * scale, f[5] * scale), f32x2_to_f16x2(f[6] * scale, f[7] * scale));
          }
        sm.wsm[qi][hd] *= inv_scale;
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&sm.qconv);
      wsync();                                      // the warpgroup's scaled weights are in place
    }
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
          // one half of the heads at a time (fewer live registers; the other
          // epilogue warps of the sub-partition cover the load latency)
          uint32_t r[32];
          tc::tmem_ld_x32(col, r);
          tc::tmem_wait_ld();
          accumulate(r, wq);
          tc::tmem_ld_x32(col + 32, r);
          tc::tmem_wait_ld();
          accumulate(r, wq + 32);
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
        const uint32_t mx = __reduce_max_sync(0xffffffffu, take[qq] ? key[qq] : 0u);
        const uint32_t mn = __reduce_min_sync(0xffffffffu, take[qq] ? key[qq] : 0xFFFFFFFFu);
        if (lane == 0) {
          sm.xc[par][qi][quarter] = __popc(bal[qq]);
          sm.xmax[par][qi][quarter] = mx;
          sm.xmin[par][qi][quarter] = mn;
        }
      }
      // the tile's one barrier: the exchange, and one abort decision for the warpgroup
      if (tc::named_sync_or(1 + wg, WG_THREADS, !ok || sm.abort)) { aborted = true; break; }
#pragma unroll
      for (int qq = 0; qq < RPW; ++qq) {
        const int qi = q0 + qq;
        int tot = sm.xc[par][qi][0] + sm.xc[par][qi][1] + sm.xc[par][qi][2] + sm.xc[par][qi][3];
        if (cnt[qq] + tot > CAP) {
          // the list would overflow: cut it, raise tau, recount this tile's keys
          uint32_t thr;
          cnt[qq] = cut_list<WG_THREADS, SEG>(sm.cand_k[qi], sm.cand_p[qi], cnt[qq], a.k, CUT_LIMIT, rmin[qq],
                                              rmax[qq], &sm.scr[wg], wtid, wsync, &thr);
          tau[qq] = thr;
          rmin[qq] = thr;
          take[qq] = valid[qq] && key[qq] > tau[qq];
          bal[qq] = __ballot_sync(0xffffffffu, take[qq]);
          if (lane == 0) sm.xc[par][qi][quarter] = __popc(bal[qq]);
          wsync();
          tot = sm.xc[par][qi][0] + sm.xc[par][qi][1] + sm.xc[par][qi][2] + sm.xc[par][qi][3];
        }
        if (tot == 0) continue;
        int off = cnt[qq];
        for (int x = 0; x < quarter; ++x) off += sm.xc[par][qi][x];
        if (take[qq]) {
          const int slot = off + __popc(bal[qq] & lanes_below);
          sm.cand_k[qi][slot] = key[qq];
          sm.cand_p[qi][slot] = s_pos;
        }
        cnt[qq] += tot;
        rmax[qq] = max(rmax[qq], max(max(sm.xmax[par][qi][0], sm.xmax[par][qi][1]),
                                     max(sm.xmax[par][qi][2], sm.xmax[par][qi][3])));
        rmin[qq] = min(rmin[qq], min(min(sm.xmin[par][qi][0], sm.xmin[par][qi][1]),
                                     min(sm.xmin[par][qi][2], sm.xmin[par][qi][3])));
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
          c = cut_list<WG_THREADS, SEG>(sm.cand_k[qi], sm.cand_p[qi], c, a.k, a.k, rmin[qq], rmax[qq], &sm.scr[wg],
                                        wtid, wsync, &thr);
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

cudaError_t launch_indexer_prefill_tc(const IndexerArgs& a, int* dev_status, cudaStream_t st) {
  CUtensorMap tm_q, tm_k;
  // q as [B*T*H, 128] bf16 rows, box 256 rows; kI as [B*S_cap, 128], box 128 rows
  if (!encode_tmap_2d(&tm_q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(a.B) * a.T * HH, DD,
                      NCOL, 64))
    return cudaErrorInvalidValue;
  // e4m3 keys are read with plain loads; the key map is then unused
  if (a.e4m3) tm_k = tm_q;
  else if (!encode_tmap_2d(&tm_k, a.kI, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(a.B) * a.S_cap,
                           DD, KT, 64))
    return cudaErrorInvalidValue;
  const int n_groups = (a.T + QPB - 1) / QPB;
  const size_t smem = sizeof(TcSmem) + 1024;
  auto kern = a.e4m3 ? indexer_prefill_tc_kernel<true> : indexer_prefill_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(n_groups, a.B);
  kern<<<grid, a.e4m3 ? Layout<true>::NTHREADS : Layout<false>::NTHREADS, smem, st>>>(tm_q, tm_k, a, n_groups,
                                                                                   dev_status);
  return cudaGetLastError();
}

}  // namespace ic
