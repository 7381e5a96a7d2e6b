// Decode indexer scores on the 5th-generation tensor cores: one query row
// per sequence (the decode step) against its whole key cache, for the
// production indexer shape H_I = 64 heads, d_I = 128, keys in e4m3 (with a
// per-row scale) or bf16.
//
// Score (DSA lightning-indexer score, the Full layers of IndexCache; notes
// page "NLP--IndexCache", section "背景 & 问题提出"):
//     I[b,s] = k_scale[b,s] * sum_h w[b,h] * ReLU(q[b,h,:] . kI[b,s,:]),  s <= pos
// (a positive scale commutes with ReLU).  One fp32 score row per sequence
// goes to the workspace, and the select kernels of the decode path pick the
// top k from it.  When given a histogram buffer, the kernel also counts the
// scores of each sequence by the top kDecHistBits bits of their order-
// preserving key (a shared-memory histogram per epilogue warpgroup, added
// into the global one at the end of each sequence), which lets the select
// find its threshold without a pass over the row.
//
// e4m3 keys go to the tensor cores as they are stored (kind::f8f6f4), so no
// thread touches a key byte.  The bf16 query is carried exactly by two e4m3
// operands: per head h a power of two 2^e_h brings max|q_h| into [128, 256),
// q_h 2^e_h = hi + lo with hi = e4m3(q_h 2^e_h) and lo = e4m3(q_h 2^e_h - hi).
// A bf16 value has 8 significant bits and an e4m3 one 4, so the remainder
// has at most 4 significant bits and lo is exact whenever it is not below the
// e4m3 subnormal step 2^-9, i.e. for every element within 2^-10 of the
// head's largest (smaller ones are off by at most 2^-10 after scaling, a
// relative 2^-17 of the head's largest term).  The MMA takes the hi and lo
// rows together as N = 128 columns (four MMAs of K = 32 per tile: the issue
// of a tcgen05.mma costs the issuing thread about as much as a small MMA
// takes to run, so fewer and larger ones keep the tensor core fed), and the
// epilogue recombines: ReLU(acc_hi + acc_lo) * (w_h 2^-e_h).
//
// The work is a stream over the key cache (132 bytes per key for e4m3), so
// the kernel is laid out to keep HBM busy: persistent CTAs each take a
// contiguous range of (sequence, 128-key tile) pairs, and
//   warp 0      TMA: key tiles (e4m3: 128 rows x 128 B, eight stages; bf16:
//               two 64-feature halves, four stages), and each sequence's q
//   warps 1, 3  MMA issuers, alternate tiles, into four TMEM accumulators
//               (keys on the lanes, heads on the columns): the issue of a
//               tcgen05.mma holds its thread for about as long as a small MMA
//               runs, so two issuers keep the tensor core busier
//   warp 2      per sequence: the q split above (e4m3) and the head weights
//   warps 4-11  epilogue, two warpgroups taking alternate tiles: thread =
//               key; the weighted ReLU sum of its 64 heads, times the key's
//               scale, written to the score row
//
// Every wait is bounded; a wait that gives up sets the CTA's abort flag and
// the device status word, every role winds down, in-flight MMAs and copies
// are waited for (bounded), and tensor memory is released before returning.
#include <cuda_fp16.h>

#include "ic_common.cuh"
#include "ic_kernels.h"
#include "tc_utils.cuh"

namespace ic {
namespace {

constexpr int HH = 64;                   // indexer heads
constexpr int DD = 128;                  // indexer feature dim
constexpr int KT = 128;                  // keys per tile (MMA M)
constexpr int KSTAGE_BYTES = 128 * 1024; // key stage ring
constexpr int RAW_TILE = KT * DD;        // e4m3 tile bytes
constexpr int BF_TILE = 2 * KT * 128;    // bf16 tile bytes (two halves)
constexpr int RSTAGES = KSTAGE_BYTES / RAW_TILE;   // 8
constexpr int BSTAGES = KSTAGE_BYTES / BF_TILE;    // 4
constexpr int NACC = 4;                  // TMEM accumulators
constexpr int ACC_COLS = 2 * HH;         // 128 columns each (bf16 keys use the first 64)
constexpr uint32_t TMEM_COLS = NACC * ACC_COLS;
constexpr int NTHREADS = 12 * 32;
constexpr int PREP_THREADS = 32;         // thread = two heads
constexpr int MMA_ISSUERS = 2;           // warps 1 and 3, alternate tiles
constexpr int EPI_GROUPS = 2;
constexpr int EPI_THREADS = 128;         // per group
constexpr int HBINS = 1 << kDecHistBits;
constexpr uint32_t IDESC_BF16 = tc::idesc_bf16_f32(KT, HH);
constexpr uint32_t IDESC_E4M3 = tc::idesc_e4m3_f32(KT, 2 * HH);

struct __align__(1024) DecTcSmem {
  uint8_t kst[KSTAGE_BYTES];             // key tiles (128 B rows, SW128)
  uint8_t qs[2][2][HH * 128];            // bf16 q of a sequence: two 64-feature halves, 64 rows x 128 B (SW128)
  uint8_t qsp[2][2 * HH * 128];          // e4m3 q split: hi rows 0-63, lo rows 64-127, 128 B each (SW128)
  float wsm[2][HH];                      // per-head weight (times 2^-e_h for e4m3)
  int hist[EPI_GROUPS][HBINS];           // per epilogue warpgroup: score keys of the current sequence
  uint64_t kfull[RSTAGES], kempty[RSTAGES];
  uint64_t qfull[2], qempty[2];          // bf16 q buffer
  uint64_t pfull[2], pempty[2];          // q split + weights ready / split free
  uint64_t wempty[2];                    // weights free
  uint64_t afull[NACC], aempty[NACC];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void set_abort(DecTcSmem& sm, int* status) {
  sm.abort = 1;
  if (status) atomicExch(status, kDevTimeout);
}

// Two floats -> two e4m3 bytes (round to nearest even, saturating): `lo_f`
// in the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo_f, float hi_f) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi_f), "f"(lo_f));
  return r;
}

// Two e4m3 bytes (low byte first) -> two floats, exactly.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(v)));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
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

template <bool E4M3>
__global__ void __launch_bounds__(NTHREADS, 1)
indexer_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         IndexerArgs a, float* scores, size_t pitch, int* hist, int ntile, int* status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  DecTcSmem& sm = *reinterpret_cast<DecTcSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr bool e4m3 = E4M3;
  constexpr int nst = E4M3 ? RSTAGES : BSTAGES;
  // this CTA's contiguous range of (sequence, tile) pairs
  const long long total = static_cast<long long>(a.B) * ntile;
  const long long u0 = total * blockIdx.x / gridDim.x;
  const long long u1 = total * (blockIdx.x + 1) / gridDim.x;
  const int n_it = static_cast<int>(u1 - u0);
  const int pos = a.q_pos0;                // the query row's position (T = 1)
  for (int i = tid; i < EPI_GROUPS * HBINS; i += NTHREADS) (&sm.hist[0][0])[i] = 0;

  if (tid == 0) {
    for (int s = 0; s < RSTAGES; ++s) { tc::mbar_init(&sm.kfull[s], 1); tc::mbar_init(&sm.kempty[s], 1); }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&sm.qfull[s], 1);
      tc::mbar_init(&sm.qempty[s], e4m3 ? PREP_THREADS : MMA_ISSUERS);
      tc::mbar_init(&sm.pfull[s], PREP_THREADS);
      tc::mbar_init(&sm.pempty[s], MMA_ISSUERS);
      tc::mbar_init(&sm.wempty[s], EPI_GROUPS * EPI_THREADS);
    }
    for (int s = 0; s < NACC; ++s) { tc::mbar_init(&sm.afull[s], 1); tc::mbar_init(&sm.aempty[s], EPI_THREADS); }
    tc::mbar_init(&sm.drain, MMA_ISSUERS);
    sm.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // The set-up above may overlap the kernel before.  With a histogram, that
  // kernel is the histogram clear, which writes nothing else and started
  // only once everything before it had completed: the roles that never
  // touch the histogram read the keys, q, w and scales at once, and only
  // the epilogue waits.  Without one, every role waits.
  if (hist == nullptr || warp >= 4) grid_dep_wait();
  grid_dep_trigger();

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      tc::tma_prefetch_map(&tm_q);
      tc::tma_prefetch_map(&tm_k);
      // every key is read once: its lines go first when L2 needs room, so the
      // stream does not push out the score rows the select reads next
      const uint64_t pol_k = tc::l2_evict_first();
      bool ok = true;
      int nseq = 0, cur_b = -1, issued_k = 0, issued_q = 0;
      int b = static_cast<int>(u0 / ntile), kt = static_cast<int>(u0 % ntile);
      for (int i = 0; ok && i < n_it; ++i, kt = kt + 1 == ntile ? 0 : kt + 1, b += kt == 0) {
        if (b != cur_b) {
          const int qb = nseq & 1;
          if (!tc::mbar_wait(&sm.qempty[qb], ((nseq >> 1) & 1) ^ 1, &sm.abort)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(&sm.qfull[qb], 2 * HH * 128);
          tc::tma_load_2d(sm.qs[qb][0], &tm_q, &sm.qfull[qb], 0, b * HH);
          tc::tma_load_2d(sm.qs[qb][1], &tm_q, &sm.qfull[qb], 64, b * HH);
          issued_q = nseq + 1;
          cur_b = b;
          ++nseq;
        }
        const int krow = b * a.S_cap + kt * KT;
        const int s = i % nst;
        if (!tc::mbar_wait(&sm.kempty[s], ((i / nst) & 1) ^ 1, &sm.abort)) { ok = false; break; }
        if (e4m3) {
          tc::mbar_arrive_expect_tx(&sm.kfull[s], RAW_TILE);
          tc::tma_load_2d_hint(sm.kst + s * RAW_TILE, &tm_k, &sm.kfull[s], 0, krow, pol_k);
        } else {
          tc::mbar_arrive_expect_tx(&sm.kfull[s], BF_TILE);
          tc::tma_load_2d_hint(sm.kst + s * BF_TILE, &tm_k, &sm.kfull[s], 0, krow, pol_k);
          tc::tma_load_2d_hint(sm.kst + s * BF_TILE + KT * 128, &tm_k, &sm.kfull[s], 64, krow, pol_k);
        }
        issued_k = i + 1;
      }
      if (!ok) set_abort(sm, status);
      // no copy of ours may still be landing in shared memory when the CTA exits
      for (int i = (issued_k > nst ? issued_k - nst : 0); i < issued_k; ++i)
        tc::mbar_wait(&sm.kfull[i % nst], (i / nst) & 1, nullptr);
      for (int n = (issued_q > 2 ? issued_q - 2 : 0); n < issued_q; ++n)
        tc::mbar_wait(&sm.qfull[n & 1], (n >> 1) & 1, nullptr);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 3) {
    // ================= MMA issuers (tile i: issuer i % 2) =================
    const int mi = warp == 1 ? 0 : 1;
    if (lane == 0) {
      bool ok = true;
      int nseq = 0, cur_b = -1, qb = 0;
      int b = static_cast<int>(u0 / ntile), kt = static_cast<int>(u0 % ntile);
      // operand descriptors are built once; a tile or K step only moves the
      // start address (16-byte units in the low bits)
      const uint64_t da0 = tc::sdesc_k_sw128(tc::smem_u32(sm.kst));
      const uint64_t dq0 = tc::sdesc_k_sw128(tc::smem_u32(E4M3 ? sm.qsp[0] : sm.qs[0][0]));
      constexpr uint32_t kTileStep = (E4M3 ? RAW_TILE : BF_TILE) >> 4;
      constexpr uint32_t kQStep = (E4M3 ? sizeof(sm.qsp[0]) : sizeof(sm.qs[0])) >> 4;
      uint64_t dq = dq0;
      for (int i = 0; ok && i < n_it; ++i, kt = kt + 1 == ntile ? 0 : kt + 1, b += kt == 0) {
        const bool last_of_seq = i + 1 == n_it || kt + 1 == ntile;
        if (b != cur_b) {
          qb = nseq & 1;
          dq = dq0 + qb * kQStep;
          uint64_t* ready = e4m3 ? &sm.pfull[qb] : &sm.qfull[qb];
          if (!tc::mbar_wait(ready, (nseq >> 1) & 1, &sm.abort)) { ok = false; break; }
          cur_b = b;
          ++nseq;
        }
        if (i % MMA_ISSUERS == mi) {
        const int acc = i % NACC;
        const int s = i % nst;
        if (!tc::mbar_wait(&sm.aempty[acc], ((i / NACC) & 1) ^ 1, &sm.abort)) { ok = false; break; }
        if (!tc::mbar_wait(&sm.kfull[s], (i / nst) & 1, &sm.abort)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t d_tmem = tmem + acc * ACC_COLS;
        const uint64_t da = da0 + s * kTileStep;
        if (e4m3) {
          // B: hi rows 0-63, lo rows 64-127 of the split q; K step = 32 B
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) tc::mma_f8f6f4(d_tmem, da + 2 * kk, dq + 2 * kk, IDESC_E4M3, kk != 0);
        } else {
          // two 64-feature halves of (KT x 128 B) for keys and (HH x 128 B) for q; K step = 32 B
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_f16(d_tmem, da + h * ((KT * 128) >> 4) + 2 * kk, dq + h * ((HH * 128) >> 4) + 2 * kk,
                          IDESC_BF16, (h | kk) != 0);
        }
        tc::mma_commit(&sm.kempty[s]);
        tc::mma_commit(&sm.afull[acc]);
        }
        // the q operand of this sequence is free once both issuers' MMAs on it are done
        if (last_of_seq) tc::mma_commit(e4m3 ? &sm.pempty[qb] : &sm.qempty[qb]);
      }
      if (!ok) set_abort(sm, status);
      tc::mma_commit(&sm.drain);
      if (!tc::mbar_wait(&sm.drain, 0, nullptr, 4000000000ull)) set_abort(sm, status);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ================= per-sequence q split and weights (thread = heads lane, lane + 32) =================
    bool ok = true;
    if (n_it > 0) {
      const int b_first = static_cast<int>(u0 / ntile), b_last = static_cast<int>((u1 - 1) / ntile);
      for (int b = b_first, n = 0; ok && b <= b_last; ++b, ++n) {
        const int qb = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        if (!tc::mbar_wait(&sm.wempty[qb], ph ^ 1, &sm.abort)) { ok = false; break; }
        if (!e4m3) {
          sm.wsm[qb][lane] = a.w[static_cast<size_t>(b) * HH + lane];
          sm.wsm[qb][lane + 32] = a.w[static_cast<size_t>(b) * HH + lane + 32];
          tc::mbar_arrive(&sm.pfull[qb]);
          continue;
        }
        if (!tc::mbar_wait(&sm.qfull[qb], ph, &sm.abort)) { ok = false; break; }
        if (!tc::mbar_wait(&sm.pempty[qb], ph ^ 1, &sm.abort)) { ok = false; break; }
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          const int h = lane + 32 * hh;
          const int sw = h & 7;
          const float w = a.w[static_cast<size_t>(b) * HH + h];
          float amax = 0.0f;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const uint8_t* src = sm.qs[qb][hf] + h * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float f[8];
              bf16x8_to_f32(*reinterpret_cast<const uint4*>(src + ((j ^ sw) << 4)), f);
#pragma unroll
              for (int t = 0; t < 8; ++t) amax = fmaxf(amax, fabsf(f[t]));
            }
          }
          // 2^e with max|q| 2^e in [128, 256); e kept where 2^e and 2^-e are normal
          const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
          const int e = amax > 0.0f ? max(-120, min(126, 134 - ex)) : 0;
          const float scale = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
          const float inv_scale = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
          uint8_t* dst_hi = sm.qsp[qb] + h * 128;
          uint8_t* dst_lo = sm.qsp[qb] + (HH + h) * 128;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            // e4m3 chunk cc = features 16cc .. 16cc+15 = bf16 chunks 2(cc&3), 2(cc&3)+1 of half cc/4
            const uint8_t* src = sm.qs[qb][cc >> 2] + h * 128;
            const int c0 = 2 * (cc & 3);
            float f[16];
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(src + ((c0 ^ sw) << 4)), f);
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(src + (((c0 + 1) ^ sw) << 4)), f + 8);
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const float x0 = f[4 * t] * scale, x1 = f[4 * t + 1] * scale;
              const float x2 = f[4 * t + 2] * scale, x3 = f[4 * t + 3] * scale;
              const uint32_t h01 = f32x2_to_e4m3x2(x0, x1), h23 = f32x2_to_e4m3x2(x2, x3);
              const float2 b01 = e4m3x2_to_f32x2(h01), b23 = e4m3x2_to_f32x2(h23);
              const uint32_t l01 = f32x2_to_e4m3x2(x0 - b01.x, x1 - b01.y);
              const uint32_t l23 = f32x2_to_e4m3x2(x2 - b23.x, x3 - b23.y);
              hw[t] = h01 | (h23 << 16);
              lw[t] = l01 | (l23 << 16);
            }
            *reinterpret_cast<uint4*>(dst_hi + ((cc ^ sw) << 4)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(dst_lo + ((cc ^ sw) << 4)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
          sm.wsm[qb][h] = w * inv_scale;
        }
        // the bf16 q buffer is released only now that its values have been
        // used, so that the next copy into it cannot overtake a load
        tc::mbar_arrive(&sm.qempty[qb]);
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&sm.pfull[qb]);
      }
    }
    if (!ok) set_abort(sm, status);
  } else {
    // ================= epilogue (thread = key lane) =================
    const int quarter = warp & 3;                   // TMEM lane quarter this warp may read
    const int grp = (warp - 4) >> 2;                // takes the tiles i with i % 2 == grp
    const int kl = quarter * 32 + lane;             // key within the tile
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    int nseq = 0, cur_b = -1, wb = 0;
    int b = static_cast<int>(u0 / ntile), kt = static_cast<int>(u0 % ntile);
    // key scales are loaded two of this group's tiles ahead so that their
    // latency stays hidden; the cursor (pb, pkt) is at tile j
    int pb = b, pkt = kt, pj = 0;
    auto scale_at = [&](int j) -> float {   // j >= pj
      for (; pj < j; ++pj)
        if (++pkt == ntile) { pkt = 0; ++pb; }
      const int ps = pkt * KT + kl;
      return (e4m3 && j < n_it && ps <= pos) ? __ldg(a.kscale + static_cast<size_t>(pb) * a.S_cap + ps) : 1.0f;
    };
    float ks_a = scale_at(grp), ks_b = scale_at(grp + EPI_GROUPS);
    // A thread whose wait gives up stops working but stays in the loop until
    // the end of the sequence, where the warpgroup decides together (one
    // barrier vote) to stop, so that no thread is left at a barrier.
    const int etid = (tid - 128) & (EPI_THREADS - 1);
    for (int i = 0; i < n_it; ++i, kt = kt + 1 == ntile ? 0 : kt + 1, b += kt == 0) {
      const bool last_of_seq = i + 1 == n_it || kt + 1 == ntile;
      if (b != cur_b) {
        wb = nseq & 1;
        if (ok && !tc::mbar_wait(&sm.pfull[wb], (nseq >> 1) & 1, &sm.abort)) { ok = false; set_abort(sm, status); }
        cur_b = b;
        ++nseq;
      }
      if (ok && i % EPI_GROUPS == grp) {
        const int s = kt * KT + kl;
        const bool valid = s <= pos;
        const float ks = ks_a;
        ks_a = ks_b;
        ks_b = scale_at(i + 2 * EPI_GROUPS);
        const int acc = i % NACC;
        if (!tc::mbar_wait(&sm.afull[acc], (i / NACC) & 1, &sm.abort)) {
          ok = false;
          set_abort(sm, status);
        } else {
          tc::tc_fence_after();
          const uint32_t ta = tmem + lane_field + acc * ACC_COLS;
          const float* wq = sm.wsm[wb];
          float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
          if (e4m3) {
#pragma unroll
            for (int hb = 0; hb < HH; hb += 32) {         // heads hb .. hb+31: hi columns, then lo columns
              uint32_t hi[32], lo[32];
              tc::tmem_ld_x32(ta + hb, hi);
              tc::tmem_ld_x32(ta + HH + hb, lo);
              tc::tmem_wait_ld();
              if (hb + 32 == HH) {
                tc::tc_fence_before();
                tc::mbar_arrive(&sm.aempty[acc]);
              }
#pragma unroll
              for (int h = 0; h < 32; h += 4) {
                const float4 w4 = *reinterpret_cast<const float4*>(wq + hb + h);
                s0 = fmaf(w4.x, fmaxf(__uint_as_float(hi[h + 0]) + __uint_as_float(lo[h + 0]), 0.0f), s0);
                s1 = fmaf(w4.y, fmaxf(__uint_as_float(hi[h + 1]) + __uint_as_float(lo[h + 1]), 0.0f), s1);
                s2 = fmaf(w4.z, fmaxf(__uint_as_float(hi[h + 2]) + __uint_as_float(lo[h + 2]), 0.0f), s2);
                s3 = fmaf(w4.w, fmaxf(__uint_as_float(hi[h + 3]) + __uint_as_float(lo[h + 3]), 0.0f), s3);
              }
            }
          } else {
            uint32_t r0[32], r1[32];
            tc::tmem_ld_x32(ta, r0);
            tc::tmem_ld_x32(ta + 32, r1);
            tc::tmem_wait_ld();
            tc::tc_fence_before();
            tc::mbar_arrive(&sm.aempty[acc]);
#pragma unroll
            for (int h = 0; h < 32; h += 4) {
              const float4 w4 = *reinterpret_cast<const float4*>(wq + h);
              s0 = fmaf(w4.x, fmaxf(__uint_as_float(r0[h + 0]), 0.0f), s0);
              s1 = fmaf(w4.y, fmaxf(__uint_as_float(r0[h + 1]), 0.0f), s1);
              s2 = fmaf(w4.z, fmaxf(__uint_as_float(r0[h + 2]), 0.0f), s2);
              s3 = fmaf(w4.w, fmaxf(__uint_as_float(r0[h + 3]), 0.0f), s3);
            }
#pragma unroll
            for (int h = 0; h < 32; h += 4) {
              const float4 w4 = *reinterpret_cast<const float4*>(wq + 32 + h);
              s0 = fmaf(w4.x, fmaxf(__uint_as_float(r1[h + 0]), 0.0f), s0);
              s1 = fmaf(w4.y, fmaxf(__uint_as_float(r1[h + 1]), 0.0f), s1);
              s2 = fmaf(w4.z, fmaxf(__uint_as_float(r1[h + 2]), 0.0f), s2);
              s3 = fmaf(w4.w, fmaxf(__uint_as_float(r1[h + 3]), 0.0f), s3);
            }
          }
          const float sc = ((s0 + s1) + (s2 + s3)) * ks;
          if (valid) {
            scores[static_cast<size_t>(b) * pitch + s] = sc;
            if (hist) atomicAdd(&sm.hist[grp][float_key(sc) >> (32 - kDecHistBits)], 1);
          }
        }
      }
      if (last_of_seq) {
        if (hist) {
          const bool stop = tc::named_sync_or(1 + grp, EPI_THREADS, !ok || sm.abort != 0);
          if (!stop) {
            int* hg = hist + static_cast<size_t>(b) * HBINS;
            for (int bin = etid; bin < HBINS; bin += EPI_THREADS) {
              const int v = sm.hist[grp][bin];
              if (v) { atomicAdd(hg + bin, v); sm.hist[grp][bin] = 0; }
            }
          }
          tc::named_sync(1 + grp, EPI_THREADS);   // the group's bins are clear before the next sequence
          if (stop) break;
        } else if (!ok) {
          break;
        }
        // the weights of this sequence are no longer read by this group
        tc::mbar_arrive(&sm.wempty[wb]);
      }
    }
    if (!ok) set_abort(sm, status);
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

bool indexer_decode_tc_supported(const IndexerArgs& a) {
  return a.T == 1 && a.H == HH && a.D == DD && static_cast<long long>(a.B) * a.S_cap < (1ll << 31) &&
         static_cast<long long>(a.B) * HH < (1ll << 31);
}

cudaError_t launch_indexer_decode_tc(const IndexerArgs& a, float* scores, size_t pitch, int* hist, int* dev_status,
                                     cudaStream_t st) {
  CUtensorMap tm_q, tm_k;
  if (!encode_tmap_2d(&tm_q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(a.B) * HH, DD, HH, 64))
    return cudaErrorInvalidValue;
  const uint64_t krows = static_cast<uint64_t>(a.B) * a.S_cap;
  const bool ok = a.e4m3 ? encode_tmap_2d(&tm_k, a.kI, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, krows, DD, KT, 128)
                         : encode_tmap_2d(&tm_k, a.kI, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, krows, DD, KT, 64);
  if (!ok) return cudaErrorInvalidValue;
  const int ntile = (a.q_pos0 + 1 + KT - 1) / KT;
  int dev = 0, n_sm = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  const long long total = static_cast<long long>(a.B) * ntile;
  const int grid = static_cast<int>(total < n_sm ? total : n_sm);
  const size_t smem = sizeof(DecTcSmem) + 1024;
  auto kern = a.e4m3 ? indexer_decode_tc_kernel<true> : indexer_decode_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(NTHREADS), smem, st, tm_q, tm_k, a, scores, pitch, hist, ntile, dev_status);
}

}  // namespace ic
