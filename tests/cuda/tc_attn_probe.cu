// Test probe for the attention building blocks:
//   * TMA tile::gather4 of 128 arbitrary rows (two 64-column halves, 128 B swizzle)
//   * S[128 keys x 32] = Kg . Q^T   (A = gathered rows, K-major; B = Q, K-major)
//   * D[128 d x 32]   = Kg^T . P    (A = gathered rows read MN-major; B = P [keys][32], MN-major, 64 B swizzle)
// The MN-major descriptors are the ones the sparse-attention kernel uses:
// A: leading byte offset = the distance between the two 64-column halves,
// stride byte offset = 1024 (8 rows of 128 B); B: stride byte offset = 512
// (8 rows of 64 B).
#include <cuda_bf16.h>

#include "../../cross_layer_top_indexer_b300/csrc/ic_kernels.h"
#include "../../cross_layer_top_indexer_b300/csrc/tc_utils.cuh"

namespace {
using namespace ic::tc;

struct __align__(1024) AttnProbeSmem {
  uint8_t a[48 * 1024];        // gathered rows: half 0 at 0, half 1 at 16 KB (+ slack)
  uint8_t q[2][32 * 128];      // Q, K-major SW128
  uint8_t p[24 * 1024];        // P [128 keys][32] bf16, 64 B rows, SW64 (+ slack)
  uint64_t full, done;
  uint32_t tmem;
};

__device__ __forceinline__ void gather4(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int r0, int r1,
                                        int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint64_t make_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(layout) << 61;
  return d;
}

__global__ void __launch_bounds__(128, 1) attn_probe_kernel(const __grid_constant__ CUtensorMap tk,
                                                            const __grid_constant__ CUtensorMap tq,
                                                            const int* idx, const __nv_bfloat16* P, float* S,
                                                            float* Dv, int* status) {
  extern __shared__ __align__(1024) unsigned char raw[];
  AttnProbeSmem& sm =
      *reinterpret_cast<AttnProbeSmem*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) { mbar_init(&sm.full, 1); mbar_init(&sm.done, 1); fence_mbar_init(); }
  if (warp == 0) { tmem_alloc(&sm.tmem, 128); tmem_relinquish(); }
  // P -> shared, MN-major rows of 64 B with the 64-byte swizzle (chunk ^= (row >> 1) & 3)
  {
    const int k = tid;   // one key row per thread
    const uint4* src = reinterpret_cast<const uint4*>(P + k * 32);
    for (int c = 0; c < 4; ++c) {
      uint4 v = src[c];
      *reinterpret_cast<uint4*>(sm.p + k * 64 + ((c ^ ((k >> 1) & 3)) * 16)) = v;
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  if (tid == 0) {
    mbar_arrive_expect_tx(&sm.full, 2 * 128 * 128 + 2 * 32 * 128);
    for (int r = 0; r < 128; r += 4) {
      gather4(sm.a + r * 128, &tk, &sm.full, 0, idx[r], idx[r + 1], idx[r + 2], idx[r + 3]);
      gather4(sm.a + 16384 + r * 128, &tk, &sm.full, 64, idx[r], idx[r + 1], idx[r + 2], idx[r + 3]);
    }
    tma_load_2d(sm.q[0], &tq, &sm.full, 0, 0);
    tma_load_2d(sm.q[1], &tq, &sm.full, 64, 0);
    if (!mbar_wait(&sm.full, 0, nullptr)) { *status = 1; }
    else {
      tc_fence_after();
      const uint32_t a0 = smem_u32(sm.a), q0 = smem_u32(sm.q[0]), q1 = smem_u32(sm.q[1]), p0 = smem_u32(sm.p);
      // S = Kg . Q^T  (K-major both, M=128, N=32)
      const uint32_t id_qk = idesc_bf16_f32(128, 32);
      for (int h = 0; h < 2; ++h)
        for (int kk = 0; kk < 4; ++kk)
          mma_f16(tmem, sdesc_k_sw128(a0 + h * 16384 + kk * 32), sdesc_k_sw128((h ? q1 : q0) + kk * 32), id_qk,
                  (h | kk) != 0);
      // D = Kg^T . P  (MN-major both, M=128 (d), N=32, K=128 keys)
      const uint32_t id_pv = idesc_bf16_f32(128, 32) | (1u << 15) | (1u << 16);
      for (int kk = 0; kk < 8; ++kk)
        mma_f16(tmem + 32, make_desc(a0 + kk * 2048, 16384, 1024, 2), make_desc(p0 + kk * 1024, 0, 512, 4), id_pv,
                kk != 0);
      mma_commit(&sm.done);
    }
  }
  __syncwarp();
  __syncthreads();
  if (!mbar_wait(&sm.done, 0, nullptr)) { if (tid == 0) *status = 2; }
  tc_fence_after();
  for (int c = 0; c < 64; c += 32) {
    uint32_t r[32];
    tmem_ld_x32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, r);
    tmem_wait_ld();
    const int row = warp * 32 + (tid & 31);
    for (int j = 0; j < 32; ++j) {
      if (c == 0) S[row * 32 + j] = __uint_as_float(r[j]);
      else Dv[row * 32 + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 128);
}
}  // namespace

extern "C" int tc_attn_probe(const void* Kmat, int rows, const void* Q, const int* idx, const void* P, float* S,
                             float* Dv, int* status) {
  CUtensorMap tk, tq;
  if (!ic::encode_tmap_2d(&tk, Kmat, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, 128, 1, 64)) return 10;
  if (!ic::encode_tmap_2d(&tq, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 32, 128, 32, 64)) return 11;
  const size_t smem = sizeof(AttnProbeSmem) + 1024;
  if (cudaFuncSetAttribute(attn_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return 12;
  attn_probe_kernel<<<1, 128, smem>>>(tk, tq, idx, reinterpret_cast<const __nv_bfloat16*>(P), S, Dv, status);
  if (cudaGetLastError() != cudaSuccess) return 13;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 14;
}
