// Test probe: one 128 x 256 x 128 bf16 tile through the same TMA, shared-memory
// descriptor, tcgen05.mma and tensor-memory load helpers the indexer uses.
// D[m][n] = sum_k A[m][k] * B[n][k], written to global memory as fp32.
#include "../../cross_layer_top_indexer_b300/csrc/ic_kernels.h"
#include "../../cross_layer_top_indexer_b300/csrc/tc_utils.cuh"

namespace {
using namespace ic::tc;

struct __align__(1024) ProbeSmem {
  uint8_t a[2][128 * 128];
  uint8_t b[2][256 * 128];
  uint64_t full, done;
  uint32_t tmem;
  int abort;
};

__global__ void __launch_bounds__(128, 1) probe_kernel(const __grid_constant__ CUtensorMap ta,
                                                       const __grid_constant__ CUtensorMap tb, float* D,
                                                       int* status) {
  extern __shared__ __align__(1024) unsigned char raw[];
  ProbeSmem& sm = *reinterpret_cast<ProbeSmem*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&sm.full, 1);
    mbar_init(&sm.done, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) { tmem_alloc(&sm.tmem, 256); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  bool ok = true;
  if (tid == 0) {
    mbar_arrive_expect_tx(&sm.full, 2 * 128 * 128 + 2 * 256 * 128);
    tma_load_2d(sm.a[0], &ta, &sm.full, 0, 0);
    tma_load_2d(sm.a[1], &ta, &sm.full, 64, 0);
    tma_load_2d(sm.b[0], &tb, &sm.full, 0, 0);
    tma_load_2d(sm.b[1], &tb, &sm.full, 64, 0);
    ok = mbar_wait(&sm.full, 0, nullptr);
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, 256);
      for (int h = 0; h < 2; ++h)
        for (int kk = 0; kk < 4; ++kk)
          mma_f16(tmem, sdesc_k_sw128(smem_u32(sm.a[h]) + kk * 32), sdesc_k_sw128(smem_u32(sm.b[h]) + kk * 32),
                  idesc, (h | kk) != 0);
      mma_commit(&sm.done);
    }
    if (!ok) { sm.abort = 1; *status = 1; }
  }
  __syncwarp();
  __syncthreads();
  if (!sm.abort) {
    if (!mbar_wait(&sm.done, 0, nullptr)) { *status = 2; }
    tc_fence_after();
    for (int c = 0; c < 256; c += 32) {
      uint32_t r[32];
      tmem_ld_x32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, r);
      tmem_wait_ld();
      for (int j = 0; j < 32; ++j) D[(warp * 32 + lane) * 256 + c + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
}
}  // namespace

extern "C" int tc_tile_probe(const void* A, const void* B, float* D, int* status) {
  CUtensorMap ta, tb;
  if (!ic::encode_tmap_2d(&ta, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 128, 128, 128, 64)) return 10;
  if (!ic::encode_tmap_2d(&tb, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 256, 128, 256, 64)) return 11;
  const size_t smem = sizeof(ProbeSmem) + 1024;
  if (cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 12;
  probe_kernel<<<1, 128, smem>>>(ta, tb, D, status);
  if (cudaGetLastError() != cudaSuccess) return 13;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 14;
}
