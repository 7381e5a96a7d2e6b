// Cross-layer overlap of two top-k index tensors, per query row:
//
//     Overlap(a, b) = |I_a ∩ I_b| / k
//
// (deep-read page, "IndexCache：跨层复用稀疏注意力的索引", section
// "相邻层重叠很高，但“重叠率”不是搜索目标": the overlap of the top-k sets of
// two layers, which the page's measurement order ("一个实用的测量顺序") asks
// to record per layer next to the indexer and attention times).
//
// I_a and I_b are the SETS of valid (>= 0) positions of a row: empty (-1)
// slots and repeated positions count once at most, and the order inside a
// row does not matter.  Rows written by ic_indexer_topk are already strictly
// ascending with the -1 padding at the end; such rows skip the sort below.
//
// One CTA per row: both rows go to shared memory (invalid slots become
// INT_MAX, above every position); a row that is not already ascending is
// sorted with a bitonic network; then every thread takes entries of a that
// are valid and differ from their predecessor (so each position of a counts
// once) and binary-searches them in b.  Integer work only: the count is
// exact, and the ratio is count / k in fp32.
#include <limits.h>

#include "ic_common.cuh"
#include "ic_kernels.h"

namespace ic {
namespace {

constexpr int OV_THREADS = 256;

// Bitonic sort of n (a power of two) ints in shared memory, ascending.
__device__ void bitonic_sort(int* v, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (n >> 1); i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));   // first index of the pair
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const int x = v[lo], y = v[hi];
        if ((x > y) == up) { v[lo] = y; v[hi] = x; }
      }
      __syncthreads();
    }
  }
}

// Loads a row, maps invalid slots to INT_MAX, pads to n with INT_MAX, and
// sorts it unless it is already ascending.
__device__ void load_sorted(int* v, const int32_t* row, int k, int n, int* flag) {
  if (threadIdx.x == 0) *flag = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    int x = i < k ? row[i] : -1;
    v[i] = x >= 0 ? x : INT_MAX;
  }
  __syncthreads();
  for (int i = threadIdx.x; i + 1 < n; i += blockDim.x)
    if (v[i] > v[i + 1]) *flag = 1;   // benign race: every writer stores 1
  __syncthreads();
  if (*flag) bitonic_sort(v, n);
}

__global__ void __launch_bounds__(OV_THREADS) overlap_kernel(const int32_t* __restrict__ ia,
                                                             const int32_t* __restrict__ ib, int k, int n,
                                                             float* __restrict__ ratio, int32_t* __restrict__ count) {
  extern __shared__ int ov_smem[];
  int* va = ov_smem;
  int* vb = ov_smem + n;
  __shared__ int flag;
  __shared__ int warp_cnt[OV_THREADS / 32];
  const size_t r = blockIdx.x;
  load_sorted(va, ia + r * k, k, n, &flag);
  load_sorted(vb, ib + r * k, k, n, &flag);
  int c = 0;
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    const int x = va[i];
    if (x == INT_MAX || (i > 0 && va[i - 1] == x)) continue;
    int lo = 0, hi = k;   // first slot of b holding a value >= x
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (vb[mid] < x) lo = mid + 1; else hi = mid;
    }
    c += (lo < k && vb[lo] == x) ? 1 : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) warp_cnt[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < OV_THREADS / 32; ++w) t += warp_cnt[w];
    ratio[r] = static_cast<float>(t) / static_cast<float>(k);
    if (count) count[r] = t;
  }
}

}  // namespace

cudaError_t launch_overlap(int R, int k, const int32_t* ia, const int32_t* ib, float* ratio, int32_t* count,
                           cudaStream_t st) {
  int n = 1;
  while (n < k) n <<= 1;
  const size_t smem = 2 * static_cast<size_t>(n) * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(overlap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  overlap_kernel<<<R, OV_THREADS, smem, st>>>(ia, ib, k, n, ratio, count);
  return cudaGetLastError();
}

}  // namespace ic
