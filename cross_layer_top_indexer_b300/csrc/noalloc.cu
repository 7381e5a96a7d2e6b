// ic_indexer_topk_noalloc: the few-rows (decode) indexer + top-k with its
// scratch memory in a fixed device array instead of a caller workspace.
//
// Who needs it: code that may not call cudaMalloc at the point where it runs
// the indexer.  Examples: a serving process whose memory manager has already
// reserved the whole GPU (for its KV-cache pool) and forbids allocations
// outside it; a plugin inside a host application that does not hand out its
// allocator; latency-critical loops where cudaMalloc is not acceptable
// because it can synchronise the device and stall other streams.  Such
// callers still pass their inputs and the index output; the score rows the
// decode path stages live in the array below.
//
// The array is a file-scope static device array of kScratchBytes.  Every GPU
// that loads this part of the library holds it until the process exits.
// All calls on a device share it and it keeps whatever the last call left:
// nothing in it needs to start at zero (every score the selection reads is
// written earlier by the same call), but two calls whose kernels overlap on
// the GPU (different streams, no ordering between them) race on it.
#include <stdio.h>

#include <mutex>

#include "ic_common.cuh"
#include "ic_kernels.h"

namespace {

constexpr size_t kScratchBytes = 32ull << 20;   // 32 MiB: 32 rows of 262144 scores

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// In host code `g_noalloc_scratch` names a host-side stand-in, not device
// memory: its device address is looked up per device, with that device
// current, and passed to the kernels.  Only a successful lookup is kept, so
// a failed first attempt (for instance one made during a stream capture) is
// retried by the next call.
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

ic_status bad(ic_status st, const char* fmt, long long a = 0, long long b = 0) {
  char buf[256];
  snprintf(buf, sizeof(buf), fmt, a, b);
  return ic::report_error(st, buf);
}

}  // namespace

extern "C" __attribute__((visibility("default"))) ic_status ic_indexer_topk_noalloc(
    int B, int T, int S, int S_cap, int H, int D, int k, int q_pos0, const void* q, const void* kI, int k_dtype,
    const float* k_scale, const float* w, int32_t* idx_out, void* stream) {
  ic::clear_error();
  if (S_cap == 0) S_cap = S;
  // the checks of ic_indexer_topk, then this entry point's own limits
  const ic_status st =
      ic::check_indexer_args(B, T, S, S_cap, H, D, k, q_pos0, q, kI, k_dtype, k_scale, w, idx_out);
  if (st != IC_OK) return st;
  if (T > ic::kDecodeMaxT)
    return bad(IC_ERR_UNSUPPORTED, "T=%lld: this entry point serves at most %lld query rows per sequence", T,
               ic::kDecodeMaxT);
  const size_t need = ic::indexer_decode_ws_bytes(B, T, S);
  if (need > kScratchBytes)
    return bad(IC_ERR_UNSUPPORTED, "these sizes need %lld bytes of scratch; the fixed array holds %lld",
               (long long)need, (long long)kScratchBytes);
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess || !scratch) {
    char buf[200];
    snprintf(buf, sizeof(buf), "cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
    return ic::report_error(IC_ERR_CUDA, buf);
  }
  ic::IndexerArgs a{q, kI, k_scale, w, idx_out, B, T, S, S_cap, H, D, k, q_pos0, k_dtype == IC_E4M3};
  e = ic::launch_indexer_decode(a, scratch, kScratchBytes, ic::device_status(), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    char buf[200];
    snprintf(buf, sizeof(buf), "indexer launch: %s", cudaGetErrorString(e));
    return ic::report_error(IC_ERR_CUDA, buf);
  }
  return IC_OK;
}
