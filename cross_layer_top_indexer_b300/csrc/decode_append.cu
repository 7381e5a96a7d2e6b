// Decode step, first part: append the new token's rows to every layer's
// caches (indexer keys and their scales on Full layers, K and V on all
// layers), in one launch for the whole stack.
//
// In decode each sequence gains one token per step; its indexer key and its
// K/V rows join the caches before the step's query runs, so the query at
// position pos attends to keys 0 .. pos, itself included (notes page
// "NLP--IndexCache", "背景 & 问题提出": the indexer scores all previous
// tokens; the deep-read page's speed section measures decode at 200K).
//
// Grid (n_layers, B): one CTA copies one sequence's rows of one layer with
// 16-byte loads and stores.  Shared layers have no indexer cache of their
// own (they reuse the indices of the last Full layer), so only Full layers
// get an indexer key appended.
#include <string.h>

#include <string>

#include "ic_common.cuh"
#include "ic_kernels.h"

namespace ic {
namespace {

constexpr int kMaxAppendLayers = 64;

struct AppendLayer {
  uint8_t* kI;            // destination rows [B, S_cap, kI_bytes]
  float* ks;              // [B, S_cap] (e4m3 only)
  uint8_t* K;             // [B, S_cap, row_bytes]
  uint8_t* V;
  const uint8_t* kI_src;  // [B, kI_bytes]
  const float* ks_src;    // [B]
  const uint8_t* K_src;   // [B, row_bytes]
  const uint8_t* V_src;
};

struct AppendParams {
  int n_layers, B, S_cap, pos, kI_bytes, row_bytes;
  AppendLayer L[kMaxAppendLayers];
};

__device__ __forceinline__ void copy_row(uint8_t* dst, const uint8_t* src, int bytes) {
  for (int i = threadIdx.x; i < bytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
}

__global__ void __launch_bounds__(64) decode_append_kernel(const __grid_constant__ AppendParams p) {
  grid_dep_wait();
  grid_dep_trigger();
  const AppendLayer& L = p.L[blockIdx.x];
  const size_t b = blockIdx.y;
  const size_t row = b * p.S_cap + p.pos;
  copy_row(L.K + row * p.row_bytes, L.K_src + b * p.row_bytes, p.row_bytes);
  copy_row(L.V + row * p.row_bytes, L.V_src + b * p.row_bytes, p.row_bytes);
  if (L.kI) {
    copy_row(L.kI + row * p.kI_bytes, L.kI_src + b * p.kI_bytes, p.kI_bytes);
    if (L.ks && threadIdx.x == 0) L.ks[row] = L.ks_src[b];
  }
}

bool aligned16(const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }

ic_status fail_msg(ic_status st, const std::string& m) { return report_error(st, m.c_str()); }

}  // namespace
}  // namespace ic

extern "C" __attribute__((visibility("default"))) ic_status ic_decode_append(
    const char* pattern, int n_layers, const ic_layer* layers, const ic_append_src* src, const ic_dims* dims,
    int pos, void* stream) {
  using ic::fail_msg;
  ic::clear_error();
  if (!pattern || n_layers < 1) return fail_msg(IC_ERR_PATTERN, "pattern is NULL or n_layers < 1");
  if (strnlen(pattern, (size_t)n_layers + 1) != (size_t)n_layers)
    return fail_msg(IC_ERR_PATTERN, "pattern length differs from n_layers");
  if (pattern[0] != 'F') return fail_msg(IC_ERR_PATTERN, "the first layer must be 'F'");
  for (int l = 0; l < n_layers; ++l)
    if (pattern[l] != 'F' && pattern[l] != 'S')
      return fail_msg(IC_ERR_PATTERN, "role '" + std::string(1, pattern[l]) + "' at layer " + std::to_string(l) +
                                          ": every role must be 'F' or 'S'");
  if (!layers || !src || !dims) return fail_msg(IC_ERR_ARG, "null layers, src or dims");
  if (n_layers > ic::kMaxAppendLayers)
    return fail_msg(IC_ERR_UNSUPPORTED, "at most " + std::to_string(ic::kMaxAppendLayers) + " layers per call");
  const int B = dims->B, D = dims->D, Dh = dims->Dh;
  const int S_cap = dims->S_cap ? dims->S_cap : dims->S;
  if (B < 1 || S_cap < 1 || pos < 0 || pos >= S_cap)
    return fail_msg(IC_ERR_ARG, "need B >= 1 and 0 <= pos < S_cap (pos " + std::to_string(pos) + ", S_cap " +
                                    std::to_string(S_cap) + ")");
  if (D != 32 && D != 64 && D != 128) return fail_msg(IC_ERR_UNSUPPORTED, "indexer dim must be 32, 64 or 128");
  if (Dh != 64 && Dh != 128) return fail_msg(IC_ERR_UNSUPPORTED, "head dim must be 64 or 128");
  if (dims->k_dtype != IC_BF16 && dims->k_dtype != IC_E4M3) return fail_msg(IC_ERR_ARG, "unknown k_dtype");
  const bool e4m3 = dims->k_dtype == IC_E4M3;
  ic::AppendParams p;
  memset(&p, 0, sizeof(p));
  p.n_layers = n_layers;
  p.B = B;
  p.S_cap = S_cap;
  p.pos = pos;
  p.kI_bytes = D * (e4m3 ? 1 : 2);
  p.row_bytes = Dh * 2;
  for (int l = 0; l < n_layers; ++l) {
    const ic_layer& L = layers[l];
    const ic_append_src& s = src[l];
    const std::string at = "layer " + std::to_string(l) + ": ";
    if (!L.K || !L.V || !s.K || !s.V) return fail_msg(IC_ERR_ARG, at + "null K/V pointer");
    if (!ic::aligned16(L.K) || !ic::aligned16(L.V) || !ic::aligned16(s.K) || !ic::aligned16(s.V))
      return fail_msg(IC_ERR_ARG, at + "pointers must be 16-byte aligned");
    ic::AppendLayer& A = p.L[l];
    A.K = (uint8_t*)const_cast<void*>(L.K);
    A.V = (uint8_t*)const_cast<void*>(L.V);
    A.K_src = (const uint8_t*)s.K;
    A.V_src = (const uint8_t*)s.V;
    if (pattern[l] == 'F') {
      if (!L.kI || !s.kI) return fail_msg(IC_ERR_ARG, at + "a Full layer needs kI and its source");
      if (!ic::aligned16(L.kI) || !ic::aligned16(s.kI)) return fail_msg(IC_ERR_ARG, at + "kI must be 16-byte aligned");
      if (e4m3 != (L.k_scale != nullptr) || e4m3 != (s.k_scale != nullptr))
        return fail_msg(IC_ERR_ARG, at + "k_scale (and its source) must be given for e4m3 keys and only for them");
      A.kI = (uint8_t*)const_cast<void*>(L.kI);
      A.kI_src = (const uint8_t*)s.kI;
      A.ks = const_cast<float*>(L.k_scale);
      A.ks_src = s.k_scale;
    }
  }
  const cudaError_t e =
      ic::launch_pdl(ic::decode_append_kernel, dim3(n_layers, B), dim3(64), 0, static_cast<cudaStream_t>(stream), p);
  if (e != cudaSuccess) return fail_msg(IC_ERR_CUDA, std::string("append launch: ") + cudaGetErrorString(e));
  return IC_OK;
}
