// C-ABI entry points of the IndexCache library: argument checks, workspace
// sizing, the F/S layer loop and the device status word.
//
// The layer loop restates the refresh/share schedule of the deep-read page
// (wineandchord.com, "IndexCache：跨层复用稀疏注意力的索引", section
// "从 DSA 的成本分解开始") and the reuse rule f(l) = max{j < l : c_j = F} of
// the notes page ("NLP--IndexCache", section "IndexCache 方法"): a Full
// layer runs the indexer and overwrites the one cached index tensor, a
// Shared layer reads it unchanged, every layer runs sparse attention.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <math.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/indexcache.h"
#include "ic_common.cuh"
#include "ic_kernels.h"

namespace {

thread_local char g_msg[512] = "";

ic_status fail(ic_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

// One device error word per GPU, written by bounded device waits.
__device__ int g_dev_status;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices];
std::once_flag g_status_once[kMaxDevices];

int* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::call_once(g_status_once[dev], [dev] {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_status) == cudaSuccess) g_status_ptr[dev] = static_cast<int*>(p);
  });
  return g_status_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Limit of the tensor-core prefill indexer's waits on other roles; 0 means
// the default (ic::kWaitLimitNs).  Set only through ic_debug_set_wait_limit_ns.
std::atomic<uint64_t> g_wait_ns{0};

}  // namespace

namespace ic {
// Message hook for entry points defined in other files of the library.
ic_status report_error(ic_status st, const char* msg) { return fail(st, "%s", msg); }
void clear_error() { g_msg[0] = 0; }
int* device_status() { return device_status_ptr(); }
}  // namespace ic

namespace {

ic_status check_indexer(int B, int T, int S, int S_cap, int H, int D, int k, int q_pos0, const void* q,
                        const void* kI, int k_dtype, const float* k_scale, const float* w, const void* idx) {
  if (B < 1 || T < 1 || S < 1 || H < 1 || D < 1 || k < 1 || q_pos0 < 0)
    return fail(IC_ERR_ARG, "sizes must be positive (B=%d T=%d S=%d H=%d D=%d k=%d q_pos0=%d)", B, T, S, H, D,
                k, q_pos0);
  if ((long long)q_pos0 + T > S) return fail(IC_ERR_ARG, "q_pos0 + T (%d + %d) exceeds S (%d)", q_pos0, T, S);
  if (S_cap < S) return fail(IC_ERR_ARG, "S_cap (%d) is smaller than S (%d)", S_cap, S);
  if (k_dtype != IC_BF16 && k_dtype != IC_E4M3) return fail(IC_ERR_ARG, "k_dtype %d unknown", k_dtype);
  if (!q || !kI || !w || !idx) return fail(IC_ERR_ARG, "null tensor pointer");
  if (k_dtype == IC_E4M3 && !k_scale) return fail(IC_ERR_ARG, "e4m3 keys need k_scale");
  if (k_dtype == IC_BF16 && k_scale) return fail(IC_ERR_ARG, "k_scale must be NULL for bf16 keys");
  if (!aligned16(q) || !aligned16(kI) || !aligned16(w) || !aligned16(idx) || (k_scale && !aligned16(k_scale)))
    return fail(IC_ERR_ARG, "tensor pointers must be 16-byte aligned");
  if (H > 64) return fail(IC_ERR_UNSUPPORTED, "H=%d: at most 64 indexer heads", H);
  if (D != 32 && D != 64 && D != 128) return fail(IC_ERR_UNSUPPORTED, "D=%d: indexer dim must be 32, 64 or 128", D);
  if (k > ic::kMaxK) return fail(IC_ERR_UNSUPPORTED, "k=%d: at most %d", k, ic::kMaxK);
  if ((long long)B * S_cap * D >= (1ll << 40)) return fail(IC_ERR_UNSUPPORTED, "key buffer too large");
  return IC_OK;
}

ic_status check_attn(int B, int T, int S, int S_cap, int Hq, int Dh, int k, const void* Q, const void* K,
                     const void* V, const void* idx, const void* O) {
  if (B < 1 || T < 1 || S < 1 || Hq < 1 || Dh < 1 || k < 1)
    return fail(IC_ERR_ARG, "sizes must be positive (B=%d T=%d S=%d Hq=%d Dh=%d k=%d)", B, T, S, Hq, Dh, k);
  if (S_cap < S) return fail(IC_ERR_ARG, "S_cap (%d) is smaller than S (%d)", S_cap, S);
  if (!Q || !K || !V || !idx || !O) return fail(IC_ERR_ARG, "null tensor pointer");
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(idx) || !aligned16(O))
    return fail(IC_ERR_ARG, "tensor pointers must be 16-byte aligned");
  if (Hq > 32) return fail(IC_ERR_UNSUPPORTED, "Hq=%d: at most 32 query heads", Hq);
  if (Dh != 64 && Dh != 128) return fail(IC_ERR_UNSUPPORTED, "Dh=%d: head dim must be 64 or 128", Dh);
  if (k > ic::kMaxK) return fail(IC_ERR_UNSUPPORTED, "k=%d: at most %d", k, ic::kMaxK);
  return IC_OK;
}

}  // namespace

namespace ic {
// Argument checks of ic_indexer_topk, shared with the other indexer entry points.
ic_status check_indexer_args(int B, int T, int S, int S_cap, int H, int D, int k, int q_pos0, const void* q,
                             const void* kI, int k_dtype, const float* k_scale, const float* w, const void* idx) {
  return check_indexer(B, T, S, S_cap, H, D, k, q_pos0, q, kI, k_dtype, k_scale, w, idx);
}
}  // namespace ic

namespace {

size_t indexer_ws(const ic_dims* d) {
  if (d->T <= ic::kDecodeMaxT) return ic::indexer_decode_ws_fast_bytes(d->B, d->T, d->S);
  return ic::indexer_prefill_tc_ws_bytes(d->B, d->T, d->S, d->H, d->D, d->k_dtype == IC_E4M3);
}

ic_status cuda_fail(cudaError_t e, const char* what) {
  return fail(IC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

ic_status run_indexer(ic::IndexerArgs a, void* ws, size_t ws_bytes, cudaStream_t st) {
  int* status = device_status_ptr();
  a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  cudaError_t e;
  if (a.T <= ic::kDecodeMaxT) {
    const size_t need = ic::indexer_decode_ws_bytes(a.B, a.T, a.S);
    if (ws_bytes < need || (need && !ws))
      return fail(IC_ERR_ARG, "workspace of %zu bytes is smaller than the %zu needed", ws_bytes, need);
    if (need && !aligned16(ws)) return fail(IC_ERR_ARG, "workspace must be 16-byte aligned");
    e = ic::launch_indexer_decode(a, ws, ws_bytes, status, st);
  } else if (ic::indexer_prefill_tc_supported(a)) {
    const size_t need = ic::indexer_prefill_tc_ws_bytes(a.B, a.T, a.S, a.H, a.D, a.e4m3 != 0);
    if (ws_bytes < need || (need && !ws))
      return fail(IC_ERR_ARG, "workspace of %zu bytes is smaller than the %zu needed", ws_bytes, need);
    if (need && !aligned16(ws)) return fail(IC_ERR_ARG, "workspace must be 16-byte aligned");
    e = ic::launch_indexer_prefill_tc(a, ws, ws_bytes, status, st);
  } else {
    e = ic::launch_indexer_prefill(a, status, st);
  }
  return e == cudaSuccess ? IC_OK : cuda_fail(e, "indexer launch");
}

ic_status run_attn(const ic::AttnArgs& a, void* ws, size_t ws_bytes, cudaStream_t st) {
  const size_t need = ic::attn_ws_bytes(a.B, a.T, a.Hq, a.Dh, a.k);
  if (ws_bytes < need || (need && !ws))
    return fail(IC_ERR_ARG, "workspace of %zu bytes is smaller than the %zu needed", ws_bytes, need);
  if (need && !aligned16(ws)) return fail(IC_ERR_ARG, "workspace must be 16-byte aligned");
  cudaError_t e = ic::launch_sparse_attn(a, ws, ws_bytes, device_status_ptr(), st);
  return e == cudaSuccess ? IC_OK : cuda_fail(e, "sparse attention launch");
}

}  // namespace

#define IC_EXPORT __attribute__((visibility("default")))

struct ic_trace {
  int n_layers = 0;
  int max_forwards = 0;
  int used = 0;
  std::vector<cudaEvent_t> events;   // [max_forwards][n_layers][4]
  std::string roles;                  // pattern of every recorded forward
};

extern "C" {

IC_EXPORT int ic_abi_version(void) { return 1; }

IC_EXPORT const char* ic_last_error(void) { return g_msg; }

IC_EXPORT size_t ic_workspace_size(const ic_dims* d) {
  if (!d || d->B < 1 || d->T < 1 || d->S < 1 || d->k < 1 || d->Hq < 1 || d->Dh < 1) return (size_t)-1;
  const size_t a = indexer_ws(d);
  const size_t b = ic::attn_ws_bytes(d->B, d->T, d->Hq, d->Dh, d->k);
  return a > b ? a : b;
}

IC_EXPORT ic_status ic_indexer_topk(int B, int T, int S, int S_cap, int H, int D, int k, int q_pos0, const void* q,
                          const void* kI, int k_dtype, const float* k_scale, const float* w, int32_t* idx_out,
                          void* ws, size_t ws_bytes, void* stream) {
  g_msg[0] = 0;
  if (S_cap == 0) S_cap = S;
  ic_status st = check_indexer(B, T, S, S_cap, H, D, k, q_pos0, q, kI, k_dtype, k_scale, w, idx_out);
  if (st != IC_OK) return st;
  ic::IndexerArgs a{q, kI, k_scale, w, idx_out, B, T, S, S_cap, H, D, k, q_pos0, k_dtype == IC_E4M3};
  return run_indexer(a, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

IC_EXPORT ic_status ic_indexer_topk_fp8(int B, int T, int S, int S_cap, int H, int D, int k, int q_pos0,
                                        const void* q, const float* q_scale, const void* kI, const float* k_scale,
                                        const float* w, int32_t* idx_out, void* stream) {
  g_msg[0] = 0;
  if (S_cap == 0) S_cap = S;
  ic_status st = check_indexer(B, T, S, S_cap, H, D, k, q_pos0, q, kI, IC_E4M3, k_scale, w, idx_out);
  if (st != IC_OK) return st;
  if (!q_scale) return fail(IC_ERR_ARG, "e4m3 queries need q_scale");
  if (!aligned16(q_scale)) return fail(IC_ERR_ARG, "tensor pointers must be 16-byte aligned");
  if (H != 64 || D != 128 || T <= ic::kDecodeMaxT)
    return fail(IC_ERR_UNSUPPORTED, "e4m3 queries: the kernel covers H=64, D=128 and more than %d query rows "
                "(got H=%d D=%d T=%d)", ic::kDecodeMaxT, H, D, T);
  ic::IndexerArgs a{q, kI, k_scale, w, idx_out, B, T, S, S_cap, H, D, k, q_pos0, 1};
  a.qscale = q_scale;
  a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  cudaError_t e = ic::launch_indexer_prefill_tc(a, nullptr, 0, device_status_ptr(), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? IC_OK : cuda_fail(e, "indexer launch");
}

IC_EXPORT ic_status ic_sparse_attn(int B, int T, int S, int S_cap, int Hq, int Dh, int k, const void* Q, const void* K,
                         const void* V, const int32_t* idx, float scale, void* O, void* ws, size_t ws_bytes,
                         void* stream) {
  g_msg[0] = 0;
  if (S_cap == 0) S_cap = S;
  ic_status st = check_attn(B, T, S, S_cap, Hq, Dh, k, Q, K, V, idx, O);
  if (st != IC_OK) return st;
  if (!(scale >= 0.0f)) return fail(IC_ERR_ARG, "scale must be >= 0");
  if (scale == 0.0f) scale = 1.0f / sqrtf((float)Dh);
  ic::AttnArgs a{Q, K, V, idx, O, B, T, S, S_cap, Hq, Dh, k, scale, 0};
  return run_attn(a, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

// Do the byte ranges [a, a + na) and [b, b + nb) share a byte?
static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

static ic_status forward_impl(const char* pattern, int n_layers, const ic_layer* layers, const ic_dims* dims,
                              int32_t* index_cache, int* indexer_calls, void* ws, size_t ws_bytes, void* stream,
                              ic_trace* trace) {
  g_msg[0] = 0;
  if (indexer_calls) *indexer_calls = 0;
  // --- the whole pattern first (nothing is launched for a bad one) ---
  if (!pattern) return fail(IC_ERR_PATTERN, "pattern is NULL");
  if (n_layers < 1) return fail(IC_ERR_PATTERN, "n_layers must be >= 1");
  const size_t len = strnlen(pattern, (size_t)n_layers + 1);
  if (len != (size_t)n_layers)
    return fail(IC_ERR_PATTERN, "pattern length %zu differs from n_layers %d", len, n_layers);
  if (pattern[0] != 'F') return fail(IC_ERR_PATTERN, "the first layer must be 'F' (a Shared layer needs an earlier Full layer)");
  for (int l = 0; l < n_layers; ++l)
    if (pattern[l] != 'F' && pattern[l] != 'S')
      return fail(IC_ERR_PATTERN, "role '%c' at layer %d: every role must be 'F' or 'S'", pattern[l], l);
  // --- sizes and every layer's pointers ---
  if (!layers || !dims || !index_cache) return fail(IC_ERR_ARG, "null layers, dims or index_cache");
  ic_dims d = *dims;
  if (d.S_cap == 0) d.S_cap = d.S;
  float scale = d.scale;
  if (!(scale >= 0.0f)) return fail(IC_ERR_ARG, "scale must be >= 0");
  if (scale == 0.0f) scale = 1.0f / sqrtf((float)(d.Dh > 0 ? d.Dh : 1));
  for (int l = 0; l < n_layers; ++l) {
    const ic_layer& L = layers[l];
    ic_status st;
    if (pattern[l] == 'F') {
      st = check_indexer(d.B, d.T, d.S, d.S_cap, d.H, d.D, d.k, d.q_pos0, L.q, L.kI, d.k_dtype, L.k_scale, L.w,
                         index_cache);
      if (st != IC_OK) return fail(st, "layer %d indexer: %s", l, std::string(g_msg).c_str());
    }
    st = check_attn(d.B, d.T, d.S, d.S_cap, d.Hq, d.Dh, d.k, L.Q, L.K, L.V, index_cache, L.O);
    if (st != IC_OK) return fail(st, "layer %d attention: %s", l, std::string(g_msg).c_str());
  }
  const size_t need = ic_workspace_size(&d);
  if (ws_bytes < need || (need && !ws))
    return fail(IC_ERR_ARG, "workspace of %zu bytes is smaller than the %zu needed", ws_bytes, need);
  cudaEvent_t* ev = nullptr;
  if (trace) {
    if (trace->n_layers != n_layers) return fail(IC_ERR_ARG, "trace made for %d layers, forward has %d", trace->n_layers, n_layers);
    if (trace->used >= trace->max_forwards) return fail(IC_ERR_ARG, "trace is full (%d forwards); read it first", trace->max_forwards);
    ev = trace->events.data() + (size_t)trace->used * 4 * n_layers;
    trace->roles.append(pattern, n_layers);
    trace->used++;
  }
  // --- the layer loop: refresh on F, share on S, attention everywhere ---
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int calls = 0;
  for (int l = 0; l < n_layers; ++l) {
    const ic_layer& L = layers[l];
    if (pattern[l] == 'F') {
      ic::IndexerArgs a{L.q, L.kI, L.k_scale, L.w, index_cache, d.B, d.T, d.S, d.S_cap, d.H, d.D, d.k, d.q_pos0,
                        d.k_dtype == IC_E4M3};
      if (ev) cudaEventRecord(ev[4 * l + 0], st);
      ic_status r = run_indexer(a, ws, ws_bytes, st);
      if (r != IC_OK) { if (indexer_calls) *indexer_calls = calls; return r; }
      if (ev) cudaEventRecord(ev[4 * l + 1], st);
      ++calls;
    }
    ic::AttnArgs a{L.Q, L.K, L.V, index_cache, L.O, d.B, d.T, d.S, d.S_cap, d.Hq, d.Dh, d.k, scale, 0};
    // a Shared layer's attention follows the previous layer's, which writes
    // only that layer's O: unless that O overlaps this layer's inputs, they
    // are complete when the launch starts
    if (pattern[l] == 'S' && l > 0) {
      const size_t q_bytes = (size_t)d.B * d.T * d.Hq * d.Dh * 2, kv_bytes = (size_t)d.B * d.S_cap * d.Dh * 2;
      const void* po = layers[l - 1].O;
      a.inputs_ready = !overlaps(po, q_bytes, L.Q, q_bytes) && !overlaps(po, q_bytes, L.K, kv_bytes) &&
                       !overlaps(po, q_bytes, L.V, kv_bytes) &&
                       !overlaps(po, q_bytes, index_cache, (size_t)d.B * d.T * d.k * 4);
    }
    if (ev) cudaEventRecord(ev[4 * l + 2], st);
    ic_status r = run_attn(a, ws, ws_bytes, st);
    if (r != IC_OK) { if (indexer_calls) *indexer_calls = calls; return r; }
    if (ev) cudaEventRecord(ev[4 * l + 3], st);
  }
  if (indexer_calls) *indexer_calls = calls;
  return IC_OK;
}

IC_EXPORT ic_status ic_forward_pattern(const char* pattern, int n_layers, const ic_layer* layers,
                                       const ic_dims* dims, int32_t* index_cache, int* indexer_calls, void* ws,
                                       size_t ws_bytes, void* stream) {
  return forward_impl(pattern, n_layers, layers, dims, index_cache, indexer_calls, ws, ws_bytes, stream, nullptr);
}

IC_EXPORT ic_status ic_forward_pattern_traced(const char* pattern, int n_layers, const ic_layer* layers,
                                              const ic_dims* dims, int32_t* index_cache, int* indexer_calls,
                                              void* ws, size_t ws_bytes, void* stream, ic_trace* trace) {
  if (!trace) { g_msg[0] = 0; return fail(IC_ERR_ARG, "trace is NULL"); }
  return forward_impl(pattern, n_layers, layers, dims, index_cache, indexer_calls, ws, ws_bytes, stream, trace);
}

IC_EXPORT ic_status ic_trace_create(int n_layers, int max_forwards, ic_trace** out) {
  g_msg[0] = 0;
  if (!out || n_layers < 1 || max_forwards < 1) return fail(IC_ERR_ARG, "bad trace arguments");
  *out = nullptr;
  ic_trace* t = new ic_trace;
  t->n_layers = n_layers;
  t->max_forwards = max_forwards;
  t->events.assign((size_t)n_layers * max_forwards * 4, nullptr);
  for (auto& e : t->events) {
    cudaError_t err = cudaEventCreate(&e);
    if (err != cudaSuccess) {
      for (auto& x : t->events) if (x) cudaEventDestroy(x);
      delete t;
      return cuda_fail(err, "cudaEventCreate");
    }
  }
  *out = t;
  return IC_OK;
}

IC_EXPORT ic_status ic_trace_destroy(ic_trace* t) {
  g_msg[0] = 0;
  if (!t) return IC_OK;
  for (auto& e : t->events) if (e) cudaEventDestroy(e);
  delete t;
  return IC_OK;
}

IC_EXPORT ic_status ic_trace_read(ic_trace* t, int* n_forwards, float* indexer_ms, float* attn_ms) {
  g_msg[0] = 0;
  if (!t) return fail(IC_ERR_ARG, "trace is NULL");
  const int L = t->n_layers;
  for (int l = 0; l < L; ++l) {
    if (indexer_ms) indexer_ms[l] = 0.0f;
    if (attn_ms) attn_ms[l] = 0.0f;
  }
  for (int f = 0; f < t->used; ++f) {
    cudaEvent_t* ev = t->events.data() + (size_t)f * 4 * L;
    cudaError_t e = cudaEventSynchronize(ev[4 * (L - 1) + 3]);
    if (e != cudaSuccess) return cuda_fail(e, "trace event");
    for (int l = 0; l < L; ++l) {
      float ms = 0.0f;
      if (t->roles[(size_t)f * L + l] == 'F') {
        e = cudaEventElapsedTime(&ms, ev[4 * l + 0], ev[4 * l + 1]);
        if (e != cudaSuccess) return cuda_fail(e, "trace elapsed");
        if (indexer_ms) indexer_ms[l] += ms;
      }
      e = cudaEventElapsedTime(&ms, ev[4 * l + 2], ev[4 * l + 3]);
      if (e != cudaSuccess) return cuda_fail(e, "trace elapsed");
      if (attn_ms) attn_ms[l] += ms;
    }
  }
  if (n_forwards) *n_forwards = t->used;
  t->used = 0;
  t->roles.clear();
  return IC_OK;
}

IC_EXPORT ic_status ic_overlap(int R, int k, const int32_t* idx_a, const int32_t* idx_b, float* ratio_out,
                               int32_t* count_out, void* stream) {
  g_msg[0] = 0;
  if (R < 1 || k < 1) return fail(IC_ERR_ARG, "sizes must be positive (R=%d k=%d)", R, k);
  if (!idx_a || !idx_b || !ratio_out) return fail(IC_ERR_ARG, "null tensor pointer");
  if (!aligned16(idx_a) || !aligned16(idx_b) || !aligned16(ratio_out) || (count_out && !aligned16(count_out)))
    return fail(IC_ERR_ARG, "tensor pointers must be 16-byte aligned");
  if (k > ic::kMaxK) return fail(IC_ERR_UNSUPPORTED, "k=%d: at most %d", k, ic::kMaxK);
  cudaError_t e = ic::launch_overlap(R, k, idx_a, idx_b, ratio_out, count_out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? IC_OK : cuda_fail(e, "overlap launch");
}

IC_EXPORT ic_status ic_debug_set_wait_limit_ns(unsigned long long ns) {
  g_msg[0] = 0;
  g_wait_ns.store(static_cast<uint64_t>(ns), std::memory_order_relaxed);
  return IC_OK;
}

IC_EXPORT ic_status ic_stream_status(void* stream) {
  g_msg[0] = 0;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream");
  int* p = device_status_ptr();
  if (!p) return fail(IC_ERR_CUDA, "device status word unavailable");
  int v = 0;
  e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (v != ic::kDevOk) {
    const int zero = 0;
    cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
    return fail(IC_ERR_DEVICE_TIMEOUT, "a bounded device wait gave up (code %d)", v);
  }
  return IC_OK;
}

}  // extern "C"
