// Host-side launchers of the IndexCache kernels (internal to the library).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ic {

// Default limit of a bounded device wait on another role's progress.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct IndexerArgs {
  const void* q;         // [B,T,H,D] bf16
  const void* kI;        // [B,S_cap,D] bf16 or e4m3
  const float* kscale;   // [B,S_cap] (e4m3 only)
  const float* w;        // [B,T,H]
  int32_t* idx;          // [B,T,k]
  int B, T, S, S_cap, H, D, k, q_pos0, e4m3;
  uint64_t wait_ns = 0;  // limit of the tensor-core prefill kernel's waits; 0 = kWaitLimitNs
  const float* qscale = nullptr;   // [B,T,H] > 0: q given as e4m3 bytes (tensor-core prefill kernel only)
};

struct AttnArgs {
  const void* Q;         // [B,T,Hq,Dh] bf16
  const void* K;         // [B,S_cap,Dh] bf16
  const void* V;         // [B,S_cap,Dh] bf16
  const int32_t* idx;    // [B,T,k]
  void* O;               // [B,T,Hq,Dh] bf16
  int B, T, S, S_cap, Hq, Dh, k;
  float scale;
  // Nonzero: Q, K, V and idx are not written by the kernel just before this
  // launch on the stream, and everything before that kernel has completed,
  // so the tensor-core kernel reads them before its programmatic-launch wait
  // (it still waits before writing O).  Set for the Shared layers of a
  // forward, whose launch follows the previous layer's attention.
  int inputs_ready;
};

// Fused prefill indexer + streaming top-k (scores never leave the SM).
// Tensor-core (tcgen05/TMA) kernel for H = 64, D = 128, bf16 keys:
bool indexer_prefill_tc_supported(const IndexerArgs& a);
// Workspace of the tensor-core prefill path (e4m3 keys: their bf16 widening).
size_t indexer_prefill_tc_ws_bytes(int B, int T, int S, int H, int D, bool e4m3);
cudaError_t launch_indexer_prefill_tc(const IndexerArgs& a, void* ws, size_t ws_bytes, int* dev_status,
                                      cudaStream_t st);
// mma.sync kernel for every other supported shape:
cudaError_t launch_indexer_prefill(const IndexerArgs& a, int* dev_status, cudaStream_t st);

// 2-D TMA map over a row-major [rows, cols] tensor with a [box_rows, box_cols]
// box (128-byte swizzle when a box row is 128 bytes).
bool encode_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elt_bytes, uint64_t rows,
                    uint64_t cols, uint32_t box_rows, uint32_t box_cols);

// Decode indexer: score rows into ws, then an exact select per row.
// indexer_decode_ws_bytes is the least workspace the path needs (the score
// rows); indexer_decode_ws_fast_bytes adds the score-key histogram of the
// clustered select, which the path uses when the workspace holds it.
size_t indexer_decode_ws_bytes(int B, int T, int S);
size_t indexer_decode_ws_fast_bytes(int B, int T, int S);
cudaError_t launch_indexer_decode(const IndexerArgs& a, void* ws, size_t ws_bytes, int* dev_status,
                                  cudaStream_t st);
// Rows per sequence at or below which the indexer takes the decode path.
constexpr int kDecodeMaxT = 8;
// Decode select: bins of the score-key histogram the decode scorer builds
// (the top kDecHistBits bits of the order-preserving key).
constexpr int kDecHistBits = 11;
// Tensor-core decode scores for one query row per sequence, H = 64, D = 128:
bool indexer_decode_tc_supported(const IndexerArgs& a);
cudaError_t launch_indexer_decode_tc(const IndexerArgs& a, float* scores, size_t pitch, int* hist, int* dev_status,
                                     cudaStream_t st);

// Sparse attention; splits the k rows over CTAs (partials in ws) when few rows.
size_t attn_ws_bytes(int B, int T, int Hq, int Dh, int k);
cudaError_t launch_sparse_attn(const AttnArgs& a, void* ws, size_t ws_bytes, int* dev_status, cudaStream_t st);
// Tensor-core (tcgen05 + TMA gather) kernel for Hq = 32, Dh = 128 and many rows:
// The tcgen05 attention: 0 when it does not take these shapes, 1 for whole
// rows per CTA, n > 1 when each row is shared among n CTAs (few rows, e.g.
// decode), whose per-share partials (max, sum, unnormalised O; the split
// kernel's layout) are merged in a thread block cluster or by the combine
// kernel.
constexpr int kTcTargetCtas = 148;
int sparse_attn_tc_splits(const AttnArgs& a);
// nsplit > 1 with partials == nullptr: the shares of a row run as one thread
// block cluster and are merged in it (sparse_attn_tc_cluster_merge says when
// that launch is possible); otherwise they go to `partials`.
cudaError_t launch_sparse_attn_tc(const AttnArgs& a, int nsplit, float* partials, int* dev_status, cudaStream_t st);
constexpr int kTcMaxClusterSplit = 8;   // portable cluster size
bool sparse_attn_tc_cluster_merge(const AttnArgs& a, int nsplit);

// Per-row overlap |I_a ∩ I_b| / k of two index tensors [R, k] (count optional).
cudaError_t launch_overlap(int R, int k, const int32_t* ia, const int32_t* ib, float* ratio, int32_t* count,
                           cudaStream_t st);

}  // namespace ic

#include "../../include/indexcache.h"

namespace ic {
// Shared by the entry points of the library (defined in abi.cu).
ic_status report_error(ic_status st, const char* msg);
// The argument checks of ic_indexer_topk (message set on failure).
ic_status check_indexer_args(int B, int T, int S, int S_cap, int H, int D, int k, int q_pos0, const void* q,
                             const void* kI, int k_dtype, const float* k_scale, const float* w, const void* idx);
void clear_error();
int* device_status();
}  // namespace ic
