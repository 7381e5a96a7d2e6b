/*
 * indexcache.h -- C ABI of the IndexCache hot path on NVIDIA B300 (sm_103a).
 *
 * IndexCache ("Accelerating Sparse Attention via Cross-Layer Index Reuse",
 * arXiv 2603.12201) splits the layers of a DeepSeek-Sparse-Attention model
 * into Full (F) layers, which run the lightning indexer and refresh a single
 * cached top-k index tensor, and Shared (S) layers, which skip the indexer and
 * reuse the indices of the nearest preceding F layer.  Every layer then runs
 * core attention over its k selected key/value rows only.
 *
 *   notes page (joezjh.github.io, "NLP--IndexCache"), "IndexCache 方法":
 *       roles c_l in {F, S}; an S layer uses the indices of
 *       f(l) = max{ j < l : c_j = F }.
 *   deep-read page (wineandchord.com, "IndexCache：跨层复用稀疏注意力的索引"),
 *       "从 DSA 的成本分解开始": the executable refresh/share schedule,
 *       which refuses a length mismatch, a first role other than F, and any
 *       role other than F or S.
 *   notes page, "背景 & 问题提出": for every query the indexer scores the
 *       previous tokens and keeps the top k (k = 2048); core attention cost
 *       drops from O(L^2) to O(Lk).
 *
 * Conventions for every call
 * --------------------------
 *  - Tensor arguments are DEVICE pointers owned by the caller, row-major with
 *    the innermost axis last, each 16-byte aligned.  The library never
 *    allocates device memory and keeps no pointer after a call returns.
 *  - All work is enqueued asynchronously on `stream` (a cudaStream_t, passed
 *    as void*; NULL = the legacy default stream).  No call synchronises,
 *    except ic_stream_status.
 *  - Arguments are checked before anything is enqueued: a call that returns
 *    an error has launched nothing.  ic_last_error() then returns a message
 *    (per calling thread, valid until that thread's next call).
 *  - Positions are absolute: query row t of a call sits at position
 *    q_pos0 + t and may attend to key rows 0 .. q_pos0 + t (its own position
 *    included).  Key buffers hold S_cap >= S rows per sequence; rows S ..
 *    S_cap-1 are never read (room for later decode appends).
 *  - Indices are int32, ascending within a row, padded with -1 when fewer
 *    than k positions are causal.  Ties in score go to the lower position.
 */
#ifndef INDEXCACHE_H
#define INDEXCACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ic_status {
  IC_OK = 0,
  IC_ERR_PATTERN = 1,        /* bad F/S pattern (see ic_forward_pattern)           */
  IC_ERR_ARG = 2,            /* null/misaligned pointer, bad size, small workspace */
  IC_ERR_UNSUPPORTED = 3,    /* a size the kernels do not cover (see each call)    */
  IC_ERR_CUDA = 4,           /* a CUDA launch or runtime call failed                */
  IC_ERR_DEVICE_TIMEOUT = 5  /* a bounded device-side wait gave up (reported by
                                ic_stream_status after the stream drained)         */
} ic_status;

/* Storage type of the indexer keys kI. */
enum { IC_BF16 = 0, IC_E4M3 = 1 /* OCP FP8 E4M3 (e4m3fn) with a per-row fp32 scale */ };

/* Sizes shared by the calls of one forward. */
typedef struct ic_dims {
  int B;        /* sequences in the batch                                        */
  int T;        /* query rows per sequence in this call                          */
  int S;        /* key rows visible per sequence; q_pos0 + T <= S                */
  int S_cap;    /* key rows allocated per sequence (>= S); 0 means S             */
  int H;        /* indexer heads, 1..64                                          */
  int D;        /* indexer feature dim: 32, 64 or 128                            */
  int k;        /* top-k, 1..2048                                                */
  int q_pos0;   /* absolute position of query row 0                              */
  int k_dtype;  /* IC_BF16 or IC_E4M3                                            */
  int Hq;       /* core-attention query heads, 1..32 (all share the one K/V head) */
  int Dh;       /* core-attention head dim: 64 or 128                            */
  float scale;  /* softmax scale; 0 means 1/sqrt(Dh)                             */
} ic_dims;

/* Device pointers of one layer.  q, kI, k_scale, w are read on F layers only
 * (they may be NULL on S layers); k_scale is used iff k_dtype == IC_E4M3. */
typedef struct ic_layer {
  const void* q;        /* [B, T, H, D] bf16                                      */
  const void* kI;       /* [B, S_cap, D] bf16, or e4m3 bytes                      */
  const float* k_scale; /* [B, S_cap] fp32 > 0 (IC_E4M3 only)                     */
  const float* w;       /* [B, T, H] fp32                                         */
  const void* Q;        /* [B, T, Hq, Dh] bf16                                    */
  const void* K;        /* [B, S_cap, Dh] bf16 (one K/V head shared by all Hq)    */
  const void* V;        /* [B, S_cap, Dh] bf16                                    */
  void* O;              /* [B, T, Hq, Dh] bf16 output                             */
} ic_layer;

/* Bytes of device workspace the calls below need for these sizes (the
 * maximum over ic_indexer_topk, ic_sparse_attn and ic_forward_pattern).
 * Returns 0 for sizes that need none; (size_t)-1 for invalid dims.  A
 * workspace passed to those calls is caller-owned device memory, 16-byte
 * aligned (IC_ERR_ARG otherwise). */
size_t ic_workspace_size(const ic_dims* dims);

/* Lightning indexer + top-k, one Full layer
 * (notes page, "背景 & 问题提出"; the score is the DSA indexer score):
 *
 *   I[b,t,s] = sum_h w[b,t,h] * ReLU( q[b,t,h,:] . kI[b,s,:] * k_scale[b,s] )
 *   for 0 <= s <= q_pos0 + t, and
 *   idx_out[b,t,:] = the k positions of highest I (ties: lower s), ascending,
 *                    -1 padded when q_pos0 + t + 1 < k.
 *
 * k_scale must be NULL for IC_BF16 (factor 1) and non-NULL for IC_E4M3.
 * The L x L scores are never written to memory on the prefill path; rows with
 * few queries per sequence (decode) stage one score row per query in `ws`,
 * and e4m3 keys on the prefill path take their exact bf16 widening there.
 * Errors: IC_ERR_ARG (pointers, sizes, q_pos0 + T > S, S > S_cap, workspace
 * smaller than ic_workspace_size), IC_ERR_UNSUPPORTED (H > 64, D not in
 * {32,64,128}, k > 2048), IC_ERR_CUDA. */
ic_status ic_indexer_topk(int B, int T, int S, int S_cap, int H, int D, int k, int q_pos0,
                          const void* q, const void* kI, int k_dtype, const float* k_scale,
                          const float* w, int32_t* idx_out, void* ws, size_t ws_bytes,
                          void* stream);

/* ic_indexer_topk with fp8 queries and keys (e4m3, as stored), for the
 * tensor-core fp8 rate (notes page, "背景 & 问题提出": the indexer is the
 * O(L^2) term; DSA's lightning indexer runs in low precision):
 *
 *   I[b,t,s] = sum_h w[b,t,h] * ReLU( q_scale[b,t,h] * (q8[b,t,h,:] . kI8[b,s,:]) * k_scale[b,s] )
 *
 * q [B,T,H,D] e4m3 bytes, q_scale [B,T,H] fp32 > 0, kI [B,S_cap,D] e4m3
 * bytes, k_scale [B,S_cap] fp32 > 0; the rest as for ic_indexer_topk.  The
 * scales are positive, so both leave the ReLU: the kernel multiplies w by
 * q_scale and the head sum by k_scale, and the tensor cores take the e4m3
 * bytes as stored (kind::f8f6f4).  No workspace.
 * Errors: as ic_indexer_topk; IC_ERR_UNSUPPORTED unless H = 64, D = 128 and
 * T > 8 (prefill rows). */
ic_status ic_indexer_topk_fp8(int B, int T, int S, int S_cap, int H, int D, int k, int q_pos0,
                              const void* q, const float* q_scale, const void* kI, const float* k_scale,
                              const float* w, int32_t* idx_out, void* stream);

/* Sparse core attention over selected rows (notes page, "背景 & 问题提出":
 * core attention only on the k selected tokens):
 *
 *   O[b,t,h,:] = sum_j softmax_j( scale * Q[b,t,h,:] . K[b,idx_j,:] ) V[b,idx_j,:]
 *   over the valid idx_j = idx[b,t,j] >= 0; a row with no valid index gives 0.
 *
 * Indices outside [0, S) (such as -1) are empty slots.  fp32 accumulation, bf16 output.
 * `ws` is used when few query rows are given (decode split over the k rows).
 * Errors: IC_ERR_ARG, IC_ERR_UNSUPPORTED (Hq > 32, Dh not 64/128,
 * k > 2048), IC_ERR_CUDA. */
ic_status ic_sparse_attn(int B, int T, int S, int S_cap, int Hq, int Dh, int k,
                         const void* Q, const void* K, const void* V, const int32_t* idx,
                         float scale, void* O, void* ws, size_t ws_bytes, void* stream);

/* ic_indexer_topk for few query rows (T <= 8 per sequence: the decode
 * path) that allocates nothing and takes no workspace.  The paper has no
 * counterpart to this call; it exists for callers that cannot call
 * cudaMalloc where they run the indexer, e.g. a server whose memory manager
 * owns all free device memory, a plugin without access to its host's
 * allocator, or a loop that must not take cudaMalloc's implicit device
 * synchronisation.  The score rows it stages live in a fixed 32 MiB device
 * array inside the library (held by every GPU that loads it, until exit):
 * B * T * S * 4 bytes (S rounded up to a multiple of 4) must fit, or the call
 * returns IC_ERR_UNSUPPORTED; T > 8 also returns IC_ERR_UNSUPPORTED.  The
 * first successful call on a device looks up the array's device address,
 * with that device current, and keeps it (a failed lookup is retried by the
 * next call); make that first call before any stream capture.  All calls
 * share the array: calls whose kernels may
 * overlap on the GPU race on it and must be ordered by the caller.  Nothing
 * in it needs to start at zero.  Arguments, results and other errors as for
 * ic_indexer_topk. */
ic_status ic_indexer_topk_noalloc(int B, int T, int S, int S_cap, int H, int D, int k, int q_pos0,
                                  const void* q, const void* kI, int k_dtype, const float* k_scale,
                                  const float* w, int32_t* idx_out, void* stream);

/* The F/S layer loop (deep-read page, "从 DSA 的成本分解开始"; notes page,
 * "IndexCache 方法").  `pattern` is a NUL-terminated string of n_layers
 * characters, each 'F' or 'S', the first 'F'.  The whole pattern and every
 * layer's pointers are validated before any launch (IC_ERR_PATTERN /
 * IC_ERR_ARG, nothing enqueued).  Then, for l = 0 .. n_layers-1:
 *   'F': ic_indexer_topk of layer l writes `index_cache` [B, T, k];
 *   both: ic_sparse_attn of layer l reads `index_cache`, writes layers[l].O.
 * `layers` is a HOST array of n_layers entries.  *indexer_calls (host, may be
 * NULL) receives the number of indexer launches, i.e. the count of 'F'. */
ic_status ic_forward_pattern(const char* pattern, int n_layers, const ic_layer* layers,
                             const ic_dims* dims, int32_t* index_cache, int* indexer_calls,
                             void* ws, size_t ws_bytes, void* stream);

/* Rows of one new token per sequence, for ic_decode_append (device
 * pointers; kI and k_scale are read on Full layers only). */
typedef struct ic_append_src {
  const void* kI;        /* [B, D] bf16, or e4m3 bytes                             */
  const float* k_scale;  /* [B] fp32 > 0 (IC_E4M3 only)                            */
  const void* K;         /* [B, Dh] bf16                                           */
  const void* V;         /* [B, Dh] bf16                                           */
} ic_append_src;

/* Decode step, append (notes page, "背景 & 问题提出": each query's indexer
 * scores all tokens before it; a decoded token's own keys join the caches
 * before its query runs): for every layer l and sequence b, copies
 * src[l].K[b], src[l].V[b] into layers[l].K / .V at row pos of sequence b, and
 * on Full layers src[l].kI[b] (and k_scale[b]) into layers[l].kI (.k_scale).
 * One launch for the whole stack.  `layers` and `src` are HOST arrays of
 * n_layers entries (at most 64); the pattern is checked as in
 * ic_forward_pattern.  Uses dims->B, S_cap (0 means S), D, Dh and k_dtype;
 * 0 <= pos < S_cap.  A decode step is this call, then ic_forward_pattern
 * with q_pos0 = pos, T = 1 and S = pos + 1.
 * Errors: IC_ERR_PATTERN, IC_ERR_ARG (null or misaligned pointers, pos out of
 * range), IC_ERR_UNSUPPORTED (more than 64 layers, D or Dh unsupported),
 * IC_ERR_CUDA. */
ic_status ic_decode_append(const char* pattern, int n_layers, const ic_layer* layers, const ic_append_src* src,
                           const ic_dims* dims, int pos, void* stream);

/* Per-layer tracing of the F/S loop.  The deep-read page's measurement
 * section ("一个实用的测量顺序") asks for the indexer time and the core
 * sparse-attention time of every layer before any end-to-end figure.  A
 * trace owns CUDA events (no device memory) for up to `max_forwards` traced
 * forwards of `n_layers` layers. */
typedef struct ic_trace ic_trace;
ic_status ic_trace_create(int n_layers, int max_forwards, ic_trace** out);
ic_status ic_trace_destroy(ic_trace* trace);

/* ic_forward_pattern that also records events around every launch into the
 * next free slot of `trace` (IC_ERR_ARG when the trace is full or was made
 * for another layer count). */
ic_status ic_forward_pattern_traced(const char* pattern, int n_layers, const ic_layer* layers,
                                    const ic_dims* dims, int32_t* index_cache, int* indexer_calls,
                                    void* ws, size_t ws_bytes, void* stream, ic_trace* trace);

/* Waits for the traced forwards, writes per-layer times summed over them
 * (milliseconds; indexer_ms[l] = 0 for S layers) into the HOST arrays
 * indexer_ms[n_layers] and attn_ms[n_layers] (either may be NULL),
 * *n_forwards = how many forwards were summed, and empties the trace. */
ic_status ic_trace_read(ic_trace* trace, int* n_forwards, float* indexer_ms, float* attn_ms);

/* Cross-layer overlap of two index tensors (deep-read page,
 * "相邻层重叠很高，但“重叠率”不是搜索目标": Overlap(l, j) = |I_l ∩ I_j| / k;
 * the page's measurement order, "一个实用的测量顺序", records it per layer):
 *
 *   ratio_out[r] = |A_r ∩ B_r| / k,   count_out[r] = |A_r ∩ B_r|
 *
 * where A_r and B_r are the sets of valid (>= 0) positions in row r of
 * idx_a and idx_b ([R, k] int32, device).  Empty (-1) slots and repeated
 * positions count at most once; the order within a row does not matter.
 * ratio_out [R] fp32 (device, required); count_out [R] int32 (device, may be
 * NULL).  Asynchronous on `stream`; no workspace.
 * Errors: IC_ERR_ARG (sizes < 1, null or misaligned pointers),
 * IC_ERR_UNSUPPORTED (k > 2048), IC_ERR_CUDA. */
ic_status ic_overlap(int R, int k, const int32_t* idx_a, const int32_t* idx_b, float* ratio_out,
                     int32_t* count_out, void* stream);

/* Loss of the model under an F/S pattern: `pattern` is a NUL-terminated
 * string of n_layers characters 'F'/'S'; `user` is passed through.  Return
 * NaN to stop the search with an error. */
typedef double (*ic_loss_fn)(const char* pattern, void* user);

/* Training-free greedy layer selection (notes page, "核心算法：Greedy Layer
 * Selection"; deep-read page, "Training-free：直接用语言模型损失选择 Full 层").
 * Starts from all-F; layer 0 is never removed.  Each of `removals` rounds
 * calls evaluate_loss on every pattern that turns one remaining F layer
 * (other than layer 0) into S, in ascending layer order, and commits the flip
 * with the lowest loss (ties: the lower layer).  Host code only: the loss
 * callback runs the caller's model.  Writes the final pattern (n_layers
 * characters + NUL) to the HOST buffer pattern_out and the number of loss
 * evaluations, K(N-1) - K(K-1)/2, to *forwards_out (may be NULL).
 * Errors: IC_ERR_ARG (n_layers < 1, removals outside [0, n_layers-1], null
 * callback or output, or a NaN loss; pattern_out then holds the flips
 * committed so far). */
ic_status ic_greedy_full_layers(int n_layers, int removals, ic_loss_fn evaluate_loss, void* user,
                                char* pattern_out, long long* forwards_out);

/* Waits for `stream`, then reports and clears the device error word that
 * bounded waits inside the kernels set when they give up
 * (IC_ERR_DEVICE_TIMEOUT), or IC_ERR_CUDA for a failed stream. */
ic_status ic_stream_status(void* stream);

/* Debugging aid, off by default: sets the limit, in nanoseconds of device
 * time, of every wait that the tensor-core prefill indexer (the kernel behind
 * ic_indexer_topk for H = 64, D = 128 and more than 8 query rows) makes on
 * another part of the same kernel; 0 restores the default (2 s).  A wait that
 * runs out makes the kernel wind down cleanly (no trap, no hang): its copies
 * and tensor-core work already issued are waited for, its tensor memory is
 * released, the index rows it owns are left unspecified, and the next
 * ic_stream_status returns IC_ERR_DEVICE_TIMEOUT.  Only a test of that path
 * has a reason to set a small limit.  Process-wide; affects later launches. */
ic_status ic_debug_set_wait_limit_ns(unsigned long long ns);

/* Message of the calling thread's last failed call ("" if none). */
const char* ic_last_error(void);

/* ABI version of this header: 1. */
int ic_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* INDEXCACHE_H */
