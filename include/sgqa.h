/*
 * sgqa.h -- C ABI of the Sparse GQA full-attention layer on NVIDIA B300 (sm_103a).
 *
 * The layer (Step 5 Preview pages):
 *   - ai4snews.wisdomeyes.cn news item "Step 5 Preview bets on depth over width",
 *     Interpretation, second paragraph: the indexer keys of adjacent historical
 *     positions are compressed into block representations with block size 8, which cuts
 *     the indexer and top-k cost by 8x; the selected blocks feed a sparse
 *     flash-attention operator.
 *   - ai.info article "StepFun Details Step 5 Preview's 92-Block Agent Design":
 *     "Why StepFun chose 92 transformer blocks" (the full-attention path is Gated GQA)
 *     and "Sparse GQA targets million-token context" (blocks of eight, top-k 4,096
 *     tokens, contexts up to 1M tokens).
 *   - phantomic12 catalog entry "Step 5 Preview": 64 query heads, 4 KV groups,
 *     head_dim 192, sparse indexer with topk 512 (blocks) and proxy_dim 256.
 *
 * Conventions shared by every entry point:
 *   - bf16 tensors are passed as `const void*` / `void*` and hold IEEE bfloat16 payloads.
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; the library never
 *     allocates, frees or retains device memory beyond the call.  Tensors are dense
 *     and contiguous in the layout stated next to them (row-major, last index fastest).
 *   - Every call is asynchronous on `stream`: it validates its arguments on the host,
 *     enqueues kernels and returns.  The return value reports host-detectable errors
 *     only; nothing is launched when it is not SGQA_OK.  Errors found on the device
 *     (a bounded wait that ran out, an index out of range) are recorded in a sticky
 *     per-device error word that sgqa_get_device_error() reads and clears.
 *   - Nothing aborts or throws across the ABI.
 *   - Symbols: G = num_kv_groups, Hg = heads_per_group, H = G*Hg, D = head_dim,
 *     P = proxy_dim, B = block_size, k = top_k_blocks.  A query at absolute position t
 *     owns block b_t = floor(t / B).
 */
#ifndef SGQA_H_
#define SGQA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols of the shared library (the build hides everything else). */
#if defined(SGQA_BUILD) && defined(__GNUC__)
#define SGQA_API __attribute__((visibility("default")))
#else
#define SGQA_API
#endif

/* The stream type of the CUDA runtime (cudaStream_t); 0 is the legacy default stream. */
typedef struct CUstream_st* sgqa_stream_t;

#define SGQA_ABI_VERSION 2

typedef enum {
  SGQA_OK = 0,
  SGQA_ERR_INVALID_ARGUMENT = 1,   /* null pointer, negative size, inconsistent ranges */
  SGQA_ERR_UNSUPPORTED_SHAPE = 2,  /* a dimension the library does not implement */
  SGQA_ERR_WORKSPACE_TOO_SMALL = 3,/* ws_bytes below sgqa_workspace_bytes() */
  SGQA_ERR_CUDA = 4,               /* a CUDA runtime call failed (launch, attribute, ...) */
  SGQA_ERR_DEVICE_TIMEOUT = 5,     /* a device-side bounded wait ran out */
  SGQA_ERR_DEVICE_BOUNDS = 6       /* a device-side index check failed (bad sel_idx entry) */
} sgqa_status;

typedef struct {
  int32_t num_kv_groups;    /* G >= 1 (4 on the pages) */
  int32_t heads_per_group;  /* Hg in 1..16 (16 on the pages; the 16 heads are the MMA M dim) */
  int32_t head_dim;         /* D; the library implements 192 */
  int32_t proxy_dim;        /* P in {64, 128, 192, 256} (256 on the pages) */
  int32_t block_size;       /* B in {1, 2, 4, 8, 16} (8 on the pages; 1 = token-level reference) */
  int32_t top_k_blocks;     /* k >= 1 (512 on the pages = 4,096 tokens) */
  int32_t gate_per_dim;     /* 1: gate is [T, H, D] (element-wise); 0: gate is [T, H] (per head) */
  float softmax_scale;      /* scale on q.k; <= 0 selects 1/sqrt(D) */
  int32_t attn_kernel;      /* prefill attention kernel: SGQA_ATTN_AUTO (0, the default), or
                               SGQA_ATTN_WARP / _TC_UNION / _ROUTED / _GROUPED to force one (see
                               sgqa_attention_kernel); other values are INVALID_ARGUMENT */
} sgqa_params;

/* Prefill attention kernels (sgqa_params.attn_kernel, sgqa_attention_kernel()). */
#define SGQA_ATTN_AUTO 0      /* the union kernel where its shape holds, else the warp-level one */
#define SGQA_ATTN_WARP 1      /* one warp per (row, group) on warp-level MMAs: every shape */
#define SGQA_ATTN_TC_UNION 2  /* 8 query rows per unit over the union of their selected blocks,
                                 tcgen05 with the (row, head) pairs as the MMA's M */
#define SGQA_ATTN_ROUTED 3    /* each unit of 8 query rows to the union kernel when its union is
                                 small against its rows' selections (they share many blocks),
                                 else to the warp-level kernel (needs the attention workspace) */
#define SGQA_ATTN_GROUPED 4   /* as SGQA_ATTN_ROUTED, with units of 8 rows drawn from each window of
                                 4,096 rows in the order of a MinHash signature of their
                                 selections, so rows that share blocks share units */

/* Operation selector for sgqa_workspace_bytes(). */
enum { SGQA_OP_INDEX_TOPK = 1, SGQA_OP_PREFILL = 2, SGQA_OP_DECODE = 3, SGQA_OP_ATTN = 4, SGQA_OP_PREFILL_HOST = 5 };

/* ---------------------------------------------------------------------------------
 * Block index (ai4snews item, Interpretation para 2: "compresses indexers for adjacent
 * historical positions into block representations with block size 8").
 *
 * k_blk[g, b, :] = bf16( mean of k_proxy[g, j, :] over the tokens j of block b that lie
 * before tok_end ), accumulated in fp32 in token order and rounded once to nearest-even
 * (the fp32 sum divided by the token count rounds as the exact quotient would), for every
 * block b that holds a token of [tok_begin, tok_end).  A block that is only
 * partly filled averages the tokens present; it is rebuilt when more tokens arrive.
 *
 *   k_proxy  [G, ctx_cap, P] bf16, read
 *   k_blk    [G, nb_cap, P]  bf16, written for blocks tok_begin/B .. ceil(tok_end/B)-1
 * Errors: INVALID_ARGUMENT if 0 <= tok_begin <= tok_end <= ctx_cap fails or the blocks
 * do not fit in nb_cap; UNSUPPORTED_SHAPE for P or B outside the sets above.
 * ------------------------------------------------------------------------------- */
SGQA_API sgqa_status sgqa_build_block_index(const sgqa_params* prm, const void* k_proxy, int64_t ctx_cap,
                                   int64_t tok_begin, int64_t tok_end, void* k_blk, int64_t nb_cap,
                                   sgqa_stream_t stream);

/* ---------------------------------------------------------------------------------
 * Indexer + top-k block selection (ai4snews item, Interpretation para 2; phantomic12
 * entry: "sparse indexer (topk 512, proxy_dim 256)"; ai.info article, "Sparse GQA
 * targets million-token context").
 *
 * For each query row i in [0, T) at absolute position t = q_start + i and each group g:
 *   score[b] = sum_p q_proxy[g, i, p] * k_blk[g, b, p]     for candidates 0 <= b < b_t
 *   (fp32 accumulation on the tensor cores; a plain dot product, no scale)
 *   selection = { b_t } U top-(k-1) candidates by (score descending, b descending)
 * written ascending to sel_idx[g, i, 0 .. sel_cnt[g, i]-1], the rest of the row = -1.
 * sel_cnt[g, i] = min(k, b_t + 1).
 *
 *   q_proxy  [G, T, P]       bf16, read
 *   k_blk    [G, nb_cap, P]  bf16, read; blocks 0 .. b_(q_start+T-1) - 1 must be built
 *   sel_idx  [G, T, k]       int32, written
 *   sel_cnt  [G, T]          int32, written
 *   ws       scratch of at least sgqa_workspace_bytes(prm, SGQA_OP_INDEX_TOPK, T,
 *            q_start + T, 1) bytes; a larger workspace lets more rows share one pass.
 * Rows of more than 16,384 (and 8 (k - 1)) candidates, up to 131,072, are selected without
 * writing their scores when the workspace holds that path's buffers for 8,192 rows (the
 * size sgqa_workspace_bytes returns does): the indexer writes the largest score of every 8
 * candidates, the (k-1)-th largest of those is a lower bound on the row's (k-1)-th score,
 * and only the candidates that reach it (their keys, a bit each) go to the exact
 * selection; a row with more than 4,096 of them is redone from its scores.  The selection
 * is the same either way.
 * Errors: INVALID_ARGUMENT (nulls, q_start < 0, blocks beyond nb_cap),
 * WORKSPACE_TOO_SMALL, UNSUPPORTED_SHAPE.
 * ------------------------------------------------------------------------------- */
SGQA_API sgqa_status sgqa_index_topk(const sgqa_params* prm, const void* q_proxy, int64_t T, int64_t q_start,
                            const void* k_blk, int64_t nb_cap, int32_t* sel_idx, int32_t* sel_cnt,
                            void* ws, size_t ws_bytes, sgqa_stream_t stream);

/* ---------------------------------------------------------------------------------
 * Gated sparse attention (ai.info article, "Why StepFun chose 92 transformer blocks":
 * Gated GQA; ai4snews item, Interpretation para 2: sparse flash attention over the
 * selected blocks).
 *
 * For query row i (position t = q_start + i), head h of group g = h / Hg:
 *   J = { j in blocks sel_idx[g, i, 0..sel_cnt-1] : j <= t }   (dense_mode: all j <= t)
 *   s_j = softmax_scale * q[i, h, :] . k[g, j, :]
 *   o   = sum_j softmax(s)_j v[g, j, :]             (online softmax in fp32)
 *   out[i, h, :] = bf16( o * sigmoid(gate[i, h, :]) )     (gate[i, h] if gate_per_dim=0)
 *   lse[i, h]    = log sum_j exp(s_j)                      (natural log, fp32)
 *
 *   q, gate  [T, H, D] bf16 (gate [T, H] when gate_per_dim = 0), read
 *   k, v     [G, ctx_cap, D] bf16, read (group-major: a block of a group is contiguous)
 *   sel_idx  [G, T, k] int32 ascending, sel_cnt [G, T] int32, read (ignored in dense_mode)
 *   out      [T, H, D] bf16, written;  lse [T, H] fp32, written (may be NULL)
 *   ws       scratch of sgqa_workspace_bytes(prm, SGQA_OP_ATTN, T, q_start + T, 1) bytes
 *            (about G * T * 13.5 bytes: 7.1 MB at T = 131,072), 16-byte aligned, or NULL / too
 *            small: the grouped mode (SGQA_ATTN_GROUPED, the default where the union kernel's
 *            shape holds) keeps its row order, per-unit choice and unit lists there; without
 *            it every unit runs on the union kernel.
 * A sel_idx entry outside [0, b_t] sets SGQA_ERR_DEVICE_BOUNDS on the device and the
 * entry is skipped.  Errors: INVALID_ARGUMENT, UNSUPPORTED_SHAPE (a forced kernel outside
 * its shape), WORKSPACE_TOO_SMALL (SGQA_ATTN_ROUTED / _GROUPED forced without the workspace).
 * ------------------------------------------------------------------------------- */
SGQA_API sgqa_status sgqa_sparse_attn_fwd(const sgqa_params* prm, const void* q, const void* k, const void* v,
                                 int64_t ctx_cap, const void* gate, const int32_t* sel_idx,
                                 const int32_t* sel_cnt, int64_t T, int64_t q_start, void* out, float* lse,
                                 int32_t dense_mode, void* ws, size_t ws_bytes, sgqa_stream_t stream);

/* ---------------------------------------------------------------------------------
 * Fused prefill of one Sparse GQA layer: block index over [q_start, q_start+T), then
 * indexer + top-k, then gated sparse attention, all enqueued on `stream` with no host
 * round trip.  Chunked prefill passes q_start > 0 with the blocks before q_start
 * already built in k_blk and the caches holding tokens [0, q_start+T).
 *
 *   q, gate [T, H, D]; q_proxy [G, T, P]; k, v [G, ctx_cap, D]; k_proxy [G, ctx_cap, P]
 *   k_blk   [G, nb_cap, P] (read and written); sel_idx [G, T, k]; sel_cnt [G, T]
 *   out [T, H, D] bf16; lse [T, H] fp32 or NULL
 *   ws      >= sgqa_workspace_bytes(prm, SGQA_OP_PREFILL, T, q_start + T, 1): the indexer +
 *           top-k scratch, then (reused) the attention's (see sgqa_sparse_attn_fwd)
 * ------------------------------------------------------------------------------- */
SGQA_API sgqa_status sgqa_prefill(const sgqa_params* prm, const void* q, const void* k, const void* v,
                         const void* gate, const void* q_proxy, const void* k_proxy, int64_t ctx_cap,
                         int64_t T, int64_t q_start, void* k_blk, int64_t nb_cap, int32_t* sel_idx,
                         int32_t* sel_cnt, void* out, float* lse, void* ws, size_t ws_bytes,
                         sgqa_stream_t stream);

/* ---------------------------------------------------------------------------------
 * End-to-end prefill from HOST memory: the same layer as sgqa_prefill (same passages),
 * with the host-to-device copies of the inputs and the device-to-host copy of the output
 * inside the call.  The query rows are processed in chunks of `chunk_rows` (a multiple of
 * B; <= 0 selects 4,096).  Chunk j needs the caches up to its last position only
 * (causality), so its copy-in, its prefill (a chunked prefill at q_start + its first row)
 * and its copy-out run on three streams and overlap with the neighbouring chunks: the
 * library copies in on one stream of its own, computes on `stream` and copies out on a
 * second stream of its own.  Selections are identical to one sgqa_prefill over all rows,
 * and so are outputs and LSE when chunk_rows is a multiple of 4,096 (the grouped attention
 * mode's window, which then forms the same units); other chunk sizes change only the fp32
 * summation order of the attention.
 *
 * Host tensors (pinned memory for overlapped copies; pageable memory works but the
 * copies then serialise with the host):
 *   q, gate [T, H, D] (gate [T, H] when gate_per_dim = 0); q_proxy [G, T, P];
 *   k, v [G, ctx_cap, D] and k_proxy [G, ctx_cap, P]: positions [0, q_start + T) are read
 *   (a cached prefix [0, q_start) is copied too and its blocks are built on the device);
 *   out [T, H, D] bf16 written; lse [T, H] fp32 written when not NULL.
 * Device tensors (caller-owned, same layouts; they hold the inputs and outputs afterwards):
 *   q, gate, out [T, ...]; k, v, k_proxy [G, ctx_cap, ...]; k_blk [G, nb_cap, P];
 *   lse [T, H] (required when host lse is given; may be NULL otherwise);
 *   ws >= sgqa_workspace_bytes(prm, SGQA_OP_PREFILL_HOST, T, q_start + T, chunk_rows),
 *   16-byte aligned: two q_proxy chunk buffers, the chunk's selection and the indexer
 *   workspace are carved from it.
 * Ordering: all work is ordered after what `stream` had enqueued before the call, and
 * `stream` waits for the last copy-out, so an event recorded on `stream` after the call
 * completes with the whole job (synchronise `stream` before reading host out / lse).
 * The first call on a device creates two non-blocking streams and ten events, kept until
 * the process exits; calls on one device enqueue one at a time (a mutex).  No device
 * memory is allocated.  Errors: as sgqa_prefill, checked before anything is enqueued; a
 * failed CUDA call while enqueuing returns SGQA_ERR_CUDA.
 * ------------------------------------------------------------------------------- */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  const void* gate;
  const void* q_proxy;
  const void* k_proxy;
  void* out;
  float* lse;
} sgqa_host_tensors;

typedef struct {
  void* q;
  void* k;
  void* v;
  void* gate;
  void* k_proxy;
  void* k_blk;
  int64_t nb_cap;
  void* out;
  float* lse;
  void* ws;
  size_t ws_bytes;
} sgqa_device_tensors;

SGQA_API sgqa_status sgqa_prefill_host(const sgqa_params* prm, const sgqa_host_tensors* host,
                                       const sgqa_device_tensors* dev, int64_t ctx_cap, int64_t T, int64_t q_start,
                                       int64_t chunk_rows, sgqa_stream_t stream);

/* ---------------------------------------------------------------------------------
 * Decode step for `batch` sequences packed in shared caches.  Sequence s occupies cache
 * rows [kv_off[s], kv_off[s] + ctx_len[s]); kv_off[s] is a multiple of B.  Its new
 * query sits at position ctx_len[s]-1 and its K, V and proxy key are already in the
 * caches.  Steps: (optional) rebuild the block that holds the new token from
 * k_proxy_cache; score the query proxy against the sequence's earlier blocks;
 * top-k; split-K gated attention with an LSE-weighted combine.
 *
 *   ctx_len, kv_off  HOST arrays [batch] (read during the call only); batch <= 256
 *   q, gate   [batch, H, D] bf16 (gate [batch, H] when gate_per_dim = 0)
 *   q_proxy   [G, batch, P] bf16
 *   k_cache, v_cache [G, total, D] bf16; k_proxy_cache [G, total, P] bf16 or NULL
 *   k_blk_cache [G, total / B, P] bf16 (written for the new token's block when
 *             k_proxy_cache is given); total is a multiple of B
 *   sel_idx [G, batch, k] int32, sel_cnt [G, batch] int32 (written)
 *   out [batch, H, D] bf16; lse [batch, H] fp32 or NULL
 *   ws  >= sgqa_workspace_bytes(prm, SGQA_OP_DECODE, 1, max ctx_len, batch)
 * ------------------------------------------------------------------------------- */
SGQA_API sgqa_status sgqa_decode(const sgqa_params* prm, int32_t batch, const int64_t* ctx_len, const int64_t* kv_off,
                        const void* q, const void* q_proxy, const void* gate, const void* k_cache,
                        const void* v_cache, const void* k_proxy_cache, void* k_blk_cache, int64_t total,
                        int32_t* sel_idx, int32_t* sel_cnt, void* out, float* lse, void* ws, size_t ws_bytes,
                        sgqa_stream_t stream);

/* ---------------------------------------------------------------------------------
 * Indexer + top-k without a caller-provided workspace.  No counterpart on the pages: it
 * exists for callers that cannot allocate device memory at the point of the call, for
 * example an inference engine that reserves nearly all of HBM for its KV cache at
 * start-up and hands its kernels only input and output pointers, or a plugin interface
 * whose contract passes tensors but no scratch buffer.
 *
 * Same operation, arguments and results as sgqa_index_topk, minus ws / ws_bytes.  The
 * score scratch is a file-scope device array of SGQA_NOALLOC_SCRATCH_BYTES inside this
 * library; every GPU that loads the library holds it until the process exits.  The call
 * allocates nothing (no cudaMalloc / cudaFree, no allocating library routine).
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current); make that first call before any stream capture.
 *   - All calls share the array and it keeps the last call's contents; nothing in it has
 *     to start at zero (every score the top-k reads is written earlier in the same call).
 *     Calls that overlap on the GPU (different streams, or another thread) race on it.
 *   - A request whose smallest pass (min(T, 128) query rows x G groups x the candidate
 *     count of the last row, rounded up to 4, in fp32) does not fit in the array returns
 *     SGQA_ERR_WORKSPACE_TOO_SMALL before anything is launched; larger requests that do
 *     fit run in as many passes as needed.
 * ------------------------------------------------------------------------------- */
#define SGQA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
SGQA_API sgqa_status sgqa_index_topk_noalloc(const sgqa_params* prm, const void* q_proxy, int64_t T, int64_t q_start,
                                             const void* k_blk, int64_t nb_cap, int32_t* sel_idx, int32_t* sel_cnt,
                                             sgqa_stream_t stream);

/* ---------------------------------------------------------------------------------
 * FP8 block-proxy cache (decode variant).  The pages deploy the model in FP8 (ai.info
 * article, "Why StepFun chose 92 transformer blocks") but do not say how the indexer's
 * block proxies are stored; these two entries keep them as FP8 E4M3 codes (1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits; largest finite 448), which halves the
 * bytes the decode indexer streams.
 *
 * sgqa_build_block_index_fp8: as sgqa_build_block_index, but k_blk_e4m3 is uint8 codes
 *   [G, nb_cap, P]; each block mean (fp32 sum of the bf16 proxies over the tokens
 *   present, divided by their number) is rounded once to E4M3 as the exact quotient would
 *   be, to nearest, ties to even, saturating at +-448.  Base 16-byte aligned.
 * sgqa_decode_fp8: as sgqa_decode, but k_blk_cache_e4m3 is uint8 codes [G, total / B, P]
 *   (the rebuilt block is written as E4M3).  Scores widen the codes exactly to fp32.
 * ------------------------------------------------------------------------------- */
SGQA_API sgqa_status sgqa_build_block_index_fp8(const sgqa_params* prm, const void* k_proxy, int64_t ctx_cap,
                                                int64_t tok_begin, int64_t tok_end, void* k_blk_e4m3,
                                                int64_t nb_cap, sgqa_stream_t stream);
SGQA_API sgqa_status sgqa_decode_fp8(const sgqa_params* prm, int32_t batch, const int64_t* ctx_len,
                                     const int64_t* kv_off, const void* q, const void* q_proxy, const void* gate,
                                     const void* k_cache, const void* v_cache, const void* k_proxy_cache,
                                     void* k_blk_cache_e4m3, int64_t total, int32_t* sel_idx, int32_t* sel_cnt,
                                     void* out, float* lse, void* ws, size_t ws_bytes, sgqa_stream_t stream);

/* Workspace bytes needed by `op` for T query rows ending at context length ctx_len
 * (decode: the largest ctx_len of the batch; SGQA_OP_PREFILL_HOST: `batch` carries the
 * call's chunk_rows, <= 0 for the default).  Returns 0 for an invalid request. */
SGQA_API size_t sgqa_workspace_bytes(const sgqa_params* prm, int32_t op, int64_t T, int64_t ctx_len, int32_t batch);

/* Synchronizes `stream`, then returns and clears the current device's sticky device
 * error word (SGQA_OK if no kernel recorded an error); SGQA_ERR_CUDA if the
 * synchronization itself failed. */
SGQA_API sgqa_status sgqa_get_device_error(sgqa_stream_t stream);

/* Limit, in nanoseconds, of every device-side bounded wait (mbarrier / flag polls) of
 * later launches on the current device.  Default 1e9 (one second).  0 makes each wait
 * give up at its first unsuccessful poll (used to test the timeout path). */
SGQA_API sgqa_status sgqa_set_wait_timeout_ns(uint64_t ns);

/* Self test of the bounded-wait path: launches one thread that waits on an mbarrier
 * nothing ever arrives at, for at most limit_ns.  Afterwards sgqa_get_device_error()
 * reports SGQA_ERR_DEVICE_TIMEOUT and the context stays usable.  No page counterpart:
 * this checks the library's own failure handling. */
SGQA_API sgqa_status sgqa_selftest_wait_timeout(uint64_t limit_ns, sgqa_stream_t stream);

/* Which attention kernel sgqa_sparse_attn_fwd / sgqa_prefill launch for these arguments
 * given a workspace of sgqa_workspace_bytes(...) bytes (no launch, no device access).  With
 * prm->attn_kernel = SGQA_ATTN_AUTO: SGQA_ATTN_GROUPED whenever the union kernel's shape
 * holds (blocks of 8, 16 heads per group, top_k_blocks <= 512, every block index of the
 * call below 2^18, i.e. positions below 2,097,152, not dense_mode), SGQA_ATTN_WARP
 * otherwise (an attention call without the workspace runs SGQA_ATTN_TC_UNION instead of
 * the grouped mode).  A forced kernel is returned when it can serve the call; a forced union,
 * routed or grouped kernel outside its shape returns -1, and the attention entries then fail with
 * SGQA_ERR_UNSUPPORTED_SHAPE.  Returns -1 for invalid parameters.  Decode always runs the
 * warp-level kernel (split over the context). */
SGQA_API int32_t sgqa_attention_kernel(const sgqa_params* prm, int64_t T, int64_t q_start, int32_t dense_mode);

/* Short English description of a status code (static storage). */
SGQA_API const char* sgqa_status_string(sgqa_status s);

/* SGQA_ABI_VERSION of the loaded library. */
SGQA_API int32_t sgqa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SGQA_H_ */
