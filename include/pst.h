/*
 * pst.h -- C ABI of the prefix-shared KV-tree attention library (libpst.so).
 *
 * ChunkAttention (Ye et al., "ChunkAttention: Efficient Self-Attention with
 * Prefix-Aware KV Cache and Two-Phase Partition"):
 *   Knowl 1  prefix-aware KV cache: K/V split into chunks of c tokens, kept in
 *            a prefix tree; sequences sharing leading full chunks share them.
 *   Knowl 2  two-phase partition decode: chunk-first over shared chunks,
 *            sequence-first over each sequence's own chunks.
 *   Knowl 3  partial_attn, attn_reduce (online-softmax merge), final divide.
 *   Knowl 5  chunk -> batch-range tables rebuilt and copied only on
 *            structural change (lazy context copy).
 * Chunked Prefill (onnx-genai wiki), sections 1-2: a W-row causal query block
 * attends to an append-only cache and equals single-pass prefill.
 *
 * Layers: a pool may hold the K/V of n_layers decoder layers under one prefix
 * tree (the tree and the chunk tables depend on token ids only, so every
 * layer shares them; Knowl 5 builds the context once per step, behind the
 * layers' earlier kernels).  Calls that take K/V for a token range without a
 * layer argument (insert, append, append_batch, prefill_attend, gather_kv)
 * take all layers at once, layer-major: [n_layers][n][Hkv][d].  Attention
 * calls without a layer argument read layer 0.  The *_layer calls and
 * pst_write_kv / pst_write_kv_last serve one layer at a time, for a model
 * whose layer l K/V exist only after layer l-1 ran.
 *
 * Conventions for every entry point:
 *   - Returns a pst_status; on failure pst_last_error() holds a message for
 *     the calling thread.  No C++ exception crosses this boundary.
 *   - "device" pointers are CUDA device memory on the pool's device; "host"
 *     pointers are ordinary host memory.  The caller owns every buffer it
 *     passes; the library never frees or retains caller pointers.
 *   - Tensors are dense, row-major, in the pool dtype (pst_config.dtype);
 *     attention outputs are fp32 instead when the pool has PST_FLAG_F32_OUT.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device work
 *     is enqueued asynchronously on it; host-side tree changes happen before
 *     the call returns.  All calls on one pool must be issued from one host
 *     thread and be ordered on the GPU (one stream, or caller-synchronised).
 *   - Attention scale is 1/sqrt(head_dim) (the textbook definition on the
 *     CachedAttention page, "Load-bearing equations"); query head h reads KV
 *     head h * n_kv_heads / n_q_heads (contiguous groups).
 */
#ifndef PST_H
#define PST_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PST_OK = 0,
  PST_ERR_INVALID = 1,   /* bad argument, shape, dtype or unsupported config */
  PST_ERR_OOM = 2,       /* chunk pool (or sequence table) exhausted; nothing was changed */
  PST_ERR_NOT_FOUND = 3, /* unknown or already removed sequence id */
  PST_ERR_CUDA = 4,      /* a CUDA runtime call failed (message has the CUDA error) */
  PST_ERR_STATE = 5,     /* call not valid in this state (e.g. device call on a host-only pool) */
  PST_ERR_DEVICE = 6     /* a kernel reported an error (bounded wait timed out, bad index) */
} pst_status;

typedef enum { PST_F16 = 0, PST_BF16 = 1, PST_F32 = 2 } pst_dtype;

/* pst_config.flags */
enum {
  PST_FLAG_NO_TENSOR_CORES = 1,  /* run the chunk-first phase on the CUDA-core kernel too */
  PST_FLAG_CONCURRENT_PHASES = 2, /* run the two phases at once on disjoint SMs (fork/join over an
                                     internal stream) instead of back to back */
  PST_FLAG_F32_OUT = 4            /* every attention call writes `out` as fp32 rows (the value the
                                     kernels would otherwise round to the pool dtype, round to
                                     nearest even); q and K/V stay in the pool dtype */
};

typedef struct {
  int32_t n_q_heads;   /* Hq >= 1 */
  int32_t n_kv_heads;  /* Hkv >= 1, divides Hq, Hq/Hkv in {1,2,4,8} */
  int32_t head_dim;    /* d in {64, 128} */
  int32_t chunk_size;  /* c in {16, 32, 64, 128}; for 16-bit K/V the chunk-first
                          phase runs on the tensor cores (tcgen05) in 64-key tiles:
                          four 16- or two 32-token chunks, one 64-token chunk, or
                          half of a 128-token chunk; fp32 K/V uses the CUDA-core
                          kernel for both phases */
  int64_t max_chunks;  /* pool capacity in chunks (>= 1) */
  int32_t dtype;       /* pst_dtype */
  int32_t min_share;   /* chunk-first threshold: a chunk covered by >= min_share live
                          sequences is computed chunk-first (Knowl 2 "covered by
                          multiple sequences"); 0 means 2; INT32_MAX disables phase 1 */
  int32_t max_seqs;    /* capacity of live sequences; 0 means 4096 */
  int32_t flags;       /* PST_FLAG_* */
  int32_t n_layers;    /* K/V layers under the one tree, in [0, 1024]; 0 means 1 */
} pst_config;

typedef struct pst_pool pst_pool;

typedef struct {
  int64_t live_seqs;
  int64_t used_chunks;     /* chunks on live paths */
  int64_t free_chunks;
  int64_t max_chunks;
  int64_t shared_chunks;   /* chunks computed chunk-first (after the last table build) */
  int64_t unique_tokens;   /* tokens stored in live chunks */
  int64_t logical_tokens;  /* sum of live sequence lengths */
  int64_t table_version;   /* bumps on every structural change */
  int64_t rebuild_count;   /* host table builds performed */
  double last_rebuild_us;  /* host time of the last table build */
  int64_t phase1_items;    /* work items of the last build (chunk-first) */
  int64_t phase2_items;    /* work items of the last build (sequence-first) */
  int64_t partial_rows;    /* (o, m, n) partial rows of the last build */
  int64_t graph_captures;  /* decode steps captured by pst_decode_attention_graph */
  int64_t phase1_ctas;     /* CTAs of the chunk-first kernel in the last build's decode step */
  int64_t phase2_ctas;     /* CTAs of the sequence-first kernel in the last build's decode step */
  int64_t simt_first;      /* 1: the last build's decode step launches the sequence-first kernel first */
} pst_stats_t;

/* Create a pool.  device >= 0: CUDA device ordinal; the pool allocates its
 * chunk slab (n_layers * 2 * max_chunks * Hkv * c * d elements), tables and scratch there
 * and keeps them until pst_pool_free.  device == -1: host-only pool that runs
 * the prefix tree and tables but owns no device memory; every call that needs
 * the GPU then returns PST_ERR_STATE (k/v must be NULL on insert).
 * On success *out receives the pool. */
pst_status pst_pool_create(const pst_config* cfg, int device, pst_pool** out);

/* Free the pool and all of its device memory (synchronises the device). */
pst_status pst_pool_free(pst_pool* pool);

/* Prefix lookup (Knowl 1, sequence arrival): *n_matched = number of leading
 * tokens (a multiple of c) covered by existing full chunks.  tokens: host
 * int32[n].  Does not modify the pool. */
pst_status pst_match(const pst_pool* pool, const int32_t* tokens, int64_t n, int64_t* n_matched);

/* Sequence arrival (Knowl 1): match the longest full-chunk prefix, share it,
 * allocate chunks for the rest and copy their K/V into the pool.
 * tokens: host int32[n], n >= 1.  k, v: device [n_layers][n][Hkv][d]; only rows
 * >= n_matched are read.  k = v = NULL: the tree changes but no K/V is
 * written; the caller then writes rows [n_matched, n) of every layer with
 * pst_write_kv before any attention reads them.
 * Atomic: on PST_ERR_OOM nothing changed.  *seq_id receives the new id (ids
 * count up from 0 and are never reused), *n_matched the shared token count. */
pst_status pst_insert(pst_pool* pool, const int32_t* tokens, int64_t n, const void* k, const void* v,
                      void* stream, int64_t* seq_id, int64_t* n_matched);

/* Decode append (Knowl 1, decoding iteration): write one token's K/V
 * (device [n_layers][Hkv][d] each) into the sequence's leaf chunk, or into a
 * new chunk when the leaf is full.  k = v = NULL: the token is added to the
 * tree only; write its K/V per layer with pst_write_kv_last. */
pst_status pst_append(pst_pool* pool, int64_t seq_id, int32_t token, const void* k, const void* v,
                      void* stream);

/* Batched decode append: n tokens for n distinct sequences.  seq_ids: host
 * int64[n]; tokens: host int32[n]; k, v: device [n_layers][n][Hkv][d], or both
 * NULL (tree only, as for pst_append).  One kernel launch per layer.  Atomic
 * on PST_ERR_OOM / NOT_FOUND / INVALID (duplicate ids). */
pst_status pst_append_batch(pst_pool* pool, int64_t n, const int64_t* seq_ids, const int32_t* tokens,
                            const void* k, const void* v, void* stream);

/* Sequence departure (Knowl 1): prune the path; chunks no live sequence
 * uses return to the free list (device memory is kept). */
pst_status pst_remove(pst_pool* pool, int64_t seq_id);

/* Batch order (Knowl 1 contiguity): the live sequence ids in the depth-first
 * order that rows of q/out follow.  seq_ids: host int64[cap] (may be NULL
 * when cap == 0); *B receives the live count (call with cap 0 to size). */
pst_status pst_batch_order(const pst_pool* pool, int64_t* seq_ids, int64_t cap, int64_t* B);

/* Length in tokens of a live sequence. */
pst_status pst_seq_length(const pst_pool* pool, int64_t seq_id, int64_t* n_tokens);

/* Decode attention (Knowl 2 + 3): out[u][h] = softmax(q[u][h] K_u^T / sqrt(d)) V_u
 * for every live sequence u in batch order, over all of its cached tokens.
 * q, out: device [B][Hq][d], B = live count.  Rebuilds and uploads the chunk
 * tables first if the tree changed (Knowl 5).  q and out must start on a
 * 16-byte boundary (PST_ERR_INVALID otherwise).  Chunk-first partials run on the
 * tensor cores (tcgen05) for f16/bf16 at every chunk size, sequence-first partials on
 * warp-level tensor-core products (f16/bf16) or the CUDA cores (f32), then a
 * merge kernel combines the partial rows (attn_reduce) and writes out. */
pst_status pst_decode_attention(pst_pool* pool, const void* q, void* out, void* stream);

/* Same as pst_decode_attention with HOST q/out: copies q host->device into a
 * library-owned device buffer, runs the decode step (from its CUDA graph, as
 * pst_decode_attention_graph does, while the tables keep their structure) and
 * copies out device->host on `stream`, then synchronises the stream.  q_host,
 * out_host: host [B][Hq][d] (pinned memory avoids staging copies inside the
 * CUDA runtime). */
pst_status pst_decode_attention_host(pst_pool* pool, const void* q_host, void* out_host, void* stream);

/* Decode attention that allocates nothing.  No counterpart in the paper: it
 * exists for callers that cannot allocate device memory at call time -- for
 * example a serving runtime that hands all GPU memory to its own allocator up
 * front, or a latency-critical loop where cudaMalloc / cudaFree would
 * synchronise the device.  Same inputs, outputs and result as
 * pst_decode_attention, but the partial rows live in a fixed 32 MiB device
 * area that the library defines at file scope.  The area is committed on a
 * device when the first pool is created there (pst_pool_create looks up its
 * device address, which loads the module that holds it) and stays until the
 * process exits; this call itself never loads a module or allocates.
 *   - It takes no per-phase timings (pst_set_profiling does not apply; after
 *     it, pst_phase_times reports nothing) and always launches the phases
 *     overlapped on `stream`, ignoring PST_FLAG_CONCURRENT_PHASES.
 *   - Needs the chunk tables already on the device: after a structural change
 *     (insert, remove, a new chunk on append) call pst_decode_attention once
 *     first; otherwise returns PST_ERR_STATE.  It never rebuilds or uploads.
 *   - A batch needing more than 32 MiB of scratch (about
 *     partial_rows * (d + 2) * 4 bytes, see pst_stats) returns
 *     PST_ERR_INVALID.
 *   - All calls share the one area, which keeps the last call's contents.
 *     Its first 4 bytes are the work-claim counter, which must start at zero:
 *     every call clears it with a 4-byte cudaMemsetAsync on `stream`; every
 *     partial row is written before it is read, so nothing else is cleared.
 *     Calls whose GPU work overlaps -- on different streams or from different
 *     pools -- race with each other.
 * Calls no cudaMalloc, cudaFree or other allocating routine. */
pst_status pst_decode_attention_noalloc(pst_pool* pool, const void* q, void* out, void* stream);

/* Decode attention replayed from a CUDA graph.  No counterpart in the paper:
 * it serves a decode loop (per step: pst_append_batch, then this call), where
 * the tables change structurally only every c-th step (ChunkAttention,
 * Knowl 5: the context is copied lazily) and launch latency would otherwise
 * show in every step.  Same inputs, outputs, result and errors as
 * pst_decode_attention.
 *   - It rebuilds and uploads the tables on the caller's stream when the tree
 *     changed structurally, like pst_decode_attention; then it captures the
 *     step's device work (counter reset, attention kernels, merge) into a CUDA
 *     graph on a library-owned stream and launches the graph on the caller's
 *     stream.  Later calls with the same table version and the same q and out
 *     pointers launch the same graph: one cudaGraphLaunch.  A structural
 *     change, or other q / out pointers, makes the next call capture again
 *     (pst_stats: graph_captures).
 *   - Appends that land in an existing leaf chunk change only device-side
 *     chunk lengths, which the graph's kernels read at run time.
 *   - Not while stream capture is active on the calling thread; with
 *     profiling on (pst_set_profiling) it behaves as pst_decode_attention. */
pst_status pst_decode_attention_graph(pst_pool* pool, const void* q, void* out, void* stream);

/* Chunked-prefill attend (Chunked Prefill, sections 1-2): append W tokens
 * (host tokens int32[W], device k_new/v_new [n_layers][W][Hkv][d]) to sequence seq_id at
 * positions [p0, p0+W), p0 = its current length, then out[t][h] =
 * softmax(q[t][h] K^T / sqrt(d)) V over keys [0, p0+t] of the sequence.
 * q, out: device [W][Hq][d], 16-byte aligned.  Appended tokens are never merged with other
 * sequences' chunks.  Attention reads layer 0.  Atomic on PST_ERR_OOM. */
pst_status pst_prefill_attend(pst_pool* pool, int64_t seq_id, const int32_t* tokens, int64_t W,
                              const void* q, const void* k_new, const void* v_new, void* out,
                              void* stream);

/* Append W tokens (host int32[W]) to sequence seq_id as a chunked-prefill
 * block, tree only: no K/V is written (pst_write_kv writes each layer's rows,
 * pst_prefill_attend_layer attends).  Appended tokens are never merged with
 * other sequences' chunks.  Atomic on PST_ERR_OOM.  Works on host-only pools. */
pst_status pst_extend(pst_pool* pool, int64_t seq_id, const int32_t* tokens, int64_t W);

/* Write layer `layer`'s K/V of the sequence's last n tokens (device k, v
 * [n][Hkv][d]), e.g. a block added by pst_extend or a prompt inserted with
 * k = v = NULL.  Rows in chunks that other live sequences share are not
 * written: PST_ERR_STATE (a shared chunk got its K/V from the insert that
 * created it).  One kernel launch. */
pst_status pst_write_kv(pst_pool* pool, int32_t layer, int64_t seq_id, int64_t n, const void* k,
                        const void* v, void* stream);

/* Write layer `layer`'s K/V of the last token of each of n sequences (host
 * seq_ids int64[n]; device k, v [n][Hkv][d]): the per-layer half of a decode
 * append made with k = v = NULL.  PST_ERR_STATE if a last token lies in a
 * shared chunk, PST_ERR_INVALID on a repeated id.  One kernel launch. */
pst_status pst_write_kv_last(pst_pool* pool, int32_t layer, int64_t n, const int64_t* seq_ids,
                             const void* k, const void* v, void* stream);

/* pst_decode_attention on layer `layer` (0 <= layer < n_layers): the same
 * tables, that layer's K/V. */
pst_status pst_decode_attention_layer(pst_pool* pool, int32_t layer, const void* q, void* out,
                                      void* stream);

/* pst_decode_attention_graph on layer `layer`: each layer keeps its own
 * captured step (a model's decode loop calls every layer once per step, each
 * with its own q / out buffers), captured again after a structural change. */
pst_status pst_decode_attention_graph_layer(pst_pool* pool, int32_t layer, const void* q, void* out,
                                            void* stream);

/* Causal attention of the W query rows at positions [p0, p0 + W) of sequence
 * seq_id over its keys [0, p0 + t] in layer `layer` (Chunked Prefill, sections
 * 1-2); appends nothing.  p0 + W <= the sequence's length; q, out: device
 * [W][Hq][d], 16-byte aligned. */
pst_status pst_prefill_attend_layer(pst_pool* pool, int32_t layer, int64_t seq_id, int64_t p0, int64_t W,
                                    const void* q, void* out, void* stream);

/* Read a sequence's cached K/V back into device k_out, v_out
 * [n_layers][n][Hkv][d] (n = its length), byte-exact. */
pst_status pst_gather_kv(const pst_pool* pool, int64_t seq_id, void* k_out, void* v_out, void* stream);

/* Canonical (chunk-id free) tables, for bit-exact comparison:
 *   shared_rows: int32[n_shared][4] = (depth, i, j, n_tokens) for every chunk
 *                covered by >= min_share sequences, in depth-first preorder;
 *                [i, j) is the half-open batch range it covers.
 *   seq_offsets: int64[B+1]; entries of batch row u are
 *                seq_entries[2*e .. 2*e+1] = (depth, kind), e in
 *                [seq_offsets[u], seq_offsets[u+1]), root to leaf;
 *                kind 1 = chunk-first, 0 = sequence-first.
 * Any buffer may be NULL with cap 0; the counts are always written.  Returns
 * PST_ERR_INVALID (counts still written) if a capacity is too small. */
pst_status pst_export_tables(const pst_pool* pool, int32_t* shared_rows, int64_t shared_cap,
                             int64_t* n_shared, int32_t* seq_entries, int64_t entries_cap,
                             int64_t* n_entries, int64_t* seq_offsets, int64_t offsets_cap, int64_t* B);

/* Pool statistics (Knowl 4 quantities: sharing, fragmentation). */
pst_status pst_stats(const pst_pool* pool, pst_stats_t* out);

/* Record CUDA events around each decode kernel and around the whole call. */
pst_status pst_set_profiling(pst_pool* pool, int enable);

/* Durations in ms of the last profiled decode: ms[0] chunk-first kernel,
 * ms[1] sequence-first kernel (0 when a kernel did not run), ms[2] the whole
 * call from its first kernel to the end of the merge.  Waits for those
 * events.  (The per-kernel events sit between the kernels and may keep them
 * from overlapping; time the whole call without profiling.)  After a
 * profiled prefill call: the attention kernel alone (and, when the block was
 * cut along the keys, the merge of its pieces), in ms[0] (tensor-core kernel)
 * or ms[1] (CUDA-core kernel). */
pst_status pst_phase_times(pst_pool* pool, float* ms3);

/* Kernel launches issued by the last pst_decode_attention call. */
pst_status pst_last_launch_count(const pst_pool* pool, int32_t* n);

/* Bits of the device error word. */
enum {
  PST_DEVICE_WAIT_TIMEOUT = 1, /* a bounded wait ran out; the kernel stopped early */
  PST_DEVICE_BAD_INDEX = 2     /* an index check failed; the access was skipped */
};

/* Read and clear the device error word written by kernels whose bounded
 * waits timed out or whose index checks failed (synchronises the device).
 * *code == 0 means no error, else an OR of PST_DEVICE_* bits. */
pst_status pst_check_device(pst_pool* pool, int32_t* code);

/* Self-test of the kernels' bounded waits (failure detection without a GPU
 * fault): on `device`, one warp waits through the attention kernels' own
 * mbarrier-wait routine on a barrier that nothing arrives on.  The wait gives
 * up after its time limit (2 s), so the call takes about that long.  On return
 * *err_code holds the device error word the kernel left (PST_DEVICE_WAIT_TIMEOUT
 * is expected) and *lanes_gave_up the lanes whose wait returned unfinished
 * (32 expected); the context stays usable. */
pst_status pst_selftest_bounded_wait(int device, int32_t* err_code, int32_t* lanes_gave_up);

/* Thread-local message of the last failing call on this thread ("" if none). */
const char* pst_last_error(void);

/* Library version string. */
const char* pst_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PST_H */
