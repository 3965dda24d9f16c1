/*
 * spd.h -- C ABI of the GB300 sparse paged decode attention library.
 *
 * Decode-phase unified sparse attention over a hierarchically paged KV cache,
 * after "LServe long-sequence LLM serving system" (the LServe write-up):
 *
 *   section 2.1  static sparsity: a fixed share of kv heads become streaming
 *                heads that see only local context; dynamic sparsity: the
 *                other heads keep a fixed KV token budget (default 4096),
 *                chosen per query from min-max pooled key features;
 *   section 2.2  hierarchical paging: large physical pages (256-1024 tokens)
 *                are the allocation unit, small logical pages (16-64 tokens)
 *                are the selection unit, a page table maps between them;
 *   section 3.2  the page selector runs once every C (= 4) decode steps and
 *                is reused in between; the budget follows
 *                min(4096, sequence length / 32); streaming heads read recent
 *                tokens through on-chip memory.
 *
 * Everything below the ABI is hand-written CUDA for sm_103a plus a C++ host
 * runtime (page pool, per-sequence tables, work partitioning).  No type from
 * PyTorch or any other framework appears here.
 *
 * Conventions
 *   - Every function returns spd_status; nothing throws across the ABI.
 *   - Pointers documented as "device" must point to memory of the GPU the
 *     context runs on and be 16-byte aligned; "host" pointers are read
 *     during the call only.
 *   - All GPU work is enqueued on the `stream` argument (a cudaStream_t;
 *     NULL means the legacy default stream).  Host-side state (lengths, step
 *     counters, page tables) advances when the call returns, before the GPU
 *     has run the work, so calls on one context must be issued in decode
 *     order on one stream.  A context is not thread-safe.
 *   - Argument errors are detected on the host before anything is enqueued
 *     and leave the context unchanged.
 *   - Kernels are launched with programmatic dependent launch: each waits
 *     for the preceding kernel on the stream before touching global memory
 *     and only then lets the next kernel start (see
 *     spd_set_early_kv_staging for the one exception).
 */
#ifndef SPD_H
#define SPD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct spd_ctx spd_ctx;
typedef struct CUstream_st *spd_stream; /* same type as cudaStream_t */

typedef enum {
  SPD_OK = 0,
  SPD_ERR_INVALID_ARG = 1,  /* bad argument or configuration               */
  SPD_ERR_NO_PAGES = 2,     /* physical page pool exhausted                 */
  SPD_ERR_BAD_SEQ = 3,      /* unknown, freed or duplicated sequence id     */
  SPD_ERR_CAPACITY = 4,     /* beyond max_context / max_seqs / budget room  */
  SPD_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed         */
  SPD_ERR_DEVICE_CHECK = 6, /* a kernel's own bounds check tripped          */
  SPD_ERR_STATE = 7         /* call out of order (e.g. no selection yet)    */
} spd_status;

typedef enum { SPD_F16 = 0, SPD_BF16 = 1 } spd_dtype;

/*
 * Configuration of one attention layer's KV cache.  Keys follow the
 * `sparse_config` block of the LServe write-up, section 5.2
 * (dynamic_token_budget, reuse_interval, physical_page_size,
 * logical_page_size; the streaming share becomes an explicit per-head mask).
 */
typedef struct {
  int num_q_heads;   /* Hq; Hq % Hkv == 0 and Hq / Hkv in {1, 2, 4, 8}      */
  int num_kv_heads;  /* Hkv, 1..128                                          */
  int head_dim;      /* d in {64, 128}                                       */
  spd_dtype dtype;   /* storage type of q, K, V and the min/max metadata     */
  int logical_page;  /* l in {16, 32, 64}: selection unit, tokens           */
  int physical_page; /* P, a multiple of l, <= 4096: allocation unit       */
  int num_physical_pages; /* pool size (shared by all sequences)            */
  int max_seqs;           /* live sequences at once                         */
  int max_context;        /* tokens per sequence                            */
  const unsigned char *kv_head_is_streaming; /* host [Hkv], copied; NULL=none */
  int sink;          /* streaming heads: attention-sink tokens S >= 0        */
  int window;        /* streaming heads: local window W >= 1 (incl. newest)  */
  int token_budget;  /* dynamic heads: tokens kept; <= 0: min(4096, L/32)    */
  int reuse_interval;/* C >= 1: selection runs when step % C == 0            */
  unsigned long long free_list_seed; /* 0: pages handed out in order;
                                        else a seeded permutation of the pool */
  /* fp8 KV storage (the LServe write-up's sparse_config, section 5.2, names
   * an fp8 KV cache).  kv_fp8 = 1: keys, values and the key min/max metadata
   * are stored as OCP fp8 E4M3 codes of value / scale -- each 16-bit input
   * divided once in fp32, rounded to nearest even, saturated at +-448 --
   * with one scale per kv head for keys and one for values (host [Hkv]
   * positive finite fp32, copied at spd_create; NULL: all 1).  q and the
   * K/V handed to the append calls stay `dtype`; page scores and attention
   * read the stored values code * scale.  Needs head_dim 128.  kv_fp8 = 0
   * (a zero-initialised config) keeps 16-bit storage and ignores the scales. */
  int kv_fp8;
  const float *k_scale;
  const float *v_scale;
} spd_config;

/*
 * Bytes of every device buffer the caller must provide.  Layouts (elements
 * of `dtype` unless noted -- one-byte E4M3 codes for k_pool, v_pool, meta,
 * stream_k and stream_v when kv_fp8 is set; Hd / Hs = number of dynamic /
 * streaming kv heads,
 * R = P / l, MP = ceil(max_context / P), KS = pages kept at the largest
 * budget):
 *   k_pool, v_pool [num_physical_pages][Hd][P][d]   keys / values of dynamic
 *                   heads; logical page j of a sequence lives in physical
 *                   page table[j / R], rows (j % R) * l ... + l - 1.
 *   meta           [num_physical_pages][Hd][R][2][d]  per logical page the
 *                   channel-wise key minimum ([..][0][:]) and maximum.
 *   stream_k, stream_v [max_seqs][Hs][S + W][d]  streaming heads: slots
 *                   0..S-1 hold positions 0..S-1, slot S + ((t - S) mod W)
 *                   holds position t >= S (a ring, never shifted).
 *   page_table     int32 [max_seqs][MP]   physical page of each sequence's
 *                   i-th P-token block (mirrors the host table).
 *   selection      int32 [max_seqs][Hd][KS]  kept logical pages, ascending.
 *   scratch        split partials, tickets, page scores and the device error
 *                   word; contents need no initialisation.
 * Every buffer must be 256-byte aligned.  Sizes of 0 mean "not used".
 */
typedef struct {
  size_t k_pool, v_pool, meta, stream_k, stream_v, page_table, selection,
      scratch;
} spd_sizes;

typedef struct {
  void *k_pool, *v_pool, *meta, *stream_k, *stream_v, *page_table, *selection,
      *scratch;
} spd_buffers;

/* Validate a configuration and report the buffer sizes it needs.  Host only.
 * SPD_ERR_INVALID_ARG on a bad configuration. */
spd_status spd_query_sizes(const spd_config *cfg, spd_sizes *out);

/*
 * Create a context over caller-owned device buffers (sizes from
 * spd_query_sizes).  The library never allocates or frees device memory for
 * the caller's data; it owns only host tables.  Host only: no GPU work is
 * enqueued and the buffers are not touched until the first append.
 */
spd_status spd_create(const spd_config *cfg, const spd_buffers *bufs,
                      spd_ctx **out);
void spd_destroy(spd_ctx *ctx);

/*
 * Page-table allocation and release (LServe write-up, section 2.2: the page
 * table maps logical pages onto larger physical pages; survey "Long-context
 * inference optimization for LLMs", section 3.4: a fixed pool with a free
 * list that reports exhaustion).  Host only.
 *   spd_seq_create  picks a free sequence slot; id in [0, max_seqs).
 *                   SPD_ERR_CAPACITY when max_seqs are live.
 *   spd_seq_free    returns the sequence's physical pages to the free list
 *                   and clears its length, step counter and selection.
 *   spd_seq_reserve makes sure physical pages exist for the next n_tokens
 *                   positions.  All or nothing: SPD_ERR_NO_PAGES (pool
 *                   exhausted) or SPD_ERR_CAPACITY (beyond max_context)
 *                   leave the pool and the sequence unchanged.  The device
 *                   page table is updated by the next spd_kv_append.
 *   spd_seq_info    length L, decode-step counter, page count at the last
 *                   selection (0 if none) and pages kept at it.
 *   spd_get_page_table copies the sequence's physical page ids (host table)
 *                   to phys_host (capacity cap entries), count to *n_host.
 */
spd_status spd_seq_create(spd_ctx *ctx, int *seq_id_out);
spd_status spd_seq_free(spd_ctx *ctx, int seq_id);
spd_status spd_seq_reserve(spd_ctx *ctx, int seq_id, int n_tokens);
spd_status spd_seq_info(spd_ctx *ctx, int seq_id, long long *length,
                        long long *step_counter, int *pages_at_selection,
                        int *pages_kept);
spd_status spd_get_page_table(spd_ctx *ctx, int seq_id, int *phys_host,
                              int cap, int *n_host);
/* Free physical pages left in the pool. */
spd_status spd_free_pages(spd_ctx *ctx, int *n_free);

/*
 * Append n_tokens key/value rows to each listed sequence and update the
 * min/max metadata of every logical page they touch (LServe write-up,
 * section 2.1: min-max pooling of each block's keys).
 *   seq_ids  host [n_seqs], distinct live sequences.
 *   k, v     device [n_seqs][n_tokens][Hkv][d] of dtype.
 * Dynamic heads go to the paged pool (pages allocated as needed, all or
 * nothing across the call: SPD_ERR_NO_PAGES / SPD_ERR_CAPACITY change
 * nothing); streaming heads go to their sink slots and ring window.
 * Metadata is exact (a min/max of stored values, no rounding).
 */
spd_status spd_kv_append(spd_ctx *ctx, const int *seq_ids, int n_seqs,
                         int n_tokens, const void *k, const void *v,
                         spd_stream stream);

/*
 * Query-aware page selection for the dynamic heads (LServe write-up,
 * section 2.1 dynamic sparsity; section 3.2 reusable selector and dynamic
 * budget).  For each listed sequence whose step counter is a multiple of C
 * (or every listed sequence if `force`):
 *   score  S(j) = max over the G query heads h of the kv head of
 *          sum_c max(q_h[c] * kmax_j[c], q_h[c] * kmin_j[c])   (fp32),
 *   keep   K_sel = max(1, budget / l) pages: the page holding the newest
 *          token plus the K_sel - 1 best other pages, ties to the lower
 *          page index; every page if there are at most K_sel.
 * Other sequences keep their stored selection untouched.
 *   q  device [n_seqs][Hq][d] of dtype.
 * SPD_ERR_STATE for a sequence with no tokens.
 */
spd_status spd_select_pages(spd_ctx *ctx, const void *q, const int *seq_ids,
                            int n_seqs, int force, spd_stream stream);

/*
 * Sparse decode attention (LServe write-up, section 2.1 unified sparse
 * kernel; split-K with exported row max and sum, Novita KV-sparsity article,
 * "attention mechanism modifications").  For query head h of kv head
 * g = h / G and the attended positions T of g:
 *   dynamic   T = tokens of (stored selection U pages created since it)
 *   streaming T = {t < S} U {t >= L - W}
 *   out[h] = sum_{t in T} softmax_t(q_h . k_t / sqrt(d)) v_t      (fp32).
 * Advances every listed sequence's decode-step counter by one.
 *   q    device [n_seqs][Hq][d] of dtype;  out device [n_seqs][Hq][d] fp32.
 * SPD_ERR_STATE if a sequence with dynamic heads has never been selected
 * or has no tokens.
 */
spd_status spd_sparse_decode_attention(spd_ctx *ctx, const void *q,
                                       const int *seq_ids, int n_seqs,
                                       float *out, spd_stream stream);

/*
 * Sparse decode attention without any device allocation by the caller or
 * the library for its temporaries.  No counterpart in the paper: this entry
 * point exists for callers that cannot allocate device memory when they run
 * attention -- code running while a CUDA stream is being captured (device
 * allocation is not allowed there), integrations whose device memory plan is
 * fixed at start-up, and plugins inside a host framework that owns every
 * device allocation.  It computes exactly what spd_sparse_decode_attention
 * computes (same arguments, same step-counter advance), but the split
 * partials and tickets of the fused combine live in a library-owned
 * file-scope device array of 4,292,608 bytes, held on every GPU that loads
 * the library until the process exits, instead of the context's scratch.
 * Limits: the array holds the partials of 1024 split items per launch.  The
 * library cuts each (sequence, kv head) into items of at most 256 tiles of 16
 * attended rows (4,096 tokens), in whole thread-block clusters of up to 16
 * items, and normally plans about one item per SM per launch; a batch that
 * needs more items is spread over several launches, and a single sequence
 * whose items alone exceed 1024 (for example 33 kv heads each attending
 * 131,072 tokens) makes the call fail with SPD_ERR_CAPACITY.  Every launch
 * is planned before anything is enqueued, so a refused call writes nothing
 * and advances no step counter.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress with that device
 * current, then the caller's current device is restored); make it before any
 * stream capture.  All calls share the array
 * and it keeps the last call's contents: tickets are cleared at each call,
 * and calls whose GPU work overlaps (other streams, other contexts) race --
 * issue them in order on one stream.  It calls no cudaMalloc, cudaFree or
 * allocating library routine.
 */
spd_status spd_sparse_decode_attention_static(spd_ctx *ctx, const void *q,
                                              const int *seq_ids, int n_seqs,
                                              float *out, spd_stream stream);

/*
 * Sparse decode attention that also exports the per-head softmax statistics
 * (the row max and row sum a split FlashAttention exports, Novita
 * KV-sparsity article, "attention mechanism modifications").  Same outputs
 * and step-counter effect as spd_sparse_decode_attention, plus, for every
 * listed sequence and query head h with logits z_t = q_h . k_t / sqrt(d)
 * over its attended positions T:
 *   row_max[h] = max_{t in T} z_t            (natural units)
 *   row_sum[h] = sum_{t in T} exp(z_t - row_max[h])
 * so that log(row_sum) + row_max is the log-sum-exp of the logits.
 *   row_max, row_sum  device [n_seqs][Hq] fp32, 4-byte aligned (caller-owned).
 * Errors as spd_sparse_decode_attention; SPD_ERR_INVALID_ARG for a null or
 * misaligned statistics pointer.
 */
spd_status spd_sparse_decode_attention_stats(spd_ctx *ctx, const void *q,
                                             const int *seq_ids, int n_seqs,
                                             float *out, float *row_max,
                                             float *row_sum, spd_stream stream);

/*
 * Sparse decode attention that also exports, per dynamic kv head, the share
 * of each query head's softmax weight that falls on each attended logical
 * page -- the per-page attention mass that completes the statistics of the
 * Novita KV-sparsity article's modified FlashAttention ("attention mechanism
 * modifications"; an eviction-style importance score, and a recall
 * diagnostic for the page selection).  Same outputs and step-counter effect
 * as spd_sparse_decode_attention (and as spd_sparse_decode_attention_stats
 * when row_max / row_sum are given), plus, for sequence b, dynamic kv head
 * index hd (kv heads that are not streaming, in increasing order), query
 * head g of its group and attended page index a:
 *   pages[b][hd][a]        the a-th attended logical page, ascending: the
 *                          stored selection, then every page created since
 *                          it was taken; -1 for a >= the attended count;
 *   page_mass[b][hd][g][a] sum over that page's attended tokens t of
 *                          exp(z_t - m) / sum_{t' in T} exp(z_t' - m), z_t =
 *                          q . k_t / sqrt(d); 0 for a >= the attended count.
 * The masses of one query head sum to 1.
 *   row_max, row_sum  device [n_seqs][Hq] fp32, or both NULL.
 *   pages      device int32 [n_seqs][Hd][max_pages] (caller-owned).
 *   page_mass  device fp32 [n_seqs][Hd][G][max_pages] (caller-owned).
 *   max_pages  capacity per (sequence, dynamic head), >= 1.
 * Pointers 4-byte aligned; with no dynamic head, pages and page_mass are not
 * touched and may be NULL.  SPD_ERR_CAPACITY (nothing enqueued) when a
 * sequence attends more than max_pages pages per dynamic head, or more than
 * the library's per-head limit: the pages a selection keeps plus 64 created
 * since it was taken.  The per-tile partial sums live in the context's
 * scratch, so calls on one context must not overlap on different streams.
 */
spd_status spd_sparse_decode_attention_page_mass(spd_ctx *ctx, const void *q,
                                                 const int *seq_ids, int n_seqs,
                                                 float *out, float *row_max,
                                                 float *row_sum, int *pages,
                                                 float *page_mass, int max_pages,
                                                 spd_stream stream);

/*
 * One decode step for each listed sequence: append one token (k, v device
 * [n_seqs][Hkv][d]), select if due, attend.  Same results as calling the
 * three entry points above in that order; enqueues fewer launches.
 */
spd_status spd_decode_step(spd_ctx *ctx, const void *q, const void *k,
                           const void *v, const int *seq_ids, int n_seqs,
                           float *out, spd_stream stream);

/* Introspection for tests.  spd_get_selection synchronises `stream` and
 * copies the kept pages of (seq, kv head) to idx_host (capacity cap). */
spd_status spd_get_selection(spd_ctx *ctx, int seq_id, int kv_head,
                             int *idx_host, int cap, int *count_host,
                             spd_stream stream);

/* Synchronise `stream` and read the device error word: SPD_OK, or
 * SPD_ERR_DEVICE_CHECK if a kernel's bounds check tripped (the word is then
 * cleared), or SPD_ERR_CUDA. */
spd_status spd_check_status(spd_ctx *ctx, spd_stream stream);

const char *spd_status_string(spd_status s);
/*
 * Early KV staging (off by default).  When on, a decode or selection kernel
 * of this context whose preceding kernel on the stream was not enqueued by
 * this context starts loading KV-cache data (page table, selection, K/V
 * tiles, page metadata) before that kernel has finished; q, the new token and
 * all writes still wait for it.  This overlaps the HBM reads with the tail of
 * the kernel before it -- in a model, the projection that produces q.  The
 * streaming heads of a decode kernel also start early when the kernel before
 * it is this context's own selection or page-table flush: neither writes the
 * streaming buffers, and q and the new token are final by then (that kernel
 * waited for its own predecessor), so they run without waiting at all.
 * Turn it on only if (a) nothing but this library's calls on this context
 * writes its KV-cache buffers, and (b) other code's kernels on the stream do
 * not release their dependents (programmatic dependent launch) before they
 * have waited for their own predecessor.  All of this library's kernels
 * meet (b).  SPD_ERR_INVALID_ARG for a NULL context.
 */
spd_status spd_set_early_kv_staging(spd_ctx *ctx, int enable);

/* Number of kernels this context has enqueued since it was created. */
spd_status spd_launch_count(spd_ctx *ctx, long long *n);
/* Human-readable detail of the last error on this context ("" if none). */
const char *spd_last_error(spd_ctx *ctx);

/* ---- prefill: block-sparse attention of a prompt ------------------------ */
/*
 * The phase before decode ("LServe long-sequence LLM serving system",
 * section 3.1): every text block's importance to every query block is
 * estimated with low-rank projections, Score(Q, K_i) ~ (Q W_q)(K_i W_k)^T /
 * sqrt(d), and exact attention runs only on the most important blocks;
 * prompts shorter than a threshold (32K in the write-up) fall back to dense
 * attention.  Readings fixed here (the write-up gives none of them): blocks
 * of `block` tokens; the score of a (query block b, key block i <= b) pair
 * is the mean of the low-rank logits over the pair's tokens, and a kv head's
 * the maximum over its query heads; query block b attends its own block and
 * the best earlier blocks (ties to the lower block), token_budget / block
 * blocks in all, or every block 0..b when the prompt is shorter than
 * dense_below; within them, causal softmax attention (key t' <= query t)
 * with scale 1 / sqrt(head_dim).  No paged cache is involved: K and V are
 * the prompt's own rows (spd_kv_append stores them in a context).
 */
typedef struct {
  int num_q_heads, num_kv_heads, head_dim; /* as spd_config: Hq % Hkv == 0,
                                               Hq / Hkv in {1,2,4,8}, d in {64,128} */
  spd_dtype dtype;                         /* of q, k and v                     */
  int rank;          /* r: columns of W_q and W_k, 1..64 (d / 8 in the write-up) */
  int block;         /* tokens per block; 64 is the size built                  */
  int token_budget;  /* key tokens a query block keeps (>= block)                */
  int dense_below;   /* prompts shorter than this attend every causal block     */
} spd_prefill_config;

/*
 * Sizes for a prompt of seq_len tokens: KB, the length of each query block's
 * list in `blocks` (nb = ceil(seq_len / block) when dense, else
 * min(nb, token_budget / block)), and the workspace bytes.  Host only.
 * SPD_ERR_INVALID_ARG on a bad configuration or seq_len < 1;
 * SPD_ERR_CAPACITY beyond 8192 blocks.
 */
spd_status spd_prefill_sizes(const spd_prefill_config *cfg, int seq_len,
                             int *blocks_per_query_block, size_t *workspace_bytes);

/*
 * Block-sparse causal attention of one prompt, enqueued on `stream` (three
 * kernels: block means, block selection, attention).
 *   q          device [seq_len][Hq][d] of dtype, 16-byte aligned.
 *   k, v       device [seq_len][Hkv][d] of dtype, 16-byte aligned.
 *   w_q, w_k   device fp32 [Hkv][d][rank]: the low-rank projections of each
 *              kv head (its query heads share w_q).
 *   out        device fp32 [seq_len][Hq][d].
 *   blocks     device int32 [Hkv][nb][KB] or NULL: the key blocks each query
 *              block attended, ascending, -1 after the last.
 *   workspace  device, 256-byte aligned, at least the spd_prefill_sizes bytes
 *              (owned by the caller; holds the block means, the lists and a
 *              device error word; one call at a time per workspace).
 * SPD_ERR_INVALID_ARG / SPD_ERR_CAPACITY on bad arguments (nothing
 * enqueued); SPD_ERR_CUDA if a launch fails.
 */
spd_status spd_prefill_block_sparse_attention(const spd_prefill_config *cfg, int seq_len,
                                              const void *q, const void *k, const void *v,
                                              const float *w_q, const float *w_k, float *out,
                                              int *blocks, void *workspace,
                                              size_t workspace_bytes, spd_stream stream);

/* Waits for `stream` and reads the workspace's device error word:
 * SPD_ERR_DEVICE_CHECK if a kernel's own check tripped, else SPD_OK. */
spd_status spd_prefill_check(const void *workspace, spd_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* SPD_H */
