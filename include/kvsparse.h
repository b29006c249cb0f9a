/*
 * kvsparse.h -- C ABI of decode-phase attention over a paged KV cache with
 * Quest-style page selection, for one GB300 (sm_103a) GPU.
 *
 * The path, per decode token and layer (KVDrive: A Holistic Multi-Tier KV
 * Cache Management System for Long-Context LLM Inference, section 2.3 "KV
 * cache offloading", steps (1)-(3); section 2.2 "Sparse attention" for the
 * Quest index):
 *   kv_page_minmax_build  -> per-page channel-wise key min/max (the index)
 *   kv_append_token       -> one new decode token per sequence into the cache,
 *                            with its page's min/max updated in place
 *   kv_page_score         -> q against the index: an upper bound on q.k
 *   (kv_page_mean_build / kv_page_score_mean: the mean-key index instead)
 *   kv_topk_select        -> the K highest-scoring pages per query head
 *                            (kv_topk_select_forced: sink and local pages first)
 *   kv_sparse_decode_attn -> softmax attention over only those pages
 *                            (kv_sparse_decode_attn_window: through a
 *                            GPU-resident window of recently critical pages)
 *   kv_dense_decode_attn  -> the same over every page (Dual-Blade, "Background
 *                            and key observations": decode reads all prior KV)
 * K/V pages live in device memory (HBM) or in pinned host memory that the GPU
 * reads in place, with no staging copy (DirectKV -- No Buffer, No Bottleneck:
 * Efficient Zero-Copy KV Cache Offloading for Long-Context LLMs, core method 1
 * "KV Cache Manager", core method 2 decode order).
 *
 * Conventions for every call:
 *  - All pointers are plain addresses.  Device arrays are device pointers; for
 *    KV_LOC_HOST_PINNED the K/V caches are host pointers from cudaHostAlloc
 *    (or cudaHostRegister) that the device can map.  Everything else is always
 *    in device memory.
 *  - The caller owns and allocates every buffer (outputs and workspaces).  The
 *    library allocates nothing, frees nothing and never synchronises, except
 *    kv_device_status, which synchronises the given stream.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls are asynchronous on it and write only their named outputs and
 *    their workspace.  Kernels are launched with programmatic dependent
 *    launch: a call's first kernel may start while the stream's previous
 *    kernel finishes, but it reads no input before griddepcontrol.wait, so a
 *    preceding kernel (of any library) that releases its dependents early and
 *    writes q, the block table or any other input afterwards is still seen
 *    complete.
 *  - Return value: KV_OK, or a negative kv_status.  Argument checks run on the
 *    host before any launch; a call that fails them launches nothing.  Checks
 *    on device-resident data (context lengths, block-table entries, selected
 *    page ids) run inside the kernels: a bad entry is skipped and recorded in a
 *    device status word that kv_device_status returns.
 *  - Alignment: q, K/V caches, minmax, scores, out and workspaces 16 bytes;
 *    int32 arrays 4 bytes.
 *
 * Shapes: B = batch, Hq = query heads, Hkv = kv heads (Hq % Hkv == 0,
 * G = Hq / Hkv), d = head_dim (128), ps = page_size (16, 32, 64 or 128), maxP =
 * max_pages_per_seq, N = num_phys_pages.  Sequence b holds context_lens[b]
 * tokens in pages 0 .. P_b - 1, P_b = ceil(context_lens[b] / ps); the last page
 * may be partial and only its first valid tokens take part anywhere.
 *
 * Layouts (row-major, innermost last):
 *   q            [B][Hq][d]          dtype
 *   k_cache      [N][Hkv][ps][d]     dtype   (v_cache the same)
 *   block_table  [B][maxP]           int32   logical page -> physical page
 *   context_lens [B]                 int32   1 <= len <= maxP * ps
 *   minmax       [N][Hkv][2][d]      dtype   [..][0][c] = min, [..][1][c] = max
 *   scores       [B][Hq][maxP]       float   -inf for p >= P_b
 *   indices      [B][Hq][k]          int32   ascending logical pages, -1 padded
 *   out          [B][Hq][d]          float
 * Query head h reads kv head h / G.
 */
#ifndef KVSPARSE_H
#define KVSPARSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { KV_F32 = 0, KV_F16 = 1, KV_BF16 = 2 } kv_dtype;
typedef enum { KV_LOC_HBM = 0, KV_LOC_HOST_PINNED = 1 } kv_location;

typedef enum {
  KV_OK = 0,
  KV_ERR_INVALID_ARG = -1,    /* null/misaligned pointer, bad shape, k < 1      */
  KV_ERR_UNSUPPORTED = -2,    /* d != 128, ps not in {16,32,64,128}, dtype,
                                 max_pages_per_seq > 524288 (attention)      */
  KV_ERR_LOCATION = -3,       /* K/V memory does not match kv_loc               */
  KV_ERR_WORKSPACE = -4,      /* workspace null or smaller than required        */
  KV_ERR_CUDA = -5,           /* a CUDA runtime call or launch failed           */
  KV_ERR_DEVICE_TIMEOUT = -6, /* a bounded device-side wait gave up             */
  KV_ERR_BOUNDS = -7          /* device data out of range (len, page id)        */
} kv_status;

typedef struct {
  int32_t batch;             /* B   >= 1                                      */
  int32_t num_q_heads;       /* Hq  >= 1                                      */
  int32_t num_kv_heads;      /* Hkv >= 1, divides Hq                          */
  int32_t head_dim;          /* d, must be 128                                */
  int32_t page_size;         /* ps, 16, 32, 64 or 128 tokens                 */
  int32_t max_pages_per_seq; /* maxP >= 1                                     */
  int64_t num_phys_pages;    /* N >= 1: pages in k_cache / v_cache / minmax   */
  int32_t dtype;             /* kv_dtype of q, K, V and minmax                */
  int32_t kv_loc;            /* kv_location of k_cache / v_cache              */
} kv_shape;

/* Index build.  For every sequence b and valid logical page p < P_b, and every
 * kv head, writes the channel-wise minimum and maximum of the page's keys
 * over its valid tokens into minmax[block_table[b][p]][kvh] (KVDrive, section
 * 2.2: Quest keeps per-block channel-wise key min and max).  Exact: the
 * outputs are elements of K, compared in IEEE totalOrder (so -0.0 < +0.0).
 * Reads k_cache from kv_loc; minmax is in device memory.  Entries of physical
 * pages no row references are not written.  A physical page shared by several
 * rows must be full in each. */
int kv_page_minmax_build(const kv_shape *shape, const void *k_cache, const int32_t *block_table,
                         const int32_t *context_lens, void *minmax, void *stream);

/* Decode append (KVDrive, section 2.1: each decode step appends the new key
 * and value vectors to the cache; DirectKV, core method 4: with the cache in
 * pinned host memory, decode appends the new token there).
 *   k_new, v_new [B][Hkv][d] dtype, device memory: the new token's K and V.
 * The token of sequence b is stored at position len_b = context_lens[b], the
 * length BEFORE the append (0 <= len_b < maxP * ps): physical page
 * block_table[b][len_b / ps], slot len_b % ps, every kv head; the bits are
 * copied unchanged.  k_cache / v_cache are written where kv_loc says (for
 * KV_LOC_HOST_PINNED, through the mapped host pointer).
 * minmax (may be NULL: no index update): the entry of that physical page
 * becomes the channel-wise min/max of its len_b % ps + 1 valid tokens, i.e.
 * min(old, k) / max(old, k) in IEEE totalOrder, or k itself when the token
 * opens the page -- bit-identical to kv_page_minmax_build on the new length.
 * Precondition: the entry holds the page's first len_b % ps tokens (from the
 * build or earlier appends), and the page is not shared with another row.
 * Calling again at the same position without advancing rewrites K/V, but the
 * min/max keeps the overwritten key too (a looser, still valid bound).
 * context_lens_out (may be NULL, may equal context_lens): receives len_b + 1.
 * A row whose len_b or block-table entry is out of range is skipped, keeps
 * its length and sets KV_ERR_BOUNDS in the device status word. */
int kv_append_token(const kv_shape *shape, const void *k_new, const void *v_new, void *k_cache,
                    void *v_cache, const int32_t *block_table, const int32_t *context_lens,
                    int32_t *context_lens_out, void *minmax, void *stream);

/* Page criticality (KVDrive, section 2.2): scores[b][h][p] =
 * sum_c max(q_c * min_c, q_c * max_c) over the minmax entry of page
 * block_table[b][p], kv head h / G -- an upper bound on q . k for every key of
 * the page.  fp32 arithmetic (the products of 16-bit inputs are exact); no
 * 1/sqrt(d) factor, since it does not change the ranking.  p >= P_b -> -inf.
 * The index rows load together with context_lens, so block-table entries
 * past P_b that hold an in-range physical page are read (never used); a
 * caller with short rows avoids those reads by setting such entries to -1. */
int kv_page_score(const kv_shape *shape, const void *q, const void *minmax,
                  const int32_t *block_table, const int32_t *context_lens, float *scores,
                  void *stream);

/* Mean-key page index (KVDrive, section 2.3: ShadowKV-style spatial chunking
 * represents a block by its mean key; section 3, Finding 2: comparing the
 * query with one mean key per block costs less than Quest's min and max; the
 * design overview: half the index bytes of the min/max pair).
 *   mean [N][Hkv][d] dtype, device memory.
 * kv_page_mean_build: for every sequence b, valid logical page p and kv head,
 * mean[block_table[b][p]][kvh][c] = (sum over the page's valid tokens of
 * K[..][t][c]) / (number of valid tokens), rounded once to dtype (nearest,
 * ties to even).  Sums run in fp32 (exact for typical 16-bit keys, whose page
 * values span few binades), the division in fp64.  Entries of unreferenced
 * pages are not written.
 * kv_page_mean_refresh: the same for the page holding each row's last token
 * only (B x Hkv entries) -- what an append changes.
 * kv_page_score_mean: scores[b][h][p] = sum_c q_c * mean_c of page
 * block_table[b][p], kv head h / G (an estimate of q . k, not a bound), fp32
 * accumulation; p >= P_b -> -inf.  Same layouts and errors as kv_page_score;
 * its output feeds kv_topk_select unchanged. */
int kv_page_mean_build(const kv_shape *shape, const void *k_cache, const int32_t *block_table,
                       const int32_t *context_lens, void *mean, void *stream);
int kv_page_mean_refresh(const kv_shape *shape, const void *k_cache, const int32_t *block_table,
                         const int32_t *context_lens, void *mean, void *stream);
int kv_page_score_mean(const kv_shape *shape, const void *q, const void *mean,
                       const int32_t *block_table, const int32_t *context_lens, float *scores,
                       void *stream);

/* Bytes of workspace kv_topk_select needs for this shape and k (may be 0). */
size_t kv_topk_workspace_bytes(const kv_shape *shape, int32_t k);

/* Top-K selection (KVDrive, section 2.2: only the Top-K blocks per query are
 * retrieved).  For each (b, h): the min(k, P_b) pages with the largest scores
 * over p < P_b, ties to the lower page index, written ascending into
 * indices[b][h][0 ..]; the remaining slots get -1.  -0.0 and +0.0 rank equal.
 * workspace may be NULL when kv_topk_workspace_bytes returns 0. */
int kv_topk_select(const kv_shape *shape, const float *scores, const int32_t *context_lens,
                   int32_t k, int32_t *indices, void *workspace, size_t workspace_bytes,
                   void *stream);

/* Top-K selection with forced pages (KVDrive, section 9.1 "Experimental
 * setup": sparse-attention systems always keep the sink tokens -- the first
 * 4 -- and the 64 most recent local tokens).  As kv_topk_select, except that
 * the pages holding tokens [0, sink_tokens) and [len_b - local_tokens, len_b)
 * are selected first; the remaining slots go to the highest-scoring other
 * pages.  Forced pages count within k: a caller that wants k dynamic pages on
 * top passes k plus the number of forced pages.  If more pages are forced
 * than k, the k lowest-index forced pages are kept.  sink_tokens = 0 and
 * local_tokens = 0 give kv_topk_select exactly.  Both must be >= 0. */
int kv_topk_select_forced(const kv_shape *shape, const float *scores,
                          const int32_t *context_lens, int32_t k, int32_t sink_tokens,
                          int32_t local_tokens, int32_t *indices, void *workspace,
                          size_t workspace_bytes, void *stream);

/* Bytes of workspace the attention calls need for this shape on the current
 * device; k = 0 for kv_dense_decode_attn, the selection size for
 * kv_sparse_decode_attn.  Split-K partial results and the per-group union of
 * selected pages live there. */
size_t kv_attn_workspace_bytes(const kv_shape *shape, int32_t k);

/* Launch plan of the attention calls on the current device: the number of
 * CTAs each (sequence, kv head, head chunk) is split over (k as for
 * kv_attn_workspace_bytes).  With more than one split, the call launches a
 * combine kernel after the attention kernel.  0 for an invalid shape. */
int32_t kv_attn_num_splits(const kv_shape *shape, int32_t k);

/* Sparse decode attention (KVDrive, section 2.3 step (3); DirectKV, core
 * method 2-3: the query and the output stay on chip and each K/V tile is read
 * once, with a streaming softmax).  For each (b, h):
 *   out[b][h] = sum_t softmax_t(scale * q . k_t) v_t
 * over the valid tokens of the pages listed in indices[b][h][0 .. k) (entries
 * < 0 skipped; ids >= P_b are a bounds error).  Pages selected by several
 * heads of one GQA group are read once.  scale is typically 1/sqrt(d). */
int kv_sparse_decode_attn(const kv_shape *shape, const void *q, const void *k_cache,
                          const void *v_cache, const int32_t *block_table,
                          const int32_t *context_lens, const int32_t *indices, int32_t k,
                          float scale, float *out, void *workspace, size_t workspace_bytes,
                          void *stream);

/* Page selection and the attention's page lists in one call: the result of
 * kv_page_score followed by kv_topk_select_forced (sink_tokens = local_tokens
 * = 0: plain kv_topk_select) -- the same indices[b][h][0 .. k) -- without the
 * scores passing through memory (KVDrive, section 2.3 steps (1)-(2): the
 * selection reads only the GPU-resident index; section 3, finding 2: the
 * selection is a large share of decode time).  For 16-bit data with G = 4 or
 * 8 it is one launch: a cluster of G CTAs per (sequence, kv head), each
 * scoring 1/G of the pages for the whole group, keeping every head's scores
 * on chip, selecting one head's pages and building the group's union of
 * selected pages; other shapes run the separate kernels.  The union lists
 * stay in `workspace` for kv_sparse_decode_attn_selected, which must follow
 * on the same stream with the same shape, k, block_table, context_lens and
 * workspace (the lists hold physical pages).  The workspace must hold
 * kv_select_workspace_bytes(shape, k) bytes (at least
 * kv_attn_workspace_bytes(shape, k)).  Errors as kv_page_score and
 * kv_topk_select_forced, and KV_ERR_WORKSPACE. */
size_t kv_select_workspace_bytes(const kv_shape *shape, int32_t k);
int kv_select_pages(const kv_shape *shape, const void *q, const void *minmax,
                    const int32_t *block_table, const int32_t *context_lens, int32_t k,
                    int32_t sink_tokens, int32_t local_tokens, int32_t *indices,
                    void *workspace, size_t workspace_bytes, void *stream);

/* Sparse decode attention over the pages the preceding kv_select_pages call
 * chose: the out of kv_sparse_decode_attn with that call's indices.  It is
 * the same bit for bit when each (sequence, kv head) group's list is split
 * over the group's own CTAs; where a CTA's share can take 100 us or more to
 * stream (long shares, e.g. 64-token pages over 64k tokens), the kernel may
 * instead cut all groups' lists into equal chunks, chosen per call from the
 * lists' lengths (a batch of rows of different lengths), and then the result
 * differs only in the order of the floating-point merge (kv_debug_split_mode
 * fixes the choice).  The workspace is the one kv_select_pages filled,
 * unchanged since. */
int kv_sparse_decode_attn_selected(const kv_shape *shape, const void *q, const void *k_cache,
                                   const void *v_cache, const int32_t *block_table,
                                   const int32_t *context_lens, int32_t k, float scale,
                                   float *out, void *workspace, size_t workspace_bytes,
                                   void *stream);

/* Dense decode attention: as kv_sparse_decode_attn over every page p < P_b
 * (Dual-Blade, "Background and key observations"). */
int kv_dense_decode_attn(const kv_shape *shape, const void *q, const void *k_cache,
                         const void *v_cache, const int32_t *block_table,
                         const int32_t *context_lens, float scale, float *out, void *workspace,
                         size_t workspace_bytes, void *stream);

/* Dense decode attention for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a convenience of this library.
 * Callers such as a plugin that a host framework hands only its input and
 * output buffers, or a latency-critical loop where cudaMalloc would
 * synchronise the device, have no workspace to pass.  This call computes
 * exactly what kv_dense_decode_attn computes, with the split-K partials kept
 * in a fixed 1 MiB scratch array inside the library's device image, which
 * every GPU that loads the library holds until the process exits.  It
 * allocates nothing and calls no allocating routine.
 *  - Limit: shapes whose partials need more than 1 MiB (see
 *    kv_attn_workspace_bytes(shape, 0)) are refused with KV_ERR_WORKSPACE
 *    before anything is launched; use kv_dense_decode_attn for them.
 *  - The first call on each device looks up the scratch array's device
 *    address (cudaGetSymbolAddress) with that device current; make that first
 *    call before any stream capture.
 *  - All calls on a device share the one array, which keeps the last call's
 *    contents; nothing in it needs to start at zero.  Calls that overlap on
 *    the GPU (concurrent streams, or several host threads) race on it.
 * Other arguments and return codes as kv_dense_decode_attn. */
int kv_dense_decode_attn_noalloc(const kv_shape *shape, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_table,
                                 const int32_t *context_lens, float scale, float *out,
                                 void *stream);

/* Streaming-read bandwidth probe (DirectKV, observation 4: host-resident
 * long-context attention is bound by the link's sustained bandwidth; this
 * measures that bandwidth).  Reads `bytes` (a multiple of 16) from `src` --
 * device memory, or pinned host memory read in place through its device
 * mapping -- with 16-byte loads from every SM, and writes one XOR word per
 * thread block into `sink` (device memory, sink_words >= 1 words; up to 4
 * blocks per SM are used).  Time it with events on `stream`. */
int kv_stream_read_probe(const void *src, size_t bytes, unsigned long long *sink,
                         int32_t sink_words, void *stream);

/* The same probe with its launch shape given: `blocks` thread blocks (sink
 * holds `blocks` words) of `threads` threads (128, 256, 512 or 1024), each
 * thread keeping `loads_in_flight` 16-byte loads in flight (4, 8 or 16).
 * For sweeping the shape that reads a buffer fastest.  KV_ERR_INVALID_ARG
 * for any other shape. */
int kv_stream_read_probe_shape(const void *src, size_t bytes, unsigned long long *sink,
                               int32_t blocks, int32_t threads, int32_t loads_in_flight,
                               void *stream);

/* One decode step of one layer on host buffers: q and context_lens come from
 * host memory, the path runs (k > 0: kv_select_pages and
 * kv_sparse_decode_attn_selected when workspace_bytes >=
 * kv_select_workspace_bytes(shape, k), else kv_page_score into `scores`,
 * kv_topk_select, kv_sparse_decode_attn; k == 0: kv_dense_decode_attn) and
 * out lands in host memory, all asynchronous on `stream`.  A host buffer the device has mapped
 * (cudaHostAlloc, or pinned and registered) is accessed across the host
 * link, the zero-copy access DirectKV applies to K/V (core method 1): out is
 * written in place; for a sparse step (k > 0), mapped q and lengths are read
 * once by a staging kernel into the device buffers q and context_lens when
 * those are given, else (and for a dense step) the kernels read them in
 * place.  Any other host buffer is copied through the matching device buffer
 * with cudaMemcpyAsync (q, context_lens, out may be NULL only for mapped
 * buffers).  The same outputs as those calls (kv_sparse_decode_attn_selected
 * says when its merge order may differ from kv_sparse_decode_attn's).  The
 * index (minmax) must be built. */
typedef struct {
  const void *q_host;               /* [B][Hq][d] dtype, host                  */
  const int32_t *context_lens_host; /* [B], host                               */
  float *out_host;                  /* [B][Hq][d], host                        */
  void *q;                          /* device copies of the three              */
  int32_t *context_lens;
  float *out;
  const void *k_cache;              /* where kv_loc says                       */
  const void *v_cache;
  const int32_t *block_table;       /* device                                  */
  const void *minmax;               /* device; sparse steps only               */
  float *scores;                    /* device [B][Hq][maxP]; sparse steps that */
                                    /* run the separate calls only (may be NULL */
                                    /* when the workspace holds the selection)  */
  int32_t *indices;                 /* device [B][Hq][k]; sparse only          */
  int32_t k;                        /* 0: dense step; else pages per head      */
  float scale;
  void *workspace;                  /* >= kv_attn_workspace_bytes(shape, k)   */
  size_t workspace_bytes;
} kv_step_io;

int kv_decode_step(const kv_shape *shape, const kv_step_io *io, void *stream);

/* GPU-resident window of critical pages (KVDrive, section 5.1 "Sliding
 * window with lookahead eviction"; section 3, Finding 1: a window of several
 * steps' critical entries cuts host-to-GPU transfer; section 6.3: with most
 * critical entries served from GPU memory, attention stays on the GPU).
 *
 * The window has one group per (sequence b, kv head) with C = cache_pages
 * slots; slot s of group (b, kvh) holds one page of that kv head at
 *   cache_k / cache_v [B * C][Hkv][ps][d] dtype, device memory,
 * page index b * C + s.  State (device memory, owned by the caller):
 *   slot_page [B][Hkv][C]     logical page in the slot, -1 = free
 *   page_slot [B][Hkv][maxP]  slot of a logical page, -1 = not cached
 *   stats     [B][Hkv][4]     (may be NULL) of the last call: pages needed,
 *                             hits, pages fetched, pages evicted.
 * kv_window_reset empties the window (both maps to -1). */
typedef struct {
  int32_t cache_pages; /* C >= min(G * k, maxP); maxP + 8 C <= 200 KiB */
  int32_t reserved;
  void *cache_k;
  void *cache_v;
  int32_t *slot_page;
  int32_t *page_slot;
  int32_t *stats;
} kv_window;

/* Workspace for kv_sparse_decode_attn_window with this shape, k and C. */
size_t kv_window_workspace_bytes(const kv_shape *shape, int32_t k, int32_t cache_pages);

int kv_window_reset(const kv_shape *shape, const kv_window *win, void *stream);

/* One decode step of sparse attention through the window.  Inputs as
 * kv_sparse_decode_attn (k_cache / v_cache where kv_loc says, typically
 * pinned host memory), plus this step's page scores [B][Hq][maxP] (the
 * kv_page_score output the indices were selected from).  Per group:
 *   need    = pages any of the G query heads selected;
 *   hits    = needed pages already in the window, misses = the rest;
 *   evict   = as many non-needed cached pages as the misses need slots,
 *             lowest score first (score = max over the G heads this step;
 *             pages at or past the row's end first; ties to the lower slot);
 *   assign  = misses in ascending page order take the free slots in
 *             ascending slot order;
 *   fetch   = the misses, and the row's last page when it is a hit (tokens
 *             may have been appended since it was copied);
 * then attention runs exactly as kv_sparse_decode_attn -- same out -- reading
 * the hits from the window (HBM) and the fetched pages from k_cache /
 * v_cache, whose valid tokens it also stores into their window slots.  When
 * G exceeds the heads one attention CTA covers (G > 8; G > 4 for fp32), a
 * page several head chunks need is read from k_cache once per chunk.
 * C must hold every needed page: C >= min(G * k, maxP), else
 * KV_ERR_INVALID_ARG.  cache_k / cache_v must be device memory
 * (KV_ERR_LOCATION).  The workspace must hold kv_window_workspace_bytes.
 * The window state marks a fetched page as cached before the attention has
 * stored it into its slot: after a call whose device status reports an error
 * (kv_device_status), reset the window (kv_window_reset) before the next. */
int kv_sparse_decode_attn_window(const kv_shape *shape, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_table,
                                 const int32_t *context_lens, const int32_t *indices, int32_t k,
                                 const float *scores, float scale, float *out,
                                 const kv_window *win, void *workspace, size_t workspace_bytes,
                                 void *stream);

/* Synchronises `stream`, then returns and clears the device status word of
 * the current device: KV_OK, KV_ERR_DEVICE_TIMEOUT or KV_ERR_BOUNDS (the
 * first error recorded since the last call), or KV_ERR_CUDA if the
 * synchronisation itself failed. */
int kv_device_status(void *stream);

/* Static, NUL-terminated name of a kv_status value. */
const char *kv_status_string(int status);

/* Testing hook for the bounded device-side waits (failure detection without
 * a GPU fault).  wait_limit_ns (1 ns .. 60 s; default 2 s) bounds every
 * pipeline wait of the attention kernels; skip_page >= 0 makes the producer
 * of every attention CTA leave its skip_page-th 16-token K/V tile unfilled, so
 * the consumer waiting for it gives up after the limit, the call's kernels finish, and
 * kv_device_status reports KV_ERR_DEVICE_TIMEOUT.  skip_page < 0 restores
 * normal operation.  Process-wide; not for concurrent use with other calls.
 * Returns KV_OK or KV_ERR_INVALID_ARG. */
int kv_debug_config(int32_t skip_page, uint64_t wait_limit_ns);

/* Testing hook for the attention over kv_select_pages' lists
 * (kv_sparse_decode_attn_selected and kv_decode_step).  Its CTAs either split
 * each (sequence, kv head) group's union list over the group's own splits, or
 * cut the lists of all groups, laid end to end, into one equal chunk per CTA
 * (possible when every group holds at least a chunk; a CTA then covers the
 * tail of one group and the head of the next at most, and the combine merges
 * the pieces).  The two give the same result up to the order of the
 * floating-point merge.  The shapes must allow equal chunks at all: 16-bit
 * data, 4 or 8 query heads per kv head, more than one split, at most 4096
 * groups.
 *   mode -1 (default): where a CTA's share of a group's list can take 100 us
 *     or more to stream, the kernel chooses per call from the groups' list
 *     lengths (equal chunks when the per-group split's longest CTA would
 *     stream more K/V than an equal chunk for longer than about 2.5 us);
 *     elsewhere the split per group, with no cost for the choice;
 *   0: always the split per group;
 *   1: equal chunks whenever possible;
 *   2: the kernel chooses, as in -1, for every call the shapes allow.
 * Process-wide; not for concurrent use with other calls.  Returns KV_OK or
 * KV_ERR_INVALID_ARG. */
int kv_debug_split_mode(int32_t mode);

#ifdef __cplusplus
}
#endif

#endif /* KVSPARSE_H */
