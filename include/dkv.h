/*
 * dkv.h -- libdkv: differentiated KV-cache compaction on one GB300 (sm_103a).
 *
 * Method: "DiffKV: Differentiated Memory Management for Large Language Models
 * with Parallel KV Compaction" (arXiv 2412.03131), as summarised on its Pith
 * review page.  For every (layer, request, KV head) -- a "unit" -- the library
 *   1. scores each token by the average attention it has received from later
 *      tokens, max-aggregated over the GQA query heads of the KV head
 *      ("What carries the argument"; Referee Report, major comment 2 on
 *      Section 4 / Algorithm 1);
 *   2. classifies it against alpha_h/N and alpha_l/N into K8V4 (keys 8-bit,
 *      values 4-bit), K4V2 or pruned ("Core claim");
 *   3. hands every unit a disjoint contiguous run of page ids from a circular
 *      free page list through a parallel prefix sum over the units' page
 *      demands, and fills the bidirectional page table ("What carries the
 *      argument"; abstract: "on-GPU memory manager that compacts fragmented
 *      free memory list into contiguous regions in parallel");
 *   4. quantises the surviving tokens per token (asymmetric min/max over the
 *      128 channels of a head, fp16 scale and zero, fp32 round-half-to-even)
 *      and packs them into unified pages ("Core claim": unified pages).
 *
 * Conventions shared by every call
 *   - Every data pointer is a DEVICE pointer, allocated and owned by the
 *     caller.  The library allocates no device memory; dkv_compact takes a
 *     caller-provided workspace sized by dkv_workspace_size.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream unless stated.
 *   - Return value: DKV_OK or a negative code.  A *synchronous* error (bad
 *     argument: DKV_E_INVAL; a CUDA launch failure: DKV_E_CUDA) means nothing
 *     was enqueued.  Conditions found on the device (DKV_E_NOMEM,
 *     DKV_E_RANGE, DKV_E_TIMEOUT, DKV_E_LENS, DKV_E_INTERNAL) are recorded in
 *     the pool's device status word and read with dkv_get_status.  A call
 *     that ends in a device-side error changes neither the cursors, nor the
 *     forward and reverse tables, nor any live page: it is all-or-nothing
 *     (pages that were free may have been scribbled and stay free).
 *   - Calls on one pool must be ordered on one stream (or synchronised by the
 *     caller); two calls on one pool in flight at once race.
 *
 * Unit order is layer-major: u = (l * R + r) * Hkv + h.  One call over L
 * layers gives bit-identical results to L one-layer calls made in layer
 * order with unit_base = l * R * Hkv and tables offset by the same unit count.
 *
 * Precision schemes (dkv_pool.scheme).  The review's free-parameter list
 * compares K8V4, K4V8, K8V2, K4V2, K2V4 and K4V1 (its Section 7.2) and keeps
 * K8V4-K4V2.  A scheme pairs a high class (K at kh bits, V at vh bits) with a
 * low class at half of each, so a low token takes exactly half a high
 * token's code bytes:
 *     DKV_SCHEME_K8V4_K4V2 (0, the default)   kh = 8, vh = 4
 *     DKV_SCHEME_K8V2_K4V1 (1)                kh = 8, vh = 2
 *     DKV_SCHEME_K4V8_K2V4 (2)                kh = 4, vh = 8
 * DKV_CLASS_K8V4 / DKV_CLASS_K4V2 below name the high / low class of
 * whichever scheme the pool uses.
 *
 * Unified page layout (P even; C = 16 (kh + vh) P bytes of codes; page bytes
 * C + 24 P: 216 P for schemes 0 and 2, 184 P for scheme 1).  A high page
 * holds P tokens, a low page 2P tokens:
 *     [0, 16 kh P)     K codes: high slot s at 16 kh s, low slot s at 8 kh s
 *     [16 kh P, C)     V codes: high slot s at 16 kh P + 16 vh s, low slot s
 *                      at 16 kh P + 8 vh s
 *     [C, C + 16P)     per slot s at C + 8 s: fp16 k_scale, k_zero, v_scale,
 *                      v_zero
 *     [C + 16P, C + 24P)  per slot s at C + 16P + 4 s: int32 token position
 * For scheme 0 that is K codes [0, 128P), V codes [128P, 192P), metadata at
 * 192P, positions at 208P.  Sub-byte codes pack lowest channel in the lowest
 * bits.  Slots fill in rank order (ascending position); unused slots,
 * including slots P..2P-1 of a high page, hold zero codes, zero metadata and
 * position -1.
 *
 * Quantiser per token row x[0..127] and bit width b (n = 2^b - 1):
 *     mn = min x, mx = max x (a zero extreme taken as +0); any non-finite x
 *     or |x| > 65504 is DKV_E_RANGE
 *     s16 = fp16_rn((mx - mn) / n), set to 2^-24 if it is 0 while mx > mn,
 *           and to 65504 if it is infinite (1-bit codes of a span > 65519)
 *     z16 = fp16_rn(mn);  s = (float)s16, z = (float)z16
 *     q   = s == 0 ? 0 : clamp(rint_even((x - z) / s), 0, n)   (fp32 ops)
 *     x'  = fma((float)q, s, z)                               (dequantised)
 */
#ifndef DKV_H
#define DKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DKV_OK 0
#define DKV_E_INVAL (-1)    /* sync: invalid argument; nothing enqueued */
#define DKV_E_NOMEM (-2)    /* device: total page demand > free pages */
#define DKV_E_RANGE (-3)    /* device: a K/V value to quantise is non-finite or > 65504 */
#define DKV_E_TIMEOUT (-4)  /* device: a bounded wait of the page scan gave up */
#define DKV_E_INTERNAL (-5) /* device: an internal consistency check failed */
#define DKV_E_CUDA (-6)     /* sync: a CUDA call failed while enqueuing */
#define DKV_E_LENS (-7)     /* device: lens[] disagree with T or max_len */

/* Token classes written to dkv_batch.classes and dkv_pool.page_cls (high /
 * low class of the pool's scheme; the names are those of scheme 0). */
#define DKV_CLASS_PRUNE 0
#define DKV_CLASS_K4V2 1
#define DKV_CLASS_K8V4 2

/* Precision schemes (dkv_pool.scheme). */
#define DKV_SCHEME_K8V4_K4V2 0
#define DKV_SCHEME_K8V2_K4V1 1
#define DKV_SCHEME_K4V8_K2V4 2

#define DKV_HEAD_DIM 128

/* One batch of prefill tokens.  T = sum(lens) tokens per layer and KV head. */
typedef struct dkv_batch {
  int32_t L, R, Hq, Hkv, D;  /* layers, requests, query heads, KV heads, D = 128 */
  int32_t max_len;           /* host-side upper bound on every lens[r] */
  int64_t T;                 /* total tokens of the batch (sum of lens) */
  int64_t unit_base;         /* global id of unit 0 of this call, stored in rev_unit */
  const void *k;             /* bf16 [L][T][Hkv][128], 16-byte aligned */
  const void *v;             /* bf16 [L][T][Hkv][128], 16-byte aligned */
  const float *sig_sum;      /* fp32 [L][T][Hq]: summed attention each token received */
  const int32_t *sig_cnt;    /* int32 [T]: how many scores were summed (N - i in prefill) */
  const int32_t *lens;       /* int32 [R]: tokens of each request, device memory */
  uint8_t *classes;          /* out: uint8 [L][T][Hkv], DKV_CLASS_* per token row */
} dkv_batch;

typedef struct dkv_params {
  float alpha_h;             /* K8V4 threshold alpha_h / N */
  float alpha_l;             /* K4V2 threshold alpha_l / N; 0 <= alpha_l <= alpha_h */
  int32_t spin_limit;        /* polls of one predecessor in the scan look-back before
                                DKV_E_TIMEOUT; 0 gives up at once (any call with
                                more than one scan partition then times out);
                                negative = library default (about a second) */
  int32_t reserved;          /* must be 0 */
  void *profiler;            /* nullable dkv_profiler*: per-kernel event timing */
} dkv_params;

/* The page pool: circular free list, cursors, reverse table and pages. */
typedef struct dkv_pool {
  int64_t F;                 /* pages; 1 <= F <= 2^31 - 1 */
  int32_t P;                 /* high-class tokens per page (low-class pages hold 2P); even */
  int32_t scheme;            /* DKV_SCHEME_*: bit widths and page layout (0 = K8V4/K4V2) */
  int32_t *free_list;        /* int32 [F]: ring of free page ids, slots [head, tail) mod F */
  uint64_t *cursors;         /* uint64 [2]: {head, tail}, monotone; free = tail - head */
  int32_t *rev_unit;         /* int32 [F]: owning global unit id, -1 if free */
  int32_t *rev_idx;          /* int32 [F]: index in the owner's forward row, -1 if free */
  uint8_t *page_cls;         /* uint8 [F]: 0 free, 1 K4V2 page, 2 K8V4 page */
  uint8_t *pages;            /* uint8 [F][dkv_page_bytes], 16-byte aligned */
  int32_t *status;           /* int32 [1]: first device-side error since last read */
} dkv_pool;

/* Forward page table of the units of one call. */
typedef struct dkv_tables {
  int32_t *fwd;              /* int32 [U][pmax]: page ids, K8V4 pages first; -1 past demand */
  int32_t pmax;              /* >= ceil(max_len / P) + 1 */
  int32_t reserved;
  int32_t *unit_hdr;         /* int32 [U][4]: {n_k8v4, n_k4v2, pages_k8v4, pages_k4v2} */
} dkv_tables;

/* Bytes of one unified page of the given scheme and P (host only):
 * (16 (kh + vh) + 24) P.  DKV_E_INVAL for an unknown scheme or P not even
 * and positive. */
int32_t dkv_page_bytes(int32_t scheme, int32_t P, int64_t *bytes);

/* Workspace bytes dkv_compact needs for this batch shape (host only; reads
 * L, R, Hkv, T and max_len of `b`).  Returns DKV_OK or DKV_E_INVAL. */
int32_t dkv_workspace_size(const dkv_batch *b, size_t *bytes);

/* Reset a pool: free_list[i] = i, head = 0, tail = F, rev_* = -1,
 * page_cls = 0, status = 0.  Page contents are left as they are. */
int32_t dkv_init_pool(const dkv_pool *pool, void *stream);

/* Prefill compaction of one batch (steps 1-4 above), asynchronous.
 * workspace: device, 256-byte aligned, >= dkv_workspace_size bytes; its
 * contents need no initialisation and are scratch after the call.
 * On success: classes written; for every unit u, fwd[u][0 .. d_u) holds the
 * page ids taken from free-list slots [head + off_u, head + off_u + d_u) mod F
 * (off_u = exclusive prefix sum of d_u = ceil(n_k8v4 / P) + ceil(n_k4v2 / 2P)),
 * rev_unit / rev_idx / page_cls describe those pages, the pages hold the
 * packed tokens, and head advanced by sum(d_u).
 * One part of the work, clearing the unused slot halves of the new K8V4
 * pages, runs on a library-owned second stream of the current device: it is
 * forked from `stream` after the page scan and joined back before the
 * commit, so the call's effects are ordered on `stream` as if it ran there
 * alone (under stream capture it becomes a fork and a join of the graph).
 * The first call in a CUDA context creates that stream and two events, kept
 * for that context until process exit (a context made after cudaDeviceReset
 * gets its own); make that first call before any stream capture.  Calls from
 * several host threads are safe (the fork and join are enqueued under a
 * lock). */
int32_t dkv_compact(const dkv_batch *b, const dkv_params *p, const dkv_pool *pool,
                    const dkv_tables *t, void *workspace, size_t workspace_bytes,
                    void *stream);

/* dkv_compact without a caller workspace, for callers that cannot allocate
 * device memory (no counterpart in the paper).  Same arguments, results and
 * errors as dkv_compact; the scratch is a library-owned __device__ array of
 * DKV_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until
 * process exit.  A batch whose dkv_workspace_size exceeds that limit is
 * rejected with DKV_E_INVAL before anything is enqueued (the Llama-3-8B-shaped
 * batch of 32 layers x 16 x 4096 tokens needs about 12.5 MiB).  Every call
 * resolves the array's device address in the current context
 * (cudaGetSymbolAddress, which loads the library's module on first use); make
 * the first call on a device before any stream capture.  The array is shared by all calls on a device and keeps the last call's contents
 * (nothing in it needs to start at zero): calls that overlap on the GPU race,
 * so order them on one stream.  Allocates no device memory (the first call
 * on a device creates dkv_compact's second stream and its events). */
#define DKV_NOALLOC_SCRATCH_BYTES (16u << 20)
int32_t dkv_compact_noalloc(const dkv_batch *b, const dkv_params *p, const dkv_pool *pool,
                            const dkv_tables *t, void *stream);

/* Dequantise one page: k_out, v_out fp32 [2P][128], pos_out int32 [2P]
 * (device).  Slots the page class does not have, unused slots and free pages
 * decode to 0 with position -1.  page_id outside [0, F) is DKV_E_INVAL. */
int32_t dkv_dequant_page(const dkv_pool *pool, int32_t page_id, float *k_out, float *v_out,
                         int32_t *pos_out, void *stream);

/* Dequantise n pages whose ids are in device memory page_ids[n]; outputs are
 * [n][2P][128] and [n][2P].  An id outside [0, F) decodes as a free page. */
int32_t dkv_dequant_pages(const dkv_pool *pool, const int32_t *page_ids, int32_t n,
                          float *k_out, float *v_out, int32_t *pos_out, void *stream);

/* ------------------------------------------------------------------------
 * Generation (decode) step.  DiffKV review, Referee Report, major comment 2
 * (Algorithm 1 classifies tokens as they age in the generation phase;
 * demotion and pruning are irreversible), with "What carries the argument"
 * and "Core claim" for classes, unified pages and the page allocator.
 *
 * The context axis of a decode batch is capacity-strided: position i of
 * request r is token row r * cap + i of sig_sum, sig_cnt, classes and
 * slot_of.  Units, pages and tables are those of dkv_compact (a prefill with
 * tables of the same pmax leaves a valid starting state).
 *
 * One step, with N = ctx_lens[r] + new_lens[r]:
 *   - every live token's class becomes min(old class, classify(score, N));
 *     the new token (position ctx_lens[r], when new_lens[r] = 1) is
 *     classified as in prefill;
 *   - per unit, each list (K8V4 slots, K4V2 slots) drops its removed tokens;
 *     with `keep` survivors, those in slots >= keep move, in ascending slot
 *     order, into the holes below keep, in ascending order (bytes copied);
 *   - tokens demoted K8V4 -> K4V2 are appended to the K4V2 list in ascending
 *     position order, requantised (4-bit K, 2-bit V, the quantiser above)
 *     from their dequantised values x = fma(q, s, z); then the new token is
 *     appended to its list (a pruned new token is dropped);
 *   - each list keeps its first min(have, need) pages, need = ceil(n / P)
 *     (K8V4) or ceil(n / 2P) (K4V2); new pages come from free-list slots
 *     head + off_u + k (mod F), off_u the exclusive prefix sum over units of
 *     their new pages, a unit's K8V4 pages first; surplus pages are appended
 *     at the tail in (unit, list, page index) order with rev -1, class 0;
 *   - unused slots of the kept pages are cleared; head and tail advance by
 *     the new and freed page counts; fwd / rev / page_cls / unit_hdr follow.
 * ------------------------------------------------------------------------ */
typedef struct dkv_decode_batch {
  int32_t L, R, Hq, Hkv, D;  /* as dkv_batch; D = 128 */
  int32_t cap;               /* positions reserved per request; a multiple of 16 */
  int64_t unit_base;         /* global id of unit 0 of this call */
  const void *k_new;         /* bf16 [L][R][Hkv][128]: each request's new token (16-byte aligned) */
  const void *v_new;         /* bf16 [L][R][Hkv][128] */
  const float *sig_sum;      /* fp32 [L][R * cap][Hq] (16-byte aligned) */
  const int32_t *sig_cnt;    /* int32 [R * cap]: scores summed for each position */
  const int32_t *ctx_lens;   /* int32 [R]: positions 0 .. ctx-1 are held; device memory */
  const int32_t *new_lens;   /* int32 [R]: 0 or 1 new token at position ctx */
  uint8_t *classes;          /* in/out uint8 [L][R * cap][Hkv] (16-byte aligned): DKV_CLASS_* of
                                positions < ctx (+ the new one after the step); other bytes are
                                not read except the new position's, which the step overwrites */
  int32_t *slot_of;          /* in/out int32 [L][R * cap][Hkv]: slot of each held token in its
                                class list, -1 when pruned; built by dkv_decode_index and
                                maintained by dkv_decode_step */
  int32_t window;            /* W >= 0: the recent window, positions [N - W, N) after the step
                                (the review's Algorithm 1 keeps the W most recent tokens at high
                                precision).  The new token enters as K8V4 when W >= 1 (and is
                                classified when W = 0); held tokens in the window keep their class */
  int32_t mode;              /* 0: every older held token is re-scored (the semantics above);
                                1: only the token the new one pushes out of the window, position
                                ctx - W, is classified, once (Algorithm 1's candidate) */
} dkv_decode_batch;

/* Workspace bytes of dkv_decode_step for this shape (host only). */
int32_t dkv_decode_workspace_size(const dkv_decode_batch *b, size_t *bytes);

/* Derive classes and slot_of of positions 0 .. ctx_lens[r]-1 from the pages
 * and tables (after a prefill, or to rebuild them).  Reads the shape,
 * ctx_lens, the tables and the pages; k_new, v_new, sig_sum, sig_cnt and
 * new_lens are not used (may be NULL).  Every byte of classes
 * and every entry of slot_of is first reset (0 and -1), then each used slot
 * of each unit's lists writes its position's class and slot.  A position or
 * page id out of range in the pages is reported as DKV_E_INTERNAL in the
 * status word.  Asynchronous; allocates nothing. */
int32_t dkv_decode_index(const dkv_decode_batch *b, const dkv_pool *pool, const dkv_tables *t,
                         void *stream);

/* One generation step (semantics above), asynchronous.  workspace: device,
 * 256-byte aligned, >= dkv_decode_workspace_size bytes, scratch.  The caller
 * advances ctx_lens by new_lens after a successful step.  A bad shape, cap
 * not a multiple of 16, window < 0 or mode not 0 or 1 is DKV_E_INVAL before
 * anything is enqueued.  Device-side errors
 * (read with dkv_get_status): DKV_E_LENS (ctx + new > cap, new not 0 or 1, a
 * list needing more than pmax pages), DKV_E_RANGE (a kept new token with a
 * non-finite value or one above 65504), DKV_E_NOMEM (new pages > free
 * pages), DKV_E_TIMEOUT (scan wait), DKV_E_INTERNAL (classes, headers,
 * slot_of or pages contradict one another).  On LENS, RANGE, NOMEM and
 * TIMEOUT, and on INTERNAL found before any page is touched, the step
 * changes nothing (classes restored); INTERNAL found while moving slots
 * leaves the state undefined.  With dkv_params.profiler the five intervals
 * are: counter reset, reclassification (or the candidate kernel in mode 1),
 * page scan, apply, requantisation of the demoted tokens. */
int32_t dkv_decode_step(const dkv_decode_batch *b, const dkv_params *p, const dkv_pool *pool,
                        const dkv_tables *t, void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Decode attention over the unified pages.
 *
 * DiffKV (arXiv 2412.03131), Figure 7 and section 6.1: the generation step's
 * attention reads the mixed-precision unified pages.  The pages do not print
 * that kernel; this is plain scaled dot-product attention.  For query head q
 * of request r in layer l (unit (l, r, q / G), G = Hq / Hkv) the attended
 * tokens are every used slot of the unit's high- and low-class lists (the
 * pool's bit-width scheme: K8V4/K4V2, K8V2/K4V1 or K4V8/K2V4), with K and V
 * the dequantised values fma(code, scale, zero) that dkv_dequant_page gives,
 * plus the step's new token (its bf16 K and V, position ctx_lens[r]) when
 * k_new is given and new_lens[r] = 1:
 *   out = sum_t p_t v_t,   p = softmax_t(scale * (q . k_t)).
 * An empty attended set gives a zero output.  With sig_sum given, each
 * attended held token's significance row receives its probability
 * (sig_sum[l][r * cap + pos][q] += p_t) and the new token's row is set to
 * its p; this is the score whose average decides the classes (Pith review,
 * "What carries the argument").  Counts (sig_cnt) are the caller's: +1 for
 * every held position, 1 for the new token.
 * Computed in fp32 (logits from the codes: scale_k (q . c) + zero_k (sum q)).
 * ------------------------------------------------------------------------ */
typedef struct dkv_attn_batch {
  int32_t L, R, Hq, Hkv;     /* the tables' shape, as in dkv_decode_batch; 1 <= Hq / Hkv <= 8 */
  int32_t cap;               /* positions per request (sig_sum rows); ctx + new <= cap */
  int32_t layer0, n_layers;  /* attend layers [layer0, layer0 + n_layers) of the tables */
  const void *q;             /* bf16 [n_layers][R][Hq][128], 16-byte aligned */
  const void *k_new;         /* bf16 [n_layers][R][Hkv][128] or NULL (no new token), 16-byte aligned */
  const void *v_new;         /* bf16, as k_new (NULL exactly when k_new is) */
  const int32_t *new_lens;   /* int32 [R], 0 or 1 (read only with k_new) */
  const int32_t *ctx_lens;   /* int32 [R]: tokens held before the step (the new token's position) */
  float scale;               /* softmax scale, finite */
  float *out;                /* out fp32 [n_layers][R][Hq][128] */
  float *sig_sum;            /* NULL, or in/out fp32 [L][R * cap][Hq] */
} dkv_attn_batch;

/* Decode attention (above), asynchronous; allocates nothing.  The pool and
 * tables are read only.  Synchronous DKV_E_INVAL: a bad shape or pointer,
 * G outside 1..8, or a shape whose per-block shared memory does not fit 220 KB
 * even with a cluster of 8 blocks per unit (a block holds 2 page buffers of
 * 216 P bytes per warp, 6 warps for G <= 4 and 8 above, plus its share of the
 * unit's logits and positions, (cap + 1) (4 G + 4) / S bytes; S is the
 * smallest cluster that fits, preferring two blocks per SM).  Device-side
 * errors (pool status word): DKV_E_LENS (a new
 * token at ctx >= cap: attended without it), DKV_E_INTERNAL (a unit header,
 * page id or stored position that contradicts the tables: that unit or token
 * is left out). */
int32_t dkv_decode_attention(const dkv_attn_batch *b, const dkv_pool *pool, const dkv_tables *t, void *stream);

/* ------------------------------------------------------------------------
 * Prefill attention that produces the significance inputs of compaction.
 *
 * DiffKV (arXiv 2412.03131), Pith review, "What carries the argument": a
 * token's significance is the average attention it receives from the tokens
 * after it; Referee Report, major comment 2: the average is over the N - i
 * scores token i receives.  For every layer, request and query head q (KV head
 * q / G), query i attends causally over keys 0 .. i of its request:
 *   out_i = sum_{j <= i} p(i, j) v_j,   p(i, .) = softmax_j(scale * q_i . k_j),
 * and the call writes sig_sum[l][t(j)][q] = sum_{i >= j} p(i, j) and
 * sig_cnt[t(j)] = N - j: the inputs dkv_compact classifies.  Computed on the
 * tensor cores (tcgen05): bf16 x bf16 products exact, fp32 accumulation; the
 * significance sums add the fp32 probabilities, the outputs use p rounded to
 * bf16 for the P V product.
 * ------------------------------------------------------------------------ */
typedef struct dkv_prefill_batch {
  int32_t L, R, Hq, Hkv;     /* 1 <= Hq / Hkv */
  int32_t max_len;           /* >= every lens[r] */
  int32_t reserved;
  int64_t T;                 /* sum of lens */
  const void *q;             /* bf16 [L][T][Hq][128], 16-byte aligned */
  const void *k;             /* bf16 [L][T][Hkv][128], 16-byte aligned (the dkv_batch layout) */
  const void *v;             /* bf16 [L][T][Hkv][128], 16-byte aligned; |v| <= 65504 */
  const int32_t *lens;       /* int32 [R] */
  float scale;               /* softmax scale, finite */
  float *out;                /* out fp32 [L][T][Hq][128] */
  float *sig_sum;            /* out fp32 [L][T][Hq] (overwritten) */
  int32_t *sig_cnt;          /* out int32 [T] (overwritten) */
} dkv_prefill_batch;

/* Prefill attention (above), asynchronous; allocates nothing.  Synchronous
 * DKV_E_INVAL for a bad shape or pointer.  Device-side (pool status word;
 * only `pool->status` is used): DKV_E_LENS when a length is negative or above
 * max_len, or the lengths do not add up to T; every block checks all of them
 * before it reads or writes anything, so out and sig_cnt are then left as
 * they were (sig_sum is zeroed first, in any case).  Significance sums are
 * added across query tiles by fp32 atomics, so their last bits depend on the
 * order. */
int32_t dkv_prefill_attention(const dkv_prefill_batch *b, const dkv_pool *pool, void *stream);

/* Synchronise `stream`, return the pool's device status word (DKV_OK or the
 * first device-side error since the last read) and clear it. */
int32_t dkv_get_status(const dkv_pool *pool, void *stream);

/* Per-kernel timing of dkv_compact with CUDA events.  A profiler holds
 * events for up to max_calls calls; every dkv_compact given it (through
 * dkv_params.profiler) records its kernels into the next call slot.
 * dkv_profiler_read synchronises and writes, for each recorded call c and
 * kernel k, ms[c * DKV_PROFILE_KERNELS + k]; it returns the number of calls
 * recorded and starts a new recording. */
#define DKV_PROFILE_KERNELS 5 /* prep, classify, page scan, quantise+scatter, commit */
int32_t dkv_profiler_create(int32_t max_calls, void **profiler);
int32_t dkv_profiler_read(void *profiler, float *ms, int32_t capacity_calls);
int32_t dkv_profiler_destroy(void *profiler);

const char *dkv_status_string(int32_t code);

/* Text of the CUDA error behind the calling thread's last DKV_E_CUDA
 * ("no error" if there was none). */
const char *dkv_last_cuda_error(void);
int32_t dkv_version(void);

/* How the library was built: DKV_BUILD_CHECKED is set in the bounds-checked
 * build (lib/libdkv_checked.so, compiled with -DDKV_CHECKED).  There every
 * page id, free-list index and page-list index that a kernel takes from the
 * tables is checked before it is used; a value outside its range records
 * DKV_E_INTERNAL in the pool status and the access is skipped (the kernel
 * does not trap).  The pool contents after such an error are unspecified.
 * The normal build keeps the checks that cost nothing measurable (page ids
 * read from the forward table or the free list before a page is touched). */
#define DKV_BUILD_CHECKED 1
int32_t dkv_build_flags(void);

#ifdef __cplusplus
}
#endif
#endif /* DKV_H */
