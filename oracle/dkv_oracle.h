/*
 * dkv_oracle.h -- plain, slow, single-threaded CPU oracle for DiffKV-style
 * differentiated KV-cache compaction.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke entry point and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA library never
 * includes this header, never links this code and shares no helper, table or
 * constant with it; the oracle is a restatement of the method from the source
 * pages, written to be checked by eye.
 *
 * Source: "DiffKV: Differentiated Memory Management for Large Language Models
 * with Parallel KV Compaction" (arXiv 2412.03131), Pith review page:
 *   - "What carries the argument": significance = average attention a token
 *     receives from subsequent tokens, max-aggregated over the GQA query heads
 *     of one KV head, compared with alpha_h/N and alpha_l/N; per-head page
 *     demand handed disjoint contiguous page IDs by a prefix sum over the
 *     circular free page list.
 *   - "Core claim": K8V4 for important tokens, K4V2 for moderately important
 *     ones, the rest pruned; unified pages, circular free page list,
 *     bidirectional page table.
 *   - Referee Report, major comment 2 (Section 4, Algorithm 1): the average is
 *     over the N-i scores token i receives; thresholds alpha/N.
 * The quantizer itself is not printed on the page; it follows the KIVI-style
 * per-token asymmetric min/max quantizer the page cites (KIVI; Nagel et al.,
 * "A white paper on neural network quantization"), with fp16 scale and zero
 * and fp32 round-half-to-even arithmetic.
 *
 * Every reading of a silent or ambiguous point is listed in the header of
 * dkv_oracle.cpp next to the function that takes it.
 */
#ifndef DKV_ORACLE_H
#define DKV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes (the values are part of the method's interface). */
#define ORACLE_OK 0
#define ORACLE_E_INVAL (-1)
#define ORACLE_E_NOMEM (-2)
#define ORACLE_E_RANGE (-3)
#define ORACLE_E_LENS (-7)

typedef struct oracle_batch {
  int32_t L, R, Hq, Hkv, D;
  int64_t T;               /* sum of lens */
  const uint16_t *k;       /* bf16 bit patterns [L][T][Hkv][D] */
  const uint16_t *v;       /* bf16 bit patterns [L][T][Hkv][D] */
  const float *sig_sum;    /* [L][T][Hq]: summed attention received */
  const int32_t *sig_cnt;  /* [T]: number of scores summed */
  const int32_t *lens;     /* [R] */
  int64_t unit_base;       /* id of this call's first unit in rev_unit; lets a
                              layer-at-a-time caller keep global unit ids */
} oracle_batch;

typedef struct oracle_pool {
  int64_t F;               /* pages in the pool */
  int32_t P;               /* high-class tokens per page; a low-class page holds 2P */
  int32_t scheme;          /* 0 K8V4/K4V2, 1 K8V2/K4V1, 2 K4V8/K2V4 (reading F) */
  int32_t *free_list;      /* [F] ring of free page ids */
  uint64_t *cursors;       /* [2] {head, tail}, monotone */
  int32_t *rev_unit;       /* [F] owning unit or -1 */
  int32_t *rev_idx;        /* [F] index in the owner's forward row or -1 */
  uint8_t *page_cls;       /* [F] 0 free, 1 K4V2 page, 2 K8V4 page */
  uint8_t *pages;          /* [F][page bytes]: 216*P for schemes 0 and 2, 184*P for scheme 1 */
} oracle_pool;

typedef struct oracle_tables {
  int32_t *fwd;            /* [U][pmax] page ids, -1 past the demand */
  int32_t pmax;
  int32_t *unit_hdr;       /* [U][4] {n_hi, n_lo, pages_hi, pages_lo} */
  uint8_t *classes;        /* [L][T][Hkv] 2 K8V4, 1 K4V2, 0 pruned */
} oracle_tables;

/* IEEE 754 binary32 -> binary16, round to nearest, ties to even. */
uint16_t oracle_fp16_rn(float x);
float oracle_fp16_to_f32(uint16_t h);
void oracle_fp16_rn_array(const float *x, uint16_t *out, int64_t n);

/* Per-token asymmetric quantizer of one row of 128 bf16 values to b bits
 * (b = 1, 2, 4 or 8).
 * Writes q[128] (unpacked codes), *s16 and *z16 (fp16 bits).  Returns
 * ORACLE_OK or ORACLE_E_RANGE. */
int32_t oracle_quant_row(const uint16_t *x, int32_t bits, uint8_t *q,
                         uint16_t *s16, uint16_t *z16);

/* Fresh pool: free_list[i] = i, head 0, tail F, rev -1, page_cls 0. */
void oracle_init_pool(oracle_pool *pool);

/* Prefill compaction.  quant_mask (nullable, [U]) restricts range checks and
 * page writes to the units it marks; classes, counts, page ids, tables and
 * cursors are always computed for every unit. */
int32_t oracle_compact(const oracle_batch *b, float alpha_h, float alpha_l,
                       oracle_pool *pool, oracle_tables *t,
                       const uint8_t *quant_mask);

/* One generation step on the pages a prefill (and earlier steps) left.
 * The context axis is capacity-strided: position i of request r is token
 * r * cap + i of sig_sum / sig_cnt / classes. */
typedef struct oracle_decode_batch {
  int32_t L, R, Hq, Hkv, D;
  int32_t cap;             /* positions reserved per request */
  int64_t unit_base;
  const uint16_t *k_new;   /* bf16 [L][R][Hkv][D]: the new token of each request */
  const uint16_t *v_new;
  const float *sig_sum;    /* [L][R * cap][Hq] */
  const int32_t *sig_cnt;  /* [R * cap] */
  const int32_t *ctx_lens; /* [R] tokens before this step */
  const int32_t *new_lens; /* [R] 0 or 1 */
  uint8_t *classes;        /* in/out [L][R * cap][Hkv] */
  int32_t window;          /* W: the last W positions are the recent window (reading D9) */
  int32_t mode;            /* 0: re-score every older held token; 1: only the token leaving the window */
} oracle_decode_batch;

/* Decode step (reading D in dkv_oracle.cpp).  t->fwd and t->unit_hdr are the
 * unit tables the previous call left (in/out); t->classes is unused. */
int32_t oracle_decode_step(const oracle_decode_batch *b, float alpha_h, float alpha_l,
                           oracle_pool *pool, oracle_tables *t);

/* Decode attention over the unified pages (reading M in dkv_oracle.cpp).
 * Layers [layer0, layer0 + n_layers) of the unit tables; unit of (layer l,
 * request r, KV head h) is (l * R + r) * Hkv + h. */
typedef struct oracle_attn_batch {
  int32_t L, R, Hq, Hkv, cap;
  int32_t layer0, n_layers;
  const uint16_t *q;       /* bf16 [n_layers][R][Hq][128] */
  const uint16_t *k_new;   /* bf16 [n_layers][R][Hkv][128], or NULL: no new token */
  const uint16_t *v_new;
  const int32_t *new_lens; /* [R] 0 or 1 (ignored when k_new is NULL) */
  const int32_t *ctx_lens; /* [R]: the new token's position */
  double scale;            /* softmax scale */
  double *out;             /* [n_layers][R][Hq][128] */
  double *p_out;           /* NULL or [n_layers][R * cap][Hq]: each attended position's
                              probability (0 elsewhere) */
} oracle_attn_batch;

int32_t oracle_decode_attention(const oracle_attn_batch *b, const oracle_pool *pool,
                                const oracle_tables *t);

/* Prefill attention with significance accumulation (reading S in
 * dkv_oracle.cpp): causal softmax attention of every query head over the
 * earlier tokens of its request, and the significance inputs of compaction. */
typedef struct oracle_prefill_batch {
  int32_t L, R, Hq, Hkv;
  int64_t T;               /* sum of lens */
  const uint16_t *q;       /* bf16 [L][T][Hq][128] */
  const uint16_t *k;       /* bf16 [L][T][Hkv][128] */
  const uint16_t *v;
  const int32_t *lens;     /* [R] */
  double scale;
  double *out;             /* [L][T][Hq][128] */
  double *sig_sum;         /* [L][T][Hq]: attention received, summed over the token's queries */
  int32_t *sig_cnt;        /* [T]: that number of queries, N - i */
} oracle_prefill_batch;

int32_t oracle_prefill_attention(const oracle_prefill_batch *b);

/* Decode a page into fp32 K, V ([2P][128] each) and positions ([2P]). */
void oracle_dequant_page(const oracle_pool *pool, int32_t page_id,
                         float *k_out, float *v_out, int32_t *pos_out);

#ifdef __cplusplus
}
#endif
#endif
