/*
 * dkv_oracle.cpp -- the CPU oracle.  TEST INFRASTRUCTURE ONLY (see the header).
 *
 * Build: g++ -std=c++17 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared.
 * -ffp-contract=off keeps every a*b+c as two roundings (GCC contracts to FMA
 * by default on aarch64), so each fp32 expression below is evaluated exactly
 * as written, one IEEE rounding per operation.
 *
 * Readings of points the source page leaves open (the page is the Pith review
 * of "DiffKV: Differentiated Memory Management for Large Language Models with
 * Parallel KV Compaction", arXiv 2412.03131):
 *
 *  S1  Token i (0-indexed) of a request of length N has score
 *      sig_sum / sig_cnt; the producer sums the attention weights of the
 *      queries j >= i (self included) and sets sig_cnt = N - i ("the average
 *      of the N-i attention scores it receives", Referee Report, major
 *      comment 2).  Division is the correctly rounded fp32 quotient.
 *  S2  GQA: query head q belongs to KV head floor(q / G); the score of a KV
 *      head is the maximum over its G query heads ("max-aggregated across GQA
 *      heads", "What carries the argument").  fmax semantics: a NaN score is
 *      ignored, an all-NaN group compares false and is pruned.
 *  S3  The threshold is alpha/N with N the request's current length, not 1/i
 *      (the review flags the 1/i wording as ambiguous; Algorithm 1 uses
 *      alpha/N).  thr = fp32(alpha / (float)N).  "At or above" is >= for both
 *      thresholds.  sig_cnt == 0 ("not yet observed") keeps the token K8V4.
 *  Q1  Quantizer per token row of 128 values and per tensor: mn, mx exact
 *      (a zero extreme canonicalised to +0);
 *      any |x| > 65504 or non-finite x is a range error; s32 = (mx-mn)/n with
 *      n = 2^b - 1; s16 = fp16_rn(s32), bumped to 2^-24 if it underflows to 0
 *      while mx > mn, and lowered to 65504 (the largest finite binary16) if
 *      it overflows to infinity -- possible only at b = 1, for a span above
 *      65519 -- so that the top codes clamp instead of dequantising to NaN;
 *      z16 = fp16_rn(mn); q = clamp(rint((x - z) / s), 0, n) with
 *      round-half-to-even, or 0 when s == 0.
 *  Q2  Dequantisation x' = fma(q, s, z) in fp32.
 *  P1  Unified page of 216*P bytes: a K8V4 page holds P tokens, a K4V2 page
 *      2P tokens (K4V2 is half the bits of K8V4, so the code region is 192*P
 *      bytes either way).  K codes at [0, 128P), V codes at [128P, 192P),
 *      fp16 {k_scale, k_zero, v_scale, v_zero} per slot at 192P + 8*slot,
 *      int32 token position per slot at 208P + 4*slot.  Unused slots: zero
 *      codes and metadata, position -1.  Sub-byte codes pack low-first.
 *  F   Precision schemes (the review's free-parameter list: the scheme
 *      K8V4-K4V2 was chosen by comparing K8V4, K4V8, K8V2, K4V2, K2V4 and
 *      K4V1 in its Section 7.2).  A scheme pairs a high class (K at kh bits,
 *      V at vh bits) with the low class at half of each: K8V4/K4V2 (scheme
 *      0, the default and the one the method states), K8V2/K4V1 (1) and
 *      K4V8/K2V4 (2).  A low token then takes exactly half the code bytes of
 *      a high one, so P1 generalises: a page of 16 (kh + vh) P + 24 P bytes
 *      holds P high or 2P low tokens; K codes at [0, 16 kh P), V codes at
 *      [16 kh P, 16 (kh + vh) P), then the metadata and positions.  The
 *      quantiser (Q1) runs at the class's widths; demotion requantises from
 *      (kh, vh) to (kh/2, vh/2).
 *  A1  Page demand of a unit (layer, request, KV head):
 *      ceil(n_hi / P) + ceil(n_lo / 2P).  An exclusive prefix sum over units
 *      in layer-major order gives each unit a contiguous run of free-list
 *      slots starting at head + offset (mod F); its K8V4 pages come first.
 *      head advances by the total; a total above tail - head is an
 *      out-of-memory error and the call changes nothing.
 *  D   Generation step (the review's Algorithm 1 classifies tokens as they
 *      age; here every live token is re-scored each step and, per the
 *      review, demotion and pruning are irreversible): with N = ctx + new,
 *      an old token's class becomes min(old class, classify(score, N)); the
 *      new token is classified.  Per unit, each list (K8V4 slots, K4V2
 *      slots) drops its removed tokens and is hole-filled: the survivors at
 *      slots >= n' move, in ascending slot order, into the holes below n' in
 *      ascending order (bytes copied unchanged).  Tokens demoted K8V4 -> K4V2
 *      are appended to the K4V2 list in ascending position order,
 *      requantised (Q1 with b = 4 for K, 2 for V) from their dequantised
 *      fp32 values x = fma(q, s, z) (no range error: those values come from
 *      finite fp16 scale and zero).  The new token is appended to its list.
 *      Each list keeps its first min(have, need) pages, need = ceil(n / cap);
 *      new pages come from the free list by the prefix sum of A1 (the unit's
 *      new K8V4 pages first); surplus pages are freed after all allocation,
 *      appended at the tail in (unit, list, page index) order.  Unused slots
 *      of the lists' pages are cleared (zero codes and metadata, position
 *      -1).  A step with new = 0 and no class change leaves everything as it
 *      was.
 *  D9  Recent window and candidate policy (the review's Algorithm 1: a
 *      window of the W most recent tokens stays at high precision, and a
 *      candidate token is classified once, irreversibly, as it leaves the
 *      window).  With window W >= 0 the window after the step is positions
 *      [N - W, N).  The new token enters as K8V4 when W >= 1 and is
 *      classified when W = 0.  Held tokens inside the window keep their
 *      class.  Mode 0 re-scores every older held token as in D; mode 1
 *      re-scores only the token the new one pushes out of the window,
 *      position ctx - W (when there is a new token and W >= 1).  W = 0 with
 *      mode 0 is D itself.
 *  M   Decode attention over the unified pages (DiffKV, Figure 7 and section
 *      6.1: attention runs over the mixed-precision pages; the page never
 *      prints the kernel, so this is plain scaled dot-product attention).
 *      For query head q of request r in layer l, the attended set is every
 *      used slot of the K8V4 and K4V2 lists of unit (l, r, q / G), plus the
 *      step's new token (bf16 K and V, position ctx) when there is one.
 *      k and v of a held token are its dequantised fp32 values fma(c, s, z)
 *      (what oracle_dequant_page returns).  Logits scale * (q . k) with the
 *      bf16 query, softmax and the weighted sum of v are taken in double.
 *      An empty attended set gives a zero output.  The probability given to
 *      each attended position is reported; it is the score that the
 *      significance sum of that position accumulates (the average attention
 *      a token receives, "What carries the argument").
 *  S   Prefill attention and the significance it produces ("What carries the
 *      argument": significance is the average attention a token receives
 *      from the tokens after it; Referee Report, major comment 2: the average
 *      is over the N - i scores token i receives).  Query i of a request
 *      attends, with causal softmax(scale * q . k), over keys 0 .. i of its
 *      request (query head q reads KV head q / G), with the bf16 K and V as
 *      they are; out_i = sum_j p(i, j) v_j.  Key j's significance sum is
 *      sum over i >= j of p(i, j), its count N - j (query j itself
 *      included).  Taken in double.
 */
#include "dkv_oracle.h"

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <utility>
#include <vector>

namespace {

float f32_from_bits(uint32_t u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

uint32_t bits_from_f32(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

float bf16_value(uint16_t h) { return f32_from_bits(static_cast<uint32_t>(h) << 16); }

/* Round the integer mantissa `mant` right by `shift` bits, nearest, ties to
 * even. */
uint32_t round_shift_even(uint32_t mant, int shift) {
  if (shift <= 0) return mant;
  if (shift >= 32) return 0;
  uint32_t keep = mant >> shift;
  uint32_t rem = mant & ((1u << shift) - 1u);
  uint32_t half = 1u << (shift - 1);
  if (rem > half || (rem == half && (keep & 1u))) keep += 1u;
  return keep;
}

void put_u16(uint8_t *p, uint16_t v) { std::memcpy(p, &v, 2); }
void put_i32(uint8_t *p, int32_t v) { std::memcpy(p, &v, 4); }
uint16_t get_u16(const uint8_t *p) {
  uint16_t v;
  std::memcpy(&v, p, 2);
  return v;
}
int32_t get_i32(const uint8_t *p) {
  int32_t v;
  std::memcpy(&v, p, 4);
  return v;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Bit widths of the precision scheme (reading F): the high class stores K
 * at kh and V at vh bits, the low class at half of each. */
int scheme_kh(int32_t scheme) { return scheme == 2 ? 4 : 8; }
int scheme_vh(int32_t scheme) { return scheme == 0 ? 4 : (scheme == 1 ? 2 : 8); }
bool scheme_ok(int32_t scheme) { return scheme >= 0 && scheme <= 2; }

/* Byte offsets inside one unified page (readings P1 and F): a high slot has
 * 128 * kh / 8 bytes of K codes and 128 * vh / 8 of V codes, a low slot half
 * of each, so the code region is 16 (kh + vh) P bytes for P high or 2P low
 * tokens; then 8 bytes of fp16 metadata and 4 of position per slot. */
struct PageLayout {
  int64_t P;
  int kh, vh;
  PageLayout(int64_t P_, int32_t scheme) : P(P_), kh(scheme_kh(scheme)), vh(scheme_vh(scheme)) {}
  int kbits(bool high) const { return high ? kh : kh / 2; }
  int vbits(bool high) const { return high ? vh : vh / 2; }
  int64_t kbytes(bool high) const { return 16 * kbits(high); }
  int64_t vbytes(bool high) const { return 16 * vbits(high); }
  int64_t codes() const { return 16 * (kh + vh) * P; }
  int64_t bytes() const { return codes() + 24 * P; }
  int64_t k_off(bool high, int64_t slot) const { return slot * kbytes(high); }
  int64_t v_off(bool high, int64_t slot) const { return 16 * kh * P + slot * vbytes(high); }
  int64_t meta_off(int64_t slot) const { return codes() + 8 * slot; }
  int64_t pos_off(int64_t slot) const { return codes() + 16 * P + 4 * slot; }
};

void clear_page(uint8_t *page, const PageLayout &lay) {
  std::memset(page, 0, static_cast<size_t>(lay.codes() + 16 * lay.P));
  for (int64_t s = 0; s < 2 * lay.P; ++s) put_i32(page + lay.pos_off(s), -1);
}

/* Pack 128 codes of width `bits` into 128*bits/8 bytes, lowest code in the
 * lowest bits of each byte. */
void pack_codes(const uint8_t *q, int bits, uint8_t *out) {
  const int per_byte = 8 / bits;
  for (int j = 0; j < 128 / per_byte; ++j) {
    unsigned byte = 0;
    for (int e = 0; e < per_byte; ++e) byte |= static_cast<unsigned>(q[j * per_byte + e]) << (e * bits);
    out[j] = static_cast<uint8_t>(byte);
  }
}

void unpack_codes(const uint8_t *in, int bits, uint8_t *q) {
  const int per_byte = 8 / bits;
  const unsigned mask = (1u << bits) - 1u;
  for (int d = 0; d < 128; ++d) q[d] = static_cast<uint8_t>((in[d / per_byte] >> ((d % per_byte) * bits)) & mask);
}

}  // namespace

extern "C" {

/* IEEE 754 binary32 -> binary16 conversion, round to nearest, ties to even,
 * written from the format definitions: binary16 has 5 exponent bits (bias
 * 15) and 10 fraction bits; values below 2^-14 are subnormal multiples of
 * 2^-24; values that round to 2^16 or beyond become infinity. */
uint16_t oracle_fp16_rn(float x) {
  const uint32_t u = bits_from_f32(x);
  const uint16_t sign = static_cast<uint16_t>((u >> 16) & 0x8000u);
  const int e = static_cast<int>((u >> 23) & 0xffu);
  const uint32_t frac = u & 0x7fffffu;
  if (e == 0xff) return static_cast<uint16_t>(sign | (frac ? 0x7e00u : 0x7c00u));
  if (e == 0) return sign; /* binary32 subnormal: below 2^-126, rounds to 0 */
  const uint32_t mant = frac | 0x800000u; /* value = mant * 2^(e - 150) */
  const int E = e - 127 + 15;             /* binary16 biased exponent */
  if (E >= 31) return static_cast<uint16_t>(sign | 0x7c00u);
  if (E >= 1) {
    /* normal: keep 11 significant bits; a carry out of the fraction bumps the
     * exponent, and a carry out of exponent 30 lands on infinity (0x7c00). */
    uint32_t keep = round_shift_even(mant, 13);
    uint32_t h = (static_cast<uint32_t>(E) << 10) + (keep - 0x400u);
    return static_cast<uint16_t>(sign | h);
  }
  /* subnormal: count of 2^-24 units = mant * 2^(e - 150 + 24) */
  const int shift = 126 - e;
  return static_cast<uint16_t>(sign | round_shift_even(mant, shift));
}

float oracle_fp16_to_f32(uint16_t h) {
  const uint32_t sign = static_cast<uint32_t>(h & 0x8000u) << 16;
  const int e = (h >> 10) & 0x1f;
  const uint32_t frac = h & 0x3ffu;
  if (e == 0) {
    float mag = std::ldexp(static_cast<float>(frac), -24);
    return sign ? -mag : mag;
  }
  if (e == 31) return f32_from_bits(sign | 0x7f800000u | (frac << 13));
  return f32_from_bits(sign | (static_cast<uint32_t>(e - 15 + 127) << 23) | (frac << 13));
}

void oracle_fp16_rn_array(const float *x, uint16_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp16_rn(x[i]);
}

/* Reading Q1. */
int32_t oracle_quant_row(const uint16_t *x, int32_t bits, uint8_t *q, uint16_t *s16_out,
                         uint16_t *z16_out) {
  float xf[128];
  for (int d = 0; d < 128; ++d) {
    xf[d] = bf16_value(x[d]);
    if (!std::isfinite(xf[d]) || std::fabs(xf[d]) > 65504.0f) return ORACLE_E_RANGE;
  }
  float mn = xf[0], mx = xf[0];
  for (int d = 1; d < 128; ++d) {
    if (xf[d] < mn) mn = xf[d];
    if (xf[d] > mx) mx = xf[d];
  }
  /* reading Q1: a zero extreme is taken as +0 (IEEE min/max leave the sign
   * of a zero result open when both zeros occur) */
  mn = mn + 0.0f;
  mx = mx + 0.0f;
  const int n = (1 << bits) - 1;
  const float span = mx - mn;
  const float s32 = span / static_cast<float>(n);
  uint16_t s16 = oracle_fp16_rn(s32);
  if (mx > mn && s16 == 0) s16 = 0x0001; /* smallest subnormal, 2^-24 */
  if (s16 == 0x7c00) s16 = 0x7bff;       /* reading Q1 step 3: largest finite, 65504 */
  const uint16_t z16 = oracle_fp16_rn(mn);
  const float s = oracle_fp16_to_f32(s16);
  const float z = oracle_fp16_to_f32(z16);
  for (int d = 0; d < 128; ++d) {
    if (s == 0.0f) {
      q[d] = 0;
      continue;
    }
    const float diff = xf[d] - z;
    const float t = diff / s;
    float r = std::nearbyint(t); /* default rounding mode: ties to even */
    if (r < 0.0f) r = 0.0f;
    if (r > static_cast<float>(n)) r = static_cast<float>(n);
    q[d] = static_cast<uint8_t>(r);
  }
  *s16_out = s16;
  *z16_out = z16;
  return ORACLE_OK;
}

/* Reading Q1 on fp32 inputs (used to requantise demoted tokens). */
static void quant_row_f32(const float *xf, int32_t bits, uint8_t *q, uint16_t *s16_out, uint16_t *z16_out) {
  float mn = xf[0], mx = xf[0];
  for (int d = 1; d < 128; ++d) {
    if (xf[d] < mn) mn = xf[d];
    if (xf[d] > mx) mx = xf[d];
  }
  mn = mn + 0.0f;
  mx = mx + 0.0f;
  const int n = (1 << bits) - 1;
  const float span = mx - mn;
  const float s32 = span / static_cast<float>(n);
  uint16_t s16 = oracle_fp16_rn(s32);
  if (mx > mn && s16 == 0) s16 = 0x0001;
  if (s16 == 0x7c00) s16 = 0x7bff;
  const uint16_t z16 = oracle_fp16_rn(mn);
  const float s = oracle_fp16_to_f32(s16);
  const float z = oracle_fp16_to_f32(z16);
  for (int d = 0; d < 128; ++d) {
    if (s == 0.0f) {
      q[d] = 0;
      continue;
    }
    const float diff = xf[d] - z;
    const float t = diff / s;
    float r = std::nearbyint(t);
    if (r < 0.0f) r = 0.0f;
    if (r > static_cast<float>(n)) r = static_cast<float>(n);
    q[d] = static_cast<uint8_t>(r);
  }
  *s16_out = s16;
  *z16_out = z16;
}

void oracle_init_pool(oracle_pool *pool) {
  for (int64_t i = 0; i < pool->F; ++i) {
    pool->free_list[i] = static_cast<int32_t>(i);
    pool->rev_unit[i] = -1;
    pool->rev_idx[i] = -1;
    pool->page_cls[i] = 0;
  }
  pool->cursors[0] = 0;
  pool->cursors[1] = static_cast<uint64_t>(pool->F);
}

int32_t oracle_compact(const oracle_batch *b, float alpha_h, float alpha_l, oracle_pool *pool,
                       oracle_tables *t, const uint8_t *quant_mask) {
  /* argument checks */
  if (b->D != 128 || b->L < 1 || b->R < 1 || b->Hkv < 1 || b->Hq < b->Hkv || b->Hq % b->Hkv != 0)
    return ORACLE_E_INVAL;
  if (!(alpha_l >= 0.0f) || !(alpha_h >= alpha_l) || !std::isfinite(alpha_h)) return ORACLE_E_INVAL;
  if (pool->P < 2 || pool->P % 2 != 0 || pool->F < 1 || t->pmax < 1 || !scheme_ok(pool->scheme))
    return ORACLE_E_INVAL;

  const int64_t L = b->L, R = b->R, Hq = b->Hq, Hkv = b->Hkv, T = b->T, P = pool->P;
  const int64_t G = Hq / Hkv;
  const int64_t U = L * R * Hkv;

  /* lengths must tile [0, T) and fit the forward table */
  std::vector<int64_t> tok_off(R);
  int64_t sum = 0;
  for (int64_t r = 0; r < R; ++r) {
    const int64_t N = b->lens[r];
    if (N < 0 || N > static_cast<int64_t>(t->pmax - 1) * P) return ORACLE_E_LENS;
    tok_off[r] = sum;
    sum += N;
  }
  if (sum != T) return ORACLE_E_LENS;

  /* significance, three-tier classification and per-unit counts
   * (readings S1-S3) */
  std::vector<int64_t> n_hi(U, 0), n_lo(U, 0);
  for (int64_t l = 0; l < L; ++l)
    for (int64_t r = 0; r < R; ++r) {
      const int64_t N = b->lens[r];
      const float thr_h = alpha_h / static_cast<float>(N);
      const float thr_l = alpha_l / static_cast<float>(N);
      for (int64_t h = 0; h < Hkv; ++h) {
        const int64_t u = (l * R + r) * Hkv + h;
        for (int64_t i = 0; i < N; ++i) {
          const int64_t tok = tok_off[r] + i;
          const int32_t cnt = b->sig_cnt[tok];
          uint8_t cls;
          if (cnt == 0) {
            cls = 2;
          } else {
            float s = NAN;
            for (int64_t g = 0; g < G; ++g) {
              const float score = b->sig_sum[(l * T + tok) * Hq + h * G + g] / static_cast<float>(cnt);
              s = std::fmax(s, score);
            }
            cls = (s >= thr_h) ? 2 : (s >= thr_l) ? 1 : 0;
          }
          t->classes[(l * T + tok) * Hkv + h] = cls;
          if (cls == 2) ++n_hi[u];
          if (cls == 1) ++n_lo[u];
        }
      }
    }

  /* page demand and serial exclusive prefix sum (reading A1) */
  std::vector<int64_t> p_hi(U), p_lo(U), off(U);
  int64_t total = 0;
  for (int64_t u = 0; u < U; ++u) {
    p_hi[u] = ceil_div(n_hi[u], P);
    p_lo[u] = ceil_div(n_lo[u], 2 * P);
    off[u] = total;
    total += p_hi[u] + p_lo[u];
  }
  const uint64_t head = pool->cursors[0], tail = pool->cursors[1];
  if (static_cast<uint64_t>(total) > tail - head) return ORACLE_E_NOMEM;

  /* range check of every row that will be quantised, before any write */
  for (int64_t l = 0; l < L; ++l)
    for (int64_t r = 0; r < R; ++r)
      for (int64_t h = 0; h < Hkv; ++h) {
        const int64_t u = (l * R + r) * Hkv + h;
        if (quant_mask && !quant_mask[u]) continue;
        for (int64_t i = 0; i < b->lens[r]; ++i) {
          const int64_t tok = tok_off[r] + i;
          const int64_t row = (l * T + tok) * Hkv + h;
          if (t->classes[row] == 0) continue;
          for (int d = 0; d < 128; ++d) {
            const float kx = bf16_value(b->k[row * 128 + d]);
            const float vx = bf16_value(b->v[row * 128 + d]);
            if (!std::isfinite(kx) || std::fabs(kx) > 65504.0f) return ORACLE_E_RANGE;
            if (!std::isfinite(vx) || std::fabs(vx) > 65504.0f) return ORACLE_E_RANGE;
          }
        }
      }

  /* tables, page classes and page contents */
  const PageLayout lay(P, pool->scheme);
  const int64_t F = pool->F;
  for (int64_t l = 0; l < L; ++l)
    for (int64_t r = 0; r < R; ++r)
      for (int64_t h = 0; h < Hkv; ++h) {
        const int64_t u = (l * R + r) * Hkv + h;
        const int64_t d = p_hi[u] + p_lo[u];
        const bool write_pages = !quant_mask || quant_mask[u];
        int32_t *fwd = t->fwd + u * t->pmax;
        for (int64_t k = 0; k < t->pmax; ++k) {
          if (k >= d) {
            fwd[k] = -1;
            continue;
          }
          const int64_t slot = static_cast<int64_t>((head + static_cast<uint64_t>(off[u] + k)) % static_cast<uint64_t>(F));
          const int32_t id = pool->free_list[slot];
          fwd[k] = id;
          pool->rev_unit[id] = static_cast<int32_t>(b->unit_base + u);
          pool->rev_idx[id] = static_cast<int32_t>(k);
          pool->page_cls[id] = (k < p_hi[u]) ? 2 : 1;
          if (write_pages) clear_page(pool->pages + static_cast<int64_t>(id) * lay.bytes(), lay);
        }
        int32_t *hdr = t->unit_hdr + u * 4;
        hdr[0] = static_cast<int32_t>(n_hi[u]);
        hdr[1] = static_cast<int32_t>(n_lo[u]);
        hdr[2] = static_cast<int32_t>(p_hi[u]);
        hdr[3] = static_cast<int32_t>(p_lo[u]);
        if (!write_pages) continue;

        int64_t rank_hi = 0, rank_lo = 0;
        for (int64_t i = 0; i < b->lens[r]; ++i) {
          const int64_t tok = tok_off[r] + i;
          const int64_t row = (l * T + tok) * Hkv + h;
          const uint8_t cls = t->classes[row];
          if (cls == 0) continue;
          const bool high = (cls == 2);
          int64_t k_idx, slot;
          if (high) {
            k_idx = rank_hi / P;
            slot = rank_hi % P;
            ++rank_hi;
          } else {
            k_idx = p_hi[u] + rank_lo / (2 * P);
            slot = rank_lo % (2 * P);
            ++rank_lo;
          }
          uint8_t qk[128], qv[128];
          uint16_t ks, kz, vs, vz;
          oracle_quant_row(b->k + row * 128, lay.kbits(high), qk, &ks, &kz);
          oracle_quant_row(b->v + row * 128, lay.vbits(high), qv, &vs, &vz);
          uint8_t *page = pool->pages + static_cast<int64_t>(fwd[k_idx]) * lay.bytes();
          pack_codes(qk, lay.kbits(high), page + lay.k_off(high, slot));
          pack_codes(qv, lay.vbits(high), page + lay.v_off(high, slot));
          uint8_t *meta = page + lay.meta_off(slot);
          put_u16(meta + 0, ks);
          put_u16(meta + 2, kz);
          put_u16(meta + 4, vs);
          put_u16(meta + 6, vz);
          put_i32(page + lay.pos_off(slot), static_cast<int32_t>(i));
        }
      }
  pool->cursors[0] = head + static_cast<uint64_t>(total);
  return ORACLE_OK;
}


namespace {

/* One list of a unit: slot s lives in page pages[s / cap], slot s % cap. */
struct ListRef {
  bool high;
  int64_t cap;
  const int32_t *pages;
};

uint8_t *slot_k(uint8_t *pool_pages, const PageLayout &lay, const ListRef &lr, int64_t s) {
  return pool_pages + static_cast<int64_t>(lr.pages[s / lr.cap]) * lay.bytes() + lay.k_off(lr.high, s % lr.cap);
}

void copy_slot(uint8_t *pp, const PageLayout &lay, const ListRef &lr, int64_t from, int64_t to) {
  const int64_t kb = lay.kbytes(lr.high), vb = lay.vbytes(lr.high);
  uint8_t *fp = pp + static_cast<int64_t>(lr.pages[from / lr.cap]) * lay.bytes();
  uint8_t *tp = pp + static_cast<int64_t>(lr.pages[to / lr.cap]) * lay.bytes();
  const int64_t fs = from % lr.cap, ts = to % lr.cap;
  std::memcpy(tp + lay.k_off(lr.high, ts), fp + lay.k_off(lr.high, fs), static_cast<size_t>(kb));
  std::memcpy(tp + lay.v_off(lr.high, ts), fp + lay.v_off(lr.high, fs), static_cast<size_t>(vb));
  std::memcpy(tp + lay.meta_off(ts), fp + lay.meta_off(fs), 8);
  std::memcpy(tp + lay.pos_off(ts), fp + lay.pos_off(fs), 4);
}

void clear_slot(uint8_t *pp, const PageLayout &lay, const ListRef &lr, int64_t s) {
  const int64_t kb = lay.kbytes(lr.high), vb = lay.vbytes(lr.high);
  uint8_t *pg = pp + static_cast<int64_t>(lr.pages[s / lr.cap]) * lay.bytes();
  const int64_t ss = s % lr.cap;
  std::memset(pg + lay.k_off(lr.high, ss), 0, static_cast<size_t>(kb));
  std::memset(pg + lay.v_off(lr.high, ss), 0, static_cast<size_t>(vb));
  std::memset(pg + lay.meta_off(ss), 0, 8);
  put_i32(pg + lay.pos_off(ss), -1);
}

void write_slot(uint8_t *pp, const PageLayout &lay, const ListRef &lr, int64_t s, const uint8_t *qk, const uint8_t *qv,
                uint16_t ks, uint16_t kz, uint16_t vs, uint16_t vz, int32_t pos) {
  uint8_t *pg = pp + static_cast<int64_t>(lr.pages[s / lr.cap]) * lay.bytes();
  const int64_t ss = s % lr.cap;
  pack_codes(qk, lay.kbits(lr.high), pg + lay.k_off(lr.high, ss));
  pack_codes(qv, lay.vbits(lr.high), pg + lay.v_off(lr.high, ss));
  put_u16(pg + lay.meta_off(ss) + 0, ks);
  put_u16(pg + lay.meta_off(ss) + 2, kz);
  put_u16(pg + lay.meta_off(ss) + 4, vs);
  put_u16(pg + lay.meta_off(ss) + 6, vz);
  put_i32(pg + lay.pos_off(ss), pos);
}

/* Hole-fill of one list: survivors at slots >= n_keep move, in ascending
 * order, into the holes below n_keep, in ascending order. */
void hole_fill(uint8_t *pp, const PageLayout &lay, const ListRef &lr, const std::vector<uint8_t> &keep, int64_t n_keep) {
  std::vector<int64_t> holes, movers;
  for (int64_t s = 0; s < static_cast<int64_t>(keep.size()); ++s) {
    if (s < n_keep && !keep[s]) holes.push_back(s);
    if (s >= n_keep && keep[s]) movers.push_back(s);
  }
  for (size_t k = 0; k < holes.size(); ++k) copy_slot(pp, lay, lr, movers[k], holes[k]);
}

}  // namespace

extern "C" int32_t oracle_decode_step(const oracle_decode_batch *b, float alpha_h, float alpha_l, oracle_pool *pool,
                                      oracle_tables *t) {
  if (b->D != 128 || b->L < 1 || b->R < 1 || b->Hkv < 1 || b->Hq < b->Hkv || b->Hq % b->Hkv != 0 || b->cap < 1)
    return ORACLE_E_INVAL;
  if (!(alpha_l >= 0.0f) || !(alpha_h >= alpha_l) || !std::isfinite(alpha_h)) return ORACLE_E_INVAL;
  if (pool->P < 2 || pool->P % 2 != 0 || pool->F < 1 || t->pmax < 1 || !scheme_ok(pool->scheme))
    return ORACLE_E_INVAL;
  if (b->window < 0 || (b->mode != 0 && b->mode != 1)) return ORACLE_E_INVAL;
  const int64_t L = b->L, R = b->R, Hq = b->Hq, Hkv = b->Hkv, cap = b->cap, P = pool->P, F = pool->F;
  const int64_t G = Hq / Hkv, U = L * R * Hkv, pmax = t->pmax;
  for (int64_t r = 0; r < R; ++r) {
    const int64_t c = b->ctx_lens[r], n = b->new_lens[r];
    if (c < 0 || n < 0 || n > 1 || c + n > cap || c + n > (pmax - 1) * P) return ORACLE_E_LENS;
  }
  const PageLayout lay(P, pool->scheme);
  auto row_of = [&](int64_t l, int64_t r, int64_t i, int64_t h) { return ((l * R + r) * cap + i) * Hkv + h; };

  /* classes after the step (readings S1-S3, D) */
  std::vector<uint8_t> ncls(b->classes, b->classes + L * R * cap * Hkv);
  for (int64_t l = 0; l < L; ++l)
    for (int64_t r = 0; r < R; ++r) {
      const int64_t N = b->ctx_lens[r] + b->new_lens[r];
      if (N == 0) continue;
      const float thr_h = alpha_h / static_cast<float>(N);
      const float thr_l = alpha_l / static_cast<float>(N);
      const int64_t ctx = b->ctx_lens[r], W = b->window;
      for (int64_t i = 0; i < N; ++i) {
        const bool is_new = i >= ctx;
        /* reading D9: which positions are (re)classified this step */
        if (!is_new) {
          if (i >= N - W) continue;                               /* in the window: kept */
          if (b->mode == 1 && !(b->new_lens[r] == 1 && W >= 1 && i == ctx - W)) continue;
        }
        const int64_t tok = r * cap + i;
        const int32_t cnt = b->sig_cnt[tok];
        for (int64_t h = 0; h < Hkv; ++h) {
          uint8_t cls;
          if (is_new && W >= 1) {
            cls = 2;                                               /* enters the window */
          } else if (cnt == 0) {
            cls = 2;
          } else {
            float s = NAN;
            for (int64_t g = 0; g < G; ++g)
              s = std::fmax(s, b->sig_sum[(l * R * cap + tok) * Hq + h * G + g] / static_cast<float>(cnt));
            cls = (s >= thr_h) ? 2 : (s >= thr_l) ? 1 : 0;
          }
          const int64_t row = row_of(l, r, i, h);
          if (i < b->ctx_lens[r] && b->classes[row] < cls) cls = b->classes[row];
          ncls[row] = cls;
        }
      }
    }

  /* per-unit plan */
  struct Plan {
    int64_t keep_hi, keep_lo, dem, n_hi, n_lo, have_hi, have_lo, need_hi, need_lo, d, f;
    int new_cls;
  };
  std::vector<Plan> plan(U);
  std::vector<int64_t> off_d(U), off_f(U);
  int64_t dsum = 0, fsum = 0;
  for (int64_t l = 0; l < L; ++l)
    for (int64_t r = 0; r < R; ++r)
      for (int64_t h = 0; h < Hkv; ++h) {
        const int64_t u = (l * R + r) * Hkv + h;
        const int32_t *hdr = t->unit_hdr + u * 4;
        const int32_t *fw = t->fwd + u * pmax;
        Plan pl{};
        const int64_t n_hi = hdr[0], n_lo = hdr[1];
        pl.have_hi = hdr[2];
        pl.have_lo = hdr[3];
        if (pl.have_hi + pl.have_lo > pmax) return ORACLE_E_INVAL;
        for (int64_t k = 0; k < pl.have_hi + pl.have_lo; ++k)
          if (fw[k] < 0 || fw[k] >= F) return ORACLE_E_INVAL;
        for (int64_t s = 0; s < n_hi; ++s) {
          const uint8_t *pg = pool->pages + static_cast<int64_t>(fw[s / P]) * lay.bytes();
          const int32_t pos = get_i32(pg + lay.pos_off(s % P));
          if (pos < 0 || pos >= b->ctx_lens[r]) return ORACLE_E_INVAL;
          const uint8_t c = ncls[row_of(l, r, pos, h)];
          if (c == 2) ++pl.keep_hi;
          if (c == 1) ++pl.dem;
        }
        for (int64_t s = 0; s < n_lo; ++s) {
          const uint8_t *pg = pool->pages + static_cast<int64_t>(fw[pl.have_hi + s / (2 * P)]) * lay.bytes();
          const int32_t pos = get_i32(pg + lay.pos_off(s % (2 * P)));
          if (pos < 0 || pos >= b->ctx_lens[r]) return ORACLE_E_INVAL;
          const uint8_t c = ncls[row_of(l, r, pos, h)];
          if (c == 2) return ORACLE_E_INVAL;  /* a K4V2 token cannot climb back */
          if (c == 1) ++pl.keep_lo;
        }
        pl.new_cls = b->new_lens[r] ? ncls[row_of(l, r, b->ctx_lens[r], h)] : 0;
        if (pl.new_cls != 0) {
          const int64_t nr = (l * R + r) * Hkv + h;
          for (int d = 0; d < 128; ++d) {
            const float kx = bf16_value(b->k_new[nr * 128 + d]);
            const float vx = bf16_value(b->v_new[nr * 128 + d]);
            if (!std::isfinite(kx) || std::fabs(kx) > 65504.0f) return ORACLE_E_RANGE;
            if (!std::isfinite(vx) || std::fabs(vx) > 65504.0f) return ORACLE_E_RANGE;
          }
        }
        pl.n_hi = pl.keep_hi + (pl.new_cls == 2);
        pl.n_lo = pl.keep_lo + pl.dem + (pl.new_cls == 1);
        pl.need_hi = ceil_div(pl.n_hi, P);
        pl.need_lo = ceil_div(pl.n_lo, 2 * P);
        if (pl.need_hi + pl.need_lo > pmax) return ORACLE_E_LENS;
        pl.d = std::max<int64_t>(0, pl.need_hi - pl.have_hi) + std::max<int64_t>(0, pl.need_lo - pl.have_lo);
        pl.f = std::max<int64_t>(0, pl.have_hi - pl.need_hi) + std::max<int64_t>(0, pl.have_lo - pl.need_lo);
        off_d[u] = dsum;
        off_f[u] = fsum;
        dsum += pl.d;
        fsum += pl.f;
        plan[u] = pl;
      }
  const uint64_t head = pool->cursors[0], tail = pool->cursors[1];
  if (static_cast<uint64_t>(dsum) > tail - head) return ORACLE_E_NOMEM;

  /* apply, unit by unit */
  std::vector<int32_t> freed;
  for (int64_t l = 0; l < L; ++l)
    for (int64_t r = 0; r < R; ++r)
      for (int64_t h = 0; h < Hkv; ++h) {
        const int64_t u = (l * R + r) * Hkv + h;
        const Plan &pl = plan[u];
        int32_t *hdr = t->unit_hdr + u * 4;
        int32_t *fw = t->fwd + u * pmax;
        const int64_t n_hi = hdr[0], n_lo = hdr[1];
        std::vector<int32_t> old_hi(fw, fw + pl.have_hi), old_lo(fw + pl.have_hi, fw + pl.have_hi + pl.have_lo);
        std::vector<int32_t> new_ids;
        for (int64_t k = 0; k < pl.d; ++k)
          new_ids.push_back(pool->free_list[(head + static_cast<uint64_t>(off_d[u] + k)) % static_cast<uint64_t>(F)]);
        std::vector<int32_t> hi_pages(old_hi), lo_pages(old_lo);
        size_t nx = 0;
        std::vector<int32_t> created;
        while (static_cast<int64_t>(hi_pages.size()) < pl.need_hi) {
          hi_pages.push_back(new_ids[nx]);
          created.push_back(new_ids[nx++]);
        }
        while (static_cast<int64_t>(lo_pages.size()) < pl.need_lo) {
          lo_pages.push_back(new_ids[nx]);
          created.push_back(new_ids[nx++]);
        }
        for (int32_t id : created) clear_page(pool->pages + static_cast<int64_t>(id) * lay.bytes(), lay);
        const ListRef HI{true, P, hi_pages.data()}, LO{false, 2 * P, lo_pages.data()};
        /* keep flags and demoted slots */
        std::vector<uint8_t> keep_hi(n_hi), keep_lo(n_lo);
        std::vector<std::pair<int32_t, int64_t>> dem_by_pos;  /* (position, K8V4 slot) */
        for (int64_t s = 0; s < n_hi; ++s) {
          const int32_t pos = get_i32(pool->pages + static_cast<int64_t>(HI.pages[s / P]) * lay.bytes() + lay.pos_off(s % P));
          const uint8_t c = ncls[row_of(l, r, pos, h)];
          keep_hi[s] = c == 2;
          if (c == 1) dem_by_pos.emplace_back(pos, s);
        }
        std::sort(dem_by_pos.begin(), dem_by_pos.end());
        std::vector<int64_t> demoted;
        for (const auto &e : dem_by_pos) demoted.push_back(e.second);
        for (int64_t s = 0; s < n_lo; ++s) {
          const int32_t pos =
              get_i32(pool->pages + static_cast<int64_t>(LO.pages[s / (2 * P)]) * lay.bytes() + lay.pos_off(s % (2 * P)));
          keep_lo[s] = ncls[row_of(l, r, pos, h)] == 1;
        }
        /* K4V2 list first (its appends need the holes filled), then the
         * demoted tokens, then the K8V4 list (after its demoted slots were
         * read), then the new token */
        hole_fill(pool->pages, lay, LO, keep_lo, pl.keep_lo);
        for (size_t k = 0; k < demoted.size(); ++k) {
          const int64_t s = demoted[k];
          const uint8_t *pg = pool->pages + static_cast<int64_t>(HI.pages[s / P]) * lay.bytes();
          const int64_t ss = s % P;
          uint8_t qk[128], qv[128];
          unpack_codes(pg + lay.k_off(true, ss), lay.kbits(true), qk);
          unpack_codes(pg + lay.v_off(true, ss), lay.vbits(true), qv);
          const uint8_t *meta = pg + lay.meta_off(ss);
          const float ks = oracle_fp16_to_f32(get_u16(meta + 0)), kz = oracle_fp16_to_f32(get_u16(meta + 2));
          const float vs = oracle_fp16_to_f32(get_u16(meta + 4)), vz = oracle_fp16_to_f32(get_u16(meta + 6));
          float xk[128], xv[128];
          for (int d = 0; d < 128; ++d) {
            xk[d] = std::fma(static_cast<float>(qk[d]), ks, kz);
            xv[d] = std::fma(static_cast<float>(qv[d]), vs, vz);
          }
          uint8_t nk[128], nv[128];
          uint16_t s1, z1, s2, z2;
          quant_row_f32(xk, lay.kbits(false), nk, &s1, &z1);
          quant_row_f32(xv, lay.vbits(false), nv, &s2, &z2);
          write_slot(pool->pages, lay, LO, pl.keep_lo + static_cast<int64_t>(k), nk, nv, s1, z1, s2, z2,
                     get_i32(pg + lay.pos_off(ss)));
        }
        hole_fill(pool->pages, lay, HI, keep_hi, pl.keep_hi);
        if (pl.new_cls != 0) {
          const int64_t nr = (l * R + r) * Hkv + h;
          const bool high = pl.new_cls == 2;
          uint8_t qk[128], qv[128];
          uint16_t ks, kz, vs, vz;
          oracle_quant_row(b->k_new + nr * 128, lay.kbits(high), qk, &ks, &kz);
          oracle_quant_row(b->v_new + nr * 128, lay.vbits(high), qv, &vs, &vz);
          const int64_t slot = high ? pl.keep_hi : pl.keep_lo + pl.dem;
          write_slot(pool->pages, lay, high ? HI : LO, slot, qk, qv, ks, kz, vs, vz,
                     static_cast<int32_t>(b->ctx_lens[r]));
        }
        for (int64_t s = pl.n_hi; s < pl.need_hi * P; ++s) clear_slot(pool->pages, lay, HI, s);
        for (int64_t s = pl.n_lo; s < pl.need_lo * 2 * P; ++s) clear_slot(pool->pages, lay, LO, s);
        /* freed pages of this unit, in (list, page index) order */
        for (int64_t k = pl.need_hi; k < pl.have_hi; ++k) freed.push_back(old_hi[k]);
        for (int64_t k = pl.need_lo; k < pl.have_lo; ++k) freed.push_back(old_lo[k]);
        /* tables */
        for (int64_t k = 0; k < pmax; ++k) {
          int32_t id = -1;
          if (k < pl.need_hi) id = hi_pages[k];
          else if (k < pl.need_hi + pl.need_lo) id = lo_pages[k - pl.need_hi];
          fw[k] = id;
          if (id >= 0) {
            pool->rev_unit[id] = static_cast<int32_t>(b->unit_base + u);
            pool->rev_idx[id] = static_cast<int32_t>(k);
            pool->page_cls[id] = k < pl.need_hi ? 2 : 1;
          }
        }
        hdr[0] = static_cast<int32_t>(pl.n_hi);
        hdr[1] = static_cast<int32_t>(pl.n_lo);
        hdr[2] = static_cast<int32_t>(pl.need_hi);
        hdr[3] = static_cast<int32_t>(pl.need_lo);
      }
  /* frees after all allocation */
  uint64_t tl = tail;
  for (int32_t id : freed) {
    pool->free_list[tl % static_cast<uint64_t>(F)] = id;
    ++tl;
    pool->rev_unit[id] = -1;
    pool->rev_idx[id] = -1;
    pool->page_cls[id] = 0;
  }
  pool->cursors[0] = head + static_cast<uint64_t>(dsum);
  pool->cursors[1] = tl;
  std::memcpy(b->classes, ncls.data(), ncls.size());
  return ORACLE_OK;
}

/* Reading Q2: x' = fma(q, s, z) per element; slots a page does not have (the
 * upper half of a K8V4 page) and free pages decode to 0 with position -1. */
int32_t oracle_decode_attention(const oracle_attn_batch *b, const oracle_pool *pool,
                                const oracle_tables *t) {
  if (!b || !pool || !t || b->R < 0 || b->Hkv <= 0 || b->Hq <= 0 || b->Hq % b->Hkv != 0 ||
      b->layer0 < 0 || b->n_layers < 0 || b->layer0 + b->n_layers > b->L || !b->q || !b->out ||
      !b->ctx_lens || (b->k_new && (!b->v_new || !b->new_lens)) || !scheme_ok(pool->scheme))
    return ORACLE_E_INVAL;
  const PageLayout lay(pool->P, pool->scheme);
  const int64_t P = pool->P, R = b->R, Hq = b->Hq, Hkv = b->Hkv, G = Hq / Hkv, cap = b->cap;
  if (b->p_out)
    std::fill(b->p_out, b->p_out + static_cast<int64_t>(b->n_layers) * R * cap * Hq, 0.0);
  for (int64_t li = 0; li < b->n_layers; ++li) {
    for (int64_t r = 0; r < R; ++r) {
      for (int64_t h = 0; h < Hkv; ++h) {
        const int64_t u = ((b->layer0 + li) * R + r) * Hkv + h;
        const int32_t *hdr = t->unit_hdr + 4 * u;
        const int32_t *fwd = t->fwd + u * t->pmax;
        /* the attended tokens: dequantised K, V and positions */
        std::vector<float> ks, vs;
        std::vector<int64_t> pos;
        for (int list = 0; list < 2; ++list) {
          const bool high = (list == 0);
          const int64_t n = hdr[list], per = high ? P : 2 * P, first = high ? 0 : hdr[2];
          for (int64_t i = 0; i < n; ++i) {
            const uint8_t *pg = pool->pages + static_cast<int64_t>(fwd[first + i / per]) * lay.bytes();
            const int64_t sl = i % per;
            uint8_t qk[128], qv[128];
            unpack_codes(pg + lay.k_off(high, sl), lay.kbits(high), qk);
            unpack_codes(pg + lay.v_off(high, sl), lay.vbits(high), qv);
            const uint8_t *meta = pg + lay.meta_off(sl);
            const float k_s = oracle_fp16_to_f32(get_u16(meta + 0)), k_z = oracle_fp16_to_f32(get_u16(meta + 2));
            const float v_s = oracle_fp16_to_f32(get_u16(meta + 4)), v_z = oracle_fp16_to_f32(get_u16(meta + 6));
            for (int d = 0; d < 128; ++d) {
              ks.push_back(std::fma(static_cast<float>(qk[d]), k_s, k_z));
              vs.push_back(std::fma(static_cast<float>(qv[d]), v_s, v_z));
            }
            pos.push_back(get_i32(pg + lay.pos_off(sl)));
          }
        }
        if (b->k_new && b->new_lens[r] == 1) {
          const int64_t row = ((li * R + r) * Hkv + h) * 128;
          for (int d = 0; d < 128; ++d) {
            ks.push_back(bf16_value(b->k_new[row + d]));
            vs.push_back(bf16_value(b->v_new[row + d]));
          }
          pos.push_back(b->ctx_lens[r]);
        }
        const int64_t n = static_cast<int64_t>(pos.size());
        for (int64_t g = 0; g < G; ++g) {
          const int64_t qh = h * G + g;
          const uint16_t *qrow = b->q + ((li * R + r) * Hq + qh) * 128;
          double *o = b->out + ((li * R + r) * Hq + qh) * 128;
          for (int d = 0; d < 128; ++d) o[d] = 0.0;
          if (n == 0) continue;
          std::vector<double> lg(n);
          double mx = -INFINITY;
          for (int64_t i = 0; i < n; ++i) {
            double dot = 0.0;
            for (int d = 0; d < 128; ++d) dot += static_cast<double>(bf16_value(qrow[d])) * ks[i * 128 + d];
            lg[i] = b->scale * dot;
            mx = std::max(mx, lg[i]);
          }
          double den = 0.0;
          for (int64_t i = 0; i < n; ++i) {
            lg[i] = std::exp(lg[i] - mx);
            den += lg[i];
          }
          for (int64_t i = 0; i < n; ++i) {
            const double p = lg[i] / den;
            for (int d = 0; d < 128; ++d) o[d] += p * vs[i * 128 + d];
            if (b->p_out) b->p_out[(li * R * cap + r * cap + pos[i]) * Hq + qh] = p;
          }
        }
      }
    }
  }
  return ORACLE_OK;
}

int32_t oracle_prefill_attention(const oracle_prefill_batch *b) {
  if (!b || b->L < 1 || b->R < 0 || b->Hkv < 1 || b->Hq < b->Hkv || b->Hq % b->Hkv != 0 || !b->q || !b->k ||
      !b->v || !b->lens || !b->out || !b->sig_sum || !b->sig_cnt)
    return ORACLE_E_INVAL;
  const int64_t T = b->T, Hq = b->Hq, Hkv = b->Hkv, G = Hq / Hkv;
  int64_t start = 0;
  for (int64_t r = 0; r < b->R; ++r) {
    const int64_t n = b->lens[r];
    for (int64_t i = 0; i < n; ++i) b->sig_cnt[start + i] = static_cast<int32_t>(n - i);
    for (int64_t l = 0; l < b->L; ++l) {
      for (int64_t qh = 0; qh < Hq; ++qh) {
        const int64_t h = qh / G;
        for (int64_t j = 0; j < n; ++j) b->sig_sum[(l * T + start + j) * Hq + qh] = 0.0;
        std::vector<double> lg(static_cast<size_t>(n));
        for (int64_t i = 0; i < n; ++i) {
          const uint16_t *qi = b->q + ((l * T + start + i) * Hq + qh) * 128;
          double mx = -INFINITY;
          for (int64_t j = 0; j <= i; ++j) {
            const uint16_t *kj = b->k + ((l * T + start + j) * Hkv + h) * 128;
            double dot = 0.0;
            for (int d = 0; d < 128; ++d) dot += static_cast<double>(bf16_value(qi[d])) * bf16_value(kj[d]);
            lg[j] = b->scale * dot;
            mx = std::max(mx, lg[j]);
          }
          double den = 0.0;
          for (int64_t j = 0; j <= i; ++j) {
            lg[j] = std::exp(lg[j] - mx);
            den += lg[j];
          }
          double *o = b->out + ((l * T + start + i) * Hq + qh) * 128;
          for (int d = 0; d < 128; ++d) o[d] = 0.0;
          for (int64_t j = 0; j <= i; ++j) {
            const double p = lg[j] / den;
            const uint16_t *vj = b->v + ((l * T + start + j) * Hkv + h) * 128;
            for (int d = 0; d < 128; ++d) o[d] += p * bf16_value(vj[d]);
            b->sig_sum[(l * T + start + j) * Hq + qh] += p;
          }
        }
      }
    }
    start += n;
  }
  return start == T ? ORACLE_OK : ORACLE_E_INVAL;
}

void oracle_dequant_page(const oracle_pool *pool, int32_t page_id, float *k_out, float *v_out,
                         int32_t *pos_out) {
  const PageLayout lay(pool->P, pool->scheme);
  const int64_t P = pool->P;
  const uint8_t cls = pool->page_cls[page_id];
  const uint8_t *page = pool->pages + static_cast<int64_t>(page_id) * lay.bytes();
  for (int64_t s = 0; s < 2 * P; ++s) {
    float *ko = k_out + s * 128;
    float *vo = v_out + s * 128;
    const bool exists = (cls == 1) || (cls == 2 && s < P);
    if (!exists) {
      for (int d = 0; d < 128; ++d) ko[d] = vo[d] = 0.0f;
      pos_out[s] = -1;
      continue;
    }
    const bool high = (cls == 2);
    uint8_t qk[128], qv[128];
    unpack_codes(page + lay.k_off(high, s), lay.kbits(high), qk);
    unpack_codes(page + lay.v_off(high, s), lay.vbits(high), qv);
    const uint8_t *meta = page + lay.meta_off(s);
    const float ks = oracle_fp16_to_f32(get_u16(meta + 0));
    const float kz = oracle_fp16_to_f32(get_u16(meta + 2));
    const float vs = oracle_fp16_to_f32(get_u16(meta + 4));
    const float vz = oracle_fp16_to_f32(get_u16(meta + 6));
    for (int d = 0; d < 128; ++d) {
      ko[d] = std::fma(static_cast<float>(qk[d]), ks, kz);
      vo[d] = std::fma(static_cast<float>(qv[d]), vs, vz);
    }
    pos_out[s] = get_i32(page + lay.pos_off(s));
  }
}

}  // extern "C"
