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
 *      while mx > mn; z16 = fp16_rn(mn); q = clamp(rint((x - z) / s), 0, n)
 *      with round-half-to-even, or 0 when s == 0.
 *  Q2  Dequantisation x' = fma(q, s, z) in fp32.
 *  P1  Unified page of 216*P bytes: a K8V4 page holds P tokens, a K4V2 page
 *      2P tokens (K4V2 is half the bits of K8V4, so the code region is 192*P
 *      bytes either way).  K codes at [0, 128P), V codes at [128P, 192P),
 *      fp16 {k_scale, k_zero, v_scale, v_zero} per slot at 192P + 8*slot,
 *      int32 token position per slot at 208P + 4*slot.  Unused slots: zero
 *      codes and metadata, position -1.  Nibbles and crumbs pack low-first.
 *  A1  Page demand of a unit (layer, request, KV head):
 *      ceil(n_hi / P) + ceil(n_lo / 2P).  An exclusive prefix sum over units
 *      in layer-major order gives each unit a contiguous run of free-list
 *      slots starting at head + offset (mod F); its K8V4 pages come first.
 *      head advances by the total; a total above tail - head is an
 *      out-of-memory error and the call changes nothing.
 */
#include "dkv_oracle.h"

#include <cmath>
#include <cstdint>
#include <cstring>
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

/* Byte offsets inside one unified page (reading P1). */
struct PageLayout {
  int64_t P;
  int64_t bytes() const { return 216 * P; }
  int64_t k_off(bool high, int64_t slot) const { return slot * (high ? 128 : 64); }
  int64_t v_off(bool high, int64_t slot) const { return 128 * P + slot * (high ? 64 : 32); }
  int64_t meta_off(int64_t slot) const { return 192 * P + 8 * slot; }
  int64_t pos_off(int64_t slot) const { return 208 * P + 4 * slot; }
};

void clear_page(uint8_t *page, const PageLayout &lay) {
  std::memset(page, 0, static_cast<size_t>(208 * lay.P));
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
  if (pool->P < 2 || pool->P % 2 != 0 || pool->F < 1 || t->pmax < 1) return ORACLE_E_INVAL;

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
  const PageLayout lay{P};
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
          oracle_quant_row(b->k + row * 128, high ? 8 : 4, qk, &ks, &kz);
          oracle_quant_row(b->v + row * 128, high ? 4 : 2, qv, &vs, &vz);
          uint8_t *page = pool->pages + static_cast<int64_t>(fwd[k_idx]) * lay.bytes();
          pack_codes(qk, high ? 8 : 4, page + lay.k_off(high, slot));
          pack_codes(qv, high ? 4 : 2, page + lay.v_off(high, slot));
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

/* Reading Q2: x' = fma(q, s, z) per element; slots a page does not have (the
 * upper half of a K8V4 page) and free pages decode to 0 with position -1. */
void oracle_dequant_page(const oracle_pool *pool, int32_t page_id, float *k_out, float *v_out,
                         int32_t *pos_out) {
  const PageLayout lay{pool->P};
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
    unpack_codes(page + lay.k_off(high, s), high ? 8 : 4, qk);
    unpack_codes(page + lay.v_off(high, s), high ? 4 : 2, qv);
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
