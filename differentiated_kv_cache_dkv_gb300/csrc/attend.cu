// attend.cu -- decode attention over the unified pages (dkv_decode_attention).
//
// DiffKV (arXiv 2412.03131), Figure 7 and section 6.1: the generation step's
// attention runs over the mixed-precision unified pages.  The pages do not
// print that kernel, so this is plain scaled dot-product attention: each query
// head attends over the held tokens of its KV head (the dequantised K8V4 and
// K4V2 slots) plus the step's new token.  The probability a token receives is
// the score its significance sum accumulates (Pith review, "What carries the
// argument": significance is the average attention a token receives).
//
// One cluster of S blocks per unit (layer, request, KV head); S = 1 whenever
// a unit's logits fit one block's shared memory.  Block `rank` takes a
// contiguous share of the unit's token sequence (the K8V4 list, then the
// K4V2 list, then the new token) and the pages that hold it.  Each of its
// warps takes its share of those pages, round robin, and streams them through a private
// ring of page buffers (bulk async copies completing on mbarriers), so each
// page is read from HBM once, whole and contiguous.  Per 16-slot tile of a
// page the warp
//   - computes the logits on the tensor cores (codes x query), keeps them in
//     shared memory for the significance update,
//   - folds them into its running softmax (maximum per query head, rescaled
//     lazily when it grows by more than 8), and
//   - accumulates the weighted values on the tensor cores (codes x p s_v).
// The warps of a block, then the blocks of the cluster (distributed shared
// memory), merge (max, sum, output); each rank writes a share of the outputs,
// and every block adds its tokens' probabilities to their significance rows.
//
// Arithmetic: with codes c, scale s and zero z of a row,
//   q . k   = s (q . c) + z (sum of q),
//   sum p v = sum (p s_v) c + sum p z_v,
// the two contractions over codes run on the tensor cores (fp16 inputs that
// hold every code and 22 bits of the fp32 factors, fp32 accumulation), the
// rest in fp32.  The step's new token (bf16 K and V) is one more term of its
// block's merge.
//
// Waits: every mbarrier wait is bounded (on expiry the warp records
// DKV_E_TIMEOUT, waits boundedly for its own copies in flight and stops
// reading pages).  The cluster barriers are hardware barriers that every
// thread of every block reaches exactly twice: no thread returns early.
#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <type_traits>

#include "dkv_internal.cuh"

namespace cg = cooperative_groups;

namespace dkv {

namespace {

constexpr int kNS = kAttendStages;
constexpr unsigned kFull = 0xffffffffu;
constexpr int64_t kWaitLimit = 1ll << 24;  // polls of one mbarrier before giving up
constexpr float kRescale = 8.0f;           // lazy softmax rescale threshold (natural log units)

// ------------------------------------------------------------ PTX helpers --

__device__ __forceinline__ uint32_t saddr(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void bar_init(uint64_t *bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(bar)) : "memory");
}

__device__ __forceinline__ void bar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(bar)) : "memory");
}

// Bounded wait for the phase of the given parity.
__device__ __forceinline__ bool bar_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t addr = saddr(bar);
  for (int64_t i = 0; i < kWaitLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// One lane: expect `bytes` on `bar` and start the copies of a page's used
// regions into `dst`: a high-class page its codes and the metadata of its P
// slots, then its positions; a low-class page the whole page.  For scheme SC
// the codes take 16 (kh + vh) P bytes (K8V4/K4V2: [0, 192P)).  Sizes and
// addresses are multiples of 16 bytes.
template <int SC>
__device__ __forceinline__ void fetch_page(uint8_t *dst, const uint8_t *src, int kind, int P, uint64_t *bar) {
  constexpr uint32_t KH = scheme_kh(SC), VH = scheme_vh(SC);
  const uint32_t meta = 16u * (KH + VH) * P, pos = meta + 16u * P;
  const uint32_t b = saddr(bar);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (kind == 1) {
    const uint32_t n0 = meta + 8u * P, n1 = (4u * P + 15u) & ~15u;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(n0 + n1) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     saddr(dst)),
                 "l"(src), "r"(n0), "r"(b)
                 : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     saddr(dst + pos)),
                 "l"(src + pos), "r"(n1), "r"(b)
                 : "memory");
  } else {
    const uint32_t n = meta + 24u * P;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(n) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     saddr(dst)),
                 "l"(src), "r"(n), "r"(b)
                 : "memory");
  }
}

// Code i (of W bits) of a little-endian run of words; i a constant after
// unrolling, so the word and the shift are too.
template <int W>
__device__ __forceinline__ uint32_t code_at_w(const uint32_t *x, int i) {
  return (x[(i * W) >> 5] >> ((i * W) & 31)) & ((1u << W) - 1u);
}

// ---------------------------------------------------------- tensor cores --

// D = A B + D on the tensor cores: A 16x16 and B 16x8 fp16, D fp32.  Lane
// (g, t) = (lane / 4, lane % 4) holds A rows g, g + 8 at columns 2t, 2t + 1
// (a0, a1) and 2t + 8, 2t + 9 (a2, a3); B rows 2t, 2t + 1 (b0) and
// 2t + 8, 2t + 9 (b1) of column g; D rows g, g + 8 at columns 2t, 2t + 1.
__device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                    uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f16bits(float x) { return __half_as_ushort(__float2half_rn(x)); }
__device__ __forceinline__ uint32_t pack2(uint32_t lo, uint32_t hi) { return lo | (hi << 16); }

// Part `lo` (0: nearest fp16, 1: fp16 of the remainder) of x.
__device__ __forceinline__ uint32_t f16part(float x, int lo) {
  const __half h = __float2half_rn(x);
  return lo ? f16bits(x - __half2float(h)) : __half_as_ushort(h);
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }  // -126 <= e <= 127

__device__ __forceinline__ float bf16_at(const uint32_t *w, int e) {
  const uint32_t x = w[e >> 1];
  return __uint_as_float((e & 1) ? (x & 0xffff0000u) : (x << 16));
}

__device__ __forceinline__ float half_lo(uint32_t x) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(x & 0xffffu)));
}
__device__ __forceinline__ float half_hi(uint32_t x) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(x >> 16)));
}

// Byte selector for __byte_perm: byte b of the first word to byte 0 and
// byte b of the second to byte 2 (bytes 1 and 3 are masked off later).
__device__ __forceinline__ uint32_t sel_pair(int b) { return b | (b << 4) | ((4 + b) << 8) | ((4 + b) << 12); }

// A code c as the fp16 bit pattern c (the subnormal c * 2^-24, exact): a byte
// or a masked nibble / crumb moved into the low bits of a half.  The tensor
// core multiplies it exactly; the 2^24 (and the mask's own power of two) is
// undone on the fp32 result.
//
// Layouts (tile = 16 consecutive slots of a page; lane (g, t)):
//   logits   D[row = slot][col = 2 h + part] = sum_k codes . q_part, with the
//            128 channels ordered per 16-column step kc so that lane t's A
//            words are 4 consecutive code bytes of its slot rows:
//              K8V4 (8-bit): columns 2t, 2t+1, 2t+8, 2t+9 = channels
//                32t + 4kc + {0, 1, 2, 3};
//              K4V2 (4-bit): bytes j = 16t + 2kc, j + 1; columns 2t, 2t+1 =
//                their low nibbles (channels 2j, 2j + 2), 2t+8, 2t+9 = their
//                high nibbles (channels 2j + 1, 2j + 3; the query is divided
//                by 16 there to undo the nibble's position);
//   values   D[row = channel][col = 2 h + part] = sum_k codes . (p s_v)_part,
//            k = the tile's slots, lane t's columns 2t, 2t+1, 2t+8, 2t+9 =
//            slots 4t .. 4t+3; rows g, g + 8 of step mt = channels
//            16 g + 2 mt and 16 g + 2 mt + 1 (so lane g's outputs are the 16
//            consecutive channels 16 g ..): K8V4 low / high nibble of byte
//            mt of the lane's 8 bytes, K4V2 crumbs 2 (mt & 1), +1 of byte
//            mt / 2 of its 4 bytes.
// The other bit-width schemes (K8V2/K4V1, K4V8/K2V4) take one code per
// half by shift and mask, in the K8V4 channel order for the logits and the
// value order above for the outputs, at their own widths (1, 2, 4 or 8 bits).
// fp32 inputs become two fp16 parts (nearest, then the remainder) in two
// columns, so the products carry 22 bits of them; query heads are scaled by
// a power of two into fp16 range, and the weights p s_v by the power of two
// that puts the largest weight seen so far there.
constexpr int kChunkTiles = 1;

// Element (4 - t + i) & 3 of four words, i.e. undo the rotated load order.
template <typename T>
__device__ __forceinline__ T unrot(const T (&z)[4], int t, int i) {
  const int k = (4 - t + i) & 3;
  return k == 0 ? z[0] : (k == 1 ? z[1] : (k == 2 ? z[2] : z[3]));
}

// NT: n-tiles of four query heads (G <= 4 NT); SC: the pool's bit-width scheme
template <int NT, int SC>
__global__ void __launch_bounds__(32 * attend_warps(4 * NT), attend_blocks_per_sm(4 * NT)) k_attend(AttnArgs a) {
  constexpr int KH = scheme_kh(SC), VH = scheme_vh(SC);  // high-class K and V widths (the low class: half)
  constexpr int kWarps = attend_warps(4 * NT);
  constexpr int kAttendThreads = 32 * kWarps;
  cg::cluster_group cluster = cg::this_cluster();
  const int32_t S = static_cast<int32_t>(cluster.num_blocks());
  const int32_t rank = static_cast<int32_t>(cluster.block_rank());
  const int64_t ui = blockIdx.x / S;  // unit of this call: (layer, request, KV head)
  const int32_t h = static_cast<int32_t>(ui % a.Hkv);
  const int32_t r = static_cast<int32_t>((ui / a.Hkv) % a.R);
  const int32_t li = static_cast<int32_t>(ui / (static_cast<int64_t>(a.Hkv) * a.R));
  const int64_t u = static_cast<int64_t>(a.layer0) * a.R * a.Hkv + ui;  // unit id in the tables
  const int P = a.P, G = a.G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, tq = lane & 3;

  extern __shared__ __align__(128) uint8_t smem[];
  const AttnLayout lay = attend_layout(a.cmax, G, a.pmax, P);
  const int32_t pbytes = 216 * P;  // a ring slot: the largest page of any scheme
  // the scheme's page: K codes [0, vbase), V codes [vbase, moff), metadata, positions
  const int32_t vbase = 16 * KH * P, moff = 16 * (KH + VH) * P, poff = moff + 16 * P;
  const int64_t gbytes = moff + 24 * static_cast<int64_t>(P);
  uint8_t *stage = smem + lay.stage + static_cast<size_t>(warp) * kNS * pbytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + lay.bar) + warp * kNS;
  float *lg = reinterpret_cast<float *>(smem + lay.lg);
  int32_t *ps = reinterpret_cast<int32_t *>(smem + lay.ps);
  int32_t *fw = reinterpret_cast<int32_t *>(smem + lay.fw);
  float *red = reinterpret_cast<float *>(smem + lay.red);  // [warps][G][128]
  float *wm = reinterpret_cast<float *>(smem + lay.st);    // [warps][8] maxima
  float *wl = wm + kWarps * kAttendMaxG;                   // [warps][8] sums
  float *bM = wl + kWarps * kAttendMaxG, *bL = bM + kAttendMaxG;  // block max / sum (read remotely)
  float *gM = bL + kAttendMaxG, *gL = gM + kAttendMaxG;           // cluster max / sum
  float *bF = gL + kAttendMaxG;  // [8 blocks][8 heads]: exp(block max - cluster max)

  __shared__ int failed;  // a warp gave up on a copy: the significance update is skipped
  __shared__ float nlg_s[kAttendMaxG];  // the new token's logit per query head
  __shared__ float vnew_s[128];         // and its V row
  if (threadIdx.x == 0) failed = 0;
  if (lane == 0) {
    for (int s = 0; s < kNS; ++s) bar_init(bars + s);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // ---- the unit: header, new token, this block's share
  const int4 hd = *reinterpret_cast<const int4 *>(a.unit_hdr + 4 * u);
  int32_t n_hi = hd.x, n_lo = hd.y;
  const int32_t p_hi = hd.z, p_lo = hd.w;
  const int32_t ctx = __ldg(a.ctx_lens + r);
  bool has_new = a.k_new != nullptr && __ldg(a.new_lens + r) == 1;
  if (has_new && (ctx < 0 || ctx >= a.cap)) {
    if (threadIdx.x == 0) set_error(a.status, DKV_E_LENS);
    has_new = false;
  }
  const bool bad = n_hi < 0 || n_lo < 0 || p_hi != (n_hi + P - 1) / P || p_lo != (n_lo + 2 * P - 1) / (2 * P) ||
                   p_hi + p_lo > a.pmax ||
                   static_cast<int64_t>(n_hi) + n_lo + has_new > static_cast<int64_t>(S) * a.cmax;
  if (bad) {
    if (threadIdx.x == 0) set_error(a.status, DKV_E_INTERNAL);
    n_hi = n_lo = 0;
  }
  const int32_t n_held = n_hi + n_lo;
  const int32_t n_tot = n_held + (has_new ? 1 : 0);
  const int32_t chunk = (n_tot + S - 1) / S;
  const int32_t c0 = min(n_tot, rank * chunk), c1 = min(n_tot, c0 + chunk);
  // this block's pages: K8V4 pages [kh0, kh1), then K4V2 pages [kl0, kl1)
  const int32_t h0 = min(c0, n_hi), h1 = min(c1, n_hi);
  const int32_t kh0 = h0 / P, kh1 = h1 > h0 ? (h1 + P - 1) / P : kh0;
  const int32_t l0 = max(c0, n_hi) - n_hi, l1 = max(min(c1, n_held), n_hi) - n_hi;
  const int32_t kl0 = l0 / (2 * P), kl1 = l1 > l0 ? (l1 + 2 * P - 1) / (2 * P) : kl0;
  const int32_t nph = kh1 - kh0, npw = nph + (kl1 - kl0);
  const int32_t npg = bad ? 0 : p_hi + p_lo;
  for (int k = threadIdx.x; k < npg; k += kAttendThreads) {
    const int32_t id = a.fwd[u * a.pmax + k];
    const bool ok = id >= 0 && id < a.F;
    if (!ok) set_error(a.status, DKV_E_INTERNAL);
    fw[k] = ok ? id : -1;
  }
  for (int k = threadIdx.x; k < c1 - c0; k += kAttendThreads) ps[k] = -1;  // tokens never read stay out

  // ---- query fragments.  As a B operand lane (g, t) holds column g: head
  // 4j + g/2, part g & 1, channels 32t .. 32t + 31 (both orders above).  As a
  // D operand it holds head 4j + t: its scale and channel sum.
  const int64_t qrow = (static_cast<int64_t>(li) * a.R + r) * a.Hq + static_cast<int64_t>(h) * G;
  // the same for every warp of the block: warp 0 forms them into shared
  // memory (lane-major, so each lane's 8-byte read is conflict-free)
  __shared__ uint2 frag_h[NT][8][32], frag_l[NT][8][32];  // K8V4 / K4V2 channel orders
  __shared__ float frag_sum[NT][4], frag_inv[NT][4];      // per D-operand head 4j + t
  if (warp == 0) {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int hb = 4 * j + (gq >> 1), part = gq & 1;
      float qv[32];
      float mx = 0.0f, sm = 0.0f;
      if (hb < G) {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.q + (qrow + hb) * 128 + 32 * tq);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = __ldg(src + k);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) qv[8 * k + e] = bf16_at(w, e);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) qv[e] = 0.0f;
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        mx = fmaxf(mx, fabsf(qv[e]));
        sm += qv[e];
      }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
        sm += __shfl_xor_sync(kFull, sm, off);
      }
      // head scale: max |q| into [2^14, 2^15)
      const int ex = mx > 0.0f ? static_cast<int>((__float_as_uint(mx) >> 23) & 0xff) - 127 : 0;
      const int ke = min(max(14 - ex, -100), 100);
      const float sc = pow2f(ke);
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) {
        const float *x = qv + 4 * kc;  // channels 32t + 4kc + {0, 1, 2, 3}
        frag_h[j][kc][lane] = make_uint2(pack2(f16part(x[0] * sc, part), f16part(x[1] * sc, part)),
                                         pack2(f16part(x[2] * sc, part), f16part(x[3] * sc, part)));
        frag_l[j][kc][lane] = make_uint2(pack2(f16part(x[0] * sc, part), f16part(x[2] * sc, part)),
                                         pack2(f16part(x[1] * sc * 0.0625f, part), f16part(x[3] * sc * 0.0625f, part)));
      }
      // the D-operand head 4j + t is the B-operand head of lane 8t
      const float qs = __shfl_sync(kFull, sm, 8 * tq);
      const float qi = pow2f(-__shfl_sync(kFull, ke, 8 * tq)) * 16777216.0f;  // undoes 2^ke and the codes' 2^-24
      if (gq == 0) {
        frag_sum[j][tq] = qs;
        frag_inv[j][tq] = qi;
      }
    }
  }
  __syncthreads();  // fw, barriers, query fragments
  float qsum[NT], qinv[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    qsum[j] = frag_sum[j][tq];
    qinv[j] = frag_inv[j][tq];
  }

  // page item q of this block: kind, page id, first token index, used slots
  auto item = [&](int32_t q, int &kind, int32_t &pid, int32_t &tok0, int32_t &ntok) {
    if (q < nph) {
      const int32_t k = kh0 + q;
      kind = 1;
      pid = fw[k];
      tok0 = k * P;
      ntok = min(P, n_hi - tok0);
    } else {
      const int32_t k = kl0 + (q - nph);
      kind = 2;
      pid = fw[p_hi + k];
      tok0 = n_hi + k * 2 * P;
      ntok = min(2 * P, n_held - tok0);
    }
  };

  // running softmax of head 4j + t: reference maximum m, partial sum l, the
  // zero-point term o0 = sum p z_v, and the tensor-core accumulators cv of
  // sum (p s_v 2^(14 - ew)) c 2^-24 over channels 16g + {2mt, 2mt + 1}; ew is
  // the largest weight exponent seen (it only grows; cv is rescaled by the
  // exact power of two when it does)
  float m[NT], l[NT], o0[NT], cv[NT][8][4];
  int ew[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.0f;
    o0[j] = 0.0f;
    ew[j] = -100;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) cv[j][mt][0] = cv[j][mt][1] = cv[j][mt][2] = cv[j][mt][3] = 0.0f;
  }

  // ---- stream this warp's pages: items warp, warp + 8, ...
  const int32_t nmine = npw > warp ? (npw - warp + kWarps - 1) / kWarps : 0;
  auto issue = [&](int32_t n) {
    int kind;
    int32_t pid, tok0, ntok;
    item(warp + n * kWarps, kind, pid, tok0, ntok);
    uint64_t *bar = bars + n % kNS;
    if (pid >= 0) fetch_page<SC>(stage + (n % kNS) * pbytes, a.pages + pid * gbytes, kind, P, bar);
    else bar_arrive(bar);
  };
  if (lane == 0) {
    for (int32_t n = 0; n < min(nmine, kNS); ++n) issue(n);
  }
  __syncwarp();
  bool ok = true;
  int32_t n = 0;
  for (; n < nmine; ++n) {
    const int s = n % kNS;
    int kind;
    int32_t pid, tok0, ntok;
    item(warp + n * kWarps, kind, pid, tok0, ntok);
    if (!__all_sync(kFull, bar_wait(bars + s, (n / kNS) & 1))) {  // warp-uniform
      ok = false;
      break;
    }
    const uint8_t *pg = stage + s * pbytes;
    const int32_t slo = pid >= 0 ? max(c0 - tok0, 0) : 0;
    const int32_t shi = pid >= 0 ? min(c1 - tok0, ntok) : 0;  // this block's slots of the page
    const int32_t ntiles = shi > slo ? (shi + 15) / 16 : 0;
    for (int32_t ct = slo / 16; ct < ntiles; ct += kChunkTiles) {
      const int nt = min(kChunkTiles, ntiles - ct);
      float w0[kChunkTiles][NT], w1[kChunkTiles][NT];  // p s_v of slots g and g + 8 of each tile
#pragma unroll
      for (int k = 0; k < kChunkTiles; ++k) {
        if (k >= nt) break;
        const int32_t sb = (ct + k) * 16;
        const int32_t s0 = sb + gq, s1 = s0 + 8;
        const bool v0 = s0 >= slo && s0 < shi, v1 = s1 >= slo && s1 < shi;
        const int32_t r0 = min(s0, ntok - 1), r1 = min(s1, ntok - 1);  // rows read (inside the page)
        float c[NT][4], c2[NT][4];  // two accumulators: even and odd column steps
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) c[j][e] = c2[j][e] = 0.0f;
        // other schemes: each code extracted by shift and mask in the K8V4
        // channel order (lane t: channels 32t + 4kc + {0..3} of step kc)
        auto qk_generic = [&](auto wtag) {
          constexpr int W = decltype(wtag)::value;  // K bits
          uint32_t x0[W], x1[W];                    // the lane's 32 channels: 4W bytes of each row
#pragma unroll
          for (int i = 0; i < W; ++i) {
            x0[i] = reinterpret_cast<const uint32_t *>(pg + r0 * 16 * W + 4 * W * tq)[i];
            x1[i] = reinterpret_cast<const uint32_t *>(pg + r1 * 16 * W + 4 * W * tq)[i];
          }
#pragma unroll
          for (int kc = 0; kc < 8; ++kc) {
            const uint32_t a0 = code_at_w<W>(x0, 4 * kc) | (code_at_w<W>(x0, 4 * kc + 1) << 16);
            const uint32_t a2 = code_at_w<W>(x0, 4 * kc + 2) | (code_at_w<W>(x0, 4 * kc + 3) << 16);
            const uint32_t a1 = code_at_w<W>(x1, 4 * kc) | (code_at_w<W>(x1, 4 * kc + 1) << 16);
            const uint32_t a3 = code_at_w<W>(x1, 4 * kc + 2) | (code_at_w<W>(x1, 4 * kc + 3) << 16);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              const uint2 f = frag_h[j][kc][lane];
              mma((kc & 1) ? c2[j] : c[j], a0, a1, a2, a3, f.x, f.y);
            }
          }
        };
        // 8-bit and 4-bit keys take the byte-permute extraction (either class
        // of any scheme), other widths the generic one
        auto qk_k8 = [&]() {
          uint32_t x0[8], x1[8];
          const uint4 *k0 = reinterpret_cast<const uint4 *>(pg + r0 * 128 + 32 * tq);
          const uint4 *k1 = reinterpret_cast<const uint4 *>(pg + r1 * 128 + 32 * tq);
          const uint4 pa = k0[0], pb = k0[1], qa = k1[0], qb = k1[1];
          x0[0] = pa.x; x0[1] = pa.y; x0[2] = pa.z; x0[3] = pa.w; x0[4] = pb.x; x0[5] = pb.y; x0[6] = pb.z; x0[7] = pb.w;
          x1[0] = qa.x; x1[1] = qa.y; x1[2] = qa.z; x1[3] = qa.w; x1[4] = qb.x; x1[5] = qb.y; x1[6] = qb.z; x1[7] = qb.w;
#pragma unroll
          for (int kc = 0; kc < 8; ++kc) {
            const uint32_t a0 = __byte_perm(x0[kc], 0, 0x4140), a2 = __byte_perm(x0[kc], 0, 0x4342);
            const uint32_t a1 = __byte_perm(x1[kc], 0, 0x4140), a3 = __byte_perm(x1[kc], 0, 0x4342);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              const uint2 f = frag_h[j][kc][lane];
              mma((kc & 1) ? c2[j] : c[j], a0, a1, a2, a3, f.x, f.y);
            }
          }
        };
        auto qk_k4 = [&]() {
          const uint4 y0 = *reinterpret_cast<const uint4 *>(pg + r0 * 64 + 16 * tq);
          const uint4 y1 = *reinterpret_cast<const uint4 *>(pg + r1 * 64 + 16 * tq);
          const uint32_t x0[4] = {y0.x, y0.y, y0.z, y0.w}, x1[4] = {y1.x, y1.y, y1.z, y1.w};
#pragma unroll
          for (int kc = 0; kc < 8; ++kc) {
            const uint32_t sel = (kc & 1) ? 0x4342 : 0x4140;
            const uint32_t e0 = __byte_perm(x0[kc >> 1], 0, sel), e1 = __byte_perm(x1[kc >> 1], 0, sel);
            const uint32_t a0 = e0 & 0x000F000Fu, a2 = e0 & 0x00F000F0u;
            const uint32_t a1 = e1 & 0x000F000Fu, a3 = e1 & 0x00F000F0u;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              const uint2 f = frag_l[j][kc][lane];
              mma((kc & 1) ? c2[j] : c[j], a0, a1, a2, a3, f.x, f.y);
            }
          }
        };
        auto qk_width = [&](auto wtag) {
          constexpr int W = decltype(wtag)::value;
          if constexpr (W == 8) qk_k8();
          else if constexpr (W == 4) qk_k4();
          else qk_generic(wtag);
        };
        if (kind == 1) qk_width(std::integral_constant<int, KH>{});
        else qk_width(std::integral_constant<int, KH / 2>{});
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) c[j][e] += c2[j][e];
        const uint2 mt0 = *reinterpret_cast<const uint2 *>(pg + moff + 8 * r0);
        const uint2 mt1 = *reinterpret_cast<const uint2 *>(pg + moff + 8 * r1);
        const float ks0 = half_lo(mt0.x), kz0 = half_hi(mt0.x), sv0 = half_lo(mt0.y), zv0 = half_hi(mt0.y);
        const float ks1 = half_lo(mt1.x), kz1 = half_hi(mt1.x), sv1 = half_lo(mt1.y), zv1 = half_hi(mt1.y);
        if (tq == 0) {
          if (v0) ps[tok0 + s0 - c0] = *reinterpret_cast<const int32_t *>(pg + poff + 4 * r0);
          if (v1) ps[tok0 + s1 - c0] = *reinterpret_cast<const int32_t *>(pg + poff + 4 * r1);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int hh = 4 * j + tq;
          const bool hv = hh < G;
          const float d0 = (c[j][0] + c[j][1]) * qinv[j], d1 = (c[j][2] + c[j][3]) * qinv[j];
          const float lg0 = (v0 && hv) ? a.scale * fmaf(ks0, d0, kz0 * qsum[j]) : -INFINITY;
          const float lg1 = (v1 && hv) ? a.scale * fmaf(ks1, d1, kz1 * qsum[j]) : -INFINITY;
          if (v0 && hv) lg[(tok0 + s0 - c0) * G + hh] = lg0;
          if (v1 && hv) lg[(tok0 + s1 - c0) * G + hh] = lg1;
          // the head's maximum over the tile is taken (a butterfly) only when
          // some lane of the warp needs the reference to move
          float tmx = fmaxf(lg0, lg1);
          const bool up = tmx > m[j] + kRescale || (m[j] == -INFINITY && tmx > -INFINITY);
          if (__any_sync(kFull, up)) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) tmx = fmaxf(tmx, __shfl_xor_sync(kFull, tmx, off));
          }
          if (tmx > m[j] + kRescale || (m[j] == -INFINITY && tmx > -INFINITY)) {  // uniform per head
            const float f = m[j] == -INFINITY ? 0.0f : __expf(m[j] - tmx);
            l[j] *= f;
            o0[j] *= f;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) cv[j][mt][e] *= f;
#pragma unroll
            for (int kk = 0; kk < kChunkTiles; ++kk) {
              if (kk < k) {
                w0[kk][j] *= f;
                w1[kk][j] *= f;
              }
            }
            m[j] = tmx;
          }
          const float p0 = lg0 == -INFINITY ? 0.0f : __expf(lg0 - m[j]);
          const float p1 = lg1 == -INFINITY ? 0.0f : __expf(lg1 - m[j]);
          l[j] += p0 + p1;
          o0[j] = fmaf(p0, zv0, o0[j]);
          o0[j] = fmaf(p1, zv1, o0[j]);
          w0[k][j] = p0 * sv0;
          w1[k][j] = p1 * sv1;
        }
      }
      // the weights' exponent: grow ew to the group's largest weight (cv
      // rescaled exactly), so every weight times 2^(14 - ew) fits fp16
      float sw[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float wx = 0.0f;
#pragma unroll
        for (int k = 0; k < kChunkTiles; ++k)
          if (k < nt) wx = fmaxf(wx, fmaxf(w0[k][j], w1[k][j]));
        int ex = wx > 0.0f ? min(static_cast<int>((__float_as_uint(wx) >> 23) & 0xff) - 127, 100) : -100;
        if (__any_sync(kFull, ex > ew[j])) {  // rare: the head's largest exponent (a butterfly)
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) ex = max(ex, __shfl_xor_sync(kFull, ex, off));
        } else {
          ex = ew[j];
        }
        if (ex > ew[j]) {  // uniform per head
          const float f = pow2f(max(ew[j] - ex, -126));
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) cv[j][mt][e] *= f;
          ew[j] = ex;
        }
        sw[j] = pow2f(14 - ew[j]);
      }
#pragma unroll
      for (int k = 0; k < kChunkTiles; ++k) {
        if (k >= nt) break;
        const int32_t sb = (ct + k) * 16;
        // B: weights of slots t, t + 4 (b0) and t + 8, t + 12 (b1) for this
        // lane's column (head 4j + g/2, part g & 1).  The lane holding slots
        // g, g + 8 of head 4j + t packs (nearest, remainder) of each weight.
        uint32_t b[NT][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const float x0 = w0[k][j] * sw[j], x1 = w1[k][j] * sw[j];
          const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
          const uint32_t pk0 = pack2(__half_as_ushort(h0), f16bits(x0 - __half2float(h0)));
          const uint32_t pk1 = pack2(__half_as_ushort(h1), f16bits(x1 - __half2float(h1)));
          const int sa = (tq << 2) | (gq >> 1), sb4 = ((tq + 4) << 2) | (gq >> 1);
          const uint32_t va = __shfl_sync(kFull, pk0, sa), vb = __shfl_sync(kFull, pk0, sb4);
          const uint32_t vc = __shfl_sync(kFull, pk1, sa), vd = __shfl_sync(kFull, pk1, sb4);
          const uint32_t hs = (gq & 1) ? 0x7632u : 0x5410u;  // remainder halves for odd columns
          b[j][0] = __byte_perm(va, vb, hs);
          b[j][1] = __byte_perm(vc, vd, hs);
        }
        // A: value codes of slots t, t + 4, t + 8, t + 12, channels 16g ..,
        // each code moved to the low bits of its half
        int32_t rr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) rr[i] = min(sb + tq + 4 * i, ntok - 1);
        // other schemes: lane g's 16 channels 16g .. of each of its 4 slots are
        // 2W bytes; each code extracted by shift and mask
        auto pv_generic = [&](auto wtag) {
          constexpr int W = decltype(wtag)::value;  // V bits
          constexpr int NZ = W >= 2 ? W / 2 : 1;     // words of 16 channels
          uint32_t z[4][NZ];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint8_t *src = pg + vbase + rr[i] * 16 * W + 2 * W * gq;
            if (W == 1) {
              z[i][0] = *reinterpret_cast<const uint16_t *>(src);
            } else {
#pragma unroll
              for (int q = 0; q < NZ; ++q) z[i][q] = reinterpret_cast<const uint32_t *>(src)[q];
            }
          }
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const uint32_t a0 = code_at_w<W>(z[0], 2 * mt) | (code_at_w<W>(z[1], 2 * mt) << 16);
            const uint32_t a1 = code_at_w<W>(z[0], 2 * mt + 1) | (code_at_w<W>(z[1], 2 * mt + 1) << 16);
            const uint32_t a2 = code_at_w<W>(z[2], 2 * mt) | (code_at_w<W>(z[3], 2 * mt) << 16);
            const uint32_t a3 = code_at_w<W>(z[2], 2 * mt + 1) | (code_at_w<W>(z[3], 2 * mt + 1) << 16);
#pragma unroll
            for (int j = 0; j < NT; ++j) mma(cv[j][mt], a0, a1, a2, a3, b[j][0], b[j][1]);
          }
        };
        // 4-bit and 2-bit values take the byte-permute extraction (either
        // class of any scheme), other widths the generic one
        auto pv_v4 = [&]() {
          const uint8_t *vb8 = pg + vbase + 8 * gq;
          uint2 z[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) z[i] = *reinterpret_cast<const uint2 *>(vb8 + rr[i] * 64);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const uint32_t sl = sel_pair(mt & 3);
            const uint32_t x01 = __byte_perm(mt < 4 ? z[0].x : z[0].y, mt < 4 ? z[1].x : z[1].y, sl);
            const uint32_t x23 = __byte_perm(mt < 4 ? z[2].x : z[2].y, mt < 4 ? z[3].x : z[3].y, sl);
            const uint32_t a0 = x01 & 0x000F000Fu, a1 = (x01 >> 4) & 0x000F000Fu;
            const uint32_t a2 = x23 & 0x000F000Fu, a3 = (x23 >> 4) & 0x000F000Fu;
#pragma unroll
            for (int j = 0; j < NT; ++j) mma(cv[j][mt], a0, a1, a2, a3, b[j][0], b[j][1]);
          }
        };
        auto pv_v2 = [&]() {
          const uint8_t *vb8 = pg + vbase + 4 * gq;
          uint32_t z[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) z[i] = *reinterpret_cast<const uint32_t *>(vb8 + rr[i] * 32);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const uint32_t sl = sel_pair(mt >> 1);
            const int s0 = (mt & 1) ? 4 : 0;  // crumbs 0, 1 or 2, 3 of the byte
            const uint32_t x01 = __byte_perm(z[0], z[1], sl), x23 = __byte_perm(z[2], z[3], sl);
            const uint32_t a0 = (x01 >> s0) & 0x00030003u, a1 = (x01 >> (s0 + 2)) & 0x00030003u;
            const uint32_t a2 = (x23 >> s0) & 0x00030003u, a3 = (x23 >> (s0 + 2)) & 0x00030003u;
#pragma unroll
            for (int j = 0; j < NT; ++j) mma(cv[j][mt], a0, a1, a2, a3, b[j][0], b[j][1]);
          }
        };
        auto pv_width = [&](auto wtag) {
          constexpr int W = decltype(wtag)::value;
          if constexpr (W == 4) pv_v4();
          else if constexpr (W == 2) pv_v2();
          else pv_generic(wtag);
        };
        if (kind == 1) pv_width(std::integral_constant<int, VH>{});
        else pv_width(std::integral_constant<int, VH / 2>{});
      }
    }
    __syncwarp();  // every lane is done with stage s
    if (lane == 0 && n + kNS < nmine) issue(n + kNS);
  }
  if (!ok) {  // a copy never completed: record it, drain what is in flight (bounded), read no more
    if (lane == 0) {
      set_error(a.status, DKV_E_TIMEOUT);
      failed = 1;
    }
    for (int32_t q = n; q < min(nmine, n + kNS); ++q) bar_wait(bars + q % kNS, (q / kNS) & 1);
  }

  // ---- the step's new token, when this block holds it: its logits and its V
  // row, formed by the last warp as soon as its own pages are done (others may
  // still be streaming), so the merge below finds them in shared memory
  const bool own_new = has_new && n_held >= c0 && n_held < c1;
  const int64_t new_row = ((static_cast<int64_t>(li) * a.R + r) * a.Hkv + h) * 128;
  if (own_new && warp == kWarps - 1) {
    constexpr int kG = 4 * NT;  // query heads a block can hold
    const uint2 kk = __ldg(reinterpret_cast<const uint2 *>(a.k_new + new_row) + lane);  // channels 4 lane ..
    const uint2 vv = __ldg(reinterpret_cast<const uint2 *>(a.v_new + new_row) + lane);
    uint2 qq[kG];
#pragma unroll
    for (int g = 0; g < kG; ++g)
      qq[g] = g < G ? __ldg(reinterpret_cast<const uint2 *>(a.q + (qrow + g) * 128) + lane) : make_uint2(0u, 0u);
    const uint32_t kw[2] = {kk.x, kk.y}, vw[2] = {vv.x, vv.y};
#pragma unroll
    for (int e = 0; e < 4; ++e) vnew_s[4 * lane + e] = bf16_at(vw, e);
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      const uint32_t qw[2] = {qq[g].x, qq[g].y};
      float d = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) d = fmaf(bf16_at(qw, e), bf16_at(kw, e), d);
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) d += __shfl_xor_sync(kFull, d, off);
      if (lane == 0 && g < G) nlg_s[g] = a.scale * d;
    }
  }

  // ---- merge the warp's lanes (same head: lanes of equal t), then the block's warps
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int hh = 4 * j + tq;
    float lw = l[j], zw = o0[j];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      lw += __shfl_xor_sync(kFull, lw, off);
      zw += __shfl_xor_sync(kFull, zw, off);
    }
    if (hh < G) {
      const float so = pow2f(ew[j] + 10);  // 2^24 of the codes times 2^(ew - 14) of the weights
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        red[(warp * G + hh) * 128 + 16 * gq + 2 * mt] = fmaf(cv[j][mt][0] + cv[j][mt][1], so, zw);
        red[(warp * G + hh) * 128 + 16 * gq + 2 * mt + 1] = fmaf(cv[j][mt][2] + cv[j][mt][3], so, zw);
      }
      if (gq == 0) {
        wm[warp * kAttendMaxG + hh] = m[j];
        wl[warp * kAttendMaxG + hh] = lw;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < G) {  // thread g owns column g of wm / wl: it turns maxima into factors
    const int g = threadIdx.x;
    float mx = -INFINITY;
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, wm[w * kAttendMaxG + g]);
    float sum = 0.0f;
    for (int w = 0; w < kWarps; ++w) {
      const float mw = wm[w * kAttendMaxG + g];
      const float f = mw > -INFINITY ? expf(mw - mx) : 0.0f;
      sum = fmaf(wl[w * kAttendMaxG + g], f, sum);
      wm[w * kAttendMaxG + g] = f;
    }
    bM[g] = mx;
    bL[g] = sum;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G * 128; e += kAttendThreads) {
    const int g = e >> 7;
    float sum = 0.0f;
    for (int w = 0; w < kWarps; ++w) sum = fmaf(red[w * G * 128 + e], wm[w * kAttendMaxG + g], sum);
    red[e] = sum;  // each e is read and written by this thread alone
  }

  // ---- the new token (last in the unit's order): one more term of the block's merge
  if (own_new) {
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int g = 0; g < G; ++g) {
        const float x = nlg_s[g];
        lg[(n_held - c0) * G + g] = x;
        const float mx = fmaxf(bM[g], x);
        const float fo = bM[g] == -INFINITY ? 0.0f : expf(bM[g] - mx);
        const float fn = expf(x - mx);
        bL[g] = bL[g] * fo + fn;
        bM[g] = mx;
        wm[g] = fo;  // reused: factors for the outputs below
        wl[g] = fn;
      }
      ps[n_held - c0] = ctx;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < G * 128; e += kAttendThreads) {
      const int g = e >> 7, d = e & 127;
      red[e] = fmaf(wl[g], vnew_s[d], red[e] * wm[g]);
    }
  }
  cluster.sync();  // 1: every block's (max, sum, output) is final

  // ---- merge the cluster's blocks.  The remote reads of every rank are
  // issued together (S <= 8, unrolled), so the merge waits for one
  // distributed-shared-memory round trip, not one per rank.
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    float mq[8], lq[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      mq[q] = -INFINITY;
      lq[q] = 0.0f;
      if (q < S) {
        mq[q] = cluster.map_shared_rank(bM, q)[g];
        lq[q] = cluster.map_shared_rank(bL, q)[g];
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < S) mx = fmaxf(mx, mq[q]);
    float sum = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (q < S) {
        const float f = mq[q] > -INFINITY ? expf(mq[q] - mx) : 0.0f;
        sum = fmaf(lq[q], f, sum);
        bF[q * kAttendMaxG + g] = f;
      }
    }
    gM[g] = mx;
    gL[g] = sum;
  }
  __syncthreads();
  {  // every rank writes its share of the outputs
    float *out = a.out + qrow * 128;
    const int per = (G * 128 + S - 1) / S;
    const int e1 = min(G * 128, (rank + 1) * per);
    for (int e = rank * per + threadIdx.x; e < e1; e += kAttendThreads) {
      const int g = e >> 7;
      float part[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) part[q] = q < S ? cluster.map_shared_rank(red, q)[e] : 0.0f;
      float sum = 0.0f;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < S) sum = fmaf(part[q], bF[q * kAttendMaxG + g], sum);
      const float lsum = gL[g];
      out[e] = lsum > 0.0f ? __fdiv_rn(sum, lsum) : 0.0f;
    }
  }

  // ---- significance: add each token's probability to its row.
  if (a.sig_sum != nullptr && !failed) {
    const int64_t row0 = (static_cast<int64_t>(a.layer0 + li) * a.R + r) * a.cap;
    const int32_t nloc = c1 - c0;
    // one block owns each (position, head) of the call, so an add in the
    // memory system (no value returned: nothing waits on it) equals the
    // read-add-write; the new token's row is set, not added to
    if (G == 4 && (reinterpret_cast<uintptr_t>(a.sig_sum) & 15) == 0) {
      // a token's four heads are 16 contiguous bytes: one vector add
      float mg[4], linv[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        mg[g] = gM[g];
        linv[g] = gL[g] > 0.0f ? 1.0f / gL[g] : 0.0f;
      }
      for (int t = threadIdx.x; t < nloc; t += kAttendThreads) {
        const int32_t pos = ps[t];
        if (pos == -1) continue;  // a token whose page id was rejected
        if (pos < 0 || pos >= a.cap) {
          set_error(a.status, DKV_E_INTERNAL);
          continue;
        }
        float *dst = a.sig_sum + (row0 + pos) * a.Hq + static_cast<int64_t>(h) * 4;
        const float4 l4 = *reinterpret_cast<const float4 *>(lg + t * 4);
        const float p0 = __expf(l4.x - mg[0]) * linv[0], p1 = __expf(l4.y - mg[1]) * linv[1];
        const float p2 = __expf(l4.z - mg[2]) * linv[2], p3 = __expf(l4.w - mg[3]) * linv[3];
        if (c0 + t < n_held)
          asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(p0), "f"(p1), "f"(p2),
                       "f"(p3)
                       : "memory");
        else
          *reinterpret_cast<float4 *>(dst) = make_float4(p0, p1, p2, p3);
      }
    } else {
      // thread (t0, g) = (tid / G, tid % G) takes head g of tokens t0,
      // t0 + T, ... (T = threads / G), so a warp's adds are consecutive
      const int T = kAttendThreads / G;
      const int t0 = threadIdx.x / G, g = threadIdx.x - t0 * G;
      const float lsum = gL[g < G ? g : 0];
      const float linv = lsum > 0.0f ? 1.0f / lsum : 0.0f, mg = gM[g < G ? g : 0];
      if (t0 < T) {
        for (int t = t0; t < nloc; t += T) {
          const int32_t pos = ps[t];
          if (pos == -1) continue;
          if (pos < 0 || pos >= a.cap) {
            set_error(a.status, DKV_E_INTERNAL);
            continue;
          }
          float *dst = a.sig_sum + (row0 + pos) * a.Hq + static_cast<int64_t>(h) * G + g;
          const float pv = __expf(lg[t * G + g] - mg) * linv;
          if (c0 + t < n_held) atomicAdd(dst, pv);
          else *dst = pv;
        }
      }
    }
  }
  cluster.sync();  // 2: no block leaves while another may still read its shared memory
}

template <int NT, int SC>
cudaError_t launch_nt(const AttnArgs &a, int32_t S, size_t smem, cudaStream_t s) {
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(k_attend<NT, SC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.units * S), 1, 1);
  cfg.blockDim = dim3(32 * attend_warps(4 * NT), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_attend<NT, SC>, a);
}

}  // namespace

cudaError_t launch_attend(const AttnArgs &a, int32_t S, cudaStream_t s) {
  if (a.units == 0) return cudaSuccess;
  const size_t smem = attend_layout(a.cmax, a.G, a.pmax, a.P).bytes;
  if (a.G < 1 || a.G > 8) return cudaErrorInvalidValue;
  if (a.scheme == 1) return a.G <= 4 ? launch_nt<1, 1>(a, S, smem, s) : launch_nt<2, 1>(a, S, smem, s);
  if (a.scheme == 2) return a.G <= 4 ? launch_nt<1, 2>(a, S, smem, s) : launch_nt<2, 2>(a, S, smem, s);
  return a.G <= 4 ? launch_nt<1, 0>(a, S, smem, s) : launch_nt<2, 0>(a, S, smem, s);
}

}  // namespace dkv
