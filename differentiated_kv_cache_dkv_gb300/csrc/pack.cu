// pack.cu -- quantise, pack and scatter every surviving token row into its
// unified-page slot (k_pack).
//
// DiffKV (arXiv 2412.03131), Pith review, "Core claim": important tokens are
// stored as K8V4 (keys 8-bit, values 4-bit), moderately important ones as
// K4V2, in unified pages.  The quantiser is per token and per tensor over the
// 128 channels of a head: asymmetric min/max, fp16 scale and zero, codes
// rint((x - z) / s) with ties to even (the KIVI-style per-token quantiser the
// paper cites).
//
// Exactness.  The reference result is q = rint(RN(RN(x - z) / s)) in fp32.
// The kernel computes d = RN(x - z) exactly as the definition, then
// y = RN(d * RN(1/s) + 1536.5) with one fused multiply-add (packed two
// channels at a time with sub.rn.f32x2 / fma.rn.f32x2, which round each half
// like the scalar operation).  y lies in [1024, 2048), so it carries t + 0.5
// in fixed point with 13 fraction bits.  The error of that fixed-point value
// against RN(d / s) + 0.5 is below 0.75 * 2^-13 (quotient <= 256: 2^-24
// relative for the reciprocal, half an ulp of y, 2^-24 relative for the
// reference's own rounding), so bits(y) >> 13 carries the round-to-nearest-even
// code in its low bits unless the 13 fraction bits are all zero -- only then
// can the quotient sit on a tie or on the other side of one.  Those elements,
// and rows whose end points would need clamping (checked exactly per row), are
// recomputed with the IEEE division.  Codes are therefore bit-identical to
// the definition.
//
// Work layout (one CTA per SM, persistent over unit tiles = 128 tokens of one
// (layer, request, KV head)), a warp-specialised pipeline over a ring of
// kStages shared-memory stages:
//   one producer warp issues two TMA tile loads per tile (cp.async.bulk.tensor
//       3-D: the 128 consecutive token rows of one KV head, 32 KB of K and 32
//       KB of V) into the stage, completing on its "full" mbarrier, then
//       stores the list of surviving rows (K8V4 first, ranks by popcount of
//       the class bitmasks) with page id (from the circular free list), slot
//       and position, and arrives on it.
//   consumer warps (19) claim 8-row groups of a stage from a shared counter
//       (low-class rows start at a multiple of 8, so a group is
//       class-uniform: one pair of K / V widths of the pool's scheme),
//       one row per 4-lane group: bf16x2 min / max reduced over the group,
//       one lane each computes the K and the V scale / zero / reciprocal and
//       stores the slot's metadata and position, then every lane quantises
//       its 32 K and 32 V channels as four jobs of 16 channels through one
//       quantiser body (a rolled loop: the consumer code stays small enough
//       for the instruction cache, which bounded the unrolled form) and
//       stores their packed codes at the class's 8, 4, 2 or 1 bits.  A lane's 16-byte chunks are rotated by its
//       group, so the 8 rows a warp reads at once (256 bytes apart) fall on
//       all 32 shared-memory banks.  A warp
//       that finds no group left arrives on the stage's "empty" mbarrier and
//       moves on; the stage is refilled once every consumer warp has left it.
// Unused slots of the pages are filled by k_commit, which walks every page.
// Every mbarrier wait is bounded by the global timer (about a second); on
// expiry the CTA records DKV_E_TIMEOUT, drains its own copies in flight
// (again bounded) and leaves.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kStages = 3;
constexpr int kProducerWarps = 1;
// 19 consumer warps: the most whose registers (88 a thread) fit one block per
// SM without spilling; 18 measured 1.2% slower on the Llama prefill (same GPU,
// alternating runs), 16 slower still, and 20 spill.
constexpr int kConsumerWarps = 19;
constexpr int kPackThreads = 32 * (kConsumerWarps + kProducerWarps);
constexpr uint64_t kWaitNs = 1000000000ull;  // an mbarrier wait gives up after about a second
constexpr uint32_t kWaitPolls = 1u << 26;    // ... or after this many polls, whichever is first

// 1536 = 1.5 * 2^10 puts y in [1024, 2048) (ulp 2^-13); the extra 0.5 turns
// the floor of the 13-bit shift into round-to-nearest.  bits(1536) is a
// multiple of 2^21, so bits(y) >> 13 carries the code in its low 8 bits and
// bits(y) & 8191 is the fixed-point fraction of t + 0.5.
constexpr float kMagicHalf = 1536.5f;

struct __align__(128) Stage {
  uint8_t k[kTileTokens][256];   // bf16 K rows of the tile's 128 tokens
  uint8_t v[kTileTokens][256];   // bf16 V rows
  int4 ent[kTileTokens + 8];     // per listed row: page id, slot, position, token in tile
  int32_t info[4];               // entries spanned, K8V4 rows, first K4V2 entry, row groups
  int32_t next_group;            // claim counter of the consumer warps
};

struct PackSmem {
  Stage st[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
};
constexpr size_t kPackSmemBytes = sizeof(PackSmem) + 128;  // + alignment slack

// ------------------------------------------------------------ PTX helpers --

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for the phase with the given parity to complete: false after
// about kWaitNs of the global timer (or kWaitPolls polls, whichever first).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t addr = smem_addr(bar);
  uint64_t t0 = 0;
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
    if ((i & 63) == 63) {
      const uint64_t t = global_ns();
      if (t0 == 0) t0 = t;
      else if (t - t0 > kWaitNs) return false;
    }
  }
  return false;
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// TMA load of one box of a 3-D tensor map at coordinates (c0, c1, c2),
// completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

// -------------------------------------------------------------- numerics --

__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmin2_nan(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmax2_nan(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Min and max over the 32 bf16 channels a lane holds (16 words), reduced
// over the 4 lanes of a group.  Returns the pair packed as bf16x2
// {min, -max} (NaN propagates).
__device__ __forceinline__ uint32_t row_minmax(const uint4 &a, const uint4 &b, const uint4 &c, const uint4 &d) {
  const uint32_t m0 = bmin2(bmin2(bmin2(a.x, a.y), bmin2(a.z, a.w)), bmin2(bmin2(b.x, b.y), bmin2(b.z, b.w)));
  const uint32_t m1 = bmin2(bmin2(bmin2(c.x, c.y), bmin2(c.z, c.w)), bmin2(bmin2(d.x, d.y), bmin2(d.z, d.w)));
  const uint32_t x0 = bmax2(bmax2(bmax2(a.x, a.y), bmax2(a.z, a.w)), bmax2(bmax2(b.x, b.y), bmax2(b.z, b.w)));
  const uint32_t x1 = bmax2(bmax2(bmax2(c.x, c.y), bmax2(c.z, c.w)), bmax2(bmax2(d.x, d.y), bmax2(d.z, d.w)));
  const uint32_t mn = bmin2(m0, m1), mx = bmax2(x0, x1);
  const uint32_t p0 = __byte_perm(mn, mx, 0x5410) ^ 0x80000000u;  // {mn.lo, -mx.lo}
  const uint32_t p1 = __byte_perm(mn, mx, 0x7632) ^ 0x80000000u;  // {mn.hi, -mx.hi}
  uint32_t p = bmin2(p0, p1);
  p = bmin2(p, __shfl_xor_sync(0xffffffffu, p, 1));
  p = bmin2(p, __shfl_xor_sync(0xffffffffu, p, 2));
  return p;
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

// Result bits of two channels held as one bf16x2 word: the subtraction reads
// each bf16 half directly (mixed precision, no integer unpacking), the
// multiply-add is packed fp32 math
// (each half rounded exactly like the scalar IEEE operation):
//   y = RN(RN(x - z) * r + 1536.5)
__device__ __forceinline__ void fast_pair(uint32_t w, float z, uint64_t rr, uint64_t mm, uint32_t &b0,
                                          uint32_t &b1) {
  // RN(x - z) straight from each bf16 half (mixed-precision subtract: the
  // bf16 operand is widened exactly, the difference rounded once in fp32)
  float d0, d1;
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; sub.rn.f32.bf16 %0, l, %3; sub.rn.f32.bf16 %1, h, %3; }"
      : "=f"(d0), "=f"(d1)
      : "r"(w), "f"(z));
  uint64_t y;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(y) : "l"(pack2(d0, d1)), "l"(rr), "l"(mm));
  asm("mov.b64 {%0, %1}, %2;" : "=r"(b0), "=r"(b1) : "l"(y));
}

// Codes of 16 channels (a: channels 0-7, b: 8-15) with the exact division
// wherever the fast code may differ from the definition, or everywhere for a
// row that needs clamping (r < 0); one code per byte.  Rare, so out of line.
__device__ __noinline__ uint4 exact16(uint4 a, uint4 b, float z, float r, float s, float n) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t out[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float x = (i & 1) ? bf_hi(w[i >> 1]) : bf_lo(w[i >> 1]);
    const float d = __fsub_rn(x, z);
    const uint32_t bits = __float_as_uint(__fmaf_rn(d, r, kMagicHalf));
    uint32_t q = (bits >> 13) & 255u;
    if (r < 0.0f || (bits & 8191u) == 0u) q = static_cast<uint32_t>(fminf(fmaxf(rintf(__fdiv_rn(d, s)), 0.0f), n));
    out[i >> 2] |= q << (8 * (i & 3));
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Per channel the bits of y; the code sits in bits [13, 13 + width).
struct Bits16 {
  uint32_t b[16];
};

__device__ __forceinline__ void quant16(const uint4 &a, const uint4 &b, float z, float r, float s, float n,
                                        Bits16 &q) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  const uint64_t rr = pack2(r, r), mm = pack2(kMagicHalf, kMagicHalf);
  uint32_t flag = 0xffffffffu;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    fast_pair(w[i], z, rr, mm, q.b[2 * i], q.b[2 * i + 1]);
    // the two channels' 13 fraction bits side by side in 16-bit halves: a
    // half of the running minimum becomes zero once a fraction is zero
    flag = __vminu2(flag, __byte_perm(q.b[2 * i], q.b[2 * i + 1], 0x5410) & 0x1fff1fffu);
  }
  if ((flag & 0xffffu) == 0u || (flag >> 16) == 0u || r < 0.0f) {
    const uint4 e = exact16(a, b, z, r, s, n);
    const uint32_t ew[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
    for (int i = 0; i < 16; ++i) q.b[i] = ((ew[i >> 2] >> (8 * (i & 3))) & 255u) << 13;
  }
}

// Pack `count` codes of `width` bits starting at channel `first`, lowest
// channel in the lowest bits: one shift and one and-or per code.
template <int kWidth, int kCount>
__device__ __forceinline__ uint32_t pack_codes(const Bits16 &q, int first) {
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < kCount; ++i) {
    const int sh = 13 - kWidth * i;
    const uint32_t x = sh >= 0 ? (q.b[first + i] >> sh) : (q.b[first + i] << -sh);
    w |= x & (((1u << kWidth) - 1u) << (kWidth * i));
  }
  return w;
}

// Four 8-bit codes (bits 13..20 of each y) into one word by byte permutes.
__device__ __forceinline__ uint32_t pack8x4(const Bits16 &q, int first) {
  const uint32_t c0 = q.b[first] >> 13, c1 = q.b[first + 1] >> 13, c2 = q.b[first + 2] >> 13, c3 = q.b[first + 3] >> 13;
  return __byte_perm(__byte_perm(c0, c1, 0x0040), __byte_perm(c2, c3, 0x0040), 0x5410);
}

// Quantise a lane's 32 K and 32 V channels of one row and store their packed
// codes into the row's slot: four jobs of 16 channels (K chunks l4, l4+4;
// K chunks l4+8, l4+12; the same for V), one quantiser body for all of them,
// the operands re-read from the staged tile.  The class's K and V widths come
// from the scheme's high widths (kKH, kVH), halved for the low class: 8, 4,
// 2 or 1 bits (the 1-bit packing is compiled only for a scheme that has it).
template <int kKH, int kVH>
__device__ __forceinline__ void store_row(uint8_t *pg, int32_t P, int32_t slot_, bool high, int l4,
                                          const uint4 *kr, const uint4 *vr, float kz, float kq, float ks,
                                          float vz, float vq, float vs) {
  constexpr bool kOneBit = kKH == 2 || kVH == 2;
  const int64_t slot = slot_;
  const int kw = high ? kKH : kKH / 2, vw = high ? kVH : kVH / 2;
  uint8_t *kd = pg + slot * 16 * kw;
  uint8_t *vd = pg + static_cast<int64_t>(16 * kKH) * P + slot * 16 * vw;
#pragma unroll 2
  for (int j = 0; j < 4; ++j) {
    const bool isv = j >= 2;
    const int c = (l4 + 8 * (j & 1)) & 15;  // first chunk of the job; the second is c + 4 (mod 16)
    const int c2 = (c + 4) & 15;
    const uint4 *src = isv ? vr : kr;
    const uint4 a = src[c], b = src[c2];
    const float z = isv ? vz : kz, r = isv ? vq : kq, s = isv ? vs : ks;
    const int width = isv ? vw : kw;
    Bits16 q;
    quant16(a, b, z, r, s, static_cast<float>((1 << width) - 1), q);
    uint8_t *d = isv ? vd : kd;
    if (width == 8) {
      *reinterpret_cast<uint2 *>(d + 8 * c) = make_uint2(pack8x4(q, 0), pack8x4(q, 4));
      *reinterpret_cast<uint2 *>(d + 8 * c2) = make_uint2(pack8x4(q, 8), pack8x4(q, 12));
    } else if (width == 4) {
      *reinterpret_cast<uint32_t *>(d + 4 * c) = pack_codes<4, 8>(q, 0);
      *reinterpret_cast<uint32_t *>(d + 4 * c2) = pack_codes<4, 8>(q, 8);
    } else if (!kOneBit || width == 2) {
      *reinterpret_cast<uint16_t *>(d + 2 * c) = static_cast<uint16_t>(pack_codes<2, 8>(q, 0));
      *reinterpret_cast<uint16_t *>(d + 2 * c2) = static_cast<uint16_t>(pack_codes<2, 8>(q, 8));
    } else {
      d[c] = static_cast<uint8_t>(pack_codes<1, 8>(q, 0));
      d[c2] = static_cast<uint8_t>(pack_codes<1, 8>(q, 8));
    }
  }
}

// ---------------------------------------------------------------- kernel --

__device__ __forceinline__ TileDesc load_desc(const CompactArgs &a, int32_t tau) {
  const uint4 *p = reinterpret_cast<const uint4 *>(a.desc + tau);
  TileDesc d;
  uint4 *q = reinterpret_cast<uint4 *>(&d);
  q[0] = __ldg(p);
  q[1] = __ldg(p + 1);
  q[2] = __ldg(p + 2);
  q[3] = __ldg(p + 3);
  return d;
}

__device__ __forceinline__ uint32_t word_of(const uint4 &m, int w) {
  return w == 0 ? m.x : (w == 1 ? m.y : (w == 2 ? m.z : m.w));
}

struct ProducerRows {
  int ent[kMaskWords], slot[kMaskWords];
  int32_t id[kMaskWords];
  int nsurv, nh_t;
};

__device__ __forceinline__ void list_rows(const CompactArgs &a, const TileDesc &m, int lane, int32_t P,
                                          ProducerRows &o) {
  int nh_t = 0, nl_t = 0, pre_h[kMaskWords], pre_l[kMaskWords];
#pragma unroll
  for (int x = 0; x < kMaskWords; ++x) {
    pre_h[x] = nh_t;
    pre_l[x] = nl_t;
    nh_t += __popc(word_of(m.hm, x));
    nl_t += __popc(word_of(m.lm, x));
  }
  // K4V2 entries start at a multiple of 8, so no 8-row group mixes classes
  const int lo0 = (nh_t + 7) & ~7;
  const uint32_t below = (1u << lane) - 1u;
#pragma unroll
  for (int x = 0; x < kMaskWords; ++x) {
    const uint32_t hw = word_of(m.hm, x), lw = word_of(m.lm, x);
    const bool is_hi = (hw >> lane) & 1u;
    const bool is_lo = (lw >> lane) & 1u;
    int pidx = 0;
    o.ent[x] = -1;
    o.slot[x] = 0;
    if (is_hi) {
      o.ent[x] = pre_h[x] + __popc(hw & below);
      const int32_t rho = m.base_hi + o.ent[x];
      pidx = rho / P;
      o.slot[x] = rho - pidx * P;
    } else if (is_lo) {
      const int rl = pre_l[x] + __popc(lw & below);
      o.ent[x] = lo0 + rl;
      const int32_t rho = m.base_lo + rl;
      const int32_t pl = rho / (2 * P);
      pidx = m.p_hi + pl;
      o.slot[x] = rho - pl * 2 * P;
    }
    int64_t idx = static_cast<int64_t>(m.ring) + pidx;
    if (idx >= a.F) idx -= a.F;
    o.id[x] = o.ent[x] >= 0 ? (in_range(idx, a.F, &a.ws->err) ? __ldg(a.free_list + idx) : -1) : 0;
  }
  o.nsurv = lo0 + nl_t;  // entries spanned
  o.nh_t = nh_t;
}

// kS: the pool's precision scheme, so the class widths are constants.
template <int kS>
__global__ void __launch_bounds__(kPackThreads, 1)
    k_pack(CompactArgs a, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ unsigned char smem_raw[];
  PackSmem &sm = *reinterpret_cast<PackSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (a.ws->err != 0) return;

  const int32_t TR = a.ws->TR;
  const int32_t ntiles = TR * a.Hkv * a.L;  // < 2^31: rows are validated below 2^31
  const int32_t P = a.P;
  constexpr int kh = scheme_kh(kS), vh = scheme_vh(kS);
  const int64_t page_bytes = static_cast<int64_t>(16 * (kh + vh) + 24) * P;
  const int64_t meta_off = static_cast<int64_t>(16 * (kh + vh)) * P;
  const int64_t pos_off = meta_off + 16 * static_cast<int64_t>(P);

  if (warp >= kConsumerWarps) {
    int64_t it = 0;
    bool ok = true;
    const int32_t g = gridDim.x;
    const int32_t t0 = blockIdx.x;
    TileDesc cur{}, nxt{}, nxt2{};
    if (t0 < ntiles) cur = load_desc(a, t0);
    if (t0 + g < ntiles) nxt = load_desc(a, t0 + g);
    ProducerRows rows_cur, rows_nxt;
    if (t0 < ntiles) list_rows(a, cur, lane, P, rows_cur);
    for (int32_t tau = t0; tau < ntiles; tau += g, ++it) {
      if (tau + 2 * g < ntiles) nxt2 = load_desc(a, tau + 2 * g);
      const int s = static_cast<int>(it % kStages);
      const uint32_t ph = static_cast<uint32_t>((it / kStages) & 1);
      if (it >= kStages && !mbar_wait(&sm.empty[s], ph ^ 1u)) {
        ok = false;
        break;
      }
      Stage &st = sm.st[s];
      if (lane == 0) {
        mbar_expect_tx(&sm.full[s], 2u * kTileTokens * 256u);
        tma_load_3d(st.k, &kmap, 0, cur.h, cur.tok_row, &sm.full[s]);
        tma_load_3d(st.v, &vmap, 0, cur.h, cur.tok_row, &sm.full[s]);
      }
      if (tau + g < ntiles) list_rows(a, nxt, lane, P, rows_nxt);
#pragma unroll
      for (int x = 0; x < kMaskWords; ++x) {
        if (rows_cur.ent[x] < 0) continue;
        const int k = 32 * x + lane;
        st.ent[rows_cur.ent[x]] = make_int4(rows_cur.id[x], rows_cur.slot[x], cur.pos0 + k, k);
      }
      if (lane == 0) {
        st.info[0] = rows_cur.nsurv;
        st.info[1] = rows_cur.nh_t;
        st.info[2] = (rows_cur.nh_t + 7) & ~7;
        st.info[3] = (rows_cur.nsurv + 7) >> 3;
        st.next_group = 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.full[s]);
      cur = nxt;
      nxt = nxt2;
      rows_cur = rows_nxt;
    }
    if (!ok) set_error(&a.ws->err, DKV_E_TIMEOUT);
    for (int64_t q = (it > kStages ? it - kStages : 0); q < it; ++q)
      mbar_wait(&sm.full[q % kStages], static_cast<uint32_t>((q / kStages) & 1));
    return;
  }

  // -------------------------------------------------------------- consumers
  // Warps claim 8-row groups of a stage from its shared counter, so a warp
  // that is fast on one stage takes more groups or moves on; a stage is
  // released once every warp has left it.
  const int grp = lane >> 2, l4 = lane & 3;
  int64_t it = 0;
  for (int32_t tau = blockIdx.x; tau < ntiles; tau += gridDim.x, ++it) {
    const int s = static_cast<int>(it % kStages);
    const uint32_t ph = static_cast<uint32_t>((it / kStages) & 1);
    if (!mbar_wait(&sm.full[s], ph)) {
      set_error(&a.ws->err, DKV_E_TIMEOUT);
      return;
    }
    Stage &st = sm.st[s];
    const int n_ent = st.info[0];
    const int nh_t = st.info[1];
    const int lo0 = st.info[2];
    const int ngroups = st.info[3];
    for (;;) {
      int g = 0;
      if (lane == 0) g = atomicAdd(&st.next_group, 1);
      g = __shfl_sync(0xffffffffu, g, 0);
      if (g >= ngroups) break;
      const int e = 8 * g + grp;
      const bool valid = e < nh_t || (e >= lo0 && e < n_ent);  // entries [nh, lo0) are padding
      const int4 en = st.ent[valid ? e : 0];  // page id, slot, position, token in tile
      // channels 8c..8c+7 for the chunks c = l4 + 4j, j = 0..3
      const uint4 *kr = reinterpret_cast<const uint4 *>(st.k[en.w]);
      const uint4 *vr = reinterpret_cast<const uint4 *>(st.v[en.w]);
      // the lane's chunks are cb, cb+4, cb+8, cb+12 (mod 16) with cb rotated by
      // the group, so the 8 groups of a warp, reading 8 rows 256 bytes apart,
      // spread their 16-byte loads over all 32 banks
      const int cb = (l4 + grp) & 15;
      const uint4 k0 = kr[cb], k1 = kr[(cb + 4) & 15], k2 = kr[(cb + 8) & 15], k3 = kr[(cb + 12) & 15];
      const uint4 v0 = vr[cb], v1 = vr[(cb + 4) & 15], v2 = vr[(cb + 8) & 15], v3 = vr[(cb + 12) & 15];
      const uint32_t kmm = row_minmax(k0, k1, k2, k3);
      const uint32_t vmm = row_minmax(v0, v1, v2, v3);
      const bool high = 8 * g < nh_t;  // class-uniform group
      // scalar job: lane 0 of the group for K, lane 1 for V
      const int jt = l4 & 1;
      const uint32_t mine = jt ? vmm : kmm;
      constexpr float kNh = (1 << kh) - 1, kNl = (1 << (kh / 2)) - 1, vNh = (1 << vh) - 1, vNl = (1 << (vh / 2)) - 1;
      const float nmax = jt == 0 ? (high ? kNh : kNl) : (high ? vNh : vNl);  // top code of the class's width
      // a zero extreme is +0 (min / max leave the sign of a zero open)
      const float mn = __fadd_rn(bf_lo(mine), 0.0f);
      const float mx = __fadd_rn(-bf_hi(mine), 0.0f);
      const float s32 = __fdiv_rn(__fsub_rn(mx, mn), nmax);
      __half hs = __float2half_rn(s32);
      if (mx > mn && __half_as_ushort(hs) == 0) hs = __ushort_as_half(1);  // 2^-24
      const bool big = __half_as_ushort(hs) == 0x7c00u;  // 1-bit codes of a span above 65519
      if (big) hs = __ushort_as_half(0x7bff);              // 65504: the top codes clamp
      const __half hz = __float2half_rn(mn);
      const float js = __half2float(hs);
      const float jz = __half2float(hz);
      float jr = 0.0f;
      if (js != 0.0f) {
        jr = __frcp_rn(js);
        // Clamping can only be needed when the zero point is not the minimum
        // itself, the scale lost precision as an fp16 subnormal, or it was
        // lowered from infinity; then check the end points exactly.
        if (jz != mn || js < 6.103515625e-05f || big) {
          const float qlo = rintf(__fdiv_rn(__fsub_rn(mn, jz), js));
          const float qhi = rintf(__fdiv_rn(__fsub_rn(mx, jz), js));
          if (!(qlo >= 0.0f && qhi <= nmax)) jr = -1.0f;  // row needs clamping: exact path
        }
      }
      const bool pid_ok = en.x >= 0 && en.x < a.F;  // a corrupt free list is reported, not followed
      if (valid && !pid_ok && l4 == 0) set_error(&a.ws->err, DKV_E_INTERNAL);
      const bool write = valid && pid_ok;
      uint8_t *pg = a.pages + static_cast<int64_t>(write ? en.x : 0) * page_bytes;
      if (write && l4 < 2) {
        if (!(fabsf(mn) <= 65504.0f && fabsf(mx) <= 65504.0f)) set_error(&a.ws->err, DKV_E_RANGE);
        const uint32_t meta = static_cast<uint32_t>(__half_as_ushort(hs)) |
                              (static_cast<uint32_t>(__half_as_ushort(hz)) << 16);
        *reinterpret_cast<uint32_t *>(pg + meta_off + 8 * static_cast<int64_t>(en.y) + 4 * jt) = meta;
        if (jt == 0) *reinterpret_cast<int32_t *>(pg + pos_off + 4 * static_cast<int64_t>(en.y)) = en.z;
      }
      const int src = grp << 2;
      const float kz = __shfl_sync(0xffffffffu, jz, src), kq = __shfl_sync(0xffffffffu, jr, src);
      const float ks = __shfl_sync(0xffffffffu, js, src);
      const float vz = __shfl_sync(0xffffffffu, jz, src + 1), vq = __shfl_sync(0xffffffffu, jr, src + 1);
      const float vs = __shfl_sync(0xffffffffu, js, src + 1);
      if (write) store_row<kh, vh>(pg, P, en.y, high, cb, kr, vr, kz, kq, ks, vz, vq, vs);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
  }
}

// 3-D tensor map over a bf16 [L * T][Hkv][128] array whose box is the 128
// channels of one KV head for 128 consecutive tokens.
cudaError_t make_tile_map(CUtensorMap *map, const void *base, int64_t tokens, int32_t Hkv) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(tokens)};
  const cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(Hkv) * 256};
  const cuuint32_t box[3] = {128, 1, kTileTokens};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

int pack_blocks_per_sm() { return 1; }

cudaError_t launch_pack(const CompactArgs &a, int grid, cudaStream_t s) {
  const int64_t tokens = static_cast<int64_t>(a.L) * a.T;
  if (tokens < 1) return cudaSuccess;  // nothing can survive
  alignas(64) CUtensorMap kmap, vmap;
  cudaError_t e = make_tile_map(&kmap, a.k, tokens, a.Hkv);
  if (e != cudaSuccess) return e;
  e = make_tile_map(&vmap, a.v, tokens, a.Hkv);
  if (e != cudaSuccess) return e;
  const int smem = static_cast<int>(kPackSmemBytes);
  void (*kern)(CompactArgs, const CUtensorMap, const CUtensorMap) =
      a.pg.vh == 2 ? k_pack<1> : (a.pg.kh == 4 ? k_pack<2> : k_pack<0>);
  static_assert(scheme_vh(1) == 2 && scheme_kh(2) == 4, "scheme dispatch");
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kPackThreads, smem, s>>>(a, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace dkv
