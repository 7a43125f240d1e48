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
// y = RN(d * RN(1/s) + 1536) with one fused multiply-add.  y lies in
// [1024, 2048), so it carries the quotient in fixed point with 13 fraction
// bits: w = bits(y) - bits(1536).  The error of w * 2^-13 against RN(d / s)
// is below 0.75 * 2^-13 (quotient <= 256: 2^-24 relative for the reciprocal,
// half an ulp of y, 2^-24 relative for the reference's own rounding), so
// (w + 4096) >> 13 equals the round-to-nearest-even code unless
// w + 4096 is a multiple of 2^13 exactly -- only then can the quotient sit on
// a tie or on the other side of one.  Those elements, and rows whose end
// points would need clamping (checked exactly per row), are recomputed with
// the IEEE division.  Codes are therefore bit-identical to the definition.
//
// Work layout.  A block takes unit tiles (128 tokens of one (layer, request,
// KV head)) in a grid-stride loop.  From the tile's two class bitmasks it
// lists the surviving rows, K8V4 first, with their page id and slot (ranks
// come from popcounts plus the tile's rank bases from the scan), so pruned
// rows are never read and most warps see a single class.  A warp takes 16
// list entries: 4 groups of 8 lanes, each group 4 rows, each lane 16 channels
// (two 128-bit loads per tensor).  Row min / max are bf16x2 min / max
// (NaN-propagating) reduced over the 8 lanes; the per-row scalar work (scale,
// zero, reciprocal, end-point check, metadata store) is spread one job per
// lane; codes are packed in registers and stored 4-16 bytes per lane, so the
// four groups of a warp write neighbouring slots of a page.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kPackThreads = 256;
constexpr int kPackWarps = kPackThreads / 32;
constexpr int kRowsPerWarp = 16;
static_assert(kPackWarps * kRowsPerWarp == kTileTokens, "one warp pass per tile");

constexpr float kMagic = 1536.0f;           // 1.5 * 2^10: y in [1024, 2048), ulp 2^-13
constexpr uint32_t kMagicBits = 0x44C00000u;  // bits of 1536.0f
constexpr uint32_t kBias = 4096u - kMagicBits;  // v = w + 4096 (mod 2^32)

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

// Min and max over 16 bf16 channels (8 words), reduced over the 8 lanes of a
// group.  Returns the pair packed as bf16x2 {min, -max}.
__device__ __forceinline__ uint32_t row_minmax(const uint4 &a, const uint4 &b) {
  uint32_t mn = bmin2(bmin2(bmin2(a.x, a.y), bmin2(a.z, a.w)), bmin2(bmin2(b.x, b.y), bmin2(b.z, b.w)));
  uint32_t mx = bmax2(bmax2(bmax2(a.x, a.y), bmax2(a.z, a.w)), bmax2(bmax2(b.x, b.y), bmax2(b.z, b.w)));
  // {min(lo, hi) of mn, min(lo, hi) of -mx}: pair (mn.lo, -mx.lo) vs (mn.hi, -mx.hi)
  const uint32_t p0 = __byte_perm(mn, mx, 0x5410) ^ 0x80000000u;  // {mn.lo, -mx.lo}
  const uint32_t p1 = __byte_perm(mn, mx, 0x7632) ^ 0x80000000u;  // {mn.hi, -mx.hi}
  uint32_t p = bmin2(p0, p1);
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) p = bmin2(p, __shfl_xor_sync(0xffffffffu, p, o));
  return p;
}

// Fast code of one element (see the file header); `zero` accumulates the
// minimum of the low 13 bits, 0 flags a possible tie.
__device__ __forceinline__ uint32_t fast_code(float x, float z, float r, uint32_t &flag) {
  const float d = __fsub_rn(x, z);
  const float y = __fmaf_rn(d, r, kMagic);
  const uint32_t v = __float_as_uint(y) + kBias;
  flag = min(flag, v & 8191u);
  return v >> 13;
}

__device__ __forceinline__ uint32_t exact_code(float x, float z, float s, float n) {
  const float t = __fdiv_rn(__fsub_rn(x, z), s);
  const float q = fminf(fmaxf(rintf(t), 0.0f), n);
  return static_cast<uint32_t>(q);
}

// Codes of 16 channels held as 8 bf16x2 words.
struct Codes16 {
  uint32_t c[16];
};

__device__ __forceinline__ void quant16(const uint4 &a, const uint4 &b, float z, float r, float s, float n,
                                        Codes16 &q) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t flag = 0xffffffffu;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    q.c[2 * i] = fast_code(bf_lo(w[i]), z, r, flag);
    q.c[2 * i + 1] = fast_code(bf_hi(w[i]), z, r, flag);
  }
  if (flag == 0u || r < 0.0f) {  // rare: a possible tie, or a row that needs clamping
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float x = (i & 1) ? bf_hi(w[i >> 1]) : bf_lo(w[i >> 1]);
      const float y = __fmaf_rn(__fsub_rn(x, z), r, kMagic);
      if (r < 0.0f || ((__float_as_uint(y) + kBias) & 8191u) == 0u) q.c[i] = exact_code(x, z, s, n);
    }
  }
}

// Pack 16 codes of `bits` bits, lowest channel in the lowest bits.
__device__ __forceinline__ uint32_t pack_word(const Codes16 &q, int first, int count, int bits) {
  uint32_t w = 0;
#pragma unroll
  for (int i = count - 1; i >= 0; --i) w = (w << bits) | q.c[first + i];
  return w;
}

__device__ __forceinline__ void fill_words(uint8_t *p, int64_t nwords, uint32_t value, int tid) {
  uint32_t *w = reinterpret_cast<uint32_t *>(p);
  for (int64_t i = tid; i < nwords; i += kPackThreads) w[i] = value;
}

__global__ void __launch_bounds__(kPackThreads, 2) k_pack(CompactArgs a) {
  __shared__ int32_t ent_tok[kTileTokens];
  __shared__ int32_t ent_page[kTileTokens];
  __shared__ int32_t ent_slot[kTileTokens];
  if (a.ws->err != 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane >> 3, l8 = lane & 7;
  const int32_t TR = a.ws->TR;
  const int64_t head_mod = a.ws->head_mod;
  const int64_t per_layer = static_cast<int64_t>(TR) * a.Hkv;
  const int64_t ntiles = per_layer * a.L;
  const int64_t P = a.P;
  const int64_t page_bytes = 216 * P;

  for (int64_t tau = blockIdx.x; tau < ntiles; tau += gridDim.x) {
    // ---- which unit tile
    const int64_t l = tau / per_layer;
    const int64_t rem = tau - l * per_layer;
    const int r = find_segment(a.tile_off, a.R + 1, rem, a.Hkv);
    const int32_t tr0 = __ldg(a.tile_off + r);
    const int32_t nt = __ldg(a.tile_off + r + 1) - tr0;
    const int32_t q = static_cast<int32_t>(rem - static_cast<int64_t>(tr0) * a.Hkv);
    const int32_t h = q / nt;
    const int32_t j = q - h * nt;
    const int64_t u = (l * a.R + r) * a.Hkv + h;
    const int64_t t0 = __ldg(a.tok_off + r) + static_cast<int64_t>(j) * kTileTokens;

    const uint4 *mp = reinterpret_cast<const uint4 *>(a.mask + tau * (2 * kMaskWords));
    const uint4 hm = mp[0], lm = mp[1];
    const int2 base = a.base[tau];
    const UnitInfo inf = a.unit[u];
    const uint32_t hw[4] = {hm.x, hm.y, hm.z, hm.w};
    const uint32_t lw[4] = {lm.x, lm.y, lm.z, lm.w};
    const int nh_t = __popc(hw[0]) + __popc(hw[1]) + __popc(hw[2]) + __popc(hw[3]);
    const int nl_t = __popc(lw[0]) + __popc(lw[1]) + __popc(lw[2]) + __popc(lw[3]);
    const int nsurv = nh_t + nl_t;
    int64_t ring = head_mod + inf.off;
    if (ring >= a.F) ring -= a.F;

    // ---- list the surviving rows: K8V4 first, each with page id and slot
    if (tid < kTileTokens) {
      const int k = tid, wi = k >> 5;
      const uint32_t below = (1u << (k & 31)) - 1u;
      int rh = __popc(hw[wi] & below), rl = __popc(lw[wi] & below);
#pragma unroll
      for (int x = 0; x < 4; ++x)
        if (x < wi) {
          rh += __popc(hw[x]);
          rl += __popc(lw[x]);
        }
      const bool is_hi = (hw[wi] >> (k & 31)) & 1u;
      const bool is_lo = (lw[wi] >> (k & 31)) & 1u;
      if (is_hi || is_lo) {
        int e;
        int64_t pidx, slot;
        if (is_hi) {
          e = rh;
          const int64_t rho = base.x + rh;
          pidx = rho / P;
          slot = rho - pidx * P;
        } else {
          e = nh_t + rl;
          const int64_t rho = base.y + rl;
          const int64_t pl = rho / (2 * P);
          pidx = inf.p_hi + pl;
          slot = rho - pl * 2 * P;
        }
        int64_t idx = ring + pidx;
        if (idx >= a.F) idx -= a.F;
        int32_t id = a.free_list[idx];
        if (id < 0 || id >= a.F) {
          set_error(&a.ws->err, DKV_E_INTERNAL);
          id = -1;
        }
        ent_tok[e] = k;
        ent_page[e] = id;
        ent_slot[e] = static_cast<int32_t>(slot);
      }
    }
    __syncthreads();

    // ---- quantise + pack + scatter: warp `warp` takes entries [16 warp, 16 warp + 16)
    const int e0 = warp * kRowsPerWarp;
    if (e0 < nsurv) {
      uint4 kr[4][2], vr[4][2];
      const uint16_t *kbase = a.k + ((l * a.T + t0) * a.Hkv + h) * 128 + 16 * l8;
      const uint16_t *vbase = a.v + ((l * a.T + t0) * a.Hkv + h) * 128 + 16 * l8;
      const int64_t tok_stride = static_cast<int64_t>(a.Hkv) * 128;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = e0 + grp + 4 * i;
        if (e < nsurv) {
          const int64_t off = ent_tok[e] * tok_stride;
          const uint4 *kp = reinterpret_cast<const uint4 *>(kbase + off);
          const uint4 *vp = reinterpret_cast<const uint4 *>(vbase + off);
          kr[i][0] = __ldcs(kp);
          kr[i][1] = __ldcs(kp + 1);
          vr[i][0] = __ldcs(vp);
          vr[i][1] = __ldcs(vp + 1);
        } else {
          kr[i][0] = kr[i][1] = vr[i][0] = vr[i][1] = make_uint4(0, 0, 0, 0);
        }
      }
      // row min / max per (row, tensor), reduced over the 8 lanes of the group
      uint32_t mm[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        mm[2 * i] = row_minmax(kr[i][0], kr[i][1]);
        mm[2 * i + 1] = row_minmax(vr[i][0], vr[i][1]);
      }
      // one scalar job per lane: row l8 >> 1, tensor l8 & 1
      uint32_t mine = mm[0];
#pragma unroll
      for (int x = 1; x < 8; ++x) mine = (l8 == x) ? mm[x] : mine;
      const int ji = l8 >> 1, jt = l8 & 1;
      const int ej = e0 + grp + 4 * ji;
      const bool jvalid = ej < nsurv;
      const bool jhigh = ej < nh_t;
      const int bits = jt == 0 ? (jhigh ? 8 : 4) : (jhigh ? 4 : 2);
      const float nmax = static_cast<float>((1 << bits) - 1);
      // a zero extreme is +0 (min / max leave the sign of a zero open)
      const float mn = __fadd_rn(bf_lo(mine), 0.0f);
      const float mx = __fadd_rn(-bf_hi(mine), 0.0f);
      if (jvalid && !(fabsf(mn) <= 65504.0f && fabsf(mx) <= 65504.0f)) set_error(&a.ws->err, DKV_E_RANGE);
      const float s32 = __fdiv_rn(__fsub_rn(mx, mn), nmax);
      __half hs = __float2half_rn(s32);
      if (mx > mn && __half_as_ushort(hs) == 0) hs = __ushort_as_half(1);  // 2^-24
      const __half hz = __float2half_rn(mn);
      const float js = __half2float(hs);
      const float jz = __half2float(hz);
      float jr = 0.0f;
      if (js != 0.0f) {
        jr = __frcp_rn(js);
        const float qlo = rintf(__fdiv_rn(__fsub_rn(mn, jz), js));
        const float qhi = rintf(__fdiv_rn(__fsub_rn(mx, jz), js));
        if (!(qlo >= 0.0f && qhi <= nmax)) jr = -1.0f;  // row needs clamping: exact path
      }
      if (jvalid) {
        const int32_t pid = ent_page[ej];
        if (pid >= 0) {
          uint8_t *pg = a.pages + pid * page_bytes;
          const int64_t slot = ent_slot[ej];
          const uint32_t meta = static_cast<uint32_t>(__half_as_ushort(hs)) |
                                (static_cast<uint32_t>(__half_as_ushort(hz)) << 16);
          *reinterpret_cast<uint32_t *>(pg + 192 * P + 8 * slot + 4 * jt) = meta;
          if (jt == 0)
            *reinterpret_cast<int32_t *>(pg + 208 * P + 4 * slot) = j * kTileTokens + ent_tok[ej];
        }
      }
      // codes, row by row
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int src = (grp << 3) + 2 * i;
        const float kz = __shfl_sync(0xffffffffu, jz, src);
        const float kq = __shfl_sync(0xffffffffu, jr, src);
        const float ks = __shfl_sync(0xffffffffu, js, src);
        const float vz = __shfl_sync(0xffffffffu, jz, src + 1);
        const float vq = __shfl_sync(0xffffffffu, jr, src + 1);
        const float vs = __shfl_sync(0xffffffffu, js, src + 1);
        const int e = e0 + grp + 4 * i;
        if (e >= nsurv) continue;
        const int32_t pid = ent_page[e];
        if (pid < 0) continue;
        const int64_t slot = ent_slot[e];
        uint8_t *pg = a.pages + pid * page_bytes;
        const bool high = e < nh_t;
        Codes16 ck, cv;
        if (high) {
          quant16(kr[i][0], kr[i][1], kz, kq, ks, 255.0f, ck);
          quant16(vr[i][0], vr[i][1], vz, vq, vs, 15.0f, cv);
          const uint4 kw = make_uint4(pack_word(ck, 0, 4, 8), pack_word(ck, 4, 4, 8), pack_word(ck, 8, 4, 8),
                                      pack_word(ck, 12, 4, 8));
          const uint2 vw = make_uint2(pack_word(cv, 0, 8, 4), pack_word(cv, 8, 8, 4));
          *reinterpret_cast<uint4 *>(pg + slot * 128 + 16 * l8) = kw;
          *reinterpret_cast<uint2 *>(pg + 128 * P + slot * 64 + 8 * l8) = vw;
        } else {
          quant16(kr[i][0], kr[i][1], kz, kq, ks, 15.0f, ck);
          quant16(vr[i][0], vr[i][1], vz, vq, vs, 3.0f, cv);
          const uint2 kw = make_uint2(pack_word(ck, 0, 8, 4), pack_word(ck, 8, 8, 4));
          const uint32_t vw = pack_word(cv, 0, 16, 2);
          *reinterpret_cast<uint2 *>(pg + slot * 64 + 8 * l8) = kw;
          *reinterpret_cast<uint32_t *>(pg + 128 * P + slot * 32 + 4 * l8) = vw;
        }
      }
    }

    // ---- unused slots.  (a) every K8V4 page whose slot 0 is in this tile:
    // metadata and positions of slots P..2P-1 (the page has no such slots).
    {
      const int64_t first = (base.x + P - 1) / P;         // first page starting at rank >= base.x
      const int64_t last = (base.x + nh_t - 1) / P;       // page of the last rank in the tile
      const int64_t npages = (nh_t > 0 && last >= first) ? last - first + 1 : 0;
      const int64_t per_page = 3 * P;                      // 2P words of metadata, P of positions
      for (int64_t w = tid; w < npages * per_page; w += kPackThreads) {
        const int64_t pk = first + w / per_page;
        const int64_t ww = w % per_page;
        const int32_t pid = ent_page[pk * P - base.x];
        if (pid < 0) continue;
        uint8_t *pg = a.pages + pid * page_bytes;
        if (ww < 2 * P) reinterpret_cast<uint32_t *>(pg + 200 * P)[ww] = 0u;
        else reinterpret_cast<int32_t *>(pg + 212 * P)[ww - 2 * P] = -1;
      }
    }
    // (b) tail of the unit's last K8V4 page, (c) tail of its last K4V2 page
    if (nh_t > 0 && base.x + nh_t == inf.n_hi && (inf.n_hi % P) != 0) {
      const int32_t pid = ent_page[nh_t - 1];
      if (pid >= 0) {
        uint8_t *pg = a.pages + pid * page_bytes;
        const int64_t s0 = inf.n_hi % P;
        fill_words(pg + 128 * s0, 32 * (P - s0), 0u, tid);
        fill_words(pg + 128 * P + 64 * s0, 16 * (P - s0), 0u, tid);
        fill_words(pg + 192 * P + 8 * s0, 2 * (P - s0), 0u, tid);
        fill_words(pg + 208 * P + 4 * s0, P - s0, 0xffffffffu, tid);
      }
    }
    if (nl_t > 0 && base.y + nl_t == inf.n_lo && (inf.n_lo % (2 * P)) != 0) {
      const int32_t pid = ent_page[nsurv - 1];
      if (pid >= 0) {
        uint8_t *pg = a.pages + pid * page_bytes;
        const int64_t s0 = inf.n_lo % (2 * P);
        fill_words(pg + 64 * s0, 16 * (2 * P - s0), 0u, tid);
        fill_words(pg + 128 * P + 32 * s0, 8 * (2 * P - s0), 0u, tid);
        fill_words(pg + 192 * P + 8 * s0, 2 * (2 * P - s0), 0u, tid);
        fill_words(pg + 208 * P + 4 * s0, 2 * P - s0, 0xffffffffu, tid);
      }
    }
    __syncthreads();
  }
}

}  // namespace

int pack_blocks_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_pack, kPackThreads, 0) != cudaSuccess || n < 1) n = 1;
  return n;
}

cudaError_t launch_pack(const CompactArgs &a, int grid, cudaStream_t s) {
  k_pack<<<grid, kPackThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dkv
