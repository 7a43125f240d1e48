// classify.cu -- request prefix sums and per-tile records (k_prep) and the
// significance reduce + three-tier classification (k_classify_rows for the
// common head shapes, k_classify otherwise).
//
// DiffKV (arXiv 2412.03131), Pith review: a token's significance is the
// average attention it receives from subsequent tokens, max-aggregated over
// the query heads that share its KV head; tokens at or above alpha_h/N are
// K8V4, between alpha_l/N and alpha_h/N K4V2, below alpha_l/N pruned ("What
// carries the argument"; Referee Report, major comment 2 on Algorithm 1).
//
// The average is sig_sum / sig_cnt rounded once in fp32.  Because rounding a
// quotient by a positive count is monotone, the maximum over the G query
// heads of the rounded quotients equals the rounded quotient of the maximum
// sum (and of the minimum sum for a negative count), so each (token, KV head)
// costs one IEEE division instead of G with bit-identical results.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kPrepThreads = 1024;
constexpr int kClassifyThreads = 256;

__global__ void __launch_bounds__(kPrepThreads) k_prep(CompactArgs a, int32_t npart) {
  __shared__ int64_t warp_tok[32];
  __shared__ int32_t warp_tile[32];
  __shared__ int64_t carry_tok;
  __shared__ int32_t carry_tile;
  __shared__ int32_t bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    carry_tok = 0;
    carry_tile = 0;
    bad = 0;
  }
  __syncthreads();
  for (int64_t base = 0; base < a.R; base += blockDim.x) {
    const int64_t r = base + tid;
    int64_t n = 0;
    if (r < a.R) {
      n = a.lens[r];
      if (n < 0 || n > a.max_len) bad = 1;
      if (n < 0) n = 0;
    }
    int32_t nt = static_cast<int32_t>((n + kTileTokens - 1) / kTileTokens);
    // inclusive warp scans
    int64_t it = n;
    int32_t il = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t xt = __shfl_up_sync(0xffffffffu, it, o);
      const int32_t xl = __shfl_up_sync(0xffffffffu, il, o);
      if (lane >= o) {
        it += xt;
        il += xl;
      }
    }
    if (lane == 31) {
      warp_tok[warp] = it;
      warp_tile[warp] = il;
    }
    __syncthreads();
    if (warp == 0) {
      const int nw = blockDim.x >> 5;
      int64_t wt = lane < nw ? warp_tok[lane] : 0;
      int32_t wl = lane < nw ? warp_tile[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t xt = __shfl_up_sync(0xffffffffu, wt, o);
        const int32_t xl = __shfl_up_sync(0xffffffffu, wl, o);
        if (lane >= o) {
          wt += xt;
          wl += xl;
        }
      }
      if (lane < nw) {
        warp_tok[lane] = wt;   // inclusive over warps
        warp_tile[lane] = wl;
      }
    }
    __syncthreads();
    const int64_t before_tok = carry_tok + (warp ? warp_tok[warp - 1] : 0);
    const int32_t before_tile = carry_tile + (warp ? warp_tile[warp - 1] : 0);
    if (r < a.R) {
      a.tok_off[r] = before_tok + it - n;
      a.tile_off[r] = before_tile + il - nt;
    }
    __syncthreads();
    if (tid == blockDim.x - 1) {
      carry_tok = before_tok + it;
      carry_tile = before_tile + il;
    }
    __syncthreads();
  }
  // every tile's record (bounded by the workspace's room), one thread per
  // tile: its request by bisection of the tile offsets written above, first
  // token, size, and the thresholds alpha / N, each an IEEE division
  {
    const int64_t room = a.T / kTileTokens + a.R;
    const int64_t ntiles = carry_tile < room ? carry_tile : room;
    for (int64_t x = tid; x < ntiles; x += blockDim.x) {
      int lo = 0, hi = a.R - 1;  // the last request whose first tile is <= x
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.tile_off[mid] <= x) lo = mid; else hi = mid - 1;
      }
      const int64_t tok0 = a.tok_off[lo];
      const int64_t n = static_cast<int64_t>(a.lens[lo]) < 0 ? 0 : a.lens[lo];
      const int64_t done = (x - a.tile_off[lo]) * kTileTokens;
      TileInfo ti;
      ti.t0 = tok0 + done;
      ti.cnt = static_cast<int32_t>(n - done < kTileTokens ? n - done : kTileTokens);
      ti.N = static_cast<int32_t>(n);
      ti.thr_h = __fdiv_rn(a.alpha_h, static_cast<float>(n));
      ti.thr_l = __fdiv_rn(a.alpha_l, static_cast<float>(n));
      ti.pad[0] = ti.pad[1] = 0;
      a.tile_info[x] = ti;
    }
  }
  if (tid == 0) {
    a.tok_off[a.R] = carry_tok;
    a.tile_off[a.R] = carry_tile;
    if (carry_tok != a.T) bad = 1;
    a.ws->err = bad ? DKV_E_LENS : 0;
    a.ws->ticket = 0;
    a.ws->TR = carry_tile;
    a.ws->npart = npart;
    a.ws->total = 0;
    a.ws->head = 0;
  }
  for (int32_t i = tid; i < npart; i += blockDim.x) a.part[i] = 0;
}

// One tile of a layer: where its scores start, how many tokens it holds and
// its request's thresholds.
struct ClassifyItem {
  int64_t l, t0;
  int32_t rt, cnt;
  float thr_h, thr_l;
};

__device__ __forceinline__ TileInfo load_tile_info(const TileInfo *p) {
  const int4 x = __ldg(reinterpret_cast<const int4 *>(p));
  const int4 y = __ldg(reinterpret_cast<const int4 *>(p) + 1);
  TileInfo t;
  t.t0 = static_cast<int64_t>((static_cast<uint64_t>(static_cast<uint32_t>(x.y)) << 32) | static_cast<uint32_t>(x.x));
  t.cnt = x.z;
  t.N = x.w;
  t.thr_h = __int_as_float(y.x);
  t.thr_l = __int_as_float(y.y);
  t.pad[0] = t.pad[1] = 0;
  return t;
}

__device__ __forceinline__ ClassifyItem classify_item(const CompactArgs &a, int64_t item, int32_t TR) {
  ClassifyItem it;
  it.l = item / TR;
  it.rt = static_cast<int32_t>(item - it.l * TR);
  const TileInfo ti = load_tile_info(a.tile_info + it.rt);
  it.t0 = ti.t0;
  it.cnt = ti.cnt;
  it.thr_h = ti.thr_h;
  it.thr_l = ti.thr_l;
  return it;
}

// The class of one (token, KV head) from m, the largest summed score over
// the head's query heads (the smallest when the count n is negative), and n
// (non-zero).  Reciprocal test: with rc the hardware reciprocal of n (within
// 1 ulp), y = RN(m * rc) is within 2^-22 (relative) of m / n, so
// y >= thr (1 + 2^-19) proves RN(m / n) >= thr and y <= thr (1 - 2^-19)
// proves RN(m / n) < thr (the margins, themselves rounded, stay far from
// 2^-22); in between, and for thresholds below 2^-100 where a tiny quotient
// could leave the relative bound, the IEEE division decides.  A NaN fails
// every test and goes to the division: pruned.
struct Thresholds {
  float thr_h, thr_l, hi_h, lo_h, hi_l, lo_l;
  bool exact_only;
};

__device__ __forceinline__ Thresholds thresholds(float thr_h, float thr_l) {
  Thresholds t;
  t.thr_h = thr_h;
  t.thr_l = thr_l;
  t.exact_only = !(thr_l >= 0x1p-100f);
  t.hi_h = __fmul_rn(thr_h, 1.0f + 0x1p-19f);
  t.lo_h = __fmul_rn(thr_h, 1.0f - 0x1p-19f);
  t.hi_l = __fmul_rn(thr_l, 1.0f + 0x1p-19f);
  t.lo_l = __fmul_rn(thr_l, 1.0f - 0x1p-19f);
  return t;
}

__device__ __forceinline__ int classify_score(float m, float cf, float rc, const Thresholds &t) {
  const float y = __fmul_rn(m, rc);
  if (!t.exact_only && y >= t.hi_h) return DKV_CLASS_K8V4;
  if (!t.exact_only && !(y > t.lo_h) && y >= t.hi_l) return DKV_CLASS_K4V2;
  if (!t.exact_only && !(y > t.lo_h) && !(y > t.lo_l)) return DKV_CLASS_PRUNE;
  const float s = __fdiv_rn(m, cf);
  return s >= t.thr_h ? DKV_CLASS_K8V4 : (s >= t.thr_l ? DKV_CLASS_K4V2 : DKV_CLASS_PRUNE);
}

// Scores held in registers for the next tile (the first kPre float4 per
// thread: every score of a tile when Hq <= 32), loaded while the current tile
// is classified.
constexpr int kPre = 4;

template <bool kVec>
__global__ void __launch_bounds__(kClassifyThreads) k_classify(CompactArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  float *sig_s = reinterpret_cast<float *>(smem);                     // [tile][Hq + 1]
  int32_t *cnt_s = reinterpret_cast<int32_t *>(sig_s + kTileTokens * (a.Hq + 1));  // [tile]
  uint8_t *cls_s = reinterpret_cast<uint8_t *>(cnt_s + kTileTokens);  // [tile][Hkv]
  if (a.ws->err != 0) return;
  const int32_t TR = a.ws->TR;
  const int64_t items = static_cast<int64_t>(a.L) * TR;
  const int tid = threadIdx.x;
  const int G = a.G;
  const int ld = a.Hq + 1;
  // (4 i) / Hq by a multiply: exact for 4 i < 2^32 / Hq (4 i <= 128 Hq here)
  const uint32_t inv_hq = static_cast<uint32_t>((0x100000000ull + a.Hq - 1) / a.Hq);

  float4 pre[kPre];
  int32_t pre_cnt = 0;
  auto prefetch = [&](const ClassifyItem &it) {
    const float4 *s4 = reinterpret_cast<const float4 *>(a.sig_sum + (it.l * a.T + it.t0) * a.Hq);
    const int nv = (it.cnt * a.Hq) >> 2;
#pragma unroll
    for (int q = 0; q < kPre; ++q) {
      const int i = tid + q * kClassifyThreads;
      pre[q] = i < nv ? __ldcs(s4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pre_cnt = tid < it.cnt ? __ldg(a.sig_cnt + it.t0 + tid) : 0;
  };

  int64_t item = blockIdx.x;
  ClassifyItem cur{};
  if (kVec && item < items) {
    cur = classify_item(a, item, TR);
    prefetch(cur);
  }
  for (; item < items; item += gridDim.x) {
    if (!kVec) cur = classify_item(a, item, TR);
    const int cnt = cur.cnt;
    const Thresholds thr = thresholds(cur.thr_h, cur.thr_l);

    // stage the tile's summed scores [cnt][Hq] into rows padded to Hq + 1
    // floats, so the per-token reads below hit 32 different banks
    const float *src = a.sig_sum + (cur.l * a.T + cur.t0) * a.Hq;
    const int nf = cnt * a.Hq;
    if (kVec) {
      const float4 *s4 = reinterpret_cast<const float4 *>(src);
      const int nv = nf >> 2;
#pragma unroll
      for (int q = 0; q < kPre; ++q) {
        const int i = tid + q * kClassifyThreads;
        if (i < nv) {
          const int k = static_cast<int>(__umulhi(static_cast<uint32_t>(4 * i), inv_hq));
          float *d = sig_s + k * ld + (4 * i - k * a.Hq);
          d[0] = pre[q].x;
          d[1] = pre[q].y;
          d[2] = pre[q].z;
          d[3] = pre[q].w;
        }
      }
      for (int i = tid + kPre * kClassifyThreads; i < nv; i += blockDim.x) {  // Hq > 32: the rest, now
        const float4 x = __ldcs(s4 + i);
        const int k = static_cast<int>(__umulhi(static_cast<uint32_t>(4 * i), inv_hq));
        float *d = sig_s + k * ld + (4 * i - k * a.Hq);
        d[0] = x.x;
        d[1] = x.y;
        d[2] = x.z;
        d[3] = x.w;
      }
      if (tid < cnt) cnt_s[tid] = pre_cnt;
    } else {
      for (int i = tid; i < nf; i += blockDim.x) {
        const int k = i / a.Hq;
        sig_s[k * ld + (i - k * a.Hq)] = __ldcs(src + i);
      }
      for (int i = tid; i < cnt; i += blockDim.x) cnt_s[i] = __ldg(a.sig_cnt + cur.t0 + i);
    }
    __syncthreads();
    // the next tile's scores are loaded while this one is classified
    const int64_t next = item + gridDim.x;
    ClassifyItem nxt{};
    if (kVec && next < items) {
      nxt = classify_item(a, next, TR);
      prefetch(nxt);
    }

    const int64_t tau0 = cur.l * a.Hkv * TR + cur.rt;  // unit tile of head 0
    for (int p = tid; p < a.Hkv * kTileTokens; p += blockDim.x) {
      const int h = p / kTileTokens;
      const int k = p % kTileTokens;
      int c = DKV_CLASS_PRUNE;
      if (k < cnt) {
        const int32_t n = cnt_s[k];
        if (n == 0) {
          c = DKV_CLASS_K8V4;  // not yet observed: keep at high precision
        } else {
          const float *row = sig_s + k * (a.Hq + 1) + h * G;
          float m = row[0];
          if (n > 0) {
            for (int g = 1; g < G; ++g) m = fmaxf(m, row[g]);
          } else {
            for (int g = 1; g < G; ++g) m = fminf(m, row[g]);
          }
          const float cf = static_cast<float>(n);
          float rc;
          asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rc) : "f"(cf));
          c = classify_score(m, cf, rc, thr);
        }
        cls_s[k * a.Hkv + h] = static_cast<uint8_t>(c);
      }
      const uint32_t hi = __ballot_sync(0xffffffffu, c == DKV_CLASS_K8V4);
      const uint32_t lo = __ballot_sync(0xffffffffu, c == DKV_CLASS_K4V2);
      if ((tid & 31) == 0) {
        uint32_t *m = a.mask + (tau0 + static_cast<int64_t>(h) * TR) * (2 * kMaskWords);
        m[k >> 5] = hi;
        m[kMaskWords + (k >> 5)] = lo;
      }
    }
    __syncthreads();
    uint8_t *dst = a.classes + (cur.l * a.T + cur.t0) * a.Hkv;
    const int nb = cnt * a.Hkv;
    if ((reinterpret_cast<uintptr_t>(dst) & 3) == 0) {  // whole words, then the tail
      for (int b = tid; b < (nb >> 2); b += blockDim.x)
        reinterpret_cast<uint32_t *>(dst)[b] = reinterpret_cast<const uint32_t *>(cls_s)[b];
      for (int b = (nb & ~3) + tid; b < nb; b += blockDim.x) dst[b] = cls_s[b];
    } else {
      for (int b = tid; b < nb; b += blockDim.x) dst[b] = cls_s[b];
    }
    __syncthreads();
    cur = nxt;
  }
}

// The same classification with one thread per token, for the head shapes of
// common models (Hq and G known at compile time).  A warp takes 32
// consecutive tokens of one tile (a quarter), so one ballot per KV head is
// one word of that unit tile's class mask, and streams its quarters through
// a private ring of kRowStages shared-memory buffers: one lane starts a bulk
// asynchronous copy of the quarter's summed scores (32 contiguous rows of Hq
// floats) that completes on the stage's mbarrier, kRowStages quarters ahead
// of their use.  Each lane then reads its own token's row from shared memory,
// reduces it per KV head, classifies, and stores the token's Hkv class bytes
// as words.  Rows of 8 or 16 float4 chunks would put a warp's reads of one
// chunk in one bank group, so those lanes take the KV heads in a rotated
// order (lane i starts at head i).

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

constexpr int kRowWarps = kClassifyThreads / 32;
constexpr int64_t kRowWaitLimit = 1ll << 24;  // polls of one mbarrier before giving up

__host__ __device__ constexpr int row_stages(int hq) { return kRowWarps * 3 * 128 * hq <= 100 * 1024 ? 3 : 2; }
__host__ __device__ constexpr size_t rows_smem(int hq) {
  return static_cast<size_t>(kRowWarps) * row_stages(hq) * (128 * hq + sizeof(uint64_t) + sizeof(TileInfo));
}

__device__ __forceinline__ bool row_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  for (int64_t i = 0; i < kRowWaitLimit; ++i) {
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

template <int HQ, int G>
__global__ void __launch_bounds__(kClassifyThreads) k_classify_rows(CompactArgs a) {
  constexpr int HKV = HQ / G, NV = HQ / 4, NW = (HKV + 3) / 4, S = row_stages(HQ);
  constexpr bool kRotate = NV % 8 == 0 && G % 4 == 0 && (HKV & (HKV - 1)) == 0;
  static_assert(HQ % 4 == 0 && HQ % G == 0, "rows of whole 16-byte chunks, whole KV heads");
  static_assert(HKV <= 16, "the 2-bit classes of every KV head in one word");
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *buf = reinterpret_cast<float *>(smem) + static_cast<size_t>(warp) * S * 32 * HQ;  // [S][32][HQ]
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(kRowWarps) * S * 128 * HQ) + warp * S;
  TileInfo *tinf = reinterpret_cast<TileInfo *>(smem + static_cast<size_t>(kRowWarps) * S * (128 * HQ + 8)) +
                   warp * S;
  if (a.ws->err != 0) return;
  if (lane == 0) {
    for (int st = 0; st < S; ++st)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bars + st)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  const int32_t TR = a.ws->TR;
  const int64_t items = static_cast<int64_t>(a.L) * TR * kMaskWords;  // (layer, tile, quarter)
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kRowWarps;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kRowWarps + warp;
  const int64_t nmine = first < items ? (items - first + nw - 1) / nw : 0;
  if (nmine == 0) return;
  // The warp's items first, first + nw, ... as (layer, tile quarter) pairs,
  // stepped without a division per item: three cursors (the quarter in use,
  // the next to copy, the one after it, whose tile record is loaded early).
  const int32_t nq = TR * kMaskWords;  // quarters per layer
  const int64_t dl = nw / nq;
  const int32_t dq = static_cast<int32_t>(nw - dl * nq);
  struct Cursor {
    int64_t l;
    int32_t tq;  // rt * kMaskWords + q
  };
  auto step = [&](Cursor &c) {
    c.l += dl;
    c.tq += dq;
    if (c.tq >= nq) {
      c.tq -= nq;
      ++c.l;
    }
  };
  Cursor use{first / nq, static_cast<int32_t>(first % nq)};
  Cursor put = use, ahead_c = use;
  // quarter c of this warp into stage st: lane 0 records its tile and starts
  // the copy (a bare arrive when the quarter lies past the tile's end); every
  // lane loads its token's count
  int32_t cn[S];
  auto issue = [&](const Cursor &c, int st, const TileInfo &ti) -> int32_t {
    const int q = c.tq % kMaskWords;
    const int nvalid = min(max(ti.cnt - 32 * q, 0), 32);
    if (lane == 0) {
      tinf[st] = ti;
      const uint32_t b = smem_u32(bars + st);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      if (nvalid > 0) {
        const uint32_t bytes = static_cast<uint32_t>(nvalid) * HQ * 4u;
        const float *src = a.sig_sum + (c.l * a.T + ti.t0 + 32 * q) * HQ;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         smem_u32(buf + static_cast<size_t>(st) * 32 * HQ)),
                     "l"(src), "r"(bytes), "r"(b)
                     : "memory");
      } else {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
      }
    }
    return lane < nvalid ? __ldg(a.sig_cnt + ti.t0 + 32 * q + lane) : 0;
  };
#pragma unroll
  for (int st = 0; st < S; ++st) {
    cn[st] = 0;
    if (st < nmine) {
      cn[st] = issue(put, st, load_tile_info(a.tile_info + put.tq / kMaskWords));
      step(put);
    }
  }
  ahead_c = put;
  TileInfo ahead = S < nmine ? load_tile_info(a.tile_info + ahead_c.tq / kMaskWords) : TileInfo{};
  __syncwarp();

  const bool words = HKV % 4 == 0 && (reinterpret_cast<uintptr_t>(a.classes) & 3) == 0;
  int64_t m = 0;
  bool ok = true;
  for (; m < nmine; ++m) {
    const int st = static_cast<int>(m % S);
    if (!__all_sync(0xffffffffu, row_wait(bars + st, static_cast<uint32_t>((m / S) & 1)))) {
      ok = false;
      break;
    }
    const int64_t l = use.l;
    const int q = use.tq % kMaskWords;
    const int32_t rt = use.tq / kMaskWords;
    step(use);
    const TileInfo ti = tinf[st];
    const int32_t n = cn[0];
#pragma unroll
    for (int i = 0; i + 1 < S; ++i) cn[i] = cn[i + 1];
    const int k = 32 * q + lane;
    const bool valid = k < ti.cnt;
    const Thresholds thr = thresholds(ti.thr_h, ti.thr_l);
    const float cf = static_cast<float>(n);
    float rc;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rc) : "f"(cf));
    const float *rowp = buf + static_cast<size_t>(st) * 32 * HQ + lane * HQ;
    auto classify_head = [&](const float *v) -> int {
      if (n == 0) return DKV_CLASS_K8V4;  // not yet observed: keep at high precision
      float mx = v[0];
      if (n > 0) {
#pragma unroll
        for (int g = 1; g < G; ++g) mx = fmaxf(mx, v[g]);
      } else {
#pragma unroll
        for (int g = 1; g < G; ++g) mx = fminf(mx, v[g]);
      }
      return classify_score(mx, cf, rc, thr);
    };
    uint32_t cls2 = 0;  // 2-bit class of every KV head
    if (valid) {
      if (kRotate) {
#pragma unroll
        for (int s = 0; s < HKV; ++s) {
          const int hh = (s + lane) & (HKV - 1);
          float v[G];
#pragma unroll
          for (int j = 0; j < G / 4; ++j) {
            const float4 x4 = reinterpret_cast<const float4 *>(rowp + hh * G)[j];
            v[4 * j] = x4.x;
            v[4 * j + 1] = x4.y;
            v[4 * j + 2] = x4.z;
            v[4 * j + 3] = x4.w;
          }
          cls2 |= static_cast<uint32_t>(classify_head(v)) << (2 * hh);
        }
      } else {
        float x[HQ];
#pragma unroll
        for (int j = 0; j < NV; ++j) {
          const float4 x4 = reinterpret_cast<const float4 *>(rowp)[j];
          x[4 * j] = x4.x;
          x[4 * j + 1] = x4.y;
          x[4 * j + 2] = x4.z;
          x[4 * j + 3] = x4.w;
        }
#pragma unroll
        for (int h = 0; h < HKV; ++h) cls2 |= static_cast<uint32_t>(classify_head(x + h * G)) << (2 * h);
      }
    }
    __syncwarp();  // every lane is done with the stage: refill it
    if (m + S < nmine) {
      cn[S - 1] = issue(put, st, ahead);
      step(put);
      step(ahead_c);
      if (m + S + 1 < nmine) ahead = load_tile_info(a.tile_info + ahead_c.tq / kMaskWords);
    }
    uint32_t mh = 0, ml = 0;  // lane h < HKV: word q of head h's masks
    uint32_t cw[NW];
#pragma unroll
    for (int w = 0; w < NW; ++w) cw[w] = 0;
#pragma unroll
    for (int h = 0; h < HKV; ++h) {
      const uint32_t c = (cls2 >> (2 * h)) & 3u;  // PRUNE (0) for the lanes past the tile's end
      const uint32_t hi = __ballot_sync(0xffffffffu, c == DKV_CLASS_K8V4);
      const uint32_t lo = __ballot_sync(0xffffffffu, c == DKV_CLASS_K4V2);
      if (lane == h) {
        mh = hi;
        ml = lo;
      }
      cw[h / 4] |= c << (8 * (h % 4));
    }
    if (lane < HKV) {
      uint32_t *mk = a.mask + ((l * HKV + lane) * TR + rt) * (2 * kMaskWords);
      mk[q] = mh;
      mk[kMaskWords + q] = ml;
    }
    if (valid) {
      uint8_t *dst = a.classes + (l * a.T + ti.t0 + k) * HKV;
      if (words && NW == 2 && (reinterpret_cast<uintptr_t>(a.classes) & 7) == 0) {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(cw[0], cw[NW - 1]);
      } else if (words) {
#pragma unroll
        for (int w = 0; w < NW; ++w) reinterpret_cast<uint32_t *>(dst)[w] = cw[w];
      } else {
#pragma unroll
        for (int h = 0; h < HKV; ++h) dst[h] = static_cast<uint8_t>(cw[h / 4] >> (8 * (h % 4)));
      }
    }
  }
  if (!ok) {  // a copy never completed: record it, wait (bounded) for the ones in flight, stop
    if (lane == 0) set_error(&a.ws->err, DKV_E_TIMEOUT);
    for (int64_t r = m; r < min(nmine, m + S); ++r) row_wait(bars + r % S, static_cast<uint32_t>((r / S) & 1));
  }
}

template <int HQ, int G>
cudaError_t launch_rows(const CompactArgs &a, int sms, cudaStream_t s) {
  static std::atomic<int> bps{0};  // resident blocks per SM, queried once
  constexpr size_t smem = rows_smem(HQ);
  if (bps.load() == 0) {
    cudaError_t e = cudaFuncSetAttribute(k_classify_rows<HQ, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_classify_rows<HQ, G>, kClassifyThreads, smem);
    if (e != cudaSuccess) return e;
    bps.store(n > 0 ? n : 1);
  }
  const int64_t items = static_cast<int64_t>(a.L) * (a.T / kTileTokens + a.R) * kMaskWords;
  const int64_t want = (items + kRowWarps - 1) / kRowWarps;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(sms) * bps.load())));
  k_classify_rows<HQ, G><<<grid, kClassifyThreads, smem, s>>>(a);
  return cudaGetLastError();
}

size_t classify_smem(int Hq, int Hkv) {
  return sizeof(float) * kTileTokens * (Hq + 1) + sizeof(int32_t) * kTileTokens + kTileTokens * Hkv;
}

}  // namespace

cudaError_t launch_prep(const CompactArgs &a, cudaStream_t s) {
  const int32_t npart = static_cast<int32_t>((a.U + kScanUnits - 1) / kScanUnits);
  k_prep<<<1, kPrepThreads, 0, s>>>(a, npart);
  return cudaGetLastError();
}

cudaError_t launch_classify(const CompactArgs &a, int grid, int sms, cudaStream_t s) {
  // the head shapes with a per-token kernel: (Hq, G) of Llama-3 8B / 70B,
  // Qwen2.5 7B / 32B, and a small grouped shape
  const int hq = a.Hq, g = a.G;
  if (hq == 32 && g == 4) return launch_rows<32, 4>(a, sms, s);
  if (hq == 64 && g == 8) return launch_rows<64, 8>(a, sms, s);
  if (hq == 28 && g == 7) return launch_rows<28, 7>(a, sms, s);
  if (hq == 40 && g == 5) return launch_rows<40, 5>(a, sms, s);
  if (hq == 12 && g == 4) return launch_rows<12, 4>(a, sms, s);
  {
    const size_t smem = classify_smem(a.Hq, a.Hkv);
    const bool vec = (a.Hq % 4) == 0;
    if (smem > 48 * 1024) {
      const int limit = static_cast<int>(smem);
      cudaError_t e = vec ? cudaFuncSetAttribute(k_classify<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit)
                          : cudaFuncSetAttribute(k_classify<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
      if (e != cudaSuccess) return e;
    }
    if (vec) k_classify<true><<<grid, kClassifyThreads, smem, s>>>(a);
    else k_classify<false><<<grid, kClassifyThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace dkv
