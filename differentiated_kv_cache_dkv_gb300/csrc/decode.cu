// decode.cu -- one generation step on the unified pages (dkv_decode_step) and
// the per-position index it keeps (dkv_decode_index).
//
// DiffKV (arXiv 2412.03131), Pith review: tokens are K8V4, K4V2 or pruned by
// their significance against alpha_h/N and alpha_l/N ("What carries the
// argument", "Core claim"); in the generation phase tokens are classified as
// they age and demotion and pruning are irreversible (Referee Report, major
// comment 2 on Section 4 / Algorithm 1); pages come from a circular free page
// list through a parallel prefix sum and are tracked by a bidirectional page
// table ("What carries the argument").
//
// Step semantics (with N = ctx + new for a request):
//   - every live token's class becomes min(old, classify(score, N)); the new
//     token is classified;
//   - per unit (layer, request, KV head) each list (K8V4 slots, K4V2 slots)
//     drops its removed tokens; the survivors in slots >= the survivor count
//     move, ascending, into the holes below it, ascending (bytes copied);
//   - tokens demoted K8V4 -> K4V2 are requantised (4-bit K, 2-bit V) from
//     their dequantised fp32 values and appended to the K4V2 list in
//     ascending position order; then the new token is appended to its list;
//   - a list keeps its first min(have, need) pages, need = ceil(n / capacity);
//     new pages come from the free-list head by an exclusive scan over units
//     (a unit's new K8V4 pages first); surplus pages are freed to the tail in
//     (unit, list, page) order; unused slots are cleared.
//
// With a recent window W (the review's Algorithm 1) held tokens at positions
// >= N - W keep their class and the new token enters as K8V4 (W >= 1); in the
// single-candidate mode only the token leaving the window, position ctx - W,
// is classified, instead of every older held token.
//
// Kernels, in stream order (after a memset of the call's counters):
//   k_reclass  streams sig_sum / sig_cnt, reclassifies every live row and
//              marks each changed class byte in place (0x80 | old << 2 | new;
//              old = 3 for the new token) -- the step's only full pass over
//              the significance sums, which dominate its bytes (in the
//              single-candidate mode k_candidate does the same for the
//              candidate and new rows alone);
//   k_dscan    per-unit plan (survivors, page needs, new and freed pages),
//              block scan + decoupled look-back over partitions of units,
//              capacity check;
//   k_apply    one block per (layer, request, head group): turns the marks
//              into final classes (or reverts them if the call failed),
//              builds per-unit bitmaps of removed slots and demoted
//              positions in shared memory, then one warp per unit clears new
//              pages, hole-fills, requantises, appends, clears vacated slots
//              and rewrites its tables.
// All waits are bounded (look-back polls by spin_limit); nothing traps.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kReclassThreads = 512;
constexpr int kReclassRows = 2;           // rows in flight per thread (4 blocks of 512 per SM)
constexpr int kCandThreads = 64;          // candidate kernel: 2 Hkv rows per (layer, request)
constexpr int kDScanThreads = 256;        // one unit per thread
constexpr int kMarkCap = 256;             // listed marks per unit in the apply block

__device__ __forceinline__ void st_release(uint64_t *p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_acquire(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int32_t cdiv(int32_t a, int32_t b) { return (a + b - 1) / b; }

// |x| > 65504 or non-finite for a bf16 bit pattern: bf16 0x477f is 65280, the
// largest value not above 65504, and 0x4780 (65536) the next.
__device__ __forceinline__ bool bf16_out_of_range(uint32_t h) { return (h & 0x7fffu) >= 0x4780u; }

__device__ __forceinline__ bool words_out_of_range(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) bad |= bf16_out_of_range(w[i] & 0xffffu) | bf16_out_of_range(w[i] >> 16);
  return bad;
}

// ---------------------------------------------------------------- k_reclass --

// Starts the copy of [p, p + bytes) from HBM into L2 (whole 16-byte pieces
// inside the range); nothing waits on it, the loads that follow hit L2.
__device__ __forceinline__ void prefetch_l2(const void *p, uint64_t bytes) {
  const uintptr_t b = reinterpret_cast<uintptr_t>(p);
  const uintptr_t e = (b + bytes) & ~static_cast<uintptr_t>(15);
  const uintptr_t st = (b + 15) & ~static_cast<uintptr_t>(15);
  if (e > st) asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(st), "r"(static_cast<uint32_t>(e - st)));
}

// The new token's class mark, its saved prior byte and class, and the range
// check of a kept new token's K and V.  Once per unit, so out of line.
__device__ __noinline__ void new_token(const DecodeArgs &a, uint8_t *c, int64_t u, uint32_t prior, uint32_t cn) {
  *c = static_cast<uint8_t>(0x80u | (3u << 2) | cn);
  a.ucnt[u].w = static_cast<int32_t>(prior | (cn << 8) | (1u << 16));
  if (cn != DKV_CLASS_PRUNE) {
    const uint4 *kr = reinterpret_cast<const uint4 *>(a.k_new + u * DKV_HEAD_DIM);
    const uint4 *vr = reinterpret_cast<const uint4 *>(a.v_new + u * DKV_HEAD_DIM);
    bool oor = false;
    for (int q = 0; q < DKV_HEAD_DIM / 8; ++q) oor |= words_out_of_range(__ldg(kr + q)) | words_out_of_range(__ldg(vr + q));
    if (oor) set_error(&a.ws->err, DKV_E_RANGE);
  }
}

__device__ __forceinline__ bool lens_bad(const DecodeArgs &a, int32_t ctx, int32_t nw) {
  return ctx < 0 || nw < 0 || nw > 1 || static_cast<int64_t>(ctx) + nw > a.cap ||
         static_cast<int64_t>(ctx) + nw > static_cast<int64_t>(a.pmax - 1) * a.P;
}

// With a recent window the new token enters as K8V4 without a score: its
// class mark, saved prior byte and list entry, and the range check of its K
// and V words (32 threads per KV head: 16 K words, 16 V words).
__device__ __noinline__ void window_new_token(const DecodeArgs &a, int32_t r, int32_t l, int32_t ctx) {
  const int Hkv = a.Hkv;
  const int64_t lr = static_cast<int64_t>(l) * a.R + r;
  const int64_t u0 = lr * Hkv;
  for (int t = threadIdx.x; t < Hkv * 32; t += blockDim.x) {
    const int h = t >> 5, q = t & 31;
    const uint4 *src = reinterpret_cast<const uint4 *>((q < 16 ? a.k_new : a.v_new) + (u0 + h) * DKV_HEAD_DIM);
    if (words_out_of_range(__ldg(src + (q & 15)))) set_error(&a.ws->err, DKV_E_RANGE);
    if (q != 0) continue;
    uint8_t *c = a.classes + (lr * a.cap + ctx) * Hkv + h;
    a.ucnt[u0 + h].w = static_cast<int32_t>(*c | (DKV_CLASS_K8V4 << 8) | (1u << 16));
    *c = static_cast<uint8_t>(0x80u | (3u << 2) | DKV_CLASS_K8V4);
    const int32_t m = atomicAdd(a.lcnt + lr, 1);
    if (m < kMarkList)
      a.list[lr * kMarkList + m] = (static_cast<uint32_t>(ctx) << 11) | (h << 4) | (3u << 2) | DKV_CLASS_K8V4;
  }
}

// 4 blocks of 512 per SM (32 registers); the paired-row loop of G = 4 runs
// at 3 (40 registers: at 32 it spills)
template <int kV4>  // float4 loads per row (G / 4); 0 = scalar loads
__global__ void __launch_bounds__(kReclassThreads, kV4 == 1 ? 3 : 4) k_reclass(DecodeArgs a) {
  __shared__ int32_t ev_s[kMaxHq * 3];  // per head: demoted, K8V4 pruned, K4V2 pruned
  __shared__ uint32_t mk_s[kMarkList];  // this block's changes, listed for the apply kernel
  __shared__ int32_t mk_n, mk_base;
  const int32_t r = blockIdx.y, l = blockIdx.z;
  const int32_t i0 = static_cast<int32_t>(blockIdx.x) << (31 - __clz(a.rchunk));  // rchunk: a power of two
  const int32_t ctx = __ldg(a.ctx_lens + r), nw = __ldg(a.new_lens + r);
  if (lens_bad(a, ctx, nw)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(&a.ws->err, DKV_E_LENS);
    return;
  }
  if (a.window >= 1 && blockIdx.x == gridDim.x - 1) {  // a block of its own (code here makes the loop spill)
    if (nw == 1) window_new_token(a, r, l, ctx);
    return;
  }
  const int32_t N = ctx + nw;
  if (i0 >= N) return;
  const int32_t i1 = min(N, i0 + a.rchunk);
  // With a recent window the scored rows end where it starts (N - W; the
  // held rows in it keep their class, the new token enters as K8V4 below)
  const int32_t is = a.window >= 1 ? max(i0, min(i1, N - a.window)) : i1;
  // The block's significance rows are one contiguous range: one bulk
  // prefetch into L2 keeps HBM busy with far more bytes in flight than the
  // threads' own loads (2 rows each at 32 registers) hold.  Issued here,
  // before the loop's registers are live, it costs the loop none.
  if (threadIdx.x == 0 && is > i0)
    prefetch_l2(a.sig_sum + ((static_cast<int64_t>(l) * a.R + r) * a.cap + i0) * a.Hq,
                static_cast<uint64_t>(is - i0) * a.Hq * 4u);
  const int Hkv = a.Hkv, G = a.G;
  for (int t = threadIdx.x; t < Hkv * 3; t += blockDim.x) ev_s[t] = 0;
  if (threadIdx.x == 0) mk_n = 0;
  __syncthreads();
  const float thr_h = __fdiv_rn(a.alpha_h, static_cast<float>(N));
  const float thr_l = __fdiv_rn(a.alpha_l, static_cast<float>(N));
  // Reciprocal test: with rc the hardware reciprocal of c (within 1 ulp),
  // y = RN(m * rc) is within 2^-22 (relative) of m / c, so y >= thr (1 + 2^-19)
  // proves RN(m / c) >= thr and y <= thr (1 - 2^-19) proves RN(m / c) < thr
  // (the margins, themselves rounded, stay far from 2^-22); in between, and for
  // thresholds below 2^-100 where a tiny quotient could leave the relative
  // bound, the IEEE division decides.  A NaN fails every test: pruned, as by
  // the division.
  const bool exact_only = !(thr_l >= 0x1p-100f);
  const float hi_h = __fmul_rn(thr_h, 1.0f + 0x1p-19f), lo_h = __fmul_rn(thr_h, 1.0f - 0x1p-19f);
  const float hi_l = __fmul_rn(thr_l, 1.0f + 0x1p-19f), lo_l = __fmul_rn(thr_l, 1.0f - 0x1p-19f);
  const int sh = (Hkv & (Hkv - 1)) == 0 ? __ffs(Hkv) - 1 : -1;
  const int64_t tok0 = static_cast<int64_t>(r) * a.cap + i0;
  const int64_t lrow = static_cast<int64_t>(l) * a.R * a.cap;  // first token row of the layer
  uint8_t *cls = a.classes + (lrow + tok0) * Hkv;
  const float *sig = a.sig_sum + (lrow + tok0) * a.Hq;
  const int32_t *cnt = a.sig_cnt + tok0;
  const int nrows = (is - i0) * Hkv;
  const int64_t u0 = (static_cast<int64_t>(l) * a.R + r) * Hkv;
  if (kV4 == 1 && sh >= 1) {
    // G = 4 and an even power-of-two Hkv: a thread takes the two rows of one
    // token and head pair (32 contiguous bytes of sums, 2 class bytes),
    // sharing the token's count, reciprocal and new-token test
    // the reciprocal test's bounds, opened to +-inf when only the division
    // decides: then the first test passes only y = +inf and the third only
    // y = -inf or NaN, where the division gives the same class
    const float fhh = exact_only ? INFINITY : hi_h, fhl = exact_only ? -INFINITY : lo_h;
    const float flh = exact_only ? INFINITY : hi_l, fll = exact_only ? -INFINITY : lo_l;
    auto decide = [&](float mm, float cf, float rc) -> uint32_t {
      const float yv = __fmul_rn(mm, rc);
      if (yv >= fhh) return DKV_CLASS_K8V4;
      if (!(yv > fhl) && yv >= flh) return DKV_CLASS_K4V2;
      if (!(yv > fhl) && !(yv > fll)) return DKV_CLASS_PRUNE;
      const float sq = __fdiv_rn(mm, cf);
      return sq >= thr_h ? DKV_CLASS_K8V4 : (sq >= thr_l ? DKV_CLASS_K4V2 : DKV_CLASS_PRUNE);
    };
    auto update = [&](int j, int ii, bool is_new, uint32_t o, uint32_t cn) {
      const int h = j - (ii << sh);
      if (!is_new) {
        if (o == DKV_CLASS_PRUNE) return;  // min(0, x) = 0: nothing can change
        if (o > DKV_CLASS_K8V4) {
          set_error(&a.ws->err, DKV_E_INTERNAL);
          return;
        }
        if (cn < o) {
          cls[j] = static_cast<uint8_t>(0x80u | (o << 2) | cn);
          atomicAdd(&ev_s[h * 3 + (o == DKV_CLASS_K4V2 ? 2 : (cn == DKV_CLASS_K4V2 ? 0 : 1))], 1);
          const int32_t q = atomicAdd(&mk_n, 1);
          if (q < kMarkList) mk_s[q] = (static_cast<uint32_t>(i0 + ii) << 11) | (h << 4) | (o << 2) | cn;
        }
      } else {  // the new token (position ctx)
        new_token(a, cls + j, u0 + h, o, cn);
        const int32_t q = atomicAdd(&mk_n, 1);
        if (q < kMarkList) mk_s[q] = (static_cast<uint32_t>(i0 + ii) << 11) | (h << 4) | (3u << 2) | cn;
      }
    };
    const float4 *sp = reinterpret_cast<const float4 *>(sig);
    const int npairs = nrows >> 1;
    for (int jp = threadIdx.x; jp < npairs; jp += kReclassThreads) {
      const int j = 2 * jp;
      const int ii = j >> sh;
      const int32_t cc = __ldg(cnt + ii);
      const uint32_t o2 = *reinterpret_cast<const uint16_t *>(cls + j);
      const float4 x = __ldcs(sp + j), y = __ldcs(sp + j + 1);
      const bool is_new = i0 + ii >= ctx;
      const uint32_t o0 = o2 & 0xffu, o1 = o2 >> 8;
      if (!is_new && o0 == DKV_CLASS_PRUNE && o1 == DKV_CLASS_PRUNE) continue;
      // max over the group of the rounded quotients == rounded quotient of
      // the max sum (min for a negative count): division is monotone
      float m0, m1;
      if (cc > 0) {
        m0 = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
        m1 = fmaxf(fmaxf(y.x, y.y), fmaxf(y.z, y.w));
      } else {
        m0 = fminf(fminf(x.x, x.y), fminf(x.z, x.w));
        m1 = fminf(fminf(y.x, y.y), fminf(y.z, y.w));
      }
      uint32_t cn0 = DKV_CLASS_K8V4, cn1 = DKV_CLASS_K8V4;  // a count of 0: not yet observed
      if (cc != 0) {
        const float cf = static_cast<float>(cc);
        float rc;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rc) : "f"(cf));
        cn0 = decide(m0, cf, rc);
        cn1 = decide(m1, cf, rc);
      }
      update(j, ii, is_new, o0, cn0);
      update(j + 1, ii, is_new, o1, cn1);
    }
  } else
  for (int jb = 0; jb < nrows; jb += kReclassRows * kReclassThreads) {
    float m[kReclassRows];
    int32_t c[kReclassRows];
    uint32_t old[kReclassRows];
#pragma unroll
    for (int k = 0; k < kReclassRows; ++k) {
      const int j = jb + k * kReclassThreads + threadIdx.x;
      m[k] = 0.0f;
      c[k] = 0;
      old[k] = 0;
      if (j < nrows) {
        const int ii = sh >= 0 ? (j >> sh) : j / Hkv;
        c[k] = __ldg(cnt + ii);
        old[k] = cls[j];
        if (kV4 > 0) {
          const float4 *p = reinterpret_cast<const float4 *>(sig + static_cast<int64_t>(j) * G);
          const float4 x = __ldcs(p);
          float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
          float mn = fminf(fminf(x.x, x.y), fminf(x.z, x.w));
#pragma unroll
          for (int q = 1; q < kV4; ++q) {
            const float4 y = __ldcs(p + q);
            mx = fmaxf(mx, fmaxf(fmaxf(y.x, y.y), fmaxf(y.z, y.w)));
            mn = fminf(mn, fminf(fminf(y.x, y.y), fminf(y.z, y.w)));
          }
          m[k] = c[k] > 0 ? mx : mn;
        } else {
          const float *p = sig + static_cast<int64_t>(j) * G;
          float mx = __ldcs(p), mn = mx;
          for (int q = 1; q < G; ++q) {
            const float y = __ldcs(p + q);
            mx = fmaxf(mx, y);
            mn = fminf(mn, y);
          }
          m[k] = c[k] > 0 ? mx : mn;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kReclassRows; ++k) {
      const int j = jb + k * kReclassThreads + threadIdx.x;
      if (j >= nrows) continue;
      const int ii = sh >= 0 ? (j >> sh) : j / Hkv;
      const int h = j - ii * Hkv;
      const bool is_new = i0 + ii >= ctx;
      const uint32_t o = old[k];
      if (!is_new && o == DKV_CLASS_PRUNE) continue;  // min(0, x) = 0: nothing can change
      uint32_t cn = DKV_CLASS_K8V4;  // a count of 0: not yet observed
      if (c[k] != 0) {
        // max over the group of the rounded quotients == rounded quotient
        // of the max sum (min for a negative count): division is monotone
        const float cf = static_cast<float>(c[k]);
        float rc;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rc) : "f"(cf));
        const float y = __fmul_rn(m[k], rc);
        if (!exact_only && y >= hi_h) {
          cn = DKV_CLASS_K8V4;
        } else if (!exact_only && !(y > lo_h) && y >= hi_l) {
          cn = DKV_CLASS_K4V2;
        } else if (!exact_only && !(y > lo_h) && !(y > lo_l)) {
          cn = DKV_CLASS_PRUNE;
        } else {
          const float s = __fdiv_rn(m[k], cf);
          cn = s >= thr_h ? DKV_CLASS_K8V4 : (s >= thr_l ? DKV_CLASS_K4V2 : DKV_CLASS_PRUNE);
        }
      }
      if (!is_new) {
        if (o > DKV_CLASS_K8V4) {
          set_error(&a.ws->err, DKV_E_INTERNAL);
          continue;
        }
        if (cn < o) {
          cls[j] = static_cast<uint8_t>(0x80u | (o << 2) | cn);
          atomicAdd(&ev_s[h * 3 + (o == DKV_CLASS_K4V2 ? 2 : (cn == DKV_CLASS_K4V2 ? 0 : 1))], 1);
          const int32_t q = atomicAdd(&mk_n, 1);
          if (q < kMarkList) mk_s[q] = (static_cast<uint32_t>(i0 + ii) << 11) | (h << 4) | (o << 2) | cn;
        }
      } else {  // the new token (position ctx)
        new_token(a, cls + j, u0 + h, o, cn);
        const int32_t q = atomicAdd(&mk_n, 1);
        if (q < kMarkList) mk_s[q] = (static_cast<uint32_t>(i0 + ii) << 11) | (h << 4) | (3u << 2) | cn;
      }
    }
  }
  __syncthreads();
  // the block's changes join its (layer, request) list; a block with more
  // than the buffer holds pushes the list past its capacity, so the apply
  // kernel scans the class bytes of that (layer, request) instead
  const int32_t nmk = mk_n;
  if (threadIdx.x == 0 && nmk > 0)
    mk_base = atomicAdd(a.lcnt + (static_cast<int64_t>(l) * a.R + r), nmk <= kMarkList ? nmk : (1 << 24));
  __syncthreads();
  if (nmk > 0 && nmk <= kMarkList) {
    uint32_t *dst = a.list + (static_cast<int64_t>(l) * a.R + r) * kMarkList;
    for (int q = threadIdx.x; q < nmk; q += blockDim.x)
      if (mk_base + q < kMarkList) dst[mk_base + q] = mk_s[q];
  }
  for (int t = threadIdx.x; t < Hkv * 3; t += blockDim.x) {
    const int32_t n = ev_s[t];
    if (n == 0) continue;
    int4 *uc = a.ucnt + u0 + t / 3;
    int *dst = (t % 3 == 0) ? &uc->x : (t % 3 == 1 ? &uc->y : &uc->z);
    atomicAdd(dst, n);
  }
}

// -------------------------------------------------------------- k_candidate --

// The single-candidate policy of the review's Algorithm 1 (Referee Report,
// major comment 2): per (layer, request) only the token that the new one
// pushes out of the recent window, position ctx - W, is classified (its class
// becomes min(old, classify)), and the new token enters as K8V4 (W >= 1) or
// is classified (W = 0).  Every other class byte stays as it is, so this
// replaces k_reclass's pass over the significance sums with 2 Hkv rows per
// (layer, request); it leaves the same marks, counters and change lists.
__global__ void __launch_bounds__(kCandThreads) k_candidate(DecodeArgs a) {
  const int32_t r = blockIdx.x, l = blockIdx.y;
  const int32_t ctx = __ldg(a.ctx_lens + r), nw = __ldg(a.new_lens + r);
  if (lens_bad(a, ctx, nw)) {
    if (threadIdx.x == 0) set_error(&a.ws->err, DKV_E_LENS);
    return;
  }
  if (nw == 0) return;  // no new token: nothing leaves the window
  const int32_t N = ctx + 1, W = a.window, pc = ctx - W;
  const int Hkv = a.Hkv, G = a.G;
  const float thr_h = __fdiv_rn(a.alpha_h, static_cast<float>(N));
  const float thr_l = __fdiv_rn(a.alpha_l, static_cast<float>(N));
  const int64_t lr = static_cast<int64_t>(l) * a.R + r;
  const int64_t u0 = lr * Hkv;
  for (int j = threadIdx.x; j < 2 * Hkv; j += blockDim.x) {
    const bool is_new = j >= Hkv;
    const int h = is_new ? j - Hkv : j;
    if (!is_new && (W < 1 || pc < 0)) continue;  // no held token leaves the window
    const int32_t i = is_new ? ctx : pc;
    const int64_t row = lr * a.cap + i;
    uint8_t *c = a.classes + row * Hkv + h;
    const uint32_t o = *c;
    if (!is_new && o == DKV_CLASS_PRUNE) continue;
    uint32_t cn = DKV_CLASS_K8V4;
    const int32_t cnt = __ldg(a.sig_cnt + static_cast<int64_t>(r) * a.cap + i);
    if (cnt != 0 && !(is_new && W >= 1)) {
      const float *p = a.sig_sum + row * a.Hq + h * G;
      float mx = __ldg(p), mn = mx;
      for (int q = 1; q < G; ++q) {
        const float y = __ldg(p + q);
        mx = fmaxf(mx, y);
        mn = fminf(mn, y);
      }
      const float sc = __fdiv_rn(cnt > 0 ? mx : mn, static_cast<float>(cnt));
      cn = sc >= thr_h ? DKV_CLASS_K8V4 : (sc >= thr_l ? DKV_CLASS_K4V2 : DKV_CLASS_PRUNE);
    }
    uint32_t e;
    if (!is_new) {
      if (o > DKV_CLASS_K8V4) {
        set_error(&a.ws->err, DKV_E_INTERNAL);
        continue;
      }
      if (cn >= o) continue;
      *c = static_cast<uint8_t>(0x80u | (o << 2) | cn);
      int4 *uc = a.ucnt + u0 + h;
      atomicAdd(o == DKV_CLASS_K4V2 ? &uc->z : (cn == DKV_CLASS_K4V2 ? &uc->x : &uc->y), 1);
      e = (static_cast<uint32_t>(i) << 11) | (h << 4) | (o << 2) | cn;
    } else {
      new_token(a, c, u0 + h, o, cn);
      e = (static_cast<uint32_t>(i) << 11) | (h << 4) | (3u << 2) | cn;
    }
    // at most 2 Hkv <= 256 entries: the list never overflows
    const int32_t q = atomicAdd(a.lcnt + lr, 1);
    if (q < kMarkList) a.list[lr * kMarkList + q] = e;
  }
}

// ------------------------------------------------------------------ k_dscan --

// 64-bit look-back word: flags in bits 62-63, new pages in bits 31-61, freed
// pages in bits 0-30 (both sums stay below 2^31: units * pmax < 2^31).
constexpr uint64_t kHalfMask = (1ull << 31) - 1;

__global__ void __launch_bounds__(kDScanThreads) k_dscan(DecodeArgs a) {
  __shared__ uint64_t wsum_s[kDScanThreads / 32];
  __shared__ int32_t part_s, fail_s;
  __shared__ uint64_t prefix_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    part_s = atomicAdd(&a.ws->ticket, 1);
    fail_s = 0;
  }
  __syncthreads();
  const int32_t part = part_s;
  const int32_t npart = static_cast<int32_t>((a.U + kDScanThreads - 1) / kDScanThreads);
  if (part >= npart) return;
  const int64_t u = static_cast<int64_t>(part) * kDScanThreads + tid;

  DecPlan pl{};
  uint64_t v = 0;
  if (u < a.U) {
    const int4 hdr = reinterpret_cast<const int4 *>(a.unit_hdr)[u];
    const int4 uc = a.ucnt[u];
    pl.n_hi = hdr.x;
    pl.n_lo = hdr.y;
    pl.have_hi = hdr.z;
    pl.have_lo = hdr.w;
    pl.dem = uc.x;
    pl.keep_hi = hdr.x - uc.x - uc.y;
    pl.keep_lo = hdr.y - uc.z;
    pl.new_cls = (uc.w & (1 << 16)) ? ((uc.w >> 8) & 3) : 0;
    const int32_t n2_hi = pl.keep_hi + (pl.new_cls == DKV_CLASS_K8V4);
    const int32_t n2_lo = pl.keep_lo + pl.dem + (pl.new_cls == DKV_CLASS_K4V2);
    pl.need_hi = cdiv(n2_hi, a.P);
    pl.need_lo = cdiv(n2_lo, 2 * a.P);
    const int32_t ctx = __ldg(a.ctx_lens + (u / a.Hkv) % a.R);
    if (pl.keep_hi < 0 || pl.keep_lo < 0 || pl.have_hi < 0 || pl.have_lo < 0 || hdr.x < 0 || hdr.y < 0 ||
        pl.have_hi + pl.have_lo > a.pmax || static_cast<int64_t>(hdr.x) > static_cast<int64_t>(pl.have_hi) * a.P ||
        static_cast<int64_t>(hdr.y) > static_cast<int64_t>(pl.have_lo) * 2 * a.P ||
        static_cast<int64_t>(hdr.x) + hdr.y > ctx) {
      set_error(&a.ws->err, DKV_E_INTERNAL);
      pl.need_hi = pl.have_hi > 0 ? pl.have_hi : 0;
      pl.need_lo = pl.have_lo > 0 ? pl.have_lo : 0;
    } else if (pl.need_hi + pl.need_lo > a.pmax) {
      set_error(&a.ws->err, DKV_E_LENS);
      pl.need_hi = pl.have_hi;
      pl.need_lo = pl.have_lo;
    }
    const int32_t d = max(0, pl.need_hi - pl.have_hi) + max(0, pl.need_lo - pl.have_lo);
    const int32_t f = max(0, pl.have_hi - pl.need_hi) + max(0, pl.have_lo - pl.need_lo);
    v = (static_cast<uint64_t>(d) << 31) | static_cast<uint64_t>(f);
  }
  // block-wide inclusive scan of the packed (new, freed) counts
  uint64_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) wsum_s[warp] = incl;
  __syncthreads();
  uint64_t before = 0;
  for (int w = 0; w < warp; ++w) before += wsum_s[w];
  const uint64_t excl = before + incl - v;

  if (tid == 0) {
    uint64_t agg = 0;
    for (int w = 0; w < kDScanThreads / 32; ++w) agg += wsum_s[w];
    uint64_t prefix = 0;
    bool fail = false;
    if (part == 0) {
      st_release(a.part, kFlagPrefix | agg);
    } else {
      st_release(a.part + part, kFlagAggregate | agg);
      if (a.spin_limit == 0) {
        fail = true;
      } else {
        int32_t pred = part - 1;
        for (;;) {
          uint64_t st = ld_acquire(a.part + pred);
          int64_t spins = 0;
          while ((st >> 62) == 0) {
            if (++spins > a.spin_limit) {
              fail = true;
              break;
            }
            __nanosleep(64);
            st = ld_acquire(a.part + pred);
          }
          if (fail) break;
          prefix += st & kValueMask;
          if ((st & kFlagPrefix) != 0) break;
          --pred;  // partition 0 always publishes a prefix
        }
      }
      if (!fail) st_release(a.part + part, kFlagPrefix | (prefix + agg));
    }
    if (fail) {
      set_error(&a.ws->err, DKV_E_TIMEOUT);
      fail_s = 1;
    }
    prefix_s = prefix;
    if (!fail && part == npart - 1) {
      const uint64_t tot = prefix + agg;
      const int64_t dsum = static_cast<int64_t>(tot >> 31), fsum = static_cast<int64_t>(tot & kHalfMask);
      const uint64_t head = a.cursors[0], tail = a.cursors[1];
      a.ws->dsum = dsum;
      a.ws->fsum = fsum;
      a.ws->head = head;
      a.ws->tail = tail;
      if (tail - head > static_cast<uint64_t>(a.F) || static_cast<uint64_t>(dsum) > tail - head)
        set_error(&a.ws->err, DKV_E_NOMEM);
    }
  }
  __syncthreads();
  if (fail_s || u >= a.U) return;
  const uint64_t off = prefix_s + excl;
  pl.off_d = static_cast<int32_t>(off >> 31);
  pl.off_f = static_cast<int32_t>(off & kHalfMask);
  a.plan[u] = pl;
}

// ------------------------------------------------------------------ k_apply --

// Up to 32 next indices s in [cur, hi) whose bit in bm is `want`, ascending,
// into buf[0..); advances cur past the last one taken.  Warp-collective.
__device__ int next_bits(const uint32_t *bm, int32_t &cur, int32_t hi, bool want, int32_t *buf, int lane) {
  int got = 0;
  while (got < 32 && cur < hi) {
    const int32_t w = (cur >> 5) + lane;
    const int32_t s0 = w << 5;
    uint32_t bits = 0;
    if (s0 < hi) {
      bits = want ? bm[w] : ~bm[w];
      if (s0 < cur) bits &= ~0u << (cur - s0);
      if (hi - s0 < 32) bits &= (1u << (hi - s0)) - 1u;
    }
    const int n = __popc(bits);
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    const int room = 32 - got;
    int rk = incl - n;
    uint32_t b = bits;
    while (b != 0u && rk < room) {
      const int j = __ffs(b) - 1;
      b &= b - 1u;
      buf[got + rk] = s0 + j;
      ++rk;
    }
    __syncwarp();
    if (total <= room) {
      got += total;
      const int32_t nxt = ((cur >> 5) + 32) << 5;
      cur = nxt < hi ? nxt : hi;
    } else {
      got = 32;
      cur = buf[31] + 1;
    }
  }
  return got;
}

// Everything one warp needs about its unit.
struct UnitView {
  int64_t u;
  int64_t row0;        // classes / slot_of index of (position 0, this head)
  int32_t ctx;         // live positions before the step
  int32_t Hkv;
  const int32_t *fw;   // forward row (old contents until the table phase)
  DecPlan p;
  int64_t new_base;    // head + off_d (free-list cursor of the unit's first new page)
  int32_t xh;          // new K8V4 pages
};

__device__ __forceinline__ int32_t new_page(const DecodeArgs &a, const UnitView &v, int32_t j) {
  const uint64_t idx = static_cast<uint64_t>(v.new_base + j) % static_cast<uint64_t>(a.F);
  return a.free_list[idx];
}

// Page id of page k of the unit's K8V4 (hi) or K4V2 list: the old pages
// first, then the new ones.  -1 (and an error) for an id outside the pool.
__device__ __forceinline__ int32_t list_page(const DecodeArgs &a, const UnitView &v, bool hi, int32_t k) {
  int32_t id;
  if (!in_range(k, hi ? max(v.p.have_hi, v.p.need_hi) : max(v.p.have_lo, v.p.need_lo), a.status)) return -1;
  if (hi) id = k < v.p.have_hi ? v.fw[k] : new_page(a, v, k - v.p.have_hi);
  else id = k < v.p.have_lo ? v.fw[v.p.have_hi + k] : new_page(a, v, v.xh + k - v.p.have_lo);
  if (id < 0 || id >= a.F) {
    atomicCAS(a.status, 0, DKV_E_INTERNAL);
    return -1;
  }
  return id;
}

struct SlotAddr {
  uint8_t *k, *v, *meta, *pos;
};

__device__ __forceinline__ bool slot_addr(const DecodeArgs &a, const UnitView &v, bool hi, int32_t s, SlotAddr &o) {
  const int32_t per = hi ? a.P : 2 * a.P;
  const int32_t id = list_page(a, v, hi, s / per);
  if (id < 0) return false;
  const PageGeom &g = a.pg;
  const int64_t ss = s % per;
  uint8_t *pg = a.pages + static_cast<int64_t>(id) * g.bytes;
  o.k = pg + ss * 16 * (hi ? g.kh : g.kh >> 1);
  o.v = pg + g.vbase + ss * 16 * (hi ? g.vh : g.vh >> 1);
  o.meta = pg + g.meta + 8 * ss;
  o.pos = pg + g.pos + 4 * ss;
  return true;
}

// 16-byte units of K and V codes in one slot of the high (hi) or low list of
// scheme S (the bit widths of the high class).
template <int S>
__device__ __forceinline__ int k_units(bool hi) { return hi ? scheme_kh(S) : scheme_kh(S) >> 1; }
template <int S>
__device__ __forceinline__ int v_units(bool hi) { return hi ? scheme_vh(S) : scheme_vh(S) >> 1; }

// Copy one slot of a list to another slot of the same list (codes, metadata,
// position); kn, vn: 16-byte units of K and V codes per slot.  Returns the
// moved token's position.
__device__ __forceinline__ int32_t copy_slot(const SlotAddr &f, const SlotAddr &t, int kn, int vn) {
  const uint4 *fk = reinterpret_cast<const uint4 *>(f.k);
  const uint4 *fv = reinterpret_cast<const uint4 *>(f.v);
  uint4 *tk = reinterpret_cast<uint4 *>(t.k);
  uint4 *tv = reinterpret_cast<uint4 *>(t.v);
  uint4 x[8];  // K, then V (distinct slots: no overlap)
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < kn) x[i] = fk[i];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < kn) tk[i] = x[i];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < vn) x[i] = fv[i];
  const uint2 m = *reinterpret_cast<const uint2 *>(f.meta);
  const int32_t pos = *reinterpret_cast<const int32_t *>(f.pos);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < vn) tv[i] = x[i];
  *reinterpret_cast<uint2 *>(t.meta) = m;
  *reinterpret_cast<int32_t *>(t.pos) = pos;
  return pos;
}

__device__ __forceinline__ void clear_slot(const SlotAddr &t, int kn, int vn) {
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  uint4 *tk = reinterpret_cast<uint4 *>(t.k);
  uint4 *tv = reinterpret_cast<uint4 *>(t.v);
  for (int i = 0; i < kn; ++i) tk[i] = z;
  for (int i = 0; i < vn; ++i) tv[i] = z;
  *reinterpret_cast<uint2 *>(t.meta) = make_uint2(0u, 0u);
  *reinterpret_cast<int32_t *>(t.pos) = -1;
}

// Hole-fill of one list: survivors in slots >= keep move, ascending, into the
// removed slots below keep, ascending; the moved tokens' index entries follow.
template <int S>
__device__ void hole_fill(const DecodeArgs &a, const UnitView &v, bool hi, const uint32_t *rm, int32_t keep,
                          int32_t n, int32_t *buf, int lane) {
  int32_t hc = 0, mc = keep;
  for (;;) {
    const int nh = next_bits(rm, hc, keep, true, buf, lane);
    if (nh == 0) break;
    int32_t hole = lane < nh ? buf[lane] : 0;
    __syncwarp();
    const int nm = next_bits(rm, mc, n, false, buf, lane);
    int32_t mover = lane < nm ? buf[lane] : 0;
    __syncwarp();
    if (nm != nh) {
      if (lane == 0) atomicCAS(a.status, 0, DKV_E_INTERNAL);
      return;
    }
    if (lane < nh) {
      SlotAddr f, t;
      if (slot_addr(a, v, hi, mover, f) && slot_addr(a, v, hi, hole, t)) {
        const int32_t pos = copy_slot(f, t, k_units<S>(hi), v_units<S>(hi));
        if (pos >= 0 && pos < v.ctx) a.slot_of[v.row0 + static_cast<int64_t>(pos) * v.Hkv] = hole;
        else atomicCAS(a.status, 0, DKV_E_INTERNAL);
      }
    }
  }
  __syncwarp();
}

// The per-token quantiser on fp32 values spread over kGroup lanes (kPer
// channels each): exact min / max (a zero extreme taken as +0), fp16 scale
// (raised to 2^-24 from 0, lowered to 65504 from infinity) and zero,
// q = clamp(rint_even(RN(x - z) / s), 0, n).
//
// The code of an element is read from y = RN(d * RN(1/s) + 1536.5), d =
// RN(x - z): y lies on a grid of 2^-13 and bits(y) >> 13 holds floor(t + 0.5)
// for t = y - 1536.5.  |d * RN(1/s) - d / s| <= 2^-16 for codes below 256, far
// inside half the grid step, so when y is not an integer (t not a
// half-integer) floor(t + 0.5) is the rounded quotient of the definition.
// A lane holding an integer y (low 13 bits zero) re-evaluates all its
// elements with the IEEE division, as does every lane of a row whose codes
// would need clamping.
template <int kPer, int kGroup>
__device__ __forceinline__ void quant_vals(const float (&x)[kPer], int nmax, uint32_t (&q)[kPer], uint16_t &s16o,
                                           uint16_t &z16o) {
  float mn = x[0], mx = x[0];
#pragma unroll
  for (int i = 1; i < kPer; ++i) {
    mn = fminf(mn, x[i]);
    mx = fmaxf(mx, x[i]);
  }
#pragma unroll
  for (int o = 1; o < kGroup; o <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  mn = __fadd_rn(mn, 0.0f);
  mx = __fadd_rn(mx, 0.0f);
  const float nf = static_cast<float>(nmax);
  const float s32 = __fdiv_rn(__fsub_rn(mx, mn), nf);
  uint16_t s16 = __half_as_ushort(__float2half_rn(s32));
  if (mx > mn && s16 == 0) s16 = 1;
  if (s16 == 0x7c00u) s16 = 0x7bffu;  // 65504: 1-bit codes of a span above 65519 clamp
  const uint16_t z16 = __half_as_ushort(__float2half_rn(mn));
  const float s = __half2float(__ushort_as_half(s16));
  const float z = __half2float(__ushort_as_half(z16));
  s16o = s16;
  z16o = z16;
  if (s == 0.0f) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) q[i] = 0u;
    return;
  }
  const float r = __frcp_rn(s);
  const bool clamp_row = __fmul_rn(__fsub_rn(mn, z), r) < -0.25f || __fmul_rn(__fsub_rn(mx, z), r) > nf + 0.25f;
  // fast codes first, with the smallest fraction field seen; one branch for
  // the lane's codes: where any fraction is zero (a code that may differ from
  // the definition) or the row clamps, every code is taken by the division
  // (equal to the fast code wherever that one is right)
  uint32_t frac = clamp_row ? 0u : 8191u;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const float d = __fsub_rn(x[i], z);
    const uint32_t bits = __float_as_uint(__fmaf_rn(d, r, 1536.5f));
    q[i] = (bits >> 13) & 255u;
    frac = min(frac, bits & 8191u);
  }
  if (frac == 0u) {
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      q[i] = static_cast<uint32_t>(fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(x[i], z), s)), 0.0f), nf));
  }
}

template <int kPer>
__device__ __forceinline__ uint64_t pack_bits(const uint32_t (&q)[kPer], int width) {
  uint64_t w = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) w |= static_cast<uint64_t>(q[i]) << (width * i);
  return w;
}

// Code i (of width w bits) of a run of packed codes held in a uint4.
__device__ __forceinline__ uint32_t code_at(const uint4 &c, int i, int w) {
  const int o = i * w;
  const int wi = o >> 5;
  const uint32_t word = wi == 0 ? c.x : (wi == 1 ? c.y : (wi == 2 ? c.z : c.w));
  return (word >> (o & 31)) & ((1u << w) - 1u);
}

// n bytes (4, 8 or 16; 16-byte-aligned runs of them) into a uint4, the rest zero.
__device__ __forceinline__ uint4 load_bytes(const uint8_t *p, int n) {
  if (n == 16) return *reinterpret_cast<const uint4 *>(p);
  if (n == 8) {
    const uint2 x = *reinterpret_cast<const uint2 *>(p);
    return make_uint4(x.x, x.y, 0u, 0u);
  }
  return make_uint4(*reinterpret_cast<const uint32_t *>(p), 0u, 0u, 0u);
}

// The low 2 w bytes of v (16 codes of w bits) at p (w = 1, 2 or 4).
__device__ __forceinline__ void store_codes16(uint8_t *p, uint64_t v, int w) {
  if (w == 4) *reinterpret_cast<uint2 *>(p) = make_uint2(static_cast<uint32_t>(v), static_cast<uint32_t>(v >> 32));
  else if (w == 2) *reinterpret_cast<uint32_t *>(p) = static_cast<uint32_t>(v);
  else *reinterpret_cast<uint16_t *>(p) = static_cast<uint16_t>(v);
}

// Requantise one demoted token, 8 lanes (lane t: channels 16t .. 16t+15):
// dequantise its high-class codes (fma(q, s, z)) at the scheme's (kh, vh)
// widths, quantise them at (kh/2, vh/2) and store them, with the metadata and
// position, into low-class slot ds of page dpg.  kc, vc: the lane's 2 kh and
// 2 vh code bytes.  Every lane of the warp calls it (the reductions shuffle
// within 8 lanes).
template <int S>
__device__ __forceinline__ void requant8(const DecodeArgs &a, uint4 kc, uint4 vc, uint2 meta, bool ok, uint8_t *dpg,
                                         int64_t ds, int32_t pos, int t) {
  const PageGeom &g = a.pg;
  constexpr int KH = scheme_kh(S), VH = scheme_vh(S), kl = KH >> 1, vl = VH >> 1;
  float x[16];
  uint32_t q[16];
  uint16_t ks2, kz2, vs2, vz2;
  {  // K then V, one 16-channel piece at a time (fewer live registers)
    const float ks = __half2float(__ushort_as_half(static_cast<uint16_t>(meta.x & 0xffffu)));
    const float kz = __half2float(__ushort_as_half(static_cast<uint16_t>(meta.x >> 16)));
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = __fmaf_rn(static_cast<float>(code_at(kc, i, KH)), ks, kz);
    quant_vals<16, 8>(x, (1 << kl) - 1, q, ks2, kz2);
    if (ok) store_codes16(dpg + ds * 16 * kl + 2 * kl * t, pack_bits<16>(q, kl), kl);
  }
  {
    const float vs = __half2float(__ushort_as_half(static_cast<uint16_t>(meta.y & 0xffffu)));
    const float vz = __half2float(__ushort_as_half(static_cast<uint16_t>(meta.y >> 16)));
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = __fmaf_rn(static_cast<float>(code_at(vc, i, VH)), vs, vz);
    quant_vals<16, 8>(x, (1 << vl) - 1, q, vs2, vz2);
    if (ok) store_codes16(dpg + g.vbase + ds * 16 * vl + 2 * vl * t, pack_bits<16>(q, vl), vl);
  }
  if (ok && t == 0) {
    *reinterpret_cast<uint2 *>(dpg + g.meta + 8 * ds) =
        make_uint2(static_cast<uint32_t>(ks2) | (static_cast<uint32_t>(kz2) << 16),
                   static_cast<uint32_t>(vs2) | (static_cast<uint32_t>(vz2) << 16));
    *reinterpret_cast<int32_t *>(dpg + g.pos + 4 * ds) = pos;
  }
}

// The demoted tokens (high -> low class) go to low-class slots keep_lo + k in
// ascending position order.  Normally each token's high slot bytes are
// copied, one lane per token, into a job for k_demote (the copy must happen
// before the high list's hole-fill may overwrite the slot; the
// requantisation runs later, spread over the whole GPU); when the call's job
// buffer is full, this warp requantises them in place, 8 lanes per token.
template <int S>
__device__ void demote(const DecodeArgs &a, const UnitView &v, const uint32_t *dem, int32_t *buf, int lane) {
  int32_t cur = 0, k = 0;
  const int grp = lane >> 3, t = lane & 7;
  const PageGeom &g = a.pg;
  constexpr int KH = scheme_kh(S), VH = scheme_vh(S);
  const int64_t P = a.P;
  for (;;) {
    const int nd = next_bits(dem, cur, v.ctx, true, buf, lane);
    if (nd == 0) break;
    // one lane per demoted token: its high slot, then the ids of its source
    // and destination pages (two rounds of loads for up to 32 tokens)
    int32_t my_hs = -1, my_src = -1, my_dst = -1;
    if (lane < nd) my_hs = a.slot_of[v.row0 + static_cast<int64_t>(buf[lane]) * v.Hkv];
    if (lane < nd) {
      if (my_hs >= 0 && my_hs < v.p.n_hi) my_src = list_page(a, v, true, my_hs / a.P);
      my_dst = list_page(a, v, false, (v.p.keep_lo + k + lane) / (2 * a.P));
    }
    int32_t base = 0;
    if (lane == 0) base = atomicAdd(&a.ws->job_n, nd);
    base = __shfl_sync(0xffffffffu, base, 0);
    if (static_cast<int64_t>(base) + nd <= a.njobs) {
      if (lane < nd) {
        const int32_t pos = buf[lane];
        DemJob &jb = a.jobs[base + lane];
        bool ok = my_hs >= 0 && my_hs < v.p.n_hi && my_src >= 0 && my_dst >= 0;
        if (ok) {
          const int64_t ss = my_hs % P;
          const uint8_t *spg = a.pages + static_cast<int64_t>(my_src) * g.bytes;
          const uint4 *kk = reinterpret_cast<const uint4 *>(spg + 16 * KH * ss);
          const uint4 *vv = reinterpret_cast<const uint4 *>(spg + g.vbase + 16 * VH * ss);
          uint4 c[8];  // K codes, then V codes
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i < KH) c[i] = kk[i];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i < KH) jb.c[i] = c[i];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i < VH) c[i] = vv[i];
          const uint2 meta = *reinterpret_cast<const uint2 *>(spg + g.meta + 8 * ss);
          const int32_t spos = *reinterpret_cast<const int32_t *>(spg + g.pos + 4 * ss);
          ok = spos == pos;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i < VH) jb.c[KH + i] = c[i];
          jb.meta = meta;
        }
        if (!ok) atomicCAS(a.status, 0, DKV_E_INTERNAL);
        const int32_t slot = v.p.keep_lo + k + lane;
        jb.dst_page = ok ? my_dst : -1;
        jb.dst_slot = slot % (2 * a.P);
        jb.pos = pos;
        if (ok) a.slot_of[v.row0 + static_cast<int64_t>(pos) * v.Hkv] = slot;
      }
    } else {
      // the reservation ran past the buffer: its entries inside the buffer
      // are marked empty (k_demote reads every reserved entry below the end)
      if (lane < nd && static_cast<int64_t>(base) + lane < a.njobs) a.jobs[base + lane].dst_page = -1;
      for (int gq = 0; gq < nd; gq += 4) {
        const int j = gq + grp;
        const bool act = j < nd;
        const int32_t hs = __shfl_sync(0xffffffffu, my_hs, j & 31);
        const int32_t sid = __shfl_sync(0xffffffffu, my_src, j & 31);
        const int32_t did = __shfl_sync(0xffffffffu, my_dst, j & 31);
        const int32_t pos = act ? buf[j] : 0;
        bool ok = act && hs >= 0 && hs < v.p.n_hi && sid >= 0 && did >= 0;
        const int64_t ss = hs % P, ds = (v.p.keep_lo + k + j) % (2 * P);
        const uint8_t *spg = a.pages + static_cast<int64_t>(sid) * g.bytes;
        uint4 kc = make_uint4(0u, 0u, 0u, 0u), vc = kc;
        uint2 meta = make_uint2(0u, 0u);
        int32_t spos = -1;
        if (ok) {
          kc = load_bytes(spg + 16 * KH * ss + 2 * KH * t, 2 * KH);
          vc = load_bytes(spg + g.vbase + 16 * VH * ss + 2 * VH * t, 2 * VH);
          meta = *reinterpret_cast<const uint2 *>(spg + g.meta + 8 * ss);
          spos = *reinterpret_cast<const int32_t *>(spg + g.pos + 4 * ss);
        }
        if (ok && spos != pos) ok = false;
        if (act && !ok && t == 0) atomicCAS(a.status, 0, DKV_E_INTERNAL);
        requant8<S>(a, kc, vc, meta, ok, a.pages + static_cast<int64_t>(did) * g.bytes, ds, pos, t);
        if (ok && t == 0) a.slot_of[v.row0 + static_cast<int64_t>(pos) * v.Hkv] = v.p.keep_lo + k + j;
      }
    }
    k += nd;
    __syncwarp();
  }
}

// Four codes of w bits per lane (channels 4 lane .. 4 lane + 3) packed into a
// slot's code bytes at d: 32, 16 or 8 bits a lane, or, at 1 bit, the nibbles
// of two lanes joined into one byte.  Every lane of the warp calls it.
__device__ __forceinline__ void store_lane4(uint8_t *d, const uint32_t (&q)[4], int w, int lane, bool ok) {
  const uint32_t bits = static_cast<uint32_t>(pack_bits<4>(q, w));
  if (w == 8) {
    if (ok) reinterpret_cast<uint32_t *>(d)[lane] = bits;
  } else if (w == 4) {
    if (ok) reinterpret_cast<uint16_t *>(d)[lane] = static_cast<uint16_t>(bits);
  } else if (w == 2) {
    if (ok) d[lane] = static_cast<uint8_t>(bits);
  } else {
    const uint32_t up = __shfl_down_sync(0xffffffffu, bits, 1);
    if (ok && (lane & 1) == 0) d[lane >> 1] = static_cast<uint8_t>(bits | (up << 4));
  }
}

// Quantise and store the new token (bf16 row of 128 channels, 4 per lane).
template <int S>
__device__ void append_new(const DecodeArgs &a, const UnitView &v, int lane) {
  const bool hi = v.p.new_cls == DKV_CLASS_K8V4;
  const int32_t slot = hi ? v.p.keep_hi : v.p.keep_lo + v.p.dem;
  SlotAddr d;
  const bool ok = slot_addr(a, v, hi, slot, d);  // warp-uniform
  if (!ok) return;
  const int kw = k_units<S>(hi), vw = v_units<S>(hi);  // widths in bits = 16-byte units per slot
  const uint2 kr = reinterpret_cast<const uint2 *>(a.k_new + v.u * DKV_HEAD_DIM)[lane];
  const uint2 vr = reinterpret_cast<const uint2 *>(a.v_new + v.u * DKV_HEAD_DIM)[lane];
  float xk[4] = {__uint_as_float(kr.x << 16), __uint_as_float(kr.x & 0xffff0000u), __uint_as_float(kr.y << 16),
                 __uint_as_float(kr.y & 0xffff0000u)};
  float xv[4] = {__uint_as_float(vr.x << 16), __uint_as_float(vr.x & 0xffff0000u), __uint_as_float(vr.y << 16),
                 __uint_as_float(vr.y & 0xffff0000u)};
  uint32_t qk[4], qv[4];
  uint16_t ks, kz, vs, vz;
  quant_vals<4, 32>(xk, (1 << kw) - 1, qk, ks, kz);
  quant_vals<4, 32>(xv, (1 << vw) - 1, qv, vs, vz);
  store_lane4(d.k, qk, kw, lane, true);
  store_lane4(d.v, qv, vw, lane, true);
  if (lane == 0) {
    *reinterpret_cast<uint2 *>(d.meta) = make_uint2(static_cast<uint32_t>(ks) | (static_cast<uint32_t>(kz) << 16),
                                                    static_cast<uint32_t>(vs) | (static_cast<uint32_t>(vz) << 16));
    *reinterpret_cast<int32_t *>(d.pos) = v.ctx;
    a.slot_of[v.row0 + static_cast<int64_t>(v.ctx) * v.Hkv] = slot;
  }
}

// Zero codes and metadata, position -1, over a whole new page.
__device__ void clear_page(const DecodeArgs &a, int32_t id, int lane) {
  uint4 *pg = reinterpret_cast<uint4 *>(a.pages + static_cast<int64_t>(id) * a.pg.bytes);
  const int64_t nz = a.pg.pos / 16, nall = a.pg.bytes / 16;  // [0, pos) zero, [pos, bytes) all ones
  for (int64_t i = lane; i < nall; i += 32)
    pg[i] = i < nz ? make_uint4(0u, 0u, 0u, 0u) : make_uint4(~0u, ~0u, ~0u, ~0u);
}

template <int S>
__device__ void apply_unit(const DecodeArgs &a, UnitView &v, uint32_t *rh, uint32_t *rl, uint32_t *dem,
                           int32_t *buf, int32_t *stage, int lane) {
  const DecPlan &p = v.p;
  const int32_t n2_hi = p.keep_hi + (p.new_cls == DKV_CLASS_K8V4);
  const int32_t n2_lo = p.keep_lo + p.dem + (p.new_cls == DKV_CLASS_K4V2);
  // the new token's K and V rows, read at the append near the end: start
  // their way into L2 now
  if (lane == 0 && p.new_cls != DKV_CLASS_PRUNE) {
    prefetch_l2(a.k_new + v.u * DKV_HEAD_DIM, 2 * DKV_HEAD_DIM);
    prefetch_l2(a.v_new + v.u * DKV_HEAD_DIM, 2 * DKV_HEAD_DIM);
  }
  // new pages start clear
  for (int32_t k = p.have_hi; k < p.need_hi; ++k) {
    const int32_t id = list_page(a, v, true, k);
    if (id >= 0) clear_page(a, id, lane);
  }
  for (int32_t k = p.have_lo; k < p.need_lo; ++k) {
    const int32_t id = list_page(a, v, false, k);
    if (id >= 0) clear_page(a, id, lane);
  }
  __syncwarp();
  // a list that lost no token has no holes, and a unit that demoted none has
  // nothing to stage: their bitmap scans are skipped (warp-uniform tests)
  if (p.keep_lo < p.n_lo) hole_fill<S>(a, v, false, rl, p.keep_lo, p.n_lo, buf, lane);  // K4V2 list
  if (p.dem > 0) demote<S>(a, v, dem, buf, lane);  // appended after its survivors
  __syncwarp();
  if (p.keep_hi < p.n_hi) hole_fill<S>(a, v, true, rh, p.keep_hi, p.n_hi, buf, lane);  // K8V4 list (demoted slots read)
  if (p.new_cls != DKV_CLASS_PRUNE) append_new<S>(a, v, lane);
  __syncwarp();
  // vacated slots of the pages the lists keep
  {
    const int32_t end_hi = min(p.n_hi, p.need_hi * a.P);
    for (int32_t s = n2_hi + lane; s < end_hi; s += 32) {
      SlotAddr t;
      if (slot_addr(a, v, true, s, t)) clear_slot(t, k_units<S>(true), v_units<S>(true));
    }
    const int32_t end_lo = min(p.n_lo, p.need_lo * 2 * a.P);
    for (int32_t s = n2_lo + lane; s < end_lo; s += 32) {
      SlotAddr t;
      if (slot_addr(a, v, false, s, t)) clear_slot(t, k_units<S>(false), v_units<S>(false));
    }
  }
  // tables: stage the kept K4V2 page ids (only when the K8V4 page count
  // changes, which moves them in the row), free the surplus, rewrite the row
  const int32_t keep_lo_pages = min(p.have_lo, p.need_lo);
  if (p.need_hi != p.have_hi)
    for (int32_t k = lane; k < keep_lo_pages; k += 32) stage[k] = v.fw[p.have_hi + k];
  int32_t fj = 0;
  const uint64_t tail = a.ws->tail + static_cast<uint64_t>(p.off_f);
  for (int32_t k = p.need_hi + lane; k < p.have_hi; k += 32) {
    const int32_t id = v.fw[k];
    const int32_t j = fj + (k - p.need_hi);
    if (id >= 0 && id < a.F) {
      a.free_list[(tail + j) % static_cast<uint64_t>(a.F)] = id;
      a.rev_unit[id] = -1;
      a.rev_idx[id] = -1;
      a.page_cls[id] = DKV_CLASS_PRUNE;
    }
  }
  fj += max(0, p.have_hi - p.need_hi);
  for (int32_t k = p.need_lo + lane; k < p.have_lo; k += 32) {
    const int32_t id = v.fw[p.have_hi + k];
    const int32_t j = fj + (k - p.need_lo);
    if (id >= 0 && id < a.F) {
      a.free_list[(tail + j) % static_cast<uint64_t>(a.F)] = id;
      a.rev_unit[id] = -1;
      a.rev_idx[id] = -1;
      a.page_cls[id] = DKV_CLASS_PRUNE;
    }
  }
  __syncwarp();
  const int32_t old_tot = p.have_hi + p.have_lo, new_tot = p.need_hi + p.need_lo;
  const int32_t k0 = p.need_hi == p.have_hi ? p.need_hi + keep_lo_pages : min(p.have_hi, p.need_hi);
  const int32_t k1 = max(old_tot, new_tot);
  int32_t *fw = a.fwd + v.u * a.pmax;
  const int32_t unit_id = static_cast<int32_t>(a.unit_base + v.u);
  for (int32_t k = k0 + lane; k < k1; k += 32) {
    int32_t id = -1;
    if (k < p.need_hi) {
      id = new_page(a, v, k - p.have_hi);  // k >= have_hi here: kept K8V4 entries are not rewritten
    } else if (k < new_tot) {
      const int32_t j = k - p.need_hi;
      id = j < keep_lo_pages ? stage[j] : new_page(a, v, v.xh + j - p.have_lo);
    }
    fw[k] = id;
    if (id >= 0 && id < a.F) {
      a.rev_unit[id] = unit_id;
      a.rev_idx[id] = k;
      a.page_cls[id] = k < p.need_hi ? DKV_CLASS_K8V4 : DKV_CLASS_K4V2;
    }
  }
  if (lane == 0) reinterpret_cast<int4 *>(a.unit_hdr)[v.u] = make_int4(n2_hi, n2_lo, p.need_hi, p.need_lo);
}

// Bits of one removed token: its slot in the removed-slot bitmap of its list,
// its position in the demoted bitmap, or its index entry cleared if pruned.
// mark = position << 4 | old class << 2 | new class.
__device__ __forceinline__ void mark_slot(const DecodeArgs &a, uint32_t mark, int64_t row0, const DecPlan &p,
                                          uint32_t *b3, int32_t words) {
  const int32_t i = static_cast<int32_t>(mark >> 4);
  const uint32_t old = (mark >> 2) & 3u, cn = mark & 3u;
  int32_t *so = a.slot_of + row0 + static_cast<int64_t>(i) * a.Hkv;
  const int32_t s = *so;
  const int32_t n = old == DKV_CLASS_K8V4 ? p.n_hi : p.n_lo;
  if (s < 0 || s >= n) {
    atomicCAS(a.status, 0, DKV_E_INTERNAL);
    return;
  }
  atomicOr(b3 + (old == DKV_CLASS_K8V4 ? 0 : words) + (s >> 5), 1u << (s & 31));
  if (cn == DKV_CLASS_K4V2) atomicOr(b3 + 2 * words + (i >> 5), 1u << (i & 31));
  else *so = -1;  // pruned
}

// One changed class byte (position i, head h; old class 3 = the new token):
// the final class (or the old one when the call failed) is written back and a
// removed token is listed for its unit's warp (or handled here if the list is
// full).
__device__ __forceinline__ void take_mark(const DecodeArgs &a, int32_t i, int32_t h, uint32_t old, uint32_t cn,
                                          int32_t h0, int32_t err, int64_t u0, int64_t blk, const DecPlan *plan_s,
                                          uint32_t *bm, int32_t words, uint32_t *mk, int32_t *mk_n) {
  uint8_t *c = a.classes + blk + static_cast<int64_t>(i) * a.Hkv + h;
  if (err != 0) {  // revert
    *c = static_cast<uint8_t>(old == 3u ? (a.ucnt[u0 + h].w & 0xff) : old);
    return;
  }
  *c = static_cast<uint8_t>(cn);
  if (old == 3u) return;  // the new token: handled from the plan
  const uint32_t mark = (static_cast<uint32_t>(i) << 4) | (old << 2) | cn;
  const int32_t k = atomicAdd(&mk_n[h - h0], 1);
  if (k < kMarkCap) mk[(h - h0) * kMarkCap + k] = mark;
  else mark_slot(a, mark, blk + h, plan_s[h - h0], bm + 3 * (h - h0) * words, words);
}

// Marks of one 16-byte vector of class bytes (the scan path).  Rare, so out
// of line.
__device__ __noinline__ void take_marks(const DecodeArgs &a, uint4 x, int32_t vi, int32_t nbytes, int32_t h0,
                                        int32_t nh, int32_t err, int64_t u0, int64_t blk, const DecPlan *plan_s,
                                        uint32_t *bm, int32_t words, uint32_t *mk, int32_t *mk_n) {
  const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
  for (int e = 0; e < 16; ++e) {
    const uint32_t b = (xw[e >> 2] >> (8 * (e & 3))) & 255u;
    if ((b & 0x80u) == 0u) continue;
    const int32_t idx = vi * 16 + e;
    if (idx >= nbytes) continue;
    const int32_t i = idx / a.Hkv, h = idx - i * a.Hkv;
    if (h < h0 || h >= h0 + nh) continue;
    take_mark(a, i, h, (b >> 2) & 3u, b & 3u, h0, err, u0, blk, plan_s, bm, words, mk, mk_n);
  }
}

// Listed changes of one (layer, request), when the list holds them all.
__device__ __noinline__ void take_list(const DecodeArgs &a, const uint32_t *list, int32_t n, int32_t h0, int32_t nh,
                                       int32_t err, int64_t u0, int64_t blk, const DecPlan *plan_s, uint32_t *bm,
                                       int32_t words, uint32_t *mk, int32_t *mk_n) {
  for (int32_t q = threadIdx.x; q < n; q += blockDim.x) {
    const uint32_t e = list[q];
    const int32_t h = static_cast<int32_t>((e >> 4) & 127u);
    if (h < h0 || h >= h0 + nh) continue;
    take_mark(a, static_cast<int32_t>(e >> 11), h, (e >> 2) & 3u, e & 3u, h0, err, u0, blk, plan_s, bm, words, mk,
              mk_n);
  }
}

template <int S>
__global__ void __launch_bounds__(32 * kMaxApplyWarps, 3) k_apply(DecodeArgs a, int32_t hpc, int32_t words) {
  extern __shared__ __align__(16) unsigned char smem[];
  DecPlan *plan_s = reinterpret_cast<DecPlan *>(smem);
  uint32_t *bm = reinterpret_cast<uint32_t *>(plan_s + hpc);        // [hpc][3][words]
  int32_t *buf = reinterpret_cast<int32_t *>(bm + 3 * hpc * words);  // [hpc][32]
  int32_t *stage = buf + 32 * hpc;                                   // [hpc][pmax]
  uint32_t *mk = reinterpret_cast<uint32_t *>(stage + a.pmax * hpc);  // [hpc][kMarkCap] marks per unit
  int32_t *mk_n = reinterpret_cast<int32_t *>(mk + kMarkCap * hpc);   // [hpc]
  const int32_t r = blockIdx.y, l = blockIdx.z;
  const int32_t h0 = blockIdx.x * hpc;
  const int32_t nh = min(hpc, a.Hkv - h0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t err = *reinterpret_cast<volatile int32_t *>(&a.ws->err);
  if (blockIdx.x == 0 && r == 0 && l == 0 && tid == 0) {
    if (err != 0) {
      atomicCAS(a.status, 0, err);
    } else {
      a.cursors[0] = a.ws->head + static_cast<uint64_t>(a.ws->dsum);
      a.cursors[1] = a.ws->tail + static_cast<uint64_t>(a.ws->fsum);
    }
  }
  int32_t ctx = a.ctx_lens[r], nw = a.new_lens[r];
  ctx = min(max(ctx, 0), a.cap);
  nw = min(max(nw, 0), a.cap - ctx);
  const int32_t N = ctx + nw;
  const int64_t u0 = (static_cast<int64_t>(l) * a.R + r) * a.Hkv;
  if (err == 0) {
    for (int i = tid; i < nh; i += blockDim.x) {
      plan_s[i] = a.plan[u0 + h0 + i];
      mk_n[i] = 0;
    }
    for (int i = tid; i < 3 * hpc * words; i += blockDim.x) bm[i] = 0u;
  }
  __syncthreads();

  // marks -> final classes (or the old ones if the call failed), bitmaps
  const int64_t blk = (static_cast<int64_t>(l) * a.R + r) * a.cap * a.Hkv;  // classes index of (l, r, 0, 0)
  uint8_t *cls = a.classes + blk;
  const int32_t nbytes = N * a.Hkv;
  const int32_t nvec = (nbytes + 15) >> 4;
  const int64_t lr = static_cast<int64_t>(l) * a.R + r;
  const int32_t n_list = a.lcnt[lr];
  if (n_list <= kMarkList) {  // every change of this (layer, request) is listed
    take_list(a, a.list + lr * kMarkList, n_list, h0, nh, err, u0, blk, plan_s, bm, words, mk, mk_n);
  } else {
  // otherwise scan the class bytes, four vectors per thread at a time; the
  // rare marked ones go out of line
  for (int32_t vb = 0; vb < nvec; vb += 4 * blockDim.x) {
    uint4 x[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int32_t vi = vb + q * blockDim.x + tid;
      x[q] = vi < nvec ? reinterpret_cast<const uint4 *>(cls)[vi] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (((x[q].x | x[q].y | x[q].z | x[q].w) & 0x80808080u) != 0u)
        take_marks(a, x[q], vb + q * blockDim.x + tid, nbytes, h0, nh, err, u0, blk, plan_s, bm, words, mk, mk_n);
  }
  }
  __syncthreads();
  if (err != 0 || warp >= nh) return;
  // this unit's listed marks: slots of the removed tokens, 32 at a time
  {
    const int32_t n_mk = min(mk_n[warp], kMarkCap);
    for (int32_t j = lane; j < n_mk; j += 32)
      mark_slot(a, mk[warp * kMarkCap + j], blk + h0 + warp, plan_s[warp], bm + 3 * warp * words, words);
  }
  __syncwarp();

  UnitView v;
  v.u = u0 + h0 + warp;
  v.row0 = blk + h0 + warp;
  v.ctx = ctx;
  v.Hkv = a.Hkv;
  v.fw = a.fwd + v.u * a.pmax;
  v.p = plan_s[warp];
  v.new_base = static_cast<int64_t>(a.ws->head % static_cast<uint64_t>(a.F)) + v.p.off_d;
  v.xh = max(0, v.p.need_hi - v.p.have_hi);
  uint32_t *b3 = bm + 3 * warp * words;
  apply_unit<S>(a, v, b3, b3 + words, b3 + 2 * words, buf + 32 * warp, stage + a.pmax * warp, lane);
}

// ----------------------------------------------------------------- k_demote --

// The staged demotions of the call, requantised across the whole GPU: each
// 8-lane group takes one job (grid-stride).  Runs after k_apply, whose K4V2
// hole-fill has emptied the destination slots and whose page clears came
// first; a failed call staged nothing.
template <int S>
__global__ void __launch_bounds__(256, 4) k_demote(DecodeArgs a) {
  if (*reinterpret_cast<volatile int32_t *>(&a.ws->err) != 0) return;
  const int64_t n = min(static_cast<int64_t>(a.ws->job_n), a.njobs);
  const int lane = threadIdx.x & 31, grp = lane >> 3, t = lane & 7;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const PageGeom &g = a.pg;
  constexpr int KH = scheme_kh(S), VH = scheme_vh(S);
  for (int64_t b = gw * 4; b < n; b += nw * 4) {
    const int64_t j = b + grp;
    const bool act = j < n;
    uint4 kc = make_uint4(0u, 0u, 0u, 0u), vc = kc;
    uint2 meta = make_uint2(0u, 0u);
    int32_t page = -1, slot = 0, pos = 0;
    if (act) {
      const DemJob &jb = a.jobs[j];
      const uint8_t *c = reinterpret_cast<const uint8_t *>(jb.c);
      kc = load_bytes(c + 2 * KH * t, 2 * KH);
      vc = load_bytes(c + 16 * KH + 2 * VH * t, 2 * VH);
      meta = jb.meta;
      page = jb.dst_page;
      slot = jb.dst_slot;
      pos = jb.pos;
    }
    const bool ok = act && page >= 0 && page < a.F;
    requant8<S>(a, kc, vc, meta, ok, a.pages + static_cast<int64_t>(ok ? page : 0) * g.bytes, slot, pos, t);
  }
}

// ------------------------------------------------------------------ k_index --

// Classes and slot index of every position from the pages: one warp per unit.
__global__ void __launch_bounds__(256) k_index(DecodeArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); u < a.U;
       u += nwarps) {
    const int32_t h = static_cast<int32_t>(u % a.Hkv);
    const int64_t lr = u / a.Hkv;
    const int32_t r = static_cast<int32_t>(lr % a.R);
    const int32_t ctx = a.ctx_lens[r];
    const int4 hdr = reinterpret_cast<const int4 *>(a.unit_hdr)[u];
    const int32_t *fw = a.fwd + u * a.pmax;
    const int64_t row0 = lr * a.cap * a.Hkv + h;
    if (ctx < 0 || ctx > a.cap || hdr.z < 0 || hdr.w < 0 || hdr.z + hdr.w > a.pmax || hdr.x < 0 || hdr.y < 0 ||
        hdr.x > hdr.z * a.P || hdr.y > hdr.w * 2 * a.P) {
      if (lane == 0) atomicCAS(a.status, 0, DKV_E_INTERNAL);
      continue;
    }
    for (int li = 0; li < 2; ++li) {
      const bool hi = li == 0;
      const int32_t n = hi ? hdr.x : hdr.y;
      const int32_t per = hi ? a.P : 2 * a.P;
      for (int32_t s = lane; s < n; s += 32) {
        const int32_t id = fw[(hi ? 0 : hdr.z) + s / per];
        if (id < 0 || id >= a.F) {
          atomicCAS(a.status, 0, DKV_E_INTERNAL);
          continue;
        }
        const int32_t pos =
            *reinterpret_cast<const int32_t *>(a.pages + static_cast<int64_t>(id) * a.pg.bytes + a.pg.pos + 4 * (s % per));
        if (pos < 0 || pos >= ctx) {
          atomicCAS(a.status, 0, DKV_E_INTERNAL);
          continue;
        }
        a.classes[row0 + static_cast<int64_t>(pos) * a.Hkv] = hi ? DKV_CLASS_K8V4 : DKV_CLASS_K4V2;
        a.slot_of[row0 + static_cast<int64_t>(pos) * a.Hkv] = s;
      }
    }
  }
}

}  // namespace

size_t apply_smem(int32_t hpc, int32_t words, int32_t pmax) {
  return sizeof(DecPlan) * hpc + sizeof(uint32_t) * 3 * hpc * words + sizeof(int32_t) * 32 * hpc +
         sizeof(int32_t) * static_cast<size_t>(pmax) * hpc + sizeof(uint32_t) * kMarkCap * hpc + sizeof(int32_t) * hpc;
}

cudaError_t launch_reclass(const DecodeArgs &a, cudaStream_t s) {
  // with a recent window one more block per (layer, request) takes the new token
  const dim3 grid((a.cap + a.rchunk - 1) / a.rchunk + (a.window >= 1 ? 1 : 0), a.R, a.L);
  if (a.G == 4) k_reclass<1><<<grid, kReclassThreads, 0, s>>>(a);
  else if (a.G == 8) k_reclass<2><<<grid, kReclassThreads, 0, s>>>(a);
  else k_reclass<0><<<grid, kReclassThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_candidate(const DecodeArgs &a, cudaStream_t s) {
  k_candidate<<<dim3(a.R, a.L), kCandThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dscan(const DecodeArgs &a, int32_t npart, cudaStream_t s) {
  k_dscan<<<npart, kDScanThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_apply(const DecodeArgs &a, int32_t hpc, int32_t words, cudaStream_t s) {
  const size_t smem = apply_smem(hpc, words, a.pmax);
  void (*kern)(DecodeArgs, int32_t, int32_t) = a.pg.vh == 2 ? k_apply<1> : (a.pg.kh == 4 ? k_apply<2> : k_apply<0>);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const dim3 grid((a.Hkv + hpc - 1) / hpc, a.R, a.L);
  kern<<<grid, 32 * hpc, smem, s>>>(a, hpc, words);
  return cudaGetLastError();
}

cudaError_t launch_demote(const DecodeArgs &a, int grid, cudaStream_t s) {
  static_assert(scheme_vh(1) == 2 && scheme_kh(2) == 4, "scheme dispatch");
  void (*kern)(DecodeArgs) = a.pg.vh == 2 ? k_demote<1> : (a.pg.kh == 4 ? k_demote<2> : k_demote<0>);
  kern<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_index(const DecodeArgs &a, int grid, cudaStream_t s) {
  k_index<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dkv
