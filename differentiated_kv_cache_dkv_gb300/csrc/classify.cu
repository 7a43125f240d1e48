// classify.cu -- request prefix sums (k_prep) and the significance reduce +
// three-tier classification (k_classify).
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
      // request of each of its tiles (bounded by the workspace's room)
      const int64_t room = a.T / kTileTokens + a.R;
      for (int32_t x = 0; x < nt; ++x)
        if (before_tile + il - nt + x < room) a.tile_req[before_tile + il - nt + x] = static_cast<int32_t>(r);
    }
    __syncthreads();
    if (tid == blockDim.x - 1) {
      carry_tok = before_tok + it;
      carry_tile = before_tile + il;
    }
    __syncthreads();
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

// One tile of a layer: where its scores start and how many tokens it holds.
struct ClassifyItem {
  int64_t l, t0, N;
  int32_t rt, cnt;
};

__device__ __forceinline__ ClassifyItem classify_item(const CompactArgs &a, int64_t item, int32_t TR) {
  ClassifyItem it;
  it.l = item / TR;
  it.rt = static_cast<int32_t>(item - it.l * TR);
  const int r = __ldg(a.tile_req + it.rt);
  const int32_t tr0 = __ldg(a.tile_off + r);
  const int32_t j = it.rt - tr0;
  const int64_t tok0 = __ldg(a.tok_off + r);
  it.N = __ldg(a.tok_off + r + 1) - tok0;
  it.t0 = tok0 + static_cast<int64_t>(j) * kTileTokens;
  const int64_t left = it.N - static_cast<int64_t>(j) * kTileTokens;
  it.cnt = static_cast<int>(left < kTileTokens ? left : kTileTokens);
  return it;
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
    const float thr_h = __fdiv_rn(a.alpha_h, static_cast<float>(cur.N));
    const float thr_l = __fdiv_rn(a.alpha_l, static_cast<float>(cur.N));
    // Reciprocal test: with rc the hardware reciprocal of n (within 1 ulp),
    // y = RN(m * rc) is within 2^-22 (relative) of m / n, so y >= thr (1 + 2^-19)
    // proves RN(m / n) >= thr and y <= thr (1 - 2^-19) proves RN(m / n) < thr
    // (the margins, themselves rounded, stay far from 2^-22); in between, and
    // for thresholds below 2^-100 where a tiny quotient could leave the
    // relative bound, the IEEE division decides.  A NaN fails every test and
    // goes to the division: pruned.
    const bool exact_only = !(thr_l >= 0x1p-100f);
    const float hi_h = __fmul_rn(thr_h, 1.0f + 0x1p-19f), lo_h = __fmul_rn(thr_h, 1.0f - 0x1p-19f);
    const float hi_l = __fmul_rn(thr_l, 1.0f + 0x1p-19f), lo_l = __fmul_rn(thr_l, 1.0f - 0x1p-19f);

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
          const float y = __fmul_rn(m, rc);
          if (!exact_only && y >= hi_h) {
            c = DKV_CLASS_K8V4;
          } else if (!exact_only && !(y > lo_h) && y >= hi_l) {
            c = DKV_CLASS_K4V2;
          } else if (!exact_only && !(y > lo_h) && !(y > lo_l)) {
            c = DKV_CLASS_PRUNE;
          } else {
            const float s = __fdiv_rn(m, cf);
            c = s >= thr_h ? DKV_CLASS_K8V4 : (s >= thr_l ? DKV_CLASS_K4V2 : DKV_CLASS_PRUNE);
          }
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

size_t classify_smem(int Hq, int Hkv) {
  return sizeof(float) * kTileTokens * (Hq + 1) + sizeof(int32_t) * kTileTokens + kTileTokens * Hkv;
}

}  // namespace

cudaError_t launch_prep(const CompactArgs &a, cudaStream_t s) {
  const int32_t npart = static_cast<int32_t>((a.U + kScanUnits - 1) / kScanUnits);
  k_prep<<<1, kPrepThreads, 0, s>>>(a, npart);
  return cudaGetLastError();
}

cudaError_t launch_classify(const CompactArgs &a, int grid, cudaStream_t s) {
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
  return cudaGetLastError();
}

}  // namespace dkv
