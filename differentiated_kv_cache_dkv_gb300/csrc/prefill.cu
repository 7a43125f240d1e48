// prefill.cu -- causal prefill attention that also produces the significance
// inputs of compaction (dkv_prefill_attention).
//
// DiffKV (arXiv 2412.03131), Pith review, "What carries the argument": a
// token's significance is the average attention it receives from the tokens
// after it; Referee Report, major comment 2: the average is over the N - i
// scores token i receives.  So the prefill attention that computes
//   out_i = sum_{j <= i} p(i, j) v_j,   p(i, .) = softmax_j(scale q_i . k_j)
// is also where sig_sum[j] = sum_{i >= j} p(i, j) and sig_cnt[j] = N - j are
// produced; the compaction reads exactly these.
//
// One block of 4 warps per (64-query tile, request, layer x query head); a
// warp owns 16 query rows.  Key tiles of 64 are staged in shared memory: K as
// bf16 rows (padded against bank conflicts), V transposed to fp16.
//   pass 1   S = Q K^T on the tensor cores (bf16 x bf16, exact products, fp32
//            accumulation); the running row maximum and sum;
//   pass 2   S again; P = exp(S - m) / l exactly normalised; O += P V on the
//            tensor cores (P as two fp16 parts: nearest and remainder), and
//            the column sums of P over the block's rows are added to the
//            keys' significance sums (fp32 atomics across query tiles).
// Two passes over K because a column sum needs the final normaliser of every
// row it crosses.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kQ = 64;          // queries per block (16 per warp)
constexpr int kK = 64;          // keys per tile
constexpr int kWarpsP = 4;
constexpr int kThreadsP = 32 * kWarpsP;
constexpr int kKStride = 136;   // bf16 per staged K row (128 + 8: spreads the rows over the banks)
constexpr int kVStride = 72;    // fp16 per staged V^T row (64 keys + 8)
constexpr unsigned kFullP = 0xffffffffu;

struct PrefillSmem {
  uint16_t k[kK][kKStride];   // bf16 bits
  __half vt[128][kVStride];
  float cs[kWarpsP][kK];
  int64_t start;
  int32_t lens_ok;
};

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (nearest, remainder) fp16 parts of two floats, packed as two half2 words.
__device__ __forceinline__ void split2(float x, float y, uint32_t &hi, uint32_t &lo) {
  const __half hx = __float2half_rn(x), hy = __float2half_rn(y);
  const __half lx = __float2half_rn(x - __half2float(hx)), ly = __float2half_rn(y - __half2float(hy));
  hi = static_cast<uint32_t>(__half_as_ushort(hx)) | (static_cast<uint32_t>(__half_as_ushort(hy)) << 16);
  lo = static_cast<uint32_t>(__half_as_ushort(lx)) | (static_cast<uint32_t>(__half_as_ushort(ly)) << 16);
}

// Where request r starts in the token axis, from the lengths, validated by
// warp 0 of the block before anything is read or written: every lens[q] must
// lie in [0, max_len] and they must add up to T.  Returns false (after the
// first failing block records DKV_E_LENS) when they do not.  Every thread of
// the block must call it.
__device__ __forceinline__ bool request_start(const PrefillArgs &a, int32_t r, int64_t *start_sm, int32_t *ok_sm,
                                              int64_t &start) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int64_t before = 0, total = 0;
    int bad = 0;
    for (int32_t q = lane; q < a.R; q += 32) {
      const int32_t n = __ldg(a.lens + q);
      if (n < 0 || n > a.max_len) bad = 1;
      total += n;
      if (q < r) before += n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, o);
      total += __shfl_xor_sync(0xffffffffu, total, o);
      bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    if (lane == 0) {
      const bool ok = !bad && total == a.T;
      *start_sm = before;
      *ok_sm = ok ? 1 : 0;
      if (!ok) set_error(a.status, DKV_E_LENS);
    }
  }
  __syncthreads();
  start = *start_sm;
  return *ok_sm != 0;
}

// Stage key tile [kb, kb + kK) of (layer, KV head): K rows as they are, V
// transposed to fp16; keys at or past n are zero.
__device__ __forceinline__ void stage(PrefillSmem &sm, const PrefillArgs &a, int64_t row0, int32_t h, int32_t kb,
                                     int32_t n, bool with_v) {
  // K: 64 keys x 16 chunks of 16 bytes, a key's chunks on consecutive threads
  for (int c = threadIdx.x; c < kK * 16; c += kThreadsP) {
    const int key = c >> 4, ch = c & 15;
    uint4 kv = make_uint4(0, 0, 0, 0);
    if (kb + key < n) kv = __ldg(reinterpret_cast<const uint4 *>(a.k + ((row0 + kb + key) * a.Hkv + h) * 128 + ch * 8));
    *reinterpret_cast<uint4 *>(&sm.k[key][ch * 8]) = kv;
  }
  if (!with_v) return;
  // V transposed: consecutive threads take consecutive keys of one chunk, so
  // their 2-byte stores into a V^T row are consecutive
  for (int c = threadIdx.x; c < kK * 16; c += kThreadsP) {
    const int key = c & (kK - 1), ch = c / kK;
    uint4 vv = make_uint4(0, 0, 0, 0);
    if (kb + key < n) vv = __ldg(reinterpret_cast<const uint4 *>(a.v + ((row0 + kb + key) * a.Hkv + h) * 128 + ch * 8));
    const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t b = (e & 1) ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16);
      sm.vt[ch * 8 + e][key] = __float2half_rn(__uint_as_float(b));
    }
  }
}

// S for this warp's 16 rows and the staged 64 keys: c[nt] holds rows g, g + 8
// and keys nt * 8 + 2t, + 1 (lane (g, t)), scaled, with keys past the row, and
// every key of a row past the request, masked to -inf.
__device__ __forceinline__ void scores(const PrefillSmem &sm, const uint32_t (&qa)[8][4], float (&c)[8][4], int32_t i0,
                                       int32_t kb, int32_t n, float scale) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t b0 = *reinterpret_cast<const uint32_t *>(&sm.k[nt * 8 + g][16 * ks + 2 * t]);
      const uint32_t b1 = *reinterpret_cast<const uint32_t *>(&sm.k[nt * 8 + g][16 * ks + 2 * t + 8]);
      mma_bf16(c[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int32_t row = i0 + g + ((e & 2) ? 8 : 0);
      const int32_t key = kb + nt * 8 + 2 * t + (e & 1);
      c[nt][e] = (key <= row && row < n) ? c[nt][e] * scale : -INFINITY;  // rows past the request attend nothing
    }
  }
}

__global__ void __launch_bounds__(kThreadsP) k_prefill(PrefillArgs a) {
  __shared__ __align__(16) PrefillSmem sm;
  const int32_t r = blockIdx.y;
  const int32_t l = static_cast<int32_t>(blockIdx.z / a.Hq), qh = static_cast<int32_t>(blockIdx.z % a.Hq);
  const int32_t h = qh / a.G;
  const int32_t qb = blockIdx.x * kQ;
  int64_t start = 0;
  // no cluster or grid barrier: leaving early is safe
  if (!request_start(a, r, &sm.start, &sm.lens_ok, start)) return;
  const int32_t n = __ldg(a.lens + r);
  if (qb >= n) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
  const int32_t i0 = qb + 16 * warp;                  // this warp's first row
  const int64_t row0 = static_cast<int64_t>(l) * a.T + start;  // (layer, request) token row 0

  // Q fragments: rows i0 + g, i0 + g + 8; 16-dim steps ks
  uint32_t qa[8][4];
  {
    const int32_t ra = i0 + g, rb = i0 + g + 8;
    const uint32_t *pa = reinterpret_cast<const uint32_t *>(a.q + ((row0 + ra) * a.Hq + qh) * 128);
    const uint32_t *pb = reinterpret_cast<const uint32_t *>(a.q + ((row0 + rb) * a.Hq + qh) * 128);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa[ks][0] = ra < n ? __ldg(pa + 8 * ks + t) : 0u;
      qa[ks][1] = rb < n ? __ldg(pb + 8 * ks + t) : 0u;
      qa[ks][2] = ra < n ? __ldg(pa + 8 * ks + t + 4) : 0u;
      qa[ks][3] = rb < n ? __ldg(pb + 8 * ks + t + 4) : 0u;
    }
  }
  const int32_t kend = min(n, qb + kQ);  // keys any row of the block reaches
  const int32_t ntile = (kend + kK - 1) / kK;
  const float scale = a.scale;

  // ---- pass 1: row maximum and sum (rows g and g + 8 of the warp)
  float m[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.0f, 0.0f};
  for (int32_t kt = 0; kt < ntile; ++kt) {
    __syncthreads();  // the previous tile is no longer read
    stage(sm, a, row0, h, kt * kK, n, false);
    __syncthreads();
    float c[8][4];
    scores(sm, qa, c, i0, kt * kK, n, scale);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) mx = fmaxf(mx, fmaxf(c[nt][2 * hr], c[nt][2 * hr + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(kFullP, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kFullP, mx, 2));
      const float mn = fmaxf(m[hr], mx);
      if (mn == -INFINITY) continue;  // nothing attended yet (rows past the request)
      float s = 0.0f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) s += __expf(c[nt][2 * hr] - mn) + __expf(c[nt][2 * hr + 1] - mn);
      lsum[hr] = lsum[hr] * (m[hr] == -INFINITY ? 0.0f : __expf(m[hr] - mn)) + s;
      m[hr] = mn;
    }
  }
  float inv[2];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    lsum[hr] += __shfl_xor_sync(kFullP, lsum[hr], 1);
    lsum[hr] += __shfl_xor_sync(kFullP, lsum[hr], 2);
    inv[hr] = lsum[hr] > 0.0f ? 1.0f / lsum[hr] : 0.0f;
  }

  // ---- pass 2: probabilities, outputs, column sums
  float o[16][4];
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.0f;
  for (int32_t kt = 0; kt < ntile; ++kt) {
    __syncthreads();
    stage(sm, a, row0, h, kt * kK, n, true);
    __syncthreads();
    float c[8][4];
    scores(sm, qa, c, i0, kt * kK, n, scale);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e >> 1;
        c[nt][e] = (c[nt][e] == -INFINITY || m[hr] == -INFINITY) ? 0.0f : __expf(c[nt][e] - m[hr]) * inv[hr];
      }
      // column sums over the warp's 16 rows: keys nt * 8 + 2t, + 1
      float s0 = c[nt][0] + c[nt][2], s1 = c[nt][1] + c[nt][3];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        s0 += __shfl_xor_sync(kFullP, s0, off);
        s1 += __shfl_xor_sync(kFullP, s1, off);
      }
      if (g == 0) {
        sm.cs[warp][nt * 8 + 2 * t] = s0;
        sm.cs[warp][nt * 8 + 2 * t + 1] = s1;
      }
    }
    // O += P V: key steps kk (n-tiles 2kk, 2kk + 1 of S), 16 dim tiles nd
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t ah[4], al[4];
      split2(c[2 * kk][0], c[2 * kk][1], ah[0], al[0]);
      split2(c[2 * kk][2], c[2 * kk][3], ah[1], al[1]);
      split2(c[2 * kk + 1][0], c[2 * kk + 1][1], ah[2], al[2]);
      split2(c[2 * kk + 1][2], c[2 * kk + 1][3], ah[3], al[3]);
#pragma unroll
      for (int nd = 0; nd < 16; ++nd) {
        const uint32_t b0 = *reinterpret_cast<const uint32_t *>(&sm.vt[nd * 8 + g][16 * kk + 2 * t]);
        const uint32_t b1 = *reinterpret_cast<const uint32_t *>(&sm.vt[nd * 8 + g][16 * kk + 2 * t + 8]);
        mma_f16(o[nd], ah[0], ah[1], ah[2], ah[3], b0, b1);
        mma_f16(o[nd], al[0], al[1], al[2], al[3], b0, b1);
      }
    }
    __syncthreads();  // column sums of all warps
    if (threadIdx.x < kK) {
      const int32_t key = kt * kK + threadIdx.x;
      if (key < n) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarpsP; ++w) s += sm.cs[w][threadIdx.x];
        if (s != 0.0f) atomicAdd(a.sig_sum + (row0 + key) * a.Hq + qh, s);
      }
    }
  }
  // ---- outputs: rows g, g + 8; dims nd * 8 + 2t, + 1
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int32_t row = i0 + g + 8 * hr;
    if (row >= n) continue;
    float *dst = a.out + ((row0 + row) * a.Hq + qh) * 128;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd)
      *reinterpret_cast<float2 *>(dst + nd * 8 + 2 * t) = make_float2(o[nd][2 * hr], o[nd][2 * hr + 1]);
  }
}

// sig_cnt[start_r + i] = N_r - i.
__global__ void __launch_bounds__(256) k_sigcnt(PrefillArgs a) {
  __shared__ int64_t start_sm;
  __shared__ int32_t ok_sm;
  const int32_t r = blockIdx.y;
  int64_t start = 0;
  if (!request_start(a, r, &start_sm, &ok_sm, start)) return;
  const int32_t n = __ldg(a.lens + r);
  for (int32_t i = blockIdx.x * 256 + threadIdx.x; i < n; i += gridDim.x * 256) a.sig_cnt[start + i] = n - i;
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t s) {
  if (a.R == 0 || a.max_len == 0) return cudaSuccess;
  k_sigcnt<<<dim3(std::min((a.max_len + 255) / 256, 64), a.R), 256, 0, s>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid((a.max_len + kQ - 1) / kQ, a.R, static_cast<unsigned>(a.L) * a.Hq);
  k_prefill<<<grid, kThreadsP, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dkv
