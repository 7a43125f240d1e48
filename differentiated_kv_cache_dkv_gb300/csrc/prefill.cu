// prefill.cu -- causal prefill attention that also produces the significance
// inputs of compaction (dkv_prefill_attention), on the fifth-generation tensor
// cores (tcgen05, accumulators in tensor memory) with TMA-staged operands.
//
// DiffKV (arXiv 2412.03131), Pith review, "What carries the argument": a
// token's significance is the average attention it receives from the tokens
// after it; Referee Report, major comment 2: the average is over the N - i
// scores token i receives.  So the prefill attention that computes
//   out_i = sum_{j <= i} p(i, j) v_j,   p(i, .) = softmax_j(scale q_i . k_j)
// is also where sig_sum[j] = sum_{i >= j} p(i, j) and sig_cnt[j] = N - j are
// produced; the compaction reads exactly these.
//
// One CTA of 8 warps per (128-query tile, request, layer x query head): warp
// w reads tensor-memory lanes 32 (w mod 4) .. + 31 (the rows it owns) and
// columns 64 (w div 4) .. + 63 of each row, so two threads share a row and
// its row statistics meet once, after pass 1.  Key tiles are 128 keys.  Operands are staged by TMA with the 128-byte swizzle, 64 channels
// (128 bytes) per box row, two boxes per 128-channel tile:
//   S = Q K^T     tcgen05.mma kind::f16, A = Q (K-major, bf16), B = K
//                 (K-major, bf16), D = 128 x 128 fp32 in tensor-memory
//                 columns [0, 128); products exact, fp32 accumulation
//   O += P V      A = P rounded to bf16, held in tensor memory over the S
//                 columns already read (keys 0-63 in columns [0, 32), keys
//                 64-127 in [64, 96), two probabilities per column), B = V as
//                 it lies in memory (keys x channels: MN-major), D = O in
//                 columns [128, 256)
// Pass 1 runs S over the key tiles for each row's maximum and sum (online);
// pass 2 runs S again, forms the exact probabilities p = exp(S - m) / l in
// fp32 (one multiply-add into log2 units and ex2), adds their column sums
// (fp32, through a per-warp shared-memory transpose, then one atomic per key
// and tile) to the keys' significance sums, and accumulates O.  Rows are
// processed in rolled chunks of 32 columns, which keeps the code within the
// instruction cache and the registers at two CTAs per SM.  Two passes because a column sum needs the final
// normaliser of every row it crosses.
//
// Early prefetch: in pass 1 the V buffer is a second K buffer and two K tiles
// are in flight; in pass 2 the next K tile is requested as soon as the MMA
// that read the current one has completed, the next V tile as soon as P V
// has.  Two CTAs share an
// SM (about 107 KB of shared memory and 256 tensor-memory columns each).
// Every mbarrier wait is bounded by the global timer; a CTA that gives up
// records DKV_E_TIMEOUT, waits (bounded) for its own copies and MMAs, frees its
// tensor memory and leaves.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kTile = 128;                  // queries per CTA, keys per key tile
constexpr int kThreadsP = 256;              // two threads per query row, 64 columns each
constexpr uint32_t kTmemCols = 256;         // S in [0, 128), O in [128, 256)
constexpr uint32_t kColO = 128;
constexpr uint32_t kBoxBytes = 128 * 128;   // one TMA box: 128 rows x 64 bf16
constexpr uint32_t kTileBytes = 2 * kBoxBytes;
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr uint32_t kWaitPolls = 1u << 26;

struct __align__(1024) PrefillSmem {
  uint8_t q[kTileBytes];       // Q tile: box 0 (channels 0-63), box 1 (64-127)
  uint8_t k[kTileBytes];       // K tile
  uint8_t v[kTileBytes];       // V tile (pass 2) or the second K buffer (pass 1)
  float tr[8][32 * 8];         // per-warp transpose of 8 probability columns
  float part[4][kTile];        // column sums of the key tile per row quarter
  float2 stat[2][kTile];       // pass-1 (max, sum) of each row's two column halves
  uint64_t bar_q, bar_k, bar_v, bar_mma;
  uint32_t tmem;               // tensor-memory base address from tcgen05.alloc
  int32_t abort;               // a bounded wait gave up: skip the rest
  int64_t start;
  int32_t lens_ok;
};
constexpr size_t kPrefillSmem = sizeof(PrefillSmem) + 1024;  // + alignment slack

// ------------------------------------------------------------ PTX helpers --

__device__ __forceinline__ uint32_t saddr(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count) : "memory");
}

// Arrive (the barrier's one expected arrival) and expect `bytes` of copies.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(saddr(bar)),
               "r"(bytes)
               : "memory");
}

// Bounded wait for the phase of the given parity: false after about kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t addr = saddr(bar);
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

// TMA load of one box of a 3-D tensor map at (channel c0, head c1, row c2).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(saddr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(saddr(bar))
      : "memory");
}

// One 128-row x 128-channel tile: both 64-channel boxes on one barrier.
__device__ __forceinline__ void load_tile(uint8_t *dst, const CUtensorMap *map, int head, int row, uint64_t *bar) {
  mbar_expect_tx(bar, kTileBytes);
  tma_load_3d(dst, map, 0, head, row, bar);
  tma_load_3d(dst + kBoxBytes, map, 64, head, row, bar);
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a 128-byte-swizzled operand: start
// address, leading and stride byte offsets (16-byte units), descriptor
// version 1, swizzle mode 2 (128 bytes).  Tiles are 1024-byte aligned, so the
// base-offset field stays 0.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((addr >> 4) & 0x3fffu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3fffu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3fffu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, A
// K-major, B K-major (b_mn = false) or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// The barrier receives one arrival when every MMA this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
               : "memory");
}

// 32 consecutive fp32 columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&x)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// 2^x by the special-function unit (relative error about 2^-22; results
// below 2^-126 flush to zero, far below any probability that matters).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// bf16 pair rounded to nearest even, the lower-indexed value in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Where request r starts in the token axis, from the lengths, validated by
// warp 0 of the block before anything is read or written: every lens[q] must
// lie in [0, max_len] and they must add up to T.  Returns false (after the
// failing block records DKV_E_LENS) when they do not.  Every thread of the
// block must call it.
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

// Column sums of one 32-column chunk of this tile's probabilities over the
// warp's 32 rows: four rounds of 8 columns through the warp's shared-memory
// transpose, 8 words per row.  Row r keeps its two 4-column halves swapped
// when bit 2 of r is set, so a quarter-warp's two 16-byte stores hit 32
// distinct banks; lane (g, c) sums column c over rows 8g .. 8g + 7, group g
// taking them in the order starting at row 8g + g, so the four groups' loads
// hit distinct banks too.  off: this lane's word offsets, computed once
// (two stores, then eight loads).  Lanes 0-7 end with the sums of a round's
// columns, written to part[row quarter][column].
__device__ __forceinline__ void chunk_column_sums(PrefillSmem &sm, const float (&p)[32], int col0,
                                                  const int (&off)[10]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float *tr = sm.tr[warp];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    *reinterpret_cast<float4 *>(tr + off[0]) = make_float4(p[8 * r], p[8 * r + 1], p[8 * r + 2], p[8 * r + 3]);
    *reinterpret_cast<float4 *>(tr + off[1]) = make_float4(p[8 * r + 4], p[8 * r + 5], p[8 * r + 6], p[8 * r + 7]);
    __syncwarp();
    float s0 = tr[off[2]] + tr[off[3]], s1 = tr[off[4]] + tr[off[5]];
    float s2 = tr[off[6]] + tr[off[7]], s3 = tr[off[8]] + tr[off[9]];
    float s = (s0 + s1) + (s2 + s3);
    s += __shfl_xor_sync(0xffffffffu, s, 8);
    s += __shfl_xor_sync(0xffffffffu, s, 16);
    if (lane < 8) sm.part[warp & 3][col0 + 8 * r + lane] = s;
    __syncwarp();
  }
}

// Word offset of (row, column) in the transpose above.
__device__ __forceinline__ int tr_word(int row, int col) {
  return 8 * row + 4 * ((col >> 2) ^ ((row >> 2) & 1)) + (col & 3);
}

__global__ void __launch_bounds__(kThreadsP, 2)
    k_prefill(PrefillArgs a, const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
              const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ unsigned char smem_raw[];
  PrefillSmem &sm =
      *reinterpret_cast<PrefillSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rq = warp & 3, ch = warp >> 2;  // row quarter (tensor-memory lanes), column half
  const int32_t r = blockIdx.y;
  const int32_t l = static_cast<int32_t>(blockIdx.z / a.Hq), qh = static_cast<int32_t>(blockIdx.z % a.Hq);
  const int32_t h = qh / a.G;
  int64_t start = 0;
  // before any allocation: leaving early is safe
  if (!request_start(a, r, &sm.start, &sm.lens_ok, start)) return;
  const int32_t n = __ldg(a.lens + r);
  const int32_t ntq = (n + kTile - 1) / kTile;
  const int32_t qt = ntq - 1 - static_cast<int32_t>(blockIdx.x);  // longest rows first
  if (qt < 0) return;
  const int64_t row0 = static_cast<int64_t>(l) * a.T + start;    // (layer, request) token row 0
  const int32_t nkt = qt + 1;                                      // key tiles the causal rows reach
  const int row = 32 * rq + lane;                                  // this thread's row of the tile
  const int32_t qrow = qt * kTile + row;                           // its query position
  // a row past the request masks every key (qlim = -1); masks are applied
  // per element only in the diagonal tile and in a tile with such rows
  const int32_t qlim = qrow < n ? qrow : -1;
  const bool ragged = (qt + 1) * kTile > n;
  const float sl2 = a.scale * 1.44269504088896340736f;             // logits in log2 units
  int tro[10];  // the column-sum transpose's word offsets for this lane
  {
    const int g = lane >> 3, c = lane & 7;
    tro[0] = tr_word(lane, 0);
    tro[1] = tr_word(lane, 4);
#pragma unroll
    for (int k = 0; k < 8; ++k) tro[2 + k] = tr_word(8 * g + ((k + g) & 7), c);
  }

  if (tid == 0) {
    mbar_init(&sm.bar_q, 1);
    mbar_init(&sm.bar_k, 1);
    mbar_init(&sm.bar_v, 1);
    mbar_init(&sm.bar_mma, 1);
    sm.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&sm.tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * rq) << 16);  // this warp's lanes
  const uint32_t s_cols = lane_base + 64 * ch;                                // its 64 columns of S

  constexpr uint32_t idesc_s = idesc_bf16(128, 128, false);
  constexpr uint32_t idesc_o = idesc_bf16(128, 128, true);
  const uint32_t q_s = saddr(sm.q), k_s = saddr(sm.k), v_s = saddr(sm.v);

  // Per barrier: phases issued (copies or MMA commits requested; every
  // thread counts them, the decisions are uniform) and phases waited for
  // (the parity of the next wait).
  uint32_t iss_q = 0, iss_k = 0, iss_v = 0, iss_mma = 0;
  uint32_t ph_q = 0, ph_k = 0, ph_v = 0, ph_mma = 0;
  bool ok = true;
  // every thread waits; a failure anywhere aborts the whole CTA (the phase
  // stays counted as outstanding)
  auto wait_all = [&](uint64_t *bar, uint32_t &ph) {
    const bool w = mbar_wait(bar, ph & 1u);
    if (w) ph++;
    if (!w) {
      sm.abort = 1;
      set_error(a.status, DKV_E_TIMEOUT);
    }
    __syncthreads();
    ok = ok && sm.abort == 0;
  };

  // S = Q K^T of the key tile staged at kbuf into columns [0, 128): eight
  // K-steps of 16 channels, 32 bytes along the swizzled 128-byte rows, the
  // second four in the second box
  auto issue_s = [&](uint32_t kbuf) {
    iss_mma++;
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
        mma_ss(tmem, sw128_desc(q_s + off, 16, 1024), sw128_desc(kbuf + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
      }
      mma_commit(&sm.bar_mma);
    }
  };

  // ---- prologue: Q and the first two K tiles
  if (tid == 0) {
    load_tile(sm.q, &qmap, qh, static_cast<int>(row0 + qt * kTile), &sm.bar_q);
    load_tile(sm.k, &kmap, h, static_cast<int>(row0), &sm.bar_k);
    if (nkt > 1) load_tile(sm.v, &kmap, h, static_cast<int>(row0 + kTile), &sm.bar_v);
  }
  iss_q = 1;
  iss_k = 1;
  iss_v = nkt > 1 ? 1 : 0;
  wait_all(&sm.bar_q, ph_q);

  // ---- pass 1: row maximum and sum of this thread's 64 columns (log2
  // units).  Key tile kt sits in buffer kt & 1 (k, then v); two tiles are in
  // flight: tile kt + 2 is requested into tile kt's buffer once S of tile kt
  // is done.
  float m = -INFINITY, lsum = 0.0f;
  for (int32_t kt = 0; kt < nkt && ok; ++kt) {
    uint64_t *bar = (kt & 1) ? &sm.bar_v : &sm.bar_k;
    uint32_t &ph = (kt & 1) ? ph_v : ph_k;
    wait_all(bar, ph);
    if (!ok) break;
    issue_s((kt & 1) ? v_s : k_s);
    wait_all(&sm.bar_mma, ph_mma);
    if (!ok) break;
    if (kt + 2 < nkt) {
      if (tid == 0)
        load_tile((kt & 1) ? sm.v : sm.k, &kmap, h, static_cast<int>(row0 + (kt + 2) * kTile), bar);
      if (kt & 1) iss_v++; else iss_k++;
    }
    tc_fence_after();
    const bool masked = kt == qt || ragged;
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      float x[32];
      tmem_ld32(s_cols + 32 * c, x);
      const int32_t key0 = kt * kTile + 64 * ch + 32 * c;
      float mx = -INFINITY;
      if (masked) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = key0 + i <= qlim ? x[i] * sl2 : -INFINITY;
          mx = fmaxf(mx, x[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] *= sl2;
          mx = fmaxf(mx, x[i]);
        }
      }
      const float mn = fmaxf(m, mx);
      if (mn != -INFINITY) {
        float t = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) t += ex2(x[i] - mn);
        lsum = lsum * ex2(m - mn) + t;  // ex2(-inf) = 0 on the first chunk
        m = mn;
      }
    }
    tc_fence_before();
    __syncthreads();  // S is read: its columns may be overwritten
  }
  // the two column halves of a row meet: m = max, l = sum of rescaled sums
  sm.stat[ch][row] = make_float2(m, lsum);
  __syncthreads();
  {
    const float2 o = sm.stat[ch ^ 1][row];
    const float mn = fmaxf(m, o.x);
    if (mn != -INFINITY) {
      lsum = lsum * ex2(m - mn) + o.y * ex2(o.x - mn);
      m = mn;
    }
  }
  const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;  // 0 for a row past the request

  // ---- pass 2: probabilities, column sums, O += P V.  Tile kt + 1's K is
  // requested after S of tile kt, its V after P V of tile kt.
  if (ok) {
    if (tid == 0) {
      load_tile(sm.k, &kmap, h, static_cast<int>(row0), &sm.bar_k);
      load_tile(sm.v, &vmap, h, static_cast<int>(row0), &sm.bar_v);
    }
    iss_k++;
    iss_v++;
  }
  for (int32_t kt = 0; kt < nkt && ok; ++kt) {
    wait_all(&sm.bar_k, ph_k);
    if (!ok) break;
    issue_s(k_s);
    wait_all(&sm.bar_mma, ph_mma);
    if (!ok) break;
    if (kt + 1 < nkt) {
      if (tid == 0) load_tile(sm.k, &kmap, h, static_cast<int>(row0 + (kt + 1) * kTile), &sm.bar_k);
      iss_k++;
    }
    tc_fence_after();
    const bool masked = kt == qt || ragged;
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      float x[32];
      tmem_ld32(s_cols + 32 * c, x);
      const int32_t key0 = kt * kTile + 64 * ch + 32 * c;
      if (masked) {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = key0 + i <= qlim ? ex2(__fmaf_rn(x[i], sl2, -m)) * inv : 0.0f;
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = ex2(__fmaf_rn(x[i], sl2, -m)) * inv;
      }
      chunk_column_sums(sm, x, 64 * ch + 32 * c, tro);
      // P (bf16 pairs) of keys 64 ch + 32 c .. + 31 into columns
      // 64 ch + 16 c .. + 15: S columns this warp has already read, so no
      // other warp's S is overwritten
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = bf16x2_rn(x[2 * i], x[2 * i + 1]);
      tmem_st16(s_cols + 16 * c, w);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    {  // every column's four row-quarter sums -> one atomic per key
      const int32_t key = kt * kTile + tid;
      if (tid < kTile && key < n) {
        const float s = sm.part[0][tid] + sm.part[1][tid] + sm.part[2][tid] + sm.part[3][tid];
        if (s != 0.0f) atomicAdd(a.sig_sum + (row0 + key) * a.Hq + qh, s);
      }
    }
    wait_all(&sm.bar_v, ph_v);  // (its barrier also keeps part[] until every sum is read)
    if (!ok) break;
    iss_mma++;
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // keys 16 kk .. + 15: 8 columns of P (at 64 (kk / 4) + 8 (kk % 4)), 16 rows of V
        mma_ts(tmem + kColO, tmem + 64 * (kk >> 2) + 8 * (kk & 3), sw128_desc(v_s + kk * 2048, kBoxBytes, 1024),
               idesc_o, (kt > 0 || kk > 0) ? 1u : 0u);
      mma_commit(&sm.bar_mma);
    }
    wait_all(&sm.bar_mma, ph_mma);
    if (!ok) break;
    if (kt + 1 < nkt) {
      if (tid == 0) load_tile(sm.v, &vmap, h, static_cast<int>(row0 + (kt + 1) * kTile), &sm.bar_v);
      iss_v++;
    }
  }

  // ---- outputs: this thread's 64 channels of its row of O (the loads are
  // warp-collective, so every lane takes them; rows past the request store
  // nothing)
  if (ok) {
    tc_fence_after();
    float *dst = a.out + ((row0 + qrow) * a.Hq + qh) * 128 + 64 * ch;
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      float x[32];
      tmem_ld32(lane_base + kColO + 64 * ch + 32 * c, x);
      if (qrow < n) {
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4 *>(dst + 32 * c + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
      }
    }
  }

  // ---- teardown: after an abort, wait (bounded) for this CTA's own copies
  // and MMAs, so none outlives it; then free the tensor memory
  if (!ok && tid == 0) {
    for (; ph_q < iss_q; ++ph_q) mbar_wait(&sm.bar_q, ph_q & 1u);
    for (; ph_k < iss_k; ++ph_k) mbar_wait(&sm.bar_k, ph_k & 1u);
    for (; ph_v < iss_v; ++ph_v) mbar_wait(&sm.bar_v, ph_v & 1u);
    for (; ph_mma < iss_mma; ++ph_mma) mbar_wait(&sm.bar_mma, ph_mma & 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
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

// 3-D tensor map over a bf16 [rows][H][128] array whose box is 64 channels of
// one head for 128 consecutive rows, written to shared memory with the
// 128-byte swizzle (rows past the array read as zeros).
cudaError_t make_map(CUtensorMap *map, const void *base, int64_t rows, int32_t H) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult qr;
    void *fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr);
    if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(H) * 256};
  const cuuint32_t box[3] = {64, 1, kTile};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult res = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t s) {
  if (a.R == 0 || a.max_len == 0) return cudaSuccess;
  k_sigcnt<<<dim3(std::min((a.max_len + 255) / 256, 64), a.R), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t rows = static_cast<int64_t>(a.L) * a.T;
  if (rows < 1) return cudaSuccess;
  alignas(64) CUtensorMap qmap, kmap, vmap;
  if ((e = make_map(&qmap, a.q, rows, a.Hq)) != cudaSuccess) return e;
  if ((e = make_map(&kmap, a.k, rows, a.Hkv)) != cudaSuccess) return e;
  if ((e = make_map(&vmap, a.v, rows, a.Hkv)) != cudaSuccess) return e;
  const int smem = static_cast<int>(kPrefillSmem);
  if ((e = cudaFuncSetAttribute(k_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
  const dim3 grid((a.max_len + kTile - 1) / kTile, a.R, static_cast<unsigned>(a.L) * a.Hq);
  k_prefill<<<grid, kThreadsP, smem, s>>>(a, qmap, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace dkv
