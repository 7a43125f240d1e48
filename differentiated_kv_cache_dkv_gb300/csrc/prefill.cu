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
// Persistent: one block per SM walks the work items, a 128-query tile of one
// (request, layer x query head) each, longest first; every role keeps its
// pipeline counters running from item to item, so the next item's copies and
// S MMAs overlap the end of the current one.  A block has 8 softmax warps, an
// S-issuing warp, a P V-issuing warp and a copy warp.
// Key tiles are 128 keys; Q, K and V tiles are staged by TMA with the
// 128-byte swizzle, 64 channels per box row, two boxes per 128-channel tile,
// K and V through a ring of four tile slots.  Two passes, because a key's
// significance needs the final normaliser of every row it meets:
//   pass 1  S = Q K^T (A = Q, B = K, both K-major; D = 128 x 128 fp32 in one
//           of three tensor-memory buffers, so S of later tiles runs while
//           this one is read): each row's maximum and sum, online, in log2
//           units.
//   pass 2  S^T = K Q^T (A = K, B = Q): one tensor-memory lane per KEY, so
//           p = exp2(s scale log2e - m_q - log2 l_q) is formed per key row
//           with the queries' m + log2 l broadcast from shared memory, and the
//           key's significance is a plain row sum in fp32 (two column
//           halves per key, one atomic each per tile).  P^T, rounded to
//           bf16, goes to shared memory as rows of keys with the queries
//           contiguous, which is P in the MN-major A form: O += P V with
//           A = P (MN-major), B = V as it lies in memory (keys x channels:
//           MN-major), D = O (128 x 128 fp32) in its own tensor-memory
//           columns.
// Warp w of the softmax group reads tensor-memory lanes 32 (w mod 4) .. + 31
// and columns 64 (w div 4) .. + 63 of a tile: two threads per row (pass 1)
// or key (pass 2), whose row statistics meet once, after pass 1.  S and P V
// are issued by separate warps, so P V of a tile never queues behind the
// wait for a later K tile.
// Every mbarrier wait is bounded by the global timer; a CTA that gives up
// records DKV_E_TIMEOUT, the copy and MMA warps wait (bounded) for their own
// copies and MMAs, and the tensor memory is freed.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>

#include "dkv_internal.cuh"

namespace dkv {

namespace {
constexpr int kTile = 128;                  // queries per CTA, keys per key tile
constexpr int kSoftmaxWarps = 8;            // two threads per row or key
constexpr int kQuarters = kSoftmaxWarps / 4;  // column groups of a row (warp w: lanes of w mod 4, group w div 4)
constexpr int kCols = 128 / kQuarters;      // columns of a tile per thread
static_assert(kCols == 64, "the softmax code below handles 64 columns per thread");
constexpr int kSWarp = kSoftmaxWarps;       // issues S (or S^T)
constexpr int kPvWarp = kSoftmaxWarps + 1;  // issues P V, adds the significance
constexpr int kLoadWarp = kSoftmaxWarps + 2;  // the copy warp
constexpr int kThreadsP = 32 * (kLoadWarp + 1);
constexpr int kSBuf = 3;                    // S buffers in tensor memory
constexpr uint32_t kTmemCols = 512;         // S buffers [0, 128), [128, 256), [256, 384); O [384, 512)
constexpr uint32_t kColO = 384;
constexpr uint32_t kBox = kTile * 128;      // one box: 128 rows x 64 bf16 (16 KB)
constexpr uint32_t kTileBytes = 2 * kBox;
constexpr int kSlots = 4;                   // K / V staging ring
constexpr int kPBuf = 2;                    // P^T buffers
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr uint32_t kWaitPolls = 1u << 26;

struct __align__(1024) PrefillSmem {
  uint8_t q[kTileBytes];             // Q tile: box 0 (channels 0-63), box 1 (64-127)
  uint8_t ring[kSlots][kTileBytes];  // K or V tiles, same two-box form
  // P^T in bf16, kPBuf buffers by key tile: [query half][128 keys][64
  // queries], 128-byte swizzle.  Before pass 2 the first holds the pass-1
  // (max, sum) of each row's column groups (float2 [kQuarters][128]).
  uint8_t pt[kPBuf][kTileBytes];
  float nlse[kTile];                 // per query: -(m + log2 l), its normaliser in log2 units
  uint64_t bar_q, bar_qfree;         // the item's Q landed; the S MMAs reading it are done
  uint64_t full[kSlots], empty[kSlots];  // a ring slot landed / was read by its MMAs
  uint64_t bar_s[kSBuf];             // S (or S^T) of a tile computed into buffer b
  uint64_t bar_sfree[kSBuf];         // the softmax warps have read buffer b
  uint64_t bar_pready[kPBuf];        // P^T of a pass-2 tile is in shared-memory buffer b
  uint64_t bar_o[kPBuf], bar_done;   // P V of a tile from buffer b done; the item's P V done
  uint64_t bar_ofree;                // the softmax warps have read the item's O
  uint64_t bar_sdone, bar_pvdone;    // every S, every P V of the block done
  uint32_t tmem;                     // tensor-memory base address from tcgen05.alloc
  int32_t abort;                     // a bounded wait gave up: everyone winds down
  int64_t start;
  int32_t lens_ok;
};
constexpr size_t kPrefillSmem = sizeof(PrefillSmem) + 1024;  // + alignment slack
static_assert(kPrefillSmem <= 227 * 1024, "shared memory");

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

// Bounded wait for the phase of the given parity: false after about kWaitNs,
// or as soon as *abort (when given) is set by another thread.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const volatile int32_t *abort) {
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
      if (abort && *abort) return false;
      const uint64_t t = global_ns();
      if (t0 == 0) t0 = t;
      else if (t - t0 > kWaitNs) return false;
    }
  }
  return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(saddr(bar)) : "memory");
}

// Named barrier of the softmax warps only.
__device__ __forceinline__ void softmax_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kSoftmaxWarps) : "memory");
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

// One 128-row tile (both 64-channel boxes) on one barrier.
__device__ __forceinline__ void load_tile(uint8_t *dst, const CUtensorMap *map, int head, int row, uint64_t *bar) {
  mbar_expect_tx(bar, kTileBytes);
  tma_load_3d(dst, map, 0, head, row, bar);
  tma_load_3d(dst + kBox, map, 64, head, row, bar);
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

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, A and
// B K-major or MN-major (a_mn, b_mn), shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// The barrier receives one arrival when every MMA this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
               : "memory");
}

// 64 consecutive fp32 columns of this thread's lane.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&x)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, "
      "%38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, "
      "%60, %61, %62, %63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]),
        "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]),
        "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
        "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]),
        "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) x[i] = __uint_as_float(r[i]);
}

// 2^x by the special-function unit (relative error about 2^-22; results
// below 2^-126 flush to zero, far below any probability that matters).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (one instruction for two lanes of work, each rounded to
// nearest like the scalar operation).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of 32 values as a tree of three-input maxima.
__device__ __forceinline__ float max32(const float (&v)[32]) {
  float t[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) t[i] = max3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  t[10] = fmaxf(v[30], v[31]);
  const float u0 = max3(t[0], t[1], t[2]), u1 = max3(t[3], t[4], t[5]), u2 = max3(t[6], t[7], t[8]);
  return max3(max3(u0, u1, u2), t[9], t[10]);
}

// v[i] <- 2^(v[i] * sl2 - mo) for 32 values, in packed pairs; returns their
// sum (a tree of packed additions).
__device__ __forceinline__ float exp2_sum32(float (&v)[32], float sl2, float mo) {
  const uint64_t s2 = f2_pack(sl2, sl2), m2 = f2_pack(-mo, -mo);
  uint64_t e[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float a, b;
    f2_unpack(f2_fma(f2_pack(v[2 * i], v[2 * i + 1]), s2, m2), a, b);
    e[i] = f2_pack(ex2(a), ex2(b));
  }
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) e[i] = f2_add(e[i], e[i + w]);
  float lo, hi;
  f2_unpack(e[0], lo, hi);
  return lo + hi;
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

// One work item: a 128-query tile of one (layer, request, query head).
struct PfItem {
  int64_t row0;  // (layer, request) token row 0
  int32_t qt, n, qh, h, nk;
  bool ragged;   // rows past the request in this tile
};

// Item i of the longest-first order: the query tile counted from the end of
// its request slowest, then the request, then layer x query head.  false
// when the request has no such tile.
__device__ __forceinline__ bool pf_item(const PrefillArgs &a, int64_t i, PfItem &it) {
  const int64_t Z = static_cast<int64_t>(a.L) * a.Hq;
  const int64_t per = static_cast<int64_t>(a.R) * Z;
  const int32_t qt_rev = static_cast<int32_t>(i / per);
  const int64_t rest = i - qt_rev * per;
  const int32_t r = static_cast<int32_t>(rest / Z);
  const int32_t z = static_cast<int32_t>(rest - static_cast<int64_t>(r) * Z);
  const int32_t n = __ldg(a.lens + r);
  const int32_t ntq = (n + kTile - 1) / kTile;
  if (qt_rev >= ntq) return false;
  int64_t start = 0;
  for (int32_t q = 0; q < r; ++q) start += __ldg(a.lens + q);
  const int32_t l = z / a.Hq;
  it.qh = z - l * a.Hq;
  it.h = it.qh / a.G;
  it.n = n;
  it.qt = ntq - 1 - qt_rev;
  it.nk = it.qt + 1;
  it.ragged = (it.qt + 1) * kTile > n;
  it.row0 = static_cast<int64_t>(l) * a.T + start;
  return true;
}

// Every length must lie in [0, max_len] and they must add up to T; checked
// by warp 0 before anything is read or written (DKV_E_LENS otherwise).
// Every thread of the block must call it.
__device__ __forceinline__ bool lens_valid(const PrefillArgs &a, int32_t *ok_sm) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int64_t total = 0;
    int bad = 0;
    for (int32_t q = lane; q < a.R; q += 32) {
      const int32_t n = __ldg(a.lens + q);
      if (n < 0 || n > a.max_len) bad = 1;
      total += n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      total += __shfl_xor_sync(0xffffffffu, total, o);
      bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    if (lane == 0) {
      const bool ok = !bad && total == a.T;
      *ok_sm = ok ? 1 : 0;
      if (!ok) set_error(a.status, DKV_E_LENS);
    }
  }
  __syncthreads();
  return *ok_sm != 0;
}

// Named barrier of the softmax warps that also reduces a predicate: true in
// every thread when it was true in any.
__device__ __forceinline__ bool softmax_sync_or(bool p) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred q, o; setp.ne.u32 q, %1, 0; barrier.cta.red.or.pred o, 1, %2, q; selp.u32 %0, 1, 0, o; }"
      : "=r"(r)
      : "r"(p ? 1u : 0u), "n"(32 * kSoftmaxWarps)
      : "memory");
  return r != 0;
}

// Persistent: one block per SM walks the work items (pf_item) from blockIdx.x
// in steps of the grid.  Every role walks the same items and keeps its
// counters (S buffers, ring copies, P^T buffers, Q and O phases) running
// across them, so the next item's copies and S MMAs overlap the end of this
// one.
__global__ void __launch_bounds__(kThreadsP, 1)
    k_prefill(PrefillArgs a, const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
              const __grid_constant__ CUtensorMap vmap, int64_t n_items) {
  extern __shared__ unsigned char smem_raw[];
  PrefillSmem &sm =
      *reinterpret_cast<PrefillSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // before any allocation: leaving early is safe
  if (!lens_valid(a, &sm.lens_ok)) return;
  volatile int32_t *abort = &sm.abort;

  if (tid == 0) {
    mbar_init(&sm.bar_q, 1);
    mbar_init(&sm.bar_qfree, 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < kSBuf; ++i) {
      mbar_init(&sm.bar_s[i], 1);
      mbar_init(&sm.bar_sfree[i], kSoftmaxWarps);
    }
    for (int i = 0; i < kPBuf; ++i) {
      mbar_init(&sm.bar_pready[i], kSoftmaxWarps);
      mbar_init(&sm.bar_o[i], 1);
    }
    mbar_init(&sm.bar_done, 1);
    mbar_init(&sm.bar_ofree, kSoftmaxWarps);
    mbar_init(&sm.bar_sdone, 1);
    mbar_init(&sm.bar_pvdone, 1);
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

  // a wait that gives up records the timeout once and makes everyone stop
  auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
    if (mbar_wait(bar, parity, abort)) return true;
    if (!*abort) {
      *abort = 1;
      set_error(a.status, DKV_E_TIMEOUT);
    }
    return false;
  };
  // Within an item, tiles t = 0 .. 2 nk - 1: pass 1 (t < nk) key tile t,
  // pass 2 key tile t - nk; the block-wide tile count g picks tensor-memory
  // buffer g mod 3.  The item's copies go to ring slots by the block-wide
  // copy count: pass 1 K(t), then pass 2 K(j) and V(j) in turn.

  if (warp == kLoadWarp) {
    // ================= copy warp: lane 0 issues; a slot is refilled once
    // the MMAs that read it have completed, the Q tile once the last S^T of
    // the previous item has
    if (lane == 0) {
      int32_t L = 0, nq = 0;
      bool ok = true;
      for (int64_t i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
        PfItem it;
        if (!pf_item(a, i, it)) continue;
        if (nq > 0 && !(ok = wait(&sm.bar_qfree, (nq - 1) & 1u))) break;
        load_tile(sm.q, &qmap, it.qh, static_cast<int>(it.row0 + it.qt * kTile), &sm.bar_q);
        ++nq;
        for (int32_t p = 0; p < 3 * it.nk; ++p) {
          const int s = L % kSlots;
          if (L >= kSlots && !(ok = wait(&sm.empty[s], ((L / kSlots) - 1) & 1u))) break;
          const bool is_v = p >= it.nk && ((p - it.nk) & 1);
          const int32_t j = p < it.nk ? p : (p - it.nk) >> 1;
          load_tile(sm.ring[s], is_v ? &vmap : &kmap, it.h, static_cast<int>(it.row0 + j * kTile), &sm.full[s]);
          ++L;
        }
      }
      // every copy issued has landed before the block leaves (bounded)
      if (nq > 0) mbar_wait(&sm.bar_q, (nq - 1) & 1u, nullptr);
      for (int32_t c = max(0, L - kSlots); c < L; ++c) mbar_wait(&sm.full[c % kSlots], (c / kSlots) & 1u, nullptr);
    }
  } else if (warp == kSWarp || warp == kPvWarp) {
    // ================= MMA warps: lane 0 waits and issues.  The S warp runs
    // S (pass 1) and S^T (pass 2) of each tile as soon as its buffer has been
    // read and its K tile has landed, then hands the Q tile back; the P V
    // warp runs O += P V of each pass-2 tile once its P^T is in shared
    // memory (and, for an item's first, once O of the previous item has been
    // read), then marks the item's O complete.
    const bool leader = lane == 0;
    constexpr uint32_t kSlotStep = kTileBytes >> 4;
    if (leader) {
      int32_t L = 0, k = 0;
      bool ok = true;
      if (warp == kSWarp) {
        constexpr uint32_t idesc_s = idesc_bf16(kTile, kTile, false, false);
        // descriptors at the operands' bases; a K-step adds its byte offset / 16
        const uint64_t dq = sw128_desc(saddr(sm.q), 16, 1024);
        const uint64_t dk = sw128_desc(saddr(sm.ring[0]), 16, 1024);  // K-major (K tiles)
        int32_t g = 0;
        for (int64_t i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
          PfItem it;
          if (!pf_item(a, i, it)) continue;
          if (!(ok = wait(&sm.bar_q, k & 1u))) break;
          for (int32_t t = 0; t < 2 * it.nk; ++t, ++g) {
            const int b = g % kSBuf;
            if (g >= kSBuf && !(ok = wait(&sm.bar_sfree[b], ((g / kSBuf) - 1) & 1u))) break;
            const bool pass2 = t >= it.nk;
            const int32_t Lk = L + (pass2 ? it.nk + 2 * (t - it.nk) : t);
            if (!(ok = wait(&sm.full[Lk % kSlots], (Lk / kSlots) & 1u))) break;
            tc_fence_after();
            const uint64_t dks = dk + (Lk % kSlots) * kSlotStep;
            const uint64_t da = pass2 ? dks : dq, db = pass2 ? dq : dks;  // S = Q K^T, S^T = K Q^T
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // 16 channels a step: 32 bytes along the swizzled rows, then the next box
              const uint32_t o = ((kk >> 2) * kBox + (kk & 3) * 32) >> 4;
              mma_ss(tmem + kTile * b, da + o, db + o, idesc_s, kk > 0 ? 1u : 0u);
            }
            mma_commit(&sm.bar_s[b]);
            mma_commit(&sm.empty[Lk % kSlots]);
          }
          if (!ok) break;
          mma_commit(&sm.bar_qfree);  // the Q tile is free once these MMAs complete
          L += 3 * it.nk;
          ++k;
        }
        // every MMA of this warp done (also after an abort)
        mma_commit(&sm.bar_sdone);
        mbar_wait(&sm.bar_sdone, 0, nullptr);
      } else {
        constexpr uint32_t idesc_o = idesc_bf16(kTile, 128, true, true);
        const uint64_t dv = sw128_desc(saddr(sm.ring[0]), kBox, 1024);  // MN-major (V tiles): boxes kBox apart
        const uint64_t dp = sw128_desc(saddr(sm.pt[0]), kBox, 1024);    // MN-major (P^T): query halves kBox apart
        int32_t jj = 0;
        for (int64_t i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
          PfItem it;
          if (!pf_item(a, i, it)) continue;
          for (int32_t j = 0; j < it.nk; ++j, ++jj) {
            const int32_t Lv = L + it.nk + 2 * j + 1;
            if (j == 0 && k > 0 && !(ok = wait(&sm.bar_ofree, (k - 1) & 1u))) break;
            if (!(ok = wait(&sm.bar_pready[jj % kPBuf], (jj / kPBuf) & 1u) &&
                       wait(&sm.full[Lv % kSlots], (Lv / kSlots) & 1u)))
              break;
            tc_fence_after();
            const uint64_t dvs = dv + (Lv % kSlots) * kSlotStep;
            const uint64_t dps = dp + (jj % kPBuf) * kSlotStep;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // 16 keys a step: 16 rows (2048 bytes) of P^T and of V
              mma_ss(tmem + kColO, dps + ((kk * 2048) >> 4), dvs + ((kk * 2048) >> 4), idesc_o,
                     (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&sm.bar_o[jj % kPBuf]);
            mma_commit(&sm.empty[Lv % kSlots]);
          }
          if (!ok) break;
          mma_commit(&sm.bar_done);  // the item's O is complete
          L += 3 * it.nk;
          ++k;
        }
        // every MMA of this warp done (also after an abort)
        mma_commit(&sm.bar_pvdone);
        mbar_wait(&sm.bar_pvdone, 0, nullptr);
      }
    }
  } else {
    // ================= softmax warps: warp w reads lanes 32 (w mod 4) .. + 31
    // and columns kCols (w div 4) .. + kCols - 1 of each tile
    const int rq = warp & 3, cq = warp >> 2;
    const int row = 32 * rq + lane;  // pass 1: query row; pass 2: key row of the tile
    const float sl2 = a.scale * 1.44269504088896340736f;  // logits in log2 units
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * rq) << 16);
    const uint64_t s2 = f2_pack(sl2, sl2);
    const float4 *nl4 = reinterpret_cast<const float4 *>(sm.nlse) + (kCols / 4) * cq;
    const uint32_t prow = cq * kBox + row * 128;  // this thread's row of a P^T buffer
    bool ok = true;
    int32_t g = 0, jj = 0, k = 0;
    for (int64_t i = blockIdx.x; i < n_items; i += gridDim.x) {
      PfItem it;
      if (!pf_item(a, i, it)) continue;
      const int32_t qt = it.qt, n = it.n, nk = it.nk;
      const bool ragged = it.ragged;
      const int32_t qrow = qt * kTile + row;
      // pass 1 masks: a row past the request masks every key (qlim = -1);
      // masks are applied per element only in the diagonal tile and in a
      // tile with such rows
      const int32_t qlim = qrow < n ? qrow : -1;

      // ---- pass 1: row maximum and sum over this thread's columns (log2
      // units); the buffer is handed back as soon as it is read
      float m = -INFINITY, lsum = 0.0f;
      for (int32_t j = 0; j < nk && ok; ++j, ++g) {
        if (!(ok = wait(&sm.bar_s[g % kSBuf], (g / kSBuf) & 1u))) break;
        tc_fence_after();
        float v[kCols];
        tmem_ld64(lane_base + kTile * (g % kSBuf) + kCols * cq, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.bar_sfree[g % kSBuf]);
        if (j == qt || ragged) {
          const int32_t key0 = j * kTile + kCols * cq;
#pragma unroll
          for (int i2 = 0; i2 < kCols; ++i2) v[i2] = key0 + i2 <= qlim ? v[i2] : -INFINITY;
        }
        float(&v0)[32] = *reinterpret_cast<float(*)[32]>(&v[0]);
        float(&v1)[32] = *reinterpret_cast<float(*)[32]>(&v[32]);
        const float mn = fmaxf(m, fmaxf(max32(v0), max32(v1)) * sl2);  // scale > 0: the maximum commutes with it
        if (mn != -INFINITY) {
          const float t = exp2_sum32(v0, sl2, mn) + exp2_sum32(v1, sl2, mn);
          lsum = lsum * ex2(m - mn) + t;  // ex2(-inf) = 0 on the first tile
          m = mn;
        }
      }
      // the column groups of a row meet: m = max, l = sum of rescaled sums;
      // then -(m + log2 l) of every row is published for pass 2 (a row past
      // the request has l = 0 and gets -inf: its probabilities are 0).  The
      // second barrier also decides, for every softmax warp alike, whether
      // the block is winding down.
      float2(&stat)[kQuarters][kTile] = *reinterpret_cast<float2(*)[kQuarters][kTile]>(sm.pt[0]);
      stat[cq][row] = make_float2(m, lsum);
      softmax_sync();
      if (cq == 0) {
        float2 st[kQuarters];
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kQuarters; ++c) {
          st[c] = stat[c][row];
          mx = fmaxf(mx, st[c].x);
        }
        float ls = 0.0f;
        if (mx != -INFINITY) {
#pragma unroll
          for (int c = 0; c < kQuarters; ++c) ls += st[c].y * ex2(st[c].x - mx);
        }
        sm.nlse[row] = ls > 0.0f ? -(mx + log2f(ls)) : -INFINITY;  // a row past the request: p = 0
      }
      if (softmax_sync_or(!ok || *abort != 0)) break;

      // ---- pass 2: S^T of key tile j: this thread's key row, queries
      // q0 .. q0 + kCols - 1.  p = exp2(s sl2 - (m_q + log2 l_q)); valid
      // where key <= q < n.  The row sum is added to the key's significance
      // (one atomic per thread and tile), P^T (bf16) goes to shared memory
      // once P V of the tile that last used the buffer has read it: the
      // whole 128-byte key row `row` of query half cq, 16-byte chunk c
      // stored at c xor (row mod 8) (the 128-byte swizzle).
      const int32_t q0 = qt * kTile + kCols * cq;
      for (int32_t j = 0; j < nk && ok; ++j, ++g, ++jj) {
        if (!(ok = wait(&sm.bar_s[g % kSBuf], (g / kSBuf) & 1u))) break;
        tc_fence_after();
        float v[kCols];
        tmem_ld64(lane_base + kTile * (g % kSBuf) + kCols * cq, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.bar_sfree[g % kSBuf]);
        const int32_t key = j * kTile + row;
        const bool masked = j == qt || ragged;
        uint32_t w[kCols / 2];
        float rs = 0.0f;
#pragma unroll
        for (int c = 0; c < kCols / 32; ++c) {
          uint64_t e[16];
#pragma unroll
          for (int i2 = 0; i2 < 8; ++i2) {
            const float4 t = nl4[8 * c + i2];  // queries q0 + 32 c + 4 i2 .. + 3
            float x0, x1, x2, x3;
            f2_unpack(f2_fma(f2_pack(v[32 * c + 4 * i2], v[32 * c + 4 * i2 + 1]), s2, f2_pack(t.x, t.y)), x0, x1);
            f2_unpack(f2_fma(f2_pack(v[32 * c + 4 * i2 + 2], v[32 * c + 4 * i2 + 3]), s2, f2_pack(t.z, t.w)), x2, x3);
            e[2 * i2] = f2_pack(ex2(x0), ex2(x1));
            e[2 * i2 + 1] = f2_pack(ex2(x2), ex2(x3));
          }
          if (masked) {
            const int32_t lo = key - q0 - 32 * c, hi = n - q0 - 32 * c;  // valid queries: lo <= i < hi
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) {
              float x0, x1;
              f2_unpack(e[i2], x0, x1);
              x0 = (2 * i2 >= lo && 2 * i2 < hi) ? x0 : 0.0f;
              x1 = (2 * i2 + 1 >= lo && 2 * i2 + 1 < hi) ? x1 : 0.0f;
              e[i2] = f2_pack(x0, x1);
            }
          }
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) {
            float x0, x1;
            f2_unpack(e[i2], x0, x1);
            w[16 * c + i2] = bf16x2_rn(x0, x1);
          }
          uint64_t t[8];
#pragma unroll
          for (int i2 = 0; i2 < 8; ++i2) t[i2] = f2_add(e[i2], e[i2 + 8]);
#pragma unroll
          for (int wd = 4; wd >= 1; wd >>= 1)
#pragma unroll
            for (int i2 = 0; i2 < wd; ++i2) t[i2] = f2_add(t[i2], t[i2 + wd]);
          float lo_, hi_;
          f2_unpack(t[0], lo_, hi_);
          rs += lo_ + hi_;
        }
        if (key < n && rs != 0.0f) atomicAdd(a.sig_sum + (it.row0 + key) * a.Hq + it.qh, rs);
        // buffer jj mod kPBuf is free once P V of tile jj - kPBuf has read it
        if (jj >= kPBuf && !(ok = wait(&sm.bar_o[jj % kPBuf], ((jj - kPBuf) / kPBuf) & 1u))) break;
        uint8_t *pb = sm.pt[jj % kPBuf] + prow;
#pragma unroll
        for (int i2 = 0; i2 < kCols / 8; ++i2)
          *reinterpret_cast<uint4 *>(pb + 16 * (i2 ^ (row & 7))) =
              make_uint4(w[4 * i2], w[4 * i2 + 1], w[4 * i2 + 2], w[4 * i2 + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor cores
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.bar_pready[jj % kPBuf]);
      }

      // ---- outputs: this thread's kCols channels of its row of O (the
      // loads are warp-collective, so every lane takes them; rows past the
      // request store nothing); then O is handed back for the next item
      if (ok && (ok = wait(&sm.bar_done, k & 1u))) {
        tc_fence_after();
        float v[kCols];
        tmem_ld64(lane_base + kColO + kCols * cq, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.bar_ofree);
        if (qrow < n) {
          float *dst = a.out + ((it.row0 + qrow) * a.Hq + it.qh) * 128 + kCols * cq;
#pragma unroll
          for (int i2 = 0; i2 < kCols; i2 += 4)
            *reinterpret_cast<float4 *>(dst + i2) = make_float4(v[i2], v[i2 + 1], v[i2 + 2], v[i2 + 3]);
        }
      }
      ++k;
    }
  }

  // ---- teardown: the copy and MMA warps have waited (bounded) for this
  // block's own copies and MMAs; free the tensor memory
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
  // persistent: one block per SM over every (query tile, request, layer x
  // head) item, longest first
  const int64_t n_items = static_cast<int64_t>((a.max_len + kTile - 1) / kTile) * a.R * a.L * a.Hq;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int grid = static_cast<int>(std::min<int64_t>(n_items, std::max(sms, 1)));
  k_prefill<<<grid, kThreadsP, smem, s>>>(a, qmap, kmap, vmap, n_items);
  return cudaGetLastError();
}

}  // namespace dkv
