// alloc.cu -- page demand, parallel prefix sum over the circular free page
// list (k_scan) and the commit of tables and cursors (k_commit).
//
// DiffKV (arXiv 2412.03131), Pith review, "What carries the argument": after
// each attention head decides how many high- and low-precision pages it
// needs, a parallel prefix sum over the circular free page list assigns every
// head a disjoint contiguous region of page ids, so allocation happens on the
// GPU in one coordinated step; "Core claim": unified pages, circular free
// page list, bidirectional page table.
//
// The scan is a single pass: each block takes a ticket (its partition of
// kScanUnits units, in ticket order so every predecessor is already running),
// reduces its units' demands, publishes its aggregate, and looks back over
// the predecessors' published aggregates / inclusive prefixes (the
// decoupled look-back of Merrill and Garland, "Single-pass Parallel Prefix
// Scan with Decoupled Look-back", 2016), the block-level pieces following the
// work-efficient scan of Harris, Sengupta and Owens (GPU Gems 3, ch. 39),
// which the DiffKV paper cites.  Every wait is bounded by spin_limit polls.
#include <cuda_runtime.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kScanThreads = 1024;  // one warp per unit of the partition
constexpr int kCommitThreads = 256;
constexpr int kClearThreads = 128;

__device__ __forceinline__ void st_release(uint64_t *p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_acquire(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int32_t ceil_div(int32_t a, int32_t b) { return (a + b - 1) / b; }

__global__ void __launch_bounds__(kScanThreads) k_scan(CompactArgs a) {
  __shared__ int32_t nh_s[kScanUnits], nl_s[kScanUnits], d_s[kScanUnits], ex_s[kScanUnits];
  __shared__ int32_t wsum_s[kScanUnits / 32];
  __shared__ int32_t part_s, fail_s;
  __shared__ int64_t prefix_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.ws->err != 0) return;  // lengths rejected by k_prep
  if (tid == 0) {
    part_s = atomicAdd(&a.ws->ticket, 1);
    fail_s = 0;
  }
  __syncthreads();
  const int32_t part = part_s;
  const int32_t npart = a.ws->npart;
  if (part >= npart) return;
  const int32_t TR = a.ws->TR;
  const int64_t u0 = static_cast<int64_t>(part) * kScanUnits;

  // per unit: class counts of its tiles -> rank bases of every tile
  for (int uu = warp; uu < kScanUnits; uu += kScanThreads / 32) {
    const int64_t u = u0 + uu;
    int32_t nh = 0, nl = 0;
    if (u < a.U) {
      const int32_t h = static_cast<int32_t>(u % a.Hkv);
      const int64_t lr = u / a.Hkv;
      const int32_t r = static_cast<int32_t>(lr % a.R);
      const int64_t l = lr / a.R;
      const int32_t tr0 = a.tile_off[r];
      const int32_t nt = a.tile_off[r + 1] - tr0;
      const int64_t tau0 = (l * a.Hkv + h) * TR + tr0;
      for (int jb = 0; jb < nt; jb += 32) {
        const int j = jb + lane;
        int32_t ch = 0, cl = 0;
        uint4 hw = make_uint4(0, 0, 0, 0), lw = hw;
        if (j < nt) {
          const uint4 *m = reinterpret_cast<const uint4 *>(a.mask + (tau0 + j) * (2 * kMaskWords));
          hw = m[0];
          lw = m[1];
          ch = __popc(hw.x) + __popc(hw.y) + __popc(hw.z) + __popc(hw.w);
          cl = __popc(lw.x) + __popc(lw.y) + __popc(lw.z) + __popc(lw.w);
        }
        int32_t ih = ch, il = cl;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int32_t xh = __shfl_up_sync(0xffffffffu, ih, o);
          const int32_t xl = __shfl_up_sync(0xffffffffu, il, o);
          if (lane >= o) {
            ih += xh;
            il += xl;
          }
        }
        if (j < nt) {
          TileDesc &t = a.desc[tau0 + j];
          t.hm = hw;
          t.lm = lw;
          t.base_hi = nh + ih - ch;
          t.base_lo = nl + il - cl;
          t.tok_row = static_cast<int32_t>(l * a.T + a.tok_off[r] + static_cast<int64_t>(j) * kTileTokens);
          t.h = h;
          t.pos0 = j * kTileTokens;
        }
        nh += __shfl_sync(0xffffffffu, ih, 31);
        nl += __shfl_sync(0xffffffffu, il, 31);
      }
    }
    if (lane == 0) {
      nh_s[uu] = nh;
      nl_s[uu] = nl;
      d_s[uu] = ceil_div(nh, a.P) + ceil_div(nl, 2 * a.P);
    }
  }
  __syncthreads();

  // block-wide exclusive scan of the partition's page demands
  int32_t incl = 0;
  if (tid < kScanUnits) {
    incl = d_s[tid];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    if (lane == 31) wsum_s[warp] = incl;
  }
  __syncthreads();
  if (tid < kScanUnits) {
    int32_t before = 0;
    for (int w = 0; w < warp; ++w) before += wsum_s[w];
    ex_s[tid] = before + incl - d_s[tid];
  }

  // decoupled look-back over the preceding partitions (thread 0)
  if (tid == 0) {
    int64_t agg = 0;
    for (int w = 0; w < kScanUnits / 32; ++w) agg += wsum_s[w];
    int64_t prefix = 0;
    bool fail = false;
    if (part == 0) {
      st_release(a.part, kFlagPrefix | static_cast<uint64_t>(agg));
    } else {
      st_release(a.part + part, kFlagAggregate | static_cast<uint64_t>(agg));
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
          prefix += static_cast<int64_t>(st & kValueMask);
          if ((st & kFlagPrefix) != 0) break;
          --pred;  // partition 0 always publishes a prefix, so pred stays >= 0
        }
      }
      if (!fail) st_release(a.part + part, kFlagPrefix | static_cast<uint64_t>(prefix + agg));
    }
    if (fail) {
      set_error(&a.ws->err, DKV_E_TIMEOUT);
      fail_s = 1;
    }
    prefix_s = prefix;
    if (!fail && part == npart - 1) {
      const int64_t total = prefix + agg;
      const uint64_t head = a.cursors[0], tail = a.cursors[1];
      a.ws->total = total;
      a.ws->head = head;
      a.ws->head_mod = static_cast<int64_t>(head % static_cast<uint64_t>(a.F));
      // free pages are tail - head (never more than F for a consistent pool)
      if (static_cast<uint64_t>(total) > tail - head || total > a.F) set_error(&a.ws->err, DKV_E_NOMEM);
    }
  }
  __syncthreads();
  if (fail_s) return;
  if (tid < kScanUnits && u0 + tid < a.U) {
    const int64_t off = prefix_s + ex_s[tid];
    a.unit[u0 + tid] = UnitInfo{nh_s[tid], nl_s[tid], static_cast<int32_t>(off), ceil_div(nh_s[tid], a.P)};
  }
  // every tile of the partition's units learns where its unit's pages start
  // in the free list (meaningful only when the call does not run out of pages)
  const int64_t head_mod = static_cast<int64_t>(a.cursors[0] % static_cast<uint64_t>(a.F));
  for (int uu = warp; uu < kScanUnits; uu += kScanThreads / 32) {
    const int64_t u = u0 + uu;
    if (u >= a.U) break;
    const int32_t h = static_cast<int32_t>(u % a.Hkv);
    const int64_t lr = u / a.Hkv;
    const int32_t r = static_cast<int32_t>(lr % a.R);
    const int64_t l = lr / a.R;
    const int32_t tr0 = a.tile_off[r];
    const int32_t nt = a.tile_off[r + 1] - tr0;
    const int64_t tau0 = (l * a.Hkv + h) * TR + tr0;
    int64_t ring = head_mod + (prefix_s + ex_s[uu]) % a.F;
    if (ring >= a.F) ring -= a.F;
    const int32_t p_hi = ceil_div(nh_s[uu], a.P);
    for (int j = lane; j < nt; j += 32) {
      a.desc[tau0 + j].ring = static_cast<int32_t>(ring);
      a.desc[tau0 + j].p_hi = p_hi;
    }
  }
}

__device__ __forceinline__ void fill_words(uint8_t *p, int64_t nwords, uint32_t value, int lane) {
  uint32_t *w = reinterpret_cast<uint32_t *>(p);
  for (int64_t i = lane; i < nwords; i += 32) w[i] = value;
}

// The unused slots P..2P-1 of every new high page: their metadata (8P bytes:
// P/2 chunks of 16) and positions (4P bytes: P/2 chunks of 8; P is even) are
// cleared (zero, position -1).  It needs only the scan's placement, so it
// runs beside k_pack on a second stream, at 32 registers and no shared memory
// so that its blocks fit an SM beside a k_pack block.  One warp per unit;
// consecutive lanes write consecutive chunks of one page whose id comes from
// the lane that loaded it.  A call the scan failed writes nothing; one that
// fails later (in k_pack) has only written pages that stay free.
__global__ void __launch_bounds__(kClearThreads, 16) k_clear_hi(CompactArgs a) {
  if (a.ws->err != 0) return;
  const int lane = threadIdx.x & 31;
  const int64_t head_mod = a.ws->head_mod;
  const int32_t per = a.P;  // chunks per page
  const PageGeom &g = a.pg;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kClearThreads / 32);
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * (kClearThreads / 32) + (threadIdx.x >> 5); u < a.U;
       u += nwarps) {
    const UnitInfo inf = a.unit[u];
    int64_t ring = head_mod + inf.off;
    if (ring >= a.F) ring -= a.F;
    for (int32_t k0 = 0; k0 < inf.p_hi; k0 += 32) {
      int32_t id = -1;
      if (k0 + lane < inf.p_hi) {
        int64_t idx = ring + k0 + lane;
        if (idx >= a.F) idx -= a.F;
        if (in_range(idx, a.F, a.status)) {
          id = __ldg(a.free_list + idx);
          if (!in_range(id, a.F, a.status)) id = -1;
        }
      }
      const int32_t ne = min(inf.p_hi - k0, 32) * per;
      for (int32_t e0 = 0; e0 < ne; e0 += 32) {  // warp-uniform trip count
        const int32_t e = e0 + lane;
        const int32_t pid = __shfl_sync(0xffffffffu, id, min(e / per, 31));
        if (e < ne && pid >= 0) {
          uint8_t *pg = a.pages + static_cast<int64_t>(pid) * g.bytes;
          const int32_t c = e % per;
          if (c < per / 2) reinterpret_cast<uint4 *>(pg + g.meta + 8 * static_cast<int64_t>(per))[c] = make_uint4(0u, 0u, 0u, 0u);
          else reinterpret_cast<int2 *>(pg + g.pos + 4 * static_cast<int64_t>(per))[c - per / 2] = make_int2(-1, -1);
        }
      }
    }
  }
}

// Commit of a successful call: forward and reverse tables, page classes,
// unit headers, the head cursor; and the tail of each unit's last high and
// low page (zero codes and metadata, position -1).  A failed call only
// records its error in the pool's status word.
__global__ void __launch_bounds__(kCommitThreads) k_commit(CompactArgs a) {
  const int32_t err = a.ws->err;
  if (err != 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicCAS(a.status, 0, err);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int64_t head_mod = a.ws->head_mod;
  const int64_t P = a.P;
  const PageGeom &g = a.pg;
  const int64_t page_bytes = g.bytes;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kCommitThreads / 32);
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * (kCommitThreads / 32) + (threadIdx.x >> 5); u < a.U;
       u += nwarps) {
    const UnitInfo inf = a.unit[u];
    const int32_t p_lo = ceil_div(inf.n_lo, 2 * a.P);
    const int32_t d = inf.p_hi + p_lo;
    int64_t ring = head_mod + inf.off;
    if (ring >= a.F) ring -= a.F;
    // id of the unit's page k (-1 past its d pages; -2 where the checked build
    // finds the ring index or the id out of range: nothing is written for it)
    auto page_id = [&](int32_t k) -> int32_t {
      if (k >= d) return -1;
      int64_t idx = ring + k;
      if (idx >= a.F) idx -= a.F;
      if (!in_range(idx, a.F, a.status)) return -2;
      const int32_t id = __ldg(a.free_list + idx);
      return in_range(id, a.F, a.status) ? id : -2;
    };
    // the last K8V4 and the last K4V2 page, when partly filled (their ids
    // loaded now, beside the first group's)
    const int64_t sh = inf.n_hi % P, sl = inf.n_lo % (2 * P);
    const int32_t id_th = sh != 0 ? page_id(inf.p_hi - 1) : -1;
    const int32_t id_tl = sl != 0 ? page_id(d - 1) : -1;
    // forward entries in groups of 32, one per lane; each group's ids are
    // loaded before the previous group's stores, so the loads overlap
    int32_t *fw = a.fwd + u * a.pmax;
    int32_t id = page_id(lane);
    for (int32_t k0 = 0; k0 < a.pmax; k0 += 32) {  // d <= pmax
      const int32_t k = k0 + lane;
      const int32_t id_next = page_id(k + 32);
      if (k < a.pmax && id != -2) fw[k] = id;
      if (id >= 0) {
        a.rev_unit[id] = static_cast<int32_t>(a.unit_base + u);
        a.rev_idx[id] = k;
        a.page_cls[id] = k < inf.p_hi ? DKV_CLASS_K8V4 : DKV_CLASS_K4V2;
      }
      id = id_next;
    }
    if (lane == 0) reinterpret_cast<int4 *>(a.unit_hdr)[u] = make_int4(inf.n_hi, inf.n_lo, inf.p_hi, p_lo);
    // tails of the last K8V4 and the last K4V2 page
    if (id_th >= 0) {
      uint8_t *pg = a.pages + static_cast<int64_t>(id_th) * page_bytes;
      fill_words(pg + 16 * g.kh * sh, 4 * g.kh * (P - sh), 0u, lane);
      fill_words(pg + g.vbase + 16 * g.vh * sh, 4 * g.vh * (P - sh), 0u, lane);
      fill_words(pg + g.meta + 8 * sh, 2 * (P - sh), 0u, lane);
      fill_words(pg + g.pos + 4 * sh, P - sh, 0xffffffffu, lane);
    }
    if (id_tl >= 0) {
      uint8_t *pg = a.pages + static_cast<int64_t>(id_tl) * page_bytes;
      fill_words(pg + 8 * g.kh * sl, 2 * g.kh * (2 * P - sl), 0u, lane);
      fill_words(pg + g.vbase + 8 * g.vh * sl, 2 * g.vh * (2 * P - sl), 0u, lane);
      fill_words(pg + g.meta + 8 * sl, 2 * (2 * P - sl), 0u, lane);
      fill_words(pg + g.pos + 4 * sl, 2 * P - sl, 0xffffffffu, lane);
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) a.cursors[0] = a.ws->head + static_cast<uint64_t>(a.ws->total);
}

}  // namespace

cudaError_t launch_scan(const CompactArgs &a, int npart, cudaStream_t s) {
  k_scan<<<npart, kScanThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_clear_hi(const CompactArgs &a, int grid, cudaStream_t s) {
  k_clear_hi<<<grid, kClearThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_commit(const CompactArgs &a, int grid, cudaStream_t s) {
  k_commit<<<grid, kCommitThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dkv
