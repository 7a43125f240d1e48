// dkv_internal.cuh -- shared definitions of the libdkv kernels (device side).
//
// Work decomposition of one dkv_compact call
//   unit      (layer l, request r, KV head h), u = (l * R + r) * Hkv + h
//   tile      kTileTokens consecutive tokens of one request; rt = tile_off[r] + j
//             numbers the (request, tile) pairs, TR = sum_r ceil(N_r / tile).
//             A "unit tile" is a tile of one unit, numbered
//             tau = (l * Hkv + h) * TR + rt, so a unit's tiles are contiguous
//             and tile_info[rt] (first token, size, request length and
//             thresholds) decodes tau without a search.
//
// Kernels, in stream order (all bounded, none traps):
//   k_prep      1 block: request prefix sums, length validation, resets
//   k_classify  significance reduce + three-tier classification + per-tile
//               class bitmasks (warp ballots)
//   k_scan      per-unit page demand, block scan + decoupled look-back over
//               partitions of units, capacity check
//   k_pack      quantise + pack + scatter every surviving row into its page
//               slot, fill unused slots
//   k_commit    forward / reverse tables, page classes, head cursor, status
#pragma once

#include <cstdint>

#include "../../include/dkv.h"

namespace dkv {

// Precision schemes (dkv_pool.scheme): bits of K and V in the high class;
// the low class has half of each, so a low token takes exactly half a high
// token's code bytes and a page holds P high or 2P low tokens.
__host__ __device__ constexpr int scheme_kh(int s) { return s == 2 ? 4 : 8; }
__host__ __device__ constexpr int scheme_vh(int s) { return s == 0 ? 4 : (s == 1 ? 2 : 8); }
constexpr int kSchemes = 3;

// Byte geometry of one unified page: K codes [0, vbase), V codes
// [vbase, meta), fp16 {k_scale, k_zero, v_scale, v_zero} per slot at
// meta + 8 s, int32 position per slot at pos + 4 s.
struct PageGeom {
  int32_t P, kh, vh, pad;
  int64_t vbase;  // 16 kh P
  int64_t meta;   // 16 (kh + vh) P
  int64_t pos;    // meta + 16 P
  int64_t bytes;  // meta + 24 P
};

__host__ __device__ inline PageGeom page_geom(int scheme, int32_t P) {
  PageGeom g{};
  g.P = P;
  g.kh = scheme_kh(scheme);
  g.vh = scheme_vh(scheme);
  g.vbase = 16 * static_cast<int64_t>(g.kh) * P;
  g.meta = 16 * static_cast<int64_t>(g.kh + g.vh) * P;
  g.pos = g.meta + 16 * static_cast<int64_t>(P);
  g.bytes = g.meta + 24 * static_cast<int64_t>(P);
  return g;
}

constexpr int kTileTokens = 128;                 // tokens per tile
constexpr int kMaskWords = kTileTokens / 32;     // 32-bit words per class mask
constexpr int kScanUnits = 32;                   // units per scan partition
constexpr int kMaxHq = 128;                      // query heads supported

// Call-local state at the start of the workspace.
struct WsHeader {
  int32_t err;       // first device-side error of this call (0 = none)
  int32_t ticket;    // scan partition ticket counter
  int32_t TR;        // number of (request, tile) pairs
  int32_t npart;     // scan partitions
  int64_t total;     // sum of page demands
  uint64_t head;     // free-list head when the call started
  int64_t head_mod;  // head mod F
  int64_t pad[3];
};

// Decoupled look-back status word: flag in the top two bits.
constexpr uint64_t kFlagAggregate = 1ull << 62;
constexpr uint64_t kFlagPrefix = 2ull << 62;
constexpr uint64_t kValueMask = (1ull << 62) - 1;

// Per-unit results of the scan: {n_k8v4, n_k4v2, page offset, pages_k8v4}.
struct UnitInfo {
  int32_t n_hi, n_lo, off, p_hi;
};

// Everything the quantise + scatter kernel needs of one unit tile, written by
// the scan (64 bytes, one load per tile).
struct __align__(16) TileDesc {
  uint4 hm, lm;       // K8V4 / K4V2 bitmasks of the tile's 128 tokens
  int32_t base_hi;    // K8V4 rank of the tile's first K8V4 row within its unit
  int32_t base_lo;    // K4V2 rank likewise
  int32_t tok_row;    // l * T + first token of the tile
  int32_t h;          // KV head
  int32_t pos0;       // position of the tile's token 0 in its request
  int32_t ring;       // free-list slot of the unit's first page, (head + off) mod F
  int32_t p_hi;       // K8V4 pages of the unit
  int32_t pad;
};

// One (request, tile) pair, written by k_prep: what the classification of
// its tokens needs, in one 32-byte record.
struct __align__(16) TileInfo {
  int64_t t0;          // first token of the tile in the layer's token order
  int32_t cnt;         // tokens in the tile (1 .. kTileTokens)
  int32_t N;           // tokens of its request
  float thr_h, thr_l;  // alpha_h / N and alpha_l / N, each rounded once
  int32_t pad[2];
};

// Byte offsets of the workspace regions (all 256-byte aligned).
struct WsLayout {
  size_t tok_off;    // int64 [R + 1]
  size_t tile_off;   // int32 [R + 1]
  size_t tile_info;  // TileInfo [tr_max]: one per (request, tile) pair
  size_t part;       // uint64 [npart]
  size_t unit;       // UnitInfo [U]
  size_t mask;       // uint32 [NT][2 * kMaskWords]: K8V4 words then K4V2 words
  size_t desc;       // TileDesc [NT]
  size_t bytes;      // total
  int64_t nt_max;    // unit tiles the layout has room for
  int32_t npart;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(int64_t L, int64_t R, int64_t Hkv, int64_t T) {
  WsLayout w{};
  const int64_t U = L * R * Hkv;
  const int64_t tr_max = T / kTileTokens + R;  // >= sum_r ceil(N_r / tile)
  w.nt_max = L * Hkv * tr_max;
  w.npart = static_cast<int32_t>((U + kScanUnits - 1) / kScanUnits);
  size_t o = align256(sizeof(WsHeader));
  w.tok_off = o;  o = align256(o + sizeof(int64_t) * (R + 1));
  w.tile_off = o; o = align256(o + sizeof(int32_t) * (R + 1));
  w.tile_info = o; o = align256(o + sizeof(TileInfo) * tr_max);
  w.part = o;     o = align256(o + sizeof(uint64_t) * w.npart);
  w.unit = o;     o = align256(o + sizeof(UnitInfo) * U);
  w.mask = o;     o = align256(o + sizeof(uint32_t) * 2 * kMaskWords * w.nt_max);
  w.desc = o;     o = align256(o + sizeof(TileDesc) * w.nt_max);
  w.bytes = o;
  return w;
}

// Everything a kernel of dkv_compact needs, passed by value.
struct CompactArgs {
  PageGeom pg;                    // page layout of the pool's scheme
  int32_t L, R, Hq, Hkv, G, P, pmax, spin_limit;
  int64_t T, F, U, unit_base;
  int32_t max_len;
  float alpha_h, alpha_l;
  const uint16_t *k, *v;
  const float *sig_sum;
  const int32_t *sig_cnt, *lens;
  uint8_t *classes;
  int32_t *free_list;
  uint64_t *cursors;
  int32_t *rev_unit, *rev_idx;
  uint8_t *page_cls, *pages;
  int32_t *status;
  int32_t *fwd, *unit_hdr;
  // workspace
  WsHeader *ws;
  int64_t *tok_off;
  int32_t *tile_off;
  TileInfo *tile_info;
  uint64_t *part;
  UnitInfo *unit;
  uint32_t *mask;
  TileDesc *desc;
};

__device__ __forceinline__ void set_error(int32_t *err, int32_t code) { atomicCAS(err, 0, code); }

// Bounds checks of the DKV_CHECKED build, the stand-in for a device memory
// checker: there in_range() records DKV_E_INTERNAL and returns false when i
// lies outside [0, n), and the caller skips the access (no trap).  In the
// normal build it is the constant true and costs nothing.
#ifdef DKV_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif
__device__ __forceinline__ bool in_range(int64_t i, int64_t n, int32_t *status) {
  if (!kChecked) return true;
  if (i >= 0 && i < n) return true;
  set_error(status, DKV_E_INTERNAL);
  return false;
}

// Largest r in [0, n) with a[r] <= x (a non-decreasing, a[0] <= x).
__device__ __forceinline__ int find_segment(const int32_t *a, int n, int64_t x, int64_t scale) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(__ldg(a + mid)) * scale <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------- decode --

constexpr int kReclassChunk = 4096;   // most positions per reclassification block

// Positions per reclassification block: the longest of 4096, 2048, 1024, 512
// that still makes two waves of blocks (4 resident per SM) over the L R
// (layer, request) pairs.  Longer blocks amortise their set-up and L2
// prefetch; shorter ones keep a small batch spread over every SM.
inline int32_t reclass_chunk(int64_t lr, int32_t cap, int sms) {
  int32_t c = kReclassChunk;
  while (c > 512 && lr * ((cap + c - 1) / c) < 8ll * sms) c >>= 1;
  return c;
}
constexpr int kMaxApplyWarps = 8;     // units (KV heads) per apply block, one warp each

struct DecWsHeader {
  int32_t err;       // first device-side error of this call (0 = none)
  int32_t ticket;    // scan partition ticket counter
  int32_t npart;     // scan partitions
  int32_t job_n;     // demotion jobs staged for k_demote
  uint64_t head;     // free-list cursors when the call started
  uint64_t tail;
  int64_t dsum;      // new pages of the step
  int64_t fsum;      // freed pages of the step
  int64_t pad1[2];
};

// Per-unit plan of a generation step (48 bytes), written by the scan.
struct __align__(16) DecPlan {
  int32_t n_hi, n_lo, have_hi, have_lo;   // lists and pages before the step
  int32_t keep_hi, keep_lo, dem, new_cls; // survivors, demoted count, class of the new token
  int32_t need_hi, need_lo, off_d, off_f; // pages after the step, scan offsets (new, freed)
};

constexpr int kMarkList = 1024;       // listed changes per (layer, request); more fall back to a scan
constexpr int64_t kDemoteJobs = 1 << 20;  // staged demotions per call at most; more are done in place

// One staged demotion: the token's high-class slot bytes and where its
// low-class copy goes.
struct __align__(16) DemJob {
  uint4 c[12];         // the high slot's K codes (16 kh bytes), then its V codes (16 vh bytes)
  uint2 meta;          // fp16 k_scale, k_zero, v_scale, v_zero
  int32_t dst_page;    // -1: nothing to write
  int32_t dst_slot;
  int32_t pos;
  int32_t pad[3];
};

struct DecWsLayout {
  size_t ucnt;   // int4 [U]: demoted, K8V4 pruned, K4V2 pruned, new-token word
  size_t part;   // uint64 [npart]
  size_t lcnt;   // int32 [L * R]: changes listed per (layer, request)
  size_t plan;   // DecPlan [U]
  size_t list;   // uint32 [L * R][kMarkList]: position << 11 | head << 4 | old << 2 | new
  size_t jobs;   // DemJob [njobs]
  int64_t njobs;
  size_t reset;  // bytes zeroed at the start of a call (header, counters, partitions, list counts)
  size_t bytes;
  int32_t npart;
};

inline DecWsLayout dec_ws_layout(int64_t U, int64_t LR, int64_t rows) {
  DecWsLayout w{};
  // room for demoting one held row in 16 per call (the seeded generation
  // demotes about 1 in 200); a step that demotes more does the rest in place
  const int64_t want = rows / 16 + 64;
  w.njobs = want < kDemoteJobs ? want : kDemoteJobs;
  w.npart = static_cast<int32_t>((U + 255) / 256);
  size_t o = align256(sizeof(DecWsHeader));
  w.ucnt = o; o = align256(o + 16 * static_cast<size_t>(U));
  w.part = o; o = align256(o + sizeof(uint64_t) * w.npart);
  w.lcnt = o; o = align256(o + sizeof(int32_t) * static_cast<size_t>(LR));
  w.reset = o;
  w.plan = o; o = align256(o + sizeof(DecPlan) * static_cast<size_t>(U));
  w.list = o; o = align256(o + sizeof(uint32_t) * kMarkList * static_cast<size_t>(LR));
  w.jobs = o; o = align256(o + sizeof(DemJob) * static_cast<size_t>(w.njobs));
  w.bytes = o;
  return w;
}

struct DecodeArgs {
  PageGeom pg;                    // page layout of the pool's scheme
  int32_t L, R, Hq, Hkv, G, P, pmax, cap, spin_limit;
  int32_t window, mode;
  int32_t rchunk;  // positions per reclassification block
  int64_t F, U, unit_base;
  float alpha_h, alpha_l;
  const uint16_t *k_new, *v_new;
  const float *sig_sum;
  const int32_t *sig_cnt, *ctx_lens, *new_lens;
  uint8_t *classes;
  int32_t *slot_of;
  int32_t *free_list;
  uint64_t *cursors;
  int32_t *rev_unit, *rev_idx;
  uint8_t *page_cls, *pages;
  int32_t *status;
  int32_t *fwd, *unit_hdr;
  DecWsHeader *ws;
  int4 *ucnt;
  uint64_t *part;
  int32_t *lcnt;
  DecPlan *plan;
  uint32_t *list;
  DemJob *jobs;
  int64_t njobs;
};

// Decode attention (attend.cu): one cluster of S blocks per unit; every warp
// streams whole pages through a private ring of kAttendStages buffers.
constexpr int kAttendStages = 2;
constexpr int kAttendMaxG = 8;

// Warps per block: 6 for up to four query heads per KV head (two blocks share
// an SM, so one block's merges and significance updates overlap the other's
// page streaming), 8 above (the second group of four heads doubles the
// registers a lane holds: one block per SM).
__host__ __device__ constexpr int attend_warps(int G) { return G <= 4 ? 6 : 8; }
__host__ __device__ constexpr int attend_blocks_per_sm(int G) { return G <= 4 ? 2 : 1; }

struct AttnArgs {
  int32_t L, R, Hq, Hkv, G, P, pmax, cap, layer0, n_layers;
  int32_t scheme;               // the pool's bit-width scheme
  int32_t cmax;                 // tokens one block of a cluster holds at most
  int64_t F, units;             // units = n_layers * R * Hkv
  float scale;
  const uint16_t *q, *k_new, *v_new;
  const int32_t *new_lens, *ctx_lens;
  float *out, *sig_sum;
  const int32_t *fwd, *unit_hdr;
  const uint8_t *pages;
  int32_t *status;
};

// Byte offsets of the attention kernel's dynamic shared memory.
struct AttnLayout {
  size_t stage;   // [warps][stages][216 P] page buffers (warps = attend_warps(G))
  size_t bar;     // [warps][stages] mbarriers
  size_t lg;      // [cmax][G] logits
  size_t ps;      // [cmax] positions
  size_t fw;      // [pmax] forward row
  size_t red;     // [warps][G][128] partial outputs
  size_t st;      // statistics: [warps][8] max, [warps][8] sum, 4 x [8], [8][8] block factors
  size_t bytes;
};

__host__ __device__ inline AttnLayout attend_layout(int32_t cmax, int32_t G, int32_t pmax, int32_t P) {
  auto up = [](size_t x) { return (x + 127) / 128 * 128; };
  const size_t W = static_cast<size_t>(attend_warps(G));
  AttnLayout o{};
  size_t x = 0;
  o.stage = x; x = up(x + W * kAttendStages * 216 * static_cast<size_t>(P));
  o.bar = x; x = up(x + 8 * W * kAttendStages);
  o.lg = x; x = up(x + 4 * static_cast<size_t>(cmax) * G);
  o.ps = x; x = up(x + 4 * static_cast<size_t>(cmax));
  o.fw = x; x = up(x + 4 * static_cast<size_t>(pmax));
  o.red = x; x = up(x + 4 * W * G * 128);
  o.st = x; x = up(x + 4 * static_cast<size_t>(kAttendMaxG) * (2 * W + 12));
  o.bytes = x;
  return o;
}

// Prefill attention with significance accumulation (prefill.cu).
struct PrefillArgs {
  int32_t L, R, Hq, Hkv, G, max_len;
  int64_t T;
  float scale;
  const uint16_t *q, *k, *v;
  const int32_t *lens;
  float *out, *sig_sum;
  int32_t *sig_cnt;
  int32_t *status;
};

}  // namespace dkv

// Launchers (defined in the kernel translation units).
namespace dkv {
cudaError_t launch_prep(const CompactArgs &a, cudaStream_t s);
cudaError_t launch_classify(const CompactArgs &a, int grid, int sms, cudaStream_t s);
cudaError_t launch_scan(const CompactArgs &a, int npart, cudaStream_t s);
cudaError_t launch_pack(const CompactArgs &a, int grid, cudaStream_t s);
cudaError_t launch_commit(const CompactArgs &a, int grid, cudaStream_t s);
cudaError_t launch_clear_hi(const CompactArgs &a, int grid, cudaStream_t s);
cudaError_t launch_init_pool(const dkv_pool &p, cudaStream_t s);
cudaError_t launch_dequant(const dkv_pool &p, const int32_t *ids, int32_t one_id, int32_t n,
                           float *k_out, float *v_out, int32_t *pos_out, cudaStream_t s);
int pack_blocks_per_sm();
cudaError_t launch_reclass(const DecodeArgs &a, cudaStream_t s);
cudaError_t launch_candidate(const DecodeArgs &a, cudaStream_t s);
cudaError_t launch_dscan(const DecodeArgs &a, int32_t npart, cudaStream_t s);
cudaError_t launch_apply(const DecodeArgs &a, int32_t hpc, int32_t words, cudaStream_t s);
cudaError_t launch_demote(const DecodeArgs &a, int grid, cudaStream_t s);
cudaError_t launch_index(const DecodeArgs &a, int grid, cudaStream_t s);
size_t apply_smem(int32_t hpc, int32_t words, int32_t pmax);
cudaError_t launch_attend(const AttnArgs &a, int32_t S, cudaStream_t s);
cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t s);
}  // namespace dkv
