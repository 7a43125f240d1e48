// api.cu -- the libdkv C ABI: argument validation, workspace layout, kernel
// launches, status and profiling.  Every entry point is declared, with its
// argument meaning, layout, ownership and error behaviour, in include/dkv.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <new>
#include <vector>

#include "dkv_internal.cuh"

namespace {

using dkv::CompactArgs;

constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
int g_pack_bps[kMaxDevices];

bool device_info(int *sms, int *pack_bps) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return false;
    g_pack_bps[dev] = dkv::pack_blocks_per_sm();
    g_sms[dev] = n;
  }
  *sms = g_sms[dev];
  *pack_bps = g_pack_bps[dev];
  return true;
}

// A second stream for work that runs beside k_pack, with the events that fork
// it from the caller's stream and join it back, one set per CUDA context
// (keyed by the context's unique id, which a context made after
// cudaDeviceReset does not share, so no handle of a destroyed context is
// reused).  The events are shared, so a fork and its join are enqueued under
// the mutex.
struct SideStream {
  unsigned long long ctx = 0;
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
std::vector<SideStream> g_side;

// Unique id of the calling thread's current context (the runtime makes the
// device's primary context current if there is none yet).  Call with
// g_side_mu held (the entry points are cached in statics).
cudaError_t current_context_id(unsigned long long *id) {
  using GetCurrent = CUresult (*)(CUcontext *);
  using GetId = CUresult (*)(CUcontext, unsigned long long *);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  if (!get_current || !get_id) {
    void *f = nullptr, *g = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q1);
    if (e != cudaSuccess) return e;
    e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &g, 12000, cudaEnableDefault, &q2);
    if (e != cudaSuccess) return e;
    if (q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f || !g)
      return cudaErrorNotSupported;
    get_current = reinterpret_cast<GetCurrent>(f);
    get_id = reinterpret_cast<GetId>(g);
  }
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (!c) {  // no context current yet: the runtime makes the device's primary one current
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    if (get_current(&c) != CUDA_SUCCESS || !c) return cudaErrorDeviceUninitialized;
  }
  if (get_id(c, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

// The current context's side stream, created on first use; call with
// g_side_mu held.
cudaError_t side_stream(SideStream **out) {
  unsigned long long ctx = 0;
  cudaError_t e = current_context_id(&ctx);
  if (e != cudaSuccess) return e;
  for (SideStream &ss : g_side)
    if (ss.ctx == ctx) {
      *out = &ss;
      return cudaSuccess;
    }
  SideStream ss;
  ss.ctx = ctx;
  if ((e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
  if ((e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != cudaSuccess) {
    if (ss.fork) cudaEventDestroy(ss.fork);
    cudaStreamDestroy(ss.s);
    return e;
  }
  g_side.push_back(ss);
  *out = &g_side.back();
  return cudaSuccess;
}

thread_local cudaError_t g_last_cuda = cudaSuccess;

// Map a CUDA status to DKV_OK / DKV_E_CUDA, remembering the CUDA error.
int32_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DKV_OK;
  g_last_cuda = e;
  return DKV_E_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Profiler {
  int32_t max_calls = 0;
  int32_t next = 0;
  std::vector<cudaEvent_t> ev;  // [max_calls][DKV_PROFILE_KERNELS + 1]
};

bool valid_pool(const dkv_pool *p) {
  if (!p) return false;
  if (p->F < 1 || p->F > INT32_MAX || p->P < 2 || (p->P & 1) || p->P > (1 << 16)) return false;
  if (p->scheme < 0 || p->scheme >= dkv::kSchemes) return false;
  if (!p->free_list || !p->cursors || !p->rev_unit || !p->rev_idx || !p->page_cls || !p->pages || !p->status)
    return false;
  if (!aligned(p->pages, 16) || !aligned(p->cursors, 8) || !aligned(p->free_list, 4) || !aligned(p->rev_unit, 4) ||
      !aligned(p->rev_idx, 4) || !aligned(p->status, 4))
    return false;
  return true;
}

bool valid_shape(const dkv_batch *b) {
  if (!b) return false;
  if (b->D != DKV_HEAD_DIM || b->L < 1 || b->R < 1 || b->Hkv < 1 || b->Hq < b->Hkv || b->Hq % b->Hkv != 0 ||
      b->Hq > dkv::kMaxHq)
    return false;
  if (b->T < 0 || b->T > INT32_MAX || b->max_len < 0) return false;
  const int64_t U = static_cast<int64_t>(b->L) * b->R * b->Hkv;
  if (U > INT32_MAX || b->unit_base < 0 || b->unit_base + U > INT32_MAX) return false;
  // K / V rows are addressed with 32-bit TMA row coordinates
  if (static_cast<int64_t>(b->L) * b->T * b->Hkv > INT32_MAX) return false;
  return true;
}

bool valid_decode(const dkv_decode_batch *b) {
  if (!b) return false;
  if (b->D != DKV_HEAD_DIM || b->L < 1 || b->R < 1 || b->Hkv < 1 || b->Hq < b->Hkv || b->Hq % b->Hkv != 0 ||
      b->Hq > dkv::kMaxHq || b->R > 65535 || b->L > 65535)
    return false;
  if (b->cap < 16 || (b->cap % 16) != 0) return false;
  if (b->window < 0 || (b->mode != 0 && b->mode != 1)) return false;
  const int64_t U = static_cast<int64_t>(b->L) * b->R * b->Hkv;
  if (U > INT32_MAX || b->unit_base < 0 || b->unit_base + U > INT32_MAX) return false;
  return true;
}

bool decode_pointers(const dkv_decode_batch *b) {
  return b->k_new && b->v_new && b->sig_sum && b->sig_cnt && b->ctx_lens && b->new_lens && b->classes &&
         b->slot_of && aligned(b->k_new, 16) && aligned(b->v_new, 16) && aligned(b->sig_sum, 16) &&
         aligned(b->sig_cnt, 4) && aligned(b->ctx_lens, 4) && aligned(b->new_lens, 4) && aligned(b->classes, 16) &&
         aligned(b->slot_of, 4);
}

dkv::DecodeArgs decode_args(const dkv_decode_batch *b, const dkv_pool *pool, const dkv_tables *t) {
  dkv::DecodeArgs a{};
  a.pg = dkv::page_geom(pool->scheme, pool->P);
  a.L = b->L; a.R = b->R; a.Hq = b->Hq; a.Hkv = b->Hkv; a.G = b->Hq / b->Hkv;
  a.P = pool->P; a.pmax = t->pmax; a.cap = b->cap;
  a.window = b->window; a.mode = b->mode; a.rchunk = dkv::kReclassChunk;
  a.F = pool->F; a.U = static_cast<int64_t>(b->L) * b->R * b->Hkv; a.unit_base = b->unit_base;
  a.k_new = static_cast<const uint16_t *>(b->k_new); a.v_new = static_cast<const uint16_t *>(b->v_new);
  a.sig_sum = b->sig_sum; a.sig_cnt = b->sig_cnt; a.ctx_lens = b->ctx_lens; a.new_lens = b->new_lens;
  a.classes = b->classes; a.slot_of = b->slot_of;
  a.free_list = pool->free_list; a.cursors = pool->cursors; a.rev_unit = pool->rev_unit; a.rev_idx = pool->rev_idx;
  a.page_cls = pool->page_cls; a.pages = pool->pages; a.status = pool->status;
  a.fwd = t->fwd; a.unit_hdr = t->unit_hdr;
  return a;
}

bool valid_decode_tables(const dkv_decode_batch *b, const dkv_pool *pool, const dkv_tables *t) {
  if (!t || !t->fwd || !t->unit_hdr || !aligned(t->unit_hdr, 16) || !aligned(t->fwd, 4) || t->pmax < 2) return false;
  const int64_t U = static_cast<int64_t>(b->L) * b->R * b->Hkv;
  // the scan packs two sums of at most U * pmax pages into 31 bits each
  if (U * t->pmax >= (int64_t{1} << 31)) return false;
  (void)pool;
  return true;
}

// Largest head group per apply block whose shared memory fits; 0 if none.
int32_t apply_heads(int32_t Hkv, int32_t words, int32_t pmax) {
  int32_t hpc = Hkv < dkv::kMaxApplyWarps ? Hkv : dkv::kMaxApplyWarps;
  while (hpc > 1 && dkv::apply_smem(hpc, words, pmax) > 96 * 1024) hpc = (hpc + 1) / 2;
  return dkv::apply_smem(hpc, words, pmax) <= 200 * 1024 ? hpc : 0;
}

}  // namespace

extern "C" {

int32_t dkv_version(void) { return 100; }

int32_t dkv_build_flags(void) { return dkv::kChecked ? DKV_BUILD_CHECKED : 0; }

const char *dkv_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda); }

const char *dkv_status_string(int32_t code) {
  switch (code) {
    case DKV_OK: return "ok";
    case DKV_E_INVAL: return "invalid argument";
    case DKV_E_NOMEM: return "page demand exceeds the free pages";
    case DKV_E_RANGE: return "a value to quantise is non-finite or above 65504 in magnitude";
    case DKV_E_TIMEOUT: return "a bounded wait of the page scan gave up";
    case DKV_E_INTERNAL: return "internal consistency check failed";
    case DKV_E_CUDA: return "a CUDA call failed";
    case DKV_E_LENS: return "request lengths disagree with T or max_len";
    default: return "unknown status";
  }
}

int32_t dkv_page_bytes(int32_t scheme, int32_t P, int64_t *bytes) {
  if (!bytes || scheme < 0 || scheme >= dkv::kSchemes || P < 2 || (P & 1) || P > (1 << 16)) return DKV_E_INVAL;
  *bytes = dkv::page_geom(scheme, P).bytes;
  return DKV_OK;
}

int32_t dkv_workspace_size(const dkv_batch *b, size_t *bytes) {
  if (!bytes || !valid_shape(b)) return DKV_E_INVAL;
  *bytes = dkv::ws_layout(b->L, b->R, b->Hkv, b->T).bytes;
  return DKV_OK;
}

int32_t dkv_init_pool(const dkv_pool *pool, void *stream) {
  if (!valid_pool(pool)) return DKV_E_INVAL;
  return cuda_status(dkv::launch_init_pool(*pool, static_cast<cudaStream_t>(stream)));
}

int32_t dkv_compact(const dkv_batch *b, const dkv_params *p, const dkv_pool *pool, const dkv_tables *t,
                    void *workspace, size_t workspace_bytes, void *stream) {
  if (!valid_shape(b) || !p || !valid_pool(pool) || !t) return DKV_E_INVAL;
  if (!b->k || !b->v || !b->sig_sum || !b->sig_cnt || !b->lens || !b->classes) return DKV_E_INVAL;
  if (!aligned(b->k, 16) || !aligned(b->v, 16) || !aligned(b->sig_sum, 16) || !aligned(b->sig_cnt, 4) ||
      !aligned(b->lens, 4))
    return DKV_E_INVAL;
  if (!(std::isfinite(p->alpha_h) && std::isfinite(p->alpha_l)) || !(p->alpha_l >= 0.0f) ||
      !(p->alpha_h >= p->alpha_l) || p->reserved != 0)
    return DKV_E_INVAL;
  if (!t->fwd || !t->unit_hdr || !aligned(t->unit_hdr, 16) || !aligned(t->fwd, 4)) return DKV_E_INVAL;
  const int64_t need_pmax = (static_cast<int64_t>(b->max_len) + pool->P - 1) / pool->P + 1;
  if (t->pmax < need_pmax) return DKV_E_INVAL;
  const dkv::WsLayout lay = dkv::ws_layout(b->L, b->R, b->Hkv, b->T);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < lay.bytes) return DKV_E_INVAL;
  int sms = 0, pack_bps = 0;
  if (!device_info(&sms, &pack_bps)) return cuda_status(cudaErrorInvalidDevice);

  CompactArgs a{};
  a.pg = dkv::page_geom(pool->scheme, pool->P);
  a.L = b->L; a.R = b->R; a.Hq = b->Hq; a.Hkv = b->Hkv; a.G = b->Hq / b->Hkv;
  a.P = pool->P; a.pmax = t->pmax;
  a.spin_limit = p->spin_limit < 0 ? (1 << 22) : p->spin_limit;
  a.T = b->T; a.F = pool->F; a.U = static_cast<int64_t>(b->L) * b->R * b->Hkv; a.unit_base = b->unit_base;
  a.max_len = b->max_len;
  a.alpha_h = p->alpha_h; a.alpha_l = p->alpha_l;
  a.k = static_cast<const uint16_t *>(b->k); a.v = static_cast<const uint16_t *>(b->v);
  a.sig_sum = b->sig_sum; a.sig_cnt = b->sig_cnt; a.lens = b->lens; a.classes = b->classes;
  a.free_list = pool->free_list; a.cursors = pool->cursors; a.rev_unit = pool->rev_unit; a.rev_idx = pool->rev_idx;
  a.page_cls = pool->page_cls; a.pages = pool->pages; a.status = pool->status;
  a.fwd = t->fwd; a.unit_hdr = t->unit_hdr;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  a.ws = reinterpret_cast<dkv::WsHeader *>(ws);
  a.tok_off = reinterpret_cast<int64_t *>(ws + lay.tok_off);
  a.tile_off = reinterpret_cast<int32_t *>(ws + lay.tile_off);
  a.tile_info = reinterpret_cast<dkv::TileInfo *>(ws + lay.tile_info);
  a.part = reinterpret_cast<uint64_t *>(ws + lay.part);
  a.unit = reinterpret_cast<dkv::UnitInfo *>(ws + lay.unit);
  a.mask = reinterpret_cast<uint32_t *>(ws + lay.mask);
  a.desc = reinterpret_cast<dkv::TileDesc *>(ws + lay.desc);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Profiler *prof = static_cast<Profiler *>(p->profiler);
  cudaEvent_t *ev = nullptr;
  if (prof && prof->next < prof->max_calls) {
    ev = prof->ev.data() + static_cast<size_t>(prof->next) * (DKV_PROFILE_KERNELS + 1);
    prof->next++;
  }
  auto mark = [&](int i) {
    if (ev) cudaEventRecord(ev[i], s);
  };
  const int64_t tr_max = b->T / dkv::kTileTokens + b->R;
  const int64_t classify_items = static_cast<int64_t>(b->L) * tr_max;
  const int classify_grid = static_cast<int>(std::min<int64_t>(classify_items, static_cast<int64_t>(sms) * 8));
  const int pack_grid = sms * pack_bps;
  const int commit_grid = static_cast<int>(std::min<int64_t>((a.U + 7) / 8, static_cast<int64_t>(sms) * 8));

  mark(0);
  if (const int32_t rc = cuda_status(dkv::launch_prep(a, s))) return rc;
  mark(1);
  if (const int32_t rc = cuda_status(dkv::launch_classify(a, std::max(classify_grid, 1), sms, s))) return rc;
  mark(2);
  if (const int32_t rc = cuda_status(dkv::launch_scan(a, lay.npart, s))) return rc;
  mark(3);
  {
    // the unused halves of the new high pages are cleared on the side stream
    // while k_pack runs (they need only the scan's placement)
    std::lock_guard<std::mutex> lock(g_side_mu);
    SideStream *ss = nullptr;
    if (const int32_t rc = cuda_status(side_stream(&ss))) return rc;
    if (const int32_t rc = cuda_status(cudaEventRecord(ss->fork, s))) return rc;
    if (const int32_t rc = cuda_status(cudaStreamWaitEvent(ss->s, ss->fork, 0))) return rc;
    if (const int32_t rc = cuda_status(dkv::launch_clear_hi(a, sms, ss->s))) return rc;
    if (const int32_t rc = cuda_status(cudaEventRecord(ss->join, ss->s))) return rc;
    if (const int32_t rc = cuda_status(dkv::launch_pack(a, pack_grid, s))) return rc;
    mark(4);
    if (const int32_t rc = cuda_status(cudaStreamWaitEvent(s, ss->join, 0))) return rc;
  }
  if (const int32_t rc = cuda_status(dkv::launch_commit(a, std::max(commit_grid, 1), s))) return rc;
  mark(5);
  return DKV_OK;
}

int32_t dkv_decode_workspace_size(const dkv_decode_batch *b, size_t *bytes) {
  if (!bytes || !valid_decode(b)) return DKV_E_INVAL;
  *bytes = dkv::dec_ws_layout(static_cast<int64_t>(b->L) * b->R * b->Hkv, static_cast<int64_t>(b->L) * b->R,
                              static_cast<int64_t>(b->L) * b->R * b->cap * b->Hkv).bytes;
  return DKV_OK;
}

int32_t dkv_decode_index(const dkv_decode_batch *b, const dkv_pool *pool, const dkv_tables *t, void *stream) {
  if (!valid_decode(b) || !valid_pool(pool) || !valid_decode_tables(b, pool, t)) return DKV_E_INVAL;
  if (!b->ctx_lens || !b->classes || !b->slot_of || !aligned(b->ctx_lens, 4) || !aligned(b->slot_of, 4))
    return DKV_E_INVAL;
  int sms = 0, pack_bps = 0;
  if (!device_info(&sms, &pack_bps)) return cuda_status(cudaErrorInvalidDevice);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rows = static_cast<size_t>(b->L) * b->R * b->cap * b->Hkv;
  if (const int32_t rc = cuda_status(cudaMemsetAsync(b->classes, 0, rows, s))) return rc;
  if (const int32_t rc = cuda_status(cudaMemsetAsync(b->slot_of, 0xff, rows * sizeof(int32_t), s))) return rc;
  const dkv::DecodeArgs a = decode_args(b, pool, t);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((a.U + 7) / 8, int64_t{sms} * 8)));
  return cuda_status(dkv::launch_index(a, grid, s));
}

int32_t dkv_decode_step(const dkv_decode_batch *b, const dkv_params *p, const dkv_pool *pool, const dkv_tables *t,
                        void *workspace, size_t workspace_bytes, void *stream) {
  if (!valid_decode(b) || !p || !valid_pool(pool) || !decode_pointers(b) || !valid_decode_tables(b, pool, t))
    return DKV_E_INVAL;
  if (!(std::isfinite(p->alpha_h) && std::isfinite(p->alpha_l)) || !(p->alpha_l >= 0.0f) ||
      !(p->alpha_h >= p->alpha_l) || p->reserved != 0)
    return DKV_E_INVAL;
  const int64_t U = static_cast<int64_t>(b->L) * b->R * b->Hkv;
  const dkv::DecWsLayout lay =
      dkv::dec_ws_layout(U, static_cast<int64_t>(b->L) * b->R, static_cast<int64_t>(b->L) * b->R * b->cap * b->Hkv);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < lay.bytes) return DKV_E_INVAL;
  const int32_t words = (b->cap + 31) / 32;
  const int32_t hpc = apply_heads(b->Hkv, words, t->pmax);
  if (hpc == 0) return DKV_E_INVAL;
  int sms = 0, pack_bps = 0;
  if (!device_info(&sms, &pack_bps)) return cuda_status(cudaErrorInvalidDevice);

  dkv::DecodeArgs a = decode_args(b, pool, t);
  a.spin_limit = p->spin_limit < 0 ? (1 << 22) : p->spin_limit;
  a.alpha_h = p->alpha_h;
  a.alpha_l = p->alpha_l;
  a.rchunk = dkv::reclass_chunk(static_cast<int64_t>(b->L) * b->R, b->cap, sms);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  a.ws = reinterpret_cast<dkv::DecWsHeader *>(ws);
  a.ucnt = reinterpret_cast<int4 *>(ws + lay.ucnt);
  a.part = reinterpret_cast<uint64_t *>(ws + lay.part);
  a.plan = reinterpret_cast<dkv::DecPlan *>(ws + lay.plan);
  a.lcnt = reinterpret_cast<int32_t *>(ws + lay.lcnt);
  a.list = reinterpret_cast<uint32_t *>(ws + lay.list);
  a.jobs = reinterpret_cast<dkv::DemJob *>(ws + lay.jobs);
  a.njobs = lay.njobs;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Profiler *prof = static_cast<Profiler *>(p->profiler);
  cudaEvent_t *ev = nullptr;
  if (prof && prof->next < prof->max_calls) {
    ev = prof->ev.data() + static_cast<size_t>(prof->next) * (DKV_PROFILE_KERNELS + 1);
    prof->next++;
  }
  auto mark = [&](int i) {
    if (ev) cudaEventRecord(ev[i], s);
  };
  mark(0);
  if (const int32_t rc = cuda_status(cudaMemsetAsync(ws, 0, lay.reset, s))) return rc;
  mark(1);
  if (const int32_t rc = cuda_status(a.mode == 1 ? dkv::launch_candidate(a, s) : dkv::launch_reclass(a, s))) return rc;
  mark(2);
  if (const int32_t rc = cuda_status(dkv::launch_dscan(a, lay.npart, s))) return rc;
  mark(3);
  if (const int32_t rc = cuda_status(dkv::launch_apply(a, hpc, words, s))) return rc;
  mark(4);
  if (const int32_t rc = cuda_status(dkv::launch_demote(a, sms * 8, s))) return rc;
  mark(5);
  return DKV_OK;
}

int32_t dkv_decode_attention(const dkv_attn_batch *b, const dkv_pool *pool, const dkv_tables *t, void *stream) {
  if (!b || !valid_pool(pool) || !t || !t->fwd || !t->unit_hdr || !aligned(t->unit_hdr, 16) ||
      !aligned(t->fwd, 4) || t->pmax < 2)
    return DKV_E_INVAL;
  if (b->L < 1 || b->R < 0 || b->Hkv < 1 || b->Hq < b->Hkv || b->Hq % b->Hkv != 0 ||
      b->Hq / b->Hkv > dkv::kAttendMaxG || b->cap < 1 || b->layer0 < 0 || b->n_layers < 0 ||
      b->layer0 + static_cast<int64_t>(b->n_layers) > b->L || !std::isfinite(b->scale))
    return DKV_E_INVAL;
  if (!b->q || !b->out || !b->ctx_lens || !aligned(b->q, 16) || !aligned(b->out, 4) || !aligned(b->ctx_lens, 4))
    return DKV_E_INVAL;
  if ((b->k_new == nullptr) != (b->v_new == nullptr)) return DKV_E_INVAL;
  if (b->k_new && (!b->new_lens || !aligned(b->k_new, 16) || !aligned(b->v_new, 16) || !aligned(b->new_lens, 4)))
    return DKV_E_INVAL;
  if (b->sig_sum && !aligned(b->sig_sum, 4)) return DKV_E_INVAL;
  const int64_t units = static_cast<int64_t>(b->n_layers) * b->R * b->Hkv;
  // one cluster of S blocks per unit, the fewest whose shares of a unit's
  // logits (at most cap + 1 tokens) fit one block's shared memory
  const int32_t G = b->Hq / b->Hkv;
  // (first asking for a size that lets attend_blocks_per_sm blocks share an SM)
  int32_t S = 0, cmax = 0;
  const size_t budgets[2] = {static_cast<size_t>(220 * 1024) / dkv::attend_blocks_per_sm(G) - 1024, 220 * 1024};
  for (int pass = 0; pass < 2 && S == 0; ++pass) {
    for (int32_t s = 1; s <= 8 && S == 0; s *= 2) {
      const int32_t c = static_cast<int32_t>((static_cast<int64_t>(b->cap) + 1 + s - 1) / s);
      if (dkv::attend_layout(c, G, t->pmax, pool->P).bytes <= budgets[pass]) {
        S = s;
        cmax = c;
      }
    }
  }
  if (S == 0 || units * S > INT32_MAX) return DKV_E_INVAL;
  dkv::AttnArgs a{};
  a.L = b->L; a.R = b->R; a.Hq = b->Hq; a.Hkv = b->Hkv; a.G = G; a.P = pool->P; a.pmax = t->pmax;
  a.cap = b->cap; a.layer0 = b->layer0; a.n_layers = b->n_layers; a.cmax = cmax;
  a.scheme = pool->scheme;
  a.F = pool->F; a.units = units; a.scale = b->scale;
  a.q = static_cast<const uint16_t *>(b->q);
  a.k_new = static_cast<const uint16_t *>(b->k_new);
  a.v_new = static_cast<const uint16_t *>(b->v_new);
  a.new_lens = b->new_lens; a.ctx_lens = b->ctx_lens; a.out = b->out; a.sig_sum = b->sig_sum;
  a.fwd = t->fwd; a.unit_hdr = t->unit_hdr; a.pages = pool->pages; a.status = pool->status;
  return cuda_status(dkv::launch_attend(a, S, static_cast<cudaStream_t>(stream)));
}

int32_t dkv_prefill_attention(const dkv_prefill_batch *b, const dkv_pool *pool, void *stream) {
  if (!b || !pool || !pool->status || !aligned(pool->status, 4)) return DKV_E_INVAL;
  if (b->L < 1 || b->R < 0 || b->Hkv < 1 || b->Hq < b->Hkv || b->Hq % b->Hkv != 0 || b->max_len < 0 ||
      b->T < 0 || b->reserved != 0 || !std::isfinite(b->scale))
    return DKV_E_INVAL;
  if (b->R > 65535 || static_cast<int64_t>(b->L) * b->Hq > 65535) return DKV_E_INVAL;  // grid y and z
  if (static_cast<int64_t>(b->L) * b->T >= INT32_MAX) return DKV_E_INVAL;              // 32-bit TMA row coordinates
  if (!b->q || !b->k || !b->v || !b->lens || !b->out || !b->sig_sum || !b->sig_cnt || !aligned(b->q, 16) ||
      !aligned(b->k, 16) || !aligned(b->v, 16) || !aligned(b->lens, 4) || !aligned(b->out, 8) ||
      !aligned(b->sig_sum, 4) || !aligned(b->sig_cnt, 4))
    return DKV_E_INVAL;
  dkv::PrefillArgs a{};
  a.L = b->L; a.R = b->R; a.Hq = b->Hq; a.Hkv = b->Hkv; a.G = b->Hq / b->Hkv; a.max_len = b->max_len;
  a.T = b->T; a.scale = b->scale;
  a.q = static_cast<const uint16_t *>(b->q);
  a.k = static_cast<const uint16_t *>(b->k);
  a.v = static_cast<const uint16_t *>(b->v);
  a.lens = b->lens; a.out = b->out; a.sig_sum = b->sig_sum; a.sig_cnt = b->sig_cnt; a.status = pool->status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t sig_bytes = sizeof(float) * static_cast<size_t>(b->L) * static_cast<size_t>(b->T) * b->Hq;
  if (sig_bytes > 0)
    if (const int32_t rc = cuda_status(cudaMemsetAsync(b->sig_sum, 0, sig_bytes, s))) return rc;
  return cuda_status(dkv::launch_prefill(a, s));
}

int32_t dkv_dequant_page(const dkv_pool *pool, int32_t page_id, float *k_out, float *v_out, int32_t *pos_out,
                         void *stream) {
  if (!valid_pool(pool) || page_id < 0 || page_id >= pool->F || !k_out || !v_out || !pos_out) return DKV_E_INVAL;
  return cuda_status(
      dkv::launch_dequant(*pool, nullptr, page_id, 1, k_out, v_out, pos_out, static_cast<cudaStream_t>(stream)));
}

int32_t dkv_dequant_pages(const dkv_pool *pool, const int32_t *page_ids, int32_t n, float *k_out, float *v_out,
                          int32_t *pos_out, void *stream) {
  if (!valid_pool(pool) || n < 0 || (n > 0 && (!page_ids || !k_out || !v_out || !pos_out))) return DKV_E_INVAL;
  if (n == 0) return DKV_OK;
  return cuda_status(
      dkv::launch_dequant(*pool, page_ids, 0, n, k_out, v_out, pos_out, static_cast<cudaStream_t>(stream)));
}

int32_t dkv_get_status(const dkv_pool *pool, void *stream) {
  if (!pool || !pool->status) return DKV_E_INVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, pool->status, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess) return DKV_E_CUDA;
  if (cudaMemsetAsync(pool->status, 0, sizeof(int32_t), s) != cudaSuccess) return DKV_E_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DKV_E_CUDA;
  return host;
}

int32_t dkv_profiler_create(int32_t max_calls, void **profiler) {
  if (!profiler || max_calls < 1) return DKV_E_INVAL;
  Profiler *pr = new (std::nothrow) Profiler();
  if (!pr) return DKV_E_CUDA;
  pr->max_calls = max_calls;
  pr->ev.resize(static_cast<size_t>(max_calls) * (DKV_PROFILE_KERNELS + 1));
  for (auto &e : pr->ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      dkv_profiler_destroy(pr);
      return DKV_E_CUDA;
    }
  }
  *profiler = pr;
  return DKV_OK;
}

int32_t dkv_profiler_read(void *profiler, float *ms, int32_t capacity_calls) {
  Profiler *pr = static_cast<Profiler *>(profiler);
  if (!pr || (!ms && capacity_calls > 0)) return DKV_E_INVAL;
  const int32_t n = pr->next < capacity_calls ? pr->next : capacity_calls;
  for (int32_t c = 0; c < n; ++c) {
    cudaEvent_t *ev = pr->ev.data() + static_cast<size_t>(c) * (DKV_PROFILE_KERNELS + 1);
    if (cudaEventSynchronize(ev[DKV_PROFILE_KERNELS]) != cudaSuccess) return DKV_E_CUDA;
    for (int k = 0; k < DKV_PROFILE_KERNELS; ++k) {
      float t = 0.0f;
      if (cudaEventElapsedTime(&t, ev[k], ev[k + 1]) != cudaSuccess) return DKV_E_CUDA;
      ms[c * DKV_PROFILE_KERNELS + k] = t;
    }
  }
  pr->next = 0;
  return n;
}

int32_t dkv_profiler_destroy(void *profiler) {
  Profiler *pr = static_cast<Profiler *>(profiler);
  if (!pr) return DKV_E_INVAL;
  for (auto &e : pr->ev)
    if (e) cudaEventDestroy(e);
  delete pr;
  return DKV_OK;
}

}  // extern "C"
