"""Thin ctypes binding over libdkv.so (argument marshalling only).

Every function here forwards to the C entry point of the same name declared
in ``include/dkv.h``; all compute runs in the library's CUDA kernels.  PyTorch
only provides device memory and the current stream.  There is no fallback:
if ``libdkv.so`` has not been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# DKV_LIBRARY=checked selects the bounds-checked build (lib/libdkv_checked.so),
# DKV_LIBRARY=sanitized the one with sanitized host code (lib/libdkv_san.so)
LIB_PATH = os.path.join(HERE, "lib", {"checked": "libdkv_checked.so", "sanitized": "libdkv_san.so"}.get(
    os.environ.get("DKV_LIBRARY", ""), "libdkv.so"))

DKV_OK = 0
DKV_E_INVAL = -1
DKV_E_NOMEM = -2
DKV_E_RANGE = -3
DKV_E_TIMEOUT = -4
DKV_E_INTERNAL = -5
DKV_E_CUDA = -6
DKV_E_LENS = -7
DKV_PROFILE_KERNELS = 5
KERNEL_NAMES = ("k_prep", "k_classify", "k_scan", "k_pack", "k_commit")

_lib = None


class DkvError(RuntimeError):
    def __init__(self, code: int, what: str):
        detail = f" [{load().dkv_last_cuda_error().decode()}]" if code == DKV_E_CUDA else ""
        super().__init__(f"{what}: {status_string(code)} ({code}){detail}")
        self.code = code


class dkv_batch(ctypes.Structure):
    _fields_ = [
        ("L", ctypes.c_int32), ("R", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("D", ctypes.c_int32), ("max_len", ctypes.c_int32), ("T", ctypes.c_int64),
        ("unit_base", ctypes.c_int64), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("sig_sum", ctypes.c_void_p), ("sig_cnt", ctypes.c_void_p), ("lens", ctypes.c_void_p),
        ("classes", ctypes.c_void_p),
    ]


class dkv_params(ctypes.Structure):
    _fields_ = [("alpha_h", ctypes.c_float), ("alpha_l", ctypes.c_float), ("spin_limit", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("profiler", ctypes.c_void_p)]


class dkv_pool(ctypes.Structure):
    _fields_ = [
        ("F", ctypes.c_int64), ("P", ctypes.c_int32), ("scheme", ctypes.c_int32),
        ("free_list", ctypes.c_void_p), ("cursors", ctypes.c_void_p), ("rev_unit", ctypes.c_void_p),
        ("rev_idx", ctypes.c_void_p), ("page_cls", ctypes.c_void_p), ("pages", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
    ]


class dkv_tables(ctypes.Structure):
    _fields_ = [("fwd", ctypes.c_void_p), ("pmax", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("unit_hdr", ctypes.c_void_p)]


class dkv_decode_batch(ctypes.Structure):
    _fields_ = [
        ("L", ctypes.c_int32), ("R", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("D", ctypes.c_int32), ("cap", ctypes.c_int32), ("unit_base", ctypes.c_int64),
        ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p), ("sig_sum", ctypes.c_void_p),
        ("sig_cnt", ctypes.c_void_p), ("ctx_lens", ctypes.c_void_p), ("new_lens", ctypes.c_void_p),
        ("classes", ctypes.c_void_p), ("slot_of", ctypes.c_void_p), ("window", ctypes.c_int32),
        ("mode", ctypes.c_int32),
    ]


class dkv_attn_batch(ctypes.Structure):
    _fields_ = [
        ("L", ctypes.c_int32), ("R", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("cap", ctypes.c_int32), ("layer0", ctypes.c_int32), ("n_layers", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
        ("new_lens", ctypes.c_void_p), ("ctx_lens", ctypes.c_void_p), ("scale", ctypes.c_float),
        ("out", ctypes.c_void_p), ("sig_sum", ctypes.c_void_p),
    ]


class dkv_prefill_batch(ctypes.Structure):
    _fields_ = [
        ("L", ctypes.c_int32), ("R", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("max_len", ctypes.c_int32), ("reserved", ctypes.c_int32), ("T", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("lens", ctypes.c_void_p),
        ("scale", ctypes.c_float), ("out", ctypes.c_void_p), ("sig_sum", ctypes.c_void_p),
        ("sig_cnt", ctypes.c_void_p),
    ]


def load():
    """Load libdkv.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sigs = {
        "dkv_version": ([], i32),
        "dkv_build_flags": ([], i32),
        "dkv_status_string": ([i32], ctypes.c_char_p),
        "dkv_last_cuda_error": ([], ctypes.c_char_p),
        "dkv_page_bytes": ([i32, i32, P(ctypes.c_int64)], i32),
        "dkv_workspace_size": ([P(dkv_batch), P(ctypes.c_size_t)], i32),
        "dkv_init_pool": ([P(dkv_pool), vp], i32),
        "dkv_compact": ([P(dkv_batch), P(dkv_params), P(dkv_pool), P(dkv_tables), vp, ctypes.c_size_t, vp], i32),
        "dkv_compact_noalloc": ([P(dkv_batch), P(dkv_params), P(dkv_pool), P(dkv_tables), vp], i32),
        "dkv_dequant_page": ([P(dkv_pool), i32, vp, vp, vp, vp], i32),
        "dkv_dequant_pages": ([P(dkv_pool), vp, i32, vp, vp, vp, vp], i32),
        "dkv_get_status": ([P(dkv_pool), vp], i32),
        "dkv_decode_workspace_size": ([P(dkv_decode_batch), P(ctypes.c_size_t)], i32),
        "dkv_decode_index": ([P(dkv_decode_batch), P(dkv_pool), P(dkv_tables), vp], i32),
        "dkv_decode_step": ([P(dkv_decode_batch), P(dkv_params), P(dkv_pool), P(dkv_tables), vp, ctypes.c_size_t,
                             vp], i32),
        "dkv_decode_attention": ([P(dkv_attn_batch), P(dkv_pool), P(dkv_tables), vp], i32),
        "dkv_prefill_attention": ([P(dkv_prefill_batch), P(dkv_pool), vp], i32),
        "dkv_profiler_create": ([i32, P(vp)], i32),
        "dkv_profiler_read": ([vp, vp, i32], i32),
        "dkv_profiler_destroy": ([vp], i32),
    }
    for name, (args, res) in sigs.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def status_string(code: int) -> str:
    return load().dkv_status_string(int(code)).decode()


DKV_SCHEME_K8V4_K4V2 = 0
DKV_SCHEME_K8V2_K4V1 = 1
DKV_SCHEME_K4V8_K2V4 = 2


def dkv_page_bytes(scheme: int, P: int) -> int:
    n = ctypes.c_int64(0)
    rc = load().dkv_page_bytes(int(scheme), int(P), ctypes.byref(n))
    if rc != DKV_OK:
        raise DkvError(rc, "dkv_page_bytes")
    return int(n.value)


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _p(t) -> int | None:
    return None if t is None else t.data_ptr()


class DevicePool:
    """Pool state in device memory (torch tensors owned by this object)."""

    def __init__(self, F: int, P: int, device="cuda", scheme: int = 0):
        self.F, self.P, self.scheme = int(F), int(P), int(scheme)
        d = torch.device(device)
        self.free_list = torch.empty(self.F, dtype=torch.int32, device=d)
        self.cursors = torch.zeros(2, dtype=torch.int64, device=d)   # uint64 bit patterns
        self.rev_unit = torch.empty(self.F, dtype=torch.int32, device=d)
        self.rev_idx = torch.empty(self.F, dtype=torch.int32, device=d)
        self.page_cls = torch.empty(self.F, dtype=torch.uint8, device=d)
        self.pages = torch.empty((self.F, dkv_page_bytes(self.scheme, self.P)), dtype=torch.uint8, device=d)
        self.status = torch.zeros(1, dtype=torch.int32, device=d)

    def c(self) -> dkv_pool:
        return dkv_pool(self.F, self.P, self.scheme, _p(self.free_list), _p(self.cursors), _p(self.rev_unit),
                        _p(self.rev_idx), _p(self.page_cls), _p(self.pages), _p(self.status))


class DeviceTables:
    def __init__(self, U: int, pmax: int, device="cuda"):
        self.pmax = int(pmax)
        self.fwd = torch.empty((U, self.pmax), dtype=torch.int32, device=device)
        self.unit_hdr = torch.empty((U, 4), dtype=torch.int32, device=device)

    def c(self) -> dkv_tables:
        return dkv_tables(_p(self.fwd), self.pmax, 0, _p(self.unit_hdr))


def make_batch(inp: dict, classes: torch.Tensor, max_len: int, unit_base: int = 0) -> dkv_batch:
    return dkv_batch(int(inp["L"]), int(inp["R"]), int(inp["Hq"]), int(inp["Hkv"]), 128, int(max_len),
                     int(inp["T"]), int(unit_base), _p(inp["k"]), _p(inp["v"]), _p(inp["sig_sum"]),
                     _p(inp["sig_cnt"]), _p(inp["lens"]), _p(classes))


def dkv_workspace_size(batch: dkv_batch) -> int:
    n = ctypes.c_size_t(0)
    rc = load().dkv_workspace_size(ctypes.byref(batch), ctypes.byref(n))
    if rc != DKV_OK:
        raise DkvError(rc, "dkv_workspace_size")
    return int(n.value)


def dkv_init_pool(pool: DevicePool, stream=None) -> None:
    c = pool.c()
    rc = load().dkv_init_pool(ctypes.byref(c), _stream(stream))
    if rc != DKV_OK:
        raise DkvError(rc, "dkv_init_pool")


def dkv_compact(batch: dkv_batch, alpha_h: float, alpha_l: float, pool: DevicePool, tables: DeviceTables,
                workspace: torch.Tensor, stream=None, spin_limit: int = -1, profiler=None) -> None:
    """Enqueue one compaction; device-side errors are read with dkv_get_status."""
    params = dkv_params(float(alpha_h), float(alpha_l), int(spin_limit), 0,
                        None if profiler is None else profiler.handle)
    pc, tc = pool.c(), tables.c()
    rc = load().dkv_compact(ctypes.byref(batch), ctypes.byref(params), ctypes.byref(pc), ctypes.byref(tc),
                            _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != DKV_OK:
        raise DkvError(rc, "dkv_compact")


def dkv_compact_noalloc(batch: dkv_batch, alpha_h: float, alpha_l: float, pool: DevicePool,
                        tables: DeviceTables, stream=None, spin_limit: int = -1) -> None:
    """dkv_compact with the library's built-in scratch instead of a workspace."""
    params = dkv_params(float(alpha_h), float(alpha_l), int(spin_limit), 0, None)
    pc, tc = pool.c(), tables.c()
    rc = load().dkv_compact_noalloc(ctypes.byref(batch), ctypes.byref(params), ctypes.byref(pc), ctypes.byref(tc),
                                    _stream(stream))
    if rc != DKV_OK:
        raise DkvError(rc, "dkv_compact_noalloc")


def dkv_get_status(pool: DevicePool, stream=None) -> int:
    c = pool.c()
    return int(load().dkv_get_status(ctypes.byref(c), _stream(stream)))


def dkv_dequant_page(pool: DevicePool, page_id: int, stream=None):
    P = pool.P
    dev = pool.pages.device
    k = torch.empty((2 * P, 128), dtype=torch.float32, device=dev)
    v = torch.empty((2 * P, 128), dtype=torch.float32, device=dev)
    pos = torch.empty(2 * P, dtype=torch.int32, device=dev)
    c = pool.c()
    rc = load().dkv_dequant_page(ctypes.byref(c), int(page_id), _p(k), _p(v), _p(pos), _stream(stream))
    if rc != DKV_OK:
        raise DkvError(rc, "dkv_dequant_page")
    return k, v, pos


def dkv_dequant_pages(pool: DevicePool, page_ids: torch.Tensor, stream=None):
    P = pool.P
    n = int(page_ids.numel())
    dev = pool.pages.device
    ids = page_ids.to(device=dev, dtype=torch.int32).contiguous()
    k = torch.empty((n, 2 * P, 128), dtype=torch.float32, device=dev)
    v = torch.empty((n, 2 * P, 128), dtype=torch.float32, device=dev)
    pos = torch.empty((n, 2 * P), dtype=torch.int32, device=dev)
    c = pool.c()
    rc = load().dkv_dequant_pages(ctypes.byref(c), _p(ids), n, _p(k), _p(v), _p(pos), _stream(stream))
    if rc != DKV_OK:
        raise DkvError(rc, "dkv_dequant_pages")
    return k, v, pos


class Profiler:
    """Per-kernel CUDA-event timing of dkv_compact calls (library-owned events)."""

    def __init__(self, max_calls: int):
        h = ctypes.c_void_p()
        rc = load().dkv_profiler_create(int(max_calls), ctypes.byref(h))
        if rc != DKV_OK:
            raise DkvError(rc, "dkv_profiler_create")
        self.handle = h.value
        self.max_calls = int(max_calls)

    def read(self):
        """[(ms per kernel) for each recorded call], then starts a new recording."""
        buf = (ctypes.c_float * (self.max_calls * DKV_PROFILE_KERNELS))()
        n = load().dkv_profiler_read(self.handle, buf, self.max_calls)
        if n < 0:
            raise DkvError(n, "dkv_profiler_read")
        return [list(buf[c * DKV_PROFILE_KERNELS:(c + 1) * DKV_PROFILE_KERNELS]) for c in range(n)]

    def close(self):
        if self.handle:
            load().dkv_profiler_destroy(self.handle)
            self.handle = None


class Compactor:
    """Convenience owner of pool, tables, classes and workspace for one shape."""

    def __init__(self, L: int, R: int, Hq: int, Hkv: int, T: int, max_len: int, P: int, F: int, device="cuda",
                 scheme: int = 0):
        self.L, self.R, self.Hq, self.Hkv, self.T, self.max_len = L, R, Hq, Hkv, T, max_len
        self.U = L * R * Hkv
        self.pmax = -(-max_len // P) + 1
        self.pool = DevicePool(F, P, device, scheme=scheme)
        self.tables = DeviceTables(self.U, self.pmax, device)
        self.classes = torch.empty(max(L * T * Hkv, 1), dtype=torch.uint8, device=device)
        probe = dkv_batch(L, R, Hq, Hkv, 128, max_len, T, 0, None, None, None, None, None, None)
        self.workspace = torch.empty(dkv_workspace_size(probe), dtype=torch.uint8, device=device)
        dkv_init_pool(self.pool)

    def batch(self, inp: dict, unit_base: int = 0) -> dkv_batch:
        return make_batch(inp, self.classes, self.max_len, unit_base)

    def compact(self, inp: dict, alpha_h: float, alpha_l: float, stream=None, spin_limit: int = -1,
                profiler=None, unit_base: int = 0) -> None:
        dkv_compact(self.batch(inp, unit_base), alpha_h, alpha_l, self.pool, self.tables, self.workspace,
                    stream=stream, spin_limit=spin_limit, profiler=profiler)


# ------------------------------------------------------------------ decode --

def dkv_decode_workspace_size(batch: dkv_decode_batch) -> int:
    n = ctypes.c_size_t(0)
    rc = load().dkv_decode_workspace_size(ctypes.byref(batch), ctypes.byref(n))
    if rc != DKV_OK:
        raise DkvError(rc, "dkv_decode_workspace_size")
    return int(n.value)


def dkv_decode_index(batch: dkv_decode_batch, pool: DevicePool, tables, stream=None) -> None:
    pc, tc = pool.c(), tables.c()
    rc = load().dkv_decode_index(ctypes.byref(batch), ctypes.byref(pc), ctypes.byref(tc), _stream(stream))
    if rc != DKV_OK:
        raise DkvError(rc, "dkv_decode_index")


def dkv_decode_step(batch: dkv_decode_batch, alpha_h: float, alpha_l: float, pool: DevicePool, tables,
                    workspace: torch.Tensor, stream=None, spin_limit: int = -1, profiler=None) -> None:
    params = dkv_params(float(alpha_h), float(alpha_l), int(spin_limit), 0,
                        None if profiler is None else profiler.handle)
    pc, tc = pool.c(), tables.c()
    rc = load().dkv_decode_step(ctypes.byref(batch), ctypes.byref(params), ctypes.byref(pc), ctypes.byref(tc),
                                _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != DKV_OK:
        raise DkvError(rc, "dkv_decode_step")


def dkv_decode_attention(batch: dkv_attn_batch, pool: DevicePool, tables, stream=None) -> None:
    pc, tc = pool.c(), tables.c()
    rc = load().dkv_decode_attention(ctypes.byref(batch), ctypes.byref(pc), ctypes.byref(tc), _stream(stream))
    if rc != DKV_OK:
        raise DkvError(rc, "dkv_decode_attention")


def dkv_prefill_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, lens: torch.Tensor, max_len: int,
                          scale: float, out: torch.Tensor, sig_sum: torch.Tensor, sig_cnt: torch.Tensor,
                          pool: DevicePool, stream=None) -> None:
    """dkv_prefill_attention: q [L][T][Hq][128], k / v [L][T][Hkv][128] bf16;
    out fp32 [L][T][Hq][128], sig_sum fp32 [L][T][Hq], sig_cnt int32 [T]."""
    L, T, Hq = int(q.shape[0]), int(q.shape[1]), int(q.shape[2])
    b = dkv_prefill_batch(L, int(lens.numel()), Hq, int(k.shape[2]), int(max_len), 0, T, _p(q), _p(k), _p(v),
                          _p(lens), float(scale), _p(out), _p(sig_sum), _p(sig_cnt))
    pc = pool.c()
    rc = load().dkv_prefill_attention(ctypes.byref(b), ctypes.byref(pc), _stream(stream))
    if rc != DKV_OK:
        raise DkvError(rc, "dkv_prefill_attention")


class _TableView:
    """Tables of a contiguous run of units (pointer offsets into DeviceTables)."""

    def __init__(self, t: DeviceTables, u0: int):
        self.t, self.u0 = t, int(u0)

    def c(self) -> dkv_tables:
        return dkv_tables(_p(self.t.fwd) + 4 * self.u0 * self.t.pmax, self.t.pmax, 0,
                          _p(self.t.unit_hdr) + 16 * self.u0)


class Decoder:
    """Device state of a generation workload: pool, unit tables (pmax =
    ceil(cap / P) + 1), capacity-strided classes and slot index, workspace.
    prefill_layer() fills one layer's units with dkv_compact; index() derives
    classes and slot_of from the pages; step() runs dkv_decode_step."""

    def __init__(self, L: int, R: int, Hq: int, Hkv: int, cap: int, P: int, F: int, device="cuda",
                 window: int = 0, mode: int = 0, scheme: int = 0):
        self.L, self.R, self.Hq, self.Hkv, self.cap, self.P = L, R, Hq, Hkv, cap, P
        self.window, self.mode = int(window), int(mode)
        self.U = L * R * Hkv
        self.pmax = -(-cap // P) + 1
        self.device = torch.device(device)
        self.pool = DevicePool(F, P, device, scheme=scheme)
        self.tables = DeviceTables(self.U, self.pmax, device)
        rows = L * R * cap * Hkv
        self.classes = torch.zeros(rows, dtype=torch.uint8, device=device)
        self.slot_of = torch.full((rows,), -1, dtype=torch.int32, device=device)
        self.workspace = torch.empty(dkv_decode_workspace_size(self.batch({})), dtype=torch.uint8, device=device)
        dkv_init_pool(self.pool)
        self._pre_ws = None

    def batch(self, d: dict) -> dkv_decode_batch:
        g = d.get
        return dkv_decode_batch(self.L, self.R, self.Hq, self.Hkv, 128, self.cap, 0, _p(g("k_new")), _p(g("v_new")),
                                _p(g("sig_sum")), _p(g("sig_cnt")), _p(g("ctx_lens")), _p(g("new_lens")),
                                _p(self.classes), _p(self.slot_of), self.window, self.mode)

    def prefill_layer(self, inp: dict, layer: int, max_len: int, alpha_h: float, alpha_l: float,
                      stream=None) -> None:
        """dkv_compact of one layer's prefill inputs (L = 1) into this pool,
        units of layer `layer` (unit_base and table rows offset)."""
        T = int(inp["T"])
        cls = torch.empty(max(T * self.Hkv, 1), dtype=torch.uint8, device=self.device)
        b = make_batch(inp, cls, max_len, unit_base=layer * self.R * self.Hkv)
        need = dkv_workspace_size(b)
        if self._pre_ws is None or self._pre_ws.numel() < need:
            self._pre_ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        dkv_compact(b, alpha_h, alpha_l, self.pool, _TableView(self.tables, layer * self.R * self.Hkv),
                    self._pre_ws, stream=stream)

    def index(self, ctx_lens: torch.Tensor, stream=None) -> None:
        dkv_decode_index(self.batch({"ctx_lens": ctx_lens}), self.pool, self.tables, stream=stream)

    def step(self, d: dict, alpha_h: float, alpha_l: float, stream=None, spin_limit: int = -1,
             profiler=None) -> None:
        dkv_decode_step(self.batch(d), alpha_h, alpha_l, self.pool, self.tables, self.workspace, stream=stream,
                        spin_limit=spin_limit, profiler=profiler)

    def attend(self, q: torch.Tensor, ctx_lens: torch.Tensor, out: torch.Tensor, scale: float, layer0: int = 0,
               k_new: torch.Tensor | None = None, v_new: torch.Tensor | None = None,
               new_lens: torch.Tensor | None = None, sig_sum: torch.Tensor | None = None, stream=None) -> None:
        """dkv_decode_attention over layers [layer0, layer0 + q.shape[0])."""
        b = dkv_attn_batch(self.L, self.R, self.Hq, self.Hkv, self.cap, int(layer0), int(q.shape[0]), _p(q),
                           _p(k_new), _p(v_new), _p(new_lens), _p(ctx_lens), float(scale), _p(out), _p(sig_sum))
        dkv_decode_attention(b, self.pool, self.tables, stream=stream)
