"""CPU oracle for DiffKV-style differentiated KV-cache compaction.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg are the only callers.  The CUDA
library never imports this package and shares no code with it.

This module is a ctypes binding over ``dkv_oracle.cpp`` (a plain,
single-threaded C++ restatement of the method; every reading of the source page
is listed in that file's header) plus numpy-side page parsers used by the
tests.  Building the oracle is ``oracle.build.build_oracle()``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB_PATH, LIB_PATH_SAN, build_oracle

OK = 0
E_INVAL = -1
E_NOMEM = -2
E_RANGE = -3
E_LENS = -7
E_INTERNAL = -5

_lib = None


class _Batch(ctypes.Structure):
    _fields_ = [
        ("L", ctypes.c_int32), ("R", ctypes.c_int32), ("Hq", ctypes.c_int32),
        ("Hkv", ctypes.c_int32), ("D", ctypes.c_int32), ("T", ctypes.c_int64),
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("sig_sum", ctypes.c_void_p),
        ("sig_cnt", ctypes.c_void_p), ("lens", ctypes.c_void_p), ("unit_base", ctypes.c_int64),
    ]


class _Pool(ctypes.Structure):
    _fields_ = [
        ("F", ctypes.c_int64), ("P", ctypes.c_int32), ("scheme", ctypes.c_int32), ("free_list", ctypes.c_void_p),
        ("cursors", ctypes.c_void_p), ("rev_unit", ctypes.c_void_p),
        ("rev_idx", ctypes.c_void_p), ("page_cls", ctypes.c_void_p), ("pages", ctypes.c_void_p),
    ]


class _Tables(ctypes.Structure):
    _fields_ = [
        ("fwd", ctypes.c_void_p), ("pmax", ctypes.c_int32), ("unit_hdr", ctypes.c_void_p),
        ("classes", ctypes.c_void_p),
    ]


class _DecodeBatch(ctypes.Structure):
    _fields_ = [
        ("L", ctypes.c_int32), ("R", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("D", ctypes.c_int32), ("cap", ctypes.c_int32), ("unit_base", ctypes.c_int64),
        ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p), ("sig_sum", ctypes.c_void_p),
        ("sig_cnt", ctypes.c_void_p), ("ctx_lens", ctypes.c_void_p), ("new_lens", ctypes.c_void_p),
        ("classes", ctypes.c_void_p), ("window", ctypes.c_int32), ("mode", ctypes.c_int32),
    ]


class _AttnBatch(ctypes.Structure):
    _fields_ = [
        ("L", ctypes.c_int32), ("R", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("cap", ctypes.c_int32), ("layer0", ctypes.c_int32), ("n_layers", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
        ("new_lens", ctypes.c_void_p), ("ctx_lens", ctypes.c_void_p), ("scale", ctypes.c_double),
        ("out", ctypes.c_void_p), ("p_out", ctypes.c_void_p),
    ]


class _PrefillBatch(ctypes.Structure):
    _fields_ = [
        ("L", ctypes.c_int32), ("R", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("T", ctypes.c_int64), ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("lens", ctypes.c_void_p), ("scale", ctypes.c_double), ("out", ctypes.c_void_p),
        ("sig_sum", ctypes.c_void_p), ("sig_cnt", ctypes.c_void_p),
    ]


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        sanitized = os.environ.get("ORACLE_LIBRARY") == "sanitized"
        path = LIB_PATH_SAN if sanitized else LIB_PATH
        if not os.path.exists(path):
            build_oracle(sanitize=sanitized)
        L = ctypes.CDLL(path)
        L.oracle_fp16_rn.argtypes = [ctypes.c_float]
        L.oracle_fp16_rn.restype = ctypes.c_uint16
        L.oracle_fp16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_fp16_to_f32.restype = ctypes.c_float
        L.oracle_fp16_rn_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        L.oracle_fp16_rn_array.restype = None
        L.oracle_quant_row.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_quant_row.restype = ctypes.c_int32
        L.oracle_init_pool.argtypes = [ctypes.POINTER(_Pool)]
        L.oracle_init_pool.restype = None
        L.oracle_compact.argtypes = [ctypes.POINTER(_Batch), ctypes.c_float, ctypes.c_float,
                                     ctypes.POINTER(_Pool), ctypes.POINTER(_Tables),
                                     ctypes.c_void_p]
        L.oracle_compact.restype = ctypes.c_int32
        L.oracle_decode_step.argtypes = [ctypes.POINTER(_DecodeBatch), ctypes.c_float, ctypes.c_float,
                                         ctypes.POINTER(_Pool), ctypes.POINTER(_Tables)]
        L.oracle_decode_step.restype = ctypes.c_int32
        L.oracle_decode_attention.argtypes = [ctypes.POINTER(_AttnBatch), ctypes.POINTER(_Pool),
                                              ctypes.POINTER(_Tables)]
        L.oracle_decode_attention.restype = ctypes.c_int32
        L.oracle_prefill_attention.argtypes = [ctypes.POINTER(_PrefillBatch)]
        L.oracle_prefill_attention.restype = ctypes.c_int32
        L.oracle_dequant_page.argtypes = [ctypes.POINTER(_Pool), ctypes.c_int32, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_dequant_page.restype = None
        _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def fp16_rn(x: np.ndarray) -> np.ndarray:
    """fp32 -> fp16 bit patterns via the oracle's own IEEE conversion."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_fp16_rn_array(_ptr(x), _ptr(out), x.size)
    return out


def fp16_to_f32(h: int) -> float:
    return float(lib().oracle_fp16_to_f32(int(h)))


def quant_row(x_bf16_bits: np.ndarray, bits: int):
    """Quantise one 128-element bf16 row; returns (status, codes, s16, z16)."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    assert x.size == 128
    q = np.zeros(128, dtype=np.uint8)
    s16 = ctypes.c_uint16(0)
    z16 = ctypes.c_uint16(0)
    st = lib().oracle_quant_row(_ptr(x), bits, _ptr(q), ctypes.byref(s16), ctypes.byref(z16))
    return st, q, s16.value, z16.value


# Precision schemes (reading F of dkv_oracle.cpp): (kh, vh) of the high
# class; the low class has half of each.
SCHEMES = {0: (8, 4), 1: (8, 2), 2: (4, 8)}


def page_bytes(P: int, scheme: int = 0) -> int:
    kh, vh = SCHEMES[scheme]
    return (16 * (kh + vh) + 24) * int(P)


class Pool:
    """Host-side pool state for the oracle (numpy arrays)."""

    def __init__(self, F: int, P: int, allocate_pages: bool = True, scheme: int = 0):
        self.F, self.P, self.scheme = int(F), int(P), int(scheme)
        self.free_list = np.zeros(F, dtype=np.int32)
        self.cursors = np.zeros(2, dtype=np.uint64)
        self.rev_unit = np.zeros(F, dtype=np.int32)
        self.rev_idx = np.zeros(F, dtype=np.int32)
        self.page_cls = np.zeros(F, dtype=np.uint8)
        # np.zeros is calloc-backed: untouched pages cost no memory.
        self.pages = np.zeros((F, page_bytes(P, scheme)), dtype=np.uint8)
        self.init()

    def _c(self):
        return _Pool(self.F, self.P, self.scheme, _ptr(self.free_list), _ptr(self.cursors), _ptr(self.rev_unit),
                     _ptr(self.rev_idx), _ptr(self.page_cls), _ptr(self.pages))

    def init(self):
        p = self._c()
        lib().oracle_init_pool(ctypes.byref(p))


class Tables:
    def __init__(self, U: int, pmax: int, rows: int):
        self.pmax = int(pmax)
        self.fwd = np.full((U, pmax), -7, dtype=np.int32)
        self.unit_hdr = np.zeros((U, 4), dtype=np.int32)
        self.classes = np.full(rows, 0xEE, dtype=np.uint8)

    def _c(self):
        return _Tables(_ptr(self.fwd), self.pmax, _ptr(self.unit_hdr), _ptr(self.classes))


def compact(inp: dict, alpha_h: float, alpha_l: float, pool: Pool, tables: Tables,
            quant_mask: np.ndarray | None = None) -> int:
    """Run the oracle's prefill compaction.

    ``inp`` holds numpy arrays: k, v (uint16 bf16 bits [L][T][Hkv][128]),
    sig_sum (float32 [L][T][Hq]), sig_cnt (int32 [T]), lens (int32 [R]), the
    ints L, R, Hq, Hkv, T and optionally unit_base (global id of the first
    unit, for layer-at-a-time calls).
    """
    k = np.ascontiguousarray(inp["k"])
    v = np.ascontiguousarray(inp["v"])
    sig = np.ascontiguousarray(inp["sig_sum"], dtype=np.float32)
    cnt = np.ascontiguousarray(inp["sig_cnt"], dtype=np.int32)
    lens = np.ascontiguousarray(inp["lens"], dtype=np.int32)
    b = _Batch(int(inp["L"]), int(inp["R"]), int(inp["Hq"]), int(inp["Hkv"]), 128, int(inp["T"]),
               _ptr(k), _ptr(v), _ptr(sig), _ptr(cnt), _ptr(lens), int(inp.get("unit_base", 0)))
    p = pool._c()
    t = tables._c()
    mask = None if quant_mask is None else np.ascontiguousarray(quant_mask, dtype=np.uint8)
    return int(lib().oracle_compact(ctypes.byref(b), float(alpha_h), float(alpha_l),
                                     ctypes.byref(p), ctypes.byref(t), _ptr(mask)))


def decode_step(dinp: dict, alpha_h: float, alpha_l: float, pool: Pool, tables: Tables) -> int:
    """One generation step on the oracle's pool and tables (in place).

    ``dinp`` holds numpy arrays: k_new, v_new (uint16 bf16 bits [L][R][Hkv][128]),
    sig_sum (float32 [L][R*cap][Hq]), sig_cnt (int32 [R*cap]), ctx_lens, new_lens
    (int32 [R]), classes (uint8 [L][R*cap][Hkv], updated in place), and the ints
    L, R, Hq, Hkv, cap (and optionally unit_base, window and mode: the recent
    window W and the candidate policy, 0 = re-score all older tokens, 1 = only
    the token leaving the window).
    """
    arrs = {k: np.ascontiguousarray(dinp[k]) for k in ("k_new", "v_new", "sig_sum", "sig_cnt", "ctx_lens",
                                                        "new_lens")}
    cls = dinp["classes"]
    assert cls.flags["C_CONTIGUOUS"] and cls.dtype == np.uint8
    b = _DecodeBatch(int(dinp["L"]), int(dinp["R"]), int(dinp["Hq"]), int(dinp["Hkv"]), 128, int(dinp["cap"]),
                     int(dinp.get("unit_base", 0)), _ptr(arrs["k_new"]), _ptr(arrs["v_new"]),
                     _ptr(arrs["sig_sum"]), _ptr(arrs["sig_cnt"]), _ptr(arrs["ctx_lens"]), _ptr(arrs["new_lens"]),
                     _ptr(cls), int(dinp.get("window", 0)), int(dinp.get("mode", 0)))
    p = pool._c()
    t = tables._c()
    return int(lib().oracle_decode_step(ctypes.byref(b), float(alpha_h), float(alpha_l), ctypes.byref(p),
                                        ctypes.byref(t)))


def dequant_page(pool: Pool, page_id: int):
    P = pool.P
    k = np.zeros((2 * P, 128), dtype=np.float32)
    v = np.zeros((2 * P, 128), dtype=np.float32)
    pos = np.zeros(2 * P, dtype=np.int32)
    p = pool._c()
    lib().oracle_dequant_page(ctypes.byref(p), int(page_id), _ptr(k), _ptr(v), _ptr(pos))
    return k, v, pos


def decode_attention(a: dict, pool: Pool, tables: Tables, p_out: bool = True):
    """Decode attention (reading M).  a: L, R, Hq, Hkv, cap, layer0, n_layers,
    q (uint16 bf16 bits [n_layers, R, Hq, 128]), optional k_new / v_new
    (uint16 [n_layers, R, Hkv, 128]) with new_lens, ctx_lens, scale.
    Returns (status, out [n_layers, R, Hq, 128] float64, p [n_layers, R*cap, Hq]
    float64 or None)."""
    nl, R, Hq = int(a["n_layers"]), int(a["R"]), int(a["Hq"])
    q = np.ascontiguousarray(a["q"], dtype=np.uint16)
    kn = a.get("k_new")
    kn = None if kn is None else np.ascontiguousarray(kn, dtype=np.uint16)
    vn = a.get("v_new")
    vn = None if vn is None else np.ascontiguousarray(vn, dtype=np.uint16)
    nlens = a.get("new_lens")
    nlens = None if nlens is None else np.ascontiguousarray(nlens, dtype=np.int32)
    ctx = np.ascontiguousarray(a["ctx_lens"], dtype=np.int32)
    out = np.zeros((nl, R, Hq, 128), dtype=np.float64)
    p = np.zeros((nl, R * int(a["cap"]), Hq), dtype=np.float64) if p_out else None
    b = _AttnBatch(int(a["L"]), R, Hq, int(a["Hkv"]), int(a["cap"]), int(a["layer0"]), nl, _ptr(q), _ptr(kn),
                   _ptr(vn), _ptr(nlens), _ptr(ctx), float(a["scale"]), _ptr(out), _ptr(p))
    pp = pool._c()
    tt = tables._c()
    st = int(lib().oracle_decode_attention(ctypes.byref(b), ctypes.byref(pp), ctypes.byref(tt)))
    return st, out, p


def prefill_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, lens, scale: float):
    """Prefill attention with significance accumulation (reading S).  q, k, v:
    uint16 bf16 bits [L][T][Hq or Hkv][128].  Returns (status, out [L][T][Hq][128]
    float64, sig_sum [L][T][Hq] float64, sig_cnt [T] int32)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    L, T, Hq = q.shape[0], q.shape[1], q.shape[2]
    out = np.zeros((L, T, Hq, 128), dtype=np.float64)
    sig = np.zeros((L, T, Hq), dtype=np.float64)
    cnt = np.zeros(T, dtype=np.int32)
    b = _PrefillBatch(L, lens.size, Hq, k.shape[2], T, _ptr(q), _ptr(k), _ptr(v), _ptr(lens), float(scale),
                      _ptr(out), _ptr(sig), _ptr(cnt))
    st = int(lib().oracle_prefill_attention(ctypes.byref(b)))
    return st, out, sig, cnt
