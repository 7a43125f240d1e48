"""Test-side helpers: run the oracle on a workload and parse unified pages.

The page parser is written from the page layout the oracle documents (216*P
bytes: K codes, V codes, fp16 metadata, int32 positions) and is used to check
both the oracle's pages and the GPU's pages; it performs no quantisation.
"""
from __future__ import annotations

import numpy as np

import oracle
from differentiated_kv_cache_dkv_gb300 import workloads as W


# (kh, vh) of the high class per precision scheme; the low class has half of
# each (the documented reading: K8V4/K4V2, K8V2/K4V1, K4V8/K2V4).
SCHEME_BITS = {0: (8, 4), 1: (8, 2), 2: (4, 8)}


class Layout:
    """Byte offsets of the unified page of a scheme, from its documented
    formula: K codes [0, 16 kh P), V codes [16 kh P, 16 (kh + vh) P), fp16
    metadata 8 bytes per slot, int32 position per slot."""

    def __init__(self, P: int, scheme: int = 0):
        self.P, self.scheme = int(P), int(scheme)
        self.kh, self.vh = SCHEME_BITS[self.scheme]
        self.codes = 16 * (self.kh + self.vh) * self.P
        self.meta = self.codes
        self.pos = self.codes + 16 * self.P
        self.bytes = self.codes + 24 * self.P

    def kbits(self, high: bool) -> int:
        return self.kh if high else self.kh // 2

    def vbits(self, high: bool) -> int:
        return self.vh if high else self.vh // 2

    def k_off(self, high: bool, s: int) -> int:
        return s * 16 * self.kbits(high)

    def v_off(self, high: bool, s: int) -> int:
        return 16 * self.kh * self.P + s * 16 * self.vbits(high)


def run_oracle(w: W.Workload, inp_np: dict, alpha_h=None, alpha_l=None, pool=None, quant_mask=None):
    ah = w.alpha_h if alpha_h is None else alpha_h
    al = w.alpha_l if alpha_l is None else alpha_l
    L = int(inp_np["L"])
    if pool is None:
        pool = oracle.Pool(w.pool_pages, w.P, scheme=w.scheme)
    tab = oracle.Tables(L * w.R * w.Hkv, w.pmax, L * w.T * w.Hkv)
    st = oracle.compact(inp_np, ah, al, pool, tab, quant_mask)
    return st, pool, tab


def page_slots(page: np.ndarray, P: int, cls: int, scheme: int = 0):
    """Parse one page into per-slot (k_codes[128], v_codes[128], meta[4] u16,
    pos) for every slot the page class provides."""
    lay = Layout(P, scheme)
    high = cls == 2
    nslots = P if high else 2 * P
    kb, vb = lay.kbits(high), lay.vbits(high)
    out = []
    for s in range(nslots):
        k_bytes = page[lay.k_off(high, s):lay.k_off(high, s) + 16 * kb]
        v_bytes = page[lay.v_off(high, s):lay.v_off(high, s) + 16 * vb]
        meta = page[lay.meta + 8 * s:lay.meta + 8 * s + 8].view(np.uint16)
        pos = int(page[lay.pos + 4 * s:lay.pos + 4 * s + 4].view(np.int32)[0])
        out.append((unpack(k_bytes, kb), unpack(v_bytes, vb), meta.copy(), pos))
    return out


def unpack(b: np.ndarray, bits: int) -> np.ndarray:
    per = 8 // bits
    mask = (1 << bits) - 1
    b = b.astype(np.uint16)
    cols = [(b >> (e * bits)) & mask for e in range(per)]
    return np.stack(cols, axis=1).reshape(-1).astype(np.uint8)


def f16(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def unit_rows(w: W.Workload, L: int, u: int):
    """(layer, request, head, first token index, length) of unit u."""
    h = u % w.Hkv
    r = (u // w.Hkv) % w.R
    l = u // (w.Hkv * w.R)
    start = int(sum(w.lens[:r]))
    return l, r, h, start, w.lens[r]
