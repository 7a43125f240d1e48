"""Test-side helpers: run the oracle on a workload and parse unified pages.

The page parser is written from the page layout the oracle documents (216*P
bytes: K codes, V codes, fp16 metadata, int32 positions) and is used to check
both the oracle's pages and the GPU's pages; it performs no quantisation.
"""
from __future__ import annotations

import numpy as np

import oracle
from differentiated_kv_cache_dkv_gb300 import workloads as W


def run_oracle(w: W.Workload, inp_np: dict, alpha_h=None, alpha_l=None, pool=None, quant_mask=None):
    ah = w.alpha_h if alpha_h is None else alpha_h
    al = w.alpha_l if alpha_l is None else alpha_l
    L = int(inp_np["L"])
    if pool is None:
        pool = oracle.Pool(w.pool_pages, w.P)
    tab = oracle.Tables(L * w.R * w.Hkv, w.pmax, L * w.T * w.Hkv)
    st = oracle.compact(inp_np, ah, al, pool, tab, quant_mask)
    return st, pool, tab


def page_slots(page: np.ndarray, P: int, cls: int):
    """Parse one page into per-slot (k_codes[128], v_codes[128], meta[4] u16,
    pos) for every slot the page class provides."""
    high = cls == 2
    nslots = P if high else 2 * P
    kb = 8 if high else 4
    vb = 4 if high else 2
    out = []
    for s in range(nslots):
        k_bytes = page[s * 16 * kb:(s + 1) * 16 * kb]
        v_base = 128 * P
        v_bytes = page[v_base + s * 16 * vb:v_base + (s + 1) * 16 * vb]
        meta = page[192 * P + 8 * s:192 * P + 8 * s + 8].view(np.uint16)
        pos = int(page[208 * P + 4 * s:208 * P + 4 * s + 4].view(np.int32)[0])
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
