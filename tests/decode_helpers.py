"""Test-side helpers for the generation (decode) step: unit list parsing from
raw page bytes and the state invariants every step must keep (the oracle-side
decode state, HostDecode, lives in oracle/host_decode.py).  No quantisation
happens here."""
from __future__ import annotations

import numpy as np

from differentiated_kv_cache_dkv_gb300 import workloads as W
from oracle.host_decode import HostDecode, decode_pmax  # noqa: F401  (re-exported for the tests)
from tests.oracle_helpers import Layout, unpack


def list_slots(pages: np.ndarray, fwd_row: np.ndarray, hdr, P: int, scheme: int = 0):
    """Raw bytes of a unit's two lists: for list 0 (high class) and 1 (low
    class), a list of (K bytes, V bytes, metadata bytes, position) per slot,
    over every slot of the list's pages (used slots first)."""
    lay = Layout(P, scheme)
    n_hi, n_lo, p_hi, p_lo = (int(x) for x in hdr)
    out = []
    for high, ids, per in ((True, fwd_row[:p_hi], P), (False, fwd_row[p_hi:p_hi + p_lo], 2 * P)):
        kb, vb = 16 * lay.kbits(high), 16 * lay.vbits(high)
        slots = []
        for pid in ids:
            pg = pages[int(pid)]
            for s in range(per):
                k = pg[lay.k_off(high, s):lay.k_off(high, s) + kb]
                v = pg[lay.v_off(high, s):lay.v_off(high, s) + vb]
                meta = pg[lay.meta + 8 * s:lay.meta + 8 * s + 8]
                pos = int(pg[lay.pos + 4 * s:lay.pos + 4 * s + 4].view(np.int32)[0])
                slots.append((bytes(k), bytes(v), bytes(meta), pos))
        out.append(slots)
    return out


def check_state(w: W.Workload, cap: int, pool, fwd: np.ndarray, unit_hdr: np.ndarray, classes: np.ndarray,
                ctx_lens: np.ndarray, unit_base: int = 0, layers=None, check_ring: bool = True):
    """Invariants of a decode state (raises AssertionError):
    - every unit's header counts equal its K8V4 / K4V2 tokens in `classes`, its
      page counts are ceil(n / capacity), its forward row lists those pages
      then -1, and rev_unit / rev_idx / page_cls point back at it;
    - the used slots of each list hold exactly the positions of that class,
      each once, and every unused slot is clear (zero codes and metadata,
      position -1), slots P..2P-1 of K8V4 pages included;
    - the free ring [head, tail) and the owned pages partition the pool.
    Returns {(unit, position): (list, slot bytes)} for the checked layers."""
    P, F = pool.P, pool.F
    lay = Layout(P, getattr(pool, "scheme", 0))
    Ul = w.R * w.Hkv
    layers = range(w.L) if layers is None else layers
    owned = []
    where = {}
    for l in layers:
        for r in range(w.R):
            c = int(ctx_lens[r])
            for h in range(w.Hkv):
                u = l * Ul + r * w.Hkv + h
                n_hi, n_lo, p_hi, p_lo = (int(x) for x in unit_hdr[u])
                col = classes[l, r * cap:r * cap + c, h]
                assert n_hi == int((col == 2).sum()) and n_lo == int((col == 1).sum()), (u, n_hi, n_lo)
                assert p_hi == -(-n_hi // P) and p_lo == -(-n_lo // (2 * P)), u
                row = fwd[u]
                ids = row[:p_hi + p_lo]
                assert np.all(ids >= 0) and np.all(row[p_hi + p_lo:] == -1), u
                for k, pid in enumerate(ids):
                    assert pool.rev_unit[pid] == unit_base + u and pool.rev_idx[pid] == k, (u, k, pid)
                    assert pool.page_cls[pid] == (2 if k < p_hi else 1), (u, k)
                    if k < p_hi:
                        pg = pool.pages[pid]
                        assert not pg[lay.meta + 8 * P:lay.pos].any()
                        assert np.all(pg[lay.pos + 4 * P:lay.bytes].view(np.int32) == -1)
                owned.extend(int(x) for x in ids)
                lists = list_slots(pool.pages, row, unit_hdr[u], P, lay.scheme)
                for li, (n, cls) in enumerate(((n_hi, 2), (n_lo, 1))):
                    slots = lists[li]
                    got = [s[3] for s in slots[:n]]
                    want = np.nonzero(col == cls)[0]
                    assert sorted(got) == list(want), (u, li)
                    for s in slots[n:]:
                        assert s[3] == -1 and not any(s[0]) and not any(s[1]) and not any(s[2]), (u, li)
                    for si, s in enumerate(slots[:n]):
                        where[(u, s[3])] = (li, s[:3], si)
    if check_ring:
        head, tail = int(pool.cursors[0]), int(pool.cursors[1])
        assert 0 <= tail - head <= F
        ring = [int(pool.free_list[x % F]) for x in range(head, tail)]
        assert all(pool.page_cls[p] == 0 and pool.rev_unit[p] == -1 for p in ring)
        if len(list(layers)) == w.L:
            assert sorted(ring + owned) == list(range(F))
    return where


def slot_codes(slot_bytes, high: bool, scheme: int = 0):
    """Unpacked (K codes, V codes, fp16 metadata) of a slot's raw bytes."""
    k, v, meta = slot_bytes
    lay = Layout(2, scheme)
    kb, vb = lay.kbits(high), lay.vbits(high)
    return (unpack(np.frombuffer(k, np.uint8), kb), unpack(np.frombuffer(v, np.uint8), vb),
            np.frombuffer(meta, np.uint16))
