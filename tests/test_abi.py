"""CPU-side checks of the C ABI: the library builds, loads, exports every
symbol include/dkv.h declares, and rejects invalid arguments synchronously
(validation paths only: no kernel is launched)."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

from differentiated_kv_cache_dkv_gb300 import build as libbuild
from differentiated_kv_cache_dkv_gb300 import libdkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dkv.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return libdkv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dkv_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("dkv_init_pool", "dkv_compact", "dkv_dequant_page", "dkv_get_status", "dkv_workspace_size"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", libdkv.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\sT\s+(dkv_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in declared_functions():
        assert getattr(lib, n) is not None


def test_version_and_status_strings(lib):
    assert lib.dkv_version() >= 100
    for code in range(-7, 1):
        assert libdkv.status_string(code)


def _batch(**kw):
    b = dict(L=2, R=3, Hq=8, Hkv=2, D=128, max_len=100, T=250, unit_base=0, k=256, v=512, sig_sum=1024,
             sig_cnt=2048, lens=4096, classes=8192)
    b.update(kw)
    return libdkv.dkv_batch(**b)


def test_workspace_size_validation(lib):
    assert libdkv.dkv_workspace_size(_batch()) > 0
    for bad in (dict(D=64), dict(Hq=7), dict(L=0), dict(T=-1), dict(Hq=256, Hkv=2)):
        with pytest.raises(libdkv.DkvError) as e:
            libdkv.dkv_workspace_size(_batch(**bad))
        assert e.value.code == libdkv.DKV_E_INVAL


def _pool(**kw):
    p = dict(F=64, P=16, reserved=0, free_list=256, cursors=512, rev_unit=1024, rev_idx=2048, page_cls=4096,
             pages=8192, status=16384)
    p.update(kw)
    return libdkv.dkv_pool(**p)


def test_compact_rejects_bad_arguments_without_launching(lib):
    t = libdkv.dkv_tables(256, 16, 0, 512)
    params = libdkv.dkv_params(1.0, 0.2, -1, 0, None)
    ws = 1 << 20

    def call(b=None, p=None, pool=None, tab=None, wsp=ws, wsb=1 << 30):
        return lib.dkv_compact(ctypes.byref(b or _batch()), ctypes.byref(p or params),
                               ctypes.byref(pool or _pool()), ctypes.byref(tab or t), wsp, wsb, None)

    cases = [
        dict(b=_batch(D=96)),
        dict(b=_batch(k=257)),                                    # misaligned K
        dict(p=libdkv.dkv_params(0.1, 0.2, -1, 0, None)),         # alpha_l > alpha_h
        dict(p=libdkv.dkv_params(float("nan"), 0.2, -1, 0, None)),
        dict(pool=_pool(P=15)),                                   # odd page size
        dict(pool=_pool(F=0)),
        dict(tab=libdkv.dkv_tables(256, 3, 0, 512)),              # pmax < ceil(100/16)+1
        dict(wsp=ws + 8),                                         # misaligned workspace
        dict(wsb=16),                                             # workspace too small
    ]
    for c in cases:
        assert call(**c) == libdkv.DKV_E_INVAL, c
    assert lib.dkv_dequant_page(ctypes.byref(_pool()), 64, 256, 256, 256, None) == libdkv.DKV_E_INVAL
    assert lib.dkv_init_pool(ctypes.byref(_pool(pages=8193)), None) == libdkv.DKV_E_INVAL


def _dbatch(**kw):
    b = dict(L=2, R=3, Hq=8, Hkv=2, D=128, cap=64, unit_base=0, k_new=256, v_new=512, sig_sum=1024,
             sig_cnt=2048, ctx_lens=4096, new_lens=8192, classes=16384, slot_of=32768)
    b.update(kw)
    return libdkv.dkv_decode_batch(**b)


def test_decode_rejects_bad_arguments_without_launching(lib):
    assert libdkv.dkv_decode_workspace_size(_dbatch()) > 0
    for bad in (dict(cap=60), dict(cap=0), dict(D=64), dict(Hq=7), dict(R=0)):
        with pytest.raises(libdkv.DkvError):
            libdkv.dkv_decode_workspace_size(_dbatch(**bad))
    t = libdkv.dkv_tables(256, 6, 0, 512)
    params = libdkv.dkv_params(1.0, 0.2, -1, 0, None)

    def call(b=None, p=None, pool=None, tab=None, wsp=1 << 20, wsb=1 << 30):
        return lib.dkv_decode_step(ctypes.byref(b or _dbatch()), ctypes.byref(p or params),
                                   ctypes.byref(pool or _pool()), ctypes.byref(tab or t), wsp, wsb, None)

    cases = [
        dict(b=_dbatch(cap=40)),                                  # not a multiple of 16
        dict(b=_dbatch(classes=16385)),                           # misaligned classes
        dict(b=_dbatch(slot_of=None)),
        dict(b=_dbatch(sig_sum=1028)),                            # misaligned sig_sum
        dict(p=libdkv.dkv_params(0.1, 0.2, -1, 0, None)),
        dict(pool=_pool(P=7)),
        dict(tab=libdkv.dkv_tables(256, 1, 0, 512)),
        dict(wsp=(1 << 20) + 8),
        dict(wsb=64),
        dict(b=_dbatch(window=-1)),                               # negative recent window
        dict(b=_dbatch(mode=2)),                                  # no such decode mode
    ]
    for c in cases:
        assert call(**c) == libdkv.DKV_E_INVAL, c
    assert lib.dkv_decode_index(ctypes.byref(_dbatch(ctx_lens=None)), ctypes.byref(_pool()), ctypes.byref(t),
                                None) == libdkv.DKV_E_INVAL


def _abatch(**kw):
    b = dict(L=2, R=3, Hq=8, Hkv=2, cap=64, layer0=0, n_layers=2, q=256, k_new=None, v_new=None, new_lens=None,
             ctx_lens=4096, scale=0.088, out=8192, sig_sum=None)
    b.update(kw)
    return libdkv.dkv_attn_batch(**b)


def test_attention_rejects_bad_arguments_without_launching(lib):
    t = libdkv.dkv_tables(256, 6, 0, 512)
    cases = [
        _abatch(Hq=7),                                  # Hq not a multiple of Hkv
        _abatch(Hq=32),                                 # G = 16 > 8
        _abatch(layer0=1),                              # layers past L
        _abatch(n_layers=-1),
        _abatch(q=None), _abatch(q=264),                # missing / misaligned query
        _abatch(out=None), _abatch(ctx_lens=None),
        _abatch(k_new=256),                             # K without V
        _abatch(k_new=256, v_new=512),                  # new token without new_lens
        _abatch(k_new=264, v_new=512, new_lens=1024),   # misaligned new K
        _abatch(sig_sum=1030),                          # misaligned significance sums
        _abatch(scale=float("inf")),
        _abatch(cap=0),
        _abatch(cap=1 << 22),                           # a unit's logits do not fit one cluster
    ]
    for c in cases:
        rc = lib.dkv_decode_attention(ctypes.byref(c), ctypes.byref(_pool()), ctypes.byref(t), None)
        assert rc == libdkv.DKV_E_INVAL, c
    bad_tab = libdkv.dkv_tables(256, 6, 0, 520)         # unit headers not 16-byte aligned
    assert lib.dkv_decode_attention(ctypes.byref(_abatch()), ctypes.byref(_pool()), ctypes.byref(bad_tab),
                                    None) == libdkv.DKV_E_INVAL


def _pbatch(**kw):
    b = dict(L=2, R=3, Hq=8, Hkv=2, max_len=100, reserved=0, T=250, q=256, k=512, v=768, lens=1024, scale=0.088,
             out=2048, sig_sum=4096, sig_cnt=8192)
    b.update(kw)
    return libdkv.dkv_prefill_batch(**b)


def test_prefill_attention_rejects_bad_arguments_without_launching(lib):
    cases = [
        _pbatch(Hq=7),                      # Hq not a multiple of Hkv
        _pbatch(L=0), _pbatch(T=-1), _pbatch(max_len=-1), _pbatch(reserved=1),
        _pbatch(q=None), _pbatch(q=264),    # missing / misaligned query
        _pbatch(k=520), _pbatch(v=None),
        _pbatch(lens=None), _pbatch(out=2052), _pbatch(sig_sum=None), _pbatch(sig_cnt=8194),
        _pbatch(scale=float("nan")),
        _pbatch(R=70000),                   # more requests than a grid dimension holds
    ]
    for c in cases:
        rc = lib.dkv_prefill_attention(ctypes.byref(c), ctypes.byref(_pool()), None)
        assert rc == libdkv.DKV_E_INVAL, c
    assert lib.dkv_prefill_attention(ctypes.byref(_pbatch()), None, None) == libdkv.DKV_E_INVAL
