"""Set-up of a generation (decode) workload on the device: per-layer prefill
through dkv_compact into a Decoder's pool, the capacity-strided significance
sums and counts the steps start from, and dkv_decode_index.  Plumbing for the
benchmark and the tests; every step of the path runs in libdkv."""
from __future__ import annotations

import torch

from . import libdkv
from . import workloads as W

DECODE_SLACK = 1 << 16   # free pages between the head after prefill and the next wrap of the ring


def decode_cap(w, steps: int) -> int:
    return -(-(max(w.lens) + steps) // 16) * 16


def decode_prefill(w, dec, dev, seed: int, cap: int, head_offset: int = 0):
    """Per-layer prefill of the decode workload into dec's pool (dkv_compact,
    one layer per call) and the capacity-strided significance sums and
    counts the steps start from.  head_offset rotates the fresh ring (free
    list slot i holds page i, cursors {head_offset, head_offset + F})."""
    libdkv.dkv_init_pool(dec.pool)
    if head_offset:
        dec.pool.cursors.copy_(torch.tensor([head_offset, head_offset + dec.pool.F], dtype=torch.int64))
    req, pos = W._positions(w, dev)
    dst = req * cap + pos
    sig = torch.zeros((w.L, w.R * cap, w.Hq), dtype=torch.float32, device=dev)
    cnt = torch.zeros(w.R * cap, dtype=torch.int32, device=dev)
    cnt0 = W.sig_cnt_prefill(w, dev)
    cnt[dst] = cnt0
    lens = torch.tensor(w.lens, dtype=torch.int32, device=dev)
    for l in range(w.L):
        k = W.make_kv_layer(w, seed, l, 0, dev)[None]
        v = W.make_kv_layer(w, seed, l, 1, dev)[None]
        s = W.make_sig_layer(w, seed, l, dev)
        sig[l, dst] = s
        layer = {"L": 1, "R": w.R, "Hq": w.Hq, "Hkv": w.Hkv, "T": w.T, "k": k, "v": v, "sig_sum": s[None].contiguous(),
                 "sig_cnt": cnt0, "lens": lens}
        dec.prefill_layer(layer, l, max(w.lens), w.alpha_h, w.alpha_l)
        del k, v, s, layer
    st = libdkv.dkv_get_status(dec.pool)
    assert st == libdkv.DKV_OK, libdkv.status_string(st)
    ctx = {"L": w.L, "R": w.R, "Hq": w.Hq, "Hkv": w.Hkv, "cap": cap, "sig_sum": sig, "sig_cnt": cnt,
           "ctx_lens": lens.clone()}
    dec.index(ctx["ctx_lens"])
    st = libdkv.dkv_get_status(dec.pool)
    assert st == libdkv.DKV_OK, libdkv.status_string(st)
    return ctx


def decode_setup(w, dev, seed: int, total_steps: int, window: int = 0, mode: int = 0):
    """Decoder state after the prefill, with the pool sized so that the ring's
    head wraps within the run: a first prefill in a worst-case pool measures
    the pages it takes, the second starts the ring DECODE_SLACK pages before
    its end."""
    cap = decode_cap(w, total_steps)
    dec = libdkv.Decoder(w.L, w.R, w.Hq, w.Hkv, cap, w.P, w.pool_pages, device=dev, window=window, mode=mode,
                         scheme=w.scheme)
    decode_prefill(w, dec, dev, seed, cap)
    used = int(dec.pool.cursors[0])
    F = dec.pool.F
    offset = (F - used - DECODE_SLACK) % F
    torch.cuda.empty_cache()
    ctx = decode_prefill(w, dec, dev, seed, cap, head_offset=offset)
    return dec, ctx, cap, used
