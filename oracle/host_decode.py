"""Oracle-side state of a generation workload (TEST INFRASTRUCTURE ONLY:
used by the tests, the smoke entry point and the benchmark's CPU legs).

HostDecode holds the oracle's pool, unit tables and the capacity-strided
context (significance sums, counts, classes) after an oracle prefill of a
workload, and runs oracle generation steps on it.  Inputs come from the seeded
generators in differentiated_kv_cache_dkv_gb300.workloads; nothing here
computes any part of the method (that is dkv_oracle.cpp).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import workloads as W


def decode_pmax(cap: int, P: int) -> int:
    return -(-cap // P) + 1


class HostDecode:
    """Oracle-side decode state of a workload: pool, unit tables and the
    capacity-strided context (sig, counts, classes) after an oracle prefill."""

    def __init__(self, w: W.Workload, cap: int, F: int | None = None, seed: int | None = None, inp=None,
                 window: int = 0, mode: int = 0):
        self.w, self.cap = w, cap
        self.window, self.mode = window, mode
        self.pmax = decode_pmax(cap, w.P)
        inp = W.make_inputs(w, seed) if inp is None else inp
        self.pool = oracle.Pool(F or w.pool_pages, w.P, scheme=w.scheme)
        tab = oracle.Tables(w.U, self.pmax, w.rows)
        st = oracle.compact(W.to_numpy(inp), w.alpha_h, w.alpha_l, self.pool, tab)
        assert st == oracle.OK, st
        self.tab = tab
        self.ctx = W.decode_context(w, inp, cap)
        dst = self.ctx["dst"].numpy()
        self.classes = np.zeros((w.L, w.R * cap, w.Hkv), dtype=np.uint8)
        self.classes[:, dst] = tab.classes.reshape(w.L, w.T, w.Hkv)
        self.step_no = 0

    @property
    def ctx_lens(self) -> np.ndarray:
        return self.ctx["ctx_lens"].numpy()

    def dinp(self, upd: dict) -> dict:
        w = self.w
        return {"L": w.L, "R": w.R, "Hq": w.Hq, "Hkv": w.Hkv, "cap": self.cap,
                "k_new": upd["k_new"].contiguous().view(torch.int16).numpy().view(np.uint16),
                "v_new": upd["v_new"].contiguous().view(torch.int16).numpy().view(np.uint16),
                "sig_sum": self.ctx["sig_sum"].numpy(), "sig_cnt": self.ctx["sig_cnt"].numpy(),
                "ctx_lens": self.ctx["ctx_lens"].numpy(),
                "new_lens": upd["new_lens"].numpy().astype(np.int32), "classes": self.classes,
                "window": self.window, "mode": self.mode}

    def step(self, upd: dict | None = None, **kw) -> int:
        """Draw this step's update (unless given) and run the oracle step."""
        if upd is None:
            upd = W.decode_update_inputs(self.w, self.ctx, self.step_no, **kw)
        st = oracle.decode_step(self.dinp(upd), self.w.alpha_h, self.w.alpha_l, self.pool, self.tab)
        if st == oracle.OK:
            self.ctx["ctx_lens"] += upd["new_lens"]
            self.step_no += 1
        return st

    def snapshot(self) -> dict:
        p = self.pool
        return {"free_list": p.free_list.copy(), "cursors": p.cursors.copy(), "rev_unit": p.rev_unit.copy(),
                "rev_idx": p.rev_idx.copy(), "page_cls": p.page_cls.copy(), "pages": p.pages.copy(),
                "fwd": self.tab.fwd.copy(), "unit_hdr": self.tab.unit_hdr.copy(), "classes": self.classes.copy()}
