"""dkv_compact's second stream: the unused slot halves of new K8V4 pages are
cleared on a library-owned stream forked from the caller's and joined back
before the commit.  These tests check that the call still behaves as one
ordered operation on the caller's stream:
- two host threads compacting different batches on their own streams at the
  same time (the fork and join are enqueued under the library's lock);
- the call captured into a CUDA graph and replayed;
each compared bit for bit with the oracle (classes, tables, cursors, every
live page byte).

DiffKV, Pith review, "What carries the argument" (parallel compaction into
unified pages); the stream and graph behaviour is this library's own.
"""
from __future__ import annotations

import threading

import pytest
import torch

import oracle
from differentiated_kv_cache_dkv_gb300 import libdkv
from differentiated_kv_cache_dkv_gb300 import workloads as W
from tests.gpu_helpers import assert_same_state, fetch, make_compactor, oracle_state, to_device
from tests.oracle_helpers import run_oracle

pytestmark = pytest.mark.gpu

AH, AL = 1.0, 0.2


def _expected(w: W.Workload, inp: dict, comp: libdkv.Compactor) -> dict:
    pool = oracle.Pool(comp.pool.F, w.P, scheme=w.scheme)
    so, pool, tab = run_oracle(w, W.to_numpy(inp), AH, AL, pool=pool)
    assert so == oracle.OK
    return oracle_state(pool, tab)


def test_two_threads_two_streams_bit_exact():
    ws = [W.small("t0", lens=[300, 7, 517, 0, 129]), W.small("t1", L=3, Hq=8, Hkv=2, lens=[64, 700, 33, 256])]
    inps = [W.make_inputs(ws[0], seed=71), W.make_inputs(ws[1], seed=72)]
    comps = [make_compactor(w) for w in ws]
    exp = [_expected(w, i, c) for w, i, c in zip(ws, inps, comps)]
    dev = [to_device(i) for i in inps]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    errors = []
    start = threading.Barrier(2)

    def work(k: int) -> None:
        try:
            start.wait()
            for _ in range(6):  # each round resets the pool, so the last round's state is the expected one
                libdkv.dkv_init_pool(comps[k].pool, stream=streams[k])
                comps[k].compact(dev[k], AH, AL, stream=streams[k])
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for k in range(2):
        assert libdkv.dkv_get_status(comps[k].pool) == libdkv.DKV_OK
        assert_same_state(fetch(comps[k]), exp[k], what=f"thread {k}")


def test_graph_capture_and_replay_bit_exact():
    w = W.small("graph", L=2, Hq=8, Hkv=2, lens=[300, 7, 517, 0, 129, 128])
    inp = W.make_inputs(w, seed=73)
    comp = make_compactor(w)
    exp = _expected(w, inp, comp)
    dev = to_device(inp)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # an ordinary call first: the library's stream and events exist before capture
        libdkv.dkv_init_pool(comp.pool)
        comp.compact(dev, AH, AL)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        libdkv.dkv_init_pool(comp.pool)
        comp.compact(dev, AH, AL)
    # scribble over the outputs, then let the replay rebuild them
    comp.tables.fwd.fill_(-7)
    comp.tables.unit_hdr.fill_(-7)
    comp.classes.fill_(0x55)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert libdkv.dkv_get_status(comp.pool) == libdkv.DKV_OK
    assert_same_state(fetch(comp), exp, what="graph replay")
