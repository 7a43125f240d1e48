"""Seeded synthetic workloads for the compaction path.

This module only draws inputs.  It holds none of the method's arithmetic (no
significance averaging, classification, quantisation or allocation): it
produces K, V, the attention-received sums ``sig_sum``, their counts
``sig_cnt`` and the request lengths, with the shapes and value distributions
of the five workloads below.  Both the CUDA path and the CPU oracle consume
exactly these bytes.

Workloads (shapes from the DiffKV evaluation setting: Llama-3-8B, Qwen2.5-7B
and a 32B reasoning model producing long chains of thought; DiffKV review,
"Referee Report, Summary" and "If this is right"):

- ``tiny``: 1 layer, 1 request of 512 tokens, 8 query / 2 KV heads, page 16,
  4096 pages.  K, V ~ N(0,1) with 4 outlier channels x8; significance from an
  exact fp64 causal softmax of seeded Q ~ N(0,1) against K / sqrt(128).
- ``llama``: 32 layers, 16 x 4096 tokens, 32 / 8 heads, page 16.  2% outlier
  channels (3 of 128) x10; significance log-normal(sigma=2) per (layer, token,
  query head), normalised to mean 1/N per (layer, request, query head).
- ``qwen``: 28 layers, 64 requests with lengths uniform in [1024, 8192],
  28 / 4 heads, page 32, sigma 2.5, 5% heavy-hitter tokens per (layer,
  request, KV head) x50 on all G query heads before normalising.
- ``longcot``: 64 layers, 16 x 16384 tokens, 64 / 8 heads, page 16, sigma 2,
  x exp(-i/8192), the last 64 tokens x10 (the recent window W = 64 of the
  DiffKV review's free-parameter list).
- ``decode``: 32 layers, 256 requests holding 2048..8192 tokens, 32 / 8 heads,
  page 16, one new token per step (see ``decode_update_inputs``).

No public dataset is involved: the DiffKV path has no accuracy metric here,
only the compaction of given tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

D = 128
SEED_BASE = 0xD1FF0000


@dataclass
class Workload:
    name: str
    L: int
    Hq: int
    Hkv: int
    lens: list
    P: int
    alpha_h: float
    alpha_l: float
    sig: str = "lognormal"          # "lognormal" | "softmax" | "softmax_q0"
    sigma: float = 2.0
    n_outlier: int = 3
    outlier_scale: float = 10.0
    heavy_frac: float = 0.0
    heavy_scale: float = 50.0
    decay: float = 0.0               # positions scaled by exp(-i/decay) when > 0
    recent: int = 0                  # last `recent` tokens boosted by recent_scale
    recent_scale: float = 10.0
    F: int = 0                       # pages in the pool; 0 = worst case
    scheme: int = 0                  # precision scheme: 0 K8V4/K4V2, 1 K8V2/K4V1, 2 K4V8/K2V4
    extra: dict = field(default_factory=dict)

    @property
    def R(self) -> int:
        return len(self.lens)

    @property
    def T(self) -> int:
        return int(sum(self.lens))

    @property
    def U(self) -> int:
        return self.L * self.R * self.Hkv

    @property
    def rows(self) -> int:
        return self.L * self.T * self.Hkv

    @property
    def pmax(self) -> int:
        return -(-max(self.lens + [1]) // self.P) + 1

    @property
    def pool_pages(self) -> int:
        if self.F:
            return self.F
        # worst case: every unit needs ceil(N/P) + 1 pages
        return self.L * self.Hkv * sum(-(-n // self.P) + 1 for n in self.lens)


def _uniform_lens(R: int, lo: int, hi: int, seed: int) -> list:
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (R,), generator=g)]


def get(name: str) -> Workload:
    """The named workload (shapes and distribution parameters only)."""
    if name == "tiny":
        return Workload("tiny", L=1, Hq=8, Hkv=2, lens=[512], P=16, alpha_h=1.0, alpha_l=0.2,
                        sig="softmax", n_outlier=4, outlier_scale=8.0, F=4096)
    if name == "llama":
        return Workload("llama", L=32, Hq=32, Hkv=8, lens=[4096] * 16, P=16, alpha_h=1.0,
                        alpha_l=0.2, sigma=2.0)
    if name == "qwen":
        return Workload("qwen", L=28, Hq=28, Hkv=4, lens=_uniform_lens(64, 1024, 8192, SEED_BASE + 3),
                        P=32, alpha_h=1.5, alpha_l=0.3, sigma=2.5, heavy_frac=0.05)
    if name == "longcot":
        return Workload("longcot", L=64, Hq=64, Hkv=8, lens=[16384] * 16, P=16, alpha_h=1.0,
                        alpha_l=0.2, sigma=2.0, decay=8192.0, recent=64)
    if name == "decode":
        return Workload("decode", L=32, Hq=32, Hkv=8, lens=_uniform_lens(256, 2048, 8192, SEED_BASE + 5),
                        P=16, alpha_h=1.0, alpha_l=0.2, sigma=2.0, extra={"steps": 100})
    raise KeyError(name)


def small(name: str = "ragged", **kw) -> Workload:
    """Small parity workloads that span several token tiles with ragged tails."""
    base = dict(L=2, Hq=6, Hkv=2, lens=[300, 7, 517, 0, 129], P=16, alpha_h=1.0, alpha_l=0.2,
                sigma=2.0, n_outlier=3, outlier_scale=10.0)
    base.update(kw)
    return Workload(name, **base)


def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(int(seed) & 0xFFFFFFFFFFFF)


def make_kv_layer(w: Workload, seed: int, layer: int, which: int, device="cpu") -> torch.Tensor:
    """bf16 [T][Hkv][D] for one layer: N(0,1) with per-(layer, KV head) outlier
    channels scaled before the bf16 rounding.  which: 0 = K, 1 = V."""
    g = _gen(seed * 1000003 + layer * 2 + which, device)
    x = torch.randn((w.T, w.Hkv, D), generator=g, device=device, dtype=torch.float32)
    if w.n_outlier > 0:
        pick = torch.rand((w.Hkv, D), generator=g, device=device).argsort(dim=-1)[:, : w.n_outlier]
        mult = torch.ones((w.Hkv, D), device=device, dtype=torch.float32)
        mult.scatter_(1, pick, w.outlier_scale)
        x.mul_(mult)
    return x.to(torch.bfloat16)


def _positions(w: Workload, device) -> tuple[torch.Tensor, torch.Tensor]:
    """Per token: request index and position inside the request."""
    lens = torch.tensor(w.lens, dtype=torch.int64, device=device)
    req = torch.repeat_interleave(torch.arange(w.R, device=device), lens)
    starts = torch.cumsum(lens, 0) - lens
    pos = torch.arange(w.T, device=device) - starts[req]
    return req, pos


def sig_cnt_prefill(w: Workload, device="cpu") -> torch.Tensor:
    """Number of queries that attended to each token: N - i (self included)."""
    lens = torch.tensor(w.lens, dtype=torch.int64, device=device)
    req, pos = _positions(w, device)
    return (lens[req] - pos).to(torch.int32)


def make_sig_layer(w: Workload, seed: int, layer: int, device="cpu", k_layer=None) -> torch.Tensor:
    """fp32 sig_sum [T][Hq] for one layer (prefill: counts are N - i)."""
    if w.sig in ("softmax", "softmax_q0"):
        return _softmax_sig_layer(w, seed, layer, device, k_layer)
    g = _gen(seed * 1000003 + 500000 + layer, device)
    z = torch.randn((w.T, w.Hq), generator=g, device=device, dtype=torch.float64)
    wt = torch.exp(w.sigma * z)
    req, pos = _positions(w, device)
    lens = torch.tensor(w.lens, dtype=torch.int64, device=device)
    G = w.Hq // w.Hkv
    if w.heavy_frac > 0:
        # heavy hitters chosen per (request, KV head), applied to all G query heads
        u = torch.rand((w.T, w.Hkv), generator=g, device=device)
        heavy = (u < w.heavy_frac).to(torch.float64) * (w.heavy_scale - 1.0) + 1.0
        wt = wt * heavy.repeat_interleave(G, dim=1)
    if w.decay > 0:
        wt = wt * torch.exp(-pos.to(torch.float64) / w.decay)[:, None]
    if w.recent > 0:
        boost = torch.where(pos >= lens[req] - w.recent, w.recent_scale, 1.0).to(torch.float64)
        wt = wt * boost[:, None]
    # normalise to mean 1/N per (request, query head): scores sum to 1
    tot = torch.zeros((w.R, w.Hq), dtype=torch.float64, device=device)
    tot.index_add_(0, req, wt)
    score = wt / tot[req]
    cnt = (lens[req] - pos).to(torch.float64)
    return (score * cnt[:, None]).to(torch.float32)


def make_queries(w: Workload, seed: int, layer: int) -> torch.Tensor:
    """fp32 queries [T][Hq][D] ~ N(0,1) (zeros for the "softmax_q0" mode)."""
    g = _gen(seed * 1000003 + 700000 + layer, "cpu")
    q = torch.randn((w.T, w.Hq, D), generator=g, dtype=torch.float32)
    if w.sig == "softmax_q0":
        q.zero_()
    return q


def _softmax_sig_layer(w: Workload, seed: int, layer: int, device, k_layer) -> torch.Tensor:
    """Exact causal-softmax attention received, in fp64, then fp32.

    For query j and key i <= j of one request, p(j, i) = softmax_i(q_j . k_i /
    sqrt(128)); sig_sum[i] = sum over j >= i of p(j, i).  Query head q reads
    KV head floor(q / G).  With sig == "softmax_q0" the queries are zero, so
    p(j, i) = 1 / (j + 1)."""
    G = w.Hq // w.Hkv
    out = torch.zeros((w.T, w.Hq), dtype=torch.float64)
    q_all = make_queries(w, seed, layer)
    kf = k_layer.to("cpu").to(torch.float64)
    start = 0
    for n in w.lens:
        if n == 0:
            continue
        mask = torch.tril(torch.ones((n, n), dtype=torch.bool))
        for qh in range(w.Hq):
            qv = q_all[start:start + n, qh].to(torch.float64)
            kv = kf[start:start + n, qh // G]
            logits = (qv @ kv.T) / math.sqrt(D)
            logits = logits.masked_fill(~mask, float("-inf"))
            p = torch.softmax(logits, dim=1)         # [j][i]
            out[start:start + n, qh] = p.sum(dim=0)  # sum over queries j
        start += n
    return out.to(torch.float32).to(device)


def make_inputs(w: Workload, seed: int | None = None, device="cpu", layers=None) -> dict:
    """All inputs of the workload (or of the given layers) as torch tensors,
    filled layer by layer into preallocated tensors."""
    seed = SEED_BASE if seed is None else seed
    layers = list(range(w.L)) if layers is None else list(layers)
    n = len(layers)
    k = torch.empty((n, w.T, w.Hkv, D), dtype=torch.bfloat16, device=device)
    v = torch.empty((n, w.T, w.Hkv, D), dtype=torch.bfloat16, device=device)
    sig = torch.empty((n, w.T, w.Hq), dtype=torch.float32, device=device)
    for i, l in enumerate(layers):
        k[i] = make_kv_layer(w, seed, l, 0, device)
        v[i] = make_kv_layer(w, seed, l, 1, device)
        sig[i] = make_sig_layer(w, seed, l, device, k_layer=k[i])
    return {
        "L": n, "R": w.R, "Hq": w.Hq, "Hkv": w.Hkv, "T": w.T,
        "k": k, "v": v, "sig_sum": sig,
        "sig_cnt": sig_cnt_prefill(w, device),
        "lens": torch.tensor(w.lens, dtype=torch.int32, device=device),
    }


def to_numpy(inp: dict) -> dict:
    """Host copies of the input bytes in the layout the oracle reads."""
    out = {k: inp[k] for k in ("L", "R", "Hq", "Hkv", "T")}
    out["k"] = inp["k"].detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
    out["v"] = inp["v"].detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
    out["sig_sum"] = inp["sig_sum"].detach().to("cpu").contiguous().numpy()
    out["sig_cnt"] = inp["sig_cnt"].detach().to("cpu").contiguous().numpy()
    out["lens"] = inp["lens"].detach().to("cpu").contiguous().numpy()
    return out


# ------------------------------------------------------------- generation --

ALPHA_MID = 0.5  # significance level the demotion updates move a token to (x alpha / N)


def _i64(x: int) -> int:
    """Two's-complement int64 value of x mod 2^64."""
    x &= (1 << 64) - 1
    return x - (1 << 64) if x >= (1 << 63) else x


def _hash01(step: int, idx: torch.Tensor) -> torch.Tensor:
    """Counter-based uniform [0, 1) from integer ids: the splitmix64 finaliser
    (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
    2014) of id * golden-gamma + step key, on int64 with wrap-around; the
    same on any device."""
    x = idx.to(torch.int64) * _i64(0x9E3779B97F4A7C15) + _i64((step + 1) * 0x632BE59BD9B4E019)
    x = (x ^ ((x >> 30) & 0x3FFFFFFFF)) * _i64(0xBF58476D1CE4E5B9)
    x = (x ^ ((x >> 27) & 0x1FFFFFFFFF)) * _i64(0x94D049BB133111EB)
    x = x ^ ((x >> 31) & 0x1FFFFFFFF)
    return ((x >> 11) & ((1 << 53) - 1)).to(torch.float64) / float(1 << 53)


def decode_context(w: Workload, pre: dict, cap: int, device="cpu") -> dict:
    """Decode-layout copies (capacity-strided context axis: position i of
    request r at r * cap + i) of a prefill batch's significance sums and
    counts; classes are filled in from the prefill result by the caller."""
    lens = torch.tensor(w.lens, dtype=torch.int64, device=device)
    req, pos = _positions(w, device)
    dst = req * cap + pos
    sig = torch.zeros((w.L, w.R * cap, w.Hq), dtype=torch.float32, device=device)
    sig[:, dst] = pre["sig_sum"].to(device)
    cnt = torch.zeros(w.R * cap, dtype=torch.int32, device=device)
    cnt[dst] = pre["sig_cnt"].to(device)
    return {"L": w.L, "R": w.R, "Hq": w.Hq, "Hkv": w.Hkv, "cap": cap, "sig_sum": sig, "sig_cnt": cnt,
            "ctx_lens": lens.to(torch.int32), "dst": dst}


def decode_update_inputs(w: Workload, ctx: dict, step: int, seed: int | None = None, device="cpu",
                         p_prune: float = 0.005, p_demote: float = 0.005) -> dict:
    """Advance the context by one generation step and draw the new tokens.

    For every live position i < ctx_r of request r, layer l and KV head h a
    counter hash u over (step, l, r, h, i) picks the update of the G query
    heads of that KV head:
    u < p_prune (0.5%): sig := 0 (the token stops being attended: it is
              pruned);
    u < p_prune + p_demote (1%): sig := (ALPHA_MID / N) * cnt with
              N = ctx_r + 1 (demoted to the middle tier unless already there);
    else:     sig += sig / cnt (its average stays as it was).
    Every count then grows by one (the new query attends to every position).
    The new token at position ctx_r (none when ctx_r = cap) gets count 1 and a log-normal(sigma)
    self-attention weight with mean 1/N per query head; its K and V are drawn
    like prefill rows.  fp32 division and multiplication as written, in place
    on ctx."""
    seed = SEED_BASE if seed is None else seed
    L, R, Hq, Hkv, cap = w.L, w.R, w.Hq, w.Hkv, ctx["cap"]
    G = Hq // Hkv
    clen = ctx["ctx_lens"].to(torch.int64)
    N = (clen + 1).to(torch.float32)
    sig, cnt = ctx["sig_sum"], ctx["sig_cnt"]
    pos = torch.arange(cap, device=device)
    live = (pos[None, :] < clen[:, None])                                 # [R, cap]
    cntf = cnt.view(R, cap).to(torch.float32)[:, :, None, None]
    mid = (torch.tensor(ALPHA_MID, dtype=torch.float32, device=device) / N)[:, None, None, None]
    rh = torch.arange(R, device=device)[:, None] * Hkv + torch.arange(Hkv, device=device)[None, :]  # [R, Hkv]
    for l in range(L):
        ids = (l * R * Hkv + rh)[:, None, :] * (cap + 1) + pos[None, :, None]   # [R, cap, Hkv]
        u = _hash01(step, ids)[..., None]
        s = sig[l].view(R, cap, Hkv, G)
        upd = torch.where(u < p_prune, torch.zeros_like(s),
                          torch.where(u < p_prune + p_demote, mid * cntf, s + s / cntf))
        s.copy_(torch.where(live[:, :, None, None], upd, s))
    cnt += live.reshape(-1).to(cnt.dtype)
    # the new token of every request (no host round trip: a full request's
    # slot index points at its last position, which keeps its values)
    g = _gen(seed * 1000003 + 900000 + step, device)
    room = clen < cap                                   # a full request takes no new token
    newpos = torch.arange(R, device=device) * cap + clen.clamp(max=cap - 1)
    z = torch.randn((L, R, Hq), generator=g, device=device, dtype=torch.float64)
    wt = torch.exp(w.sigma * z - w.sigma ** 2 / 2) / (clen + 1).to(torch.float64)[None, :, None]
    sig[:, newpos] = torch.where(room[None, :, None], wt.to(torch.float32), sig[:, newpos])
    cnt[newpos] = torch.where(room, torch.ones_like(cnt[newpos]), cnt[newpos])
    kv = Workload(w.name, L=1, Hq=Hq, Hkv=Hkv, lens=[R], P=w.P, alpha_h=w.alpha_h, alpha_l=w.alpha_l,
                  n_outlier=w.n_outlier, outlier_scale=w.outlier_scale)
    k_new = torch.stack([make_kv_layer(kv, seed + 77 * step + 1, l, 0, device) for l in range(L)])
    v_new = torch.stack([make_kv_layer(kv, seed + 77 * step + 1, l, 1, device) for l in range(L)])
    return {"k_new": k_new, "v_new": v_new, "new_lens": room.to(torch.int32)}


def decode_queries(w: Workload, n_layers: int, seed: int, step: int = 0, device="cpu") -> torch.Tensor:
    """bf16 [n_layers][R][Hq][D] queries of one generation step, N(0,1)."""
    g = _gen(seed * 1000003 + 700000 + step, device)
    return torch.randn((n_layers, w.R, w.Hq, D), generator=g, device=device).to(torch.bfloat16)


def prefill_queries(w: Workload, seed: int, layer: int, device="cpu") -> torch.Tensor:
    """bf16 [T][Hq][D] prefill queries of one layer, N(0,1)."""
    g = _gen(seed * 1000003 + 800000 + layer, device)
    return torch.randn((w.T, w.Hq, D), generator=g, device=device).to(torch.bfloat16)
