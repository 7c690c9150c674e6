"""Seeded synthetic inputs for the sparse-verification hot path.

This module only draws numbers and lays them out. It holds none of the
method's arithmetic (no attention, no softmax, no selection), so both the
CUDA path and the fp64 oracle can consume the very same bytes.

Shapes follow the workloads that the Dustin pages evaluate ("Technical
Summary: Dustin", Experimental Results: Qwen2.5-72B-shaped attention at 32k
context, batched; Qwen2.5-0.5B-shaped draft heads).  The datasets named there
(PG-19, LongBench) and the model weights are not used: Gaussian bf16 tensors
with planted salient positions stand in for them.

Recipe
------
* Every tensor is drawn from N(0, 1) in fp32 by torch's seeded generator on
  the requested device (its own seed per tensor kind and layer) and rounded to
  bf16 with round-to-nearest-even.  The same call on the same device gives the
  same bytes; the GPU and CPU streams differ, so a test always hands both sides
  one set of tensors.
* Planted salient positions: for each sequence ``b`` a set of ``n_planted``
  distinct positions outside the protected sinks/window is drawn.  At each
  planted position, the key row of every KV head ``g`` (every layer, target and
  draft caches) is replaced by ``3 * sqrt(d) * u_g`` where ``u_g`` is the unit
  vector along the mean of the query rows that read head ``g`` (for the target
  cache: the historical and the verify query rows of the heads of group ``g``;
  for the draft cache: the draft query rows of the heads of its group).  Such a
  key has three times the norm of a typical N(0, 1) key and points along the
  queries, so its logits stand far above the background.
* Drift (budget/gamma sweep workload): the look-ahead set shares
  ``1 - drift`` of its positions with the historical set.  Target keys at the
  historical set point along the historical queries, target keys at the
  look-ahead-only positions along the verify queries, draft keys at the
  look-ahead set along the draft queries.
* Cache rows at or beyond ``seq_len`` (the slack left for appends) hold a
  canary: bf16 NaN by default, so any read past the context shows up.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

SEED_BASE = 0xD0571000
BF16_NAN = np.uint16(0x7FC0)

# tensor ids (one independent stream family per tensor kind)
_T_K, _T_V, _T_Q, _T_HQ, _T_KB, _T_VB, _T_DQ, _T_KD, _T_PLANT = range(1, 10)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, budget and SRH list.

    ``srh`` lists ``(channel, layer, q_head)``: channel 0 is the draft
    look-ahead signal (layer indexes the draft layers), channel 1 the target
    historical signal (layer indexes the target layers).
    """
    name: str
    B: int
    L: int
    n_layers: int
    Hq: int
    Hkv: int
    d: int
    Hq_d: int
    Hkv_d: int
    d_d: int
    gamma: int
    k: int
    sinks: int
    window: int
    m: int
    n_planted: int
    srh: tuple
    n_draft_layers: int = 1
    drift: float = 0.0
    slack: int = 64
    seed_id: int = 0

    @property
    def Lcap(self) -> int:
        return ((self.L + self.slack + 63) // 64) * 64

    @property
    def nq_verify(self) -> int:
        return self.gamma + 1

    @property
    def nq_hist(self) -> int:
        return self.gamma + 1

    @property
    def nq_draft(self) -> int:
        return self.gamma

    @property
    def seed(self) -> int:
        return SEED_BASE + self.seed_id

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _srh(target, draft):
    return tuple((1, l, h) for (l, h) in target) + tuple((0, l, h) for (l, h) in draft)


# The five workloads of the benchmark plan.
WORKLOADS = {
    "tiny": Workload(
        name="tiny B1 L1024 Hq4 Hkv1 d64 gamma4 k128", B=1, L=1024, n_layers=1,
        Hq=4, Hkv=1, d=64, Hq_d=2, Hkv_d=1, d_d=64, gamma=4,
        k=128, sinks=4, window=32, m=32, n_planted=8,
        srh=_srh([(0, 0), (0, 1)], [(0, 0), (0, 1)]), seed_id=1),
    "layer8k": Workload(
        name="qwen72b-layer B1 L8192 gamma4 k1024", B=1, L=8192, n_layers=1,
        Hq=64, Hkv=8, d=128, Hq_d=14, Hkv_d=2, d_d=64, gamma=4,
        k=1024, sinks=16, window=128, m=256, n_planted=64,
        srh=_srh([(0, 0), (0, 16), (0, 32), (0, 48)], [(0, 0), (0, 3), (0, 7), (0, 10)]),
        seed_id=2),
    "batched32k": Workload(
        name="qwen72b-layer B16 L32768 gamma5 k2048", B=16, L=32768, n_layers=1,
        Hq=64, Hkv=8, d=128, Hq_d=14, Hkv_d=2, d_d=64, gamma=5,
        k=2048, sinks=16, window=256, m=512, n_planted=256,
        srh=_srh([(0, 0), (0, 16), (0, 32), (0, 48)], [(0, 0), (0, 3), (0, 7), (0, 10)]),
        seed_id=3),
    "sweep32k": Workload(
        name="qwen72b-layer B8 L32768 sweep", B=8, L=32768, n_layers=1,
        Hq=64, Hkv=8, d=128, Hq_d=14, Hkv_d=2, d_d=64, gamma=4,
        k=2048, sinks=16, window=256, m=512, n_planted=256, drift=0.1,
        srh=_srh([(0, 0), (0, 16), (0, 32), (0, 48)], [(0, 0), (0, 3), (0, 7), (0, 10)]),
        seed_id=4),
    "stack128k": Workload(
        name="qwen72b-8layer B4 L131072 gamma4 k4096", B=4, L=131072, n_layers=8,
        Hq=64, Hkv=8, d=128, Hq_d=14, Hkv_d=2, d_d=64, gamma=4,
        k=4096, sinks=16, window=512, m=1024, n_planted=256,
        srh=_srh([(0, 0), (0, 32), (4, 16), (4, 48)], [(0, 0), (0, 3), (0, 7), (0, 10)]),
        seed_id=5),
}


def sweep_points():
    """(k, gamma) grid of the budget/gamma sweep; m = k / 4."""
    return [(k, g) for k in (512, 1024, 2048, 4096) for g in (2, 4, 8)]


# --------------------------------------------------------------------------
# bf16 helpers (bit patterns held as uint16 on the host)
# --------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_bits(t) -> np.ndarray:
    """Host uint16 bit patterns of a bf16 torch tensor (any device)."""
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def _tensor_seed(seed: int, tensor_id: int) -> int:
    return (seed * 1000003 + tensor_id * 7919 + 17) & ((1 << 62) - 1)


def normal_bf16(seed: int, tensor_id: int, shape, device="cpu"):
    """N(0,1) draws from torch's seeded generator, rounded to bf16 (RNE)."""
    import torch
    g = torch.Generator(device=device).manual_seed(_tensor_seed(seed, tensor_id))
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)


def _unit_mean(rows):
    """Unit vector (fp64) along the mean of bf16 rows of shape [..., d]."""
    import torch
    r = rows.to(torch.float64).reshape(-1, rows.shape[-1])
    mu = r.mean(dim=0)
    nrm = torch.linalg.norm(mu)
    if float(nrm) == 0.0:
        mu = torch.ones_like(mu)
        nrm = torch.linalg.norm(mu)
    return mu / nrm


def _planted_row(u, d: int):
    import torch
    return (3.0 * math.sqrt(d) * u).to(torch.float32).to(torch.bfloat16)


@dataclass
class Inputs:
    """One workload's inputs as bf16 torch tensors on ``device``."""
    wl: Workload
    K: list            # per target layer: [B][Hkv][Lcap][d]
    V: list            # per target layer: [B][Hkv][Lcap][d]
    Q: list            # per target layer: verify queries [B][gamma+1][Hq][d]
    hist_q: list       # per target layer: historical queries [B][gamma+1][Hq][d]
    Kb: list           # per target layer: draft-block keys [B][Hkv][gamma+1][d]
    Vb: list           # per target layer: draft-block values [B][Hkv][gamma+1][d]
    draft_q: list      # per draft layer: [B][gamma][Hq_d][d_d]
    Kd: list           # per draft layer: [B][Hkv_d][Lcap][d_d]
    seq_len: np.ndarray          # int32 [B]
    planted: np.ndarray          # int64 [B][n_planted] (historical set)
    planted_look: np.ndarray     # int64 [B][n_planted] (look-ahead set)
    extra: dict = field(default_factory=dict)


def _draw_planted(wl: Workload, rng: np.random.Generator, L: int):
    s_eff = min(wl.sinks, L)
    w0 = max(L - wl.window, s_eff)
    pool = np.arange(s_eff, w0)
    n = min(wl.n_planted, pool.size)
    hist = np.empty((wl.B, n), dtype=np.int64)
    look = np.empty((wl.B, n), dtype=np.int64)
    for b in range(wl.B):
        sh = np.sort(rng.choice(pool, size=n, replace=False))
        hist[b] = sh
        n_new = int(round(wl.drift * n))
        if n_new:
            rest = np.setdiff1d(pool, sh)
            keep = np.sort(rng.choice(sh, size=n - n_new, replace=False))
            new = rng.choice(rest, size=n_new, replace=False)
            look[b] = np.sort(np.concatenate([keep, new]))
        else:
            look[b] = sh
    return hist, look


def generate(wl: Workload, device="cpu", slack_fill: str = "nan", layers=None) -> Inputs:
    """Generate all inputs of ``wl`` as bf16 tensors on ``device``.

    ``layers`` restricts which target layers get K/V caches (the others get
    ``None``); the default is all of them.
    """
    import torch
    s = wl.seed
    B, L, Lcap = wl.B, wl.L, wl.Lcap
    G = wl.Hq // wl.Hkv
    Gd = wl.Hq_d // wl.Hkv_d
    layers = range(wl.n_layers) if layers is None else layers
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([s, _T_PLANT])))
    hist, look = _draw_planted(wl, rng, L)

    K, V, Q, HQ, KB, VB = [], [], [], [], [], []
    for l in range(wl.n_layers):
        q = normal_bf16(s, _T_Q * 1000 + l, (B, wl.nq_verify, wl.Hq, wl.d), device)
        hq = normal_bf16(s, _T_HQ * 1000 + l, (B, wl.nq_hist, wl.Hq, wl.d), device)
        kb = normal_bf16(s, _T_KB * 1000 + l, (B, wl.Hkv, wl.nq_verify, wl.d), device)
        vb = normal_bf16(s, _T_VB * 1000 + l, (B, wl.Hkv, wl.nq_verify, wl.d), device)
        Q.append(q); HQ.append(hq); KB.append(kb); VB.append(vb)
        if l not in layers:
            K.append(None); V.append(None)
            continue
        k = normal_bf16(s, _T_K * 1000 + l, (B, wl.Hkv, Lcap, wl.d), device)
        v = normal_bf16(s, _T_V * 1000 + l, (B, wl.Hkv, Lcap, wl.d), device)
        for b in range(B):
            ph = torch.as_tensor(hist[b], device=device)
            extra_pos = np.setdiff1d(look[b], hist[b])
            pe = torch.as_tensor(extra_pos, device=device)
            for g in range(wl.Hkv):
                heads = slice(g * G, (g + 1) * G)
                u_h = _unit_mean(torch.cat([hq[b, :, heads, :], q[b, :, heads, :]]))
                k[b, g, ph] = _planted_row(u_h, wl.d)
                if extra_pos.size:
                    k[b, g, pe] = _planted_row(_unit_mean(q[b, :, heads, :]), wl.d)
        _fill_slack(k, L, slack_fill)
        _fill_slack(v, L, slack_fill)
        K.append(k); V.append(v)

    DQ, KD = [], []
    for l in range(wl.n_draft_layers):
        dq = normal_bf16(s, _T_DQ * 1000 + l, (B, wl.nq_draft, wl.Hq_d, wl.d_d), device)
        kd = normal_bf16(s, _T_KD * 1000 + l, (B, wl.Hkv_d, Lcap, wl.d_d), device)
        for b in range(B):
            pl = torch.as_tensor(look[b], device=device)
            for g in range(wl.Hkv_d):
                u_d = _unit_mean(dq[b, :, g * Gd:(g + 1) * Gd, :])
                kd[b, g, pl] = _planted_row(u_d, wl.d_d)
        _fill_slack(kd, L, slack_fill)
        DQ.append(dq); KD.append(kd)

    seq_len = np.full((B,), L, dtype=np.int32)
    return Inputs(wl, K, V, Q, HQ, KB, VB, DQ, KD, seq_len, hist, look)


def _fill_slack(cache, L: int, how: str):
    import torch
    if cache.shape[2] <= L:
        return
    if how == "nan":
        cache[:, :, L:, :] = float("nan")
    elif how == "zero":
        cache[:, :, L:, :] = 0
    elif how != "random":
        raise ValueError(how)


def random_importance(seed: int, B: int, Lcap: int, ties: bool = False,
                      spread: float = 3.0) -> np.ndarray:
    """fp32 importance maps [B][2][Lcap] for selection-only tests.

    Values are exponentials of N(0, spread) (positive; the default spread
    gives a wide dynamic range, a small one packs most values into a few
    binary orders of magnitude, so that the top bits of many keys agree);
    with ``ties`` they are quantised to 16 levels so that many keys are equal.
    """
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 77])))
    x = np.exp(spread * g.standard_normal((B, 2, Lcap))).astype(np.float32)
    if ties:
        x = (np.floor(x.clip(0, 15.999)) + 1.0).astype(np.float32) / 16.0
    return x
