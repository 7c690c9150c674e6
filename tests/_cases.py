"""Shared set-up for the GPU parity tests: seeded inputs on the device, the
same bytes on the host for the oracle, and the comparison rules."""
from __future__ import annotations

import numpy as np
import torch

import sparse_kv_verify_gb300 as dk
from oracle import dustin_oracle as O
from synth import WORKLOADS, generate, to_bits

# Tolerances (fp32 accumulation over bf16 inputs, compared with fp64):
IMP_RTOL = 1e-4        # importance, relative
IMP_FLOOR = 1e-30      # absolute floor of the relative check (underflow)
ATT_ATOL = 1e-2        # attention outputs, max abs
TIE_RTOL = 1e-5        # selection: positions this close to a tier boundary may swap


def params_of(wl, **over):
    d = dict(B=wl.B, Lcap=wl.Lcap, gamma=wl.gamma, sinks=wl.sinks, window=wl.window, m=wl.m,
             k=wl.k)
    d.update(over)
    return dk.Params(**d)


class Case:
    def __init__(self, wl, device="cuda", seq_len=None, slack_fill="nan"):
        self.wl = wl
        self.x = generate(wl, device=device, slack_fill=slack_fill)
        if seq_len is not None:
            self.x.seq_len = np.asarray(seq_len, dtype=np.int32)
        self.seq = torch.as_tensor(self.x.seq_len, device=device)
        self.p = params_of(wl)
        self.draft = dk.Signal(self.x.draft_q, self.x.Kd)
        self.target = dk.Signal(self.x.hist_q, self.x.K)

    def bits(self, ts):
        return [to_bits(t) if t is not None else None for t in ts]

    def oracle_score(self):
        x = self.x
        return O.score(self.bits(x.draft_q), self.bits(x.Kd), self.bits(x.hist_q), self.bits(x.K),
                       self.wl.srh, x.seq_len, self.wl.Lcap)

    def oracle_verify(self, I, layer=0):
        x = self.x
        return O.verify(to_bits(x.Q[layer]), to_bits(x.K[layer]), to_bits(x.V[layer]),
                        to_bits(x.Kb[layer]), to_bits(x.Vb[layer]), I, x.seq_len)

    def oracle_dense(self, layer=0):
        x = self.x
        return O.dense(to_bits(x.Q[layer]), to_bits(x.K[layer]), to_bits(x.V[layer]),
                       to_bits(x.Kb[layer]), to_bits(x.Vb[layer]), x.seq_len)


def assert_importance(got, ref, seq_len):
    got = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    for b, L in enumerate(seq_len):
        g, r = got[b, :, :L], ref[b, :, :L]
        if L > 0:
            rel = np.abs(g - r) / np.maximum(np.abs(r), IMP_FLOOR)
            assert rel.max() <= IMP_RTOL, f"b={b}: max rel err {rel.max():.3e}"
        assert np.all(got[b, :, L:] == 0.0)


def assert_attention(got, ref, atol=ATT_ATOL):
    got = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref).max()
    assert err <= atol, f"max abs err {err:.3e}"
    return err


def assert_select_near(I_gpu, imp_ref, seq_len, k, sinks, window, m):
    """GPU selection on its own scores vs the oracle's selection on fp64
    scores: identical except for positions whose fp64 score lies within
    TIE_RTOL of the score at that tier's boundary.  The target tier is
    re-derived from the GPU's own draft tier."""
    I_gpu = I_gpu.cpu().numpy() if isinstance(I_gpu, torch.Tensor) else I_gpu
    for b, L in enumerate(seq_len):
        L = int(L)
        row = I_gpu[b]
        if k >= L:
            assert row.tolist() == list(range(L)) + [-1] * (k - L)
            continue
        s_part, w_part = O.protected_sets(L, sinks, window)
        nP = s_part.size + w_part.size
        assert row[:nP].tolist() == s_part.tolist() + w_part.tolist()
        m1 = min(m, k - nP)
        f = k - nP - m1
        U = np.arange(s_part.size, w_part[0] if w_part.size else L)
        D_gpu = row[nP:nP + m1]
        R_gpu = row[nP + m1:]
        assert np.all(np.diff(D_gpu) > 0) and np.all(np.diff(R_gpu) > 0)
        for tier, (got, sc, cand, n) in enumerate([
                (D_gpu, imp_ref[b, 0], U, m1),
                (R_gpu, imp_ref[b, 1], np.setdiff1d(U, D_gpu), f)]):
            if n == 0:
                assert got.size == 0
                continue
            assert np.all(np.isin(got, cand))
            order = np.lexsort((cand, -sc[cand]))
            ref = np.sort(cand[order[:n]])
            bound = sc[cand[order[n - 1]]]
            diff = np.setxor1d(ref, got)
            near = np.abs(sc[diff] - bound) <= TIE_RTOL * abs(bound)
            assert np.all(near), f"b={b} tier={tier}: {int((~near).sum())} positions off the boundary"


def flags_ok(ws):
    return dk.check(ws) == 0


def sampled_units(p, wl, n_layers=1, dense=False):
    """(layer, sequence, KV head) triples to check at full size: the first,
    middle and last of the units the verification kernel's stream-K split
    cuts across CTAs (their outputs come from the merge kernel), plus the
    first and last unit.  Unit u = (layer * B + b) * Hkv + g."""
    grid, tiles = dk.verify_split(p, wl.Hq, wl.Hkv, wl.d, n_layers, dense)
    cut = dk.split_units(p, wl.Hkv, n_layers, grid, tiles)
    assert len(cut) >= 2, (grid, tiles)
    n_units = n_layers * p.B * wl.Hkv
    us = sorted({cut[0], cut[len(cut) // 2], cut[-1], 0, n_units - 1})
    return [(u // (p.B * wl.Hkv), (u // wl.Hkv) % p.B, u % wl.Hkv) for u in us]
