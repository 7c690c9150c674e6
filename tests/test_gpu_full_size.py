"""GPU parity at the full sizes of the budget/gamma sweep (B=8, L=32768, twelve
(k, gamma) points, 10 % saliency drift) and of the 8-layer stack (B=4,
L=131072, about 17 GB of KV), in the launch configuration of
dustin_verify_step; the selection-policy variants the pages compare against;
and the attention-recovery report of the policies.

Outputs are checked on samples the oracle computes one by one: the importance
of one sequence in full, the selection of every sequence (bit-exact on the
GPU's own scores), attention of sampled (sequence, layer, KV head) triples,
among them units that the verification kernel's stream-K split cuts across
CTAs.
Host copies are limited to the sampled slices."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import sparse_kv_verify_gb300 as dk
from oracle import dustin_oracle as O
from synth import WORKLOADS, generate, random_importance, sweep_points, to_bits

from _cases import assert_attention, assert_importance, params_of, sampled_units

pytestmark = pytest.mark.gpu


def _score_one(x, wl, b, layers):
    """Oracle importance of sequence b from host copies of that sequence's
    SRH layers only (other layers are not read by the score)."""
    def sub(ts):
        return [to_bits(t[b:b + 1]) if l in layers else None for l, t in enumerate(ts)]
    return O.score(sub(x.draft_q), sub(x.Kd), sub(x.hist_q), sub(x.K), wl.srh,
                   x.seq_len[b:b + 1], wl.Lcap)


def _verify_one(x, wl, I_ref, b, layer, g):
    G = wl.Hq // wl.Hkv
    hs = slice(g * G, (g + 1) * G)
    return O.verify(to_bits(x.Q[layer][b:b + 1, :, hs]), to_bits(x.K[layer][b:b + 1, g:g + 1]),
                    to_bits(x.V[layer][b:b + 1, g:g + 1]), to_bits(x.Kb[layer][b:b + 1, g:g + 1]),
                    to_bits(x.Vb[layer][b:b + 1, g:g + 1]), I_ref[b:b + 1].astype(np.int64),
                    x.seq_len[b:b + 1]), hs


@pytest.mark.parametrize("k,gamma", sweep_points())
def test_sweep_full_size_sampled(k, gamma):
    wl = WORKLOADS["sweep32k"].with_(k=k, gamma=gamma, m=k // 4)
    x = generate(wl, device="cuda")
    seq = torch.as_tensor(x.seq_len, device="cuda")
    p = params_of(wl)
    layer = dk.VerifyLayer(x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0])
    call = dk.StepCall(p, dk.Signal(x.draft_q, x.Kd), dk.Signal(x.hist_q, x.K), wl.srh, [layer], seq)
    imp, I, outs = call()
    assert dk.check(call.ws) == 0
    imp_np = imp.double().cpu().numpy()
    b = gamma % wl.B
    assert_importance(imp_np[b:b + 1], _score_one(x, wl, b, {0}), x.seq_len[b:b + 1])
    I_ref, _ = O.select(imp_np, x.seq_len, wl.k, wl.sinks, wl.window, wl.m)
    assert np.array_equal(I.cpu().numpy(), I_ref)
    units = {(b, k // 512 % wl.Hkv)} | {(bb, g) for (_, bb, g) in sampled_units(p, wl)}
    for (bb, g) in sorted(units):
        ref, hs = _verify_one(x, wl, I_ref, bb, 0, g)
        assert_attention(outs[0][bb:bb + 1, :, hs], ref)


@pytest.fixture(scope="module")
def stack():
    wl = WORKLOADS["stack128k"]
    x = generate(wl, device="cuda")
    yield wl, x
    del x
    torch.cuda.empty_cache()


def test_stack_full_size_step_and_append(stack):
    """Eight layers share one selection from SRHs on layers 0 and 4; then the
    accepted rows (3 per sequence per layer) are appended."""
    wl, x = stack
    seq = torch.as_tensor(x.seq_len, device="cuda")
    p = params_of(wl)
    layers = [dk.VerifyLayer(x.Q[l], x.K[l], x.V[l], x.Kb[l], x.Vb[l]) for l in range(wl.n_layers)]
    call = dk.StepCall(p, dk.Signal(x.draft_q, x.Kd), dk.Signal(x.hist_q, x.K), wl.srh, layers, seq)
    imp, I, outs = call()
    assert dk.check(call.ws) == 0
    imp_np = imp.double().cpu().numpy()
    srh_layers = {e[1] for e in wl.srh}
    assert_importance(imp_np[:1], _score_one(x, wl, 0, srh_layers), x.seq_len[:1])
    I_ref, _ = O.select(imp_np, x.seq_len, wl.k, wl.sinks, wl.window, wl.m)
    assert np.array_equal(I.cpu().numpy(), I_ref)
    units = {(1, 4, 3)} | {(b, l, g) for (l, b, g) in sampled_units(p, wl, wl.n_layers)}
    for (b, l, g) in sorted(units):
        ref, hs = _verify_one(x, wl, I_ref, b, l, g)
        assert_attention(outs[l][b:b + 1, :, hs], ref)

    # append the first 3 draft-block rows of every sequence in every layer
    n_acc = torch.full((wl.B,), 3, dtype=torch.int32, device="cuda")
    before = x.seq_len.copy()
    ws = dk.workspace(p)
    dk.dustin_kv_append(p, x.K, x.V, x.Kb, x.Vb, n_acc, seq, ws=ws)
    assert dk.check(ws) == 0
    assert np.array_equal(seq.cpu().numpy(), before + 3)
    for (b, l, g) in [(0, 0, 0), (wl.B - 1, wl.n_layers - 1, wl.Hkv - 1)]:
        L0 = int(before[b])
        assert torch.equal(x.K[l][b, g, L0:L0 + 3], x.Kb[l][b, g, :3])
        assert torch.equal(x.V[l][b, g, L0:L0 + 3], x.Vb[l][b, g, :3])


# ------------------------------------------------------- selection policies
# The pages compare Dustin's tiered selection with a sink + recent-window cache
# (StreamingLLM) and with single-signal selection; all three are settings of
# the same budget parameters.


def _policies(k, sinks, window):
    return {
        "dustin": dict(sinks=sinks, window=window, m=k // 4, k=k),
        "streaming": dict(sinks=sinks, window=k - sinks, m=0, k=k),
        "draft_only": dict(sinks=sinks, window=window, m=k - sinks - window, k=k),
        "target_only": dict(sinks=sinks, window=window, m=0, k=k),
    }


@pytest.mark.parametrize("policy", ["dustin", "streaming", "draft_only", "target_only"])
def test_selection_policies_bit_exact(policy):
    B, L, Lcap = 3, 6000, 6016
    keys = random_importance(123, B, Lcap, ties=policy == "target_only")
    seq = np.array([L, 4000, 5999], dtype=np.int32)
    pp = _policies(512, 8, 64)[policy]
    p = dk.Params(B, Lcap, 4, pp["sinks"], pp["window"], pp["m"], pp["k"])
    I = dk.dustin_select(p, torch.as_tensor(keys, device="cuda"), torch.as_tensor(seq, device="cuda"))
    ref, _ = O.select(keys.astype(np.float64), seq, pp["k"], pp["sinks"], pp["window"], pp["m"])
    I = I.cpu().numpy()
    assert np.array_equal(I, ref)
    if policy == "streaming":
        for b, Lb in enumerate(seq):
            w = pp["window"]
            assert np.array_equal(I[b], np.r_[np.arange(pp["sinks"]), np.arange(Lb - w, Lb)])


def test_attention_recovery_of_policies():
    """Share of the dense verification attention mass captured by each
    policy's I_verify, on the 8 K-position layer with planted salient keys:
    the tiered selection recovers more than the sink + window cache and at
    least as much as the weaker of the two single signals."""
    wl = WORKLOADS["layer8k"]
    x = generate(wl, device="cuda")
    seq = torch.as_tensor(x.seq_len, device="cuda")
    imp = dk.dustin_score(params_of(wl), dk.Signal(x.draft_q, x.Kd), dk.Signal(x.hist_q, x.K),
                          wl.srh, seq)
    Q, K = to_bits(x.Q[0]), to_bits(x.K[0])
    arr = {}
    for name, pp in _policies(wl.k, wl.sinks, wl.window).items():
        p = dk.Params(wl.B, wl.Lcap, wl.gamma, pp["sinks"], pp["window"], pp["m"], pp["k"])
        I = dk.dustin_select(p, imp, seq).cpu().numpy()
        arr[name] = float(O.attention_recovery(Q, K, I, x.seq_len).mean())
    print("attention recovery by policy:", {k: round(v, 4) for k, v in arr.items()})
    assert arr["dustin"] > arr["streaming"]
    assert arr["dustin"] >= min(arr["draft_only"], arr["target_only"])
    assert all(0.0 < v <= 1.0 + 1e-12 for v in arr.values())


def test_attention_recovery_by_policy_sweep(capsys):
    """Attention recovery rate of each policy on the drift workload (B=8,
    L=32768, k=2048, gamma=4; the historical and look-ahead planted sets share
    90 %): GPU scores and GPU selection for every policy, the oracle's dense
    probabilities for the recovery of the first sampled sequences.  Prints a
    table of the rates; asserts only that they are rates and that the budgeted
    signal-driven selection recovers more than sinks plus a window."""
    wl = WORKLOADS["sweep32k"].with_(k=2048, gamma=4, m=512)
    x = generate(wl, device="cuda")
    seq = torch.as_tensor(x.seq_len, device="cuda")
    imp = dk.dustin_score(params_of(wl), dk.Signal(x.draft_q, x.Kd), dk.Signal(x.hist_q, x.K),
                          wl.srh, seq)
    n = 2   # sampled sequences
    Q, K = to_bits(x.Q[0][:n]), to_bits(x.K[0][:n])
    arr = {}
    for name, pp in _policies(wl.k, wl.sinks, wl.window).items():
        p = dk.Params(wl.B, wl.Lcap, wl.gamma, pp["sinks"], pp["window"], pp["m"], pp["k"])
        I = dk.dustin_select(p, imp, seq).cpu().numpy()[:n]
        arr[name] = (pp, O.attention_recovery(Q, K, I, x.seq_len[:n]))
    with capsys.disabled():
        print("\n| policy | sinks | window | m (draft tier) | f (target tier) | "
              + " | ".join(f"ARR seq {b}" for b in range(n)) + " | mean |")
        print("|---|---|---|---|---|" + "---|" * (n + 1))
        for name, (pp, r) in arr.items():
            f = pp["k"] - pp["sinks"] - pp["window"] - pp["m"]
            print(f"| {name} | {pp['sinks']} | {pp['window']} | {pp['m']} | {f} | "
                  + " | ".join(f"{v:.4f}" for v in r) + f" | {r.mean():.4f} |")
    assert all(np.all((r > 0.0) & (r <= 1.0 + 1e-12)) for _, r in arr.values())
    assert arr["dustin"][1].mean() > arr["streaming"][1].mean()


def test_collect_two_query_scoring():
    """Scoring on two query rows only (the first draft look-ahead row and the
    bonus row of the historical target queries): the caller passes signals
    holding just those rows, and the scores match the oracle on the same rows."""
    wl = WORKLOADS["layer8k"]
    x = generate(wl, device="cuda")
    seq = torch.as_tensor(x.seq_len, device="cuda")
    dq = [t[:, :1].contiguous() for t in x.draft_q]          # first draft row
    hq = [t[:, -1:].contiguous() for t in x.hist_q]          # bonus row
    imp = dk.dustin_score(params_of(wl), dk.Signal(dq, x.Kd), dk.Signal(hq, x.K), wl.srh, seq)
    ref = O.score([to_bits(t) for t in dq], [to_bits(t) for t in x.Kd], [to_bits(t) for t in hq],
                  [to_bits(t) for t in x.K], wl.srh, x.seq_len, wl.Lcap)
    assert_importance(imp, ref, x.seq_len)
    # each channel's mass is one per (head, row): 4 heads x 1 row
    assert np.allclose(ref[0, :, : x.seq_len[0]].sum(axis=1), [4.0, 4.0])
