"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test checks the oracle against one of: a hand-derived golden fixture
(tests/golden), a closed form, an invariant the Dustin pages fix, a special
case that reduces to a library routine (scipy / torch), or brute force on a
tiny input.  None of them calls the CUDA path.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import dustin_oracle as O
from synth import WORKLOADS, generate, to_bits, f32_to_bf16_bits, random_importance

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def bits(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def rnd_bits(rng, shape, scale=1.0):
    return bits(scale * rng.standard_normal(shape))


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# score
# ---------------------------------------------------------------------------


def _score_case(rng, B=2, L=(37, 50), Lcap=64, hq=4, hkv=2, d=8, hq_d=2, hkv_d=1, d_d=8,
                nq_t=3, nq_d=2, srh=((1, 0, 0), (1, 0, 3), (0, 0, 1))):
    hist_q = [rnd_bits(rng, (B, nq_t, hq, d))]
    K = [rnd_bits(rng, (B, hkv, Lcap, d))]
    draft_q = [rnd_bits(rng, (B, nq_d, hq_d, d_d))]
    Kd = [rnd_bits(rng, (B, hkv_d, Lcap, d_d))]
    seq_len = np.array(L, dtype=np.int32)
    return draft_q, Kd, hist_q, K, list(srh), seq_len, Lcap


def test_score_mass_closed_form():
    """Each pair's softmax sums to 1, so channel c sums to its number of pairs."""
    rng = np.random.default_rng(1)
    args = _score_case(rng)
    imp = O.score(*args)
    srh, seq_len = args[4], args[5]
    n_t = sum(1 for s in srh if s[0] == 1) * args[2][0].shape[1]
    n_d = sum(1 for s in srh if s[0] == 0) * args[0][0].shape[1]
    for b in range(len(seq_len)):
        assert imp[b, 1].sum() == pytest.approx(n_t, rel=1e-13)
        assert imp[b, 0].sum() == pytest.approx(n_d, rel=1e-13)
        assert np.all(imp[b, :, seq_len[b]:] == 0.0)
        assert np.all(imp[b, :, : seq_len[b]] > 0.0)


def test_score_equal_keys_uniform():
    """All keys equal -> every position gets exactly n_pairs / L."""
    rng = np.random.default_rng(2)
    draft_q, Kd, hist_q, K, srh, seq_len, Lcap = _score_case(rng, B=1, L=(45,))
    K[0][:] = bits(rng.standard_normal(8))[None, None, None, :]
    Kd[0][:] = bits(rng.standard_normal(8))[None, None, None, :]
    imp = O.score(draft_q, Kd, hist_q, K, srh, seq_len, Lcap)
    assert np.allclose(imp[0, 1, :45], 2 * 3 / 45, rtol=1e-14, atol=0)
    assert np.allclose(imp[0, 0, :45], 1 * 2 / 45, rtol=1e-14, atol=0)


def test_score_golden_two_keys():
    g = load("score_two_keys.json")
    d = g["d"]
    hist_q = [bits(np.array(g["q"]).reshape(1, 1, 1, d))]
    K = [bits(np.array(g["keys"]).reshape(1, 1, 2, d))]
    draft_q = [bits(np.zeros((1, 1, 1, d)))]
    Kd = [bits(np.zeros((1, 1, 2, d)))]
    imp = O.score(draft_q, Kd, hist_q, K, [(1, 0, 0)], np.array([2], np.int32), 2)
    assert imp[0, 1].tolist() == pytest.approx(g["expected_importance"], rel=1e-15)
    assert imp[0, 0].tolist() == [0.0, 0.0]


def test_score_single_pair_is_library_softmax():
    """One SRH with one query row: the map is scipy's softmax of the logits."""
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(3)
    d, L = 16, 29
    q = rnd_bits(rng, (1, 1, 1, d))
    K = rnd_bits(rng, (1, 1, L, d))
    imp = O.score([q], [K], [q], [K], [(0, 0, 0)], np.array([L], np.int32), L)
    qf = O.bf16(q).reshape(d)
    Kf = O.bf16(K).reshape(L, d)
    ref = sp.softmax(Kf @ qf * (1.0 / 4.0))       # 1/sqrt(16)
    assert np.allclose(imp[0, 0], ref, rtol=1e-13, atol=0)


def test_score_gqa_group_mapping():
    """Query head h reads KV head h // (Hq / Hkv): a spike planted at position
    p_g in KV head g shows up for exactly the heads of group g."""
    hq, hkv, d, L = 8, 4, 8, 16
    q = np.zeros((1, 1, hq, d)); q[..., 0] = 4.0
    K = np.zeros((1, hkv, L, d))
    spikes = [3, 7, 11, 14]
    for g, p in enumerate(spikes):
        K[0, g, p, 0] = 8.0                     # logit 32/sqrt(8) ~ 11.3 vs 0
    for h in range(hq):
        imp = O.score([bits(q)], [bits(K)], [bits(q)], [bits(K)], [(1, 0, h)],
                      np.array([L], np.int32), L)
        assert int(np.argmax(imp[0, 1])) == spikes[h // 2]


def test_score_channels_are_separate():
    rng = np.random.default_rng(4)
    args = list(_score_case(rng))
    a = O.score(*args)
    args[1] = [rnd_bits(rng, args[1][0].shape)]          # new draft cache
    b = O.score(*args)
    assert np.array_equal(a[:, 1], b[:, 1])
    assert not np.allclose(a[:, 0], b[:, 0])


def test_score_position_permutation_equivariance():
    rng = np.random.default_rng(5)
    draft_q, Kd, hist_q, K, srh, seq_len, Lcap = _score_case(rng, B=1, L=(64,))
    perm = rng.permutation(64)
    a = O.score(draft_q, Kd, hist_q, K, srh, seq_len, Lcap)
    b = O.score(draft_q, [Kd[0][:, :, perm]], hist_q, [K[0][:, :, perm]], srh, seq_len, Lcap)
    assert np.allclose(b[0][:, :], a[0][:, perm], rtol=1e-12, atol=0)


def test_score_ignores_slack_canary():
    wl = WORKLOADS["tiny"]
    x = generate(wl, slack_fill="nan")
    imp = O.score([to_bits(t) for t in x.draft_q], [to_bits(t) for t in x.Kd],
                  [to_bits(t) for t in x.hist_q], [to_bits(t) for t in x.K], wl.srh,
                  x.seq_len, wl.Lcap)
    assert np.all(np.isfinite(imp))
    assert imp[0, 1].sum() == pytest.approx(2 * wl.nq_hist, rel=1e-13)
    assert imp[0, 0].sum() == pytest.approx(2 * wl.nq_draft, rel=1e-13)


# ---------------------------------------------------------------------------
# select
# ---------------------------------------------------------------------------


def _brute_tier(scores, cand, n):
    """Membership by counting: i is in the tier iff fewer than n candidates
    beat it (higher score, or equal score at a lower index)."""
    chosen = []
    for i in cand:
        beat = sum(1 for j in cand if scores[j] > scores[i] or (scores[j] == scores[i] and j < i))
        if beat < n:
            chosen.append(i)
    return sorted(chosen)


def _check_select(I, tiers, imp, L, k, sinks, window, m):
    ns, nw, m1, f = tiers
    row = list(I)
    assert len(row) == k
    if k >= L:
        assert row == list(range(L)) + [-1] * (k - L)
        return
    assert len(set(row)) == k
    sink_part = list(range(min(sinks, L)))
    w0 = max(L - window, len(sink_part))
    win_part = list(range(w0, L))
    assert row[:ns] == sink_part and row[ns:ns + nw] == win_part
    U = list(range(len(sink_part), w0))
    D = row[ns + nw: ns + nw + m1]
    R = row[ns + nw + m1:]
    assert m1 == min(m, k - ns - nw) and len(R) == f
    assert D == _brute_tier(imp[0], U, m1)
    rest = [i for i in U if i not in set(D)]
    assert R == _brute_tier(imp[1], rest, f)


@pytest.mark.parametrize("seed", range(12))
def test_select_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    L = int(rng.integers(8, 48))
    Lcap = 48
    k = int(rng.integers(1, 56))
    sinks = int(rng.integers(0, 5))
    window = int(rng.integers(0, 6))
    if sinks + window > k:
        k = sinks + window + int(rng.integers(0, 4))
    m = int(rng.integers(0, k + 2))
    ties = seed % 2 == 0
    imp = random_importance(seed, 1, Lcap, ties=ties).astype(np.float64)
    I, tiers = O.select(imp, np.array([L]), k, sinks, window, m)
    _check_select(I[0], tiers[0], imp[0], L, k, sinks, window, m)


def test_select_golden_hand_example():
    g = load("select_hand.json")
    imp = np.zeros((1, 2, g["L"]))
    imp[0, 0] = g["draft"]
    imp[0, 1] = g["target"]
    I, tiers = O.select(imp, np.array([g["L"]]), g["k"], g["sinks"], g["window"], g["m"])
    assert I[0].tolist() == g["expected"]
    assert list(tiers[0]) == g["expected_tiers"]


def test_select_all_equal_keys_closed_form():
    """Equal scores everywhere: the draft tier is the first m' unprotected
    positions and the target tier the next f (lower index wins every tie)."""
    L, k, s, w, m = 100, 30, 4, 10, 7
    imp = np.ones((1, 2, L))
    I, tiers = O.select(imp, np.array([L]), k, s, w, m)
    U0 = s
    assert I[0].tolist() == (list(range(s)) + list(range(L - w, L))
                             + list(range(U0, U0 + 7)) + list(range(U0 + 7, U0 + 7 + 9)))


def test_select_budget_covers_context():
    imp = np.random.default_rng(0).random((2, 2, 16))
    I, _ = O.select(imp, np.array([10, 16]), 16, 2, 3, 4)
    assert I[0].tolist() == list(range(10)) + [-1] * 6
    assert I[1].tolist() == list(range(16))


def test_select_protected_overflow_rejected():
    with pytest.raises(ValueError):
        O.select(np.ones((1, 2, 64)), np.array([64]), 8, 5, 5, 0)


# ---------------------------------------------------------------------------
# verify / dense
# ---------------------------------------------------------------------------


def _verify_case(rng, B=2, L=(40, 33), Lcap=48, hq=4, hkv=2, d=8, gamma=2):
    T = gamma + 1
    Q = rnd_bits(rng, (B, T, hq, d))
    K = rnd_bits(rng, (B, hkv, Lcap, d))
    V = rnd_bits(rng, (B, hkv, Lcap, d))
    Kb = rnd_bits(rng, (B, hkv, T, d))
    Vb = rnd_bits(rng, (B, hkv, T, d))
    return Q, K, V, Kb, Vb, np.array(L, dtype=np.int32)


def test_verify_full_budget_equals_dense():
    """k >= L selects every row, and sparse verification equals dense."""
    rng = np.random.default_rng(7)
    Q, K, V, Kb, Vb, sl = _verify_case(rng)
    I = np.full((2, 48), -1)
    for b in range(2):
        I[b, : sl[b]] = np.arange(sl[b])
    a = O.verify(Q, K, V, Kb, Vb, I, sl)
    b = O.dense(Q, K, V, Kb, Vb, sl)
    assert np.array_equal(a, b)


def test_verify_equal_keys_mean_of_values():
    """Equal keys -> uniform weights: O is the mean of V over the selected rows
    and the block rows u <= t (so each t sees a different set)."""
    rng = np.random.default_rng(8)
    Q, K, V, Kb, Vb, sl = _verify_case(rng, B=1, L=(30,))
    kr = bits(rng.standard_normal(8))
    K[:] = kr
    Kb[:] = kr
    I = np.array([[3, 5, 8, 13, 21, -1]])
    Ov = O.verify(Q, K, V, Kb, Vb, I, sl)
    Vf, Vbf = O.bf16(V), O.bf16(Vb)
    for h in range(4):
        g = h // 2
        for t in range(3):
            rows = np.concatenate([Vf[0, g, [3, 5, 8, 13, 21]], Vbf[0, g, : t + 1]])
            assert np.allclose(Ov[0, t, h], rows.mean(axis=0), rtol=1e-13, atol=1e-15)


def test_verify_gamma0_empty_selection_is_block_row():
    rng = np.random.default_rng(9)
    Q, K, V, Kb, Vb, sl = _verify_case(rng, B=1, L=(20,), gamma=0)
    Ov = O.verify(Q, K, V, Kb, Vb, np.full((1, 4), -1), sl)
    for h in range(4):
        assert np.array_equal(Ov[0, 0, h], O.bf16(Vb[0, h // 2, 0]))


def test_verify_golden_two_keys():
    g = load("verify_two_keys.json")
    d = g["d"]
    Q = bits(np.tile(np.array(g["q"]), (1, 2, 1, 1)))
    K = bits(np.array(g["cache_k"]).reshape(1, 1, 1, d))
    V = bits(np.array(g["cache_v"]).reshape(1, 1, 1, d))
    Kb = bits(np.array(g["block_k"]).reshape(1, 1, 2, d))
    Vb = bits(np.array(g["block_v"]).reshape(1, 1, 2, d))
    Ov = O.verify(Q, K, V, Kb, Vb, np.array([[0]]), np.array([1], np.int32))
    assert Ov[0, :, 0, :].tolist()[0] == pytest.approx(g["expected_O"][0], rel=1e-14, abs=1e-16)
    assert Ov[0, :, 0, :].tolist()[1] == pytest.approx(g["expected_O"][1], rel=1e-14, abs=1e-16)


def test_dense_matches_torch_sdpa():
    """Dense verification is torch's scaled_dot_product_attention (fp64, CPU)
    with the context fully visible and the draft block causal."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(10)
    Q, K, V, Kb, Vb, sl = _verify_case(rng)
    Od = O.dense(Q, K, V, Kb, Vb, sl)
    T, hq, d, G = 3, 4, 8, 2
    for b in range(2):
        L = int(sl[b])
        for h in range(hq):
            g = h // G
            keys = np.concatenate([O.bf16(K[b, g, :L]), O.bf16(Kb[b, g])])
            vals = np.concatenate([O.bf16(V[b, g, :L]), O.bf16(Vb[b, g])])
            mask = np.ones((T, L + T), dtype=bool)
            for t in range(T):
                mask[t, L + t + 1:] = False
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(O.bf16(Q[b, :, h]))[None], torch.tensor(keys)[None],
                torch.tensor(vals)[None], attn_mask=torch.tensor(mask)[None])[0].numpy()
            assert np.allclose(Od[b, :, h], ref, rtol=1e-12, atol=1e-14)


def test_verify_rejects_index_beyond_context():
    rng = np.random.default_rng(11)
    Q, K, V, Kb, Vb, sl = _verify_case(rng, B=1, L=(20,))
    with pytest.raises(ValueError):
        O.verify(Q, K, V, Kb, Vb, np.array([[1, 20]]), sl)


# ---------------------------------------------------------------------------
# append and attention recovery
# ---------------------------------------------------------------------------


def test_kv_append_exact_copy():
    rng = np.random.default_rng(12)
    K = rnd_bits(rng, (2, 2, 16, 4))
    V = rnd_bits(rng, (2, 2, 16, 4))
    Kb = rnd_bits(rng, (2, 2, 3, 4))
    Vb = rnd_bits(rng, (2, 2, 3, 4))
    K2, V2, sl2 = O.kv_append(K, V, Kb, Vb, np.array([2, 0]), np.array([5, 9]))
    assert sl2.tolist() == [7, 9]
    assert np.array_equal(K2[0, :, 5:7], Kb[0, :, :2]) and np.array_equal(V2[0, :, 5:7], Vb[0, :, :2])
    untouched = np.ones(16, bool); untouched[5:7] = False
    assert np.array_equal(K2[0][:, untouched], K[0][:, untouched])
    assert np.array_equal(K2[1], K[1]) and np.array_equal(V2[1], V[1])


def test_attention_recovery_bounds():
    rng = np.random.default_rng(13)
    Q, K, V, Kb, Vb, sl = _verify_case(rng, B=1, L=(30,))
    full = np.arange(30)[None]
    assert O.attention_recovery(Q, K, full, sl)[0] == pytest.approx(1.0, rel=1e-13)
    assert O.attention_recovery(Q, K, np.full((1, 3), -1), sl)[0] == 0.0


def test_attention_recovery_golden_two_heads():
    """Hand-derived recovery rates (tests/golden/arr_two_heads.json): the
    per-head KV mapping, the 1/sqrt(d) scale, the seq_len cut and the mean
    over heads and queries each change the value if wrong."""
    g = load("arr_two_heads.json")
    Q = bits(np.array(g["q"])[None])            # [1][T=2][hq=2][d]
    K = bits(np.array(g["k"])[None])            # [1][hkv=2][3][d]
    sl = np.array([g["seq_len"]], np.int32)
    e = g["expected"]
    for key, sel in (("sel_1", [1]), ("sel_0", [0, -1]), ("sel_0_1", [0, 1]), ("sel_none", [-1])):
        got = O.attention_recovery(Q, K, np.array([sel]), sl)[0]
        assert got == pytest.approx(e[key], rel=1e-14, abs=1e-16), key


def test_planted_positions_are_recovered_on_tiny():
    """End-to-end sanity on the tiny workload: planted salient positions end up
    in I_verify (a sanity signal of the input recipe, not a parity pin)."""
    wl = WORKLOADS["tiny"]
    x = generate(wl)
    imp = O.score([to_bits(t) for t in x.draft_q], [to_bits(t) for t in x.Kd],
                  [to_bits(t) for t in x.hist_q], [to_bits(t) for t in x.K], wl.srh,
                  x.seq_len, wl.Lcap)
    I, _ = O.select(imp, x.seq_len, wl.k, wl.sinks, wl.window, wl.m)
    assert np.isin(x.planted[0], I[0]).all()
