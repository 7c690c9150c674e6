"""Parity of every CUDA stage with the fp64 oracle on seeded inputs.

Small workloads (tiny, qwen72b-layer 8k) are compared element by element;
the 32k batched workload runs in the launch configuration the benchmark
times and is checked on samples the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU too
    pytest.skip("needs a GPU", allow_module_level=True)

import sparse_kv_verify_gb300 as dk  # noqa: E402
from oracle import dustin_oracle as O  # noqa: E402
from synth import WORKLOADS, random_importance, to_bits  # noqa: E402

from _cases import (Case, params_of, assert_importance, assert_attention,  # noqa: E402
                    assert_select_near, sampled_units)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


# ------------------------------------------------------------------ score


@pytest.mark.parametrize("name", ["tiny", "layer8k"])
def test_score_parity(name):
    c = Case(WORKLOADS[name])
    ws = dk.workspace(c.p, c.draft, c.target, c.wl.srh)
    imp = dk.dustin_score(c.p, c.draft, c.target, c.wl.srh, c.seq, ws=ws)
    assert dk.check(ws) == 0
    assert_importance(imp, c.oracle_score(), c.x.seq_len)


def test_score_ragged_lengths_multi_batch():
    wl = WORKLOADS["tiny"].with_(B=3, L=1024)
    c = Case(wl, seq_len=[1024, 777, 65])
    imp = dk.dustin_score(c.p, c.draft, c.target, wl.srh, c.seq)
    assert_importance(imp, c.oracle_score(), c.x.seq_len)


def test_score_long_caches_in_sequence_groups():
    """Long caches and batches whose logits exceed the L2 budget are scored in
    groups of sequences (here 5 sequences of up to 2^20 - 64 positions)."""
    for L, B in ((40000, 1), (140000, 2), ((1 << 20) - 64, 5)):
        wl = WORKLOADS["tiny"].with_(L=L, B=B, n_planted=16)
        c = Case(wl, seq_len=[L - 777 * i for i in range(B)])
        imp = dk.dustin_score(c.p, c.draft, c.target, wl.srh, c.seq)
        assert_importance(imp, c.oracle_score(), c.x.seq_len)


def test_score_strided_cache_views():
    """Caches that are views with padded strides (not densely packed) are read
    through the general 4-D tensor maps; results are unchanged."""
    wl = WORKLOADS["tiny"].with_(B=2)
    c = Case(wl, seq_len=[1024, 700])
    x = c.x
    pad = lambda t: torch.cat([t, torch.zeros_like(t[:, :, :96])], dim=2)[:, :, : t.shape[2]]
    K2, Kd2 = [pad(t) for t in x.K], [pad(t) for t in x.Kd]
    assert K2[0].stride(1) != K2[0].shape[2] * K2[0].shape[3]
    imp = dk.dustin_score(c.p, dk.Signal(x.draft_q, Kd2), dk.Signal(x.hist_q, K2), wl.srh, c.seq)
    assert_importance(imp, c.oracle_score(), c.x.seq_len)


def test_score_deterministic():
    c = Case(WORKLOADS["layer8k"])
    a = dk.dustin_score(c.p, c.draft, c.target, c.wl.srh, c.seq).clone()
    b = dk.dustin_score(c.p, c.draft, c.target, c.wl.srh, c.seq)
    assert torch.equal(a, b)


# ------------------------------------------------------------------ select


@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("L,k,s,w,m", [(1024, 128, 4, 32, 32), (8192, 1024, 16, 128, 256),
                                        (5000, 700, 0, 0, 700), (300, 299, 3, 5, 0),
                                        (2000, 64, 16, 48, 512), (100, 128, 4, 8, 16)])
def test_select_bit_exact_on_identical_keys(ties, L, k, s, w, m):
    B, Lcap = 3, ((L + 64 + 63) // 64) * 64
    keys = random_importance(L * 7 + k, B, Lcap, ties=ties)
    seq = np.array([L, max(1, L // 2), max(1, L - 3)], dtype=np.int32)
    p = dk.Params(B, Lcap, 4, s, w, m, k)
    I = dk.dustin_select(p, torch.as_tensor(keys, device="cuda"), torch.as_tensor(seq, device="cuda"))
    ref, _ = O.select(keys.astype(np.float64), seq, k, s, w, m)
    assert np.array_equal(I.cpu().numpy(), ref)


@pytest.mark.parametrize("spread", [0.1, 0.02, 0.0003])
@pytest.mark.parametrize("B,L,k,s,w,m", [(2, 131072, 4096, 16, 512, 1024),
                                          (16, 32768, 2048, 16, 256, 512),
                                          (1, 20000, 3000, 8, 64, 700)])
def test_select_narrow_keys(spread, B, L, k, s, w, m):
    """Keys packed into a narrow range: the 12-bit threshold bins hold tens of
    thousands of keys, so the candidate lists are first narrowed by the next
    10 key bits across the cluster (spreads 0.1 and 0.02), or, when even
    those sub-bins are too full (0.0003), the general path runs; every case
    is exact."""
    Lcap = L + 64
    keys = random_importance(int(spread * 1e4) + B, B, Lcap, spread=spread)
    seq = np.array([L - 37 * b for b in range(B)], dtype=np.int32)
    p = dk.Params(B, Lcap, 4, s, w, m, k)
    ws = dk.workspace(p)
    I = dk.dustin_select(p, torch.as_tensor(keys, device="cuda"), torch.as_tensor(seq, device="cuda"),
                         ws=ws)
    assert dk.check(ws) == 0
    ref, _ = O.select(keys.astype(np.float64), seq, k, s, w, m)
    assert np.array_equal(I.cpu().numpy(), ref)


def test_select_long_cache_global_keys():
    """Caches too long to stage keys on chip select from global memory."""
    B, L, k = 2, 131072, 4096
    Lcap = L + 64
    keys = random_importance(5, B, Lcap, ties=True)
    seq = np.array([L, 100000], dtype=np.int32)
    p = dk.Params(B, Lcap, 4, 16, 512, 1024, k)
    I = dk.dustin_select(p, torch.as_tensor(keys, device="cuda"), torch.as_tensor(seq, device="cuda"))
    ref, _ = O.select(keys.astype(np.float64), seq, k, 16, 512, 1024)
    assert np.array_equal(I.cpu().numpy(), ref)


@pytest.mark.parametrize("B", [20, 48, 100, 300])
def test_select_many_sequences(B):
    """Batches too large for one 8-CTA cluster per sequence at once run with
    smaller clusters (down to one CTA per sequence); results stay exact."""
    L, k, s, w, m = 3000, 400, 8, 64, 100
    Lcap = L + 64
    keys = random_importance(B, B, Lcap, ties=bool(B % 2))
    rng = np.random.default_rng(B)
    seq = rng.integers(k - 50, L + 1, size=B).astype(np.int32)
    p = dk.Params(B, Lcap, 4, s, w, m, k)
    I = dk.dustin_select(p, torch.as_tensor(keys, device="cuda"), torch.as_tensor(seq, device="cuda"))
    ref, _ = O.select(keys.astype(np.float64), seq, k, s, w, m)
    assert np.array_equal(I.cpu().numpy(), ref)


def test_select_uncached_keys():
    """Slices too long for shared memory read their keys from global memory."""
    B, L, k = 2, 500000, 4096
    Lcap = L + 64
    keys = random_importance(11, B, Lcap, ties=False)
    seq = np.array([L, 480001], dtype=np.int32)
    p = dk.Params(B, Lcap, 4, 16, 512, 1024, k)
    I = dk.dustin_select(p, torch.as_tensor(keys, device="cuda"), torch.as_tensor(seq, device="cuda"))
    ref, _ = O.select(keys.astype(np.float64), seq, k, 16, 512, 1024)
    assert np.array_equal(I.cpu().numpy(), ref)


def test_select_nan_key_flagged():
    B, L, Lcap = 1, 512, 576
    keys = random_importance(9, B, Lcap)
    keys[0, 0, 100] = np.nan
    p = dk.Params(B, Lcap, 4, 4, 8, 16, 64)
    ws = dk.workspace(p)
    dk.dustin_select(p, torch.as_tensor(keys, device="cuda"),
                     torch.as_tensor(np.array([L], np.int32), device="cuda"), ws=ws)
    assert dk.check(ws) & dk.DEV_NAN


@pytest.mark.parametrize("name", ["tiny", "layer8k"])
def test_select_on_own_scores_vs_oracle_scores(name):
    c = Case(WORKLOADS[name])
    imp = dk.dustin_score(c.p, c.draft, c.target, c.wl.srh, c.seq)
    I = dk.dustin_select(c.p, imp, c.seq)
    wl = c.wl
    assert_select_near(I, c.oracle_score(), c.x.seq_len, wl.k, wl.sinks, wl.window, wl.m)


# ------------------------------------------------------------------ verify


@pytest.mark.parametrize("name", ["tiny", "layer8k"])
def test_verify_parity(name):
    c = Case(WORKLOADS[name])
    wl, x = c.wl, c.x
    I_ref, _ = O.select(c.oracle_score(), x.seq_len, wl.k, wl.sinks, wl.window, wl.m)
    I = torch.as_tensor(I_ref.astype(np.int32), device="cuda")
    ws = dk.workspace(c.p, verify=(wl.Hq, wl.Hkv, wl.d, 1))
    o = dk.dustin_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], I, c.seq, ws=ws)
    assert dk.check(ws) == 0
    assert_attention(o, c.oracle_verify(I_ref))


@pytest.mark.parametrize("name", ["tiny", "layer8k"])
def test_dense_parity(name):
    c = Case(WORKLOADS[name])
    x = c.x
    ws = dk.workspace(c.p, verify=(c.wl.Hq, c.wl.Hkv, c.wl.d, 1))
    o = dk.dense_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], c.seq, ws=ws)
    assert dk.check(ws) == 0
    assert_attention(o, c.oracle_dense())


@pytest.mark.parametrize("gamma", [0, 1, 2, 8, 15])
def test_verify_gamma_range(gamma):
    """gamma from 0 up to 15 (one to eight 16-row m-tiles of queries, G = 8)."""
    wl = WORKLOADS["layer8k"].with_(gamma=gamma, L=2048, k=256, sinks=4, window=64, m=64,
                                    n_planted=16)
    c = Case(wl)
    x = c.x
    rng = np.random.default_rng(gamma)
    I_ref = np.stack([np.sort(rng.choice(wl.L, wl.k, replace=False))]).astype(np.int64)
    I = torch.as_tensor(I_ref.astype(np.int32), device="cuda")
    o = dk.dustin_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], I, c.seq)
    assert_attention(o, c.oracle_verify(I_ref))
    od = dk.dense_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], c.seq)
    assert_attention(od, c.oracle_dense())


@pytest.mark.parametrize("gamma,hq,hkv,d", [(12, 24, 8, 128), (6, 64, 8, 128), (18, 24, 8, 128),
                                             (7, 64, 8, 128), (20, 3, 1, 64), (21, 3, 1, 64)])
def test_verify_query_rows_near_mma_width(gamma, hq, hkv, d):
    """(gamma + 1) * Hq / Hkv query rows of 39, 56, 57, 64, 63 and 66: up to
    64 the verification MMAs are 64 rows wide (16 rows in each tensor-memory
    lane quarter, the last quarter partly or wholly in use), beyond it 128
    rows wide; at d = 128 two CTAs share an SM up to 56 rows and one runs
    alone from 57; row counts that are not multiples of 8 included."""
    wl = WORKLOADS["tiny"].with_(gamma=gamma, Hq=hq, Hkv=hkv, d=d, L=1024, k=256, sinks=4,
                                 window=64, m=64)
    c = Case(wl)
    x = c.x
    rng = np.random.default_rng(gamma * 7 + d)
    I_ref = np.stack([np.sort(rng.choice(wl.L, wl.k, replace=False)) for _ in range(wl.B)]).astype(np.int64)
    I = torch.as_tensor(I_ref.astype(np.int32), device="cuda")
    ws = dk.workspace(c.p, verify=(hq, hkv, d, 1))
    o = dk.dustin_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], I, c.seq, ws=ws)
    assert dk.check(ws) == 0
    assert_attention(o, c.oracle_verify(I_ref))
    od = dk.dense_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], c.seq, ws=ws)
    assert_attention(od, c.oracle_dense())


@pytest.mark.parametrize("gamma,hq,hkv,d,per_sm", [(5, 64, 8, 128, 2), (12, 24, 8, 128, 2),
                                                    (6, 64, 8, 128, 2), (18, 24, 8, 128, 1),
                                                    (7, 64, 8, 128, 1), (20, 3, 1, 64, 2),
                                                    (21, 3, 1, 64, 1)])
def test_verify_ctas_per_sm(gamma, hq, hkv, d, per_sm):
    """Two verification CTAs per SM while the query rows fit 64-row MMAs and
    two CTAs' shared memory fits an SM (48, 39 and 56 rows at d = 128, 63 at
    d = 64); one beyond (57 and 64 rows at d = 128: a query buffer and three
    stages no longer fit twice; 66 rows: 128-row MMAs need 512 tensor-memory
    columns).  The parity tests above run the boundary shapes."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = dk.Params(B=16, Lcap=32768, gamma=gamma, sinks=16, window=256, m=512, k=2048)
    grid, tiles = dk.verify_split(p, hq, hkv, d, 1, False)
    assert tiles == 2048 // 64 + 1
    assert grid == per_sm * sms


@pytest.mark.parametrize("d,hq,hkv", [(64, 2, 1), (128, 16, 8)])
def test_verify_largest_draft_block(d, hq, hkv):
    """gamma + 1 = 64 draft-block rows (one whole block tile under the causal
    mask) and (gamma + 1) * Hq/Hkv = 128 query rows, the largest shape; one
    more draft row is refused with DUSTIN_ERANGE before anything runs."""
    wl = WORKLOADS["tiny"].with_(gamma=63, Hq=hq, Hkv=hkv, d=d, L=1024, k=256, sinks=4,
                                 window=64, m=64)
    c = Case(wl)
    x = c.x
    rng = np.random.default_rng(63)
    I_ref = np.stack([np.sort(rng.choice(wl.L, wl.k, replace=False))]).astype(np.int64)
    I = torch.as_tensor(I_ref.astype(np.int32), device="cuda")
    ws = dk.workspace(c.p, verify=(hq, hkv, d, 1))
    o = dk.dustin_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], I, c.seq, ws=ws)
    assert dk.check(ws) == 0
    assert_attention(o, c.oracle_verify(I_ref))
    od = dk.dense_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], c.seq, ws=ws)
    assert_attention(od, c.oracle_dense())
    p65 = params_of(wl, gamma=64)
    q65 = torch.zeros((wl.B, 65, hq, d), dtype=torch.bfloat16, device="cuda")
    kb65 = torch.zeros((wl.B, hkv, 65, d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dk.DustinError):
        dk.dustin_verify_attn(p65, q65, x.K[0], x.V[0], kb65, kb65, I, c.seq, ws=ws)


def test_verify_full_budget_matches_dense():
    """k >= L: I_verify is every context row, so sparse equals dense."""
    wl = WORKLOADS["tiny"].with_(k=1100)
    c = Case(wl)
    x = c.x
    I = dk.dustin_select(c.p, dk.dustin_score(c.p, c.draft, c.target, wl.srh, c.seq), c.seq)
    assert I[0, :wl.L].tolist() == list(range(wl.L)) and bool((I[0, wl.L:] == -1).all())
    o_s = dk.dustin_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], I, c.seq)
    o_d = dk.dense_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], c.seq)
    assert torch.allclose(o_s, o_d, atol=2e-6, rtol=0)
    assert_attention(o_d, c.oracle_dense())


def test_verify_many_segments_per_cta():
    """Short units (two tiles) and many of them: every CTA of the stream-K
    split runs several units in turn and reloads its query buffers; the
    kernels end cleanly (no wait gives up) and match the oracle.  (80
    sequences keep three or more units per CTA with two CTAs per SM.)"""
    wl = WORKLOADS["tiny"].with_(B=80, Hq=16, Hkv=8, L=512, k=64, sinks=4, window=16, m=16,
                                 n_planted=4)
    c = Case(wl)
    x = c.x
    for dense in (False, True):
        grid, tiles = dk.verify_split(c.p, wl.Hq, wl.Hkv, wl.d, 1, dense)
        T = wl.B * wl.Hkv * tiles
        segs = max(len({t // tiles for t in range(cta * T // grid, (cta + 1) * T // grid)})
                   for cta in range(grid))
        assert segs >= 3, (grid, tiles, segs)
    rng = np.random.default_rng(5)
    I_ref = np.stack([np.sort(rng.choice(wl.L, wl.k, replace=False)) for _ in range(wl.B)])
    I = torch.as_tensor(I_ref.astype(np.int32), device="cuda")
    ws = dk.workspace(c.p, verify=(wl.Hq, wl.Hkv, wl.d, 1))
    o = dk.dustin_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], I, c.seq, ws=ws)
    assert dk.check(ws) == 0
    assert_attention(o, c.oracle_verify(I_ref))
    od = dk.dense_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], c.seq, ws=ws)
    assert dk.check(ws) == 0
    assert_attention(od, c.oracle_dense())


def test_verify_padding_and_bad_index():
    """-1 entries are skipped silently; an index past the context is skipped
    and flagged."""
    c = Case(WORKLOADS["tiny"])
    x, wl = c.x, c.wl
    rng = np.random.default_rng(3)
    I_ref = np.sort(rng.choice(wl.L, 100, replace=False))
    I_pad = np.concatenate([I_ref, -np.ones(wl.k - 100, np.int64)])[None]
    ws = dk.workspace(c.p, verify=(wl.Hq, wl.Hkv, wl.d, 1))
    o = dk.dustin_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0],
                              torch.as_tensor(I_pad.astype(np.int32), device="cuda"), c.seq, ws=ws)
    assert dk.check(ws) == 0
    assert_attention(o, c.oracle_verify(I_pad))
    I_bad = I_pad.copy()
    I_bad[0, 120] = wl.L + 5
    o = dk.dustin_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0],
                              torch.as_tensor(I_bad.astype(np.int32), device="cuda"), c.seq, ws=ws)
    assert dk.check(ws) & dk.DEV_INDEX
    assert_attention(o, c.oracle_verify(I_pad))


def test_verify_ragged_lengths():
    wl = WORKLOADS["tiny"].with_(B=3)
    c = Case(wl, seq_len=[1024, 500, 90])
    x = c.x
    imp = dk.dustin_score(c.p, c.draft, c.target, wl.srh, c.seq)
    I = dk.dustin_select(c.p, imp, c.seq)
    I_np = I.cpu().numpy().astype(np.int64)
    o = dk.dustin_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], I, c.seq)
    assert_attention(o, c.oracle_verify(I_np))
    od = dk.dense_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], c.seq)
    assert_attention(od, c.oracle_dense())


def test_empty_and_one_position_sequences():
    """seq_len[b] = 0 and 1 beside ordinary lengths, through scoring,
    selection, sparse and dense verification and the fused step, against the
    oracle.  An empty context scores 0 everywhere, selects nothing (all -1)
    and its queries attend to the draft block alone; a one-position context
    gives that position the number of (SRH head, query row) pairs of each
    channel (each softmax over one position is 1)."""
    wl = WORKLOADS["tiny"].with_(B=4)
    c = Case(wl, seq_len=[0, 1, 1024, 2])
    x = c.x
    ws = dk.workspace(c.p, c.draft, c.target, wl.srh, verify=(wl.Hq, wl.Hkv, wl.d, 1))
    imp = dk.dustin_score(c.p, c.draft, c.target, wl.srh, c.seq, ws=ws)
    assert dk.check(ws) == 0
    assert_importance(imp, c.oracle_score(), x.seq_len)
    imp_np = imp.double().cpu().numpy()
    n_draft = sum(wl.gamma for e in wl.srh if e[0] == 0)
    n_target = sum(wl.gamma + 1 for e in wl.srh if e[0] == 1)
    assert np.all(imp_np[0] == 0.0)
    assert np.allclose(imp_np[1, :, 0], [n_draft, n_target], rtol=1e-6, atol=0)
    I = dk.dustin_select(c.p, imp, c.seq, ws=ws)
    assert dk.check(ws) == 0
    I_ref, _ = O.select(imp_np, x.seq_len, wl.k, wl.sinks, wl.window, wl.m)
    I_np = I.cpu().numpy()
    assert np.array_equal(I_np, I_ref)
    assert np.all(I_np[0] == -1) and I_np[1, 0] == 0 and np.all(I_np[1, 1:] == -1)
    o = dk.dustin_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], I, c.seq, ws=ws)
    assert dk.check(ws) == 0
    assert_attention(o, c.oracle_verify(I_ref))
    od = dk.dense_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], c.seq, ws=ws)
    assert dk.check(ws) == 0
    assert_attention(od, c.oracle_dense())
    layer = dk.VerifyLayer(x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0])
    call = dk.StepCall(c.p, c.draft, c.target, wl.srh, [layer], c.seq)
    imp2, I2, outs = call()
    assert dk.check(call.ws) == 0
    assert torch.equal(imp2, imp) and torch.equal(I2, I)
    assert_attention(outs[0], c.oracle_verify(I_ref))


# ------------------------------------------------------------------ append


def test_kv_append_and_overflow_flag():
    wl = WORKLOADS["tiny"].with_(B=3, n_layers=2)
    c = Case(wl, seq_len=[1000, 1010, wl.Lcap - 2])
    x = c.x
    before = [(to_bits(k).copy(), to_bits(v).copy()) for k, v in zip(x.K, x.V)]
    n_acc = torch.tensor([3, 0, 4], dtype=torch.int32, device="cuda")
    ws = dk.workspace(c.p)
    dk.dustin_kv_append(c.p, x.K, x.V, x.Kb, x.Vb, n_acc, c.seq, ws=ws)
    flags = dk.check(ws)
    assert flags & dk.DEV_APPEND    # sequence 2 would pass the capacity
    assert c.seq.cpu().tolist() == [1003, 1010, wl.Lcap - 2]
    for l in range(2):
        K2, V2, sl = O.kv_append(before[l][0][:2], before[l][1][:2], to_bits(x.Kb[l])[:2],
                                 to_bits(x.Vb[l])[:2], [3, 0], [1000, 1010])
        assert np.array_equal(to_bits(x.K[l])[:2], K2)
        assert np.array_equal(to_bits(x.V[l])[:2], V2)
        assert np.array_equal(to_bits(x.K[l])[2], before[l][0][2])


def test_kv_append_twice_in_a_row():
    """Two appends back to back on one stream, nothing in between: the second
    copies at the seq_len the first one left, in every sequence and layer
    (gamma + 1 = 5 rows at most per call)."""
    wl = WORKLOADS["tiny"].with_(B=3, n_layers=2)
    c = Case(wl, seq_len=[1000, 1010, 900])
    x = c.x
    before = [(to_bits(k).copy(), to_bits(v).copy()) for k, v in zip(x.K, x.V)]
    n1, n2 = [3, 0, 5], [1, 4, 0]
    ws = dk.workspace(c.p)
    for n in (n1, n2):
        dk.dustin_kv_append(c.p, x.K, x.V, x.Kb, x.Vb, torch.tensor(n, dtype=torch.int32, device="cuda"),
                            c.seq, ws=ws)
    assert dk.check(ws) == 0
    assert c.seq.cpu().tolist() == [1004, 1014, 905]
    for l in range(2):
        kb, vb = to_bits(x.Kb[l]), to_bits(x.Vb[l])
        K1, V1, s1 = O.kv_append(before[l][0], before[l][1], kb, vb, n1, [1000, 1010, 900])
        K2, V2, s2 = O.kv_append(K1, V1, kb, vb, n2, s1)
        assert s2.tolist() == [1004, 1014, 905]
        assert np.array_equal(to_bits(x.K[l]), K2)
        assert np.array_equal(to_bits(x.V[l]), V2)


# ------------------------------------------------------------------ fused step


@pytest.mark.parametrize("name", ["tiny", "layer8k"])
def test_verify_step_end_to_end(name):
    c = Case(WORKLOADS[name])
    wl, x = c.wl, c.x
    layer = dk.VerifyLayer(x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0])
    call = dk.StepCall(c.p, c.draft, c.target, wl.srh, [layer], c.seq)
    imp, I, outs = call()
    assert dk.check(call.ws) == 0
    assert_importance(imp, c.oracle_score(), x.seq_len)
    # selection is bit-exact on the GPU's own fp32 scores
    I_ref, _ = O.select(imp.double().cpu().numpy(), x.seq_len, wl.k, wl.sinks, wl.window, wl.m)
    assert np.array_equal(I.cpu().numpy(), I_ref)
    assert_attention(outs[0], c.oracle_verify(I_ref))
    # planted salient positions are recovered (sanity of the recipe)
    assert np.isin(x.planted, I.cpu().numpy()).mean() > 0.99


def test_verify_step_in_sequence_groups():
    """A batch whose logits exceed the L2 budget is scored by the fused step in
    groups of sequences (here 3 sequences of about 2^19 positions, 37.7 MB of
    logits each: groups of 2 and 1); every stage still matches the oracle."""
    wl = WORKLOADS["tiny"].with_(B=3, L=(1 << 19) - 64, n_planted=16)
    c = Case(wl, seq_len=[wl.L, wl.L - 1000, 70000])
    x = c.x
    layer = dk.VerifyLayer(x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0])
    call = dk.StepCall(c.p, c.draft, c.target, wl.srh, [layer], c.seq)
    n, g = call.launches()
    assert g == 2 and n == 2 * 2 + 3
    imp, I, outs = call()
    assert dk.check(call.ws) == 0
    assert_importance(imp, c.oracle_score(), x.seq_len)
    I_ref, _ = O.select(imp.double().cpu().numpy(), x.seq_len, wl.k, wl.sinks, wl.window, wl.m)
    assert np.array_equal(I.cpu().numpy(), I_ref)
    assert_attention(outs[0], c.oracle_verify(I_ref))


def test_verify_step_multi_layer_shared_selection():
    wl = WORKLOADS["tiny"].with_(n_layers=3, srh=((1, 0, 0), (1, 2, 3), (0, 0, 1)))
    c = Case(wl)
    x = c.x
    layers = [dk.VerifyLayer(x.Q[l], x.K[l], x.V[l], x.Kb[l], x.Vb[l]) for l in range(3)]
    imp, I, outs = dk.dustin_verify_step(c.p, c.draft, c.target, wl.srh, layers, c.seq)
    assert_importance(imp, c.oracle_score(), x.seq_len)
    I_np = I.cpu().numpy().astype(np.int64)
    for l in range(3):
        assert_attention(outs[l], c.oracle_verify(I_np, layer=l))


# ------------------------------------------------------------------ full size


@pytest.fixture(scope="module")
def big():
    return Case(WORKLOADS["batched32k"])


def test_full_size_step_sampled(big):
    """The 32k batched workload in the launch configuration the benchmark
    times: importance of two sequences in full, selection of every sequence
    bit-exact on the GPU's scores, attention of sampled (sequence, KV head)
    pairs against the oracle."""
    c = big
    wl, x = c.wl, c.x
    layer = dk.VerifyLayer(x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0])
    call = dk.StepCall(c.p, c.draft, c.target, wl.srh, [layer], c.seq)
    imp, I, outs = call()
    assert dk.check(call.ws) == 0
    imp_np = imp.double().cpu().numpy()
    for b in (0, wl.B - 1):
        sub = lambda ts: [to_bits(t[b:b + 1]) for t in ts]
        ref = O.score(sub(x.draft_q), sub(x.Kd), sub(x.hist_q), sub(x.K), wl.srh,
                      x.seq_len[b:b + 1], wl.Lcap)
        assert_importance(imp_np[b:b + 1], ref, x.seq_len[b:b + 1])
    I_ref, _ = O.select(imp_np, x.seq_len, wl.k, wl.sinks, wl.window, wl.m)
    I_np = I.cpu().numpy()
    assert np.array_equal(I_np, I_ref)
    G = wl.Hq // wl.Hkv
    o = outs[0]
    for (_, b, g) in sampled_units(c.p, wl, dense=False):
        hs = slice(g * G, (g + 1) * G)
        ref = O.verify(to_bits(x.Q[0][b:b + 1, :, hs]), to_bits(x.K[0][b:b + 1, g:g + 1]),
                       to_bits(x.V[0][b:b + 1, g:g + 1]), to_bits(x.Kb[0][b:b + 1, g:g + 1]),
                       to_bits(x.Vb[0][b:b + 1, g:g + 1]), I_ref[b:b + 1].astype(np.int64),
                       x.seq_len[b:b + 1])
        assert_attention(o[b:b + 1, :, hs], ref)


def test_full_size_dense_sampled(big):
    c = big
    wl, x = c.wl, c.x
    o = dk.dense_verify_attn(c.p, x.Q[0], x.K[0], x.V[0], x.Kb[0], x.Vb[0], c.seq)
    G = wl.Hq // wl.Hkv
    for (_, b, g) in sampled_units(c.p, wl, dense=True):
        hs = slice(g * G, (g + 1) * G)
        ref = O.dense(to_bits(x.Q[0][b:b + 1, :, hs]), to_bits(x.K[0][b:b + 1, g:g + 1]),
                      to_bits(x.V[0][b:b + 1, g:g + 1]), to_bits(x.Kb[0][b:b + 1, g:g + 1]),
                      to_bits(x.Vb[0][b:b + 1, g:g + 1]), x.seq_len[b:b + 1])
        assert_attention(o[b:b + 1, :, hs], ref)


@pytest.mark.parametrize("name,over", [("layer8k", {}), ("tiny", dict(k=1100, n_layers=2))])
def test_compact_kv_then_dense_equals_sparse_verify(name, over):
    """The compacted-cache variant: the selected rows copied into compact
    caches and verified densely match the oracle's sparse verification, and
    bit-for-bit the CUDA sparse verification of the full caches (same keys in
    the same order), in every layer; every (sequence, KV head) pair's K and V
    rows equal a gather of the full caches, zero past the compact length."""
    c = Case(WORKLOADS[name].with_(**over))
    wl, x = c.wl, c.x
    I_ref, _ = O.select(c.oracle_score(), x.seq_len, wl.k, wl.sinks, wl.window, wl.m)
    I = torch.as_tensor(I_ref.astype(np.int32), device="cuda")
    ws = dk.workspace(c.p)
    kcs, vcs, slc = dk.dustin_compact_kv(c.p, x.K, x.V, I, c.seq, ws=ws)
    assert dk.check(ws) == 0
    valid = (I_ref >= 0).sum(axis=1)
    assert np.array_equal(slc.cpu().numpy(), valid)
    pc = params_of(wl, Lcap=wl.k)
    for l in range(wl.n_layers):
        o_sparse = dk.dustin_verify_attn(c.p, x.Q[l], x.K[l], x.V[l], x.Kb[l], x.Vb[l], I, c.seq)
        o_dense = dk.dense_verify_attn(pc, x.Q[l], kcs[l], vcs[l], x.Kb[l], x.Vb[l], slc)
        assert_attention(o_dense, c.oracle_verify(I_ref, layer=l))
        assert torch.equal(o_sparse, o_dense)
        for b in range(wl.B):
            rows = torch.as_tensor(I_ref[b][: valid[b]], device="cuda")
            for g in range(x.K[l].shape[1]):
                for full, comp in ((x.K[l], kcs[l]), (x.V[l], vcs[l])):
                    assert torch.equal(comp[b, g, : valid[b]], full[b, g, rows]), (l, b, g)
                    assert torch.all(comp[b, g, valid[b]:wl.k] == 0), (l, b, g)
