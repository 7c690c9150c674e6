"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a private copy of the oracle's source (a
wrong index, sign, scale, mask bound or tie rule) and checks that at least one
pin of test_oracle_pins fails against the mutated copy.  The real oracle
module is never modified.
"""
import os
import types

import pytest

import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "dustin_oracle.py")

MUTATIONS = [
    ("gqa group as modulo", "return h // (hq // hkv)", "return h % hkv",
     [P.test_score_gqa_group_mapping]),
    ("scale 1/d", "logits = keys @ q / math.sqrt(d)", "logits = keys @ q / d",
     [P.test_score_golden_two_keys, P.test_score_single_pair_is_library_softmax]),
    ("channel swapped", "imp[b, channel, :L] += softmax(logits)",
     "imp[b, 1 - channel, :L] += softmax(logits)",
     [P.test_score_golden_two_keys, P.test_score_channels_are_separate]),
    ("softmax not normalised", "return e / np.sum(e, axis=axis, keepdims=True)", "return e",
     [P.test_score_mass_closed_form]),
    ("ties to the higher index", "order = np.lexsort((cand, -scores[cand]))",
     "order = np.lexsort((-cand, -scores[cand]))",
     [P.test_select_golden_hand_example, P.test_select_all_equal_keys_closed_form]),
    ("ascending score order", "order = np.lexsort((cand, -scores[cand]))",
     "order = np.lexsort((cand, scores[cand]))",
     [P.test_select_golden_hand_example]),
    ("budget split ignores protected", "m1 = min(m, k - n_p)", "m1 = min(m, k)",
     [P.test_select_golden_hand_example] + [lambda s=s: P.test_select_matches_brute_force(s)
                                            for s in range(12)]),
    ("target tier may repeat draft", "rest = np.setdiff1d(U, D)", "rest = U",
     [P.test_select_golden_hand_example]),
    ("block mask off by one", "keys = np.concatenate([kc, kb[: t + 1]])\n                    vals = np.concatenate([vc, vb[: t + 1]])",
     "keys = np.concatenate([kc, kb[: t + 2]])\n                    vals = np.concatenate([vc, vb[: t + 2]])",
     [P.test_verify_golden_two_keys, P.test_verify_equal_keys_mean_of_values]),
    ("block never visible", "keys = np.concatenate([kc, kb[: t + 1]])\n                    vals = np.concatenate([vc, vb[: t + 1]])",
     "keys = np.concatenate([kc, kb[:1]])\n                    vals = np.concatenate([vc, vb[:1]])",
     [P.test_verify_golden_two_keys, P.test_dense_matches_torch_sdpa]),
    ("values from keys", "O[b, t, h, :] = p @ vals", "O[b, t, h, :] = p @ keys",
     [P.test_verify_equal_keys_mean_of_values, P.test_verify_golden_two_keys]),
    ("dense drops last context row", "return _attend(Q, K, V, Kb, Vb, lambda b: np.arange(int(seq_len[b])))",
     "return _attend(Q, K, V, Kb, Vb, lambda b: np.arange(int(seq_len[b]) - 1))",
     [P.test_verify_full_budget_equals_dense, P.test_dense_matches_torch_sdpa]),
    ("recovery reads the other KV head", "keys = bf16(K[b, kv_group(h, hq, hkv), :L, :])",
     "keys = bf16(K[b, hkv - 1 - kv_group(h, hq, hkv), :L, :])",
     [P.test_attention_recovery_golden_two_heads]),
    ("recovery without 1/sqrt(d)", "p = softmax(keys @ bf16(Q[b, t, h, :]) / math.sqrt(d))",
     "p = softmax(keys @ bf16(Q[b, t, h, :]))", [P.test_attention_recovery_golden_two_heads]),
    ("recovery past seq_len", "keys = bf16(K[b, kv_group(h, hq, hkv), :L, :])",
     "keys = bf16(K[b, kv_group(h, hq, hkv), :, :])", [P.test_attention_recovery_golden_two_heads]),
    ("recovery averaged over heads only", "arr[b] = tot / (hq * T)", "arr[b] = tot / hq",
     [P.test_attention_recovery_golden_two_heads]),
    ("append shifted", "K2[b, :, L:L + n, :] = Kb[b, :, :n, :]",
     "K2[b, :, L + 1:L + n + 1, :] = Kb[b, :, :n, :]", [P.test_kv_append_exact_copy]),
]


def _mutant(old, new):
    src = open(SRC).read()
    assert old in src, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(monkeypatch, name, old, new, pins):
    monkeypatch.setattr(P, "O", _mutant(old, new))
    caught = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught += 1
    assert caught > 0, f"no pin caught mutation '{name}'"
