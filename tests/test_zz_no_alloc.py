"""dustin_score_noalloc: scoring for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (or any allocator) at the moment they
score, so they cannot hand the library a workspace; this entry point keeps its
scratch in a static device array inside the library instead.  Its output must
match dustin_score's on the same inputs, call after call, while the static
array keeps the previous call's contents, and its device error word must
reach the caller through dustin_score_noalloc_check.  This file runs last so that a
stop-at-first-failure run has already run every other test.
"""
import dataclasses

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import sparse_kv_verify_gb300 as dk  # noqa: E402
from synth import WORKLOADS  # noqa: E402

from _cases import Case, IMP_RTOL, IMP_FLOOR, assert_importance  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _close(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    rel = np.abs(a - b) / np.maximum(np.abs(b), IMP_FLOOR)
    return rel.max() <= IMP_RTOL


@pytest.mark.parametrize("name", ["tiny", "layer8k"])
def test_noalloc_matches_workspace_score_twice(name):
    c = Case(WORKLOADS[name])
    ref = dk.dustin_score(c.p, c.draft, c.target, c.wl.srh, c.seq)
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        dk.dustin_score_noalloc(c.p, c.draft, c.target, c.wl.srh, c.seq, importance=out)
        assert dk.noalloc_check() == 0
        assert _close(out, ref)


def test_noalloc_two_groups_matches_oracle():
    """Sixteen 8K-position sequences with 36 (SRH head, query row) pairs each
    need 16 x 36 x Lcap x 4 bytes of logits, more than the 16 MiB array, so the
    call scores them in at least two groups of sequences; every sequence must
    still match the fp64 oracle."""
    wl = dataclasses.replace(WORKLOADS["layer8k"], B=16)
    c = Case(wl, seq_len=[8192 - 97 * b for b in range(16)])
    n_pairs = sum((wl.gamma + 1) if s[0] == 1 else wl.gamma for s in wl.srh)
    assert n_pairs == 36 and 16 * n_pairs * wl.Lcap * 4 > (16 << 20)
    out = torch.full((wl.B, 2, wl.Lcap), float("nan"), dtype=torch.float32, device="cuda")
    dk.dustin_score_noalloc(c.p, c.draft, c.target, c.wl.srh, c.seq, importance=out)
    assert dk.noalloc_check() == 0
    assert_importance(out, c.oracle_score(), c.x.seq_len)


def test_noalloc_error_word_is_sticky_until_checked():
    """A seq_len beyond the cache capacity is flagged (the sequence is
    skipped); the flag survives a later clean call and is cleared by the
    check that reports it."""
    c = Case(WORKLOADS["tiny"])
    out = torch.empty((1, 2, c.wl.Lcap), dtype=torch.float32, device="cuda")
    bad = torch.tensor([c.wl.Lcap + 1], dtype=torch.int32, device="cuda")
    dk.dustin_score_noalloc(c.p, c.draft, c.target, c.wl.srh, bad, importance=out)
    dk.dustin_score_noalloc(c.p, c.draft, c.target, c.wl.srh, c.seq, importance=out)
    assert dk.noalloc_check() == dk.DEV_SEQLEN
    assert dk.noalloc_check() == 0
    dk.dustin_score_noalloc(c.p, c.draft, c.target, c.wl.srh, c.seq, importance=out)
    assert dk.noalloc_check() == 0
    assert_importance(out, c.oracle_score(), c.x.seq_len)


def test_noalloc_rejects_oversize():
    """Scratch beyond the array's 16 MiB is refused with DUSTIN_ERANGE before
    any launch: here one sequence alone needs 18 pairs x 2^20 positions x 4
    bytes = 72 MiB of logits."""
    c = Case(WORKLOADS["tiny"])
    big = dk.Params(1, 1 << 20, 4, 4, 32, 32, 128)
    imp = torch.empty((1, 2, 16), dtype=torch.float32, device="cuda")
    with pytest.raises(dk.DustinError) as e:
        dk.dustin_score_noalloc(big, c.draft, c.target, c.wl.srh, c.seq, importance=imp)
    assert e.value.status == -2
