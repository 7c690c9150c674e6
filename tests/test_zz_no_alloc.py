"""dustin_score_noalloc: scoring for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (or any allocator) at the moment they
score, so they cannot hand the library a workspace; this entry point keeps its
scratch in a static device array inside the library instead.  Its output must
match dustin_score's on the same inputs, call after call, while the static
array keeps the previous call's contents.  This file runs last so that a
stop-at-first-failure run has already run every other test.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import sparse_kv_verify_gb300 as dk  # noqa: E402
from synth import WORKLOADS  # noqa: E402

from _cases import Case, IMP_RTOL, IMP_FLOOR  # noqa: E402


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
        torch.cuda.synchronize()
        assert _close(out, ref)


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
