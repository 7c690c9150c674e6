"""The give-up path of the bounded on-chip waits, run on the GPU.

Every mbarrier wait in the kernels gives up after a time limit, flags
DUSTIN_DEV_TIMEOUT and raises the CTA's abort flag so that its other waits
stop too.  Making a real kernel's wait run out would need a copy or an MMA that
never completes; instead dustin_wait_selftest runs the same wait helper in one
CTA on an mbarrier that nothing arrives on, with nothing in flight.  The test
checks the reported status, both waiters' times, and that the context still
runs a scoring call correctly afterwards."""
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import sparse_kv_verify_gb300 as dk  # noqa: E402
from synth import WORKLOADS  # noqa: E402

from _cases import Case, assert_importance  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def test_wait_gives_up_and_aborts_the_other_waiter():
    c = Case(WORKLOADS["tiny"])
    ws = dk.workspace(c.p, c.draft, c.target, c.wl.srh)
    limit = 2_000_000                                   # 2 ms
    waited = dk.wait_selftest(limit, ws).cpu().tolist()
    assert dk.check(ws) == dk.DEV_TIMEOUT
    assert limit <= waited[0] < 500_000_000
    # the second waiter (own limit 2 s) stopped on the abort flag, soon after
    assert waited[0] <= waited[1] < 500_000_000
    assert dk.check(ws) == 0                            # the check cleared the word
    # the context is still usable
    imp = dk.dustin_score(c.p, c.draft, c.target, c.wl.srh, c.seq, ws=ws)
    assert dk.check(ws) == 0
    assert_importance(imp, c.oracle_score(), c.x.seq_len)
