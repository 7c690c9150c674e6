"""The seeded generator is deterministic and plants what its recipe says."""
import math

import numpy as np
import torch

from synth import WORKLOADS, generate, to_bits, f32_to_bf16_bits, bf16_bits_to_f32


def test_same_seed_same_bytes():
    a = generate(WORKLOADS["tiny"])
    b = generate(WORKLOADS["tiny"])
    for x, y in zip(a.K + a.V + a.Q + a.hist_q + a.Kd + a.draft_q, b.K + b.V + b.Q + b.hist_q + b.Kd + b.draft_q):
        assert np.array_equal(to_bits(x), to_bits(y))
    assert np.array_equal(a.planted, b.planted)


def test_planted_rows_point_along_queries():
    wl = WORKLOADS["tiny"]
    x = generate(wl)
    k = x.K[0].float()
    for p in x.planted[0]:
        row = k[0, 0, p]
        assert abs(float(row.norm()) - 3 * math.sqrt(wl.d)) < 0.1
        q = torch.cat([x.hist_q[0][0, :, :, :], x.Q[0][0, :, :, :]]).float().reshape(-1, wl.d).mean(0)
        cos = float(row @ q / (row.norm() * q.norm()))
        assert cos > 0.999
    s_eff, w0 = wl.sinks, wl.L - wl.window
    assert np.all((x.planted >= s_eff) & (x.planted < w0))
    assert len(set(x.planted[0].tolist())) == wl.n_planted


def test_slack_canary_and_rounding():
    wl = WORKLOADS["tiny"]
    x = generate(wl, slack_fill="nan")
    assert torch.isnan(x.K[0][:, :, wl.L:].float()).all()
    assert not torch.isnan(x.K[0][:, :, :wl.L].float()).any()
    v = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5], dtype=np.float32)
    assert bf16_bits_to_f32(f32_to_bf16_bits(v)).tolist() == [1.0, 1.015625, -2.5]
