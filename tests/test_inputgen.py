"""The seeded input generator: determinism, index addressing, bf16 rounding
(against torch's own conversion), the value distributions of the recipe."""
import numpy as np
import pytest
import torch

import inputgen
from inputgen import workloads as W


def test_deterministic_and_addressable():
    a = inputgen.normal(7, 1, 0.0, 1.0, 1000, 5000, False)
    b = inputgen.normal(7, 1, 0.0, 1.0, 0, 6000, False)
    np.testing.assert_array_equal(a, b[1000:])
    idx = np.array([5999, 0, 1234, 1000])
    np.testing.assert_array_equal(inputgen.normal_at(7, 1, 0.0, 1.0, idx, False), b[idx])
    assert not np.array_equal(inputgen.normal(8, 1, 0.0, 1.0, 0, 100, False), b[:100])
    assert not np.array_equal(inputgen.normal(7, 2, 0.0, 1.0, 0, 100, False), b[:100])


def test_bf16_matches_torch_round_to_nearest_even():
    f = inputgen.normal(3, 4, 0.0, 3.0, 0, 200_000, False)
    bits = inputgen.normal(3, 4, 0.0, 3.0, 0, 200_000, True)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, ref)
    np.testing.assert_array_equal(inputgen.bf16_to_f32(bits),
                                  torch.from_numpy(f).to(torch.bfloat16).float().numpy())


def test_normal_distribution():
    from scipy import stats
    x = inputgen.normal(11, 2, 0.0, 0.5, 0, 400_000, False).astype(np.float64)
    assert abs(x.mean()) < 0.005 and abs(x.std() - 0.5) < 0.005
    assert stats.kstest(x / 0.5, "norm").pvalue > 1e-3


def test_delta_bias_recipe():
    w = W.WORKLOADS["mamba130m"]
    bias = W.bias_vector(w).astype(np.float64)
    dt = np.log1p(np.exp(bias))
    assert dt.min() >= 1e-3 * (1 - 1e-5) and dt.max() <= 1e-1 * (1 + 1e-5)
    # log-uniform: log(dt) roughly uniform over [ln 1e-3, ln 1e-1]
    q = (np.log(dt) - np.log(1e-3)) / (np.log(1e-1) - np.log(1e-3))
    assert 0.4 < q.mean() < 0.6


def test_workload_table():
    ws = W.WORKLOADS
    assert (ws["tiny"].batch, ws["tiny"].L, ws["tiny"].d_inner, ws["tiny"].d_state) == (1, 64, 16, 4)
    assert ws["mamba130m"].elements == 2 * 2048 * 1536
    assert ws["mamba2p8b"].bf16 and ws["long"].L == 1 << 20 and ws["decode"].decode
    A = W.A_matrix(ws["tiny"])
    np.testing.assert_array_equal(A[5], -np.arange(1, 5, dtype=np.float32))


def test_sampled_inputs_match_full():
    w = W.WORKLOADS["tiny"]
    full = W.host_scan_inputs(w)
    part = W.host_scan_inputs(w, b_sel=[0], d_sel=[2, 9, 15], t_count=20)
    for k in ("u", "delta", "z"):
        np.testing.assert_array_equal(part[k], full[k][:, :20][:, :, [2, 9, 15]])
    for k in ("B", "C"):
        np.testing.assert_array_equal(part[k], full[k][:, :20])
