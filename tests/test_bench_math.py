"""The bench's roofline arithmetic (CPU): algorithmic bytes and ALU clocks per element, checked
against the same quantities worked out term by term for the named workloads."""
import pytest

import bench
from inputgen import workloads as W


def test_forward_bytes_of_the_mamba_2p8b_shape():
    # 8 x 2048 x 5120 x 16, bf16 I/O: u, delta, z read and y written (2 bytes each), B and C
    # rows (2 bytes per state and step), A / D / bias once (fp32), last_state once (fp32)
    acts = 8 * 2048 * 5120 * 4 * 2
    bc = 8 * 2048 * 16 * 2 * 2
    params = 5120 * 16 * 4 + 5120 * 4 * 2
    last = 8 * 5120 * 16 * 4
    assert bench.algorithmic_bytes(W.WORKLOADS["mamba2p8b"]) == acts + bc + params + last == 675127296


def test_forward_bytes_of_the_long_context_shape():
    acts = 1048576 * 2048 * 4 * 2
    bc = 1048576 * 16 * 2 * 2
    params = 2048 * 16 * 4 + 2048 * 4 * 2
    last = 2048 * 16 * 4
    assert bench.algorithmic_bytes(W.WORKLOADS["long"]) == acts + bc + params + last


def test_forward_bytes_fp32_io():
    acts = 2 * 2048 * 1536 * 4 * 4
    bc = 2 * 2048 * 16 * 2 * 4
    params = 1536 * 16 * 4 + 1536 * 4 * 2
    last = 2 * 1536 * 16 * 4
    assert bench.algorithmic_bytes(W.WORKLOADS["mamba130m"]) == acts + bc + params + last


def test_ssd_bytes():
    # x, z read and y written (bf16), dt per head, B and C shared by the heads, the fp32 last
    # state, and A / dt_bias per head and D per channel
    acts = 8 * 2048 * 5120 * 3 * 2
    dt = 8 * 2048 * 80 * 2
    bc = 8 * 2048 * 2 * 128 * 2
    last = 8 * 5120 * 128 * 4
    params = (2 * 80 + 5120) * 4
    assert bench.ssd_algorithmic_bytes(W.WORKLOADS["ssd2p7b"]) == acts + dt + bc + last + params


def test_alu_bound_of_the_scan():
    # d_state 16: 4 FP32 per state + 6 per element = 70 FP32 operations; 16 + 2 exponentials
    # and a reciprocal (two SFU slots) = 20 SFU slots; the softplus logarithm either as 10 more
    # FP32 operations or as an lg2 (two SFU slots): max(80/128, 20/32) = 0.625 clocks per
    # element beats max(70/128, 22/32) = 0.6875
    assert bench.alu_clocks_per_element(16) == pytest.approx(0.625)
    assert 148 * 2032e6 / bench.alu_clocks_per_element(16) / 1e9 == pytest.approx(481.18, abs=0.01)
    # conv1d + SiLU in front: 7 more FP32, one more exponential and one more reciprocal
    assert bench.alu_clocks_per_element(16, conv=True) == pytest.approx(max(87 / 128, 23 / 32))


def test_alu_bound_of_the_backward():
    # 15 FP32 per state + 16 per element = 256; 2 ex2 per state + 4 + 4 reciprocal/log (two
    # slots each) = 44 SFU slots: FP32-bound at 2 clocks per element
    assert bench.bwd_alu_clocks_per_element(16) == pytest.approx(2.0)
