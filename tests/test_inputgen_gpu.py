"""Device-filled inputs equal the host draws bit for bit (fp32 and bf16)."""
import numpy as np
import pytest
import torch

import inputgen

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bf16", [False, True])
def test_device_fill_matches_host(bf16):
    n = 3_000_017
    t = torch.empty(n, dtype=torch.bfloat16 if bf16 else torch.float32, device="cuda")
    inputgen.dev_fill_normal(9, 3, 0.0, 0.5, 1234, n, bf16, t.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    host = inputgen.normal(9, 3, 0.0, 0.5, 1234, n, bf16)
    got = t.view(torch.int16).cpu().numpy().view(np.uint16) if bf16 else t.cpu().numpy()
    np.testing.assert_array_equal(got, host)
