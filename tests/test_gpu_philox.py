"""The device Philox4x32-10 agrees bit for bit with the oracle's independent
implementation (itself pinned to PyTorch's engine) on 10^6 counters."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def test_device_philox_matches_oracle(vas_lib):
    rng = np.random.default_rng(123)
    n = 1_000_000
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    ctr[:1000, 2:] = 0                        # the (position, sequence, 0, 0) form
    key = (0x9ABCDEF0, 0x12345678)
    ref = oracle.philox4x32_10(ctr, np.array(key, dtype=np.uint32))
    c = torch.from_numpy(ctr.view(np.int32)).cuda()
    out = torch.empty_like(c)
    vas_lib.vas_philox4x32_10(c, key[0], key[1], out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), ref)
