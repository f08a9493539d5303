"""The device-side failure path: a bounded wait that cannot complete gives up
after its limit, the error reaches the host as MSA_ERR_TIMEOUT, and the
context stays usable.  No fault, no hang: the wait is the library's own
bounded mbarrier wait on a barrier that nothing arrives on."""
import time

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O

pytestmark = pytest.mark.gpu

MSA_ERR_TIMEOUT = 5


def test_bounded_wait_times_out_and_context_survives(cuda_dev):
    from block_sparse_long_proxy_gb300 import msa
    t0 = time.perf_counter()
    with pytest.raises(msa.MsaError) as e:
        msa.selftest_wait_timeout()
    elapsed = time.perf_counter() - t0
    assert e.value.status == MSA_ERR_TIMEOUT
    assert 1.5 < elapsed < 60.0  # the wait's 2 s limit, not an early exit
    # the context still runs kernels: a small top-k against the oracle
    rng = np.random.default_rng(3)
    ms = rng.standard_normal((5, 2, 40)).astype(np.float32)
    nvp = np.array([1, 10, 20, 39, 40], np.int32)
    got = msa.topk_select(torch.from_numpy(ms).to(cuda_dev), 4, torch.from_numpy(nvp).to(cuda_dev)).cpu().numpy()
    assert np.array_equal(got, O.topk_select(ms, 4, nvp))
