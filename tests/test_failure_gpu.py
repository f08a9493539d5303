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


def test_plan_allocation_failure_is_reported(cuda_dev):
    """Host-side failure injection: a plan whose device allocation fails
    returns MSA_ERR_NO_MEMORY with nothing allocated, and the next plan (the
    injection used up) is built and works."""
    from block_sparse_long_proxy_gb300 import msa
    MSA_ERR_NO_MEMORY = 4
    before = torch.cuda.mem_get_info()[0]
    msa.inject_plan_alloc_failures(2)
    try:
        for _ in range(2):
            with pytest.raises(msa.MsaError) as e:
                msa.Plan([256], [256], 4, 2, 2, 128, 64, 2, num_pages=2)
            assert e.value.status == MSA_ERR_NO_MEMORY and "injected" in str(e.value)
    finally:
        msa.inject_plan_alloc_failures(0)
    assert torch.cuda.mem_get_info()[0] >= before - (1 << 20)
    plan = msa.Plan([256], [256], 4, 2, 2, 128, 64, 2, num_pages=2)
    rng = np.random.default_rng(1)
    ms = torch.from_numpy(rng.standard_normal((plan.n_tiles, 2, plan.max_blocks)).astype(np.float32)).to(cuda_dev)
    got = msa.topk_select(ms, 2, plan.num_valid_pages).cpu().numpy()
    assert np.array_equal(got, O.topk_select(ms.cpu().numpy(), 2, O.num_valid_pages([256], [256])))


def test_checks_mode_flags_nan_outputs(cuda_dev, monkeypatch):
    """MSA_CHECKS: a plan created with it set scans each call's inputs and
    outputs; a NaN planted in pq (which the block maxima would not carry: a
    max drops NaN operands) and one planted in q both come back as
    MSA_ERR_NONFINITE.  Clean inputs, and the same NaN under a plan made
    without the variable, raise nothing."""
    from block_sparse_long_proxy_gb300 import msa, synth
    from tests.gpu_cases import make_plan
    MSA_ERR_NONFINITE = 7
    case = synth.Case("checks", [300], [300], 4, 2, 128, 2, 64, 2)
    inp = synth.make_inputs(case, device=cuda_dev)
    monkeypatch.setenv("MSA_CHECKS", "1")
    plan = make_plan(case, inp)
    monkeypatch.delenv("MSA_CHECKS")
    plain = make_plan(case, inp)
    ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    idx = msa.topk_select(ms, case.topk, plan.num_valid_pages)
    plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx)
    plan.check_errors()  # clean inputs: nothing to report
    bad_pq = inp["pq"].clone()
    bad_pq[5, 1, 3] = float("nan")
    plan.proxy_maxscore(bad_pq, inp["pk_pages"], inp["kv_indices"])
    with pytest.raises(msa.MsaError) as e:
        plan.check_errors()
    assert e.value.status == MSA_ERR_NONFINITE
    plain.proxy_maxscore(bad_pq, inp["pk_pages"], inp["kv_indices"])
    plain.check_errors()  # no scan without MSA_CHECKS
    bad_q = inp["q"].clone()
    bad_q[7, 2, 11] = float("nan")
    plan.sparse_attn(bad_q, inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx)
    with pytest.raises(msa.MsaError) as e:
        plan.check_errors()
    assert e.value.status == MSA_ERR_NONFINITE
    plan.check_errors()  # the word was cleared by the read
    bad_k = inp["k_pages"].clone()
    bad_k[int(inp["kv_indices"][1]), 1, 17, 5] = float("nan")  # a referenced page
    plan.sparse_attn(inp["q"], bad_k, inp["v_pages"], inp["kv_indices"], idx)
    with pytest.raises(msa.MsaError) as e:
        plan.check_errors()
    assert e.value.status == MSA_ERR_NONFINITE
