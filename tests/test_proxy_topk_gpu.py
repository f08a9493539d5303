"""msa_proxy_topk (the proxy pass with the top-k selection fused in) on the
GPU: equal to msa_proxy_maxscore + msa_topk_select, bit-exact against the
oracle's selection over the same scores, and within the score-gap rule of
the oracle's own chain."""
import numpy as np
import pytest
import torch

from block_sparse_long_proxy_gb300 import synth
from oracle import msa_oracle as O
from tests.gpu_cases import MS_ATOL, check_indices_with_gap, make_plan

pytestmark = pytest.mark.gpu

CASES = [
    synth.tiny(),
    synth.Case("ragged varlen", [300, 77, 128, 129], [300, 1000, 128, 500], 8, 2, 128, 2, 64, 3,
               page_perm_seed=3, extra_pages=5),
    synth.Case("40-block rows, two chunks", [5120], [5120], 8, 2, 128, 2, 64, 16, page_perm_seed=11),
    synth.Case("topk 32 over 100 blocks", [2048], [12800], 4, 2, 64, 2, 32, 32, page_perm_seed=2),
    synth.Case("topk 1", [640], [4500], 4, 2, 64, 2, 32, 1),
    synth.Case("16 proxy heads, two head groups", [1024], [5000], 16, 16, 64, 16, 64, 8),
    synth.Case("empty query sequence mid-batch", [300, 0, 129], [300, 500, 129], 8, 2, 128, 2, 64, 3,
               page_perm_seed=6),
]


def _fused(plan, inp):
    ms = torch.empty((plan.n_tiles, plan.hp, plan.max_blocks), dtype=torch.float32, device=inp["pq"].device)
    idx = plan.proxy_topk(inp["pq"], inp["pk_pages"], inp["kv_indices"], max_score=ms)
    torch.cuda.synchronize()
    plan.check_errors()
    return ms, idx


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_fused_equals_separate_calls(cuda_dev, case):
    from block_sparse_long_proxy_gb300 import msa
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = make_plan(case, inp)
    ms, idx = _fused(plan, inp)
    ms2 = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    idx2 = msa.topk_select(ms2, case.topk, plan.num_valid_pages)
    torch.cuda.synchronize()
    assert torch.equal(ms, ms2)
    assert torch.equal(idx, idx2)
    nvp = O.num_valid_pages(case.qo_lens, case.kv_lens)
    assert np.array_equal(idx.cpu().numpy(), O.topk_select(ms.cpu().numpy(), case.topk, nvp))
    # repeated launches on one plan: the row counters reset themselves
    for _ in range(2):
        _, again = _fused(plan, inp)
        assert torch.equal(again, idx)


def test_fused_against_oracle_chain(cuda_dev):
    case = CASES[2]
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = make_plan(case, inp)
    ms, idx = _fused(plan, inp)
    nvp = O.num_valid_pages(case.qo_lens, case.kv_lens)
    ms_ref = O.proxy_max_score(synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]), inp["kv_indices"].cpu().numpy(),
                               case.qo_lens, case.kv_lens)
    fin = np.isfinite(ms_ref)
    assert np.abs(ms.cpu().numpy()[fin] - ms_ref[fin]).max() <= MS_ATOL
    check_indices_with_gap(idx.cpu().numpy(), ms_ref, nvp, case.topk, np.arange(len(nvp)))


def test_fused_ties_across_chunks(cuda_dev):
    """pq = 0: every visible block scores 0, so each row takes the lowest
    topk-1 blocks below the diagonal, wherever their chunk sits, plus the
    diagonal."""
    case = synth.Case("all-equal scores", [4096], [9000], 4, 2, 64, 2, 32, 12)
    inp = synth.make_inputs(case, device=cuda_dev)
    inp["pq"].zero_()
    plan = make_plan(case, inp)
    ms, idx = _fused(plan, inp)
    nvp = O.num_valid_pages(case.qo_lens, case.kv_lens)
    got = idx.cpu().numpy()
    assert np.array_equal(got, O.topk_select(ms.cpu().numpy(), case.topk, nvp))
    for t, n in enumerate(nvp):
        want = list(range(min(case.topk - 1, n - 1))) + [n - 1] if case.topk < n else list(range(n))
        want += [-1] * (case.topk - len(want))
        assert (got[t] == np.array(want)).all()


def test_fused_unsupported_configs(cuda_dev):
    from block_sparse_long_proxy_gb300 import msa
    big = synth.Case("topk 33", [1024], [9000], 4, 2, 64, 2, 32, 33)
    inp = synth.make_inputs(big, device=cuda_dev)
    with pytest.raises(msa.MsaError):
        make_plan(big, inp).proxy_topk(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    dec = synth.Case("decode", [1, 1], [700, 300], 4, 2, 64, 2, 32, 4)
    inp = synth.make_inputs(dec, device=cuda_dev)
    with pytest.raises(msa.MsaError):
        make_plan(dec, inp).proxy_topk(inp["pq"], inp["pk_pages"], inp["kv_indices"])
