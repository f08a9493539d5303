"""FP8 (e4m3) K/V sparse prefill on the GPU against the oracle: msa_sparse_attn
with a prefill plan whose K/V pages hold e4m3 codes with one fp32 scale per
KV head (tolerance: max-abs 6e-2 and cosine >= 0.99 on out; lse within
1e-2; rows without a visible key exactly 0 / -inf)."""
import numpy as np
import pytest
import torch

from block_sparse_long_proxy_gb300 import synth
from oracle import msa_oracle as O
from tests.gpu_cases import O_ATOL_FP8, compare_out, irregular_idx, make_plan, random_idx, rows_of_tiles

pytestmark = pytest.mark.gpu

CASES = [
    synth.Case("S=256 G=4", [256], [256], 8, 2, 128, 2, 64, 2, kv_dtype="e4m3"),
    synth.Case("ragged varlen paged", [300, 77, 128, 129], [300, 1000, 128, 500], 8, 2, 128, 2, 64, 3,
               kv_dtype="e4m3", page_perm_seed=3, extra_pages=5),
    synth.Case("G=1", [256], [256], 2, 2, 128, 2, 64, 2, kv_dtype="e4m3"),
    synth.Case("G=3 odd group", [200], [333], 6, 2, 128, 2, 64, 2, kv_dtype="e4m3", page_perm_seed=1),
    synth.Case("topk above blocks", [640], [640], 4, 1, 128, 1, 64, 9, kv_dtype="e4m3"),
    synth.Case("topk 1 straddling tile", [128, 100], [200, 300], 2, 1, 128, 1, 64, 1, kv_dtype="e4m3"),
    synth.Case("empty query sequence mid-batch", [300, 0, 129], [300, 500, 129], 8, 2, 128, 2, 64, 3,
               kv_dtype="e4m3", page_perm_seed=6),
    synth.Case("topk 1024 (the maximum) over 16 blocks", [2048], [2048], 4, 1, 128, 1, 64, 1024, kv_dtype="e4m3",
               page_perm_seed=7),
    synth.Case("long 40-block rows topk 16", [5120], [5120], 8, 2, 128, 2, 64, 16, kv_dtype="e4m3",
               page_perm_seed=11),
]


def _run(case, inp, idx, dev):
    plan = make_plan(case, inp)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"],
                                torch.from_numpy(idx).to(dev), k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    torch.cuda.synchronize()
    plan.check_errors()
    return plan, out, lse


def _oracle(case, inp, idx, tile_ids=None):
    return O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                              inp["kv_indices"].cpu().numpy(), idx, case.qo_lens, case.kv_lens,
                              k_scale=inp["k_scale"].cpu().numpy(), v_scale=inp["v_scale"].cpu().numpy(),
                              tile_ids=tile_ids)


def _compare(out, lse, o_ref, lse_ref):
    compare_out(out, o_ref, O_ATOL_FP8)
    assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    assert np.abs(lse[fin] - lse_ref[fin]).max() <= 1e-2
    assert (out[np.isneginf(lse_ref)] == 0.0).all()


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_fp8_prefill_random_indexes(cuda_dev, case):
    inp = synth.make_inputs(case, device=cuda_dev)
    idx = random_idx(case, np.random.default_rng(5))
    _, out, lse = _run(case, inp, idx, cuda_dev)
    o_ref, lse_ref = _oracle(case, inp, idx)
    _compare(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref)


def test_fp8_prefill_irregular_indexes(cuda_dev):
    """Selections in random order, -1 entries anywhere, every fifth row
    empty (its query rows get out = 0, lse = -inf)."""
    case = synth.Case("shuffled and empty rows", [1024, 700, 300], [1024, 900, 300], 8, 2, 128, 2, 64, 6,
                      kv_dtype="e4m3", page_perm_seed=4)
    inp = synth.make_inputs(case, device=cuda_dev)
    idx = irregular_idx(case, np.random.default_rng(9))
    _, out, lse = _run(case, inp, idx, cuda_dev)
    o_ref, lse_ref = _oracle(case, inp, idx)
    assert np.isneginf(lse_ref).any()
    _compare(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref)


def test_fp8_prefill_two_calls(cuda_dev):
    """A second call with other selections on the same plan (the converted
    stages and Q tiles are rebuilt every call)."""
    case = CASES[1]
    inp = synth.make_inputs(case, device=cuda_dev)
    for seed in (1, 2):
        idx = random_idx(case, np.random.default_rng(seed))
        _, out, lse = _run(case, inp, idx, cuda_dev)
        o_ref, lse_ref = _oracle(case, inp, idx)
        _compare(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref)


def test_fp8_prefill_32k_sampled(cuda_dev):
    """The S=32768 prefill workload (32q/8kv heads, d=128, topk 16) with
    e4m3 K/V: the GPU's own proxy -> top-k -> FP8 attention; the oracle
    checks the first, last and some middle tiles on the GPU's indexes."""
    from block_sparse_long_proxy_gb300 import msa
    case = synth.prefill_32k()
    case.kv_dtype = "e4m3"
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = make_plan(case, inp)
    ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    idx_t = msa.topk_select(ms, case.topk, plan.num_valid_pages)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx_t,
                                k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    torch.cuda.synchronize()
    plan.check_errors()
    tiles = [0, 1, 77, 128, 200, 255]
    idx = idx_t.cpu().numpy()
    o_ref, lse_ref = _oracle(case, inp, idx, tile_ids=tiles)
    rows = rows_of_tiles(case, tiles)
    _compare(out.float().cpu().numpy()[rows], lse.cpu().numpy()[rows], o_ref[rows], lse_ref[rows])


def test_fp8_prefill_head_dim_64_unsupported(cuda_dev):
    from block_sparse_long_proxy_gb300 import msa
    case = synth.Case("fp8 d64", [256], [256], 4, 2, 64, 2, 32, 2, kv_dtype="e4m3")
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = make_plan(case, inp)
    idx = torch.from_numpy(random_idx(case, np.random.default_rng(0))).to(cuda_dev)
    with pytest.raises(msa.MsaError) as e:
        plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx,
                         k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    assert e.value.status == 2
