"""FP8 (e4m3) paged sparse decode on the GPU against the oracle
(tolerance: max-abs 6e-2 and cosine >= 0.99 on out; lse within 1e-2)."""
import numpy as np
import pytest
import torch

from block_sparse_long_proxy_gb300 import synth
from oracle import msa_oracle as O
from tests.gpu_cases import O_ATOL_FP8, O_ATOL_BF16, compare_out, random_idx, make_plan, check_indices_with_gap

pytestmark = pytest.mark.gpu

CASES = [
    synth.Case("G=8 ragged kv", [1] * 5, [700, 129, 128, 1, 5000], 16, 2, 128, 2, 64, 4, kv_dtype="e4m3",
               page_perm_seed=2, extra_pages=3),
    synth.Case("G=4 padded heads", [1] * 3, [4096, 300, 1000], 8, 2, 128, 2, 64, 16, kv_dtype="e4m3",
               page_perm_seed=4),
    synth.Case("G=16 two n-tiles", [1] * 2, [2048, 777], 32, 2, 128, 2, 64, 5, kv_dtype="e4m3", page_perm_seed=6),
    synth.Case("G=1", [1] * 4, [1024, 200, 3000, 129], 3, 3, 128, 3, 32, 3, kv_dtype="e4m3", page_perm_seed=8),
    synth.Case("topk above blocks", [1] * 2, [256, 1000], 8, 1, 128, 1, 64, 12, kv_dtype="e4m3"),
    # topk at the largest value a plan accepts, over a 1094-block sequence (and a 24-block one)
    synth.Case("topk 1024 (the maximum)", [1] * 2, [140000, 3000], 8, 1, 128, 1, 64, 1024, kv_dtype="e4m3",
               page_perm_seed=12),
]


def _check(case, dev, idx=None):
    inp = synth.make_inputs(case, device=dev)
    if idx is None:
        idx = random_idx(case, np.random.default_rng(3))
    plan = make_plan(case, inp)
    kw = {}
    if case.kv_dtype == "e4m3":
        kw = dict(k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"],
                                torch.from_numpy(idx).to(dev), **kw)
    torch.cuda.synchronize()
    plan.check_errors()
    okw = {}
    if case.kv_dtype == "e4m3":
        okw = dict(k_scale=inp["k_scale"].cpu().numpy(), v_scale=inp["v_scale"].cpu().numpy())
    o_ref, lse_ref = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                                        inp["kv_indices"].cpu().numpy(), idx, case.qo_lens, case.kv_lens, **okw)
    compare_out(out.float().cpu().numpy(), o_ref, O_ATOL_FP8 if case.kv_dtype == "e4m3" else O_ATOL_BF16)
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-2
    return plan, inp


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_fp8_decode_random_indexes(cuda_dev, case):
    _check(case, cuda_dev)


# batches with at least as many (sequence, group) rows as SMs take the
# warp-streaming kernel (one CTA per row); these cover it at sizes the
# oracle runs in seconds: ragged kv, padded slots (topk above a sequence's
# blocks), G = 8 and G = 4, partial last pages.
_LENS = [int(x) for x in np.random.default_rng(21).integers(1, 3000, size=40)]
WS_CASES = [
    synth.Case("rows>=SMs G=8 ragged", [1] * 20, _LENS[:20], 64, 8, 128, 8, 64, 8, kv_dtype="e4m3",
               page_perm_seed=9, extra_pages=5),
    synth.Case("rows>=SMs G=4 padded slots", [1] * 40, _LENS, 16, 4, 128, 4, 64, 12, kv_dtype="e4m3",
               page_perm_seed=10),
    # topk above the warp-streaming kernel's limit: the ring kernel, one CTA per row
    synth.Case("rows>=SMs topk 80", [1] * 20, _LENS[:20], 64, 8, 128, 8, 64, 80, kv_dtype="e4m3",
               page_perm_seed=11),
]


@pytest.mark.parametrize("case", WS_CASES, ids=lambda c: c.name)
def test_fp8_decode_one_cta_per_row(cuda_dev, case):
    assert len(case.qo_lens) * case.hkv >= torch.cuda.get_device_properties(cuda_dev).multi_processor_count
    _check(case, cuda_dev)


def test_fp8_decode_two_calls_reuse_workspace(cuda_dev):
    """The split-K partials live in the plan; a second call with other
    indexes overwrites them completely."""
    case = CASES[0]
    _check(case, cuda_dev, random_idx(case, np.random.default_rng(11)))
    _check(case, cuda_dev, random_idx(case, np.random.default_rng(12)))


def test_bf16_decode_batch(cuda_dev):
    """A decode batch with bf16 K/V runs the prefill kernel (one-row tiles)."""
    _check(synth.Case("bf16 decode", [1] * 4, [900, 128, 129, 4000], 16, 2, 128, 2, 64, 4, page_perm_seed=5),
           cuda_dev)


def test_paged_decode_full_size_sampled(cuda_dev):
    """32 sequences x 131072 keys, 64/8 heads, topk 16: the whole chain on
    the GPU, the oracle on sampled sequences (indices with the gap rule,
    attention on the GPU's indices)."""
    from block_sparse_long_proxy_gb300 import msa
    case = synth.paged_decode()
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = make_plan(case, inp)
    ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    idx = msa.topk_select(ms, case.topk, plan.num_valid_pages)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx,
                                k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    torch.cuda.synchronize()
    plan.check_errors()
    ids = [0, 5, 17, 31]
    table = inp["kv_indices"].cpu().numpy()
    nvp = O.num_valid_pages(case.qo_lens, case.kv_lens)
    ms_ref = O.proxy_max_score(synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]), table, case.qo_lens,
                               case.kv_lens, tile_ids=ids)
    idx_g = idx.cpu().numpy()
    assert np.array_equal(idx_g[ids], O.topk_select(ms.cpu().numpy()[ids], case.topk, nvp[ids]))
    check_indices_with_gap(idx_g, ms_ref, nvp, case.topk, ids)
    o_ref, _ = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]), table,
                                  idx_g, case.qo_lens, case.kv_lens, k_scale=inp["k_scale"].cpu().numpy(),
                                  v_scale=inp["v_scale"].cpu().numpy(), tile_ids=ids)
    compare_out(out[ids].float().cpu().numpy(), o_ref[ids], O_ATOL_FP8)
