"""msa_sparse_attn (bf16 prefill) on the GPU against the oracle, and the
whole three-stage path end to end."""
import numpy as np
import pytest
import torch

from block_sparse_long_proxy_gb300 import synth
from oracle import msa_oracle as O
from tests.gpu_cases import (O_ATOL_BF16, compare_out, random_idx, irregular_idx, make_plan, rows_of_tiles,
                             check_indices_with_gap, MS_ATOL)

pytestmark = pytest.mark.gpu

SMALL = [
    synth.tiny(),
    synth.Case("ragged varlen d128 paged", [300, 77, 128, 129], [300, 1000, 128, 500], 8, 2, 128, 2, 64, 3,
               page_perm_seed=3, extra_pages=5),
    synth.Case("G=1 single head per CTA", [256], [256], 2, 2, 128, 2, 64, 2),
    synth.Case("G=3 odd group", [200], [333], 6, 2, 64, 2, 32, 2, page_perm_seed=1),
    synth.Case("topk above blocks", [640], [640], 4, 1, 128, 1, 64, 9),
    synth.Case("topk 1 straddling tile", [128, 100], [200, 300], 2, 1, 64, 1, 32, 1),
    synth.Case("long 40-block rows topk 16", [5120], [5120], 8, 2, 128, 2, 64, 16, page_perm_seed=11),
    # a sequence with keys but no query rows: no tiles, its pages still in the page table
    synth.Case("empty query sequence mid-batch", [300, 0, 129], [300, 500, 129], 8, 2, 128, 2, 64, 3,
               page_perm_seed=6),
    # topk at the largest value a plan accepts; every tile takes all of its blocks
    synth.Case("topk 1024 (the maximum) over 16 blocks", [2048], [2048], 4, 1, 128, 1, 64, 1024, page_perm_seed=7),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c.name)
def test_sparse_attn_random_indexes(cuda_dev, case):
    inp = synth.make_inputs(case, device=cuda_dev)
    idx = random_idx(case, np.random.default_rng(5))
    plan = make_plan(case, inp)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"],
                                torch.from_numpy(idx).to(cuda_dev))
    torch.cuda.synchronize()
    plan.check_errors()
    o_ref, lse_ref = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                                        inp["kv_indices"].cpu().numpy(), idx, case.qo_lens, case.kv_lens)
    compare_out(out.float().cpu().numpy(), o_ref, O_ATOL_BF16)
    lg = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    assert np.abs(lg[fin] - lse_ref[fin]).max() <= 1e-3


IRREGULAR = [
    # more selected blocks than one 32-lane pass of the unit-list builder
    synth.Case("topk 36 over 40 blocks", [5120], [5120], 2, 1, 128, 1, 64, 36, page_perm_seed=2),
    synth.Case("shuffled and empty rows", [1024, 700, 300], [1024, 900, 300], 8, 2, 128, 2, 64, 6,
               page_perm_seed=4),
]


@pytest.mark.parametrize("case", IRREGULAR, ids=lambda c: c.name)
def test_sparse_attn_irregular_indexes(cuda_dev, case):
    inp = synth.make_inputs(case, device=cuda_dev)
    idx = irregular_idx(case, np.random.default_rng(9))
    plan = make_plan(case, inp)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"],
                                torch.from_numpy(idx).to(cuda_dev))
    torch.cuda.synchronize()
    plan.check_errors()
    o_ref, lse_ref = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                                        inp["kv_indices"].cpu().numpy(), idx, case.qo_lens, case.kv_lens)
    compare_out(out.float().cpu().numpy(), o_ref, O_ATOL_BF16)
    lg = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(lse_ref))
    assert np.isneginf(lse_ref).any()  # the empty rows are in the case
    fin = np.isfinite(lse_ref)
    assert np.abs(lg[fin] - lse_ref[fin]).max() <= 1e-3


@pytest.mark.parametrize("case", [synth.tiny(),
                                  synth.Case("varlen planted small", [1024, 2048, 640], [1024, 2048, 900],
                                             8, 2, 128, 2, 64, 4, page_perm_seed=1, planted=True),
                                  synth.Case("empty query sequence mid-batch, chain", [300, 0, 129],
                                             [300, 500, 129], 8, 2, 128, 2, 64, 3, page_perm_seed=6)],
                         ids=lambda c: c.name)
def test_end_to_end_small(cuda_dev, case):
    """proxy -> top-k -> attention, every stage against the oracle: max_score
    within 1e-3, indices bit-exact on the GPU's own max_score and equal to
    the oracle's chain except at score gaps below 1e-3, attention on the
    GPU's indices within the bf16 tolerance."""
    from block_sparse_long_proxy_gb300 import msa
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = make_plan(case, inp)
    ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    idx = msa.topk_select(ms, case.topk, plan.num_valid_pages)
    out, _ = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx)
    torch.cuda.synchronize()
    plan.check_errors()
    nvp = O.num_valid_pages(case.qo_lens, case.kv_lens)
    ms_g = ms.cpu().numpy()
    ms_ref = O.proxy_max_score(synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]), inp["kv_indices"].cpu().numpy(),
                               case.qo_lens, case.kv_lens)
    fin = np.isfinite(ms_ref)
    assert np.abs(ms_g[fin] - ms_ref[fin]).max() <= MS_ATOL
    idx_g = idx.cpu().numpy()
    assert np.array_equal(idx_g, O.topk_select(ms_g, case.topk, nvp))
    check_indices_with_gap(idx_g, ms_ref, nvp, case.topk, np.arange(len(nvp)))
    o_ref, _ = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                                  inp["kv_indices"].cpu().numpy(), idx_g, case.qo_lens, case.kv_lens)
    compare_out(out.float().cpu().numpy(), o_ref, O_ATOL_BF16)


def test_bad_page_id_raises_device_check(cuda_dev):
    """An out-of-range page id is caught by the kernels' own bounds check:
    the block is read from page 0 instead and msa_check_errors reports
    MSA_ERR_DEVICE_CHECK."""
    from block_sparse_long_proxy_gb300 import msa
    case = synth.Case("bad page", [256], [256], 2, 1, 64, 1, 32, 2)
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = make_plan(case, inp)
    table = inp["kv_indices"].clone()
    table[1] = 10 ** 6
    idx = torch.tensor([[[0, -1]], [[0, 1]]], dtype=torch.int32, device=cuda_dev)
    plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], table, idx)
    with pytest.raises(msa.MsaError) as e:
        plan.check_errors()
    assert e.value.status == 6
    plan.check_errors()   # the word was cleared


def _full_size(case, cuda_dev, tile_ids):
    from block_sparse_long_proxy_gb300 import msa
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = make_plan(case, inp)
    ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    idx = msa.topk_select(ms, case.topk, plan.num_valid_pages)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx)
    torch.cuda.synchronize()
    plan.check_errors()
    nvp = O.num_valid_pages(case.qo_lens, case.kv_lens)
    table = inp["kv_indices"].cpu().numpy()
    ms_ref = O.proxy_max_score(synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]), table, case.qo_lens,
                               case.kv_lens, tile_ids=tile_ids)
    ms_g = ms.cpu().numpy()
    fin = np.isfinite(ms_ref[tile_ids])
    assert np.abs(ms_g[tile_ids][fin] - ms_ref[tile_ids][fin]).max() <= MS_ATOL
    idx_g = idx.cpu().numpy()
    assert np.array_equal(idx_g[tile_ids], O.topk_select(ms_g[tile_ids], case.topk, nvp[tile_ids]))
    check_indices_with_gap(idx_g, ms_ref, nvp, case.topk, tile_ids)
    o_ref, lse_ref = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                                        table, idx_g, case.qo_lens, case.kv_lens, tile_ids=tile_ids)
    rows = rows_of_tiles(case, tile_ids)
    compare_out(out[torch.from_numpy(rows).to(cuda_dev)].float().cpu().numpy(), o_ref[rows], O_ATOL_BF16)
    assert np.abs(lse[torch.from_numpy(rows).to(cuda_dev)].cpu().numpy() - lse_ref[rows]).max() <= 1e-3


def test_prefill_32k_sampled(cuda_dev):
    _full_size(synth.prefill_32k(), cuda_dev, [0, 1, 15, 16, 100, 200, 255])


def test_varlen_paged_sampled(cuda_dev):
    case = synth.varlen_paged()
    # first/last tiles of each sequence plus a few inside
    tl = O.tiles_of(case.qo_lens, case.kv_lens)
    starts = [i for i, t in enumerate(tl) if i == 0 or tl[i - 1].seq != t.seq]
    ids = sorted(set(starts + [s + 1 for s in starts] + [len(tl) - 1, len(tl) - 2, 700, 1100]))
    _full_size(case, cuda_dev, ids)


def test_training_64k_forward_sampled(cuda_dev):
    _full_size(synth.training_64k(), cuda_dev, [0, 3, 300, 511])
