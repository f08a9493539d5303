"""msa_proxy_maxscore on the GPU against the oracle.

Tolerance: |gpu - oracle| <= 1e-3 on every finite entry (the parity bound
for proxy scores, equal to the score-gap rule of the selections; the fp32
accumulation of exact bf16 products is ~1e-6 off in practice) and an
identical -inf pattern."""
import numpy as np
import pytest
import torch

from block_sparse_long_proxy_gb300 import synth
from oracle import msa_oracle as O

pytestmark = pytest.mark.gpu
ATOL = 1e-3


def _run(case, dev, tile_ids=None):
    from block_sparse_long_proxy_gb300 import msa
    inp = synth.make_inputs(case, device=dev)
    plan = msa.Plan(case.qo_lens, case.kv_lens, case.hq, case.hkv, case.hp, case.d, case.dp, case.topk,
                    num_pages=inp["k_pages"].shape[0])
    ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    torch.cuda.synchronize()
    plan.check_errors()
    got = ms.cpu().numpy()
    ref = O.proxy_max_score(synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]), inp["kv_indices"].cpu().numpy(),
                            case.qo_lens, case.kv_lens, tile_ids=tile_ids)
    if tile_ids is not None:
        got, ref = got[tile_ids], ref[tile_ids]
    assert got.shape == ref.shape
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    fin = np.isfinite(ref)
    err = np.abs(got[fin] - ref[fin]).max() if fin.any() else 0.0
    assert err <= ATOL, err
    return err


@pytest.mark.parametrize("case", [
    synth.tiny(),
    synth.Case("ragged offsets dp64", [200, 77, 300], [1000, 300, 300], 4, 4, 64, 4, 64, 4, page_perm_seed=3,
               extra_pages=3),
    synth.Case("ragged offsets dp32", [129, 1], [129, 77], 2, 2, 64, 2, 32, 4, page_perm_seed=5),
    synth.Case("12 proxy heads (two head groups)", [384], [500], 12, 12, 64, 12, 64, 4, page_perm_seed=7),
    synth.Case("long tile rows, 40 blocks", [5000], [5000], 8, 8, 64, 8, 64, 4),
], ids=lambda c: c.name)
def test_proxy_prefill_small(cuda_dev, case):
    _run(case, cuda_dev)


@pytest.mark.parametrize("case", [
    synth.Case("decode dp64", [1] * 5, [700, 129, 128, 1, 5000], 16, 8, 128, 8, 64, 4, page_perm_seed=2),
    synth.Case("decode dp32 3 heads", [1] * 3, [300, 4096, 77], 6, 3, 64, 3, 32, 4, page_perm_seed=4),
], ids=lambda c: c.name)
def test_proxy_decode_small(cuda_dev, case):
    _run(case, cuda_dev)


def test_proxy_prefill_32k_sampled(cuda_dev):
    case = synth.prefill_32k()
    _run(case, cuda_dev, tile_ids=[0, 1, 31, 32, 33, 100, 200, 254, 255])


def test_proxy_decode_full_size_sampled(cuda_dev):
    case = synth.paged_decode()
    _run(case, cuda_dev, tile_ids=[0, 7, 31])


def _run_fp8(case, dev, tile_ids=None):
    """msa_proxy_maxscore_fp8 (e4m3 proxy K with one scale) against the
    oracle's R11 route on the same codes."""
    from block_sparse_long_proxy_gb300 import msa
    inp = synth.make_inputs(case, device=dev)
    plan = msa.Plan(case.qo_lens, case.kv_lens, case.hq, case.hkv, case.hp, case.d, case.dp, case.topk,
                    num_pages=inp["k_pages"].shape[0], kv_dtype=case.kv_dtype)
    ms = plan.proxy_maxscore_fp8(inp["pq"], inp["pk_pages_e4m3"], inp["pk_scale"], inp["kv_indices"])
    torch.cuda.synchronize()
    plan.check_errors()
    got = ms.cpu().numpy()
    ref = O.proxy_max_score(synth.bits(inp["pq"]), synth.bits(inp["pk_pages_e4m3"]), inp["kv_indices"].cpu().numpy(),
                            case.qo_lens, case.kv_lens, tile_ids=tile_ids, pk_scale=float(inp["pk_scale"][0]))
    if tile_ids is not None:
        got, ref = got[tile_ids], ref[tile_ids]
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    fin = np.isfinite(ref)
    err = np.abs(got[fin] - ref[fin]).max() if fin.any() else 0.0
    assert err <= ATOL, err
    return err


@pytest.mark.parametrize("case", [
    synth.Case("fp8 proxy decode ragged", [1] * 5, [700, 129, 128, 1, 5000], 16, 8, 128, 8, 64, 4,
               kv_dtype="e4m3", page_perm_seed=2, extra_pages=3),
    synth.Case("fp8 proxy decode 3 heads", [1] * 3, [300, 4096, 77], 6, 3, 128, 3, 64, 4, kv_dtype="e4m3",
               page_perm_seed=4),
], ids=lambda c: c.name)
def test_proxy_decode_fp8_small(cuda_dev, case):
    _run_fp8(case, cuda_dev)


def test_proxy_decode_fp8_full_size_sampled(cuda_dev):
    _run_fp8(synth.paged_decode(), cuda_dev, tile_ids=[0, 7, 31])


def test_proxy_fp8_rejects_prefill_plans(cuda_dev):
    from block_sparse_long_proxy_gb300 import msa
    case = synth.Case("fp8 proxy prefill", [256], [256], 4, 2, 128, 2, 64, 2, kv_dtype="e4m3")
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = msa.Plan(case.qo_lens, case.kv_lens, case.hq, case.hkv, case.hp, case.d, case.dp, case.topk,
                    num_pages=inp["k_pages"].shape[0], kv_dtype=case.kv_dtype)
    with pytest.raises(msa.MsaError) as e:
        plan.proxy_maxscore_fp8(inp["pq"], inp["pk_pages_e4m3"], inp["pk_scale"], inp["kv_indices"])
    assert e.value.status == 2


def _run_nvfp4(case, dev, tile_ids=None):
    """msa_proxy_maxscore_nvfp4 (the FP4 block-score indexer) against the
    oracle's R12 route on the same codes and scales; the top-k of the GPU's
    scores equals the oracle's top-k of them (bit-exact)."""
    from block_sparse_long_proxy_gb300 import msa
    inp = synth.make_inputs(case, device=dev)
    plan = msa.Plan(case.qo_lens, case.kv_lens, case.hq, case.hkv, case.hp, case.d, case.dp, case.topk,
                    num_pages=inp["k_pages"].shape[0], kv_dtype=case.kv_dtype)
    ms = plan.proxy_maxscore_nvfp4(inp["pq"], inp["pk_fp4_codes"], inp["pk_fp4_scales"], inp["pk_fp4_global"],
                                   inp["kv_indices"])
    idx = msa.topk_select(ms, case.topk, plan.num_valid_pages)
    torch.cuda.synchronize()
    plan.check_errors()
    got = ms.cpu().numpy()
    ref = O.proxy_max_score(synth.bits(inp["pq"]), inp["pk_fp4_codes"].cpu().numpy(), inp["kv_indices"].cpu().numpy(),
                            case.qo_lens, case.kv_lens, tile_ids=tile_ids,
                            pk_nvfp4=(synth.bits(inp["pk_fp4_scales"]), float(inp["pk_fp4_global"][0])))
    nvp = O.num_valid_pages(case.qo_lens, case.kv_lens)
    ids = list(range(len(nvp))) if tile_ids is None else tile_ids
    assert np.array_equal(idx.cpu().numpy()[ids], O.topk_select(got[ids], case.topk, nvp[ids]))
    got, ref = got[ids], ref[ids]
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    fin = np.isfinite(ref)
    err = np.abs(got[fin] - ref[fin]).max() if fin.any() else 0.0
    assert err <= ATOL, err
    return err


@pytest.mark.parametrize("case", [
    synth.Case("nvfp4 proxy decode ragged", [1] * 5, [700, 129, 128, 1, 5000], 16, 8, 128, 8, 64, 4,
               kv_dtype="e4m3", page_perm_seed=2, extra_pages=3),
    synth.Case("nvfp4 proxy decode 3 heads", [1] * 3, [300, 4096, 77], 6, 3, 128, 3, 64, 4, kv_dtype="e4m3",
               page_perm_seed=4),
    synth.Case("nvfp4 proxy decode 70 sequences", [1] * 70, [int(x) for x in np.arange(70) * 211 + 1], 16, 8, 128, 8,
               64, 6, kv_dtype="e4m3", page_perm_seed=5),
], ids=lambda c: c.name)
def test_proxy_decode_nvfp4_small(cuda_dev, case):
    _run_nvfp4(case, cuda_dev)


def test_proxy_decode_nvfp4_full_size_sampled(cuda_dev):
    _run_nvfp4(synth.paged_decode(), cuda_dev, tile_ids=[0, 7, 31])


def test_proxy_nvfp4_rejects_prefill_plans(cuda_dev):
    from block_sparse_long_proxy_gb300 import msa
    case = synth.Case("nvfp4 proxy prefill", [256], [256], 4, 2, 128, 2, 64, 2, kv_dtype="e4m3")
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = msa.Plan(case.qo_lens, case.kv_lens, case.hq, case.hkv, case.hp, case.d, case.dp, case.topk,
                    num_pages=inp["k_pages"].shape[0], kv_dtype=case.kv_dtype)
    with pytest.raises(msa.MsaError) as e:
        plan.proxy_maxscore_nvfp4(inp["pq"], inp["pk_fp4_codes"], inp["pk_fp4_scales"], inp["pk_fp4_global"],
                                  inp["kv_indices"])
    assert e.value.status == 2
