"""Several proxy heads per GQA group (Hp = 2 Hkv) on the GPU against the
oracle: every proxy head scores and selects its own blocks, and the Hq/Hp
query heads that use a proxy head attend over its blocks of their KV head
(forward bf16 and e4m3, decode, backward)."""
import numpy as np
import pytest
import torch

from block_sparse_long_proxy_gb300 import synth
from oracle import msa_oracle as O
from tests.gpu_cases import (MS_ATOL, O_ATOL_BF16, O_ATOL_FP8, check_indices_with_gap, compare_out, make_plan,
                             random_idx)

pytestmark = pytest.mark.gpu


def _ms_check(case, inp, ms):
    ref = O.proxy_max_score(synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]), inp["kv_indices"].cpu().numpy(),
                            case.qo_lens, case.kv_lens)
    got = ms.cpu().numpy()
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    fin = np.isfinite(ref)
    assert np.abs(got[fin] - ref[fin]).max() <= MS_ATOL
    return ref


def test_hp2_prefill_chain(cuda_dev):
    """proxy -> top-k -> attention with 16 proxy heads over 8 KV heads (32
    query heads: two per proxy head), S = 4096 and a ragged second
    sequence, paged: max_score, bit-exact top-k, end-to-end indices under
    the gap rule, and the output against the oracle on the GPU's indexes."""
    from block_sparse_long_proxy_gb300 import msa
    case = synth.Case("hp 16 / hkv 8", [4096, 300], [4096, 700], 32, 8, 128, 16, 64, 8, page_perm_seed=2)
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = make_plan(case, inp)
    ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    idx_t = msa.topk_select(ms, case.topk, plan.num_valid_pages)
    assert tuple(idx_t.shape) == (plan.n_tiles, 16, case.topk)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx_t)
    torch.cuda.synchronize()
    plan.check_errors()
    ms_ref = _ms_check(case, inp, ms)
    nvp = O.num_valid_pages(case.qo_lens, case.kv_lens)
    idx = idx_t.cpu().numpy()
    assert np.array_equal(idx, O.topk_select(ms.cpu().numpy(), case.topk, nvp))
    check_indices_with_gap(idx, ms_ref, nvp, case.topk, list(range(len(nvp))))
    # the proxy heads of one group do pick different blocks
    assert (idx[:, 0::2] != idx[:, 1::2]).any()
    o_ref, lse_ref = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                                        inp["kv_indices"].cpu().numpy(), idx, case.qo_lens, case.kv_lens)
    compare_out(out.float().cpu().numpy(), o_ref, O_ATOL_BF16)
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3


def test_hp2_fused_proxy_topk(cuda_dev):
    case = synth.Case("hp 4 / hkv 2 fused", [2048, 200], [2048, 900], 8, 2, 128, 4, 64, 6, page_perm_seed=3)
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = make_plan(case, inp)
    from block_sparse_long_proxy_gb300 import msa
    ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    sep = msa.topk_select(ms, case.topk, plan.num_valid_pages)
    fused = plan.proxy_topk(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    torch.cuda.synchronize()
    plan.check_errors()
    assert torch.equal(sep, fused)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_hp2_attention_random_indexes(cuda_dev, kv_dtype):
    case = synth.Case("hp 4 / hkv 2", [300, 77, 129], [300, 1000, 500], 8, 2, 128, 4, 64, 3, kv_dtype=kv_dtype,
                      page_perm_seed=3, extra_pages=2)
    inp = synth.make_inputs(case, device=cuda_dev)
    idx = random_idx(case, np.random.default_rng(7))
    plan = make_plan(case, inp)
    kw, okw = {}, {}
    if kv_dtype == "e4m3":
        kw = dict(k_scale=inp["k_scale"], v_scale=inp["v_scale"])
        okw = dict(k_scale=inp["k_scale"].cpu().numpy(), v_scale=inp["v_scale"].cpu().numpy())
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"],
                                torch.from_numpy(idx).to(cuda_dev), **kw)
    torch.cuda.synchronize()
    plan.check_errors()
    o_ref, lse_ref = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                                        inp["kv_indices"].cpu().numpy(), idx, case.qo_lens, case.kv_lens, **okw)
    compare_out(out.float().cpu().numpy(), o_ref, O_ATOL_FP8 if kv_dtype == "e4m3" else O_ATOL_BF16)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lse.cpu().numpy()), np.isneginf(lse_ref))
    assert np.abs(lse.cpu().numpy()[fin] - lse_ref[fin]).max() <= 1e-2


_LENS = [int(x) for x in np.random.default_rng(5).integers(1, 3000, size=20)]


@pytest.mark.parametrize("case", [
    synth.Case("decode hp 4 / hkv 2 (split rows)", [1] * 5, [700, 129, 128, 1, 5000], 16, 2, 128, 4, 64, 4,
               kv_dtype="e4m3", page_perm_seed=2, extra_pages=3),
    synth.Case("decode hp 16 / hkv 8 (row per CTA)", [1] * 20, _LENS, 64, 8, 128, 16, 64, 8, kv_dtype="e4m3",
               page_perm_seed=9),
], ids=lambda c: c.name)
def test_hp2_fp8_decode(cuda_dev, case):
    """Both decode kernels: rows are (sequence, proxy head)."""
    from block_sparse_long_proxy_gb300 import msa
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = make_plan(case, inp)
    ms = plan.proxy_maxscore(inp["pq"], inp["pk_pages"], inp["kv_indices"])
    idx_t = msa.topk_select(ms, case.topk, plan.num_valid_pages)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx_t,
                                k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    torch.cuda.synchronize()
    plan.check_errors()
    _ms_check(case, inp, ms)
    idx = idx_t.cpu().numpy()
    o_ref, lse_ref = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                                        inp["kv_indices"].cpu().numpy(), idx, case.qo_lens, case.kv_lens,
                                        k_scale=inp["k_scale"].cpu().numpy(), v_scale=inp["v_scale"].cpu().numpy())
    compare_out(out.float().cpu().numpy(), o_ref, O_ATOL_FP8)
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-2


@pytest.mark.parametrize("case,w", [
    (synth.Case("bwd hp 4 / hkv 2 ragged", [300, 77, 129], [300, 500, 129], 8, 2, 128, 4, 64, 3,
                page_perm_seed=3, extra_pages=2), 0.7),
    (synth.Case("bwd hp 8 / hkv 2, one head per proxy head", [512], [512], 8, 2, 128, 8, 64, 2,
                page_perm_seed=4), 1.0),
], ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_hp2_backward(cuda_dev, case, w):
    """All five gradients: dK / dV of a KV head sum the selections of all of
    its proxy heads; dpq of a proxy head distils its own query heads."""
    inp = synth.make_inputs(case, device=cuda_dev, with_dout=True)
    idx = random_idx(case, np.random.default_rng(11))
    plan = make_plan(case, inp)
    idx_t = torch.from_numpy(idx).to(cuda_dev)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx_t)
    grads = plan.sparse_attn_bwd(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx_t, out, lse,
                                 inp["dout"], inp["pq"], inp["pk_pages"], kl_weight=w)
    torch.cuda.synchronize()
    plan.check_errors()
    ref = O.sparse_attention_bwd(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                                 inp["kv_indices"].cpu().numpy(), idx, case.qo_lens, case.kv_lens,
                                 synth.bits(inp["dout"]), synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]),
                                 kl_weight=w)
    for name in ("dq", "dpq", "dk", "dv", "dpk"):
        g = grads[name].cpu().numpy()
        assert np.isfinite(g).all(), name
        compare_out(g, ref[name], O_ATOL_BF16, name)
