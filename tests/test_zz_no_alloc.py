"""The allocation-free FP8 decode entry point (msa_sparse_decode_noalloc).

Callers that cannot allocate device memory while they decode (a server whose
memory pool owns the whole GPU, a latency-bound loop that cannot take
cudaMalloc's implicit synchronisation) cannot build a plan, so they use this
call: its scratch is a fixed array inside libmsa.  Its output must match the
planned entry point (msa_sparse_attn) on the same inputs, call after call,
even though every call reuses the same scratch.  This file is collected last
so that a run stopping at the first failure has run every other test."""
import numpy as np
import pytest
import torch

from block_sparse_long_proxy_gb300 import synth
from tests.gpu_cases import O_ATOL_FP8, make_plan, random_idx

pytestmark = pytest.mark.gpu


def _batch_arrays(case, dev):
    lens = torch.tensor(case.kv_lens, dtype=torch.int32, device=dev)
    nb = [(k + 127) // 128 for k in case.kv_lens]
    indptr = torch.tensor(np.concatenate([[0], np.cumsum(nb)]), dtype=torch.int32, device=dev)
    return lens, indptr


@pytest.mark.parametrize("case", [
    synth.Case("G=8 ragged", [1] * 6, [700, 129, 128, 1, 5000, 300], 16, 2, 128, 2, 64, 4, kv_dtype="e4m3",
               page_perm_seed=2, extra_pages=3),
    synth.Case("G=16", [1] * 3, [2048, 777, 4096], 32, 2, 128, 2, 64, 6, kv_dtype="e4m3", page_perm_seed=6),
    synth.Case("32 x 16384, 64/8 heads, topk 16", [1] * 32, [16384] * 32, 64, 8, 128, 8, 64, 16, kv_dtype="e4m3",
               page_perm_seed=1),
], ids=lambda c: c.name)
def test_noalloc_matches_planned_decode_two_calls(cuda_dev, case):
    from block_sparse_long_proxy_gb300 import msa
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = make_plan(case, inp)
    lens, indptr = _batch_arrays(case, cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    for call in range(2):
        idx = torch.from_numpy(random_idx(case, np.random.default_rng(100 + call))).to(cuda_dev)
        ref, ref_lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx,
                                        k_scale=inp["k_scale"], v_scale=inp["v_scale"])
        out = torch.full_like(inp["q"], float("nan"))
        lse = torch.full((case.total_q, case.hq), float("nan"), dtype=torch.float32, device=cuda_dev)
        msa.sparse_decode_noalloc(inp["q"], inp["k_pages"], inp["v_pages"], lens, indptr, inp["kv_indices"], idx,
                                  inp["k_scale"], inp["v_scale"], out=out, lse=lse, err_word=err)
        torch.cuda.synchronize()
        plan.check_errors()
        assert int(err.item()) == 0
        diff = (out.float() - ref.float()).abs().max().item()
        assert diff <= O_ATOL_FP8, (call, diff)
        assert (lse - ref_lse).abs().max().item() <= 1e-3


def test_noalloc_rejects_oversized_batch(cuda_dev):
    """batch * num_qo_heads * topk above the static scratch's capacity is
    refused on the host before any work is enqueued."""
    from block_sparse_long_proxy_gb300 import msa
    b, hq, hkv, topk = 64, 64, 8, 16          # 65536 > 47,639 partial rows
    q = torch.zeros((b, hq, 128), dtype=torch.bfloat16, device=cuda_dev)
    kp = torch.zeros((8, hkv, 128, 128), dtype=torch.float8_e4m3fn, device=cuda_dev)
    lens = torch.full((b,), 128, dtype=torch.int32, device=cuda_dev)
    indptr = torch.arange(b + 1, dtype=torch.int32, device=cuda_dev)
    table = torch.zeros((b,), dtype=torch.int32, device=cuda_dev)
    idx = torch.zeros((b, hkv, topk), dtype=torch.int32, device=cuda_dev)
    sc = torch.ones(hkv, dtype=torch.float32, device=cuda_dev)
    with pytest.raises(msa.MsaError) as e:
        msa.sparse_decode_noalloc(q, kp, kp, lens, indptr, table, idx, sc, sc)
    assert e.value.status == 1 and "static scratch" in str(e.value)


def test_noalloc_capacity_boundary(cuda_dev):
    """The capacity is 47,639 partial rows (batch * num_qo_heads * topk) at
    head_dim 128.  47,639 is prime, so the largest product a valid shape can
    reach is 47,637 = 67 * 9 * 79: it runs and matches the planned decode;
    47,640 = 40 * 3 * 397 is refused."""
    from block_sparse_long_proxy_gb300 import msa
    case = synth.Case("67 x 12800, 9/1 heads, topk 79", [1] * 67, [12800] * 67, 9, 1, 128, 1, 64, 79,
                      kv_dtype="e4m3", page_perm_seed=3)
    assert 67 * 9 * 79 == 47637
    inp = synth.make_inputs(case, device=cuda_dev)
    plan = make_plan(case, inp)
    lens, indptr = _batch_arrays(case, cuda_dev)
    idx = torch.from_numpy(random_idx(case, np.random.default_rng(7))).to(cuda_dev)
    ref, _ = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx,
                              k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out, _ = msa.sparse_decode_noalloc(inp["q"], inp["k_pages"], inp["v_pages"], lens, indptr, inp["kv_indices"],
                                       idx, inp["k_scale"], inp["v_scale"], err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert (out.float() - ref.float()).abs().max().item() <= O_ATOL_FP8

    b, hq, hkv, topk = 40, 3, 1, 397
    assert b * hq * topk == 47640
    q = torch.zeros((b, hq, 128), dtype=torch.bfloat16, device=cuda_dev)
    kp = torch.zeros((8, hkv, 128, 128), dtype=torch.float8_e4m3fn, device=cuda_dev)
    lens = torch.full((b,), 128, dtype=torch.int32, device=cuda_dev)
    indptr = torch.arange(b + 1, dtype=torch.int32, device=cuda_dev)
    table = torch.zeros((b,), dtype=torch.int32, device=cuda_dev)
    idx = torch.zeros((b, hkv, topk), dtype=torch.int32, device=cuda_dev)
    sc = torch.ones(hkv, dtype=torch.float32, device=cuda_dev)
    with pytest.raises(msa.MsaError) as e:
        msa.sparse_decode_noalloc(q, kp, kp, lens, indptr, table, idx, sc, sc)
    assert e.value.status == 1 and "static scratch" in str(e.value)
