"""msa_sparse_attn_bwd on the GPU against the oracle: dq, dk, dv and the KL
proxy gradients dpq, dpk, each within max-abs 2e-2 and cosine >= 0.99."""
import numpy as np
import pytest
import torch

from block_sparse_long_proxy_gb300 import synth
from oracle import msa_oracle as O
from tests.gpu_cases import O_ATOL_BF16, compare_out, irregular_idx, make_plan, random_idx, rows_of_tiles

pytestmark = pytest.mark.gpu
PAGE = 128


def _run_gpu(case, inp, idx_t, w):
    plan = make_plan(case, inp)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx_t)
    grads = plan.sparse_attn_bwd(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx_t, out, lse,
                                 inp["dout"], inp["pq"], inp["pk_pages"], kl_weight=w)
    torch.cuda.synchronize()
    plan.check_errors()
    return {k: v.cpu().numpy() for k, v in grads.items()}


def _oracle(case, inp, idx, w, tile_ids=None):
    return O.sparse_attention_bwd(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                                  inp["kv_indices"].cpu().numpy(), idx, case.qo_lens, case.kv_lens,
                                  synth.bits(inp["dout"]), synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]),
                                  kl_weight=w, tile_ids=tile_ids)


SMALL = [
    (synth.Case("S=256 G=4", [256], [256], 8, 2, 128, 2, 64, 2), 1.0),
    (synth.Case("ragged varlen paged offsets", [300, 77, 129], [300, 500, 129], 8, 2, 128, 2, 64, 3,
                page_perm_seed=3, extra_pages=2), 0.5),
    (synth.Case("G=1", [384], [384], 2, 2, 128, 2, 64, 2, page_perm_seed=1), 1.0),
    (synth.Case("long rows topk 16", [2048], [2048], 8, 2, 128, 2, 64, 16, page_perm_seed=5), 1.0),
    # dq runs the G heads of a proxy head in one CTA: G = 3 and G = 2 (Hp = 2 Hkv), with tiles of one,
    # two and more cached blocks (the head's Q sits in a different K stage for each)
    (synth.Case("G=3 ragged", [300, 129, 77], [900, 129, 333], 6, 2, 128, 2, 64, 3, page_perm_seed=9), 0.9),
    (synth.Case("G=2 Hp=2Hkv", [640, 200], [640, 700], 8, 2, 128, 4, 64, 5, page_perm_seed=10), 1.0),
    # an odd number of proxy heads: the proxy softmax pairs heads 0 and 1 and runs head 2 alone
    (synth.Case("Hp=3", [300, 129], [300, 500], 6, 3, 128, 3, 64, 3, page_perm_seed=11), 0.7),
    # a sequence with keys but no query rows: its pages are never selected, so their dK, dV, dpk are 0
    (synth.Case("empty query sequence mid-batch", [300, 0, 129], [300, 500, 129], 8, 2, 128, 2, 64, 3,
                page_perm_seed=6), 1.0),
    # topk at the largest value a plan accepts: every tile caches all of its blocks
    (synth.Case("topk 1024 (the maximum) over 16 blocks", [2048], [2048], 4, 1, 128, 1, 64, 1024,
                page_perm_seed=7), 1.0),
]


@pytest.mark.parametrize("case,w", SMALL, ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_bwd_small(cuda_dev, case, w):
    inp = synth.make_inputs(case, device=cuda_dev, with_dout=True)
    idx = random_idx(case, np.random.default_rng(9))
    got = _run_gpu(case, inp, torch.from_numpy(idx).to(cuda_dev), w)
    ref = _oracle(case, inp, idx, w)
    for name in ("dq", "dpq", "dk", "dv", "dpk"):
        compare_out(got[name], ref[name], O_ATOL_BF16, name)


def _check_all(got, ref):
    for name in ("dq", "dpq", "dk", "dv", "dpk"):
        assert np.isfinite(got[name]).all(), "%s has non-finite entries" % name
        assert np.isfinite(ref[name]).all(), "oracle %s has non-finite entries" % name
        compare_out(got[name], ref[name], O_ATOL_BF16, name)


def test_bwd_rows_without_visible_keys(cuda_dev):
    """Tiles straddling two blocks with topk 1 (only the diagonal block): the
    early rows see no key (R7), so their dq and dpq are exactly 0 and they
    add nothing to dk, dv, dpk; everything else matches the oracle."""
    case = synth.Case("straddle topk 1", [128, 100, 64], [200, 300, 1000], 8, 2, 128, 2, 64, 1,
                      page_perm_seed=6, extra_pages=1)
    inp = synth.make_inputs(case, device=cuda_dev, with_dout=True)
    idx = random_idx(case, np.random.default_rng(2))
    got = _run_gpu(case, inp, torch.from_numpy(idx).to(cuda_dev), 1.0)
    ref = _oracle(case, inp, idx, 1.0)
    empty = np.isneginf(ref["lse"])
    assert empty.any()
    assert (got["dq"][empty] == 0.0).all()
    grp = case.hq // case.hkv
    empty_g = empty.reshape(case.total_q, case.hkv, grp).all(2)
    assert (got["dpq"][empty_g] == 0.0).all()
    _check_all(got, ref)


@pytest.mark.parametrize("case", [
    synth.Case("shuffled and empty rows", [1024, 700, 300], [1024, 900, 300], 8, 2, 128, 2, 64, 6,
               page_perm_seed=4),
    synth.Case("shuffled, ragged, topk 3", [300, 77, 129], [300, 500, 129], 4, 2, 128, 2, 64, 3,
               page_perm_seed=3, extra_pages=2),
], ids=lambda c: c.name)
def test_bwd_irregular_indexes(cuda_dev, case):
    """Selections in random order with -1 entries anywhere in the row and
    every fifth (tile, group) row holding only -1 (R7 for all its rows)."""
    inp = synth.make_inputs(case, device=cuda_dev, with_dout=True)
    idx = irregular_idx(case, np.random.default_rng(4))
    got = _run_gpu(case, inp, torch.from_numpy(idx).to(cuda_dev), 0.8)
    ref = _oracle(case, inp, idx, 0.8)
    assert np.isneginf(ref["lse"]).any()
    _check_all(got, ref)


def test_bwd_shared_pages(cuda_dev):
    """Several page-table entries naming one physical page (a shared prefix,
    and one page listed twice): dK, dV and dpk of that page are the sums over
    every entry, as the oracle's scatter-add gives them."""
    case = synth.Case("shared prefix", [256, 300, 129], [512, 600, 384], 8, 2, 128, 2, 64, 3,
                      page_perm_seed=8, extra_pages=1)
    inp = synth.make_inputs(case, device=cuda_dev, with_dout=True)
    table = inp["kv_indices"].clone()
    # entries: seq 0 -> 0..3, seq 1 -> 4..8, seq 2 -> 9..11
    table[4] = table[0]          # seq 1 block 0 = seq 0 block 0
    table[5] = table[1]          # seq 1 block 1 = seq 0 block 1
    table[9] = table[0]          # seq 2 block 0 = the same page again
    table[11] = table[6]         # seq 2 block 2 = seq 1 block 2
    inp["kv_indices"] = table
    idx = random_idx(case, np.random.default_rng(3))
    # make sure the shared blocks are selected by several sequences
    tl = O.tiles_of(case.qo_lens, case.kv_lens)
    for t, tile in enumerate(tl):
        for g in range(case.hkv):
            if tile.nvp > 2 and case.topk >= 3:
                idx[t, g, :3] = sorted({0, 1, tile.nvp - 1}) + [-1] * (3 - len({0, 1, tile.nvp - 1}))
    got = _run_gpu(case, inp, torch.from_numpy(idx).to(cuda_dev), 1.0)
    ref = _oracle(case, inp, idx, 1.0)
    _check_all(got, ref)


def test_bwd_bitwise_reproducible(cuda_dev):
    """No gradient is reduced by atomics: repeated backward calls give the same
    bits for all five gradients, with four query heads per proxy head (the dpq
    sum over heads), several KV heads (the dpk sum over them), shared pages and
    ragged tiles."""
    case = synth.Case("repro", [700, 300, 129], [900, 600, 384], 16, 4, 128, 4, 64, 4,
                      page_perm_seed=12, extra_pages=1)
    inp = synth.make_inputs(case, device=cuda_dev, with_dout=True)
    table = inp["kv_indices"].clone()
    table[8] = table[0]  # seq 1 block 0 = seq 0 block 0
    inp["kv_indices"] = table
    idx_t = torch.from_numpy(random_idx(case, np.random.default_rng(21))).to(cuda_dev)
    plan = make_plan(case, inp)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx_t)
    runs = []
    for _ in range(3):
        g = plan.sparse_attn_bwd(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx_t, out, lse,
                                 inp["dout"], inp["pq"], inp["pk_pages"], kl_weight=0.7)
        torch.cuda.synchronize()
        plan.check_errors()
        runs.append({k: v.clone() for k, v in g.items()})
    for name in ("dq", "dpq", "dk", "dv", "dpk"):
        for r in runs[1:]:
            assert torch.equal(runs[0][name], r[name]), "%s differs between runs" % name
    ref = _oracle(case, inp, idx_t.cpu().numpy(), 0.7)
    _check_all({k: v.cpu().numpy() for k, v in runs[0].items()}, ref)


NARROW = [
    (synth.tiny(), 1.0),
    (synth.Case("d64 dp32", [256], [256], 4, 2, 64, 2, 32, 2), 1.0),
    (synth.Case("d64 dp32 ragged paged G=4", [300, 77, 129], [300, 500, 129], 8, 2, 64, 2, 32, 3,
                page_perm_seed=3, extra_pages=2), 0.6),
    (synth.Case("d128 dp32", [384, 129], [384, 700], 8, 2, 128, 2, 32, 3, page_perm_seed=2), 1.0),
    (synth.Case("d64 dp64 Hp=4", [700, 129], [900, 384], 16, 2, 64, 4, 64, 4, page_perm_seed=7), 0.8),
]


@pytest.mark.parametrize("case,w", NARROW, ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_bwd_narrow_heads(cuda_dev, case, w):
    """head_dim 64 and proxy_head_dim 32: the d = 128 / dp = 64 kernels read
    the narrow tensors through 64-column boxes whose columns past the edge
    are zero; every gradient matches the oracle at the true width and the
    scales of the true widths."""
    inp = synth.make_inputs(case, device=cuda_dev, with_dout=True)
    idx = random_idx(case, np.random.default_rng(11))
    got = _run_gpu(case, inp, torch.from_numpy(idx).to(cuda_dev), w)
    ref = _oracle(case, inp, idx, w)
    for name, shape in (("dq", (case.total_q, case.hq, case.d)), ("dpq", (case.total_q, case.hp, case.dp))):
        assert got[name].shape == shape, name
    _check_all(got, ref)


def test_bwd_refuses_misaligned_gradients(cuda_dev):
    """The gradients are written with 32-byte stores: a buffer that is only
    16-byte aligned is refused on the host (MSA_ERR_INVALID_ARG) and nothing
    is launched."""
    from block_sparse_long_proxy_gb300 import msa
    case = synth.Case("align", [256], [256], 4, 2, 128, 2, 64, 2)
    inp = synth.make_inputs(case, device=cuda_dev, with_dout=True)
    idx = torch.from_numpy(random_idx(case, np.random.default_rng(0))).to(cuda_dev)
    plan = make_plan(case, inp)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx)
    n = inp["q"].numel()
    buf = torch.zeros(n + 8, dtype=torch.float32, device=cuda_dev)
    grads = dict(dq=buf[4:4 + n].view(inp["q"].shape),  # 16 bytes past a 256-byte boundary
                 dk=torch.zeros(inp["k_pages"].shape, dtype=torch.float32, device=cuda_dev),
                 dv=torch.zeros(inp["v_pages"].shape, dtype=torch.float32, device=cuda_dev),
                 dpq=torch.zeros(inp["pq"].shape, dtype=torch.float32, device=cuda_dev),
                 dpk=torch.zeros(inp["pk_pages"].shape, dtype=torch.float32, device=cuda_dev))
    with pytest.raises(msa.MsaError) as e:
        plan.sparse_attn_bwd(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx, out, lse,
                             inp["dout"], inp["pq"], inp["pk_pages"], grads=grads)
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert (buf == 0).all()


def test_bwd_long_selection_list_is_sorted_in_place(cuda_dev):
    """1025 one-tile sequences whose page tables all name one physical page,
    with two proxy heads per KV head: 2050 selections of that page by one KV
    head, more than the key-side kernel sorts in shared memory, so the list
    is sorted in place in the inverse index.  All five gradients match the
    oracle (dK, dV and dpk of the shared page sum every sequence) and two
    runs give the same bits."""
    n_seq = 1025
    case = synth.Case("long list", [128] * n_seq, [128] * n_seq, 2, 1, 64, 2, 32, 1)
    inp = synth.make_inputs(case, device=cuda_dev, with_dout=True)
    inp["kv_indices"] = torch.zeros_like(inp["kv_indices"])  # every sequence's only block is physical page 0
    idx_np = random_idx(case, np.random.default_rng(5))
    idx_t = torch.from_numpy(idx_np).to(cuda_dev)
    plan = make_plan(case, inp)
    out, lse = plan.sparse_attn(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx_t)
    runs = []
    for _ in range(2):
        g = plan.sparse_attn_bwd(inp["q"], inp["k_pages"], inp["v_pages"], inp["kv_indices"], idx_t, out, lse,
                                 inp["dout"], inp["pq"], inp["pk_pages"], kl_weight=0.9)
        torch.cuda.synchronize()
        plan.check_errors()
        runs.append({k: v.clone() for k, v in g.items()})
    for name in ("dq", "dpq", "dk", "dv", "dpk"):
        assert torch.equal(runs[0][name], runs[1][name]), "%s differs between runs" % name
    ref = _oracle(case, inp, idx_np, 0.9)
    got = {k: v.cpu().numpy() for k, v in runs[0].items()}
    for name in ("dq", "dpq"):
        compare_out(got[name], ref[name], O_ATOL_BF16, name)
    # the shared page's dK, dV and dpk sum 2050 selections (magnitudes up to
    # ~740): the bar is the same relative precision as for an O(1) output
    for name in ("dk", "dv", "dpk"):
        assert np.isfinite(got[name]).all(), name
        compare_out(got[name], ref[name], O_ATOL_BF16 * max(1.0, float(np.abs(ref[name]).max())), name)
