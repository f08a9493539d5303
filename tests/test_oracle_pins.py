"""Pins for the fp64 oracle: every check here compares the oracle with a
route that does not go through the oracle's own formula -- torch's library
attention and autograd, max-pooling, closed forms, brute force over subsets
and central finite differences -- chosen so that a dropped term, a wrong
sign, index, mask boundary or a transposed operand in the oracle fails."""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import msa_oracle as O
from block_sparse_long_proxy_gb300 import synth

PAGE = 128


# ---------------------------------------------------------------- decoding --

def test_bf16_decode_all_patterns():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.bf16_to_f64(pats)
    ref = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2  # 0x7f and 0xff
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9
    # the K/V decode of the attention oracle looks the codes up in a table of
    # this function's values: same bytes in any shape, same results
    grid = np.random.default_rng(0).integers(0, 256, (3, 5, 7), dtype=np.uint8)
    looked = O._decode_kv(grid, True)
    assert looked.shape == grid.shape
    assert np.array_equal(looked, O.e4m3_to_f64(grid), equal_nan=True)


# ------------------------------------------------------------------ tiling --

def test_tiles_closed_form():
    tl = O.tiles_of([1024], [1024])
    assert [t.nvp for t in tl] == list(range(1, 9))
    assert all(t.pos0 == 128 * i for i, t in enumerate(tl))
    dec = O.tiles_of([1] * 3, [131072, 200, 129])
    assert [t.nvp for t in dec] == [1024, 2, 2]
    # ragged tail with a prefix: offset 800, rows 0..199
    rag = O.tiles_of([200], [1000])
    assert [(t.q_begin, t.q_end, t.pos0, t.nvp) for t in rag] == [(0, 128, 800, 8), (128, 200, 928, 8)]
    assert list(O.kv_indptr([1000, 128, 129])) == [0, 8, 9, 11]
    assert O.tiles_of([0, 5], [10, 5])[0].seq == 1


# ------------------------------------------------------------------- top-k --

def _precedes(a, b, s):
    return (s[a] > s[b]) or (s[a] == s[b] and a < b)


def _brute_topk(scores, nvp, k):
    """Unique subset where every member precedes every non-member, by
    enumeration over all subsets of the right size."""
    jd = nvp - 1
    if k >= nvp:
        return list(range(nvp))
    cands = [j for j in range(jd) if scores[j] > -np.inf]
    m = min(k - 1, len(cands))
    hits = []
    for sub in itertools.combinations(cands, m):
        rest = [j for j in cands if j not in sub]
        if all(_precedes(a, b, scores) for a in sub for b in rest):
            hits.append(sorted(list(sub) + [jd]))
    assert len(hits) == 1
    return hits[0]


def test_topk_brute_force_tiny():
    rng = np.random.default_rng(0)
    for trial in range(400):
        nb = int(rng.integers(1, 10))
        nvp = int(rng.integers(1, nb + 1))
        k = int(rng.integers(1, 7))
        # few distinct values -> many ties; some -inf; a -0.0 next to +0.0
        vals = np.array([-np.inf, -1.5, -0.0, 0.0, 0.25, 2.0], dtype=np.float32)
        sc = vals[rng.integers(0, len(vals), nb)]
        assert O.topk_row(sc, nvp, k) == _brute_topk(sc, nvp, k), (sc, nvp, k)


def test_topk_special_cases():
    eq = np.zeros(10, dtype=np.float32)
    assert O.topk_row(eq, 10, 4) == [0, 1, 2, 9]            # ties -> lower index
    ninf = np.full(10, -np.inf, dtype=np.float32)
    assert O.topk_row(ninf, 10, 4) == [9]                    # never picks -inf
    assert O.topk_row(eq, 3, 4) == [0, 1, 2]                 # K >= nvp: all valid
    sc = np.array([5, 1, 9, 3, -100, 7], dtype=np.float32)
    assert O.topk_row(sc, 5, 3) == [0, 2, 4]                 # diagonal forced even if lowest
    ms = np.stack([sc[None].repeat(2, 0)])                   # [1, 2, 6]
    out = O.topk_select(ms, 4, np.array([5]))
    assert out.shape == (1, 2, 4) and list(out[0, 0]) == [0, 2, 3, 4]
    pad = O.topk_select(np.stack([ninf[None]]), 4, np.array([10]))
    assert list(pad[0, 0]) == [9, -1, -1, -1]


# -------------------------------------------------------------- proxy max --

def _mk(case):
    return synth.make_inputs(case)


def _pool_route(inp, case):
    """max_score by a different route: dense masked logits with torch.matmul,
    then F.max_pool2d over 128x128 windows (ceil mode)."""
    pq = inp["pq"].double()
    pk = inp["pk_pages"].double()
    table = inp["kv_indices"].long()
    outs = []
    q0, p0 = 0, 0
    nbmax = max((k + PAGE - 1) // PAGE for k in case.kv_lens)
    for ql, kl in zip(case.qo_lens, case.kv_lens):
        nb = (kl + PAGE - 1) // PAGE
        keys = torch.cat([pk[table[p0 + j], 0] for j in range(nb)], 0)[:kl]     # [kl, dp]
        qs = pq[q0:q0 + ql]                                                     # [ql, hp, dp]
        lg = torch.einsum("rhc,kc->hrk", qs, keys) / math.sqrt(case.dp)
        qpos = (kl - ql) + torch.arange(ql)
        vis = torch.arange(kl)[None, :] <= qpos[:, None]
        lg = lg.masked_fill(~vis[None], -math.inf)
        pooled = F.max_pool2d(lg[:, None], kernel_size=PAGE, stride=PAGE, ceil_mode=True)[:, 0]
        pooled = pooled.permute(1, 0, 2)                                        # [tiles, hp, nb]
        full = torch.full((pooled.shape[0], case.hp, nbmax), -math.inf, dtype=torch.float64)
        full[:, :, :nb] = pooled
        outs.append(full)
        q0 += ql
        p0 += nb
    return torch.cat(outs, 0).float().numpy()


@pytest.mark.parametrize("qo,kv,perm", [([1024], [1024], None), ([200, 77], [1000, 300], 3),
                                        ([1, 1], [700, 129], 5)])
def test_proxy_max_pool_route(qo, kv, perm):
    case = synth.Case("t", qo, kv, 4, 2, 64, 2, 32, 4, page_perm_seed=perm, extra_pages=2)
    inp = _mk(case)
    ms = O.proxy_max_score(synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]),
                           inp["kv_indices"].numpy(), qo, kv)
    ref = _pool_route(inp, case)
    assert ms.shape == ref.shape
    assert np.array_equal(np.isneginf(ms), np.isneginf(ref))
    fin = np.isfinite(ref)
    np.testing.assert_allclose(ms[fin], ref[fin], rtol=1e-6, atol=1e-6)


def test_proxy_closed_form_constant_keys():
    """All proxy keys equal c and pq[i] = (i+1) c: logit = (i+1)|c|^2/sqrt(dp),
    so max_score[t, j] is attained at the last row of tile t that sees any
    key of block j."""
    qo, kv, dp = 300, 500, 32
    off = kv - qo
    c = np.zeros(dp)
    c[3] = 0.5
    nb = (kv + PAGE - 1) // PAGE
    pk = torch.zeros(nb, 1, PAGE, dp, dtype=torch.float64)
    pk[:, 0, :, :] = torch.from_numpy(c)
    pq = torch.from_numpy(np.arange(1, qo + 1)[:, None, None] * c[None, None, :])  # [qo,1,dp]
    ms = O.proxy_max_score(synth.bits(pq.to(torch.bfloat16)), synth.bits(pk.to(torch.bfloat16)),
                           np.arange(nb), [qo], [kv])
    for t in range(3):
        r_last = min((t + 1) * 128, qo) - 1
        for j in range(nb):
            rows = [r for r in range(t * 128, r_last + 1) if off + r >= j * PAGE]
            want = (max(rows) + 1) * 0.25 / math.sqrt(dp) if rows else -math.inf
            got = float(ms[t, 0, j])
            assert (got == want) or abs(got - want) <= 1e-6 * abs(want), (t, j, got, want)


def test_proxy_mask_boundary():
    """One planted large pair on the causal boundary counts; one key further
    right does not."""
    qo = kv = 256
    dp = 32
    pq = torch.zeros(qo, 1, dp)
    pk = torch.zeros(2, 1, PAGE, dp)
    pq[130, 0, 0] = 4.0
    pk[1, 0, 130 - 128, 0] = 2.0      # key 130 is visible to row 130
    pk[1, 0, 140 - 128, 1] = 9.0      # key 140: future for rows < 140
    pq[135, 0, 1] = 1.0               # row 135 must not see key 140
    ms = O.proxy_max_score(synth.bits(pq.to(torch.bfloat16)), synth.bits(pk.to(torch.bfloat16)),
                           np.arange(2), [qo], [kv])
    assert float(ms[1, 0, 1]) == pytest.approx(8.0 / math.sqrt(dp))
    assert float(ms[1, 0, 0]) == 0.0
    assert float(ms[0, 0, 1]) == -math.inf


def test_proxy_fp8_keys_reduce_to_bf16_route():
    """R11: with e4m3 codes and a power-of-two scale every code * scale is a
    bf16 value, so the e4m3 route of proxy_max_score must equal the (pinned)
    bf16 route on those values exactly; a wrong scale or decode would not."""
    qo, kv, dp = [1, 1, 1], [700, 129, 300], 64
    gen = torch.Generator().manual_seed(4)
    nb = sum((k + PAGE - 1) // PAGE for k in kv)
    codes = (torch.randn(nb + 2, 1, PAGE, dp, generator=gen) * 60).to(torch.float8_e4m3fn)
    scale = 0.125
    values = codes.to(torch.float64) * scale
    assert torch.equal(values.to(torch.bfloat16).to(torch.float64), values)   # exact in bf16
    pq = torch.randn(3, 2, dp, generator=gen).to(torch.bfloat16)
    table = torch.randperm(nb + 2, generator=gen)[:nb].numpy()
    ref = O.proxy_max_score(synth.bits(pq), synth.bits(values.to(torch.bfloat16)), table, qo, kv)
    got = O.proxy_max_score(synth.bits(pq), synth.bits(codes), table, qo, kv, pk_scale=scale)
    assert np.array_equal(got, ref)
    assert np.isfinite(got[:, :, 0]).all()


# ----------------------------------------------------- sparse attention ----

def _dense_route(inp, case, idx, fp8=False):
    """Attention by torch's library routine with an explicit boolean mask:
    visible (bottom-right causal) and block selected for (tile, group)."""
    q = inp["q"].double()
    if fp8:
        k = inp["k_pages"].double() * inp["k_scale"].double().view(1, -1, 1, 1)
        v = inp["v_pages"].double() * inp["v_scale"].double().view(1, -1, 1, 1)
    else:
        k, v = inp["k_pages"].double(), inp["v_pages"].double()
    table = inp["kv_indices"].long()
    grp = case.hq // case.hkv
    outs = []
    q0, p0, t0 = 0, 0, 0
    for ql, kl in zip(case.qo_lens, case.kv_lens):
        nb = (kl + PAGE - 1) // PAGE
        ks = torch.cat([k[table[p0 + j]] for j in range(nb)], 1)[:, :kl]  # [hkv, kl, d]
        vs = torch.cat([v[table[p0 + j]] for j in range(nb)], 1)[:, :kl]
        qpos = (kl - ql) + torch.arange(ql)
        vis = torch.arange(kl)[None, :] <= qpos[:, None]
        o = torch.zeros(ql, case.hq, case.d, dtype=torch.float64)
        for h in range(case.hq):
            g = h // grp
            sel = torch.zeros(ql, kl, dtype=torch.bool)
            for r in range(ql):
                for j in idx[t0 + r // 128, h // (case.hq // idx.shape[1])]:
                    if j >= 0:
                        sel[r, j * PAGE:(j + 1) * PAGE] = True
            o[:, h] = F.scaled_dot_product_attention(q[q0:q0 + ql, h][None], ks[g][None],
                                                     vs[g][None], attn_mask=(vis & sel)[None])[0]
        outs.append(o)
        q0 += ql
        p0 += nb
        t0 += (ql + 127) // 128
    return torch.cat(outs, 0).numpy()


def _rand_idx(case, rng):
    """Random valid selections, one row per proxy head (R8)."""
    tl = O.tiles_of(case.qo_lens, case.kv_lens)
    idx = np.full((len(tl), case.hp, case.topk), -1, np.int32)
    for t, tile in enumerate(tl):
        for g in range(case.hp):
            others = rng.permutation(tile.nvp - 1)[: case.topk - 1]
            sel = sorted(list(others) + [tile.nvp - 1])
            idx[t, g, :len(sel)] = sel
    return idx


@pytest.mark.parametrize("qo,kv,topk", [([1024], [1024], 8), ([1024], [1024], 3),
                                        ([200, 64], [333, 64], 2), ([1, 1], [500, 128], 2)])
def test_sparse_attention_vs_library(qo, kv, topk):
    case = synth.Case("t", qo, kv, 4, 2, 64, 2, 32, topk, page_perm_seed=2)
    inp = _mk(case)
    idx = _rand_idx(case, np.random.default_rng(1))
    o, lse = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]),
                                synth.bits(inp["v_pages"]), inp["kv_indices"].numpy(), idx, qo, kv)
    ref = _dense_route(inp, case, idx)
    np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12)
    assert np.all(np.isfinite(lse))


def test_topk_all_blocks_is_dense_causal():
    case = synth.tiny()
    case.topk = 8
    inp = _mk(case)
    nvp = O.num_valid_pages(case.qo_lens, case.kv_lens)
    ms = O.proxy_max_score(synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]),
                           inp["kv_indices"].numpy(), case.qo_lens, case.kv_lens)
    idx = O.topk_select(ms, 8, nvp)
    o, _ = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]),
                              synth.bits(inp["v_pages"]), inp["kv_indices"].numpy(), idx,
                              case.qo_lens, case.kv_lens)
    q = inp["q"].double().permute(1, 0, 2)                          # [hq, S, d]
    k = inp["k_pages"].double().permute(1, 0, 2, 3).reshape(2, 1024, 64)
    v = inp["v_pages"].double().permute(1, 0, 2, 3).reshape(2, 1024, 64)
    ref = F.scaled_dot_product_attention(q, k.repeat_interleave(4, 0), v.repeat_interleave(4, 0),
                                         is_causal=True).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12)


def test_zero_keys_closed_form():
    """K == 0: every visible logit is 0, so O is the mean of V over the
    visible selected keys and LSE = ln(count)."""
    case = synth.Case("t", [300], [300], 2, 1, 64, 1, 32, 2)
    inp = _mk(case)
    inp["k_pages"].zero_()
    idx = _rand_idx(case, np.random.default_rng(4))
    o, lse = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]),
                                synth.bits(inp["v_pages"]), inp["kv_indices"].numpy(), idx, [300], [300])
    v = inp["v_pages"].double()[:, 0].reshape(-1, 64)[:300].numpy()
    for r in [0, 5, 127, 128, 200, 299]:
        keys = [kk for j in idx[r // 128, 0] if j >= 0 for kk in range(j * 128, min(j * 128 + 128, 300))
                if kk <= r]
        np.testing.assert_allclose(o[r, 0], v[keys].mean(0), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse[r, 0], math.log(len(keys)), rtol=1e-12)


def test_fp8_scales_vs_library():
    case = synth.Case("t", [1, 1, 1], [640, 300, 129], 8, 2, 64, 2, 32, 3, kv_dtype="e4m3",
                      page_perm_seed=9)
    inp = _mk(case)
    idx = _rand_idx(case, np.random.default_rng(3))
    o, _ = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]),
                              synth.bits(inp["v_pages"]), inp["kv_indices"].numpy(), idx,
                              case.qo_lens, case.kv_lens, inp["k_scale"].numpy(), inp["v_scale"].numpy())
    ref = _dense_route(inp, case, idx, fp8=True)
    np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------- backward --

def _autograd_route(inp, case, idx, w):
    """Main gradients by autograd through torch's attention with the block
    mask; proxy gradients by autograd through torch's kl_div."""
    grp = case.hq // case.hkv
    q = inp["q"].double().requires_grad_()
    kp = inp["k_pages"].double().requires_grad_()
    vp = inp["v_pages"].double().requires_grad_()
    pq = inp["pq"].double().requires_grad_()
    pk = inp["pk_pages"].double().requires_grad_()
    do = inp["dout"].double()
    table = inp["kv_indices"].long()
    loss_main = 0.0
    loss_kl = 0.0
    q0, p0, t0 = 0, 0, 0
    for ql, kl in zip(case.qo_lens, case.kv_lens):
        nb = (kl + PAGE - 1) // PAGE
        ks = torch.cat([kp[table[p0 + j]] for j in range(nb)], 1)[:, :kl]
        vs = torch.cat([vp[table[p0 + j]] for j in range(nb)], 1)[:, :kl]
        pks = torch.cat([pk[table[p0 + j], 0] for j in range(nb)], 0)[:kl]
        qpos = (kl - ql) + torch.arange(ql)
        vis = torch.arange(kl)[None, :] <= qpos[:, None]
        msa_grp = case.hq // case.hp                 # query heads per proxy head (R8)
        for p in range(case.hp):
            g = p // (case.hp // case.hkv)
            sel = torch.zeros(ql, kl, dtype=torch.bool)
            for r in range(ql):
                for j in idx[t0 + r // 128, p]:
                    if j >= 0:
                        sel[r, j * PAGE:(j + 1) * PAGE] = True
            # rows that see no selected key (R7) are left out of both losses:
            # the library softmax would give 0/0 there
            live = (vis & sel).any(1)
            rows = torch.arange(q0, q0 + ql)[live]
            m = (vis & sel)[live]
            pmain = 0.0
            for h in range(p * msa_grp, (p + 1) * msa_grp):
                qh = q[rows, h]
                oh = F.scaled_dot_product_attention(qh[None], ks[g][None], vs[g][None], attn_mask=m[None])[0]
                loss_main = loss_main + (oh * do[rows, h]).sum()
                s = (qh @ ks[g].T / math.sqrt(case.d)).masked_fill(~m, -math.inf)
                pmain = pmain + torch.softmax(s, -1).detach() / msa_grp
            z = (pq[rows, p] @ pks.T / math.sqrt(case.dp)).masked_fill(~m, -math.inf)
            logp = torch.log_softmax(z, -1).masked_fill(~m, 0.0)
            loss_kl = loss_kl + w * F.kl_div(logp, pmain, reduction="sum")
        q0 += ql
        p0 += nb
        t0 += (ql + 127) // 128
    (loss_main + loss_kl).backward()
    grads = [t.grad if t.grad is not None else torch.zeros_like(t) for t in (q, kp, vp, pq, pk)]
    return tuple(gr.numpy() for gr in grads)


@pytest.mark.parametrize("qo,kv,topk,w", [([256], [256], 2, 1.0), ([150, 40], [300, 200], 2, 0.5)])
def test_bwd_vs_autograd(qo, kv, topk, w):
    case = synth.Case("t", qo, kv, 4, 2, 64, 2, 32, topk, page_perm_seed=4, extra_pages=1)
    inp = synth.make_inputs(case, with_dout=True)
    idx = _rand_idx(case, np.random.default_rng(5))
    g = O.sparse_attention_bwd(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                               inp["kv_indices"].numpy(), idx, qo, kv, synth.bits(inp["dout"]),
                               synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]), kl_weight=w)
    dq, dk, dv, dpq, dpk = _autograd_route(inp, case, idx, w)
    for name, ref in [("dq", dq), ("dk", dk), ("dv", dv), ("dpq", dpq), ("dpk", dpk)]:
        np.testing.assert_allclose(g[name], ref, rtol=1e-9, atol=1e-11, err_msg=name)


def _r7_cases():
    """Selections that leave query rows with no visible key (R7): a tile
    straddling two blocks with only its diagonal block selected; a group
    whose selection row holds only -1; -1 entries between valid ones."""
    a = synth.Case("straddle topk 1", [128], [200], 4, 2, 64, 2, 32, 1)
    ia = np.array([[[1], [1]]], dtype=np.int32)             # rows 0..55 sit in block 0
    b = synth.Case("ragged, -1 rows", [150, 40, 1], [300, 200, 129], 4, 2, 64, 2, 32, 3,
                   page_perm_seed=4, extra_pages=1)
    ib = _rand_idx(b, np.random.default_rng(12))
    ib[0, 0, :] = [2, -1, -1]          # tile 0 of seq 0 (positions 150..277): rows < 256 see nothing
    ib[1, 1, :] = -1                   # tile 1, group 1: no block at all
    ib[2, 0, :] = [-1, 1, -1]          # seq 1 tile: diagonal block only, -1 on both sides
    return [(a, ia), (b, ib)]


@pytest.mark.parametrize("ci", [0, 1])
def test_bwd_rows_without_visible_keys(ci):
    """R7 in the backward: rows that see no selected key get zero dq and
    dpq and send nothing into dk, dv or dpk; every gradient is finite and
    the rest equals autograd with those rows left out of both losses."""
    case, idx = _r7_cases()[ci]
    inp = synth.make_inputs(case, with_dout=True)
    g = O.sparse_attention_bwd(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                               inp["kv_indices"].numpy(), idx, case.qo_lens, case.kv_lens, synth.bits(inp["dout"]),
                               synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]), kl_weight=0.7)
    for name in ("dq", "dk", "dv", "dpq", "dpk", "o"):
        assert np.isfinite(g[name]).all(), name
    empty = np.isneginf(g["lse"])                                 # [total_q, Hq]
    assert empty.any() and (~empty).any()
    assert (g["dq"][empty] == 0.0).all() and (g["o"][empty] == 0.0).all()
    grp = case.hq // case.hkv
    empty_g = empty.reshape(case.total_q, case.hkv, grp).all(2)   # [total_q, Hkv]: same for the group's heads
    assert (empty_g == empty.reshape(case.total_q, case.hkv, grp).any(2)).all()
    assert (g["dpq"][empty_g] == 0.0).all()
    dq, dk, dv, dpq, dpk = _autograd_route(inp, case, idx, 0.7)
    for name, ref in [("dq", dq), ("dk", dk), ("dv", dv), ("dpq", dpq), ("dpk", dpk)]:
        np.testing.assert_allclose(g[name], ref, rtol=1e-9, atol=1e-11, err_msg=name)


def test_kl_objective_finite_with_empty_rows():
    """The KL objective is defined (finite) when some rows see no key, and
    its finite differences still match the closed-form proxy gradient."""
    case, idx = _r7_cases()[0]
    inp = synth.make_inputs(case, with_dout=True)
    args = (synth.bits(inp["q"]), synth.bits(inp["k_pages"]), inp["kv_indices"].numpy(), idx,
            case.qo_lens, case.kv_lens)
    g = O.sparse_attention_bwd(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                               inp["kv_indices"].numpy(), idx, case.qo_lens, case.kv_lens,
                               synth.bits(inp["dout"]), synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]))
    pq = O.bf16_to_f64(synth.bits(inp["pq"]))
    pk = O.bf16_to_f64(synth.bits(inp["pk_pages"]))
    assert np.isfinite(O.kl_objective(pq, pk, *args))
    h = 1e-6
    for i, hh, c in [(3, 0, 5), (100, 1, 17), (127, 0, 31), (60, 1, 0)]:   # rows 0..55 are empty
        a, b = pq.copy(), pq.copy()
        a[i, hh, c] += h
        b[i, hh, c] -= h
        fd = (O.kl_objective(a, pk, *args) - O.kl_objective(b, pk, *args)) / (2 * h)
        assert abs(fd - g["dpq"][i, hh, c]) <= 1e-6 * max(1.0, abs(fd)), (i, hh, c, fd, g["dpq"][i, hh, c])


def test_kl_grad_finite_differences():
    """The closed-form proxy gradient equals central differences of the
    fp64 KL objective (w=1), for entries of pq and of pk."""
    case = synth.Case("t", [256], [256], 4, 2, 64, 2, 32, 2)
    inp = synth.make_inputs(case, with_dout=True)
    idx = _rand_idx(case, np.random.default_rng(6))
    args = (synth.bits(inp["q"]), synth.bits(inp["k_pages"]), inp["kv_indices"].numpy(), idx,
            case.qo_lens, case.kv_lens)
    g = O.sparse_attention_bwd(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                               inp["kv_indices"].numpy(), idx, case.qo_lens, case.kv_lens,
                               synth.bits(inp["dout"]), synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]))
    pq = O.bf16_to_f64(synth.bits(inp["pq"]))
    pk = O.bf16_to_f64(synth.bits(inp["pk_pages"]))
    h = 1e-6
    rng = np.random.default_rng(7)
    for _ in range(6):
        i, hh, c = int(rng.integers(0, 256)), int(rng.integers(0, 2)), int(rng.integers(0, 32))
        a, b = pq.copy(), pq.copy()
        a[i, hh, c] += h
        b[i, hh, c] -= h
        fd = (O.kl_objective(a, pk, *args) - O.kl_objective(b, pk, *args)) / (2 * h)
        assert abs(fd - g["dpq"][i, hh, c]) <= 1e-6 * max(1.0, abs(fd)), (i, hh, c, fd, g["dpq"][i, hh, c])
    for _ in range(6):
        p, r, c = int(rng.integers(0, 2)), int(rng.integers(0, 128)), int(rng.integers(0, 32))
        a, b = pk.copy(), pk.copy()
        a[p, 0, r, c] += h
        b[p, 0, r, c] -= h
        fd = (O.kl_objective(pq, a, *args) - O.kl_objective(pq, b, *args)) / (2 * h)
        assert abs(fd - g["dpk"][p, 0, r, c]) <= 1e-6 * max(1.0, abs(fd)), (p, r, c, fd)


def test_main_bwd_finite_differences():
    """dq/dk/dv equal central differences of sum(O * dO)."""
    case = synth.Case("t", [256], [256], 2, 1, 64, 1, 32, 2)
    inp = synth.make_inputs(case, with_dout=True)
    idx = _rand_idx(case, np.random.default_rng(8))
    bits = {k: synth.bits(inp[k]) for k in ("q", "k_pages", "v_pages", "dout", "pq", "pk_pages")}
    g = O.sparse_attention_bwd(bits["q"], bits["k_pages"], bits["v_pages"], inp["kv_indices"].numpy(), idx,
                               [256], [256], bits["dout"], bits["pq"], bits["pk_pages"])
    do = O.bf16_to_f64(bits["dout"])

    def objective(qf, kf, vf):
        # forward in float64 from float inputs, through the oracle's own
        # attention applied to exactly-representable perturbed inputs is not
        # possible (bf16 inputs), so evaluate the masked softmax directly
        ks = np.concatenate([np.arange(j * 128, j * 128 + 128) for j in idx[0, 0] if j >= 0] or [[]])
        tot = 0.0
        for t in range(2):
            ks_t = np.concatenate([np.arange(j * 128, j * 128 + 128) for j in idx[t, 0] if j >= 0])
            for r in range(t * 128, t * 128 + 128):
                kk = ks_t[ks_t <= r]
                for hh in range(2):
                    s = kf.reshape(-1, 64)[kk] @ qf[r, hh] / 8.0
                    p = np.exp(s - s.max())
                    p /= p.sum()
                    tot += (p @ vf.reshape(-1, 64)[kk]) @ do[r, hh]
        del ks
        return tot

    qf = O.bf16_to_f64(bits["q"])
    kf = O.bf16_to_f64(bits["k_pages"])[:, 0]
    vf = O.bf16_to_f64(bits["v_pages"])[:, 0]
    eps = 1e-6
    rng = np.random.default_rng(9)
    for name, arr, grad in [("q", qf, g["dq"]), ("k", kf, g["dk"][:, 0]), ("v", vf, g["dv"][:, 0])]:
        for _ in range(4):
            ix = tuple(int(rng.integers(0, n)) for n in arr.shape)
            a, b = arr.copy(), arr.copy()
            a[ix] += eps
            b[ix] -= eps
            qa, ka, va = (a if name == "q" else qf), (a if name == "k" else kf), (a if name == "v" else vf)
            qb, kb, vb = (b if name == "q" else qf), (b if name == "k" else kf), (b if name == "v" else vf)
            fd = (objective(qa, ka, va) - objective(qb, kb, vb)) / (2 * eps)
            assert abs(fd - grad[ix]) <= 1e-6 * max(1.0, abs(fd)), (name, ix, fd, grad[ix])


def test_kl_grad_constant_proxy_keys_is_zero():
    """sum_k (p_proxy - p_main) = 0 per row, so with every proxy key equal
    the pq gradient vanishes."""
    case = synth.Case("t", [256], [256], 4, 2, 64, 2, 32, 2)
    inp = synth.make_inputs(case, with_dout=True)
    inp["pk_pages"][:] = inp["pk_pages"][0, 0, 0]
    idx = _rand_idx(case, np.random.default_rng(10))
    g = O.sparse_attention_bwd(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                               inp["kv_indices"].numpy(), idx, [256], [256], synth.bits(inp["dout"]),
                               synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]))
    assert np.abs(g["dpq"]).max() < 1e-12


def test_rows_without_visible_keys():
    """R7: a tile straddling two blocks with only its diagonal block
    selected leaves its early rows without keys: O = 0, LSE = -inf; the
    other rows still match the library attention."""
    case = synth.Case("t", [128], [200], 2, 1, 64, 1, 32, 1)   # offset 72: rows 0..55 sit in block 0
    inp = _mk(case)
    idx = np.array([[[1]]], dtype=np.int32)                       # diagonal block only
    o, lse = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                                inp["kv_indices"].numpy(), idx, [128], [200])
    early = np.arange(128) + 72 < 128
    assert np.all(o[early] == 0.0) and np.all(np.isneginf(lse[early]))
    ref = _dense_route(inp, case, idx)
    np.testing.assert_allclose(o[~early], ref[~early], rtol=1e-10, atol=1e-12)


def test_unit_values_give_unit_output():
    """V == 1: O = sum_k P[k] * 1, so every row with a visible key has O = 1
    (the rows of P sum to 1) and every row without one has O = 0."""
    case = synth.Case("ragged", [200, 64, 1], [333, 64, 500], 4, 2, 64, 2, 32, 2, page_perm_seed=1)
    inp = _mk(case)
    inp["v_pages"].fill_(1.0)
    idx = _rand_idx(case, np.random.default_rng(11))
    # tile 0 (positions 133..260) keeps only its diagonal block 2 (keys 256..):
    # its rows at positions below 256 see nothing (R7)
    idx[0, 0, :] = [2, -1]
    o, lse = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                                inp["kv_indices"].numpy(), idx, case.qo_lens, case.kv_lens)
    seen = np.isfinite(lse)
    assert seen.any() and (~seen).any()
    np.testing.assert_allclose(o[seen], 1.0, rtol=0, atol=1e-12)
    assert (o[~seen] == 0.0).all()


def test_topk_diagonal_always_present():
    """Every selected row holds the diagonal block num_valid_pages - 1, is
    ascending, and has min(topk, nvp) entries followed by -1 padding."""
    rng = np.random.default_rng(17)
    for topk in (1, 2, 5, 16):
        nb = 40
        ms = rng.standard_normal((60, 3, nb)).astype(np.float32)
        ms[rng.random(ms.shape) < 0.2] = -np.inf
        nvp = rng.integers(1, nb + 1, 60).astype(np.int32)
        idx = O.topk_select(ms, topk, nvp)
        for t in range(60):
            for h in range(3):
                row = idx[t, h]
                n = min(topk, int(nvp[t]))
                sel = row[row >= 0]
                assert int(nvp[t]) - 1 in sel
                assert len(sel) <= n and (row[len(sel):] == -1).all()
                assert (np.diff(sel) > 0).all()


def test_proxy_max_dominates_visible_pairs():
    """Each block score is at least every visible pair's logit in that block
    (a sample of pairs, computed here straight from the definition): a mask
    that drops visible keys, or a wrong pairing of rows and keys, fails."""
    case = synth.Case("t", [300], [460], 2, 2, 64, 2, 32, 2, page_perm_seed=2)
    inp = _mk(case)
    ms = O.proxy_max_score(synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]), inp["kv_indices"].numpy(),
                           case.qo_lens, case.kv_lens)
    pq = inp["pq"].double().numpy()
    pk = inp["pk_pages"].double().numpy()[:, 0]                  # [pages, 128, dp]
    table = inp["kv_indices"].numpy()
    off = 460 - 300
    rng = np.random.default_rng(5)
    for _ in range(400):
        i = int(rng.integers(0, 300))
        k = int(rng.integers(0, off + i + 1))                      # visible to row i
        h = int(rng.integers(0, 2))
        logit = float(pq[i, h] @ pk[table[k // PAGE], k % PAGE]) / math.sqrt(case.dp)
        assert logit <= float(ms[i // 128, h, k // PAGE]) * (1 + 1e-6) + 1e-6


# ------------------------------------- several proxy heads per group (R8) --

def _hp2_case(**kw):
    """Hp = 2 Hkv: two proxy heads (two block sets) per GQA group of 4."""
    return synth.Case("hp2", kw.get("qo", [300, 129]), kw.get("kv", [460, 129]), 8, 2, 64, 4, 32,
                      kw.get("topk", 2), page_perm_seed=3, extra_pages=1)


def test_hp2_attention_vs_library():
    """Each query head attends over its own proxy head's blocks: the oracle
    equals torch's attention with the per-head block mask."""
    case = _hp2_case()
    inp = _mk(case)
    idx = _rand_idx(case, np.random.default_rng(21))
    assert idx.shape[1] == 4
    o, _ = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                              inp["kv_indices"].numpy(), idx, case.qo_lens, case.kv_lens)
    ref = _dense_route(inp, case, idx)
    np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12)


def test_hp2_attention_reduces_to_one_proxy_head_per_group():
    """With Hp = 2 Hkv, head h of group g gives what the one-proxy-head
    attention gives when group g's block set is proxy head 2g + s's, s the
    half of the group h sits in: heads 0-1 of a group of 4 use s = 0,
    heads 2-3 use s = 1."""
    case = _hp2_case()
    inp = _mk(case)
    idx = _rand_idx(case, np.random.default_rng(22))
    args = (synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
            inp["kv_indices"].numpy())
    o2, l2 = O.sparse_attention(*args, idx, case.qo_lens, case.kv_lens)
    for s in range(2):
        o1, l1 = O.sparse_attention(*args, np.ascontiguousarray(idx[:, s::2]), case.qo_lens, case.kv_lens)
        for h in range(case.hq):
            if (h % 4) // 2 == s:
                np.testing.assert_array_equal(o2[:, h], o1[:, h])
                np.testing.assert_array_equal(l2[:, h], l1[:, h])


def test_hp2_bwd_vs_autograd():
    """All five gradients with Hp = 2 Hkv against autograd: each proxy head
    distils the mean distribution of its own two query heads over its own
    blocks; dK / dV of a KV head sum both proxy heads' selections."""
    case = _hp2_case(qo=[150, 40], kv=[300, 200])
    inp = synth.make_inputs(case, with_dout=True)
    idx = _rand_idx(case, np.random.default_rng(23))
    g = O.sparse_attention_bwd(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                               inp["kv_indices"].numpy(), idx, case.qo_lens, case.kv_lens, synth.bits(inp["dout"]),
                               synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]), kl_weight=0.6)
    dq, dk, dv, dpq, dpk = _autograd_route(inp, case, idx, 0.6)
    for name, ref in [("dq", dq), ("dk", dk), ("dv", dv), ("dpq", dpq), ("dpk", dpk)]:
        np.testing.assert_allclose(g[name], ref, rtol=1e-9, atol=1e-11, err_msg=name)


def test_hp2_kl_grad_finite_differences():
    """The closed-form dpq of every proxy head equals central differences of
    the fp64 KL objective with Hp = 2 Hkv."""
    case = _hp2_case(qo=[256], kv=[256])
    inp = synth.make_inputs(case, with_dout=True)
    idx = _rand_idx(case, np.random.default_rng(24))
    args = (synth.bits(inp["q"]), synth.bits(inp["k_pages"]), inp["kv_indices"].numpy(), idx,
            case.qo_lens, case.kv_lens)
    g = O.sparse_attention_bwd(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]),
                               inp["kv_indices"].numpy(), idx, case.qo_lens, case.kv_lens,
                               synth.bits(inp["dout"]), synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]))
    pq = O.bf16_to_f64(synth.bits(inp["pq"]))
    pk = O.bf16_to_f64(synth.bits(inp["pk_pages"]))
    h = 1e-6
    for i, hh, c in [(10, 0, 3), (130, 1, 7), (200, 2, 30), (255, 3, 0)]:
        a, b = pq.copy(), pq.copy()
        a[i, hh, c] += h
        b[i, hh, c] -= h
        fd = (O.kl_objective(a, pk, *args) - O.kl_objective(b, pk, *args)) / (2 * h)
        assert abs(fd - g["dpq"][i, hh, c]) <= 1e-6 * max(1.0, abs(fd)), (i, hh, c, fd, g["dpq"][i, hh, c])


# ------------------------------------------------ NVFP4 proxy K (R12) -------

def test_e2m1_decode_all_codes():
    """The 16 e2m1 codes decode to the format's published values: +-{0, 0.5,
    1, 1.5, 2, 3, 4, 6} (code 8 is -0)."""
    got = O.e2m1_to_f64(np.arange(16))
    want = np.array(list(synth.E2M1_MAGNITUDES) + [-m for m in synth.E2M1_MAGNITUDES])
    assert np.array_equal(got, want)
    assert np.signbit(got[8])


def test_proxy_nvfp4_reduces_to_bf16_route():
    """NVFP4 proxy keys whose values are exact in bf16 (a power-of-two global
    scale) give exactly the scores of the bf16 route on those values, which
    this test builds from the published e2m1 table and torch's e4m3
    conversion: a swapped nibble order, a wrong 16-dim scale grouping or a
    dropped scale fails."""
    qo, kv, dp = [1, 1, 2], [300, 129, 700], 64
    gen = torch.Generator().manual_seed(13)
    nb = sum((k + PAGE - 1) // PAGE for k in kv)
    codes = torch.randint(0, 256, (nb + 1, 1, PAGE, dp // 2), generator=gen, dtype=torch.int32).to(torch.uint8)
    scales = (torch.rand(nb + 1, 1, PAGE, dp // 16, generator=gen) * 30 + 0.01).to(torch.float8_e4m3fn)
    gscale = 0.125
    mags = torch.tensor(synth.E2M1_MAGNITUDES, dtype=torch.float64)
    lo, hi = codes.long() & 0xF, codes.long() >> 4
    nib = torch.stack([lo, hi], -1).reshape(nb + 1, 1, PAGE, dp)
    vals = torch.where(nib >= 8, -1.0, 1.0).double() * mags[nib & 7]
    vals = vals * scales.double().repeat_interleave(16, -1) * gscale
    assert torch.equal(vals.to(torch.bfloat16).double(), vals)          # exact in bf16
    pq = torch.randn(4, 2, dp, generator=gen).to(torch.bfloat16)
    table = torch.randperm(nb + 1, generator=gen)[:nb].numpy()
    ref = O.proxy_max_score(synth.bits(pq), synth.bits(vals.to(torch.bfloat16)), table, qo, kv)
    got = O.proxy_max_score(synth.bits(pq), codes.numpy(), table, qo, kv, pk_nvfp4=(synth.bits(scales), gscale))
    assert np.array_equal(got, ref)
    assert np.isfinite(got[:, :, 0]).all()
