"""Shared helpers of the GPU parity tests: run the CUDA path through the
binding and compare with the oracle on the same inputs."""
import numpy as np
import torch

from block_sparse_long_proxy_gb300 import synth
from oracle import msa_oracle as O

# parity tolerances: outputs and gradients max-abs 2e-2 (bf16) / 6e-2 (e4m3)
# and cosine >= 0.99 against the fp64 oracle
O_ATOL_BF16 = 2e-2
O_ATOL_FP8 = 6e-2
COS_MIN = 0.99
MS_ATOL = 1e-3
GAP = 1e-3


def random_idx(case, rng):
    """Valid kv_block_indexes, one row per proxy head: the diagonal block plus
    topk-1 random others, ascending, -1 padded."""
    tl = O.tiles_of(case.qo_lens, case.kv_lens)
    idx = np.full((len(tl), case.hp, case.topk), -1, np.int32)
    for t, tile in enumerate(tl):
        for g in range(case.hp):
            others = rng.permutation(tile.nvp - 1)[: case.topk - 1]
            sel = sorted(list(others) + [tile.nvp - 1])
            idx[t, g, :len(sel)] = sel
    return idx


def irregular_idx(case, rng):
    """Selections in random order with the -1 padding spread through the row,
    and every fifth (tile, group) row empty: its rows get out = 0, lse = -inf."""
    idx = random_idx(case, rng)
    nt, hkv, _ = idx.shape
    for t in range(nt):
        for g in range(hkv):
            idx[t, g] = idx[t, g][rng.permutation(case.topk)]
            if (t * hkv + g) % 5 == 3:
                idx[t, g] = -1
    return idx


def make_plan(case, inp):
    from block_sparse_long_proxy_gb300 import msa
    return msa.Plan(case.qo_lens, case.kv_lens, case.hq, case.hkv, case.hp, case.d, case.dp, case.topk,
                    num_pages=inp["k_pages"].shape[0], kv_dtype=case.kv_dtype)


def rows_of_tiles(case, tile_ids):
    tl = O.tiles_of(case.qo_lens, case.kv_lens)
    return np.concatenate([np.arange(tl[t].q_begin, tl[t].q_end) for t in tile_ids])


def compare_out(got, ref, atol, what="out"):
    """max-abs and cosine similarity of bf16 GPU output vs fp64 oracle."""
    g = got.astype(np.float64).ravel()
    r = ref.astype(np.float64).ravel()
    err = np.abs(g - r).max()
    cos = float(g @ r / (np.linalg.norm(g) * np.linalg.norm(r) + 1e-300))
    assert err <= atol, "%s max-abs %g > %g" % (what, err, atol)
    assert cos >= COS_MIN, "%s cosine %g" % (what, cos)
    return err, cos


def check_indices_with_gap(idx_gpu, ms_ref, nvp, topk, tile_ids):
    """End-to-end indices (from the GPU's own max_score) equal the oracle's
    (from the oracle's max_score) except where the oracle's scores of the
    swapped blocks differ by less than GAP from its selection threshold."""
    idx_ref = O.topk_select(ms_ref[tile_ids], topk, nvp[tile_ids])
    bad = 0
    for a, t in enumerate(tile_ids):
        for h in range(idx_ref.shape[1]):
            got = set(int(x) for x in idx_gpu[t, h] if x >= 0)
            want = set(int(x) for x in idx_ref[a, h] if x >= 0)
            if got == want:
                continue
            row = ms_ref[t, h]
            sel_scores = [row[j] for j in want if j != nvp[t] - 1]
            thr = min(sel_scores) if sel_scores else -np.inf
            for j in got.symmetric_difference(want):
                if not abs(float(row[j]) - float(thr)) < GAP:
                    bad += 1
    assert bad == 0, "%d index mismatches beyond the score-gap rule" % bad
