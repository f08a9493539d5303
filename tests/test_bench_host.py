"""Host-side accounting of bench.py, checked on the CPU."""
import numpy as np

import bench
from block_sparse_long_proxy_gb300 import synth


def test_visible_pairs_of_all_blocks_is_the_causal_count():
    """With every valid block selected the exact visible-pair FLOPs equal the
    dense bottom-right causal count: query i of a sequence sees off + i + 1
    keys, each pair costing 4*d FLOPs per head."""
    case = synth.Case("ragged", [300, 128, 1], [300, 500, 1000], 4, 2, 64, 2, 32, 9)
    tiles = bench._tiles_nvp(case)
    idx = np.full((len(tiles), case.hkv, case.topk), -1, np.int32)
    for t, n in enumerate(tiles):
        idx[t, :, :n] = np.arange(n)
    pairs = sum(sum(kl - ql + i + 1 for i in range(ql)) for ql, kl in zip(case.qo_lens, case.kv_lens))
    assert bench.visible_pair_flops(idx, case) == pairs * case.hq * 4 * case.d


def test_visible_pairs_of_one_diagonal_block():
    """A single 128-row tile choosing only its diagonal block: the causal
    triangle of 128 * 129 / 2 pairs."""
    case = synth.Case("one tile", [128], [128], 2, 1, 64, 1, 32, 1)
    idx = np.array([[[0]]], np.int32)
    assert bench.visible_pair_flops(idx, case) == 128 * 129 // 2 * 2 * 4 * 64
    assert bench.selected_flops(idx, case)[0] == 128 * 128 * 2 * 4 * 64
