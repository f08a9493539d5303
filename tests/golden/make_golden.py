"""Writes tests/golden/tiny_chain.json from the fp64 oracle alone.

The pages print no worked example, so the stored values here are the
oracle's own outputs on a tiny seeded case; the test that reads them
(tests/test_golden.py) guards the oracle against unnoticed changes.  Inputs
come from the seeded generator, which holds none of the method's arithmetic.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from block_sparse_long_proxy_gb300 import synth  # noqa: E402
from oracle import msa_oracle as O  # noqa: E402


def golden_case():
    # ragged, paged, with a prefix offset: 2 sequences, 3 tiles
    return synth.Case("golden", [200, 60], [300, 130], 4, 2, 64, 2, 32, 2, page_perm_seed=3, seed=11)


def compute():
    case = golden_case()
    inp = synth.make_inputs(case)
    table = inp["kv_indices"].numpy()
    nvp = O.num_valid_pages(case.qo_lens, case.kv_lens)
    ms = O.proxy_max_score(synth.bits(inp["pq"]), synth.bits(inp["pk_pages"]), table, case.qo_lens, case.kv_lens)
    idx = O.topk_select(ms, case.topk, nvp)
    o, lse = O.sparse_attention(synth.bits(inp["q"]), synth.bits(inp["k_pages"]), synth.bits(inp["v_pages"]), table,
                                idx, case.qo_lens, case.kv_lens)
    return {
        "case": {"qo_lens": case.qo_lens, "kv_lens": case.kv_lens, "hq": case.hq, "hkv": case.hkv, "d": case.d,
                 "hp": case.hp, "dp": case.dp, "topk": case.topk, "page_perm_seed": 3, "seed": 11},
        "num_valid_pages": nvp.tolist(),
        "max_score": [[[None if not np.isfinite(v) else float(v) for v in row] for row in t] for t in ms],
        "kv_block_indexes": idx.tolist(),
        "o_row_sums": [float(x) for x in o.sum(axis=(1, 2))],
        "lse_rows": [float(x) for x in lse[:, 0]],
    }


if __name__ == "__main__":
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_chain.json"), "w") as f:
        json.dump(compute(), f, indent=1)
