"""The oracle reproduces its stored outputs on the tiny golden case
(tests/golden/tiny_chain.json, written by tests/golden/make_golden.py)."""
import json
import os

import numpy as np

from tests.golden.make_golden import compute

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_stored_golden():
    want = json.load(open(os.path.join(HERE, "golden", "tiny_chain.json")))
    got = compute()
    assert got["num_valid_pages"] == want["num_valid_pages"]
    assert got["kv_block_indexes"] == want["kv_block_indexes"]
    gm = np.array([[[np.nan if v is None else v for v in r] for r in t] for t in got["max_score"]])
    wm = np.array([[[np.nan if v is None else v for v in r] for r in t] for t in want["max_score"]])
    assert np.array_equal(np.isnan(gm), np.isnan(wm))
    np.testing.assert_allclose(gm[~np.isnan(gm)], wm[~np.isnan(wm)], rtol=0, atol=0)
    np.testing.assert_allclose(got["o_row_sums"], want["o_row_sums"], rtol=1e-12)
    np.testing.assert_allclose(got["lse_rows"], want["lse_rows"], rtol=1e-12)
