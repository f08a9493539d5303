"""msa_topk_select on the GPU against the oracle, bit-exact on identical
max_score inputs (ties, -inf, signed zeros, ragged num_valid_pages)."""
import numpy as np
import pytest
import torch

from oracle import msa_oracle as O

pytestmark = pytest.mark.gpu


def _scores(rng, n, h, nb, kind):
    if kind == "ties":
        vals = np.array([-np.inf, -2.0, -0.0, 0.0, 0.5, 1.0, 3.0], dtype=np.float32)
        return vals[rng.integers(0, len(vals), (n, h, nb))]
    x = rng.standard_normal((n, h, nb)).astype(np.float32)
    x[rng.random((n, h, nb)) < 0.05] = -np.inf
    return x


@pytest.mark.parametrize("nb,topk,kind", [(8, 4, "ties"), (8, 1, "normal"), (200, 16, "normal"),
                                          (256, 16, "ties"), (257, 16, "normal"), (1000, 40, "ties"),
                                          (1024, 16, "normal"), (3000, 16, "ties"), (3000, 300, "normal"),
                                          (64, 64, "normal"), (64, 65, "normal"),
                                          # the maxima the API accepts: topk 1024, 65536 blocks per row
                                          (1025, 1024, "ties"), (65536, 1024, "normal"), (65536, 1024, "ties")])
def test_topk_bit_exact(cuda_dev, nb, topk, kind):
    from block_sparse_long_proxy_gb300 import msa
    rng = np.random.default_rng(nb * 7 + topk)
    n, h = 37, 3
    ms = _scores(rng, n, h, nb, kind)
    nvp = rng.integers(1, nb + 1, n).astype(np.int32)
    nvp[0], nvp[1] = 1, nb
    got = msa.topk_select(torch.from_numpy(ms).to(cuda_dev), topk,
                          torch.from_numpy(nvp).to(cuda_dev)).cpu().numpy()
    want = O.topk_select(ms, topk, nvp)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("n,h,nb", [(256, 8, 256), (1472, 8, 1024), (32, 8, 1024)])
def test_topk_config_shapes(cuda_dev, n, h, nb):
    """Shapes of the 32K prefill, the varlen prefill and the decode batch."""
    from block_sparse_long_proxy_gb300 import msa
    rng = np.random.default_rng(n)
    ms = rng.standard_normal((n, h, nb)).astype(np.float32)
    nvp = np.minimum(np.arange(n) % nb + 1, nb).astype(np.int32)
    if n == 32:
        nvp[:] = nb
    for t in range(n):                       # -inf past the valid blocks
        ms[t, :, nvp[t]:] = -np.inf
    got = msa.topk_select(torch.from_numpy(ms).to(cuda_dev), 16, torch.from_numpy(nvp).to(cuda_dev)).cpu().numpy()
    assert np.array_equal(got, O.topk_select(ms, 16, nvp))


@pytest.mark.parametrize("nb", [8, 600, 2000])
def test_topk_out_of_range_nvp_selects_nothing(cuda_dev, nb):
    """num_valid_pages outside [1, max_blocks] is outside the contract: the
    row is written as all -1 (no clamping to a valid count); the other rows
    are unaffected."""
    from block_sparse_long_proxy_gb300 import msa
    rng = np.random.default_rng(nb)
    n, h, topk = 6, 2, 5
    ms = rng.standard_normal((n, h, nb)).astype(np.float32)
    nvp = np.array([0, -3, nb + 1, nb, 1, 1 << 30], dtype=np.int32)
    got = msa.topk_select(torch.from_numpy(ms).to(cuda_dev), topk, torch.from_numpy(nvp).to(cuda_dev)).cpu().numpy()
    for t in (0, 1, 2, 5):
        assert (got[t] == -1).all(), (t, got[t])
    good = [3, 4]
    assert np.array_equal(got[good], O.topk_select(ms[good], topk, nvp[good]))
