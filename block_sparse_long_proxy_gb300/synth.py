"""Seeded synthetic inputs for the MSA hot path.

This module only draws random tensors and lays them out; it holds none of the
method's arithmetic.  The same tensors feed both the CUDA library and the
fp64 oracle (the oracle reads the identical bf16 / e4m3 bytes).

Layouts (shared contract, see include/msa.h):
  q, dout        [total_q, Hq, d]          bf16
  k_pages,v_pages[P, Hkv, 128, d]          bf16, or e4m3 with k_scale/v_scale [Hkv] fp32
  pk_pages_e4m3 [P, 1, 128, dp], pk_scale [1]  e4m3 proxy K (e4m3 cases only)
  pk_fp4_codes [P, 1, 128, dp/2] uint8, pk_fp4_scales [P, 1, 128, dp/16] e4m3,
  pk_fp4_global [1]                          NVFP4 proxy K (e4m3 cases only)
  pq             [total_q, Hp, dp]         bf16
  pk_pages       [P, 1, 128, dp]           bf16 (one shared proxy K head)
  kv_indices     [sum_s ceil(kv_len_s/128)] int32 page table, logical -> physical
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

PAGE = 128


@dataclass
class Case:
    name: str
    qo_lens: list
    kv_lens: list
    hq: int
    hkv: int
    d: int
    hp: int
    dp: int
    topk: int
    kv_dtype: str = "bf16"          # "bf16" or "e4m3"
    page_perm_seed: int | None = None  # None: identity page table
    planted: bool = False
    seed: int = 0
    extra_pages: int = 0            # unused pages in the pool (page ids never referenced)
    meta: dict = field(default_factory=dict)

    @property
    def total_q(self):
        return int(sum(self.qo_lens))

    @property
    def n_pages_used(self):
        return int(sum((k + PAGE - 1) // PAGE for k in self.kv_lens))


# The five workloads of the method's evaluation, at their stated sizes.
def tiny():
    return Case("tiny causal MSA forward S=1024", [1024], [1024], 8, 2, 64, 2, 32, 4)


def prefill_32k():
    return Case("sparse prefill S=32768", [32768], [32768], 32, 8, 128, 8, 64, 16)


def varlen_paged():
    lens = [8192, 16384, 32768, 131072]
    return Case("varlen paged prefill 8K/16K/32K/128K", lens, list(lens), 32, 8, 128, 8, 64, 16,
                page_perm_seed=1, planted=True)


def paged_decode():
    return Case("paged sparse decode B=32 kv=131072 fp8", [1] * 32, [131072] * 32, 64, 8, 128, 8, 64,
                16, kv_dtype="e4m3", page_perm_seed=1)


def training_64k():
    return Case("training step S=65536", [65536], [65536], 32, 8, 128, 8, 64, 16)


CONFIGS = {"tiny": tiny, "prefill_32k": prefill_32k, "varlen_paged": varlen_paged,
           "paged_decode": paged_decode, "training_64k": training_64k}


def _randn(shape, gen, device):
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)


def _orthonormal(n, dim, gen, device):
    a = _randn((dim, n), gen, device).double().cpu()
    qm, _ = torch.linalg.qr(a)
    return qm.T.contiguous().float().to(device)        # [n, dim], orthonormal rows


def make_inputs(case: Case, device="cpu", with_dout=False):
    """Draw every input of one workload with torch generators seeded from
    case.seed (values: N(0,1)); page table from case.page_perm_seed."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(case.seed)
    tq = case.total_q
    n_pages = case.n_pages_used + case.extra_pages
    out = {}
    q = _randn((tq, case.hq, case.d), gen, dev)
    k = _randn((n_pages, case.hkv, PAGE, case.d), gen, dev)
    v = _randn((n_pages, case.hkv, PAGE, case.d), gen, dev)
    pq = _randn((tq, case.hp, case.dp), gen, dev)
    pk = _randn((n_pages, 1, PAGE, case.dp), gen, dev)

    # page table: logical block j of sequence s -> physical page
    if case.page_perm_seed is None:
        table = torch.arange(case.n_pages_used, dtype=torch.int32)
    else:
        pg = torch.Generator().manual_seed(case.page_perm_seed)
        table = torch.randperm(n_pages, generator=pg)[: case.n_pages_used].to(torch.int32)
    out["kv_indices"] = table.to(dev)

    if case.planted:
        # low-rank planted-block signal so that block selections are not
        # uniform: 32 planted blocks per (sequence, group) share a direction
        # with every query of that group.
        groups = case.hkv
        u = _orthonormal(groups, case.dp, gen, dev)       # proxy directions
        w = _orthonormal(groups, case.d, gen, dev)        # main directions
        gsz = case.hq // case.hkv
        pl = torch.Generator().manual_seed(case.seed + 7)
        start = 0
        for s, kl in enumerate(case.kv_lens):
            nb = (kl + PAGE - 1) // PAGE
            for g in range(groups):
                blocks = torch.randperm(nb, generator=pl)[: min(32, nb)]
                phys = table[start + blocks].long().to(dev)
                pk[phys, 0] += 3.0 * u[g]
                k[phys, g] += 2.0 * w[g]
            start += nb
        for g in range(groups):
            pq[:, g] += 3.0 * u[g]
            q[:, g * gsz:(g + 1) * gsz] += 2.0 * w[g]

    out["q"] = q.to(torch.bfloat16)
    out["pq"] = pq.to(torch.bfloat16)
    out["pk_pages"] = pk.to(torch.bfloat16)
    if case.kv_dtype == "bf16":
        out["k_pages"] = k.to(torch.bfloat16)
        out["v_pages"] = v.to(torch.bfloat16)
    else:
        # e4m3 codes with one fp32 scale per KV head: scale = amax / 448
        ks = k.abs().amax(dim=(0, 2, 3)) / 448.0
        vs = v.abs().amax(dim=(0, 2, 3)) / 448.0
        out["k_pages"] = (k / ks.view(1, -1, 1, 1)).to(torch.float8_e4m3fn)
        out["v_pages"] = (v / vs.view(1, -1, 1, 1)).to(torch.float8_e4m3fn)
        out["k_scale"] = ks.float().contiguous()
        out["v_scale"] = vs.float().contiguous()
        # the shared proxy K head as e4m3 codes with one fp32 scale (decode)
        ps = pk.abs().amax() / 448.0
        out["pk_pages_e4m3"] = (pk / ps).to(torch.float8_e4m3fn)
        out["pk_scale"] = ps.float().reshape(1).contiguous()
        # ... and in NVFP4: e2m1 code pairs, e4m3 scales of 16 dims, one fp32 scale
        out.update(nvfp4_quantize(pk))
    if with_dout:
        out["dout"] = _randn((tq, case.hq, case.d), gen, dev).to(torch.bfloat16)
    del q, k, v, pq, pk
    return out


E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)   # codes 0..7 of the OCP FP4 E2M1 format


def nvfp4_quantize(x):
    """Quantise x [..., D] (D a multiple of 16) to NVFP4 inputs: each block of
    16 dims gets an e4m3 scale amax/6 (relative to one fp32 global scale
    amax/(448*6)), and each value the nearest e2m1 code (ties to the smaller
    magnitude); code pairs are packed with the even dim in the low nibble.
    Returns pk_fp4_codes uint8 [..., D/2], pk_fp4_scales e4m3 [..., D/16],
    pk_fp4_global fp32 [1]."""
    x = x.float()
    gs = (x.abs().amax() / (448.0 * 6.0)).clamp_min(1e-30)
    blk = x.reshape(*x.shape[:-1], x.shape[-1] // 16, 16)
    bs = (blk.abs().amax(-1) / (6.0 * gs)).to(torch.float8_e4m3fn)
    denom = (bs.float() * gs).unsqueeze(-1)
    y = torch.where(denom > 0, blk / torch.where(denom > 0, denom, torch.ones_like(denom)), torch.zeros_like(blk))
    mags = torch.tensor(E2M1_MAGNITUDES, dtype=torch.float32, device=x.device)
    k = (y.abs().unsqueeze(-1) - mags).abs().argmin(-1)                  # nearest magnitude, lower on ties
    code = (k | ((y < 0) & (k > 0)).to(k.dtype) << 3).to(torch.uint8).reshape(x.shape)
    packed = code[..., 0::2] | (code[..., 1::2] << 4)
    return {"pk_fp4_codes": packed.contiguous(), "pk_fp4_scales": bs.contiguous(),
            "pk_fp4_global": gs.reshape(1).float().contiguous()}


def bits(t: torch.Tensor):
    """Raw bit pattern of a bf16 / e4m3 tensor as a numpy array (uint16 or
    uint8), for the oracle."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    raise TypeError(t.dtype)
