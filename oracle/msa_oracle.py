"""fp64 CPU oracle for the MiniMax Sparse Attention (MSA) hot path.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package's smoke check and
the benchmark's CPU-baseline leg may import this module; the product path
(the CUDA library and its Python binding) never does, and it shares no code
with them.  Everything here is plain numpy in float64, written for a reader
to check against the pages by eye: no tiling, fusion or reordering beyond
what the method states.

Sources (page title, section):
  [README]  "MiniMax-AI/MSA" README (pigsec.cn mirror), section "Usage":
            the three-stage flow -- a dense proxy pass with
            num_kv_heads=1 and output_maxscore=True that yields a per-block
            max score, sparse_topk_select(max_score, topk, num_valid_pages)
            that yields kv_block_indexes, and a plan with kv_block_num=topk
            whose attention visits only those blocks through the page table
            kv_indices; page_size 128.
  [NEWS]    news.ditty.ir, "MSA: MiniMax sparse attention kernels for SM100
            GPUs", paragraph on the three-stage flow (same three stages).
  [FLASH]   iitog.ru, "Flash-MSA: open kernels for training models with
            sparse attention on millions of tokens":
              - "three key differences" paragraph: whole 128-token blocks
                picked by max-pooling proxy scores; GQA main attention;
                each proxy head picks its own block set per GQA group;
              - "kernel design" paragraph: the token's own (local) block is
                always visible, block indexes are cached from the forward
                and reused by the backward;
              - "backward pass" paragraph: the gradient of the KL loss with
                respect to a proxy score is p_proxy - p_main.

Readings where the pages are silent:
  R1  causal alignment is bottom-right: query row r of a sequence with
      qo_len rows and kv_len keys sits at position kv_len - qo_len + r and
      sees key k iff k <= that position.
  R2  the proxy pools LOGITS (q.k/sqrt(dp)), not probabilities; -inf where a
      block holds no visible key for any row of the tile.
  R3  the diagonal block of a tile is the block holding the tile's last
      row's position: j_d = num_valid_pages - 1; it is selected first and
      counts inside topk.  The other topk-1 blocks are the largest finite
      max_score values among j < j_d, ties to the lower block index.
      Output is ascending, padded with -1.  If topk >= num_valid_pages all
      valid blocks are selected.
  R4  main attention scale is 1/sqrt(d); LSE is natural-log.
  R5  FP8 e4m3 K/V carry one fp32 scale per KV head: logit =
      (q.k_code)*k_scale/sqrt(d), value = v_code*v_scale.
  R6  the KL term is KL(p_main || p_proxy) per (query row, GQA group) over
      the selected visible keys, p_main = mean of the group's G head
      distributions (detached), summed over rows, weight w; the LM loss
      sends no gradient into the proxy and the KL none into main Q/K/V.
      Parity of R6's domain and mean is unpinned by the pages.
  R7  a query row that sees no key of its tile's selected blocks (possible
      only when a tile straddles two blocks and its earlier block is not
      selected, or when its selection row holds only -1) has O = 0 and
      LSE = -inf; in the backward its P and p_proxy are 0, so its KL term,
      dZ and every gradient it sends are 0.
  R8  several proxy heads per GQA group: with Hp = m * Hkv proxy heads (m >=
      1, Hq divisible by Hp) each proxy head picks its own block set, and
      the G = Hq/Hkv query heads of a GQA group are split into m equal
      "MSA groups" of Hq/Hp consecutive heads: query head h attends over the
      blocks kv_block_indexes[t, h // (Hq/Hp)] of KV head h // (Hq/Hkv), and
      proxy head p = h // (Hq/Hp) distils the mean distribution of its own
      Hq/Hp heads.  m = 1 is one proxy head per GQA group.
  R11 an FP8 e4m3 proxy K (decode) carries one fp32 scale for the single
      shared proxy head, dequantised like R5: logit =
      (pq.pk_code)*pk_scale/sqrt(dp).
  R12 an NVFP4 proxy K (the FP4 block-score indexer) follows the public
      NVFP4 format: e2m1 codes, two per byte with the even dimension in the
      low nibble, one e4m3 scale per 16 consecutive dimensions of a key and
      one fp32 scale for the head; pk = code * block scale * global scale.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

PAGE = 128   # tokens per KV block / page  ([README] "page_size, topk = 128, 16")
TILE = 128   # query rows per tile


# ---------------------------------------------------------------------------
# exact decoding of the stored bit patterns
# ---------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, exactly (bf16 is the upper
    half of an IEEE binary32)."""
    u = np.ascontiguousarray(bits).view(np.uint16).astype(np.uint32) << np.uint32(16)
    # signalling-NaN patterns raise the invalid flag when widened; they stay NaN
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


def e4m3_to_f64(bits) -> np.ndarray:
    """OCP FP8 E4M3 ("e4m3fn") bit patterns -> float64 from the format's
    definition: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent
    field 0 is subnormal (2^-6 * m/8); S.1111.111 is NaN; no infinities."""
    b = np.ascontiguousarray(bits).view(np.uint8).astype(np.int64)
    sign = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = np.ldexp(m / 8.0, -6)
    v = sign * np.where(e == 0, sub, normal)
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return v


def e2m1_to_f64(nibbles) -> np.ndarray:
    """OCP FP4 E2M1 4-bit codes -> float64 from the format's definition:
    1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; exponent field 0
    is subnormal (m * 2^-1); no infinities or NaN."""
    b = np.asarray(nibbles).astype(np.int64) & 0xF
    sign = np.where(b >> 3, -1.0, 1.0)
    e = (b >> 1) & 0x3
    m = b & 0x1
    normal = np.ldexp(1.0 + m / 2.0, (e - 1).astype(np.int64))
    return sign * np.where(e == 0, m * 0.5, normal)


def nvfp4_to_f64(code_bytes, scale_bits, global_scale) -> np.ndarray:
    """NVFP4 values (R12): code bytes [..., D/2] (byte b holds dims 2b in
    its low nibble and 2b+1 in its high nibble), e4m3 block scales
    [..., D/16] (one per 16 consecutive dims) and one fp32 global scale ->
    float64 [..., D] = e2m1(code) * e4m3(block scale) * global_scale."""
    cb = np.ascontiguousarray(code_bytes).view(np.uint8)
    vals = np.stack([e2m1_to_f64(cb & 0xF), e2m1_to_f64(cb >> 4)], axis=-1)
    vals = vals.reshape(cb.shape[:-1] + (2 * cb.shape[-1],))
    sc = np.repeat(e4m3_to_f64(scale_bits), 16, axis=-1)
    return vals * sc * float(global_scale)


# ---------------------------------------------------------------------------
# tiling and page table (R1, R3)
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Tile:
    seq: int        # sequence index in the batch
    q_begin: int    # first global query row of the tile
    q_end: int      # one past the last global query row
    pos0: int       # key position of the tile's first row (R1)
    kv_len: int     # keys in the tile's sequence
    nvp: int        # num_valid_pages: blocks holding a key visible to some row


def kv_indptr(kv_lens) -> np.ndarray:
    """Start of each sequence's pages in the flat kv_indices list: one page
    per 128 keys, ceil(kv_len/128) pages per sequence."""
    nb = [(int(k) + PAGE - 1) // PAGE for k in kv_lens]
    return np.concatenate([[0], np.cumsum(nb)]).astype(np.int64)


def tiles_of(qo_lens, kv_lens) -> list[Tile]:
    """Query tiles of 128 rows, numbered across the whole batch (R1, R3)."""
    out = []
    q0 = 0
    for s, (ql, kl) in enumerate(zip(qo_lens, kv_lens)):
        ql, kl = int(ql), int(kl)
        assert 0 <= ql <= kl
        off = kl - ql
        for t in range((ql + TILE - 1) // TILE):
            r0, r1 = t * TILE, min((t + 1) * TILE, ql)
            last_pos = off + r1 - 1
            out.append(Tile(s, q0 + r0, q0 + r1, off + r0, kl, last_pos // PAGE + 1))
        q0 += ql
    return out


def num_valid_pages(qo_lens, kv_lens) -> np.ndarray:
    return np.array([t.nvp for t in tiles_of(qo_lens, kv_lens)], dtype=np.int32)


def max_blocks(kv_lens) -> int:
    return max([(int(k) + PAGE - 1) // PAGE for k in kv_lens] + [0])


def gather_seq(pages: np.ndarray, kv_indices, indptr, seq: int, kv_len: int) -> np.ndarray:
    """Keys of one sequence in logical order through the page table
    ([README] "kv_indices"): pages [P, H, 128, D] -> [kv_len, H, D]."""
    nb = (kv_len + PAGE - 1) // PAGE
    ids = np.asarray(kv_indices[indptr[seq]: indptr[seq] + nb], dtype=np.int64)
    blocks = pages[ids]                                  # [nb, H, 128, D]
    return blocks.transpose(0, 2, 1, 3).reshape(nb * PAGE, pages.shape[1], pages.shape[3])[:kv_len]


# ---------------------------------------------------------------------------
# stage 1: proxy max score (R2)
# ---------------------------------------------------------------------------

def proxy_max_score(pq_bits, pk_bits, kv_indices, qo_lens, kv_lens, tile_ids=None, pk_scale=None,
                    pk_nvfp4=None):
    """max_score[t, h, j] = max over rows i of tile t and keys k of block j
    with k visible to i of pq[i,h].pk[k]/sqrt(dp), rounded once to fp32;
    -inf where no pair is visible.  pq: [total_q, Hp, dp] bf16 bits;
    pk: [P, 1, 128, dp] bf16 bits (one shared proxy K head, [README]
    "num_kv_heads=1"), or e4m3 codes (uint8) with pk_scale, pk = code *
    pk_scale (R11), or NVFP4 code bytes [P, 1, 128, dp/2] with pk_nvfp4 =
    (block scale bits [P, 1, 128, dp/16], global scale) (R12).  Returns
    float32 [n_tiles, Hp, nb_max]; tiles not in tile_ids stay -inf."""
    # bit patterns are decoded per tile (the decode is exact), so that large
    # page pools never need a float64 copy
    pq_bits, pk_bits = np.asarray(pq_bits), np.asarray(pk_bits)
    tiles = tiles_of(qo_lens, kv_lens)
    indptr = kv_indptr(kv_lens)
    hp, dp = pq_bits.shape[1], pq_bits.shape[2]
    out = np.full((len(tiles), hp, max_blocks(kv_lens)), -np.inf, dtype=np.float64)
    for ti in (range(len(tiles)) if tile_ids is None else tile_ids):
        tl = tiles[ti]
        nk = min(tl.nvp * PAGE, tl.kv_len)
        raw = gather_seq(pk_bits, kv_indices, indptr, tl.seq, tl.kv_len)[:nk, 0, :]
        if pk_nvfp4 is not None:
            sbits = gather_seq(np.asarray(pk_nvfp4[0]), kv_indices, indptr, tl.seq, tl.kv_len)[:nk, 0, :]
            keys = nvfp4_to_f64(raw, sbits, pk_nvfp4[1])                          # [nk, dp]
        elif pk_scale is not None:
            keys = e4m3_to_f64(raw) * float(pk_scale)
        else:
            keys = bf16_to_f64(raw)
        qrows = bf16_to_f64(pq_bits[tl.q_begin: tl.q_end])                     # [R, hp, dp]
        logits = np.matmul(qrows.transpose(1, 0, 2), keys.T) / math.sqrt(dp)   # [hp, R, nk]
        qpos = tl.pos0 + np.arange(tl.q_end - tl.q_begin)
        visible = np.arange(nk)[None, :] <= qpos[:, None]                       # [R, nk]
        logits = np.where(visible[None], logits, -np.inf)
        for j in range(tl.nvp):
            out[ti, :, j] = logits[:, :, j * PAGE: (j + 1) * PAGE].max(axis=(1, 2))
    return out.astype(np.float32)


# ---------------------------------------------------------------------------
# stage 2: top-k block selection (R3)
# ---------------------------------------------------------------------------

def topk_row(scores, nvp: int, topk: int) -> list[int]:
    """Block indexes selected for one (tile, proxy head) row of max_score."""
    jd = nvp - 1
    if topk >= nvp:
        return list(range(nvp))
    cands = [j for j in range(jd) if scores[j] > -np.inf]
    # descending score, then ascending block index; -0.0 == +0.0 here
    cands.sort(key=lambda j: (-float(scores[j]), j))
    return sorted(cands[: topk - 1] + [jd])


def topk_select(max_score, topk: int, nvp) -> np.ndarray:
    """kv_block_indexes [n_tiles, H, topk] int32, ascending, -1 padded
    ([README] sparse_topk_select(max_score, topk, num_valid_pages);
    [FLASH] local block always visible, one block set per proxy head)."""
    ms = np.asarray(max_score, dtype=np.float32)
    n, h, _ = ms.shape
    out = np.full((n, h, topk), -1, dtype=np.int32)
    for t in range(n):
        for g in range(h):
            sel = topk_row(ms[t, g], int(nvp[t]), topk)
            out[t, g, : len(sel)] = sel
    return out


# ---------------------------------------------------------------------------
# stage 3: block-sparse GQA attention (R1, R4, R5)
# ---------------------------------------------------------------------------

def _selected_keys(tl: Tile, idx_row) -> np.ndarray:
    """Logical key positions of the selected blocks, ascending."""
    blocks = [int(j) for j in idx_row if j >= 0]
    ks = [np.arange(j * PAGE, min((j + 1) * PAGE, tl.kv_len)) for j in blocks]
    return np.concatenate(ks) if ks else np.zeros(0, dtype=np.int64)


def _decode_kv(bits, fp8: bool):
    if not fp8:
        return bf16_to_f64(bits)
    # the definition evaluated once on all 256 codes, then looked up by byte
    # (the same values as e4m3_to_f64(bits), without redoing it per element)
    table = e4m3_to_f64(np.arange(256, dtype=np.uint8))
    return table[np.ascontiguousarray(bits).view(np.uint8)]


def sparse_attention(q_bits, k_bits, v_bits, kv_indices, kv_block_indexes, qo_lens, kv_lens,
                     k_scale=None, v_scale=None, tile_ids=None):
    """For query i of tile t and head h (KV head g = h // (Hq/Hkv), proxy
    head p = h // (Hq/Hp), R8): softmax over the keys of the blocks
    kv_block_indexes[t, p, :] that are visible to i of q.k_g/sqrt(d),
    O = P.V_g, LSE = ln sum exp.  Hp is kv_block_indexes.shape[1].  bf16
    K/V, or e4m3 K/V with per-KV-head scales when k_scale/v_scale are given.
    Returns (O, LSE) in float64; rows of tiles not in tile_ids are NaN."""
    fp8 = k_scale is not None
    q_bits, k_bits, v_bits = np.asarray(q_bits), np.asarray(k_bits), np.asarray(v_bits)
    tiles = tiles_of(qo_lens, kv_lens)
    indptr = kv_indptr(kv_lens)
    hq, d = q_bits.shape[1], q_bits.shape[2]
    hkv = k_bits.shape[1]
    grp = hq // hkv
    hs = kv_block_indexes.shape[1]                     # proxy heads = block sets per tile
    assert hs % hkv == 0 and hq % hs == 0
    msa_grp = hq // hs                                 # query heads per proxy head
    o = np.full(q_bits.shape, np.nan)
    lse = np.full(q_bits.shape[:2], np.nan)
    for ti in (range(len(tiles)) if tile_ids is None else tile_ids):
        tl = tiles[ti]
        # only the selected keys' bit patterns are decoded (exactly)
        kseq = gather_seq(k_bits, kv_indices, indptr, tl.seq, tl.kv_len)
        vseq = gather_seq(v_bits, kv_indices, indptr, tl.seq, tl.kv_len)
        qt = bf16_to_f64(q_bits[tl.q_begin: tl.q_end])
        qpos = tl.pos0 + np.arange(tl.q_end - tl.q_begin)
        for h in range(hq):
            g = h // grp
            ks = _selected_keys(tl, kv_block_indexes[ti, h // msa_grp])
            kmat = _decode_kv(kseq[ks, g, :], fp8)
            vmat = _decode_kv(vseq[ks, g, :], fp8)
            if fp8:
                kmat = kmat * float(k_scale[g])
                vmat = vmat * float(v_scale[g])
            s = qt[:, h, :] @ kmat.T / math.sqrt(d)
            s = np.where(ks[None, :] <= qpos[:, None], s, -np.inf)
            m = s.max(axis=1, keepdims=True) if s.shape[1] else np.full((s.shape[0], 1), -np.inf)
            empty = np.isneginf(m)                      # R7: no visible key
            m = np.where(empty, 0.0, m)
            e = np.exp(s - m)
            l = e.sum(axis=1, keepdims=True)
            with np.errstate(divide="ignore", invalid="ignore"):
                lse[tl.q_begin: tl.q_end, h] = np.where(empty, -np.inf, m + np.log(l))[:, 0]
                o[tl.q_begin: tl.q_end, h, :] = np.where(empty, 0.0, (e / np.where(empty, 1.0, l)) @ vmat)
    return o, lse


# ---------------------------------------------------------------------------
# training extension: backward with the KL-coupled proxy gradient (R6)
# ---------------------------------------------------------------------------

def _masked_softmax(s, empty):
    """Row softmax of logits s [R, n] whose masked entries are -inf, and its
    natural-log LSE [R, 1].  Rows flagged in empty [R, 1] (no visible key,
    R7) get probabilities 0 and LSE -inf instead of 0/0."""
    m = np.where(empty, 0.0, s.max(axis=1, keepdims=True, initial=-np.inf))
    e = np.where(empty, 0.0, np.exp(s - m))
    l = np.where(empty, 1.0, e.sum(axis=1, keepdims=True))
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, m + np.log(l))
    return e / l, lse


def sparse_attention_bwd(q_bits, k_bits, v_bits, kv_indices, kv_block_indexes, qo_lens, kv_lens,
                         dout_bits, pq_bits, pk_bits, kl_weight=1.0, tile_ids=None):
    """Gradients of sum(O * dO) with respect to q, k, v restricted to the
    cached blocks, plus the proxy gradients of w * sum_rows KL(p_main ||
    p_proxy), whose logit gradient is w*(p_proxy - p_main) ([FLASH]
    backward-pass paragraph).  bf16 inputs.  Returns a dict of float64
    arrays: dq [total_q,Hq,d], dk, dv [P,Hkv,128,d], dpq [total_q,Hp,dp],
    dpk [P,1,128,dp], plus o and lse of the forward.  Only tiles in tile_ids
    contribute (rows of other tiles in dq/dpq are NaN)."""
    q = bf16_to_f64(q_bits)
    kp = bf16_to_f64(k_bits)
    vp = bf16_to_f64(v_bits)
    do = bf16_to_f64(dout_bits)
    pq = bf16_to_f64(pq_bits)
    pk = bf16_to_f64(pk_bits)
    tiles = tiles_of(qo_lens, kv_lens)
    indptr = kv_indptr(kv_lens)
    hq, d = q.shape[1], q.shape[2]
    hkv = kp.shape[1]
    hs = pq.shape[1]                                   # proxy heads (R8)
    assert kv_block_indexes.shape[1] == hs and hs % hkv == 0 and hq % hs == 0
    msa_grp = hq // hs                                 # query heads per proxy head
    dp = pq.shape[2]
    dq = np.full(q.shape, np.nan)
    dpq = np.full(pq.shape, np.nan)
    dk = np.zeros(kp.shape)
    dv = np.zeros(vp.shape)
    dpk = np.zeros(pk.shape)
    o = np.full(q.shape, np.nan)
    lse = np.full(q.shape[:2], np.nan)
    for ti in (range(len(tiles)) if tile_ids is None else tile_ids):
        tl = tiles[ti]
        rows = slice(tl.q_begin, tl.q_end)
        nb = (tl.kv_len + PAGE - 1) // PAGE
        page_ids = np.asarray(kv_indices[indptr[tl.seq]: indptr[tl.seq] + nb], dtype=np.int64)
        kseq = gather_seq(kp, kv_indices, indptr, tl.seq, tl.kv_len)
        vseq = gather_seq(vp, kv_indices, indptr, tl.seq, tl.kv_len)
        pkseq = gather_seq(pk, kv_indices, indptr, tl.seq, tl.kv_len)[:, 0, :]
        qpos = tl.pos0 + np.arange(tl.q_end - tl.q_begin)
        for hp_ in range(hs):
            g = hp_ // (hs // hkv)                       # KV head of proxy head hp_
            ks = _selected_keys(tl, kv_block_indexes[ti, hp_])
            vis = ks[None, :] <= qpos[:, None]
            # R7: a row that sees no selected key has P = 0, O = 0, LSE = -inf,
            # and so no gradient; its proxy distribution is empty as well
            # (p_proxy = 0), which makes its KL term and dZ zero
            empty = ~vis.any(axis=1, keepdims=True)                      # [R, 1]
            kmat, vmat = kseq[ks, g, :], vseq[ks, g, :]
            dkmat = np.zeros_like(kmat)
            dvmat = np.zeros_like(vmat)
            p_main = np.zeros(vis.shape)
            for h in range(hp_ * msa_grp, (hp_ + 1) * msa_grp):
                s = np.where(vis, q[rows, h, :] @ kmat.T / math.sqrt(d), -np.inf)
                p, lse_h = _masked_softmax(s, empty)                    # [R, n], [R, 1]
                oh = p @ vmat
                o[rows, h, :] = oh
                lse[rows, h] = lse_h[:, 0]
                dov = do[rows, h, :]
                dP = dov @ vmat.T
                D = (dov * oh).sum(axis=1, keepdims=True)
                dS = p * (dP - D)
                dq[rows, h, :] = dS @ kmat / math.sqrt(d)
                dkmat += dS.T @ q[rows, h, :] / math.sqrt(d)
                dvmat += p.T @ dov
                p_main += p / msa_grp
            # proxy distribution over the same selected, visible keys
            z = np.where(vis, pq[rows, hp_, :] @ pkseq[ks].T / math.sqrt(dp), -np.inf)
            p_proxy, _ = _masked_softmax(z, empty)
            dz = kl_weight * (p_proxy - p_main)
            dpq[rows, hp_, :] = dz @ pkseq[ks] / math.sqrt(dp)
            dpk_keys = dz.T @ pq[rows, hp_, :] / math.sqrt(dp)          # [n, dp]
            # scatter per-key gradients back to physical pages
            pg = page_ids[ks // PAGE]
            np.add.at(dk, (pg, g, ks % PAGE), dkmat)
            np.add.at(dv, (pg, g, ks % PAGE), dvmat)
            np.add.at(dpk, (pg, 0, ks % PAGE), dpk_keys)
    return dict(dq=dq, dk=dk, dv=dv, dpq=dpq, dpk=dpk, o=o, lse=lse)


def kl_objective(pq, pk, q_bits, k_bits, kv_indices, kv_block_indexes, qo_lens, kv_lens,
                 kl_weight=1.0):
    """w * sum over rows and proxy heads of KL(p_main || p_proxy) as a function of
    float64 proxy inputs pq [total_q,Hp,dp], pk [P,1,128,dp], with p_main
    from the bf16 main q/k (held fixed).  Used to pin the closed-form proxy
    gradient by finite differences."""
    q = bf16_to_f64(q_bits)
    kp = bf16_to_f64(k_bits)
    tiles = tiles_of(qo_lens, kv_lens)
    indptr = kv_indptr(kv_lens)
    hq, d = q.shape[1], q.shape[2]
    hkv = kp.shape[1]
    hs = pq.shape[1]
    msa_grp = hq // hs
    dp = pq.shape[2]
    total = 0.0
    for ti, tl in enumerate(tiles):
        rows = slice(tl.q_begin, tl.q_end)
        kseq = gather_seq(kp, kv_indices, indptr, tl.seq, tl.kv_len)
        pkseq = gather_seq(pk, kv_indices, indptr, tl.seq, tl.kv_len)[:, 0, :]
        qpos = tl.pos0 + np.arange(tl.q_end - tl.q_begin)
        for hp_ in range(hs):
            g = hp_ // (hs // hkv)
            ks = _selected_keys(tl, kv_block_indexes[ti, hp_])
            vis = ks[None, :] <= qpos[:, None]
            empty = ~vis.any(axis=1, keepdims=True)        # R7 rows contribute nothing
            p_main = np.zeros(vis.shape)
            for h in range(hp_ * msa_grp, (hp_ + 1) * msa_grp):
                s = np.where(vis, q[rows, h, :] @ kseq[ks, g, :].T / math.sqrt(d), -np.inf)
                p_main += _masked_softmax(s, empty)[0] / msa_grp
            z = np.where(vis, pq[rows, hp_, :] @ pkseq[ks].T / math.sqrt(dp), -np.inf)
            _, lse_z = _masked_softmax(z, empty)
            with np.errstate(divide="ignore", invalid="ignore"):
                log_pp = z - lse_z
                terms = np.where(p_main > 0, p_main * (np.log(p_main) - log_pp), 0.0)
            total += kl_weight * terms.sum()
    return total
