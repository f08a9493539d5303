/*
 * libmsa -- the MiniMax Sparse Attention (MSA) hot path on one NVIDIA GB300
 * (sm_103a), as a C ABI.
 *
 * The method (sources named by page title and section):
 *   [README] "MiniMax-AI/MSA" README (pigsec.cn mirror), section "Usage":
 *            a dense proxy pass (plan with num_kv_heads=1,
 *            output_maxscore=True) gives a per-block max score;
 *            sparse_topk_select(max_score, topk, num_valid_pages) turns it
 *            into kv_block_indexes; a plan with kv_block_num=topk runs
 *            attention over only those blocks of the paged K/V
 *            (k_pages, v_pages, kv_indices), page_size 128.
 *   [STACKS] same README, section "Stacks": paged FP8 decode
 *            (SparseDecodePagedAttentionWrapper) next to BF16 sparse prefill.
 *   [FLASH]  iitog.ru, "Flash-MSA: open kernels for training models with
 *            sparse attention on millions of tokens": whole 128-token blocks
 *            chosen by max-pooling proxy scores; GQA main attention; one
 *            block set per proxy head / GQA group; the token's own block is
 *            always visible; indexes cached from the forward feed the
 *            backward; the KL-loss gradient with respect to a proxy score is
 *            p_proxy - p_main.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every tensor argument is a DEVICE pointer to a dense row-major array
 *    owned by the caller; layouts are given per call.  The library never
 *    frees or retains them past the call.
 *  - Compute calls enqueue work on `stream` and return without waiting; they
 *    allocate nothing (any scratch lives in the plan, allocated once by
 *    msa_plan) and never synchronise the host.
 *  - Tiles: a sequence with qo_len query rows and kv_len keys (qo_len <=
 *    kv_len) places row r at key position kv_len - qo_len + r (bottom-right
 *    causal alignment) and row r sees key k iff k <= that position.  Query
 *    rows are cut into tiles of 128 rows per sequence; tiles are numbered
 *    across the batch in sequence order ("global tile index").  Tile t's
 *    num_valid_pages is the number of 128-key blocks up to and including the
 *    block of its last row's position; that last block is its diagonal
 *    block.
 *  - Page table: kv_indices is the flat list of physical page ids, sequence
 *    by sequence, ceil(kv_len/128) entries per sequence (logical block j of
 *    sequence s is page kv_indices[sum_{s'<s} ceil(kv_len_s'/128) + j]).
 *    Page ids must lie in [0, num_pages); a kernel that meets one outside
 *    skips that block and raises MSA_ERR_DEVICE_CHECK in the plan's error
 *    word (read with msa_check_errors).
 *  - Errors: host-side argument checks return MSA_ERR_INVALID_ARG or
 *    MSA_ERR_UNSUPPORTED before anything is enqueued; a failed launch
 *    returns MSA_ERR_CUDA.  msa_last_error() gives a message for the
 *    calling thread's last failure.
 *  - NaN inputs are outside the contract and are not scanned for.  A plan
 *    created while the environment variable MSA_CHECKS is set (to anything
 *    but "0") adds, after each of its calls, scans of that call's
 *    floating-point inputs (the query-side arrays q, pq, dout, and the pages
 *    of k/v/pk that kv_indices names; bf16 or e4m3, not the NVFP4 codes) and
 *    outputs (max_score, out, lse, dq, dpq; not dk/dv/dpk, whose unreferenced
 *    pages keep the caller's contents), and raises MSA_ERR_NONFINITE in the
 *    error word when one holds a NaN.  -inf in max_score and lse is a
 *    defined value (no visible key) and is not flagged.  Each scan is one
 *    read of its array.
 */
#ifndef MSA_H
#define MSA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* msa_stream_t;

typedef enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1,   /* bad pointer, size or layout */
  MSA_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels implement */
  MSA_ERR_CUDA = 3,          /* CUDA runtime / launch failure */
  MSA_ERR_NO_MEMORY = 4,     /* plan workspace allocation failed */
  MSA_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up */
  MSA_ERR_DEVICE_CHECK = 6,  /* a device-side bounds check fired (bad page id) */
  MSA_ERR_NONFINITE = 7      /* MSA_CHECKS: a NaN reached an output */
} msa_status;

typedef enum {
  MSA_KV_BF16 = 0,           /* K/V pages are bfloat16 */
  MSA_KV_FP8_E4M3 = 1        /* K/V pages are OCP e4m3 with one fp32 scale per KV head */
} msa_kv_dtype;

typedef struct msa_plan_s* msa_plan_t;

/*
 * msa_plan -- validate a batch shape and build the device tables every
 * other call reads ([README] "Usage": fmha_sm100_plan(qo_lens, kv_lens,
 * heads, num_kv_heads, page_size, kv_block_num=topk)).
 *
 *  qo_lens, kv_lens  HOST int32[batch]; 0 <= qo_lens[s] <= kv_lens[s],
 *                    kv_lens[s] >= 1, and at least one qo_lens[s] > 0 (a
 *                    sequence with qo_len 0 has no tiles; its pages keep
 *                    their page-table entries).  Otherwise
 *                    MSA_ERR_INVALID_ARG.  Copied; the caller keeps
 *                    ownership.
 *  num_qo_heads      Hq, query heads of the main attention.
 *  num_kv_heads      Hkv, KV heads (GQA groups); Hq % Hkv == 0.
 *  num_proxy_heads   Hp, proxy query heads, a multiple of Hkv that divides
 *                    Hq ([FLASH]: at least one proxy head per GQA group,
 *                    each with its own block set).  Proxy head p serves
 *                    query heads [p*Hq/Hp, (p+1)*Hq/Hp), all of KV head
 *                    p / (Hp/Hkv): with Hp = Hkv that is one proxy head per
 *                    GQA group; with Hp = m*Hkv each group's query heads
 *                    split into m sets with a block set each.
 *  head_dim          d in {64, 128}.
 *  proxy_head_dim    dp in {32, 64}.
 *  page_size         must be 128 ([README] "page_size, topk = 128, 16").
 *  topk              K >= 1 selected blocks per (tile, proxy head), the
 *                    diagonal block included.
 *  num_pages         physical pages in the K/V page pool (and the proxy K
 *                    pool, which shares page ids).
 *  kv_dtype          element type of k_pages / v_pages.
 *  flags             reserved, pass 0.
 *  stream            stream for the one host->device copy of the tables.
 *  out               receives the plan; release with msa_plan_destroy.
 *
 * Allocates the plan's device tables and workspace (this is the only call
 * that allocates) and waits for their upload.
 */
msa_status msa_plan(const int32_t* qo_lens, const int32_t* kv_lens, int32_t batch,
                    int32_t num_qo_heads, int32_t num_kv_heads, int32_t num_proxy_heads,
                    int32_t head_dim, int32_t proxy_head_dim, int32_t page_size, int32_t topk,
                    int64_t num_pages, msa_kv_dtype kv_dtype, uint32_t flags,
                    msa_stream_t stream, msa_plan_t* out);

void msa_plan_destroy(msa_plan_t plan);

/* Shape queries of a plan. */
int32_t msa_plan_num_tiles(msa_plan_t plan);     /* tiles across the batch */
int32_t msa_plan_max_blocks(msa_plan_t plan);    /* max_s ceil(kv_len_s/128) */
int64_t msa_plan_total_q(msa_plan_t plan);       /* sum of qo_lens */
/* DEVICE int32[num_tiles]: num_valid_pages per tile (owned by the plan). */
const int32_t* msa_plan_num_valid_pages(msa_plan_t plan);

/*
 * msa_proxy_maxscore -- stage 1, the proxy pass ([README] "Usage": dense
 * proxy pass with output_o=False, output_maxscore=True; [FLASH]: blocks of
 * 128 tokens chosen by max-pooling over proxy scores).
 *
 *   max_score[t, h, j] = max over rows i of tile t and keys k of block j
 *                        with k visible to i of  pq[i,h] . pk[k] / sqrt(dp)
 *                        (-inf where no pair is visible, and for j beyond
 *                        the tile's num_valid_pages).
 *
 *  pq         bf16 [total_q, Hp, dp].
 *  pk_pages   bf16 [num_pages, 1, 128, dp]: one shared proxy K head, paged
 *             with the same kv_indices as the main K/V.
 *  kv_indices int32 page table (see conventions).
 *  max_score  fp32 [num_tiles, Hp, max_blocks], written entirely.
 * The proxy V of the reference call is not taken: nothing reads it when no
 * output O is produced.
 */
msa_status msa_proxy_maxscore(msa_plan_t plan, const void* pq, const void* pk_pages,
                              const int32_t* kv_indices, float* max_score, msa_stream_t stream);

/*
 * msa_proxy_maxscore_fp8 -- stage 1 at decode with the proxy K stored as
 * FP8 e4m3 ("MiniMax-AI/MSA" README, section "Stacks": the FP8 paged decode
 * stack; an FP8 proxy K halves the proxy scan, which is the largest read of
 * a decode step).  The logit of a pair is (pq[i,h] . pk_code[k]) *
 * pk_scale[0] / sqrt(dp), the same dequantisation as the FP8 main K;
 * otherwise max_score is defined as in msa_proxy_maxscore.
 *
 *  pq         bf16 [total_q, Hp, dp].
 *  pk_pages   e4m3 codes [num_pages, 1, 128, dp], 16-byte aligned.
 *  pk_scale   device pointer to one fp32 scale (> 0) for the shared proxy head.
 * Plans whose sequences all have qo_len = 1, dp = 64 and Hp <= 8 only;
 * others return MSA_ERR_UNSUPPORTED.
 */
msa_status msa_proxy_maxscore_fp8(msa_plan_t plan, const void* pq, const void* pk_pages,
                                  const float* pk_scale, const int32_t* kv_indices, float* max_score,
                                  msa_stream_t stream);

/*
 * msa_proxy_maxscore_nvfp4 -- stage 1 at decode with the proxy K stored in
 * NVFP4, the FP4 block-score indexer ("MiniMax-AI/MSA" README, section
 * "Stacks": the FP4 block-score indexer; Flash-MSA article, "what's next":
 * the indexer in low precision).  The shared proxy head's keys are e2m1
 * codes with one e4m3 scale per 16 consecutive dimensions and one fp32
 * scale for the head:
 *   pk[k, d] = e2m1(code[k, d]) * e4m3(block_scale[k, d / 16]) * global_scale
 * and the logit of a pair is pq[i,h] . pk[k] / sqrt(dp); otherwise max_score
 * is defined as in msa_proxy_maxscore.  The proxy K read is a quarter of the
 * bf16 one (plus 1/8 for the scales).
 *
 *  pq               bf16 [total_q, Hp, dp].
 *  pk_codes         uint8 [num_pages, 1, 128, dp / 2], 16-byte aligned: byte
 *                   b of a key holds dims 2b (low nibble) and 2b + 1 (high
 *                   nibble), each e2m1 (1 sign, 2 exponent bits with bias 1,
 *                   1 mantissa bit; exponent 0 is 0 or 0.5).
 *  pk_block_scales  e4m3 [num_pages, 1, 128, dp / 16], 16-byte aligned.
 *  pk_global_scale  device pointer to one fp32 scale (> 0).
 * Decode plans (every qo_len == 1) with dp = 64 and Hp <= 8 only; others
 * return MSA_ERR_UNSUPPORTED.  The products run on f16 tensor cores with pq
 * rounded to f16 (exact for |pq| in [2^-14, 65504]); code * block scale is
 * exact in f16.
 */
msa_status msa_proxy_maxscore_nvfp4(msa_plan_t plan, const void* pq, const void* pk_codes,
                                    const void* pk_block_scales, const float* pk_global_scale,
                                    const int32_t* kv_indices, float* max_score, msa_stream_t stream);

/*
 * msa_topk_select -- stage 2 ([README] sparse_topk_select(max_score, topk,
 * num_valid_pages); [FLASH]: each proxy head picks its own block set, the
 * local block is always visible).  Plan-free, like the reference call.
 *
 * For each row (t, h) with n = num_valid_pages[t] and diagonal block
 * j_d = n - 1: if topk >= n the row selects blocks 0..n-1; otherwise it
 * selects j_d plus the topk-1 largest max_score[t,h,j] over j < j_d,
 * ignoring -inf, ordered by (score descending, j ascending); -0.0 and +0.0
 * are equal.  Selected indexes are written ascending, padded with -1.
 * Scores are compared exactly (bit-exact result); NaN inputs are outside
 * the contract.
 *
 *  max_score        fp32 [n_tiles, heads, max_blocks].
 *  num_valid_pages  int32 [n_tiles], each in [1, max_blocks].  A row whose
 *                   value lies outside that range selects nothing: it is
 *                   written as topk entries of -1 (the attention then
 *                   treats its query rows as seeing no key).
 *  kv_block_indexes int32 [n_tiles, heads, topk] (output).
 *  1 <= topk <= 1024, max_blocks <= 65536.
 */
msa_status msa_topk_select(const float* max_score, int32_t n_tiles, int32_t heads,
                           int32_t max_blocks, int32_t topk, const int32_t* num_valid_pages,
                           int32_t* kv_block_indexes, msa_stream_t stream);

/*
 * msa_proxy_topk -- stages 1 and 2 fused ([FLASH], kernel-design
 * paragraph: the forward proxy pass keeps a streaming top-k over blocks in
 * registers instead of accumulating outputs).  The proxy pass and the
 * selection of msa_proxy_maxscore + msa_topk_select in one launch, with no
 * max_score round trip.
 *
 * Writes the same kv_block_indexes as msa_topk_select(max_score, ...,
 * plan topk, msa_plan_num_valid_pages(plan), ...) would on the scores that
 * msa_proxy_maxscore writes: bit-exact, ties to the lower block, ascending,
 * -1 padded.  The work units of one tile report their candidates and the
 * last of them merges; nothing waits on another CTA.
 *
 *  pq, pk_pages, kv_indices  as for msa_proxy_maxscore.
 *  max_score         fp32 [num_tiles, Hp, max_blocks] (output) or NULL.
 *  kv_block_indexes  int32 [num_tiles, Hp, topk] (output).
 * Prefill plans with topk <= 32 and at most 1024 blocks per sequence;
 * others return MSA_ERR_UNSUPPORTED (use the two separate calls).  The
 * plan's counters are reset by every complete launch, so two calls on one
 * plan must not overlap in time; after a launch that failed with a device
 * error the plan must be rebuilt.
 */
msa_status msa_proxy_topk(msa_plan_t plan, const void* pq, const void* pk_pages,
                          const int32_t* kv_indices, float* max_score, int32_t* kv_block_indexes,
                          msa_stream_t stream);

/*
 * msa_sparse_attn -- stage 3, GQA block-sparse attention forward ([README]
 * "Usage": fmha_sm100(q, k_pages, v_pages, sparse_plan, kv_indices,
 * kv_block_indexes); [STACKS]: paged FP8 decode; [FLASH]: GQA main
 * attention over the selected blocks).
 *
 * For query row i of tile t and head h (KV head g = h / (Hq/Hkv), proxy
 * head p = h / (Hq/Hp)): softmax over the keys k of KV head g in blocks
 * kv_block_indexes[t, p, :] (entries < 0 are skipped) with k visible to i
 * of s = q[i,h].k[k] / sqrt(d); out = P.V, lse = natural-log logsumexp of
 * s.  With FP8 K/V: s uses k*k_scale[g] and V is v*v_scale[g]
 * ([STACKS]: FP8 for the paged decode and the sparse prefill).
 *
 *  q                 bf16 [total_q, Hq, d].
 *  k_pages, v_pages  [num_pages, Hkv, 128, d], bf16 or e4m3 per the plan
 *                    (e4m3 prefill: head_dim 128; the MMAs run in f16, with
 *                    q rounded to f16, exact for |q| in [2^-14, 65504]).
 *  kv_indices        int32 page table.
 *  kv_block_indexes  int32 [num_tiles, Hp, topk], as msa_topk_select writes
 *                    them.  Any order of distinct valid blocks is accepted,
 *                    with -1 entries anywhere.  In prefill a query row that
 *                    sees no key of its selection gets out = 0 and
 *                    lse = -inf (a row of only -1 included); decode
 *                    selections must hold the diagonal (last) block.
 *  k_scale, v_scale  fp32 [Hkv] for FP8 K/V, NULL for bf16.
 *  out               bf16 [total_q, Hq, d] (output).
 *  lse               fp32 [total_q, Hq] (output) or NULL.
 * Decode batches (every qo_len == 1) run a split-K kernel whose partial
 * results live in the plan's workspace: two calls on one plan must not
 * overlap in time (issue them on one stream, or order the streams).
 */
msa_status msa_sparse_attn(msa_plan_t plan, const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* kv_indices, const int32_t* kv_block_indexes,
                           const float* k_scale, const float* v_scale,
                           void* out, float* lse, msa_stream_t stream);

/*
 * msa_sparse_attn_bwd -- training extension: the fused backward ([FLASH]
 * backward-pass paragraph: the KL between the proxy and main attention
 * distributions needs both, so both gradients come from one pass; the KL
 * gradient with respect to a proxy logit is p_proxy - p_main; block indexes
 * are the ones cached from the forward).
 *
 * Main part, restricted to the cached blocks and the causal mask, for the
 * scalar sum(out * dout):  D = rowsum(dout*out), dS = P*(dP - D),
 * dq = dS.K/sqrt(d), dk = dS^T.q/sqrt(d) and dv = P^T.dout summed over the
 * heads (and selections) of a KV head.  KL part, per row i and proxy head p
 * over the same keys as p's query heads: p_main = mean of the P of the
 * Hq/Hp heads that use p's blocks (no gradient), p_proxy = softmax of
 * pq[i,p].pk/sqrt(dp), dZ = kl_weight*(p_proxy - p_main), dpq =
 * dZ.pk/sqrt(dp), dpk = dZ^T.pq/sqrt(dp).  A page named by several
 * page-table entries (a shared prefix) gets the sum over all of them in
 * dk_pages, dv_pages and dpk_pages.  Rows that see no key of their
 * selection get dq = 0 and dpq = 0 and add nothing elsewhere.
 *
 *  q, k_pages, v_pages, kv_indices, kv_block_indexes  as in the forward
 *                    (bf16 K/V only).
 *  out, lse          the forward's bf16 out and fp32 lse.
 *  dout              bf16 [total_q, Hq, d].
 *  pq, pk_pages      the proxy inputs of msa_proxy_maxscore.
 *  dq                fp32 [total_q, Hq, d]            (output, overwritten)
 *  dk_pages,dv_pages fp32 [num_pages, Hkv, 128, d]    (output; pages the
 *                    plan's sequences reference are overwritten, others
 *                    untouched)
 *  dpq               fp32 [total_q, Hp, dp]           (output, overwritten)
 *  dpk_pages         fp32 [num_pages, 1, 128, dp]     (output, as dk_pages)
 * q, k_pages, v_pages, out, dout, pq and pk_pages must be 16-byte aligned and
 * the five gradients 32-byte aligned (MSA_ERR_INVALID_ARG otherwise).
 */
msa_status msa_sparse_attn_bwd(msa_plan_t plan, const void* q, const void* k_pages,
                               const void* v_pages, const int32_t* kv_indices,
                               const int32_t* kv_block_indexes, const void* out, const float* lse,
                               const void* dout, const void* pq, const void* pk_pages,
                               float kl_weight, float* dq, float* dk_pages, float* dv_pages,
                               float* dpq, float* dpk_pages, msa_stream_t stream);

/*
 * msa_sparse_decode_noalloc -- the FP8 paged decode of msa_sparse_attn for
 * callers that cannot allocate device memory when they decode (for example
 * a server that gives the GPU's memory to its own pool at start-up, or a
 * decode loop that must not pay for cudaMalloc's implicit synchronisation;
 * neither can create a plan, since msa_plan allocates).  The paper has no
 * counterpart: this is a deployment variant of the decode kernel.
 *
 * Computes exactly what msa_sparse_attn computes for a decode batch (one
 * query row per sequence) with e4m3 K/V, head_dim 128, up to 16 query heads
 * per KV head.  The batch comes as DEVICE arrays instead of a plan:
 *   kv_lens    int32 [batch], keys per sequence (>= 1);
 *   kv_indptr  int32 [batch+1], offset of each sequence's pages in
 *              kv_indices (kv_indptr[s+1] - kv_indptr[s] >= ceil(kv_len/128)).
 * q, k_pages, v_pages, kv_indices, kv_block_indexes ([batch, Hkv, topk]),
 * k_scale, v_scale, out and lse (nullable) are as in msa_sparse_attn.
 * err_word: optional DEVICE uint32 that the kernels OR status bits into;
 * NULL discards them.  Bit 0: a device-side bounds check fired (a bad page
 * id or page range; that block is skipped or read from page 0).  Bit 1: a
 * bounded device-side wait gave up; the call's out and lse are then
 * unspecified.  The caller clears the word.
 *
 * Scratch: all of it (a tile table and the split-K partials) lives in one
 * fixed 24 MiB device array inside libmsa, held by every GPU that loads the
 * library until the process exits.  The call allocates nothing and calls no
 * allocating routine.  Each call clears the split-K counters of its own rows
 * before using them, so a call that failed does not disturb later ones.  It rejects, with MSA_ERR_INVALID_ARG, batch > 4096 or
 * batch * num_qo_heads * topk above 47,639 (the partials that fit in the
 * array at head_dim 128) or batch * num_kv_heads above 65,536.  The first call on a device looks up the array's
 * device address for that device (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  Every call on a
 * device shares the one array and overwrites what it needs: calls that
 * overlap on the GPU (other streams, or other host threads) race and give
 * wrong results; issue them one after another.
 */
msa_status msa_sparse_decode_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                     const int32_t* kv_lens, const int32_t* kv_indptr,
                                     const int32_t* kv_indices, const int32_t* kv_block_indexes,
                                     const float* k_scale, const float* v_scale, int32_t batch,
                                     int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                                     int32_t topk, int64_t num_pages, void* out, float* lse,
                                     uint32_t* err_word, msa_stream_t stream);

/*
 * msa_check_errors -- waits for `stream`, then reads and clears the plan's
 * device error word: MSA_OK, MSA_ERR_TIMEOUT (a bounded wait inside a kernel
 * gave up; that kernel's outputs are unspecified), MSA_ERR_DEVICE_CHECK (a
 * kernel skipped a block whose page id was out of range) or, for plans
 * created under MSA_CHECKS, MSA_ERR_NONFINITE (an output held a NaN), in
 * that order when several are set.
 */
msa_status msa_check_errors(msa_plan_t plan, msa_stream_t stream);

/*
 * msa_selftest_wait_timeout -- the failure-detection path, on the device:
 * launches one kernel whose bounded mbarrier wait cannot complete (nothing
 * arrives on the barrier).  The wait gives up after its 2 s limit, the
 * kernel records the timeout in an error word and returns, the context stays
 * usable, and the call reports what msa_check_errors reports for any kernel
 * whose wait ran out: MSA_ERR_TIMEOUT.  Any other error word gives
 * MSA_ERR_CUDA.  Synchronises `stream`; allocates and frees 4 bytes.
 */
msa_status msa_selftest_wait_timeout(msa_stream_t stream);

/*
 * msa_test_fail_plan_allocs -- failure injection on the host, for tests of a
 * caller's out-of-memory handling: the next `count` calls of msa_plan that
 * reach their device allocation fail there exactly as a failed cudaMalloc
 * does (MSA_ERR_NO_MEMORY, nothing allocated, *out left NULL), without
 * calling cudaMalloc.  count <= 0 cancels what is left.  Process-wide.
 */
void msa_test_fail_plan_allocs(int32_t count);

/* Message for the calling thread's last failed call ("" if none). */
const char* msa_last_error(void);

/* Library version, "major.minor.patch". */
const char* msa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MSA_H */
