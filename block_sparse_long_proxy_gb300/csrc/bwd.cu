// Training extension: the backward of block-sparse GQA attention on the
// cached blocks, fused with the KL-coupled proxy gradient (Flash-MSA
// article, backward-pass paragraph: the KL between proxy and main attention
// needs both distributions, so both gradients come from one backward; the
// gradient of the KL loss with respect to a proxy score is p_proxy - p_main;
// the block indexes are the ones cached by the forward).
//
// For row i, head h (KV head g, proxy head p: the G = Hq/Hp heads of p use
// p's blocks), key set Omega = visible keys of the cached blocks of (tile, p):
//   P = exp(q.k/sqrt(d) - lse), D = rowsum(dout*out), dS = P*(dout.v - D)
//   dq = dS.K/sqrt(d), dk = sum_h dS^T.q/sqrt(d), dv = sum_h P^T.dout
//   p_proxy = softmax_Omega(pq_p.pk/sqrt(dp)), p_main = mean over p's heads of P
//   dZ = w*(p_proxy - p_main), dpq = dZ.pk/sqrt(dp), dpk = dZ^T.pq/sqrt(dp)
// Both dpq and dpk split into a proxy term and a main term:
//   dpq = w/sqrt(dp) * (p_proxy.pk - (1/G) sum_h P_h.pk)
//   dpk = w/sqrt(dp) * (p_proxy^T.pq - (1/G) sum_h P_h^T.pq)
//
// Kernels, in stream order:
//   proxy    the proxy softmax over Omega on the tensor cores: the forward
//            attention kernel (attn_fwd.cu) with pq as queries and the shared
//            proxy K head as keys and values gives p_proxy . pk and its LSE
//   prep     per (tile, proxy head p): D of p's heads and lse * log2(e),
//            both stored [head][row]; the proxy LSE in log2 units
//            ([proxy head][row]) and dpq's proxy term (plain store)
//   index    page owners, then the page -> selections inverse index
//   dq       per (tile, proxy head), tcgen05 (bwd_dq.cu): the proxy head's
//            G query heads one after the other; dq (owned, plain store) and
//            dpq's main term (accumulated over the G heads in tensor memory,
//            then added to the proxy term)
//   dkv      per (physical page, group), tcgen05 (bwd_dkv.cu): loops over
//            the selections of the page by any page-table entry (sorted, so
//            sums are deterministic); dk, dv (owned, plain store) and dpk
//            (both terms; a partial per KV head, the last of them adds them
//            in KV-head order)
// No gradient is reduced by atomics: every sum has a fixed order, so the
// backward gives the same bits on every run.
//
// The tensor-core kernels are built for d = 128 and dp = 64.  At d = 64 or
// dp = 32 they read q, out, dout, K, V, pq and pk through tensor maps of the
// true width with the same 64-column boxes: the columns past the edge arrive
// as zeros, every contraction over d (or dp) is unchanged, and the products
// whose columns run over d (dq, dk, dv) or dp (dpq, dpk) have zeros there,
// which the kernels do not store.  The scales are those of the true widths.

#include "msa_internal.h"
#include "ptx.cuh"

#include <algorithm>
#include <vector>

namespace msa {
namespace {

constexpr int kDP = 64;    // columns of the proxy softmax's Op and of the partials
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ prep

// Per (tile, proxy head g): D[row, h] = rowsum(dout * out) and lse * log2(e)
// of the G query heads that use g's blocks, both stored [head][row]; the
// proxy LSE of g in log2 units, [proxy head][row]; and dpq's proxy term
// w/sqrt(dp) * p_proxy . pk, from the proxy softmax (launch_proxy_softmax)
// run just before.  out and dout are [total_q, Hq, d] (d = 64 or 128), dpq
// [total_q, Hp, dp] (dp = 32 or 64); the proxy softmax's Op keeps 64 columns.
__global__ void __launch_bounds__(kThreads)
    bwd_prep_kernel(const TileInfo* __restrict__ tiles, const __nv_bfloat16* __restrict__ out,
                    const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse,
                    const __nv_bfloat16* __restrict__ op, const float* __restrict__ lse_p,
                    float* __restrict__ dsumt, float* __restrict__ lse2t, float* __restrict__ lsept,
                    float* __restrict__ dpq, int32_t hq, int32_t hsel, int32_t total_q, int32_t d, int32_t dp,
                    float kl_weight) {
  pdl_wait();  // launched with programmatic dependent launch: the previous kernel's writes first
  const int t = blockIdx.x / hsel, g = blockIdx.x % hsel;
  const TileInfo tl = tiles[t];
  const int lane = threadIdx.x & 31;
  const int G = hq / hsel;

  // D = rowsum(dout * out): eight lanes per (row, head), d / 8 values each
  // (two 16-byte loads apiece at d = 128, one at d = 64), so that every
  // thread has its few loads in flight at once and the block's 256 threads
  // cover 32 rows per pass
  static_assert(kThreads % 8 == 0 && 128 % (kThreads / 8) == 0, "row passes");
  const int sub = lane & 7;
  const int nv = d >> 6;  // 16-byte loads per lane
  for (int e = threadIdx.x >> 3; e < G * 128; e += kThreads / 8) {
    const int h = g * G + e / 128, r = e % 128;
    float acc = 0.f;
    if (r < tl.rows) {
      const int64_t off = (static_cast<int64_t>(tl.q_begin + r) * hq + h) * d + sub * nv * 8;
      const uint4* a = reinterpret_cast<const uint4*>(out + off);
      const uint4* b = reinterpret_cast<const uint4*>(dout + off);
      const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
      const uint4 x0 = a[0], y0 = b[0];
      const uint4 x1 = nv > 1 ? a[1] : zero, y1 = nv > 1 ? b[1] : zero;
      const uint32_t xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const uint32_t ys[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float2 fx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[c]));
        const float2 fy = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[c]));
        acc += fx.x * fy.x + fx.y * fy.y;
      }
    }
    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 2);
    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 4);
    if (sub == 0 && r < tl.rows) {
      const int64_t q_row = tl.q_begin + r;
      dsumt[static_cast<int64_t>(h) * total_q + q_row] = acc;
      lse2t[static_cast<int64_t>(h) * total_q + q_row] = lse[q_row * hq + h] * kLog2e;
    }
  }

  // proxy LSE in log2 units, and dpq's proxy term
  const float f = kl_weight * rsqrtf(static_cast<float>(dp));
  for (int r = threadIdx.x; r < tl.rows; r += blockDim.x) {
    const int64_t q_row = tl.q_begin + r;
    lsept[static_cast<int64_t>(g) * total_q + q_row] = lse_p[q_row * hsel + g] * kLog2e;
  }
  const int cpr = dp / 8;  // 8-column groups of a dpq row
  for (int e = threadIdx.x; e < tl.rows * cpr; e += blockDim.x) {
    const int r = e / cpr, c = e % cpr;
    const int64_t row = static_cast<int64_t>(tl.q_begin + r) * hsel + g;
    const uint4 v = *reinterpret_cast<const uint4*>(op + row * kDP + c * 8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float4* dst = reinterpret_cast<float4*>(dpq + row * dp + c * 8);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[2 * k]));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[2 * k + 1]));
      dst[k] = make_float4(lo.x * f, lo.y * f, hi.x * f, hi.y * f);
    }
  }
}

// ------------------------------------------------------------ inverse index
//
// The key-side kernel has one CTA per (page-table entry, group) and writes
// dK / dV of the entry's physical page with plain stores.  Several entries
// may name one physical page (a prefix shared by sequences), so every
// selection is filed under the page's owner, the lowest entry that names
// it; the owner's CTA sums the contributions of all of them and the other
// entries' CTAs leave the page alone.

// owner[page] = min over entries e with kv_indices[e] == page of e (owner
// starts at INT_MAX).  Entries with a page id out of range own themselves.
__global__ void bwd_owner_kernel(const int32_t* __restrict__ kv_indices, int32_t n_entries, int64_t num_pages,
                                 int32_t* __restrict__ owner) {
  pdl_wait();  // launched with programmatic dependent launch: the previous kernel's writes first
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n_entries) return;
  const int64_t page = kv_indices[e];
  if (page >= 0 && page < num_pages) atomicMin(owner + page, e);
}

__device__ __forceinline__ int32_t owner_of(const int32_t* __restrict__ kv_indices, const int32_t* __restrict__ owner,
                                            int64_t num_pages, int32_t e) {
  const int64_t page = kv_indices[e];
  return (page >= 0 && page < num_pages) ? owner[page] : e;
}

// count[o*hkv + g] = number of selections (tile, proxy head p, slot) of a
// proxy head p of KV head g = p / kv_div whose block maps to a page owned by
// entry o.
__global__ void bwd_count_kernel(const TileInfo* __restrict__ tiles, const int32_t* __restrict__ idx, int32_t n_tiles,
                                 int32_t hsel, int32_t kv_div, int32_t topk, const int32_t* __restrict__ kv_indices,
                                 const int32_t* __restrict__ owner, int64_t num_pages, int32_t* __restrict__ count) {
  pdl_wait();  // launched with programmatic dependent launch: the previous kernel's writes first
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<int64_t>(n_tiles) * hsel * topk) return;
  const int hkv = hsel / kv_div;
  const int t = static_cast<int>(e / (static_cast<int64_t>(hsel) * topk));
  const int g = static_cast<int>((e / topk) % hsel) / kv_div;
  const int j = idx[e];
  const TileInfo tl = tiles[t];
  if (j < 0 || j >= tl.nvp) return;
  atomicAdd(count + owner_of(kv_indices, owner, num_pages, tl.page_base + j) * hkv + g, 1);
}

// Exclusive scan of n counts into off[0..n] (one CTA of 1024 threads);
// cursor[] is reset to off[].
__global__ void __launch_bounds__(1024) bwd_scan_kernel(const int32_t* __restrict__ count, int32_t n,
                                                        int32_t* __restrict__ off, int32_t* __restrict__ cursor) {
  pdl_wait();  // launched with programmatic dependent launch: the previous kernel's writes first
  __shared__ int32_t part[1024];
  const int per = (n + 1023) / 1024;
  const int b = threadIdx.x * per, e = min(n, b + per);
  // a list longer than the key-side kernel sorts in shared memory gets a
  // power-of-two capacity (at most twice its length) to be sorted in place
  auto cap = [](int c) {
    if (c <= kBwdSmemList) return c;
    int p2 = 1;
    while (p2 < c) p2 <<= 1;
    return p2;
  };
  int s = 0;
  for (int i = b; i < e; ++i) s += cap(count[i]);
  part[threadIdx.x] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const int v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int run = part[threadIdx.x] - s;
  for (int i = b; i < e; ++i) {
    off[i] = run;
    cursor[i] = run;
    run += cap(count[i]);
  }
  if (threadIdx.x == 1023) off[n] = part[1023];
}

// Files each selection under its page owner and KV head; the list item is
// the flat selection index (t * hsel + p) * topk + slot, which gives the
// tile, the proxy head and the logical block (and sorts by tile).
__global__ void bwd_fill_kernel(const TileInfo* __restrict__ tiles, const int32_t* __restrict__ idx, int32_t n_tiles,
                                int32_t hsel, int32_t kv_div, int32_t topk, const int32_t* __restrict__ kv_indices,
                                const int32_t* __restrict__ owner, int64_t num_pages, int32_t* __restrict__ cursor,
                                int32_t* __restrict__ list) {
  pdl_wait();  // launched with programmatic dependent launch: the previous kernel's writes first
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<int64_t>(n_tiles) * hsel * topk) return;
  const int hkv = hsel / kv_div;
  const int t = static_cast<int>(e / (static_cast<int64_t>(hsel) * topk));
  const int g = static_cast<int>((e / topk) % hsel) / kv_div;
  const int j = idx[e];
  const TileInfo tl = tiles[t];
  if (j < 0 || j >= tl.nvp) return;
  list[atomicAdd(cursor + owner_of(kv_indices, owner, num_pages, tl.page_base + j) * hkv + g, 1)] =
      static_cast<int32_t>(e);
}

}  // namespace

// The backward's plan table: the tiles, heaviest first (the dq CTAs, one
// per tile and proxy head, run the most blocks first so the last wave is
// the lightest).
void bwd_plan_tables(msa_plan_s* p, std::vector<int32_t>& aux) {
  std::vector<int32_t> order(p->n_tiles);
  for (int t = 0; t < p->n_tiles; ++t) order[t] = t;
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
    return std::min(p->tiles[a].nvp, p->topk) > std::min(p->tiles[b].nvp, p->topk);
  });
  p->heavy_tiles_off = static_cast<int64_t>(aux.size());
  aux.insert(aux.end(), order.begin(), order.end());
}

// The backward scratch, each part 256-byte aligned: dsumt, lse2t ([Hq][total_q]
// fp32), lsept ([Hp][total_q] fp32), the proxy softmax's Op (bf16 [total_q,
// Hp, dp]) and LSE (fp32 [total_q, Hp]), the inverse index (int32), the page
// owners (int32 [num_pages]), dpk's per-KV-head partials (fp32 [entries]
// [Hkv][128][dp]) and their counters ([entries]).
static size_t al256(size_t b) { return (b + 255) & ~size_t(255); }

size_t bwd_scratch_bytes(const msa_plan_s* p) {
  if (p->decode) return 0;
  const size_t tq = static_cast<size_t>(p->total_q);
  const size_t ent = static_cast<size_t>(p->n_page_entries) * p->hkv;
  return 2 * al256(4 * tq * p->hq) + al256(4 * tq * p->hp) + al256(2 * tq * p->hp * kDP) + al256(4 * tq * p->hp) +
         al256(sizeof(int32_t) * (3 * ent + 1 + 2 * static_cast<size_t>(p->n_tiles) * p->hp * p->topk)) +
         al256(sizeof(int32_t) * static_cast<size_t>(p->num_pages)) +
         al256(4 * ent * 128 * kDP) + al256(4 * static_cast<size_t>(p->n_page_entries));
}

msa_status launch_attn_bwd(const msa_plan_s* p, const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* kv_indices, const int32_t* idx, const void* out, const float* lse,
                           const void* dout, const void* pq, const void* pk_pages, float kl_weight, float* dq,
                           float* dk, float* dv, float* dpq, float* dpk, cudaStream_t st) {
  if (p->decode) return set_error(MSA_ERR_UNSUPPORTED, "msa_sparse_attn_bwd: decode batches have no backward");
  if (p->bwd_d == nullptr) return set_error(MSA_ERR_UNSUPPORTED, "msa_sparse_attn_bwd: plan has no backward scratch");
  const int n_ent = p->n_page_entries;
  const size_t ent = static_cast<size_t>(n_ent) * p->hkv;
  const size_t tq = static_cast<size_t>(p->total_q);
  char* sp = static_cast<char*>(p->bwd_d);
  float* dsumt = reinterpret_cast<float*>(sp);                        // [hq][total_q]
  sp += al256(4 * tq * p->hq);
  float* lse2t = reinterpret_cast<float*>(sp);                        // [hq][total_q], lse * log2(e)
  sp += al256(4 * tq * p->hq);
  float* lsept = reinterpret_cast<float*>(sp);                        // [hp][total_q], log2 units
  sp += al256(4 * tq * p->hp);
  auto* op = reinterpret_cast<__nv_bfloat16*>(sp);                    // [total_q, hp, dp] bf16
  sp += al256(2 * tq * p->hp * kDP);
  float* lse_p = reinterpret_cast<float*>(sp);                        // [total_q, hp], natural log
  sp += al256(4 * tq * p->hp);
  int32_t* cnt = reinterpret_cast<int32_t*>(sp);
  int32_t* off = cnt + ent;
  int32_t* cur = off + ent + 1;
  int32_t* list = cur + ent;
  sp += al256(sizeof(int32_t) * (3 * ent + 1 + 2 * static_cast<size_t>(p->n_tiles) * p->hp * p->topk));
  int32_t* owner = reinterpret_cast<int32_t*>(sp);                    // [num_pages]
  sp += al256(sizeof(int32_t) * static_cast<size_t>(p->num_pages));
  float* dpk_part = reinterpret_cast<float*>(sp);                     // [entries][hkv][128][dp]
  sp += al256(4 * ent * 128 * kDP);
  int32_t* dpk_cnt = reinterpret_cast<int32_t*>(sp);                  // [entries]
  const auto* O = static_cast<const __nv_bfloat16*>(out);
  const auto* dO = static_cast<const __nv_bfloat16*>(dout);
  const int64_t n_sel = static_cast<int64_t>(p->n_tiles) * p->hp * p->topk;
  const int kv_div = p->hp / p->hkv;

  // the counters first, so that the kernels follow one another with
  // programmatic dependent launch (each waits for its predecessor's writes)
  msa_status s = cuda_check(cudaMemsetAsync(cnt, 0, sizeof(int32_t) * ent, st), "msa_sparse_attn_bwd: memset");
  if (s == MSA_OK)
    s = cuda_check(cudaMemsetAsync(dpk_cnt, 0, 4 * static_cast<size_t>(n_ent), st), "msa_sparse_attn_bwd: memset");
  if (s == MSA_OK)  // 0x7F7F7F7F: above every entry index
    s = cuda_check(cudaMemsetAsync(owner, 0x7F, sizeof(int32_t) * static_cast<size_t>(p->num_pages), st),
                   "msa_sparse_attn_bwd: memset");
  if (s == MSA_OK) s = launch_proxy_softmax(p, pq, pk_pages, kv_indices, idx, op, lse_p, st);
  if (s != MSA_OK) return s;
  const int sel_blocks = static_cast<int>((n_sel + 255) / 256);
  cudaError_t e = launch_pdl(bwd_prep_kernel, dim3(p->n_tiles * p->hp), dim3(kThreads), 0, st, p->tiles_d, O, dO,
                             lse, static_cast<const __nv_bfloat16*>(op), static_cast<const float*>(lse_p), dsumt,
                             lse2t, lsept, dpq, p->hq, p->hp, static_cast<int32_t>(p->total_q), p->d, p->dp,
                             kl_weight);
  if (e == cudaSuccess)
    e = launch_pdl(bwd_owner_kernel, dim3((n_ent + 255) / 256), dim3(256), 0, st, kv_indices, n_ent, p->num_pages,
                   owner);
  if (e == cudaSuccess)
    e = launch_pdl(bwd_count_kernel, dim3(sel_blocks), dim3(256), 0, st, static_cast<const TileInfo*>(p->tiles_d),
                   idx, p->n_tiles, p->hp, kv_div, p->topk, kv_indices, static_cast<const int32_t*>(owner),
                   p->num_pages, cnt);
  if (e == cudaSuccess)
    e = launch_pdl(bwd_scan_kernel, dim3(1), dim3(1024), 0, st, static_cast<const int32_t*>(cnt),
                   static_cast<int32_t>(ent), off, cur);
  if (e == cudaSuccess)
    e = launch_pdl(bwd_fill_kernel, dim3(sel_blocks), dim3(256), 0, st, static_cast<const TileInfo*>(p->tiles_d), idx,
                   p->n_tiles, p->hp, kv_div, p->topk, kv_indices, static_cast<const int32_t*>(owner),
                   p->num_pages, cur, list);
  s = cuda_check(e, "msa_sparse_attn_bwd: launch");
  if (s != MSA_OK) return s;
  s = launch_bwd_dq_tc(p, q, k_pages, v_pages, dout, pk_pages, idx, kv_indices, lse2t, dsumt, dq, dpq, kl_weight, st);
  if (s != MSA_OK) return s;
  return launch_bwd_dkv_tc(p, q, k_pages, v_pages, dout, pq, pk_pages, kv_indices, idx, owner, off, cnt, list,
                           lse2t, dsumt, lsept, dk, dv, dpk, dpk_part, dpk_cnt, kl_weight, st);
}

}  // namespace msa
