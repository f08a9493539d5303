// Stage 2: per-(tile, proxy head) top-k block selection over max_score.
//
// The selection ("MiniMax-AI/MSA" README, section "Usage":
// sparse_topk_select(max_score, topk, num_valid_pages); Flash-MSA article,
// kernel-design paragraph: the token's own block is always visible):
// the diagonal block j_d = num_valid_pages - 1 is always taken; the other
// topk-1 are the largest finite scores among blocks j < j_d, ties broken
// towards the lower block index; output ascending, padded with -1.
//
// One warp per row.  Scores map to order-preserving 32-bit keys (-0.0 is
// folded onto +0.0, -inf and everything past the candidates become key 0,
// which no finite score maps to).  The threshold T -- the (topk-1)-th
// largest key -- is found exactly by a 32-step binary search on the key
// bits, each step one warp-wide count of keys >= a probe value.  A final
// ascending scan emits blocks with key > T, then as many key == T blocks as
// are still needed in ascending j order, then j_d: the result is bit-exact
// and already sorted.  HBM traffic is one coalesced read of the row.
#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kWarpsPerBlock = 8;


// Keys held in registers: KPL per lane covers rows of up to 32*KPL blocks.
template <int KPL>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    topk_kernel(const float* __restrict__ max_score, int32_t rows, int32_t heads, int32_t max_blocks,
                int32_t topk, const int32_t* __restrict__ nvp_arr, int32_t* __restrict__ out) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int tile = static_cast<int>(row / heads);
  const float* src = max_score + row * max_blocks;
  int32_t* dst = out + row * topk;
  const int n = nvp_arr[tile];
  if (n < 1 || n > max_blocks) {  // outside the contract: select nothing
    for (int j = lane; j < topk; j += 32) dst[j] = -1;
    return;
  }
  const uint32_t lt_mask = (1u << lane) - 1u;

  if (topk >= n) {  // every valid block is selected
    for (int j = lane; j < topk; j += 32) dst[j] = j < n ? j : -1;
    return;
  }
  const int jd = n - 1;
  const int need_total = topk - 1;

  uint32_t key[KPL];
  int count_valid = 0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int j = i * 32 + lane;
    key[i] = j < jd ? order_key(__ldg(src + j)) : 0u;
    count_valid += key[i] != 0u;
  }
  count_valid = __reduce_add_sync(0xFFFFFFFFu, count_valid);

  uint32_t thr = 1u;          // take every candidate (key >= 1) when there are few
  int eq_take = 1 << 30;
  if (count_valid > need_total && need_total > 0) {
    // largest T with #{key >= T} >= need_total: exactly the need_total-th key
    uint32_t t = 0u;
    for (int bit = 31; bit >= 0; --bit) {
      const uint32_t probe = t | (1u << bit);
      int c = 0;
#pragma unroll
      for (int i = 0; i < KPL; ++i) c += key[i] >= probe;
      c = __reduce_add_sync(0xFFFFFFFFu, c);
      if (c >= need_total) t = probe;
    }
    thr = t;
    int above = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) above += key[i] > thr;
    above = __reduce_add_sync(0xFFFFFFFFu, above);
    eq_take = need_total - above;  // >= 1 by the choice of T
  } else if (need_total == 0) {
    thr = 0xFFFFFFFFu;
    eq_take = 0;
  }

  int written = 0, eq_seen = 0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    if (i * 32 >= n) break;
    const int j = i * 32 + lane;
    const bool is_eq = key[i] != 0u && key[i] == thr;
    const uint32_t eq_ballot = __ballot_sync(0xFFFFFFFFu, is_eq);
    const int eq_rank = eq_seen + __popc(eq_ballot & lt_mask);
    bool sel = (key[i] != 0u && key[i] > thr) || (is_eq && eq_rank < eq_take) || j == jd;
    const uint32_t sel_ballot = __ballot_sync(0xFFFFFFFFu, sel);
    if (sel) dst[written + __popc(sel_ballot & lt_mask)] = j;
    written += __popc(sel_ballot);
    eq_seen += __popc(eq_ballot);
  }
  for (int j = written + lane; j < topk; j += 32) dst[j] = -1;
}

// Rows longer than 1024 blocks: keys re-read from global (L2) each step.
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    topk_kernel_long(const float* __restrict__ max_score, int32_t rows, int32_t heads, int32_t max_blocks,
                     int32_t topk, const int32_t* __restrict__ nvp_arr, int32_t* __restrict__ out) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int tile = static_cast<int>(row / heads);
  const float* src = max_score + row * max_blocks;
  int32_t* dst = out + row * topk;
  const int n = nvp_arr[tile];
  if (n < 1 || n > max_blocks) {  // outside the contract: select nothing
    for (int j = lane; j < topk; j += 32) dst[j] = -1;
    return;
  }
  const uint32_t lt_mask = (1u << lane) - 1u;
  if (topk >= n) {
    for (int j = lane; j < topk; j += 32) dst[j] = j < n ? j : -1;
    return;
  }
  const int jd = n - 1;
  const int need_total = topk - 1;
  auto key_at = [&](int j) -> uint32_t { return j < jd ? order_key(__ldg(src + j)) : 0u; };
  int count_valid = 0;
  for (int j = lane; j < jd; j += 32) count_valid += key_at(j) != 0u;
  count_valid = __reduce_add_sync(0xFFFFFFFFu, count_valid);
  uint32_t thr = 1u;
  int eq_take = 1 << 30;
  if (count_valid > need_total && need_total > 0) {
    uint32_t t = 0u;
    for (int bit = 31; bit >= 0; --bit) {
      const uint32_t probe = t | (1u << bit);
      int c = 0;
      for (int j = lane; j < jd; j += 32) c += key_at(j) >= probe;
      c = __reduce_add_sync(0xFFFFFFFFu, c);
      if (c >= need_total) t = probe;
    }
    thr = t;
    int above = 0;
    for (int j = lane; j < jd; j += 32) above += key_at(j) > thr;
    above = __reduce_add_sync(0xFFFFFFFFu, above);
    eq_take = need_total - above;
  } else if (need_total == 0) {
    thr = 0xFFFFFFFFu;
    eq_take = 0;
  }
  int written = 0, eq_seen = 0;
  for (int base = 0; base < n; base += 32) {
    const int j = base + lane;
    const uint32_t k = j < n ? key_at(j) : 0u;
    const bool is_eq = k != 0u && k == thr;
    const uint32_t eq_ballot = __ballot_sync(0xFFFFFFFFu, is_eq);
    const int eq_rank = eq_seen + __popc(eq_ballot & lt_mask);
    const bool sel = (k != 0u && k > thr) || (is_eq && eq_rank < eq_take) || j == jd;
    const uint32_t sel_ballot = __ballot_sync(0xFFFFFFFFu, sel);
    if (sel) dst[written + __popc(sel_ballot & lt_mask)] = j;
    written += __popc(sel_ballot);
    eq_seen += __popc(eq_ballot);
  }
  for (int j = written + lane; j < topk; j += 32) dst[j] = -1;
}

}  // namespace

msa_status launch_topk(const float* max_score, int32_t n_tiles, int32_t heads, int32_t max_blocks, int32_t topk,
                       const int32_t* nvp, int32_t* out, cudaStream_t st) {
  const int32_t rows = n_tiles * heads;
  const dim3 grid((rows + kWarpsPerBlock - 1) / kWarpsPerBlock), block(32 * kWarpsPerBlock);
  cudaError_t e;
  if (max_blocks <= 256)
    e = launch_pdl(topk_kernel<8>, grid, block, 0, st, max_score, rows, heads, max_blocks, topk, nvp, out);
  else if (max_blocks <= 1024)
    e = launch_pdl(topk_kernel<32>, grid, block, 0, st, max_score, rows, heads, max_blocks, topk, nvp, out);
  else
    e = launch_pdl(topk_kernel_long, grid, block, 0, st, max_score, rows, heads, max_blocks, topk, nvp, out);
  return cuda_check(e, "msa_topk_select: launch");
}

}  // namespace msa
