// Host side of libmsa: argument validation, the plan (tile table, page
// offsets, workspace), dispatch to the kernels, error reporting.
#include <cudaTypedefs.h>
#include <cuda.h>
#include <stdarg.h>
#include <stdlib.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {

static thread_local std::string g_last_error;
// Allocation failures still to inject into msa_plan (msa_test_fail_plan_allocs).
static std::atomic<int32_t> g_fail_allocs{0};

msa_status set_error(msa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

msa_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MSA_OK;
  return set_error(MSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_tensor_map(void* map, int rank, const void* base, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, int dtype_bf16_or_u8,
                       int swizzle_bytes) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i > 0) gstride[i - 1] = strides_bytes[i - 1];
  }
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle_bytes == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (swizzle_bytes == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
  if (swizzle_bytes == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
  const CUtensorMapDataType dt = dtype_bf16_or_u8 == 2   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dtype_bf16_or_u8 == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = fn(reinterpret_cast<CUtensorMap*>(map), dt, rank, const_cast<void*>(base), gdim, gstride, bdim,
                  estride, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace msa

using namespace msa;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

namespace msa {
namespace {
// One thread waits on a barrier that nothing arrives on.  The bounded wait
// gives up after its limit, sets kErrTimeout in the error word and returns,
// as any kernel's wait would; a completed wait would set the top bit.
__global__ void selftest_wait_kernel(uint32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && mbar_wait(&bar, 0, err)) atomicOr(err, 0x80000000u);
}
}  // namespace
}  // namespace msa

namespace msa {
namespace {

// MSA_CHECKS: one read of a call's inputs and outputs; any NaN raises
// kErrNonFinite.  The test is on the bits, so infinities pass: fp32 and bf16
// NaN have an all-ones exponent and a non-zero mantissa, an e4m3 NaN is
// S.1111.111.
template <typename T>
__device__ __forceinline__ bool nan_bits(T v) {
  const uint32_t u = static_cast<uint32_t>(v);
  if (sizeof(T) == 4) return (u & 0x7FFFFFFFu) > 0x7F800000u;
  if (sizeof(T) == 2) return (u & 0x7FFFu) > 0x7F80u;
  return (u & 0x7Fu) == 0x7Fu;
}

template <typename T>
__global__ void nan_scan_kernel(const T* __restrict__ x, int64_t n, uint32_t* err) {
  bool bad = false;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    bad |= nan_bits(x[i]);
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(err, kErrNonFinite);
}

// The pages a plan's page table names, per_page elements each (out-of-range
// ids are skipped: the compute kernels report those).
template <typename T>
__global__ void nan_scan_pages_kernel(const T* __restrict__ pool, const int32_t* __restrict__ kv_indices,
                                      int32_t n_entries, int64_t num_pages, int64_t per_page, uint32_t* err) {
  for (int e = blockIdx.x; e < n_entries; e += gridDim.x) {
    const int64_t page = kv_indices[e];
    if (page < 0 || page >= num_pages) continue;  // uniform over the CTA
    const T* x = pool + page * per_page;
    bool bad = false;
    for (int64_t i = threadIdx.x; i < per_page; i += blockDim.x) bad |= nan_bits(x[i]);
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(err, kErrNonFinite);
  }
}

// n elements of `elem` bytes (4: fp32, 2: bf16, 1: e4m3) of an array, when
// the plan was created under MSA_CHECKS; otherwise nothing.
msa_status scan_rows(const msa_plan_s* p, const void* x, int64_t n, int elem, cudaStream_t st) {
  if (!p->checks || x == nullptr || n <= 0) return MSA_OK;
  const int grid = static_cast<int>(std::min<int64_t>(int64_t(p->num_sms) * 8, (n + 255) / 256));
  if (elem == 4)
    nan_scan_kernel<uint32_t><<<grid, 256, 0, st>>>(static_cast<const uint32_t*>(x), n, p->err_d);
  else if (elem == 2)
    nan_scan_kernel<uint16_t><<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(x), n, p->err_d);
  else
    nan_scan_kernel<uint8_t><<<grid, 256, 0, st>>>(static_cast<const uint8_t*>(x), n, p->err_d);
  return cuda_check(cudaGetLastError(), "MSA_CHECKS: scan launch");
}

// The referenced pages of a pool, per_page elements of `elem` bytes each.
msa_status scan_pages(const msa_plan_s* p, const void* pool, const int32_t* kv_indices, int64_t per_page, int elem,
                      cudaStream_t st) {
  if (!p->checks || pool == nullptr) return MSA_OK;
  const int grid = std::min(p->n_page_entries, p->num_sms * 8);
  const int n = p->n_page_entries;
  if (elem == 2)
    nan_scan_pages_kernel<uint16_t><<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(pool), kv_indices, n,
                                                          p->num_pages, per_page, p->err_d);
  else
    nan_scan_pages_kernel<uint8_t><<<grid, 256, 0, st>>>(static_cast<const uint8_t*>(pool), kv_indices, n,
                                                         p->num_pages, per_page, p->err_d);
  return cuda_check(cudaGetLastError(), "MSA_CHECKS: scan launch");
}

// After a proxy call: its pq rows and referenced pk pages (bf16 or e4m3),
// then its max_score.
msa_status scan_proxy(const msa_plan_s* p, msa_status s, const void* pq, const void* pk_pages,
                      const int32_t* kv_indices, int pk_elem, const float* ms, cudaStream_t st) {
  if (s == MSA_OK) s = scan_rows(p, pq, p->total_q * p->hp * p->dp, 2, st);
  if (s == MSA_OK && pk_elem > 0) s = scan_pages(p, pk_pages, kv_indices, int64_t(128) * p->dp, pk_elem, st);
  if (s == MSA_OK) s = scan_rows(p, ms, int64_t(p->n_tiles) * p->hp * p->max_blocks, 4, st);
  return s;
}

}  // namespace
}  // namespace msa

extern "C" {

const char* msa_last_error(void) { return g_last_error.c_str(); }
const char* msa_version(void) { return "0.1.0"; }

msa_status msa_plan(const int32_t* qo_lens, const int32_t* kv_lens, int32_t batch, int32_t num_qo_heads,
                    int32_t num_kv_heads, int32_t num_proxy_heads, int32_t head_dim, int32_t proxy_head_dim,
                    int32_t page_size, int32_t topk, int64_t num_pages, msa_kv_dtype kv_dtype, uint32_t flags,
                    msa_stream_t stream, msa_plan_t* out) {
  if (!out) return set_error(MSA_ERR_INVALID_ARG, "msa_plan: out is NULL");
  *out = nullptr;
  if (batch < 1 || !qo_lens || !kv_lens) return set_error(MSA_ERR_INVALID_ARG, "msa_plan: empty batch");
  if (num_qo_heads < 1 || num_kv_heads < 1 || num_proxy_heads < 1)
    return set_error(MSA_ERR_INVALID_ARG, "msa_plan: head counts must be >= 1");
  if (num_qo_heads % num_kv_heads != 0)
    return set_error(MSA_ERR_INVALID_ARG, "msa_plan: num_qo_heads %% num_kv_heads != 0");
  if (num_proxy_heads % num_kv_heads != 0 || num_qo_heads % num_proxy_heads != 0)
    return set_error(MSA_ERR_UNSUPPORTED,
                     "msa_plan: num_proxy_heads must be a multiple of num_kv_heads and divide num_qo_heads");
  if (head_dim != 64 && head_dim != 128) return set_error(MSA_ERR_UNSUPPORTED, "msa_plan: head_dim must be 64 or 128");
  if (proxy_head_dim != 32 && proxy_head_dim != 64)
    return set_error(MSA_ERR_UNSUPPORTED, "msa_plan: proxy_head_dim must be 32 or 64");
  if (page_size != kPage) return set_error(MSA_ERR_UNSUPPORTED, "msa_plan: page_size must be 128");
  if (topk < 1 || topk > 1024) return set_error(MSA_ERR_INVALID_ARG, "msa_plan: topk must be in [1, 1024]");
  if (num_pages < 1 || num_pages > (int64_t(1) << 24))
    return set_error(MSA_ERR_INVALID_ARG, "msa_plan: num_pages out of range");
  if (kv_dtype != MSA_KV_BF16 && kv_dtype != MSA_KV_FP8_E4M3)
    return set_error(MSA_ERR_INVALID_ARG, "msa_plan: unknown kv_dtype");
  if (flags != 0) return set_error(MSA_ERR_INVALID_ARG, "msa_plan: flags must be 0");

  auto* p = new msa_plan_s();
  p->batch = batch;
  p->hq = num_qo_heads;
  p->hkv = num_kv_heads;
  p->hp = num_proxy_heads;
  p->d = head_dim;
  p->dp = proxy_head_dim;
  p->topk = topk;
  p->num_pages = num_pages;
  p->kv_dtype = kv_dtype;
  p->qo_lens.assign(qo_lens, qo_lens + batch);
  p->kv_lens.assign(kv_lens, kv_lens + batch);

  int64_t q0 = 0, page_base = 0;
  bool all_one = true;
  for (int s = 0; s < batch; ++s) {
    const int64_t ql = qo_lens[s], kl = kv_lens[s];
    if (ql < 0 || kl < 1 || ql > kl) {
      delete p;
      return set_error(MSA_ERR_INVALID_ARG, "msa_plan: sequence %d needs 0 <= qo_len <= kv_len and kv_len >= 1", s);
    }
    if (ql != 1) all_one = false;
    const int64_t nb = (kl + kPage - 1) / kPage;
    p->max_blocks = static_cast<int32_t>(std::max<int64_t>(p->max_blocks, nb));
    const int64_t off = kl - ql;
    for (int64_t t = 0; t * kTile < ql; ++t) {
      TileInfo ti{};
      const int64_t r0 = t * kTile, r1 = std::min<int64_t>(ql, r0 + kTile);
      ti.seq = s;
      ti.q_begin = static_cast<int32_t>(q0 + r0);
      ti.rows = static_cast<int32_t>(r1 - r0);
      ti.pos0 = static_cast<int32_t>(off + r0);
      ti.kv_len = static_cast<int32_t>(kl);
      ti.nvp = static_cast<int32_t>((off + r1 - 1) / kPage + 1);
      ti.page_base = static_cast<int32_t>(page_base);
      p->tiles.push_back(ti);
    }
    q0 += ql;
    page_base += nb;
    if (q0 > (int64_t(1) << 31) - 1 || page_base > (int64_t(1) << 31) - 1) {
      delete p;
      return set_error(MSA_ERR_INVALID_ARG, "msa_plan: batch too large for 32-bit row / page indexing");
    }
  }
  p->total_q = q0;
  p->n_page_entries = static_cast<int32_t>(page_base);
  p->n_tiles = static_cast<int32_t>(p->tiles.size());
  p->decode = all_one;
  {  // debug mode: scan every call's outputs for NaN
    const char* c = getenv("MSA_CHECKS");
    p->checks = c != nullptr && c[0] != '\0' && strcmp(c, "0") != 0;
  }
  if (p->n_tiles == 0) {
    delete p;
    return set_error(MSA_ERR_INVALID_ARG, "msa_plan: no query rows in the batch");
  }

  if (cudaGetDevice(&p->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
    delete p;
    return set_error(MSA_ERR_CUDA, "msa_plan: no CUDA device");
  }

  std::vector<int32_t> aux;
  proxy_plan_tables(p, aux);
  attn_plan_tables(p, aux);
  bwd_plan_tables(p, aux);

  // device block: tiles | nvp | error word | aux tables | decode partials |
  // backward scratch | fused top-k counters and candidates
  const size_t tiles_bytes = sizeof(TileInfo) * p->n_tiles;
  const size_t nvp_off = (tiles_bytes + 255) & ~size_t(255);
  const size_t err_off = nvp_off + ((sizeof(int32_t) * p->n_tiles + 255) & ~size_t(255));
  const size_t aux_off = err_off + 256;
  const size_t part_off = aux_off + ((sizeof(int32_t) * aux.size() + 255) & ~size_t(255));
  const size_t part_bytes = (sizeof(float) * decode_partial_floats(p) + 255) & ~size_t(255);
  const size_t bwd_off = part_off + part_bytes;
  const size_t fz_off = bwd_off + ((bwd_scratch_bytes(p) + 255) & ~size_t(255));
  const size_t total = fz_off + fused_topk_scratch_bytes(p);
  int32_t inject = g_fail_allocs.load();
  while (inject > 0 && !g_fail_allocs.compare_exchange_weak(inject, inject - 1)) {
  }
  if (inject > 0) {  // an injected failure: the same path as a real one, without the call
    delete p;
    return set_error(MSA_ERR_NO_MEMORY, "msa_plan: cudaMalloc of %zu bytes failed (injected)", total);
  }
  if (cudaMalloc(&p->dev_block, total) != cudaSuccess) {
    cudaGetLastError();
    delete p;
    return set_error(MSA_ERR_NO_MEMORY, "msa_plan: cudaMalloc of %zu bytes failed", total);
  }
  char* base = static_cast<char*>(p->dev_block);
  p->tiles_d = reinterpret_cast<TileInfo*>(base);
  p->nvp_d = reinterpret_cast<int32_t*>(base + nvp_off);
  p->err_d = reinterpret_cast<uint32_t*>(base + err_off);
  p->aux_d = reinterpret_cast<int32_t*>(base + aux_off);
  p->partial_d = part_bytes ? reinterpret_cast<float*>(base + part_off) : nullptr;
  p->bwd_d = bwd_scratch_bytes(p) ? base + bwd_off : nullptr;
  p->fused_topk_d = fused_topk_scratch_bytes(p) ? base + fz_off : nullptr;

  std::vector<char> host(part_off, 0);
  memcpy(host.data(), p->tiles.data(), tiles_bytes);
  for (int t = 0; t < p->n_tiles; ++t)
    memcpy(host.data() + nvp_off + sizeof(int32_t) * t, &p->tiles[t].nvp, sizeof(int32_t));
  if (!aux.empty()) memcpy(host.data() + aux_off, aux.data(), sizeof(int32_t) * aux.size());
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  msa_status s = cuda_check(cudaMemcpyAsync(p->dev_block, host.data(), part_off, cudaMemcpyHostToDevice, st),
                            "msa_plan: upload");
  if (s == MSA_OK && part_bytes)  // decode partials and per-row counters start at zero
    s = cuda_check(cudaMemsetAsync(base + part_off, 0, part_bytes, st), "msa_plan: clear decode workspace");
  if (s == MSA_OK && p->fused_topk_d)  // the fused top-k's row counters start at zero
    s = cuda_check(cudaMemsetAsync(p->fused_topk_d, 0, fused_topk_counter_bytes(p), st), "msa_plan: clear counters");
  if (s == MSA_OK) s = cuda_check(cudaStreamSynchronize(st), "msa_plan: upload sync");
  if (s != MSA_OK) {
    cudaFree(p->dev_block);
    delete p;
    return s;
  }
  *out = p;
  return MSA_OK;
}

void msa_plan_destroy(msa_plan_t plan) {
  if (!plan) return;
  if (plan->dev_block) cudaFree(plan->dev_block);
  delete plan;
}

int32_t msa_plan_num_tiles(msa_plan_t plan) { return plan ? plan->n_tiles : 0; }
int32_t msa_plan_max_blocks(msa_plan_t plan) { return plan ? plan->max_blocks : 0; }
int64_t msa_plan_total_q(msa_plan_t plan) { return plan ? plan->total_q : 0; }
const int32_t* msa_plan_num_valid_pages(msa_plan_t plan) { return plan ? plan->nvp_d : nullptr; }

msa_status msa_proxy_maxscore(msa_plan_t plan, const void* pq, const void* pk_pages, const int32_t* kv_indices,
                              float* max_score, msa_stream_t stream) {
  if (!plan || !pq || !pk_pages || !kv_indices || !max_score)
    return set_error(MSA_ERR_INVALID_ARG, "msa_proxy_maxscore: NULL argument");
  if (!aligned16(pq) || !aligned16(pk_pages))
    return set_error(MSA_ERR_INVALID_ARG, "msa_proxy_maxscore: pq and pk_pages must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const msa_status s = plan->decode ? launch_proxy_decode(plan, pq, pk_pages, kv_indices, max_score, st)
                                    : launch_proxy_prefill(plan, pq, pk_pages, kv_indices, max_score, st);
  return scan_proxy(plan, s, pq, pk_pages, kv_indices, 2, max_score, st);
}

msa_status msa_proxy_maxscore_fp8(msa_plan_t plan, const void* pq, const void* pk_pages, const float* pk_scale,
                                  const int32_t* kv_indices, float* max_score, msa_stream_t stream) {
  if (!plan || !pq || !pk_pages || !pk_scale || !kv_indices || !max_score)
    return set_error(MSA_ERR_INVALID_ARG, "msa_proxy_maxscore_fp8: NULL argument");
  if (!aligned16(pq) || !aligned16(pk_pages))
    return set_error(MSA_ERR_INVALID_ARG, "msa_proxy_maxscore_fp8: pq and pk_pages must be 16-byte aligned");
  if (!plan->decode)
    return set_error(MSA_ERR_UNSUPPORTED, "msa_proxy_maxscore_fp8: FP8 proxy K is implemented for decode batches only");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return scan_proxy(plan, launch_proxy_decode_fp8(plan, pq, pk_pages, pk_scale, kv_indices, max_score, st), pq,
                    pk_pages, kv_indices, 1, max_score, st);
}

msa_status msa_proxy_maxscore_nvfp4(msa_plan_t plan, const void* pq, const void* pk_codes,
                                    const void* pk_block_scales, const float* pk_global_scale,
                                    const int32_t* kv_indices, float* max_score, msa_stream_t stream) {
  if (!plan || !pq || !pk_codes || !pk_block_scales || !pk_global_scale || !kv_indices || !max_score)
    return set_error(MSA_ERR_INVALID_ARG, "msa_proxy_maxscore_nvfp4: NULL argument");
  if (!aligned16(pq) || !aligned16(pk_codes) || !aligned16(pk_block_scales))
    return set_error(MSA_ERR_INVALID_ARG,
                     "msa_proxy_maxscore_nvfp4: pq, pk_codes and pk_block_scales must be 16-byte aligned");
  if (!plan->decode)
    return set_error(MSA_ERR_UNSUPPORTED,
                     "msa_proxy_maxscore_nvfp4: the NVFP4 proxy K is implemented for decode batches only");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // e2m1 codes have no NaN: pq and max_score are scanned
  return scan_proxy(plan,
                    launch_proxy_decode_nvfp4(plan, pq, pk_codes, pk_block_scales, pk_global_scale, kv_indices,
                                              max_score, st),
                    pq, nullptr, kv_indices, 0, max_score, st);
}

msa_status msa_proxy_topk(msa_plan_t plan, const void* pq, const void* pk_pages, const int32_t* kv_indices,
                          float* max_score, int32_t* kv_block_indexes, msa_stream_t stream) {
  if (!plan || !pq || !pk_pages || !kv_indices || !kv_block_indexes)
    return set_error(MSA_ERR_INVALID_ARG, "msa_proxy_topk: NULL argument");
  if (!aligned16(pq) || !aligned16(pk_pages))
    return set_error(MSA_ERR_INVALID_ARG, "msa_proxy_topk: pq and pk_pages must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return scan_proxy(plan, launch_proxy_topk(plan, pq, pk_pages, kv_indices, max_score, kv_block_indexes, st), pq,
                    pk_pages, kv_indices, 2, max_score, st);
}

msa_status msa_topk_select(const float* max_score, int32_t n_tiles, int32_t heads, int32_t max_blocks,
                           int32_t topk, const int32_t* num_valid_pages, int32_t* kv_block_indexes,
                           msa_stream_t stream) {
  if (!max_score || !num_valid_pages || !kv_block_indexes)
    return set_error(MSA_ERR_INVALID_ARG, "msa_topk_select: NULL argument");
  if (n_tiles < 1 || heads < 1 || max_blocks < 1 || max_blocks > 65536 || topk < 1 || topk > 1024)
    return set_error(MSA_ERR_INVALID_ARG, "msa_topk_select: sizes out of range");
  if (int64_t(n_tiles) * heads > (int64_t(1) << 31) - 1)
    return set_error(MSA_ERR_INVALID_ARG, "msa_topk_select: too many rows");
  return launch_topk(max_score, n_tiles, heads, max_blocks, topk, num_valid_pages, kv_block_indexes,
                     reinterpret_cast<cudaStream_t>(stream));
}

msa_status msa_sparse_attn(msa_plan_t plan, const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* kv_indices, const int32_t* kv_block_indexes, const float* k_scale,
                           const float* v_scale, void* out, float* lse, msa_stream_t stream) {
  if (!plan || !q || !k_pages || !v_pages || !kv_indices || !kv_block_indexes || !out)
    return set_error(MSA_ERR_INVALID_ARG, "msa_sparse_attn: NULL argument");
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out))
    return set_error(MSA_ERR_INVALID_ARG, "msa_sparse_attn: q, k_pages, v_pages, out must be 16-byte aligned");
  const bool fp8 = plan->kv_dtype == MSA_KV_FP8_E4M3;
  if (fp8 != (k_scale != nullptr) || fp8 != (v_scale != nullptr))
    return set_error(MSA_ERR_INVALID_ARG, "msa_sparse_attn: k_scale/v_scale must be given exactly for FP8 K/V");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  msa_status s = fp8 && plan->decode
                     ? launch_attn_decode(plan, q, k_pages, v_pages, kv_indices, kv_block_indexes, k_scale, v_scale,
                                          out, lse, st)
                     : launch_attn_prefill(plan, q, k_pages, v_pages, kv_indices, kv_block_indexes, k_scale, v_scale,
                                           out, lse, st);
  const int64_t rows = plan->total_q * plan->hq;
  const int kv_elem = fp8 ? 1 : 2;
  const int64_t per_page = int64_t(plan->hkv) * 128 * plan->d;
  if (s == MSA_OK) s = scan_rows(plan, q, rows * plan->d, 2, st);
  if (s == MSA_OK) s = scan_pages(plan, k_pages, kv_indices, per_page, kv_elem, st);
  if (s == MSA_OK) s = scan_pages(plan, v_pages, kv_indices, per_page, kv_elem, st);
  if (s == MSA_OK) s = scan_rows(plan, out, rows * plan->d, 2, st);
  if (s == MSA_OK) s = scan_rows(plan, lse, rows, 4, st);
  return s;
}

msa_status msa_sparse_attn_bwd(msa_plan_t plan, const void* q, const void* k_pages, const void* v_pages,
                               const int32_t* kv_indices, const int32_t* kv_block_indexes, const void* out,
                               const float* lse, const void* dout, const void* pq, const void* pk_pages,
                               float kl_weight, float* dq, float* dk_pages, float* dv_pages, float* dpq,
                               float* dpk_pages, msa_stream_t stream) {
  if (!plan || !q || !k_pages || !v_pages || !kv_indices || !kv_block_indexes || !out || !lse || !dout || !pq ||
      !pk_pages || !dq || !dk_pages || !dv_pages || !dpq || !dpk_pages)
    return set_error(MSA_ERR_INVALID_ARG, "msa_sparse_attn_bwd: NULL argument");
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out) || !aligned16(dout) ||
      !aligned16(pq) || !aligned16(pk_pages) || !aligned32(dq) || !aligned32(dk_pages) || !aligned32(dv_pages) ||
      !aligned32(dpq) || !aligned32(dpk_pages))
    return set_error(MSA_ERR_INVALID_ARG,
                     "msa_sparse_attn_bwd: inputs must be 16-byte aligned and gradients 32-byte aligned");
  if (plan->kv_dtype != MSA_KV_BF16)
    return set_error(MSA_ERR_UNSUPPORTED, "msa_sparse_attn_bwd: bf16 K/V only");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  msa_status s = launch_attn_bwd(plan, q, k_pages, v_pages, kv_indices, kv_block_indexes, out, lse, dout, pq,
                                 pk_pages, kl_weight, dq, dk_pages, dv_pages, dpq, dpk_pages, st);
  const int64_t rows = plan->total_q * plan->hq;
  const int64_t per_page = int64_t(plan->hkv) * 128 * plan->d;
  if (s == MSA_OK) s = scan_rows(plan, q, rows * plan->d, 2, st);
  if (s == MSA_OK) s = scan_rows(plan, dout, rows * plan->d, 2, st);
  if (s == MSA_OK) s = scan_rows(plan, pq, plan->total_q * plan->hp * plan->dp, 2, st);
  if (s == MSA_OK) s = scan_pages(plan, k_pages, kv_indices, per_page, 2, st);
  if (s == MSA_OK) s = scan_pages(plan, v_pages, kv_indices, per_page, 2, st);
  if (s == MSA_OK) s = scan_pages(plan, pk_pages, kv_indices, int64_t(128) * plan->dp, 2, st);
  if (s == MSA_OK) s = scan_rows(plan, dq, rows * plan->d, 4, st);
  if (s == MSA_OK) s = scan_rows(plan, dpq, plan->total_q * plan->hp * plan->dp, 4, st);
  return s;
}

void msa_test_fail_plan_allocs(int32_t count) { g_fail_allocs.store(count > 0 ? count : 0); }

msa_status msa_selftest_wait_timeout(msa_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* word_d = nullptr;
  if (cudaMalloc(&word_d, sizeof(uint32_t)) != cudaSuccess) {
    cudaGetLastError();
    return set_error(MSA_ERR_NO_MEMORY, "msa_selftest_wait_timeout: cudaMalloc failed");
  }
  msa_status s = cuda_check(cudaMemsetAsync(word_d, 0, sizeof(uint32_t), st), "msa_selftest_wait_timeout: memset");
  if (s == MSA_OK) {
    selftest_wait_kernel<<<1, 32, 0, st>>>(word_d);
    s = cuda_check(cudaGetLastError(), "msa_selftest_wait_timeout: launch");
  }
  if (s == MSA_OK) s = cuda_check(cudaStreamSynchronize(st), "msa_selftest_wait_timeout: sync");
  uint32_t word = 0;
  if (s == MSA_OK) s = cuda_check(cudaMemcpy(&word, word_d, sizeof(word), cudaMemcpyDeviceToHost), "msa_selftest_wait_timeout: read");
  cudaFree(word_d);
  if (s != MSA_OK) return s;
  if (word == kErrTimeout) return set_error(MSA_ERR_TIMEOUT, "msa_selftest_wait_timeout: the bounded wait gave up (word 0x%x)", word);
  return set_error(MSA_ERR_CUDA, "msa_selftest_wait_timeout: unexpected error word 0x%x", word);
}

msa_status msa_check_errors(msa_plan_t plan, msa_stream_t stream) {
  if (!plan) return set_error(MSA_ERR_INVALID_ARG, "msa_check_errors: NULL plan");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  msa_status s = cuda_check(cudaStreamSynchronize(st), "msa_check_errors: sync");
  if (s != MSA_OK) return s;
  s = cuda_check(cudaMemcpy(&word, plan->err_d, sizeof(word), cudaMemcpyDeviceToHost), "msa_check_errors: read");
  if (s != MSA_OK) return s;
  if (word == 0) return MSA_OK;
  s = cuda_check(cudaMemset(plan->err_d, 0, sizeof(uint32_t)), "msa_check_errors: clear");
  if (s != MSA_OK) return s;
  if (word & kErrTimeout) return set_error(MSA_ERR_TIMEOUT, "a bounded device-side wait gave up (word 0x%x)", word);
  if (word & kErrDeviceCheck)
    return set_error(MSA_ERR_DEVICE_CHECK, "a device-side bounds check fired: page id out of range (word 0x%x)", word);
  return set_error(MSA_ERR_NONFINITE, "MSA_CHECKS: an output held a NaN (word 0x%x)", word);
}

}  // extern "C"
