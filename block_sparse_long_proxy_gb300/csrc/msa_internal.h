// Internal declarations of libmsa: plan layout, device tables and the kernel
// launchers each translation unit provides.  Host-only C++ plus plain
// structs shared with device code.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/msa.h"

namespace msa {

constexpr int kPage = 128;   // tokens per KV block / page
constexpr int kTile = 128;   // query rows per tile

// One query tile.  Positions follow bottom-right causal alignment: row r of
// a sequence with qo_len rows and kv_len keys sits at key position
// kv_len - qo_len + r.
struct TileInfo {
  int32_t seq;        // sequence index
  int32_t q_begin;    // global index of the tile's first query row
  int32_t rows;       // rows in this tile, 1..128
  int32_t pos0;       // key position of the first row
  int32_t kv_len;     // keys of the sequence
  int32_t nvp;        // num_valid_pages: blocks up to the diagonal block
  int32_t page_base;  // offset of the sequence's pages in kv_indices
  int32_t pad;
};
static_assert(sizeof(TileInfo) == 32, "TileInfo is uploaded as raw bytes");

// Bits of the device error word.
enum : uint32_t { kErrDeviceCheck = 1u, kErrTimeout = 2u, kErrNonFinite = 4u };

#ifdef __CUDACC__
// Order-preserving 32-bit key of a block score for the top-k selection:
// -0.0 is folded onto +0.0, and -inf maps to 0, which no finite score maps
// to (0 marks "not a candidate").
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;                        // -0.0 == +0.0
  if (u == 0xFF800000u) return 0u;                     // -inf is never a candidate
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);   // monotone in the float order
}
#endif

}  // namespace msa

struct msa_plan_s {
  int device = 0;
  int num_sms = 0;
  int32_t batch = 0, hq = 0, hkv = 0, hp = 0, d = 0, dp = 0, topk = 0;
  int64_t num_pages = 0;
  msa_kv_dtype kv_dtype = MSA_KV_BF16;
  int32_t n_tiles = 0, max_blocks = 0;
  int64_t total_q = 0;
  bool decode = false;               // every qo_len == 1
  bool checks = false;               // MSA_CHECKS set at plan creation: scan outputs for NaN
  std::vector<int32_t> qo_lens, kv_lens;
  std::vector<msa::TileInfo> tiles;  // host copy
  // device memory owned by the plan (one allocation, carved up)
  void* dev_block = nullptr;
  msa::TileInfo* tiles_d = nullptr;
  int32_t* nvp_d = nullptr;
  uint32_t* err_d = nullptr;
  float* partial_d = nullptr;        // decode split-K partials (O, m, l)
  int32_t decode_ctas = 0;           // persistent decode grid size
  // per-kernel work tables, one int32 array carved by offsets
  int32_t* aux_d = nullptr;
  int64_t proxy_units_off = 0;       // prefill proxy work units, grouped by persistent CTA
  int32_t n_proxy_units = 0;
  int64_t proxy_cta_off = 0;         // prefill proxy: first unit of each CTA, [proxy_n_ctas + 1]
  int32_t proxy_n_ctas = 0;
  int64_t proxy_unit_start_off = 0;  // decode proxy: first unit of each tile
  int64_t proxy_chunk_base_off = 0;  // prefill proxy: first 32-block chunk of each tile
  int32_t proxy_n_chunks = 0;        // sum over tiles of ceil(nvp / 32)
  void* fused_topk_d = nullptr;      // msa_proxy_topk scratch: per-row counters, chunk candidates
  int64_t attn_units_off = 0;        // prefill attention work units
  int32_t n_attn_units = 0;
  int64_t proxy_attn_units_off = 0;  // backward proxy softmax work units
  int32_t n_proxy_attn_units = 0;
  int64_t heavy_tiles_off = 0;       // tile ids, most cached blocks first (the backward's dq order)
  int32_t n_page_entries = 0;        // sum over sequences of ceil(kv_len / 128)
  void* bwd_d = nullptr;             // backward scratch (D, proxy LSE, inverse index)
};

namespace msa {

// Launches `kernel` with programmatic stream serialization: its CTAs may be
// scheduled while the previous kernel in the stream drains, which hides the
// launch gap between the short kernels of a decode step; the kernel must
// call pdl_wait() (ptx.cuh) before it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

msa_status set_error(msa_status s, const char* fmt, ...);
msa_status cuda_check(cudaError_t e, const char* what);

// ---- plan-time tables (host), appended to the plan's aux array ----
void proxy_plan_tables(msa_plan_s* p, std::vector<int32_t>& aux);
void attn_plan_tables(msa_plan_s* p, std::vector<int32_t>& aux);
void bwd_plan_tables(msa_plan_s* p, std::vector<int32_t>& aux);
size_t bwd_scratch_bytes(const msa_plan_s* p);
size_t fused_topk_scratch_bytes(const msa_plan_s* p);  // 0 when msa_proxy_topk is unsupported
size_t fused_topk_counter_bytes(const msa_plan_s* p);  // leading part that starts at zero
// The backward's proxy softmax (attn_fwd.cu): Op = sum_k p_proxy(k) pk[k]
// (bf16 [total_q, Hp, 64]) and its natural-log LSE ([total_q, Hp]).
msa_status launch_proxy_softmax(const msa_plan_s* p, const void* pq, const void* pk_pages, const int32_t* kv_indices,
                                const int32_t* idx, void* op, float* lse, cudaStream_t st);
// dQ and dpq's main term on the tensor cores (bwd_dq.cu); dpq holds the
// proxy term on entry and gets the main term added.
msa_status launch_bwd_dq_tc(const msa_plan_s* p, const void* q, const void* k_pages, const void* v_pages,
                            const void* dout, const void* pk_pages, const int32_t* idx, const int32_t* kv_indices,
                            const float* lse2t, const float* dsumt, float* dq, float* dpq, float kl_weight,
                            cudaStream_t st);
// dK, dV and dpk on the tensor cores (bwd_dkv.cu); lse2t, dsumt, lsept are
// the row statistics written by the prep kernel, [heads][total_q]; dpk_part
// is [page-table entries][hkv][128][64] fp32 scratch, dpk_cnt [entries]
// int32 zeroed.
// Selection lists (per page owner and KV head) of up to kBwdSmemList entries
// are sorted in shared memory by the key-side kernel; a longer list gets a
// power-of-two capacity in the inverse index and is sorted in place there.
constexpr int kBwdSmemList = 2048;
msa_status launch_bwd_dkv_tc(const msa_plan_s* p, const void* q, const void* k_pages, const void* v_pages,
                             const void* dout, const void* pq, const void* pk_pages, const int32_t* kv_indices,
                             const int32_t* idx, const int32_t* owner, const int32_t* inv_off,
                             const int32_t* inv_cnt, int32_t* inv_list,
                             const float* lse2t, const float* dsumt, const float* lsept, float* dk, float* dv,
                             float* dpk, float* dpk_part, int32_t* dpk_cnt, float kl_weight, cudaStream_t st);

// ---- launchers (each returns MSA_OK or an error with its message set) ----
msa_status launch_topk(const float* max_score, int32_t n_tiles, int32_t heads, int32_t max_blocks,
                       int32_t topk, const int32_t* nvp, int32_t* out, cudaStream_t st);

msa_status launch_proxy_prefill(const msa_plan_s* p, const void* pq, const void* pk_pages,
                                const int32_t* kv_indices, float* max_score, cudaStream_t st);
msa_status launch_proxy_topk(const msa_plan_s* p, const void* pq, const void* pk_pages,
                             const int32_t* kv_indices, float* max_score, int32_t* kv_block_indexes,
                             cudaStream_t st);
msa_status launch_proxy_decode(const msa_plan_s* p, const void* pq, const void* pk_pages,
                               const int32_t* kv_indices, float* max_score, cudaStream_t st);
// decode proxy scan over e4m3 proxy K pages with one fp32 scale (device pointer)
msa_status launch_proxy_decode_fp8(const msa_plan_s* p, const void* pq, const void* pk_pages, const float* pk_scale,
                                   const int32_t* kv_indices, float* max_score, cudaStream_t st);
// decode proxy scan over an NVFP4 proxy K (proxy_fp4.cu): e2m1 codes [P, 128, dp/2],
// e4m3 block scales [P, 128, dp/16] and one fp32 scale (device pointer)
msa_status launch_proxy_decode_nvfp4(const msa_plan_s* p, const void* pq, const void* pk_codes,
                                     const void* pk_block_scales, const float* pk_global_scale,
                                     const int32_t* kv_indices, float* max_score, cudaStream_t st);

msa_status launch_attn_prefill(const msa_plan_s* p, const void* q, const void* k_pages,
                               const void* v_pages, const int32_t* kv_indices, const int32_t* idx,
                               const float* k_scale, const float* v_scale, void* out, float* lse,
                               cudaStream_t st);
// one CTA per (sequence, group) row with warp-private half-block streams
// (decode_ws.cu); used by launch_attn_decode when decode_ws_applies(p)
bool decode_ws_applies(const msa_plan_s* p);
msa_status launch_attn_decode_ws(const msa_plan_s* p, const void* q, const void* k_pages, const void* v_pages,
                                 const int32_t* kv_indices, const int32_t* idx, const float* k_scale,
                                 const float* v_scale, void* out, float* lse, cudaStream_t st);
msa_status launch_attn_decode(const msa_plan_s* p, const void* q, const void* k_pages,
                              const void* v_pages, const int32_t* kv_indices, const int32_t* idx,
                              const float* k_scale, const float* v_scale, void* out, float* lse,
                              cudaStream_t st);
size_t decode_partial_floats(const msa_plan_s* p);

msa_status launch_attn_bwd(const msa_plan_s* p, const void* q, const void* k_pages,
                           const void* v_pages, const int32_t* kv_indices, const int32_t* idx,
                           const void* out, const float* lse, const void* dout, const void* pq,
                           const void* pk_pages, float kl_weight, float* dq, float* dk, float* dv,
                           float* dpq, float* dpk, cudaStream_t st);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
// dtype_bf16_or_u8: 0 uint8, 1 bf16, 2 fp32.
bool encode_tensor_map(void* map, int rank, const void* base, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, int dtype_bf16_or_u8,
                       int swizzle_bytes);

}  // namespace msa
