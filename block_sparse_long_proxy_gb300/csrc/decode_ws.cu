// Stage 3 (decode), one CTA per (sequence, group) row: paged sparse
// attention with FP8 e4m3 K/V ("MiniMax-AI/MSA" README, section "Stacks":
// paged FP8 decode), the same arithmetic as decode_kernel in decode.cu:
// softmax over the selected blocks' keys of q.(k_code*k_scale)/sqrt(d),
// out = P.(v_code*v_scale).
//
// Used when the batch has at least as many (sequence, group) rows as SMs and
// G <= 8.  Every warp of the CTA streams its own units (kKeys keys of K
// and of V of one selected block) through a private buffer and keeps its own
// online-softmax state; the warps' states are merged once, at the end of the
// row.  With two CTAs per SM that is 16 independent warps per SM, each with
// one load in flight, and no producer warp or per-block CTA barrier.  Unit
// u of the row (slot u / kParts of kv_block_indexes, keys kKeys (u % kParts)
// ...) goes to warp u % kWsWarps.
//
// Per unit, on mma.sync (f16 in, f32 out), exactly as decode_kernel:
//   S^T = K . q^T     M = kKeys keys, N = 8 heads, K = d (e4m3 -> f16 in registers)
//   O^T += V^T . P^T  M = d,  N = 8 heads, K = kKeys keys (P^T by movmatrix)
// with d permuted so that every shared-memory read is one conflict-free word.
#include "msa_internal.h"
#include "ptx.cuh"

#include <cuda_fp16.h>

namespace msa {
namespace {

constexpr int kD = 128;
// a unit is kKeys keys of one selected block (K and V), streamed by one warp
// through kStg private stages; kWsWarps warps per CTA, two CTAs per SM.
// Measured at 32 x 131072 (keys, stages, warps): (64,1,6) 29.9 us,
// (32,2,6) 30.4, (64,2,3) 31.0, (64,1,4) 29.7, (32,1,12) 35.5 (spills),
// (32,1,8) 28.9: 16 warps per SM and the same unit count for every warp.
constexpr int kKeys = 32;
constexpr int kStg = 1;
constexpr int kWsWarps = 8;
constexpr int kWsThreads = 32 * kWsWarps;
constexpr int kParts = 128 / kKeys;             // units per block
constexpr int kPartBytes = kKeys * kD;          // K (or V) bytes of one unit
constexpr int kStageBytes = 2 * kPartBytes;     // K part | V part
constexpr int kBufBytes = kStg * kStageBytes;   // one warp's stages
constexpr int kMT = kKeys / 16;                 // 16-key m-tiles of a unit
constexpr int kMaxTopk = (32 * kWsWarps) / kParts;  // a warp's units fit one lane each
static_assert(kBufBytes >= 8 * (kD + 2) * 4, "a warp's merge scratch fits its stages");

struct WsSmem {
  static constexpr int kBufOff = 0;
  static constexpr int kBarOff = kWsWarps * kBufBytes;
  static constexpr int kBytes = kBarOff + 8 * kWsWarps * kStg;
};

// byte offset of (row, byte col) in a tile of 128-byte rows written by TMA
// with 128-byte swizzle: the 16-byte chunk index is XORed with row % 8.
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return row * 128 + ((((col >> 4) ^ row) & 7) << 4) + (col & 15);
}

__global__ void __launch_bounds__(kWsThreads, 2)
    decode_ws_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                     const __nv_bfloat16* __restrict__ q, const TileInfo* __restrict__ tiles,
                     const int32_t* __restrict__ idx, const int32_t* __restrict__ kv_indices, int64_t num_pages,
                     const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                     __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int32_t hq, int32_t hsel,
                     int32_t kv_div, int32_t topk, float scale_log2, uint32_t* err) {
  pdl_wait();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // row = (sequence, proxy head g): the G = hq / hsel query heads of g over
  // g's blocks of KV head g / kv_div
  const int row = blockIdx.x;
  const int t = row / hsel, g = row % hsel;
  const int G = hq / hsel;
  const int hkv = hsel / kv_div, kvh = g / kv_div;
  const TileInfo tl = tiles[t];
  uint8_t* buf = smem + WsSmem::kBufOff + warp * kBufBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + WsSmem::kBarOff) + warp * kStg;
  if (lane == 0) {
    prefetch_tmap(&k_map);
    prefetch_tmap(&v_map);
    for (int s = 0; s < kStg; ++s) mbar_init(bar + s, 1);
    fence_mbar_init();
  }
  __syncwarp();

  // this warp's units u = warp, warp + W, ...: lane l holds the l-th one's
  // first key position (-1 for a padding slot) and page row
  const int n_units = kParts * topk;
  const int my_n = n_units > warp ? (n_units - warp + kWsWarps - 1) / kWsWarps : 0;
  int ukey = -1, urow = 0;
  if (lane < my_n) {
    const int u = warp + lane * kWsWarps;
    const int j = idx[static_cast<int64_t>(row) * topk + u / kParts];
    if (j >= tl.nvp) {
      atomicOr(err, kErrDeviceCheck);
    } else if (j >= 0) {
      int64_t page = kv_indices[tl.page_base + j];
      if (page < 0 || page >= num_pages) {
        atomicOr(err, kErrDeviceCheck);
        page = 0;
      }
      ukey = j * 128 + (u % kParts) * kKeys;
      urow = static_cast<int>((page * hkv + kvh) * 128 + (u % kParts) * kKeys);
    }
  }
  // compact the valid units to the low lanes (padding slots load nothing)
  const unsigned vmask = __ballot_sync(0xFFFFFFFFu, lane < my_n && ukey >= 0);
  const int n_valid = __popc(vmask);
  {
    int src = 0;  // lane holding the (lane+1)-th valid unit
    for (int k = 0, r = 0; k < 32; ++k)
      if ((vmask >> k) & 1u) {
        if (r == lane) src = k;
        ++r;
      }
    const int k2 = __shfl_sync(0xFFFFFFFFu, ukey, src);
    const int r2 = __shfl_sync(0xFFFFFFFFu, urow, src);
    ukey = k2;
    urow = r2;
  }

  // q^T fragments: head gi of the group, d = 16 kc + 4 t4 + {0,1} | {2,3}
  const int gi = lane >> 2, t4 = lane & 3;
  uint32_t qf[kD / 16][2];
  {
    const __nv_bfloat16* qr = q + (static_cast<int64_t>(tl.q_begin) * hq + g * G + gi) * kD;
#pragma unroll
    for (int kc = 0; kc < kD / 16; ++kc) {
      if (gi < G) {
        const uint2 v = *reinterpret_cast<const uint2*>(qr + kc * 16 + 4 * t4);
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
        const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
        qf[kc][0] = pack_f16x2(f0.x, f0.y);
        qf[kc][1] = pack_f16x2(f1.x, f1.y);
      } else {
        qf[kc][0] = qf[kc][1] = 0u;
      }
    }
  }
  const float sl2 = scale_log2 * k_scale[kvh];
  const int qpos = tl.pos0;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f}, oacc[8][4];
#pragma unroll
  for (int md = 0; md < 8; ++md) oacc[md][0] = oacc[md][1] = oacc[md][2] = oacc[md][3] = 0.f;

  auto issue = [&](int i) {  // load unit i of the warp into stage i % kStg
    if (i >= n_valid) return;
    const int r = __shfl_sync(0xFFFFFFFFu, urow, i);
    if (lane == 0) {
      uint64_t* b = bar + i % kStg;
      uint8_t* st = buf + (i % kStg) * kStageBytes;
      mbar_expect_tx(b, kStageBytes);
      tma_load_2d(st, &k_map, b, 0, r);
      tma_load_2d(st + kPartBytes, &v_map, b, 0, r);
    }
  };
  for (int i = 0; i < kStg - 1; ++i) issue(i);
  bool ok = true;
  for (int i = 0; ok && i < n_valid; ++i) {
    issue(i + kStg - 1);  // the stage it fills was released at the end of unit i - 1
    const int key0 = __shfl_sync(0xFFFFFFFFu, ukey, i);
    if (!(ok = mbar_wait(bar + i % kStg, (i / kStg) & 1, err))) break;
    const uint32_t kb = smem_u32(buf + (i % kStg) * kStageBytes), vb = kb + kPartBytes;

    // S^T for the unit's keys
    float sacc[kMT][4];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) sacc[mt][0] = sacc[mt][1] = sacc[mt][2] = sacc[mt][3] = 0.f;
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      const int ra = 16 * mt + gi, rb = ra + 8;
#pragma unroll
      for (int kc = 0; kc < kD / 16; ++kc) {
        const uint32_t wa = lds32(kb + swz(ra, kc * 16 + 4 * t4));
        const uint32_t wb = lds32(kb + swz(rb, kc * 16 + 4 * t4));
        mma_f16(sacc[mt], e4m3x2_to_f16x2(wa), e4m3x2_to_f16x2(wb), e4m3x2_to_f16x2(wa >> 16),
                e4m3x2_to_f16x2(wb >> 16), qf[kc][0], qf[kc][1]);
      }
    }
    // keys past the query position (and past kv_len) are masked; log2 domain
    const int kpos0 = key0 + gi;
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      const bool va = kpos0 + 16 * mt <= qpos, vb2 = kpos0 + 16 * mt + 8 <= qpos;
      sacc[mt][0] = va ? sacc[mt][0] * sl2 : -INFINITY;
      sacc[mt][1] = va ? sacc[mt][1] * sl2 : -INFINITY;
      sacc[mt][2] = vb2 ? sacc[mt][2] * sl2 : -INFINITY;
      sacc[mt][3] = vb2 ? sacc[mt][3] * sl2 : -INFINITY;
    }
    uint32_t pb[kMT][2];
    float alpha[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float mx = fmaxf(sacc[0][c], sacc[0][2 + c]);
#pragma unroll
      for (int mt = 1; mt < kMT; ++mt) mx = fmaxf(mx, fmaxf(sacc[mt][c], sacc[mt][2 + c]));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
      const float m_new = fmaxf(m[c], mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      alpha[c] = ex2_approx(m[c] - m_use);
      m[c] = m_new;
      float sum = 0.f;
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        sacc[mt][c] = ex2_approx(sacc[mt][c] - m_use);
        sacc[mt][2 + c] = ex2_approx(sacc[mt][2 + c] - m_use);
        sum += sacc[mt][c] + sacc[mt][2 + c];
      }
      l[c] = l[c] * alpha[c] + sum;
    }
#pragma unroll
    for (int md = 0; md < 8; ++md) {
      oacc[md][0] *= alpha[0];
      oacc[md][2] *= alpha[0];
      oacc[md][1] *= alpha[1];
      oacc[md][3] *= alpha[1];
    }
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      pb[mt][0] = movmatrix_t(pack_f16x2(sacc[mt][0], sacc[mt][1]));
      pb[mt][1] = movmatrix_t(pack_f16x2(sacc[mt][2], sacc[mt][3]));
    }
    // O^T += V^T P^T over the unit's keys
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      const int r0 = 16 * mt + 2 * t4;
#pragma unroll
      for (int qg = 0; qg < kD / 32; ++qg) {
        const int col = 32 * qg + 4 * gi;
        const uint32_t w0 = lds32(vb + swz(r0, col)), w1 = lds32(vb + swz(r0 + 1, col));
        const uint32_t w2 = lds32(vb + swz(r0 + 8, col)), w3 = lds32(vb + swz(r0 + 9, col));
        const uint32_t x01 = prmt(w0, w1, 0x5140), x23 = prmt(w2, w3, 0x5140);
        const uint32_t y01 = prmt(w0, w1, 0x7362), y23 = prmt(w2, w3, 0x7362);
        mma_f16(oacc[2 * qg], e4m3x2_to_f16x2(x01), e4m3x2_to_f16x2(x01 >> 16), e4m3x2_to_f16x2(x23),
                e4m3x2_to_f16x2(x23 >> 16), pb[mt][0], pb[mt][1]);
        mma_f16(oacc[2 * qg + 1], e4m3x2_to_f16x2(y01), e4m3x2_to_f16x2(y01 >> 16), e4m3x2_to_f16x2(y23),
                e4m3x2_to_f16x2(y23 >> 16), pb[mt][0], pb[mt][1]);
      }
    }
    __syncwarp();  // every lane has read the buffer before the next load overwrites it
  }

  // merge the warps' states: each warp's (m, l, O) goes to its own buffer
  // ([head slot][128 + 2] floats), then thread e takes one (head, d)
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    l[c] += __shfl_xor_sync(0xFFFFFFFFu, l[c], 4);
    l[c] += __shfl_xor_sync(0xFFFFFFFFu, l[c], 8);
    l[c] += __shfl_xor_sync(0xFFFFFFFFu, l[c], 16);
  }
  float* sc = reinterpret_cast<float*>(buf);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int h = 2 * t4 + c;
    if (h < G) {
      if (gi == 0) {
        sc[h * (kD + 2) + kD] = ok ? m[c] : -INFINITY;
        sc[h * (kD + 2) + kD + 1] = l[c];
      }
#pragma unroll
      for (int md = 0; md < 8; ++md) {
        const int d0 = 32 * (md >> 1) + 4 * gi + 2 * (md & 1);
        sc[h * (kD + 2) + d0] = oacc[md][c];
        sc[h * (kD + 2) + d0 + 1] = oacc[md][2 + c];
      }
    }
  }
  __syncthreads();
  const float vs = v_scale[kvh];
  for (int e = threadIdx.x; e < G * kD; e += kWsThreads) {
    const int h = e / kD, d = e % kD;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWsWarps; ++w)
      mm = fmaxf(mm, reinterpret_cast<const float*>(smem + w * kBufBytes)[h * (kD + 2) + kD]);
    float Lsum = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kWsWarps; ++w) {
      const float* p = reinterpret_cast<const float*>(smem + w * kBufBytes) + h * (kD + 2);
      const float s = p[kD] == -INFINITY ? 0.f : ex2_approx(p[kD] - mm);
      Lsum += p[kD + 1] * s;
      o += p[d] * s;
    }
    const int64_t orow = static_cast<int64_t>(tl.q_begin) * hq + g * G + h;
    out[orow * kD + d] = __float2bfloat16_rn(Lsum > 0.f ? o / Lsum * vs : 0.f);
    if (d == 0 && lse != nullptr) lse[orow] = Lsum > 0.f ? (mm + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
  }
}

}  // namespace

bool decode_ws_applies(const msa_plan_s* p) {
  return p->n_tiles * p->hp >= p->num_sms && p->hq / p->hp <= 8 && p->topk <= kMaxTopk && p->d == kD;
}

msa_status launch_attn_decode_ws(const msa_plan_s* p, const void* q, const void* k_pages, const void* v_pages,
                                 const int32_t* kv_indices, const int32_t* idx, const float* k_scale,
                                 const float* v_scale, void* out, float* lse, cudaStream_t st) {
  CUtensorMap km, vm;
  const uint64_t dims[2] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(p->num_pages) * p->hkv * 128};
  const uint64_t str[1] = {static_cast<uint64_t>(kD)};
  const uint32_t box[2] = {static_cast<uint32_t>(kD), static_cast<uint32_t>(kKeys)};
  if (!encode_tensor_map(&km, 2, k_pages, dims, str, box, 0, 128) ||
      !encode_tensor_map(&vm, 2, v_pages, dims, str, box, 0, 128))
    return set_error(MSA_ERR_CUDA, "msa_sparse_attn: tensor map encoding failed");
  const int smem = WsSmem::kBytes + 1024;
  cudaFuncSetAttribute(decode_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return cuda_check(launch_pdl(decode_ws_kernel, dim3(p->n_tiles * p->hp), dim3(kWsThreads), smem, st, km, vm,
                                static_cast<const __nv_bfloat16*>(q), p->tiles_d, idx, kv_indices, p->num_pages,
                                k_scale, v_scale, static_cast<__nv_bfloat16*>(out), lse, p->hq, p->hp,
                                p->hp / p->hkv, p->topk, 1.4426950408889634f / sqrtf(static_cast<float>(kD)),
                                p->err_d),
                    "msa_sparse_attn: decode launch");
}

}  // namespace msa
