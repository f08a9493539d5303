// Stage 1 at decode with an NVFP4 proxy K: the FP4 block-score indexer
// ("MiniMax-AI/MSA" README, section "Stacks": an FP4 block-score indexer next
// to the FP8 paged decode; Flash-MSA article, "what's next": training the
// indexer in low precision).
//
// The shared proxy K head is stored in NVFP4: e2m1 codes, two per byte (the
// low nibble holds the even dimension), one e4m3 scale per 16 consecutive
// dimensions of a key, and one fp32 scale for the whole head.  A key's value
// is pk[k, d] = code(k, d) * block_scale(k, d / 16) * global_scale, so the
// logit of a pair is (pq . (code * block_scale))[k] * global_scale / sqrt(dp),
// and max_score is defined as for msa_proxy_maxscore.  code * block_scale is
// exact in f16 (at most 2 x 4 significant bits, magnitudes 2^-10 .. 2688),
// so the dot products run on f16 mma.sync with pq rounded to f16; the global
// scale is positive and is applied once to each block maximum.
//
// A decode proxy pass reads every valid block of every sequence once: an HBM
// stream of 4 KB of codes and 512 B of scales per (sequence, block), a
// quarter of the bf16 proxy K.  Each warp takes a contiguous range of
// (sequence, block) units and streams them through its own bulk copies; per unit it computes S^T = K . pq^T (M = 128 keys, N = 8 heads,
// K = 64 dims) and a max over keys.  Lane (g, t4) reads the 32-bit words t4
// and t4 + 4 of key rows g and g + 8 of an m-tile (eight dims each) and the
// pq fragments use the same dimension order (a dot product does not depend
// on the order of its terms).
#include "msa_internal.h"
#include "ptx.cuh"

#include <algorithm>

namespace msa {
namespace {

constexpr int kDP = 64;
constexpr int kCodeBytes = 128 * kDP / 2;    // e2m1 codes of one page
constexpr int kScaleBytes = 128 * kDP / 16;  // e4m3 block scales of one page
constexpr int kStageBytes = kCodeBytes + kScaleBytes;
// warps per CTA and ring stages per warp, one CTA per SM; measured at 32 x
// 131072 keys (warps x stages): 16 x 2 40.3 us, 16 x 3 41.4, 12 x 4 42.8, 8 x 6
// 49.4, 32 x 1 36.5, 24 x 1 36.0; with the m-tile loop fully unrolled 16 x 2
// 38.5 and 24 x 1 35.3 us: the loads in flight come from many warps
constexpr int kFp4Warps = 24;
constexpr int kFp4Stages = 1;

__device__ __forceinline__ int unit_range_start(int w, int total, int nw) {
  const int q = total / nw, r = total % nw;
  return w * q + (w < r ? w : r);
}

// four bytes of e2m1 pairs -> four f16x2 (byte b -> out[b], low nibble in the low half)
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t* out) {
  asm("{\n\t.reg .b8 a, b, c, d;\n\t"
      "mov.b32 {a, b, c, d}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, a;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, c;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, d;\n\t}"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(w));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// e4m3 byte `b` of w as an f16 in both halves
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t w, int b) {
  const uint32_t h = e4m3x2_to_f16x2(w >> (8 * b));  // low half: byte b
  return prmt(h, h, 0x1010);
}

template <int W, int S>
__global__ void __launch_bounds__(32 * W)
    proxy_decode_nvfp4_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ bscale,
                              const float* __restrict__ gscale, const __nv_bfloat16* __restrict__ pq,
                              const TileInfo* __restrict__ tiles, const int32_t* __restrict__ unit_start,
                              int32_t n_tiles, const int32_t* __restrict__ kv_indices, int64_t num_pages,
                              float* __restrict__ max_score, int32_t hp, int32_t max_blocks, float scale,
                              uint32_t* err) {
  pdl_wait();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + warp * S * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + W * S * kStageBytes) + warp * S;
  const float out_scale = scale * gscale[0];

  const int total_units = unit_start[n_tiles];
  // -inf past each sequence's valid blocks
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       e < static_cast<int64_t>(n_tiles) * hp * max_blocks; e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(e % max_blocks);
    const int t = static_cast<int>(e / (static_cast<int64_t>(hp) * max_blocks));
    if (j >= tiles[t].nvp) max_score[e] = -INFINITY;
  }

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(bars + s, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const int nw = gridDim.x * W;
  const int gw = blockIdx.x * W + warp;
  const int ub = unit_range_start(gw, total_units, nw), ue = unit_range_start(gw + 1, total_units, nw);
  const int n = ue - ub;

  // lane l holds the tile, block and page of the warp's unit base + l
  auto meta = [&](int base, int& t, int& j, int64_t& page) {
    const int unit = base + lane;
    t = 0;
    j = 0;
    page = 0;
    if (unit < ue) {
      int lo = 0, hi = n_tiles - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(unit_start + mid) <= unit) lo = mid; else hi = mid - 1;
      }
      t = lo;
      j = unit - __ldg(unit_start + lo);
      page = kv_indices[tiles[t].page_base + j];
      if (page < 0 || page >= num_pages) {
        atomicOr(err, kErrDeviceCheck);
        page = 0;
      }
    }
  };
  int ct, cj, nt_, nj;
  int64_t cpage, npage;
  meta(ub, ct, cj, cpage);
  meta(ub + 32, nt_, nj, npage);
  int chunk = 0;
  auto issue = [&](int i) {  // the warp's i-th unit into stage i % S
    if (i >= n) return;
    const int ii = i - 32 * chunk;
    const long long p_cur = __shfl_sync(0xFFFFFFFFu, static_cast<long long>(cpage), ii & 31);
    const long long p_nxt = __shfl_sync(0xFFFFFFFFu, static_cast<long long>(npage), ii & 31);
    const int64_t page = (ii >> 5) == 0 ? p_cur : p_nxt;
    if (lane == 0) {
      uint64_t* bar = bars + (i % S);
      uint8_t* st = ring + (i % S) * kStageBytes;
      mbar_expect_tx(bar, kStageBytes);
      bulk_load(st, codes + page * kCodeBytes, kCodeBytes, bar);
      bulk_load(st + kCodeBytes, bscale + page * kScaleBytes, kScaleBytes, bar);
    }
  };
  for (int i = 0; i < S; ++i) issue(i);

  const int g = lane >> 2, t4 = lane & 3;
  for (int i = 0; i < n; ++i) {
    if (i - 32 * chunk == 32) {
      ct = nt_;
      cj = nj;
      cpage = npage;
      ++chunk;
      meta(ub + 32 * (chunk + 1), nt_, nj, npage);
    }
    const int t = __shfl_sync(0xFFFFFFFFu, ct, i & 31);
    const int j = __shfl_sync(0xFFFFFFFFu, cj, i & 31);
    const TileInfo tl = tiles[t];
    // B fragments of k-chunk kc: head g, the dims 32 (kc / 2) + 8 t4 + 4 (kc % 2) + {0,1} | {2,3}
    uint32_t bf[kDP / 16][2];
    const __nv_bfloat16* qrow = pq + (static_cast<int64_t>(tl.q_begin) * hp + g) * kDP;
#pragma unroll
    for (int kc = 0; kc < kDP / 16; ++kc) {
      if (g < hp) {
        const uint2 v = *reinterpret_cast<const uint2*>(qrow + 32 * (kc >> 1) + 8 * t4 + 4 * (kc & 1));
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
        const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
        bf[kc][0] = pack_f16x2(f0.x, f0.y);
        bf[kc][1] = pack_f16x2(f1.x, f1.y);
      } else {
        bf[kc][0] = bf[kc][1] = 0u;
      }
    }
    const int s = i % S;
    if (!mbar_wait(bars + s, (i / S) & 1, err)) break;
    const uint32_t cbase = smem_u32(ring + s * kStageBytes);
    const uint32_t sbase = cbase + kCodeBytes;
    const int nkeys = min(128, tl.kv_len - j * 128);
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      const int ra = mt * 16 + g, rb = ra + 8;
      // word h of a row holds dims 32 h' + 8 t4 .. +7 for h = t4 + 4 h'; their
      // scale is byte 2 h' + t4 / 2 of the row's four block scales
      const uint32_t swa = lds32(sbase + ra * 4), swb = lds32(sbase + rb * 4);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t wa = lds32(cbase + ra * 32 + 4 * (t4 + 4 * hh));
        const uint32_t wb = lds32(cbase + rb * 32 + 4 * (t4 + 4 * hh));
        const uint32_t sa = scale_f16x2(swa, 2 * hh + (t4 >> 1)), sb = scale_f16x2(swb, 2 * hh + (t4 >> 1));
        uint32_t xa[4], xb[4];
        e2m1x8_to_f16x2x4(wa, xa);
        e2m1x8_to_f16x2x4(wb, xb);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          xa[q] = hmul2(xa[q], sa);
          xb[q] = hmul2(xb[q], sb);
        }
        // k-chunk 2 hh takes this lane's dims +0..3 (pairs 0, 1), k-chunk 2 hh + 1 dims +4..7
        mma_f16(c, xa[0], xb[0], xa[1], xb[1], bf[2 * hh][0], bf[2 * hh][1]);
        mma_f16(c, xa[2], xb[2], xa[3], xb[3], bf[2 * hh + 1][0], bf[2 * hh + 1][1]);
      }
      if (ra < nkeys) { mx0 = fmaxf(mx0, c[0]); mx1 = fmaxf(mx1, c[1]); }
      if (rb < nkeys) { mx0 = fmaxf(mx0, c[2]); mx1 = fmaxf(mx1, c[3]); }
    }
    __syncwarp();
    issue(i + S);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, o));
    }
    if (lane < 4) {
      const int h0 = 2 * lane, h1 = 2 * lane + 1;
      float* dst = max_score + static_cast<int64_t>(t) * hp * max_blocks + j;
      if (h0 < hp) dst[static_cast<int64_t>(h0) * max_blocks] = mx0 * out_scale;
      if (h1 < hp) dst[static_cast<int64_t>(h1) * max_blocks] = mx1 * out_scale;
    }
  }
}

}  // namespace

msa_status launch_proxy_decode_nvfp4(const msa_plan_s* p, const void* pq, const void* pk_codes,
                                     const void* pk_block_scales, const float* pk_global_scale,
                                     const int32_t* kv_indices, float* max_score, cudaStream_t st) {
  if (p->hp > 8) return set_error(MSA_ERR_UNSUPPORTED, "msa_proxy_maxscore_nvfp4: up to 8 proxy heads");
  if (p->dp != kDP) return set_error(MSA_ERR_UNSUPPORTED, "msa_proxy_maxscore_nvfp4: proxy_head_dim 64 only");
  const int32_t* ustart = p->aux_d + p->proxy_unit_start_off;
  constexpr int W = kFp4Warps, S = kFp4Stages;
  const int smem = W * S * kStageBytes + W * S * 8 + 1024;
  cudaFuncSetAttribute(proxy_decode_nvfp4_kernel<W, S>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return cuda_check(launch_pdl(proxy_decode_nvfp4_kernel<W, S>, dim3(p->num_sms), dim3(32 * W), smem, st,
                                static_cast<const uint8_t*>(pk_codes), static_cast<const uint8_t*>(pk_block_scales),
                                pk_global_scale, static_cast<const __nv_bfloat16*>(pq), p->tiles_d, ustart,
                                p->n_tiles, kv_indices, p->num_pages, max_score, p->hp, p->max_blocks,
                                1.0f / sqrtf(static_cast<float>(kDP)), p->err_d),
                    "msa_proxy_maxscore_nvfp4: launch");
}

}  // namespace msa
