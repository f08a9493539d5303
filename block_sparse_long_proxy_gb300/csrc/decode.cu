// Stage 3 (decode): paged sparse attention with FP8 e4m3 K/V, one query row
// per sequence ("MiniMax-AI/MSA" README, section "Stacks": paged FP8 decode
// next to the BF16 sparse prefill).  For each sequence and query head h of
// group g: softmax over the keys of the blocks kv_block_indexes[t, g, :] of
// q.(k_code*k_scale[g])/sqrt(d); out = P.(v_code*v_scale[g]).
//
// The work is HBM-bound (every selected block is read once; 8 query heads
// share it), so the kernel is a stream over (tile, group, slot) units:
// CTA c takes a contiguous range of units, a producer warp gathers each
// selected block's K and V page (16 KB each at d = 128) through a 3-stage
// TMA ring with 128-byte swizzle, and four consumer warps each take 32 of
// the block's 128 keys.  Tensor cores via mma.sync (f16 in, f32 out):
//   S^T = K . q^T     M = keys, N = 8 heads, K = d   (e4m3 -> f16 in registers)
//   O^T += V^T . P^T  M = d,    N = 8 heads, K = keys (P^T by movmatrix)
// The d index of both products is permuted so that every shared-memory
// read is one conflict-free 32-bit word; the output is un-permuted on store.
// Each warp keeps its own online-softmax state (m, l, O); the four warps'
// states are merged in shared memory whenever the CTA's range leaves a
// (tile, group) row, giving one partial per row segment.  A second kernel
// merges the (at most a few) segments of each row, applies v_scale and
// writes out and lse.
#include "msa_internal.h"
#include "ptx.cuh"

#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

namespace msa {
namespace {

constexpr int kD = 128;                 // head dim of this kernel
constexpr int kCWarps = 4;              // consumer warps
constexpr int kKeysW = 128 / kCWarps;   // keys of a block per consumer warp
constexpr int kMT = kKeysW / 16;        // 16-key m-tiles per consumer warp
constexpr int kRounds = 2;              // the merge moves d in kRounds slices
constexpr int kDR = 128 / kRounds;      // d per merge slice
static_assert(kRounds == 1 || kRounds == 2 || kRounds == 4, "a merge slice holds whole m-tile pairs");
static_assert(kMT >= 1 && kKeysW % 16 == 0, "consumer warps take whole 16-key m-tiles");
constexpr int kDThreads = 32 * (kCWarps + 1);
constexpr int kDStages = 3;
constexpr int kBlk = 128 * kD;          // bytes of one e4m3 K (or V) block

// byte offset of (row, byte col) in a 128-row x 128-byte tile written by TMA
// with 128-byte swizzle: the 16-byte chunk index is XORed with row % 8.
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return row * 128 + ((((col >> 4) ^ row) & 7) << 4) + (col & 15);
}

// first unit of CTA c when U units are cut into C near-equal ranges
__host__ __device__ __forceinline__ int range_start(int c, int U, int C) {
  const int q = U / C, r = U % C;
  return c * q + (c < r ? c : r);
}
// the CTA whose range holds unit u (inverse of range_start)
__device__ __forceinline__ int range_owner(int u, int U, int C) {
  const int q = U / C, r = U % C;
  return u < r * (q + 1) ? u / (q + 1) : r + (u - r * (q + 1)) / q;
}

template <int NT>
struct DecodeSmem {
  static constexpr int kRingOff = 0;
  static constexpr int kScratchOff = kDStages * 2 * kBlk;
  // per-warp merge scratch, one slice of d at a time: [warp][head slot][kDR + 2]
  static constexpr int kScratchFloats = kCWarps * 8 * NT * (kDR + 2);
  static constexpr int kBarOff = kScratchOff + kScratchFloats * 4;
  static constexpr int kStageJOff = kBarOff + 8 * 2 * kDStages;
  static constexpr int kFlagOff = kStageJOff + 4 * kDStages;
  static constexpr int kBytes = kFlagOff + 4;
};

template <int NT>  // n-tiles of 8 heads: group size G <= 8*NT
__global__ void __launch_bounds__(kDThreads, NT == 1 ? 2 : 1)
    decode_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                  const __nv_bfloat16* __restrict__ q, const TileInfo* __restrict__ tiles,
                  const int32_t* __restrict__ idx, const int32_t* __restrict__ kv_indices, int64_t num_pages,
                  const float* __restrict__ k_scale, const float* __restrict__ v_scale, float* __restrict__ part_o,
                  float* __restrict__ part_ml, int32_t* __restrict__ row_cnt, __nv_bfloat16* __restrict__ out,
                  float* __restrict__ lse, int32_t n_units, int32_t hq, int32_t hsel, int32_t kv_div, int32_t topk,
                  float scale_log2, uint32_t* err) {
  pdl_wait();
  // A row is (sequence, proxy head p): the G = hq / hsel query heads of p
  // attend over p's blocks of KV head p / kv_div (kv_div proxy heads per KV
  // head; 1 when there is one proxy head per GQA group).
  const int hkv = hsel / kv_div;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using L = DecodeSmem<NT>;
  constexpr int kSlots = 8 * NT;  // head slots of the per-warp scratch
  constexpr int kHalf = kDR;
  uint8_t* ring = smem + L::kRingOff;
  float* scratch = reinterpret_cast<float*>(smem + L::kScratchOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + kDStages;
  volatile int32_t* stage_j = reinterpret_cast<int32_t*>(smem + L::kStageJOff);
  volatile int32_t* merge_flag = reinterpret_cast<int32_t*>(smem + L::kFlagOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = hq / hsel;
  const int ub = range_start(blockIdx.x, n_units, gridDim.x);
  const int ue = range_start(blockIdx.x + 1, n_units, gridDim.x);

  if (threadIdx.x == 0) {
    prefetch_tmap(&k_map);
    prefetch_tmap(&v_map);
    for (int s = 0; s < kDStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kCWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kCWarps) {
    // ---------------------------------------------------------- producer
    // One ring stage per unit, in unit order.  The block index travels with
    // the stage (stage_j, -1 for a padding slot, which loads nothing).  The
    // metadata of 32 units at a time is fetched lane-parallel so that its
    // dependent global loads stay off the per-unit critical path.
    bool ok = true;
    int i = 0;
    for (int base = ub; ok && base < ue; base += 32) {
      const int u = base + lane;
      int j = -1, row_off = 0;
      if (u < ue) {
        const int row = u / topk;
        const int t = row / hsel, g = row % hsel;
        j = idx[u];
        const TileInfo tl = tiles[t];
        if (j >= tl.nvp) {
          atomicOr(err, kErrDeviceCheck);
          j = -1;
        }
        if (j >= 0) {
          int64_t page = kv_indices[tl.page_base + j];
          if (page < 0 || page >= num_pages) {
            atomicOr(err, kErrDeviceCheck);
            page = 0;
          }
          row_off = static_cast<int>((page * hkv + g / kv_div) * 128);
        }
      }
      const int n = min(32, ue - base);
      for (int k = 0; k < n; ++k, ++i) {
        const int jk = __shfl_sync(0xFFFFFFFFu, j, k);
        const int rk = __shfl_sync(0xFFFFFFFFu, row_off, k);
        if (lane == 0) {
          const int s = i % kDStages;
          if (!(ok = mbar_wait(empty + s, ((i / kDStages) & 1) ^ 1, err))) {
            // leave the loop below too
          } else {
            stage_j[s] = jk;
            if (jk >= 0) {
              mbar_expect_tx(full + s, 2 * kBlk);
              tma_load_2d(ring + s * 2 * kBlk, &k_map, full + s, 0, rk);
              tma_load_2d(ring + s * 2 * kBlk + kBlk, &v_map, full + s, 0, rk);
            } else {
              mbar_arrive(full + s);
            }
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int gi = lane >> 2, t4 = lane & 3;
  const int w = warp;
  int cur_row = -1, seg = 0, i = 0;
  float m[NT][2], l[NT][2], oacc[8][NT][4];
  uint32_t qf[NT][kD / 16][2];
  float sl2 = 0.f;
  int qpos = 0;
  bool ok = true;

  auto flush = [&](int row, int slot) {
    const bool whole = slot == row * topk && ue >= (row + 1) * topk;
    // per-warp totals of l (sum over the 8 key lanes of each head column)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float v = l[nt][c];
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
        l[nt][c] = v;
      }
    // merge the consumer warps' states one slice of d at a time
    float* wsc = scratch + w * kSlots * (kHalf + 2);  // [head slot][kDR + 2]: O slice, m, l
#pragma unroll
    for (int rnd = 0; rnd < kRounds; ++rnd) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int h = 8 * nt + 2 * t4 + c;
          if (h < G) {
            if (gi == 0) {
              wsc[h * (kHalf + 2) + kHalf] = m[nt][c];
              wsc[h * (kHalf + 2) + kHalf + 1] = l[nt][c];
            }
#pragma unroll
            for (int mh = 0; mh < 8 / kRounds; ++mh) {
              const int md = 8 / kRounds * rnd + mh;  // m-tile md holds d in [32(md/2), 32(md/2)+32)
              const int d0 = 32 * (md >> 1) + 4 * gi + 2 * (md & 1) - kHalf * rnd;
              wsc[h * (kHalf + 2) + d0] = oacc[md][nt][c];
              wsc[h * (kHalf + 2) + d0 + 1] = oacc[md][nt][2 + c];
            }
          }
        }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kCWarps) : "memory");
      for (int e = threadIdx.x; e < G * kHalf; e += 32 * kCWarps) {
        const int h = e / kHalf, d = e % kHalf;
        float mm = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < kCWarps; ++ww) mm = fmaxf(mm, scratch[(ww * kSlots + h) * (kHalf + 2) + kHalf]);
        float Lsum = 0.f, o = 0.f;
#pragma unroll
        for (int ww = 0; ww < kCWarps; ++ww) {
          const float* p = scratch + (ww * kSlots + h) * (kHalf + 2);
          const float sc = p[kHalf] == -INFINITY ? 0.f : ex2_approx(p[kHalf] - mm);
          Lsum += p[kHalf + 1] * sc;
          o += p[d] * sc;
        }
        if (whole) {  // this CTA holds the whole row: write the result directly
          const int t = row / hsel, g = row % hsel;
          const int64_t orow = static_cast<int64_t>(tiles[t].q_begin) * hq + g * G + h;
          out[orow * kD + kHalf * rnd + d] = __float2bfloat16_rn(Lsum > 0.f ? o / Lsum * v_scale[g / kv_div] : 0.f);
          if (d == 0 && rnd == 0 && lse != nullptr)
            lse[orow] = Lsum > 0.f ? (mm + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
        } else {
          const int64_t base = static_cast<int64_t>(slot) * G + h;
          part_o[base * kD + kHalf * rnd + d] = o;
          if (d == 0 && rnd == 0) {
            part_ml[base * 2] = mm;
            part_ml[base * 2 + 1] = Lsum;
          }
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kCWarps) : "memory");
    }
    if (whole) return;
    // The CTA that completes a row's last segment merges all of them:
    // partials are made visible with a fence, then counted per row.
    __threadfence();
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kCWarps) : "memory");
    // The row's segments start at u0 and at every range start inside it:
    // one per CTA from the owner of u0 to the owner of its last unit.
    const int u0 = row * topk;
    const int c0 = range_owner(u0, n_units, gridDim.x);
    const int c1 = range_owner(u0 + topk - 1, n_units, gridDim.x);
    const int rq = n_units / gridDim.x, rr = n_units % gridDim.x;
    if (threadIdx.x == 0) {
      const int old = atomicAdd(row_cnt + row, 1);
      const bool last = old == c1 - c0;
      if (last) row_cnt[row] = 0;  // ready for the next call
      *merge_flag = last;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kCWarps) : "memory");
    if (*merge_flag) {
      // Online merge over the row's segments, one segment per step: every
      // thread owns one d column of all G heads, so the loads of a segment
      // (m, l and O of each head) are independent and issue together.
      __threadfence();
      const int t = row / hsel, g = row % hsel;
      const float vs = v_scale[g / kv_div];
      const int64_t q_row = tiles[t].q_begin;
      for (int d = threadIdx.x; d < kD; d += 32 * kCWarps)
#pragma unroll 1
        for (int hb = 0; hb < G; hb += 8) {  // eight heads at a time
          float M[8], Ls[8], Od[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) M[k] = -INFINITY, Ls[k] = 0.f, Od[k] = 0.f;
          for (int c = c0; c <= c1; ++c) {
            const int64_t b0 = static_cast<int64_t>(max(u0, c * rq + min(c, rr))) * G + hb;
            float ms[8], ls[8], po[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              if (hb + k < G) {
                ms[k] = __ldcg(part_ml + (b0 + k) * 2);
                ls[k] = __ldcg(part_ml + (b0 + k) * 2 + 1);
                po[k] = __ldcg(part_o + (b0 + k) * kD + d);
              }
#pragma unroll
            for (int k = 0; k < 8; ++k)
              if (hb + k < G && ms[k] != -INFINITY) {
                const float mn = fmaxf(M[k], ms[k]);
                const float a = ex2_approx(M[k] - mn), sc = ex2_approx(ms[k] - mn);
                Ls[k] = Ls[k] * a + ls[k] * sc;
                Od[k] = Od[k] * a + po[k] * sc;
                M[k] = mn;
              }
          }
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (hb + k < G) {
              const int64_t orow = q_row * hq + g * G + hb + k;
              out[orow * kD + d] = __float2bfloat16_rn(Ls[k] > 0.f ? Od[k] / Ls[k] * vs : 0.f);
              if (d == 0 && lse != nullptr)
                lse[orow] = Ls[k] > 0.f ? (M[k] + log2f(Ls[k])) * 0.69314718055994531f : -INFINITY;
            }
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kCWarps) : "memory");
  };

  for (int u = ub; u < ue; ++u) {
    const int row = u / topk;
    const int t = row / hsel, g = row % hsel;
    if (row != cur_row) {
      if (cur_row >= 0) flush(cur_row, seg);
      cur_row = row;
      seg = u;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
        for (int md = 0; md < 8; ++md) oacc[md][nt][0] = oacc[md][nt][1] = oacc[md][nt][2] = oacc[md][nt][3] = 0.f;
      }
      const TileInfo tl = tiles[t];
      qpos = tl.pos0;
      sl2 = scale_log2 * k_scale[g / kv_div];
      // q^T fragments: head n = gi + 8nt of the group, d = 16kc + 4t4 + {0,1} | {2,3}
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int hl = gi + 8 * nt;
        const __nv_bfloat16* qr = q + (static_cast<int64_t>(tl.q_begin) * hq + g * G + hl) * kD;
#pragma unroll
        for (int kc = 0; kc < kD / 16; ++kc) {
          if (hl < G) {
            const uint2 v = *reinterpret_cast<const uint2*>(qr + kc * 16 + 4 * t4);
            const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
            const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
            qf[nt][kc][0] = pack_f16x2(f0.x, f0.y);
            qf[nt][kc][1] = pack_f16x2(f1.x, f1.y);
          } else {
            qf[nt][kc][0] = qf[nt][kc][1] = 0u;
          }
        }
      }
    }
    const int s = i % kDStages;
    ++i;
    if (!ok || !(ok = mbar_wait(full + s, ((i - 1) / kDStages) & 1, err))) continue;  // after a timeout: no
    const int j = stage_j[s];                                                         // compute, but every
    if (j < 0) {                                                                      // flush still runs
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
      continue;
    }
    const uint32_t kb = smem_u32(ring + s * 2 * kBlk);
    const uint32_t vb = kb + kBlk;

    // S^T for this warp's 32 keys
    float sacc[kMT][NT][4];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) sacc[mt][nt][0] = sacc[mt][nt][1] = sacc[mt][nt][2] = sacc[mt][nt][3] = 0.f;
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      const int ra = kKeysW * w + 16 * mt + gi, rb = ra + 8;
#pragma unroll
      for (int kc = 0; kc < kD / 16; ++kc) {
        const uint32_t wa = lds32(kb + swz(ra, kc * 16 + 4 * t4));
        const uint32_t wb = lds32(kb + swz(rb, kc * 16 + 4 * t4));
        const uint32_t a0 = e4m3x2_to_f16x2(wa), a1 = e4m3x2_to_f16x2(wb);
        const uint32_t a2 = e4m3x2_to_f16x2(wa >> 16), a3 = e4m3x2_to_f16x2(wb >> 16);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_f16(sacc[mt][nt], a0, a1, a2, a3, qf[nt][kc][0], qf[nt][kc][1]);
      }
    }
    // mask keys past the query position, scale into the log2 domain
    const int kpos0 = j * 128 + kKeysW * w + gi;
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      const bool va = kpos0 + 16 * mt <= qpos, vb2 = kpos0 + 16 * mt + 8 <= qpos;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        sacc[mt][nt][0] = va ? sacc[mt][nt][0] * sl2 : -INFINITY;
        sacc[mt][nt][1] = va ? sacc[mt][nt][1] * sl2 : -INFINITY;
        sacc[mt][nt][2] = vb2 ? sacc[mt][nt][2] * sl2 : -INFINITY;
        sacc[mt][nt][3] = vb2 ? sacc[mt][nt][3] * sl2 : -INFINITY;
      }
    }
    // online softmax per head column
    uint32_t pb[kMT][NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float alpha[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float mx = fmaxf(sacc[0][nt][c], sacc[0][nt][2 + c]);
#pragma unroll
        for (int mt = 1; mt < kMT; ++mt) mx = fmaxf(mx, fmaxf(sacc[mt][nt][c], sacc[mt][nt][2 + c]));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
        const float m_new = fmaxf(m[nt][c], mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        alpha[c] = ex2_approx(m[nt][c] - m_use);
        m[nt][c] = m_new;
        float sum = 0.f;
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          sacc[mt][nt][c] = ex2_approx(sacc[mt][nt][c] - m_use);
          sacc[mt][nt][2 + c] = ex2_approx(sacc[mt][nt][2 + c] - m_use);
          sum += sacc[mt][nt][c] + sacc[mt][nt][2 + c];
        }
        l[nt][c] = l[nt][c] * alpha[c] + sum;
      }
#pragma unroll
      for (int md = 0; md < 8; ++md) {
        oacc[md][nt][0] *= alpha[0];
        oacc[md][nt][2] *= alpha[0];
        oacc[md][nt][1] *= alpha[1];
        oacc[md][nt][3] *= alpha[1];
      }
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        pb[mt][nt][0] = movmatrix_t(pack_f16x2(sacc[mt][nt][0], sacc[mt][nt][1]));
        pb[mt][nt][1] = movmatrix_t(pack_f16x2(sacc[mt][nt][2], sacc[mt][nt][3]));
      }
    }
    // O^T += V^T P^T over this warp's 32 keys
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      const int r0 = kKeysW * w + 16 * mt + 2 * t4;
#pragma unroll
      for (int qg = 0; qg < kD / 32; ++qg) {
        const int col = 32 * qg + 4 * gi;
        const uint32_t w0 = lds32(vb + swz(r0, col)), w1 = lds32(vb + swz(r0 + 1, col));
        const uint32_t w2 = lds32(vb + swz(r0 + 8, col)), w3 = lds32(vb + swz(r0 + 9, col));
        const uint32_t x01 = prmt(w0, w1, 0x5140), x23 = prmt(w2, w3, 0x5140);
        const uint32_t y01 = prmt(w0, w1, 0x7362), y23 = prmt(w2, w3, 0x7362);
        const uint32_t a0 = e4m3x2_to_f16x2(x01), a1 = e4m3x2_to_f16x2(x01 >> 16);
        const uint32_t a2 = e4m3x2_to_f16x2(x23), a3 = e4m3x2_to_f16x2(x23 >> 16);
        const uint32_t b0 = e4m3x2_to_f16x2(y01), b1 = e4m3x2_to_f16x2(y01 >> 16);
        const uint32_t b2 = e4m3x2_to_f16x2(y23), b3 = e4m3x2_to_f16x2(y23 >> 16);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_f16(oacc[2 * qg][nt], a0, a1, a2, a3, pb[mt][nt][0], pb[mt][nt][1]);
          mma_f16(oacc[2 * qg + 1][nt], b0, b1, b2, b3, pb[mt][nt][0], pb[mt][nt][1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + s);
  }
  if (cur_row >= 0) flush(cur_row, seg);
}

// One CTA per (sequence, group) row when there are enough rows to fill the
// GPU (no partials, no merge); otherwise rows are cut into near-equal unit
// ranges over all SMs and merged by the last CTA of each row.
int decode_grid_rows(int rows, int topk, int num_sms, int G) {
  if (rows >= num_sms) return rows;
  const int per_sm = G <= 8 ? 2 : 1;
  return std::max(1, std::min(rows * topk, num_sms * per_sm));
}

}  // namespace

size_t decode_partial_floats(const msa_plan_s* p) {
  if (!p->decode) return 0;
  // rows are (sequence, proxy head): one block set each
  const size_t units = static_cast<size_t>(p->n_tiles) * p->hp * p->topk;
  const size_t g = p->hq / p->hp;
  return units * g * (kD + 2) + static_cast<size_t>(p->n_tiles) * p->hp;  // partials + per-row counters
}

msa_status launch_attn_decode(const msa_plan_s* p, const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* kv_indices, const int32_t* idx, const float* k_scale,
                              const float* v_scale, void* out, float* lse, cudaStream_t st) {
  if (p->d != kD) return set_error(MSA_ERR_UNSUPPORTED, "msa_sparse_attn: FP8 decode needs head_dim 128");
  if (p->hq / p->hp > 16)
    return set_error(MSA_ERR_UNSUPPORTED, "msa_sparse_attn: FP8 decode needs at most 16 query heads per proxy head");
  if (decode_ws_applies(p))
    return launch_attn_decode_ws(p, q, k_pages, v_pages, kv_indices, idx, k_scale, v_scale, out, lse, st);
  CUtensorMap km, vm;
  const uint64_t dims[2] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(p->num_pages) * p->hkv * 128};
  const uint64_t str[1] = {static_cast<uint64_t>(kD)};
  const uint32_t box[2] = {static_cast<uint32_t>(kD), 128};
  if (!encode_tensor_map(&km, 2, k_pages, dims, str, box, 0, 128) ||
      !encode_tensor_map(&vm, 2, v_pages, dims, str, box, 0, 128))
    return set_error(MSA_ERR_CUDA, "msa_sparse_attn: tensor map encoding failed");
  const int n_units = p->n_tiles * p->hp * p->topk;
  const int grid = decode_grid_rows(p->n_tiles * p->hp, p->topk, p->num_sms, p->hq / p->hp);
  const size_t units = static_cast<size_t>(n_units);
  const int G = p->hq / p->hp;
  const int kv_div = p->hp / p->hkv;
  float* part_o = p->partial_d;
  float* part_ml = p->partial_d + units * G * kD;
  int32_t* row_cnt = reinterpret_cast<int32_t*>(part_ml + units * G * 2);  // zeroed by msa_plan
  auto* o_ptr = static_cast<__nv_bfloat16*>(out);
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kD));
  const auto* qq = static_cast<const __nv_bfloat16*>(q);
  cudaError_t e;
  if (G <= 8) {
    const int smem = DecodeSmem<1>::kBytes + 1024;
    cudaFuncSetAttribute(decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    e = launch_pdl(decode_kernel<1>, dim3(grid), dim3(kDThreads), smem, st, km, vm, qq, p->tiles_d, idx, kv_indices,
                   p->num_pages, k_scale, v_scale, part_o, part_ml, row_cnt, o_ptr, lse, n_units, p->hq, p->hp, kv_div,
                   p->topk, scale_log2, p->err_d);
  } else {
    const int smem = DecodeSmem<2>::kBytes + 1024;
    cudaFuncSetAttribute(decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    e = launch_pdl(decode_kernel<2>, dim3(grid), dim3(kDThreads), smem, st, km, vm, qq, p->tiles_d, idx, kv_indices,
                   p->num_pages, k_scale, v_scale, part_o, part_ml, row_cnt, o_ptr, lse, n_units, p->hq, p->hp, kv_div,
                   p->topk, scale_log2, p->err_d);
  }
  return cuda_check(e, "msa_sparse_attn: decode launch");
}

}  // namespace msa

// ---------------------------------------------------------------------------
// Allocation-free FP8 decode (msa_sparse_decode_noalloc).
//
// Some callers cannot allocate device memory at the time they decode: a
// serving process that hands all of the GPU's memory to its own pool at
// start-up, or a decode loop that must not pay for cudaMalloc's implicit
// synchronisation.  Such a caller cannot create a plan (msa_plan
// allocates), so this entry point takes the batch description as device
// arrays and keeps every piece of scratch -- the tile table and the split-K
// partials of the decode kernel above -- in one file-scope device array of
// fixed size, which every GPU that loads libmsa holds until the process
// exits.  Its device address is fetched once per device with
// cudaGetSymbolAddress; host code never hands the symbol itself to a kernel.
// ---------------------------------------------------------------------------

namespace msa {

constexpr size_t kStaticScratchBytes = size_t(24) << 20;  // 24 MiB
constexpr int kStaticMaxBatch = 4096;
constexpr size_t kStaticTilesBytes = sizeof(TileInfo) * kStaticMaxBatch;
constexpr size_t kStaticErrOff = kStaticTilesBytes;
constexpr int kStaticMaxRows = 65536;  // batch * num_kv_heads
constexpr size_t kStaticCntOff = kStaticTilesBytes + 256;
constexpr size_t kStaticPartOff = kStaticCntOff + sizeof(int32_t) * kStaticMaxRows;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

namespace {

struct StaticDevice {
  unsigned char* base = nullptr;  // device address of g_decode_scratch on this device
  int num_sms = 0;
  bool ready = false;
};
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
StaticDevice g_static[kMaxDevices];

// One-time set-up per device, run with that device current.
msa_status static_scratch(StaticDevice* out) {
  int dev = -1;
  msa_status s = cuda_check(cudaGetDevice(&dev), "msa_sparse_decode_noalloc: cudaGetDevice");
  if (s != MSA_OK) return s;
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(MSA_ERR_UNSUPPORTED, "msa_sparse_decode_noalloc: device index %d above %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_static_mu);
  StaticDevice& sd = g_static[dev];
  if (!sd.ready) {
    void* ptr = nullptr;
    s = cuda_check(cudaGetSymbolAddress(&ptr, g_decode_scratch), "msa_sparse_decode_noalloc: cudaGetSymbolAddress");
    if (s != MSA_OK) return s;
    int sms = 0;
    s = cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                   "msa_sparse_decode_noalloc: SM count");
    if (s != MSA_OK) return s;
    sd.base = static_cast<unsigned char*>(ptr);
    sd.num_sms = sms;
    sd.ready = true;
  }
  *out = sd;
  return MSA_OK;
}

// Tile table of a decode batch (one query row per sequence) from device
// kv_lens / kv_indptr.  A sequence whose page range is shorter than its
// kv_len needs gets no valid blocks and raises the device-check bit.  The
// split-K arrival counters of the sequence's rows are cleared here on every
// call, so a row left half-counted by an earlier call that failed (a wait
// that gave up) cannot make this call merge too early or never.
__global__ void decode_tiles_kernel(const int32_t* __restrict__ kv_lens, const int32_t* __restrict__ kv_indptr,
                                    int32_t batch, int32_t num_kv_heads, TileInfo* __restrict__ tiles,
                                    int32_t* __restrict__ row_cnt, uint32_t* err) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= batch) return;
  for (int g = 0; g < num_kv_heads; ++g) row_cnt[static_cast<int64_t>(t) * num_kv_heads + g] = 0;
  TileInfo ti;
  const int kl = kv_lens[t];
  const int base = kv_indptr[t], next = kv_indptr[t + 1];
  ti.seq = t;
  ti.q_begin = t;
  ti.rows = 1;
  ti.kv_len = kl;
  ti.pos0 = kl - 1;
  ti.nvp = kl >= 1 ? (kl + 127) / 128 : 0;
  ti.page_base = base;
  ti.pad = 0;
  if (kl < 1 || next - base < ti.nvp) {
    atomicOr(err, kErrDeviceCheck);
    ti.nvp = 0;
  }
  tiles[t] = ti;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" msa_status msa_sparse_decode_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                                const int32_t* kv_lens, const int32_t* kv_indptr,
                                                const int32_t* kv_indices, const int32_t* kv_block_indexes,
                                                const float* k_scale, const float* v_scale, int32_t batch,
                                                int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                                                int32_t topk, int64_t num_pages, void* out, float* lse,
                                                uint32_t* err_word, msa_stream_t stream) {
  const char* fn = "msa_sparse_decode_noalloc";
  if (!q || !k_pages || !v_pages || !kv_lens || !kv_indptr || !kv_indices || !kv_block_indexes || !k_scale ||
      !v_scale || !out)
    return set_error(MSA_ERR_INVALID_ARG, "%s: NULL argument", fn);
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_pages) | reinterpret_cast<uintptr_t>(v_pages) |
       reinterpret_cast<uintptr_t>(out)) & 15u)
    return set_error(MSA_ERR_INVALID_ARG, "%s: q, k_pages, v_pages, out must be 16-byte aligned", fn);
  if (batch < 1 || batch > kStaticMaxBatch)
    return set_error(MSA_ERR_INVALID_ARG, "%s: batch %d outside [1, %d]", fn, batch, kStaticMaxBatch);
  if (static_cast<int64_t>(batch) * num_kv_heads > kStaticMaxRows)
    return set_error(MSA_ERR_INVALID_ARG, "%s: batch * num_kv_heads above %d", fn, kStaticMaxRows);
  if (num_qo_heads < 1 || num_kv_heads < 1 || num_qo_heads % num_kv_heads != 0)
    return set_error(MSA_ERR_INVALID_ARG, "%s: bad head counts", fn);
  if (head_dim != kD) return set_error(MSA_ERR_UNSUPPORTED, "%s: head_dim must be 128", fn);
  const int G = num_qo_heads / num_kv_heads;
  if (G > 16) return set_error(MSA_ERR_UNSUPPORTED, "%s: at most 16 query heads per KV head", fn);
  if (topk < 1 || topk > 1024) return set_error(MSA_ERR_INVALID_ARG, "%s: topk outside [1, 1024]", fn);
  if (num_pages < 1 || num_pages > (int64_t(1) << 24)) return set_error(MSA_ERR_INVALID_ARG, "%s: num_pages", fn);
  const size_t n_units = static_cast<size_t>(batch) * num_kv_heads * topk;
  const size_t part_bytes = n_units * G * (kD + 2) * sizeof(float);
  if (n_units > size_t(1) << 30 || part_bytes > kStaticScratchBytes - kStaticPartOff)
    return set_error(MSA_ERR_INVALID_ARG,
                     "%s: batch*num_kv_heads*topk*(num_qo_heads/num_kv_heads) = %zu exceeds the static scratch "
                     "limit of %zu (24 MiB at head_dim 128)",
                     fn, n_units * G, (kStaticScratchBytes - kStaticPartOff) / ((kD + 2) * sizeof(float)));

  StaticDevice sd;
  msa_status s = static_scratch(&sd);
  if (s != MSA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  TileInfo* tiles = reinterpret_cast<TileInfo*>(sd.base);
  uint32_t* err = err_word ? err_word : reinterpret_cast<uint32_t*>(sd.base + kStaticErrOff);
  float* part_o = reinterpret_cast<float*>(sd.base + kStaticPartOff);
  float* part_ml = part_o + n_units * G * kD;
  // per-row arrival counters: cleared for this call's rows by the tile-table
  // kernel, which runs first on the same stream
  int32_t* row_cnt = reinterpret_cast<int32_t*>(sd.base + kStaticCntOff);
  auto* o_ptr = static_cast<__nv_bfloat16*>(out);

  CUtensorMap km, vm;
  const uint64_t dims[2] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(num_pages) * num_kv_heads * 128};
  const uint64_t str[1] = {static_cast<uint64_t>(kD)};
  const uint32_t box[2] = {static_cast<uint32_t>(kD), 128};
  if (!encode_tensor_map(&km, 2, k_pages, dims, str, box, 0, 128) ||
      !encode_tensor_map(&vm, 2, v_pages, dims, str, box, 0, 128))
    return set_error(MSA_ERR_CUDA, "%s: tensor map encoding failed", fn);

  decode_tiles_kernel<<<(batch + 127) / 128, 128, 0, st>>>(kv_lens, kv_indptr, batch, num_kv_heads, tiles, row_cnt,
                                                           err);
  s = cuda_check(cudaGetLastError(), "msa_sparse_decode_noalloc: tile table launch");
  if (s != MSA_OK) return s;
  const int nu = static_cast<int>(n_units);
  const int grid = decode_grid_rows(batch * num_kv_heads, topk, sd.num_sms, G);
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kD));
  const auto* qq = static_cast<const __nv_bfloat16*>(q);
  if (G <= 8) {
    const int smem = DecodeSmem<1>::kBytes + 1024;
    cudaFuncSetAttribute(decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    decode_kernel<1><<<grid, kDThreads, smem, st>>>(km, vm, qq, tiles, kv_block_indexes, kv_indices, num_pages,
                                                     k_scale, v_scale, part_o, part_ml, row_cnt, o_ptr, lse, nu,
                                                     num_qo_heads, num_kv_heads, 1, topk, scale_log2, err);
  } else {
    const int smem = DecodeSmem<2>::kBytes + 1024;
    cudaFuncSetAttribute(decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    decode_kernel<2><<<grid, kDThreads, smem, st>>>(km, vm, qq, tiles, kv_block_indexes, kv_indices, num_pages,
                                                     k_scale, v_scale, part_o, part_ml, row_cnt, o_ptr, lse, nu,
                                                     num_qo_heads, num_kv_heads, 1, topk, scale_log2, err);
  }
  return cuda_check(cudaGetLastError(), "msa_sparse_decode_noalloc: decode launch");
}
