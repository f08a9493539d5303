// Training extension, key side: dK, dV and the proxy-key gradient dpk of
// block-sparse GQA attention with the KL-coupled proxy (Flash-MSA article,
// backward-pass paragraph), on the tcgen05 tensor cores.
//
// One CTA per (page-table entry e, KV head g).  The lowest entry that names
// a physical page owns it: its CTA walks every selection of that page by a
// proxy head of KV head g (a group has Hp/Hkv proxy heads, each with its own
// blocks), by this entry or any other that names the same page (the inverse
// index, sorted so sums are deterministic), 64 query rows at a time, and the
// CTAs of the other entries return at once.  Per selection by proxy head p,
// for each of the G = Hq/Hp query heads that use p's blocks:
//   S^T  = K . Q_h^T            dP^T = V . dO_h^T       (M = keys, N = rows)
//   P^T  = exp2(S^T sl2 - lse2)  dS^T = P^T * (dP^T - D)  (masked: causal, ragged)
//   dV  += P^T . dO_h           dK  += dS^T . Q_h       (P^T, dS^T from TMEM)
//   dpk += P^T . pq
// and once per 64 rows, before the heads, for the proxy distribution over
// the same keys (in the dP^T columns):
//   Sp^T = pk . pq^T,  Pp^T = exp2(Sp^T zsl2 - lsep),  dpk += (-G Pp^T) . pq
// so that at the end dpk * (-w / (G sqrt(dp))) = w/sqrt(dp) (Pp - mean_h P_h)^T pq,
// this KV head's share of the KL gradient with respect to the proxy keys.
//
// Tensor memory (512 columns): S^T 64 | dP^T 64 | dV 128 | dpk 64 | dK 128 | K 64.
// K is copied into tensor memory once, so S^T = K . Q^T reads only Q from
// shared memory.  The softmax warps overwrite S^T (or Sp^T) and dP^T in
// place with bf16 pairs, handing P^T over before dS^T.  The MMA stream is
// pipelined across heads: S^T of head h+1 goes out as soon as dV and dpk of
// head h have taken P^T out of the S^T columns, dP^T of h+1 right after dK of
// h (after the last head, the next 64 rows' Sp^T), so the softmax of one
// head overlaps the products of the other; a half's first S^T goes out
// before its proxy term, while the proxy softmax runs.
// Each warpgroup owns 32 of the 64 rows, and each writes its packed pairs
// into the first half of its own 32 columns, so a k-step of 16 rows of an
// A operand in TMEM starts at column (kk / 2) * 32 + (kk % 2) * 8.
// dV and dpk sit side by side in tensor memory and share their A operand
// P^T, and each stage holds pq right after dO's two chunks, so one N = 192
// product P^T . [dO | pq] adds to both (an N = 64 product takes as long as
// an N = 128 one).
// Roles: warps 0-7 softmax (warp w reads TMEM lanes 32 (w % 4) ...), warp 8
// TMA producer (K, V, pk once; then a ring of Q/dO/pq halves, with their
// per-row lse2 / D / lsep staged by the same warp), warp 9 MMA.
#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kD = 128;
constexpr int kDP = 64;
constexpr int kQStages = 3;
constexpr int kSoftWarps = 8;
constexpr int kThreads = 32 * (kSoftWarps + 2);
constexpr int kMaxList = kBwdSmemList;
constexpr float kLog2e = 1.4426950408889634f;

constexpr uint32_t kColS = 0, kColDP = 64, kColDV = 128, kColDPK = 256, kColDK = 320, kColK = 448;

struct DkvSmem {
  static constexpr int kKOff = 0;                               // K block: 2 x [128 keys][128 B]
  static constexpr int kVOff = kKOff + 32768;                   // V block
  static constexpr int kPkOff = kVOff + 32768;                  // pk block: [128 keys][128 B]
  // ring: Q half 2 x [64][128 B] | dO half 2 x [64][128 B] | pq half [64][128 B]:
  // dO's two chunks and pq sit 8 KB apart, one rows-major operand of N = 192
  static constexpr int kQdOff = kPkOff + 16384;
  static constexpr int kQdBytes = 40960;
  static constexpr int kRowOff = kQdOff + kQStages * kQdBytes;  // stage s: lse2[64], D[64], lsep[64]
  static constexpr int kListOff = kRowOff + kQStages * 192 * 4;
  static constexpr int kBarOff = kListOff + kMaxList * 4;
  static constexpr int kFlagOff = kBarOff + 8 * 26;  // the dpk reduction's "last" flag
  static constexpr int kBytes = kFlagOff + 16;
};

__device__ __forceinline__ uint32_t ts_col(uint32_t base, int kk) {
  return base + static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8);
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap do_map,
                      const __grid_constant__ CUtensorMap pq_map, const __grid_constant__ CUtensorMap k_map,
                      const __grid_constant__ CUtensorMap v_map, const __grid_constant__ CUtensorMap pk_map,
                      const __grid_constant__ CUtensorMap dk_map, const __grid_constant__ CUtensorMap dv_map,
                      const TileInfo* __restrict__ tiles, const int32_t* __restrict__ idx,
                      const int32_t* __restrict__ owner, const int32_t* __restrict__ inv_off,
                      const int32_t* __restrict__ inv_cnt, int32_t* __restrict__ inv_list, int32_t topk,
                      const int32_t* __restrict__ kv_indices, int64_t num_pages, const float* __restrict__ lse2t,
                      const float* __restrict__ dsumt, const float* __restrict__ lsept, float* __restrict__ dk,
                      float* __restrict__ dv, float* __restrict__ dpk, float* __restrict__ dpk_part,
                      int32_t* __restrict__ dpk_cnt, int32_t hq, int32_t hkv, int32_t hsel,
                      int32_t total_q, int32_t d, int32_t dp, float kl_weight, uint32_t* err) {
  pdl_wait();  // launched with programmatic dependent launch: the previous kernel's writes first
  using L = DkvSmem;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int e = blockIdx.x / hkv, g = blockIdx.x % hkv;
  const int G = hq / hsel;  // query heads per proxy head
  int64_t page = kv_indices[e];
  const bool page_ok = page >= 0 && page < num_pages;
  if (page_ok && owner[page] != e) return;  // another entry's CTA owns this page
  if (!page_ok) page = 0;
  const int lb = inv_off[e * hkv + g], n = inv_cnt[e * hkv + g];
  const int64_t kv_off = (page * hkv + g) * 128 * d;

  // dpk of the page: each of its hkv CTAs leaves a partial, and the last of
  // them to count itself adds the partials in KV-head order (the same sum on
  // every run).  Threads [0, nthr) of the CTA take part.
  float* const part_e = dpk_part + (static_cast<int64_t>(e) * hkv + g) * 128 * kDP;
  auto finish_dpk = [&](int tid, int nthr, int bar_id) {
    __threadfence();
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(nthr) : "memory");
    int32_t* const flag = reinterpret_cast<int32_t*>(smem + DkvSmem::kFlagOff);
    if (tid == 0) {
      int32_t prev;
      asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(dpk_cnt + e) : "memory");
      *flag = prev == hkv - 1;
    }
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(nthr) : "memory");
    if (!*flag) return;
    // partials keep 64 columns a row; dpk rows have dp (columns [dp, 64) are
    // padding at dp = 32)
    float4* dst = reinterpret_cast<float4*>(dpk + page * 128 * dp);
    const float4* src0 = reinterpret_cast<const float4*>(dpk_part + static_cast<int64_t>(e) * hkv * 128 * kDP);
    // each thread keeps up to eight outputs (2048 float4s at most over 256 or
    // more threads) and sums the KV heads' partials in head order, one load
    // per output in flight for each head
    const int q4 = dp / 4;  // float4s of a dpk row
    constexpr int kPer = 8;
    float4 acc[kPer];
    int src_i[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = tid + k * nthr;
      src_i[k] = i < 128 * q4 ? (i / q4) * (kDP / 4) + i % q4 : -1;
    }
    for (int gg = 0; gg < hkv; ++gg) {
      const float4* src = src0 + static_cast<int64_t>(gg) * 128 * kDP / 4;
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        if (src_i[k] < 0) continue;
        const float4 v = __ldcg(src + src_i[k]);
        if (gg == 0) {
          acc[k] = v;
        } else {
          acc[k].x += v.x;
          acc[k].y += v.y;
          acc[k].z += v.z;
          acc[k].w += v.w;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (src_i[k] >= 0) dst[tid + k * nthr] = acc[k];
  };

  if (n == 0) {  // never cached: dK = dV = 0 and a zero dpk partial
    if (!page_ok) return;
    float4* a = reinterpret_cast<float4*>(dk + kv_off);
    float4* b = reinterpret_cast<float4*>(dv + kv_off);
    float4* c = reinterpret_cast<float4*>(part_e);
    for (int i = threadIdx.x; i < 128 * d / 4; i += blockDim.x) {
      a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      b[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int i = threadIdx.x; i < 128 * kDP / 4; i += blockDim.x) c[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    finish_dpk(threadIdx.x, kThreads, 2);
    return;
  }

  uint8_t* k_s = smem + L::kKOff;
  uint8_t* v_s = smem + L::kVOff;
  uint8_t* pk_s = smem + L::kPkOff;
  uint8_t* qd_s = smem + L::kQdOff;
  float* row_s = reinterpret_cast<float*>(smem + L::kRowOff);
  int32_t* list = reinterpret_cast<int32_t*>(smem + L::kListOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* kv_full = bars;
  uint64_t* init_done = bars + 1;  // accumulators zeroed, K in tensor memory
  uint64_t* qd_full = bars + 2;                 // [kQStages]
  uint64_t* qd_empty = qd_full + kQStages;      // [kQStages]
  uint64_t* sp_full = qd_empty + kQStages;
  uint64_t* pp_full = sp_full + 1;
  uint64_t* s_full = pp_full + 1;    // S^T computed
  uint64_t* dp_full = s_full + 1;    // dP^T computed
  uint64_t* p_full = dp_full + 1;    // P^T written (bf16, in place of S^T)
  uint64_t* ds_full = p_full + 1;    // dS^T written (bf16, in place of dP^T)
  uint64_t* done = ds_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    prefetch_tmap(&q_map);
    prefetch_tmap(&do_map);
    prefetch_tmap(&pq_map);
    prefetch_tmap(&k_map);
    prefetch_tmap(&v_map);
    prefetch_tmap(&pk_map);
    mbar_init(kv_full, 1);
    mbar_init(init_done, kSoftWarps);
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(qd_full + s, 2);  // expect_tx arrival + the staged lse2 / D
      mbar_init(qd_empty + s, 1);
    }
    mbar_init(sp_full, 1);
    mbar_init(pp_full, kSoftWarps);
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_full, kSoftWarps);
    mbar_init(ds_full, kSoftWarps);
    mbar_init(done, 1);
    fence_mbar_init();
  }
  // the selection list (flat indexes (t * hsel + p) * topk + slot), sorted so
  // that every run sums in the same order: in registers (up to 32 entries),
  // in shared memory (up to kMaxList) or in place in the inverse index
  const bool sorted = n <= kMaxList;
  if (n <= 32) {  // one warp, in registers (bitonic network over lanes)
    if (warp == 0) {
      int v = lane < n ? inv_list[lb + lane] : 0x7FFFFFFF;
#pragma unroll
      for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          const int o = __shfl_xor_sync(0xFFFFFFFFu, v, stride);
          const bool up = (lane & size) == 0, lower = (lane & stride) == 0;
          v = lower == up ? min(v, o) : max(v, o);  // the lower lane of an ascending pair keeps the smaller
        }
      if (lane < n) list[lane] = v;
    }
  } else if (sorted) {
    int pow2 = 1;
    while (pow2 < n) pow2 <<= 1;
    for (int i = threadIdx.x; i < pow2; i += blockDim.x) list[i] = i < n ? inv_list[lb + i] : 0x7FFFFFFF;
    __syncthreads();
    for (int size = 2; size <= pow2; size <<= 1)
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = threadIdx.x; i < pow2; i += blockDim.x) {
          const int o = i ^ stride;
          if (o > i) {
            const bool up = (i & size) == 0;
            const int a = list[i], b = list[o];
            if ((a > b) == up) {
              list[i] = b;
              list[o] = a;
            }
          }
        }
        __syncthreads();
      }
  } else {
    // a list too long for shared memory: sorted in place in the inverse
    // index, whose capacity for it is the next power of two (the scan gives
    // it that), padded with the largest key; rare, and off the common path
    int pow2 = 1;
    while (pow2 < n) pow2 <<= 1;
    int32_t* gl = inv_list + lb;
    for (int i = n + threadIdx.x; i < pow2; i += blockDim.x) gl[i] = 0x7FFFFFFF;
    __syncthreads();
    for (int size = 2; size <= pow2; size <<= 1)
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = threadIdx.x; i < pow2; i += blockDim.x) {
          const int o = i ^ stride;
          if (o > i) {
            const bool up = (i & size) == 0;
            const int a = gl[i], b = gl[o];
            if ((a > b) == up) {
              gl[i] = b;
              gl[o] = a;
            }
          }
        }
        __syncthreads();
      }
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto sel_at = [&](int it) { return sorted ? list[it] : inv_list[lb + it]; };
  const int sel_per_tile = hsel * topk;

  if (warp == 8) {
    // ---------------------------------------------------------- producer
    bool ok = true;
    if (lane == 0) {
      mbar_expect_tx(kv_full, 2 * 32768 + 16384);
      const int row = static_cast<int>((page * hkv + g) * 128);
      for (int c = 0; c < 2; ++c) {
        tma_load_2d(k_s + c * 16384, &k_map, kv_full, c * 64, row);
        tma_load_2d(v_s + c * 16384, &v_map, kv_full, c * 64, row);
      }
      tma_load_2d(pk_s, &pk_map, kv_full, 0, static_cast<int>(page * 128));
    }
    int qi = 0;
    for (int it = 0; ok && it < n; ++it) {
      const int sel = sel_at(it);
      const TileInfo tl = tiles[sel / sel_per_tile];
      const int pp = (sel / topk) % hsel;  // the selecting proxy head
      const int halves = tl.rows > 64 ? 2 : 1;
      for (int hf = 0; ok && hf < halves; ++hf) {
        const int r0 = tl.q_begin + hf * 64;
        for (int hh = 0; hh < G; ++hh, ++qi) {
          const int h = pp * G + hh;
          const int s = qi % kQStages;
          if (!(ok = mbar_wait(qd_empty + s, ((qi / kQStages) & 1) ^ 1, err))) break;
          uint8_t* st = qd_s + s * L::kQdBytes;
          if (lane == 0) {
            mbar_expect_tx(qd_full + s, L::kQdBytes);
            for (int c = 0; c < 2; ++c) {
              tma_load_3d(st + c * 8192, &q_map, qd_full + s, c * 64, h, r0);
              tma_load_3d(st + 16384 + c * 8192, &do_map, qd_full + s, c * 64, h, r0);
            }
            tma_load_3d(st + 32768, &pq_map, qd_full + s, 0, pp, r0);
          }
          for (int rr = lane; rr < 64; rr += 32) {
            const int r = hf * 64 + rr;
            const bool rok = r < tl.rows;
            const int64_t ei = static_cast<int64_t>(h) * total_q + tl.q_begin + r;
            row_s[s * 192 + rr] = rok ? -lse2t[ei] : 0.f;  // negated: the softmax adds them
            row_s[s * 192 + 64 + rr] = rok ? -dsumt[ei] : 0.f;
            row_s[s * 192 + 128 + rr] = rok ? -lsept[static_cast<int64_t>(pp) * total_q + tl.q_begin + r] : 0.f;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(qd_full + s);
        }
      }
    }
  } else if (warp == 9) {
    // --------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 64, false, false);   // S^T, dP^T, Sp^T
      constexpr uint32_t id_d = idesc_bf16_f32(128, 128, false, true);   // dV, dK (B rows-major)
      constexpr uint32_t id_p = idesc_bf16_f32(128, 64, false, true);    // dpk (proxy term)
      constexpr uint32_t id_vp = idesc_bf16_f32(128, 192, false, true);  // [dV | dpk] += P^T [dO | pq]
      // descriptors precomputed (one add per MMA): the issuing thread runs
      // only a step ahead of the tensor pipe
      constexpr uint64_t kQdDesc = L::kQdBytes >> 4;
      const uint64_t v_km = smem_desc(smem_u32(v_s), 16, 1024, kSwizzle128);
      const uint64_t pk_km = smem_desc(smem_u32(pk_s), 16, 1024, kSwizzle128);
      const uint64_t q_km = smem_desc(smem_u32(qd_s), 16, 1024, kSwizzle128);         // Q half (S^T = K Q^T)
      const uint64_t do_km = smem_desc(smem_u32(qd_s) + 16384, 16, 1024, kSwizzle128); // dO half (dP^T = V dO^T)
      const uint64_t q_mn = smem_desc(smem_u32(qd_s), 8192, 1024, kSwizzle128);       // Q as rows-major B (dK)
      const uint64_t do_mn = smem_desc(smem_u32(qd_s) + 16384, 8192, 1024, kSwizzle128);
      const uint64_t pq_km = smem_desc(smem_u32(qd_s) + 32768, 16, 1024, kSwizzle128);
      const uint64_t pq_mn = smem_desc(smem_u32(qd_s) + 32768, 8192, 1024, kSwizzle128);
      bool ok = mbar_wait(kv_full, 0, err) && mbar_wait(init_done, 0, err);
      tc_fence_after();
      // Sp^T = pk . pq^T of the half whose first head sits in stage qa, in
      // the dP^T columns (so that the half's first S^T can go out while the
      // proxy softmax runs)
      auto sp = [&](int qa) -> bool {
        const uint64_t po = static_cast<uint64_t>(qa % kQStages) * kQdDesc;
        if (!mbar_wait(qd_full + qa % kQStages, (qa / kQStages) & 1, err)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kDP / 16; ++kk) mma_ss(tmem + kColDP, pk_km + kk * 2, pq_km + po + kk * 2, id_s, kk > 0);
        mma_commit(sp_full);
        return true;
      };
      int qi = 0, pi = 0;
      bool sp_issued = false;  // the current half's Sp^T went out with the previous half's last head
      for (int it = 0; ok && it < n; ++it) {
        const TileInfo tl = tiles[sel_at(it) / sel_per_tile];
        const int halves = tl.rows > 64 ? 2 : 1;
        for (int hf = 0; ok && hf < halves; ++hf, ++pi) {
          const uint64_t po = static_cast<uint64_t>(qi % kQStages) * kQdDesc;  // the half's pq: its first head's stage
          const bool more_halves = hf + 1 < halves || it + 1 < n;
          if (!sp_issued && !(ok = sp(qi))) break;
          sp_issued = false;
          auto dpt = [&](uint64_t so) {  // dP^T = V . dO^T
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_ss(tmem + kColDP, v_km + (((kk / 4) * 16384 + (kk % 4) * 32) >> 4),
                     do_km + so + (((kk / 4) * 8192 + (kk % 4) * 32) >> 4), id_s, kk > 0);
            mma_commit(dp_full);
          };
          auto st = [&](uint64_t so) {  // S^T = K . Q^T (K from tensor memory)
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_ts(tmem + kColS, tmem + kColK + kk * 8, q_km + so + (((kk / 4) * 8192 + (kk % 4) * 32) >> 4), id_s,
                     kk > 0);
            mma_commit(s_full);
          };
          // head 0: S^T overlaps the proxy softmax, then the proxy term of
          // dpk reads -G Pp^T from the dP^T columns before dP^T overwrites them
          {
            const int s = qi % kQStages;
            const uint64_t so = static_cast<uint64_t>(s) * kQdDesc;
            if (!(ok = mbar_wait(qd_full + s, (qi / kQStages) & 1, err))) break;
            tc_fence_after();
            st(so);
            if (!(ok = mbar_wait(pp_full, pi & 1, err))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(tmem + kColDPK, ts_col(tmem + kColDP, kk), pq_mn + po + kk * 128, id_p, 1);
            dpt(so);
          }
          // heads pipelined: S^T of head h+1 is issued as soon as dV, dpk of
          // head h have taken P^T out of its columns, so the softmax of h+1
          // can start right after dS^T of h; dP^T of h+1 follows dK of h,
          // which takes dS^T out of the dP^T columns
          for (int hh = 0; ok && hh < G; ++hh, ++qi) {
            const int s = qi % kQStages;
            const uint64_t so = static_cast<uint64_t>(s) * kQdDesc;
            if (!(ok = mbar_wait(p_full, qi & 1, err))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // dV and dpk (side by side in TMEM) in one product
              mma_ts(tmem + kColDV, ts_col(tmem + kColS, kk), do_mn + so + kk * 128, id_vp, 1);
            const bool next = hh + 1 < G;
            const int s1 = (qi + 1) % kQStages;
            const uint64_t so1 = static_cast<uint64_t>(s1) * kQdDesc;
            if (next) {
              if (!(ok = mbar_wait(qd_full + s1, ((qi + 1) / kQStages) & 1, err))) break;
              tc_fence_after();
              st(so1);
            }
            if (!(ok = mbar_wait(ds_full, qi & 1, err))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(tmem + kColDK, ts_col(tmem + kColDP, kk), q_mn + so + kk * 128, id_d, 1);
            mma_commit(qd_empty + s);
            if (next) {
              dpt(so1);
            } else if (more_halves) {  // the next half's proxy scores, once dK has read dS^T out of their columns
              if (!(ok = sp(qi + 1))) break;
              sp_issued = true;
            }
          }
          if (!ok) break;
        }
      }
      mma_commit(done);
    }
    // dV and dK out of the softmax warps' staging boxes (see their epilogue)
    const bool staged = bar_sync_and(1, 32 * kSoftWarps + 32, true);
    if (staged && lane == 0) {
      const int nbox = d / 32;
      const int row0 = static_cast<int>((page * hkv + g) * 128);
      for (int b = 0; b < nbox; ++b) {
        tma_store_2d(&dv_map, smem + b * 16384, 32 * b, row0);
        tma_store_2d(&dk_map, smem + (nbox + b) * 16384, 32 * b, row0);
      }
      bulk_commit_group();
      bulk_wait_group_read0();  // the boxes are read before the CTA's memory goes
    }
  } else {
    // ----------------------------------------------------------- softmax
    const int wg = warp >> 2, quarter = warp & 3;
    const int key = quarter * 32 + lane;
    const int c0 = wg * 32;  // this warpgroup's rows within the 64-row half
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = kLog2e * rsqrtf(static_cast<float>(d));
    const float zsl2 = kLog2e * rsqrtf(static_cast<float>(dp));
    const float neg_g = -static_cast<float>(G);
    bool ok = mbar_wait(kv_full, 0, err);
    {  // dV, dpk, dK start at zero (columns 128..447, 160 per warpgroup); K row
       // `key`, d in [64 wg, 64 wg + 64), goes to tensor memory as bf16 pairs
      uint32_t z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
      for (int c = 0; c < 10; ++c) tmem_st16(lane_base + kColDV + wg * 160 + c * 16, z);
      const uint8_t* krow = k_s + wg * 16384 + key * 128;
      uint32_t kv[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 v = *reinterpret_cast<const uint4*>(krow + ((u ^ (key & 7)) << 4));
        kv[4 * u] = v.x;
        kv[4 * u + 1] = v.y;
        kv[4 * u + 2] = v.z;
        kv[4 * u + 3] = v.w;
      }
      tmem_st16(lane_base + kColK + 32 * wg, kv);
      tmem_st16(lane_base + kColK + 32 * wg + 16, kv + 16);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(init_done);
    }
    int qi = 0, pi = 0;
    for (int it = 0; ok && it < n; ++it) {
      const int sel = sel_at(it);
      const TileInfo tl = tiles[sel / sel_per_tile];
      const int j = idx[sel];  // the block's logical index in the selecting tile's sequence
      const int kpos = j * 128 + key;
      const int halves = tl.rows > 64 ? 2 : 1;
      for (int hf = 0; ok && hf < halves; ++hf, ++pi) {
        const int s0 = qi % kQStages;  // the half's first head's stage: its pq and proxy LSE
        const int rbase = hf * 64 + c0;  // tile row of column 0 of this warpgroup
        // every key of the block visible to all 32 rows: no per-element mask
        const bool need_mask = j * 128 + 127 > tl.pos0 + rbase || rbase + 32 > tl.rows;
        // proxy probabilities over this block's keys, scaled by -G
        if (!(ok = mbar_wait(qd_full + s0, (qi / kQStages) & 1, err))) break;
        if (!(ok = mbar_wait(sp_full, pi & 1, err))) break;
        tc_fence_after();
        {
          uint32_t sv[32], pk[16];
          tmem_ld32(lane_base + kColDP + c0, sv);
          tmem_wait_ld();
          const float2* nlp = reinterpret_cast<const float2*>(row_s + s0 * 192 + 128 + c0);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 nl = nlp[c >> 1];
            float x0, x1;
            ffma2v(x0, x1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), zsl2, zsl2, nl.x, nl.y);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if (need_mask) {
              const int r = rbase + c;
              if (!(r < tl.rows && kpos <= tl.pos0 + r)) p0 = 0.f;
              if (!(r + 1 < tl.rows && kpos <= tl.pos0 + r + 1)) p1 = 0.f;
            }
            pk[c >> 1] = pack_bf16x2(p0 * neg_g, p1 * neg_g);
          }
          tmem_st16(lane_base + kColDP + c0, pk);
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pp_full);
        for (int hh = 0; ok && hh < G; ++hh, ++qi) {
          const int s = qi % kQStages;
          if (!(ok = mbar_wait(qd_full + s, (qi / kQStages) & 1, err))) break;
          if (!(ok = mbar_wait(s_full, qi & 1, err))) break;
          tc_fence_after();
          // P^T first (dP^T may still be running), then dS^T
          uint32_t sv[32], pa[16], da[16];
          float pr[32];
          tmem_ld32(lane_base + kColS + c0, sv);
          tmem_wait_ld();
          const float2* nl2 = reinterpret_cast<const float2*>(row_s + s * 192 + c0);
          const float2* ndd = reinterpret_cast<const float2*>(row_s + s * 192 + 64 + c0);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 nl = nl2[c >> 1];
            float x0, x1;
            ffma2v(x0, x1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), sl2, sl2, nl.x, nl.y);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if (need_mask) {
              const int r = rbase + c;
              if (!(r < tl.rows && kpos <= tl.pos0 + r)) p0 = 0.f;
              if (!(r + 1 < tl.rows && kpos <= tl.pos0 + r + 1)) p1 = 0.f;
            }
            pr[c] = p0;
            pr[c + 1] = p1;
            pa[c >> 1] = pack_bf16x2(p0, p1);
          }
          tmem_st16(lane_base + kColS + c0, pa);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_full);
          if (!(ok = mbar_wait(dp_full, qi & 1, err))) break;
          tc_fence_after();
          tmem_ld32(lane_base + kColDP + c0, sv);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 nd = ndd[c >> 1];
            float t0, t1, d0, d1;
            fadd2v(t0, t1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), nd.x, nd.y);
            fmul2(d0, d1, t0, t1, pr[c], pr[c + 1]);
            da[c >> 1] = pack_bf16x2(d0, d1);
          }
          tmem_st16(lane_base + kColDP + c0, da);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(ds_full);
        }
      }
    }
    // epilogue: dV and dK rows are owned (plain stores); this KV head's dpk
    // partial goes to the scratch for the page's reduction
    if (ok) ok = mbar_wait(done, 0, err);
    tc_fence_after();
    ok = __all_sync(0xFFFFFFFFu, ok);  // the TMEM loads below are warp-collective
    // dV and dK of the CTA's 128 keys leave through shared memory (all of it
    // is free once every product is complete): 32-column fp32 TMA boxes in
    // the 128-byte swizzled layout, so the 16-byte writes here meet no bank
    // conflicts and the stores write whole lines
    const int nbox = d / 32;  // boxes per tensor
    if (ok && page_ok) {
      const float ks = rsqrtf(static_cast<float>(d));
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (wg * 64 >= d) break;  // at d = 64 the second warpgroup's columns are padding
        uint32_t a[32], b[32];
        tmem_ld32(lane_base + kColDV + wg * 64 + c * 32, a);
        tmem_ld32(lane_base + kColDK + wg * 64 + c * 32, b);
        tmem_wait_ld();
        uint8_t* bv = smem + (wg * 2 + c) * 16384 + key * 128;
        uint8_t* bk = smem + (nbox + wg * 2 + c) * 16384 + key * 128;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int off = (e ^ (key & 7)) << 4;
          *reinterpret_cast<float4*>(bv + off) =
              make_float4(__uint_as_float(a[4 * e]), __uint_as_float(a[4 * e + 1]), __uint_as_float(a[4 * e + 2]),
                          __uint_as_float(a[4 * e + 3]));
          *reinterpret_cast<float4*>(bk + off) =
              make_float4(__uint_as_float(b[4 * e]) * ks, __uint_as_float(b[4 * e + 1]) * ks,
                          __uint_as_float(b[4 * e + 2]) * ks, __uint_as_float(b[4 * e + 3]) * ks);
        }
      }
      fence_async_shared();  // the TMA stores read the boxes through the async proxy
    }
    // every softmax thread has staged its rows (or none of the CTA's stores
    // go out); the MMA warp, idle by now, issues the stores
    bar_sync_and(1, 32 * kSoftWarps + 32, ok && page_ok);
    // this KV head's dpk partial (full 32-byte sectors), then the page's sum
    if (ok && page_ok) {
      const float f_main = -kl_weight * rsqrtf(static_cast<float>(dp)) / static_cast<float>(G);
      uint32_t a[32];
      tmem_ld32(lane_base + kColDPK + wg * 32, a);
      tmem_wait_ld();
      float* pr = part_e + key * kDP + wg * 32;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        st_global_v8(pr + 8 * i, __uint_as_float(a[8 * i]) * f_main, __uint_as_float(a[8 * i + 1]) * f_main,
                     __uint_as_float(a[8 * i + 2]) * f_main, __uint_as_float(a[8 * i + 3]) * f_main,
                     __uint_as_float(a[8 * i + 4]) * f_main, __uint_as_float(a[8 * i + 5]) * f_main,
                     __uint_as_float(a[8 * i + 6]) * f_main, __uint_as_float(a[8 * i + 7]) * f_main);
    }
    if (page_ok) finish_dpk(threadIdx.x, 32 * kSoftWarps, 1);  // the softmax warps: threads 0-255
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

}  // namespace

msa_status launch_bwd_dkv_tc(const msa_plan_s* p, const void* q, const void* k_pages, const void* v_pages,
                             const void* dout, const void* pq, const void* pk_pages, const int32_t* kv_indices,
                             const int32_t* idx, const int32_t* owner, const int32_t* inv_off,
                             const int32_t* inv_cnt, int32_t* inv_list,
                             const float* lse2t, const float* dsumt, const float* lsept, float* dk, float* dv,
                             float* dpk, float* dpk_part, int32_t* dpk_cnt, float kl_weight, cudaStream_t st) {
  // tensors of their true width d (dp); the 64-column boxes read zeros past
  // the edge at d = 64 (dp = 32)
  CUtensorMap qm, dom, pqm, km, vm, pkm, dkm, dvm;
  const uint64_t d = static_cast<uint64_t>(p->d), dp = static_cast<uint64_t>(p->dp);
  const uint64_t qdims[3] = {d, static_cast<uint64_t>(p->hq), static_cast<uint64_t>(p->total_q)};
  const uint64_t qstr[2] = {d * 2, static_cast<uint64_t>(p->hq) * d * 2};
  const uint32_t qbox[3] = {64, 1, 64};
  const uint64_t pqdims[3] = {dp, static_cast<uint64_t>(p->hp), static_cast<uint64_t>(p->total_q)};
  const uint64_t pqstr[2] = {dp * 2, static_cast<uint64_t>(p->hp) * dp * 2};
  const uint64_t kdims[2] = {d, static_cast<uint64_t>(p->num_pages) * p->hkv * 128};
  const uint64_t kstr[1] = {d * 2};
  const uint32_t kbox[2] = {64, 128};
  const uint64_t pkdims[2] = {dp, static_cast<uint64_t>(p->num_pages) * 128};
  const uint64_t pkstr[1] = {dp * 2};
  // dK / dV pages, fp32 [num_pages * Hkv * 128][d]: 32-column boxes of 128 rows
  const uint64_t gstr[1] = {d * 4};
  const uint32_t gbox[2] = {32, 128};
  if (!encode_tensor_map(&qm, 3, q, qdims, qstr, qbox, 1, 128) ||
      !encode_tensor_map(&dom, 3, dout, qdims, qstr, qbox, 1, 128) ||
      !encode_tensor_map(&pqm, 3, pq, pqdims, pqstr, qbox, 1, 128) ||
      !encode_tensor_map(&km, 2, k_pages, kdims, kstr, kbox, 1, 128) ||
      !encode_tensor_map(&vm, 2, v_pages, kdims, kstr, kbox, 1, 128) ||
      !encode_tensor_map(&pkm, 2, pk_pages, pkdims, pkstr, kbox, 1, 128) ||
      !encode_tensor_map(&dkm, 2, dk, kdims, gstr, gbox, 2, 128) ||
      !encode_tensor_map(&dvm, 2, dv, kdims, gstr, gbox, 2, 128))
    return set_error(MSA_ERR_CUDA, "msa_sparse_attn_bwd: tensor map encoding failed");
  const int smem = DkvSmem::kBytes + 1024;
  cudaFuncSetAttribute(bwd_dkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
return cuda_check(launch_pdl(bwd_dkv_tc_kernel, dim3(p->n_page_entries * p->hkv), dim3(kThreads), smem, st, qm,
                               dom, pqm, km, vm, pkm, dkm, dvm, p->tiles_d, idx, owner, inv_off, inv_cnt, inv_list,
                               p->topk, kv_indices, p->num_pages, lse2t, dsumt, lsept, dk, dv, dpk, dpk_part, dpk_cnt,
                               p->hq, p->hkv, p->hp, static_cast<int32_t>(p->total_q), p->d, p->dp, kl_weight,
                               p->err_d),
                    "msa_sparse_attn_bwd: dkv launch");
}

}  // namespace msa
