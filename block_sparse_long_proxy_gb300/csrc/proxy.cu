// Stage 1: the proxy pass.  max_score[t, h, j] = max over rows i of tile t and
// keys k of block j with k visible to i of pq[i,h].pk[k]/sqrt(dp), -inf where
// nothing is visible ("MiniMax-AI/MSA" README, section "Usage": the dense
// proxy pass with num_kv_heads=1 and output_maxscore=True; Flash-MSA
// article, "three key differences": 128-token blocks chosen by max-pooling
// proxy scores).  Only the logits' block maxima leave the chip: no softmax,
// no P.V.
//
// Prefill kernel (tcgen05): one CTA per work unit = (tile, up to 8 proxy
// heads, a chunk of up to 32 KV blocks).  Warp 0 streams the tile's Q slices
// once and the paged proxy-K blocks through a 4-stage TMA ring; warp 1 issues
// one 128x256xdp MMA per (pair of consecutive blocks, head) -- N = 256 keeps
// the shared-memory operand traffic below the SMEM bandwidth, which a
// 128x128 MMA saturates -- into two 256-column TMEM accumulators; warps 2-9,
// as two groups each owning one accumulator, read it back (tcgen05.ld),
// apply the causal mask on diagonal blocks, and reduce each block to one
// value.  The proxy K
// block is read once per tile and shared by all heads (there is one proxy K
// head).
//
// Decode kernel (every qo_len == 1): one query row per sequence, so the pass
// is an HBM stream over the proxy-K pages.  Each warp owns a 3-stage TMA ring
// of pages and computes S^T = K_block . pq^T with mma.sync (M = 128 keys,
// N = 8 heads), then a max over keys.
#include "msa_internal.h"
#include "ptx.cuh"

#include <algorithm>

namespace msa {
namespace {

constexpr int kHeadsPerCta = 8;
constexpr int kChunk = 32;
constexpr int kStages = 4;
constexpr int kNBuf = 2;  // TMEM accumulators of 256 columns (one per epilogue group)
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);

// work unit of the prefill kernel
struct ProxyUnit {
  int32_t tile, h0, nh, j0, j1, fill_tail, pad0, pad1;
};

__device__ __forceinline__ int32_t f2ord(float f) {
  const int32_t b = __float_as_int(f);
  return b ^ ((b >> 31) & 0x7FFFFFFF);
}
__device__ __forceinline__ float ord2f(int32_t o) { return __int_as_float(o ^ ((o >> 31) & 0x7FFFFFFF)); }

// The top-k selection fused into the proxy pass (msa_proxy_topk; Flash-MSA
// article, kernel-design paragraph: the proxy pass keeps a streaming top-k
// of blocks instead of accumulating outputs).  Each
// chunk CTA of a (tile, group of 8 proxy heads) leaves, per head, its best
// topk-1 candidates among the blocks below the diagonal; the last of those
// CTAs to finish (a counter per row group, no waiting) merges them, adds the
// diagonal block and writes the ascending, -1 padded index row: the same
// selection as msa_topk_select on the same scores, since the best topk-1 of
// a union are among the best topk-1 of its parts.  A candidate is the 64-bit
// key (order_key(score) << 32) | ~j, so larger is better and ties go to the
// lower block; 0 is "none".
struct FusedTopk {
  int32_t* out;                // kv_block_indexes [n_tiles, hp, topk]; nullptr: max_score only
  int32_t* counters;           // [n_tiles * n_hgroups], zero between launches
  unsigned long long* cand;    // [((chunk_base[t] + c) * n_hgroups + hg) * 8 + h][32]
  const int32_t* chunk_base;   // [n_tiles]
  int32_t topk, n_hgroups;
};
constexpr int kFusedMaxTopk = 32;     // one lane per selected block
constexpr int kFusedMaxChunks = 32;   // max_blocks <= 1024

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
  const uint32_t hi = static_cast<uint32_t>(v >> 32);
  const uint32_t mhi = __reduce_max_sync(0xFFFFFFFFu, hi);
  const uint32_t mlo = __reduce_max_sync(0xFFFFFFFFu, hi == mhi ? static_cast<uint32_t>(v) : 0u);
  return (static_cast<unsigned long long>(mhi) << 32) | mlo;
}

template <int DP>
struct ProxySmem {
  static constexpr int kQBytes = 128 * DP * 2;   // one head's Q tile
  static constexpr int kKBytes = 128 * DP * 2;   // one proxy K block
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kHeadsPerCta * kQBytes;
  static constexpr int kPartOff = kKOff + kStages * kKBytes;
  static constexpr int kBarOff = kPartOff + kChunk * kHeadsPerCta * kEpiWarps * 4;
  static constexpr int kBytes = kBarOff + 8 * (1 + 2 * kStages + 2 * kNBuf + 1 + kHeadsPerCta) + 16;
};

// Persistent: CTA b takes the units cta_off[b] .. cta_off[b + 1] - 1, dealt at
// plan time longest first to the least-loaded CTA.  The
// K ring, the two TMEM accumulators and every barrier live across units; the
// ring counter and the accumulator counter run on across units (a unit's
// block count is padded to even with an empty stage, so that block pairs
// always sit in adjacent stages), and each head's Q tile is reloaded as soon
// as the previous unit's last MMA of that head has read it, so the next
// unit's loads overlap the current unit's last products and its epilogue
// (the block maxima and the fused selection).
template <int DP>
__global__ void __launch_bounds__(kThreads, 1)
    proxy_prefill_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                         const ProxyUnit* __restrict__ units, const int32_t* __restrict__ cta_off,
                         const TileInfo* __restrict__ tiles,
                         const int32_t* __restrict__ kv_indices, int64_t num_pages, float* __restrict__ max_score,
                         int32_t hp, int32_t max_blocks, float scale, FusedTopk fz, uint32_t* err) {
  pdl_wait();
  using L = ProxySmem<DP>;
  static_assert(kStages % 2 == 0, "block pairs occupy adjacent stages");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem + L::kQOff;
  uint8_t* k_s = smem + L::kKOff;
  int32_t* part = reinterpret_cast<int32_t*>(smem + L::kPartOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + kStages;
  uint64_t* t_full = k_empty + kStages;
  uint64_t* t_empty = t_full + kNBuf;
  uint64_t* drain = t_empty + kNBuf;
  uint64_t* q_empty = drain + 1;  // [kHeadsPerCta]: head h's Q tile read by the unit's last MMA of h
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_empty + kHeadsPerCta);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    prefetch_tmap(&q_map);
    prefetch_tmap(&k_map);
    mbar_init(q_full, 1);
    for (int h = 0; h < kHeadsPerCta; ++h) mbar_init(q_empty + h, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
    }
    for (int b = 0; b < kNBuf; ++b) {
      mbar_init(t_full + b, 1);
      mbar_init(t_empty + b, kEpiWarps / 2);  // the group of four warps reading accumulator b
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int kit = 0;  // ring position, across units
      bool ok = true;
      for (int k = 0, ui = cta_off[blockIdx.x]; ok && ui < cta_off[blockIdx.x + 1]; ++k, ++ui) {
        const ProxyUnit u = units[ui];
        const TileInfo tl = tiles[u.tile];
        const int nblk = u.j1 - u.j0;
        for (int h = 0; ok && h < u.nh; ++h) {
          if (k > 0 && !(ok = mbar_wait(q_empty + h, (k - 1) & 1, err))) break;
          // after head 0's slot is free the previous unit's q_full phase is
          // complete (its MMAs waited for it), so this arrival opens the next
          if (h == 0) mbar_expect_tx(q_full, u.nh * L::kQBytes);
          tma_load_3d(q_s + h * L::kQBytes, &q_map, q_full, 0, u.h0 + h, tl.q_begin);
        }
        if (!ok) break;
        for (int i = 0; i < nblk + (nblk & 1); ++i, ++kit) {
          const int s = kit % kStages;
          if (!(ok = mbar_wait(k_empty + s, ((kit / kStages) & 1) ^ 1, err))) break;
          if (i == nblk) {  // the empty stage that keeps the next unit's pairs aligned
            mbar_arrive(k_full + s);
            continue;
          }
          int64_t page = kv_indices[tl.page_base + u.j0 + i];
          if (page < 0 || page >= num_pages) {
            atomicOr(err, kErrDeviceCheck);
            page = 0;
          }
          mbar_expect_tx(k_full + s, L::kKBytes);
          tma_load_2d(k_s + s * L::kKBytes, &k_map, k_full + s, 0, static_cast<int>(page * 128));
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // one MMA covers two consecutive K blocks (N = 256): the pair sits in
      // adjacent ring stages, so its 256 rows form one K-major operand
      constexpr uint32_t id256 = idesc_bf16_f32(128, 256, false, false);
      constexpr uint32_t id128 = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t sw = DP == 64 ? kSwizzle128 : kSwizzle64;
      constexpr uint32_t sbo = DP == 64 ? 1024 : 512;
      int kit = 0, item = 0;
      bool ok = true;
      for (int k = 0, ui = cta_off[blockIdx.x]; ok && ui < cta_off[blockIdx.x + 1]; ++k, ++ui) {
        const ProxyUnit u = units[ui];
        const int nblk = u.j1 - u.j0;
        if (!(ok = mbar_wait(q_full, k & 1, err))) break;
        for (int i = 0; ok && i < nblk; i += 2, kit += 2) {
          const bool pair = i + 1 < nblk;
          const int s = kit % kStages;
          // the second stage of a pair (or the empty stage after an odd last block)
          if (!(ok = mbar_wait(k_full + s, (kit / kStages) & 1, err))) break;
          if (!(ok = mbar_wait(k_full + s + 1, ((kit + 1) / kStages) & 1, err))) break;
          tc_fence_after();
          const uint32_t kaddr = smem_u32(k_s + s * L::kKBytes);
          for (int h = 0; h < u.nh; ++h, ++item) {
            const int b = item & 1;  // accumulator b: 256 columns, read by epilogue group b
            if (!(ok = mbar_wait(t_empty + b, ((item >> 1) & 1) ^ 1, err))) break;
            tc_fence_after();
            const uint32_t qaddr = smem_u32(q_s + h * L::kQBytes);
#pragma unroll
            for (int kk = 0; kk < DP / 16; ++kk)
              mma_ss(tmem + b * 256, smem_desc(qaddr + kk * 32, 16, sbo, sw), smem_desc(kaddr + kk * 32, 16, sbo, sw),
                     pair ? id256 : id128, kk > 0);
            mma_commit(t_full + b);
            if (i + 2 >= nblk) mma_commit(q_empty + h);  // the unit's last MMA of head h
          }
          mma_commit(k_empty + s);
          mma_commit(k_empty + s + 1);
        }
        // heads the unit does not have: their Q slots are free as well (every
        // unit completes each q_empty once)
        for (int h = u.nh; ok && h < kHeadsPerCta; ++h) mma_commit(q_empty + h);
      }
      mma_commit(drain);
      mbar_wait(drain, 0, err);
    }
  } else {
    // epilogue: two groups of four warps, group b reading accumulator b
    // (items alternate between them, so one group's TMEM loads overlap the
    // other group's reduction); an item is one head over a pair of blocks;
    // warp w reads TMEM lanes 32*(w%4).. and each block's 128 columns
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int grp = ew >> 2;
    const int r = quarter * 32 + lane;
    const int et = threadIdx.x - 64;
    int item = 0;
    bool ok = true;
    for (int k = 0, ui = cta_off[blockIdx.x]; ui < cta_off[blockIdx.x + 1]; ++k, ++ui) {
      const ProxyUnit u = units[ui];
      const TileInfo tl = tiles[u.tile];
      const int nblk = u.j1 - u.j0;
      const bool row_ok = r < tl.rows;
      const int qpos = tl.pos0 + r;
      for (int i = 0; i < nblk; i += 2) {
        const int nb = i + 1 < nblk ? 2 : 1;
        for (int h = 0; h < u.nh; ++h, ++item) {
          if ((item & 1) != grp || !ok) continue;
          if (!(ok = mbar_wait(t_full + grp, (item >> 1) & 1, err))) continue;
          tc_fence_after();
          for (int bi = 0; bi < nb; ++bi) {
            uint32_t v[128];
            const uint32_t taddr = tmem + grp * 256 + bi * 128 + (static_cast<uint32_t>(quarter * 32) << 16);
            tmem_ld32(taddr, v);
            tmem_ld32(taddr + 32, v + 32);
            tmem_ld32(taddr + 64, v + 64);
            tmem_ld32(taddr + 96, v + 96);
            tmem_wait_ld();
            if (bi == nb - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(t_empty + grp);
            }
            const int j = u.j0 + i + bi;
            if ((j * 128 + 127 > tl.pos0) || (tl.rows < 128)) {  // diagonal / ragged: mask the future
              const int limit = row_ok ? qpos - j * 128 : -1;
#pragma unroll
              for (int c = 0; c < 128; ++c)
                if (c > limit) v[c] = __float_as_uint(-INFINITY);
            }
            float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; c += 8) {
              m0 = fmax3(m0, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
              m1 = fmax3(m1, __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
              m2 = fmax3(m2, __uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
              m3 = fmax3(m3, __uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
            }
            const float m = fmax3(fmaxf(m0, m1), m2, m3);
            const int32_t wm = __reduce_max_sync(0xFFFFFFFFu, f2ord(m));
            if (lane == 0) part[((i + bi) * kHeadsPerCta + h) * kEpiWarps + quarter] = wm;
          }
        }
      }
      ok = __all_sync(0xFFFFFFFFu, ok);  // warp-uniform: the barriers and selections below are collective
      // all epilogue warps: combine the eight partial maxima of each item
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
      if (ok) {
        for (int it = et; it < nblk * u.nh; it += 32 * kEpiWarps) {
          const int h = it / nblk, i = it % nblk;
          int32_t m = part[(i * kHeadsPerCta + h) * kEpiWarps];
#pragma unroll
          for (int w = 1; w < 4; ++w) m = max(m, part[(i * kHeadsPerCta + h) * kEpiWarps + w]);
          const float v = ord2f(m) * scale;
          if (max_score) max_score[(static_cast<int64_t>(u.tile) * hp + u.h0 + h) * max_blocks + u.j0 + i] = v;
          part[(i * kHeadsPerCta + h) * kEpiWarps + 4] = __float_as_int(v);  // the fused selection reads it
        }
      }
      if (fz.out) {
        // ---- fused top-k: this chunk's candidates, then the row group's merge
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
        const bool wok = ok;
        const int hg = u.h0 / kHeadsPerCta;
        const int n = tl.nvp < 1 ? 1 : (tl.nvp > max_blocks ? max_blocks : tl.nvp);
        const int need = fz.topk - 1;
        const bool all = fz.topk >= n;  // every valid block is selected
        const int n_chunks = (tl.nvp + kChunk - 1) / kChunk;
        auto slot = [&](int c, int h) -> int64_t {
          return ((static_cast<int64_t>(fz.chunk_base[u.tile] + c) * fz.n_hgroups + hg) * kHeadsPerCta + h) * 32;
        };
        if (wok && !all && ew < u.nh) {
          const int j = u.j0 + lane;
          unsigned long long ck = 0ull;
          if (lane < nblk && j < n - 1) {
            const uint32_t key = order_key(__int_as_float(part[(lane * kHeadsPerCta + ew) * kEpiWarps + 4]));
            if (key) ck = (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(j));
          }
          unsigned long long mine = 0ull;
          bool taken = false;
          for (int q = 0; q < need; ++q) {
            const unsigned long long m = warp_max_u64(taken ? 0ull : ck);
            if (m == 0ull) break;
            if (ck == m) taken = true;
            if (lane == q) mine = m;
          }
          if (lane < need) fz.cand[slot(u.j0 / kChunk, ew) + lane] = mine;
        }
        // the CTA barrier orders every thread's candidates before thread 0's
        // release; its acquire (in the last CTA) orders the merge's reads after
        // every chunk's release
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
        if (et == 0) {
          int32_t* ctr = fz.counters + static_cast<int64_t>(u.tile) * fz.n_hgroups + hg;
          int32_t prev;
          asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(ctr) : "memory");
          const bool last = prev == n_chunks - 1;
          if (last) *ctr = 0;  // every chunk of the row group has counted: ready for the next launch
          part[5] = last;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
        if (part[5] && wok && ew < u.nh) {
          int32_t* dst = fz.out + (static_cast<int64_t>(u.tile) * hp + u.h0 + ew) * fz.topk;
          if (all) {
            if (lane < fz.topk) dst[lane] = lane < n ? lane : -1;
          } else {
            // a k-way merge of the chunks' lists, each already best-first:
            // lane c holds chunk c's list and shifts it as its head is taken
            unsigned long long v[kFusedMaxTopk - 1];
#pragma unroll
            for (int rr = 0; rr < kFusedMaxTopk - 1; ++rr)
              v[rr] = (lane < n_chunks && rr < need) ? __ldcg(fz.cand + slot(lane, ew) + rr) : 0ull;
            uint32_t sel = 0xFFFFFFFFu;  // lane q: the q-th best block
            int found = 0;
            for (int q = 0; q < need; ++q) {
              const unsigned long long m = warp_max_u64(v[0]);
              if (m == 0ull) break;
              if (v[0] == m) {
#pragma unroll
                for (int rr = 0; rr < kFusedMaxTopk - 2; ++rr) v[rr] = v[rr + 1];
                v[kFusedMaxTopk - 2] = 0ull;
              }
              if (lane == q) sel = 0xFFFFFFFFu - static_cast<uint32_t>(m);
              ++found;
            }
            if (lane == found) sel = static_cast<uint32_t>(n - 1);  // the diagonal block
            // ascending: each selected block's rank among the selected ones
            int rank = 0;
            for (int l = 0; l < 32; ++l) rank += __shfl_sync(0xFFFFFFFFu, sel, l) < sel;
            if (sel != 0xFFFFFFFFu) dst[rank] = static_cast<int32_t>(sel);
            if (lane > found && lane < fz.topk) dst[lane] = -1;
          }
        }
      }
      if (u.fill_tail && max_score) {
        const int tail = max_blocks - tl.nvp;
        for (int it = et; it < tail * u.nh; it += 32 * kEpiWarps) {
          const int h = it / tail, j = tl.nvp + it % tail;
          max_score[(static_cast<int64_t>(u.tile) * hp + u.h0 + h) * max_blocks + j] = -INFINITY;
        }
      }
      // the next unit's partial maxima may overwrite this unit's
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ decode

// Warps x ring stages per warp, one CTA per SM: measured at 32 x 131072,
// dp = 64: 4 x 3 103 us, 6 x 2 97.8, 12 x 1 94.6, 10 x 1 90.4, 8 x 1 90.1.
constexpr int kDecWarps = 8;
constexpr int kDecStages = 1;

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Units are (sequence, block) pairs in order; unit_start[t] is the first unit
// of tile (sequence) t.  Warp w takes the contiguous unit range
// [U*w/W, U*(w+1)/W).  Unit metadata (sequence, block, page row) is computed
// lane-parallel 32 units at a time, one chunk ahead of the loads, so that
// the dependent global lookups stay off the per-unit path.
__device__ __forceinline__ int warp_range_start(int w, int U, int W) {
  const int q = U / W, r = U % W;
  return w * q + (w < r ? w : r);
}

template <int DP>
__global__ void __launch_bounds__(32 * kDecWarps)
    proxy_decode_kernel(const __grid_constant__ CUtensorMap k_map, const __nv_bfloat16* __restrict__ pq,
                        const TileInfo* __restrict__ tiles, const int32_t* __restrict__ unit_start, int32_t n_tiles,
                        const int32_t* __restrict__ kv_indices, int64_t num_pages, float* __restrict__ max_score,
                        int32_t hp, int32_t max_blocks, float scale, uint32_t* err) {
  pdl_wait();
  constexpr int kBlk = 128 * DP * 2;
  constexpr int kRowBytes = DP * 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + warp * kDecStages * kBlk;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDecWarps * kDecStages * kBlk) + warp * kDecStages;

  const int total_units = unit_start[n_tiles];
  // -inf past each sequence's valid blocks
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       e < static_cast<int64_t>(n_tiles) * hp * max_blocks; e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(e % max_blocks);
    const int t = static_cast<int>(e / (static_cast<int64_t>(hp) * max_blocks));
    if (j >= tiles[t].nvp) max_score[e] = -INFINITY;
  }

  if (lane == 0) {
    for (int s = 0; s < kDecStages; ++s) mbar_init(bars + s, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const int nw = gridDim.x * kDecWarps;
  const int gw = blockIdx.x * kDecWarps + warp;
  const int ub = warp_range_start(gw, total_units, nw), ue = warp_range_start(gw + 1, total_units, nw);
  const int n = ue - ub;

  // lane l: metadata of unit (chunk_base + l)
  auto meta = [&](int chunk_base, int& t, int& j, int& row) {
    const int unit = chunk_base + lane;
    t = 0;
    j = 0;
    row = 0;
    if (unit < ue) {
      int lo = 0, hi = n_tiles - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(unit_start + mid) <= unit) lo = mid; else hi = mid - 1;
      }
      t = lo;
      j = unit - __ldg(unit_start + lo);
      int64_t page = kv_indices[tiles[t].page_base + j];
      if (page < 0 || page >= num_pages) {
        atomicOr(err, kErrDeviceCheck);
        page = 0;
      }
      row = static_cast<int>(page * 128);
    }
  };
  int ct, cj, crow, nt_, nj, nrow;  // current chunk and next chunk metadata
  meta(ub, ct, cj, crow);
  meta(ub + 32, nt_, nj, nrow);
  auto row_of = [&](int i) {  // page row of the warp's i-th unit (i in this or the next chunk)
    const int c = i >> 5, cur = 0;
    (void)cur;
    const int r_cur = __shfl_sync(0xFFFFFFFFu, crow, i & 31);
    const int r_nxt = __shfl_sync(0xFFFFFFFFu, nrow, i & 31);
    return c == 0 ? r_cur : r_nxt;
  };
  int chunk = 0;  // index of the chunk held in (ct, cj, crow)
  auto issue = [&](int i) {  // load the warp's i-th unit into stage i % kDecStages
    if (i >= n) return;
    const int r = row_of(i - 32 * chunk);
    if (lane == 0) {
      uint64_t* bar = bars + (i % kDecStages);
      mbar_expect_tx(bar, kBlk);
      tma_load_2d(ring + (i % kDecStages) * kBlk, &k_map, bar, 0, r);
    }
  };
  for (int i = 0; i < kDecStages; ++i) issue(i);

  const int g = lane >> 2, t4 = lane & 3;
  for (int i = 0; i < n; ++i) {
    if (i - 32 * chunk == 32) {  // move to the next chunk of metadata
      ct = nt_;
      cj = nj;
      crow = nrow;
      ++chunk;
      meta(ub + 32 * (chunk + 1), nt_, nj, nrow);
    }
    const int t = __shfl_sync(0xFFFFFFFFu, ct, i & 31);
    const int j = __shfl_sync(0xFFFFFFFFu, cj, i & 31);
    const TileInfo tl = tiles[t];
    // B fragments: pq[row, head n = hb + g, dims] of eight heads from hb;
    // heads >= hp contribute zeros
    uint32_t bf[DP / 16][2];
    const __nv_bfloat16* qrow0 = pq + static_cast<int64_t>(tl.q_begin) * hp * DP;
    auto load_bf = [&](int hb) {
      const __nv_bfloat16* qrow = qrow0 + static_cast<int64_t>(hb + g) * DP;
#pragma unroll
      for (int kt = 0; kt < DP / 16; ++kt) {
        if (hb + g < hp) {
          bf[kt][0] = *reinterpret_cast<const uint32_t*>(qrow + kt * 16 + 2 * t4);
          bf[kt][1] = *reinterpret_cast<const uint32_t*>(qrow + kt * 16 + 8 + 2 * t4);
        } else {
          bf[kt][0] = bf[kt][1] = 0u;
        }
      }
    };
    load_bf(0);
    const int s = i % kDecStages;
    if (!mbar_wait(bars + s, (i / kDecStages) & 1, err)) break;
    const uint32_t base = smem_u32(ring + s * kBlk);
    const int nkeys = min(128, tl.kv_len - j * 128);  // keys past kv_len are not visible
    for (int hb = 0;;) {  // eight proxy heads per pass over the page (one pass when hp <= 8)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kt = 0; kt < DP / 16; ++kt) {
          const int row = mt * 16 + (lane & 15);
          const int chunk16 = kt * 2 + (lane >> 4);
          const int sw = DP == 64 ? (chunk16 ^ (row & 7)) : (chunk16 ^ ((row >> 1) & 3));
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4(base + row * kRowBytes + sw * 16, a0, a1, a2, a3);
          mma_16816(c, a0, a1, a2, a3, bf[kt][0], bf[kt][1]);
        }
        const int r0 = mt * 16 + g, r1 = r0 + 8;
        if (r0 < nkeys) { mx0 = fmaxf(mx0, c[0]); mx1 = fmaxf(mx1, c[1]); }
        if (r1 < nkeys) { mx0 = fmaxf(mx0, c[2]); mx1 = fmaxf(mx1, c[3]); }
      }
      const bool last = hb + 8 >= hp;
      if (last) {  // the stage is free once the last pass has read it
        __syncwarp();
        issue(i + kDecStages);
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, o));
      }
      if (lane < 4) {
        const int h0 = hb + 2 * lane, h1 = h0 + 1;
        float* dst = max_score + static_cast<int64_t>(t) * hp * max_blocks + j;
        if (h0 < hp) dst[static_cast<int64_t>(h0) * max_blocks] = mx0 * scale;
        if (h1 < hp) dst[static_cast<int64_t>(h1) * max_blocks] = mx1 * scale;
      }
      if (last) break;
      hb += 8;
      load_bf(hb);
    }
  }
}

// FP8 proxy K at decode: the same scan over e4m3 proxy K pages (64 bytes a
// row at dp = 64) with one fp32 scale for the shared proxy head, so the
// dominant decode read is halved.  logit = (pq . pk_code) * pk_scale / sqrt(dp)
// and, the scale being positive, the block max is taken on the codes' dot
// products and scaled once.  A row of a page is loaded by TMA with 64-byte
// swizzle; lane (g, t4) reads the 4 bytes at dims 16 kc + 4 t4 of keys g and
// g + 8 of an m-tile, which is one conflict-free 32-bit word per lane, and the
// pq fragments use the same dim order (the dot product is order-free).
constexpr int kDec8Warps = 24;  // warps per CTA, one CTA per SM (measured best of 4..24)
constexpr int kDec8Stages = 1;  // ring stages per warp: the parallelism is across warps

template <int W, int S>
__global__ void __launch_bounds__(32 * W)
    proxy_decode_fp8_kernel(const __grid_constant__ CUtensorMap k_map, const __nv_bfloat16* __restrict__ pq,
                            const float* __restrict__ pk_scale, const TileInfo* __restrict__ tiles,
                            const int32_t* __restrict__ unit_start, int32_t n_tiles,
                            const int32_t* __restrict__ kv_indices, int64_t num_pages, float* __restrict__ max_score,
                            int32_t hp, int32_t max_blocks, float scale, uint32_t* err) {
  pdl_wait();
  constexpr int DP = 64;
  constexpr int kBlk = 128 * DP;  // bytes of one e4m3 proxy K page
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + warp * S * kBlk;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + W * S * kBlk) + warp * S;
  const float out_scale = scale * pk_scale[0];

  const int total_units = unit_start[n_tiles];
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
  const int ub = warp_range_start(gw, total_units, nw), ue = warp_range_start(gw + 1, total_units, nw);
  const int n = ue - ub;

  auto meta = [&](int chunk_base, int& t, int& j, int& row) {
    const int unit = chunk_base + lane;
    t = 0;
    j = 0;
    row = 0;
    if (unit < ue) {
      int lo = 0, hi = n_tiles - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(unit_start + mid) <= unit) lo = mid; else hi = mid - 1;
      }
      t = lo;
      j = unit - __ldg(unit_start + lo);
      int64_t page = kv_indices[tiles[t].page_base + j];
      if (page < 0 || page >= num_pages) {
        atomicOr(err, kErrDeviceCheck);
        page = 0;
      }
      row = static_cast<int>(page * 128);
    }
  };
  int ct, cj, crow, nt_, nj, nrow;
  meta(ub, ct, cj, crow);
  meta(ub + 32, nt_, nj, nrow);
  int chunk = 0;
  auto issue = [&](int i) {
    if (i >= n) return;
    const int ii = i - 32 * chunk;
    const int r_cur = __shfl_sync(0xFFFFFFFFu, crow, ii & 31);
    const int r_nxt = __shfl_sync(0xFFFFFFFFu, nrow, ii & 31);
    const int r = (ii >> 5) == 0 ? r_cur : r_nxt;
    if (lane == 0) {
      uint64_t* bar = bars + (i % S);
      mbar_expect_tx(bar, kBlk);
      tma_load_2d(ring + (i % S) * kBlk, &k_map, bar, 0, r);
    }
  };
  for (int i = 0; i < S; ++i) issue(i);

  const int g = lane >> 2, t4 = lane & 3;
  for (int i = 0; i < n; ++i) {
    if (i - 32 * chunk == 32) {
      ct = nt_;
      cj = nj;
      crow = nrow;
      ++chunk;
      meta(ub + 32 * (chunk + 1), nt_, nj, nrow);
    }
    const int t = __shfl_sync(0xFFFFFFFFu, ct, i & 31);
    const int j = __shfl_sync(0xFFFFFFFFu, cj, i & 31);
    const TileInfo tl = tiles[t];
    // B fragments: pq[row, head g, dims 16 kc + 4 t4 .. +3] as f16 pairs
    uint32_t bf[DP / 16][2];
    const __nv_bfloat16* qrow = pq + (static_cast<int64_t>(tl.q_begin) * hp + g) * DP;
#pragma unroll
    for (int kc = 0; kc < DP / 16; ++kc) {
      if (g < hp) {
        const uint2 v = *reinterpret_cast<const uint2*>(qrow + kc * 16 + 4 * t4);
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
    const uint32_t base = smem_u32(ring + s * kBlk);
    const int nkeys = min(128, tl.kv_len - j * 128);
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      const int ra = mt * 16 + g, rb = ra + 8;
#pragma unroll
      for (int kc = 0; kc < DP / 16; ++kc) {
        const uint32_t wa = lds32(base + ra * 64 + ((kc ^ ((ra >> 1) & 3)) << 4) + 4 * t4);
        const uint32_t wb = lds32(base + rb * 64 + ((kc ^ ((rb >> 1) & 3)) << 4) + 4 * t4);
        mma_f16(c, e4m3x2_to_f16x2(wa), e4m3x2_to_f16x2(wb), e4m3x2_to_f16x2(wa >> 16), e4m3x2_to_f16x2(wb >> 16),
                bf[kc][0], bf[kc][1]);
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

// --------------------------------------------------------------- host side

void proxy_plan_tables(msa_plan_s* p, std::vector<int32_t>& aux) {
  // prefill work units, longest first
  std::vector<ProxyUnit> us;
  for (int t = 0; t < p->n_tiles; ++t) {
    const int nvp = p->tiles[t].nvp;
    for (int h0 = 0; h0 < p->hp; h0 += kHeadsPerCta)
      for (int j0 = 0; j0 < nvp; j0 += kChunk) {
        ProxyUnit u{};
        u.tile = t;
        u.h0 = h0;
        u.nh = std::min(kHeadsPerCta, p->hp - h0);
        u.j0 = j0;
        u.j1 = std::min(nvp, j0 + kChunk);
        u.fill_tail = (u.j1 == nvp) && (nvp < p->max_blocks);
        us.push_back(u);
      }
  }
  std::stable_sort(us.begin(), us.end(),
                   [](const ProxyUnit& a, const ProxyUnit& b) { return (a.j1 - a.j0) > (b.j1 - b.j0); });
  // the fused top-k's candidate slots: chunk c of tile t is slot chunk_base[t] + c
  p->proxy_chunk_base_off = static_cast<int64_t>(aux.size());
  int32_t chunks = 0;
  for (int t = 0; t < p->n_tiles; ++t) {
    aux.push_back(chunks);
    chunks += (p->tiles[t].nvp + kChunk - 1) / kChunk;
  }
  p->proxy_n_chunks = chunks;
  // persistent CTAs: units dealt longest first to the least-loaded CTA (a
  // unit costs its block-head products plus a fixed tail), each CTA's units
  // stored contiguously; proxy_cta_off[b] .. [b + 1] are CTA b's
  const int n_ctas = std::max(1, std::min(static_cast<int>(us.size()), p->num_sms));
  std::vector<std::vector<ProxyUnit>> per(n_ctas);
  std::vector<std::pair<int64_t, int>> heap;  // (load, cta), a min-heap
  for (int b = 0; b < n_ctas; ++b) heap.push_back({0, b});
  auto later = [](const std::pair<int64_t, int>& a, const std::pair<int64_t, int>& b) { return a > b; };
  for (const ProxyUnit& u : us) {
    std::pop_heap(heap.begin(), heap.end(), later);
    auto& top = heap.back();
    per[top.second].push_back(u);
    top.first += static_cast<int64_t>(u.j1 - u.j0) * u.nh + 8;
    std::push_heap(heap.begin(), heap.end(), later);
  }
  p->proxy_cta_off = static_cast<int64_t>(aux.size());
  p->proxy_n_ctas = n_ctas;
  int32_t off = 0;
  for (int b = 0; b < n_ctas; ++b) {
    aux.push_back(off);
    off += static_cast<int32_t>(per[b].size());
  }
  aux.push_back(off);
  p->proxy_units_off = static_cast<int64_t>(aux.size());
  p->n_proxy_units = static_cast<int32_t>(us.size());
  for (int b = 0; b < n_ctas; ++b) {
    const int32_t* raw = reinterpret_cast<const int32_t*>(per[b].data());
    aux.insert(aux.end(), raw, raw + per[b].size() * (sizeof(ProxyUnit) / 4));
  }
  // decode: first unit of each tile
  p->proxy_unit_start_off = static_cast<int64_t>(aux.size());
  int32_t acc = 0;
  for (int t = 0; t < p->n_tiles; ++t) {
    aux.push_back(acc);
    acc += p->tiles[t].nvp;
  }
  aux.push_back(acc);
}

static bool make_pk_map(CUtensorMap* m, const msa_plan_s* p, const void* pk_pages) {
  const uint64_t dims[2] = {static_cast<uint64_t>(p->dp), static_cast<uint64_t>(p->num_pages) * 128};
  const uint64_t strides[1] = {static_cast<uint64_t>(p->dp) * 2};
  const uint32_t box[2] = {static_cast<uint32_t>(p->dp), 128};
  return encode_tensor_map(m, 2, pk_pages, dims, strides, box, 1, p->dp * 2);
}

static msa_status proxy_prefill(const msa_plan_s* p, const void* pq, const void* pk_pages, const int32_t* kv_indices,
                                float* max_score, const FusedTopk& fz, cudaStream_t st) {
  CUtensorMap qm, km;
  const uint64_t qdims[3] = {static_cast<uint64_t>(p->dp), static_cast<uint64_t>(p->hp),
                             static_cast<uint64_t>(p->total_q)};
  const uint64_t qstr[2] = {static_cast<uint64_t>(p->dp) * 2, static_cast<uint64_t>(p->hp) * p->dp * 2};
  const uint32_t qbox[3] = {static_cast<uint32_t>(p->dp), 1, 128};
  if (!encode_tensor_map(&qm, 3, pq, qdims, qstr, qbox, 1, p->dp * 2) || !make_pk_map(&km, p, pk_pages))
    return set_error(MSA_ERR_CUDA, "msa_proxy_maxscore: tensor map encoding failed");
  const ProxyUnit* units = reinterpret_cast<const ProxyUnit*>(p->aux_d + p->proxy_units_off);
  const int32_t* cta_off = p->aux_d + p->proxy_cta_off;
  const float scale = 1.0f / sqrtf(static_cast<float>(p->dp));
  const int grid = p->proxy_n_ctas;  // persistent: one CTA per SM
  cudaError_t e;
  if (p->dp == 64) {
    const int smem = ProxySmem<64>::kBytes + 1024;
    cudaFuncSetAttribute(proxy_prefill_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    e = launch_pdl(proxy_prefill_kernel<64>, dim3(grid), dim3(kThreads), smem, st, qm, km, units, cta_off,
                   p->tiles_d, kv_indices, p->num_pages, max_score, p->hp, p->max_blocks, scale, fz, p->err_d);
  } else {
    const int smem = ProxySmem<32>::kBytes + 1024;
    cudaFuncSetAttribute(proxy_prefill_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    e = launch_pdl(proxy_prefill_kernel<32>, dim3(grid), dim3(kThreads), smem, st, qm, km, units, cta_off,
                   p->tiles_d, kv_indices, p->num_pages, max_score, p->hp, p->max_blocks, scale, fz, p->err_d);
  }
  return cuda_check(e, "msa_proxy_maxscore: prefill launch");
}

msa_status launch_proxy_prefill(const msa_plan_s* p, const void* pq, const void* pk_pages, const int32_t* kv_indices,
                                float* max_score, cudaStream_t st) {
  return proxy_prefill(p, pq, pk_pages, kv_indices, max_score, FusedTopk{}, st);
}

size_t fused_topk_counter_bytes(const msa_plan_s* p) {
  if (p->decode || p->topk > kFusedMaxTopk || p->max_blocks > kChunk * kFusedMaxChunks) return 0;
  const int64_t hg = (p->hp + kHeadsPerCta - 1) / kHeadsPerCta;
  return (sizeof(int32_t) * p->n_tiles * hg + 255) & ~size_t(255);
}

size_t fused_topk_scratch_bytes(const msa_plan_s* p) {
  const size_t c = fused_topk_counter_bytes(p);
  if (c == 0) return 0;
  const int64_t hg = (p->hp + kHeadsPerCta - 1) / kHeadsPerCta;
  return c + sizeof(unsigned long long) * static_cast<size_t>(p->proxy_n_chunks) * hg * kHeadsPerCta * 32;
}

msa_status launch_proxy_topk(const msa_plan_s* p, const void* pq, const void* pk_pages, const int32_t* kv_indices,
                             float* max_score, int32_t* kv_block_indexes, cudaStream_t st) {
  if (p->decode) return set_error(MSA_ERR_UNSUPPORTED, "msa_proxy_topk: prefill plans only");
  if (!p->fused_topk_d)
    return set_error(MSA_ERR_UNSUPPORTED, "msa_proxy_topk: needs topk <= %d and at most %d blocks per sequence",
                     kFusedMaxTopk, kChunk * kFusedMaxChunks);
  FusedTopk fz{};
  fz.out = kv_block_indexes;
  fz.counters = static_cast<int32_t*>(p->fused_topk_d);
  fz.cand = reinterpret_cast<unsigned long long*>(static_cast<char*>(p->fused_topk_d) + fused_topk_counter_bytes(p));
  fz.chunk_base = p->aux_d + p->proxy_chunk_base_off;
  fz.topk = p->topk;
  fz.n_hgroups = (p->hp + kHeadsPerCta - 1) / kHeadsPerCta;
  return proxy_prefill(p, pq, pk_pages, kv_indices, max_score, fz, st);
}

msa_status launch_proxy_decode(const msa_plan_s* p, const void* pq, const void* pk_pages, const int32_t* kv_indices,
                               float* max_score, cudaStream_t st) {
  CUtensorMap km;
  if (!make_pk_map(&km, p, pk_pages)) return set_error(MSA_ERR_CUDA, "msa_proxy_maxscore: tensor map encoding failed");
  const int32_t* ustart = p->aux_d + p->proxy_unit_start_off;
  const float scale = 1.0f / sqrtf(static_cast<float>(p->dp));
  const int grid = p->num_sms;
  const auto* q = static_cast<const __nv_bfloat16*>(pq);
  cudaError_t e;
  if (p->dp == 64) {
    const int smem = kDecWarps * kDecStages * 128 * 64 * 2 + kDecWarps * kDecStages * 8 + 1024;
    cudaFuncSetAttribute(proxy_decode_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    e = launch_pdl(proxy_decode_kernel<64>, dim3(grid), dim3(32 * kDecWarps), smem, st, km, q, p->tiles_d, ustart,
                   p->n_tiles, kv_indices, p->num_pages, max_score, p->hp, p->max_blocks, scale, p->err_d);
  } else {
    const int smem = kDecWarps * kDecStages * 128 * 32 * 2 + kDecWarps * kDecStages * 8 + 1024;
    cudaFuncSetAttribute(proxy_decode_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    e = launch_pdl(proxy_decode_kernel<32>, dim3(grid), dim3(32 * kDecWarps), smem, st, km, q, p->tiles_d, ustart,
                   p->n_tiles, kv_indices, p->num_pages, max_score, p->hp, p->max_blocks, scale, p->err_d);
  }
  return cuda_check(e, "msa_proxy_maxscore: decode launch");
}

msa_status launch_proxy_decode_fp8(const msa_plan_s* p, const void* pq, const void* pk_pages, const float* pk_scale,
                                   const int32_t* kv_indices, float* max_score, cudaStream_t st) {
  if (p->hp > 8) return set_error(MSA_ERR_UNSUPPORTED, "msa_proxy_maxscore_fp8: up to 8 proxy heads");
  if (p->dp != 64) return set_error(MSA_ERR_UNSUPPORTED, "msa_proxy_maxscore_fp8: proxy_head_dim 64 only");
  CUtensorMap km;
  const uint64_t dims[2] = {64, static_cast<uint64_t>(p->num_pages) * 128};
  const uint64_t strides[1] = {64};
  const uint32_t box[2] = {64, 128};
  if (!encode_tensor_map(&km, 2, pk_pages, dims, strides, box, 0, 64))
    return set_error(MSA_ERR_CUDA, "msa_proxy_maxscore_fp8: tensor map encoding failed");
  const int32_t* ustart = p->aux_d + p->proxy_unit_start_off;
  const float scale = 1.0f / sqrtf(64.0f);
  constexpr int W = kDec8Warps, S = kDec8Stages;
  const int smem = W * S * 128 * 64 + W * S * 8 + 1024;
  cudaFuncSetAttribute(proxy_decode_fp8_kernel<W, S>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return cuda_check(launch_pdl(proxy_decode_fp8_kernel<W, S>, dim3(p->num_sms), dim3(32 * W), smem, st, km,
                                static_cast<const __nv_bfloat16*>(pq), pk_scale, p->tiles_d, ustart, p->n_tiles,
                                kv_indices, p->num_pages, max_score, p->hp, p->max_blocks, scale, p->err_d),
                    "msa_proxy_maxscore_fp8: launch");
}

}  // namespace msa
