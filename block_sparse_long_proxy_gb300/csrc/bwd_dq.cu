// Training extension, query side: dQ and the main term of the proxy-query
// gradient dpq of block-sparse GQA attention with the KL-coupled proxy
// (Flash-MSA article, backward-pass paragraph), on the tcgen05 tensor cores.
//
// One CTA per (query tile t, proxy head p): it runs the G = Hq/Hp query
// heads that use p's cached blocks one after the other.  Each head's Q_h is
// copied into tensor memory, dO_h stays in shared memory, and the tile's
// cached blocks stream through TMA rings (K three stages, V and pk two),
// one continuous stream over the G heads.  Per head h and block j:
//   S  = Q_h . K_j^T (Q from TMEM)   dP = dO_h . V_j^T        (M = rows, N = 128 keys)
//   P  = exp2(S sl2 - lse2) (masked)   dS = P * (dP - D)
//   dQ += dS . K_j       dpq += P . pk_j                     (dS, P from TMEM)
// Blocks are pipelined through split handoffs: the softmax hands P over
// before dS, and the MMA thread issues S of block j+1 right after dpq of
// block j and dP of j+1 right after dQ of j, so the tensor pipe has work
// while the softmax runs (its two warpgroups split the 128 keys).
// After each head dQ / sqrt(d) is stored.  dpq accumulates over all G heads
// in tensor memory (the pk rows are the same for the G heads), and at the
// end dpq * (-w / (G sqrt(dp))) is added to the proxy term the prep kernel
// stored: no partial sums leave the CTA and the order of the sum is fixed.
//
// Head switches: Q of the next head goes into the K stage of the previous
// head's last block; the next head's first two blocks are loaded while the
// previous head finishes, and its Q and dO once the previous head's
// products are done (dO's shared memory is theirs until then).
//
// Tensor memory: S 128 | dP 128 | dQ 128 | dpq 64 | Q 64 columns.  Warpgroup
// w owns keys 64w..64w+63 and writes its bf16 pairs into the first 32 of
// its 64 S / dP columns, so k-step kk (16 keys) of an A operand in TMEM
// starts at column (kk / 4) * 64 + (kk % 4) * 8.
// Roles: warps 0-7 softmax (thread = query row), warp 8 TMA producer,
// warp 9 MMA issuer.
#include "msa_internal.h"
#include "ptx.cuh"

namespace msa {
namespace {

constexpr int kD = 128;
// K, V and pk of a block stream through rings of their own: V is read by
// dP and pk by dpq early in a block's turn, K last (by dQ), so K's ring is
// one deeper (one of its stages holds a head's Q until Q is in tensor
// memory)
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kSoftWarps = 8;
constexpr int kThreads = 32 * (kSoftWarps + 2);
constexpr float kLog2e = 1.4426950408889634f;

constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDPQ = 384, kColQ = 448;

struct DqSmem {
  static constexpr int kDOOff = 0;                                  // dO_h: 2 x [128 rows][128 B]
  static constexpr int kKOff = 32768;                               // K ring: kKStages x 32 KB
  static constexpr int kVOff = kKOff + kKStages * 32768;            // V ring: kVStages x 32 KB
  static constexpr int kPkOff = kVOff + kVStages * 32768;           // pk ring: kVStages x 16 KB
  static constexpr int kBarOff = kPkOff + kVStages * 16384;
  static constexpr int kNbOff = kBarOff + 8 * 24;  // the tile's cached block count
  static constexpr int kBytes = kNbOff + 16;
};

__device__ __forceinline__ bool valid_block(int j, int nvp) { return j >= 0 && j < nvp; }

// 64 fp32 values times s, from registers to a 32-byte aligned row: full
// 32-byte sectors
__device__ __forceinline__ void store_row_v8(float* dst, const uint32_t (&a)[64], float s) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    st_global_v8(dst + 8 * i, __uint_as_float(a[8 * i]) * s, __uint_as_float(a[8 * i + 1]) * s,
                 __uint_as_float(a[8 * i + 2]) * s, __uint_as_float(a[8 * i + 3]) * s,
                 __uint_as_float(a[8 * i + 4]) * s, __uint_as_float(a[8 * i + 5]) * s,
                 __uint_as_float(a[8 * i + 6]) * s, __uint_as_float(a[8 * i + 7]) * s);
}

// K stage that holds head hh's Q until it is in tensor memory: the stage of
// the previous head's last block (stage 2 for the first head), never one of
// the head's first two blocks
__device__ __forceinline__ int q_stage(int hh, int nb) { return (hh * nb + 2) % kKStages; }

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap do_map,
                     const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                     const __grid_constant__ CUtensorMap pk_map, const TileInfo* __restrict__ tiles,
                     const int32_t* __restrict__ idx, const int32_t* __restrict__ kv_indices, int64_t num_pages,
                     const float* __restrict__ lse2t, const float* __restrict__ dsumt, float* __restrict__ dq,
                     float* __restrict__ dpq, const int32_t* __restrict__ heavy_tiles, int32_t hq, int32_t hkv,
                     int32_t hsel, int32_t topk, int32_t total_q, int32_t d, int32_t dp, float kl_weight,
                     uint32_t* err) {
  pdl_wait();  // launched with programmatic dependent launch: the previous kernel's writes first
  using L = DqSmem;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int t = heavy_tiles[blockIdx.x / hsel], ps = blockIdx.x % hsel;  // heaviest tiles first
  // the G heads ps*G .. ps*G+G-1 read KV head g and the blocks of proxy head ps
  const int G = hq / hsel, g = ps / (hsel / hkv);
  const TileInfo tl = tiles[t];
  const int32_t* row_idx = idx + (static_cast<int64_t>(t) * hsel + ps) * topk;

  uint8_t* do_s = smem + L::kDOOff;
  uint8_t* k_s = smem + L::kKOff;
  uint8_t* v_s = smem + L::kVOff;
  uint8_t* pk_s = smem + L::kPkOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* q_full = bars;                   // Q_h and dO_h loaded
  uint64_t* q_tm = bars + 1;                 // Q_h copied into tensor memory (its K stage free)
  uint64_t* k_full = bars + 2;               // [kKStages]
  uint64_t* k_empty = k_full + kKStages;     // [kKStages]
  uint64_t* v_full = k_empty + kKStages;     // [kVStages]
  uint64_t* v_empty = v_full + kVStages;     // [kVStages]
  uint64_t* pk_full = v_empty + kVStages;    // [kVStages]
  uint64_t* pk_empty = pk_full + kVStages;   // [kVStages]
  uint64_t* s_full = pk_empty + kVStages;  // S computed
  uint64_t* p_full = s_full + 1;           // P written (bf16, over S)
  uint64_t* dp_full = p_full + 1;          // dP computed
  uint64_t* ds_full = dp_full + 1;         // dS written (bf16, over dP)
  uint64_t* done = ds_full + 1;            // a head's products complete
  uint64_t* dq_free = done + 1;            // a head's dQ read out of tensor memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dq_free + 1);
  int32_t* nb_s = reinterpret_cast<int32_t*>(smem + L::kNbOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    prefetch_tmap(&q_map);
    prefetch_tmap(&do_map);
    prefetch_tmap(&k_map);
    prefetch_tmap(&v_map);
    prefetch_tmap(&pk_map);
    mbar_init(q_full, 1);
    mbar_init(q_tm, kSoftWarps);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 1);
      mbar_init(pk_full + s, 1);
      mbar_init(pk_empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, kSoftWarps);
    mbar_init(dp_full, 1);
    mbar_init(ds_full, kSoftWarps);
    mbar_init(done, 1);
    mbar_init(dq_free, kSoftWarps);
    fence_mbar_init();
  }
  if (warp == 8) {  // the tile's cached blocks (the same for the G heads)
    int c = 0;
    for (int k = lane; k < topk; k += 32) c += valid_block(row_idx[k], tl.nvp) ? 1 : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
    if (lane == 0) *nb_s = c;
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nb = *nb_s;

  if (nb == 0) {
    // no cached block: dQ = 0 for the G heads; dpq keeps the proxy term
    if (warp < kSoftWarps) {
      const int wg = warp >> 2, r = (warp & 3) * 32 + lane;
      if (r < tl.rows && wg * 64 < d)
        for (int hh = 0; hh < G; ++hh) {
          float4* dqr = reinterpret_cast<float4*>(
              dq + (static_cast<int64_t>(tl.q_begin + r) * hq + ps * G + hh) * d + wg * 64);
#pragma unroll
          for (int i = 0; i < 16; ++i) dqr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
  } else if (warp == 8) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      bool ok = true;
      int pend = -1;  // head whose Q sits in a K stage and is not yet known to be in tensor memory
      // confirms the pending Q copy, at the latest before the next head's Q
      // load (so that q_tm never runs two phases ahead of this wait)
      auto confirm_q = [&]() -> bool {
        if (pend < 0) return true;
        const bool r = mbar_wait(q_tm, pend & 1, err);
        pend = -1;
        return r;
      };
      auto load_qd = [&](int hh) -> bool {
        if (!confirm_q()) return false;
        if (hh > 0 && !mbar_wait(done, (hh - 1) & 1, err)) return false;  // dO and Q's stage free
        const int h = ps * G + hh;
        uint8_t* q_s = k_s + q_stage(hh, nb) * 32768;
        mbar_expect_tx(q_full, 65536);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(q_s + c * 16384, &q_map, q_full, c * 64, h, tl.q_begin);
          tma_load_3d(do_s + c * 16384, &do_map, q_full, c * 64, h, tl.q_begin);
        }
        pend = hh;
        return true;
      };
      // K, V and pk of the tile's block j as block gi of the stream
      auto load_block = [&](int gi, int j) -> bool {
        int64_t page = kv_indices[tl.page_base + j];
        if (page < 0 || page >= num_pages) page = 0;  // reported by the prep kernel
        const int row = static_cast<int>((page * hkv + g) * 128);
        const int ks = gi % kKStages, vs = gi % kVStages;
        if (!mbar_wait(k_empty + ks, ((gi / kKStages) & 1) ^ 1, err)) return false;
        if (pend >= 0 && ks == q_stage(pend, nb) && !confirm_q()) return false;  // the stage holds Q
        mbar_expect_tx(k_full + ks, 32768);
        for (int c = 0; c < 2; ++c) tma_load_2d(k_s + ks * 32768 + c * 16384, &k_map, k_full + ks, c * 64, row);
        if (!mbar_wait(v_empty + vs, ((gi / kVStages) & 1) ^ 1, err)) return false;
        mbar_expect_tx(v_full + vs, 32768);
        for (int c = 0; c < 2; ++c) tma_load_2d(v_s + vs * 32768 + c * 16384, &v_map, v_full + vs, c * 64, row);
        if (!mbar_wait(pk_empty + vs, ((gi / kVStages) & 1) ^ 1, err)) return false;
        mbar_expect_tx(pk_full + vs, 16384);
        tma_load_2d(pk_s + vs * 16384, &pk_map, pk_full + vs, 0, static_cast<int>(page * 128));
        return true;
      };
      // head hh's blocks: the first two before its Q and dO (from the second
      // head on they stream in while the previous head finishes)
      for (int hh = 0; ok && hh < G; ++hh) {
        if (hh == 0) ok = load_qd(0);
        int b = 0;
        for (int k = 0; ok && k < topk; ++k) {
          const int j = row_idx[k];
          if (!valid_block(j, tl.nvp)) continue;
          if (hh > 0 && b == 2 && !(ok = load_qd(hh))) break;
          ok = load_block(hh * nb + b, j);
          ++b;
        }
        if (ok && hh > 0 && b < 3) ok = load_qd(hh);  // a head of one or two blocks
      }
    }
  } else if (warp == 9) {
    // --------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);  // S, dP
      constexpr uint32_t id_q = idesc_bf16_f32(128, 128, false, true);   // dQ (B keys-major)
      constexpr uint32_t id_p = idesc_bf16_f32(128, 64, false, true);    // dpq
      // descriptors precomputed (one add per MMA): the issuing thread runs
      // only a step ahead of the tensor pipe
      const uint64_t k_km = smem_desc(smem_u32(k_s), 16, 1024, kSwizzle128);       // K, keys x d (S = Q K^T)
      const uint64_t v_km = smem_desc(smem_u32(v_s), 16, 1024, kSwizzle128);       // V (dP = dO V^T)
      const uint64_t k_mn = smem_desc(smem_u32(k_s), 16384, 1024, kSwizzle128);    // K as keys-major B (dQ += dS K)
      const uint64_t pk_mn = smem_desc(smem_u32(pk_s), 16384, 1024, kSwizzle128);  // pk (dpq += P pk)
      const uint64_t do_km = smem_desc(smem_u32(do_s), 16, 1024, kSwizzle128);
      constexpr uint64_t kTile = 32768 >> 4, kPkTile = 16384 >> 4;
      bool ok = true;
      auto sq = [&](int gi) -> bool {  // S = Q . K^T (Q from tensor memory) of stream block gi
        const int ks = gi % kKStages;
        if (!mbar_wait(k_full + ks, (gi / kKStages) & 1, err)) return false;
        tc_fence_after();
        const uint64_t so = static_cast<uint64_t>(ks) * kTile;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
          mma_ts(tmem + kColS, tmem + kColQ + kk * 8, k_km + so + off, id_s, kk > 0);
        }
        mma_commit(s_full);
        return true;
      };
      auto dpv = [&](int gi) -> bool {  // dP = dO . V^T of stream block gi, then V's stage is free
        const int vs = gi % kVStages;
        if (!mbar_wait(v_full + vs, (gi / kVStages) & 1, err)) return false;
        tc_fence_after();
        const uint64_t so = static_cast<uint64_t>(vs) * kTile;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
          mma_ss(tmem + kColDP, do_km + off, v_km + so + off, id_s, kk > 0);
        }
        mma_commit(dp_full);
        mma_commit(v_empty + vs);
        return true;
      };
      // Blocks are pipelined: S of block i+1 goes out as soon as dpq of block
      // i has taken P out of the S columns, and dP of i+1 as soon as dQ of i
      // has taken dS out of the dP columns, so the softmax computes P of i+1
      // while dQ of i runs and dS of i+1 while dpq of i+1 runs.
      for (int hh = 0; ok && hh < G; ++hh) {
        const int base = hh * nb;
        ok = mbar_wait(q_full, hh & 1, err) && mbar_wait(q_tm, hh & 1, err);  // dO_h in smem, Q_h in TMEM
        tc_fence_after();
        ok = ok && sq(base) && dpv(base);
        for (int b = 0; ok && b < nb; ++b) {
          const int gi = base + b;
          const bool next = b + 1 < nb;
          const int vs = gi % kVStages, ks = gi % kKStages;
          if (!(ok = mbar_wait(p_full, gi & 1, err))) break;
          if (!(ok = mbar_wait(pk_full + vs, (gi / kVStages) & 1, err))) break;
          tc_fence_after();
          const uint64_t po = static_cast<uint64_t>(vs) * kPkTile;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t a_col = (kk >> 2) * 64 + (kk & 3) * 8;  // warpgroup kk/4 packed its keys there
            mma_ts(tmem + kColDPQ, tmem + kColS + a_col, pk_mn + po + kk * 128, id_p, gi > 0 || kk > 0);
          }
          mma_commit(pk_empty + vs);
          if (next && !(ok = sq(gi + 1))) break;
          if (!(ok = mbar_wait(ds_full, gi & 1, err))) break;
          // the head's first dQ overwrites the previous head's, once read out
          if (b == 0 && hh > 0 && !(ok = mbar_wait(dq_free, (hh - 1) & 1, err))) break;
          tc_fence_after();
          const uint64_t so = static_cast<uint64_t>(ks) * kTile;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t a_col = (kk >> 2) * 64 + (kk & 3) * 8;
            mma_ts(tmem + kColDQ, tmem + kColDP + a_col, k_mn + so + kk * 128, id_q, b > 0 || kk > 0);
          }
          mma_commit(k_empty + ks);
          if (next && !(ok = dpv(gi + 1))) break;
        }
        mma_commit(done);
      }
    }
  } else {
    // ----------------------------------------------------------- softmax
    const int wg = warp >> 2, quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row of the tile
    const int kc0 = wg * 64;            // this warpgroup's keys within the block
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool row_ok = r < tl.rows;
    const int qpos = tl.pos0 + r;
    const int64_t q_row = tl.q_begin + r;
    const float sl2 = kLog2e * rsqrtf(static_cast<float>(d));
    const float qsc = rsqrtf(static_cast<float>(d));
    bool ok = true;
    for (int hh = 0; hh < G; ++hh) {
      const int h = ps * G + hh, base = hh * nb;
      const int64_t ei = static_cast<int64_t>(h) * total_q + q_row;
      const float l2 = row_ok ? lse2t[ei] : 0.f;
      const float dd = row_ok ? dsumt[ei] : 0.f;
      if (ok) ok = mbar_wait(q_full, hh & 1, err);
      ok = __all_sync(0xFFFFFFFFu, ok);  // the TMEM stores below are warp-collective
      if (!ok) break;
      {  // Q_h row r, d in [64 wg, 64 wg + 64), into tensor memory as bf16 pairs
        const uint8_t* qrow = k_s + q_stage(hh, nb) * 32768 + wg * 16384 + r * 128;
        uint32_t qv[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = *reinterpret_cast<const uint4*>(qrow + ((u ^ (r & 7)) << 4));
          qv[4 * u] = v.x;
          qv[4 * u + 1] = v.y;
          qv[4 * u + 2] = v.z;
          qv[4 * u + 3] = v.w;
        }
        tmem_st16(lane_base + kColQ + 32 * wg, qv);
        tmem_st16(lane_base + kColQ + 32 * wg + 16, qv + 16);
        tmem_wait_st();
        tc_fence_before();
        fence_async_shared();  // Q's shared memory is a K stage next: TMA writes follow these reads
        __syncwarp();
        if (lane == 0) mbar_arrive(q_tm);
      }
      int b = 0;
      for (int k = 0; ok && k < topk; ++k) {
        const int j = row_idx[k];
        if (!valid_block(j, tl.nvp)) continue;
        const int gi = base + b;
        if (!(ok = mbar_wait(s_full, gi & 1, err))) break;
        tc_fence_after();
        const int kbase = j * 128 + kc0;
        const bool need_mask = j * 128 + 127 > tl.pos0 || tl.rows < 128;  // diagonal block or ragged tile
        // P first (dpq needs only P; dP may still be running), then dS
        float pr[64];
#pragma unroll
        for (int c = 0; c < 2; ++c) {  // 32 keys at a time; packed pairs land in columns already read
          uint32_t sv[32], pa[16];
          tmem_ld32(lane_base + kColS + kc0 + 32 * c, sv);
          tmem_wait_ld();
          if (!need_mask) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float x0, x1;
              ffma2(x0, x1, __uint_as_float(sv[i]), __uint_as_float(sv[i + 1]), sl2, -l2);
              pr[32 * c + i] = ex2_approx(x0);
              pr[32 * c + i + 1] = ex2_approx(x1);
              pa[i >> 1] = pack_bf16x2(pr[32 * c + i], pr[32 * c + i + 1]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const int kp = kbase + 32 * c + i;
              const bool ok0 = row_ok && kp <= qpos, ok1 = row_ok && kp + 1 <= qpos;
              pr[32 * c + i] = ok0 ? ex2_approx(__uint_as_float(sv[i]) * sl2 - l2) : 0.f;
              pr[32 * c + i + 1] = ok1 ? ex2_approx(__uint_as_float(sv[i + 1]) * sl2 - l2) : 0.f;
              pa[i >> 1] = pack_bf16x2(pr[32 * c + i], pr[32 * c + i + 1]);
            }
          }
          tmem_st16(lane_base + kColS + kc0 + 16 * c, pa);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
        if (!(ok = mbar_wait(dp_full, gi & 1, err))) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dv_[32], da[16];
          tmem_ld32(lane_base + kColDP + kc0 + 32 * c, dv_);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float t0, t1, d0, d1;
            fadd2v(t0, t1, __uint_as_float(dv_[i]), __uint_as_float(dv_[i + 1]), -dd, -dd);
            fmul2(d0, d1, t0, t1, pr[32 * c + i], pr[32 * c + i + 1]);
            da[i >> 1] = pack_bf16x2(d0, d1);
          }
          tmem_st16(lane_base + kColDP + kc0 + 16 * c, da);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_full);
        ++b;
      }
      // the head's dQ: read out of tensor memory (the next head's dQ may then
      // start), then stored while the next head's Q and dO load
      if (ok) ok = mbar_wait(done, hh & 1, err);
      tc_fence_after();
      ok = __all_sync(0xFFFFFFFFu, ok);  // tcgen05.ld is warp-collective: every lane loads, valid rows store
      if (!ok) break;
      uint32_t a[64];
      tmem_ld32(lane_base + kColDQ + wg * 64, a);
      tmem_ld32(lane_base + kColDQ + wg * 64 + 32, a + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && hh + 1 < G) mbar_arrive(dq_free);
      // at d = 64 the second warpgroup's columns are padding
      if (row_ok && wg * 64 < d) store_row_v8(dq + (q_row * hq + h) * d + wg * 64, a, qsc);
    }
    // dpq: the main term over the G heads, added to the proxy term the prep
    // kernel stored (the last head's products are complete: waited above)
    if (ok) {
      const float f = -kl_weight * rsqrtf(static_cast<float>(dp)) / static_cast<float>(G);
      uint32_t a[32];
      tmem_ld32(lane_base + kColDPQ + wg * 32, a);
      tmem_wait_ld();
      if (row_ok && wg * 32 < dp) {  // at dp = 32 the second warpgroup's columns are padding
        float4* dpr = reinterpret_cast<float4*>(dpq + (q_row * hsel + ps) * dp + wg * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float4 v = dpr[i];
          v.x += __uint_as_float(a[4 * i]) * f;
          v.y += __uint_as_float(a[4 * i + 1]) * f;
          v.z += __uint_as_float(a[4 * i + 2]) * f;
          v.w += __uint_as_float(a[4 * i + 3]) * f;
          dpr[i] = v;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

}  // namespace

msa_status launch_bwd_dq_tc(const msa_plan_s* p, const void* q, const void* k_pages, const void* v_pages,
                            const void* dout, const void* pk_pages, const int32_t* idx, const int32_t* kv_indices,
                            const float* lse2t, const float* dsumt, float* dq, float* dpq, float kl_weight,
                            cudaStream_t st) {
  // tensors of their true width d (dp); the 64-column boxes read zeros past
  // the edge at d = 64 (dp = 32)
  CUtensorMap qm, dom, km, vm, pkm;
  const uint64_t d = static_cast<uint64_t>(p->d), dp = static_cast<uint64_t>(p->dp);
  const uint64_t qdims[3] = {d, static_cast<uint64_t>(p->hq), static_cast<uint64_t>(p->total_q)};
  const uint64_t qstr[2] = {d * 2, static_cast<uint64_t>(p->hq) * d * 2};
  const uint32_t qbox[3] = {64, 1, 128};
  const uint64_t kdims[2] = {d, static_cast<uint64_t>(p->num_pages) * p->hkv * 128};
  const uint64_t kstr[1] = {d * 2};
  const uint32_t kbox[2] = {64, 128};
  const uint64_t pkdims[2] = {dp, static_cast<uint64_t>(p->num_pages) * 128};
  const uint64_t pkstr[1] = {dp * 2};
  if (!encode_tensor_map(&qm, 3, q, qdims, qstr, qbox, 1, 128) ||
      !encode_tensor_map(&dom, 3, dout, qdims, qstr, qbox, 1, 128) ||
      !encode_tensor_map(&km, 2, k_pages, kdims, kstr, kbox, 1, 128) ||
      !encode_tensor_map(&vm, 2, v_pages, kdims, kstr, kbox, 1, 128) ||
      !encode_tensor_map(&pkm, 2, pk_pages, pkdims, pkstr, kbox, 1, 128))
    return set_error(MSA_ERR_CUDA, "msa_sparse_attn_bwd: tensor map encoding failed");
  const int smem = DqSmem::kBytes + 1024;
  cudaFuncSetAttribute(bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  // one CTA per (tile, proxy head), looping over the proxy head's query heads
  return cuda_check(launch_pdl(bwd_dq_tc_kernel, dim3(p->n_tiles * p->hp), dim3(kThreads), smem, st, qm, dom, km, vm,
                               pkm, p->tiles_d, idx, kv_indices, p->num_pages, lse2t, dsumt, dq, dpq,
                               p->aux_d + p->heavy_tiles_off, p->hq, p->hkv, p->hp, p->topk,
                               static_cast<int32_t>(p->total_q), p->d, p->dp, kl_weight, p->err_d),
                    "msa_sparse_attn_bwd: dq launch");
}

}  // namespace msa
