// Stage 3 (prefill): GQA block-sparse flash attention forward, bf16 or FP8 K/V.
//
// For query row i of tile t and head h (KV head g = h / (Hq/Hkv), proxy
// head p = h / (Hq/Hp)): softmax over the keys of the selected blocks
// kv_block_indexes[t, p, :] that are visible to i, of q.k_g/sqrt(d); out =
// P.V_g and lse = ln sum exp ("MiniMax-AI/MSA" README, section "Usage":
// fmha_sm100(q, k_pages, v_pages, sparse_plan, kv_indices,
// kv_block_indexes); Flash-MSA article, "three key differences": the main
// attention is GQA and each proxy head picks its own block set).  With one
// proxy head per GQA group, p = g.
//
// A work unit is (tile, proxy head, pair of the query heads that use its
// blocks): both heads share every K/V block the TMA producer gathers
// through the page table.  Tensor memory holds S0, S1 (128 columns each) and O0, O1 (d
// columns each); the bf16 probabilities P_h overwrite the first 64 columns
// of S_h and feed the P.V MMA straight from tensor memory.  Roles:
//   warps 0-3  softmax of head 0 (thread = query row), warps 4-7 head 1,
//   warp 8     producer: builds each unit's block list (top-k row and page
//              rows, all 32 lanes at once) into a two-slot ring, loads Q per
//              unit and the K/V blocks into a 2-stage ring (one barrier per
//              stage for K and V),
//   warp 9     MMA issuer: S_h = Q_h K^T (smem x smem), O_h += P_h V
//              (tmem x smem), ordered QK0 QK1 | PV0 QK0' PV1 QK1' | ... so
//              that one head's softmax overlaps the other head's MMAs.
// The issuing thread runs only about one MMA ahead of the tensor pipe, so
// its loop does nothing between MMA groups that it can avoid: three waits
// and three commits per block step, descriptors precomputed.
// Online softmax in the log2 domain; the O rescale runs in the softmax
// warps between P.V steps, and the epilogue releases O_h to the next unit
// as soon as it is in registers.
//
// FP8 K/V ("MiniMax-AI/MSA" README, section "Stacks": sparse prefill in FP8
// next to BF16).  K/V pages hold e4m3 codes with one fp32 scale per KV
// head: logit = (q . k_code) * k_scale / sqrt(d), v = v_code * v_scale.  The
// producer gathers the 16 KB code blocks by TMA into the upper half of the
// K / V ring stages, and two converter warps (warps 10-11) expand them in
// place to f16 (exact: every e4m3 value is an f16) in the 128-byte-swizzled
// layout the MMAs read, and convert each unit's Q tiles in place from bf16
// to f16.  The MMAs then run kind::f16 with f16 operands (Q, K, P and V),
// k_scale folds into the softmax scale and v_scale into the epilogue.
// Rounding: Q to f16 is exact for |q| in [2^-14, 65504] (smaller values
// lose at most 2^-25, larger ones saturate) and P is rounded to f16 instead
// of bf16.
#include "msa_internal.h"
#include "ptx.cuh"

#include <algorithm>

namespace msa {
namespace {

constexpr int kStages = 2;
constexpr int kSoftWarps = 8;
constexpr int kConvWarps = 2;  // FP8 K/V only
constexpr int kEpiWarp0 = 12;  // warps 12-15: epilogue
constexpr int kMaxTopk = 1024;
// Four warpgroups: softmax (two), producer / MMA / FP8 converters, epilogue.
// Launched at 128 registers a thread; the softmax warpgroups then take
// kSoftRegs and the other two give theirs back down to kWg2Regs and
// kEpiRegs, which adds up to the launch's 512 x 128 (an increase waits for
// the decreases otherwise).
constexpr int kAttnThreads = 512;
constexpr int kLaunchRegs = 128;
constexpr int kSoftRegs = 168;
constexpr int kWg2Regs = 104;
constexpr int kEpiRegs = 72;
static_assert(256 * kSoftRegs + 128 * kWg2Regs + 128 * kEpiRegs == kAttnThreads * kLaunchRegs, "register split");

struct AttnUnit {
  int32_t tile, g, h0, nh;
};

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  tmem_st16(taddr, r);
  tmem_st16(taddr + 16, r + 16);
}

// One unit's cached blocks, built once by the producer warp (its lanes read
// the top-k row and the page table in parallel) for the MMA and softmax
// warps: a 16-int header, then j[cap] (selected blocks, padding and
// out-of-range entries dropped) and row[cap] (their first K/V tensor-map
// row), cap >= topk.
struct UnitHdr {
  int32_t n, nh, h0, q_begin, rows, pos0, g, pad[9];
};
constexpr int kListSlots = 2;
constexpr int kHdrInts = 16;

// A head's row statistics at the end of a unit, from the softmax warps to
// the epilogue warps (two buffers per head, alternating by unit).
struct UnitStats {
  int32_t n, active, ok, h0, q_begin, rows, g, pad[9];
  float m[128], l[128];
};

// Shared memory: Q (two heads), the K and V rings, the O staging buffer
// (kStageO: one 64-column box of a head's bf16 O tile, for the TMA stores of
// full tiles), barriers, the units' row statistics, then the two list slots,
// whose size follows topk.
template <int D, bool kStageO, int kLists = 1>
struct AttnSmem {
  static constexpr int kTileBytes = 128 * D * 2;  // 128 rows x D bf16, in D/64 swizzled chunks of 16 KB
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kOOff = kVOff + kStages * kTileBytes;
  static constexpr int kOChunkBytes = 128 * 64 * 2;  // 64 columns of 128 rows
  static constexpr int kBarOff = kOOff + (kStageO ? kOChunkBytes : 0);
  static constexpr int kStatOff = kBarOff + 8 * 64;
  static constexpr int kListOff = kStatOff + 4 * static_cast<int>(sizeof(UnitStats));
  static __host__ __device__ constexpr int slot_ints(int cap) { return kHdrInts + 2 * kLists * cap; }
  static __host__ __device__ constexpr int bytes(int cap) { return kListOff + kListSlots * slot_ints(cap) * 4; }
};

// Persistent: CTA b takes units b, b + gridDim.x, ... (heaviest first).
// Tensor memory, barriers and the K/V ring live across units; every
// barrier's phase comes from a running count (per head for the S / P / O
// barriers), and Q is released right after a unit's last QK so the next
// unit's Q load overlaps the tail of the current one.
template <int D, bool kOneKvHead, bool kFp8, bool kStageO>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const __grid_constant__ CUtensorMap o_map,
                    int32_t list_cap, const AttnUnit* __restrict__ units, int32_t n_units,
                    const TileInfo* __restrict__ tiles, const int32_t* __restrict__ idx,
                    const int32_t* __restrict__ kv_indices, int64_t num_pages, __nv_bfloat16* __restrict__ out,
                    float* __restrict__ lse, int32_t hq, int32_t hsel, int32_t kv_div, int32_t topk,
                    float scale_log2, const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                    uint32_t* err) {
  pdl_wait();
  // hsel block sets (proxy heads) per tile; a unit's u.g is its proxy head,
  // whose blocks are read from KV head u.g / kv_div of hsel / kv_div
  const int hkv = hsel / kv_div;
  // a one-head K/V pool (the backward's proxy softmax) pairs two proxy heads
  // per unit, each over its own blocks: one (j, row) list per head
  using L = AttnSmem<D, kStageO, kOneKvHead ? 2 : 1>;
  constexpr int kChunks = D / 64;
  static_assert(!kFp8 || (D == 128 && !kOneKvHead), "FP8 K/V: head_dim 128, main attention");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem + L::kQOff;
  uint8_t* k_s = smem + L::kKOff;
  uint8_t* v_s = smem + L::kVOff;
  int32_t* const list_base = reinterpret_cast<int32_t*>(smem + L::kListOff);
  // the staged layout sizes the list slots by topk; the other keeps them at
  // the compile-time maximum (constant offsets in the issue loops)
  const int cap = kStageO ? list_cap : kMaxTopk;
  const int slot_ints = L::slot_ints(cap);
  auto lhdr = [&](int k) -> UnitHdr& { return *reinterpret_cast<UnitHdr*>(list_base + (k % kListSlots) * slot_ints); };
  auto lj = [&](int k) -> int32_t* { return list_base + (k % kListSlots) * slot_ints + kHdrInts; };
  auto lrow = [&](int k) -> int32_t* { return list_base + (k % kListSlots) * slot_ints + kHdrInts + cap; };
  auto lj1 = [&](int k) -> int32_t* { return list_base + (k % kListSlots) * slot_ints + kHdrInts + 2 * cap; };
  auto lrow1 = [&](int k) -> int32_t* { return list_base + (k % kListSlots) * slot_ints + kHdrInts + 3 * cap; };
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* kv_full = bars + 2;              // [kStages]: K and V of a block
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;  // [2]
  uint64_t* p_full = s_full + 2;          // [2]
  uint64_t* o_done = p_full + 2;          // [2]: a unit's last P.V of head h
  uint64_t* o_free = o_done + 2;          // [2]
  uint64_t* list_full = o_free + 2;       // [kListSlots]
  uint64_t* list_empty = list_full + kListSlots;
  uint64_t* drain = list_empty + kListSlots;
  uint64_t* raw_full = drain + 1;          // [kStages], FP8: e4m3 K and V codes landed
  uint64_t* q_ready = raw_full + kStages;  // FP8: Q converted to f16
  uint64_t* ost_ready = q_ready + 1;       // a head's O staged (kStageO)
  uint64_t* ost_free = ost_ready + 1;      // the TMA store has read it
  uint64_t* stat_full = ost_free + 1;      // [head * 2 + buffer]
  uint64_t* stat_empty = stat_full + 4;    // [head * 2 + buffer]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stat_empty + 4);
  UnitStats* const stats = reinterpret_cast<UnitStats*>(smem + L::kStatOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    prefetch_tmap(&q_map);
    prefetch_tmap(&k_map);
    prefetch_tmap(&v_map);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kv_full + s, kFp8 ? kConvWarps : 1);
      mbar_init(kv_empty + s, 1);
      mbar_init(raw_full + s, 1);
    }
    mbar_init(q_ready, kConvWarps);
    mbar_init(ost_ready, 4);  // the four epilogue warps
    mbar_init(ost_free, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(stat_full + i, 4);   // the head's four softmax warps
      mbar_init(stat_empty + i, 4);  // the four epilogue warps
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(s_full + h, 1);
      mbar_init(p_full + h, 4);
      mbar_init(o_done + h, 1);
      mbar_init(o_free + h, 4);  // the epilogue warps
    }
    for (int i = 0; i < kListSlots; ++i) {
      mbar_init(list_full + i, 1);
      mbar_init(list_empty + i, 1 + kSoftWarps + (kFp8 ? kConvWarps : 0));  // MMA thread, softmax (and converter) warps
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // each role's branch starts with its warpgroup's register share

  if (warp == 8) {
    // ---------------------------------------------------------- producer
    setmaxnreg_dec<kWg2Regs>();
    int kv_it = 0;
    bool ok = true;
    for (int k = 0, ui = blockIdx.x; ok && ui < n_units; ++k, ui += gridDim.x) {
      UnitHdr& ls = lhdr(k);
      int32_t* const ls_j = lj(k);
      int32_t* const ls_row = lrow(k);
      const AttnUnit u = units[ui];
      const TileInfo tl = tiles[u.tile];
      const int32_t* sel = idx + (static_cast<int64_t>(u.tile) * hsel + u.g) * topk;
      if (lane == 0) ok = mbar_wait_inl(list_empty + k % kListSlots, ((k / kListSlots) & 1) ^ 1, err);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      __syncwarp();
      if (!ok) break;
      // the unit's blocks: padding skipped, entries past the tile's valid
      // blocks dropped and reported, pages checked against the pool
      int n = 0;
      for (int b = 0; b < topk; b += 32) {
        const int kk = b + lane;
        const int j = kk < topk ? sel[kk] : -1;
        const bool valid = j >= 0 && j < tl.nvp;
        if (j >= tl.nvp) atomicOr(err, kErrDeviceCheck);
        int row = 0;
        if (valid) {
          int64_t page = kv_indices[tl.page_base + j];
          if (page < 0 || page >= num_pages) {
            atomicOr(err, kErrDeviceCheck);
            page = 0;
          }
          // K/V head of the unit's proxy head, or the single head of a one-head pool
          row = static_cast<int>((kOneKvHead ? page : page * hkv + u.g / kv_div) * 128);
        }
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, valid);
        if (valid) {
          const int o = n + __popc(m & ((1u << lane) - 1u));
          ls_j[o] = j;
          ls_row[o] = row;
        }
        n += __popc(m);
      }
      const bool pair = kOneKvHead && u.nh == 2;
      if (pair) {
        // the second proxy head's own blocks (selection row g + 1); the
        // shorter list is padded with j = -1 (fully masked, page row 0)
        int32_t* const ls_j1 = lj1(k);
        int32_t* const ls_row1 = lrow1(k);
        const int32_t* sel1 = sel + topk;
        int n1 = 0;
        for (int b = 0; b < topk; b += 32) {
          const int kk = b + lane;
          const int j = kk < topk ? sel1[kk] : -1;
          const bool valid = j >= 0 && j < tl.nvp;
          if (j >= tl.nvp) atomicOr(err, kErrDeviceCheck);
          int row = 0;
          if (valid) {
            int64_t page = kv_indices[tl.page_base + j];
            if (page < 0 || page >= num_pages) {
              atomicOr(err, kErrDeviceCheck);
              page = 0;
            }
            row = static_cast<int>(page * 128);
          }
          const uint32_t m = __ballot_sync(0xFFFFFFFFu, valid);
          if (valid) {
            const int o = n1 + __popc(m & ((1u << lane) - 1u));
            ls_j1[o] = j;
            ls_row1[o] = row;
          }
          n1 += __popc(m);
        }
        for (int i = n + lane; i < n1; i += 32) {
          ls_j[i] = -1;
          ls_row[i] = 0;
        }
        for (int i = n1 + lane; i < n; i += 32) {
          ls_j1[i] = -1;
          ls_row1[i] = 0;
        }
        n = n > n1 ? n : n1;
      }
      if (lane == 0) {
        ls.n = n;
        ls.nh = u.nh;
        ls.h0 = u.h0;
        ls.q_begin = tl.q_begin;
        ls.rows = tl.rows;
        ls.pos0 = tl.pos0;
        ls.g = u.g / kv_div;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(list_full + k % kListSlots);
        if (k > 0) ok = mbar_wait_inl(q_empty, (k - 1) & 1, err);
        if (ok) {
          mbar_expect_tx(q_full, u.nh * L::kTileBytes);
          for (int h = 0; h < u.nh; ++h)
            for (int c = 0; c < kChunks; ++c)
              tma_load_3d(q_s + h * L::kTileBytes + c * 16384, &q_map, q_full, c * 64, u.h0 + h, tl.q_begin);
        }
        for (int i = 0; ok && i < n; ++i, ++kv_it) {
          const int s = kv_it % kStages;
          if (!(ok = mbar_wait_inl(kv_empty + s, ((kv_it / kStages) & 1) ^ 1, err))) break;
          const int row = ls_row[i];
          if (kFp8) {  // e4m3 codes into the upper half of the stage; the converters expand them
            mbar_expect_tx(raw_full + s, 2 * 16384);
            tma_load_2d(k_s + s * L::kTileBytes + 16384, &k_map, raw_full + s, 0, row);
            tma_load_2d(v_s + s * L::kTileBytes + 16384, &v_map, raw_full + s, 0, row);
            continue;
          }
          // a one-head pool's keys are its values: one load serves both, and
          // a paired unit's second head reads its own block from the V region
          const bool pair = kOneKvHead && u.nh == 2;
          const int row1 = pair ? lrow1(k)[i] : row;
          mbar_expect_tx(kv_full + s, (kOneKvHead && !pair ? 1 : 2) * L::kTileBytes);
          for (int c = 0; c < kChunks; ++c)
            tma_load_2d(k_s + s * L::kTileBytes + c * 16384, &k_map, kv_full + s, c * 64, row);
          if (!kOneKvHead || pair)
            for (int c = 0; c < kChunks; ++c)
              tma_load_2d(v_s + s * L::kTileBytes + c * 16384, &v_map, kv_full + s, c * 64, row1);
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    }
  } else if (warp == 9) {
    // --------------------------------------------------------------- MMA
    setmaxnreg_dec<kWg2Regs>();
    if (lane == 0) {
      // The issuing thread runs only a step ahead of the tensor pipe, so
      // anything between two MMA groups (a wait, a commit, address
      // arithmetic) idles the pipe: descriptors are precomputed, K and V of
      // a block share one barrier, O_h's barrier is committed once per unit
      // (a block's S_h commit already covers the previous P_h.V), and the
      // per-head phase counters are scalars.
      constexpr uint32_t id_qk = kFp8 ? idesc_f16_f32(128, 128, false, false) : idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_pv = kFp8 ? idesc_f16_f32(128, D, false, true) : idesc_bf16_f32(128, D, false, true);
      constexpr uint64_t kTileDesc = L::kTileBytes >> 4;
      const uint64_t qd0 = smem_desc(smem_u32(q_s), 16, 1024, kSwizzle128);
      const uint64_t kd0 = smem_desc(smem_u32(k_s), 16, 1024, kSwizzle128);
      const uint64_t vd0 = smem_desc(smem_u32(kOneKvHead ? k_s : v_s), 16384, 1024, kSwizzle128);
      // a paired one-head unit: head 1's block sits in the V region, as its
      // keys (K-major) and its values (rows-major)
      const uint64_t kd1 = smem_desc(smem_u32(v_s), 16, 1024, kSwizzle128);
      const uint64_t vd1 = smem_desc(smem_u32(v_s), 16384, 1024, kSwizzle128);
      auto qk = [&](int h, int s) {
        const uint64_t qd = qd0 + h * kTileDesc, kd = (kOneKvHead && h == 1 ? kd1 : kd0) + s * kTileDesc;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
          mma_ss(tmem + h * 128, qd + off, kd + off, id_qk, kk > 0);
        }
        mma_commit(s_full + h);
      };
      auto pv = [&](int h, int s, bool acc) {
        const uint64_t vd = (kOneKvHead && h == 1 ? vd1 : vd0) + s * kTileDesc;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + 256 + h * D, tmem + h * 128 + kk * 8, vd + ((kk * 2048) >> 4), id_pv, acc || (kk > 0));
      };
      int kv_it = 0, ch0 = 0, ch1 = 0;
      bool ok = true;
      for (int k = 0, ui = blockIdx.x; ok && ui < n_units; ++k, ui += gridDim.x) {
        if (!(ok = mbar_wait_inl(list_full + k % kListSlots, (k / kListSlots) & 1, err))) break;
        const int n = lhdr(k).n;
        const bool two = lhdr(k).nh == 2;
        mbar_arrive(list_empty + k % kListSlots);
        if (!(ok = mbar_wait_inl(kFp8 ? q_ready : q_full, k & 1, err))) break;
        tc_fence_after();
        // O_h of every unit is released by the epilogue once per unit; the
        // MMA thread waits for that release in every unit (also where it
        // issues nothing into O_h), so that a parity wait never meets a
        // barrier two phases behind
        if (n == 0) {
          mma_commit(q_empty);
          if (k > 0 && !(ok = mbar_wait_inl(o_free, (k - 1) & 1, err) && mbar_wait_inl(o_free + 1, (k - 1) & 1, err)))
            break;
          continue;
        }
        if (!(ok = mbar_wait_inl(kv_full + (kv_it & 1), (kv_it >> 1) & 1, err))) break;
        tc_fence_after();
        qk(0, kv_it & 1);
        if (two) qk(1, kv_it & 1);
        if (n == 1) mma_commit(q_empty);  // the unit's last QK is issued
        for (int i = 0; i < n; ++i) {
          const int it = kv_it + i;
          const int s = it & 1, s1 = s ^ 1;
          const bool more = i + 1 < n;
          // head 0: P_0 . V, then S_0 of the next block
          if (!(ok = mbar_wait_inl(p_full, (ch0 + i) & 1, err))) break;
          // the first P.V of a unit overwrites O_h: the previous unit's
          // epilogue must have read it (the QKs above already overlap it)
          if (i == 0 && k > 0 && !(ok = mbar_wait_inl(o_free, (k - 1) & 1, err))) break;
          if (i == 0 && k > 0 && !two && !(ok = mbar_wait_inl(o_free + 1, (k - 1) & 1, err))) break;
          tc_fence_after();
          pv(0, s, i > 0);
          if (!two) mma_commit(kv_empty + s);
          if (more) {
            if (!(ok = mbar_wait_inl(kv_full + s1, ((it + 1) >> 1) & 1, err))) break;
            tc_fence_after();
            qk(0, s1);
            if (!two && i + 1 == n - 1) mma_commit(q_empty);
          } else {
            mma_commit(o_done);
          }
          if (!two) continue;
          // head 1
          if (!(ok = mbar_wait_inl(p_full + 1, (ch1 + i) & 1, err))) break;
          if (i == 0 && k > 0 && !(ok = mbar_wait_inl(o_free + 1, (k - 1) & 1, err))) break;
          tc_fence_after();
          pv(1, s, i > 0);
          mma_commit(kv_empty + s);
          if (more) {
            qk(1, s1);
            if (i + 1 == n - 1) mma_commit(q_empty);
          } else {
            mma_commit(o_done + 1);
          }
        }
        ch0 += n;
        if (two) ch1 += n;
        kv_it += n;
      }
      mma_commit(drain);
      mbar_wait_inl(drain, 0, err);
    }
  } else if (warp < kSoftWarps) {
    // ----------------------------------------------------------- softmax
    setmaxnreg_inc<kSoftRegs>();
    // Each unit's row statistics go to the epilogue warps, which normalise
    // and store O while these warps go on to the next unit's blocks.
    const int h = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + h * 128;
    const uint32_t o_addr = tmem + lane_base + 256 + h * D;
    int ch = 0;  // blocks of head h so far
    bool ok = true;
    for (int k = 0, ui = blockIdx.x; ui < n_units; ++k, ui += gridDim.x) {
      const UnitHdr& ls = lhdr(k);
      const int32_t* const ls_j = kOneKvHead && h == 1 ? lj1(k) : lj(k);  // a paired unit's heads: own blocks
      if (ok) ok = mbar_wait_inl(list_full + k % kListSlots, (k / kListSlots) & 1, err);
      ok = __all_sync(0xFFFFFFFFu, ok);
      const int n = ok ? ls.n : 0, nh = ok ? ls.nh : 0;
      const int rows = ls.rows, pos0 = ls.pos0;
      // FP8: the scores are q . k_code, scaled by k_scale of the unit's KV head
      const float sl2 = kFp8 ? scale_log2 * k_scale[ls.g] : scale_log2;
      const bool active = ok && h < nh;
      const bool row_ok = r < rows;
      const int qpos = pos0 + r;
      float m = -INFINITY, l = 0.f;
      for (int i = 0; active && ok && i < n; ++i) {
        if (!(ok = mbar_wait_inl(s_full + h, (ch + i) & 1, err))) break;
        tc_fence_after();
        uint32_t sv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, sv + c * 32);
        tmem_wait_ld();
        const int j = ls_j[i];
        const bool pad = kOneKvHead && j < 0;  // the shorter list of a paired unit: every key masked
        const bool need_mask = pad || (j * 128 + 127 > pos0) || (rows < 128);
        if (need_mask) {  // only diagonal / ragged blocks: -inf past the row's position
          const int limit = row_ok && !pad ? qpos - j * 128 : -1;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > limit) sv[c] = __float_as_uint(-INFINITY);
        }
        float mx;
        {  // four independent chains keep the max off the latency path
          float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
          for (int c = 0; c < 128; c += 8) {
            a0 = fmax3(a0, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
            a1 = fmax3(a1, __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]));
            a2 = fmax3(a2, __uint_as_float(sv[c + 4]), __uint_as_float(sv[c + 5]));
            a3 = fmax3(a3, __uint_as_float(sv[c + 6]), __uint_as_float(sv[c + 7]));
          }
          mx = fmax3(fmaxf(a0, a1), a2, a3);
        }
        // lazy rescaling: the reference max moves only when the row max grows
        // by more than 2^8, so probabilities stay below 256 and O is rescaled
        // rarely
        const float mx2 = mx * sl2;
        const float m_new = mx2 > m + 8.f ? mx2 : m;
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = m_new == m ? 1.f : ex2_approx(m - m_use);
        float sum0 = 0.f, sum1 = 0.f, sum2 = 0.f, sum3 = 0.f;
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float x0, x1;
          ffma2(x0, x1, __uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1]), sl2, -m_use);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          if (c & 1)
            fadd2(sum2, sum3, p0, p1);
          else
            fadd2(sum0, sum1, p0, p1);
          pk[c] = kFp8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
        }
        sum0 += sum2;
        sum1 += sum3;
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_st16(s_addr + c * 16, pk + c * 16);
        l = l * alpha + (sum0 + sum1);
        // rescale O_h (written by P.V of the previous block, already complete
        // because the S_h MMA of this block was issued after it)
        // (P_h.V of the previous block is complete: the MMA thread issued
        // this block's S_h after it, and s_full covers every earlier MMA)
        if (i > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(o_addr + c * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(o_addr + c * 32, ov);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full + h);
        m = m_new;
      }
      // this head's statistics (buffer k % 2, reused once the epilogue has
      // read its contents from two units back)
      const int b = k & 1;
      UnitStats& st = stats[h * 2 + b];
      if (k >= 2 && ok) ok = mbar_wait_inl(stat_empty + h * 2 + b, ((k >> 1) - 1) & 1, err);
      ok = __all_sync(0xFFFFFFFFu, ok);
      st.m[r] = m;
      st.l[r] = l;
      if (quarter == 0 && lane == 0) {
        st.n = n;
        st.active = active ? 1 : 0;
        st.ok = ok ? 1 : 0;
        st.h0 = ls.h0;
        st.q_begin = ls.q_begin;
        st.rows = rows;
        st.g = ls.g;
      }
      if (h < nh) ch += n;
      // the list slot may be refilled (every warp arrives once per unit, active or not)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(stat_full + h * 2 + b);
        mbar_arrive(list_empty + k % kListSlots);
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ---------------------------------------------------------- epilogue
    setmaxnreg_dec<kEpiRegs>();
    // Per unit, head 0 then head 1: wait for the softmax's statistics and
    // for the unit's last P.V, read O_h in 32-column chunks, release it to
    // the next unit's P.V, and write bf16 O = O_h / l (times v_scale for
    // FP8) and the natural-log LSE.  Full tiles of FP8 plans go through the
    // shared staging buffer and TMA tensor stores.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int od0 = 0, od1 = 0;  // units with blocks of head 0 / head 1 so far
    int ost_uses = 0;      // 64-column boxes staged so far
    bool ok = true;
    for (int k = 0, ui = blockIdx.x; ui < n_units; ++k, ui += gridDim.x) {
      const int b = k & 1;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        const UnitStats& st = stats[h * 2 + b];
        if (ok) ok = mbar_wait_inl(stat_full + h * 2 + b, (k >> 1) & 1, err);
        ok = __all_sync(0xFFFFFFFFu, ok);
        const int n = st.n, rows = st.rows, q_begin = st.q_begin, h0 = st.h0;
        const bool active = ok && st.active != 0;
        const bool unit_ok = ok && st.ok != 0;
        const float m = st.m[r], l = st.l[r];
        const float o_scale = kFp8 ? v_scale[st.g] : 1.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(stat_empty + h * 2 + b);
        if (!active) {
          __syncwarp();
          if (lane == 0) mbar_arrive(o_free + h);
          continue;
        }
        const bool has_o = n > 0;
        if (has_o && ok) ok = mbar_wait_inl(o_done + h, (h == 0 ? od0++ : od1++) & 1, err);
        ok = __all_sync(0xFFFFFFFFu, ok);
        tc_fence_after();
        const uint32_t o_addr = tmem + lane_base + 256 + h * D;
        const float inv_l = l > 0.f ? o_scale / l : 0.f;
        const bool row_ok = r < rows;
        const int64_t orow = static_cast<int64_t>(q_begin + r) * hq + h0 + h;
        const bool staged = kStageO && rows == 128;
        uint8_t* const ob = smem + L::kOOff + r * 128;
        uint4* const dst = reinterpret_cast<uint4*>(out + orow * D);
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          if (has_o) {
            tmem_ld32(o_addr + c * 32, ov);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = 0u;
          }
          if (c == D / 32 - 1) {  // all of O_h is in registers: the next unit's P.V may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free + h);
          }
          // staged: one 64-column box at a time, once the previous box's
          // store has read the buffer
          if (staged && (c & 1) == 0 && ost_uses > 0 && ok) ok = mbar_wait_inl(ost_free, (ost_uses - 1) & 1, err);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t* x = ov + 8 * e;
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(x[0]) * inv_l, __uint_as_float(x[1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(x[2]) * inv_l, __uint_as_float(x[3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(x[4]) * inv_l, __uint_as_float(x[5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(x[6]) * inv_l, __uint_as_float(x[7]) * inv_l);
            if (staged) {
              // the TMA box layout: 64-column chunks of 128-byte rows, 16-byte
              // units swizzled by row % 8
              const int unit = (c & 1) * 4 + e;
              *reinterpret_cast<uint4*>(ob + ((unit ^ (r & 7)) << 4)) = w;
            } else if (unit_ok && row_ok) {
              dst[c * 4 + e] = w;
            }
          }
          if (staged && (c & 1) == 1) {  // the box is complete: one thread stores it
            fence_async_shared();        // the TMA store reads it through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(ost_ready);
            if (quarter == 0 && lane == 0) {
              if (ok) ok = mbar_wait_inl(ost_ready, ost_uses & 1, err);
              if (ok && unit_ok) {
                tma_store_3d(&o_map, smem + L::kOOff, 64 * (c >> 1), h0 + h, q_begin);
                bulk_commit_group();
              }
              bulk_wait_group_read0();
              mbar_arrive(ost_free);
            }
            ++ost_uses;
          }
        }
        if (unit_ok && row_ok && lse != nullptr)
          lse[orow] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
      }
    }
    if (kStageO && quarter == 0 && lane == 0) bulk_wait_group0();  // the stores are complete
  } else if (kFp8) {
    // -------------------------------------------------- FP8 converters
    setmaxnreg_dec<kWg2Regs>();
    // Thread ct of the two warps owns rows ct and ct + 64 of every K / V
    // block: it reads a row's 128 e4m3 codes (eight 16-byte units of the
    // swizzled upper half of the stage) before it writes any of the row's
    // f16 units, and the only f16 units that land in that upper half are the
    // same row's, so no other thread's codes are overwritten.
    const int ct = threadIdx.x - 32 * (kSoftWarps + 2);
    auto expand = [&](uint8_t* buf) {  // buf: one ring stage, 2 chunks x [128 rows][128 B] of f16
#pragma unroll 1
      for (int rr = 0; rr < 2; ++rr) {
        const int r = ct + 64 * rr, sw = r & 7;
        const uint8_t* raw = buf + 16384 + r * 128;
        uint4 u[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) u[c] = *reinterpret_cast<const uint4*>(raw + ((c ^ sw) << 4));
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // codes of d in [16c, 16c + 16) -> two f16 units
          uint4 lo, hi;
          lo.x = e4m3x2_to_f16x2(u[c].x);
          lo.y = e4m3x2_to_f16x2(u[c].x >> 16);
          lo.z = e4m3x2_to_f16x2(u[c].y);
          lo.w = e4m3x2_to_f16x2(u[c].y >> 16);
          hi.x = e4m3x2_to_f16x2(u[c].z);
          hi.y = e4m3x2_to_f16x2(u[c].z >> 16);
          hi.z = e4m3x2_to_f16x2(u[c].w);
          hi.w = e4m3x2_to_f16x2(u[c].w >> 16);
          uint8_t* dst = buf + (c >> 2) * 16384 + r * 128;
          const int u0 = (c & 3) * 2;
          *reinterpret_cast<uint4*>(dst + ((u0 ^ sw) << 4)) = lo;
          *reinterpret_cast<uint4*>(dst + (((u0 + 1) ^ sw) << 4)) = hi;
        }
      }
    };
    int kv_it = 0;
    bool ok = true;
    for (int k = 0, ui = blockIdx.x; ok && ui < n_units; ++k, ui += gridDim.x) {
      const UnitHdr& ls = lhdr(k);
      ok = mbar_wait_inl(list_full + k % kListSlots, (k / kListSlots) & 1, err);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      const int n = ls.n, nh = ls.nh;
      __syncwarp();
      if (lane == 0) mbar_arrive(list_empty + k % kListSlots);
      // Q of the unit's heads, bf16 -> f16 in place
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait_inl(q_full, k & 1, err)))) break;
      for (int hh = 0; hh < nh; ++hh) {
        uint4* qv = reinterpret_cast<uint4*>(q_s + hh * L::kTileBytes);
#pragma unroll 4
        for (int e = ct; e < L::kTileBytes / 16; e += 32 * kConvWarps) {
          uint4 v = qv[e];
          v.x = bf16x2_to_f16x2(v.x);
          v.y = bf16x2_to_f16x2(v.y);
          v.z = bf16x2_to_f16x2(v.z);
          v.w = bf16x2_to_f16x2(v.w);
          qv[e] = v;
        }
      }
      fence_async_shared();  // the MMAs read these through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(q_ready);
      for (int i = 0; i < n; ++i, ++kv_it) {
        const int s = kv_it % kStages;
        if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait_inl(raw_full + s, (kv_it / kStages) & 1, err)))) break;
        expand(k_s + s * L::kTileBytes);
        expand(v_s + s * L::kTileBytes);
        fence_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(kv_full + s);
      }
    }
  } else {
    setmaxnreg_dec<kWg2Regs>();  // warps 10-11 without FP8 K/V: idle
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

}  // namespace

void attn_plan_tables(msa_plan_s* p, std::vector<int32_t>& aux) {
  // a unit: (tile, proxy head g, a pair of the query heads that use g's
  // blocks); with one proxy head per GQA group g is the group
  std::vector<AttnUnit> us;
  const int grp = p->hq / p->hp;
  for (int t = 0; t < p->n_tiles; ++t)
    for (int g = 0; g < p->hp; ++g)
      for (int h = 0; h < grp; h += 2) us.push_back(AttnUnit{t, g, g * grp + h, std::min(2, grp - h)});
  // heaviest first: a unit visits at most min(num_valid_pages, topk) blocks
  std::stable_sort(us.begin(), us.end(), [&](const AttnUnit& a, const AttnUnit& b) {
    return std::min(p->tiles[a.tile].nvp, p->topk) > std::min(p->tiles[b.tile].nvp, p->topk);
  });
  p->attn_units_off = static_cast<int64_t>(aux.size());
  p->n_attn_units = static_cast<int32_t>(us.size());
  const int32_t* raw = reinterpret_cast<const int32_t*>(us.data());
  aux.insert(aux.end(), raw, raw + us.size() * 4);
  // the proxy softmax of the backward: proxy heads g and g + 1 of a tile in
  // one unit, each over its own blocks (the two heads' softmaxes overlap each
  // other's products)
  std::vector<AttnUnit> ps;
  for (int t = 0; t < p->n_tiles; ++t)
    for (int g = 0; g < p->hp; g += 2) ps.push_back(AttnUnit{t, g, g, std::min(2, p->hp - g)});
  std::stable_sort(ps.begin(), ps.end(), [&](const AttnUnit& a, const AttnUnit& b) {
    return std::min(p->tiles[a.tile].nvp, p->topk) > std::min(p->tiles[b.tile].nvp, p->topk);
  });
  p->proxy_attn_units_off = static_cast<int64_t>(aux.size());
  p->n_proxy_attn_units = static_cast<int32_t>(ps.size());
  raw = reinterpret_cast<const int32_t*>(ps.data());
  aux.insert(aux.end(), raw, raw + ps.size() * 4);
}

namespace {

constexpr int kMaxSmem = 232448;  // 227 KB of dynamic shared memory per CTA

// Launches one instantiation: with O staged through shared memory (full
// tiles stored by TMA) for FP8 K/V when the list slots for this topk leave
// room for the staging buffer, else with per-thread stores.  Measured at
// S=32768: FP8 973 -> 1019 TFLOP/s staged; bf16 0.808 -> 0.826 ms staged,
// so bf16 keeps the per-thread stores.
// The register split above assumes the kernel is launched at exactly
// kLaunchRegs a thread; any other count would leave an increase waiting, so
// such a build is not launched.
template <typename K>
cudaError_t check_launch_regs(K kern) {
  cudaFuncAttributes a;
  const cudaError_t e = cudaFuncGetAttributes(&a, kern);
  if (e != cudaSuccess) return e;
  return a.numRegs == kLaunchRegs ? cudaSuccess : cudaErrorInvalidConfiguration;
}

template <int D, bool kOneKvHead, bool kFp8>
cudaError_t launch_attn_variant(dim3 grid, cudaStream_t st, const CUtensorMap& qm, const CUtensorMap& km,
                                const CUtensorMap& vm, const CUtensorMap& om, int32_t topk, const AttnUnit* units,
                                int32_t n_units, const TileInfo* tiles, const int32_t* idx,
                                const int32_t* kv_indices, int64_t num_pages, __nv_bfloat16* o, float* lse,
                                int32_t hq, int32_t hsel, int32_t kv_div, float scale_log2, const float* k_scale,
                                const float* v_scale, uint32_t* err) {
  const int cap = (topk + 3) & ~3;
  if constexpr (kFp8) {
    const int staged = AttnSmem<D, true, kOneKvHead ? 2 : 1>::bytes(cap) + 1024;
    if (staged <= kMaxSmem) {
      auto kern = attn_fwd_kernel<D, kOneKvHead, kFp8, true>;
      if (const cudaError_t e = check_launch_regs(kern)) return e;
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, staged);
      return launch_pdl(kern, grid, dim3(kAttnThreads), staged, st, qm, km, vm, om, cap, units, n_units,
                        tiles, idx, kv_indices, num_pages, o, lse, hq, hsel, kv_div, topk, scale_log2, k_scale,
                        v_scale, err);
    }
  }
  const int plain = AttnSmem<D, false, kOneKvHead ? 2 : 1>::bytes(kMaxTopk) + 1024;
  auto kern = attn_fwd_kernel<D, kOneKvHead, kFp8, false>;
  if (const cudaError_t e = check_launch_regs(kern)) return e;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plain);
  return launch_pdl(kern, grid, dim3(kAttnThreads), plain, st, qm, km, vm, om, cap, units, n_units, tiles, idx,
                    kv_indices, num_pages, o, lse, hq, hsel, kv_div, topk, scale_log2, k_scale, v_scale, err);
}

// [total_q, heads, D] bf16 rows as 3-D boxes of 64 columns x 1 head x 128 rows, 128-byte swizzle
bool rows_map(CUtensorMap* m, const void* base, int d, int heads, int64_t total_q) {
  const uint64_t dims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(heads), static_cast<uint64_t>(total_q)};
  const uint64_t str[2] = {static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(heads) * d * 2};
  const uint32_t box[3] = {64, 1, 128};
  return encode_tensor_map(m, 3, base, dims, str, box, 1, 128);
}

}  // namespace

msa_status launch_attn_prefill(const msa_plan_s* p, const void* q, const void* k_pages, const void* v_pages,
                               const int32_t* kv_indices, const int32_t* idx, const float* k_scale,
                               const float* v_scale, void* out, float* lse, cudaStream_t st) {
  if (p->topk > kMaxTopk) return set_error(MSA_ERR_UNSUPPORTED, "msa_sparse_attn: topk above 1024");
  const bool fp8 = p->kv_dtype == MSA_KV_FP8_E4M3;
  if (fp8 && p->d != 128)
    return set_error(MSA_ERR_UNSUPPORTED, "msa_sparse_attn: FP8 K/V prefill needs head_dim 128");
  CUtensorMap qm, km, vm, om;
  const int kv_elem = fp8 ? 1 : 2;
  const uint64_t kdims[2] = {static_cast<uint64_t>(p->d), static_cast<uint64_t>(p->num_pages) * p->hkv * 128};
  const uint64_t kstr[1] = {static_cast<uint64_t>(p->d) * kv_elem};
  // bf16: 64-column boxes (128 B rows); e4m3: whole 128-byte rows of codes
  const uint32_t kbox[2] = {fp8 ? 128u : 64u, 128};
  if (!rows_map(&qm, q, p->d, p->hq, p->total_q) || !rows_map(&om, out, p->d, p->hq, p->total_q) ||
      !encode_tensor_map(&km, 2, k_pages, kdims, kstr, kbox, fp8 ? 0 : 1, 128) ||
      !encode_tensor_map(&vm, 2, v_pages, kdims, kstr, kbox, fp8 ? 0 : 1, 128))
    return set_error(MSA_ERR_CUDA, "msa_sparse_attn: tensor map encoding failed");
  const AttnUnit* units = reinterpret_cast<const AttnUnit*>(p->aux_d + p->attn_units_off);
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(p->d));
  auto* o = static_cast<__nv_bfloat16*>(out);
  const dim3 grid(std::min(p->n_attn_units, p->num_sms));  // persistent: one CTA per SM
  const int kv_div = p->hp / p->hkv;
  cudaError_t e;
  if (fp8)
    e = launch_attn_variant<128, false, true>(grid, st, qm, km, vm, om, p->topk, units, p->n_attn_units, p->tiles_d,
                                              idx, kv_indices, p->num_pages, o, lse, p->hq, p->hp, kv_div, scale_log2,
                                              k_scale, v_scale, p->err_d);
  else if (p->d == 128)
    e = launch_attn_variant<128, false, false>(grid, st, qm, km, vm, om, p->topk, units, p->n_attn_units, p->tiles_d,
                                               idx, kv_indices, p->num_pages, o, lse, p->hq, p->hp, kv_div,
                                               scale_log2, nullptr, nullptr, p->err_d);
  else
    e = launch_attn_variant<64, false, false>(grid, st, qm, km, vm, om, p->topk, units, p->n_attn_units, p->tiles_d,
                                              idx, kv_indices, p->num_pages, o, lse, p->hq, p->hp, kv_div, scale_log2,
                                              nullptr, nullptr, p->err_d);
  return cuda_check(e, "msa_sparse_attn: prefill launch");
}

// The proxy softmax of the backward (the KL term's p_proxy): for proxy head g
// of each tile, over group g's cached visible keys, Op = sum_k p(k) pk[k]
// and its natural-log LSE, with scores pq.pk/sqrt(dp).  It is the forward
// above with pq as the queries, the one shared proxy K head as both keys and
// values, and one head per unit.  Op: bf16 [total_q, Hp, 64]; lse: fp32
// [total_q, Hp].
msa_status launch_proxy_softmax(const msa_plan_s* p, const void* pq, const void* pk_pages, const int32_t* kv_indices,
                                const int32_t* idx, void* op, float* lse, cudaStream_t st) {
  if (p->topk > kMaxTopk) return set_error(MSA_ERR_UNSUPPORTED, "msa_sparse_attn_bwd: topk above 1024");
  CUtensorMap qm, km, om;
  // pq and pk at dp = 32 are read as 64-column boxes whose upper half lies
  // past the tensor's edge: TMA fills it with zeros, so the dp = 64 kernel
  // computes the same scores and an Op whose columns [dp, 64) are zero
  const uint64_t kdims[2] = {static_cast<uint64_t>(p->dp), static_cast<uint64_t>(p->num_pages) * 128};
  const uint64_t kstr[1] = {static_cast<uint64_t>(p->dp) * 2};
  const uint32_t kbox[2] = {64, 128};
  if (!rows_map(&qm, pq, p->dp, p->hp, p->total_q) || !rows_map(&om, op, 64, p->hp, p->total_q) ||
      !encode_tensor_map(&km, 2, pk_pages, kdims, kstr, kbox, 1, 128))
    return set_error(MSA_ERR_CUDA, "msa_sparse_attn_bwd: tensor map encoding failed");
  const AttnUnit* units = reinterpret_cast<const AttnUnit*>(p->aux_d + p->proxy_attn_units_off);
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(p->dp));
  const dim3 grid(std::min(p->n_proxy_attn_units, p->num_sms));
  return cuda_check(launch_attn_variant<64, true, false>(grid, st, qm, km, km, om, p->topk, units,
                                                          p->n_proxy_attn_units, p->tiles_d, idx, kv_indices,
                                                          p->num_pages, static_cast<__nv_bfloat16*>(op), lse, p->hp,
                                                          p->hp, p->hp, scale_log2, nullptr, nullptr, p->err_d),
                    "msa_sparse_attn_bwd: proxy softmax launch");
}

}  // namespace msa
