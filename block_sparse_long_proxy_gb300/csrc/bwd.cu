// Training extension: the backward of block-sparse GQA attention on the
// cached blocks, fused with the KL-coupled proxy gradient (Flash-MSA
// article, backward-pass paragraph: the KL between proxy and main attention
// needs both distributions, so both gradients come from one backward; the
// gradient of the KL loss with respect to a proxy score is p_proxy - p_main;
// the block indexes are the ones cached by the forward).
//
// For row i, head h (group g), key set Omega = visible keys of the cached
// blocks of (tile, g):
//   P = exp(q.k/sqrt(d) - lse), D = rowsum(dout*out), dS = P*(dout.v - D)
//   dq = dS.K/sqrt(d), dk = sum_h dS^T.q/sqrt(d), dv = sum_h P^T.dout
//   p_proxy = softmax_Omega(pq.pk/sqrt(dp)), p_main = mean_h P
//   dZ = w*(p_proxy - p_main), dpq = dZ.pk/sqrt(dp), dpk = dZ^T.pq/sqrt(dp)
// Both dpq and dpk split into a proxy term and a main term:
//   dpq = w/sqrt(dp) * (p_proxy.pk - (1/G) sum_h P_h.pk)
//   dpk = w/sqrt(dp) * (p_proxy^T.pq - (1/G) sum_h P_h^T.pq)
//
// Kernels, in stream order:
//   zero     dpk rows of every referenced page (it is reduced by atomics)
//   prep     per (tile, group): D of the group's heads and lse * log2(e),
//            both stored [head][row]; the proxy LSE over Omega (online
//            softmax, [group][row]) and dpq's proxy term (plain store)
//   index    block -> tiles inverse index of the cached selections
//   dq       per (tile, head), tcgen05 (bwd_dq.cu): dq (owned, plain
//            store) and dpq's main term (fp32 atomics, G per element)
//   dkv      per (cached block, group), tcgen05 (bwd_dkv.cu): loops over
//            the tiles that selected the block (sorted, so sums are
//            deterministic); dk, dv (owned, plain store) and dpk (both
//            terms, fp32 atomics across groups)
// The prep kernel's small products use mma.sync m16n8k16 (bf16 in, f32
// accumulate) with ldmatrix fragments from padded shared-memory tiles.
#include "msa_internal.h"
#include "ptx.cuh"

#include <algorithm>

namespace msa {
namespace {

constexpr int kD = 128;    // head dim of this kernel
constexpr int kDP = 64;    // proxy head dim of this kernel
constexpr int kLdP = kDP + 8;  // padded smem row of 64-wide tiles: 144 B
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// cp.async of 16 bytes; src_bytes = 0 zero-fills the destination.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// A fragment (16 x 16, row-major) at (r0, c0) of a bf16 smem tile with row
// pitch `ld` elements.
__device__ __forceinline__ void frag_a(const __nv_bfloat16* tile, int ld, int r0, int c0, uint32_t* a) {
  const int lane = threadIdx.x & 31;
  ldsm_x4(smem_u32(tile + (r0 + (lane & 15)) * ld + c0 + (lane >> 4) * 8), a);
}
// B fragments of two n8-tiles for S = A . T^T where T is stored row-major
// with rows = n: n in [n0, n0+16), k in [k0, k0+16).
// b[0..1]: n-tile n0, b[2..3]: n-tile n0+8.
__device__ __forceinline__ void frag_b_nk(const __nv_bfloat16* tile, int ld, int n0, int k0, uint32_t* b) {
  const int lane = threadIdx.x & 31;
  ldsm_x4(smem_u32(tile + (n0 + (lane & 7) + ((lane >> 4) << 3)) * ld + k0 + ((lane >> 3) & 1) * 8), b);
}
// B fragments of two n8-tiles for O = A . T where T is stored row-major with
// rows = k: k in [k0, k0+16), n in [n0, n0+16).
__device__ __forceinline__ void frag_b_kn(const __nv_bfloat16* tile, int ld, int k0, int n0, uint32_t* b) {
  const int lane = threadIdx.x & 31;
  ldsm_x4_t(smem_u32(tile + (k0 + (lane & 7) + ((lane >> 3) & 1) * 8) * ld + n0 + (lane >> 4) * 8), b);
}
// Load `rows` valid rows (others zero) of a [128 x W] bf16 tile from global
// rows at `src` with row stride `stride` elements into a padded smem tile.
template <int W>
__device__ __forceinline__ void load_tile(__nv_bfloat16* dst, const __nv_bfloat16* src, int64_t stride, int rows) {
  constexpr int kChunks = W / 8;  // 16-byte chunks per row
  for (int e = threadIdx.x; e < 128 * kChunks; e += blockDim.x) {
    const int r = e / kChunks, c = e % kChunks;
    const bool ok = r < rows;
    cp_async16(dst + r * (W + 8) + c * 8, ok ? src + r * stride + c * 8 : src, ok ? 16 : 0);
  }
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) { return pack_bf16x2(lo, hi); }

// ------------------------------------------------------------------ prep

// Per (tile, group): D[row, h] for the group's heads, the proxy LSE over the
// cached visible keys (log2 units, scale included) and dpq's proxy term.
__global__ void __launch_bounds__(kThreads)
    bwd_prep_kernel(const TileInfo* __restrict__ tiles, const int32_t* __restrict__ idx,
                    const int32_t* __restrict__ kv_indices, int64_t num_pages, const __nv_bfloat16* __restrict__ out,
                    const __nv_bfloat16* __restrict__ dout, const __nv_bfloat16* __restrict__ pq,
                    const __nv_bfloat16* __restrict__ pk, const float* __restrict__ lse, float* __restrict__ dsumt,
                    float* __restrict__ lse2t, float* __restrict__ lsept, float* __restrict__ dpq, int32_t hq,
                    int32_t hkv, int32_t topk, int32_t total_q, float kl_weight, uint32_t* err) {
  __shared__ __align__(16) __nv_bfloat16 pqs[128 * kLdP];
  __shared__ __align__(16) __nv_bfloat16 pks[128 * kLdP];
  const int t = blockIdx.x / hkv, g = blockIdx.x % hkv;
  const TileInfo tl = tiles[t];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, t4 = lane & 3;
  const int G = hq / hkv;

  // D = rowsum(dout * out): two lanes per row, 64 d values each
  for (int h = g * G; h < (g + 1) * G; ++h)
    for (int r = warp * 16 + (lane >> 1); r < 128; r += 128) {
      float acc = 0.f;
      if (r < tl.rows) {
        const int64_t off = (static_cast<int64_t>(tl.q_begin + r) * hq + h) * kD + (lane & 1) * 64;
        const uint4* a = reinterpret_cast<const uint4*>(out + off);
        const uint4* b = reinterpret_cast<const uint4*>(dout + off);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 x = a[c], y = b[c];
          const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 fx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[e]));
            const float2 fy = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[e]));
            acc += fx.x * fy.x + fx.y * fy.y;
          }
        }
      }
      acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
      if ((lane & 1) == 0 && r < tl.rows) {
        const int64_t q_row = tl.q_begin + r;
        dsumt[static_cast<int64_t>(h) * total_q + q_row] = acc;
        lse2t[static_cast<int64_t>(h) * total_q + q_row] = lse[q_row * hq + h] * kLog2e;
      }
    }

  // proxy softmax over the cached visible keys (online), O_proxy = p_proxy.pk
  load_tile<kDP>(pqs, pq + (static_cast<int64_t>(tl.q_begin) * hkv + g) * kDP, static_cast<int64_t>(hkv) * kDP,
                 tl.rows);
  const float zsl2 = kLog2e * rsqrtf(static_cast<float>(kDP));
  const int r0 = warp * 16 + gr, r1 = r0 + 8;
  const int qp0 = tl.pos0 + r0, qp1 = tl.pos0 + r1;
  const bool ok0 = r0 < tl.rows, ok1 = r1 < tl.rows;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  const int32_t* row_idx = idx + (static_cast<int64_t>(t) * hkv + g) * topk;
  for (int k = 0; k < topk; ++k) {
    const int j = row_idx[k];
    if (j < 0 || j >= tl.nvp) continue;
    int64_t page = kv_indices[tl.page_base + j];
    if (page < 0 || page >= num_pages) {
      if (threadIdx.x == 0) atomicOr(err, kErrDeviceCheck);
      page = 0;
    }
    __syncthreads();  // previous block's pks reads are done
    load_tile<kDP>(pks, pk + page * 128 * kDP, kDP, 128);
    cp_async_wait_all();
    __syncthreads();
    float z[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i][0] = z[i][1] = z[i][2] = z[i][3] = 0.f;
#pragma unroll
    for (int kc = 0; kc < kDP / 16; ++kc) {
      uint32_t a[4];
      frag_a(pqs, kLdP, warp * 16, kc * 16, a);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t b[4];
        frag_b_nk(pks, kLdP, np * 16, kc * 16, b);
        mma_bf16(z[2 * np], a, b[0], b[1]);
        mma_bf16(z[2 * np + 1], a, b[2], b[3]);
      }
    }
    // mask and row max (rows r0: z[.][0..1], r1: z[.][2..3])
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int kp = j * 128 + nt * 8 + 2 * t4 + c;
        z[nt][c] = (ok0 && kp <= qp0) ? z[nt][c] * zsl2 : -INFINITY;
        z[nt][2 + c] = (ok1 && kp <= qp1) ? z[nt][2 + c] * zsl2 : -INFINITY;
        mx0 = fmaxf(mx0, z[nt][c]);
        mx1 = fmaxf(mx1, z[nt][2 + c]);
      }
#pragma unroll
    for (int s = 1; s < 4; s <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, s));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, s));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = ex2_approx(m0 - mu0), al1 = ex2_approx(m1 - mu1);
    m0 = mn0;
    m1 = mn1;
    float s0 = 0.f, s1 = 0.f;
    uint32_t pa[8][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const float p00 = ex2_approx(z[nt][0] - mu0), p01 = ex2_approx(z[nt][1] - mu0);
      const float p10 = ex2_approx(z[nt][2] - mu1), p11 = ex2_approx(z[nt][3] - mu1);
      s0 += p00 + p01;
      s1 += p10 + p11;
      // C -> A fragment: k chunk nt/2; even n-tile fills a0a1/a2a3, odd a4a5/a6a7
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack2(p00, p01);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack2(p10, p11);
    }
    l0 = l0 * al0 + s0;
    l1 = l1 * al1 + s1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o[i][0] *= al0;
      o[i][1] *= al0;
      o[i][2] *= al1;
      o[i][3] *= al1;
    }
#pragma unroll
    for (int kc = 0; kc < 8; ++kc)
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b[4];
        frag_b_kn(pks, kLdP, kc * 16, np * 16, b);
        mma_bf16(o[2 * np], pa[kc], b[0], b[1]);
        mma_bf16(o[2 * np + 1], pa[kc], b[2], b[3]);
      }
  }
  cp_async_wait_all();
#pragma unroll
  for (int s = 1; s < 4; s <<= 1) {
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, s);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, s);
  }
  const float f = kl_weight * rsqrtf(static_cast<float>(kDP));
  const float i0 = l0 > 0.f ? f / l0 : 0.f, i1 = l1 > 0.f ? f / l1 : 0.f;
  if (ok0 && t4 == 0) lsept[static_cast<int64_t>(g) * total_q + tl.q_begin + r0] = l0 > 0.f ? m0 + log2f(l0) : -INFINITY;
  if (ok1 && t4 == 0) lsept[static_cast<int64_t>(g) * total_q + tl.q_begin + r1] = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int c = nt * 8 + 2 * t4;
    if (ok0)
      *reinterpret_cast<float2*>(dpq + (static_cast<int64_t>(tl.q_begin + r0) * hkv + g) * kDP + c) =
          make_float2(o[nt][0] * i0, o[nt][1] * i0);
    if (ok1)
      *reinterpret_cast<float2*>(dpq + (static_cast<int64_t>(tl.q_begin + r1) * hkv + g) * kDP + c) =
          make_float2(o[nt][2] * i1, o[nt][3] * i1);
  }
}

// ------------------------------------------------------------ inverse index

// count[e*hkv + g] = number of tiles whose cached blocks of group g include
// page-table entry e (entry = sequence's page_base + logical block).
__global__ void bwd_count_kernel(const TileInfo* __restrict__ tiles, const int32_t* __restrict__ idx, int32_t n_tiles,
                                 int32_t hkv, int32_t topk, int32_t* __restrict__ count) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<int64_t>(n_tiles) * hkv * topk) return;
  const int t = static_cast<int>(e / (static_cast<int64_t>(hkv) * topk));
  const int g = static_cast<int>((e / topk) % hkv);
  const int j = idx[e];
  const TileInfo tl = tiles[t];
  if (j < 0 || j >= tl.nvp) return;
  atomicAdd(count + (tl.page_base + j) * hkv + g, 1);
}

// Exclusive scan of n counts into off[0..n] (one CTA of 1024 threads);
// cursor[] is reset to off[].
__global__ void __launch_bounds__(1024) bwd_scan_kernel(const int32_t* __restrict__ count, int32_t n,
                                                        int32_t* __restrict__ off, int32_t* __restrict__ cursor) {
  __shared__ int32_t part[1024];
  const int per = (n + 1023) / 1024;
  const int b = threadIdx.x * per, e = min(n, b + per);
  int s = 0;
  for (int i = b; i < e; ++i) s += count[i];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const int v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int run = part[threadIdx.x] - s;
  for (int i = b; i < e; ++i) {
    off[i] = run;
    cursor[i] = run;
    run += count[i];
  }
  if (threadIdx.x == 1023) off[n] = part[1023];
}

__global__ void bwd_fill_kernel(const TileInfo* __restrict__ tiles, const int32_t* __restrict__ idx, int32_t n_tiles,
                                int32_t hkv, int32_t topk, int32_t* __restrict__ cursor, int32_t* __restrict__ list) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<int64_t>(n_tiles) * hkv * topk) return;
  const int t = static_cast<int>(e / (static_cast<int64_t>(hkv) * topk));
  const int g = static_cast<int>((e / topk) % hkv);
  const int j = idx[e];
  const TileInfo tl = tiles[t];
  if (j < 0 || j >= tl.nvp) return;
  list[atomicAdd(cursor + (tl.page_base + j) * hkv + g, 1)] = t;
}

// dpk rows of every referenced page start at zero (they are reduced by
// atomics across groups).
__global__ void bwd_zero_dpk_kernel(const int32_t* __restrict__ kv_indices, int32_t n_entries, int64_t num_pages,
                                    float* __restrict__ dpk) {
  const int e = blockIdx.x;
  if (e >= n_entries) return;
  const int64_t page = kv_indices[e];
  if (page < 0 || page >= num_pages) return;
  float4* p = reinterpret_cast<float4*>(dpk + page * 128 * kDP);
  for (int i = threadIdx.x; i < 128 * kDP / 4; i += blockDim.x) p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

}  // namespace

size_t bwd_scratch_bytes(const msa_plan_s* p) {
  if (p->decode) return 0;
  const size_t ent = static_cast<size_t>(p->n_page_entries) * p->hkv;
  const size_t bytes = sizeof(float) * static_cast<size_t>(p->total_q) * (2 * p->hq + p->hkv) +
                       sizeof(int32_t) * (3 * ent + 1 + static_cast<size_t>(p->n_tiles) * p->hkv * p->topk);
  return (bytes + 255) & ~size_t(255);
}

void bwd_plan_tables(msa_plan_s* p, std::vector<int32_t>& aux) {
  p->blk_j_off = static_cast<int64_t>(aux.size());
  for (int s = 0; s < p->batch; ++s) {
    const int nb = (p->kv_lens[s] + kPage - 1) / kPage;
    for (int j = 0; j < nb; ++j) aux.push_back(j);
  }
}

msa_status launch_attn_bwd(const msa_plan_s* p, const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* kv_indices, const int32_t* idx, const void* out, const float* lse,
                           const void* dout, const void* pq, const void* pk_pages, float kl_weight, float* dq,
                           float* dk, float* dv, float* dpq, float* dpk, cudaStream_t st) {
  if (p->decode) return set_error(MSA_ERR_UNSUPPORTED, "msa_sparse_attn_bwd: decode batches have no backward");
  if (p->d != kD || p->dp != kDP)
    return set_error(MSA_ERR_UNSUPPORTED, "msa_sparse_attn_bwd: head_dim 128 and proxy_head_dim 64 only");
  if (p->bwd_d == nullptr) return set_error(MSA_ERR_UNSUPPORTED, "msa_sparse_attn_bwd: plan has no backward scratch");
  const int n_ent = p->n_page_entries;
  const size_t ent = static_cast<size_t>(n_ent) * p->hkv;
  float* dsumt = reinterpret_cast<float*>(p->bwd_d);               // [hq][total_q]
  float* lse2t = dsumt + static_cast<size_t>(p->total_q) * p->hq;  // [hq][total_q], lse * log2(e)
  float* lsept = lse2t + static_cast<size_t>(p->total_q) * p->hq;  // [hkv][total_q], log2 units
  int32_t* cnt = reinterpret_cast<int32_t*>(lsept + static_cast<size_t>(p->total_q) * p->hkv);
  int32_t* off = cnt + ent;
  int32_t* cur = off + ent + 1;
  int32_t* list = cur + ent;
  const int32_t* blk_j = p->aux_d + p->blk_j_off;
  const auto* O = static_cast<const __nv_bfloat16*>(out);
  const auto* dO = static_cast<const __nv_bfloat16*>(dout);
  const auto* PQ = static_cast<const __nv_bfloat16*>(pq);
  const auto* PK = static_cast<const __nv_bfloat16*>(pk_pages);
  const int64_t n_sel = static_cast<int64_t>(p->n_tiles) * p->hkv * p->topk;

  bwd_zero_dpk_kernel<<<n_ent, 256, 0, st>>>(kv_indices, n_ent, p->num_pages, dpk);
  bwd_prep_kernel<<<p->n_tiles * p->hkv, kThreads, 0, st>>>(p->tiles_d, idx, kv_indices, p->num_pages, O, dO, PQ, PK,
                                                           lse, dsumt, lse2t, lsept, dpq, p->hq, p->hkv, p->topk,
                                                           static_cast<int32_t>(p->total_q), kl_weight, p->err_d);
  msa_status s = cuda_check(cudaMemsetAsync(cnt, 0, sizeof(int32_t) * ent, st), "msa_sparse_attn_bwd: memset");
  if (s != MSA_OK) return s;
  const int sel_blocks = static_cast<int>((n_sel + 255) / 256);
  bwd_count_kernel<<<sel_blocks, 256, 0, st>>>(p->tiles_d, idx, p->n_tiles, p->hkv, p->topk, cnt);
  bwd_scan_kernel<<<1, 1024, 0, st>>>(cnt, static_cast<int32_t>(ent), off, cur);
  bwd_fill_kernel<<<sel_blocks, 256, 0, st>>>(p->tiles_d, idx, p->n_tiles, p->hkv, p->topk, cur, list);
  s = cuda_check(cudaGetLastError(), "msa_sparse_attn_bwd: launch");
  if (s != MSA_OK) return s;
  s = launch_bwd_dq_tc(p, q, k_pages, v_pages, dout, pk_pages, idx, kv_indices, lse2t, dsumt, dq, dpq, kl_weight, st);
  if (s != MSA_OK) return s;
  return launch_bwd_dkv_tc(p, q, k_pages, v_pages, dout, pq, pk_pages, kv_indices, blk_j, off, list, lse2t, dsumt,
                           lsept, dk, dv, dpk, kl_weight, st);
}

}  // namespace msa
