// LoRA shrink and expand over virtual-expert blocks (sm_103a).
//
// Shrink: fork PR #24 "Root cause" commit -- the MoL shrink stage is a
// fused-MoE GEMM over the virtual experts with N = S*r and K = the input width;
// code-review commit -- weight laid out [E, N, K].
// Expand: fork PR #24 PR body "Background (measured attribution)" -- the
// down-delta expand is an M x 6144 output from a K = rank = 32 contraction
// whose real traffic is a few MB; "Fix" -- expand weight view [E, N, K].
//
// Both stages are small-M grouped contractions: for each routed block, the
// gathered rows (1..BLOCK_M real pairs) times one virtual expert's weight,
// transposed. The weight is the HBM stream; rows are few. Each block of the
// grid is one (routed block, weight tile) work item, and items whose routed
// block is past num_tokens_post_padded or a sentinel block return at once, so
// the work done follows the real rows, not the padded worst case: a block
// with c real rows runs ceil(c/16) row tiles, never BLOCK_M rows of padding.
//
// The contraction runs on mma.sync m16n8k16 (bf16 in, fp32 accumulate).
// Because a dot product does not depend on the order of its terms, the k
// index is permuted identically in both operands so that every lane's
// fragment is one contiguous 16-byte run of a K-contiguous row: thread
// (g, t) of a warp reads row g at k = 8t..8t+7 of each 32-wide k block
// (16-byte loads, every 32-byte sector fully used), for both the activation
// rows and the weight rows. For the expand, the output column order inside a
// warp tile is permuted the same way so that each thread ends with 8
// adjacent outputs per row, read-modified-written with one 16-byte access.
//
// The expand's A operand is the fp32 intermediate, split into a bf16 head
// and a bf16 tail (two mma per step): 16 significant bits per value, error
// about 2^-17 relative -- far below the final bf16 rounding of the output.

#include <algorithm>

#include "mol_device.cuh"
#include "mol_internal.h"

namespace mol {

constexpr int kShrinkThreads = 128;  // 4 warps split the K range of one item
constexpr int kShrinkNT = 2;         // 8-column mma tiles per item -> 16 weight rows
constexpr int kShrinkUnroll = 4;     // 32-wide k blocks in flight per warp
constexpr int kExpandThreads = 128;  // 4 warps x 32 output columns
constexpr int kExpandCols = 128;

template <int NT, int UNROLL>
__global__ void __launch_bounds__(kShrinkThreads)
lora_shrink_kernel(const uint16_t* __restrict__ x, int64_t x_stride, int x_div, int K,
                   const uint16_t* __restrict__ lora_a, int R, const int* __restrict__ sorted_ids,
                   const int* __restrict__ expert_ids, const int* __restrict__ ntpp_ptr,
                   int block_m, int64_t numel, int num_vexperts, float* __restrict__ inter,
                   int n_jt) {
  constexpr int JT = 8 * NT;
  constexpr int NW = kShrinkThreads / 32;
  __shared__ int rows[128];
  __shared__ int wcnt[NW];
  __shared__ float red[NW - 1][NT * 4][32];

  const int t = blockIdx.x / n_jt;
  const int jt = blockIdx.x - t * n_jt;
  if ((int64_t)t * block_m >= (int64_t)__ldg(ntpp_ptr)) return;
  const int v = __ldg(expert_ids + t);
  if (v < 0 || v >= num_vexperts) return;
  const int c = compact_block_rows(sorted_ids + (int64_t)t * block_m, block_m, numel, rows, wcnt);
  if (c == 0) return;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, tq = lane & 3;
  const int nkb = (K + 31) >> 5;
  const int kb0 = warp * nkb / NW, kb1 = (warp + 1) * nkb / NW;
  const int j0 = jt * JT;
  const uint16_t* arow[NT];
#pragma unroll
  for (int u = 0; u < NT; ++u) arow[u] = lora_a + ((int64_t)v * R + j0 + 8 * u + g) * K + 8 * tq;
  const uint4 zero = make_uint4(0, 0, 0, 0);

  for (int m0 = 0; m0 < c; m0 += 16) {
    const int r0 = m0 + g, r1 = m0 + 8 + g;
    const uint16_t* xr0 = r0 < c ? x + (int64_t)(rows[r0] / x_div) * x_stride + 8 * tq : nullptr;
    const uint16_t* xr1 = r1 < c ? x + (int64_t)(rows[r1] / x_div) * x_stride + 8 * tq : nullptr;
    float acc[NT][4];
#pragma unroll
    for (int u = 0; u < NT; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;

    for (int kb = kb0; kb < kb1; kb += UNROLL) {
      uint4 a[UNROLL][NT], x0[UNROLL], x1[UNROLL];
#pragma unroll
      for (int uu = 0; uu < UNROLL; ++uu) {
        const int k = (kb + uu) * 32;
        const bool kin = (kb + uu < kb1) && (k + 8 * tq < K);
#pragma unroll
        for (int u = 0; u < NT; ++u) a[uu][u] = kin ? ld_stream16(arow[u] + k) : zero;
        x0[uu] = (kin && xr0) ? ld_keep16(xr0 + k) : zero;
        x1[uu] = (kin && xr1) ? ld_keep16(xr1 + k) : zero;
      }
#pragma unroll
      for (int uu = 0; uu < UNROLL; ++uu) {
#pragma unroll
        for (int u = 0; u < NT; ++u) {
          // k step 0 <- elements 8t..8t+3, k step 1 <- 8t+4..8t+7 (same map in both operands)
          mma_16816(acc[u], x0[uu].x, x1[uu].x, x0[uu].y, x1[uu].y, a[uu][u].x, a[uu][u].y);
          mma_16816(acc[u], x0[uu].z, x1[uu].z, x0[uu].w, x1[uu].w, a[uu][u].z, a[uu][u].w);
        }
      }
    }

    // Sum the four K-range partials in a fixed order (deterministic).
    if (warp > 0) {
#pragma unroll
      for (int u = 0; u < NT; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e) red[warp - 1][u * 4 + e][lane] = acc[u][e];
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int u = 0; u < NT; ++u) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int w = 0; w < NW - 1; ++w) acc[u][e] += red[w][u * 4 + e][lane];
        const int col = j0 + 8 * u + 2 * tq;
        if (r0 < c)
          *reinterpret_cast<float2*>(inter + (int64_t)rows[r0] * R + col) =
              make_float2(acc[u][0], acc[u][1]);
        if (r1 < c)
          *reinterpret_cast<float2*>(inter + (int64_t)rows[r1] * R + col) =
              make_float2(acc[u][2], acc[u][3]);
      }
    }
    __syncthreads();
  }
}

template <int RK>
__global__ void __launch_bounds__(kExpandThreads)
lora_expand_kernel(const float* __restrict__ inter, int R, const uint16_t* __restrict__ lora_b,
                   int S, int Ns, float scale, const float* __restrict__ topk_w,
                   const int* __restrict__ sorted_ids, const int* __restrict__ expert_ids,
                   const int* __restrict__ ntpp_ptr, int block_m, int64_t numel,
                   int num_vexperts, uint16_t* __restrict__ out, int64_t out_stride,
                   int chunks_per_slice) {
  constexpr bool K16 = (RK == 16);
  constexpr int KB = K16 ? 1 : RK / 32;  // k blocks (32 wide, or one 16-wide block)
  __shared__ int rows[128];
  __shared__ int wcnt[kExpandThreads / 32];

  const int per_block = S * chunks_per_slice;
  const int t = blockIdx.x / per_block;
  const int rem = blockIdx.x - t * per_block;
  const int s = rem / chunks_per_slice;
  const int chunk = rem - s * chunks_per_slice;
  if ((int64_t)t * block_m >= (int64_t)__ldg(ntpp_ptr)) return;
  const int v = __ldg(expert_ids + t);
  if (v < 0 || v >= num_vexperts) return;
  const int c = compact_block_rows(sorted_ids + (int64_t)t * block_m, block_m, numel, rows, wcnt);
  if (c == 0) return;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, tq = lane & 3;
  const int n_base = chunk * kExpandCols + warp * 32;  // column inside the slice
  if (n_base >= Ns) return;                            // warp-uniform; no block sync follows

  // Weight fragments. Lane (g, t) of 8-column tile u holds the weight row of
  // output column n_base + 8*(g/2) + 2u + (g%2), so thread t finishes with
  // columns n_base + 8t .. n_base + 8t + 7 of each row.
  const int grp = n_base + 8 * (g >> 1);
  const bool bvalid = grp < Ns;
  const uint16_t* bw =
      lora_b + ((int64_t)v * S * Ns + (int64_t)s * Ns + grp + (g & 1)) * RK;
  uint4 bf[KB][4];
#pragma unroll
  for (int kb = 0; kb < KB; ++kb)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if constexpr (K16) {
        const uint2 q = bvalid ? ld_stream8(bw + 2 * u * RK + 4 * tq) : make_uint2(0, 0);
        bf[kb][u] = make_uint4(q.x, q.y, 0, 0);
      } else {
        bf[kb][u] = bvalid ? ld_stream16(bw + 2 * u * RK + kb * 32 + 8 * tq) : make_uint4(0, 0, 0, 0);
      }
    }

  const bool ovalid = (n_base + 8 * tq) < Ns;
  const int64_t ocol = (int64_t)s * Ns + n_base + 8 * tq;
  const float4 zf = make_float4(0.f, 0.f, 0.f, 0.f);

  for (int m0 = 0; m0 < c; m0 += 16) {
    const int r0 = m0 + g, r1 = m0 + 8 + g;
    const int i0 = r0 < c ? rows[r0] : -1;
    const int i1 = r1 < c ? rows[r1] : -1;
    float acc[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;

#pragma unroll
    for (int kb = 0; kb < KB; ++kb) {
      const int koff = s * RK + (K16 ? 4 * tq : kb * 32 + 8 * tq);
      const float* p0 = inter + (int64_t)i0 * R + koff;
      const float* p1 = inter + (int64_t)i1 * R + koff;
      const float4 a0 = i0 >= 0 ? ld_keep_f4(p0) : zf;
      const float4 a1 = i1 >= 0 ? ld_keep_f4(p1) : zf;
      uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
      split_bf16x2(a0.x, a0.y, h0, l0);
      split_bf16x2(a1.x, a1.y, h1, l1);
      split_bf16x2(a0.z, a0.w, h2, l2);
      split_bf16x2(a1.z, a1.w, h3, l3);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        mma_16816(acc[u], h0, h1, h2, h3, bf[kb][u].x, bf[kb][u].y);
        mma_16816(acc[u], l0, l1, l2, l3, bf[kb][u].x, bf[kb][u].y);
      }
      if constexpr (!K16) {
        const float4 b0 = i0 >= 0 ? ld_keep_f4(p0 + 4) : zf;
        const float4 b1 = i1 >= 0 ? ld_keep_f4(p1 + 4) : zf;
        split_bf16x2(b0.x, b0.y, h0, l0);
        split_bf16x2(b1.x, b1.y, h1, l1);
        split_bf16x2(b0.z, b0.w, h2, l2);
        split_bf16x2(b1.z, b1.w, h3, l3);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          mma_16816(acc[u], h0, h1, h2, h3, bf[kb][u].z, bf[kb][u].w);
          mma_16816(acc[u], l0, l1, l2, l3, bf[kb][u].z, bf[kb][u].w);
        }
      }
    }

    if (ovalid) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = h ? i1 : i0;
        if (i < 0) continue;
        const float sw = topk_w ? scale * __ldg(topk_w + i) : scale;
        uint4* po = reinterpret_cast<uint4*>(out + (int64_t)i * out_stride + ocol);
        uint4 o = *po;
        uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float lo = fmaf(sw, acc[u][2 * h], bf16_lo(ow[u]));
          const float hi = fmaf(sw, acc[u][2 * h + 1], bf16_hi(ow[u]));
          ow[u] = pack_bf16x2(lo, hi);
        }
        *po = o;
      }
    }
  }
}

cudaError_t launch_shrink(const void* x, int64_t x_stride, int x_div, int K, const void* lora_a,
                          int R, const int32_t* sorted_ids, const int32_t* expert_ids,
                          const int32_t* ntpp, int64_t capacity, int block_m, int64_t numel,
                          int num_vexperts, float* inter, cudaStream_t stream) {
  const int64_t nblk = capacity / block_m;
  if (numel == 0 || nblk == 0) return cudaSuccess;
  const int n_jt = R / (8 * kShrinkNT);
  const int64_t grid = nblk * n_jt;
  lora_shrink_kernel<kShrinkNT, kShrinkUnroll><<<(unsigned)grid, kShrinkThreads, 0, stream>>>(
      static_cast<const uint16_t*>(x), x_stride, x_div, K, static_cast<const uint16_t*>(lora_a),
      R, sorted_ids, expert_ids, ntpp, block_m, numel, num_vexperts, inter, n_jt);
  return cudaGetLastError();
}

cudaError_t launch_expand(const float* inter, const void* lora_b, int S, int r, int Ns, float scale,
                          const float* topk_weights, const int32_t* sorted_ids,
                          const int32_t* expert_ids, const int32_t* ntpp, int64_t capacity,
                          int block_m, int64_t numel, int num_vexperts, void* out,
                          int64_t out_stride, cudaStream_t stream) {
  const int64_t nblk = capacity / block_m;
  if (numel == 0 || nblk == 0) return cudaSuccess;
  const int cps = (Ns + kExpandCols - 1) / kExpandCols;
  const int64_t grid = nblk * S * cps;
  const int R = S * r;
  const uint16_t* b = static_cast<const uint16_t*>(lora_b);
  uint16_t* o = static_cast<uint16_t*>(out);
#define MOL_EXPAND_CASE(RK)                                                                  \
  case RK:                                                                                   \
    lora_expand_kernel<RK><<<(unsigned)grid, kExpandThreads, 0, stream>>>(                   \
        inter, R, b, S, Ns, scale, topk_weights, sorted_ids, expert_ids, ntpp, block_m, numel, \
        num_vexperts, o, out_stride, cps);                                                   \
    break;
  switch (r) {
    MOL_EXPAND_CASE(16)
    MOL_EXPAND_CASE(32)
    MOL_EXPAND_CASE(64)
    MOL_EXPAND_CASE(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOL_EXPAND_CASE
  return cudaGetLastError();
}

}  // namespace mol
