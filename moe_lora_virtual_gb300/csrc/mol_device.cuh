// Device helpers shared by the MoL kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MOL_DEV __device__ __forceinline__

namespace mol {

// bf16 pair packed in one 32-bit register: low half = first (lower-k) element.
MOL_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
MOL_DEV float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
MOL_DEV float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Split an fp32 pair into a bf16 "head" pair and the bf16 pair of what is
// left. head + tail carries 16 significant bits of each value; the tail is
// exact (v - head has at most 16 significant bits of which bf16 keeps 8).
MOL_DEV void split_bf16x2(float a, float b, uint32_t& head, uint32_t& tail) {
  head = pack_bf16x2(a, b);
  tail = pack_bf16x2(a - bf16_lo(head), b - bf16_hi(head));
}

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col). Fragment layout
// (lane = 4*g + t): a0 = A[g][2t..], a1 = A[g+8][2t..], a2 = A[g][2t+8..],
// a3 = A[g+8][2t+8..]; b0 = B[2t..][g], b1 = B[2t+8..][g];
// d0 = D[g][2t], d1 = D[g][2t+1], d2 = D[g+8][2t], d3 = D[g+8][2t+1].
MOL_DEV void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                       uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte load of data read once (adapter weights): no L1 allocation.
MOL_DEV uint4 ld_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}
MOL_DEV uint2 ld_stream8(const void* p) {
  uint2 r;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
// 16-byte load of data other blocks reuse (activations, intermediates).
MOL_DEV uint4 ld_keep16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
MOL_DEV float4 ld_keep_f4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

MOL_DEV unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Compact the valid pair ids of one block (ids in [0, numel)) into `rows`,
// keeping slot order. Needs blockDim.x >= block_m and blockDim.x % 32 == 0;
// every thread of the block must call it. Returns the number of rows.
MOL_DEV int compact_block_rows(const int* __restrict__ slot_ids, int block_m, int64_t numel,
                               int* rows, int* warp_counts) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  int id = -1;
  if (tid < block_m) id = slot_ids[tid];
  const bool ok = tid < block_m && id >= 0 && (int64_t)id < numel;
  const unsigned bal = __ballot_sync(0xffffffffu, ok);
  if (lane == 0) warp_counts[warp] = __popc(bal);
  __syncthreads();
  int before = 0, total = 0;
  for (int w = 0; w < nwarps; ++w) {
    const int cw = warp_counts[w];
    before += (w < warp) ? cw : 0;
    total += cw;
  }
  if (ok) rows[before + __popc(bal & lanemask_lt())] = id;
  __syncthreads();
  return total;
}

}  // namespace mol
