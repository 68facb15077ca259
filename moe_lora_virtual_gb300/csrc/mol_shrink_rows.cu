// LoRA shrink for routed blocks that hold many rows (sm_103a).
//
// fork PR #24 "Root cause" commit: the shrink is a grouped GEMM over the
// virtual experts with N = S*r and K = the input width; code-review commit:
// weights laid out [E, N, K]. For every routed block t of virtual expert v:
//   inter[i, j] = sum_k x[i / x_div, k] * lora_a[v, j, k],   j < R.
//
// When a routed block holds many rows (expert-parallel prefill: about eight
// real pairs per virtual expert), the shrink that streams (block, 8 lora_a
// rows) items copies the block's activation rows again for every 8-row job,
// and those rows take half of every stage: the HBM bytes in flight per SM
// halve and the jobs no longer fit a stage whole. Here each block of the grid
// (one per SM) walks routed blocks t = b, b + G, ...; it copies a block's
// activation rows (tiles of 16 rows, or 8 when K > 1024; one bulk copy per
// row) once into one of two resident 32 KB buffers, and streams only lora_a
// through a ring of four 32 KB stages: the rows of several 8-row groups at
// once when K is small, one bulk copy per stage since a virtual expert's rows
// are adjacent in memory. While the consumers work on one tile the producer
// fills the other buffer and the free stages with the next tile's rows and
// weights. A block with more rows than a tile streams its weights once per
// tile (the later passes mostly from L2).
//
// Roles (160 threads): warp 4 produces (routing words, row compaction, every
// bulk copy, stage headers); warps 0-3 consume (mma.sync m16n8k16, each warp a
// quarter of the k range, partial sums added in a fixed order: the same
// arithmetic as the item shrink, so the two give bit-identical results on the
// same rows). Every wait is bounded; a timeout records a fault bit, lets the
// issued copies land (bounded) and leaves.

#include <algorithm>

#include "mol_device.cuh"
#include "mol_internal.h"

namespace mol {

__device__ unsigned int g_rows_fault_flags;

cudaError_t take_rows_faults(unsigned* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_rows_fault_flags, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_rows_fault_flags, &zero, sizeof(unsigned));
}

namespace xr {
constexpr int kConsumers = 4;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kJT = 8;                      // lora_a rows per group (one n8 mma tile)
constexpr int kXR = 16;                     // most activation rows per tile (one m16 mma tile)
constexpr int kMaxK = 2048;
constexpr int kMaxJ = 4;                    // groups per stage
constexpr int kStageBytes = 32 * 1024;
constexpr int kStages = 4;
constexpr int kXBytes = 32 * 1024;          // one activation buffer: 16 rows to K = 1024, else 8
constexpr int kHeader = 1024;
constexpr size_t kSmem = kHeader + (size_t)kStages * kStageBytes + 2 * (size_t)kXBytes;
constexpr uint32_t kPolls = 1u << 22;
struct Hdr {
  int jt0;   // first 8-row group of the stage; -1 = end of work
  int nj;    // groups in the stage
  int cm;    // rows of the tile
  int m0;    // first compacted row of the tile
  int first; // first stage of the tile (wait for its activation buffer)
  int last;  // last stage of the tile (release its activation buffer)
};
static_assert(2 * (2 * kStages + 4) * 8 + kStages * (int)sizeof(Hdr) <= kHeader, "header");
}  // namespace xr

// Groups per stage and rows per activation tile for a contraction width K.
static inline int rows_groups(int K, int R) {
  return std::max(1, std::min({xr::kMaxJ, xr::kStageBytes / (xr::kJT * K * 2), R / xr::kJT}));
}
static inline int rows_tile(int K) { return xr::kXR * K * 2 <= xr::kXBytes ? xr::kXR : 8; }

__global__ void __launch_bounds__(xr::kThreads, 1)
lora_shrink_rows_kernel(const uint16_t* __restrict__ x, int64_t x_stride, int x_div, int K,
                        const uint16_t* __restrict__ lora_a, int R,
                        const int* __restrict__ sorted_ids, const int* __restrict__ expert_ids,
                        const int* __restrict__ ntpp_ptr, int block_m, int64_t numel,
                        int num_vexperts, float* __restrict__ inter, int64_t nblk, int J,
                        int TR, int early) {
  using namespace xr;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kStages;
  uint64_t* xfull = empty + kStages;
  uint64_t* xempty = xfull + 2;
  Hdr* hdr = reinterpret_cast<Hdr*>(smem + 2 * (2 * kStages + 4) * 8);
  unsigned char* stages = smem + kHeader;
  unsigned char* xbuf = stages + (size_t)kStages * kStageBytes;
  __shared__ float red[kConsumers - 1][kMaxJ][4][32];
  __shared__ int prow[128];  // producer: compacted rows of the current block
  __shared__ int trow[2][kXR];  // pair ids of the rows in each activation buffer

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kConsumers);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&xfull[b], 1);
      mbar_init(&xempty[b], kConsumers);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int xpitch = K * 2;

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    // With `early` the routing and the weights are older than the kernel
    // before this one and are read before griddepcontrol.wait; the
    // activations, after it.
    bool waited = !early;
    if (!early) {
      pdl_wait();
      pdl_launch_dependents();
    }
    const int ntpp = __ldg(ntpp_ptr);
    const int njt = R / kJT;
    uint32_t q = 0;   // stage uses issued
    uint32_t nt = 0;  // tiles issued
    bool fault = false;
    auto wait_free = [&](uint64_t* bar, uint32_t use) -> bool {  // bounded, lane 0 waits
      bool ok = true;
      if (lane == 0) ok = mbar_wait(bar, ((use) & 1) ^ 1, kPolls);
      return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    };
    for (int64_t t = blockIdx.x; t < nblk && !fault; t += gridDim.x) {
      if (t * block_m >= ntpp) break;  // blocks are in order: the rest are padding
      const int e = __ldg(expert_ids + t);
      if (e < 0 || e >= num_vexperts) continue;
      int c = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = u * 32 + lane;
        const int sl = idx < block_m ? __ldg(sorted_ids + t * block_m + idx) : -1;
        const bool ok = sl >= 0 && (int64_t)sl < numel;
        const unsigned bal = __ballot_sync(0xffffffffu, ok);
        if (ok) prow[c + __popc(bal & lanemask_lt())] = sl;
        c += __popc(bal);
      }
      __syncwarp();
      const uint16_t* wv = lora_a + (int64_t)e * R * K;
      for (int m0 = 0; m0 < c && !fault; m0 += TR, ++nt) {
        const int cm = min(TR, c - m0);
        const int xb = (int)(nt & 1);
        if (!wait_free(&xempty[xb], nt >> 1)) {
          fault = true;
          break;
        }
        if (lane < cm) trow[xb][lane] = prow[m0 + lane];
        __syncwarp();
        if (!waited) {
          pdl_wait();
          pdl_launch_dependents();
          waited = true;
        }
        if (lane == 0) mbar_arrive_expect_tx(&xfull[xb], (uint32_t)(cm * xpitch));
        __syncwarp();
        if (lane < cm)
          bulk_g2s(xbuf + (size_t)xb * kXBytes + lane * xpitch,
                   x + (int64_t)(prow[m0 + lane] / x_div) * x_stride, (uint32_t)xpitch, &xfull[xb]);
        for (int jt0 = 0; jt0 < njt; jt0 += J) {
          const int nj = min(J, njt - jt0);
          const int st = (int)(q % kStages);
          if (!wait_free(&empty[st], q / kStages)) {
            fault = true;
            break;
          }
          if (lane == 0) {
            hdr[st] = Hdr{jt0, nj, cm, m0, jt0 == 0 ? 1 : 0, jt0 + nj >= njt ? 1 : 0};
            const uint32_t bytes = (uint32_t)(nj * kJT * xpitch);
            mbar_arrive_expect_tx(&full[st], bytes);
            bulk_g2s(stages + (size_t)st * kStageBytes, wv + (int64_t)jt0 * kJT * K, bytes,
                     &full[st]);
          }
          ++q;
        }
      }
    }
    if (!waited) {
      pdl_wait();
      pdl_launch_dependents();
    }
    if (!fault) {
      const int st = (int)(q % kStages);
      if (wait_free(&empty[st], q / kStages)) {
        if (lane == 0) {
          hdr[st].jt0 = -1;
          mbar_arrive(&full[st]);
        }
      } else {
        fault = true;
      }
    }
    if (fault && lane == 0) {
      atomicOr(&g_rows_fault_flags, kFaultBulkTimeout);
      // let the copies already issued land before the block's shared memory goes
      for (uint32_t u = q > (uint32_t)kStages ? q - kStages : 0; u < q; ++u)
        mbar_wait(&full[u % kStages], (u / kStages) & 1, kPolls);
      for (uint32_t u = nt > 2u ? nt - 2 : 0; u < nt; ++u)
        mbar_wait(&xfull[u & 1], (u >> 1) & 1, kPolls);
    }
    __syncwarp();
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();  // they store the intermediate
  pdl_launch_dependents();
  const int g = lane >> 2, tq = lane & 3;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  uint32_t nt = 0;  // tiles started
  const int nkb = (K + 31) >> 5;
  const int kb0 = warp * nkb / kConsumers, kb1 = (warp + 1) * nkb / kConsumers;
  for (uint32_t q = 0;; ++q) {
    const int st = (int)(q % kStages);
    if (!mbar_wait(&full[st], (q / kStages) & 1, kPolls)) {
      if (lane == 0) atomicOr(&g_rows_fault_flags, kFaultBulkTimeout);
      return;
    }
    const Hdr h = hdr[st];
    if (h.jt0 < 0) break;
    const int xb = (int)(nt & 1);
    if (h.first) {
      if (!mbar_wait(&xfull[xb], (nt >> 1) & 1, kPolls)) {
        if (lane == 0) atomicOr(&g_rows_fault_flags, kFaultBulkTimeout);
        return;
      }
    }
    const unsigned char* W = stages + (size_t)st * kStageBytes;
    const unsigned char* X = xbuf + (size_t)xb * kXBytes;
    const int cm = h.cm, nj = h.nj;
    float acc[kMaxJ][4], acc2[kMaxJ][4];
#pragma unroll
    for (int j = 0; j < kMaxJ; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = acc2[j][e] = 0.f;
#pragma unroll 2
    for (int kb = kb0; kb < kb1; kb += 2) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int kk = (kb + hh) * 32 + 8 * tq;
        const bool kin = kb + hh < kb1 && kk < K;
        const uint4 xa = (kin && g < cm) ? lds16(X + g * xpitch + kk * 2) : zero;
        const uint4 xv = (kin && g + 8 < cm) ? lds16(X + (g + 8) * xpitch + kk * 2) : zero;
#pragma unroll
        for (int j = 0; j < kMaxJ; ++j) {
          if (j >= nj) break;
          const uint4 a = kin ? lds16(W + (j * kJT + g) * xpitch + kk * 2) : zero;
          // k step 0 <- elements 8t..8t+3, k step 1 <- 8t+4..8t+7 (same map in both operands)
          if (hh == 0) {
            mma_16816(acc[j], xa.x, xv.x, xa.y, xv.y, a.x, a.y);
            mma_16816(acc[j], xa.z, xv.z, xa.w, xv.w, a.z, a.w);
          } else {
            mma_16816(acc2[j], xa.x, xv.x, xa.y, xv.y, a.x, a.y);
            mma_16816(acc2[j], xa.z, xv.z, xa.w, xv.w, a.z, a.w);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    // add the four warps' partial sums in a fixed order, store
#pragma unroll
    for (int j = 0; j < kMaxJ; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] += acc2[j][e];
    if (warp > 0) {
#pragma unroll
      for (int j = 0; j < kMaxJ; ++j) {
        if (j >= nj) break;
#pragma unroll
        for (int e = 0; e < 4; ++e) red[warp - 1][j][e][lane] = acc[j][e];
      }
    }
    named_sync(1, kConsumers * 32);
    if (warp == 0) {
#pragma unroll
      for (int j = 0; j < kMaxJ; ++j) {
        if (j >= nj) break;
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int w = 0; w < kConsumers - 1; ++w) acc[j][e] += red[w][j][e][lane];
        const int col = (h.jt0 + j) * kJT + 2 * tq;
        if (g < cm)
          *reinterpret_cast<float2*>(inter + (int64_t)trow[xb][g] * R + col) =
              make_float2(acc[j][0], acc[j][1]);
        if (g + 8 < cm)
          *reinterpret_cast<float2*>(inter + (int64_t)trow[xb][g + 8] * R + col) =
              make_float2(acc[j][2], acc[j][3]);
      }
    }
    named_sync(1, kConsumers * 32);
    if (h.last) {
      if (lane == 0) mbar_arrive(&xempty[xb]);
      ++nt;
    }
  }
}

// --- host side ----------------------------------------------------------------

bool shrink_rows_fits(int64_t numel, int num_vexperts, int R, int K, int block_m,
                      bool adapter_ranks) {
  if (adapter_ranks || numel <= 0 || K > xr::kMaxK || R % xr::kJT != 0) return false;
  if (block_m < 32) return false;
  // many rows per virtual expert: on average at least four pairs each
  return numel >= 4 * std::min<int64_t>(numel, num_vexperts);
}

cudaError_t prepare_rows_kernels() {
  return cudaFuncSetAttribute(lora_shrink_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)xr::kSmem);
}

cudaError_t launch_shrink_rows(const void* x, int64_t x_stride, int x_div, int K,
                               const void* lora_a, int R, const int32_t* sorted_ids,
                               const int32_t* expert_ids, const int32_t* ntpp, int64_t capacity,
                               int block_m, int64_t numel, int num_vexperts, float* inter,
                               bool early, cudaStream_t stream) {
  const int64_t nblk = capacity / block_m;
  if (numel == 0 || nblk == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)std::min<int64_t>(nblk, sms));
  return launch_pdl(lora_shrink_rows_kernel, grid, dim3(xr::kThreads), xr::kSmem, stream,
                    static_cast<const uint16_t*>(x), x_stride, x_div, K,
                    static_cast<const uint16_t*>(lora_a), R, sorted_ids, expert_ids, ntpp, block_m,
                    numel, num_vexperts, inter, nblk, rows_groups(K, R), rows_tile(K),
                    early ? 1 : 0);
}

}  // namespace mol
