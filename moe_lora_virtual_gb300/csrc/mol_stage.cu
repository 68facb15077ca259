// One LoRA stage fused into one launch: shrink then expand per routed block (sm_103a).
//
// fork PR #24 PR body "Background (measured attribution)": a MoE layer runs
// five fused_moe_kernel launches, three of them MoL, and the MoL stages pay
// for their launch structure rather than for their bytes. With the shrink and
// the expand as separate launches every stage boundary costs a routing round
// trip, a pipeline ramp and a drain, and the expand's weight stream cannot
// start before the whole shrink grid has finished.
//
// Here one thread block takes one routed block of the routing -- one virtual
// expert v and the block's real pairs -- and runs the whole stage for it:
//   inter[i, j]      = sum_k x[i / x_div, k] * lora_a[v, j, k]                    (j < R)
//   out[i, s*Ns + n] = bf16_rn(out + scale * w_i * sum_j inter[i, s*r + j] * lora_b[v, s*Ns + n, j])
// (fork PR #24 "Root cause" commit: the shrink is a grouped GEMM over the
// virtual experts with N = S*r; code-review commit: weights laid out [E, N, K];
// "Fix": the expand's weight view is [E, N, K] with K = r.)
// The intermediate of the block's rows stays in shared memory between the two
// halves (it is also stored, as the call's contract asks). The weight stream
// runs on without a break: the producer warp streams the lora_a jobs, then the
// lora_b tiles with the output rows they update, through the same ring of
// stages, while the consumer warps are still on the shrink. A stage that
// reuses a routing (the down stage) reads the routing and issues its first
// weight copies before griddepcontrol.wait, so its blocks stream weights while
// the previous stage drains.
//
// Two blocks share an SM up to R = 64 (2 x 111 KB of shared memory).
// Roles (160 threads): warp 4 is the producer -- routing words, row
// compaction, every bulk copy (cp.async.bulk) and the stage headers. Warps 0-3
// consume: shrink chunks on mma.sync m16n8k16 (each warp a quarter of the
// chunk's k range, partial sums added in a fixed order), then expand tiles
// (each warp 64 of the tile's 256 output columns, the intermediate split into
// bf16 head and tail as in the separate expand). Rows are taken in tiles of
// 16 (one m16 tile); a block with more real rows repeats the stage per tile.
// Every wait is bounded; a timeout records a fault bit and the block leaves.

#include <algorithm>

#include "mol_device.cuh"
#include "mol_internal.h"

namespace mol {

__device__ unsigned int g_stage_fault_flags;

cudaError_t take_stage_checks(unsigned long long* first, unsigned long long* count) {
  CheckRecord r;
  const cudaError_t e = take_check_record_here(&r);
  *first = r.first;
  *count = r.count;
  return e;
}

cudaError_t take_stage_faults(unsigned* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_stage_fault_flags, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_stage_fault_flags, &zero, sizeof(unsigned));
}

namespace fs {
constexpr int kConsumers = 4;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kJT = 8;                 // lora_a rows per shrink job (one n8 mma tile)
constexpr int kMR = 16;                // pair rows per row tile (one m16 mma tile)
// The shrink's stage size: jobs are cut along k exactly as in the separate
// shrink, so both give bit-identical intermediates.
constexpr int kStageBytes = 52 * 1024;
constexpr int kStages = 2;
constexpr int kHeader = 1024;          // barriers and stage headers
constexpr int kCols = 256;             // output columns per expand tile
constexpr int kOutPitch = kCols * 2 + 64;  // bytes between staged output rows (bank skew)
constexpr uint32_t kPolls = 1u << 22;
struct Hdr {
  int kind;   // 0 shrink chunk, 1 expand tile, -1 end of work
  int m0;     // first compacted row of the row tile
  int cm;     // rows in the row tile
  int a;      // shrink: 8-row group jt;   expand: slice s
  int k0;     // shrink: first k;          expand: first output column of the slice
  int len;    // shrink: k values;         expand: output columns
  int pitch;  // shrink: bytes between staged rows
};
static_assert(2 * kStages * 8 + kStages * (int)sizeof(Hdr) <= kHeader, "header");
constexpr size_t smem_bytes(int R) { return kHeader + (size_t)kStages * kStageBytes + (size_t)kMR * (R + 4) * 4; }

// k chunk of a shrink job with cm activation rows: all of K with unpadded rows
// when that fits a stage, else equal chunks (multiples of 64) of rows padded by
// 64 bytes.
MOL_DEV void chunk(int K, int cm, int& len, int& pitch) {
  const int rows = kJT + cm;
  if (rows * K * 2 <= kStageBytes) {
    len = K;
    pitch = K * 2;
    return;
  }
  const int lmax = (kStageBytes / rows - 64) / 2 / 64 * 64;
  const int n = (K + lmax - 1) / lmax;
  len = ((K + n - 1) / n + 63) / 64 * 64;
  pitch = len * 2 + 64;
}
}  // namespace fs

template <int RK, bool EARLY>
__global__ void __launch_bounds__(fs::kThreads, 2)
lora_stage_kernel(const uint16_t* __restrict__ x, int64_t x_stride, int x_div, int K,
                  const uint16_t* __restrict__ lora_a, int R, const uint16_t* __restrict__ lora_b,
                  int S, int Ns, float scale, const float* __restrict__ topk_w,
                  const int* __restrict__ sorted_ids, const int* __restrict__ expert_ids,
                  const int* __restrict__ ntpp_ptr, int block_m, int64_t numel, int num_vexperts,
                  float* __restrict__ inter, uint16_t* __restrict__ out, int64_t out_stride) {
  using namespace fs;
  static_assert(RK == 8 || RK == 16 || RK == 32 || RK == 64, "fused stage: rank 8, 16, 32 or 64");
  constexpr bool K16 = (RK <= 16);
  constexpr int KB = K16 ? 1 : RK / 32;  // expand k blocks (32 wide, or one 16-wide block)
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kStages;
  Hdr* hdr = reinterpret_cast<Hdr*>(smem + 2 * kStages * 8);
  unsigned char* stages = smem + kHeader;
  float* inter_s = reinterpret_cast<float*>(stages + (size_t)kStages * kStageBytes);  // [kMR][R + 4]
  const int ipitch = R + 4;
  __shared__ float red[kConsumers - 1][4][32];
  __shared__ int prow[128];  // the block's real pair ids, in slot order

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kConsumers);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    // Routing words and (EARLY: the routing is older than the kernel before
    // this one) the first weight copies go out before griddepcontrol.wait;
    // activations and output rows, which that kernel may write, after it.
    bool waited = !EARLY;
    if (!EARLY) {
      pdl_wait();
      pdl_launch_dependents();
    }
    const int t = blockIdx.x;
    const int ntpp = __ldg(ntpp_ptr);
    const int e = __ldg(expert_ids + t);
    int sl[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = u * 32 + lane;
      sl[u] = idx < block_m ? __ldg(sorted_ids + (int64_t)t * block_m + idx) : -1;
    }
    const int v = ((int64_t)t * block_m < ntpp && e >= 0 && e < num_vexperts) ? e : -1;
    if (kChecked) {  // the caller's routing words
      if (lane == 0) {
        (void)MOL_NOTE(ntpp >= 0 && ntpp <= (int64_t)gridDim.x * block_m && ntpp % block_m == 0,
                       MOL_CHECK_ROUTE_NTPP, ntpp);
        if ((int64_t)t * block_m < ntpp)
          (void)MOL_NOTE(e >= -1 && e < num_vexperts, MOL_CHECK_ROUTE_EXPERT, t);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v >= 0 && u * 32 + lane < block_m)
          (void)MOL_NOTE(sl[u] >= 0 && (int64_t)sl[u] <= numel, MOL_CHECK_ROUTE_PAIR,
                         (int64_t)t * block_m + u * 32 + lane);
    }
    int c = 0;
    if (v >= 0) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool ok = sl[u] >= 0 && (int64_t)sl[u] < numel;
        const unsigned bal = __ballot_sync(0xffffffffu, ok);
        if (ok) prow[c + __popc(bal & lanemask_lt())] = sl[u];
        c += __popc(bal);
      }
    }
    __syncwarp();
    uint32_t q = 0;
    bool fault = false;
    auto acquire = [&](int& st) -> bool {  // wait until stage use q is free
      st = (int)(q % kStages);
      const uint32_t ph = (q / kStages) & 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&empty[st], ph ^ 1, kPolls);
      return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    };
    const int njt = R / kJT;
    bool stop = false;  // checked build: a failed check ends the block's work
    for (int m0 = 0; m0 < c && !fault && !stop; m0 += kMR) {
      const int cm = min(kMR, c - m0);
      const uint16_t* xsrc =
          (lane >= 16 && lane - 16 < cm) ? x + (int64_t)(prow[m0 + lane - 16] / x_div) * x_stride
                                         : nullptr;
      int len, pitch;
      chunk(K, cm, len, pitch);
      const bool whole = (len == K && pitch == K * 2);
      if (kChecked) {  // the tile's rows fit a stage and the intermediate tile; x rows exist
        const int xr = lane >= 16 && lane - 16 < cm ? prow[m0 + lane - 16] / x_div : 0;
        const bool ok =
            (lane != 0 ||
             (MOL_CHECK((kJT + cm) * pitch <= kStageBytes && pitch >= 2 * min(len, K),
                        MOL_CHECK_SMEM, (kJT + cm) * pitch) &&
              MOL_CHECK(R <= 128 && R % kJT == 0, MOL_CHECK_SMEM, kMR * (R + 4) * 4))) &&
            MOL_CHECK(xr >= 0 && (int64_t)xr < (numel + x_div - 1) / x_div, MOL_CHECK_ROW, xr);
        stop = !__all_sync(0xffffffffu, ok);
        if (stop) break;
      }
      // shrink: 8 lora_a rows (and the tile's activation rows) per stage
      for (int jt = 0; jt < njt && !fault && !stop; ++jt) {
        if (kChecked) {
          const int64_t wr = (int64_t)v * R + jt * kJT;
          stop = !__all_sync(0xffffffffu, lane != 0 || MOL_CHECK(wr + kJT <= (int64_t)num_vexperts * R,
                                                                 MOL_CHECK_WEIGHT_ROW, wr));
          if (stop) break;
        }
        const uint16_t* wrows = lora_a + ((int64_t)v * R + jt * kJT) * K;
        for (int k0 = 0; k0 < K; k0 += len) {
          int st;
          if (!acquire(st)) {
            fault = true;
            break;
          }
          const int cl = min(len, K - k0);
          unsigned char* base = stages + (size_t)st * kStageBytes;
          if (lane == 0) {
            hdr[st] = Hdr{0, m0, cm, jt, k0, cl, pitch};
            mbar_arrive_expect_tx(&full[st], (uint32_t)((kJT + cm) * cl * 2));
          }
          __syncwarp();
          if (whole) {
            if (lane == 0) bulk_g2s(base, wrows, kJT * K * 2, &full[st]);
          } else if (lane < kJT) {
            bulk_g2s(base + lane * pitch, wrows + (int64_t)lane * K + k0, cl * 2, &full[st]);
          }
          if (!waited) {
            pdl_wait();
            pdl_launch_dependents();
            waited = true;
          }
          if (xsrc) bulk_g2s(base + (kJT + lane - 16) * pitch, xsrc + k0, cl * 2, &full[st]);
          ++q;
        }
      }
      // expand: per slice, 256 output columns of lora_b and the rows they update
      for (int s = 0; s < S && !fault && !stop; ++s) {
        for (int col0 = 0; col0 < Ns; col0 += kCols) {
          const int ncols = min(kCols, Ns - col0);
          if (kChecked) {  // lora_b rows of the tile exist; weights and output rows fit a stage
            const int64_t wr = ((int64_t)v * S + s) * Ns + col0;
            const bool ok =
                lane != 0 ||
                (MOL_CHECK(wr + ncols <= (int64_t)num_vexperts * S * Ns, MOL_CHECK_WEIGHT_ROW, wr) &&
                 MOL_CHECK(ncols * RK * 2 + (cm - 1) * kOutPitch + ncols * 2 <= kStageBytes,
                           MOL_CHECK_SMEM, ncols * RK * 2 + cm * kOutPitch));
            stop = !__all_sync(0xffffffffu, ok);
            if (stop) break;
          }
          int st;
          if (!acquire(st)) {
            fault = true;
            break;
          }
          unsigned char* base = stages + (size_t)st * kStageBytes;
          const uint32_t wbytes = (uint32_t)ncols * RK * 2;
          if (lane == 0) {
            hdr[st] = Hdr{1, m0, cm, s, col0, ncols, 0};
            mbar_arrive_expect_tx(&full[st], wbytes + (uint32_t)(cm * ncols * 2));
            bulk_g2s(base, lora_b + (((int64_t)v * S + s) * Ns + col0) * RK, wbytes, &full[st]);
          }
          if (lane < cm)
            bulk_g2s(base + wbytes + lane * kOutPitch,
                     out + (int64_t)prow[m0 + lane] * out_stride + (int64_t)s * Ns + col0,
                     (uint32_t)ncols * 2, &full[st]);
          ++q;
        }
      }
    }
    if (!waited) {
      pdl_wait();
      pdl_launch_dependents();
    }
    if (!fault) {
      int st;
      if (acquire(st)) {
        if (lane == 0) {
          hdr[st].kind = -1;
          mbar_arrive(&full[st]);
        }
      } else {
        fault = true;
      }
    }
    if (fault && lane == 0) {
      atomicOr(&g_stage_fault_flags, kFaultBulkTimeout);
      // the last uses of each stage: let their copies land before the block exits
      for (uint32_t u = q > (uint32_t)kStages ? q - kStages : 0; u < q; ++u)
        mbar_wait(&full[u % kStages], (u / kStages) & 1, kPolls);
    }
    __syncwarp();
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();  // they write the intermediate and the output
  pdl_launch_dependents();
  const int g = lane >> 2, tq = lane & 3;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  const float4 zf = make_float4(0.f, 0.f, 0.f, 0.f);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float acc2[4] = {0.f, 0.f, 0.f, 0.f};
  for (uint32_t q = 0;; ++q) {
    const int st = (int)(q % kStages);
    if (!mbar_wait(&full[st], (q / kStages) & 1, kPolls)) {
      if (lane == 0) atomicOr(&g_stage_fault_flags, kFaultBulkTimeout);
      return;
    }
    const Hdr h = hdr[st];
    if (h.kind < 0) break;
    const unsigned char* W = stages + (size_t)st * kStageBytes;
    const int cm = h.cm, m0 = h.m0;
    if (h.kind == 0) {
      // ---- shrink chunk: rows of the tile x 8 lora_a rows over k in [k0, k0 + len)
      const int k0 = h.k0, len = h.len, pitch = h.pitch;
      if (k0 == 0) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = acc2[e] = 0.f;
      }
      const unsigned char* X = W + kJT * pitch;
      const int nkb = (len + 31) >> 5;
      const int kb0 = warp * nkb / kConsumers, kb1 = (warp + 1) * nkb / kConsumers;
#pragma unroll 2
      for (int kb = kb0; kb < kb1; kb += 2) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int kk = (kb + hh) * 32 + 8 * tq;
          const bool kin = kb + hh < kb1 && kk < len;
          const uint4 xa = (kin && g < cm) ? lds16(X + g * pitch + kk * 2) : zero;
          const uint4 xb = (kin && g + 8 < cm) ? lds16(X + (g + 8) * pitch + kk * 2) : zero;
          const uint4 a = kin ? lds16(W + g * pitch + kk * 2) : zero;
          // k step 0 <- elements 8t..8t+3, k step 1 <- 8t+4..8t+7 (same map in both operands)
          if (hh == 0) {
            mma_16816(acc, xa.x, xb.x, xa.y, xb.y, a.x, a.y);
            mma_16816(acc, xa.z, xb.z, xa.w, xb.w, a.z, a.w);
          } else {
            mma_16816(acc2, xa.x, xb.x, xa.y, xb.y, a.x, a.y);
            mma_16816(acc2, xa.z, xb.z, xa.w, xb.w, a.z, a.w);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (k0 + len >= K) {  // last chunk of the job: add the four partials, store
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] += acc2[e];
        if (warp > 0) {
#pragma unroll
          for (int e = 0; e < 4; ++e) red[warp - 1][e][lane] = acc[e];
        }
        named_sync(1, kConsumers * 32);
        if (warp == 0) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int w = 0; w < kConsumers - 1; ++w) acc[e] += red[w][e][lane];
          const int col = h.a * kJT + 2 * tq;
          const bool cok = MOL_CHECK(col + 2 <= R, MOL_CHECK_COLUMN, col);
          if (g < cm && cok &&
              MOL_CHECK((int64_t)prow[m0 + g] < numel, MOL_CHECK_ROW, prow[m0 + g])) {
            const float2 v2 = make_float2(acc[0], acc[1]);
            *reinterpret_cast<float2*>(inter + (int64_t)prow[m0 + g] * R + col) = v2;
            *reinterpret_cast<float2*>(inter_s + g * ipitch + col) = v2;
          }
          if (g + 8 < cm && cok &&
              MOL_CHECK((int64_t)prow[m0 + g + 8] < numel, MOL_CHECK_ROW, prow[m0 + g + 8])) {
            const float2 v2 = make_float2(acc[2], acc[3]);
            *reinterpret_cast<float2*>(inter + (int64_t)prow[m0 + g + 8] * R + col) = v2;
            *reinterpret_cast<float2*>(inter_s + (g + 8) * ipitch + col) = v2;
          }
        }
        named_sync(1, kConsumers * 32);  // the tile's intermediate in shared memory is complete
      }
      continue;
    }
    // ---- expand tile: slice s, output columns [col0, col0 + ncols) of the slice
    const int s = h.a, col0 = h.k0, ncols = h.len;
    const uint16_t* wsm = reinterpret_cast<const uint16_t*>(W);           // [ncols][RK]
    const unsigned char* osm = W + (size_t)ncols * RK * 2;               // [cm][kOutPitch]
    const bool kq = RK != 8 || tq < 2;  // rank 8: quads 2 and 3 hold k columns 8..15 (zero)
    const int i0 = g < cm ? prow[m0 + g] : -1;
    const int i1 = g + 8 < cm ? prow[m0 + g + 8] : -1;
    // intermediate fragments of rows g and g + 8, split into bf16 head and tail
    uint32_t hf[KB][8], lf[KB][8];
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) {
      const int j = s * RK + (K16 ? 4 * tq : kb * 32 + 8 * tq);
      const float* p0 = inter_s + g * ipitch + j;
      const float* p1 = inter_s + (g + 8) * ipitch + j;
      const float4 a0 = (kq && i0 >= 0) ? *reinterpret_cast<const float4*>(p0) : zf;
      const float4 a1 = (kq && i1 >= 0) ? *reinterpret_cast<const float4*>(p1) : zf;
      split_bf16x2(a0.x, a0.y, hf[kb][0], lf[kb][0]);
      split_bf16x2(a1.x, a1.y, hf[kb][1], lf[kb][1]);
      split_bf16x2(a0.z, a0.w, hf[kb][2], lf[kb][2]);
      split_bf16x2(a1.z, a1.w, hf[kb][3], lf[kb][3]);
      if constexpr (!K16) {
        const float4 b0 = i0 >= 0 ? *reinterpret_cast<const float4*>(p0 + 4) : zf;
        const float4 b1 = i1 >= 0 ? *reinterpret_cast<const float4*>(p1 + 4) : zf;
        split_bf16x2(b0.x, b0.y, hf[kb][4], lf[kb][4]);
        split_bf16x2(b1.x, b1.y, hf[kb][5], lf[kb][5]);
        split_bf16x2(b0.z, b0.w, hf[kb][6], lf[kb][6]);
        split_bf16x2(b1.z, b1.w, hf[kb][7], lf[kb][7]);
      }
    }
    const float sw0 = i0 >= 0 ? (topk_w ? scale * __ldg(topk_w + i0) : scale) : 0.f;
    const float sw1 = i1 >= 0 ? (topk_w ? scale * __ldg(topk_w + i1) : scale) : 0.f;
#pragma unroll
    for (int cg = 0; cg < 2; ++cg) {
      const int nb = warp * 64 + cg * 32;  // the group's first column inside the tile
      if (nb >= ncols) break;              // warp-uniform
      float d[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) d[u][0] = d[u][1] = d[u][2] = d[u][3] = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        // weight row of output column nb + 8*(g/2) + 2u + (g%2): thread tq ends with
        // columns nb + 8tq .. nb + 8tq + 7
        const int wr = nb + 8 * (g >> 1) + 2 * u + (g & 1);
        const bool bv = wr < ncols;
        if constexpr (K16) {
          const uint2 q2 = (bv && kq) ? lds8(wsm + wr * RK + 4 * tq) : make_uint2(0, 0);
          mma_16816(d[u], hf[0][0], hf[0][1], hf[0][2], hf[0][3], q2.x, q2.y);
          mma_16816(d[u], lf[0][0], lf[0][1], lf[0][2], lf[0][3], q2.x, q2.y);
        } else {
#pragma unroll
          for (int kb = 0; kb < KB; ++kb) {
            const uint4 w4 = bv ? lds16(wsm + wr * RK + kb * 32 + 8 * tq) : zero;
            mma_16816(d[u], hf[kb][0], hf[kb][1], hf[kb][2], hf[kb][3], w4.x, w4.y);
            mma_16816(d[u], lf[kb][0], lf[kb][1], lf[kb][2], lf[kb][3], w4.x, w4.y);
            mma_16816(d[u], hf[kb][4], hf[kb][5], hf[kb][6], hf[kb][7], w4.z, w4.w);
            mma_16816(d[u], lf[kb][4], lf[kb][5], lf[kb][6], lf[kb][7], w4.z, w4.w);
          }
        }
      }
      if (nb + 8 * tq < ncols) {
        const int64_t oc = (int64_t)s * Ns + col0 + nb + 8 * tq;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i = hh ? i1 : i0;
          if (i < 0) continue;
          if (!MOL_CHECK((int64_t)i < numel, MOL_CHECK_ROW, i) ||
              !MOL_CHECK(oc + 8 <= (int64_t)S * Ns, MOL_CHECK_COLUMN, oc))
            continue;
          const float sw = hh ? sw1 : sw0;
          uint4 ov = lds16(osm + (8 * hh + g) * kOutPitch + (nb + 8 * tq) * 2);
          uint32_t* ow = reinterpret_cast<uint32_t*>(&ov);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float lo = fmaf(sw, d[u][2 * hh], bf16_lo(ow[u]));
            const float hi = fmaf(sw, d[u][2 * hh + 1], bf16_hi(ow[u]));
            ow[u] = pack_bf16x2(lo, hi);
          }
          *reinterpret_cast<uint4*>(out + (int64_t)i * out_stride + oc) = ov;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
}

// --- host side ----------------------------------------------------------------

static int stage_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

bool stage_fused_fits(int64_t numel, int num_vexperts, int R, int r, int K, int N, int block_m,
                      int64_t capacity, bool adapter_arrays) {
  if (adapter_arrays || numel <= 0) return false;
  if (!(r == 8 || r == 16 || r == 32 || r == 64) || R > 128) return false;
  if (shrink_tc_fits(numel, num_vexperts, R, K, block_m)) return false;
  // One block per routed block streams its virtual expert's weights through two
  // stages: that is about one round trip only when every routed block has an SM
  // of its own and a block's weights fill about two stages. Past that the
  // persistent shrink and the separate expand keep more bytes in flight per SM
  // and are faster.
  const int64_t weight_bytes = 2 * ((int64_t)R * K + (int64_t)N * r);
  return capacity / block_m <= stage_sms() && weight_bytes <= 2 * fs::kStageBytes;
}

template <int RK>
static cudaError_t prepare_stage_rk() {
  const int bytes = (int)fs::smem_bytes(128);
  cudaError_t e = cudaFuncSetAttribute(lora_stage_kernel<RK, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(lora_stage_kernel<RK, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t prepare_stage_kernels() {
  cudaError_t e = prepare_stage_rk<8>();
  if (e == cudaSuccess) e = prepare_stage_rk<16>();
  if (e == cudaSuccess) e = prepare_stage_rk<32>();
  if (e == cudaSuccess) e = prepare_stage_rk<64>();
  return e;
}

cudaError_t launch_stage(const void* x, int64_t x_stride, int x_div, int K, const void* lora_a,
                         const void* lora_b, int S, int r, int Ns, float scale,
                         const float* topk_weights, const int32_t* sorted_ids,
                         const int32_t* expert_ids, const int32_t* ntpp, int64_t capacity,
                         int block_m, int64_t numel, int num_vexperts, float* inter, void* out,
                         int64_t out_stride, bool early, cudaStream_t stream) {
  const int64_t nblk = capacity / block_m;
  if (numel == 0 || nblk == 0) return cudaSuccess;
  if (nblk > INT32_MAX) return cudaErrorInvalidConfiguration;
  const int R = S * r;
  const dim3 grid((unsigned)nblk);
  const size_t smem = fs::smem_bytes(R);
  const uint16_t* xp = static_cast<const uint16_t*>(x);
  const uint16_t* a = static_cast<const uint16_t*>(lora_a);
  const uint16_t* b = static_cast<const uint16_t*>(lora_b);
  uint16_t* o = static_cast<uint16_t*>(out);
#define MOL_STAGE(RK, E)                                                                       \
  launch_pdl(lora_stage_kernel<RK, E>, grid, dim3(fs::kThreads), smem, stream, xp, x_stride,   \
             x_div, K, a, R, b, S, Ns, scale, topk_weights, sorted_ids, expert_ids, ntpp,       \
             block_m, numel, num_vexperts, inter, o, out_stride)
  switch (r) {
    case 8:
      return early ? MOL_STAGE(8, true) : MOL_STAGE(8, false);
    case 16:
      return early ? MOL_STAGE(16, true) : MOL_STAGE(16, false);
    case 32:
      return early ? MOL_STAGE(32, true) : MOL_STAGE(32, false);
    case 64:
      return early ? MOL_STAGE(64, true) : MOL_STAGE(64, false);
    default:
      return cudaErrorInvalidValue;
  }
#undef MOL_STAGE
}

}  // namespace mol
