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

constexpr uint32_t kWaitPolls = 1u << 22;  // bounded mbarrier waits

// Faults recorded instead of hanging (see kFaultBulkTimeout).
__device__ unsigned int g_fault_flags;

// Test controls of the shrink's bounded waits, set only through
// mol_debug_wait_test: bit 0 of g_test_stall makes the producer warp leave
// before it issues any copy (so the consumers' waits run out with nothing in
// flight), and g_wait_limit_ns is the wall-clock limit of every wait of the
// shrink. Both are read once per block.
__device__ unsigned int g_test_stall;
__device__ unsigned long long g_wait_limit_ns = kWaitLimitNs;

cudaError_t take_lora_faults(unsigned* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_fault_flags, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_fault_flags, &zero, sizeof(unsigned));
}

cudaError_t set_wait_test(unsigned stall, unsigned long long limit_ns) {
  cudaError_t e = cudaDeviceSynchronize();  // no kernel may be running while they change
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_test_stall, &stall, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_wait_limit_ns, &limit_ns, sizeof(unsigned long long));
  if (e != cudaSuccess) return e;
  return set_expand_tc_wait_test(stall, limit_ns);
}

// Routing words of one work item as loaded: a producer fetches them one item
// ahead and evaluates them only when it reaches the item.
struct Raw {
  int64_t t;  // routed block, -1 past the last item
  int ntpp, e;
  int sl[4];  // slot ids of lanes u * 32 + lane
};

// Shrink: a persistent, warp-specialised TMA pipeline.
//
// Work item = (routed block t, 8 weight rows jt). Block b of the grid (two per
// SM) walks items b, b+G, b+2G, ... . Warp 4 is the producer: it fetches the
// next item's routing (expert id, slot ids) one item ahead, compacts the
// block's real rows with warp ballots, splits them into jobs of at most 16
// rows and streams each job through a ring of two shared-memory stages. A job
// whose 8 weight rows and activation rows fit one stage at the full width K
// takes one stage: the weight rows, adjacent in memory, arrive in ONE bulk
// copy and each activation row in one more. Otherwise the job is cut along k
// into equal chunks, the widest that fit, and every row of a chunk is its own
// copy into a row padded by 64 bytes (the 16-byte fragment reads of a quarter
// warp then fall in distinct banks). Copies stay kilobytes long: one thread
// issuing 1 KB copies cannot keep up with HBM, with 4 KB and more it can. Small
// items (8 rows) keep the blocks' shares of the weight stream even.
// Warps 0-3 consume: they wait for a stage, run the mma over their quarter of
// its k range from shared memory only (two accumulator chains), release the
// stage on its "empty" mbarrier and, after a job's last chunk, add their four
// partial sums in a fixed order and store the job's fp32 rows. Every wait is
// bounded; a timeout records a fault bit and leaves the kernel instead of
// hanging.
namespace sp {
constexpr int kConsumers = 4;                    // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;  // + the producer warp
constexpr int kXR = 16;                          // activation rows per job (one 16-row mma tile)
constexpr int kStageBytes = 52 * 1024;
constexpr int kStages = 2;
constexpr int kBlocksPerSM = 2;                  // two issuing producers per SM
constexpr int kMeta = kStages + 2;               // jobs whose rows a consumer may still read
constexpr int kHeader = 1024;                    // barriers, stage headers, job meta
constexpr size_t kSmem = kHeader + (size_t)kStages * kStageBytes;
struct Job {
  int v, jt, cm, ncols;  // ncols: leading columns of the item inside the adapter's rank
  int rows[kXR];
};
struct StageHdr {
  int job;    // meta slot, -1 = end of work
  int k0;     // first k of the chunk
  int len;    // k values in the chunk
  int pitch;  // bytes between rows in the stage
};
static_assert(2 * kStages * 8 + kStages * (int)sizeof(StageHdr) + kMeta * (int)sizeof(Job) <= kHeader,
              "header");

// k chunk of a job of JT weight rows and cm activation rows: all of K with
// unpadded rows when that fits a stage, else equal chunks (multiples of 64) of
// padded rows.
template <int JT>
MOL_DEV void job_chunk(int K, int cm, int& len, int& pitch) {
  const int rows = JT + cm;
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
}  // namespace sp

// JT: weight rows per item, one (8) or two (16) 8-column mma tiles.
template <bool RANKS, int JT>
__global__ void __launch_bounds__(sp::kThreads, sp::kBlocksPerSM)
lora_shrink_kernel(const uint16_t* __restrict__ x, int64_t x_stride, int x_div, int K,
                   const uint16_t* __restrict__ lora_a, int R, const int* __restrict__ sorted_ids,
                   const int* __restrict__ expert_ids, const int* __restrict__ ntpp_ptr,
                   int block_m, int64_t numel, int num_vexperts, float* __restrict__ inter,
                   int n_jt, int64_t n_items, int early, int r1,
                   const int* __restrict__ lora_ranks, int num_experts, int num_loras,
                   RoutingIds pf) {
  using namespace sp;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kStages;
  StageHdr* hdr = reinterpret_cast<StageHdr*>(smem + 2 * kStages * 8);
  Job* meta = reinterpret_cast<Job*>(smem + 2 * kStages * 8 + kStages * sizeof(StageHdr));
  unsigned char* stages = smem + kHeader;
  __shared__ float red[kConsumers - 1][4][32];
  __shared__ int prow[128];  // producer: compacted rows of the current block
  __shared__ uint16_t s_rank[RANKS ? kMaxLoraTable : 1];  // producer: adapter ranks in [0, r1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kConsumers);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t wlim = g_wait_limit_ns;
  const int64_t G = gridDim.x;
  // L2 prefetch (pf.topk_ids set: this shrink follows the align of the same call,
  // whose caller declared the ids complete before the kernel preceding the call
  // began, so they may be read before any wait). Block b asks L2 for the lora_a
  // rows of the virtual experts v = b + j * G (j < 32) that have pairs, so the
  // weight stream from HBM starts while the align still runs and is spread over
  // every SM's copy engine (one SM's engine alone is far too slow for it).
  if (pf.topk_ids != nullptr && warp == kConsumers) {
    const int b = (int)blockIdx.x;
    unsigned own = 0;
    for (int i = lane; i < pf.numel; i += 32) {
      const int v = remap_one(ld_cg_i32(pf.topk_ids + i), ld_cg_i32(pf.lora_ids + i / pf.topk),
                              pf.num_experts, pf.max_loras);
      if (v >= 0 && v < num_vexperts && v % G == b) own |= 1u << (v / G);
    }
    own = __reduce_or_sync(0xffffffffu, own);
    if ((own >> lane) & 1u)
      prefetch_l2(lora_a + (int64_t)(b + lane * G) * R * K, (int64_t)R * K * 2);
  }
  // The activations may come from the kernel right before this one: only the
  // producer reads global memory, and it reads them after griddepcontrol.wait.
  // With `early` (inside mol_lora_forward, routing reused) routing words and
  // weight rows are older than that kernel and the producer reads them before
  // the wait. Consumers wait before they store.
  if (!early || warp != kConsumers) {
    pdl_wait();
    pdl_launch_dependents();
  }

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    if (g_test_stall & 1u) return;  // test control: nothing is issued, the consumers' waits run out
    uint32_t q = 0;   // stage uses issued
    uint32_t jn = 0;  // jobs issued
    bool waited = !early;
    auto acquire = [&](int& st) -> bool {  // wait until stage q is free
      st = (int)(q % kStages);
      const uint32_t ph = (q / kStages) & 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&empty[st], ph ^ 1, kWaitPolls, wlim);
      return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    };
    auto fetch = [&](int64_t it, Raw& r) {
      r.t = it < n_items ? it / n_jt : -1;
      r.ntpp = 0;
      r.e = -1;
#pragma unroll
      for (int u = 0; u < 4; ++u) r.sl[u] = -1;
      if (r.t < 0) return;
      r.ntpp = __ldg(ntpp_ptr);
      r.e = __ldg(expert_ids + r.t);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = u * 32 + lane;
        if (idx < block_m) r.sl[u] = __ldg(sorted_ids + r.t * block_m + idx);
      }
    };
    Raw nxt;
    int64_t item = blockIdx.x;
    fetch(item, nxt);
    if constexpr (RANKS) {  // per-adapter ranks, read like the weights
      for (int l = lane; l < num_loras; l += 32) {
        const int rk = __ldg(lora_ranks + l);
        s_rank[l] = (uint16_t)(rk < 0 ? 0 : (rk > r1 ? r1 : rk));
      }
      __syncwarp();
    }
    bool fault = false;
    bool stop = false;  // checked build: a failed check ends the block's work
    while (item < n_items && !fault && !stop) {
      const Raw cur_r = nxt;
      const int64_t cur = item;
      item += G;
      fetch(item, nxt);  // next item's routing is in flight while this one streams
      const int jt_c = (int)(cur % n_jt);
      const bool below = cur_r.t * block_m < cur_r.ntpp;
      if (kChecked && jt_c == 0 && lane == 0) {  // the caller's routing words, once per block
        const int64_t cap = n_items / n_jt * block_m;
        (void)MOL_NOTE(cur_r.ntpp >= 0 && cur_r.ntpp <= cap && cur_r.ntpp % block_m == 0,
                       MOL_CHECK_ROUTE_NTPP, cur_r.ntpp);
        if (below)
          (void)MOL_NOTE(cur_r.e >= -1 && cur_r.e < num_vexperts, MOL_CHECK_ROUTE_EXPERT, cur_r.t);
      }
      if (!below) break;  // the block's later items lie further past the routed blocks
      const int v = cur_r.e;
      if (v < 0 || v >= num_vexperts) continue;
      if (kChecked && jt_c == 0) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int idx = u * 32 + lane;
          if (idx < block_m)
            (void)MOL_NOTE(cur_r.sl[u] >= 0 && (int64_t)cur_r.sl[u] <= numel, MOL_CHECK_ROUTE_PAIR,
                           cur_r.t * block_m + idx);
        }
      }
      // Columns of this item inside the adapter's rank: rank 0 writes nothing,
      // an item wholly past the rank writes zeros (its weights are padding).
      int in_rank = JT;  // columns of the item below the rank (r1 % JT == 0 with ranks)
      if constexpr (RANKS) {
        const int rl = (int)s_rank[v / num_experts];
        if (rl == 0) continue;
        in_rank = rl - (jt_c * JT) % r1;
      }
      int c = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int slu = cur_r.sl[u];
        const bool ok = slu >= 0 && (int64_t)slu < numel;
        const unsigned bal = __ballot_sync(0xffffffffu, ok);
        if (ok) prow[c + __popc(bal & lanemask_lt())] = slu;
        c += __popc(bal);
      }
      __syncwarp();
      const int jt = jt_c;
      if (RANKS && in_rank <= 0) {
        if (!waited) {  // the zeros overwrite rows the previous kernel may still read
          pdl_wait();
          pdl_launch_dependents();
          waited = true;
        }
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        constexpr int kQ = JT / 4;  // float4 pieces of the item's columns per row
        for (int q2 = lane; q2 < kQ * c; q2 += 32)
          *reinterpret_cast<float4*>(inter + (int64_t)prow[q2 / kQ] * R + jt * JT + 4 * (q2 % kQ)) = z;
        __syncwarp();
        continue;
      }
      const uint16_t* wrows = lora_a + ((int64_t)v * R + jt * JT) * K;
      if (kChecked) {
        const int64_t wr = (int64_t)v * R + jt * JT;
        stop = !__all_sync(0xffffffffu, lane != 0 || MOL_CHECK(jt * JT + JT <= R && wr + JT <=
                                                                   (int64_t)num_vexperts * R,
                                                               MOL_CHECK_WEIGHT_ROW, wr));
        if (stop) break;
      }
      for (int m0 = 0; m0 < c && !fault; m0 += kXR) {
        const int cm = min(kXR, c - m0);
        int len, pitch;
        job_chunk<JT>(K, cm, len, pitch);
        const bool whole = (len == K && pitch == K * 2);
        if (kChecked) {  // the job's rows fit a stage; its activation rows exist
          const int xr = lane >= 16 && lane - 16 < cm ? prow[m0 + lane - 16] / x_div : 0;
          const bool ok =
              (lane != 0 || MOL_CHECK((JT + cm) * pitch <= kStageBytes && pitch >= 2 * min(len, K),
                                      MOL_CHECK_SMEM, (JT + cm) * pitch)) &&
              MOL_CHECK(xr >= 0 && (int64_t)xr < (numel + x_div - 1) / x_div, MOL_CHECK_ROW, xr);
          stop = !__all_sync(0xffffffffu, ok);
          if (stop) break;
        }
        const int slot = (int)(jn % kMeta);
        Job& jb = meta[slot];
        if (lane == 0) {
          jb.v = v;
          jb.jt = jt;
          jb.cm = cm;
          jb.ncols = in_rank < JT ? in_rank : JT;
        }
        if (lane < cm) jb.rows[lane] = prow[m0 + lane];
        const uint16_t* xsrc =
            (lane >= 16 && lane - 16 < cm) ? x + (int64_t)(prow[m0 + lane - 16] / x_div) * x_stride
                                           : nullptr;
        __syncwarp();
        for (int k0 = 0; k0 < K; k0 += len) {
          int st;
          if (!acquire(st)) {
            fault = true;
            break;
          }
          const int cl = min(len, K - k0);
          unsigned char* base = stages + (size_t)st * kStageBytes;
          if (lane == 0) {
            hdr[st].job = slot;
            hdr[st].k0 = k0;
            hdr[st].len = cl;
            hdr[st].pitch = pitch;
            mbar_arrive_expect_tx(&full[st], (uint32_t)((JT + cm) * cl * 2));
          }
          __syncwarp();
          if (whole) {
            if (lane == 0) bulk_g2s(base, wrows, JT * K * 2, &full[st]);
          } else if (lane < JT) {
            bulk_g2s(base + lane * pitch, wrows + (int64_t)lane * K + k0, cl * 2, &full[st]);
          }
          if (!waited) {  // the weight copy is on its way; activations wait for the producer kernel
            pdl_wait();
            pdl_launch_dependents();
            waited = true;
          }
          if (xsrc)
            bulk_g2s(base + (JT + lane - 16) * pitch, xsrc + k0, cl * 2, &full[st]);
          ++q;
        }
        ++jn;
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
          hdr[st].job = -1;
          mbar_arrive(&full[st]);
        }
      } else {
        fault = true;
      }
    }
    if (fault && lane == 0) {
      atomicOr(&g_fault_flags, kFaultBulkTimeout);
      // Let the copies of the last uses of each stage land (bounded) before the
      // block exits and its shared memory is released: a stage's full barrier
      // completes when its copies have arrived, whether or not anyone reads them.
      for (uint32_t u = q > (uint32_t)kStages ? q - kStages : 0; u < q; ++u)
        mbar_wait(&full[u % kStages], (u / kStages) & 1, kWaitPolls, wlim);
    }
    __syncwarp();
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, tq = lane & 3;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  constexpr int NT = JT / 8;  // 8-column mma tiles per item
  float acc[NT][4] = {};
  float acc2[NT][4] = {};  // odd k blocks: a second, independent mma chain
  for (uint32_t q = 0;; ++q) {
    const int st = (int)(q % kStages);
    if (!mbar_wait(&full[st], (q / kStages) & 1, kWaitPolls, wlim)) {
      if (lane == 0) atomicOr(&g_fault_flags, kFaultBulkTimeout);
      return;
    }
    const int slot = hdr[st].job;
    if (slot < 0) break;
    const int k0 = hdr[st].k0, len = hdr[st].len, pitch = hdr[st].pitch;
    const Job& jb = meta[slot];
    const int cm = jb.cm;
    if (k0 == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = acc2[nt][e] = 0.f;
    }
    const unsigned char* W = stages + (size_t)st * kStageBytes;
    const unsigned char* X = W + JT * pitch;
    const int nkb = (len + 31) >> 5;
    const int kb0 = warp * nkb / kConsumers, kb1 = (warp + 1) * nkb / kConsumers;
#pragma unroll 2
    for (int kb = kb0; kb < kb1; kb += 2) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kk = (kb + h) * 32 + 8 * tq;
        const bool kin = kb + h < kb1 && kk < len;
        const uint4 xa = (kin && g < cm) ? lds16(X + g * pitch + kk * 2) : zero;
        const uint4 xb = (kin && g + 8 < cm) ? lds16(X + (g + 8) * pitch + kk * 2) : zero;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {  // weight row nt * 8 + g
          const uint4 a = kin ? lds16(W + (nt * 8 + g) * pitch + kk * 2) : zero;
          // k step 0 <- elements 8t..8t+3, k step 1 <- 8t+4..8t+7 (same map in both operands)
          if (h == 0) {
            mma_16816(acc[nt], xa.x, xb.x, xa.y, xb.y, a.x, a.y);
            mma_16816(acc[nt], xa.z, xb.z, xa.w, xb.w, a.z, a.w);
          } else {
            mma_16816(acc2[nt], xa.x, xb.x, xa.y, xb.y, a.x, a.y);
            mma_16816(acc2[nt], xa.z, xb.z, xa.w, xb.w, a.z, a.w);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    if (k0 + len >= K) {  // last chunk of the job: add the four partials, store
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {  // one 8-column tile at a time through `red`
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] += acc2[nt][e];
        if (warp > 0) {
#pragma unroll
          for (int e = 0; e < 4; ++e) red[warp - 1][e][lane] = acc[nt][e];
        }
        named_sync(1, kConsumers * 32);
        if (warp == 0) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int w = 0; w < kConsumers - 1; ++w) acc[nt][e] += red[w][e][lane];
          const int cin = nt * 8 + 2 * tq;  // column inside the item
          const int col = jb.jt * JT + cin;
          // columns past the adapter's rank are zero padding: written as 0
          const bool k0v = !RANKS || cin < jb.ncols, k1v = !RANKS || cin + 1 < jb.ncols;
          const bool cok = MOL_CHECK(col >= 0 && col + 2 <= R, MOL_CHECK_COLUMN, col);
          if (g < cm && cok &&
              MOL_CHECK(jb.rows[g] >= 0 && (int64_t)jb.rows[g] < numel, MOL_CHECK_ROW, jb.rows[g]))
            *reinterpret_cast<float2*>(inter + (int64_t)jb.rows[g] * R + col) =
                make_float2(k0v ? acc[nt][0] : 0.f, k1v ? acc[nt][1] : 0.f);
          if (g + 8 < cm && cok &&
              MOL_CHECK(jb.rows[g + 8] >= 0 && (int64_t)jb.rows[g + 8] < numel, MOL_CHECK_ROW,
                        jb.rows[g + 8]))
            *reinterpret_cast<float2*>(inter + (int64_t)jb.rows[g + 8] * R + col) =
                make_float2(k0v ? acc[nt][2] : 0.f, k1v ? acc[nt][3] : 0.f);
        }
        named_sync(1, kConsumers * 32);
      }
    }
  }
}

// Expand with the weight fragments in registers (rank 128; ranks 16-64 take
// the staged expand below). One item = (routed block t, slice s, 128 output
// columns), 4 warps x 32 columns. Three waves of loads: the routing words
// together, then the weight fragments and the output rows to update, then the
// intermediate. With EARLY (inside mol_lora_forward, right after this stage's
// shrink) the first two run before griddepcontrol.wait, overlapping the
// shrink's tail.
constexpr int kExpandThreads = 128;
constexpr int kExpandCols = 128;

// Zeroes the elements of a (columns j .. j+3) at or past column rl.
MOL_DEV void mask_cols(float4& a, int j, int rl) {
  if (j >= rl) a.x = 0.f;
  if (j + 1 >= rl) a.y = 0.f;
  if (j + 2 >= rl) a.z = 0.f;
  if (j + 3 >= rl) a.w = 0.f;
}
// Zeroes the bf16 elements of b (columns j .. j+7, two per word, lower column
// in the low half) at or past column rl.
MOL_DEV void mask_bf16x8(uint4& b, int j, int rl) {
  uint32_t* w = reinterpret_cast<uint32_t*>(&b);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int c = j + 2 * q;
    if (c >= rl) w[q] = 0u;
    else if (c + 1 >= rl) w[q] &= 0xFFFFu;
  }
}

template <int RK, bool EARLY, bool ADAPT>
__global__ void __launch_bounds__(kExpandThreads, RK == 16 ? 9 : RK == 32 ? 8 : RK == 64 ? 5 : 4)
lora_expand_kernel(const float* __restrict__ inter, int R, const uint16_t* __restrict__ lora_b,
                   int S, int Ns, float scale, const float* __restrict__ topk_w,
                   const int* __restrict__ sorted_ids, const int* __restrict__ expert_ids,
                   const int* __restrict__ ntpp_ptr, int block_m, int64_t numel,
                   int num_vexperts, uint16_t* __restrict__ out, int64_t out_stride,
                   int chunks_per_slice, const int* __restrict__ lora_ranks,
                   const float* __restrict__ lora_scalings, int num_experts) {
  constexpr bool K16 = (RK == 16);
  constexpr int KB = K16 ? 1 : RK / 32;  // k blocks (32 wide, or one 16-wide block)
  __shared__ int rows[128];
  __shared__ int wcnt[kExpandThreads / 32];

  const int tid = threadIdx.x;
  const int per_block = S * chunks_per_slice;
  const int t = blockIdx.x / per_block;
  const int rem = blockIdx.x - t * per_block;
  const int s = rem / chunks_per_slice;
  const int chunk = rem - s * chunks_per_slice;
  if (!EARLY) {
    pdl_wait();
    pdl_launch_dependents();
  }
  const int ntpp = __ldg(ntpp_ptr);
  const int v = __ldg(expert_ids + t);
  const int slot = tid < block_m ? __ldg(sorted_ids + (int64_t)t * block_m + tid) : -1;
  if (kChecked && rem == 0)
    note_block_routing(t, ntpp, v, slot, block_m, numel, num_vexperts,
                       (int64_t)(gridDim.x / per_block) * block_m);
  if ((int64_t)t * block_m >= ntpp || v < 0 || v >= num_vexperts) return;
  // the adapter's rank and scaling, loaded with the weights below
  int rk_raw = RK;
  float scl = 1.f;
  if constexpr (ADAPT) {
    if (lora_ranks) rk_raw = __ldg(lora_ranks + v / num_experts);
    if (lora_scalings) scl = __ldg(lora_scalings + v / num_experts);
  }
  // rank 0: the adapter writes no delta; past rank rl the intermediate and
  // the weight columns are padding and take no part in the sum
  const int rl = rk_raw < 0 ? 0 : (rk_raw > RK ? RK : rk_raw);
  const int c = compact_block_rows(slot, numel, rows, wcnt);
  if (c == 0) return;

  const int lane = tid & 31, warp = tid >> 5, g = lane >> 2, tq = lane & 3;
  const int n_base = chunk * kExpandCols + warp * 32;  // column inside the slice
  if (n_base >= Ns) return;                            // warp-uniform; no block sync follows

  // Weight fragments. Lane (g, t) of 8-column tile u holds the weight row of
  // output column n_base + 8*(g/2) + 2u + (g%2), so thread t finishes with
  // columns n_base + 8t .. n_base + 8t + 7 of each row.
  const int grp = n_base + 8 * (g >> 1);
  const bool bvalid = grp < Ns;
  const uint16_t* bw = lora_b + ((int64_t)v * S * Ns + (int64_t)s * Ns + grp + (g & 1)) * RK;
  uint4 bf[KB][4];
#pragma unroll
  for (int kb = 0; kb < KB; ++kb)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      // with ranks, weight columns wholly past rl are not read
      const int j0 = K16 ? 4 * tq : kb * 32 + 8 * tq;
      const bool kin = bvalid && (!ADAPT || j0 < rl);
      if constexpr (K16) {
        const uint2 q = kin ? ld_stream8(bw + 2 * u * RK + 4 * tq) : make_uint2(0, 0);
        bf[kb][u] = make_uint4(q.x, q.y, 0, 0);
      } else {
        bf[kb][u] = kin ? ld_stream16(bw + 2 * u * RK + kb * 32 + 8 * tq) : make_uint4(0, 0, 0, 0);
      }
    }

  const bool ovalid = (n_base + 8 * tq) < Ns;
  const int64_t ocol = (int64_t)s * Ns + n_base + 8 * tq;
  if (kChecked && !MOL_CHECK(s * RK + RK <= R, MOL_CHECK_COLUMN, s * RK)) return;
  const float4 zf = make_float4(0.f, 0.f, 0.f, 0.f);
  const uint4 zu = make_uint4(0, 0, 0, 0);
  // output rows of the first row tile, fetched with the weights
  int i0 = g < c ? rows[g] : -1;
  int i1 = 8 + g < c ? rows[8 + g] : -1;
  uint4 o0 = (ovalid && i0 >= 0) ? *reinterpret_cast<const uint4*>(out + (int64_t)i0 * out_stride + ocol) : zu;
  uint4 o1 = (ovalid && i1 >= 0) ? *reinterpret_cast<const uint4*>(out + (int64_t)i1 * out_stride + ocol) : zu;
  if (EARLY) {
    pdl_wait();  // the intermediate comes from the shrink that precedes this kernel
    pdl_launch_dependents();
  }
  if (ADAPT && rl == 0) return;
  if (ADAPT && rl < RK) {  // the chunk that straddles rl keeps only its columns below rl
#pragma unroll
    for (int kb = 0; kb < KB; ++kb)
#pragma unroll
      for (int u = 0; u < 4; ++u) mask_bf16x8(bf[kb][u], K16 ? 4 * tq : kb * 32 + 8 * tq, rl);
  }
  const float scale_v = ADAPT ? scale * scl : scale;

  for (int m0 = 0; m0 < c; m0 += 16) {
    if (m0 > 0) {
      i0 = m0 + g < c ? rows[m0 + g] : -1;
      i1 = m0 + 8 + g < c ? rows[m0 + 8 + g] : -1;
      o0 = (ovalid && i0 >= 0) ? *reinterpret_cast<const uint4*>(out + (int64_t)i0 * out_stride + ocol) : zu;
      o1 = (ovalid && i1 >= 0) ? *reinterpret_cast<const uint4*>(out + (int64_t)i1 * out_stride + ocol) : zu;
    }
    float acc[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;

#pragma unroll
    for (int kb = 0; kb < KB; ++kb) {
      const int koff = s * RK + (K16 ? 4 * tq : kb * 32 + 8 * tq);
      const float* p0 = inter + (int64_t)(i0 >= 0 ? i0 : 0) * R + koff;
      const float* p1 = inter + (int64_t)(i1 >= 0 ? i1 : 0) * R + koff;
      float4 a0 = i0 >= 0 ? ld_l2_f4(p0) : zf;
      float4 a1 = i1 >= 0 ? ld_l2_f4(p1) : zf;
      float4 b0 = zf, b1 = zf;
      if constexpr (!K16) {
        b0 = i0 >= 0 ? ld_l2_f4(p0 + 4) : zf;
        b1 = i1 >= 0 ? ld_l2_f4(p1 + 4) : zf;
      }
      if (ADAPT && rl < RK) {  // intermediate columns j >= rl count as zero
        const int j = K16 ? 4 * tq : kb * 32 + 8 * tq;
        mask_cols(a0, j, rl);
        mask_cols(a1, j, rl);
        mask_cols(b0, j + 4, rl);
        mask_cols(b1, j + 4, rl);
      }
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
        if (!MOL_CHECK((int64_t)i < numel, MOL_CHECK_ROW, i) ||
            !MOL_CHECK(ocol + 8 <= (int64_t)S * Ns, MOL_CHECK_COLUMN, ocol))
          continue;
        const float sw = topk_w ? scale_v * __ldg(topk_w + i) : scale_v;
        uint4 o = h ? o1 : o0;
        uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float lo = fmaf(sw, acc[u][2 * h], bf16_lo(ow[u]));
          const float hi = fmaf(sw, acc[u][2 * h + 1], bf16_hi(ow[u]));
          ow[u] = pack_bf16x2(lo, hi);
        }
        *reinterpret_cast<uint4*>(out + (int64_t)i * out_stride + ocol) = o;
      }
    }
  }
}

// Staged expand, rank 8, 16, 32 or 64. One item = (routed block t, slice s, COLS
// output columns: 256, 512 or 768). One thread copies the item's lora_b rows (COLS x
// RK bf16, contiguous in [V, N, r]) into shared memory with a bulk copy, and
// every thread copies its pieces of the output rows to update with cp.async, so
// neither takes registers while in flight; each warp covers COLS / 4 columns
// (32-column groups) with the intermediate it loads once. At rank 32, 64
// registers and 26 KB let eight blocks share an SM, enough to run the decode
// expands in about one wave. Fragment layout, MMA order per accumulator,
// rounding and the handling of adapter arrays (ADAPT: rank 0 writes nothing;
// both operands are zeroed past the adapter's rank; the delta is scaled by its
// scaling) are those of lora_expand_kernel, so both kernels give bit-identical
// outputs. DB (blocks of many rows): two staged row tiles, the next tile's
// output rows are copied while the current one computes. Rank 8 runs the
// rank-16 step (k = 16) with the upper eight k columns zero in both operands:
// quads tq = 2, 3 of a warp, which would hold them, load nothing.
// COLS: output columns per item, 256, or 512 or 768 (ranks 8 and 16, one staged tile)
__host__ __device__ constexpr int st_out_pitch(int cols) { return cols + 32; }  // elements (64-byte skew per row)
// dynamic shared memory of one block: the lora_b tile, then the output row tile(s), then
// (two staged tiles) the next tile's intermediate fragments
constexpr size_t expand_st_smem(int rk, bool db, int cols) {
  return (size_t)cols * rk * 2 + (size_t)(db ? 2 : 1) * 16 * st_out_pitch(cols) * 2 +
         (db ? (size_t)16 * rk * 4 : 0);
}

// Outcome of one staged expand item: skipped (nothing copied), done (its weight tile
// consumed one phase of the weight barrier), past the routed blocks, or the block leaves
// (a wait ran out or a check failed).
enum StItem : int { kStSkip = 0, kStDone = 1, kStPast = 2, kStLeave = 3 };

// Item `it` of the staged expand (lora_expand_st_kernel). Every return is block-uniform.
template <int RK, bool EARLY, bool ADAPT, bool DB, int COLS, bool LOOP>
MOL_DEV int expand_st_item(int it, uint32_t wphase, bool& waited, unsigned char* st_smem,
                           uint64_t* wbar, int* rows, int* wcnt, const float* __restrict__ inter,
                           int R, const uint16_t* __restrict__ lora_b, int S, int Ns, float scale,
                           const float* __restrict__ topk_w, const int* __restrict__ sorted_ids,
                           const int* __restrict__ expert_ids, const int* __restrict__ ntpp_ptr,
                           int block_m, int64_t numel, int num_vexperts,
                           uint16_t* __restrict__ out, int64_t out_stride, int chunks_per_slice,
                           int n_items, const int* __restrict__ lora_ranks,
                           const float* __restrict__ lora_scalings, int num_experts) {
  static_assert(RK == 8 || RK == 16 || RK == 32 || RK == 64, "staged expand: rank 8, 16, 32 or 64");
  static_assert(COLS == 256 || COLS == 512 || COLS == 768,
                "staged expand: 256, 512 or 768 columns per item");
  constexpr int kStCols = COLS;
  constexpr int kStGroups = kStCols / (kExpandThreads / 32) / 32;  // column groups per warp
  constexpr int kStOutPitch = st_out_pitch(kStCols);
  constexpr bool K16 = (RK <= 16);
  constexpr int KB = K16 ? 1 : RK / 32;  // k blocks (32 wide, or one 16-wide block)
  uint16_t* wsm = reinterpret_cast<uint16_t*>(st_smem);  // kStCols x RK lora_b rows
  uint16_t* osm = wsm + kStCols * RK;                     // (DB ? 2 : 1) x 16 output rows
  float* ism = reinterpret_cast<float*>(osm + (DB ? 2 : 1) * 16 * kStOutPitch);  // DB: 16 x RK
  const int tid = threadIdx.x;
  const int per_block = S * chunks_per_slice;
  const int t = it / per_block;
  const int rem = it - t * per_block;
  const int s = rem / chunks_per_slice;
  const int chunk = rem - s * chunks_per_slice;
  const int ntpp = __ldg(ntpp_ptr);
  const int v = __ldg(expert_ids + t);
  const int slot = tid < block_m ? __ldg(sorted_ids + (int64_t)t * block_m + tid) : -1;
  if (kChecked && rem == 0)
    note_block_routing(t, ntpp, v, slot, block_m, numel, num_vexperts,
                       (int64_t)(n_items / per_block) * block_m);
  if ((int64_t)t * block_m >= ntpp) return kStPast;
  if (v < 0 || v >= num_vexperts) return kStSkip;
  // the adapter's rank and scaling, in flight over the row compaction
  int rk_raw = RK;
  float scl = 1.f;
  if constexpr (ADAPT) {
    if (lora_ranks) rk_raw = __ldg(lora_ranks + v / num_experts);
    if (lora_scalings) scl = __ldg(lora_scalings + v / num_experts);
  }
  const int c = compact_block_rows(slot, numel, rows, wcnt);
  if (c == 0) return kStSkip;
  // rank 0: the adapter writes no delta (nothing is copied); past rank rl the
  // intermediate and the weight columns are padding and take no part
  const int rl = rk_raw < 0 ? 0 : (rk_raw > RK ? RK : rk_raw);
  if (ADAPT && rl == 0) return kStSkip;
  const float scale_v = ADAPT ? scale * scl : scale;
  // columns [col0, col0 + ncols) of the slice; ncols > 0 (chunk < ceil(Ns / kStCols)) and a
  // multiple of 8, so the copy is a multiple of 16 bytes from a 16-byte aligned row
  const int col0 = chunk * kStCols;
  const int ncols = min(kStCols, Ns - col0);
  if (kChecked) {  // block-uniform: the whole block leaves before the copy is issued
    const int64_t wr = (int64_t)v * S * Ns + (int64_t)s * Ns + col0;
    const bool wok = ncols > 0 && ncols <= kStCols && wr + ncols <= (int64_t)num_vexperts * S * Ns;
    const bool cok = s * RK + RK <= R;
    if (tid == 0) {
      (void)MOL_CHECK(wok, MOL_CHECK_WEIGHT_ROW, wr);
      (void)MOL_CHECK(cok, MOL_CHECK_COLUMN, s * RK);
    }
    if (!wok || !cok) return kStLeave;
  }
  if (tid == 0) {
    const uint32_t bytes = (uint32_t)ncols * RK * 2;
    mbar_arrive_expect_tx(wbar, bytes);
    bulk_g2s(wsm, lora_b + ((int64_t)v * S * Ns + (int64_t)s * Ns + col0) * RK, bytes, wbar);
  }

  const int lane = tid & 31, warp = tid >> 5, g = lane >> 2, tq = lane & 3;
  const bool kq = RK != 8 || tq < 2;       // this quad's k columns exist (rank 8: the first two)
  const int wcol = warp * 32 * kStGroups;  // the warp's first column inside the item
  const float4 zf = make_float4(0.f, 0.f, 0.f, 0.f);
  const uint4 zu = make_uint4(0, 0, 0, 0);
  int i0 = g < c ? rows[g] : -1;
  int i1 = 8 + g < c ? rows[8 + g] : -1;
  // output rows to update (rows r0 and r1 of a row tile), every column group of
  // the warp (thread tq: 8 columns each), staged at
  // osm[(16 * buf + 8 * hh + g) * kStOutPitch + column inside the item]; each
  // thread later reads back only what it copied itself
  auto osm_at = [&](int buf, int hh, int col) {
    return osm + ((DB ? 16 * buf : 0) + 8 * hh + g) * kStOutPitch + col;
  };
  auto load_out = [&](int buf, int r0, int r1) {
#pragma unroll
    for (int cg = 0; cg < kStGroups; ++cg) {
      const int col = wcol + cg * 32 + 8 * tq;
      const bool ok = col0 + col < Ns;
      const int64_t oc = (int64_t)s * Ns + col0 + col;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = hh ? r1 : r0;
        if (ok && i >= 0 && MOL_CHECK((int64_t)i < numel, MOL_CHECK_ROW, i) &&
            MOL_CHECK(oc + 8 <= (int64_t)S * Ns, MOL_CHECK_COLUMN, oc))
          cp_async16_zfill(osm_at(buf, hh, col), out + (int64_t)i * out_stride + oc, 16u);
      }
    }
  };
  // DB: the intermediate fragments of rows r0 and r1 (columns of the quad in
  // every k block), staged at ism[(8 * hh + g) * RK + column]; the four warps
  // copy the same values to the same places, each thread reads back what it
  // copied, and a block barrier separates every warp's reads of one tile from
  // the copies of the next
  auto ism_at = [&](int hh, int j) { return ism + (8 * hh + g) * RK + j; };
  auto load_inter = [&](int r0, int r1) {
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) {
      const int j = K16 ? 4 * tq : kb * 32 + 8 * tq;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = hh ? r1 : r0;
        if (!kq || i < 0 || !MOL_CHECK((int64_t)i < numel, MOL_CHECK_ROW, i)) continue;
        const float* src = inter + (int64_t)i * R + s * RK + j;
        cp_async16_zfill(ism_at(hh, j), src, 16u);
        if constexpr (!K16) cp_async16_zfill(ism_at(hh, j + 4), src + 4, 16u);
      }
    }
  };
  load_out(0, i0, i1);
  cp_async_commit();
  if (!waited) {
    pdl_wait();  // the intermediate comes from the shrink that precedes this kernel
    pdl_launch_dependents();
    waited = true;
  }
  if constexpr (DB) {
    load_inter(i0, i1);
    cp_async_commit();
  }

  bool landed = false;
  for (int m0 = 0; m0 < c; m0 += 16) {
    const int buf = DB ? (m0 >> 4) & 1 : 0;
    if (m0 > 0) {
      i0 = m0 + g < c ? rows[m0 + g] : -1;
      i1 = m0 + 8 + g < c ? rows[m0 + 8 + g] : -1;
      if (!DB) {
        load_out(0, i0, i1);
        cp_async_commit();
      }
    }
    const bool ahead = DB && m0 + 16 < c;
    const int n0 = ahead && m0 + 16 + g < c ? rows[m0 + 16 + g] : -1;
    const int n1 = ahead && m0 + 24 + g < c ? rows[m0 + 24 + g] : -1;
    if (ahead) {  // the next tile's output rows, into the other buffer
      load_out(buf ^ 1, n0, n1);
      cp_async_commit();
    }
    // the intermediate fragments, split into bf16 head and tail, serve every column
    // group: from global memory (L2) at once with one staged tile, from the staged
    // copies (after their wait below) with two
    const int koff = s * RK + (K16 ? 4 * tq : 8 * tq);
    const float* p0 = inter + (int64_t)(i0 >= 0 ? i0 : 0) * R + koff;
    const float* p1 = inter + (int64_t)(i1 >= 0 ? i1 : 0) * R + koff;
    uint32_t h[KB][8], l[KB][8];
    auto build = [&]() {
#pragma unroll
      for (int kb = 0; kb < KB; ++kb) {
        const int j = K16 ? 4 * tq : kb * 32 + 8 * tq;
        float4 a0, a1;
        if constexpr (DB) {
          a0 = (kq && i0 >= 0) ? *reinterpret_cast<const float4*>(ism_at(0, j)) : zf;
          a1 = (kq && i1 >= 0) ? *reinterpret_cast<const float4*>(ism_at(1, j)) : zf;
        } else {
          a0 = (kq && i0 >= 0) ? ld_l2_f4(p0 + kb * 32) : zf;
          a1 = (kq && i1 >= 0) ? ld_l2_f4(p1 + kb * 32) : zf;
        }
        if (ADAPT && rl < RK) {
          mask_cols(a0, j, rl);
          mask_cols(a1, j, rl);
        }
        split_bf16x2(a0.x, a0.y, h[kb][0], l[kb][0]);
        split_bf16x2(a1.x, a1.y, h[kb][1], l[kb][1]);
        split_bf16x2(a0.z, a0.w, h[kb][2], l[kb][2]);
        split_bf16x2(a1.z, a1.w, h[kb][3], l[kb][3]);
        if constexpr (!K16) {
          float4 b0, b1;
          if constexpr (DB) {
            b0 = i0 >= 0 ? *reinterpret_cast<const float4*>(ism_at(0, j + 4)) : zf;
            b1 = i1 >= 0 ? *reinterpret_cast<const float4*>(ism_at(1, j + 4)) : zf;
          } else {
            b0 = i0 >= 0 ? ld_l2_f4(p0 + kb * 32 + 4) : zf;
            b1 = i1 >= 0 ? ld_l2_f4(p1 + kb * 32 + 4) : zf;
          }
          if (ADAPT && rl < RK) {
            mask_cols(b0, j + 4, rl);
            mask_cols(b1, j + 4, rl);
          }
          split_bf16x2(b0.x, b0.y, h[kb][4], l[kb][4]);
          split_bf16x2(b1.x, b1.y, h[kb][5], l[kb][5]);
          split_bf16x2(b0.z, b0.w, h[kb][6], l[kb][6]);
          split_bf16x2(b1.z, b1.w, h[kb][7], l[kb][7]);
        }
      }
    };
    if (!DB) build();
    if (!landed) {  // every thread sees the weight copy land before it reads the tile
      bool ok = mbar_wait(wbar, wphase, kWaitPolls);
      // two staged tiles, or more items to come: barriers follow, so the block leaves
      // together or not at all (one item: each thread may leave alone)
      if constexpr (DB || LOOP) ok = __syncthreads_and(ok ? 1 : 0) != 0;
      if (!ok) {
        atomicOr(&g_fault_flags, kFaultBulkTimeout);
        cp_async_wait_all();
        return kStLeave;
      }
      landed = true;
    }
    if (ahead)
      cp_async_wait_group<1>();  // this tile's pieces; the next tile's output rows stay in flight
    else
      cp_async_wait_all();  // this thread's pieces
    if constexpr (DB) {
      build();
      if (ahead) {  // every warp has this tile's fragments in registers: stage the next tile's
        named_sync(1, kExpandThreads);
        load_inter(n0, n1);
        cp_async_commit();
      }
    }
#pragma unroll
    for (int cg = 0; cg < kStGroups; ++cg) {
      const int nb = wcol + cg * 32;  // the group's first column inside the item
      if (nb >= ncols) break;         // warp-uniform
      float acc[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        // weight row of output column nb + 8*(g/2) + 2u + (g%2): thread tq ends with
        // columns nb + 8tq .. nb + 8tq + 7
        const int wr = nb + 8 * (g >> 1) + 2 * u + (g & 1);
        const bool bv = wr < ncols;
        if constexpr (K16) {
          const uint2 q2 = (bv && kq) ? lds8(wsm + wr * RK + 4 * tq) : make_uint2(0, 0);
          uint4 q = make_uint4(q2.x, q2.y, 0, 0);
          if (ADAPT && rl < RK) mask_bf16x8(q, 4 * tq, rl);
          mma_16816(acc[u], h[0][0], h[0][1], h[0][2], h[0][3], q.x, q.y);
          mma_16816(acc[u], l[0][0], l[0][1], l[0][2], l[0][3], q.x, q.y);
        } else {
#pragma unroll
          for (int kb = 0; kb < KB; ++kb) {
            uint4 q = bv ? lds16(wsm + wr * RK + kb * 32 + 8 * tq) : zu;
            if (ADAPT && rl < RK) mask_bf16x8(q, kb * 32 + 8 * tq, rl);
            mma_16816(acc[u], h[kb][0], h[kb][1], h[kb][2], h[kb][3], q.x, q.y);
            mma_16816(acc[u], l[kb][0], l[kb][1], l[kb][2], l[kb][3], q.x, q.y);
            mma_16816(acc[u], h[kb][4], h[kb][5], h[kb][6], h[kb][7], q.z, q.w);
            mma_16816(acc[u], l[kb][4], l[kb][5], l[kb][6], l[kb][7], q.z, q.w);
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
          const float sw = topk_w ? scale_v * __ldg(topk_w + i) : scale_v;
          uint4 ov = lds16(osm_at(buf, hh, nb + 8 * tq));
          uint32_t* ow = reinterpret_cast<uint32_t*>(&ov);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float lo = fmaf(sw, acc[u][2 * hh], bf16_lo(ow[u]));
            const float hi = fmaf(sw, acc[u][2 * hh + 1], bf16_hi(ow[u]));
            ow[u] = pack_bf16x2(lo, hi);
          }
          *reinterpret_cast<uint4*>(out + (int64_t)i * out_stride + oc) = ov;
        }
      }
    }
  }
  return kStDone;
}

// LOOP (more than four items per resident block): a wave of resident blocks, block b
// taking items b + j * gridDim.x in order of the routed block t, so once t lies past the
// routed blocks so do all later ones and the block leaves; the row compaction's first
// barrier comes after every thread has finished the previous item (its rows, its weight
// tile, its weight barrier phase). Otherwise one block per item.
template <int RK, bool EARLY, bool ADAPT, bool DB, int COLS, bool LOOP>
__global__ void __launch_bounds__(kExpandThreads, RK == 64 ? (DB ? 4 : 5)
                                                  : COLS == 768 ? 4 : COLS == 512 ? 6 : (DB ? 6 : 8))
lora_expand_st_kernel(const float* __restrict__ inter, int R, const uint16_t* __restrict__ lora_b,
                      int S, int Ns, float scale, const float* __restrict__ topk_w,
                      const int* __restrict__ sorted_ids, const int* __restrict__ expert_ids,
                      const int* __restrict__ ntpp_ptr, int block_m, int64_t numel,
                      int num_vexperts, uint16_t* __restrict__ out, int64_t out_stride,
                      int chunks_per_slice, int n_items, const int* __restrict__ lora_ranks,
                      const float* __restrict__ lora_scalings, int num_experts) {
  extern __shared__ __align__(128) unsigned char st_smem[];
  __shared__ uint64_t wbar;
  __shared__ int rows[128];
  __shared__ int wcnt[kExpandThreads / 32];
  if (threadIdx.x == 0) {
    mbar_init(&wbar, 1);
    fence_mbar_init();  // the first row compaction's barriers publish the init
  }
  if (!EARLY) {
    pdl_wait();
    pdl_launch_dependents();
  }
  bool waited = !EARLY;
#define MOL_ST_ITEM_ARGS                                                                       \
  st_smem, &wbar, rows, wcnt, inter, R, lora_b, S, Ns, scale, topk_w, sorted_ids, expert_ids, \
      ntpp_ptr, block_m, numel, num_vexperts, out, out_stride, chunks_per_slice, n_items,      \
      lora_ranks, lora_scalings, num_experts
  if constexpr (!LOOP) {
    (void)expand_st_item<RK, EARLY, ADAPT, DB, COLS, false>(blockIdx.x, 0u, waited, MOL_ST_ITEM_ARGS);
  } else {
    uint32_t wphase = 0;  // parity of the weight barrier's next phase
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
      const int r = expand_st_item<RK, EARLY, ADAPT, DB, COLS, true>(it, wphase, waited, MOL_ST_ITEM_ARGS);
      if (r == kStPast || r == kStLeave) break;
      if (r == kStDone) wphase ^= 1;
    }
  }
#undef MOL_ST_ITEM_ARGS
}

static int device_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

// Blocks of kernel K (kExpandThreads threads, `smem` dynamic bytes) resident on the
// device at once: its SM count times its occupancy, cached per kernel and device.
template <auto K>
static int64_t resident_blocks(size_t smem) {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, K, kExpandThreads, smem) != cudaSuccess ||
        n <= 0)
      n = 1;
    cache[dev] = n;
  }
  return (int64_t)device_sms() * cache[dev];
}

// Opts the staged expand instances above 48 KB of dynamic shared memory in (the looping
// ones exist for one staged tile and without early reads).
template <int RK, bool DB, int COLS = 256>
static cudaError_t prepare_expand_st() {
  const int bytes = (int)expand_st_smem(RK, DB, COLS);
  cudaError_t e = cudaSuccess;
  for (auto k : {lora_expand_st_kernel<RK, false, false, DB, COLS, false>,
                 lora_expand_st_kernel<RK, false, true, DB, COLS, false>,
                 lora_expand_st_kernel<RK, true, false, DB, COLS, false>,
                 lora_expand_st_kernel<RK, true, true, DB, COLS, false>,
                 lora_expand_st_kernel<RK, false, false, false, COLS, true>,
                 lora_expand_st_kernel<RK, false, true, false, COLS, true>})
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e;
}

cudaError_t prepare_lora_kernels() {
  cudaError_t e = prepare_tc_kernels();
  if (e != cudaSuccess) return e;
  e = prepare_expand_tc_kernels();
  if (e != cudaSuccess) return e;
  e = prepare_expand_st<64, true>();
  if (e != cudaSuccess) return e;
  e = prepare_expand_st<64, false>();
  if (e != cudaSuccess) return e;
  e = prepare_expand_st<32, true>();
  if (e != cudaSuccess) return e;
  e = prepare_expand_st<32, false>();
  if (e != cudaSuccess) return e;
  e = prepare_expand_st<16, true>();
  if (e != cudaSuccess) return e;
  e = prepare_expand_st<16, false>();
  if (e != cudaSuccess) return e;
  e = prepare_expand_st<8, true>();
  if (e != cudaSuccess) return e;
  e = prepare_expand_st<8, false>();
  if (e != cudaSuccess) return e;
  e = prepare_expand_st<16, false, 512>();
  if (e == cudaSuccess) e = prepare_expand_st<16, false, 768>();
  if (e == cudaSuccess) e = prepare_expand_st<8, false, 512>();
  if (e == cudaSuccess) e = prepare_expand_st<8, false, 768>();
  if (e != cudaSuccess) return e;
  for (auto k : {lora_shrink_kernel<false, 8>, lora_shrink_kernel<true, 8>,
                 lora_shrink_kernel<false, 16>, lora_shrink_kernel<true, 16>})
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp::kSmem);
  return e;
}

cudaError_t launch_shrink(const void* x, int64_t x_stride, int x_div, int K, const void* lora_a,
                          int R, const int32_t* sorted_ids, const int32_t* expert_ids,
                          const int32_t* ntpp, int64_t capacity, int block_m, int64_t numel,
                          int num_vexperts, float* inter, bool early, cudaStream_t stream,
                          int r1, const int32_t* lora_ranks, int num_experts,
                          const RoutingIds* prefetch) {
  const int64_t nblk = capacity / block_m;
  if (numel == 0 || nblk == 0) return cudaSuccess;
  if (!lora_ranks && shrink_tc_fits(numel, num_vexperts, R, K, block_m))
    return launch_shrink_tc(x, x_stride, x_div, K, lora_a, R, sorted_ids, expert_ids, ntpp,
                            capacity, block_m, numel, num_vexperts, inter, stream);
  // Items of 16 weight rows where an item with the average row count is copied whole at
  // full K (one weight copy, half as many items: decode down 4.98 -> 4.14 us), or where
  // routed blocks average at least four pairs and 8-row items would not be whole either
  // (each item's activation rows are copied once for twice the weight bytes); otherwise
  // items of 8 weight rows (whole at full K, and twice as many to share among the blocks)
  const int64_t avg_rows = (numel + std::min<int64_t>(numel, num_vexperts) - 1) /
                           std::min<int64_t>(numel, num_vexperts);
  const bool whole8 = (8 + avg_rows) * K * 2 <= sp::kStageBytes;
  const bool whole16 = (16 + avg_rows) * K * 2 <= sp::kStageBytes;
  const bool many = numel >= 4 * std::min<int64_t>(numel, num_vexperts);
  const int JT = (r1 % 16 == 0 && (whole16 || (many && !whole8))) ? 16 : 8;
  const int n_jt = R / JT;
  const int num_loras = lora_ranks ? num_vexperts / num_experts : 0;
  const int64_t n_items = nblk * n_jt;
  const int64_t G = std::min<int64_t>(n_items, (int64_t)device_sms() * sp::kBlocksPerSM);
  // the L2 prefetch (ids declared ready early): few pairs, every virtual expert owned by one
  // of 32 slots of a block, and the lora_a rows of as many virtual experts as there can be
  // pairs within the budget
  RoutingIds pf{nullptr, nullptr, 0, 1, 1, 1, false};
  if (prefetch && prefetch->ready_early && prefetch->numel <= kPrefetchPairsMax &&
      num_vexperts <= 32 * G &&
      std::min<int64_t>(numel, num_vexperts) * R * K * 2 <= kPrefetchBudget)
    pf = *prefetch;
  auto kernel = JT == 16 ? (lora_ranks ? lora_shrink_kernel<true, 16> : lora_shrink_kernel<false, 16>)
                         : (lora_ranks ? lora_shrink_kernel<true, 8> : lora_shrink_kernel<false, 8>);
  return launch_pdl(kernel,
                    dim3((unsigned)G), dim3(sp::kThreads), sp::kSmem, stream,
                    static_cast<const uint16_t*>(x), x_stride, x_div, K,
                    static_cast<const uint16_t*>(lora_a), R, sorted_ids, expert_ids, ntpp, block_m,
                    numel, num_vexperts, inter, n_jt, n_items, early ? 1 : 0, r1, lora_ranks,
                    num_experts < 1 ? 1 : num_experts, num_loras, pf);
}

// One staged expand instance over n_items items. One staged tile and more than four
// items per resident block: one wave of resident blocks, each looping over items (no block
// launch, barrier set-up and routing read per item; the blocks past the routed ones leave
// at their first item there); otherwise one block per item, which the hardware deals to
// the SMs as they free up (measured faster with few items per block).
template <int RK, bool E, bool A, bool D, int C>
static cudaError_t launch_expand_st(cudaStream_t stream, int64_t n_items, const float* inter, int R,
                                    const uint16_t* b, int S, int Ns, float scale, const float* w,
                                    const int32_t* sorted_ids, const int32_t* expert_ids,
                                    const int32_t* ntpp, int block_m, int64_t numel,
                                    int num_vexperts, uint16_t* o, int64_t out_stride, int cps,
                                    const int32_t* ranks, const float* scalings, int ne) {
  const size_t smem = expand_st_smem(RK, D, C);
  const int64_t resident =
      D ? 0 : resident_blocks<lora_expand_st_kernel<RK, false, A, false, C, true>>(smem);
  // every block starts at once, after the previous kernel (no early launch, so no early reads)
  if (!D && n_items > 4 * resident)
    return launch_ordered(lora_expand_st_kernel<RK, false, A, false, C, true>, dim3((unsigned)resident),
                          dim3(kExpandThreads), smem, stream, inter, R, b, S, Ns, scale, w,
                          sorted_ids, expert_ids, ntpp, block_m, numel, num_vexperts, o,
                          out_stride, cps, (int)n_items, ranks, scalings, ne);
  return launch_pdl(lora_expand_st_kernel<RK, E, A, D, C, false>, dim3((unsigned)n_items),
                    dim3(kExpandThreads), smem, stream, inter, R, b, S, Ns, scale, w, sorted_ids,
                    expert_ids, ntpp, block_m, numel, num_vexperts, o, out_stride, cps,
                    (int)n_items, ranks, scalings, ne);
}

template <int RK, bool EARLY>
static cudaError_t expand_rk(dim3 grid, cudaStream_t stream, const float* inter, int R,
                             const uint16_t* b, int S, int Ns, float scale, const float* w,
                             const int32_t* sorted_ids, const int32_t* expert_ids,
                             const int32_t* ntpp, int block_m, int64_t numel, int num_vexperts,
                             uint16_t* o, int64_t out_stride, int cps, const int32_t* ranks,
                             const float* scalings, int num_experts) {
  const bool adapt = ranks != nullptr || scalings != nullptr;
  return launch_pdl(adapt ? lora_expand_kernel<RK, EARLY, true> : lora_expand_kernel<RK, EARLY, false>,
                    grid, dim3(kExpandThreads), 0, stream, inter, R,
                    b, S, Ns, scale, w, sorted_ids, expert_ids, ntpp, block_m, numel, num_vexperts,
                    o, out_stride, cps, ranks, scalings, num_experts < 1 ? 1 : num_experts);
}

cudaError_t launch_expand(const float* inter, const void* lora_b, int S, int r, int Ns, float scale,
                          const float* topk_weights, const int32_t* sorted_ids,
                          const int32_t* expert_ids, const int32_t* ntpp, int64_t capacity,
                          int block_m, int64_t numel, int num_vexperts, void* out,
                          int64_t out_stride, bool early, cudaStream_t stream,
                          const int32_t* lora_ranks, const float* lora_scalings, int num_experts) {
  const int64_t nblk = capacity / block_m;
  if (numel == 0 || nblk == 0) return cudaSuccess;
  const int R = S * r;
  const uint16_t* b = static_cast<const uint16_t*>(lora_b);
  uint16_t* o = static_cast<uint16_t*>(out);
  if (expand_tc_fits(numel, num_vexperts, r, Ns, block_m, out_stride,
                     lora_ranks != nullptr || lora_scalings != nullptr))
    return launch_expand_tc(inter, lora_b, S, Ns, scale, topk_weights, sorted_ids, expert_ids, ntpp,
                            capacity, block_m, numel, num_vexperts, out, out_stride, stream);
  if (r == 8 || r == 16 || r == 32 || r == 64) {
    // many rows per virtual expert (on average at least 32 pairs each): blocks hold
    // several row tiles, so the output rows of the next one are prefetched
    const bool db = numel >= 32 * std::min<int64_t>(numel, num_vexperts);
    // ranks 8 and 16 with at least four pairs per virtual expert on average: items of 768
    // columns where they tile the slice, else 512, so a block moves at least as many
    // bytes as a rank-32 item of 256 and the grid has fewer items (each pays the routing
    // reads and the row compaction); measured: 768 where a slice is 768 wide beats 512,
    // 1024 on a 2048-wide slice loses to 512 (three blocks per SM instead of six)
    const bool wide = r <= 16 && !db && numel >= 4 * std::min<int64_t>(numel, num_vexperts);
    const int cols = wide ? (Ns % 768 == 0 ? 768 : 512) : 256;
    const int cps_st = (Ns + cols - 1) / cols;
    const int64_t n_items = nblk * S * cps_st;
    if (n_items > INT32_MAX) return cudaErrorInvalidConfiguration;
    const bool adapt = lora_ranks != nullptr || lora_scalings != nullptr;
    const int ne = num_experts < 1 ? 1 : num_experts;
#define MOL_EXPAND_ST(RK, E, A, D, C)                                                            \
  launch_expand_st<RK, E, A, D, C>(stream, n_items, inter, R, b, S, Ns, scale, topk_weights,     \
                                   sorted_ids, expert_ids, ntpp, block_m, numel, num_vexperts, o, \
                                   out_stride, cps_st, lora_ranks, lora_scalings, ne)
#define MOL_EXPAND_ST_A(RK, E, A) \
  (db ? MOL_EXPAND_ST(RK, E, A, true, 256) : MOL_EXPAND_ST(RK, E, A, false, 256))
#define MOL_EXPAND_ST_W(RK, E, A)                                                     \
  (cols == 768 ? MOL_EXPAND_ST(RK, E, A, false, 768)                                 \
   : cols == 512 ? MOL_EXPAND_ST(RK, E, A, false, 512) : MOL_EXPAND_ST_A(RK, E, A))
#define MOL_EXPAND_ST_RK(RK, M)                                                  \
  return early ? (adapt ? M(RK, true, true) : M(RK, true, false))                \
               : (adapt ? M(RK, false, true) : M(RK, false, false))
    if (r == 8) MOL_EXPAND_ST_RK(8, MOL_EXPAND_ST_W);
    if (r == 16) MOL_EXPAND_ST_RK(16, MOL_EXPAND_ST_W);
    if (r == 32) MOL_EXPAND_ST_RK(32, MOL_EXPAND_ST_A);
    MOL_EXPAND_ST_RK(64, MOL_EXPAND_ST_A);
#undef MOL_EXPAND_ST_RK
#undef MOL_EXPAND_ST_W
#undef MOL_EXPAND_ST_A
#undef MOL_EXPAND_ST
  }
  const int cps = (Ns + kExpandCols - 1) / kExpandCols;
  if (nblk * S * cps > INT32_MAX) return cudaErrorInvalidConfiguration;
  const dim3 grid((unsigned)(nblk * S * cps));
#define MOL_EXPAND_CASE(RK)                                                                     \
  case RK:                                                                                      \
    return early ? expand_rk<RK, true>(grid, stream, inter, R, b, S, Ns, scale, topk_weights,   \
                                       sorted_ids, expert_ids, ntpp, block_m, numel,            \
                                       num_vexperts, o, out_stride, cps, lora_ranks,            \
                                       lora_scalings, num_experts)                              \
                 : expand_rk<RK, false>(grid, stream, inter, R, b, S, Ns, scale, topk_weights,  \
                                        sorted_ids, expert_ids, ntpp, block_m, numel,           \
                                        num_vexperts, o, out_stride, cps, lora_ranks,           \
                                        lora_scalings, num_experts);
  switch (r) {
    MOL_EXPAND_CASE(16)
    MOL_EXPAND_CASE(32)
    MOL_EXPAND_CASE(64)
    MOL_EXPAND_CASE(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOL_EXPAND_CASE
}

cudaError_t take_lora_checks(unsigned long long* first, unsigned long long* count) {
  CheckRecord r;
  const cudaError_t e = take_check_record_here(&r);
  *first = r.first;
  *count = r.count;
  return e;
}

}  // namespace mol
