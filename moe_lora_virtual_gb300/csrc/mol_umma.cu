// LoRA shrink on the fifth-generation tensor cores (tcgen05, accumulators in
// tensor memory) for batches where each virtual expert holds many rows.
//
// When every token runs the same adapter the routed blocks are full (64 or
// 128 rows of one virtual expert) and the shrink is a real dense contraction:
// fork PR #24 "Root cause" commit, the MoL shrink is a fused-MoE GEMM over the
// virtual experts with N = S*r and K = the input width; code-review commit,
// weights laid out [E, N, K]. This kernel computes, per routed block t of
// virtual expert v and per 128 lora_a rows (mt; when R is not a multiple of
// 128 the last tile holds the expert's last 64 rows only: a 64-row weight box
// fills the first half of the stage's weight tile, the MMA's other 64 rows
// read whatever the stage held before and are computed but not stored),
//   D[j, n] = sum_k lora_a[v, mt*128 + j, k] * x[row(n), k]     (j < 128, n < BM)
// as tcgen05.mma M=128 x N=BM x K=16 steps (bf16 in, fp32 in tensor memory),
// and writes inter[pair(n), mt*128 + j] = D[j, n] for the block's real rows.
//
// Layout. A persistent grid; each block walks items (t, mt) b, b+G, ... with
// ten warps in four roles:
//   warp 0     TMA producer: one cp.async.bulk.tensor per stage moves the
//              128 x 64 weight tile (128-byte swizzle) into the stage;
//   warp 1     allocates the tensor memory (two accumulators of BM columns),
//              and one lane issues the MMAs of a stage (four K=16 steps) and
//              commits them to the stage's "empty" barrier and, after the
//              item's last stage, to the accumulator's "full" barrier;
//   warps 2-5  gather: the block's x rows, 128 bytes of each per stage (eight
//              lanes per row, whole lines per instruction), with cp.async into
//              the same 128-byte-swizzled layout (zeros for padding slots);
//              each thread's arrival on the stage's "full" barrier fires when
//              its copies land (cp.async.mbarrier.arrive.noinc), so the gather
//              never waits for data, and the MMA lane fences the generic and
//              async proxies before the MMAs read the stage;
//   warps 6-9  epilogue: wait for an accumulator, read it with tcgen05.ld
//              (each warp its 32-lane quarter of tensor memory = 32 lora_a
//              rows), release it to the MMA warp, store fp32 rows.
// The two accumulators let the epilogue of one item overlap the next item's
// MMAs. Every wait is bounded: a timeout sets a fault bit, the roles leave
// their loops, and the tensor memory is freed before the block exits.

#include <algorithm>
#include <mutex>

#include "mol_device.cuh"
#include "mol_internal.h"
#include "mol_tc.cuh"

namespace mol {

namespace tc {
constexpr int kM = 128;                   // lora_a rows per item (MMA M)
constexpr int kKStep = 64;                // k per stage: one 128-byte swizzled row
constexpr int kStages = 4;
constexpr int kATile = kM * 128;          // 16 KB
constexpr int kGatherWarps = 4;
constexpr int kEpiWarps = 4;
constexpr int kThreads = (2 + kGatherWarps + kEpiWarps) * 32;
constexpr uint32_t kPolls = 1u << 22;
template <int BN>
struct Geo {
  static constexpr int kXTile = BN * 128;
  static constexpr int kStageBytes = kATile + kXTile;  // multiple of 1024
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;
  static constexpr int kBlocksPerSM = BN == 64 ? 2 : 1;
};
}  // namespace tc

__device__ unsigned int g_tc_fault_flags;

cudaError_t take_tc_faults(unsigned* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_tc_fault_flags, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_tc_fault_flags, &zero, sizeof(unsigned));
}

template <int BN>
__global__ void __launch_bounds__(tc::kThreads, tc::Geo<BN>::kBlocksPerSM)
lora_shrink_tc_kernel(const __grid_constant__ CUtensorMap tmap_a,
                      const __grid_constant__ CUtensorMap tmap_h,
                      const uint16_t* __restrict__ x, int64_t x_stride, int x_div, int K, int R,
                      const int* __restrict__ sorted_ids, const int* __restrict__ expert_ids,
                      const int* __restrict__ ntpp_ptr, int64_t numel, int num_vexperts,
                      float* __restrict__ inter, int64_t n_items, int mtiles) {
  using namespace tc;
  using G = Geo<BN>;
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full[kStages], empty[kStages], accf[2], acce[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int s_fault;
  unsigned char* smem =
      smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1024-byte aligned stages
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1 + kGatherWarps * 32);  // TMA arrival + every gather thread
      mbar_init(&empty[s], 1);                     // MMA commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf[a], 1);          // MMA commit
      mbar_init(&acce[a], kEpiWarps);  // one arrival per epilogue warp
    }
    s_fault = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, G::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  pdl_wait();  // routing, activations and weights may come from the kernel before
  pdl_launch_dependents();

  const int64_t Gs = gridDim.x;
  const int nk = K / kKStep;
  const int ntpp = __ldg(ntpp_ptr);
  auto item = [&](int64_t it, int64_t& t, int& mt, int& v) -> bool {
    t = it / mtiles;
    mt = (int)(it - t * mtiles);
    if (t * BN >= ntpp) return false;
    v = __ldg(expert_ids + t);
    return v >= 0 && v < num_vexperts;
  };
  auto stageA = [&](uint32_t q) { return smem + (size_t)(q % kStages) * G::kStageBytes; };
  bool fault = false;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t q = 0;
      for (int64_t it = blockIdx.x; it < n_items && !fault; it += Gs) {
        int64_t t;
        int mt, v;
        if (kChecked && it % mtiles == 0) {  // the caller's routing words, once per block
          const int64_t tb = it / mtiles;
          const int64_t cap = n_items / mtiles * BN;
          (void)MOL_NOTE(ntpp >= 0 && ntpp <= cap && ntpp % BN == 0, MOL_CHECK_ROUTE_NTPP, ntpp);
          if (tb * BN < ntpp) {
            const int e = __ldg(expert_ids + tb);
            (void)MOL_NOTE(e >= -1 && e < num_vexperts, MOL_CHECK_ROUTE_EXPERT, tb);
          }
        }
        if (!item(it, t, mt, v)) continue;
        const int y = v * R + mt * kM;
        const bool half = R - mt * kM < kM;  // the expert's last 64 rows: the 64-row box
        for (int ks = 0; ks < nk; ++ks, ++q) {
          const int s = (int)(q % kStages);
          if (!mbar_wait(&empty[s], ((q / kStages) & 1) ^ 1, kPolls)) {
            fault = true;
            break;
          }
          // checked build: the box starts on a 16-byte boundary and lies inside the tensor;
          // a failed check skips the copy (the stage then holds stale data)
          const bool in_box =
              MOL_CHECK((ks * kKStep) % 8 == 0 && ks * kKStep + kKStep <= K, MOL_CHECK_TMA_COORD,
                        ks * kKStep) &&
              MOL_CHECK(y >= 0 && (int64_t)y + (half ? kM / 2 : kM) <= (int64_t)num_vexperts * R,
                        MOL_CHECK_TMA_COORD, y);
          if (kChecked && !in_box) {
            mbar_arrive_expect_tx(&full[s], 0u);
            continue;
          }
          mbar_arrive_expect_tx(&full[s], (uint32_t)(half ? kATile / 2 : kATile));
          tma_load_2d(stageA(q), half ? &tmap_h : &tmap_a, ks * kKStep, y, &full[s]);
        }
      }
      // after a timeout, wait (bounded) for the last uses of each stage to complete: their
      // barriers also count the gather's row copies, so a stage whose rows never came
      // costs one more bounded wait
      if (fault)
        for (uint32_t u = q > (uint32_t)kStages ? q - kStages : 0; u < q; ++u)
          mbar_wait(&full[u % kStages], (u / kStages) & 1, kPolls);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = IDesc<tc::kM, BN>::kValue;
      uint32_t q = 0, n = 0;
      for (int64_t it = blockIdx.x; it < n_items && !fault; it += Gs) {
        int64_t t;
        int mt, v;
        if (!item(it, t, mt, v)) continue;
        const int a = (int)(n & 1);
        if (!mbar_wait(&acce[a], ((n >> 1) & 1) ^ 1, kPolls)) {
          fault = true;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(a * BN);
        for (int ks = 0; ks < nk; ++ks, ++q) {
          const int s = (int)(q % kStages);
          if (!mbar_wait(&full[s], (q / kStages) & 1, kPolls)) {
            fault = true;
            break;
          }
          // the x rows arrived through cp.async (generic proxy); the MMAs read
          // them through the async proxy
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t sa = smem_u32(stageA(q));
          const uint32_t sx = sa + kATile;
#pragma unroll
          for (int kk = 0; kk < kKStep / 16; ++kk)  // 16 k = 32 bytes along the swizzled row
            umma_bf16(d, sw128_desc(sa + kk * 32), sw128_desc(sx + kk * 32), idesc,
                      (ks | kk) != 0 ? 1u : 0u);
          umma_commit(&empty[s]);  // the stage is free once these MMAs have read it
        }
        if (fault) break;
        umma_commit(&accf[a]);
        ++n;
      }
    }
  } else if (warp < 2 + kGatherWarps) {
    // ------------------------------------------------------------ x gather
    // Eight lanes cover one row's 128 bytes, so each instruction of a warp
    // moves four whole rows (full lines); thread g takes chunk g % 8 of rows
    // g / 8, g / 8 + kRowStep, ... .
    const int g = tid - 64;
    constexpr int kRowStep = kGatherWarps * 32 / 8;
    constexpr int kRowsPerThr = BN / kRowStep;
    const int c = g & 7, r0 = g >> 3;
    uint32_t q = 0;
    for (int64_t it = blockIdx.x; it < n_items && !fault; it += Gs) {
      int64_t t;
      int mt, v;
      if (!item(it, t, mt, v)) continue;
      const uint16_t* src[kRowsPerThr];
      uint32_t nbytes[kRowsPerThr];
#pragma unroll
      for (int i = 0; i < kRowsPerThr; ++i) {
        const int pid = __ldg(sorted_ids + t * BN + r0 + kRowStep * i);
        if (kChecked && mt == 0 && c == 0)
          (void)MOL_NOTE(pid >= 0 && (int64_t)pid <= numel, MOL_CHECK_ROUTE_PAIR,
                         t * BN + r0 + kRowStep * i);
        const bool ok = pid >= 0 && (int64_t)pid < numel &&
                        MOL_CHECK((int64_t)(pid / x_div) < (numel + x_div - 1) / x_div,
                                  MOL_CHECK_ROW, pid / x_div);
        src[i] = (ok ? x + (int64_t)(pid / x_div) * x_stride : x) + c * 8;
        nbytes[i] = ok ? 16u : 0u;
      }
      for (int ks = 0; ks < nk; ++ks, ++q) {
        const int s = (int)(q % kStages);
        if (!mbar_wait(&empty[s], ((q / kStages) & 1) ^ 1, kPolls)) {
          fault = true;
          break;
        }
        unsigned char* tile = stageA(q) + kATile;
#pragma unroll
        for (int i = 0; i < kRowsPerThr; ++i) {
          const int r = r0 + kRowStep * i;
          cp_async16_zfill(tile + r * 128 + ((c ^ (r & 7)) << 4), src[i] + ks * kKStep, nbytes[i]);
        }
        cp_async_arrive_noinc(&full[s]);
      }
    }
    cp_async_wait_all();  // no copy of this thread is left in flight at exit
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // tensor-memory lanes 32*quarter .. +31
    uint32_t n = 0;
    for (int64_t it = blockIdx.x; it < n_items && !fault; it += Gs) {
      int64_t t;
      int mt, v;
      if (!item(it, t, mt, v)) continue;
      const int a = (int)(n & 1);
      // tcgen05.ld is warp-collective: the lanes agree on the outcome of the wait
      if (!__all_sync(0xffffffffu, mbar_wait(&accf[a], (n >> 1) & 1, kPolls))) {
        fault = true;
        break;
      }
      tc_fence_after();
      // pair ids of the block's rows, two per lane, shared through shuffles
      int p_lo = __ldg(sorted_ids + t * BN + lane);
      int p_hi = __ldg(sorted_ids + t * BN + 32 + lane);
      int p_x2 = BN == 128 ? __ldg(sorted_ids + t * BN + 64 + lane) : -1;
      int p_x3 = BN == 128 ? __ldg(sorted_ids + t * BN + 96 + lane) : -1;
      const int j = mt * kM + quarter * 32 + lane;
      const uint32_t base = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(a * BN);
#pragma unroll 1
      for (int n0 = 0; n0 < BN; n0 += 8) {
        float val[8];
        tmem_ld8(base + (uint32_t)n0, val);
        const int src = n0 < 32 ? p_lo : n0 < 64 ? p_hi : n0 < 96 ? p_x2 : p_x3;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int pid = __shfl_sync(0xffffffffu, src, (n0 + e) & 31);
          if (j < R && pid >= 0 && (int64_t)pid < numel) inter[(int64_t)pid * R + j] = val[e];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[a]);
      ++n;
    }
  }

  if (fault) {
    atomicOr(&g_tc_fault_flags, kFaultBulkTimeout);
    s_fault = 1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, G::kTmemCols);
}

// --- host side ----------------------------------------------------------------

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_status = cudaSuccess;

int tc_device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}
}  // namespace

bool shrink_tc_fits(int64_t numel, int num_vexperts, int R, int K, int block_m) {
  if (numel <= 0 || R % 64 != 0 || K % tc::kKStep != 0) return false;
  if (block_m != 64 && block_m != 128) return false;
  // many rows per virtual expert: on average at least 32 pairs each
  return numel >= 32 * std::min<int64_t>(numel, num_vexperts);
}

cudaError_t prepare_tc_kernels() {
  cudaError_t e = cudaFuncSetAttribute(lora_shrink_tc_kernel<64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tc::Geo<64>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(lora_shrink_tc_kernel<128>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)tc::Geo<128>::kSmem);
}

cudaError_t launch_shrink_tc(const void* x, int64_t x_stride, int x_div, int K, const void* lora_a,
                             int R, const int32_t* sorted_ids, const int32_t* expert_ids,
                             const int32_t* ntpp, int64_t capacity, int block_m, int64_t numel,
                             int num_vexperts, float* inter, cudaStream_t stream) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    g_encode_status = cudaGetDriverEntryPointByVersion(
        "cuTensorMapEncodeTiled", reinterpret_cast<void**>(&g_encode), 12000, cudaEnableDefault, &q);
    if (g_encode_status == cudaSuccess && (q != cudaDriverEntryPointSuccess || !g_encode))
      g_encode_status = cudaErrorNotSupported;
  });
  if (g_encode_status != cudaSuccess) return g_encode_status;
  const int64_t nblk = capacity / block_m;
  if (numel == 0 || nblk == 0) return cudaSuccess;
  // lora_a as a 2-D tensor: num_vexperts * R rows of K bf16, row pitch 2K bytes
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)num_vexperts * (cuuint64_t)R};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)tc::kKStep, (cuuint32_t)tc::kM};
  const cuuint32_t estr[2] = {1, 1};
  CUresult cr = g_encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(lora_a), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // the same tensor with a 64-row box, for the last tile when R % 128 == 64
  CUtensorMap map_h;
  const cuuint32_t box_h[2] = {(cuuint32_t)tc::kKStep, (cuuint32_t)(tc::kM / 2)};
  cr = g_encode(&map_h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(lora_a), dims,
                strides, box_h, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const int mtiles = (R + tc::kM - 1) / tc::kM;
  const int64_t n_items = nblk * mtiles;
  const uint16_t* xp = static_cast<const uint16_t*>(x);
  if (block_m == 64) {
    const dim3 grid((unsigned)std::min<int64_t>(n_items, (int64_t)tc_device_sms() * 2));
    return launch_pdl(lora_shrink_tc_kernel<64>, grid, dim3(tc::kThreads), tc::Geo<64>::kSmem,
                      stream, map, map_h, xp, x_stride, x_div, K, R, sorted_ids, expert_ids, ntpp,
                      numel, num_vexperts, inter, n_items, mtiles);
  }
  const dim3 grid((unsigned)std::min<int64_t>(n_items, (int64_t)tc_device_sms()));
  return launch_pdl(lora_shrink_tc_kernel<128>, grid, dim3(tc::kThreads), tc::Geo<128>::kSmem,
                    stream, map, map_h, xp, x_stride, x_div, K, R, sorted_ids, expert_ids, ntpp,
                    numel, num_vexperts, inter, n_items, mtiles);
}

cudaError_t take_tc_checks(unsigned long long* first, unsigned long long* count) {
  CheckRecord r;
  const cudaError_t e = take_check_record_here(&r);
  *first = r.first;
  *count = r.count;
  return e;
}

}  // namespace mol
