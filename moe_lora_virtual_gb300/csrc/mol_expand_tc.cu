// LoRA expand on the fifth-generation tensor cores (tcgen05, accumulators in
// tensor memory) for full routed blocks of rank 64.
//
// fork PR #24 PR body "Background (measured attribution)": the expand is an
// M x N output with a narrow K = rank contraction added into the MoE output;
// "Fix" commit: its weight view is [E, N, K]. Per routed block t of virtual
// expert v (BN = BLOCK_M rows), slice s and 128 output columns (m-tile m):
//   D[n, j] = sum_k inter[pair(n), s*64 + k] * lora_b[v, s*Ns + m*128 + j, k]
//   out[pair(n), s*Ns + m*128 + j] = bf16(out + scale * w_pair * D[n, j])
// The fp32 intermediate enters the tensor cores as two bf16 operands, its
// head and the bf16 of what is left (tail), so the product keeps 16
// significant bits of it: D = head . lora_b + tail . lora_b, both K = 64 in
// four K = 16 steps of tcgen05.mma M = 128 (rows; with BLOCK_M 64 the upper
// half is not read back), N = 128 (output columns).
//
// When every token runs the same adapter the routed blocks are full and the
// expand streams hundreds of MB of output rows (read, add, write back), with
// little arithmetic per byte; the mma.sync expand is latency-bound there
// (long dependency chains in few resident warps). Here the products run
// asynchronously in the tensor cores and a thread of the epilogue owns
// contiguous columns of one row.
//
// Layout. A persistent grid (one block per SM); block b walks items
// (unit of 128 rows, slice s, group of up to eight m-tiles) b, b+G, ..., so the
// blocks that run at the same time hold neighbouring units and load each lora_b
// tile from DRAM once between them; eighteen warps:
//   warp 0     TMA producer: per m-tile, one cp.async.bulk.tensor for the
//              128 x 64 lora_b tile (128-byte swizzle);
//   warp 1     allocates the tensor memory (two accumulators of 128 columns);
//              one lane issues each m-tile's eight MMAs and commits them to
//              the lora_b tile's "empty" barrier, the accumulator's "full"
//              barrier and, after a run's last m-tile, to its operand
//              buffer's "empty" barrier;
//   warps 2-5  converters: per run of items with the same rows and slice, the
//              rows' pair ids and weights and the intermediate rows as head /
//              tail operands (128-byte swizzle) in one of two buffers, one run
//              ahead;
//   warps 6-9  copiers: per m-tile, the output rows (16-byte cp.async into a
//              staged tile of their own ring), arriving on its "full" barrier
//              as they land;
//   warps 10-17 epilogue: a thread reads 32 columns of its row at a time
//              (tensor-memory lane = row; two warps per 32-lane quarter, one
//              per half of the columns), adds them to the staged output row
//              and the warp stores its rows' bf16 sums, 128 bytes of a row per
//              eight lanes; then the staged tile and the accumulator are
//              released.
// Every wait is bounded: a timeout sets a fault bit, the roles leave their
// loops, and the tensor memory is freed before the block exits.

#include <algorithm>
#include <mutex>

#include "mol_device.cuh"
#include "mol_internal.h"
#include "mol_tc.cuh"

namespace mol {

namespace xt {
constexpr int kM = 128;        // output columns per m-tile (MMA N)
constexpr int kRows = 128;     // MMA M: rows of the operand buffers
constexpr int kRank = 64;      // rank: one 128-byte swizzled row of k
constexpr int kMGroup = 8;     // most m-tiles per item
constexpr int kBTile = kM * kRank * 2;        // 16 KB lora_b tile
constexpr int kATile = kRows * kRank * 2;     // 16 KB head (or tail) operand
constexpr int kConverters = 128;              // warps 2-5
constexpr int kCopiers = 128;                 // warps 6-9
constexpr int kEpiWarps = 8;                  // warps 10-17
constexpr int kThreads = (10 + kEpiWarps) * 32;
constexpr uint32_t kPolls = 1u << 22;
constexpr int kOutPitch = kM * 2 + 16;  // staged output row: 256 bytes + a 16-byte skew
constexpr int round1k(int b) { return (b + 1023) / 1024 * 1024; }
constexpr int kBStages = 3;  // lora_b tiles in flight
constexpr int kAccs = 2;     // accumulators in tensor memory (256 of the 512 columns)
constexpr int kOStages = 3;                        // staged output-row tiles in flight
constexpr int kOTile = round1k(kRows * kOutPitch);
constexpr int kABytes = 2 * kATile;  // head + tail
constexpr size_t kSmem =
    1024 + (size_t)kBStages * kBTile + (size_t)kOStages * kOTile + 2 * (size_t)kABytes;
constexpr uint32_t kTmemCols = kAccs * kM;
}  // namespace xt

__device__ unsigned int g_xt_fault_flags;
// Test controls of the bounded waits, set only through mol_debug_wait_test: bit 0
// of g_xt_test_stall makes the weight producer issue no copy (so every other
// role's waits run out), g_xt_wait_limit_ns is the wall-clock limit of every wait.
__device__ unsigned int g_xt_test_stall;
__device__ unsigned long long g_xt_wait_limit_ns = kWaitLimitNs;

cudaError_t set_expand_tc_wait_test(unsigned stall, unsigned long long limit_ns) {
  cudaError_t e = cudaMemcpyToSymbol(g_xt_test_stall, &stall, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_xt_wait_limit_ns, &limit_ns, sizeof(unsigned long long));
}

cudaError_t take_expand_tc_faults(unsigned* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_xt_fault_flags, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_xt_fault_flags, &zero, sizeof(unsigned));
}

template <int BN>
__global__ void __launch_bounds__(xt::kThreads, 1)
lora_expand_tc_kernel(const __grid_constant__ CUtensorMap tmap_b, const float* __restrict__ inter,
                      int R, int S, int Ns, float scale, const float* __restrict__ topk_w,
                      const int* __restrict__ sorted_ids, const int* __restrict__ expert_ids,
                      const int* __restrict__ ntpp_ptr, int64_t numel, int num_vexperts,
                      uint16_t* __restrict__ out, int64_t out_stride, int64_t nblk, int mgroups,
                      int mtiles) {
  using namespace xt;
  constexpr int NB = kBStages, NO = kOStages;
  extern __shared__ unsigned char smem_raw[];
  // lora_b ring (TMA -> MMA), output-row ring (copiers -> epilogue), accumulators,
  // operand buffers
  __shared__ uint64_t wfull[NB], wempty[NB], ofull[NO], oempty[NO], accf[kAccs], acce[kAccs],
      bfull[2], bempty[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int m_pid[2][kRows];  // per operand buffer: pair of each row, -1 for none
  __shared__ float m_w[2][kRows];  // and its scale * routed weight
  unsigned char* smem =
      smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1024-byte aligned
  unsigned char* wbuf = smem;                                  // lora_b tiles
  unsigned char* obuf = wbuf + (size_t)NB * kBTile;             // staged output rows
  unsigned char* abuf = obuf + (size_t)NO * kOTile;             // two head + tail buffers
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    for (int s = 0; s < NB; ++s) {
      mbar_init(&wfull[s], 1);   // the TMA arrival
      mbar_init(&wempty[s], 1);  // MMA commit
    }
    for (int s = 0; s < NO; ++s) {
      mbar_init(&ofull[s], kCopiers);   // every copier thread
      mbar_init(&oempty[s], kEpiWarps);  // every epilogue warp
    }
    for (int a = 0; a < kAccs; ++a) {
      mbar_init(&accf[a], 1);
      mbar_init(&acce[a], kEpiWarps);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bfull[a], kConverters);
      mbar_init(&bempty[a], 1 + kEpiWarps);  // MMA commit + every epilogue warp
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint64_t wlim = g_xt_wait_limit_ns;
  pdl_wait();  // routing, intermediate and output rows come from earlier kernels
  pdl_launch_dependents();

  const int ntpp = __ldg(ntpp_ptr);
  const int per = S * mgroups;
  // Units: routed blocks (BLOCK_M 128) or pairs of routed blocks (BLOCK_M 64). A unit
  // is one 128-row sub-unit (a block, or a pair whose two blocks have the same
  // virtual expert) or two 64-row ones (the blocks of a pair on their own). An item is
  // a unit, a slice and a group of its m-tiles; the items cover the units below ntpp.
  constexpr int kPer = kRows / BN;  // routed blocks per unit
  const int64_t nunits = (nblk + kPer - 1) / kPer;
  const int64_t ueff = min(nunits, (int64_t)((max(ntpp, 0) + kRows - 1) / kRows));
  // items b, b + G, ... of the grid: blocks that run at the same time hold neighbouring
  // items, so the units of one virtual expert load the same lora_b tiles together
  const int64_t nitems = ueff * per, G = gridDim.x;
  // work x (2 per item: item x / 2, sub-unit x % 2) -> its first routing slot, slice,
  // m-tiles [m0, m1), rows and virtual expert; false when there is no such sub-unit
  auto work = [&](int64_t x, int64_t& slot0, int& s, int& m0, int& m1, int& nrows, int& v,
                  bool note = false) -> bool {
    const int64_t it = x >> 1;
    const int k = (int)(x & 1);
    const int64_t u = it / per;
    const int rem = (int)(it - u * per);
    s = rem / mgroups;
    const int g = rem - s * mgroups;  // the slice's m-tiles in mgroups equal groups
    m0 = g * mtiles / mgroups;
    m1 = (g + 1) * mtiles / mgroups;
    auto block = [&](int64_t t) -> int {  // expert of routed block t, -1 if none
      if (t >= nblk || t * BN >= ntpp) return -1;
      const int e = __ldg(expert_ids + t);
      if (kChecked && note && s == 0 && m0 == 0)  // the caller's expert ids, once per block
        (void)MOL_NOTE(e >= -1 && e < num_vexperts, MOL_CHECK_ROUTE_EXPERT, t);
      return e >= 0 && e < num_vexperts ? e : -1;
    };
    if (kPer == 1) {
      v = block(u);
      slot0 = u * BN;
      nrows = BN;
      return k == 0 && v >= 0;
    }
    const int e0 = block(2 * u), e1 = block(2 * u + 1);
    if (e0 >= 0 && e0 == e1) {  // one 128-row sub-unit
      v = e0;
      slot0 = 2 * u * BN;
      nrows = 2 * BN;
      return k == 0;
    }
    v = k ? e1 : e0;
    slot0 = (2 * u + k) * BN;
    nrows = BN;
    return v >= 0;
  };
  auto wtile = [&](uint32_t q) { return wbuf + (size_t)(q % NB) * kBTile; };
  auto otile = [&](uint32_t q) { return obuf + (size_t)(q % NO) * kOTile; };
  bool fault = false;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && !(g_xt_test_stall & 1u)) {  // test control: no copy, every wait runs out
      if (kChecked && blockIdx.x == 0)  // the caller's post-padded count
        (void)MOL_NOTE(ntpp >= 0 && ntpp <= nblk * BN && ntpp % BN == 0, MOL_CHECK_ROUTE_NTPP, ntpp);
      uint32_t q = 0;
      for (int64_t x = 2 * blockIdx.x; x < 2 * nitems && !fault; x += (x & 1) ? 2 * G - 1 : 1) {
        int64_t slot0;
        int s, m0, m1, nrows, v;
        if (!work(x, slot0, s, m0, m1, nrows, v, true)) continue;
        for (int m = m0; m < m1; ++m, ++q) {
          const int st = (int)(q % NB);
          if (!mbar_wait(&wempty[st], ((q / NB) & 1) ^ 1, kPolls, wlim)) {
            fault = true;
            break;
          }
          const int64_t row = ((int64_t)v * S + s) * Ns + (int64_t)m * kM;
          if (kChecked &&
              !MOL_CHECK(row >= 0 && row + kM <= (int64_t)num_vexperts * S * Ns,
                         MOL_CHECK_TMA_COORD, row)) {
            mbar_arrive_expect_tx(&wfull[st], 0u);  // the tile keeps stale data
            continue;
          }
          mbar_arrive_expect_tx(&wfull[st], (uint32_t)kBTile);
          tma_load_2d(wtile(q), &tmap_b, 0, (int)row, &wfull[st]);
        }
      }
      // after a timeout, let the last copies into each tile land (bounded) before the
      // block's shared memory is released
      if (fault)
        for (uint32_t u = q > (uint32_t)NB ? q - NB : 0; u < q; ++u)
          mbar_wait(&wfull[u % NB], (u / NB) & 1, kPolls, wlim);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = IDesc<kRows, kM>::kValue;
      uint32_t q = 0, n = 0, rn = 0;  // m-tiles, accumulators, runs of one (block, slice)
      int64_t key = -1;
      int j = 0;
      uint32_t ah = 0, at = 0;
      for (int64_t x = 2 * blockIdx.x; x < 2 * nitems && !fault; x += (x & 1) ? 2 * G - 1 : 1) {
        int64_t slot0;
        int s, m0, m1, nrows, v;
        if (!work(x, slot0, s, m0, m1, nrows, v)) continue;
        if (slot0 * S + s != key) {  // a new run: its operand buffer
          if (key >= 0) umma_commit(&bempty[j]);  // the last run's buffer, once its MMAs are done
          key = slot0 * S + s;
          j = (int)(rn & 1);
          if (!mbar_wait(&bfull[j], (rn >> 1) & 1, kPolls, wlim)) {
            fault = true;
            break;
          }
          ++rn;
          ah = smem_u32(abuf + (size_t)j * kABytes);
          at = ah + kATile;
        }
        for (int m = m0; m < m1; ++m, ++q, ++n) {
          const int st = (int)(q % NB);
          const int a = (int)(n % kAccs);
          if (!mbar_wait(&acce[a], ((n / kAccs) & 1) ^ 1, kPolls, wlim) ||
              !mbar_wait(&wfull[st], (q / NB) & 1, kPolls, wlim)) {
            fault = true;
            break;
          }
          // the head / tail operands were written through the generic proxy
          // (st.shared); the MMAs read them through the async proxy
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(a * kM);
          const uint32_t sb = smem_u32(wtile(q));
#pragma unroll
          for (int kk = 0; kk < kRank / 16; ++kk)  // 16 k = 32 bytes along the swizzled row
            umma_bf16(d, sw128_desc(ah + kk * 32), sw128_desc(sb + kk * 32), idesc, kk ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < kRank / 16; ++kk)
            umma_bf16(d, sw128_desc(at + kk * 32), sw128_desc(sb + kk * 32), idesc, 1u);
          umma_commit(&wempty[st]);  // the lora_b tile is free once these MMAs have read it
          umma_commit(&accf[a]);
        }
      }
      if (key >= 0 && !fault) umma_commit(&bempty[j]);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ converters
    const int l = tid - 64;  // 0 .. kConverters-1
    uint32_t rn = 0;
    int64_t key = -1;
    for (int64_t x = 2 * blockIdx.x; x < 2 * nitems && !fault; x += (x & 1) ? 2 * G - 1 : 1) {
      int64_t slot0;
      int s, m0, m1, nrows, v;
      if (!work(x, slot0, s, m0, m1, nrows, v)) continue;
      if (slot0 * S + s == key) continue;  // the run's operands are in place already
      key = slot0 * S + s;
      const int j = (int)(rn & 1);
      // the converters take every wait's outcome together (they meet at named barriers)
      if (!named_sync_and(2, kConverters, mbar_wait(&bempty[j], ((rn >> 1) & 1) ^ 1, kPolls, wlim))) {
        fault = true;
        break;
      }
      ++rn;
      // pair ids and weights of the sub-unit's rows
      for (int r = l; r < kRows; r += kConverters) {
        const int pid = r < nrows ? __ldg(sorted_ids + slot0 + r) : -1;
        if (kChecked && r < nrows)  // the caller's slots
          (void)MOL_NOTE(pid >= 0 && (int64_t)pid <= numel, MOL_CHECK_ROUTE_PAIR, slot0 + r);
        const bool ok = pid >= 0 && (int64_t)pid < numel;
        m_pid[j][r] = ok ? pid : -1;
        m_w[j][r] = ok && topk_w ? scale * __ldg(topk_w + pid) : scale;
      }
      named_sync(2, kConverters);  // every converter sees the sub-unit's pair ids
      // intermediate rows (slice s) as bf16 head and tail, 128-byte swizzled:
      // 16-byte chunk c (8 values) of row r at r * 128 + ((c ^ (r & 7)) << 4)
      unsigned char* ah = abuf + (size_t)j * kABytes;
      unsigned char* at = ah + kATile;
#pragma unroll
      for (int k = l; k < kRows * 8; k += kConverters) {
        if (k >= nrows * 8) break;
        const int r = k >> 3, c = k & 7;
        const int pid = m_pid[j][r];
        uint4 h = make_uint4(0, 0, 0, 0), tl = make_uint4(0, 0, 0, 0);
        if (pid >= 0) {
          const float* src = inter + (int64_t)pid * R + s * kRank + c * 8;
          const float4 a0 = ld_l2_f4(src), a1 = ld_l2_f4(src + 4);
          split_bf16x2(a0.x, a0.y, h.x, tl.x);
          split_bf16x2(a0.z, a0.w, h.y, tl.y);
          split_bf16x2(a1.x, a1.y, h.z, tl.z);
          split_bf16x2(a1.z, a1.w, h.w, tl.w);
        }
        const int off = r * 128 + ((c ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(ah + off) = h;
        *reinterpret_cast<uint4*>(at + off) = tl;
      }
      fence_proxy_async_smem();  // generic writes, read next through the async proxy
      mbar_arrive(&bfull[j]);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ copiers
    const int l = tid - 192;  // 0 .. kCopiers-1
    // a copier always moves 16-byte chunk c of rows r0, r0 + kRowStep, ... of an m-tile
    constexpr int kRowStep = kCopiers / 16, kMine = kRows / kRowStep;
    const int c = l & 15, r0 = l >> 4;
    const uint16_t* src[kMine];  // per run: the rows' first output column of the slice
    uint32_t q = 0, rn = 0;
    int64_t key = -1;
    int j = 0;
    for (int64_t x = 2 * blockIdx.x; x < 2 * nitems && !fault; x += (x & 1) ? 2 * G - 1 : 1) {
      int64_t slot0;
      int s, m0, m1, nrows, v;
      if (!work(x, slot0, s, m0, m1, nrows, v)) continue;
      if (slot0 * S + s != key) {  // a new run: its pair ids (the copiers meet at named barriers)
        key = slot0 * S + s;
        j = (int)(rn & 1);
        if (!named_sync_and(3, kCopiers, mbar_wait(&bfull[j], (rn >> 1) & 1, kPolls, wlim))) {
          fault = true;
          break;
        }
        ++rn;
#pragma unroll
        for (int i = 0; i < kMine; ++i) {
          const int pid = m_pid[j][r0 + i * kRowStep];
          src[i] = pid >= 0 ? out + (int64_t)pid * out_stride + (int64_t)s * Ns + c * 8 : nullptr;
        }
      }
      // output rows of each m-tile: 256 bytes per real row, 16 chunks of 16 bytes
      for (int m = m0; m < m1 && !fault; ++m, ++q) {
        const int st = (int)(q % NO);
        if (!named_sync_and(3, kCopiers, mbar_wait(&oempty[st], ((q / NO) & 1) ^ 1, kPolls, wlim))) {
          fault = true;
          break;
        }
        unsigned char* ot = otile(q) + r0 * kOutPitch + c * 16;
#pragma unroll
        for (int i = 0; i < kMine; ++i)
          if (src[i]) cp_async16_zfill(ot + i * kRowStep * kOutPitch, src[i] + m * kM, 16u);
        cp_async_arrive_noinc(&ofull[st]);
      }
    }
    cp_async_wait_all();  // no copy of this thread is left in flight at exit
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;             // tensor-memory lanes 32*quarter .. +31 = rows
    const int half = (warp - 10) >> 2;        // output columns [64 * half, 64 * half + 64)
    const int r = quarter * 32 + lane;        // this thread's row of the sub-unit
    bool has_rows = false;                    // a 64-row sub-unit: two quarters hold no row
    uint32_t q = 0, n = 0, rn = 0;
    int64_t key = -1;
    int j = 0;
    float w = 0.f;
    for (int64_t x = 2 * blockIdx.x; x < 2 * nitems && !fault; x += (x & 1) ? 2 * G - 1 : 1) {
      int64_t slot0;
      int s, m0, m1, nrows, v;
      if (!work(x, slot0, s, m0, m1, nrows, v)) continue;
      if (slot0 * S + s != key) {  // a new run
        if (key >= 0 && lane == 0) mbar_arrive(&bempty[j]);  // done with the last run's buffer
        key = slot0 * S + s;
        j = (int)(rn & 1);
        // the block's pair ids and weights (written before the buffer's "full" arrival)
        if (!__all_sync(0xffffffffu, mbar_wait(&bfull[j], (rn >> 1) & 1, kPolls, wlim))) {
          fault = true;
          break;
        }
        ++rn;
        has_rows = quarter * 32 < nrows;
        w = has_rows ? m_w[j][r] : 0.f;
      }
      for (int m = m0; m < m1; ++m, ++q, ++n) {
        const int st = (int)(q % NO);
        const int a = (int)(n % kAccs);
        // tcgen05.ld is warp-collective: the lanes agree on the outcome of the waits
        if (!__all_sync(0xffffffffu, mbar_wait(&accf[a], (n / kAccs) & 1, kPolls, wlim) &&
                                         mbar_wait(&ofull[st], (q / NO) & 1, kPolls, wlim))) {
          fault = true;
          break;
        }
        tc_fence_after();
        unsigned char* ot = otile(q);
        if (has_rows) {
          // this thread's 64 columns of its row: the sums back into the staged row
          unsigned char* orow = ot + r * kOutPitch + half * 128;
          const uint32_t base =
              tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(a * kM + half * 64);
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 32) {
            float val[32];
            tmem_ld32(base + (uint32_t)c0, val);
#pragma unroll
            for (int g = 0; g < 4; ++g) {  // 8 columns: one 16-byte piece of the row
              uint4 o = *reinterpret_cast<const uint4*>(orow + (c0 + 8 * g) * 2);
              uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float lo = fmaf(w, val[8 * g + 2 * u], bf16_lo(ow[u]));
                const float hi = fmaf(w, val[8 * g + 2 * u + 1], bf16_hi(ow[u]));
                ow[u] = pack_bf16x2(lo, hi);
              }
              *reinterpret_cast<uint4*>(orow + (c0 + 8 * g) * 2) = o;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (has_rows) {
          // the warp's 32 rows x 64 columns back to global memory, 128 contiguous
          // bytes per row: eight lanes per row, four rows per instruction
          const int64_t col = (int64_t)s * Ns + (int64_t)m * kM + half * 64 + (lane & 7) * 8;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = quarter * 32 + i * 4 + (lane >> 3);
            const int p = m_pid[j][rr];
            if (p >= 0 && MOL_CHECK((int64_t)p < numel, MOL_CHECK_ROW, p))
              *reinterpret_cast<uint4*>(out + (int64_t)p * out_stride + col) =
                  *reinterpret_cast<const uint4*>(ot + rr * kOutPitch + half * 128 + (lane & 7) * 16);
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&acce[a]);
          mbar_arrive(&oempty[st]);
        }
      }
      if (fault) break;
    }
    if (key >= 0 && !fault && lane == 0) mbar_arrive(&bempty[j]);
  }

  if (fault) atomicOr(&g_xt_fault_flags, kFaultBulkTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// --- host side ----------------------------------------------------------------

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_xt_encode = nullptr;
std::once_flag g_xt_encode_once;
cudaError_t g_xt_encode_status = cudaSuccess;

int xt_device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}
}  // namespace

bool expand_tc_fits(int64_t numel, int num_vexperts, int r, int Ns, int block_m,
                    int64_t out_stride, bool adapter_arrays) {
  if (adapter_arrays || numel <= 0 || r != xt::kRank || Ns % xt::kM != 0) return false;
  if (block_m != 64 && block_m != 128) return false;
  if (out_stride % 8 != 0) return false;
  // many rows per virtual expert: on average at least 32 pairs each
  return numel >= 32 * std::min<int64_t>(numel, num_vexperts);
}

cudaError_t prepare_expand_tc_kernels() {
  cudaError_t e = cudaFuncSetAttribute(lora_expand_tc_kernel<64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)xt::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(lora_expand_tc_kernel<128>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)xt::kSmem);
}

cudaError_t launch_expand_tc(const float* inter, const void* lora_b, int S, int Ns, float scale,
                             const float* topk_weights, const int32_t* sorted_ids,
                             const int32_t* expert_ids, const int32_t* ntpp, int64_t capacity,
                             int block_m, int64_t numel, int num_vexperts, void* out,
                             int64_t out_stride, cudaStream_t stream) {
  std::call_once(g_xt_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    g_xt_encode_status = cudaGetDriverEntryPointByVersion(
        "cuTensorMapEncodeTiled", reinterpret_cast<void**>(&g_xt_encode), 12000, cudaEnableDefault,
        &q);
    if (g_xt_encode_status == cudaSuccess && (q != cudaDriverEntryPointSuccess || !g_xt_encode))
      g_xt_encode_status = cudaErrorNotSupported;
  });
  if (g_xt_encode_status != cudaSuccess) return g_xt_encode_status;
  const int64_t nblk = capacity / block_m;
  if (numel == 0 || nblk == 0) return cudaSuccess;
  // lora_b as a 2-D tensor: V * S * Ns rows of 64 bf16 (128-byte rows)
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)xt::kRank,
                              (cuuint64_t)num_vexperts * (cuuint64_t)S * (cuuint64_t)Ns};
  const cuuint64_t strides[1] = {(cuuint64_t)xt::kRank * 2};
  const cuuint32_t box[2] = {(cuuint32_t)xt::kRank, (cuuint32_t)xt::kM};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult cr = g_xt_encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(lora_b),
                                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const int mtiles = Ns / xt::kM;
  const int mgroups = (mtiles + xt::kMGroup - 1) / xt::kMGroup;
  const int64_t n_items = (nblk * block_m + xt::kRows - 1) / xt::kRows * S * mgroups;
  const dim3 grid((unsigned)std::min<int64_t>(n_items, (int64_t)xt_device_sms()));
  const int R = S * xt::kRank;
  uint16_t* o = static_cast<uint16_t*>(out);
  if (block_m == 64)
    return launch_pdl(lora_expand_tc_kernel<64>, grid, dim3(xt::kThreads), xt::kSmem,
                      stream, map, inter, R, S, Ns, scale, topk_weights, sorted_ids, expert_ids,
                      ntpp, numel, num_vexperts, o, out_stride, nblk, mgroups, mtiles);
  return launch_pdl(lora_expand_tc_kernel<128>, grid, dim3(xt::kThreads), xt::kSmem,
                    stream, map, inter, R, S, Ns, scale, topk_weights, sorted_ids, expert_ids, ntpp,
                    numel, num_vexperts, o, out_stride, nblk, mgroups, mtiles);
}

cudaError_t take_expand_tc_checks(unsigned long long* first, unsigned long long* count) {
  CheckRecord r;
  const cudaError_t e = take_check_record_here(&r);
  *first = r.first;
  *count = r.count;
  return e;
}

}  // namespace mol
