// Device helpers shared by the MoL kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mol.h"

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
// 16-byte load that bypasses L1 (data written by the preceding grid).
MOL_DEV float4 ld_l2_f4(const float* p) {
  float4 r;
  asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

// Programmatic dependent launch. wait: block until the preceding grid in the
// stream has completed and its writes are visible (a no-op when the launch
// has no programmatic dependency). launch_dependents: let the next grid's
// blocks be scheduled once every block of this grid has issued it.
MOL_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOL_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// mbarrier + bulk async copy (TMA, 1-D) into shared memory.
MOL_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
MOL_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
MOL_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
MOL_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Copy `bytes` (multiple of 16; both addresses 16-byte aligned) from global to
// shared memory; completion is counted on `bar`.
MOL_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
MOL_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
MOL_DEV uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Longest time a barrier wait may take before it gives up (the waits inside
// these kernels last microseconds; no kernel runs for more than milliseconds).
constexpr uint64_t kWaitLimitNs = 1000000000ull;
// Bounded wait: gives up, returning false, after `max_iter` polls or
// `limit_ns` of wall-clock time (one second by default), whichever comes first
// (a poll may suspend the thread for a hardware-defined time, so the clock
// bounds the total).
MOL_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_iter,
                       uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < max_iter; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
  return false;
}

MOL_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Barrier 1 among the first `threads` threads of the block (0 is __syncthreads).
MOL_DEV void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
// Barrier `id` among `threads` threads that also ANDs a predicate over them:
// every participant returns true only if every participant passed true.
MOL_DEV bool named_sync_and(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}
MOL_DEV uint4 lds16(const void* p) { return *reinterpret_cast<const uint4*>(p); }
MOL_DEV uint2 lds8(const void* p) { return *reinterpret_cast<const uint2*>(p); }
// 16-byte copy global -> shared through L2 (cp.async): src_bytes of 16 are
// read, the rest of the 16 bytes zero-filled (0: nothing is read).
MOL_DEV void cp_async16_zfill(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
// Virtual id of one (token, slot) pair: negative ids stay as they are; a token
// without a valid adapter, or an expert id past the experts, gives -1; else
// base + lora * E.
MOL_DEV int remap_one(int base, int lora, int num_experts, int max_loras) {
  if (base < 0) return base;
  if (lora < 0 || lora >= max_loras || base >= num_experts) return -1;
  return base + lora * num_experts;
}
// 32-bit load from L2 (no L1 allocation, so no stale L1 line is read).
MOL_DEV int ld_cg_i32(const int* p) {
  int v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
// Asks L2 to load `bytes` (a multiple of 16) from 16-byte aligned global memory,
// asynchronously, in 32 KB requests; nothing waits for it.
MOL_DEV void prefetch_l2(const void* p, int64_t bytes) {
  const char* c = static_cast<const char*>(p);
  for (int64_t o = 0; o < bytes; o += 32768) {
    const uint32_t n = (uint32_t)(bytes - o < 32768 ? bytes - o : 32768);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c + o), "r"(n) : "memory");
  }
}
// Waits until every cp.async this thread issued has landed.
MOL_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Closes this thread's current group of cp.async copies.
MOL_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's committed groups are still in flight.
template <int N>
MOL_DEV void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Error bits a kernel records instead of hanging or trapping.
constexpr unsigned kFaultBulkTimeout = 1u;

// Device-side index checks. Each translation unit owns one check record: the
// first failed check's site and value, and the number of failed checks.
// MOL_CHECK(cond, site, value) guards an access whose bounds hold by
// construction: the release build compiles it to `true`; the checked build
// (MOL_CHECKED) records a false `cond` and yields it, and the caller skips the
// access. MOL_NOTE(cond, site, value) guards against caller data that every
// build skips when `cond` is false: it yields `cond` in both builds and the
// checked build also records it. `kChecked` lets a caller guard a skip that
// only the checked build takes (`if (kChecked && !ok) return;`).
struct CheckRecord {
  unsigned long long first;  // (site << 48) | (value & 0xFFFFFFFFFFFF), 0 = none
  unsigned long long count;
};
#ifdef MOL_CHECKED
static __device__ CheckRecord g_check_record;
__device__ __noinline__ static void check_record(unsigned site, long long value) {
  const unsigned long long code =
      ((unsigned long long)site << 48) | ((unsigned long long)value & 0xFFFFFFFFFFFFull);
  atomicCAS(&g_check_record.first, 0ull, code);
  atomicAdd(&g_check_record.count, 1ull);
}
MOL_DEV bool check_cond(bool cond, unsigned site, long long value) {
  if (!cond) check_record(site, value);
  return cond;
}
#define MOL_CHECK(cond, site, value) (::mol::check_cond((cond), (site), (long long)(value)))
#define MOL_NOTE(cond, site, value) (::mol::check_cond((cond), (site), (long long)(value)))
// Host: reads and clears this translation unit's record on the current device.
static inline cudaError_t take_check_record_here(CheckRecord* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_check_record, sizeof(CheckRecord));
  if (e != cudaSuccess) return e;
  const CheckRecord zero = {0ull, 0ull};
  return cudaMemcpyToSymbol(g_check_record, &zero, sizeof(CheckRecord));
}
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
// (the operands stay unevaluated: sizeof only marks them used)
#define MOL_CHECK(cond, site, value) ((void)sizeof(cond), (void)sizeof(value), true)
#define MOL_NOTE(cond, site, value) ((void)sizeof(value), (cond))
static inline cudaError_t take_check_record_here(CheckRecord* out) {
  out->first = 0ull;
  out->count = 0ull;
  return cudaSuccess;
}
#endif

MOL_DEV unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive scan of one int per thread over the block; `total` = sum of all.
template <int THREADS>
MOL_DEV int block_exclusive_scan(int v, int* sh, int& total) {
  constexpr int NW = THREADS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < NW ? sh[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < NW) sh[lane] = wi - w;
    if (lane == NW - 1) sh[NW] = wi;
  }
  __syncthreads();
  const int res = sh[warp] + incl - v;
  total = sh[NW];
  __syncthreads();
  return res;
}

// Checked build: records the caller's routing words of routed block t that
// every build skips (a bad num_tokens_post_padded, an expert id outside
// [-1, V) below it, a slot outside [0, numel] of a block with an expert).
// Every thread of one item of the block calls it with its slot (-1 past block_m).
MOL_DEV void note_block_routing(int64_t t, int ntpp, int v, int slot, int block_m, int64_t numel,
                                int num_vexperts, int64_t capacity) {
  if (!kChecked) return;
  const int tid = threadIdx.x;
  const bool below = t * block_m < ntpp;
  if (tid == 0) {
    (void)MOL_NOTE(ntpp >= 0 && ntpp <= capacity && ntpp % block_m == 0, MOL_CHECK_ROUTE_NTPP, ntpp);
    if (below) (void)MOL_NOTE(v >= -1 && v < num_vexperts, MOL_CHECK_ROUTE_EXPERT, t);
  }
  if (below && v >= 0 && v < num_vexperts && tid < block_m)
    (void)MOL_NOTE(slot >= 0 && (int64_t)slot <= numel, MOL_CHECK_ROUTE_PAIR, t * block_m + tid);
}

// Compact the valid pair ids of one block into `rows`, keeping slot order.
// `id` is this thread's slot of the block (-1 for threads past block_m); ids
// outside [0, numel) are padding. Needs blockDim.x >= block_m and a multiple
// of 32; every thread of the block must call it. Returns the row count.
MOL_DEV int compact_block_rows(int id, int64_t numel, int* rows, int* warp_counts) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const bool ok = id >= 0 && (int64_t)id < numel;
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
