// Virtual top-k remap and align_block_size with a sentinel bucket (sm_103a).
//
// Remap: sglang PR 24171 prhub summary, "Key source snippets"
// (_fused_virtual_topk_ids_kernel: keep negative ids, else base + lora * E);
// fork PR #24 "fix(lora): -1 = no adapter" commit (no-adapter tokens get no
// delta, so they are remapped to -1).
// Align: sglang PR 24171 prhub summary, "Key source snippets"
// (_align_block_size_torch: sentinel bucket V, bucket_count = V + 1, sentinel
// blocks keep -1); sglang PR 24262 prhub summary, "Implementation breakdown"
// (histogram, prefix sum, expert_ids, scatter in a few launches, no host
// synchronisation; up to 8192 buckets).
//
// Design. The order inside a bucket is ascending flat index, so the scatter
// is a stable counting sort. Pairs are cut into tiles (one thread block each);
// a tile is cut into 8 (or 16) contiguous warp segments; a warp walks its
// segment in rounds of 32 pairs in order. Inside a round, __match_any_sync
// gives each lane the lanes holding the same bucket; a per-warp shared-memory
// table of 16-bit counters (one per bucket) carries the running count across
// rounds. Pass 1 counts, a column scan over the warp tables turns counts into
// per-warp bases, pass 2 recomputes each pair's stable rank inside the tile.
// Everything is ordered by construction (tile < warp < round < lane), so the
// result is bit-reproducible with no atomics. With one tile the same block
// finishes the job (bucket scan, expert_ids, scatter): one launch. Up to
// 131072 pairs the tiles are the thread blocks of one cluster (up to 16) and
// the cross-tile steps go through distributed shared memory: each block sums
// the tiles' counts of its share of the buckets and writes, into every tile's
// shared memory, that tile's base in each bucket relative to the share, and
// the shares' padded totals are exchanged -- one launch, no workspace, two
// cluster barriers. Beyond that, per-tile histograms go to the workspace, one
// block scans them, and a third launch scatters.

#include <algorithm>

#include "mol_device.cuh"
#include "mol_internal.h"

namespace mol {

constexpr int kAlignThreads = 256;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kScanThreads = 1024;
constexpr int kTileMin = 4096;
constexpr int kMaxTiles = 128;
constexpr int kAlignSmemMax = 200 * 1024;
constexpr int kClusterTileMax = 16384;  // pairs per block of the cluster align
constexpr int kClusterMax = 16;         // blocks in one cluster (above 8 where the device allows)
constexpr int64_t kClusterPairs = 8LL * kClusterTileMax;  // largest numel of the cluster align

MOL_DEV int bucket_of(int vid, int num_vexperts) {
  return (vid >= 0 && vid < num_vexperts) ? vid : num_vexperts;
}

__global__ void virtual_topk_kernel(const int* __restrict__ topk_ids, const int* __restrict__ lora_ids,
                                    int64_t numel, int topk, int num_experts, int max_loras,
                                    int* __restrict__ vtopk) {
  pdl_wait();
  pdl_launch_dependents();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < numel;
       i += (int64_t)gridDim.x * blockDim.x) {
    vtopk[i] = remap_one(topk_ids[i], lora_ids[i / topk], num_experts, max_loras);
  }
}

// Per-token adapter ids (fork PR #24, "feat(lora): base takes no pool slot"
// and "fix(lora): complete the '-1 = no adapter' sentinel guards"): token t
// takes the slot of the request whose segment [seg[q], seg[q+1]) holds it,
// found by binary search; a negative slot, one >= max_loras, or (checked only
// after those two) an adapter of rank 0 gives -1, as does a token outside
// every segment.
__global__ void token_lora_ids_kernel(const int* __restrict__ weight_indices,
                                      const int* __restrict__ seg_indptr, int num_reqs,
                                      int64_t num_tokens, int max_loras,
                                      const int* __restrict__ lora_ranks, int* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < num_tokens;
       t += (int64_t)gridDim.x * blockDim.x) {
    int lo = 0, hi = num_reqs;  // first q with seg[q] > t
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if ((int64_t)__ldg(seg_indptr + mid) <= t)
        lo = mid + 1;
      else
        hi = mid;
    }
    const int q = lo - 1;
    int id = -1;
    if (q >= 0 && t < (int64_t)__ldg(seg_indptr + q + 1)) {
      const int w = __ldg(weight_indices + q);
      if (w >= 0 && w < max_loras && (!lora_ranks || __ldg(lora_ranks + w) > 0)) id = w;
    }
    out[t] = id;
  }
}

// counts[b] -> exclusive offsets of the BM-padded buckets (in place); returns
// the padded total. block_m is a power of two (validated on the host): padding
// and block indices are masks and shifts.
template <int THREADS>
MOL_DEV int bucket_scan(int* counts, int nb, int block_m, int* sh) {
  const int pad = block_m - 1;
  const int per = (nb + THREADS - 1) / THREADS;
  const int b0 = min((int)threadIdx.x * per, nb), b1 = min(b0 + per, nb);
  int local = 0;
  for (int b = b0; b < b1; ++b) local += (counts[b] + pad) & ~pad;
  int total;
  int run = block_exclusive_scan<THREADS>(local, sh, total);
  for (int b = b0; b < b1; ++b) {
    const int pb = (counts[b] + pad) & ~pad;
    counts[b] = run;
    run += pb;
  }
  return total;
}

// expert_ids of every block and num_tokens_post_padded from the offsets of
// bucket_scan (every thread of the block, after a barrier that follows it).
template <int THREADS>
MOL_DEV void write_blocks(const int* offs, int nb, int num_vexperts, int block_m, int64_t capacity,
                          int total, int* __restrict__ expert_ids, int* __restrict__ ntpp_out) {
  const int lg = __ffs(block_m) - 1;
  const int per = (nb + THREADS - 1) / THREADS;
  const int b0 = min((int)threadIdx.x * per, nb), b1 = min(b0 + per, num_vexperts);
  for (int b = b0; b < b1; ++b) {
    const int t0 = offs[b] >> lg, t1 = (b + 1 < nb ? offs[b + 1] : total) >> lg;
    for (int t = t0; t < t1; ++t)
      if (MOL_CHECK(t < (capacity >> lg), MOL_CHECK_ALIGN_BLOCK, t)) expert_ids[t] = b;
  }
  const int64_t nblk = capacity >> lg;
  for (int64_t t = (offs[num_vexperts] >> lg) + threadIdx.x; t < nblk; t += THREADS)
    expert_ids[t] = -1;
  if (threadIdx.x == 0) {
    (void)MOL_CHECK(total <= capacity, MOL_CHECK_ALIGN_TOTAL, total);
    *ntpp_out = total;
  }
}

// Both: offsets in place, then expert_ids and num_tokens_post_padded.
template <int THREADS>
MOL_DEV void bucket_offsets(int* counts, int nb, int num_vexperts, int block_m, int64_t capacity,
                            int* __restrict__ expert_ids, int* __restrict__ ntpp_out, int* sh) {
  const int total = bucket_scan<THREADS>(counts, nb, block_m, sh);
  __syncthreads();
  write_blocks<THREADS>(counts, nb, num_vexperts, block_m, capacity, total, expert_ids, ntpp_out);
}

// Pass 1: the warp's bucket counts over its contiguous segment [s0, s1) of the
// tile's keys, in rounds of 32 in order, into its 16-bit table `mine`.
MOL_DEV void warp_count(const uint16_t* keys, int s0, int s1, uint16_t* mine, int lane) {
  for (int r = s0; r < s1; r += 32) {
    const int q = r + lane;
    const bool valid = q < s1;
    const unsigned key = valid ? keys[q] : 0xFFFFu;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (valid && lane == __ffs(peers) - 1) mine[key] = (uint16_t)(mine[key] + __popc(peers));
    __syncwarp();
  }
}

// Pass 2: the same rounds again; `mine` holds the warp's base in each bucket
// inside the tile. emit(q, key, rank) gets each pair's stable rank in the tile.
template <typename F>
MOL_DEV void warp_rank(const uint16_t* keys, int s0, int s1, uint16_t* mine, int lane, F&& emit) {
  for (int r = s0; r < s1; r += 32) {
    const int q = r + lane;
    const bool valid = q < s1;
    const unsigned key = valid ? keys[q] : 0xFFFFu;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int base = valid ? (int)mine[key] : 0;
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) mine[key] = (uint16_t)(base + __popc(peers));
    __syncwarp();
    if (valid) emit(q, (int)key, base + __popc(peers & lanemask_lt()));
  }
}

// Pass 1 that also keeps each pair's stable rank inside its warp's segment
// (lrank[q]), so that no second pass of matches is needed: with the column-
// scanned tables, a pair's rank inside the tile is tbl[warp][key] + lrank[q].
MOL_DEV void warp_count_rank(const uint16_t* keys, int s0, int s1, uint16_t* mine, int lane,
                             uint16_t* lrank) {
  warp_rank(keys, s0, s1, mine, lane, [&](int q, int, int lr) { lrank[q] = (uint16_t)lr; });
}

// Column scan: the warp tables become exclusive per-warp bases inside the tile;
// total(b, n) receives the tile's count of bucket b.
// Two buckets per thread and access (32-bit words of two 16-bit counters, rows
// of nb_pad, a multiple of 8, counters: 16-byte aligned rows), every warp's
// word loaded first: the scan moves the tables through shared memory at full
// width.
template <int WARPS, typename F>
MOL_DEV void column_scan(uint16_t* tbl, int nb, int nb_pad, F&& total) {
  uint32_t* t32 = reinterpret_cast<uint32_t*>(tbl);
  const int row = nb_pad / 2;
  for (int j = threadIdx.x; 2 * j < nb; j += WARPS * 32) {
    uint32_t c[WARPS];
#pragma unroll
    for (int w = 0; w < WARPS; ++w) c[w] = t32[w * row + j];
    uint32_t lo = 0, hi = 0;  // running sums of bucket 2j and 2j + 1
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      t32[w * row + j] = lo | (hi << 16);
      lo += c[w] & 0xFFFFu;
      hi += c[w] >> 16;
    }
    total(2 * j, (int)lo);
    if (2 * j + 1 < nb) total(2 * j + 1, (int)hi);
  }
}

// ONE: pass 1 keeps each pair's rank inside its warp's segment (lrank, in
// shared memory after the keys), and pass 2 needs no matches.
template <bool REMAP, bool ONE>
__global__ void __launch_bounds__(kAlignThreads, 1)
align_tile_kernel(const int* __restrict__ src, const int* __restrict__ lora_ids, int topk,
                  int num_experts, int max_loras, int* __restrict__ vtopk_out, int64_t numel,
                  int num_vexperts, int block_m, int64_t capacity, int tile, int tiles, int nb_pad,
                  int* __restrict__ sorted_ids, int* __restrict__ expert_ids,
                  int* __restrict__ ntpp_out, int* __restrict__ ws_hist,
                  int* __restrict__ ws_rank, int trigger) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int sh_scan[kAlignWarps + 1];
  const int nb = num_vexperts + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint16_t* tbl = reinterpret_cast<uint16_t*>(smem);   // [kAlignWarps][nb_pad]
  uint16_t* keys = tbl + kAlignWarps * nb_pad;         // [tile]
  uint16_t* lrank = keys + tile;                       // ONE: [tile]
  int* offs = reinterpret_cast<int*>(keys + (ONE ? 2 : 1) * tile);  // [nb], single-tile only
  const bool fused = (tiles == 1);

  if ((int)blockIdx.x < tiles) {  // shared memory only: may overlap the previous kernel
    uint4* t4 = reinterpret_cast<uint4*>(tbl);
    const int n4 = kAlignWarps * nb_pad / 8;
    for (int q = tid; q < n4; q += kAlignThreads) t4[q] = make_uint4(0, 0, 0, 0);
  }
  // The single-block align writes the final routing. Called on its own
  // (trigger = 0) it lets its dependents start only when it exits, so a kernel
  // that follows it may read the routing before its own griddepcontrol.wait.
  // Inside mol_lora_forward the next kernel waits before reading the routing:
  // it may start once this kernel has waited for the previous one (trigger = 1),
  // or at once when the caller's ids were complete before the previous kernel
  // began (trigger = 2: the next kernel reads the ids early). With several
  // tiles the scatter kernel is the last writer and plays that role.
  if (trigger == 2) pdl_launch_dependents();
  const int64_t t0 = (int64_t)blockIdx.x * tile;
  const int tlen = (int)max((int64_t)0, min((int64_t)tile, numel - t0));
  const int seg = tile / kAlignWarps;
  const int s0 = warp * seg, s1 = min(s0 + seg, tlen);
  uint16_t* mine = tbl + warp * nb_pad;
  // Keys, per-warp counts, the tile's bucket counts and (one tile) the bucket
  // offsets: in shared memory only, from the ids.
  auto count_keys = [&]() {
    __syncthreads();
    if constexpr (ONE)  // pass 1: per-warp counts over the warp's segment (and the ranks)
      warp_count_rank(keys, s0, s1, mine, lane, lrank);
    else
      warp_count(keys, s0, s1, mine, lane);
    __syncthreads();
    // column scan: warp tables become exclusive bases; the tile total per bucket
    // goes to shared memory (one tile) or to the workspace histogram
    column_scan<kAlignWarps>(tbl, nb, nb_pad, [&](int b, int n) {
      const int64_t w = (int64_t)blockIdx.x * nb + b;
      if (fused)
        offs[b] = n;
      else if (MOL_CHECK(w < (int64_t)tiles * nb, MOL_CHECK_ALIGN_WORKSPACE, w))
        ws_hist[w] = n;
    });
    __syncthreads();
  };
  // trigger = 2, one tile: the ids are older than the previous kernel, so all of
  // that runs before the wait; only the writes wait (the virtual ids stay in
  // registers until then: one tile holds at most kTileMin pairs).
  const bool ids_early = trigger == 2 && fused;
  int total = 0;
  int vkeep[kTileMin / kAlignThreads];
  if (ids_early) {
#pragma unroll
    for (int j = 0; j < kTileMin / kAlignThreads; ++j) {
      const int q = tid + j * kAlignThreads;
      vkeep[j] = 0;
      if (q < tlen) {
        const int64_t i = t0 + q;
        vkeep[j] = REMAP ? remap_one(src[i], lora_ids[i / topk], num_experts, max_loras) : src[i];
        keys[q] = (uint16_t)bucket_of(vkeep[j], num_vexperts);
      }
    }
    count_keys();
    total = bucket_scan<kAlignThreads>(offs, nb, block_m, sh_scan);
    __syncthreads();  // every bucket's offset is in place
  }
  pdl_wait();  // inputs and the routing buffers belong to earlier kernels until here
  if (trigger == 1 || (trigger == 0 && tiles > 1)) pdl_launch_dependents();

  // One tile, ids read after the wait: they are loaded before the padding fill, so that
  // their latency overlaps it (raw ids and adapter ids in registers).
  const bool ids_first = fused && !ids_early;
  int lkeep[kTileMin / kAlignThreads];
  if (ids_first) {
#pragma unroll
    for (int j = 0; j < kTileMin / kAlignThreads; ++j) {
      const int q = tid + j * kAlignThreads;
      vkeep[j] = q < tlen ? src[t0 + q] : -1;
      lkeep[j] = (REMAP && q < tlen) ? lora_ids[(t0 + q) / topk] : -1;
    }
  }

  // Every slot starts as padding (value numel); real pairs overwrite theirs.
  for (int64_t q = (int64_t)blockIdx.x * kAlignThreads + tid; q < capacity;
       q += (int64_t)gridDim.x * kAlignThreads)
    sorted_ids[q] = (int)numel;
  if ((int)blockIdx.x >= tiles) return;  // fill-only block

  if (ids_early) {
    if (REMAP) {
#pragma unroll
      for (int j = 0; j < kTileMin / kAlignThreads; ++j) {
        const int q = tid + j * kAlignThreads;
        if (q < tlen) vtopk_out[t0 + q] = vkeep[j];
      }
    }
    write_blocks<kAlignThreads>(offs, nb, num_vexperts, block_m, capacity, total, expert_ids,
                                ntpp_out);
    __syncthreads();  // the padding fill lands before the scatter overwrites it
  } else {
    if (ids_first) {
#pragma unroll
      for (int j = 0; j < kTileMin / kAlignThreads; ++j) {
        const int q = tid + j * kAlignThreads;
        if (q < tlen) {
          const int vid = REMAP ? remap_one(vkeep[j], lkeep[j], num_experts, max_loras) : vkeep[j];
          if (REMAP) vtopk_out[t0 + q] = vid;
          keys[q] = (uint16_t)bucket_of(vid, num_vexperts);
        }
      }
    } else {
      for (int q = tid; q < tlen; q += kAlignThreads) {
        const int64_t i = t0 + q;
        int vid;
        if (REMAP) {
          vid = remap_one(src[i], lora_ids[i / topk], num_experts, max_loras);
          vtopk_out[i] = vid;
        } else {
          vid = src[i];
        }
        keys[q] = (uint16_t)bucket_of(vid, num_vexperts);
      }
    }
    count_keys();
    if (fused)
      bucket_offsets<kAlignThreads>(offs, nb, num_vexperts, block_m, capacity, expert_ids,
                                    ntpp_out, sh_scan);
  }

  // Pass 2: stable rank of every pair inside the tile.
  auto emit = [&](int q, int key, int lr) {
    const int64_t i = t0 + q;
    if (fused) {
      const int64_t pos = (int64_t)offs[key] + lr;
      if (MOL_CHECK(pos >= 0 && pos < capacity, MOL_CHECK_ALIGN_SLOT, pos)) sorted_ids[pos] = (int)i;
    } else {
      ws_rank[i] = lr;
    }
  };
  if constexpr (ONE) {  // every thread any pair: the ranks are in shared memory
    for (int q = tid; q < tlen; q += kAlignThreads) {
      const int key = keys[q];
      emit(q, key, (int)tbl[(q / seg) * nb_pad + key] + (int)lrank[q]);
    }
  } else {
    warp_rank(keys, s0, s1, mine, lane, emit);
  }
}

// ---------------------------------------------------------------------------
// Cluster align: the tiles are the blocks of one thread-block cluster.

MOL_DEV uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
MOL_DEV uint32_t cluster_blocks() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Every thread of every block of the cluster: memory operations before it are
// visible to every thread of the cluster after it (shared and global memory).
MOL_DEV void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Address of the same shared-memory word in block `rank` of the cluster.
MOL_DEV uint32_t peer_smem(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
MOL_DEV int ld_peer(uint32_t a) {
  int v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
MOL_DEV void st_peer(uint32_t a, int v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Block p of the cluster holds tile p (`tile` pairs from p * tile). After the
// tile's counts (cnt[b]), block c takes buckets [c * per, (c + 1) * per):
// it sums the tiles' counts of each (remote reads), pads and scans its share;
// with the offset o_b of each of its buckets inside the share it writes
// o_b + (counts of the tiles before p) into block p's cnt[b] (remote writes),
// and it sends the share's padded total to every block. After the second
// barrier every block knows where each share starts: it writes its buckets'
// expert_ids and scatters its pairs to cnt[key] + the start of key's share +
// the pair's stable rank in the tile (the padding fill of every slot comes
// before the second barrier). Every block reaches every barrier (no
// early exit, no data-dependent wait), and no block reads or writes another's
// shared memory after the last.
template <bool REMAP, int WARPS, bool ONEPASS>
__global__ void __launch_bounds__(WARPS * 32, 1)
align_cluster_kernel(const int* __restrict__ src, const int* __restrict__ lora_ids, int topk,
                     int num_experts, int max_loras, int* __restrict__ vtopk_out, int64_t numel,
                     int num_vexperts, int block_m, int64_t capacity, int tile, int nb_pad,
                     int* __restrict__ sorted_ids, int* __restrict__ expert_ids,
                     int* __restrict__ ntpp_out, int trigger) {
  constexpr int THREADS = WARPS * 32;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int sh_scan[WARPS + 1];
  __shared__ int rsum[kClusterMax];  // padded total of each block's share of the buckets
  __shared__ int s_sentinel;         // offset of the sentinel bucket (in the block that holds it)
  __shared__ int sbase[kClusterMax];  // where each block's share of the buckets starts
  const int nb = num_vexperts + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int CL = (int)cluster_blocks(), me = (int)cluster_rank();
  uint16_t* tbl = reinterpret_cast<uint16_t*>(smem);  // [WARPS][nb_pad]
  uint16_t* keys = tbl + WARPS * nb_pad;              // [tile]
  uint16_t* lrank = keys + tile;                      // ONEPASS: [tile] ranks inside warp segments
  int* cnt = reinterpret_cast<int*>(keys + (ONEPASS ? 2 : 1) * tile);  // [nb]: counts, then bases
  int* opad = cnt + nb;                               // [per]: offsets inside this block's share

  {
    uint4* t4 = reinterpret_cast<uint4*>(tbl);
    const int n4 = WARPS * nb_pad / 8;
    for (int q = tid; q < n4; q += THREADS) t4[q] = make_uint4(0, 0, 0, 0);
  }
  if (trigger == 2) pdl_launch_dependents();  // see align_tile_kernel
  pdl_wait();  // inputs and routing buffers belong to earlier kernels until here
  if (trigger == 1) pdl_launch_dependents();

  const int64_t t0 = (int64_t)me * tile;
  const int tlen = (int)max((int64_t)0, min((int64_t)tile, numel - t0));
  // the tile's ids, kLd per thread in flight at once, then its keys
  constexpr int kLd = 8;
  for (int q0 = 0; q0 < tlen; q0 += kLd * THREADS) {
    int sv[kLd], lv[kLd];
#pragma unroll
    for (int j = 0; j < kLd; ++j) {
      const int q = q0 + j * THREADS + tid;
      sv[j] = q < tlen ? src[t0 + q] : -1;
      lv[j] = (REMAP && q < tlen) ? lora_ids[(t0 + q) / topk] : -1;
    }
#pragma unroll
    for (int j = 0; j < kLd; ++j) {
      const int q = q0 + j * THREADS + tid;
      if (q < tlen) {
        const int vid = REMAP ? remap_one(sv[j], lv[j], num_experts, max_loras) : sv[j];
        if (REMAP) vtopk_out[t0 + q] = vid;
        keys[q] = (uint16_t)bucket_of(vid, num_vexperts);
      }
    }
  }
  __syncthreads();
  const int seg = tile / WARPS;
  const int s0 = warp * seg, s1 = min(s0 + seg, tlen);
  uint16_t* mine = tbl + warp * nb_pad;
  if constexpr (ONEPASS)
    warp_count_rank(keys, s0, s1, mine, lane, lrank);
  else
    warp_count(keys, s0, s1, mine, lane);
  __syncthreads();
  column_scan<WARPS>(tbl, nb, nb_pad, [&](int b, int n) { cnt[b] = n; });
  cluster_barrier();  // 1: every tile's counts are in its block's shared memory
  // every slot starts as padding (the pairs overwrite theirs after barrier 2, which
  // orders these stores before them)
  for (int64_t q = (int64_t)me * THREADS + tid; q < capacity; q += (int64_t)CL * THREADS)
    sorted_ids[q] = (int)numel;

  const int per = (nb + CL - 1) / CL;
  const int b0 = min(me * per, nb), b1 = min(b0 + per, nb);
  const int ppt = (per + THREADS - 1) / THREADS;
  const int c0 = min(b0 + tid * ppt, b1), c1 = min(c0 + ppt, b1);
  const int pad = block_m - 1, lg = __ffs(block_m) - 1;
  int ck[kClusterMax];  // one bucket per thread: its tiles' counts stay in registers
  int local = 0;
  for (int b = c0; b < c1; ++b) {
    int c[kClusterMax];  // every tile's count of b: independent remote loads, all in flight
#pragma unroll
    for (int p = 0; p < kClusterMax; ++p) c[p] = p < CL ? ld_peer(peer_smem(cnt + b, p)) : 0;
    int tot = 0;
#pragma unroll
    for (int p = 0; p < kClusterMax; ++p) {
      tot += c[p];
      ck[p] = c[p];
    }
    const int pb = (tot + pad) & ~pad;
    opad[b - b0] = pb;
    local += pb;
  }
  int share_total;
  int run = block_exclusive_scan<THREADS>(local, sh_scan, share_total);
  for (int b = c0; b < c1; ++b) {
    const int o = run;  // the bucket's offset inside the share
    run += opad[b - b0];
    opad[b - b0] = o;
    int c[kClusterMax];
#pragma unroll
    for (int p = 0; p < kClusterMax; ++p)
      c[p] = ppt == 1 ? ck[p] : (p < CL ? ld_peer(peer_smem(cnt + b, p)) : 0);
    int r = o;  // tile p's base in b, relative to the share's start
#pragma unroll
    for (int p = 0; p < kClusterMax; ++p) {
      if (p < CL) st_peer(peer_smem(cnt + b, p), r);
      r += c[p];
    }
  }
  if (tid < CL) st_peer(peer_smem(rsum + me, tid), share_total);
  cluster_barrier();  // 2: every tile's relative bases and every share's padded total are in place

  int base = 0, ntpp = 0;
  for (int c = 0; c < CL; ++c) {
    const int v = rsum[c];
    base += c < me ? v : 0;
    ntpp += v;
  }
  if (tid < CL) {  // where each share starts
    int a = 0;
    for (int c = 0; c < tid; ++c) a += rsum[c];
    sbase[tid] = a;
  }
  for (int b = c0; b < c1; ++b) {
    const int o = base + opad[b - b0];
    const int pb = (b + 1 < b1 ? opad[b + 1 - b0] : share_total) - opad[b - b0];
    if (b < num_vexperts) {
      const int nblk = pb >> lg;
      for (int k = 0; k < nblk; ++k)
        if (MOL_CHECK((o >> lg) + k < (capacity >> lg), MOL_CHECK_ALIGN_BLOCK, (o >> lg) + k))
          expert_ids[(o >> lg) + k] = b;
    } else {
      s_sentinel = o;  // b == V: the last bucket
    }
  }
  if (me == 0 && tid == 0) {
    (void)MOL_CHECK(ntpp <= capacity, MOL_CHECK_ALIGN_TOTAL, ntpp);
    *ntpp_out = ntpp;
  }
  __syncthreads();  // s_sentinel and sbase
  if (b0 < nb && b1 == nb) {  // the sentinel's blocks and every block past them carry -1
    for (int64_t t = (s_sentinel >> lg) + tid; t < (capacity >> lg); t += THREADS)
      expert_ids[t] = -1;
  }

  auto scatter = [&](int q, int key, int lr) {
    const int64_t pos = (int64_t)cnt[key] + sbase[key / per] + lr;
    if (MOL_CHECK(pos >= 0 && pos < capacity, MOL_CHECK_ALIGN_SLOT, pos)) sorted_ids[pos] = (int)(t0 + q);
  };
  if constexpr (ONEPASS) {  // every thread any pair: the ranks are in shared memory
    for (int q = tid; q < tlen; q += THREADS) {
      const int key = keys[q];
      scatter(q, key, (int)tbl[(q / seg) * nb_pad + key] + (int)lrank[q]);
    }
  } else {
    warp_rank(keys, s0, s1, mine, lane, scatter);
  }
}

// Multi-tile: per-bucket prefix over tiles, bucket offsets, expert_ids, ntpp.
__global__ void __launch_bounds__(kScanThreads, 1)
align_scan_kernel(int* __restrict__ ws_hist, int* __restrict__ ws_offs, int tiles,
                  int num_vexperts, int block_m, int64_t capacity, int* __restrict__ expert_ids,
                  int* __restrict__ ntpp_out) {
  extern __shared__ __align__(16) int counts[];
  __shared__ int sh_scan[kScanThreads / 32 + 1];
  const int nb = num_vexperts + 1;
  pdl_wait();
  pdl_launch_dependents();
  for (int b = threadIdx.x; b < nb; b += kScanThreads) {
    int run = 0;
    int p = 0;
    for (; p + 8 <= tiles; p += 8) {
      int c[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) c[u] = ws_hist[(int64_t)(p + u) * nb + b];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        ws_hist[(int64_t)(p + u) * nb + b] = run;
        run += c[u];
      }
    }
    for (; p < tiles; ++p) {
      const int c = ws_hist[(int64_t)p * nb + b];
      ws_hist[(int64_t)p * nb + b] = run;
      run += c;
    }
    counts[b] = run;
  }
  __syncthreads();
  bucket_offsets<kScanThreads>(counts, nb, num_vexperts, block_m, capacity, expert_ids, ntpp_out,
                               sh_scan);
  __syncthreads();
  for (int b = threadIdx.x; b < nb; b += kScanThreads) ws_offs[b] = counts[b];
}

__global__ void align_scatter_kernel(const int* __restrict__ vtopk, int64_t numel, int num_vexperts,
                                     int tile, const int* __restrict__ ws_hist,
                                     const int* __restrict__ ws_offs,
                                     const int* __restrict__ ws_rank, int* __restrict__ sorted_ids,
                                     int64_t capacity, int trigger) {
  // last writer of the routing: dependents start when it exits unless trigger (see
  // align_tile_kernel)
  if (trigger == 2) pdl_launch_dependents();
  pdl_wait();
  if (trigger == 1) pdl_launch_dependents();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= numel) return;
  const int key = bucket_of(vtopk[i], num_vexperts);
  const int64_t p = i / tile;
  const int64_t pos = (int64_t)ws_offs[key] + ws_hist[p * (num_vexperts + 1) + key] + ws_rank[i];
  if (MOL_CHECK(pos >= 0 && pos < capacity, MOL_CHECK_ALIGN_SLOT, pos)) sorted_ids[pos] = (int)i;
}

// ---------------------------------------------------------------------------

AlignPlan make_align_plan(int64_t numel, int num_vexperts, int block_m) {
  AlignPlan p{};
  p.numel = numel;
  p.nb = num_vexperts + 1;
  p.nb_pad = (p.nb + 7) & ~7;
  p.block_m = block_m;
  const int64_t nonempty = std::min<int64_t>(numel, p.nb);
  p.capacity = (numel + nonempty * (block_m - 1) + block_m - 1) / block_m * block_m;
  p.cluster = false;
  if (numel <= kTileMin) {
    p.tile = (int)std::max<int64_t>(256, (numel + 255) / 256 * 256);
    p.tiles = 1;
  } else if (numel <= kClusterPairs) {
    p.cluster = true;  // tile and block count are chosen at launch for the device
    p.tile = 0;
    p.tiles = 0;
    p.one_pass = false;  // chosen at launch too
    p.smem_tile = 0;
    p.ws_bytes = 0;
    return p;
  } else {
    const int64_t want = (numel + kMaxTiles - 1) / kMaxTiles;
    p.tile = (int)std::max<int64_t>(kTileMin, (want + 255) / 256 * 256);
    p.tiles = (int)((numel + p.tile - 1) / p.tile);
  }
  size_t smem = (size_t)kAlignWarps * p.nb_pad * 2 + (size_t)p.tile * 2;
  if (p.tiles == 1) smem += (size_t)p.nb * 4;
  // one pass of matches where the pairs' ranks fit beside the tables
  p.one_pass = smem + (size_t)p.tile * 2 <= (size_t)kAlignSmemMax;
  if (p.one_pass) smem += (size_t)p.tile * 2;
  p.smem_tile = (smem + 15) / 16 * 16;
  if (p.tiles == 1) {
    p.ws_bytes = 0;
  } else {
    const size_t ints = (size_t)p.tiles * p.nb + p.nb + (size_t)numel;
    p.ws_bytes = (ints * 4 + 255) / 256 * 256;
  }
  return p;
}

// Largest cluster of the cluster align on each device (8, or 16 where a
// 16-block cluster of its shared-memory size can be scheduled).
static int g_cluster_max[64] = {0};

static cudaError_t prepare_cluster_align() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  for (auto k : {align_cluster_kernel<true, 8, false>, align_cluster_kernel<false, 8, false>,
                 align_cluster_kernel<true, 16, false>, align_cluster_kernel<false, 16, false>,
                 align_cluster_kernel<true, 8, true>, align_cluster_kernel<false, 8, true>,
                 align_cluster_kernel<true, 16, true>, align_cluster_kernel<false, 16, true>}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlignSmemMax);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kClusterMax);
  cfg.blockDim = dim3(kAlignThreads);
  cfg.dynamicSmemBytes = kAlignSmemMax;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterMax;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, (void*)align_cluster_kernel<true, 8, false>, &cfg);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // a refused query leaves the portable size
    n = 0;
  }
  if (dev >= 0 && dev < 64) g_cluster_max[dev] = n >= 1 ? kClusterMax : 8;
  return cudaSuccess;
}

static int sm_count(int device) {
  static int cache[64] = {0};
  if (device < 0 || device >= 64) return 148;
  if (cache[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0)
      n = 148;
    cache[device] = n;
  }
  return cache[device];
}

cudaError_t prepare_lora_kernels();

cudaError_t prepare_kernels() {
  cudaError_t e = cudaSuccess;
  for (auto k : {align_tile_kernel<true, false>, align_tile_kernel<false, false>,
                 align_tile_kernel<true, true>, align_tile_kernel<false, true>})
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlignSmemMax);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(align_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kAlignSmemMax);
  if (e != cudaSuccess) return e;
  e = prepare_cluster_align();
  if (e != cudaSuccess) return e;
  e = prepare_stage_kernels();
  if (e != cudaSuccess) return e;
  return prepare_lora_kernels();
}

cudaError_t launch_token_lora_ids(const int32_t* weight_indices, const int32_t* seg_indptr,
                                  int num_reqs, int64_t num_tokens, int max_loras,
                                  const int32_t* lora_ranks, int32_t* lora_ids,
                                  cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((num_tokens + threads - 1) / threads, 4096);
  return launch_pdl(token_lora_ids_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                    weight_indices, seg_indptr, num_reqs, num_tokens, max_loras, lora_ranks,
                    lora_ids);
}

cudaError_t launch_virtual_topk(const int32_t* topk_ids, const int32_t* lora_ids, int64_t numel,
                                int topk, int num_experts, int max_loras, int32_t* vtopk,
                                cudaStream_t stream) {
  if (numel == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((numel + threads - 1) / threads, 4096);
  return launch_pdl(virtual_topk_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream, topk_ids,
                    lora_ids, numel, topk, num_experts, max_loras, vtopk);
}

cudaError_t launch_align(const AlignPlan& plan, bool remap, const int32_t* src,
                         const int32_t* lora_ids, int topk, int num_experts, int max_loras,
                         int32_t* vtopk_out, int num_vexperts, int32_t* sorted_ids,
                         int32_t* expert_ids, int32_t* ntpp, void* workspace, int trigger,
                         cudaStream_t stream) {
  const int trig = trigger;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (plan.cluster) {
    // blocks of 2048 pairs, up to the device's cluster size, then larger tiles (the tile
    // passes, rounds of 32 pairs per warp, are the longest steps: more blocks, fewer rounds)
    const int cmax = (device >= 0 && device < 64 && g_cluster_max[device]) ? g_cluster_max[device] : 8;
    const int cl = (int)std::min<int64_t>(cmax, (plan.numel + kTileMin / 2 - 1) / (kTileMin / 2));
    const int tile = (int)(((plan.numel + cl - 1) / cl + 255) / 256 * 256);
    if (tile > kClusterTileMax) return cudaErrorInvalidConfiguration;
    const int per = (plan.nb + cl - 1) / cl;
    // shared memory of a block with `warps` warp tables (and, one pass, the pairs' ranks)
    auto smem_of = [&](int warps, bool one) {
      return (size_t)warps * plan.nb_pad * 2 + (size_t)tile * (one ? 4 : 2) + (size_t)plan.nb * 4 +
             (size_t)per * 4;
    };
    // sixteen warps where their tables fit (half the match rounds per warp), else eight;
    // one pass of matches where the pairs' ranks fit too
    const bool w16 = smem_of(16, false) <= (size_t)kAlignSmemMax;
    const int warps = w16 ? 16 : 8;
    const bool one = smem_of(warps, true) <= (size_t)kAlignSmemMax;
    const size_t smem = smem_of(warps, one);
    if (smem > (size_t)kAlignSmemMax) return cudaErrorInvalidConfiguration;
    const int32_t* lids = remap ? lora_ids : nullptr;
    int32_t* vout = remap ? vtopk_out : nullptr;
    const int tk = remap ? topk : 1, ne = remap ? num_experts : 1, ml = remap ? max_loras : 1;
#define MOL_ALIGN_CLUSTER(R, W, O)                                                                 \
  launch_pdl_cluster(align_cluster_kernel<R, W, O>, cl, dim3(W * 32), smem, stream, src, lids, tk, \
                     ne, ml, vout, plan.numel, num_vexperts, plan.block_m, plan.capacity, tile,     \
                     plan.nb_pad, sorted_ids, expert_ids, ntpp, trig)
#define MOL_ALIGN_CLUSTER_W(R, O) (w16 ? MOL_ALIGN_CLUSTER(R, 16, O) : MOL_ALIGN_CLUSTER(R, 8, O))
    if (remap) return one ? MOL_ALIGN_CLUSTER_W(true, true) : MOL_ALIGN_CLUSTER_W(true, false);
    return one ? MOL_ALIGN_CLUSTER_W(false, true) : MOL_ALIGN_CLUSTER_W(false, false);
#undef MOL_ALIGN_CLUSTER_W
#undef MOL_ALIGN_CLUSTER
  }
  int* ws_hist = nullptr;
  int* ws_offs = nullptr;
  int* ws_rank = nullptr;
  unsigned grid = 1;
  if (plan.tiles > 1) {
    ws_hist = static_cast<int*>(workspace);
    ws_offs = ws_hist + (size_t)plan.tiles * plan.nb;
    ws_rank = ws_offs + plan.nb;
    const int64_t fill_blocks = (plan.capacity + 16383) / 16384;
    grid = (unsigned)std::max<int64_t>(plan.tiles, std::min<int64_t>(sm_count(device), fill_blocks));
  }
  {
    const int32_t* lids = remap ? lora_ids : nullptr;
    int32_t* vout = remap ? vtopk_out : nullptr;
    const int tk = remap ? topk : 1, ne = remap ? num_experts : 1, ml = remap ? max_loras : 1;
#define MOL_ALIGN_TILE(R, O)                                                                      \
  launch_pdl(align_tile_kernel<R, O>, dim3(grid), dim3(kAlignThreads), plan.smem_tile, stream, src, \
             lids, tk, ne, ml, vout, plan.numel, num_vexperts, plan.block_m, plan.capacity,        \
             plan.tile, plan.tiles, plan.nb_pad, sorted_ids, expert_ids, ntpp, ws_hist, ws_rank,   \
             trig)
    if (remap)
      e = plan.one_pass ? MOL_ALIGN_TILE(true, true) : MOL_ALIGN_TILE(true, false);
    else
      e = plan.one_pass ? MOL_ALIGN_TILE(false, true) : MOL_ALIGN_TILE(false, false);
#undef MOL_ALIGN_TILE
  }
  if (e != cudaSuccess || plan.tiles == 1) return e;
  e = launch_pdl(align_scan_kernel, dim3(1), dim3(kScanThreads), (size_t)plan.nb * 4, stream, ws_hist,
                 ws_offs, plan.tiles, num_vexperts, plan.block_m, plan.capacity, expert_ids, ntpp);
  if (e != cudaSuccess) return e;
  const int64_t sblocks = (plan.numel + 255) / 256;
  const int32_t* vt = remap ? vtopk_out : src;
  return launch_pdl(align_scatter_kernel, dim3((unsigned)sblocks), dim3(256), 0, stream, vt,
                    plan.numel, num_vexperts, plan.tile, ws_hist, ws_offs, ws_rank, sorted_ids,
                    plan.capacity, trig);
}

cudaError_t take_align_checks(unsigned long long* first, unsigned long long* count) {
  CheckRecord r;
  const cudaError_t e = take_check_record_here(&r);
  *first = r.first;
  *count = r.count;
  return e;
}

}  // namespace mol
