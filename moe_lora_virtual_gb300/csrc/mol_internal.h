// Host-side launchers behind the C ABI (not exported).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mol {

// Kernels this library has enqueued in this process (read by mol_launch_count).
void count_launch();

// Geometry of the align step for given sizes (host arithmetic).
struct AlignPlan {
  int64_t numel;
  int nb;          // buckets = V + 1
  int nb_pad;      // nb rounded up to 8
  int block_m;
  int64_t capacity;
  int tile;        // pairs per tile block
  int tiles;       // number of tile blocks (1 = single fused block)
  bool cluster;    // the tiles are the blocks of one cluster (sized at launch): no workspace
  bool one_pass;   // tile kernel: the pairs' ranks kept in shared memory, one pass of matches
  size_t smem_tile;
  size_t ws_bytes;  // workspace (0 with one tile or one cluster), 256-byte multiple
};

AlignPlan make_align_plan(int64_t numel, int num_vexperts, int block_m);

// Sets shared-memory limits of every kernel on the current device.
cudaError_t prepare_kernels();

// Launch with programmatic stream serialization: the kernel's blocks may be
// scheduled while the previous kernel in the stream finishes; each kernel
// guards its reads of that kernel's output with griddepcontrol.wait.
// The same for a grid that is one thread-block cluster of `blocks` blocks.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), int blocks, dim3 block, size_t smem,
                               cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = blocks;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// A launch in plain stream order: it starts once the previous kernel has finished
// (for grids of resident blocks with a fixed share of work each, which would
// otherwise start one by one as the previous kernel's blocks leave).
template <typename... KArgs, typename... Args>
cudaError_t launch_ordered(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.numAttrs = 0;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Per-token adapter ids from per-request slots (seg_indptr non-decreasing).
cudaError_t launch_token_lora_ids(const int32_t* weight_indices, const int32_t* seg_indptr,
                                  int num_reqs, int64_t num_tokens, int max_loras,
                                  const int32_t* lora_ranks, int32_t* lora_ids,
                                  cudaStream_t stream);

cudaError_t launch_virtual_topk(const int32_t* topk_ids, const int32_t* lora_ids, int64_t numel,
                                int topk, int num_experts, int max_loras, int32_t* vtopk,
                                cudaStream_t stream);

// remap != 0: `src` is topk_ids and the remap is fused (vtopk written);
// remap == 0: `src` is vtopk_ids.
// trigger: when the align's dependents may start. 0: when it exits (called on
// its own: a following kernel may read the routing early); 1: once it has waited
// for the previous kernel (the next kernel reads the routing after its own
// griddepcontrol.wait, as in mol_lora_forward); 2: at once, and with one tile the
// align counts and scans before its own wait (the caller's ids were complete
// before the previous kernel began; the next kernel may read them early).
cudaError_t launch_align(const AlignPlan& plan, bool remap, const int32_t* src,
                         const int32_t* lora_ids, int topk, int num_experts, int max_loras,
                         int32_t* vtopk_out, int num_vexperts, int32_t* sorted_ids,
                         int32_t* expert_ids, int32_t* ntpp, void* workspace, int trigger,
                         cudaStream_t stream);

// r1: rank per slice; lora_ranks (per adapter, adapter = v / num_experts, may
// be NULL) limit the columns computed: rank 0 writes nothing, columns past
// the rank are written as 0. Ranks are read like the weights (before
// griddepcontrol.wait with `early`).
// early = true only inside mol_lora_forward reusing a routing (compute_routing
// = 0): the routing and the weights are then read before griddepcontrol.wait,
// the activations after it. The routing is then older than the kernel that
// precedes the call (or was written by a standalone align, which lets its
// dependents start only once it has exited).
// The top-k ids and adapter ids the routing of a mol_lora_forward call is computed
// from. With ready_early (compute_routing = 2: the ids were complete before the
// previous kernel began) the shrink that follows the align asks L2 for the lora_a
// rows of every virtual expert with pairs while the align still runs (see
// launch_shrink).
struct RoutingIds {
  const int32_t* topk_ids;  // [numel]
  const int32_t* lora_ids;  // [numel / topk]
  int numel, topk, num_experts, max_loras;
  bool ready_early;
};
// Most pairs, and most bytes of weight rows, for which the shrink prefetches.
constexpr int kPrefetchPairsMax = 4096;
constexpr int64_t kPrefetchBudget = 64ll << 20;

cudaError_t launch_shrink(const void* x, int64_t x_stride, int x_div, int K, const void* lora_a,
                          int R, const int32_t* sorted_ids, const int32_t* expert_ids,
                          const int32_t* ntpp, int64_t capacity, int block_m, int64_t numel,
                          int num_vexperts, float* inter, bool early, cudaStream_t stream,
                          int r1, const int32_t* lora_ranks, int num_experts,
                          const RoutingIds* prefetch = nullptr);

// early = true only when the preceding kernel is this library's shrink of the
// same stage (mol_lora_forward): routing, weights and output rows are then read
// before griddepcontrol.wait, the intermediate after it. The shrink waits for
// its own predecessor before it lets this kernel start, so everything older
// than the shrink is complete.
cudaError_t launch_expand(const float* inter, const void* lora_b, int S, int r, int Ns, float scale,
                          const float* topk_weights, const int32_t* sorted_ids,
                          const int32_t* expert_ids, const int32_t* ntpp, int64_t capacity,
                          int block_m, int64_t numel, int num_vexperts, void* out,
                          int64_t out_stride, bool early, cudaStream_t stream,
                          const int32_t* lora_ranks, const float* lora_scalings, int num_experts);

// Per-adapter ranks: the shrink keeps one rank per adapter in shared memory.
constexpr int kMaxLoraTable = 2048;

// Shrink on tcgen05 tensor cores for batches with many rows per virtual
// expert: R % 64 == 0, K % 64 == 0, block_m in {64, 128}, at least 32 pairs per
// virtual expert on average, no per-adapter ranks. Reads everything after
// griddepcontrol.wait.
bool shrink_tc_fits(int64_t numel, int num_vexperts, int R, int K, int block_m);
cudaError_t prepare_tc_kernels();
cudaError_t launch_shrink_tc(const void* x, int64_t x_stride, int x_div, int K, const void* lora_a,
                             int R, const int32_t* sorted_ids, const int32_t* expert_ids,
                             const int32_t* ntpp, int64_t capacity, int block_m, int64_t numel,
                             int num_vexperts, float* inter, cudaStream_t stream);

// The expand of full routed blocks of rank 64 on tcgen05 (many rows per virtual
// expert, no adapter arrays, Ns a multiple of 128, BLOCK_M 64 or 128).
bool expand_tc_fits(int64_t numel, int num_vexperts, int r, int Ns, int block_m,
                    int64_t out_stride, bool adapter_arrays);
cudaError_t prepare_expand_tc_kernels();
cudaError_t launch_expand_tc(const float* inter, const void* lora_b, int S, int Ns, float scale,
                             const float* topk_weights, const int32_t* sorted_ids,
                             const int32_t* expert_ids, const int32_t* ntpp, int64_t capacity,
                             int block_m, int64_t numel, int num_vexperts, void* out,
                             int64_t out_stride, cudaStream_t stream);

// One stage fused into one launch (shrink then expand per routed block, the
// block's intermediate kept in shared memory and also stored): for small
// layers (every routed block on an SM of its own, a virtual expert's weights
// in about two stages), ranks 8-64, R <= 128, no per-adapter arrays.
// early = true when the routing is older than the kernel before the call
// (mol_lora_forward reusing a routing): routing words and the first weight
// copies are then issued before griddepcontrol.wait.
bool stage_fused_fits(int64_t numel, int num_vexperts, int R, int r, int K, int N, int block_m,
                      int64_t capacity, bool adapter_arrays);
cudaError_t prepare_stage_kernels();
cudaError_t launch_stage(const void* x, int64_t x_stride, int x_div, int K, const void* lora_a,
                         const void* lora_b, int S, int r, int Ns, float scale,
                         const float* topk_weights, const int32_t* sorted_ids,
                         const int32_t* expert_ids, const int32_t* ntpp, int64_t capacity,
                         int block_m, int64_t numel, int num_vexperts, float* inter, void* out,
                         int64_t out_stride, bool early, cudaStream_t stream);
cudaError_t take_stage_faults(unsigned* out);

// Fault words of the pipelined kernels (bit 0: a bounded barrier or copy wait
// ran out); read and cleared by mol_take_fault_flags.
cudaError_t take_lora_faults(unsigned* out);
cudaError_t take_tc_faults(unsigned* out);
cudaError_t take_expand_tc_faults(unsigned* out);
// Check records of the checked build, per kernel file (read and cleared; zero
// in the release build): the first failed check's (site << 48 | value) and the
// number of failed checks.
cudaError_t take_align_checks(unsigned long long* first, unsigned long long* count);
cudaError_t take_lora_checks(unsigned long long* first, unsigned long long* count);
cudaError_t take_tc_checks(unsigned long long* first, unsigned long long* count);
cudaError_t take_stage_checks(unsigned long long* first, unsigned long long* count);
cudaError_t take_expand_tc_checks(unsigned long long* first, unsigned long long* count);
// Test controls of the bounded waits (mol_debug_wait_test): the item shrink's and
// the tcgen05 expand's producers.
cudaError_t set_wait_test(unsigned stall, unsigned long long limit_ns);
cudaError_t set_expand_tc_wait_test(unsigned stall, unsigned long long limit_ns);

// Largest contraction width accepted by the shrink (it streams K in chunks).
constexpr int kShrinkMaxK = 1 << 16;

}  // namespace mol
