// Exported C ABI of the MoL LoRA library (declared in include/mol.h).
// Host code only: validation, device checks, dispatch to the launchers.

#include <algorithm>
#include <atomic>
#include <mutex>

#include "mol.h"
#include "mol_internal.h"


namespace {
std::atomic<int64_t> g_launches{0};
}  // namespace

void mol::count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

thread_local int32_t g_last_cuda_error = 0;

int32_t cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int32_t)e;
  return MOL_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_block_m(int32_t bm) { return bm == 16 || bm == 32 || bm == 64 || bm == 128; }

// Per device: 0 = unchecked, 1 = ready (sm_103, kernels prepared), 2 = unsupported.
// Read without the lock on every call; written under it once per device.
constexpr int kMaxDevices = 64;
std::atomic<int> g_device_state[kMaxDevices] = {};
std::mutex g_device_mutex;

// Checks the current device is an sm_103 part and prepares kernel attributes
// once per device. Returns MOL_OK, MOL_ERR_UNSUPPORTED or MOL_ERR_CUDA.
int32_t ensure_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return MOL_ERR_UNSUPPORTED;
  if (g_device_state[dev].load(std::memory_order_acquire) == 1) return MOL_OK;
  std::lock_guard<std::mutex> lock(g_device_mutex);
  if (g_device_state[dev].load(std::memory_order_relaxed) == 0) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (major != 10 || minor != 3) {
      g_device_state[dev].store(2, std::memory_order_release);
    } else {
      e = mol::prepare_kernels();
      if (e != cudaSuccess) return cuda_fail(e);
      g_device_state[dev].store(1, std::memory_order_release);
    }
  }
  return g_device_state[dev].load(std::memory_order_relaxed) == 1 ? MOL_OK : MOL_ERR_UNSUPPORTED;
}

int32_t check_align_args(int64_t numel, int32_t num_vexperts, int32_t block_m) {
  if (numel < 0 || num_vexperts < 1) return MOL_ERR_INVALID_ARG;
  if (!valid_block_m(block_m)) return MOL_ERR_UNSUPPORTED;
  if (numel > MOL_MAX_NUMEL || num_vexperts + 1 > MOL_MAX_BUCKETS) return MOL_ERR_UNSUPPORTED;
  return MOL_OK;
}

int32_t check_routing_in(const int32_t* sorted_ids, const int32_t* expert_ids, const int32_t* ntpp,
                         int64_t capacity, int32_t block_m, int64_t numel, int32_t num_vexperts) {
  if (numel < 0 || capacity < 0 || num_vexperts < 1) return MOL_ERR_INVALID_ARG;
  if (!valid_block_m(block_m)) return MOL_ERR_UNSUPPORTED;
  if (numel > MOL_MAX_NUMEL) return MOL_ERR_UNSUPPORTED;
  if (capacity % block_m != 0) return MOL_ERR_INVALID_ARG;
  if (numel > 0 && capacity > 0 && (!sorted_ids || !expert_ids || !ntpp)) return MOL_ERR_INVALID_ARG;
  return MOL_OK;
}

int32_t check_shrink_args(const void* x, int64_t x_row_stride, int32_t x_row_div, int32_t K,
                          const void* lora_a, int32_t num_slices, int32_t rank, const float* inter,
                          int64_t numel) {
  if (K <= 0 || x_row_div < 1 || num_slices < 1 || rank < 1 || x_row_stride < K)
    return MOL_ERR_INVALID_ARG;
  const int64_t R = (int64_t)num_slices * rank;
  if (K % 8 != 0 || K > mol::kShrinkMaxK || x_row_stride % 8 != 0 || R % 8 != 0 || R > 1024)
    return MOL_ERR_UNSUPPORTED;
  if (numel > 0 && (!x || !lora_a || !inter)) return MOL_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(lora_a) || !aligned16(inter)) return MOL_ERR_UNSUPPORTED;
  return MOL_OK;
}

int32_t check_expand_args(const float* inter, const void* lora_b, int32_t num_slices, int32_t rank,
                          int32_t slice_n, const void* out, int64_t out_row_stride,
                          int64_t numel) {
  if (num_slices < 1 || rank < 1 || slice_n < 1) return MOL_ERR_INVALID_ARG;
  if (out_row_stride < (int64_t)num_slices * slice_n) return MOL_ERR_INVALID_ARG;
  if (!(rank == 8 || rank == 16 || rank == 32 || rank == 64 || rank == 128))
    return MOL_ERR_UNSUPPORTED;
  if (slice_n % 8 != 0 || out_row_stride % 8 != 0) return MOL_ERR_UNSUPPORTED;
  if (numel > 0 && (!inter || !lora_b || !out)) return MOL_ERR_INVALID_ARG;
  if (!aligned16(inter) || !aligned16(lora_b) || !aligned16(out)) return MOL_ERR_UNSUPPORTED;
  return MOL_OK;
}

// Per-adapter ranks / scalings (either may be NULL): the adapter of virtual
// expert v is v / num_experts; the shrink keeps the ranks in shared memory.
int32_t check_adapter_args(const int32_t* lora_ranks, const float* lora_scalings,
                           int32_t num_experts, int32_t num_vexperts, int32_t rank) {
  if (!lora_ranks && !lora_scalings) return MOL_OK;
  if (num_experts < 1 || num_vexperts % num_experts != 0) return MOL_ERR_INVALID_ARG;
  if (lora_ranks && (num_vexperts / num_experts > mol::kMaxLoraTable || rank % 8 != 0))
    return MOL_ERR_UNSUPPORTED;
  return MOL_OK;
}

}  // namespace

extern "C" {

int32_t mol_version(void) { return 100; }

const char* mol_status_string(int32_t status) {
  switch (status) {
    case MOL_OK:
      return "ok";
    case MOL_ERR_INVALID_ARG:
      return "invalid argument";
    case MOL_ERR_CAPACITY:
      return "routing buffer or workspace too small";
    case MOL_ERR_UNSUPPORTED:
      return "shape, alignment or device outside the supported contract";
    case MOL_ERR_CUDA:
      return "CUDA error (see mol_last_cuda_error)";
    default:
      return "unknown status";
  }
}

int32_t mol_last_cuda_error(void) { return g_last_cuda_error; }

int64_t mol_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int64_t mol_align_capacity(int64_t numel, int32_t num_vexperts, int32_t block_m) {
  if (numel < 0 || num_vexperts < 1 || block_m < 1) return -1;
  const int64_t nonempty = numel < (int64_t)num_vexperts + 1 ? numel : (int64_t)num_vexperts + 1;
  return (numel + nonempty * (block_m - 1) + block_m - 1) / block_m * block_m;
}

size_t mol_workspace_bytes(int64_t numel, int32_t num_vexperts, int32_t block_m) {
  if (check_align_args(numel, num_vexperts, block_m) != MOL_OK) return 0;
  return mol::make_align_plan(numel, num_vexperts, block_m).ws_bytes;
}

int32_t mol_virtual_topk(const int32_t* topk_ids, const int32_t* lora_ids, int64_t num_tokens,
                         int32_t topk, int32_t num_experts, int32_t max_loras,
                         int32_t* vtopk_ids, void* stream) {
  if (num_tokens < 0 || topk < 1 || num_experts < 1 || max_loras < 1) return MOL_ERR_INVALID_ARG;
  const int64_t numel = num_tokens * topk;
  if (numel > MOL_MAX_NUMEL) return MOL_ERR_UNSUPPORTED;
  if ((int64_t)num_experts * max_loras > (int64_t)1 << 30) return MOL_ERR_UNSUPPORTED;
  if (numel == 0) return MOL_OK;
  if (!topk_ids || !lora_ids || !vtopk_ids) return MOL_ERR_INVALID_ARG;
  int32_t st = ensure_device();
  if (st != MOL_OK) return st;
  cudaError_t e = mol::launch_virtual_topk(topk_ids, lora_ids, numel, topk, num_experts, max_loras,
                                           vtopk_ids, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOL_OK : cuda_fail(e);
}

int32_t mol_take_fault_flags(uint32_t* flags) {
  if (!flags) return MOL_ERR_INVALID_ARG;
  int32_t st = ensure_device();
  if (st != MOL_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned a = 0, b = 0, c = 0, d = 0;
  e = mol::take_lora_faults(&a);
  if (e == cudaSuccess) e = mol::take_tc_faults(&b);
  if (e == cudaSuccess) e = mol::take_stage_faults(&c);
  if (e == cudaSuccess) e = mol::take_expand_tc_faults(&d);
  if (e != cudaSuccess) return cuda_fail(e);
  *flags = a | b | c | d;
  return MOL_OK;
}

int32_t mol_debug_wait_test(uint32_t stall_producer, uint64_t wait_limit_ns) {
  if (stall_producer > 1) return MOL_ERR_INVALID_ARG;
  int32_t st = ensure_device();
  if (st != MOL_OK) return st;
  const unsigned long long lim = wait_limit_ns == 0 ? 1000000000ull : wait_limit_ns;
  cudaError_t e = mol::set_wait_test(stall_producer, lim);
  return e == cudaSuccess ? MOL_OK : cuda_fail(e);
}

int32_t mol_checked_build(void) {
#ifdef MOL_CHECKED
  return 1;
#else
  return 0;
#endif
}

int32_t mol_take_check_record(uint64_t* first, uint64_t* count) {
  int32_t st = ensure_device();
  if (st != MOL_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  // in the path's order: align, item shrink and expands, tcgen05 shrink, fused stage,
  // tcgen05 expand
  cudaError_t (*const take[5])(unsigned long long*, unsigned long long*) = {
      mol::take_align_checks, mol::take_lora_checks, mol::take_tc_checks,
      mol::take_stage_checks, mol::take_expand_tc_checks};
  unsigned long long f = 0, n = 0;
  for (auto fn : take) {
    unsigned long long fi = 0, ni = 0;
    e = fn(&fi, &ni);
    if (e != cudaSuccess) return cuda_fail(e);
    if (f == 0) f = fi;
    n += ni;
  }
  if (first) *first = f;
  if (count) *count = n;
  return MOL_OK;
}

int32_t mol_token_lora_ids(const int32_t* weight_indices, const int32_t* seg_indptr,
                           int32_t num_reqs, int64_t num_tokens, int32_t max_loras,
                           const int32_t* lora_ranks, int32_t* lora_ids, void* stream) {
  if (num_reqs < 0 || num_tokens < 0 || max_loras < 1) return MOL_ERR_INVALID_ARG;
  if (num_tokens > MOL_MAX_NUMEL) return MOL_ERR_UNSUPPORTED;
  if (num_tokens == 0) return MOL_OK;
  if (!lora_ids || (num_reqs > 0 && (!weight_indices || !seg_indptr))) return MOL_ERR_INVALID_ARG;
  int32_t st = ensure_device();
  if (st != MOL_OK) return st;
  cudaError_t e = mol::launch_token_lora_ids(weight_indices, seg_indptr, num_reqs, num_tokens,
                                             max_loras, lora_ranks, lora_ids,
                                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOL_OK : cuda_fail(e);
}

int32_t mol_align_block_size(const int32_t* vtopk_ids, int64_t numel, int32_t num_vexperts,
                             int32_t block_m, int32_t* sorted_token_ids, int64_t capacity,
                             int32_t* expert_ids, int32_t* num_tokens_post_padded,
                             void* workspace, size_t workspace_bytes, void* stream) {
  int32_t st = check_align_args(numel, num_vexperts, block_m);
  if (st != MOL_OK) return st;
  if (!num_tokens_post_padded || (numel > 0 && !vtopk_ids) ||
      (capacity > 0 && (!sorted_token_ids || !expert_ids)))
    return MOL_ERR_INVALID_ARG;
  const mol::AlignPlan plan = mol::make_align_plan(numel, num_vexperts, block_m);
  if (capacity < plan.capacity || capacity % block_m != 0) return MOL_ERR_CAPACITY;
  if (plan.ws_bytes > 0 && (!workspace || workspace_bytes < plan.ws_bytes)) return MOL_ERR_CAPACITY;
  if (plan.ws_bytes > 0 && !aligned16(workspace)) return MOL_ERR_UNSUPPORTED;
  st = ensure_device();
  if (st != MOL_OK) return st;
  mol::AlignPlan p = plan;
  p.capacity = capacity;  // fill the caller's whole buffer
  cudaError_t e = mol::launch_align(p, false, vtopk_ids, nullptr, 1, 1, 1, nullptr, num_vexperts,
                                    sorted_token_ids, expert_ids, num_tokens_post_padded,
                                    workspace, 0, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOL_OK : cuda_fail(e);
}

int32_t mol_lora_shrink(const void* x, int64_t x_row_stride, int32_t x_row_div, int32_t K,
                        const void* lora_a, int32_t num_slices, int32_t rank,
                        const int32_t* sorted_token_ids, const int32_t* expert_ids,
                        const int32_t* num_tokens_post_padded, int64_t capacity,
                        int32_t block_m, int64_t numel, int32_t num_vexperts, float* inter,
                        int32_t num_experts, const int32_t* lora_ranks, void* stream) {
  int32_t st = check_routing_in(sorted_token_ids, expert_ids, num_tokens_post_padded, capacity,
                                block_m, numel, num_vexperts);
  if (st != MOL_OK) return st;
  st = check_shrink_args(x, x_row_stride, x_row_div, K, lora_a, num_slices, rank, inter, numel);
  if (st != MOL_OK) return st;
  st = check_adapter_args(lora_ranks, nullptr, num_experts, num_vexperts, rank);
  if (st != MOL_OK) return st;
  if (numel == 0 || capacity == 0) return MOL_OK;
  st = ensure_device();
  if (st != MOL_OK) return st;
  cudaError_t e = mol::launch_shrink(x, x_row_stride, x_row_div, K, lora_a, num_slices * rank,
                                     sorted_token_ids, expert_ids, num_tokens_post_padded,
                                     capacity, block_m, numel, num_vexperts, inter, false,
                                     static_cast<cudaStream_t>(stream), rank, lora_ranks,
                                     num_experts);
  return e == cudaSuccess ? MOL_OK : cuda_fail(e);
}

int32_t mol_lora_expand(const float* inter, const void* lora_b, int32_t num_slices, int32_t rank,
                        int32_t slice_n, float scale, const float* topk_weights,
                        const int32_t* sorted_token_ids, const int32_t* expert_ids,
                        const int32_t* num_tokens_post_padded, int64_t capacity, int32_t block_m,
                        int64_t numel, int32_t num_vexperts, void* out, int64_t out_row_stride,
                        int32_t num_experts, const int32_t* lora_ranks,
                        const float* lora_scalings, void* stream) {
  int32_t st = check_routing_in(sorted_token_ids, expert_ids, num_tokens_post_padded, capacity,
                                block_m, numel, num_vexperts);
  if (st != MOL_OK) return st;
  st = check_expand_args(inter, lora_b, num_slices, rank, slice_n, out, out_row_stride, numel);
  if (st != MOL_OK) return st;
  st = check_adapter_args(lora_ranks, lora_scalings, num_experts, num_vexperts, rank);
  if (st != MOL_OK) return st;
  if (numel == 0 || capacity == 0) return MOL_OK;
  st = ensure_device();
  if (st != MOL_OK) return st;
  cudaError_t e = mol::launch_expand(inter, lora_b, num_slices, rank, slice_n, scale, topk_weights,
                                     sorted_token_ids, expert_ids, num_tokens_post_padded,
                                     capacity, block_m, numel, num_vexperts, out, out_row_stride,
                                     false, static_cast<cudaStream_t>(stream), lora_ranks,
                                     lora_scalings, num_experts);
  return e == cudaSuccess ? MOL_OK : cuda_fail(e);
}

int32_t mol_lora_forward(const void* x, int64_t x_row_stride, int32_t x_row_div, int32_t K,
                         const int32_t* topk_ids, const int32_t* lora_ids, int64_t num_tokens,
                         int32_t topk, int32_t num_experts, int32_t max_loras,
                         const void* lora_a, const void* lora_b, int32_t num_slices,
                         int32_t rank, int32_t slice_n, float scale,
                         const float* topk_weights, void* out, int64_t out_row_stride,
                         int32_t block_m, int32_t compute_routing, int32_t* vtopk_ids,
                         int32_t* sorted_token_ids, int64_t capacity, int32_t* expert_ids,
                         int32_t* num_tokens_post_padded, float* inter,
                         const int32_t* lora_ranks, const float* lora_scalings,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (num_tokens < 0 || topk < 1 || num_experts < 1 || max_loras < 1) return MOL_ERR_INVALID_ARG;
  if (compute_routing < 0 || compute_routing > 2) return MOL_ERR_INVALID_ARG;
  const int64_t V64 = (int64_t)num_experts * max_loras;
  if (V64 + 1 > MOL_MAX_BUCKETS) return MOL_ERR_UNSUPPORTED;
  const int32_t V = (int32_t)V64;
  const int64_t numel = num_tokens * topk;
  int32_t st = check_align_args(numel, V, block_m);
  if (st != MOL_OK) return st;
  st = check_routing_in(sorted_token_ids, expert_ids, num_tokens_post_padded, capacity, block_m,
                        numel, V);
  if (st != MOL_OK) return st;
  st = check_shrink_args(x, x_row_stride, x_row_div, K, lora_a, num_slices, rank, inter, numel);
  if (st != MOL_OK) return st;
  st = check_expand_args(inter, lora_b, num_slices, rank, slice_n, out, out_row_stride, numel);
  if (st != MOL_OK) return st;
  st = check_adapter_args(lora_ranks, lora_scalings, num_experts, V, rank);
  if (st != MOL_OK) return st;
  const mol::AlignPlan plan = mol::make_align_plan(numel, V, block_m);
  if (compute_routing) {
    if (!num_tokens_post_padded) return MOL_ERR_INVALID_ARG;
    if (numel > 0 && (!topk_ids || !lora_ids || !vtopk_ids)) return MOL_ERR_INVALID_ARG;
    if (capacity > 0 && (!sorted_token_ids || !expert_ids)) return MOL_ERR_INVALID_ARG;
    if (capacity < plan.capacity) return MOL_ERR_CAPACITY;
    if (plan.ws_bytes > 0 && (!workspace || workspace_bytes < plan.ws_bytes))
      return MOL_ERR_CAPACITY;
    if (plan.ws_bytes > 0 && !aligned16(workspace)) return MOL_ERR_UNSUPPORTED;
  }
  st = ensure_device();
  if (st != MOL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (compute_routing) {
    mol::AlignPlan p = plan;
    p.capacity = capacity;
    e = mol::launch_align(p, true, topk_ids, lora_ids, topk, num_experts, max_loras, vtopk_ids, V,
                          sorted_token_ids, expert_ids, num_tokens_post_padded, workspace,
                          compute_routing == 2 ? 2 : 1, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (numel == 0 || capacity == 0) return MOL_OK;
  if (mol::stage_fused_fits(numel, V, num_slices * rank, rank, K, num_slices * slice_n, block_m,
                            capacity, lora_ranks != nullptr || lora_scalings != nullptr)) {
    e = mol::launch_stage(x, x_row_stride, x_row_div, K, lora_a, lora_b, num_slices, rank, slice_n,
                          scale, topk_weights, sorted_token_ids, expert_ids,
                          num_tokens_post_padded, capacity, block_m, numel, V, inter, out,
                          out_row_stride, compute_routing == 0, s);
    return e == cudaSuccess ? MOL_OK : cuda_fail(e);
  }
  // ids declared ready early: the shrink asks L2 for its weight rows while the align runs
  const mol::RoutingIds ids{topk_ids, lora_ids, (int)numel, topk, num_experts, max_loras,
                            compute_routing == 2};
  e = mol::launch_shrink(x, x_row_stride, x_row_div, K, lora_a, num_slices * rank,
                         sorted_token_ids, expert_ids, num_tokens_post_padded, capacity, block_m,
                         numel, V, inter, compute_routing == 0, s, rank, lora_ranks, num_experts,
                         compute_routing ? &ids : nullptr);
  if (e != cudaSuccess) return cuda_fail(e);
  e = mol::launch_expand(inter, lora_b, num_slices, rank, slice_n, scale, topk_weights,
                         sorted_token_ids, expert_ids, num_tokens_post_padded, capacity, block_m,
                         numel, V, out, out_row_stride, true, s, lora_ranks, lora_scalings,
                         num_experts);
  return e == cudaSuccess ? MOL_OK : cuda_fail(e);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Align without any allocation: the scratch lives in this library.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they route a batch: an inference runtime that has already reserved nearly
// all of device memory for its own pool and hands an operator only its input
// and output buffers, or a latency-critical loop where an allocation's implicit
// device synchronisation is not acceptable. For them, this variant of
// mol_align_block_size takes no workspace argument and uses a fixed 1 MiB
// array compiled into the library instead. Every GPU that loads the library
// holds that 1 MiB until the process exits.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
// Device address of g_noalloc_scratch, per device. In host code the array's
// name is only a host-side stand-in, so the address is looked up once per
// device with that device current; later calls read the cached address
// without taking a lock.
std::atomic<void*> g_noalloc_scratch_addr[kMaxDevices] = {};

int32_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return MOL_ERR_UNSUPPORTED;
  void* p = g_noalloc_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_device_mutex);
    p = g_noalloc_scratch_addr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return cuda_fail(e);
      g_noalloc_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return MOL_OK;
}

}  // namespace

extern "C" int32_t mol_align_block_size_noalloc(const int32_t* vtopk_ids, int64_t numel,
                                                int32_t num_vexperts, int32_t block_m,
                                                int32_t* sorted_token_ids, int64_t capacity,
                                                int32_t* expert_ids,
                                                int32_t* num_tokens_post_padded, void* stream) {
  int32_t st = check_align_args(numel, num_vexperts, block_m);
  if (st != MOL_OK) return st;
  if (!num_tokens_post_padded || (numel > 0 && !vtopk_ids) ||
      (capacity > 0 && (!sorted_token_ids || !expert_ids)))
    return MOL_ERR_INVALID_ARG;
  const mol::AlignPlan plan = mol::make_align_plan(numel, num_vexperts, block_m);
  if (capacity < plan.capacity || capacity % block_m != 0) return MOL_ERR_CAPACITY;
  if (plan.ws_bytes > kNoAllocScratchBytes) return MOL_ERR_CAPACITY;
  st = ensure_device();
  if (st != MOL_OK) return st;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != MOL_OK) return st;
  mol::AlignPlan p = plan;
  p.capacity = capacity;
  cudaError_t e = mol::launch_align(p, false, vtopk_ids, nullptr, 1, 1, 1, nullptr, num_vexperts,
                                    sorted_token_ids, expert_ids, num_tokens_post_padded, scratch,
                                    0, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOL_OK : cuda_fail(e);
}
