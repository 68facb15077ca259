/*
 * mol.h -- C ABI of the MoL ("virtual experts") LoRA hot path on GB300 (sm_103a).
 *
 * Each (routed expert, LoRA adapter) pair is one virtual expert of a larger
 * MoE: V = num_experts * max_loras (fork PR #24 "feat(mol):
 * SGLANG_OPT_MOL_LORA_STAGE_CFG", the "...and grid blowup / Root cause"
 * commit). One LoRA stage of a MoE layer runs four steps:
 *
 *   1. mol_virtual_topk      remap top-k expert ids to virtual ids;
 *   2. mol_align_block_size  group pairs by virtual expert into BLOCK_M-padded
 *                            blocks, invalid ids in a trailing sentinel bucket;
 *   3. mol_lora_shrink       inter = x . lora_a^T per block (fp32 out);
 *   4. mol_lora_expand       out += scale * inter . lora_b^T per block (bf16 RMW).
 *
 * mol_lora_forward runs 1-4 (or 3-4 on an existing routing) in one call.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Data pointers are DEVICE pointers, owned by the caller, on the current
 *   CUDA device; the library never allocates, frees or keeps them.
 * - bf16 tensors are passed as raw 16-bit storage (const void* / void*).
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Every call only enqueues work on `stream` and returns: it does not
 *   synchronize, allocate, or read device memory on the host, so a sequence of
 *   calls can be captured into a CUDA graph.
 * - Arguments are validated on the host before anything is enqueued. On an
 *   error status nothing is launched and no output is touched.
 * - Bad device *data* never faults: ids outside [0, V) go to the sentinel
 *   bucket; sorted_token_ids entries outside [0, numel) are skipped, and so
 *   are blocks whose expert id is outside [0, V) (the checked build below
 *   records such entries).
 * - Return value: MOL_OK (0) or a negative MOL_ERR_* status;
 *   mol_status_string() names it, mol_last_cuda_error() gives the cudaError_t
 *   behind MOL_ERR_CUDA (per host thread).
 * - Scalars and pointers only; no struct is passed by value.
 * - Routing layout (all int32):
 *     vtopk_ids         [num_tokens * topk]  virtual ids, negative = sentinel
 *     sorted_token_ids  [capacity]           flat pair ids grouped by bucket,
 *                                            ascending inside a bucket, pads = numel
 *     expert_ids        [capacity / block_m] virtual expert of each block, -1 for
 *                                            sentinel blocks and blocks past the end
 *     num_tokens_post_padded [1]             number of filled slots (multiple of block_m)
 *   capacity must be >= mol_align_capacity(numel, V, block_m).
 */
#ifndef MOL_H_
#define MOL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOL_OK 0
#define MOL_ERR_INVALID_ARG (-1)  /* null pointer, negative size, inconsistent sizes */
#define MOL_ERR_CAPACITY (-2)     /* routing buffer or workspace smaller than required */
#define MOL_ERR_UNSUPPORTED (-3)  /* shape/alignment outside the kernels' contract, or not sm_103 */
#define MOL_ERR_CUDA (-4)         /* a CUDA call failed; see mol_last_cuda_error() */

/* Bucket cap of align: V + 1 (sentinel) <= 8192 (sglang PR 24262 prhub summary,
 * "Implementation breakdown" item 2 and "Risks" item 2: at most 8191 virtual experts). */
#define MOL_MAX_BUCKETS 8192
/* Largest number of (token, slot) pairs one call accepts: 4 Mi pairs (half a
 * million tokens at top-8). The align sets it: a tile of pairs keeps its
 * bucket keys in shared memory (2 bytes each, at most 32768 per tile), at
 * most 128 tiles take part, and each warp counts its pairs per bucket in
 * 16-bit counters. */
#define MOL_MAX_NUMEL (1 << 22)

/* Library ABI version (major * 100 + minor). */
int32_t mol_version(void);

/* Text for a status code; never NULL. */
const char* mol_status_string(int32_t status);

/* cudaError_t of the last MOL_ERR_CUDA returned on this host thread (0 if none). */
int32_t mol_last_cuda_error(void);

/* Kernels this library has enqueued in this process so far (all threads; a
 * launch captured into a CUDA graph counts once, when it is captured). Lets a
 * caller see how many launches a call makes. */
int64_t mol_launch_count(void);

/*
 * Slots of sorted_token_ids needed for any routing of `numel` pairs:
 * ceil_BM(numel + min(numel, V + 1) * (block_m - 1)). The fork PR #24
 * code-review commit calls this the worst-case untrimmed routing buffer; the
 * bound is tight (one pair per bucket reaches it). Pure host arithmetic.
 * Returns -1 on invalid arguments.
 */
int64_t mol_align_capacity(int64_t numel, int32_t num_vexperts, int32_t block_m);

/*
 * Bytes of device workspace mol_align_block_size / mol_lora_forward need for
 * these sizes: 0 up to 131072 pairs (one thread block, or one thread-block
 * cluster, does the whole align), else per-tile histograms and ranks. Pure
 * host arithmetic. Returns 0 on invalid arguments (the call itself then fails).
 */
size_t mol_workspace_bytes(int64_t numel, int32_t num_vexperts, int32_t block_m);


/*
 * Step 1: virtual top-k remap (sglang PR 24171 prhub summary, "Key source
 * snippets", _fused_virtual_topk_ids_kernel; fork PR #24 "fix(lora): -1 = no
 * adapter" commit).
 *   vtopk[i] = base                       if base < 0 (sentinel kept verbatim)
 *            = -1                         if lora < 0, lora >= max_loras or base >= num_experts
 *            = base + lora * num_experts  otherwise
 * with base = topk_ids[i], lora = lora_ids[i / topk].
 *   topk_ids  int32 [num_tokens, topk], row-major, device
 *   lora_ids  int32 [num_tokens], device (per-token adapter slot, -1 = none)
 *   vtopk_ids int32 [num_tokens, topk], device, written (may not alias inputs)
 * num_tokens >= 0, topk >= 1, num_experts >= 1, max_loras >= 1,
 * num_tokens * topk <= MOL_MAX_NUMEL. num_tokens == 0 enqueues nothing.
 */
int32_t mol_virtual_topk(const int32_t* topk_ids, const int32_t* lora_ids, int64_t num_tokens,
                         int32_t topk, int32_t num_experts, int32_t max_loras,
                         int32_t* vtopk_ids, void* stream);

/*
 * Step 2: align_block_size with a sentinel bucket (sglang PR 24171 prhub
 * summary, "Key source snippets", _align_block_size_torch; sglang PR 24262
 * prhub summary, "Implementation breakdown": histogram, prefix sum, expert_ids,
 * scatter, no host synchronisation).
 * bucket(i) = vtopk[i] if 0 <= vtopk[i] < V else V. Bucket b holds c_b pairs
 * and p_b = ceil(c_b / block_m) * block_m slots at offset o_b = sum_{b'<b} p_b'.
 *   sorted_token_ids[o_b + j] = j-th smallest i with bucket(i) == b (j < c_b),
 *                               numel in [o_b + c_b, o_b + p_b) and [ntpp, capacity)
 *   expert_ids[t]             = b for t in [o_b, o_b + p_b) / block_m when b < V, else -1
 *   *num_tokens_post_padded   = ntpp = sum_b p_b (the sentinel bucket is counted)
 * All three outputs are written in full. Deterministic and bit-reproducible.
 *   vtopk_ids    int32 [numel], device
 *   num_vexperts V >= 1, V + 1 <= MOL_MAX_BUCKETS
 *   block_m      one of 16, 32, 64, 128
 *   capacity     >= mol_align_capacity(numel, V, block_m), multiple of block_m
 *   workspace    device, >= mol_workspace_bytes(numel, V, block_m) bytes, 16-byte
 *                aligned (may be NULL when that is 0); contents are scratch
 */
int32_t mol_align_block_size(const int32_t* vtopk_ids, int64_t numel, int32_t num_vexperts,
                             int32_t block_m, int32_t* sorted_token_ids, int64_t capacity,
                             int32_t* expert_ids, int32_t* num_tokens_post_padded,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * mol_align_block_size without a workspace argument, for callers that cannot
 * allocate device memory where they route a batch: a runtime that has already
 * reserved nearly all of HBM for its own pool and gives an operator only its
 * inputs and outputs, or a latency-critical loop where an allocation's
 * implicit device synchronisation is not acceptable. The pages have no
 * counterpart of this call; it is a convenience of this library.
 * The scratch is a fixed 1 MiB array compiled into the library (every GPU that
 * loads the library holds it until the process exits). Sizes whose workspace
 * (mol_workspace_bytes) exceeds 1 MiB are rejected with MOL_ERR_CAPACITY. That
 * workspace is 0 up to 131072 pairs (one block, or one cluster of blocks,
 * does the whole align) and, from there to 524288 pairs,
 * 4 * (tiles * (V + 1) + (V + 1) + numel) bytes rounded up to 256 with
 * tiles = ceil(numel / 4096): the largest accepted size is 131072 pairs at
 * V = 8191 or 4095, more with fewer buckets. Outputs, capacity and
 * the other arguments are those of mol_align_block_size, and so are the results
 * (bit-identical). No allocation of any kind is made.
 * Every call shares the one array and it keeps the previous call's contents;
 * nothing in it needs to start at zero (each word a call reads was written
 * earlier by the same call). Calls that overlap on the GPU (several streams, or
 * several host threads) race on it and must be serialised by the caller.
 * The first call on each device looks the array's device address up
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.
 */
int32_t mol_align_block_size_noalloc(const int32_t* vtopk_ids, int64_t numel,
                                     int32_t num_vexperts, int32_t block_m,
                                     int32_t* sorted_token_ids, int64_t capacity,
                                     int32_t* expert_ids, int32_t* num_tokens_post_padded,
                                     void* stream);

/*
 * Step 3: LoRA shrink per block (fork PR #24 "Root cause" commit: the MoL
 * shrink stage is a fused-MoE GEMM over virtual experts with N = S*r, K = the
 * input width; code-review commit: weight layout [E, N, K]).
 * For every block t with t * block_m < ntpp and v = expert_ids[t] >= 0, and
 * every slot whose pair id i = sorted_token_ids[t*block_m + m] is in [0, numel):
 *   inter[i, j] = sum_k x[i / x_row_div, k] * lora_a[v, j, k],  j < R = num_slices*rank
 * accumulated in fp32. Rows of pairs in no such block are not written.
 *   x          bf16, row q at x + q * x_row_stride (elements), K valid columns
 *   x_row_div  topk for token-row input (gate_up), 1 for per-pair input (down)
 *   lora_a     bf16 [num_vexperts, R, K], contiguous
 *   inter      fp32 [numel, R], contiguous
 * Contract: K % 8 == 0, K <= 65536, R % 8 == 0, R <= 1024, x_row_stride % 8 == 0,
 * x, lora_a, inter 16-byte aligned, capacity % block_m == 0. x must hold
 * ceil(numel / x_row_div) rows.
 * Per-adapter ranks (fork PR #24 "fix(lora): complete the '-1 = no adapter'
 * sentinel guards": kernels index lora_ranks per adapter slot and return
 * early on rank 0):
 *   lora_ranks   int32 [num_vexperts / num_experts] or NULL (all adapters of
 *                rank `rank`). The adapter of virtual expert v is
 *                v / num_experts. With rank r_l (clamped to [0, rank]) the
 *                adapter's lora_a rows past r_l are padding: inter columns
 *                [s*rank + r_l, (s+1)*rank) of each slice are written as 0,
 *                whatever those rows hold (8-row groups wholly past r_l are
 *                not read); r_l = 0 writes nothing.
 *                Needs rank % 8 == 0 and num_vexperts / num_experts <= 2048;
 *                read like lora_a (not produced by the kernel right before).
 *   num_experts  routed experts (used only with lora_ranks).
 */
int32_t mol_lora_shrink(const void* x, int64_t x_row_stride, int32_t x_row_div, int32_t K,
                        const void* lora_a, int32_t num_slices, int32_t rank,
                        const int32_t* sorted_token_ids, const int32_t* expert_ids,
                        const int32_t* num_tokens_post_padded, int64_t capacity,
                        int32_t block_m, int64_t numel, int32_t num_vexperts, float* inter,
                        int32_t num_experts, const int32_t* lora_ranks, void* stream);

/*
 * Step 4: LoRA expand per block, added into the MoE output (fork PR #24 PR
 * body "Background (measured attribution)": M x N output from a K = rank
 * contraction; "Fix": weight view [E, N, K]).
 * For the same blocks and pairs as the shrink, for slice s < num_slices and
 * n < slice_n:
 *   out[i, s*slice_n + n] = bf16_rn( out + scale * w_i *
 *                           sum_j inter[i, s*rank + j] * lora_b[v, s*slice_n + n, j] )
 * with w_i = topk_weights[i] (or 1 when topk_weights is NULL); accumulation,
 * scale and add in fp32, one round-to-nearest-even to bf16. Rows of pairs in
 * no processed block are bit-unchanged ("-1 = no adapter": no delta).
 *   inter        fp32 [numel, num_slices*rank]
 *   lora_b       bf16 [num_vexperts, num_slices*slice_n, rank], contiguous
 *   topk_weights fp32 [numel] or NULL
 *   out          bf16, row i at out + i * out_row_stride (elements), updated in place
 * Contract: rank in {8, 16, 32, 64, 128}, slice_n % 8 == 0, out_row_stride % 8 == 0,
 * out_row_stride >= num_slices * slice_n, inter/lora_b/out 16-byte aligned.
 * Per-adapter rank and scaling (adapter of v = v / num_experts):
 *   lora_ranks     int32 [num_vexperts / num_experts] or NULL: the sum runs over
 *                  j < r_l (clamped to [0, rank]), so inter columns and lora_b
 *                  columns at or past r_l take no part, whatever they hold
 *                  (they may still be read); r_l = 0 leaves the pair's output
 *                  rows bit-unchanged. Needs rank % 8 == 0 and at most 2048
 *                  adapters.
 *   lora_scalings  fp32 [num_vexperts / num_experts] or NULL: the delta is
 *                  multiplied by scale * lora_scalings[adapter].
 *   num_experts    routed experts (used only with either array).
 * Both arrays are read like lora_b.
 */
int32_t mol_lora_expand(const float* inter, const void* lora_b, int32_t num_slices, int32_t rank,
                        int32_t slice_n, float scale, const float* topk_weights,
                        const int32_t* sorted_token_ids, const int32_t* expert_ids,
                        const int32_t* num_tokens_post_padded, int64_t capacity, int32_t block_m,
                        int64_t numel, int32_t num_vexperts, void* out, int64_t out_row_stride,
                        int32_t num_experts, const int32_t* lora_ranks,
                        const float* lora_scalings, void* stream);

/*
 * One MoL LoRA stage end to end (fork PR #24 PR body "Background": per layer
 * one routing feeds every MoL stage). With compute_routing = 1 the call runs
 * steps 1-2 into the given routing buffers (vtopk_ids, sorted_token_ids,
 * expert_ids, num_tokens_post_padded), then 3-4; with 0 it reads those
 * buffers as they are (the down stage reusing the gate_up routing) and
 * topk_ids / lora_ids / workspace may be NULL. Arguments are those of the
 * four calls above; numel = num_tokens * topk; V = num_experts * max_loras.
 * Routing buffers passed with compute_routing = 0 must be complete when the
 * call's first kernel starts (true unless the kernel just before the call
 * lets its dependents start early, before writing them). compute_routing = 2
 * computes the routing like 1 and declares that topk_ids and lora_ids were
 * complete before the kernel just before the call on `stream` began, or that
 * the call is ordered after their writer by an event or a copy on `stream` (in
 * a MoE layer the router's top-k runs before the expert GEMMs that precede the
 * LoRA stage): the align then counts the pairs, and the shrink starts and asks
 * L2 for the weight rows the ids select, while that kernel still runs. With 1
 * the ids may come from the kernel just before the call; both give the same
 * results. lora_ranks and lora_scalings (each NULL or one entry per adapter)
 * are those of the shrink and the expand.
 * compute_routing outside {0, 1, 2} is MOL_ERR_INVALID_ARG.
 */
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
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * The step before step 1: per-token adapter ids from per-request adapter
 * slots (fork PR #24, "feat(lora): base takes no pool slot": a request
 * without an adapter has weight index -1; "fix(lora): complete the '-1 = no
 * adapter' sentinel guards": consumers check for a negative index before
 * indexing lora_ranks, with the meaning of the rank == 0 branch, and the
 * per-token mapping of _compute_moe_lora_info filters negatives first).
 *   lora_ids[t] = w = weight_indices[q]  for t in [seg_indptr[q], seg_indptr[q+1]),
 *                                        if 0 <= w < max_loras and (lora_ranks
 *                                        is NULL or lora_ranks[w] > 0)
 *               = -1                     otherwise, and for tokens in no segment.
 *   weight_indices int32 [num_reqs]; seg_indptr int32 [num_reqs + 1],
 *   non-decreasing (token offsets of the requests); lora_ranks int32
 *   [max_loras] or NULL; lora_ids int32 [num_tokens] (written in full).
 * lora_ranks is indexed only after the range check, so -1 never reads it.
 * Contract: num_tokens <= MOL_MAX_NUMEL. With a decreasing seg_indptr every
 * token still gets some value in {-1} U [0, max_loras) and nothing is read out
 * of bounds.
 */
int32_t mol_token_lora_ids(const int32_t* weight_indices, const int32_t* seg_indptr,
                           int32_t num_reqs, int64_t num_tokens, int32_t max_loras,
                           const int32_t* lora_ranks, int32_t* lora_ids, void* stream);


/*
 * Every wait inside this library's kernels (on a barrier, a bulk copy or a
 * tensor-core accumulator) is bounded; when one runs out the kernel records a
 * fault bit, stops its work early and exits instead of hanging. This call
 * waits for the current device to be idle (cudaDeviceSynchronize), writes the
 * bits recorded since the last call to *flags (0 = none; bit 0 = a wait ran
 * out) and clears them. It synchronizes, so it belongs in checks and tests,
 * not in a captured or timed sequence.
 * After a wait ran out, the outputs of the call that recorded it are undefined
 * (rows may be missing or partial). Before a block exits after a timeout, the
 * producers wait, bounded, for the copies they issued, and the threads that
 * copy rows with cp.async wait for their own; if one of those waits runs out
 * too (the tensor-core shrink's stage barriers also count the gathered rows),
 * the block may exit with a copy in flight.
 * (No counterpart on the pages: the pages' kernels have no bounded waits.)
 */
int32_t mol_take_fault_flags(uint32_t* flags);

/*
 * Test hook of the bounded waits (no counterpart on the pages). With
 * stall_producer = 1 the producer warp of every block of mol_lora_shrink (and
 * of the shrink inside mol_lora_forward, on the mma path) leaves before it
 * issues any copy, and so does the weight producer of the tensor-core expand
 * (full routed blocks of rank 64), so the other roles' waits run out with
 * nothing in flight and record bit 0 of mol_take_fault_flags; 0 restores
 * normal operation. wait_limit_ns bounds every wait of those two kernels (0 =
 * the default, one second). Synchronizes the device; for tests only, never while another
 * thread uses the library. Returns MOL_ERR_INVALID_ARG for stall_producer > 1.
 */
int32_t mol_debug_wait_test(uint32_t stall_producer, uint64_t wait_limit_ns);

/*
 * Checked build (no counterpart on the pages). The same sources compiled with
 * MOL_CHECKED (libmol_checked.so, built beside libmol.so) test the index
 * arithmetic of every kernel on the device: before a guarded access a kernel
 * checks the index against its buffer; a failed check records its site and
 * the offending value and the access is skipped (no trap, no fault; a kernel
 * whose pipeline a skip would stall ends its work early instead, so outputs
 * after a failed check are undefined). Routing data passed in by the caller
 * is checked the same way: entries that the release build silently skips
 * (see the conventions above) are recorded as well. The release build
 * compiles every check out.
 *
 * Sites (the value recorded with each):
 */
#define MOL_CHECK_ROUTE_EXPERT 1  /* a block below num_tokens_post_padded has an expert id
                                     outside [-1, V); value: the block */
#define MOL_CHECK_ROUTE_PAIR 2    /* a sorted_token_ids entry of such a block is outside
                                     [0, numel]; value: the slot */
#define MOL_CHECK_ROUTE_NTPP 3    /* num_tokens_post_padded is negative, above capacity or not a
                                     multiple of block_m; value: num_tokens_post_padded */
#define MOL_CHECK_ALIGN_SLOT 4    /* the align writes a slot outside [0, capacity); value: slot */
#define MOL_CHECK_ALIGN_BLOCK 5   /* the align writes expert_ids outside [0, capacity / block_m);
                                     value: the index */
#define MOL_CHECK_ALIGN_TOTAL 6   /* the align's padded total exceeds capacity; value: total */
#define MOL_CHECK_ALIGN_WORKSPACE 7 /* a workspace index past the tile histograms or ranks;
                                       value: the index */
#define MOL_CHECK_ROW 8           /* a pair row of x, inter or out outside the tensor (x:
                                     numel / x_row_div rows); value: the row */
#define MOL_CHECK_COLUMN 9        /* a column range of inter or out outside its row; value: the
                                     first column */
#define MOL_CHECK_SMEM 10         /* a copy into or a read of shared memory past its region;
                                     value: the byte offset of its end */
#define MOL_CHECK_TMA_COORD 11    /* a tensor copy whose inner coordinate is not a multiple of 16
                                     bytes or lies outside the tensor; value: the coordinate */
#define MOL_CHECK_WEIGHT_ROW 12   /* a lora_a / lora_b row outside [0, V * rows per expert);
                                     value: the row */

/* 1 for the checked build, 0 for the release build. */
int32_t mol_checked_build(void);

/*
 * Reads and clears the check record of the current device: *count = failed
 * checks since the last call (0 in the release build), *first = (site << 48)
 * | (value & 0xFFFFFFFFFFFF) of the first one recorded by the earliest kernel
 * file in the path's order (align, shrink/expand, tcgen05 shrink, fused
 * stage), 0 if none. Synchronizes the device. Either pointer may be NULL.
 */
int32_t mol_take_check_record(uint64_t* first, uint64_t* count);

#ifdef __cplusplus
}
#endif

#endif /* MOL_H_ */
