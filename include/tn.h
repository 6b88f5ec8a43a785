/*
 * tn.h: C ABI of the GB300 exact tensor-network contraction executor.
 *
 * A network is contracted pairwise along a fixed binary tree.  Before any
 * device work, tn_plan() fixes the storage order of every tensor by the
 * GEMM-oriented "lifetime ordering" of "Crossing the single-GPU memory wall:
 * multi-GPU large-scale tensor network contraction" (digest of arXiv
 * 2606.01852), section 1.4: walking the tree back from the root, each
 * operand stores the output's modes it owns, in the output's order, followed
 * by the summed modes.  Every step A x B -> C then reads A as a row-major
 * [m, k] matrix and B as a row-major [n, k] matrix (section 1.1 names M, N
 * and K); no intermediate is ever transposed.  Only leaves are permuted.
 * Intermediates larger than memory are handled by slicing (section 1.1):
 * fixing the sliced modes splits the contraction into independent
 * sub-contractions whose results add up in the output.
 *
 * Conventions for every call:
 *   - Storage is row-major: the last listed mode varies fastest.
 *   - Values are complex64: interleaved (re, im) float pairs, 8 bytes each.
 *   - Mode ids are 0 .. n_modes-1.  A closed mode appears in exactly two
 *     tensors, an open mode in exactly one.  Hyperedges, traces (a mode twice
 *     in one tensor) and modes that appear nowhere are rejected.
 *   - No call throws; every failure is a tn_status.  A plan is not
 *     thread-safe: use it from one host thread and one stream at a time.
 *   - tn_plan() does no device work.  The library never allocates device
 *     memory: the caller provides the workspace.
 */
#ifndef TN_GB300_H
#define TN_GB300_H

#include <stdint.h>

#if defined(__GNUC__)
#define TN_API __attribute__((visibility("default")))
#else
#define TN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tn_status {
    TN_OK = 0,
    TN_EINVAL = 1,     /* malformed network, tree, slice set or argument */
    TN_ENOMEM = 2,     /* workspace missing or smaller than required */
    TN_EOVERFLOW = 3,  /* a size or FLOP count exceeds 64 bits */
    TN_ECUDA = 4,      /* a CUDA runtime call failed (see tn_last_error) */
    TN_EDEVICE = 5,    /* a kernel reported an inconsistency on the device */
    TN_ETIMEOUT = 6,   /* a bounded device-side wait gave up */
    TN_ENOTIMPL = 7    /* valid request this build does not support */
} tn_status;

/* Arithmetic of the tensor-core contraction of dense nodes.  Small and
 * bandwidth-bound nodes use fp32 CUDA-core arithmetic in every mode.
 * Intermediates are complex64 in HBM in every mode. */
enum {
    TN_PREC_TF32X3 = 0, /* split precision: x = hi + lo (hi = x rounded to
                           tf32, lo = x - hi); products hi*hi + hi*lo + lo*hi
                           accumulated in fp32 (fp32-level accuracy) */
    TN_PREC_BF16 = 1,   /* tensor-core operands rounded to bf16 (round to
                           nearest even), fp32 accumulation */
    TN_PREC_FP32 = 2,   /* every node on CUDA-core fp32 FMA */
    TN_PREC_BF16X3 = 3  /* split bf16: x = hi + lo (hi = x rounded to bf16,
                           lo = x - hi rounded to bf16, 16 significant bits);
                           products hi*hi + hi*lo + lo*hi on the bf16 tensor
                           path accumulated in fp32: half the tensor-core time
                           and operand bytes of TN_PREC_TF32X3, about 32 times
                           its representation error (2^-17 against 2^-22 of
                           each operand entry) */
};

/* Node classes reported by tn_plan_node_class and forced by
 * tn_plan_set_policy. */
enum {
    TN_NODE_SIMT = 0,      /* general CUDA-core tiled kernel */
    TN_NODE_DENSE = 1,     /* tcgen05 tensor-core kernel */
    TN_NODE_STREAM = 2,    /* bandwidth-bound kernel (small n or k) */
    TN_NODE_TINY = 3,      /* batched tiny nodes, many per launch */
    TN_NODE_FUSED = 4      /* inside a fused leaf subtree (tn_plan_set_fusion) */
};

enum {
    TN_POLICY_AUTO = 0,    /* classify every node by its shape */
    TN_POLICY_SIMT = 1,    /* every node on the general CUDA-core kernel */
    TN_POLICY_NO_TINY = 2  /* auto, but no batched tiny-node launches */
};

/*
 * Network description (section 1.1; section 3.1 describes the same data as
 * an einsum string plus per-mode extents).  All arrays are caller-owned and
 * only read during tn_plan(), which copies what it needs.
 *   n_tensors     number of leaves (>= 1)
 *   ranks[t]      number of modes of leaf t (0 allowed: a scalar)
 *   modes[t]      the ranks[t] mode ids of leaf t, in its storage order
 *   n_modes       number of mode ids
 *   extents[x]    dimension of mode x (>= 1)
 *   n_open        number of open modes
 *   open_modes    open mode ids in the order of the result's axes (the
 *                 root order that section 1.4 takes as given)
 *   precision     one of TN_PREC_*
 */
typedef struct tn_network {
    int32_t n_tensors;
    const int32_t *ranks;
    const int32_t *const *modes;
    int32_t n_modes;
    const int64_t *extents;
    int32_t n_open;
    const int32_t *open_modes;
    int32_t precision;
} tn_network;

/*
 * Contraction tree in SSA form (section 3.4 lists a tree as ordered steps
 * with two operands and an output each).  Step s contracts the ids
 * pairs[2s] (operand A, whose kept modes form M) and pairs[2s+1] (operand B,
 * kept modes N); leaves are ids 0 .. n_tensors-1 and step s produces id
 * n_tensors + s.  Every id is consumed exactly once; the last step is the
 * root.  n_steps must be n_tensors - 1.
 */
typedef struct tn_tree {
    int32_t n_steps;
    const int32_t *pairs;
} tn_tree;

/* Sliced modes (section 1.1): closed modes only.  Slices run in
 * lexicographic order of the sliced indices, the first listed mode most
 * significant.  n = 0 (or a NULL pointer to this struct) means no slicing. */
typedef struct tn_slices {
    int32_t n;
    const int32_t *modes;
} tn_slices;

typedef struct tn_plan_s tn_plan_t;

/* Stream handle; the same type as cudaStream_t (NULL = legacy stream). */
typedef struct CUstream_st *tn_stream_t;

/*
 * Validate the inputs, compute mode lifetimes, the lifetime order of every
 * tensor, every node's GEMM shape (m, n, k), C_t = sum of 8 m n k over the
 * nodes times the number of slices, C_s = the largest intermediate in
 * elements, the kernel class of every node, and the workspace layout.
 * Host only.  On success *out owns a new plan (free with tn_plan_destroy).
 * Errors: TN_EINVAL (malformed input; see tn_last_error(NULL)),
 * TN_EOVERFLOW, TN_ENOTIMPL (more modes per tensor than supported).
 */
TN_API tn_status tn_plan(const tn_network *network, const tn_tree *tree,
                  const tn_slices *slices, tn_plan_t **out);

/* Release a plan (NULL is ignored).  Does not free the workspace. */
TN_API void tn_plan_destroy(tn_plan_t *plan);

/* C_t over all slices: sum over nodes of 8 m n k (one complex multiply-add
 * counted as 8 real flops), times the number of slices. */
TN_API tn_status tn_plan_flops(const tn_plan_t *plan, uint64_t *ct);

/* C_s: the largest step output, in elements (per slice). */
TN_API tn_status tn_plan_peak(const tn_plan_t *plan, uint64_t *cs);

/* Number of slices: product of the sliced modes' extents (1 if none). */
TN_API tn_status tn_plan_num_slices(const tn_plan_t *plan, uint64_t *n);

/* Number of steps (n_tensors - 1). */
TN_API tn_status tn_plan_num_steps(const tn_plan_t *plan, int32_t *n);

/* Lifetime order of tensor `id` (leaf or step output, SSA numbering):
 * writes min(len, cap) mode ids into buf and the full length into *len.
 * Sliced modes are not part of any order. */
TN_API tn_status tn_plan_mode_order(const tn_plan_t *plan, int32_t id, int32_t *buf,
                             int32_t cap, int32_t *len);

/* GEMM shape of step `step`: mnk[0] = m, mnk[1] = n, mnk[2] = k. */
TN_API tn_status tn_plan_node_mnk(const tn_plan_t *plan, int32_t step, uint64_t mnk[3]);

/* Kernel class (TN_NODE_*) the executor will use for step `step`. */
TN_API tn_status tn_plan_node_class(const tn_plan_t *plan, int32_t step, int32_t *cls);

/* Choose how nodes are classified (TN_POLICY_*).  Call before
 * tn_plan_workspace_bytes / tn_plan_set_workspace; it resets the workspace
 * binding.  Errors: TN_EINVAL (NULL plan or a value not listed above). */
TN_API tn_status tn_plan_set_policy(tn_plan_t *plan, int32_t policy);

/* Device workspace the plan needs, in bytes (intermediates, permuted
 * leaves, descriptor tables and a device status word). */
TN_API tn_status tn_plan_workspace_bytes(const tn_plan_t *plan, uint64_t *bytes);

/*
 * Bind device memory as the workspace: dev_ptr must be 256-byte aligned
 * device memory of at least tn_plan_workspace_bytes() bytes, owned by the
 * caller and left alone by everyone else until the plan is destroyed or
 * rebound.  Uploads the plan's descriptor tables (synchronous copy) on the
 * current device.  Errors: TN_EINVAL (NULL or misaligned), TN_ENOMEM (too
 * small), TN_ECUDA.
 */
TN_API tn_status tn_plan_set_workspace(tn_plan_t *plan, void *dev_ptr, uint64_t bytes);

/*
 * Contract the network: enqueue all slices and all steps on `stream`.
 *   leaf_ptrs[t]  device pointer to leaf t in its own storage order
 *                 (complex64, contiguous, 8-byte aligned); read only, must
 *                 stay valid until the enqueued work completes.
 *   out_ptr       device pointer to the result (complex64, open-mode order,
 *                 product of the open extents entries; 1 entry if none).
 *                 Overwritten with the sum over all slices.
 * Asynchronous: returns after enqueueing.  Launch-time failures give
 * TN_ECUDA; device-side problems surface through tn_plan_check().
 * Replay: the first call with a given set of leaf, output and workspace
 * pointers launches directly and also records the launch sequence into a
 * CUDA graph (on a stream the plan creates); later calls with the same
 * pointers replay that graph on `stream`.  Different pointers re-record.
 * Turn this off with tn_plan_set_replay(plan, 0).
 * Errors: TN_EINVAL (NULL pointers), TN_ENOMEM (no workspace bound).
 */
TN_API tn_status tn_execute(tn_plan_t *plan, const void *const *leaf_ptrs, void *out_ptr,
                     tn_stream_t stream);

/*
 * tn_execute for callers that cannot allocate device memory (the paper has
 * no counterpart; this is a convenience of this library).  Some callers may
 * not allocate after start-up: real-time loops, plugins inside a host
 * runtime that owns all device memory, code running where the allocator is
 * off limits.  This call needs no tn_plan_set_workspace: it runs the same
 * kernels as tn_execute with a 32 MiB scratch array that the library keeps
 * in device global memory (every GPU that loads the library holds it until
 * the process exits).  It calls no allocating routine.
 *   - Plans whose tn_plan_workspace_bytes exceeds 32 MiB: TN_ENOMEM, with
 *     nothing enqueued.
 *   - All calls share the array.  Each call clears the status word and
 *     uploads its plan's descriptor table on `stream` before its kernels;
 *     calls whose GPU work overlaps (other streams, unordered threads) race
 *     on the array.  Order them on one stream.
 *   - The first call on a device looks up the array's address on that
 *     device (which must be current) and caches it: make that first call
 *     before any stream capture.
 *   - The device status word of these calls lives at the start of the
 *     array: after a static call (stream synchronised), tn_plan_check() on
 *     the same plan reads and clears it there, with the device of that
 *     call current.  Launch timing is suspended during these calls.
 * Arguments, result and other errors as for tn_execute.
 */
TN_API tn_status tn_execute_static(tn_plan_t *plan, const void *const *leaf_ptrs, void *out_ptr,
                                   tn_stream_t stream);

/*
 * tn_execute restricted to the slices first, first + step, first + 2 step,
 * ... below tn_plan_num_slices: out_ptr receives their sum (zero when the
 * range is empty).  Slices are independent sub-contractions whose results
 * add up (section 1.1 slicing), so R processes that take first = r,
 * step = R and add their outputs obtain the full result; that sum is the
 * only exchange between them.  step >= 1, first >= 0.  Launches directly
 * (no graph replay); otherwise as tn_execute.
 */
TN_API tn_status tn_execute_slices(tn_plan_t *plan, const void *const *leaf_ptrs, void *out_ptr,
                                   tn_stream_t stream, uint64_t first, uint64_t step);

/*
 * End to end from host memory: copy each caller leaf host_leaves[t] (its
 * whole storage, complex64, caller's order) into the device buffer
 * dev_leaves[t] (caller-owned, at least as large), contract into dev_out as
 * tn_execute does, and copy the result (open-mode order) into host_out.
 * Leaves in pinned (page-locked) host memory are read through their device
 * mapping by one gather kernel for all of them; other leaves are copied one
 * cudaMemcpyAsync each (synchronous for pageable memory).  Asynchronous on
 * `stream` for pinned buffers: synchronise the stream before reading
 * host_out.  The host buffers must stay valid until then.  When every host
 * buffer (leaves and host_out) is pinned and graph replay is on, the whole
 * call (gather, contraction, copy out) is recorded after its first run and
 * replayed by later calls with the same buffers and workspace; the buffers'
 * contents are read afresh on every call.
 * Errors: as tn_execute; TN_EINVAL for NULL pointers.
 */
TN_API tn_status tn_execute_host(tn_plan_t *plan, const void *const *host_leaves, void *host_out,
                                 void *const *dev_leaves, void *dev_out, tn_stream_t stream);

/* ---- verification of intermediates ------------------------------------
 *
 * The value of a contraction does not depend on the tree ("Crossing the
 * single-GPU memory wall", section 1.1), so every node can be checked on its
 * own: its output must be the [m, k] x [n, k] product of its two operands
 * (section 1.4 layouts).  These two calls expose one node's operands and
 * output as they lie in the workspace, so that sampled outputs of a
 * full-size node can be recomputed independently from the data the node
 * actually read.
 */

/*
 * Run the first slice's launches, in issue order and without graph replay,
 * up to and including the launch that computes step `step` (its split-K
 * reduction included), then stop.  Leaves and out_ptr as for tn_execute
 * (out_ptr receives the root's slice-0 value only if `step` is the root).
 * Afterwards, until the next execute of any kind, the step's two operands
 * and its output are still in place for tn_plan_tensor_gather.  Other
 * launches of the same tiny-node batch as `step` also run.
 * Errors: TN_EINVAL (NULL pointers, step out of range), TN_ENOMEM (no
 * workspace bound), TN_ECUDA.
 */
TN_API tn_status tn_execute_prefix(tn_plan_t *plan, const void *const *leaf_ptrs, void *out_ptr,
                                   int32_t step, tn_stream_t stream);

/*
 * Read entries of tensor `id` (SSA numbering: an operand or the output of
 * the step the last tn_execute_prefix stopped at) as complex64, after that
 * call and on a stream ordered after it.  idx: device array of `count`
 * logical indices, row-major over the tensor's lifetime order
 * (tn_plan_mode_order; sliced modes at slice 0).  dst: device array of
 * `count` complex64, receives the entries.  Tensors the planner stores in a
 * planar split format (operands of tensor-core nodes) are returned as
 * hi + lo, the value the tensor-core kernel multiplies; K-tiling is undone.
 * An index outside the tensor gives 0 and makes tn_plan_check report
 * TN_EDEVICE.  Asynchronous on `stream`.
 * Errors: TN_EINVAL (no prefix run, or `id` not an operand or the output of
 * its step, NULL arrays), TN_ECUDA.
 */
TN_API tn_status tn_plan_tensor_gather(tn_plan_t *plan, int32_t id, const int64_t *idx,
                                       uint64_t count, void *dst, tn_stream_t stream);

/* Enable (1, the default) or disable (0) graph replay in tn_execute; any
 * recorded graph is released either way. */
TN_API tn_status tn_plan_set_replay(tn_plan_t *plan, int32_t enable);

/*
 * Complex products on the tensor cores in the split-tf32 precision: with
 * `enable` = 1 a tensor-core node whose time is dominated by its arithmetic
 * forms C = A B from three real products, Ar Br, Ai Bi and (Ar + Ai)(Br + Bi)
 * (re = ArBr - AiBi, im = (Ar + Ai)(Br + Bi) - ArBr - AiBi), instead of four:
 * 25 % fewer tensor-core operations, but operands of 24 instead of 16 bytes
 * per entry, whose 96 KiB pipeline stages leave room for only two stages in
 * shared memory; rounding errors of the imaginary part are about twice as
 * large (still within the complex64 tolerance).  On a GB300 this is slower
 * today (a 4096^3 node: 2.28 ms against 1.76 ms with four products), so the
 * default is 0: always four products.  The pages do not describe this; it
 * is the classic three-multiplication complex product.  Re-plans the layout
 * (like tn_plan_set_policy): bind the workspace again afterwards.
 * Errors: TN_EINVAL (NULL plan).
 */
TN_API tn_status tn_plan_set_three_products(tn_plan_t *plan, int32_t enable);

/*
 * Promotion chunk of the tensor-core nodes: the number of complex k whose
 * products the tensor core accumulates in its fp32 TMEM accumulator before
 * the sum is added (round to nearest) into fp32 registers.  The tensor
 * core's accumulation rounds toward zero, so every node's sums shrink by a
 * relative bias that grows with the chunk (measured ~1.3e-6 per node with
 * 256, ~0.33e-6 with 64), and the nodes' biases add up at the root; shorter
 * chunks cost throughput (4096^3 node: ~352 TFLOP/s with 256, ~340 with 128).
 * chunk_k = 0 (the default) picks, per plan, the longest of 256, 128 and 64
 * whose bias times the number of tensor-core nodes stays within 4e-6 (2048
 * for plain bf16 operands, whose own rounding is ~1e-3); otherwise a
 * multiple of 32 in [32, 4096] for every tensor-core node (CTA pairs use
 * half of it).  Re-plans the layout (like
 * tn_plan_set_policy): bind the workspace again afterwards.
 * Errors: TN_EINVAL (NULL plan or a value outside that set).
 */
TN_API tn_status tn_plan_set_promotion_chunk(tn_plan_t *plan, int32_t chunk_k);

/*
 * Tensor-core nodes on CTA pairs (tcgen05 cta_group::2): with `enable` = 1,
 * a tensor-core node whose longer side has at least 256 entries runs on
 * clusters of two CTAs, each pair computing tiles of 256 x 128 complex
 * outputs with MMAs of M = 256 (each SM holds half of the tile's A rows and
 * half of its B rows, so it reads half as much of B per MMA) and the real
 * and imaginary parts accumulated directly (negated-A MMAs for -Ai Bi) in
 * double-buffered TMEM.  Measured on a GB300 it is not faster than the
 * single-CTA kernel at equal accuracy (4096^3 node, split tf32: 318 against
 * 349 TFLOP/s with 256-k chunks; under the power cap it draws less power but
 * still takes longer), so the default is 0.  Re-plans the layout (like
 * tn_plan_set_policy): bind the workspace again afterwards.
 * Errors: TN_EINVAL (NULL plan).
 */
TN_API tn_status tn_plan_set_cta_pairs(tn_plan_t *plan, int32_t enable);

/*
 * Fused leaf subtrees ("leaf-gate absorption").  Lifetime ordering leaves
 * the leaves as the only tensors to reorder ("Crossing the single-GPU memory
 * wall", section 1.3), and near the leaves a tree is mostly chains of tiny
 * steps: gates absorbed into wires, small tensors meeting.  With `enable` =
 * 1 (the default) every maximal subtree whose leaves and intermediates all
 * have at most 2048 entries (a subtree's tensors together at most 8192 =
 * 64 KiB, leaves of at most 12 axes after merging) runs as one CTA of one
 * launch at the start of each slice: the CTA reads its leaves straight from
 * the caller's buffers (their permutation into lifetime order done on the
 * load), computes the subtree's steps in shared memory and writes only the
 * subtree's root.  Those leaves get no permutation job, the inner steps no
 * launch and no workspace (tn_plan_node_class reports TN_NODE_FUSED; their
 * tensors cannot be read with tn_plan_tensor_gather).  Only with
 * TN_POLICY_AUTO.  Results equal the unfused plan's up to fp32 rounding
 * order.  Re-plans the layout (like tn_plan_set_policy): bind the workspace
 * again afterwards.  Errors: TN_EINVAL (NULL plan).
 */
TN_API tn_status tn_plan_set_fusion(tn_plan_t *plan, int32_t enable);

/*
 * Slice-invariant hoisting ("Crossing the single-GPU memory wall", section
 * 1.1: slicing repeats the whole contraction once per slice; a node none of
 * whose leaves carries a sliced mode computes the same tensor in every
 * slice).  With `enable` = 1 (the default) the first slice an execute runs
 * takes every launch and each later slice only the launches that depend on
 * a sliced leaf; invariant intermediates that those launches read stay in
 * the workspace for the whole execute (the workspace may grow: query
 * tn_plan_workspace_bytes again).  Results are those of the plain slice
 * loop; tn_plan_launches counts the launches of one execute either way.
 * No effect without slices.  Re-plans the layout (like tn_plan_set_policy):
 * bind the workspace again afterwards.
 * Errors: TN_EINVAL (NULL plan).
 */
TN_API tn_status tn_plan_set_hoisting(tn_plan_t *plan, int32_t enable);

/* After the stream has been synchronised: read and clear the device status
 * word of the plan's last execute (in the bound workspace, or in the static
 * scratch array when that execute was tn_execute_static).  TN_OK,
 * TN_EDEVICE (a kernel saw an inconsistent descriptor) or TN_ETIMEOUT (a
 * bounded wait inside a kernel gave up; the plan's descriptor tables are
 * restored, so the next execute runs normally). */
TN_API tn_status tn_plan_check(tn_plan_t *plan);

/* ---- measurement ------------------------------------------------------ */

/* Kernel ids in launch records. */
enum {
    TN_KERNEL_PERMUTE = 0,      /* leaf permutation batch */
    TN_KERNEL_SIMT = 1,         /* general CUDA-core node kernel */
    TN_KERNEL_DENSE_TF32X3 = 2, /* tcgen05 node kernel, split tf32 */
    TN_KERNEL_DENSE_BF16 = 3,   /* tcgen05 node kernel, bf16 operands */
    TN_KERNEL_STREAM = 4,       /* bandwidth-bound node kernel */
    TN_KERNEL_TINY = 5,         /* batched tiny-node kernel */
    TN_KERNEL_REDUCE = 6,       /* ordered sum of split-K partials */
    TN_KERNEL_DENSE_TF32X3_3P = 7, /* tcgen05 node kernel, split tf32, three real products */
    TN_KERNEL_DENSE_BF16X3 = 8,    /* tcgen05 node kernel, split bf16 */
    TN_KERNEL_FUSED = 9            /* fused leaf subtrees */
};

/* One kernel launch of a profiled tn_execute.  flops = 8 m n k of the
 * node(s) it ran; bytes = the algorithmic HBM bytes (every operand read
 * once, the output written once, plus read once more when accumulating). */
typedef struct tn_launch_record {
    int32_t kernel;   /* TN_KERNEL_* */
    int32_t step;     /* tree step, or -1 for launches covering many */
    float ms;         /* device time between CUDA events around the launch */
    uint64_t flops;
    uint64_t bytes;
} tn_launch_record;

/* Number of kernel launches one tn_execute makes (all slices). */
TN_API tn_status tn_plan_launches(const tn_plan_t *plan, uint64_t *n);

/* Enable (1) or disable (0) launch timing.  While enabled, tn_execute
 * records a CUDA event before and after every launch on its stream (events
 * are created by the plan and freed with it).  Off by default. */
TN_API tn_status tn_plan_set_profiling(tn_plan_t *plan, int32_t enable);

/* After a profiled tn_execute has completed (stream synchronised): copy up
 * to cap records into buf and the number recorded into *len. */
TN_API tn_status tn_plan_profile_read(tn_plan_t *plan, tn_launch_record *buf, int32_t cap,
                                      int32_t *len);

/* Static text for a status code. */
TN_API const char *tn_status_string(tn_status status);

/* Text of the last failure on this plan; with plan == NULL, of the last
 * failed tn_plan() call on this thread.  Valid until the next call. */
TN_API const char *tn_last_error(const tn_plan_t *plan);

#ifdef __cplusplus
}
#endif

#endif /* TN_GB300_H */
