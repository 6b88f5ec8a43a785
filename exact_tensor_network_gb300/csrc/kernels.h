// Launchers of the device kernels and the small structs they take by value.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "plan.h"

namespace tn {

// Device status word layout at the start of the workspace.
enum : int32_t { ERR_NONE = 0, ERR_DESC = 1, ERR_TIMEOUT = 2 };
struct DevStatus {
    int32_t code;      // first error seen (ERR_*), 0 if none
    int32_t where;     // kernel-specific detail
};

// One GEMM-shaped node: C[offM(i) + offN(j)] (+)= sum_k A[i*k + kk] * B[j*k + kk].
struct NodeArgs {
    const float2 *A;
    const float2 *B;
    void *C;
    int64_t m, n, k;
    SepLayout lm, ln;
    int32_t accumulate;   // 1: add into C (later slices of the root)
    int32_t out_fmt;      // Fmt of C; planes are m*n entries apart
    PlanarTile out_tile;  // K-tiling of a planar C
    DevStatus *status;
    // split-K: with ksplit > 1, split s sums k in [s*kchunk, (s+1)*kchunk)
    // and writes plain partials part[(s*m + i)*n + j]; splitk_reduce stores C
    int32_t ksplit;
    int64_t kchunk;
    float2 *part;
};

// Bandwidth-bound node: B (n <= kStreamMaxN rows) is small and staged in
// shared memory k-chunk by k-chunk; the rows of A stream through once.
// Same output conventions as NodeArgs; split-K partials are reduced by the
// kernel itself (cnt).
constexpr int kStreamMaxN = 16;
constexpr int kStreamKc = 256;     // k entries of B staged per chunk (<= 32 KiB)
struct StreamArgs {
    const float2 *A;
    const float2 *B;
    void *C;
    float2 *part;
    int64_t m, n, k, kchunk;
    int32_t ksplit;
    int32_t lanes;        // threads that share one row of A (power of two <= 32)
    int32_t rows_per_cta;
    SepLayout lm, ln;
    int32_t accumulate;
    int32_t out_fmt;
    PlanarTile out_tile;
    int32_t rows_contig;  // set by the launcher: entry (i, j) lies at i n + j
    // split-K: one counter per row-block CTA (zero between runs); the last
    // split of a block to finish reduces the block's partials into C
    int32_t *cnt;
};

// Ordered sum of split-K partials into the node's output.
struct ReduceArgs {
    const float2 *part;
    void *C;
    int64_t m, n;
    int32_t ksplit;
    SepLayout lm, ln;
    int32_t accumulate;
    int32_t out_fmt;
    PlanarTile out_tile;
};

// One batched launch of tiny nodes: descriptors [first, first + count) of
// the workspace table.
// A batch holds at most kTinyLaunchNodes nodes; base[i] is the first CTA of
// node first + i (base[count] = the launch's CTAs).  The bases travel in the
// launch parameters, so a CTA finds its node without reading the table.
struct TinyLaunch {
    const TinyDesc *table;
    int32_t first, count;
    char *arena;
    float2 *out;
    int32_t accumulate_root;   // later slices: the root adds into out
    int32_t base[kTinyLaunchNodes + 1];
};

cudaError_t launch_tiny_batch(const TinyLaunch &args, int ctas, cudaStream_t stream);
cudaError_t launch_stream_node(const StreamArgs &args, cudaStream_t stream);
cudaError_t launch_splitk_reduce(const ReduceArgs &args, cudaStream_t stream);

// One tensor-core node.  A and B are planar (FMT_SPLIT4, FMT_GAUSS6 or
// FMT_BF2) and reached through 3-D TMA maps over (k, rows, plane), or 4-D
// maps when K-tiled.
struct DenseArgs {
    CUtensorMap tmA;
    CUtensorMap tmB;
    void *C;
    int64_t m, n, k;
    SepLayout lm, ln;
    int32_t accumulate;
    int32_t out_fmt;
    PlanarTile out_tile;
    int32_t bf16;         // operands are FMT_BF2
    int32_t bf16x3;       // operands are FMT_BF4 (split bf16)
    int32_t three;        // operands are FMT_GAUSS6: three real products
    int32_t narrow;       // 128 x 64 tiles (B boxes of 64 rows, MMA N = 128)
    int32_t ktiled;       // operands K-tiled (4-D maps) rather than row-major (3-D)
    int32_t pair;         // clusters of two CTAs (tiles of 256 rows; B maps of 64-row boxes)
    int32_t chunk_kb;     // k-blocks (stages) accumulated in TMEM per promotion
    DevStatus *status;
    // split-K as in NodeArgs (kchunk a multiple of 256)
    int32_t ksplit;
    int64_t kchunk;
    float2 *part;
    const EpTable *ep;    // address-order store table, or null
    // tail split (see NodePlan::tail_first): halves' sums in `part`, one
    // counter per tail tile; tail_first < 0 when off
    int64_t tail_first;
    int32_t *tail_cnt;
};

cudaError_t launch_dense(const DenseArgs &args, int num_sms, cudaStream_t stream);

// Build the TMA map of a planar operand in format `fmt` (FMT_SPLIT4,
// FMT_GAUSS6 or FMT_BF2): rows x k entries per plane.  Returns false (with a
// message) when the driver call is unavailable or rejects the shape.
// A TMA box is 64 bytes of k by box_rows rows (128, or 64 for the B side of
// a narrow node).
bool encode_operand_map(CUtensorMap *map, const void *base, int64_t rows, int64_t k, int32_t fmt,
                        bool tiled, int32_t box_rows, std::string *err);

constexpr int kPermBatch = 512;   // permutation jobs per launch

struct PermLaunch {
    int32_t njobs;
    int32_t accumulate;
    const PermDesc *table;          // device table (workspace)
    char *arena;                    // workspace arena
    float2 *out;
    int32_t job[kPermBatch];        // table index of job j
    int32_t cta_start[kPermBatch + 1];
    const float2 *src[kPermBatch];  // slice-shifted source pointers
};

cudaError_t launch_permute(const PermLaunch &args, int total_ctas, cudaStream_t stream);
cudaError_t launch_simt_node(const NodeArgs &args, cudaStream_t stream);

// CTAs a permutation job of `size` elements gets.
int permute_ctas(int64_t size);
// CTAs for one leaf job of permute_kernel (K-tiled conversions take several
// 32 x 128 blocks per CTA)
int permute_job_ctas(const PermDesc &d);

// Copy of whole leaves from pinned host memory (read through its device
// mapping over the host link) into device buffers: one launch for many
// leaves instead of one copy each.
constexpr int kGatherBatch = 256;
struct GatherLaunch {
    int32_t njobs;
    int32_t cta_start[kGatherBatch + 1];
    const float2 *src[kGatherBatch];   // device addresses of the pinned host leaves
    float2 *dst[kGatherBatch];
    int64_t size[kGatherBatch];        // elements
};
cudaError_t launch_gather(const GatherLaunch &args, int total_ctas, cudaStream_t stream);

// One launch of fused leaf subtrees (FuseGroup in plan.h): CTA x runs group
// group[x], whose leaves' slice-shifted caller pointers are
// src[src_first[x] ...].
struct FuseLaunch {
    int32_t ngroups;
    int32_t accumulate_root;   // later slices: a group rooted at the tree's root adds into out
    const FuseGroup *groups;   // device tables (workspace)
    const FuseNode *nodes;
    const FuseGather *gather;
    const int32_t *levels;
    const int32_t *offs;
    const int32_t *chunks;
    char *arena;
    float2 *out;
    int32_t group[kFuseBatch];
    int32_t src_first[kFuseBatch];
    const float2 *src[kFuseSrc];
};
cudaError_t launch_fused(const FuseLaunch &args, int smem_bytes, cudaStream_t stream);

// Entries of one stored tensor read back as complex64 (tn_plan_tensor_gather):
// dst[t] = the value of logical entry idx[t] (row-major in the tensor's
// lifetime order) of a tensor of `size` entries stored at src in format
// `fmt` with K-tiling `tile`; planar split formats give hi + lo.  An index
// outside [0, size) yields 0 and records ERR_DESC in the status word.
struct GatherArgs {
    const void *src;
    int64_t size;
    int32_t fmt;
    int32_t pad;
    PlanarTile tile;
    const int64_t *idx;
    int64_t count;
    float2 *dst;
    DevStatus *status;
};
cudaError_t launch_tensor_gather(const GatherArgs &args, cudaStream_t stream);

}  // namespace tn
