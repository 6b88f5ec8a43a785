// Internal plan structures shared by the host planner and the executor.
//
// The planner turns (network, tree, slices) into: the lifetime order of
// every tensor ("Crossing the single-GPU memory wall", section 1.4), one
// GEMM descriptor per tree step (section 1.1: A = [m, k], B = [n, k], both
// row-major, output entry (i, j) stored at offM(i) + offN(j)), one
// permutation job per leaf that is not already stored in lifetime order,
// and a workspace layout built from buffer lifetimes.
#pragma once

#include <cuda.h>   // CUtensorMap (type only; the driver is reached at run time)

#include <cstdint>
#include <string>
#include <vector>

#include "../../include/tn.h"

namespace tn {

constexpr int kMaxRank = 64;       // modes per tensor accepted by tn_plan
constexpr int kMaxPermRank = 16;   // leaf permutation rank after merging axes
constexpr int kMaxRuns = 12;       // runs per side of a separable output layout
constexpr uint64_t kAlign = 256;   // workspace alignment of every buffer

// Node policy beyond the public TN_POLICY_* values, for tests of the
// tensor-core kernel only: every node it can take (k a multiple of 4, of 8
// for bf16 operands) goes to it, whatever its shape.  Deep chains of such
// nodes carry split-tf32 operands (22 significant bits) through every level,
// so their results are not held to the complex64 tolerance; that is why the
// setting is not part of the C ABI.
constexpr int32_t kPolicyForceDense = 3;

// Output side layout.  An index i in [0, prod ext) is split mixed-radix into
// digits (run 0 most significant); its offset is sum digit[r] * stride[r]
// (in elements).  The modes of M (or N) that sit next to each other in the
// output's order form one run.
struct SepLayout {
    int32_t nrun;
    int32_t pad;
    int64_t ext[kMaxRuns];
    int64_t stride[kMaxRuns];
    int32_t shift[kMaxRuns];   // log2(ext) when ext is a power of two, else -1
};

inline int32_t log2_exact(int64_t e) {
    if (e <= 0 || (e & (e - 1)) != 0) return -1;
    int32_t s = 0;
    while ((int64_t(1) << s) < e) ++s;
    return s;
}

// Storage format of a tensor in HBM.  Every tensor is C64 except the
// operands of tensor-core (dense) nodes, which their producer writes in the
// planar form the tensor-core kernel loads with TMA:
//   FMT_SPLIT4: four fp32 planes [re_hi, im_hi, re_lo, im_lo], each the
//               tensor's row-major entries; hi = x rounded to tf32,
//               lo = (x - hi) rounded to tf32 (16 bytes per entry)
//   FMT_BF2:    two bf16 planes [re, im] (4 bytes per entry)
//   FMT_GAUSS6: six fp32 planes [re_hi, im_hi, s_hi, re_lo, im_lo, s_lo]
//               with s = re + im (rounded in fp32), split as in FMT_SPLIT4
//               (24 bytes per entry): operands of nodes that form the
//               complex product from three real products (see NodePlan)
//   FMT_BF4:    four bf16 planes [re_hi, im_hi, re_lo, im_lo]; hi = x
//               rounded to bf16 (nearest even), lo = (x - hi) rounded to
//               bf16 (8 bytes per entry): the split-bf16 precision
enum Fmt : int32_t { FMT_C64 = 0, FMT_SPLIT4 = 1, FMT_BF2 = 2, FMT_GAUSS6 = 3, FMT_BF4 = 4 };
inline uint64_t fmt_bytes(int32_t f) {
    return f == FMT_SPLIT4 ? 16 : f == FMT_BF2 ? 4 : f == FMT_GAUSS6 ? 24 : 8;   // C64, BF4: 8
}
// Planes of a planar format.
inline int32_t fmt_planes(int32_t f) {
    return f == FMT_SPLIT4 || f == FMT_BF4 ? 4 : f == FMT_BF2 ? 2 : f == FMT_GAUSS6 ? 6 : 0;
}
// Planar formats with bf16 entries.
inline bool fmt_bf16(int32_t f) { return f == FMT_BF2 || f == FMT_BF4; }

// K-tiling of a planar operand.  The consumer reads the operand as a
// row-major [rows][k] matrix; with kt > 0 each plane is stored as
// [k / kt][rows][kt], so that one tensor-core stage (kt entries of 128 rows)
// is a single contiguous 8 KiB block rather than 128 pieces one row
// (possibly megabytes) apart.  Producers map the row-major index
// r * k + c to ((c / kt) * rows + r) * kt + c % kt.  kt = 0: row-major.
struct PlanarTile {
    int64_t k;
    int64_t rows;
    int32_t kshift;   // log2(k) when k is a power of two, else -1
    int32_t kt;       // 0, 16 (tf32 planes) or 32 (bf16 planes)
};

// Entries per K tile for a planar format (64 bytes of one row).
inline int32_t planar_kt(int32_t fmt) {
    return fmt_bf16(fmt) ? 32 : (fmt == FMT_SPLIT4 || fmt == FMT_GAUSS6) ? 16 : 0;
}

// Where a tensor lives during execution.
enum PlaceKind : int32_t { PLACE_WS = 0, PLACE_LEAF = 1, PLACE_OUT = 2 };
struct Place {
    int32_t kind;
    int32_t leaf;     // PLACE_LEAF: user leaf index
    uint64_t off;     // PLACE_WS: byte offset into the workspace arena
};

// Device-side leaf permutation job (lives in the workspace descriptor
// table).  Destination index is row-major over dims (lifetime order);
// source offset is sum digit[d] * sstride[d] from the (slice-shifted) user
// pointer.
struct PermDesc {
    int64_t size;           // elements
    int64_t dst_off;        // byte offset into the arena, or -1 = output
    int32_t rank;
    int32_t fmt;            // destination format (Fmt); planes are `size` apart
    PlanarTile tile;        // destination K-tiling (planar formats)
    int64_t dims[kMaxPermRank];
    int64_t sstride[kMaxPermRank];
    int32_t dshift[kMaxPermRank];   // log2(dims) for powers of two, else -1
    // 1: the innermost dimension is contiguous in the source and a multiple
    // of 4 long, and size is a multiple of 4: a thread moves four
    // consecutive entries at a time
    int32_t vec4;
    // 1: the source holds the entries in the destination's order (a format
    // conversion, possibly K-tiled, of a leaf already in lifetime order) and
    // size is a multiple of 16: a thread moves runs of 16 entries, 16-byte
    // loads and stores
    int32_t contig;
    // a true transpose: the source's contiguous axis tax is not the
    // destination's innermost one; 32 x 32 tiles over (tax, innermost) go
    // through shared memory so that both sides move whole 32-entry rows.
    // -1 when not used
    int32_t tax;
    int32_t pad;
};

struct LeafPlan {
    int32_t leaf;
    bool identity;          // caller's layout already is the lifetime order
    bool in_place;          // consumed straight from the caller's pointer
    int64_t size;           // elements after slicing
    int64_t full_size;      // elements of the caller's leaf (all its modes)
    Place place;            // where the consumer reads it
    PermDesc perm;          // valid when !in_place
    // slicing: sliced modes this leaf carries, as (slice position, stride)
    std::vector<std::pair<int32_t, int64_t>> slice_terms;
};

struct NodePlan {
    int32_t step, a, b, out;
    uint64_t m, n, k;
    Place pa, pb, pc;
    SepLayout lm, ln;
    int32_t cls;
    int32_t level;          // 1 + max level of operand nodes (leaves: 0)
    bool is_root;
    int32_t layout;         // 0: C = [M|N], 1: C = [N|M], 2: interleaved
    int32_t out_fmt;        // format the output is stored in (Fmt)
    PlanarTile out_tile;    // K-tiling of the output (planar formats)
    int32_t ktiled;         // dense class: operands are K-tiled
    // split-K (CUDA-core classes): ksplit ranges of kchunk entries each write
    // fp32 complex partial sums [split][i][j] into `part`, then an ordered
    // reduction stores the node's output
    int32_t ksplit;
    int64_t kchunk;
    Place part;
    // stream and dense classes: operands swapped (the kernel computes
    // C^T = B A^T, rows n and columns m, through the swapped layouts) so that
    // B is the small side
    int32_t swap;
    // dense class: tiles of 128 x 64 (n <= 64 after the swap): B stacked
    // [Br; Bi] fills one N = 128 MMA instead of half an N = 256 one
    int32_t narrow;
    // dense class: runs on CTA pairs (tiles of 256 x 128, cta_group::2)
    int32_t pair;
    // dense class: complex k accumulated in TMEM per promotion into fp32
    // registers (the tensor core's accumulation rounds toward zero: shorter
    // chunks, smaller bias; see choose_chunks)
    int32_t chunk_k;
    // dense class: byte offset (from the workspace start) of the node's
    // address-order store table (EpTable), or -1 when it has none
    int64_t ep_off;
    // dense class, tail split: tiles from tail_first on (those past the last
    // full wave) run as two k halves; each half writes its fp32 sums to
    // `part` and counts itself in, per drain warp, in a counter (block of
    // counters at tail_cnt_off: byte offset from the workspace start); the
    // second to arrive adds the other half and stores.  -1: no tail split.
    int64_t tail_first;
    int64_t tail_cnt_off;
    // stream class with split-K: CTAs per split (row blocks) and their
    // counters (byte offset from the workspace start); the kernel reduces
    // its own partials, so the node has no separate reduction launch
    int64_t red_ctas;
    int64_t red_cnt_off;
    // dense class, tf32x3: the complex product from three real products
    // (Ar Br, Ai Bi, (Ar + Ai)(Br + Bi)) instead of four; operands are
    // FMT_GAUSS6
    int32_t three_products;
};

// Tensor-core tile (complex entries), its drain warps (one tail-tile
// counter each) and the bytes of a node's fp32 partial sums: split-K
// partials, or the two halves of every tail tile.
constexpr int64_t kDenseBM = 128, kDenseBN = 128;
constexpr uint64_t kDrainWarps = 8;
// Kernel view of a dense node: rows and columns after the operand swap.
inline uint64_t dense_rows(const NodePlan &nd) { return nd.swap ? nd.n : nd.m; }
inline uint64_t dense_cols(const NodePlan &nd) { return nd.swap ? nd.m : nd.n; }
inline uint64_t dense_tiles(const NodePlan &nd) {
    const uint64_t bn = nd.narrow ? kDenseBN / 2 : kDenseBN;
    const uint64_t bm = nd.pair ? 2 * kDenseBM : kDenseBM;
    return ((dense_rows(nd) + bm - 1) / bm) * ((dense_cols(nd) + bn - 1) / bn);
}
inline uint64_t part_bytes(const NodePlan &nd) {
    if (nd.ksplit > 1) return (uint64_t)nd.ksplit * nd.m * nd.n * 8;
    if (nd.tail_first >= 0)
        return (dense_tiles(nd) - (uint64_t)nd.tail_first) * 2 * kDenseBM * kDenseBN * 8;
    return 0;
}

// Address-order store table of a tensor-core node.  Every warp of the
// kernel's epilogue owns 32 output rows x 16 columns at a time; when the
// output layout repeats identically from one such block to the next, the
// entry (r, c) of a block lies at block_base + lo_m[r] + lo_n[c], and
// perm lists the 512 entries (r * 16 + c) by increasing address so that the
// warp's stores walk memory in order.
struct EpTable {
    int64_t lo_m[32];
    int64_t lo_n[16];
    uint16_t perm[512];
    // 1: the output is K-tiled with power-of-two rows and k, so tiling is a
    // permutation of address bits; lo_m / lo_n (and the sort) are then in
    // tiled addresses and the block base is tiled before they are added
    int32_t pretiled;
    // 1: in every full block the sorted entries form runs of four at
    // consecutive offsets, the first a multiple of 4 (block bases and the
    // plane size too), so a lane stores four entries at once
    int32_t vec;
};

inline int64_t tiled_offset_host(const PlanarTile &t, int64_t off) {
    if (t.kt == 0) return off;
    const int64_t r = off / t.k, c = off % t.k;
    return ((c / t.kt) * t.rows + r) * t.kt + c % t.kt;
}

// One tiny node inside a batched launch (device table).  Its operands and
// output live in the workspace arena (c_off < 0: the caller's output).
struct TinyDesc {
    int64_t a_off, b_off, c_off;
    int32_t m, n, k;
    int32_t out_fmt;
    int32_t is_root;
    PlanarTile out_tile;
    int32_t cta_base;      // first CTA of this node within its launch
    int32_t ctas;
    int32_t lanes;         // threads that share one output's k range (a power of two <= 32)
    // Output walk, so that consecutive threads store consecutive addresses:
    // address p (< m n <= 2^23) splits mixed-radix over the wn runs of the
    // output's modes, fastest first; digit d of run t adds d * wt[t] to i
    // (bit t of wside clear) or to j (bit t set).
    int32_t wn;
    uint32_t wside;
    int32_t wext[2 * kMaxRuns];
    int32_t wshift[2 * kMaxRuns];   // log2(wext) or -1
    int32_t wt[2 * kMaxRuns];
};

// Launch schedule: every node gets a stage one past its operands' stages;
// stage by stage, the tiny nodes of the stage run as one batched launch and
// the other nodes one launch each.
enum LaunchKind : int32_t { LAUNCH_PERMUTE = 0, LAUNCH_NODE = 1, LAUNCH_TINY = 2, LAUNCH_FUSED = 3 };
struct Launch {
    int32_t kind;
    int32_t node;          // LAUNCH_NODE: step
    int32_t first, count;  // LAUNCH_TINY: range in the tiny table; LAUNCH_FUSED:
                           // range in the program's fused-group list
    int32_t ctas;          // LAUNCH_TINY: CTAs of the launch
    uint64_t flops, bytes; // algorithmic work of the launch (measurement)
};

// Fused leaf subtrees ("leaf-gate absorption").  Near the leaves, a tree is
// mostly chains of tiny steps (gates absorbed into wires, small tensors
// meeting); each would cost a batched launch per tree level and a round
// trip through HBM.  A fused group is a maximal subtree whose leaves and
// intermediates are all small: one CTA reads its leaves straight from the
// caller's buffers (their permutation into lifetime order absorbed into the
// load: a list of source offsets), computes every step in shared memory
// level by level, and writes only the subtree's root, in its consumer's
// format.  All groups of a slice are independent of every other launch, so
// they run in one launch at the start.  Limits: leaves and step outputs of
// at most kFuseMaxTensor entries, a group's tensors together at most
// kFuseSmemEntries (they all stay in shared memory: no reuse), at most
// kFuseMaxMacs multiply-adds per group (one CTA does them all) and
// kFuseMaxDescBytes of step descriptors and output offsets.
constexpr int64_t kFuseMaxTensor = 2048;
constexpr int64_t kFuseSmemEntries = 8192;   // 64 KiB of complex64
constexpr int64_t kFuseMaxMacs = 1 << 15;    // complex multiply-adds of a group (one CTA)
constexpr int64_t kFuseMaxDescBytes = 24 * 1024;
constexpr int kFuseBatch = 256;              // groups per launch
constexpr int kFuseSrc = 2048;               // leaf pointers per launch
struct FuseLeaf {        // one leaf of a group (host side: its launch pointer)
    int32_t slot;        // shared-memory offset (complex entries)
    int32_t size;        // entries after slicing
    int32_t leaf;        // caller's leaf index
};
struct FuseGather {      // one leaf entry loaded into shared memory: entry e of
                         // a group's list goes to shared-memory slot e
    int32_t src;         // element offset in the (slice-shifted) caller's leaf
    int32_t leaf;        // the group's leaf (0 .. n_leaves - 1)
};
struct FuseNode {        // one step of a group (copied to shared memory)
    int32_t a, b;        // shared-memory offsets of the operands
    int32_t c;           // shared-memory offset of the output; -1: the group's root
    int32_t m, n, k;
    int32_t lshift;      // log2 of the threads that split one output's k range (<= 5)
    int32_t nshift;      // log2(n) when n is a power of two, else -1
    int32_t obase;       // first thread item of this step in its level (a multiple of
                         // 32: a warp never holds two steps)
    int32_t off;         // output offsets: offM(i) at off + i, offN(j) at off + m + j
};
struct FuseGroup {
    int32_t first_leaf, n_leaves;    // host leaf list (launch pointers)
    int32_t first_gather, n_gather;  // leaf entries (= shared-memory slots 0 .. n_gather-1)
    int32_t first_node, n_nodes;
    int32_t first_level, n_levels;   // level l: nodes [lvl[l], lvl[l + 1]) of the node list;
                                     // then lvl[n_levels + 1 + l]: its first warp chunk
    int32_t first_chunk, n_chunks;   // warp chunk (32 thread items) -> its step
    int32_t first_off, n_off;        // output offset table
    int32_t smem;                    // shared-memory entries of the group's tensors
    int32_t smem_bytes;              // tensors + descriptors (nodes, levels, offsets)
    int32_t is_root;                 // the root is the tree's root (caller's output)
    int32_t out_fmt;
    int64_t out_off;                 // arena byte offset of the root's output (-1: caller's)
    int32_t step;                    // tree step of the group's root
    int32_t pad;
    PlanarTile out_tile;
};
// Tiny nodes: at most this many complex multiply-adds (m n k), a k short
// enough for one pass of a thread group over it, and few outputs (each
// output reads its own A and B rows, which a tiled kernel would share).
// Such a node costs the batched dot-product kernel a few microseconds, less
// than a launch of its own.
constexpr uint64_t kTinyMacs = 1ull << 23;
constexpr uint64_t kTinyMaxK = 512;
constexpr uint64_t kTinyMaxOut = 1ull << 17;
constexpr int kTinyLaunchNodes = 256;   // tiny nodes per batched launch (at most)

inline int64_t sep_offset_host(const SepLayout &L, int64_t i) {
    int64_t off = 0;
    for (int r = L.nrun - 1; r >= 0; --r) {
        off += (i % L.ext[r]) * L.stride[r];
        i /= L.ext[r];
    }
    return off;
}

// True when offsets of index i0 + r (i0 a multiple of B, r < B) split as
// off(i0) + off(r): B is a product of whole innermost runs times a divisor
// of the next run.
inline bool block_invariant(const SepLayout &L, int64_t B) {
    int64_t c = 1;
    for (int r = L.nrun - 1; r >= 0; --r) {
        const int64_t e = L.ext[r];
        if (B % (c * e) == 0) {
            c *= e;
            if (c == B) return true;
            continue;
        }
        return (c * e) % B == 0 && B % c == 0;
    }
    return true;
}

// Aim of the split-K choice: at least this many CTAs per launch (two per
// SM of a GB300).
constexpr int kTargetCtas = 2 * 152;

// Launch data of a tensor-core node, built when the workspace is bound:
// 3-D TMA maps (k, rows, planes) over the planar operands.
struct DenseMaps {
    CUtensorMap a, b;
    int32_t node;
};

struct Plan {
    // inputs (copied)
    int32_t n_tensors = 0, n_modes = 0, precision = 0;
    std::vector<int64_t> extents;
    std::vector<std::vector<int32_t>> leaf_modes;
    std::vector<int32_t> open_modes;
    std::vector<int32_t> pairs;       // 2 per step
    std::vector<int32_t> slice_modes;

    // derived
    std::vector<std::vector<int32_t>> orders;   // per SSA id
    std::vector<NodePlan> nodes;
    std::vector<LeafPlan> leaves;
    std::vector<int32_t> consumer;              // per SSA id, -1 for root
    uint64_t ct_slice = 0, ct_total = 0, cs = 0, n_slices = 1;
    uint64_t out_elems = 1;
    std::vector<int64_t> slice_ext;             // extents of sliced modes

    // execution layout
    int32_t policy = TN_POLICY_AUTO;
    int32_t three_products = 0;   // tn_plan_set_three_products
    int32_t cta_pairs = 0;        // tn_plan_set_cta_pairs
    int32_t chunk_k = 0;          // tn_plan_set_promotion_chunk (0: per-plan rule)
    int32_t hoist = 1;            // tn_plan_set_hoisting
    uint64_t table_off = 0, table_bytes = 0;    // PermDesc table
    uint64_t arena_off = 0, arena_bytes = 0;
    uint64_t ws_bytes = 0;
    std::vector<PermDesc> perm_table;
    std::vector<int32_t> perm_leaves;           // leaf of each table entry
    std::vector<unsigned char> table_blob;      // device tables: PermDesc[], EpTable[], TinyDesc[]
    std::vector<Launch> sched;                  // launches of one slice, in order
    std::vector<int32_t> launch_of;             // per step: its launch's index in sched
    // Slice-invariant hoisting (with slices and hoist set): a tensor is
    // variant when a sliced leaf lies below it.  The first slice an execute
    // runs takes `sched` and every leaf job; later slices take `sched_rest`
    // (the variant launches) and `perm_rest` (the variant leaves' jobs),
    // since the invariant tensors they read are still in the arena.
    std::vector<uint8_t> variant;               // per SSA id
    std::vector<Launch> sched_rest;
    std::vector<int32_t> perm_all, perm_rest;   // perm_table entries of each program
    uint64_t tiny_off = 0;                      // workspace offset of the TinyDesc table
    // fused leaf subtrees (tn_plan_set_fusion): groups and their tables
    int32_t fuse = 1;
    std::vector<int32_t> fused;                 // per step: index of its group, or -1
    std::vector<FuseGroup> fuse_groups;
    std::vector<int32_t> fuse_all, fuse_rest;   // groups each program runs
    uint64_t fuse_off = 0;                      // workspace offsets of FuseGroup[], FuseNode[],
    uint64_t fuse_node_off = 0, fuse_gather_off = 0, fuse_lvl_off = 0, fuse_offs_off = 0;   // FuseGather[], levels, offsets
    uint64_t fuse_chunk_off = 0;                // chunk -> step tables
    int32_t fuse_smem = 0;                      // largest group's shared memory (bytes)
    std::vector<FuseLeaf> fuse_leaves_host;     // host copy of FuseLeaf[] (launch parameters)
    std::vector<int32_t> fmt;                   // per SSA id (Fmt)
    std::vector<DenseMaps> dense_maps;          // per dense node, set at bind
    void *maps_ws = nullptr;                    // workspace the maps point into
    int num_sms = 0;

    // measurement
    bool profiling = false;
    std::vector<void *> events;                 // cudaEvent_t pairs
    std::vector<tn_launch_record> records;
    uint64_t launches_per_exec = 0;

    // replay: the launch sequence of the last (leaves, output, workspace)
    // captured as a CUDA graph (graph exec and capture stream as opaque
    // handles; exec.cu)
    bool use_graph = true;
    void *graph_exec = nullptr;
    void *capture_stream = nullptr;
    std::vector<void *> lane_streams;           // recording: extra streams for independent launches
    // tn_execute_host: host leaf pointers seen last and their device mappings
    // (null: pageable, copied with cudaMemcpyAsync)
    std::vector<const void *> host_leaves_seen, host_leaves_dev;
    // tn_execute_host with pinned leaves and output: the whole call (gather,
    // contraction, copy out) recorded as one graph for these buffers
    void *host_graph_exec = nullptr;
    std::vector<const void *> hg_key;           // host leaves, host out, device leaves, device out, workspace
    std::vector<void *> dag_events;             // recording: one event per launch
    std::vector<const void *> graph_leaves;
    void *graph_out = nullptr;
    void *graph_ws = nullptr;

    // tn_execute_prefix: the step it stopped after (-1: none since the last
    // full execute) and the slice-0 pointers of its leaves and output, read
    // by tn_plan_tensor_gather
    int32_t prefix_step = -1;
    std::vector<const void *> prefix_leaves;
    void *prefix_out = nullptr;

    // the last execute of this plan ran on the library's static scratch
    // array (tn_execute_static): tn_plan_check reads that array's status word
    bool last_static = false;

    // binding
    void *ws = nullptr;
    uint64_t ws_size = 0;
    int device = -1;

    std::string last_error;
};

// Build the plan; returns TN_OK or an error with plan->last_error (or err)
// describing it.
tn_status build_plan(const tn_network *net, const tn_tree *tree, const tn_slices *sl,
                     Plan *plan, std::string *err);

// Classify nodes under plan->policy and lay out the workspace.
tn_status layout_plan(Plan *plan);

// Destroy the plan's CUDA events, recorded graph and capture stream (exec.cu).
void release_events(Plan *plan);

// Forget the recorded launch graph (exec.cu).
void drop_graph(Plan *plan);

}  // namespace tn

// The opaque handle behind tn_plan_t.
struct tn_plan_s {
    tn::Plan p;
    ~tn_plan_s() { tn::release_events(&p); }
};
