// Node classes, launch schedule, workspace layout and device tables.
//
// Runs after build_plan (and again whenever the policy changes); host only.
//   1. classify every node (tensor-core, streaming, general, tiny) and
//      choose its split-K;
//   2. storage formats: operands of tensor-core nodes are written planar by
//      their producers, everything else is complex64;
//   3. schedule: a node's stage is one past the stages of its operands; stage
//      by stage, all tiny nodes of the stage form one batched launch and
//      every other node gets its own launch (the root, which depends on
//      everything, comes last);
//   4. buffer lifetimes on that launch order and an offline placement into
//      one arena (largest first, lowest free offset);
//   5. device tables: leaf permutation jobs, address-order store tables of
//      tensor-core nodes, tiny-node descriptors.
#include <algorithm>
#include <cstring>

#include "plan.h"

namespace tn {

int classify(const Plan &p, const NodePlan &nd);   // exec.cu
void choose_split(const Plan &p, NodePlan &nd);    // exec.cu
uint64_t launches_of(const Plan &p, bool first);  // exec.cu

namespace {

struct Interval {
    uint64_t bytes;
    int start, end;   // launch indices; leaf copies start at -1
    int id;
    uint64_t off;
};

// Largest buffers first, each at the lowest offset that overlaps no placed
// buffer alive at the same time.  Operands end at the launch that reads
// them and outputs start there, so a launch never aliases its own buffers.
uint64_t place_buffers(std::vector<Interval> &iv) {
    std::vector<int> order(iv.size());
    for (size_t i = 0; i < iv.size(); ++i) order[i] = (int)i;
    std::sort(order.begin(), order.end(), [&](int x, int y) {
        if (iv[x].bytes != iv[y].bytes) return iv[x].bytes > iv[y].bytes;
        return iv[x].start < iv[y].start;
    });
    std::vector<int> placed;
    uint64_t peak = 0;
    for (int i : order) {
        std::vector<std::pair<uint64_t, uint64_t>> busy;
        for (int j : placed)
            if (!(iv[j].end < iv[i].start || iv[i].end < iv[j].start))
                busy.push_back({iv[j].off, iv[j].off + iv[j].bytes});
        std::sort(busy.begin(), busy.end());
        uint64_t off = 0;
        for (auto &b : busy) {
            if (off + iv[i].bytes <= b.first) break;
            off = std::max(off, (b.second + kAlign - 1) / kAlign * kAlign);
        }
        iv[i].off = off;
        peak = std::max(peak, off + iv[i].bytes);
        placed.push_back(i);
    }
    return (peak + kAlign - 1) / kAlign * kAlign;
}

uint64_t align_up(uint64_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Three real products instead of four (FMT_GAUSS6 operands) where the node
// stays bound by its arithmetic with 24-byte operand entries (flops per byte
// well above the ratio of the tensor and HBM peaks, about 50) and its
// operands stay below 64 GiB in that format.
bool three_products_pay(const NodePlan &nd) {
    const double m = (double)nd.m, n = (double)nd.n, k = (double)nd.k;
    const double in_b = 24.0 * (m * k + n * k);
    const double intensity = 8.0 * m * n * k / (in_b + 8.0 * m * n);
    return nd.k >= 256 && intensity >= 64.0 && in_b <= 64.0 * (1ull << 30);
}

// Whether the sorted order of a full 32 x 16 block splits into runs of four
// consecutive offsets starting at multiples of 4, with every block base and
// the plane size multiples of 4 as well.  (K-tiling keeps such runs
// contiguous: its tiles hold 16 or 32 entries and tiling keeps the low bits.)
bool quad_stores_ok(const NodePlan &nd, const EpTable &t) {
    if (nd.m < 32 || nd.n < 16) return false;
    if (nd.out_fmt != FMT_C64 && (nd.m * nd.n) % 4 != 0) return false;
    for (int g = 0; g < 128; ++g) {
        const int e0 = t.perm[4 * g];
        const int64_t o = t.lo_m[e0 >> 4] + t.lo_n[e0 & 15];
        if (o % 4 != 0) return false;
        for (int u = 1; u < 4; ++u) {
            const int e = t.perm[4 * g + u];
            if (t.lo_m[e >> 4] + t.lo_n[e & 15] != o + u) return false;
        }
    }
    for (uint64_t i0 = 0; i0 < nd.m; i0 += 32)
        if (sep_offset_host(nd.lm, (int64_t)i0) % 4 != 0) return false;
    for (uint64_t j0 = 0; j0 < nd.n; j0 += 16)
        if (sep_offset_host(nd.ln, (int64_t)j0) % 4 != 0) return false;
    return true;
}

// The output walk of a tiny node (see TinyDesc): the runs of M and N,
// each with its digit's weight in i or j, sorted by their stride in the
// output.  Those strides nest (1, e0, e0 e1, ...) because the output is a
// dense row-major tensor over the M and N modes.
bool make_walk(const NodePlan &nd, TinyDesc *d) {
    struct Run {
        int64_t ext, stride, weight;
        int side;
    };
    std::vector<Run> runs;
    auto add = [&](const SepLayout &L, int side) {
        int64_t w = 1;
        for (int r = L.nrun - 1; r >= 0; --r) {
            if (L.ext[r] > 1) runs.push_back({L.ext[r], L.stride[r], w, side});
            w *= L.ext[r];
        }
    };
    add(nd.lm, 0);
    add(nd.ln, 1);
    std::sort(runs.begin(), runs.end(), [](const Run &x, const Run &y) { return x.stride < y.stride; });
    if (runs.size() > 2 * (size_t)kMaxRuns) return false;
    int64_t expect = 1;
    d->wn = (int32_t)runs.size();
    d->wside = 0;
    for (size_t t = 0; t < runs.size(); ++t) {
        if (runs[t].stride != expect) return false;
        expect *= runs[t].ext;
        d->wext[t] = (int32_t)runs[t].ext;
        d->wshift[t] = log2_exact(runs[t].ext);
        d->wt[t] = (int32_t)runs[t].weight;
        if (runs[t].side) d->wside |= 1u << t;
    }
    return expect == (int64_t)(nd.m * nd.n);
}

bool make_ep_table(const NodePlan &nd, EpTable *t) {
    if (!block_invariant(nd.lm, 32) || !block_invariant(nd.ln, 16)) return false;
    std::memset(t, 0, sizeof(*t));
    for (int r = 0; r < 32; ++r) t->lo_m[r] = r < (int64_t)nd.m ? sep_offset_host(nd.lm, r) : 0;
    for (int c = 0; c < 16; ++c) t->lo_n[c] = c < (int64_t)nd.n ? sep_offset_host(nd.ln, c) : 0;
    std::vector<uint16_t> idx(512);
    for (int e = 0; e < 512; ++e) idx[e] = (uint16_t)e;
    auto key = [&](uint16_t e) -> int64_t {
        const int r = e >> 4, c = e & 15;
        if (r >= (int64_t)nd.m || c >= (int64_t)nd.n) return INT64_MAX;
        return t->lo_m[r] + t->lo_n[c];
    };
    // power-of-two extents: every mode owns its own address bits, and K-tiling
    // with power-of-two rows and k only moves bits, so the tiled address of
    // base + lo_m[r] + lo_n[c] is the sum of the three tiled parts
    const PlanarTile &tl = nd.out_tile;
    auto pow2_layout = [](const SepLayout &L) {
        for (int r = 0; r < L.nrun; ++r)
            if (L.shift[r] < 0 || log2_exact(L.stride[r]) < 0) return false;
        return true;
    };
    if (tl.kt != 0 && tl.kshift >= 0 && log2_exact(tl.rows) >= 0 && pow2_layout(nd.lm) &&
        pow2_layout(nd.ln)) {
        t->pretiled = 1;
        for (int r = 0; r < 32; ++r) t->lo_m[r] = tiled_offset_host(tl, t->lo_m[r]);
        for (int c = 0; c < 16; ++c) t->lo_n[c] = tiled_offset_host(tl, t->lo_n[c]);
    }
    std::stable_sort(idx.begin(), idx.end(), [&](uint16_t x, uint16_t y) { return key(x) < key(y); });
    for (int e = 0; e < 512; ++e) t->perm[e] = idx[e];
    t->vec = quad_stores_ok(nd, *t) ? 1 : 0;
    return true;
}

// Fused leaf subtrees (FuseGroup in plan.h).  A step may sit in a group when
// it is tiny, its output and its k have at most kFuseMaxTensor entries, each
// operand is a small leaf (at most kFuseMaxTensor entries) or such a step,
// and its subtree's tensors together fit kFuseSmemEntries, its multiply-adds
// kFuseMaxMacs and its descriptors kFuseMaxDescBytes.  A group is a maximal
// such subtree (at least one step); its root is a step whose consumer cannot
// join it.
int64_t fuse_desc_bytes(int64_t nodes, int64_t offsets, int64_t levels, int64_t chunks) {
    return nodes * (int64_t)sizeof(FuseNode) + 4 * (offsets + 2 * (levels + 1) + chunks);
}

void form_groups(Plan *p, std::vector<FuseNode> &fnodes, std::vector<FuseGather> &fgather,
                 std::vector<int32_t> &flevels, std::vector<int32_t> &foffs,
                 std::vector<int32_t> &fchunks, std::vector<FuseLeaf> &fleaves,
                 std::vector<uint8_t> &leaf_fused) {
    const int n = p->n_tensors, S = (int)p->nodes.size();
    std::vector<uint8_t> ok(n + S, 0);
    std::vector<int64_t> cost(n + S, 0), macs(n + S, 0), nsteps(n + S, 0), noffs(n + S, 0);
    for (int t = 0; t < n; ++t) {
        const LeafPlan &lp = p->leaves[t];
        ok[t] = lp.size <= kFuseMaxTensor && lp.full_size < (int64_t(1) << 31);
        cost[t] = lp.size;
    }
    for (int s = 0; s < S; ++s) {
        const NodePlan &nd = p->nodes[s];
        const int64_t mn = (int64_t)(nd.m * nd.n);
        cost[nd.out] = cost[nd.a] + cost[nd.b] + mn;
        macs[nd.out] = macs[nd.a] + macs[nd.b] + mn * (int64_t)nd.k;
        nsteps[nd.out] = nsteps[nd.a] + nsteps[nd.b] + 1;
        noffs[nd.out] = noffs[nd.a] + noffs[nd.b] + (int64_t)(nd.m + nd.n);
        ok[nd.out] = nd.cls == TN_NODE_TINY && ok[nd.a] && ok[nd.b] && mn <= kFuseMaxTensor &&
                     (int64_t)nd.k <= kFuseMaxTensor && cost[nd.out] <= kFuseSmemEntries &&
                     macs[nd.out] <= kFuseMaxMacs &&
                     fuse_desc_bytes(nsteps[nd.out], noffs[nd.out], nsteps[nd.out],
                                     (macs[nd.out] + 31) / 32 + 32 * nsteps[nd.out]) <= kFuseMaxDescBytes;
    }
    for (int r = 0; r < S; ++r) {
        const NodePlan &rn = p->nodes[r];
        if (!ok[rn.out]) continue;
        const int cons = p->consumer[rn.out];
        if (cons >= 0 && ok[p->nodes[cons].out]) continue;   // the group goes on above
        // the subtree's steps (ascending: operands before their consumers)
        // and leaves
        std::vector<int> steps, leaves, stack{rn.out};
        while (!stack.empty()) {
            const int id = stack.back();
            stack.pop_back();
            if (id < n) {
                leaves.push_back(id);
                continue;
            }
            steps.push_back(id - n);
            stack.push_back(p->nodes[id - n].a);
            stack.push_back(p->nodes[id - n].b);
        }
        std::sort(steps.begin(), steps.end());
        std::sort(leaves.begin(), leaves.end());
        const int gi = (int)p->fuse_groups.size();
        FuseGroup G;
        std::memset(&G, 0, sizeof(G));
        G.step = r;
        G.first_leaf = (int32_t)fleaves.size();
        G.n_leaves = (int32_t)leaves.size();
        G.first_gather = (int32_t)fgather.size();
        // shared memory: leaves first (in list order: slot e holds gather
        // entry e), then the outputs of the inner steps
        std::vector<int32_t> slot(n + S, -1);
        int32_t used = 0;
        for (size_t l = 0; l < leaves.size(); ++l) {
            const int t = leaves[l];
            const LeafPlan &lp = p->leaves[t];
            fleaves.push_back(FuseLeaf{used, (int32_t)lp.size, t});
            slot[t] = used;
            // entry e (row-major over the lifetime order) comes from
            // sum digit[d] * sstride[d] of the caller's (slice-shifted) leaf
            const PermDesc &d = lp.perm;
            for (int64_t e = 0; e < lp.size; ++e) {
                int64_t rem = e, so = 0;
                for (int x = d.rank - 1; x >= 0; --x) {
                    so += (rem % d.dims[x]) * d.sstride[x];
                    rem /= d.dims[x];
                }
                fgather.push_back(FuseGather{(int32_t)so, (int32_t)l});
            }
            used += (int32_t)lp.size;
            leaf_fused[t] = 1;
        }
        G.n_gather = used;
        std::vector<int> level(n + S, 0);
        int nlev = 0;
        for (int s : steps) {
            const NodePlan &nd = p->nodes[s];
            level[nd.out] = 1 + std::max(level[nd.a], level[nd.b]);
            nlev = std::max(nlev, level[nd.out]);
            if (s != r) {
                slot[nd.out] = used;
                used += (int32_t)(nd.m * nd.n);
            }
        }
        G.smem = used;
        G.first_node = (int32_t)fnodes.size();
        G.n_nodes = (int32_t)steps.size();
        G.first_level = (int32_t)flevels.size();
        G.n_levels = nlev;
        G.first_off = (int32_t)foffs.size();
        G.first_chunk = (int32_t)fchunks.size();
        std::vector<int32_t> lchunk;
        for (int lv = 1; lv <= nlev; ++lv) {
            flevels.push_back((int32_t)(fnodes.size() - (size_t)G.first_node));
            lchunk.push_back((int32_t)(fchunks.size() - (size_t)G.first_chunk));
            int32_t obase = 0;
            for (int s : steps) {
                const NodePlan &nd = p->nodes[s];
                if (level[nd.out] != lv) continue;
                FuseNode f;
                f.a = slot[nd.a];
                f.b = slot[nd.b];
                f.c = s == r ? -1 : slot[nd.out];
                f.m = (int32_t)nd.m;
                f.n = (int32_t)nd.n;
                f.k = (int32_t)nd.k;
                // a few k entries per thread: long k ranges are split over
                // up to 32 threads (one serial chain of k multiply-adds per
                // thread would be the group's critical path)
                f.lshift = 0;
                while (f.lshift < 5 && (4 << f.lshift) < f.k) ++f.lshift;
                f.nshift = -1;
                for (int32_t t = 0; t < 31; ++t)
                    if ((int32_t(1) << t) == f.n) f.nshift = t;
                f.obase = obase;
                obase += (((f.m * f.n) << f.lshift) + 31) / 32 * 32;
                // the step of every warp chunk of this level
                for (int32_t c = f.obase; c < obase; c += 32)
                    fchunks.push_back((int32_t)(fnodes.size() - (size_t)G.first_node));
                f.off = (int32_t)(foffs.size() - (size_t)G.first_off);
                for (uint64_t i = 0; i < nd.m; ++i) foffs.push_back((int32_t)sep_offset_host(nd.lm, (int64_t)i));
                for (uint64_t j = 0; j < nd.n; ++j) foffs.push_back((int32_t)sep_offset_host(nd.ln, (int64_t)j));
                fnodes.push_back(f);
            }
        }
        flevels.push_back((int32_t)(fnodes.size() - (size_t)G.first_node));
        lchunk.push_back((int32_t)(fchunks.size() - (size_t)G.first_chunk));
        flevels.insert(flevels.end(), lchunk.begin(), lchunk.end());
        G.n_off = (int32_t)(foffs.size() - (size_t)G.first_off);
        G.n_chunks = (int32_t)(fchunks.size() - (size_t)G.first_chunk);
        G.smem_bytes = (int32_t)(8 * (int64_t)G.smem +
                                 fuse_desc_bytes(G.n_nodes, G.n_off, G.n_levels, G.n_chunks));
        for (int s : steps) p->fused[s] = gi;
        p->fuse_smem = std::max(p->fuse_smem, G.smem_bytes);
        p->fuse_groups.push_back(G);
    }
}

// Promotion chunk of the tensor-core nodes.  The tensor core accumulates in
// TMEM with rounding toward zero, which biases every node's sums toward zero
// by about 1.3e-6 (relative) with 256-k chunks, half of that with 128 and a
// quarter with 64 (measured on chains of 2^30- to 2^32-entry nodes), and the
// relative errors of a tree's nodes add up at its root.  The chunk is the
// longest whose bias times the number of tensor-core nodes stays within 4e-6
// (the complex64 tolerance is 1e-5): a longer chunk costs less bookkeeping
// per k.  The kernel makes the first chunk of a tile of eight or more chunks
// twice as long (the tile's bias grows by at most a quarter, an eighth at
// sixteen chunks), which the budget does not count: on the 7x7 x 10-cycle
// circuit (six nodes, 128-k chunks) the estimate grows from 3.9e-6 to
// 4.1e-6, still well inside the tolerance (the exact-value norm networks
// measure 4.3e-6 and 6.4e-6 in all).  CTA pairs accumulate six products per
// k-step into one accumulator instead of three: half the chunk.  Plain bf16
// operands (tolerance 2e-2,
// rounding error of the operands ~1e-3) take 2048: their stages are short on
// the tensor core, so each promotion's drain costs relatively more.
void choose_chunks(Plan *p) {
    int dense = 0;
    for (const auto &nd : p->nodes) dense += nd.cls == TN_NODE_DENSE ? 1 : 0;
    int32_t chunk = dense <= 3 ? 256 : dense <= 6 ? 128 : 64;
    if (p->precision == TN_PREC_BF16) chunk = 2048;
    if (p->chunk_k > 0) chunk = p->chunk_k;   // tn_plan_set_promotion_chunk
    // at least one pipeline stage (16 complex k of tf32 planes, 32 of bf16)
    const int32_t stage = (p->precision == TN_PREC_BF16 || p->precision == TN_PREC_BF16X3) ? 32 : 16;
    for (auto &nd : p->nodes) nd.chunk_k = std::max(stage, nd.pair ? chunk / 2 : chunk);
}

}  // namespace

tn_status layout_plan(Plan *p) {
    const int n = p->n_tensors;
    const int S = (int)p->nodes.size();
    drop_graph(p);
    for (auto &nd : p->nodes) {
        nd.cls = classify(*p, nd);
        choose_split(*p, nd);
    }

    // 2. formats
    p->fmt.assign(n + S, FMT_C64);
    const int32_t dense_fmt = p->precision == TN_PREC_BF16     ? FMT_BF2
                              : p->precision == TN_PREC_BF16X3 ? FMT_BF4
                                                               : FMT_SPLIT4;
    for (auto &nd : p->nodes) {
        nd.three_products = 0;
        if (nd.cls != TN_NODE_DENSE) continue;
        int32_t f = dense_fmt;
        if (f == FMT_SPLIT4 && p->three_products && !nd.narrow && three_products_pay(nd)) {
            nd.pair = 0;   // the three-product kernel runs on single CTAs
            f = FMT_GAUSS6;
            nd.three_products = 1;
        }
        p->fmt[nd.a] = p->fmt[nd.b] = f;
    }
    for (auto &nd : p->nodes) nd.out_fmt = nd.is_root ? FMT_C64 : p->fmt[nd.out];
    choose_chunks(p);
    // K-tiling of tensor-core operands whose k fills whole tiles
    const PlanarTile untiled{0, 0, -1, 0};
    std::vector<PlanarTile> tile(n + S, untiled);
    for (auto &nd : p->nodes) {
        nd.ktiled = 0;
        if (nd.cls != TN_NODE_DENSE) continue;
        const int32_t kt = planar_kt(p->fmt[nd.a]);
        // rows of 8 KiB and more per plane: 64-byte pieces would each cost
        // a DRAM page
        if (nd.k % (uint64_t)kt != 0 || nd.k < 2048) continue;
        nd.ktiled = 1;
        const int32_t ks = log2_exact((int64_t)nd.k);
        tile[nd.a] = PlanarTile{(int64_t)nd.k, (int64_t)nd.m, ks, kt};
        tile[nd.b] = PlanarTile{(int64_t)nd.k, (int64_t)nd.n, ks, kt};
    }
    for (auto &nd : p->nodes) nd.out_tile = nd.is_root ? untiled : tile[nd.out];

    // 2b. fused leaf subtrees (see FuseGroup in plan.h)
    std::vector<FuseNode> fnodes;
    std::vector<FuseGather> fgather;
    std::vector<FuseLeaf> fleaves;
    std::vector<int32_t> flevels, foffs, fchunks;
    std::vector<uint8_t> leaf_fused(n, 0);
    p->fused.assign(S, -1);
    p->fuse_groups.clear();
    p->fuse_smem = 0;
    if (p->fuse && p->policy == TN_POLICY_AUTO && S > 0)
        form_groups(p, fnodes, fgather, flevels, foffs, fchunks, fleaves, leaf_fused);

    // 3. schedule (group roots are ready after the fused launch at the start)
    std::vector<int> stage(n + S, 0);
    int max_stage = 0;
    for (const auto &nd : p->nodes) {
        if (p->fused[nd.step] >= 0) continue;
        stage[nd.out] = 1 + std::max(stage[nd.a], stage[nd.b]);
        max_stage = std::max(max_stage, stage[nd.out]);
    }
    std::vector<std::vector<int>> by_stage(max_stage + 1);
    for (int s = 0; s < S; ++s)
        if (p->fused[s] < 0) by_stage[stage[n + s]].push_back(s);
    // Slice-invariant subtrees (section 1.1 of "Crossing the single-GPU
    // memory wall": slicing repeats every node once per slice, although a
    // node whose subtree holds no sliced leaf computes the same tensor in
    // every slice).  With hoisting, later slices run only the variant
    // launches.
    p->variant.assign(n + S, 0);
    for (int t = 0; t < n; ++t) p->variant[t] = p->leaves[t].slice_terms.empty() ? 0 : 1;
    for (const auto &nd : p->nodes) p->variant[nd.out] = p->variant[nd.a] | p->variant[nd.b];
    const bool hoist = p->hoist && p->n_slices > 1;
    p->sched.clear();
    p->sched_rest.clear();
    std::vector<int> t_of(n + S, -1);   // launch index producing each id
    std::vector<std::vector<int>> tiny_batches, tiny_batches_rest;
    // one program: stage by stage, the stage's tiny nodes in batches of at
    // most kTinyLaunchNodes (independent launches), then its other nodes
    p->fuse_all.clear();
    p->fuse_rest.clear();
    for (int g = 0; g < (int)p->fuse_groups.size(); ++g) {
        p->fuse_all.push_back(g);
        if (hoist && p->variant[n + p->fuse_groups[g].step]) p->fuse_rest.push_back(g);
    }
    auto build = [&](std::vector<Launch> &sched, std::vector<std::vector<int>> &batches, bool rest) {
        // fused groups: batches of at most kFuseBatch groups and kFuseSrc leaves
        const std::vector<int32_t> &groups = rest ? p->fuse_rest : p->fuse_all;
        for (size_t g0 = 0; g0 < groups.size();) {
            Launch L{};
            L.kind = LAUNCH_FUSED;
            L.node = -1;
            L.first = (int32_t)g0;
            int leaves = 0;
            size_t g1 = g0;
            while (g1 < groups.size() && (int)(g1 - g0) < kFuseBatch &&
                   leaves + p->fuse_groups[groups[g1]].n_leaves <= kFuseSrc) {
                const FuseGroup &G = p->fuse_groups[groups[g1]];
                leaves += G.n_leaves;
                for (int x = G.first_node; x < G.first_node + G.n_nodes; ++x) {
                    const FuseNode &fn = fnodes[x];
                    L.flops += 8 * (uint64_t)fn.m * fn.n * fn.k;
                }
                L.bytes += 8 * (uint64_t)G.n_gather;
                const NodePlan &rn = p->nodes[G.step];
                L.bytes += fmt_bytes(rn.out_fmt) * rn.m * rn.n;
                ++g1;
            }
            L.count = (int32_t)(g1 - g0);
            L.ctas = L.count;
            if (!rest)
                for (size_t x = g0; x < g1; ++x)
                    for (int s2 = 0; s2 < S; ++s2)
                        if (p->fused[s2] == groups[x]) t_of[n + s2] = (int)sched.size();
            sched.push_back(L);
            g0 = g1;
        }
        for (int st = 1; st <= max_stage; ++st) {
            std::vector<int> tiny, other;
            for (int s : by_stage[st]) {
                if (rest && !p->variant[n + s]) continue;
                (p->nodes[s].cls == TN_NODE_TINY ? tiny : other).push_back(s);
            }
            for (size_t b0 = 0; b0 < tiny.size(); b0 += kTinyLaunchNodes) {
                const size_t b1 = std::min(tiny.size(), b0 + (size_t)kTinyLaunchNodes);
                Launch L{};
                L.kind = LAUNCH_TINY;
                L.node = -1;
                if (!rest)
                    for (size_t x = b0; x < b1; ++x) t_of[n + tiny[x]] = (int)sched.size();
                batches.emplace_back(tiny.begin() + b0, tiny.begin() + b1);
                sched.push_back(L);
            }
            for (int s : other) {
                Launch L{};
                L.kind = LAUNCH_NODE;
                L.node = s;
                if (!rest) t_of[n + s] = (int)sched.size();
                sched.push_back(L);
            }
        }
    };
    build(p->sched, tiny_batches, false);
    if (hoist) build(p->sched_rest, tiny_batches_rest, true);
    auto consume_t = [&](int id) { return p->consumer[id] < 0 ? (int)p->sched.size()
                                                               : t_of[n + p->consumer[id]]; };
    // an invariant tensor that a variant node reads is written by the first
    // slice and read by every later one: it stays live for the whole run
    auto pinned = [&](int id) {
        return hoist && !p->variant[id] && p->consumer[id] >= 0 &&
               p->variant[p->nodes[p->consumer[id]].out];
    };
    const int run_end = (int)p->sched.size() + 1;

    // 4. lifetimes and placement
    std::vector<Interval> iv;
    for (int t = 0; t < n; ++t) {
        LeafPlan &lp = p->leaves[t];
        const bool tiny_consumer = S > 0 && p->nodes[p->consumer[t]].cls == TN_NODE_TINY;
        lp.in_place = S > 0 && lp.identity && p->fmt[t] == FMT_C64 && !tiny_consumer;
        if (leaf_fused[t]) {
            // read by its group's CTA straight from the caller's buffer
            lp.in_place = true;
            lp.place = {PLACE_LEAF, t, 0};
        } else if (S == 0) {
            lp.place = {PLACE_OUT, t, 0};
        } else if (lp.in_place) {
            lp.place = {PLACE_LEAF, t, 0};
        } else {
            iv.push_back({(uint64_t)lp.size * fmt_bytes(p->fmt[t]), -1,
                          pinned(t) ? run_end : consume_t(t), t, 0});
        }
    }
    for (int s = 0; s < S; ++s) {
        const NodePlan &nd = p->nodes[s];
        const int ts = t_of[n + s];
        // inside a fused group only the group's root reaches the workspace
        if (p->fused[s] >= 0 && p->fuse_groups[p->fused[s]].step != s) continue;
        if (!nd.is_root) {
            if (pinned(nd.out))
                iv.push_back({nd.m * nd.n * fmt_bytes(nd.out_fmt), -1, run_end, nd.out, 0});
            else
                iv.push_back({nd.m * nd.n * fmt_bytes(nd.out_fmt), ts, consume_t(nd.out), nd.out, 0});
        }
        if (part_bytes(nd) > 0) iv.push_back({part_bytes(nd), ts, ts, n + S + s, 0});
    }
    p->arena_bytes = place_buffers(iv);
    std::vector<Place> where(n + 2 * S, Place{PLACE_WS, -1, 0});
    for (const auto &b : iv) where[b.id] = {PLACE_WS, -1, b.off};
    p->perm_table.clear();
    p->perm_leaves.clear();
    for (int t = 0; t < n; ++t) {
        LeafPlan &lp = p->leaves[t];
        if (S > 0 && !lp.in_place) lp.place = where[t];
        where[t] = lp.place;
        if (leaf_fused[t]) continue;
        if (S == 0 || !lp.in_place) {
            PermDesc d = lp.perm;
            d.dst_off = (lp.place.kind == PLACE_OUT) ? -1 : (int64_t)lp.place.off;
            d.fmt = (S == 0) ? FMT_C64 : p->fmt[t];
            d.tile = (S == 0) ? untiled : tile[t];
            d.vec4 = d.rank >= 1 && d.sstride[d.rank - 1] == 1 && d.dims[d.rank - 1] % 4 == 0 &&
                     d.size % 4 == 0;
            d.contig = d.rank == 1 && d.sstride[0] == 1 && d.size % 16 == 0;
            // (small leaves stay on the general path: their transposes are a
            // few loads of latency, not bandwidth)
            d.tax = -1;
            if (d.rank >= 2 && d.size >= (1 << 16) && d.sstride[d.rank - 1] != 1 &&
                d.dims[d.rank - 1] >= 8)
                for (int x = 0; x < d.rank - 1; ++x)
                    if (d.sstride[x] == 1 && d.dims[x] >= 8) d.tax = x;
            p->perm_table.push_back(d);
            p->perm_leaves.push_back(t);
        }
    }
    p->perm_all.clear();
    p->perm_rest.clear();
    for (int j = 0; j < (int)p->perm_table.size(); ++j) {
        p->perm_all.push_back(j);
        if (hoist && p->variant[p->perm_leaves[j]]) p->perm_rest.push_back(j);
    }
    auto perm_launch = [&](const std::vector<int32_t> &jobs, std::vector<Launch> &sched) {
        if (jobs.empty()) return;
        Launch L{};
        L.kind = LAUNCH_PERMUTE;
        L.node = -1;
        for (int j : jobs)
            L.bytes += (8 + fmt_bytes(p->perm_table[j].dst_off < 0 ? (int32_t)FMT_C64 : p->perm_table[j].fmt)) *
                       (uint64_t)p->perm_table[j].size;
        sched.insert(sched.begin(), L);
    };
    perm_launch(p->perm_all, p->sched);
    if (hoist) perm_launch(p->perm_rest, p->sched_rest);
    // index in sched of the launch that computes each step (after the leaf
    // permutation launch, when there is one)
    p->launch_of.assign(S, -1);
    for (int s = 0; s < S; ++s)
        p->launch_of[s] = t_of[n + s] < 0 ? -1 : t_of[n + s] + (p->perm_all.empty() ? 0 : 1);
    for (int s = 0; s < S; ++s) {
        NodePlan &nd = p->nodes[s];
        if (nd.is_root) where[nd.out] = {PLACE_OUT, -1, 0};
        nd.pa = where[nd.a];
        nd.pb = where[nd.b];
        nd.pc = where[nd.out];
        nd.part = where[n + S + s];
    }

    for (auto &G : p->fuse_groups) {
        const NodePlan &rn = p->nodes[G.step];
        G.is_root = rn.is_root ? 1 : 0;
        G.out_off = rn.pc.kind == PLACE_OUT ? -1 : (int64_t)rn.pc.off;
        G.out_fmt = rn.out_fmt;
        G.out_tile = rn.out_tile;
    }

    // 5. device tables
    p->table_off = kAlign;
    const uint64_t perm_bytes = p->perm_table.size() * sizeof(PermDesc);
    const uint64_t ep_start = align_up(perm_bytes);
    std::vector<EpTable> eps;
    for (auto &nd : p->nodes) {
        nd.ep_off = -1;
        if (nd.cls != TN_NODE_DENSE || nd.ksplit > 1) continue;
        // the table follows the kernel's view (rows and columns swapped with
        // the operands)
        NodePlan view = nd;
        if (nd.swap) {
            std::swap(view.m, view.n);
            std::swap(view.lm, view.ln);
        }
        EpTable t;
        if (!make_ep_table(view, &t)) continue;
        nd.ep_off = (int64_t)(p->table_off + ep_start + eps.size() * sizeof(EpTable));
        eps.push_back(t);
    }
    // tiny-node descriptors of each program's batches (the later slices'
    // batches hold fewer nodes: their own descriptors and CTA bases)
    std::vector<TinyDesc> tiny;
    auto describe = [&](std::vector<Launch> &sched, const std::vector<std::vector<int>> &batches) {
        size_t batch = 0;
        for (auto &L : sched) {
            if (L.kind == LAUNCH_NODE) {
                const NodePlan &nd = p->nodes[L.node];
                L.flops = 8 * nd.m * nd.n * nd.k;
            }
            if (L.kind != LAUNCH_TINY) continue;
            L.first = (int32_t)tiny.size();
            L.count = (int32_t)batches[batch].size();
            int ctas = 0;
            for (int s : batches[batch]) {
                const NodePlan &nd = p->nodes[s];
                TinyDesc d;
                std::memset(&d, 0, sizeof(d));
                d.a_off = (int64_t)nd.pa.off;
                d.b_off = (int64_t)nd.pb.off;
                d.c_off = nd.pc.kind == PLACE_OUT ? -1 : (int64_t)nd.pc.off;
                d.m = (int32_t)nd.m;
                d.n = (int32_t)nd.n;
                d.k = (int32_t)nd.k;
                d.out_fmt = nd.out_fmt;
                d.out_tile = nd.out_tile;
                d.is_root = nd.is_root ? 1 : 0;
                const uint64_t macs = nd.m * nd.n * nd.k;
                // `lanes` threads per output (a lane covers up to 16 entries
                // of k per round of loads); enough CTAs that each group of a
                // CTA computes one output (the rounds are serial memory
                // waits: one output per group measured faster than two)
                d.lanes = 1;
                while (d.lanes < 32 && (uint64_t)d.lanes * 16 < nd.k) d.lanes *= 2;
                const uint64_t per_cta = 256 / (uint64_t)d.lanes;
                d.ctas = (int32_t)std::max<uint64_t>(1, (nd.m * nd.n + per_cta - 1) / per_cta);
                d.cta_base = ctas;
                if (!make_walk(nd, &d)) return false;   // outputs are dense: not reached
                ctas += d.ctas;
                L.flops += 8 * macs;
                L.bytes += 8 * (nd.m * nd.k + nd.n * nd.k + nd.m * nd.n);
                tiny.push_back(d);
            }
            L.ctas = ctas;
            ++batch;
        }
        return true;
    };
    if (!describe(p->sched, tiny_batches) || !describe(p->sched_rest, tiny_batches_rest))
        return TN_ENOTIMPL;
    const uint64_t tiny_start = align_up(ep_start + eps.size() * sizeof(EpTable));
    p->tiny_off = p->table_off + tiny_start;
    // fused groups: FuseGroup[], FuseNode[], FuseGather[], level starts,
    // output offsets
    const uint64_t fg_start = align_up(tiny_start + tiny.size() * sizeof(TinyDesc));
    const uint64_t fn_start = align_up(fg_start + p->fuse_groups.size() * sizeof(FuseGroup));
    const uint64_t fl_start = align_up(fn_start + fnodes.size() * sizeof(FuseNode));
    const uint64_t fv_start = align_up(fl_start + fgather.size() * sizeof(FuseGather));
    const uint64_t fo_start = align_up(fv_start + flevels.size() * sizeof(int32_t));
    const uint64_t fc_start = align_up(fo_start + foffs.size() * sizeof(int32_t));
    p->fuse_chunk_off = p->table_off + fc_start;
    p->fuse_off = p->table_off + fg_start;
    p->fuse_node_off = p->table_off + fn_start;
    p->fuse_gather_off = p->table_off + fl_start;
    p->fuse_lvl_off = p->table_off + fv_start;
    p->fuse_offs_off = p->table_off + fo_start;
    // tail-tile counters (zero; every run leaves them zero again)
    const uint64_t cnt_start = align_up(fc_start + fchunks.size() * sizeof(int32_t));
    uint64_t cnt = 0;
    for (auto &nd : p->nodes) {
        nd.tail_cnt_off = -1;
        nd.red_cnt_off = -1;
        if (nd.tail_first >= 0) {
            nd.tail_cnt_off = (int64_t)(p->table_off + cnt_start + 4 * cnt);
            cnt += (dense_tiles(nd) - (uint64_t)nd.tail_first) * kDrainWarps;
        }
        if (nd.cls == TN_NODE_STREAM && nd.ksplit > 1) {
            nd.red_cnt_off = (int64_t)(p->table_off + cnt_start + 4 * cnt);
            cnt += (uint64_t)nd.red_ctas;
        }
    }
    p->table_blob.assign(cnt_start + 4 * cnt, 0);
    if (perm_bytes) std::memcpy(p->table_blob.data(), p->perm_table.data(), perm_bytes);
    if (!eps.empty())
        std::memcpy(p->table_blob.data() + ep_start, eps.data(), eps.size() * sizeof(EpTable));
    if (!tiny.empty())
        std::memcpy(p->table_blob.data() + tiny_start, tiny.data(), tiny.size() * sizeof(TinyDesc));
    if (!p->fuse_groups.empty()) {
        std::memcpy(p->table_blob.data() + fg_start, p->fuse_groups.data(),
                    p->fuse_groups.size() * sizeof(FuseGroup));
        std::memcpy(p->table_blob.data() + fn_start, fnodes.data(), fnodes.size() * sizeof(FuseNode));
        std::memcpy(p->table_blob.data() + fl_start, fgather.data(), fgather.size() * sizeof(FuseGather));
        std::memcpy(p->table_blob.data() + fv_start, flevels.data(), flevels.size() * sizeof(int32_t));
        std::memcpy(p->table_blob.data() + fo_start, foffs.data(), foffs.size() * sizeof(int32_t));
        std::memcpy(p->table_blob.data() + fc_start, fchunks.data(), fchunks.size() * sizeof(int32_t));
    }
    p->fuse_leaves_host = fleaves;
    p->table_bytes = align_up(p->table_blob.size());
    p->arena_off = p->table_off + p->table_bytes;
    p->ws_bytes = p->arena_off + p->arena_bytes;
    p->launches_per_exec = launches_of(*p, true) +
                           (p->n_slices - 1) * launches_of(*p, !(p->hoist && p->n_slices > 1));
    p->dense_maps.clear();
    p->maps_ws = nullptr;
    p->ws = nullptr;
    p->ws_size = 0;
    return TN_OK;
}

}  // namespace tn
