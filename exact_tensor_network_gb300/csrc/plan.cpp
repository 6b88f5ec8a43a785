// Host planner: validation, lifetime ordering, node descriptors, slicing,
// node classes and workspace layout.  No device work happens here.
//
// Lifetime ordering follows "Crossing the single-GPU memory wall"
// (digest of arXiv 2606.01852), section 1.4: the root keeps the caller's
// open-mode order; walking the steps from last to first, each operand is
// stored as [the output's modes it owns, in the output's order || the summed
// modes K].  The page leaves the order inside K open; it is ascending mode
// id here, the same list for both operands, which is what makes A a
// row-major [m, k] matrix and B a row-major [n, k] matrix with the same k
// index.  Section 1.1 gives the step shape (m, n, k are products of the
// extents of M, N and K) and slicing (fixing modes splits the sum).
#include "plan.h"

#include <algorithm>
#include <cstring>

namespace tn {

namespace {

bool mul_ovf(uint64_t a, uint64_t b, uint64_t *r) { return __builtin_mul_overflow(a, b, r); }
bool add_ovf(uint64_t a, uint64_t b, uint64_t *r) { return __builtin_add_overflow(a, b, r); }

bool contains(const std::vector<int32_t> &v, int32_t x) {
    return std::find(v.begin(), v.end(), x) != v.end();
}

// Runs of `side` modes inside the output order `oc`, with row-major strides
// of `oc`.  Modes of extent 1 are skipped.
bool make_runs(const std::vector<int32_t> &oc, const std::vector<int32_t> &side,
               const std::vector<int64_t> &ext, SepLayout *lay) {
    std::memset(lay, 0, sizeof(*lay));
    const int r = (int)oc.size();
    std::vector<int64_t> stride(r);
    int64_t s = 1;
    for (int i = r - 1; i >= 0; --i) {
        stride[i] = s;
        s *= ext[oc[i]];
    }
    int nrun = 0;
    bool open_run = false;
    for (int i = 0; i < r; ++i) {
        const int32_t x = oc[i];
        const bool in_side = contains(side, x);
        if (!in_side || ext[x] == 1) {
            if (!in_side) open_run = false;
            continue;
        }
        if (open_run) {
            lay->ext[nrun - 1] *= ext[x];
            lay->stride[nrun - 1] = stride[i];
        } else {
            if (nrun == kMaxRuns) return false;
            lay->ext[nrun] = ext[x];
            lay->stride[nrun] = stride[i];
            ++nrun;
            open_run = true;
        }
    }
    lay->nrun = nrun;
    for (int i = 0; i < kMaxRuns; ++i) lay->shift[i] = i < nrun ? log2_exact(lay->ext[i]) : -1;
    return true;
}

}  // namespace

tn_status build_plan(const tn_network *net, const tn_tree *tree, const tn_slices *sl,
                     Plan *p, std::string *err) {
    auto fail = [&](tn_status st, const std::string &msg) {
        *err = msg;
        return st;
    };
    if (!net || !tree) return fail(TN_EINVAL, "network and tree are required");
    const int32_t n = net->n_tensors;
    if (n < 1) return fail(TN_EINVAL, "n_tensors must be >= 1");
    if (net->n_modes < 0) return fail(TN_EINVAL, "n_modes must be >= 0");
    if (net->n_modes > 0 && !net->extents) return fail(TN_EINVAL, "extents is NULL");
    if (!net->ranks || !net->modes) return fail(TN_EINVAL, "ranks/modes is NULL");
    if (net->n_open < 0 || (net->n_open > 0 && !net->open_modes))
        return fail(TN_EINVAL, "bad open-mode list");
    if (net->precision < TN_PREC_TF32X3 || net->precision > TN_PREC_BF16X3)
        return fail(TN_EINVAL, "unknown precision");
    p->n_tensors = n;
    p->n_modes = net->n_modes;
    p->precision = net->precision;
    p->extents.assign(net->extents, net->extents + net->n_modes);
    for (int64_t e : p->extents)
        if (e < 1) return fail(TN_EINVAL, "extent must be >= 1");

    std::vector<int> count(p->n_modes, 0);
    p->leaf_modes.resize(n);
    for (int t = 0; t < n; ++t) {
        const int32_t r = net->ranks[t];
        if (r < 0) return fail(TN_EINVAL, "negative rank");
        if (r > kMaxRank) return fail(TN_ENOTIMPL, "tensor rank above 64");
        if (r > 0 && !net->modes[t]) return fail(TN_EINVAL, "modes[t] is NULL");
        p->leaf_modes[t].assign(net->modes[t], net->modes[t] + r);
        for (int i = 0; i < r; ++i) {
            const int32_t x = p->leaf_modes[t][i];
            if (x < 0 || x >= p->n_modes) return fail(TN_EINVAL, "mode id out of range");
            for (int j = 0; j < i; ++j)
                if (p->leaf_modes[t][j] == x)
                    return fail(TN_EINVAL, "mode repeated within one tensor (trace)");
            ++count[x];
        }
    }
    std::vector<char> is_open(p->n_modes, 0);
    p->open_modes.assign(net->open_modes, net->open_modes + net->n_open);
    for (int32_t x : p->open_modes) {
        if (x < 0 || x >= p->n_modes) return fail(TN_EINVAL, "open mode out of range");
        if (is_open[x]) return fail(TN_EINVAL, "open mode listed twice");
        is_open[x] = 1;
    }
    for (int x = 0; x < p->n_modes; ++x) {
        const int want = is_open[x] ? 1 : 2;
        if (count[x] != want)
            return fail(TN_EINVAL, "mode " + std::to_string(x) + " appears in " +
                                       std::to_string(count[x]) + " tensors, expected " +
                                       std::to_string(want));
    }

    const int32_t S = tree->n_steps;
    if (S != n - 1) return fail(TN_EINVAL, "tree must have n_tensors - 1 steps");
    if (S > 0 && !tree->pairs) return fail(TN_EINVAL, "pairs is NULL");
    const int total = n + S;
    p->pairs.assign(tree->pairs, tree->pairs + 2 * S);
    p->consumer.assign(total, -1);
    for (int s = 0; s < S; ++s) {
        const int32_t a = p->pairs[2 * s], b = p->pairs[2 * s + 1];
        if (a == b) return fail(TN_EINVAL, "step contracts a tensor with itself");
        for (int32_t id : {a, b}) {
            if (id < 0 || id >= n + s)
                return fail(TN_EINVAL, "tree id out of range or used before it exists");
            if (p->consumer[id] != -1) return fail(TN_EINVAL, "tree uses an id twice");
            p->consumer[id] = s;
        }
    }

    std::vector<char> is_sliced(p->n_modes, 0);
    if (sl && sl->n > 0) {
        if (!sl->modes) return fail(TN_EINVAL, "slice modes is NULL");
        for (int i = 0; i < sl->n; ++i) {
            const int32_t x = sl->modes[i];
            if (x < 0 || x >= p->n_modes) return fail(TN_EINVAL, "slice mode out of range");
            if (is_open[x]) return fail(TN_EINVAL, "only closed modes can be sliced");
            if (is_sliced[x]) return fail(TN_EINVAL, "slice mode listed twice");
            is_sliced[x] = 1;
            p->slice_modes.push_back(x);
            p->slice_ext.push_back(p->extents[x]);
        }
    }
    p->n_slices = 1;
    for (int64_t e : p->slice_ext)
        if (mul_ovf(p->n_slices, (uint64_t)e, &p->n_slices))
            return fail(TN_EOVERFLOW, "slice count overflows");

    // Mode sets of every SSA id on the sliced network: an output keeps the
    // operands' modes that the two do not share.
    std::vector<std::vector<int32_t>> ms(total);
    for (int t = 0; t < n; ++t)
        for (int32_t x : p->leaf_modes[t])
            if (!is_sliced[x]) ms[t].push_back(x);
    for (int s = 0; s < S; ++s) {
        const auto &A = ms[p->pairs[2 * s]], &B = ms[p->pairs[2 * s + 1]];
        auto &C = ms[n + s];
        for (int32_t x : A)
            if (!contains(B, x)) C.push_back(x);
        for (int32_t x : B)
            if (!contains(A, x)) C.push_back(x);
        if ((int)C.size() > kMaxRank) return fail(TN_ENOTIMPL, "intermediate rank above 64");
    }

    // Reverse walk (section 1.4).
    p->orders.assign(total, {});
    const int root = total - 1;
    p->orders[root] = p->open_modes;
    {
        std::vector<int32_t> a_sorted = ms[root], b_sorted = p->open_modes;
        std::sort(a_sorted.begin(), a_sorted.end());
        std::sort(b_sorted.begin(), b_sorted.end());
        if (a_sorted != b_sorted) return fail(TN_EINVAL, "root modes differ from the open modes");
    }
    for (int s = S - 1; s >= 0; --s) {
        const int32_t a = p->pairs[2 * s], b = p->pairs[2 * s + 1];
        const auto &oc = p->orders[n + s];
        std::vector<int32_t> K;
        for (int32_t x : ms[a])
            if (contains(ms[b], x)) K.push_back(x);
        std::sort(K.begin(), K.end());
        for (int32_t side : {a, b}) {
            auto &o = p->orders[side];
            o.clear();
            for (int32_t x : oc)
                if (contains(ms[side], x)) o.push_back(x);
            o.insert(o.end(), K.begin(), K.end());
        }
    }

    // Node descriptors.
    std::vector<int32_t> level(total, 0);
    p->nodes.resize(S);
    p->ct_slice = 0;
    p->cs = 0;
    for (int s = 0; s < S; ++s) {
        NodePlan &nd = p->nodes[s];
        std::memset(&nd, 0, sizeof(nd));
        nd.step = s;
        nd.a = p->pairs[2 * s];
        nd.b = p->pairs[2 * s + 1];
        nd.out = n + s;
        nd.is_root = (nd.out == root);
        const auto &oc = p->orders[nd.out];
        std::vector<int32_t> M, N;
        for (int32_t x : oc) (contains(ms[nd.a], x) ? M : N).push_back(x);
        uint64_t m = 1, nn = 1, k = 1;
        for (int32_t x : M)
            if (mul_ovf(m, (uint64_t)p->extents[x], &m)) return fail(TN_EOVERFLOW, "m overflows");
        for (int32_t x : N)
            if (mul_ovf(nn, (uint64_t)p->extents[x], &nn)) return fail(TN_EOVERFLOW, "n overflows");
        const auto &oa = p->orders[nd.a];
        for (size_t i = M.size(); i < oa.size(); ++i)
            if (mul_ovf(k, (uint64_t)p->extents[oa[i]], &k)) return fail(TN_EOVERFLOW, "k overflows");
        nd.m = m;
        nd.n = nn;
        nd.k = k;
        uint64_t f = 8, mn = 0;
        if (mul_ovf(f, m, &f) || mul_ovf(f, nn, &f) || mul_ovf(f, k, &f) ||
            add_ovf(p->ct_slice, f, &p->ct_slice) || mul_ovf(m, nn, &mn))
            return fail(TN_EOVERFLOW, "FLOP count overflows 64 bits");
        p->cs = std::max(p->cs, mn);
        if (!make_runs(oc, M, p->extents, &nd.lm) || !make_runs(oc, N, p->extents, &nd.ln))
            return fail(TN_ENOTIMPL, "output layout interleaves M and N more than 12 times");
        // layout class of C
        int first_n = -1, last_m = -1, first_m = -1, last_n = -1;
        for (int i = 0; i < (int)oc.size(); ++i) {
            if (contains(M, oc[i])) {
                if (first_m < 0) first_m = i;
                last_m = i;
            } else {
                if (first_n < 0) first_n = i;
                last_n = i;
            }
        }
        nd.layout = (first_n < 0 || last_m < first_n) ? 0 : (first_m < 0 || last_n < first_m) ? 1 : 2;
        level[nd.out] = 1 + std::max(level[nd.a], level[nd.b]);
        nd.level = level[nd.out];
    }
    if (S == 0) {
        uint64_t sz = 1;
        for (int32_t x : ms[0])
            if (mul_ovf(sz, (uint64_t)p->extents[x], &sz)) return fail(TN_EOVERFLOW, "size overflows");
        p->cs = sz;
    }
    if (mul_ovf(p->ct_slice, p->n_slices, &p->ct_total))
        return fail(TN_EOVERFLOW, "total FLOP count overflows 64 bits");
    p->out_elems = 1;
    for (int32_t x : p->open_modes)
        if (mul_ovf(p->out_elems, (uint64_t)p->extents[x], &p->out_elems))
            return fail(TN_EOVERFLOW, "output size overflows");

    // Leaves: user layout -> lifetime order.
    p->leaves.resize(n);
    for (int t = 0; t < n; ++t) {
        LeafPlan &lp = p->leaves[t];
        lp.leaf = t;
        std::memset(&lp.perm, 0, sizeof(lp.perm));
        const auto &um = p->leaf_modes[t];
        const int r = (int)um.size();
        std::vector<int64_t> ustride(r);
        int64_t s = 1;
        for (int i = r - 1; i >= 0; --i) {
            ustride[i] = s;
            s *= p->extents[um[i]];
        }
        lp.full_size = s;
        for (int i = 0; i < r; ++i)
            if (is_sliced[um[i]]) {
                const int pos = (int)(std::find(p->slice_modes.begin(), p->slice_modes.end(), um[i]) -
                                      p->slice_modes.begin());
                lp.slice_terms.push_back({pos, ustride[i]});
            }
        std::vector<int64_t> dims, sst;
        for (int32_t x : p->orders[t]) {
            if (p->extents[x] == 1) continue;
            const int i = (int)(std::find(um.begin(), um.end(), x) - um.begin());
            if (!dims.empty() && sst.back() == ustride[i] * p->extents[x]) {
                dims.back() *= p->extents[x];
                sst.back() = ustride[i];
            } else {
                dims.push_back(p->extents[x]);
                sst.push_back(ustride[i]);
            }
        }
        int64_t size = 1;
        for (int64_t d : dims) size *= d;
        lp.size = size;
        lp.identity = dims.empty() || (dims.size() == 1 && sst[0] == 1);
        lp.in_place = lp.identity;
        if ((int)dims.size() > kMaxPermRank)
            return fail(TN_ENOTIMPL, "leaf permutation needs more than 16 axes after merging");
        lp.perm.size = size;
        lp.perm.rank = (int32_t)dims.size();
        for (size_t i = 0; i < dims.size(); ++i) {
            lp.perm.dims[i] = dims[i];
            lp.perm.sstride[i] = sst[i];
            lp.perm.dshift[i] = log2_exact(dims[i]);
        }
    }
    return TN_OK;
}

}  // namespace tn
