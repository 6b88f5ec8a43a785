// Executor: node classification and the stream-ordered launch sequence.
//
// For every slice (section 1.1 of "Crossing the single-GPU memory wall":
// the sliced sub-contractions are independent and their results add up) the
// executor permutes the leaves that need it, then runs the tree's steps in
// order, each on the kernel its class selects; the root step writes the
// caller's output on the first slice and adds into it on later ones.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <string>

#include "kernels.h"
#include "plan.h"

namespace tn {

int classify(const Plan &p, const NodePlan &nd) {
    (void)nd;
    if (p.policy == TN_POLICY_SIMT || p.precision == TN_PREC_FP32) return TN_NODE_SIMT;
    return TN_NODE_SIMT;
}

uint64_t launches_per_slice(const Plan &p) {
    const uint64_t perm = (p.perm_table.size() + kPermBatch - 1) / kPermBatch;
    return perm + p.nodes.size();
}

void release_events(Plan *p) {
    for (void *e : p->events)
        if (e) cudaEventDestroy(static_cast<cudaEvent_t>(e));
    p->events.clear();
}

namespace {

// Brackets launches with CUDA events when the plan is being profiled.
struct Recorder {
    Plan *p;
    cudaStream_t s;
    size_t i = 0;
    bool ok = true;
    void begin(int32_t kernel, int32_t step, uint64_t flops, uint64_t bytes) {
        if (!p->profiling || !ok) return;
        while (p->events.size() < 2 * (i + 1)) {
            cudaEvent_t e;
            if (cudaEventCreate(&e) != cudaSuccess) {
                ok = false;
                return;
            }
            p->events.push_back(e);
        }
        cudaEventRecord(static_cast<cudaEvent_t>(p->events[2 * i]), s);
        p->records.push_back(tn_launch_record{kernel, step, 0.f, flops, bytes});
    }
    void end() {
        if (!p->profiling || !ok) return;
        cudaEventRecord(static_cast<cudaEvent_t>(p->events[2 * i + 1]), s);
        ++i;
    }
};

uint64_t node_bytes(const NodePlan &nd, bool accumulate) {
    return 8 * (nd.m * nd.k + nd.n * nd.k + nd.m * nd.n * (accumulate ? 2 : 1));
}

tn_status cuda_fail(Plan *p, cudaError_t e, const char *what) {
    p->last_error = std::string(what) + ": " + cudaGetErrorString(e);
    return TN_ECUDA;
}

}  // namespace

tn_status upload_tables(Plan *p) {
    cudaError_t e = cudaMemset(p->ws, 0, p->table_off);
    if (e != cudaSuccess) return cuda_fail(p, e, "clearing the status word");
    if (!p->perm_table.empty()) {
        e = cudaMemcpy(static_cast<char *>(p->ws) + p->table_off, p->perm_table.data(),
                       p->perm_table.size() * sizeof(PermDesc), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(p, e, "uploading the permutation table");
    }
    return TN_OK;
}

tn_status execute_plan(Plan *p, const void *const *leaf_ptrs, void *out_ptr,
                       cudaStream_t stream) {
    char *ws = static_cast<char *>(p->ws);
    char *arena = ws + p->arena_off;
    DevStatus *status = reinterpret_cast<DevStatus *>(ws);
    const PermDesc *table = reinterpret_cast<const PermDesc *>(ws + p->table_off);
    float2 *out = static_cast<float2 *>(out_ptr);
    const int n = p->n_tensors;
    const int nsl = (int)p->slice_modes.size();
    std::vector<int64_t> digit(nsl, 0);
    std::vector<const float2 *> leaf_src(n);
    PermLaunch *pl = new PermLaunch;
    tn_status st = TN_OK;
    Recorder rec{p, stream};
    p->records.clear();

    for (uint64_t sigma = 0; sigma < p->n_slices && st == TN_OK; ++sigma) {
        // slice digits, first slice mode most significant
        uint64_t rem = sigma;
        for (int i = nsl - 1; i >= 0; --i) {
            digit[i] = (int64_t)(rem % (uint64_t)p->slice_ext[i]);
            rem /= (uint64_t)p->slice_ext[i];
        }
        for (int t = 0; t < n; ++t) {
            int64_t off = 0;
            for (const auto &term : p->leaves[t].slice_terms) off += digit[term.first] * term.second;
            leaf_src[t] = static_cast<const float2 *>(leaf_ptrs[t]) + off;
        }
        // leaf permutations, batched
        const int njobs = (int)p->perm_table.size();
        for (int j0 = 0; j0 < njobs; j0 += kPermBatch) {
            const int cnt = std::min(kPermBatch, njobs - j0);
            pl->njobs = cnt;
            pl->accumulate = 0;
            pl->table = table;
            pl->arena = arena;
            pl->out = out;
            int ctas = 0;
            for (int j = 0; j < cnt; ++j) {
                pl->job[j] = j0 + j;
                pl->cta_start[j] = ctas;
                pl->src[j] = leaf_src[p->perm_leaves[j0 + j]];
                ctas += permute_ctas(p->perm_table[j0 + j].size);
            }
            pl->cta_start[cnt] = ctas;
            uint64_t bytes = 0;
            for (int j = 0; j < cnt; ++j) bytes += 16 * (uint64_t)p->perm_table[j0 + j].size;
            rec.begin(TN_KERNEL_PERMUTE, -1, 0, bytes);
            cudaError_t e = launch_permute(*pl, ctas, stream);
            rec.end();
            if (e != cudaSuccess) {
                st = cuda_fail(p, e, "launching the leaf permutation");
                break;
            }
        }
        if (st != TN_OK) break;
        for (const NodePlan &nd : p->nodes) {
            auto resolve = [&](const Place &pl_) -> float2 * {
                switch (pl_.kind) {
                    case PLACE_WS: return reinterpret_cast<float2 *>(arena + pl_.off);
                    case PLACE_LEAF: return const_cast<float2 *>(leaf_src[pl_.leaf]);
                    default: return out;
                }
            };
            NodeArgs a;
            std::memset(&a, 0, sizeof(a));
            a.A = resolve(nd.pa);
            a.B = resolve(nd.pb);
            a.C = resolve(nd.pc);
            a.m = (int64_t)nd.m;
            a.n = (int64_t)nd.n;
            a.k = (int64_t)nd.k;
            a.lm = nd.lm;
            a.ln = nd.ln;
            a.accumulate = (nd.is_root && sigma > 0) ? 1 : 0;
            a.precision = p->precision;
            a.status = status;
            rec.begin(TN_KERNEL_SIMT, nd.step, 8 * nd.m * nd.n * nd.k, node_bytes(nd, a.accumulate));
            cudaError_t e = launch_simt_node(a, stream);
            rec.end();
            if (e != cudaSuccess) {
                st = cuda_fail(p, e, "launching a node kernel");
                break;
            }
        }
    }
    delete pl;
    return st;
}

tn_status read_profile(Plan *p, tn_launch_record *buf, int32_t cap, int32_t *len) {
    const size_t n = p->records.size();
    for (size_t i = 0; i < n; ++i) {
        float ms = 0.f;
        cudaError_t e = cudaEventElapsedTime(&ms, static_cast<cudaEvent_t>(p->events[2 * i]),
                                             static_cast<cudaEvent_t>(p->events[2 * i + 1]));
        if (e != cudaSuccess) return cuda_fail(p, e, "reading launch events");
        p->records[i].ms = ms;
    }
    *len = (int32_t)n;
    for (size_t i = 0; i < n && (int32_t)i < cap; ++i) buf[i] = p->records[i];
    return TN_OK;
}

tn_status check_plan(Plan *p) {
    DevStatus h{0, 0};
    cudaError_t e = cudaMemcpy(&h, p->ws, sizeof(h), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(p, e, "reading the status word");
    if (h.code != ERR_NONE) {
        e = cudaMemset(p->ws, 0, sizeof(h));
        if (e != cudaSuccess) return cuda_fail(p, e, "clearing the status word");
        p->last_error = "device status " + std::to_string(h.code) + " at " + std::to_string(h.where);
        return h.code == ERR_TIMEOUT ? TN_ETIMEOUT : TN_EDEVICE;
    }
    return TN_OK;
}

}  // namespace tn
