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

// Node classes.  A node goes to the tensor cores when its operands can be
// TMA-tiled (k entries per row a multiple of 16 bytes in the planar
// format), its tiles are reasonably full (m, n >= 64, k >= 16), and its
// arithmetic intensity with planar operand bytes (16 per tf32x3 entry,
// 4 per bf16 entry, 8 per output entry) is high enough to be
// compute-bound rather than bandwidth-bound.
int classify(const Plan &p, const NodePlan &nd) {
    if (p.policy == TN_POLICY_SIMT || p.precision == TN_PREC_FP32) return TN_NODE_SIMT;
    const bool bf16 = p.precision == TN_PREC_BF16;
    const uint64_t kq = bf16 ? 8 : 4;
    if (p.policy == TN_POLICY_DENSE) return nd.k % kq == 0 ? TN_NODE_DENSE : TN_NODE_SIMT;
    if (nd.k % kq == 0 && nd.k >= 16 && nd.m >= 64 && nd.n >= 64) {
        const double in_b = bf16 ? 4.0 : 16.0;
        const double m = (double)nd.m, n = (double)nd.n, k = (double)nd.k;
        const double intensity = 8.0 * m * n * k / (in_b * (m * k + n * k) + 8.0 * m * n);
        if (intensity >= 24.0) return TN_NODE_DENSE;
    }
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

// TMA maps of every tensor-core node's planar operands inside the current
// workspace (host-side encoding only; rebuilt when the workspace moves).
tn_status build_dense_maps(Plan *p) {
    p->dense_maps.clear();
    char *arena = static_cast<char *>(p->ws) + p->arena_off;
    const bool bf16 = p->precision == TN_PREC_BF16;
    for (size_t s = 0; s < p->nodes.size(); ++s) {
        const NodePlan &nd = p->nodes[s];
        if (nd.cls != TN_NODE_DENSE) continue;
        if (nd.pa.kind != PLACE_WS || nd.pb.kind != PLACE_WS) {
            p->last_error = "tensor-core operand not in the workspace";
            return TN_EDEVICE;
        }
        DenseMaps dm;
        std::memset(&dm, 0, sizeof(dm));
        dm.node = (int32_t)s;
        std::string err;
        if (!encode_operand_map(&dm.a, arena + nd.pa.off, (int64_t)nd.m, (int64_t)nd.k, bf16, &err) ||
            !encode_operand_map(&dm.b, arena + nd.pb.off, (int64_t)nd.n, (int64_t)nd.k, bf16, &err)) {
            p->last_error = "step " + std::to_string(s) + ": " + err;
            return TN_ECUDA;
        }
        p->dense_maps.push_back(dm);
    }
    p->maps_ws = p->ws;
    return TN_OK;
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
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(p, e, "querying the SM count");
    return build_dense_maps(p);
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
    tn_status st = TN_OK;
    if (p->maps_ws != p->ws) {
        st = build_dense_maps(p);
        if (st != TN_OK) return st;
    }
    if (p->num_sms <= 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(p, e, "querying the SM count");
    }
    std::vector<int32_t> map_of(p->nodes.size(), -1);
    for (size_t i = 0; i < p->dense_maps.size(); ++i) map_of[p->dense_maps[i].node] = (int32_t)i;
    PermLaunch *pl = new PermLaunch;
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
            const int32_t accumulate = (nd.is_root && sigma > 0) ? 1 : 0;
            const uint64_t flops = 8 * nd.m * nd.n * nd.k;
            cudaError_t e;
            if (nd.cls == TN_NODE_DENSE) {
                alignas(128) DenseArgs dargs;
                std::memset(&dargs, 0, sizeof(dargs));
                DenseArgs *d = &dargs;
                const DenseMaps &dm = p->dense_maps[map_of[nd.step]];
                std::memcpy(&d->tmA, &dm.a, sizeof(CUtensorMap));
                std::memcpy(&d->tmB, &dm.b, sizeof(CUtensorMap));
                d->C = resolve(nd.pc);
                d->m = (int64_t)nd.m;
                d->n = (int64_t)nd.n;
                d->k = (int64_t)nd.k;
                d->lm = nd.lm;
                d->ln = nd.ln;
                d->accumulate = accumulate;
                d->out_fmt = nd.out_fmt;
                d->bf16 = p->precision == TN_PREC_BF16;
                d->status = status;
                const uint64_t in_b = d->bf16 ? 4 : 16;
                rec.begin(d->bf16 ? TN_KERNEL_DENSE_BF16 : TN_KERNEL_DENSE_TF32X3, nd.step, flops,
                          in_b * (nd.m * nd.k + nd.n * nd.k) +
                              fmt_bytes(nd.out_fmt) * nd.m * nd.n * (accumulate ? 2 : 1));
                e = launch_dense(*d, p->num_sms, stream);
                rec.end();
            } else {
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
                a.accumulate = accumulate;
                a.out_fmt = nd.out_fmt;
                a.status = status;
                rec.begin(TN_KERNEL_SIMT, nd.step, flops, node_bytes(nd, accumulate));
                e = launch_simt_node(a, stream);
                rec.end();
            }
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
