// C ABI of the executor (declared in include/tn.h).  Argument checks and
// plumbing only: planning is in plan.cpp, launching in exec.cu.
#include <cuda_runtime.h>

#include <new>
#include <string>

#include "../../include/tn.h"
#include "plan.h"

namespace tn {
tn_status upload_tables(Plan *p);
tn_status execute_plan(Plan *p, const void *const *leaf_ptrs, void *out_ptr, cudaStream_t stream);
tn_status check_plan(Plan *p);
tn_status execute_replayed(Plan *p, const void *const *leaf_ptrs, void *out_ptr,
                           cudaStream_t stream);
tn_status execute_range(Plan *p, const void *const *leaf_ptrs, void *out_ptr, cudaStream_t stream,
                        uint64_t first, uint64_t step);
tn_status read_profile(Plan *p, tn_launch_record *buf, int32_t cap, int32_t *len);
tn_status check_static(Plan *p);
tn_status execute_prefix(Plan *p, const void *const *leaf_ptrs, void *out_ptr, int32_t step,
                         cudaStream_t stream);
tn_status tensor_gather(Plan *p, int32_t id, const int64_t *idx, uint64_t count, void *dst,
                        cudaStream_t stream);
tn_status execute_host(Plan *p, const void *const *host_leaves, void *host_out,
                       void *const *dev_leaves, void *dev_out, cudaStream_t stream);
}  // namespace tn

namespace {
thread_local std::string g_plan_error;
}

extern "C" {

tn_status tn_plan(const tn_network *network, const tn_tree *tree, const tn_slices *slices,
                  tn_plan_t **out) {
    if (!out) {
        g_plan_error = "out is NULL";
        return TN_EINVAL;
    }
    *out = nullptr;
    tn_plan_s *h = new (std::nothrow) tn_plan_s;
    if (!h) {
        g_plan_error = "host allocation failed";
        return TN_ENOMEM;
    }
    std::string err;
    tn_status st = tn::build_plan(network, tree, slices, &h->p, &err);
    if (st == TN_OK) st = tn::layout_plan(&h->p);
    if (st != TN_OK) {
        g_plan_error = err.empty() ? h->p.last_error : err;
        delete h;
        return st;
    }
    g_plan_error.clear();
    *out = h;
    return TN_OK;
}

void tn_plan_destroy(tn_plan_t *plan) { delete plan; }

tn_status tn_plan_flops(const tn_plan_t *plan, uint64_t *ct) {
    if (!plan || !ct) return TN_EINVAL;
    *ct = plan->p.ct_total;
    return TN_OK;
}

tn_status tn_plan_peak(const tn_plan_t *plan, uint64_t *cs) {
    if (!plan || !cs) return TN_EINVAL;
    *cs = plan->p.cs;
    return TN_OK;
}

tn_status tn_plan_num_slices(const tn_plan_t *plan, uint64_t *n) {
    if (!plan || !n) return TN_EINVAL;
    *n = plan->p.n_slices;
    return TN_OK;
}

tn_status tn_plan_num_steps(const tn_plan_t *plan, int32_t *n) {
    if (!plan || !n) return TN_EINVAL;
    *n = (int32_t)plan->p.nodes.size();
    return TN_OK;
}

tn_status tn_plan_mode_order(const tn_plan_t *plan, int32_t id, int32_t *buf, int32_t cap,
                             int32_t *len) {
    if (!plan || !len || cap < 0 || (cap > 0 && !buf)) return TN_EINVAL;
    if (id < 0 || id >= (int32_t)plan->p.orders.size()) return TN_EINVAL;
    const auto &o = plan->p.orders[id];
    *len = (int32_t)o.size();
    for (int32_t i = 0; i < cap && i < (int32_t)o.size(); ++i) buf[i] = o[i];
    return TN_OK;
}

tn_status tn_plan_node_mnk(const tn_plan_t *plan, int32_t step, uint64_t mnk[3]) {
    if (!plan || !mnk || step < 0 || step >= (int32_t)plan->p.nodes.size()) return TN_EINVAL;
    const auto &nd = plan->p.nodes[step];
    mnk[0] = nd.m;
    mnk[1] = nd.n;
    mnk[2] = nd.k;
    return TN_OK;
}

tn_status tn_plan_node_class(const tn_plan_t *plan, int32_t step, int32_t *cls) {
    if (!plan || !cls || step < 0 || step >= (int32_t)plan->p.nodes.size()) return TN_EINVAL;
    const tn::Plan &p = plan->p;
    *cls = (step < (int32_t)p.fused.size() && p.fused[step] >= 0) ? TN_NODE_FUSED : p.nodes[step].cls;
    return TN_OK;
}

tn_status tn_plan_set_promotion_chunk(tn_plan_t *plan, int32_t chunk_k) {
    if (!plan) return TN_EINVAL;
    if (chunk_k != 0 && (chunk_k < 32 || chunk_k > 4096 || chunk_k % 32 != 0)) {
        plan->p.last_error = "promotion chunk must be 0 or a multiple of 32 in [32, 4096]";
        return TN_EINVAL;
    }
    plan->p.chunk_k = chunk_k;
    return tn::layout_plan(&plan->p);
}

tn_status tn_plan_set_cta_pairs(tn_plan_t *plan, int32_t enable) {
    if (!plan) return TN_EINVAL;
    plan->p.cta_pairs = enable ? 1 : 0;
    return tn::layout_plan(&plan->p);
}

tn_status tn_plan_set_fusion(tn_plan_t *plan, int32_t enable) {
    if (!plan) return TN_EINVAL;
    plan->p.fuse = enable ? 1 : 0;
    return tn::layout_plan(&plan->p);
}

tn_status tn_plan_set_policy(tn_plan_t *plan, int32_t policy) {
    // tn::kPolicyForceDense is a test setting outside the ABI (see plan.h)
    if (!plan || policy < TN_POLICY_AUTO || policy > tn::kPolicyForceDense) return TN_EINVAL;
    plan->p.policy = policy;
    return tn::layout_plan(&plan->p);
}

tn_status tn_execute_host(tn_plan_t *plan, const void *const *host_leaves, void *host_out,
                          void *const *dev_leaves, void *dev_out, tn_stream_t stream) {
    if (!plan) return TN_EINVAL;
    tn::Plan &p = plan->p;
    if (!host_leaves || !host_out || !dev_leaves || !dev_out) {
        p.last_error = "host_leaves, host_out, dev_leaves and dev_out are required";
        return TN_EINVAL;
    }
    for (int t = 0; t < p.n_tensors; ++t)
        if (!host_leaves[t] || !dev_leaves[t]) {
            p.last_error = "leaf pointer " + std::to_string(t) + " is NULL";
            return TN_EINVAL;
        }
    if (!p.ws) {
        p.last_error = "no workspace bound (tn_plan_set_workspace)";
        return TN_ENOMEM;
    }
    p.last_static = false;
    return tn::execute_host(&p, host_leaves, host_out, dev_leaves, dev_out,
                            reinterpret_cast<cudaStream_t>(stream));
}

tn_status tn_plan_set_three_products(tn_plan_t *plan, int32_t enable) {
    if (!plan) return TN_EINVAL;
    plan->p.three_products = enable ? 1 : 0;
    return tn::layout_plan(&plan->p);
}

tn_status tn_plan_set_hoisting(tn_plan_t *plan, int32_t enable) {
    if (!plan) return TN_EINVAL;
    plan->p.hoist = enable ? 1 : 0;
    return tn::layout_plan(&plan->p);
}

tn_status tn_plan_workspace_bytes(const tn_plan_t *plan, uint64_t *bytes) {
    if (!plan || !bytes) return TN_EINVAL;
    *bytes = plan->p.ws_bytes;
    return TN_OK;
}

tn_status tn_plan_set_workspace(tn_plan_t *plan, void *dev_ptr, uint64_t bytes) {
    if (!plan) return TN_EINVAL;
    tn::Plan &p = plan->p;
    if (!dev_ptr || (reinterpret_cast<uintptr_t>(dev_ptr) % tn::kAlign) != 0) {
        p.last_error = "workspace must be a non-NULL 256-byte aligned device pointer";
        return TN_EINVAL;
    }
    if (bytes < p.ws_bytes) {
        p.last_error = "workspace of " + std::to_string(bytes) + " bytes is smaller than the " +
                       std::to_string(p.ws_bytes) + " bytes the plan needs";
        return TN_ENOMEM;
    }
    p.ws = dev_ptr;
    p.ws_size = bytes;
    tn_status st = tn::upload_tables(&p);
    if (st != TN_OK) {
        p.ws = nullptr;
        p.ws_size = 0;
    }
    return st;
}

tn_status tn_execute(tn_plan_t *plan, const void *const *leaf_ptrs, void *out_ptr,
                     tn_stream_t stream) {
    if (!plan) return TN_EINVAL;
    tn::Plan &p = plan->p;
    if (!leaf_ptrs || !out_ptr) {
        p.last_error = "leaf_ptrs and out_ptr are required";
        return TN_EINVAL;
    }
    for (int t = 0; t < p.n_tensors; ++t)
        if (!leaf_ptrs[t]) {
            p.last_error = "leaf pointer " + std::to_string(t) + " is NULL";
            return TN_EINVAL;
        }
    if (!p.ws) {
        p.last_error = "no workspace bound (tn_plan_set_workspace)";
        return TN_ENOMEM;
    }
    p.last_static = false;
    return tn::execute_replayed(&p, leaf_ptrs, out_ptr, reinterpret_cast<cudaStream_t>(stream));
}

tn_status tn_plan_check(tn_plan_t *plan) {
    if (!plan) return TN_EINVAL;
    if (plan->p.last_static) return tn::check_static(&plan->p);
    if (!plan->p.ws) return TN_OK;
    return tn::check_plan(&plan->p);
}

tn_status tn_execute_slices(tn_plan_t *plan, const void *const *leaf_ptrs, void *out_ptr,
                            tn_stream_t stream, uint64_t first, uint64_t step) {
    if (!plan) return TN_EINVAL;
    tn::Plan &p = plan->p;
    if (!leaf_ptrs || !out_ptr || step < 1) {
        p.last_error = "leaf_ptrs and out_ptr are required and step must be >= 1";
        return TN_EINVAL;
    }
    for (int t = 0; t < p.n_tensors; ++t)
        if (!leaf_ptrs[t]) {
            p.last_error = "leaf pointer " + std::to_string(t) + " is NULL";
            return TN_EINVAL;
        }
    if (!p.ws) {
        p.last_error = "no workspace bound (tn_plan_set_workspace)";
        return TN_ENOMEM;
    }
    p.last_static = false;
    return tn::execute_range(&p, leaf_ptrs, out_ptr, reinterpret_cast<cudaStream_t>(stream), first,
                             step);
}

tn_status tn_execute_prefix(tn_plan_t *plan, const void *const *leaf_ptrs, void *out_ptr,
                            int32_t step, tn_stream_t stream) {
    if (!plan) return TN_EINVAL;
    tn::Plan &p = plan->p;
    if (!leaf_ptrs || !out_ptr) {
        p.last_error = "leaf_ptrs and out_ptr are required";
        return TN_EINVAL;
    }
    for (int t = 0; t < p.n_tensors; ++t)
        if (!leaf_ptrs[t]) {
            p.last_error = "leaf pointer " + std::to_string(t) + " is NULL";
            return TN_EINVAL;
        }
    if (step < 0 || step >= (int32_t)p.nodes.size()) {
        p.last_error = "step out of range";
        return TN_EINVAL;
    }
    if (!p.ws) {
        p.last_error = "no workspace bound (tn_plan_set_workspace)";
        return TN_ENOMEM;
    }
    p.last_static = false;
    return tn::execute_prefix(&p, leaf_ptrs, out_ptr, step, reinterpret_cast<cudaStream_t>(stream));
}

tn_status tn_plan_tensor_gather(tn_plan_t *plan, int32_t id, const int64_t *idx, uint64_t count,
                                void *dst, tn_stream_t stream) {
    if (!plan) return TN_EINVAL;
    tn::Plan &p = plan->p;
    if ((count > 0 && (!idx || !dst)) || id < 0 || id >= (int32_t)p.orders.size()) {
        p.last_error = "bad tensor id or NULL index / destination";
        return TN_EINVAL;
    }
    return tn::tensor_gather(&p, id, idx, count, dst, reinterpret_cast<cudaStream_t>(stream));
}

tn_status tn_plan_set_replay(tn_plan_t *plan, int32_t enable) {
    if (!plan) return TN_EINVAL;
    tn::drop_graph(&plan->p);
    plan->p.use_graph = enable != 0;
    return TN_OK;
}

tn_status tn_plan_launches(const tn_plan_t *plan, uint64_t *n) {
    if (!plan || !n) return TN_EINVAL;
    *n = plan->p.launches_per_exec;
    return TN_OK;
}

tn_status tn_plan_set_profiling(tn_plan_t *plan, int32_t enable) {
    if (!plan) return TN_EINVAL;
    plan->p.profiling = enable != 0;
    plan->p.records.clear();
    return TN_OK;
}

tn_status tn_plan_profile_read(tn_plan_t *plan, tn_launch_record *buf, int32_t cap,
                               int32_t *len) {
    if (!plan || !len || cap < 0 || (cap > 0 && !buf)) return TN_EINVAL;
    return tn::read_profile(&plan->p, buf, cap, len);
}

const char *tn_status_string(tn_status status) {
    switch (status) {
        case TN_OK: return "ok";
        case TN_EINVAL: return "invalid argument";
        case TN_ENOMEM: return "workspace missing or too small";
        case TN_EOVERFLOW: return "size or FLOP count overflows 64 bits";
        case TN_ECUDA: return "CUDA runtime error";
        case TN_EDEVICE: return "device-side inconsistency";
        case TN_ETIMEOUT: return "device-side wait timed out";
        case TN_ENOTIMPL: return "not supported by this build";
    }
    return "unknown status";
}

const char *tn_last_error(const tn_plan_t *plan) {
    if (!plan) return g_plan_error.c_str();
    return plan->p.last_error.c_str();
}

}  // extern "C"
