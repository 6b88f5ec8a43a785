// tn_execute_static: tn_execute without any caller-provided workspace.
//
// Some callers cannot hand the library device memory: code that runs after
// its start-up phase under a rule of "no allocation from here on" (real-time
// loops, plugins inside a host runtime that owns every byte of device memory
// and forbids side allocations), or code that runs where calling the
// allocator is unsafe.  For them this file keeps one fixed scratch array in
// device global memory, sized at build time, and runs the ordinary executor
// with that array as its workspace.  Nothing here calls cudaMalloc,
// cudaFree or any allocating routine.
//
// Limits and behaviour a caller must know:
//   - The array holds kStaticScratchBytes (32 MiB).  A plan whose workspace
//     (tn_plan_workspace_bytes) is larger is rejected with TN_ENOMEM before
//     anything is enqueued.
//   - The array is a global of this library: every GPU that loads the
//     library keeps those 32 MiB reserved until the process exits.
//   - All calls share the one array, and it keeps whatever the last call
//     left in it.  Each call re-uploads its plan's descriptor table and
//     clears the device status word on the caller's stream before the
//     kernels run; everything else is written before it is read.  Two calls
//     whose GPU work overlaps (different streams, or different threads
//     without ordering) race on the array and give wrong results: order them
//     on one stream.
//   - The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it; make
//     that first call before any stream capture.
//   - The device status word of these calls lives at the start of the
//     array.  After a static call, tn_plan_check() on that plan reads it
//     there (and clears it), as it reads a bound workspace's otherwise.
//   - Launch timing (tn_plan_set_profiling) is suspended for these calls,
//     since it would create CUDA events.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/tn.h"
#include "kernels.h"
#include "plan.h"

namespace tn {
tn_status execute_plan(Plan *p, const void *const *leaf_ptrs, void *out_ptr, cudaStream_t stream);
}  // namespace tn

namespace {

constexpr unsigned long long kStaticScratchBytes = 32ull << 20;
constexpr int kMaxDevices = 64;

// Host code must not use this name as a device address: in host code it
// names a host-side stand-in.  The device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

tn_status scratch_address(tn::Plan &p, void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        p.last_error = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return TN_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        p.last_error = "device index above 63";
        return TN_ENOTIMPL;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_scratch);
        if (e != cudaSuccess || !ptr) {
            p.last_error = std::string("cudaGetSymbolAddress of the static scratch array: ") +
                           cudaGetErrorString(e);
            return TN_ECUDA;
        }
        g_addr[dev] = ptr;
    }
    *out = g_addr[dev];
    return TN_OK;
}

}  // namespace

namespace tn {

// tn_plan_check after a static call: the status word at offset 0 of the
// array on the current device (zero when no static call ran there yet).
tn_status check_static(Plan *p) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        p->last_error = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return TN_ECUDA;
    }
    void *addr = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (dev >= 0 && dev < kMaxDevices) addr = g_addr[dev];
    }
    if (!addr) return TN_OK;
    DevStatus h{0, 0};
    e = cudaMemcpy(&h, addr, sizeof(h), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
        p->last_error = std::string("reading the static status word: ") + cudaGetErrorString(e);
        return TN_ECUDA;
    }
    if (h.code == ERR_NONE) return TN_OK;
    // the next static call uploads the tables (tail-tile counters included)
    // again, so clearing the word is all that is left to do
    e = cudaMemset(addr, 0, sizeof(h));
    if (e != cudaSuccess) {
        p->last_error = std::string("clearing the static status word: ") + cudaGetErrorString(e);
        return TN_ECUDA;
    }
    p->last_error = "device status " + std::to_string(h.code) + " at " + std::to_string(h.where);
    return h.code == ERR_TIMEOUT ? TN_ETIMEOUT : TN_EDEVICE;
}

}  // namespace tn

extern "C" TN_API tn_status tn_execute_static(tn_plan_t *plan, const void *const *leaf_ptrs,
                                              void *out_ptr, tn_stream_t stream) {
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
    if (p.ws_bytes > kStaticScratchBytes) {
        p.last_error = "plan needs a workspace of " + std::to_string(p.ws_bytes) +
                       " bytes; the static scratch array holds " +
                       std::to_string(kStaticScratchBytes) + " bytes";
        return TN_ENOMEM;
    }
    void *scratch = nullptr;
    tn_status st = scratch_address(p, &scratch);
    if (st != TN_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Status word back to zero, then this plan's descriptor table.
    cudaError_t e = cudaMemsetAsync(scratch, 0, p.table_off, s);
    if (e == cudaSuccess && !p.table_blob.empty())
        e = cudaMemcpyAsync(static_cast<char *>(scratch) + p.table_off, p.table_blob.data(),
                            p.table_blob.size(), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) {
        p.last_error = std::string("preparing the static scratch array: ") + cudaGetErrorString(e);
        return TN_ECUDA;
    }
    void *saved_ws = p.ws;
    const uint64_t saved_size = p.ws_size;
    const bool saved_prof = p.profiling;
    p.ws = scratch;
    p.ws_size = kStaticScratchBytes;
    p.profiling = false;
    st = tn::execute_plan(&p, leaf_ptrs, out_ptr, s);
    p.ws = saved_ws;
    p.ws_size = saved_size;
    p.profiling = saved_prof;
    p.last_static = true;
    return st;
}
