// Batched kernel for tiny nodes.
//
// Most nodes near the leaves of a tree are tiny (a few hundred to a few
// million complex multiply-adds: single-qubit gates absorbed into wires,
// small random tensors meeting).  One launch per node would cost several
// microseconds of launch and memory latency each, far more than their
// arithmetic.  All tiny nodes of one schedule stage are independent, so one
// launch runs them all: each node owns CTAs (its cta_base range in the
// descriptor table), enough that every thread group computes about one
// output, since each output is a serial chain of memory waits; `lanes`
// threads cooperate on one output's k range (k <= 512: one round of loads,
// 16 entries per lane) and combine with warp shuffles.  One lane decodes
// each output's address into (i, j) and passes it to the lanes that compute
// it.  Operands are complex64 in the workspace arena; the output goes
// through the node's separable offsets in its consumer's format (the root
// adds into the caller's output on later slices).
#include "common.cuh"
#include "kernels.h"

namespace tn {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) tiny_batch_kernel(const __grid_constant__ TinyLaunch a) {
    __shared__ int node_s;
    __shared__ __align__(16) TinyDesc ds;
    pdl_trigger();
    // This CTA's node: the one whose CTA range holds blockIdx.x, found with
    // one compare per thread over the launch parameters; then its
    // descriptor, copied once into shared memory, where the output loop
    // reads it.  The table is written once, before any launch, so both
    // steps may run before the previous launch has finished.
    const int b = blockIdx.x;
    if (threadIdx.x == 0) node_s = 0;   // (every CTA matches one node)
    __syncthreads();
    for (int t = threadIdx.x; t < a.count; t += kThreads)
        if (a.base[t] <= b && b < a.base[t + 1]) node_s = t;
    __syncthreads();
    {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(a.table + a.first + node_s);
        uint32_t *dst = reinterpret_cast<uint32_t *>(&ds);
        for (int x = threadIdx.x; x < (int)(sizeof(TinyDesc) / 4); x += kThreads) dst[x] = src[x];
    }
    __syncthreads();
    pdl_wait();
    const TinyDesc &d = ds;
    const int local = b - d.cta_base;
    const float2 *A = reinterpret_cast<const float2 *>(a.arena + d.a_off);
    const float2 *B = reinterpret_cast<const float2 *>(a.arena + d.b_off);
    void *C = d.c_off < 0 ? static_cast<void *>(a.out) : static_cast<void *>(a.arena + d.c_off);
    const int64_t mn = (int64_t)d.m * d.n;
    const int64_t per = (mn + d.ctas - 1) / d.ctas;
    const int64_t o0 = (int64_t)local * per;
    const int64_t o1 = min(mn, o0 + per);
    const int lanes = d.lanes;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int opw = 32 / lanes;                        // outputs per warp and pass
    const int chunk = opw;                             // outputs of one decode pass
    const int l = lane % lanes, gq = lane / lanes;
    const int accumulate = d.is_root ? a.accumulate_root : 0;
    const int k = d.k;
    // rows of even length on 16-byte boundaries load two entries at a time
    const bool pairs = (k & 1) == 0 && ((reinterpret_cast<uintptr_t>(A) |
                                         reinterpret_cast<uintptr_t>(B)) & 15) == 0;
    // Each warp takes `chunk` consecutive addresses at a time: lane q
    // decodes address cb + q into (i, j) (the walk; m n <= 2^23 here, so
    // 32-bit index arithmetic is exact), then groups of `lanes` lanes take
    // the outputs in address order, reading (i, j) from the decoding lane.
    for (int64_t cb = o0 + (int64_t)warp * chunk; cb < o1; cb += (int64_t)(kThreads / 32) * chunk) {
        int wi = 0, wj = 0;
        if (lane < chunk && cb + lane < o1) {
            int rem = static_cast<int>(cb + lane);
#pragma unroll 1
            for (int t = 0; t < d.wn; ++t) {
                int dg;
                if (d.wshift[t] >= 0) {
                    dg = rem & (d.wext[t] - 1);
                    rem >>= d.wshift[t];
                } else {
                    const int q = rem / d.wext[t];
                    dg = rem - q * d.wext[t];
                    rem = q;
                }
                if ((d.wside >> t) & 1u) wj += dg * d.wt[t];
                else wi += dg * d.wt[t];
            }
        }
#pragma unroll 1
        for (int q0 = 0; q0 < chunk; q0 += opw) {
            const int q = q0 + gq;
            const int64_t o = cb + q;
            const int i = __shfl_sync(0xffffffffu, wi, q);
            const int j = __shfl_sync(0xffffffffu, wj, q);
            float2 acc = make_float2(0.f, 0.f);
            if (o < o1) {
                const float2 *ar = A + (int64_t)i * k, *br = B + (int64_t)j * k;
                if (pairs) {
                    // eight independent 16-byte load pairs in flight per round
                    const float4 *ar4 = reinterpret_cast<const float4 *>(ar);
                    const float4 *br4 = reinterpret_cast<const float4 *>(br);
                    const int k2 = k >> 1;
                    for (int kk = l; kk < k2; kk += 8 * lanes) {
                        float4 av[8], bv[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int idx = kk + u * lanes;
                            av[u] = idx < k2 ? ar4[idx] : make_float4(0.f, 0.f, 0.f, 0.f);
                            bv[u] = idx < k2 ? br4[idx] : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            cfma(acc, make_float2(av[u].x, av[u].y), make_float2(bv[u].x, bv[u].y));
                            cfma(acc, make_float2(av[u].z, av[u].w), make_float2(bv[u].z, bv[u].w));
                        }
                    }
                } else {
                    // eight independent load pairs in flight per round
                    for (int kk = l; kk < k; kk += 8 * lanes) {
                        float2 av[8], bv[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int idx = kk + u * lanes;
                            av[u] = idx < k ? ar[idx] : make_float2(0.f, 0.f);
                            bv[u] = idx < k ? br[idx] : make_float2(0.f, 0.f);
                        }
#pragma unroll
                        for (int u = 0; u < 8; ++u) cfma(acc, av[u], bv[u]);
                    }
                }
            }
            for (int off = lanes >> 1; off > 0; off >>= 1) {
                acc.x += __shfl_down_sync(0xffffffffu, acc.x, off, lanes);
                acc.y += __shfl_down_sync(0xffffffffu, acc.y, off, lanes);
            }
            if (l == 0 && o < o1) store_entry(C, d.out_fmt, mn, o, acc, accumulate, d.out_tile);
        }
    }
}

}  // namespace

cudaError_t launch_tiny_batch(const TinyLaunch &args, int ctas, cudaStream_t stream) {
    if (ctas <= 0) return cudaSuccess;
    return launch_pdl(tiny_batch_kernel, dim3(ctas), dim3(kThreads), 0, stream, args);
}

}  // namespace tn
