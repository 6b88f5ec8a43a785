// Fused leaf subtrees: one CTA computes a whole small subtree near the
// leaves ("leaf-gate absorption").
//
// In circuit networks most steps near the leaves absorb a single-qubit gate
// into a wire or join two small gate tensors; in random networks small
// leaves meet.  Run one launch per tree level (the batched tiny kernel),
// such a chain costs a launch and a round trip through HBM per level.  Here
// each fused group (FuseGroup in plan.h: a maximal subtree whose leaves and
// intermediates are all small) is one CTA: it gathers its leaves from the
// caller's buffers straight into shared memory in lifetime order (the leaf
// permutation of "Crossing the single-GPU memory wall", section 1.3, done on
// the load through a precomputed list of source offsets, all loads
// independent), computes its steps level by level in shared memory (every
// step C[i, j] = sum_k A[i, k] B[j, k] of section 1.1 on the section 1.4
// layouts, C stored at offM(i) + offN(j)), and stores only the group's root,
// in its consumer's format.  The steps of one level are independent: their
// outputs form one flat index space over the CTA's threads, and the level
// ends with a barrier.  Step descriptors and output offsets are copied to
// shared memory first, so the level loop touches no global memory.
#include "common.cuh"
#include "kernels.h"

namespace tn {

namespace {

constexpr int kThreads = 512;

__global__ void __launch_bounds__(kThreads) fused_kernel(const __grid_constant__ FuseLaunch a) {
    extern __shared__ float2 sm[];
    __shared__ FuseGroup gs;
    pdl_trigger();
    const int x = blockIdx.x;
    // the group's descriptor (tables are written once, before any launch)
    {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(a.groups + a.group[x]);
        uint32_t *dst = reinterpret_cast<uint32_t *>(&gs);
        for (int w = threadIdx.x; w < (int)(sizeof(FuseGroup) / 4); w += kThreads) dst[w] = src[w];
    }
    __syncthreads();
    const FuseGroup g = gs;
    // descriptors after the tensors: steps, level starts (steps, then warp
    // chunks), output offsets, the step of every warp chunk; like the group
    // descriptor they are written before any launch, so they are read
    // before waiting for the previous grid
    FuseNode *nodes = reinterpret_cast<FuseNode *>(sm + g.smem);
    int32_t *levels = reinterpret_cast<int32_t *>(nodes + g.n_nodes);
    int32_t *lchunk = levels + g.n_levels + 1;
    int32_t *offs = lchunk + g.n_levels + 1;
    int32_t *cnode = offs + g.n_off;
    {
        const int32_t *src = reinterpret_cast<const int32_t *>(a.nodes + g.first_node);
        int32_t *dst = reinterpret_cast<int32_t *>(nodes);
        const int words = g.n_nodes * (int)(sizeof(FuseNode) / 4);
        for (int w = threadIdx.x; w < words; w += kThreads) dst[w] = src[w];
        for (int w = threadIdx.x; w < 2 * (g.n_levels + 1); w += kThreads)
            levels[w] = a.levels[g.first_level + w];
        for (int w = threadIdx.x; w < g.n_off; w += kThreads) offs[w] = a.offs[g.first_off + w];
        for (int w = threadIdx.x; w < g.n_chunks; w += kThreads) cnode[w] = a.chunks[g.first_chunk + w];
    }
    // leaves: slot e <- the caller's leaf at its source offset.  The (leaf,
    // offset) pairs are static too: each thread parks its slots' pairs in the
    // slots themselves, then, once the previous grid (which may have written
    // the leaves) is done, replaces each by the leaf entry: one round trip
    // after the wait instead of two
    for (int e = threadIdx.x; e < g.n_gather; e += kThreads) {
        const FuseGather ge = a.gather[g.first_gather + e];
        reinterpret_cast<int2 *>(sm)[e] = make_int2(ge.leaf, ge.src);
    }
    pdl_wait();
    const float2 *const *src = a.src + a.src_first[x];
    for (int e = threadIdx.x; e < g.n_gather; e += kThreads) {
        const int2 ge = reinterpret_cast<const int2 *>(sm)[e];
        sm[e] = src[ge.x][ge.y];
    }
    __syncthreads();
    void *out = g.out_off < 0 ? static_cast<void *>(a.out) : static_cast<void *>(a.arena + g.out_off);
    const int accumulate = g.is_root ? a.accumulate_root : 0;
    const int lane = threadIdx.x & 31;
    for (int lv = 0; lv < g.n_levels; ++lv) {
        const int c0 = lchunk[lv], total = (lchunk[lv + 1] - c0) * 32;
        // warp by warp over the level's items (a step's items start at a
        // multiple of 32, so a warp's lanes all belong to one step, read from
        // the chunk table)
        for (int base = threadIdx.x - lane; base < total; base += kThreads) {
            const FuseNode &nd = nodes[cnode[c0 + (base >> 5)]];
            // shifts, not divisions: every level waits for its slowest chain
            const int L = 1 << nd.lshift;
            const int item = base + lane - nd.obase;
            const int o = item >> nd.lshift, l = item & (L - 1);
            const bool valid = o < nd.m * nd.n;
            float2 acc = make_float2(0.f, 0.f);
            int i = 0, j = 0;
            if (valid) {
                if (nd.nshift >= 0) {
                    i = o >> nd.nshift;
                    j = o & (nd.n - 1);
                } else {
                    i = o / nd.n;
                    j = o - i * nd.n;
                }
                const float2 *ar = sm + nd.a + i * nd.k, *br = sm + nd.b + j * nd.k;
                // two independent chains of multiply-adds
                float2 acc1 = make_float2(0.f, 0.f);
                int kk = l;
                for (; kk + L < nd.k; kk += 2 * L) {
                    cfma(acc, ar[kk], br[kk]);
                    cfma(acc1, ar[kk + L], br[kk + L]);
                }
                if (kk < nd.k) cfma(acc, ar[kk], br[kk]);
                acc.x += acc1.x;
                acc.y += acc1.y;
            }
            for (int off = L >> 1; off > 0; off >>= 1) {
                acc.x += __shfl_down_sync(0xffffffffu, acc.x, off, L);
                acc.y += __shfl_down_sync(0xffffffffu, acc.y, off, L);
            }
            if (valid && l == 0) {
                const int dst = offs[nd.off + i] + offs[nd.off + nd.m + j];
                if (nd.c >= 0) sm[nd.c + dst] = acc;
                else store_entry(out, g.out_fmt, (int64_t)nd.m * nd.n, dst, acc, accumulate, g.out_tile);
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_fused(const FuseLaunch &args, int smem_bytes, cudaStream_t stream) {
    if (args.ngroups <= 0) return cudaSuccess;
    static int attr_bytes = 0;
    const int bytes = (smem_bytes + 15) / 16 * 16;
    if (bytes > 48 * 1024 && bytes > attr_bytes) {
        cudaError_t e = cudaFuncSetAttribute(fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             bytes);
        if (e != cudaSuccess) return e;
        attr_bytes = bytes;
    }
    return launch_pdl(fused_kernel, dim3(args.ngroups), dim3(kThreads), (size_t)bytes, stream, args);
}

}  // namespace tn
