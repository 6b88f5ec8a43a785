// Leaf permutation: caller's storage order -> lifetime order.
//
// Lifetime ordering ("Crossing the single-GPU memory wall", section 1.4)
// removes every runtime transpose of intermediates; what is left is one
// reordering of each leaf that is not already stored in lifetime order,
// done here once per slice (a sliced leaf is read at the slice's offset).
// Many small leaves share one launch: each job owns a contiguous range of
// CTAs.  Destination writes are linear and coalesced; the source side is a
// gather through the job's strides.
#include "common.cuh"
#include "kernels.h"

namespace tn {

namespace {

constexpr int kThreads = 256;
constexpr int kItems = 4;

__global__ void __launch_bounds__(kThreads) permute_kernel(const __grid_constant__ PermLaunch a) {
    pdl_trigger();
    pdl_wait();
    // Find this CTA's job (uniform across the CTA).
    int lo = 0, hi = a.njobs - 1;
    const int b = blockIdx.x;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.cta_start[mid] <= b) lo = mid;
        else hi = mid - 1;
    }
    const int j = lo;
    const PermDesc &d = a.table[a.job[j]];
    const int ctas = a.cta_start[j + 1] - a.cta_start[j];
    const int local = b - a.cta_start[j];
    const float2 *src = a.src[j];
    void *dst = d.dst_off < 0 ? static_cast<void *>(a.out) : static_cast<void *>(a.arena + d.dst_off);
    const int32_t fmt = d.dst_off < 0 ? (int32_t)FMT_C64 : d.fmt;
    const int rank = d.rank;
    const int64_t size = d.size;
    // source offset of destination entry e (mixed radix over dims)
    auto source = [&](int64_t e) {
        int64_t rem = e, so = 0;
#pragma unroll 1
        for (int r = rank - 1; r >= 0; --r) {
            const int64_t dim = d.dims[r];
            if (d.dshift[r] >= 0) {
                so += (rem & (dim - 1)) * d.sstride[r];
                rem >>= d.dshift[r];
            } else {
                const int64_t q = rem / dim;
                so += (rem - q * dim) * d.sstride[r];
                rem = q;
            }
        }
        return so;
    };
    if (d.vec4 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
        // four consecutive entries per thread: consecutive in the source
        // too; all loads of the pass first, then one store per plane each
        // K-tiled destinations are walked in their physical order (whole
        // 64-byte tile rows per plane in turn); q * 4 is then a physical
        // index, and its logical index comes from undoing the tiling
        const PlanarTile &tl = d.tile;
        const bool phys = tl.kt != 0;
        const PlanarTile untiled{0, 0, -1, 0};
        const int64_t n4 = size / 4;
        const int64_t step4 = (int64_t)ctas * kThreads * kItems;
        for (int64_t base = (int64_t)local * kThreads * kItems; base < n4; base += step4) {
            float2 v[kItems][4];
#pragma unroll
            for (int it = 0; it < kItems; ++it) {
                const int64_t q = base + it * kThreads + threadIdx.x;
                if (q < n4) {
                    int64_t e = q * 4;
                    if (phys) {
                        // physical ((c / kt) * rows + r) * kt + c % kt
                        const int64_t cl = e % tl.kt, t2 = e / tl.kt;
                        const int64_t r = t2 % tl.rows, ct = t2 / tl.rows;
                        e = r * tl.k + ct * tl.kt + cl;
                    }
                    const float2 *p = src + source(e);
#pragma unroll
                    for (int u = 0; u < 4; ++u) v[it][u] = p[u];
                }
            }
#pragma unroll
            for (int it = 0; it < kItems; ++it) {
                const int64_t q = base + it * kThreads + threadIdx.x;
                if (q < n4) store_quad(dst, fmt, size, q * 4, v[it], a.accumulate, phys ? untiled : d.tile);
            }
        }
        return;
    }
    const int64_t step = (int64_t)ctas * kThreads * kItems;
    for (int64_t base = (int64_t)local * kThreads * kItems; base < size; base += step) {
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int64_t e = base + it * kThreads + threadIdx.x;
            if (e >= size) break;
            store_entry(dst, fmt, size, e, src[source(e)], a.accumulate, d.tile);
        }
    }
}

__global__ void __launch_bounds__(kThreads) gather_kernel(const __grid_constant__ GatherLaunch a) {
    pdl_trigger();
    pdl_wait();
    int lo = 0, hi = a.njobs - 1;
    const int b = blockIdx.x;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.cta_start[mid] <= b) lo = mid;
        else hi = mid - 1;
    }
    const int ctas = a.cta_start[lo + 1] - a.cta_start[lo];
    const int local = b - a.cta_start[lo];
    const float2 *src = a.src[lo];
    float2 *dst = a.dst[lo];
    const int64_t size = a.size[lo];
    const int64_t step = (int64_t)ctas * kThreads * kItems;
    for (int64_t base = (int64_t)local * kThreads * kItems; base < size; base += step) {
        // all loads of the pass in flight before the stores (host-link latency)
        float2 v[kItems];
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int64_t e = base + it * kThreads + threadIdx.x;
            v[it] = e < size ? src[e] : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int64_t e = base + it * kThreads + threadIdx.x;
            if (e < size) dst[e] = v[it];
        }
    }
}

__global__ void __launch_bounds__(kThreads) tensor_gather_kernel(const __grid_constant__ GatherArgs a) {
    pdl_trigger();
    pdl_wait();
    for (int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x; t < a.count;
         t += (int64_t)gridDim.x * kThreads) {
        const int64_t e = a.idx[t];
        float2 v = make_float2(0.f, 0.f);
        if (e < 0 || e >= a.size) {
            if (a.status) atomicCAS(&a.status->code, ERR_NONE, ERR_DESC);
        } else if (a.fmt == FMT_C64) {
            v = static_cast<const float2 *>(a.src)[e];
        } else {
            const int64_t o = tiled_offset(a.tile, e), pl = a.size;
            if (a.fmt == FMT_BF2 || a.fmt == FMT_BF4) {
                const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.src) + o;
                v.x = __bfloat162float(q[0]);
                v.y = __bfloat162float(q[pl]);
                if (a.fmt == FMT_BF4) {
                    v.x += __bfloat162float(q[2 * pl]);
                    v.y += __bfloat162float(q[3 * pl]);
                }
            } else {
                // FMT_SPLIT4: [re_hi, im_hi, re_lo, im_lo]; FMT_GAUSS6:
                // [re_hi, im_hi, s_hi, re_lo, im_lo, s_lo]
                const float *q = static_cast<const float *>(a.src) + o;
                const int64_t lo = a.fmt == FMT_GAUSS6 ? 3 * pl : 2 * pl;
                v.x = q[0] + q[lo];
                v.y = q[pl] + q[lo + pl];
            }
        }
        a.dst[t] = v;
    }
}

}  // namespace

cudaError_t launch_tensor_gather(const GatherArgs &args, cudaStream_t stream) {
    if (args.count <= 0) return cudaSuccess;
    int64_t blocks = (args.count + kThreads - 1) / kThreads;
    if (blocks > 152 * 8) blocks = 152 * 8;
    return launch_pdl(tensor_gather_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream, args);
}

int permute_ctas(int64_t size) {
    const int64_t per = (int64_t)kThreads * kItems;
    int64_t c = (size + per - 1) / per;
    if (c < 1) c = 1;
    if (c > 4096) c = 4096;
    return (int)c;
}

cudaError_t launch_permute(const PermLaunch &args, int total_ctas, cudaStream_t stream) {
    if (args.njobs <= 0) return cudaSuccess;
    return launch_pdl(permute_kernel, dim3(total_ctas), dim3(kThreads), 0, stream, args);
}

cudaError_t launch_gather(const GatherLaunch &args, int total_ctas, cudaStream_t stream) {
    if (args.njobs <= 0) return cudaSuccess;
    return launch_pdl(gather_kernel, dim3(total_ctas), dim3(kThreads), 0, stream, args);
}

}  // namespace tn
