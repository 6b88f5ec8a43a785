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

__global__ void __launch_bounds__(kThreads, 3) permute_kernel(const __grid_constant__ PermLaunch a) {
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
    if (d.tax >= 0) {
        // True transpose through shared memory.  Tiles of 32 entries along
        // axis tax (contiguous in the source) by 32 along the destination's
        // innermost axis L: a warp reads 32 consecutive source entries, and
        // after the tile turns in shared memory a warp writes 32 consecutive
        // destination entries.  The other axes index the tiles.
        __shared__ float2 tile[32][33];
        const int L = rank - 1, ax = d.tax;
        const int64_t na = (d.dims[ax] + 31) / 32, nl = (d.dims[L] + 31) / 32;
        int64_t dstride_a = 1;
        for (int x = ax + 1; x < rank; ++x) dstride_a *= d.dims[x];
        const int64_t ntiles = size / (d.dims[ax] * d.dims[L]) * na * nl;
        const int lane = threadIdx.x & 31, wrp = threadIdx.x >> 5;
        for (int64_t t = local; t < ntiles; t += ctas) {
            // tile t -> (rest, ta, tl): tl fastest, then ta, then the other
            // axes in destination order (row-major)
            int64_t rem = t;
            const int64_t tl = rem % nl;
            rem /= nl;
            const int64_t ta = rem % na;
            rem /= na;
            int64_t sbase = 0, dbase = 0, dstr = d.dims[L];
#pragma unroll 1
            for (int x = L - 1; x >= 0; --x) {
                if (x == ax) {
                    dstr *= d.dims[x];
                    continue;
                }
                const int64_t dg = rem % d.dims[x];
                rem /= d.dims[x];
                sbase += dg * d.sstride[x];
                dbase += dg * dstr;
                dstr *= d.dims[x];
            }
            const int64_t a0 = ta * 32, l0 = tl * 32;
            __syncthreads();   // the previous tile's readers are done
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int r = wrp + 8 * it;   // along L
                const int64_t ia = a0 + lane, il = l0 + r;
                if (ia < d.dims[ax] && il < d.dims[L])
                    tile[r][lane] = src[sbase + ia + il * d.sstride[L]];
            }
            __syncthreads();
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int c = wrp + 8 * it;   // along tax
                const int64_t ia = a0 + c, il = l0 + lane;
                if (ia < d.dims[ax] && il < d.dims[L])
                    store_entry(dst, fmt, size, dbase + ia * dstride_a + il, tile[lane][c], a.accumulate,
                                d.tile);
            }
        }
        return;
    }
    if (d.contig && d.tile.kt != 0 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        // A conversion into a K-tiled planar operand: the source is row-major
        // [rows][k], the destination per plane [k / kt][rows][kt].  Read
        // along rows and write along tile rows are both strided the other
        // way, so blocks of 32 rows x 128 entries turn through shared
        // memory: a warp reads 512 contiguous source bytes, and a warp writes
        // whole 64-byte tile rows of 32 consecutive rows (contiguous in every
        // plane).
        __shared__ __align__(16) float2 blk[32][128 + 4];
        const PlanarTile &tl = d.tile;
        const int64_t rows = tl.rows, kk = tl.k;
        const int kt = tl.kt;
        const int64_t nrb = (rows + 31) / 32, ncb = (kk + 127) / 128;
        const PlanarTile untiled{0, 0, -1, 0};
        // each CTA takes several blocks; the next block's loads are in flight
        // while this one's tile rows are stored
        const int64_t nblk = nrb * ncb;
        // thread: rows trow + 4 i of the block, entries c2, c2 + 1 (64 pairs
        // of entries per row)
        const int trow = threadIdx.x >> 6, c2 = (threadIdx.x & 63) * 2;
        float4 nxt[8];
        auto load_block = [&](int64_t u) {
            const int64_t r0 = (u / ncb) * 32, c0 = (u % ncb) * 128;
            if (c2 >= (int)min((int64_t)128, kk - c0)) return;
            const float4 *p = reinterpret_cast<const float4 *>(src + (r0 + trow) * kk + c0 + c2);
            const int64_t rstep = 2 * kk;   // four rows, in float4 units
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (r0 + trow + 4 * i < rows) nxt[i] = p[i * rstep];
        };
        if (local < nblk) load_block(local);
        for (int64_t u = local; u < nblk; u += ctas) {
            const int64_t r0 = (u / ncb) * 32, c0 = (u % ncb) * 128;
            const int cw = (int)min((int64_t)128, kk - c0);   // a multiple of kt
            __syncthreads();   // the previous block's readers are done
            if (c2 < cw) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (r0 + trow + 4 * i < rows) *reinterpret_cast<float4 *>(&blk[trow + 4 * i][c2]) = nxt[i];
            }
            __syncthreads();
            if (u + ctas < nblk) load_block(u + ctas);
            // quads of 4 entries: 8 kt quads per tile row block of 32 rows
            const int quads = (cw / kt) * 8 * kt;
            for (int q = threadIdx.x; q < quads; q += kThreads) {
                const int ct = q / (8 * kt), e = (q - ct * 8 * kt) * 4;
                const int row = e / kt, cl = e - row * kt;
                if (r0 + row >= rows) continue;
                const float2 v4[4] = {blk[row][ct * kt + cl], blk[row][ct * kt + cl + 1],
                                      blk[row][ct * kt + cl + 2], blk[row][ct * kt + cl + 3]};
                const int64_t phys = (((c0 / kt) + ct) * rows + r0 + row) * kt + cl;
                store_quad(dst, fmt, size, phys, v4, a.accumulate, untiled);
            }
        }
        return;
    }
    if (d.contig && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
        // a format conversion: source entry e is destination entry e.  Runs
        // of 16 entries are walked in the destination's physical order
        // (consecutive threads write consecutive addresses of every plane);
        // a K-tiled run (16 entries of one tile row) comes from 16
        // consecutive entries of one source row: 128 bytes, eight 16-byte
        // loads when the source is 16-byte aligned
        const PlanarTile &tl = d.tile;
        const PlanarTile untiled{0, 0, -1, 0};
        const bool src16 = (reinterpret_cast<uintptr_t>(src) & 15) == 0;
        const int64_t runs = size / 16;
        const int64_t stride = (int64_t)ctas * kThreads;
        for (int64_t u = (int64_t)local * kThreads + threadIdx.x; u < runs; u += stride) {
            const int64_t p0 = u * 16;
            int64_t e0 = p0;
            if (tl.kt != 0) {
                // physical ((c / kt) * rows + r) * kt + c % kt -> r * k + c
                const int sh = tl.kt == 32 ? 5 : 4;
                const int64_t cl = p0 & (tl.kt - 1), t2 = p0 >> sh;
                const int64_t ct = t2 / tl.rows, r = t2 - ct * tl.rows;
                e0 = r * tl.k + (ct << sh) + cl;
            }
            float2 v[16];
            if (src16) {
                const float4 *s4 = reinterpret_cast<const float4 *>(src + e0);
                float4 w[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) w[q] = s4[q];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    v[2 * q] = make_float2(w[q].x, w[q].y);
                    v[2 * q + 1] = make_float2(w[q].z, w[q].w);
                }
            } else {
#pragma unroll
                for (int q = 0; q < 16; ++q) v[q] = src[e0 + q];
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 v4[4] = {v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]};
                store_quad(dst, fmt, size, p0 + 4 * q, v4, a.accumulate, untiled);
            }
        }
        return;
    }
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

int permute_job_ctas(const PermDesc &d) {
    if (d.tax < 0 && d.contig && d.tile.kt != 0) {
        // K-tiled conversion: blocks of 32 rows x 128 entries, at least four
        // per CTA (the next block's loads overlap this one's stores), and at
        // most one full wave of CTAs (three per SM) per leaf: a large leaf's
        // CTAs then walk its blocks in one wave instead of several
        const int64_t blocks = ((d.tile.rows + 31) / 32) * ((d.tile.k + 127) / 128);
        int64_t c = (blocks + 3) / 4;
        if (c < 1) c = 1;
        if (c > 3 * 152) c = 3 * 152;
        return (int)c;
    }
    return permute_ctas(d.size);
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
