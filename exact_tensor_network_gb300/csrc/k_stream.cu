// Bandwidth-bound node kernel and the split-K reduction.
//
// Nodes with a small side (n <= 16 after swapping the operands when m is
// the small one) are gate-like contractions, outer products and dot products:
// their time is reading the big operand A once (the t_gemm bandwidth term
// of "Crossing the single-GPU memory wall", section 1.6).  B is staged in
// shared memory one k-chunk at a time; each row of A is read once, by
// `lanes` threads that split its k range and then combine their partial
// sums with warp shuffles.  Long k ranges are cut into ksplit chunks run by
// different CTAs; their fp32 partial sums land in the workspace and the
// last split of each row block adds them in a fixed order (deterministic),
// then stores the node's output through its separable offsets in the
// consumer's format.  splitk_reduce does the same for the other classes.
#include "common.cuh"
#include "kernels.h"

namespace tn {

namespace {

constexpr int kThreads = 256;

// NB: a bound on n (4, 8 or 16) that sizes the unrolled column loops.
template <int FMT, int NB>
__global__ void __launch_bounds__(kThreads) stream_node_kernel(const __grid_constant__ StreamArgs a) {
    __shared__ float2 Bs[NB * kStreamKc];
    pdl_trigger();
    pdl_wait();
    const int s = blockIdx.y;
    const int64_t k0 = (int64_t)s * a.kchunk;
    const int64_t k1 = min(a.k, k0 + a.kchunk);
    const int n = (int)a.n;
    const int lanes = a.lanes;
    const int g = threadIdx.x / lanes, l = threadIdx.x % lanes;
    const int groups = kThreads / lanes;
    const int64_t r0 = (int64_t)blockIdx.x * a.rows_per_cta;
    const int64_t r1 = min(a.m, r0 + a.rows_per_cta);

    // accumulators per row, B staged chunk by chunk
    for (int64_t rb = r0; rb < r1; rb += groups) {
        const int64_t r = rb + g;
        float2 acc[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j) acc[j] = make_float2(0.f, 0.f);
        for (int64_t c0 = k0; c0 < k1; c0 += kStreamKc) {
            const int clen = (int)min((int64_t)kStreamKc, k1 - c0);
            // this lane's first eight entries of the row are in flight while
            // B is staged; later batches keep eight loads in flight as well
            const float2 *arow = a.A + r * a.k + c0;
            float2 av[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int idx = l + u * lanes;
                av[u] = (r < r1 && idx < clen) ? arow[idx] : make_float2(0.f, 0.f);
            }
            __syncthreads();
#pragma unroll 4
            for (int e = threadIdx.x; e < n * clen; e += kThreads) {
                const int j = e / clen, kk = e - j * clen;
                Bs[j * kStreamKc + kk] = a.B[(int64_t)j * a.k + c0 + kk];
            }
            __syncthreads();
            if (r < r1) {
                for (int kb = l; kb < clen; kb += 8 * lanes) {
                    if (kb != l) {
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int idx = kb + u * lanes;
                            av[u] = idx < clen ? arow[idx] : make_float2(0.f, 0.f);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int idx = kb + u * lanes;
                        if (idx < clen) {
#pragma unroll
                            for (int j = 0; j < NB; ++j)
                                if (j < n) cfma(acc[j], av[u], Bs[j * kStreamKc + idx]);
                        }
                    }
                }
            }
        }
        // combine the lanes of a row
        for (int off = lanes >> 1; off > 0; off >>= 1) {
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                if (j < n) {
                    acc[j].x += __shfl_down_sync(0xffffffffu, acc[j].x, off, lanes);
                    acc[j].y += __shfl_down_sync(0xffffffffu, acc[j].y, off, lanes);
                }
            }
        }
        if (l == 0 && r < r1) {
            if (a.ksplit > 1) {
                float2 *dst = a.part + ((int64_t)s * a.m + r) * a.n;
#pragma unroll
                for (int j = 0; j < NB; ++j)
                    if (j < n) dst[j] = acc[j];
            } else {
                const int64_t offm = sep_offset(a.lm, r);
#pragma unroll
                for (int j = 0; j < NB; ++j)
                    if (j < n)
                        store_entry_t<FMT>(a.C, a.m * a.n, offm + sep_offset(a.ln, j), acc[j],
                                           a.accumulate, a.out_tile);
            }
        }
    }
    if (a.ksplit > 1) {
        // The last split of this row block to finish sums the partials of
        // all splits and stores the rows; a counter, not a wait.  Row blocks
        // are small (often a few dozen entries) and splits many, so the
        // threads split both: E threads (a power of two covering the block,
        // at most all of them) per entry, G = 256 / E groups over the splits
        // (group g takes splits g, g + G, ...: four loads in flight), then
        // group 0 adds the G group sums in order.  The order is fixed, so
        // runs are bit-identical.
        __shared__ int last;
        __shared__ float2 red_s[kThreads];
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) last = atomicAdd(a.cnt + blockIdx.x, 1) == a.ksplit - 1;
        __syncthreads();
        if (!last) return;
        __threadfence();
        // rows r0..r1 are one contiguous run of each split's partials
        const int64_t cnt = (r1 - r0) * n, plane = a.m * a.n;
        const float2 *base = a.part + r0 * a.n;
        int E = 1;
        while (E < cnt && E < kThreads) E <<= 1;
        const int G = kThreads / E;
        const int eg = threadIdx.x % E, gi = threadIdx.x / E;
        for (int64_t e0 = 0; e0 < cnt; e0 += E) {
            const int64_t e = e0 + eg;
            float2 v = make_float2(0.f, 0.f);
            if (e < cnt) {
                const float2 *pe = base + e;
                int sp = gi;
                for (; sp + 3 * G < a.ksplit; sp += 4 * G) {
                    float2 x[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) x[u] = __ldcg(pe + (int64_t)(sp + u * G) * plane);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        v.x += x[u].x;
                        v.y += x[u].y;
                    }
                }
                for (; sp < a.ksplit; sp += G) {
                    const float2 x = __ldcg(pe + (int64_t)sp * plane);
                    v.x += x.x;
                    v.y += x.y;
                }
            }
            if (G > 1) {
                red_s[threadIdx.x] = v;
                __syncthreads();
                if (gi == 0 && e < cnt) {
                    for (int g2 = 1; g2 < G; ++g2) {
                        const float2 x = red_s[g2 * E + eg];
                        v.x += x.x;
                        v.y += x.y;
                    }
                }
                __syncthreads();
            }
            if (gi == 0 && e < cnt) {
                const int64_t r = r0 + e / n;
                const int j = (int)(e - (r - r0) * n);
                store_entry_t<FMT>(a.C, plane, sep_offset(a.lm, r) + sep_offset(a.ln, j), v,
                                   a.accumulate, a.out_tile);
            }
        }
        if (threadIdx.x == 0) a.cnt[blockIdx.x] = 0;   // ready for the next run
    }
}

// Streaming node with k <= 16 (gate-like, outer products): B (n x k) is
// staged once per CTA; each thread takes 16 / K rows per pass (K = k rounded
// up to a power of two), issues all their loads before any arithmetic
// (16-byte loads when k = K is even) and then computes and stores the rows
// one by one.  Consecutive threads own consecutive rows, so A is read and
// (for outputs whose M side is innermost) C written in whole lines.
template <int K>
__global__ void __launch_bounds__(kThreads) stream_rows_kernel(const __grid_constant__ StreamArgs a) {
    constexpr int RPT = 16 / K;   // rows per thread and pass
    __shared__ __align__(16) float2 Bs[kStreamMaxN * K];
    // B read two entries (16 bytes, the same address in every lane) at a time
    const float4 *Bs2 = reinterpret_cast<const float4 *>(Bs);
    __shared__ int64_t offn_s[kStreamMaxN];
    // row-major [m, n] outputs: each warp's 32 rows are one contiguous run,
    // staged here and stored by consecutive lanes
    __shared__ float2 Cs[kThreads / 32][32 * (kStreamMaxN + 1)];
    pdl_trigger();
    pdl_wait();
    const int n = (int)a.n, k = (int)a.k;
    for (int e = threadIdx.x; e < n * K; e += kThreads) {
        const int j = e / K, kk = e - j * K;
        Bs[e] = kk < k ? a.B[(int64_t)j * k + kk] : make_float2(0.f, 0.f);
    }
    if (threadIdx.x < n) offn_s[threadIdx.x] = sep_offset(a.ln, threadIdx.x);
    __syncthreads();
    const bool vec = (k == K) && (K % 2 == 0);
    const int64_t pass = (int64_t)kThreads * RPT;
    for (int64_t base = (int64_t)blockIdx.x * pass; base < a.m; base += (int64_t)gridDim.x * pass) {
        float2 av[RPT][K];
#pragma unroll
        for (int u = 0; u < RPT; ++u) {
            const int64_t r = base + u * kThreads + threadIdx.x;
            const float2 *row = a.A + r * k;
            if (r < a.m && vec) {
                const float4 *row4 = reinterpret_cast<const float4 *>(row);
#pragma unroll
                for (int h = 0; h < K / 2; ++h) {
                    const float4 v = row4[h];
                    av[u][2 * h] = make_float2(v.x, v.y);
                    av[u][2 * h + 1] = make_float2(v.z, v.w);
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < K; ++kk)
                    av[u][kk] = (r < a.m && kk < k) ? row[kk] : make_float2(0.f, 0.f);
            }
        }
        if (a.rows_contig) {
            const int lane = threadIdx.x & 31;
            float2 *tile = Cs[threadIdx.x >> 5];
            const int ts = n | 1;   // odd row stride: lanes' rows in distinct banks
            const int dr = 32 / n, dc = 32 - dr * n;
#pragma unroll
            for (int u = 0; u < RPT; ++u) {
                const int64_t r = base + u * kThreads + threadIdx.x;
                if (r < a.m) {
#pragma unroll 1
                    for (int j = 0; j < n; ++j) {
                        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                        for (int kk = 0; kk < K; kk += 2) {
                            const float4 b2 = Bs2[(j * K + kk) >> 1];
                            cfma(acc, av[u][kk], make_float2(b2.x, b2.y));
                            cfma(acc, av[u][kk + 1], make_float2(b2.z, b2.w));
                        }
                        tile[lane * ts + j] = acc;
                    }
                }
                __syncwarp();
                const int64_t r0 = base + u * kThreads + (threadIdx.x & ~31);
                const int64_t cnt = r0 < a.m ? min((int64_t)32, a.m - r0) * n : 0;
                // entry e = rr n + cc of the warp's run; e steps by 32
                int rr = lane / n, cc = lane - rr * n;
#pragma unroll 1
                for (int e = lane; e < (int)cnt; e += 32) {
                    store_entry(a.C, a.out_fmt, a.m * a.n, r0 * n + e, tile[rr * ts + cc],
                                a.accumulate, a.out_tile);
                    rr += dr;
                    cc += dc;
                    if (cc >= n) {
                        cc -= n;
                        ++rr;
                    }
                }
                __syncwarp();
            }
            continue;
        }
#pragma unroll
        for (int u = 0; u < RPT; ++u) {
            const int64_t r = base + u * kThreads + threadIdx.x;
            if (r >= a.m) continue;
            const int64_t offm = sep_offset(a.lm, r);
#pragma unroll 1
            for (int j = 0; j < n; ++j) {
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int kk = 0; kk < K; kk += 2) {
                    const float4 b2 = Bs2[(j * K + kk) >> 1];
                    cfma(acc, av[u][kk], make_float2(b2.x, b2.y));
                    cfma(acc, av[u][kk + 1], make_float2(b2.z, b2.w));
                }
                store_entry(a.C, a.out_fmt, a.m * a.n, offm + offn_s[j], acc, a.accumulate,
                            a.out_tile);
            }
        }
    }
}

// Gate-like node with n = k = 16 (a 4-mode gate on a large state): 1024 fp32
// FMAs per 256 bytes of HBM traffic, so on the shared-memory B of
// stream_rows_kernel the loads of B and the store loop cost as many issue
// slots as the arithmetic.  Here eight lanes share a row: lane (h, q) owns
// the outputs 8h .. 8h+7 and the complex k entries {2q, 2q+1, 8+2q, 9+2q},
// and keeps the matching 8 x 4 slice of B in registers for the whole
// launch, so the inner loop is FMAs only (and the registers leave room for
// four warps per scheduler).  The four lanes of an output half combine
// their partial sums by a reduce-scatter (two shuffle steps), after which
// lane (h, q) holds outputs 8h + 2q and 8h + 2q + 1.  So that every lane
// runs the same code, lane q's register i holds output 8h + (i ^ 2q): the
// partner lane q ^ 2 keeps the same outputs in registers i ^ 4, and lane
// q ^ 1 in registers i ^ 2.  Rows arrive through a per-warp ring of
// cp.async copies (kG16Depth groups of 4 rows, 512 bytes, per warp; each
// lane copies 16 bytes, and one warp sync per group makes the group
// readable and frees the slot read last for the next copy).
constexpr int kG16Warps = 16;
constexpr int kG16Depth = 16;
constexpr int kG16Smem = kG16Warps * kG16Depth * 512;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, int src_bytes) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kG16Warps * 32, 1) stream_g16_kernel(const __grid_constant__ StreamArgs a) {
    extern __shared__ __align__(16) float4 g16_ring[];
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rr = lane >> 3, h = (lane >> 2) & 1, q = lane & 3;
    float4 *ring = g16_ring + warp * kG16Depth * 32;
    // B slice: register i, entry t holds B[8h + (i ^ 2q)][kt], kt = 2q + (t & 1) + 8 (t >> 1)
    float2 b[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int j = 8 * h + (i ^ (2 * q));
#pragma unroll
        for (int t = 0; t < 4; ++t) b[i][t] = a.B[j * 16 + 2 * q + (t & 1) + 8 * (t >> 1)];
    }
    int64_t offn[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) offn[i] = a.rows_contig ? 8 * h + 2 * q + i : sep_offset(a.ln, 8 * h + 2 * q + i);
    const int64_t ngroups = (a.m + 3) / 4;
    const int64_t g0 = (int64_t)blockIdx.x * kG16Warps + warp;
    const int64_t gstride = (int64_t)gridDim.x * kG16Warps;
    // the warp's group g is rows 4g .. 4g+3, 512 contiguous bytes: lane l
    // copies bytes 16 l .. 16 l + 15 (zero-filled past the last row)
    auto issue = [&](int64_t g, int slot) {
        const int64_t r = g * 4 + (lane >> 3);
        const bool ok = r < a.m;
        const float2 *src = a.A + (ok ? g * 64 + 2 * lane : 0);
        cp_async16(ring + slot * 32 + lane, src, ok ? 16 : 0);
    };
#pragma unroll
    for (int s = 0; s < kG16Depth - 1; ++s) {
        const int64_t g = g0 + s * gstride;
        if (g < ngroups) issue(g, s);
        cp_async_commit();
    }
    int slot = 0;
    for (int64_t g = g0; g < ngroups; g += gstride) {
        // this group's copies (every lane's) are complete and visible, and
        // every lane has read the previous slot: it can be refilled
        cp_async_wait<kG16Depth - 2>();
        __syncwarp();
        // row rr's entries 2q, 2q+1 (16 bytes at 16 q) and 8+2q, 9+2q (at 64 + 16 q)
        const float4 p0 = ring[slot * 32 + rr * 8 + q], p1 = ring[slot * 32 + rr * 8 + 4 + q];
        const int64_t gn = g + (kG16Depth - 1) * gstride;
        if (gn < ngroups) issue(gn, slot == 0 ? kG16Depth - 1 : slot - 1);
        cp_async_commit();
        slot = slot == kG16Depth - 1 ? 0 : slot + 1;
        const float2 av[4] = {make_float2(p0.x, p0.y), make_float2(p0.z, p0.w), make_float2(p1.x, p1.y),
                              make_float2(p1.z, p1.w)};
        float2 acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            acc[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int t = 0; t < 4; ++t) cfma(acc[i], av[t], b[i][t]);
        }
        // reduce-scatter over the four lanes of the output half: keep
        // registers 0..3 and receive lane ^ 2's 4..7 (the same outputs),
        // then keep 0..1 and receive lane ^ 1's 2..3
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[i].x += __shfl_xor_sync(0xffffffffu, acc[i + 4].x, 2);
            acc[i].y += __shfl_xor_sync(0xffffffffu, acc[i + 4].y, 2);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            acc[i].x += __shfl_xor_sync(0xffffffffu, acc[i + 2].x, 1);
            acc[i].y += __shfl_xor_sync(0xffffffffu, acc[i + 2].y, 1);
        }
        const int64_t r = g * 4 + rr;
        if (r < a.m) {
            if (a.rows_contig && a.out_fmt == FMT_C64) {
                float4 *p = reinterpret_cast<float4 *>(static_cast<float2 *>(a.C) + r * 16 + 8 * h + 2 * q);
                float4 v = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
                if (a.accumulate) {
                    const float4 o = *p;
                    v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
                }
                *p = v;
            } else {
                const int64_t offm = a.rows_contig ? r * 16 : sep_offset(a.lm, r);
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    store_entry(a.C, a.out_fmt, a.m * 16, offm + offn[i], acc[i], a.accumulate,
                                a.out_tile);
            }
        }
    }
    cp_async_wait<0>();
}

__global__ void __launch_bounds__(kThreads) splitk_reduce_kernel(const __grid_constant__ ReduceArgs a) {
    pdl_trigger();
    pdl_wait();
    const int64_t mn = a.m * a.n;
    for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < mn;
         e += (int64_t)gridDim.x * kThreads) {
        // splits added in order, four loads in flight
        float2 v = make_float2(0.f, 0.f);
        int s = 0;
        for (; s + 4 <= a.ksplit; s += 4) {
            float2 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) x[u] = __ldcg(a.part + (int64_t)(s + u) * mn + e);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                v.x += x[u].x;
                v.y += x[u].y;
            }
        }
        for (; s < a.ksplit; ++s) {
            const float2 p = __ldcg(a.part + (int64_t)s * mn + e);
            v.x += p.x;
            v.y += p.y;
        }
        const int64_t i = e / a.n, j = e - i * a.n;
        store_entry(a.C, a.out_fmt, mn, sep_offset(a.lm, i) + sep_offset(a.ln, j), v, a.accumulate,
                    a.out_tile);
    }
}

template <int NB>
cudaError_t launch_stream_nb(const StreamArgs &args, dim3 grid, cudaStream_t stream) {
    if (args.out_fmt == FMT_SPLIT4)
        return launch_pdl(stream_node_kernel<FMT_SPLIT4, NB>, grid, dim3(kThreads), 0, stream, args);
    else if (args.out_fmt == FMT_GAUSS6)
        return launch_pdl(stream_node_kernel<FMT_GAUSS6, NB>, grid, dim3(kThreads), 0, stream, args);
    else if (args.out_fmt == FMT_BF2)
        return launch_pdl(stream_node_kernel<FMT_BF2, NB>, grid, dim3(kThreads), 0, stream, args);
    else if (args.out_fmt == FMT_BF4)
        return launch_pdl(stream_node_kernel<FMT_BF4, NB>, grid, dim3(kThreads), 0, stream, args);
    return launch_pdl(stream_node_kernel<FMT_C64, NB>, grid, dim3(kThreads), 0, stream, args);
}

}  // namespace

cudaError_t launch_stream_node(const StreamArgs &args, cudaStream_t stream) {
    if (args.k <= 16 && args.ksplit <= 1) {
        // output entry (i, j) at i n + j (plain row-major [m, n]) with n >= 4:
        // stage each warp's rows; with n < 4 a thread's own entries already
        // fill most of a sector
        StreamArgs a2 = args;
        a2.rows_contig = args.n >= 4 &&
                         (args.lm.nrun == 0 || (args.lm.nrun == 1 && args.lm.stride[0] == args.n)) &&
                         (args.ln.nrun == 0 || (args.ln.nrun == 1 && args.ln.stride[0] == 1));
        const bool a_aligned = (reinterpret_cast<uintptr_t>(args.A) & 15) == 0;
        const bool c_aligned = (reinterpret_cast<uintptr_t>(args.C) & 15) == 0;
        if (args.k == 16 && args.n == 16 && a_aligned && (c_aligned || !a2.rows_contig)) {
            static bool attr_set = false;
            if (!attr_set) {
                cudaError_t e = cudaFuncSetAttribute(stream_g16_kernel,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kG16Smem);
                if (e != cudaSuccess) return e;
                attr_set = true;
            }
            const int64_t groups = (args.m + 3) / 4;   // groups of four rows, one per warp pass
            int64_t blocks = (groups + kG16Warps - 1) / kG16Warps;
            if (blocks > 152) blocks = 152;
            return launch_pdl(stream_g16_kernel, dim3((unsigned)blocks), dim3(kG16Warps * 32),
                              (size_t)kG16Smem, stream, a2);
        }
        const int K = args.k <= 2 ? 2 : args.k <= 4 ? 4 : args.k <= 8 ? 8 : 16;
        const int64_t pass = (int64_t)kThreads * (16 / K);
        int64_t blocks = (args.m + pass - 1) / pass;
        if (blocks > 152 * 8) blocks = 152 * 8;
        if (blocks < 1) blocks = 1;
        cudaError_t e;
        switch (K) {
            case 2: e = launch_pdl(stream_rows_kernel<2>, dim3((unsigned)blocks), dim3(kThreads), 0, stream, a2); break;
            case 4: e = launch_pdl(stream_rows_kernel<4>, dim3((unsigned)blocks), dim3(kThreads), 0, stream, a2); break;
            case 8: e = launch_pdl(stream_rows_kernel<8>, dim3((unsigned)blocks), dim3(kThreads), 0, stream, a2); break;
            default: e = launch_pdl(stream_rows_kernel<16>, dim3((unsigned)blocks), dim3(kThreads), 0, stream, a2); break;
        }
        return e;
    }
    const int64_t blocks = (args.m + args.rows_per_cta - 1) / args.rows_per_cta;
    dim3 grid((unsigned)blocks, (unsigned)args.ksplit);
    if (args.n <= 4) return launch_stream_nb<4>(args, grid, stream);
    if (args.n <= 8) return launch_stream_nb<8>(args, grid, stream);
    return launch_stream_nb<16>(args, grid, stream);
}

cudaError_t launch_splitk_reduce(const ReduceArgs &args, cudaStream_t stream) {
    const int64_t mn = args.m * args.n;
    int64_t blocks = (mn + kThreads - 1) / kThreads;
    if (blocks > 152 * 8) blocks = 152 * 8;
    return launch_pdl(splitk_reduce_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream, args);
}

}  // namespace tn
