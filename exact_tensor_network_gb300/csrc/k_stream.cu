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
