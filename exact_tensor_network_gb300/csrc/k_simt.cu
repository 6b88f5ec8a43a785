// General node kernel on CUDA cores (fp32 complex FMA).
//
// Computes one pairwise step of "Crossing the single-GPU memory wall"
// (section 1.1) in the GEMM form that lifetime ordering (section 1.4) gives
// every node: A is a row-major [m, k] matrix, B a row-major [n, k] matrix,
// and output entry (i, j) = sum_k A[i, k] * B[j, k] lands at
// offM(i) + offN(j), which covers outputs whose order interleaves M and N
// modes without any transpose pass.
//
// 64 x 64 output tile per CTA, 256 threads each owning 4 x 4 complex
// accumulators (rows ty + 16r, columns tx + 16c, so that 16 lanes store 16
// consecutive columns); K staged through shared memory 16 entries at a
// time.  Any shape works (ragged edges are masked); the tensor-core and
// streaming kernels take the shapes they are faster on.
#include "common.cuh"
#include "kernels.h"

namespace tn {

namespace {

constexpr int BM = 64, BN = 64, BK = 16, TM = 4, TN = 4;
constexpr int kThreads = (BM / TM) * (BN / TN);

template <int FMT>
__global__ void __launch_bounds__(kThreads) simt_node_kernel(const __grid_constant__ NodeArgs a) {
    __shared__ float2 As[BK][BM + 1];
    __shared__ float2 Bs[BK][BN + 1];
    __shared__ int64_t offm_s[BM], offn_s[BN];   // the tile's row and column offsets
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x;
    const int tx = tid % (BN / TN), ty = tid / (BN / TN);
    const int64_t mt = (a.m + BM - 1) / BM, nt = (a.n + BN - 1) / BN;
    const int64_t tiles = mt * nt;
    const int64_t work = tiles * a.ksplit;
    for (int64_t w = blockIdx.x; w < work; w += gridDim.x) {
        const int64_t tile = w / a.ksplit;
        const int split = (int)(w - tile * a.ksplit);
        const int64_t kbeg = a.ksplit > 1 ? split * a.kchunk : 0;
        const int64_t kend = a.ksplit > 1 ? min(a.k, kbeg + a.kchunk) : a.k;
        const int64_t i0 = (tile / nt) * BM, j0 = (tile % nt) * BN;
        float2 acc[TM][TN];
#pragma unroll
        for (int r = 0; r < TM; ++r)
#pragma unroll
            for (int c = 0; c < TN; ++c) acc[r][c] = make_float2(0.f, 0.f);
        for (int64_t k0 = kbeg; k0 < kend; k0 += BK) {
            // stage A[i0:i0+BM, k0:k0+BK] and B[j0:j0+BN, k0:k0+BK]
            for (int e = tid; e < BM * BK; e += kThreads) {
                const int r = e / BK, c = e % BK;
                const int64_t i = i0 + r, kk = k0 + c;
                As[c][r] = (i < a.m && kk < kend) ? a.A[i * a.k + kk] : make_float2(0.f, 0.f);
            }
            for (int e = tid; e < BN * BK; e += kThreads) {
                const int r = e / BK, c = e % BK;
                const int64_t j = j0 + r, kk = k0 + c;
                Bs[c][r] = (j < a.n && kk < kend) ? a.B[j * a.k + kk] : make_float2(0.f, 0.f);
            }
            __syncthreads();
            // the stage's valid k entries only (small-k nodes: one short stage)
            const int kn = (int)min((int64_t)BK, kend - k0);
#pragma unroll 2
            for (int kk = 0; kk < kn; ++kk) {
                float2 av[TM], bv[TN];
#pragma unroll
                for (int r = 0; r < TM; ++r) av[r] = As[kk][ty + r * (BM / TM)];
#pragma unroll
                for (int c = 0; c < TN; ++c) bv[c] = Bs[kk][tx + c * (BN / TN)];
#pragma unroll
                for (int r = 0; r < TM; ++r)
#pragma unroll
                    for (int c = 0; c < TN; ++c) cfma(acc[r][c], av[r], bv[c]);
            }
            __syncthreads();
        }
        if (a.ksplit > 1) {
            // plain partial sums of this k range
#pragma unroll
            for (int r = 0; r < TM; ++r) {
                const int64_t i = i0 + ty + r * (BM / TM);
                if (i >= a.m) continue;
                float2 *dst = a.part + ((int64_t)split * a.m + i) * a.n;
#pragma unroll
                for (int c = 0; c < TN; ++c) {
                    const int64_t j = j0 + tx + c * (BN / TN);
                    if (j < a.n) dst[j] = acc[r][c];
                }
            }
            continue;
        }
        // separable offsets of the tile's rows and columns, once per tile
        for (int e = tid; e < BM + BN; e += kThreads) {
            if (e < BM) {
                const int64_t i = i0 + e;
                offm_s[e] = i < a.m ? sep_offset(a.lm, i) : 0;
            } else {
                const int64_t j = j0 + (e - BM);
                offn_s[e - BM] = j < a.n ? sep_offset(a.ln, j) : 0;
            }
        }
        __syncthreads();
        // rows rolled (the selects keep acc in registers): one copy of the
        // store code per column instead of one per entry
#pragma unroll 1
        for (int r = 0; r < TM; ++r) {
            const int64_t i = i0 + ty + r * (BM / TM);
            if (i >= a.m) continue;
            const int64_t offm = offm_s[ty + r * (BM / TM)];
#pragma unroll
            for (int c = 0; c < TN; ++c) {
                const int64_t j = j0 + tx + c * (BN / TN);
                if (j >= a.n) continue;
                const float2 v = r == 0 ? acc[0][c] : r == 1 ? acc[1][c] : r == 2 ? acc[2][c] : acc[3][c];
                store_entry_t<FMT>(a.C, a.m * a.n, offm + offn_s[tx + c * (BN / TN)], v, a.accumulate,
                                   a.out_tile);
            }
        }
        __syncthreads();   // the next tile rewrites the offsets
    }
}

}  // namespace

cudaError_t launch_simt_node(const NodeArgs &args, cudaStream_t stream) {
    const int64_t tiles = ((args.m + BM - 1) / BM) * ((args.n + BN - 1) / BN) * args.ksplit;
    const int64_t grid = tiles < 152 * 16 ? tiles : 152 * 16;
    if (args.out_fmt == FMT_SPLIT4)
        return launch_pdl(simt_node_kernel<FMT_SPLIT4>, dim3((unsigned)grid), dim3(kThreads), 0, stream, args);
    else if (args.out_fmt == FMT_GAUSS6)
        return launch_pdl(simt_node_kernel<FMT_GAUSS6>, dim3((unsigned)grid), dim3(kThreads), 0, stream, args);
    else if (args.out_fmt == FMT_BF2)
        return launch_pdl(simt_node_kernel<FMT_BF2>, dim3((unsigned)grid), dim3(kThreads), 0, stream, args);
    else if (args.out_fmt == FMT_BF4)
        return launch_pdl(simt_node_kernel<FMT_BF4>, dim3((unsigned)grid), dim3(kThreads), 0, stream, args);
    return launch_pdl(simt_node_kernel<FMT_C64>, dim3((unsigned)grid), dim3(kThreads), 0, stream, args);
}

}  // namespace tn
