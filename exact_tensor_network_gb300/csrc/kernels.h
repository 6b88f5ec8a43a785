// Launchers of the device kernels and the small structs they take by value.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"

namespace tn {

// Device status word layout at the start of the workspace.
enum : int32_t { ERR_NONE = 0, ERR_DESC = 1, ERR_TIMEOUT = 2 };
struct DevStatus {
    int32_t code;      // first error seen (ERR_*), 0 if none
    int32_t where;     // kernel-specific detail
};

// One GEMM-shaped node: C[offM(i) + offN(j)] (+)= sum_k A[i*k + kk] * B[j*k + kk].
struct NodeArgs {
    const float2 *A;
    const float2 *B;
    float2 *C;
    int64_t m, n, k;
    SepLayout lm, ln;
    int32_t accumulate;   // 1: add into C (later slices of the root)
    int32_t precision;
    DevStatus *status;
};

constexpr int kPermBatch = 512;   // permutation jobs per launch

struct PermLaunch {
    int32_t njobs;
    int32_t accumulate;
    const PermDesc *table;          // device table (workspace)
    char *arena;                    // workspace arena
    float2 *out;
    int32_t job[kPermBatch];        // table index of job j
    int32_t cta_start[kPermBatch + 1];
    const float2 *src[kPermBatch];  // slice-shifted source pointers
};

cudaError_t launch_permute(const PermLaunch &args, int total_ctas, cudaStream_t stream);
cudaError_t launch_simt_node(const NodeArgs &args, cudaStream_t stream);

// CTAs a permutation job of `size` elements gets.
int permute_ctas(int64_t size);

}  // namespace tn
