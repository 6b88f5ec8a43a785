// Small device helpers shared by the kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"

namespace tn {

// Offset of index i under a separable output layout: split i mixed-radix
// over the runs (run 0 most significant) and sum digit * stride.
__device__ __forceinline__ int64_t sep_offset(const SepLayout &L, int64_t i) {
    int64_t off = 0;
    for (int r = L.nrun - 1; r >= 0; --r) {
        const int64_t e = L.ext[r];
        const int64_t q = i / e;
        off += (i - q * e) * L.stride[r];
        i = q;
    }
    return off;
}

__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}

__device__ __forceinline__ void cfma(float2 &acc, float2 a, float2 b) {
    acc.x = fmaf(a.x, b.x, acc.x);
    acc.x = fmaf(-a.y, b.y, acc.x);
    acc.y = fmaf(a.x, b.y, acc.y);
    acc.y = fmaf(a.y, b.x, acc.y);
}

}  // namespace tn
