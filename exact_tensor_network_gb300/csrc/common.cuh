// Small device helpers shared by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"

namespace tn {

// Offset of index i under a separable output layout: split i mixed-radix
// over the runs (run 0 most significant) and sum digit * stride.
// Power-of-two extents use shifts and masks; other extents divide (32-bit
// when the index fits, which avoids the slow 64-bit division).
__device__ __forceinline__ int64_t sep_offset(const SepLayout &L, int64_t i) {
    int64_t off = 0;
    for (int r = L.nrun - 1; r >= 0; --r) {
        const int64_t e = L.ext[r];
        int64_t d;
        if (L.shift[r] >= 0) {
            d = i & (e - 1);
            i >>= L.shift[r];
        } else if (i < 0x7fffffff && e < 0x7fffffff) {
            const uint32_t q = static_cast<uint32_t>(i) / static_cast<uint32_t>(e);
            d = i - static_cast<int64_t>(q) * e;
            i = q;
        } else {
            const int64_t q = i / e;
            d = i - q * e;
            i = q;
        }
        off += d * L.stride[r];
    }
    return off;
}

// x rounded to tf32 (10-bit mantissa, round to nearest, ties away), as fp32.
__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Store entry `off` of a tensor in the compile-time format FMT (see Fmt in
// plan.h); planes are `plane` entries apart.  `accumulate` adds into a C64
// destination.  Kernels instantiated per format keep one store path.
// Physical index of row-major index `off` in a K-tiled planar operand (see
// PlanarTile in plan.h).
__device__ __forceinline__ int64_t tiled_offset(const PlanarTile &t, int64_t off) {
    if (t.kt == 0) return off;
    int64_t r, c;
    if (t.kshift >= 0) {
        r = off >> t.kshift;
        c = off & (t.k - 1);
    } else {
        r = off / t.k;
        c = off - r * t.k;
    }
    const int sh = t.kt == 32 ? 5 : 4;
    return (((c >> sh) * t.rows + r) << sh) + (c & (t.kt - 1));
}

template <int FMT>
__device__ __forceinline__ void store_entry_t(void *dst, int64_t plane, int64_t off, float2 v,
                                              int32_t accumulate, const PlanarTile &tile) {
    if constexpr (FMT != FMT_C64) off = tiled_offset(tile, off);
    if constexpr (FMT == FMT_C64) {
        float2 *p = static_cast<float2 *>(dst) + off;
        if (accumulate) {
            const float2 o = *p;
            v.x += o.x;
            v.y += o.y;
        }
        *p = v;
    } else if constexpr (FMT == FMT_SPLIT4) {
        float *p = static_cast<float *>(dst) + off;
        const float rh = to_tf32(v.x), ih = to_tf32(v.y);
        p[0] = rh;
        p[plane] = ih;
        p[2 * plane] = to_tf32(v.x - rh);
        p[3 * plane] = to_tf32(v.y - ih);
    } else {
        __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(dst) + off;
        p[0] = __float2bfloat16_rn(v.x);
        p[plane] = __float2bfloat16_rn(v.y);
    }
}

// Same with the format chosen at run time.
__device__ __forceinline__ void store_entry(void *dst, int32_t fmt, int64_t plane, int64_t off,
                                            float2 v, int32_t accumulate, const PlanarTile &tile) {
    if (fmt != FMT_C64) off = tiled_offset(tile, off);
    if (fmt == FMT_C64) {
        float2 *p = static_cast<float2 *>(dst) + off;
        if (accumulate) {
            const float2 o = *p;
            v.x += o.x;
            v.y += o.y;
        }
        *p = v;
    } else if (fmt == FMT_SPLIT4) {
        float *p = static_cast<float *>(dst) + off;
        const float rh = to_tf32(v.x), ih = to_tf32(v.y);
        p[0] = rh;
        p[plane] = ih;
        p[2 * plane] = to_tf32(v.x - rh);
        p[3 * plane] = to_tf32(v.y - ih);
    } else {
        __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(dst) + off;
        p[0] = __float2bfloat16_rn(v.x);
        p[plane] = __float2bfloat16_rn(v.y);
    }
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
