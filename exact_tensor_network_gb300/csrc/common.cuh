// Small device helpers shared by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"

namespace tn {

// Programmatic dependent launch.  Every kernel is launched with programmatic
// stream serialization (launch_pdl), signals at its start that the next
// kernel on the stream may be scheduled (its CTAs then wait on the SMs this
// grid leaves free), and waits before its first global memory access until
// the previous grid has completed and its writes are visible.  The wait is a
// hardware dependency (no spin); a dependent grid is only launched once every
// CTA of this grid has started, so waiting CTAs never starve this grid.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Offset of index i under a separable output layout: split i mixed-radix
// over the runs (run 0 most significant) and sum digit * stride.
// Power-of-two extents use shifts and masks; other extents divide (32-bit
// when the index fits, which avoids the slow 64-bit division).
__device__ __forceinline__ int64_t sep_offset(const SepLayout &L, int64_t i) {
    int64_t off = 0;
    // rolled: inlined at many call sites, an unrolled copy per site would
    // swell the kernels' code (and their instruction-cache misses)
#pragma unroll 1
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

// One entry in FMT_GAUSS6 (see Fmt in plan.h): re, im and s = re + im, each
// as tf32 hi and lo, planes `plane` entries apart.
__device__ __forceinline__ void store_gauss6(float *p, int64_t plane, float2 v) {
    const float sum = v.x + v.y;
    const float rh = to_tf32(v.x), ih = to_tf32(v.y), sh = to_tf32(sum);
    p[0] = rh;
    p[plane] = ih;
    p[2 * plane] = sh;
    p[3 * plane] = to_tf32(v.x - rh);
    p[4 * plane] = to_tf32(v.y - ih);
    p[5 * plane] = to_tf32(sum - sh);
}

// x as a bf16 pair: hi = x rounded to bf16, lo = (x - hi) rounded to bf16
// (x - hi is exact in fp32).
__device__ __forceinline__ void bf16_split(float x, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

__device__ __forceinline__ void store_bf4(__nv_bfloat16 *p, int64_t plane, float2 v) {
    __nv_bfloat16 rh, rl, ih, il;
    bf16_split(v.x, rh, rl);
    bf16_split(v.y, ih, il);
    p[0] = rh;
    p[plane] = ih;
    p[2 * plane] = rl;
    p[3 * plane] = il;
}

// Store entry `off` of a tensor in the compile-time format FMT (see Fmt in
// plan.h); planes are `plane` entries apart.  `accumulate` adds into a C64
// destination.  Kernels instantiated per format keep one store path.
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
    } else if constexpr (FMT == FMT_GAUSS6) {
        store_gauss6(static_cast<float *>(dst) + off, plane, v);
    } else if constexpr (FMT == FMT_BF4) {
        store_bf4(static_cast<__nv_bfloat16 *>(dst) + off, plane, v);
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
    } else if (fmt == FMT_GAUSS6) {
        store_gauss6(static_cast<float *>(dst) + off, plane, v);
    } else if (fmt == FMT_BF4) {
        store_bf4(static_cast<__nv_bfloat16 *>(dst) + off, plane, v);
    } else {
        __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(dst) + off;
        p[0] = __float2bfloat16_rn(v.x);
        p[plane] = __float2bfloat16_rn(v.y);
    }
}

// Four entries at offsets off .. off + 3 (off a multiple of 4, planes a
// multiple of 4 entries apart, dst 16-byte aligned): the conversions of
// store_entry, then one 16-byte store per plane (8 bytes per bf16 plane).
// K-tiling keeps such a run contiguous because tiles hold 16 or 32 entries.
__device__ __forceinline__ void store_quad(void *dst, int32_t fmt, int64_t plane, int64_t off,
                                           const float2 (&v)[4], int32_t accumulate,
                                           const PlanarTile &tile) {
    if (fmt != FMT_C64) off = tiled_offset(tile, off);
    if (fmt == FMT_C64) {
        float4 *p = reinterpret_cast<float4 *>(static_cast<float2 *>(dst) + off);
        float4 x0 = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
        float4 x1 = make_float4(v[2].x, v[2].y, v[3].x, v[3].y);
        if (accumulate) {
            const float4 o0 = p[0], o1 = p[1];
            x0.x += o0.x; x0.y += o0.y; x0.z += o0.z; x0.w += o0.w;
            x1.x += o1.x; x1.y += o1.y; x1.z += o1.z; x1.w += o1.w;
        }
        p[0] = x0;
        p[1] = x1;
    } else if (fmt == FMT_SPLIT4) {
        float *p = static_cast<float *>(dst) + off;
        float rh[4], ih[4], rl[4], il[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            rh[t] = to_tf32(v[t].x);
            ih[t] = to_tf32(v[t].y);
            rl[t] = to_tf32(v[t].x - rh[t]);
            il[t] = to_tf32(v[t].y - ih[t]);
        }
        *reinterpret_cast<float4 *>(p) = make_float4(rh[0], rh[1], rh[2], rh[3]);
        *reinterpret_cast<float4 *>(p + plane) = make_float4(ih[0], ih[1], ih[2], ih[3]);
        *reinterpret_cast<float4 *>(p + 2 * plane) = make_float4(rl[0], rl[1], rl[2], rl[3]);
        *reinterpret_cast<float4 *>(p + 3 * plane) = make_float4(il[0], il[1], il[2], il[3]);
    } else if (fmt == FMT_GAUSS6) {
        float *p = static_cast<float *>(dst) + off;
        float q[6][4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float sum = v[t].x + v[t].y;
            q[0][t] = to_tf32(v[t].x);
            q[1][t] = to_tf32(v[t].y);
            q[2][t] = to_tf32(sum);
            q[3][t] = to_tf32(v[t].x - q[0][t]);
            q[4][t] = to_tf32(v[t].y - q[1][t]);
            q[5][t] = to_tf32(sum - q[2][t]);
        }
#pragma unroll
        for (int c = 0; c < 6; ++c)
            *reinterpret_cast<float4 *>(p + c * plane) = make_float4(q[c][0], q[c][1], q[c][2], q[c][3]);
    } else if (fmt == FMT_BF4) {
        // planes re_hi, im_hi, re_lo, im_lo: four bf16 (8 bytes) each
        __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(dst) + off;
        __nv_bfloat16 q[4][4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            bf16_split(v[t].x, q[0][t], q[2][t]);
            bf16_split(v[t].y, q[1][t], q[3][t]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const __nv_bfloat162 x0 = __halves2bfloat162(q[c][0], q[c][1]);
            const __nv_bfloat162 x1 = __halves2bfloat162(q[c][2], q[c][3]);
            uint2 w;
            w.x = *reinterpret_cast<const uint32_t *>(&x0);
            w.y = *reinterpret_cast<const uint32_t *>(&x1);
            *reinterpret_cast<uint2 *>(p + c * plane) = w;
        }
    } else {
        __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(dst) + off;
        __nv_bfloat162 re0 = __halves2bfloat162(__float2bfloat16_rn(v[0].x), __float2bfloat16_rn(v[1].x));
        __nv_bfloat162 re1 = __halves2bfloat162(__float2bfloat16_rn(v[2].x), __float2bfloat16_rn(v[3].x));
        __nv_bfloat162 im0 = __halves2bfloat162(__float2bfloat16_rn(v[0].y), __float2bfloat16_rn(v[1].y));
        __nv_bfloat162 im1 = __halves2bfloat162(__float2bfloat16_rn(v[2].y), __float2bfloat16_rn(v[3].y));
        uint2 re, im;
        re.x = *reinterpret_cast<uint32_t *>(&re0);
        re.y = *reinterpret_cast<uint32_t *>(&re1);
        im.x = *reinterpret_cast<uint32_t *>(&im0);
        im.y = *reinterpret_cast<uint32_t *>(&im1);
        *reinterpret_cast<uint2 *>(p) = re;
        *reinterpret_cast<uint2 *>(p + plane) = im;
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
