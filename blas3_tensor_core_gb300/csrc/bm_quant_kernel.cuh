// bm_quant_kernel.cuh -- BF16 -> MXFP8 quantization for sm_103a: E4M3 codes plus
// one UE8M0 scale per group of 32 consecutive elements of a row, the scales
// written in the tiled atom layout that the block-scaled GEMM reads.
//
// This is the "W quantize BF16 -> MXFP8" step of the SM103 MXFP8 path in "fused
// A2A/GEMM Perfetto profile protocol" (per group of 32: read BF16, amax
// reduction, UE8M0 scale, E4M3 conversion, write). The page names the steps;
// the conversion rule is the OCP Microscaling (MX) v1.0 one: shared exponent
// e = floor(log2(amax)) - 8 (8 being the largest E4M3 exponent), clamped to
// [-127, 127]; scale code e + 127; each element is X / 2^e rounded to the
// nearest E4M3 value, ties to even, with magnitudes beyond 448 saturated to
// 448. A group of zeros gets code 0; a group holding a NaN or an infinity gets
// code 255 (NaN) and NaN elements.
//
// The work is HBM-bound (2 bytes read and about 1.03 written per element): one
// thread per group reads its 64 bytes with four 16-byte loads, consecutive
// threads take consecutive groups of a row, and the grid strides over the
// groups, padding entries of the scale array included.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

#include "bm_ptx.cuh"

namespace bm {

struct QuantParams {
    int64_t rows, k;
    const uint16_t *X;  // bf16 bits, row-major, leading dimension ldx
    int64_t ldx;
    uint8_t *Q;         // E4M3 codes, row-major, leading dimension ldq
    int64_t ldq;
    uint8_t *S;         // UE8M0 codes, tiled: ceil(rows / 128) x ceil(k / 128) atoms of 512 bytes
    int64_t groups;     // ceil(k / 32): groups of a row
    int64_t groups_pad; // 4 * ceil(k / 128): groups of a row in the scale array, padding included
    int64_t rows_pad;   // 128 * ceil(rows / 128)
};

// Byte of the scale of row r, group g in the tiled layout.
__device__ __forceinline__ int64_t scale_offset(int64_t r, int64_t g, int64_t groups_pad)
{
    return ((r >> 7) * (groups_pad >> 2) + (g >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (g & 3);
}

// Scale code of a group from the bits of its (finite) amax: for a normal amax with
// exponent field f, floor(log2(amax)) = f - 127, so the code e + 127 is f - 8;
// zero and subnormal amax (f = 0) and any f < 8 clamp to code 0.
__device__ __forceinline__ uint32_t ue8m0_code(float amax)
{
    const int f = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
    return f > 8 ? static_cast<uint32_t>(f - 8) : 0u;
}

// Four E4M3 codes from four values (already divided by the scale), rounded to
// nearest even, saturating at +-448.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d)
{
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__global__ void __launch_bounds__(256) bm_quantize_mxfp8_kernel(const QuantParams p)
{
    griddep_launch_dependents();
    griddep_wait();
    const int64_t total = p.rows_pad * p.groups_pad;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = idx / p.groups_pad;
        const int64_t g = idx - r * p.groups_pad;
        uint8_t *s_at = p.S + scale_offset(r, g, p.groups_pad);
        if (r >= p.rows || g >= p.groups) {  // padding of the scale array
            *s_at = 0;
            continue;
        }
        const int64_t p0 = 32 * g;
        const int n = p.k - p0 < 32 ? static_cast<int>(p.k - p0) : 32;
        const uint16_t *src = p.X + r * p.ldx + p0;
        float v[32];
        if (n == 32) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 w = __ldg(reinterpret_cast<const uint4 *>(src) + q);
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    v[8 * q + 2 * e] = __uint_as_float(u[e] << 16);
                    v[8 * q + 2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
                }
            }
        } else {  // the short last group of a row: elements past k count as zeros and are not written
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = e < n ? __uint_as_float(static_cast<uint32_t>(src[e]) << 16) : 0.0f;
        }
        float amax = 0.0f;
        bool special = false;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const float a = fabsf(v[e]);
            special |= !(a <= 3.402823466e38f);  // NaN or infinity
            amax = fmaxf(amax, a);
        }
        uint32_t code = special ? 255u : ue8m0_code(amax);
        *s_at = static_cast<uint8_t>(code);
        uint32_t out[8];
        if (special) {
#pragma unroll
            for (int q = 0; q < 8; ++q) out[q] = 0x7F7F7F7Fu;
        } else {
            // 1 / 2^e = 2^(127 - code): exponent field 254 - code, in [8, 254] (code <= 246)
            const float inv = __uint_as_float((254u - code) << 23);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                out[q] = e4m3x4(v[4 * q] * inv, v[4 * q + 1] * inv, v[4 * q + 2] * inv, v[4 * q + 3] * inv);
        }
        uint8_t *dst = p.Q + r * p.ldq + p0;
        if (n == 32) {
            reinterpret_cast<uint4 *>(dst)[0] = make_uint4(out[0], out[1], out[2], out[3]);
            reinterpret_cast<uint4 *>(dst)[1] = make_uint4(out[4], out[5], out[6], out[7]);
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (e < n) dst[e] = static_cast<uint8_t>(out[e >> 2] >> (8 * (e & 3)));
        }
    }
}

}  // namespace bm
