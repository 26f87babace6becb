// Device helpers for the q8_row row-group interleaved layout (see
// qmv_internal.cuh): one 16-byte lane chunk = 4 rows x 4 int8 columns.
#pragma once

#include "qmv_internal.cuh"

namespace qmv {

// 128-bit streaming load that does not allocate in L1 (weights are read
// exactly once per call).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Asks L2 to fetch [p, p + bytes) from HBM (no data comes to the SM);
// p 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Activations are re-read by every warp: keep them in L1.  They may be the
// output of the previous kernel in the stream, which can still be running
// while this one starts (programmatic dependent launch), so they are read
// after pdl_wait() with ordinary coherent loads, never the non-coherent
// read-only path.
__device__ __forceinline__ float4 ld_act_f4(const float* p) {
    return __ldca(reinterpret_cast<const float4*>(p));
}

// Exact int8 -> f32 without the (quarter-rate) integer-to-float converter:
// flip the sign bit (two's complement -> offset binary, u = b + 128), move
// byte t into the low mantissa byte of 2^23 (bits 0x4B0000uu = 2^23 + u), and
// subtract 2^23 + 128.  Every step is exact.
__device__ __forceinline__ float2 i8pair_lo(uint32_t u) {
    return make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)),
                       __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441)));
}
__device__ __forceinline__ float2 i8pair_hi(uint32_t u) {
    return make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)),
                       __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443)));
}

// acc[r] += q[r][0..3] . x[0..3] for the 4 rows of one lane chunk.  Each row
// keeps two fp32 partial sums (a packed f32x2 pair).
__device__ __forceinline__ void q8_chunk_fma(const uint4 w, const float4 x, float2 acc[4]) {
    const float2 bias = make_float2(-8388736.0f, -8388736.0f);
    const float2 x01 = make_float2(x.x, x.y);
    const float2 x23 = make_float2(x.z, x.w);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const uint32_t u = ws[r] ^ 0x80808080u;
        const float2 v01 = __fadd2_rn(i8pair_lo(u), bias);
        const float2 v23 = __fadd2_rn(i8pair_hi(u), bias);
        acc[r] = __ffma2_rn(v01, x01, acc[r]);
        acc[r] = __ffma2_rn(v23, x23, acc[r]);
    }
}

// Activation float4 of lane `lane` for 128-column block `blk`; zero past
// `cols` (x 16-byte aligned; nothing at or past x[cols] is read).
__device__ __forceinline__ float4 act_for_block(const float* x, int64_t blk, int lane, int64_t cols) {
    const int64_t c = blk * 128 + lane * 4;
    if (c + 4 <= cols) return ld_act_f4(x + c);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < cols) v.x = __ldca(x + c);
    if (c + 1 < cols) v.y = __ldca(x + c + 1);
    if (c + 2 < cols) v.z = __ldca(x + c + 2);
    return v;
}

// Sum of a float over the 32 lanes, result in every lane.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Codes of blocks [b0, b0 + U) of row group `rg` (zero at and past b1): the
// batch a kernel loads before its dependency wait.
template <int U>
__device__ __forceinline__ void q8_first_codes(uint4 (&w)[U], const int8_t* __restrict__ qbase, int64_t cols_pad,
                                               int64_t rg, int64_t b0, int64_t b1, int lane) {
    const int8_t* p = qbase + rg * 4 * cols_pad + lane * 16;
#pragma unroll
    for (int u = 0; u < U; ++u) w[u] = b0 + u < b1 ? ld_stream_u4(p + (b0 + u) * 512) : make_uint4(0u, 0u, 0u, 0u);
}

// Dot products of the 4 rows of row group `rg` (qbase: packed codes of the
// matrix) with x over blocks [b0, b1), when the codes of [b0, b0 + U) are
// already in w0 (from q8_first_codes; zero codes contribute exactly 0).
// Returns the 4 per-lane partials.
template <int U>
__device__ __forceinline__ void q8_rowgroup_dot_from(const uint4 (&w0)[U], const int8_t* __restrict__ qbase,
                                                     int64_t cols_pad, int64_t rg, int64_t b0, int64_t b1,
                                                     const float* __restrict__ x, int64_t cols, int lane,
                                                     float out[4]) {
    float2 acc[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[r] = make_float2(0.f, 0.f);
    {
        float4 xv[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            xv[u] = b0 + u < b1 ? act_for_block(x, b0 + u, lane, cols) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < U; ++u) q8_chunk_fma(w0[u], xv[u], acc);
    }
    const int8_t* p = qbase + rg * 4 * cols_pad + lane * 16;
    int64_t b = b0 + U;
    for (; b + U <= b1; b += U) {
        uint4 w[U];
        float4 xv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) w[u] = ld_stream_u4(p + (b + u) * 512);
#pragma unroll
        for (int u = 0; u < U; ++u) xv[u] = act_for_block(x, b + u, lane, cols);
#pragma unroll
        for (int u = 0; u < U; ++u) q8_chunk_fma(w[u], xv[u], acc);
    }
    for (; b < b1; ++b) {
        const uint4 w = ld_stream_u4(p + b * 512);
        q8_chunk_fma(w, act_for_block(x, b, lane, cols), acc);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) out[r] = acc[r].x + acc[r].y;
}

}  // namespace qmv
