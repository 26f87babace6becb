// Q2 (2-bit, g64 / g128) decode GEMV:
//   y[m] = sum_g d[m,g] * sum_{k in g} (q[m,k] - 1) * x[k]
//
// qxmx_gpu.cpp, `gemv_dpas8` (8-row DPAS tiles, split-K over the K groups,
// per-group scale FMA in f32) and `gemv_reduce` are the prior art.  On
// sm_103a the 2-bit decode, not the multiply, is the cost: at the HBM roofline
// the GPU must retire ~2e13 weights/s, under two issue slots per weight.  So
// the multiply-add goes to the tensor cores (mma.sync m16n8k16, bf16 in, fp32
// accumulate) and the decode is two ALU ops per pair of weights:
//   * codes are repacked at load time into the MMA A-fragment order;
//   * one LOP3 ORs a pair of codes into the mantissas of two bf16 1.0s,
//     giving 1 + q*2^(p-7); one bf16x2 FMA maps that to q - 1 exactly;
//   * the activation x is split exactly into three bf16 parts
//     (x = hi + mid + lo, 24 significant bits) that form B columns 0..2, so
//     (q-1)*x is formed without rounding and summed in fp32;
//   * the per-group scale d (f16 -> f32, exact) multiplies the fp32 group sum.
// The persistent kernel (q2_gemv_v3_kernel) halves the decode again: one AND
// per pair of weights leaves q * 2^(p-133) as an exact bf16 subnormal, x
// enters as three base-256 digits on a common grid so that every group sum
// the tensor core forms is exact, and the bias -sum(x) of each group is added
// in fp32 from the digit sums (exact where all weights of a group are 0).
// The K range is split across the warps of a CTA; partial sums are reduced
// in shared memory in a fixed order (deterministic).  The persistent kernel
// is a programmatic dependent launch: its producer warp starts fetching the
// constant codes and scales while the previous kernel in the stream is still
// running, and the consumers wait for that kernel before reading x.
#include "tma_util.cuh"

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kBLanes = 12;   // lanes 0..11 carry the three activation parts

__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// (a & b) | c as one LOP3.  Written out because the compiler, left to
// itself, did not fuse the mask and the OR of the decode below (the explicit
// form made the persistent Q2 kernel 14 % faster).
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// Decodes one packed word (16 codes) into the 8 bf16x2 A registers of two
// consecutive k-steps.  Register t holds the codes at bits 2t and 2t+16.
// Constants: bf16 pairs of (2^(7-p), -(2^(7-p)+1)) for p = 0, 2, 4.
__device__ __forceinline__ void q2_decode_word(uint32_t w, uint32_t a[8]) {
    const uint32_t one = 0x3F803F80u;              // bf16 1.0, 1.0
    const uint32_t m0 = 0x00030003u, m2 = 0x000C000Cu, m4 = 0x00300030u;
    const uint32_t s0 = 0x43004300u, c0 = 0xC301C301u;  //  128, -129
    const uint32_t s2 = 0x42004200u, c2 = 0xC204C204u;  //   32,  -33
    const uint32_t s4 = 0x41004100u, c4 = 0xC110C110u;  //    8,   -9
    const uint32_t w6 = w >> 6, w12 = w >> 12;
    a[0] = bf16x2_fma(and_or(w, m0, one), s0, c0);
    a[1] = bf16x2_fma(and_or(w, m2, one), s2, c2);
    a[2] = bf16x2_fma(and_or(w, m4, one), s4, c4);
    a[3] = bf16x2_fma(and_or(w6, m0, one), s0, c0);
    a[4] = bf16x2_fma(and_or(w6, m2, one), s2, c2);
    a[5] = bf16x2_fma(and_or(w6, m4, one), s4, c4);
    a[6] = bf16x2_fma(and_or(w12, m0, one), s0, c0);
    a[7] = bf16x2_fma(and_or(w12, m2, one), s2, c2);
}

__device__ __forceinline__ void mma_bf16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint2 b) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y));
}

// x = hi + mid + lo exactly, each part a bf16 (round to nearest even).
__device__ __forceinline__ void split3(float x, __nv_bfloat16& hi, __nv_bfloat16& mid, __nv_bfloat16& lo) {
    hi = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(hi);
    mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    lo = __float2bfloat16_rn(r2);
}

__device__ __forceinline__ uint32_t pack_bf16x2(__nv_bfloat16 lo, __nv_bfloat16 hi) {
    return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

// Decode for the persistent kernel: the right shifts run as IMAD.HI on the
// FMA pipe (multipliers 2^26 and 2^20 arrive as kernel arguments, so they
// are not folded back into shifts), leaving the ALU pipe -- half the issue
// rate on this part -- to the eight LOP3s.  Same output as q2_decode_word.
__device__ __forceinline__ void q2_decode_word_hi(uint32_t w, uint32_t mul6, uint32_t mul12, uint32_t a[8]) {
    const uint32_t one = 0x3F803F80u;
    const uint32_t m0 = 0x00030003u, m2 = 0x000C000Cu, m4 = 0x00300030u;
    const uint32_t s0 = 0x43004300u, c0 = 0xC301C301u;
    const uint32_t s2 = 0x42004200u, c2 = 0xC204C204u;
    const uint32_t s4 = 0x41004100u, c4 = 0xC110C110u;
    const uint32_t w6 = __umulhi(w, mul6), w12 = __umulhi(w, mul12);
    a[0] = bf16x2_fma(and_or(w, m0, one), s0, c0);
    a[1] = bf16x2_fma(and_or(w, m2, one), s2, c2);
    a[2] = bf16x2_fma(and_or(w, m4, one), s4, c4);
    a[3] = bf16x2_fma(and_or(w6, m0, one), s0, c0);
    a[4] = bf16x2_fma(and_or(w6, m2, one), s2, c2);
    a[5] = bf16x2_fma(and_or(w6, m4, one), s4, c4);
    a[6] = bf16x2_fma(and_or(w12, m0, one), s0, c0);
    a[7] = bf16x2_fma(and_or(w12, m2, one), s2, c2);
}

// MMA with a zero accumulator input (first k-step of a group).
__device__ __forceinline__ void mma_bf16_z(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
    const float z = 0.f;
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}
__device__ __forceinline__ void mma_bf16_acc(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Both tiles of a pair for one 128-column chunk.  bq: the lane's activation
// fragments of the chunk's 8 k-steps ({step 2i, step 2i+1} in bq[i]); sa/sb:
// the raw f16 scales of the two tiles for this lane's rows.
template <int G>
__device__ __forceinline__ void q2_pair_chunk(const uint4 wa, const uint4 wb, const uint4 bq[4], uint32_t sa,
                                              uint32_t sb, uint32_t sa2, uint32_t sb2, bool two, uint32_t mul6,
                                              uint32_t mul12, float acc[2][2]) {
    // scales: G=64: sa = (row r: g0, g1), sa2 = (row r+8: g0, g1); G=128: sa = (row r, row r+8)
    float2 fa, fb, fa2, fb2;
    if (G == 64) {
        fa = __half22float2(*reinterpret_cast<const __half2*>(&sa));
        fa2 = __half22float2(*reinterpret_cast<const __half2*>(&sa2));
        fb = __half22float2(*reinterpret_cast<const __half2*>(&sb));
        fb2 = __half22float2(*reinterpret_cast<const __half2*>(&sb2));
    } else {
        fa = __half22float2(*reinterpret_cast<const __half2*>(&sa));
        fb = __half22float2(*reinterpret_cast<const __half2*>(&sb));
        fa2 = fa;
        fb2 = fb;
    }
    const uint32_t wsa[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t wsb[4] = {wb.x, wb.y, wb.z, wb.w};
    float ca[4], cb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t a[8];
        q2_decode_word_hi(wsa[j], mul6, mul12, a);
        const bool first = (G == 64) ? ((j & 1) == 0) : (j == 0);
        if (first) mma_bf16_z(ca, a[0], a[1], a[2], a[3], bq[j].x, bq[j].y);
        else mma_bf16_acc(ca, a[0], a[1], a[2], a[3], bq[j].x, bq[j].y);
        mma_bf16_acc(ca, a[4], a[5], a[6], a[7], bq[j].z, bq[j].w);
        if (two) {
            uint32_t b[8];
            q2_decode_word_hi(wsb[j], mul6, mul12, b);
            if (first) mma_bf16_z(cb, b[0], b[1], b[2], b[3], bq[j].x, bq[j].y);
            else mma_bf16_acc(cb, b[0], b[1], b[2], b[3], bq[j].x, bq[j].y);
            mma_bf16_acc(cb, b[4], b[5], b[6], b[7], bq[j].z, bq[j].w);
        }
        if ((G == 64 && (j & 1)) || (G == 128 && j == 3)) {
            const bool g1 = G == 64 && j == 3;
            // rows r (c0: hi, c1: mid/lo parts) and r+8 (c2, c3)
            acc[0][0] = fmaf(g1 ? fa.y : fa.x, ca[0] + ca[1], acc[0][0]);
            acc[0][1] = fmaf(G == 64 ? (g1 ? fa2.y : fa2.x) : fa.y, ca[2] + ca[3], acc[0][1]);
            if (two) {
                acc[1][0] = fmaf(g1 ? fb.y : fb.x, cb[0] + cb[1], acc[1][0]);
                acc[1][1] = fmaf(G == 64 ? (g1 ? fb2.y : fb2.x) : fb.y, cb[2] + cb[3], acc[1][1]);
            }
        }
    }
}

// Decode for the persistent kernel: the code bits are moved into the low
// mantissa bits of a zero-exponent bf16, which is the subnormal (or, for
// bit 7, the smallest normal) number q * 2^(p-133) -- exactly, because
// bf16 values below 2^-125 are evenly spaced at 2^-133.  One AND per pair
// of weights and one shift per word, no bias FMA; the bias (q - 1) is
// applied per group in fp32 (see q2_gemv_v3_kernel).  Register t takes the
// codes at bits 2t and 2t+16 as before, so p = 0, 2, 4, 6 for the four
// A registers of a k-step: row r gets p = 0 (columns 0-7 of the step) and
// 4 (columns 8-15), row r+8 gets 2 and 6.  The activation for columns 8-15
// is pre-scaled by 2^-4, so every product carries the same factor, times
// 4 on rows r+8.
__device__ __forceinline__ void q2_decode_word_sub(uint32_t w, uint32_t a[8]) {
    const uint32_t w8 = w >> 8;
    a[0] = w & 0x00030003u;
    a[1] = w & 0x000C000Cu;
    a[2] = w & 0x00300030u;
    a[3] = w & 0x00C000C0u;
    a[4] = w8 & 0x00030003u;
    a[5] = w8 & 0x000C000Cu;
    a[6] = w8 & 0x00300030u;
    a[7] = w8 & 0x00C000C0u;
}

// One 16-row tile x 128-column chunk from shared memory: 8 MMA k-steps with
// zero-initialised group accumulators, d applied per group in fp32.
// bq: the lane's activation fragments for the chunk ({step 2i, 2i+1} in
// bq[i]); s01/s23: the lane's raw f16 scales (G=64: (row r: g0, g1) and
// (row r+8: g0, g1); G=128: s01 = (row r, row r+8)); kk: the lane's bias
// terms of the chunk's groups (G=64: g0, g1; G=128: .x).  The MMA sums are
// exact (see q2_gemv_v3_kernel), so adding kk to the rounded column-pair
// sum cancels exactly where the weights are all zero.
template <int G>
__device__ __forceinline__ void q2_tile_chunk_v3(const uint4 w, const uint4 bq[4], uint32_t s01, uint32_t s23,
                                                 float2 kk, float acc[2]) {
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&s01));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&s23));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    float c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t a[8];
        q2_decode_word_sub(ws[j], a);
        const bool first = (G == 64) ? ((j & 1) == 0) : (j == 0);
        if (first) mma_bf16_z(c, a[0], a[1], a[2], a[3], bq[j].x, bq[j].y);
        else mma_bf16_acc(c, a[0], a[1], a[2], a[3], bq[j].x, bq[j].y);
        mma_bf16_acc(c, a[4], a[5], a[6], a[7], bq[j].z, bq[j].w);
        if (G == 64 && (j & 1)) {
            const bool g1 = j == 3;
            const float k = g1 ? kk.y : kk.x;
            acc[0] = fmaf(g1 ? f01.y : f01.x, (c[0] + c[1]) + k, acc[0]);
            acc[1] = fmaf(g1 ? f23.y : f23.x, fmaf(4.f, k, c[2] + c[3]), acc[1]);
        } else if (G == 128 && j == 3) {
            acc[0] = fmaf(f01.x, (c[0] + c[1]) + kk.x, acc[0]);
            acc[1] = fmaf(f01.y, fmaf(4.f, kk.x, c[2] + c[3]), acc[1]);
        }
    }
}

// Per-(tile, chunk) scale fetch: G=64 -> 4 f16 (2 row halves x 2 groups),
// G=128 -> 2 f16 (2 row halves).
template <int G> struct Scales;
template <> struct Scales<64> {
    uint2 v;
    __device__ __forceinline__ void load(const __half* d, int64_t tc, int lane) {
        v = __ldg(reinterpret_cast<const uint2*>(d + tc * 32) + (lane >> 2));
    }
    __device__ __forceinline__ void load_shared(const __half* p, int lane) {
        v = reinterpret_cast<const uint2*>(p)[lane >> 2];
    }
    __device__ __forceinline__ float get(int rhi, int gi) const {
        const uint32_t u = rhi ? v.y : v.x;
        return __half2float(__ushort_as_half((unsigned short)(gi ? (u >> 16) : (u & 0xffffu))));
    }
};
template <> struct Scales<128> {
    uint32_t v;
    __device__ __forceinline__ void load(const __half* d, int64_t tc, int lane) {
        v = __ldg(reinterpret_cast<const uint32_t*>(d + tc * 16) + (lane >> 2));
    }
    __device__ __forceinline__ void load_shared(const __half* p, int lane) {
        v = reinterpret_cast<const uint32_t*>(p)[lane >> 2];
    }
    __device__ __forceinline__ float get(int rhi, int) const {
        return __half2float(__ushort_as_half((unsigned short)(rhi ? (v >> 16) : (v & 0xffffu))));
    }
};

// One 16-row tile x 128-column chunk: 8 MMA k-steps, d applied per group.
template <int G>
__device__ __forceinline__ void q2_tile_chunk(const uint4 w, const Scales<G>& sc, const uint2* bfrag,
                                              int lane, float acc[2]) {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t a[8];
        q2_decode_word(ws[j], a);
        const uint2 b0 = lane < kBLanes ? bfrag[(2 * j) * kBLanes + lane] : make_uint2(0u, 0u);
        const uint2 b1 = lane < kBLanes ? bfrag[(2 * j + 1) * kBLanes + lane] : make_uint2(0u, 0u);
        mma_bf16(c, a[0], a[1], a[2], a[3], b0);
        mma_bf16(c, a[4], a[5], a[6], a[7], b1);
        if ((G == 64 && (j & 1)) || (G == 128 && j == 3)) {
            const int gi = G == 64 ? (j >> 1) : 0;
            acc[0] = fmaf(sc.get(0, gi), c[0] + c[1], acc[0]);
            acc[1] = fmaf(sc.get(1, gi), c[2] + c[3], acc[1]);
            c[0] = c[1] = c[2] = c[3] = 0.f;
        }
    }
}

// CTA: kWarps warps = (kWarps/S) tile pairs x S K-splits; persistent over
// units of (kWarps/S) tile pairs.  Dynamic shared memory: B fragments for all
// k-steps ([KC*8][12] uint2), then the split-K partials.
template <int G>
__global__ void __launch_bounds__(kThreads) q2_gemv_kernel(const uint4* __restrict__ codes,
                                                          const __half* __restrict__ d,
                                                          const float* __restrict__ x, float* __restrict__ y,
                                                          int64_t rows, int64_t cols, int KC, int S,
                                                          int64_t n_units) {
    extern __shared__ uint2 smem[];
    uint2* bfrag = smem;
    float* part = reinterpret_cast<float*>(smem + (size_t)KC * 8 * kBLanes);
    const int nsteps = KC * 8;
    for (int idx = threadIdx.x; idx < nsteps * kBLanes; idx += kThreads) {
        const int s = idx / kBLanes, l = idx % kBLanes;
        const int part_id = l >> 2, kq = l & 3;
        const int64_t k0 = 16 * (int64_t)s + 2 * kq;
        const int64_t ks[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
        __nv_bfloat16 p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float xv = ks[e] < cols ? x[ks[e]] : 0.f;
            __nv_bfloat16 hi, mid, lo;
            split3(xv, hi, mid, lo);
            p[e] = part_id == 0 ? hi : part_id == 1 ? mid : lo;
        }
        bfrag[idx] = make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]));
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int tpc = kWarps / S;          // tile pairs per unit
    const int ksplit = warp % S;
    const int tpl = warp / S;
    const int kc0 = KC * ksplit / S, kc1 = KC * (ksplit + 1) / S;

    for (int64_t unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
        const int64_t rt0 = (unit * tpc + tpl) * 2;   // first of the warp's two 16-row tiles
        float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        if (rt0 * 16 < rows) {
            const uint4* pa = codes + (rt0 * KC) * 32 + lane;
            const uint4* pb = codes + ((rt0 + 1) * KC) * 32 + lane;
            uint4 wa = ld_stream_u4(pa + (int64_t)kc0 * 32);
            uint4 wb = ld_stream_u4(pb + (int64_t)kc0 * 32);
            Scales<G> sa, sb;
            sa.load(d, rt0 * KC + kc0, lane);
            sb.load(d, (rt0 + 1) * KC + kc0, lane);
            for (int kc = kc0; kc < kc1; ++kc) {
                uint4 na = wa, nb = wb;
                Scales<G> nsa = sa, nsb = sb;
                if (kc + 1 < kc1) {
                    na = ld_stream_u4(pa + (int64_t)(kc + 1) * 32);
                    nb = ld_stream_u4(pb + (int64_t)(kc + 1) * 32);
                    nsa.load(d, rt0 * KC + kc + 1, lane);
                    nsb.load(d, (rt0 + 1) * KC + kc + 1, lane);
                }
                const uint2* bf = bfrag + (size_t)kc * 8 * kBLanes;
                q2_tile_chunk<G>(wa, sa, bf, lane, acc[0]);
                q2_tile_chunk<G>(wb, sb, bf, lane, acc[1]);
                wa = na; wb = nb; sa = nsa; sb = nsb;
            }
        }
        // quad reduce: lanes 4r..4r+3 hold the parts of rows r and r+8
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v = acc[t][h];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                acc[t][h] = v;
            }
        if (S == 1) {
            if ((lane & 3) == 0) {
#pragma unroll
                for (int t = 0; t < 2; ++t)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int64_t row = (rt0 + t) * 16 + 8 * h + (lane >> 2);
                        if (row < rows) y[row] = acc[t][h];
                    }
            }
            continue;
        }
        if ((lane & 3) == 0) {
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    part[(ksplit * tpc + tpl) * 32 + t * 16 + 8 * h + (lane >> 2)] = acc[t][h];
        }
        __syncthreads();
        if (threadIdx.x < tpc * 32) {
            float s = 0.f;
            for (int k = 0; k < S; ++k) s += part[k * tpc * 32 + threadIdx.x];
            const int64_t row = unit * tpc * 32 + threadIdx.x;
            if (row < rows) y[row] = s;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Persistent, bulk-copy-fed variant (used for cols <= 16384).
//
// One CTA per SM: 16 consumer warps and 1 producer warp.  The CTA owns a
// contiguous range of 16-row tiles; the producer streams each tile pair's
// codes and scales for a K slab (contiguous in the packed layout) into a
// ring of shared-memory stages with cp.async.bulk, so up to ~180 KB per SM
// are in flight.  Consumer warp w decodes and multiplies chunks
// [w*n/16, (w+1)*n/16) of every slab from shared memory; at the last slab of a
// pair the 16 partial sums of each row are added in warp order by warp 0
// (deterministic).  Hand-offs use mbarriers with bounded waits only.
// ---------------------------------------------------------------------------
constexpr int kConsumerWarps = 16;
constexpr int kTmaThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 6;
constexpr int kTmaMaxChunks = 128;   // cols <= 16384

struct Q2Plan {
    int KC, slab, nslab, stages;
    uint32_t code_stage, scale_stage;
    size_t smem;
};

template <int G>
Q2Plan q2_plan(int KC) {
    constexpr int gpc = 128 / G;
    const size_t limit = 227 * 1024;
    const size_t fixed = (size_t)KC * 52 * sizeof(uint4) + 2 * kConsumerWarps * 32 * sizeof(float) +
                         (2 * kMaxStages + 4) * sizeof(uint64_t) + 16 + 128;
    Q2Plan p{};
    p.KC = KC;
    p.nslab = 1;
    p.slab = KC;
    auto stage_bytes = [&](int slab) { return (size_t)2 * slab * (512 + 32 * gpc); };
    while (p.slab > 8 && fixed + 3 * stage_bytes(p.slab) > limit) {
        ++p.nslab;
        p.slab = (KC + p.nslab - 1) / p.nslab;
    }
    p.code_stage = (uint32_t)(2 * p.slab * 512);
    p.scale_stage = (uint32_t)(2 * p.slab * 32 * gpc);
    size_t st = (limit - fixed) / stage_bytes(p.slab);
    p.stages = (int)(st > (size_t)kMaxStages ? kMaxStages : st);
    p.smem = fixed + (size_t)p.stages * stage_bytes(p.slab);
    return p;
}

template <int G>
__global__ void __launch_bounds__(kTmaThreads, 1) q2_gemv_tma_kernel(
    const uint4* __restrict__ codes, const __half* __restrict__ d, const float* __restrict__ x,
    float* __restrict__ y, int64_t rows, int64_t cols, int KC, int slab, int nslab, int stages,
    uint32_t code_stage, uint32_t scale_stage, int64_t n_tiles, uint32_t mul6, uint32_t mul12,
    int* __restrict__ status) {
    constexpr int gpc = 128 / G;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
    const uint32_t stage_bytes = code_stage + scale_stage;
    // activation fragments: per chunk 13 blocks of 64 B; block l (< 12) holds
    // lane l's B registers for the chunk's 8 k-steps, block 12 is zero
    uint4* bfrag = reinterpret_cast<uint4*>(base + (size_t)stages * stage_bytes);
    float* red = reinterpret_cast<float*>(bfrag + (size_t)KC * 52);   // [2][warps][32]
    uint64_t* full = reinterpret_cast<uint64_t*>(red + 2 * kConsumerWarps * 32);
    uint64_t* empty = full + kMaxStages;
    uint64_t* rdone = empty + kMaxStages;   // [2]
    uint64_t* rfree = rdone + 2;            // [2]
    int* abort_flag = reinterpret_cast<int*>(rfree + 2);
    volatile int* abort = abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = (int64_t)blockIdx.x * n_tiles / gridDim.x;
    const int64_t t1 = (int64_t)(blockIdx.x + 1) * n_tiles / gridDim.x;
    const int64_t npairs = (t1 - t0 + 1) / 2;
    const int64_t nitems = npairs * nslab;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            qmv::mbar_init(&full[s], 1);
            qmv::mbar_init(&empty[s], kConsumerWarps);
        }
        for (int b = 0; b < 2; ++b) {
            qmv::mbar_init(&rdone[b], kConsumerWarps);
            qmv::mbar_init(&rfree[b], 1);
        }
        *abort_flag = 0;
        qmv::mbar_fence_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int64_t i = 0;
            for (; i < nitems; ++i) {
                const int s = (int)(i % stages);
                const uint32_t ph = (uint32_t)(i / stages) & 1u;
                if (!qmv::mbar_wait(&empty[s], ph ^ 1u, abort, status)) break;
                const int64_t pr = i / nslab;
                const int sl = (int)(i % nslab);
                const int64_t t = t0 + 2 * pr;
                const int nt = (int)(t1 - t < 2 ? t1 - t : 2);
                const int c0 = sl * slab;
                const int nc = KC - c0 < slab ? KC - c0 : slab;
                const uint32_t cb = (uint32_t)nc * 512, sb = (uint32_t)nc * 32 * gpc;
                qmv::mbar_arrive_tx(&full[s], (uint32_t)nt * (cb + sb));
                uint8_t* st_codes = base + (size_t)s * stage_bytes;
                uint8_t* st_scales = st_codes + code_stage;
                for (int tt = 0; tt < nt; ++tt) {
                    const int64_t tc = (t + tt) * KC + c0;
                    qmv::bulk_g2s(st_codes + (size_t)tt * slab * 512, codes + tc * 32, cb, &full[s]);
                    qmv::bulk_g2s(st_scales + (size_t)tt * slab * 32 * gpc, d + tc * 16 * gpc, sb, &full[s]);
                }
            }
            // drain: every issued copy lands before the CTA may exit
            for (int k = 0; k < stages && i - 1 - k >= 0; ++k) {
                const int64_t j = i - 1 - k;
                qmv::mbar_wait(&full[j % stages], (uint32_t)(j / stages) & 1u, abort, status);
            }
        }
        return;
    }

    // ---------------- consumers: activation split into B fragments ----------------
    for (int e = threadIdx.x; e < KC * 8 * 4; e += kConsumerWarps * 32) {
        const int s = e >> 2, kq = e & 3;           // global k-step, lane quarter
        const int64_t k0 = 16 * (int64_t)s + 2 * kq;
        float2 lo2 = make_float2(0.f, 0.f), hi2 = make_float2(0.f, 0.f);
        if (k0 < cols) {   // cols % 64 == 0: then k0 + 9 < cols too
            lo2 = *reinterpret_cast<const float2*>(x + k0);
            hi2 = *reinterpret_cast<const float2*>(x + k0 + 8);
        }
        const float xv[4] = {lo2.x, lo2.y, hi2.x, hi2.y};
        __nv_bfloat16 p[3][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) split3(xv[q], p[0][q], p[1][q], p[2][q]);
        uint2* chunk = reinterpret_cast<uint2*>(bfrag + (size_t)(s >> 3) * 52);
#pragma unroll
        for (int part = 0; part < 3; ++part)
            chunk[(part * 4 + kq) * 8 + (s & 7)] =
                make_uint2(pack_bf16x2(p[part][0], p[part][1]), pack_bf16x2(p[part][2], p[part][3]));
    }
    for (int c = threadIdx.x; c < KC * 4; c += kConsumerWarps * 32)
        bfrag[(size_t)(c >> 2) * 52 + 48 + (c & 3)] = make_uint4(0u, 0u, 0u, 0u);
    qmv::named_bar(1, kConsumerWarps * 32);

    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    for (int64_t i = 0; i < nitems; ++i) {
        const int s = (int)(i % stages);
        const uint32_t ph = (uint32_t)(i / stages) & 1u;
        if (!qmv::mbar_wait(&full[s], ph, abort, status)) break;
        const int64_t pr = i / nslab;
        const int sl = (int)(i % nslab);
        const int64_t t = t0 + 2 * pr;
        const int nt = (int)(t1 - t < 2 ? t1 - t : 2);
        const int c0 = sl * slab;
        const int nc = KC - c0 < slab ? KC - c0 : slab;
        const uint4* st_codes = reinterpret_cast<const uint4*>(base + (size_t)s * stage_bytes);
        const __half* st_scales = reinterpret_cast<const __half*>(base + (size_t)s * stage_bytes + code_stage);
        const int ca = nc * warp / kConsumerWarps, cz = nc * (warp + 1) / kConsumerWarps;
        const int bl = lane < kBLanes ? lane : kBLanes;   // lanes 12..31 read the zero block
        for (int c = ca; c < cz; ++c) {
            const uint4* bsrc = bfrag + (size_t)(c0 + c) * 52 + bl * 4;
            const uint4 bq[4] = {bsrc[0], bsrc[1], bsrc[2], bsrc[3]};
            const uint4 wa = st_codes[(size_t)c * 32 + lane];
            const uint4 wb = st_codes[(size_t)(slab + c) * 32 + lane];
            uint32_t sa, sb, sa2 = 0, sb2 = 0;
            if (G == 64) {
                const uint2 va = reinterpret_cast<const uint2*>(st_scales + (size_t)c * 32)[lane >> 2];
                const uint2 vb = reinterpret_cast<const uint2*>(st_scales + (size_t)(slab + c) * 32)[lane >> 2];
                sa = va.x; sa2 = va.y; sb = vb.x; sb2 = vb.y;
            } else {
                sa = reinterpret_cast<const uint32_t*>(st_scales + (size_t)c * 16)[lane >> 2];
                sb = reinterpret_cast<const uint32_t*>(st_scales + (size_t)(slab + c) * 16)[lane >> 2];
            }
            q2_pair_chunk<G>(wa, wb, bq, sa, sb, sa2, sb2, nt > 1, mul6, mul12, acc);
        }
        __syncwarp();
        if (lane == 0) qmv::mbar_arrive(&empty[s]);
        if (sl != nslab - 1) continue;

        // last slab of the pair: reduce the 8 warps' partials in warp order
        const int buf = (int)(pr & 1);
        const uint32_t use = (uint32_t)(pr >> 1) & 1u;
#pragma unroll
        for (int tt = 0; tt < 2; ++tt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v = acc[tt][h];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                acc[tt][h] = v;
            }
        if (!qmv::mbar_wait(&rfree[buf], use ^ 1u, abort, status)) break;
        if ((lane & 3) == 0) {
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    red[(buf * kConsumerWarps + warp) * 32 + tt * 16 + 8 * h + (lane >> 2)] = acc[tt][h];
        }
        acc[0][0] = acc[0][1] = acc[1][0] = acc[1][1] = 0.f;
        __syncwarp();
        if (lane == 0) qmv::mbar_arrive(&rdone[buf]);
        if (warp == 0) {
            if (!qmv::mbar_wait(&rdone[buf], use, abort, status)) break;
            if (lane < nt * 16) {
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) sum += red[(buf * kConsumerWarps + w) * 32 + lane];
                const int64_t row = t * 16 + lane;
                if (row < rows) y[row] = sum;
            }
            __syncwarp();
            if (lane == 0) qmv::mbar_arrive(&rfree[buf]);
        }
    }
}

// ---------------------------------------------------------------------------
// Whole-tile variant (used when a round of tiles fits in shared memory; the
// 17408 x 5120 workload loads every tile a CTA owns at once).
//
// One CTA per SM with 16 consumer warps and 1 producer warp.  The CTA owns a
// contiguous range of 16-row tiles and processes them in rounds of TR tiles:
// the producer copies each tile's codes and scales (contiguous in the packed
// layout) with two cp.async.bulk into its own buffer, signalled on the tile's
// mbarrier.  WPT = 16/TR warps share a tile, each taking a contiguous K range
// of it, so every warp runs one long uninterrupted chunk loop; the WPT
// partial sums of each row are added in warp order by the tile's first warp
// (deterministic).  All hand-offs are mbarriers with bounded waits.
// ---------------------------------------------------------------------------
constexpr int kV3Warps = 16;
constexpr int kV3Threads = (kV3Warps + 1) * 32;
constexpr int kV3MaxTR = 8;

struct Q2PlanV3 {
    int TR, WPT;
    uint32_t tile_bytes, code_bytes;
    size_t smem;
    bool ok;
};

template <int G>
Q2PlanV3 q2_plan_v3(int KC) {
    constexpr int gpc = 128 / G;
    const size_t limit = 227 * 1024;
    Q2PlanV3 p{};
    p.code_bytes = (uint32_t)KC * 512;
    p.tile_bytes = p.code_bytes + (uint32_t)KC * 32 * gpc;
    const size_t fixed = (size_t)KC * 52 * sizeof(uint4) + (size_t)KC * 4 * sizeof(float2) +
                         kV3Warps * 32 * sizeof(float) + (2 * kV3MaxTR + 2) * sizeof(uint64_t) + 16 + 128;
    p.ok = false;
    if (KC > kTmaMaxChunks) return p;   // the activation prologue covers at most kTmaMaxChunks chunks
    for (int tr = kV3MaxTR; tr >= 1; tr >>= 1) {
        if (fixed + (size_t)tr * p.tile_bytes <= limit && KC >= kV3Warps / tr) {
            p.TR = tr;
            p.WPT = kV3Warps / tr;
            p.smem = fixed + (size_t)tr * p.tile_bytes;
            p.ok = true;
            break;
        }
    }
    return p;
}

template <int G>
__global__ void __launch_bounds__(kV3Threads, 1) q2_gemv_v3_kernel(
    const uint4* __restrict__ codes, const __half* __restrict__ d, const float* __restrict__ x,
    float* __restrict__ y, int64_t rows, int64_t cols, int KC, int TR, int WPT, uint32_t tile_bytes,
    uint32_t code_bytes, int64_t n_tiles, int* __restrict__ status) {
    constexpr int gpc = 128 / G;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
    uint4* bfrag = reinterpret_cast<uint4*>(base + (size_t)TR * tile_bytes);
    float2* ktab = reinterpret_cast<float2*>(bfrag + (size_t)KC * 52);   // [KC][lane % 4] bias terms
    float* red = reinterpret_cast<float*>(ktab + (size_t)KC * 4);         // [16 warps][32]
    uint64_t* tfull = reinterpret_cast<uint64_t*>(red + kV3Warps * 32);   // [TR]
    uint64_t* cdone = tfull + kV3MaxTR;                                   // [TR]
    uint64_t* rdone = cdone + kV3MaxTR;                                   // round finished
    int* abort_flag = reinterpret_cast<int*>(rdone + 2);
    volatile int* abort = abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = (int64_t)blockIdx.x * n_tiles / gridDim.x;
    const int64_t t1 = (int64_t)(blockIdx.x + 1) * n_tiles / gridDim.x;
    const int64_t ntl = t1 - t0;
    const int64_t rounds = (ntl + TR - 1) / TR;

    if (threadIdx.x == 0) {
        for (int i = 0; i < TR; ++i) {
            qmv::mbar_init(&tfull[i], 1);
            qmv::mbar_init(&cdone[i], WPT);
        }
        qmv::mbar_init(&rdone[0], kV3Warps);
        *abort_flag = 0;
        qmv::mbar_fence_init();
    }
    __syncthreads();

    if (warp == kV3Warps) {
        // ---------------- producer ----------------
        if (lane == 0) {
            // the codes and scales are constant: the first round is fetched
            // before the consumers' dependency wait (programmatic launch)
            int64_t issued_rounds = 0;
            for (int64_t r = 0; r < rounds; ++r) {
                if (r > 0 && !qmv::mbar_wait(&rdone[0], (uint32_t)(r - 1) & 1u, abort, status)) break;
                // one round done: the consumers have passed their wait
                if (r == 1) qmv::pdl_launch_dependents();
                for (int i = 0; i < TR; ++i) {
                    const int64_t t = t0 + r * TR + i;
                    if (t >= t1) break;
                    uint8_t* buf = base + (size_t)i * tile_bytes;
                    qmv::mbar_arrive_tx(&tfull[i], tile_bytes);
                    qmv::bulk_g2s(buf, codes + t * KC * 32, code_bytes, &tfull[i]);
                    qmv::bulk_g2s(buf + code_bytes, d + t * KC * 16 * gpc, tile_bytes - code_bytes, &tfull[i]);
                }
                issued_rounds = r + 1;
            }
            // drain the last round's copies before the CTA may exit
            if (issued_rounds > 0) {
                const int64_t r = issued_rounds - 1;
                for (int i = 0; i < TR && t0 + r * TR + i < t1; ++i) qmv::mbar_drain(&tfull[i], (uint32_t)r & 1u);
            }
        }
        return;
    }

    // x (and y) may belong to the previous kernel in the stream
    qmv::pdl_wait();
    qmv::pdl_launch_dependents();

    // ---------------- activation digits into B fragments ----------------
    // x is written as three base-256 digits on one grid set by the largest
    // |x| (exponent emax): x ~= 2^(emax-7) * (n0 + n1/256 + n2/65536) with
    // integers |n0| <= 256, |n1|, |n2| <= 128, an error of at most
    // 2^(emax-24) per element.  B column p holds digit n_p as the bf16
    // n_p * 2^(118-8p) for columns 0-7 of a k-step and n_p * 2^(114-8p) for
    // columns 8-15.  Against the decoded weights q * 2^(p'-133), every
    // product in column p is then an integer multiple of 2^(-15-8p) (of
    // 2^(-13-8p) on rows r+8) and a group's sum stays below 2^17 of those
    // units, so the MMA sums are exact whatever order the tensor core adds
    // in.  The bias -sum_{k in g} x_k enters through ktab: -N_p * 2^(-15-8p)
    // with N_p the group's (exact) digit sum, added once per group to the
    // column-pair sum of lane class 0 (columns 0 and 1, rounded once, as the
    // pair sum is) and of lane class 1 (column 2).  The loop therefore
    // leaves rows r scaled by 2^(-8-emax) and rows r+8 by 2^(-6-emax).
    //
    // Fragment layout per chunk: [k-step pair j][13 slots] uint4; slot l
    // (< 12) holds lane l's registers for k-steps 2j and 2j+1, slot 12 is
    // zero, so the four 128-bit loads of a chunk are conflict-free
    // (consecutive lanes, consecutive 16-byte slots; lanes 12..31 broadcast
    // the zero slot).  Every thread issues all of its activation loads before
    // using any.
    int emax;
    {
        constexpr int kMaxPer = (kTmaMaxChunks * 32 + kV3Warps * 32 - 1) / (kV3Warps * 32);
        constexpr int kItemsPerGroup = G / 4;   // 4 threads per 16-column k-step
        const int n = KC * 32;
        float2 lo[kMaxPer], hi[kMaxPer];
#pragma unroll
        for (int u = 0; u < kMaxPer; ++u) {
            const int e = threadIdx.x + u * kV3Warps * 32;
            lo[u] = hi[u] = make_float2(0.f, 0.f);
            if (e < n) {
                const int64_t k0 = 16 * (int64_t)(e >> 2) + 2 * (e & 3);
                if (k0 < cols) {   // cols % 64 == 0: then k0 + 9 < cols too
                    lo[u] = __ldca(reinterpret_cast<const float2*>(x + k0));
                    hi[u] = __ldca(reinterpret_cast<const float2*>(x + k0 + 8));
                }
            }
        }
        float m = 0.f;
#pragma unroll
        for (int u = 0; u < kMaxPer; ++u)
            m = fmaxf(m, fmaxf(fmaxf(fabsf(lo[u].x), fabsf(lo[u].y)), fmaxf(fabsf(hi[u].x), fabsf(hi[u].y))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) red[warp] = m;
        qmv::named_bar(1, kV3Warps * 32);
        float mx = 0.f;
#pragma unroll
        for (int w = 0; w < kV3Warps; ++w) mx = fmaxf(mx, red[w]);
        // clamped so that 2^(7-emax) and every scale below is a normal float
        emax = min(max((int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127, -120), 127);
        const float sc = __uint_as_float((uint32_t)(134 - emax) << 23);   // 2^(7-emax)
        const float kLo[3] = {0x1p118f, 0x1p110f, 0x1p102f};
        const float kHi[3] = {0x1p114f, 0x1p106f, 0x1p98f};
#pragma unroll
        for (int u = 0; u < kMaxPer; ++u) {
            const int e = threadIdx.x + u * kV3Warps * 32;
            if (e < n) {   // n is a multiple of 32: uniform across the warp
                const int s = e >> 2, kq = e & 3;
                const float xv[4] = {lo[u].x, lo[u].y, hi[u].x, hi[u].y};
                float dg[3][4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float t = xv[q] * sc;
                    dg[0][q] = rintf(t);
                    const float r1 = (t - dg[0][q]) * 256.f;
                    dg[1][q] = rintf(r1);
                    dg[2][q] = rintf((r1 - dg[1][q]) * 256.f);
                }
                uint2* chunk = reinterpret_cast<uint2*>(bfrag + (size_t)(s >> 3) * 52);
                const int j = (s & 7) >> 1, half = s & 1;
#pragma unroll
                for (int p = 0; p < 3; ++p) {
                    const __nv_bfloat162 b0 = __floats2bfloat162_rn(dg[p][0] * kLo[p], dg[p][1] * kLo[p]);
                    const __nv_bfloat162 b1 = __floats2bfloat162_rn(dg[p][2] * kHi[p], dg[p][3] * kHi[p]);
                    chunk[(j * 13 + p * 4 + kq) * 2 + half] =
                        make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
                }
                // the group's digit sums (integers below 2^15: exact)
                float ns[3];
#pragma unroll
                for (int p = 0; p < 3; ++p) ns[p] = (dg[p][0] + dg[p][1]) + (dg[p][2] + dg[p][3]);
#pragma unroll
                for (int o = 1; o < kItemsPerGroup; o <<= 1)
#pragma unroll
                    for (int p = 0; p < 3; ++p) ns[p] += __shfl_xor_sync(0xffffffffu, ns[p], o);
                const int gl = e & (kItemsPerGroup - 1);
                if (gl < 4) {   // item gl writes the bias of lane class gl
                    const float b01 = -ns[0] * 0x1p-15f + -ns[1] * 0x1p-23f;
                    const float kv = gl == 0 ? b01 : (gl == 1 ? -ns[2] * 0x1p-31f : 0.f);
                    const int grp = e / kItemsPerGroup;
                    float* kt = reinterpret_cast<float*>(ktab + (size_t)(grp / gpc) * 4 + gl);
                    kt[grp % gpc] = kv;
                    if (gpc == 1) kt[1] = 0.f;
                }
            }
        }
        for (int c = threadIdx.x; c < KC * 4; c += kV3Warps * 32)
            bfrag[(size_t)(c >> 2) * 52 + (c & 3) * 13 + 12] = make_uint4(0u, 0u, 0u, 0u);
    }
    qmv::named_bar(1, kV3Warps * 32);

    const int ti = warp / WPT;              // tile slot this warp works on
    const int part = warp % WPT;            // its K range within the tile
    const int ca = KC * part / WPT, cz = KC * (part + 1) / WPT;
    const int bl = lane < kBLanes ? lane : kBLanes;
    for (int64_t r = 0; r < rounds; ++r) {
        const int64_t t = t0 + r * TR + ti;
        if (t < t1) {
            if (!qmv::mbar_wait(&tfull[ti], (uint32_t)r & 1u, abort, status)) break;
            const uint4* tc = reinterpret_cast<const uint4*>(base + (size_t)ti * tile_bytes);
            const uint8_t* ts = base + (size_t)ti * tile_bytes + code_bytes;
            float acc[2] = {0.f, 0.f};
            float acc2[2] = {0.f, 0.f};
            auto chunk_args = [&](int c, uint4 (&bq)[4], uint4& w, uint32_t& s01, uint32_t& s23, float2& kk) {
                const uint4* bsrc = bfrag + (size_t)c * 52 + bl;
#pragma unroll
                for (int j = 0; j < 4; ++j) bq[j] = bsrc[j * 13];
                w = tc[(size_t)c * 32 + lane];
                kk = ktab[(size_t)c * 4 + (lane & 3)];
                if (G == 64) {
                    const uint2 v = reinterpret_cast<const uint2*>(ts + (size_t)c * 64)[lane >> 2];
                    s01 = v.x;
                    s23 = v.y;
                } else {
                    s01 = reinterpret_cast<const uint32_t*>(ts + (size_t)c * 32)[lane >> 2];
                    s23 = 0;
                }
            };
            int c = ca;
            for (; c + 1 < cz; c += 2) {   // two chunks per step: two independent MMA chains
                uint4 bq0[4], bq1[4], w0, w1;
                uint32_t s0a, s0b, s1a, s1b;
                float2 k0, k1;
                chunk_args(c, bq0, w0, s0a, s0b, k0);
                chunk_args(c + 1, bq1, w1, s1a, s1b, k1);
                q2_tile_chunk_v3<G>(w0, bq0, s0a, s0b, k0, acc);
                q2_tile_chunk_v3<G>(w1, bq1, s1a, s1b, k1, acc2);
            }
            if (c < cz) {
                uint4 bq0[4], w0;
                uint32_t s0a, s0b;
                float2 k0;
                chunk_args(c, bq0, w0, s0a, s0b, k0);
                q2_tile_chunk_v3<G>(w0, bq0, s0a, s0b, k0, acc);
            }
            acc[0] += acc2[0];
            acc[1] += acc2[1];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 1);
                acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 2);
            }
            if ((lane & 3) == 0) {
                red[warp * 32 + (lane >> 2)] = acc[0];
                red[warp * 32 + 8 + (lane >> 2)] = acc[1];
            }
            __syncwarp();
            if (lane == 0) qmv::mbar_arrive(&cdone[ti]);
            if (part == 0) {
                if (!qmv::mbar_wait(&cdone[ti], (uint32_t)r & 1u, abort, status)) break;
                if (lane < 16) {
                    float sum = 0.f;
                    for (int k = 0; k < WPT; ++k) sum += red[(warp + k) * 32 + lane];
                    const int64_t row = t * 16 + lane;
                    // undo the digit grid and the 4x of rows r+8 (exact)
                    if (row < rows) y[row] = ldexpf(sum, (lane < 8 ? 8 : 6) + emax);
                }
                __syncwarp();
            }
        }
        if (lane == 0) qmv::mbar_arrive(&rdone[0]);
    }
}

int choose_split(int64_t n_tp, int KC) {
    const int64_t target = (int64_t)qmv::sm_count() * 16;
    int S = 1;
    while (S < kWarps && n_tp * S < target && KC / (2 * S) >= 2) S *= 2;
    return S;
}

template <int G>
qmv_status launch_q2_tma(const qmv_weights* w, const float* x, float* y, cudaStream_t st) {
    const int KC = (int)(w->cols_pad / 128);
    const Q2Plan p = q2_plan<G>(KC);
    int* status = qmv::device_status();
    if (!status) return qmv::fail(QMV_ERR_CUDA, "qmv_q2: no CUDA device");
    static int configured[64] = {0};
    const int dev = qmv::current_device();
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaFuncSetAttribute(q2_gemv_tma_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        configured[dev] = 1;
    }
    const int64_t n_tiles = w->rows_pad / 16;
    int64_t grid = qmv::sm_count();
    if (grid > (n_tiles + 1) / 2) grid = (n_tiles + 1) / 2;
    q2_gemv_tma_kernel<G><<<(unsigned)grid, kTmaThreads, p.smem, st>>>(
        w->codes, w->d, x, y, w->rows, w->cols, KC, p.slab, p.nslab, p.stages, p.code_stage, p.scale_stage,
        n_tiles, 1u << 26, 1u << 20, status);
    return qmv::check_launch("q2_gemv_tma_kernel");
}

template <int G>
qmv_status launch_q2_v3(const qmv_weights* w, const Q2PlanV3& p, const float* x, float* y, cudaStream_t st) {
    const int KC = (int)(w->cols_pad / 128);
    int* status = qmv::device_status();
    if (!status) return qmv::fail(QMV_ERR_CUDA, "qmv_q2: no CUDA device");
    static int configured[64] = {0};
    const int dev = qmv::current_device();
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaFuncSetAttribute(q2_gemv_v3_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        configured[dev] = 1;
    }
    const int64_t n_tiles = w->rows_pad / 16;
    int64_t grid = qmv::sm_count();
    if (grid > n_tiles) grid = n_tiles;
    return qmv::launch_pdl(q2_gemv_v3_kernel<G>, dim3((unsigned)grid), dim3(kV3Threads), p.smem, st, w->codes, w->d, x,
                           y, w->rows, w->cols, KC, p.TR, p.WPT, p.tile_bytes, p.code_bytes, n_tiles, status);
}

template <int G>
qmv_status launch_q2(const qmv_weights* w, const float* x, float* y, cudaStream_t st) {
    const int KC = (int)(w->cols_pad / 128);
    const Q2PlanV3 p3 = q2_plan_v3<G>(KC);
    if (p3.ok) return launch_q2_v3<G>(w, p3, x, y, st);
    if (KC <= kTmaMaxChunks) return launch_q2_tma<G>(w, x, y, st);
    const int64_t n_tp = w->rows_pad / 32;
    const int S = choose_split(n_tp, KC);
    const int tpc = kWarps / S;
    const int64_t n_units = (n_tp + tpc - 1) / tpc;
    const size_t smem = (size_t)KC * 8 * kBLanes * sizeof(uint2) + (size_t)kWarps * 32 * sizeof(float);
    static int configured[64] = {0};
    const int dev = qmv::current_device();
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaFuncSetAttribute(q2_gemv_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        configured[dev] = 1;
    }
    int64_t grid = (int64_t)qmv::sm_count() * (smem <= 64 * 1024 ? 3 : smem <= 100 * 1024 ? 2 : 1);
    if (grid > n_units) grid = n_units;
    q2_gemv_kernel<G><<<(unsigned)grid, kThreads, smem, st>>>(w->codes, w->d, x, y, w->rows, w->cols, KC, S,
                                                              n_units);
    return qmv::check_launch("q2_gemv_kernel");
}

qmv_status q2_entry(const qmv_weights* w, const float* x, float* y, qmv_stream st, int group,
                    const char* name) {
    QMV_REQUIRE(w && x && y, QMV_ERR_INVALID_ARG, "%s: null argument", name);
    QMV_REQUIRE(w->format == (group == 64 ? QMV_FMT_Q2G64 : QMV_FMT_Q2G128), QMV_ERR_UNSUPPORTED,
                "%s: handle is not Q2 g%d", name, group);
    QMV_REQUIRE(qmv::aligned16(x) && qmv::aligned16(y), QMV_ERR_INVALID_ARG,
                "%s: x and y must be 16-byte aligned", name);
    return group == 64 ? launch_q2<64>(w, x, y, (cudaStream_t)st) : launch_q2<128>(w, x, y, (cudaStream_t)st);
}

}  // namespace

extern "C" qmv_status qmv_q2g64(const qmv_weights* w, const float* x, float* y, qmv_stream st) {
    return q2_entry(w, x, y, st, 64, "qmv_q2g64");
}

extern "C" qmv_status qmv_q2g128(const qmv_weights* w, const float* x, float* y, qmv_stream st) {
    return q2_entry(w, x, y, st, 128, "qmv_q2g128");
}
