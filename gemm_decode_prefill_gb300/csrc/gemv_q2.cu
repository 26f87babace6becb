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
// The K range is split across the warps of a CTA; partial sums are reduced
// in shared memory in a fixed order (deterministic).
#include "qmv_internal.cuh"

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
    a[0] = bf16x2_fma((w & m0) | one, s0, c0);
    a[1] = bf16x2_fma((w & m2) | one, s2, c2);
    a[2] = bf16x2_fma((w & m4) | one, s4, c4);
    a[3] = bf16x2_fma((w6 & m0) | one, s0, c0);
    a[4] = bf16x2_fma((w6 & m2) | one, s2, c2);
    a[5] = bf16x2_fma((w6 & m4) | one, s4, c4);
    a[6] = bf16x2_fma((w12 & m0) | one, s0, c0);
    a[7] = bf16x2_fma((w12 & m2) | one, s2, c2);
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

// Per-(tile, chunk) scale fetch: G=64 -> 4 f16 (2 row halves x 2 groups),
// G=128 -> 2 f16 (2 row halves).
template <int G> struct Scales;
template <> struct Scales<64> {
    uint2 v;
    __device__ __forceinline__ void load(const __half* d, int64_t tc, int lane) {
        v = __ldg(reinterpret_cast<const uint2*>(d + tc * 32) + (lane >> 2));
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

int choose_split(int64_t n_tp, int KC) {
    const int64_t target = (int64_t)qmv::sm_count() * 16;
    int S = 1;
    while (S < kWarps && n_tp * S < target && KC / (2 * S) >= 2) S *= 2;
    return S;
}

template <int G>
qmv_status launch_q2(const qmv_weights* w, const float* x, float* y, cudaStream_t st) {
    const int KC = (int)(w->cols_pad / 128);
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
