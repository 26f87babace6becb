// MoE decode step: router select and the expert FFN over the selected slots.
//
// Router select (cortiq-engine 0.5.43 src/gpu_wgpu.rs, WGSL `moe_select_sg`
// and `moe_select`): one CTA, all-parallel.  The shared-expert gate dot is
// compensated (Ogita-Rump-Oishi Dot2: TwoProduct via FMA + TwoSum), so the
// sigmoid weight stays within 1e-6 relative of the exact value; the softmax
// max and denominator are block reductions; the top-k is k rounds of a
// block argmax on the raw f32 logits with the lowest index winning equal
// values, and chosen experts are excluded by a flag (not by overwriting the
// logit with a sentinel), so every finite logit is handled.
//
// Expert FFN (cortiq-engine 0.5.43 src/gpu_wgpu.rs, WGSL `moe_gate_up` and
// `moe_down`; cortiq-engine 0.3.7 src/gpu_metal.rs, host `moe_block`): two
// kernels.  gate/up: a warp owns a 4-row group of BOTH matrices of one slot
// (they share the x reads) and writes act = silu(g) * u.  down: a warp owns
// a 4-row group of the output and a share of the slots; per slot it forms
// the row dot with act, scales by rs and the router weight, and the shares
// are reduced in shared memory in a fixed order.
#include <cfloat>
#include <climits>

#include "q8_block.cuh"

namespace {

constexpr int kSelThreads = 256;
constexpr int kSelMaxPerThread = 4;   // n_exp <= 1024

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// (value, index) better-than: larger value, or equal value and lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(kSelThreads) moe_select_kernel(
    const float* __restrict__ logits, int n, int k, int renorm, const float* __restrict__ sgw,
    const float* __restrict__ x, int hidden, const float* __restrict__ sg_logit, int32_t* __restrict__ sel,
    float* __restrict__ wout) {
    __shared__ float s_a[kSelThreads / 32];
    __shared__ float s_b[kSelThreads / 32];
    __shared__ int s_i[kSelThreads / 32];
    __shared__ float s_gate;
    __shared__ int s_pick;
    __shared__ float s_wsel[1024];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    constexpr int nw = kSelThreads / 32;

    // ---- shared-expert gate: compensated dot product (Dot2) ----
    if (sgw) {
        float s = 0.f, c = 0.f;
        for (int i = tid; i < hidden; i += kSelThreads) {
            const float a = sgw[i], b = x[i];
            const float p = a * b;
            const float pe = fmaf(a, b, -p);
            float t, e;
            two_sum(s, p, t, e);
            s = t;
            c += e + pe;
        }
        for (int off = 16; off > 0; off >>= 1) {
            const float so = __shfl_xor_sync(0xffffffffu, s, off);
            const float co = __shfl_xor_sync(0xffffffffu, c, off);
            float t, e;
            two_sum(s, so, t, e);
            s = t;
            c += co + e;
        }
        if (lane == 0) { s_a[wid] = s; s_b[wid] = c; }
        __syncthreads();
        if (tid == 0) {
            float ss = s_a[0], cc = s_b[0];
            for (int w = 1; w < nw; ++w) {
                float t, e;
                two_sum(ss, s_a[w], t, e);
                ss = t;
                cc += s_b[w] + e;
            }
            s_gate = ss + cc;
        }
        __syncthreads();
    } else if (sg_logit) {
        if (tid == 0) s_gate = *sg_logit;
        __syncthreads();
    }

    // ---- logits, max, softmax denominator ----
    float v[kSelMaxPerThread];
    bool live[kSelMaxPerThread];
    float m = -FLT_MAX;
#pragma unroll
    for (int j = 0; j < kSelMaxPerThread; ++j) {
        const int idx = tid + j * kSelThreads;
        live[j] = idx < n;
        v[j] = live[j] ? logits[idx] : -FLT_MAX;
        if (live[j]) m = fmaxf(m, v[j]);
    }
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) s_a[wid] = m;
    __syncthreads();
    float mx = s_a[0];
    for (int w = 1; w < nw; ++w) mx = fmaxf(mx, s_a[w]);
    __syncthreads();
    // softmax denominator: compensated (TwoSum) summation, so its error is
    // ~1 ulp however many logits there are
    float es = 0.f, ec = 0.f;
#pragma unroll
    for (int j = 0; j < kSelMaxPerThread; ++j)
        if (live[j]) {
            float t, e;
            two_sum(es, expf(v[j] - mx), t, e);
            es = t;
            ec += e;
        }
    for (int off = 16; off > 0; off >>= 1) {
        const float so = __shfl_xor_sync(0xffffffffu, es, off);
        const float co = __shfl_xor_sync(0xffffffffu, ec, off);
        float t, e;
        two_sum(es, so, t, e);
        es = t;
        ec += co + e;
    }
    if (lane == 0) { s_a[wid] = es; s_b[wid] = ec; }
    __syncthreads();
    float den_s = s_a[0], den_c = s_b[0];
    for (int w = 1; w < nw; ++w) {
        float t, e;
        two_sum(den_s, s_a[w], t, e);
        den_s = t;
        den_c += s_b[w] + e;
    }
    const float den = den_s + den_c;

    // ---- k rounds of block argmax over the unchosen logits ----
    bool chosen[kSelMaxPerThread] = {false, false, false, false};
    for (int s = 0; s < k; ++s) {
        float bv = -FLT_MAX;
        int bi = INT_MAX;
#pragma unroll
        for (int j = 0; j < kSelMaxPerThread; ++j) {
            const int idx = tid + j * kSelThreads;
            if (live[j] && !chosen[j] && (bi == INT_MAX || better(v[j], idx, bv, bi))) {
                bv = v[j];
                bi = idx;
            }
        }
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (oi != INT_MAX && (bi == INT_MAX || better(ov, oi, bv, bi))) { bv = ov; bi = oi; }
        }
        __syncthreads();  // previous round's s_a / s_i reads are done
        if (lane == 0) { s_a[wid] = bv; s_i[wid] = bi; }
        __syncthreads();
        if (tid == 0) {
            float fv = s_a[0];
            int fi = s_i[0];
            for (int w = 1; w < nw; ++w)
                if (s_i[w] != INT_MAX && (fi == INT_MAX || better(s_a[w], s_i[w], fv, fi))) {
                    fv = s_a[w];
                    fi = s_i[w];
                }
            s_pick = fi;
            sel[s] = fi;
            s_wsel[s] = expf(fv - mx);   // unnormalised; divided below
        }
        __syncthreads();
        const int pick = s_pick;
#pragma unroll
        for (int j = 0; j < kSelMaxPerThread; ++j)
            if (tid + j * kSelThreads == pick) chosen[j] = true;
    }

    if (tid == 0) {
        // renormalised weights are e_s / sum_selected e (the softmax
        // denominator cancels); the selected sum is compensated as well
        float ws = 0.f, wc = 0.f;
        for (int s = 0; s < k; ++s) {
            float t, e;
            two_sum(ws, s_wsel[s], t, e);
            ws = t;
            wc += e;
        }
        const float norm = renorm ? ws + wc : den;
        for (int s = 0; s < k; ++s) wout[s] = s_wsel[s] / norm;
        if (sgw || sg_logit) {
            sel[k] = n;
            wout[k] = 1.0f / (1.0f + expf(-s_gate));
        }
    }
}

// ---- expert FFN ----

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

// grid.x: row-group chunks of `inter`, grid.y: slot.  act[slot][row].
__global__ void __launch_bounds__(kThreads) moe_gate_up_kernel(
    const int8_t* __restrict__ gq, const float* __restrict__ grs, const int8_t* __restrict__ uq,
    const float* __restrict__ urs, int64_t n_experts, int64_t inter, int64_t rows_pad, int64_t cols_pad,
    int64_t hidden, const int32_t* __restrict__ sel, const float* __restrict__ x, float* __restrict__ act,
    int* __restrict__ status) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slot = blockIdx.y;
    const int64_t rg = (int64_t)blockIdx.x * kWarps + warp;
    if (rg * 4 >= inter) return;
    const int e = sel[slot];
    if (e < 0 || e >= n_experts) {
        if (lane == 0) atomicCAS(status, 0, qmv::kDevBadExpert);
        if (lane < 4 && rg * 4 + lane < inter) act[slot * inter + rg * 4 + lane] = 0.f;
        return;
    }
    const int64_t nblk = cols_pad / 128;
    const int8_t* gbase = gq + (int64_t)e * rows_pad * cols_pad;
    const int8_t* ubase = uq + (int64_t)e * rows_pad * cols_pad;
    float2 ag[4], au[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) { ag[r] = make_float2(0.f, 0.f); au[r] = make_float2(0.f, 0.f); }
    const int8_t* pg = gbase + rg * 4 * cols_pad + lane * 16;
    const int8_t* pu = ubase + rg * 4 * cols_pad + lane * 16;
    int64_t b = 0;
    constexpr int U = 4;
    for (; b + U <= nblk; b += U) {
        uint4 wg[U], wu[U];
        float4 xv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            wg[u] = qmv::ld_stream_u4(pg + (b + u) * 512);
            wu[u] = qmv::ld_stream_u4(pu + (b + u) * 512);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) xv[u] = qmv::act_for_block(x, b + u, lane, hidden);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            qmv::q8_chunk_fma(wg[u], xv[u], ag);
            qmv::q8_chunk_fma(wu[u], xv[u], au);
        }
    }
    for (; b < nblk; ++b) {
        const float4 xv = qmv::act_for_block(x, b, lane, hidden);
        qmv::q8_chunk_fma(qmv::ld_stream_u4(pg + b * 512), xv, ag);
        qmv::q8_chunk_fma(qmv::ld_stream_u4(pu + b * 512), xv, au);
    }
    float g[4], u[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        g[r] = qmv::warp_sum(ag[r].x + ag[r].y);
        u[r] = qmv::warp_sum(au[r].x + au[r].y);
    }
    if (lane < 4) {
        const int64_t row = rg * 4 + lane;
        if (row < inter) {
            const float gs = (lane == 0 ? g[0] : lane == 1 ? g[1] : lane == 2 ? g[2] : g[3]) *
                             grs[(int64_t)e * rows_pad + row];
            const float us = (lane == 0 ? u[0] : lane == 1 ? u[1] : lane == 2 ? u[2] : u[3]) *
                             urs[(int64_t)e * rows_pad + row];
            act[slot * inter + row] = gs / (1.0f + expf(-gs)) * us;
        }
    }
}

// Warp w: row group blockIdx.x * (kWarps/S) + w / S, slots s = w % S, w % S + S, ...
__global__ void __launch_bounds__(kThreads) moe_down_kernel(
    const int8_t* __restrict__ dq, const float* __restrict__ drs, int64_t n_experts, int64_t hidden,
    int64_t rows_pad, int64_t cols_pad, int64_t inter, const int32_t* __restrict__ sel,
    const float* __restrict__ wsel, int slots, const float* __restrict__ act, float* __restrict__ out, int S) {
    __shared__ float part[kWarps * 4];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gpc = kWarps / S;
    const int ks = warp % S, rgl = warp / S;
    const int64_t rg = (int64_t)blockIdx.x * gpc + rgl;
    const int64_t nblk = cols_pad / 128;
    float tot[4] = {0.f, 0.f, 0.f, 0.f};
    if (rg * 4 < hidden) {
        for (int s = ks; s < slots; s += S) {
            const int e = sel[s];
            if (e < 0 || e >= n_experts) continue;  // reported by the gate/up kernel
            float v[4];
            qmv::q8_rowgroup_dot<2>(dq + (int64_t)e * rows_pad * cols_pad, cols_pad, rg, 0, nblk,
                                    act + (int64_t)s * inter, inter, lane, v);
            const float ws = wsel[s];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int64_t row = rg * 4 + r;
                const float rsv = row < hidden ? drs[(int64_t)e * rows_pad + row] : 0.f;
                tot[r] = fmaf(ws * rsv, qmv::warp_sum(v[r]), tot[r]);
            }
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < 4; ++r) part[(ks * gpc + rgl) * 4 + r] = tot[r];
    }
    __syncthreads();
    if (threadIdx.x < gpc * 4) {
        float s = 0.f;
        for (int k = 0; k < S; ++k) s += part[k * gpc * 4 + threadIdx.x];
        const int64_t row = (int64_t)blockIdx.x * gpc * 4 + threadIdx.x;
        if (row < hidden) out[row] = s;
    }
}

}  // namespace

extern "C" qmv_status moe_select_topk(const float* logits, int n_exp, int top_k, int renorm,
                                      const float* sg_w, const float* x, int hidden, const float* sg_logit,
                                      int32_t* sel, float* w, qmv_stream st) {
    QMV_REQUIRE(logits && sel && w, QMV_ERR_INVALID_ARG, "moe_select_topk: null argument");
    QMV_REQUIRE(n_exp >= 1 && n_exp <= kSelThreads * kSelMaxPerThread, QMV_ERR_INVALID_ARG,
                "moe_select_topk: need 1 <= n_exp <= %d (got %d)", kSelThreads * kSelMaxPerThread, n_exp);
    QMV_REQUIRE(top_k >= 1 && top_k <= n_exp, QMV_ERR_INVALID_ARG,
                "moe_select_topk: need 1 <= top_k <= n_exp (got %d)", top_k);
    QMV_REQUIRE(!sg_w || (x && hidden >= 1), QMV_ERR_INVALID_ARG,
                "moe_select_topk: sg_w needs x and hidden >= 1");
    moe_select_kernel<<<1, kSelThreads, 0, (cudaStream_t)st>>>(logits, n_exp, top_k, renorm, sg_w, x, hidden,
                                                              sg_w ? nullptr : sg_logit, sel, w);
    return qmv::check_launch("moe_select_kernel");
}

extern "C" qmv_status moe_ffn_q8row(const qmv_weights* gate, const qmv_weights* up, const qmv_weights* down,
                                    const int32_t* sel, const float* w, int slots, const float* x, float* out,
                                    qmv_stream st) {
    QMV_REQUIRE(gate && up && down && sel && w && x && out, QMV_ERR_INVALID_ARG, "moe_ffn_q8row: null argument");
    QMV_REQUIRE(gate->format == QMV_FMT_Q8ROW && up->format == QMV_FMT_Q8ROW && down->format == QMV_FMT_Q8ROW,
                QMV_ERR_UNSUPPORTED, "moe_ffn_q8row: handles must be q8_row");
    QMV_REQUIRE(slots >= 1 && slots <= 64, QMV_ERR_INVALID_ARG, "moe_ffn_q8row: need 1 <= slots <= 64");
    const int64_t E = gate->experts, inter = gate->rows, hidden = gate->cols;
    QMV_REQUIRE(up->experts == E && up->rows == inter && up->cols == hidden && down->experts == E &&
                    down->rows == hidden && down->cols == inter,
                QMV_ERR_INVALID_ARG, "moe_ffn_q8row: gate/up [E][inter][hidden] and down [E][hidden][inter] "
                                     "shapes disagree");
    QMV_REQUIRE(qmv::aligned16(x) && qmv::aligned16(out), QMV_ERR_INVALID_ARG,
                "moe_ffn_q8row: x and out must be 16-byte aligned");
    int* status = qmv::device_status();
    QMV_REQUIRE(status, QMV_ERR_CUDA, "moe_ffn_q8row: no CUDA device");
    cudaStream_t cs = (cudaStream_t)st;
    float* act = nullptr;
    const size_t act_bytes = (size_t)slots * (size_t)inter * sizeof(float);
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&act), act_bytes, cs);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return qmv::fail(QMV_ERR_ALLOC, "moe_ffn_q8row: scratch allocation failed: %s", cudaGetErrorString(e));
    }
    const dim3 g1((unsigned)(((inter + 3) / 4 + kWarps - 1) / kWarps), (unsigned)slots);
    moe_gate_up_kernel<<<g1, kThreads, 0, cs>>>(gate->q, gate->rs, up->q, up->rs, E, inter, gate->rows_pad,
                                                gate->cols_pad, hidden, sel, x, act, status);
    const int S = slots >= 4 ? 4 : slots >= 2 ? 2 : 1;
    const int gpc = kWarps / S;
    const int64_t n_rg = (hidden + 3) / 4;
    moe_down_kernel<<<(unsigned)((n_rg + gpc - 1) / gpc), kThreads, 0, cs>>>(
        down->q, down->rs, E, hidden, down->rows_pad, down->cols_pad, inter, sel, w, slots, act, out, S);
    qmv_status s = qmv::check_launch("moe kernels");
    cudaFreeAsync(act, cs);
    return s;
}

// ---------------------------------------------------------------------------
// moe_ffn_q8row_static: the same expert FFN, allocating nothing.
//
// Some callers cannot allocate device memory once they are serving: engines
// that hand all device memory to their own allocator at start-up and refuse
// allocations afterwards, and plugins loaded into such engines.  For them the
// activation scratch of the two FFN kernels lives in the fixed array below.
// Every GPU that loads this library holds it (256 KiB) until the process
// exits; calls with slots * inter above its size are rejected.
//
// All calls on a device share the array and it keeps the last call's
// contents; nothing has to start at zero, because the gate/up kernel writes
// every element (slot, row) that the down kernel then reads.  Two calls whose
// work overlaps on the GPU (e.g. on different streams without ordering) race
// on the array: order them.
//
// The array's name is only a host-side stand-in in host code, so its device
// address is looked up once per device with cudaGetSymbolAddress, with that
// device current, by the first call made on the device.  That first call
// should come before any stream capture.
// ---------------------------------------------------------------------------
#include <mutex>

constexpr int64_t kStaticActFloats = 1 << 16;   // slots * inter <= 65536
static __device__ __align__(256) float g_static_act[kStaticActFloats];

namespace {

std::mutex g_static_mu;
float* g_static_act_ptr[64] = {};

qmv_status static_act_address(float** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64)
        return qmv::fail(QMV_ERR_CUDA, "moe_ffn_q8row_static: no usable CUDA device");
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_act_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_act);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return qmv::fail(QMV_ERR_CUDA, "moe_ffn_q8row_static: cudaGetSymbolAddress failed: %s",
                             cudaGetErrorString(e));
        }
        g_static_act_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_static_act_ptr[dev];
    return QMV_OK;
}

}  // namespace

extern "C" qmv_status moe_ffn_q8row_static(const qmv_weights* gate, const qmv_weights* up,
                                           const qmv_weights* down, const int32_t* sel, const float* w,
                                           int slots, const float* x, float* out, qmv_stream st) {
    QMV_REQUIRE(gate && up && down && sel && w && x && out, QMV_ERR_INVALID_ARG,
                "moe_ffn_q8row_static: null argument");
    QMV_REQUIRE(gate->format == QMV_FMT_Q8ROW && up->format == QMV_FMT_Q8ROW && down->format == QMV_FMT_Q8ROW,
                QMV_ERR_UNSUPPORTED, "moe_ffn_q8row_static: handles must be q8_row");
    QMV_REQUIRE(slots >= 1 && slots <= 64, QMV_ERR_INVALID_ARG, "moe_ffn_q8row_static: need 1 <= slots <= 64");
    const int64_t E = gate->experts, inter = gate->rows, hidden = gate->cols;
    QMV_REQUIRE(up->experts == E && up->rows == inter && up->cols == hidden && down->experts == E &&
                    down->rows == hidden && down->cols == inter,
                QMV_ERR_INVALID_ARG, "moe_ffn_q8row_static: gate/up [E][inter][hidden] and down [E][hidden][inter] "
                                     "shapes disagree");
    QMV_REQUIRE((int64_t)slots * inter <= kStaticActFloats, QMV_ERR_UNSUPPORTED,
                "moe_ffn_q8row_static: slots * inter = %lld exceeds the fixed scratch of %lld floats",
                (long long)((int64_t)slots * inter), (long long)kStaticActFloats);
    QMV_REQUIRE(qmv::aligned16(x) && qmv::aligned16(out), QMV_ERR_INVALID_ARG,
                "moe_ffn_q8row_static: x and out must be 16-byte aligned");
    int* status = qmv::device_status();
    QMV_REQUIRE(status, QMV_ERR_CUDA, "moe_ffn_q8row_static: no CUDA device");
    float* act = nullptr;
    const qmv_status sa = static_act_address(&act);
    if (sa != QMV_OK) return sa;
    cudaStream_t cs = (cudaStream_t)st;
    const dim3 g1((unsigned)(((inter + 3) / 4 + kWarps - 1) / kWarps), (unsigned)slots);
    moe_gate_up_kernel<<<g1, kThreads, 0, cs>>>(gate->q, gate->rs, up->q, up->rs, E, inter, gate->rows_pad,
                                                gate->cols_pad, hidden, sel, x, act, status);
    const int S = slots >= 4 ? 4 : slots >= 2 ? 2 : 1;
    const int gpc = kWarps / S;
    const int64_t n_rg = (hidden + 3) / 4;
    moe_down_kernel<<<(unsigned)((n_rg + gpc - 1) / gpc), kThreads, 0, cs>>>(
        down->q, down->rs, E, hidden, down->rows_pad, down->cols_pad, inter, sel, w, slots, act, out, S);
    return qmv::check_launch("moe_ffn_q8row_static kernels");
}
