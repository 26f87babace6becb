// q8_row decode GEMV:  y[o] = rs[o] * sum_i q[o,i] * xs[i].
//
// cortiq-engine 0.5.43 src/gpu_wgpu.rs, WGSL `q8_matvec` (one workgroup per
// row, tree reduction) and cortiq-engine 0.3.7 src/gpu_metal.rs, MSL
// `q8_matvec` (one simdgroup per row, coalesced char4 reads) are the prior
// art.  Here a warp owns a 4-row group and streams it with 128-bit loads
// (512 contiguous bytes per warp per step), converts the int8 codes to f32
// exactly in registers and accumulates with packed f32x2 FMAs; the K range
// is split across the warps of a CTA when the row count alone cannot fill
// the GPU, and the S partial sums are reduced in shared memory in a fixed
// order (deterministic).
#include "q8_block.cuh"

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kUnroll = 4;

// Warp w of a CTA: row group (blockIdx.x * (kWarps/S) + w / S), K split w % S.
__global__ void __launch_bounds__(kThreads) q8row_gemv_kernel(
    const int8_t* __restrict__ q, const float* __restrict__ rs, const float* __restrict__ xs,
    float* __restrict__ y, int64_t rows, int64_t cols, int64_t cols_pad, int S) {
    __shared__ float part[kWarps * 4];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int gpc = kWarps / S;                       // row groups per CTA
    const int ks = warp % S;
    const int rgl = warp / S;
    const int64_t rg = (int64_t)blockIdx.x * gpc + rgl;
    const int64_t nblk = cols_pad / 128;
    const int64_t b0 = nblk * ks / S, b1 = nblk * (ks + 1) / S;
    const bool live = rg * 4 < rows;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (live) qmv::q8_rowgroup_dot<kUnroll>(q, cols_pad, rg, b0, b1, xs, cols, lane, v);
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] = qmv::warp_sum(v[r]);
    if (S == 1) {
        if (live && lane < 4) {
            const int64_t row = rg * 4 + lane;
            const float vv = lane == 0 ? v[0] : lane == 1 ? v[1] : lane == 2 ? v[2] : v[3];
            if (row < rows) y[row] = rs[row] * vv;
        }
        return;
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < 4; ++r) part[(ks * gpc + rgl) * 4 + r] = v[r];
    }
    __syncthreads();
    if (threadIdx.x < gpc * 4) {
        const int rl = threadIdx.x;  // row within the CTA
        float s = 0.f;
        for (int k = 0; k < S; ++k) s += part[k * gpc * 4 + rl];
        const int64_t row = (int64_t)blockIdx.x * gpc * 4 + rl;
        if (row < rows) y[row] = rs[row] * s;
    }
}

// Number of warps a row group's K range is split across: enough warps to
// fill the GPU several times over, but at least 4 blocks of 128 columns each.
int choose_split(int64_t n_rg, int64_t nblk) {
    const int64_t target = (int64_t)qmv::sm_count() * 32;  // resident warps across the GPU
    int S = 1;
    while (S < kWarps && n_rg * S < target && nblk / (2 * S) >= 4) S *= 2;
    return S;
}

}  // namespace

extern "C" qmv_status qmv_q8row(const qmv_weights* w, const float* xs, float* y, qmv_stream st) {
    QMV_REQUIRE(w && xs && y, QMV_ERR_INVALID_ARG, "qmv_q8row: null argument");
    QMV_REQUIRE(w->format == QMV_FMT_Q8ROW, QMV_ERR_UNSUPPORTED, "qmv_q8row: handle is not q8_row");
    QMV_REQUIRE(w->experts == 1, QMV_ERR_UNSUPPORTED, "qmv_q8row: handle is an expert stack");
    QMV_REQUIRE(qmv::aligned16(xs) && qmv::aligned16(y), QMV_ERR_INVALID_ARG,
                "qmv_q8row: xs and y must be 16-byte aligned");
    const int64_t n_rg = (w->rows + 3) / 4;
    const int64_t nblk = w->cols_pad / 128;
    const int S = choose_split(n_rg, nblk);
    const int gpc = kWarps / S;
    const int64_t grid = (n_rg + gpc - 1) / gpc;
    q8row_gemv_kernel<<<(unsigned)grid, kThreads, 0, (cudaStream_t)st>>>(
        w->q, w->rs, xs, y, w->rows, w->cols, w->cols_pad, S);
    return qmv::check_launch("q8row_gemv_kernel");
}
