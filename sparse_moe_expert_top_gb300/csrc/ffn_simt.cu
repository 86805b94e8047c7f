// Grouped expert FFN in fp32 on the SIMT pipes (operand type MOE_F32).
//
// The fp32 workload's tolerance (1e-5 relative) rules out tf32 tensor-core
// arithmetic, so this path multiplies with fp32 FMAs.  One CTA owns one
// expert and a 64-wide slice of the output columns and walks the expert's
// compact rows 32 at a time; shared-memory tiles of 32 rows x 32 K and
// 64 columns x 32 K feed 2x4 register blocks per thread.
//
// Page "perf(ds4): batch heterogeneous MoE prefill by expert" (Luce-Org/
// lucebox PR #640), Summary: grouped gate/up and down projections over the
// expert-major compact rows, one grouped launch for all active experts.

#include <cuda_runtime.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRows = 32, kCols = 64, kK = 32, kThreads = 256;

// GATED: h[i][m] = silu(xs[i].wa[e][m]) * (xs[i].wb[e][m]); otherwise
// y[i][m] = xs[i].wa[e][m].  `a` is [cap][K], wa/wb are [E][M][K].
template <bool GATED>
__global__ void __launch_bounds__(kThreads) ffn_simt_kernel(const float* __restrict__ a,
                                                            const int32_t* __restrict__ offsets, int cap, int K,
                                                            int M, const float* __restrict__ wa,
                                                            const float* __restrict__ wb, float* __restrict__ out,
                                                            unsigned* err) {
    __shared__ float sa[kRows][kK + 1];
    __shared__ float sw0[kCols][kK + 1];
    __shared__ float sw1[GATED ? kCols : 1][kK + 1];
    const int e = blockIdx.y, m0 = blockIdx.x * kCols, tid = threadIdx.x;
    const int lo = offsets[e], hi = offsets[e + 1];
    if (lo < 0 || hi < lo || hi > cap) {
        if (tid == 0) atomicOr(err, DEVERR_OFFSETS);
        return;
    }
    const int tx = tid & 15, ty = tid >> 4;  // 4 columns x 2 rows per thread
    const float* wa_e = wa + static_cast<size_t>(e) * M * K;
    const float* wb_e = GATED ? wb + static_cast<size_t>(e) * M * K : nullptr;

    for (int r0 = lo + blockIdx.z * kRows; r0 < hi; r0 += gridDim.z * kRows) {
        float acc0[2][4] = {}, acc1[2][4] = {};
        for (int k0 = 0; k0 < K; k0 += kK) {
            for (int i = tid; i < kRows * kK; i += kThreads) {
                const int r = i / kK, c = i % kK;
                sa[r][c] = (r0 + r < hi && k0 + c < K) ? a[static_cast<size_t>(r0 + r) * K + k0 + c] : 0.f;
            }
            for (int i = tid; i < kCols * kK; i += kThreads) {
                const int r = i / kK, c = i % kK;
                const bool ok = m0 + r < M && k0 + c < K;
                sw0[r][c] = ok ? wa_e[static_cast<size_t>(m0 + r) * K + k0 + c] : 0.f;
                if (GATED) sw1[r][c] = ok ? wb_e[static_cast<size_t>(m0 + r) * K + k0 + c] : 0.f;
            }
            __syncthreads();
#pragma unroll 8
            for (int j = 0; j < kK; ++j) {
                const float x0 = sa[ty * 2][j], x1 = sa[ty * 2 + 1][j];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float w0 = sw0[tx * 4 + c][j];
                    acc0[0][c] = fmaf(x0, w0, acc0[0][c]);
                    acc0[1][c] = fmaf(x1, w0, acc0[1][c]);
                    if (GATED) {
                        const float w1 = sw1[tx * 4 + c][j];
                        acc1[0][c] = fmaf(x0, w1, acc1[0][c]);
                        acc1[1][c] = fmaf(x1, w1, acc1[1][c]);
                    }
                }
            }
            __syncthreads();
        }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int row = r0 + ty * 2 + rr;
            if (row >= hi) continue;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int m = m0 + tx * 4 + c;
                if (m >= M) continue;
                float v = acc0[rr][c];
                if (GATED) {
                    const float g = acc0[rr][c];
                    v = g / (1.f + expf(-g)) * acc1[rr][c];
                }
                out[static_cast<size_t>(row) * M + m] = v;
            }
        }
    }
}

// Zero-fills rows offsets[E] .. cap-1 of a [cap][row_elems] fp32 buffer.
__global__ void zero_tail_rows_kernel(float* __restrict__ buf, const int32_t* __restrict__ offsets, int E, int cap,
                                      int row_elems) {
    const int R = offsets[E];
    if (R < 0 || R > cap) return;
    const size_t begin = static_cast<size_t>(R) * row_elems, end = static_cast<size_t>(cap) * row_elems;
    for (size_t i = begin + blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < end;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        buf[i] = 0.f;
}

moe_status launch(bool gated, const float* a, const int32_t* offsets, int cap, int E, int K, int M,
                  const float* wa, const float* wb, float* out, cudaStream_t st, const DeviceInfo& di) {
    // enough row-slices to fill the GPU when few experts are active
    const int col_tiles = (M + kCols - 1) / kCols;
    int zsplit = (2 * di.sm_count + E * col_tiles - 1) / (E * col_tiles);
    const int max_z = (cap + kRows - 1) / kRows;
    zsplit = zsplit < 1 ? 1 : (zsplit > max_z ? max_z : zsplit);
    dim3 grid(col_tiles, E, zsplit);
    if (gated)
        ffn_simt_kernel<true><<<grid, kThreads, 0, st>>>(a, offsets, cap, K, M, wa, wb, out, di.error_word);
    else
        ffn_simt_kernel<false><<<grid, kThreads, 0, st>>>(a, offsets, cap, K, M, wa, wb, out, di.error_word);
    MOE_CUDA_TRY(cudaGetLastError());
    zero_tail_rows_kernel<<<2 * di.sm_count, 256, 0, st>>>(out, offsets, E, cap, M);
    return cuda_status(cudaGetLastError());
}

}  // namespace

moe_status launch_ffn_simt_gate_up(const float* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                   const float* w_gate, const float* w_up, float* h, cudaStream_t st,
                                   const DeviceInfo& di) {
    return launch(true, xs, offsets, cap, E, d, f, w_gate, w_up, h, st, di);
}

moe_status launch_ffn_simt_down(const float* h, const int32_t* offsets, int cap, int E, int d, int f,
                                const float* w_down, float* y, cudaStream_t st, const DeviceInfo& di) {
    return launch(false, h, offsets, cap, E, f, d, w_down, nullptr, y, st, di);
}

}  // namespace moe
