// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Bits of the sticky device error word.
enum : unsigned {
    DEVERR_TIMEOUT = 1u,   // a bounded wait ran out
    DEVERR_OFFSETS = 2u,   // offsets failed the device-side consistency check
    DEVERR_RANGE = 4u,     // a value did not fit the fp16 operands of the FP8-weight path
};

constexpr int kMaxExperts = 256;
constexpr int kMaxK = 16;
// Chunks with T*k <= kSmallRoutes and T <= kSmallTokens can take A1-A4 in one
// launch (moe_route_scatter_small); moe_forward does so.
constexpr int kSmallRoutes = 512;
constexpr int kSmallTokens = 128;

// Workspace layout (int32 words): [0] completion counter, [1..31] reserved,
// then chunk_counts[n_chunks][256] (written by the histogram), local_rank[T*k]
// (histogram), chunk_bases[n_chunks][256] (prefix).  The prefix reads the
// counts and writes the bases elsewhere, so it can be repeated.
// Chunks are token-aligned: chunk c holds the routes of tokens
// [c*ct, (c+1)*ct), ct = ws_chunk_tokens(T), a multiple of 32 chosen so that
// there are at most kMaxChunks chunks (one CTA of the histogram each).
constexpr int kWsHeaderWords = 32;
constexpr int kChunkTokenQuantum = 32;
constexpr int kMaxChunks = 256;
inline int ws_chunk_tokens(int T) {
    const int m = (T + kChunkTokenQuantum * kMaxChunks - 1) / (kChunkTokenQuantum * kMaxChunks);
    return kChunkTokenQuantum * (m > 1 ? m : 1);
}
inline int ws_chunks(int T, int /*k*/) { return (T + ws_chunk_tokens(T) - 1) / ws_chunk_tokens(T); }
inline size_t ws_rank_offset(int T, int k) {
    return kWsHeaderWords + static_cast<size_t>(ws_chunks(T, k)) * kMaxExperts;
}
inline size_t ws_bases_offset(int T, int k) { return ws_rank_offset(T, k) + static_cast<size_t>(T) * k; }
inline size_t ws_words(int T, int k) {
    return ws_bases_offset(T, k) + static_cast<size_t>(ws_chunks(T, k)) * kMaxExperts;
}

#ifdef __CUDACC__
// Order-preserving 64-bit top-k key: high word = the logit's bits mapped so
// that unsigned order equals float order (with -0.0 folded onto +0.0), low
// word = 0xFFFF - expert so that equal logits rank the lower expert first.
// Key 0 is below every real key and marks "taken" or "no expert".
__device__ __forceinline__ unsigned long long topk_order_key(float v, int e) {
    unsigned u = __float_as_uint(v);
    if ((u << 1) == 0u) u = 0u;
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(u) << 32) | static_cast<unsigned>(0xFFFF - e);
}

__device__ __forceinline__ float topk_key_value(unsigned long long key) {
    unsigned u = static_cast<unsigned>(key >> 32);
    u = (u & 0x80000000u) ? (u & 0x7fffffffu) : ~u;
    return __uint_as_float(u);
}
#endif

struct DeviceInfo {
    int sm_count;
    int cc_major, cc_minor;
    int l2_bytes;
    unsigned* error_word;   // device address of the sticky error word
};

// Per-device cache; returns MOE_OK and fills *info for the current device.
// The device addresses in it are those of the current CUDA context.
moe_status device_info(DeviceInfo* info);

// Unique id of the calling thread's current CUDA context (cuCtxGetId), 0
// when no context is current yet.
moe_status current_context_id(unsigned long long* id);

// Records `err` as this thread's last CUDA error and returns MOE_ERR_CUDA
// (or MOE_OK when err == cudaSuccess).
moe_status cuda_status(cudaError_t err);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned128(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 127u) == 0; }

// Slot counters of the fused combine: one per token and 128-feature slice.
inline int tile_counts_per_token(int d) { return (d + 127) / 128; }

inline int dtype_size(int dtype) { return dtype == MOE_BF16 ? 2 : (dtype == MOE_F32 ? 4 : 0); }

// A launch of the bf16 tensor-core grouped FFN kernel (gate/up + SwiGLU, or
// down) prepared on the host: its TMA tensor maps encoded once, with the
// launch arguments.  Replaying it needs no host work beyond the launch.
struct FfnTcLaunch {
    CUtensorMap a0, a1, b, bb;   // weight tiles (gate, up / down twice), rows (64-row and big-item boxes)
    const int32_t* offsets;
    int cap, E, K, M;
    bool narrow, gated;
    void* out;                   // h (bf16) or y (fp32)
};

moe_status prepare_ffn_tc_gate_up(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                  const void* w_gate, const void* w_up, void* h, const DeviceInfo& di,
                                  FfnTcLaunch* p);
moe_status prepare_ffn_tc_down(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                               const void* w_down, float* y, const DeviceInfo& di, FfnTcLaunch* p);
moe_status launch_ffn_tc_prepared(const FfnTcLaunch& p, cudaStream_t st, const DeviceInfo& di);
// The paired-SM kernels (clusters of two CTAs, M = 256 MMAs) for chunks of
// many routes; the tensor maps are the one-SM kernels' (weights: 128-row
// boxes; rows: 16- and 64-row boxes).
bool use_pair_ffn(int cap);
moe_status launch_ffn_pair_prepared(const FfnTcLaunch& p, cudaStream_t st, const DeviceInfo& di);
moe_status launch_ffn_pair_w8a8(bool gated, const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                                const CUtensorMap& bb, const int32_t* offsets, int cap, int E, int K, int M, void* out,
                                const float* sa0, const float* sa1, const float* sb, cudaStream_t st,
                                const DeviceInfo& di);

// Kernel launchers implemented in the other translation units.
moe_status launch_ffn_tc_gate_up(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                 const void* w_gate, const void* w_up, void* h, cudaStream_t st,
                                 const DeviceInfo& di);
moe_status launch_ffn_tc_down(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                              const void* w_down, float* y, cudaStream_t st, const DeviceInfo& di);
moe_status launch_ffn_simt_gate_up(const float* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                   const float* w_gate, const float* w_up, float* h, cudaStream_t st,
                                   const DeviceInfo& di);
moe_status launch_ffn_simt_down(const float* h, const int32_t* offsets, int cap, int E, int d, int f,
                                const float* w_down, float* y, cudaStream_t st, const DeviceInfo& di);

moe_status launch_ffn_tc_gate_up_gather(const void* x, int T, int k, const int32_t* route_of_row,
                                        const int32_t* offsets, int E, int d, int f, const void* w_gate,
                                        const void* w_up, void* h, cudaStream_t st, const DeviceInfo& di);
moe_status launch_ffn_tc_down_combine(const void* h, const int32_t* offsets, int T, int k, int E, int d, int f,
                                      const void* w_down, const int32_t* route_of_row,
                                      const int32_t* row_of_route, const float* w, float* y,
                                      int32_t* tile_counts, float* out, cudaStream_t st, const DeviceInfo& di);

moe_status launch_ffn_fp8_gate_up(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                  const uint8_t* q_gate, const float* s_gate, const uint8_t* q_up, const float* s_up,
                                  void* h, cudaStream_t st, const DeviceInfo& di);
moe_status launch_ffn_fp8_down(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                               const uint8_t* q_down, const float* s_down, float* y, cudaStream_t st,
                               const DeviceInfo& di);
moe_status launch_ffn_w8a8_gate_up(const uint8_t* xs, const float* xs_scale, const int32_t* offsets, int cap, int E,
                                   int d, int f, const uint8_t* q_gate, const float* s_gate, const uint8_t* q_up,
                                   const float* s_up, void* h, cudaStream_t st, const DeviceInfo& di);
moe_status launch_ffn_w8a8_down(const uint8_t* hq, const float* h_scale, const int32_t* offsets, int cap, int E,
                                int d, int f, const uint8_t* q_down, const float* s_down, float* y, cudaStream_t st,
                                const DeviceInfo& di);
moe_status launch_ffn_fp4_gate_up(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                  const uint8_t* q_gate, const uint8_t* b_gate, const float* s_gate,
                                  const uint8_t* q_up, const uint8_t* b_up, const float* s_up, void* h,
                                  cudaStream_t st, const DeviceInfo& di);
moe_status launch_ffn_fp4_down(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                               const uint8_t* q_down, const uint8_t* b_down, const float* s_down, float* y,
                               cudaStream_t st, const DeviceInfo& di);
moe_status launch_quantize_fp4(const void* w, int dtype, int E, int M, int K, uint8_t* codes, uint8_t* block_scales,
                               float* scales, cudaStream_t st, const DeviceInfo& di);
moe_status launch_quantize_rows_fp4(const void* a, int dtype, int rows, int ld, int K, uint8_t* codes,
                                    uint8_t* block_scales, float* scales, cudaStream_t st, const DeviceInfo& di);
moe_status launch_ffn_w4a4_gate_up(const uint8_t* xs, const uint8_t* xs_bs, int ld, const float* xs_s,
                                   const int32_t* offsets, int cap, int E, int d, int f, const uint8_t* q_gate,
                                   const uint8_t* b_gate, const float* s_gate, const uint8_t* q_up,
                                   const uint8_t* b_up, const float* s_up, void* h, cudaStream_t st,
                                   const DeviceInfo& di);
moe_status launch_ffn_w4a4_down(const uint8_t* hq, const uint8_t* h_bs, int ld, const float* h_s,
                                const int32_t* offsets, int cap, int E, int d, int f, const uint8_t* q_down,
                                const uint8_t* b_down, const float* s_down, float* y, cudaStream_t st,
                                const DeviceInfo& di);
moe_status launch_router_topk(const void* x, const void* wr, int T, int E, int d, int k, float* logits,
                              int32_t* ids, float* w, cudaStream_t st, const DeviceInfo& di);
// moe_route_scatter_small for the fused path: xs may be NULL (no row copy);
// tile_counts [T][n_counts] are zeroed and out rows of all-masked tokens set
// to +0.0.
moe_status launch_route_scatter_small_fused(const float* logits, const void* x, const uint8_t* mask, int T, int E,
                                            int k, int d, int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                                            void* xs, int32_t* row_of_route, int32_t* route_of_row,
                                            int32_t* tile_counts, float* out, cudaStream_t st, const DeviceInfo& di);
moe_status launch_quantize_fp8(const void* w, int dtype, long long rows, int K, uint8_t* codes, float* scales,
                               cudaStream_t st, const DeviceInfo& di);

}  // namespace moe

// Host-side argument check helper: returns MOE_ERR_INVALID_ARG from the
// enclosing function when `cond` is false.
#define MOE_REQUIRE(cond)                          \
    do {                                           \
        if (!(cond)) return MOE_ERR_INVALID_ARG;   \
    } while (0)

#define MOE_CUDA_TRY(expr)                                      \
    do {                                                        \
        cudaError_t e_ = (expr);                                \
        if (e_ != cudaSuccess) return ::moe::cuda_status(e_);   \
    } while (0)
