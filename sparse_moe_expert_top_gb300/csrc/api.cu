// C-ABI plumbing: device cache, sticky device error word, status strings,
// grouped FFN dispatch and the whole-path convenience call.

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <new>

#include "moe_internal.cuh"

// Sticky device error word (bits moe::DEVERR_*), one per device that loads
// the library.  Kernels receive its address as an argument.
__device__ unsigned g_moe_device_error;

namespace moe {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
bool g_ready[kMaxDevices];
unsigned long long g_context[kMaxDevices];   // context the cached device addresses belong to
DeviceInfo g_info[kMaxDevices];
thread_local int g_last_cuda_error = 0;

std::once_flag g_ctx_fn_once;
PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;

}  // namespace

moe_status cuda_status(cudaError_t err) {
    if (err == cudaSuccess) return MOE_OK;
    g_last_cuda_error = static_cast<int>(err);
    return MOE_ERR_CUDA;
}

moe_status current_context_id(unsigned long long* id) {
    std::call_once(g_ctx_fn_once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) return MOE_ERR_UNSUPPORTED;
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return cuda_status(cudaErrorUnknown);
    *id = 0;
    if (ctx != nullptr && g_ctx_get_id(ctx, id) != CUDA_SUCCESS) return cuda_status(cudaErrorUnknown);
    return MOE_OK;
}

moe_status device_info(DeviceInfo* info) {
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    unsigned long long ctx = 0;
    moe_status st = current_context_id(&ctx);
    if (st != MOE_OK) return st;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_ready[dev]) {
        DeviceInfo di{};
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev));
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&di.cc_major, cudaDevAttrComputeCapabilityMajor, dev));
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&di.cc_minor, cudaDevAttrComputeCapabilityMinor, dev));
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&di.l2_bytes, cudaDevAttrL2CacheSize, dev));
        if (di.cc_major != 10 || di.cc_minor != 3) return MOE_ERR_UNSUPPORTED;
        g_info[dev] = di;
        g_ready[dev] = true;
    }
    // A device address belongs to one context: after cudaDeviceReset the
    // runtime makes a new primary context and loads the module again, so the
    // address is looked up again whenever the current context is another one
    // (or none was current yet: the lookup itself makes the primary context).
    if (ctx == 0 || g_context[dev] != ctx) {
        void* p = nullptr;
        MOE_CUDA_TRY(cudaGetSymbolAddress(&p, g_moe_device_error));
        if ((st = current_context_id(&ctx)) != MOE_OK) return st;
        g_info[dev].error_word = static_cast<unsigned*>(p);
        g_context[dev] = ctx;
    }
    *info = g_info[dev];
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" int moe_version(void) { return 100; }

extern "C" const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported device or operand type";
        case MOE_ERR_CUDA: return "CUDA call failed";
        case MOE_ERR_TIMEOUT: return "a bounded device wait ran out";
        case MOE_ERR_RANGE: return "a value out of the fp16 operand range";
        default: return "unknown status";
    }
}

extern "C" int moe_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" moe_status moe_check_device_error(void* stream) {
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    unsigned word = 0;
    MOE_CUDA_TRY(cudaMemcpy(&word, di.error_word, sizeof(word), cudaMemcpyDeviceToHost));
    if (word == 0) return MOE_OK;
    const unsigned zero = 0;
    MOE_CUDA_TRY(cudaMemcpy(di.error_word, &zero, sizeof(zero), cudaMemcpyHostToDevice));
    if (word & DEVERR_TIMEOUT) return MOE_ERR_TIMEOUT;
    if (word & DEVERR_OFFSETS) return MOE_ERR_INVALID_ARG;
    return MOE_ERR_RANGE;
}

extern "C" moe_status moe_clear_device_error(void* stream) {
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    return cuda_status(cudaMemsetAsync(di.error_word, 0, sizeof(unsigned), static_cast<cudaStream_t>(stream)));
}

namespace {

moe_status check_ffn_args(const int32_t* offsets, int cap, int E, int d, int f, int dtype) {
    const int es = dtype_size(dtype);
    if (es == 0) return MOE_ERR_UNSUPPORTED;
    MOE_REQUIRE(offsets && cap >= 0 && E >= 1 && E <= kMaxExperts && d >= 1 && f >= 1);
    MOE_REQUIRE((static_cast<size_t>(d) * es) % 16 == 0 && (static_cast<size_t>(f) * es) % 16 == 0);
    if (dtype == MOE_BF16) MOE_REQUIRE(d % 128 == 0 && f % 128 == 0);
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_grouped_gate_up(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                          const void* w_gate, const void* w_up, int dtype, void* h,
                                          void* stream) {
    moe_status st = check_ffn_args(offsets, cap, E, d, f, dtype);
    if (st != MOE_OK) return st;
    if (cap == 0) return MOE_OK;
    MOE_REQUIRE(xs && w_gate && w_up && h);
    MOE_REQUIRE(aligned16(xs) && aligned16(w_gate) && aligned16(w_up) && aligned16(h));
    DeviceInfo di;
    st = device_info(&di);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == MOE_BF16) return launch_ffn_tc_gate_up(xs, offsets, cap, E, d, f, w_gate, w_up, h, s, di);
    return launch_ffn_simt_gate_up(static_cast<const float*>(xs), offsets, cap, E, d, f,
                                   static_cast<const float*>(w_gate), static_cast<const float*>(w_up),
                                   static_cast<float*>(h), s, di);
}

extern "C" moe_status moe_grouped_down(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                                       const void* w_down, int dtype, float* y, void* stream) {
    moe_status st = check_ffn_args(offsets, cap, E, d, f, dtype);
    if (st != MOE_OK) return st;
    if (cap == 0) return MOE_OK;
    MOE_REQUIRE(h && w_down && y);
    MOE_REQUIRE(aligned16(h) && aligned16(w_down) && aligned16(y));
    DeviceInfo di;
    st = device_info(&di);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == MOE_BF16) return launch_ffn_tc_down(h, offsets, cap, E, d, f, w_down, y, s, di);
    return launch_ffn_simt_down(static_cast<const float*>(h), offsets, cap, E, d, f,
                                static_cast<const float*>(w_down), y, s, di);
}

extern "C" moe_status moe_grouped_ffn(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                      const void* w_gate, const void* w_up, const void* w_down, int dtype,
                                      void* h, float* y, void* stream) {
    moe_status st = moe_grouped_gate_up(xs, offsets, cap, E, d, f, w_gate, w_up, dtype, h, stream);
    if (st != MOE_OK) return st;
    return moe_grouped_down(h, offsets, cap, E, d, f, w_down, dtype, y, stream);
}

extern "C" moe_status moe_forward(const float* logits, const void* x, const uint8_t* mask, int T, int E, int k,
                                  int d, int f, const void* w_gate, const void* w_up, const void* w_down, int dtype,
                                  int32_t* ids, float* w, int32_t* counts, int32_t* offsets, void* xs,
                                  int32_t* row_of_route, int32_t* route_of_row, void* h, float* y, float* out,
                                  void* ws, void* stream) {
    // validate everything before the first launch so that a bad argument
    // enqueues nothing
    moe_status st = check_ffn_args(offsets, T * k, E, d, f, dtype);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= kMaxK && k <= E && d % 4 == 0);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && x && w_gate && w_up && w_down && ids && w && counts && xs && row_of_route &&
                route_of_row && h && y && out && ws);
    MOE_REQUIRE(aligned16(x) && aligned16(xs) && aligned16(h) && aligned16(y) && aligned16(out) &&
                aligned16(ws) && aligned16(w_gate) && aligned16(w_up) && aligned16(w_down));
    const int cap = T * k;
    if (T <= kSmallTokens && cap <= kSmallRoutes) {
        if ((st = moe_route_scatter_small(logits, x, dtype, 0, mask, T, E, k, d, ids, w, counts, offsets, xs,
                                          row_of_route, route_of_row, stream)) != MOE_OK)
            return st;
    } else {
        if ((st = moe_route_topk_offsets(logits, mask, T, E, k, ids, w, counts, offsets, ws, stream)) != MOE_OK)
            return st;
        if ((st = moe_scatter_rows(x, dtype, ids, mask, offsets, T, k, d, E, xs, row_of_route, route_of_row, ws,
                                   stream)) != MOE_OK)
            return st;
    }
    if ((st = moe_grouped_ffn(xs, offsets, cap, E, d, f, w_gate, w_up, w_down, dtype, h, y, stream)) != MOE_OK)
        return st;
    return moe_combine(y, row_of_route, w, T, k, d, out, stream);
}

// ---------------------------------------------------------------------------
// FP8 E4M3 expert weights
// ---------------------------------------------------------------------------

extern "C" moe_status moe_quantize_weights_fp8(const void* w, int dtype, long long rows, int K, uint8_t* codes,
                                               float* scales, void* stream) {
    if (dtype_size(dtype) == 0) return MOE_ERR_UNSUPPORTED;
    MOE_REQUIRE(rows >= 0 && K >= 16 && K % 16 == 0);
    if (rows == 0) return MOE_OK;
    MOE_REQUIRE(w && codes && scales && aligned16(w) && aligned16(codes));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    return launch_quantize_fp8(w, dtype, rows, K, codes, scales, static_cast<cudaStream_t>(stream), di);
}

extern "C" moe_status moe_grouped_gate_up_fp8(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                              const uint8_t* w_gate_q, const float* s_gate, const uint8_t* w_up_q,
                                              const float* s_up, void* h, void* stream) {
    moe_status st = check_ffn_args(offsets, cap, E, d, f, MOE_BF16);
    if (st != MOE_OK) return st;
    if (cap == 0) return MOE_OK;
    MOE_REQUIRE(xs && w_gate_q && s_gate && w_up_q && s_up && h);
    MOE_REQUIRE(aligned16(xs) && aligned16(w_gate_q) && aligned16(w_up_q) && aligned16(h));
    DeviceInfo di;
    st = device_info(&di);
    if (st != MOE_OK) return st;
    return launch_ffn_fp8_gate_up(xs, offsets, cap, E, d, f, w_gate_q, s_gate, w_up_q, s_up, h,
                                  static_cast<cudaStream_t>(stream), di);
}

extern "C" moe_status moe_grouped_down_fp8(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                                           const uint8_t* w_down_q, const float* s_down, float* y, void* stream) {
    moe_status st = check_ffn_args(offsets, cap, E, d, f, MOE_BF16);
    if (st != MOE_OK) return st;
    if (cap == 0) return MOE_OK;
    MOE_REQUIRE(h && w_down_q && s_down && y);
    MOE_REQUIRE(aligned16(h) && aligned16(w_down_q) && aligned16(y));
    DeviceInfo di;
    st = device_info(&di);
    if (st != MOE_OK) return st;
    return launch_ffn_fp8_down(h, offsets, cap, E, d, f, w_down_q, s_down, y, static_cast<cudaStream_t>(stream), di);
}

extern "C" moe_status moe_grouped_ffn_fp8(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                          const uint8_t* w_gate_q, const float* s_gate, const uint8_t* w_up_q,
                                          const float* s_up, const uint8_t* w_down_q, const float* s_down, void* h,
                                          float* y, void* stream) {
    moe_status st = moe_grouped_gate_up_fp8(xs, offsets, cap, E, d, f, w_gate_q, s_gate, w_up_q, s_up, h, stream);
    if (st != MOE_OK) return st;
    return moe_grouped_down_fp8(h, offsets, cap, E, d, f, w_down_q, s_down, y, stream);
}

extern "C" moe_status moe_forward_fp8(const float* logits, const void* x, const uint8_t* mask, int T, int E, int k,
                                      int d, int f, const uint8_t* w_gate_q, const float* s_gate,
                                      const uint8_t* w_up_q, const float* s_up, const uint8_t* w_down_q,
                                      const float* s_down, int32_t* ids, float* w, int32_t* counts,
                                      int32_t* offsets, void* xs, int32_t* row_of_route, int32_t* route_of_row,
                                      void* h, float* y, float* out, void* ws, void* stream) {
    moe_status st = check_ffn_args(offsets, T * k, E, d, f, MOE_BF16);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= kMaxK && k <= E);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && x && w_gate_q && s_gate && w_up_q && s_up && w_down_q && s_down && ids && w && counts &&
                xs && row_of_route && route_of_row && h && y && out && ws);
    MOE_REQUIRE(aligned16(x) && aligned16(xs) && aligned16(h) && aligned16(y) && aligned16(out) &&
                aligned16(ws) && aligned16(w_gate_q) && aligned16(w_up_q) && aligned16(w_down_q));
    const int cap = T * k;
    if (T <= kSmallTokens && cap <= kSmallRoutes) {
        if ((st = moe_route_scatter_small(logits, x, MOE_BF16, 1, mask, T, E, k, d, ids, w, counts, offsets, xs,
                                          row_of_route, route_of_row, stream)) != MOE_OK)
            return st;
    } else {
        if ((st = moe_route_topk_offsets(logits, mask, T, E, k, ids, w, counts, offsets, ws, stream)) != MOE_OK)
            return st;
        if ((st = moe_scatter_rows_f16(x, ids, mask, offsets, T, k, d, E, xs, row_of_route, route_of_row, ws,
                                       stream)) != MOE_OK)
            return st;
    }
    if ((st = moe_grouped_ffn_fp8(xs, offsets, cap, E, d, f, w_gate_q, s_gate, w_up_q, s_up, w_down_q, s_down, h, y,
                                  stream)) != MOE_OK)
        return st;
    return moe_combine(y, row_of_route, w, T, k, d, out, stream);
}

// ---------------------------------------------------------------------------
// 4-bit block-scaled expert weights
// ---------------------------------------------------------------------------

extern "C" moe_status moe_quantize_weights_fp4(const void* w, int dtype, int E, int M, int K, uint8_t* codes,
                                               uint8_t* block_scales, float* scales, void* stream) {
    if (dtype_size(dtype) == 0) return MOE_ERR_UNSUPPORTED;
    MOE_REQUIRE(E >= 0 && M >= 0 && K >= 64 && K % 64 == 0);
    if (static_cast<long long>(E) * M == 0) return MOE_OK;
    MOE_REQUIRE(w && codes && block_scales && scales && aligned16(w) && aligned16(codes) && aligned16(block_scales));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    return launch_quantize_fp4(w, dtype, E, M, K, codes, block_scales, scales, static_cast<cudaStream_t>(stream), di);
}

extern "C" moe_status moe_grouped_gate_up_fp4(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                              const uint8_t* w_gate_q, const uint8_t* b_gate, const float* s_gate,
                                              const uint8_t* w_up_q, const uint8_t* b_up, const float* s_up, void* h,
                                              void* stream) {
    moe_status st = check_ffn_args(offsets, cap, E, d, f, MOE_BF16);
    if (st != MOE_OK) return st;
    if (cap == 0) return MOE_OK;
    MOE_REQUIRE(xs && w_gate_q && b_gate && s_gate && w_up_q && b_up && s_up && h);
    MOE_REQUIRE(aligned16(xs) && aligned16(w_gate_q) && aligned16(w_up_q) && aligned16(b_gate) && aligned16(b_up) &&
                aligned16(h));
    DeviceInfo di;
    if ((st = device_info(&di)) != MOE_OK) return st;
    return launch_ffn_fp4_gate_up(xs, offsets, cap, E, d, f, w_gate_q, b_gate, s_gate, w_up_q, b_up, s_up, h,
                                  static_cast<cudaStream_t>(stream), di);
}

extern "C" moe_status moe_grouped_down_fp4(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                                           const uint8_t* w_down_q, const uint8_t* b_down, const float* s_down,
                                           float* y, void* stream) {
    moe_status st = check_ffn_args(offsets, cap, E, d, f, MOE_BF16);
    if (st != MOE_OK) return st;
    if (cap == 0) return MOE_OK;
    MOE_REQUIRE(h && w_down_q && b_down && s_down && y);
    MOE_REQUIRE(aligned16(h) && aligned16(w_down_q) && aligned16(b_down) && aligned16(y));
    DeviceInfo di;
    if ((st = device_info(&di)) != MOE_OK) return st;
    return launch_ffn_fp4_down(h, offsets, cap, E, d, f, w_down_q, b_down, s_down, y,
                               static_cast<cudaStream_t>(stream), di);
}

extern "C" moe_status moe_forward_fp4(const float* logits, const void* x, const uint8_t* mask, int T, int E, int k,
                                      int d, int f, const uint8_t* w_gate_q, const uint8_t* b_gate,
                                      const float* s_gate, const uint8_t* w_up_q, const uint8_t* b_up,
                                      const float* s_up, const uint8_t* w_down_q, const uint8_t* b_down,
                                      const float* s_down, int32_t* ids, float* w, int32_t* counts,
                                      int32_t* offsets, void* xs, int32_t* row_of_route, int32_t* route_of_row,
                                      void* h, float* y, float* out, void* ws, void* stream) {
    moe_status st = check_ffn_args(offsets, T * k, E, d, f, MOE_BF16);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= kMaxK && k <= E);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && x && ids && w && counts && xs && row_of_route && route_of_row && h && y && out && ws);
    const int cap = T * k;
    if (T <= kSmallTokens && cap <= kSmallRoutes) {
        if ((st = moe_route_scatter_small(logits, x, MOE_BF16, 1, mask, T, E, k, d, ids, w, counts, offsets, xs,
                                          row_of_route, route_of_row, stream)) != MOE_OK)
            return st;
    } else {
        if ((st = moe_route_topk_offsets(logits, mask, T, E, k, ids, w, counts, offsets, ws, stream)) != MOE_OK)
            return st;
        if ((st = moe_scatter_rows_f16(x, ids, mask, offsets, T, k, d, E, xs, row_of_route, route_of_row, ws,
                                       stream)) != MOE_OK)
            return st;
    }
    if ((st = moe_grouped_gate_up_fp4(xs, offsets, cap, E, d, f, w_gate_q, b_gate, s_gate, w_up_q, b_up, s_up, h,
                                      stream)) != MOE_OK)
        return st;
    if ((st = moe_grouped_down_fp4(h, offsets, cap, E, d, f, w_down_q, b_down, s_down, y, stream)) != MOE_OK)
        return st;
    return moe_combine(y, row_of_route, w, T, k, d, out, stream);
}

// ---------------------------------------------------------------------------
// FP8 E4M3 weights and activations (kind::f8f6f4 tensor-core MMAs)
// ---------------------------------------------------------------------------

namespace {

moe_status check_w8a8_args(const int32_t* offsets, int cap, int E, int d, int f) {
    MOE_REQUIRE(offsets && cap >= 0 && E >= 1 && E <= kMaxExperts && d >= 128 && f >= 128);
    MOE_REQUIRE(d % 128 == 0 && f % 128 == 0);
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_grouped_gate_up_w8a8(const uint8_t* xs, const float* xs_scales, const int32_t* offsets,
                                               int cap, int E, int d, int f, const uint8_t* w_gate_q,
                                               const float* s_gate, const uint8_t* w_up_q, const float* s_up,
                                               void* h, void* stream) {
    moe_status st = check_w8a8_args(offsets, cap, E, d, f);
    if (st != MOE_OK) return st;
    if (cap == 0) return MOE_OK;
    MOE_REQUIRE(xs && xs_scales && w_gate_q && s_gate && w_up_q && s_up && h);
    MOE_REQUIRE(aligned16(xs) && aligned16(w_gate_q) && aligned16(w_up_q) && aligned16(h));
    DeviceInfo di;
    if ((st = device_info(&di)) != MOE_OK) return st;
    return launch_ffn_w8a8_gate_up(xs, xs_scales, offsets, cap, E, d, f, w_gate_q, s_gate, w_up_q, s_up, h,
                                   static_cast<cudaStream_t>(stream), di);
}

extern "C" moe_status moe_grouped_down_w8a8(const uint8_t* h_q, const float* h_scales, const int32_t* offsets,
                                            int cap, int E, int d, int f, const uint8_t* w_down_q,
                                            const float* s_down, float* y, void* stream) {
    moe_status st = check_w8a8_args(offsets, cap, E, d, f);
    if (st != MOE_OK) return st;
    if (cap == 0) return MOE_OK;
    MOE_REQUIRE(h_q && h_scales && w_down_q && s_down && y);
    MOE_REQUIRE(aligned16(h_q) && aligned16(w_down_q) && aligned16(y));
    DeviceInfo di;
    if ((st = device_info(&di)) != MOE_OK) return st;
    return launch_ffn_w8a8_down(h_q, h_scales, offsets, cap, E, d, f, w_down_q, s_down, y,
                                static_cast<cudaStream_t>(stream), di);
}

extern "C" moe_status moe_forward_w8a8(const float* logits, const void* x, const uint8_t* mask, int T, int E, int k,
                                       int d, int f, const uint8_t* w_gate_q, const float* s_gate,
                                       const uint8_t* w_up_q, const float* s_up, const uint8_t* w_down_q,
                                       const float* s_down, int32_t* ids, float* w, int32_t* counts,
                                       int32_t* offsets, uint8_t* x_q, float* x_scales, uint8_t* xs,
                                       float* xs_scales, int32_t* row_of_route, int32_t* route_of_row, void* h,
                                       uint8_t* h_q, float* h_scales, float* y, float* out, void* ws,
                                       void* stream) {
    moe_status st = check_w8a8_args(offsets, T * k, E, d, f);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= kMaxK && k <= E);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && x && ids && w && counts && x_q && x_scales && xs && xs_scales && row_of_route &&
                route_of_row && h && h_q && h_scales && y && out && ws);
    MOE_REQUIRE(aligned16(x) && aligned16(x_q) && aligned16(xs) && aligned16(h) && aligned16(h_q) &&
                aligned16(y) && aligned16(out) && aligned16(ws));
    const int cap = T * k;
    if (T <= kSmallTokens && cap <= kSmallRoutes) {
        // small chunks: routing, quantization and scatter in one launch
        if ((st = moe_route_scatter_quant_small_e4m3(logits, x, mask, T, E, k, d, ids, w, counts, offsets, x_q,
                                                     x_scales, xs, xs_scales, row_of_route, route_of_row, stream)) !=
            MOE_OK)
            return st;
    } else if ((st = moe_route_topk_offsets(logits, mask, T, E, k, ids, w, counts, offsets, ws, stream)) != MOE_OK) {
        return st;
    } else if (d <= 8 * 128 * 8) {
        // E4M3 codes of the token rows, one scale per row (the weights' quantizer's arithmetic), scattered
        if ((st = moe_scatter_rows_quant_e4m3(x, ids, mask, offsets, T, k, d, E, x_q, x_scales, xs, xs_scales,
                                              row_of_route, route_of_row, ws, stream)) != MOE_OK)
            return st;
    } else {
        if ((st = moe_quantize_weights_fp8(x, MOE_BF16, T, d, x_q, x_scales, stream)) != MOE_OK) return st;
        if ((st = moe_scatter_rows_e4m3(x_q, x_scales, ids, mask, offsets, T, k, d, E, xs, xs_scales, row_of_route,
                                        route_of_row, ws, stream)) != MOE_OK)
            return st;
    }
    if ((st = moe_grouped_gate_up_w8a8(xs, xs_scales, offsets, cap, E, d, f, w_gate_q, s_gate, w_up_q, s_up, h,
                                       stream)) != MOE_OK)
        return st;
    // E4M3 codes of the rows of h (bf16), one scale per row
    if (f <= 8 * 32 * 8)
        st = moe_quantize_rows_e4m3(h, offsets, E, cap, f, h_q, h_scales, stream);
    else
        st = moe_quantize_weights_fp8(h, MOE_BF16, cap, f, h_q, h_scales, stream);
    if (st != MOE_OK) return st;
    if ((st = moe_grouped_down_w8a8(h_q, h_scales, offsets, cap, E, d, f, w_down_q, s_down, y, stream)) != MOE_OK)
        return st;
    return moe_combine(y, row_of_route, w, T, k, d, out, stream);
}

// ---------------------------------------------------------------------------
// 4-bit operands on both sides (block-scaled tensor-core MMAs)
// ---------------------------------------------------------------------------

extern "C" moe_status moe_quantize_rows_fp4(const void* a, int dtype, int rows, int ld, int K, uint8_t* codes,
                                            uint8_t* block_scales, float* scales, void* stream) {
    if (dtype_size(dtype) == 0) return MOE_ERR_UNSUPPORTED;
    MOE_REQUIRE(rows >= 0 && ld >= rows && ld % 4 == 0 && K >= 64 && K % 64 == 0);
    if (rows == 0) return MOE_OK;
    MOE_REQUIRE(a && codes && block_scales && scales && aligned16(a) && aligned16(codes) && aligned16(block_scales));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    return launch_quantize_rows_fp4(a, dtype, rows, ld, K, codes, block_scales, scales,
                                    static_cast<cudaStream_t>(stream), di);
}

namespace {
int rows_ld(int rows) { return (rows + 3) / 4 * 4; }
}  // namespace

extern "C" moe_status moe_grouped_gate_up_w4a4(const uint8_t* xs_codes, const uint8_t* xs_block_scales, int ld,
                                               const float* xs_scales, const int32_t* offsets, int cap, int E, int d,
                                               int f, const uint8_t* w_gate_q, const uint8_t* b_gate,
                                               const float* s_gate, const uint8_t* w_up_q, const uint8_t* b_up,
                                               const float* s_up, void* h, void* stream) {
    moe_status st = check_w8a8_args(offsets, cap, E, d, f);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(ld >= cap && ld % 4 == 0);
    if (cap == 0) return MOE_OK;
    MOE_REQUIRE(xs_codes && xs_block_scales && xs_scales && w_gate_q && b_gate && s_gate && w_up_q && b_up && s_up &&
                h);
    MOE_REQUIRE(aligned16(xs_codes) && aligned16(xs_block_scales) && aligned16(w_gate_q) && aligned16(b_gate) &&
                aligned16(w_up_q) && aligned16(b_up) && aligned16(h));
    DeviceInfo di;
    if ((st = device_info(&di)) != MOE_OK) return st;
    return launch_ffn_w4a4_gate_up(xs_codes, xs_block_scales, ld, xs_scales, offsets, cap, E, d, f, w_gate_q, b_gate,
                                   s_gate, w_up_q, b_up, s_up, h, static_cast<cudaStream_t>(stream), di);
}

extern "C" moe_status moe_grouped_down_w4a4(const uint8_t* h_codes, const uint8_t* h_block_scales, int ld,
                                            const float* h_scales, const int32_t* offsets, int cap, int E, int d,
                                            int f, const uint8_t* w_down_q, const uint8_t* b_down,
                                            const float* s_down, float* y, void* stream) {
    moe_status st = check_w8a8_args(offsets, cap, E, d, f);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(ld >= cap && ld % 4 == 0);
    if (cap == 0) return MOE_OK;
    MOE_REQUIRE(h_codes && h_block_scales && h_scales && w_down_q && b_down && s_down && y);
    MOE_REQUIRE(aligned16(h_codes) && aligned16(h_block_scales) && aligned16(w_down_q) && aligned16(b_down) &&
                aligned16(y));
    DeviceInfo di;
    if ((st = device_info(&di)) != MOE_OK) return st;
    return launch_ffn_w4a4_down(h_codes, h_block_scales, ld, h_scales, offsets, cap, E, d, f, w_down_q, b_down, s_down,
                                y, static_cast<cudaStream_t>(stream), di);
}

extern "C" moe_status moe_forward_w4a4(const float* logits, const void* x, const uint8_t* mask, int T, int E, int k,
                                       int d, int f, const uint8_t* w_gate_q, const uint8_t* b_gate,
                                       const float* s_gate, const uint8_t* w_up_q, const uint8_t* b_up,
                                       const float* s_up, const uint8_t* w_down_q, const uint8_t* b_down,
                                       const float* s_down, int32_t* ids, float* w, int32_t* counts,
                                       int32_t* offsets, uint8_t* x_codes, uint8_t* x_block_scales,
                                       float* x_scales, uint8_t* xs_codes, uint8_t* xs_block_scales,
                                       float* xs_scales, int32_t* row_of_route, int32_t* route_of_row, void* h,
                                       uint8_t* h_codes, uint8_t* h_block_scales, float* h_scales, float* y,
                                       float* out, void* ws, void* stream) {
    moe_status st = check_w8a8_args(offsets, T * k, E, d, f);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= kMaxK && k <= E);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && x && ids && w && counts && x_codes && x_block_scales && x_scales && xs_codes &&
                xs_block_scales && xs_scales && row_of_route && route_of_row && h && h_codes && h_block_scales &&
                h_scales && y && out && ws);
    MOE_REQUIRE(aligned16(x) && aligned16(h) && aligned16(y) && aligned16(out) && aligned16(ws));
    const int cap = T * k;
    if (T <= kSmallTokens && cap <= kSmallRoutes) {
        // small chunks: routing, quantization and scatter in one launch
        if ((st = moe_route_scatter_quant_small_fp4(logits, x, mask, T, E, k, d, ids, w, counts, offsets, x_codes,
                                                    x_block_scales, rows_ld(T), x_scales, xs_codes, xs_block_scales,
                                                    rows_ld(cap), xs_scales, row_of_route, route_of_row, stream)) !=
            MOE_OK)
            return st;
    } else if ((st = moe_route_topk_offsets(logits, mask, T, E, k, ids, w, counts, offsets, ws, stream)) != MOE_OK) {
        return st;
    } else if (d <= 4 * 128 * 16) {
        // 4-bit token rows, scattered to the compact rows (one kernel up to d = 8192)
        if ((st = moe_scatter_rows_quant_fp4(x, ids, mask, offsets, T, k, d, E, x_codes, x_block_scales, rows_ld(T),
                                             x_scales, xs_codes, xs_block_scales, rows_ld(cap), xs_scales,
                                             row_of_route, route_of_row, ws, stream)) != MOE_OK)
            return st;
    } else {
        if ((st = moe_quantize_rows_fp4(x, MOE_BF16, T, rows_ld(T), d, x_codes, x_block_scales, x_scales, stream)) !=
            MOE_OK)
            return st;
        if ((st = moe_scatter_rows_fp4(x_codes, x_block_scales, rows_ld(T), x_scales, ids, mask, offsets, T, k, d, E,
                                       xs_codes, xs_block_scales, rows_ld(cap), xs_scales, row_of_route,
                                       route_of_row, ws, stream)) != MOE_OK)
            return st;
    }
    if ((st = moe_grouped_gate_up_w4a4(xs_codes, xs_block_scales, rows_ld(cap), xs_scales, offsets, cap, E, d, f,
                                       w_gate_q, b_gate, s_gate, w_up_q, b_up, s_up, h, stream)) != MOE_OK)
        return st;
    // NVFP4 rows of h (bf16; the unused rows are zero and quantize to zero codes)
    if ((st = moe_quantize_rows_fp4(h, MOE_BF16, cap, rows_ld(cap), f, h_codes, h_block_scales, h_scales, stream)) !=
        MOE_OK)
        return st;
    if ((st = moe_grouped_down_w4a4(h_codes, h_block_scales, rows_ld(cap), h_scales, offsets, cap, E, d, f, w_down_q,
                                    b_down, s_down, y, stream)) != MOE_OK)
        return st;
    return moe_combine(y, row_of_route, w, T, k, d, out, stream);
}

// ---------------------------------------------------------------------------
// Fused permutation (bf16)
// ---------------------------------------------------------------------------

extern "C" moe_status moe_grouped_gate_up_gather(const void* x, int T, int k, const int32_t* route_of_row,
                                                 const int32_t* offsets, int E, int d, int f, const void* w_gate,
                                                 const void* w_up, void* h, void* stream) {
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= kMaxK && static_cast<long long>(T) * k < (1ll << 30));
    moe_status st = check_ffn_args(offsets, T * k, E, d, f, MOE_BF16);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(x && route_of_row && w_gate && w_up && h);
    MOE_REQUIRE(aligned16(x) && aligned16(w_gate) && aligned16(w_up) && aligned16(h));
    DeviceInfo di;
    st = device_info(&di);
    if (st != MOE_OK) return st;
    return launch_ffn_tc_gate_up_gather(x, T, k, route_of_row, offsets, E, d, f, w_gate, w_up, h,
                                        static_cast<cudaStream_t>(stream), di);
}

extern "C" moe_status moe_grouped_down_combine(const void* h, const int32_t* offsets, int T, int k, int E, int d,
                                               int f, const void* w_down, const int32_t* route_of_row,
                                               const int32_t* row_of_route, const float* w, float* y,
                                               int32_t* tile_counts, float* out, void* stream) {
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= kMaxK && static_cast<long long>(T) * k < (1ll << 30));
    moe_status st = check_ffn_args(offsets, T * k, E, d, f, MOE_BF16);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(h && w_down && route_of_row && row_of_route && w && y && tile_counts && out);
    MOE_REQUIRE(aligned16(h) && aligned16(w_down) && aligned128(y) && aligned16(out));
    DeviceInfo di;
    st = device_info(&di);
    if (st != MOE_OK) return st;
    return launch_ffn_tc_down_combine(h, offsets, T, k, E, d, f, w_down, route_of_row, row_of_route, w, y,
                                      tile_counts, out, static_cast<cudaStream_t>(stream), di);
}

// moe_forward_fused's automatic mode: gather the token rows inside the
// gate/up kernel while the chunk averages at most this many routes per expert
// (above it the compact copy's large TMA boxes are cheaper than per-row
// copies), and fuse the combine into the down kernel while y (T*k*d fp32,
// the exchange between the CTAs that own a token's slots) fits in twice the
// L2; above that the separate combine kernel is faster.
#ifndef MOE_FUSED_GATHER_MAX_ROUTES_PER_EXPERT
#define MOE_FUSED_GATHER_MAX_ROUTES_PER_EXPERT 16
#endif

namespace {

int fused_auto_mode(long long cap, int E, int d, bool have_xs, const DeviceInfo& di) {
    if (!have_xs || cap <= static_cast<long long>(E) * MOE_FUSED_GATHER_MAX_ROUTES_PER_EXPERT)
        return MOE_FUSED_GATHER;
    if (cap * d * 4 <= 2LL * di.l2_bytes) return MOE_FUSED_COMPACT;
    return MOE_FUSED_NONE;
}

}  // namespace

extern "C" moe_status moe_ffn_paired(int cap, int* paired) {
    MOE_REQUIRE(paired && cap >= 0);
    *paired = use_pair_ffn(cap) ? 1 : 0;
    return MOE_OK;
}

extern "C" moe_status moe_forward_fused_mode(int T, int E, int k, int d, int have_xs, int* mode) {
    MOE_REQUIRE(mode && T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E && d >= 1);
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    *mode = fused_auto_mode(static_cast<long long>(T) * k, E, d, have_xs != 0, di);
    return MOE_OK;
}

extern "C" moe_status moe_forward_fused(const float* logits, const void* x, const uint8_t* mask, int T, int E,
                                        int k, int d, int f, const void* w_gate, const void* w_up,
                                        const void* w_down, int mode, int32_t* ids, float* w, int32_t* counts,
                                        int32_t* offsets, void* xs, int32_t* row_of_route, int32_t* route_of_row,
                                        void* h, float* y, int32_t* tile_counts, float* out, void* ws,
                                        void* stream) {
    moe_status st = check_ffn_args(offsets, T * k, E, d, f, MOE_BF16);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= kMaxK && k <= E);
    MOE_REQUIRE(mode == MOE_FUSED_AUTO || mode == MOE_FUSED_GATHER || mode == MOE_FUSED_COMPACT ||
                mode == MOE_FUSED_NONE);
    MOE_REQUIRE((mode != MOE_FUSED_COMPACT && mode != MOE_FUSED_NONE) || xs != nullptr);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && x && w_gate && w_up && w_down && ids && w && counts && row_of_route && route_of_row && h &&
                y && tile_counts && out && ws);
    MOE_REQUIRE(aligned16(x) && aligned16(h) && aligned128(y) && aligned16(out) && aligned16(ws) &&
                aligned16(w_gate) && aligned16(w_up) && aligned16(w_down) && (xs == nullptr || aligned16(xs)));
    DeviceInfo di;
    st = device_info(&di);
    if (st != MOE_OK) return st;
    const long long cap = static_cast<long long>(T) * k;
    if (mode == MOE_FUSED_AUTO) mode = fused_auto_mode(cap, E, d, xs != nullptr, di);
    if (mode == MOE_FUSED_NONE)
        return moe_forward(logits, x, mask, T, E, k, d, f, w_gate, w_up, w_down, MOE_BF16, ids, w, counts, offsets, xs,
                           row_of_route, route_of_row, h, y, out, ws, stream);
    const bool gather = mode == MOE_FUSED_GATHER;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T <= kSmallTokens && cap <= kSmallRoutes) {
        // A1-A4 in one launch, with the fused combine's preparation
        if ((st = launch_route_scatter_small_fused(logits, x, mask, T, E, k, d, ids, w, counts, offsets,
                                                   gather ? nullptr : xs, row_of_route, route_of_row, tile_counts,
                                                   out, s, di)) != MOE_OK)
            return st;
    } else {
        if ((st = moe_route_topk_offsets(logits, mask, T, E, k, ids, w, counts, offsets, ws, stream)) != MOE_OK)
            return st;
        if ((st = moe_scatter_index(ids, mask, offsets, T, k, d, E, gather ? nullptr : x, gather ? nullptr : xs,
                                    row_of_route, route_of_row, tile_counts, out, ws, stream)) != MOE_OK)
            return st;
    }
    if (gather)
        st = moe_grouped_gate_up_gather(x, T, k, route_of_row, offsets, E, d, f, w_gate, w_up, h, stream);
    else
        st = moe_grouped_gate_up(xs, offsets, T * k, E, d, f, w_gate, w_up, MOE_BF16, h, stream);
    if (st != MOE_OK) return st;
    return moe_grouped_down_combine(h, offsets, T, k, E, d, f, w_down, route_of_row, row_of_route, w, y,
                                    tile_counts, out, stream);
}

// ---------------------------------------------------------------------------
// Router projection + top-k
// ---------------------------------------------------------------------------

extern "C" moe_status moe_router_topk(const void* x, const void* wr, int T, int E, int d, int k, float* logits,
                                      int32_t* ids, float* w, void* stream) {
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E && d >= 64 && d % 64 == 0);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(x && wr && ids && w && aligned16(x) && aligned16(wr));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    return launch_router_topk(x, wr, T, E, d, k, logits, ids, w, static_cast<cudaStream_t>(stream), di);
}

// ---------------------------------------------------------------------------
// Plans: the path for fixed shapes, weights and buffers, prepared once
// ---------------------------------------------------------------------------

struct moe_plan {
    int device;
    unsigned long long context;
    int T, E, k, d, f, dtype;
    const void *w_gate, *w_up, *w_down;
    int32_t* ids;
    float* w;
    int32_t *counts, *offsets;
    void* xs;
    int32_t *row_of_route, *route_of_row;
    void* h;
    float* y;
    void* ws;
    moe::DeviceInfo di;
    moe::FfnTcLaunch gate_up, down;   // bf16: the tensor maps, encoded once
};

extern "C" moe_status moe_plan_create(int T, int E, int k, int d, int f, int dtype, const void* w_gate,
                                      const void* w_up, const void* w_down, int32_t* ids, float* w,
                                      int32_t* counts, int32_t* offsets, void* xs, int32_t* row_of_route,
                                      int32_t* route_of_row, void* h, float* y, void* ws, moe_plan** plan) {
    MOE_REQUIRE(plan != nullptr);
    *plan = nullptr;
    moe_status st = check_ffn_args(offsets, T * k, E, d, f, dtype);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(T >= 1 && k >= 1 && k <= kMaxK && k <= E && d % 4 == 0);
    MOE_REQUIRE(static_cast<long long>(T) * k < (1ll << 30));
    MOE_REQUIRE(w_gate && w_up && w_down && ids && w && counts && xs && row_of_route && route_of_row && h && y &&
                ws);
    MOE_REQUIRE(aligned16(xs) && aligned16(h) && aligned16(y) && aligned16(ws) && aligned16(w_gate) &&
                aligned16(w_up) && aligned16(w_down));
    moe_plan p{};
    MOE_CUDA_TRY(cudaGetDevice(&p.device));
    if ((st = device_info(&p.di)) != MOE_OK) return st;
    if ((st = current_context_id(&p.context)) != MOE_OK) return st;
    p.T = T;
    p.E = E;
    p.k = k;
    p.d = d;
    p.f = f;
    p.dtype = dtype;
    p.w_gate = w_gate;
    p.w_up = w_up;
    p.w_down = w_down;
    p.ids = ids;
    p.w = w;
    p.counts = counts;
    p.offsets = offsets;
    p.xs = xs;
    p.row_of_route = row_of_route;
    p.route_of_row = route_of_row;
    p.h = h;
    p.y = y;
    p.ws = ws;
    if (dtype == MOE_BF16) {
        const int cap = T * k;
        if ((st = prepare_ffn_tc_gate_up(xs, offsets, cap, E, d, f, w_gate, w_up, h, p.di, &p.gate_up)) != MOE_OK)
            return st;
        if ((st = prepare_ffn_tc_down(h, offsets, cap, E, d, f, w_down, y, p.di, &p.down)) != MOE_OK) return st;
    }
    moe_plan* heap = new (std::nothrow) moe_plan(p);
    if (heap == nullptr) return MOE_ERR_CUDA;
    *plan = heap;
    return MOE_OK;
}

extern "C" moe_status moe_plan_destroy(moe_plan* plan) {
    delete plan;
    return MOE_OK;
}

namespace {

// The plan belongs to the device and context it was made in.
moe_status check_plan(const moe_plan* plan) {
    MOE_REQUIRE(plan != nullptr);
    int dev = -1;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    unsigned long long ctx = 0;
    moe_status st = current_context_id(&ctx);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(dev == plan->device && ctx == plan->context);
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_plan_grouped_gate_up(const moe_plan* plan, void* stream) {
    moe_status st = check_plan(plan);
    if (st != MOE_OK) return st;
    const moe_plan& p = *plan;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.dtype == MOE_BF16) return launch_ffn_tc_prepared(p.gate_up, s, p.di);
    return launch_ffn_simt_gate_up(static_cast<const float*>(p.xs), p.offsets, p.T * p.k, p.E, p.d, p.f,
                                   static_cast<const float*>(p.w_gate), static_cast<const float*>(p.w_up),
                                   static_cast<float*>(p.h), s, p.di);
}

extern "C" moe_status moe_plan_grouped_down(const moe_plan* plan, void* stream) {
    moe_status st = check_plan(plan);
    if (st != MOE_OK) return st;
    const moe_plan& p = *plan;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.dtype == MOE_BF16) return launch_ffn_tc_prepared(p.down, s, p.di);
    return launch_ffn_simt_down(static_cast<const float*>(p.h), p.offsets, p.T * p.k, p.E, p.d, p.f,
                                static_cast<const float*>(p.w_down), p.y, s, p.di);
}

extern "C" moe_status moe_plan_forward(const moe_plan* plan, const float* logits, const void* x,
                                       const uint8_t* mask, float* out, void* stream) {
    moe_status st = check_plan(plan);
    if (st != MOE_OK) return st;
    const moe_plan& p = *plan;
    MOE_REQUIRE(logits && x && out && aligned16(x) && aligned16(out));
    const int T = p.T, E = p.E, k = p.k, d = p.d, cap = T * k;
    if (T <= kSmallTokens && cap <= kSmallRoutes) {
        if ((st = moe_route_scatter_small(logits, x, p.dtype, 0, mask, T, E, k, d, p.ids, p.w, p.counts, p.offsets,
                                          p.xs, p.row_of_route, p.route_of_row, stream)) != MOE_OK)
            return st;
    } else {
        if ((st = moe_route_topk_offsets(logits, mask, T, E, k, p.ids, p.w, p.counts, p.offsets, p.ws, stream)) !=
            MOE_OK)
            return st;
        if ((st = moe_scatter_rows(x, p.dtype, p.ids, mask, p.offsets, T, k, d, E, p.xs, p.row_of_route,
                                   p.route_of_row, p.ws, stream)) != MOE_OK)
            return st;
    }
    if ((st = moe_plan_grouped_gate_up(plan, stream)) != MOE_OK) return st;
    if ((st = moe_plan_grouped_down(plan, stream)) != MOE_OK) return st;
    return moe_combine(p.y, p.row_of_route, p.w, T, k, d, out, stream);
}
