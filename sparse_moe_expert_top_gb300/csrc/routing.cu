// Routing-side kernels of grouped MoE prefill: top-k routing (A1), route
// histogram (A2), exclusive prefix (A3), expert-major scatter (A4) and the
// weighted combine (A7).  These steps move a few MB to a few hundred MB per
// chunk and are bound by HBM bandwidth or by launch latency; none of them is
// a contraction, so they run on the SIMT pipes with 128-bit accesses.
//
// Page "perf(ds4): batch heterogeneous MoE prefill by expert" (Luce-Org/
// lucebox PR #640), Summary: GPU-native route histogram, prefix and scatter
// for up to 256 experts; masked owner routes are exact zero contributions.
// Page "perf(ds4): accelerate ROCm decode and long-context selection"
// (PR #667), lucebox8 A/B: one fused expert-major combine launch replaces the
// reduce/multiply launches.

#include <cuda_runtime.h>

#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// A1: top-k routing, one warp per token.
// ---------------------------------------------------------------------------

// Order-preserving 64-bit key: high word = the logit's bits mapped so that
// unsigned order equals float order (with -0.0 folded onto +0.0), low word =
// 0xFFFF - expert so that equal logits rank the lower expert first.  Key 0 is
// below every real key and marks "taken" or "no expert".
__device__ __forceinline__ unsigned long long topk_key(float v, int e) {
    unsigned u = __float_as_uint(v);
    if ((u << 1) == 0u) u = 0u;
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(u) << 32) | static_cast<unsigned>(0xFFFF - e);
}

__device__ __forceinline__ float key_value(unsigned long long key) {
    unsigned u = static_cast<unsigned>(key >> 32);
    u = (u & 0x80000000u) ? (u & 0x7fffffffu) : ~u;
    return __uint_as_float(u);
}

template <int EPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int32_t* __restrict__ ids, float* __restrict__ w) {
    const int lane = threadIdx.x & 31;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const float* row = logits + static_cast<size_t>(t) * E;

    unsigned long long key[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const int e = lane + 32 * j;
        key[j] = (e < E) ? topk_key(__ldg(row + e), e) : 0ull;
    }

    float sel_val = 0.f;
    int sel_id = 0;
    for (int s = 0; s < k; ++s) {
        unsigned long long best = key[0];
#pragma unroll
        for (int j = 1; j < EPL; ++j) best = key[j] > best ? key[j] : best;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(kFull, best, off);
            best = o > best ? o : best;
        }
        const int e = 0xFFFF - static_cast<int>(best & 0xFFFFu);
#pragma unroll
        for (int j = 0; j < EPL; ++j)
            if (lane + 32 * j == e) key[j] = 0ull;
        if (lane == s) {
            sel_val = key_value(best);
            sel_id = e;
        }
    }

    // softmax over the k selected logits; lane 0 holds the largest
    const float top = __shfl_sync(kFull, sel_val, 0);
    const float z = (lane < k) ? expf(sel_val - top) : 0.f;
    float sum = z;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    if (lane < k) {
        ids[static_cast<size_t>(t) * k + lane] = sel_id;
        w[static_cast<size_t>(t) * k + lane] = z / sum;
    }
}

// ---------------------------------------------------------------------------
// A2: route histogram with stable in-chunk ranks.
//
// CTA c owns routes [c*2048, (c+1)*2048); warp w of the CTA owns 256 of them
// and walks them 32 at a time in route order.  __match_any_sync groups the
// lanes that hit the same expert; a lane's rank is the warp's running count
// for that expert plus the number of lower lanes in its group, so ranks
// follow route order.  The per-warp counts are then scanned across warps in
// warp order, giving every route its stable rank inside the chunk and the
// chunk's per-expert count.  The last CTA to finish (completion counter in
// the workspace) sums the chunk counts into counts[] and resets the counter.
// ---------------------------------------------------------------------------

constexpr int kHistWarps = 8;
constexpr int kHistSteps = kHistChunk / (kHistWarps * 32);

__global__ void __launch_bounds__(256) route_histogram_kernel(const int32_t* __restrict__ ids,
                                                              const uint8_t* __restrict__ mask, int n_routes,
                                                              int E, int32_t* __restrict__ ws,
                                                              int32_t* __restrict__ counts, unsigned* err) {
    __shared__ int cnt[kHistWarps][kMaxExperts];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t* chunk_counts = ws + kWsHeaderWords;
    int32_t* lrank = chunk_counts + static_cast<size_t>(gridDim.x) * kMaxExperts;

    for (int i = tid; i < kHistWarps * kMaxExperts; i += blockDim.x) (&cnt[0][0])[i] = 0;
    __syncthreads();

    const unsigned lt_mask = (1u << lane) - 1u;
    const int base = blockIdx.x * kHistChunk + warp * (kHistSteps * 32);
    int my_e[kHistSteps], my_rank[kHistSteps];
    bool bad = false;
#pragma unroll
    for (int step = 0; step < kHistSteps; ++step) {
        const int r = base + step * 32 + lane;
        int e = -1;
        if (r < n_routes) {
            e = __ldg(ids + r);
            if (e < 0 || e >= E) {
                bad = true;
                e = -1;
            } else if (mask != nullptr && __ldg(mask + r) != 0) {
                e = -1;
            }
        }
        const unsigned peers = __match_any_sync(kFull, e);
        int rank = -1;
        if (e >= 0) rank = cnt[warp][e] + __popc(peers & lt_mask);
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) cnt[warp][e] += __popc(peers);
        __syncwarp();
        my_e[step] = e;
        my_rank[step] = rank;
    }
    if (bad) atomicOr(err, DEVERR_OFFSETS);
    __syncthreads();

    // exclusive scan over warps, per expert
    for (int e = tid; e < kMaxExperts; e += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kHistWarps; ++w) {
            const int c = cnt[w][e];
            cnt[w][e] = run;
            run += c;
        }
        chunk_counts[static_cast<size_t>(blockIdx.x) * kMaxExperts + e] = run;
    }
    __syncthreads();
#pragma unroll
    for (int step = 0; step < kHistSteps; ++step) {
        const int r = base + step * 32 + lane;
        if (r < n_routes) lrank[r] = my_e[step] >= 0 ? my_rank[step] + cnt[warp][my_e[step]] : -1;
    }

    // last CTA reduces the chunk counts
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(reinterpret_cast<unsigned*>(ws), 1u) == gridDim.x - 1);
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int e = tid; e < E; e += blockDim.x) {
            int sum = 0;
            for (int c = 0; c < static_cast<int>(gridDim.x); ++c)
                sum += __ldcg(chunk_counts + static_cast<size_t>(c) * kMaxExperts + e);
            counts[e] = sum;
        }
        if (tid == 0) atomicExch(reinterpret_cast<unsigned*>(ws), 0u);
    }
}

// ---------------------------------------------------------------------------
// A3: exclusive prefix over expert counts (one CTA of 256 threads), and the
// per-chunk row bases: base[c][e] = offsets[e] + sum of chunk counts c' < c.
// The chunk counts are only read, so the call can be repeated.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) prefix_offsets_kernel(const int32_t* __restrict__ counts, int E,
                                                             int n_chunks, int32_t* __restrict__ offsets,
                                                             const int32_t* __restrict__ chunk_counts,
                                                             int32_t* __restrict__ chunk_bases) {
    __shared__ int warp_sum[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = tid < E ? counts[tid] : 0;
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += warp_sum[w];
    const int excl = before + incl - c;
    if (tid < E) offsets[tid] = excl;
    if (tid == E - 1) offsets[E] = excl + c;

    if (tid < E) {
        int run = excl;
        for (int ch = 0; ch < n_chunks; ++ch) {
            chunk_bases[static_cast<size_t>(ch) * kMaxExperts + tid] = run;
            run += chunk_counts[static_cast<size_t>(ch) * kMaxExperts + tid];
        }
    }
}

// ---------------------------------------------------------------------------
// A4: scatter, one CTA per token.  The token row is read once with 128-bit
// loads and written to each of its unmasked compact rows; the CTA also
// zero-fills k of the unused tail rows R .. T*k-1.  Expert ids, compact rows
// and R are checked against their ranges before any write: a workspace that
// the histogram and prefix did not prepare for these ids sets
// DEVERR_OFFSETS instead of writing outside xs.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(128) scatter_rows_kernel(const uint4* __restrict__ x,
                                                           const int32_t* __restrict__ ids,
                                                           const int32_t* __restrict__ offsets, int T, int k,
                                                           int E, int row_vecs, const int32_t* __restrict__ lrank,
                                                           const int32_t* __restrict__ bases,
                                                           uint4* __restrict__ xs,
                                                           int32_t* __restrict__ row_of_route,
                                                           int32_t* __restrict__ route_of_row, unsigned* err) {
    __shared__ int rows[kMaxK];
    __shared__ int tails[kMaxK];
    const int t = blockIdx.x, tid = threadIdx.x;
    const int n_routes = T * k;
    if (tid < k) {
        const int r = t * k + tid;
        const int lr = lrank[r];
        int row = -1;
        bool bad = false;
        if (lr >= 0) {
            const int e = ids[r];
            if (e >= 0 && e < E) row = bases[static_cast<size_t>(r / kHistChunk) * kMaxExperts + e] + lr;
            if (row < 0 || row >= n_routes) {
                bad = true;
                row = -1;
            }
        }
        rows[tid] = row;
        row_of_route[r] = row;
        if (row >= 0) route_of_row[row] = r;
        const int R = __ldg(offsets + E);
        int tail = -1;
        if (R < 0 || R > n_routes) bad = true;
        else if (R + r < n_routes) tail = R + r;
        tails[tid] = tail;
        if (tail >= 0) route_of_row[tail] = -1;
        if (bad) atomicOr(err, DEVERR_OFFSETS);
    }
    __syncthreads();
    const uint4* src = x + static_cast<size_t>(t) * row_vecs;
    for (int v = tid; v < row_vecs; v += blockDim.x) {
        const uint4 val = __ldg(src + v);
        for (int s = 0; s < k; ++s) {
            const int row = rows[s];
            if (row >= 0) xs[static_cast<size_t>(row) * row_vecs + v] = val;
            const int tail = tails[s];
            if (tail >= 0) xs[static_cast<size_t>(tail) * row_vecs + v] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// ---------------------------------------------------------------------------
// A7: combine, one CTA per token; slots are added in ascending order with
// fp32 FMAs starting from +0.0, masked slots are skipped.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(128) combine_kernel(const float4* __restrict__ y,
                                                      const int32_t* __restrict__ row_of_route,
                                                      const float* __restrict__ w, int k, int d4, int cap,
                                                      float4* __restrict__ out, unsigned* err) {
    __shared__ int rows[kMaxK];
    __shared__ float wt[kMaxK];
    const int t = blockIdx.x, tid = threadIdx.x;
    if (tid < k) {
        int row = row_of_route[static_cast<size_t>(t) * k + tid];
        if (row >= cap) {  // not a row of y: flagged, treated as masked
            atomicOr(err, DEVERR_OFFSETS);
            row = -1;
        }
        rows[tid] = row;
        wt[tid] = w[static_cast<size_t>(t) * k + tid];
    }
    __syncthreads();
    float4* dst = out + static_cast<size_t>(t) * d4;
    for (int v = tid; v < d4; v += blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < k; ++s) {
            const int row = rows[s];
            if (row < 0) continue;
            const float4 yy = __ldg(y + static_cast<size_t>(row) * d4 + v);
            const float ws = wt[s];
            acc.x = fmaf(ws, yy.x, acc.x);
            acc.y = fmaf(ws, yy.y, acc.y);
            acc.z = fmaf(ws, yy.z, acc.z);
            acc.w = fmaf(ws, yy.w, acc.w);
        }
        dst[v] = acc;
    }
}

moe_status launch_status() { return cuda_status(cudaGetLastError()); }

// Largest chunk the allocation-free histogram accepts, and its scratch size:
// header + per-chunk counts + one in-chunk rank per route (295 KB).
constexpr int kNoAllocMaxRoutes = 65536;
constexpr int kNoAllocWords =
    kWsHeaderWords + ((kNoAllocMaxRoutes + kHistChunk - 1) / kHistChunk) * kMaxExperts + kNoAllocMaxRoutes;

}  // namespace
}  // namespace moe

// Scratch of moe_route_histogram_noalloc.  Every GPU that loads the library
// holds this array until the process exits, and every call of that entry
// point on a device uses the same copy.
static __device__ __align__(256) int32_t g_noalloc_hist_scratch[moe::kNoAllocWords];

using namespace moe;

namespace {

std::mutex g_noalloc_mutex;
int32_t* g_noalloc_scratch[64];

// Device address of g_noalloc_hist_scratch on the current device.  In host
// code the array's name is only a host-side stand-in, so the address is
// looked up once per device (with that device current) and cached.
moe_status noalloc_scratch(int32_t** out) {
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_scratch[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_hist_scratch);
        if (e != cudaSuccess) return cuda_status(e);
        g_noalloc_scratch[dev] = static_cast<int32_t*>(p);
    }
    *out = g_noalloc_scratch[dev];
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_workspace_size(int T, int k, size_t* bytes) {
    MOE_REQUIRE(bytes != nullptr && T >= 0 && k >= 1 && k <= kMaxK);
    MOE_REQUIRE(static_cast<long long>(T) * k < (1ll << 30));
    *bytes = ws_words(T, k) * sizeof(int32_t);
    return MOE_OK;
}

extern "C" moe_status moe_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                                     void* stream) {
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && ids && w);
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    const int threads = 256, warps_per_block = threads / 32;
    const int blocks = (T + warps_per_block - 1) / warps_per_block;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (E <= 32)
        route_topk_kernel<1><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w);
    else if (E <= 64)
        route_topk_kernel<2><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w);
    else if (E <= 128)
        route_topk_kernel<4><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w);
    else
        route_topk_kernel<8><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w);
    return launch_status();
}

extern "C" moe_status moe_route_histogram(const int32_t* ids, const uint8_t* mask, int T, int k, int E,
                                          int32_t* counts, void* ws, void* stream) {
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E);
    MOE_REQUIRE(counts && ws && aligned16(ws));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) return cuda_status(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s));
    MOE_REQUIRE(ids);
    const int n_routes = T * k;
    route_histogram_kernel<<<ws_chunks(T, k), 256, 0, s>>>(ids, mask, n_routes, E, static_cast<int32_t*>(ws),
                                                          counts, di.error_word);
    return launch_status();
}

extern "C" moe_status moe_prefix_offsets(const int32_t* counts, int T, int k, int E, int32_t* offsets, void* ws,
                                         void* stream) {
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E);
    MOE_REQUIRE(counts && offsets && ws && aligned16(ws));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* w32 = static_cast<int32_t*>(ws);
    prefix_offsets_kernel<<<1, 256, 0, s>>>(counts, E, T == 0 ? 0 : ws_chunks(T, k), offsets, w32 + kWsHeaderWords,
                                            w32 + ws_bases_offset(T, k));
    return launch_status();
}

extern "C" moe_status moe_scatter_rows(const void* x, int dtype, const int32_t* ids, const uint8_t* mask,
                                       const int32_t* offsets, int T, int k, int d, int E, void* xs,
                                       int32_t* row_of_route, int32_t* route_of_row, void* ws, void* stream) {
    (void)mask;  // the histogram already folded the mask into the workspace ranks
    const int es = dtype_size(dtype);
    if (es == 0) return MOE_ERR_UNSUPPORTED;
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E && d >= 1);
    MOE_REQUIRE((static_cast<size_t>(d) * es) % 16 == 0);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(x && ids && offsets && xs && row_of_route && route_of_row && ws);
    MOE_REQUIRE(aligned16(x) && aligned16(xs) && aligned16(ws));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    const int row_vecs = static_cast<int>(static_cast<size_t>(d) * es / 16);
    const int32_t* w32 = static_cast<const int32_t*>(ws);
    scatter_rows_kernel<<<T, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(x), ids, offsets, T, k, E, row_vecs, w32 + ws_rank_offset(T, k),
        w32 + ws_bases_offset(T, k), static_cast<uint4*>(xs), row_of_route, route_of_row, di.error_word);
    return launch_status();
}

extern "C" moe_status moe_combine(const float* y, const int32_t* row_of_route, const float* w, int T, int k, int d,
                                  float* out, void* stream) {
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= kMaxK && d >= 1 && d % 4 == 0);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(y && row_of_route && w && out && aligned16(y) && aligned16(out));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    combine_kernel<<<T, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float4*>(y), row_of_route, w, k, d / 4, T * k, reinterpret_cast<float4*>(out),
        di.error_word);
    return launch_status();
}

// Allocation-free route histogram: the counts of moe_route_histogram, with
// the scratch taken from g_noalloc_hist_scratch instead of a caller
// workspace.  It allocates nothing; it clears the scratch's completion
// counter before the launch because the array keeps the previous call's
// contents.
extern "C" moe_status moe_route_histogram_noalloc(const int32_t* ids, const uint8_t* mask, int T, int k, int E,
                                                  int32_t* counts, void* stream) {
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E);
    MOE_REQUIRE(counts != nullptr);
    MOE_REQUIRE(static_cast<long long>(T) * k <= kNoAllocMaxRoutes);
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    int32_t* scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) return cuda_status(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s));
    MOE_REQUIRE(ids != nullptr);
    MOE_CUDA_TRY(cudaMemsetAsync(scratch, 0, sizeof(int32_t), s));
    route_histogram_kernel<<<ws_chunks(T, k), 256, 0, s>>>(ids, mask, T * k, E, scratch, counts, di.error_word);
    return launch_status();
}
