// Router projection with the top-k routing in its epilogue, on the sm_103a
// tensor cores: logits[t][e] = x[t] . wr[e] (bf16 operands, fp32
// accumulation), then the k largest logits per token (descending, ties to the
// lower expert id) and their softmax weights.
//
// Page "perf(ds4): extend sparse prefill scheduling to 10K", Summary: tokens
// take their native top-6 of the routed experts; the router logits are the
// token rows times the router matrix (stored K-contiguous, wr [E][d], like
// the expert weights).
//
// GB300 design: a cluster of 4 CTAs per 64-token tile, each CTA one quarter
// of K.  The router matrix (E <= 256 rows, at most two 128-row tiles) is the
// A operand of tcgen05.mma (M = 128), the token rows the B operand (N = 64);
// a CTA's K range streams through a 4-stage TMA ring of 40 KB stages.  After
// its last MMA each CTA reads its accumulators (one 64-column region per
// expert tile) with tcgen05.ld and writes them transposed into shared memory
// (the ring is free by then), [token][expert].  After a cluster barrier, CTA
// r sums the four partial tiles for tokens 16r .. 16r+15 over distributed
// shared memory in rank order (fixed, so the logits are reproducible) and
// one warp per token selects the top-k with order keys and writes ids,
// weights and, when asked, the logits row.  A second cluster barrier keeps
// every CTA's tile alive until its neighbours have read it.  Bounded waits as
// in the FFN kernels; every thread reaches both cluster barriers, also after
// an abandoned wait.

#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int RM = 128;          // router rows (experts) per A tile
constexpr int RT = 64;           // tokens per CTA (MMA N)
constexpr int RK = 64;           // K per stage
constexpr int kRStages = 4;
constexpr int kRThreads = 192;   // warp 0 TMA, 1 MMA, 2-5 epilogue
constexpr int kRATile = RM * RK * 2;                 // 16 KB
constexpr int kRBTile = RT * RK * 2;                 // 8 KB
constexpr int kRStage = 2 * kRATile + kRBTile;       // 40 KB
constexpr int kRRing = kRStages * kRStage;           // 160 KB
constexpr int kRLogitPitch = kMaxExperts + 1;        // floats per token row in shared memory
constexpr int kRCtrl = 256;
constexpr int kRSmem = kRRing + kRCtrl + 1024;
constexpr int kRCluster = 4;                          // CTAs per token tile (K split)
static_assert(RT * kRLogitPitch * 4 <= kRRing, "the logit tile fits the ring");

__global__ void __launch_bounds__(kRThreads, 1)
    router_topk_kernel(const __grid_constant__ CUtensorMap map_wr, const __grid_constant__ CUtensorMap map_x, int T,
                       int E, int d, int k, float* __restrict__ logits, int32_t* __restrict__ ids,
                       float* __restrict__ w, unsigned* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* ctrl = smem + kRRing;
    uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
    uint64_t* empty = full + kRStages;
    uint64_t* acc_full = empty + kRStages;
    uint64_t* drain = acc_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* issued = reinterpret_cast<int*>(tmem_slot + 2);  // kRStages entries
    volatile int* epi_ok = issued + kRStages;
    float* tile = reinterpret_cast<float*>(smem);          // [RT][kRLogitPitch], after the MMAs

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const int t0 = (blockIdx.x / kRCluster) * RT;
    // this CTA's k-blocks: [kb_lo, kb_hi) of d / RK, split as evenly as possible
    const int n_all = d / RK;
    const int kb_lo = (n_all * static_cast<int>(rank)) / kRCluster;
    const int kb_hi = (n_all * (static_cast<int>(rank) + 1)) / kRCluster;
    const int n_kb = kb_hi - kb_lo;
    const bool two = E > RM;                                // a second expert tile
    const uint32_t stage_tx = (two ? 2 : 1) * kRATile + kRBTile;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            issued[s] = -1;
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&map_wr);
        prefetch_tmap(&map_x);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(2 * RT)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = l2_policy(2);   // every CTA reads the router matrix: keep it in L2
            const uint64_t pol_x = l2_policy(1);
            int s = 0;
            uint32_t ph = 0;
            for (int j = 0; j < n_kb; ++j) {
                const int kb = kb_lo + j;
                if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, err)) break;
                uint8_t* st = smem + s * kRStage;
                mbar_arrive_expect_tx(&full[s], stage_tx);
                issued[s] = static_cast<int>(ph);
                tma_load_2d(st, &map_wr, &full[s], kb * RK, 0, pol_w);
                if (two) tma_load_2d(st + kRATile, &map_wr, &full[s], kb * RK, RM, pol_w);
                tma_load_2d(st + 2 * kRATile, &map_x, &full[s], kb * RK, t0, pol_x);
                if (++s == kRStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // bf16 A and B, fp32 accumulator, M = 128, N = 64
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(RT >> 3) << 17) |
                                   (static_cast<uint32_t>(RM >> 4) << 24);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int kb = 0; kb < n_kb; ++kb) {
                if (!mbar_wait(&full[s], ph, abort_flag, err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = sdesc_lo(smem_u32(smem + s * kRStage));
                const uint32_t a1 = a0 + (kRATile >> 4);
                const uint32_t b = a0 + ((2 * kRATile) >> 4);
#pragma unroll
                for (int kk = 0; kk < RK / 16; ++kk) {
                    const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
                    const uint64_t bd = sdesc_from_lo(b + 2 * kk);
                    umma_bf16(tmem_base, sdesc_from_lo(a0 + 2 * kk), bd, idesc, acc);
                    if (two) umma_bf16(tmem_base + RT, sdesc_from_lo(a1 + 2 * kk), bd, idesc, acc);
                }
                umma_commit(&empty[s]);
                if (++s == kRStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (ok) umma_commit(acc_full);   // (with no k-blocks it arrives at once; the epilogue writes zeros)
            umma_commit(drain);
            mbar_drain(drain, 0);
        }
    } else {
        // ---- epilogue (warps 2..5): TMEM -> shared [token][expert] -> top-k per token
        const int q = warp & 3;   // TMEM lanes [32q, 32q + 32): experts 32q + lane (+ 128)
        const int et = threadIdx.x - 64;
        if (et == 0) *epi_ok = mbar_wait(acc_full, 0, abort_flag, err) ? 1 : 0;
        epilogue_sync();
        if (*epi_ok) {
            tc_fence_after();
            const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            for (int r = 0; r < (two ? 2 : 1); ++r) {
                const int e = r * RM + q * 32 + lane;
#pragma unroll
                for (int c0 = 0; c0 < RT; c0 += 32) {
                    uint32_t v[32];
                    if (n_kb > 0) {
                        tmem_ld32(lane_addr + static_cast<uint32_t>(r * RT + c0), v);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = 0u;
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) tile[(c0 + j) * kRLogitPitch + e] = __uint_as_float(v[j]);
                }
            }
        }
        tc_fence_before();
    }

    // every CTA's partial tile is complete: CTA `rank` reduces tokens
    // [16 rank, 16 rank + 16) over the four tiles and routes them
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (warp >= 2) {
        const int q = warp & 3;
        if (*epi_ok && *abort_flag == 0) {
            uint32_t peer[kRCluster];
            const uint32_t tile_addr = smem_u32(tile);
#pragma unroll
            for (int c = 0; c < kRCluster; ++c)
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(peer[c]) : "r"(tile_addr), "r"(c));
            // warp per token: sum the partials in rank order, then k rounds of a warp arg-max
            for (int tt = static_cast<int>(rank) * (RT / kRCluster) + q; tt < (static_cast<int>(rank) + 1) * (RT / kRCluster);
                 tt += 4) {
                const int t = t0 + tt;
                if (t >= T) break;
                unsigned long long key[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int e = lane + 32 * j;
                    float acc = 0.f;
                    if (e < E) {
#pragma unroll
                        for (int c = 0; c < kRCluster; ++c) {
                            float pv;
                            asm volatile("ld.shared::cluster.f32 %0, [%1];"
                                         : "=f"(pv)
                                         : "r"(peer[c] + static_cast<uint32_t>((tt * kRLogitPitch + e) * 4)));
                            acc = c == 0 ? pv : acc + pv;
                        }
                    }
                    key[j] = e < E ? topk_order_key(acc, e) : 0ull;
                    if (logits != nullptr && e < E) logits[static_cast<size_t>(t) * E + e] = acc;
                }
                float sel_val = 0.f;
                int sel_id = 0;
                for (int sl = 0; sl < k; ++sl) {
                    unsigned long long best = key[0];
#pragma unroll
                    for (int j = 1; j < 8; ++j) best = key[j] > best ? key[j] : best;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
                        best = o > best ? o : best;
                    }
                    const int e = 0xFFFF - static_cast<int>(best & 0xFFFFu);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (lane + 32 * j == e) key[j] = 0ull;
                    if (lane == sl) {
                        sel_val = topk_key_value(best);
                        sel_id = e;
                    }
                }
                // softmax over the k selected logits, summed in slot order
                const float top = __shfl_sync(0xffffffffu, sel_val, 0);
                float sum = 0.f;
                for (int r = 0; r < k; ++r) sum += expf(__shfl_sync(0xffffffffu, sel_val, r) - top);
                const float inv = 1.f / sum;
                if (lane < k) {
                    ids[static_cast<size_t>(t) * k + lane] = sel_id;
                    w[static_cast<size_t>(t) * k + lane] = expf(sel_val - top) * inv;
                }
            }
        }
    }
    // keep this CTA's tile until every neighbour has read it
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        for (int s = 0; s < kRStages; ++s)
            if (issued[s] >= 0) mbar_drain(&full[s], static_cast<uint32_t>(issued[s]));
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(2 * RT)
                     : "memory");
    }
}

std::mutex g_router_mutex;
bool g_router_attr[64];

}  // namespace

moe_status launch_router_topk(const void* x, const void* wr, int T, int E, int d, int k, float* logits,
                              int32_t* ids, float* w, cudaStream_t st, const DeviceInfo& di) {
    CUtensorMap mw, mx;
    moe_status s;
    if ((s = encode_2d_map(&mw, wr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, E, RK, RM,
                           CU_TENSOR_MAP_SWIZZLE_128B)) != MOE_OK)
        return s;
    if ((s = encode_2d_map(&mx, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, T, RK, RT,
                           CU_TENSOR_MAP_SWIZZLE_128B)) != MOE_OK)
        return s;
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lock(g_router_mutex);
        if (!g_router_attr[dev]) {
            MOE_CUDA_TRY(cudaFuncSetAttribute(router_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem));
            g_router_attr[dev] = true;
        }
    }
    // clusters of kRCluster CTAs, one cluster per 64-token tile
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(((T + RT - 1) / RT) * kRCluster));
    cfg.blockDim = dim3(kRThreads);
    cfg.dynamicSmemBytes = kRSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kRCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, router_topk_kernel, mw, mx, T, E, d, k, logits, ids, w,
                                          di.error_word));
}

}  // namespace moe
