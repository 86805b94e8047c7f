// Grouped expert FFN on the sm_103a tensor cores (operand type MOE_BF16).
//
// Page "perf(ds4): batch heterogeneous MoE prefill by expert" (Luce-Org/
// lucebox PR #640), Summary: one grouped gate/up and one grouped down
// projection over all active experts instead of a serial graph per expert.
// Page "perf(ds4): unify gfx1151 sparse-prefill stack" (PR #685),
// Composition: adaptive sparse-MoE tiles and a persistent compact work queue.
//
// GB300 design
// ------------
// Prefill chunks give each expert few rows (median 9 at 401 tokens, ~19 at
// 2048), so the work is streaming the touched experts' weights from HBM.
// The kernel therefore swaps the GEMM operands: the WEIGHT tile is the
// M = 128 operand of tcgen05.mma and the expert's compact token rows form N
// (a multiple of 16, at most 128 per work item, 256 in big-item mode).  Each
// weight byte is loaded once per row slice, and an expert with 9 rows issues
// N = 16 MMAs instead of padding 9 rows up to an M = 128 tile.  (The pages'
// adaptive tile width on RDNA is the same idea.)
//
// Work item = (expert e, a slice mt of the output features -- 128 for
// gate/up, 256 (two tiles) for down -- and a slice nt of the expert's
// compact rows: 128 rows, or 256 when most rows belong to heavy experts).
// Chunks of at most 64 routes use narrow items instead -- 64 features for
// gate/up (gate and up rows stacked in one MMA tile), one 128-row tile for
// down -- so that a handful of tokens still gives several waves of items.
// Items are numbered expert by expert (expert-id order; heaviest expert
// first in the fused down kernel), then mt, then nt, so CTAs working at the
// same time on the nt slices of one expert share its weight tile through L2.
// The kernel is persistent: one CTA per SM takes items blockIdx.x,
// blockIdx.x + gridDim.x, ...; every CTA derives the same item table from
// `offsets` in its prologue, so ragged per-expert row counts (including empty
// experts) need no host round trip.
//
// Roles: warp 0 lane 0 issues TMA loads into a ring of shared-memory stages
// (128B-swizzled, 64 K-elements per stage); warp 1 lane 0 issues
// tcgen05.mma into a double-buffered TMEM accumulator (gate and up
// accumulators side by side for the SwiGLU stage); the epilogue warps (4 for
// gate/up, 8 for down) read the accumulator with tcgen05.ld, apply SwiGLU
// (gate/up) and store rows; the fused instantiations add a row-gather warp
// (gate/up) or four combine warps (down), below.
// Every mbarrier wait is bounded: when it runs out the kernel records
// DEVERR_TIMEOUT, lets its copies and MMAs drain, frees TMEM and returns.
//
// Fused permutation (the FUSED instantiations)
// --------------------------------------------
// Pages "perf(ds4): accelerate ROCm decode and long-context selection"
// (PR #667), its gfx1151 fused-combine A/B, and "perf(ds4): extend sparse
// prefill scheduling to 10K" (PR #684), its historical fused-combine
// discriminator: the combine is a fused expert-major kernel there; here the
// whole row permutation moves into the GEMMs.
// * Gate/up: no compact copy xs.  A gather warp (next to the TMA warp, which
//   keeps streaming the weight tiles) copies the item's token rows from x
//   with 16-byte cp.async copies (token = route_of_row[row] / k) into the
//   128B-swizzled layout of the MMA operand; each lane's copies arrive on the
//   stage's full barrier when they land (cp.async.mbarrier.arrive), and the
//   MMA thread fences the generic proxy against the async proxy before it
//   reads them.  (TMA row gathers, four rows per copy, were measured slower:
//   their per-copy cost exceeds what the compact copy costs.)
// * Down: four combine warps follow the epilogue.  After an item's y rows
//   are stored they count, per (token, feature slice), the slots stored so
//   far (one global counter each); the CTA that stores a token's last slot
//   adds its slots in ascending slot order from +0.0 (the unfused combine's
//   arithmetic, so out is bit-identical) and drops the y lines it read from
//   L2 without write-back.  y is scratch here and laid out slice-major
//   ([feature slice][row][slice width]), so that the items running at the
//   same time write contiguous memory.

#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace moe {
namespace {

// silu(g) = g / (1 + e^-g) with the fast exponential and division
// intrinsics (a few ulp of fp32; the result is rounded to a 16-bit h).  For
// g < -88 the exponential overflows to +inf and the quotient is -0.
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.f + __expf(-g)); }

// Big-item mode (row slices of up to 256 rows, 3 stages of 64 KB) is taken
// when the rows beyond the first 128 of each expert reach this percentage
// of all rows; otherwise row slices of 128 rows and 4 stages of 48 KB.
#ifndef MOE_TC_BIG_MODE_PCT
#define MOE_TC_BIG_MODE_PCT 50
#endif
// L2 eviction priority of the TMA loads: 0 normal, 1 evict_first, 2 evict_last.
// Weight tiles read by one work item only are streamed with evict_first;
// tiles of experts with several row slices (read once per slice, by CTAs
// that run at about the same time) are kept with MOE_TC_SHARED_W_POLICY.
#ifndef MOE_TC_SHARED_W_POLICY
#define MOE_TC_SHARED_W_POLICY 2
#endif
#ifndef MOE_TC_X_POLICY
#define MOE_TC_X_POLICY 2
#endif

constexpr int BM = 128;        // MMA M: weight rows per tile
constexpr int BN = 128;        // rows of a light work item / of one accumulator slot
constexpr int BK = 64;         // K elements per stage (one 128-byte swizzle atom of bf16)
constexpr int UMMA_K = 16;     // K per tcgen05.mma of kind::f16
constexpr int kBoxRows = 16;   // compact rows per small TMA box (the granule of N)
#ifndef MOE_TC_BIG_BOX_ROWS
#define MOE_TC_BIG_BOX_ROWS 64
#endif
constexpr int kBigBoxRows = MOE_TC_BIG_BOX_ROWS;  // compact rows per large TMA box
// Warps 0 (TMA) and 1 (MMA), then the epilogue: 4 warps for gate/up, 8 for
// down.  In big-item mode the down kernel's 8 epilogue warps work as two
// groups, two warps per tensor-memory lane quarter taking alternate 32-row
// chunks: the fp32 stores of 256-row items otherwise set the pace instead of
// the MMAs.  In the other modes the second group only takes part in the
// barriers (a second group there was measured slower).
#ifndef MOE_TC_DOWN_EPI_WARPS
#define MOE_TC_DOWN_EPI_WARPS 8
#endif
// The fused kernels add warps after the epilogue warps: one row-gather warp
// (gate/up) or four combine warps (down).
template <bool GATED, bool FUSED>
struct Roles {
    static constexpr int kEpiWarps = GATED ? 4 : MOE_TC_DOWN_EPI_WARPS;
    static constexpr int kCombWarps = (!GATED && FUSED) ? 4 : 0;
    static constexpr int kGatherWarps = (GATED && FUSED) ? 1 : 0;
    static constexpr int kThreads = 64 + 32 * (kEpiWarps + kCombWarps + kGatherWarps);
};
__device__ __forceinline__ void epilogue_sync_n(int threads) {
    asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
}
__device__ __forceinline__ void combine_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
// Slots whose loads the combine warps keep in flight together (top-6 routing
// takes one group).
constexpr int kSlotGroup = 6;

// Arguments of the fused permutation (unused by the plain instantiations).
struct FusedArgs {
    const uint8_t* x;             // gate/up: token rows, bf16 [T][d]
    const int32_t* route_of_row;  // compact row -> route t*k+s
    const int32_t* row_of_route;  // down: route -> compact row, -1 if masked
    const float* w;               // down: gate weights [T][k]
    float* out;                   // down: [T][d]
    int32_t* tile_counts;         // down: [T][cstride] slot counters, zero on entry
    int T, k, cstride;
};

// Scales of the E4M3 instantiations (unused by the bf16 ones): the
// accumulator of weight row m and compact row n is multiplied by a0[e*M + m]
// (gate/up: the gate rows; down: the w_down rows) or a1[e*M + m] (the up
// rows) and by b[n] (the compact row's own scale).
struct OpScales {
    const float* a0;
    const float* a1;
    const float* b;
};

// Shared memory: a 192 KB ring, carved per launch into 4 stages of 48 KB
// (two 16 KB weight tiles + up to 128 rows; narrow items: two k-blocks of one
// weight tile + up to 64 rows each) or, in big-item mode, 3 stages of 64 KB
// (two weight tiles + up to 256 rows).  TMEM: 512 columns, region r
// (weight tile r) at columns 256r, each region in two 128-column slots; a
// light item uses slot s of both regions (consecutive light items alternate
// slots, so one item's epilogue overlaps the next item's MMAs), a big item
// uses both slots, i.e. 256 contiguous columns per region.
template <bool GATED>
struct Cfg {
    static constexpr int kA = 2;  // weight tiles per stage (gate+up, or two w_down feature tiles)
    static constexpr int kATileBytes = BM * BK * 2;
    static constexpr int kMaxStages = 4;
    static constexpr int kRingBytes = 4 * (kA * kATileBytes + BN * BK * 2);  // = 3 x 64 KB
    static constexpr int kTmemCols = 512;
    static constexpr int kCtrlBytes = 4096;  // barriers, TMEM slot, flags, item table (<= 3.3 KB)
    // the first kList items of the CTA's hand-out sequence, decoded once at
    // the start (a decode -- a search over the experts and two loads of the
    // offsets -- takes microseconds under load, on every role's path between items)
    static constexpr int kList = 512;
    static constexpr int kListBytes = kList * 16;
    // gate/up: a 32-row x 128-feature bf16 tile of h staged for row-contiguous
    // stores, then (narrow items) the up half of a stacked tile, 64 features x 32
    // rows of fp32 padded to 33 columns
    static constexpr int kOutStageBytes = GATED ? 32 * BM * 2 + 64 * 33 * 4 : 0;
    // fused kernels only: the token of each row of the current item (gate/up),
    // or the combine warps' barriers, list of completed tokens and their
    // compact rows (down)
    static constexpr int kFusedBytes = GATED ? 2048 : 1024 + 2 * BN * 4 + 2 * BN * kMaxK * 4;
    static constexpr int kSmemBytes = kRingBytes + kCtrlBytes + kListBytes + kOutStageBytes + 1024;
    static constexpr int smem_bytes(bool fused) { return kSmemBytes + (fused ? kFusedBytes : 0); }
    static_assert(kSmemBytes + kFusedBytes <= 232448, "shared memory budget of one CTA");
    static_assert(kRingBytes == 3 * (kA * kATileBytes + 2 * BN * BK * 2), "both carve-ups fill the ring");
    static_assert(kRingBytes / 4 >= kA * kATileBytes + 2 * 64 * BK * 2, "narrow carve-up: two k-blocks per stage");
};

// ---------------------------------------------------------------------------
// The kernel.  GATED: out = h (bf16 [cap][M]) = silu(A0 . xs) * (A1 . xs) with
// A0 = w_gate, A1 = w_up, M = f, K = d.  Otherwise out = y (fp32 [cap][M]) =
// A0 . h with A0 = w_down, M = d, K = f.
// ---------------------------------------------------------------------------

template <bool GATED, bool FUSED, bool F8 = false>
__global__ void __launch_bounds__(Roles<GATED, FUSED>::kThreads, 1)
    ffn_tc_kernel(const __grid_constant__ CUtensorMap map_a0, const __grid_constant__ CUtensorMap map_a1,
                  const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_b_big,
                  const int32_t* __restrict__ offsets, int cap, int E,
                  int K, int M, int narrow, void* __restrict__ out, unsigned* err, const FusedArgs fa,
                  const OpScales sc) {
    using C = Cfg<GATED>;
    using Ro = Roles<GATED, FUSED>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* ctrl = smem + C::kRingBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
    uint64_t* empty = full + C::kMaxStages;
    uint64_t* acc_full = empty + C::kMaxStages;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* issued = reinterpret_cast<int*>(tmem_slot + 2);  // last phase issued per stage, -1 = none
    int* item_off = issued + C::kMaxStages;               // E + 1 entries
    int* ntiles = item_off + kMaxExperts + 1;             // E entries
    // outcome of the epilogue's accumulator wait, double-buffered by item
    // parity (the four epilogue warps are never more than one item apart)
    volatile int* epi_flag = reinterpret_cast<volatile int*>(ntiles + kMaxExperts);  // 2 entries
    int* mode_big = const_cast<int*>(reinterpret_cast<volatile int*>(epi_flag + 2));   // launch-wide carve-up
    int* order = mode_big + 1;   // experts by descending row count (E entries; row counts while ranking)
    Item* ilist = reinterpret_cast<Item*>(ctrl + C::kCtrlBytes);   // this CTA's items, in hand-out order
    uint8_t* after_list = ctrl + C::kCtrlBytes + C::kListBytes;
    __nv_bfloat16* out_stage = reinterpret_cast<__nv_bfloat16*>(after_list);  // gate/up only
    float* up_stage = reinterpret_cast<float*>(after_list + 32 * BM * 2);     // narrow gate/up only
    uint8_t* fused_smem = after_list + C::kOutStageBytes;
    int* tok_s = reinterpret_cast<int*>(fused_smem);                  // gather: token of each row of the item
    uint64_t* comb_done = reinterpret_cast<uint64_t*>(fused_smem);    // combine: an item's y rows are stored (2)
    uint64_t* comb_free = comb_done + 2;                               // combine: that barrier phase was consumed (2)
    volatile int* comb_flag = reinterpret_cast<volatile int*>(comb_free + 2);
    volatile int* list_n = comb_flag + 1;                              // tokens completed by this CTA's item
    int* list = reinterpret_cast<int*>(fused_smem + 1024);             // up to 2 * BN of them
    int* list_rows = list + 2 * BN;                                    // their compact rows, kMaxK per token

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // K elements per k-block: one 128-byte swizzle row of the operand type
    constexpr int KBE = F8 ? 128 : BK;
    const int n_kb = K / KBE;
    // Output features per work item.  Normal items: 128 (gate/up: a gate tile
    // and an up tile, two MMAs) or 256 (down: two tiles).  Narrow items (small
    // chunks, chosen on the host so that there are more items than waves of
    // SMs): 64 for gate/up -- 64 gate rows stacked on 64 up rows in one 128-row
    // A tile, one MMA -- or 128 for down (one tile).
    const int fw = GATED ? (narrow ? BM / 2 : BM) : (narrow ? BM : 2 * BM);
    const int n_mt = (M + fw - 1) / fw;

    // ---- prologue: barriers, TMEM, item table --------------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kMaxStages; ++s) {
            // gather: one arrival with the weight bytes, one per gather-warp lane when its rows have landed
            mbar_init(&full[s], GATED && FUSED ? 33 : 1);
            mbar_init(&empty[s], 1);
            issued[s] = -1;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], Ro::kEpiWarps);
            if (!GATED && FUSED) {
                mbar_init(&comb_done[b], Ro::kEpiWarps);
                mbar_init(&comb_free[b], Ro::kCombWarps);
            }
        }
        if (!GATED && FUSED) *list_n = 0;
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&map_a0);
        if (GATED) prefetch_tmap(&map_a1);
        prefetch_tmap(&map_b);
        prefetch_tmap(&map_b_big);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp >= 2 && warp < 2 + Ro::kEpiWarps) {
        // The epilogue warps build the item table.  Warp 2 validates the
        // segments, picks the carve-up and counts every expert's row slices.
        // The fused down kernel then ranks the experts by row count (largest
        // first, ties to the lower id; all epilogue threads), which spreads the
        // tokens' completions, and so the combine warps' work, more evenly
        // over the launch (measured: 2,048 tokens 0.76 -> 0.66 ms); the other
        // kernels keep the expert-id order, which streams the weight bank and
        // the compact rows in address order (the ranked order made them 3-5 %
        // slower).  Warp 2 finally numbers the items in the chosen order.
        constexpr int kEpiThreads = 32 * Ro::kEpiWarps;
        constexpr bool kRanked = !GATED && FUSED;
        const int et = threadIdx.x - 64;
        if (warp == 2) {
            bool bad = false;
            long long rows = 0, excess = 0;
            for (int e = lane; e < E; e += 32) {
                const int lo = offsets[e], hi = offsets[e + 1];
                bad |= lo < 0 || hi < lo || hi > cap;
                const int n = hi - lo;
                rows += n > 0 ? n : 0;
                excess += n > BN ? n - BN : 0;
            }
            bad = __any_sync(0xffffffffu, bad);
            for (int off = 16; off > 0; off >>= 1) {
                rows += __shfl_xor_sync(0xffffffffu, rows, off);
                excess += __shfl_xor_sync(0xffffffffu, excess, off);
            }
            const bool big = !narrow && rows > 0 && excess * 100 >= static_cast<long long>(MOE_TC_BIG_MODE_PCT) * rows;
            if (lane == 0) {
                *mode_big = big ? 1 : 0;
                epi_flag[0] = bad ? 1 : 0;   // (reused once the table is built)
            }
            for (int e = lane; e < E; e += 32) {
                const int n = bad ? 0 : max(offsets[e + 1] - offsets[e], 0);
                ntiles[e] = n == 0 ? 0 : (big && n > BN ? (n + 2 * BN - 1) / (2 * BN) : (n + BN - 1) / BN);
                order[e] = kRanked ? n : e;
            }
        }
        epilogue_sync_n(kEpiThreads);
        if (kRanked) {
            int rank[(kMaxExperts + 127) / 128];
#pragma unroll
            for (int i = 0; i < (kMaxExperts + 127) / 128; ++i) {
                const int e = et + i * kEpiThreads;
                rank[i] = 0;
                if (e < E) {
                    const int n = order[e];
                    int r = 0;
                    for (int j = 0; j < E; ++j) {
                        const int m = order[j];
                        r += (m > n || (m == n && j < e)) ? 1 : 0;
                    }
                    rank[i] = r;
                }
            }
            epilogue_sync_n(kEpiThreads);
#pragma unroll
            for (int i = 0; i < (kMaxExperts + 127) / 128; ++i) {
                const int e = et + i * kEpiThreads;
                if (e < E) order[rank[i]] = e;
            }
            epilogue_sync_n(kEpiThreads);
        }
        if (warp == 2) {
            const bool bad = epi_flag[0] != 0;
            // exclusive scan of the item counts in expert order: lane j owns
            // positions [j*per, (j+1)*per)
            const int per = (E + 31) / 32;
            int local = 0;
            for (int i = 0; i < per; ++i) {
                const int p = lane * per + i;
                if (p < E) local += ntiles[order[p]] * n_mt;
            }
            int incl = local;
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            int run = incl - local;
            for (int i = 0; i < per; ++i) {
                const int p = lane * per + i;
                if (p < E) {
                    item_off[p] = run;
                    run += ntiles[order[p]] * n_mt;
                }
            }
            if (lane == 31) item_off[E] = run;
            if (bad && lane == 0) atomicOr(err, DEVERR_OFFSETS);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n_items = item_off[E];
    const bool big = *mode_big != 0;
    // stages: 3 x 64 KB (big items), else 4 x 48 KB.  A narrow stage holds two
    // consecutive k-blocks (two 16 KB A tiles and their rows, at most 64), so
    // that it carries as many weight bytes as a normal one.
    const int S = big ? 3 : 4;
    const int stage_bytes = C::kRingBytes / S;
    const int kpb = narrow ? 2 : 1;          // k-blocks per stage
    const int n_st = n_kb / kpb;             // stages per item (K is a multiple of 128)
    const int slice = big ? 2 * BN : BN;                           // rows per work item at most
    auto item_at = [&](int it) { return decode_item_ordered(it, item_off, order, ntiles, offsets, E, slice); };
    // item j of this CTA is hand-out position blockIdx.x + j * gridDim.x
    const int n_list = static_cast<int>(blockIdx.x) < n_items
                           ? min((n_items - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                                     static_cast<int>(gridDim.x),
                                 C::kList)
                           : 0;
    if (warp >= 2)
        for (int j = threadIdx.x - 64; j < n_list; j += blockDim.x - 64) ilist[j] = item_at(blockIdx.x + j * gridDim.x);
    __syncthreads();
    auto my_item = [&](int j, int it) { return j < C::kList ? ilist[j] : item_at(it); };

    if (warp == 0) {
        // ---- TMA producer -------------------------------------------------
        if (lane == 0) {
            const uint64_t pol_once = l2_policy(1);
            const uint64_t pol_shared = l2_policy(MOE_TC_SHARED_W_POLICY);
            const uint64_t pol_x = l2_policy(MOE_TC_X_POLICY);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int it = blockIdx.x, j = 0; ok && it < n_items; it += gridDim.x, ++j) {
                const Item item = my_item(j, it);
                const int n16 = (item.rows + kBoxRows - 1) / kBoxRows;
                const int row_bytes = n16 * kBoxRows * BK * 2;   // one k-block of the item's rows
                // (the fused gate/up kernel's rows come from the gather warp)
                const uint32_t bytes = C::kA * C::kATileBytes + (GATED && FUSED ? 0 : kpb * row_bytes);
                // w_down tiles past the expert's last feature (M not a multiple
                // of 256) read the next expert's rows, or zero fill past the
                // end of the bank; the epilogue stores none of their results
                const int wy = item.e * M + item.mt * fw;
                const int wy1 = GATED ? wy : wy + BM;
                const uint64_t pol_w = ntiles[item.e] > 1 ? pol_shared : pol_once;
                for (int js = 0; js < n_st; ++js) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + s * stage_bytes;
                    mbar_arrive_expect_tx(&full[s], bytes);
                    issued[s] = static_cast<int>(ph);
                    for (int hk = 0; hk < kpb; ++hk) {
                        const int kb = js * kpb + hk;
                        if (narrow) {
                            // k-block hk: A tile at hk * 16 KB (gate/up: 64 gate rows, then 64 up rows)
                            uint8_t* at = st + hk * C::kATileBytes;
                            tma_load_2d(at, &map_a0, &full[s], kb * KBE, wy, pol_w);
                            if (GATED) tma_load_2d(at + C::kATileBytes / 2, &map_a1, &full[s], kb * KBE, wy, pol_w);
                        } else {
                            tma_load_2d(st, &map_a0, &full[s], kb * KBE, wy, pol_w);
                            tma_load_2d(st + C::kATileBytes, &map_a1, &full[s], kb * KBE, wy1, pol_w);
                        }
                        if (GATED && FUSED) continue;
                        uint8_t* bdst = st + C::kA * C::kATileBytes + hk * row_bytes;
                        // the rows in as few boxes as possible: 64-row boxes, then 16-row ones
                        int r = 0;
                        for (; r + kBigBoxRows <= n16 * kBoxRows; r += kBigBoxRows)
                            tma_load_2d(bdst + r * 128, &map_b_big, &full[s], kb * KBE, item.row0 + r, pol_x);
                        for (; r < n16 * kBoxRows; r += kBoxRows)
                            tma_load_2d(bdst + r * 128, &map_b, &full[s], kb * KBE, item.row0 + r, pol_x);
                    }
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer ---------------------------------------------------
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int toggle = 0;            // slot of the next light item
            uint32_t use0 = 0, use1 = 0;  // uses of each accumulator slot so far
            bool ok = true;
            for (int it = blockIdx.x, j = 0; ok && it < n_items; it += gridDim.x, ++j) {
                const Item item = my_item(j, it);
                const int n16 = (item.rows + kBoxRows - 1) / kBoxRows;
                const uint32_t idesc = F8 ? idesc_e4m3(BM, n16 * kBoxRows) : idesc_bf16(BM, n16 * kBoxRows);
                const bool both = item.rows > BN;
                const int slot = both ? 0 : toggle;
                const uint32_t use_s = slot ? use1 : use0;
                if (!mbar_wait(&acc_empty[slot], (use_s & 1u) ^ 1u, abort_flag, err)) break;
                if (both && !mbar_wait(&acc_empty[1], (use1 & 1u) ^ 1u, abort_flag, err)) break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(slot * BN);
                const int row_bytes = n16 * kBoxRows * BK * 2;
                for (int js = 0; js < n_st; ++js) {
                    if (!mbar_wait(&full[s], ph, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    // gathered rows were written by the generic proxy (cp.async)
                    if (GATED && FUSED) fence_proxy_async_smem();
                    tc_fence_after();
                    // descriptors advance by 32 bytes of K (2 in the low half) per MMA
                    const uint32_t a0 = sdesc_lo(smem_u32(smem + s * stage_bytes));
                    const uint32_t a1 = a0 + (C::kATileBytes >> 4);
                    const uint32_t b = a0 + ((C::kA * C::kATileBytes) >> 4);
                    if (narrow) {
                        // two k-blocks, each one MMA per 16 K on its own A tile and rows
#pragma unroll
                        for (int hk = 0; hk < 2; ++hk) {
                            const uint32_t ah = hk ? a1 : a0;
                            const uint32_t bh = b + static_cast<uint32_t>((hk * row_bytes) >> 4);
#pragma unroll
                            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                                const uint32_t acc = (js | hk | kk) != 0 ? 1u : 0u;
                                if (F8)
                                    umma_e4m3(d0, sdesc_from_lo(ah + 2 * kk), sdesc_from_lo(bh + 2 * kk), idesc, acc);
                                else
                                    umma_bf16(d0, sdesc_from_lo(ah + 2 * kk), sdesc_from_lo(bh + 2 * kk), idesc, acc);
                            }
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                            const uint32_t acc = (js | kk) != 0 ? 1u : 0u;
                            const uint64_t bd = sdesc_from_lo(b + 2 * kk);
                            if (F8) {
                                umma_e4m3(d0, sdesc_from_lo(a0 + 2 * kk), bd, idesc, acc);
                                umma_e4m3(d0 + 2 * BN, sdesc_from_lo(a1 + 2 * kk), bd, idesc, acc);
                            } else {
                                umma_bf16(d0, sdesc_from_lo(a0 + 2 * kk), bd, idesc, acc);
                                umma_bf16(d0 + 2 * BN, sdesc_from_lo(a1 + 2 * kk), bd, idesc, acc);
                            }
                        }
                    }
                    umma_commit(&empty[s]);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&acc_full[slot]);
                if (slot) ++use1;
                else ++use0;
                if (both) {
                    umma_commit(&acc_full[1]);
                    ++use1;
                    toggle = 0;
                } else {
                    toggle ^= 1;
                }
            }
            // every MMA issued above has completed once `drain` flips
            umma_commit(drain);
            mbar_drain(drain, 0);
        }
    } else if (warp < 2 + Ro::kEpiWarps) {
        // ---- epilogue (warps 2..) ----------------------------------------
        // One thread waits (bounded) for the accumulator and publishes the
        // outcome; every epilogue barrier below is reached by all epilogue warps
        // in every iteration, so an abandoned wait cannot leave a warp behind
        // at a barrier.
        const int q = warp & 3;               // TMEM lanes [32q, 32q+32) belong to this warp
        const int et = threadIdx.x - 64;      // 0 .. 32 * epilogue warps - 1
        constexpr int kEpiThreads = 32 * Ro::kEpiWarps;
        const int grp = (warp - 2) >> 2;      // down: chunk group (alternate 32-row chunks)
        const int n_groups = big ? Ro::kEpiWarps / 4 : 1;
        int local = 0;
        int toggle = 0;
        uint32_t use0 = 0, use1 = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++local) {
            const Item item = my_item(local, it);
            const bool both = item.rows > BN;
            const int slot = both ? 0 : toggle;
            const int buf = local & 1;  // flag parity
            if (et == 0) {
                bool got = mbar_wait(&acc_full[slot], (slot ? use1 : use0) & 1u, abort_flag, err);
                if (got && both) got = mbar_wait(&acc_full[1], use1 & 1u, abort_flag, err);
                epi_flag[buf] = got ? 1 : 0;
            }
            epilogue_sync_n(kEpiThreads);
            if (!epi_flag[buf]) {
                ok = false;
                break;
            }
            tc_fence_after();
            // output feature of this lane: gated -> one 128-feature tile (narrow:
            // lanes 0-63 gate, 64-127 up of a 64-feature tile); down -> tile 0 at
            // m, tile 1 at m + 128
            const int m = item.mt * fw + q * 32 + lane;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(slot * BN);
            for (int c0 = 32 * grp; grp < n_groups && c0 < item.rows; c0 += 32 * n_groups) {
                uint32_t g[32], g1[32];
                tmem_ld32(taddr + c0, g);
                if (!narrow) tmem_ld32(taddr + 2 * BN + c0, g1);
                tmem_ld_wait();
                // E4M3 operands: the weight row's scale times the compact row's scale
                float rs[32];
                if (F8) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) rs[j] = c0 + j < item.rows ? __ldg(sc.b + item.row0 + c0 + j) : 0.f;
                }
                if (GATED && narrow) {
                    // the up half (warps of lane quarters 2, 3) goes through shared memory
                    float ws = 1.f;
                    if (F8)
                        ws = __ldg((q < 2 ? sc.a0 : sc.a1) + static_cast<size_t>(item.e) * M + item.mt * fw +
                                   (q & 1) * 32 + lane);
                    if (q >= 2) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            up_stage[((q - 2) * 32 + lane) * 33 + j] =
                                F8 ? __uint_as_float(g[j]) * ws * rs[j] : __uint_as_float(g[j]);
                    }
                    epilogue_sync_n(kEpiThreads);
                    if (q < 2) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float gv = F8 ? __uint_as_float(g[j]) * ws * rs[j] : __uint_as_float(g[j]);
                            const float hv = silu_fast(gv) * up_stage[(q * 32 + lane) * 33 + j];
                            out_stage[j * (BM / 2) + q * 32 + lane] = __float2bfloat16_rn(hv);
                        }
                    }
                    epilogue_sync_n(kEpiThreads);
                    // each row's 64 features (128 bytes) leave as 8 x 16-byte stores
                    __nv_bfloat16* h = static_cast<__nv_bfloat16*>(out);
                    const int chunk = et & 7;
#pragma unroll
                    for (int pass = 0; pass < 2; ++pass) {
                        const int j = pass * 16 + (et >> 3);
                        const int n = c0 + j;
                        if (n < item.rows) {
                            const uint4 v = *reinterpret_cast<const uint4*>(out_stage + j * (BM / 2) + chunk * 8);
                            *reinterpret_cast<uint4*>(h + static_cast<size_t>(item.row0 + n) * M + item.mt * fw +
                                                      chunk * 8) = v;
                        }
                    }
                    epilogue_sync_n(kEpiThreads);
                } else if (GATED) {
                    // SwiGLU into the staged tile: row j, feature q*32 + lane
                    float wsg = 1.f, wsu = 1.f;
                    if (F8) {
                        wsg = __ldg(sc.a0 + static_cast<size_t>(item.e) * M + m);
                        wsu = __ldg(sc.a1 + static_cast<size_t>(item.e) * M + m);
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float gv = F8 ? __uint_as_float(g[j]) * wsg * rs[j] : __uint_as_float(g[j]);
                        const float uv = F8 ? __uint_as_float(g1[j]) * wsu * rs[j] : __uint_as_float(g1[j]);
                        const float hv = silu_fast(gv) * uv;
                        out_stage[j * BM + q * 32 + lane] = __float2bfloat16_rn(hv);
                    }
                    epilogue_sync_n(kEpiThreads);
                    // each row's 128 features (256 bytes) leave as 16 x 16-byte stores
                    __nv_bfloat16* h = static_cast<__nv_bfloat16*>(out);
                    const int chunk = et & 15;
#pragma unroll
                    for (int pass = 0; pass < 4; ++pass) {
                        const int j = pass * 8 + (et >> 4);
                        const int n = c0 + j;
                        if (n < item.rows) {
                            const uint4 v = *reinterpret_cast<const uint4*>(out_stage + j * BM + chunk * 8);
                            *reinterpret_cast<uint4*>(h + static_cast<size_t>(item.row0 + n) * M + item.mt * BM +
                                                      chunk * 8) = v;
                        }
                    }
                    epilogue_sync_n(kEpiThreads);
                } else {
                    const bool has1 = !narrow && m + BM < M;
                    // y row-major [cap][M]; the fused kernel's scratch y is
                    // slice-major instead: slice mt is [cap][its width] at
                    // mt * fw * cap, so concurrent items of one slice write
                    // contiguous memory
                    const int ystride = FUSED ? min(fw, M - item.mt * fw) : M;
                    float* y = static_cast<float*>(out) + (FUSED ? static_cast<size_t>(item.mt) * fw * cap : 0);
                    const int mo = FUSED ? m - item.mt * fw : m;
                    float ws0 = 1.f, ws1 = 1.f;
                    if (F8) {
                        ws0 = __ldg(sc.a0 + static_cast<size_t>(item.e) * M + m);
                        if (has1) ws1 = __ldg(sc.a0 + static_cast<size_t>(item.e) * M + m + BM);
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int n = c0 + j;
                        if (n < item.rows) {
                            float* yr = y + static_cast<size_t>(item.row0 + n) * ystride;
                            yr[mo] = F8 ? __uint_as_float(g[j]) * ws0 * rs[j] : __uint_as_float(g[j]);
                            if (has1) yr[mo + BM] = F8 ? __uint_as_float(g1[j]) * ws1 * rs[j] : __uint_as_float(g1[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&acc_empty[slot]);
                if (both) mbar_arrive(&acc_empty[1]);
                // fused down: hand the stored item to the combine warps (at most
                // two items ahead of them; a failed wait has raised the abort flag)
                if (!GATED && FUSED && mbar_wait(&comb_free[buf], ((local >> 1) & 1) ^ 1u, abort_flag, err))
                    mbar_arrive(&comb_done[buf]);
            }
            if (slot) ++use1;
            else ++use0;
            if (both) {
                ++use1;
                toggle = 0;
            } else {
                toggle ^= 1;
            }
        }
        // zero-fill the unused compact rows R .. cap-1 (the fused down kernel's
        // y is scratch)
        const int R = offsets[E];
        if (ok && !(FUSED && !GATED) && R >= 0 && R <= cap) {
            const int vecs = M * (GATED ? 2 : 4) / 16;
            const int gw = blockIdx.x * Ro::kEpiWarps + (warp - 2);
            const int nw = gridDim.x * Ro::kEpiWarps;
            uint4* o = static_cast<uint4*>(out);
            for (int row = R + gw; row < cap; row += nw)
                for (int v = lane; v < vecs; v += 32) o[static_cast<size_t>(row) * vecs + v] = make_uint4(0, 0, 0, 0);
        }
    } else if (GATED && FUSED) {
        // ---- row-gather warp (fused gate/up) -------------------------------
        // Waits for each stage's slot like the TMA warp and copies 16-byte
        // chunks of token rows -- lane l takes chunk l % 8 of rows l / 8,
        // l / 8 + 4, ... -- then arrives on the stage's full barrier when its
        // copies have landed.
        const uint64_t pol_x = l2_policy(MOE_TC_X_POLICY);
        const size_t xrow = static_cast<size_t>(K) * 2;   // bytes per token row
        const int n_routes = fa.T * fa.k;
        const int chunk = lane & 7;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int it = blockIdx.x, j = 0; ok && it < n_items; it += gridDim.x, ++j) {
            const Item item = my_item(j, it);
            const int N = (item.rows + kBoxRows - 1) / kBoxRows * kBoxRows;
            const int row_bytes = N * BK * 2;
            // the token of every row; padding rows repeat the first row
            __syncwarp();
            for (int n = lane; n < N; n += 32) {
                const int r = fa.route_of_row[item.row0 + (n < item.rows ? n : 0)];
                const bool good = r >= 0 && r < n_routes;
                if (!good) atomicOr(err, DEVERR_OFFSETS);
                tok_s[n] = good ? r / fa.k : 0;
            }
            __syncwarp();
            for (int js = 0; js < n_st; ++js) {
                int got = 1;
                if (lane == 0) got = mbar_wait(&empty[s], ph ^ 1u, abort_flag, err) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    ok = false;
                    break;
                }
                uint8_t* st = smem + s * stage_bytes;
                for (int hk = 0; hk < kpb; ++hk) {
                    const int kb = js * kpb + hk;
                    const uint32_t bdst = smem_u32(st + C::kA * C::kATileBytes + hk * row_bytes);
                    const uint8_t* src = fa.x + kb * (BK * 2) + chunk * 16;
                    // 128B swizzle: chunk c of row n sits at chunk position c ^ (n % 8)
                    for (int n = lane >> 3; n < N; n += 4)
                        cp_async16(bdst + n * 128 + ((chunk ^ (n & 7)) << 4), src + tok_s[n] * xrow, pol_x);
                }
                cp_async_arrive_noinc(&full[s]);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        // every copy lands before the CTA ends (also after an abandoned wait)
        cp_async_wait_all();
    } else if (!GATED && FUSED) {
        // ---- combine warps (fused down) -----------------------------------
        // For each item, once the epilogue has stored its y rows: count every
        // row's slot on its (token, feature slice) counter; the CTA whose count
        // completes the token's unmasked slots adds them into out.  The
        // epilogue's stores reach the counters through its mbarrier arrive (CTA
        // scope) and a gpu-scope release fence here; the completing CTA fences
        // again (acquire) before it reads the other CTAs' rows.
        const int ct = threadIdx.x - 32 * (2 + Ro::kEpiWarps);
        constexpr int kCombThreads = 32 * Ro::kCombWarps;
        const int k = fa.k;
        const int n_routes = fa.T * k;
        const int d4 = M / 4;
        const int per = fw / 4;                 // float4 columns of a token's slice (64 or 32)
        const int tpp = kCombThreads / per;     // tokens per pass
        const int c = ct % per, jt = ct / per;
        const float4* y4 = static_cast<const float4*>(out);
        float4* out4 = reinterpret_cast<float4*>(fa.out);
        int local = 0;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++local) {
            const Item item = my_item(local, it);
            const int b = local & 1;
            if (ct == 0) *comb_flag = mbar_wait(&comb_done[b], (local >> 1) & 1u, abort_flag, err) ? 1 : 0;
            combine_sync();
            if (!*comb_flag) break;
            if (lane == 0) mbar_arrive(&comb_free[b]);
            fence_acq_rel_gpu();
            for (int n = ct; n < item.rows; n += kCombThreads) {
                const int r = fa.route_of_row[item.row0 + n];
                if (r < 0 || r >= n_routes) {
                    atomicOr(err, DEVERR_OFFSETS);
                    continue;
                }
                const int t = r / k;
                const int32_t* rows_t = fa.row_of_route + static_cast<size_t>(t) * k;
                int rows[kMaxK];
                int nv = 0;
#pragma unroll
                for (int sl = 0; sl < kMaxK; ++sl) {
                    rows[sl] = sl < k ? __ldg(rows_t + sl) : -1;
                    if (rows[sl] >= cap) rows[sl] = -1;
                    nv += rows[sl] >= 0 ? 1 : 0;
                }
                const int old = atomicAdd(fa.tile_counts + static_cast<size_t>(t) * fa.cstride + item.mt, 1);
                if (old == nv - 1) {
                    const int p = atomicAdd(const_cast<int*>(list_n), 1);
                    list[p] = t;
#pragma unroll
                    for (int sl = 0; sl < kMaxK; ++sl) list_rows[p * kMaxK + sl] = rows[sl];
                }
            }
            fence_acq_rel_gpu();
            combine_sync();
            const int n_list = *list_n;
            // y is slice-major: slice mt holds rows of w4 float4 columns
            const int w4 = min(per, d4 - item.mt * per);
            const float4* ys = y4 + static_cast<size_t>(item.mt) * per * cap;
            const int col = item.mt * per + c;   // float4 column of out
            // d is a multiple of 128, so a warp's 32 columns are all in range or all out.
            // Two tokens per thread and pass, slots in groups of kSlotGroup, every
            // load of a group in flight before the fixed-order sum.
            if (c < w4) {
                for (int j0 = jt; j0 < n_list; j0 += 2 * tpp) {
                    const bool two = j0 + tpp < n_list;
                    const int jj[2] = {j0, two ? j0 + tpp : j0};
                    float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
                    for (int s0 = 0; s0 < k; s0 += kSlotGroup) {
                        float4 yv[2][kSlotGroup];
                        float ws[2][kSlotGroup];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int* rj = list_rows + jj[u] * kMaxK + s0;
                            const float* w_t = fa.w + static_cast<size_t>(list[jj[u]]) * k + s0;
#pragma unroll
                            for (int sl = 0; sl < kSlotGroup; ++sl) {
                                const int row = s0 + sl < k ? rj[sl] : -1;
                                if (row >= 0) {
                                    yv[u][sl] = __ldcg(ys + static_cast<size_t>(row) * w4 + c);
                                    ws[u][sl] = __ldg(w_t + sl);
                                }
                            }
                        }
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int* rj = list_rows + jj[u] * kMaxK + s0;
#pragma unroll
                            for (int sl = 0; sl < kSlotGroup; ++sl) {
                                if (s0 + sl < k && rj[sl] >= 0) {
                                    acc[u].x = fmaf(ws[u][sl], yv[u][sl].x, acc[u].x);
                                    acc[u].y = fmaf(ws[u][sl], yv[u][sl].y, acc[u].y);
                                    acc[u].z = fmaf(ws[u][sl], yv[u][sl].z, acc[u].z);
                                    acc[u].w = fmaf(ws[u][sl], yv[u][sl].w, acc[u].w);
                                }
                            }
                        }
                    }
                    out4[static_cast<size_t>(list[jj[0]]) * d4 + col] = acc[0];
                    if (two) out4[static_cast<size_t>(list[jj[1]]) * d4 + col] = acc[1];
                    // the y lines of these tokens' slices are dead: drop them from L2
                    __syncwarp();
                    if ((c & 7) == 0) {
                        for (int u = 0; u < (two ? 2 : 1); ++u) {
                            const int* rj = list_rows + jj[u] * kMaxK;
                            for (int sl = 0; sl < k; ++sl)
                                if (rj[sl] >= 0) l2_discard128(ys + static_cast<size_t>(rj[sl]) * w4 + c);
                        }
                    }
                }
            }
            combine_sync();
            if (ct == 0) *list_n = 0;
        }
    }

    // ---- teardown ----------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        // let every TMA copy still in flight land before the CTA's shared
        // memory is released
        for (int s = 0; s < S; ++s)
            if (issued[s] >= 0) mbar_drain(&full[s], static_cast<uint32_t>(issued[s]));
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(C::kTmemCols)
                     : "memory");
    }
}

// Diagnostic of the bounded waits: one thread waits, through mbar_wait, for
// an mbarrier phase that nothing completes, and gives up after limit_ns.
__global__ void bounded_wait_probe_kernel(unsigned long long limit_ns, unsigned* err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, err, limit_ns);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

std::mutex g_mutex;
bool g_attr_set[64][8];

// 2-D bf16 tensor map over a row-major [rows][K] matrix with a box of
// 64 K-elements x box_rows rows and 128-byte swizzle.
moe_status encode_2d(CUtensorMap* map, const void* base, int K, long long rows, int box_rows) {
    return encode_2d_map(map, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, rows, BK, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}

// 2-D E4M3 (one byte per element) tensor map with a box of 128 K-elements
// (one 128-byte swizzle row, like 64 bf16 elements) x box_rows rows.
moe_status encode_2d_u8(CUtensorMap* map, const void* base, int K, long long rows, int box_rows) {
    return encode_2d_map(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, rows, 128, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}

template <bool GATED, bool FUSED, bool F8>
moe_status set_smem_attr() {
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    constexpr int v = (GATED ? 1 : 0) + (FUSED ? 2 : 0) + (F8 ? 4 : 0);
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_attr_set[dev][v]) {
        MOE_CUDA_TRY(cudaFuncSetAttribute(ffn_tc_kernel<GATED, FUSED, F8>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<GATED>::smem_bytes(FUSED)));
        g_attr_set[dev][v] = true;
    }
    return MOE_OK;
}

template <bool GATED, bool FUSED, bool F8 = false>
moe_status launch(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b, const CUtensorMap& bb,
                  const int32_t* offsets, int cap, int E, int K, int M, bool narrow, void* out, const FusedArgs& fa,
                  cudaStream_t st, const DeviceInfo& di, const OpScales& sc = OpScales{}) {
    moe_status s;
    if ((s = set_smem_attr<GATED, FUSED, F8>()) != MOE_OK) return s;
    ffn_tc_kernel<GATED, FUSED, F8>
        <<<di.sm_count, Roles<GATED, FUSED>::kThreads, Cfg<GATED>::smem_bytes(FUSED), st>>>(
            a0, a1, b, bb, offsets, cap, E, K, M, narrow ? 1 : 0, out, di.error_word, fa, sc);
    return cuda_status(cudaGetLastError());
}

}  // namespace

// Narrow items for chunks of at most 64 routes (no expert can have more than
// 64 rows, so two k-blocks of rows fit a stage and the big-item carve-up
// never applies) when even
// an upper bound on the normal items -- min(E, cap) touched experts times
// the feature tiles per expert -- stays under four waves of CTAs.
bool use_narrow(int cap, int E, int tiles_per_expert, const DeviceInfo& di) {
    const long long experts = E < cap ? E : cap;
    return cap <= BN / 2 && experts * tiles_per_expert < 4LL * di.sm_count;
}

moe_status prepare_ffn_tc_gate_up(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                  const void* w_gate, const void* w_up, void* h, const DeviceInfo& di,
                                  FfnTcLaunch* p) {
    moe_status s;
    p->narrow = use_narrow(cap, E, f / BM, di);
    const int wbox = p->narrow ? BM / 2 : BM;
    if ((s = encode_2d(&p->a0, w_gate, d, static_cast<long long>(E) * f, wbox)) != MOE_OK) return s;
    if ((s = encode_2d(&p->a1, w_up, d, static_cast<long long>(E) * f, wbox)) != MOE_OK) return s;
    if ((s = encode_2d(&p->b, xs, d, cap, kBoxRows)) != MOE_OK) return s;
    if ((s = encode_2d(&p->bb, xs, d, cap, kBigBoxRows)) != MOE_OK) return s;
    p->gated = true;
    p->offsets = offsets;
    p->cap = cap;
    p->E = E;
    p->K = d;
    p->M = f;
    p->out = h;
    return MOE_OK;
}

moe_status prepare_ffn_tc_down(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                               const void* w_down, float* y, const DeviceInfo& di, FfnTcLaunch* p) {
    moe_status s;
    if ((s = encode_2d(&p->a0, w_down, f, static_cast<long long>(E) * d, BM)) != MOE_OK) return s;
    p->a1 = p->a0;
    if ((s = encode_2d(&p->b, h, f, cap, kBoxRows)) != MOE_OK) return s;
    if ((s = encode_2d(&p->bb, h, f, cap, kBigBoxRows)) != MOE_OK) return s;
    p->narrow = use_narrow(cap, E, (d + 2 * BM - 1) / (2 * BM), di);
    p->gated = false;
    p->offsets = offsets;
    p->cap = cap;
    p->E = E;
    p->K = f;
    p->M = d;
    p->out = y;
    return MOE_OK;
}

moe_status launch_ffn_tc_prepared(const FfnTcLaunch& p, cudaStream_t st, const DeviceInfo& di) {
    if (!p.narrow && use_pair_ffn(p.cap)) return launch_ffn_pair_prepared(p, st, di);
    if (p.gated)
        return launch<true, false>(p.a0, p.a1, p.b, p.bb, p.offsets, p.cap, p.E, p.K, p.M, p.narrow, p.out,
                                   FusedArgs{}, st, di);
    return launch<false, false>(p.a0, p.a1, p.b, p.bb, p.offsets, p.cap, p.E, p.K, p.M, p.narrow, p.out,
                                FusedArgs{}, st, di);
}

moe_status launch_ffn_tc_gate_up(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                 const void* w_gate, const void* w_up, void* h, cudaStream_t st,
                                 const DeviceInfo& di) {
    FfnTcLaunch p;
    moe_status s = prepare_ffn_tc_gate_up(xs, offsets, cap, E, d, f, w_gate, w_up, h, di, &p);
    if (s != MOE_OK) return s;
    return launch_ffn_tc_prepared(p, st, di);
}

moe_status launch_ffn_tc_down(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                              const void* w_down, float* y, cudaStream_t st, const DeviceInfo& di) {
    FfnTcLaunch p;
    moe_status s = prepare_ffn_tc_down(h, offsets, cap, E, d, f, w_down, y, di, &p);
    if (s != MOE_OK) return s;
    return launch_ffn_tc_prepared(p, st, di);
}

// A5 with E4M3 weights and E4M3 compact rows (kind::f8f6f4 MMAs).  Narrow
// items hold two 128-element k-blocks per stage, so they need K to be a
// multiple of 256.
moe_status launch_ffn_w8a8_gate_up(const uint8_t* xs, const float* xs_scale, const int32_t* offsets, int cap, int E,
                                   int d, int f, const uint8_t* q_gate, const float* s_gate, const uint8_t* q_up,
                                   const float* s_up, void* h, cudaStream_t st, const DeviceInfo& di) {
    CUtensorMap ma0, ma1, mb, mbb;
    moe_status s;
    const bool narrow = use_narrow(cap, E, f / BM, di) && d % 256 == 0;
    const int wbox = narrow ? BM / 2 : BM;
    if ((s = encode_2d_u8(&ma0, q_gate, d, static_cast<long long>(E) * f, wbox)) != MOE_OK) return s;
    if ((s = encode_2d_u8(&ma1, q_up, d, static_cast<long long>(E) * f, wbox)) != MOE_OK) return s;
    if ((s = encode_2d_u8(&mb, xs, d, cap, kBoxRows)) != MOE_OK) return s;
    if ((s = encode_2d_u8(&mbb, xs, d, cap, kBigBoxRows)) != MOE_OK) return s;
    if (!narrow && use_pair_ffn(cap))
        return launch_ffn_pair_w8a8(true, ma0, ma1, mb, mbb, offsets, cap, E, d, f, h, s_gate, s_up, xs_scale, st, di);
    return launch<true, false, true>(ma0, ma1, mb, mbb, offsets, cap, E, d, f, narrow, h, FusedArgs{}, st, di,
                                     OpScales{s_gate, s_up, xs_scale});
}

// A6 with E4M3 weights and E4M3 rows of h.
moe_status launch_ffn_w8a8_down(const uint8_t* hq, const float* h_scale, const int32_t* offsets, int cap, int E,
                                int d, int f, const uint8_t* q_down, const float* s_down, float* y, cudaStream_t st,
                                const DeviceInfo& di) {
    CUtensorMap ma0, mb, mbb;
    moe_status s;
    if ((s = encode_2d_u8(&ma0, q_down, f, static_cast<long long>(E) * d, BM)) != MOE_OK) return s;
    if ((s = encode_2d_u8(&mb, hq, f, cap, kBoxRows)) != MOE_OK) return s;
    if ((s = encode_2d_u8(&mbb, hq, f, cap, kBigBoxRows)) != MOE_OK) return s;
    const bool narrow = use_narrow(cap, E, (d + 2 * BM - 1) / (2 * BM), di) && f % 256 == 0;
    if (!narrow && use_pair_ffn(cap))
        return launch_ffn_pair_w8a8(false, ma0, ma0, mb, mbb, offsets, cap, E, f, d, y, s_down, nullptr, h_scale, st,
                                    di);
    return launch<false, false, true>(ma0, ma0, mb, mbb, offsets, cap, E, f, d, narrow, y, FusedArgs{}, st, di,
                                      OpScales{s_down, nullptr, h_scale});
}

moe_status launch_ffn_tc_gate_up_gather(const void* x, int T, int k, const int32_t* route_of_row,
                                        const int32_t* offsets, int E, int d, int f, const void* w_gate,
                                        const void* w_up, void* h, cudaStream_t st, const DeviceInfo& di) {
    CUtensorMap ma0, ma1, mb;
    moe_status s;
    const int cap = T * k;
    const bool narrow = use_narrow(cap, E, f / BM, di);
    const int wbox = narrow ? BM / 2 : BM;
    if ((s = encode_2d(&ma0, w_gate, d, static_cast<long long>(E) * f, wbox)) != MOE_OK) return s;
    if ((s = encode_2d(&ma1, w_up, d, static_cast<long long>(E) * f, wbox)) != MOE_OK) return s;
    // the row maps are not used by the gather warp; a valid map over x stands in
    if ((s = encode_2d(&mb, x, d, T, 1)) != MOE_OK) return s;
    FusedArgs fa{};
    fa.x = static_cast<const uint8_t*>(x);
    fa.route_of_row = route_of_row;
    fa.T = T;
    fa.k = k;
    return launch<true, true>(ma0, ma1, mb, mb, offsets, cap, E, d, f, narrow, h, fa, st, di);
}

moe_status launch_ffn_tc_down_combine(const void* h, const int32_t* offsets, int T, int k, int E, int d, int f,
                                      const void* w_down, const int32_t* route_of_row,
                                      const int32_t* row_of_route, const float* w, float* y,
                                      int32_t* tile_counts, float* out, cudaStream_t st, const DeviceInfo& di) {
    CUtensorMap ma0, mb, mbb;
    moe_status s;
    const int cap = T * k;
    if ((s = encode_2d(&ma0, w_down, f, static_cast<long long>(E) * d, BM)) != MOE_OK) return s;
    if ((s = encode_2d(&mb, h, f, cap, kBoxRows)) != MOE_OK) return s;
    if ((s = encode_2d(&mbb, h, f, cap, kBigBoxRows)) != MOE_OK) return s;
    const bool narrow = use_narrow(cap, E, (d + 2 * BM - 1) / (2 * BM), di);
    FusedArgs fa{};
    fa.route_of_row = route_of_row;
    fa.row_of_route = row_of_route;
    fa.w = w;
    fa.out = out;
    fa.tile_counts = tile_counts;
    fa.T = T;
    fa.k = k;
    fa.cstride = tile_counts_per_token(d);
    return launch<false, true>(ma0, ma0, mb, mbb, offsets, cap, E, f, d, narrow, y, fa, st, di);
}

}  // namespace moe

extern "C" moe_status moe_selftest_bounded_wait(int limit_ms, void* stream) {
    using namespace moe;
    MOE_REQUIRE(limit_ms >= 1 && limit_ms <= 5000);
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    bounded_wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<unsigned long long>(limit_ms) * 1000000ull, di.error_word);
    return cuda_status(cudaGetLastError());
}
