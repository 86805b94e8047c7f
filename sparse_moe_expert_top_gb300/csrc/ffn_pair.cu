// Grouped expert FFN (A5 gate/up + SwiGLU, A6 down) on pairs of SMs.
//
// The same work as the one-SM tensor-core kernel, for chunks with many rows
// per expert: a cluster of two CTAs issues tcgen05.mma.cta_group::2 with
// M = 256, so one MMA instruction covers 256 weight rows (128 in each CTA's
// shared memory) against up to 256 compact rows (the CTA's own half of them
// in its shared memory, exchanged between the two SMs by the tensor cores).
// Per 64-K stage each SM then loads 32 KB of weights and at most 16 KB of
// rows, where the one-SM kernel loads 32 KB and up to 32 KB for the same
// MMA work, and each SM's shared memory serves half the operand reads.
//
// Roles per CTA: warp 0 TMA producer, warp 1 MMA issuer (active in the even
// CTA of the pair only), then eight epilogue warps (two groups of four taking
// alternate 32-row chunks).  Both CTAs run the same item sequence, which the
// even CTA's producer takes from a per-launch counter and publishes to both.
// The odd CTA's TMA loads complete on the even CTA's full barrier (the
// cta_group::2 form of the bulk tensor copy); the MMA thread's commits arrive
// on the barriers of both CTAs (multicast); the odd CTA's epilogue releases
// an accumulator on the even CTA's barrier.
//
// Work item: (expert e, a 256-feature tile of gate/up or a 512-feature tile
// of down, a slice of at most 256 of the expert's compact rows).  The item's
// rows are padded to N = 32 * ceil(rows / 32); the even CTA holds rows
// [0, N/2) of the slice and the odd CTA rows [N/2, N), so accumulator column
// c belongs to compact row row0 + c in both CTAs' tensor memory.
#include <cuda_bf16.h>

#include "tc_common.cuh"

#ifndef MOE_PAIR_MIN_ROUTES
#define MOE_PAIR_MIN_ROUTES 24576
#endif

namespace moe {
namespace {

constexpr int PBM = 128;                 // weight rows per CTA and tile
constexpr int kRowBytes = 128;           // one 128-byte swizzle row of K per operand row and stage
constexpr int kPairSlice = 256;          // compact rows per item at most (the MMA's N)
constexpr int kPairStages = 4;
constexpr int kATile = PBM * kRowBytes;  // 16 KB
constexpr int kBTile = 128 * kRowBytes;  // 16 KB: the CTA's half of N rows
constexpr int kStageBytes = 2 * kATile + kBTile;
constexpr int kRingBytes = kPairStages * kStageBytes;  // 192 KB
constexpr int kCtrlBytes = 4096;
// Dynamic hand-out: the even CTA's producer takes each next position of the
// hand-out order from a per-launch counter and publishes the decoded item in
// a ring of kSched slots of both CTAs (one mbarrier per slot).  The decode
// reads shared copies of the offsets and of the block starts of the order.
constexpr int kSched = 16;
constexpr int kListBytes = 8192;
constexpr int kSchedOff = 0;                                   // kSched items of 16 bytes
constexpr int kItemFullOff = kSchedOff + kSched * 16;          // kSched mbarriers
constexpr int kOffsOff = kItemFullOff + kSched * 8;            // offsets[0 .. E]
constexpr int kBstartOff = kOffsOff + (kMaxExperts + 4) * 4;   // block starts of the hand-out order
constexpr int kBstartCap = (kListBytes - kBstartOff) / 4;
static_assert(kBstartCap > 1024, "room for the block-start table");
constexpr int kSmallBox = 16;            // rows per small TMA box
constexpr int kLargeBox = 64;            // rows per large TMA box
constexpr int kTmemCols = 512;           // gate (tile 0) at 0, up (tile 1) at 256; two 128-column slots each

template <bool GATED>
struct PairCfg {
    // two groups of 4 epilogue warps take alternate 32-row chunks of an item
    static constexpr int kEpiWarps = 8;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
    static constexpr int kFeat = GATED ? 2 * PBM : 4 * PBM;  // output features per item (the pair's)
    static constexpr int kOutStage = GATED ? 2 * 32 * PBM * 2 : 0;   // a 32-row bf16 tile of h per group
    static constexpr int kSmemBytes = kRingBytes + kCtrlBytes + kListBytes + kOutStage + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
};

__device__ __forceinline__ float silu_pair(float g) { return __fdividef(g, 1.f + __expf(-g)); }

// Named barrier 1 among the epilogue threads of this CTA.
__device__ __forceinline__ void epilogue_sync_n_pair(int threads) {
    asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
}

// Named barrier 2 + g among the 128 threads of epilogue group g.
__device__ __forceinline__ void group_sync(int g) { asm volatile("bar.sync %0, 128;" ::"r"(2 + g) : "memory"); }

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// All threads of both CTAs; returns once every thread of the pair has arrived.
__device__ __forceinline__ void pair_sync() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// Arrive on an mbarrier of either CTA of the pair without release semantics.
// Used where the only thing the waiting side depends on is tensor-memory
// reads that have already completed (tcgen05.wait::ld, then the tcgen05
// fence): a release at cluster scope would also hold the warp until its
// global stores are performed, about a microsecond on every item (measured:
// 8,192-token chunk, gate/up 1.364 -> 1.352 ms, down 0.783 -> 0.768 ms).
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// 2-D tile load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int x,
                                                 int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

template <bool F8>
__device__ __forceinline__ void umma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    if (F8)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Arrives on the barrier at this shared-memory offset in both CTAs once every
// MMA issued so far has completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
    const uint16_t both = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(both)
        : "memory");
}

// Rows of the item held by each CTA (a multiple of 16).
__device__ __forceinline__ int half_rows(int rows) { return 16 * ((rows + 31) / 32); }

// ---------------------------------------------------------------------------
// GATED: out = h (bf16 [cap][M]) = silu(A0 . xs) * (A1 . xs), A0 = w_gate,
// A1 = w_up, M = f, K = d.  Otherwise out = y (fp32 [cap][M]) = A0 . h,
// A0 = w_down, M = d, K = f.  F8: E4M3 operands (kind::f8f6f4), the
// accumulators scaled in the epilogue by the weight row's and the compact
// row's scales.
// ---------------------------------------------------------------------------
template <bool GATED, bool F8>
__global__ void __launch_bounds__(PairCfg<GATED>::kThreads, 1)
    ffn_pair_kernel(const __grid_constant__ CUtensorMap map_a0, const __grid_constant__ CUtensorMap map_a1,
                    const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_b_big,
                    const int32_t* __restrict__ offsets, int cap, int E, int K, int M, void* __restrict__ out,
                    unsigned* err, const float* __restrict__ sa0, const float* __restrict__ sa1,
                    const float* __restrict__ sb, int* __restrict__ ticket) {
    using C = PairCfg<GATED>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* ctrl = smem + kRingBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
    uint64_t* empty = full + kPairStages;
    uint64_t* acc_full = empty + kPairStages;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* issued = reinterpret_cast<int*>(tmem_slot + 2);
    int* item_off = issued + kPairStages;           // E + 1 entries
    int* ntiles = item_off + kMaxExperts + 1;        // E entries
    volatile int* epi_flag = reinterpret_cast<volatile int*>(ntiles + kMaxExperts);  // 2 entries
    int* order = const_cast<int*>(epi_flag + 2);     // experts: the heavy ones, then the light ones (E entries)
    int* heavy_items = order + kMaxExperts;          // items of the heavy experts
    int* heavy_experts = heavy_items + 1;            // how many experts are heavy
    uint8_t* lreg = ctrl + kCtrlBytes;
    Item* sched = reinterpret_cast<Item*>(lreg + kSchedOff);               // published items, slot j % kSched
    uint64_t* item_full = reinterpret_cast<uint64_t*>(lreg + kItemFullOff);
    int* soffs = reinterpret_cast<int*>(lreg + kOffsOff);
    int* bstart = reinterpret_cast<int*>(lreg + kBstartOff);
    __nv_bfloat16* out_stage = reinterpret_cast<__nv_bfloat16*>(ctrl + kCtrlBytes + kListBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    constexpr int KBE = F8 ? 128 : 64;   // K elements per stage
    const int n_kb = K / KBE;
    const int n_mt = (M + C::kFeat - 1) / C::kFeat;

    // ---- prologue ------------------------------------------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            issued[s] = -1;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 2 * C::kEpiWarps);   // the epilogue warps of both CTAs
        }
        for (int i = 0; i < kSched; ++i) mbar_init(&item_full[i], 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&map_a0);
        if (GATED) prefetch_tmap(&map_a1);
        prefetch_tmap(&map_b);
        prefetch_tmap(&map_b_big);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    if (warp == 2) {
        // Item table (identical in both CTAs).  Experts with more than one
        // row slice ("heavy": their weight tiles serve several slices from L2,
        // the MMAs set the pace) come first in `order`, the others ("light":
        // each weight tile streamed from HBM for one slice) after them, each
        // group in expert-id order; item_off is the exclusive scan of the item
        // counts in that order.  The items are then handed out interleaved
        // (item_at below), so that at any time some pairs run tensor-bound
        // heavy items while others stream light ones.
        bool bad = false;
        for (int e = lane; e < E; e += 32) {
            const int lo = offsets[e], hi = offsets[e + 1];
            bad |= lo < 0 || hi < lo || hi > cap;
        }
        bad = __any_sync(0xffffffffu, bad);
        const int per = (E + 31) / 32;                 // lane j owns experts / positions [j*per, (j+1)*per)
        const int first = min(lane * per, E);
        int nheavy = 0;
        for (int i = 0; i < per; ++i) {
            const int e = lane * per + i;
            if (e < E) {
                const int n = bad ? 0 : offsets[e + 1] - offsets[e];
                ntiles[e] = (n + kPairSlice - 1) / kPairSlice;
                nheavy += ntiles[e] > 1 ? 1 : 0;
            }
        }
        int hincl = nheavy;
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, hincl, off);
            if (lane >= off) hincl += o;
        }
        const int n_heavy = __shfl_sync(0xffffffffu, hincl, 31);
        int hpos = hincl - nheavy;                      // heavy experts before this lane's
        int lpos = n_heavy + (first - hpos);            // light experts go after all heavy ones
        for (int i = 0; i < per; ++i) {
            const int e = lane * per + i;
            if (e < E) order[ntiles[e] > 1 ? hpos++ : lpos++] = e;
        }
        __syncwarp();
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
        __syncwarp();
        if (lane == 0) {
            *heavy_items = item_off[n_heavy];
            *heavy_experts = n_heavy;
        }
        if (bad && lane == 0 && rank == 0) atomicOr(err, DEVERR_OFFSETS);
    }
    tc_fence_before();
    __syncthreads();
    pair_sync();   // both CTAs' barriers are initialised before either signals the other's
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n_items = item_off[E];
    const int n_heavy_items = *heavy_items;
    const int n_groups = *heavy_experts * n_mt;       // heavy (expert, feature tile) groups
    const int n_light = n_items - n_heavy_items;
    // The hand-out order is a sequence of blocks, one per heavy group b (in
    // expert, feature-tile order): the group's row slices, consecutive so
    // that pairs running them at the same time share its weight tiles in L2,
    // then light items in proportion to the group's slices, so that heavy
    // and light items keep one ratio along the whole order.  With H_b the
    // heavy items before block b (H of them, L light ones), block b starts at
    //   B(b) = H_b + floor(H_b L / H),  H_b = item_off[b / n_mt] + (b % n_mt) * ntiles.
    const bool table = n_groups <= kBstartCap;
    auto block_start_of = [&](int b) {
        const int ei = b / n_mt, mt = b - ei * n_mt;
        const int hb = item_off[ei] + mt * ntiles[order[ei]];
        return hb + static_cast<int>(static_cast<long long>(hb) * n_light / n_heavy_items);
    };
    if (warp >= 2) {
        // shared copies for the decode: the block starts and the offsets
        for (int b = threadIdx.x - 64; table && b < n_groups; b += 32 * C::kEpiWarps) bstart[b] = block_start_of(b);
        for (int e = threadIdx.x - 64; e <= E; e += 32 * C::kEpiWarps) soffs[e] = offsets[e];
    }
    __syncthreads();
    auto item_at = [&](int p) {
        int u = p;
        if (n_groups > 0) {
            auto block_start = [&](int b) { return table ? bstart[b] : block_start_of(b); };
            int lo = 0, hi = n_groups - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (block_start(mid) <= p) lo = mid;
                else hi = mid - 1;
            }
            const int ei = lo / n_mt, mt = lo - ei * n_mt;
            const int size = ntiles[order[ei]];
            const int head = item_off[ei] + mt * size;    // the group's first item
            const int b0 = block_start(lo);
            const int o = p - b0;
            // light items handed out before block lo: b0 - head
            u = o < size ? head + o : n_heavy_items + (b0 - head) + (o - size);
        }
        int lo = 0, hi = E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (item_off[mid] <= u) lo = mid;
            else hi = mid - 1;
        }
        Item r;
        r.e = order[lo];
        const int local = u - item_off[lo];
        const int n = ntiles[r.e];
        r.mt = local / n;
        const int nt = local - r.mt * n;
        r.row0 = soffs[r.e] + nt * kPairSlice;
        r.rows = min(kPairSlice, soffs[r.e + 1] - r.row0);
        return r;
    };

    // Item j of this pair: the even CTA's producer takes hand-out position
    // `pair` first, then n_pairs + (the counter's next value) for each further
    // item, and publishes the decoded item (e = -1 past the last position) in
    // slot j % kSched of both CTAs; every other role waits for the slot.  No
    // role is kSched items behind the producer: the producer runs at most the
    // stage ring ahead of the MMA thread, which runs at most two items ahead of
    // the epilogues of both CTAs.
    auto publish = [&](int j, const Item& it) {
        const int q = j % kSched;
        sched[q] = it;
        mbar_arrive(&item_full[q]);
        // the odd CTA's copy: an asynchronous store that completes on its slot barrier
        const uint32_t rbar = map_to_rank(smem_u32(&item_full[q]), 1);
        const uint32_t rdst = map_to_rank(smem_u32(&sched[q]), 1);
        asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], 16;" ::"r"(rbar)
                     : "memory");
        asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                         rdst),
                     "r"(it.e), "r"(it.mt), "r"(it.row0), "r"(it.rows), "r"(rbar)
                     : "memory");
    };
    auto wait_item = [&](int j) {
        return mbar_wait(&item_full[j % kSched], static_cast<uint32_t>(j / kSched) & 1u, abort_flag, err);
    };

    if (warp == 0) {
        // ---- TMA producer (both CTAs) ------------------------------------------
        if (lane == 0) {
            const uint64_t pol_once = l2_policy(1);
            const uint64_t pol_shared = l2_policy(2);
            const uint64_t pol_x = l2_policy(2);
            const uint32_t full_lead = map_to_rank(smem_u32(full), 0);   // the even CTA's full[0]
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            int t_next = pair;
            for (int j = 0; ok; ++j) {
                Item item;
                if (rank == 0) {
                    const int t = t_next;
                    // the next position now, used one item later (the atomic's latency hides behind this item)
                    if (t < n_items) t_next = n_pairs + atomicAdd(ticket, 1);
                    if (t < n_items) {
                        item = item_at(t);
                    } else {
                        item.e = -1;
                        item.mt = item.row0 = item.rows = 0;
                    }
                    publish(j, item);
                } else {
                    if (!wait_item(j)) break;
                    item = sched[j % kSched];
                }
                if (item.e < 0) break;
                const int nh = half_rows(item.rows);
                const int my0 = item.row0 + static_cast<int>(rank) * nh;
                const uint32_t bytes = 2 * kATile + nh * kRowBytes;   // this CTA's share of a stage
                // weight tiles past the expert's last feature read the next
                // expert's rows (or zero fill past the bank); none of their
                // results is stored
                const int wy0 = item.e * M + item.mt * C::kFeat + static_cast<int>(rank) * PBM;
                const int wy1 = GATED ? wy0 : wy0 + 2 * PBM;
                const uint64_t pol_w = ntiles[item.e] > 1 ? pol_shared : pol_once;
                for (int kb = 0; kb < n_kb; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + s * kStageBytes;
                    if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * bytes);
                    issued[s] = static_cast<int>(ph);
                    const uint32_t bar = full_lead + 8u * static_cast<uint32_t>(s);
                    tma_load_2d_pair(st, &map_a0, bar, kb * KBE, wy0, pol_w);
                    tma_load_2d_pair(st + kATile, GATED ? &map_a1 : &map_a0, bar, kb * KBE, wy1, pol_w);
                    uint8_t* bdst = st + 2 * kATile;
                    int r = 0;
                    for (; r + kLargeBox <= nh; r += kLargeBox)
                        tma_load_2d_pair(bdst + r * kRowBytes, &map_b_big, bar, kb * KBE, my0 + r, pol_x);
                    for (; r < nh; r += kSmallBox)
                        tma_load_2d_pair(bdst + r * kRowBytes, &map_b, bar, kb * KBE, my0 + r, pol_x);
                    if (++s == kPairStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer (even CTA) ---------------------------------------------
        if (lane == 0 && rank == 0) {
            int s = 0;
            uint32_t ph = 0;
            int toggle = 0;
            uint32_t use0 = 0, use1 = 0;
            bool ok = true;
            for (int j = 0; ok; ++j) {
                if (!wait_item(j)) break;
                const Item item = sched[j % kSched];
                if (item.e < 0) break;
                const int N = 2 * half_rows(item.rows);
                const uint32_t idesc = F8 ? idesc_e4m3(2 * PBM, N) : idesc_bf16(2 * PBM, N);
                const bool both = item.rows > 128;
                const int slot = both ? 0 : toggle;
                const uint32_t use_s = slot ? use1 : use0;
                if (!mbar_wait(&acc_empty[slot], (use_s & 1u) ^ 1u, abort_flag, err)) break;
                if (both && !mbar_wait(&acc_empty[1], (use1 & 1u) ^ 1u, abort_flag, err)) break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(slot * 128);
                for (int kb = 0; kb < n_kb; ++kb) {
                    if (!mbar_wait(&full[s], ph, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sdesc_lo(smem_u32(smem + s * kStageBytes));
                    const uint32_t a1 = a0 + (kATile >> 4);
                    const uint32_t b = a0 + ((2 * kATile) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
                        const uint64_t bd = sdesc_from_lo(b + 2 * kk);
                        umma_pair<F8>(d0, sdesc_from_lo(a0 + 2 * kk), bd, idesc, acc);
                        umma_pair<F8>(d0 + 256, sdesc_from_lo(a1 + 2 * kk), bd, idesc, acc);
                    }
                    umma_commit_pair(&empty[s]);
                    if (++s == kPairStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair(&acc_full[slot]);
                if (slot) ++use1;
                else ++use0;
                if (both) {
                    umma_commit_pair(&acc_full[1]);
                    ++use1;
                    toggle = 0;
                } else {
                    toggle ^= 1;
                }
            }
            // every MMA issued above has completed once `drain` flips (in both CTAs)
            umma_commit_pair(drain);
            mbar_drain(drain, 0);
        }
    } else {
        // ---- epilogue (both CTAs) ----------------------------------------------
        const int q = warp & 3;
        const int et = threadIdx.x - 64;
        constexpr int kEpiThreads = 32 * C::kEpiWarps;
        const int grp = (warp - 2) >> 2;
        __nv_bfloat16* stage_g = out_stage + grp * 32 * PBM;   // gate/up: this group's staging tile
        const uint32_t acc_empty_lead = map_to_rank(smem_u32(acc_empty), 0);
        int local = 0;
        int toggle = 0;
        uint32_t use0 = 0, use1 = 0;
        bool ok = true;
        for (;; ++local) {
            const int buf = local & 1;
            if (et == 0) {
                // 1: the item's accumulators are ready; 2: no further item; 0: a wait timed out
                int flag = wait_item(local) ? 1 : 0;
                if (flag) {
                    const Item it0 = sched[local % kSched];
                    if (it0.e < 0) {
                        flag = 2;
                    } else {
                        const bool both0 = it0.rows > 128;
                        const int slot0 = both0 ? 0 : toggle;
                        bool got = mbar_wait(&acc_full[slot0], (slot0 ? use1 : use0) & 1u, abort_flag, err);
                        if (got && both0) got = mbar_wait(&acc_full[1], use1 & 1u, abort_flag, err);
                        flag = got ? 1 : 0;
                    }
                }
                epi_flag[buf] = flag;
            }
            epilogue_sync_n_pair(kEpiThreads);
            const int flag = epi_flag[buf];
            if (flag == 2) break;
            if (flag == 0) {
                ok = false;
                break;
            }
            // the slot's phase has completed (seen by thread 0 of the epilogue): each
            // thread takes it too before reading the slot
            for (int spin = 0;
                 spin < 4096 && !mbar_try_wait(smem_u32(&item_full[local % kSched]), static_cast<uint32_t>(local / kSched) & 1u);
                 ++spin) {
            }
            const Item item = sched[local % kSched];
            const bool both = item.rows > 128;
            const int slot = both ? 0 : toggle;
            tc_fence_after();
            // this CTA's features: tile 0 at fb + [0, 128), tile 1 (down) at fb + 256 + [0, 128)
            const int fb = item.mt * C::kFeat + static_cast<int>(rank) * PBM;
            const int m = fb + q * 32 + lane;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(slot * 128);
            // down: the second group only for 256-row items (light items' stores are few)
            const int n_groups = (GATED || both) ? 2 : 1;
            // Hands the accumulator slots back to the MMA thread of the even CTA,
            // once per warp and item, as soon as the warp's tensor-memory reads of
            // the item are done: before its last chunk's stores, which need no
            // ordering against the next MMAs.
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_remote_relaxed(acc_empty_lead + 8u * static_cast<uint32_t>(slot));
                    if (both) mbar_arrive_remote_relaxed(acc_empty_lead + 8u);
                }
            };
            bool released = false;
            for (int c0 = 32 * grp; grp < n_groups && c0 < item.rows; c0 += 32 * n_groups) {
                uint32_t g[32], g1[32];
                tmem_ld32(taddr + c0, g);
                tmem_ld32(taddr + 256 + c0, g1);
                tmem_ld_wait();
                if (c0 + 32 * n_groups >= item.rows) {   // the warp's last chunk of the item
                    release();
                    released = true;
                }
                float rs[32];
                if (F8) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) rs[j] = c0 + j < item.rows ? __ldg(sb + item.row0 + c0 + j) : 0.f;
                }
                if (GATED) {
                    const bool valid = fb < M;   // the whole 128-feature tile, f being a multiple of 128
                    float wsg = 1.f, wsu = 1.f;
                    if (F8 && valid) {
                        wsg = __ldg(sa0 + static_cast<size_t>(item.e) * M + m);
                        wsu = __ldg(sa1 + static_cast<size_t>(item.e) * M + m);
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float gv = F8 ? __uint_as_float(g[j]) * wsg * rs[j] : __uint_as_float(g[j]);
                        const float uv = F8 ? __uint_as_float(g1[j]) * wsu * rs[j] : __uint_as_float(g1[j]);
                        stage_g[j * PBM + q * 32 + lane] = __float2bfloat16_rn(silu_pair(gv) * uv);
                    }
                    group_sync(grp);
                    __nv_bfloat16* h = static_cast<__nv_bfloat16*>(out);
                    const int eg = et - 128 * grp;   // thread of the group
                    const int chunk = eg & 15;
#pragma unroll
                    for (int pass = 0; pass < 4; ++pass) {
                        const int j = pass * 8 + (eg >> 4);
                        const int n = c0 + j;
                        if (valid && n < item.rows) {
                            const uint4 v = *reinterpret_cast<const uint4*>(stage_g + j * PBM + chunk * 8);
                            *reinterpret_cast<uint4*>(h + static_cast<size_t>(item.row0 + n) * M + fb + chunk * 8) = v;
                        }
                    }
                    group_sync(grp);   // (the groups run different numbers of chunks: no CTA-wide barrier here)
                } else {
                    const bool has0 = m < M, has1 = m + 2 * PBM < M;
                    float ws0 = 1.f, ws1 = 1.f;
                    if (F8) {
                        if (has0) ws0 = __ldg(sa0 + static_cast<size_t>(item.e) * M + m);
                        if (has1) ws1 = __ldg(sa0 + static_cast<size_t>(item.e) * M + m + 2 * PBM);
                    }
                    float* y = static_cast<float*>(out);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int n = c0 + j;
                        if (n < item.rows) {
                            float* yr = y + static_cast<size_t>(item.row0 + n) * M;
                            if (has0) yr[m] = F8 ? __uint_as_float(g[j]) * ws0 * rs[j] : __uint_as_float(g[j]);
                            if (has1)
                                yr[m + 2 * PBM] = F8 ? __uint_as_float(g1[j]) * ws1 * rs[j] : __uint_as_float(g1[j]);
                        }
                    }
                }
            }
            if (!released) release();   // a warp without a chunk of this item
            if (slot) ++use1;
            else ++use0;
            if (both) {
                ++use1;
                toggle = 0;
            } else {
                toggle ^= 1;
            }
        }
        // zero-fill the unused compact rows R .. cap-1
        const int R = offsets[E];
        if (ok && R >= 0 && R <= cap) {
            const int vecs = M * (GATED ? 2 : 4) / 16;
            const int gw = blockIdx.x * C::kEpiWarps + (warp - 2);
            const int nw = gridDim.x * C::kEpiWarps;
            uint4* o = static_cast<uint4*>(out);
            for (int row = R + gw; row < cap; row += nw)
                for (int v = lane; v < vecs; v += 32) o[static_cast<size_t>(row) * vecs + v] = make_uint4(0, 0, 0, 0);
        }
    }

    // ---- teardown ----------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        // the last CTA out clears the launch's counter line for the next launch on it
        __threadfence();
        if (atomicAdd(ticket + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            ticket[0] = 0;
            ticket[1] = 0;
        }
    }
    if (threadIdx.x == 0) {
        if (rank == 0 && *abort_flag) {
            // copies still in flight (both CTAs' shares count on these barriers)
            for (int s = 0; s < kPairStages; ++s)
                if (issued[s] >= 0) mbar_drain(&full[s], static_cast<uint32_t>(issued[s]));
        }
        // the even CTA's final commit reaches this CTA's drain barrier too
        if (rank == 1) mbar_drain(drain, 0);
    }
    __syncthreads();
    // neither CTA leaves while the other may still signal its barriers or
    // the tensor cores may still read its shared memory
    pair_sync();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
}


// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

struct PairCache {
    unsigned long long ctx;
    int pairs;   // co-resident clusters of two
};
std::mutex g_pair_mutex;
PairCache g_pair_cache[64][4];

// Hand-out counters: one 128-byte line per launch slot ([0] the counter,
// [1] the CTAs done).  Each launch takes the next line, so that launches on
// different streams do not share one, and the last CTA of a launch clears
// its line for the next launch on it.  (A captured graph keeps its line:
// replays of one graph run one after another.)
constexpr int kTicketSlots = 64;
__device__ int g_pair_tickets[kTicketSlots * 32];
int* g_ticket_base[64];
unsigned long long g_ticket_ctx[64];
unsigned g_ticket_seq[64];

moe_status next_ticket(int dev, unsigned long long ctx, int** out) {
    std::lock_guard<std::mutex> lock(g_pair_mutex);
    if (g_ticket_base[dev] == nullptr || g_ticket_ctx[dev] != ctx) {
        void* p = nullptr;
        MOE_CUDA_TRY(cudaGetSymbolAddress(&p, g_pair_tickets));
        g_ticket_base[dev] = static_cast<int*>(p);
        g_ticket_ctx[dev] = ctx;
    }
    *out = g_ticket_base[dev] + (g_ticket_seq[dev]++ % kTicketSlots) * 32;
    return MOE_OK;
}

template <bool GATED, bool F8>
moe_status launch_pair(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b, const CUtensorMap& bb,
                       const int32_t* offsets, int cap, int E, int K, int M, void* out, const float* sa0,
                       const float* sa1, const float* sb, cudaStream_t st, const DeviceInfo& di) {
    using C = PairCfg<GATED>;
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    unsigned long long ctx = 0;
    moe_status s = current_context_id(&ctx);
    if (s != MOE_OK) return s;
    auto kern = ffn_pair_kernel<GATED, F8>;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int pairs = 0;
    {
        constexpr int v = (GATED ? 1 : 0) + (F8 ? 2 : 0);
        std::lock_guard<std::mutex> lock(g_pair_mutex);
        PairCache& pc = g_pair_cache[dev][v];
        if (pc.ctx != ctx || pc.pairs <= 0) {
            MOE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes));
            cfg.gridDim = dim3(di.sm_count / 2 * 2);
            int n = 0;
            MOE_CUDA_TRY(cudaOccupancyMaxActiveClusters(&n, kern, &cfg));
            pc.ctx = ctx;
            pc.pairs = n < di.sm_count / 2 ? n : di.sm_count / 2;
        }
        pairs = pc.pairs;
    }
    if (pairs < 1) return MOE_ERR_UNSUPPORTED;
    int* ticket = nullptr;
    if ((s = next_ticket(dev, ctx, &ticket)) != MOE_OK) return s;
    cfg.gridDim = dim3(2 * pairs);
    MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, a0, a1, b, bb, offsets, cap, E, K, M, out, di.error_word, sa0, sa1,
                                    sb, ticket));
    return MOE_OK;
}

}  // namespace

// Chunks of at least this many routes (T * k) take the paired kernels.
bool use_pair_ffn(int cap) { return cap >= MOE_PAIR_MIN_ROUTES; }

moe_status launch_ffn_pair_prepared(const FfnTcLaunch& p, cudaStream_t st, const DeviceInfo& di) {
    if (p.gated)
        return launch_pair<true, false>(p.a0, p.a1, p.b, p.bb, p.offsets, p.cap, p.E, p.K, p.M, p.out, nullptr,
                                        nullptr, nullptr, st, di);
    return launch_pair<false, false>(p.a0, p.a1, p.b, p.bb, p.offsets, p.cap, p.E, p.K, p.M, p.out, nullptr, nullptr,
                                     nullptr, st, di);
}

moe_status launch_ffn_pair_w8a8(bool gated, const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                                const CUtensorMap& bb, const int32_t* offsets, int cap, int E, int K, int M, void* out,
                                const float* sa0, const float* sa1, const float* sb, cudaStream_t st,
                                const DeviceInfo& di) {
    if (gated) return launch_pair<true, true>(a0, a1, b, bb, offsets, cap, E, K, M, out, sa0, sa1, sb, st, di);
    return launch_pair<false, true>(a0, a1, b, bb, offsets, cap, E, K, M, out, sa0, sa1, sb, st, di);
}

}  // namespace moe
