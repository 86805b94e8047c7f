// Grouped expert FFN (A5 gate/up + SwiGLU, A6 down) with 4-bit operands on
// both sides: tcgen05.mma kind::mxf4nvf4 with block scaling.
//
// The weights are the 4-bit banks of moe_quantize_weights_fp4 (E2M1 codes,
// an E4M3 scale per 16 values, an fp32 scale per row); the compact rows of x
// and h carry the same format, made by moe_quantize_rows_fp4.  The tensor
// cores read the packed codes straight from shared memory and apply the
// per-16 block scales themselves (one MMA: K = 64, four block scales per row
// of each operand); the epilogue applies the two row scales.
//
// Block scales in tensor memory.  For an M = 128 MMA the hardware reads the
// scales of operand row r from lane r % 32 and column r / 32 of the scale
// address (four E4M3 scales, one per 16 K, in the 32-bit cell), and a lane
// quarter q of the accumulator reads them from its own quarter: the layout
// is 32 lanes wide and repeated in each of the four lane quarters.  Four
// scale warps (one per lane quarter) write it per stage from the scale words
// the TMA brought into shared memory (on a barrier of their own, loaded ahead
// of the codes), then signal the MMA thread; scale groups start at multiples
// of four columns.
//
// Per stage (256 K): two 16 KB code tiles of 128 weight rows, up to 64
// compact rows (8 KB), the weight rows' block-scale words (2 x 2 KB) and the
// compact rows' (1,088 bytes); four stages of 46 KB.  Work item: (expert, 128
// output features -- 256 for down, as two tiles -- and a slice of at most 64
// of the expert's compact rows; 128 in big-item mode, three stages of 55 KB).
// Tensor memory: accumulators of two item slots of 64 columns per weight tile
// (columns 0-255; an item of more than 64 rows takes both), block scales of
// the stages after them.
#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int NBM = 128;                                  // weight rows per tile (MMA M)
constexpr int kSliceN = 64;                               // compact rows per item at most (MMA N)
constexpr int kNStages = 4;
constexpr int kStageK = 256;                              // K per stage: one 128-byte row of packed codes
constexpr int kMmasPerStage = kStageK / 64;               // MMAs of K = 64 per weight tile and stage
constexpr int kCodeTile = NBM * 128;                      // 16 KB
constexpr int kRowsTile = kSliceN * 128;                  // 8 KB
constexpr int kSfaTile = kMmasPerStage * NBM * 4;         // 2 KB of block-scale words per weight tile
// The compact rows' scale words come in a box of 68 rows starting at the
// item's first row rounded down to a multiple of 4 (a tiled copy's innermost
// coordinate must be a multiple of 16 bytes).
constexpr int kSfbRows = kSliceN + 4;
constexpr int kSfbTile = kMmasPerStage * kSfbRows * 4;    // 1,088 bytes
constexpr int kOffA1 = kCodeTile;
constexpr int kOffB = 2 * kCodeTile;
constexpr int kOffSa0 = kOffB + kRowsTile;
constexpr int kOffSa1 = kOffSa0 + kSfaTile;
constexpr int kOffSb = kOffSa1 + kSfaTile;
constexpr int kNStageBytes = (kOffSb + kSfbTile + 1023) / 1024 * 1024;   // 46 KB
static_assert(kNStageBytes % 1024 == 0, "stages keep the code tiles 1024-byte aligned");
constexpr int kNRingBytes = kNStages * kNStageBytes;
// Big-item mode (chunks where most rows lie beyond the first 64 of their
// expert): slices of up to 128 rows (N <= 128, both accumulator slots), three
// stages of 55 KB (16 KB of rows, the row scales' box 132 rows).
constexpr int kSliceBig = 128;
constexpr int kNStagesBig = 3;
constexpr int kSfbRowsBig = kSliceBig + 4;
constexpr int kNStageBytesBig = (2 * kCodeTile + kSliceBig * 128 + 2 * kSfaTile + kMmasPerStage * kSfbRowsBig * 4 +
                                 1023) / 1024 * 1024;
static_assert(kNStagesBig * kNStageBytesBig <= kNRingBytes, "both carve-ups fit the ring");
#ifndef MOE_NVF4_BIG_MODE_PCT
#define MOE_NVF4_BIG_MODE_PCT 50
#endif
constexpr int kNCtrlBytes = 4096;
// The first kNList items of a CTA's hand-out sequence, decoded once at the
// start (an item's decode -- a search over the experts and two loads of the
// offsets -- takes microseconds under load, on every role's path between items).
constexpr int kNList = 512;
constexpr int kNListBytes = kNList * 16;
constexpr int kNOutStage = 32 * NBM * 2;                  // gate/up: a 32-row x 128-feature bf16 tile of h
constexpr int kNSmemBytes = kNRingBytes + kNCtrlBytes + kNListBytes + kNOutStage + 1024;
static_assert(kNSmemBytes <= 232448, "shared memory budget of one CTA");
constexpr int kNTmemCols = 512;
constexpr int kAccCols = 64;                              // one item slot of one weight tile
constexpr int kSfBase = 4 * kAccCols;                     // block scales after the accumulators
constexpr int kSfStageCols = 48;                          // per stage: 16 (tile 0) + 16 (tile 1) + 16 (rows)
static_assert(kSfBase + kNStages * kSfStageCols <= kNTmemCols, "tensor memory budget");
constexpr int kNEpiWarps = 4;
constexpr int kSfWarps = 4;
constexpr int kSfWarp0 = 2 + kNEpiWarps;
constexpr int kNThreads = 32 * (kSfWarp0 + kSfWarps);

__device__ __forceinline__ float silu_nvf4(float g) { return __fdividef(g, 1.f + __expf(-g)); }

// Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (format 1 in bits
// 7-9 and 10-12), both K-major, N >> 3 at bit 17, block scales E4M3 (bit 23
// clear), M >> 4 at bit 24, scale-data selectors 0.
__device__ __forceinline__ uint32_t idesc_nvf4(int M, int N) {
    return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.block16 [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// One lane waits (bounded) and the warp shares the outcome.
__device__ __forceinline__ bool warp_wait_nvf4(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                               unsigned* err) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, err) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// ---------------------------------------------------------------------------
// GATED: out = h (bf16 [cap][M]) = silu(A0 . xs) * (A1 . xs) with A0, A1 the
// gate and up banks, M = f, K = d.  Otherwise out = y (fp32 [cap][M]) = A0 . h,
// A0 = w_down, M = d, K = f.  Weight row scales sa0 (gate / down) and sa1
// (up), compact row scales sb.
// ---------------------------------------------------------------------------
// Item at hand-out position p.  The order is a sequence of blocks, one per
// heavy group b (heavy expert, feature tile; in expert, feature-tile order):
// the group's row slices, consecutive so that CTAs running them at the same
// time share its weight tiles in L2, then light items in proportion to the
// group's slices, so that the MMA-bound heavy items and the HBM-bound light
// ones keep one ratio along the whole order.  With H_b the heavy items before
// block b (H of them, L light ones), block b starts at B(b) = H_b + floor(H_b L / H).
// heavy[0] = H, heavy[1] = the number of heavy experts; items are numbered in
// `order` (heavy experts first) by item_off.
__device__ __noinline__ Item decode_interleaved(int p, const int* item_off, const int* order, const int* ntiles,
                                                const int* heavy, const int32_t* offsets, int E, int n_mt,
                                                int slice) {
    const int n_heavy_items = heavy[0];
    const int n_groups = heavy[1] * n_mt;
    int u = p;
    if (n_groups > 0) {
        const long long n_light = item_off[E] - n_heavy_items;
        auto head_of = [&](int b) {
            const int ei = b / n_mt, mt = b - ei * n_mt;
            return item_off[ei] + mt * ntiles[order[ei]];
        };
        auto block_start = [&](int b) {
            const int hb = head_of(b);
            return hb + static_cast<int>(static_cast<long long>(hb) * n_light / n_heavy_items);
        };
        int lo = 0, hi = n_groups - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (block_start(mid) <= p) lo = mid;
            else hi = mid - 1;
        }
        const int head = head_of(lo);
        const int size = ntiles[order[lo / n_mt]];
        const int b0 = block_start(lo);
        const int o = p - b0;
        u = o < size ? head + o : n_heavy_items + (b0 - head) + (o - size);
    }
    return decode_item_ordered(u, item_off, order, ntiles, offsets, E, slice);
}

template <bool GATED>
__global__ void __launch_bounds__(kNThreads, 1)
    ffn_nvf4_kernel(const __grid_constant__ CUtensorMap map_a0, const __grid_constant__ CUtensorMap map_a1,
                    const __grid_constant__ CUtensorMap map_sa0, const __grid_constant__ CUtensorMap map_sa1,
                    const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_b_big,
                    const __grid_constant__ CUtensorMap map_sb, const __grid_constant__ CUtensorMap map_sb_big,
                    const int32_t* __restrict__ offsets, int cap, int E, int K, int M, void* __restrict__ out,
                    unsigned* err, const float* __restrict__ sa0, const float* __restrict__ sa1,
                    const float* __restrict__ sb) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* ctrl = smem + kNRingBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
    uint64_t* sf_full = full + kNStages;
    uint64_t* empty = sf_full + kNStages;
    uint64_t* acc_full = empty + kNStages;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint64_t* sf_in = drain + 1;                     // a stage's block-scale words have landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_in + kNStages);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* issued = reinterpret_cast<int*>(tmem_slot + 2);
    int* item_off = issued + kNStages;               // E + 1 entries
    int* ntiles = item_off + kMaxExperts + 1;        // E entries
    volatile int* epi_flag = reinterpret_cast<volatile int*>(ntiles + kMaxExperts);  // 2 entries
    int* mode_big = const_cast<int*>(epi_flag + 2);   // launch-wide carve-up
    int* order = mode_big + 1;                        // experts: the heavy ones, then the light ones (E entries)
    int* heavy_items = order + kMaxExperts;           // items of the heavy experts
    int* heavy_experts = heavy_items + 1;             // how many experts are heavy
    Item* ilist = reinterpret_cast<Item*>(ctrl + kNCtrlBytes);   // this CTA's items, in hand-out order
    __nv_bfloat16* out_stage = reinterpret_cast<__nv_bfloat16*>(ctrl + kNCtrlBytes + kNListBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int fw = GATED ? NBM : 2 * NBM;            // output features per item
    const int n_mt = (M + fw - 1) / fw;
    const int n_st = (K + kStageK - 1) / kStageK;   // stages per item (a half-empty last one when K % 256 = 128)

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&sf_in[s], 1);
            mbar_init(&sf_full[s], kSfWarps);
            mbar_init(&empty[s], 1);
            issued[s] = -1;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kNEpiWarps);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&map_a0);
        prefetch_tmap(&map_a1);
        prefetch_tmap(&map_sa0);
        prefetch_tmap(&map_sa1);
        prefetch_tmap(&map_b);
        prefetch_tmap(&map_b_big);
        prefetch_tmap(&map_sb);
        prefetch_tmap(&map_sb_big);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kNTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 2) {
        // item table in expert order: row slices of 64 per expert, or of 128
        // when more than half of the rows lie beyond the first 64 of their expert
        bool bad = false;
        long long rows = 0, excess = 0;
        for (int e = lane; e < E; e += 32) {
            const int lo = offsets[e], hi = offsets[e + 1];
            bad |= lo < 0 || hi < lo || hi > cap;
            const int n = hi - lo;
            rows += n > 0 ? n : 0;
            excess += n > kSliceN ? n - kSliceN : 0;
        }
        bad = __any_sync(0xffffffffu, bad);
        for (int off = 16; off > 0; off >>= 1) {
            rows += __shfl_xor_sync(0xffffffffu, rows, off);
            excess += __shfl_xor_sync(0xffffffffu, excess, off);
        }
        // (the down projection keeps 64-row items: its fp32 stores of a 128-row item
        // would hold the tensor cores longer than the halved weight re-reads save)
        const bool big =
            GATED && rows > 0 && excess * 100 >= static_cast<long long>(MOE_NVF4_BIG_MODE_PCT) * rows;
        const int slice = big ? kSliceBig : kSliceN;
        if (lane == 0) *mode_big = big ? 1 : 0;
        // Experts with more than one row slice ("heavy": their weight tiles serve
        // several slices from L2, the MMAs set the pace) come first in `order`,
        // the others ("light": each weight tile streamed from HBM for one slice)
        // after them, each group in expert-id order; item_off is the exclusive
        // scan of the item counts in that order.  The items are then handed out
        // interleaved (item_at below).
        const int per = (E + 31) / 32;                 // lane j owns experts / positions [j*per, (j+1)*per)
        const int first = min(lane * per, E);
        int nheavy = 0;
        for (int i = 0; i < per; ++i) {
            const int e = lane * per + i;
            if (e < E) {
                const int n = bad ? 0 : offsets[e + 1] - offsets[e];
                ntiles[e] = (n + slice - 1) / slice;
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
        if (bad && lane == 0) atomicOr(err, DEVERR_OFFSETS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n_items = item_off[E];
    const bool big = *mode_big != 0;
    const int S = big ? kNStagesBig : kNStages;
    const int stage_bytes = big ? kNStageBytesBig : kNStageBytes;
    const int off_sa0 = kOffB + (big ? kSliceBig : kSliceN) * 128;   // after the rows
    const int off_sa1 = off_sa0 + kSfaTile;
    const int off_sb = off_sa1 + kSfaTile;
    const int sfb_rows = big ? kSfbRowsBig : kSfbRows;
    auto item_at = [&](int p) {
        return decode_interleaved(p, item_off, order, ntiles, heavy_items, offsets, E, n_mt, big ? kSliceBig : kSliceN);
    };
    // item j of this CTA is hand-out position blockIdx.x + j * gridDim.x
    const int n_list = static_cast<int>(blockIdx.x) < n_items
                           ? min((n_items - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                                     static_cast<int>(gridDim.x),
                                 kNList)
                           : 0;
    if (warp >= 2)
        for (int j = threadIdx.x - 64; j < n_list; j += kNThreads - 64) ilist[j] = item_at(blockIdx.x + j * gridDim.x);
    __syncthreads();
    auto my_item = [&](int j, int it) { return j < kNList ? ilist[j] : item_at(it); };

    if (warp == 0) {
        // ---- TMA producer --------------------------------------------------------
        if (lane == 0) {
            const uint64_t pol_once = l2_policy(1);
            const uint64_t pol_shared = l2_policy(2);
            const uint64_t pol_x = l2_policy(2);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int it = blockIdx.x, j = 0; ok && it < n_items; it += gridDim.x, ++j) {
                const Item item = my_item(j, it);
                const int n16 = (item.rows + 15) / 16;
                const uint32_t bytes = 2 * kCodeTile + n16 * 16 * 128;              // codes and rows
                const uint32_t sf_bytes = 2 * kSfaTile + kMmasPerStage * sfb_rows * 4;   // their block scales
                const int m0 = item.mt * fw;                  // first feature of tile 0
                const int m1 = GATED ? m0 : m0 + NBM;         // tile 1: the up rows, or the next 128 features
                const uint64_t pol_w = ntiles[item.e] > 1 ? pol_shared : pol_once;
                for (int js = 0; js < n_st; ++js) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + s * stage_bytes;
                    issued[s] = static_cast<int>(ph);
                    // the small block-scale loads first, on their own barrier, so that the scale
                    // warps have them in tensor memory by the time the codes land
                    mbar_arrive_expect_tx(&sf_in[s], sf_bytes);
                    tma_load_3d(st + off_sa0, &map_sa0, &sf_in[s], m0, js * kMmasPerStage, item.e, pol_w);
                    tma_load_3d(st + off_sa1, &map_sa1, &sf_in[s], m1, js * kMmasPerStage, item.e, pol_w);
                    tma_load_2d(st + off_sb, big ? &map_sb_big : &map_sb, &sf_in[s], item.row0 & ~3,
                                js * kMmasPerStage, pol_x);
                    // codes: x = byte offset in the row (two values per byte); scales: 3-D (word, 64-K tile, expert)
                    mbar_arrive_expect_tx(&full[s], bytes);
                    tma_load_2d(st, &map_a0, &full[s], js * 128, item.e * M + m0, pol_w);
                    tma_load_2d(st + kOffA1, &map_a1, &full[s], js * 128, item.e * M + m1, pol_w);
                    // the rows in as few boxes as possible: 64-row boxes, then 16-row ones
                    int r = 0;
                    for (; r + 64 <= n16 * 16; r += 64)
                        tma_load_2d(st + kOffB + r * 128, &map_b_big, &full[s], js * 128, item.row0 + r, pol_x);
                    for (; r < n16 * 16; r += 16)
                        tma_load_2d(st + kOffB + r * 128, &map_b, &full[s], js * 128, item.row0 + r, pol_x);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer ------------------------------------------------------------
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int slot = 0;
            uint32_t use0 = 0, use1 = 0;   // uses of each accumulator slot so far
            bool ok = true;
            for (int it = blockIdx.x, j = 0; ok && it < n_items; it += gridDim.x, ++j) {
                const Item item = my_item(j, it);
                const int N = (item.rows + 15) / 16 * 16;
                const uint32_t idesc = idesc_nvf4(NBM, N);
                // an item of more than 64 rows takes both slots (128 columns per weight tile)
                const bool both = item.rows > kSliceN;
                if (both) slot = 0;
                if (!mbar_wait(&acc_empty[slot], ((slot ? use1 : use0) & 1u) ^ 1u, abort_flag, err)) break;
                if (both && !mbar_wait(&acc_empty[1], (use1 & 1u) ^ 1u, abort_flag, err)) break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(slot * kAccCols);
                const uint32_t d1 = d0 + 2 * kAccCols;
                for (int js = 0; js < n_st; ++js) {
                    if (!mbar_wait(&full[s], ph, abort_flag, err) || !mbar_wait(&sf_full[s], ph, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sdesc_lo(smem_u32(smem + s * stage_bytes));
                    const uint32_t a1 = a0 + (kOffA1 >> 4);
                    const uint32_t b = a0 + (kOffB >> 4);
                    const uint32_t sf = tmem_base + static_cast<uint32_t>(kSfBase + s * kSfStageCols);
#pragma unroll
                    for (int c = 0; c < kMmasPerStage; ++c) {
                        // 32 bytes (64 values) of K per MMA; scale group c of each operand at 4 c
                        const uint32_t acc = (js | c) != 0 ? 1u : 0u;
                        const uint64_t bd = sdesc_from_lo(b + 2 * c);
                        umma_nvf4(d0, sdesc_from_lo(a0 + 2 * c), bd, idesc, sf + 4 * c, sf + 32 + 4 * c, acc);
                        umma_nvf4(d1, sdesc_from_lo(a1 + 2 * c), bd, idesc, sf + 16 + 4 * c, sf + 32 + 4 * c, acc);
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
                    slot = 0;
                } else {
                    slot ^= 1;
                }
            }
            umma_commit(drain);
            mbar_drain(drain, 0);
        }
    } else if (warp < kSfWarp0) {
        // ---- epilogue (warps 2-5) ----------------------------------------------
        const int q = warp & 3;
        const int et = threadIdx.x - 64;
        int local = 0;
        int slot = 0;
        uint32_t use0 = 0, use1 = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++local) {
            const Item item = my_item(local, it);
            const int buf = local & 1;
            const bool both = item.rows > kSliceN;
            if (both) slot = 0;
            if (et == 0) {
                bool got = mbar_wait(&acc_full[slot], (slot ? use1 : use0) & 1u, abort_flag, err);
                if (got && both) got = mbar_wait(&acc_full[1], use1 & 1u, abort_flag, err);
                epi_flag[buf] = got ? 1 : 0;
            }
            epi_sync();
            if (!epi_flag[buf]) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int m = item.mt * fw + q * 32 + lane;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(slot * kAccCols);
            // the slots go back to the MMA thread as soon as the warp's tensor-memory
            // reads of the item are done, before its last chunk's stores
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&acc_empty[slot]);
                    if (both) mbar_arrive(&acc_empty[1]);
                }
            };
            bool released = false;
            for (int c0 = 0; c0 < item.rows; c0 += 32) {
                uint32_t g[32], g1[32];
                tmem_ld32(taddr + c0, g);
                tmem_ld32(taddr + 2 * kAccCols + c0, g1);
                tmem_ld_wait();
                if (c0 + 32 >= item.rows) {   // the last chunk
                    release();
                    released = true;
                }
                float rs[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) rs[j] = c0 + j < item.rows ? __ldg(sb + item.row0 + c0 + j) : 0.f;
                if (GATED) {
                    const float wsg = __ldg(sa0 + static_cast<size_t>(item.e) * M + m);
                    const float wsu = __ldg(sa1 + static_cast<size_t>(item.e) * M + m);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float gv = __uint_as_float(g[j]) * wsg * rs[j];
                        const float uv = __uint_as_float(g1[j]) * wsu * rs[j];
                        out_stage[j * NBM + q * 32 + lane] = __float2bfloat16_rn(silu_nvf4(gv) * uv);
                    }
                    epi_sync();
                    __nv_bfloat16* h = static_cast<__nv_bfloat16*>(out);
                    const int chunk = et & 15;
#pragma unroll
                    for (int pass = 0; pass < 4; ++pass) {
                        const int j = pass * 8 + (et >> 4);
                        const int n = c0 + j;
                        if (n < item.rows) {
                            const uint4 v = *reinterpret_cast<const uint4*>(out_stage + j * NBM + chunk * 8);
                            *reinterpret_cast<uint4*>(h + static_cast<size_t>(item.row0 + n) * M + item.mt * NBM +
                                                      chunk * 8) = v;
                        }
                    }
                    epi_sync();
                } else {
                    const bool has1 = m + NBM < M;
                    const float ws0 = __ldg(sa0 + static_cast<size_t>(item.e) * M + m);
                    const float ws1 = has1 ? __ldg(sa0 + static_cast<size_t>(item.e) * M + m + NBM) : 0.f;
                    float* y = static_cast<float*>(out);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int n = c0 + j;
                        if (n < item.rows) {
                            float* yr = y + static_cast<size_t>(item.row0 + n) * M;
                            yr[m] = __uint_as_float(g[j]) * ws0 * rs[j];
                            if (has1) yr[m + NBM] = __uint_as_float(g1[j]) * ws1 * rs[j];
                        }
                    }
                }
            }
            if (!released) release();   // an item without rows
            if (slot) ++use1;
            else ++use0;
            if (both) {
                ++use1;
                slot = 0;
            } else {
                slot ^= 1;
            }
        }
        const int R = offsets[E];
        if (ok && R >= 0 && R <= cap) {
            const int vecs = M * (GATED ? 2 : 4) / 16;
            const int gw = blockIdx.x * kNEpiWarps + (warp - 2);
            const int nw = gridDim.x * kNEpiWarps;
            uint4* o = static_cast<uint4*>(out);
            for (int row = R + gw; row < cap; row += nw)
                for (int v = lane; v < vecs; v += 32) o[static_cast<size_t>(row) * vecs + v] = make_uint4(0, 0, 0, 0);
        }
    } else {
        // ---- block-scale warps: shared memory -> tensor memory, per stage --------
        // Warp w writes lane quarter w % 4; every quarter gets the same 32-lane
        // layout: column 4 c + j, lane i = the block-scale word of operand row
        // 32 j + i for MMA c of the stage.
        const int q = warp & 3;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int it = blockIdx.x, j = 0; ok && it < n_items; it += gridDim.x, ++j) {
            const int off = my_item(j, it).row0 & 3;   // the item's first row within the scale box
            for (int js = 0; js < n_st; ++js) {
                if (!warp_wait_nvf4(&sf_in[s], ph, abort_flag, err)) {
                    ok = false;
                    break;
                }
                const uint32_t* st = reinterpret_cast<const uint32_t*>(smem + s * stage_bytes);
                const uint32_t* sa_0 = st + off_sa0 / 4;   // [c][128] words
                const uint32_t* sa_1 = st + off_sa1 / 4;
                const uint32_t* sbw = st + off_sb / 4 + off;   // [c][sfb_rows] words
                uint32_t v[16];
                const uint32_t col = lane_base + static_cast<uint32_t>(kSfBase + s * kSfStageCols);
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[4 * c + j] = sa_0[c * NBM + 32 * j + lane];
                tmem_st16(col, v);
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[4 * c + j] = sa_1[c * NBM + 32 * j + lane];
                tmem_st16(col + 16, v);
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        v[4 * c + j] = (j < 2 || big) ? sbw[c * sfb_rows + 32 * j + lane] : 0u;
                tmem_st16(col + 32, v);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sf_full[s]);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    }

    // ---- teardown ----------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        for (int s = 0; s < S; ++s)
            if (issued[s] >= 0) {
                mbar_drain(&full[s], static_cast<uint32_t>(issued[s]));
                mbar_drain(&sf_in[s], static_cast<uint32_t>(issued[s]));
            }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kNTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

std::mutex g_nvf4_mutex;
bool g_nvf4_attr[64][2];

// Codes: a row-major [rows][K/2] byte matrix, boxes of 128 bytes x box_rows rows, 128-byte swizzle.
moe_status encode_codes_nvf4(CUtensorMap* map, const uint8_t* base, int K, long long rows, int box_rows) {
    return encode_2d_map(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, rows, 128, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}

// Weight block scales [E][K/64][M][4] as 32-bit words: dims (M, K/64, E), box (128, 4, 1).
moe_status encode_wscales_nvf4(CUtensorMap* map, const uint8_t* base, int E, int M, int K) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    moe_status st = get_encode(&enc);
    if (st != MOE_OK) return st;
    const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64),
                                static_cast<cuuint64_t>(E)};
    const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(M) * 4, static_cast<cuuint64_t>(K / 64) * M * 4};
    const cuuint32_t box[3] = {NBM, kMmasPerStage, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t*>(base), gdim, gstride, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

// Row block scales [K/64][ld][4] as 32-bit words: dims (ld, K/64), box (box_rows, 4).
moe_status encode_rscales_nvf4(CUtensorMap* map, const uint8_t* base, int ld, int K, int box_rows) {
    return encode_2d_map(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, ld, K / 64, box_rows, kMmasPerStage,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <bool GATED>
moe_status launch_nvf4(const uint8_t* a0, const uint8_t* sa0b, const float* sa0, const uint8_t* a1,
                       const uint8_t* sa1b, const float* sa1, const uint8_t* b, const uint8_t* sbb, int ld,
                       const float* sb, const int32_t* offsets, int cap, int E, int K, int M, void* out,
                       cudaStream_t st, const DeviceInfo& di) {
    CUtensorMap ma0, ma1, msa0, msa1, mb, mbb, msb, msbb;
    moe_status s;
    if ((s = encode_codes_nvf4(&ma0, a0, K, static_cast<long long>(E) * M, NBM)) != MOE_OK) return s;
    if ((s = encode_codes_nvf4(&ma1, a1, K, static_cast<long long>(E) * M, NBM)) != MOE_OK) return s;
    if ((s = encode_wscales_nvf4(&msa0, sa0b, E, M, K)) != MOE_OK) return s;
    if ((s = encode_wscales_nvf4(&msa1, sa1b, E, M, K)) != MOE_OK) return s;
    if ((s = encode_codes_nvf4(&mb, b, K, cap, 16)) != MOE_OK) return s;
    if ((s = encode_codes_nvf4(&mbb, b, K, cap, 64)) != MOE_OK) return s;
    if ((s = encode_rscales_nvf4(&msb, sbb, ld, K, kSfbRows)) != MOE_OK) return s;
    if ((s = encode_rscales_nvf4(&msbb, sbb, ld, K, kSfbRowsBig)) != MOE_OK) return s;
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lock(g_nvf4_mutex);
        if (!g_nvf4_attr[dev][GATED ? 1 : 0]) {
            MOE_CUDA_TRY(cudaFuncSetAttribute(ffn_nvf4_kernel<GATED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              kNSmemBytes));
            g_nvf4_attr[dev][GATED ? 1 : 0] = true;
        }
    }
    ffn_nvf4_kernel<GATED><<<di.sm_count, kNThreads, kNSmemBytes, st>>>(
        ma0, ma1, msa0, msa1, mb, mbb, msb, msbb, offsets, cap, E, K, M, out, di.error_word, sa0, sa1, sb);
    return cuda_status(cudaGetLastError());
}

}  // namespace

moe_status launch_ffn_w4a4_gate_up(const uint8_t* xs, const uint8_t* xs_bs, int ld, const float* xs_s,
                                   const int32_t* offsets, int cap, int E, int d, int f, const uint8_t* q_gate,
                                   const uint8_t* b_gate, const float* s_gate, const uint8_t* q_up,
                                   const uint8_t* b_up, const float* s_up, void* h, cudaStream_t st,
                                   const DeviceInfo& di) {
    return launch_nvf4<true>(q_gate, b_gate, s_gate, q_up, b_up, s_up, xs, xs_bs, ld, xs_s, offsets, cap, E, d, f, h,
                             st, di);
}

moe_status launch_ffn_w4a4_down(const uint8_t* hq, const uint8_t* h_bs, int ld, const float* h_s,
                                const int32_t* offsets, int cap, int E, int d, int f, const uint8_t* q_down,
                                const uint8_t* b_down, const float* s_down, float* y, cudaStream_t st,
                                const DeviceInfo& di) {
    return launch_nvf4<false>(q_down, b_down, s_down, q_down, b_down, s_down, hq, h_bs, ld, h_s, offsets, cap, E, f,
                              d, y, st, di);
}

}  // namespace moe
