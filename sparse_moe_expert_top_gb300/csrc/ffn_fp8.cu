// Grouped expert FFN with FP8 E4M3 expert weights on the sm_103a tensor
// cores, and the quantizer that produces those weights.
//
// The pages run their routed experts on low-bit weights: page "perf(ds4):
// batch heterogeneous MoE prefill by expert", "Fresh main-snapshot
// requalification" (a ROCmFP2 expert model), and page "perf(ggml): reuse
// ROCmFP4 weights across q=4 columns" (ROCmFP4/FPX expert weights streamed
// once per group of columns).  A prefill chunk of up to ~2k tokens gives each
// expert a few dozen rows, so the grouped FFN streams the touched experts'
// weights from HBM and the bytes per weight set its time.
//
// Format: OCP FP8 E4M3 codes (1 byte per weight) with one fp32 scale per
// output channel, w ~= scale[channel] * e4m3(code); the quantizer below makes
// them from bf16 or fp32 weights (scale = max|row| / 448, code = E4M3
// round-to-nearest-even of w / scale in fp32, saturating).
//
// GB300 design
// ------------
// The weights are widened inside the SM, between the TMA and the tensor
// core, to fp16: one cvt.rn.f16x2.e4m3x2 per pair of codes, exact (every
// E4M3 value is an fp16 value).  tcgen05.mma kind::f16 takes A and B in one
// type, so the token rows of this path are fp16 too (xs from the fp16
// scatter, h written as fp16 here).
//  - warp 0 (TMA): 64(K) x 128-row fp8 tiles of the two weight banks
//    (64-byte swizzle) into an 8-stage ring (released by the converters);
//  - the last warp (TMA): the item's fp16 token rows (128-byte swizzle) into
//    a 4-stage ring (released by the MMA);
//  - warps 6.. (converters, groups of 4): thread r owns weight row r of the
//    tile, which is tensor-memory lane r.  It reads its 64 codes of each
//    tile, widens them and writes the 32 f16x2 words to tensor memory with
//    tcgen05.st;
//  - warp 1 (MMA): tcgen05.mma with A (weights) read from tensor memory and
//    B (token rows) from shared memory, fp32 accumulators in tensor memory;
//  - warps 2-5 (epilogue): accumulator * scale[channel], then SwiGLU and an
//    fp16 h (gate/up) or an fp32 y (down).
// Keeping the widened weights in tensor memory spares shared memory the
// widened tile's write and the MMA's read of it.  At a few dozen rows per
// expert the MMA warp issues M=128, K=16 MMAs of small N, each worth ~50
// cycles of the tensor pipe, and a tcgen05.commit costs about two of them:
// so there is one commit per stage, shared by both rings the MMA consumes.
//
// Tensor memory (512 columns): accumulator region 0 (gate, or w_down tile 0)
// at columns 0..127, region 1 (up, or w_down tile 1) at 128..255, four
// widened A stages of 64 columns (two 32-column tiles of 64 fp16 K-values
// each) at 256..511.  Work items and their order are those of the bf16
// kernel with row slices of at most 128 rows.  Every wait is bounded (2 s);
// on a time-out the kernel records DEVERR_TIMEOUT, drains and returns.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_common.cuh"

namespace moe {
namespace {

// silu(g) = g / (1 + e^-g) with the fast exponential and division
// intrinsics (a few ulp of fp32; the result is rounded to a 16-bit h).  For
// g < -88 the exponential overflows to +inf and the quotient is -0.
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.f + __expf(-g)); }

// Compact rows per work item at most (MMA N): 64 leaves tensor memory for
// six widened stages, 128 for four.
#ifndef MOE_FP8_BN
#define MOE_FP8_BN 128
#endif
constexpr int BM = 128;          // weight rows per tile (MMA M)
constexpr int BN = MOE_FP8_BN;
constexpr int BK = 64;           // K per stage
constexpr int UMMA_K = 16;
constexpr int kBoxRows = 16;
constexpr int kBigBoxRows = 64;
// Converter warps: groups of 4 (one warp per tensor-memory lane quarter);
// group g widens both weight tiles of the stages j with j % groups == g.
#ifndef MOE_FP8_CONV_WARPS
#define MOE_FP8_CONV_WARPS 4
#endif
constexpr int kConvWarps = MOE_FP8_CONV_WARPS;
constexpr int kConvGroups = kConvWarps / 4;
static_assert(kConvWarps % 4 == 0 && kConvGroups >= 1, "converter warps");
constexpr int kRowWarp = 6 + kConvWarps;        // TMA of the token rows
// warp 0 TMA of the codes, 1 MMA, 2-5 epilogue, 6.. converters, then the row TMA warp
constexpr int kThreads = 32 * (kRowWarp + 1);
constexpr int kQStages = 8;      // ring of code tiles (TMA -> converters)
// Token-row stages (TMA -> MMA) and converted weight stages in tensor memory
// (converters -> MMA) advance together: stage j of both is freed by one
// tcgen05.commit (a commit costs the issuing thread about as much as two
// MMAs at these N, so there is one per stage, not one per ring).
constexpr int kAStages = (512 - 2 * BN) / 64;
constexpr int kBStages = kAStages;
static_assert(kBStages == kAStages, "one release barrier per stage of both rings");
constexpr int kQTileBytes = BM * BK;          // 8 KB of codes per weight tile
constexpr int kQStageBytes = 2 * kQTileBytes;
constexpr int kBBytes = BN * BK * 2;          // 16 KB of fp16 rows
constexpr int kRingBytes = kQStages * kQStageBytes + kBStages * kBBytes;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 2 * BN;
constexpr int kACols = 64;                   // per converted stage: 2 tiles x 32 columns
constexpr int kCtrlBytes = 3072;
constexpr int kOutStageBytes = 32 * BM * 2;  // gate/up: a 32-row x 128-feature fp16 tile of h
constexpr int kSmemBytes = kRingBytes + kCtrlBytes + kOutStageBytes + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
static_assert(kAccCols + kAStages * kACols == kTmemCols, "tensor memory map");
// A group publishes stage j after waiting for the MMA to free stage
// j + groups - kAStages: that must be an earlier stage than j.
static_assert(kConvGroups < kAStages, "converter groups must be fewer than the tensor-memory stages");

// Four codes (one 32-bit word; the low byte is the lowest K index) -> two
// f16x2 words.
__device__ __forceinline__ void convert4(uint32_t v, uint32_t& lo, uint32_t& hi) {
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"(static_cast<unsigned short>(v)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"(static_cast<unsigned short>(v >> 16)));
}

// Instruction descriptor of tcgen05.mma kind::f16 with fp16 A and B, fp32
// accumulator, both K-major.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// 4-bit weights (E2M1 codes, two per byte with the lower K index in the low
// nibble, and an E4M3 scale per 16 codes): one code pair -> one f16x2 word
// (cvt.rn.f16x2.e2m1x2), exact -- every E2M1 value times every E4M3 value
// is an fp16 value (at most 6 significant bits, magnitudes from 2^-10 to
// 2688).

// {value(b), value(b)} as f16x2 for the E4M3 code b.
__device__ __forceinline__ uint32_t f16x2_splat_e4m3(uint32_t b) {
    uint32_t d;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(static_cast<unsigned short>(b | (b << 8))));
    return d;
}

__device__ __forceinline__ uint32_t hmul2_rn(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// The eight codes of a 32-bit word (four code pairs, the lowest byte first)
// -> four f16x2 words: the word is split into its bytes by one mov.
__device__ __forceinline__ void f16x2_from_e2m1x8(uint32_t word, uint32_t (&d)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(word));
}

// Row r of a 4-bit weight tile: 32 bytes of codes (64 K-values) at r * 32,
// then, past the tile's CODE_BYTES, its four block scales as one word at
// r * 4 (block j in byte j).  -> 32 f16x2 words of code value * block scale.
template <int CODE_BYTES>
__device__ __forceinline__ void convert_row_fp4(const uint8_t* tile, int r, uint32_t (&w)[32]) {
    const uint4 v0 = *reinterpret_cast<const uint4*>(tile + r * 32);
    const uint4 v1 = *reinterpret_cast<const uint4*>(tile + r * 32 + 16);
    const uint32_t sw = *reinterpret_cast<const uint32_t*>(tile + CODE_BYTES + r * 4);
    const uint32_t words[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
        const uint32_t sc = f16x2_splat_e4m3((sw >> (8 * blk)) & 0xFFu);   // 16 codes = 2 words per block
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int q = 2 * blk + h;
            uint32_t d[4];
            f16x2_from_e2m1x8(words[q], d);
#pragma unroll
            for (int b = 0; b < 4; ++b) w[4 * q + b] = hmul2_rn(d[b], sc);
        }
    }
}

__device__ __forceinline__ void convert16(const uint4 v, uint32_t* w) {
    convert4(v.x, w[0], w[1]);
    convert4(v.y, w[2], w[3]);
    convert4(v.z, w[4], w[5]);
    convert4(v.w, w[6], w[7]);
}

// Row r of a 64-byte-swizzled tile of 64-byte rows: 16-byte chunk c sits at
// chunk c ^ ((r >> 1) & 3) (address bits 4-5 XOR bits 7-8).
__device__ __forceinline__ void convert_row(const uint8_t* tile, int r, uint32_t (&w)[32]) {
    const uint8_t* row = tile + r * BK;
    const int x = (r >> 1) & 3;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + ((c ^ x) << 4));
        convert16(v, w + 8 * c);
    }
}

// One lane waits (bounded) and the warp shares the outcome, so that the
// warp stays converged for the .sync.aligned tensor-memory instructions.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, unsigned* err) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, err) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// ---------------------------------------------------------------------------
// GATED: h (fp16 [cap][M]) = silu(s_g * (Q_g . xs)) * (s_u * (Q_u . xs)),
// M = f, K = d.  Otherwise y (fp32 [cap][M]) = s_d * (Q_d . h), M = d, K = f,
// two 128-feature tiles per item.
// ---------------------------------------------------------------------------
template <bool GATED, bool FP4 = false>
__global__ void __launch_bounds__(kThreads, 1)
    ffn_fp8_kernel(const __grid_constant__ CUtensorMap map_q0, const __grid_constant__ CUtensorMap map_q1,
                   const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_b_big,
                   const float* __restrict__ scale0, const float* __restrict__ scale1,
                   const int32_t* __restrict__ offsets, int cap, int E, int K, int M, void* __restrict__ out,
                   unsigned* err, const __grid_constant__ CUtensorMap map_s0,
                   const __grid_constant__ CUtensorMap map_s1) {
    // Bytes of one weight tile (128 rows x 64 K) in the code ring: FP8 codes,
    // or 4-bit codes followed by the tile's block scales (one word per row).
    constexpr int kQCode = FP4 ? BM * BK / 2 : kQTileBytes;
    constexpr int kQTile = FP4 ? kQCode + BM * 4 : kQTileBytes;
    constexpr int kQStage = 2 * kQTile;
    static_assert(kQStage <= kQStageBytes, "the code ring's stages hold either format");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* qring = smem;
    uint8_t* bring = smem + kQStages * kQStageBytes;
    uint8_t* ctrl = smem + kRingBytes;
    uint64_t* q_full = reinterpret_cast<uint64_t*>(ctrl);
    uint64_t* q_empty = q_full + kQStages;     // the 4 warps of one converter group
    uint64_t* b_full = q_empty + kQStages;
    uint64_t* a_full = b_full + kBStages;      // the 4 warps of one converter group
    uint64_t* done = a_full + kAStages;        // MMA commit: stage s of both rings is free
    uint64_t* acc_full = done + kAStages;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* drain = acc_empty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // last phase issued per stage of the two TMA rings (-1 = none)
    int* issued = reinterpret_cast<int*>(tmem_slot + 2);
    int* item_off = issued + kQStages + kBStages;         // E + 1 entries
    int* ntiles = item_off + kMaxExperts + 1;             // E entries
    volatile int* epi_flag = reinterpret_cast<volatile int*>(ntiles + kMaxExperts);  // 2 entries
    __half* out_stage = reinterpret_cast<__half*>(ctrl + kCtrlBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_kb = K / BK;
    const int n_mt = GATED ? M / BM : (M + 2 * BM - 1) / (2 * BM);

    // ---- prologue ---------------------------------------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], 4);
        }
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&a_full[s], 4);
            mbar_init(&done[s], 1);
        }
        for (int s = 0; s < kQStages + kBStages; ++s) issued[s] = -1;
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&map_q0);
        if (GATED) prefetch_tmap(&map_q1);
        if (FP4) {
            prefetch_tmap(&map_s0);
            if (GATED) prefetch_tmap(&map_s1);
        }
        prefetch_tmap(&map_b);
        prefetch_tmap(&map_b_big);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 2) {
        // validate the segments and count the 128-row slices of every expert
        bool bad = false;
        for (int e = lane; e < E; e += 32) {
            const int lo = offsets[e], hi = offsets[e + 1];
            bad |= lo < 0 || hi < lo || hi > cap;
        }
        bad = __any_sync(0xffffffffu, bad);
        for (int e = lane; e < E; e += 32) {
            const int n = offsets[e + 1] - offsets[e];
            ntiles[e] = bad || n <= 0 ? 0 : (n + BN - 1) / BN;
        }
        __syncwarp();
        const int per = (E + 31) / 32;
        int local = 0;
        for (int i = 0; i < per; ++i) {
            const int e = lane * per + i;
            if (e < E && !bad) local += ntiles[e] * n_mt;
        }
        int incl = local;
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        int run = incl - local;
        for (int i = 0; i < per; ++i) {
            const int e = lane * per + i;
            if (e < E) {
                item_off[e] = run;
                run += bad ? 0 : ntiles[e] * n_mt;
            }
        }
        if (lane == 31) item_off[E] = run;
        if (bad && lane == 0) atomicOr(err, DEVERR_OFFSETS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n_items = item_off[E];

    if (warp == 0) {
        // ---- TMA of the code tiles ------------------------------------------
        if (lane == 0) {
            const uint64_t pol_once = l2_policy(1);
            const uint64_t pol_shared = l2_policy(2);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                const Item item = decode_item(it, item_off, ntiles, offsets, E, BN);
                const int wy = item.e * M + item.mt * (GATED ? BM : 2 * BM);
                const int wy1 = GATED ? wy : wy + BM;
                const uint64_t pol_w = ntiles[item.e] > 1 ? pol_shared : pol_once;
                for (int kb = 0; kb < n_kb; ++kb) {
                    if (!mbar_wait(&q_empty[s], ph ^ 1u, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = qring + s * kQStage;
                    mbar_arrive_expect_tx(&q_full[s], kQStage);
                    issued[s] = static_cast<int>(ph);
                    if (FP4) {
                        // codes: 32 bytes of each of the 128 rows; block scales [E][K/64][M] words:
                        // the words of rows m .. m+127 of k-tile kb
                        const int m0 = item.mt * (GATED ? BM : 2 * BM), m1 = GATED ? m0 : m0 + BM;
                        const int sy = item.e * n_kb + kb;
                        tma_load_2d(st, &map_q0, &q_full[s], kb * (BK / 2), wy, pol_w);
                        tma_load_2d(st + kQCode, &map_s0, &q_full[s], m0, sy, pol_w);
                        tma_load_2d(st + kQTile, &map_q1, &q_full[s], kb * (BK / 2), wy1, pol_w);
                        tma_load_2d(st + kQTile + kQCode, &map_s1, &q_full[s], m1, sy, pol_w);
                    } else {
                        tma_load_2d(st, &map_q0, &q_full[s], kb * BK, wy, pol_w);
                        tma_load_2d(st + kQTileBytes, &map_q1, &q_full[s], kb * BK, wy1, pol_w);
                    }
                    if (++s == kQStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else if (warp == kRowWarp) {
        // ---- TMA of the token rows ------------------------------------------
        if (lane == 0) {
            const uint64_t pol_x = l2_policy(2);
            int j = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                const Item item = decode_item(it, item_off, ntiles, offsets, E, BN);
                const int n16 = (item.rows + kBoxRows - 1) / kBoxRows;
                for (int kb = 0; kb < n_kb; ++kb, ++j) {
                    const int s = j % kBStages;
                    const uint32_t ph = static_cast<uint32_t>(j / kBStages) & 1u;
                    if (!mbar_wait(&done[s], ph ^ 1u, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    uint8_t* bdst = bring + s * kBBytes;
                    mbar_arrive_expect_tx(&b_full[s], n16 * kBoxRows * BK * 2);
                    issued[kQStages + s] = static_cast<int>(ph);
                    int r = 0;
                    for (; r + kBigBoxRows <= n16 * kBoxRows; r += kBigBoxRows)
                        tma_load_2d(bdst + r * 128, &map_b_big, &b_full[s], kb * BK, item.row0 + r, pol_x);
                    for (; r < n16 * kBoxRows; r += kBoxRows)
                        tma_load_2d(bdst + r * 128, &map_b, &b_full[s], kb * BK, item.row0 + r, pol_x);
                }
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer ---------------------------------------------------
        if (lane == 0) {
            int j = 0;
            uint32_t use = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                const Item item = decode_item(it, item_off, ntiles, offsets, E, BN);
                const int n16 = (item.rows + kBoxRows - 1) / kBoxRows;
                const uint32_t idesc = idesc_f16(BM, n16 * kBoxRows);
                if (!mbar_wait(acc_empty, (use & 1u) ^ 1u, abort_flag, err)) break;
                tc_fence_after();
                for (int kb = 0; kb < n_kb; ++kb, ++j) {
                    const int s = j % kBStages;
                    const uint32_t ph = static_cast<uint32_t>(j / kBStages) & 1u;
                    if (!mbar_wait(&b_full[s], ph, abort_flag, err) || !mbar_wait(&a_full[s], ph, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b = sdesc_lo(smem_u32(bring + s * kBBytes));
                    const uint32_t a = tmem_base + static_cast<uint32_t>(kAccCols + s * kACols);
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
                        const uint64_t bd = sdesc_from_lo(b + 2 * kk);
                        umma_f16_tmem_a(tmem_base, a + kk * (UMMA_K / 2), bd, idesc, acc);
                        umma_f16_tmem_a(tmem_base + BN, a + 32 + kk * (UMMA_K / 2), bd, idesc, acc);
                    }
                    umma_commit(&done[s]);
                }
                if (!ok) break;
                umma_commit(acc_full);
                ++use;
            }
            umma_commit(drain);
            mbar_drain(drain, 0);
        }
    } else if (warp >= 6) {
        // ---- converters (warps 6..): thread r widens weight row r ------------
        // Stage j (counted over this CTA's items) uses ring slot j % kQStages
        // and tensor-memory stage j % kAStages.  A group publishes stage j
        // (a_full) only after it has read and widened its next stage, so the
        // tensor-memory stores of stage j complete behind that work.
        const int q = warp & 3;  // tensor-memory lanes [32q, 32q + 32)
        const int r = q * 32 + lane;
        const int g = (warp - 6) >> 2;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kAccCols;
        int pending = -1;
        auto publish = [&](int c) {
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[c]);
        };
        const int n_my_items = n_items > static_cast<int>(blockIdx.x)
                                   ? (n_items - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                                   : 0;
        const int n_stages = n_my_items * n_kb;
        bool ok = true;
        for (int j = g; j < n_stages; j += kConvGroups) {
            const int s = j % kQStages, cs = j % kAStages;
            const uint32_t ph = static_cast<uint32_t>(j / kQStages) & 1u;
            const uint32_t cph = static_cast<uint32_t>(j / kAStages) & 1u;
            // tensor-memory stage cs is free once the MMAs of stage j - kAStages completed
            if (!warp_wait(&q_full[s], ph, abort_flag, err) || !warp_wait(&done[cs], cph ^ 1u, abort_flag, err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint8_t* st = qring + s * kQStage;
            uint32_t w0[32], w1[32];
            if (FP4) {
                convert_row_fp4<kQCode>(st, r, w0);
                convert_row_fp4<kQCode>(st + kQTile, r, w1);
            } else {
                convert_row(st, r, w0);
                convert_row(st + kQTileBytes, r, w1);
            }
            // the codes are in registers: the ring slot may be refilled
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_empty[s]);
            if (pending >= 0) publish(pending);
            tmem_st32(lane_base + cs * kACols, w0);
            tmem_st32(lane_base + cs * kACols + 32, w1);
            pending = cs;
        }
        if (pending >= 0) {
            if (ok) publish(pending);
            else tmem_st_wait();
        }
    } else {
        // ---- epilogue (warps 2..5) ----------------------------------------
        const int q = warp & 3;
        const int et = threadIdx.x - 64;  // 0..127
        int local = 0;
        uint32_t use = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++local) {
            const Item item = decode_item(it, item_off, ntiles, offsets, E, BN);
            const int buf = local & 1;
            if (et == 0) epi_flag[buf] = mbar_wait(acc_full, use & 1u, abort_flag, err) ? 1 : 0;
            epilogue_sync();
            if (!epi_flag[buf]) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int m = item.mt * (GATED ? BM : 2 * BM) + q * 32 + lane;
            const size_t srow = static_cast<size_t>(item.e) * M;
            const bool has1 = GATED || m + BM < M;
            const float sc0 = __ldg(scale0 + srow + m);
            const float sc1 = GATED ? __ldg(scale1 + srow + m) : (has1 ? __ldg(scale0 + srow + m + BM) : 0.f);
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            bool range = false;
            for (int c0 = 0; c0 < item.rows; c0 += 32) {
                uint32_t g[32], g1[32];
                tmem_ld32(taddr + c0, g);
                tmem_ld32(taddr + BN + c0, g1);
                tmem_ld_wait();
                if (GATED) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float gv = __uint_as_float(g[j]) * sc0;
                        const float uv = __uint_as_float(g1[j]) * sc1;
                        const float hv = silu_fast(gv) * uv;
                        range |= !(fabsf(hv) <= 65504.f) && c0 + j < item.rows;
                        out_stage[j * BM + q * 32 + lane] = __float2half_rn(hv);
                    }
                    epilogue_sync();
                    __half* h = static_cast<__half*>(out);
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
                    epilogue_sync();
                } else {
                    float* y = static_cast<float*>(out);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int n = c0 + j;
                        if (n < item.rows) {
                            float* yr = y + static_cast<size_t>(item.row0 + n) * M;
                            yr[m] = __uint_as_float(g[j]) * sc0;
                            if (has1) yr[m + BM] = __uint_as_float(g1[j]) * sc1;
                        }
                    }
                }
            }
            if (GATED && __any_sync(0xffffffffu, range) && lane == 0) atomicOr(err, DEVERR_RANGE);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            ++use;
        }
        // zero-fill the unused compact rows R .. cap-1
        const int R = offsets[E];
        if (ok && R >= 0 && R <= cap) {
            const int vecs = M * (GATED ? 2 : 4) / 16;
            const int gw = blockIdx.x * 4 + (warp - 2), nw = gridDim.x * 4;
            uint4* o = static_cast<uint4*>(out);
            for (int row = R + gw; row < cap; row += nw)
                for (int v = lane; v < vecs; v += 32) o[static_cast<size_t>(row) * vecs + v] = make_uint4(0, 0, 0, 0);
        }
    }

    // ---- teardown ----------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        for (int s = 0; s < kQStages; ++s)
            if (issued[s] >= 0) mbar_drain(&q_full[s], static_cast<uint32_t>(issued[s]));
        for (int s = 0; s < kBStages; ++s)
            if (issued[kQStages + s] >= 0) mbar_drain(&b_full[s], static_cast<uint32_t>(issued[kQStages + s]));
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// Quantizer: one warp per weight row.  scale = max|w| / 448 (1 for an
// all-zero row), code = E4M3 RNE of w / scale (IEEE fp32 division),
// saturating at +-448.  Input bf16 or fp32, K a multiple of 16.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
    unsigned short v;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(v) : "f"(hi), "f"(lo));
    return v;
}

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&v)[8]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename T>
__global__ void __launch_bounds__(256) quantize_fp8_kernel(const T* __restrict__ w, long long rows, int K,
                                                           uint8_t* __restrict__ codes, float* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long row = gw; row < rows; row += nw) {
        const T* wr = w + row * K;
        float amax = 0.f;
        for (int k = lane * 8; k < K; k += 256) {
            float v[8];
            load8(wr + k, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
        }
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
        uint8_t* cr = codes + row * K;
        for (int k = lane * 8; k < K; k += 256) {
            float v[8];
            load8(wr + k, v);
            uint32_t p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                p[i] = e4m3x2_from_f32(__fdiv_rn(v[2 * i], s), __fdiv_rn(v[2 * i + 1], s));
            *reinterpret_cast<uint2*>(cr + k) = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
        }
        if (lane == 0) scales[row] = s;
    }
}

// The 4-bit quantizer, a warp per row (lane j takes the 16-value blocks j,
// j + 32, ...), in the fp32 arithmetic of its definition:
//   s = max|w| / 2688 (1 for an all-zero row);
//   b = E4M3 code (nearest even, saturating) of (block max / 6) / s;
//   q = E2M1 code (nearest even, saturating at 6) of w / (value(b) * s),
//       0 when value(b) is 0.
// Codes: two per byte, the lower K index in the low nibble.  Block scales:
// [E][K/64][M] words, block j of row m in byte j % 4 of word (e, j / 4, m).
__device__ __forceinline__ uint32_t e2m1x2_from_f32(float lo, float hi) {
    unsigned short v;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(v)
        : "f"(hi), "f"(lo));
    return v & 0xFFu;
}

template <typename T>
__global__ void __launch_bounds__(256) quantize_fp4_kernel(const T* __restrict__ w, long long rows, int M, int K,
                                                           uint8_t* __restrict__ codes, uint8_t* __restrict__ bscales,
                                                           float* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const int n_blk = K / 16;
    for (long long row = gw; row < rows; row += nw) {
        const T* wr = w + row * K;
        float amax = 0.f;
        for (int j = lane; j < n_blk; j += 32) {
            float v[8];
            load8(wr + 16 * j, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
            load8(wr + 16 * j + 8, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
        }
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float s = amax > 0.f ? __fdiv_rn(amax, 2688.f) : 1.f;
        const long long e = row / M, m = row - e * M;
        for (int j = lane; j < n_blk; j += 32) {
            float v[16];
            load8(wr + 16 * j, *reinterpret_cast<float(*)[8]>(v));
            load8(wr + 16 * j + 8, *reinterpret_cast<float(*)[8]>(v + 8));
            float bmax = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
            const uint32_t b = e4m3x2_from_f32(__fdiv_rn(__fdiv_rn(bmax, 6.f), s), 0.f) & 0xFFu;
            uint32_t half2;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(half2) : "h"(static_cast<unsigned short>(b)));
            const float vb = __half2float(__ushort_as_half(static_cast<unsigned short>(half2 & 0xFFFFu)));
            const float denom = __fmul_rn(vb, s);
            uint32_t p[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                p[i] = vb > 0.f ? e2m1x2_from_f32(__fdiv_rn(v[2 * i], denom), __fdiv_rn(v[2 * i + 1], denom)) : 0u;
            *reinterpret_cast<uint2*>(codes + row * (K / 2) + 8 * j) =
                make_uint2(p[0] | (p[1] << 8) | (p[2] << 16) | (p[3] << 24), p[4] | (p[5] << 8) | (p[6] << 16) |
                                                                                  (p[7] << 24));
            bscales[((e * (K / 64) + j / 4) * M + m) * 4 + (j & 3)] = static_cast<uint8_t>(b);
        }
        if (lane == 0) scales[row] = s;
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

std::mutex g_attr_mutex;
bool g_attr_set[64][4];

template <bool GATED, bool FP4 = false>
moe_status set_smem_attr() {
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    constexpr int v = (GATED ? 1 : 0) + (FP4 ? 2 : 0);
    if (!g_attr_set[dev][v]) {
        MOE_CUDA_TRY(cudaFuncSetAttribute(ffn_fp8_kernel<GATED, FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          kSmemBytes));
        g_attr_set[dev][v] = true;
    }
    return MOE_OK;
}

// fp8 code tiles: 64 codes (64 bytes) x 128 rows, 64-byte swizzle
moe_status encode_codes(CUtensorMap* map, const void* base, int K, long long rows) {
    return encode_2d_map(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, rows, BK, BM, CU_TENSOR_MAP_SWIZZLE_64B);
}

// fp16 token rows: 64 K-values (128 bytes) x box_rows rows, 128-byte swizzle
moe_status encode_rows(CUtensorMap* map, const void* base, int K, long long rows, int box_rows) {
    return encode_2d_map(map, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, K, rows, BK, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

moe_status launch_ffn_fp8_gate_up(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                  const uint8_t* q_gate, const float* s_gate, const uint8_t* q_up, const float* s_up,
                                  void* h, cudaStream_t st, const DeviceInfo& di) {
    CUtensorMap m0, m1, mb, mbb;
    moe_status s;
    if ((s = encode_codes(&m0, q_gate, d, static_cast<long long>(E) * f)) != MOE_OK) return s;
    if ((s = encode_codes(&m1, q_up, d, static_cast<long long>(E) * f)) != MOE_OK) return s;
    if ((s = encode_rows(&mb, xs, d, cap, kBoxRows)) != MOE_OK) return s;
    if ((s = encode_rows(&mbb, xs, d, cap, kBigBoxRows)) != MOE_OK) return s;
    if ((s = set_smem_attr<true>()) != MOE_OK) return s;
    ffn_fp8_kernel<true><<<di.sm_count, kThreads, kSmemBytes, st>>>(m0, m1, mb, mbb, s_gate, s_up, offsets, cap, E,
                                                                    d, f, h, di.error_word, m0, m1);
    return cuda_status(cudaGetLastError());
}

moe_status launch_ffn_fp8_down(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                               const uint8_t* q_down, const float* s_down, float* y, cudaStream_t st,
                               const DeviceInfo& di) {
    CUtensorMap m0, mb, mbb;
    moe_status s;
    if ((s = encode_codes(&m0, q_down, f, static_cast<long long>(E) * d)) != MOE_OK) return s;
    if ((s = encode_rows(&mb, h, f, cap, kBoxRows)) != MOE_OK) return s;
    if ((s = encode_rows(&mbb, h, f, cap, kBigBoxRows)) != MOE_OK) return s;
    if ((s = set_smem_attr<false>()) != MOE_OK) return s;
    ffn_fp8_kernel<false><<<di.sm_count, kThreads, kSmemBytes, st>>>(m0, m0, mb, mbb, s_down, s_down, offsets, cap,
                                                                     E, f, d, y, di.error_word, m0, m0);
    return cuda_status(cudaGetLastError());
}

// 4-bit code tiles: 32 bytes (64 K-values) x 128 rows, no swizzle
moe_status encode_codes_fp4(CUtensorMap* map, const void* base, int K, long long rows) {
    return encode_2d_map(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, rows, BK / 2, BM,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
}

// 4-bit block scales [E][K/64][M] 32-bit words (a row's four block scales of
// one 64-K tile in one word): 128 rows x one k-tile per box
moe_status encode_scales_fp4(CUtensorMap* map, const void* base, int M, int E, int K) {
    return encode_2d_map(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, M, static_cast<long long>(E) * (K / BK), BM, 1,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
}

moe_status launch_ffn_fp4_gate_up(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                  const uint8_t* q_gate, const uint8_t* b_gate, const float* s_gate,
                                  const uint8_t* q_up, const uint8_t* b_up, const float* s_up, void* h,
                                  cudaStream_t st, const DeviceInfo& di) {
    CUtensorMap m0, m1, mb, mbb, ms0, ms1;
    moe_status s;
    if ((s = encode_codes_fp4(&m0, q_gate, d, static_cast<long long>(E) * f)) != MOE_OK) return s;
    if ((s = encode_codes_fp4(&m1, q_up, d, static_cast<long long>(E) * f)) != MOE_OK) return s;
    if ((s = encode_scales_fp4(&ms0, b_gate, f, E, d)) != MOE_OK) return s;
    if ((s = encode_scales_fp4(&ms1, b_up, f, E, d)) != MOE_OK) return s;
    if ((s = encode_rows(&mb, xs, d, cap, kBoxRows)) != MOE_OK) return s;
    if ((s = encode_rows(&mbb, xs, d, cap, kBigBoxRows)) != MOE_OK) return s;
    if ((s = set_smem_attr<true, true>()) != MOE_OK) return s;
    ffn_fp8_kernel<true, true><<<di.sm_count, kThreads, kSmemBytes, st>>>(m0, m1, mb, mbb, s_gate, s_up, offsets, cap,
                                                                          E, d, f, h, di.error_word, ms0, ms1);
    return cuda_status(cudaGetLastError());
}

moe_status launch_ffn_fp4_down(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                               const uint8_t* q_down, const uint8_t* b_down, const float* s_down, float* y,
                               cudaStream_t st, const DeviceInfo& di) {
    CUtensorMap m0, mb, mbb, ms0;
    moe_status s;
    if ((s = encode_codes_fp4(&m0, q_down, f, static_cast<long long>(E) * d)) != MOE_OK) return s;
    if ((s = encode_scales_fp4(&ms0, b_down, d, E, f)) != MOE_OK) return s;
    if ((s = encode_rows(&mb, h, f, cap, kBoxRows)) != MOE_OK) return s;
    if ((s = encode_rows(&mbb, h, f, cap, kBigBoxRows)) != MOE_OK) return s;
    if ((s = set_smem_attr<false, true>()) != MOE_OK) return s;
    ffn_fp8_kernel<false, true><<<di.sm_count, kThreads, kSmemBytes, st>>>(m0, m0, mb, mbb, s_down, s_down, offsets,
                                                                           cap, E, f, d, y, di.error_word, ms0, ms0);
    return cuda_status(cudaGetLastError());
}

moe_status launch_quantize_fp4(const void* w, int dtype, int E, int M, int K, uint8_t* codes, uint8_t* block_scales,
                               float* scales, cudaStream_t st, const DeviceInfo& di) {
    const long long rows = static_cast<long long>(E) * M;
    const long long blocks_needed = (rows + 7) / 8;
    const int blocks = static_cast<int>(blocks_needed < di.sm_count * 16LL ? blocks_needed : di.sm_count * 16LL);
    if (dtype == MOE_BF16)
        quantize_fp4_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(w), rows, M, K,
                                                                    codes, block_scales, scales);
    else
        quantize_fp4_kernel<float><<<blocks, 256, 0, st>>>(static_cast<const float*>(w), rows, M, K, codes,
                                                            block_scales, scales);
    return cuda_status(cudaGetLastError());
}

// Rows of activations: block scales [K/64][ld][4] (the weights' layout with
// one expert of ld rows, of which the first `rows` are written).
moe_status launch_quantize_rows_fp4(const void* a, int dtype, int rows, int ld, int K, uint8_t* codes,
                                    uint8_t* block_scales, float* scales, cudaStream_t st, const DeviceInfo& di) {
    const long long blocks_needed = (rows + 7) / 8;
    const int blocks = static_cast<int>(blocks_needed < di.sm_count * 16LL ? blocks_needed : di.sm_count * 16LL);
    if (dtype == MOE_BF16)
        quantize_fp4_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(a), rows, ld, K,
                                                                    codes, block_scales, scales);
    else
        quantize_fp4_kernel<float><<<blocks, 256, 0, st>>>(static_cast<const float*>(a), rows, ld, K, codes,
                                                            block_scales, scales);
    return cuda_status(cudaGetLastError());
}

moe_status launch_quantize_fp8(const void* w, int dtype, long long rows, int K, uint8_t* codes, float* scales,
                               cudaStream_t st, const DeviceInfo& di) {
    const long long warps = rows;
    const long long blocks_needed = (warps + 7) / 8;
    const int blocks = static_cast<int>(blocks_needed < di.sm_count * 16LL ? blocks_needed : di.sm_count * 16LL);
    if (dtype == MOE_BF16)
        quantize_fp8_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(w), rows, K,
                                                                    codes, scales);
    else
        quantize_fp8_kernel<float><<<blocks, 256, 0, st>>>(static_cast<const float*>(w), rows, K, codes, scales);
    return cuda_status(cudaGetLastError());
}

}  // namespace moe
