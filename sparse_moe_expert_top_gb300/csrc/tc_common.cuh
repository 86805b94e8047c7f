// Building blocks of the tensor-core kernels: PTX wrappers for mbarriers,
// TMA, tcgen05 and tensor memory; the bounded waits; the work-item table of
// the grouped FFN; tensor-map encoding on the host.  Everything sits in an
// anonymous namespace, so each translation unit that includes this header
// gets its own copy.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per bounded wait

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase of `bar` with parity `parity` to complete.
// Returns false (after flagging the CTA and the device error word on a
// time-out) when the wait is abandoned.  The common case (the phase is
// already complete) costs one try_wait inline; the polling loop is out of line.
__device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag, unsigned* err,
                                            unsigned long long limit_ns) {
    const uint32_t addr = smem_u32(bar);
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(addr, parity)) return true;
        if ((i & 63u) == 0u) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicOr(err, DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, unsigned* err,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(smem_u32(bar), parity)) return true;
    return mbar_wait_slow(bar, parity, abort_flag, err, limit_ns);
}

// Bounded wait that ignores the abort flag: used while draining copies and
// MMAs that are already in flight.
__device__ __noinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
    const uint32_t addr = smem_u32(bar);
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(addr, parity) && global_ns() - t0 < kWaitLimitNs) {
    }
}

// L2 cache policy for TMA loads: 0 evict_normal, 1 evict_first, 2 evict_last.
__device__ __forceinline__ uint64_t l2_policy(int kind) {
    uint64_t p;
    if (kind == 1)
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    else if (kind == 2)
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    else
        asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// 16-byte asynchronous copy global -> shared (L1 bypassed) with an L2 policy;
// both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
                 : "memory");
}
// One arrival on `bar` once every cp.async this thread issued so far has
// landed (the arrival is part of the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Release/acquire fence at GPU scope.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// Orders shared-memory writes of the generic proxy that this thread has
// written or observed (cp.async included, once complete) before its later
// accesses through the async proxy (tcgen05.mma).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Drops a 128-byte line from L2 without writing it back (its contents become
// undefined); the address is 128-byte aligned.
__device__ __forceinline__ void l2_discard128(const void* p) {
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major, 128B-swizzled operand tile:
// rows of 128 bytes, 8-row core groups 1024 bytes apart (stride byte
// offset), descriptor version 1, swizzle mode 2 (128B).  The leading byte
// offset is unused for this layout.
// The descriptor is built from two 32-bit halves: the low half carries the
// start address (bits 0-13, in 16-byte units) and the leading byte offset
// (bit 16); the high half is the same for every tile.  Advancing a tile by
// 32 bytes of K adds 2 to the low half, so the MMA issue loop needs no
// 64-bit arithmetic.
constexpr uint32_t kSdescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr) { return ((saddr & 0x3FFFFu) >> 4) | (1u << 16); }
__device__ __forceinline__ uint64_t sdesc_from_lo(uint32_t lo) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(kSdescHi));
    return d;
}
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) { return sdesc_from_lo(sdesc_lo(saddr)); }

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, bf16 A
// and B, both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4: fp32 accumulator,
// A and B both E4M3 (format 0 in bits 7-9 and 10-12), both K-major, N >> 3 at
// bit 17, M >> 4 at bit 24.  One MMA consumes K = 32 one-byte elements, the
// same 32 bytes of a 128B-swizzled row as a kind::f16 MMA's K = 16.
__device__ __forceinline__ uint32_t idesc_e4m3(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Barrier 1 among the 128 epilogue threads (warps 2-5).
__device__ __forceinline__ void epilogue_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// tcgen05.mma kind::f16 with A read from tensor memory (lane = row of A,
// two 16-bit K-values per 32-bit column) and B from shared memory; the
// instruction descriptor is the one of the shared-memory form (A K-major).
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 consecutive 32-bit tensor-memory columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Work-item table
// ---------------------------------------------------------------------------

struct Item {
    int e, mt, row0, rows;
};

// item_off[e] = first item of expert e (exclusive scan), ntiles[e] = compact
// row slices of expert e.  Items of one expert are ordered mt-major, nt-minor.
__device__ __forceinline__ Item decode_item(int it, const int* item_off, const int* ntiles, const int32_t* offsets,
                                            int E, int slice) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (item_off[mid] <= it) lo = mid;
        else hi = mid - 1;
    }
    Item r;
    r.e = lo;
    const int local = it - item_off[lo];
    const int n = ntiles[lo];
    r.mt = local / n;
    const int nt = local - r.mt * n;
    const int seg_lo = __ldg(offsets + lo), seg_hi = __ldg(offsets + lo + 1);
    r.row0 = seg_lo + nt * slice;
    r.rows = min(slice, seg_hi - r.row0);
    return r;
}

// Item `it` of the table built in expert order: item_off[p] = first item of
// the p-th expert in that order, order[p] = that expert, ntiles[e] = its
// compact row slices.  Items of one expert are ordered mt-major, nt-minor.
__device__ __forceinline__ Item decode_item_ordered(int it, const int* item_off, const int* order, const int* ntiles,
                                                    const int32_t* offsets, int E, int slice) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (item_off[mid] <= it) lo = mid;
        else hi = mid - 1;
    }
    Item r;
    r.e = order[lo];
    const int local = it - item_off[lo];
    const int n = ntiles[r.e];
    r.mt = local / n;
    const int nt = local - r.mt * n;
    const int seg_lo = __ldg(offsets + r.e), seg_hi = __ldg(offsets + r.e + 1);
    r.row0 = seg_lo + nt * slice;
    r.rows = min(slice, seg_hi - r.row0);
    return r;
}

// ---------------------------------------------------------------------------
// Host side: tensor maps
// ---------------------------------------------------------------------------

std::mutex g_encode_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

moe_status get_encode(PFN_cuTensorMapEncodeTiled_v12000* fn) {
    std::lock_guard<std::mutex> lock(g_encode_mutex);
    if (g_encode == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        MOE_CUDA_TRY(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q));
        if (q != cudaDriverEntryPointSuccess || p == nullptr) return MOE_ERR_UNSUPPORTED;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    *fn = g_encode;
    return MOE_OK;
}

// 2-D tensor map over a row-major [rows][K] matrix of `elem_bytes`-byte
// elements with a box of box_k K-elements x box_rows rows.
moe_status encode_2d_map(CUtensorMap* map, const void* base, CUtensorMapDataType type, int elem_bytes, int K,
                         long long rows, int box_k, int box_rows, CUtensorMapSwizzle swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    moe_status st = get_encode(&enc);
    if (st != MOE_OK) return st;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(K) * static_cast<cuuint64_t>(elem_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_k), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, type, 2, const_cast<void*>(base), gdim, gstride, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

}  // namespace
}  // namespace moe
