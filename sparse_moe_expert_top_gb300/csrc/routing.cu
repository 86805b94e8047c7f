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
        key[j] = (e < E) ? topk_order_key(__ldg(row + e), e) : 0ull;
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
            sel_val = topk_key_value(best);
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
// A1, streaming form (E a multiple of 4, E <= 256): four lanes per token,
// eight tokens per warp.  Lane q of a token's quad holds float4 columns
// q, q+4, ..., q+60 of the logit row (a quad load covers 64 contiguous bytes).
//   1. Lower bound: every lane sorts the maxima of its float4 groups; two
//      shuffle rounds merge the quad's sorted lists (the top of two sorted
//      lists is the pairwise maximum of one with the other reversed), and
//      tau = the k-th largest group maximum.  k group maxima are distinct
//      logits >= tau, so every top-k logit is >= tau.
//   2. Candidates: the logits >= tau (typically k plus a few) are appended
//      to a per-token list in shared memory.
//   3. Selection: a candidate's rank is the number of candidates that beat
//      it under (logit descending, expert id ascending) -- a strict total
//      order with -0.0 == +0.0 in the float comparisons -- and the ranks
//      below k are the result, exactly.
// A token whose candidates overflow the list (many ties at tau) is solved by
// an exact insertion scan instead.  Few instructions per logit, no
// divergent insertions on the common path: large chunks stream.
// ---------------------------------------------------------------------------

__device__ __forceinline__ bool topk_beats(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

// Offers (x, e) to a sorted top-k list (v, id) whose last entry is thr: a
// strictly larger x shifts the smaller entries down and lands after every
// entry >= x.
template <int KMAX>
__device__ __forceinline__ void topk_offer(float (&v)[KMAX], int (&id)[KMAX], float& thr, int k, float x, int e) {
    if (!(x > thr)) return;
    bool placed = false;
#pragma unroll
    for (int i = KMAX - 1; i >= 0; --i) {
        if (i < k && !placed) {
            if (i > 0 && x > v[i - 1]) {
                v[i] = v[i - 1];
                id[i] = id[i - 1];
            } else {
                v[i] = x;
                id[i] = e;
                placed = true;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < KMAX; ++i)
        if (i == k - 1) thr = v[i];
}

// Sorts g[0..N) into descending order (bitonic network, branch-free).
template <int N>
__device__ __forceinline__ void sort_desc(float (&g)[N]) {
#pragma unroll
    for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    const float hi = fmaxf(g[i], g[j]), lo = fminf(g[i], g[j]);
                    const bool desc = (i & size) == 0;
                    g[i] = desc ? hi : lo;
                    g[j] = desc ? lo : hi;
                }
            }
        }
    }
}

// Sorts a bitonic sequence g[0..N) into descending order.
template <int N>
__device__ __forceinline__ void bitonic_merge_desc(float (&g)[N]) {
#pragma unroll
    for (int stride = N >> 1; stride > 0; stride >>= 1) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            if ((i & stride) == 0) {
                const float hi = fmaxf(g[i], g[i + stride]), lo = fminf(g[i], g[i + stride]);
                g[i] = hi;
                g[i + stride] = lo;
            }
        }
    }
}

constexpr int kTopkCand = 32;  // candidate slots per token

// Top-k of token t by the four lanes q = 0..3 of one quad (mask `quad`);
// cv/ce/sv: the token's candidate list and selected values in shared memory.
// Every synchronisation is among the quad's lanes.
template <int KMAX>
__device__ __forceinline__ void topk_quad_token(const float* __restrict__ logits, int t, int E, int k,
                                                int32_t* __restrict__ ids, float* __restrict__ w, float* cv,
                                                int* ce, float* sv, int q, unsigned quad) {
    constexpr int kNone = 0x7fffffff;
    const int nvec = E >> 2;

    // this lane's 16 float4 groups (experts 4c .. 4c+3 for c = q + 4i)
    float4 f[16];
    const float4* row = reinterpret_cast<const float4*>(logits + static_cast<size_t>(t) * E);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int c = q + 4 * i;
        f[i] = c < nvec ? __ldg(row + c) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }

    // 1. tau: the k-th largest group maximum of the quad
    float g[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) g[i] = fmaxf(fmaxf(f[i].x, f[i].y), fmaxf(f[i].z, f[i].w));
    sort_desc<16>(g);
    float top[KMAX];
#pragma unroll
    for (int i = 0; i < KMAX; ++i) top[i] = g[i];
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
        float other[KMAX];
#pragma unroll
        for (int i = 0; i < KMAX; ++i) other[i] = __shfl_xor_sync(quad, top[i], m);
#pragma unroll
        for (int i = 0; i < KMAX; ++i) top[i] = fmaxf(top[i], other[KMAX - 1 - i]);
        bitonic_merge_desc<KMAX>(top);
    }
    float tau = top[0];
#pragma unroll
    for (int i = 0; i < KMAX; ++i)
        if (i == k - 1) tau = top[i];

    // 2. candidates: logits >= tau, appended in (lane, group) order
    int mine = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        mine += (f[i].x >= tau) + (f[i].y >= tau) + (f[i].z >= tau) + (f[i].w >= tau);
    int incl = mine;
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        const int o = __shfl_up_sync(quad, incl, off, 4);
        if (q >= off) incl += o;
    }
    const int n_cand = __shfl_sync(quad, incl, 3, 4);
    if (n_cand <= kTopkCand) {
        int pos = incl - mine;
        auto append = [&](float x, int e) {
            if (x >= tau) {
                cv[pos] = x;
                ce[pos] = e;
                ++pos;
            }
        };
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int e0 = 4 * (q + 4 * i);
            append(f[i].x, e0);
            append(f[i].y, e0 + 1);
            append(f[i].z, e0 + 2);
            append(f[i].w, e0 + 3);
        }
        __syncwarp(quad);
        // 3. exact ranks among the candidates
        for (int j = q; j < n_cand; j += 4) {
            const float vj = cv[j];
            const int ej = ce[j];
            int rank = 0;
            for (int i = 0; i < n_cand; ++i) rank += topk_beats(cv[i], ce[i], vj, ej) ? 1 : 0;
            if (rank < k) {
                ids[static_cast<size_t>(t) * k + rank] = ej;
                sv[rank] = vj;
            }
        }
    } else {
        // many ties at tau: exact insertion scan of all logits, then a merge
        float v[KMAX];
        int id[KMAX];
#pragma unroll
        for (int i = 0; i < KMAX; ++i) {
            v[i] = -INFINITY;
            id[i] = kNone;
        }
        float thr = -INFINITY;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int e0 = 4 * (q + 4 * i);
            topk_offer<KMAX>(v, id, thr, k, f[i].x, e0);
            topk_offer<KMAX>(v, id, thr, k, f[i].y, e0 + 1);
            topk_offer<KMAX>(v, id, thr, k, f[i].z, e0 + 2);
            topk_offer<KMAX>(v, id, thr, k, f[i].w, e0 + 3);
        }
#pragma unroll
        for (int m = 1; m <= 2; m <<= 1) {
            float pv[KMAX];
            int pid[KMAX];
#pragma unroll
            for (int i = 0; i < KMAX; ++i) {
                pv[i] = __shfl_xor_sync(quad, v[i], m);
                pid[i] = __shfl_xor_sync(quad, id[i], m);
            }
            float nv[KMAX];
            int nid[KMAX];
#pragma unroll
            for (int r = 0; r < KMAX; ++r) {
                nv[r] = -INFINITY;
                nid[r] = kNone;
                if (r < k) {
                    const bool take_a = topk_beats(v[0], id[0], pv[0], pid[0]);
                    nv[r] = take_a ? v[0] : pv[0];
                    nid[r] = take_a ? id[0] : pid[0];
#pragma unroll
                    for (int i = 0; i < KMAX - 1; ++i) {
                        v[i] = take_a ? v[i + 1] : v[i];
                        id[i] = take_a ? id[i + 1] : id[i];
                        pv[i] = take_a ? pv[i] : pv[i + 1];
                        pid[i] = take_a ? pid[i] : pid[i + 1];
                    }
                    if (take_a) {
                        v[KMAX - 1] = -INFINITY;
                        id[KMAX - 1] = kNone;
                    } else {
                        pv[KMAX - 1] = -INFINITY;
                        pid[KMAX - 1] = kNone;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < KMAX; ++i) {
                v[i] = nv[i];
                id[i] = nid[i];
            }
        }
        if (q == 0) {
#pragma unroll
            for (int r = 0; r < KMAX; ++r)
                if (r < k) {
                    ids[static_cast<size_t>(t) * k + r] = id[r];
                    sv[r] = v[r];
                }
        }
    }
    __syncwarp(quad);
    if (q == 0) {
        // softmax over the k selected logits, summed in slot order
        float sum = 0.f;
        for (int r = 0; r < k; ++r) sum += expf(sv[r] - sv[0]);
        const float inv = 1.f / sum;
        float* w_t = w + static_cast<size_t>(t) * k;
        for (int r = 0; r < k; ++r) w_t[r] = expf(sv[r] - sv[0]) * inv;
    }
}

template <int KMAX>
__global__ void __launch_bounds__(128, 1) route_topk_quad_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                              int32_t* __restrict__ ids, float* __restrict__ w) {
    __shared__ float cand_v[4][8][kTopkCand];
    __shared__ int cand_e[4][8][kTopkCand];
    __shared__ float sel_v[4][8][KMAX];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = lane & 3, tw = lane >> 2;
    const unsigned quad = 0xfu << (lane & ~3);
    const int t = blockIdx.x * 32 + warp * 8 + tw;
    // every synchronisation is among the four lanes of one token, so the
    // quads of padding tokens past T leave at once (their -inf logits would
    // all tie at tau and take the slow exact path)
    if (t >= T) return;
    topk_quad_token<KMAX>(logits, t, E, k, ids, w, cand_v[warp][tw], cand_e[warp][tw], sel_v[warp][tw], q, quad);
}

// ---------------------------------------------------------------------------
// A2 (with TOPK and PREFIX: A1-A3 in one launch): route histogram with
// stable ranks inside token-aligned chunks.
//
// Chunk c holds the routes of tokens [c*ct, (c+1)*ct), ct = ws_chunk_tokens(T)
// (a multiple of 32), and CTA c (32 warps) owns it.  The CTA walks its tokens
// 32 at a time: warp w takes token w of the pass -- with TOPK it routes it
// first (k rounds of a warp arg-max over order keys, the softmax summed in
// slot order, as the small-chunk kernel does), else it reads the token's ids --
// and leaves the experts of its unmasked routes in shared memory.  Warp 0
// then ranks the pass's routes in route order, 32 at a time:
// __match_any_sync groups the lanes that hit one expert, and a route's rank
// inside the chunk is its expert's running count plus the number of lower
// lanes of its group.  After the last pass the running counts are the
// chunk's per-expert counts.  The last CTA to finish (completion counter in
// the workspace header) sums the chunk counts into counts[], four threads
// per expert each over a quarter of the chunks; with PREFIX it also writes
// the exclusive prefix offsets[] and every chunk's row bases (base[c][e] =
// offsets[e] + the counts of expert e in the chunks before c), as
// prefix_offsets_kernel does.  The counter is left at zero for the next call.
// A warp per token keeps the latency of a pass short: at prefill chunk
// sizes every token of the chunk is in flight at once.
// ---------------------------------------------------------------------------

constexpr int kChunkThreads = 1024;
constexpr int kChunkWarps = kChunkThreads / 32;   // tokens per pass
static_assert(kChunkThreads == 4 * kMaxExperts, "the tail takes four threads per expert");

template <bool TOPK, bool PREFIX>
__global__ void __launch_bounds__(kChunkThreads) route_chunks_kernel(const float* __restrict__ logits,
                                                                     const uint8_t* __restrict__ mask, int T, int E,
                                                                     int k, int chunk_tokens, int32_t* ids,
                                                                     float* __restrict__ w, int32_t* __restrict__ ws,
                                                                     int32_t* __restrict__ counts,
                                                                     int32_t* __restrict__ offsets, unsigned* err) {
    __shared__ int s_e[kChunkWarps * kMaxK];   // expert of each route of the pass (-1: masked)
    __shared__ int s_cnt[kMaxExperts];         // running per-expert counts of the chunk; later the offsets
    __shared__ int psum[4][kMaxExperts];       // the tail's partial sums over quarters of the chunks
    __shared__ int warp_sum[8];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, n_chunks = gridDim.x;
    int32_t* chunk_counts = ws + kWsHeaderWords;
    int32_t* lrank = chunk_counts + static_cast<size_t>(n_chunks) * kMaxExperts;
    const int t_begin = c * chunk_tokens, t_end = min(T, t_begin + chunk_tokens);

    if (tid < kMaxExperts) s_cnt[tid] = 0;
    bool bad = false;
    for (int p0 = t_begin; p0 < t_end; p0 += kChunkWarps) {
        const int t = p0 + warp;
        const int nt = min(kChunkWarps, t_end - p0);
        if (t < t_end) {
            int e = -1;   // lane s < k: the expert of slot s
            if (TOPK) {
                const float* row = logits + static_cast<size_t>(t) * E;
                unsigned long long key[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int ee = lane + 32 * jj;
                    key[jj] = (ee < E) ? topk_order_key(__ldg(row + ee), ee) : 0ull;
                }
                float sel_val = 0.f;
                int sel_id = 0;
                for (int sl = 0; sl < k; ++sl) {
                    unsigned long long best = key[0];
#pragma unroll
                    for (int jj = 1; jj < 8; ++jj) best = key[jj] > best ? key[jj] : best;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        const unsigned long long o = __shfl_xor_sync(kFull, best, off);
                        best = o > best ? o : best;
                    }
                    const int eb = 0xFFFF - static_cast<int>(best & 0xFFFFu);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        if (lane + 32 * jj == eb) key[jj] = 0ull;
                    if (lane == sl) {
                        sel_val = topk_key_value(best);
                        sel_id = eb;
                    }
                }
                // softmax over the k selected logits, summed in slot order
                const float top = __shfl_sync(kFull, sel_val, 0);
                float sum = 0.f;
                for (int r = 0; r < k; ++r) sum += expf(__shfl_sync(kFull, sel_val, r) - top);
                const float inv = 1.f / sum;
                if (lane < k) {
                    ids[static_cast<size_t>(t) * k + lane] = sel_id;
                    w[static_cast<size_t>(t) * k + lane] = expf(sel_val - top) * inv;
                    e = sel_id;
                }
            } else if (lane < k) {
                e = ids[static_cast<size_t>(t) * k + lane];
                if (e < 0 || e >= E) {
                    bad = true;
                    e = -1;
                }
            }
            if (lane < k) {
                if (e >= 0 && mask != nullptr && mask[static_cast<size_t>(t) * k + lane] != 0) e = -1;
                s_e[warp * k + lane] = e;
            }
        }
        __syncthreads();
        if (warp == 0) {
            // the pass's routes in route order: local route j is slot j % k of token p0 + j / k
            const unsigned lt_mask = (1u << lane) - 1u;
            const int n_r = nt * k;
            const size_t r0 = static_cast<size_t>(p0) * k;
            for (int j0 = 0; j0 < n_r; j0 += 32) {
                const int j = j0 + lane;
                const int e = j < n_r ? s_e[j] : -1;
                const unsigned peers = __match_any_sync(kFull, e);
                const int rank = e >= 0 ? s_cnt[e] + __popc(peers & lt_mask) : -1;
                __syncwarp();
                if (e >= 0 && lane == __ffs(peers) - 1) s_cnt[e] += __popc(peers);
                __syncwarp();
                if (j < n_r) lrank[r0 + j] = rank;
            }
        }
        __syncthreads();
    }
    if (bad) atomicOr(err, DEVERR_OFFSETS);
    if (tid < kMaxExperts) chunk_counts[static_cast<size_t>(c) * kMaxExperts + tid] = s_cnt[tid];

    // the last CTA reduces the chunk counts (and, with PREFIX, scans them)
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(reinterpret_cast<unsigned*>(ws), 1u) == static_cast<unsigned>(n_chunks - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int e = tid & (kMaxExperts - 1), part = tid / kMaxExperts;
    const int per = (n_chunks + 3) / 4;
    const int c_lo = min(n_chunks, part * per), c_hi = min(n_chunks, c_lo + per);
    int part_sum = 0;
    if (e < E)
        for (int cc = c_lo; cc < c_hi; ++cc) part_sum += __ldcg(chunk_counts + static_cast<size_t>(cc) * kMaxExperts + e);
    psum[part][e] = part_sum;
    __syncthreads();
    const int total = psum[0][e] + psum[1][e] + psum[2][e] + psum[3][e];
    if (part == 0 && e < E) counts[e] = total;
    if (PREFIX) {
        // exclusive scan of the totals over the experts, by the 256 threads of part 0
        int incl = total;
        if (part == 0) {
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(kFull, incl, off);
                if (lane >= off) incl += o;
            }
            if (lane == 31) warp_sum[warp] = incl;
        }
        __syncthreads();
        if (part == 0) {
            int before = 0;
            for (int ww = 0; ww < warp; ++ww) before += warp_sum[ww];
            const int excl = before + incl - total;
            s_cnt[e] = excl;
            if (e < E) offsets[e] = excl;
            if (e == E - 1) offsets[E] = excl + total;
        }
        __syncthreads();
        int32_t* bases = lrank + static_cast<size_t>(T) * k;
        if (e < E) {
            int run = s_cnt[e];
            for (int pp = 0; pp < part; ++pp) run += psum[pp][e];
            for (int cc = c_lo; cc < c_hi; ++cc) {
                bases[static_cast<size_t>(cc) * kMaxExperts + e] = run;
                run += __ldcg(chunk_counts + static_cast<size_t>(cc) * kMaxExperts + e);
            }
        }
    }
    if (tid == 0) atomicExch(reinterpret_cast<unsigned*>(ws), 0u);
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

// bf16x2 -> f16x2 (exact for |v| <= 65504 down to 2^-17; smaller values
// round to fp16 subnormals).  Sets `range` when a value is beyond 65504.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v, bool& range) {
    const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xFFFF0000u);
    range |= !(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f);
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <bool TO_F16>
__global__ void __launch_bounds__(128) scatter_rows_kernel(const uint4* __restrict__ x,
                                                           const int32_t* __restrict__ ids,
                                                           const int32_t* __restrict__ offsets, int T, int k,
                                                           int E, int row_vecs, const int32_t* __restrict__ lrank,
                                                           const int32_t* __restrict__ bases,
                                                           uint4* __restrict__ xs,
                                                           int32_t* __restrict__ row_of_route,
                                                           int32_t* __restrict__ route_of_row, unsigned* err,
                                                           int32_t* __restrict__ tile_counts, int n_counts,
                                                           float4* __restrict__ out, int d4, int chunk_tokens,
                                                           const float* __restrict__ scale_in = nullptr,
                                                           float* __restrict__ scale_out = nullptr,
                                                           const uint32_t* __restrict__ sf_in = nullptr,
                                                           int ld_in = 0, uint32_t* __restrict__ sf_out = nullptr,
                                                           int ld_out = 0, int n_sf = 0) {
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
            if (e >= 0 && e < E) row = bases[static_cast<size_t>(t / chunk_tokens) * kMaxExperts + e] + lr;
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
        if (scale_out != nullptr) {
            // rows carrying E4M3 codes: each compact row gets its token row's scale
            if (row >= 0) scale_out[row] = __ldg(scale_in + t);
            if (tail >= 0) scale_out[tail] = 0.f;
        }
    }
    __syncthreads();
    if (tile_counts != nullptr) {
        // the fused combine's preparation, as in scatter_index_kernel
        bool any = false;
        for (int s = 0; s < k; ++s) any |= rows[s] >= 0;
        for (int j = tid; j < n_counts; j += blockDim.x) tile_counts[static_cast<size_t>(t) * n_counts + j] = 0;
        if (!any)
            for (int v = tid; v < d4; v += blockDim.x) out[static_cast<size_t>(t) * d4 + v] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const uint4* src = x + static_cast<size_t>(t) * row_vecs;
    bool range = false;
    for (int v = tid; v < row_vecs; v += blockDim.x) {
        uint4 val = __ldg(src + v);
        if (TO_F16) {
            val.x = bf16x2_to_f16x2(val.x, range);
            val.y = bf16x2_to_f16x2(val.y, range);
            val.z = bf16x2_to_f16x2(val.z, range);
            val.w = bf16x2_to_f16x2(val.w, range);
        }
        for (int s = 0; s < k; ++s) {
            const int row = rows[s];
            if (row >= 0) xs[static_cast<size_t>(row) * row_vecs + v] = val;
            const int tail = tails[s];
            if (tail >= 0) xs[static_cast<size_t>(tail) * row_vecs + v] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if (sf_out != nullptr) {
        // 4-bit rows: the token's block-scale words [tile][ld] go to its compact rows' columns
        for (int j = tid; j < n_sf; j += blockDim.x) {
            const uint32_t v = __ldg(sf_in + static_cast<size_t>(j) * ld_in + t);
            for (int s = 0; s < k; ++s) {
                const int row = rows[s];
                if (row >= 0) sf_out[static_cast<size_t>(j) * ld_out + row] = v;
                const int tail = tails[s];
                if (tail >= 0) sf_out[static_cast<size_t>(j) * ld_out + tail] = 0u;
            }
        }
    }
    if (TO_F16 && __syncthreads_or(range) && tid == 0) atomicOr(err, DEVERR_RANGE);
}

// ---------------------------------------------------------------------------
// E4M3 activation rows (the FP8-activation path).  The arithmetic is the
// weights' quantizer's: scale = max|row| / 448 (IEEE fp32 division; 1 for an
// all-zero row), code = E4M3 of the IEEE fp32 quotient v / scale, rounded to
// nearest even and saturating -- so that the codes are the weight
// quantizer's bit for bit.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t e4m3x2_rn(float lo, float hi) {
    unsigned short v;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(v) : "f"(hi), "f"(lo));
    return v;
}

// The 8 bf16 values of `u` as 8 E4M3 codes of v / s.
__device__ __forceinline__ uint2 e4m3x8_of_bf16x8(uint4 u, float s) {
    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        p[i] = e4m3x2_rn(__fdiv_rn(__uint_as_float(wv[i] << 16), s), __fdiv_rn(__uint_as_float(wv[i] & 0xFFFF0000u), s));
    return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

__device__ __forceinline__ float amax_bf16x8(uint4 u) {
    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(wv[i] << 16)), fabsf(__uint_as_float(wv[i] & 0xFFFF0000u))));
    return m;
}

// Largest `v` of the CTA, returned to every thread (red: one float per warp).
__device__ __forceinline__ float block_max(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, off));
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float m = 0.f;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    return m;
}

constexpr int kQuantWarps = 8;   // rows per CTA of the row quantizer
constexpr int kQuantVec = 8;     // uint4 (8 bf16) per lane: rows of up to 2048 values in registers

// Rows of a bf16 matrix [cap][K] to E4M3 codes and one scale per row, a warp
// per row holding its row in registers (read once, reduced with shuffles).
// Rows at or beyond R = offsets[E] are the zero-filled unused compact rows:
// their codes are 0 and their scale 1 (an all-zero row), without reading them.
__global__ void __launch_bounds__(32 * kQuantWarps) quantize_rows_e4m3_kernel(const uint4* __restrict__ a, int K8,
                                                                            int cap, const int32_t* __restrict__ offsets,
                                                                            int E, uint2* __restrict__ codes,
                                                                            float* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
    if (row >= cap) return;
    uint2* crow = codes + static_cast<size_t>(row) * K8;
    if (row >= __ldg(offsets + E)) {
        for (int v = lane; v < K8; v += 32) crow[v] = make_uint2(0u, 0u);
        if (lane == 0) scales[row] = 1.f;
        return;
    }
    uint4 u[kQuantVec];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < kQuantVec; ++j) {
        const int v = lane + 32 * j;
        if (v < K8) {
            u[j] = __ldg(a + static_cast<size_t>(row) * K8 + v);
            amax = fmaxf(amax, amax_bf16x8(u[j]));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
#pragma unroll
    for (int j = 0; j < kQuantVec; ++j) {
        const int v = lane + 32 * j;
        if (v < K8) crow[v] = e4m3x8_of_bf16x8(u[j], s);
    }
    if (lane == 0) scales[row] = s;
}

// A4 of the FP8-activation path straight from the bf16 token rows, a CTA per
// token: the row is read once, quantized (codes x_q and scale x_scales of the
// token) and its codes written to the token's compact rows with their scale;
// k of the unused tail rows R .. T*k-1 get zero codes and scale 0.  The
// compact rows come from the workspace exactly as in scatter_rows_kernel.
template <int VPT>
__global__ void __launch_bounds__(128) scatter_quant_e4m3_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ ids, const int32_t* __restrict__ offsets, int T, int k,
    int E, int d8, const int32_t* __restrict__ lrank, const int32_t* __restrict__ bases, int chunk_tokens,
    uint2* __restrict__ x_q, float* __restrict__ x_scales, uint2* __restrict__ xs, float* __restrict__ xs_scales,
    int32_t* __restrict__ row_of_route, int32_t* __restrict__ route_of_row, unsigned* err) {
    __shared__ int rows[kMaxK];
    __shared__ int tails[kMaxK];
    __shared__ float red[4];
    const int t = blockIdx.x, tid = threadIdx.x;
    const int n_routes = T * k;
    if (tid < k) {
        const int r = t * k + tid;
        const int lr = lrank[r];
        int row = -1;
        bool bad = false;
        if (lr >= 0) {
            const int e = ids[r];
            if (e >= 0 && e < E) row = bases[static_cast<size_t>(t / chunk_tokens) * kMaxExperts + e] + lr;
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
    uint4 u[VPT];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = tid + j * 128;
        if (v < d8) {
            u[j] = __ldg(x + static_cast<size_t>(t) * d8 + v);
            amax = fmaxf(amax, amax_bf16x8(u[j]));
        }
    }
    amax = block_max(amax, red);   // its barrier also publishes rows[] and tails[]
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = tid + j * 128;
        if (v < d8) {
            const uint2 q = e4m3x8_of_bf16x8(u[j], s);
            x_q[static_cast<size_t>(t) * d8 + v] = q;
            for (int sl = 0; sl < k; ++sl) {
                const int row = rows[sl];
                if (row >= 0) xs[static_cast<size_t>(row) * d8 + v] = q;
                const int tail = tails[sl];
                if (tail >= 0) xs[static_cast<size_t>(tail) * d8 + v] = make_uint2(0u, 0u);
            }
        }
    }
    if (tid < k) {
        if (rows[tid] >= 0) xs_scales[rows[tid]] = s;
        if (tails[tid] >= 0) xs_scales[tails[tid]] = 0.f;
    }
    if (tid == 0) x_scales[t] = s;
}

// ---------------------------------------------------------------------------
// 4-bit activation rows (the 4-bit-activation path), quantized in the
// scatter.  The arithmetic is the 4-bit weight quantizer's, bit for bit: row
// scale s = max|row| / 2688 (1 for an all-zero row); per block of 16 values
// the E4M3 block scale b of (block max / 6) / s (two IEEE fp32 divisions,
// nearest even, saturating); codes = E2M1 of v / (value(b) * s), nearest
// even, saturating at 6; 0 when value(b) is 0.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t e2m1x2_rn(float lo, float hi) {
    unsigned short v;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(v)
        : "f"(hi), "f"(lo));
    return v & 0xFFu;
}

__device__ __forceinline__ float e4m3_code_value(uint32_t b) {
    uint32_t half2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(half2) : "h"(static_cast<unsigned short>(b)));
    float v;
    asm("cvt.f32.f16 %0, %1;" : "=f"(v) : "h"(static_cast<unsigned short>(half2 & 0xFFFFu)));
    return v;
}

// The 16 bf16 values of (a, b) as 8 bytes of E2M1 codes (the lower value of
// each pair in the low nibble) under row scale s; *bscale gets the block's
// E4M3 scale code.
__device__ __forceinline__ uint2 quant_block_fp4(uint4 a, uint4 b, float s, uint32_t& bscale) {
    float val[16];
    const uint32_t wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float bmax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        val[2 * i] = __uint_as_float(wv[i] << 16);
        val[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
        bmax = fmaxf(bmax, fmaxf(fabsf(val[2 * i]), fabsf(val[2 * i + 1])));
    }
    const uint32_t bs = e4m3x2_rn(__fdiv_rn(__fdiv_rn(bmax, 6.f), s), 0.f) & 0xFFu;
    const float vb = e4m3_code_value(bs);
    const float denom = __fmul_rn(vb, s);
    uint32_t p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        p[i] = vb > 0.f ? e2m1x2_rn(__fdiv_rn(val[2 * i], denom), __fdiv_rn(val[2 * i + 1], denom)) : 0u;
    bscale = bs;
    return make_uint2(p[0] | (p[1] << 8) | (p[2] << 16) | (p[3] << 24), p[4] | (p[5] << 8) | (p[6] << 16) | (p[7] << 24));
}

// One CTA of 128 threads per token; thread i takes blocks of 16 values i, i +
// 128, ... (at most VPB of them: d <= VPB * 2048).  Writes the token's codes,
// block scales and scale (x_codes [T][d/2], x_bs [d/64][ld_x][4], x_scales [T])
// and the same to each of its compact rows (xs_*), zeros to rows R .. T*k-1.
template <int VPB>
__global__ void __launch_bounds__(128) scatter_quant_fp4_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ ids, const int32_t* __restrict__ offsets, int T, int k,
    int E, int n_blk, const int32_t* __restrict__ lrank, const int32_t* __restrict__ bases, int chunk_tokens,
    uint2* __restrict__ x_codes, uint8_t* __restrict__ x_bs, int ld_x, float* __restrict__ x_scales,
    uint2* __restrict__ xs_codes, uint8_t* __restrict__ xs_bs, int ld_xs, float* __restrict__ xs_scales,
    int32_t* __restrict__ row_of_route, int32_t* __restrict__ route_of_row, unsigned* err) {
    __shared__ int rows[kMaxK];
    __shared__ int tails[kMaxK];
    __shared__ float red[4];
    const int t = blockIdx.x, tid = threadIdx.x;
    const int n_routes = T * k;
    if (tid < k) {
        const int r = t * k + tid;
        const int lr = lrank[r];
        int row = -1;
        bool bad = false;
        if (lr >= 0) {
            const int e = ids[r];
            if (e >= 0 && e < E) row = bases[static_cast<size_t>(t / chunk_tokens) * kMaxExperts + e] + lr;
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
    uint4 u[VPB][2];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < VPB; ++j) {
        const int v = tid + j * 128;
        if (v < n_blk) {
            u[j][0] = __ldg(x + (static_cast<size_t>(t) * n_blk + v) * 2);
            u[j][1] = __ldg(x + (static_cast<size_t>(t) * n_blk + v) * 2 + 1);
            amax = fmaxf(amax, fmaxf(amax_bf16x8(u[j][0]), amax_bf16x8(u[j][1])));
        }
    }
    amax = block_max(amax, red);   // its barrier also publishes rows[] and tails[]
    const float s = amax > 0.f ? __fdiv_rn(amax, 2688.f) : 1.f;
#pragma unroll
    for (int j = 0; j < VPB; ++j) {
        const int v = tid + j * 128;
        if (v < n_blk) {
            uint32_t b;
            const uint2 q = quant_block_fp4(u[j][0], u[j][1], s, b);
            const size_t sf = static_cast<size_t>(v >> 2);   // 64-value tile of this block
            x_codes[static_cast<size_t>(t) * n_blk + v] = q;
            x_bs[(sf * ld_x + t) * 4 + (v & 3)] = static_cast<uint8_t>(b);
            for (int sl = 0; sl < k; ++sl) {
                const int row = rows[sl];
                if (row >= 0) {
                    xs_codes[static_cast<size_t>(row) * n_blk + v] = q;
                    xs_bs[(sf * ld_xs + row) * 4 + (v & 3)] = static_cast<uint8_t>(b);
                }
                const int tail = tails[sl];
                if (tail >= 0) {
                    xs_codes[static_cast<size_t>(tail) * n_blk + v] = make_uint2(0u, 0u);
                    xs_bs[(sf * ld_xs + tail) * 4 + (v & 3)] = 0;
                }
            }
        }
    }
    if (tid < k) {
        if (rows[tid] >= 0) xs_scales[rows[tid]] = s;
        if (tails[tid] >= 0) xs_scales[tails[tid]] = 0.f;
    }
    if (tid == 0) x_scales[t] = s;
}

// A4 without the row copy, for the fused path (the gate/up kernel gathers
// the token rows itself).  One warp per token: the compact row of each slot
// exactly as scatter_rows_kernel computes it, both index maps, and the
// token's preparation for the fused combine -- its slot counters cleared and,
// when every slot is masked, its output row set to +0.0.
__global__ void __launch_bounds__(256) scatter_index_kernel(const int32_t* __restrict__ ids,
                                                            const int32_t* __restrict__ offsets, int T, int k,
                                                            int E, const int32_t* __restrict__ lrank,
                                                            const int32_t* __restrict__ bases,
                                                            int32_t* __restrict__ row_of_route,
                                                            int32_t* __restrict__ route_of_row,
                                                            int32_t* __restrict__ tile_counts, int n_counts,
                                                            float4* __restrict__ out, int d4, unsigned* err,
                                                            int chunk_tokens) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const int n_routes = T * k;
    int row = -1;
    if (lane < k) {
        const int r = t * k + lane;
        const int lr = lrank[r];
        bool bad = false;
        if (lr >= 0) {
            const int e = ids[r];
            if (e >= 0 && e < E) row = bases[static_cast<size_t>(t / chunk_tokens) * kMaxExperts + e] + lr;
            if (row < 0 || row >= n_routes) {
                bad = true;
                row = -1;
            }
        }
        row_of_route[r] = row;
        if (row >= 0) route_of_row[row] = r;
        const int R = __ldg(offsets + E);
        if (R < 0 || R > n_routes) bad = true;
        else if (R + r < n_routes) route_of_row[R + r] = -1;
        if (bad) atomicOr(err, DEVERR_OFFSETS);
    }
    const bool any = __ballot_sync(0xffffffffu, row >= 0) != 0u;
    for (int j = lane; j < n_counts; j += 32) tile_counts[static_cast<size_t>(t) * n_counts + j] = 0;
    if (!any)
        for (int v = lane; v < d4; v += 32) out[static_cast<size_t>(t) * d4 + v] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------------------
// A7: combine, one CTA per token; slots are added in ascending order with
// fp32 FMAs starting from +0.0, masked slots are skipped.
// ---------------------------------------------------------------------------

// CTA (t, c) combines float4 columns [c * chunk4, (c + 1) * chunk4) of token
// t (one chunk spanning the row unless the chunk is small); U float4 columns
// per thread and pass (2 for wide rows; 1 keeps the registers, and so the
// resident CTAs, of short rows).
template <int U>
__global__ void __launch_bounds__(128) combine_kernel(const float4* __restrict__ y,
                                                      const int32_t* __restrict__ row_of_route,
                                                      const float* __restrict__ w, int k, int d4, int chunk4,
                                                      int cap, float4* __restrict__ out, unsigned* err) {
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
    const int v_end = min(d4, static_cast<int>(blockIdx.y + 1) * chunk4);
    // U float4 columns per thread and pass; the loads of a group of slots are
    // all in flight before the fixed-order sum (slots ascending from +0.0,
    // masked slots skipped, as above)
    constexpr int kGroup = 6;
    const int step = blockDim.x;
    for (int v0 = static_cast<int>(blockIdx.y) * chunk4 + tid; v0 < v_end; v0 += U * step) {
        int vv[U];
        bool in[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            in[u] = v0 + u * step < v_end;
            vv[u] = in[u] ? v0 + u * step : v0;
        }
        float4 acc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < k; s0 += kGroup) {
            float4 yv[U][kGroup];
#pragma unroll
            for (int sl = 0; sl < kGroup; ++sl) {
                const int row = s0 + sl < k ? rows[s0 + sl] : -1;
                if (row >= 0) {
#pragma unroll
                    for (int u = 0; u < U; ++u) yv[u][sl] = __ldg(y + static_cast<size_t>(row) * d4 + vv[u]);
                }
            }
#pragma unroll
            for (int sl = 0; sl < kGroup; ++sl) {
                if (s0 + sl < k && rows[s0 + sl] >= 0) {
                    const float ws = wt[s0 + sl];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        acc[u].x = fmaf(ws, yv[u][sl].x, acc[u].x);
                        acc[u].y = fmaf(ws, yv[u][sl].y, acc[u].y);
                        acc[u].z = fmaf(ws, yv[u][sl].z, acc[u].z);
                        acc[u].w = fmaf(ws, yv[u][sl].w, acc[u].w);
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (in[u]) dst[vv[u]] = acc[u];
    }
}

// ---------------------------------------------------------------------------
// A1-A4 in one launch for small chunks (T*k <= kSmallRoutes, T <= kSmallTokens):
// every CTA recomputes the routing of the whole chunk (a few tokens: cheaper
// than a launch) and copies its share of the token rows; CTA 0 alone writes
// ids, w, counts, offsets, row_of_route and route_of_row.  The results are
// those of moe_route_topk (streaming form: slot-order softmax sum) +
// moe_route_histogram + moe_prefix_offsets + moe_scatter_rows, bit for bit.
// ---------------------------------------------------------------------------

constexpr int kSmallThreads = 512;

// A1-A3 of a small chunk in shared memory, by every CTA of the launch: the
// top-k (warp per token), stable ranks in route order, the prefix; s_row gets
// each route's compact row (-1 masked).  The CTA with `writer` set also
// writes ids, w, counts, offsets and both index maps.  Returns R.  Ends with a
// barrier.
__device__ __forceinline__ int small_chunk_routing(const float* __restrict__ logits,
                                                   const uint8_t* __restrict__ mask, int T, int E, int k,
                                                   bool writer, int32_t* __restrict__ ids, float* __restrict__ w,
                                                   int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                   int32_t* __restrict__ row_of_route,
                                                   int32_t* __restrict__ route_of_row, int* s_e, int* s_row,
                                                   int* s_cnt, int* s_off) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kWarps = kSmallThreads / 32;
    const int n_routes = T * k;
    for (int e = tid; e < kMaxExperts; e += kSmallThreads) s_cnt[e] = 0;

    // A1: warp per token, k rounds of a warp arg-max over order keys
    for (int t = warp; t < T; t += kWarps) {
        const float* row = logits + static_cast<size_t>(t) * E;
        unsigned long long key[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane + 32 * j;
            key[j] = (e < E) ? topk_order_key(__ldg(row + e), e) : 0ull;
        }
        float sel_val = 0.f;
        int sel_id = 0;
        for (int sl = 0; sl < k; ++sl) {
            unsigned long long best = key[0];
#pragma unroll
            for (int j = 1; j < 8; ++j) best = key[j] > best ? key[j] : best;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const unsigned long long o = __shfl_xor_sync(kFull, best, off);
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
        const float top = __shfl_sync(kFull, sel_val, 0);
        float sum = 0.f;
        for (int r = 0; r < k; ++r) sum += expf(__shfl_sync(kFull, sel_val, r) - top);
        const float inv = 1.f / sum;
        if (lane < k) {
            const int r = t * k + lane;
            const bool masked = mask != nullptr && __ldg(mask + r) != 0;
            s_e[r] = masked ? -1 : sel_id;
            if (writer) {
                ids[r] = sel_id;
                w[r] = expf(sel_val - top) * inv;
            }
        }
    }
    __syncthreads();

    // A2: stable ranks in route order (one warp, 32 routes at a time)
    if (warp == 0) {
        const unsigned lt_mask = (1u << lane) - 1u;
        for (int base = 0; base < n_routes; base += 32) {
            const int r = base + lane;
            const int e = r < n_routes ? s_e[r] : -1;
            const unsigned peers = __match_any_sync(kFull, e);
            const int rank = e >= 0 ? s_cnt[e] + __popc(peers & lt_mask) : -1;
            __syncwarp();
            if (e >= 0 && lane == __ffs(peers) - 1) s_cnt[e] += __popc(peers);
            __syncwarp();
            if (r < n_routes) s_row[r] = rank;
        }
        // A3: exclusive prefix over the experts (8 consecutive experts per lane)
        int c[8], local = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane * 8 + i;
            c[i] = e < E ? s_cnt[e] : 0;
            local += c[i];
        }
        int incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(kFull, incl, off);
            if (lane >= off) incl += o;
        }
        int run = incl - local;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane * 8 + i;
            if (e < E) s_off[e] = run;
            run += c[i];
        }
        if (lane == 31) s_off[E] = incl;
    }
    __syncthreads();
    const int R = s_off[E];
    for (int r = tid; r < n_routes; r += kSmallThreads) {
        const int e = s_e[r], rank = s_row[r];
        const int row = e >= 0 ? s_off[e] + rank : -1;
        s_row[r] = row;
        if (writer) {
            row_of_route[r] = row;
            if (row >= 0) route_of_row[row] = r;
        }
    }
    if (writer) {
        for (int e = tid; e < E; e += kSmallThreads) {
            counts[e] = s_cnt[e];
            offsets[e] = s_off[e];
        }
        if (tid == 0) offsets[E] = R;
        for (int j = R + tid; j < n_routes; j += kSmallThreads) route_of_row[j] = -1;
    }
    __syncthreads();
    return R;
}

template <bool TO_F16>
__global__ void __launch_bounds__(kSmallThreads) route_scatter_small_kernel(
    const float* __restrict__ logits, const uint4* __restrict__ x, const uint8_t* __restrict__ mask, int T, int E,
    int k, int row_vecs, int32_t* __restrict__ ids, float* __restrict__ w, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, uint4* __restrict__ xs, int32_t* __restrict__ row_of_route,
    int32_t* __restrict__ route_of_row, unsigned* err, int32_t* __restrict__ tile_counts, int n_counts,
    float4* __restrict__ out, int d4) {
    __shared__ int s_e[kSmallRoutes];     // expert of route r, -1 when masked
    __shared__ int s_row[kSmallRoutes];   // compact row of route r (-1 masked)
    __shared__ int s_cnt[kMaxExperts];
    __shared__ int s_off[kMaxExperts + 1];
    const int tid = threadIdx.x;
    const int n_routes = T * k;
    const bool writer = blockIdx.x == 0;
    const int R = small_chunk_routing(logits, mask, T, E, k, writer, ids, w, counts, offsets, row_of_route,
                                      route_of_row, s_e, s_row, s_cnt, s_off);
    __syncthreads();

    // the fused combine's preparation (fused path): this CTA's share of the
    // tokens gets its slot counters cleared, and +0.0 rows when every slot is
    // masked
    if (tile_counts != nullptr) {
        for (int t = blockIdx.x; t < T; t += gridDim.x) {
            bool any = false;
            for (int s = 0; s < k; ++s) any |= s_row[t * k + s] >= 0;
            for (int j = tid; j < n_counts; j += kSmallThreads) tile_counts[static_cast<size_t>(t) * n_counts + j] = 0;
            if (!any)
                for (int v = tid; v < d4; v += kSmallThreads)
                    out[static_cast<size_t>(t) * d4 + v] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    if (xs == nullptr) return;   // the gate/up kernel gathers the rows itself

    // A4: this CTA's share of the compact rows, and of the zero-filled tail
    bool range = false;
    for (int r = blockIdx.x; r < n_routes; r += gridDim.x) {
        const int row = s_row[r];
        if (row < 0) continue;
        const uint4* src = x + static_cast<size_t>(r / k) * row_vecs;
        uint4* dst = xs + static_cast<size_t>(row) * row_vecs;
        for (int v = tid; v < row_vecs; v += kSmallThreads) {
            uint4 val = __ldg(src + v);
            if (TO_F16) {
                val.x = bf16x2_to_f16x2(val.x, range);
                val.y = bf16x2_to_f16x2(val.y, range);
                val.z = bf16x2_to_f16x2(val.z, range);
                val.w = bf16x2_to_f16x2(val.w, range);
            }
            dst[v] = val;
        }
    }
    for (int j = R + static_cast<int>(blockIdx.x); j < n_routes; j += gridDim.x)
        for (int v = tid; v < row_vecs; v += kSmallThreads)
            xs[static_cast<size_t>(j) * row_vecs + v] = make_uint4(0u, 0u, 0u, 0u);
    if (TO_F16 && __syncthreads_or(range) && tid == 0) atomicOr(err, DEVERR_RANGE);
}

moe_status launch_status() { return cuda_status(cudaGetLastError()); }

// Largest chunk the allocation-free histogram accepts, and its scratch size:
// header + per-chunk counts (at most kMaxChunks chunks) + one in-chunk rank
// per route (512 KB).
constexpr int kNoAllocMaxRoutes = 65536;
constexpr int kNoAllocWords = kWsHeaderWords + kMaxChunks * kMaxExperts + kNoAllocMaxRoutes;

// A2 (histogram only) over the token-aligned chunks of `ws`.
moe_status launch_histogram(const int32_t* ids, const uint8_t* mask, int T, int k, int E, int32_t* counts,
                            int32_t* ws, cudaStream_t s, const DeviceInfo& di) {
    route_chunks_kernel<false, false><<<ws_chunks(T, k), kChunkThreads, 0, s>>>(
        nullptr, mask, T, E, k, ws_chunk_tokens(T), const_cast<int32_t*>(ids), nullptr, ws, counts, nullptr,
        di.error_word);
    return launch_status();
}

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
unsigned long long g_noalloc_context[64];   // context the cached address belongs to

// Device address of g_noalloc_hist_scratch on the current device.  In host
// code the array's name is only a host-side stand-in, so the address is
// looked up (with the device current) and cached per device, together with
// the id of the CUDA context it belongs to: when another context is current
// (after cudaDeviceReset the runtime makes a new primary context and loads
// the module again) the address is looked up again.
moe_status noalloc_scratch(int32_t** out) {
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    unsigned long long ctx = 0;
    moe_status st = current_context_id(&ctx);
    if (st != MOE_OK) return st;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_scratch[dev] == nullptr || ctx == 0 || g_noalloc_context[dev] != ctx) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_hist_scratch);
        if (e != cudaSuccess) return cuda_status(e);
        if ((st = current_context_id(&ctx)) != MOE_OK) return st;
        g_noalloc_scratch[dev] = static_cast<int32_t*>(p);
        g_noalloc_context[dev] = ctx;
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
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (E % 4 == 0 && aligned16(logits)) {  // E <= 256: 16 float4 groups per lane at most
        const int blocks = (T + 31) / 32;  // 4 warps x 8 tokens
        if (k <= 8)
            route_topk_quad_kernel<8><<<blocks, 128, 0, s>>>(logits, T, E, k, ids, w);
        else
            route_topk_quad_kernel<16><<<blocks, 128, 0, s>>>(logits, T, E, k, ids, w);
        return launch_status();
    }
    const int threads = 256, warps_per_block = threads / 32;
    const int blocks = (T + warps_per_block - 1) / warps_per_block;
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
    return launch_histogram(ids, mask, T, k, E, counts, static_cast<int32_t*>(ws), s, di);
}

extern "C" moe_status moe_route_topk_offsets(const float* logits, const uint8_t* mask, int T, int E, int k,
                                             int32_t* ids, float* w, int32_t* counts, int32_t* offsets, void* ws,
                                             void* stream) {
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E);
    MOE_REQUIRE(counts && offsets && ws && aligned16(ws));
    if (T == 0) {
        moe_status st = moe_route_histogram(nullptr, nullptr, 0, k, E, counts, ws, stream);
        return st != MOE_OK ? st : moe_prefix_offsets(counts, 0, k, E, offsets, ws, stream);
    }
    MOE_REQUIRE(logits && ids && w);
    if (ws_chunk_tokens(T) > kChunkWarps) {
        // beyond kMaxChunks chunks of one pass the CTAs would walk their tokens
        // serially: the streaming top-k kernel and the histogram scale better
        moe_status st = moe_route_topk(logits, T, E, k, ids, w, stream);
        if (st == MOE_OK) st = moe_route_histogram(ids, mask, T, k, E, counts, ws, stream);
        if (st == MOE_OK) st = moe_prefix_offsets(counts, T, k, E, offsets, ws, stream);
        return st;
    }
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int chunks = ws_chunks(T, k), ct = ws_chunk_tokens(T);
    int32_t* w32 = static_cast<int32_t*>(ws);
    route_chunks_kernel<true, true><<<chunks, kChunkThreads, 0, s>>>(logits, mask, T, E, k, ct, ids, w, w32, counts,
                                                                    offsets, di.error_word);
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

namespace {

moe_status scatter_rows(const void* x, int es, bool to_f16, const int32_t* ids, const int32_t* offsets, int T,
                        int k, int d, int E, void* xs, int32_t* row_of_route, int32_t* route_of_row, void* ws,
                        void* stream) {
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
    auto kernel = to_f16 ? scatter_rows_kernel<true> : scatter_rows_kernel<false>;
    kernel<<<T, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(x), ids, offsets, T, k, E, row_vecs, w32 + ws_rank_offset(T, k),
        w32 + ws_bases_offset(T, k), static_cast<uint4*>(xs), row_of_route, route_of_row, di.error_word, nullptr, 0,
        nullptr, 0, ws_chunk_tokens(T), nullptr, nullptr, nullptr, 0, nullptr, 0, 0);
    return launch_status();
}

}  // namespace

extern "C" moe_status moe_scatter_rows(const void* x, int dtype, const int32_t* ids, const uint8_t* mask,
                                       const int32_t* offsets, int T, int k, int d, int E, void* xs,
                                       int32_t* row_of_route, int32_t* route_of_row, void* ws, void* stream) {
    (void)mask;  // the histogram already folded the mask into the workspace ranks
    const int es = dtype_size(dtype);
    if (es == 0) return MOE_ERR_UNSUPPORTED;
    return scatter_rows(x, es, false, ids, offsets, T, k, d, E, xs, row_of_route, route_of_row, ws, stream);
}

extern "C" moe_status moe_tile_counts_size(int T, int d, size_t* bytes) {
    MOE_REQUIRE(bytes != nullptr && T >= 0 && d >= 1);
    *bytes = static_cast<size_t>(T) * tile_counts_per_token(d) * sizeof(int32_t);
    return MOE_OK;
}

extern "C" moe_status moe_scatter_index(const int32_t* ids, const uint8_t* mask, const int32_t* offsets, int T,
                                        int k, int d, int E, const void* x, void* xs, int32_t* row_of_route,
                                        int32_t* route_of_row, int32_t* tile_counts, float* out, void* ws,
                                        void* stream) {
    (void)mask;  // folded into the workspace ranks by the histogram
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E && d >= 8 && d % 8 == 0);
    MOE_REQUIRE((x == nullptr) == (xs == nullptr));
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(ids && offsets && row_of_route && route_of_row && tile_counts && out && ws);
    MOE_REQUIRE(aligned16(out) && aligned16(ws));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    const int32_t* w32 = static_cast<const int32_t*>(ws);
    if (x != nullptr) {
        // with the compact copy of the bf16 token rows
        MOE_REQUIRE(aligned16(x) && aligned16(xs));
        scatter_rows_kernel<false><<<T, 128, 0, static_cast<cudaStream_t>(stream)>>>(
            static_cast<const uint4*>(x), ids, offsets, T, k, E, d / 8, w32 + ws_rank_offset(T, k),
            w32 + ws_bases_offset(T, k), static_cast<uint4*>(xs), row_of_route, route_of_row, di.error_word,
            tile_counts, tile_counts_per_token(d), reinterpret_cast<float4*>(out), d / 4, ws_chunk_tokens(T));
        return launch_status();
    }
    scatter_index_kernel<<<(T + 7) / 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        ids, offsets, T, k, E, w32 + ws_rank_offset(T, k), w32 + ws_bases_offset(T, k), row_of_route, route_of_row,
        tile_counts, tile_counts_per_token(d), reinterpret_cast<float4*>(out), d / 4, di.error_word,
        ws_chunk_tokens(T));
    return launch_status();
}

extern "C" moe_status moe_scatter_rows_e4m3(const uint8_t* x_codes, const float* x_scales, const int32_t* ids,
                                            const uint8_t* mask, const int32_t* offsets, int T, int k, int d, int E,
                                            uint8_t* xs, float* xs_scales, int32_t* row_of_route,
                                            int32_t* route_of_row, void* ws, void* stream) {
    (void)mask;  // folded into the workspace ranks by the histogram
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E && d >= 16 && d % 16 == 0);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(x_codes && x_scales && ids && offsets && xs && xs_scales && row_of_route && route_of_row && ws);
    MOE_REQUIRE(aligned16(x_codes) && aligned16(xs) && aligned16(ws));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    const int32_t* w32 = static_cast<const int32_t*>(ws);
    scatter_rows_kernel<false><<<T, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const uint4*>(x_codes), ids, offsets, T, k, E, d / 16, w32 + ws_rank_offset(T, k),
        w32 + ws_bases_offset(T, k), reinterpret_cast<uint4*>(xs), row_of_route, route_of_row, di.error_word,
        nullptr, 0, nullptr, 0, ws_chunk_tokens(T), x_scales, xs_scales);
    return launch_status();
}

extern "C" moe_status moe_scatter_rows_fp4(const uint8_t* x_codes, const uint8_t* x_block_scales, int ld_x,
                                           const float* x_scales, const int32_t* ids, const uint8_t* mask,
                                           const int32_t* offsets, int T, int k, int d, int E, uint8_t* xs_codes,
                                           uint8_t* xs_block_scales, int ld_xs, float* xs_scales,
                                           int32_t* row_of_route, int32_t* route_of_row, void* ws, void* stream) {
    (void)mask;  // folded into the workspace ranks by the histogram
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E && d >= 64 && d % 64 == 0);
    MOE_REQUIRE(ld_x >= T && ld_x % 4 == 0 && ld_xs >= T * k && ld_xs % 4 == 0);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(x_codes && x_block_scales && x_scales && ids && offsets && xs_codes && xs_block_scales &&
                xs_scales && row_of_route && route_of_row && ws);
    MOE_REQUIRE(aligned16(x_codes) && aligned16(xs_codes) && aligned16(x_block_scales) &&
                aligned16(xs_block_scales) && aligned16(ws));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    const int32_t* w32 = static_cast<const int32_t*>(ws);
    scatter_rows_kernel<false><<<T, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const uint4*>(x_codes), ids, offsets, T, k, E, d / 32, w32 + ws_rank_offset(T, k),
        w32 + ws_bases_offset(T, k), reinterpret_cast<uint4*>(xs_codes), row_of_route, route_of_row, di.error_word,
        nullptr, 0, nullptr, 0, ws_chunk_tokens(T), x_scales, xs_scales,
        reinterpret_cast<const uint32_t*>(x_block_scales), ld_x, reinterpret_cast<uint32_t*>(xs_block_scales), ld_xs,
        d / 64);
    return launch_status();
}

extern "C" moe_status moe_scatter_rows_quant_fp4(const void* x, const int32_t* ids, const uint8_t* mask,
                                                  const int32_t* offsets, int T, int k, int d, int E,
                                                  uint8_t* x_codes, uint8_t* x_block_scales, int ld_x,
                                                  float* x_scales, uint8_t* xs_codes, uint8_t* xs_block_scales,
                                                  int ld_xs, float* xs_scales, int32_t* row_of_route,
                                                  int32_t* route_of_row, void* ws, void* stream) {
    (void)mask;  // folded into the workspace ranks by the histogram
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E && d >= 64 && d % 64 == 0);
    MOE_REQUIRE(d <= 4 * 128 * 16);
    MOE_REQUIRE(ld_x >= T && ld_x % 4 == 0 && ld_xs >= T * k && ld_xs % 4 == 0);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(x && ids && offsets && x_codes && x_block_scales && x_scales && xs_codes && xs_block_scales &&
                xs_scales && row_of_route && route_of_row && ws);
    MOE_REQUIRE(aligned16(x) && aligned16(x_codes) && aligned16(xs_codes) && aligned16(ws));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    const int32_t* w32 = static_cast<const int32_t*>(ws);
    const int n_blk = d / 16;
    auto kernel = n_blk <= 2 * 128 ? scatter_quant_fp4_kernel<2> : scatter_quant_fp4_kernel<4>;
    kernel<<<T, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(x), ids, offsets, T, k, E, n_blk, w32 + ws_rank_offset(T, k),
        w32 + ws_bases_offset(T, k), ws_chunk_tokens(T), reinterpret_cast<uint2*>(x_codes), x_block_scales, ld_x,
        x_scales, reinterpret_cast<uint2*>(xs_codes), xs_block_scales, ld_xs, xs_scales, row_of_route, route_of_row,
        di.error_word);
    return launch_status();
}

extern "C" moe_status moe_scatter_rows_quant_e4m3(const void* x, const int32_t* ids, const uint8_t* mask,
                                                   const int32_t* offsets, int T, int k, int d, int E, uint8_t* x_q,
                                                   float* x_scales, uint8_t* xs, float* xs_scales,
                                                   int32_t* row_of_route, int32_t* route_of_row, void* ws,
                                                   void* stream) {
    (void)mask;  // folded into the workspace ranks by the histogram
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E && d >= 16 && d % 16 == 0);
    MOE_REQUIRE(d <= 8 * 128 * 8);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(x && ids && offsets && x_q && x_scales && xs && xs_scales && row_of_route && route_of_row && ws);
    MOE_REQUIRE(aligned16(x) && aligned16(x_q) && aligned16(xs) && aligned16(ws));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    const int32_t* w32 = static_cast<const int32_t*>(ws);
    const int d8 = d / 8;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto kernel = d8 <= 4 * 128 ? scatter_quant_e4m3_kernel<4> : scatter_quant_e4m3_kernel<8>;
    kernel<<<T, 128, 0, s>>>(static_cast<const uint4*>(x), ids, offsets, T, k, E, d8, w32 + ws_rank_offset(T, k),
                             w32 + ws_bases_offset(T, k), ws_chunk_tokens(T), reinterpret_cast<uint2*>(x_q),
                             x_scales, reinterpret_cast<uint2*>(xs), xs_scales, row_of_route, route_of_row,
                             di.error_word);
    return launch_status();
}

extern "C" moe_status moe_quantize_rows_e4m3(const void* a, const int32_t* offsets, int E, int cap, int K,
                                             uint8_t* codes, float* scales, void* stream) {
    MOE_REQUIRE(E >= 1 && E <= kMaxExperts && cap >= 0 && K >= 16 && K % 16 == 0 && K <= 8 * 32 * kQuantVec);
    if (cap == 0) return MOE_OK;
    MOE_REQUIRE(a && offsets && codes && scales && aligned16(a) && aligned16(codes));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    quantize_rows_e4m3_kernel<<<(cap + kQuantWarps - 1) / kQuantWarps, 32 * kQuantWarps, 0,
                                static_cast<cudaStream_t>(stream)>>>(static_cast<const uint4*>(a), K / 8, cap, offsets,
                                                                     E, reinterpret_cast<uint2*>(codes), scales);
    return launch_status();
}

extern "C" moe_status moe_scatter_rows_f16(const void* x, const int32_t* ids, const uint8_t* mask,
                                           const int32_t* offsets, int T, int k, int d, int E, void* xs,
                                           int32_t* row_of_route, int32_t* route_of_row, void* ws, void* stream) {
    (void)mask;
    return scatter_rows(x, 2, true, ids, offsets, T, k, d, E, xs, row_of_route, route_of_row, ws, stream);
}

namespace moe {
namespace {

// A1-A4 with 4-bit rows in one launch for small chunks (T <= kSmallTokens,
// T*k <= kSmallRoutes): CTA t takes the chunk's routing in shared memory (CTA
// 0 writes the index outputs), quantizes token row t with the 4-bit
// quantizer's arithmetic and writes its codes, block scales and scale to x_*
// and to the token's compact rows; the rows R .. T*k-1 get zeros, spread
// over the CTAs.
__global__ void __launch_bounds__(kSmallThreads) route_scatter_quant_small_fp4_kernel(
    const float* __restrict__ logits, const uint4* __restrict__ x, const uint8_t* __restrict__ mask, int T, int E,
    int k, int n_blk, int32_t* __restrict__ ids, float* __restrict__ w, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, uint2* __restrict__ x_codes, uint8_t* __restrict__ x_bs, int ld_x,
    float* __restrict__ x_scales, uint2* __restrict__ xs_codes, uint8_t* __restrict__ xs_bs, int ld_xs,
    float* __restrict__ xs_scales, int32_t* __restrict__ row_of_route, int32_t* __restrict__ route_of_row) {
    __shared__ int s_e[kSmallRoutes];
    __shared__ int s_row[kSmallRoutes];
    __shared__ int s_cnt[kMaxExperts];
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ float red[kSmallThreads / 32];
    const int t = blockIdx.x, tid = threadIdx.x;
    const int n_routes = T * k;
    const int R = small_chunk_routing(logits, mask, T, E, k, t == 0, ids, w, counts, offsets, row_of_route,
                                      route_of_row, s_e, s_row, s_cnt, s_off);
    const uint4* xr = x + static_cast<size_t>(t) * n_blk * 2;
    float amax = 0.f;
    for (int v = tid; v < n_blk; v += kSmallThreads)
        amax = fmaxf(amax, fmaxf(amax_bf16x8(__ldg(xr + 2 * v)), amax_bf16x8(__ldg(xr + 2 * v + 1))));
    amax = block_max(amax, red);
    const float s = amax > 0.f ? __fdiv_rn(amax, 2688.f) : 1.f;
    for (int v = tid; v < n_blk; v += kSmallThreads) {
        uint32_t b;
        const uint2 q = quant_block_fp4(__ldg(xr + 2 * v), __ldg(xr + 2 * v + 1), s, b);
        const size_t sf = static_cast<size_t>(v >> 2);
        x_codes[static_cast<size_t>(t) * n_blk + v] = q;
        x_bs[(sf * ld_x + t) * 4 + (v & 3)] = static_cast<uint8_t>(b);
        for (int sl = 0; sl < k; ++sl) {
            const int row = s_row[t * k + sl];
            if (row >= 0) {
                xs_codes[static_cast<size_t>(row) * n_blk + v] = q;
                xs_bs[(sf * ld_xs + row) * 4 + (v & 3)] = static_cast<uint8_t>(b);
            }
        }
    }
    if (tid < k && s_row[t * k + tid] >= 0) xs_scales[s_row[t * k + tid]] = s;
    if (tid == 0) x_scales[t] = s;
    for (int j = R + t; j < n_routes; j += gridDim.x) {
        for (int v = tid; v < n_blk; v += kSmallThreads) {
            xs_codes[static_cast<size_t>(j) * n_blk + v] = make_uint2(0u, 0u);
            xs_bs[((static_cast<size_t>(v) >> 2) * ld_xs + j) * 4 + (v & 3)] = 0;
        }
        if (tid == 0) xs_scales[j] = 0.f;
    }
}

// The same for E4M3 rows (the FP8-activation path): one scale per token row
// (max|row| / 448), codes x_q [T][d] and, per compact row, xs [T*k][d].
__global__ void __launch_bounds__(kSmallThreads) route_scatter_quant_small_e4m3_kernel(
    const float* __restrict__ logits, const uint4* __restrict__ x, const uint8_t* __restrict__ mask, int T, int E,
    int k, int d8, int32_t* __restrict__ ids, float* __restrict__ w, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, uint2* __restrict__ x_q, float* __restrict__ x_scales, uint2* __restrict__ xs,
    float* __restrict__ xs_scales, int32_t* __restrict__ row_of_route, int32_t* __restrict__ route_of_row) {
    __shared__ int s_e[kSmallRoutes];
    __shared__ int s_row[kSmallRoutes];
    __shared__ int s_cnt[kMaxExperts];
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ float red[kSmallThreads / 32];
    const int t = blockIdx.x, tid = threadIdx.x;
    const int n_routes = T * k;
    const int R = small_chunk_routing(logits, mask, T, E, k, t == 0, ids, w, counts, offsets, row_of_route,
                                      route_of_row, s_e, s_row, s_cnt, s_off);
    const uint4* xr = x + static_cast<size_t>(t) * d8;
    float amax = 0.f;
    for (int v = tid; v < d8; v += kSmallThreads) amax = fmaxf(amax, amax_bf16x8(__ldg(xr + v)));
    amax = block_max(amax, red);
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    for (int v = tid; v < d8; v += kSmallThreads) {
        const uint2 q = e4m3x8_of_bf16x8(__ldg(xr + v), s);
        x_q[static_cast<size_t>(t) * d8 + v] = q;
        for (int sl = 0; sl < k; ++sl) {
            const int row = s_row[t * k + sl];
            if (row >= 0) xs[static_cast<size_t>(row) * d8 + v] = q;
        }
    }
    if (tid < k && s_row[t * k + tid] >= 0) xs_scales[s_row[t * k + tid]] = s;
    if (tid == 0) x_scales[t] = s;
    for (int j = R + t; j < n_routes; j += gridDim.x) {
        for (int v = tid; v < d8; v += kSmallThreads) xs[static_cast<size_t>(j) * d8 + v] = make_uint2(0u, 0u);
        if (tid == 0) xs_scales[j] = 0.f;
    }
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_scatter_quant_small_e4m3(const float* logits, const void* x, const uint8_t* mask,
                                                          int T, int E, int k, int d, int32_t* ids, float* w,
                                                          int32_t* counts, int32_t* offsets, uint8_t* x_q,
                                                          float* x_scales, uint8_t* xs, float* xs_scales,
                                                          int32_t* row_of_route, int32_t* route_of_row,
                                                          void* stream) {
    using namespace moe;
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E && d >= 16 && d % 16 == 0);
    MOE_REQUIRE(T <= kSmallTokens && T * k <= kSmallRoutes);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && x && ids && w && counts && offsets && x_q && x_scales && xs && xs_scales && row_of_route &&
                route_of_row);
    MOE_REQUIRE(aligned16(x) && aligned16(x_q) && aligned16(xs));
    route_scatter_quant_small_e4m3_kernel<<<T, kSmallThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        logits, static_cast<const uint4*>(x), mask, T, E, k, d / 8, ids, w, counts, offsets,
        reinterpret_cast<uint2*>(x_q), x_scales, reinterpret_cast<uint2*>(xs), xs_scales, row_of_route,
        route_of_row);
    return launch_status();
}

extern "C" moe_status moe_route_scatter_quant_small_fp4(const float* logits, const void* x, const uint8_t* mask,
                                                         int T, int E, int k, int d, int32_t* ids, float* w,
                                                         int32_t* counts, int32_t* offsets, uint8_t* x_codes,
                                                         uint8_t* x_block_scales, int ld_x, float* x_scales,
                                                         uint8_t* xs_codes, uint8_t* xs_block_scales, int ld_xs,
                                                         float* xs_scales, int32_t* row_of_route,
                                                         int32_t* route_of_row, void* stream) {
    using namespace moe;
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E && d >= 64 && d % 64 == 0);
    MOE_REQUIRE(T <= kSmallTokens && T * k <= kSmallRoutes);
    MOE_REQUIRE(ld_x >= T && ld_x % 4 == 0 && ld_xs >= T * k && ld_xs % 4 == 0);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && x && ids && w && counts && offsets && x_codes && x_block_scales && x_scales && xs_codes &&
                xs_block_scales && xs_scales && row_of_route && route_of_row);
    MOE_REQUIRE(aligned16(x) && aligned16(x_codes) && aligned16(xs_codes));
    route_scatter_quant_small_fp4_kernel<<<T, kSmallThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        logits, static_cast<const uint4*>(x), mask, T, E, k, d / 16, ids, w, counts, offsets,
        reinterpret_cast<uint2*>(x_codes), x_block_scales, ld_x, x_scales, reinterpret_cast<uint2*>(xs_codes),
        xs_block_scales, ld_xs, xs_scales, row_of_route, route_of_row);
    return launch_status();
}

extern "C" moe_status moe_route_scatter_small(const float* logits, const void* x, int dtype, int xs_f16,
                                              const uint8_t* mask, int T, int E, int k, int d, int32_t* ids,
                                              float* w, int32_t* counts, int32_t* offsets, void* xs,
                                              int32_t* row_of_route, int32_t* route_of_row, void* stream) {
    const int es = dtype_size(dtype);
    if (es == 0) return MOE_ERR_UNSUPPORTED;
    MOE_REQUIRE(T >= 0 && T <= kSmallTokens && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E &&
                T * k <= kSmallRoutes && d >= 1);
    MOE_REQUIRE(!xs_f16 || dtype == MOE_BF16);
    MOE_REQUIRE((static_cast<size_t>(d) * es) % 16 == 0);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && x && ids && w && counts && offsets && xs && row_of_route && route_of_row);
    MOE_REQUIRE(aligned16(x) && aligned16(xs));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    const int row_vecs = static_cast<int>(static_cast<size_t>(d) * es / 16);
    const int grid = T * k < 2 * di.sm_count ? T * k : 2 * di.sm_count;
    auto kernel = xs_f16 ? route_scatter_small_kernel<true> : route_scatter_small_kernel<false>;
    kernel<<<grid, kSmallThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        logits, static_cast<const uint4*>(x), mask, T, E, k, row_vecs, ids, w, counts, offsets,
        static_cast<uint4*>(xs), row_of_route, route_of_row, di.error_word, nullptr, 0, nullptr, 0);
    return launch_status();
}

extern "C" moe_status moe_route_scatter_small_fused(const float* logits, const void* x, const uint8_t* mask, int T,
                                                    int E, int k, int d, int32_t* ids, float* w, int32_t* counts,
                                                    int32_t* offsets, void* xs, int32_t* row_of_route,
                                                    int32_t* route_of_row, int32_t* tile_counts, float* out,
                                                    void* stream) {
    MOE_REQUIRE(T >= 0 && T <= kSmallTokens && E >= 1 && E <= kMaxExperts && k >= 1 && k <= kMaxK && k <= E &&
                T * k <= kSmallRoutes && d >= 8 && d % 8 == 0);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && x && ids && w && counts && offsets && row_of_route && route_of_row && tile_counts && out);
    MOE_REQUIRE(aligned16(x) && aligned16(out) && (xs == nullptr || aligned16(xs)));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    return launch_route_scatter_small_fused(logits, x, mask, T, E, k, d, ids, w, counts, offsets, xs, row_of_route,
                                            route_of_row, tile_counts, out, static_cast<cudaStream_t>(stream), di);
}

namespace moe {

moe_status launch_route_scatter_small_fused(const float* logits, const void* x, const uint8_t* mask, int T, int E,
                                            int k, int d, int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                                            void* xs, int32_t* row_of_route, int32_t* route_of_row,
                                            int32_t* tile_counts, float* out, cudaStream_t st, const DeviceInfo& di) {
    const int row_vecs = d / 8;   // bf16 rows
    const int grid = T * k < 2 * di.sm_count ? T * k : 2 * di.sm_count;
    route_scatter_small_kernel<false><<<grid, kSmallThreads, 0, st>>>(
        logits, static_cast<const uint4*>(x), mask, T, E, k, row_vecs, ids, w, counts, offsets,
        static_cast<uint4*>(xs), row_of_route, route_of_row, di.error_word, tile_counts, tile_counts_per_token(d),
        reinterpret_cast<float4*>(out), d / 4);
    return launch_status();
}

}  // namespace moe

extern "C" moe_status moe_combine(const float* y, const int32_t* row_of_route, const float* w, int T, int k, int d,
                                  float* out, void* stream) {
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= kMaxK && d >= 1 && d % 4 == 0);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(y && row_of_route && w && out && aligned16(y) && aligned16(out));
    DeviceInfo di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    // a small chunk splits every row over CTAs of 128 float4 columns so that all SMs take part
    const int d4 = d / 4;
    const int chunk4 = T < 2 * di.sm_count ? 128 : d4;
    const dim3 grid(T, (d4 + chunk4 - 1) / chunk4);
    // two columns per thread once a CTA's span has at least 512 float4 (2 KB per thread pass)
    auto kernel = chunk4 >= 512 ? combine_kernel<2> : combine_kernel<1>;
    kernel<<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float4*>(y), row_of_route, w, k, d4, chunk4, T * k, reinterpret_cast<float4*>(out),
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
    return launch_histogram(ids, mask, T, k, E, counts, scratch, s, di);
}
