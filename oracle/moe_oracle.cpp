/*
 * CPU oracle of grouped MoE prefill -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain C++17, every floating-point result in double precision.  Only the
 * test suite, __graft_entry__.smoke() and the CPU-baseline / reference legs of
 * bench.py load this library (through oracle/moe_oracle.py, which only
 * marshals arguments).  The product path -- the CUDA library and its Python
 * binding -- never loads it, and this file includes nothing from the product.
 *
 * What it computes follows the page "perf(ds4): batch heterogeneous MoE
 * prefill by expert" (Luce-Org/lucebox PR #640), Summary: every token is
 * routed to its top-k of up to 256 routed experts; a route histogram, an
 * exclusive prefix over the expert counts and a scatter put the token rows in
 * expert-major order; grouped gate/up projections with SwiGLU and a grouped
 * down projection run per expert; a weighted combine brings the expert
 * outputs back to token order, and masked (non-owned) routes contribute
 * exactly zero ("Summary", "Correctness and validation").  The combine is the
 * fused expert-major route combine of the page "perf(ds4): accelerate ROCm
 * decode and long-context selection" (PR #667), lucebox8 A/B section.
 *
 * Readings of points the pages leave open:
 *   - top-k order: logit descending, equal logits to the lower expert id;
 *     -0.0 and +0.0 compare equal (IEEE comparison);
 *   - gate weights: softmax over the k selected logits, which equals a full
 *     softmax renormalised over the selected k;
 *   - the mask applies after selection: a masked route keeps its slot and
 *     its weight but is left out of the histogram, the scatter and the
 *     combine, and the other weights are not renormalised;
 *   - rows inside an expert segment keep ascending route order r = t*k + s;
 *   - SwiGLU: silu(x.Wg) * (x.Wu), silu(a) = a / (1 + e^-a), no clamp;
 *   - combine: out[t] starts at +0.0 and adds w[t,s] * y(t,s) for ascending
 *     s, skipping masked slots (never multiplying them).
 *
 * Arithmetic: operands are read exactly into doubles (bf16 and fp32 values
 * are doubles; an FP8 E4M3 weight is its fp32 channel scale times its code's
 * value, an exact product in double).  Every dot product is summed in
 * ascending index order.  The FFN evaluates several independent dot products
 * in one pass over the index (four rows against one gate row and one up row,
 * or against two down rows); each of them is still the same ascending sum,
 * so the result is bit for bit that of one dot product at a time.  The build
 * disables floating-point contraction (-ffp-contract=off): every operation
 * rounds once, as written.  OpenMP spreads independent outputs over cores;
 * no sum is split across threads.
 *
 * Storage: expert weights are K-contiguous (the nn.Linear convention):
 * w_gate and w_up [E][f][d], w_down [E][d][f].  A weight bank may be given
 * for a range of experts e0 .. e1-1, its first matrix being expert e0's.
 *
 * Pins (tests marked "not gpu" check this file against facts it does not
 * compute itself): hand-derived golden fixtures, brute-force top-k over all
 * orderings on tiny inputs, a closed-form softmax, counting and permutation
 * invariants, the E=1/k=1 reduction to a dense SwiGLU FFN in PyTorch, the
 * k=E reduction to a full softmax mixture, the all-masked exact +0.0 case,
 * the E4M3 rounding against PyTorch's float8_e4m3fn cast and the format's
 * bit layout, and the router projection against one-hot rows and a
 * hand-worked case.  A mutation suite plants plausible mistakes in a copy of
 * this source and checks that some pin fails for each.  No function here is
 * unpinned.
 *
 * Every entry point returns 0 on success and 1 on a bad argument.
 */

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// Storage types of oracle operands.
enum : int {
    ORC_F64 = 0,
    ORC_F32 = 1,
    ORC_BF16 = 2,   // raw bfloat16 bits (the high half of an fp32)
    ORC_E4M3 = 3,   // OCP FP8 E4M3 codes, with one fp32 scale per row
    ORC_FP4 = 4,    // E2M1 codes, two per byte, an E4M3 scale per 16 values and an fp32 scale per row
};

// ---------------------------------------------------------------------------
// Exact decoding of the storage types
// ---------------------------------------------------------------------------

double bf16_value(uint16_t bits) {
    const uint32_t u = static_cast<uint32_t>(bits) << 16;
    float v;
    std::memcpy(&v, &u, sizeof v);
    return v;
}

// OCP FP8 E4M3: sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
// exponent field 0 holds the subnormals m/8 * 2^-6.  (Code 0x7F/0xFF is NaN
// and is never produced by the quantizer below.)
double e4m3_value(uint8_t code) {
    const double sign = (code & 0x80) ? -1.0 : 1.0;
    const int e = (code >> 3) & 0xF;
    const int m = code & 0x7;
    const double mag = e > 0 ? std::ldexp(1.0 + m / 8.0, e - 7) : std::ldexp(m / 8.0, -6);
    return sign * mag;
}

// E2M1 (the 4-bit OCP MX element type): sign bit 3, exponent bits 2-1 with
// bias 1, mantissa bit 0; exponent field 0 holds the subnormal 0.5 * m.
// Values 0, 0.5, 1, 1.5, 2, 3, 4, 6.
double e2m1_value(uint8_t code) {
    const double sign = (code & 0x8) ? -1.0 : 1.0;
    const int e = (code >> 1) & 0x3;
    const int m = code & 0x1;
    const double mag = e > 0 ? std::ldexp(1.0 + m / 2.0, e - 1) : 0.5 * m;
    return sign * mag;
}

double element(const void* p, int dtype, size_t i) {
    switch (dtype) {
        case ORC_F64: return static_cast<const double*>(p)[i];
        case ORC_F32: return static_cast<const float*>(p)[i];
        case ORC_BF16: return bf16_value(static_cast<const uint16_t*>(p)[i]);
        default: return NAN;
    }
}

bool plain_dtype(int dtype) { return dtype == ORC_F64 || dtype == ORC_F32 || dtype == ORC_BF16; }
bool weight_dtype(int dtype) { return plain_dtype(dtype) || dtype == ORC_E4M3 || dtype == ORC_FP4; }

// The 4-bit bank: codes [rows][K/2] (element 2i in the low nibble of byte
// i), block scales [rows][K/16] (E4M3 codes), row scales [rows] (fp32).
struct Fp4Bank {
    const uint8_t* codes;
    const uint8_t* block_scales;
};

// Rows row0 .. row0+n_rows-1 of a [rows][K] weight matrix as doubles.
void decode_rows(const void* base, int dtype, const float* row_scale, size_t row0, size_t n_rows, size_t K,
                 double* out) {
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < static_cast<long long>(n_rows); ++r) {
        const size_t row = row0 + static_cast<size_t>(r);
        double* dst = out + static_cast<size_t>(r) * K;
        if (dtype == ORC_E4M3) {
            const uint8_t* codes = static_cast<const uint8_t*>(base) + row * K;
            const double s = row_scale[row];
            for (size_t c = 0; c < K; ++c) dst[c] = s * e4m3_value(codes[c]);
        } else if (dtype == ORC_FP4) {
            // w = row scale * block scale * E2M1 value, an exact product in double
            const Fp4Bank* bank = static_cast<const Fp4Bank*>(base);
            const uint8_t* codes = bank->codes + row * (K / 2);
            const uint8_t* bs = bank->block_scales + row * (K / 16);
            const double s = row_scale[row];
            for (size_t c = 0; c < K; ++c) {
                const uint8_t code = (c & 1) ? (codes[c / 2] >> 4) : (codes[c / 2] & 0xF);
                dst[c] = s * e4m3_value(bs[c / 16]) * e2m1_value(code);
            }
        } else {
            for (size_t c = 0; c < K; ++c) dst[c] = element(base, dtype, row * K + c);
        }
    }
}

// ---------------------------------------------------------------------------
// Dot products, each summed in ascending index order
// ---------------------------------------------------------------------------

// ra[r] = x_r . a and rb[r] = x_r . b for the NR rows x_r = x + r*ld.
template <int NR>
void dots_rows2(const double* x, size_t ld, size_t K, const double* a, const double* b, double* ra, double* rb) {
    double sa[NR], sb[NR];
    for (int r = 0; r < NR; ++r) sa[r] = sb[r] = 0.0;
    for (size_t c = 0; c < K; ++c) {
        const double av = a[c], bv = b[c];
        for (int r = 0; r < NR; ++r) {
            const double xv = x[r * ld + c];
            sa[r] += xv * av;
            sb[r] += xv * bv;
        }
    }
    for (int r = 0; r < NR; ++r) {
        ra[r] = sa[r];
        rb[r] = sb[r];
    }
}

void dots_rows2_n(int nr, const double* x, size_t ld, size_t K, const double* a, const double* b, double* ra,
                  double* rb) {
    switch (nr) {
        case 4: dots_rows2<4>(x, ld, K, a, b, ra, rb); break;
        case 3: dots_rows2<3>(x, ld, K, a, b, ra, rb); break;
        case 2: dots_rows2<2>(x, ld, K, a, b, ra, rb); break;
        default: dots_rows2<1>(x, ld, K, a, b, ra, rb); break;
    }
}

constexpr int kRowBlock = 4;

double silu(double a) { return a / (1.0 + std::exp(-a)); }

bool check_offsets(const int32_t* offsets, int e0, int e1) {
    if (offsets == nullptr || e0 < 0 || e1 < e0) return false;
    for (int e = e0; e < e1; ++e)
        if (offsets[e] < 0 || offsets[e + 1] < offsets[e]) return false;
    return true;
}

// E4M3 nearest value, ties to even (the default rounding mode of nearbyint),
// saturating at +-448; the result keeps the sign of x, also when it is zero.
double e4m3_round_one(double x) {
    const double a = std::fabs(x);
    int ex = 0;
    std::frexp(a > 0.0 ? a : 1.0, &ex);            // a in [2^(ex-1), 2^ex)
    const int binade = std::max(ex - 1, -6);        // subnormals share the spacing of the 2^-6 binade
    const double quantum = std::ldexp(1.0, binade - 3);
    double r = std::nearbyint(a / quantum) * quantum;
    r = std::min(r, 448.0);
    return std::copysign(r, x);
}

// E2M1 nearest value (ties to even), saturating at +-6; the sign of x is
// kept, also when the result is zero.
double e2m1_round_one(double x) {
    const double a = std::fabs(x);
    int ex = 0;
    std::frexp(a > 0.0 ? a : 1.0, &ex);             // a in [2^(ex-1), 2^ex)
    const int binade = std::max(ex - 1, 0);          // the subnormal 0.5 shares the 2^0 binade's spacing
    const double quantum = std::ldexp(1.0, binade - 1);
    double r = std::nearbyint(a / quantum) * quantum;
    r = std::min(r, 6.0);
    return std::copysign(r, x);
}

uint8_t e2m1_encode_one(double v) {
    const uint8_t sign = std::signbit(v) ? 0x8 : 0x0;
    const double a = std::fabs(v);
    if (a == 0.0) return sign;
    if (a < 1.0) return sign | 0x1;                  // 0.5
    int ex = 0;
    std::frexp(a, &ex);
    const int e_field = ex;                          // a in [2^(ex-1), 2^ex): biased exponent (ex - 1) + 1
    const int mant = static_cast<int>(std::nearbyint(a / std::ldexp(1.0, ex - 1) * 2.0 - 2.0));
    return static_cast<uint8_t>(sign | (e_field << 1) | mant);
}

// bf16 nearest value (ties to even): 8 significant bits with fp32's
// exponent range; subnormals keep the 2^-133 spacing, magnitudes that round
// beyond the largest finite bf16 become infinities.
double bf16_round_one(double x) {
    const double a = std::fabs(x);
    if (!(a > 0.0) || std::isinf(a)) return x;
    int ex = 0;
    std::frexp(a, &ex);                             // a in [2^(ex-1), 2^ex)
    const int binade = std::max(ex - 1, -126);
    const double quantum = std::ldexp(1.0, binade - 7);
    double r = std::nearbyint(a / quantum) * quantum;
    if (r > std::ldexp(255.0 / 128.0, 127)) r = INFINITY;
    return std::copysign(r, x);
}

uint8_t e4m3_encode_one(double v) {
    const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
    const double a = std::fabs(v);
    if (a == 0.0) return sign;
    int ex = 0;
    std::frexp(a, &ex);
    int e_field, mant;
    if (a >= std::ldexp(1.0, -6)) {
        e_field = ex - 1 + 7;
        mant = static_cast<int>(std::nearbyint(a / std::ldexp(1.0, ex - 1) * 8.0 - 8.0));
    } else {
        e_field = 0;
        mant = static_cast<int>(std::nearbyint(a / std::ldexp(1.0, -9)));
    }
    return static_cast<uint8_t>(sign | (e_field << 3) | mant);
}

}  // namespace

extern "C" {

int oracle_version(void) { return 2; }

// Threads the parallel loops use (OpenMP's default team size).
int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

// ---------------------------------------------------------------------------
// A1: top-k routing.  Page "perf(ds4): batch heterogeneous MoE prefill by
// expert", Summary (routed experts, up to 256); page "perf(ds4): extend
// sparse prefill scheduling to 10K", Summary (native top-6 routing).
// ids[t][s]: the s-th expert of token t in (logit descending, id ascending)
// order; w[t][s] = exp(l_s - l_0) / sum over the k selected of exp(l_j - l_0).
// ---------------------------------------------------------------------------
int oracle_route_topk(const float* logits, long long T, int E, int k, int32_t* ids, double* w) {
    if (T < 0 || E < 1 || k < 1 || k > E || (T > 0 && (!logits || !ids || !w))) return 1;
#pragma omp parallel for schedule(static)
    for (long long t = 0; t < T; ++t) {
        const float* row = logits + t * E;
        std::vector<int> order(E);
        std::iota(order.begin(), order.end(), 0);
        // a stable sort keeps equal logits in ascending id order
        std::stable_sort(order.begin(), order.end(), [row](int a, int b) { return row[a] > row[b]; });
        const double l0 = row[order[0]];   // the largest selected logit
        double sum = 0.0;
        for (int s = 0; s < k; ++s) sum += std::exp(static_cast<double>(row[order[s]]) - l0);
        for (int s = 0; s < k; ++s) {
            ids[t * k + s] = order[s];
            w[t * k + s] = std::exp(static_cast<double>(row[order[s]]) - l0) / sum;
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// A2: route histogram.  Same page, Summary (GPU-native route histogram);
// masked owner routes are not counted.  mask may be NULL (nothing masked).
// ---------------------------------------------------------------------------
int oracle_route_histogram(const int32_t* ids, const uint8_t* mask, long long T, int k, int E, int32_t* counts) {
    if (T < 0 || k < 1 || E < 1 || !counts || (T > 0 && !ids)) return 1;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (long long r = 0; r < T * k; ++r) {
        if (mask && mask[r]) continue;
        if (ids[r] < 0 || ids[r] >= E) return 1;
        counts[ids[r]] += 1;
    }
    return 0;
}

// ---------------------------------------------------------------------------
// A3: exclusive prefix.  Same page, Summary (GPU-native prefix).
// offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e].
// ---------------------------------------------------------------------------
int oracle_prefix_offsets(const int32_t* counts, int E, int32_t* offsets) {
    if (E < 1 || !counts || !offsets) return 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    return 0;
}

// ---------------------------------------------------------------------------
// A4: the expert-major permutation.  Same page, Summary (GPU-native
// scatter); page "perf(ds4): extend sparse prefill scheduling to 10K",
// Summary (selected-row order is preserved).  The unmasked route indices,
// stably sorted by expert id: route_of_row[i] = the route in compact row i
// (-1 for i >= R), row_of_route[r] = the compact row of route r (-1 masked).
// ---------------------------------------------------------------------------
int oracle_scatter_permutation(const int32_t* ids, const uint8_t* mask, long long T, int k, int32_t* row_of_route,
                               int32_t* route_of_row) {
    if (T < 0 || k < 1 || (T > 0 && (!ids || !row_of_route || !route_of_row))) return 1;
    const long long n = T * k;
    std::vector<long long> routes;
    for (long long r = 0; r < n; ++r)
        if (!(mask && mask[r])) routes.push_back(r);
    std::stable_sort(routes.begin(), routes.end(), [ids](long long a, long long b) { return ids[a] < ids[b]; });
    for (long long i = 0; i < n; ++i) route_of_row[i] = row_of_route[i] = -1;
    for (size_t i = 0; i < routes.size(); ++i) {
        route_of_row[i] = static_cast<int32_t>(routes[i]);
        row_of_route[routes[i]] = static_cast<int32_t>(i);
    }
    return 0;
}

// xs[i] = x[route_of_row[i] / k] for the n_rows compact rows (as doubles).
int oracle_gather_rows(const void* x, int dtype, long long T, int d, const int32_t* route_of_row, long long n_rows,
                       int k, double* xs) {
    if (!plain_dtype(dtype) || T < 0 || d < 0 || k < 1 || n_rows < 0) return 1;
    if (n_rows > 0 && (!x || !route_of_row || !xs)) return 1;
    for (long long i = 0; i < n_rows; ++i) {
        const long long r = route_of_row[i];
        if (r < 0 || r / k >= T) return 1;
    }
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < n_rows; ++i) {
        const size_t t = static_cast<size_t>(route_of_row[i] / k);
        for (int c = 0; c < d; ++c) xs[i * d + c] = element(x, dtype, t * d + c);
    }
    return 0;
}

// ---------------------------------------------------------------------------
// A5: grouped gate/up with SwiGLU.  Same page, Summary (grouped gate/up
// projections); the SwiGLU is the "DS4 SwiGLU split op" of the page
// "perf(ggml): reuse ROCmFP4 weights across q=4 columns".
// For every expert e in [e0, e1) and compact row i of its segment
// offsets[e] .. offsets[e+1]-1:
//   h[i][j] = silu(g) * u,  g = xs[i] . w_gate_e[j],  u = xs[i] . w_up_e[j].
// w_gate / w_up hold the matrices of experts e0 .. e1-1 ([f][d] each);
// s_gate / s_up their row scales for ORC_E4M3 (else unused).
// ---------------------------------------------------------------------------
int oracle_grouped_swiglu(const double* xs, const int32_t* offsets, int e0, int e1, int d, int f,
                          const void* w_gate, const void* w_up, int wdtype, const float* s_gate, const float* s_up,
                          double* h) {
    if (!weight_dtype(wdtype) || d < 1 || f < 1 || !check_offsets(offsets, e0, e1)) return 1;
    if ((wdtype == ORC_E4M3 || wdtype == ORC_FP4) && (!s_gate || !s_up)) return 1;
    std::vector<double> wg, wu;
    for (int e = e0; e < e1; ++e) {
        const long long lo = offsets[e], n = static_cast<long long>(offsets[e + 1]) - offsets[e];
        if (n == 0) continue;
        if (!xs || !h || !w_gate || !w_up) return 1;
        wg.resize(static_cast<size_t>(f) * d);
        wu.resize(static_cast<size_t>(f) * d);
        decode_rows(w_gate, wdtype, s_gate, static_cast<size_t>(e - e0) * f, f, d, wg.data());
        decode_rows(w_up, wdtype, s_up, static_cast<size_t>(e - e0) * f, f, d, wu.data());
        const long long blocks = (n + kRowBlock - 1) / kRowBlock;
#pragma omp parallel for schedule(dynamic, 8)
        for (long long q = 0; q < blocks * f; ++q) {
            const long long i0 = (q / f) * kRowBlock;
            const int j = static_cast<int>(q % f);
            const int nr = static_cast<int>(std::min<long long>(kRowBlock, n - i0));
            double g[kRowBlock], u[kRowBlock];
            dots_rows2_n(nr, xs + (lo + i0) * d, d, d, wg.data() + static_cast<size_t>(j) * d,
                         wu.data() + static_cast<size_t>(j) * d, g, u);
            for (int r = 0; r < nr; ++r) h[(lo + i0 + r) * f + j] = silu(g[r]) * u[r];
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// A6: grouped down projection.  Same page, Summary (grouped down).
//   y[i][j] = h[i] . w_down_e[j]   (w_down_e [d][f]).
// ---------------------------------------------------------------------------
int oracle_grouped_down(const double* h, const int32_t* offsets, int e0, int e1, int d, int f, const void* w_down,
                        int wdtype, const float* s_down, double* y) {
    if (!weight_dtype(wdtype) || d < 1 || f < 1 || !check_offsets(offsets, e0, e1)) return 1;
    if ((wdtype == ORC_E4M3 || wdtype == ORC_FP4) && !s_down) return 1;
    std::vector<double> wd;
    for (int e = e0; e < e1; ++e) {
        const long long lo = offsets[e], n = static_cast<long long>(offsets[e + 1]) - offsets[e];
        if (n == 0) continue;
        if (!h || !y || !w_down) return 1;
        wd.resize(static_cast<size_t>(d) * f);
        decode_rows(w_down, wdtype, s_down, static_cast<size_t>(e - e0) * d, d, f, wd.data());
        const long long blocks = (n + kRowBlock - 1) / kRowBlock;
        const int pairs = (d + 1) / 2;
#pragma omp parallel for schedule(dynamic, 8)
        for (long long q = 0; q < blocks * pairs; ++q) {
            const long long i0 = (q / pairs) * kRowBlock;
            const int j = 2 * static_cast<int>(q % pairs);
            const int j2 = std::min(j + 1, d - 1);
            const int nr = static_cast<int>(std::min<long long>(kRowBlock, n - i0));
            double a[kRowBlock], b[kRowBlock];
            dots_rows2_n(nr, h + (lo + i0) * f, f, f, wd.data() + static_cast<size_t>(j) * f,
                         wd.data() + static_cast<size_t>(j2) * f, a, b);
            for (int r = 0; r < nr; ++r) {
                y[(lo + i0 + r) * d + j] = a[r];
                if (j2 != j) y[(lo + i0 + r) * d + j2] = b[r];
            }
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// A7: weighted combine.  Page "perf(ds4): accelerate ROCm decode and
// long-context selection", lucebox8 A/B (fused expert-major route combine);
// page "perf(ds4): batch heterogeneous MoE prefill by expert", Summary
// (masked owner routes are exact zero contributions).
//   out[t] = +0.0, then += w[t][s] * y[row_of_route[t*k+s]] for ascending s,
//   masked slots (row -1) skipped.  n_rows = rows of y (checked).
// ---------------------------------------------------------------------------
int oracle_combine(const double* y, long long n_rows, const int32_t* row_of_route, const double* w, long long T,
                   int k, int d, double* out) {
    if (T < 0 || k < 1 || d < 0 || n_rows < 0) return 1;
    if (T > 0 && (!row_of_route || !w || !out)) return 1;
    for (long long r = 0; r < T * k; ++r)
        if (row_of_route[r] >= n_rows || (row_of_route[r] >= 0 && !y)) return 1;
#pragma omp parallel for schedule(static)
    for (long long t = 0; t < T; ++t) {
        double* o = out + t * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        for (int s = 0; s < k; ++s) {
            const long long row = row_of_route[t * k + s];
            if (row < 0) continue;
            const double ws = w[t * k + s];
            for (int c = 0; c < d; ++c) o[c] += ws * y[row * d + c];
        }
    }
    return 0;
}

int oracle_silu(const double* a, long long n, double* out) {
    if (n < 0 || (n > 0 && (!a || !out))) return 1;
    for (long long i = 0; i < n; ++i) out[i] = silu(a[i]);
    return 0;
}

// ---------------------------------------------------------------------------
// FP8 E4M3 expert weights with one scale per output channel (the low-bit
// expert weights of the page "perf(ds4): batch heterogeneous MoE prefill by
// expert", "Fresh main-snapshot requalification", and of the page
// "perf(ggml): reuse ROCmFP4 weights across q=4 columns").  For a row w of K
// values (fp32, or bf16 read exactly as fp32):
//   scale = max|w| / 448 in fp32 (1 for an all-zero row),
//   code  = E4M3 code of the nearest E4M3 value (ties to even, saturating)
//           to the fp32 quotient w / scale.
// The weight the FFN uses is scale * value(code).  (A float64 row is read
// as its nearest fp32 values.)  The same quantizer, applied to the rows of x
// and of h, gives the activations of the FP8-activation path.
// ---------------------------------------------------------------------------
int oracle_e4m3_round(const double* x, long long n, double* out) {
    if (n < 0 || (n > 0 && (!x || !out))) return 1;
    for (long long i = 0; i < n; ++i) out[i] = e4m3_round_one(x[i]);
    return 0;
}

// An intermediate stored in bf16 (the h of the bf16 and FP8-activation
// paths): the nearest bf16 value of each element, ties to even.
int oracle_round_bf16(const double* x, long long n, double* out) {
    if (n < 0 || (n > 0 && (!x || !out))) return 1;
    for (long long i = 0; i < n; ++i) out[i] = bf16_round_one(x[i]);
    return 0;
}

int oracle_e4m3_encode(const double* v, long long n, uint8_t* codes) {
    if (n < 0 || (n > 0 && (!v || !codes))) return 1;
    for (long long i = 0; i < n; ++i) codes[i] = e4m3_encode_one(v[i]);
    return 0;
}

int oracle_e4m3_decode(const uint8_t* codes, long long n, double* v) {
    if (n < 0 || (n > 0 && (!v || !codes))) return 1;
    for (long long i = 0; i < n; ++i) v[i] = e4m3_value(codes[i]);
    return 0;
}

int oracle_quantize_fp8(const void* w, int dtype, long long rows, int K, uint8_t* codes, float* scales) {
    if (!plain_dtype(dtype) || rows < 0 || K < 1) return 1;
    if (rows > 0 && (!w || !codes || !scales)) return 1;
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int c = 0; c < K; ++c)
            amax = std::max(amax, std::fabs(static_cast<float>(element(w, dtype, r * K + c))));
        const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
        scales[r] = scale;
        for (int c = 0; c < K; ++c) {
            const float q = static_cast<float>(element(w, dtype, r * K + c)) / scale;
            codes[r * K + c] = e4m3_encode_one(e4m3_round_one(q));
        }
    }
    return 0;
}

int oracle_dequantize_fp8(const uint8_t* codes, const float* scales, long long rows, int K, double* w) {
    if (rows < 0 || K < 1 || (rows > 0 && (!codes || !scales || !w))) return 1;
    decode_rows(codes, ORC_E4M3, scales, 0, static_cast<size_t>(rows), static_cast<size_t>(K), w);
    return 0;
}

// ---------------------------------------------------------------------------
// 4-bit expert weights: E2M1 codes with an E4M3 scale per block of 16
// consecutive K-values and an fp32 scale per row (output channel) -- the
// block-scaled 4-bit format of NVIDIA's NVFP4, its per-tensor scale taken
// per channel.  For a row w of K values (fp32, or bf16 read exactly), in
// fp32 arithmetic:
//   s   = max|w| / 2688 (2688 = 6 * 448; 1 for an all-zero row),
//   b_j = E4M3 code (nearest, ties to even, saturating) of
//         (max over block j of |w|) / 6 / s (two divisions, in this order),
//   q_i = E2M1 code (nearest, ties to even, saturating at 6) of
//         w_i / (value(b_j) * s) for i in block j; 0 when value(b_j) is 0.
// The weight the FFN uses is s * value(b_j) * value(q_i), exactly.
// ---------------------------------------------------------------------------
int oracle_e2m1_round(const double* x, long long n, double* out) {
    if (n < 0 || (n > 0 && (!x || !out))) return 1;
    for (long long i = 0; i < n; ++i) out[i] = e2m1_round_one(x[i]);
    return 0;
}

int oracle_e2m1_encode(const double* v, long long n, uint8_t* codes) {
    if (n < 0 || (n > 0 && (!v || !codes))) return 1;
    for (long long i = 0; i < n; ++i) codes[i] = e2m1_encode_one(v[i]);
    return 0;
}

int oracle_e2m1_decode(const uint8_t* codes, long long n, double* v) {
    if (n < 0 || (n > 0 && (!v || !codes))) return 1;
    for (long long i = 0; i < n; ++i) v[i] = e2m1_value(codes[i] & 0xF);
    return 0;
}

int oracle_quantize_fp4(const void* w, int dtype, long long rows, int K, uint8_t* codes, uint8_t* block_scales,
                        float* scales) {
    if (!plain_dtype(dtype) || rows < 0 || K < 16 || K % 16 != 0) return 1;
    if (rows > 0 && (!w || !codes || !block_scales || !scales)) return 1;
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < rows; ++r) {
        auto wv = [&](int c) { return static_cast<float>(element(w, dtype, static_cast<size_t>(r) * K + c)); };
        float amax = 0.0f;
        for (int c = 0; c < K; ++c) amax = std::max(amax, std::fabs(wv(c)));
        const float s = amax > 0.0f ? amax / 2688.0f : 1.0f;
        scales[r] = s;
        uint8_t* cr = codes + static_cast<size_t>(r) * (K / 2);
        for (int c = 0; c < K / 2; ++c) cr[c] = 0;
        for (int j = 0; j < K / 16; ++j) {
            float bmax = 0.0f;
            for (int i = 16 * j; i < 16 * j + 16; ++i) bmax = std::max(bmax, std::fabs(wv(i)));
            const float t = bmax / 6.0f / s;
            const uint8_t b = e4m3_encode_one(e4m3_round_one(t));
            block_scales[static_cast<size_t>(r) * (K / 16) + j] = b;
            const float vb = static_cast<float>(e4m3_value(b));
            const float denom = vb * s;
            for (int i = 16 * j; i < 16 * j + 16; ++i) {
                const uint8_t q = vb > 0.0f ? e2m1_encode_one(e2m1_round_one(wv(i) / denom)) : 0;
                cr[i / 2] |= static_cast<uint8_t>(q << (4 * (i & 1)));
            }
        }
    }
    return 0;
}

int oracle_dequantize_fp4(const uint8_t* codes, const uint8_t* block_scales, const float* scales, long long rows,
                          int K, double* w) {
    if (rows < 0 || K < 16 || K % 16 != 0 || (rows > 0 && (!codes || !block_scales || !scales || !w))) return 1;
    const Fp4Bank bank{codes, block_scales};
    decode_rows(&bank, ORC_FP4, scales, 0, static_cast<size_t>(rows), static_cast<size_t>(K), w);
    return 0;
}

// ---------------------------------------------------------------------------
// The router projection in front of A1 (page "perf(ds4): extend sparse
// prefill scheduling to 10K", Summary: native top-6 routing from router
// logits): logits[t][e] = x[t] . wr[e], wr [E][d] K-contiguous.
// ---------------------------------------------------------------------------
int oracle_router_logits(const void* x, int xdtype, const void* wr, int wdtype, long long T, int E, int d,
                         double* logits) {
    if (!plain_dtype(xdtype) || !plain_dtype(wdtype) || T < 0 || E < 1 || d < 1) return 1;
    if (T > 0 && (!x || !wr || !logits)) return 1;
#pragma omp parallel for schedule(static)
    for (long long q = 0; q < T * E; ++q) {
        const long long t = q / E;
        const int e = static_cast<int>(q % E);
        double s = 0.0;
        for (int c = 0; c < d; ++c)
            s += element(x, xdtype, static_cast<size_t>(t) * d + c) * element(wr, wdtype, static_cast<size_t>(e) * d + c);
        logits[q] = s;
    }
    return 0;
}

}  // extern "C"
