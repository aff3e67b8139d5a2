// combine.cu -- moe_combine and moe_combine_backward.
//
// The combine of "03 · Combine 与 forward / backward 对称性" §1,
//   out[t] = sum_j w[t,j] * y[slot_pos[t,j]],
// done as a deterministic gather-reduce (a warp reads a token's k rows and
// writes its output row; eight-slot rows are cut into column parts taken by
// neighbouring warps) instead of the scatter-add of §2.3.
//
// Accuracy contract: the result is the double-precision slot-order sum
// rounded once to the output type.  The fast path accumulates s = sum w*y
// with float FMAs in slot order together with a = sum |w|*|y|.  The float
// error of s is at most k*2^-24*(1+2^-15)*a (plus the double sum's own error,
// far smaller), so if the whole interval [s-B, s+B] rounds to a single bf16
// value, that value is the rounding of the double sum (rounding is monotone).
// Elements whose interval straddles a rounding boundary -- about 2^-12 of them
// on typical data -- are recomputed in double in the same slot order.
// float32 outputs always take the double path.
//
// The backward (§4): grad_y[slot_pos[t,j]] = w[t,j]*grad_out[t] is the exact
// product rounded once (float product plus an error-free tie check), and
// grad_probs[t,j] = <grad_out[t], y[slot_pos[t,j]]> is a double-float
// (Knuth TwoSum) accumulation per lane followed by a fixed butterfly of
// double-float additions (and, for a row cut into column parts, the parts'
// double-float partials added in part order), so it is deterministic and far
// more accurate than a plain float dot.
#include "pipeline.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kFull = 0xFFFFFFFFu;

int grid_for(const void* kernel, int threads, size_t smem, int64_t work_blocks) {
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t cap = int64_t(sm_count()) * per_sm;
    return int(work_blocks < cap ? (work_blocks > 0 ? work_blocks : 1) : cap);
}

int grid_for(const void* kernel, int threads, int64_t work_blocks) {
    return grid_for(kernel, threads, 0, work_blocks);
}

// Float error bound factor for a k-term FMA chain, rounded up (see header).
float combine_bound_factor(int k) { return float(k) * 0x1p-24f * (1.0f + 0x1p-15f); }

// Double-float error bound factor (see dd_sum_bf16), rounded up generously.
float dd_bound_factor(int k) {
    const float n = 2.0f * float(k);
    return 4.0f * n * n * 0x1p-48f + float(k) * 0x1p-52f;
}

// Column parts of an eight-slot row: about 7 lane steps of 32 vectors each,
// and a power of two that divides the block's warps (1, 2 or 4).  The
// backward stops at 2: each part restarts its copy pipeline and meets its
// sibling parts at two barriers, which at 4 parts cost more than the balance
// gains when every slot is live (DeepSeek shape: 1 part 687 us, 2 parts
// 665 us, 4 parts 705 us; the forward: 343, 341, 338 us).
int column_parts(int64_t nvec) {
    const int64_t steps = (nvec + 31) / 32;
    return steps >= 28 ? 4 : steps >= 14 ? 2 : 1;
}

int column_parts_bwd(int64_t nvec) { return column_parts(nvec) >= 2 ? 2 : 1; }
static_assert(kWarps % 4 == 0, "column parts divide the block's warps");

// Stage the token's slot rows and weights in shared memory (lanes < k).
__device__ __forceinline__ void stage_slots(int32_t* s_pos, float* s_w, const int32_t* slot_pos,
                                            const float* topk_w, int64_t t, int k,
                                            int64_t n_rows, int lane) {
    if (lane < k) {
        const int32_t p = slot_pos[t * k + lane];
        s_pos[lane] = (p >= 0 && p < n_rows) ? p : -1;
        s_w[lane] = topk_w ? topk_w[t * k + lane] : 1.0f;
    }
    __syncwarp();
}

// Two floats in one 64-bit register (low word = even element): Blackwell's
// packed f32x2 add/sub/mul run two lanes of float arithmetic per instruction.
typedef unsigned long long f2_t;

__device__ __forceinline__ f2_t f2_pack(float lo, float hi) {
    f2_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(f2_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2_t f2_add(f2_t a, f2_t b) {
    f2_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2_t f2_sub(f2_t a, f2_t b) {
    f2_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2_t f2_mul(f2_t a, f2_t b) {
    f2_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// bf16 pair (low half = even element) -> two floats
__device__ __forceinline__ f2_t f2_from_bf16x2(uint32_t p) {
    return f2_pack(bf16lo_to_f32(p), bf16hi_to_f32(p));
}
// Knuth TwoSum on both lanes: (hi, lo) += q with the rounding error of
// hi + q kept exactly in lo's input.
__device__ __forceinline__ void f2_two_sum_acc(f2_t& hi, f2_t& lo, f2_t q) {
    const f2_t s = f2_add(hi, q);
    const f2_t bp = f2_sub(s, hi);
    const f2_t e = f2_add(f2_sub(hi, f2_sub(s, bp)), f2_sub(q, bp));
    hi = s;
    lo = f2_add(lo, e);
}

// w * (g0, g1) -> bf16 pair of the exact products.  The packed float products
// are correctly rounded floats; a bf16 midpoint (low half 0x8000) in either
// one sends the pair to the error-free tie break.
__device__ __forceinline__ uint32_t scale_pair_bf16_f2(f2_t w2, f2_t g2) {
    float p0, p1;
    f2_unpack(f2_mul(w2, g2), p0, p1);
    const uint32_t lows = __byte_perm(__float_as_uint(p0), __float_as_uint(p1), 0x5410) ^ 0x80008000u;
    if (((lows - 0x00010001u) & ~lows & 0x80008000u) != 0) {   // a half equal to 0x8000
        float w, w_hi, g0, g1;
        f2_unpack(w2, w, w_hi);
        f2_unpack(g2, g0, g1);
        return mul_bf16_rn(w, g0) | (mul_bf16_rn(w, g1) << 16);
    }
    return pack_bf16x2_rn(p0, p1);
}

// A bf16 pair with any -0 half turned into +0 (a sum that starts from +0
// never ends on -0).
__device__ __forceinline__ uint32_t plus_zero_bf16x2(uint32_t r) {
    if ((r & 0xFFFFu) == 0x8000u) r &= 0xFFFF0000u;
    if ((r >> 16) == 0x8000u) r &= 0x0000FFFFu;
    return r;
}

constexpr int kBwdStages = 3;

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))), "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

// -------------------------------------------------------- combine, bf16 rows

constexpr int kU = 2;   // 16-byte vectors per lane per batch
constexpr int kJ = 4;   // slot rows loaded per batch

__device__ __forceinline__ float unpack_bf16(const uint4& d, int i) {
    const uint32_t w = i < 2 ? d.x : i < 4 ? d.y : i < 6 ? d.z : d.w;
    return (i & 1) ? bf16hi_to_f32(w) : bf16lo_to_f32(w);
}

__device__ __forceinline__ void set_word(uint4& d, int q, uint32_t v) {
    if (q == 0) d.x = v; else if (q == 1) d.y = v; else if (q == 2) d.z = v; else d.w = v;
}
__device__ __forceinline__ uint32_t get_word(const uint4& d, int q) {
    return q == 0 ? d.x : q == 1 ? d.y : q == 2 ? d.z : d.w;
}

// Interval that certainly holds both the exact slot-order sum and its double
// evaluation, from the float sum s and a = sum |w|*|y|.  a == 0 means every
// term is an exact zero: the sum is exactly +0 (a float or double chain of
// zero products starting from +0 stays +0), so the interval is the point s.
// Otherwise the float error is at most cbound * a, plus an absolute k*2^-149
// for results in the subnormal range.
__device__ __forceinline__ void certify_interval(float s, float a, float cbound, int k,
                                                 float& lo, float& hi) {
    if (a == 0.0f) {
        lo = s;
        hi = s;
        return;
    }
    const float b = __fmaf_ru(a, cbound, float(k) * 0x1p-149f);
    lo = __fsub_rd(s, b);
    hi = __fadd_ru(s, b);
}

// Double path for one bf16 element: exact slot order, one rounding.
__device__ __noinline__ uint16_t combine_elem_f64_bf16(const uint16_t* y, int64_t H, int64_t h,
                                                       const int32_t* s_pos, const float* s_w,
                                                       int k) {
    double acc = 0.0;
    for (int j = 0; j < k; ++j) {
        const int32_t p = s_pos[j];
        if (p < 0) continue;
        acc = fma(double(s_w[j]), double(bf16_to_f32(y[int64_t(p) * H + h])), acc);
    }
    return f64_to_bf16_rn(acc);
}

// Knuth TwoSum: s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// Middle tier for an element the float fast path could not certify: the
// slot-order sum in double-float arithmetic (Dekker/Knuth error-free
// TwoProduct and TwoSum, all on the float pipes), certified against the exact
// bf16 rounding midpoints around it.  Its error is below
// 2*(2k*2^-24)^2 * sum|w*y| (Ogita-Rump-Oishi Sum2 bound), plus the double
// sum's own k*2^-53 * sum|w*y|; if the whole interval lies strictly between
// the two midpoints of one bf16 value, that value is the rounding of the
// double slot-order sum.  An interval cannot decide a sum that sits exactly
// on a midpoint, which unweighted sums of bf16 rows often do, so the chain
// also records whether every product and every partial sum was exact: then
// each prefix of the slot-order sum is a float, the double chain computes the
// same prefixes exactly, and the float sum rounds directly.  Returns false
// when it cannot decide.
__device__ __forceinline__ bool dd_sum_bf16(const float* w, const float* y, const bool* valid,
                                            int n, float dd_bound, uint16_t* out) {
    float hi = 0.0f, lo = 0.0f, a = 0.0f;
    bool exact = true;
    for (int j = 0; j < n; ++j) {
        if (!valid[j]) continue;
        const float p = __fmul_rn(w[j], y[j]);
        const float ep = __fmaf_rn(w[j], y[j], -p);          // w*y == p + ep exactly
        float sum, es;
        two_sum(hi, p, sum, es);
        exact = exact && ep == 0.0f && es == 0.0f;
        hi = sum;
        lo = __fadd_rn(lo, __fadd_rn(es, ep));
        a = __fmaf_rn(fabsf(w[j]), fabsf(y[j]), a);
    }
    if (exact) { *out = f32_to_bf16_rn(hi); return true; }   // hi is the exact sum
    const float s = __fadd_rn(hi, lo);
    const float b = __fmaf_ru(a, dd_bound, 0x1p-126f);
    // r = bf16(s); its rounding midpoints m_lo < r < m_hi are exact floats
    const uint16_t r = f32_to_bf16_rn(s);
    const float rv = bf16_to_f32(r);
    const float up = bf16_to_f32(uint16_t(r + 1)), dn = bf16_to_f32(uint16_t(r - 1));
    const float m_hi = rv >= 0 ? __fmul_rn(__fadd_rn(rv, up), 0.5f) : __fmul_rn(__fadd_rn(rv, dn), 0.5f);
    const float m_lo = rv >= 0 ? __fmul_rn(__fadd_rn(rv, dn), 0.5f) : __fmul_rn(__fadd_rn(rv, up), 0.5f);
    if (!(fabsf(rv) > 0x1p-120f && fabsf(rv) < 0x1p120f)) return false;   // leave extremes to double
    // (hi + lo) - b > m_lo and (hi + lo) + b < m_hi, evaluated so that rounding
    // can only make the test fail: hi - m_lo is exact (Sterbenz), then round down
    const float below = __fadd_rd(__fsub_rn(hi, m_lo), __fsub_rd(lo, b));
    const float above = __fadd_rd(__fsub_rn(m_hi, hi), __fsub_rd(-lo, b));
    if (below > 0.0f && above > 0.0f) { *out = r; return true; }
    return false;
}

// At most one live term: the double slot-order sum is fma(w, y, +0), the
// exact product (a zero product gives +0), rounded once; 4 vectors in flight
// per lane (a lone row per step would leave the warp latency-bound).  Writes
// columns [vb, ve) of the token's output row.
__device__ __forceinline__ void combine_single(const uint4* __restrict__ y, int64_t nvec,
                                               int64_t vb, int64_t ve, int lane, bool live,
                                               int64_t p, float w, uint4* __restrict__ orow) {
    const f2_t w2 = f2_pack(w, w);
    for (int64_t v0 = vb + lane; v0 < ve; v0 += 32 * 4) {
        uint4 d[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t v = v0 + 32 * u;
            d[u] = (live && v < ve) ? __ldcs(y + p * nvec + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t v = v0 + 32 * u;
            if (v >= ve) break;
            uint4 r = make_uint4(0, 0, 0, 0);
            if (live) {
                r.x = plus_zero_bf16x2(scale_pair_bf16_f2(w2, f2_from_bf16x2(d[u].x)));
                r.y = plus_zero_bf16x2(scale_pair_bf16_f2(w2, f2_from_bf16x2(d[u].y)));
                r.z = plus_zero_bf16x2(scale_pair_bf16_f2(w2, f2_from_bf16x2(d[u].z)));
                r.w = plus_zero_bf16x2(scale_pair_bf16_f2(w2, f2_from_bf16x2(d[u].w)));
            }
            __stcs(orow + v, r);
        }
    }
}

// One 16-byte column (8 bf16 elements) of a token's combine from its k slot
// vectors d[j] (rows pj[j] < 0 are empty): the certified float sum, else the
// double-float tier, else double -- the double slot-order sum rounded once.
template <int KMAX, bool PLAIN>   // PLAIN: unit weights (plain sum)
__device__ __forceinline__ uint4 combine_vector(const uint4 (&d)[KMAX], const int32_t (&pj)[KMAX],
                                                const float (&wj)[KMAX], int k, float cbound,
                                                float dd_bound) {
    if constexpr (PLAIN) {
        // plain sum (permute backward): every product is exact, so a
        // TwoSum chain shows whether the float sum is the exact
        // slot-order sum (then the double chain computes the same
        // prefixes and it rounds directly); the rare inexact element
        // goes through the certified tiers.  The chain runs on both
        // elements of a 32-bit word at once (packed f32x2 add/sub
        // round each half like the scalar operations).
        uint4 res;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            f2_t hi2 = 0ull;
            uint32_t err0 = 0, err1 = 0;      // error terms' magnitude bits
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (pj[j] < 0) continue;
                const uint32_t wd = q == 0 ? d[j].x : q == 1 ? d[j].y : q == 2 ? d[j].z : d[j].w;
                const f2_t y2 = f2_from_bf16x2(wd);
                const f2_t s2 = f2_add(hi2, y2);
                const f2_t bp = f2_sub(s2, hi2);
                const f2_t e2 = f2_add(f2_sub(hi2, f2_sub(s2, bp)), f2_sub(y2, bp));
                hi2 = s2;
                err0 |= uint32_t(e2) & 0x7FFFFFFFu;
                err1 |= uint32_t(e2 >> 32) & 0x7FFFFFFFu;
            }
            float hsum[2];
            f2_unpack(hi2, hsum[0], hsum[1]);
            uint16_t half[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = 2 * q + h;
                if ((h == 0 ? err0 : err1) == 0) {
                    half[h] = f32_to_bf16_rn(hsum[h]);
                    continue;
                }
                float yv[KMAX];
                bool valid[KMAX];
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    valid[j] = pj[j] >= 0;
                    yv[j] = unpack_bf16(d[j], i);
                }
                if (!dd_sum_bf16(wj, yv, valid, KMAX, dd_bound, &half[h])) {
                    double acc = 0.0;
#pragma unroll
                    for (int j = 0; j < KMAX; ++j)
                        if (valid[j]) acc = fma(double(wj[j]), double(yv[j]), acc);
                    half[h] = f64_to_bf16_rn(acc);
                }
            }
            set_word(res, q, uint32_t(half[0]) | (uint32_t(half[1]) << 16));
        }
        return res;
    } else {
        float s[8], a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) { s[i] = 0.0f; a[i] = 0.0f; }
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (pj[j] < 0) continue;
            const float w = wj[j], aw = fabsf(w);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float yv = unpack_bf16(d[j], i);
                s[i] = __fmaf_rn(w, yv, s[i]);
                a[i] = __fmaf_rn(aw, fabsf(yv), a[i]);
            }
        }
        uint4 res;
        uint32_t open = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float lo0, hi0, lo1, hi1;
            certify_interval(s[2 * q], a[2 * q], cbound, k, lo0, hi0);
            certify_interval(s[2 * q + 1], a[2 * q + 1], cbound, k, lo1, hi1);
            const uint32_t lo = pack_bf16x2_rn(lo0, lo1);
            const uint32_t hi = pack_bf16x2_rn(hi0, hi1);
            set_word(res, q, lo);
            const uint32_t diff = lo ^ hi;              // bit 2q + h: element 2q + h is open
            open |= ((diff & 0xFFFFu) ? 1u : 0u) << (2 * q);
            open |= ((diff >> 16) ? 1u : 0u) << (2 * q + 1);
        }
        if (open) {
            // only the open elements take the slower tiers (about 1 in 600
            // on GEMM outputs; a warp runs the union of its lanes' open ones)
            bool valid[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j) valid[j] = pj[j] >= 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (!(open & (1u << i))) continue;
                float yv[KMAX];
#pragma unroll
                for (int j = 0; j < KMAX; ++j) yv[j] = unpack_bf16(d[j], i);
                uint16_t half;
                if (!dd_sum_bf16(wj, yv, valid, KMAX, dd_bound, &half)) {
                    // last resort: double, slot order, one rounding
                    double acc = 0.0;
#pragma unroll
                    for (int j = 0; j < KMAX; ++j)
                        if (valid[j]) acc = fma(double(wj[j]), double(yv[j]), acc);
                    half = f64_to_bf16_rn(acc);
                }
                const uint32_t w = get_word(res, i >> 1);
                set_word(res, i >> 1, (i & 1) ? (w & 0xFFFFu) | (uint32_t(half) << 16)
                                              : (w & 0xFFFF0000u) | uint32_t(half));
            }
        }
        return res;
    }
}

// k <= 8: one 16-byte column per lane step with every slot row of it held in
// registers, so an element whose rounding cannot be certified is recomputed
// in double from the same registers (no reload).  (A cp.async ring as in
// the backward measured slower here: 352 vs 345 us at T=16384, H=7168, k=8.)
// Up to six slots the kernel is held to 64 registers (4 blocks, 32 warps per
// SM; a few bytes of rare-path spill): at one wave of tokens it is bound by
// instruction latency, which more resident warps hide.  Eight slots keep
// up to 128 (2 blocks, 16 warps per SM: the DeepSeek-shaped workload is
// HBM-bound there).
template <int KMAX, bool PLAIN>   // PLAIN: topk_w == NULL (plain sum)
__global__ void __launch_bounds__(kThreads, KMAX <= 6 ? 4 : 2)
combine_bf16_regs_kernel(const uint4* __restrict__ y, int64_t T, int64_t nvec, int k, int64_t n_rows,
                         const int32_t* __restrict__ slot_pos, const float* __restrict__ topk_w,
                         uint4* __restrict__ out, float cbound, float dd_bound, int parts) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // work item = (token, column part): consecutive warps take the parts of
    // one token, so a token whose every slot is live does not hold one warp
    // for its whole row while lighter tokens finish elsewhere (capacity drops
    // leave a few such tokens among many with none).  Eight-slot rows only;
    // the host passes parts = 1 for the smaller instantiations.
    const int lp = 31 - __clz(parts);                   // parts is a power of two
    const int64_t P = int64_t(1) << lp;
    const int64_t chunk = ((nvec + P - 1) / P + 31) / 32 * 32;
    const int64_t items = T * P, step = int64_t(gridDim.x) * kWarps;
    // lane j < k holds slot j of an item; the next item's slot is loaded
    // while this one is combined, so a warp waits on the slot arrays only
    // once (on layouts where most tokens keep one slot or none, that wait
    // was most of the kernel)
    int32_t next_p = -1;
    float next_w = 0.0f;
    auto load_slot = [&](int64_t it) {
        if (it < items && lane < k) {
            const int64_t tt = it >> lp;
            const int32_t p = slot_pos[tt * k + lane];
            next_p = (p >= 0 && p < n_rows) ? p : -1;
            next_w = topk_w ? topk_w[tt * k + lane] : 1.0f;
        }
    };
    load_slot(int64_t(blockIdx.x) * kWarps + warp);
    for (int64_t item = int64_t(blockIdx.x) * kWarps + warp; item < items; item += step) {
        const int32_t my_p = next_p;
        const float my_w = next_w;
        load_slot(item + step);
        const int64_t t = item >> lp;
        const int64_t vb = (item & (P - 1)) * chunk, ve = min64(vb + chunk, nvec);
        if (vb >= ve) continue;
        int32_t pj[KMAX];
        float wj[KMAX];
        int nv = 0;
        int32_t p0 = 0;
        float w0 = 0.0f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            const int32_t pv = __shfl_sync(kFull, my_p, j);
            const float wv = __shfl_sync(kFull, my_w, j);
            pj[j] = j < k ? pv : -1;
            wj[j] = j < k ? wv : 0.0f;
            if (pj[j] >= 0 && nv++ == 0) { p0 = pj[j]; w0 = wj[j]; }
        }
        if (nv <= 1) {
            combine_single(y, nvec, vb, ve, lane, nv > 0, int64_t(p0), w0, out + t * nvec);
            continue;
        }
        for (int64_t v = vb + lane; v < ve; v += 32) {
            uint4 d[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                d[j] = pj[j] >= 0 ? __ldcs(y + int64_t(pj[j]) * nvec + v) : make_uint4(0, 0, 0, 0);
            __stcs(out + t * nvec + v, combine_vector<KMAX, PLAIN>(d, pj, wj, k, cbound, dd_bound));
        }
    }
}

// k <= 8 with a token's slot rows together at most kCbStageMax bytes (the
// layer, mid and virtual-EP shapes): one CTA of 8 warps per token at a time.
// Lanes 0..k-1 of warp 0 each bulk-copy one whole slot row (cp.async.bulk,
// a few KB contiguous, so HBM sees long runs instead of 512-byte pieces of
// scattered rows) into a ring stage; every thread then takes 16-byte columns
// of the token from shared memory through the same column arithmetic as the
// register kernel and writes the output row.  The ring holds kCbStages
// tokens, so the next tokens' rows stream in while one is combined.
constexpr int kCbStages = 3;
constexpr int kCbStageMax = 32768;
constexpr int kCbThreads = 256;

template <int KMAX, bool PLAIN>
__global__ void __launch_bounds__(kCbThreads)
combine_bf16_bulk_kernel(const uint8_t* __restrict__ y, int64_t T, int64_t nvec, int k,
                         int64_t n_rows, const int32_t* __restrict__ slot_pos,
                         const float* __restrict__ topk_w, uint4* __restrict__ out, float cbound,
                         float dd_bound, uint32_t* __restrict__ status) {
    extern __shared__ __align__(128) uint8_t cb_smem[];         // [kCbStages][KMAX][row]
    __shared__ __align__(8) uint64_t full_bar[kCbStages];
    __shared__ int32_t s_pos[kCbStages][KMAX];
    __shared__ float s_w[kCbStages][KMAX];
    __shared__ int s_failed;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t row_bytes = uint32_t(nvec) * 16u;
    const int64_t first = blockIdx.x;
    const int64_t my = first < T ? (T - first + gridDim.x - 1) / gridDim.x : 0;
    const uint32_t smem0 = smem_addr(cb_smem);
    if (tid == 0) {
        for (int s = 0; s < kCbStages; ++s) mbar_init(smem_addr(&full_bar[s]), 1);
        mbar_fence_init();
        s_failed = 0;
    }
    __syncthreads();
    // warp 0: slot rows and weights of token q into stage q % kCbStages
    auto issue = [&](int64_t q) {
        const int64_t t = first + q * int64_t(gridDim.x);
        const int st = int(q % kCbStages);
        int32_t p = -1;
        if (lane < k) {
            p = slot_pos[t * k + lane];
            if (p < 0 || p >= n_rows) p = -1;
            s_pos[st][lane] = p;
            s_w[st][lane] = PLAIN ? 1.0f : topk_w[t * k + lane];
        }
        const uint32_t live = __ballot_sync(0xFFFFFFFFu, p >= 0);
        const uint32_t bar = smem_addr(&full_bar[st]);
        if (lane == 0) mbar_expect_tx(bar, uint32_t(__popc(live)) * row_bytes);
        __syncwarp();
        if (p >= 0)
            bulk_load(smem0 + (uint32_t(st) * KMAX + uint32_t(lane)) * row_bytes,
                      y + int64_t(p) * row_bytes, row_bytes, bar);
    };
    if (warp == 0)
        for (int64_t q = 0; q < my && q < kCbStages; ++q) issue(q);
    int64_t q_fail = -1;
    for (int64_t q = 0; q < my; ++q) {
        const int64_t t = first + q * int64_t(gridDim.x);
        const int st = int(q % kCbStages);
        if (!mbar_wait(smem_addr(&full_bar[st]), uint32_t(q / kCbStages) & 1u)) s_failed = 1;
        __syncthreads();
        if (s_failed) {
            q_fail = q;
            break;
        }
        int32_t pj[KMAX];
        float wj[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            pj[j] = j < k ? s_pos[st][j] : -1;
            wj[j] = j < k ? s_w[st][j] : 0.0f;
        }
        const uint4* stage = reinterpret_cast<const uint4*>(cb_smem + size_t(st) * KMAX * row_bytes);
        for (int64_t v = tid; v < nvec; v += kCbThreads) {
            uint4 d[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                d[j] = pj[j] >= 0 ? stage[j * nvec + v] : make_uint4(0, 0, 0, 0);
            __stcs(out + t * nvec + v, combine_vector<KMAX, PLAIN>(d, pj, wj, k, cbound, dd_bound));
        }
        __syncthreads();                        // every thread is done with the stage
        if (warp == 0 && q + kCbStages < my) issue(q + kCbStages);
    }
    if (q_fail >= 0 && tid == 0) {
        // rows still landing in the stages of tokens q_fail .. q_fail + stages - 1
        for (int64_t i = q_fail; i < my && i < q_fail + kCbStages; ++i)
            mbar_wait(smem_addr(&full_bar[i % kCbStages]), uint32_t(i / kCbStages) & 1u);
        if (status) atomicExch(status, uint32_t(MOE_ERR_TIMEOUT));
    }
}

__global__ void __launch_bounds__(kThreads)
combine_bf16_vec_kernel(const uint4* __restrict__ y, int64_t T, int64_t nvec, int k, int64_t n_rows,
                        const int32_t* __restrict__ slot_pos, const float* __restrict__ topk_w,
                        uint4* __restrict__ out, float cbound) {
    __shared__ int32_t s_pos[kWarps][kMaxTopK];
    __shared__ float s_w[kWarps][kMaxTopK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t H = nvec * 8;
    for (int64_t t = int64_t(blockIdx.x) * kWarps + warp; t < T;
         t += int64_t(gridDim.x) * kWarps) {
        stage_slots(s_pos[warp], s_w[warp], slot_pos, topk_w, t, k, n_rows, lane);
        for (int64_t v0 = lane; v0 < nvec; v0 += 32 * kU) {
            float s[kU][8], a[kU][8];
#pragma unroll
            for (int u = 0; u < kU; ++u)
#pragma unroll
                for (int i = 0; i < 8; ++i) { s[u][i] = 0.0f; a[u][i] = 0.0f; }
            for (int j0 = 0; j0 < k; j0 += kJ) {
                uint4 d[kJ][kU];
#pragma unroll
                for (int jj = 0; jj < kJ; ++jj) {
                    const int j = j0 + jj;
                    const int32_t p = j < k ? s_pos[warp][j] : -1;
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int64_t v = v0 + 32 * u;
                        d[jj][u] = (p >= 0 && v < nvec) ? __ldcs(y + int64_t(p) * nvec + v)
                                                        : make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int jj = 0; jj < kJ; ++jj) {
                    const int j = j0 + jj;
                    if (j >= k || s_pos[warp][j] < 0) continue;
                    const float w = s_w[warp][j];
                    const float aw = fabsf(w);
#pragma unroll
                    for (int u = 0; u < kU; ++u)
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float yv = unpack_bf16(d[jj][u], i);
                            s[u][i] = __fmaf_rn(w, yv, s[u][i]);
                            a[u][i] = __fmaf_rn(aw, fabsf(yv), a[u][i]);
                        }
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t v = v0 + 32 * u;
                if (v >= nvec) continue;
                uint4 res;
                uint32_t open = 0;           // bit q: word q not certified
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float lo0, hi0, lo1, hi1;
                    certify_interval(s[u][2 * q], a[u][2 * q], cbound, k, lo0, hi0);
                    certify_interval(s[u][2 * q + 1], a[u][2 * q + 1], cbound, k, lo1, hi1);
                    const uint32_t lo = pack_bf16x2_rn(lo0, lo1);
                    const uint32_t hi = pack_bf16x2_rn(hi0, hi1);
                    set_word(res, q, lo);
                    if (lo != hi) open |= 1u << q;
                }
                if (open) {
                    const uint16_t* yb = reinterpret_cast<const uint16_t*>(y);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (!(open & (1u << q))) continue;
                        const int64_t h = v * 8 + 2 * q;
                        const uint32_t e0 = combine_elem_f64_bf16(yb, H, h, s_pos[warp], s_w[warp], k);
                        const uint32_t e1 = combine_elem_f64_bf16(yb, H, h + 1, s_pos[warp], s_w[warp], k);
                        set_word(res, q, e0 | (e1 << 16));
                    }
                }
                __stcs(out + t * nvec + v, res);
            }
        }
        __syncwarp();
    }
}

// ---------------------------------------------- combine, element-wise paths
// float32 rows (any alignment) and bf16 rows that are not 16-byte multiples:
// the double slot-order sum, rounded once.
template <typename E>
__global__ void __launch_bounds__(kThreads)
combine_elem_kernel(const E* __restrict__ y, int64_t T, int64_t H, int k, int64_t n_rows,
                    const int32_t* __restrict__ slot_pos, const float* __restrict__ topk_w,
                    E* __restrict__ out) {
    __shared__ int32_t s_pos[kWarps][kMaxTopK];
    __shared__ float s_w[kWarps][kMaxTopK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t t = int64_t(blockIdx.x) * kWarps + warp; t < T;
         t += int64_t(gridDim.x) * kWarps) {
        stage_slots(s_pos[warp], s_w[warp], slot_pos, topk_w, t, k, n_rows, lane);
        for (int64_t h = lane; h < H; h += 32) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                const int32_t p = s_pos[warp][j];
                if (p < 0) continue;
                double yv;
                if constexpr (sizeof(E) == 4) yv = double(y[int64_t(p) * H + h]);
                else yv = double(bf16_to_f32(y[int64_t(p) * H + h]));
                acc = fma(double(s_w[warp][j]), yv, acc);
            }
            if constexpr (sizeof(E) == 4) out[t * H + h] = f64_to_f32_rn(acc);
            else out[t * H + h] = f64_to_bf16_rn(acc);
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------- backward

// Double-float accumulate: (hi, lo) += q.
__device__ __forceinline__ void dd_add1(float& hi, float& lo, float q) {
    float s, e;
    two_sum(hi, q, s, e);
    hi = s;
    lo = __fadd_rn(lo, e);
}

// Butterfly sum of a double-float over the warp; every lane ends with the
// same bits (TwoSum's error term does not depend on operand order).
__device__ __forceinline__ void dd_warp_sum_pair(float& hi, float& lo) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float h2 = __shfl_xor_sync(kFull, hi, off);
        const float l2 = __shfl_xor_sync(kFull, lo, off);
        float s, e;
        two_sum(hi, h2, s, e);
        e = __fadd_rn(e, __fadd_rn(lo, l2));
        hi = __fadd_rn(s, e);
        lo = __fsub_rn(e, __fsub_rn(hi, s));
    }
}

__device__ __forceinline__ float dd_warp_sum(float hi, float lo) {
    dd_warp_sum_pair(hi, lo);
    return __fadd_rn(hi, lo);
}

// Double-float partial sums of a dot product, one per column part of the row,
// added in part order (fixed, so the result is deterministic).
__device__ __forceinline__ float dd_parts_sum(const float (*part)[8][2], int nparts, int j) {
    float hi = part[0][j][0], lo = part[0][j][1];
    for (int q = 1; q < nparts; ++q) {
        float s, e;
        two_sum(hi, part[q][j][0], s, e);
        e = __fadd_rn(e, __fadd_rn(lo, part[q][j][1]));
        hi = __fadd_rn(s, e);
        lo = __fsub_rn(e, __fsub_rn(hi, s));
    }
    return __fadd_rn(hi, lo);
}

// the P warps that hold the column parts of one token (named barrier 1 + warp / P)
__device__ __forceinline__ void parts_sync(int warp, int nparts) {
    asm volatile("bar.sync %0, %1;" :: "r"(1 + warp / nparts), "r"(32 * nparts) : "memory");
}


// k <= 8: one 16-byte column per lane step; the k slot rows and grad_out of
// a step are fetched kBwdStages - 1 steps ahead into a per-warp shared-memory
// ring with cp.async (16-byte LDGSTS), so the loads in flight do not occupy
// registers.  Two CTAs per SM (at most 128 registers a thread).
template <int KMAX>
constexpr size_t bwd_ring_bytes() { return size_t(kWarps) * kBwdStages * (KMAX + 1) * 32 * 16; }
template <int KMAX>
__global__ void __launch_bounds__(kThreads, 2)
combine_bwd_bf16_vec_kernel(const uint4* __restrict__ gout, const uint4* __restrict__ y,
                            int64_t T, int64_t nvec, int k, int64_t n_rows,
                            const int32_t* __restrict__ slot_pos,
                            const float* __restrict__ topk_w, uint4* __restrict__ gy,
                            float* __restrict__ grad_probs, int parts) {
    static_assert(KMAX <= 8, "packed accumulators for up to 8 slots");
    extern __shared__ uint4 bwd_ring[];               // [kWarps][kBwdStages][KMAX + 1][32]
    __shared__ int32_t s_pos[kWarps][kMaxTopK];
    __shared__ float s_w[kWarps][kMaxTopK];
    __shared__ float s_part[kWarps][8][2];            // per-warp partial dots (parts > 1)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint4* ring = bwd_ring + warp * kBwdStages * (KMAX + 1) * 32;
    // work item = (token, column part), as in the forward combine (eight-slot
    // rows only).  parts divides the block's warps and every stride of the
    // item loop, so the parts of one token are warps part_base..part_base+P-1
    // of one block in the same round; each leaves its partial dot products in
    // s_part and the first of them adds them up in part order.  Every warp of
    // such a group takes the same branches (the token and its slots are
    // shared), so the group barriers always meet.
    const int P = KMAX >= 8 ? parts : 1;
    const int64_t chunk = ((nvec + P - 1) / P + 31) / 32 * 32;
    const int part_base = (warp / P) * P;
    for (int64_t item = int64_t(blockIdx.x) * kWarps + warp; item < T * P;
         item += int64_t(gridDim.x) * kWarps) {
        const int64_t t = item / P;
        const int part = int(item - t * P);
        const int64_t vb = part * chunk, ve = min64(vb + chunk, nvec);
        stage_slots(s_pos[warp], s_w[warp], slot_pos, topk_w, t, k, n_rows, lane);
        int32_t pj[KMAX];
        f2_t wj[KMAX], hi[KMAX], lo[KMAX];
        int nv = 0, j0 = 0;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            pj[j] = j < k ? s_pos[warp][j] : -1;
            if (pj[j] >= 0 && nv++ == 0) j0 = j;
            const float w = j < k ? s_w[warp][j] : 0.0f;
            wj[j] = f2_pack(w, w);
            hi[j] = 0ull;
            lo[j] = 0ull;
        }
        if (nv == 0) {              // every slot empty or dropped: nothing reads grad_out
            if (part == 0 && lane < k) grad_probs[t * k + lane] = 0.0f;
            __syncwarp();
            continue;
        }
        if (nv == 1) {
            // one live slot: the same per-lane accumulation order, 4 column
            // vectors in flight per lane instead of one row pair per step
            const int64_t p = s_pos[warp][j0];
            const float w = s_w[warp][j0];
            const f2_t w2 = f2_pack(w, w);
            f2_t h1 = 0ull, l1 = 0ull;
            for (int64_t v0 = vb + lane; v0 < ve; v0 += 32 * 4) {
                uint4 gv[4], yv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t v = v0 + 32 * u;
                    const bool in = v < ve;
                    gv[u] = in ? __ldcs(gout + t * nvec + v) : make_uint4(0, 0, 0, 0);
                    yv[u] = in ? __ldcs(y + p * nvec + v) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t v = v0 + 32 * u;
                    if (v >= ve) break;
                    const f2_t g0 = f2_from_bf16x2(gv[u].x), g1 = f2_from_bf16x2(gv[u].y);
                    const f2_t g2 = f2_from_bf16x2(gv[u].z), g3 = f2_from_bf16x2(gv[u].w);
                    uint4 r;
                    r.x = scale_pair_bf16_f2(w2, g0);
                    r.y = scale_pair_bf16_f2(w2, g1);
                    r.z = scale_pair_bf16_f2(w2, g2);
                    r.w = scale_pair_bf16_f2(w2, g3);
                    __stcs(gy + p * nvec + v, r);
                    f2_two_sum_acc(h1, l1, f2_mul(g0, f2_from_bf16x2(yv[u].x)));
                    f2_two_sum_acc(h1, l1, f2_mul(g1, f2_from_bf16x2(yv[u].y)));
                    f2_two_sum_acc(h1, l1, f2_mul(g2, f2_from_bf16x2(yv[u].z)));
                    f2_two_sum_acc(h1, l1, f2_mul(g3, f2_from_bf16x2(yv[u].w)));
                }
            }
            float a0, a1, b0, b1;
            f2_unpack(h1, a0, a1);
            f2_unpack(l1, b0, b1);
            float s1, e1;
            two_sum(a0, a1, s1, e1);
            e1 = __fadd_rn(e1, __fadd_rn(b0, b1));
            dd_warp_sum_pair(s1, e1);
            if (P == 1) {
                const float r = __fadd_rn(s1, e1);
                if (lane < k) grad_probs[t * k + lane] = lane == j0 ? r : 0.0f;
            } else {
                if (lane == 0) {
                    s_part[warp][0][0] = s1;
                    s_part[warp][0][1] = e1;
                }
                parts_sync(warp, P);
                if (part == 0 && lane < k) {
                    const float r = dd_parts_sum(&s_part[part_base], P, 0);
                    grad_probs[t * k + lane] = lane == j0 ? r : 0.0f;
                }
                parts_sync(warp, P);
            }
            __syncwarp();
            continue;
        }
        // software pipeline over this lane's column steps: the loads of step
        // i + kBwdStages - 1 go to the warp's shared-memory ring (cp.async)
        // while step i is computed, so the bytes in flight live in shared
        // memory, not registers; each lane reads back only its own copies
        const int64_t nsteps = ve > vb ? (ve - vb + 31) / 32 : 0;
        auto issue = [&](int64_t i) {
            const int64_t v = vb + lane + 32 * i;
            if (i < nsteps && v < ve) {
                uint4* st = ring + (i % kBwdStages) * (KMAX + 1) * 32;
#pragma unroll
                for (int j = 0; j < KMAX; ++j)
                    if (pj[j] >= 0) cp_async16(st + j * 32 + lane, y + int64_t(pj[j]) * nvec + v);
                cp_async16(st + KMAX * 32 + lane, gout + t * nvec + v);
            }
            cp_async_commit();
        };
#pragma unroll
        for (int i = 0; i < kBwdStages - 1; ++i) issue(i);
        for (int64_t i = 0; i < nsteps; ++i) {
            issue(i + kBwdStages - 1);
            cp_async_wait<kBwdStages - 1>();               // step i has landed
            const int64_t v = vb + lane + 32 * i;
            if (v >= ve) continue;
            const uint4* st = ring + (i % kBwdStages) * (KMAX + 1) * 32;
            const uint4 gv = st[KMAX * 32 + lane];
            uint4 yv[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                yv[j] = pj[j] >= 0 ? st[j * 32 + lane] : make_uint4(0, 0, 0, 0);
            const f2_t g0 = f2_from_bf16x2(gv.x), g1 = f2_from_bf16x2(gv.y);
            const f2_t g2 = f2_from_bf16x2(gv.z), g3 = f2_from_bf16x2(gv.w);
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (pj[j] < 0) continue;
                uint4 r;
                r.x = scale_pair_bf16_f2(wj[j], g0);
                r.y = scale_pair_bf16_f2(wj[j], g1);
                r.z = scale_pair_bf16_f2(wj[j], g2);
                r.w = scale_pair_bf16_f2(wj[j], g3);
                __stcs(gy + int64_t(pj[j]) * nvec + v, r);
                // bf16 x bf16 products have 16 significant bits: exact in float
                f2_two_sum_acc(hi[j], lo[j], f2_mul(g0, f2_from_bf16x2(yv[j].x)));
                f2_two_sum_acc(hi[j], lo[j], f2_mul(g1, f2_from_bf16x2(yv[j].y)));
                f2_two_sum_acc(hi[j], lo[j], f2_mul(g2, f2_from_bf16x2(yv[j].z)));
                f2_two_sum_acc(hi[j], lo[j], f2_mul(g3, f2_from_bf16x2(yv[j].w)));
            }
        }
        cp_async_wait<0>();
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j >= k) break;
            float h0, h1, l0, l1;
            f2_unpack(hi[j], h0, h1);
            f2_unpack(lo[j], l0, l1);
            float s, e;
            two_sum(h0, h1, s, e);                     // fold the odd lane into the even one
            e = __fadd_rn(e, __fadd_rn(l0, l1));
            dd_warp_sum_pair(s, e);
            if (P == 1) {
                if (lane == 0) grad_probs[t * k + j] = pj[j] >= 0 ? __fadd_rn(s, e) : 0.0f;
            } else if (lane == 0) {
                s_part[warp][j][0] = s;
                s_part[warp][j][1] = e;
            }
        }
        if (P > 1) {
            parts_sync(warp, P);
            if (part == 0 && lane < k)
                grad_probs[t * k + lane] =
                    s_pos[warp][lane] >= 0 ? dd_parts_sum(&s_part[part_base], P, lane) : 0.0f;
            parts_sync(warp, P);
        }
        __syncwarp();
    }
}

// Element-wise backward (float32 rows, or bf16 rows that are not 16-byte
// multiples): same arithmetic, one element per lane step.
template <typename E, int KMAX>
__global__ void __launch_bounds__(kThreads)
combine_bwd_elem_kernel(const E* __restrict__ gout, const E* __restrict__ y, int64_t T,
                        int64_t H, int k, int64_t n_rows, const int32_t* __restrict__ slot_pos,
                        const float* __restrict__ topk_w, E* __restrict__ gy,
                        float* __restrict__ grad_probs) {
    __shared__ int32_t s_pos[kWarps][kMaxTopK];
    __shared__ float s_w[kWarps][kMaxTopK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t t = int64_t(blockIdx.x) * kWarps + warp; t < T;
         t += int64_t(gridDim.x) * kWarps) {
        stage_slots(s_pos[warp], s_w[warp], slot_pos, topk_w, t, k, n_rows, lane);
        float hi[KMAX], lo[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) { hi[j] = 0.0f; lo[j] = 0.0f; }
        for (int64_t h = lane; h < H; h += 32) {
            float g;
            if constexpr (sizeof(E) == 4) g = gout[t * H + h];
            else g = bf16_to_f32(gout[t * H + h]);
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (j >= k) break;
                const int32_t p = s_pos[warp][j];
                if (p < 0) continue;
                const float w = s_w[warp][j];
                const int64_t at = int64_t(p) * H + h;
                float yv;
                if constexpr (sizeof(E) == 4) {
                    yv = y[at];
                    gy[at] = __fmul_rn(w, g);
                    const float q = __fmul_rn(g, yv);
                    const float eq = __fmaf_rn(g, yv, -q);     // exact product = q + eq
                    dd_add1(hi[j], lo[j], q);
                    lo[j] = __fadd_rn(lo[j], eq);
                } else {
                    yv = bf16_to_f32(y[at]);
                    gy[at] = uint16_t(mul_bf16_rn(w, g));
                    dd_add1(hi[j], lo[j], __fmul_rn(g, yv));
                }
            }
        }
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j >= k) break;
            const float r = dd_warp_sum(hi[j], lo[j]);
            if (lane == 0) grad_probs[t * k + j] = s_pos[warp][j] >= 0 ? r : 0.0f;
        }
        __syncwarp();
    }
}

moe_status_t check_common(const void* a, const void* b, moe_dtype_t dtype, int64_t T, int64_t H,
                          int k, int64_t n_rows, const int32_t* slot_pos) {
    if (!dtype_ok(dtype) || T < 0 || H < 0 || k < 1 || n_rows < 0) return MOE_ERR_INVALID_ARG;
    if (k > kMaxTopK || T * int64_t(k) >= (int64_t(1) << 31) || n_rows >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!slot_pos || (H > 0 && (!a || !b)))) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

template <int KMAX>
moe_status_t launch_bwd(const void* gout, const void* y, moe_dtype_t dtype, int64_t T, int64_t H, int k,
                int64_t n_rows, const int32_t* slot_pos, const float* topk_w, void* gy, float* gp,
                bool vec, cudaStream_t s) {
    const int64_t want = (T + kWarps - 1) / kWarps;
    if (vec && KMAX <= 8) {
        constexpr int KV = KMAX <= 8 ? KMAX : 8;
        const auto kern = combine_bwd_bf16_vec_kernel<KV>;
        constexpr size_t smem = bwd_ring_bytes<KV>();
        if (!opt_in_smem((const void*)kern, int(smem))) return MOE_ERR_CUDA;
        const int parts = KV >= 8 ? column_parts_bwd(H / 8) : 1;
        const int64_t want_p = (T * parts + kWarps - 1) / kWarps;
        kern<<<grid_for((const void*)kern, kThreads, smem, want_p), kThreads, smem, s>>>(
            static_cast<const uint4*>(gout), static_cast<const uint4*>(y), T, H / 8, k, n_rows,
            slot_pos, topk_w, static_cast<uint4*>(gy), gp, parts);
    } else if (dtype == MOE_F32) {
        const auto kern = combine_bwd_elem_kernel<float, KMAX>;
        kern<<<grid_for((const void*)kern, kThreads, want), kThreads, 0, s>>>(
            static_cast<const float*>(gout), static_cast<const float*>(y), T, H, k, n_rows,
            slot_pos, topk_w, static_cast<float*>(gy), gp);
    } else {
        const auto kern = combine_bwd_elem_kernel<uint16_t, KMAX>;
        kern<<<grid_for((const void*)kern, kThreads, want), kThreads, 0, s>>>(
            static_cast<const uint16_t*>(gout), static_cast<const uint16_t*>(y), T, H, k, n_rows,
            slot_pos, topk_w, static_cast<uint16_t*>(gy), gp);
    }
    return launch_status();
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_combine(const void* expert_out, moe_dtype_t dtype, int64_t T,
                                    int64_t H, int k, int64_t n_rows, const int32_t* slot_pos,
                                    const float* topk_w, void* out, void* stream) {
    MOE_TRACE(__func__);
    const moe_status_t st = check_common(expert_out, out, dtype, T, H, k, n_rows, slot_pos);
    if (st != MOE_OK) return st;
    if (T == 0 || H == 0) return MOE_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t want = (T + kWarps - 1) / kWarps;
    const size_t row = size_t(H) * elem_size(dtype);
    if (dtype == MOE_BF16 && row % 16 == 0 && aligned16(expert_out) && aligned16(out)) {
        const uint4* yv = static_cast<const uint4*>(expert_out);
        uint4* ov = static_cast<uint4*>(out);
        const float cb = combine_bound_factor(k);
        const bool plain = topk_w == nullptr;
        const size_t stage_bytes = size_t(k <= 2 ? 2 : k <= 4 ? 4 : k <= 6 ? 6 : 8) * row;
        // the staged kernel wins on rows of at most two slots (mid shape: 63.6 ->
        // 42.1 us); at six slots of 4 KB rows the register kernel is faster
        // (32 vs 41 us), so wider slot counts keep it
        if (k >= 2 && k <= 4 && stage_bytes <= size_t(kCbStageMax)) {
            const auto kern =
                k <= 2 ? (plain ? combine_bf16_bulk_kernel<2, true> : combine_bf16_bulk_kernel<2, false>)
                : k <= 4 ? (plain ? combine_bf16_bulk_kernel<4, true> : combine_bf16_bulk_kernel<4, false>)
                : k <= 6 ? (plain ? combine_bf16_bulk_kernel<6, true> : combine_bf16_bulk_kernel<6, false>)
                         : (plain ? combine_bf16_bulk_kernel<8, true> : combine_bf16_bulk_kernel<8, false>);
            const size_t smem = kCbStages * stage_bytes;
            if (!opt_in_smem((const void*)kern, int(kCbStages * kCbStageMax))) return MOE_ERR_CUDA;
            kern<<<grid_for((const void*)kern, kCbThreads, smem, T), kCbThreads, smem, s>>>(
                static_cast<const uint8_t*>(expert_out), T, H / 8, k, n_rows, slot_pos, topk_w, ov,
                cb, dd_bound_factor(k), device_status_word());
        } else if (k <= 8) {
            const auto kern =
                k <= 1 ? (plain ? combine_bf16_regs_kernel<1, true> : combine_bf16_regs_kernel<1, false>)
                : k <= 2 ? (plain ? combine_bf16_regs_kernel<2, true> : combine_bf16_regs_kernel<2, false>)
                : k <= 4 ? (plain ? combine_bf16_regs_kernel<4, true> : combine_bf16_regs_kernel<4, false>)
                : k <= 6 ? (plain ? combine_bf16_regs_kernel<6, true> : combine_bf16_regs_kernel<6, false>)
                         : (plain ? combine_bf16_regs_kernel<8, true> : combine_bf16_regs_kernel<8, false>);
            // whole rows up to six slots: at T = 4096, H = 2048, k = 6, 2 or 4
            // column parts measured 29.7 / 30.6 us against 29.6
            const int parts = k > 6 ? column_parts(H / 8) : 1;
            const int64_t want_p = (T * parts + kWarps - 1) / kWarps;
            kern<<<grid_for((const void*)kern, kThreads, want_p), kThreads, 0, s>>>(
                yv, T, H / 8, k, n_rows, slot_pos, topk_w, ov, cb, dd_bound_factor(k), parts);
        } else {
            combine_bf16_vec_kernel<<<grid_for((const void*)combine_bf16_vec_kernel, kThreads, want),
                                      kThreads, 0, s>>>(yv, T, H / 8, k, n_rows, slot_pos, topk_w,
                                                        ov, cb);
        }
    } else if (dtype == MOE_F32) {
        const auto kern = combine_elem_kernel<float>;
        kern<<<grid_for((const void*)kern, kThreads, want), kThreads, 0, s>>>(
            static_cast<const float*>(expert_out), T, H, k, n_rows, slot_pos, topk_w,
            static_cast<float*>(out));
    } else {
        const auto kern = combine_elem_kernel<uint16_t>;
        kern<<<grid_for((const void*)kern, kThreads, want), kThreads, 0, s>>>(
            static_cast<const uint16_t*>(expert_out), T, H, k, n_rows, slot_pos, topk_w,
            static_cast<uint16_t*>(out));
    }
    return launch_status();
}

extern "C" moe_status_t moe_combine_backward(const void* grad_out, const void* expert_out,
                                             moe_dtype_t dtype, int64_t T, int64_t H, int k,
                                             int64_t n_rows, const int32_t* slot_pos,
                                             const float* topk_w, void* grad_expert_out,
                                             float* grad_probs, void* stream) {
    MOE_TRACE(__func__);
    moe_status_t st = check_common(grad_out, expert_out, dtype, T, H, k, n_rows, slot_pos);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    if (!grad_probs || (H > 0 && !grad_expert_out)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t row = size_t(H) * elem_size(dtype);
    const bool vec = dtype == MOE_BF16 && row % 16 == 0 && aligned16(grad_out) &&
                     aligned16(expert_out) && aligned16(grad_expert_out);
    if (k <= 1) return launch_bwd<1>(grad_out, expert_out, dtype, T, H, k, n_rows, slot_pos, topk_w, grad_expert_out, grad_probs, vec, s);
    else if (k <= 2) return launch_bwd<2>(grad_out, expert_out, dtype, T, H, k, n_rows, slot_pos, topk_w, grad_expert_out, grad_probs, vec, s);
    else if (k <= 4) return launch_bwd<4>(grad_out, expert_out, dtype, T, H, k, n_rows, slot_pos, topk_w, grad_expert_out, grad_probs, vec, s);
    else if (k <= 8) return launch_bwd<8>(grad_out, expert_out, dtype, T, H, k, n_rows, slot_pos, topk_w, grad_expert_out, grad_probs, vec, s);
    else if (k <= 16) return launch_bwd<16>(grad_out, expert_out, dtype, T, H, k, n_rows, slot_pos, topk_w, grad_expert_out, grad_probs, vec, s);
    return launch_bwd<32>(grad_out, expert_out, dtype, T, H, k, n_rows, slot_pos, topk_w, grad_expert_out, grad_probs, vec, s);
}
