// grouped_swiglu.cu -- moe_grouped_swiglu_pack, moe_grouped_swiglu,
// moe_grouped_swiglu_fp8, and the training path (save, dgrad, wgrad).
//
// The expert FFN of "从零理解 MoE 算子" §8 over expert-contiguous rows
// (group_list segments, §7): GMM1 (x @ w_up[e], [n,2I]) -> hidden =
// silu(gate) * up (gate = first I columns, up = last I) -> GMM2 (hidden @
// w_down[e], [n,H]).
//
// Tensor-core path for sm_103a: each CTA owns one SM (persistent), tiles of
// 128 rows x 256 columns, fp32 accumulators in tensor memory.
//   warp 0       TMA producer: 128x64 A and 256x64 B bf16 tiles (128-byte
//                swizzle) into a 4-stage shared-memory ring
//   warp 1       one thread issues tcgen05.mma (M=128, N=256, K=16) and
//                tcgen05.commit to release ring stages / publish the tile
//   warp 2       allocates / frees 512 tensor-memory columns: two 256-column
//                accumulators, so the MMAs of the next tile run while the
//                epilogue drains the previous one
//   warps 4..7   epilogue: tcgen05.ld of their 32-lane quadrant, SwiGLU (GMM1)
//                or conversion (GMM2), bf16 stores, rows past the expert's
//                segment masked
//   warps 8..15  (moe_grouped_swiglu_fp8's GMM1 only) turn each stage's e4m3
//                codes and block scales into the bf16 A tile before the MMA
//                issuer may use it
// Both operands are K-major: moe_grouped_swiglu_pack lays the weights out
// once as w_up_packed [E, 2I, H] (rows in 128-blocks [gate j0..j0+127 | up
// j0..j0+127], so one 256-column tile holds matching gate and up columns) and
// w_down_packed [E, H, I].  The tile schedule is built on the device from
// offsets (no host synchronisation): experts in order, within an expert the
// N tiles, within those the M tiles, so the CTAs running at once share an
// expert's weights through L2.
// Every wait on an mbarrier is bounded; a wait that gives up records
// MOE_ERR_TIMEOUT in the workspace status word and the kernel winds down.
#include "pipeline.cuh"

namespace moe {
namespace {

constexpr int BM = 128;             // rows per tile (TMEM lanes)
constexpr int BN = 256;             // columns per tile (TMEM columns)
constexpr int BK = 64;              // K per stage: one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kThreads = 256;
constexpr int kConvWarps = 8;       // converter warps of the e4m3-A kernel (2 a row)
constexpr int kThreadsA8 = kThreads + 32 * kConvWarps;
constexpr int kConvPerRow = 32 * kConvWarps / 128;   // threads sharing one A row
constexpr int kTileABytes = BM * BK * 2;      // 16 KB
constexpr int kTileBBytes = BN * BK * 2;      // 32 KB
constexpr int kStageBytes = kTileABytes + kTileBBytes;
constexpr int kSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack
constexpr int kTmemCols = 2 * BN;              // double-buffered accumulator
constexpr int kTileA8Bytes = BM * BK;          // 8 KB of e4m3 A codes
constexpr int kA8Offset = kTileABytes - kTileA8Bytes;   // where they land in the A slot
constexpr int kScaleBox = 4;                   // scale columns per TMA box (16 bytes)
constexpr int kScaleBytes = BM * kScaleBox * 4;           // a stage's scale box: 2 KB
constexpr int kSmemBytesA8 = kSmemBytes + kStages * kScaleBytes;

// ------------------------------------------------------------- PTX helpers

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor, K-major operand with 128-byte swizzle:
// start address >> 4 in bits 0-13, leading byte offset (unused for swizzled
// K-major; 16 B) in bits 16-29, stride byte offset (1024 B between 8-row
// groups) >> 4 in bits 32-45, descriptor version 1 in bits 46-47, layout
// SWIZZLE_128B (2) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_k128(uint32_t addr) {
    uint64_t d = 0;
    d |= uint64_t((addr >> 4) & 0x3FFFu);
    d |= uint64_t(1) << 16;
    d |= uint64_t(1024 >> 4) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;
    return d;
}

// Instruction descriptor for kind::f16: D f32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) |
                            (uint32_t(BM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
        :: "r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Or-reduction of `v` over the `nthreads` threads (whole warps) that meet at
// named barrier `id`; every one of them gets the result.
__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n"
        " bar.red.or.pred p, %2, %3, q;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(r) : "r"(uint32_t(v)), "r"(id), "r"(nthreads) : "memory");
    return r != 0;
}

// The float value of the e4m3 code in byte k of w by integer arithmetic (the
// hardware conversions through f16 measured about 2 codes per SM cycle,
// several times slower than the tensor cores consume them): the code moved
// to the top byte and shifted right by 4 (arithmetic) leaves the sign in bit
// 31 and exponent:mantissa in bits 26..20; adding (127 - 7) << 23 rebiases a
// normal code's exponent.  Selects take an exponent field of 0 (subnormal:
// 2^-6 (1 + m/8) - 2^-6, exact; a zero keeps its sign) and the NaN codes.
template <int K>
__device__ __forceinline__ float e4m3_to_f32(uint32_t w) {
    const uint32_t t = __byte_perm(w, 0u, (K << 12) | 0x0444);
    const uint32_t a = uint32_t(int32_t(t) >> 4) & 0x87F00000u;
    const uint32_t sign = t & 0x80000000u;
    const float f = (t & 0x78000000u) ? __uint_as_float(a + (120u << 23))
                                      : __fsub_rn(__uint_as_float(a + (121u << 23)),
                                                  __uint_as_float(sign | (121u << 23)));
    const float z = (t & 0x7F000000u) ? f : __uint_as_float(sign);
    return (t & 0x7F000000u) == 0x7F000000u ? __uint_as_float(0x7FC00000u) : z;
}

// bf16 pairs (lo, hi) of bf16(code * sc) for the four e4m3 codes of w, each
// the exact product rounded once to nearest even, with no branch (branches
// here measured several times slower): the four products in packed float
// multiplies, their rounding errors in packed FMAs; a product whose float
// value lies exactly on a bf16 rounding midpoint while the exact product does
// not -- 2% of products, as the block scales amax/448 share 1/7's repeating
// bits -- moves one float ulp toward the exact product, so the packed
// conversion rounds as the exact product would (mul_bf16_rn's rule).
__device__ __forceinline__ uint32_t nudge_off_midpoint(float p, float e) {
    const uint32_t u = __float_as_uint(p);
    const bool tie = (u & 0xFFFFu) == 0x8000u && e != 0.0f;
    const uint32_t toward = ((__float_as_uint(e) ^ u) >> 31) ? 0xFFFFFFFFu : 1u;   // -1 or +1
    return u + (tie ? toward : 0u);
}

__device__ __forceinline__ void e4m3x4_scaled_bf16(uint32_t w, float sc, uint32_t& lo,
                                                   uint32_t& hi) {
    const float f0 = e4m3_to_f32<0>(w), f1 = e4m3_to_f32<1>(w);
    const float f2 = e4m3_to_f32<2>(w), f3 = e4m3_to_f32<3>(w);
    float p0, p1, p2, p3, e0, e1, e2, e3;
    asm("{\n .reg .b64 x, y, s, p, q, np, nq, r, t;\n mov.b64 x, {%8, %9};\n"
        " mov.b64 y, {%10, %11};\n mov.b64 s, {%12, %12};\n"
        " mul.rn.f32x2 p, x, s;\n mul.rn.f32x2 q, y, s;\n"
        " xor.b64 np, p, 0x8000000080000000;\n xor.b64 nq, q, 0x8000000080000000;\n"
        " fma.rn.f32x2 r, x, s, np;\n fma.rn.f32x2 t, y, s, nq;\n"
        " mov.b64 {%0, %1}, p;\n mov.b64 {%2, %3}, q;\n"
        " mov.b64 {%4, %5}, r;\n mov.b64 {%6, %7}, t;\n}"
        : "=f"(p0), "=f"(p1), "=f"(p2), "=f"(p3), "=f"(e0), "=f"(e1), "=f"(e2), "=f"(e3)
        : "f"(f0), "f"(f1), "f"(f2), "f"(f3), "f"(sc));
    lo = pack_bf16x2_rn(__uint_as_float(nudge_off_midpoint(p0, e0)),
                        __uint_as_float(nudge_off_midpoint(p1, e1)));
    hi = pack_bf16x2_rn(__uint_as_float(nudge_off_midpoint(p2, e2)),
                        __uint_as_float(nudge_off_midpoint(p3, e3)));
}

// ------------------------------------------------------------- tile schedule

// Tile t -> (expert e, m tile m, n tile n).  s_tile_start[e] = first tile of
// expert e (prefix of ceil(n_e/BM) * n_tiles), s_tile_start[E] = total.
__device__ __forceinline__ void tile_coords(int t, const int* s_tile_start, const int* s_mt,
                                            int E, int n_tiles, int& e, int& m, int& n) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_tile_start[mid] <= t) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int r = t - s_tile_start[e];
    n = r / s_mt[e];
    m = r % s_mt[e];
}

// Epilogues of the m-grouped GEMM.
enum Epi : int {
    kPlain = 0,       // bf16 store of the accumulator (GMM2, GMM1 backward)
    kSwiglu = 1,      // [gate | up] tile -> silu(gate) * up (GMM1)
    kSwigluSave = 2,  // kSwiglu, and also store gate and up as bf16 for the backward
    kSwigluBwd = 3,   // dh tile -> [d_gate | d_up] at the stored gate / up (GMM2 backward)
};

struct GemmArgs {
    const int32_t* offsets;     // [E+1] row segments
    int64_t n_rows;             // rows of the activation buffers: segments are clamped to it
    int E;
    int K;                      // reduction length
    int n_tiles;                // BN-column tiles per expert
    int64_t w_rows_per_expert;  // rows of the (K-major) weight per expert
    void* out;                  // bf16 [N_rows, out_cols]
    int64_t out_cols;           // columns of out
    int64_t valid_cols;         // accumulator columns that exist (kPlain / kSwigluBwd)
    int64_t I;                  // intermediate size (kSwigluSave / kSwigluBwd)
    const uint16_t* gate_up;    // kSwigluBwd: stored [N_rows, 2I] bf16
    uint16_t* aux_out;          // kSwigluSave: gate_up [N_rows, 2I]
    WsHeader* header;
    const float* a_scales;      // e4m3 A operand: one scale per 128 columns, [N_rows, K/128]
};

// 32 floats -> 4 x 16-byte bf16 stores
__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const float* a) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int i0 = v * 8;
        d[v] = make_uint4(pack_bf16x2_rn(a[i0], a[i0 + 1]), pack_bf16x2_rn(a[i0 + 2], a[i0 + 3]),
                          pack_bf16x2_rn(a[i0 + 4], a[i0 + 5]), pack_bf16x2_rn(a[i0 + 6], a[i0 + 7]));
    }
}

// 32 bf16 held as four 16-byte words -> floats
__device__ __forceinline__ void unpack_bf16x32(const uint4* s, float* a) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const uint4 w = s[v];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            a[v * 8 + 2 * h] = __uint_as_float(ws[h] << 16);
            a[v * 8 + 2 * h + 1] = __uint_as_float(ws[h] & 0xFFFF0000u);
        }
    }
}

// A8: the A operand is e4m3 codes with per-128-column scales (map_a over
// the codes, map_s over the scales).  TMA brings a stage's 128 x 64 codes
// into the upper half of its A slot and the scale columns around its block
// into a small ring; kConvWarps converter warps (kConvPerRow threads an A
// row) read them, meet at a named barrier (the bf16 rows they write overlap
// the codes), write bf16(code * scale) -- the exact product rounded once, as
// moe_dequantize_fp8 -- in the 128-byte-swizzled layout the MMA reads, and
// release the stage to the MMA issuer on conv_bar.
template <int EPI, bool A8 = false>
__global__ void __launch_bounds__(A8 ? kThreadsA8 : kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_b, GemmArgs args,
                    const __grid_constant__ CUtensorMap map_s) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(8) uint64_t conv_bar[kStages];
    __shared__ __align__(8) uint64_t tmem_full_bar[2];
    __shared__ __align__(8) uint64_t tmem_empty_bar[2];
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_tile_start[kMaxExperts + 1];
    __shared__ int s_mt[kMaxExperts];
    __shared__ int s_row0[kMaxExperts + 1];
    __shared__ int s_failed;
    __shared__ int s_bad;

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    float* s_scale = reinterpret_cast<float*>(smem + kStages * kStageBytes);   // A8: [stage][BM][4]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = args.E;

    // schedule from the device-side offsets (single warp scan, E <= 1024);
    // offsets are clamped into [0, n_rows], so no row outside the buffers is
    // ever written, and offsets that needed it are reported
    if (warp == 0) {
        int carry = 0;
        bool bad = false;
        const int nr = int(args.n_rows);
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            int mt = 0;
            if (e < E) {
                const int raw0 = args.offsets[e], raw1 = args.offsets[e + 1];
                bad |= raw0 < 0 || raw1 < raw0 || raw1 > nr;
                const int r0 = min(max(raw0, 0), nr), r1 = min(max(raw1, 0), nr);
                mt = r1 > r0 ? (r1 - r0 + BM - 1) / BM : 0;
                s_mt[e] = mt > 0 ? mt : 1;
                s_row0[e] = r0;
            }
            int incl = mt * args.n_tiles;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
                if (lane >= off) incl += o;
            }
            if (e < E) s_tile_start[e] = carry + incl - mt * args.n_tiles;
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        bad = __any_sync(0xFFFFFFFFu, bad);
        if (lane == 0) {
            s_tile_start[E] = carry;
            s_row0[E] = min(max(args.offsets[E], 0), nr);
            s_failed = 0;
            s_bad = bad;
        }
    }
    if (threadIdx.x == 32) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&full_bar[s]), 1);
            mbar_init(smem_addr(&empty_bar[s]), 1);
            mbar_init(smem_addr(&conv_bar[s]), kConvWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&tmem_full_bar[b]), 1);
            mbar_init(smem_addr(&tmem_empty_bar[b]), 128);
        }
        mbar_fence_init();
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_addr(&s_tmem_base)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const int total_tiles = s_tile_start[E];
    const int k_steps = args.K / BK;
    const uint32_t tmem_base = s_tmem_base;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------ TMA producer
        uint32_t it = 0;
        for (int t = blockIdx.x; t < total_tiles && !s_failed; t += gridDim.x) {
            int e, m, n;
            tile_coords(t, s_tile_start, s_mt, E, args.n_tiles, e, m, n);
            const int row_a = s_row0[e] + m * BM;
            const int row_b = int(e * args.w_rows_per_expert) + n * BN;
            for (int ks = 0; ks < k_steps; ++ks, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1u;
                if (!mbar_wait(smem_addr(&empty_bar[s]), ph ^ 1u)) { s_failed = 1; break; }
                const uint32_t a_dst = smem_addr(smem + s * kStageBytes);
                const uint32_t b_dst = a_dst + kTileABytes;
                const uint32_t fb = smem_addr(&full_bar[s]);
                mbar_expect_tx(fb, A8 ? kTileA8Bytes + kTileBBytes + kScaleBytes : kStageBytes);
                tma_load_2d(A8 ? a_dst + kA8Offset : a_dst, &map_a, ks * BK, row_a, fb);
                tma_load_2d(b_dst, &map_b, ks * BK, row_b, fb);
                if (A8)   // the 4 scale columns around this stage's block (x a multiple of 4)
                    tma_load_2d(smem_addr(s_scale + s * BM * kScaleBox), &map_s,
                                ((ks * BK) / 128) & ~(kScaleBox - 1), row_a, fb);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------ MMA issuer
        uint32_t it = 0, tile_iter = 0;
        for (int t = blockIdx.x; t < total_tiles && !s_failed; t += gridDim.x, ++tile_iter) {
            const uint32_t buf = tile_iter & 1u, use = tile_iter >> 1;
            if (!mbar_wait(smem_addr(&tmem_empty_bar[buf]), (use & 1u) ^ 1u)) { s_failed = 1; break; }
            tc_fence_after();
            const uint32_t tmem_d = tmem_base + buf * BN;
            for (int ks = 0; ks < k_steps; ++ks, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1u;
                // (A8: the converters waited for the TMA of this stage)
                if (!mbar_wait(smem_addr(A8 ? &conv_bar[s] : &full_bar[s]), ph)) {
                    s_failed = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a_base = smem_addr(smem + s * kStageBytes);
                const uint32_t b_base = a_base + kTileABytes;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    // advance 16 bf16 = 32 bytes along K inside the swizzled row
                    mma_bf16(tmem_d, smem_desc_k128(a_base + kk * 32),
                             smem_desc_k128(b_base + kk * 32), (ks | kk) != 0);
                }
                mma_commit(smem_addr(&empty_bar[s]));     // frees the stage when done
            }
            if (s_failed) break;
            mma_commit(smem_addr(&tmem_full_bar[buf]));   // the tile's accumulator is ready
        }
    } else if (A8 && warp >= 8) {
        // ------------------------------------------------------ e4m3 -> bf16
        // kConvPerRow threads a row: thread (r, part) converts columns
        // [part, part + 1) * BK / kConvPerRow of A row r
        const int ct = int(threadIdx.x) - kThreads;
        const int r = ct / kConvPerRow, part = ct % kConvPerRow;
        constexpr int kCodes = BK / kConvPerRow;          // codes a thread converts
        constexpr int kVecs = kCodes / 16;                // 16-byte code vectors
        constexpr int kChunks = kCodes / 8;               // 16-byte bf16 chunks
        uint32_t it = 0;
        bool stop = false;
        for (int t = blockIdx.x; t < total_tiles && !stop; t += gridDim.x) {
            for (int ks = 0; ks < k_steps; ++ks, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1u;
                const bool ok = mbar_wait(smem_addr(&full_bar[s]), ph);
                uint8_t* slot = smem + s * kStageBytes;
                uint4 q[kVecs];
                float sc = 0.0f;
                if (ok) {
                    const uint4* src =
                        reinterpret_cast<const uint4*>(slot + kA8Offset + r * BK + part * kCodes);
#pragma unroll
                    for (int v = 0; v < kVecs; ++v) q[v] = src[v];
                    sc = s_scale[(s * BM + r) * kScaleBox + (((ks * BK) / 128) & (kScaleBox - 1))];
                }
                // every converter has its codes before any bf16 row is
                // written over them; a failure anywhere stops all of them
                stop = bar_red_or(1, 32 * kConvWarps, !ok || s_failed);
                if (stop) break;
                uint8_t* row = slot + r * (BK * 2);
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {       // chunk: 8 columns, 2 code words
                    const uint4 v = q[c >> 1];
                    const uint32_t w0 = (c & 1) ? v.z : v.x, w1 = (c & 1) ? v.w : v.y;
                    uint32_t o0, o1, o2, o3;
                    e4m3x4_scaled_bf16(w0, sc, o0, o1);
                    e4m3x4_scaled_bf16(w1, sc, o2, o3);
                    // 128-byte swizzle: chunk j of row r sits at chunk j ^ (r % 8)
                    const int j = part * kChunks + c;
                    *reinterpret_cast<uint4*>(row + ((j ^ (r & 7)) << 4)) = make_uint4(o0, o1, o2, o3);
                }
                // each thread orders its own writes before the tensor core's
                // reads; the warp's lane 0 then arrives for all 32
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&conv_bar[s]));
            }
        }
        if (stop) s_failed = 1;
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------ epilogue
        const int q = warp - 4;                           // TMEM lane quadrant
        const uint32_t lane_base = uint32_t(q * 32) << 16;
        uint32_t tile_iter = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++tile_iter) {
            const uint32_t buf = tile_iter & 1u, use = tile_iter >> 1;
            int e, m, n;
            tile_coords(t, s_tile_start, s_mt, E, args.n_tiles, e, m, n);
            const int64_t row = int64_t(s_row0[e]) + m * BM + q * 32 + lane;
            const bool row_ok = row < s_row0[e + 1];
            // kSwigluBwd: the first chunk's stored gate/up, fetched while the
            // accumulator is still being computed
            uint4 cg[4], cu[4];
            int nchunks = 0;
            if (EPI == kSwigluBwd) {
                const int64_t left = args.valid_cols - int64_t(n) * BN;
                nchunks = int((left < BN ? left : BN) / 32);
                if (row_ok && nchunks > 0) {
                    const uint4* gp = reinterpret_cast<const uint4*>(
                        args.gate_up + row * 2 * args.I + int64_t(n) * BN);
                    const uint4* up = reinterpret_cast<const uint4*>(
                        args.gate_up + row * 2 * args.I + args.I + int64_t(n) * BN);
#pragma unroll
                    for (int v = 0; v < 4; ++v) { cg[v] = gp[v]; cu[v] = up[v]; }
                }
            }
            if (s_failed || !mbar_wait(smem_addr(&tmem_full_bar[buf]), use & 1u)) {
                s_failed = 1;
                break;
            }
            tc_fence_after();
            const uint32_t tmem_acc = tmem_base + buf * BN;
            uint16_t* out = static_cast<uint16_t*>(args.out);
            if (EPI == kSwiglu || EPI == kSwigluSave) {
                // columns [0,128) gate, [128,256) up, for hidden j0 = n*128
                const int64_t j0 = int64_t(n) * (BN / 2);
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 32) {
                    float g[32], u[32], hv[32];
                    tmem_ld32(tmem_acc + lane_base + c, g);
                    tmem_ld32(tmem_acc + lane_base + BN / 2 + c, u);
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            hv[i] = __fdividef(g[i], 1.0f + __expf(-g[i])) * u[i];
                        store_bf16x32(out + row * args.out_cols + j0 + c, hv);
                        if (EPI == kSwigluSave) {
                            uint16_t* gu = args.aux_out + row * 2 * args.I;
                            store_bf16x32(gu + j0 + c, g);
                            store_bf16x32(gu + args.I + j0 + c, u);
                        }
                    }
                }
            } else if (EPI == kSwigluBwd) {
                // accumulator columns = hidden columns j = n*BN + c (< I):
                // d_up = dh*silu(g), d_gate = dh*u*s*(1 + g*(1-s)), s = sigmoid(g);
                // the stored gate/up of chunk c+1 load while chunk c is computed
#pragma unroll 1
                for (int ci = 0; ci < nchunks; ++ci) {
                    const int c = ci * 32;
                    const int64_t j = int64_t(n) * BN + c;
                    uint4 ng[4], nu[4];
                    if (row_ok && ci + 1 < nchunks) {
                        const uint4* gp = reinterpret_cast<const uint4*>(
                            args.gate_up + row * 2 * args.I + j + 32);
                        const uint4* up = reinterpret_cast<const uint4*>(
                            args.gate_up + row * 2 * args.I + args.I + j + 32);
#pragma unroll
                        for (int v = 0; v < 4; ++v) { ng[v] = gp[v]; nu[v] = up[v]; }
                    }
                    float dh[32];
                    tmem_ld32(tmem_acc + lane_base + c, dh);
                    if (row_ok) {
                        float g[32], u[32], dg[32], du[32];
                        unpack_bf16x32(cg, g);
                        unpack_bf16x32(cu, u);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float sg = __fdividef(1.0f, 1.0f + __expf(-g[i]));
                            du[i] = dh[i] * (g[i] * sg);
                            dg[i] = dh[i] * u[i] * (sg * (1.0f + g[i] * (1.0f - sg)));
                        }
                        uint16_t* o = out + row * 2 * args.I;
                        store_bf16x32(o + j, dg);
                        store_bf16x32(o + args.I + j, du);
                    }
#pragma unroll
                    for (int v = 0; v < 4; ++v) { cg[v] = ng[v]; cu[v] = nu[v]; }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    const int64_t j = int64_t(n) * BN + c;
                    if (j >= args.valid_cols) break;              // uniform over the warp
                    float a[32];
                    tmem_ld32(tmem_acc + lane_base + c, a);
                    if (row_ok) store_bf16x32(out + row * args.out_cols + j, a);
                }
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&tmem_empty_bar[buf]));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (s_failed && threadIdx.x == 0) {
        args.header->status = MOE_ERR_TIMEOUT;
        args.header->detail = blockIdx.x;
    } else if (s_bad && threadIdx.x == 0 && blockIdx.x == 0) {
        atomicCAS(&args.header->status, uint32_t(MOE_OK), uint32_t(MOE_ERR_DEVICE_CHECK));
    }
    if (warp == 2) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem_base), "r"(kTmemCols) : "memory");
    }
}

// ------------------------------------------------------ k-grouped wgrad
// dW[e] = P_e^T Q_e over the rows of expert e's segment: P [N_rows, M] and
// Q [N_rows, Ncols] row-major, dW [E, M, Ncols] fp32.  Both operands are read
// MN-major: a stage holds 64 token rows (the reduction) of a 256-column P
// panel (four 64-column TMA boxes, two per 128-row half of the tile) and a
// 256-column Q panel (four boxes), each box 64 rows x 128 bytes with the
// 128-byte swizzle -- the canonical MN-major
// SW128 layout, 8-row K groups 1024 bytes apart (SBO) and 64-element MN
// blocks one box (8 KB) apart (LBO).  The instruction descriptor marks A and B
// as MN-major.  Rows past the segment's end in its last stage belong to the
// next expert.  One MMA reduces 16 token rows, so the last stage issues MMAs
// only up to the first multiple of 16 at or past the segment's end, and only
// the rows between the end and that multiple (at most 15) must read as zero:
// the producer warp zeroes them in shared memory (whole 128-byte rows, so the
// swizzle does not matter) and publishes the stage on a second barrier.  A
// segment that ends on a 16-row boundary needs no fix-up.  The producer never
// waits on a stage it has issued: while it waits for a free ring slot it
// polls the partial stages in flight and fixes up each one once it lands, so
// the next tile's loads go out as early as they would without a fix-up.  An
// expert with no rows gets zeros.  The epilogue writes each 32x32 fp32 block
// of its quadrant into a 128-byte-swizzled staging tile (kEpiBufs per warp)
// and hands it to the TMA store engine, so the warp moves on to the next
// block while full 128-byte rows stream out.
constexpr int kBoxBytes = 64 * 128;
constexpr int kEpiTileBytes = 32 * 32 * 4;            // one 32x32 fp32 block
// A tile is 256 rows of dW (two 128-row halves with their own TMEM
// accumulators, all 512 columns) x 256 columns: both halves share every Q
// panel, so a stage of 64 token rows (P 256 columns + Q 256 columns = 64 KB)
// feeds twice the MMA work of a 128-row tile, and there are half as many
// tiles (and partial last stages).  The price: one accumulator set, so a
// tile's MMAs wait for the previous tile's epilogue.
constexpr int kWM = 256;                       // dW rows per tile
constexpr int kWStages = 3;
// bound on the producer's non-blocking polls for a free ring slot (each poll
// is at least two shared-memory round trips: well over half a second)
constexpr uint32_t kPollLimit = 1u << 24;
constexpr int kEpiBufs = 2;
constexpr int kWA = kWM / 64;                  // P boxes per stage (2 per half)
constexpr int kWB = BN / 64;                   // Q boxes per stage
constexpr int kWStageBytes = (kWA + kWB) * kBoxBytes;
constexpr int kWgradSmemBytes = kWStages * kWStageBytes + 4 * kEpiBufs * kEpiTileBytes + 1024;
static_assert(kWgradSmemBytes <= 227 * 1024 - 256, "wgrad shared memory");

__device__ __forceinline__ uint64_t smem_desc_mn128(uint32_t addr) {
    uint64_t d = 0;
    d |= uint64_t((addr >> 4) & 0x3FFFu);
    d |= uint64_t(kBoxBytes >> 4) << 16;       // LBO: next 64-element MN block
    d |= uint64_t(1024 >> 4) << 32;            // SBO: next 8-row K group
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;
    return d;
}

constexpr uint32_t kIdescMN = kIdesc | (1u << 15) | (1u << 16);   // A and B MN-major

__device__ __forceinline__ void mma_bf16_mn(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
        :: "r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(kIdescMN), "r"(accumulate) : "memory");
}

struct WgradArgs {
    const int32_t* offsets;
    int64_t n_rows;             // rows of the operands (rows past it read as zeros)
    int E;
    int M, Ncols;               // dW[e] is [M, Ncols]
    int m_tiles, n_tiles;       // ceil(M / kWM), Ncols / BN
    float* out;                 // [E, M, Ncols]
    WsHeader* header;
};

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int c0, int c1, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(src) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
grouped_wgrad_kernel(const __grid_constant__ CUtensorMap map_p,
                     const __grid_constant__ CUtensorMap map_q,
                     const __grid_constant__ CUtensorMap map_out, WgradArgs args) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kWStages];
    __shared__ __align__(8) uint64_t ready_bar[kWStages];
    __shared__ __align__(8) uint64_t empty_bar[kWStages];
    __shared__ __align__(8) uint64_t tmem_full_bar;
    __shared__ __align__(8) uint64_t tmem_empty_bar;
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_failed;
    __shared__ int s_bad;

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 3) {            // offsets outside [0, n_rows] or decreasing are reported
        bool bad = false;
        for (int e = lane; e < args.E; e += 32) {
            const int64_t raw0 = args.offsets[e], raw1 = args.offsets[e + 1];
            bad |= raw0 < 0 || raw1 < raw0 || raw1 > args.n_rows;
        }
        bad = __any_sync(0xFFFFFFFFu, bad);
        if (lane == 0) s_bad = bad;
    }
    if (threadIdx.x == 32) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(smem_addr(&full_bar[s]), 1);
            mbar_init(smem_addr(&ready_bar[s]), 1);
            mbar_init(smem_addr(&empty_bar[s]), 1);
        }
        mbar_init(smem_addr(&tmem_full_bar), 1);
        mbar_init(smem_addr(&tmem_empty_bar), 128);
        mbar_fence_init();
        s_failed = 0;
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_addr(&s_tmem_base)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const int per_expert = args.m_tiles * args.n_tiles;
    const int total_tiles = args.E * per_expert;
    const uint32_t tmem_base = s_tmem_base;
    auto coords = [&](int t, int& e, int& m, int& n) {
        e = t / per_expert;
        const int r = t - e * per_expert;
        n = r / args.m_tiles;
        m = r - n * args.m_tiles;
    };

    if (warp == 0) {
        // ------------------------------------------ TMA producer + tail fix-up
        // Any ring slot may hold a partial stage awaiting its fix-up: bit s of
        // `pend`, with the stage's full-barrier parity and valid-row count in
        // byte s of `pend_info` (parity << 7 | valid, valid < 64).  While it
        // waits for a free slot the warp polls the pending stages and fixes up
        // each one as soon as it lands, so it never parks on a stage it has
        // just issued while later loads could be going out.
        uint32_t it = 0;
        bool failed = false;
        uint32_t pend = 0, pend_info = 0;
        auto poll = [&]() {
            for (int ps = 0; ps < kWStages; ++ps) {
                if (!((pend >> ps) & 1u)) continue;
                const uint32_t info = (pend_info >> (8 * ps)) & 0xFFu;
                bool landed = false;
                if (lane == 0) landed = mbar_test(smem_addr(&full_bar[ps]), info >> 7);
                if (!__shfl_sync(0xFFFFFFFFu, landed, 0)) continue;
                // zero rows [valid, next multiple of 16) of every box: 16-byte chunks
                const int valid = int(info & 63u);
                const int chunks = (((valid + 15) & ~15) - valid) * 8;
                for (int b = 0; b < kWA + kWB; ++b) {
                    uint8_t* box = smem + ps * kWStageBytes + b * kBoxBytes + valid * 128;
                    for (int c = lane; c < chunks; c += 32)
                        *reinterpret_cast<uint4*>(box + c * 16) = make_uint4(0, 0, 0, 0);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&ready_bar[ps]));
                pend &= ~(1u << ps);
            }
        };
        for (int t = blockIdx.x; t < total_tiles && !failed; t += gridDim.x) {
            int e, m, n;
            coords(t, e, m, n);
            const int r0 = args.offsets[e], r1 = args.offsets[e + 1];
            const int ksteps = r1 > r0 ? (r1 - r0 + 63) / 64 : 0;
            for (int ks = 0; ks < ksteps; ++ks, ++it) {
                const int s = it % kWStages;
                const uint32_t ph = (it / kWStages) & 1u;
                // slot s is free once the MMAs of its last stage have completed
                // (that stage, if partial, was fixed up here first)
                bool got = false;
                for (uint32_t i = 0; i < kPollLimit && !got; ++i) {
                    poll();
                    bool ok = false;
                    if (lane == 0) ok = mbar_test(smem_addr(&empty_bar[s]), ph ^ 1u);
                    got = __shfl_sync(0xFFFFFFFFu, ok, 0);
                }
                if (!got) { failed = true; break; }
                const uint32_t base = smem_addr(smem + s * kWStageBytes);
                const uint32_t fb = smem_addr(&full_bar[s]);
                const int row = r0 + ks * 64;
                if (lane == 0) {
                    mbar_expect_tx(fb, kWStageBytes);
                    for (int b = 0; b < kWA; ++b)
                        tma_load_2d(base + b * kBoxBytes, &map_p, m * kWM + b * 64, row, fb);
                    for (int b = 0; b < kWB; ++b)
                        tma_load_2d(base + (kWA + b) * kBoxBytes, &map_q, n * BN + b * 64, row, fb);
                }
                const int valid = min(64, r1 - row);
                if (valid % 16 != 0) {
                    pend |= 1u << s;
                    pend_info = (pend_info & ~(0xFFu << (8 * s))) |
                                (((ph << 7) | uint32_t(valid)) << (8 * s));
                }
            }
        }
        for (uint32_t i = 0; i < kPollLimit && pend && !failed; ++i) poll();
        if (pend) failed = true;
        if (failed && lane == 0) s_failed = 1;
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------ MMA issuer
        uint32_t it = 0, tile_iter = 0, ready_phase = 0;
        for (int t = blockIdx.x; t < total_tiles && !s_failed; t += gridDim.x, ++tile_iter) {
            int e, m, n;
            coords(t, e, m, n);
            const int r0 = args.offsets[e], r1 = args.offsets[e + 1];
            const int ksteps = r1 > r0 ? (r1 - r0 + 63) / 64 : 0;
            // the previous tile's epilogue has drained both accumulators
            if (!mbar_wait(smem_addr(&tmem_empty_bar), (tile_iter & 1u) ^ 1u)) { s_failed = 1; break; }
            tc_fence_after();
            for (int ks = 0; ks < ksteps; ++ks, ++it) {
                const int s = it % kWStages;
                const uint32_t ph = (it / kWStages) & 1u;
                if (!mbar_wait(smem_addr(&full_bar[s]), ph)) { s_failed = 1; break; }
                const int valid = min(64, r1 - (r0 + ks * 64));
                if (valid % 16 != 0) {
                    if (!mbar_wait(smem_addr(&ready_bar[s]), (ready_phase >> s) & 1u)) {
                        s_failed = 1;
                        break;
                    }
                    ready_phase ^= 1u << s;
                }
                tc_fence_after();
                const uint32_t a_base = smem_addr(smem + s * kWStageBytes);
                const uint32_t b_base = a_base + kWA * kBoxBytes;
                const int nk = (valid + 15) / 16;
#pragma unroll
                for (int kk = 0; kk < 64 / 16; ++kk) {    // 16 token rows = 2 K groups
                    if (kk >= nk) break;
                    const uint64_t bdesc = smem_desc_mn128(b_base + kk * 2048);
#pragma unroll
                    for (int h = 0; h < 2; ++h)           // rows [128h, 128h+128) of the tile
                        mma_bf16_mn(tmem_base + h * BN,
                                    smem_desc_mn128(a_base + h * 2 * kBoxBytes + kk * 2048), bdesc,
                                    (ks | kk) != 0);
                }
                mma_commit(smem_addr(&empty_bar[s]));
            }
            if (s_failed) break;
            mma_commit(smem_addr(&tmem_full_bar));
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------ epilogue
        const int q = warp - 4;
        const uint32_t lane_base = uint32_t(q * 32) << 16;
        // kEpiBufs staging tiles for this warp, 1024-byte aligned (128-byte swizzle)
        const uint32_t stage0 = smem_addr(smem + kWStages * kWStageBytes + q * kEpiBufs * kEpiTileBytes);
        uint32_t chunk_iter = 0;
        uint32_t tile_iter = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++tile_iter) {
            if (s_failed || !mbar_wait(smem_addr(&tmem_full_bar), tile_iter & 1u)) {
                s_failed = 1;
                break;
            }
            tc_fence_after();
            int e, m, n;
            coords(t, e, m, n);
            const bool empty = args.offsets[e + 1] <= args.offsets[e];
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const int row_in = m * kWM + h * BM + q * 32;   // this quadrant's first dW row
                if (row_in >= args.M) continue;                // past M (a partial last tile)
                const int out_row = e * args.M + row_in;
                const uint32_t tmem_acc = tmem_base + h * BN;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32, ++chunk_iter) {
                    float a[32];
                    if (!empty) {
                        tmem_ld32(tmem_acc + lane_base + c, a);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) a[i] = 0.0f;
                    }
                    // the store that last used this staging tile has finished reading it
                    if (lane == 0 && chunk_iter >= kEpiBufs) bulk_wait_read<kEpiBufs - 1>();
                    __syncwarp();
                    const uint32_t tile = stage0 + (chunk_iter % kEpiBufs) * kEpiTileBytes;
                    // row `lane`, 16-byte chunk j at j ^ (row % 8): the 128-byte swizzle
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t dst = tile + lane * 128 + ((j ^ (lane & 7)) << 4);
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
                                     :: "r"(dst), "f"(a[4 * j]), "f"(a[4 * j + 1]), "f"(a[4 * j + 2]),
                                        "f"(a[4 * j + 3]) : "memory");
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&map_out, n * BN + c, out_row, tile);
                        bulk_commit();
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&tmem_empty_bar));
        }
        if (lane == 0) bulk_wait_all();                 // every store has landed
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (s_failed && threadIdx.x == 0) {
        args.header->status = MOE_ERR_TIMEOUT;
        args.header->detail = blockIdx.x;
    } else if (s_bad && threadIdx.x == 0 && blockIdx.x == 0) {
        atomicCAS(&args.header->status, uint32_t(MOE_OK), uint32_t(MOE_ERR_DEVICE_CHECK));
    }
    if (warp == 2) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem_base), "r"(kTmemCols) : "memory");
    }
}

__global__ void reset_status_kernel(WsHeader* header) {
    header->status = MOE_OK;
    header->detail = 0;
}

// --------------------------------------------------------------- prepack
// w_up [E,H,2I] -> [E,2I,H] with rows in 128-blocks [gate | up];
// w_down [E,I,H] -> [E,H,I].  32x32 tiles through shared memory.
__global__ void pack_transpose_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                                      int64_t R, int64_t C, int interleave_I) {
    // src [E][R][C] -> dst [E][C'][R] where C' is C with the gate/up
    // interleave applied when interleave_I > 0 (then C = 2I)
    __shared__ uint16_t tile[32][33];
    const int64_t e = blockIdx.z;
    const int64_t r0 = int64_t(blockIdx.y) * 32, c0 = int64_t(blockIdx.x) * 32;
    const uint16_t* s = src + e * R * C;
    uint16_t* d = dst + e * R * C;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int64_t r = r0 + i, c = c0 + threadIdx.x;
        if (r < R && c < C) tile[i][threadIdx.x] = s[r * C + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int64_t c = c0 + i, r = r0 + threadIdx.x;
        if (r < R && c < C) {
            int64_t pr = c;
            if (interleave_I > 0) {
                const int64_t I = interleave_I;
                const int64_t j = c < I ? c : c - I;
                pr = (j / 128) * 256 + (c < I ? 0 : 128) + (j % 128);
            }
            d[pr * R + r] = tile[threadIdx.x][i];
        }
    }
}

// ------------------------------------------------------------ tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2D bf16 map over a row-major [rows, cols] matrix, box [box_rows, 64 cols],
// 128-byte swizzle; reads past the last row return zeros.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
    const cuuint32_t box[2] = {cuuint32_t(BK), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// 2D map over row-major e4m3 codes [rows, cols] (one byte each), box
// [box_rows, 64 codes], no swizzle (the converter warps place the bf16 rows);
// reads past the last row return zeros.
bool make_map_u8(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols)};
    const cuuint32_t box[2] = {cuuint32_t(BK), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// 2D fp32 map over the block scales [rows, cols] of e4m3 rows, box
// [box rows BM, kScaleBox columns] (cols * 4 bytes must be a multiple of 16).
bool make_map_scales(CUtensorMap* map, const float* base, int64_t rows, int64_t cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * 4};
    const cuuint32_t box[2] = {cuuint32_t(kScaleBox), cuuint32_t(BM)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D fp32 map over the row-major [rows, cols] weight-gradient output, box
// 32 x 32 with the 128-byte swizzle of the epilogue's staging tiles.
bool make_out_map(CUtensorMap* map, float* base, int64_t rows, int64_t cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Opt every tensor-core kernel into its dynamic shared memory.
bool smem_attrs_set() {
    const void* kernels[] = {(const void*)grouped_gemm_kernel<kPlain>,
                             (const void*)grouped_gemm_kernel<kSwiglu>,
                             (const void*)grouped_gemm_kernel<kSwigluSave>,
                             (const void*)grouped_gemm_kernel<kSwigluBwd>};
    for (const void* k : kernels)
        if (!opt_in_smem(k, kSmemBytes)) return false;
    if (!opt_in_smem((const void*)grouped_gemm_kernel<kSwiglu, true>, kSmemBytesA8)) return false;
    return opt_in_smem((const void*)grouped_wgrad_kernel, kWgradSmemBytes);
}

// The status header a call resets and its kernels report into.
moe_status_t status_workspace(void* workspace, size_t workspace_bytes, WsHeader** header) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kWsAlign - 1)) ||
        workspace_bytes < kWsAlign)
        return MOE_ERR_WORKSPACE;
    *header = static_cast<WsHeader*>(workspace);
    return MOE_OK;
}

moe_status_t check_shapes(int64_t N, int E, int64_t H, int64_t I) {
    if (N < 0 || E < 1 || H < 1 || I < 1) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || H % BN != 0 || I % 128 != 0 || H % BK != 0 || I % BK != 0)
        return MOE_ERR_UNSUPPORTED;
    if (N >= (int64_t(1) << 31) || int64_t(E) * 2 * I >= (int64_t(1) << 31) ||
        int64_t(E) * H >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_grouped_swiglu_pack(const void* w_up, const void* w_down, int E,
                                                int64_t H, int64_t I, void* w_up_packed,
                                                void* w_down_packed, void* stream) {
    MOE_TRACE(__func__);
    const moe_status_t st = check_shapes(0, E, H, I);
    if (st != MOE_OK) return st;
    if (!w_up || !w_down || !w_up_packed || !w_down_packed) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 block(32, 8);
    const dim3 g_up(unsigned((2 * I + 31) / 32), unsigned((H + 31) / 32), unsigned(E));
    pack_transpose_kernel<<<g_up, block, 0, s>>>(static_cast<const uint16_t*>(w_up),
                                                 static_cast<uint16_t*>(w_up_packed), H, 2 * I,
                                                 int(I));
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    const dim3 g_down(unsigned((H + 31) / 32), unsigned((I + 31) / 32), unsigned(E));
    pack_transpose_kernel<<<g_down, block, 0, s>>>(static_cast<const uint16_t*>(w_down),
                                                   static_cast<uint16_t*>(w_down_packed), I, H, 0);
    return launch_status();
}

extern "C" moe_status_t moe_grouped_swiglu_workspace_size(int64_t N, int E, int64_t H, int64_t I,
                                                          size_t* bytes) {
    if (!bytes) return MOE_ERR_INVALID_ARG;
    const moe_status_t st = check_shapes(N, E, H, I);
    if (st != MOE_OK) return st;
    *bytes = kWsAlign + align_up(size_t(N > 0 ? N : 1) * size_t(I) * 2, kWsAlign);
    return MOE_OK;
}

extern "C" moe_status_t moe_grouped_swiglu(const void* x, const void* w_up_packed,
                                           const void* w_down_packed, const int32_t* offsets,
                                           int64_t N, int E, int64_t H, int64_t I, void* y,
                                           void* workspace, size_t workspace_bytes,
                                           void* stream) {
    MOE_TRACE(__func__);
    moe_status_t st = check_shapes(N, E, H, I);
    if (st != MOE_OK) return st;
    if (!offsets || (N > 0 && (!x || !w_up_packed || !w_down_packed || !y)))
        return MOE_ERR_INVALID_ARG;
    size_t need = 0;
    moe_grouped_swiglu_workspace_size(N, E, H, I, &need);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kWsAlign - 1)) ||
        workspace_bytes < need)
        return MOE_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(w_up_packed) || !aligned16(w_down_packed) || !aligned16(y))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsHeader* header = static_cast<WsHeader*>(workspace);
    reset_status_kernel<<<1, 1, 0, s>>>(header);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    if (N == 0) return MOE_OK;
    void* hidden = static_cast<char*>(workspace) + kWsAlign;

    CUtensorMap m_x, m_up, m_h, m_down;
    if (!make_map(&m_x, x, N, H, BM) || !make_map(&m_up, w_up_packed, int64_t(E) * 2 * I, H, BN) ||
        !make_map(&m_h, hidden, N, I, BM) || !make_map(&m_down, w_down_packed, int64_t(E) * H, I, BN))
        return MOE_ERR_CUDA;

    if (!smem_attrs_set()) return MOE_ERR_CUDA;
    const int grid = sm_count();
    GemmArgs a1{offsets, N, E, int(H), int(I / 128), 2 * I, hidden, I, I, I, nullptr, nullptr, header};
    grouped_gemm_kernel<kSwiglu><<<grid, kThreads, kSmemBytes, s>>>(m_x, m_up, a1, m_x);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    GemmArgs a2{offsets, N, E, int(I), int(H / BN), H, y, H, H, I, nullptr, nullptr, header};
    grouped_gemm_kernel<kPlain><<<grid, kThreads, kSmemBytes, s>>>(m_h, m_down, a2, m_h);
    return launch_status();
}

extern "C" moe_status_t moe_grouped_swiglu_fp8(const void* x_q, const float* scales,
                                               const void* w_up_packed, const void* w_down_packed,
                                               const int32_t* offsets, int64_t N, int E,
                                               int64_t H, int64_t I, void* y, void* workspace,
                                               size_t workspace_bytes, void* stream) {
    MOE_TRACE(__func__);
    moe_status_t st = check_shapes(N, E, H, I);
    if (st != MOE_OK) return st;
    if (H % 512 != 0) return MOE_ERR_UNSUPPORTED;        // scale rows of a multiple of 16 bytes
    if (!offsets || (N > 0 && (!x_q || !scales || !w_up_packed || !w_down_packed || !y)))
        return MOE_ERR_INVALID_ARG;
    size_t need = 0;
    moe_grouped_swiglu_workspace_size(N, E, H, I, &need);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kWsAlign - 1)) ||
        workspace_bytes < need)
        return MOE_ERR_WORKSPACE;
    if (!aligned16(x_q) || !aligned16(scales) ||
        !aligned16(w_up_packed) || !aligned16(w_down_packed) || !aligned16(y))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsHeader* header = static_cast<WsHeader*>(workspace);
    reset_status_kernel<<<1, 1, 0, s>>>(header);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    if (N == 0) return MOE_OK;
    void* hidden = static_cast<char*>(workspace) + kWsAlign;

    CUtensorMap m_x, m_up, m_h, m_down, m_s;
    if (!make_map_u8(&m_x, x_q, N, H, BM) || !make_map_scales(&m_s, scales, N, H / 128) ||
        !make_map(&m_up, w_up_packed, int64_t(E) * 2 * I, H, BN) ||
        !make_map(&m_h, hidden, N, I, BM) || !make_map(&m_down, w_down_packed, int64_t(E) * H, I, BN))
        return MOE_ERR_CUDA;

    if (!smem_attrs_set()) return MOE_ERR_CUDA;
    const int grid = sm_count();
    GemmArgs a1{offsets, N, E, int(H), int(I / 128), 2 * I, hidden, I, I, I, nullptr, nullptr,
                header, scales};
    grouped_gemm_kernel<kSwiglu, true><<<grid, kThreadsA8, kSmemBytesA8, s>>>(m_x, m_up, a1, m_s);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    GemmArgs a2{offsets, N, E, int(I), int(H / BN), H, y, H, H, I, nullptr, nullptr, header};
    grouped_gemm_kernel<kPlain><<<grid, kThreads, kSmemBytes, s>>>(m_h, m_down, a2, m_h);
    return launch_status();
}

extern "C" moe_status_t moe_grouped_swiglu_save(const void* x, const void* w_up_packed,
                                                const void* w_down_packed, const int32_t* offsets,
                                                int64_t N, int E, int64_t H, int64_t I, void* y,
                                                void* hidden, void* gate_up, void* workspace,
                                                size_t workspace_bytes, void* stream) {
    MOE_TRACE(__func__);
    moe_status_t st = check_shapes(N, E, H, I);
    if (st != MOE_OK) return st;
    if (!offsets || (N > 0 && (!x || !w_up_packed || !w_down_packed || !y || !hidden || !gate_up)))
        return MOE_ERR_INVALID_ARG;
    WsHeader* header = nullptr;
    if ((st = status_workspace(workspace, workspace_bytes, &header)) != MOE_OK) return st;
    if (!aligned16(x) || !aligned16(w_up_packed) || !aligned16(w_down_packed) || !aligned16(y) ||
        !aligned16(hidden) || !aligned16(gate_up))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    reset_status_kernel<<<1, 1, 0, s>>>(header);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    if (N == 0) return MOE_OK;
    CUtensorMap m_x, m_up, m_h, m_down;
    if (!make_map(&m_x, x, N, H, BM) || !make_map(&m_up, w_up_packed, int64_t(E) * 2 * I, H, BN) ||
        !make_map(&m_h, hidden, N, I, BM) || !make_map(&m_down, w_down_packed, int64_t(E) * H, I, BN))
        return MOE_ERR_CUDA;
    if (!smem_attrs_set()) return MOE_ERR_CUDA;
    const int grid = sm_count();
    GemmArgs a1{offsets, N, E, int(H), int(I / 128), 2 * I, hidden, I, I, I, nullptr,
                static_cast<uint16_t*>(gate_up), header};
    grouped_gemm_kernel<kSwigluSave><<<grid, kThreads, kSmemBytes, s>>>(m_x, m_up, a1, m_x);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    GemmArgs a2{offsets, N, E, int(I), int(H / BN), H, y, H, H, I, nullptr, nullptr, header};
    grouped_gemm_kernel<kPlain><<<grid, kThreads, kSmemBytes, s>>>(m_h, m_down, a2, m_h);
    return launch_status();
}

extern "C" moe_status_t moe_grouped_swiglu_dgrad(const void* dy, const void* w_up,
                                                 const void* w_down, const int32_t* offsets,
                                                 const void* gate_up, int64_t N, int E, int64_t H,
                                                 int64_t I, void* dgate_up, void* dx,
                                                 void* workspace, size_t workspace_bytes,
                                                 void* stream) {
    MOE_TRACE(__func__);
    moe_status_t st = check_shapes(N, E, H, I);
    if (st != MOE_OK) return st;
    if (!offsets || (N > 0 && (!dy || !w_up || !w_down || !gate_up || !dgate_up || !dx)))
        return MOE_ERR_INVALID_ARG;
    WsHeader* header = nullptr;
    if ((st = status_workspace(workspace, workspace_bytes, &header)) != MOE_OK) return st;
    if (!aligned16(dy) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(gate_up) ||
        !aligned16(dgate_up) || !aligned16(dx))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    reset_status_kernel<<<1, 1, 0, s>>>(header);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    if (N == 0) return MOE_OK;
    CUtensorMap m_dy, m_wd, m_dgu, m_wu;
    if (!make_map(&m_dy, dy, N, H, BM) || !make_map(&m_wd, w_down, int64_t(E) * I, H, BN) ||
        !make_map(&m_dgu, dgate_up, N, 2 * I, BM) || !make_map(&m_wu, w_up, int64_t(E) * H, 2 * I, BN))
        return MOE_ERR_CUDA;
    if (!smem_attrs_set()) return MOE_ERR_CUDA;
    const int grid = sm_count();
    // GMM2 backward + SwiGLU backward: dh = dy @ w_down[e]^T (w_down [E,I,H] is
    // already K-major for this product), [d_gate | d_up] into dgate_up
    GemmArgs d2{offsets, N, E, int(H), int((I + BN - 1) / BN), I, dgate_up, 2 * I, I, I,
                static_cast<const uint16_t*>(gate_up), nullptr, header};
    grouped_gemm_kernel<kSwigluBwd><<<grid, kThreads, kSmemBytes, s>>>(m_dy, m_wd, d2, m_dy);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    // GMM1 backward: dx = dgate_up @ w_up[e]^T (w_up [E,H,2I] is K-major here)
    GemmArgs d1{offsets, N, E, int(2 * I), int(H / BN), H, dx, H, H, I, nullptr, nullptr, header};
    grouped_gemm_kernel<kPlain><<<grid, kThreads, kSmemBytes, s>>>(m_dgu, m_wu, d1, m_dgu);
    return launch_status();
}

extern "C" moe_status_t moe_grouped_swiglu_wgrad(const void* x, const void* hidden,
                                                 const void* dy, const void* dgate_up,
                                                 const int32_t* offsets, int64_t N, int E,
                                                 int64_t H, int64_t I, float* dw_up,
                                                 float* dw_down, void* workspace,
                                                 size_t workspace_bytes, void* stream) {
    MOE_TRACE(__func__);
    moe_status_t st = check_shapes(N, E, H, I);
    if (st != MOE_OK) return st;
    if (!offsets) return MOE_ERR_INVALID_ARG;
    if (dw_up && N > 0 && (!x || !dgate_up)) return MOE_ERR_INVALID_ARG;
    if (dw_down && N > 0 && (!hidden || !dy)) return MOE_ERR_INVALID_ARG;
    WsHeader* header = nullptr;
    if ((st = status_workspace(workspace, workspace_bytes, &header)) != MOE_OK) return st;
    if ((dw_up && (!aligned16(dw_up) || (N > 0 && (!aligned16(x) || !aligned16(dgate_up))))) ||
        (dw_down && (!aligned16(dw_down) || (N > 0 && (!aligned16(hidden) || !aligned16(dy))))))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    reset_status_kernel<<<1, 1, 0, s>>>(header);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    if (N == 0) {                        // no rows: every expert's gradient is zero
        if (dw_up && cudaMemsetAsync(dw_up, 0, size_t(E) * H * 2 * I * sizeof(float), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (dw_down && cudaMemsetAsync(dw_down, 0, size_t(E) * I * H * sizeof(float), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (!smem_attrs_set()) return MOE_ERR_CUDA;
    const int grid = sm_count();
    if (dw_down) {          // dW_down[e] [I,H] = hidden_e^T dy_e
        CUtensorMap m_p, m_q, m_o;
        if (!make_map(&m_p, hidden, N, I, 64) || !make_map(&m_q, dy, N, H, 64) ||
            !make_out_map(&m_o, dw_down, int64_t(E) * I, H))
            return MOE_ERR_CUDA;
        WgradArgs a{offsets, N, E, int(I), int(H), int((I + kWM - 1) / kWM), int(H / BN), dw_down,
                    header};
        grouped_wgrad_kernel<<<grid, kThreads, kWgradSmemBytes, s>>>(m_p, m_q, m_o, a);
        if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    }
    if (dw_up) {            // dW_up[e] [H,2I] = x_e^T dgate_up_e
        CUtensorMap m_p, m_q, m_o;
        if (!make_map(&m_p, x, N, H, 64) || !make_map(&m_q, dgate_up, N, 2 * I, 64) ||
            !make_out_map(&m_o, dw_up, int64_t(E) * H, 2 * I))
            return MOE_ERR_CUDA;
        WgradArgs a{offsets, N, E, int(H), int(2 * I), int((H + kWM - 1) / kWM), int(2 * I / BN),
                    dw_up, header};
        grouped_wgrad_kernel<<<grid, kThreads, kWgradSmemBytes, s>>>(m_p, m_q, m_o, a);
        if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}
