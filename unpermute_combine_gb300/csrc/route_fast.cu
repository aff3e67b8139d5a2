// route_fast.cu -- moe_route / moe_route_grouped for up to 256 experts.
//
// The same outputs as the general route in route.cu: top-k over the router
// logits with a softmax over the k chosen scores ("从零理解 MoE 算子" §3;
// group-limited variant §21), tokens per expert and their prefixes
// (group_list, §7), and the expert-major, token-ascending sorted_indices of a
// masked_select over the transposed routing map ("token dispatcher +
// fuse_a2a" §1.1) with its inverse slot_pos.  K1 then K2, as one
// cooperative launch when every block fits on the GPU at once:
//
//   K1  one block per SM, each a contiguous run of at most 128 tokens.  The
//       block's logits arrive in shared memory by bulk copy (8-token chunks,
//       one mbarrier each), so every byte the block needs is in flight from
//       the start.  Every expert gets a unique 32-bit key: the top 24 bits of
//       the order-preserving bit pattern of its logit above the 8-bit
//       complement of its id, so equal keys cannot occur and a larger key is
//       a larger logit (or an equal one with a lower id) -- except that two
//       logits in the same 24-bit bucket order by id rather than by value.
//       The k winners and the (k+1)-th are checked for that, and such a token
//       (about 1e-3 of tokens on continuous logits, none on exact ties) is
//       ranked again on the exact 32-bit patterns.
//         k <= 8, no group limit: four (E <= 32) or eight threads a token,
//         each keeping a sorted top 8 of its share of the experts with
//         compare-exchange networks, merged over the token's lanes
//         (route_coop_topk_kernel).
//         Otherwise: a warp a token, k+1 rounds of one warp max-reduction
//         each, every lane keeping its best two keys and rescanning only
//         when popped a second time (route_fast_topk_kernel).
//       Then the fp32 softmax, and for every slot a bit in a per-expert token
//       mask of the block: an expert's count is the popcount of its mask, a
//       slot's rank inside the block the popcount of the bits below its
//       token.  Writes topk_idx, topk_w and a row of 16-bit counts per block.
//   K2  per block: the per-expert totals and the sum of the earlier blocks'
//       rows (read straight from the rows for up to 256 blocks, else from a
//       scan kernel's exclusive prefixes), the exclusive scan of the totals
//       (offsets), and the final position offsets[e] + before[e] + rank of
//       every slot.
//   Fused (k <= 8, no group limit, every block resident): K2 runs in the
//       same blocks after a grid barrier, from the masks and ranks still in
//       shared memory.  Otherwise K1 leaves the in-block ranks in slot_pos
//       and K2 is a programmatic dependent launch.
//
// Position of (t, e) = offsets[e] + #{t' < t : e in topk(t')}: integer
// arithmetic throughout, so the result is bit-exact and independent of
// scheduling.  Only the fused launch waits on other blocks, all of them
// resident, with a time limit.
#include <cmath>
#include <map>
#include <mutex>

#include "pipeline.cuh"
#include "route_fast.cuh"

namespace moe {
namespace {

constexpr int kKThreads = 1024;                  // K1: 32 warps
constexpr int kKWarps = kKThreads / 32;
constexpr int kMinTokens = 32;                   // tokens per K1 block, at least
constexpr int kMaxTokens = 128;                  // ... at most: 4 mask words per expert
constexpr int kChunkTokens = 8;                  // tokens per bulk-load chunk
constexpr int kChunks = kMaxTokens / kChunkTokens;
constexpr int kSizingSms = 512;                  // SM count assumed when sizing the workspace
constexpr int kFusedMaxBlocks = 256;             // K2 sums the histogram rows itself up to here
constexpr int kPThreads = 1024;                  // K2
constexpr uint32_t kFull = 0xFFFFFFFFu;

// 16-bit histogram counts, rows padded to 16 bytes
__host__ __device__ inline int hist_stride(int E) { return (E + 7) & ~7; }

int values_per_lane(int E) { return E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : 8; }

int64_t tokens_per_block(int64_t T, int sms) {
    const int64_t tpb = (T + sms - 1) / sms;
    return tpb < kMinTokens ? kMinTokens : tpb > kMaxTokens ? kMaxTokens : tpb;
}

// Histogram rows any T can need: G = ceil(T / tpb) with tpb as above and at
// most kSizingSms SMs, so G <= max(min(kSizingSms, ceil(T/32)), ceil(T/128)).
int64_t max_blocks(int64_t T) {
    const int64_t a = (T + kMinTokens - 1) / kMinTokens;
    const int64_t b = (T + kMaxTokens - 1) / kMaxTokens;
    const int64_t lo = a < kSizingSms ? a : kSizingSms;
    return lo > b ? lo : b;
}

// Order-preserving 32-bit pattern of a float (larger value -> larger
// pattern); -0 is folded onto +0 so the two compare equal.  Every finite
// value maps above 0.
__device__ __forceinline__ uint32_t exact_key(float f) {
    const uint32_t u = __float_as_uint(f + 0.0f);
    return u ^ (uint32_t(int32_t(u) >> 31) | 0x80000000u);
}

__device__ __forceinline__ float exact_key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// ------------------------------------------------------------------------ K1

// Best two keys of a lane (h > r, 0 where there are fewer).
template <int V>
__device__ __forceinline__ void top2(const uint32_t (&key)[V], uint32_t& h, uint32_t& r) {
    h = 0u;
    r = 0u;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const uint32_t lo = min(h, key[v]);
        h = max(h, key[v]);
        r = max(r, lo);
    }
}

// Best two keys of a lane below `below`.
template <int V>
__device__ __forceinline__ void top2_below(const uint32_t (&key)[V], uint32_t below, uint32_t& h,
                                           uint32_t& r) {
    h = 0u;
    r = 0u;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const uint32_t x = key[v] < below ? key[v] : 0u;
        const uint32_t lo = min(h, x);
        h = max(h, x);
        r = max(r, lo);
    }
}

// V logits per lane (expert e = lane*V + v); up to KMAX slots (rounds
// unrolled); FULL: E == 32*V (no lane holds a missing expert).
template <int V, int KMAX, bool GROUPED, bool FULL>
__global__ void __launch_bounds__(kKThreads, 1)
route_fast_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k, int tpb,
                       bool bulk, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                       uint8_t* __restrict__ routing_map, uint16_t* __restrict__ hist,
                       int32_t* __restrict__ rank_out, int n_groups, int topk_groups,
                       uint32_t* __restrict__ dev_status) {
    // the scatter kernel may be scheduled now; it waits for this grid to end
    asm volatile("griddepcontrol.launch_dependents;");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[kChunks];
    __shared__ uint32_t s_m[kKWarps][KMAX + 2];      // the rounds' winning keys, per warp
    __shared__ int s_fail;
    const int W = (tpb + 31) >> 5;                                   // mask words per expert
    float* s_logits = reinterpret_cast<float*>(smem_raw);          // [tpb*E + 32*V] if bulk
    uint32_t* s_mask = reinterpret_cast<uint32_t*>(
        smem_raw + (bulk ? (size_t(tpb) * E + 32 * V) * sizeof(float) : 0));   // [E][W]
    int32_t* s_idx = reinterpret_cast<int32_t*>(s_mask + size_t(E) * W);        // [tpb*k]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = int64_t(blockIdx.x) * tpb;
    const int nt = int(min64(tpb, T - t0));
    const int nchunks = (nt + kChunkTokens - 1) / kChunkTokens;
    if (threadIdx.x == 0) {
        s_fail = 0;
        if (bulk) {
            for (int c = 0; c < nchunks; ++c) mbar_init(smem_addr(&bars[c]), 1);
            mbar_fence_init();
        }
    }
    for (int i = threadIdx.x; i < E * W; i += kKThreads) s_mask[i] = 0u;
    for (int i = threadIdx.x; i < nt * k; i += kKThreads) s_idx[i] = -1;
    __syncthreads();
    if (bulk && threadIdx.x == 0) {
        for (int c = 0; c < nchunks; ++c) {
            const int n = min(kChunkTokens, nt - kChunkTokens * c);
            const uint32_t bytes = uint32_t(n) * uint32_t(E) * 4u;
            const uint32_t bar = smem_addr(&bars[c]);
            mbar_expect_tx(bar, bytes);
            bulk_load(smem_addr(s_logits + size_t(kChunkTokens * c) * E),
                      logits + (t0 + kChunkTokens * c) * E, bytes, bar);
        }
    }

    // group-limited routing: lanes per group (a power of two)
    const int lpg = GROUPED ? E / n_groups / V : 1;
    // low byte of every key: 255 - expert id
    uint32_t nid[V];
#pragma unroll
    for (int v = 0; v < V; ++v) nid[v] = uint32_t(255 - (lane * V + v));
    uint32_t* sm = s_m[warp];

    for (int tl = warp; tl < nt; tl += kKWarps) {
        const int64_t t = t0 + tl;
        const float* grow = logits + t * E;
        const float* srow = s_logits + size_t(tl) * E;
        float val[V];
        if (bulk) {
            const bool ok = __all_sync(kFull, mbar_wait(smem_addr(&bars[tl / kChunkTokens]), 0));
            if (!ok) {
                if (lane == 0) s_fail = 1;
                continue;
            }
            if (V >= 4) {
#pragma unroll
                for (int q = 0; q < V / 4; ++q) {
                    const float4 f = *reinterpret_cast<const float4*>(srow + lane * V + 4 * q);
                    val[4 * q] = f.x; val[4 * q + 1] = f.y; val[4 * q + 2] = f.z; val[4 * q + 3] = f.w;
                }
            } else if (V == 2) {
                const float2 f = *reinterpret_cast<const float2*>(srow + lane * V);
                val[0] = f.x;
                val[V - 1] = f.y;
            } else {
                val[0] = srow[lane];
            }
        } else {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int e = lane * V + v;
                val[v] = (FULL || e < E) ? __ldg(grow + e) : 0.0f;
            }
        }
        uint32_t key[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            key[v] = (exact_key(val[v]) & 0xFFFFFF00u) | nid[v];
            if (!FULL && lane * V + v >= E) key[v] = 0u;
        }
        if (GROUPED) {
            // group score = largest logit of the group (exact patterns); keep
            // the topk_groups best groups, equal scores to the lower group id
            uint32_t gm = 0u;
#pragma unroll
            for (int v = 0; v < V; ++v)
                if (FULL || lane * V + v < E) gm = max(gm, exact_key(val[v]));
            for (int off = 1; off < lpg; off <<= 1) gm = max(gm, __shfl_xor_sync(kFull, gm, off));
            const bool lead = (lane & (lpg - 1)) == 0 && lane * V < E;
            uint32_t cand = lead ? gm : 0u;
            uint32_t kept = 0u;
            for (int i = 0; i < topk_groups; ++i) {
                const uint32_t m = __reduce_max_sync(kFull, cand);
                const uint32_t l = __reduce_min_sync(kFull, cand == m ? uint32_t(lane) : 32u);
                kept |= 1u << l;
                if (uint32_t(lane) == l) cand = 0u;
            }
            if (!((kept >> (lane & ~(lpg - 1))) & 1u)) {
#pragma unroll
                for (int v = 0; v < V; ++v) key[v] = 0u;
            }
        }

        // k + 1 rounds, each one warp max: round j's key is the j-th largest
        // (kept in sm[j]); the last round finds the runner-up that the
        // exactness check needs.  Once every candidate is taken the max is 0
        // and nothing changes.
        uint32_t h, r;
        top2(key, h, r);
        bool rvalid = true;
#pragma unroll
        for (int j = 0; j <= KMAX; ++j) {
            if (j > k) break;
            const uint32_t m = __reduce_max_sync(kFull, h);
            if (lane == 0) sm[j] = m;
            const bool own = h == m;
            const bool scan = own && !rvalid;
            h = own ? r : h;
            rvalid = rvalid && !own;
            if (__any_sync(kFull, scan)) {
                if (scan) {                      // second pop: the best two below m
                    top2_below(key, m, h, r);
                    rvalid = true;
                }
            }
        }
        __syncwarp();
        const uint32_t mine = lane < k ? sm[lane] : 0u;
        const uint32_t nkey = sm[lane + 1 <= KMAX ? lane + 1 : KMAX];
        const uint32_t mk = sm[k - 1], mk1 = sm[k];
        int ej = lane < k ? 255 - int(mine & 0xFFu) : 0;
        float fj = 0.0f;
        if (lane < k) fj = bulk ? srow[ej] : __ldg(grow + ej);
        // exact order: adjacent winners that share a bucket must be equal
        const uint32_t vkj = exact_key(fj);
        const uint32_t nvk = __shfl_down_sync(kFull, vkj, 1);
        bool bad = lane + 1 < k && (mine >> 8) == (nkey >> 8) && vkj != nvk;
        // exact set: if the (k+1)-th shares the k-th's bucket, every
        // candidate of that bucket must hold the same logit
        if (mk1 != 0u && (mk1 >> 8) == (mk >> 8)) {
            const uint32_t beta = mk >> 8;
            uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                if (key[v] != 0u && (key[v] >> 8) == beta) {
                    const uint32_t x = exact_key(val[v]);
                    lo = min(lo, x);
                    hi = max(hi, x);
                }
            }
            if (__reduce_min_sync(kFull, lo) != __reduce_max_sync(kFull, hi)) bad = true;
        }
        if (__any_sync(kFull, bad)) {
            // rank this token again on the exact patterns: largest value,
            // then the lowest expert id holding it
            uint32_t taken = 0u;
            for (int j = 0; j < k; ++j) {
                uint32_t bk = 0u;
                int bv = 0;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    if (key[v] == 0u || ((taken >> v) & 1u)) continue;
                    const uint32_t x = exact_key(val[v]);
                    if (x > bk) { bk = x; bv = v; }
                }
                const uint32_t m = __reduce_max_sync(kFull, bk);
                const int e = int(__reduce_min_sync(kFull, bk == m && bk != 0u
                                                              ? uint32_t(lane * V + bv) : kFull));
                if (lane == j) { ej = e; fj = exact_key_value(m); }
                if (e >= 0 && e / V == lane) taken |= 1u << (e % V);
            }
        }
        // softmax over the k chosen scores, stabilised by the largest (slot 0)
        const float s0 = __shfl_sync(kFull, fj, 0);
        const float ex = lane < k ? expf(fj - s0) : 0.0f;
        float total = ex;
#pragma unroll
        for (int off = KMAX >= 32 ? 16 : KMAX / 2; off > 0; off >>= 1)
            total += __shfl_xor_sync(kFull, total, off);
        if (lane < k) {
            topk_idx[t * k + lane] = ej;
            topk_w[t * k + lane] = ex / total;
            s_idx[tl * k + lane] = ej;
            atomicOr(&s_mask[ej * W + (tl >> 5)], 1u << (tl & 31));
        }
        if (routing_map) {
            uint8_t* mrow = routing_map + t * E;
#pragma unroll
            for (int v = 0; v < V; ++v)
                if (FULL || lane * V + v < E) mrow[lane * V + v] = 0;
            __syncwarp();
            if (lane < k) mrow[ej] = 1;
        }
        __syncwarp();                    // sm is rewritten by the next token
    }
    __syncthreads();
    if (bulk && threadIdx.x == 0) {
        // a chunk whose wait gave up may still be landing: wait for every
        // chunk (bounded) before the block's shared memory is released
        for (int c = 0; c < nchunks; ++c) mbar_wait(smem_addr(&bars[c]), 0);
    }
    if (s_fail && threadIdx.x == 0 && dev_status) atomicExch(dev_status, uint32_t(MOE_ERR_TIMEOUT));
    // this block's histogram row: 16-bit counts (at most tpb <= 128 each)
    const int stride = hist_stride(E);
    uint16_t* hrow = hist + int64_t(blockIdx.x) * stride;
    for (int e = threadIdx.x; e < stride; e += kKThreads) {
        int32_t c = 0;
        if (e < E)
            for (int w = 0; w < W; ++w) c += __popc(s_mask[e * W + w]);
        hrow[e] = uint16_t(c);
    }
    for (int i = threadIdx.x; i < nt * k; i += kKThreads) {
        const int tl = i / k;
        const int e = s_idx[i];
        int32_t rank = -1;
        if (e >= 0 && e < E) {
            const uint32_t* m = s_mask + e * W;
            const int q = tl >> 5;
            rank = __popc(m[q] & ((1u << (tl & 31)) - 1u));
            for (int w = 0; w < q; ++w) rank += __popc(m[w]);
        }
        rank_out[t0 * k + i] = rank;
    }
}

// Exclusive scan of s_in[0..n) into s_out[0..n] (s_out[n] = total), n <= 1024;
// every thread of the block calls it.
__device__ void scan_experts(const int32_t* s_in, int32_t* s_out, int n) {
    __shared__ int32_t s_warp[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t v = int(threadIdx.x) < n ? s_in[threadIdx.x] : 0;
    int32_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    // the totals of the warps before this one: one load a lane, one add-reduce
    const int32_t pre = int32_t(__reduce_add_sync(
        kFull, uint32_t(lane < warp && 32 * lane < n ? s_warp[lane] : 0)));
    if (int(threadIdx.x) < n) s_out[threadIdx.x] = pre + incl - v;
    if (int(threadIdx.x) == n - 1) s_out[n] = pre + incl;
    if (n == 0 && threadIdx.x == 0) s_out[0] = 0;
    __syncthreads();
}

// Outputs of the placement, for the fused route.
struct PlaceOut {
    int32_t* counts;
    int32_t* offsets;
    int32_t* group_list;
    int32_t* sorted_indices;
    int32_t* slot_pos;
    float* permuted_probs;
    WsHeader* header;
    uint32_t* counter;          // grid-barrier count (workspace): arrivals, then departures
    uint32_t* go;               // [2] this call's way, published by block 0 (tag: count,
                                // tag ^ 1: flags), 8 bytes after the count: one load reads both
    uint64_t* marker;           // tag of the last call whose blocks all left the barrier
    uint64_t* flags;            // [G] arrival flags, for a workspace in an unknown state
    uint64_t tag;               // this call's tag (distinct for every call in the process)
    uint64_t expect;            // the marker a clean workspace holds (the previous call's tag)
};

// The placement of route_fast_place_kernel inside the fused route, from this
// block's shared memory: wait until every block has written its count row
// (a grid barrier; every block is resident, so the wait is only for blocks
// still ranking, and it gives up after kWaitLimitNs), sum the rows -- all of
// them for the totals, those before this block for its prefix -- scan the
// totals into offsets and place this block's slots.
__device__ void place_from_block(const uint16_t* __restrict__ hist, int E, int k, int tpb,
                                 int64_t T, const uint32_t* s_mask, int W, const int32_t* s_idx,
                                 const float* s_w, const PlaceOut& po, const uint32_t* s_count0,
                                 uint32_t* __restrict__ dev_status) {
    __shared__ __align__(16) uint32_t s_ptot[kPThreads * 4];   // [P][stride/2] packed partials
    __shared__ __align__(16) uint32_t s_pbef[kPThreads * 4];
    __shared__ int32_t s_tot[kFastMaxExperts];
    __shared__ int32_t s_bef[kFastMaxExperts];
    __shared__ int32_t s_off[kFastMaxExperts + 1];
    const int G = int(gridDim.x), b = int(blockIdx.x), nthreads = int(blockDim.x);
    const int stride = hist_stride(E);
    const int64_t t0 = int64_t(b) * tpb;
    const int nt = int(max64(0, min64(tpb, T - t0)));
    // The grid barrier, without clearing the workspace between calls.  Block 0
    // loaded the count and the marker (the tag of the last call whose blocks
    // all left the barrier) when it started, before any block of this call
    // could arrive, and published the way in the word `go` after its top-k:
    // this call's tag for the count (the marker held the tag of the previous
    // call on this workspace and the count was zero), the tag ^ 1 for the
    // flags.  (With the marker alone, a write over the count that left the
    // marker intact would let blocks through before every row is written.)
    // Every block adds 1 to the count with a release reduction (which
    // releases the block's count row, written before the __syncthreads below,
    // at GPU scope), then reads `go` and the count together:
    //  - count: done once all G blocks have arrived.  Leaving, each block adds
    //    1 more, and the last of the 2G resets the count to zero and stores
    //    the tag in the marker.
    //  - flags (a new workspace, other data written over it or over its
    //    count, a call that timed out): the block stores the tag in its own
    //    flag and warp 0 polls the G flags until all hold it -- correct
    //    whatever the workspace held, as a foreign flag or `go` matches only
    //    by a 2^-63 chance.  Block 0 then takes *s_count0 (the count it
    //    found) plus G off the count -- zero once every arrival has landed,
    //    in whatever order -- and stores the marker.  (Should an arrival have
    //    come before block 0 read the count, the count ends nonzero and the
    //    next call takes the flags again, which clears it.)
    // (A memset of the count before every call measured 1.9 us per call; a
    // self-initialising compare-and-swap count was 90 us slower.)
    __shared__ int s_ok, s_way;
    __syncthreads();
    if (threadIdx.x < 32) {
        const uint64_t start = global_ns();
        bool ok = true;
        int way = 0;                         // 0 not yet published, 1 count, 2 flags
        if (threadIdx.x == 0) {
            // a release reduction (a fence plus a relaxed add measured 0.3 us
            // slower); the flag below, on the flags way only, is a release store
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(po.counter) : "memory");
            for (;;) {
                // the count and `go` in one load (two loads would be two
                // round trips: an acquire load holds back every later load)
                uint32_t w[4];               // count, unused, `go` low, `go` high
                asm volatile("ld.acquire.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                             : "l"(po.counter) : "memory");
                const uint32_t c = w[0];
                const uint64_t g = (uint64_t(w[3]) << 32) | w[2];
                if (g == (po.tag ^ 1u)) { way = 2; break; }
                if (g == po.tag) way = 1;
                if (way == 1 && c >= uint32_t(G)) break;
                if (global_ns() - start > kWaitLimitNs) { ok = false; break; }
                __nanosleep(32);
            }
            if (way == 2)
                asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(po.flags + b),
                             "l"(po.tag) : "memory");
        }
        way = __shfl_sync(kFull, way, 0);
        ok = __shfl_sync(kFull, int(ok), 0) != 0;
        while (way == 2 && ok) {             // the whole warp polls the G flags
            bool mine = true;
            for (int i = int(threadIdx.x); i < G; i += 32) {
                uint64_t v;
                asm volatile("ld.acquire.gpu.global.u64 %0, [%1];"
                             : "=l"(v) : "l"(po.flags + i) : "memory");
                mine = mine && v == po.tag;
            }
            if (__all_sync(kFull, mine)) break;
            const bool late = global_ns() - start > kWaitLimitNs;
            if (__any_sync(kFull, late)) { ok = false; break; }
            __nanosleep(32);
        }
        if (threadIdx.x == 0) { s_ok = ok; s_way = way; }
    }
    __syncthreads();
    if (!s_ok) {
        if (threadIdx.x == 0 && dev_status) atomicExch(dev_status, uint32_t(MOE_ERR_TIMEOUT));
        return;
    }
    if (threadIdx.x == 0) {                  // leaving: leave the count zero for the next call
        if (s_way == 1) {
            if (atomicAdd(po.counter, 1u) == 2u * uint32_t(G) - 1u) {
                *po.counter = 0u;
                *po.marker = po.tag;
            }
        } else if (b == 0) {
            // the count is *s_count0 plus the G arrivals, whenever they land
            atomicSub(po.counter, *s_count0 + uint32_t(G));
            *po.marker = po.tag;
        }
    }
    // rows of 16-bit counts, summed as packed pairs (every sum is at most
    // T <= 152 * kMaxTokens: no carry crosses a half); the rows were written
    // in this launch, so they are read through L2 (ld.global.cg)
    const int Q = stride >> 3;
    const int P = nthreads / Q;
    const int qc = threadIdx.x % Q, p = threadIdx.x / Q;
    if (p < P) {
        uint4 tot = make_uint4(0, 0, 0, 0), bef = make_uint4(0, 0, 0, 0);
        for (int r0 = p; r0 < G; r0 += 8 * P) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int r = r0 + u * P;
                v[u] = r < G ? __ldcg(reinterpret_cast<const uint4*>(hist + int64_t(r) * stride) + qc)
                             : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int r = r0 + u * P;
                tot.x += v[u].x; tot.y += v[u].y; tot.z += v[u].z; tot.w += v[u].w;
                if (r < b) {
                    bef.x += v[u].x; bef.y += v[u].y; bef.z += v[u].z; bef.w += v[u].w;
                }
            }
        }
        reinterpret_cast<uint4*>(s_ptot)[p * Q + qc] = tot;
        reinterpret_cast<uint4*>(s_pbef)[p * Q + qc] = bef;
    }
    __syncthreads();
    // word w of a row holds experts 2w (low half) and 2w+1 (high half); one
    // thread a word adds its P partials (a measured tie with splitting the P
    // over several lanes, which needs one more block barrier)
    for (int w = threadIdx.x; w < (E + 1) / 2; w += nthreads) {
        uint32_t a = 0u, c = 0u;
        for (int pp = 0; pp < P; ++pp) {
            a += s_ptot[pp * (stride / 2) + w];
            c += s_pbef[pp * (stride / 2) + w];
        }
        s_tot[2 * w] = int32_t(a & 0xFFFFu);
        s_bef[2 * w] = int32_t(c & 0xFFFFu);
        if (2 * w + 1 < E) {
            s_tot[2 * w + 1] = int32_t(a >> 16);
            s_bef[2 * w + 1] = int32_t(c >> 16);
        }
    }
    __syncthreads();
    scan_experts(s_tot, s_off, E);
    if (b == 0) {
        for (int e = threadIdx.x; e < E; e += nthreads) {
            po.counts[e] = s_tot[e];
            po.offsets[e] = s_off[e];
            po.group_list[e] = s_off[e + 1];
        }
        if (threadIdx.x == 0) {
            po.offsets[E] = s_off[E];
            po.header->status = MOE_OK;
            po.header->detail = 0;
        }
    }
    for (int i = threadIdx.x; i < nt * k; i += nthreads) {
        const int tk = i / k;
        const int e = s_idx[i];
        if (e < 0 || e >= E) {                           // a token whose logits never arrived
            po.slot_pos[t0 * k + i] = -1;
            continue;
        }
        const uint32_t* m = s_mask + e * W;
        const int qw = tk >> 5;
        int32_t rank = __popc(m[qw] & ((1u << (tk & 31)) - 1u));
        for (int w = 0; w < qw; ++w) rank += __popc(m[w]);
        const int32_t pos = s_off[e] + s_bef[e] + rank;
        po.slot_pos[t0 * k + i] = pos;
        po.sorted_indices[pos] = int32_t(t0 + tk);
        if (po.permuted_probs) po.permuted_probs[pos] = s_w[i];
    }
}

// ------------------------------------------- K1, four or eight threads a token
// For k <= 8 without group limits.  Thread q of a token keeps a sorted top 8
// of its NG*8 experts [q*NG*8, (q+1)*NG*8): each group of 8 keys is sorted by
// a 19-comparator network (Batcher's odd-even merge sort) and merged into the
// running list (the larger of list[i] and group[7-i] form a bitonic sequence
// holding the top 8 of both, sorted by a 12-comparator half-cleaner; the
// smaller ones are the rejects, whose maximum is kept as the best key outside
// the list).  Two butterfly merges over the token's four lanes leave every
// lane with the token's top 8 and its ninth key.  No per-round warp
// reduction: the work is compare-exchanges, with every lane busy.  A token
// whose truncated keys may not order like the logits (the check of the warp
// version) is queued and ranked after the main pass by a warp on the exact
// patterns.


__device__ __forceinline__ void cex(uint32_t& a, uint32_t& b) {   // a >= b afterwards
    const uint32_t hi = max(a, b);
    b = min(a, b);
    a = hi;
}

__device__ __forceinline__ void sort8_desc(uint32_t (&c)[8]) {
    cex(c[0], c[1]); cex(c[2], c[3]); cex(c[4], c[5]); cex(c[6], c[7]);
    cex(c[0], c[2]); cex(c[1], c[3]); cex(c[4], c[6]); cex(c[5], c[7]);
    cex(c[1], c[2]); cex(c[5], c[6]);
    cex(c[0], c[4]); cex(c[1], c[5]); cex(c[2], c[6]); cex(c[3], c[7]);
    cex(c[2], c[4]); cex(c[3], c[5]);
    cex(c[1], c[2]); cex(c[3], c[4]); cex(c[5], c[6]);
}

__device__ __forceinline__ void bitonic8_desc(uint32_t (&m)[8]) {
    cex(m[0], m[4]); cex(m[1], m[5]); cex(m[2], m[6]); cex(m[3], m[7]);
    cex(m[0], m[2]); cex(m[1], m[3]); cex(m[4], m[6]); cex(m[5], m[7]);
    cex(m[0], m[1]); cex(m[2], m[3]); cex(m[4], m[5]); cex(m[6], m[7]);
}

// list <- top 8 of list and c (both sorted descending); ninth <- the largest
// key that is in neither the new list nor below an earlier ninth.
__device__ __forceinline__ void merge8(uint32_t (&list)[8], const uint32_t (&c)[8],
                                       uint32_t& ninth) {
    uint32_t m[8], rej = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        m[i] = max(list[i], c[7 - i]);
        rej = max(rej, min(list[i], c[7 - i]));
    }
    ninth = max(ninth, rej);
    bitonic8_desc(m);
#pragma unroll
    for (int i = 0; i < 8; ++i) list[i] = m[i];
}

// FUSED: the whole route in this one launch -- all blocks resident at once
// (a cooperative launch), a grid barrier after the count rows are written,
// then the placement of route_fast_place_kernel straight from this block's
// shared memory (place_from_block below).
// TPT threads a token (4 or 8), each with NG groups of 8 experts:
// E <= 8 * NG * TPT.
template <int NG, int TPT, bool FULL, bool FUSED>
__global__ void __launch_bounds__(kMaxTokens * TPT, 1)
route_coop_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k, int tpb,
                       bool bulk, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                       uint8_t* __restrict__ routing_map, uint16_t* __restrict__ hist,
                       int32_t* __restrict__ rank_out, uint32_t* __restrict__ dev_status,
                       PlaceOut po) {
    if (!FUSED) asm volatile("griddepcontrol.launch_dependents;");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[kChunks];
    __shared__ int s_fail, s_nfb;
    __shared__ uint32_t s_count0;
    __shared__ int s_fb[kMaxTokens];                 // tokens left for the exact pass
    constexpr int V = NG * 8 * TPT / 32;             // experts per lane in the exact pass
    constexpr int SPT = 8 / TPT;                     // slots per thread (k <= 8)
    constexpr int TPW = 32 / TPT;                    // tokens per warp
    const int nthreads = int(blockDim.x);
    const int W = (tpb + 31) >> 5;
    float* s_logits = reinterpret_cast<float*>(smem_raw);          // [tpb*E + 32*V] if bulk
    uint32_t* s_mask = reinterpret_cast<uint32_t*>(
        smem_raw + (bulk ? (size_t(tpb) * E + 32 * V) * sizeof(float) : 0));   // [E][W]
    int32_t* s_idx = reinterpret_cast<int32_t*>(s_mask + size_t(E) * W);        // [tpb*k]
    float* s_w = reinterpret_cast<float*>(s_idx + size_t(tpb) * k);              // [tpb*k] if FUSED

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tl = threadIdx.x / TPT, q = threadIdx.x % TPT;
    const int64_t t0 = int64_t(blockIdx.x) * tpb;
    const int nt = int(min64(tpb, T - t0));
    const int nchunks = (nt + kChunkTokens - 1) / kChunkTokens;
    // the fused barrier's way (place_from_block): block 0 loads the marker and
    // the count before anything else -- before any block of this call can
    // arrive -- and publishes the way after its top-k
    uint64_t marker = 0;
    uint32_t count0 = 0;
    if (FUSED && threadIdx.x == 0 && blockIdx.x == 0) {
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(marker) : "l"(po.marker) : "memory");
        asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(count0) : "l"(po.counter) : "memory");
    }
    if (threadIdx.x == 0) {
        s_fail = 0;
        s_nfb = 0;
        if (bulk) {
            // the logits go out first, before the block's shared-memory set-up
            for (int c = 0; c < nchunks; ++c) mbar_init(smem_addr(&bars[c]), 1);
            mbar_fence_init();
            for (int c = 0; c < nchunks; ++c) {
                const int n = min(kChunkTokens, nt - kChunkTokens * c);
                const uint32_t bytes = uint32_t(n) * uint32_t(E) * 4u;
                const uint32_t bar = smem_addr(&bars[c]);
                mbar_expect_tx(bar, bytes);
                bulk_load(smem_addr(s_logits + size_t(kChunkTokens * c) * E),
                          logits + (t0 + kChunkTokens * c) * E, bytes, bar);
            }
        }
    }
    for (int i = threadIdx.x; i < E * W; i += nthreads) s_mask[i] = 0u;
    for (int i = threadIdx.x; i < nt * k; i += nthreads) s_idx[i] = -1;
    __syncthreads();

    // warp w holds tokens TPW*w .. TPW*w + TPW - 1, all in one 8-token chunk
    const bool active = tl < nt;
    const bool warp_live = warp * TPW < nt;
    bool ok = true;
    if (bulk && warp_live)
        ok = __all_sync(kFull, mbar_wait(smem_addr(&bars[warp * TPW / kChunkTokens]), 0));
    if (!ok && lane == 0) s_fail = 1;
    if (ok && warp_live) {
        const int64_t t = t0 + (active ? tl : 0);
        const float* grow = logits + t * E;
        const float* srow = s_logits + size_t(active ? tl : 0) * E;
        const int ebase = q * NG * 8;
        uint32_t list[8], ninth = 0u;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            // groups taken in an order rotated by q, so the four lanes of a
            // token read different shared-memory banks
            const int gg = (g + q) & (NG - 1);
            const int e0 = ebase + gg * 8;
            float f[8];
            if (bulk) {
                const float4 a = *reinterpret_cast<const float4*>(srow + e0);
                const float4 b = *reinterpret_cast<const float4*>(srow + e0 + 4);
                f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
                f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
            } else {
#pragma unroll
                for (int v = 0; v < 8; ++v) f[v] = (FULL || e0 + v < E) ? __ldg(grow + e0 + v) : 0.0f;
            }
            uint32_t c[8];
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                c[v] = (exact_key(f[v]) & 0xFFFFFF00u) | uint32_t(255 - (e0 + v));
                if (!FULL && e0 + v >= E) c[v] = 0u;
            }
            sort8_desc(c);
            if (g == 0) {
#pragma unroll
                for (int i = 0; i < 8; ++i) list[i] = c[i];
            } else {
                merge8(list, c, ninth);
            }
        }
#pragma unroll
        for (int off = 1; off < TPT; off <<= 1) {     // the token's TPT lanes
            uint32_t c[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) c[i] = __shfl_xor_sync(kFull, list[i], off);
            const uint32_t n2 = __shfl_xor_sync(kFull, ninth, off);
            merge8(list, c, ninth);
            ninth = max(ninth, n2);
        }
        // the k-th key (smallest of the first k), the (k+1)-th (largest of
        // the rest and the ninth), and this lane's slots q*SPT .. -- as
        // reductions and masks, so the list stays in registers
        uint32_t kth = 0xFFFFFFFFu, k1th = ninth, a = 0u, b = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            kth = i < k ? min(kth, list[i]) : kth;
            k1th = i >= k ? max(k1th, list[i]) : k1th;
        }
#pragma unroll
        for (int qq = 0; qq < TPT; ++qq) {
            const uint32_t sel = q == qq ? 0xFFFFFFFFu : 0u;
            a |= list[SPT * qq] & sel;
            if (SPT == 2) b |= list[SPT * qq + 1] & sel;
        }
        const int j0 = SPT * q, j1 = SPT == 2 ? SPT * q + 1 : 8;   // 8: no second slot
        int e_a = 255 - int(a & 0xFFu);
        const int e_b = 255 - int(b & 0xFFu);
        float fa = 0.0f, fb = 0.0f;
        if (active && j0 < k) fa = bulk ? srow[e_a] : __ldg(grow + e_a);
        if (active && j1 < k) fb = bulk ? srow[e_b] : __ldg(grow + e_b);
        uint32_t vka = exact_key(fa);
        const uint32_t vkb = exact_key(fb);
        // exact order: adjacent winners that share a bucket must be equal
        const uint32_t na = __shfl_down_sync(kFull, a, 1), nvka = __shfl_down_sync(kFull, vka, 1);
        bool bad_order = SPT == 2
            ? (j1 < k && (a >> 8) == (b >> 8) && vka != vkb) ||
              (q < TPT - 1 && j1 + 1 < k && (b >> 8) == (na >> 8) && vkb != nvka)
            : (q < TPT - 1 && j0 + 1 < k && (a >> 8) == (na >> 8) && vka != nvka);
        // exact set: if the (k+1)-th shares the k-th's bucket, every
        // candidate of that bucket must hold the same logit
        const bool amb = k1th != 0u && (k1th >> 8) == (kth >> 8);
        bool bad_set = false;
        if (__any_sync(kFull, amb)) {
            uint32_t lo = 0xFFFFFFFFu, hi = 0u;
            if (amb) {
                const uint32_t beta = kth >> 8;
#pragma unroll 8
                for (int i = 0; i < NG * 8; ++i) {
                    const int e = ebase + i;
                    if (!FULL && e >= E) break;
                    const uint32_t x = exact_key(bulk ? srow[e] : __ldg(grow + e));
                    const bool in = (x >> 8) == beta;
                    lo = in ? min(lo, x) : lo;
                    hi = in ? max(hi, x) : hi;
                }
            }
#pragma unroll
            for (int off = 1; off < TPT; off <<= 1) {
                lo = min(lo, __shfl_xor_sync(kFull, lo, off));
                hi = max(hi, __shfl_xor_sync(kFull, hi, off));
            }
            if (amb && lo != hi) bad_set = true;
        }
        // both flags token-wide (every lane takes part in every shuffle: no
        // short-circuit)
#pragma unroll
        for (int off = 1; off < TPT; off <<= 1) {
            const int o1 = __shfl_xor_sync(kFull, int(bad_order), off);
            const int o2 = __shfl_xor_sync(kFull, int(bad_set), off);
            bad_order = bad_order || o1 != 0;
            bad_set = bad_set || o2 != 0;
        }
        const bool any_order_only = __any_sync(kFull, bad_order && !bad_set);
        if (TPT == 8 && any_order_only) {
            // the set is right and only the order within a bucket is not:
            // sort the token's winners (one per lane) on the exact key --
            // value, then the lower id -- with a bitonic network over its
            // eight lanes.  A token already in order comes out unchanged.
            uint64_t key = j0 < k ? (uint64_t(vka) << 32) | uint64_t(0xFFFFFFFFu - uint32_t(e_a))
                                  : 0ull;
#pragma unroll
            for (int size = 2; size <= 8; size <<= 1) {
#pragma unroll
                for (int st = size >> 1; st > 0; st >>= 1) {
                    const uint64_t other = __shfl_xor_sync(kFull, key, st);
                    const bool take_max = ((q & st) == 0) != ((q & size) != 0);
                    key = take_max ? (key > other ? key : other) : (key < other ? key : other);
                }
            }
            if (bad_order && !bad_set && j0 < k) {
                vka = uint32_t(key >> 32);
                e_a = int(0xFFFFFFFFu - uint32_t(key));
                fa = exact_key_value(vka);
            }
        }
        const bool bad = bad_set || (TPT != 8 && bad_order);
        if (active && bad && q == 0) s_fb[atomicAdd(&s_nfb, 1)] = tl;
        // softmax over the k chosen scores, stabilised by the largest (slot 0)
        const float s0 = __shfl_sync(kFull, fa, lane & ~(TPT - 1));
        const float xa = j0 < k ? expf(fa - s0) : 0.0f;
        const float xb = j1 < k ? expf(fb - s0) : 0.0f;
        float total = xa + xb;
#pragma unroll
        for (int off = 1; off < TPT; off <<= 1) total += __shfl_xor_sync(kFull, total, off);
        if (active && !bad) {
            if (j0 < k) {
                const float w = xa / total;
                topk_idx[t * k + j0] = e_a;
                topk_w[t * k + j0] = w;
                s_idx[tl * k + j0] = e_a;
                if (FUSED) s_w[tl * k + j0] = w;
                atomicOr(&s_mask[e_a * W + (tl >> 5)], 1u << (tl & 31));
            }
            if (j1 < k) {
                const float w = xb / total;
                topk_idx[t * k + j1] = e_b;
                topk_w[t * k + j1] = w;
                s_idx[tl * k + j1] = e_b;
                if (FUSED) s_w[tl * k + j1] = w;
                atomicOr(&s_mask[e_b * W + (tl >> 5)], 1u << (tl & 31));
            }
        }
        if (routing_map && active && !bad) {
            uint8_t* mrow = routing_map + t * E;
            for (int e = ebase; e < ebase + NG * 8; ++e)
                if (FULL || e < E) mrow[e] = 0;
        }
        __syncwarp();
        if (routing_map && active && !bad) {
            uint8_t* mrow = routing_map + t * E;
            if (j0 < k) mrow[e_a] = 1;
            if (j1 < k) mrow[e_b] = 1;
        }
    }
    __syncthreads();
    if (FUSED && threadIdx.x == 0 && blockIdx.x == 0) {
        // the way, published after the top-k: by now the two loads are long
        // back (storing it at the start would hold this block's first warp,
        // and with it the block, until they were)
        const bool clean = marker == po.expect && count0 == 0u;
        const uint64_t g = clean ? po.tag : po.tag ^ 1u;
        asm volatile("st.relaxed.gpu.global.v2.u32 [%0], {%1, %2};"
                     :: "l"(po.go), "r"(uint32_t(g)), "r"(uint32_t(g >> 32)) : "memory");
        s_count0 = count0;
    }
    // the queued tokens, one warp each, ranked on the exact patterns: the
    // largest value, then the lowest expert id holding it
    for (int i = warp; i < s_nfb; i += nthreads / 32) {
        const int ftl = s_fb[i];
        const int64_t t = t0 + ftl;
        const float* grow = logits + t * E;
        const float* srow = s_logits + size_t(ftl) * E;
        uint32_t ek[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int e = lane * V + v;
            ek[v] = (FULL || e < E) ? exact_key(bulk ? srow[e] : __ldg(grow + e)) : 0u;
        }
        uint32_t taken = 0u;
        int ej = 0;
        float fj = 0.0f;
        for (int j = 0; j < k; ++j) {
            uint32_t bk = 0u;
            int bv = 0;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                if ((taken >> v) & 1u) continue;
                if (ek[v] > bk) { bk = ek[v]; bv = v; }
            }
            const uint32_t m = __reduce_max_sync(kFull, bk);
            const int e = int(__reduce_min_sync(kFull, bk == m && bk != 0u
                                                          ? uint32_t(lane * V + bv) : kFull));
            if (lane == j) { ej = e; fj = exact_key_value(m); }
            if (e >= 0 && e / V == lane) taken |= 1u << (e % V);
        }
        const float s0 = __shfl_sync(kFull, fj, 0);
        const float ex = lane < k ? expf(fj - s0) : 0.0f;
        float total = ex;
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) total += __shfl_xor_sync(kFull, total, off);
        if (lane < k) {
            const float w = ex / total;
            topk_idx[t * k + lane] = ej;
            topk_w[t * k + lane] = w;
            s_idx[ftl * k + lane] = ej;
            if (FUSED) s_w[ftl * k + lane] = w;
            atomicOr(&s_mask[ej * W + (ftl >> 5)], 1u << (ftl & 31));
        }
        if (routing_map) {
            uint8_t* mrow = routing_map + t * E;
#pragma unroll
            for (int v = 0; v < V; ++v)
                if (FULL || lane * V + v < E) mrow[lane * V + v] = 0;
            __syncwarp();
            if (lane < k) mrow[ej] = 1;
        }
    }
    __syncthreads();
    if (bulk && s_fail && threadIdx.x == 0)          // a chunk that never arrived may still land
        for (int c = 0; c < nchunks; ++c) mbar_wait(smem_addr(&bars[c]), 0);
    if (s_fail && threadIdx.x == 0 && dev_status) atomicExch(dev_status, uint32_t(MOE_ERR_TIMEOUT));
    const int stride = hist_stride(E);
    uint16_t* hrow = hist + int64_t(blockIdx.x) * stride;
    for (int e = threadIdx.x; e < stride; e += nthreads) {
        int32_t c = 0;
        if (e < E)
            for (int w = 0; w < W; ++w) c += __popc(s_mask[e * W + w]);
        hrow[e] = uint16_t(c);
    }
    if constexpr (FUSED) {
        place_from_block(hist, E, k, tpb, T, s_mask, W, s_idx, s_w, po, &s_count0, dev_status);
    } else {
        for (int i = threadIdx.x; i < nt * k; i += nthreads) {
            const int tk = i / k;
            const int e = s_idx[i];
            int32_t rank = -1;
            if (e >= 0 && e < E) {
                const uint32_t* m = s_mask + e * W;
                const int qw = tk >> 5;
                rank = __popc(m[qw] & ((1u << (tk & 31)) - 1u));
                for (int w = 0; w < qw; ++w) rank += __popc(m[w]);
            }
            rank_out[t0 * k + i] = rank;
        }
    }
}

// ------------------------------------------------------- scan (beyond K2's reach)
// Block x owns experts [32x, 32x+32); thread (g, c) owns expert 32x+c and row
// group g: pre[b][e] = sum of rows before b (exclusive prefix), pre[G][e] =
// the total.
__global__ void __launch_bounds__(1024)
route_fast_scan_kernel(const uint16_t* __restrict__ hist, int32_t* __restrict__ pre, int64_t G,
                       int E) {
    wait_for_predecessor();
    __shared__ int32_t s_part[32][33];
    const int stride = hist_stride(E);
    const int c = threadIdx.x & 31, g = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + c;
    const int64_t rows = (G + 31) / 32;
    const int64_t b0 = min64(G, g * rows), b1 = min64(G, b0 + rows);
    int32_t sum = 0;
    if (e < E)
        for (int64_t b = b0; b < b1; ++b) sum += hist[b * stride + e];
    s_part[g][c] = sum;
    __syncthreads();
    int32_t run = 0;
    for (int q = 0; q < g; ++q) run += s_part[q][c];
    if (e < E) {
        for (int64_t b = b0; b < b1; ++b) {
            pre[b * E + e] = run;
            run += hist[b * stride + e];
        }
        if (g == 31) pre[G * E + e] = run;
    }
}

// ------------------------------------------------------------------------ K2

template <bool FUSED>
__global__ void __launch_bounds__(kPThreads)
route_fast_place_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
                        int64_t T, int E, int k, int tpb, int64_t G,
                        const uint16_t* __restrict__ hist, const int32_t* __restrict__ pre,
                        int32_t* __restrict__ counts,
                        int32_t* __restrict__ offsets, int32_t* __restrict__ group_list,
                        int32_t* __restrict__ sorted_indices, int32_t* __restrict__ slot_pos,
                        float* __restrict__ permuted_probs, WsHeader* __restrict__ header) {
    wait_for_predecessor();
    __shared__ __align__(16) uint32_t s_ptot[kPThreads * 4];   // [P][stride/2] packed partial totals
    __shared__ __align__(16) uint32_t s_pbef[kPThreads * 4];   // [P][stride/2] packed "before"
    __shared__ int32_t s_tot[kFastMaxExperts];
    __shared__ int32_t s_bef[kFastMaxExperts];
    __shared__ int32_t s_off[kFastMaxExperts + 1];
    const int stride = hist_stride(E);
    const int64_t b = blockIdx.x;
    const int64_t t0 = b * tpb;
    const int nt = int(max64(0, min64(tpb, T - t0)));

    // this block's slots, fetched before the histogram work (at most
    // tpb*k/kPThreads = 4 per thread)
    constexpr int kPer = kMaxTokens * kMaxTopK / kPThreads;
    int32_t se[kPer], sr[kPer];
    float sw[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int i = threadIdx.x + u * kPThreads;
        se[u] = -1;
        sr[u] = -1;
        sw[u] = 0.0f;
        if (i < nt * k) {
            se[u] = topk_idx[t0 * k + i];
            sr[u] = slot_pos[t0 * k + i];
            sw[u] = topk_w[t0 * k + i];
        }
    }

    if (FUSED) {
        // rows of 16-bit counts: Q 16-byte columns of 8 counts per row, P rows
        // at a time, up to 8 loads in flight.  Counts are summed as packed
        // 16-bit pairs (no carry crosses a half: every sum is at most
        // T <= kFusedMaxBlocks * kMaxTokens = 32768).
        const int Q = stride >> 3;
        const int P = kPThreads / Q;
        const int q = threadIdx.x % Q, p = threadIdx.x / Q;
        uint4 tot = make_uint4(0, 0, 0, 0), bef = make_uint4(0, 0, 0, 0);
        if (p < P) {
            for (int64_t r0 = p; r0 < G; r0 += 8 * int64_t(P)) {
                uint4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int64_t r = r0 + int64_t(u) * P;
                    v[u] = r < G ? __ldg(reinterpret_cast<const uint4*>(hist + r * stride) + q)
                                 : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int64_t r = r0 + int64_t(u) * P;
                    tot.x += v[u].x; tot.y += v[u].y; tot.z += v[u].z; tot.w += v[u].w;
                    if (r < b) {
                        bef.x += v[u].x; bef.y += v[u].y; bef.z += v[u].z; bef.w += v[u].w;
                    }
                }
            }
            reinterpret_cast<uint4*>(s_ptot)[p * Q + q] = tot;
            reinterpret_cast<uint4*>(s_pbef)[p * Q + q] = bef;
        }
        __syncthreads();
        // word w of a row holds experts 2w (low half) and 2w+1 (high half)
        for (int w = threadIdx.x; w < (E + 1) / 2; w += kPThreads) {
            uint32_t a = 0u, c = 0u;
            for (int pp = 0; pp < P; ++pp) {
                a += s_ptot[pp * (stride / 2) + w];
                c += s_pbef[pp * (stride / 2) + w];
            }
            s_tot[2 * w] = int32_t(a & 0xFFFFu);
            s_bef[2 * w] = int32_t(c & 0xFFFFu);
            if (2 * w + 1 < E) {
                s_tot[2 * w + 1] = int32_t(a >> 16);
                s_bef[2 * w + 1] = int32_t(c >> 16);
            }
        }
    } else {
        for (int e = threadIdx.x; e < E; e += kPThreads) {
            s_bef[e] = b < G ? pre[b * E + e] : 0;
            s_tot[e] = pre[G * E + e];
        }
    }
    __syncthreads();
    scan_experts(s_tot, s_off, E);
    if (b == 0) {
        for (int e = threadIdx.x; e < E; e += kPThreads) {
            counts[e] = s_tot[e];
            offsets[e] = s_off[e];
            group_list[e] = s_off[e + 1];
        }
        if (threadIdx.x == 0) {
            offsets[E] = s_off[E];
            header->status = MOE_OK;
            header->detail = 0;
        }
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int i = threadIdx.x + u * kPThreads;
        if (i >= nt * k) continue;
        const int e = se[u];
        if (e < 0 || e >= E || sr[u] < 0) {          // a token whose logits never arrived
            slot_pos[t0 * k + i] = -1;
            continue;
        }
        const int32_t pos = s_off[e] + s_bef[e] + sr[u];
        slot_pos[t0 * k + i] = pos;
        sorted_indices[pos] = int32_t(t0 + i / k);
        if (permuted_probs) permuted_probs[pos] = sw[u];
    }
}

// logits [tpb*E + 32*V] (bulk), masks [E][W], ids [tpb*k], weights [tpb*k]
size_t topk_smem_bytes(int64_t tpb, int E, int k, int V, bool bulk) {
    const int W = int((tpb + 31) / 32);
    return (bulk ? (size_t(tpb) * E + 32 * V) * sizeof(float) : 0) +
           sizeof(uint32_t) * size_t(E) * W + 2 * sizeof(int32_t) * size_t(tpb) * k;
}

template <int V, int KMAX, bool GROUPED, bool FULL>
moe_status_t launch_topk(const float* logits, int64_t T, int E, int k, int tpb, int64_t G,
                         bool bulk, int32_t* topk_idx, float* topk_w, uint8_t* routing_map,
                         uint16_t* hist, int32_t* rank_out, int n_groups, int topk_groups,
                         cudaStream_t s) {
    const auto kern = route_fast_topk_kernel<V, KMAX, GROUPED, FULL>;
    const int max_smem = int(topk_smem_bytes(kMaxTokens, kFastMaxExperts, kMaxTopK, 8, true));
    if (!opt_in_smem((const void*)kern, max_smem)) return MOE_ERR_CUDA;
    kern<<<unsigned(G), kKThreads, topk_smem_bytes(tpb, E, k, V, bulk), s>>>(
        logits, T, E, k, tpb, bulk, topk_idx, topk_w, routing_map, hist, rank_out, n_groups,
        topk_groups, device_status_word());
    return launch_status();
}

template <int V, bool GROUPED, bool FULL>
moe_status_t launch_topk_k(const float* logits, int64_t T, int E, int k, int tpb, int64_t G,
                           bool bulk, int32_t* topk_idx, float* topk_w, uint8_t* routing_map,
                           uint16_t* hist, int32_t* rank_out, int n_groups, int topk_groups,
                           cudaStream_t s) {
    return k <= 8
        ? launch_topk<V, 8, GROUPED, FULL>(logits, T, E, k, tpb, G, bulk, topk_idx, topk_w,
                                           routing_map, hist, rank_out, n_groups, topk_groups, s)
        : launch_topk<V, kMaxTopK, GROUPED, FULL>(logits, T, E, k, tpb, G, bulk, topk_idx, topk_w,
                                                  routing_map, hist, rank_out, n_groups,
                                                  topk_groups, s);
}

// The fused route's barrier tags: a distinct value for every call in the
// process (the SplitMix64 output function -- Steele, Lea and Flood, "Fast
// splittable pseudorandom number generators", OOPSLA 2014 -- of a call
// counter: its odd Weyl step and xor-shift-multiply mix are bijections of
// 64-bit words), and the tag the previous call on the same workspace
// received, which the workspace's marker holds if that call completed.
void barrier_tags(const void* workspace, uint64_t* tag, uint64_t* expect) {
    static std::mutex m;
    static std::map<std::pair<int, const void*>, uint64_t> last;
    static uint64_t calls = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(m);
    uint64_t z = (++calls) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    *tag = z ^ (z >> 31);
    const auto key = std::make_pair(dev, workspace);
    const auto it = last.find(key);
    *expect = it != last.end() ? it->second : ~*tag;    // unknown workspace: no match
    if (it == last.end() && last.size() >= 4096) last.clear();
    last[key] = *tag;
}

// The few-threads-a-token top-k (TPT threads a token, NG groups of 8
// experts each).  When every block can be resident at once the whole route
// runs in this one cooperative launch (*fused = true); otherwise the kernel
// leaves count rows and in-block ranks for the place kernel.
template <int NG, int TPT, bool FULL>
moe_status_t launch_coop(const float* logits, int64_t T, int E, int k, int tpb, int64_t G,
                         bool bulk, int32_t* topk_idx, float* topk_w, uint8_t* routing_map,
                         uint16_t* hist, int32_t* rank_out, const PlaceOut& po, bool* fused,
                         cudaStream_t s) {
    constexpr int V = NG * 8 * TPT / 32;
    constexpr int threads = kMaxTokens * TPT;
    static_assert(threads <= kPThreads, "place_from_block sizes its arrays for kPThreads");
    const int max_smem = int(topk_smem_bytes(kMaxTokens, kFastMaxExperts, 8, 8, true));
    const size_t smem = topk_smem_bytes(tpb, E, k, V, bulk);
    const auto kfused = route_coop_topk_kernel<NG, TPT, FULL, true>;
    const auto kplain = route_coop_topk_kernel<NG, TPT, FULL, false>;
    if (!opt_in_smem((const void*)kfused, max_smem) || !opt_in_smem((const void*)kplain, max_smem))
        return MOE_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfused, threads, smem) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    uint32_t* dev_status = device_status_word();
    *fused = G <= int64_t(per_sm) * sm_count() && G <= kFusedMaxBlocks;
    if (!*fused) {
        kplain<<<unsigned(G), threads, smem, s>>>(logits, T, E, k, tpb, bulk, topk_idx, topk_w,
                                                 routing_map, hist, rank_out, dev_status, po);
        return launch_status();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(G));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    PlaceOut pt = po;
    barrier_tags(po.counter, &pt.tag, &pt.expect);
    return cudaLaunchKernelEx(&cfg, kfused, logits, T, E, k, tpb, bulk, topk_idx, topk_w,
                              routing_map, hist, rank_out, dev_status, pt) == cudaSuccess
               ? MOE_OK : MOE_ERR_CUDA;
}

// E <= 32: four threads a token, one group each; more experts: eight threads
// a token (twice the resident warps of four, half the chain per thread)
template <int V>
moe_status_t launch_coop_v(const float* logits, int64_t T, int E, int k, int tpb, int64_t G,
                           bool bulk, int32_t* topk_idx, float* topk_w, uint8_t* routing_map,
                           uint16_t* hist, int32_t* rank_out, const PlaceOut& po, bool* fused,
                           cudaStream_t s) {
    constexpr int TPT = V == 1 ? 4 : 8;
    constexpr int NG = V * 4 / TPT;
    return E == 32 * V
        ? launch_coop<NG, TPT, true>(logits, T, E, k, tpb, G, bulk, topk_idx, topk_w,
                                     routing_map, hist, rank_out, po, fused, s)
        : launch_coop<NG, TPT, false>(logits, T, E, k, tpb, G, bulk, topk_idx, topk_w,
                                      routing_map, hist, rank_out, po, fused, s);
}

template <int V>
moe_status_t launch_topk_v(const float* logits, int64_t T, int E, int k, int tpb, int64_t G,
                           bool bulk, int32_t* topk_idx, float* topk_w, uint8_t* routing_map,
                           uint16_t* hist, int32_t* rank_out, int n_groups, int topk_groups,
                           cudaStream_t s) {
    const bool full = E == 32 * V;
    if (n_groups > 0)
        return full ? launch_topk_k<V, true, true>(logits, T, E, k, tpb, G, bulk, topk_idx, topk_w,
                                                   routing_map, hist, rank_out, n_groups,
                                                   topk_groups, s)
                    : launch_topk_k<V, true, false>(logits, T, E, k, tpb, G, bulk, topk_idx,
                                                    topk_w, routing_map, hist, rank_out, n_groups,
                                                    topk_groups, s);
    return full ? launch_topk_k<V, false, true>(logits, T, E, k, tpb, G, bulk, topk_idx, topk_w,
                                                routing_map, hist, rank_out, 0, 0, s)
                : launch_topk_k<V, false, false>(logits, T, E, k, tpb, G, bulk, topk_idx, topk_w,
                                                 routing_map, hist, rank_out, 0, 0, s);
}

// Workspace after the header: 16-bit histogram rows [G][stride], the fused
// route's barrier (a 256-byte unit holding the count at 0, `go` at 8 and
// the marker at 16, then kFusedMaxBlocks uint64 flags), then (when G can exceed
// kFusedMaxBlocks) the scan kernel's int32 prefixes [G+1][E].
constexpr size_t kBarrierBytes = kWsAlign + kFusedMaxBlocks * sizeof(uint64_t);
static_assert(kBarrierBytes % kWsAlign == 0, "the barrier word keeps the prefixes aligned");
size_t counts_bytes(int64_t T, int E) {
    return align_up(size_t(max_blocks(T)) * size_t(hist_stride(E)) * sizeof(uint16_t), kWsAlign);
}
size_t prefix_bytes(int64_t T, int E) {
    const int64_t g = max_blocks(T);
    return g > kFusedMaxBlocks ? align_up(size_t(g + 1) * size_t(E) * sizeof(int32_t), kWsAlign)
                               : 0;
}

}  // namespace

bool fast_route_supported(int E, int n_groups) {
    if (E < 1 || E > kFastMaxExperts) return false;
    if (n_groups > 0) {
        const int V = values_per_lane(E);
        const int gsize = E / n_groups;
        if (gsize % V != 0) return false;
        const int lpg = gsize / V;
        if (lpg & (lpg - 1)) return false;
    }
    return true;
}

size_t fast_hist_bytes(int64_t T, int E) {
    return counts_bytes(T, E) + kBarrierBytes + prefix_bytes(T, E);
}

moe_status_t fast_route(const float* logits, int64_t T, int E, int k, int n_groups,
                        int topk_groups, int32_t* topk_idx, float* topk_w, int32_t* counts,
                        int32_t* offsets, int32_t* group_list, int32_t* sorted_indices,
                        int32_t* slot_pos, float* permuted_probs, uint8_t* routing_map,
                        WsHeader* header, int32_t* scratch, cudaStream_t s) {
    int sms = sm_count();
    if (sms > kSizingSms) sms = kSizingSms;
    const int64_t tpb = T > 0 ? tokens_per_block(T, sms) : kMinTokens;
    const int64_t G = (T + tpb - 1) / tpb;
    const bool bulk = E % 4 == 0 && aligned16(logits);
    uint16_t* hist = reinterpret_cast<uint16_t*>(scratch);
    char* barrier = reinterpret_cast<char*>(scratch) + counts_bytes(T, E);
    int32_t* pre = reinterpret_cast<int32_t*>(barrier + kBarrierBytes);
    if (G > 0 && n_groups == 0 && k <= 8) {
        // a few threads a token, compare-exchange networks; the whole route
        // in one cooperative launch when every block fits at once
        const int NG = values_per_lane(E);      // logits per lane of a 32-lane token
        const PlaceOut po{counts, offsets, group_list, sorted_indices, slot_pos, permuted_probs,
                          header, reinterpret_cast<uint32_t*>(barrier),
                          reinterpret_cast<uint32_t*>(barrier + 8),
                          reinterpret_cast<uint64_t*>(barrier + 16),
                          reinterpret_cast<uint64_t*>(barrier + kWsAlign), 0, 0};
        bool fused = false;
        moe_status_t st;
        if (NG == 1)
            st = launch_coop_v<1>(logits, T, E, k, int(tpb), G, bulk, topk_idx, topk_w,
                                   routing_map, hist, slot_pos, po, &fused, s);
        else if (NG == 2)
            st = launch_coop_v<2>(logits, T, E, k, int(tpb), G, bulk, topk_idx, topk_w,
                                   routing_map, hist, slot_pos, po, &fused, s);
        else if (NG == 4)
            st = launch_coop_v<4>(logits, T, E, k, int(tpb), G, bulk, topk_idx, topk_w,
                                   routing_map, hist, slot_pos, po, &fused, s);
        else
            st = launch_coop_v<8>(logits, T, E, k, int(tpb), G, bulk, topk_idx, topk_w,
                                   routing_map, hist, slot_pos, po, &fused, s);
        if (st != MOE_OK || fused) return st;
    } else if (G > 0) {
        const int V = values_per_lane(E);
        const int g = n_groups, kg = topk_groups;
        moe_status_t st;
        if (V == 1)
            st = launch_topk_v<1>(logits, T, E, k, int(tpb), G, bulk, topk_idx, topk_w,
                                  routing_map, hist, slot_pos, g, kg, s);
        else if (V == 2)
            st = launch_topk_v<2>(logits, T, E, k, int(tpb), G, bulk, topk_idx, topk_w,
                                  routing_map, hist, slot_pos, g, kg, s);
        else if (V == 4)
            st = launch_topk_v<4>(logits, T, E, k, int(tpb), G, bulk, topk_idx, topk_w,
                                  routing_map, hist, slot_pos, g, kg, s);
        else
            st = launch_topk_v<8>(logits, T, E, k, int(tpb), G, bulk, topk_idx, topk_w,
                                  routing_map, hist, slot_pos, g, kg, s);
        if (st != MOE_OK) return st;
    }
    const bool fused = G <= kFusedMaxBlocks;
    if (!fused && launch_dependent(route_fast_scan_kernel, unsigned((E + 31) / 32), 1024, 0, s,
                                   (const uint16_t*)hist, pre, G, E) != cudaSuccess)
        return MOE_ERR_CUDA;
    const cudaError_t err = fused
        ? launch_dependent(route_fast_place_kernel<true>, unsigned(G > 0 ? G : 1), kPThreads, 0,
                           s, (const int32_t*)topk_idx, (const float*)topk_w, T, E, k, int(tpb),
                           G, (const uint16_t*)hist, (const int32_t*)pre, counts, offsets,
                           group_list, sorted_indices, slot_pos, permuted_probs, header)
        : launch_dependent(route_fast_place_kernel<false>, unsigned(G), kPThreads, 0, s,
                           (const int32_t*)topk_idx, (const float*)topk_w, T, E, k, int(tpb), G,
                           (const uint16_t*)hist, (const int32_t*)pre, counts, offsets,
                           group_list, sorted_indices, slot_pos, permuted_probs, header);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
