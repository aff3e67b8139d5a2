// route.cu -- moe_route / moe_route_indices.
//
// Top-k over the router logits with a softmax over the k chosen scores
// ("从零理解 MoE 算子" §3), then the routing map, tokens per expert, the
// exclusive/inclusive prefixes (group_list, §7) and the expert-major,
// token-ascending sorted_indices of a masked_select over the transposed
// routing map ("token dispatcher + fuse_a2a" §1.1), with its inverse slot_pos.
//
// Three kernels, no inter-block waiting:
//   R1  one warp per token: top-k by repeated warp arg-max over order-
//       preserving 64-bit keys (value, then lower id), fp32 softmax, routing
//       map row, and a per-block expert histogram (shared-memory integer
//       atomics: order-independent).  The index-only variant validates given
//       choices instead.
//   R2  one thread per (expert, row group): turns the [blocks x E] histogram
//       into per-block exclusive prefixes in place and writes counts[E]; block
//       0 also folds the per-block error flags into the workspace status.
//   R3  one block per token block: scans counts into offsets, ranks its
//       tokens' choices stably (warp-serial groups of 32/k tokens resolved
//       with __match_any_sync), adds the block and warp prefixes and scatters
//       slot_pos, sorted_indices and permuted_probs.
// Position of (t, e) = offsets[e] + #{t' < t : e in topk(t')}: exact integer
// arithmetic, so the result is bit-exact and independent of scheduling.
#include <cmath>

#include "common.cuh"
#include "route_fast.cuh"

namespace moe {
namespace {

constexpr int kTokensPerBlock = 128;
constexpr int kThreads = 512;                              // R3 and the check kernel
constexpr int kWarps = kThreads / 32;
constexpr int kTokensPerWarp = kTokensPerBlock / kWarps;   // R3: 8 tokens per warp
constexpr uint32_t kFull = 0xFFFFFFFFu;


__host__ __device__ inline int64_t num_blocks(int64_t T) {
    return (T + kTokensPerBlock - 1) / kTokensPerBlock;
}

// [B rows x (E+1)] block histograms (column E: error flags), then one row of
// raw per-expert totals written by the scan kernel when it runs.
size_t hist_bytes(int64_t T, int E) {
    return align_up(size_t(num_blocks(T) + 1) * size_t(E + 1) * sizeof(int32_t), kWsAlign);
}

// Order-preserving 32-bit key of a float: larger value -> larger key.  -0 is
// folded onto +0 so the two compare equal (ties then go to the lower id).
// Every finite value maps above 0, which marks an empty or taken entry.
__device__ __forceinline__ uint32_t value_key(float f) {
    uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_value(uint32_t u) {
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// ------------------------------------------------------------------------ R1

// Block size of R1 for NV logits per lane (register budget: at most 64
// registers per thread at 1024 threads).
__host__ __device__ constexpr int topk_threads(int nv) {
    return nv <= 8 ? 1024 : nv <= 16 ? 512 : 256;
}

// GROUPED: group-limited routing ("从零理解 MoE 算子" §21).  The E experts form
// n_groups consecutive groups (n_groups <= 32, one lane per group); a group's
// score is its largest logit; the topk_groups best groups (equal scores: the
// lower group id) are kept and the experts of the others are masked before
// the top-k.
template <int NV, bool GROUPED>  // logits per lane: expert e = v*32 + lane, v < NV
__global__ void __launch_bounds__(topk_threads(NV))
route_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                  uint8_t* __restrict__ routing_map, int32_t* __restrict__ hist,
                  int n_groups, int topk_groups) {
    constexpr int kTopkThreads = topk_threads(NV);
    constexpr int kTopkWarps = kTopkThreads / 32;
    __shared__ int s_hist[kMaxExperts];
    for (int e = threadIdx.x; e < E; e += kTopkThreads) s_hist[e] = 0;
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t t0 = int64_t(blockIdx.x) * kTokensPerBlock;

    // each warp walks tokens warp, warp+kTopkWarps, ... of the block; the next
    // token's logits are loaded while the current one is ranked
    float cur[NV], nxt[NV];
    auto load_row = [&](int64_t t, float* dst) {
        const float* row = logits + t * E;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int e = v * 32 + lane;
            dst[v] = e < E ? __ldcs(row + e) : 0.0f;
        }
    };
    if (t0 + warp < T) load_row(t0 + warp, cur);
    for (int i = warp; i < kTokensPerBlock; i += kTopkWarps) {
        const int64_t t = t0 + i;
        if (t >= T) break;
        const bool more = i + kTopkWarps < kTokensPerBlock && t + kTopkWarps < T;
        if (more) load_row(t + kTopkWarps, nxt);
        uint32_t key[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int e = v * 32 + lane;
            key[v] = e < E ? value_key(cur[v]) : 0u;
        }
        if (GROUPED) {
            const int gsize = E / n_groups;
            int gv[NV];
#pragma unroll
            for (int v = 0; v < NV; ++v) gv[v] = (v * 32 + lane) / gsize;
            uint32_t cand = 0;                     // lane g: group g's score
            for (int g = 0; g < n_groups; ++g) {
                uint32_t local = 0;
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    if (gv[v] == g && key[v] > local) local = key[v];
                const uint32_t m = __reduce_max_sync(kFull, local);
                if (lane == g) cand = m;
            }
            uint32_t kept = 0;                     // bit g: group g kept
            for (int i = 0; i < topk_groups; ++i) {
                const uint32_t m = __reduce_max_sync(kFull, cand);
                const int g = int(__reduce_min_sync(kFull, cand == m ? uint32_t(lane) : 0xFFFFFFFFu));
                kept |= 1u << g;
                if (lane == g) cand = 0;
            }
#pragma unroll
            for (int v = 0; v < NV; ++v)
                if (!((kept >> gv[v]) & 1u)) key[v] = 0;   // padding lanes are 0 already
        }
        // this lane's two best entries (largest key, lowest v = lowest id on
        // ties): the head bk/bv and the runner-up b2/v2
        uint32_t bk = 0, b2 = 0;
        int bv = 0, v2 = 0;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            if (key[v] > bk) {
                b2 = bk; v2 = bv; bk = key[v]; bv = v;
            } else if (key[v] > b2) {
                b2 = key[v]; v2 = v;
            }
        }
        bool have2 = true;       // b2/v2 is the runner-up of what is left

        uint32_t taken = 0;      // bit v: my expert v*32+lane was chosen
        int my_e = -1;           // lane j keeps slot j
        float my_val = 0.0f;
        for (int j = 0; j < k; ++j) {
            // winner: the largest value, then the lowest expert id holding it
            const uint32_t m = __reduce_max_sync(kFull, bk);
            const int e = int(__reduce_min_sync(kFull, bk == m ? uint32_t(bv * 32 + lane) : 0xFFFFFFFFu));
            if (lane == j) { my_e = e; my_val = key_to_value(m); }
            if ((e & 31) == lane) {            // the owner drops the winner
                taken |= 1u << bv;
                if (have2) {                   // the runner-up is the new head
                    bk = b2;
                    bv = v2;
                    have2 = false;
                } else {                       // a second pop: rescan what is left
                    bk = 0; bv = 0; b2 = 0; v2 = 0;
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        if ((taken >> v) & 1u) continue;
                        if (key[v] > bk) {
                            b2 = bk; v2 = bv; bk = key[v]; bv = v;
                        } else if (key[v] > b2) {
                            b2 = key[v]; v2 = v;
                        }
                    }
                    have2 = true;
                }
            }
        }
        // softmax over the k chosen scores, stabilised by the largest (slot 0)
        const float s0 = __shfl_sync(kFull, my_val, 0);
        const float ex = lane < k ? expf(my_val - s0) : 0.0f;
        float total = ex;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(kFull, total, off);
        if (lane < k) {
            topk_idx[t * k + lane] = my_e;
            topk_w[t * k + lane] = ex / total;
            atomicAdd(&s_hist[my_e], 1);
        }
        if (routing_map) {
            uint8_t* mrow = routing_map + t * E;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int e = v * 32 + lane;
                if (e < E) mrow[e] = uint8_t((taken >> v) & 1u);
            }
        }
        if (more) {
#pragma unroll
            for (int v = 0; v < NV; ++v) cur[v] = nxt[v];
        }
    }
    __syncthreads();
    int32_t* h = hist + int64_t(blockIdx.x) * (E + 1);
    for (int e = threadIdx.x; e < E; e += kTopkThreads) h[e] = s_hist[e];
    if (threadIdx.x == 0) h[E] = 0;
}

// Slot j of a token is valid if its id is in [0, E) and no earlier slot of the
// same token names it.  *bad is set for an id outside [-1, E) or a repeat.
__device__ __forceinline__ bool slot_valid(const int32_t* ids, int j, int E, bool* bad) {
    const int e = ids[j];
    if (e == -1) return false;
    if (e < 0 || e >= E) { *bad = true; return false; }
    for (int q = 0; q < j; ++q)
        if (ids[q] == e) { *bad = true; return false; }
    return true;
}

// R1 for given choices: validate, histogram, routing map.
__global__ void __launch_bounds__(kThreads)
route_check_kernel(const int32_t* __restrict__ topk_idx, int64_t T, int E, int k,
                   uint8_t* __restrict__ routing_map, int32_t* __restrict__ hist) {
    extern __shared__ int32_t smem[];
    int* s_hist = smem;                       // [E]
    int32_t* s_idx = smem + E;                // [kTokensPerBlock * k]
    __shared__ int s_bad;
    const int64_t t0 = int64_t(blockIdx.x) * kTokensPerBlock;
    const int nt = int(min64(kTokensPerBlock, T - t0));
    for (int e = threadIdx.x; e < E; e += kThreads) s_hist[e] = 0;
    for (int i = threadIdx.x; i < nt * k; i += kThreads) s_idx[i] = topk_idx[t0 * k + i];
    if (threadIdx.x == 0) s_bad = 0;
    if (routing_map) {
        uint8_t* m = routing_map + t0 * E;
        for (int64_t i = threadIdx.x; i < int64_t(nt) * E; i += kThreads) m[i] = 0;
    }
    __syncthreads();
    bool bad = false;
    for (int i = threadIdx.x; i < nt * k; i += kThreads) {
        const int tl = i / k, j = i % k;
        if (slot_valid(s_idx + tl * k, j, E, &bad)) {
            const int e = s_idx[i];
            atomicAdd(&s_hist[e], 1);
            if (routing_map) routing_map[(t0 + tl) * E + e] = 1;
        }
    }
    if (bad) atomicOr(&s_bad, 1);
    __syncthreads();
    int32_t* h = hist + int64_t(blockIdx.x) * (E + 1);
    for (int e = threadIdx.x; e < E; e += kThreads) h[e] = s_hist[e];
    if (threadIdx.x == 0) h[E] = s_bad;
}

// ------------------------------------------------------------------------ R2
// Block x owns experts [32x, 32x+32); thread (g, c) owns expert 32x+c and
// the row group g of the histogram.
__global__ void __launch_bounds__(1024)
route_scan_kernel(int32_t* __restrict__ hist, int64_t B, int E, WsHeader* __restrict__ header) {
    wait_for_predecessor();
    __shared__ int32_t s_part[32][33];
    const int c = threadIdx.x & 31, g = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + c;
    const int64_t rows = (B + 31) / 32;
    const int64_t b0 = min64(B, g * rows), b1 = min64(B, b0 + rows);
    int32_t sum = 0;
    if (e < E)
        for (int64_t b = b0; b < b1; ++b) sum += hist[b * (E + 1) + e];
    s_part[g][c] = sum;
    __syncthreads();
    int32_t run = 0;
    for (int q = 0; q < g; ++q) run += s_part[q][c];
    if (e < E) {
        for (int64_t b = b0; b < b1; ++b) {
            const int32_t v = hist[b * (E + 1) + e];
            hist[b * (E + 1) + e] = run;
            run += v;
        }
        if (g == 31) hist[B * (E + 1) + e] = run;      // raw totals row
    }
    if (blockIdx.x == 0) {                   // fold the per-block error flags
        __shared__ int s_bad;
        if (threadIdx.x == 0) s_bad = 0;
        __syncthreads();
        int bad = 0;
        for (int64_t b = threadIdx.x; b < B; b += blockDim.x) bad |= hist[b * (E + 1) + E];
        if (bad) atomicOr(&s_bad, 1);
        __syncthreads();
        if (threadIdx.x == 0) {
            header->status = s_bad ? MOE_ERR_DEVICE_CHECK : MOE_OK;
            header->detail = 0;
        }
    }
}

// ------------------------------------------------------------------------ R3

// Exclusive scan of n <= 1024 ints held in s_in into s_out[0..n] (s_out[n]
// = total).  All kThreads threads must call it.
__device__ void block_exclusive_scan(const int32_t* s_in, int32_t* s_out, int n) {
    __shared__ int32_t s_warp[kWarps];
    constexpr int kPer = kMaxExperts / kThreads;     // items per thread
    const int base = threadIdx.x * kPer;
    int32_t v[kPer];
    int32_t local = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        v[i] = base + i < n ? s_in[base + i] : 0;
        local += v[i];
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int32_t wpre = 0;
    for (int q = 0; q < warp; ++q) wpre += s_warp[q];
    int32_t run = wpre + incl - local;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        if (base + i < n) s_out[base + i] = run;
        run += v[i];
    }
    if (threadIdx.x == kThreads - 1) {
        int32_t total = 0;
        for (int q = 0; q < kWarps; ++q) total += s_warp[q];
        s_out[n] = total;
    }
    __syncthreads();
}

// FUSED: this kernel also does R2's work (B <= kFusedMaxBlocks): every block
// sums the raw histogram rows itself -- the rows before it for its own
// prefix, all rows for the counts -- and block 0 publishes counts and the
// status word.  Otherwise `hist` already holds R2's per-block prefixes.
constexpr int kFusedMaxBlocks = 256;

// Layout of the permuted rows ("从零理解 MoE 算子" §18 capacity, the
// drop_and_pad branch of "token dispatcher + fuse_a2a" §1.1, DeepEP's
// expert_alignment): an expert keeps its first `capacity` tokens in token
// order (capacity 0: all); its segment is `capacity` rows when `pad`, else its
// kept count rounded up to a multiple of `alignment`.  max_rows bounds the
// rows the outputs may hold.
struct Layout {
    int capacity;
    int pad;
    int alignment;
    int64_t max_rows;
};

template <bool FUSED>
__global__ void __launch_bounds__(kThreads)
route_scatter_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
                     int64_t T, int E, int k, bool check_ids,
                     const int32_t* __restrict__ hist, int32_t* __restrict__ counts,
                     int32_t* __restrict__ offsets, int32_t* __restrict__ group_list,
                     int32_t* __restrict__ sorted_indices, int32_t* __restrict__ slot_pos,
                     float* __restrict__ permuted_probs, WsHeader* __restrict__ header,
                     Layout lay) {
    wait_for_predecessor();
    extern __shared__ int32_t smem[];
    int32_t* s_cnt = smem;                                   // [kWarps][E] -> warp prefixes
    int32_t* s_off = s_cnt + kWarps * E;                     // [E+1]
    int32_t* s_bpre = s_off + (E + 1);                       // [E]
    int32_t* s_kept = s_bpre + E;                            // [E]
    int32_t* s_idx = s_kept + E;                             // [kTokensPerBlock*k]
    int32_t* s_rank = s_idx + kTokensPerBlock * k;           // [kTokensPerBlock*k]
    float* s_w = reinterpret_cast<float*>(s_rank + kTokensPerBlock * k);   // [kTokensPerBlock*k]
    __shared__ int s_bad;

    const int64_t B = num_blocks(T);
    const int64_t t0 = int64_t(blockIdx.x) * kTokensPerBlock;
    const int nt = int(max64(0, min64(kTokensPerBlock, T - t0)));

    // every global read this block needs, issued before the first barrier
    for (int i = threadIdx.x; i < nt * k; i += kThreads) {
        s_idx[i] = topk_idx[t0 * k + i];
        if (permuted_probs) s_w[i] = topk_w[t0 * k + i];
    }
    if (FUSED) {
        // P threads per expert column, each summing every P-th row with 16
        // independent loads in flight; partial sums meet in s_cnt (scratch
        // until it is zeroed below)
        const int P = E >= kThreads ? 1 : (kThreads / E >= 8 ? 8 : kThreads / E >= 4 ? 4 :
                                           kThreads / E >= 2 ? 2 : 1);
        int32_t* s_tot = s_cnt;             // [P][E]
        int32_t* s_bef = s_cnt + P * E;     // [P][E]
        for (int id = threadIdx.x; id < P * E; id += kThreads) {
            const int e = id % E, part = id / E;
            int32_t before = 0, total = 0;
            for (int64_t b0 = part; b0 < B; b0 += 16 * P) {
                int32_t c[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int64_t b = b0 + int64_t(u) * P;
                    c[u] = b < B ? hist[b * (E + 1) + e] : 0;
                }
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    total += c[u];
                    before += b0 + int64_t(u) * P < int64_t(blockIdx.x) ? c[u] : 0;
                }
            }
            s_tot[part * E + e] = total;
            s_bef[part * E + e] = before;
        }
        if (blockIdx.x == 0) {
            int bad = 0;
            for (int64_t b = threadIdx.x; b < B; b += kThreads) bad |= hist[b * (E + 1) + E];
            if (threadIdx.x == 0) s_bad = 0;
            __syncthreads();
            if (bad) atomicOr(&s_bad, 1);
        }
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += kThreads) {
            int32_t before = 0, total = 0;
            for (int q = 0; q < P; ++q) {
                total += s_tot[q * E + e];
                before += s_bef[q * E + e];
            }
            s_bpre[e] = before;
            s_off[e] = total;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < kWarps * E; i += kThreads) s_cnt[i] = 0;
    } else {
        const bool has_hist = t0 < T;
        for (int e = threadIdx.x; e < E; e += kThreads) {
            s_bpre[e] = has_hist ? hist[int64_t(blockIdx.x) * (E + 1) + e] : 0;
            s_off[e] = hist[B * (E + 1) + e];              // raw totals from the scan kernel
        }
        for (int i = threadIdx.x; i < kWarps * E; i += kThreads) s_cnt[i] = 0;
    }
    __syncthreads();
    // kept tokens and segment length of every expert
    for (int e = threadIdx.x; e < E; e += kThreads) {
        const int32_t total = s_off[e];
        const int32_t kept = lay.capacity > 0 && total > lay.capacity ? lay.capacity : total;
        s_kept[e] = kept;
        s_off[e] = lay.pad ? lay.capacity : (kept + lay.alignment - 1) / lay.alignment * lay.alignment;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += kThreads) counts[e] = s_kept[e];
        if (FUSED && threadIdx.x == 0) {
            header->status = s_bad ? MOE_ERR_DEVICE_CHECK : MOE_OK;
            header->detail = 0;
        }
    }
    // offsets = exclusive scan of the segments (every block recomputes it)
    block_exclusive_scan(s_off, s_off, E);
    const bool overflow = int64_t(s_off[E]) > lay.max_rows;
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e <= E; e += kThreads) offsets[e] = s_off[e];
        for (int e = threadIdx.x; e < E; e += kThreads) group_list[e] = s_off[e + 1];
        if (overflow && threadIdx.x == 0) {
            header->status = MOE_ERR_DEVICE_CHECK;     // rows past max_rows are not written
            header->detail = 1;
        }
    }
    if (check_ids) {
        bool bad = false;   // already reported by the check kernel
        for (int i = threadIdx.x; i < nt * k; i += kThreads) {
            const int tl = i / k, j = i % k;
            s_rank[i] = slot_valid(s_idx + tl * k, j, E, &bad) ? s_idx[i] : -1;  // staged
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nt * k; i += kThreads) s_idx[i] = s_rank[i];
        __syncthreads();
    }

    // warp-serial stable ranking: warp w owns tokens [w*TPW, (w+1)*TPW) of the
    // block and walks them in order, G = 32/k tokens per step
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = 32 / k;
    const int ti = lane / k, j = lane % k;
    int32_t* cnt = s_cnt + warp * E;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int base = warp * kTokensPerWarp; base < (warp + 1) * kTokensPerWarp; base += G) {
        const int tl = base + ti;
        const bool active = ti < G && tl < (warp + 1) * kTokensPerWarp && tl < nt;
        const int e = active ? s_idx[tl * k + j] : -1;
        const bool valid = e >= 0;
        const unsigned grp = __match_any_sync(kFull, valid ? e : -2 - lane);
        const int before = __popc(grp & lt_mask);
        int32_t r = 0;
        if (valid) r = cnt[e] + before;
        __syncwarp();
        if (valid) {
            s_rank[tl * k + j] = r;
            if ((grp >> lane) == 1u) cnt[e] += __popc(grp);   // highest lane of the group
        }
        __syncwarp();
    }
    __syncthreads();
    // per-expert exclusive prefix across warps (in place)
    for (int e = threadIdx.x; e < E; e += kThreads) {
        int32_t run = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int32_t c = s_cnt[w * E + e];
            s_cnt[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nt * k; i += kThreads) {
        const int tl = i / k;
        const int e = s_idx[i];
        const int64_t t = t0 + tl;
        const int32_t rank = e < 0 ? 0 : s_bpre[e] + s_cnt[(tl / kTokensPerWarp) * E + e] + s_rank[i];
        const int64_t pos = e < 0 ? -1 : int64_t(s_off[e]) + rank;
        if (e < 0 || (lay.capacity > 0 && rank >= lay.capacity) || pos >= lay.max_rows) {
            slot_pos[t * k + (i % k)] = -1;                 // empty, dropped or out of room
            continue;
        }
        slot_pos[t * k + (i % k)] = int32_t(pos);
        sorted_indices[pos] = int32_t(t);
        if (permuted_probs) permuted_probs[pos] = s_w[i];
    }
    // padding rows inside the segments, then every row from offsets[E] on
    for (int e = blockIdx.x; e < E; e += gridDim.x) {
        const int64_t p1 = min64(s_off[e + 1], lay.max_rows);
        for (int64_t p = int64_t(s_off[e]) + s_kept[e] + threadIdx.x; p < p1; p += kThreads) {
            sorted_indices[p] = -1;
            if (permuted_probs) permuted_probs[p] = 0.0f;
        }
    }
    for (int64_t p = min64(s_off[E], lay.max_rows) + int64_t(blockIdx.x) * kThreads + threadIdx.x;
         p < lay.max_rows; p += int64_t(gridDim.x) * kThreads) {
        sorted_indices[p] = -1;
        if (permuted_probs) permuted_probs[p] = 0.0f;
    }
}

size_t scatter_smem_bytes(int E, int k) {
    return sizeof(int32_t) * (size_t(kWarps) * E + (E + 1) + 2 * size_t(E) +
                              3 * size_t(kTokensPerBlock) * k);
}

size_t check_smem_bytes(int E, int k) {
    return sizeof(int32_t) * (size_t(E) + size_t(kTokensPerBlock) * k);
}

moe_status_t validate_sizes(int64_t T, int E, int k) {
    if (T < 0 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > kMaxTopK || k > E) return MOE_ERR_UNSUPPORTED;
    if (T * int64_t(k) >= (int64_t(1) << 31) || T * int64_t(E) >= (int64_t(1) << 40))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

template <int NV>
void launch_topk(const float* logits, int64_t T, int E, int k, int32_t* topk_idx, float* topk_w,
                 uint8_t* routing_map, int32_t* hist, int n_groups, int topk_groups,
                 cudaStream_t s) {
    if (n_groups > 0)
        route_topk_kernel<NV, true><<<unsigned(num_blocks(T)), topk_threads(NV), 0, s>>>(
            logits, T, E, k, topk_idx, topk_w, routing_map, hist, n_groups, topk_groups);
    else
        route_topk_kernel<NV, false><<<unsigned(num_blocks(T)), topk_threads(NV), 0, s>>>(
            logits, T, E, k, topk_idx, topk_w, routing_map, hist, 0, 0);
}

moe_status_t finish_route(const int32_t* topk_idx, const float* topk_w, int64_t T, int E, int k,
                          bool check_ids, int32_t* hist, WsHeader* header, int32_t* counts,
                          int32_t* offsets, int32_t* group_list, int32_t* sorted_indices,
                          int32_t* slot_pos, float* permuted_probs, cudaStream_t s,
                          Layout lay = Layout{0, 0, 1, -1}) {
    const int64_t B = num_blocks(T);
    const bool fused = B <= kFusedMaxBlocks;
    if (lay.max_rows < 0) lay.max_rows = T * k;
    if (!fused && launch_dependent(route_scan_kernel, unsigned((E + 31) / 32), 1024, 0, s, hist,
                                   B, E, header) != cudaSuccess)
        return MOE_ERR_CUDA;
    const size_t smem = scatter_smem_bytes(E, k);
    const int max_smem = int(scatter_smem_bytes(kMaxExperts, kMaxTopK));
    if (!opt_in_smem((const void*)route_scatter_kernel<true>, max_smem) ||
        !opt_in_smem((const void*)route_scatter_kernel<false>, max_smem))
        return MOE_ERR_CUDA;
    const cudaError_t err = fused
        ? launch_dependent(route_scatter_kernel<true>, unsigned(B > 0 ? B : 1), kThreads, smem, s,
                           topk_idx, topk_w, T, E, k, check_ids, (const int32_t*)hist, counts,
                           offsets, group_list, sorted_indices, slot_pos, permuted_probs, header,
                           lay)
        : launch_dependent(route_scatter_kernel<false>, unsigned(B > 0 ? B : 1), kThreads, smem, s,
                           topk_idx, topk_w, T, E, k, check_ids, (const int32_t*)hist, counts,
                           offsets, group_list, sorted_indices, slot_pos, permuted_probs, header,
                           lay);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Scratch after the header: the larger of what the general kernels and the
// route_fast kernels (up to 256 experts) need.
size_t route_hist_bytes(int64_t T, int E) {
    const size_t a = hist_bytes(T, E);
    const size_t b = E <= kFastMaxExperts ? fast_hist_bytes(T, E) : 0;
    return a > b ? a : b;
}

moe_status_t check_workspace(const void* ws, size_t ws_bytes, int64_t T, int E) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kWsAlign - 1))) return MOE_ERR_WORKSPACE;
    if (ws_bytes < kWsAlign + route_hist_bytes(T, E)) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_route_workspace_size(int64_t T, int E, int k, size_t* bytes) {
    if (!bytes) return MOE_ERR_INVALID_ARG;
    const moe_status_t st = validate_sizes(T, E, k);
    if (st != MOE_OK) return st;
    *bytes = kWsAlign + route_hist_bytes(T, E);
    return MOE_OK;
}

namespace moe {
namespace {
moe_status_t route_from_logits(const float* logits, int64_t T, int E, int k, int n_groups,
                               int topk_groups, int32_t* topk_idx, float* topk_w,
                               int32_t* counts, int32_t* offsets, int32_t* group_list,
                               int32_t* sorted_indices, int32_t* slot_pos, float* permuted_probs,
                               uint8_t* routing_map, void* workspace, size_t workspace_bytes,
                               void* stream) {
    moe_status_t st = validate_sizes(T, E, k);
    if (st != MOE_OK) return st;
    if (!counts || !offsets || !group_list) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !topk_idx || !topk_w || !sorted_indices || !slot_pos ||
                  !permuted_probs))
        return MOE_ERR_INVALID_ARG;
    st = check_workspace(workspace, workspace_bytes, T, E);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsHeader* header = static_cast<WsHeader*>(workspace);
    int32_t* hist = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + kWsAlign);
    if (fast_route_supported(E, n_groups))
        return fast_route(logits, T, E, k, n_groups, topk_groups, topk_idx, topk_w, counts,
                          offsets, group_list, sorted_indices, slot_pos, permuted_probs,
                          routing_map, header, hist, s);
    if (T > 0) {
        const int nv = (E + 31) / 32;
        const int g = n_groups, kg = topk_groups;
        if (nv <= 1) launch_topk<1>(logits, T, E, k, topk_idx, topk_w, routing_map, hist, g, kg, s);
        else if (nv <= 2) launch_topk<2>(logits, T, E, k, topk_idx, topk_w, routing_map, hist, g, kg, s);
        else if (nv <= 4) launch_topk<4>(logits, T, E, k, topk_idx, topk_w, routing_map, hist, g, kg, s);
        else if (nv <= 8) launch_topk<8>(logits, T, E, k, topk_idx, topk_w, routing_map, hist, g, kg, s);
        else if (nv <= 16) launch_topk<16>(logits, T, E, k, topk_idx, topk_w, routing_map, hist, g, kg, s);
        else launch_topk<32>(logits, T, E, k, topk_idx, topk_w, routing_map, hist, g, kg, s);
        if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    }
    return finish_route(topk_idx, topk_w, T, E, k, false, hist, header, counts, offsets,
                        group_list, sorted_indices, slot_pos, permuted_probs, s);
}
}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_route(const float* logits, int64_t T, int E, int k,
                                  int32_t* topk_idx, float* topk_w, int32_t* counts,
                                  int32_t* offsets, int32_t* group_list, int32_t* sorted_indices,
                                  int32_t* slot_pos, float* permuted_probs, uint8_t* routing_map,
                                  void* workspace, size_t workspace_bytes, void* stream) {
    MOE_TRACE(__func__);
    return route_from_logits(logits, T, E, k, 0, 0, topk_idx, topk_w, counts, offsets,
                             group_list, sorted_indices, slot_pos, permuted_probs, routing_map,
                             workspace, workspace_bytes, stream);
}

extern "C" moe_status_t moe_route_grouped(const float* logits, int64_t T, int E, int k,
                                          int n_groups, int topk_groups, int32_t* topk_idx,
                                          float* topk_w, int32_t* counts, int32_t* offsets,
                                          int32_t* group_list, int32_t* sorted_indices,
                                          int32_t* slot_pos, float* permuted_probs,
                                          uint8_t* routing_map, void* workspace,
                                          size_t workspace_bytes, void* stream) {
    MOE_TRACE(__func__);
    if (n_groups < 1 || topk_groups < 1 || topk_groups > n_groups || E < 1 || E % n_groups != 0)
        return MOE_ERR_INVALID_ARG;
    if (n_groups > 32) return MOE_ERR_UNSUPPORTED;
    if (int64_t(k) > int64_t(topk_groups) * (E / n_groups)) return MOE_ERR_INVALID_ARG;
    return route_from_logits(logits, T, E, k, n_groups, topk_groups, topk_idx, topk_w, counts,
                             offsets, group_list, sorted_indices, slot_pos, permuted_probs,
                             routing_map, workspace, workspace_bytes, stream);
}

extern "C" moe_status_t moe_route_indices(const int32_t* topk_idx, const float* topk_w,
                                          int64_t T, int E, int k, int32_t* counts,
                                          int32_t* offsets, int32_t* group_list,
                                          int32_t* sorted_indices, int32_t* slot_pos,
                                          float* permuted_probs, uint8_t* routing_map,
                                          void* workspace, size_t workspace_bytes,
                                          void* stream) {
    MOE_TRACE(__func__);
    moe_status_t st = validate_sizes(T, E, k);
    if (st != MOE_OK) return st;
    if (!counts || !offsets || !group_list) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !sorted_indices || !slot_pos)) return MOE_ERR_INVALID_ARG;
    if (permuted_probs && !topk_w && T > 0) return MOE_ERR_INVALID_ARG;
    st = check_workspace(workspace, workspace_bytes, T, E);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsHeader* header = static_cast<WsHeader*>(workspace);
    int32_t* hist = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + kWsAlign);
    if (T > 0) {
        route_check_kernel<<<unsigned(num_blocks(T)), kThreads, check_smem_bytes(E, k), s>>>(
            topk_idx, T, E, k, routing_map, hist);
        if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    }
    return finish_route(topk_idx, topk_w, T, E, k, true, hist, header, counts, offsets,
                        group_list, sorted_indices, slot_pos, permuted_probs, s);
}

// ------------------------------------------------- capacity / padded layout

namespace moe {
namespace {
moe_status_t layout_rows(int64_t T, int E, int k, int capacity, int pad, int alignment,
                         int64_t* rows) {
    if (capacity < 0 || alignment < 1 || (pad && capacity < 1)) return MOE_ERR_INVALID_ARG;
    const int64_t r = pad ? int64_t(E) * capacity : T * k + int64_t(E) * (alignment - 1);
    if (r >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    *rows = r;
    return MOE_OK;
}
}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_expert_capacity(int64_t tokens, int top_k, int num_experts,
                                            double capacity_factor, int64_t* capacity) {
    if (!capacity || tokens < 0 || top_k < 1 || num_experts < 1 || !(capacity_factor > 0.0))
        return MOE_ERR_INVALID_ARG;
    const double c = std::ceil(double(tokens) * double(top_k) / double(num_experts) *
                               capacity_factor);
    if (c >= 2147483648.0) return MOE_ERR_UNSUPPORTED;
    *capacity = int64_t(c);
    return MOE_OK;
}

extern "C" moe_status_t moe_route_layout_rows(int64_t T, int E, int k, int capacity, int pad,
                                              int alignment, int64_t* max_rows) {
    if (!max_rows) return MOE_ERR_INVALID_ARG;
    const moe_status_t st = validate_sizes(T, E, k);
    if (st != MOE_OK) return st;
    return layout_rows(T, E, k, capacity, pad, alignment, max_rows);
}

extern "C" moe_status_t moe_route_layout(const int32_t* topk_idx, const float* topk_w, int64_t T,
                                         int E, int k, int capacity, int pad, int alignment,
                                         int64_t max_rows, int32_t* counts, int32_t* offsets,
                                         int32_t* group_list, int32_t* sorted_indices,
                                         int32_t* slot_pos, float* permuted_probs,
                                         void* workspace, size_t workspace_bytes, void* stream) {
    MOE_TRACE(__func__);
    moe_status_t st = validate_sizes(T, E, k);
    if (st != MOE_OK) return st;
    int64_t bound = 0;
    st = layout_rows(T, E, k, capacity, pad, alignment, &bound);
    if (st != MOE_OK) return st;
    if (max_rows < 0 || max_rows >= (int64_t(1) << 31)) return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets || !group_list) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !slot_pos)) return MOE_ERR_INVALID_ARG;
    if (max_rows > 0 && !sorted_indices) return MOE_ERR_INVALID_ARG;
    if (permuted_probs && !topk_w && T > 0) return MOE_ERR_INVALID_ARG;
    st = check_workspace(workspace, workspace_bytes, T, E);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsHeader* header = static_cast<WsHeader*>(workspace);
    int32_t* hist = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + kWsAlign);
    if (T > 0) {
        route_check_kernel<<<unsigned(num_blocks(T)), kThreads, check_smem_bytes(E, k), s>>>(
            topk_idx, T, E, k, nullptr, hist);
        if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    }
    return finish_route(topk_idx, topk_w, T, E, k, true, hist, header, counts, offsets,
                        group_list, sorted_indices, slot_pos, permuted_probs, s,
                        Layout{capacity, pad, alignment, max_rows});
}

// ------------------------------------------------------- no-allocation route
// moe_route for callers that cannot provide a workspace.  The histogram
// scratch lives in a fixed array in this library's device image instead of
// caller memory: every GPU that loads the library holds it until the process
// exits.  Nothing in it needs to start at zero -- each call writes every
// scratch byte before it reads it -- but all calls share it, so calls that
// overlap on the GPU (different streams, or different host threads) race.
#include <mutex>

static __device__ __align__(256) unsigned char g_route_scratch[MOE_ROUTE_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_scratch[kNoallocMaxDevices] = {};

// Device address of g_route_scratch on the current device, looked up once
// per device (host code cannot use the array's name as an address).
moe_status_t noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kNoallocMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_scratch[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_noalloc_scratch[dev] = p;
    }
    *out = g_noalloc_scratch[dev];
    return MOE_OK;
}
}  // namespace

extern "C" moe_status_t moe_route_noalloc(const float* logits, int64_t T, int E, int k,
                                          int32_t* topk_idx, float* topk_w, int32_t* counts,
                                          int32_t* offsets, int32_t* group_list,
                                          int32_t* sorted_indices, int32_t* slot_pos,
                                          float* permuted_probs, uint8_t* routing_map,
                                          void* stream) {
    MOE_TRACE(__func__);
    const moe_status_t st = validate_sizes(T, E, k);
    if (st != MOE_OK) return st;
    if (kWsAlign + route_hist_bytes(T, E) > MOE_ROUTE_NOALLOC_SCRATCH_BYTES)
        return MOE_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const moe_status_t sst = noalloc_scratch(&scratch);
    if (sst != MOE_OK) return sst;
    return moe_route(logits, T, E, k, topk_idx, topk_w, counts, offsets, group_list,
                     sorted_indices, slot_pos, permuted_probs, routing_map, scratch,
                     MOE_ROUTE_NOALLOC_SCRATCH_BYTES, stream);
}
