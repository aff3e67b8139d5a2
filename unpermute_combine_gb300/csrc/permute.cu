// permute.cu -- moe_permute, moe_sort_chunks, moe_chunk_idxs, moe_expert_scale.
//
// Row movement is HBM-bound: every source row is read once and every
// destination row written once, in 16-byte vectors, coalesced along the row.
// permute is token-centric ("token dispatcher + fuse_a2a" §1.1
// index_select, done in the dedup direction): one warp per token reads x[t]
// once and writes it to its k permuted rows.
#include "pipeline.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;     // 16-byte vectors in flight per lane

// One warp per token; lane l moves vectors l, l+32, ... of the row.
template <typename V>
__global__ void __launch_bounds__(kThreads)
permute_kernel(const V* __restrict__ x, int64_t T, int64_t nvec, int k, int64_t n_rows,
               const int32_t* __restrict__ slot_pos, V* __restrict__ out) {
    __shared__ int32_t s_pos[kWarps][kMaxTopK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t t = int64_t(blockIdx.x) * kWarps + warp; t < T;
         t += int64_t(gridDim.x) * kWarps) {
        if (lane < k) {
            const int32_t p = slot_pos[t * k + lane];
            s_pos[warp][lane] = (p >= 0 && p < n_rows) ? p : -1;
        }
        __syncwarp();
        const V* src = x + t * nvec;
        for (int64_t v0 = lane; v0 < nvec; v0 += 32 * kUnroll) {
            V d[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t v = v0 + 32 * u;
                if (v < nvec) d[u] = __ldcs(src + v);
            }
            for (int j = 0; j < k; ++j) {
                const int32_t p = s_pos[warp][j];
                if (p < 0) continue;
                V* dst = out + int64_t(p) * nvec;
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int64_t v = v0 + 32 * u;
                    if (v < nvec) __stcs(dst + v, d[u]);
                }
            }
        }
        __syncwarp();
    }
}

// Bulk-copy permute: one warp per CTA.  Lane 0 loads x[t] (in pieces of at
// most kPieceMax bytes) into a ring of shared-memory stages with bulk copies;
// once a piece has landed, lanes 0..k-1 each write it to their slot row with
// a bulk store, so a whole row leaves in one instruction per slot instead of
// one 16-byte store per lane.  A stage is refilled only after this lane's
// stores from it have finished reading it (bulk wait_group.read).  Waits on
// the stage mbarriers are bounded; a timeout stops the CTA and is recorded in
// *status.
//
// An optional side row (side_bytes > 0: the FP8 scale row of the token) rides
// in the same stage as the token's first piece and goes to the same slot rows
// of side_out, so one launch moves both.
constexpr int kPieceMax = 16384;
constexpr int kSideMax = 4096;
constexpr int kPermStages = 3;

__global__ void __launch_bounds__(32)
permute_bulk_kernel(const uint8_t* __restrict__ x, int64_t T, int64_t row_bytes, int piece,
                    int pieces, int k, int64_t n_rows, const int32_t* __restrict__ slot_pos,
                    uint8_t* __restrict__ out, const uint8_t* __restrict__ side,
                    uint32_t side_bytes, uint8_t* __restrict__ side_out,
                    uint32_t* __restrict__ status) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[kPermStages];
    const int lane = threadIdx.x;
    const int64_t total = T * pieces;
    const int64_t first = blockIdx.x;
    const int64_t my_items = first < total ? (total - first + gridDim.x - 1) / gridDim.x : 0;
    const uint32_t smem0 = smem_addr(smem);
    const uint32_t stage_bytes = uint32_t(piece) + side_bytes;
    if (lane == 0) {
        for (int s = 0; s < kPermStages; ++s) mbar_init(smem_addr(&full_bar[s]), 1);
        mbar_fence_init();
    }
    __syncwarp();

    auto item_coords = [&](int64_t q, int64_t& t, uint32_t& off, uint32_t& bytes) {
        const int64_t item = first + q * gridDim.x;
        t = item / pieces;
        off = uint32_t(item % pieces) * uint32_t(piece);
        bytes = uint32_t(min64(piece, row_bytes - off));
    };
    auto issue_load = [&](int64_t q) {
        int64_t t;
        uint32_t off, bytes;
        item_coords(q, t, off, bytes);
        const int s = int(q % kPermStages);
        const uint32_t fb = smem_addr(&full_bar[s]);
        const bool with_side = side_bytes != 0 && off == 0;
        mbar_expect_tx(fb, bytes + (with_side ? side_bytes : 0u));
        bulk_load(smem0 + uint32_t(s) * stage_bytes, x + t * row_bytes + off, bytes, fb);
        if (with_side)
            bulk_load(smem0 + uint32_t(s) * stage_bytes + uint32_t(piece), side + t * side_bytes,
                      side_bytes, fb);
    };
    auto slot_of = [&](int64_t q) -> int32_t {
        if (q >= my_items || lane >= k) return -1;
        int64_t t;
        uint32_t off, bytes;
        item_coords(q, t, off, bytes);
        const int32_t p = slot_pos[t * k + lane];
        return (p >= 0 && p < n_rows) ? p : -1;
    };

    if (lane == 0)
        for (int64_t q = 0; q < my_items && q < kPermStages; ++q) issue_load(q);
    int32_t p_cur = slot_of(0);
    bool failed = false;
    int64_t q_fail = 0;
    for (int64_t q = 0; q < my_items; ++q) {
        const int32_t p_next = slot_of(q + 1);               // in flight meanwhile
        const int s = int(q % kPermStages);
        const uint32_t ph = uint32_t(q / kPermStages) & 1u;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_addr(&full_bar[s]), ph))) {
            failed = true;
            q_fail = q;
            break;
        }
        int64_t t;
        uint32_t off, bytes;
        item_coords(q, t, off, bytes);
        if (p_cur >= 0) {
            bulk_store(out + int64_t(p_cur) * row_bytes + off, smem0 + uint32_t(s) * stage_bytes,
                       bytes);
            if (side_bytes != 0 && off == 0)
                bulk_store(side_out + int64_t(p_cur) * side_bytes,
                           smem0 + uint32_t(s) * stage_bytes + uint32_t(piece), side_bytes);
        }
        bulk_commit();
        // the stores of item q-1 have read their stage: refill it with item q-1+S
        bulk_wait_read<1>();
        __syncwarp();
        if (lane == 0 && q >= 1 && q - 1 + kPermStages < my_items) issue_load(q - 1 + kPermStages);
        p_cur = p_next;
    }
    bulk_wait_all();
    if (failed && lane == 0) {
        // loads issued but never consumed (items q_fail .. the last one
        // issued) may still be landing in this CTA's shared memory: wait for
        // each (bounded) before the CTA exits and the memory is reused
        const int64_t last = min64(my_items - 1, max64(kPermStages - 1, q_fail + kPermStages - 2));
        for (int64_t i = q_fail; i <= last; ++i)
            mbar_wait(smem_addr(&full_bar[i % kPermStages]), uint32_t(i / kPermStages) & 1u);
        if (status) atomicExch(status, uint32_t(MOE_ERR_TIMEOUT));
    }
}

int grid_for(const void* kernel, int threads, size_t smem, int64_t work_blocks) {
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t cap = int64_t(sm_count()) * per_sm;
    return int(work_blocks < cap ? (work_blocks > 0 ? work_blocks : 1) : cap);
}

// ----------------------------------------------------------------- sort_chunks
// Prep kernel (one block): validate the splits and the chunk order, then write
// per output chunk i: dst_start[i] (exclusive prefix of split_sizes[idx[i]],
// dst_start[C] = N) and src_start[i] (start row of chunk idx[i] in `in`).
struct ChunkPlan {
    int32_t* dst_start;   // [C+1]
    int32_t* src_start;   // [C]
    int32_t* src_prefix;  // [C+1] exclusive prefix of split_sizes in input order
};

constexpr int kPrepThreads = 1024;
constexpr int kMaxChunks = 65536;

__device__ int32_t block_scan_exclusive_1024(int32_t v, int32_t* s_warp, int32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t w = s_warp[lane];
        int32_t wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t o = __shfl_up_sync(0xFFFFFFFFu, wi, off);
            if (lane >= off) wi += o;
        }
        s_warp[lane] = wi - w;              // exclusive warp prefix
        if (lane == 31) s_warp[32] = wi;    // block total
    }
    __syncthreads();
    const int32_t r = s_warp[warp] + incl - v;
    *total = s_warp[32];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kPrepThreads)
sort_chunks_prep_kernel(const int32_t* __restrict__ split_sizes,
                        const int32_t* __restrict__ sorted_idxs, int C, int64_t N,
                        ChunkPlan plan, WsHeader* __restrict__ header) {
    __shared__ int32_t s_warp[33];
    __shared__ uint32_t s_seen[kMaxChunks / 32];
    __shared__ int s_bad;
    for (int i = threadIdx.x; i < (C + 31) / 32; i += kPrepThreads) s_seen[i] = 0;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    bool bad = false;
    for (int i = threadIdx.x; i < C; i += kPrepThreads) {
        const int32_t c = sorted_idxs[i];
        if (c < 0 || c >= C || split_sizes[i] < 0) { bad = true; continue; }
        const uint32_t bit = 1u << (c & 31);
        if (atomicOr(&s_seen[c >> 5], bit) & bit) bad = true;   // named twice
    }
    if (bad) atomicOr(&s_bad, 1);
    __syncthreads();
    // prefix of split_sizes in input order (64-bit guard against overflow)
    int64_t carry = 0;
    for (int base = 0; base < C; base += kPrepThreads) {
        const int i = base + threadIdx.x;
        const int32_t v = i < C ? split_sizes[i] : 0;
        int32_t total;
        const int32_t ex = block_scan_exclusive_1024(v, s_warp, &total);
        if (i < C) plan.src_prefix[i] = int32_t(carry + ex);
        carry += total;
    }
    if (threadIdx.x == 0) {
        plan.src_prefix[C] = int32_t(carry);
        if (carry != N) s_bad = 1;
    }
    __syncthreads();
    // prefix of split_sizes[idx[i]] in output order
    int64_t carry2 = 0;
    for (int base = 0; base < C; base += kPrepThreads) {
        const int i = base + threadIdx.x;
        int32_t c = i < C ? sorted_idxs[i] : 0;
        c = (c >= 0 && c < C) ? c : 0;
        const int32_t v = i < C ? split_sizes[c] : 0;
        int32_t total;
        const int32_t ex = block_scan_exclusive_1024(v, s_warp, &total);
        if (i < C) {
            plan.dst_start[i] = int32_t(carry2 + ex);
            plan.src_start[i] = plan.src_prefix[c];
        }
        carry2 += total;
    }
    if (threadIdx.x == 0) {
        plan.dst_start[C] = int32_t(carry2);
        header->status = s_bad ? MOE_ERR_DEVICE_CHECK : MOE_OK;
        header->detail = 0;
    }
}

// Copy kernel: each warp owns a contiguous range of output rows; it finds the
// chunk of its first row by binary search and walks forward.
template <typename V>
__global__ void __launch_bounds__(kThreads)
sort_chunks_copy_kernel(const V* __restrict__ in, int64_t N, int64_t nvec, int C,
                        ChunkPlan plan, const WsHeader* __restrict__ header,
                        V* __restrict__ out) {
    if (header->status != MOE_OK) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * kWarps;
    const int64_t gw = int64_t(blockIdx.x) * kWarps + warp;
    const int64_t per = (N + nwarps - 1) / nwarps;
    const int64_t r0 = gw * per, r1 = min64(N, r0 + per);
    if (r0 >= r1) return;
    // last chunk i with dst_start[i] <= r0
    int lo = 0, hi = C - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (plan.dst_start[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    int i = lo;
    int64_t chunk_end = plan.dst_start[i + 1];
    for (int64_t r = r0; r < r1; ++r) {
        while (r >= chunk_end) { ++i; chunk_end = plan.dst_start[i + 1]; }
        const int64_t s = plan.src_start[i] + (r - plan.dst_start[i]);
        const V* src = in + s * nvec;
        V* dst = out + r * nvec;
        for (int64_t v0 = lane; v0 < nvec; v0 += 32 * kUnroll) {
            V d[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t v = v0 + 32 * u;
                if (v < nvec) d[u] = __ldcs(src + v);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t v = v0 + 32 * u;
                if (v < nvec) __stcs(dst + v, d[u]);
            }
        }
    }
}

// ------------------------------------------------- sort_chunks, fused bulk
// Every chunk is one contiguous run of rows in the input and in the output,
// so for up to kFusedChunks chunks of 16-byte-multiple rows one launch does
// everything: each single-warp CTA builds and checks the chunk plan in shared
// memory (two warp scans over the C split sizes -- cheaper than a separate
// plan launch), then copies its share of the output as pieces of at most
// kScPiece bytes, each inside one chunk, through a ring of shared-memory
// stages with bulk copies (one bulk load and one bulk store per piece).
// Every CTA reaches the same verdict on the plan; an invalid plan writes
// nothing and CTA 0 records MOE_ERR_DEVICE_CHECK.  Launched as a
// programmatic dependent of the previous kernel in the stream.
constexpr int kFusedChunks = 1024;
constexpr int kScPiece = 16384;
constexpr int kScStages = 3;

__device__ __forceinline__ int32_t warp_incl_scan(int32_t v, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t o = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += o;
    }
    return v;
}

__global__ void __launch_bounds__(32)
sort_chunks_bulk_kernel(const uint8_t* __restrict__ in, int64_t N, int64_t row_bytes,
                        const int32_t* __restrict__ split_sizes,
                        const int32_t* __restrict__ sorted_idxs, int C, uint8_t* __restrict__ out,
                        WsHeader* __restrict__ header, uint32_t* __restrict__ status) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[kScStages];
    __shared__ int32_t s_srcpre[kFusedChunks];     // first input row of input chunk c
    __shared__ int32_t s_src[kFusedChunks];        // first input row of output chunk j
    __shared__ int32_t s_dst[kFusedChunks + 1];    // first output row of output chunk j
    __shared__ int32_t s_item[kFusedChunks + 1];   // first piece of output chunk j
    __shared__ uint32_t s_seen[kFusedChunks / 32];
    const int lane = threadIdx.x;
    const uint32_t full = 0xFFFFFFFFu;
    wait_for_predecessor();

    // ---- plan
    for (int i = lane; i < kFusedChunks / 32; i += 32) s_seen[i] = 0;
    bool bad = false;
    int64_t carry = 0;
    for (int base = 0; base < C; base += 32) {
        const int i = base + lane;
        int32_t v = i < C ? split_sizes[i] : 0;
        if (v < 0) { bad = true; v = 0; }
        const int32_t incl = warp_incl_scan(v, lane);
        if (i < C) s_srcpre[i] = int32_t(carry + incl - v);
        carry += __shfl_sync(full, incl, 31);
    }
    if (carry != N) bad = true;
    __syncwarp();
    int64_t rcarry = 0, icarry = 0;
    for (int base = 0; base < C; base += 32) {
        const int j = base + lane;
        int32_t rows = 0, c = -1;
        if (j < C) {
            c = sorted_idxs[j];
            if (c < 0 || c >= C) {
                bad = true;
                c = -1;
            } else {
                const uint32_t bit = 1u << (c & 31);
                if (atomicOr(&s_seen[c >> 5], bit) & bit) bad = true;     // named twice
                rows = max(split_sizes[c], 0);
            }
        }
        const int32_t items = int32_t((int64_t(rows) * row_bytes + kScPiece - 1) / kScPiece);
        const int32_t rincl = warp_incl_scan(rows, lane);
        const int32_t iincl = warp_incl_scan(items, lane);
        if (j < C) {
            s_dst[j] = int32_t(rcarry + rincl - rows);
            s_src[j] = c >= 0 ? s_srcpre[c] : 0;
            s_item[j] = int32_t(icarry + iincl - items);
        }
        rcarry += __shfl_sync(full, rincl, 31);
        icarry += __shfl_sync(full, iincl, 31);
    }
    if (lane == 0) {
        s_dst[C] = int32_t(rcarry);
        s_item[C] = int32_t(icarry);
    }
    bad = __any_sync(full, bad);
    if (blockIdx.x == 0 && lane == 0) {
        header->status = bad ? MOE_ERR_DEVICE_CHECK : MOE_OK;
        header->detail = 0;
    }
    if (bad) return;
    __syncwarp();

    // ---- copy
    const int64_t total = s_item[C];
    const int64_t first = blockIdx.x;
    const int64_t my_items = first < total ? (total - first + gridDim.x - 1) / gridDim.x : 0;
    const uint32_t smem0 = smem_addr(smem);
    if (lane == 0) {
        for (int st = 0; st < kScStages; ++st) mbar_init(smem_addr(&full_bar[st]), 1);
        mbar_fence_init();
    }
    __syncwarp();
    auto piece_of = [&](int64_t q, int64_t& src, int64_t& dst, uint32_t& bytes) {
        const int32_t item = int32_t(first + q * gridDim.x);
        int lo = 0, hi = C - 1;                        // last chunk starting at or before item
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_item[mid] <= item) lo = mid; else hi = mid - 1;
        }
        const int64_t off = int64_t(item - s_item[lo]) * kScPiece;
        const int64_t cbytes = int64_t(s_dst[lo + 1] - s_dst[lo]) * row_bytes;
        bytes = uint32_t(min64(kScPiece, cbytes - off));
        src = int64_t(s_src[lo]) * row_bytes + off;
        dst = int64_t(s_dst[lo]) * row_bytes + off;
    };
    auto issue_load = [&](int64_t q) {
        int64_t src, dst;
        uint32_t bytes;
        piece_of(q, src, dst, bytes);
        const int st = int(q % kScStages);
        const uint32_t fb = smem_addr(&full_bar[st]);
        mbar_expect_tx(fb, bytes);
        bulk_load(smem0 + uint32_t(st) * kScPiece, in + src, bytes, fb);
    };
    if (lane == 0)
        for (int64_t q = 0; q < my_items && q < kScStages; ++q) issue_load(q);
    bool failed = false;
    int64_t q_fail = 0;
    for (int64_t q = 0; q < my_items; ++q) {
        const int st = int(q % kScStages);
        const uint32_t ph = uint32_t(q / kScStages) & 1u;
        if (!__all_sync(full, mbar_wait(smem_addr(&full_bar[st]), ph))) {
            failed = true;
            q_fail = q;
            break;
        }
        if (lane == 0) {
            int64_t src, dst;
            uint32_t bytes;
            piece_of(q, src, dst, bytes);
            bulk_store(out + dst, smem0 + uint32_t(st) * kScPiece, bytes);
            bulk_commit();
            // the store of piece q-1 has read its stage: refill it with piece q-1+S
            bulk_wait_read<1>();
            if (q >= 1 && q - 1 + kScStages < my_items) issue_load(q - 1 + kScStages);
        }
        __syncwarp();
    }
    if (lane == 0) bulk_wait_all();
    if (failed && lane == 0) {
        // pieces loaded but never stored may still be landing in this CTA's
        // shared memory: wait for each (bounded) before the CTA exits
        const int64_t last = min64(my_items - 1, max64(kScStages - 1, q_fail + kScStages - 2));
        for (int64_t i = q_fail; i <= last; ++i)
            mbar_wait(smem_addr(&full_bar[i % kScStages]), uint32_t(i / kScStages) & 1u);
        if (status) atomicExch(status, uint32_t(MOE_ERR_TIMEOUT));
    }
}

size_t chunk_plan_bytes(int C) {
    return align_up(sizeof(int32_t) * (size_t(C + 1) * 2 + size_t(C)), kWsAlign);
}

ChunkPlan chunk_plan(void* ws, int C) {
    int32_t* base = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kWsAlign);
    return ChunkPlan{base, base + (C + 1), base + (C + 1) + C};
}

// -------------------------------------------------------------- expert scale
template <typename T>
__global__ void __launch_bounds__(kThreads)
expert_scale_kernel(const T* __restrict__ in, int64_t n_rows, int64_t H, int E,
                    const int32_t* __restrict__ offsets, const float* __restrict__ scale,
                    T* __restrict__ out) {
    __shared__ int32_t s_off[kMaxExperts + 1];
    __shared__ float s_scale[kMaxExperts];
    for (int e = threadIdx.x; e <= E; e += kThreads) s_off[e] = offsets[e];
    for (int e = threadIdx.x; e < E; e += kThreads) s_scale[e] = scale[e];
    __syncthreads();
    const int64_t rows = min64(n_rows, s_off[E]);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t p = int64_t(blockIdx.x) * kWarps + warp; p < rows;
         p += int64_t(gridDim.x) * kWarps) {
        int lo = 0, hi = E - 1;          // last e with offsets[e] <= p
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_off[mid] <= p) lo = mid; else hi = mid - 1;
        }
        const float s = s_scale[lo];
        for (int64_t h = lane; h < H; h += 32) {
            if constexpr (sizeof(T) == 4) {
                out[p * H + h] = __fmul_rn(in[p * H + h], s);
            } else {
                out[p * H + h] = uint16_t(mul_bf16_rn(bf16_to_f32(in[p * H + h]), s));
            }
        }
    }
}

// bf16 rows that are 16-byte multiples: one warp per row, 16-byte vectors,
// four in flight per lane; each element is the exact product rounded once
// (the same arithmetic as expert_scale_kernel).
__global__ void __launch_bounds__(kThreads)
expert_scale_vec_kernel(const uint4* __restrict__ in, int64_t n_rows, int64_t nvec, int E,
                        const int32_t* __restrict__ offsets, const float* __restrict__ scale,
                        uint4* __restrict__ out) {
    __shared__ int32_t s_off[kMaxExperts + 1];
    __shared__ float s_scale[kMaxExperts];
    for (int e = threadIdx.x; e <= E; e += kThreads) s_off[e] = offsets[e];
    for (int e = threadIdx.x; e < E; e += kThreads) s_scale[e] = scale[e];
    __syncthreads();
    const int64_t rows = min64(n_rows, s_off[E]);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t p = int64_t(blockIdx.x) * kWarps + warp; p < rows;
         p += int64_t(gridDim.x) * kWarps) {
        int lo = 0, hi = E - 1;          // last e with offsets[e] <= p
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_off[mid] <= p) lo = mid; else hi = mid - 1;
        }
        const float sc = s_scale[lo];
        const uint4* src = in + p * nvec;
        uint4* dst = out + p * nvec;
        for (int64_t v0 = lane; v0 < nvec; v0 += 32 * 4) {
            uint4 d[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t v = v0 + 32 * u;
                d[u] = v < nvec ? __ldcs(src + v) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t v = v0 + 32 * u;
                if (v >= nvec) break;
                const uint32_t w[4] = {d[u].x, d[u].y, d[u].z, d[u].w};
                uint32_t r[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    r[i] = mul_bf16_rn(bf16lo_to_f32(w[i]), sc) |
                           (mul_bf16_rn(bf16hi_to_f32(w[i]), sc) << 16);
                __stcs(dst + v, make_uint4(r[0], r[1], r[2], r[3]));
            }
        }
    }
}

// Zero the padding rows of a padded / aligned layout: expert e's rows
// [offsets[e] + counts[e], offsets[e+1]), clipped to max_rows.  One block per
// expert (grid-stride), 16-byte stores when the rows allow.
template <typename V>
__global__ void __launch_bounds__(kThreads)
fill_pad_rows_kernel(V* __restrict__ rows, int64_t max_rows, int64_t nvec,
                     const int32_t* __restrict__ offsets, const int32_t* __restrict__ counts,
                     int E) {
    for (int e = blockIdx.x; e < E; e += gridDim.x) {
        // first pad row and the segment end, kept inside [0, max_rows)
        const int64_t p0 = max64(int64_t(offsets[e]) + max64(counts[e], 0), 0);
        const int64_t p1 = min64(offsets[e + 1], max_rows);
        if (p0 >= p1) continue;
        const int64_t n = (p1 - p0) * nvec;
        V* base = rows + p0 * nvec;
        for (int64_t i = threadIdx.x; i < n; i += kThreads) base[i] = V{};
    }
}

// Rows of row_bytes (a multiple of 16, 16-byte aligned buffers) plus an
// optional side row of side_bytes (a multiple of 16, at most kSideMax).
bool launch_permute_bulk(const void* x, int64_t T, size_t row, int k, int64_t n_rows,
                         const int32_t* slot_pos, void* out, const void* side, size_t side_bytes,
                         void* side_out, cudaStream_t s) {
    const int pieces = int((row + kPieceMax - 1) / kPieceMax);
    const int piece = int(((row + pieces - 1) / pieces + 15) / 16 * 16);
    const size_t smem = size_t(kPermStages) * (size_t(piece) + side_bytes);
    if (!opt_in_smem((const void*)permute_bulk_kernel, kPermStages * (kPieceMax + kSideMax)))
        return false;
    const int64_t items = T * pieces;
    const int g = int(min64(items, int64_t(sm_count()) * 4));
    permute_bulk_kernel<<<g, 32, smem, s>>>(
        static_cast<const uint8_t*>(x), T, int64_t(row), piece, pieces, k, n_rows, slot_pos,
        static_cast<uint8_t*>(out), static_cast<const uint8_t*>(side), uint32_t(side_bytes),
        static_cast<uint8_t*>(side_out), device_status_word());
    return true;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_permute_fp8(const void* x_q, const float* scales, int64_t T,
                                        int64_t H, int block, int k, int64_t n_rows,
                                        const int32_t* slot_pos, void* out_q, float* out_scales,
                                        void* stream) {
    MOE_TRACE(__func__);
    if (T < 0 || H < 0 || k < 1 || n_rows < 0) return MOE_ERR_INVALID_ARG;
    if (block != 32 && block != 64 && block != 128 && block != 256) return MOE_ERR_UNSUPPORTED;
    if (H % block != 0) return MOE_ERR_INVALID_ARG;
    if (k > kMaxTopK || T * int64_t(k) >= (int64_t(1) << 31) || n_rows >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    if (T == 0 || H == 0 || n_rows == 0) return MOE_OK;
    if (!x_q || !scales || !slot_pos || !out_q || !out_scales) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t row = size_t(H), side = size_t(H / block) * sizeof(float);
    if (row % 16 == 0 && side % 16 == 0 && side <= size_t(kSideMax) && aligned16(x_q) &&
        aligned16(out_q) && aligned16(scales) && aligned16(out_scales)) {
        if (!launch_permute_bulk(x_q, T, row, k, n_rows, slot_pos, out_q, scales, side,
                                 out_scales, s))
            return MOE_ERR_CUDA;
        return launch_status();
    }
    // rows the bulk path cannot take: the two row sets one after the other
    const moe_status_t st = moe_permute(x_q, MOE_FP8_E4M3, T, H, k, n_rows, slot_pos, out_q,
                                        stream);
    if (st != MOE_OK) return st;
    return moe_permute(scales, MOE_F32, T, H / block, k, n_rows, slot_pos, out_scales, stream);
}

extern "C" moe_status_t moe_permute(const void* x, moe_dtype_t dtype, int64_t T, int64_t H, int k,
                                    int64_t n_rows, const int32_t* slot_pos, void* out,
                                    void* stream) {
    MOE_TRACE(__func__);
    if (!dtype_ok_move(dtype) || T < 0 || H < 0 || k < 1 || n_rows < 0) return MOE_ERR_INVALID_ARG;
    if (k > kMaxTopK || T * int64_t(k) >= (int64_t(1) << 31) || n_rows >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    if (T == 0 || H == 0 || n_rows == 0) return MOE_OK;
    if (!x || !slot_pos || !out) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t row = size_t(H) * elem_size(dtype);
    const int64_t blocks = (T + kWarps - 1) / kWarps;
    if (row % 16 == 0 && aligned16(x) && aligned16(out)) {
        if (!launch_permute_bulk(x, T, row, k, n_rows, slot_pos, out, nullptr, 0, nullptr, s))
            return MOE_ERR_CUDA;
    } else if (dtype == MOE_F32) {
        const int g = grid_for((const void*)permute_kernel<float>, kThreads, 0, blocks);
        permute_kernel<float><<<g, kThreads, 0, s>>>(
            static_cast<const float*>(x), T, H, k, n_rows, slot_pos, static_cast<float*>(out));
    } else if (dtype == MOE_BF16) {
        const int g = grid_for((const void*)permute_kernel<uint16_t>, kThreads, 0, blocks);
        permute_kernel<uint16_t><<<g, kThreads, 0, s>>>(
            static_cast<const uint16_t*>(x), T, H, k, n_rows, slot_pos, static_cast<uint16_t*>(out));
    } else {
        const int g = grid_for((const void*)permute_kernel<uint8_t>, kThreads, 0, blocks);
        permute_kernel<uint8_t><<<g, kThreads, 0, s>>>(
            static_cast<const uint8_t*>(x), T, H, k, n_rows, slot_pos, static_cast<uint8_t*>(out));
    }
    return launch_status();
}

extern "C" moe_status_t moe_sort_chunks_workspace_size(int C, size_t* bytes) {
    if (!bytes || C < 1) return MOE_ERR_INVALID_ARG;
    if (C > kMaxChunks) return MOE_ERR_UNSUPPORTED;
    *bytes = kWsAlign + chunk_plan_bytes(C);
    return MOE_OK;
}

extern "C" moe_status_t moe_sort_chunks(const void* in, moe_dtype_t dtype, int64_t N, int64_t H,
                                        const int32_t* split_sizes, const int32_t* sorted_idxs,
                                        int C, void* out, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    MOE_TRACE(__func__);
    if (!dtype_ok_move(dtype) || N < 0 || H < 0 || C < 1) return MOE_ERR_INVALID_ARG;
    if (C > kMaxChunks || N >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (!split_sizes || !sorted_idxs) return MOE_ERR_INVALID_ARG;
    if (N > 0 && H > 0 && (!in || !out)) return MOE_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kWsAlign - 1)) ||
        workspace_bytes < kWsAlign + chunk_plan_bytes(C))
        return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsHeader* header = static_cast<WsHeader*>(workspace);
    const size_t row_b = size_t(H) * elem_size(dtype);
    if (C <= kFusedChunks && row_b % 16 == 0 && (N == 0 || H == 0 || (aligned16(in) && aligned16(out)))) {
        if (!opt_in_smem((const void*)sort_chunks_bulk_kernel, kScStages * kScPiece))
            return MOE_ERR_CUDA;
        const int64_t pieces = (N * int64_t(row_b) + kScPiece - 1) / kScPiece + C;
        const int g = int(max64(1, min64(pieces, int64_t(sm_count()) * 3)));
        if (launch_dependent(sort_chunks_bulk_kernel, unsigned(g), 32, size_t(kScStages) * kScPiece,
                             s, static_cast<const uint8_t*>(in), N, int64_t(row_b), split_sizes,
                             sorted_idxs, C, static_cast<uint8_t*>(out), header,
                             device_status_word()) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    const ChunkPlan plan = chunk_plan(workspace, C);
    sort_chunks_prep_kernel<<<1, kPrepThreads, 0, s>>>(split_sizes, sorted_idxs, C, N, plan,
                                                      header);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
    if (N == 0 || H == 0) return MOE_OK;
    const size_t row = size_t(H) * elem_size(dtype);
    const int64_t want = (N + kWarps - 1) / kWarps;
    if (row % 16 == 0 && aligned16(in) && aligned16(out)) {
        const int g = grid_for((const void*)sort_chunks_copy_kernel<uint4>, kThreads, 0, want);
        sort_chunks_copy_kernel<uint4><<<g, kThreads, 0, s>>>(
            static_cast<const uint4*>(in), N, int64_t(row / 16), C, plan, header,
            static_cast<uint4*>(out));
    } else if (dtype == MOE_F32) {
        const int g = grid_for((const void*)sort_chunks_copy_kernel<float>, kThreads, 0, want);
        sort_chunks_copy_kernel<float><<<g, kThreads, 0, s>>>(
            static_cast<const float*>(in), N, H, C, plan, header, static_cast<float*>(out));
    } else if (dtype == MOE_BF16) {
        const int g = grid_for((const void*)sort_chunks_copy_kernel<uint16_t>, kThreads, 0, want);
        sort_chunks_copy_kernel<uint16_t><<<g, kThreads, 0, s>>>(
            static_cast<const uint16_t*>(in), N, H, C, plan, header,
            static_cast<uint16_t*>(out));
    } else {
        const int g = grid_for((const void*)sort_chunks_copy_kernel<uint8_t>, kThreads, 0, want);
        sort_chunks_copy_kernel<uint8_t><<<g, kThreads, 0, s>>>(
            static_cast<const uint8_t*>(in), N, H, C, plan, header, static_cast<uint8_t*>(out));
    }
    return launch_status();
}

extern "C" moe_status_t moe_chunk_idxs(int R, int L, int inverse, int32_t* idxs) {
    if (R < 1 || L < 1 || !idxs) return MOE_ERR_INVALID_ARG;
    if (int64_t(R) * L > kMaxChunks) return MOE_ERR_UNSUPPORTED;
    // Numbering an [A x B] grid row-major and reading it column by column
    // puts entry (a, b) = a*B + b at position b*A + a.
    for (int r = 0; r < R; ++r)
        for (int l = 0; l < L; ++l) {
            if (!inverse) idxs[l * R + r] = r * L + l;
            else idxs[r * L + l] = l * R + r;
        }
    return MOE_OK;
}

extern "C" moe_status_t moe_expert_scale(const void* in, moe_dtype_t dtype, int64_t n_rows,
                                         int64_t H, int E, const int32_t* offsets,
                                         const float* scale, void* out, void* stream) {
    MOE_TRACE(__func__);
    if (!dtype_ok(dtype) || n_rows < 0 || H < 0 || E < 1) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || n_rows >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (!offsets || !scale) return MOE_ERR_INVALID_ARG;
    if (n_rows == 0 || H == 0) return MOE_OK;
    if (!in || !out) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t want = (n_rows + kWarps - 1) / kWarps;
    if (dtype == MOE_F32) {
        const int g = grid_for((const void*)expert_scale_kernel<float>, kThreads, 0, want);
        expert_scale_kernel<float><<<g, kThreads, 0, s>>>(
            static_cast<const float*>(in), n_rows, H, E, offsets, scale, static_cast<float*>(out));
    } else if ((H * 2) % 16 == 0 && aligned16(in) && aligned16(out)) {
        const int g = grid_for((const void*)expert_scale_vec_kernel, kThreads, 0, want);
        expert_scale_vec_kernel<<<g, kThreads, 0, s>>>(
            static_cast<const uint4*>(in), n_rows, H / 8, E, offsets, scale,
            static_cast<uint4*>(out));
    } else {
        const int g = grid_for((const void*)expert_scale_kernel<uint16_t>, kThreads, 0, want);
        expert_scale_kernel<uint16_t><<<g, kThreads, 0, s>>>(
            static_cast<const uint16_t*>(in), n_rows, H, E, offsets, scale,
            static_cast<uint16_t*>(out));
    }
    return launch_status();
}

extern "C" moe_status_t moe_fill_pad_rows(void* rows, moe_dtype_t dtype, int64_t max_rows,
                                         int64_t H, const int32_t* offsets,
                                         const int32_t* counts, int E, void* stream) {
    MOE_TRACE(__func__);
    if (!dtype_ok_move(dtype) || max_rows < 0 || H < 0 || E < 1) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
    if (!offsets || !counts) return MOE_ERR_INVALID_ARG;
    if (max_rows == 0 || H == 0) return MOE_OK;
    if (!rows) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t row = size_t(H) * elem_size(dtype);
    const int g = int(min64(E, int64_t(sm_count()) * 4));
    if (row % 16 == 0 && aligned16(rows))
        fill_pad_rows_kernel<uint4><<<g, kThreads, 0, s>>>(static_cast<uint4*>(rows), max_rows,
                                                          int64_t(row / 16), offsets, counts, E);
    else if (dtype == MOE_F32)
        fill_pad_rows_kernel<float><<<g, kThreads, 0, s>>>(static_cast<float*>(rows), max_rows, H,
                                                           offsets, counts, E);
    else if (dtype == MOE_BF16)
        fill_pad_rows_kernel<uint16_t><<<g, kThreads, 0, s>>>(static_cast<uint16_t*>(rows),
                                                              max_rows, H, offsets, counts, E);
    else
        fill_pad_rows_kernel<uint8_t><<<g, kThreads, 0, s>>>(static_cast<uint8_t*>(rows),
                                                             max_rows, H, offsets, counts, E);
    return launch_status();
}
