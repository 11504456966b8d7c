// Grouping of the 2T slots by expert: per-expert counts, their exclusive
// prefix sum, and a stable (token-ascending) rank inside each expert. The
// pages note only that different tokens pick different experts and that some
// experts get none (tokentrails.org "Mixtral", step "Two experts per token");
// the expert-contiguous order is this library's own structure, and it is what
// lets each expert's weights be read once per batch.
//
// One CTA of 1024 threads: thread i owns a contiguous run of tokens, counts
// its slots per expert, a block-wide scan gives each thread its starting rank
// per expert, and a second pass writes rows in token order. There are no
// atomics, so the result is the unique stable order.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kPermuteThreads = 1024;

__global__ void __launch_bounds__(kPermuteThreads)
    permute_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
                   int64_t T_tokens, int E, int32_t* __restrict__ counts,
                   int32_t* __restrict__ offsets, int32_t* __restrict__ perm_token,
                   int32_t* __restrict__ slot_row, float* __restrict__ perm_w,
                   const unsigned char* __restrict__ x, int64_t row_bytes, unsigned char* __restrict__ x_perm) {
    __shared__ int warp_tot[kPermuteThreads / 32][kMaxExperts];
    __shared__ int s_off[kMaxExperts + 1];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t chunk = (T_tokens + kPermuteThreads - 1) / kPermuteThreads;
    const int64_t t0 = ((int64_t)tid * chunk < T_tokens) ? (int64_t)tid * chunk : T_tokens;
    const int64_t t1 = (t0 + chunk < T_tokens) ? t0 + chunk : T_tokens;

    int cnt[kMaxExperts];
#pragma unroll
    for (int e = 0; e < kMaxExperts; ++e) cnt[e] = 0;
    bool bad = false;
    for (int64_t t = t0; t < t1; ++t) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int e = topk_idx[2 * t + j];
            if (e >= 0 && e < E) {
#pragma unroll
                for (int q = 0; q < kMaxExperts; ++q) cnt[q] += (q == e);
            } else {
                bad = true;
            }
        }
    }
    if (bad) report_error(MOE_ERR_DEVICE_CHECK, K_PERMUTE, W_INDEX);

    // exclusive scan over threads, one expert at a time: warp scan, then a
    // scan of the 32 warp totals
    int excl[kMaxExperts];
#pragma unroll
    for (int e = 0; e < kMaxExperts; ++e) {
        int v = cnt[e];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        excl[e] = v - cnt[e];
        if (lane == 31) warp_tot[warp][e] = v;
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e) {
            const int tot = warp_tot[lane][e];
            int v = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            warp_tot[lane][e] = v - tot;  // exclusive prefix of warps
            if (lane == 31 && e < E) s_off[e + 1] = v;  // expert total for now
        }
    }
    __syncthreads();
    if (tid == 0) {
        s_off[0] = 0;
        for (int e = 0; e < E; ++e) {
            const int c = s_off[e + 1];
            counts[e] = c;
            s_off[e + 1] = s_off[e] + c;
        }
        for (int e = 0; e <= E; ++e) offsets[e] = s_off[e];
    }
    __syncthreads();
    int next[kMaxExperts];
#pragma unroll
    for (int e = 0; e < kMaxExperts; ++e) next[e] = (e < E ? s_off[e] : 0) + warp_tot[warp][e] + excl[e];

    for (int64_t t = t0; t < t1; ++t) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int e = topk_idx[2 * t + j];
            int r = -1;
            if (e >= 0 && e < E) {
#pragma unroll
                for (int q = 0; q < kMaxExperts; ++q)
                    if (q == e) r = next[q]++;
                perm_token[r] = (int32_t)t;
                perm_w[r] = topk_w[2 * t + j];
            }
            slot_row[2 * t + j] = r;
        }
    }
    // Small batches: the same CTA copies the token rows into expert order
    // (x != nullptr; row_bytes % 16 == 0), saving a launch.
    if (x != nullptr) {
        __syncthreads();
        const int64_t rows = s_off[E];
        const int64_t c16 = row_bytes / 16;
        for (int64_t i = tid; i < rows * c16; i += kPermuteThreads) {
            const int64_t r = i / c16, c = i - r * c16;
            const int64_t tk = perm_token[r];
            reinterpret_cast<uint4*>(x_perm + r * row_bytes)[c] = reinterpret_cast<const uint4*>(x + tk * row_bytes)[c];
        }
    }
}

// ---------------------------------------------------------------------------
// Grouping of small batches (2T <= 512 slots) on several CTAs. Every CTA
// ranks all the slots itself (16 warps, one slot per thread, warp ballots per
// expert, integer counts: the same unique stable order as permute_kernel), CTA
// 0 writes the grouping, and every CTA copies its share of the token rows into
// x_perm. A single CTA copying all the rows waits on one memory round trip per
// handful of rows; spread over the grid the copies are in flight together.
// ---------------------------------------------------------------------------
constexpr int kSmallPermuteThreads = 512;
constexpr int kSmallPermuteMaxSlots = kSmallPermuteThreads;

__global__ void __launch_bounds__(kSmallPermuteThreads)
    permute_small_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int64_t T_tokens,
                         int E, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                         int32_t* __restrict__ perm_token, int32_t* __restrict__ slot_row,
                         float* __restrict__ perm_w, const unsigned char* __restrict__ x, int64_t row_bytes,
                         unsigned char* __restrict__ x_perm) {
    constexpr int W = kSmallPermuteThreads / 32;
    __shared__ int wcnt[W][kMaxExperts];
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int row_token[kSmallPermuteMaxSlots];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = (int)(2 * T_tokens);
    const bool lead = blockIdx.x == 0;
    int e = -1;
    if (tid < R) e = topk_idx[tid];
    const bool valid = e >= 0 && e < E;
    if (tid < R && !valid && lead) report_error(MOE_ERR_DEVICE_CHECK, K_PERMUTE, W_INDEX);
    const unsigned lt = (1u << lane) - 1u;
    int before = 0;
#pragma unroll
    for (int q = 0; q < kMaxExperts; ++q) {
        const unsigned m = __ballot_sync(0xffffffffu, valid && e == q);
        if (e == q) before = __popc(m & lt);
        if (lane == 0) wcnt[warp][q] = __popc(m);
    }
    __syncthreads();
    if (tid < kMaxExperts) {
        // exclusive prefix over warps (in place); the total goes to s_off
        int run = 0;
        for (int w = 0; w < W; ++w) {
            const int c = wcnt[w][tid];
            wcnt[w][tid] = run;
            run += c;
        }
        s_off[tid + 1] = run;
    }
    __syncthreads();
    if (tid == 0) {
        s_off[0] = 0;
        for (int q = 0; q < E; ++q) {
            if (lead) counts[q] = s_off[q + 1];
            s_off[q + 1] += s_off[q];
        }
        if (lead)
            for (int q = 0; q <= E; ++q) offsets[q] = s_off[q];
    }
    __syncthreads();
    if (tid < R) {
        const int r = valid ? s_off[e] + wcnt[warp][e] + before : -1;
        if (valid) row_token[r] = tid >> 1;
        if (lead) {
            slot_row[tid] = r;
            if (valid) {
                perm_token[r] = tid >> 1;
                perm_w[r] = topk_w[tid];
            }
        }
    }
    __syncthreads();
    // rows [0, s_off[E]) of x_perm, 16-byte chunks spread over the grid, four
    // loads in flight per thread before their stores
    const int64_t c16 = row_bytes / 16;
    const int64_t n = (int64_t)s_off[E] * c16;
    const int64_t stride = (int64_t)gridDim.x * kSmallPermuteThreads;
    for (int64_t i0 = (int64_t)blockIdx.x * kSmallPermuteThreads + tid; i0 < n; i0 += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < n) {
                const int64_t r = i / c16, c = i - r * c16;
                v[u] = reinterpret_cast<const uint4*>(x + (int64_t)row_token[r] * row_bytes)[c];
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < n) {
                const int64_t r = i / c16, c = i - r * c16;
                reinterpret_cast<uint4*>(x_perm + r * row_bytes)[c] = v[u];
            }
        }
    }
}

// x_perm[r] = x[perm_token[r]]: one row per warp-group, 16-byte copies when
// the row size allows, 4-byte copies otherwise.
__global__ void __launch_bounds__(256)
    gather_rows_kernel(const unsigned char* __restrict__ x, const int32_t* __restrict__ perm_token,
                       const int32_t* __restrict__ offsets, int E, int64_t rows, int64_t row_bytes,
                       unsigned char* __restrict__ x_perm) {
    pdl_trigger();
    pdl_wait();
    const int64_t valid_rows = ((int64_t)offsets[E] < rows) ? (int64_t)offsets[E] : rows;
    const int64_t chunks16 = (row_bytes % 16 == 0) ? row_bytes / 16 : 0;
    for (int64_t r = blockIdx.x; r < valid_rows; r += gridDim.x) {
        const int64_t t = perm_token[r];
        const unsigned char* src = x + t * row_bytes;
        unsigned char* dst = x_perm + r * row_bytes;
        if (chunks16) {
            for (int64_t c = threadIdx.x; c < chunks16; c += blockDim.x)
                reinterpret_cast<uint4*>(dst)[c] = reinterpret_cast<const uint4*>(src)[c];
        } else {
            for (int64_t c = threadIdx.x; c < row_bytes / 4; c += blockDim.x)
                reinterpret_cast<uint32_t*>(dst)[c] = reinterpret_cast<const uint32_t*>(src)[c];
        }
    }
}

}  // namespace moe

namespace moe {

// ---------------------------------------------------------------------------
// Grouping for large batches on many CTAs. The result is the same unique
// stable order as permute_kernel (all sums are integer counts, so no order of
// summation can change them).
//   pass 1 (permute_count_kernel): CTA c counts the slots of its token chunk
//            per expert -> chunk_counts[c][e];
//   pass 2 (permute_place_kernel): CTA c adds up the counts of all chunks
//            (totals -> offsets) and of the chunks before it (its base), ranks
//            its tokens 64 at a time with warp ballots, writes slot_row,
//            perm_token and perm_w, and copies each token row of x to the
//            token's two rows of x_perm (one read, two writes).
// ---------------------------------------------------------------------------
constexpr int kPlaceThreads = 256;
constexpr int kPlaceSub = 64;  // tokens ranked together (two warps)

__global__ void __launch_bounds__(kPlaceThreads)
    permute_count_kernel(const int32_t* __restrict__ topk_idx, int64_t T_tokens, int E, int64_t chunk,
                         int32_t* __restrict__ chunk_counts) {
    __shared__ int wc[kPlaceThreads / 32][kMaxExperts];
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t0 = (int64_t)blockIdx.x * chunk;
    const int64_t t1 = (t0 + chunk < T_tokens) ? t0 + chunk : T_tokens;
    int cnt[kMaxExperts];
#pragma unroll
    for (int e = 0; e < kMaxExperts; ++e) cnt[e] = 0;
    bool bad = false;
    for (int64_t base = t0; base < t1; base += kPlaceThreads) {
        const int64_t t = base + threadIdx.x;
        int i0 = -1, i1 = -1;
        if (t < t1) {
            i0 = topk_idx[2 * t];
            i1 = topk_idx[2 * t + 1];
            bad |= !(i0 >= 0 && i0 < E) || !(i1 >= 0 && i1 < E);
        }
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e)
            cnt[e] += __popc(__ballot_sync(0xffffffffu, i0 == e)) + __popc(__ballot_sync(0xffffffffu, i1 == e));
    }
    if (bad) report_error(MOE_ERR_DEVICE_CHECK, K_PERMUTE, W_INDEX);
    if (lane == 0) {
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e) wc[warp][e] = cnt[e];
    }
    __syncthreads();
    if (threadIdx.x < kMaxExperts) {
        int s = 0;
        for (int w = 0; w < kPlaceThreads / 32; ++w) s += wc[w][threadIdx.x];
        chunk_counts[(int64_t)blockIdx.x * kMaxExperts + threadIdx.x] = s;
    }
}

__global__ void __launch_bounds__(kPlaceThreads)
    permute_place_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int64_t T_tokens,
                         int E, int64_t chunk, int nchunks, const int32_t* __restrict__ chunk_counts,
                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                         int32_t* __restrict__ perm_token, int32_t* __restrict__ slot_row,
                         float* __restrict__ perm_w, const unsigned char* __restrict__ x, int64_t row_bytes,
                         unsigned char* __restrict__ x_perm) {
    __shared__ int red[kPlaceThreads / 32][2 * kMaxExperts];
    __shared__ int base_s[kMaxExperts];
    __shared__ int wtot[2][kMaxExperts];
    __shared__ int rows_s[kPlaceSub][2];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int me = blockIdx.x;

    // totals of every chunk and of the chunks before this one (integer sums)
    int tot[kMaxExperts], pre[kMaxExperts];
#pragma unroll
    for (int e = 0; e < kMaxExperts; ++e) tot[e] = pre[e] = 0;
    for (int c = tid; c < nchunks; c += kPlaceThreads) {
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e) {
            const int v = chunk_counts[(int64_t)c * kMaxExperts + e];
            tot[e] += v;
            pre[e] += (c < me) ? v : 0;
        }
    }
#pragma unroll
    for (int e = 0; e < kMaxExperts; ++e) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            tot[e] += __shfl_xor_sync(0xffffffffu, tot[e], o);
            pre[e] += __shfl_xor_sync(0xffffffffu, pre[e], o);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e) {
            red[warp][e] = tot[e];
            red[warp][kMaxExperts + e] = pre[e];
        }
    }
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int e = 0; e < E; ++e) {
            int te = 0, pe = 0;
            for (int w = 0; w < kPlaceThreads / 32; ++w) {
                te += red[w][e];
                pe += red[w][kMaxExperts + e];
            }
            if (me == 0) {
                counts[e] = te;
                offsets[e] = run;
            }
            base_s[e] = run + pe;
            run += te;
        }
        if (me == 0) offsets[E] = run;
    }
    __syncthreads();

    const int64_t t0 = (int64_t)me * chunk;
    const int64_t t1 = (t0 + chunk < T_tokens) ? t0 + chunk : T_tokens;
    const int64_t c16 = row_bytes / 16;
    for (int64_t sub = t0; sub < t1; sub += kPlaceSub) {
        // ---- ranks of 64 tokens (warps 0 and 1), in token order
        if (tid < kPlaceSub) {
            const int64_t t = sub + tid;
            int i0 = -1, i1 = -1;
            if (t < t1) {
                i0 = topk_idx[2 * t];
                i1 = topk_idx[2 * t + 1];
            }
            const unsigned lt = (1u << lane) - 1u;
            int r0 = -1, r1 = -1;
#pragma unroll
            for (int e = 0; e < kMaxExperts; ++e) {
                const unsigned m0 = __ballot_sync(0xffffffffu, i0 == e);
                const unsigned m1 = __ballot_sync(0xffffffffu, i1 == e);
                const int before = __popc(m0 & lt) + __popc(m1 & lt);
                if (lane == 0) wtot[warp][e] = __popc(m0) + __popc(m1);
                if (i0 == e) r0 = before;
                if (i1 == e) r1 = before + (i0 == e ? 1 : 0);
            }
            rows_s[tid][0] = r0;
            rows_s[tid][1] = r1;
        }
        __syncthreads();
        if (tid < kPlaceSub) {
            const int64_t t = sub + tid;
            if (t < t1) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int e = topk_idx[2 * t + j];
                    int r = -1;
                    if (e >= 0 && e < E) {
                        r = base_s[e] + (warp == 1 ? wtot[0][e] : 0) + rows_s[tid][j];
                        perm_token[r] = (int32_t)t;
                        perm_w[r] = topk_w[2 * t + j];
                    }
                    slot_row[2 * t + j] = r;
                    rows_s[tid][j] = r;
                }
            }
        }
        __syncthreads();
        if (tid == 0) {
            for (int e = 0; e < E; ++e) base_s[e] += wtot[0][e] + wtot[1][e];
        }
        // ---- copy each token row to its two rows (all 8 warps)
        if (x != nullptr) {
            const int64_t n_sub = ((t1 - sub) < kPlaceSub) ? (t1 - sub) : kPlaceSub;
            for (int q = warp; q < n_sub; q += kPlaceThreads / 32) {
                const int64_t t = sub + q;
                const int ra = rows_s[q][0], rb = rows_s[q][1];
                const uint4* src = reinterpret_cast<const uint4*>(x + t * row_bytes);
                uint4* da = reinterpret_cast<uint4*>(x_perm + (int64_t)(ra >= 0 ? ra : 0) * row_bytes);
                uint4* db = reinterpret_cast<uint4*>(x_perm + (int64_t)(rb >= 0 ? rb : 0) * row_bytes);
                // four loads in flight per lane before their stores
                for (int64_t c0 = lane; c0 < c16; c0 += 4 * 32) {
                    uint4 v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (c0 + 32 * u < c16) v[u] = src[c0 + 32 * u];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int64_t c = c0 + 32 * u;
                        if (c < c16) {
                            if (ra >= 0) da[c] = v[u];
                            if (rb >= 0) db[c] = v[u];
                        }
                    }
                }
            }
        }
        __syncthreads();
    }
}

// dst[r] = src[index[r]] for r < rows, 16-byte copies, four in flight per
// thread; an index outside [0, src_rows) gives a row of zeros and latches
// MOE_ERR_DEVICE_CHECK. Used to move rows between the ranks' buffers of an
// expert-parallel layer laid out in one allocation, and to regroup them.
__global__ void __launch_bounds__(256)
    gather_index_kernel(const unsigned char* __restrict__ src, int64_t src_rows, const int32_t* __restrict__ index,
                        int64_t rows, int64_t row_bytes, unsigned char* __restrict__ dst) {
    pdl_trigger();
    pdl_wait();
    const int64_t c16 = row_bytes / 16;
    const int64_t n = rows * c16;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    bool bad = false;
    for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < n; i0 += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t i = i0 + u * stride;
            v[u] = make_uint4(0, 0, 0, 0);
            if (i < n) {
                const int64_t r = i / c16, c = i - r * c16;
                const int64_t s = index[r];
                if (s >= 0 && s < src_rows) v[u] = reinterpret_cast<const uint4*>(src + s * row_bytes)[c];
                else bad = true;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < n) {
                const int64_t r = i / c16, c = i - r * c16;
                reinterpret_cast<uint4*>(dst + r * row_bytes)[c] = v[u];
            }
        }
    }
    if (bad) report_error(MOE_ERR_DEVICE_CHECK, K_GATHER, W_INDEX);
}

}  // namespace moe
