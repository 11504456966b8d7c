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
