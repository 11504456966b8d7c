// fp32 expert FFNs on the CUDA cores (FFMA; no TF32), for layers stored in
// fp32. Same grouping as the tensor-core path: expert e owns rows
// [offsets[e], offsets[e+1]) of x_perm.
//   up:   H[r][f] = SiLU(W1_e[f] . x_perm[r]) * (W3_e[f] . x_perm[r])     (fp32)
//   down: y_slot[r][c] = perm_w[r] * (W2_e[c] . H[r])
// A CTA computes a 32 x 32 output tile of one expert; its row tile is found
// from the device-side offsets, so the host never reads the counts.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kF32Tile = 32;

__device__ __forceinline__ bool f32_find_tile(const int32_t* offsets, int E, int tile_y, int& e,
                                              int& r0, int& r1) {
    int base = 0;
    for (int q = 0; q < E; ++q) {
        const int a = offsets[q], b = offsets[q + 1];
        const int nt = (b - a + kF32Tile - 1) / kF32Tile;
        if (tile_y < base + nt) {
            e = q;
            r0 = a + (tile_y - base) * kF32Tile;
            r1 = b;
            return true;
        }
        base += nt;
    }
    return false;
}

// grid: (ceil(N / 32), upper bound on row tiles); block (32, 8).
template <bool UP>
__global__ void __launch_bounds__(256)
    f32_ffn_kernel(const float* __restrict__ act, const int32_t* __restrict__ offsets, int E,
                   const float* __restrict__ wa, const float* __restrict__ wb, const float* __restrict__ perm_w,
                   int K, int N, float* __restrict__ out) {
    __shared__ float sx[kF32Tile][kF32Tile + 1];
    __shared__ float sa[kF32Tile][kF32Tile + 1];
    __shared__ float sb[kF32Tile][kF32Tile + 1];
    pdl_trigger();
    pdl_wait();
    int e, r0, r1;
    if (!f32_find_tile(offsets, E, blockIdx.y, e, r0, r1)) return;
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int n0 = blockIdx.x * kF32Tile;
    const float* A = wa + (int64_t)e * N * K;
    const float* B = UP ? wb + (int64_t)e * N * K : nullptr;
    float accu[4] = {0.f, 0.f, 0.f, 0.f};
    float accv[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < K; k0 += kF32Tile) {
        for (int i = ty; i < kF32Tile; i += 8) {
            const int r = r0 + i, k = k0 + tx, n = n0 + i;
            sx[i][tx] = (r < r1 && k < K) ? act[(int64_t)r * K + k] : 0.f;
            sa[i][tx] = (n < N && k < K) ? A[(int64_t)n * K + k] : 0.f;
            if (UP) sb[i][tx] = (n < N && k < K) ? B[(int64_t)n * K + k] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kF32Tile; ++kk) {
            const float w = sa[tx][kk];
            const float w3 = UP ? sb[tx][kk] : 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float xv = sx[ty + 8 * q][kk];
                accu[q] = fmaf(xv, w, accu[q]);
                if (UP) accv[q] = fmaf(xv, w3, accv[q]);
            }
        }
        __syncthreads();
    }
    const int n = n0 + tx;
    if (n >= N) return;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int r = r0 + ty + 8 * q;
        if (r >= r1 || r >= r0 + kF32Tile) continue;
        if (UP) out[(int64_t)r * N + n] = silu_f32(accu[q]) * accv[q];
        else out[(int64_t)r * N + n] = perm_w[r] * accu[q];
    }
}

// y[t] = y_slot[slot_row[t][0]] + y_slot[slot_row[t][1]], rounded once.
template <typename T>
__global__ void __launch_bounds__(256)
    combine_kernel(const float* __restrict__ y_slot, const int32_t* __restrict__ slot_row, int64_t T_tokens,
                   int d, T* __restrict__ y) {
    pdl_trigger();
    pdl_wait();
    const int64_t n = T_tokens * d;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / d;
        const int64_t c = i - t * d;
        const int r0 = slot_row[2 * t], r1 = slot_row[2 * t + 1];
        const float a = r0 >= 0 ? y_slot[(int64_t)r0 * d + c] : 0.f;
        const float b = r1 >= 0 ? y_slot[(int64_t)r1 * d + c] : 0.f;
        const float s = a + b;
        if constexpr (sizeof(T) == 2) y[i] = __float2bfloat16_rn(s);
        else y[i] = s;
    }
}

// Vectorised combine for d % 4 == 0: 4 columns per thread.
template <typename T>
__global__ void __launch_bounds__(256)
    combine4_kernel(const float* __restrict__ y_slot, const int32_t* __restrict__ slot_row, int64_t T_tokens,
                    int d, T* __restrict__ y) {
    pdl_trigger();
    pdl_wait();
    const int d4 = d / 4;
    const int64_t n = T_tokens * d4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / d4;
        const int64_t c4 = i - t * d4;
        const int r0 = slot_row[2 * t], r1 = slot_row[2 * t + 1];
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 a = r0 >= 0 ? reinterpret_cast<const float4*>(y_slot + (int64_t)r0 * d)[c4] : z;
        const float4 b = r1 >= 0 ? reinterpret_cast<const float4*>(y_slot + (int64_t)r1 * d)[c4] : z;
        const float s0 = a.x + b.x, s1 = a.y + b.y, s2 = a.z + b.z, s3 = a.w + b.w;
        if constexpr (sizeof(T) == 2) {
            uint2 pk = make_uint2(pack_bf16x2(s0, s1), pack_bf16x2(s2, s3));
            reinterpret_cast<uint2*>(y + t * d)[c4] = pk;
        } else {
            reinterpret_cast<float4*>(y + t * d)[c4] = make_float4(s0, s1, s2, s3);
        }
    }
}

// Load-balancing statistics (tokentrails.org "Mixtral", step "Load balancing"):
// f_i = counts_i / (2T), P_i = mean_t softmax(l_t)_i over all E scores,
// L_aux = E * sum_i f_i P_i. One cluster of kAuxCtas CTAs: CTA r takes the
// r-th of kAuxCtas equal blocks of tokens and reduces its softmax rows in a
// fixed order (threads, warps); CTA 0 then adds the CTAs' sums in rank order
// through distributed shared memory. The order depends only on T.
constexpr int kAuxThreads = 1024;
constexpr int kAuxCtas = 8;
__global__ void __launch_bounds__(kAuxThreads)
    aux_stats_kernel(const float* __restrict__ logits, const int32_t* __restrict__ counts, int64_t T_tokens,
                     int E, float* __restrict__ f, float* __restrict__ P, float* __restrict__ l_aux) {
    __shared__ float red[kAuxThreads / 32][kMaxExperts];
    __shared__ float part[kMaxExperts];
    pdl_trigger();
    pdl_wait();
    const uint32_t rank = cluster_ctarank();
    const int64_t per = (T_tokens + kAuxCtas - 1) / kAuxCtas;
    const int64_t t_begin = (int64_t)rank * per;
    const int64_t t_end = t_begin + per < T_tokens ? t_begin + per : T_tokens;
    float acc[kMaxExperts];
#pragma unroll
    for (int e = 0; e < kMaxExperts; ++e) acc[e] = 0.f;
    // a thread's tokens t = t_begin + tid, + 1024, ... in order; the score rows of
    // four of them are loaded before any is used
    constexpr int G = 4;
    for (int64_t t0 = t_begin + threadIdx.x; t0 < t_end; t0 += (int64_t)G * kAuxThreads) {
        float lv[G][kMaxExperts];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int64_t t = t0 + (int64_t)g * kAuxThreads;
#pragma unroll
            for (int e = 0; e < kMaxExperts; ++e) lv[g][e] = (t < t_end && e < E) ? logits[t * E + e] : 0.f;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (t0 + (int64_t)g * kAuxThreads >= t_end) break;
            float m = lv[g][0];
#pragma unroll
            for (int e = 1; e < kMaxExperts; ++e)
                if (e < E) m = fmaxf(m, lv[g][e]);
            float p[kMaxExperts];
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < kMaxExperts; ++e) {
                p[e] = e < E ? expf(lv[g][e] - m) : 0.f;
                s += p[e];
            }
            const float inv = 1.0f / s;
#pragma unroll
            for (int e = 0; e < kMaxExperts; ++e) acc[e] += p[e] * inv;
        }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int e = 0; e < kMaxExperts; ++e) {
        float v = acc[e];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[warp][e] = v;
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e) {
            float v = red[lane][e];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) part[e] = v;
        }
    }
    // every CTA's sums are in its shared memory before CTA 0 reads them
    cluster_sync();
    if (rank == 0 && threadIdx.x == 0) {
        float L = 0.f;
        for (int e = 0; e < E; ++e) {
            float v = 0.f;
            for (int r = 0; r < kAuxCtas; ++r) {
                float pr;
                asm volatile("ld.shared::cluster.f32 %0, [%1];"
                             : "=f"(pr)
                             : "r"(mapa_shared(smem_u32(&part[e]), (uint32_t)r))
                             : "memory");
                v += pr;
            }
            const float fe = (float)counts[e] / (float)(2 * T_tokens);
            const float pe = v / (float)T_tokens;
            f[e] = fe;
            P[e] = pe;
            L += fe * pe;
        }
        l_aux[0] = (float)E * L;
    }
    // no CTA leaves while CTA 0 may still read its shared memory
    cluster_sync();
}

}  // namespace moe
