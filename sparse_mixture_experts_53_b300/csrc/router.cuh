// Router: scores l = x . W_g, top-2 selection and the softmax over the two
// kept scores ("Mixtral of Experts" lecture, router walkthrough;
// tokentrails.org "Mixtral", step "The router").
//
// Large batches: W_g (E x d, 64 KB in bf16 at d = 4096) is staged once per CTA
// in shared memory and a warp scores four tokens at a time; each lane
// accumulates a fixed, strided share of the d products of each token for all
// E experts in fp32, then a butterfly of warp shuffles leaves the E totals in
// every lane. Small batches split one token over a CTA. The reduction order
// of a token's scores is fixed, so the result does not depend on the grid.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kRouterWarps = 8;

template <typename T>
struct Vec16;  // 16-byte vector of stored elements
template <>
struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
};
template <>
struct Vec16<float> {
    static constexpr int N = 4;
};

template <typename T>
__device__ __forceinline__ void unpack_vec(const uint4 raw, float (&v)[Vec16<T>::N]) {
    if constexpr (sizeof(T) == 2) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(h[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    } else {
        const float* f = reinterpret_cast<const float*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = f[i];
    }
}

template <typename T>
__device__ __forceinline__ void load_vec(const T* p, float (&v)[Vec16<T>::N]) {
    unpack_vec<T>(*reinterpret_cast<const uint4*>(p), v);
}

constexpr int kRouterGroup = 8;  // 16-byte chunks each thread loads before storing them (W_g staging)
constexpr int kRouterTokensPerWarp = 4;  // tokens a warp scores together (large batches)
constexpr int kRouterChunks = 2;         // 16-byte chunks of each token a lane loads before using them

// Top-2 selection and the two-way softmax from the E scores of one token.
__device__ __forceinline__ void top2_softmax(const float (&acc)[kMaxExperts], int E, int32_t* idx, float* w) {
    // strict '>' keeps the lower index among equal scores
    int a = 0;
    float la = acc[0];
#pragma unroll
    for (int e = 1; e < kMaxExperts; ++e)
        if (e < E && acc[e] > la) { la = acc[e]; a = e; }
    int b = -1;
    float lb = 0.f;
#pragma unroll
    for (int e = 0; e < kMaxExperts; ++e)
        if (e < E && e != a && (b < 0 || acc[e] > lb)) { lb = acc[e]; b = e; }
    const float r = expf(lb - la);
    const float inv = 1.0f / (1.0f + r);
    idx[0] = a;
    idx[1] = b;
    w[0] = inv;
    w[1] = r * inv;
}

// use_smem: W_g is copied to shared memory (E * d * sizeof(T) bytes of
// dynamic shared memory); otherwise it is read through L1/L2.
// vec: rows are 16-byte aligned and d is a multiple of the vector width.
template <typename T>
__global__ void __launch_bounds__(kRouterWarps * 32, 2)
    router_top2_kernel(const T* __restrict__ x, const T* __restrict__ wg, int64_t T_tokens, int d,
                       int E, int use_smem, int vec, int32_t* __restrict__ topk_idx,
                       float* __restrict__ topk_w, float* __restrict__ logits) {
    extern __shared__ __align__(16) unsigned char router_smem[];
    pdl_trigger();
    pdl_wait();
    const T* w = wg;
    if (use_smem) {
        T* s = reinterpret_cast<T*>(router_smem);
        const int64_t n = (int64_t)E * d;
        if (vec) {
            // several independent 16-byte loads in flight per thread
            const int64_t nv = n / Vec16<T>::N;
            const uint4* src = reinterpret_cast<const uint4*>(wg);
            uint4* dst = reinterpret_cast<uint4*>(s);
            for (int64_t i0 = threadIdx.x; i0 < nv; i0 += (int64_t)blockDim.x * kRouterGroup) {
                uint4 tmp[kRouterGroup];
#pragma unroll
                for (int u = 0; u < kRouterGroup; ++u) {
                    const int64_t i = i0 + (int64_t)u * blockDim.x;
                    if (i < nv) tmp[u] = src[i];
                }
#pragma unroll
                for (int u = 0; u < kRouterGroup; ++u) {
                    const int64_t i = i0 + (int64_t)u * blockDim.x;
                    if (i < nv) dst[i] = tmp[u];
                }
            }
        } else {
            for (int64_t i = threadIdx.x; i < n; i += blockDim.x) s[i] = wg[i];
        }
        __syncthreads();
        w = s;
    }
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    constexpr int V = Vec16<T>::N;

    if (vec) {
        // A warp scores kRouterTokensPerWarp consecutive tokens together, so
        // each W_g chunk read from shared memory (and widened to fp32) serves
        // all of them. Per token the sums are the single-token ones: lane
        // chunks c = lane, lane + 32, ... in increasing order, then a butterfly.
        constexpr int TPW = kRouterTokensPerWarp;
        const int nchunks = d / V;
        for (int64_t t0 = ((int64_t)blockIdx.x * kRouterWarps + warp) * TPW; t0 < T_tokens;
             t0 += (int64_t)gridDim.x * kRouterWarps * TPW) {
            float acc[TPW][kMaxExperts];
#pragma unroll
            for (int k = 0; k < TPW; ++k)
#pragma unroll
                for (int e = 0; e < kMaxExperts; ++e) acc[k][e] = 0.f;
            for (int c0 = lane; c0 < nchunks; c0 += 32 * kRouterChunks) {
                uint4 xg[kRouterChunks][TPW];
#pragma unroll
                for (int u = 0; u < kRouterChunks; ++u)
#pragma unroll
                    for (int k = 0; k < TPW; ++k) {
                        const int c = c0 + 32 * u;
                        xg[u][k] = (c < nchunks && t0 + k < T_tokens)
                                       ? *reinterpret_cast<const uint4*>(x + (t0 + k) * d + c * V)
                                       : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                for (int u = 0; u < kRouterChunks; ++u) {
                    const int c = c0 + 32 * u;
                    if (c < nchunks) {
                        float xv[TPW][V];
#pragma unroll
                        for (int k = 0; k < TPW; ++k) unpack_vec<T>(xg[u][k], xv[k]);
#pragma unroll
                        for (int e = 0; e < kMaxExperts; ++e) {
                            if (e < E) {
                                float wv[V];
                                load_vec<T>(w + (int64_t)e * d + c * V, wv);
#pragma unroll
                                for (int k = 0; k < TPW; ++k)
#pragma unroll
                                    for (int i = 0; i < V; ++i) acc[k][e] = fmaf(xv[k][i], wv[i], acc[k][e]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < TPW; ++k) {
#pragma unroll
                for (int e = 0; e < kMaxExperts; ++e) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) acc[k][e] += __shfl_xor_sync(0xffffffffu, acc[k][e], o);
                }
                const int64_t t = t0 + k;
                if (t >= T_tokens) break;
                if (logits != nullptr && lane < E) {
                    float v = acc[k][0];
#pragma unroll
                    for (int e = 1; e < kMaxExperts; ++e)
                        if (lane == e) v = acc[k][e];
                    logits[t * E + lane] = v;
                }
                if (lane == 0) top2_softmax(acc[k], E, topk_idx + 2 * t, topk_w + 2 * t);
            }
        }
        return;
    }

    // scalar path (rows not 16-byte aligned or d not a multiple of the vector width)
    for (int64_t t = (int64_t)blockIdx.x * kRouterWarps + warp; t < T_tokens;
         t += (int64_t)gridDim.x * kRouterWarps) {
        const T* xr = x + t * d;
        float acc[kMaxExperts];
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e) acc[e] = 0.f;
        for (int j = lane; j < d; j += 32) {
            const float xv = to_f32<T>(xr[j]);
#pragma unroll
            for (int e = 0; e < kMaxExperts; ++e)
                if (e < E) acc[e] = fmaf(xv, to_f32<T>(w[(int64_t)e * d + j]), acc[e]);
        }
        // butterfly: every lane ends with the full sums, in the same order
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
        }
        if (logits != nullptr && lane < E) {
            float v = acc[0];
#pragma unroll
            for (int e = 1; e < kMaxExperts; ++e)
                if (lane == e) v = acc[e];
            logits[t * E + lane] = v;
        }
        if (lane == 0) top2_softmax(acc, E, topk_idx + 2 * t, topk_w + 2 * t);
    }
}

// Small batches: one CTA per token, the d products split over 8 warps. Each
// lane sums its own chunks in order, a butterfly adds the lanes, and warp 0
// adds the 8 warp totals in warp order, so the result is deterministic and the
// longest chain of additions is d/256 + 13 terms. W_g is read through L1/L2
// (64 KB), so no CTA waits for a whole copy of it.
template <typename T>
__global__ void __launch_bounds__(kRouterWarps * 32)
    router_top2_split_kernel(const T* __restrict__ x, const T* __restrict__ wg, int64_t T_tokens, int d, int E,
                             int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, float* __restrict__ logits) {
    __shared__ float part[kRouterWarps][kMaxExperts];
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    constexpr int V = Vec16<T>::N;
    const int nchunks = d / V;  // d % V == 0 and 16-byte rows (checked on the host)
    for (int64_t t = blockIdx.x; t < T_tokens; t += gridDim.x) {
        const T* xr = x + t * d;
        float acc[kMaxExperts];
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e) acc[e] = 0.f;
        for (int c = warp * 32 + lane; c < nchunks; c += kRouterWarps * 32) {
            float xv[V];
            load_vec<T>(xr + c * V, xv);
#pragma unroll
            for (int e = 0; e < kMaxExperts; ++e) {
                if (e < E) {
                    float wv[V];
                    load_vec<T>(wg + (int64_t)e * d + c * V, wv);
#pragma unroll
                    for (int i = 0; i < V; ++i) acc[e] = fmaf(xv[i], wv[i], acc[e]);
                }
            }
        }
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
        }
        if (lane == 0) {
#pragma unroll
            for (int e = 0; e < kMaxExperts; ++e) part[warp][e] = acc[e];
        }
        __syncthreads();
        if (warp == 0) {
            float tot[kMaxExperts];
#pragma unroll
            for (int e = 0; e < kMaxExperts; ++e) {
                float v = part[0][e];
#pragma unroll
                for (int q = 1; q < kRouterWarps; ++q) v += part[q][e];
                tot[e] = v;
            }
            if (logits != nullptr && lane < E) {
                float v = tot[0];
#pragma unroll
                for (int e = 1; e < kMaxExperts; ++e)
                    if (lane == e) v = tot[e];
                logits[t * E + lane] = v;
            }
            if (lane == 0) top2_softmax(tot, E, topk_idx + 2 * t, topk_w + 2 * t);
        }
        __syncthreads();
    }
}

}  // namespace moe
