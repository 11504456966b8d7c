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
//
// bf16 batches above the small-batch size run on the tensor cores instead
// (router_tc_kernel): the scores of 128 tokens are one M = 128, N = 16, K = d
// tcgen05 product of the token tile and W_g (rows E..15 zero), accumulated in
// fp32 in tensor memory; the epilogue's thread for a token reads its E scores
// and makes the top-2 choice. That leaves the kernel bound by reading x.
#pragma once

#include "common.cuh"
#include "ffn_tc.cuh"

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

// ---------------------------------------------------------------------------
// Router on the tensor cores (bf16, d a multiple of 64). Persistent CTAs take
// 128-token tiles; warp 0 streams the tile's x (TMA, 64 K x 128 rows) and the
// matching 64 K x 8 rows of W_g into a stage, warp 1 issues four M = 128,
// N = 16, K = 16 MMAs per stage into one of two 16-column accumulators, and
// warps 2-5 (one token per thread) read the scores back, choose the top two
// and write idx, w and the scores. Rows 8..15 of each stage's W_g slot are
// zero (written once before the first copy), and TMA fills W_g rows >= E and
// token rows >= T with zeros, so those scores and rows are never used.
// ---------------------------------------------------------------------------
constexpr int kRtStages = 8;
constexpr int kRtM = 128;                                  // tokens per tile
constexpr int kRtN = 16;                                   // MMA columns (E <= 8 used)
constexpr uint32_t kRtABytes = kRtM * kBK * 2;             // 16 KB of x per stage
constexpr uint32_t kRtBBytes = kRtN * kBK * 2;             // 2 KB slot of W_g per stage
constexpr uint32_t kRtBLoad = 8 * kBK * 2;                 // the 1 KB TMA writes (rows 0-7)
constexpr uint32_t kRtStageBytes = kRtABytes + kRtBBytes;  // 18 KB, a multiple of 1 KB
constexpr int kRtThreads = 192;

struct RouterTcControl {
    uint64_t full[kRtStages];
    uint64_t empty[kRtStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr size_t kRtSmemBytes = 1024 + (size_t)kRtStages * kRtStageBytes + sizeof(RouterTcControl);

__device__ __forceinline__ void rt_abort(RouterTcControl* c, int where) {
    report_error(MOE_ERR_TIMEOUT, K_ROUTER, where);
    *reinterpret_cast<volatile int*>(&c->abort_flag) = 1;
}

__global__ void __launch_bounds__(kRtThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                     int64_t T_tokens, int d, int E, uint64_t timeout_ns, int32_t* __restrict__ topk_idx,
                     float* __restrict__ topk_w, float* __restrict__ logits) {
    extern __shared__ unsigned char rt_smem_raw[];
    unsigned char* smem = align1024(rt_smem_raw);
    RouterTcControl* ctl = reinterpret_cast<RouterTcControl*>(smem + (size_t)kRtStages * kRtStageBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t tmo = timeout_ns;
    volatile int* abort_flag = &ctl->abort_flag;
    const int n_tiles = (int)((T_tokens + kRtM - 1) / kRtM);
    const int KB = d / kBK;

    // rows 8..15 of every W_g slot: zeros the tensor core reads (async proxy)
    for (int i = threadIdx.x; i < kRtStages * (int)(kRtBBytes - kRtBLoad) / 16; i += blockDim.x) {
        const int st = i / ((kRtBBytes - kRtBLoad) / 16), j = i % ((kRtBBytes - kRtBLoad) / 16);
        reinterpret_cast<uint4*>(smem + (size_t)st * kRtStageBytes + kRtABytes + kRtBLoad)[j] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        for (int q = 0; q < kRtStages; ++q) {
            mbar_init(smem_u32(&ctl->full[q]), 1);
            mbar_init(smem_u32(&ctl->empty[q]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&ctl->tfull[b]), 1);
            mbar_init(smem_u32(&ctl->tempty[b]), 4);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&map_x);
        tma_prefetch_desc(&map_w);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), 2 * kRtN);
        tmem_relinquish();
    }
    pdl_trigger();
    pdl_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_x = policy_evict_first();   // each token row is read once
            const uint64_t pol_w = policy_evict_last();    // W_g is read by every tile
            uint32_t s = 0, ph = 0;
            uint32_t issued_mask = 0, issued_ph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1, tmo, abort_flag)) {
                        rt_abort(ctl, W_PRODUCER);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&ctl->full[s]);
                    const uint32_t sa = smem_u32(smem + (size_t)s * kRtStageBytes);
                    mbar_arrive_expect_tx(fb, kRtABytes + kRtBLoad);
                    tma_load_2d(sa, &map_x, fb, kb * kBK, tile * kRtM, pol_x);
                    tma_load_2d(sa + kRtABytes, &map_w, fb, kb * kBK, 0, pol_w);
                    issued_mask |= 1u << s;
                    issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                    if (++s == kRtStages) { s = 0; ph ^= 1; }
                }
            }
            if (!ok) {
                for (int q = 0; q < kRtStages; ++q)
                    if (issued_mask & (1u << q))
                        drain_wait(smem_u32(&ctl->full[q]), (issued_ph >> q) & 1u, tmo, K_ROUTER);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kRtM, kRtN);
            uint32_t s = 0, ph = 0;
            bool ok = true, any = false;
            int it = 0;
            for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++it) {
                const int b = it & 1;
                const uint32_t aph = (it >> 1) & 1;
                if (!mbar_wait(smem_u32(&ctl->tempty[b]), aph ^ 1, tmo, abort_flag)) {
                    rt_abort(ctl, W_MMA);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * kRtN;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(smem_u32(&ctl->full[s]), ph, tmo, abort_flag)) {
                        rt_abort(ctl, W_MMA);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)s * kRtStageBytes);
                    const uint64_t adesc = sw128_kmajor_desc(sa);
                    const uint64_t bdesc = sw128_kmajor_desc(sa + kRtABytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
                    any = true;
                    mma_commit(smem_u32(&ctl->empty[s]));
                    if (++s == kRtStages) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                mma_commit(smem_u32(&ctl->tfull[b]));
            }
            if (any) {
                mma_commit(smem_u32(&ctl->drain));
                drain_wait(smem_u32(&ctl->drain), 0, tmo, K_ROUTER);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2-5): one token per thread
        const int sub = warp & 3;   // tensor-memory lanes 32 sub .. 32 sub + 31
        int it = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
            const int b = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            if (!mbar_wait(smem_u32(&ctl->tfull[b]), aph, tmo, abort_flag)) {
                rt_abort(ctl, W_EPILOGUE);
                break;
            }
            tc_fence_after();
            uint32_t v[16];
            tmem_ld16(tmem_base + b * kRtN + ((uint32_t)(sub * 32) << 16), v);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[b]));
            const int64_t t = (int64_t)tile * kRtM + sub * 32 + lane;
            if (t < T_tokens) {
                float acc[kMaxExperts];
#pragma unroll
                for (int e = 0; e < kMaxExperts; ++e) acc[e] = __uint_as_float(v[e]);
                if (logits != nullptr) {
#pragma unroll
                    for (int e = 0; e < kMaxExperts; ++e)
                        if (e < E) logits[t * E + e] = acc[e];
                }
                top2_softmax(acc, E, topk_idx + 2 * t, topk_w + 2 * t);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 2 * kRtN);
}

}  // namespace moe
