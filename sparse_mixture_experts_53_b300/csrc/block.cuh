// Memory-bound steps of the decoder block around the MoE layer: RMSNorm (with
// the residual add in front of it), RoPE on the fused Q/K/V projection, and
// the final residual add. Mixtral keeps LLaMA's block and swaps only the MLP
// for the MoE layer; the two residual branches are attention on the
// normalised input, then the MoE layer on the normalised sum ("Mixtral"
// lineage page, step "GPT-2 vs Mixtral" and its Code).
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kNormThreads = 256;
constexpr int kRopeTokens = 4;        // tokens per RoPE block (blockDim.y)
constexpr int kRopeMaxPairs = 128;    // head_dim <= 256

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float (&v)[8]) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(p[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&v)[8]) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
}

// One warp per row. ADD: h = bf16(x + add) is written to h_out and normalised;
// otherwise x itself. y = g * h / sqrt(mean(h^2) + eps), rounded to bf16.
// The sum of squares is taken over the bf16 values of h, the values the next
// step reads. d is a multiple of 8 (16-byte chunks).
template <bool ADD>
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const __nv_bfloat16* __restrict__ x,
                                                               const float* __restrict__ add,
                                                               const __nv_bfloat16* __restrict__ g, float eps,
                                                               int64_t rows, int d, __nv_bfloat16* h_out,
                                                               __nv_bfloat16* __restrict__ y) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nch = d >> 3;
    const uint4* gv = reinterpret_cast<const uint4*>(g);
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nwarps) {
        const uint4* xr = reinterpret_cast<const uint4*>(x + r * d);
        uint4* hr = reinterpret_cast<uint4*>(h_out + (ADD ? r * d : 0));
        float ss = 0.f;
#pragma unroll 4
        for (int c = lane; c < nch; c += 32) {
            float v[8];
            unpack_bf16x8(xr[c], v);
            if (ADD) {
                const float4* ar = reinterpret_cast<const float4*>(add + r * d) + 2 * c;
                const float4 a0 = ar[0], a1 = ar[1];
                v[0] += a0.x; v[1] += a0.y; v[2] += a0.z; v[3] += a0.w;
                v[4] += a1.x; v[5] += a1.y; v[6] += a1.z; v[7] += a1.w;
                const uint4 hb = pack_bf16x8(v);
                hr[c] = hb;
                unpack_bf16x8(hb, v);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = rsqrtf(ss / (float)d + eps);
        // each lane reads back the chunks it wrote itself
        const uint4* src = ADD ? reinterpret_cast<const uint4*>(hr) : xr;
        uint4* yr = reinterpret_cast<uint4*>(y + r * d);
#pragma unroll 4
        for (int c = lane; c < nch; c += 32) {
            float v[8], w[8];
            unpack_bf16x8(src[c], v);
            unpack_bf16x8(gv[c], w);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = w[i] * (v[i] * inv);
            yr[c] = pack_bf16x8(v);
        }
    }
}

struct RopeArgs {
    const float* qkv;     // [T][(Hq + 2 Hkv) hd] fp32: the fused projection's output
    __nv_bfloat16* q;     // [T][Hq hd]
    __nv_bfloat16* k;     // [T][Hkv hd] (nullable: keys only to the cache)
    __nv_bfloat16* v;     // [T][Hkv hd] (nullable)
    int64_t T;
    int64_t S;            // tokens per sequence (prefill): position = t mod S, sequence t / S
    const int32_t* pos;   // decode: token t is sequence t's next token, at position pos[t] (nullable)
    __nv_bfloat16* k_cache;  // [B][Hkv][cache_max][hd] (nullable): keys appended at their position
    __nv_bfloat16* v_cache;
    int64_t cache_max;
    int Hq, Hkv, hd;
    double theta[kRopeMaxPairs];  // base^(-2i/hd), i = 0 .. hd/2 - 1
};

// Block (hd/2, kRopeTokens): thread x handles channel pair x of every head of
// one token. The angle pos * theta_i is formed and reduced modulo 2 pi in
// double precision (pos reaches 32767 and beyond, where a float product would
// be off by 1e-3 rad), then the reduced angle goes to sincosf. With caches,
// the token's keys and values are also stored at their position in the
// head-major caches (prefill: positions 0 .. S-1 of every sequence; decode:
// position pos[t] of sequence t).
__global__ void __launch_bounds__(256) rope_split_kernel(const __grid_constant__ RopeArgs a) {
    pdl_trigger();
    pdl_wait();
    const int i = threadIdx.x;
    const int64_t t = (int64_t)blockIdx.x * kRopeTokens + threadIdx.y;
    if (t >= a.T) return;
    const int64_t seq = a.pos != nullptr ? t : t / a.S;
    const int64_t p = a.pos != nullptr ? (int64_t)a.pos[t] : t % a.S;
    // a cache write needs a slot: a full cache is reported and not written
    bool to_cache = a.k_cache != nullptr;
    if (to_cache && (p < 0 || p >= a.cache_max)) {
        if (i == 0) report_error(MOE_ERR_DEVICE_CHECK, K_ROPE, W_INDEX);
        to_cache = false;
    }
    const double pos = (double)p;
    const double twopi = 6.283185307179586476925;
    double ang = pos * a.theta[i];
    ang -= twopi * rint(ang / twopi);
    float sn, cs;
    sincosf((float)ang, &sn, &cs);
    const int W = (a.Hq + 2 * a.Hkv) * a.hd;
    const float2* row = reinterpret_cast<const float2*>(a.qkv + t * W);
    const int P = a.hd >> 1;
    uint32_t* q = reinterpret_cast<uint32_t*>(a.q + t * (int64_t)a.Hq * a.hd);
    uint32_t* k = a.k != nullptr ? reinterpret_cast<uint32_t*>(a.k + t * (int64_t)a.Hkv * a.hd) : nullptr;
    uint32_t* v = a.v != nullptr ? reinterpret_cast<uint32_t*>(a.v + t * (int64_t)a.Hkv * a.hd) : nullptr;
    for (int h = 0; h < a.Hq; ++h) {
        const float2 z = row[h * P + i];
        q[h * P + i] = pack_bf16x2(z.x * cs - z.y * sn, z.x * sn + z.y * cs);
    }
    for (int h = 0; h < a.Hkv; ++h) {
        const float2 z = row[(a.Hq + h) * P + i];
        const uint32_t kv = pack_bf16x2(z.x * cs - z.y * sn, z.x * sn + z.y * cs);
        if (k != nullptr) k[h * P + i] = kv;
        if (to_cache)
            reinterpret_cast<uint32_t*>(a.k_cache + ((seq * a.Hkv + h) * a.cache_max + p) * a.hd)[i] = kv;
    }
    for (int h = 0; h < a.Hkv; ++h) {
        const float2 z = row[(a.Hq + a.Hkv + h) * P + i];
        const uint32_t vv = pack_bf16x2(z.x, z.y);
        if (v != nullptr) v[h * P + i] = vv;
        if (to_cache)
            reinterpret_cast<uint32_t*>(a.v_cache + ((seq * a.Hkv + h) * a.cache_max + p) * a.hd)[i] = vv;
    }
}

// out = bf16(a + b), n a multiple of 8.
__global__ void __launch_bounds__(256) residual_add_kernel(const __nv_bfloat16* __restrict__ a,
                                                           const __nv_bfloat16* __restrict__ b, int64_t n,
                                                           __nv_bfloat16* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    const int64_t n8 = n >> 3;
    const uint4* av = reinterpret_cast<const uint4*>(a);
    const uint4* bv = reinterpret_cast<const uint4*>(b);
    uint4* ov = reinterpret_cast<uint4*>(out);
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < n8; c += (int64_t)gridDim.x * blockDim.x) {
        float x[8], y[8];
        unpack_bf16x8(av[c], x);
        unpack_bf16x8(bv[c], y);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] += y[i];
        ov[c] = pack_bf16x8(x);
    }
}

}  // namespace moe
