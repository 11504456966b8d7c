// Causal grouped-query attention on the 5th-generation tensor cores.
//
// Mixtral keeps LLaMA's attention: rotary positions and grouped-query heads
// ("Mixtral" lineage page, step "GPT-2 vs Mixtral"); the Mixtral notes
// (royalroad.pages.dev, Architecture) give 32 query heads and 8 KV heads, and
// the breakdown's 41.9M attention parameters per layer make a head 128 wide.
//
// One CTA computes 128 queries of one head of one sequence against the keys at
// or before them, 128 keys at a time, with the running-maximum softmax (the
// exact result, accumulated tile by tile with rescaling):
//   S = Q K^T            tcgen05.mma, M = 128 queries, N = 128 keys, K = 128
//                        channels; Q and K tiles K-major in shared memory
//                        (TMA, 128-byte swizzle), S in tensor memory
//   P = exp(S - m)       4 softmax warps, one query row per thread, written to
//                        shared memory in bf16 in the swizzled K-major layout
//   O += P V             tcgen05.mma, M = 128, N = 128 channels, K = 128 keys;
//                        V read as stored ([key][channel], MN-major), O in
//                        tensor memory, rescaled in place when a row's maximum
//                        grows
// Warp 0 issues TMA loads (Q once, then K and V tiles through two stages),
// warp 1 issues the MMAs (S of the next tile is issued before P V of the
// current one, so it overlaps the softmax), warps 2-5 run the softmax and the
// epilogue O / l. Every wait is bounded; on a timeout the CTA latches
// MOE_ERR_TIMEOUT, lets its copies and MMAs land and returns.
#pragma once

#include "ffn_tc.cuh"

namespace moe {

constexpr int kAttnHD = 128;                       // head width
constexpr int kAttnTile = 128;                     // queries per CTA, keys per step
constexpr int kAttnThreads = 192;
constexpr uint32_t kAttnBox = 128 * 64 * 2;        // 16 KB: 128 rows x 64 channels
constexpr uint32_t kAttnTileBytes = 2 * kAttnBox;  // 32 KB: 128 rows x 128 channels

struct AttnControl {
    uint64_t q_full;
    uint64_t kv_full[2];
    uint64_t kv_empty[2];
    uint64_t s_full, s_free, p_full, p_free, drain;
    uint32_t tmem_base;
    int abort_flag;
};

// Q | K0 | V0 | K1 | V1 | P | control
constexpr size_t kAttnSmemBytes = 1024 + 6 * (size_t)kAttnTileBytes + sizeof(AttnControl);
static_assert(kAttnSmemBytes <= 227 * 1024, "attention CTA exceeds the shared memory of a CTA");

struct AttnArgs {
    __nv_bfloat16* o;   // [T][Hq hd]
    int64_t S;          // tokens per sequence
    int B, Hq, Hkv;
    int n_qt;           // query tiles per sequence
    float scale_log2;   // log2(e) / sqrt(hd)
    uint64_t timeout_ns;
};

__device__ __forceinline__ void unpack_bf16x8_attn(const uint4& u, float (&v)[8]) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(p[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (a0, a1) * (b0, b1) + (c0, c1) as one paired fp32 FMA.
__device__ __forceinline__ void ffma2(float a0, float a1, float b0, float b1, float c0, float c1, float& d0, float& d1) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// (a0, a1) + (b0, b1) as one paired fp32 add.
__device__ __forceinline__ void fadd2(float a0, float a1, float b0, float b1, float& d0, float& d1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void attn_abort(AttnControl* c, int where) {
    report_error(MOE_ERR_TIMEOUT, K_ATTN, where);
    *reinterpret_cast<volatile int*>(&c->abort_flag) = 1;
}

// Grid: n_qt * B * Hq CTAs, the query tiles with the most keys first; the
// heads that share a KV head are neighbours, so their K and V tiles meet in L2.
__global__ void __launch_bounds__(kAttnThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v, const AttnArgs a) {
    extern __shared__ unsigned char attn_smem_raw[];
    unsigned char* smem = align1024(attn_smem_raw);
    AttnControl* ctl = reinterpret_cast<AttnControl*>(smem + 6 * (size_t)kAttnTileBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t tmo = a.timeout_ns;
    volatile int* abort_flag = &ctl->abort_flag;

    const int per_qt = a.B * a.Hq;
    const int qt = a.n_qt - 1 - (int)(blockIdx.x / per_qt);
    const int rem = (int)(blockIdx.x % per_qt);
    const int b = rem / a.Hq;
    const int h = rem - b * a.Hq;
    const int kvh = h / (a.Hq / a.Hkv);
    const int64_t row0 = (int64_t)b * a.S;   // first token of the sequence
    const int q0 = qt * kAttnTile;           // first query position of the tile
    const int nkv = qt + 1;                  // key tiles at or before the queries

    const uint32_t sQ = smem_u32(smem);
    auto sK = [&](int st) { return sQ + (uint32_t)(1 + 2 * st) * kAttnTileBytes; };
    auto sV = [&](int st) { return sQ + (uint32_t)(2 + 2 * st) * kAttnTileBytes; };
    const uint32_t sP = sQ + 5 * kAttnTileBytes;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&ctl->q_full), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&ctl->kv_full[s]), 1);
            mbar_init(smem_u32(&ctl->kv_empty[s]), 1);
        }
        mbar_init(smem_u32(&ctl->s_full), 1);
        mbar_init(smem_u32(&ctl->s_free), 4);
        mbar_init(smem_u32(&ctl->p_full), 4);
        mbar_init(smem_u32(&ctl->p_free), 1);
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), 256);
        tmem_relinquish();
    }
    pdl_trigger();
    pdl_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = ctl->tmem_base;          // columns 0-127: scores
    const uint32_t tO = ctl->tmem_base + 128;    // columns 128-255: output accumulator

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_normal();  // re-read by the group's heads and later tiles
            const uint32_t qb = smem_u32(&ctl->q_full);
            mbar_arrive_expect_tx(qb, kAttnTileBytes);
            tma_load_2d(sQ, &map_q, qb, h * kAttnHD, (int)(row0 + q0), pol_q);
            tma_load_2d(sQ + kAttnBox, &map_q, qb, h * kAttnHD + 64, (int)(row0 + q0), pol_q);
            uint32_t issued = 0, issued_ph = 0;
            for (int j = 0; j < nkv; ++j) {
                const int st = j & 1;
                const uint32_t ph = (uint32_t)(j >> 1) & 1u;
                if (!mbar_wait(smem_u32(&ctl->kv_empty[st]), ph ^ 1u, tmo, abort_flag)) {
                    attn_abort(ctl, W_PRODUCER);
                    break;
                }
                const uint32_t fb = smem_u32(&ctl->kv_full[st]);
                mbar_arrive_expect_tx(fb, 2 * kAttnTileBytes);
                const int ky = (int)(row0 + (int64_t)j * kAttnTile);
                tma_load_2d(sK(st), &map_k, fb, kvh * kAttnHD, ky, pol_kv);
                tma_load_2d(sK(st) + kAttnBox, &map_k, fb, kvh * kAttnHD + 64, ky, pol_kv);
                tma_load_2d(sV(st), &map_v, fb, kvh * kAttnHD, ky, pol_kv);
                tma_load_2d(sV(st) + kAttnBox, &map_v, fb, kvh * kAttnHD + 64, ky, pol_kv);
                issued |= 1u << st;
                issued_ph = (issued_ph & ~(1u << st)) | (ph << st);
            }
            // every copy this CTA started lands before it leaves (immediate on the normal path)
            drain_wait(smem_u32(&ctl->q_full), 0, tmo, K_ATTN);
            for (int st = 0; st < 2; ++st)
                if (issued & (1u << st)) drain_wait(smem_u32(&ctl->kv_full[st]), (issued_ph >> st) & 1u, tmo, K_ATTN);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128);
            constexpr uint32_t idesc_o = idesc_bf16_f32(128, 128, false, true);
            bool ok = mbar_wait(smem_u32(&ctl->q_full), 0, tmo, abort_flag);
            if (!ok) attn_abort(ctl, W_MMA);
            bool any = false;
            for (int j = 0; ok && j <= nkv; ++j) {
                if (j < nkv) {
                    // S = Q K_j^T, once the softmax has read S of the previous tile
                    const int st = j & 1;
                    if (!mbar_wait(smem_u32(&ctl->kv_full[st]), (uint32_t)(j >> 1) & 1u, tmo, abort_flag) ||
                        (j > 0 && !mbar_wait(smem_u32(&ctl->s_free), (uint32_t)(j - 1) & 1u, tmo, abort_flag))) {
                        attn_abort(ctl, W_MMA);
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kAttnHD / 16; ++kk) {
                        const uint32_t off = (uint32_t)(kk >> 2) * kAttnBox;
                        const uint64_t ad = sw128_kmajor_desc(sQ + off) + 2ull * (kk & 3);
                        const uint64_t bd = sw128_kmajor_desc(sK(st) + off) + 2ull * (kk & 3);
                        mma_bf16(tS, ad, bd, idesc_s, kk > 0);
                    }
                    any = true;
                    mma_commit(smem_u32(&ctl->s_full));
                }
                if (j > 0) {
                    // O += P_{j-1} V_{j-1}
                    const int jj = j - 1, st = jj & 1;
                    if (!mbar_wait(smem_u32(&ctl->p_full), (uint32_t)jj & 1u, tmo, abort_flag)) {
                        attn_abort(ctl, W_MMA);
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kAttnTile / 16; ++kk) {
                        const uint64_t ad = sw128_kmajor_desc(sP + (uint32_t)(kk >> 2) * kAttnBox) + 2ull * (kk & 3);
                        const uint64_t bd = sw128_mnmajor_desc(sV(st), kAttnBox) + 128ull * kk;
                        mma_bf16(tO, ad, bd, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&ctl->kv_empty[st]));
                    mma_commit(smem_u32(&ctl->p_free));
                }
            }
            if (any) {
                mma_commit(smem_u32(&ctl->drain));
                drain_wait(smem_u32(&ctl->drain), 0, tmo, K_ATTN);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int sub = warp & 3;                  // tensor-memory lanes 32 sub .. 32 sub + 31
        const int row = sub * 32 + lane;           // query row of the tile
        const int qpos = q0 + row;
        const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
        const float sl2 = a.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            // waits are voted warp-wide: the tensor-memory loads below need all 32 lanes
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->s_full), (uint32_t)j & 1u, tmo, abort_flag))) {
                attn_abort(ctl, W_EPILOGUE);
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[128];
#pragma unroll
            for (int c = 0; c < 8; ++c) tmem_ld16(tS + lane_off + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&sv[16 * c]));
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->s_free));
            // causal and end-of-sequence mask: only the diagonal tile has keys after a query
            const int kbase = j * kAttnTile;
            float mx = -INFINITY;
            if (j == qt) {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    const int key = kbase + c;
                    const bool masked = key > qpos || (int64_t)key >= a.S;
                    const float s = masked ? -INFINITY : __uint_as_float(sv[c]);
                    sv[c] = __float_as_uint(s);
                    mx = fmaxf(mx, s);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 128; ++c) mx = fmaxf(mx, __uint_as_float(sv[c]));
            }
            const float m_new = fmaxf(m, mx * sl2);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = fast_exp2(m - m_use);
            float sum = 0.f;
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const float p0 = fast_exp2(fmaf(__uint_as_float(sv[2 * c]), sl2, -m_use));
                const float p1 = fast_exp2(fmaf(__uint_as_float(sv[2 * c + 1]), sl2, -m_use));
                sum += p0 + p1;
                pk[c] = pack_bf16x2(p0, p1);
            }
            l = fmaf(l, alpha, sum);
            m = m_new;
            if (j > 0) {
                // P V of the previous tile has finished with P and with O
                if (!__all_sync(0xffffffffu,
                                mbar_wait(smem_u32(&ctl->p_free), (uint32_t)(j - 1) & 1u, tmo, abort_flag))) {
                    attn_abort(ctl, W_EPILOGUE);
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha < 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        uint32_t o[16];
                        tmem_ld16(tO + lane_off + 16 * c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st16(tO + lane_off + 16 * c, o);
                    }
                    tmem_wait_st();
                }
            }
            // P row in the 128-byte-swizzled K-major layout: two 64-key blocks,
            // 16-byte chunk q of row r stored at chunk q ^ (r % 8)
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const uint32_t addr = sP + (uint32_t)(q >> 3) * kAttnBox + (uint32_t)row * 128u +
                                      ((uint32_t)((q & 7) ^ (row & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * q]),
                             "r"(pk[4 * q + 1]), "r"(pk[4 * q + 2]), "r"(pk[4 * q + 3])
                             : "memory");
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full));
        }
        if (ok && __all_sync(0xffffffffu,
                             mbar_wait(smem_u32(&ctl->p_free), (uint32_t)(nkv - 1) & 1u, tmo, abort_flag))) {
            tc_fence_after();
            const float inv_l = 1.f / l;
            const bool valid = (int64_t)qpos < a.S;
            __nv_bfloat16* out = a.o + (row0 + qpos) * (int64_t)a.Hq * kAttnHD + (int64_t)h * kAttnHD;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t o[16];
                tmem_ld16(tO + lane_off + 16 * c, o);
                tmem_wait_ld();
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(out + 16 * c);
                    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
            }
        } else if (ok) {
            attn_abort(ctl, W_EPILOGUE);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(ctl->tmem_base, 256);
}

// ---------------------------------------------------------------------------
// Two query heads of one KV group per CTA (grouped-query attention with an
// even group): both heads read the same K and V tiles, loaded once. Each head
// has its own 4 softmax warps, score tile S and accumulator O in tensor
// memory (512 columns); the MMA warp alternates between the heads, so one
// head's S = Q K^T and O += P V run on the tensor core while the other head's
// softmax runs on the CUDA cores. P (bf16) is written into the head's S
// columns with tcgen05.st and read from there as the A operand of P V: the
// MMAs of one thread run in issue order, so O += P_j V_j has read P_j before
// the next S = Q K_{j+1} overwrites those columns, and the completion of that
// S also tells the softmax warps that O holds P_j V_j. The running maximum is
// rescaled lazily: O and l keep their reference until a row's maximum grows by
// more than 2^8 (the result is exact either way; the reference only bounds
// the size of P).
// ---------------------------------------------------------------------------
constexpr int kAttnPairThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-5 head 0, warps 6-9 head 1
constexpr float kAttnRescaleLog2 = 8.f;

struct AttnPairControl {
    uint64_t q_full;
    uint64_t kv_full[2];
    uint64_t kv_empty[2];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_full[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// Q0 | Q1 | K0 | V0 | K1 | V1 | control
constexpr size_t kAttnPairSmemBytes = 1024 + 6 * (size_t)kAttnTileBytes + sizeof(AttnPairControl);
static_assert(kAttnPairSmemBytes <= 227 * 1024, "attention CTA exceeds the shared memory of a CTA");

__device__ __forceinline__ void attn_pair_abort(AttnPairControl* c, int where) {
    report_error(MOE_ERR_TIMEOUT, K_ATTN, where);
    *reinterpret_cast<volatile int*>(&c->abort_flag) = 1;
}

// Grid: n_qt * B * Hq / 2 CTAs, the query tiles with the most keys first.
__global__ void __launch_bounds__(kAttnPairThreads, 1)
    attention_pair_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                          const __grid_constant__ CUtensorMap map_v, const AttnArgs a) {
    extern __shared__ unsigned char attn_smem_raw[];
    unsigned char* smem = align1024(attn_smem_raw);
    AttnPairControl* ctl = reinterpret_cast<AttnPairControl*>(smem + 6 * (size_t)kAttnTileBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t tmo = a.timeout_ns;
    volatile int* abort_flag = &ctl->abort_flag;

    const int pairs = a.Hq >> 1;
    const int per_qt = a.B * pairs;
    const int qt = a.n_qt - 1 - (int)(blockIdx.x / per_qt);
    const int rem = (int)(blockIdx.x % per_qt);
    const int b = rem / pairs;
    const int h0 = 2 * (rem - b * pairs);          // heads h0 and h0 + 1
    const int kvh = h0 / (a.Hq / a.Hkv);
    const int64_t row0 = (int64_t)b * a.S;
    const int q0 = qt * kAttnTile;
    const int nkv = qt + 1;

    const uint32_t sQ = smem_u32(smem);
    auto sQh = [&](int x) { return sQ + (uint32_t)x * kAttnTileBytes; };
    auto sK = [&](int st) { return sQ + (uint32_t)(2 + 2 * st) * kAttnTileBytes; };
    auto sV = [&](int st) { return sQ + (uint32_t)(3 + 2 * st) * kAttnTileBytes; };

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&ctl->q_full), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&ctl->kv_full[s]), 1);
            mbar_init(smem_u32(&ctl->kv_empty[s]), 1);
            mbar_init(smem_u32(&ctl->s_full[s]), 1);
            mbar_init(smem_u32(&ctl->p_full[s]), 4);
            mbar_init(smem_u32(&ctl->o_full[s]), 1);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), 512);
        tmem_relinquish();
    }
    pdl_trigger();
    pdl_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // head x: S (and P) at columns 256 x .. 256 x + 127, O at 256 x + 128 .. 256 x + 255
    const uint32_t tmem = ctl->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_normal();
            const uint32_t qb = smem_u32(&ctl->q_full);
            mbar_arrive_expect_tx(qb, 2 * kAttnTileBytes);
            for (int x = 0; x < 2; ++x) {
                tma_load_2d(sQh(x), &map_q, qb, (h0 + x) * kAttnHD, (int)(row0 + q0), pol_q);
                tma_load_2d(sQh(x) + kAttnBox, &map_q, qb, (h0 + x) * kAttnHD + 64, (int)(row0 + q0), pol_q);
            }
            uint32_t issued = 0, issued_ph = 0;
            for (int j = 0; j < nkv; ++j) {
                const int st = j & 1;
                const uint32_t ph = (uint32_t)(j >> 1) & 1u;
                if (!mbar_wait(smem_u32(&ctl->kv_empty[st]), ph ^ 1u, tmo, abort_flag)) {
                    attn_pair_abort(ctl, W_PRODUCER);
                    break;
                }
                const uint32_t fb = smem_u32(&ctl->kv_full[st]);
                mbar_arrive_expect_tx(fb, 2 * kAttnTileBytes);
                const int ky = (int)(row0 + (int64_t)j * kAttnTile);
                tma_load_2d(sK(st), &map_k, fb, kvh * kAttnHD, ky, pol_kv);
                tma_load_2d(sK(st) + kAttnBox, &map_k, fb, kvh * kAttnHD + 64, ky, pol_kv);
                tma_load_2d(sV(st), &map_v, fb, kvh * kAttnHD, ky, pol_kv);
                tma_load_2d(sV(st) + kAttnBox, &map_v, fb, kvh * kAttnHD + 64, ky, pol_kv);
                issued |= 1u << st;
                issued_ph = (issued_ph & ~(1u << st)) | (ph << st);
            }
            drain_wait(smem_u32(&ctl->q_full), 0, tmo, K_ATTN);
            for (int st = 0; st < 2; ++st)
                if (issued & (1u << st)) drain_wait(smem_u32(&ctl->kv_full[st]), (issued_ph >> st) & 1u, tmo, K_ATTN);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128);
            constexpr uint32_t idesc_o = idesc_bf16_f32(128, 128, false, true);
            bool ok = mbar_wait(smem_u32(&ctl->q_full), 0, tmo, abort_flag) &&
                      mbar_wait(smem_u32(&ctl->kv_full[0]), 0, tmo, abort_flag);
            bool any = false;
            auto issue_s = [&](int x, int st) {
                const uint32_t d = tmem + 256u * (uint32_t)x;
#pragma unroll
                for (int kk = 0; kk < kAttnHD / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * kAttnBox;
                    const uint64_t ad = sw128_kmajor_desc(sQh(x) + off) + 2ull * (kk & 3);
                    const uint64_t bd = sw128_kmajor_desc(sK(st) + off) + 2ull * (kk & 3);
                    mma_bf16(d, ad, bd, idesc_s, kk > 0);
                }
                mma_commit(smem_u32(&ctl->s_full[x]));
            };
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                issue_s(1, 0);
                any = true;
            } else {
                attn_pair_abort(ctl, W_MMA);
            }
            for (int j = 0; ok && j < nkv; ++j) {
                const int st = j & 1;
                for (int x = 0; ok && x < 2; ++x) {
                    if (!mbar_wait(smem_u32(&ctl->p_full[x]), (uint32_t)j & 1u, tmo, abort_flag)) {
                        attn_pair_abort(ctl, W_MMA);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t p_tmem = tmem + 256u * (uint32_t)x;
                    const uint32_t o_tmem = p_tmem + 128u;
#pragma unroll
                    for (int kk = 0; kk < kAttnTile / 16; ++kk) {
                        const uint64_t bd = sw128_mnmajor_desc(sV(st), kAttnBox) + 128ull * kk;
                        mma_bf16_ts(o_tmem, p_tmem + 8u * (uint32_t)kk, bd, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    if (x == 1) mma_commit(smem_u32(&ctl->kv_empty[st]));  // both heads are done with K_j, V_j
                    if (j + 1 < nkv) {
                        if (x == 0 &&
                            !mbar_wait(smem_u32(&ctl->kv_full[st ^ 1]), (uint32_t)((j + 1) >> 1) & 1u, tmo, abort_flag)) {
                            attn_pair_abort(ctl, W_MMA);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_s(x, st ^ 1);
                    } else {
                        mma_commit(smem_u32(&ctl->o_full[x]));
                    }
                }
            }
            if (any) {
                mma_commit(smem_u32(&ctl->drain));
                drain_wait(smem_u32(&ctl->drain), 0, tmo, K_ATTN);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue of one head
        const int x = (warp - 2) >> 2;             // head slot
        const int sub = warp & 3;                  // tensor-memory lanes 32 sub .. 32 sub + 31
        const int row = sub * 32 + lane;
        const int qpos = q0 + row;
        const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
        const uint32_t tS = tmem + 256u * (uint32_t)x + lane_off;
        const uint32_t tO = tS + 128u;
        const float sl2 = a.scale_log2;
        float m_ref = 0.f, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            // warp-wide vote: the tensor-memory loads and stores below need all 32 lanes
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->s_full[x]), (uint32_t)j & 1u, tmo, abort_flag))) {
                attn_pair_abort(ctl, W_EPILOGUE);
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, &sv[32 * c]);
            tmem_wait_ld();
            const bool diag = j == qt;
            if (diag) {
                // the diagonal tile: keys after the query, and past the sequence's end, drop out
                const int kbase = j * kAttnTile;
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    const int key = kbase + c;
                    if (key > qpos || (int64_t)key >= a.S) sv[c] = __float_as_uint(-INFINITY);
                }
            }
            // row maximum: three-input max over 4 independent chains
            float mx4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) mx4[i] = fmaxf(__uint_as_float(sv[i]), __uint_as_float(sv[4 + i]));
#pragma unroll
            for (int c = 8; c < 128; c += 8)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    mx4[i] = fmax3f(mx4[i], __uint_as_float(sv[c + i]), __uint_as_float(sv[c + 4 + i]));
            const float mx = fmax3f(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
            const float m_tile = mx * sl2;
            if (j == 0) {
                m_ref = m_tile == -INFINITY ? 0.f : m_tile;
            } else {
                const bool grow = m_tile > m_ref + kAttnRescaleLog2;
                if (__any_sync(0xffffffffu, grow)) {
                    // O holds P_{j-1} V_{j-1} (the MMA that wrote S_j ran after it): rescale it in place
                    const float m_new = grow ? m_tile : m_ref;
                    const float alpha = fast_exp2(m_ref - m_new);
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        uint32_t o[16];
                        tmem_ld16(tO + 16 * c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st16(tO + 16 * c, o);
                    }
                    l *= alpha;
                    m_ref = m_new;
                }
            }
            // p = 2^(s log2(e) / sqrt(hd) - m): the scaling as paired FMAs, row
            // sums over 4 paired chains. (Moving a share of the exponentials to
            // a polynomial on the FMA pipe measured slower: the softmax is
            // bound by instruction issue, not by the special-function unit.)
            float sa[4], sb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) sa[i] = sb[i] = 0.f;
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                float x0, x1;
                ffma2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1]), sl2, sl2, -m_ref, -m_ref, x0, x1);
                const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                fadd2(sa[c & 3], sb[c & 3], p0, p1, sa[c & 3], sb[c & 3]);
                pk[c] = pack_bf16x2(p0, p1);
            }
            l += ((sa[0] + sb[0]) + (sa[1] + sb[1])) + ((sa[2] + sb[2]) + (sa[3] + sb[3]));
            // P over the first 64 columns of S: keys 2c and 2c + 1 in column c
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_st16(tS + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&pk[16 * c]));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full[x]));
        }
        if (ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->o_full[x]), 0, tmo, abort_flag))) {
            tc_fence_after();
            const float inv_l = 1.f / l;
            const bool valid = (int64_t)qpos < a.S;
            __nv_bfloat16* out = a.o + (row0 + qpos) * (int64_t)a.Hq * kAttnHD + (int64_t)(h0 + x) * kAttnHD;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t o[16];
                tmem_ld16(tO + 16 * c, o);
                tmem_wait_ld();
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(out + 16 * c);
                    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
            }
        } else if (ok) {
            attn_pair_abort(ctl, W_EPILOGUE);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(ctl->tmem_base, 512);
}

// ---------------------------------------------------------------------------
// Decode: one new token per sequence against its key/value cache. The cache
// is head-major, [B][Hkv][cache_max][128] bf16, so a KV head's keys are one
// contiguous run. CTA (split s, KV head, sequence) takes an equal share of the
// n = len + 1 valid keys (the new token's were appended by the RoPE step), 64
// keys per step, for the G query heads that share the KV head:
//   S = Q K^T     tcgen05.mma M = 128 (rows 0 .. G-1 are the heads; the other
//                 rows are not read), N = 64 keys, K = 128 channels; Q held in
//                 tensor memory (A operand), K by TMA (128-byte swizzle), S in
//                 tensor memory
//   softmax       warp 0, one row per lane: running maximum and sum, O
//                 rescaled in place when the maximum grows, P (bf16) written
//                 over S
//   O += P V      tcgen05.mma M = 128, N = 128 channels, K = 64 keys, P from
//                 tensor memory, V as stored (MN-major)
// Keys and values stream through three shared-memory stages, so the tensor
// core only waits on HBM. Each CTA writes one unnormalised partial (O, m, l) per
// head; a second kernel merges the splits in order (flash decoding).
// ---------------------------------------------------------------------------
constexpr int kDecChunk = 64;                        // keys per step
constexpr int kDecThreads = 96;                      // warp 0 softmax, warp 1 TMA, warp 2 MMA
constexpr int kDecMaxGroup = 32;                     // query heads per KV head (one row per lane)
constexpr int kDecCtasPerSm = 2;
constexpr int kDecStages = 3;
constexpr uint32_t kDecBox = 64 * 64 * 2;            // 8 KB: 64 keys x 64 channels
constexpr uint32_t kDecStageBytes = 4 * kDecBox;     // keys (two boxes) + values (two boxes)

struct DecControl {
    uint64_t q_ready;
    uint64_t kv_full[kDecStages];
    uint64_t kv_empty[kDecStages];
    uint64_t s_full, p_full, o_full, drain;
    uint32_t tmem_base;
    int abort_flag;
};

// stages | control
constexpr size_t kDecSmemBytes = 1024 + (size_t)kDecStages * kDecStageBytes + sizeof(DecControl);

struct DecodeArgs {
    const __nv_bfloat16* q;       // [B][Hq hd]
    const int32_t* len;           // [B] keys cached before this token
    float* part_o;                // [B][Hq][splits][hd]
    float* part_ml;               // [B][Hq][splits][2]
    int64_t cache_max;
    int Hq, Hkv, splits;
    float scale_log2;
    uint64_t timeout_ns;
};

__device__ __forceinline__ void dec_abort(DecControl* c, int where) {
    report_error(MOE_ERR_TIMEOUT, K_ATTN, where);
    *reinterpret_cast<volatile int*>(&c->abort_flag) = 1;
}

// map_k, map_v: the caches viewed as [B Hkv cache_max][128], boxes of 64
// channels x 64 keys.
__global__ void __launch_bounds__(kDecThreads, 1)
    attention_decode_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                            const DecodeArgs a) {
    extern __shared__ unsigned char dec_smem_raw[];
    unsigned char* smem = align1024(dec_smem_raw);
    DecControl* ctl = reinterpret_cast<DecControl*>(smem + (size_t)kDecStages * kDecStageBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t tmo = a.timeout_ns;
    volatile int* abort_flag = &ctl->abort_flag;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int G = a.Hq / a.Hkv;
    const uint32_t sbase = smem_u32(smem);
    auto sK = [&](int st) { return sbase + (uint32_t)st * kDecStageBytes; };
    auto sV = [&](int st) { return sK(st) + 2 * kDecBox; };

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&ctl->q_ready), 1);
        for (int s = 0; s < kDecStages; ++s) {
            mbar_init(smem_u32(&ctl->kv_full[s]), 1);
            mbar_init(smem_u32(&ctl->kv_empty[s]), 1);
        }
        mbar_init(smem_u32(&ctl->s_full), 1);
        mbar_init(smem_u32(&ctl->p_full), 1);
        mbar_init(smem_u32(&ctl->o_full), 1);
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&ctl->tmem_base), 256);
        tmem_relinquish();
    }
    if (warp == 1 && lane == 0) {
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
    }
    pdl_trigger();
    pdl_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = ctl->tmem_base;         // columns 0-63: scores (P over columns 0-31)
    const uint32_t tQ = ctl->tmem_base + 64;    // columns 64-127: the queries, two bf16 per column
    const uint32_t tO = ctl->tmem_base + 128;   // columns 128-255: output accumulator

    const int64_t n_all = (int64_t)a.len[b] + 1;
    const int64_t n = n_all < a.cache_max ? n_all : a.cache_max;
    const int64_t nch = (n + kDecChunk - 1) / kDecChunk;
    const int64_t per = (nch + a.splits - 1) / a.splits;
    const int64_t c_begin = split * per;
    const int64_t c_end = c_begin + per < nch ? c_begin + per : nch;
    const int steps = c_end > c_begin ? (int)(c_end - c_begin) : 0;
    const int64_t row0 = ((int64_t)b * a.Hkv + kvh) * a.cache_max;

    if (warp == 1) {
        // ------------------------------------------------------------ TMA
        if (lane == 0 && steps > 0) {
            const uint64_t pol = policy_evict_first();
            uint32_t issued = 0, issued_ph = 0;
            for (int i = 0; i < steps; ++i) {
                const int st = i % kDecStages;
                const uint32_t ph = (uint32_t)(i / kDecStages) & 1u;
                if (!mbar_wait(smem_u32(&ctl->kv_empty[st]), ph ^ 1u, tmo, abort_flag)) {
                    dec_abort(ctl, W_PRODUCER);
                    break;
                }
                const uint32_t fb = smem_u32(&ctl->kv_full[st]);
                mbar_arrive_expect_tx(fb, kDecStageBytes);
                const int ky = (int)(row0 + (c_begin + i) * kDecChunk);
                tma_load_2d(sK(st), &map_k, fb, 0, ky, pol);
                tma_load_2d(sK(st) + kDecBox, &map_k, fb, 64, ky, pol);
                tma_load_2d(sV(st), &map_v, fb, 0, ky, pol);
                tma_load_2d(sV(st) + kDecBox, &map_v, fb, 64, ky, pol);
                issued |= 1u << st;
                issued_ph = (issued_ph & ~(1u << st)) | (ph << st);
            }
            for (int st = 0; st < kDecStages; ++st)
                if (issued & (1u << st)) drain_wait(smem_u32(&ctl->kv_full[st]), (issued_ph >> st) & 1u, tmo, K_ATTN);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ MMA
        if (lane == 0 && steps > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, kDecChunk);
            constexpr uint32_t idesc_o = idesc_bf16_f32(128, 128, false, true);
            bool ok = mbar_wait(smem_u32(&ctl->q_ready), 0, tmo, abort_flag);
            if (!ok) dec_abort(ctl, W_MMA);
            bool any = false;
            for (int i = 0; ok && i < steps; ++i) {
                const int st = i % kDecStages;
                if (!mbar_wait(smem_u32(&ctl->kv_full[st]), (uint32_t)(i / kDecStages) & 1u, tmo, abort_flag)) {
                    dec_abort(ctl, W_MMA);
                    break;
                }
                tc_fence_after();
                // S = Q K^T (issued after the previous P V, which read P from these columns)
#pragma unroll
                for (int kk = 0; kk < kAttnHD / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2);
                    const uint64_t bd = sw128_kmajor_desc(sK(st) + off * kDecBox) + 2ull * (kk & 3);
                    mma_bf16_ts(tS, tQ + 8u * (uint32_t)kk, bd, idesc_s, kk > 0);
                }
                any = true;
                mma_commit(smem_u32(&ctl->s_full));
                if (!mbar_wait(smem_u32(&ctl->p_full), (uint32_t)i & 1u, tmo, abort_flag)) {
                    dec_abort(ctl, W_MMA);
                    break;
                }
                tc_fence_after();
                // O += P V
#pragma unroll
                for (int kk = 0; kk < kDecChunk / 16; ++kk) {
                    const uint64_t bd = sw128_mnmajor_desc(sV(st), kDecBox) + 128ull * kk;
                    mma_bf16_ts(tO, tS + 8u * (uint32_t)kk, bd, idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(smem_u32(&ctl->kv_empty[st]));
                if (i + 1 == steps) mma_commit(smem_u32(&ctl->o_full));
            }
            if (any) {
                mma_commit(smem_u32(&ctl->drain));
                drain_wait(smem_u32(&ctl->drain), 0, tmo, K_ATTN);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + partial (warp 0: lanes = rows)
        const int row = lane;
        const float sl2 = a.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        if (steps > 0) {
            // the group's queries into tensor memory, one head per lane (rows G .. 31 zero)
            const uint4* qr = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * a.Hq + kvh * G + row) * kAttnHD);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[16];
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4) {
                    const uint4 u = row < G ? qr[4 * c + v4] : make_uint4(0u, 0u, 0u, 0u);
                    w[4 * v4] = u.x;
                    w[4 * v4 + 1] = u.y;
                    w[4 * v4 + 2] = u.z;
                    w[4 * v4 + 3] = u.w;
                }
                tmem_st16(tQ + 16 * c, w);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->q_ready));
        }
        for (int i = 0; i < steps; ++i) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->s_full), (uint32_t)i & 1u, tmo, abort_flag))) {
                dec_abort(ctl, W_EPILOGUE);
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[kDecChunk];
            tmem_ld32(tS, &sv[0]);
            tmem_ld32(tS + 32, &sv[32]);
            tmem_wait_ld();
            const int64_t k0 = (c_begin + i) * kDecChunk;
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kDecChunk; ++c) {
                if (k0 + c >= n) sv[c] = __float_as_uint(-INFINITY);
                mx = fmaxf(mx, __uint_as_float(sv[c]));
            }
            const float m_new = fmaxf(m_run, mx * sl2);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = m_run == -INFINITY ? 0.f : fast_exp2(m_run - m_use);
            if (i > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
                // O holds P_{i-1} V_{i-1} (the MMA that wrote S_i ran after it): rescale it in place
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    uint32_t o[16];
                    tmem_ld16(tO + 16 * c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 16; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
                    tmem_st16(tO + 16 * c, o);
                }
            }
            float sum = 0.f;
            uint32_t pk[kDecChunk / 2];
#pragma unroll
            for (int c = 0; c < kDecChunk / 2; ++c) {
                const float p0 = fast_exp2(fmaf(__uint_as_float(sv[2 * c]), sl2, -m_use));
                const float p1 = fast_exp2(fmaf(__uint_as_float(sv[2 * c + 1]), sl2, -m_use));
                sum += p0 + p1;
                pk[c] = pack_bf16x2(p0, p1);
            }
            l_run = l_run * alpha + sum;
            m_run = m_new;
            tmem_st16(tS, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
            tmem_st16(tS + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full));
        }
        const int64_t part = ((int64_t)b * a.Hq + kvh * G + row) * a.splits + split;
        if (ok && steps > 0 &&
            __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->o_full), 0, tmo, abort_flag))) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t o[16];
                tmem_ld16(tO + 16 * c, o);
                tmem_wait_ld();
                if (row < G) {
                    float4* dst = reinterpret_cast<float4*>(a.part_o + part * kAttnHD + 16 * c);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                             __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3]));
                }
            }
        } else if (ok && steps > 0) {
            dec_abort(ctl, W_EPILOGUE);
        } else if (steps == 0 && row < G) {
            // no keys for this split: an empty partial
            for (int c = 0; c < kAttnHD; c += 4)
                *reinterpret_cast<float4*>(a.part_o + part * kAttnHD + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (row < G) {
            a.part_ml[2 * part] = m_run;
            a.part_ml[2 * part + 1] = l_run;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(ctl->tmem_base, 256);
}

// out[b][h] = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c over the splits c
// in order (empty ones carry m = -inf, l = 0), bf16. Block (h, b), one thread per
// channel. The block of head 0 then advances the sequence's cache length
// (nothing later in the step reads it).
__global__ void __launch_bounds__(kAttnHD) attention_decode_merge_kernel(const float* __restrict__ part_o,
                                                                         const float* __restrict__ part_ml, int Hq,
                                                                         int chunks, int32_t* len, int64_t cache_max,
                                                                         __nv_bfloat16* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    const int h = blockIdx.x, b = blockIdx.y, e = threadIdx.x;
    const int64_t hb = (int64_t)b * Hq + h;
    const float* ml = part_ml + hb * chunks * 2;
    const float* po = part_o + hb * chunks * kAttnHD + e;
    float M = -INFINITY;
#pragma unroll 8
    for (int c = 0; c < chunks; ++c) M = fmaxf(M, ml[2 * c]);
    float L = 0.f, O = 0.f;
#pragma unroll 8
    for (int c = 0; c < chunks; ++c) {
        const float m = ml[2 * c];
        const float w = m == -INFINITY ? 0.f : fast_exp2(m - M);
        L = fmaf(w, ml[2 * c + 1], L);
        O = fmaf(w, po[(int64_t)c * kAttnHD], O);
    }
    out[hb * kAttnHD + e] = __float2bfloat16_rn(O / L);
    __syncthreads();
    if (h == 0 && e == 0 && len[b] < cache_max) len[b] += 1;
}

}  // namespace moe
