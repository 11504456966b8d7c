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
// n = len + 1 valid keys (the new token's were appended by the RoPE step), 128
// keys per step, for the G <= 16 query heads that share the KV head. The keys
// sit on the MMA's 128-row side and the G heads on its N = 16 side, so the
// softmax runs one key per thread and computes only G exponentials per key:
//   S^T = K Q^T     tcgen05.mma M = 128 keys, N = 16 (heads G .. 15 are zero
//                   rows of Q), K = 128 channels; K by TMA (128-byte swizzle,
//                   K-major), Q K-major in shared memory; S^T in tensor
//                   memory, two buffers, so the scores of step i + 1 are
//                   computed while the softmax of step i runs
//   softmax         warps 0-3, thread t = key t of the step: each head's
//                   maximum over the 128 keys (warp butterflies, then the four
//                   warps' values through shared memory behind a bounded
//                   mbarrier wait), p = 2^(s - m), a per-thread partial sum
//                   rescaled with the running maximum; P^T (bf16, heads x
//                   keys, K-major) into shared memory, two buffers
//   O^T += V^T P^T  M = 128 channels, N = 16 heads, K = 128 keys: V read as
//                   stored ([key][channel] is the MN-major A), O^T in tensor
//                   memory (16 columns), rescaled in place when a maximum grows
// Keys and values stream through three 64 KB stages. Key rows past the valid
// ones in the last step are masked (score -inf) and their value rows are
// zeroed in shared memory before P V, so whatever the cache holds past its
// length cannot reach the result. Each CTA writes one unnormalised partial
// (O, m, l) per head; a second kernel merges the splits in order (flash
// decoding).
// ---------------------------------------------------------------------------
constexpr int kDecChunk = 128;                       // keys per step
constexpr int kDecN = 16;                            // MMA N: the group's query heads, zero-padded
constexpr int kDecThreads = 192;                     // warps 0-3 softmax, warp 4 TMA, warp 5 MMA
constexpr int kDecMaxGroup = kDecN;                  // query heads per KV head
constexpr int kDecCtasPerSm = 1;
constexpr int kDecStages = 3;
constexpr uint32_t kDecBox = 128 * 64 * 2;           // 16 KB: 128 keys x 64 channels
constexpr uint32_t kDecStageBytes = 4 * kDecBox;     // keys (two boxes) + values (two boxes)
constexpr uint32_t kDecQBytes = 2 * kDecN * 128;     // Q: two 64-channel blocks of 16 rows x 128 bytes
constexpr uint32_t kDecPBytes = 2 * kDecN * 128;     // one P^T buffer: two 64-key blocks of 16 rows

struct DecControl {
    uint64_t q_ready;
    uint64_t kv_full[kDecStages];
    uint64_t kv_empty[kDecStages];
    uint64_t s_full[2], p_full[2], red_full[2], o_ready[2];
    uint64_t o_full, fin_full, drain;
    float red[2][4][kDecN];                          // per step parity, per softmax warp, per head
    float fin[4][kDecN];
    uint32_t tmem_base;
    int abort_flag;
};

// stages | Q | P^T x 2 | control
constexpr size_t kDecSmemBytes =
    1024 + (size_t)kDecStages * kDecStageBytes + kDecQBytes + 2 * (size_t)kDecPBytes + sizeof(DecControl);
static_assert(kDecSmemBytes <= 227 * 1024, "decode attention CTA exceeds the shared memory of a CTA");

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

// Bounded wait on an mbarrier by a whole warp; true when every lane saw the phase complete.
__device__ __forceinline__ bool dec_wait_warp(uint32_t bar, uint32_t parity, uint64_t tmo, volatile int* abort_flag) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, tmo, abort_flag));
}

// map_k, map_v: the caches viewed as [B Hkv cache_max][128], boxes of 64
// channels x 128 keys. GP: the group size rounded up to a power of two
// (1 .. 16); the softmax's per-head loops run GP times, heads G .. GP-1 are
// zero rows of Q whose results are dropped.
template <int GP>
__global__ void __launch_bounds__(kDecThreads, 1)
    attention_decode_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                            const DecodeArgs a) {
    extern __shared__ unsigned char dec_smem_raw[];
    unsigned char* smem = align1024(dec_smem_raw);
    DecControl* ctl = reinterpret_cast<DecControl*>(smem + (size_t)kDecStages * kDecStageBytes + kDecQBytes +
                                                    2 * (size_t)kDecPBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t tmo = a.timeout_ns;
    volatile int* abort_flag = &ctl->abort_flag;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int G = a.Hq / a.Hkv;
    const uint32_t sbase = smem_u32(smem);
    auto sK = [&](int st) { return sbase + (uint32_t)st * kDecStageBytes; };
    auto sV = [&](int st) { return sK(st) + 2 * kDecBox; };
    const uint32_t sQ = sbase + kDecStages * kDecStageBytes;
    auto sP = [&](int buf) { return sQ + kDecQBytes + (uint32_t)buf * kDecPBytes; };

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&ctl->q_ready), 4);
        for (int s = 0; s < kDecStages; ++s) {
            mbar_init(smem_u32(&ctl->kv_full[s]), 1);
            mbar_init(smem_u32(&ctl->kv_empty[s]), 1);
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(smem_u32(&ctl->s_full[p]), 1);
            mbar_init(smem_u32(&ctl->p_full[p]), 4);
            mbar_init(smem_u32(&ctl->red_full[p]), 4);
            mbar_init(smem_u32(&ctl->o_ready[p]), 1);
        }
        mbar_init(smem_u32(&ctl->o_full), 1);
        mbar_init(smem_u32(&ctl->fin_full), 4);
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&ctl->tmem_base), 64);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
    }
    pdl_trigger();
    pdl_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = ctl->tmem_base;          // columns 0-15 and 16-31: S^T of even and odd steps
    const uint32_t tO = ctl->tmem_base + 32;     // columns 32-47: O^T

    const int64_t n_all = (int64_t)a.len[b] + 1;
    const int64_t n = n_all < a.cache_max ? n_all : a.cache_max;
    const int64_t nch = (n + kDecChunk - 1) / kDecChunk;
    const int64_t per = (nch + a.splits - 1) / a.splits;
    const int64_t c_begin = split * per;
    const int64_t c_end = c_begin + per < nch ? c_begin + per : nch;
    const int steps = c_end > c_begin ? (int)(c_end - c_begin) : 0;
    const int64_t row0 = ((int64_t)b * a.Hkv + kvh) * a.cache_max;

    if (warp == 4) {
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
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA
        if (lane == 0 && steps > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, kDecN);
            constexpr uint32_t idesc_o = idesc_bf16_f32(128, kDecN, true, false);
            bool ok = mbar_wait(smem_u32(&ctl->q_ready), 0, tmo, abort_flag);
            if (!ok) dec_abort(ctl, W_MMA);
            bool any = false;
            // O^T += V^T P^T of step j, once the softmax has written P^T_j
            auto pv = [&](int j) -> bool {
                if (!mbar_wait(smem_u32(&ctl->p_full[j & 1]), (uint32_t)(j >> 1) & 1u, tmo, abort_flag)) return false;
                tc_fence_after();
                const int st = j % kDecStages;
#pragma unroll
                for (int kk = 0; kk < kDecChunk / 16; ++kk) {
                    const uint64_t ad = sw128_mnmajor_desc(sV(st), kDecBox) + 128ull * kk;
                    const uint64_t bd = sw128_kmajor_desc(sP(j & 1) + (uint32_t)(kk >> 2) * (kDecN * 128)) +
                                        2ull * (kk & 3);
                    mma_bf16(tO, ad, bd, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(smem_u32(&ctl->kv_empty[st]));
                mma_commit(smem_u32(&ctl->o_ready[j & 1]));
                return true;
            };
            for (int i = 0; ok && i < steps; ++i) {
                const int st = i % kDecStages;
                if (!mbar_wait(smem_u32(&ctl->kv_full[st]), (uint32_t)(i / kDecStages) & 1u, tmo, abort_flag)) {
                    dec_abort(ctl, W_MMA);
                    ok = false;
                    break;
                }
                tc_fence_after();
                // S^T_i = K_i Q^T into buffer i & 1 (its scores of step i - 2 were read before P^T_{i-2},
                // whose P V was issued before this)
#pragma unroll
                for (int kk = 0; kk < kAttnHD / 16; ++kk) {
                    const uint32_t blk = (uint32_t)(kk >> 2);
                    const uint64_t ad = sw128_kmajor_desc(sK(st) + blk * kDecBox) + 2ull * (kk & 3);
                    const uint64_t bd = sw128_kmajor_desc(sQ + blk * (kDecN * 128)) + 2ull * (kk & 3);
                    mma_bf16(tS + kDecN * (uint32_t)(i & 1), ad, bd, idesc_s, kk > 0);
                }
                any = true;
                mma_commit(smem_u32(&ctl->s_full[i & 1]));
                if (i > 0 && !pv(i - 1)) {
                    dec_abort(ctl, W_MMA);
                    ok = false;
                    break;
                }
            }
            if (ok) {
                if (pv(steps - 1)) {
                    mma_commit(smem_u32(&ctl->o_full));
                } else {
                    dec_abort(ctl, W_MMA);
                }
            }
            if (any) {
                mma_commit(smem_u32(&ctl->drain));
                drain_wait(smem_u32(&ctl->drain), 0, tmo, K_ATTN);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + partial (warps 0-3: t = key / channel)
        const int t = threadIdx.x;                               // 0 .. 127
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;   // this warp's tensor-memory lane quarter
        const float sl2 = a.scale_log2;
        float m_run[GP], l_part[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            m_run[h] = -INFINITY;
            l_part[h] = 0.f;
        }
        bool ok = true;
        if (steps > 0) {
            // Q (the group's heads, zero rows past G) and both P^T buffers (rows past G stay zero) into
            // shared memory, K-major in the 128-byte swizzle: thread t writes row t / 8, 16-byte chunk t % 8
            // of both 64-channel blocks, and zeroes the same chunks of both P^T buffers
            const int hq = t >> 3, c = t & 7;
            const uint32_t off = (uint32_t)hq * 128u + ((uint32_t)(c ^ (hq & 7)) << 4);
            const uint4* qr = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * a.Hq + kvh * G + hq) * kAttnHD);
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                const uint4 u = hq < G ? qr[blk * 8 + c] : make_uint4(0u, 0u, 0u, 0u);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sQ + blk * (kDecN * 128) + off),
                             "r"(u.x), "r"(u.y), "r"(u.z), "r"(u.w)
                             : "memory");
#pragma unroll
                for (int pb = 0; pb < 2; ++pb)
                    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(sP(pb) + blk * (kDecN * 128) + off),
                                 "r"(0u)
                                 : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->q_ready));
        }
        for (int i = 0; i < steps; ++i) {
            const int par = i & 1;
            if (!dec_wait_warp(smem_u32(&ctl->s_full[par]), (uint32_t)(i >> 1) & 1u, tmo, abort_flag)) {
                dec_abort(ctl, W_EPILOGUE);
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[kDecN];
            tmem_ld16(tS + kDecN * (uint32_t)par + lane_off, sv);
            tmem_wait_ld();
            const int64_t key = (c_begin + i) * kDecChunk + t;
            const bool valid = key < n;
            float sc[GP], wmax[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                sc[h] = valid ? __uint_as_float(sv[h]) * sl2 : -INFINITY;
                wmax[h] = sc[h];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int h = 0; h < GP; ++h) wmax[h] = fmaxf(wmax[h], __shfl_xor_sync(0xffffffffu, wmax[h], o));
            if (lane == 0) {
#pragma unroll
                for (int h = 0; h < GP; ++h) ctl->red[par][warp][h] = wmax[h];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->red_full[par]));
            if (!dec_wait_warp(smem_u32(&ctl->red_full[par]), (uint32_t)(i >> 1) & 1u, tmo, abort_flag)) {
                dec_abort(ctl, W_EPILOGUE);
                ok = false;
                break;
            }
            if (i >= 2) {
                // P V of step i - 2 has finished reading this P^T buffer
                if (!dec_wait_warp(smem_u32(&ctl->o_ready[par]), (uint32_t)((i - 2) >> 1) & 1u, tmo, abort_flag)) {
                    dec_abort(ctl, W_EPILOGUE);
                    ok = false;
                    break;
                }
            }
            float alpha[GP];
            bool grow = false;
            // P^T[h][t]: block t / 64, row h, 16-byte chunk (t % 64) / 8 swizzled by h % 8
            const uint32_t prow = sP(par) + (uint32_t)(t >> 6) * (kDecN * 128) + (uint32_t)(t & 7) * 2u;
            const uint32_t pchunk = (uint32_t)((t & 63) >> 3);
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                const float mc = fmax3f(fmaxf(ctl->red[par][0][h], ctl->red[par][1][h]), ctl->red[par][2][h],
                                        ctl->red[par][3][h]);
                const float m_new = fmaxf(m_run[h], mc);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                alpha[h] = m_run[h] == -INFINITY ? 0.f : fast_exp2(m_run[h] - m_use);
                grow |= alpha[h] < 1.f;
                const float p = fast_exp2(sc[h] - m_use);
                l_part[h] = fmaf(l_part[h], alpha[h], p);
                m_run[h] = m_new;
                const uint32_t addr = prow + (uint32_t)h * 128u + ((pchunk ^ (uint32_t)(h & 7)) << 4);
                const __nv_bfloat16 pb = __float2bfloat16_rn(p);
                asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(*reinterpret_cast<const uint16_t*>(&pb))
                             : "memory");
            }
            if (!valid) {
                // the value row of a key past the valid ones is zeroed, so it cannot reach O
                const uint32_t vrow = sV((int)(i % kDecStages)) + (uint32_t)t * 128u;
#pragma unroll
                for (int blk = 0; blk < 2; ++blk)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(vrow + blk * kDecBox + q * 16u),
                                     "r"(0u)
                                     : "memory");
            }
            if (i > 0 && grow) {
                // a maximum grew: once P V of the previous step has finished with O, rescale O in place
                // (with no growth O needs no change, and P V of this step may follow the previous one at once)
                if (!dec_wait_warp(smem_u32(&ctl->o_ready[par ^ 1]), (uint32_t)((i - 1) >> 1) & 1u, tmo,
                                   abort_flag)) {
                    dec_abort(ctl, W_EPILOGUE);
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    uint32_t o[kDecN];
                    tmem_ld16(tO + lane_off, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < GP; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
                    tmem_st16(tO + lane_off, o);
                    tmem_wait_st();
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full[par]));
        }
        // each head's sum over the keys: the threads' partial sums, warp by warp, then the four warps
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int h = 0; h < GP; ++h) l_part[h] += __shfl_xor_sync(0xffffffffu, l_part[h], o);
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < GP; ++h) ctl->fin[warp][h] = l_part[h];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->fin_full));
        const bool fin_ok = dec_wait_warp(smem_u32(&ctl->fin_full), 0, tmo, abort_flag);
        const int64_t part0 = ((int64_t)b * a.Hq + kvh * G) * a.splits + split;
        if (ok && fin_ok && steps > 0 && dec_wait_warp(smem_u32(&ctl->o_full), 0, tmo, abort_flag)) {
            tc_fence_after();
            uint32_t o[kDecN];
            tmem_ld16(tO + lane_off, o);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < GP; ++h)
                if (h < G) a.part_o[(part0 + (int64_t)h * a.splits) * kAttnHD + t] = __uint_as_float(o[h]);
        } else if (steps > 0) {
            dec_abort(ctl, W_EPILOGUE);
        } else {
            // no keys for this split: an empty partial
#pragma unroll
            for (int h = 0; h < GP; ++h)
                if (h < G) a.part_o[(part0 + (int64_t)h * a.splits) * kAttnHD + t] = 0.f;
        }
        if (t < G) {
            const float l = fin_ok ? ctl->fin[0][t] + ctl->fin[1][t] + ctl->fin[2][t] + ctl->fin[3][t] : 0.f;
            float m = -INFINITY;
#pragma unroll
            for (int h = 0; h < GP; ++h)
                if (h == t) m = m_run[h];
            a.part_ml[2 * (part0 + (int64_t)t * a.splits)] = m;
            a.part_ml[2 * (part0 + (int64_t)t * a.splits) + 1] = l;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(ctl->tmem_base, 64);
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
