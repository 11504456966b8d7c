// Causal grouped-query attention on the 5th-generation tensor cores.
//
// The block's attention is LLaMA's ("Mixtral" lineage page, step "GPT-2 vs
// Mixtral": RMSNorm, RoPE, grouped-query attention); the Mixtral notes
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

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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

}  // namespace moe
