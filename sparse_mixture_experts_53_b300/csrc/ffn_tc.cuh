// Expert FFNs on the 5th-generation tensor cores (tcgen05.mma kind::f16,
// bf16 operands, fp32 accumulators in tensor memory), operands staged by TMA
// into 128-byte-swizzled shared memory.
//
// Each expert is a SwiGLU block, E(x) = W2 (SiLU(W1 x) * W3 x)
// (tokentrails.org "Mixtral", Code; fdeinterviews.com breakdown "The paper in
// one minute"). Rows are in expert-contiguous order, so expert e owns rows
// [offsets[e], offsets[e+1]); experts with no rows produce no work and none of
// their weights are read (lecture, router walkthrough: unused experts are not
// touched).
//
// Two kernel families, both persistent (one CTA per SM) and warp-specialised:
// warp 0 issues TMA loads, warp 1 issues MMAs, warps 2-5 run the epilogue
// (warp w reads tensor-memory lanes 32*(w%4) .. 32*(w%4)+31).
//
//  * token-tile kernels (many tokens per expert): a tile is 128 rows of one
//    expert x 256 output columns, K stepped by 64.
//      up:   columns are 128 rows of W1 followed by the same 128 rows of W3, so
//            one N=256 MMA yields u and v side by side and the epilogue writes
//            h = SiLU(u) * v in bf16;
//      down: columns are 256 rows of W2; the epilogue writes perm_w[r] * acc.
//    Tiles run expert-major, then column tile, then row tile, so the CTAs
//    running at one time share weight tiles and activations through L2.
//
//  * weight-streaming kernels (few tokens per expert): the MMA's M side is 128
//    weight rows and its N side is the expert's tokens (<= 64), so all SMs
//    stream weights at full width. The reduction dimension is split into
//    slices so that the units of work outnumber the SMs; each unit writes an
//    fp32 partial, and a separate pass sums the partials in a fixed order.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kTcThreads = 192;
constexpr int kBK = 64;          // K elements per stage (128 bytes of bf16)
constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kTileStages = 4;
constexpr uint32_t kTileABytes = kTileM * kBK * 2;   // 16 KB
constexpr uint32_t kTileBBytes = kTileN * kBK * 2;   // 32 KB
constexpr uint32_t kTileStageBytes = kTileABytes + kTileBBytes;
constexpr int kTileAccCols = 256;
constexpr int kMaxStreamStages = 12;
constexpr int kStreamAcc = 4;
constexpr int kStreamMaxNB = 64;
constexpr uint32_t kStreamABytes = 128 * kBK * 2;     // 16 KB of weights per stage

constexpr int kUnitRing = 8;

struct TcControl {
    uint64_t full[kMaxStreamStages];
    uint64_t empty[kMaxStreamStages];
    uint64_t tfull[kStreamAcc];
    uint64_t tempty[kStreamAcc];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int n_work;
    int n_act;
    int off[kMaxExperts + 1];
    int cnt[kMaxExperts];
    int mt[kMaxExperts];
    int base[kMaxExperts + 1];
    int act[kMaxExperts];
    int koff[kMaxExperts + 1];  // expert groups padded to multiples of 64 rows
    int half_ok;                // pair kernel, forward modes: last tiles of <= 128 rows run as half tiles
    // pair kernel with a shared unit counter: the even CTA's producer claims each unit and passes it
    // to every other role of both CTAs through this ring
    uint64_t ring_full[kUnitRing];   // the slot holds a claimed unit (-1: no more)
    uint64_t ring_empty[kUnitRing];  // (even CTA) every reader of both CTAs has taken the slot
    int ring_unit[kUnitRing];
};

constexpr size_t kTileSmemBytes = 1024 + (size_t)kTileStages * kTileStageBytes + sizeof(TcControl);

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
    return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Waits for the last issued phase of a barrier without looking at the abort
// flag: used on the way out to let in-flight copies and MMAs land.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                           int kernel) {
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > timeout_ns) {
            report_error(MOE_ERR_TIMEOUT, kernel, W_DRAIN);
            return;
        }
    }
}

__device__ __forceinline__ void raise_abort(TcControl* c, int kernel, int where) {
    report_error(MOE_ERR_TIMEOUT, kernel, where);
    *reinterpret_cast<volatile int*>(&c->abort_flag) = 1;
}

struct TileArgs {
    const int32_t* offsets;  // [E+1]
    const float* perm_w;     // [R] (down only; nullptr = no scale)
    void* out;               // up: H bf16 [R][ldo]; down: y_slot fp32 [R][ldo]; see the backward modes
    int E;
    int K;          // reduction length (d for up, ffn for down)
    int n_tiles_n;  // column tiles per expert
    int w_rows;     // rows of one expert in the weight maps (ffn for up, d for down)
    int ldo;        // output row stride in elements
    uint64_t timeout_ns;
    // training forward (up): also keep u = W1 x and v = W3 x in bf16 [R][ldo] (nullable)
    __nv_bfloat16* u_out;
    __nv_bfloat16* v_out;
    // backward of the SwiGLU (pair kernel, PM_BWD_DH): the kept u and v
    const __nv_bfloat16* u_in;
    const __nv_bfloat16* v_in;
    // weight gradients (pair kernel, PM_WGRAD): rows >= split_rows go to out2
    float* out2;
    int m_tiles;           // 256-row tiles of the gradient per expert
    int split_rows;        // rows of the first gradient matrix
    int64_t out_estride;   // elements per expert in each gradient matrix
    // plain linear layer (pair kernel, PM_DOWN with offsets == nullptr): one group of this many rows
    int dense_rows;
    // pair kernel: order of an expert's tiles. 0 = row tiles fastest: the tiles running at one time share
    // a block of B, and all of the expert's A stays in L2 across B's blocks (right when A is the smaller
    // operand); 1 = column tiles fastest: they share a block of A and all of B stays in L2 (right when B
    // is the smaller one). The order does not change any tile's arithmetic.
    int n_fast;
    // down projection with the combine (pair kernel, PM_DOWN, y non-null): a slot whose token's other slot
    // lies in a lower-numbered expert adds that slot's y_slot row to its own and writes the token's row of
    // y (bf16); every other slot writes y_slot. done[unit] (zero at launch) counts the epilogue warps that
    // have finished the unit's stores.
    const int32_t* perm_token;
    const int32_t* slot_row;
    __nv_bfloat16* y;
    int* done;
    // pair kernel (up projection): zero these counts once its predecessors are done (the down
    // projection that follows reads them only after this kernel has completed)
    int* zero_counts;
    int n_zero_counts;
    // pair kernel: nullptr = pair p takes units p, p + pairs, ...; otherwise a counter, zero at launch,
    // from which the pairs claim units in order as they become free (any pair may compute any unit: the
    // results do not depend on the assignment)
    int* sched;
};

// Epilogue of one token tile for one thread (one row): reads the row's
// accumulator columns from tensor memory and writes
//   up:   h = SiLU(u) * v in bf16 (u in columns j, v in columns v_off + j),
//   down: perm_w[r] * acc in fp32.
// Every thread of the warp must call it (tcgen05.ld is warp-collective);
// `valid` only predicates the stores.
// [j_begin, j_end): the columns this thread handles (up: of the u, v pairs;
// down: of the accumulator columns), multiples of 16; col0: the output column
// of j = 0 (up: in H, down: in y_slot).
template <bool UP>
__device__ __forceinline__ void tile_epilogue(uint32_t taddr, bool valid, int64_t r, int nt, const TileArgs& args,
                                              int j_begin = 0, int j_end = UP ? kTileM : kTileN,
                                              int v_off = kTileM, int col0 = -1) {
    if (col0 < 0) col0 = nt * (UP ? kTileM : kTileN);
    if (UP) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out) + r * args.ldo + col0;
#pragma unroll 1
        for (int j = j_begin; j < j_end; j += 16) {
            uint32_t u[16], v[16];
            tmem_ld16(taddr + j, u);
            tmem_ld16(taddr + v_off + j, v);
            tmem_wait_ld();
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float h0 = silu_f32(__uint_as_float(u[2 * i])) * __uint_as_float(v[2 * i]);
                const float h1 = silu_f32(__uint_as_float(u[2 * i + 1])) * __uint_as_float(v[2 * i + 1]);
                pk[i] = pack_bf16x2(h0, h1);
            }
            if (valid) {
                uint4* dst = reinterpret_cast<uint4*>(out + j);
                dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                if (args.u_out != nullptr) {
                    // training forward: keep u and v (bf16) for the backward pass
                    const int64_t at = r * args.ldo + col0 + j;
#pragma unroll
                    for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
                    uint4* du = reinterpret_cast<uint4*>(args.u_out + at);
                    du[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    du[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    uint4* dv = reinterpret_cast<uint4*>(args.v_out + at);
                    dv[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dv[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
            }
        }
    } else {
        const float pw = valid ? (args.perm_w != nullptr ? args.perm_w[r] : 1.0f) : 0.f;
        float* out = reinterpret_cast<float*>(args.out) + r * args.ldo + col0;
#pragma unroll 1
        for (int j = j_begin; j < j_end; j += 16) {
            uint32_t a[16];
            tmem_ld16(taddr + j, a);
            tmem_wait_ld();
            if (valid) {
                float4* dst = reinterpret_cast<float4*>(out + j);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_float4(pw * __uint_as_float(a[4 * i]), pw * __uint_as_float(a[4 * i + 1]),
                                         pw * __uint_as_float(a[4 * i + 2]), pw * __uint_as_float(a[4 * i + 3]));
            }
        }
    }
}

// Down-projection epilogue with the combine fused in, for one thread (one slot row r); every thread of
// the warp calls it with the same columns (tcgen05.ld is warp-collective: the per-thread choice below
// only selects which stores it makes). A slot that finishes its token (`finish`) adds the same columns
// of the token's other slot (row pr of y_slot, already written; pr < 0: no other slot) to its own value
// (the accumulator scaled by its gate weight, rounded once as in y_slot), sums in fp32 and rounds once
// to bf16 into row t of y; any other slot writes its y_slot row as tile_epilogue<false> does. Two fp32
// operands add the same in either order, so y equals the separate combine pass bit for bit.
__device__ __forceinline__ void down_combine_epilogue(uint32_t taddr, bool valid, bool finish, int64_t r, int64_t pr,
                                                      int64_t t, const TileArgs& args, int j_begin, int j_end,
                                                      int col0) {
    const float pw = valid ? (args.perm_w != nullptr ? args.perm_w[r] : 1.0f) : 0.f;
    float* ys = reinterpret_cast<float*>(args.out) + r * args.ldo + col0;
    const float* other = reinterpret_cast<const float*>(args.out) + (pr >= 0 ? pr : 0) * args.ldo + col0;
    __nv_bfloat16* yo = args.y + t * args.ldo + col0;
    const bool read_other = valid && finish && pr >= 0;
#pragma unroll 1
    for (int j = j_begin; j < j_end; j += 16) {
        float4 o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = read_other ? reinterpret_cast<const float4*>(other + j)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        uint32_t a[16];
        __syncwarp();
        tmem_ld16(taddr + j, a);
        tmem_wait_ld();
        float v[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) v[c] = __fmul_rn(pw, __uint_as_float(a[c]));
        if (valid && finish) {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                pk[2 * i] = pack_bf16x2(__fadd_rn(v[4 * i], o[i].x), __fadd_rn(v[4 * i + 1], o[i].y));
                pk[2 * i + 1] = pack_bf16x2(__fadd_rn(v[4 * i + 2], o[i].z), __fadd_rn(v[4 * i + 3], o[i].w));
            }
            uint4* dst = reinterpret_cast<uint4*>(yo + j);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        } else if (valid) {
            float4* dst = reinterpret_cast<float4*>(ys + j);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
    }
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.global.acquire.gpu.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// UP = true: SwiGLU up-projection; UP = false: W2 down-projection + gate scale.
template <bool UP>
__global__ void __launch_bounds__(kTcThreads, 1)
    tile_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                     const __grid_constant__ CUtensorMap map_b1, const TileArgs args) {
    extern __shared__ unsigned char tc_smem_raw[];
    unsigned char* smem = align1024(tc_smem_raw);
    TcControl* ctl = reinterpret_cast<TcControl*>(smem + (size_t)kTileStages * kTileStageBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int kid = UP ? K_TILE_UP : K_TILE_DOWN;
    const uint64_t tmo = args.timeout_ns;
    volatile int* abort_flag = &ctl->abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTileStages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
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
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b0);
        if (UP) tma_prefetch_desc(&map_b1);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), 2 * kTileAccCols);
        tmem_relinquish();
    }
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x == 0) {
        int tiles = 0;
        if (args.offsets != nullptr) {
            for (int e = 0; e <= args.E; ++e) ctl->off[e] = args.offsets[e];
        } else {
            ctl->off[0] = 0;
            ctl->off[1] = args.dense_rows;
        }
        for (int e = 0; e < args.E; ++e) {
            const int c = ctl->off[e + 1] - ctl->off[e];
            ctl->cnt[e] = c;
            ctl->mt[e] = (c + kTileM - 1) / kTileM;
            ctl->base[e] = tiles;
            tiles += ctl->mt[e] * args.n_tiles_n;
        }
        ctl->base[args.E] = tiles;
        ctl->n_work = tiles;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int n_work = ctl->n_work;
    const int E = args.E;
    const int KB = args.K / kBK;

    auto decode = [&](int tile, int& e, int& nt, int& mt) {
        e = 0;
        while (e < E - 1 && tile >= ctl->base[e + 1]) ++e;
        const int rem = tile - ctl->base[e];
        nt = rem / ctl->mt[e];
        mt = rem - nt * ctl->mt[e];
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            // activations are re-read for every column tile: keep them; a
            // weight tile is shared by the CTAs working on the expert's row
            // tiles at the same time: normal priority
            const uint64_t pol_act = policy_evict_last();
            const uint64_t pol_w = policy_evict_normal();
            uint32_t s = 0, ph = 0;
            uint32_t issued_mask = 0, issued_ph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < n_work; tile += gridDim.x) {
                int e, nt, mt;
                decode(tile, e, nt, mt);
                const int arow = ctl->off[e] + mt * kTileM;
                const int brow = e * args.w_rows + nt * (UP ? kTileM : kTileN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1, tmo, abort_flag)) {
                        raise_abort(ctl, kid, W_PRODUCER);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&ctl->full[s]);
                    const uint32_t sa = smem_u32(smem + (size_t)s * kTileStageBytes);
                    const uint32_t sb = sa + kTileABytes;
                    mbar_arrive_expect_tx(fb, kTileStageBytes);
                    tma_load_2d(sa, &map_a, fb, kb * kBK, arow, pol_act);
                    if (UP) {
                        tma_load_2d(sb, &map_b0, fb, kb * kBK, brow, pol_w);
                        tma_load_2d(sb + kTileBBytes / 2, &map_b1, fb, kb * kBK, brow, pol_w);
                    } else {
                        tma_load_2d(sb, &map_b0, fb, kb * kBK, brow, pol_w);
                    }
                    issued_mask |= 1u << s;
                    issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                    if (++s == kTileStages) { s = 0; ph ^= 1; }
                }
            }
            if (!ok) {
                for (int q = 0; q < kTileStages; ++q)
                    if (issued_mask & (1u << q))
                        drain_wait(smem_u32(&ctl->full[q]), (issued_ph >> q) & 1u, tmo, kid);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kTileM, kTileN);
            uint32_t s = 0, ph = 0;
            bool ok = true, any = false;
            int it = 0;
            for (int tile = blockIdx.x; ok && tile < n_work; tile += gridDim.x, ++it) {
                const int b = it & 1;
                const uint32_t aph = (it >> 1) & 1;
                if (!mbar_wait(smem_u32(&ctl->tempty[b]), aph ^ 1, tmo, abort_flag)) {
                    raise_abort(ctl, kid, W_MMA);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * kTileAccCols;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(smem_u32(&ctl->full[s]), ph, tmo, abort_flag)) {
                        raise_abort(ctl, kid, W_MMA);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)s * kTileStageBytes);
                    const uint64_t adesc = sw128_kmajor_desc(sa);
                    const uint64_t bdesc = sw128_kmajor_desc(sa + kTileABytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
                    any = true;
                    mma_commit(smem_u32(&ctl->empty[s]));
                    if (++s == kTileStages) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                mma_commit(smem_u32(&ctl->tfull[b]));
            }
            if (any) {
                mma_commit(smem_u32(&ctl->drain));
                drain_wait(smem_u32(&ctl->drain), 0, tmo, kid);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2-5)
        const int sub = warp & 3;
        const int row_in_tile = sub * 32 + lane;
        int it = 0;
        for (int tile = blockIdx.x; tile < n_work; tile += gridDim.x, ++it) {
            int e, nt, mt;
            decode(tile, e, nt, mt);
            const int b = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            if (!mbar_wait(smem_u32(&ctl->tfull[b]), aph, tmo, abort_flag)) {
                raise_abort(ctl, kid, W_EPILOGUE);
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + b * kTileAccCols + ((uint32_t)(sub * 32) << 16);
            const int grow = mt * kTileM + row_in_tile;
            const bool valid = grow < ctl->cnt[e];
            const int64_t r = ctl->off[e] + grow;
            tile_epilogue<UP>(taddr, valid, r, nt, args);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[b]));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 2 * kTileAccCols);
}

// ---------------------------------------------------------------------------
// token tiles on CTA pairs: one tcgen05.mma.cta_group::2 spans the tensor cores
// of two SMs. The pair owns a 256-token x 256-column tile: each CTA stages 128
// token rows of A and 128 rows of B (up: CTA 0 the W1 rows, CTA 1 the W3 rows;
// down: the two halves of the 256 W2 rows) and holds the accumulator of its
// own 128 token rows. Per FLOP, each SM reads two thirds of the operand bytes
// of the single-CTA tile (L2 -> shared memory and shared memory -> tensor
// core). The even CTA (rank 0) issues the MMAs; the TMA loads of both CTAs
// count on its `full` barrier, its commits arrive on `empty`/`tfull` of both
// CTAs, and the epilogues of both CTAs arrive on its `tempty`.
// ---------------------------------------------------------------------------
constexpr int kPairM = 256;
constexpr int kPairStages = 6;
// CTA-pair kernels: warp 0 TMA, warp 1 MMA, warps 2-9 the epilogue (two warps
// per tensor-memory lane quarter, each taking half of the tile's columns)
constexpr int kPairThreads = 320;
constexpr int kPairEpiWarps = 8;
constexpr uint32_t kPairHalfBytes = 128 * kBK * 2;          // 16 KB: one CTA's half of A or of B
constexpr uint32_t kPairStageBytes = 2 * kPairHalfBytes;     // 32 KB per CTA and stage
// readers of a unit-ring slot: the MMA issuer, the odd CTA's producer and the epilogue warps of both CTAs
constexpr int kRingReaders = 2 + 2 * kPairEpiWarps;
constexpr size_t kPairSmemBytes = 1024 + (size_t)kPairStages * kPairStageBytes + sizeof(TcControl);
// the weight-gradient epilogue's staging arrays, one per epilogue warp, after the control block
constexpr size_t kWgradStageBytes = 16 + (size_t)kPairEpiWarps * 32 * 33 * sizeof(float);
static_assert(kPairSmemBytes + kWgradStageBytes <= 227 * 1024, "CTA-pair kernel exceeds the shared memory of a CTA");

// What a CTA-pair tile kernel computes (the tile loop, the TMA ring and the
// MMA issue are shared; the operands' rows, their major-ness, the K range and
// the epilogue differ):
//   PM_UP      H = SiLU(X W1^T) * (X W3^T) per expert (forward)
//   PM_DOWN    y_slot = perm_w * (H W2^T) per expert (forward)
//   PM_BWD_DH  dh = dYs W2 per expert, W2 read as stored ([d][ffn]: MN-major
//              B); the epilogue applies the SwiGLU backward with the kept u,
//              v: du = dh v SiLU'(u), dv = dh SiLU(u), written side by side
//              as dUV [.][2 ffn] (bf16)
//   PM_BWD_DX  dXp = dUV [W1; W3] per expert, fp32, W1 and W3 read as stored
//              ([ffn][d]: MN-major B), K = 2 ffn
//   PM_WGRAD   weight gradients, fp32: per expert, A^T B over the expert's
//              tokens, both operands read as stored (token rows: MN-major);
//              A is a backward activation whose expert groups start at
//              multiples of 64 rows with zero rows between them, so a K step
//              that runs past the group adds nothing; an expert with no tokens
//              gets zeros
// dYs and dUV (the A operands of the backward modes) use that padded row
// order; x_perm, H and the outputs y_slot, dXp use the plain one.
enum PairMode : int { PM_UP = 0, PM_DOWN = 1, PM_BWD_DH = 2, PM_BWD_DX = 3, PM_WGRAD = 4 };

// Epilogue of one row of a PM_BWD_DH tile: 256 columns f of dh, the kept u
// and v of the same row and columns, du and dv out in bf16. The u, v loads of
// the next 16 columns are issued before the current ones are used, so their
// latency overlaps the tensor-memory load and the arithmetic.
__device__ __forceinline__ void bwd_dh_epilogue(uint32_t taddr, bool valid, int64_t r, int64_t pr, int nt,
                                                const TileArgs& args, int j_begin, int j_end) {
    const int F = args.ldo / 2;
    const int64_t col0 = (int64_t)nt * kTileN;
    const uint4* urow = reinterpret_cast<const uint4*>(args.u_in + r * F + col0);
    const uint4* vrow = reinterpret_cast<const uint4*>(args.v_in + r * F + col0);
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out) + pr * args.ldo + col0;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    uint4 un[2] = {zero, zero}, vn[2] = {zero, zero};
    if (valid) {
        un[0] = urow[j_begin / 8]; un[1] = urow[j_begin / 8 + 1];
        vn[0] = vrow[j_begin / 8]; vn[1] = vrow[j_begin / 8 + 1];
    }
#pragma unroll 1
    for (int j = j_begin; j < j_end; j += 16) {
        const uint4 uc[2] = {un[0], un[1]}, vc[2] = {vn[0], vn[1]};
        if (valid && j + 16 < j_end) {
            un[0] = urow[(j + 16) / 8]; un[1] = urow[(j + 16) / 8 + 1];
            vn[0] = vrow[(j + 16) / 8]; vn[1] = vrow[(j + 16) / 8 + 1];
        }
        uint32_t a[16];
        tmem_ld16(taddr + j, a);
        tmem_wait_ld();
        const __nv_bfloat16* uu = reinterpret_cast<const __nv_bfloat16*>(uc);
        const __nv_bfloat16* vv = reinterpret_cast<const __nv_bfloat16*>(vc);
        uint32_t pdu[8], pdv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float du2[2], dv2[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float dh = __uint_as_float(a[2 * i + q]);
                const float u = __bfloat162float(uu[2 * i + q]);
                const float v = __bfloat162float(vv[2 * i + q]);
                const float sg = __fdividef(1.0f, 1.0f + __expf(-u));
                du2[q] = dh * v * (sg * (1.0f + u * (1.0f - sg)));
                dv2[q] = dh * (u * sg);
            }
            pdu[i] = pack_bf16x2(du2[0], du2[1]);
            pdv[i] = pack_bf16x2(dv2[0], dv2[1]);
        }
        if (valid) {
            uint4* d0 = reinterpret_cast<uint4*>(out + j);
            d0[0] = make_uint4(pdu[0], pdu[1], pdu[2], pdu[3]);
            d0[1] = make_uint4(pdu[4], pdu[5], pdu[6], pdu[7]);
            uint4* d1 = reinterpret_cast<uint4*>(out + F + j);
            d1[0] = make_uint4(pdv[0], pdv[1], pdv[2], pdv[3]);
            d1[1] = make_uint4(pdv[4], pdv[5], pdv[6], pdv[7]);
        }
    }
}

// Epilogue of a PM_WGRAD tile for one warp (32 rows of the gradient, 256
// fp32 columns; zeros when the expert had no tokens, i.e. no MMA wrote the
// accumulator). Each 32-column block goes through the warp's 32 x 33 staging
// array in shared memory, so every store writes 32 consecutive floats of one
// row (one 128-byte line) instead of 16 bytes of 32 different rows.
constexpr int kWgradStageFloats = 32 * 33;

__device__ __forceinline__ void wgrad_epilogue(uint32_t taddr, bool any_k, int e, int row0, int nt, int lane,
                                               float* stage, const TileArgs& args, int j_begin, int j_end) {
    // the warp's rows lie in one gradient matrix (split_rows is a multiple of 256)
    float* base = row0 < args.split_rows ? reinterpret_cast<float*>(args.out) : args.out2;
    const int r0 = row0 < args.split_rows ? row0 : row0 - args.split_rows;
    float* out = base + (int64_t)e * args.out_estride + (int64_t)r0 * args.ldo + (int64_t)nt * kTileN + lane;
#pragma unroll 1
    for (int j = j_begin; j < j_end; j += 32) {
        uint32_t a[16], b[16];
        tmem_ld16(taddr + j, a);
        tmem_ld16(taddr + j + 16, b);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            stage[lane * 33 + c] = any_k ? __uint_as_float(a[c]) : 0.f;
            stage[lane * 33 + 16 + c] = any_k ? __uint_as_float(b[c]) : 0.f;
        }
        __syncwarp();
#pragma unroll 4
        for (int rr = 0; rr < 32; ++rr) out[(int64_t)rr * args.ldo + j] = stage[rr * 33 + lane];
        __syncwarp();
    }
}

// One CTA pair per thread-block cluster (launched with cluster size 2).
//
// Half tiles (forward modes): an expert's last row tile with at most 128 real
// rows runs one M = 128 MMA across the pair instead of M = 256, at about half
// the tensor-core time. Each CTA then supplies 64 token rows (from row
// 64 * rank of the tile), and its accumulator holds those 64 rows twice over
// the lanes: lanes 0-63 carry the tile's columns 0-127, lanes 64-127 columns
// 128-255. For the up projection each CTA's 128 weight rows are 64 rows of W1
// followed by the same 64 rows of W3 (map_b0h / map_b1h: boxes of 64 rows),
// so a lane still finds u and v of the same f, 64 columns apart.
template <int MODE>
__global__ void __launch_bounds__(kPairThreads, 1)
    tile_pair_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                          const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_b0h,
                          const __grid_constant__ CUtensorMap map_b1h, const TileArgs args) {
    constexpr bool UP = MODE == PM_UP;
    constexpr bool WG = MODE == PM_WGRAD;
    constexpr bool A_MN = WG;                      // A read as stored with K = token rows
    constexpr bool B_MN = MODE >= PM_BWD_DH;       // B read as stored (weights, or token rows)
    constexpr bool A_PAD = MODE >= PM_BWD_DH;      // A rows in the padded group order
    extern __shared__ unsigned char tc_smem_raw[];
    unsigned char* smem = align1024(tc_smem_raw);
    TcControl* ctl = reinterpret_cast<TcControl*>(smem + (size_t)kPairStages * kPairStageBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();     // CTA of the pair
    const uint32_t lead = 0;                     // the pair's even CTA
    const bool leader = rank == 0;
    const int pair = blockIdx.x / 2;             // cluster index: the unit sequence
    const int n_pairs = gridDim.x / 2;
    const uint16_t pair_mask = 0x3u;
    const int kid = UP ? K_TILE_UP : (MODE == PM_DOWN ? K_TILE_DOWN : K_TILE_BWD);
    const uint64_t tmo = args.timeout_ns;
    volatile int* abort_flag = &ctl->abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&ctl->tfull[b]), 1);
            mbar_init(smem_u32(&ctl->tempty[b]), 2 * kPairEpiWarps);  // the epilogue warps of both CTAs
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        for (int q = 0; q < kUnitRing; ++q) {
            mbar_init(smem_u32(&ctl->ring_full[q]), 1);
            mbar_init(smem_u32(&ctl->ring_empty[q]), kRingReaders);
        }
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b0);
        if (UP) {
            tma_prefetch_desc(&map_b1);
            tma_prefetch_desc(&map_b0h);
            tma_prefetch_desc(&map_b1h);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&ctl->tmem_base), 2 * kTileAccCols);
        tmem_relinquish_pair();
    }
    pdl_trigger();
    pdl_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < args.n_zero_counts; i += gridDim.x * blockDim.x)
        args.zero_counts[i] = 0;
    if (threadIdx.x == 0) {
        int tiles = 0;
        if (args.offsets != nullptr) {
            for (int e = 0; e <= args.E; ++e) ctl->off[e] = args.offsets[e];
        } else {
            ctl->off[0] = 0;
            ctl->off[1] = args.dense_rows;
        }
        for (int e = 0; e < args.E; ++e) {
            const int c = ctl->off[e + 1] - ctl->off[e];
            ctl->cnt[e] = c;
            // token modes: 256-token row tiles; weight gradients: fixed row tiles, every expert
            ctl->mt[e] = WG ? args.m_tiles : (c + kPairM - 1) / kPairM;
            ctl->base[e] = tiles;
            tiles += ctl->mt[e] * args.n_tiles_n;
        }
        ctl->base[args.E] = tiles;
        ctl->n_work = tiles;
        ctl->koff[0] = 0;
        for (int e = 0; e < args.E; ++e) ctl->koff[e + 1] = ctl->koff[e] + (ctl->cnt[e] + kBK - 1) / kBK * kBK;
        // Half tiles pay when they save a large share of the MMA work (few row tiles per expert): a
        // half tile finishes early, which puts its pair out of step with the pairs that share its
        // weight tiles. Measured at the Mixtral shape: 5.6 % of the MMA rows saved (T = 4096) made the
        // expert GEMMs 0.5-4 % faster; 2.9 % (the skewed T = 8192 batch) made the up projection 1 %
        // slower; 1.9 % (T = 16384) changed nothing measurable. So they run from 4 % on.
        int rows = 0, saved = 0;
        for (int e = 0; e < args.E; ++e) {
            rows += ctl->mt[e] * kPairM;
            const int tail = ctl->cnt[e] - (ctl->mt[e] - 1) * kPairM;
            if (ctl->mt[e] > 0 && tail <= 128) saved += 128;
        }
        ctl->half_ok = MODE <= PM_DOWN && saved * 25 >= rows;
    }
    // both CTAs' barriers are initialised and both halves of tensor memory are
    // allocated before any CTA signals the other
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int n_work = ctl->n_work;
    const int E = args.E;
    const int KB = args.K / kBK;

    // unit -> expert, column tile, row tile
    auto decode = [&](int tile, int& e, int& nt, int& mt) {
        e = 0;
        while (e < E - 1 && tile >= ctl->base[e + 1]) ++e;
        const int rem = tile - ctl->base[e];
        if (args.n_fast) {
            mt = rem / args.n_tiles_n;
            nt = rem - mt * args.n_tiles_n;
        } else {
            nt = rem / ctl->mt[e];
            mt = rem - nt * ctl->mt[e];
        }
    };
    // K steps of a tile: fixed, or the expert's padded token count
    auto ksteps = [&](int e) { return WG ? (ctl->koff[e + 1] - ctl->koff[e]) / kBK : KB; };
    // a forward tile with at most 128 real rows runs as a half tile (M = 128)
    auto is_half = [&](int e, int mt) { return MODE <= PM_DOWN && ctl->half_ok && ctl->cnt[e] - mt * kPairM <= 128; };

    // The pair's it-th unit (-1: none left). Static: pair + it * n_pairs. With a counter: the even CTA's
    // producer claims it (claim_unit) and every other role of both CTAs takes it from the ring slot
    // (take_unit, one thread per role or warp), then frees the slot (give_back).
    const bool shared_counter = args.sched != nullptr;
    // `claimed`: the unit the even CTA's producer took from the counter one iteration ahead, so that the
    // atomic's round trip overlaps the previous unit's loads
    auto claim_unit = [&](int it, int& claimed, int& tile) -> bool {
        const int q = it & (kUnitRing - 1);
        const uint32_t rph = (uint32_t)(it / kUnitRing) & 1u;
        if (!mbar_wait_cluster(smem_u32(&ctl->ring_empty[q]), rph ^ 1u, tmo, abort_flag)) return false;
        int u = claimed < n_work ? claimed : -1;
        if (u >= 0) claimed = atomicAdd(args.sched, 1);
        ctl->ring_unit[q] = u;
        st_cluster_s32(mapa_shared(smem_u32(&ctl->ring_unit[q]), 1), u);
        mbar_arrive(smem_u32(&ctl->ring_full[q]));
        mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->ring_full[q]), 1));
        tile = u;
        return true;
    };
    auto take_unit = [&](int it, int& tile) -> bool {
        const int q = it & (kUnitRing - 1);
        const uint32_t rph = (uint32_t)(it / kUnitRing) & 1u;
        if (!mbar_wait_cluster(smem_u32(&ctl->ring_full[q]), rph, tmo, abort_flag)) return false;
        tile = *reinterpret_cast<volatile int*>(&ctl->ring_unit[q]);
        return true;
    };
    auto give_back = [&](int it) {
        mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->ring_empty[it & (kUnitRing - 1)]), lead));
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            // token rows are re-read for every column tile: keep them in L2;
            // a weight tile is shared by the pairs working on the expert's
            // row tiles at the same time: normal priority (and both operands
            // of the weight gradients, which together exceed L2)
            const uint64_t pol_act = policy_evict_last();
            const uint64_t pol_w = policy_evict_normal();
            const CUtensorMap* map_b = (UP && rank == 1) ? &map_b1 : &map_b0;
            uint32_t s = 0, ph = 0;
            uint32_t issued_mask = 0, issued_ph = 0;
            bool ok = true;
            int claimed = (shared_counter && leader) ? atomicAdd(args.sched, 1) : 0;
            for (int it = 0; ok; ++it) {
                int tile = pair + it * n_pairs;
                if (shared_counter) {
                    if (!(leader ? claim_unit(it, claimed, tile) : take_unit(it, tile))) {
                        raise_abort(ctl, kid, W_PRODUCER);
                        ok = false;
                        break;
                    }
                    if (!leader) give_back(it);
                }
                if (tile < 0 || tile >= n_work) break;
                int e, nt, mt;
                decode(tile, e, nt, mt);
                // this CTA's 128 rows (K-major) or 128 columns (MN-major) of each operand; a half tile's
                // CTA supplies 64 token rows
                const bool half = is_half(e, mt);
                const int a0 = WG ? mt * kPairM + 128 * (int)rank
                                  : (A_PAD ? ctl->koff[e] : ctl->off[e]) + mt * kPairM + (half ? 64 : 128) * (int)rank;
                const int b0 = UP ? e * args.w_rows + nt * kTileM
                                  : (B_MN ? nt * kTileN + 128 * (int)rank
                                          : e * args.w_rows + nt * kTileN + 128 * (int)rank);
                const int nk = ksteps(e);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1, tmo, abort_flag)) {
                        raise_abort(ctl, kid, W_PRODUCER);
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = smem_u32(&ctl->full[s]);
                    const uint32_t fb = mapa_shared(fb_local, lead);  // the pair's even CTA counts both CTAs
                    if (leader) mbar_arrive_expect_tx(fb_local, 2 * kPairStageBytes);
                    const uint32_t sa = smem_u32(smem + (size_t)s * kPairStageBytes);
                    const uint32_t sb = sa + kPairHalfBytes;
                    const int kx = kb * kBK;
                    if (A_MN) {
                        // two boxes of 64 columns x 64 token rows of the padded activation
                        const int ky = ctl->koff[e] + kx;
                        tma_load_2d_pair(sa, &map_a, fb, a0, ky, pol_w);
                        tma_load_2d_pair(sa + kPairHalfBytes / 2, &map_a, fb, a0 + 64, ky, pol_w);
                    } else {
                        tma_load_2d_pair(sa, &map_a, fb, kx, a0, pol_act);
                    }
                    if (B_MN) {
                        // two boxes of 64 columns x 64 K rows, read as stored
                        const CUtensorMap* mb = &map_b0;
                        int ky;
                        if (WG) {
                            ky = ctl->off[e] + kx;                    // token rows of x_perm or H
                        } else if (MODE == PM_BWD_DX) {
                            mb = kx < args.w_rows ? &map_b0 : &map_b1;  // rows of W1, then of W3
                            ky = e * args.w_rows + (kx < args.w_rows ? kx : kx - args.w_rows);
                        } else {
                            ky = e * args.w_rows + kx;                // rows of W2
                        }
                        tma_load_2d_pair(sb, mb, fb, b0, ky, pol_w);
                        tma_load_2d_pair(sb + kPairHalfBytes / 2, mb, fb, b0 + 64, ky, pol_w);
                    } else if (UP && half) {
                        // 64 rows of W1, then the same 64 rows of W3
                        const int bh = e * args.w_rows + nt * kTileM + 64 * (int)rank;
                        tma_load_2d_pair(sb, &map_b0h, fb, kx, bh, pol_w);
                        tma_load_2d_pair(sb + kPairHalfBytes / 2, &map_b1h, fb, kx, bh, pol_w);
                    } else {
                        tma_load_2d_pair(sb, map_b, fb, kx, b0, pol_w);
                    }
                    issued_mask |= 1u << s;
                    issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                    if (++s == kPairStages) { s = 0; ph ^= 1; }
                }
            }
            if (!ok && leader) {
                for (int q = 0; q < kPairStages; ++q)
                    if (issued_mask & (1u << q))
                        drain_wait(smem_u32(&ctl->full[q]), (issued_ph >> q) & 1u, tmo, kid);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA only)
        if (lane == 0 && leader) {
            constexpr uint32_t idesc_full = idesc_bf16_f32(kPairM, kTileN, A_MN, B_MN);
            constexpr uint32_t idesc_half = idesc_bf16_f32(kPairM / 2, kTileN, A_MN, B_MN);
            // descriptor start advance per K step of 16, in 16-byte units:
            // 32 bytes inside a K-major swizzle row, two 1 KB atoms MN-major
            constexpr uint64_t a_step = A_MN ? 128 : 2;
            constexpr uint64_t b_step = B_MN ? 128 : 2;
            uint32_t s = 0, ph = 0;
            bool ok = true, any = false;
            for (int it = 0; ok; ++it) {
                int tile = pair + it * n_pairs;
                if (shared_counter) {
                    if (!take_unit(it, tile)) {
                        raise_abort(ctl, kid, W_MMA);
                        ok = false;
                        break;
                    }
                    give_back(it);
                }
                if (tile < 0 || tile >= n_work) break;
                int e, nt, mt;
                decode(tile, e, nt, mt);
                const int nk = ksteps(e);
                const uint32_t idesc = is_half(e, mt) ? idesc_half : idesc_full;
                const int b = it & 1;
                const uint32_t aph = (it >> 1) & 1;
                if (!mbar_wait_cluster(smem_u32(&ctl->tempty[b]), aph ^ 1, tmo, abort_flag)) {
                    raise_abort(ctl, kid, W_MMA);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * kTileAccCols;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(smem_u32(&ctl->full[s]), ph, tmo, abort_flag)) {
                        raise_abort(ctl, kid, W_MMA);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)s * kPairStageBytes);
                    const uint32_t sb = sa + kPairHalfBytes;
                    const uint64_t adesc = A_MN ? sw128_mnmajor_desc(sa, kPairHalfBytes / 2) : sw128_kmajor_desc(sa);
                    const uint64_t bdesc = B_MN ? sw128_mnmajor_desc(sb, kPairHalfBytes / 2) : sw128_kmajor_desc(sb);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16_pair(d_tmem, adesc + a_step * kk, bdesc + b_step * kk, idesc, (kb | kk) != 0);
                    any = true;
                    mma_commit_pair(smem_u32(&ctl->empty[s]), pair_mask);
                    if (++s == kPairStages) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                mma_commit_pair(smem_u32(&ctl->tfull[b]), pair_mask);
            }
            if (any) {
                mma_commit_pair(smem_u32(&ctl->drain), (uint16_t)1u);
                drain_wait(smem_u32(&ctl->drain), 0, tmo, kid);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2-9, both CTAs)
        const int sub = warp & 3;                 // tensor-memory lanes 32 sub .. 32 sub + 31
        const int half = (warp - 2) >> 2;         // which half of the tile's columns
        const int row_in_tile = 128 * (int)rank + sub * 32 + lane;
        constexpr int ncols = UP ? kTileM : kTileN;  // up: u, v pairs
        const int j_begin = half * (ncols / 2), j_end = j_begin + ncols / 2;
        uint32_t tempty_leader[2];
        for (int b = 0; b < 2; ++b) tempty_leader[b] = mapa_shared(smem_u32(&ctl->tempty[b]), lead);
        for (int it = 0;; ++it) {
            int tile = pair + it * n_pairs;
            if (shared_counter) {
                int got = 1;
                if (lane == 0) got = take_unit(it, tile) ? 1 : 0;
                got = __shfl_sync(0xffffffffu, got, 0);
                tile = __shfl_sync(0xffffffffu, tile, 0);
                if (!got) {
                    if (lane == 0) raise_abort(ctl, kid, W_EPILOGUE);
                    break;
                }
                __syncwarp();
                if (lane == 0) give_back(it);
            }
            if (tile < 0 || tile >= n_work) break;
            int e, nt, mt;
            decode(tile, e, nt, mt);
            const int b = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            if (!mbar_wait(smem_u32(&ctl->tfull[b]), aph, tmo, abort_flag)) {
                raise_abort(ctl, kid, W_EPILOGUE);
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + b * kTileAccCols + ((uint32_t)(sub * 32) << 16);
            if (WG) {
                float* stage = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(ctl) +
                                                        ((sizeof(TcControl) + 15) & ~size_t(15))) +
                               (warp - 2) * kWgradStageFloats;
                wgrad_epilogue(taddr, ksteps(e) > 0, e, mt * kPairM + row_in_tile - lane, nt, lane, stage, args,
                               j_begin, j_end);
            } else {
                // half tile: lane l holds row l mod 64 of this CTA's 64 rows, the tile's columns
                // 128 (l / 64) .. 128 (l / 64) + 127 (up: u and v of f = 64 (l / 64) + j at j, 64 + j)
                const bool hf = is_half(e, mt);
                const int gl = sub * 32 + lane;
                const int grow = hf ? mt * kPairM + 64 * (int)rank + (gl & 63) : mt * kPairM + row_in_tile;
                const bool valid = grow < ctl->cnt[e];
                const int64_t r = ctl->off[e] + grow;
                const int hb = half * (UP ? 32 : 64);
                const int jb = hf ? hb : j_begin, je = hf ? hb + (UP ? 32 : 64) : j_end;
                const int col0 = hf ? nt * (UP ? kTileM : kTileN) + (UP ? 64 : 128) * (gl >> 6) : -1;
                if (MODE == PM_DOWN && args.y != nullptr) {
                    // the combine fused in: does this slot finish its token? (the token's other slot lies
                    // in a lower-numbered expert, whose units come first; wait until that unit is stored)
                    int64_t t = 0, pr = -1;
                    bool finish = false;
                    if (valid) {
                        t = args.perm_token[r];
                        const int s0 = args.slot_row[2 * t], s1 = args.slot_row[2 * t + 1];
                        pr = s0 == r ? s1 : s0;
                        int pe = -1;
                        if (pr >= 0)
                            for (int q = 0; q < E; ++q)
                                if (pr >= ctl->off[q] && pr < ctl->off[q + 1]) pe = q;
                        finish = pr < 0 || pe < e;
                        if (pr >= 0 && pe == e) report_error(MOE_ERR_DEVICE_CHECK, kid, W_INDEX);
                        if (finish && pr >= 0) {
                            const int pm = (int)(pr - ctl->off[pe]) / kPairM;
                            const int* flag = args.done + ctl->base[pe] + nt * ctl->mt[pe] + pm;
                            const uint64_t t0 = global_ns();
                            while (ld_acquire_gpu(flag) < 2 * kPairEpiWarps) {
                                if (global_ns() - t0 > tmo) {
                                    raise_abort(ctl, kid, W_EPILOGUE);
                                    break;
                                }
                                __nanosleep(256);
                            }
                        }
                    }
                    __syncwarp();
                    down_combine_epilogue(taddr, valid, finish, r, pr, t, args, jb, je, col0 < 0 ? nt * kTileN : col0);
                    // the unit's y_slot rows are visible to every SM before the warp counts itself done
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) atomicAdd(args.done + tile, 1);
                } else if (hf) {
                    if (UP)
                        tile_epilogue<true>(taddr, valid, r, nt, args, hb, hb + 32, 64, col0);
                    else
                        tile_epilogue<false>(taddr, valid, r, nt, args, hb, hb + 64, 0, col0);
                } else if (MODE == PM_BWD_DH) {
                    bwd_dh_epilogue(taddr, valid, r, (int64_t)ctl->koff[e] + grow, nt, args, j_begin, j_end);
                } else {
                    tile_epilogue<UP>(taddr, valid, r, nt, args, j_begin, j_end);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader[b]);
        }
    }

    // no CTA of the pair frees tensor memory or leaves while the other may
    // still be signalled or read
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, 2 * kTileAccCols);
}

// ---------------------------------------------------------------------------
// weight-streaming kernels
// ---------------------------------------------------------------------------
struct StreamArgs {
    const int32_t* offsets;  // [E+1]
    float* part;             // fp32 partials
    int E;
    int R;          // rows of x_perm / H (= 2T)
    int kslice;     // K elements per unit
    int S;          // K slices
    int RB;         // 128-row blocks per weight matrix of one expert
    int nmat;       // 2 (W1 and W3) or 1 (W2)
    int w_rows;     // rows of one expert in the weight map (ffn or d)
    int nb;         // token rows per MMA (N), multiple of 16, <= 64
    int stages;     // pipeline depth
    uint32_t stage_bytes;
    uint64_t timeout_ns;
    int dense_rows;  // plain linear layer (offsets == nullptr, E == 1): one group of this many rows
    // Weight bytes of this call that should stay in L2 for the next call (decode-time expert cache,
    // 0 = none): spread evenly over the experts the call touches, each keeps the leading 128-row
    // blocks of its matrices.
    uint64_t keep_bytes;
};

inline size_t stream_smem_bytes(int nb, int stages) {
    const size_t stage = kStreamABytes + (size_t)((nb * 128 + 1023) / 1024) * 1024;
    return 1024 + stage * stages + sizeof(TcControl);
}

// UP = true: partials of W1 x and W3 x, layout [S][2][R][ffn].
// UP = false: partials of W2 h, layout [S][R][d].
template <bool UP>
__global__ void __launch_bounds__(kTcThreads, 1)
    stream_gemm_kernel(const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_w1,
                       const __grid_constant__ CUtensorMap map_x, const StreamArgs args) {
    extern __shared__ unsigned char tc_smem_raw[];
    unsigned char* smem = align1024(tc_smem_raw);
    TcControl* ctl = reinterpret_cast<TcControl*>(smem + (size_t)args.stages * args.stage_bytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int kid = UP ? K_STREAM_UP : K_STREAM_DOWN;
    const uint64_t tmo = args.timeout_ns;
    volatile int* abort_flag = &ctl->abort_flag;
    const int stages = args.stages;
    const int units_per_expert = args.nmat * args.RB * args.S;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < kStreamAcc; ++b) {
            mbar_init(smem_u32(&ctl->tfull[b]), 1);
            mbar_init(smem_u32(&ctl->tempty[b]), 4);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&map_w0);
        if (UP) tma_prefetch_desc(&map_w1);
        tma_prefetch_desc(&map_x);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), kStreamAcc * kStreamMaxNB);
        tmem_relinquish();
    }
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x == 0) {
        int n_act = 0;
        if (args.offsets != nullptr) {
            for (int e = 0; e <= args.E; ++e) ctl->off[e] = args.offsets[e];
        } else {
            ctl->off[0] = 0;
            ctl->off[1] = args.dense_rows;
        }
        bool too_many = false;
        for (int e = 0; e < args.E; ++e) {
            const int c = ctl->off[e + 1] - ctl->off[e];
            ctl->cnt[e] = c;
            if (c > args.nb) too_many = true;
            if (c > 0) ctl->act[n_act++] = e;
        }
        if (too_many) {
            report_error(MOE_ERR_DEVICE_CHECK, kid, W_COUNT);
            n_act = 0;
        }
        ctl->n_act = n_act;
        ctl->n_work = n_act * units_per_expert;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int n_work = ctl->n_work;
    const int KB = args.kslice / kBK;
    const int S = args.S, RB = args.RB;

    auto decode = [&](int u, int& e, int& m, int& rb, int& ks) {
        const int ae = u / units_per_expert;
        int rem = u - ae * units_per_expert;
        ks = rem % S;
        rem /= S;
        rb = rem % RB;
        m = rem / RB;
        e = ctl->act[ae];
    };

    if (warp == 0) {
        if (lane == 0) {
            // Weights are read once per call: evict-first, except the leading row blocks that an expert
            // cache keeps for the next call (the router's choices of consecutive tokens repeat more often
            // than chance: lecture, router walkthrough), which are loaded with the evict-last priority.
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_keep = policy_evict_last();
            const uint64_t pol_x = policy_evict_last();
            const uint32_t x_bytes = (uint32_t)args.nb * 128u;
            int keep_rb = 0;
            if (args.keep_bytes > 0 && ctl->n_act > 0) {
                const uint64_t blk = 128ull * (uint64_t)args.kslice * (uint64_t)S * 2ull;  // one row block of one matrix
                const uint64_t per = args.keep_bytes / (blk * (uint64_t)ctl->n_act * (uint64_t)args.nmat);
                keep_rb = (int)(per < (uint64_t)RB ? per : (uint64_t)RB);
            }
            uint32_t s = 0, ph = 0;
            uint32_t issued_mask = 0, issued_ph = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < n_work; u += gridDim.x) {
                int e, m, rb, ks;
                decode(u, e, m, rb, ks);
                const int wrow = e * args.w_rows + rb * 128;
                const int xrow = ctl->off[e];
                const CUtensorMap* mw = (UP && m == 1) ? &map_w1 : &map_w0;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1, tmo, abort_flag)) {
                        raise_abort(ctl, kid, W_PRODUCER);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&ctl->full[s]);
                    const uint32_t sa = smem_u32(smem + (size_t)s * args.stage_bytes);
                    const int kx = ks * args.kslice + kb * kBK;
                    mbar_arrive_expect_tx(fb, kStreamABytes + x_bytes);
                    tma_load_2d(sa, mw, fb, kx, wrow, rb < keep_rb ? pol_keep : pol_w);
                    tma_load_2d(sa + kStreamABytes, &map_x, fb, kx, xrow, pol_x);
                    issued_mask |= 1u << s;
                    issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                    if (++s == (uint32_t)stages) { s = 0; ph ^= 1; }
                }
            }
            if (!ok) {
                for (int q = 0; q < stages; ++q)
                    if (issued_mask & (1u << q))
                        drain_wait(smem_u32(&ctl->full[q]), (issued_ph >> q) & 1u, tmo, kid);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)args.nb);
            uint32_t s = 0, ph = 0;
            bool ok = true, any = false;
            int it = 0;
            for (int u = blockIdx.x; ok && u < n_work; u += gridDim.x, ++it) {
                const int b = it % kStreamAcc;
                const uint32_t aph = (it / kStreamAcc) & 1;
                if (!mbar_wait(smem_u32(&ctl->tempty[b]), aph ^ 1, tmo, abort_flag)) {
                    raise_abort(ctl, kid, W_MMA);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * kStreamMaxNB;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(smem_u32(&ctl->full[s]), ph, tmo, abort_flag)) {
                        raise_abort(ctl, kid, W_MMA);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)s * args.stage_bytes);
                    const uint64_t adesc = sw128_kmajor_desc(sa);
                    const uint64_t bdesc = sw128_kmajor_desc(sa + kStreamABytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
                    any = true;
                    mma_commit(smem_u32(&ctl->empty[s]));
                    if (++s == (uint32_t)stages) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                mma_commit(smem_u32(&ctl->tfull[b]));
            }
            if (any) {
                mma_commit(smem_u32(&ctl->drain));
                drain_wait(smem_u32(&ctl->drain), 0, tmo, kid);
            }
        }
        __syncwarp();
    } else {
        const int sub = warp & 3;
        const int wr = sub * 32 + lane;  // weight row inside the 128-row block
        int it = 0;
        for (int u = blockIdx.x; u < n_work; u += gridDim.x, ++it) {
            int e, m, rb, ks;
            decode(u, e, m, rb, ks);
            const int b = it % kStreamAcc;
            const uint32_t aph = (it / kStreamAcc) & 1;
            if (!mbar_wait(smem_u32(&ctl->tfull[b]), aph, tmo, abort_flag)) {
                raise_abort(ctl, kid, W_EPILOGUE);
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + b * kStreamMaxNB + ((uint32_t)(sub * 32) << 16);
            const int cnt = ctl->cnt[e];
            const int64_t plane = UP ? ((int64_t)ks * 2 + m) : (int64_t)ks;
            float* dst = args.part + (plane * args.R + ctl->off[e]) * (int64_t)args.w_rows + rb * 128 + wr;
            for (int n0 = 0; n0 < args.nb; n0 += 16) {
                uint32_t a[16];
                tmem_ld16(taddr + n0, a);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (n0 + i < cnt) dst[(int64_t)(n0 + i) * args.w_rows] = __uint_as_float(a[i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[b]));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kStreamAcc * kStreamMaxNB);
}

// H[r][f] = bf16( SiLU(sum_s U_s[r][f]) * sum_s V_s[r][f] ), partials [S][2][R][F]
// u_out, v_out (nullable, training forward): the summed u and v in bf16.
__global__ void __launch_bounds__(256)
    reduce_swiglu_kernel(const float* __restrict__ part, int S, int64_t R, int F,
                         __nv_bfloat16* __restrict__ H, __nv_bfloat16* __restrict__ u_out,
                         __nv_bfloat16* __restrict__ v_out) {
    pdl_trigger();
    pdl_wait();
    const int64_t n = R * F;
    const int64_t plane = R * F;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        // groups of four slices are loaded before they are added (in slice order)
        float u = 0.f, v = 0.f;
        int s = 0;
        for (; s + 4 <= S; s += 4) {
            float pu[4], pv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                pu[q] = part[(2 * (int64_t)(s + q)) * plane + i];
                pv[q] = part[(2 * (int64_t)(s + q) + 1) * plane + i];
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                u += pu[q];
                v += pv[q];
            }
        }
        for (; s < S; ++s) {
            u += part[(2 * (int64_t)s) * plane + i];
            v += part[(2 * (int64_t)s + 1) * plane + i];
        }
        H[i] = __float2bfloat16_rn(silu_f32(u) * v);
        if (u_out != nullptr) {
            u_out[i] = __float2bfloat16_rn(u);
            v_out[i] = __float2bfloat16_rn(v);
        }
    }
}

// y_slot[r][c] = perm_w[r] * sum_s P_s[r][c], partials [S][R][d]
__global__ void __launch_bounds__(256)
    reduce_down_kernel(const float* __restrict__ part, int S, int64_t R, int d,
                       const float* __restrict__ perm_w, float* __restrict__ y_slot) {
    pdl_trigger();
    pdl_wait();
    const int64_t n = R * d;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < S; ++s) acc += part[(int64_t)s * n + i];
        y_slot[i] = perm_w != nullptr ? perm_w[i / d] * acc : acc;
    }
}

// Weight-streaming path of the whole layer: the K-slice sum, the gate scale and
// the two-slot combine in one pass,
//   y[t] = (perm_w[r0] * sum_s P_s[r0]) + (perm_w[r1] * sum_s P_s[r1]),
// with the same operations in the same order as reduce_down_kernel followed
// by the combine, so both routes give bit-identical y.
template <typename T>
__global__ void __launch_bounds__(256)
    reduce_combine_kernel(const float* __restrict__ part, int S, int64_t R, int d, const float* __restrict__ perm_w,
                          const int32_t* __restrict__ slot_row, int64_t T_tokens, T* __restrict__ y) {
    pdl_trigger();
    pdl_wait();
    const int64_t n = T_tokens * d;
    const int64_t plane = R * d;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / d;
        const int64_t c = i - t * d;
        float ab[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int r = slot_row[2 * t + j];
            float v = 0.f;
            if (r >= 0) {
                // groups of eight slices are loaded before they are added (in slice order)
                const float* p = part + (int64_t)r * d + c;
                float acc = 0.f;
                int s = 0;
                for (; s + 8 <= S; s += 8) {
                    float pv[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) pv[q] = p[(int64_t)(s + q) * plane];
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc += pv[q];
                }
                for (; s < S; ++s) acc += p[(int64_t)s * plane];
                v = perm_w[r] * acc;
            }
            ab[j] = v;
        }
        const float sum = ab[0] + ab[1];
        if constexpr (sizeof(T) == 2) y[i] = __float2bfloat16_rn(sum);
        else y[i] = sum;
    }
}

}  // namespace moe
