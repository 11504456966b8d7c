// Backward pass of the MoE layer: the small kernels around the CTA-pair GEMMs
// (ffn_tc.cuh, modes PM_BWD_DH, PM_BWD_DX and PM_WGRAD).
//
// The pages train the router and the experts end to end with the
// load-balancing term added to the loss (tokentrails.org "Mixtral", step "Load
// balancing"; "Mixtral of Experts" lecture, router walkthrough). For an
// upstream gradient dy these kernels and the GEMMs give the gradients of
//   L = sum_t <dy_t, y_t> + aux_coef * L_aux
// by the chain rule through the forward definition:
//   dg_k = <dy, E_k(x)>                         (per slot, bwd_slot_kernel)
//   dYs  = g_k dy                               (per slot, bwd_slot_kernel)
//   dl_j = g_j (dg_j - sum_i g_i dg_i)          (kept scores; k = 2 softmax)
//        + aux_coef (E/T) p_j (f_j - sum_i f_i p_i)   (P_i through the full softmax p;
//                                                f_i, a count, is piecewise constant)
//   dx   = dXp[slot 0] + dXp[slot 1] + dl W_g   (bwd_combine_kernel)
//   dW_g = dl^T x                               (dwg kernels, fixed-order sums)
// Everything is deterministic: sums run in a fixed order and no result depends
// on atomics.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kTrTile = 64;        // transpose tile (elements per side)
constexpr int kTrThreads = 256;

// out[b][c][col_off + r] = in[b][r][c] for r < rows, c < cols (bf16); rows and
// cols are multiples of 64. Batched over experts (blockIdx.z).
__global__ void __launch_bounds__(kTrThreads)
    transpose_w_kernel(const __nv_bfloat16* __restrict__ in, int rows, int cols, __nv_bfloat16* __restrict__ out,
                       int ld_out, int col_off) {
    __shared__ __nv_bfloat16 tile[kTrTile][kTrTile + 8];
    pdl_trigger();
    pdl_wait();
    const int r0 = blockIdx.y * kTrTile, c0 = blockIdx.x * kTrTile;
    const __nv_bfloat16* src = in + (int64_t)blockIdx.z * rows * cols;
    __nv_bfloat16* dst = out + (int64_t)blockIdx.z * cols * ld_out;
    // load: 64 rows x 8 chunks of 8 elements
    for (int i = threadIdx.x; i < kTrTile * 8; i += kTrThreads) {
        const int rr = i >> 3, cc = (i & 7) * 8;
        const uint4 v = *reinterpret_cast<const uint4*>(src + (int64_t)(r0 + rr) * cols + c0 + cc);
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
        for (int q = 0; q < 8; ++q) tile[rr][cc + q] = e[q];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kTrTile * 8; i += kTrThreads) {
        const int cc = i >> 3, rr = (i & 7) * 8;
        __align__(16) __nv_bfloat16 e[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) e[q] = tile[rr + q][cc];
        *reinterpret_cast<uint4*>(dst + (int64_t)(c0 + cc) * ld_out + col_off + r0 + rr) =
            *reinterpret_cast<const uint4*>(e);
    }
}

// Token transpose of an activation in expert-contiguous row order:
// out[c][j] = in[r][c] with j = kofs[e] + (r - offsets[e]), where expert e's
// group starts at kofs[e] = sum over q < e of cnt[q] rounded up to 64; the
// columns of a group past its cnt[e] tokens are zero. A 64-column tile of the
// output lies inside one group. cols is a multiple of 64.
__global__ void __launch_bounds__(kTrThreads)
    transpose_tok_kernel(const __nv_bfloat16* __restrict__ in, const int32_t* __restrict__ offsets, int E, int cols,
                         __nv_bfloat16* __restrict__ out, int64_t ld_out) {
    __shared__ __nv_bfloat16 tile[kTrTile][kTrTile + 8];
    __shared__ int grp[3];  // expert, first token row, tokens
    pdl_trigger();
    pdl_wait();
    const int64_t j0 = (int64_t)blockIdx.y * kTrTile;
    const int c0 = blockIdx.x * kTrTile;
    if (threadIdx.x == 0) {
        int k = 0, e = -1, r0 = 0, n = 0;
        for (int q = 0; q < E; ++q) {
            const int c = offsets[q + 1] - offsets[q];
            const int kp = (c + kBK - 1) / kBK * kBK;
            if (j0 >= k && j0 < k + kp) { e = q; r0 = offsets[q] + (int)(j0 - k); n = c - (int)(j0 - k); }
            k += kp;
        }
        grp[0] = e; grp[1] = r0; grp[2] = n;
    }
    __syncthreads();
    if (grp[0] < 0) return;  // past the last group: never read
    const int r0 = grp[1], n = grp[2];
    for (int i = threadIdx.x; i < kTrTile * 8; i += kTrThreads) {
        const int rr = i >> 3, cc = (i & 7) * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (rr < n) v = *reinterpret_cast<const uint4*>(in + (int64_t)(r0 + rr) * cols + c0 + cc);
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
        for (int q = 0; q < 8; ++q) tile[rr][cc + q] = e[q];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kTrTile * 8; i += kTrThreads) {
        const int cc = i >> 3, rr = (i & 7) * 8;
        __align__(16) __nv_bfloat16 e[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) e[q] = tile[rr + q][cc];
        *reinterpret_cast<uint4*>(out + (int64_t)(c0 + cc) * ld_out + j0 + rr) = *reinterpret_cast<const uint4*>(e);
    }
}

// Per slot row r (one warp each): dYs[r] = perm_w[r] * dy[token], and
// dg[r] = <dy[token], y_slot[r]> / perm_w[r], i.e. <dy, E_e(x)>. Each lane sums
// its own 8-element chunks in order, then a butterfly adds the lanes.
__global__ void __launch_bounds__(256)
    bwd_slot_kernel(const __nv_bfloat16* __restrict__ dy, const float* __restrict__ y_slot,
                    const int32_t* __restrict__ perm_token, const float* __restrict__ perm_w,
                    const int32_t* __restrict__ offsets, int E, int d, __nv_bfloat16* __restrict__ dys,
                    float* __restrict__ dg) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t rows = offsets[E];
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows;
         r += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const int64_t t = perm_token[r];
        const float w = perm_w[r];
        const __nv_bfloat16* dyr = dy + t * d;
        const float* ys = y_slot + r * d;
        __nv_bfloat16* out = dys + r * d;
        float acc = 0.f;
        for (int c = lane * 8; c < d; c += 32 * 8) {
            const uint4 raw = *reinterpret_cast<const uint4*>(dyr + c);
            const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(&raw);
            const float4 y0 = *reinterpret_cast<const float4*>(ys + c);
            const float4 y1 = *reinterpret_cast<const float4*>(ys + c + 4);
            const float yv[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
            uint32_t pk[4];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc = fmaf(__bfloat162float(v[q]), yv[q], acc);
#pragma unroll
            for (int q = 0; q < 4; ++q) pk[q] = pack_bf16x2(w * __bfloat162float(v[2 * q]), w * __bfloat162float(v[2 * q + 1]));
            *reinterpret_cast<uint4*>(out + c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) dg[r] = acc / w;
    }
}

// Per token: the scores' gradient dl[t][E] from the kept weights' gradient
// (two-way softmax Jacobian) plus aux_coef times the load-balancing term's.
__global__ void __launch_bounds__(256)
    bwd_router_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
                      const int32_t* __restrict__ slot_row, const float* __restrict__ dg,
                      const float* __restrict__ logits, const int32_t* __restrict__ counts, int64_t T_tokens, int E,
                      float aux_coef, float* __restrict__ dl) {
    __shared__ float f[kMaxExperts];
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x < kMaxExperts)
        f[threadIdx.x] = threadIdx.x < E ? (float)counts[threadIdx.x] / (float)(2 * T_tokens) : 0.f;
    __syncthreads();
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T_tokens; t += (int64_t)gridDim.x * blockDim.x) {
        float out[kMaxExperts];
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e) out[e] = 0.f;
        const int a = topk_idx[2 * t], b = topk_idx[2 * t + 1];
        const float ga = topk_w[2 * t], gb = topk_w[2 * t + 1];
        const int ra = slot_row[2 * t], rb = slot_row[2 * t + 1];
        const float dga = ra >= 0 ? dg[ra] : 0.f, dgb = rb >= 0 ? dg[rb] : 0.f;
        const float sdg = ga * dga + gb * dgb;
        const float dla = ga * (dga - sdg), dlb = gb * (dgb - sdg);
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e) {
            if (e == a) out[e] += dla;
            if (e == b) out[e] += dlb;
        }
        if (aux_coef != 0.f) {
            float l[kMaxExperts], m = -INFINITY;
#pragma unroll
            for (int e = 0; e < kMaxExperts; ++e) {
                l[e] = e < E ? logits[t * E + e] : -INFINITY;
                m = fmaxf(m, l[e]);
            }
            float p[kMaxExperts], z = 0.f;
#pragma unroll
            for (int e = 0; e < kMaxExperts; ++e) {
                p[e] = e < E ? expf(l[e] - m) : 0.f;
                z += p[e];
            }
            float c = 0.f;
#pragma unroll
            for (int e = 0; e < kMaxExperts; ++e) {
                p[e] /= z;
                c += f[e] * p[e];
            }
            const float scale = aux_coef * (float)E / (float)T_tokens;
#pragma unroll
            for (int e = 0; e < kMaxExperts; ++e) out[e] += scale * p[e] * (f[e] - c);
        }
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e)
            if (e < E) dl[t * E + e] = out[e];
    }
}

// dx[t][c] = dXp[slot_row[t][0]][c] + dXp[slot_row[t][1]][c] + sum_e dl[t][e] W_g[e][c],
// added in that order, rounded once to bf16.
__global__ void __launch_bounds__(256)
    bwd_combine_kernel(const float* __restrict__ dxp, const int32_t* __restrict__ slot_row,
                       const float* __restrict__ dl, const __nv_bfloat16* __restrict__ wg, int64_t T_tokens, int d,
                       int E, __nv_bfloat16* __restrict__ dx) {
    pdl_trigger();
    pdl_wait();
    const int64_t n = T_tokens * (d / 4);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / (d / 4);
        const int c = (int)(i - t * (d / 4)) * 4;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int r = slot_row[2 * t + j];
            if (r >= 0) {
                const float4 v = *reinterpret_cast<const float4*>(dxp + (int64_t)r * d + c);
                acc[0] += v.x; acc[1] += v.y; acc[2] += v.z; acc[3] += v.w;
            }
        }
        for (int e = 0; e < E; ++e) {
            const float g = dl[t * E + e];
            const uint2 raw = *reinterpret_cast<const uint2*>(wg + (int64_t)e * d + c);
            const __nv_bfloat16* w = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = fmaf(g, __bfloat162float(w[q]), acc[q]);
        }
        uint2 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        *reinterpret_cast<uint2*>(dx + t * d + c) = o;
    }
}

constexpr int kDwgChunk = 128;  // tokens per partial sum of the router's weight gradient

// part[chunk][e][c] = sum over the chunk's tokens t (in order) of dl[t][e] x[t][c]
__global__ void __launch_bounds__(256)
    dwg_partial_kernel(const float* __restrict__ dl, const __nv_bfloat16* __restrict__ x, int64_t T_tokens, int d,
                       int E, float* __restrict__ part) {
    pdl_trigger();
    pdl_wait();
    const int c = blockIdx.y * blockDim.x + threadIdx.x;
    const int64_t t0 = (int64_t)blockIdx.x * kDwgChunk;
    const int64_t t1 = t0 + kDwgChunk < T_tokens ? t0 + kDwgChunk : T_tokens;
    if (c >= d) return;
    float acc[kMaxExperts];
#pragma unroll
    for (int e = 0; e < kMaxExperts; ++e) acc[e] = 0.f;
    for (int64_t t = t0; t < t1; ++t) {
        const float xv = __bfloat162float(x[t * d + c]);
#pragma unroll
        for (int e = 0; e < kMaxExperts; ++e)
            if (e < E) acc[e] = fmaf(dl[t * E + e], xv, acc[e]);
    }
    for (int e = 0; e < E; ++e) part[((int64_t)blockIdx.x * E + e) * d + c] = acc[e];
}

// dw_gate[e][c] = sum over chunks, in order, of part[chunk][e][c]
__global__ void __launch_bounds__(256)
    dwg_final_kernel(const float* __restrict__ part, int nchunks, int d, int E, float* __restrict__ dwg) {
    pdl_trigger();
    pdl_wait();
    const int64_t n = (int64_t)E * d;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float acc = 0.f;
        for (int k = 0; k < nchunks; ++k) acc += part[(int64_t)k * n + i];
        dwg[i] = acc;
    }
}

}  // namespace moe
