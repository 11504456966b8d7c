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

// Rows of dYs and dUV are in the padded group order the backward GEMMs read:
// expert e's rows start at koff[e] = sum over q < e of its count rounded up to
// 64, and the rows between groups are zero. One warp per padded row pr:
//   a row of expert e's group (k = pr - koff[e] < count): r = offsets[e] + k,
//     dYs[pr] = perm_w[r] * dy[token], dg[r] = <dy[token], y_slot[r]> / perm_w[r]
//     (= <dy, E_e(x)>); each lane sums its own 8-element chunks in order, then
//     a butterfly adds the lanes;
//   a pad row: dYs[pr] = 0 and dUV[pr] = 0.
__global__ void __launch_bounds__(256)
    bwd_slot_kernel(const __nv_bfloat16* __restrict__ dy, const float* __restrict__ y_slot,
                    const int32_t* __restrict__ perm_token, const float* __restrict__ perm_w,
                    const int32_t* __restrict__ offsets, int E, int d, int F, int64_t padded_rows,
                    __nv_bfloat16* __restrict__ dys, __nv_bfloat16* __restrict__ duv, float* __restrict__ dg) {
    __shared__ int koff[kMaxExperts + 1];
    __shared__ int off[kMaxExperts + 1];
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x == 0) {
        koff[0] = 0;
        for (int e = 0; e <= E; ++e) off[e] = offsets[e];
        for (int e = 0; e < E; ++e) koff[e + 1] = koff[e] + (off[e + 1] - off[e] + 63) / 64 * 64;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t used = koff[E] < padded_rows ? koff[E] : padded_rows;
    for (int64_t pr = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; pr < used;
         pr += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        int e = 0;
        while (e < E - 1 && pr >= koff[e + 1]) ++e;
        const int64_t k = pr - koff[e];
        __nv_bfloat16* out = dys + pr * d;
        if (k >= off[e + 1] - off[e]) {
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int c = lane * 8; c < d; c += 32 * 8) *reinterpret_cast<uint4*>(out + c) = z;
            for (int c = lane * 8; c < 2 * F; c += 32 * 8) *reinterpret_cast<uint4*>(duv + pr * 2 * F + c) = z;
            continue;
        }
        const int64_t r = off[e] + k;
        const int64_t t = perm_token[r];
        const float w = perm_w[r];
        const __nv_bfloat16* dyr = dy + t * d;
        const float* ys = y_slot + r * d;
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
