/*
 * moe.h — C ABI of the top-2 sparse mixture-of-experts feed-forward layer
 * (Mixtral shape: d = 4096, ffn = 14336, E = 8 experts, k = 2), for NVIDIA
 * B300 (sm_103a).
 *
 * The operation, as stated on the web pages about "Mixtral of Experts"
 * (arXiv 2401.04088):
 *   - router: one linear layer gives E scores l = x . W_g; a top-2 mask keeps
 *     the two largest and a softmax over them gives two weights that sum to 1
 *     ("Mixtral of Experts" lecture, router walkthrough; flashpapers.ai
 *     summary, "How It Works"; tokentrails.org "Mixtral", step "The router");
 *   - experts: E_i(x) = W2_i (SiLU(W1_i x) * W3_i x), a SwiGLU block
 *     (tokentrails.org "Mixtral", Code; fdeinterviews.com breakdown, "The paper
 *     in one minute");
 *   - output: y = g_a E_a(x) + g_b E_b(x); the other experts are not run and
 *     their weights are not read (tokentrails.org step "Two experts per token";
 *     lecture, router walkthrough);
 *   - training statistic: L_aux = E * sum_i f_i P_i (tokentrails.org step
 *     "Load balancing").
 *
 * Conventions shared by every call:
 *   - Layouts are row-major and contiguous. Weights use the [out][in] layout of
 *     a linear layer: w_gate [E][d] (row e is the page's column e of W_g),
 *     w1 and w3 [E][ffn][d], w2 [E][d][ffn]. Activations: x [T][d], y [T][d].
 *   - Element type of x, weights, x_perm and y is shape->dtype (MOE_F32 or
 *     MOE_BF16). Router scores, gate weights, y_slot and statistics are float;
 *     indices are int32.
 *   - Every data pointer is DEVICE memory owned by the caller, 16-byte aligned
 *     (the bf16 path reads x_perm, the hidden activations and the weights with
 *     TMA). The library allocates no device memory in any call; intermediates
 *     live in a caller-provided workspace sized by the *_workspace_bytes calls.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls only
 *     enqueue work: they do not synchronise the host and copy nothing back.
 *   - Errors: argument checks happen on the host before anything is enqueued
 *     and return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_WORKSPACE
 *     synchronously. A failed launch returns MOE_ERR_CUDA. Faults found on the
 *     device (a bounded wait that ran out, an index out of range) are latched
 *     in a per-device status word and read with moe_get_device_status().
 *   - Results are deterministic: no floating-point atomics; every reduction
 *     has a fixed order for a given shape.
 *   - Slot order ("expert-contiguous order"): one slot is a (token t, choice j)
 *     pair, j = 0 for the higher score. Rows of x_perm / y_slot list the 2T
 *     slots by expert ascending, then token ascending. offsets[e] is the first
 *     row of expert e; offsets[E] = 2T.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null pointer, negative size, misaligned pointer */
    MOE_ERR_UNSUPPORTED = 2,  /* shape the kernels do not cover (E != 8, k != 2, d or ffn not a tile multiple) */
    MOE_ERR_WORKSPACE = 3,    /* workspace smaller than the *_workspace_bytes figure */
    MOE_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    MOE_ERR_TIMEOUT = 5,      /* device: a bounded wait ran out (kernel returned early) */
    MOE_ERR_DEVICE_CHECK = 6  /* device: an index or count was out of range */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef struct {
    int64_t T;     /* tokens, >= 0 */
    int32_t d;     /* model dimension */
    int32_t ffn;   /* expert hidden dimension */
    int32_t E;     /* experts; must be 8 */
    int32_t k;     /* experts per token; must be 2 */
    int32_t dtype; /* moe_dtype */
} moe_shape;

/* Supported shapes:
 *   MOE_F32 : any d, ffn >= 1 (CUDA-core FFMA path, no TF32).
 *   MOE_BF16: d % 256 == 0 and ffn % 128 == 0 (tcgen05 tensor-core path). */

/* Library version string (static storage). */
const char* moe_version(void);

/* Human-readable name of a status code (static storage). */
const char* moe_status_string(moe_status s);

/* Workspace bytes needed by moe_layer_forward for this shape (0 on a bad
 * shape). Covers routing arrays, x_perm, the hidden activations and y_slot. */
size_t moe_workspace_bytes(const moe_shape* s);

/* Workspace bytes needed by moe_expert_ffn for this shape (0 on a bad shape).
 * moe_expert_ffn and this call accept any s->E from 1 to 8 (a rank of an
 * expert-parallel layer holds a share of the experts); the other calls need
 * E = 8, k = 2. */
size_t moe_ffn_workspace_bytes(const moe_shape* s);

/* Router (lecture router walkthrough; flashpapers "How It Works";
 * tokentrails step "The router").
 *   x        [T][d]   dtype      token rows
 *   w_gate   [E][d]   dtype      router weights
 *   topk_idx [T][2]   int32 out  selected experts, higher score first; equal
 *                                scores go to the lower expert index
 *   topk_w   [T][2]   float out  softmax of the two selected scores
 *   logits   [T][E]   float out  router scores, or NULL to skip writing them
 * Scores are accumulated in fp32 from the stored values. */
moe_status moe_route_top2(const moe_shape* s, const void* x, const void* w_gate,
                          int32_t* topk_idx, float* topk_w, float* logits, void* stream);

/* Grouping of slots by expert (this library's structure; the pages say only
 * that different tokens pick different experts and some experts get none).
 *   topk_idx, topk_w  [T][2]       from moe_route_top2
 *   x                 [T][d]       dtype
 *   counts            [E]   out    slots per expert
 *   offsets           [E+1] out    exclusive prefix sum of counts
 *   perm_token        [2T]  out    token of each row (expert-contiguous order)
 *   slot_row          [T][2] out   row of slot (t, j)
 *   perm_w            [2T]  out    gate weight of each row
 *   x_perm            [2T][d] out  x_perm[r] = x[perm_token[r]]
 *   ws / ws_bytes                  optional scratch of moe_permute_workspace_bytes(s)
 *                                  bytes; with it, batches of 2048 tokens or more are
 *                                  grouped by many CTAs (per-chunk counts, then ranks),
 *                                  without it by one CTA. Both give the same result.
 * An index outside [0, E) latches MOE_ERR_DEVICE_CHECK; that slot gets row -1.
 * A non-NULL ws smaller than required returns MOE_ERR_WORKSPACE. */
moe_status moe_permute(const moe_shape* s, const int32_t* topk_idx, const float* topk_w,
                       const void* x, int32_t* counts, int32_t* offsets, int32_t* perm_token,
                       int32_t* slot_row, float* perm_w, void* x_perm, void* ws, size_t ws_bytes,
                       void* stream);

/* Scratch bytes for moe_permute's many-CTA grouping (0 on a bad shape). */
size_t moe_permute_workspace_bytes(const moe_shape* s);

/* Expert FFNs on the grouped rows, scaled by the gate weight (tokentrails
 * Code: expert = w2(silu(w1 x) * w3 x)):
 *   y_slot[r] = perm_w[r] * W2_e (SiLU(W1_e x_perm[r]) * (W3_e x_perm[r])),
 *   for offsets[e] <= r < offsets[e+1].
 *   x_perm [2T][d] dtype, offsets [E+1] int32 (device), perm_w [2T] float,
 *   w1, w3 [E][ffn][d] dtype, w2 [E][d][ffn] dtype, y_slot [2T][d] float out.
 *   ws / ws_bytes: workspace of at least moe_ffn_workspace_bytes(s) bytes.
 * The bf16 path accumulates in fp32 and rounds SiLU(u)*v to bf16 before the
 * W2 product. Experts with no rows read none of their weights. The row counts
 * stay on the device: the host never waits for them. Each expert may hold at
 * most T rows (true of any top-2 routing, where a token picks two different
 * experts); a larger group latches MOE_ERR_DEVICE_CHECK on the decode-sized
 * path (T <= 64), which then skips the experts' work. */
moe_status moe_expert_ffn(const moe_shape* s, const void* x_perm, const int32_t* offsets,
                          const float* perm_w, const void* w1, const void* w3, const void* w2,
                          float* y_slot, void* ws, size_t ws_bytes, void* stream);

/* Weighted sum back in token order (tokentrails step "Two experts per token"):
 *   y[t] = y_slot[slot_row[t][0]] + y_slot[slot_row[t][1]]  (in that order,
 *   fp32, rounded once to dtype). */
moe_status moe_combine(const moe_shape* s, const float* y_slot, const int32_t* slot_row,
                       void* y, void* stream);

/* Load-balancing statistics (tokentrails step "Load balancing"):
 *   f[i] = counts[i] / (2T), P[i] = mean over tokens of softmax(logits[t])[i]
 *   (all E scores), l_aux[0] = E * sum_i f[i] P[i].
 *   logits [T][E] float, counts [E] int32, f [E], P [E], l_aux [1] float out. */
moe_status moe_aux_stats(const moe_shape* s, const float* logits, const int32_t* counts,
                         float* f, float* P, float* l_aux, void* stream);

/* The whole layer: route, group, expert FFNs, combine (and, when aux_f,
 * aux_P and aux_l_aux are all non-NULL, the load-balancing statistics).
 *   x [T][d], w_gate [E][d], w1, w3 [E][ffn][d], w2 [E][d][ffn], y [T][d] out.
 *   ws / ws_bytes: at least moe_workspace_bytes(s) bytes of device memory.
 * Nothing is copied to the host and the host never waits. */
moe_status moe_layer_forward(const moe_shape* s, const void* x, const void* w_gate,
                             const void* w1, const void* w3, const void* w2, void* y,
                             float* aux_f, float* aux_P, float* aux_l_aux,
                             void* ws, size_t ws_bytes, void* stream);

/* The whole layer without any caller-provided workspace and without any
 * device allocation (the pages have no counterpart: this is a library
 * convenience). It is for callers that cannot call cudaMalloc at the point
 * where they run the layer: for example a plugin inside a host application
 * that reserves all device memory through its own pool, or a latency-critical
 * serving loop that must not call cudaMalloc because an allocation can
 * synchronise the device.
 *   Same arguments and results as moe_layer_forward without statistics; the
 *   caller still passes x, the weights and y (device memory).
 *   Intermediates live in one 24 MiB array of static device memory inside the
 *   library; every GPU that loads the library holds it until the process
 *   exits. A shape whose moe_workspace_bytes() exceeds 24 MiB (25165824 bytes)
 *   is rejected with MOE_ERR_WORKSPACE before anything is enqueued; the
 *   Mixtral decode batch (bf16, d = 4096, ffn = 14336, T <= 16) fits.
 *   The first call on each device looks up the array's device address with
 *   that device current; make that first call before any stream capture.
 *   All calls share the one array and it keeps the previous call's contents
 *   (no part of it needs to start at zero). Calls whose work overlaps on the
 *   GPU (other streams, other host threads) race on it: serialise them. */
moe_status moe_layer_forward_noalloc(const moe_shape* s, const void* x, const void* w_gate,
                                     const void* w1, const void* w3, const void* w2, void* y,
                                     void* stream);

/* Row gather (library plumbing for expert parallelism; the pages have no
 * counterpart): dst[r] = src[index[r]] for r < rows, rows of row_bytes bytes
 * (a multiple of 16). An index outside [0, src_rows) writes a row of zeros and
 * latches MOE_ERR_DEVICE_CHECK. src, index, dst: device memory, 16-byte
 * aligned; src and dst must not overlap. */
moe_status moe_gather_rows(const void* src, int64_t src_rows, const int32_t* index, int64_t rows,
                           int64_t row_bytes, void* dst, void* stream);

/* ---------------------------------------------------------------- training
 * The pages train the router and the experts end to end and add the
 * load-balancing term to the loss (tokentrails.org "Mixtral", step "Load
 * balancing"; lecture, router walkthrough: the router is a learned linear
 * layer). They print no backward pass; these calls give, for an upstream
 * gradient dy, the gradients of
 *     L = sum_t <dy_t, y_t> + aux_coef * L_aux
 * by the chain rule through the forward definition: the top-2 choice and the
 * routed counts f_i are piecewise constant (not differentiated), the two kept
 * weights are the softmax of the two kept scores, L_aux reaches the scores
 * through P_i (the full softmax), SiLU'(z) = s (1 + z (1 - s)).
 * Training needs shape->dtype == MOE_BF16 and d, ffn multiples of 256. */

/* Bytes of the state moe_layer_forward_train keeps for moe_layer_backward
 * (0 on an unsupported shape): the forward workspace plus u = W1 x and
 * v = W3 x of every slot row in bf16. */
size_t moe_train_state_bytes(const moe_shape* s);

/* Bytes of the workspace of moe_layer_backward (0 on an unsupported shape):
 * the per-slot gradients g*dy, [du dv] and dx before the combine (about 160 KB
 * per token at the Mixtral shape) and the router's partial sums. No weight is
 * copied: the backward GEMMs read W1, W3, W2 as stored. */
size_t moe_backward_workspace_bytes(const moe_shape* s);

/* Forward pass that keeps its intermediates for the backward pass.
 *   Same arguments and results as moe_layer_forward (y bit-identical for the
 *   same inputs), with the workspace replaced by
 *   state / state_bytes: at least moe_train_state_bytes(s) bytes of device
 *     memory, owned by the caller and passed unchanged to moe_layer_backward. */
moe_status moe_layer_forward_train(const moe_shape* s, const void* x, const void* w_gate,
                                   const void* w1, const void* w3, const void* w2, void* y,
                                   float* aux_f, float* aux_P, float* aux_l_aux,
                                   void* state, size_t state_bytes, void* stream);

/* Backward pass for an upstream gradient dy [T][d] (bf16).
 *   x, w_gate, w1, w3, w2   the forward's inputs (unchanged since the forward)
 *   aux_coef                weight of L_aux in the loss (0 = none)
 *   state / state_bytes     from moe_layer_forward_train on the same inputs
 *   dx       [T][d]        bf16 out
 *   dw_gate  [E][d]        float out
 *   dw1, dw3 [E][ffn][d]   float out
 *   dw2      [E][d][ffn]   float out
 *   ws / ws_bytes          at least moe_backward_workspace_bytes(s) bytes
 * Gradients are written, not accumulated; an expert no token selected gets
 * zeros. All sums run in a fixed order: results are deterministic. */
moe_status moe_layer_backward(const moe_shape* s, const void* x, const void* w_gate,
                              const void* w1, const void* w3, const void* w2, const void* dy,
                              float aux_coef, const void* state, size_t state_bytes, void* dx,
                              float* dw_gate, float* dw1, float* dw3, float* dw2,
                              void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------------------
 * Decoder block around the layer. Mixtral keeps the Mistral/LLaMA block and
 * replaces its MLP by the MoE layer ("Mixtral" lineage page, step "GPT-2 vs
 * Mixtral" and its Code):
 *   h   = x + Wo . attention(RoPE(Wq xn), RoPE(Wk xn), Wv xn),  xn = RMSNorm(x)
 *   out = h + MoE(RMSNorm(h))
 * with 32 query heads and 8 KV heads of width 128 at d = 4096 (royalroad.pages.dev
 * notes, Architecture; fdeinterviews.com breakdown, layer diagram: 41.9M
 * attention parameters per layer). Readings where the pages are silent:
 * RMSNorm(x) = g * x / sqrt(mean(x^2) + eps); RoPE turns channel pairs
 * (2i, 2i+1) of every query and key head by pos * rope_base^(-2i/head_dim),
 * pos = index inside the sequence; scores q.k / sqrt(head_dim), causal, no
 * sliding window, no biases; query head h reads KV head h / (n_heads /
 * n_kv_heads). A batch is B sequences of S tokens, token-major [B*S][d].
 * Everything here is bf16 storage with fp32 accumulation; the residual stream
 * h is rounded to bf16.
 * ------------------------------------------------------------------------- */
typedef struct {
    int64_t B;           /* sequences, >= 1 */
    int64_t S;           /* tokens per sequence, >= 1 */
    int32_t d;           /* model width, multiple of 256 */
    int32_t n_heads;     /* query heads */
    int32_t n_kv_heads;  /* key/value heads, divides n_heads */
    int32_t head_dim;    /* must be 128 */
    int32_t ffn;         /* the MoE layer's expert width (multiple of 256) */
    int32_t E;           /* experts: 8 */
    int32_t k;           /* experts per token: 2 */
    float eps;           /* RMSNorm epsilon */
    float rope_base;     /* RoPE base */
    int64_t cache_max;   /* key/value cache capacity per sequence (0: no cache) */
} moe_block_shape;

typedef struct {
    const void* attn_norm;  /* [d] bf16 gain of the first RMSNorm */
    const void* wqkv;       /* [(n_heads + 2 n_kv_heads) head_dim][d] bf16: Wq rows, then Wk, then Wv */
    const void* wo;         /* [d][n_heads head_dim] bf16 */
    const void* ffn_norm;   /* [d] bf16 gain of the second RMSNorm */
    const void* w_gate;     /* [E][d] bf16, the MoE layer's weights as for moe_layer_forward */
    const void* w1;         /* [E][ffn][d] */
    const void* w3;         /* [E][ffn][d] */
    const void* w2;         /* [E][d][ffn] */
} moe_block_weights;

/* Workspace of moe_block_forward (0 for an unsupported shape). */
size_t moe_block_workspace_bytes(const moe_block_shape* s);

/* out [B*S][d] bf16 = the decoder block applied to x [B*S][d] bf16 (device
 * pointers, 16-byte aligned; out may not alias x). Enqueues RMSNorm, the fused
 * Q/K/V projection, RoPE, attention, the Wo projection, the residual add fused
 * with the second RMSNorm, moe_layer_forward and the last residual add.
 * k_cache, v_cache (nullable, both or neither): [B][n_kv_heads][cache_max]
 * [head_dim] bf16; when given, every sequence's keys (after RoPE) and values
 * are also stored at positions 0 .. S-1 (needs S <= cache_max), ready for
 * moe_block_decode. */
moe_status moe_block_forward(const moe_block_shape* s, const void* x, const moe_block_weights* w, void* k_cache,
                             void* v_cache, void* out, void* ws, size_t ws_bytes, void* stream);

/* Workspace of moe_block_decode (0 for an unsupported shape). */
size_t moe_block_decode_workspace_bytes(const moe_block_shape* s);

/* One decode step: B sequences, one new token each (s->S must be 1).
 * x [B][d] bf16 holds the new tokens; cache_len [B] int32 (device) the number
 * of tokens each sequence has cached, so the new token sits at that position.
 * The step appends the token's key and value to the caches, attends over the
 * cache (cache_len[b] + 1 keys), runs the rest of the block (the MoE layer on
 * its weight-streaming path for up to 64 sequences) into out [B][d] bf16, and
 * advances cache_len[b] by one, all on the device, so steps follow each other
 * without a host round trip. A sequence whose cache is full (cache_len[b] >=
 * cache_max) latches MOE_ERR_DEVICE_CHECK and is not appended. */
moe_status moe_block_decode(const moe_block_shape* s, const void* x, const moe_block_weights* w, void* k_cache,
                            void* v_cache, int32_t* cache_len, void* out, void* ws, size_t ws_bytes, void* stream);

/* The block's steps, one call each (the same kernels moe_block_forward runs). */

/* y [rows][d] = RMSNorm(h) * g in bf16. With `add` (fp32 [rows][d], nullable)
 * h = bf16(x + add) is formed first and written to h_out [rows][d]; without it
 * h = x and h_out is unused. d % 8 == 0. */
moe_status moe_rmsnorm(int64_t rows, int32_t d, const void* x, const float* add, const void* g, float eps,
                       void* h_out, void* y, void* stream);

/* y [rows][n_out] fp32 = x [rows][n_in] . w^T, w [n_out][n_in] bf16 (a linear
 * layer). n_in % 64 == 0, n_out % 256 == 0. Up to 64 rows with a workspace of
 * moe_linear_workspace_bytes: weight streaming (128 weight rows x the rows per
 * tcgen05 MMA, K split over the SMs, partials summed in slice order);
 * otherwise (or ws NULL) CTA-pair tiles of 256 rows x 256 columns. */
size_t moe_linear_workspace_bytes(int64_t rows, int32_t n_in, int32_t n_out);
moe_status moe_linear(int64_t rows, int32_t n_in, int32_t n_out, const void* x, const void* w, float* y, void* ws,
                      size_t ws_bytes, void* stream);

/* Splits the fused projection qkv [B*S][(n_heads + 2 n_kv_heads) head_dim]
 * fp32 into q [B*S][n_heads head_dim], k and v [B*S][n_kv_heads head_dim]
 * (bf16), turning the channel pairs of q and k by RoPE. Positions are t mod S
 * within each sequence, or, with pos (device int32 [B], s->S == 1, decode),
 * pos[b] for sequence b's one token. k_cache, v_cache (nullable, both or
 * neither; [B][n_kv_heads][cache_max][head_dim]) also receive each key and
 * value at its position; k and v may then be NULL. A position outside the
 * cache latches MOE_ERR_DEVICE_CHECK and is not written. */
moe_status moe_rope_split(const moe_block_shape* s, const float* qkv, const int32_t* pos, void* q, void* k, void* v,
                          void* k_cache, void* v_cache, void* stream);

/* Causal grouped-query attention of each sequence: o [B*S][n_heads head_dim]
 * bf16 from q, k, v as moe_rope_split writes them. head_dim must be 128. */
moe_status moe_attention(const moe_block_shape* s, const void* q, const void* k, const void* v, void* o,
                         void* stream);

/* Decode attention of one new token per sequence: q [B][n_heads head_dim]
 * bf16 against the head-major caches ([B][n_kv_heads][cache_max][head_dim],
 * the token's own key and value already stored at position cache_len[b]),
 * cache_len[b] + 1 keys; o [B][n_heads head_dim] bf16. Splits each
 * sequence's keys over CTAs per KV head (each streams its share in steps of
 * 128 keys through shared memory by TMA, S^T = K Q^T and O^T += V^T P^T on
 * the tensor cores, a running softmax with one key per thread) and merges the
 * partials; advances cache_len[b] by one (up to cache_max). Cache rows at or
 * past a sequence's key count are never used, whatever they hold. ws:
 * moe_attention_decode_workspace_bytes. head_dim 128, n_heads / n_kv_heads
 * <= 16. */
size_t moe_attention_decode_workspace_bytes(const moe_block_shape* s);
moe_status moe_attention_decode(const moe_block_shape* s, const void* q, const void* k_cache, const void* v_cache,
                                int32_t* cache_len, void* o, void* ws, size_t ws_bytes, void* stream);

/* out [n] = bf16(a + b), bf16, n % 8 == 0. */
moe_status moe_residual_add(int64_t n, const void* a, const void* b, void* out, void* stream);

/* Synchronises the current device, then reports and clears its status word.
 * *code receives MOE_OK or the first device-side error since the last read;
 * *detail (nullable) receives 100 * kernel + where for diagnostics, with
 * kernel 1 router, 2 grouping, 3 row gather, 4 up tiles, 5 down tiles,
 * 6 streaming up, 7 streaming down, 12 the wait self-test, 13 backward tiles,
 * 15 RoPE / cache append, 16 attention, and where 1 TMA producer, 2 MMA issuer, 3 epilogue, 4 drain of in-flight
 * work, 5 index check, 6 group larger than the kernel allows. Returns
 * MOE_ERR_CUDA if the device itself reports an error. */
moe_status moe_get_device_status(int32_t* code, int32_t* detail);

/* Waits for `stream`, then reads and clears the device status word like
 * moe_get_device_status, and returns the latched device error (MOE_OK if
 * none, MOE_ERR_CUDA if the device itself failed). */
moe_status moe_check_device_status(void* stream);

/* Self-test of the device-side timeout path (no counterpart on the pages):
 * one CTA waits on an mbarrier that nothing arrives on, with the same bounded
 * wait as the tensor-core kernels. After timeout_ns (1 ns .. 10 s) the wait
 * gives up, *gave_up (device int32) is set to 1 and MOE_ERR_TIMEOUT is latched
 * in the status word, as a real stall would; the device stays usable. */
moe_status moe_selftest_wait_timeout(uint64_t timeout_ns, int32_t* gave_up, void* stream);

/* Read-bandwidth probe (a measurement utility; the pages have no counterpart):
 * reads `bytes` (a multiple of 16) of device memory at `buf` (16-byte aligned)
 * once, with streaming loads, and writes nothing but possibly one word to
 * `sink` (a device uint32, 4-byte aligned). Timed over a buffer much larger
 * than L2 it gives the HBM read rate, the roofline of the weight-streaming
 * kernels, which read and do not write. Enqueued on `stream`; argument errors
 * return MOE_ERR_INVALID_ARG before anything is enqueued. */
moe_status moe_read_probe(const void* buf, size_t bytes, uint32_t* sink, void* stream);

/* Upper bound, in nanoseconds, on every device-side wait of the tensor-core
 * kernels (default 2e9). A wait that runs out latches MOE_ERR_TIMEOUT and the
 * kernel returns early after its in-flight copies and MMAs have landed. */
moe_status moe_set_wait_timeout_ns(uint64_t ns);

/* Tuning / test knobs (host-side, process-wide):
 *   MOE_KNOB_FFN_PATH   0 = automatic, 1 = token-tile path (128 tokens x 256
 *                       columns per tile), 2 = weight-streaming path (128
 *                       weight rows x up to 64 tokens per tile; needs T <= 64)
 *   MOE_KNOB_KSLICE     K-slice of the weight-streaming path (multiple of 64;
 *                       0 = automatic)
 *   MOE_KNOB_GRID       CTAs of the persistent tensor-core kernels (0 = one
 *                       per SM)
 *   MOE_KNOB_PDL        1 (default) = launch each kernel with programmatic
 *                       dependent launch, so it starts while its predecessor
 *                       drains (it still waits for the predecessor's results
 *                       before touching memory); 0 = plain serialised launches
 *   MOE_KNOB_TILE_CTAS  0 (default) = automatic: 128-token tiles on single
 *                       CTAs up to 384 tokens, 256-token tiles on CTA pairs
 *                       (one tcgen05 MMA spans two SMs) above; 1 = single
 *                       CTAs; 2 = CTA pairs. The single-CTA kernel also
 *                       runs when no CTA pair fits.
 *   MOE_KNOB_L2_KEEP_KB decode-time expert cache of the weight-streaming path
 *                       (0 .. 131072 KiB; default 0 = off): about this many
 *                       KiB of each call's expert weights are loaded with the
 *                       L2 evict-last priority so that a following call that
 *                       routes to the same experts finds them in L2 (the
 *                       router's choices of consecutive tokens repeat more
 *                       often than chance: "Mixtral of Experts" lecture,
 *                       router walkthrough). The budget is spread evenly over
 *                       the experts a call touches, each keeping the leading
 *                       rows of W1, W3 (two thirds) and W2 (one third); the
 *                       rest is loaded evict-first. Results do not change.
 *   MOE_KNOB_TILE_SCHED CTA-pair GEMMs, a bit mask (0 .. 7; default 0): bit 0
 *                       for the up projection, bit 1 for the down projection,
 *                       bit 2 for the four GEMMs of moe_layer_backward. Clear:
 *                       pair p computes units p, p + pairs, p + 2 pairs, ...;
 *                       set: the pairs claim units in order from a counter in
 *                       the workspace (zeroed on the stream before the
 *                       launches) as they become free, so the units in flight
 *                       stay a window of consecutive units. At the Mixtral
 *                       shape with T = 16384 this halves the up projection's
 *                       DRAM reads but takes 0.4 % longer (T = 4096: 2 %; the
 *                       backward's GEMMs: 2-7 %). Results do not change.
 *   MOE_KNOB_ROUTER_TC  1 (default) = bf16 batches of more than 256 tokens
 *                       compute the router's scores on the tensor cores (fp32
 *                       accumulation in tensor memory, 128 tokens per tile);
 *                       0 = on the CUDA cores (the fixed per-lane order with a
 *                       butterfly, as for small batches). The two sum the d
 *                       products in different orders, so scores can differ in
 *                       the last bits.
 *   MOE_KNOB_FUSE_COMBINE 1 (default) = moe_layer_forward on CTA-pair token
 *                       tiles runs the combine inside the down projection: the
 *                       slot of a token in the higher-numbered of its two
 *                       experts waits for the unit holding the other slot,
 *                       adds that slot's y_slot row to its own and writes the
 *                       token's row of y (bf16), so y_slot is written only for
 *                       the other slots and the separate combine pass is
 *                       skipped; 0 = y_slot for every slot, then the combine.
 *                       Results are bit-identical. The fused form needs all
 *                       CTA pairs resident at once, so with MOE_KNOB_GRID above
 *                       one CTA per SM the separate combine runs.
 *   MOE_KNOB_DEBUG      1 = debug mode: every launch is followed by a wait on
 *                       its stream and a look at the device status word, so a
 *                       device-side error (timeout, index check) is returned by
 *                       the call that launched the kernel and the kernel is
 *                       named on stderr; 0 (default) = asynchronous
 * Returns MOE_ERR_INVALID_ARG for an unknown knob or value.
 * Environment, read when the library loads: MOE_DEBUG=1 starts in debug mode;
 * MOE_WAIT_TIMEOUT_NS sets the initial wait limit (as moe_set_wait_timeout_ns). */
enum { MOE_KNOB_FFN_PATH = 1, MOE_KNOB_KSLICE = 2, MOE_KNOB_GRID = 3, MOE_KNOB_PDL = 4, MOE_KNOB_TILE_CTAS = 5,
       MOE_KNOB_DEBUG = 6, MOE_KNOB_L2_KEEP_KB = 7, MOE_KNOB_TILE_SCHED = 8, MOE_KNOB_ROUTER_TC = 9,
       MOE_KNOB_FUSE_COMBINE = 10 };
moe_status moe_set_knob(int32_t knob, int64_t value);

/* Per-kernel timing with CUDA events recorded on the launching stream.
 * moe_timing_enable(1) starts recording every kernel this library launches;
 * moe_timing_read() synchronises on the recorded events, writes a JSON object
 * {"kernel": [launches, total_ms], ...} into buf (NUL-terminated, truncated to
 * n bytes) and clears the record. Returns MOE_ERR_CUDA on an event error. */
moe_status moe_timing_enable(int32_t enable);
moe_status moe_timing_read(char* buf, size_t n);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
