// C ABI of the top-2 sparse MoE layer (declared in include/moe.h): argument
// checks, workspace layout, tensor-map encoding, kernel dispatch, per-kernel
// timing and the device status word. All device work is in the kernels
// included below; this file only marshals arguments and enqueues launches on
// the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <utility>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "common.cuh"
#include "ffn_f32.cuh"
#include "ffn_tc.cuh"
#include "bwd.cuh"
#include "permute.cuh"
#include "router.cuh"
#include "block.cuh"
#include "attention.cuh"

namespace moe {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 1024;
constexpr int kStreamMaxTokens = 64;     // weight-streaming path needs T <= 64
constexpr int64_t kRouterSplitMaxTokens = 256;  // one CTA per token below this
constexpr int64_t kFusedGatherBytes = 512 * 1024;  // the permutation CTA gathers x_perm below this
constexpr int64_t kPermuteMultiMinTokens = 2048;  // many-CTA grouping from this batch size on
constexpr int64_t kPermuteMaxChunks = 4096;       // token chunks (CTAs) of the many-CTA grouping
// Token tiles on single CTAs (128 tokens) up to this batch size, on CTA pairs
// (256 tokens) above: with few tokens per expert the smaller tile pads less and
// keeps more weight bytes in flight. Measured at the Mixtral shape: T = 128
// 0.499 vs 0.530 ms, T = 256 0.511 vs 0.553 ms, T = 512 0.628 vs 0.585 ms.
constexpr int64_t kSingleCtaMaxTokens = 384;
constexpr size_t kSmemBudget = 225 * 1024;
constexpr size_t kStreamInflightBytes = 20u << 20;  // weight bytes in flight, whole GPU

struct TimingRecord {
    const char* name;
    cudaEvent_t start, stop;
};

// Initial wait limit: MOE_WAIT_TIMEOUT_NS from the environment (1 ns .. 10 s), else 2 s.
uint64_t env_timeout_ns() {
    const char* v = std::getenv("MOE_WAIT_TIMEOUT_NS");
    if (v == nullptr) return 2000000000ull;
    char* end = nullptr;
    const unsigned long long t = std::strtoull(v, &end, 10);
    return (end != v && *end == '\0' && t >= 1 && t <= 10000000000ull) ? (uint64_t)t : 2000000000ull;
}

bool env_flag(const char* name) {
    const char* v = std::getenv(name);
    return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
}

struct HostState {
    int ffn_path = 0;          // 0 auto, 1 token tiles, 2 weight streaming
    int64_t kslice = 0;        // 0 auto
    int grid = 0;              // 0 = one CTA per SM
    uint64_t timeout_ns = env_timeout_ns();
    bool debug = env_flag("MOE_DEBUG");  // synchronise after every launch and report device errors at once
    bool timing = false;
    bool pdl = true;           // programmatic dependent launch between the library's kernels
    int tile_ctas = 0;         // token tiles: 0 auto, 1 single CTAs, 2 CTA pairs
    int tile_sched = 0;        // CTA-pair GEMMs claiming units from a counter: bit 0 up, 1 down, 2 backward
    bool router_tc = true;     // bf16 router above the small-batch size on the tensor cores
    bool fuse_combine = true;  // whole-layer call on CTA pairs: the combine runs in the down projection
    uint64_t l2_keep_bytes = 0;  // weight-streaming path: bytes per call kept in L2 for the next call
    int pair_cap[kMaxDevices][8] = {{0}};  // resident clusters per pair kernel (0 = not queried)
    std::vector<TimingRecord> records;
    std::vector<cudaEvent_t> pool;
    int sms[kMaxDevices] = {0};
    bool attr_set[kMaxDevices][32] = {{false}};
};
HostState g;

// NVTX range around an ABI call, so profilers show the library's calls on the
// host timeline (the NVTX header is self-contained; it costs nothing when no
// tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 148;
    if (g.sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g.sms[dev] = n;
    }
    return g.sms[dev];
}

// Raises a kernel's dynamic shared-memory limit once per device.
template <typename K>
bool ensure_smem(K kernel, int slot, size_t bytes) {
    const int dev = current_device();
    if (dev >= 0 && dev < kMaxDevices && g.attr_set[dev][slot]) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return false;
    if (dev >= 0 && dev < kMaxDevices) g.attr_set[dev][slot] = true;
    return true;
}

cudaEvent_t take_event() {
    if (!g.pool.empty()) {
        cudaEvent_t e = g.pool.back();
        g.pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Launches a kernel with programmatic dependent launch allowed (unless the
// knob turned it off): the kernel may start while its predecessor in the
// stream drains, and waits inside (griddepcontrol.wait) before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t klaunch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                    Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// As klaunch, for a kernel that runs in thread-block clusters of `cluster` CTAs.
template <typename... KArgs, typename... Args>
cudaError_t klaunch_cluster(void (*kernel)(KArgs...), int cluster, dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename F>
moe_status launch(const char* name, cudaStream_t st, F&& f) {
    cudaEvent_t a = nullptr, b = nullptr;
    if (g.timing) {
        a = take_event();
        b = take_event();
        cudaEventRecord(a, st);
    }
    const cudaError_t lerr = f();
    const cudaError_t err = lerr != cudaSuccess ? lerr : cudaGetLastError();
    if (g.timing) {
        cudaEventRecord(b, st);
        g.records.push_back({name, a, b});
    }
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    if (g.debug) {
        // debug mode: wait for this kernel and return a device-side error from the call that
        // launched it, naming the kernel (the status word is left latched for the next read)
        if (cudaStreamSynchronize(st) != cudaSuccess) {
            std::fprintf(stderr, "moe debug: %s: %s\n", name, cudaGetErrorString(cudaGetLastError()));
            return MOE_ERR_CUDA;
        }
        int h[4] = {0, 0, 0, 0};
        if (cudaMemcpyFromSymbol(h, g_status, sizeof(h)) != cudaSuccess) return MOE_ERR_CUDA;
        if (h[0] != 0) {
            std::fprintf(stderr, "moe debug: %s: device status %d (kernel %d, where %d, block %d)\n", name, h[0],
                         h[1], h[2], h[3]);
            return static_cast<moe_status>(h[0]);
        }
    }
    return MOE_OK;
}

#define MOE_TRY(expr)                         \
    do {                                      \
        const moe_status _st = (expr);        \
        if (_st != MOE_OK) return _st;        \
    } while (0)

// ------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D bf16 matrix [rows][inner], boxes of box_rows x 64 elements, 128-byte
// swizzle (the layout the MMA descriptors expect), zero fill outside.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------ validation
moe_status check_shape(const moe_shape* s) {
    if (s == nullptr) return MOE_ERR_INVALID_ARG;
    if (s->T < 0 || s->T > (int64_t(1) << 29) || s->d <= 0 || s->ffn <= 0) return MOE_ERR_INVALID_ARG;
    if (s->dtype != MOE_F32 && s->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (s->E != 8 || s->k != 2) return MOE_ERR_UNSUPPORTED;
    if (s->dtype == MOE_BF16 && (s->d % 256 != 0 || s->ffn % 128 != 0)) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)s->d * s->ffn > (int64_t(1) << 31) / 8) return MOE_ERR_UNSUPPORTED;  // int32 weight rows
    return MOE_OK;
}

// The expert FFN alone runs any number of experts from 1 to 8 (an
// expert-parallel rank holds a share of them); k does not enter it.
moe_status check_ffn_shape(const moe_shape* s) {
    if (s == nullptr || s->E < 1 || s->E > kMaxExperts) return s == nullptr ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED;
    moe_shape t = *s;
    t.E = 8;
    t.k = 2;
    return check_shape(&t);
}

bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }

size_t esize(const moe_shape& s) { return s.dtype == MOE_BF16 ? 2 : 4; }

// K slice of a weight-streaming kernel whose units are `rows_units` weight
// row blocks (of all experts) times the K slices. Slices of 1024-2048 elements
// that divide K are tried, and the one whose units fill the last wave of CTAs
// best wins (ties: the wider slice, fewer partial sums); smaller K fall back to
// the widest divisor up to 1024. Decode batch, Mixtral shape: the up
// projection keeps 1024 (7168 units, 48.4 waves); the down projection takes
// 1792 (2048 units, 13.8 waves) instead of 1024 (3584 units, 24.2 waves),
// 146 vs 150 us and fewer partials to sum.
int pick_kslice(int K, int64_t rows_units) {
    if (g.kslice > 0 && g.kslice % kBK == 0 && K % g.kslice == 0) return (int)g.kslice;
    const int64_t grid = sm_count();
    int best = 0;
    double best_fill = -1.0;
    for (int ks = 1024; ks <= 2048 && ks <= K; ks += kBK) {
        if (K % ks != 0) continue;
        const int64_t units = rows_units * (K / ks);
        const double waves = (double)units / (double)grid;
        const double fill = waves / std::ceil(waves);
        if (fill >= best_fill) {
            best_fill = fill;
            best = ks;
        }
    }
    if (best > 0) return best;
    for (int ks = 1024; ks >= kBK; ks -= kBK)
        if (K % ks == 0) return ks;
    return K;
}

// 1 = token tiles, 2 = weight streaming, 0 = unsupported request
int choose_path(const moe_shape& s) {
    if (s.dtype != MOE_BF16) return 0;
    if (g.ffn_path == 1) return 1;
    if (g.ffn_path == 2) return s.T <= kStreamMaxTokens ? 2 : 0;
    return s.T <= kStreamMaxTokens ? 2 : 1;
}

// Tokens per CTA of the many-CTA grouping and the number of chunks.
int64_t permute_chunk(int64_t T) {
    const int64_t c = (T + kPermuteMaxChunks - 1) / kPermuteMaxChunks;
    return std::max<int64_t>(kPlaceSub, (c + kPlaceSub - 1) / kPlaceSub * kPlaceSub);
}

size_t permute_ws_bytes(const moe_shape& s) {
    const int64_t chunks = (std::max<int64_t>(s.T, 1) + permute_chunk(s.T) - 1) / permute_chunk(s.T);
    return align_up((size_t)chunks * kMaxExperts * sizeof(int32_t), 256);
}

struct FfnLayout {
    int path = 0;
    int nb = 0, ks_up = 0, ks_down = 0, S_up = 0, S_down = 0;
    size_t h = 0, part_up = 0, part_down = 0, sched = 0, done = 0, total = 0;
};

FfnLayout ffn_layout(const moe_shape& s) {
    FfnLayout L;
    const size_t R = (size_t)(2 * s.T);
    size_t off = 0;
    L.h = off;
    off = align_up(off + R * s.ffn * esize(s), kAlign);
    if (s.dtype == MOE_BF16) {
        L.path = choose_path(s);
        if (L.path == 2) {
            L.nb = (int)align_up((size_t)(s.T > 0 ? s.T : 1), 16);
            // units: weight row blocks of 128 of every expert (two matrices up)
            L.ks_up = pick_kslice(s.d, (int64_t)s.E * 2 * (s.ffn / 128));
            L.ks_down = pick_kslice(s.ffn, (int64_t)s.E * (s.d / 128));
            L.S_up = s.d / L.ks_up;
            L.S_down = s.ffn / L.ks_down;
            L.part_up = off;
            off = align_up(off + (size_t)L.S_up * 2 * R * s.ffn * 4, kAlign);
            L.part_down = off;
            off = align_up(off + (size_t)L.S_down * R * s.d * 4, kAlign);
        } else if (L.path == 1) {
            // the unit counters of the CTA-pair kernels (up, down), on separate lines
            L.sched = off;
            off = align_up(off + 256, kAlign);
            // the down projection's per-unit completion counts (combine fused in)
            L.done = off;
            off = align_up(off + (size_t)((R + 255) / 256 + s.E) * (s.d / 256) * sizeof(int), kAlign);
        }
    }
    L.total = off;
    return L;
}

struct FwdLayout {
    size_t idx, w, logits, counts, offsets, perm_token, slot_row, perm_w, perm_ws, x_perm, y_slot, ffn, total;
    FfnLayout f;
};

FwdLayout fwd_layout(const moe_shape& s) {
    FwdLayout L;
    const size_t T = (size_t)s.T, R = 2 * T, E = (size_t)s.E;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, kAlign);
        return at;
    };
    L.idx = take(R * 4);
    L.w = take(R * 4);
    L.logits = take(T * E * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.perm_token = take(R * 4);
    L.slot_row = take(R * 4);
    L.perm_w = take(R * 4);
    L.perm_ws = take(permute_ws_bytes(s));
    L.x_perm = take(R * s.d * esize(s));
    L.y_slot = take(R * s.d * 4);
    L.f = ffn_layout(s);
    L.ffn = take(L.f.total);
    L.total = off;
    return L;
}

// --------------------------------------------------------------- stages
moe_status run_router(const moe_shape& s, const void* x, const void* wg, int32_t* idx, float* w, float* logits,
                      cudaStream_t st) {
    if (s.T == 0) return MOE_OK;
    const size_t es = esize(s);
    const size_t wbytes = (size_t)s.E * s.d * es;
    const int use_smem = wbytes <= 200 * 1024 ? 1 : 0;
    const int V = (int)(16 / es);
    const int vec = (s.d % V == 0 && aligned16(x) && aligned16(wg)) ? 1 : 0;
    const int64_t blocks = (s.T + kRouterWarps * kRouterTokensPerWarp - 1) / (kRouterWarps * kRouterTokensPerWarp);
    // as many CTAs as fit at once (W_g staged in shared memory limits them)
    // (126 registers x 256 threads: two CTAs per SM)
    const int per_sm = use_smem ? (int)std::max<size_t>(1, std::min<size_t>(2, (200 * 1024) / std::max<size_t>(1, wbytes))) : 2;
    const int grid = (int)std::min<int64_t>(blocks, (int64_t)sm_count() * per_sm);
    const size_t smem = use_smem ? wbytes : 0;
    if (vec && s.T <= kRouterSplitMaxTokens) {
        // small batch: one CTA per token, the model dimension split over 8 warps
        const int sgrid = (int)s.T;
        if (s.dtype == MOE_BF16)
            return launch("router_top2", st, [&] {
                return klaunch(router_top2_split_kernel<__nv_bfloat16>, sgrid, kRouterWarps * 32, 0, st, 
                    static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(wg), s.T, s.d, s.E, idx,
                    w, logits);
            });
        return launch("router_top2", st, [&] {
            return klaunch(router_top2_split_kernel<float>, sgrid, kRouterWarps * 32, 0, st, 
                static_cast<const float*>(x), static_cast<const float*>(wg), s.T, s.d, s.E, idx, w, logits);
        });
    }
    if (s.dtype == MOE_BF16 && vec && s.d % kBK == 0 && g.router_tc) {
        // tensor cores: 128-token tiles, one CTA per SM
        CUtensorMap mx, mw;
        if (!make_map(&mx, x, (uint64_t)s.d, (uint64_t)s.T, kRtM) || !make_map(&mw, wg, (uint64_t)s.d, (uint64_t)s.E, 8))
            return MOE_ERR_CUDA;
        if (!ensure_smem(router_tc_kernel, 25, kRtSmemBytes)) return MOE_ERR_CUDA;
        const int tiles = (int)((s.T + kRtM - 1) / kRtM);
        const int tgrid = std::max(1, std::min(tiles, sm_count()));
        return launch("router_top2", st, [&] {
            return klaunch(router_tc_kernel, tgrid, kRtThreads, kRtSmemBytes, st, mx, mw, s.T, s.d, s.E,
                           g.timeout_ns, idx, w, logits);
        });
    }
    if (s.dtype == MOE_BF16) {
        if (!ensure_smem(router_top2_kernel<__nv_bfloat16>, 0, 200 * 1024)) return MOE_ERR_CUDA;
        return launch("router_top2", st, [&] {
            return klaunch(router_top2_kernel<__nv_bfloat16>, grid, kRouterWarps * 32, smem, st, 
                static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(wg), s.T, s.d, s.E,
                use_smem, vec, idx, w, logits);
        });
    }
    if (!ensure_smem(router_top2_kernel<float>, 1, 200 * 1024)) return MOE_ERR_CUDA;
    return launch("router_top2", st, [&] {
        return klaunch(router_top2_kernel<float>, grid, kRouterWarps * 32, smem, st, 
            static_cast<const float*>(x), static_cast<const float*>(wg), s.T, s.d, s.E, use_smem, vec, idx, w,
            logits);
    });
}

moe_status run_permute(const moe_shape& s, const int32_t* idx, const float* w, const void* x, int32_t* counts,
                       int32_t* offsets, int32_t* perm_token, int32_t* slot_row, float* perm_w, void* x_perm,
                       void* ws, size_t ws_bytes, cudaStream_t st) {
    const int64_t R = 2 * s.T;
    const int64_t row_bytes = (int64_t)s.d * esize(s);
    const bool rows16 = row_bytes % 16 == 0 && aligned16(x) && aligned16(x_perm);
    if (s.T >= kPermuteMultiMinTokens && ws != nullptr && ws_bytes >= permute_ws_bytes(s)) {
        // large batch: per-chunk counts, then ranks + rows + row copies on many CTAs
        const int64_t chunk = permute_chunk(s.T);
        const int nchunks = (int)((s.T + chunk - 1) / chunk);
        int32_t* chunk_counts = static_cast<int32_t*>(ws);
        MOE_TRY(launch("permute_count", st, [&] {
            return klaunch(permute_count_kernel, nchunks, kPlaceThreads, 0, st, idx, s.T, s.E, chunk, chunk_counts);
        }));
        MOE_TRY(launch("permute_place", st, [&] {
            return klaunch(permute_place_kernel, nchunks, kPlaceThreads, 0, st, idx, w, s.T, s.E, chunk, nchunks,
                           static_cast<const int32_t*>(chunk_counts), counts, offsets, perm_token, slot_row, perm_w,
                           rows16 ? static_cast<const unsigned char*>(x) : nullptr, row_bytes,
                           static_cast<unsigned char*>(x_perm));
        }));
        if (rows16) return MOE_OK;
    } else if (s.T > 0 && R <= kSmallPermuteMaxSlots && rows16) {
        // small batch: every CTA ranks all slots, CTA 0 writes the grouping,
        // the grid copies the rows
        const int64_t chunks = R * (row_bytes / 16);
        const int grid = (int)std::max<int64_t>(
            1, std::min<int64_t>((chunks + 2 * kSmallPermuteThreads - 1) / (2 * kSmallPermuteThreads), sm_count()));
        return launch("permute", st, [&] {
            return klaunch(permute_small_kernel, grid, kSmallPermuteThreads, 0, st, idx, w, s.T, s.E, counts,
                           offsets, perm_token, slot_row, perm_w, static_cast<const unsigned char*>(x), row_bytes,
                           static_cast<unsigned char*>(x_perm));
        });
    } else {
        // one CTA; it also copies the rows when they are few
        const bool fused = s.T > 0 && rows16 && R * row_bytes <= kFusedGatherBytes;
        MOE_TRY(launch("permute", st, [&] {
            return klaunch(permute_kernel, 1, kPermuteThreads, 0, st, idx, w, s.T, s.E, counts, offsets, perm_token,
                           slot_row, perm_w, fused ? static_cast<const unsigned char*>(x) : nullptr, row_bytes,
                           static_cast<unsigned char*>(x_perm));
        }));
        if (s.T == 0 || fused) return MOE_OK;
    }
    const int grid = (int)std::min<int64_t>(R, (int64_t)sm_count() * 8);
    return launch("gather_rows", st, [&] {
        return klaunch(gather_rows_kernel, grid, 256, 0, st, static_cast<const unsigned char*>(x), perm_token,
                       offsets, s.E, R, row_bytes, static_cast<unsigned char*>(x_perm));
    });
}

int tc_grid(int64_t work_upper) {
    const int sms = g.grid > 0 ? g.grid : sm_count();
    return (int)std::max<int64_t>(1, std::min<int64_t>(work_upper, sms));
}

// Clusters of `cluster` CTAs (CTA pairs: 2) of a kernel that fit on the GPU
// at once (queried once per device and slot); -1 if none fits.
template <typename K>
int pair_capacity(K kernel, size_t smem, int slot, int cluster = 2) {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return -1;
    int& cap = g.pair_cap[dev][slot];
    if (cap == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cluster * (sm_count() / cluster));
        cfg.blockDim = dim3(kPairThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = -1;
        }
        cap = n;
    }
    return cap;
}

// Grid of a persistent CTA-pair kernel: an even number of CTAs.
int pair_grid(int64_t pairs_upper, int cap) {
    int pairs = g.grid > 0 ? std::max(1, g.grid / 2) : cap;
    pairs = (int)std::max<int64_t>(1, std::min<int64_t>(pairs_upper, pairs));
    return 2 * pairs;
}

// Both expert GEMMs on CTA-pair token tiles.
// MOE_ERR_UNSUPPORTED (nothing enqueued) when the kernels do not fit.
moe_status run_pair_ffn(const moe_shape& s, const void* x_perm, const int32_t* offsets, const float* perm_w,
                        const void* w1, const void* w3, const void* w2, float* y_slot, __nv_bfloat16* H,
                        __nv_bfloat16* u_out, __nv_bfloat16* v_out, int* sched, const int32_t* perm_token,
                        const int32_t* slot_row, __nv_bfloat16* y, int* done, cudaStream_t st) {
    const int64_t R = 2 * s.T;
    const int d = s.d, F = s.ffn, E = s.E;
    auto kup = tile_pair_gemm_kernel<PM_UP>;
    auto kdown = tile_pair_gemm_kernel<PM_DOWN>;
    const int slot = 6;
    const int cap_slot = 0;  // the backward kernels use slots 2-4
    const int cap_up = ensure_smem(kup, slot, kPairSmemBytes) ? pair_capacity(kup, kPairSmemBytes, cap_slot) : -1;
    const int cap_down =
        ensure_smem(kdown, slot + 1, kPairSmemBytes) ? pair_capacity(kdown, kPairSmemBytes, cap_slot + 1) : -1;
    if (cap_up <= 0 || cap_down <= 0) {
        cudaGetLastError();
        return MOE_ERR_UNSUPPORTED;
    }
    CUtensorMap ma, mb0, mb1, mb0h, mb1h;
    if (!make_map(&ma, x_perm, d, R, 128) || !make_map(&mb0, w1, d, (uint64_t)E * F, 128) ||
        !make_map(&mb1, w3, d, (uint64_t)E * F, 128) || !make_map(&mb0h, w1, d, (uint64_t)E * F, 64) ||
        !make_map(&mb1h, w3, d, (uint64_t)E * F, 64))
        return MOE_ERR_CUDA;
    TileArgs up{offsets, perm_w, H, E, d, F / kTileM, F, F, g.timeout_ns, u_out, v_out};
    const int64_t units_up = ((R + kPairM - 1) / kPairM + E) * (F / kTileM);
    const int grid_up = pair_grid(units_up, cap_up);
    if (y != nullptr) {
        up.zero_counts = done;
        up.n_zero_counts = (int)(((R + kPairM - 1) / kPairM + E) * (d / kTileN));
    }
    const int sched_bits = g.tile_sched;
    if (sched_bits & 3) {
        // the kernels claim their units from counters that start at zero
        if (cudaMemsetAsync(sched, 0, 256, st) != cudaSuccess) return MOE_ERR_CUDA;
        if (sched_bits & 1) up.sched = sched;
    }
    MOE_TRY(launch("tile_up_swiglu", st, [&] {
        return klaunch_cluster(kup, 2, grid_up, kPairThreads, kPairSmemBytes, st, ma, mb0, mb1, mb0h, mb1h, up);
    }));
    CUtensorMap mh, mw2;
    if (!make_map(&mh, H, F, R, 128) || !make_map(&mw2, w2, F, (uint64_t)E * d, 128)) return MOE_ERR_CUDA;
    TileArgs down{offsets, perm_w, y_slot, E, F, d / kTileN, d, d, g.timeout_ns};
    if (sched_bits & 2) down.sched = sched + 32;
    const int64_t units_down = ((R + kPairM - 1) / kPairM + E) * (d / kTileN);
    if (y != nullptr) {
        // the combine fused into the down projection's epilogue: per-unit completion counts, zeroed by
        // the up projection (launched above) so that no memset separates the two kernels
        down.perm_token = perm_token;
        down.slot_row = slot_row;
        down.y = y;
        down.done = done;
    }
    return launch("tile_down_scale", st, [&] {
        return klaunch_cluster(kdown, 2, pair_grid(units_down, cap_down), kPairThreads, kPairSmemBytes, st, mh, mw2,
                               mw2, mw2, mw2, down);
    });
}

// With slot_row and y given (the whole-layer call), the weight-streaming path
// finishes with the fused K-slice sum + gate scale + combine, and the CTA-pair
// path (given perm_token too) with the combine fused into the down
// projection, and both set *combined; otherwise the expert FFN writes y_slot.
moe_status run_ffn(const moe_shape& s, const void* x_perm, const int32_t* offsets, const float* perm_w,
                   const void* w1, const void* w3, const void* w2, float* y_slot, unsigned char* ws,
                   const FfnLayout& L, cudaStream_t st, const int32_t* slot_row = nullptr, void* y = nullptr,
                   bool* combined = nullptr, __nv_bfloat16* u_out = nullptr, __nv_bfloat16* v_out = nullptr,
                   const int32_t* perm_token = nullptr) {
    if (s.T == 0) return MOE_OK;
    const int64_t R = 2 * s.T;
    const int d = s.d, F = s.ffn, E = s.E;
    if (s.dtype == MOE_F32) {
        float* H = reinterpret_cast<float*>(ws + L.h);
        const int gy = (int)((R + kF32Tile - 1) / kF32Tile + E);
        MOE_TRY(launch("f32_up", st, [&] {
            return klaunch(f32_ffn_kernel<true>, dim3((F + kF32Tile - 1) / kF32Tile, gy), dim3(32, 8), 0, st, 
                static_cast<const float*>(x_perm), offsets, E, static_cast<const float*>(w1),
                static_cast<const float*>(w3), nullptr, d, F, H);
        }));
        return launch("f32_down", st, [&] {
            return klaunch(f32_ffn_kernel<false>, dim3((d + kF32Tile - 1) / kF32Tile, gy), dim3(32, 8), 0, st, 
                H, offsets, E, static_cast<const float*>(w2), nullptr, perm_w, F, d, y_slot);
        });
    }
    __nv_bfloat16* H = reinterpret_cast<__nv_bfloat16*>(ws + L.h);
    const int tile_ctas = g.tile_ctas != 0 ? g.tile_ctas : (s.T <= kSingleCtaMaxTokens ? 1 : 2);
    if (L.path == 1 && tile_ctas == 2) {
        // CTA pairs: each CTA stages 128 token rows and 128 weight rows per stage
        const bool fuse = perm_token != nullptr && slot_row != nullptr && y != nullptr && combined != nullptr &&
                          g.fuse_combine;
        const moe_status rc =
            run_pair_ffn(s, x_perm, offsets, perm_w, w1, w3, w2, y_slot, H, u_out, v_out,
                         reinterpret_cast<int*>(ws + L.sched), fuse ? perm_token : nullptr,
                         fuse ? slot_row : nullptr, fuse ? static_cast<__nv_bfloat16*>(y) : nullptr,
                         reinterpret_cast<int*>(ws + L.done), st);
        if (rc == MOE_OK && fuse) *combined = true;
        if (rc != MOE_ERR_UNSUPPORTED) return rc;
    }
    if (L.path == 1) {
        CUtensorMap ma, mb0, mb1;
        if (!make_map(&ma, x_perm, d, R, kTileM) || !make_map(&mb0, w1, d, (uint64_t)E * F, kTileM) ||
            !make_map(&mb1, w3, d, (uint64_t)E * F, kTileM))
            return MOE_ERR_CUDA;
        if (!ensure_smem(tile_gemm_kernel<true>, 2, kTileSmemBytes)) return MOE_ERR_CUDA;
        TileArgs up{offsets, perm_w, H, E, d, F / kTileM, F, F, g.timeout_ns, u_out, v_out};
        const int64_t tiles_up = ((R + kTileM - 1) / kTileM + E) * (F / kTileM);
        MOE_TRY(launch("tile_up_swiglu", st, [&] {
            return klaunch(tile_gemm_kernel<true>, tc_grid(tiles_up), kTcThreads, kTileSmemBytes, st, ma, mb0, mb1, up);
        }));
        CUtensorMap mh, mw2;
        if (!make_map(&mh, H, F, R, kTileM) || !make_map(&mw2, w2, F, (uint64_t)E * d, kTileN)) return MOE_ERR_CUDA;
        if (!ensure_smem(tile_gemm_kernel<false>, 3, kTileSmemBytes)) return MOE_ERR_CUDA;
        TileArgs down{offsets, perm_w, y_slot, E, F, d / kTileN, d, d, g.timeout_ns};
        const int64_t tiles_down = ((R + kTileM - 1) / kTileM + E) * (d / kTileN);
        return launch("tile_down_scale", st, [&] {
            return klaunch(tile_gemm_kernel<false>, tc_grid(tiles_down), kTcThreads, kTileSmemBytes, st, mh, mw2, mw2, down);
        });
    }
    if (L.path != 2) return MOE_ERR_UNSUPPORTED;
    float* part_up = reinterpret_cast<float*>(ws + L.part_up);
    float* part_down = reinterpret_cast<float*>(ws + L.part_down);
    const uint32_t stage_bytes = kStreamABytes + (uint32_t)align_up((size_t)L.nb * 128, 1024);
    // About 20 MB of weight tiles in flight over the whole GPU keep HBM busy;
    // measured on B300 at T = 16 and 64, more outstanding copies (12 stages on
    // every SM, 32 MB) cost 5-7 % of the streaming rate, fewer (6 stages) 3-5 %.
    const int grid_up = tc_grid((int64_t)E * 2 * (F / 128) * L.S_up);
    const int grid_down = tc_grid((int64_t)E * (d / 128) * L.S_down);
    auto stages_for = [&](int grid) {
        const size_t per_cta = kStreamInflightBytes / ((size_t)grid * kStreamABytes);
        const size_t fit = (kSmemBudget - 1024 - sizeof(TcControl)) / stage_bytes;
        return (int)std::max<size_t>(2, std::min<size_t>({per_cta, fit, (size_t)kMaxStreamStages}));
    };
    const int stages = stages_for(grid_up);
    const int stages_down = stages_for(grid_down);
    const size_t smem = stream_smem_bytes(L.nb, stages);
    const size_t smem_down = stream_smem_bytes(L.nb, stages_down);
    CUtensorMap mw1, mw3, mx;
    if (!make_map(&mw1, w1, d, (uint64_t)E * F, 128) || !make_map(&mw3, w3, d, (uint64_t)E * F, 128) ||
        !make_map(&mx, x_perm, d, R, L.nb))
        return MOE_ERR_CUDA;
    if (!ensure_smem(stream_gemm_kernel<true>, 4, kSmemBudget)) return MOE_ERR_CUDA;
    StreamArgs up{offsets, part_up, E, (int)R, L.ks_up, L.S_up, F / 128, 2, F, L.nb, stages, stage_bytes,
                  g.timeout_ns};
    up.keep_bytes = g.l2_keep_bytes / 3 * 2;  // W1 and W3 hold two thirds of an expert's bytes
    MOE_TRY(launch("stream_up", st, [&] {
        return klaunch(stream_gemm_kernel<true>, grid_up, kTcThreads, smem, st, mw1, mw3, mx, up);
    }));
    const int rgrid = (int)std::min<int64_t>((R * F + 255) / 256, (int64_t)sm_count() * 8);
    MOE_TRY(launch("reduce_swiglu", st, [&] {
        return klaunch(reduce_swiglu_kernel, rgrid, 256, 0, st, part_up, L.S_up, R, F, H, u_out, v_out);
    }));
    CUtensorMap mw2, mh;
    if (!make_map(&mw2, w2, F, (uint64_t)E * d, 128) || !make_map(&mh, H, F, R, L.nb)) return MOE_ERR_CUDA;
    if (!ensure_smem(stream_gemm_kernel<false>, 5, kSmemBudget)) return MOE_ERR_CUDA;
    StreamArgs down{offsets, part_down, E, (int)R, L.ks_down, L.S_down, d / 128, 1, d, L.nb, stages_down,
                    stage_bytes, g.timeout_ns};
    down.keep_bytes = g.l2_keep_bytes / 3;
    MOE_TRY(launch("stream_down", st, [&] {
        return klaunch(stream_gemm_kernel<false>, grid_down, kTcThreads, smem_down, st, mw2, mw2, mh, down);
    }));
    if (slot_row != nullptr && y != nullptr && combined != nullptr) {
        const int cgrid = (int)std::min<int64_t>((s.T * d + 255) / 256, (int64_t)sm_count() * 8);
        *combined = true;
        return launch("reduce_combine", st, [&] {
            return klaunch(reduce_combine_kernel<__nv_bfloat16>, cgrid, 256, 0, st, part_down, L.S_down, R, d,
                           perm_w, slot_row, s.T, static_cast<__nv_bfloat16*>(y));
        });
    }
    const int dgrid = (int)std::min<int64_t>((R * d + 255) / 256, (int64_t)sm_count() * 8);
    return launch("reduce_down", st, [&] {
        return klaunch(reduce_down_kernel, dgrid, 256, 0, st, part_down, L.S_down, R, d, perm_w, y_slot);
    });
}

moe_status run_combine(const moe_shape& s, const float* y_slot, const int32_t* slot_row, void* y,
                       cudaStream_t st) {
    if (s.T == 0) return MOE_OK;
    const bool v4 = (s.d % 4 == 0) && aligned16(y_slot) && aligned16(y);
    const int64_t n = v4 ? s.T * (s.d / 4) : s.T * s.d;
    const int grid = (int)std::min<int64_t>((n + 255) / 256, (int64_t)sm_count() * 8);
    if (s.dtype == MOE_BF16) {
        return launch("combine", st, [&] {
            if (v4)
                return klaunch(combine4_kernel<__nv_bfloat16>, grid, 256, 0, st, y_slot, slot_row, s.T, s.d,
                                                                     static_cast<__nv_bfloat16*>(y));
            else
                return klaunch(combine_kernel<__nv_bfloat16>, grid, 256, 0, st, y_slot, slot_row, s.T, s.d,
                                                                    static_cast<__nv_bfloat16*>(y));
        });
    }
    return launch("combine", st, [&] {
        if (v4)
            return klaunch(combine4_kernel<float>, grid, 256, 0, st, y_slot, slot_row, s.T, s.d, static_cast<float*>(y));
        else
            return klaunch(combine_kernel<float>, grid, 256, 0, st, y_slot, slot_row, s.T, s.d, static_cast<float*>(y));
    });
}

moe_status run_aux(const moe_shape& s, const float* logits, const int32_t* counts, float* f, float* P,
                   float* l_aux, cudaStream_t st) {
    if (s.T == 0) {
        if (cudaMemsetAsync(f, 0, sizeof(float) * s.E, st) != cudaSuccess ||
            cudaMemsetAsync(P, 0, sizeof(float) * s.E, st) != cudaSuccess ||
            cudaMemsetAsync(l_aux, 0, sizeof(float), st) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    return launch("aux_stats", st, [&] {
        return klaunch_cluster(aux_stats_kernel, kAuxCtas, kAuxCtas, kAuxThreads, 0, st, logits, counts, s.T, s.E, f,
                               P, l_aux);
    });
}

// ------------------------------------------------------------- training
// State kept by the training forward: the forward workspace (routing, grouping,
// x_perm, H, y_slot, scores) plus u = W1 x and v = W3 x per row (bf16).
struct TrainLayout {
    FwdLayout f;
    size_t u = 0, v = 0, total = 0;
};

TrainLayout train_layout(const moe_shape& s) {
    TrainLayout L;
    L.f = fwd_layout(s);
    const size_t uv = align_up((size_t)(2 * s.T) * s.ffn * 2, kAlign);
    L.u = L.f.total;
    L.v = L.u + uv;
    L.total = L.v + uv;
    return L;
}

// Workspace of the backward pass. dYs and dUV rows are in the padded group
// order (each expert's rows from a multiple of 64, zero rows between groups).
struct BwdLayout {
    size_t dg, dl, dys, duv, dxp, dwg, sched, total;
    int64_t rp;   // padded rows: 2T + 64 E, rounded up to 64
    int nchunks;  // token chunks of the router's weight gradient
};

BwdLayout bwd_layout(const moe_shape& s) {
    BwdLayout L;
    const size_t T = (size_t)s.T, R = 2 * T, E = (size_t)s.E, d = (size_t)s.d, F = (size_t)s.ffn;
    L.rp = (int64_t)align_up(R + (size_t)kBK * E, kBK);
    L.nchunks = (int)((T + kDwgChunk - 1) / kDwgChunk);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, kAlign);
        return at;
    };
    L.dg = take(R * 4);
    L.dl = take(T * E * 4);
    L.dys = take((size_t)L.rp * d * 2);
    L.duv = take((size_t)L.rp * 2 * F * 2);
    L.dxp = take(R * d * 4);
    L.dwg = take((size_t)std::max(L.nchunks, 1) * E * d * 4);
    L.sched = take(512);  // unit counters of the four CTA-pair GEMMs, on separate lines
    L.total = off;
    return L;
}

bool train_supported(const moe_shape& s) { return s.dtype == MOE_BF16 && s.d % 256 == 0 && s.ffn % 256 == 0; }

// One CTA-pair GEMM of the backward pass; MOE_ERR_UNSUPPORTED when no CTA pair fits.
template <int MODE>
moe_status launch_pair(const char* name, int slot, int cap_slot, const CUtensorMap& ma, const CUtensorMap& mb0,
                       const CUtensorMap& mb1, const TileArgs& a, int64_t pairs_upper, cudaStream_t st) {
    // the weight-gradient epilogue stages its stores in 4 warps' arrays after the control block
    const size_t smem = kPairSmemBytes + (MODE == PM_WGRAD ? kWgradStageBytes : 0);
    auto kern = tile_pair_gemm_kernel<MODE>;
    if (!ensure_smem(kern, slot, smem)) return MOE_ERR_CUDA;
    const int cap = pair_capacity(kern, smem, cap_slot);
    if (cap <= 0) return MOE_ERR_UNSUPPORTED;
    return launch(name, st, [&] {
        return klaunch_cluster(kern, 2, pair_grid(pairs_upper, cap), kPairThreads, smem, st, ma, mb0, mb1, mb0, mb1,
                               a);
    });
}

moe_status run_backward(const moe_shape& s, const __nv_bfloat16* x, const __nv_bfloat16* wg,
                        const __nv_bfloat16* w1, const __nv_bfloat16* w3, const __nv_bfloat16* w2,
                        const __nv_bfloat16* dy, float aux_coef, const unsigned char* state, __nv_bfloat16* dx,
                        float* dwg, float* dw1, float* dw3, float* dw2, unsigned char* ws, cudaStream_t st) {
    const TrainLayout TL = train_layout(s);
    const BwdLayout B = bwd_layout(s);
    const int64_t T = s.T, R = 2 * T;
    const int d = s.d, F = s.ffn, E = s.E;
    const int32_t* idx = reinterpret_cast<const int32_t*>(state + TL.f.idx);
    const float* gw = reinterpret_cast<const float*>(state + TL.f.w);
    const float* logits = reinterpret_cast<const float*>(state + TL.f.logits);
    const int32_t* counts = reinterpret_cast<const int32_t*>(state + TL.f.counts);
    const int32_t* offsets = reinterpret_cast<const int32_t*>(state + TL.f.offsets);
    const int32_t* perm_token = reinterpret_cast<const int32_t*>(state + TL.f.perm_token);
    const int32_t* slot_row = reinterpret_cast<const int32_t*>(state + TL.f.slot_row);
    const float* perm_w = reinterpret_cast<const float*>(state + TL.f.perm_w);
    const __nv_bfloat16* x_perm = reinterpret_cast<const __nv_bfloat16*>(state + TL.f.x_perm);
    const float* y_slot = reinterpret_cast<const float*>(state + TL.f.y_slot);
    const __nv_bfloat16* H = reinterpret_cast<const __nv_bfloat16*>(state + TL.f.ffn + TL.f.f.h);
    const __nv_bfloat16* U = reinterpret_cast<const __nv_bfloat16*>(state + TL.u);
    const __nv_bfloat16* V = reinterpret_cast<const __nv_bfloat16*>(state + TL.v);
    float* dg = reinterpret_cast<float*>(ws + B.dg);
    float* dl = reinterpret_cast<float*>(ws + B.dl);
    __nv_bfloat16* dys = reinterpret_cast<__nv_bfloat16*>(ws + B.dys);
    __nv_bfloat16* duv = reinterpret_cast<__nv_bfloat16*>(ws + B.duv);
    float* dxp = reinterpret_cast<float*>(ws + B.dxp);
    float* part = reinterpret_cast<float*>(ws + B.dwg);
    const int sms = sm_count();
    int* sched = (g.tile_sched & 4) ? reinterpret_cast<int*>(ws + B.sched) : nullptr;
    if (sched != nullptr && cudaMemsetAsync(sched, 0, 512, st) != cudaSuccess) return MOE_ERR_CUDA;

    // per slot: dYs = g dy (padded order, pad rows of dYs and dUV zeroed),
    // dg = <dy, E(x)>; per token: the scores' gradient
    MOE_TRY(launch("bwd_slot", st, [&] {
        return klaunch(bwd_slot_kernel, (int)std::max<int64_t>(1, std::min<int64_t>((B.rp + 7) / 8, (int64_t)sms * 8)),
                       256, 0, st, dy, y_slot, perm_token, perm_w, offsets, E, d, F, B.rp, dys, duv, dg);
    }));
    MOE_TRY(launch("bwd_router", st, [&] {
        return klaunch(bwd_router_kernel, (int)std::min<int64_t>((T + 255) / 256, (int64_t)sms * 4), 256, 0, st, idx,
                       gw, slot_row, dg, logits, counts, T, E, aux_coef, dl);
    }));
    // dh = dYs W2 (W2 read as stored), then du, dv with the kept u, v
    const int64_t token_tiles = (R + kPairM - 1) / kPairM + E;
    CUtensorMap ma, mb0, mb1;
    if (!make_map(&ma, dys, d, (uint64_t)B.rp, 128) || !make_map(&mb0, w2, F, (uint64_t)E * d, 64))
        return MOE_ERR_CUDA;
    TileArgs a_dh{offsets, nullptr, duv, E, d, F / kTileN, d, 2 * F, g.timeout_ns};
    a_dh.u_in = U;
    a_dh.v_in = V;
    if (sched != nullptr) a_dh.sched = sched;
    MOE_TRY(launch_pair<PM_BWD_DH>("bwd_dh_swiglu", 8, 2, ma, mb0, mb0, a_dh, token_tiles * (F / kTileN), st));
    // dXp = [du dv] [W1; W3] (W1, W3 read as stored)
    if (!make_map(&ma, duv, 2 * F, (uint64_t)B.rp, 128) || !make_map(&mb0, w1, d, (uint64_t)E * F, 64) ||
        !make_map(&mb1, w3, d, (uint64_t)E * F, 64))
        return MOE_ERR_CUDA;
    TileArgs a_dx{offsets, nullptr, dxp, E, 2 * F, d / kTileN, F, d, g.timeout_ns};
    if (sched != nullptr) a_dx.sched = sched + 32;
    MOE_TRY(launch_pair<PM_BWD_DX>("bwd_dx", 9, 3, ma, mb0, mb1, a_dx, token_tiles * (d / kTileN), st));
    // dx = both slots + the router's part
    MOE_TRY(launch("bwd_combine", st, [&] {
        return klaunch(bwd_combine_kernel, (int)std::min<int64_t>((T * (d / 4) + 255) / 256, (int64_t)sms * 8), 256, 0,
                       st, dxp, slot_row, dl, wg, T, d, E, dx);
    }));
    // dW_g = dl^T x
    MOE_TRY(launch("bwd_dwg", st, [&] {
        return klaunch(dwg_partial_kernel, dim3(B.nchunks, (d + 255) / 256), 256, 0, st, dl, x, T, d, E, part);
    }));
    MOE_TRY(launch("bwd_dwg", st, [&] {
        return klaunch(dwg_final_kernel, (int)std::min<int64_t>(((int64_t)E * d + 255) / 256, (int64_t)sms * 4), 256,
                       0, st, part, B.nchunks, d, E, dwg);
    }));
    // dW2[e] = dYs_e^T H_e, both read as stored (token rows)
    if (!make_map(&ma, dys, d, (uint64_t)B.rp, 64) || !make_map(&mb0, H, F, R, 64)) return MOE_ERR_CUDA;
    TileArgs a_w2{offsets, nullptr, dw2, E, 0, F / kTileN, 0, F, g.timeout_ns};
    a_w2.m_tiles = d / kPairM;
    a_w2.split_rows = d;
    a_w2.out_estride = (int64_t)d * F;
    if (sched != nullptr) a_w2.sched = sched + 64;
    MOE_TRY(launch_pair<PM_WGRAD>("bwd_dw2", 10, 4, ma, mb0, mb0, a_w2, (int64_t)E * (d / kPairM) * (F / kTileN), st));
    // [dW1; dW3][e] = [du dv]_e^T Xp_e
    if (!make_map(&ma, duv, 2 * (uint64_t)F, (uint64_t)B.rp, 64) || !make_map(&mb0, x_perm, d, R, 64))
        return MOE_ERR_CUDA;
    TileArgs a_w13{offsets, nullptr, dw1, E, 0, d / kTileN, 0, d, g.timeout_ns};
    a_w13.out2 = dw3;
    a_w13.m_tiles = 2 * F / kPairM;
    a_w13.split_rows = F;
    a_w13.out_estride = (int64_t)F * d;
    // [du dv] (2 ffn columns per token) is the larger operand: column tiles fastest, so each of its
    // 256-column blocks is shared by the tiles running at one time and x_perm (d columns) stays in L2
    // (DRAM reads per launch at T = 4096: 4.07 GB row tiles fastest, 0.55 GB column tiles fastest)
    a_w13.n_fast = 1;
    if (sched != nullptr) a_w13.sched = sched + 96;
    return launch_pair<PM_WGRAD>("bwd_dw13", 10, 4, ma, mb0, mb0, a_w13,
                                 (int64_t)E * (2 * F / kPairM) * (d / kTileN), st);
}

// Scratch of moe_layer_forward_noalloc: a fixed array of static device memory,
// one copy per device that loads the library, held until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(24) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device. The array's name
// is only a host-side stand-in in host code, so its address is looked up once
// per device (with that device current) and cached. Host threads that make
// their first call on one device at the same time may both look it up; they
// store the same value, and the atomic slots keep that well defined.
void* noalloc_scratch() {
    static std::atomic<void*> addr[kMaxDevices];
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    void* p = addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
        addr[dev].store(p, std::memory_order_release);
    }
    return p;
}

// ------------------------------------------------------------ decoder block
moe_status check_block_shape(const moe_block_shape* s) {
    if (s == nullptr) return MOE_ERR_INVALID_ARG;
    if (s->B < 1 || s->S < 1 || s->d <= 0 || s->n_heads <= 0 || s->n_kv_heads <= 0 || s->head_dim <= 0 ||
        s->ffn <= 0 || !(s->eps >= 0.f) || !std::isfinite(s->eps) || !(s->rope_base > 0.f) ||
        !std::isfinite(s->rope_base))
        return MOE_ERR_INVALID_ARG;
    if (s->n_heads % s->n_kv_heads != 0 || s->cache_max < 0) return MOE_ERR_INVALID_ARG;
    if (s->head_dim != kAttnHD || s->d % 256 != 0 || s->ffn % 256 != 0 || s->E != 8 || s->k != 2)
        return MOE_ERR_UNSUPPORTED;
    // the fused projection runs on 256-column tiles
    if ((int64_t)(s->n_heads + 2 * s->n_kv_heads) * s->head_dim % 256 != 0) return MOE_ERR_UNSUPPORTED;
    if (s->B > (int64_t)INT32_MAX / s->S) return MOE_ERR_UNSUPPORTED;  // TMA row coordinates are int32
    return MOE_OK;
}

moe_shape block_layer_shape(const moe_block_shape& s) {
    moe_shape m;
    m.T = s.B * s.S;
    m.d = s.d;
    m.ffn = s.ffn;
    m.E = s.E;
    m.k = s.k;
    m.dtype = MOE_BF16;
    return m;
}

struct BlockLayout {
    size_t xn, qkv, q, k, v, attn, h, y, moe, total;
};

// xn (later the second norm's output), qkv (later Wo's fp32 output), q, k, v,
// attention output, residual stream h, MoE output y, the MoE layer's workspace
BlockLayout block_layout(const moe_block_shape& s) {
    const size_t T = (size_t)(s.B * s.S), d = (size_t)s.d;
    const size_t wq = (size_t)s.n_heads * s.head_dim, wkv = (size_t)s.n_kv_heads * s.head_dim;
    BlockLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, kAlign);
        return at;
    };
    L.xn = take(T * d * 2);
    L.qkv = take(T * std::max(wq + 2 * wkv, d) * 4);
    L.q = take(T * wq * 2);
    L.k = take(T * wkv * 2);
    L.v = take(T * wkv * 2);
    L.attn = take(T * wq * 2);
    L.h = take(T * d * 2);
    L.y = take(T * d * 2);
    const moe_shape m = block_layer_shape(s);
    L.moe = take(std::max<size_t>(moe_workspace_bytes(&m), 16));
    L.total = off;
    return L;
}

moe_status run_rmsnorm(int64_t rows, int d, const void* x, const float* add, const void* gain, float eps, void* h_out,
                       void* y, cudaStream_t st) {
    if (rows == 0) return MOE_OK;
    const int64_t blocks_needed = (rows + kNormThreads / 32 - 1) / (kNormThreads / 32);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(blocks_needed, (int64_t)sm_count() * 8));
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const auto* gb = static_cast<const __nv_bfloat16*>(gain);
    auto* hb = static_cast<__nv_bfloat16*>(h_out);
    auto* yb = static_cast<__nv_bfloat16*>(y);
    if (add != nullptr)
        return launch("rmsnorm_add", st, [&] {
            return klaunch(rmsnorm_kernel<true>, grid, kNormThreads, 0, st, xb, add, gb, eps, rows, d, hb, yb);
        });
    return launch("rmsnorm", st, [&] {
        return klaunch(rmsnorm_kernel<false>, grid, kNormThreads, 0, st, xb, add, gb, eps, rows, d, hb, yb);
    });
}

// Weight streaming for a linear layer of few rows (<= 64, a decode batch):
// the streaming kernel's M side is 128 weight rows and its N side the rows of
// x, K split into slices so that the units fill the GPU; fp32 partials per
// slice, summed in slice order.
struct LinearStreamPlan {
    int ks = 0, S = 0, nb = 0;
    size_t part_bytes = 0;
};

LinearStreamPlan linear_stream_plan(int64_t rows, int n_in, int n_out) {
    LinearStreamPlan L;
    if (rows < 1 || rows > kStreamMaxTokens || n_out % 128 != 0) return L;
    const int64_t rb = n_out / 128, grid = sm_count();
    double best_fill = -1.0;
    // the largest slice (256 .. 2048, dividing n_in) whose units fill the last wave best
    for (int ks = 256; ks <= 2048 && ks <= n_in; ks += kBK) {
        if (n_in % ks != 0) continue;
        const double waves = (double)(rb * (n_in / ks)) / (double)grid;
        const double fill = waves / std::ceil(waves);
        if (fill >= best_fill - 1e-9) {
            best_fill = fill;
            L.ks = ks;
        }
    }
    if (L.ks == 0) L.ks = n_in;  // n_in < 256: one slice
    L.S = n_in / L.ks;
    L.nb = (int)align_up((size_t)rows, 16);
    L.part_bytes = align_up((size_t)L.S * (size_t)rows * (size_t)n_out * 4, kAlign);
    return L;
}

moe_status run_linear(int64_t rows, int n_in, int n_out, const void* x, const void* w, float* y, cudaStream_t st,
                      const char* name = "linear", unsigned char* ws = nullptr, size_t ws_bytes = 0) {
    if (rows == 0) return MOE_OK;
    const LinearStreamPlan P = linear_stream_plan(rows, n_in, n_out);
    if (P.S > 0 && ws != nullptr && ws_bytes >= P.part_bytes) {
        float* part = reinterpret_cast<float*>(ws);
        const uint32_t stage_bytes = kStreamABytes + (uint32_t)align_up((size_t)P.nb * 128, 1024);
        const int grid = tc_grid((int64_t)(n_out / 128) * P.S);
        const size_t per_cta = kStreamInflightBytes / ((size_t)grid * kStreamABytes);
        const size_t fit = (kSmemBudget - 1024 - sizeof(TcControl)) / stage_bytes;
        const int stages = (int)std::max<size_t>(2, std::min<size_t>({per_cta, fit, (size_t)kMaxStreamStages}));
        CUtensorMap mw, mx;
        if (!make_map(&mw, w, (uint64_t)n_in, (uint64_t)n_out, 128) ||
            !make_map(&mx, x, (uint64_t)n_in, (uint64_t)rows, (uint32_t)P.nb))
            return MOE_ERR_CUDA;
        if (!ensure_smem(stream_gemm_kernel<false>, 5, kSmemBudget)) return MOE_ERR_CUDA;
        StreamArgs a{nullptr, part, 1, (int)rows, P.ks, P.S, n_out / 128, 1, n_out, P.nb, stages, stage_bytes,
                     g.timeout_ns};
        a.dense_rows = (int)rows;
        MOE_TRY(launch(name, st, [&] {
            return klaunch(stream_gemm_kernel<false>, grid, kTcThreads, stream_smem_bytes(P.nb, stages), st, mw, mw,
                           mx, a);
        }));
        const int rgrid = (int)std::min<int64_t>((rows * n_out + 255) / 256, (int64_t)sm_count() * 8);
        return launch("linear_reduce", st, [&] {
            return klaunch(reduce_down_kernel, rgrid, 256, 0, st, part, P.S, rows, n_out, (const float*)nullptr, y);
        });
    }
    CUtensorMap ma, mb;
    if (!make_map(&ma, x, (uint64_t)n_in, (uint64_t)rows, 128) || !make_map(&mb, w, (uint64_t)n_in, (uint64_t)n_out, 128))
        return MOE_ERR_CUDA;
    TileArgs a{nullptr, nullptr, y, 1, n_in, n_out / kTileN, n_out, n_out, g.timeout_ns};
    a.dense_rows = (int)rows;
    const int64_t units = (rows + kPairM - 1) / kPairM * (n_out / kTileN);
    // the same kernel (and attribute slots) as the expert FFN's down projection
    return launch_pair<PM_DOWN>(name, 7, 1, ma, mb, mb, a, units, st);
}

moe_status run_rope(const moe_block_shape& s, const float* qkv, void* q, void* k, void* v, cudaStream_t st,
                    const int32_t* pos = nullptr, void* k_cache = nullptr, void* v_cache = nullptr) {
    const int64_t T = s.B * s.S;
    if (T == 0) return MOE_OK;
    RopeArgs a{};
    a.qkv = qkv;
    a.q = static_cast<__nv_bfloat16*>(q);
    a.k = static_cast<__nv_bfloat16*>(k);
    a.v = static_cast<__nv_bfloat16*>(v);
    a.T = T;
    a.S = s.S;
    a.pos = pos;
    a.k_cache = static_cast<__nv_bfloat16*>(k_cache);
    a.v_cache = static_cast<__nv_bfloat16*>(v_cache);
    a.cache_max = s.cache_max;
    a.Hq = s.n_heads;
    a.Hkv = s.n_kv_heads;
    a.hd = s.head_dim;
    for (int i = 0; i < s.head_dim / 2; ++i)
        a.theta[i] = std::pow((double)s.rope_base, -2.0 * (double)i / (double)s.head_dim);
    const dim3 block(s.head_dim / 2, kRopeTokens);
    const int64_t grid = (T + kRopeTokens - 1) / kRopeTokens;
    return launch("rope_split", st, [&] { return klaunch(rope_split_kernel, dim3((unsigned)grid), block, 0, st, a); });
}

moe_status run_attention(const moe_block_shape& s, const void* q, const void* k, const void* v, void* o,
                         cudaStream_t st) {
    const int64_t T = s.B * s.S;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, (uint64_t)s.n_heads * kAttnHD, (uint64_t)T, 128) ||
        !make_map(&mk, k, (uint64_t)s.n_kv_heads * kAttnHD, (uint64_t)T, 128) ||
        !make_map(&mv, v, (uint64_t)s.n_kv_heads * kAttnHD, (uint64_t)T, 128))
        return MOE_ERR_CUDA;
    AttnArgs a{};
    a.o = static_cast<__nv_bfloat16*>(o);
    a.S = s.S;
    a.B = (int)s.B;
    a.Hq = s.n_heads;
    a.Hkv = s.n_kv_heads;
    a.n_qt = (int)((s.S + kAttnTile - 1) / kAttnTile);
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.head_dim));
    a.timeout_ns = g.timeout_ns;
    // heads of an even GQA group go two per CTA and share their K and V tiles
    const bool paired = (s.n_heads / s.n_kv_heads) % 2 == 0;
    const int64_t grid = (int64_t)a.n_qt * s.B * (paired ? s.n_heads / 2 : s.n_heads);
    if (grid > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    if (paired) {
        if (!ensure_smem(attention_pair_kernel, 14, kAttnPairSmemBytes)) return MOE_ERR_CUDA;
        return launch("attention", st, [&] {
            return klaunch(attention_pair_kernel, dim3((unsigned)grid), dim3(kAttnPairThreads), kAttnPairSmemBytes, st,
                           mq, mk, mv, a);
        });
    }
    if (!ensure_smem(attention_kernel, 11, kAttnSmemBytes)) return MOE_ERR_CUDA;
    return launch("attention", st, [&] {
        return klaunch(attention_kernel, dim3((unsigned)grid), dim3(kAttnThreads), kAttnSmemBytes, st, mq, mk, mv, a);
    });
}

// CTAs per (sequence, KV head) of the decode attention: enough that the grid fills every SM
// with kDecCtasPerSm CTAs once, but no more splits than chunks of the cache.
int decode_splits(const moe_block_shape& s) {
    const int64_t pairs = std::max<int64_t>(1, s.B * s.n_kv_heads);
    const int64_t want = std::max<int64_t>(1, (int64_t)kDecCtasPerSm * sm_count() / pairs);
    const int64_t chunks = (s.cache_max + kDecChunk - 1) / kDecChunk;
    return (int)std::max<int64_t>(1, std::min<int64_t>(want, chunks));
}

size_t decode_attention_ws_bytes(const moe_block_shape& s) {
    const size_t parts = (size_t)s.B * s.n_heads * decode_splits(s);
    return align_up(parts * kAttnHD * 4, kAlign) + align_up(parts * 2 * 4, kAlign);
}

bool decode_supported(const moe_block_shape& s) {
    const int group = s.n_heads / s.n_kv_heads;
    return s.S == 1 && s.cache_max >= 1 && group <= kDecMaxGroup && s.B <= 65535 && s.n_kv_heads <= 65535 &&
           s.B * s.n_kv_heads * s.cache_max <= INT32_MAX && s.B * s.n_heads <= INT32_MAX;
}

moe_status run_attention_decode(const moe_block_shape& s, const void* q, const void* kc, const void* vc,
                                int32_t* len, void* o, unsigned char* ws, cudaStream_t st) {
    const int splits = decode_splits(s);
    const size_t parts = (size_t)s.B * s.n_heads * splits;
    const int group = s.n_heads / s.n_kv_heads;
    CUtensorMap mk, mv;
    const uint64_t cache_rows = (uint64_t)s.B * s.n_kv_heads * s.cache_max;
    if (!make_map(&mk, kc, kAttnHD, cache_rows, kDecChunk) || !make_map(&mv, vc, kAttnHD, cache_rows, kDecChunk))
        return MOE_ERR_CUDA;
    DecodeArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.len = len;
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_ml = reinterpret_cast<float*>(ws + align_up(parts * kAttnHD * 4, kAlign));
    a.cache_max = s.cache_max;
    a.Hq = s.n_heads;
    a.Hkv = s.n_kv_heads;
    a.splits = splits;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.head_dim));
    a.timeout_ns = g.timeout_ns;
    // the softmax's per-head loops are unrolled for the group size rounded up to a power of two
    const int gp = group <= 1 ? 1 : group <= 2 ? 2 : group <= 4 ? 4 : group <= 8 ? 8 : 16;
    auto kern = gp == 1 ? attention_decode_kernel<1>
                : gp == 2 ? attention_decode_kernel<2>
                : gp == 4 ? attention_decode_kernel<4>
                : gp == 8 ? attention_decode_kernel<8>
                          : attention_decode_kernel<16>;
    const int slot = gp == 1 ? 20 : gp == 2 ? 21 : gp == 4 ? 22 : gp == 8 ? 23 : 24;
    if (!ensure_smem(kern, slot, kDecSmemBytes)) return MOE_ERR_CUDA;
    MOE_TRY(launch("attention_decode", st, [&] {
        return klaunch(kern, dim3((unsigned)splits, (unsigned)s.n_kv_heads, (unsigned)s.B), dim3(kDecThreads),
                       kDecSmemBytes, st, mk, mv, a);
    }));
    return launch("attention_decode_merge", st, [&] {
        return klaunch(attention_decode_merge_kernel, dim3((unsigned)s.n_heads, (unsigned)s.B), dim3(kAttnHD), 0, st,
                       (const float*)a.part_o, (const float*)a.part_ml, s.n_heads, splits, len, s.cache_max,
                       static_cast<__nv_bfloat16*>(o));
    });
}

struct DecodeLayout {
    size_t xn, qkv, q, attn, h, y, lin, att, moe, total;
    size_t lin_bytes;
};

// One decode step's buffers: xn [B][d] (later the second norm's output), the
// projection output [B][max((Hq+2Hkv) hd, d)] fp32 (later Wo's), q and the
// attention output [B][Hq hd], h and y [B][d], the linear layers' K-slice
// partials, the attention partials, the MoE layer's workspace.
DecodeLayout decode_layout(const moe_block_shape& s) {
    const size_t B = (size_t)s.B, d = (size_t)s.d;
    const size_t wq = (size_t)s.n_heads * s.head_dim, wqkv = wq + 2 * (size_t)s.n_kv_heads * s.head_dim;
    DecodeLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, kAlign);
        return at;
    };
    L.xn = take(B * d * 2);
    L.qkv = take(B * std::max(wqkv, d) * 4);
    L.q = take(B * wq * 2);
    L.attn = take(B * wq * 2);
    L.h = take(B * d * 2);
    L.y = take(B * d * 2);
    L.lin_bytes = std::max(linear_stream_plan(s.B, s.d, (int)wqkv).part_bytes,
                           linear_stream_plan(s.B, (int)wq, s.d).part_bytes);
    L.lin = take(std::max<size_t>(L.lin_bytes, 16));
    L.att = take(decode_attention_ws_bytes(s));
    const moe_shape m = block_layer_shape(s);
    L.moe = take(std::max<size_t>(moe_workspace_bytes(&m), 16));
    L.total = off;
    return L;
}

moe_status run_residual_add(int64_t n, const void* a, const void* b, void* out, cudaStream_t st) {
    if (n == 0) return MOE_OK;
    const int64_t chunks = n / 8;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((chunks + 255) / 256, (int64_t)sm_count() * 8));
    return launch("residual_add", st, [&] {
        return klaunch(residual_add_kernel, grid, 256, 0, st, static_cast<const __nv_bfloat16*>(a),
                       static_cast<const __nv_bfloat16*>(b), n, static_cast<__nv_bfloat16*>(out));
    });
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_version(void) { return "moe-b300 0.1 (sm_103a)"; }

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "device wait timed out";
        case MOE_ERR_DEVICE_CHECK: return "device index check failed";
    }
    return "unknown status";
}

size_t moe_workspace_bytes(const moe_shape* s) {
    if (check_shape(s) != MOE_OK) return 0;
    if (s->dtype == MOE_BF16 && choose_path(*s) == 0) return 0;
    return fwd_layout(*s).total;
}

size_t moe_ffn_workspace_bytes(const moe_shape* s) {
    if (check_ffn_shape(s) != MOE_OK) return 0;
    if (s->dtype == MOE_BF16 && choose_path(*s) == 0) return 0;
    return ffn_layout(*s).total;
}

moe_status moe_route_top2(const moe_shape* s, const void* x, const void* w_gate, int32_t* topk_idx, float* topk_w,
                          float* logits, void* stream) {
    NvtxRange nvtx("moe_route_top2");
    MOE_TRY(check_shape(s));
    if (s->T > 0 && (!ok_ptr(x) || !ok_ptr(w_gate) || !ok_ptr(topk_idx) || !ok_ptr(topk_w) ||
                     (logits != nullptr && !aligned16(logits))))
        return MOE_ERR_INVALID_ARG;
    return run_router(*s, x, w_gate, topk_idx, topk_w, logits, static_cast<cudaStream_t>(stream));
}

size_t moe_permute_workspace_bytes(const moe_shape* s) {
    if (check_shape(s) != MOE_OK) return 0;
    return permute_ws_bytes(*s);
}

moe_status moe_permute(const moe_shape* s, const int32_t* topk_idx, const float* topk_w, const void* x,
                       int32_t* counts, int32_t* offsets, int32_t* perm_token, int32_t* slot_row, float* perm_w,
                       void* x_perm, void* ws, size_t ws_bytes, void* stream) {
    NvtxRange nvtx("moe_permute");
    MOE_TRY(check_shape(s));
    if (!ok_ptr(counts) || !ok_ptr(offsets)) return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && (!ok_ptr(topk_idx) || !ok_ptr(topk_w) || !ok_ptr(x) || !ok_ptr(perm_token) ||
                     !ok_ptr(slot_row) || !ok_ptr(perm_w) || !ok_ptr(x_perm)))
        return MOE_ERR_INVALID_ARG;
    if (ws != nullptr && (!aligned16(ws) || ws_bytes < permute_ws_bytes(*s))) return MOE_ERR_WORKSPACE;
    return run_permute(*s, topk_idx, topk_w, x, counts, offsets, perm_token, slot_row, perm_w, x_perm, ws, ws_bytes,
                       static_cast<cudaStream_t>(stream));
}

moe_status moe_expert_ffn(const moe_shape* s, const void* x_perm, const int32_t* offsets, const float* perm_w,
                          const void* w1, const void* w3, const void* w2, float* y_slot, void* ws, size_t ws_bytes,
                          void* stream) {
    NvtxRange nvtx("moe_expert_ffn");
    MOE_TRY(check_ffn_shape(s));
    if (s->T == 0) return MOE_OK;
    if (!ok_ptr(x_perm) || !ok_ptr(offsets) || !ok_ptr(perm_w) || !ok_ptr(w1) || !ok_ptr(w3) || !ok_ptr(w2) ||
        !ok_ptr(y_slot) || !ok_ptr(ws))
        return MOE_ERR_INVALID_ARG;
    if (s->dtype == MOE_BF16 && choose_path(*s) == 0) return MOE_ERR_UNSUPPORTED;
    const FfnLayout L = ffn_layout(*s);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    return run_ffn(*s, x_perm, offsets, perm_w, w1, w3, w2, y_slot, static_cast<unsigned char*>(ws), L,
                   static_cast<cudaStream_t>(stream));
}

moe_status moe_combine(const moe_shape* s, const float* y_slot, const int32_t* slot_row, void* y, void* stream) {
    NvtxRange nvtx("moe_combine");
    MOE_TRY(check_shape(s));
    if (s->T > 0 && (!ok_ptr(y_slot) || !ok_ptr(slot_row) || !ok_ptr(y))) return MOE_ERR_INVALID_ARG;
    return run_combine(*s, y_slot, slot_row, y, static_cast<cudaStream_t>(stream));
}

moe_status moe_aux_stats(const moe_shape* s, const float* logits, const int32_t* counts, float* f, float* P,
                         float* l_aux, void* stream) {
    NvtxRange nvtx("moe_aux_stats");
    MOE_TRY(check_shape(s));
    if (!ok_ptr(counts) || !ok_ptr(f) || !ok_ptr(P) || !ok_ptr(l_aux)) return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && !ok_ptr(logits)) return MOE_ERR_INVALID_ARG;
    return run_aux(*s, logits, counts, f, P, l_aux, static_cast<cudaStream_t>(stream));
}

moe_status moe_layer_forward(const moe_shape* s, const void* x, const void* w_gate, const void* w1, const void* w3,
                             const void* w2, void* y, float* aux_f, float* aux_P, float* aux_l_aux, void* ws,
                             size_t ws_bytes, void* stream) {
    NvtxRange nvtx("moe_layer_forward");
    MOE_TRY(check_shape(s));
    const bool aux = aux_f != nullptr && aux_P != nullptr && aux_l_aux != nullptr;
    if ((aux_f != nullptr || aux_P != nullptr || aux_l_aux != nullptr) && !aux) return MOE_ERR_INVALID_ARG;
    if (aux && (!ok_ptr(aux_f) || !ok_ptr(aux_P) || !ok_ptr(aux_l_aux))) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (s->T == 0) return aux ? run_aux(*s, nullptr, nullptr, aux_f, aux_P, aux_l_aux, st) : MOE_OK;
    if (!ok_ptr(x) || !ok_ptr(w_gate) || !ok_ptr(w1) || !ok_ptr(w3) || !ok_ptr(w2) || !ok_ptr(y) || !ok_ptr(ws))
        return MOE_ERR_INVALID_ARG;
    if (s->dtype == MOE_BF16 && choose_path(*s) == 0) return MOE_ERR_UNSUPPORTED;
    const FwdLayout L = fwd_layout(*s);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    unsigned char* w = static_cast<unsigned char*>(ws);
    int32_t* idx = reinterpret_cast<int32_t*>(w + L.idx);
    float* gw = reinterpret_cast<float*>(w + L.w);
    float* logits = aux ? reinterpret_cast<float*>(w + L.logits) : nullptr;
    int32_t* counts = reinterpret_cast<int32_t*>(w + L.counts);
    int32_t* offsets = reinterpret_cast<int32_t*>(w + L.offsets);
    int32_t* perm_token = reinterpret_cast<int32_t*>(w + L.perm_token);
    int32_t* slot_row = reinterpret_cast<int32_t*>(w + L.slot_row);
    float* perm_w = reinterpret_cast<float*>(w + L.perm_w);
    void* x_perm = w + L.x_perm;
    float* y_slot = reinterpret_cast<float*>(w + L.y_slot);
    MOE_TRY(run_router(*s, x, w_gate, idx, gw, logits, st));
    MOE_TRY(run_permute(*s, idx, gw, x, counts, offsets, perm_token, slot_row, perm_w, x_perm, w + L.perm_ws,
                        permute_ws_bytes(*s), st));
    bool combined = false;
    // The fused combine makes a pair wait for units of other pairs, so it needs every pair resident at
    // once: with MOE_KNOB_GRID above one CTA per SM the separate combine pass runs instead.
    const bool all_pairs_resident = g.grid == 0 || g.grid <= sm_count();
    MOE_TRY(run_ffn(*s, x_perm, offsets, perm_w, w1, w3, w2, y_slot, w + L.ffn, L.f, st, slot_row, y, &combined,
                    nullptr, nullptr, all_pairs_resident ? perm_token : nullptr));
    if (!combined) MOE_TRY(run_combine(*s, y_slot, slot_row, y, st));
    if (aux) MOE_TRY(run_aux(*s, logits, counts, aux_f, aux_P, aux_l_aux, st));
    return MOE_OK;
}

moe_status moe_layer_forward_noalloc(const moe_shape* s, const void* x, const void* w_gate, const void* w1,
                                     const void* w3, const void* w2, void* y, void* stream) {
    NvtxRange nvtx("moe_layer_forward_noalloc");
    MOE_TRY(check_shape(s));
    if (s->T == 0) return MOE_OK;
    if (s->dtype == MOE_BF16 && choose_path(*s) == 0) return MOE_ERR_UNSUPPORTED;
    if (fwd_layout(*s).total > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;
    void* scratch = noalloc_scratch();
    if (scratch == nullptr) return MOE_ERR_CUDA;
    return moe_layer_forward(s, x, w_gate, w1, w3, w2, y, nullptr, nullptr, nullptr, scratch, kNoAllocScratchBytes,
                             stream);
}

size_t moe_block_workspace_bytes(const moe_block_shape* s) {
    if (check_block_shape(s) != MOE_OK) return 0;
    return block_layout(*s).total;
}

bool block_weights_ok(const moe_block_weights* w) {
    return w != nullptr && ok_ptr(w->attn_norm) && ok_ptr(w->wqkv) && ok_ptr(w->wo) && ok_ptr(w->ffn_norm) &&
           ok_ptr(w->w_gate) && ok_ptr(w->w1) && ok_ptr(w->w3) && ok_ptr(w->w2);
}

moe_status moe_block_forward(const moe_block_shape* s, const void* x, const moe_block_weights* w, void* k_cache,
                             void* v_cache, void* out, void* ws, size_t ws_bytes, void* stream) {
    NvtxRange nvtx("moe_block_forward");
    MOE_TRY(check_block_shape(s));
    if (!block_weights_ok(w) || !ok_ptr(x) || !ok_ptr(out) || !ok_ptr(ws) || x == out)
        return MOE_ERR_INVALID_ARG;
    if ((k_cache == nullptr) != (v_cache == nullptr)) return MOE_ERR_INVALID_ARG;
    if (k_cache != nullptr && (!ok_ptr(k_cache) || !ok_ptr(v_cache) || s->S > s->cache_max)) return MOE_ERR_INVALID_ARG;
    const BlockLayout L = block_layout(*s);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char* b = static_cast<unsigned char*>(ws);
    const int64_t T = s->B * s->S;
    const int d = s->d;
    const int wq = s->n_heads * s->head_dim, wkv = s->n_kv_heads * s->head_dim;
    void* xn = b + L.xn;
    float* qkv = reinterpret_cast<float*>(b + L.qkv);
    void* q = b + L.q;
    void* k = b + L.k;
    void* v = b + L.v;
    void* attn = b + L.attn;
    void* h = b + L.h;
    void* y = b + L.y;
    // h = x + Wo attention(RoPE(Wq xn), RoPE(Wk xn), Wv xn), xn = RMSNorm(x)
    MOE_TRY(run_rmsnorm(T, d, x, nullptr, w->attn_norm, s->eps, nullptr, xn, st));
    MOE_TRY(run_linear(T, d, wq + 2 * wkv, xn, w->wqkv, qkv, st, "linear_qkv"));
    MOE_TRY(run_rope(*s, qkv, q, k, v, st, nullptr, k_cache, v_cache));
    MOE_TRY(run_attention(*s, q, k, v, attn, st));
    float* o = qkv;  // the projection output is consumed: Wo's output takes its place
    MOE_TRY(run_linear(T, wq, d, attn, w->wo, o, st, "linear_o"));
    // out = h + MoE(RMSNorm(h)); the second norm's output takes xn's place
    MOE_TRY(run_rmsnorm(T, d, x, o, w->ffn_norm, s->eps, h, xn, st));
    const moe_shape m = block_layer_shape(*s);
    MOE_TRY(moe_layer_forward(&m, xn, w->w_gate, w->w1, w->w3, w->w2, y, nullptr, nullptr, nullptr, b + L.moe,
                              L.total - L.moe, stream));
    return run_residual_add(T * d, h, y, out, st);
}

size_t moe_block_decode_workspace_bytes(const moe_block_shape* s) {
    if (check_block_shape(s) != MOE_OK || !decode_supported(*s)) return 0;
    return decode_layout(*s).total;
}

moe_status moe_block_decode(const moe_block_shape* s, const void* x, const moe_block_weights* w, void* k_cache,
                            void* v_cache, int32_t* cache_len, void* out, void* ws, size_t ws_bytes, void* stream) {
    NvtxRange nvtx("moe_block_decode");
    MOE_TRY(check_block_shape(s));
    if (s->S != 1 || s->cache_max < 1) return MOE_ERR_INVALID_ARG;
    if (!decode_supported(*s)) return MOE_ERR_UNSUPPORTED;
    if (!block_weights_ok(w) || !ok_ptr(x) || !ok_ptr(out) || !ok_ptr(ws) || !ok_ptr(k_cache) || !ok_ptr(v_cache) ||
        cache_len == nullptr || x == out)
        return MOE_ERR_INVALID_ARG;
    const DecodeLayout L = decode_layout(*s);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char* b = static_cast<unsigned char*>(ws);
    const int64_t B = s->B;
    const int d = s->d;
    const int wq = s->n_heads * s->head_dim, wkv = s->n_kv_heads * s->head_dim;
    void* xn = b + L.xn;
    float* qkv = reinterpret_cast<float*>(b + L.qkv);
    void* q = b + L.q;
    void* attn = b + L.attn;
    void* h = b + L.h;
    void* y = b + L.y;
    unsigned char* lin = b + L.lin;
    MOE_TRY(run_rmsnorm(B, d, x, nullptr, w->attn_norm, s->eps, nullptr, xn, st));
    MOE_TRY(run_linear(B, d, wq + 2 * wkv, xn, w->wqkv, qkv, st, "linear_qkv", lin, L.lin_bytes));
    // q to the workspace; the new key and value straight into the caches at position cache_len[b]
    moe_block_shape one = *s;
    one.S = 1;
    MOE_TRY(run_rope(one, qkv, q, nullptr, nullptr, st, cache_len, k_cache, v_cache));
    MOE_TRY(run_attention_decode(*s, q, k_cache, v_cache, cache_len, attn, b + L.att, st));
    float* o = qkv;
    MOE_TRY(run_linear(B, wq, d, attn, w->wo, o, st, "linear_o", lin, L.lin_bytes));
    MOE_TRY(run_rmsnorm(B, d, x, o, w->ffn_norm, s->eps, h, xn, st));
    const moe_shape m = block_layer_shape(*s);
    MOE_TRY(moe_layer_forward(&m, xn, w->w_gate, w->w1, w->w3, w->w2, y, nullptr, nullptr, nullptr, b + L.moe,
                              L.total - L.moe, stream));
    return run_residual_add(B * d, h, y, out, st);
}

size_t moe_attention_decode_workspace_bytes(const moe_block_shape* s) {
    if (check_block_shape(s) != MOE_OK || !decode_supported(*s)) return 0;
    return decode_attention_ws_bytes(*s);
}

moe_status moe_attention_decode(const moe_block_shape* s, const void* q, const void* k_cache, const void* v_cache,
                                int32_t* cache_len, void* o, void* ws, size_t ws_bytes, void* stream) {
    NvtxRange nvtx("moe_attention_decode");
    MOE_TRY(check_block_shape(s));
    if (s->S != 1 || s->cache_max < 1) return MOE_ERR_INVALID_ARG;
    if (!decode_supported(*s)) return MOE_ERR_UNSUPPORTED;
    if (!ok_ptr(q) || !ok_ptr(k_cache) || !ok_ptr(v_cache) || cache_len == nullptr || !ok_ptr(o) || !ok_ptr(ws))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < decode_attention_ws_bytes(*s)) return MOE_ERR_WORKSPACE;
    return run_attention_decode(*s, q, k_cache, v_cache, cache_len, o, static_cast<unsigned char*>(ws),
                                static_cast<cudaStream_t>(stream));
}

moe_status moe_rmsnorm(int64_t rows, int32_t d, const void* x, const float* add, const void* g, float eps,
                       void* h_out, void* y, void* stream) {
    NvtxRange nvtx("moe_rmsnorm");
    if (rows < 0 || d <= 0 || d % 8 != 0 || !(eps >= 0.f) || !std::isfinite(eps)) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!ok_ptr(x) || !ok_ptr(g) || !ok_ptr(y) || (add != nullptr && (!ok_ptr(add) || !ok_ptr(h_out))))
        return MOE_ERR_INVALID_ARG;
    return run_rmsnorm(rows, d, x, add, g, eps, add != nullptr ? h_out : nullptr, y, static_cast<cudaStream_t>(stream));
}

size_t moe_linear_workspace_bytes(int64_t rows, int32_t n_in, int32_t n_out) {
    if (rows <= 0 || n_in <= 0 || n_out <= 0 || n_in % kBK != 0 || n_out % kTileN != 0) return 0;
    return linear_stream_plan(rows, n_in, n_out).part_bytes;
}

moe_status moe_linear(int64_t rows, int32_t n_in, int32_t n_out, const void* x, const void* w, float* y, void* ws,
                      size_t ws_bytes, void* stream) {
    NvtxRange nvtx("moe_linear");
    if (rows < 0 || n_in <= 0 || n_out <= 0) return MOE_ERR_INVALID_ARG;
    if (n_in % kBK != 0 || n_out % kTileN != 0 || rows > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    if (rows == 0) return MOE_OK;
    if (!ok_ptr(x) || !ok_ptr(w) || !ok_ptr(y) || (ws != nullptr && !ok_ptr(ws))) return MOE_ERR_INVALID_ARG;
    return run_linear(rows, n_in, n_out, x, w, y, static_cast<cudaStream_t>(stream), "linear",
                      static_cast<unsigned char*>(ws), ws != nullptr ? ws_bytes : 0);
}

moe_status moe_rope_split(const moe_block_shape* s, const float* qkv, const int32_t* pos, void* q, void* k, void* v,
                          void* k_cache, void* v_cache, void* stream) {
    NvtxRange nvtx("moe_rope_split");
    MOE_TRY(check_block_shape(s));
    if (!ok_ptr(qkv) || !ok_ptr(q) || (k != nullptr && !ok_ptr(k)) || (v != nullptr && !ok_ptr(v)) ||
        (k == nullptr) != (v == nullptr) || (k_cache == nullptr) != (v_cache == nullptr))
        return MOE_ERR_INVALID_ARG;
    if (k_cache != nullptr && (!ok_ptr(k_cache) || !ok_ptr(v_cache) || s->cache_max < 1)) return MOE_ERR_INVALID_ARG;
    if (pos != nullptr && s->S != 1) return MOE_ERR_INVALID_ARG;
    if (k == nullptr && k_cache == nullptr) return MOE_ERR_INVALID_ARG;
    if (pos == nullptr && k_cache != nullptr && s->S > s->cache_max) return MOE_ERR_INVALID_ARG;
    return run_rope(*s, qkv, q, k, v, static_cast<cudaStream_t>(stream), pos, k_cache, v_cache);
}

moe_status moe_attention(const moe_block_shape* s, const void* q, const void* k, const void* v, void* o,
                         void* stream) {
    NvtxRange nvtx("moe_attention");
    MOE_TRY(check_block_shape(s));
    if (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(o)) return MOE_ERR_INVALID_ARG;
    return run_attention(*s, q, k, v, o, static_cast<cudaStream_t>(stream));
}

moe_status moe_residual_add(int64_t n, const void* a, const void* b, void* out, void* stream) {
    NvtxRange nvtx("moe_residual_add");
    if (n < 0 || n % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    if (!ok_ptr(a) || !ok_ptr(b) || !ok_ptr(out)) return MOE_ERR_INVALID_ARG;
    return run_residual_add(n, a, b, out, static_cast<cudaStream_t>(stream));
}

moe_status moe_gather_rows(const void* src, int64_t src_rows, const int32_t* index, int64_t rows, int64_t row_bytes,
                           void* dst, void* stream) {
    NvtxRange nvtx("moe_gather_rows");
    if (rows < 0 || src_rows < 0 || row_bytes <= 0 || row_bytes % 16 != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!ok_ptr(src) || !ok_ptr(index) || !ok_ptr(dst)) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t chunks = rows * (row_bytes / 16);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((chunks + 1023) / 1024, (int64_t)sm_count() * 8));
    return launch("gather_rows", st, [&] {
        return klaunch(gather_index_kernel, grid, 256, 0, st, static_cast<const unsigned char*>(src), src_rows, index,
                       rows, row_bytes, static_cast<unsigned char*>(dst));
    });
}

size_t moe_train_state_bytes(const moe_shape* s) {
    if (check_shape(s) != MOE_OK || !train_supported(*s) || choose_path(*s) == 0) return 0;
    return train_layout(*s).total;
}

size_t moe_backward_workspace_bytes(const moe_shape* s) {
    if (check_shape(s) != MOE_OK || !train_supported(*s)) return 0;
    return bwd_layout(*s).total;
}

moe_status moe_layer_forward_train(const moe_shape* s, const void* x, const void* w_gate, const void* w1,
                                   const void* w3, const void* w2, void* y, float* aux_f, float* aux_P,
                                   float* aux_l_aux, void* state, size_t state_bytes, void* stream) {
    NvtxRange nvtx("moe_layer_forward_train");
    MOE_TRY(check_shape(s));
    if (!train_supported(*s)) return MOE_ERR_UNSUPPORTED;
    const bool aux = aux_f != nullptr && aux_P != nullptr && aux_l_aux != nullptr;
    if ((aux_f != nullptr || aux_P != nullptr || aux_l_aux != nullptr) && !aux) return MOE_ERR_INVALID_ARG;
    if (aux && (!ok_ptr(aux_f) || !ok_ptr(aux_P) || !ok_ptr(aux_l_aux))) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (s->T == 0) return aux ? run_aux(*s, nullptr, nullptr, aux_f, aux_P, aux_l_aux, st) : MOE_OK;
    if (!ok_ptr(x) || !ok_ptr(w_gate) || !ok_ptr(w1) || !ok_ptr(w3) || !ok_ptr(w2) || !ok_ptr(y) || !ok_ptr(state))
        return MOE_ERR_INVALID_ARG;
    if (choose_path(*s) == 0) return MOE_ERR_UNSUPPORTED;
    const TrainLayout L = train_layout(*s);
    if (state_bytes < L.total) return MOE_ERR_WORKSPACE;
    unsigned char* w = static_cast<unsigned char*>(state);
    int32_t* idx = reinterpret_cast<int32_t*>(w + L.f.idx);
    float* gw = reinterpret_cast<float*>(w + L.f.w);
    float* logits = reinterpret_cast<float*>(w + L.f.logits);
    int32_t* counts = reinterpret_cast<int32_t*>(w + L.f.counts);
    int32_t* offsets = reinterpret_cast<int32_t*>(w + L.f.offsets);
    int32_t* perm_token = reinterpret_cast<int32_t*>(w + L.f.perm_token);
    int32_t* slot_row = reinterpret_cast<int32_t*>(w + L.f.slot_row);
    float* perm_w = reinterpret_cast<float*>(w + L.f.perm_w);
    void* x_perm = w + L.f.x_perm;
    float* y_slot = reinterpret_cast<float*>(w + L.f.y_slot);
    MOE_TRY(run_router(*s, x, w_gate, idx, gw, logits, st));
    MOE_TRY(run_permute(*s, idx, gw, x, counts, offsets, perm_token, slot_row, perm_w, x_perm, w + L.f.perm_ws,
                        permute_ws_bytes(*s), st));
    // y_slot stays in the state (the backward reads each expert's output), so
    // the expert outputs are combined by the separate pass
    MOE_TRY(run_ffn(*s, x_perm, offsets, perm_w, w1, w3, w2, y_slot, w + L.f.ffn, L.f.f, st, nullptr, nullptr,
                    nullptr, reinterpret_cast<__nv_bfloat16*>(w + L.u), reinterpret_cast<__nv_bfloat16*>(w + L.v)));
    MOE_TRY(run_combine(*s, y_slot, slot_row, y, st));
    if (aux) MOE_TRY(run_aux(*s, logits, counts, aux_f, aux_P, aux_l_aux, st));
    return MOE_OK;
}

moe_status moe_layer_backward(const moe_shape* s, const void* x, const void* w_gate, const void* w1, const void* w3,
                              const void* w2, const void* dy, float aux_coef, const void* state, size_t state_bytes,
                              void* dx, float* dw_gate, float* dw1, float* dw3, float* dw2, void* ws, size_t ws_bytes,
                              void* stream) {
    NvtxRange nvtx("moe_layer_backward");
    MOE_TRY(check_shape(s));
    if (!train_supported(*s)) return MOE_ERR_UNSUPPORTED;
    if (!ok_ptr(dw_gate) || !ok_ptr(dw1) || !ok_ptr(dw3) || !ok_ptr(dw2)) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (s->T == 0) {
        // no tokens: every gradient is zero
        const size_t we = (size_t)s->E * s->ffn * s->d * sizeof(float);
        if (cudaMemsetAsync(dw_gate, 0, (size_t)s->E * s->d * sizeof(float), st) != cudaSuccess ||
            cudaMemsetAsync(dw1, 0, we, st) != cudaSuccess || cudaMemsetAsync(dw3, 0, we, st) != cudaSuccess ||
            cudaMemsetAsync(dw2, 0, we, st) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (!ok_ptr(x) || !ok_ptr(w_gate) || !ok_ptr(w1) || !ok_ptr(w3) || !ok_ptr(w2) || !ok_ptr(dy) ||
        !ok_ptr(state) || !ok_ptr(dx) || !ok_ptr(ws))
        return MOE_ERR_INVALID_ARG;
    if (choose_path(*s) == 0) return MOE_ERR_UNSUPPORTED;
    if (state_bytes < train_layout(*s).total || ws_bytes < bwd_layout(*s).total) return MOE_ERR_WORKSPACE;
    return run_backward(*s, static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w_gate),
                        static_cast<const __nv_bfloat16*>(w1), static_cast<const __nv_bfloat16*>(w3),
                        static_cast<const __nv_bfloat16*>(w2), static_cast<const __nv_bfloat16*>(dy), aux_coef,
                        static_cast<const unsigned char*>(state), static_cast<__nv_bfloat16*>(dx), dw_gate, dw1, dw3,
                        dw2, static_cast<unsigned char*>(ws), st);
}

moe_status moe_selftest_wait_timeout(uint64_t timeout_ns, int32_t* gave_up, void* stream) {
    if (timeout_ns == 0 || timeout_ns > 10000000000ull || !ok_ptr(gave_up)) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return launch("wait_selftest", st, [&] {
        wait_selftest_kernel<<<1, 32, 0, st>>>(timeout_ns, gave_up);
        return cudaGetLastError();
    });
}

moe_status moe_read_probe(const void* buf, size_t bytes, uint32_t* sink, void* stream) {
    if (!ok_ptr(buf) || !ok_ptr(sink) || bytes == 0 || bytes % 16 != 0) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t n16 = bytes / 16;
    const int grid = (int)std::max<size_t>(1, std::min<size_t>((size_t)sm_count() * 4, (n16 + 511) / 512));
    return launch("read_probe", st, [&] {
        return klaunch(read_probe_kernel, grid, 512, 0, st, static_cast<const uint4*>(buf), n16, sink);
    });
}

moe_status moe_get_device_status(int32_t* code, int32_t* detail) {
    if (code == nullptr) return MOE_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    int h[4] = {0, 0, 0, 0};
    if (cudaMemcpyFromSymbol(h, g_status, sizeof(h)) != cudaSuccess) return MOE_ERR_CUDA;
    const int zero[4] = {0, 0, 0, 0};
    if (cudaMemcpyToSymbol(g_status, zero, sizeof(zero)) != cudaSuccess) return MOE_ERR_CUDA;
    *code = h[0];
    if (detail != nullptr) *detail = h[1] * 100 + h[2];
    return MOE_OK;
}

moe_status moe_check_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
    int32_t code = MOE_OK;
    const moe_status rc = moe_get_device_status(&code, nullptr);
    return rc != MOE_OK ? rc : static_cast<moe_status>(code);
}

moe_status moe_set_wait_timeout_ns(uint64_t ns) {
    if (ns == 0) return MOE_ERR_INVALID_ARG;
    g.timeout_ns = ns;
    return MOE_OK;
}

moe_status moe_set_knob(int32_t knob, int64_t value) {
    switch (knob) {
        case MOE_KNOB_FFN_PATH:
            if (value < 0 || value > 4 || value == 3) return MOE_ERR_INVALID_ARG;
            g.ffn_path = (int)value;
            return MOE_OK;
        case MOE_KNOB_KSLICE:
            if (value < 0 || value % kBK != 0) return MOE_ERR_INVALID_ARG;
            g.kslice = value;
            return MOE_OK;
        case MOE_KNOB_GRID:
            if (value < 0 || value > 65535) return MOE_ERR_INVALID_ARG;
            g.grid = (int)value;
            return MOE_OK;
        case MOE_KNOB_PDL:
            if (value < 0 || value > 1) return MOE_ERR_INVALID_ARG;
            g.pdl = value != 0;
            return MOE_OK;
        case MOE_KNOB_TILE_CTAS:
            if (value < 0 || value > 2) return MOE_ERR_INVALID_ARG;
            g.tile_ctas = (int)value;
            return MOE_OK;
        case MOE_KNOB_TILE_SCHED:
            if (value < 0 || value > 7) return MOE_ERR_INVALID_ARG;
            g.tile_sched = (int)value;
            return MOE_OK;
        case MOE_KNOB_FUSE_COMBINE:
            if (value < 0 || value > 1) return MOE_ERR_INVALID_ARG;
            g.fuse_combine = value != 0;
            return MOE_OK;
        case MOE_KNOB_ROUTER_TC:
            if (value < 0 || value > 1) return MOE_ERR_INVALID_ARG;
            g.router_tc = value != 0;
            return MOE_OK;
        case MOE_KNOB_L2_KEEP_KB:
            if (value < 0 || value > 128 * 1024) return MOE_ERR_INVALID_ARG;
            g.l2_keep_bytes = (uint64_t)value * 1024u;
            return MOE_OK;
        case MOE_KNOB_DEBUG:
            if (value < 0 || value > 1) return MOE_ERR_INVALID_ARG;
            g.debug = value != 0;
            return MOE_OK;
    }
    return MOE_ERR_INVALID_ARG;
}

moe_status moe_timing_enable(int32_t enable) {
    g.timing = enable != 0;
    return MOE_OK;
}

moe_status moe_timing_read(char* buf, size_t n) {
    std::map<std::string, std::pair<long, double>> agg;
    moe_status rc = MOE_OK;
    for (const TimingRecord& r : g.records) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
            rc = MOE_ERR_CUDA;
        auto& a = agg[r.name];
        a.first += 1;
        a.second += ms;
        g.pool.push_back(r.start);
        g.pool.push_back(r.stop);
    }
    g.records.clear();
    std::string out = "{";
    bool first = true;
    for (const auto& kv : agg) {
        char line[160];
        std::snprintf(line, sizeof(line), "%s\"%s\": [%ld, %.6f]", first ? "" : ", ", kv.first.c_str(),
                      kv.second.first, kv.second.second);
        out += line;
        first = false;
    }
    out += "}";
    if (buf != nullptr && n > 0) {
        std::strncpy(buf, out.c_str(), n - 1);
        buf[n - 1] = '\0';
    }
    return rc;
}

}  // extern "C"
