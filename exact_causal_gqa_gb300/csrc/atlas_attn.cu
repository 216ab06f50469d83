// atlas_attn.cu -- the C ABI: argument checks, the split plan, tensor-map
// encoding and kernel launches.  Declared in include/atlas_attn.h.
#include "internal.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <limits.h>
#include <math.h>
#include <stdint.h>
#include <algorithm>
#include <atomic>
#include <mutex>

namespace atlas {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult res;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &res) == cudaSuccess &&
            res == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// CTAs the automatic split plan aims for at the largest context the page table
// allows: SMs x 2 resident CTAs x 2 waves, with splits of at most kMaxSplit keys
// (measured best at 2.5K-4K keys, ~1.3-2 MB of K/V per CTA, on the decode
// workloads).  A pure function of the call's sizes and the SM count, so a given
// problem on a given part always gets the same split (and the same bits).
int64_t plan_ctas(int sms) { return (int64_t)sms * 2 * 2; }
constexpr int64_t kMaxSplit = 2560;
// The fp32 ring kernel with 4 or 8 columns runs 4-warp CTAs three to an SM: its
// splits aim for SMs x 3 x 4 CTAs, so that a small batch still fills every slot
// (a lone 4-warp CTA on an SM runs at about half the rate of 12 warps).
int64_t f32_ring_plan_ctas(int sms) { return (int64_t)sms * 3 * 4; }

// The tensor-core path's split plan aims for SMs x 1 CTA x 3 waves at the largest
// context (splits of 1K-8K keys; 8K measured best for the suffix workload); it
// writes the output directly once a call has at least SMs x 2 query tiles.
int64_t tc_plan_ctas(int sms) { return (int64_t)sms * 3; }
int64_t tc_direct_tiles(int sms) { return (int64_t)sms * 2; }
// Query tiles whose rows see fewer keys than this use a hi + lo split of P:
// with few keys (or a peaked softmax) a single bf16 rounding of P moves the
// output by up to 2^-8 |v| (bf16 keeps 8 significant bits).  Scores sharper than
// unit-variance inputs at scale 1/sqrt(D) (|scale| sqrt(D) above kHiLoScale) use
// the split on every tile.  Elsewhere the kernel decides per block (fmha_tc.cu).
constexpr int kHiLoBelow = 512;
constexpr float kHiLoScale = 1.25f;

// A bf16 decode-like call whose whole context per (sequence, kv head) holds at most
// this many K/V bytes runs as one split per (sequence, kv head, column tile) that
// writes its output directly: at that size the merge launch (a few microseconds)
// costs more than the parallelism the splits add.
constexpr int64_t kDirectMaxBytes = 256 * 1024;
// An fp32 ring-kernel call whose automatic plan has at most this many splits runs
// them as one thread-block cluster per (sequence, kv head, column tile), merged in
// distributed shared memory (the portable cluster size limit).
constexpr int kClusterMaxSplits = 8;

// One GB300: the count the plan assumes when no device is visible.
constexpr int kDefaultSms = 152;

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

std::atomic<int> g_sm_count[64];

}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return kDefaultSms;
    }
    const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
    if (cached > 0) return cached;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return kDefaultSms;
    }
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

atlas_status make_plan(atlas_kind kind, int32_t Hq, int32_t Hkv, int32_t D, int32_t P,
                       const atlas_launch *L, Plan *plan) {
    if (!L) return ATLAS_ERR_INVALID_ARG;
    if (L->sm_count < 0) return ATLAS_ERR_INVALID_ARG;
    const int sms = L->sm_count > 0 ? L->sm_count : device_sm_count();
    if (kind != ATLAS_KIND_DECODE && kind != ATLAS_KIND_SUFFIX && kind != ATLAS_KIND_PREFILL)
        return ATLAS_ERR_INVALID_ARG;
    if (L->batch < 1 || L->max_pages_per_seq < 1 || L->num_pages < 1 || L->q_len < 1 || Hq < 1 ||
        Hkv < 1 || Hq % Hkv != 0)
        return ATLAS_ERR_INVALID_ARG;
    if (kind == ATLAS_KIND_DECODE && L->q_len != 1) return ATLAS_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return ATLAS_ERR_UNSUPPORTED;
    if (!is_pow2(P) || P < 8 || P > 128) return ATLAS_ERR_UNSUPPORTED;
    if (L->q_dtype != L->kv_dtype) return ATLAS_ERR_UNSUPPORTED;
    if (L->kv_dtype == ATLAS_F32) {
        if (L->out_dtype != ATLAS_F32) return ATLAS_ERR_UNSUPPORTED;
    } else if (L->kv_dtype == ATLAS_BF16) {
        if (L->out_dtype != ATLAS_F32 && L->out_dtype != ATLAS_BF16) return ATLAS_ERR_UNSUPPORTED;
    } else {
        return ATLAS_ERR_UNSUPPORTED;
    }
    const int64_t max_ctx = (int64_t)L->max_pages_per_seq * P;
    if (max_ctx > INT32_MAX / 2) return ATLAS_ERR_INVALID_ARG;
    // Keys one (sequence, kv head) may need: a window bounds them.  Splits are
    // sized from this; the split count still covers the whole context (splits
    // below every row's window exit at once).
    const int64_t work_ctx =
        L->window > 0 ? std::min(max_ctx, (int64_t)L->window + L->q_len + 127) : max_ctx;
    if ((int64_t)L->num_pages * Hkv * P >= INT32_MAX) return ATLAS_ERR_INVALID_ARG;
    if (L->q_len > max_ctx) return ATLAS_ERR_INVALID_ARG;
    // Output rows are indexed in 32 bits (the merge, the tensor-core tiles).
    if ((int64_t)L->batch * Hq * L->q_len >= INT32_MAX) return ATLAS_ERR_INVALID_ARG;
    if (L->split_tokens < 0 || L->split_tokens % kSplitBlockTokens != 0)
        return ATLAS_ERR_INVALID_ARG;
    if (L->phase != ATLAS_PHASE_ALL && L->phase != ATLAS_PHASE_CHUNKS &&
        L->phase != ATLAS_PHASE_MERGE)
        return ATLAS_ERR_INVALID_ARG;

    const int G = Hq / Hkv;
    plan->G = G;
    plan->direct = plan->cluster = plan->balanced = 0;
    plan->tc_split = 0;
    plan->tiles_per_unit = plan->tiles_per_head = 0;
    if ((int64_t)G * L->q_len > 16) {
        // Many query rows per (sequence, kv head): 128-row tiles on tcgen05 (bf16
        // products, or three tf32 products per fp32 product).
        plan->path = L->kv_dtype == ATLAS_BF16 ? Path::TensorCore : Path::TensorCoreF32;
        const int64_t tiles_per_unit = ((int64_t)G * L->q_len + 127) / 128;
        const int64_t tiles = (int64_t)L->batch * Hkv * tiles_per_unit;
        plan->tiles_per_unit = (int)tiles_per_unit;
        plan->col_tiles = 0;
        int64_t chunk = 0;
        if (L->split_tokens > 0) {
            chunk = round_up(L->split_tokens, 128);
        } else if ((tiles < tc_direct_tiles(sms) || L->phase != ATLAS_PHASE_ALL) &&
                   !(L->debug_flags & ATLAS_DEBUG_TC_DIRECT)) {
            const int64_t target = tc_plan_ctas(sms);
            chunk = round_up((work_ctx * tiles + target - 1) / target, 128);
            if (chunk < 1024) chunk = 1024;
            if (chunk > 8192) chunk = 8192;
        }
        if (chunk > 0) {
            if (chunk > round_up(max_ctx, 128)) chunk = round_up(max_ctx, 128);
            if (tiles > 65535) return ATLAS_ERR_UNSUPPORTED;
            plan->tc_split = 1;
            // An automatic whole call cuts each sequence into equal splits taken
            // longest-first (the chunked phases keep fixed chunks: their passes
            // are defined on them).
            plan->balanced = L->split_tokens == 0 && L->phase == ATLAS_PHASE_ALL &&
                             !L->chunk_range && L->batch <= kTcOrderMaxSeqs;
            plan->chunk = (int)chunk;
            plan->n_chunks = (int)((max_ctx + chunk - 1) / chunk);
            const int64_t rows = (int64_t)L->batch * Hq * L->q_len;
            plan->acc_bytes = (size_t)rows * plan->n_chunks * D * sizeof(float);
            plan->ml_offset = (size_t)round_up((int64_t)plan->acc_bytes, 256);
            plan->ws_bytes = plan->ml_offset + (size_t)rows * plan->n_chunks * 2 * sizeof(float);
        } else {
            if (tiles > INT32_MAX || L->phase != ATLAS_PHASE_ALL) return ATLAS_ERR_UNSUPPORTED;
            plan->chunk = plan->n_chunks = 0;
            plan->tiles_per_head = (L->q_len % 128 == 0) ? L->q_len / 128 : 0;
            plan->acc_bytes = plan->ml_offset = plan->ws_bytes = 0;
        }
        return ATLAS_OK;
    }
    plan->path = L->kv_dtype == ATLAS_BF16 ? Path::SplitBF16 : Path::SplitF32;
    const int cols = plan->path == Path::SplitBF16      ? split_bf16_cols_per_cta(G, L->q_len)
                                                        : split_f32_cols_per_cta(G, L->q_len);
    plan->col_tiles = (G * L->q_len + cols - 1) / cols;
    if ((int64_t)Hkv * plan->col_tiles > 65535 || L->batch > 65535) return ATLAS_ERR_UNSUPPORTED;

    int64_t chunk = L->split_tokens;
    const int64_t unit_bytes = max_ctx * 2 * D * (L->kv_dtype == ATLAS_BF16 ? 2 : 4);
    const bool whole_call = chunk == 0 && L->phase == ATLAS_PHASE_ALL && !L->chunk_range;
    if (whole_call && plan->path == Path::SplitBF16 && unit_bytes <= kDirectMaxBytes) {
        plan->direct = 1;
        plan->chunk = (int)round_up(max_ctx, kSplitBlockTokens);
        plan->n_chunks = 1;
        plan->acc_bytes = plan->ml_offset = plan->ws_bytes = 0;
        return ATLAS_OK;
    }
    if (chunk == 0) {
        const int64_t units = (int64_t)L->batch * Hkv * plan->col_tiles;
        const int64_t target =
            plan->path == Path::SplitF32 && cols <= 8 ? f32_ring_plan_ctas(sms) : plan_ctas(sms);
        chunk = round_up((work_ctx * units + target - 1) / target, kSplitBlockTokens);
        // The f32 kernel has no pipeline to fill: small splits just add CTAs.
        const int64_t min_chunk = plan->path == Path::SplitF32 ? kSplitBlockTokens : 512;
        if (chunk > kMaxSplit) chunk = kMaxSplit;
        if (chunk < min_chunk) chunk = min_chunk;
    }
    if (chunk > max_ctx) chunk = round_up(max_ctx, kSplitBlockTokens);
    plan->chunk = (int)chunk;
    plan->n_chunks = (int)((max_ctx + chunk - 1) / chunk);
    if (whole_call && plan->path == Path::SplitF32 && plan->n_chunks <= kClusterMaxSplits) {
        plan->cluster = 1;
        plan->acc_bytes = plan->ml_offset = plan->ws_bytes = 0;
        return ATLAS_OK;
    }

    const int64_t rows = (int64_t)L->batch * Hq * L->q_len;
    plan->acc_bytes = (size_t)rows * plan->n_chunks * D * sizeof(float);
    plan->ml_offset = (size_t)round_up((int64_t)plan->acc_bytes, 256);
    plan->ws_bytes = plan->ml_offset + (size_t)rows * plan->n_chunks * 2 * sizeof(float);
    return ATLAS_OK;
}

namespace {

// 2-D view of a bf16 (or fp32) tensor with D elements per row: `rows` rows; boxes
// of one 128-byte row slab (64 bf16 or 32 fp32 elements) x box_rows rows with
// 128-byte swizzling.
atlas_status encode_rows_map(CUtensorMap *map, const void *base, int64_t rows, int32_t D,
                             int32_t box_rows, bool f32 = false) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return ATLAS_ERR_CUDA;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * (f32 ? 4 : 2)};
    const cuuint32_t box[2] = {f32 ? 32u : 64u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATLAS_OK : ATLAS_ERR_CUDA;
}

// View of a page pool (rows = num_pages*Hkv*P, D bf16 per row, 128-byte swizzle)
// for the split kernel.  Pages of fewer than 64 tokens: a 3-D view [D/64 slabs]
// [rows][64 elements] whose box is one page's P rows x all slabs, so one TMA load
// brings a whole page (slab-major in shared memory: the 128-byte rows keep the
// row & 7 swizzle).  This measured ~5 % faster than one box per slab at P = 16.
// Larger pages: a 2-D view with boxes of 64 elements x 64 rows, one per slab.
atlas_status encode_pool_map(CUtensorMap *map, const void *pool, int32_t num_pages, int32_t Hkv,
                             int32_t P, int32_t D) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return ATLAS_ERR_CUDA;
    const cuuint64_t rows = (cuuint64_t)num_pages * Hkv * P;
    CUresult r;
    if (P < kSplitBlockTokens) {
        const cuuint64_t dims[3] = {64u, rows, (cuuint64_t)D / 64};
        const cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128u};
        const cuuint32_t box[3] = {64u, (cuuint32_t)P, (cuuint32_t)D / 64};
        const cuuint32_t estr[3] = {1u, 1u, 1u};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[2] = {(cuuint64_t)D, rows};
        const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
        const cuuint32_t box[2] = {64u, (cuuint32_t)kSplitBlockTokens};
        const cuuint32_t estr[2] = {1u, 1u};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS ? ATLAS_OK : ATLAS_ERR_CUDA;
}

atlas_status run(atlas_kind kind, const void *q, const void *k_pages, const void *v_pages,
                 const int32_t *page_table, const int32_t *seq_lens, int32_t Hq, int32_t Hkv,
                 int32_t D, int32_t P, float scale, const atlas_launch *L) {
    if (!q || !k_pages || !v_pages || !page_table || !seq_lens || !L ||
        (!L->out && L->phase != ATLAS_PHASE_CHUNKS))
        return ATLAS_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(L->out) ||
        !aligned16(L->workspace))
        return ATLAS_ERR_INVALID_ARG;
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return ATLAS_ERR_INVALID_ARG;
    if (L->window < 0 || !(L->softcap >= 0.f) || L->softcap == INFINITY)
        return ATLAS_ERR_INVALID_ARG;
    Plan plan;
    atlas_status st = make_plan(kind, Hq, Hkv, D, P, L, &plan);
    if (st != ATLAS_OK) return st;
    if (plan.ws_bytes > 0 && (!L->workspace || L->workspace_bytes < plan.ws_bytes))
        return ATLAS_ERR_WORKSPACE;

    cudaStream_t stream = static_cast<cudaStream_t>(L->stream);
    // A sticky error from earlier work is not ours to report as a launch failure,
    // but a pending non-sticky one would be picked up by our launch check.
    (void)cudaGetLastError();

    SplitParams sp{};
    sp.q = q;
    sp.k_pages = k_pages;
    sp.v_pages = v_pages;
    sp.page_table = page_table;
    sp.seq_lens = seq_lens;
    sp.B = L->batch;
    sp.Hq = Hq;
    sp.Hkv = Hkv;
    sp.G = plan.G;
    sp.D = D;
    sp.P = P;
    sp.q_len = L->q_len;
    sp.max_pages = L->max_pages_per_seq;
    sp.num_pages = L->num_pages;
    sp.chunk = plan.chunk;
    sp.n_chunks = plan.n_chunks;
    sp.col_tiles = plan.col_tiles;
    sp.require_full = kind == ATLAS_KIND_PREFILL;
    sp.scale_log2 = scale * kLog2e;
    sp.window = L->window;
    sp.q_lens = L->q_lens;
    sp.chunk_range = L->chunk_range;
    sp.softcap_log2 = L->softcap > 0.f ? L->softcap * kLog2e : 0.f;
    sp.softcap_inv = L->softcap > 0.f ? scale / L->softcap : 0.f;
    sp.ws_acc = static_cast<float *>(L->workspace);
    sp.ws_ml = reinterpret_cast<float *>(static_cast<char *>(L->workspace) + plan.ml_offset);
    sp.status = L->status_word;
    sp.debug_flags = L->debug_flags;
    sp.direct = plan.direct;
    sp.cluster = plan.cluster;
    sp.out = L->out;
    sp.out_bf16 = L->out_dtype == ATLAS_BF16;
    sp.lse = L->lse;
    sp.sinks = L->sinks;

    cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
    if (L->events)
        for (int i = 0; i < 3; ++i) ev[i] = static_cast<cudaEvent_t>(L->events[i]);
    cudaError_t err;
    if (L->phase == ATLAS_PHASE_MERGE) {
        if (ev[0] && cudaEventRecord(ev[0], stream) != cudaSuccess) return ATLAS_ERR_CUDA;
        if (ev[1] && cudaEventRecord(ev[1], stream) != cudaSuccess) return ATLAS_ERR_CUDA;
    } else if (plan.path == Path::TensorCore || plan.path == Path::TensorCoreF32) {
        CUtensorMap tmQ, tmK, tmV;
        const bool f32 = plan.path == Path::TensorCoreF32;
        const int bn = f32 ? 64 : 128;  // keys per block of the kernel
        const int box = P < bn ? P : bn;
        st = encode_rows_map(&tmQ, q, (int64_t)L->batch * Hq * L->q_len, D, 128, f32);
        if (st == ATLAS_OK)
            st = encode_rows_map(&tmK, k_pages, (int64_t)L->num_pages * Hkv * P, D, box, f32);
        if (st == ATLAS_OK)
            st = encode_rows_map(&tmV, v_pages, (int64_t)L->num_pages * Hkv * P, D, box, f32);
        if (st != ATLAS_OK) return st;
        TcParams tp{};
        tp.page_table = page_table;
        tp.seq_lens = seq_lens;
        tp.B = L->batch;
        tp.Hq = Hq;
        tp.Hkv = Hkv;
        tp.G = plan.G;
        tp.D = D;
        tp.P = P;
        tp.q_len = L->q_len;
        tp.max_pages = L->max_pages_per_seq;
        tp.num_pages = L->num_pages;
        tp.tiles_per_unit = plan.tiles_per_unit;
        tp.tiles_per_head = plan.tiles_per_head;
        tp.split = plan.tc_split;
        tp.chunk = plan.chunk;
        tp.n_chunks = plan.n_chunks;
        tp.balanced = plan.balanced;
        tp.require_full = kind == ATLAS_KIND_PREFILL;
        tp.hilo_below = fabsf(scale) * sqrtf((float)D) > kHiLoScale ? INT32_MAX : kHiLoBelow;
        tp.negate_scores = scale < 0.f;
        tp.scale_log2 = fabsf(scale) * kLog2e;
        tp.window = L->window;
        tp.softcap_log2 = L->softcap > 0.f ? L->softcap * kLog2e : 0.f;
        tp.softcap_inv = L->softcap > 0.f ? fabsf(scale) / L->softcap : 0.f;
        tp.sinks = L->sinks;
        tp.q_lens = L->q_lens;
        tp.chunk_range = L->chunk_range;
        tp.out = L->out;
        tp.out_bf16 = L->out_dtype == ATLAS_BF16;
        tp.lse = L->lse;
        tp.ws_acc = sp.ws_acc;
        tp.ws_ml = sp.ws_ml;
        tp.status = L->status_word;
        tp.sms = L->sm_count > 0 ? L->sm_count : device_sm_count();
        if (ev[0] && cudaEventRecord(ev[0], stream) != cudaSuccess) return ATLAS_ERR_CUDA;
        err = f32 ? launch_fmha_tc_f32(tp, tmQ, tmK, tmV, stream)
                  : launch_fmha_tc(tp, tmQ, tmK, tmV, stream);
        if (err != cudaSuccess) return ATLAS_ERR_CUDA;
        if (ev[1] && cudaEventRecord(ev[1], stream) != cudaSuccess) return ATLAS_ERR_CUDA;
        if (!plan.tc_split) {
            if (ev[2] && cudaEventRecord(ev[2], stream) != cudaSuccess) return ATLAS_ERR_CUDA;
            return ATLAS_OK;
        }
    } else {
    if (ev[0] && cudaEventRecord(ev[0], stream) != cudaSuccess) return ATLAS_ERR_CUDA;
    if (plan.path == Path::SplitBF16) {
        CUtensorMap tmK, tmV;
        st = encode_pool_map(&tmK, k_pages, L->num_pages, Hkv, P, D);
        if (st == ATLAS_OK) st = encode_pool_map(&tmV, v_pages, L->num_pages, Hkv, P, D);
        if (st != ATLAS_OK) return st;
        err = launch_split_bf16(sp, tmK, tmV, stream);
    } else {
        err = launch_split_f32(sp, stream);
    }
    if (err != cudaSuccess) return ATLAS_ERR_CUDA;
    if (ev[1] && cudaEventRecord(ev[1], stream) != cudaSuccess) return ATLAS_ERR_CUDA;
    }
    if (L->phase == ATLAS_PHASE_CHUNKS || plan.direct || plan.cluster) {
        if (ev[2] && cudaEventRecord(ev[2], stream) != cudaSuccess) return ATLAS_ERR_CUDA;
        return ATLAS_OK;
    }

    MergeParams mp{};
    mp.seq_lens = seq_lens;
    mp.B = L->batch;
    mp.Hq = Hq;
    mp.D = D;
    mp.q_len = L->q_len;
    mp.max_pages = L->max_pages_per_seq;
    mp.P = P;
    mp.chunk = plan.chunk;
    mp.n_chunks = plan.n_chunks;
    mp.balanced = plan.balanced;
    mp.require_full = sp.require_full;
    mp.window = L->window;
    mp.sinks = L->sinks;
    mp.q_lens = L->q_lens;
    mp.ws_acc = sp.ws_acc;
    mp.ws_ml = sp.ws_ml;
    mp.out = L->out;
    mp.out_bf16 = L->out_dtype == ATLAS_BF16;
    mp.lse = L->lse;
    mp.sms = L->sm_count > 0 ? L->sm_count : device_sm_count();
    err = launch_merge(mp, stream);
    if (err != cudaSuccess) return ATLAS_ERR_CUDA;
    if (ev[2] && cudaEventRecord(ev[2], stream) != cudaSuccess) return ATLAS_ERR_CUDA;
    return ATLAS_OK;
}

}  // namespace
}  // namespace atlas

extern "C" {

atlas_status atlas_attn_decode(const void *q, const void *k_pages, const void *v_pages,
                               const int32_t *page_table, const int32_t *seq_lens,
                               int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                               int32_t page_tokens, float scale, const atlas_launch *L) {
    return atlas::run(ATLAS_KIND_DECODE, q, k_pages, v_pages, page_table, seq_lens, n_q_heads,
                      n_kv_heads, head_dim, page_tokens, scale, L);
}

atlas_status atlas_attn_suffix(const void *q, const void *k_pages, const void *v_pages,
                               const int32_t *page_table, const int32_t *seq_lens,
                               int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                               int32_t page_tokens, float scale, const atlas_launch *L) {
    return atlas::run(ATLAS_KIND_SUFFIX, q, k_pages, v_pages, page_table, seq_lens, n_q_heads,
                      n_kv_heads, head_dim, page_tokens, scale, L);
}

atlas_status atlas_attn_prefill(const void *q, const void *k_pages, const void *v_pages,
                                const int32_t *page_table, const int32_t *seq_lens,
                                int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                int32_t page_tokens, float scale, const atlas_launch *L) {
    return atlas::run(ATLAS_KIND_PREFILL, q, k_pages, v_pages, page_table, seq_lens, n_q_heads,
                      n_kv_heads, head_dim, page_tokens, scale, L);
}

atlas_status atlas_kv_append(const void *k_new, const void *v_new, void *k_pages, void *v_pages,
                             const int32_t *page_table, const int32_t *seq_lens,
                             const int32_t *n_new, int32_t n_kv_heads, int32_t head_dim,
                             int32_t page_tokens, const atlas_append *A) {
    if (!A || !k_new || !v_new || !k_pages || !v_pages || !page_table || !seq_lens)
        return ATLAS_ERR_INVALID_ARG;
    if (A->batch < 1 || A->max_pages_per_seq < 1 || A->num_pages < 1 || A->max_new < 0 ||
        n_kv_heads < 1)
        return ATLAS_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return ATLAS_ERR_UNSUPPORTED;
    if (page_tokens < 1 || page_tokens > 128 || (page_tokens & (page_tokens - 1)))
        return ATLAS_ERR_UNSUPPORTED;
    if (A->kv_dtype != ATLAS_F32 && A->kv_dtype != ATLAS_BF16) return ATLAS_ERR_UNSUPPORTED;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
                          reinterpret_cast<uintptr_t>(k_pages) | reinterpret_cast<uintptr_t>(v_pages);
    if (mis & 15u) return ATLAS_ERR_INVALID_ARG;
    if (A->max_new == 0) return ATLAS_OK;
    atlas::AppendParams ap{};
    ap.k_new = k_new;
    ap.v_new = v_new;
    ap.k_pages = k_pages;
    ap.v_pages = v_pages;
    ap.page_table = page_table;
    ap.seq_lens = seq_lens;
    ap.n_new = n_new;
    ap.B = A->batch;
    ap.Hkv = n_kv_heads;
    ap.max_new = A->max_new;
    ap.P = page_tokens;
    ap.max_pages = A->max_pages_per_seq;
    ap.num_pages = A->num_pages;
    ap.row_bytes = head_dim * (A->kv_dtype == ATLAS_BF16 ? 2 : 4);
    ap.status = A->status_word;
    (void)cudaGetLastError();
    return atlas::launch_kv_append(ap, static_cast<cudaStream_t>(A->stream)) == cudaSuccess
               ? ATLAS_OK
               : ATLAS_ERR_CUDA;
}

size_t atlas_attn_workspace_size(atlas_kind kind, int32_t n_q_heads, int32_t n_kv_heads,
                                 int32_t head_dim, int32_t page_tokens, const atlas_launch *L) {
    atlas::Plan plan;
    if (atlas::make_plan(kind, n_q_heads, n_kv_heads, head_dim, page_tokens, L, &plan) != ATLAS_OK)
        return SIZE_MAX;
    return plan.ws_bytes;
}

int32_t atlas_attn_split_tokens(atlas_kind kind, int32_t n_q_heads, int32_t n_kv_heads,
                                int32_t head_dim, int32_t page_tokens, const atlas_launch *L) {
    atlas::Plan plan;
    if (atlas::make_plan(kind, n_q_heads, n_kv_heads, head_dim, page_tokens, L, &plan) != ATLAS_OK)
        return -1;
    return plan.n_chunks > 0 && !plan.direct && !plan.cluster ? plan.chunk : 0;
}

const char *atlas_attn_status_string(atlas_status status) {
    switch (status) {
        case ATLAS_OK: return "ok";
        case ATLAS_ERR_INVALID_ARG: return "invalid argument";
        case ATLAS_ERR_UNSUPPORTED: return "unsupported head_dim, page_tokens or dtype";
        case ATLAS_ERR_WORKSPACE: return "workspace missing or too small";
        case ATLAS_ERR_CUDA: return "CUDA runtime or driver call failed";
        case ATLAS_ERR_DEVICE: return "a kernel reported a device-side error";
    }
    return "unknown status";
}

}  // extern "C"
