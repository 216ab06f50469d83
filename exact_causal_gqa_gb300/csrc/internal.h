// internal.h -- parameter blocks and launchers shared by the host entry points
// (atlas_attn.cu) and the kernel translation units.  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "atlas_attn.h"

namespace atlas {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// A bounded wait gives up after this long and reports ATLAS_DEV_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Keys per pipeline stage of the split-KV kernels.
constexpr int kSplitBlockTokens = 64;

// Balanced split geometry of the tensor-core path: a context of L keys is cut into
// n = ceil(L / chunk) splits of round_up(ceil(L / n), 128) keys (the last one
// shorter), split s covering keys [s * size, (s + 1) * size).  The kernels and the
// merge derive it from seq_lens alike.
__host__ __device__ inline int balanced_split(int L, int chunk) {
    const int Lc = L < 1 ? 1 : L;
    const int n = (Lc + chunk - 1) / chunk;
    const int per = (Lc + n - 1) / n;
    return (per + 127) / 128 * 128;
}
// Largest batch whose splits the tensor-core kernels order longest-first (each CTA
// ranks the batch's sequences itself).
constexpr int kTcOrderMaxSeqs = 128;

// Everything the split-KV kernels (bf16 mma.sync and f32) and the merge need.
// "Columns" are the query rows one (sequence, kv head) owns: column n is q head
// g = n / q_len of the group and query row i = n % q_len.
struct SplitParams {
    const void *q;              // [B][Hq][q_len][D]
    const void *k_pages;        // f32 path reads the pools directly
    const void *v_pages;
    const int32_t *page_table;  // [B][max_pages]
    const int32_t *seq_lens;    // [B]
    int32_t B, Hq, Hkv, G, D, P, q_len, max_pages, num_pages;
    int32_t chunk;              // keys per split (multiple of 64)
    int32_t n_chunks;           // splits per (sequence, kv head): ceil(max_pages*P / chunk)
    int32_t col_tiles;          // ceil(G*q_len / columns per CTA)
    int32_t require_full;       // prefill: seq_len must equal q_len
    float scale_log2;           // scale * log2(e)
    int32_t window;             // > 0: keys pos - window < t <= pos only
    float softcap_log2;         // > 0: s2 = softcap_log2 * tanh(raw * softcap_inv)
    float softcap_inv;          // scale / softcap
    const int32_t *q_lens;      // [B] ragged query rows (<= q_len) or null
    const int32_t *chunk_range; // [B][2] splits [lo, hi) this launch computes, or null (all)
    float *ws_acc;              // [B*Hq*q_len][n_chunks][D]   unnormalised accumulators
    float *ws_ml;               // [B*Hq*q_len][n_chunks][2]   (m in log2 units, l)
    uint32_t *status;           // may be null
    uint32_t debug_flags;
    // Direct mode (bf16): one split covers the whole context; the split kernel
    // writes the output rows itself (no workspace, no merge).
    int32_t direct;
    // Cluster mode (f32): the n_chunks (<= 8) splits of one (sequence, kv head,
    // column tile) run as one thread-block cluster and merge through distributed
    // shared memory; rank 0 writes the output rows (no workspace, no merge launch).
    int32_t cluster;
    void *out;
    int32_t out_bf16;
    float *lse;
    const float *sinks;         // [Hq] natural-log logits or null (direct mode only)
};

struct MergeParams {
    const int32_t *seq_lens;
    int32_t B, Hq, D, q_len, max_pages, P, chunk, n_chunks, require_full;
    int32_t balanced;           // splits of balanced_split(seq_len, chunk) keys
    int32_t window;             // splits below a row's window hold nothing for it
    const float *sinks;         // [Hq] natural-log logits or null: one more state (m, 1, 0)
    const int32_t *q_lens;      // [B] ragged query rows or null; padding rows untouched
    const float *ws_acc;
    const float *ws_ml;
    void *out;
    int32_t out_bf16;
    float *lse;
    int32_t sms;            // SM count: sizes the warps per row
    int32_t warps_per_row;  // set by launch_merge
};

// Tensor-core (tcgen05 / TMEM) path for many query rows per (sequence, kv head):
// 128-row query tiles x 128-key blocks (bf16) or 64-key blocks (fp32 as 3 x tf32),
// head_dim 64 or 128.  Either writes the
// normalised output directly (one CTA per tile, all its keys) or, when there are
// too few tiles to fill the GPU, split partials in the SplitParams layout.
struct TcParams {
    const int32_t *page_table;
    const int32_t *seq_lens;
    int32_t B, Hq, Hkv, G, D, P, q_len, max_pages, num_pages;
    int32_t tiles_per_unit;   // ceil(G * q_len / 128)
    int32_t tiles_per_head;   // q_len / 128 when q_len % 128 == 0 (heavy-first order), else 0
    int32_t split;            // 1: write split partials; 0: write the output
    int32_t chunk, n_chunks;  // split geometry (chunk a multiple of 128)
    int32_t balanced;         // split mode: balanced splits in longest-first order
                              // (tc_order.cuh); the grid's CTAs are work items
    int32_t require_full;
    int32_t hilo_below;       // tiles whose rows see fewer keys use a hi+lo split of P
    int32_t negate_scores;    // scale < 0: S = -Q K^T with |scale| (keeps the max exact)
    float scale_log2;         // |scale| * log2(e)
    int32_t window;           // > 0: keys pos - window < t <= pos only
    float softcap_log2;       // > 0: s2 = softcap_log2 * tanh(raw * softcap_inv)
    float softcap_inv;        // |scale| / softcap
    const float *sinks;       // [Hq] or null (direct mode folds it into the epilogue)
    const int32_t *q_lens;    // [B] ragged query rows (<= q_len) or null
    const int32_t *chunk_range;  // split mode: [B][2] splits [lo, hi) to compute, or null
    void *out;
    int32_t out_bf16;
    float *lse;
    float *ws_acc, *ws_ml;
    uint32_t *status;
    int32_t sms;         // SM count (sizes the persistent prefill grid)
};

// Paged KV append (kv_append.cu).
struct AppendParams {
    const void *k_new, *v_new;  // [B][Hkv][max_new][D]
    void *k_pages, *v_pages;    // [num_pages][Hkv][P][D]
    const int32_t *page_table, *seq_lens, *n_new;
    int32_t B, Hkv, max_new, P, max_pages, num_pages, row_bytes;
    uint32_t *status;
};
cudaError_t launch_kv_append(const AppendParams &p, cudaStream_t stream);

cudaError_t launch_fmha_tc(const TcParams &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                           const CUtensorMap &tmV, cudaStream_t stream);
// The same for fp32 q/K/V: three tf32 products per fp32 product (fmha_tc_f32.cu).
cudaError_t launch_fmha_tc_f32(const TcParams &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                               const CUtensorMap &tmV, cudaStream_t stream);

// Columns handled by one CTA of the bf16 split kernel.
int split_bf16_cols_per_cta(int G, int q_len);

cudaError_t launch_split_bf16(const SplitParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                              cudaStream_t stream);
// fp32 with few columns: 4, 8 or 16 columns per CTA by G x q_len.
int split_f32_cols_per_cta(int G, int q_len);
cudaError_t launch_split_f32(const SplitParams &p, cudaStream_t stream);
cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream);

// Multiprocessor count of the current device (cached per device); 152 (one
// GB300) when no device is visible.
int device_sm_count();

// The split plan of a call: which kernel path, split geometry and workspace.  A
// pure function of the call's sizes and the SM count (atlas_launch.sm_count, else
// device_sm_count()).
enum class Path { SplitBF16, SplitF32, TensorCore, TensorCoreF32 };

struct Plan {
    Path path;
    int direct;   // bf16 split kernel: one split, output written directly
    int cluster;  // f32 split kernel: splits merged inside one thread-block cluster
    int balanced; // tensor-core split mode: equal splits per sequence, longest first
    int chunk, n_chunks, col_tiles, G;
    int tc_split, tiles_per_unit, tiles_per_head;
    size_t acc_bytes, ml_offset, ws_bytes;
};

atlas_status make_plan(atlas_kind kind, int32_t Hq, int32_t Hkv, int32_t D, int32_t P,
                       const atlas_launch *L, Plan *plan);

}  // namespace atlas
