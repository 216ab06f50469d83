// split_kv.cu -- split-KV attention over paged K/V for few query rows per
// (sequence, kv head): decode (one row per q head) and short suffixes.
//
// Each CTA owns one (split of the key axis, kv head, sequence) and up to 8 or 16
// "columns" (q head of the GQA group x query row).  It folds its pages into an
// online-softmax state (m, l, acc) -- the page-by-page fold of the CFR-Atlas
// README (opening paragraph, "Core contract") -- and writes that partial state;
// merge.cu combines the splits (CPUAttn README, "Operator model": split-K only
// with a structured merge).
//
// bf16 path, per CTA: one producer warp gathers the split's pages through the
// page table with TMA loads (128-byte swizzle) into a STAGES-deep ring of
// 64-key K/V blocks -- pages of fewer than 64 tokens come in one box per page
// (a 3-D view [D/64 slabs][rows][64]), larger pages in one box per 64-column
// slab; four consumer warps each take 16 keys of every block and
// run both contractions on mma.sync tensor-core tiles with the keys on M:
//   S^T[16 keys x 8 cols]  = K[16 x D] . Q^T[D x 8]      (ldmatrix from the ring)
//   O^T[D x 8 cols]       += V^T[D x 16] . P^T[16 x 8]    (ldmatrix.trans; P^T via movmatrix)
// P is fed as bf16 hi + lo parts, so the PV product keeps ~16 bits of P.
// Column max / sum reductions are quad shuffles.
#include "internal.h"
#include "ptx.cuh"

#include <math.h>

namespace atlas {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kSplitThreads = (kConsumerWarps + 1) * 32;
constexpr int BT = kSplitBlockTokens;

__device__ __forceinline__ void record(uint32_t *status, uint32_t bit) {
    if (status) atomicOr(status, bit);
}

// qn: the sequence's query rows (q_lens[b] when ragged, else q_len).
__device__ __forceinline__ bool seq_len_bad(const SplitParams &p, int L, int qn) {
    return qn < 0 || qn > p.q_len || L < qn || L > p.max_pages * p.P ||
           (p.require_full && L != qn);
}

// Flat output row of column n of (b, hkv).
__device__ __forceinline__ int64_t column_row(const SplitParams &p, int b, int hkv, int n) {
    // q head hkv * G + n / q_len, row n % q_len: together (hkv * G) * q_len + n
    return ((int64_t)b * p.Hq + (int64_t)hkv * p.G) * p.q_len + n;
}

// Keys visible to column n (absolute count), as defined by the suffix rule.  L
// here is the sequence length shifted by q_len - qn (see split_prologue), so the
// same formula serves ragged batches.
__device__ __forceinline__ int column_visible(const SplitParams &p, int L, int n) {
    return L - p.q_len + (n % p.q_len) + 1;
}

// First key column n may see: the lower end of its window, or 0.
__device__ __forceinline__ int column_first(const SplitParams &p, int L, int n) {
    return p.window > 0 ? max(0, column_visible(p, L, n) - p.window) : 0;
}

// Score in log2 units from a raw dot product: scale (and the softcap, if any).
__device__ __forceinline__ float score_log2(const SplitParams &p, float raw) {
    return p.softcap_log2 > 0.f ? p.softcap_log2 * tanh_acc(raw * p.softcap_inv)
                                : raw * p.scale_log2;
}

// Direct mode (p.direct): NaN for every row of columns [col0, col0 + ncols) of
// (b, hkv) that is a query (all of them when `all_rows`, as for a bad seq_len).
__device__ void direct_nan_rows(const SplitParams &p, int b, int hkv, int col0, int ncols,
                                int qn, bool all_rows) {
    const float nan = __int_as_float(0x7fc00000);
    for (int idx = threadIdx.x; idx < ncols * p.D; idx += blockDim.x) {
        const int c = idx / p.D, d = idx % p.D;
        if (!all_rows && (col0 + c) % p.q_len >= qn) continue;
        const int64_t row = column_row(p, b, hkv, col0 + c);
        if (p.out_bf16)
            static_cast<__nv_bfloat16 *>(p.out)[row * p.D + d] = __float2bfloat16_rn(nan);
        else
            static_cast<float *>(p.out)[row * p.D + d] = nan;
        if (d == 0 && p.lse) p.lse[row] = nan;
    }
}

// Shared prologue: decides whether this CTA has work.  Returns false when the
// CTA must exit (nothing visible, or an error that has been recorded).
// Returns L shifted to L - qn + q_len: with it, row i (< qn) of a ragged sequence
// sits at position L_shifted - q_len + i = seq_len - qn + i, as in a full batch.
// Columns with row index >= qn are padding (qn out).
// Why split_prologue found no work for the CTA.
constexpr int kNoWork = 1;   // nothing of this split is visible to its columns
constexpr int kBadPage = 2;  // a page id outside the pool (recorded)
constexpr int kBadLen = 3;   // the sequence's seq_len / q_lens are invalid (recorded)

template <int NCOLS>
__device__ bool split_prologue(const SplitParams &p, int ct, int &L, int &kv_begin, int &kv_end,
                               int &col0, int &ncols, int &qn, int &why) {
    const int b = blockIdx.z;
    const int hkv = blockIdx.y / p.col_tiles;
    // A pass of a call spread over several launches computes some splits only.
    if (p.chunk_range &&
        ((int)blockIdx.x < p.chunk_range[2 * b] || (int)blockIdx.x >= p.chunk_range[2 * b + 1]))
        return false;
    L = p.seq_lens[b];
    qn = p.q_lens ? p.q_lens[b] : p.q_len;
    col0 = ct * NCOLS;
    ncols = min(NCOLS, p.G * p.q_len - col0);
    why = kNoWork;
    if (seq_len_bad(p, L, qn)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) record(p.status, ATLAS_DEV_BAD_SEQLEN);
        // split mode: the merge writes NaN rows for this sequence; cluster mode:
        // the cluster's rank 0 does
        if (p.direct) direct_nan_rows(p, b, hkv, col0, ncols, qn, true);
        why = kBadLen;
        return false;
    }
    L = L - qn + p.q_len;
    int i_max = -1, i_min = p.q_len;
    for (int c = 0; c < ncols; ++c) {
        const int i = (col0 + c) % p.q_len;
        if (i >= qn) continue;  // padding row of a ragged batch
        i_max = max(i_max, i);
        i_min = min(i_min, i);
    }
    if (i_max < 0) return false;  // only padding rows
    const int kv_hi = L - p.q_len + i_max + 1;
    // Keys below every column's window are skipped whole (64-key blocks).
    const int kv_lo = p.window > 0 ? max(0, L - p.q_len + i_min + 1 - p.window) : 0;
    kv_begin = max((int)blockIdx.x * p.chunk, kv_lo / kSplitBlockTokens * kSplitBlockTokens);
    kv_end = min(kv_hi, (int)blockIdx.x * p.chunk + p.chunk);
    if (kv_begin >= kv_end) return false;

    // Every page id this split will touch must be inside the pool.
    const int pg0 = kv_begin / p.P, pg1 = (kv_end - 1) / p.P;
    bool bad = false;
    for (int pg = pg0 + (int)threadIdx.x; pg <= pg1; pg += blockDim.x) {
        const int id = p.page_table[(int64_t)b * p.max_pages + pg];
        bad |= (id < 0 || id >= p.num_pages);
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) record(p.status, ATLAS_DEV_BAD_PAGE);
        why = kBadPage;
        if (p.direct) {
            direct_nan_rows(p, b, hkv, col0, ncols, qn, false);
            return false;
        }
        if (p.cluster) return false;  // a NaN state for this split, merged in the cluster
        for (int c = threadIdx.x; c < ncols; c += blockDim.x) {
            float *ml = p.ws_ml + (column_row(p, b, hkv, col0 + c) * p.n_chunks + blockIdx.x) * 2;
            ml[0] = __int_as_float(0x7fc00000);
            ml[1] = __int_as_float(0x7fc00000);
        }
        return false;
    }
    return true;
}

// Combine the per-warp states held in shared memory and write this split's
// partial (m, l, acc) for every valid column.  cm/cl: [W][NCOLS]; cacc: [W][NCOLS][D].
// Direct mode (one split covers the whole context): write the output row itself
// with the merge's arithmetic on that single state (the sink, if any, as one more
// state m = sink log2 e, l = 1, acc = 0), so the bits equal split + merge of it;
// padding rows of a ragged batch are not written.
// Cluster mode: the state (acc[D], m, l) of each column goes to `part` in this
// CTA's shared memory ([NCOLS][D + 2]) for the cluster merge.
template <int W, int NCOLS, int D>
__device__ void write_partials(const SplitParams &p, const float *cm, const float *cl,
                               const float *cacc, int col0, int ncols, int qn, bool failed,
                               float *part = nullptr) {
    const int b = blockIdx.z;
    const int hkv = blockIdx.y / p.col_tiles;
    if (p.direct && failed) {
        direct_nan_rows(p, b, hkv, col0, ncols, qn, false);
        return;
    }
    for (int idx = threadIdx.x; idx < NCOLS * D; idx += blockDim.x) {
        const int c = idx / D, d = idx % D;
        if (c >= ncols) continue;
        const int64_t row = column_row(p, b, hkv, col0 + c);
        const int64_t slot = row * p.n_chunks + blockIdx.x;
        if (part && failed) {
            part[c * (D + 2) + d] = __int_as_float(0x7fc00000);
            if (d == 0) part[c * (D + 2) + D] = part[c * (D + 2) + D + 1] = __int_as_float(0x7fc00000);
            continue;
        }
        if (failed) {
            if (d == 0) {
                p.ws_ml[slot * 2] = __int_as_float(0x7fc00000);
                p.ws_ml[slot * 2 + 1] = __int_as_float(0x7fc00000);
            }
            continue;
        }
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, cm[w * NCOLS + c]);
        float a = 0.f, l = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const float f = ex2(cm[w * NCOLS + c] - M);
                a += f * cacc[(w * NCOLS + c) * D + d];
                l += f * cl[w * NCOLS + c];
            }
        }
        if (part) {
            part[c * (D + 2) + d] = a;
            if (d == 0) {
                part[c * (D + 2) + D] = M;
                part[c * (D + 2) + D + 1] = l;
            }
            continue;
        }
        if (p.direct) {
            if ((col0 + c) % p.q_len >= qn) continue;  // padding row: not written
            const float sink2 = p.sinks ? p.sinks[(row / p.q_len) % p.Hq] * kLog2e : -INFINITY;
            float M2 = sink2;
            if (l > 0.f) M2 = fmaxf(M2, M);
            float o, lse;
            if (isnan(l) || isnan(M) || isnan(sink2) || M2 == -INFINITY) {
                o = lse = __int_as_float(0x7fc00000);
            } else {
                const float w = l > 0.f ? ex2(M - M2) : 0.f;
                const float lsum = fmaf(w, l, p.sinks ? ex2(sink2 - M2) : 0.f);
                o = fmaf(w, a, 0.f) / lsum;
                lse = kLn2 * (M2 + log2f(lsum));
            }
            if (p.out_bf16)
                static_cast<__nv_bfloat16 *>(p.out)[row * D + d] = __float2bfloat16_rn(o);
            else
                static_cast<float *>(p.out)[row * D + d] = o;
            if (d == 0 && p.lse) p.lse[row] = lse;
            continue;
        }
        p.ws_acc[slot * D + d] = a;
        if (d == 0) {
            p.ws_ml[slot * 2] = M;
            p.ws_ml[slot * 2 + 1] = l;
        }
    }
}

// 3-D tiled TMA load into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap *map, int32_t x,
                                                 int32_t y, int32_t z, uint32_t bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// Byte offset of block row r (0..63) in the ring layout the producer writes:
// rows come in boxes of 2^lg_br rows, each box holding all D/64 slabs of its rows.
template <int D>
__device__ __forceinline__ uint32_t box_row_offset(int r, int lg_br) {
    const uint32_t box = (uint32_t)r >> lg_br, in_box = (uint32_t)r & ((1u << lg_br) - 1u);
    return (((box << lg_br) * (D / 64)) + in_box) * 128u;
}

template <int D, int NT, int STAGES>
struct SplitLayout {
    static constexpr int kTile = BT * D * 2;           // one 64-key K or V block, bf16
    static constexpr int kStage = 2 * kTile;           // K then V
    static constexpr int kBars = STAGES * kStage;      // full[STAGES], empty[STAGES]
    static constexpr int kFlags = kBars + 2 * STAGES * 8;
    static constexpr int kBytes = kFlags + 16 + 1024;  // + alignment slack
    static constexpr int kCombine = kConsumerWarps * NT * 8 * (D + 2) * 4;
    static_assert(kCombine <= kBars, "combine scratch must fit in the ring");
};

template <int D, int NT, int STAGES>
__global__ void __launch_bounds__(kSplitThreads, 2)
    split_bf16_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
    allow_dependent_launch();  // the merge may start its CTAs (it waits for this grid)
    using Lay = SplitLayout<D, NT, STAGES>;
    constexpr int NCOLS = NT * 8;
    constexpr int KSTEPS = D / 16;
    constexpr int SLAB = BT * 128;  // bytes of one 64-element-wide slab of a block

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full0 = sbase + Lay::kBars;
    const uint32_t empty0 = full0 + STAGES * 8;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Lay::kFlags);

    int L, kv_begin, kv_end, col0, ncols, qn, why;
    if (!split_prologue<NCOLS>(p, blockIdx.y % p.col_tiles, L, kv_begin, kv_end, col0, ncols,
                               qn, why))
        return;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int b = blockIdx.z;
    const int hkv = blockIdx.y / p.col_tiles;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const int nblocks = (kv_end - kv_begin + BT - 1) / BT;
    bool failed = false;

    // Per-thread softmax state for columns nt*8 + 2*(lane%4) + {0,1}.
    float m_run[NT][2], l_run[NT][2];
    float acc[KSTEPS][NT][4];

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer warp
        // The whole warp walks the blocks (page ids from a warp-wide cache, one
        // coalesced table read per 32 pages); lanes 0..subs-1 issue the boxes.
        if (lane == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
        }
        const uint64_t policy = policy_evict_first();
        const int BR = p.P < BT ? p.P : BT;  // rows per box
        const int subs = BT / BR;           // boxes per block (<= 8)
        const int lp = 31 - __clz(p.P);     // log2(P)
        PageIdCache pages{p.page_table + (int64_t)b * p.max_pages, (kv_end - 1) >> lp};
        int issued = 0;
        for (int j = 0; j < nblocks; ++j) {
            const int s = j % STAGES;
            if (j >= STAGES &&
                !__all_sync(0xffffffffu, mbar_wait_bounded(empty0 + 8 * s, ((j / STAGES) - 1) & 1,
                                                           abort_flag, kWaitLimitNs))) {
                failed = true;
                break;
            }
            // A block starts on a multiple of 64 keys: with P <= 64 box sb is page
            // t0 / P + sb from its first row, else the block lies inside one page.
            // The block's pages share one 32-page line of the cache, so lane sb
            // finds its page with one shuffle.
            const int t0 = kv_begin + j * BT;
            const int nsub = min(subs, (kv_end - t0 + BR - 1) / BR);
            const int my_y =
                (pages.get_line(t0 >> lp, lane < nsub ? lane : 0) * p.Hkv + hkv) * p.P +
                ((t0 + (lane < nsub ? lane : 0) * BR) & (p.P - 1));
            if ((p.debug_flags & ATLAS_DEBUG_WITHHOLD_STAGE) && j == 0) continue;
            if (lane < nsub) {
                if (lane == 0)
                    mbar_arrive_expect_tx(full0 + 8 * s, (uint32_t)(nsub * BR * D * 2 * 2));
                __syncwarp((1u << nsub) - 1u);
                const uint32_t kdst = sbase + s * Lay::kStage;
                const uint32_t vdst = kdst + Lay::kTile;
                if (BR < BT) {
                    // One box per page: all D/64 slabs of its BR rows.
                    const uint32_t off = (uint32_t)(lane * BR * (D / 64) * 128);
                    tma_load_3d_hint(kdst + off, &tmK, 0, my_y, 0, full0 + 8 * s, policy);
                    tma_load_3d_hint(vdst + off, &tmV, 0, my_y, 0, full0 + 8 * s, policy);
                } else {
#pragma unroll
                    for (int slab = 0; slab < D / 64; ++slab) {
                        tma_load_2d_hint(kdst + slab * SLAB, &tmK, slab * 64, my_y, full0 + 8 * s,
                                         policy);
                        tma_load_2d_hint(vdst + slab * SLAB, &tmV, slab * 64, my_y, full0 + 8 * s,
                                         policy);
                    }
                }
            }
            __syncwarp();
            issued = j + 1;
        }
        if (failed && lane == 0) {
            *abort_flag = 1;
            // Let the copies already in flight land before the CTA exits.
            int no_abort = 0;
            for (int j = max(0, issued - STAGES); j < issued; ++j) {
                if ((p.debug_flags & ATLAS_DEBUG_WITHHOLD_STAGE) && j == 0) continue;
                mbar_wait_bounded(full0 + 8 * (j % STAGES), (j / STAGES) & 1,
                                  (volatile int *)&no_abort, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ consumer warps
        // Q^T as mma B fragments: element k = d, n = column lane/4.
        uint32_t qf[KSTEPS][NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int c = nt * 8 + lane / 4;
            const __nv_bfloat16 *qrow = nullptr;
            if (c < ncols) qrow = static_cast<const __nv_bfloat16 *>(p.q) +
                                   column_row(p, b, hkv, col0 + c) * D;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                const int d0 = kk * 16 + 2 * (lane % 4);
                qf[kk][nt][0] = qrow ? *reinterpret_cast<const uint32_t *>(qrow + d0) : 0u;
                qf[kk][nt][1] = qrow ? *reinterpret_cast<const uint32_t *>(qrow + d0 + 8) : 0u;
            }
        }
        // Visible key range [lo, lim) of each of this thread's score columns
        // (empty for padding columns).
        int lim[NT][2], lo[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int c = nt * 8 + 2 * (lane % 4) + e;
                const bool real = c < ncols && (col0 + c) % p.q_len < qn;
                lim[nt][e] = real ? min(kv_end, column_visible(p, L, col0 + c)) : 0;
                lo[nt][e] = real ? column_first(p, L, col0 + c) : 0;
                m_run[nt][e] = -INFINITY;
                l_run[nt][e] = 0.f;
            }
#pragma unroll
        for (int dt = 0; dt < KSTEPS; ++dt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[dt][nt][e] = 0.f;

        // Ring layout of a block: box b (rows b*BR .. b*BR+BR-1) at b * BR * D/64 * 128
        // bytes, slab-major inside (slab s at s * BR * 128), 128-byte rows swizzled by
        // row & 7 (BR >= 8).  With BR = 64 this is the plain slab-major tile.
        const int lg_br = 31 - __clz(p.P < BT ? p.P : BT);
        const uint32_t slab_step = 128u << lg_br;
        const int rk = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;  // K row of this lane
        const int rv = 16 * warp + (lane & 7) + (lane >> 4) * 8;         // V row of this lane
        const uint32_t row_k = box_row_offset<D>(rk, lg_br);
        const uint32_t row_v = box_row_offset<D>(rv, lg_br);
        for (int j = 0; j < nblocks; ++j) {
            const int s = j % STAGES;
            // Warp-uniform decision: the mma.sync below needs every lane.
            const bool landed = __all_sync(
                0xffffffffu, mbar_wait_bounded(full0 + 8 * s, (j / STAGES) & 1, abort_flag,
                                               kWaitLimitNs));
            if (!landed) {
                failed = true;
                *abort_flag = 1;
                break;
            }
            const int key0 = kv_begin + j * BT + 16 * warp;
            const int valid = kv_end - key0;
            if (valid > 0) {
                const uint32_t kt = sbase + s * Lay::kStage;
                const uint32_t vt = kt + Lay::kTile;
                // ---- S^T = K . Q^T
                float sc[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const int d = kk * 16 + (lane >> 4) * 8;
                    uint32_t a[4];
                    ldmatrix_x4(kt + row_k + (d / 64) * slab_step + ((((d % 64) / 8) ^ (rk & 7)) << 4),
                                a[0], a[1], a[2], a[3]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(sc[nt], a, qf[kk][nt][0],
                                                                   qf[kk][nt][1]);
                }
                // ---- mask, scale (log2 units), online softmax per column
                uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float pr[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = key0 + lane / 4 + 8 * (e >> 1);
                        sc[nt][e] = key < lim[nt][e & 1] && key >= lo[nt][e & 1]
                                        ? score_log2(p, sc[nt][e])
                                        : -INFINITY;
                    }
#pragma unroll
                    for (int ce = 0; ce < 2; ++ce) {
                        float mx = fmaxf(sc[nt][ce], sc[nt][ce + 2]);
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                        const float m_new = fmaxf(m_run[nt][ce], mx);
                        const float m_use = m_new == -INFINITY ? 0.f : m_new;
                        const float corr = ex2(m_run[nt][ce] - m_use);
                        pr[ce] = ex2(sc[nt][ce] - m_use);
                        pr[ce + 2] = ex2(sc[nt][ce + 2] - m_use);
                        l_run[nt][ce] = l_run[nt][ce] * corr + pr[ce] + pr[ce + 2];
                        m_run[nt][ce] = m_new;
#pragma unroll
                        for (int dt = 0; dt < KSTEPS; ++dt) {
                            acc[dt][nt][ce] *= corr;
                            acc[dt][nt][ce + 2] *= corr;
                        }
                    }
                    // P (rows = keys lane/4 and +8, cols 2*(lane%4)+{0,1}) as bf16 hi + lo,
                    // transposed into the B-fragment layout of the PV product.
                    const __nv_bfloat162 h01 = __floats2bfloat162_rn(pr[0], pr[1]);
                    const __nv_bfloat162 h23 = __floats2bfloat162_rn(pr[2], pr[3]);
                    const float2 f01 = __bfloat1622float2(h01);
                    const float2 f23 = __bfloat1622float2(h23);
                    bh[nt][0] = movmatrix_trans(*reinterpret_cast<const uint32_t *>(&h01));
                    bh[nt][1] = movmatrix_trans(*reinterpret_cast<const uint32_t *>(&h23));
                    bl[nt][0] = movmatrix_trans(pack_bf16(pr[0] - f01.x, pr[1] - f01.y));
                    bl[nt][1] = movmatrix_trans(pack_bf16(pr[2] - f23.x, pr[3] - f23.y));
                }
                // ---- O^T += V^T . P^T
                // Key index of the low half of a0/a1 (and +8 for a2/a3).
                const int kq = 2 * (lane % 4);
                uint32_t keep01 = 0xffffffffu, keep23 = 0xffffffffu;
                if (valid < 16) {
                    keep01 = (kq < valid ? 0x0000ffffu : 0u) | (kq + 1 < valid ? 0xffff0000u : 0u);
                    keep23 = (kq + 8 < valid ? 0x0000ffffu : 0u) |
                             (kq + 9 < valid ? 0xffff0000u : 0u);
                }
#pragma unroll
                for (int dt = 0; dt < KSTEPS; ++dt) {
                    const int d = dt * 16 + ((lane >> 3) & 1) * 8;
                    uint32_t a[4];
                    ldmatrix_x4_trans(vt + row_v + (d / 64) * slab_step +
                                          ((((d % 64) / 8) ^ (rv & 7)) << 4),
                                      a[0], a[1], a[2], a[3]);
                    // Keys past the split end may hold stale or NaN rows: zero them.
                    a[0] &= keep01;
                    a[1] &= keep01;
                    a[2] &= keep23;
                    a[3] &= keep23;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_bf16_16816(acc[dt][nt], a, bh[nt][0], bh[nt][1]);
                        mma_bf16_16816(acc[dt][nt], a, bl[nt][0], bl[nt][1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
        }
        // Full column sums: lanes sharing lane%4 hold the same columns.
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int ce = 0; ce < 2; ++ce) {
                float l = l_run[nt][ce];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                l_run[nt][ce] = l;
            }
    }

    const bool any_failed = __syncthreads_or(failed) != 0;
    if (any_failed && threadIdx.x == 0) record(p.status, ATLAS_DEV_TIMEOUT);

    // Reuse the ring as combine scratch (all loads have landed or been drained).
    float *cm = reinterpret_cast<float *>(smem);
    float *cl = cm + kConsumerWarps * NCOLS;
    float *cacc = cl + kConsumerWarps * NCOLS;
    if (!any_failed && warp < kConsumerWarps) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int ce = 0; ce < 2; ++ce) {
                const int c = nt * 8 + 2 * (lane % 4) + ce;
                if (lane < 4) {
                    cm[warp * NCOLS + c] = m_run[nt][ce];
                    cl[warp * NCOLS + c] = l_run[nt][ce];
                }
#pragma unroll
                for (int dt = 0; dt < KSTEPS; ++dt) {
                    const int d = dt * 16 + lane / 4;
                    cacc[(warp * NCOLS + c) * D + d] = acc[dt][nt][ce];
                    cacc[(warp * NCOLS + c) * D + d + 8] = acc[dt][nt][ce + 2];
                }
            }
    }
    __syncthreads();
    write_partials<kConsumerWarps, NCOLS, D>(p, cm, cl, cacc, col0, ncols, qn, any_failed);
}

// ---------------------------------------------------------------- cluster merge
// Cluster mode: the n_chunks splits of one (sequence, kv head, column tile) are the
// CTAs of one thread-block cluster (rank = split index).  Each CTA keeps its partial
// state in slot `rank` of a per-CTA array of kClusterSlots slots, and every CTA but
// rank 0 copies it into the same slot of rank 0 through distributed shared memory.
// After one cluster barrier, rank 0 alone applies the structured merge (CPUAttn
// README, "Operator model") to every output element, reading the slots locally,
// with the merge kernel's arithmetic in split order, so the bits equal split + merge;
// the other CTAs leave at that barrier.  No workspace, no second launch.
// Every CTA arrives on the cluster barrier at entry (nothing may write into a CTA
// of the cluster before all of them have started) and reaches both barrier phases
// on every path (no early exit in this mode); the loops before them are bounded.
constexpr int kClusterSlots = 8;  // the portable cluster size

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The first phase of the cluster barrier, split: every thread arrives at entry and
// waits just before its first write into another CTA.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_barrier() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16-byte store into the shared memory of CTA `rank` of this cluster, at the offset
// that `local` (a shared-memory address of this CTA) has in its own.
__device__ __forceinline__ void st_cluster_v4(uint32_t local, uint32_t rank, float4 v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// slots: this CTA's kClusterSlots x [NCOLS][D + 2] array; this CTA's state is in slot
// `rank` (written before the call).
template <int NCOLS, int D>
__device__ void cluster_merge(const SplitParams &p, float *slots, int col0, int ncols, int qn,
                              bool bad_len, int seq_len) {
    constexpr int kSlot = NCOLS * (D + 2);  // floats, a multiple of 4
    static_assert(kSlot % 4 == 0, "16-byte slot copies");
    const uint32_t rank = cluster_ctarank();
    __syncthreads();  // this CTA's state is in its slot
    cluster_wait();   // every CTA of the cluster has started
    if (rank != 0) {
        const float4 *mine = reinterpret_cast<const float4 *>(slots + rank * kSlot);
        const uint32_t dst = smem_u32(slots + rank * kSlot);
        for (int i = threadIdx.x; i < kSlot / 4; i += blockDim.x)
            st_cluster_v4(dst + (uint32_t)i * 16u, 0u, mine[i]);
    }
    cluster_barrier();  // rank 0 sees every split's state
    if (rank != 0) return;
    const int b = blockIdx.z;
    const int hkv = blockIdx.y / p.col_tiles;
    const int L = seq_len;  // seq_lens[b], read at the kernel's start
    for (int idx = threadIdx.x; idx < ncols * D; idx += blockDim.x) {
        const int c = idx / D, d = idx % D;
        const int i = (col0 + c) % p.q_len;
        if (!bad_len && i >= qn) continue;  // padding row: not written
        const int64_t row = column_row(p, b, hkv, col0 + c);
        float o = __int_as_float(0x7fc00000), lse = o;
        if (!bad_len) {
            const int visible = L - qn + i + 1;
            // splits holding this row's keys: [first, nsplit)
            const int first = p.window > 0 ? max(0, visible - p.window) / p.chunk : 0;
            const int nsplit = min((visible + p.chunk - 1) / p.chunk, p.n_chunks);
            float m[kClusterSlots], l[kClusterSlots], a[kClusterSlots];
#pragma unroll
            for (int u = 0; u < kClusterSlots; ++u) {
                m[u] = l[u] = a[u] = 0.f;
                if (first + u < nsplit) {
                    const float *st = slots + (first + u) * kSlot + c * (D + 2);
                    m[u] = st[D];
                    l[u] = st[D + 1];
                    a[u] = st[d];
                }
            }
            const float sink2 = p.sinks ? p.sinks[(row / p.q_len) % p.Hq] * kLog2e : -INFINITY;
            float M = sink2;
            bool has_nan = isnan(sink2);
#pragma unroll
            for (int u = 0; u < kClusterSlots; ++u) {
                if (first + u >= nsplit) break;
                if (isnan(l[u]) || isnan(m[u])) has_nan = true;
                else if (l[u] > 0.f) M = fmaxf(M, m[u]);
            }
            if (!has_nan && M != -INFINITY) {
                float lsum = p.sinks ? ex2(sink2 - M) : 0.f, acc = 0.f;
#pragma unroll
                for (int u = 0; u < kClusterSlots; ++u) {
                    if (first + u >= nsplit) break;
                    const float w = l[u] > 0.f ? ex2(m[u] - M) : 0.f;
                    lsum = fmaf(w, l[u], lsum);
                    acc = fmaf(w, a[u], acc);
                }
                o = acc / lsum;
                lse = kLn2 * (M + log2f(lsum));
            }
        }
        if (p.out_bf16)
            static_cast<__nv_bfloat16 *>(p.out)[row * D + d] = __float2bfloat16_rn(o);
        else
            static_cast<float *>(p.out)[row * D + d] = o;
        if (d == 0 && p.lse) p.lse[row] = lse;
    }
}

// ---------------------------------------------------------------- f32 path
// Few columns per (sequence, kv head) in fp32 (decode, short suffixes).  Each of
// the W warps streams its own 8-key K/V blocks (blocks w, w+W, ... of the split)
// into a private double-buffered ring by cp.async and keeps its own online-softmax
// state per column; the warps' states are combined at the end.  Scores: lane l
// takes key l % 8 of the block and column group l / 8 (a quarter of the columns)
// and forms whole D-long dot products from shared memory, so every score and
// every exponential is computed once.  PV: lanes split the head dimension and read
// P back from shared memory.  Keys past the split's end are zero-filled, never read.
constexpr int kF32Keys = 8;

// Warps per CTA of the split form: each warp holds ~17 KB of rings (D = 128), so
// 4-warp CTAs three to an SM keep 12 warps resident where 8-warp CTAs fit one; the
// kernel is latency-bound (dependent shuffles, exponentials and shared-memory round
// trips per 8-key block), and 12 warps measured 25-31 % faster than 8.  16 columns
// need ~205 registers a thread, more than three CTAs allow.
template <int D, int NC>
struct F32Layout {
    static constexpr int W = NC == 16 ? 8 : 4;
    static constexpr int kMinCtas = NC == 16 ? 1 : 3;
    static constexpr int KS = D + 4;                      // padded row stride (floats)
    static constexpr int kBuf = kF32Keys * KS;            // one K or V block
    static constexpr int kWarp = 4 * kBuf + kF32Keys * NC;  // K[2], V[2], P[key][col]
    static constexpr int kQ = NC * KS;
    static constexpr int kBytes = (kQ + W * kWarp) * 4;
    // cluster mode only, after the rings: kClusterSlots splits' states, each
    // [NC][D + 2] (rank 0 merges them; every other CTA uses its own slot only)
    static constexpr int kPartBytes = kClusterSlots * NC * (D + 2) * 4;
    static_assert(kBytes + kPartBytes <= 232448, "shared memory budget (cluster mode)");
    static_assert(2 * W * NC + W * NC * D <= W * kWarp, "combine scratch fits the rings");
};

template <int D, int NC>
__global__ void __launch_bounds__(F32Layout<D, NC>::W * 32, F32Layout<D, NC>::kMinCtas)
    split_f32_kernel(const SplitParams p) {
    allow_dependent_launch();  // the merge may start its CTAs (it waits for this grid)
    using Lay = F32Layout<D, NC>;
    constexpr int W = Lay::W, BK = kF32Keys, DPL = D / 32, NQ = NC / 4, DV4 = D / 4;
    extern __shared__ __align__(16) float f32d_smem[];
    float *sQ = f32d_smem;
    float *sW = sQ + Lay::kQ;
    float *slots = sW + W * Lay::kWarp;  // cluster mode only
    if (p.cluster) cluster_arrive_relaxed();  // first phase, waited on before any remote write
    float *part = p.cluster ? slots + cluster_ctarank() * (NC * (D + 2)) : nullptr;

    const int b = blockIdx.z;
    const int hkv = blockIdx.y / p.col_tiles;
    // A short call is a chain of dependent memory round trips, so the reads that do
    // not depend on seq_len start now, before the prologue waits for it: the CTA's
    // query rows (cp.async; columns past the tile's end are zero-filled, padding rows
    // of a ragged batch load too and are masked with their keys) and, into L2, the
    // page-table entries of this split.
    const int seq_len_b = p.seq_lens[b];
    {
        const int c0 = (int)(blockIdx.y % p.col_tiles) * NC;
        const int nc = min(NC, p.G * p.q_len - c0);
        for (int idx = threadIdx.x; idx < NC * DV4; idx += W * 32) {
            const int c = idx / DV4, d4 = idx % DV4;
            const bool in = c < nc;
            const float *src = static_cast<const float *>(p.q) +
                               column_row(p, b, hkv, c0 + (in ? c : 0)) * D + 4 * d4;
            cp_async16(smem_u32(sQ + c * Lay::KS + 4 * d4), src, in ? 16u : 0u);
        }
        cp_async_commit();
        const int pg0 = (int)blockIdx.x * p.chunk / p.P;
        const int npg = min(p.chunk / p.P, p.max_pages - pg0);
        if ((int)threadIdx.x * 32 < npg)
            prefetch_l2(p.page_table + (int64_t)b * p.max_pages + pg0 + threadIdx.x * 32);
    }
    int L = 0, kv_begin = 0, kv_end = 0, col0 = 0, ncols = 0, qn = 0, why = 0;
    const bool work = split_prologue<NC>(p, blockIdx.y % p.col_tiles, L, kv_begin, kv_end, col0,
                                         ncols, qn, why);
    if (!work) cp_async_wait<0>();  // no copy in flight when the CTA leaves
    if (!work && !p.cluster) return;
    if (!work) {
        // an empty state (m = -inf, l = 0, acc = 0), or NaN after a bad page id
        const float nan = __int_as_float(0x7fc00000);
        for (int idx = threadIdx.x; idx < NC * (D + 2); idx += W * 32)
            part[idx] = why == kBadPage ? nan : (idx % (D + 2) == D ? -INFINITY : 0.f);
        cluster_merge<NC, D>(p, slots, col0, ncols, qn, why == kBadLen, seq_len_b);
        return;
    }
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const float *kp = static_cast<const float *>(p.k_pages);
    const float *vp = static_cast<const float *>(p.v_pages);
    const int32_t *ptab = p.page_table + (int64_t)b * p.max_pages;

    int lim[NC], lo[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const bool ok = c < ncols && (col0 + c) % p.q_len < qn;
        lim[c] = ok ? min(kv_end, column_visible(p, L, col0 + c)) : kv_begin;
        lo[c] = ok ? column_first(p, L, col0 + c) : 0;
    }

    float *wK = sW + warp * Lay::kWarp;
    float *wV = wK + 2 * Lay::kBuf;
    float *wP = wK + 4 * Lay::kBuf;
    const int lp = 31 - __clz(p.P);  // log2(P): P is a power of two
    auto load = [&](int kb, int buf) {
        const uint32_t kd = smem_u32(wK + buf * Lay::kBuf), vd = smem_u32(wV + buf * Lay::kBuf);
        for (int idx = lane; idx < BK * DV4; idx += 32) {
            const int kr = idx / DV4, d4 = idx % DV4;
            const int t = kb + kr;
            const bool in = t < kv_end;
            const int tt = in ? t : kv_begin;
            const int64_t row =
                ((int64_t)ptab[tt >> lp] * p.Hkv + hkv) * p.P + (tt & (p.P - 1));
            const uint32_t off = (uint32_t)(kr * Lay::KS + 4 * d4) * 4u;
            cp_async16(kd + off, kp + row * D + 4 * d4, in ? 16u : 0u);
            cp_async16(vd + off, vp + row * D + 4 * d4, in ? 16u : 0u);
        }
    };

    float acc[NC][DPL], m_run[NC], l_part[NQ];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        m_run[c] = -INFINITY;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[c][e] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < NQ; ++i) l_part[i] = 0.f;

    const int nblk = (kv_end - kv_begin + BK - 1) / BK;
    const int key = lane % BK, grp = lane / BK;
    // limits of this lane's columns grp*NQ + i (selected with constant indices)
    int limh[NQ], loh[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        limh[i] = grp == 0 ? lim[i] : grp == 1 ? lim[NQ + i] : grp == 2 ? lim[2 * NQ + i]
                                                                          : lim[3 * NQ + i];
        loh[i] = grp == 0 ? lo[i] : grp == 1 ? lo[NQ + i] : grp == 2 ? lo[2 * NQ + i]
                                                                     : lo[3 * NQ + i];
    }
    int j = warp;
    if (j < nblk) load(kv_begin + j * BK, 0);
    cp_async_commit();
    cp_async_wait<1>();  // the query rows (the group before this one) have landed
    __syncthreads();     // ... and every warp sees them
    for (int it = 0; j < nblk; ++it, j += W) {
        const int kb = kv_begin + j * BK;
        const int buf = it & 1;
        if (j + W < nblk) load(kb + W * BK, buf ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncwarp();
        const float *cK = wK + buf * Lay::kBuf;
        const float *cV = wV + buf * Lay::kBuf;

        // scores of this lane's key for columns grp*NQ .. grp*NQ + NQ - 1, each as four
        // partial sums (d mod 4) so that the FMAs form 4*NQ independent chains
        float s4[NQ][4];
#pragma unroll
        for (int i = 0; i < NQ; ++i)
#pragma unroll
            for (int u = 0; u < 4; ++u) s4[i][u] = 0.f;
#pragma unroll 8
        for (int d = 0; d < D; d += 4) {
            const float4 k4 = *reinterpret_cast<const float4 *>(cK + key * Lay::KS + d);
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
                const float4 q4 =
                    *reinterpret_cast<const float4 *>(sQ + (grp * NQ + i) * Lay::KS + d);
                s4[i][0] = fmaf(q4.x, k4.x, s4[i][0]);
                s4[i][1] = fmaf(q4.y, k4.y, s4[i][1]);
                s4[i][2] = fmaf(q4.z, k4.z, s4[i][2]);
                s4[i][3] = fmaf(q4.w, k4.w, s4[i][3]);
            }
        }
        float s[NQ];
#pragma unroll
        for (int i = 0; i < NQ; ++i) s[i] = (s4[i][0] + s4[i][1]) + (s4[i][2] + s4[i][3]);
        const int t = kb + key;
        float corr[NC];
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            s[i] = (t < limh[i] && t >= loh[i]) ? score_log2(p, s[i]) : -INFINITY;
            float mx = s[i];
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            // block maxima of columns g*NQ + i from the lanes of group g
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int cc = g * NQ + i;
                const float m_new = fmaxf(m_run[cc], __shfl_sync(0xffffffffu, mx, g * BK));
                const float mref = m_new == -INFINITY ? 0.f : m_new;
                corr[cc] = ex2(m_run[cc] - mref);  // 0 while nothing was visible
                m_run[cc] = m_new;
            }
        }
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            const float mr = grp == 0 ? m_run[i] : grp == 1 ? m_run[NQ + i]
                             : grp == 2 ? m_run[2 * NQ + i] : m_run[3 * NQ + i];
            const float cr = grp == 0 ? corr[i] : grp == 1 ? corr[NQ + i]
                             : grp == 2 ? corr[2 * NQ + i] : corr[3 * NQ + i];
            const float pv = ex2(s[i] - (mr == -INFINITY ? 0.f : mr));
            l_part[i] = fmaf(l_part[i], cr, pv);
            wP[key * NC + grp * NQ + i] = pv;
        }
        __syncwarp();
        // O += P V, lanes over the head dimension
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[c][e] *= corr[c];
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float pk[NC];
#pragma unroll
            for (int c4 = 0; c4 < NC; c4 += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(wP + kk * NC + c4);
                pk[c4] = v.x;
                pk[c4 + 1] = v.y;
                pk[c4 + 2] = v.z;
                pk[c4 + 3] = v.w;
            }
            float vv[DPL];
            if (DPL == 4) {
                const float4 v = *reinterpret_cast<const float4 *>(cV + kk * Lay::KS + lane * DPL);
                vv[0] = v.x;
                vv[1] = v.y;
                vv[2 % DPL] = v.z;
                vv[3 % DPL] = v.w;
            } else {
                const float2 v = *reinterpret_cast<const float2 *>(cV + kk * Lay::KS + lane * DPL);
                vv[0] = v.x;
                vv[1] = v.y;
            }
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
                for (int e = 0; e < DPL; ++e) acc[c][e] = fmaf(pk[c], vv[e], acc[c][e]);
        }
        __syncwarp();  // P and this buffer are rewritten by the next iteration
    }
    cp_async_wait<0>();
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        l_part[i] += __shfl_xor_sync(0xffffffffu, l_part[i], 1);
        l_part[i] += __shfl_xor_sync(0xffffffffu, l_part[i], 2);
        l_part[i] += __shfl_xor_sync(0xffffffffu, l_part[i], 4);
    }
    __syncthreads();  // every warp is done with its ring: reuse it for the combine
    float *cm = sW, *cl = sW + W * NC, *cacc = sW + 2 * W * NC;
    if (lane == 0) {
#pragma unroll
        for (int c = 0; c < NC; ++c) cm[warp * NC + c] = m_run[c];
    }
    if (key == 0) {
#pragma unroll
        for (int i = 0; i < NQ; ++i) cl[warp * NC + grp * NQ + i] = l_part[i];
    }
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int e = 0; e < DPL; ++e) cacc[(warp * NC + c) * D + lane * DPL + e] = acc[c][e];
    __syncthreads();
    if (p.cluster) {
        write_partials<W, NC, D>(p, cm, cl, cacc, col0, ncols, qn, false, part);
        cluster_merge<NC, D>(p, slots, col0, ncols, qn, false, seq_len_b);
        return;
    }
    write_partials<W, NC, D>(p, cm, cl, cacc, col0, ncols, qn, false);
}

template <int D, int NT, int STAGES>
cudaError_t launch_bf16_instance(const SplitParams &p, const CUtensorMap &tmK,
                                 const CUtensorMap &tmV, cudaStream_t stream) {
    using Lay = SplitLayout<D, NT, STAGES>;
    auto kern = split_bf16_kernel<D, NT, STAGES>;
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !configured[dev]) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
        if (err != cudaSuccess) return err;
        configured[dev] = 1;
    }
    dim3 grid(p.n_chunks, p.Hkv * p.col_tiles, p.B);
    kern<<<grid, kSplitThreads, Lay::kBytes, stream>>>(tmK, tmV, p);
    return cudaGetLastError();
}

}  // namespace

int split_bf16_cols_per_cta(int G, int q_len) { return G * q_len <= 8 ? 8 : 16; }

cudaError_t launch_split_bf16(const SplitParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                              cudaStream_t stream) {
    const bool wide = split_bf16_cols_per_cta(p.G, p.q_len) == 16;
    if (p.D == 128) {
        return wide ? launch_bf16_instance<128, 2, 3>(p, tmK, tmV, stream)
                    : launch_bf16_instance<128, 1, 3>(p, tmK, tmV, stream);
    }
    return wide ? launch_bf16_instance<64, 2, 4>(p, tmK, tmV, stream)
                : launch_bf16_instance<64, 1, 4>(p, tmK, tmV, stream);
}

template <int D, int NC>
cudaError_t launch_f32_instance(const SplitParams &p, cudaStream_t stream) {
    using Lay = F32Layout<D, NC>;
    auto kern = split_f32_kernel<D, NC>;
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !configured[dev]) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   Lay::kBytes + Lay::kPartBytes);
        if (err != cudaSuccess) return err;
        configured[dev] = 1;
    }
    dim3 grid(p.n_chunks, p.Hkv * p.col_tiles, p.B);
    if (!p.cluster) {
        kern<<<grid, Lay::W * 32, Lay::kBytes, stream>>>(p);
        return cudaGetLastError();
    }
    // one cluster per (sequence, kv head, column tile): its n_chunks (<= 8) splits
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(Lay::W * 32, 1, 1);
    cfg.dynamicSmemBytes = Lay::kBytes + Lay::kPartBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.n_chunks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

int split_f32_cols_per_cta(int G, int q_len) {
    const int n = G * q_len;
    return n <= 4 ? 4 : n <= 8 ? 8 : 16;
}

cudaError_t launch_split_f32(const SplitParams &p, cudaStream_t stream) {
    const int nc = split_f32_cols_per_cta(p.G, p.q_len);
    if (p.D == 128) {
        return nc == 4   ? launch_f32_instance<128, 4>(p, stream)
               : nc == 8 ? launch_f32_instance<128, 8>(p, stream)
                         : launch_f32_instance<128, 16>(p, stream);
    }
    return nc == 4   ? launch_f32_instance<64, 4>(p, stream)
           : nc == 8 ? launch_f32_instance<64, 8>(p, stream)
                     : launch_f32_instance<64, 16>(p, stream);
}

}  // namespace atlas
