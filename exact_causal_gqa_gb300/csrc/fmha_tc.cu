// fmha_tc.cu -- causal prefill and suffix-query attention on the 5th-generation
// tensor cores (tcgen05 + TMEM), fed by TMA from the page pool.
//
// A CTA owns NT (1 or 2) 128-row query tiles of one (sequence, kv head).  Tile
// rows are the G*q_len (q head, query row) pairs of the GQA group in memory
// order: one q head's 128 consecutive prompt rows (prefill) or all G heads x SQ
// rows (suffix, G*SQ = 128).  With NT = 2 the two tiles are two q heads of the
// same group at the same prompt rows, so they need exactly the same K/V blocks:
// each block is loaded once for both, and the tensor core works on one tile
// while the other tile's softmax runs.  The CTA walks 128-key blocks up to the
// last key any of its rows may see -- later blocks are never loaded (causal
// block skipping, CPUAttn README: the fused QK -> RowNorm -> PV tile pipeline
// stops at the last reachable K block) -- and folds each block into per-row
// online-softmax state (the page fold of the CFR-Atlas README, "Core contract").
// A direct prefill with more tile pairs than SMs runs persistent CTAs instead (the
// PERSIST instance): one per SM, each walking its share of the tile pairs with every
// role's barrier phases running on from one item to the next.
//
// Warp roles (128 + NT*128 threads, one CTA per SM):
//   warp 0    TMA producer: the Q tiles once, then K blocks gathered page by page
//             through the page table into a KV_STAGES-deep ring.
//   warp 3    TMA producer of the V ring (the same pages).  With one producer for
//             both rings, its per-block work (page lookups, up to 32 box copies
//             for 8-token pages) was the longest step of the suffix's pipeline.
//   warp 1    allocates TMEM; one lane issues the MMAs:
//               S  = Q K^T  (M=128, N=128, K=D; A and B from smem)  -> TMEM
//               O += P V    (M=128, N=D, K=128; A = P from TMEM, B = V from smem)
//             for head_dim D = 64 or 128 (one or two 64-element slabs per row).
//   warp 2    zeroes V rows past the last key of the final block (they may be
//             NaN-poisoned or stale, and 0 * NaN would reach O).
//   warps 4+  one softmax warpgroup per tile, one thread per query row: read the
//             S row from TMEM, mask, row max, ex2, row sum; rescale O in TMEM
//             when the row max grew by more than 2^8 (exact: acc and l always
//             share the reference max); write P as bf16 over its own S columns
//             (plus the bf16 remainder P - bf16(P) for tiles whose rows see few
//             keys, so that PV keeps ~16 bits of P there); the row max comes from
//             the TMEM loads themselves (tcgen05.ld.red).  Epilogue: O / l, written
//             row by row through shared memory (persistent CTAs: straight from
//             registers, the next item's Q being on its way into that memory).
// Every mbarrier wait is bounded; a CTA that gives up records ATLAS_DEV_TIMEOUT,
// lets its copies and MMAs finish, frees TMEM and writes NaN.
#include "internal.h"
#include "ptx.cuh"
#include "tc_order.cuh"

#include <math.h>

namespace atlas {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per block
constexpr int kMaxItems = 64;  // work items of one CTA in persistent mode
constexpr int kSlab = 128 * 128;  // one 64-element slab of a 128-row bf16 tile (128-byte rows)
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows 256x
// A block takes P as bf16 hi + lo when, for some row of the tile, its largest weight
// exceeds w = 1/12 of a lower bound of the row's total (sum so far + that weight).
// Below it the single bf16 rounding of P stays well inside the 2e-3 bound: against the
// fp64 oracle on outlier and sharp-score inputs (K rows x3..x16 on 0.2-2 % of keys,
// |scale| sqrt(D) up to the 1.25 above which every block takes hi + lo, 2048-key
// prefill and 3000-5000-key suffix rows) the largest error was 7.4e-4 at w = 1/12,
// 5.4e-4 at 1/20, 1.2e-3 at 1/10, while rows dominated by a few keys reach ~1e-2 with
// no hi + lo at all.  The test runs in the log domain against log2(w / (1 - w)).
constexpr float kLog2HiLo = -3.4594316f;  // log2(1/11)

// One work item of a CTA: NT query tiles of one (sequence, kv head) over one key
// range (all of it, or one split).
struct TcWork {
    int b, hkv, c, t0, tstep;  // tiles t0 + x * tstep, x < NT; split c
    int qn, L, rows_unit;      // query rows of the sequence; shifted length; G * q_len
    int kv_begin, kv_end, nb;  // key range and its 128-key blocks
    bool hilo, tail_fix;       // hi + lo P on every block; last block partly past kv_end
    int tail_first;            // first key row of the last block past kv_end
    int state;                 // 0: compute; 1: nothing to compute; 2: bad seq_len
};

template <int NT, int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static constexpr int kSlabs = D / 64;             // 64-element slabs per row
    static constexpr int kTileBytes = 128 * D * 2;    // a 128-row bf16 tile (Q, K or V)
    // K/V ring depth: the same bytes in flight for either head_dim
    static constexpr int kStages = (NT == 2 ? 2 : 3) * (128 / D);
    static constexpr int kSB = NT == 2 ? 1 : 2;      // S buffers per tile
    // warps 0-3: K producer (and Q), MMA issuer, tail fix-up, V producer; then NT softmax
    // warpgroups.  Each SMSP holds 16K registers and 3 of the 12 warps (NT = 2):
    // 168 registers per thread.
    static constexpr int kSoftmaxWarp0 = 4;
    static constexpr int kThreads = 32 * kSoftmaxWarp0 + NT * 128;
    static constexpr int OFF_Q = 0;
    // V stages below K stages: the PV product's MN-major B descriptor strides by a
    // 16 KB slab, and every address it can form stays inside the allocation.
    static constexpr int OFF_V = OFF_Q + NT * kTileBytes;
    static constexpr int OFF_K = OFF_V + kStages * kTileBytes;
    static constexpr int OFF_BAR = OFF_K + kStages * kTileBytes;
    // barrier indices
    static constexpr int B_Q = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_KEMPTY = B_KFULL + kStages;
    static constexpr int B_VFULL = B_KEMPTY + kStages;
    static constexpr int B_VEMPTY = B_VFULL + kStages;
    static constexpr int B_SFULL = B_VEMPTY + kStages;  // [NT][kSB]
    static constexpr int B_PFULL = B_SFULL + NT * kSB;  // [NT]
    static constexpr int B_PVDONE = B_PFULL + NT;       // [NT]
    static constexpr int B_TAIL_READY = B_PVDONE + NT;  // single use
    static constexpr int B_TAIL = B_TAIL_READY + 1;     // single use
    static constexpr int B_FINAL = B_TAIL + 1;
    static constexpr int B_QEMPTY = B_FINAL + 1;  // an item's last S products done (Q free)
    static constexpr int B_OFREE = B_QEMPTY + 1;  // [NT] an item's O read out (BM arrivals)
    static constexpr int kBars = B_OFREE + NT;
    static constexpr int OFF_TMEM = OFF_BAR + kBars * 8;
    static constexpr int OFF_FLAG = OFF_TMEM + 8;
    // [NT][2] words of 4 bytes, one byte per warp of the tile: "this block needs P as
    // hi + lo", double-buffered by block parity
    static constexpr int OFF_VOTE = OFF_FLAG + 8;
    // the CTA's work items (persistent mode: up to kMaxItems), written once at the start
    static constexpr int kItemSlots = NT == 2 ? kMaxItems : 1;
    static constexpr int OFF_MASK = OFF_VOTE + 16;  // [2] words: items with a bad page id
    static constexpr int OFF_ITEMS = OFF_MASK + 8;
    static constexpr int kSmem = OFF_ITEMS + kItemSlots * (int)sizeof(TcWork) + 1024;  // + slack
    static_assert(kSmem <= 232448, "shared memory budget");
    // TMEM columns: NT=2 -> [S0 | O0 | S1 | O1]; NT=1 -> [S(buf 0) | S(buf 1) | O]
    __device__ static constexpr uint32_t s_col(int x, int b) {
        return NT == 2 ? (uint32_t)x * 256u : (uint32_t)b * 128u;
    }
    __device__ static constexpr uint32_t o_col(int x) {
        return NT == 2 ? (uint32_t)x * 256u + 128u : 256u;
    }
};

// As umma_bf16_tmem_a, with the output rows (TMEM lanes) whose bit is set in
// mask[lane / 32] left unchanged.
__device__ __forceinline__ void umma_bf16_tmem_a_masked(uint32_t d_tmem, uint32_t a_tmem,
                                                        uint64_t b_desc, uint32_t idesc,
                                                        const uint32_t (&mask)[4]) {
    asm volatile(
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, {%4, %5, %6, %7}, 1;" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(mask[0]), "r"(mask[1]), "r"(mask[2]),
        "r"(mask[3])
        : "memory");
}

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort, kWaitLimitNs));
}

__device__ __forceinline__ int64_t tile_row(const TcParams &p, int b, int hkv, int f) {
    return ((int64_t)b * p.Hq + (int64_t)hkv * p.G) * p.q_len + f;
}

// NaN for row f of (b, hkv) in direct mode.
template <int D>
__device__ void nan_row(const TcParams &p, int b, int hkv, int f) {
    const int64_t row = tile_row(p, b, hkv, f);
    const float nan = __int_as_float(0x7fc00000);
    if (p.out_bf16) {
        uint4 v;
        v.x = v.y = v.z = v.w = 0x7fc07fc0u;
        uint4 *o = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + row * D);
        for (int k = 0; k < D / 8; ++k) o[k] = v;
    } else {
        float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + row * D);
        for (int k = 0; k < D / 4; ++k) o[k] = make_float4(nan, nan, nan, nan);
    }
    if (p.lse) p.lse[row] = nan;
}

template <int NT>
__device__ TcWork tc_work(const TcParams &p, int u, int c, int t0, int tstep, int split_keys) {
    TcWork w{};
    w.b = u / p.Hkv;
    w.hkv = u % p.Hkv;
    w.c = c;
    w.t0 = t0;
    w.tstep = tstep;
    const int seq_len = p.seq_lens[w.b];
    w.qn = p.q_lens ? p.q_lens[w.b] : p.q_len;  // query rows of this sequence
    w.rows_unit = p.G * p.q_len;
    // Both tiles cover the same prompt rows, so their key ranges agree.
    const int f0 = t0 * BM;
    const int f_last = min(f0 + BM, w.rows_unit) - 1;
    const bool spans = (f_last / p.q_len) != (f0 / p.q_len);
    const int i_min = spans ? 0 : f0 % p.q_len;
    if (w.qn < 0 || w.qn > p.q_len || seq_len < w.qn || seq_len > p.max_pages * p.P ||
        (p.require_full && seq_len != w.qn)) {
        w.state = 2;
        return w;
    }
    if (i_min >= w.qn) {  // only padding rows of a ragged sequence
        w.state = 1;
        return w;
    }
    // Last real row of the tiles; with L shifted by q_len - qn, row i sits at
    // position L - q_len + i = seq_len - qn + i as in a full batch.
    const int i_max = min(spans ? p.q_len - 1 : f_last % p.q_len, w.qn - 1);
    w.L = seq_len - w.qn + p.q_len;
    const int kv_hi = w.L - p.q_len + i_max + 1;  // keys the tiles' last row sees
    // Keys the tiles' first row sees (its window may cut that short).
    const int kv_min = p.window > 0 ? min(w.L - p.q_len + i_min + 1, p.window)
                                    : w.L - p.q_len + i_min + 1;
    // Blocks below every row's window are skipped whole.
    const int kv_lo = p.window > 0 ? max(0, w.L - p.q_len + i_min + 1 - p.window) / BN * BN : 0;
    w.kv_begin = kv_lo;
    w.kv_end = kv_hi;
    if (p.split) {
        w.kv_begin = max(c * split_keys, kv_lo);
        w.kv_end = min(kv_hi, c * split_keys + split_keys);
        if (w.kv_begin >= w.kv_end) {
            w.state = 1;
            return w;
        }
    }
    w.nb = (w.kv_end - w.kv_begin + BN - 1) / BN;
    w.hilo = kv_min < p.hilo_below;
    const int last_kb = w.kv_begin + (w.nb - 1) * BN;
    w.tail_fix = w.kv_end < last_kb + BN;
    w.tail_first = w.kv_end - last_kb;
    return w;
}

// Direct mode: item r of the heavy-first order (the latest prompt rows first).
template <int NT>
__device__ void tc_direct_item(const TcParams &p, int r, int &u, int &t0, int &tstep) {
    const int units = p.B * p.Hkv;
    if (p.tiles_per_head > 0) {
        const int heads = p.G / NT;  // head groups of NT heads
        const int per = units * heads;
        const int rest = r % per;
        u = rest / heads;
        const int qi = p.tiles_per_head - 1 - r / per;
        t0 = (rest % heads) * NT * p.tiles_per_head + qi;
        tstep = p.tiles_per_head;
    } else {
        u = r % units;
        t0 = r / units;
        tstep = 0;
    }
}

// Persistent mode: the i-th item of CTA k of `ctas`, snake order over the
// heavy-first list (a heavy item pairs with a light one in the next pass).
__device__ __forceinline__ int tc_persist_item(int k, int i, int ctas) {
    return i * ctas + ((i & 1) ? ctas - 1 - k : k);
}

template <int NT, int D, bool PERSIST>
__global__ void __launch_bounds__(Cfg<NT, D>::kThreads, 1)
    fmha_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const TcParams p) {
    allow_dependent_launch();  // the merge may start its CTAs (it waits for this grid)
    using C = Cfg<NT, D>;
    constexpr int S = C::kStages, SB = C::kSB;
    constexpr int kTileBytes = C::kTileBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEM);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#define BAR(i) (sb + C::OFF_BAR + 8u * (uint32_t)(i))

    // ------------------------------------------------------------ work items
    // One item in the grid-per-item modes.  Persistent mode (direct prefill, two
    // tiles per CTA): this CTA's items in a snake order over the heavy-first list;
    // every role walks them, and the barrier phases run on across items (counted in
    // blocks and items), so the next item's Q, K/V and first S products overlap the
    // current item's last blocks and epilogue.
    int n_items = 1;
    TcWork w0{};
    if (PERSIST) {
        const int total = p.B * p.Hkv * (p.G / NT) * p.tiles_per_head;
        n_items = 0;
        while (n_items < kMaxItems && tc_persist_item(blockIdx.x, n_items, gridDim.x) < total)
            ++n_items;
    } else {
        int u, c, t0, tstep;
        int split_keys = p.chunk;  // keys per split (split mode)
        if (p.split && p.balanced) {
            // longest-first work item (the V ring is free until the producer starts)
            const TcItem it = tc_balanced_item(p, blockIdx.x + blockIdx.y * gridDim.x,
                                               reinterpret_cast<int *>(smem + C::OFF_V));
            if (it.b < 0) return;
            c = it.split;
            u = it.b * p.Hkv + it.hkv;
            t0 = it.tile;
            tstep = 0;
            split_keys = it.split_keys;
        } else if (p.split) {
            c = blockIdx.x;
            u = blockIdx.y / p.tiles_per_unit;
            t0 = blockIdx.y % p.tiles_per_unit;
            tstep = 0;
        } else {
            c = 0;
            tc_direct_item<NT>(p, blockIdx.x, u, t0, tstep);
        }
        // A pass of a call spread over several launches computes some splits only.
        const int b = u / p.Hkv;
        if (p.split && p.chunk_range &&
            (c < p.chunk_range[2 * b] || c >= p.chunk_range[2 * b + 1]))
            return;
        w0 = tc_work<NT>(p, u, c, t0, tstep, split_keys);
    }
    TcWork *const items = reinterpret_cast<TcWork *>(smem + C::OFF_ITEMS);
    // Items not computed (bit set): a bad seq_len or a page id outside the pool (rows
    // NaN), or nothing to compute.  The page ids of every item's key range are
    // checked by the whole CTA at once; the result is the same in every thread.
    uint32_t *bad_words = reinterpret_cast<uint32_t *>(smem + C::OFF_MASK);
    if (threadIdx.x == 0) bad_words[0] = bad_words[1] = 0u;
    __syncthreads();
    uint64_t skip = 0, bad = 0;
    for (int it = 0; it < n_items; ++it) {
        TcWork w = w0;
        if (PERSIST) {
            int u, t0, tstep;
            tc_direct_item<NT>(p, tc_persist_item(blockIdx.x, it, gridDim.x), u, t0, tstep);
            w = tc_work<NT>(p, u, 0, t0, tstep, p.chunk);
            if (threadIdx.x == 0) items[it] = w;  // read by every role after the barriers
        }
        if (w.state != 0) {
            skip |= 1ull << it;
            continue;
        }
        const int pg0 = w.kv_begin / p.P, pg1 = (w.kv_end - 1) / p.P;
        for (int pg = pg0 + (int)threadIdx.x; pg <= pg1; pg += blockDim.x) {
            const int id = p.page_table[(int64_t)w.b * p.max_pages + pg];
            if (id < 0 || id >= p.num_pages) bad |= 1ull << it;
        }
    }
    if (bad) {
        atomicOr(bad_words, (uint32_t)bad);
        atomicOr(bad_words + 1, (uint32_t)(bad >> 32));
    }
    __syncthreads();
    const uint64_t bad_page = bad_words[0] | ((uint64_t)bad_words[1] << 32);
    skip |= bad_page;
    for (int it = 0; skip && it < n_items; ++it) {
        if (!((skip >> it) & 1)) continue;
        const TcWork &w = PERSIST ? items[it] : w0;
        if (w.state == 2) {
            if (threadIdx.x == 0 && w.c == 0 && p.status) atomicOr(p.status, ATLAS_DEV_BAD_SEQLEN);
            const int rows_valid = (w.qn >= 0 && w.qn <= p.q_len) ? w.qn : p.q_len;
            if (!p.split && threadIdx.x < NT * BM) {
                const int f = (w.t0 + (int)(threadIdx.x / BM) * w.tstep) * BM + threadIdx.x % BM;
                if (f < w.rows_unit && f % p.q_len < rows_valid) nan_row<D>(p, w.b, w.hkv, f);
            }
            // split mode: the merge writes NaN rows for this sequence
        } else if ((bad_page >> it) & 1) {
            if (threadIdx.x == 0 && p.status) atomicOr(p.status, ATLAS_DEV_BAD_PAGE);
            if (threadIdx.x < NT * BM) {
                const int f = (w.t0 + (int)(threadIdx.x / BM) * w.tstep) * BM + threadIdx.x % BM;
                if (f < w.rows_unit && f % p.q_len < w.qn) {
                    if (!p.split) {
                        nan_row<D>(p, w.b, w.hkv, f);
                    } else {
                        float *ml =
                            p.ws_ml + (tile_row(p, w.b, w.hkv, f) * p.n_chunks + w.c) * 2;
                        ml[0] = ml[1] = __int_as_float(0x7fc00000);
                    }
                }
            }
        }
    }
    if (skip == (n_items == 64 ? ~0ull : (1ull << n_items) - 1)) return;

    // ------------------------------------------------------------ setup
    if (threadIdx.x == 0) {
        mbar_init(BAR(C::B_Q), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(BAR(C::B_KFULL + s), 1);
            mbar_init(BAR(C::B_KEMPTY + s), 1);
            mbar_init(BAR(C::B_VFULL + s), 1);
            mbar_init(BAR(C::B_VEMPTY + s), 1);
        }
        for (int k = 0; k < NT * SB; ++k) mbar_init(BAR(C::B_SFULL + k), 1);
        for (int x = 0; x < NT; ++x) {
            mbar_init(BAR(C::B_PFULL + x), BM);
            mbar_init(BAR(C::B_PVDONE + x), 1);
        }
        mbar_init(BAR(C::B_TAIL_READY), 1);
        mbar_init(BAR(C::B_TAIL), 1);
        mbar_init(BAR(C::B_FINAL), 1);
        mbar_init(BAR(C::B_QEMPTY), 1);
        for (int x = 0; x < NT; ++x) mbar_init(BAR(C::B_OFREE + x), BM);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool failed = false;

    if (warp == 0 || warp == 3) {
        // -------------------------------------------------------- TMA producers
        // Warp 0 streams Q and the K ring, warp 3 the V ring, each through its own
        // warp-wide page-id cache.  A block starts on a multiple of 128 keys and P (a
        // power of two <= 128) divides that, so box bx of a block is page
        // kb / P + bx from its first row, and a block's pages lie in one 32-page line
        // of the cache: lane bx looks its page up with one shuffle and issues box bx.
        const int kv = warp == 0 ? 0 : 1;
        if (lane == 0) {
            prefetch_tmap(kv == 0 ? &tmK : &tmV);
            if (kv == 0) prefetch_tmap(&tmQ);
        }
        const CUtensorMap *map = kv == 0 ? &tmK : &tmV;
        const uint32_t ring = sb + (kv == 0 ? C::OFF_K : C::OFF_V);
        const int bar_full = kv == 0 ? C::B_KFULL : C::B_VFULL;
        const int bar_empty = kv == 0 ? C::B_KEMPTY : C::B_VEMPTY;
        const int lp = 31 - __clz(p.P);  // log2(P)
        int g = 0;   // blocks of this ring issued so far (all items)
        int nq = 0;  // Q tile pairs loaded so far
        for (int it = 0; it < n_items && !failed; ++it) {
            if ((skip >> it) & 1) continue;
            const TcWork &w = PERSIST ? items[it] : w0;
            if (kv == 0) {
                // The previous item's Q tiles are free once its last S products are done.
                if (nq > 0 && !wait_warp(BAR(C::B_QEMPTY), (nq - 1) & 1, abort_flag)) {
                    failed = true;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(BAR(C::B_Q), NT * kTileBytes);
                    for (int x = 0; x < NT; ++x) {
                        const int qrow = (int)tile_row(p, w.b, w.hkv, (w.t0 + x * w.tstep) * BM);
#pragma unroll
                        for (int sl = 0; sl < C::kSlabs; ++sl)
                            tma_load_2d(sb + C::OFF_Q + x * kTileBytes + sl * kSlab, &tmQ,
                                        64 * sl, qrow, BAR(C::B_Q));
                    }
                }
                ++nq;
            }
            PageIdCache pages{p.page_table + (int64_t)w.b * p.max_pages, (w.kv_end - 1) >> lp};
            for (int j = 0; j < w.nb; ++j) {
                const int s = g % S, use = g / S;
                const int kb = w.kv_begin + j * BN;
                const int nbox = (min(BN, w.kv_end - kb) + p.P - 1) >> lp;  // <= 16
                const int y =
                    (pages.get_line(kb >> lp, lane < nbox ? lane : 0) * p.Hkv + w.hkv) << lp;
                if (use > 0 && !wait_warp(BAR(bar_empty + s), (use - 1) & 1, abort_flag)) {
                    failed = true;
                    break;
                }
                if (lane < nbox) {
                    if (lane == 0)
                        mbar_arrive_expect_tx(BAR(bar_full + s),
                                              (uint32_t)(nbox << lp) * 128u * C::kSlabs);
                    __syncwarp((1u << nbox) - 1u);
#pragma unroll
                    for (int sl = 0; sl < C::kSlabs; ++sl)
                        tma_load_2d(ring + s * kTileBytes + sl * kSlab + (lane << lp) * 128, map,
                                    64 * sl, y, BAR(bar_full + s));
                }
                __syncwarp();
                ++g;
            }
        }
        if (failed && lane == 0) {
            *abort_flag = 1;
            int no_abort = 0;
            // Let the copies in flight land before the CTA's shared memory goes away.
            if (kv == 0 && nq > 0)
                mbar_wait_bounded(BAR(C::B_Q), (nq - 1) & 1, &no_abort, kWaitLimitNs);
            for (int k = max(0, g - S); k < g; ++k)
                mbar_wait_bounded(BAR(bar_full + k % S), (k / S) & 1, &no_abort, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(128, 128, false, p.negate_scores != 0);
            constexpr uint32_t idPV = idesc_bf16_f32(128, D, true);
            bool ok = true;
            int g = 0;      // blocks of earlier items
            int nq = 0;     // items so far
            int ntail = 0;  // tail fix-ups so far
            for (int it = 0; ok && it < n_items; ++it) {
                if ((skip >> it) & 1) continue;
                const TcWork &w = PERSIST ? items[it] : w0;
                const int nb = w.nb;
                ok = mbar_wait_bounded(BAR(C::B_Q), nq & 1, abort_flag, kWaitLimitNs);
                tc_fence_after();
                if (!ok) break;
                // S_x(j) = Q_x K_j^T into S buffer (g + j) % SB of tile x.  Tile 0 waits
                // for K_j; the last tile releases its stage, and after the item's last
                // block also the Q tiles.
                auto issue_s = [&](int j, int x) -> bool {
                    const int G = g + j, s = G % S;
                    if (x == 0) {
                        if (!mbar_wait_bounded(BAR(C::B_KFULL + s), (G / S) & 1, abort_flag,
                                               kWaitLimitNs))
                            return false;
                        tc_fence_after();
                    }
                    // Descriptors built once per operand base; the K slices step through
                    // the 14-bit address field (16-byte units), which no smem offset here
                    // can carry out of.
                    const uint64_t kd = sdesc_sw128(sb + C::OFF_K + s * kTileBytes, 16, 1024);
                    const uint64_t qd = sdesc_sw128(sb + C::OFF_Q + x * kTileBytes, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = ((kk >> 2) * kSlab + (kk & 3) * 32) >> 4;
                        umma_bf16(tmem + C::s_col(x, G % SB), qd + off, kd + off, idS, kk > 0);
                    }
                    umma_commit(BAR(C::B_SFULL + x * SB + G % SB));
                    if (x == NT - 1) {
                        umma_commit(BAR(C::B_KEMPTY + s));
                        if (j == nb - 1) umma_commit(BAR(C::B_QEMPTY));
                    }
                    return true;
                };
                for (int j = 0; ok && j < min(SB, nb); ++j)
#pragma unroll
                    for (int x = 0; x < NT; ++x)
                        if (ok) ok = issue_s(j, x);
                for (int j = 0; ok && j < nb; ++j) {
                    const int G = g + j, s = G % S;
#pragma unroll
                    for (int x = 0; x < NT; ++x) {
                        if (!mbar_wait_bounded(BAR(C::B_PFULL + x), G & 1, abort_flag,
                                               kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        if (x == 0) {
                            if (!mbar_wait_bounded(BAR(C::B_VFULL + s), (G / S) & 1, abort_flag,
                                                   kWaitLimitNs)) {
                                ok = false;
                                break;
                            }
                            if (j == nb - 1 && w.tail_fix) {
                                // Hand the landed last V block to the fix-up warp (only
                                // this thread observes every phase of the V ring in order).
                                mbar_arrive(BAR(C::B_TAIL_READY));
                                if (!mbar_wait_bounded(BAR(C::B_TAIL), ntail & 1, abort_flag,
                                                       kWaitLimitNs)) {
                                    ok = false;
                                    break;
                                }
                                ++ntail;
                            }
                        }
                        // The item's first PV overwrites O: the previous item's
                        // epilogue must have read it out.
                        if (j == 0 && nq > 0 &&
                            !mbar_wait_bounded(BAR(C::B_OFREE + x), (nq - 1) & 1, abort_flag,
                                               kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t vd =
                            sdesc_sw128(sb + C::OFF_V + s * kTileBytes, kSlab, 1024);
                        const uint32_t pcol = tmem + C::s_col(x, G % SB);
                        // keys 16kk .. 16kk+15 of P sit in columns 32*(kk/2) + 8*(kk%2) ..
                        // +8, their remainders 16 columns further on.  V slice kk starts
                        // 2048 bytes (128 descriptor units) after slice kk-1.
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_bf16_tmem_a(tmem + C::o_col(x),
                                             pcol + (kk >> 1) * 32 + (kk & 1) * 8,
                                             vd + kk * 128u, idPV, (j > 0 || kk > 0) ? 1u : 0u);
                        // The softmax's vote for this block (one byte per warp, written
                        // before its P arrival), read once the hi products are queued so
                        // its latency hides there.  The lo product leaves the rows of
                        // warps that did not ask for it unchanged: their lo columns hold
                        // no P.
                        const uint32_t vote = *reinterpret_cast<volatile uint32_t *>(
                            smem + C::OFF_VOTE + (x * 2 + (G & 1)) * 4);
                        if (w.hilo || vote != 0u) {
                            uint32_t off_lanes[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                off_lanes[q] =
                                    (w.hilo || ((vote >> (8 * q)) & 0xffu)) ? 0u : 0xffffffffu;
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk)
                                umma_bf16_tmem_a_masked(tmem + C::o_col(x),
                                                        pcol + (kk >> 1) * 32 + 16 + (kk & 1) * 8,
                                                        vd + kk * 128u, idPV, off_lanes);
                        }
                        umma_commit(BAR(C::B_PVDONE + x));
                        // The V stage is free once the last tile's PV has read it: release
                        // it before S_x(j + SB) waits for its K block.
                        if (x == NT - 1) umma_commit(BAR(C::B_VEMPTY + s));
                        // Ping-pong: S_x(j + SB) follows PV_x(j) at once, so tile x starts
                        // its next softmax while the other tile's P is still being made.
                        // It writes the S buffer that PV_x(j) reads P_x(j) from; the
                        // tcgen05.mma operations of one thread run in issue order, so
                        // PV_x(j) has read its operand before S_x(j + SB) writes there.
                        if (j + SB < nb && !issue_s(j + SB, x)) {
                            ok = false;
                            break;
                        }
                    }
                }
                g += nb;
                ++nq;
            }
            if (!ok) {
                failed = true;
                *abort_flag = 1;
            }
            // Every MMA issued so far completes before TMEM is released.
            umma_commit(BAR(C::B_FINAL));
            int no_abort = 0;
            mbar_wait_bounded(BAR(C::B_FINAL), 0, &no_abort, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 2) {
        // -------------------------------------------------------- tail fix-up
        int g = 0, ntail = 0;
        for (int it = 0; it < n_items && !failed; ++it) {
            if ((skip >> it) & 1) continue;
            const TcWork &w = PERSIST ? items[it] : w0;
            if (w.tail_fix) {
                const int s = (g + w.nb - 1) % S;
                if (wait_warp(BAR(C::B_TAIL_READY), ntail & 1, abort_flag)) {
                    const uint32_t vbase = sb + C::OFF_V + s * kTileBytes;
                    constexpr int kChunks = 8 * C::kSlabs;  // 16-byte chunks per V row
                    for (int idx = lane; idx < (BN - w.tail_first) * kChunks; idx += 32) {
                        const int row = w.tail_first + idx / kChunks, q = idx % kChunks;
                        st_shared_v4(vbase + (q / 8) * kSlab + row * 128 + (q % 8) * 16, 0u, 0u,
                                     0u, 0u);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(C::B_TAIL));
                    ++ntail;
                } else {
                    failed = true;
                }
            }
            g += w.nb;
        }
    } else if (warp >= C::kSoftmaxWarp0) {
        // -------------------------------------------------------- softmax
        // Four consecutive warps cover the four TMEM lane quadrants (warp % 4).
        const int x = (warp - C::kSoftmaxWarp0) / 4;  // tile of this warpgroup
        const int q4 = warp % 4;                      // TMEM lane quadrant
        const int r = q4 * 32 + lane;
        const bool capped = p.softcap_log2 > 0.f;
        const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;  // 32-byte stores
        const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
        const uint32_t to = tl + C::o_col(x);
        bool ok = true;
        int g = 0;  // blocks of earlier items
        int it = 0;
        for (; ok && it < n_items; ++it) {
        if ((skip >> it) & 1) continue;
        const TcWork &w = PERSIST ? items[it] : w0;
        const int b = w.b, hkv = w.hkv, c = w.c, kv_begin = w.kv_begin, nb = w.nb;
        const bool hilo = w.hilo;
        const int f = (w.t0 + x * w.tstep) * BM + r;
        const bool valid = f < w.rows_unit && f % p.q_len < w.qn;  // padding rows: no queries
        const int i = valid ? f % p.q_len : 0;
        const int lim_row = valid ? min(w.L - p.q_len + i + 1, w.kv_end) : 0;
        const int lo_row =
            (valid && p.window > 0) ? max(0, w.L - p.q_len + i + 1 - p.window) : 0;
        float m_used = -INFINITY, l = 0.f;
        float log2_l = -INFINITY;  // log2(l), refreshed at the end of each block
        for (int j = 0; j < nb; ++j) {
            const int G = g + j;  // block count over the CTA's items: barrier phases
            const int bsel = G % SB;
            if (!wait_warp(BAR(C::B_SFULL + x * SB + bsel), (G / SB) & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t ts = tl + C::s_col(x, bsel);
            const int nvis = lim_row - (kv_begin + j * BN);  // visible columns: [nlo, nvis)
            const int nlo = lo_row - (kv_begin + j * BN);
            // Padding rows of a ragged batch never reach the output: they may take the
            // unmasked path (their O and l are garbage but stay in their own row).
            const bool all_visible = __all_sync(0xffffffffu, !valid || (nvis >= BN && nlo <= 0));
            // A masked block, quarter by quarter (32 keys), for all the warp's real rows:
            // wholly masked (bit in q_none: nothing loaded, P = 0), wholly visible (bit in
            // q_full: the unmasked code), or mixed.  On the causal diagonal the quarters
            // before a warp's own rows are visible and those after them masked.
            int q_full = 0, q_none = 0;
            if (!all_visible) {
                const int hi = min(max(nvis, 0), BN), lo = min(max(nlo, 0), BN);
                const int hi_min = __reduce_min_sync(0xffffffffu, valid ? hi : BN);
                const int hi_max = __reduce_max_sync(0xffffffffu, valid ? hi : 0);
                const int lo_min = __reduce_min_sync(0xffffffffu, valid ? lo : BN);
                const int lo_max = __reduce_max_sync(0xffffffffu, valid ? lo : 0);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    if (32 * cc >= hi_max || 32 * cc + 32 <= lo_min) q_none |= 1 << cc;
                    else if (32 * cc >= lo_max && 32 * cc + 32 <= hi_min) q_full |= 1 << cc;
                }
            }
            // Pass 1: row max of the raw scores (scale_log2 >= 0, so the scaled
            // maximum is the maximum scaled), one per quarter, then combined.
            // Outer loops stay rolled: a fully unrolled body overflows the
            // instruction cache shared with the producer and MMA warps.
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (all_visible) {
                // The loads reduce as they read (tcgen05.ld.red): each returns its 32
                // columns' maximum (the wait names the loaded registers, which the load
                // writes until then).  Two loads in flight at a time measured slower.
                uint32_t ma[32];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    tmem_ld32_max(ts + cc * 32, ma, m4[cc]);
                    tmem_wait_ld32_max(ma, m4[cc]);
                }
            } else {
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    if ((q_none >> cc) & 1) continue;
                    uint32_t sr[32];
                    float qm;
                    tmem_ld32_max(ts + cc * 32, sr, qm);
                    tmem_wait_ld32_max(sr, qm);
                    if ((q_full >> cc) & 1) {
                        m4[0] = fmaxf(m4[0], qm);
                        continue;
                    }
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const int col = cc * 32 + e;
                        const float v0 =
                            col < nvis && col >= nlo ? __uint_as_float(sr[e]) : -INFINITY;
                        const float v1 = col + 1 < nvis && col + 1 >= nlo
                                             ? __uint_as_float(sr[e + 1])
                                             : -INFINITY;
                        m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], v0, v1);
                    }
                }
            }
            // (a padding row keeps m = -inf: it never asks for an O rescale)
            const float mraw = valid ? fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) : -INFINITY;
            // the softcap is increasing, so it maps the raw maximum to the maximum
            const float mx = mraw == -INFINITY ? -INFINITY
                             : capped ? p.softcap_log2 * tanh_acc(mraw * p.softcap_inv)
                                      : mraw * p.scale_log2;
            float corr = 1.f, log2_corr = 0.f;
            if (mx > m_used + kRescaleThreshold) {
                log2_corr = m_used - mx;  // -inf on the first visible block
                corr = ex2(log2_corr);    // 0 there
                m_used = mx;
            }
            const float mref = m_used == -INFINITY ? 0.f : m_used;
            // hi + lo P for this block?  Static per tile; else each warp decides for
            // its 32 rows and leaves its vote for the MMA thread (read after this
            // warp's P arrival), which multiplies the lo part for the rows of the warps
            // that asked for it.
            bool split_blk = hilo;
            if (!hilo) {
                // largest weight maxp = 2^(mx - mref) against w (l corr + maxp), in the
                // log domain (no exponential on this path): log2 maxp > log2(w / (1 - w))
                // + log2 l + log2 corr.  l = 0 gives -inf on the right: always hi + lo.
                const bool need = mx - mref > kLog2HiLo + log2_l + log2_corr;
                split_blk = __any_sync(0xffffffffu, need);
                if (lane == 0)
                    smem[C::OFF_VOTE + (x * 2 + (G & 1)) * 4 + q4] = split_blk ? 1 : 0;
            }

            // Pass 2: P = 2^(s * scale_log2 - m) as bf16 pairs, written over columns
            // of S already read (see quarter() below), and the row sum.
            float2 rs2[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) rs2[k] = make_float2(0.f, 0.f);
            const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
            const float2 nm2 = make_float2(-mref, -mref);
            // Keys 2k, 2k+1 of quarter cc (columns 32cc..32cc+31 of S) -> P pair k,
            // written to column 32cc + k and its remainder (hi + lo blocks) to column
            // 32cc + 16 + k: the quarter's own S columns, read just before.
            auto quarter = [&](const uint32_t (&sr)[32], int cc, uint32_t (&hw)[16],
                               uint32_t (&lw)[16], bool masked, bool split, bool cap) {
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float2 t;
                    if (cap) {
                        t.x = p.softcap_log2 * tanh_acc(__uint_as_float(sr[2 * k]) *
                                                        p.softcap_inv) - mref;
                        t.y = p.softcap_log2 * tanh_acc(__uint_as_float(sr[2 * k + 1]) *
                                                        p.softcap_inv) - mref;
                    } else {
                        t = ffma2(make_float2(__uint_as_float(sr[2 * k]),
                                              __uint_as_float(sr[2 * k + 1])),
                                  sc2, nm2);
                    }
                    if (masked) {
                        const int c0 = cc * 32 + 2 * k;
                        t.x = c0 < nvis && c0 >= nlo ? t.x : -INFINITY;
                        t.y = c0 + 1 < nvis && c0 + 1 >= nlo ? t.y : -INFINITY;
                    }
                    const float2 e2 = make_float2(ex2(t.x), ex2(t.y));
                    rs2[k & 3] = fadd2(rs2[k & 3], e2);
                    const __nv_bfloat162 hv = __floats2bfloat162_rn(e2.x, e2.y);
                    hw[k] = *reinterpret_cast<const uint32_t *>(&hv);
                    if (split) {
                        const float2 hf = __bfloat1622float2(hv);
                        lw[k] = pack_bf16(e2.x - hf.x, e2.y - hf.y);
                    }
                }
            };
            if (!split_blk && all_visible && !capped) {
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t sr[32], hw[16], lw[16];
                    tmem_ld32(ts + cc * 32, sr);
                    tmem_wait_ld();
                    quarter(sr, cc, hw, lw, false, false, false);
                    tmem_st16(ts + cc * 32, hw);
                }
            } else if (all_visible && !capped) {
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t sr[32], hw[16], lw[16];
                    tmem_ld32(ts + cc * 32, sr);
                    tmem_wait_ld();
                    quarter(sr, cc, hw, lw, false, true, false);
                    tmem_st16(ts + cc * 32, hw);
                    tmem_st16(ts + cc * 32 + 16, lw);
                }
            } else {
                // Masked (a diagonal or window block) or soft-capped: each combination of
                // the flags gets its own loop, so that no pair computes what a branch not
                // taken would need (the caps' tanh in particular).
                auto general = [&](const bool masked, const bool split, const bool cap) {
#pragma unroll 1
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t sr[32], hw[16], lw[16];
                        tmem_ld32(ts + cc * 32, sr);
                        tmem_wait_ld32(sr);
                        quarter(sr, cc, hw, lw, masked, split, cap);
                        tmem_st16(ts + cc * 32, hw);
                        if (split) tmem_st16(ts + cc * 32 + 16, lw);
                    }
                };
                // Masked, uncapped: quarter by quarter as classified above.
                auto masked_blk = [&](const bool split) {
#pragma unroll 1
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t sr[32], hw[16], lw[16];
                        if ((q_none >> cc) & 1) {
#pragma unroll
                            for (int k = 0; k < 16; ++k) hw[k] = 0u;
                            tmem_st16(ts + cc * 32, hw);
                            if (split) tmem_st16(ts + cc * 32 + 16, hw);
                            continue;
                        }
                        tmem_ld32(ts + cc * 32, sr);
                        tmem_wait_ld32(sr);
                        if ((q_full >> cc) & 1) quarter(sr, cc, hw, lw, false, split, false);
                        else quarter(sr, cc, hw, lw, true, split, false);
                        tmem_st16(ts + cc * 32, hw);
                        if (split) tmem_st16(ts + cc * 32 + 16, lw);
                    }
                };
                if (capped) {
                    if (split_blk) general(!all_visible, true, true);
                    else general(!all_visible, false, true);
                } else if (split_blk) {
                    masked_blk(true);
                } else {
                    masked_blk(false);
                }
            }
            const float2 r01 = fadd2(rs2[0], rs2[1]), r23 = fadd2(rs2[2], rs2[3]);
            const float rs = (r01.x + r01.y) + (r23.x + r23.y);
            l = l * corr + rs;
            log2_l = __log2f(l);  // for the next block's vote; -inf while l = 0
            // O must hold PV(j-1) before it is rescaled (and before PV(j) is issued,
            // which waits for this warpgroup's P).  Doing it after writing P keeps
            // PV(j-1) off the critical path.  With one S buffer S(j) was issued after
            // PV(j-1) by the same thread, and its commit tracks every earlier MMA, so
            // S being full already says so.
            if (SB > 1 && j > 0 && !wait_warp(BAR(C::B_PVDONE + x), (G - 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (j > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(to + cc * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
                    tmem_st32(to + cc * 32, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(C::B_PFULL + x));
        }
        if (ok && !wait_warp(BAR(C::B_PVDONE + x), (g + nb - 1) & 1, abort_flag)) ok = false;
        if (!ok) {
            failed = true;
            *abort_flag = 1;
        }
        // ---------------------------------------------------- epilogue
        tc_fence_after();
        if (ok) {
            const int64_t row = tile_row(p, b, hkv, valid ? f : 0);
            // Direct mode folds the sink (one more state: m = sink log2 e, l = 1,
            // acc = 0) here; split mode leaves it to the merge.
            float osc = 1.f;  // factor on acc
            if (!p.split && p.sinks && valid) {
                const float sink2 = p.sinks[(row / p.q_len) % p.Hq] * kLog2e;
                const float M = fmaxf(m_used, sink2);
                osc = ex2(m_used - M);
                l = l * osc + ex2(sink2 - M);
                m_used = M;
            }
            const float inv = p.split ? 1.f : osc / l;
            const int64_t slot = row * p.n_chunks + c;
            // The warp's 32 rows go through shared memory so that each global store
            // instruction writes whole rows: lane r holds row r of the warp, whose
            // 16-byte chunk c sits at chunk c ^ (r & 7) of its staging row, so that
            // both the row-wise writes and the chunk-wise reads are free of bank
            // conflicts.  Every MMA that reads shared memory has completed by now except
            // the other tile's last PV, whose V stage and P lie outside this tile's
            // staging area (tile 0: the Q tiles; tile 1: the V stages, written once its
            // own PV is done).
            const bool wide = p.split || !p.out_bf16;  // fp32 rows, else bf16 rows
            const int rb = wide ? D * 4 : D * 2;       // bytes per output row
            const uint32_t stage = sb + (uint32_t)(x * 4 + q4) * (32u * D * 4u);
            const uint32_t my_row = stage + (uint32_t)lane * rb;
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                tmem_ld32(to + cc * 32, o);
                tmem_wait_ld();
                if (PERSIST) {
                    // The next item's Q and K/V are landing in shared memory: rows go
                    // straight from registers (direct mode), in 32-byte stores when the
                    // output allows (each fills a whole sector of its row).
                    if (!valid) continue;
                    uint8_t *dst = static_cast<uint8_t *>(p.out) +
                                   (row * D + cc * 32) * (p.out_bf16 ? 2 : 4);
                    auto f = [&](int e) { return __uint_as_float(o[e]) * inv; };
                    if (p.out_bf16) {
#pragma unroll
                        for (int k = 0; k < 2; ++k) {  // 16 columns = 32 bytes each
                            const uint4 a = make_uint4(
                                pack_bf16(f(16 * k + 0), f(16 * k + 1)),
                                pack_bf16(f(16 * k + 2), f(16 * k + 3)),
                                pack_bf16(f(16 * k + 4), f(16 * k + 5)),
                                pack_bf16(f(16 * k + 6), f(16 * k + 7)));
                            const uint4 b = make_uint4(
                                pack_bf16(f(16 * k + 8), f(16 * k + 9)),
                                pack_bf16(f(16 * k + 10), f(16 * k + 11)),
                                pack_bf16(f(16 * k + 12), f(16 * k + 13)),
                                pack_bf16(f(16 * k + 14), f(16 * k + 15)));
                            if (out32) {
                                st_global_v8(dst + 32 * k, a, b);
                            } else {
                                reinterpret_cast<uint4 *>(dst + 32 * k)[0] = a;
                                reinterpret_cast<uint4 *>(dst + 32 * k)[1] = b;
                            }
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {  // 8 columns = 32 bytes each
                            const uint4 a = make_uint4(
                                __float_as_uint(f(8 * k + 0)), __float_as_uint(f(8 * k + 1)),
                                __float_as_uint(f(8 * k + 2)), __float_as_uint(f(8 * k + 3)));
                            const uint4 b = make_uint4(
                                __float_as_uint(f(8 * k + 4)), __float_as_uint(f(8 * k + 5)),
                                __float_as_uint(f(8 * k + 6)), __float_as_uint(f(8 * k + 7)));
                            if (out32) {
                                st_global_v8(dst + 32 * k, a, b);
                            } else {
                                reinterpret_cast<uint4 *>(dst + 32 * k)[0] = a;
                                reinterpret_cast<uint4 *>(dst + 32 * k)[1] = b;
                            }
                        }
                    }
                    continue;
                }
                if (wide) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        st_shared_v4(my_row + (uint32_t)(((cc * 8 + k) ^ (lane & 7)) * 16),
                                     __float_as_uint(__uint_as_float(o[4 * k]) * inv),
                                     __float_as_uint(__uint_as_float(o[4 * k + 1]) * inv),
                                     __float_as_uint(__uint_as_float(o[4 * k + 2]) * inv),
                                     __float_as_uint(__uint_as_float(o[4 * k + 3]) * inv));
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        st_shared_v4(my_row + (uint32_t)(((cc * 4 + k) ^ (lane & 7)) * 16),
                                     pack_bf16(__uint_as_float(o[8 * k + 0]) * inv,
                                               __uint_as_float(o[8 * k + 1]) * inv),
                                     pack_bf16(__uint_as_float(o[8 * k + 2]) * inv,
                                               __uint_as_float(o[8 * k + 3]) * inv),
                                     pack_bf16(__uint_as_float(o[8 * k + 4]) * inv,
                                               __uint_as_float(o[8 * k + 5]) * inv),
                                     pack_bf16(__uint_as_float(o[8 * k + 6]) * inv,
                                               __uint_as_float(o[8 * k + 7]) * inv));
                }
            }
            // O is read out: the next item's first PV may overwrite it.
            if (PERSIST) {
                tc_fence_before();  // the O loads are ordered before the arrival
                mbar_arrive(BAR(C::B_OFREE + x));
            }
            __syncwarp();
            // Byte offset of this thread's row in its destination, -1 for a row that
            // is not written.
            uint8_t *const dst_base = p.split ? reinterpret_cast<uint8_t *>(p.ws_acc)
                                              : static_cast<uint8_t *>(p.out);
            const int64_t my_off = !valid ? -1 : (p.split ? slot : row) * (int64_t)rb;
            const int cpr = rb / 16;       // 16-byte chunks per row: 8, 16 or 32
            const int rpi = 32 / cpr;      // rows per store instruction
            const int ch = lane % cpr;     // this lane's chunk of its row
#pragma unroll 1
            for (int r0 = 0; r0 < 32 && !PERSIST; r0 += rpi) {
                const int r = r0 + lane / cpr;
                const int64_t off = __shfl_sync(0xffffffffu, my_off, r);
                const uint4 v = ld_shared_v4(stage + (uint32_t)(r * rb + ((ch ^ (r & 7)) * 16)));
                if (off >= 0) *reinterpret_cast<uint4 *>(dst_base + off + ch * 16) = v;
            }
            if (valid) {
                if (p.split) {
                    p.ws_ml[slot * 2] = m_used;
                    p.ws_ml[slot * 2 + 1] = l;
                } else if (p.lse) {
                    p.lse[row] = kLn2 * (m_used + log2f(l));
                }
            }
        } else if (valid) {
            if (p.split) {
                const int64_t slot = tile_row(p, b, hkv, f) * p.n_chunks + c;
                p.ws_ml[slot * 2] = p.ws_ml[slot * 2 + 1] = __int_as_float(0x7fc00000);
            } else {
                nan_row<D>(p, b, hkv, f);
            }
        }
        g += nb;
        }
        // After an abort, the items this warpgroup did not reach: their rows NaN.
        for (; it < n_items; ++it) {
            if ((skip >> it) & 1) continue;
            const TcWork &w = PERSIST ? items[it] : w0;
            const int f = (w.t0 + x * w.tstep) * BM + r;
            if (f >= w.rows_unit || f % p.q_len >= w.qn) continue;
            if (p.split) {
                float *ml = p.ws_ml + (tile_row(p, w.b, w.hkv, f) * p.n_chunks + w.c) * 2;
                ml[0] = ml[1] = __int_as_float(0x7fc00000);
            } else {
                nan_row<D>(p, w.b, w.hkv, f);
            }
        }
    }

    tc_fence_before();
    const bool any_failed = __syncthreads_or(failed) != 0;
    if (any_failed && threadIdx.x == 0 && p.status) atomicOr(p.status, ATLAS_DEV_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
#undef BAR
}

template <int NT, int D>
cudaError_t launch_instance(const TcParams &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                            const CUtensorMap &tmV, cudaStream_t stream) {
    using C = Cfg<NT, D>;
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !configured[dev]) {
        err = cudaFuncSetAttribute(fmha_tc_kernel<NT, D, false>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if constexpr (NT == 2) {
            if (err == cudaSuccess)
                err = cudaFuncSetAttribute(fmha_tc_kernel<NT, D, true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        }
        if (err != cudaSuccess) return err;
        configured[dev] = 1;
    }
    const int tiles = p.B * p.Hkv * p.tiles_per_unit;
    dim3 grid = p.split ? dim3(p.n_chunks, tiles, 1) : dim3(tiles / NT, 1, 1);
    // Direct prefill with more tile pairs than SMs: one CTA per SM walks several
    // (at most kMaxItems), so that CTA start-up, the first loads and the epilogue
    // overlap the neighbouring items' work.
    bool persistent = false;
    if (NT == 2 && !p.split && p.tiles_per_head > 0 && !p.q_lens) {
        const int items = tiles / NT;
        const int ctas = max(max(p.sms, 1), (items + kMaxItems - 1) / kMaxItems);
        if (ctas < items) {
            persistent = true;
            grid = dim3(ctas, 1, 1);
        }
    }
    if constexpr (NT == 2) {
        if (persistent) {
            fmha_tc_kernel<NT, D, true><<<grid, C::kThreads, C::kSmem, stream>>>(tmQ, tmK, tmV, p);
            return cudaGetLastError();
        }
    }
    fmha_tc_kernel<NT, D, false><<<grid, C::kThreads, C::kSmem, stream>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fmha_tc(const TcParams &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                           const CUtensorMap &tmV, cudaStream_t stream) {
    // Two tiles per CTA when two q heads of a group can share every K/V block:
    // direct output, an even group, prompt rows in whole tiles.
    const bool pair = !p.split && p.tiles_per_head > 0 && p.G % 2 == 0;
    if (p.D == 64)
        return pair ? launch_instance<2, 64>(p, tmQ, tmK, tmV, stream)
                    : launch_instance<1, 64>(p, tmQ, tmK, tmV, stream);
    return pair ? launch_instance<2, 128>(p, tmQ, tmK, tmV, stream)
                : launch_instance<1, 128>(p, tmQ, tmK, tmV, stream);
}

}  // namespace atlas
