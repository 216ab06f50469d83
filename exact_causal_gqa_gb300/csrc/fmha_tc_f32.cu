// fmha_tc_f32.cu -- causal suffix and prefill attention for fp32 q/K/V on the
// 5th-generation tensor cores (tcgen05 + TMEM), each fp32 contraction done as three
// tf32 products with fp32 accumulation.
//
// Precision.  Each fp32 operand x is split as x = hi + lo with hi = x with its 13
// low mantissa bits cleared (a tf32 value, read by the tensor core exactly) and
// lo = x - hi (exact in fp32, |lo| < 2^-10 |x|).  A product a.b is taken as
//   hi(a).hi(b) + lo(a).hi(b) + hi(a).lo(b),
// dropping lo(a).lo(b) (< 2^-20 |a||b|) and the tf32 reading of the lo parts
// (< 2^-10 of them, whether the hardware truncates or rounds): each term keeps
// about 20 bits, well inside the 1e-5 bound that fp32 K/V are held to.  This
// applies to S = Q K^T and to O += P V, with fp32 accumulators in TMEM.  The lo
// products go first, the hi.hi product last.
//
// Accumulation.  The tensor core adds each product into its fp32 accumulator with
// a rounding biased towards zero, so the error of one accumulator grows with the
// number of MMAs added into it (measured: ~3e-8 relative per tf32 MMA, i.e. ~9e-5
// after 125 blocks of 24).  O is therefore accumulated in segments of kSegBlocks
// blocks: the first PV product of a segment overwrites the TMEM accumulator, and
// the converter warps fold each finished segment into a running sum with fp32
// round-to-nearest arithmetic, O_run = O_run 2^(m_run - m_seg) + O_seg, kept in
// this CTA's own output row (direct mode) or split slot (split mode).
//
// A CTA owns one 128-row query tile of one (sequence, kv head) -- the G * q_len
// (q head, query row) pairs of the GQA group in memory order, as the bf16 kernel
// -- and walks 64-key blocks up to the last key any of its rows sees (causal block
// skipping, CPUAttn README: the fused QK -> RowNorm -> PV tile pipeline stops at
// the last reachable K block), folding each into per-row online-softmax state
// (CFR-Atlas README, "Core contract").
//
// Tensor memory (512 columns): Q hi | Q lo (D each, the A operand of S) | S (64;
// overwritten by P as fp32, the A operand of PV) | P lo (64) | O (D).
// Shared memory: Q staging (once, overlaid on the K lo / V^T buffers), a ring of
// raw K blocks (the B operand of S, K-major), a ring of raw V blocks (converter
// input), and single buffers K lo, V^T hi and V^T lo (K-major B operands of S and
// PV: V^T is [D rows][64 keys], built by the converter since the tensor core reads
// both tf32 operands K-major here).
//
// Warp roles (384 threads, one CTA per SM):
//   warp 0     TMA producer: Q once, then K and V blocks page by page through the
//              page table.
//   warp 1     allocates TMEM; one lane issues the MMAs:
//                S  = Qhi K + Qlo K + Qhi Klo        (M=128, N=64, K=D; A from TMEM)
//                O += P V^T + Plo V^T + P V^Tlo      (M=128, N=D, K=64; A from TMEM)
//   warps 4-7  softmax, one thread per query row: Q into TMEM (hi, lo) at the start;
//              per block the S row from TMEM, mask, row max, ex2, row sum; P and its
//              lo part back into TMEM; O rescaled in TMEM when the row max grew by
//              more than 2^8 (exact: acc and l share the reference max).  Epilogue:
//              O / l, or the split's (m, l, acc).
//   warps 8-11 converter: K lo = K - hi(K) and K replaced by hi(K) in place; V^T hi
//              and lo from the raw V block, keys past the last visible one zeroed
//              (slots there may hold NaN); and the fold of each finished O segment
//              into the running sum.
// Every mbarrier wait is bounded; a CTA that gives up records ATLAS_DEV_TIMEOUT,
// lets its copies and MMAs finish, frees TMEM and writes NaN.
#include "internal.h"
#include "ptx.cuh"
#include "tc_order.cuh"

#include <math.h>

namespace atlas {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 64;   // keys per block
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows 256x
constexpr int kSegBlocks = 4;  // key blocks per O accumulation segment

template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static constexpr int kSlabs = D / 32;        // 32-element (128-byte) slabs per row
    static constexpr int kBlkBytes = BN * D * 4; // one fp32 K or V block
    static constexpr int kKSlab = BN * 128;      // one slab of a K or V block
    static constexpr int kQSlab = BM * 128;      // one slab of the Q tile
    static constexpr int kVtSlab = D * 128;      // one 32-key slab of V^T
    static constexpr int kStages = D == 128 ? 2 : 4;
    static constexpr int kThreads = 384;
    static constexpr int kSoftmaxWarp0 = 4;
    static constexpr int kConvWarp0 = 8;
    static constexpr int OFF_KLO = 0;
    static constexpr int OFF_VTH = OFF_KLO + kBlkBytes;
    static constexpr int OFF_VTL = OFF_VTH + kBlkBytes;
    static constexpr int OFF_Q = OFF_KLO;  // Q staging (2 blocks' bytes) until Q is in TMEM
    static constexpr int OFF_K = OFF_VTL + kBlkBytes;
    static constexpr int OFF_V = OFF_K + kStages * kBlkBytes;
    static constexpr int OFF_BAR = OFF_V + kStages * kBlkBytes;
    static_assert(BM * D * 4 <= OFF_VTL - OFF_Q, "Q staging fits the K lo / V^T hi buffers");
    // barriers
    static constexpr int B_Q = 0;             // Q landed (TMA bytes)
    static constexpr int B_QREADY = 1;        // Q in TMEM, staging consumed (128 arrivals)
    static constexpr int B_KFULL = 2;         // [kStages]
    static constexpr int B_KEMPTY = B_KFULL + kStages;
    static constexpr int B_VFULL = B_KEMPTY + kStages;
    static constexpr int B_VEMPTY = B_VFULL + kStages;  // converter done with the raw V (128)
    static constexpr int B_KLO_READY = B_VEMPTY + kStages;  // 128 arrivals
    static constexpr int B_KLO_FREE = B_KLO_READY + 1;      // S products done with K lo
    static constexpr int B_VT_READY = B_KLO_FREE + 1;       // 128 arrivals
    static constexpr int B_VT_FREE = B_VT_READY + 1;        // PV products done with V^T
    static constexpr int B_SFULL = B_VT_FREE + 1;
    static constexpr int B_PFULL = B_SFULL + 1;             // 128 arrivals
    static constexpr int B_PVDONE = B_PFULL + 1;
    static constexpr int B_SEG_DONE = B_PVDONE + 1;   // last PV of a segment done
    static constexpr int B_MSEG = B_SEG_DONE + 1;     // softmax max at a segment's end (128)
    static constexpr int B_O_DRAINED = B_MSEG + 1;    // segment read out of TMEM (128)
    static constexpr int B_FOLDED = B_O_DRAINED + 1;   // every segment but the last folded (128)
    static constexpr int B_FINAL = B_FOLDED + 1;
    static constexpr int kBars = B_FINAL + 1;
    // per row: the softmax's max at the end of a segment (by segment parity), and the
    // max the running sum is relative to after the last fold
    static constexpr int OFF_MSEG = OFF_BAR + kBars * 8;
    static constexpr int OFF_MRUN = OFF_MSEG + 2 * BM * 4;
    static constexpr int OFF_TMEM = OFF_MRUN + BM * 4;
    static constexpr int OFF_FLAG = OFF_TMEM + 8;
    static constexpr int kSmem = OFF_FLAG + 8 + 1024;  // + slack to align the base
    static_assert(kSmem <= 232448, "shared memory budget");
    // TMEM columns
    static constexpr uint32_t QH = 0, QL = D, SC = 2 * D, PL = 2 * D + BN, OC = 2 * D + 2 * BN;
    static_assert(OC + D <= kTmemCols, "TMEM budget");
};

// Instruction descriptor of kind::tf32: tf32 A and B (both K-major), f32 accumulator.
//   bits 4-5 D format (1 = f32), 7-9 A format (2 = tf32), 10-12 B format (2 = tf32),
//   bits 17-22 N >> 3, bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem desc] with tf32 operands (A: M rows = TMEM lanes,
// one 32-bit value per column along K).
__device__ __forceinline__ void umma_tf32_tmem_a(uint32_t d_tmem, uint32_t a_tmem,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// x truncated to tf32 (the value the tensor core reads) and the exact remainder.
__device__ __forceinline__ float tf32_hi(float x) {
    return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}
__device__ __forceinline__ float tf32_lo(float x) { return x - tf32_hi(x); }

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort, kWaitLimitNs));
}

__device__ __forceinline__ int64_t tile_row(const TcParams &p, int b, int hkv, int f) {
    return ((int64_t)b * p.Hq + (int64_t)hkv * p.G) * p.q_len + f;
}

template <int D>
__device__ void nan_row(const TcParams &p, int b, int hkv, int f) {
    const int64_t row = tile_row(p, b, hkv, f);
    const float nan = __int_as_float(0x7fc00000);
    float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + row * D);
    for (int k = 0; k < D / 4; ++k) o[k] = make_float4(nan, nan, nan, nan);
    if (p.lse) p.lse[row] = nan;
}

template <int D>
__global__ void __launch_bounds__(Cfg<D>::kThreads, 1)
    fmha_tf32x3_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const TcParams p) {
    allow_dependent_launch();  // the merge may start its CTAs (it waits for this grid)
    using C = Cfg<D>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEM);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#define BAR(i) (sb + C::OFF_BAR + 8u * (uint32_t)(i))

    // ------------------------------------------------------------ work item
    const int units = p.B * p.Hkv;
    int u, c, t0;
    int split_keys = p.chunk;  // keys per split (split mode)
    if (p.split && p.balanced) {
        // longest-first work item (the raw V ring is free until the producer starts)
        const TcItem it = tc_balanced_item(p, blockIdx.x + blockIdx.y * gridDim.x,
                                           reinterpret_cast<int *>(smem + C::OFF_V));
        if (it.b < 0) return;
        c = it.split;
        u = it.b * p.Hkv + it.hkv;
        t0 = it.tile;
        split_keys = it.split_keys;
    } else if (p.split) {
        c = blockIdx.x;
        u = blockIdx.y / p.tiles_per_unit;
        t0 = blockIdx.y % p.tiles_per_unit;
    } else {
        c = 0;
        const int r = blockIdx.x;
        if (p.tiles_per_head > 0) {  // heavy tiles (late prompt rows) first
            const int per = units * p.G;
            const int rest = r % per;
            u = rest / p.G;
            const int qi = p.tiles_per_head - 1 - r / per;
            t0 = (rest % p.G) * p.tiles_per_head + qi;
        } else {
            u = r % units;
            t0 = r / units;
        }
    }
    const int b = u / p.Hkv, hkv = u % p.Hkv;
    if (p.split && p.chunk_range && (c < p.chunk_range[2 * b] || c >= p.chunk_range[2 * b + 1]))
        return;
    const int seq_len = p.seq_lens[b];
    const int qn = p.q_lens ? p.q_lens[b] : p.q_len;
    const int rows_unit = p.G * p.q_len;
    const int f0 = t0 * BM;
    const int f_last = min(f0 + BM, rows_unit) - 1;
    const bool spans = (f_last / p.q_len) != (f0 / p.q_len);
    const int i_min = spans ? 0 : f0 % p.q_len;

    if (qn < 0 || qn > p.q_len || seq_len < qn || seq_len > p.max_pages * p.P ||
        (p.require_full && seq_len != qn)) {
        if (threadIdx.x == 0 && c == 0 && p.status) atomicOr(p.status, ATLAS_DEV_BAD_SEQLEN);
        const int rows_valid = (qn >= 0 && qn <= p.q_len) ? qn : p.q_len;
        if (!p.split && threadIdx.x < BM) {
            const int f = f0 + threadIdx.x;
            if (f < rows_unit && f % p.q_len < rows_valid) nan_row<D>(p, b, hkv, f);
        }
        return;  // split mode: the merge writes NaN rows for this sequence
    }
    if (i_min >= qn) return;  // only padding rows of a ragged sequence
    const int i_max = min(spans ? p.q_len - 1 : f_last % p.q_len, qn - 1);
    const int L = seq_len - qn + p.q_len;
    const int kv_hi = L - p.q_len + i_max + 1;
    const int kv_lo = p.window > 0 ? max(0, L - p.q_len + i_min + 1 - p.window) / BN * BN : 0;
    int kv_begin = kv_lo, kv_end = kv_hi;
    if (p.split) {
        kv_begin = max(c * split_keys, kv_lo);
        kv_end = min(kv_hi, c * split_keys + split_keys);
        if (kv_begin >= kv_end) return;
    }
    const int nb = (kv_end - kv_begin + BN - 1) / BN;
    {
        const int pg0 = kv_begin / p.P, pg1 = (kv_end - 1) / p.P;
        bool bad = false;
        for (int pg = pg0 + (int)threadIdx.x; pg <= pg1; pg += blockDim.x) {
            const int id = p.page_table[(int64_t)b * p.max_pages + pg];
            bad |= (id < 0 || id >= p.num_pages);
        }
        if (__syncthreads_or(bad)) {
            if (threadIdx.x == 0 && p.status) atomicOr(p.status, ATLAS_DEV_BAD_PAGE);
            if (threadIdx.x < BM) {
                const int f = f0 + threadIdx.x;
                if (f < rows_unit && f % p.q_len < qn) {
                    if (!p.split) {
                        nan_row<D>(p, b, hkv, f);
                    } else {
                        float *ml = p.ws_ml + (tile_row(p, b, hkv, f) * p.n_chunks + c) * 2;
                        ml[0] = ml[1] = __int_as_float(0x7fc00000);
                    }
                }
            }
            return;
        }
    }

    // ------------------------------------------------------------ setup
    if (threadIdx.x == 0) {
        mbar_init(BAR(C::B_Q), 1);
        mbar_init(BAR(C::B_QREADY), BM);
        for (int s = 0; s < S; ++s) {
            mbar_init(BAR(C::B_KFULL + s), 1);
            mbar_init(BAR(C::B_KEMPTY + s), 1);
            mbar_init(BAR(C::B_VFULL + s), 1);
            mbar_init(BAR(C::B_VEMPTY + s), 128);
        }
        mbar_init(BAR(C::B_KLO_READY), 128);
        mbar_init(BAR(C::B_KLO_FREE), 1);
        mbar_init(BAR(C::B_VT_READY), 128);
        mbar_init(BAR(C::B_VT_FREE), 1);
        mbar_init(BAR(C::B_SFULL), 1);
        mbar_init(BAR(C::B_PFULL), BM);
        mbar_init(BAR(C::B_PVDONE), 1);
        mbar_init(BAR(C::B_SEG_DONE), 1);
        mbar_init(BAR(C::B_MSEG), 128);
        mbar_init(BAR(C::B_O_DRAINED), 128);
        mbar_init(BAR(C::B_FOLDED), 128);
        mbar_init(BAR(C::B_FINAL), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool failed = false;

    if (warp == 0) {
        // -------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            mbar_arrive_expect_tx(BAR(C::B_Q), BM * D * 4);
            const int qrow = (int)tile_row(p, b, hkv, f0);
#pragma unroll
            for (int sl = 0; sl < C::kSlabs; ++sl)
                tma_load_2d(sb + C::OFF_Q + sl * C::kQSlab, &tmQ, 32 * sl, qrow, BAR(C::B_Q));
        }
        PageIdCache pages{p.page_table + (int64_t)b * p.max_pages, (kv_end - 1) / p.P};
        const int BR = p.P < BN ? p.P : BN;
        int issued_k = 0, issued_v = 0;
        for (int j = 0; j < nb && !failed; ++j) {
            const int s = j % S, use = j / S;
            const int kb = kv_begin + j * BN;
            const int ke = min(kb + BN, kv_end);
            const int nbox = (ke - kb + BR - 1) / BR;
            const uint32_t bytes = (uint32_t)(nbox * BR * 128 * C::kSlabs);
            int my_y = 0;
            for (int bx = 0; bx < nbox; ++bx) {
                const int tk = kb + bx * BR;
                const int y = (pages.get(tk / p.P) * p.Hkv + hkv) * p.P + (tk % p.P);
                if (lane == bx) my_y = y;
            }
            for (int kv = 0; kv < 2; ++kv) {
                const int full = (kv == 0 ? C::B_KFULL : C::B_VFULL) + s;
                const int empty = (kv == 0 ? C::B_KEMPTY : C::B_VEMPTY) + s;
                if (use > 0 && !wait_warp(BAR(empty), (use - 1) & 1, abort_flag)) {
                    failed = true;
                    break;
                }
                if (lane < nbox) {
                    const CUtensorMap *map = kv == 0 ? &tmK : &tmV;
                    const uint32_t dst = sb + (kv == 0 ? C::OFF_K : C::OFF_V) + s * C::kBlkBytes;
                    if (lane == 0) mbar_arrive_expect_tx(BAR(full), bytes);
                    __syncwarp((1u << nbox) - 1u);
#pragma unroll
                    for (int sl = 0; sl < C::kSlabs; ++sl)
                        tma_load_2d(dst + sl * C::kKSlab + lane * BR * 128, map, 32 * sl, my_y,
                                    BAR(full));
                }
                __syncwarp();
                if (kv == 0) issued_k = j + 1;
                else issued_v = j + 1;
            }
        }
        if (failed && lane == 0) {
            *abort_flag = 1;
            int no_abort = 0;
            mbar_wait_bounded(BAR(C::B_Q), 0, &no_abort, kWaitLimitNs);
            for (int j = max(0, issued_k - S); j < issued_k; ++j)
                mbar_wait_bounded(BAR(C::B_KFULL + j % S), (j / S) & 1, &no_abort, kWaitLimitNs);
            for (int j = max(0, issued_v - S); j < issued_v; ++j)
                mbar_wait_bounded(BAR(C::B_VFULL + j % S), (j / S) & 1, &no_abort, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_tf32_f32(BM, BN);
            constexpr uint32_t idPV = idesc_tf32_f32(BM, D);
            bool ok = mbar_wait_bounded(BAR(C::B_QREADY), 0, abort_flag, kWaitLimitNs);
            tc_fence_after();
            const uint64_t klod = sdesc_sw128(sb + C::OFF_KLO, 16, 1024);
            const uint64_t vthd = sdesc_sw128(sb + C::OFF_VTH, 16, 1024);
            const uint64_t vtld = sdesc_sw128(sb + C::OFF_VTL, 16, 1024);
            for (int j = 0; ok && j < nb; ++j) {
                const int s = j % S;
                ok = mbar_wait_bounded(BAR(C::B_KFULL + s), (j / S) & 1, abort_flag, kWaitLimitNs) &&
                     mbar_wait_bounded(BAR(C::B_KLO_READY), j & 1, abort_flag, kWaitLimitNs);
                if (!ok) break;
                tc_fence_after();
                // S = Qlo K + Qhi Klo + Qhi K (small terms first).  K slice kk (8
                // dims) sits 32 bytes into its 128-byte row, slab kk / 4 one K-slab on.
                const uint64_t kd = sdesc_sw128(sb + C::OFF_K + s * C::kBlkBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 8; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kKSlab + (kk & 3) * 32) >> 4;
                    umma_tf32_tmem_a(tmem + C::SC, tmem + C::QL + 8 * kk, kd + off, idS, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < D / 8; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kKSlab + (kk & 3) * 32) >> 4;
                    umma_tf32_tmem_a(tmem + C::SC, tmem + C::QH + 8 * kk, klod + off, idS, 1u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 8; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kKSlab + (kk & 3) * 32) >> 4;
                    umma_tf32_tmem_a(tmem + C::SC, tmem + C::QH + 8 * kk, kd + off, idS, 1u);
                }
                umma_commit(BAR(C::B_SFULL));
                umma_commit(BAR(C::B_KEMPTY + s));
                umma_commit(BAR(C::B_KLO_FREE));
                // O += P V^T + Plo V^T + P V^Tlo once the softmax wrote P and the
                // converter built V^T.  Key slice kk (8 keys) of V^T sits 32 bytes into
                // its 128-byte row, 32-key slab kk / 4 one V^T-slab further on.
                ok = mbar_wait_bounded(BAR(C::B_PFULL), j & 1, abort_flag, kWaitLimitNs) &&
                     mbar_wait_bounded(BAR(C::B_VT_READY), j & 1, abort_flag, kWaitLimitNs);
                // A new segment overwrites O: the previous one must have been read out.
                const bool fresh = j % kSegBlocks == 0;
                if (ok && fresh && j > 0)
                    ok = mbar_wait_bounded(BAR(C::B_O_DRAINED), (j / kSegBlocks - 1) & 1,
                                           abort_flag, kWaitLimitNs);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BN / 8; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kVtSlab + (kk & 3) * 32) >> 4;
                    umma_tf32_tmem_a(tmem + C::OC, tmem + C::PL + 8 * kk, vthd + off, idPV,
                                     (!fresh || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < BN / 8; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kVtSlab + (kk & 3) * 32) >> 4;
                    umma_tf32_tmem_a(tmem + C::OC, tmem + C::SC + 8 * kk, vtld + off, idPV, 1u);
                }
#pragma unroll
                for (int kk = 0; kk < BN / 8; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kVtSlab + (kk & 3) * 32) >> 4;
                    umma_tf32_tmem_a(tmem + C::OC, tmem + C::SC + 8 * kk, vthd + off, idPV, 1u);
                }
                umma_commit(BAR(C::B_PVDONE));
                umma_commit(BAR(C::B_VT_FREE));
                // a segment followed by another one: the converter folds it
                if ((j + 1) % kSegBlocks == 0 && j + 1 < nb) umma_commit(BAR(C::B_SEG_DONE));
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
    } else if (warp >= C::kConvWarp0) {
        // -------------------------------------------------------- converter
        const int ct = threadIdx.x - C::kConvWarp0 * 32;  // 0..127
        // The row this thread folds O for: its TMEM lane (quadrant warp % 4).
        const int r = (warp % 4) * 32 + lane;
        const uint32_t tq = tmem + ((uint32_t)((warp % 4) * 32) << 16) + C::OC;
        const int fr_row = f0 + r;
        const bool row_ok = fr_row < rows_unit && fr_row % p.q_len < qn;
        // the running sum lives in this row's own output row or split slot
        float *run = p.split
                         ? p.ws_acc + (tile_row(p, b, hkv, row_ok ? fr_row : 0) * p.n_chunks + c) * D
                         : static_cast<float *>(p.out) + tile_row(p, b, hkv, row_ok ? fr_row : 0) * D;
        const float *m_seg_s = reinterpret_cast<const float *>(smem + C::OFF_MSEG);
        float *m_run_s = reinterpret_cast<float *>(smem + C::OFF_MRUN);
        float m_run = -INFINITY;
        bool ok = wait_warp(BAR(C::B_QREADY), 0, abort_flag);  // Q staging consumed
        // K lo of block j, same layout as the raw block, and K's hi part in place:
        // element-wise on 16-byte chunks (no S product of the block is issued yet).
        auto convert_k = [&](int j) -> bool {
            const int s = j % S, use = j / S;
            if (!wait_warp(BAR(C::B_KFULL + s), use & 1, abort_flag) ||
                (j > 0 && !wait_warp(BAR(C::B_KLO_FREE), (j - 1) & 1, abort_flag)))
                return false;
            float4 *src = reinterpret_cast<float4 *>(smem + C::OFF_K + s * C::kBlkBytes);
            float4 *dst = reinterpret_cast<float4 *>(smem + C::OFF_KLO);
            for (int k = ct; k < C::kBlkBytes / 16; k += 128) {
                const float4 x = src[k];
                dst[k] = make_float4(tf32_lo(x.x), tf32_lo(x.y), tf32_lo(x.z), tf32_lo(x.w));
                src[k] = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
            }
            fence_proxy_async_smem();
            mbar_arrive(BAR(C::B_KLO_READY));
            return true;
        };
        // V^T hi / lo of block j: 4 keys x 4 dims per lane and step, transposed in
        // registers.  Warp step it covers key groups kq0 .. kq0+7 x dim groups
        // dq0 .. dq0+3 (lane: kq = kq0 + lane % 8, dq = dq0 + lane / 8): the 16-byte
        // reads of a step fall on 8 distinct chunks of 4 rows, the writes on 8 chunks
        // of 4 rows of V^T, so neither conflicts beyond its 4 wavefronts.
        auto convert_v = [&](int j) -> bool {
            const int s = j % S, use = j / S;
            if (!wait_warp(BAR(C::B_VFULL + s), use & 1, abort_flag) ||
                (j > 0 && !wait_warp(BAR(C::B_VT_FREE), (j - 1) & 1, abort_flag)))
                return false;
            const int valid = min(BN, kv_end - (kv_begin + j * BN));  // keys in this block
            const uint8_t *vraw = smem + C::OFF_V + s * C::kBlkBytes;
            constexpr int kSteps = (BN / 32) * (D / 16);  // warp steps per block
            for (int it = warp - C::kConvWarp0; it < kSteps; it += 4) {
                const int kq = (it % (BN / 32)) * 8 + lane % 8;  // 4-key group
                const int dq = (it / (BN / 32)) * 4 + lane / 8;  // 4-dim group
                float v[4][4];                                    // [key][dim]
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = 4 * kq + e;
                    const int d0 = 4 * dq;
                    // raw: slab d0/32, row key, 16-byte chunk (d0 % 32) / 4
                    const uint32_t off = (d0 / 32) * C::kKSlab + sw128(key, (d0 % 32) / 4);
                    const float4 x = *reinterpret_cast<const float4 *>(vraw + off);
                    const bool in = key < valid;
                    v[e][0] = in ? x.x : 0.f;
                    v[e][1] = in ? x.y : 0.f;
                    v[e][2] = in ? x.z : 0.f;
                    v[e][3] = in ? x.w : 0.f;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int dim = 4 * dq + e;
                    const int k0 = 4 * kq;
                    // V^T: slab k0/32, row dim, 16-byte chunk (k0 % 32) / 4
                    const uint32_t off = (k0 / 32) * C::kVtSlab + sw128(dim, (k0 % 32) / 4);
                    *reinterpret_cast<float4 *>(smem + C::OFF_VTH + off) =
                        make_float4(tf32_hi(v[0][e]), tf32_hi(v[1][e]), tf32_hi(v[2][e]),
                                    tf32_hi(v[3][e]));
                    *reinterpret_cast<float4 *>(smem + C::OFF_VTL + off) =
                        make_float4(tf32_lo(v[0][e]), tf32_lo(v[1][e]), tf32_lo(v[2][e]),
                                    tf32_lo(v[3][e]));
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(BAR(C::B_VT_READY));
            mbar_arrive(BAR(C::B_VEMPTY + s));
            return true;
        };
        // Order: V^T of block j; at a segment's first block the previous segment is
        // read out of TMEM (the next PV overwrites it once every thread here has); K lo
        // of block j + 1 (S(j + 1) waits for it); then the fold of that segment,
        // O_run = O_run 2^(m_run - m_seg) + O_seg in fp32, off the S path.
        ok = ok && convert_k(0);
        for (int j = 0; ok && j < nb; ++j) {
            if (!convert_v(j)) {
                ok = false;
                break;
            }
            const bool fold = j % kSegBlocks == 0 && j > 0;
            const int g = j / kSegBlocks - 1;  // the segment folded at block j
            uint32_t o[D / 32][32];
            float m_seg = -INFINITY;
            if (fold) {
                if (!wait_warp(BAR(C::B_SEG_DONE), g & 1, abort_flag) ||
                    !wait_warp(BAR(C::B_MSEG), g & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(tq + 32 * cc, o[cc]);
                tmem_wait_ld();
                m_seg = m_seg_s[(g & 1) * BM + r];
                tc_fence_before();
                mbar_arrive(BAR(C::B_O_DRAINED));
            }
            if (j + 1 < nb && !convert_k(j + 1)) {
                ok = false;
                break;
            }
            if (fold) {
                if (row_ok) {
                    const float fr = g == 0 || m_run == -INFINITY ? 0.f : ex2(m_run - m_seg);
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        float4 *dst = reinterpret_cast<float4 *>(run + cc * 32);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float4 a = make_float4(
                                __uint_as_float(o[cc][4 * k]), __uint_as_float(o[cc][4 * k + 1]),
                                __uint_as_float(o[cc][4 * k + 2]), __uint_as_float(o[cc][4 * k + 3]));
                            if (g == 0) {
                                dst[k] = a;
                            } else {
                                const float4 x = dst[k];
                                dst[k] = make_float4(fmaf(x.x, fr, a.x), fmaf(x.y, fr, a.y),
                                                     fmaf(x.z, fr, a.z), fmaf(x.w, fr, a.w));
                            }
                        }
                    }
                }
                m_run = m_seg;
            }
        }
        if (ok && (nb - 1) / kSegBlocks > 0) {
            m_run_s[r] = m_run;
            mbar_arrive(BAR(C::B_FOLDED));
        }
        if (!ok) {
            failed = true;
            *abort_flag = 1;
        }
    } else if (warp >= C::kSoftmaxWarp0) {
        // -------------------------------------------------------- softmax
        const int q4 = warp % 4;  // TMEM lane quadrant
        const int r = q4 * 32 + lane;
        const int f = f0 + r;
        const bool valid = f < rows_unit && f % p.q_len < qn;
        const int i = valid ? f % p.q_len : 0;
        const int lim_row = valid ? min(L - p.q_len + i + 1, kv_end) : 0;
        const int lo_row = (valid && p.window > 0) ? max(0, L - p.q_len + i + 1 - p.window) : 0;
        const bool capped = p.softcap_log2 > 0.f;
        const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
        const uint32_t to = tl + C::OC;
        bool ok = wait_warp(BAR(C::B_Q), 0, abort_flag);
        if (ok) {
            // Q row r into TMEM: hi and lo (negated for a negative scale, which is
            // exact), 32 dims per slab.
            const float sgn = p.negate_scores ? -1.f : 1.f;
#pragma unroll 1
            for (int sl = 0; sl < C::kSlabs; ++sl) {
                uint32_t hv[32], lv[32];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const float4 x = *reinterpret_cast<const float4 *>(
                        smem + C::OFF_Q + sl * C::kQSlab + sw128(r, ch));
                    const float xs[4] = {x.x * sgn, x.y * sgn, x.z * sgn, x.w * sgn};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        hv[4 * ch + e] = __float_as_uint(tf32_hi(xs[e]));
                        lv[4 * ch + e] = __float_as_uint(tf32_lo(xs[e]));
                    }
                }
                tmem_st32(tl + C::QH + 32 * sl, hv);
                tmem_st32(tl + C::QL + 32 * sl, lv);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(BAR(C::B_QREADY));  // also on failure: the waits that follow are bounded

        float m_used = -INFINITY, l = 0.f;
        for (int j = 0; ok && j < nb; ++j) {
            if (!wait_warp(BAR(C::B_SFULL), j & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t ts = tl + C::SC;
            const int nvis = lim_row - (kv_begin + j * BN);  // visible columns: [nlo, nvis)
            const int nlo = lo_row - (kv_begin + j * BN);
            // The loads also return each half's maximum (tcgen05.ld.red), used when
            // every column is visible.
            uint32_t sa[32], sb2[32];
            float qa, qb;
            tmem_ld32_max(ts, sa, qa);
            tmem_ld32_max(ts + 32, sb2, qb);
            tmem_wait_ld32_max(sa, qa);
            tmem_wait_ld32_max(sb2, qb);
            // raw scores; columns outside [nlo, nvis) are masked (they may hold
            // anything, NaN included: keys past the end or below the window)
            float sr[BN];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                sr[e] = __uint_as_float(sa[e]);
                sr[32 + e] = __uint_as_float(sb2[e]);
            }
            // Blocks whose every column is visible to every real row of the warp skip
            // the masks (padding rows never reach the output).
            const bool all_visible = __all_sync(0xffffffffu, !valid || (nvis >= BN && nlo <= 0));
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (all_visible) {
                m4[0] = qa;
                m4[1] = qb;
            } else {
#pragma unroll
                for (int e = 0; e < BN; e += 2) {
                    const float v0 = e < nvis && e >= nlo ? sr[e] : -INFINITY;
                    const float v1 = e + 1 < nvis && e + 1 >= nlo ? sr[e + 1] : -INFINITY;
                    m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], v0, v1);
                }
            }
            const float mraw = valid ? fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) : -INFINITY;
            const float mx = mraw == -INFINITY ? -INFINITY
                             : capped ? p.softcap_log2 * tanh_acc(mraw * p.softcap_inv)
                                      : mraw * p.scale_log2;
            float corr = 1.f;
            if (mx > m_used + kRescaleThreshold) {
                corr = ex2(m_used - mx);  // 0 on the first visible block
                m_used = mx;
            }
            const float mref = m_used == -INFINITY ? 0.f : m_used;
            // P = 2^(s * scale_log2 - m): its hi part over the S columns and lo part
            // into the P lo columns; the row sum takes P itself.
            float2 rs2[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) rs2[k] = make_float2(0.f, 0.f);
            const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
            const float2 nm2 = make_float2(-mref, -mref);
            auto make_p = [&](bool masked, bool cap) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t ph[32], pl[32];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int c0 = 32 * half + 2 * k;
                        const float a0 = sr[c0], a1 = sr[c0 + 1];
                        float2 t;
                        if (cap) {
                            t.x = p.softcap_log2 * tanh_acc(a0 * p.softcap_inv) - mref;
                            t.y = p.softcap_log2 * tanh_acc(a1 * p.softcap_inv) - mref;
                        } else {
                            t = ffma2(make_float2(a0, a1), sc2, nm2);
                        }
                        if (masked) {
                            t.x = c0 < nvis && c0 >= nlo ? t.x : -INFINITY;
                            t.y = c0 + 1 < nvis && c0 + 1 >= nlo ? t.y : -INFINITY;
                        }
                        const float2 e2 = make_float2(ex2(t.x), ex2(t.y));
                        rs2[k & 3] = fadd2(rs2[k & 3], e2);
                        const float2 hi = make_float2(tf32_hi(e2.x), tf32_hi(e2.y));
                        const float2 lo = fadd2(e2, make_float2(-hi.x, -hi.y));
                        ph[2 * k] = __float_as_uint(hi.x);
                        ph[2 * k + 1] = __float_as_uint(hi.y);
                        pl[2 * k] = __float_as_uint(lo.x);
                        pl[2 * k + 1] = __float_as_uint(lo.y);
                    }
                    tmem_st32(ts + 32 * half, ph);
                    tmem_st32(tl + C::PL + 32 * half, pl);
                }
            };
            if (all_visible && !capped) make_p(false, false);
            else make_p(!all_visible, capped);
            const float2 r01 = fadd2(rs2[0], rs2[1]), r23 = fadd2(rs2[2], rs2[3]);
            const float rs = (r01.x + r01.y) + (r23.x + r23.y);
            l = l * corr + rs;
            // O holds every earlier PV product of this segment: S(j) was issued after
            // PV(j-1) by the same thread, and its commit tracks every earlier MMA.  At a
            // segment's first block O holds the previous segment, which the converter
            // folds with the max it ended on (below), so nothing is rescaled here.
            if (j % kSegBlocks != 0 && __any_sync(0xffffffffu, corr != 1.f)) {
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
            mbar_arrive(BAR(C::B_PFULL));
            if ((j + 1) % kSegBlocks == 0 && j + 1 < nb) {
                // the max this segment's O is relative to, for the converter's fold
                reinterpret_cast<float *>(smem + C::OFF_MSEG)[((j / kSegBlocks) & 1) * BM + r] =
                    m_used;
                mbar_arrive(BAR(C::B_MSEG));
            }
        }
        if (ok && !wait_warp(BAR(C::B_PVDONE), (nb - 1) & 1, abort_flag)) ok = false;
        // every segment but the last one is in the running sum
        const bool folded = (nb - 1) / kSegBlocks > 0;
        if (ok && folded && !wait_warp(BAR(C::B_FOLDED), 0, abort_flag)) ok = false;
        if (!ok) {
            failed = true;
            *abort_flag = 1;
        }
        // ---------------------------------------------------- epilogue
        tc_fence_after();
        if (ok) {
            const int64_t row = tile_row(p, b, hkv, valid ? f : 0);
            const float m_pre = m_used;  // the max O is relative to (before the sink)
            float osc = 1.f;  // direct mode folds the sink: m = sink log2 e, l = 1, acc = 0
            if (!p.split && p.sinks && valid) {
                const float sink2 = p.sinks[(row / p.q_len) % p.Hq] * kLog2e;
                const float M = fmaxf(m_used, sink2);
                osc = ex2(m_used - M);
                l = l * osc + ex2(sink2 - M);
                m_used = M;
            }
            const float inv = osc / l;
            const int64_t slot = row * p.n_chunks + c;
            // O = O_run 2^(m_run - m) + O_last: the folded segments and the last one
            const float m_fold = folded ? reinterpret_cast<const float *>(smem + C::OFF_MRUN)[r]
                                        : -INFINITY;
            const float fr = m_fold == -INFINITY ? 0.f : ex2(m_fold - m_pre);
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                tmem_ld32(to + cc * 32, o);
                tmem_wait_ld();
                if (!valid) continue;
                float4 *dst = p.split
                                  ? reinterpret_cast<float4 *>(p.ws_acc + slot * D + cc * 32)
                                  : reinterpret_cast<float4 *>(static_cast<float *>(p.out) +
                                                               row * D + cc * 32);
                const float sc = p.split ? 1.f : inv;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float4 a = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                           __uint_as_float(o[4 * k + 2]),
                                           __uint_as_float(o[4 * k + 3]));
                    if (folded) {
                        const float4 x = dst[k];
                        a = make_float4(fmaf(x.x, fr, a.x), fmaf(x.y, fr, a.y),
                                        fmaf(x.z, fr, a.z), fmaf(x.w, fr, a.w));
                    }
                    dst[k] = make_float4(a.x * sc, a.y * sc, a.z * sc, a.w * sc);
                }
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

template <int D>
cudaError_t launch_instance(const TcParams &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                            const CUtensorMap &tmV, cudaStream_t stream) {
    using C = Cfg<D>;
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !configured[dev]) {
        err = cudaFuncSetAttribute(fmha_tf32x3_kernel<D>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (err != cudaSuccess) return err;
        configured[dev] = 1;
    }
    const int tiles = p.B * p.Hkv * p.tiles_per_unit;
    dim3 grid = p.split ? dim3(p.n_chunks, tiles, 1) : dim3(tiles, 1, 1);
    fmha_tf32x3_kernel<D><<<grid, C::kThreads, C::kSmem, stream>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fmha_tc_f32(const TcParams &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                               const CUtensorMap &tmV, cudaStream_t stream) {
    return p.D == 64 ? launch_instance<64>(p, tmQ, tmK, tmV, stream)
                     : launch_instance<128>(p, tmQ, tmK, tmV, stream);
}

}  // namespace atlas
