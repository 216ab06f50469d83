// fmha_tc.cu -- causal prefill and suffix-query attention on the 5th-generation
// tensor cores (tcgen05 + TMEM), fed by TMA from the page pool.
//
// One CTA owns a 128-row query tile of one (sequence, kv head): rows are the
// G*q_len (q head, query row) pairs of the GQA group in memory order, so a tile
// is one q head's 128 consecutive prompt rows (prefill) or all G heads x SQ rows
// (suffix, G*SQ = 128).  It walks 128-key blocks up to the last key any of its
// rows may see -- blocks past that are never loaded (the causal block skip of
// the CPUAttn README, "Parallel lowerings") -- and folds each block into a
// per-row online-softmax state, the page fold of the CFR-Atlas README.
//
// Warp roles (256 threads, one CTA per SM):
//   warp 0      TMA producer: the Q tile once, then K and V blocks gathered page
//               by page through the page table into a 2-stage ring.
//   warp 1      allocates TMEM; one lane issues the MMAs:
//                 S_j  = Q K_j^T  (M=128, N=128, K=128) into TMEM buffer j%2
//                 O   += P_j V_j  (M=128, N=128, K=128) into TMEM, P from smem
//   warp 2      zeroes V rows past the last key of the final block (they may be
//               NaN-poisoned or stale, and 0 * NaN would reach O).
//   warps 4-7   softmax: one thread per query row reads its S row from TMEM,
//               masks, takes the row max, exponentiates (ex2), accumulates l,
//               rescales O in TMEM when its max grew by more than 2^8, and writes
//               P (bf16; plus the bf16 remainder P - bf16(P) for tiles whose rows
//               see few keys) into smem for the PV product.  Epilogue: O / l.
// Every mbarrier wait is bounded; a CTA that gives up records ATLAS_DEV_TIMEOUT,
// lets its copies and MMAs finish, frees TMEM and writes NaN.
#include "internal.h"
#include "ptx.cuh"

#include <math.h>

namespace atlas {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per block
constexpr int KV_STAGES = 2;
constexpr int kTcThreads = 256;
constexpr int kTileBytes = 128 * 128 * 2;  // a 128 x 128 bf16 tile (Q, K, V or P)
constexpr int kSlab = 128 * 128;           // one 64-column slab of such a tile

constexpr int OFF_Q = 0;
constexpr int OFF_P = OFF_Q + kTileBytes;
constexpr int OFF_PL = OFF_P + kTileBytes;
// V stages sit below K stages: the PV product's MN-major B descriptor strides by
// a 16 KB slab, and every address it can form stays inside the CTA's allocation.
constexpr int OFF_V = OFF_PL + kTileBytes;
constexpr int OFF_K = OFF_V + KV_STAGES * kTileBytes;
constexpr int OFF_BAR = OFF_K + KV_STAGES * kTileBytes;
enum {
    B_Q = 0,
    B_KFULL = 1,
    B_KEMPTY = B_KFULL + KV_STAGES,
    B_VFULL = B_KEMPTY + KV_STAGES,
    B_VEMPTY = B_VFULL + KV_STAGES,
    B_SFULL = B_VEMPTY + KV_STAGES,
    B_SFREE = B_SFULL + 2,
    B_PFULL = B_SFREE + 2,
    B_ODONE = B_PFULL + 1,
    B_TAIL_READY = B_ODONE + 1,  // single use: the last V block has landed
    B_TAIL = B_TAIL_READY + 1,   // single use: its rows past the last key are zeroed
    B_FINAL = B_TAIL + 1,
    NUM_BARS = B_FINAL + 1
};
constexpr int OFF_TMEM = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_FLAG = OFF_TMEM + 8;
constexpr int kTcSmem = OFF_FLAG + 8 + 1024;  // + slack to align the base to 1024 B
static_assert(kTcSmem <= 232448, "shared memory budget");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_S = 0;    // two S buffers: columns [0,128) and [128,256)
constexpr uint32_t TM_O = 256;  // O accumulator: columns [256,384)
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows 256x

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort, kWaitLimitNs));
}

// Writes NaN to the rows of this tile (direct mode) -- used when the tile's
// sequence or pages are invalid, or a wait gave up.
__device__ void nan_rows(const TcParams &p, int b, int hkv, int f0, int rows_unit, int r) {
    const int f = f0 + r;
    if (f >= rows_unit) return;
    const int64_t row = ((int64_t)b * p.Hq + (int64_t)hkv * p.G) * p.q_len + f;
    const float nan = __int_as_float(0x7fc00000);
    if (p.out_bf16) {
        uint4 v;
        v.x = v.y = v.z = v.w = 0x7fc07fc0u;
        uint4 *o = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + row * 128);
        for (int k = 0; k < 16; ++k) o[k] = v;
    } else {
        float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + row * 128);
        for (int k = 0; k < 32; ++k) o[k] = make_float4(nan, nan, nan, nan);
    }
    if (p.lse) p.lse[row] = nan;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    fmha_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_FLAG);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#define BAR(i) (sb + OFF_BAR + 8u * (uint32_t)(i))

    // ------------------------------------------------------------ work item
    const int units = p.B * p.Hkv;
    int u, t, c;
    if (p.split) {
        c = blockIdx.x;
        u = blockIdx.y / p.tiles_per_unit;
        t = blockIdx.y % p.tiles_per_unit;
    } else {
        c = 0;
        const int r = blockIdx.x;
        if (p.tiles_per_head > 0) {  // heavy tiles (late prompt rows) first
            const int per = units * p.G;
            const int rest = r % per;
            u = rest / p.G;
            t = (rest % p.G) * p.tiles_per_head + (p.tiles_per_head - 1 - r / per);
        } else {
            u = r % units;
            t = r / units;
        }
    }
    const int b = u / p.Hkv, hkv = u % p.Hkv;
    const int L = p.seq_lens[b];
    const int rows_unit = p.G * p.q_len;
    const int f0 = t * BM;
    const int f_last = min(f0 + BM, rows_unit) - 1;
    const bool spans = (f_last / p.q_len) != (f0 / p.q_len);
    const int i_max = spans ? p.q_len - 1 : f_last % p.q_len;
    const int i_min = spans ? 0 : f0 % p.q_len;

    if (L < p.q_len || L > p.max_pages * p.P || (p.require_full && L != p.q_len)) {
        if (threadIdx.x == 0 && c == 0 && p.status) atomicOr(p.status, ATLAS_DEV_BAD_SEQLEN);
        if (!p.split && threadIdx.x < BM) nan_rows(p, b, hkv, f0, rows_unit, threadIdx.x);
        return;  // split mode: the merge writes NaN rows for this sequence
    }
    const int kv_hi = L - p.q_len + i_max + 1;   // keys the tile's last row sees
    const int kv_min = L - p.q_len + i_min + 1;  // keys its first row sees
    int kv_begin = 0, kv_end = kv_hi;
    if (p.split) {
        kv_begin = c * p.chunk;
        if (kv_begin >= kv_hi) return;
        kv_end = min(kv_hi, kv_begin + p.chunk);
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
                if (!p.split) {
                    nan_rows(p, b, hkv, f0, rows_unit, threadIdx.x);
                } else if (f0 + (int)threadIdx.x < rows_unit) {
                    const int64_t row =
                        ((int64_t)b * p.Hq + (int64_t)hkv * p.G) * p.q_len + f0 + threadIdx.x;
                    float *ml = p.ws_ml + (row * p.n_chunks + c) * 2;
                    ml[0] = ml[1] = __int_as_float(0x7fc00000);
                }
            }
            return;
        }
    }
    const bool hilo = kv_min < p.hilo_below;
    const int last_kb = kv_begin + (nb - 1) * BN;
    const bool tail_fix = kv_end < last_kb + BN;
    const int tail_first = kv_end - last_kb;

    // ------------------------------------------------------------ setup
    if (threadIdx.x == 0) {
        mbar_init(BAR(B_Q), 1);
        for (int s = 0; s < KV_STAGES; ++s) {
            mbar_init(BAR(B_KFULL + s), 1);
            mbar_init(BAR(B_KEMPTY + s), 1);
            mbar_init(BAR(B_VFULL + s), 1);
            mbar_init(BAR(B_VEMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(B_SFULL + s), 1);
            mbar_init(BAR(B_SFREE + s), BM);
        }
        mbar_init(BAR(B_PFULL), BM);
        mbar_init(BAR(B_ODONE), 1);
        mbar_init(BAR(B_TAIL_READY), 1);
        mbar_init(BAR(B_TAIL), 1);
        mbar_init(BAR(B_FINAL), 1);
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
            const int qrow = (b * p.Hq + hkv * p.G) * p.q_len + f0;
            mbar_arrive_expect_tx(BAR(B_Q), kTileBytes);
            tma_load_2d(sb + OFF_Q, &tmQ, 0, qrow, BAR(B_Q));
            tma_load_2d(sb + OFF_Q + kSlab, &tmQ, 64, qrow, BAR(B_Q));
            const int BR = p.P < BN ? p.P : BN;
            int issued_k = 0, issued_v = 0;
            for (int j = 0; j < nb && !failed; ++j) {
                const int s = j % KV_STAGES, use = j / KV_STAGES;
                const int kb = kv_begin + j * BN;
                const int ke = min(kb + BN, kv_end);
                const int nbox = (ke - kb + BR - 1) / BR;
                const uint32_t bytes = (uint32_t)(nbox * BR * 128 * 2);
                for (int kv = 0; kv < 2; ++kv) {
                    const int full = (kv == 0 ? B_KFULL : B_VFULL) + s;
                    const int empty = (kv == 0 ? B_KEMPTY : B_VEMPTY) + s;
                    if (use > 0 &&
                        !mbar_wait_bounded(BAR(empty), (use - 1) & 1, abort_flag, kWaitLimitNs)) {
                        failed = true;
                        break;
                    }
                    const CUtensorMap *map = kv == 0 ? &tmK : &tmV;
                    const uint32_t dst = sb + (kv == 0 ? OFF_K : OFF_V) + s * kTileBytes;
                    mbar_arrive_expect_tx(BAR(full), bytes);
                    for (int bx = 0; bx < nbox; ++bx) {
                        const int tk = kb + bx * BR;
                        const int phys = p.page_table[(int64_t)b * p.max_pages + tk / p.P];
                        const int y = (phys * p.Hkv + hkv) * p.P + (tk % p.P);
                        tma_load_2d(dst + bx * BR * 128, map, 0, y, BAR(full));
                        tma_load_2d(dst + kSlab + bx * BR * 128, map, 64, y, BAR(full));
                    }
                    if (kv == 0) issued_k = j + 1;
                    else issued_v = j + 1;
                }
            }
            if (failed) {
                *abort_flag = 1;
                int no_abort = 0;
                mbar_wait_bounded(BAR(B_Q), 0, &no_abort, kWaitLimitNs);
                for (int j = max(0, issued_k - KV_STAGES); j < issued_k; ++j)
                    mbar_wait_bounded(BAR(B_KFULL + j % KV_STAGES), (j / KV_STAGES) & 1, &no_abort,
                                      kWaitLimitNs);
                for (int j = max(0, issued_v - KV_STAGES); j < issued_v; ++j)
                    mbar_wait_bounded(BAR(B_VFULL + j % KV_STAGES), (j / KV_STAGES) & 1, &no_abort,
                                      kWaitLimitNs);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(128, 128, false);
            constexpr uint32_t idPV = idesc_bf16_f32(128, 128, true);
            bool ok = mbar_wait_bounded(BAR(B_Q), 0, abort_flag, kWaitLimitNs);
            tc_fence_after();
            auto issue_s = [&](int j) -> bool {
                const int s = j % KV_STAGES, sbuf = j & 1;
                if (!mbar_wait_bounded(BAR(B_KFULL + s), (j / KV_STAGES) & 1, abort_flag,
                                       kWaitLimitNs))
                    return false;
                if (j >= 2 && !mbar_wait_bounded(BAR(B_SFREE + sbuf), ((j >> 1) - 1) & 1,
                                                 abort_flag, kWaitLimitNs))
                    return false;
                tc_fence_after();
                const uint32_t kbase = sb + OFF_K + s * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * kSlab + (kk & 3) * 32;
                    umma_bf16(tmem + TM_S + sbuf * 128, sdesc_sw128(sb + OFF_Q + off, 16, 1024),
                              sdesc_sw128(kbase + off, 16, 1024), idS, kk > 0);
                }
                umma_commit(BAR(B_SFULL + sbuf));
                umma_commit(BAR(B_KEMPTY + s));
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 0; ok && j < nb; ++j) {
                if (j + 1 < nb && !issue_s(j + 1)) {
                    ok = false;
                    break;
                }
                const int s = j % KV_STAGES;
                if (!mbar_wait_bounded(BAR(B_PFULL), j & 1, abort_flag, kWaitLimitNs) ||
                    !mbar_wait_bounded(BAR(B_VFULL + s), (j / KV_STAGES) & 1, abort_flag,
                                       kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                if (j == nb - 1 && tail_fix) {
                    // Hand the landed last V block to the fix-up warp and wait for it.
                    // (Only this thread observes every phase of the V ring in order.)
                    mbar_arrive(BAR(B_TAIL_READY));
                    if (!mbar_wait_bounded(BAR(B_TAIL), 0, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                }
                tc_fence_after();
                const uint32_t vbase = sb + OFF_V + s * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t aoff = (kk >> 2) * kSlab + (kk & 3) * 32;
                    umma_bf16(tmem + TM_O, sdesc_sw128(sb + OFF_P + aoff, 16, 1024),
                              sdesc_sw128(vbase + kk * 2048, kSlab, 1024), idPV,
                              (j > 0 || kk > 0) ? 1u : 0u);
                }
                if (hilo) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t aoff = (kk >> 2) * kSlab + (kk & 3) * 32;
                        umma_bf16(tmem + TM_O, sdesc_sw128(sb + OFF_PL + aoff, 16, 1024),
                                  sdesc_sw128(vbase + kk * 2048, kSlab, 1024), idPV, 1u);
                    }
                }
                umma_commit(BAR(B_ODONE));
                umma_commit(BAR(B_VEMPTY + s));
            }
            if (!ok) {
                failed = true;
                *abort_flag = 1;
            }
            // Every MMA issued so far completes before TMEM is released.
            umma_commit(BAR(B_FINAL));
            int no_abort = 0;
            mbar_wait_bounded(BAR(B_FINAL), 0, &no_abort, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 2) {
        // -------------------------------------------------------- tail fix-up
        if (tail_fix) {
            const int j = nb - 1, s = j % KV_STAGES;
            if (wait_warp(BAR(B_TAIL_READY), 0, abort_flag)) {
                const uint32_t vbase = sb + OFF_V + s * kTileBytes;
                for (int idx = lane; idx < (BN - tail_first) * 16; idx += 32) {
                    const int row = tail_first + idx / 16, q = idx % 16;
                    st_shared_v4(vbase + (q / 8) * kSlab + row * 128 + (q % 8) * 16, 0u, 0u, 0u,
                                 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_TAIL));
            } else {
                failed = true;
            }
        }
    } else if (warp >= 4) {
        // -------------------------------------------------------- softmax
        const int q4 = warp - 4;
        const int r = q4 * 32 + lane;
        const int f = f0 + r;
        const bool valid = f < rows_unit;
        const int i = valid ? f % p.q_len : 0;
        const int lim_row = valid ? min(L - p.q_len + i + 1, kv_end) : 0;
        const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nb; ++j) {
            const int sbuf = j & 1;
            if (!wait_warp(BAR(B_SFULL + sbuf), (j >> 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_ld32(tl + TM_S + sbuf * 128 + cc * 32, sr[cc]);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(BAR(B_SFREE + sbuf));

            const int nvis = lim_row - (kv_begin + j * BN);  // visible columns of this row
            // Scores in log2 units; eight independent max chains keep the pipes busy.
            float mx8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mx8[k] = -INFINITY;
            if (__all_sync(0xffffffffu, nvis >= BN)) {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float v = __uint_as_float(sr[cc][e]) * p.scale_log2;
                        sr[cc][e] = __float_as_uint(v);
                        mx8[e & 7] = fmaxf(mx8[e & 7], v);
                    }
            } else {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float v = (cc * 32 + e) < nvis
                                            ? __uint_as_float(sr[cc][e]) * p.scale_log2
                                            : -INFINITY;
                        sr[cc][e] = __float_as_uint(v);
                        mx8[e & 7] = fmaxf(mx8[e & 7], v);
                    }
            }
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            float corr = 1.f;
            if (mx > m_used + kRescaleThreshold) {
                corr = ex2(m_used - mx);  // 0 on the first visible block
                m_used = mx;
            }
            const float mref = m_used == -INFINITY ? 0.f : m_used;
            float rs8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) rs8[k] = 0.f;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float pv = ex2(__uint_as_float(sr[cc][e]) - mref);
                    sr[cc][e] = __float_as_uint(pv);
                    rs8[e & 7] += pv;
                }
            const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) +
                             ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
            l = l * corr + rs;

            // PV of the previous block must be done before O is rescaled or P rewritten.
            if (j > 0 && !wait_warp(BAR(B_ODONE), (j - 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (j > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tl + TM_O + cc * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
                    tmem_st32(tl + TM_O + cc * 32, o);
                }
                tmem_wait_st();
            }
            // P row r into the K-major, 128-byte-swizzled A tile (and its remainder).
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                const int cc = ch / 4, e0 = (ch % 4) * 8;
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float a = __uint_as_float(sr[cc][e0 + 2 * k]);
                    const float bb = __uint_as_float(sr[cc][e0 + 2 * k + 1]);
                    const __nv_bfloat162 h = __floats2bfloat162_rn(a, bb);
                    hw[k] = *reinterpret_cast<const uint32_t *>(&h);
                    if (hilo) {
                        const float2 hf = __bfloat1622float2(h);
                        lw[k] = pack_bf16(a - hf.x, bb - hf.y);
                    }
                }
                const uint32_t off = (ch / 8) * kSlab + sw128(r, ch % 8);
                st_shared_v4(sb + OFF_P + off, hw[0], hw[1], hw[2], hw[3]);
                if (hilo) st_shared_v4(sb + OFF_PL + off, lw[0], lw[1], lw[2], lw[3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(BAR(B_PFULL));
        }
        if (ok && !wait_warp(BAR(B_ODONE), (nb - 1) & 1, abort_flag)) ok = false;
        if (!ok) {
            failed = true;
            *abort_flag = 1;
        }
        // ---------------------------------------------------- epilogue
        tc_fence_after();
        uint32_t o[4][32];
        if (ok) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_ld32(tl + TM_O + cc * 32, o[cc]);
            tmem_wait_ld();
        }
        if (valid) {
            const int64_t row = ((int64_t)b * p.Hq + (int64_t)hkv * p.G) * p.q_len + f;
            if (p.split) {
                const int64_t slot = row * p.n_chunks + c;
                float4 *dst = reinterpret_cast<float4 *>(p.ws_acc + slot * 128);
                if (ok) {
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        dst[k] = make_float4(__uint_as_float(o[k / 8][(k % 8) * 4]),
                                             __uint_as_float(o[k / 8][(k % 8) * 4 + 1]),
                                             __uint_as_float(o[k / 8][(k % 8) * 4 + 2]),
                                             __uint_as_float(o[k / 8][(k % 8) * 4 + 3]));
                    p.ws_ml[slot * 2] = m_used;
                    p.ws_ml[slot * 2 + 1] = l;
                } else {
                    p.ws_ml[slot * 2] = p.ws_ml[slot * 2 + 1] = __int_as_float(0x7fc00000);
                }
            } else if (ok) {
                const float inv = 1.f / l;
                if (p.out_bf16) {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) +
                                                           row * 128);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int cc = k / 4, e0 = (k % 4) * 8;
                        uint4 v;
                        v.x = pack_bf16(__uint_as_float(o[cc][e0 + 0]) * inv,
                                        __uint_as_float(o[cc][e0 + 1]) * inv);
                        v.y = pack_bf16(__uint_as_float(o[cc][e0 + 2]) * inv,
                                        __uint_as_float(o[cc][e0 + 3]) * inv);
                        v.z = pack_bf16(__uint_as_float(o[cc][e0 + 4]) * inv,
                                        __uint_as_float(o[cc][e0 + 5]) * inv);
                        v.w = pack_bf16(__uint_as_float(o[cc][e0 + 6]) * inv,
                                        __uint_as_float(o[cc][e0 + 7]) * inv);
                        dst[k] = v;
                    }
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + row * 128);
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        dst[k] = make_float4(__uint_as_float(o[k / 8][(k % 8) * 4]) * inv,
                                             __uint_as_float(o[k / 8][(k % 8) * 4 + 1]) * inv,
                                             __uint_as_float(o[k / 8][(k % 8) * 4 + 2]) * inv,
                                             __uint_as_float(o[k / 8][(k % 8) * 4 + 3]) * inv);
                }
                if (p.lse) p.lse[row] = kLn2 * (m_used + log2f(l));
            } else {
                nan_rows(p, b, hkv, f0, rows_unit, r);
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

}  // namespace

cudaError_t launch_fmha_tc(const TcParams &p, const CUtensorMap &tmQ, const CUtensorMap &tmK,
                           const CUtensorMap &tmV, cudaStream_t stream) {
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !configured[dev]) {
        err = cudaFuncSetAttribute(fmha_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kTcSmem);
        if (err != cudaSuccess) return err;
        configured[dev] = 1;
    }
    const int tiles = p.B * p.Hkv * p.tiles_per_unit;
    dim3 grid = p.split ? dim3(p.n_chunks, tiles, 1) : dim3(tiles, 1, 1);
    fmha_tc_kernel<<<grid, kTcThreads, kTcSmem, stream>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

}  // namespace atlas
