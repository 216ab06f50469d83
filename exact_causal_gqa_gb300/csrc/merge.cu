// merge.cu -- structured log-sum-exp merge of split-KV partial states
// (CPUAttn README, "Operator model": split-K is offered only with a structured
// merge).  For one output row with splits s = 0..S-1 holding (m_s, l_s, acc_s),
// m in log2 units:
//   M = max_s m_s,  w_s = 2^(m_s - M),  o = sum_s w_s acc_s / sum_s w_s l_s,
//   lse = ln 2 * (M + log2 sum_s w_s l_s).
// W warps per row (W = 1, 2 or 4, chosen from the row count so that the grid
// holds enough warps): warp k of a row takes splits k, k + W, ...; its lanes split
// the head dimension.  Each warp keeps a running maximum (its sums are rescaled
// when a group of splits raises it), so a warp's share of up to kGroup splits
// costs one round trip to memory; with W > 1 the warps' states are combined the
// same way through shared memory.  S is derived on the device from seq_lens, so
// no host sync is needed.
// Launched as a programmatic dependent of the split kernel before it: its CTAs
// may start while that kernel's last CTAs still run, read their sequence's
// length, and wait (griddepcontrol.wait) before the first partial is read.
#include "internal.h"
#include "ptx.cuh"

#include <math.h>

namespace atlas {
namespace {

constexpr int kWarps = 4;  // warps per CTA: 4 / W rows
constexpr int kGroup = 8;  // splits of one warp whose loads are in flight together

template <int D>
__global__ void __launch_bounds__(kWarps * 32) merge_kernel(const MergeParams p) {
    constexpr int DPL = D / 32;
    const int warp = (int)(threadIdx.x / 32), lane = (int)(threadIdx.x % 32);
    const int W = p.warps_per_row;
    const int sub = warp % W;  // this warp's share of its row's splits
    // rows = B * Hq * q_len < 2^31 (the plan refuses larger calls): 32-bit index math
    const int row = (int)blockIdx.x * (kWarps / W) + warp / W;
    bool active = row < p.B * p.Hq * p.q_len;
    const int bh = active ? row / p.q_len : 0;  // b * Hq + h
    const int i = active ? row - bh * p.q_len : 0;
    const int b = bh / p.Hq;
    const int L = active ? p.seq_lens[b] : 0;
    const int qn = !active ? 0 : p.q_lens ? p.q_lens[b] : p.q_len;  // ragged: rows of b
    const bool bad_len = qn < 0 || qn > p.q_len || L < qn || L > p.max_pages * p.P ||
                         (p.require_full && L != qn);
    if (!bad_len && i >= qn) active = false;  // padding row: not a query, not written
    if (W == 1 && !active) return;            // (W > 1: every warp reaches the exchange)
    // the split kernel that wrote the partials has completed, its writes visible
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // This warp's state: running max M (log2 units), sum, acc slice, NaN seen.  A
    // sink is one more state (m = sink * log2 e, l = 1, acc = 0), held by warp 0.
    float M = -INFINITY, lsum = 0.f, acc[DPL];
#pragma unroll
    for (int j = 0; j < DPL; ++j) acc[j] = 0.f;
    bool has_nan = false;
    if (active && !bad_len) {
        const int visible = L - qn + i + 1;
        // splits holding this row's keys: [first, nsplit)
        const int chunk =
            p.balanced ? balanced_split(min(L, p.max_pages * p.P), p.chunk) : p.chunk;
        const int first = p.window > 0 ? max(0, visible - p.window) / chunk : 0;
        const int nsplit = (visible + chunk - 1) / chunk;
        const float *ml = p.ws_ml + (int64_t)row * p.n_chunks * 2;
        if (p.sinks && sub == 0) {
            M = p.sinks[bh - b * p.Hq] * kLog2e;
            lsum = 1.f;
            has_nan = isnan(M);
        }
        const float *wa = p.ws_acc + (int64_t)row * p.n_chunks * D + lane * DPL;
        // [kWarps][kGroup][32 lanes] x 16 bytes (D = 128): each lane's slice of a
        // split lands here, so no registers are held while the loads are in flight
        __shared__ __align__(16) uint8_t stage[D == 128 ? kWarps * kGroup * 512 : 16];
        const uint32_t my_stage = smem_u32(stage) + (uint32_t)(warp * kGroup * 512 + lane * 16);
        for (int s0 = first + sub; s0 < nsplit; s0 += kGroup * W) {
            float m[kGroup], l[kGroup], a[kGroup][DPL];
            if (DPL == 4) {
#pragma unroll
                for (int u = 0; u < kGroup; ++u)
                    if (s0 + u * W < nsplit)
                        cp_async16(my_stage + u * 512, wa + (int64_t)(s0 + u * W) * D, 16);
                cp_async_commit();
            }
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                const int s = s0 + u * W;
                m[u] = -INFINITY;
                l[u] = 0.f;
#pragma unroll
                for (int j = 0; j < DPL; ++j) a[u][j] = 0.f;
                if (s < nsplit) {
                    m[u] = ml[2 * s];
                    l[u] = ml[2 * s + 1];
                    if (DPL != 4) {
                        const float2 v = *reinterpret_cast<const float2 *>(wa + (int64_t)s * D);
                        a[u][0] = v.x;
                        a[u][1 % DPL] = v.y;
                    }
                }
            }
            if (DPL == 4) cp_async_wait<0>();
            float Mg = M;
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                if (isnan(m[u]) || isnan(l[u])) has_nan = true;
                else if (l[u] > 0.f) Mg = fmaxf(Mg, m[u]);
            }
            if (Mg > M) {  // M = -inf only while the sums are still zero
                const float r = ex2(M - Mg);
                lsum *= r;
#pragma unroll
                for (int j = 0; j < DPL; ++j) acc[j] *= r;
                M = Mg;
            }
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                if (DPL == 4 && s0 + u * W < nsplit) {
                    const uint4 v = ld_shared_v4(my_stage + u * 512);
                    a[u][0] = __uint_as_float(v.x);
                    a[u][1 % DPL] = __uint_as_float(v.y);
                    a[u][2 % DPL] = __uint_as_float(v.z);
                    a[u][3 % DPL] = __uint_as_float(v.w);
                }
                const float w = l[u] > 0.f ? ex2(m[u] - M) : 0.f;
                lsum = fmaf(w, l[u], lsum);
#pragma unroll
                for (int j = 0; j < DPL; ++j) acc[j] = fmaf(w, a[u][j], acc[j]);
            }
        }
    }
    if (W > 1) {
        // The row's warps combine their states in warp order (sub 0 first).
        __shared__ float x_acc[kWarps][DPL][32];
        __shared__ float x_m[kWarps], x_l[kWarps];
        __shared__ int x_nan[kWarps];
#pragma unroll
        for (int j = 0; j < DPL; ++j) x_acc[warp][j][lane] = acc[j];
        if (lane == 0) {
            x_m[warp] = M;
            x_l[warp] = lsum;
            x_nan[warp] = has_nan;
        }
        __syncthreads();
        if (sub != 0 || !active) return;
        for (int k = 1; k < W; ++k) M = fmaxf(M, x_m[warp + k]);
        if (M > -INFINITY) {
            const float r0 = ex2(x_m[warp] - M);
            lsum *= r0;
#pragma unroll
            for (int j = 0; j < DPL; ++j) acc[j] *= r0;
            for (int k = 1; k < W; ++k) {
                const float r = ex2(x_m[warp + k] - M);  // 0 for a warp with no state
                lsum = fmaf(r, x_l[warp + k], lsum);
#pragma unroll
                for (int j = 0; j < DPL; ++j) acc[j] = fmaf(r, x_acc[warp + k][j][lane], acc[j]);
            }
        }
        for (int k = 1; k < W; ++k) has_nan |= x_nan[warp + k] != 0;
    }

    float o[DPL];
    float lse = __int_as_float(0x7fc00000);
    if (bad_len || has_nan || M == -INFINITY) {
#pragma unroll
        for (int j = 0; j < DPL; ++j) o[j] = __int_as_float(0x7fc00000);
    } else {
#pragma unroll
        for (int j = 0; j < DPL; ++j) o[j] = acc[j] / lsum;
        lse = kLn2 * (M + log2f(lsum));
    }
    const int64_t off = (int64_t)row * D + lane * DPL;
    if (p.out_bf16) {
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out) + off;
        if (DPL == 4) {
            uint2 v;
            v.x = pack_bf16(o[0], o[1 % DPL]);
            v.y = pack_bf16(o[2 % DPL], o[3 % DPL]);
            *reinterpret_cast<uint2 *>(out) = v;
        } else {
            *reinterpret_cast<uint32_t *>(out) = pack_bf16(o[0], o[1 % DPL]);
        }
    } else {
        float *out = static_cast<float *>(p.out) + off;
        if (DPL == 4)
            *reinterpret_cast<float4 *>(out) =
                make_float4(o[0], o[1 % DPL], o[2 % DPL], o[3 % DPL]);
        else
            *reinterpret_cast<float2 *>(out) = make_float2(o[0], o[1 % DPL]);
    }
    if (p.lse && lane == 0) p.lse[row] = lse;
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream) {
    const int64_t rows = (int64_t)p.B * p.Hq * p.q_len;
    if (rows >= INT32_MAX) return cudaErrorInvalidValue;  // make_plan refuses these
    // Several warps per row when the rows alone would leave most warp slots empty
    // and there are splits to share.
    MergeParams q = p;
    const int64_t target = (int64_t)(p.sms > 0 ? p.sms : 1) * 16;
    q.warps_per_row = 1;
    while (q.warps_per_row < kWarps && rows * q.warps_per_row < target &&
           p.n_chunks >= 2 * q.warps_per_row)
        q.warps_per_row *= 2;
    const int64_t rows_per_cta = kWarps / q.warps_per_row;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + rows_per_cta - 1) / rows_per_cta), 1, 1);
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return p.D == 128 ? cudaLaunchKernelEx(&cfg, merge_kernel<128>, q)
                      : cudaLaunchKernelEx(&cfg, merge_kernel<64>, q);
}

}  // namespace atlas
