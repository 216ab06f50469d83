// merge.cu -- structured log-sum-exp merge of split-KV partial states
// (CPUAttn README, "Operator model": split-K is offered only with a structured
// merge).  For one output row with splits s = 0..S-1 holding (m_s, l_s, acc_s),
// m in log2 units:
//   M = max_s m_s,  w_s = 2^(m_s - M),  o = sum_s w_s acc_s / sum_s w_s l_s,
//   lse = ln 2 * (M + log2 sum_s w_s l_s).
// One warp per row; lanes split the head dimension (float4 / float2 loads), and
// M is a running maximum (the sums so far are rescaled when a group of splits
// raises it), so a row with up to kGroup splits costs one round trip to memory.
// S is derived on the device from seq_lens, so no host sync is needed.
// Launched as a programmatic dependent of the split kernel before it: its CTAs
// may start while that kernel's last CTAs still run, read their sequence's
// length, and wait (griddepcontrol.wait) before the first partial is read.
#include "internal.h"
#include "ptx.cuh"

#include <math.h>

namespace atlas {
namespace {

constexpr int kRowsPerCta = 4;
constexpr int kGroup = 8;  // splits whose loads are in flight together

template <int D>
__global__ void __launch_bounds__(kRowsPerCta * 32) merge_kernel(const MergeParams p) {
    constexpr int DPL = D / 32;
    const int lane = threadIdx.x % 32;
    // rows = B * Hq * q_len < 2^31 (the plan refuses larger calls): 32-bit index math
    const int row = (int)blockIdx.x * kRowsPerCta + (int)(threadIdx.x / 32);
    if (row >= p.B * p.Hq * p.q_len) return;
    const int bh = row / p.q_len;  // b * Hq + h
    const int i = row - bh * p.q_len;
    const int b = bh / p.Hq;
    const int L = p.seq_lens[b];
    const int qn = p.q_lens ? p.q_lens[b] : p.q_len;  // ragged: query rows of sequence b
    const bool bad_len = qn < 0 || qn > p.q_len || L < qn || L > p.max_pages * p.P ||
                         (p.require_full && L != qn);
    if (!bad_len && i >= qn) return;  // padding row: not a query, not written
    // the split kernel that wrote the partials has completed, its writes visible
    asm volatile("griddepcontrol.wait;" ::: "memory");

    float o[DPL];
    float lse = __int_as_float(0x7fc00000);
    bool nan_row = bad_len;
    if (!bad_len) {
        const int visible = L - qn + i + 1;
        // splits holding this row's keys: [first, nsplit)
        const int chunk =
            p.balanced ? balanced_split(min(L, p.max_pages * p.P), p.chunk) : p.chunk;
        const int first = p.window > 0 ? max(0, visible - p.window) / chunk : 0;
        const int nsplit = (visible + chunk - 1) / chunk;
        const float *ml = p.ws_ml + (int64_t)row * p.n_chunks * 2;
        // A sink is one more state: m = sink * log2(e), l = 1, acc = 0.
        const float sink2 =
            p.sinks ? p.sinks[bh - b * p.Hq] * kLog2e : -INFINITY;
        // One pass over the splits in groups of kGroup: every load of a group (m, l
        // and the lane's slice of acc) is issued before its first use, so a row costs
        // one round trip per group.  The running max M starts at the sink's logit;
        // when a group raises it, the sums so far are rescaled (exact: they share M).
        float M = sink2;
        float lsum = p.sinks ? 1.f : 0.f;
        float acc[DPL];
#pragma unroll
        for (int j = 0; j < DPL; ++j) acc[j] = 0.f;
        bool has_nan = isnan(sink2);
        const float *wa = p.ws_acc + (int64_t)row * p.n_chunks * D + lane * DPL;
        for (int s0 = first; s0 < nsplit; s0 += kGroup) {
            float m[kGroup], l[kGroup], a[kGroup][DPL];
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                const int s = s0 + u;
                m[u] = -INFINITY;
                l[u] = 0.f;
#pragma unroll
                for (int j = 0; j < DPL; ++j) a[u][j] = 0.f;
                if (s < nsplit) {
                    m[u] = ml[2 * s];
                    l[u] = ml[2 * s + 1];
                    if (DPL == 4) {
                        const float4 v = *reinterpret_cast<const float4 *>(wa + (int64_t)s * D);
                        a[u][0] = v.x;
                        a[u][1] = v.y;
                        a[u][2 % DPL] = v.z;
                        a[u][3 % DPL] = v.w;
                    } else {
                        const float2 v = *reinterpret_cast<const float2 *>(wa + (int64_t)s * D);
                        a[u][0] = v.x;
                        a[u][1] = v.y;
                    }
                }
            }
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
                const float w = l[u] > 0.f ? ex2(m[u] - M) : 0.f;
                lsum = fmaf(w, l[u], lsum);
#pragma unroll
                for (int j = 0; j < DPL; ++j) acc[j] = fmaf(w, a[u][j], acc[j]);
            }
        }
        nan_row = has_nan || M == -INFINITY;
        if (!nan_row) {
#pragma unroll
            for (int j = 0; j < DPL; ++j) o[j] = acc[j] / lsum;
            lse = kLn2 * (M + log2f(lsum));
        }
    }
    if (nan_row) {
#pragma unroll
        for (int j = 0; j < DPL; ++j) o[j] = __int_as_float(0x7fc00000);
        lse = __int_as_float(0x7fc00000);
    }
    const int64_t off = (int64_t)row * D + lane * DPL;
    if (p.out_bf16) {
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out) + off;
        if (DPL == 4) {
            uint2 v;
            v.x = pack_bf16(o[0], o[1]);
            v.y = pack_bf16(o[2], o[3]);
            *reinterpret_cast<uint2 *>(out) = v;
        } else {
            *reinterpret_cast<uint32_t *>(out) = pack_bf16(o[0], o[1]);
        }
    } else {
        float *out = static_cast<float *>(p.out) + off;
        if (DPL == 4) *reinterpret_cast<float4 *>(out) = make_float4(o[0], o[1], o[2], o[3]);
        else *reinterpret_cast<float2 *>(out) = make_float2(o[0], o[1]);
    }
    if (p.lse && lane == 0) p.lse[row] = lse;
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream) {
    const int64_t rows = (int64_t)p.B * p.Hq * p.q_len;
    if (rows >= INT32_MAX) return cudaErrorInvalidValue;  // make_plan refuses these
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + kRowsPerCta - 1) / kRowsPerCta), 1, 1);
    cfg.blockDim = dim3(kRowsPerCta * 32, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return p.D == 128 ? cudaLaunchKernelEx(&cfg, merge_kernel<128>, p)
                      : cudaLaunchKernelEx(&cfg, merge_kernel<64>, p);
}

}  // namespace atlas
