// kv_append.cu -- the write before the attention: the new tokens' K and V rows of
// each sequence go to the page slots of positions seq_lens[b] .. seq_lens[b] +
// n_new[b] - 1, found through the page table (CFR-Atlas README, "Minimal
// integration": row-major K[token][dim] per (layer, kv head, token range);
// ferrox-core "cache" module: a KV cache grown one position at a time).
//
// A grid-stride loop moves 16 bytes of K and 16 bytes of V per thread and step;
// consecutive threads cover consecutive 16-byte pieces of a row, so both the
// reads of the new rows and the writes into a page slot are coalesced.  Memory
// bound: 2 x (read + write) x rows x head_dim x element size.
#include "internal.h"
#include "ptx.cuh"

namespace atlas {
namespace {

// Index arithmetic in I (32-bit while the piece count allows: a 64-bit division is
// a long instruction sequence); kUnroll pieces per thread are loaded before any is
// stored, so each thread keeps several independent reads in flight.
constexpr int kUnroll = 4;

template <typename I>
__global__ void __launch_bounds__(256) kv_append_kernel(const AppendParams p) {
    const I vec = (I)(p.row_bytes / 16);  // 16-byte pieces per row: 8, 16 or 32
    const int lvec = 31 - __clz((int)vec);
    const int lp = 31 - __clz(p.P);       // page_tokens is a power of two
    const I total = (I)p.B * (I)p.Hkv * (I)p.max_new * vec;
    const I stride = (I)gridDim.x * (I)blockDim.x;
    const char *kn = static_cast<const char *>(p.k_new);
    const char *vn = static_cast<const char *>(p.v_new);
    char *kp = static_cast<char *>(p.k_pages);
    char *vp = static_cast<char *>(p.v_pages);
    for (I base = (I)blockIdx.x * (I)blockDim.x + (I)threadIdx.x; base < total;
         base += stride * kUnroll) {
        uint4 kd[kUnroll], vd[kUnroll];
        int64_t dst[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            dst[u] = -1;
            const I idx = base + (I)u * stride;
            if (idx >= total) continue;
            const int piece = (int)(idx & (vec - 1));
            const I row = idx >> lvec;  // (b, g, j)
            const int j = (int)(row % (I)p.max_new);
            const I bg = row / (I)p.max_new;
            const int g = (int)(bg % (I)p.Hkv);
            const int b = (int)(bg / (I)p.Hkv);
            const int cnt = p.n_new ? p.n_new[b] : p.max_new;
            if (cnt < 0 || cnt > p.max_new) {
                if (j == 0 && g == 0 && piece == 0 && p.status)
                    atomicOr(p.status, ATLAS_DEV_BAD_SEQLEN);
                continue;
            }
            if (j >= cnt) continue;
            const int64_t t = (int64_t)p.seq_lens[b] + j;
            if (t < 0 || t >= (int64_t)p.max_pages * p.P) {
                if (p.status && piece == 0) atomicOr(p.status, ATLAS_DEV_BAD_SEQLEN);
                continue;
            }
            const int page = p.page_table[(int64_t)b * p.max_pages + (t >> lp)];
            if (page < 0 || page >= p.num_pages) {
                if (p.status && piece == 0) atomicOr(p.status, ATLAS_DEV_BAD_PAGE);
                continue;
            }
            const int64_t src = (int64_t)row * p.row_bytes + piece * 16;
            dst[u] = (((int64_t)page * p.Hkv + g) * p.P + (t & (p.P - 1))) * p.row_bytes +
                     piece * 16;
            kd[u] = *reinterpret_cast<const uint4 *>(kn + src);
            vd[u] = *reinterpret_cast<const uint4 *>(vn + src);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (dst[u] < 0) continue;
            *reinterpret_cast<uint4 *>(kp + dst[u]) = kd[u];
            *reinterpret_cast<uint4 *>(vp + dst[u]) = vd[u];
        }
    }
}

}  // namespace

cudaError_t launch_kv_append(const AppendParams &p, cudaStream_t stream) {
    const int64_t total = (int64_t)p.B * p.Hkv * p.max_new * (p.row_bytes / 16);
    int64_t blocks = (total + 255) / 256;
    // a grid-stride loop over 16 CTAs of 256 threads per SM
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    // 32-bit indices while every index of the loop (up to total + a stride) fits
    if (total + (int64_t)blocks * 256 * kUnroll < INT32_MAX)
        kv_append_kernel<int32_t><<<(unsigned)blocks, 256, 0, stream>>>(p);
    else
        kv_append_kernel<int64_t><<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace atlas
