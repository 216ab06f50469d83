// tc_order.cuh -- the longest-first order of split-KV work items shared by the
// tensor-core kernels (bf16 and fp32) in split mode.
//
// Each sequence's context is cut into equal splits (balanced_split in internal.h)
// instead of fixed-size chunks with a ragged last one, and the CTAs take the
// (sequence, split, kv head, query tile) items in order of decreasing split size,
// so that the long items start first and the last wave holds only short ones.  The
// order is a pure function of seq_lens and the call's sizes; every CTA derives it
// from seq_lens itself (no host round trip, no extra launch).
#pragma once

#include "internal.h"

namespace atlas {

struct TcItem {
    int b, hkv, tile, split, split_keys;  // b < 0: no item for this CTA
};

// All threads of the CTA call this (it synchronises the CTA).  `scratch` is shared
// memory for 4 * B + 4 ints that nothing else uses yet.  Requires B <= kTcOrderMaxSeqs.
__device__ inline TcItem tc_balanced_item(const TcParams &p, int item, int *scratch) {
    int *csz = scratch;           // [B] keys per split
    int *cnt = csz + p.B;         // [B] work items of the sequence
    int *rank = cnt + p.B;        // [B] position in the longest-first order
    int *found = rank + p.B;      // [4] the item's (b, index within its sequence)
    const int per_split = p.Hkv * p.tiles_per_unit;
    const int max_ctx = p.max_pages * p.P;
    if (threadIdx.x == 0) found[0] = -1;
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
        const int L = min(max(p.seq_lens[i], 1), max_ctx);
        const int keys = balanced_split(L, p.chunk);
        csz[i] = keys;
        cnt[i] = ((L + keys - 1) / keys) * per_split;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
        const int ci = csz[i];
        int r = 0;
        for (int k = 0; k < p.B; ++k) r += (csz[k] > ci) || (csz[k] == ci && k < i);
        rank[i] = r;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
        const int ri = rank[i];
        int start = 0;
        for (int k = 0; k < p.B; ++k) start += rank[k] < ri ? cnt[k] : 0;
        if (item >= start && item < start + cnt[i]) {
            found[0] = i;
            found[1] = item - start;
        }
    }
    __syncthreads();
    TcItem it{};
    it.b = found[0];
    if (it.b < 0) return it;
    const int li = found[1];
    it.split = li / per_split;
    const int rest = li % per_split;
    it.hkv = rest / p.tiles_per_unit;
    it.tile = rest % p.tiles_per_unit;
    it.split_keys = csz[it.b];
    __syncthreads();  // the scratch may be reused after this
    return it;
}

}  // namespace atlas
