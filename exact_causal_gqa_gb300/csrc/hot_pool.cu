// hot_pool.cu -- the bounded hot-page pool: a host-side planner that decides
// which K/V pages sit in which device slot for a decode call, and the kernel that
// copies pages in from the host tier (CFR-Atlas README, introduction: a
// byte-bounded hot cache, reusable scratch buffers for cold pages, each page
// folded into the online softmax; admission changes residency, not the result).
// The semantics are stated in include/atlas_pool.h.
#include <algorithm>
#include <new>
#include <vector>

#include "atlas_pool.h"
#include "internal.h"

struct atlas_pool {
    atlas_pool_config cfg;
    std::vector<int32_t> slot_page;  // [hot_slots] host page in the slot, -1 if free
    std::vector<int64_t> slot_used;  // [hot_slots] plan number of its last use, 0 never
    std::vector<int32_t> where;      // [host_pages] hot slot holding the page, -1 if none
    std::vector<int64_t> seen;       // [host_pages] plan number that last counted the page
    std::vector<int64_t> scr_pass;   // [host_pages] pass serial that put it in scratch
    std::vector<int32_t> scr_slot;   // [host_pages] its scratch slot in that pass
    int64_t clock = 0;               // plans so far
    int64_t pass_serial = 0;         // passes so far, over all plans
    // the last successful plan
    int32_t batch = 0, max_pages = 0;
    struct Pass {
        std::vector<int32_t> table, range, copies;
    };
    std::vector<Pass> passes;
};

namespace {

bool pow2(int32_t x) { return x > 0 && (x & (x - 1)) == 0; }

// Pages of chunk c of a sequence of L keys: logical pages [p0, p1].
void chunk_pages(int64_t c, int64_t chunk, int64_t L, int64_t P, int64_t &p0, int64_t &p1) {
    const int64_t t0 = c * chunk, t1 = std::min(t0 + chunk, L);
    p0 = t0 / P;
    p1 = (t1 - 1) / P;
}

}  // namespace

extern "C" {

atlas_status atlas_pool_create(const atlas_pool_config *cfg, atlas_pool **pool) {
    if (!cfg || !pool) return ATLAS_ERR_INVALID_ARG;
    *pool = nullptr;
    if (cfg->hot_slots < 0 || cfg->scratch_slots < 1 || cfg->host_pages < 1 ||
        !pow2(cfg->page_tokens) || cfg->page_tokens < 8 || cfg->page_tokens > 128 ||
        (int64_t)cfg->hot_slots + cfg->scratch_slots > INT32_MAX / 2)
        return ATLAS_ERR_INVALID_ARG;
    atlas_pool *p = new (std::nothrow) atlas_pool;
    if (!p) return ATLAS_ERR_INVALID_ARG;
    try {
        p->cfg = *cfg;
        p->slot_page.assign(cfg->hot_slots, -1);
        p->slot_used.assign(cfg->hot_slots, 0);
        p->where.assign(cfg->host_pages, -1);
        p->seen.assign(cfg->host_pages, 0);
        p->scr_pass.assign(cfg->host_pages, 0);
        p->scr_slot.assign(cfg->host_pages, 0);
    } catch (...) {
        delete p;
        return ATLAS_ERR_INVALID_ARG;
    }
    *pool = p;
    return ATLAS_OK;
}

void atlas_pool_destroy(atlas_pool *pool) { delete pool; }

int32_t atlas_pool_slot_of(const atlas_pool *pool, int32_t host_page) {
    if (!pool || host_page < 0 || host_page >= pool->cfg.host_pages) return -1;
    return pool->where[host_page];
}

void atlas_pool_invalidate(atlas_pool *pool, int32_t host_page) {
    if (!pool || host_page < 0 || host_page >= pool->cfg.host_pages) return;
    const int32_t s = pool->where[host_page];
    if (s >= 0) {
        pool->slot_page[s] = -1;
        pool->slot_used[s] = 0;
        pool->where[host_page] = -1;
    }
}

atlas_status atlas_pool_plan(atlas_pool *pool, const atlas_pool_request *req,
                             atlas_pool_stats *stats) {
    if (!pool || !req || !req->host_page_table || !req->seq_lens) return ATLAS_ERR_INVALID_ARG;
    const int64_t B = req->batch, MP = req->max_pages_per_seq, chunk = req->chunk_tokens;
    const int64_t P = pool->cfg.page_tokens, H = pool->cfg.hot_slots,
                  C = pool->cfg.scratch_slots, NH = pool->cfg.host_pages;
    if (B < 1 || MP < 1 || chunk < 1 || B * MP > INT32_MAX) return ATLAS_ERR_INVALID_ARG;
    const int32_t *tab = req->host_page_table;
    // -- validation: after it only an allocation can fail
    for (int64_t b = 0; b < B; ++b) {
        const int64_t L = req->seq_lens[b];
        if (L < 1 || L > MP * P) return ATLAS_ERR_INVALID_ARG;
        const int64_t np = (L + P - 1) / P;
        for (int64_t j = 0; j < np; ++j) {
            const int32_t hp = tab[b * MP + j];
            if (hp < 0 || hp >= NH) return ATLAS_ERR_INVALID_ARG;
        }
        const int64_t nch = (L + chunk - 1) / chunk;
        for (int64_t c = 0; c < nch; ++c) {
            int64_t p0, p1;
            chunk_pages(c, chunk, L, P, p0, p1);
            if (p1 - p0 + 1 > C) return ATLAS_ERR_INVALID_ARG;
        }
    }
    std::vector<atlas_pool::Pass> passes;
    std::vector<int32_t> cand;  // hot slots this call does not read, best victim first
    std::vector<int32_t> journal;  // (slot, page it held) per admission, to undo on failure
    std::vector<char> pinned;
    try {
        cand.reserve((size_t)H);
        journal.reserve((size_t)(2 * H));
        pinned.assign((size_t)H, 0);
    } catch (...) {
        return ATLAS_ERR_INVALID_ARG;
    }
    const int64_t now = pool->clock + 1;
    atlas_pool_stats st{};
    // Only an allocation can fail from here on; the journal then restores the
    // hot-slot map (the per-page stamps carry no state between plans).
    try {
    // -- pages of the call: count them and pin the hot ones
    for (int64_t b = 0; b < B; ++b) {
        const int64_t np = (req->seq_lens[b] + P - 1) / P;
        for (int64_t j = 0; j < np; ++j) {
            const int32_t hp = tab[b * MP + j];
            if (pool->seen[hp] == now) continue;
            pool->seen[hp] = now;
            ++st.pages;
            if (pool->where[hp] >= 0) {
                ++st.hits;
                pinned[pool->where[hp]] = 1;
            }
        }
    }
    for (int32_t s = 0; s < H; ++s)
        if (!pinned[s]) cand.push_back(s);
    std::sort(cand.begin(), cand.end(), [pool](int32_t a, int32_t b) {
        const bool fa = pool->slot_page[a] < 0, fb = pool->slot_page[b] < 0;
        if (fa != fb) return fa;  // free slots first
        if (pool->slot_used[a] != pool->slot_used[b])
            return pool->slot_used[a] < pool->slot_used[b];
        return a < b;
    });
    size_t next_cand = 0;

    // -- passes: chunks in (sequence, chunk) order, each pass within C scratch pages
    auto new_pass = [&]() {
        passes.emplace_back();
        atlas_pool::Pass &ps = passes.back();
        ps.table.assign((size_t)(B * MP), 0);
        ps.range.assign((size_t)(2 * B), 0);
        ++pool->pass_serial;
    };
    new_pass();
    int64_t scratch_used = 0;
    bool pass_has_work = false;
    std::vector<int32_t> admit_copies, cold;  // per chunk
    for (int64_t b = 0; b < B; ++b) {
        const int64_t L = req->seq_lens[b];
        const int64_t nch = (L + chunk - 1) / chunk;
        const int64_t recent_from =
            req->keep_recent_tokens < 0 ? 0
            : req->keep_recent_tokens == 0 ? INT64_MAX
                                           : L - req->keep_recent_tokens;  // first recent key
        for (int64_t c = 0; c < nch; ++c) {
            int64_t p0, p1;
            chunk_pages(c, chunk, L, P, p0, p1);
            admit_copies.clear();
            cold.clear();
            for (int64_t j = p0; j <= p1; ++j) {
                const int32_t hp = tab[b * MP + j];
                if (pool->where[hp] >= 0) continue;  // hot
                // last key the page holds for this sequence
                const int64_t last = std::min((j + 1) * P, L) - 1;
                if (req->admit && last >= recent_from && next_cand < cand.size()) {
                    const int32_t s = cand[next_cand++];
                    const int32_t victim = pool->slot_page[s];
                    journal.push_back(s);
                    journal.push_back(victim);
                    if (victim >= 0) {
                        pool->where[victim] = -1;
                        ++st.evicted;
                    }
                    pool->slot_page[s] = hp;
                    pool->where[hp] = s;
                    pinned[s] = 1;
                    ++st.admitted;
                    admit_copies.push_back(hp);
                    admit_copies.push_back(s);
                    continue;
                }
                if (std::find(cold.begin(), cold.end(), hp) == cold.end()) cold.push_back(hp);
            }
            int64_t need = 0;
            for (int32_t hp : cold)
                if (pool->scr_pass[hp] != pool->pass_serial) ++need;
            if (scratch_used + need > C) {
                new_pass();
                scratch_used = 0;
                pass_has_work = false;
            }
            atlas_pool::Pass &ps = passes.back();
            for (int32_t hp : cold) {
                if (pool->scr_pass[hp] == pool->pass_serial) continue;
                pool->scr_pass[hp] = pool->pass_serial;
                pool->scr_slot[hp] = (int32_t)(H + scratch_used++);
                ps.copies.push_back(hp);
                ps.copies.push_back(pool->scr_slot[hp]);
                ++st.scratch_loads;
            }
            ps.copies.insert(ps.copies.end(), admit_copies.begin(), admit_copies.end());
            for (int64_t j = p0; j <= p1; ++j) {
                const int32_t hp = tab[b * MP + j];
                ps.table[b * MP + j] = pool->where[hp] >= 0 ? pool->where[hp] : pool->scr_slot[hp];
            }
            if (ps.range[2 * b] == ps.range[2 * b + 1]) ps.range[2 * b] = (int32_t)c;
            ps.range[2 * b + 1] = (int32_t)(c + 1);
            pass_has_work = true;
        }
    }
    if (!pass_has_work && passes.size() > 1) passes.pop_back();
    } catch (...) {
        for (size_t k = journal.size(); k >= 2; k -= 2) {
            const int32_t s = journal[k - 2], old_page = journal[k - 1];
            pool->where[pool->slot_page[s]] = -1;
            pool->slot_page[s] = old_page;
            if (old_page >= 0) pool->where[old_page] = s;
        }
        pool->clock = now;  // retires this plan's page stamps (LRU order is unaffected)
        return ATLAS_ERR_INVALID_ARG;
    }
    // -- commit
    for (int64_t s = 0; s < H; ++s)
        if (pinned[s]) pool->slot_used[s] = now;
    pool->clock = now;
    pool->batch = (int32_t)B;
    pool->max_pages = (int32_t)MP;
    pool->passes.swap(passes);
    st.passes = (int32_t)pool->passes.size();
    st.copies = st.admitted + st.scratch_loads;
    if (stats) *stats = st;
    return ATLAS_OK;
}

atlas_status atlas_pool_pass(const atlas_pool *pool, int32_t k, int32_t *page_table,
                             int32_t *chunk_range, int32_t *copies, int32_t max_copies,
                             int32_t *n_copies) {
    if (!pool || k < 0 || k >= (int32_t)pool->passes.size()) return ATLAS_ERR_INVALID_ARG;
    const atlas_pool::Pass &ps = pool->passes[k];
    const int32_t n = (int32_t)(ps.copies.size() / 2);
    if (n > max_copies || (n > 0 && !copies)) return ATLAS_ERR_INVALID_ARG;
    if (page_table) std::copy(ps.table.begin(), ps.table.end(), page_table);
    if (chunk_range) std::copy(ps.range.begin(), ps.range.end(), chunk_range);
    if (copies) std::copy(ps.copies.begin(), ps.copies.end(), copies);
    if (n_copies) *n_copies = n;
    return ATLAS_OK;
}

}  // extern "C"

namespace atlas {
namespace {

constexpr int kFillThreads = 256;
constexpr int kFillUnroll = 4;  // 16-byte loads in flight per thread: host reads are far

// One CTA per (copy, K or V): a page of page_vec 16-byte words.
__global__ void __launch_bounds__(kFillThreads)
pool_fill_kernel(const uint4 *hk, const uint4 *hv, uint4 *dk, uint4 *dv, const int32_t *copies,
                 int64_t page_vec, int32_t host_pages, int32_t dev_slots, uint32_t *status) {
    const int64_t i = blockIdx.x;
    const int32_t src = copies[2 * i], dst = copies[2 * i + 1];
    if (src < 0 || src >= host_pages || dst < 0 || dst >= dev_slots) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && status) atomicOr(status, ATLAS_DEV_BAD_PAGE);
        return;
    }
    const uint4 *s = (blockIdx.y ? hv : hk) + (int64_t)src * page_vec;
    uint4 *d = (blockIdx.y ? dv : dk) + (int64_t)dst * page_vec;
    for (int64_t k0 = threadIdx.x; k0 < page_vec; k0 += (int64_t)kFillThreads * kFillUnroll) {
        uint4 r[kFillUnroll];
#pragma unroll
        for (int u = 0; u < kFillUnroll; ++u) {
            const int64_t k = k0 + (int64_t)u * kFillThreads;
            if (k < page_vec) r[u] = s[k];
        }
#pragma unroll
        for (int u = 0; u < kFillUnroll; ++u) {
            const int64_t k = k0 + (int64_t)u * kFillThreads;
            if (k < page_vec) d[k] = r[u];
        }
    }
}

// Device address of a host-tier base: page-locked host memory maps into the
// device address space; device and managed memory are used as they are.
bool device_view(const void *p, const void **out) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeHost) {
        *out = a.devicePointer;
        return *out != nullptr;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
        *out = p;
        return true;
    }
    return false;  // pageable host memory: not read from a kernel here
}

}  // namespace
}  // namespace atlas

extern "C" atlas_status atlas_pool_fill(const void *host_k, const void *host_v, void *k_slots,
                                        void *v_slots, const int32_t *copies, int32_t n_copies,
                                        int64_t page_bytes, int32_t host_pages,
                                        int32_t dev_slots, uint32_t *status_word,
                                        void *stream) {
    if (!host_k || !host_v || !k_slots || !v_slots || n_copies < 0 || page_bytes < 16 ||
        page_bytes % 16 != 0 || host_pages < 1 || dev_slots < 1)
        return ATLAS_ERR_INVALID_ARG;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(host_k) | reinterpret_cast<uintptr_t>(host_v) |
                          reinterpret_cast<uintptr_t>(k_slots) | reinterpret_cast<uintptr_t>(v_slots);
    if (mis & 15u) return ATLAS_ERR_INVALID_ARG;
    if (n_copies == 0) return ATLAS_OK;
    if (!copies) return ATLAS_ERR_INVALID_ARG;
    const void *dk_src = nullptr, *dv_src = nullptr;
    if (!atlas::device_view(host_k, &dk_src) || !atlas::device_view(host_v, &dv_src))
        return ATLAS_ERR_INVALID_ARG;
    (void)cudaGetLastError();
    const dim3 grid((unsigned)n_copies, 2, 1);
    atlas::pool_fill_kernel<<<grid, atlas::kFillThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(dk_src), static_cast<const uint4 *>(dv_src),
        static_cast<uint4 *>(k_slots), static_cast<uint4 *>(v_slots), copies, page_bytes / 16,
        host_pages, dev_slots, status_word);
    return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}
