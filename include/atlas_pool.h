/*
 * atlas_pool.h -- a bounded device pool of K/V pages fed from a host tier.
 *
 * The GPU form of CFR-Atlas's resident-memory bound (CFR-Atlas README,
 * introduction and "What CFR-Atlas is": historical K/V is a virtual address
 * space; selected pages stay in a byte-bounded hot cache, cold pages are brought
 * into reusable scratch buffers and folded into the online softmax one after
 * another; cache admission changes latency and residency, never the result).
 * Here the page contents come from a host tier (pinned host memory, read by the
 * GPU over NVLink-C2C on a Grace system) that stands in for CFR-Atlas's
 * regenerator; nothing here recomputes K/V.
 *
 * Device side: one pool of hot_slots + scratch_slots pages in the layout of the
 * attention pools, [slot][n_kv_heads][page_tokens][head_dim] for K and for V.
 * Slots 0 .. hot_slots-1 form the hot cache (kept across calls), slots
 * hot_slots .. hot_slots+scratch_slots-1 the scratch (reused pass by pass).
 * Host tier: [host_pages][n_kv_heads][page_tokens][head_dim] for K and V, the
 * same element type.  A page is named by its host-tier index.
 *
 * A decode call over the pool (one query row per sequence, as the CFR-Atlas
 * attention request is: a query over context_tokens of history) goes:
 *   1. atlas_pool_plan: the host-side planner decides, for every page of every
 *      split-KV chunk of the call, the slot it is read from, which pages are
 *      copied in (and where), and groups the chunks into passes so that each
 *      pass needs at most scratch_slots scratch pages.  Nothing is launched.
 *   2. for each pass k: atlas_pool_pass gives its page table (device slots),
 *      chunk range and copy list; atlas_pool_fill copies the listed pages from
 *      the host tier; atlas_attn_decode with ATLAS_PHASE_CHUNKS and that chunk
 *      range computes the pass's chunks into the call's workspace.
 *   3. atlas_attn_decode with ATLAS_PHASE_MERGE writes out / lse.
 * Every chunk's partial state depends only on its keys, so the output is bit for
 * bit that of one atlas_attn_decode over a fully resident pool with the same
 * sizes, whatever the pool held before the call.
 *
 * Policy (the pages name KeepRecent { recent_tokens } and an
 * admit_regenerated_pages switch without defining them; the plainest reading):
 *  - a page is "recent" for sequence b when it holds one of the last
 *    keep_recent_tokens positions of b (keep_recent_tokens < 0: every page is
 *    recent; 0: none is);
 *  - a page already in a hot slot is read from there (a hit), recent or not;
 *  - a page that is not hot, is recent, and admit != 0 is admitted: copied into
 *    a free hot slot, else into the slot of the least recently used hot page
 *    that this call does not read (ties: the lower slot), which is evicted; if
 *    every hot slot holds a page this call reads, it goes to scratch instead;
 *  - every other page is copied into a scratch slot for the pass that reads it
 *    (again in a later pass if a later pass reads it too).
 * "Used" means read by a call; the recency clock advances once per plan.
 *
 * Transactions: atlas_pool_plan either succeeds and commits the new residency,
 * or fails and leaves the pool as it was.  The caller must run the planned
 * copies before the pool is planned again (the residency assumes they ran).  A
 * host-tier page rewritten after it was copied in must be dropped with
 * atlas_pool_invalidate before the next plan.
 *
 * Threading: one pool object is not safe for concurrent use; separate objects
 * are independent.  The planner is host code and touches no CUDA state.
 */
#ifndef ATLAS_POOL_H
#define ATLAS_POOL_H

#include <stddef.h>
#include <stdint.h>

#include "atlas_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct atlas_pool atlas_pool; /* opaque planner state (host memory only) */

typedef struct {
    int32_t hot_slots;     /* >= 0: pages the hot cache holds (its byte budget / page bytes) */
    int32_t scratch_slots; /* >= 1: pages one pass may copy in besides the hot ones */
    int32_t page_tokens;   /* P, as in the attention calls */
    int32_t host_pages;    /* >= 1: pages in the host tier */
} atlas_pool_config;

typedef struct {
    int32_t batch;                  /* B >= 1 */
    int32_t max_pages_per_seq;      /* row length of host_page_table */
    const int32_t *host_page_table; /* host [batch][max_pages_per_seq]: the host-tier page
                                       of each logical page (entries past a sequence's last
                                       page are ignored) */
    const int32_t *seq_lens;        /* host [batch]: 1 <= seq_lens[b] <= max_pages*P */
    int32_t chunk_tokens;           /* >= 1: the decode call's split size
                                       (atlas_attn_split_tokens with the same sizes) */
    int32_t keep_recent_tokens;     /* KeepRecent window; < 0: every page, 0: none */
    int32_t admit;                  /* 0: pages that are not hot never become hot */
} atlas_pool_request;

typedef struct {
    int32_t passes;       /* launches of ATLAS_PHASE_CHUNKS the call needs */
    int64_t pages;        /* distinct host pages the call reads */
    int64_t hits;         /* of those, hot before the call */
    int64_t admitted;     /* copied into the hot cache by this call */
    int64_t evicted;      /* hot pages the admissions displaced */
    int64_t scratch_loads;/* scratch copies over all passes (a page may count twice) */
    int64_t copies;       /* admitted + scratch_loads: pages atlas_pool_fill moves */
} atlas_pool_stats;

/* Creates a planner with an empty hot cache.  Returns INVALID_ARG for a bad
 * configuration (page_tokens a power of two in [8, 128] as for attention). */
atlas_status atlas_pool_create(const atlas_pool_config *cfg, atlas_pool **pool);
void atlas_pool_destroy(atlas_pool *pool);

/* Plans one decode call (see above); *stats may be NULL.  INVALID_ARG for a bad
 * request: a seq_len out of range, a host page id outside [0, host_pages), or a
 * chunk whose pages cannot fit in scratch_slots even alone (scratch_slots must
 * be at least ceil(chunk_tokens / page_tokens) + 1).  The pool is then
 * unchanged. */
atlas_status atlas_pool_plan(atlas_pool *pool, const atlas_pool_request *req,
                             atlas_pool_stats *stats);

/* Pass k (0 <= k < stats.passes) of the last successful plan, into host arrays:
 *   page_table  [batch][max_pages_per_seq] device slots (entries the pass does not
 *               read are 0);
 *   chunk_range [batch][2] chunks [lo, hi) of each sequence the pass computes;
 *   copies      [n][2] (host page, device slot) pairs, *n_copies of them;
 *               max_copies >= hot_slots + scratch_slots always suffices.
 * INVALID_ARG if k is out of range or max_copies is too small. */
atlas_status atlas_pool_pass(const atlas_pool *pool, int32_t k, int32_t *page_table,
                             int32_t *chunk_range, int32_t *copies, int32_t max_copies,
                             int32_t *n_copies);

/* The hot slot holding host page `host_page`, or -1. */
int32_t atlas_pool_slot_of(const atlas_pool *pool, int32_t host_page);

/* Drops host page `host_page` from the hot cache (its contents changed). */
void atlas_pool_invalidate(atlas_pool *pool, int32_t host_page);

/*
 * atlas_pool_fill: for i < n_copies, copies host-tier page copies[i][0] of K and
 * of V (page_bytes each) into device slot copies[i][1] of k_slots / v_slots:
 *   k_slots[copies[i][1]] = host_k[copies[i][0]]   (and v), page_bytes bytes.
 * host_k / host_v: the host tier, page-locked host memory (cudaHostAlloc or
 * cudaHostRegister, read by the kernel in place) or device memory; pageable
 * memory is refused (INVALID_ARG).  k_slots / v_slots: device, dev_slots pages.
 * copies: device int32 [n_copies][2], read only.  page_bytes a multiple of 16 and
 * all four bases 16-byte aligned.  A pair outside [0, host_pages) x [0, dev_slots)
 * sets ATLAS_DEV_BAD_PAGE in *status_word (if given) and is skipped.  Enqueued on
 * `stream`; no host sync.
 */
atlas_status atlas_pool_fill(const void *host_k, const void *host_v, void *k_slots,
                             void *v_slots, const int32_t *copies, int32_t n_copies,
                             int64_t page_bytes, int32_t host_pages, int32_t dev_slots,
                             uint32_t *status_word, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ATLAS_POOL_H */
