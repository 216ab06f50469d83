/*
 * atlas_attn.h -- exact causal grouped-query softmax attention over paged K/V,
 * on one GB300 (sm_103a).
 *
 * What every entry point computes.  For each sequence b, query head h and query
 * row i in [0, q_len):
 *
 *   kv head      g = h / (n_q_heads / n_kv_heads)       (contiguous GQA groups)
 *   position     pos = seq_lens[b] - q_len + i          (the queries are the last
 *                                                        q_len positions of K/V)
 *   key t        k_t = k_pages[page_table[b][t / page_tokens]][g][t % page_tokens][:]
 *   out[b][h][i] = sum_{t <= pos} exp(s_t - M) v_t / sum_{t <= pos} exp(s_t - M),
 *                  s_t = scale * <q[b][h][i], k_t>,  M = max_t s_t
 *   lse[b][h][i] = M + ln sum_{t <= pos} exp(s_t - M)     (natural log)
 *
 * with the optional variants of atlas_launch: a window keeps only keys
 * t > pos - window, a softcap c replaces s_t by c tanh(s_t / c), and a sink
 * logit adds exp(sink[h] - M) to both denominators (M then covers it too).
 *
 * Sources (page title, section):
 *   CFR-Atlas README, "Core contract": folding exact pages into an online-softmax
 *     state gives the full-KV result, which is what is computed here;
 *   CFR-Atlas README, "Minimal integration": row-major K[token][dim], V[token][dim]
 *     pages per (layer, K/V head, token range) -> the page pools below;
 *   CPUAttn README, "Parallel example" and "Operator model": queries are the
 *     suffix of K/V (positions start at SKV - SQ); decode is the same pattern
 *     with one query row; split-K is combined by a structured merge;
 *   ferrox-core crate index: causal_gqa_attention_paged (decode) and
 *     causal_gqa_attention_prefill (prefill) name the two ends of this family.
 *
 * Layouts (all dense, row-major, C order; every pointer 16-byte aligned):
 *   q, out        [batch][n_q_heads][q_len][head_dim]
 *   k_pages,
 *   v_pages       [num_pages][n_kv_heads][page_tokens][head_dim]
 *   page_table    int32 [batch][max_pages_per_seq]; entries past a sequence's
 *                 last page are never read
 *   seq_lens      int32 [batch]; keys visible to the last query row
 *   lse           float [batch][n_q_heads][q_len]
 *
 * Ownership and asynchrony.  Every tensor pointer is a DEVICE pointer owned by
 * the caller; q, pools, page_table and seq_lens are only read.  The library
 * allocates no device memory and keeps no per-call state (it caches a driver
 * entry point and per-device kernel attributes).  All work is enqueued on
 * `stream`; no call synchronises with the host.
 *
 * Supported: head_dim 64 or 128; page_tokens a power of two in [8, 128];
 *   n_q_heads a multiple of n_kv_heads;
 *   q/K/V float32 -> out float32, or q/K/V bfloat16 -> out bfloat16 or float32.
 *   Accumulation and softmax state are float32 in every mode.
 *
 * Errors.  Host-side checks return a status before anything is enqueued.
 * Data-dependent problems are found on the device: a page id outside
 * [0, num_pages), a seq_len below q_len or above max_pages_per_seq*page_tokens,
 * or a bounded wait that ran out each OR a bit (ATLAS_DEV_*) into *status_word
 * (when given) and leave the affected output rows NaN.  The caller reads the
 * word after synchronising the stream.  Non-finite inputs are not scanned for;
 * they propagate into the rows that see them.
 */
#ifndef ATLAS_ATTN_H
#define ATLAS_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATLAS_OK = 0,
    ATLAS_ERR_INVALID_ARG = 1, /* null pointer, bad shape, misalignment, GQA ratio */
    ATLAS_ERR_UNSUPPORTED = 2, /* head_dim / page_tokens / dtype not supported */
    ATLAS_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
    ATLAS_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed */
    ATLAS_ERR_DEVICE = 5       /* reserved for callers: a status word bit was set */
} atlas_status;

typedef enum { ATLAS_F32 = 0, ATLAS_BF16 = 1 } atlas_dtype;

typedef enum { ATLAS_KIND_DECODE = 0, ATLAS_KIND_SUFFIX = 1, ATLAS_KIND_PREFILL = 2 } atlas_kind;

/* Bits the kernels OR into *status_word. */
#define ATLAS_DEV_BAD_PAGE 1u    /* a page id outside [0, num_pages) */
#define ATLAS_DEV_BAD_SEQLEN 2u  /* seq_len < q_len or > max_pages_per_seq * page_tokens */
#define ATLAS_DEV_TIMEOUT 4u     /* a bounded wait inside a kernel ran out */

/* Test-only: make the decode producer withhold one stage so that the consumers'
 * bounded wait runs out and ATLAS_DEV_TIMEOUT is reported. */
#define ATLAS_DEBUG_WITHHOLD_STAGE 1u
/* Test-only: the tensor-core path writes the output directly (no split-KV), even
 * when the call has few query tiles. */
#define ATLAS_DEBUG_TC_DIRECT 2u

/* Everything a call needs beyond the (q, k_pages, v_pages, page_table,
 * seq_lens, n_q_heads, n_kv_heads, head_dim, page_tokens, scale) list. */
typedef struct {
    int32_t batch;             /* B >= 1 */
    int32_t max_pages_per_seq; /* page_table row length */
    int32_t num_pages;         /* pages in each pool */
    int32_t q_len;             /* 1 for decode, SQ for suffix, S for prefill;
                                  batch * n_q_heads * q_len < 2^31 - 1 */
    atlas_dtype q_dtype;       /* must equal kv_dtype */
    atlas_dtype kv_dtype;
    atlas_dtype out_dtype;
    void *out;                 /* [B][Hq][q_len][D] of out_dtype; written */
    float *lse;                /* optional [B][Hq][q_len]; NULL to skip */
    void *workspace;           /* device scratch, >= atlas_attn_workspace_size() bytes */
    size_t workspace_bytes;
    uint32_t *status_word;     /* optional device word; bits OR-ed, never cleared */
    void *stream;              /* cudaStream_t; NULL = the legacy default stream */
    int32_t split_tokens;      /* keys per split-KV chunk; 0 = automatic; else a
                                  multiple of 64 */
    uint32_t debug_flags;      /* 0 in production; ATLAS_DEBUG_* for tests */
    void *const *events;       /* optional host array of 3 cudaEvent_t, recorded on
                                  `stream` before the main kernel, between it and the
                                  merge, and after the merge (profiling); NULL = none */
    /* Score / mask variants (ferrox-core: causal_gqa_attention_windowed, _softcap,
     * _sinks).  All zero / NULL gives plain causal attention. */
    int32_t window;            /* > 0: row i sees only keys pos - window < t <= pos */
    float softcap;             /* > 0: each scaled score s becomes softcap*tanh(s/softcap) */
    const float *sinks;        /* optional device [n_q_heads]: a logit per q head that joins
                                  the softmax denominator (natural-log units, like the
                                  scaled scores) with no value row; lse includes it */
    const int32_t *q_lens;     /* optional device [batch]: ragged query counts (chunked
                                  prefill).  Sequence b has q_lens[b] <= q_len query rows,
                                  the last q_lens[b] positions of its K/V: row i sits at
                                  seq_lens[b] - q_lens[b] + i.  Rows i >= q_lens[b] of q
                                  are ignored and of out / lse are not written.  NULL:
                                  every sequence has q_len rows.  Prefill then needs
                                  seq_lens[b] == q_lens[b]. */
    /* One call computed over several launches (the bounded hot-page pool of
     * atlas_pool.h serves a context larger than its device slots this way): the
     * split-KV chunks go to the same workspace pass by pass, then one merge reads
     * them all.  Each chunk's partial state depends only on its keys, so the
     * result is bit-identical to a single launch with the same sizes and split_tokens. */
    const int32_t *chunk_range; /* optional device [batch][2]: compute only chunks s with
                                   chunk_range[b][0] <= s < chunk_range[b][1] of sequence b
                                   (chunks of atlas_attn_split_tokens keys, from key 0);
                                   NULL = every chunk.  Only page_table entries of those
                                   chunks' pages are read. */
    int32_t phase;             /* ATLAS_PHASE_ALL, _CHUNKS or _MERGE (below) */
    int32_t sm_count;          /* SMs the automatic split plan fills; 0 = the multiprocessor
                                  count of the current device (cached per device), or 152
                                  (one GB300) when no device is visible, e.g. when sizing a
                                  workspace on a host without a GPU.  A caller confined to
                                  part of the GPU (a green context, an MPS share) passes its
                                  own count.  The plan, and so the workspace size and the
                                  bits of the result, is a pure function of the call's sizes
                                  and this count. */
} atlas_launch;

/* atlas_launch.phase.  With a phase other than ALL the call always takes the
 * split-KV form (the tensor-core path never writes its output directly). */
#define ATLAS_PHASE_ALL 0    /* chunks, then the merge into out / lse */
#define ATLAS_PHASE_CHUNKS 1 /* chunks only: partial states to the workspace */
#define ATLAS_PHASE_MERGE 2  /* merge only: every chunk must have been computed by
                                earlier ATLAS_PHASE_CHUNKS launches of the same sizes
                                into this workspace, on this stream */

/*
 * atlas_attn_decode: one query row per sequence (L->q_len must be 1), the
 * decode step over a paged cache (ferrox-core "causal_gqa_attention_paged";
 * CPUAttn "Operator model": decode is kv_cache=True with one query row).
 * Split-KV over the page stream, then a log-sum-exp merge.
 */
atlas_status atlas_attn_decode(const void *q, const void *k_pages, const void *v_pages,
                               const int32_t *page_table, const int32_t *seq_lens,
                               int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                               int32_t page_tokens, float scale, const atlas_launch *L);

/*
 * atlas_attn_suffix: L->q_len query rows per sequence that are the last q_len
 * positions of its K/V (CPUAttn README, "Parallel example": kv_cache=True,
 * positions start at SKV - SQ).  Row i sees keys 0 .. seq_len - q_len + i.
 */
atlas_status atlas_attn_suffix(const void *q, const void *k_pages, const void *v_pages,
                               const int32_t *page_table, const int32_t *seq_lens,
                               int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                               int32_t page_tokens, float scale, const atlas_launch *L);

/*
 * atlas_attn_prefill: causal self-attention of a whole prompt whose K/V were
 * written into pages (ferrox-core "causal_gqa_attention_prefill").  Every
 * seq_lens[b] must equal L->q_len; a sequence where it does not gets
 * ATLAS_DEV_BAD_SEQLEN and NaN rows.
 */
atlas_status atlas_attn_prefill(const void *q, const void *k_pages, const void *v_pages,
                                const int32_t *page_table, const int32_t *seq_lens,
                                int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                int32_t page_tokens, float scale, const atlas_launch *L);

/*
 * Bytes of device workspace the call of `kind` with these arguments needs (0 if
 * none).  Reads batch, max_pages_per_seq, q_len, the dtypes and split_tokens
 * from *L; ignores its pointers.  Returns SIZE_MAX if the arguments are invalid.
 */
size_t atlas_attn_workspace_size(atlas_kind kind, int32_t n_q_heads, int32_t n_kv_heads,
                                 int32_t head_dim, int32_t page_tokens, const atlas_launch *L);

/*
 * Keys per split-KV chunk of the call of `kind` with these arguments (the
 * chunks atlas_launch.chunk_range counts), 0 when the call has no chunks in
 * the workspace (the kernel writes its output itself: the tensor-core path with
 * many query tiles; a bf16 call with few query rows whose context per (sequence,
 * kv head) holds at most 256 KB of K/V; an fp32 call with few query rows whose
 * automatic plan has at most 8 splits, merged inside one thread-block cluster;
 * never with a phase other than ATLAS_PHASE_ALL, a chunk_range or a fixed
 * split_tokens), -1 if the arguments are invalid.  An automatic tensor-core plan
 * with ATLAS_PHASE_ALL cuts each sequence into equal splits of at most this many
 * keys (fewer for short sequences), taken longest-first.  Reads the same fields as
 * atlas_attn_workspace_size.
 */
int32_t atlas_attn_split_tokens(atlas_kind kind, int32_t n_q_heads, int32_t n_kv_heads,
                                int32_t head_dim, int32_t page_tokens, const atlas_launch *L);

/* Arguments of atlas_kv_append beyond its pointer / size list. */
typedef struct {
    int32_t batch;
    int32_t max_pages_per_seq;
    int32_t num_pages;
    int32_t max_new;           /* rows per sequence in k_new / v_new */
    atlas_dtype kv_dtype;      /* element type of k_new, v_new and the pools */
    uint32_t *status_word;     /* optional device word (ATLAS_DEV_* bits) */
    void *stream;              /* cudaStream_t; NULL = the legacy default stream */
} atlas_append;

/*
 * atlas_kv_append: the write before attention -- the paged KV cache grown by the
 * new tokens of each sequence (ferrox-core "cache" module: a KV cache growable one
 * position at a time; CFR-Atlas README, "Minimal integration": row-major
 * K[token][dim] per (layer, kv head, token range)).  For b < batch, kv head g and
 * j < n_new[b] (n_new NULL: all max_new rows):
 *   k_pages[page_table[b][t / page_tokens]][g][t % page_tokens][:] = k_new[b][g][j][:]
 *   (and v), with t = seq_lens[b] + j.
 * k_new, v_new: device [batch][n_kv_heads][max_new][head_dim], read only; the pools
 * are written in place; seq_lens (the lengths BEFORE the append) and n_new are
 * device int32 [batch], read only -- the caller advances seq_lens itself.  The
 * pages for the new positions must already be in page_table.  A page id outside
 * [0, num_pages) or a position past max_pages_per_seq * page_tokens sets
 * ATLAS_DEV_BAD_PAGE / ATLAS_DEV_BAD_SEQLEN and that row is skipped.
 */
atlas_status atlas_kv_append(const void *k_new, const void *v_new, void *k_pages, void *v_pages,
                             const int32_t *page_table, const int32_t *seq_lens,
                             const int32_t *n_new, int32_t n_kv_heads, int32_t head_dim,
                             int32_t page_tokens, const atlas_append *A);

/* Static, human-readable text for a status code. */
const char *atlas_attn_status_string(atlas_status status);

/* Size of the library-owned device scratch used by atlas_attn_decode_static_scratch. */
#define ATLAS_STATIC_SCRATCH_BYTES (16u << 20) /* 16 MiB per GPU that loads the library */

/*
 * atlas_attn_decode_static_scratch: atlas_attn_decode for callers that cannot
 * allocate device memory on the decode path (a host framework that owns all
 * device memory and forbids other allocations, or a serving loop where
 * cudaMalloc/cudaFree may synchronise the device).  The pages have no
 * counterpart to this entry point; it exists for such integrations.
 *
 * Same arguments and results as atlas_attn_decode, except that L->workspace and
 * L->workspace_bytes are ignored: the split-KV scratch lives in a fixed
 * ATLAS_STATIC_SCRATCH_BYTES array of device memory owned by the library (held
 * on every GPU that loads the library until the process exits).  The call
 * allocates nothing.  The caller still passes q, the pools, the page table,
 * seq_lens and the output (and optionally lse / status_word).
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.  Returns the status atlas_attn_decode would return for
 * invalid or unsupported arguments; ATLAS_ERR_UNSUPPORTED for L->phase other
 * than ATLAS_PHASE_ALL (the partials of a call spread over several launches
 * would sit in the shared array between launches); ATLAS_ERR_WORKSPACE when the
 * call would need more than ATLAS_STATIC_SCRATCH_BYTES of scratch
 * (atlas_attn_workspace_size with ATLAS_KIND_DECODE gives the need);
 * ATLAS_ERR_CUDA if the address lookup fails.  All calls on a device share the
 * array: calls whose kernels may overlap on the GPU (unordered streams) race on
 * it.  Nothing in it needs clearing between calls, since each call's merge reads
 * only partials its own split kernel wrote.
 */
atlas_status atlas_attn_decode_static_scratch(const void *q, const void *k_pages,
                                              const void *v_pages, const int32_t *page_table,
                                              const int32_t *seq_lens, int32_t n_q_heads,
                                              int32_t n_kv_heads, int32_t head_dim,
                                              int32_t page_tokens, float scale,
                                              const atlas_launch *L);

#ifdef __cplusplus
}
#endif

#endif /* ATLAS_ATTN_H */
