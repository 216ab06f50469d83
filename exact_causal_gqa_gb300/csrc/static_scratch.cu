// static_scratch.cu -- a decode entry point that allocates nothing.
//
// Who it is for: callers that cannot call cudaMalloc (or own a torch-style
// allocator) on the decode path -- for example a host framework that hands the
// library only the tensors it already owns and forbids any other device
// allocation, or a latency-critical serving loop where cudaMalloc / cudaFree may
// implicitly synchronise the device.  Such callers cannot provide the split-KV
// workspace that atlas_attn_decode needs, so this entry point keeps that scratch
// in a fixed array in device memory that belongs to the library.
//
// How: the split partials (m, l, acc per split) live in g_decode_scratch, a
// file-scope __device__ array of ATLAS_STATIC_SCRATCH_BYTES.  Every GPU that
// loads the library holds that array until the process exits.  Host code cannot
// use the array's name as a device address (on the host it names a stand-in),
// so the first call on each device looks up the real address with
// cudaGetSymbolAddress while that device is current, and later calls reuse it.
// The call then runs the ordinary decode path with that address as its
// workspace.
//
// Nothing in the array has to start at zero: every partial the merge reads is
// written by the split kernel of the same call.  That holds because the entry
// point accepts ATLAS_PHASE_ALL only: a call spread over several launches
// (ATLAS_PHASE_CHUNKS ... ATLAS_PHASE_MERGE) would leave its partials in the
// shared array between launches, where any other call could overwrite them, so
// such calls are refused.  The array is shared by all calls on a device and
// keeps the last call's contents, so two calls whose kernels overlap on the GPU
// (different streams, no ordering between them) race on it and may return wrong
// results.
#include "internal.h"

#include <cuda_runtime.h>

#include <mutex>

namespace atlas {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[ATLAS_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device (looked up once).
atlas_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return ATLAS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr)
            return ATLAS_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return ATLAS_OK;
}

}  // namespace
}  // namespace atlas

extern "C" atlas_status atlas_attn_decode_static_scratch(
    const void *q, const void *k_pages, const void *v_pages, const int32_t *page_table,
    const int32_t *seq_lens, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
    int32_t page_tokens, float scale, const atlas_launch *L) {
    if (!L) return ATLAS_ERR_INVALID_ARG;
    // The same plan atlas_attn_decode makes, with its status passed on unchanged.
    atlas::Plan plan;
    atlas_status st = atlas::make_plan(ATLAS_KIND_DECODE, n_q_heads, n_kv_heads, head_dim,
                                       page_tokens, L, &plan);
    if (st != ATLAS_OK) return st;
    if (L->phase != ATLAS_PHASE_ALL) return ATLAS_ERR_UNSUPPORTED;
    if (plan.ws_bytes > (size_t)ATLAS_STATIC_SCRATCH_BYTES) return ATLAS_ERR_WORKSPACE;
    void *scratch = nullptr;
    st = atlas::scratch_address(&scratch);
    if (st != ATLAS_OK) return st;
    atlas_launch local = *L;
    local.workspace = scratch;
    local.workspace_bytes = ATLAS_STATIC_SCRATCH_BYTES;
    return atlas_attn_decode(q, k_pages, v_pages, page_table, seq_lens, n_q_heads, n_kv_heads,
                             head_dim, page_tokens, scale, &local);
}
