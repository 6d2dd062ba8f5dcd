// Allocation-free variant of mla_verify_attn.
//
// Some callers cannot hand the library a device workspace: for example a
// plugin running inside a serving engine that owns all device memory through
// its own pool and exposes no workspace hook, or a latency-critical decode
// loop where calling cudaMalloc (which may synchronise the whole device) is
// not acceptable.  For them, mla_verify_attn_noalloc keeps its per-call scratch
// (status word, query offsets, ancestor bit sets, work list) in a file-scope
// device array instead of a caller-provided workspace, and runs the same
// kernels with a single KV split (no partial outputs to store).
//
// The array is kNoAllocScratchBytes long and lives on every GPU that loads the
// library until the process exits.  All calls share it: the prep kernel clears
// the words that must start at zero (status, item count) and writes every other
// byte before it is read, so stale contents from an earlier call never leak
// into a result, but two calls whose work overlaps on the GPU race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "mla_verify.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB per device
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device; the host-side symbol itself is not a device address).
int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return MLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MLA_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return MLA_OK;
}

}  // namespace

namespace mla_internal {
// Called by mla_init: drop the cached address of the scratch on `dev` (a reset
// device has a new context, in which the address is looked up again).
__attribute__((visibility("hidden"))) void noalloc_forget_device(int dev) {
    if (dev < 0 || dev >= kNoAllocMaxDevices) return;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    g_noalloc_ptr[dev] = nullptr;
}
}  // namespace mla_internal

extern "C" int mla_verify_noalloc_read_status(int* device_status) {
    if (!device_status) return MLA_ERR_INVALID_ARG;
    // the status word is the first word of the scratch (the workspace layout's first field)
    if (cudaMemcpyFromSymbol(device_status, g_noalloc_scratch, sizeof(int)) != cudaSuccess) return MLA_ERR_CUDA;
    return MLA_OK;
}

extern "C" int mla_verify_attn_noalloc(const void* q_lat, const void* q_rope, const void* kv_cache,
                                       const int32_t* block_table, const int32_t* seq_lens,
                                       const int32_t* tree_parent, const int32_t* n_tree, float scale,
                                       float* out, float* lse, cudaStream_t stream, int batch, int total_q,
                                       int max_tree, int max_seq_len, int num_heads, int page_size,
                                       int num_pages, int max_pages_per_seq) {
    if (batch < 0 || total_q < 0) return MLA_ERR_INVALID_ARG;
    const size_t need = mla_verify_workspace_size(batch, total_q, max_tree, max_seq_len, num_heads, 1);
    if (need == 0) return num_heads != MLA_NUM_HEADS ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
    if (need > kNoAllocScratchBytes) return MLA_ERR_WORKSPACE;  // batch / total_q beyond the static scratch
    void* scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != MLA_OK) return st;
    return mla_verify_attn(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree, scale, out, lse,
                           stream, batch, total_q, max_tree, max_seq_len, num_heads, page_size, num_pages,
                           max_pages_per_seq, 1, scratch, kNoAllocScratchBytes);
}
