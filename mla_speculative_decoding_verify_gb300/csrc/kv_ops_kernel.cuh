// Paged-cache steps around tree verification: write the draft tree's latents
// into the cache before verify, and compact the accepted root-to-node path
// after it (page "The Shared Memory Ceiling", section "The Broader Context":
// the tree's KV lives in the same paged cache, and the step after
// verification is a KV-cache defrag).  One thread block per request; rows of
// 1152 bytes are moved as 72 16-byte vectors, so the results are exact.
#pragma once

#include <cstdint>

namespace mla {

constexpr int kKvOpThreads = 256;
constexpr int kKvRowVec = 576 * 2 / 16;       // 16-byte vectors per KV row
constexpr int kKvOpMaxTree = 64;
constexpr uint32_t kAcceptSmemBytes = kKvOpMaxTree * kKvRowVec * 16;  // all accepted rows of a request
constexpr int kKvStatusBadTree = 1 << 6;
constexpr int kKvStatusBadBlock = 1 << 7;

struct KvOpParams {
    const uint4* tree_kv;        // append: [total_q, 72] (576 bf16 per tree token)
    uint4* cache;                // [num_pages * page_size, 72]
    const int32_t* block_table;  // [batch, max_pages]
    const int32_t* seq_lens;     // [batch] prefix + tree tokens
    const int32_t* n_tree;       // [batch]
    const int32_t* tree_parent;  // accept: [total_q]
    const int32_t* accept_len;   // accept: [batch]
    const int32_t* accept_idx;   // accept: [total_q] path node indices, accept_len[b] of them per request
    int32_t* new_seq_lens;       // accept: [batch]
    int* status;                 // [1], zeroed by the host before the launch
    int batch, total_q, page_size, max_pages, num_pages;
};

// Sum of n_tree[0..b) over the block, a negative count read as 0: the first
// tree token of request b (64-bit, so that no sum of counts wraps).
__device__ __forceinline__ long long request_offset(const int32_t* n_tree, int b) {
    __shared__ long long partial[kKvOpThreads / 32];
    long long v = 0;
    for (int i = threadIdx.x; i < b; i += blockDim.x) v += max(__ldg(n_tree + i), 0);
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) partial[threadIdx.x >> 5] = v;
    __syncthreads();
    long long s = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) s += partial[w];
    __syncthreads();
    return s;
}

// Cache row of KV position pos of request b; -1 if its block id is out of range.
__device__ __forceinline__ long long cache_row(const KvOpParams& p, int b, int pos) {
    const int page_idx = pos / p.page_size;
    if (page_idx >= p.max_pages) return -1;
    const int page = __ldg(p.block_table + static_cast<long long>(b) * p.max_pages + page_idx);
    if (page < 0 || page >= p.num_pages) return -1;
    return static_cast<long long>(page) * p.page_size + pos % p.page_size;
}

// Every KV position of the request's tree region maps to a valid cache row (block-uniform).
__device__ __forceinline__ bool tree_pages_ok(const KvOpParams& p, int b, int P, int T) {
    bool bad = false;
    for (int i = threadIdx.x; i < T; i += blockDim.x) bad |= cache_row(p, b, P + i) < 0;
    return !__syncthreads_or(bad);
}

__global__ void __launch_bounds__(kKvOpThreads, 1) mla_tree_append_kernel(const KvOpParams p) {
    const int b = blockIdx.x;
    const int T = __ldg(p.n_tree + b);
    const int L = __ldg(p.seq_lens + b);
    if (T < 0 || T > kKvOpMaxTree || T > L) {
        if (threadIdx.x == 0) atomicOr(p.status, kKvStatusBadTree);
        return;
    }
    const int P = L - T;
    const long long off = request_offset(p.n_tree, b);
    if (off + T > p.total_q) {   // the request's rows of tree_kv lie past the end: malformed lengths
        if (threadIdx.x == 0) atomicOr(p.status, kKvStatusBadTree);
        return;
    }
    if (!tree_pages_ok(p, b, P, T)) {
        if (threadIdx.x == 0) atomicOr(p.status, kKvStatusBadBlock);
        return;
    }
    for (int idx = threadIdx.x; idx < T * kKvRowVec; idx += blockDim.x) {
        const int i = idx / kKvRowVec, u = idx % kKvRowVec;
        const long long row = cache_row(p, b, P + i);
        p.cache[row * kKvRowVec + u] = __ldg(p.tree_kv + static_cast<long long>(off + i) * kKvRowVec + u);
    }
}

__global__ void __launch_bounds__(kKvOpThreads, 1) mla_tree_accept_kernel(const KvOpParams p) {
    extern __shared__ uint4 rows[];  // [kKvOpMaxTree][kKvRowVec]
    const int b = blockIdx.x;
    const int T = __ldg(p.n_tree + b);
    const int L = __ldg(p.seq_lens + b);
    const int A = __ldg(p.accept_len + b);
    if (T < 0 || T > kKvOpMaxTree || T > L) {
        if (threadIdx.x == 0) {
            atomicOr(p.status, kKvStatusBadTree);
            p.new_seq_lens[b] = L;
        }
        return;
    }
    const int P = L - T;
    const long long off = request_offset(p.n_tree, b);
    // the request's rows of tree_parent / accept_idx lie inside [0, total_q)
    if (off + T > p.total_q) {
        if (threadIdx.x == 0) {
            atomicOr(p.status, kKvStatusBadTree);
            p.new_seq_lens[b] = L;
        }
        return;
    }
    // the tree (parents earlier than their children) and the path (a chain from a root)
    bool bad = A < 0 || A > T;
    for (int i = threadIdx.x; i < T; i += blockDim.x) {
        const int par = __ldg(p.tree_parent + off + i);
        bad |= par < -1 || par >= i;
    }
    if (!bad) {
        for (int k = threadIdx.x; k < A; k += blockDim.x) {
            const int v = __ldg(p.accept_idx + off + k);
            const int prev = k > 0 ? __ldg(p.accept_idx + off + k - 1) : -1;
            if (v < 0 || v >= T) {
                bad = true;
            } else {
                bad |= __ldg(p.tree_parent + off + v) != prev;
            }
        }
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) {
            atomicOr(p.status, kKvStatusBadTree);
            p.new_seq_lens[b] = L;
        }
        return;
    }
    if (!tree_pages_ok(p, b, P, T)) {
        if (threadIdx.x == 0) {
            atomicOr(p.status, kKvStatusBadBlock);
            p.new_seq_lens[b] = L;
        }
        return;
    }
    // read every accepted row before writing any: a node's old position can be
    // another accepted node's new one
    for (int idx = threadIdx.x; idx < A * kKvRowVec; idx += blockDim.x) {
        const int k = idx / kKvRowVec, u = idx % kKvRowVec;
        const int v = __ldg(p.accept_idx + off + k);
        rows[idx] = p.cache[cache_row(p, b, P + v) * kKvRowVec + u];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < A * kKvRowVec; idx += blockDim.x) {
        const int k = idx / kKvRowVec, u = idx % kKvRowVec;
        p.cache[cache_row(p, b, P + k) * kKvRowVec + u] = rows[idx];
    }
    if (threadIdx.x == 0) p.new_seq_lens[b] = P + A;
}

}  // namespace mla
