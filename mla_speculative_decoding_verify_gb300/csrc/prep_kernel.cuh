// Per-call metadata for the verify kernel: query offsets of the requests,
// the ancestor-or-self bit set of every draft-tree node, input validation
// into the status word, and the list of (request, row tile) work items in
// longest-request-first order.  One thread block; integer work only.  Each
// request is handled by one warp (its tree fits in two words per lane), so
// no thread walks a long chain of dependent global loads.
#pragma once

#include <cstdint>

#include "verify_kernel.cuh"

namespace mla {

constexpr int kPrepThreads = 1024;
constexpr int kPrepWarps = kPrepThreads / 32;
constexpr int kLptMaxBatch = 1024;  // above this the items keep request order
constexpr int kMaxTree = 64;        // the ancestor bit set is one 64-bit word

struct PrepParams {
    const int32_t* block_table;  // [batch, max_pages]
    const int32_t* seq_lens;     // [batch]
    const int32_t* tree_parent;  // [total_q]
    const int32_t* n_tree;       // [batch]
    int32_t* q_off;              // [batch + 1]
    int32_t* req_state;          // [batch]
    int32_t* order;              // [batch]      scratch: requests by descending length
    int32_t* item_off;           // [batch + 1]  scratch: first item of each request
    uint64_t* anc;               // [total_q]
    int2* items;                 // [max_items]
    int32_t* item_count;         // [1]
    int* status;                 // [1]
    int batch, total_q, page_size, max_pages, num_pages, max_items;
    int32_t* tok_req;            // sparse variant: [total_q] request of each tree token (-1 if malformed), else null
    int allow_unused_rows;       // graph replay: sum(n_tree) may be below total_q; the trailing rows are unused
    int32_t* zero_words;         // words cleared before the verify kernel (its two-split merge counters), or null
    int zero_count;
    int32_t* tail_k;             // one split: how many items of the last, partial round to cut in two, or null
    int tail_cap, pairs;         // at most tail_cap; CTA pairs of the device
};

// Exclusive block-wide scan of f(i) for i in [0, n) into dst[0..n] (dst[n] = total).
template <typename F>
__device__ void block_exclusive_scan(int n, F f, int32_t* dst, int32_t* warp_sums) {
    const int tid = threadIdx.x;
    const int lane = tid & 31, wid = tid >> 5;
    int carry = 0;
    for (int base = 0; base < n; base += kPrepThreads) {
        const int i = base + tid;
        const int v = i < n ? f(i) : 0;
        int x = v;
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int w = warp_sums[lane];
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sums[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int before = (wid > 0 ? warp_sums[wid - 1] : 0) + x - v;
        if (i < n) dst[i] = carry + before;
        const int chunk_total = warp_sums[31];
        __syncthreads();
        carry += chunk_total;
    }
    if (tid == 0) dst[n] = carry;
    __syncthreads();
}

__global__ void __launch_bounds__(kPrepThreads, 1) mla_prep_kernel(const PrepParams p) {
    grid_launch_dependents();   // the verify kernel may start its launch; it waits for this grid's results
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t tree_par[kPrepWarps][kMaxTree];
    __shared__ uint64_t tree_anc[kPrepWarps][kMaxTree];
    const int tid = threadIdx.x;
    const int lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        *p.status = 0;
        *p.item_count = 0;
    }
    __syncthreads();

    // 0. sparse variant: no token belongs to a request until step 2 says so
    if (p.tok_req)
        for (int g = tid; g < p.total_q; g += kPrepThreads) p.tok_req[g] = -1;
    if (p.zero_words)
        for (int g = tid; g < p.zero_count; g += kPrepThreads) p.zero_words[g] = 0;

    // 1. query offsets (exclusive scan of n_tree)
    block_exclusive_scan(p.batch, [&](int b) { return p.n_tree[b]; }, p.q_off, warp_sums);
    if (tid == 0 && (p.allow_unused_rows ? p.q_off[p.batch] > p.total_q : p.q_off[p.batch] != p.total_q))
        atomicOr(p.status, kStatusBadTree);

    // 2. one warp per request: validate sizes, parents and block ids, then the
    //    ancestor bit sets by pointer jumping (6 rounds cover depth 64)
    for (int b = wid; b < p.batch; b += kPrepWarps) {
        const int T = p.n_tree[b];
        const int L = p.seq_lens[b];
        const int base = p.q_off[b];
        const bool shape_ok = T >= 0 && T <= kMaxTree && L >= T && base >= 0 && base + T <= p.total_q;
        bool bad_parent = false, bad_block = false;
        if (shape_ok) {
            for (int i = lane; i < T; i += 32) {
                const int par = p.tree_parent[base + i];
                const bool good = par >= -1 && par < i;
                tree_par[wid][i] = good ? par : -1;
                bad_parent |= !good;
            }
            const int pages = (L + p.page_size - 1) / p.page_size;
            if (pages > p.max_pages) {
                bad_block = true;
            } else {
                const int32_t* row = p.block_table + static_cast<long long>(b) * p.max_pages;
                for (int k = lane; k < pages; k += 32) {
                    const int pg = row[k];
                    bad_block |= pg < 0 || pg >= p.num_pages;
                }
            }
        }
        if (shape_ok && p.tok_req)
            for (int i = lane; i < T; i += 32) p.tok_req[base + i] = b;
        bad_parent = __any_sync(0xffffffffu, bad_parent);
        bad_block = __any_sync(0xffffffffu, bad_block);
        const bool all_ok = shape_ok && !bad_parent && !bad_block;
        if (lane == 0) {
            p.req_state[b] = shape_ok ? (all_ok ? 0 : 1) : 2;  // 2: outputs not written at all
            const int bits = ((!shape_ok || bad_parent) ? kStatusBadTree : 0) | (bad_block ? kStatusBadBlock : 0);
            if (bits) atomicOr(p.status, bits);
        }
        __syncwarp();
        if (shape_ok) {
            // pointer jumping: anc(i) = {i} u anc(parent(i))
            uint64_t a[2];
            int up[2];
            for (int h = 0; h < 2; ++h) {
                const int i = lane + 32 * h;
                a[h] = i < T ? (1ull << i) : 0ull;
                up[h] = i < T ? tree_par[wid][i] : -1;
                if (i < T) tree_anc[wid][i] = a[h];
            }
            __syncwarp();
            for (int round = 0; round < 6; ++round) {
                uint64_t na[2];
                int nu[2];
                for (int h = 0; h < 2; ++h) {
                    na[h] = a[h] | (up[h] >= 0 ? tree_anc[wid][up[h]] : 0ull);
                    nu[h] = up[h] >= 0 ? tree_par[wid][up[h]] : -1;
                }
                __syncwarp();
                for (int h = 0; h < 2; ++h) {
                    const int i = lane + 32 * h;
                    a[h] = na[h];
                    up[h] = nu[h];
                    if (i < T) {
                        tree_anc[wid][i] = a[h];
                        tree_par[wid][i] = up[h];
                    }
                }
                __syncwarp();
            }
            for (int h = 0; h < 2; ++h) {
                const int i = lane + 32 * h;
                if (i < T) p.anc[base + i] = all_ok ? a[h] : 0ull;
            }
        }
        __syncwarp();
    }
    __syncthreads();

    // 3. work items, longest requests first (better tail of the grid)
    const bool lpt = p.batch <= kLptMaxBatch;
    for (int b = tid; b < p.batch; b += kPrepThreads) {
        int rank = b;
        if (lpt) {
            const int Lb = p.seq_lens[b];
            rank = 0;
            for (int o = 0; o < p.batch; ++o) {
                const int Lo = p.seq_lens[o];
                rank += (Lo > Lb) || (Lo == Lb && o < b);
            }
        }
        p.order[rank] = b;
    }
    __syncthreads();
    block_exclusive_scan(
        p.batch,
        [&](int k) {
            const int b = p.order[k];
            return p.req_state[b] == 2 ? 0 : (p.n_tree[b] + kTokensPerTile - 1) / kTokensPerTile;
        },
        p.item_off, warp_sums);
    const int total_items = min(p.item_off[p.batch], p.max_items);
    for (int k = tid; k < p.batch; k += kPrepThreads) {
        const int b = p.order[k];
        if (p.req_state[b] == 2) continue;
        const int cnt = (p.n_tree[b] + kTokensPerTile - 1) / kTokensPerTile;
        for (int t = 0; t < cnt; ++t) {
            const int slot = p.item_off[k] + t;
            if (slot < p.max_items) p.items[slot] = make_int2(b, t);
        }
    }
    if (tid == 0) {
        *p.item_count = total_items;
        if (p.tail_k) {
            const int rem = p.pairs > 0 ? total_items % p.pairs : 0;
            *p.tail_k = (rem > 0 && 2 * rem <= p.pairs) ? min(rem, p.tail_cap) : 0;
        }
        if (p.item_off[p.batch] > p.max_items) atomicOr(p.status, kStatusBadTree);
    }
}

// Sparse variant: every top-k slot must be -1 or a prefix position of its
// token's request; otherwise the request's rows are written as out = 0,
// lse = -inf and the status gets kStatusBadIndex.  Grid-stride, coalesced.
constexpr int kCheckThreads = 256;

__global__ void __launch_bounds__(kCheckThreads) mla_topk_check_kernel(const int32_t* topk_idx, int topk,
                                                                     long long entries, const int32_t* tok_req,
                                                                     const int32_t* seq_lens, const int32_t* n_tree,
                                                                     int batch, int32_t* req_state, int* status) {
    grid_dependency_wait();     // the prep kernel's tok_req and req_state
    grid_launch_dependents();
    for (long long e = blockIdx.x * static_cast<long long>(kCheckThreads) + threadIdx.x; e < entries;
         e += static_cast<long long>(gridDim.x) * kCheckThreads) {
        const int v = __ldg(topk_idx + e);
        const int b = __ldg(tok_req + e / topk);
        if (b < 0 || b >= batch) continue;   // token of a malformed request
        const int P = __ldg(seq_lens + b) - __ldg(n_tree + b);
        if (v < -1 || v >= P) {
            if (req_state[b] == 0) req_state[b] = 1;
            atomicOr(status, kStatusBadIndex);
        }
    }
}

}  // namespace mla
