// Per-call metadata for the verify kernel: query offsets of the requests,
// the ancestor-or-self bit set of every draft-tree node, input validation
// into the status word, and the list of (request, row tile) work items in
// longest-request-first order.  One thread block; integer work only.
#pragma once

#include <cstdint>

#include "verify_kernel.cuh"

namespace mla {

constexpr int kPrepThreads = 1024;
constexpr int kLptMaxBatch = 1024;  // above this the items keep request order
constexpr int kMaxTree = 64;         // the ancestor bit set is one 64-bit word

struct PrepParams {
    const int32_t* block_table;  // [batch, max_pages]
    const int32_t* seq_lens;     // [batch]
    const int32_t* tree_parent;  // [total_q]
    const int32_t* n_tree;       // [batch]
    int32_t* q_off;              // [batch + 1]
    int32_t* req_state;          // [batch]
    int32_t* order;              // [batch]  scratch: requests by descending length
    int32_t* item_off;           // [batch + 1]  scratch: first item of each request
    uint64_t* anc;               // [total_q]
    int2* items;                 // [max_items]
    int32_t* item_count;         // [1]
    int* status;                 // [1]
    int batch, total_q, page_size, max_pages, num_pages, max_items;
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
    __shared__ int32_t warp_sums[32];
    const int tid = threadIdx.x;
    if (tid == 0) {
        *p.status = 0;
        *p.item_count = 0;
    }
    __syncthreads();

    // 1. query offsets (exclusive scan of n_tree)
    block_exclusive_scan(p.batch, [&](int b) { return p.n_tree[b]; }, p.q_off, warp_sums);
    if (tid == 0 && p.q_off[p.batch] != p.total_q) atomicOr(p.status, kStatusBadTree);

    // 2. validate each request: sizes, parents, block ids
    for (int b = tid; b < p.batch; b += kPrepThreads) {
        const int T = p.n_tree[b];
        const int L = p.seq_lens[b];
        int state = 0;
        int bits = 0;
        if (T < 0 || T > kMaxTree || L < T || p.q_off[b] + T > p.total_q ||
            p.q_off[b] < 0) {
            state = 2;  // outputs of this request are not written at all
            bits |= kStatusBadTree;
        } else {
            for (int i = 0; i < T; ++i) {
                const int par = p.tree_parent[p.q_off[b] + i];
                if (par < -1 || par >= i) {
                    state = 1;
                    bits |= kStatusBadTree;
                }
            }
            const int pages = (L + p.page_size - 1) / p.page_size;
            if (pages > p.max_pages) {
                state = 1;
                bits |= kStatusBadBlock;
            } else {
                for (int k = 0; k < pages; ++k) {
                    const int pg = p.block_table[static_cast<long long>(b) * p.max_pages + k];
                    if (pg < 0 || pg >= p.num_pages) {
                        state = 1;
                        bits |= kStatusBadBlock;
                        break;
                    }
                }
            }
        }
        p.req_state[b] = state;
        if (bits) atomicOr(p.status, bits);
    }
    __syncthreads();

    // 3. ancestor-or-self bit sets, one node per thread (walk bounded by the tree size)
    for (int q = tid; q < p.total_q; q += kPrepThreads) {
        int lo = 0, hi = p.batch - 1;  // request owning q: last b with q_off[b] <= q
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.q_off[mid] <= q) lo = mid; else hi = mid - 1;
        }
        const int b = lo;
        uint64_t bits = 0;
        if (p.req_state[b] == 0) {
            const int base = p.q_off[b];
            int j = q - base;
            for (int step = 0; j >= 0 && step < kMaxTree; ++step) {
                bits |= 1ull << j;
                j = p.tree_parent[base + j];
            }
        }
        p.anc[q] = bits;
    }

    // 4. work items, longest requests first (better tail of the grid)
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
        if (p.item_off[p.batch] > p.max_items) atomicOr(p.status, kStatusBadTree);
    }
}

}  // namespace mla
