// Per-call metadata for the verify kernel: query offsets of the requests,
// the ancestor-or-self bit set of every draft-tree node, input validation
// into the status word, the list of (request, row tile) work items in
// longest-request-first order, and, for the persistent schedule, each CTA
// pair's share of the sequence of all (item, KV tile) positions.  One thread
// block; integer work only.  Each request is handled by one warp (its tree
// fits in two words per lane), so no thread walks a long chain of dependent
// global loads.
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
    // persistent schedule (else null): item i holds positions [woff[i], woff[i + 1]) of the
    // sequence of all (item, KV tile) pairs, one position per KV tile (an invalid request's
    // item: one position and no tiles).  The first *rounds x sched_pairs items go whole,
    // one per CTA pair and round; CTA pair q takes positions [pair_begin[q], pair_begin[q + 1])
    // of the remaining items, an equal share moved to an item boundary when it would leave
    // a piece of fewer than min_piece tiles
    long long* woff;             // [max_items + 1]
    long long* pair_begin;       // [sched_pairs + 1]
    int32_t* pair_item;          // [sched_pairs + 1] item holding pair_begin[q] (item count at the end)
    int32_t* item_first_pair;    // [max_items] first pair whose share holds a position of the item
    int32_t* rounds;             // [1]
    int sched_pairs, min_piece;
    int topk;                    // sparse variant: slots per tree token (0 for the dense verify)
};

// Exclusive block-wide scan of f(i) for i in [0, n) into dst[0..n] (dst[n] = total).
template <typename T, typename F>
__device__ void block_exclusive_scan(int n, F f, T* dst, T* warp_sums) {
    const int tid = threadIdx.x;
    const int lane = tid & 31, wid = tid >> 5;
    T carry = 0;
    for (int base = 0; base < n; base += kPrepThreads) {
        const int i = base + tid;
        const T v = i < n ? static_cast<T>(f(i)) : T(0);
        T x = v;
        for (int o = 1; o < 32; o <<= 1) {
            const T y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[wid] = x;
        __syncthreads();
        if (wid == 0) {
            T w = lane < kPrepWarps ? warp_sums[lane] : T(0);
            for (int o = 1; o < 32; o <<= 1) {
                const T y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sums[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const T before = (wid > 0 ? warp_sums[wid - 1] : T(0)) + x - v;
        if (i < n) dst[i] = carry + before;
        const T chunk_total = warp_sums[kPrepWarps - 1];
        __syncthreads();
        carry += chunk_total;
    }
    if (tid == 0) dst[n] = carry;
    __syncthreads();
}

// Batches up to this size keep their per-request values in shared memory, so
// that no step reads back from global memory what an earlier step wrote: the
// kernel's critical path is then two rounds of global loads (the request
// sizes; the tree parents together with the block tables) instead of about ten.
constexpr int kStageBatch = 1024;
static_assert(kLptMaxBatch <= kStageBatch, "longest-first ordering reads the staged lengths");

__global__ void __launch_bounds__(kPrepThreads, 1) mla_prep_kernel(const PrepParams p) {
    grid_launch_dependents();   // the verify kernel may start its launch; it waits for this grid's results
    __shared__ int32_t warp_sums[32];
    __shared__ long long warp_sums64[32];
    __shared__ int8_t tree_par[kPrepWarps][kMaxTree];
    __shared__ uint64_t tree_anc[kPrepWarps][kMaxTree];
    __shared__ int32_t s_nt[kStageBatch], s_len[kStageBatch], s_state[kStageBatch], s_order[kStageBatch];
    __shared__ int32_t s_qoff[kStageBatch + 1], s_ioff[kStageBatch + 1];
    const int tid = threadIdx.x;
    const int lane = tid & 31, wid = tid >> 5;
    const bool staged = p.batch <= kStageBatch;
    // per-request values: shared memory for staged batches, else global memory
    // (q_off, req_state, order and item_off are written here: plain loads after a barrier)
    auto NT = [&](int b) -> int { return staged ? s_nt[b] : __ldg(p.n_tree + b); };
    auto LEN = [&](int b) -> int { return staged ? s_len[b] : __ldg(p.seq_lens + b); };
    auto QOFF = [&](int b) -> int { return staged ? s_qoff[b] : p.q_off[b]; };
    auto STATE = [&](int b) -> int { return staged ? s_state[b] : p.req_state[b]; };
    auto ORDER = [&](int k) -> int { return staged ? s_order[k] : p.order[k]; };
    auto IOFF = [&](int k) -> int { return staged ? s_ioff[k] : p.item_off[k]; };
    if (staged) {
        for (int b = tid; b < p.batch; b += kPrepThreads) {
            s_nt[b] = __ldg(p.n_tree + b);
            s_len[b] = __ldg(p.seq_lens + b);
        }
    }
    if (tid == 0) {
        *p.status = 0;
        *p.item_count = 0;
    }
    // 0. sparse variant: no token belongs to a request until step 2 says so
    if (p.tok_req)
        for (int g = tid; g < p.total_q; g += kPrepThreads) p.tok_req[g] = -1;
    if (p.zero_words)
        for (int g = tid; g < p.zero_count; g += kPrepThreads) p.zero_words[g] = 0;
    __syncthreads();

    // 1. query offsets (exclusive scan of n_tree)
    block_exclusive_scan(p.batch, NT, staged ? s_qoff : p.q_off, warp_sums);
    if (staged)
        for (int b = tid; b <= p.batch; b += kPrepThreads) p.q_off[b] = s_qoff[b];
    if (tid == 0 && (p.allow_unused_rows ? QOFF(p.batch) > p.total_q : QOFF(p.batch) != p.total_q))
        atomicOr(p.status, kStatusBadTree);

    // 2. one warp per request: validate sizes, parents and block ids, then the
    //    ancestor bit sets by pointer jumping (6 rounds cover depth 64).  The
    //    parents and the block-table entries are loaded together, before either
    //    is used, so their round trips overlap.
    for (int b = wid; b < p.batch; b += kPrepWarps) {
        const int T = NT(b);
        const int L = LEN(b);
        const int base = QOFF(b);
        const bool shape_ok = T >= 0 && T <= kMaxTree && L >= T && base >= 0 && base + T <= p.total_q;
        int par[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = lane + 32 * h;
            par[h] = shape_ok && i < T ? __ldg(p.tree_parent + base + i) : -1;
        }
        bool bad_parent = false, bad_block = false;
        if (shape_ok) {
            const int pages = (L + p.page_size - 1) / p.page_size;
            if (pages > p.max_pages) {
                bad_block = true;
            } else {
                const int32_t* row = p.block_table + static_cast<long long>(b) * p.max_pages;
                for (int k0 = 0; k0 < pages; k0 += 128) {
                    int pg[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int k = k0 + 32 * u + lane;
                        pg[u] = k < pages ? __ldg(row + k) : 0;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        bad_block |= k0 + 32 * u + lane < pages && (pg[u] < 0 || pg[u] >= p.num_pages);
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = lane + 32 * h;
                if (i < T) {
                    const bool good = par[h] >= -1 && par[h] < i;
                    tree_par[wid][i] = static_cast<int8_t>(good ? par[h] : -1);
                    bad_parent |= !good;
                }
            }
        }
        if (shape_ok && p.tok_req)
            for (int i = lane; i < T; i += 32) p.tok_req[base + i] = b;
        bad_parent = __any_sync(0xffffffffu, bad_parent);
        bad_block = __any_sync(0xffffffffu, bad_block);
        const bool all_ok = shape_ok && !bad_parent && !bad_block;
        if (lane == 0) {
            const int state = shape_ok ? (all_ok ? 0 : 1) : 2;  // 2: outputs not written at all
            p.req_state[b] = state;
            if (staged) s_state[b] = state;
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
                        tree_par[wid][i] = static_cast<int8_t>(up[h]);
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
            const int Lb = LEN(b);
            rank = 0;
            for (int o = 0; o < p.batch; ++o) {
                const int Lo = LEN(o);
                rank += (Lo > Lb) || (Lo == Lb && o < b);
            }
        }
        if (staged) s_order[rank] = b;
        else p.order[rank] = b;
    }
    __syncthreads();
    block_exclusive_scan(
        p.batch,
        [&](int k) {
            const int b = ORDER(k);
            return STATE(b) == 2 ? 0 : (NT(b) + kTokensPerTile - 1) / kTokensPerTile;
        },
        staged ? s_ioff : p.item_off, warp_sums);
    const int total_items = min(IOFF(p.batch), p.max_items);
    for (int k = tid; k < p.batch; k += kPrepThreads) {
        const int b = ORDER(k);
        if (STATE(b) == 2) continue;
        const int cnt = (NT(b) + kTokensPerTile - 1) / kTokensPerTile;
        for (int t = 0; t < cnt; ++t) {
            const int slot = IOFF(k) + t;
            if (slot < p.max_items) p.items[slot] = make_int2(b, t);
        }
    }
    if (tid == 0) {
        *p.item_count = total_items;
        if (p.tail_k) {
            const int rem = p.pairs > 0 ? total_items % p.pairs : 0;
            *p.tail_k = (rem > 0 && 2 * rem <= p.pairs) ? min(rem, p.tail_cap) : 0;
        }
        if (IOFF(p.batch) > p.max_items) atomicOr(p.status, kStatusBadTree);
    }

    // 4. persistent schedule: the CTA pairs' shares of all (item, KV tile) positions
    if (p.woff) {
        __syncthreads();   // the work items written above
        const int n = total_items;
        block_exclusive_scan(
            n,
            [&](int k) -> long long {
                const int2 it = p.items[k];
                const int b = it.x;
                if (STATE(b) != 0) return 1;   // rows written as out = 0, lse = -inf; no tiles
                const int T = NT(b);
                if (p.topk > 0) {
                    const int nA = (p.topk + kBlockN - 1) / kBlockN;
                    const int ntok = min(kTokensPerTile, T - kTokensPerTile * it.y);
                    return static_cast<long long>(nA) * (ntok > 1 ? 2 : 1) + (T + kBlockN - 1) / kBlockN;
                }
                return (LEN(b) + kBlockN - 1) / kBlockN;
            },
            p.woff, warp_sums64);
        const long long W = p.woff[n];
        const int G = p.sched_pairs;
        // Rounds of whole items first (the row tiles of a request then stream its KV
        // together, sharing it in L2); the last, partial round is shared out evenly.  A
        // partial round of fewer than G / 4 items joins the one before, so that its
        // items are not cut into many small pieces.
        int R = n / G;
        if (R > 0 && n - R * G < G / 4) --R;
        const long long X0 = p.woff[R * G], Wt = W - X0;
        if (tid == 0) *p.rounds = R;
        for (int q = tid; q <= G; q += kPrepThreads) {
            long long x = X0 + (q >= G ? Wt : Wt * q / G);
            int i = n;
            if (x < W) {
                int lo = 0, hi = n - 1;   // the item holding x: the last i with woff[i] <= x
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (p.woff[mid] <= x) lo = mid;
                    else hi = mid - 1;
                }
                i = lo;
                if (q > 0) {
                    const long long O = p.woff[i], E = p.woff[i + 1];
                    if (x - O < p.min_piece) {
                        x = O;
                    } else if (E - x < p.min_piece) {
                        x = E;
                        ++i;
                    }
                }
            }
            p.pair_begin[q] = x;
            p.pair_item[q] = i;
        }
        __syncthreads();
        for (int i = R * G + tid; i < n; i += kPrepThreads) {
            const long long O = p.woff[i];
            int lo = 0, hi = G - 1;   // the first pair whose share ends after O
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (p.pair_begin[mid + 1] > O) hi = mid;
                else lo = mid + 1;
            }
            p.item_first_pair[i] = lo;
        }
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
