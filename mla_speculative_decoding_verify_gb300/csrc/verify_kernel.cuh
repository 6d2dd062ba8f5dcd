// Fused tree-verify MLA attention kernel for sm_103a.
//
// One 2-CTA cluster computes 128 output rows (2 tree tokens x 64 heads) of one
// request over a range of its KV tiles.  The pair divides the work along the
// feature axis: CTA c owns latent dims [256c, 256c+256) and rope dims [32c, 32c+32).
//   - QK^T: each CTA multiplies its half of q by its half of every key
//     (tcgen05, q latent half resident in TMEM, keys streamed by TMA), giving
//     a partial score tile; the partials are exchanged through distributed
//     shared memory and added, so both CTAs hold the same full 576-dim score.
//   - softmax: online and lazy (page "The Shared Memory Ceiling", section
//     "Technical Deep Dive": running max and normaliser, earlier accumulators
//     rescaled when the max grows), one thread per row, tree mask applied from
//     the ancestor bit set of the row's node.
//   - PV: each CTA accumulates its 256 columns of O = P * c_kv in TMEM (V is
//     the c_kv latent, so the same shared-memory tile that served as K feeds
//     PV).  P goes to TMEM as bf16 (the A operand of PV); when a tile carries a
//     large share of a row's mass a second bf16 "low part" of P is added so the
//     result keeps close to fp32 weights.
// Pipeline: the exchange warps read a tile's partial scores out of TMEM as soon
// as QK has written them, stage them in shared memory and ship them to the
// peer; the S columns are therefore free again right after they were read, and
// the QK issuer runs ahead, bounded by the four-stage KV ring.  The softmax
// threads add the two partials, exponentiate and write P; a PV issuer (dense:
// its own warp; sparse: the QK warp, two tiles behind QK) consumes it.
// Sparse (top-k) variant (kSparse = true; page "The SMEM Ceiling", section
// "The Problem Space": each token attends to a top-k selected set of earlier
// tokens): tree token g sees the prefix positions listed in its topk slots and
// its ancestor-or-self tree tokens.  A row tile's key sequence is token 0's
// slots, then token 1's slots, then the tree keys; rows see only their own
// token's slots.  Three warps gather the rows with four-row tensor gathers
// into the same swizzled stage layout (empty slots read as zeros) and record
// which of the tile's 64 slots are real.
// Schedules (template parameter kSched):
//   - per-unit grid (kSchedPlain, kSchedMerge): one CTA pair per work unit, a
//     range of one row tile's KV tiles (split KV, flash-decoding style); two
//     splits are merged here by the second unit of each row tile to finish,
//     more by a separate combine pass;
//   - persistent (kSchedPersistent): a fixed grid of CTA pairs, each taking an
//     equal, contiguous share of the sequence of all (work item, KV tile)
//     positions.  A pair walks its share item by item with one pipeline:
//     barriers, TMEM and the cluster stay alive, the KV ring keeps streaming
//     across item boundaries.  An item cut between two or more pairs is merged
//     in the kernel by the last of its pieces to finish (LSE weights, summed in
//     piece order so that the result does not depend on the order of arrival).
// TMEM: O [0,256) | q latent half [256,384) | S [384,448) | P [448,480), its low part [480,512).
#pragma once

#include <cuda.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace mla {

constexpr int kHeads = 64;
constexpr int kDLatent = 512;
constexpr int kDRope = 64;
constexpr int kDqk = kDLatent + kDRope;
constexpr int kBlockN = 64;            // keys per KV tile
constexpr int kRows = 128;             // (token, head) rows per CTA
constexpr int kTokensPerTile = kRows / kHeads;
constexpr int kDLatentHalf = kDLatent / 2;
constexpr int kDRopeHalf = kDRope / 2;
constexpr int kStages = 4;
// Three warpgroups.  Warpgroup 0: warp 0 TMA producer, warp 1 QK MMAs, warp 2 PV MMAs
// (dense; sparse: warps 0, 2 and 3 gather the KV rows and warp 1 issues QK and PV).
// Warpgroup 1 (warps 4..7): softmax, one thread per row.  Warpgroup 2 (warps 8..11):
// the exchange, partial scores from TMEM through the staging buffer to the peer.
// Warp w reaches TMEM lanes [32 (w % 4), 32 (w % 4) + 32), so each row-owning
// warpgroup covers the 128 lanes.
constexpr int kThreads = 384;
constexpr int kThreadsSparse = 384;
constexpr int kGatherWarp2 = 3;
constexpr int kGatherWarps = 3;        // sparse: warps 0, kPvWarp and kGatherWarp2
// Sparse gather warp w (0, 1, 2) owns the four-key groups [gather_group0(w),
// gather_group0(w + 1)) of every 64-key tile: 6, 5 and 5 groups.
__host__ __device__ constexpr int gather_group0(int w) { return w == 0 ? 0 : w == 1 ? 6 : w == 2 ? 11 : 16; }
constexpr int kSoftmaxWarp0 = 4;
constexpr int kStagerWarp0 = 8;
constexpr int kPvWarp = 2;             // dense: the PV issuer; sparse: a gather warp
// Register split (setmaxnreg).  An increase draws only on the registers the block was
// launched with, so the three warpgroups' shares must add up to at most the launch's
// total: 384 threads at 168 each (the most __launch_bounds__(384, 1) allows) hold
// 64,512 = 128 x 232 (softmax) + 256 x 136 (the others).  The host checks the compiled
// register count against this before the first launch (a larger split would wait
// forever).
constexpr int kRegsAtLaunch = 168, kRegsSoftmax = 232, kRegsOther = 136;
static_assert(128 * kRegsSoftmax + 256 * kRegsOther <= 384 * kRegsAtLaunch, "register split above the launch total");
static_assert(kRegsSoftmax % 8 == 0 && kRegsOther % 8 == 0, "setmaxnreg counts are multiples of 8");
static_assert(kThreads == 3 * 128 && kThreadsSparse == 3 * 128, "three warpgroups");
static_assert(gather_group0(kGatherWarps) * 4 == 64 && 4 * gather_group0(1) <= 32,
              "gather warps cover a tile's 64 keys, at most one key per lane");
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kChunkBytes = kBlockN * 64 * 2;          // [64 keys][64 dims] bf16, 128B swizzle
constexpr uint32_t kRopeTileBytes = kBlockN * kDRopeHalf * 2;  // [64 keys][32 dims], 64B swizzle
constexpr uint32_t kStageBytes = 4 * kChunkBytes + kRopeTileBytes;
constexpr uint32_t kQRopeBytes = kRows * kDRopeHalf * 2;
constexpr uint32_t kXBufBytes = kRows * kBlockN * 4;       // one partial score tile, fp32
constexpr uint32_t kOffStages = 0;
constexpr uint32_t kOffQRope = kOffStages + kStages * kStageBytes;
constexpr uint32_t kOffXBuf = kOffQRope + kQRopeBytes;          // receive buffer (the peer's partial)
constexpr uint32_t kOffStaging = kOffXBuf + kXBufBytes;         // own partial, source of the bulk copy
constexpr uint32_t kOffCtrl = kOffStaging + kXBufBytes;
constexpr uint32_t kCtrlBytes = 512;
constexpr uint32_t kOffVis = kOffCtrl + kCtrlBytes;             // dense: per row, the visibility bits of the
constexpr uint32_t kVisBytes = kRows * 16;                      // two KV tiles that reach the draft tokens
constexpr uint32_t kSmemBytes = kOffVis + kVisBytes + 1024;     // + slack for 1 KB alignment
static_assert(kStageBytes % 1024 == 0, "stages must keep 1 KB alignment for 128B swizzle");
static_assert(kOffQRope % 1024 == 0 && kOffXBuf % 1024 == 0 && kOffStaging % 1024 == 0, "region alignment");
static_assert(kSmemBytes <= 232448, "exceeds the sm_103 opt-in shared memory per block");
// the two-split merge copies the other split's 128 rows x 1 KB over the stages, q rope and receive buffer
static_assert(kOffStaging - kOffStages >= kRows * kDLatentHalf * 4, "merge buffer");
// Outside the tile loop the staging buffer (32 KB) is scratch, per softmax warp: the q
// rows of a segment land there in two rounds of 8 KB; an epilogue's rows leave through
// its first 4 KB tile, the persistent merge reads other pieces' rows through the second.
static_assert(kXBufBytes == 4 * 8192, "staging region");

constexpr uint32_t kTmemCols = 512;
// TMEM columns: O (fp32, this CTA's 256 dims), q (bf16 pairs), S (fp32, one 64-key tile),
// P (bf16 pairs: high part, then the low part)
constexpr uint32_t kTmO = 0, kTmQ = 256, kTmS = 384, kTmP = 448, kTmPLo = 480;
constexpr uint32_t kTmAcc = 256;   // persistent merge: accumulator over the q, S and P columns (free in an epilogue)

constexpr float kLazyRescaleLog2 = 8.0f;   // rescale only when the max grows by > 2^8
constexpr float kLowPartShare = 1.0f / 16.0f;

// Status bits (1 << mla_status code).
constexpr int kStatusTimeout = 1 << 5;
constexpr int kStatusBadTree = 1 << 6;
constexpr int kStatusBadBlock = 1 << 7;
constexpr int kStatusBadIndex = 1 << 9;

// Schedules of the verify kernel.
constexpr int kSchedPlain = 0;        // one work unit per CTA pair; more than one split goes to the combine pass
constexpr int kSchedMerge = 1;        // the same, and two-split / cut units merged in the kernel
constexpr int kSchedPersistent = 2;   // a fixed grid of CTA pairs, each walking its share of all KV tiles

struct VerifyParams {
    const uint16_t* q_lat;      // [total_q, 64, 512]
    const uint16_t* q_rope;     // [total_q, 64, 64]
    const int32_t* block_table; // [batch, max_pages]
    const int32_t* seq_lens;    // [batch]
    const int32_t* n_tree;      // [batch]
    const int32_t* q_off;       // [batch + 1]   from the prep kernel
    const uint64_t* anc;        // [total_q]     ancestor-or-self bit set of each node
    const int32_t* req_state;   // [batch]       0 ok, 1 invalid (rows zeroed)
    const int2* items;          // [max_items]   (request, row tile)
    const int32_t* item_count;  // [1]
    int* status;                // [1]
    float* out;                 // [total_q, 64, 512]
    float* lse;                 // [total_q, 64]
    float* part_out;            // per-unit grid: [num_splits, total_q * 64, 512]; persistent: [2 * pairs, 128, 512]
    float* part_lse;            // per-unit grid: [num_splits, total_q * 64]; persistent: [2 * pairs, 2, 128]
    int batch, total_q, page_size, max_pages, num_pages, num_splits, max_items;
    int split_share;            // two splits: the first one's share of a work item's tiles, in 1/1024 (0 = halves)
    // one split, but the last *tail_k (<= tail_cap) work items cut in two (tail_share for the first
    // part) and merged; their partials are compact: tail_cap row tiles per split
    int tail_cap, tail_share;
    const int32_t* tail_k;      // written by the prep kernel, or null
    // this launch computes splits split_base .. split_base + gridDim.y - 1 of num_splits; their
    // partials go to part_out / part_lse slots 0 .. gridDim.y - 1 (0 unless a range of splits is asked for)
    int split_base;
    float scale_log2;           // softmax scale * log2(e)
    uint64_t timeout_ns;
    // sparse variant only
    const int32_t* topk_idx;    // [total_q, topk] prefix positions, -1 = unused slot
    const uint16_t* kv;         // the cache [num_pages * page_size, 576] (L2 prefetch of gathered rows)
    // two KV splits or cut items merged in the kernel: [max_items][2 halves][arrived, written],
    // zeroed by the prep kernel (else null)
    int32_t* merge_cnt;
    int topk;
    // persistent schedule (written by the prep kernel; else null).  Position x of the
    // sequence of all (work item, KV tile) pairs: item i holds [woff[i], woff[i + 1]).
    // Items 0 .. *rounds * pairs - 1 go whole, one per CTA pair and round (snake
    // order); the positions of the others are shared out.
    const long long* woff;        // [items + 1]
    const long long* pair_begin;  // [pairs + 1] first position of each CTA pair's share
    const int32_t* pair_item;     // [pairs + 1] item holding that position
    const int32_t* item_first_pair;  // [items] first CTA pair whose share holds a tile of the item
    const int32_t* rounds;        // [1]
    int pairs;
};

struct Ctrl {
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t kv_fixed[kStages];
    uint64_t s_full;       // QK wrote the S columns (one phase per tile)
    uint64_t s_free;       // the softmax threads read them out (QK may overwrite them)
    uint64_t p_full[2];    // P of tile j is in its TMEM columns (j & 1 selects the barrier)
    uint64_t pv_done[2];   // PV of tile j finished (P columns and O free again)
    uint64_t x_full;       // the peer's partial of the next tile landed in the receive buffer (bytes)
    uint64_t x_empty;      // the peer finished reading the partial this CTA sent it
    uint64_t stg_free;     // peer received this CTA's staging buffer (may be overwritten)
    uint64_t staged;       // the exchange warps put the own partial of the next tile in the staging buffer
    uint64_t stg_read[4];  // softmax warp w has read its 32 rows of it (exchange warp w may overwrite them)
    uint64_t q_ready;      // q of the next segment is in TMEM / shared memory (one phase per segment)
    uint64_t drain_qk;
    uint64_t drain_pv;
    uint64_t never;        // fault injection: nothing arrives on it
    uint32_t tmem_base;
    int abort;
    int lo_flag[2];
    int tile_flags[3];  // per-tile OR of the softmax threads' votes: bit 0 low part of P, bit 1 stop
    int merge_role;     // in-kernel merge: arrival rank of this unit / piece among the row tile's
    uint32_t slot_mask[kStages][kGatherWarps];  // sparse: bit k of word w set if key 4 * gather_group0(w) + k of
                                                // the stage's tile is a real slot
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

__device__ __forceinline__ void raise_status(int* status, int bit) { atomicOr(status, bit); }

// Fault injection (a test build only, compiled with MLA_FAULT_INJECTION): make
// one bounded wait run out so that the timeout paths can be tested without
// faulting or hanging the GPU.  Kinds, all in the first segment of work item 0
// (split 0) and CTA 0 of its pair:
//   1  the QK issuer waits for KV tile 1 on a barrier that nothing completes;
//   2  (two splits merged in the kernel) the first unit of the row tile never
//      marks its partial written, so the second one's poll runs out;
//   3  the exchange warps do not send the partial scores of tile 1;
//   4  (persistent schedule) the pieces of cut items other than the last never
//      mark their partials written, so the last one's poll runs out.
#ifdef MLA_FAULT_INJECTION
__device__ int g_fault_kind;
__device__ __forceinline__ int fault_kind() { return *reinterpret_cast<volatile int*>(&g_fault_kind); }
#else
__device__ __forceinline__ constexpr int fault_kind() { return 0; }
#endif

// Which KV tiles [t0, t1) split `s` of `S` covers, for a request of n tiles.  With
// two splits and share > 0 the first split takes share / 1024 of the tiles.
__device__ __forceinline__ void split_range(int n, int s, int S, int share, int& t0, int& t1) {
    if (S == 2 && share > 0) {
        const int a = static_cast<int>(min(static_cast<long long>(n), (static_cast<long long>(n) * share + 512) >> 10));
        t0 = s == 0 ? 0 : a;
        t1 = s == 0 ? a : n;
        return;
    }
    t0 = static_cast<int>((static_cast<long long>(n) * s) / S);
    t1 = static_cast<int>((static_cast<long long>(n) * (s + 1)) / S);
}

// Sparse key sequence of a row tile: tiles [0, nA) hold token 0's slots, [nA, nA + nB)
// token 1's, the rest the tree keys.  kind 0 / 1: slots of that token; kind 2: tree keys.
__device__ __forceinline__ void sparse_segment(int j, int nA, int nB, int& kind, int& base) {
    if (j < nA) {
        kind = 0;
        base = j * kBlockN;
    } else if (j < nA + nB) {
        kind = 1;
        base = (j - nA) * kBlockN;
    } else {
        kind = 2;
        base = (j - nA - nB) * kBlockN;
    }
}

// ---- segments: the pieces of work a CTA pair computes ----
// Output of a segment.
constexpr int kOutFinal = 0;      // the whole item: normalised rows into out / lse
constexpr int kOutPartial = 1;    // one split of a per-unit grid: normalised partial into its split slot
constexpr int kOutTwoSplit = 2;   // per-unit grid: two-split or cut unit, merged in the kernel
constexpr int kOutPiece = 3;      // persistent: a piece of an item cut between CTA pairs, merged in the kernel

// KV tiles [t0, t0 + n) of one work item (identical in both CTAs of the pair).
struct Seg {
    int item;          // index into the work list
    int b;             // request
    int T, L, P;       // tree tokens, KV rows and prefix length of the request
    int qbase, ntok;   // first tree token of the row tile, tokens in it (1 or 2)
    int nA, nB;        // sparse: KV tiles of token 0's and token 1's slot lists
    int t0, n;         // first KV tile (of the item's key sequence) and tile count
    int kind;          // kOut*
    int split;         // per-unit grid: split of the item; persistent: 0
    int tail_j;        // per-unit grid, cut item: its compact partial slot; else -1
    bool bad;          // invalid request: no tiles, rows written as out = 0, lse = -inf
};

// Where the next segment comes from.
struct Cursor {
    long long x, end;  // persistent: next position of the pair's share, end of the share
    int item;          // persistent: item holding x
    int round, rounds; // persistent: whole-item rounds handed out, and their number
    int pair;          // persistent: this CTA pair
    bool done;         // per-unit grid: the one segment was handed out
};

template <bool kSparse>
__device__ __forceinline__ void seg_item(const VerifyParams& p, int item, int2 it, Seg& s) {
    s.item = item;
    s.b = it.x;
    s.T = __ldg(p.n_tree + s.b);
    s.L = __ldg(p.seq_lens + s.b);
    s.P = s.L - s.T;
    s.qbase = __ldg(p.q_off + s.b) + kTokensPerTile * it.y;
    s.ntok = min(kTokensPerTile, s.T - kTokensPerTile * it.y);
    s.bad = __ldg(p.req_state + s.b) != 0;
    s.nA = s.nB = 0;
    if constexpr (kSparse) {
        s.nA = (p.topk + kBlockN - 1) / kBlockN;
        s.nB = s.ntok > 1 ? s.nA : 0;
    }
}

// KV tiles of the item's key sequence (0 for an invalid request).
template <bool kSparse>
__device__ __forceinline__ int item_kv_tiles(const Seg& s) {
    return s.bad ? 0 : (kSparse ? s.nA + s.nB + (s.T + kBlockN - 1) / kBlockN : (s.L + kBlockN - 1) / kBlockN);
}

// Per-unit grid: the unit of this CTA pair, from blockIdx.  Regular: one unit
// per (item, blockIdx.y).  With k = *tail_k > 0 the whole items come first,
// then the first parts of the last k items, then their second parts; tail_j
// numbers a cut item among the k.
template <bool kSparse, bool kMerge>
__device__ __forceinline__ bool unit_segment(const VerifyParams& p, int n_items, Seg& s) {
    int item = blockIdx.x >> 1, split = blockIdx.y + p.split_base, nsplit = p.num_splits, share = p.split_share;
    // the unit's work item, loaded before the item count is known (a cut unit of the
    // last round loads its own below): the two round trips overlap
    const int spec = min(item, p.max_items - 1);
    int2 it = spec >= 0 ? p.items[spec] : make_int2(0, 0);
    int tail_j = -1;
    if (p.tail_k != nullptr) {
        const int k = min(min(__ldg(p.tail_k), p.tail_cap), n_items), whole = n_items - k;
        if (k > 0 && item >= whole) {
            const int j = item - whole;
            if (j >= 2 * k) return false;
            tail_j = j % k;
            item = whole + tail_j;
            split = j / k;
            nsplit = 2;
            share = p.tail_share;
        }
    }
    if (item >= n_items) return false;
    if (item != spec) it = p.items[item];
    seg_item<kSparse>(p, item, it, s);
    int t0, t1;
    split_range(item_kv_tiles<kSparse>(s), split, nsplit, share, t0, t1);
    s.t0 = t0;
    s.n = t1 - t0;
    s.split = split;
    s.tail_j = tail_j;
    s.kind = (kMerge && p.merge_cnt != nullptr && nsplit == 2) ? kOutTwoSplit
             : nsplit == 1                                      ? kOutFinal
                                                                : kOutPartial;
    return true;
}

// Persistent schedule: the pair's whole item of the next round, then the next
// item piece of its share [x, end) of the remaining items.
template <bool kSparse>
__device__ __forceinline__ bool share_segment(const VerifyParams& p, int n_items, Cursor& cu, Seg& s) {
    if (cu.round < cu.rounds) {
        const int r = cu.round++;
        const int item = r * p.pairs + ((r & 1) ? p.pairs - 1 - cu.pair : cu.pair);
        seg_item<kSparse>(p, item, p.items[item], s);
        s.t0 = 0;
        s.n = item_kv_tiles<kSparse>(s);
        s.split = 0;
        s.tail_j = -1;
        s.kind = kOutFinal;
        return true;
    }
    if (cu.x >= cu.end || cu.item >= n_items) return false;
    const long long O = __ldg(p.woff + cu.item), E = __ldg(p.woff + cu.item + 1);
    seg_item<kSparse>(p, cu.item, p.items[cu.item], s);
    const long long a = cu.x - O, e = min(cu.end, E) - O;
    const long long nkv = item_kv_tiles<kSparse>(s);
    s.t0 = static_cast<int>(min(a, nkv));
    s.n = static_cast<int>(min(e, nkv)) - s.t0;
    s.split = 0;
    s.tail_j = -1;
    s.kind = (a == 0 && O + e == E) ? kOutFinal : kOutPiece;
    cu.x = O + e;
    ++cu.item;
    return true;
}

// Rows of local tile jj of segment s whose partial scores the two CTAs exchange:
// -1 for all 128, or t for the 64 rows of token t alone.  Sparse tiles of a token's
// slot list are seen by that token's rows only (the other token's rows are masked
// out), so half the scores, 16 KB, make the trip.
template <bool kSparse>
__device__ __forceinline__ int exchange_rows(const Seg& s, int jj) {
    if constexpr (kSparse) {
        int kind, base;
        sparse_segment(s.t0 + jj, s.nA, s.nB, kind, base);
        return kind < 2 ? kind : -1;
    } else {
        return -1;
    }
}
__host__ __device__ constexpr uint32_t exchange_bytes(int rows) { return rows < 0 ? kXBufBytes : kXBufBytes / 2; }

template <bool kSparse, int kSched>
__device__ __forceinline__ bool next_segment(const VerifyParams& p, int n_items, Cursor& cu, Seg& s) {
    if constexpr (kSched == kSchedPersistent) {
        return share_segment<kSparse>(p, n_items, cu, s);
    } else {
        if (cu.done) return false;
        cu.done = true;
        return unit_segment<kSparse, kSched == kSchedMerge>(p, n_items, s);
    }
}

// kSched: see the schedules above (kSchedMerge carries the in-kernel merge code,
// kept out of the plain variant: small launches run every path cold).
template <bool kSparse, int kSched>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kSparse ? kThreadsSparse : kThreads, 1)
mla_verify_kernel(const __grid_constant__ VerifyParams p, const __grid_constant__ CUtensorMap map_lat,
                  const __grid_constant__ CUtensorMap map_rope) {
    constexpr bool kPersistent = kSched == kSchedPersistent;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + kOffCtrl);

    const uint32_t c = cluster_ctarank();
    const uint32_t peer = c ^ 1u;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int pair = blockIdx.x >> 1;

    // ---- set-up: barriers, TMEM, the descriptors' prefetch, the cluster sync ----
    // first_bytes: size of the first incoming partial, posted before the peer can send
    auto setup = [&](uint32_t first_bytes) {
        if (threadIdx.x == 0) {
            for (int s = 0; s < kStages; ++s) {
                mbar_init(&ctl->kv_full[s], kSparse ? kGatherWarps : 1);  // sparse: one arrival per gather warp
                mbar_init(&ctl->kv_empty[s], 1);
                mbar_init(&ctl->kv_fixed[s], 1);
            }
            for (int x = 0; x < 2; ++x) {
                mbar_init(&ctl->p_full[x], kSoftmaxThreads);
                mbar_init(&ctl->pv_done[x], 1);
                ctl->lo_flag[x] = 0;
            }
            for (int k = 0; k < 3; ++k) ctl->tile_flags[k] = 0;
            mbar_init(&ctl->s_full, 1);
            mbar_init(&ctl->s_free, kSoftmaxThreads);
            mbar_init(&ctl->x_full, 1);
            mbar_init(&ctl->x_empty, 1);
            mbar_init(&ctl->q_ready, kSoftmaxThreads);
            mbar_init(&ctl->drain_qk, 1);
            mbar_init(&ctl->drain_pv, 1);
            mbar_init(&ctl->never, 1);
            mbar_init(&ctl->stg_free, 1);
            mbar_init(&ctl->staged, 1);
            for (int w = 0; w < 4; ++w) mbar_init(&ctl->stg_read[w], 1);
            ctl->abort = 0;
            mbar_arrive_expect_tx(&ctl->x_full, first_bytes);
            fence_mbar_init_cluster();
        }
        if (warp == 1) tmem_alloc(&ctl->tmem_base, kTmemCols);
        if (warp == 0 && lane == 0) {
            tma_prefetch_desc(&map_lat);
            tma_prefetch_desc(&map_rope);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        cluster_sync();  // the peer's barriers are initialised before any remote arrive
    };
    // The dense kernel sets up while the prep kernel still runs (its first partial
    // is always a full one); the sparse one needs its first segment for that size.
    if constexpr (!kSparse) setup(kXBufBytes);
    grid_dependency_wait();     // the prep (and slot check) kernels' work list and metadata
    grid_launch_dependents();
    const int n_items = __ldg(p.item_count);

    // ---- the first segment (identical in both CTAs of the pair) ----
    // Every role walks the segments with its own copy of the cursor, which
    // points past the first segment from here on.
    Cursor cu0{};
    if constexpr (kPersistent) {
        cu0.x = __ldg(p.pair_begin + pair);
        cu0.end = __ldg(p.pair_begin + pair + 1);
        cu0.item = __ldg(p.pair_item + pair);
        cu0.rounds = min(__ldg(p.rounds), n_items / max(p.pairs, 1));
        cu0.pair = pair;
    }
    // An exit before the pipeline starts (both CTAs of the pair take it) gives back
    // the TMEM of the dense kernel's early set-up; nothing was issued into it.
    auto release_early = [&]() {
        if constexpr (!kSparse) {
            if (warp == 1) tmem_dealloc(ctl->tmem_base, kTmemCols);
        }
    };
    Seg seg0;
    if (!next_segment<kSparse, kSched>(p, n_items, cu0, seg0)) {
        release_early();   // no work for this pair
        return;
    }

    // rows of this thread (softmax warps only)
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int tok_local = r / kHeads;
    const int head = r % kHeads;
    const bool softmax_warp = warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 4;
    const bool stager_warp = warp >= kStagerWarp0 && warp < kStagerWarp0 + 4;
    const long long out_rows = static_cast<long long>(p.total_q) * kHeads;

    // ---- two-split merge (per-unit grid; softmax warps) ----
    // With exactly two KV splits (or a cut unit) the two work units of a row
    // tile meet per CTA half c: the first to arrive writes its normalised
    // partial and lse and marks them written; the second waits for the mark,
    // copies the other split's rows of its half into shared memory in one batch
    // of async copies (the stages, q rope and receive buffer are free by then:
    // a unit is the CTA's only segment), and writes the merged rows, weighting
    // the splits by their lse and adding them in split order, so the result
    // does not depend on which unit arrives second.  Rows leave through the
    // warp's 4 KB tile of the staging buffer in whole 128-byte lines.  own(part, v)
    // fills v[32] with this unit's normalised columns 32 part .. 32 part + 31 of
    // the thread's row; lse_own is its lse.
    auto two_split_merge = [&](const Seg& sg, auto&& own, float lse_own) {
        const bool row_valid = tok_local < sg.ntok;
        const long long grow = static_cast<long long>(sg.qbase + tok_local) * kHeads + head;
        // rows of this tile in the partial buffers: its global rows, or the cut item's compact slot
        const long long part_row0 =
            sg.tail_j >= 0 ? static_cast<long long>(sg.tail_j) * kRows : static_cast<long long>(sg.qbase) * kHeads;
        const long long part_rows = sg.tail_j >= 0 ? static_cast<long long>(p.tail_cap) * kRows : out_rows;
        const int split = sg.split;
        int32_t* cnt = p.merge_cnt + (sg.item * 2 + static_cast<int>(c)) * 2;
        float* lse2 = p.part_lse + static_cast<long long>(c) * 2 * part_rows;   // [half][split][row]
        const long long prow = part_row0 + r, pwrow = part_row0 + q4 * 32;   // this row / the warp's first
        const uint32_t ebuf = smem_u32(smem + kOffStaging) + q4 * 4096;
        const long long wrow = grow - lane;   // the warp's first row
        named_bar_sync(4, kSoftmaxThreads);
        if (r == 0) ctl->merge_role = atomicAdd(cnt, 1);
        named_bar_sync(4, kSoftmaxThreads);
        const int role = *reinterpret_cast<volatile int*>(&ctl->merge_role);
        if (role == 0) {
            float* wdst = p.part_out + (static_cast<long long>(split) * part_rows + pwrow) * kDLatent + kDLatentHalf * c;
            for (int part = 0; part < kDLatentHalf / 32; ++part) {
                float v[32];
                own(part, v);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    st_shared_v4(ebuf + lane * 128 + ((u ^ (lane & 7)) << 4), v[4 * u], v[4 * u + 1], v[4 * u + 2],
                                 v[4 * u + 3]);
                __syncwarp();
                if (row_valid) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int row = 4 * i + (lane >> 3), u = lane & 7;
                        *reinterpret_cast<float4*>(wdst + static_cast<long long>(row) * kDLatent + 32 * part + 4 * u) =
                            ld_shared_v4(ebuf + row * 128 + ((u ^ (row & 7)) << 4));
                    }
                }
                __syncwarp();
            }
            if (row_valid) lse2[split * part_rows + prow] = lse_own;
            __threadfence();
            named_bar_sync(4, kSoftmaxThreads);
            const bool skip_mark = fault_kind() == 2 && sg.item == 0 && c == 0;
            if (r == 0 && !skip_mark) atomicExch(cnt + 1, 1);
            return;
        }
        if (r == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (atomicAdd(cnt + 1, 0) == 0) {
                if (globaltimer_ns() - t0 > p.timeout_ns) {
                    raise_status(p.status, kStatusTimeout);
                    break;
                }
                __nanosleep(100);
            }
        }
        named_bar_sync(4, kSoftmaxThreads);
        __threadfence();
        const int other = split ^ 1;
        // the other split's 32 rows of this warp, 1 KB each: unit u of row i at u ^ (i & 7)
        const uint32_t obuf = smem_u32(smem + kOffStages) + q4 * (32 * 1024);
        if (row_valid) {
            const float* wsrc =
                p.part_out + (static_cast<long long>(other) * part_rows + pwrow) * kDLatent + kDLatentHalf * c;
#pragma unroll 4
            for (int i = 0; i < 32; ++i) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int u = lane + 32 * h;
                    cp_async_16(obuf + i * 1024 + ((u ^ (i & 7)) << 4), wsrc + static_cast<long long>(i) * kDLatent + 4 * u);
                }
            }
            cp_async_commit();
            cp_async_wait<0>();
        }
        __syncwarp();
        const float lse_oth = row_valid ? lse2[other * part_rows + prow] : -INFINITY;
        const float l0 = split == 0 ? lse_own : lse_oth, l1 = split == 0 ? lse_oth : lse_own;
        const float m = fmaxf(l0, l1);
        float lse_tot = -INFINITY, w0 = 0.f, w1 = 0.f;
        if (m != -INFINITY) {
            lse_tot = m + __logf(__expf(l0 - m) + __expf(l1 - m));
            w0 = l0 == -INFINITY ? 0.f : __expf(l0 - lse_tot);
            w1 = l1 == -INFINITY ? 0.f : __expf(l1 - lse_tot);
        }
        float* wdst = p.out + wrow * kDLatent + kDLatentHalf * c;
        for (int part = 0; part < kDLatentHalf / 32; ++part) {
            float v[32];
            own(part, v);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int uu = 8 * part + u;
                const float4 t = ld_shared_v4(obuf + lane * 1024 + ((uu ^ (lane & 7)) << 4));
                const float o4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a0 = split == 0 ? v[4 * u + e] : o4[e], a1 = split == 0 ? o4[e] : v[4 * u + e];
                    v[4 * u + e] = w0 * a0 + w1 * a1;
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                st_shared_v4(ebuf + lane * 128 + ((u ^ (lane & 7)) << 4), v[4 * u], v[4 * u + 1], v[4 * u + 2],
                             v[4 * u + 3]);
            __syncwarp();
            if (row_valid) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = 4 * i + (lane >> 3), u = lane & 7;
                    *reinterpret_cast<float4*>(wdst + static_cast<long long>(row) * kDLatent + 32 * part + 4 * u) =
                        ld_shared_v4(ebuf + row * 128 + ((u ^ (row & 7)) << 4));
                }
            }
            __syncwarp();
        }
        if (row_valid && c == 0) p.lse[grow] = lse_tot;
    };

    if constexpr (!kPersistent) {
        if (seg0.n <= 0) {
            // Empty split or invalid request: normalised output 0, lse -inf.
            if (seg0.kind == kOutTwoSplit) {
                if (softmax_warp)
                    two_split_merge(seg0, [](int, float* v) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) v[k] = 0.f;
                    }, -INFINITY);
                release_early();
                return;
            }
            if (softmax_warp && tok_local < seg0.ntok) {
                const long long grow = static_cast<long long>(seg0.qbase + tok_local) * kHeads + head;
                const long long slot_row = static_cast<long long>(seg0.split - p.split_base) * out_rows + grow;
                float* dst = seg0.kind == kOutFinal ? p.out + grow * kDLatent + kDLatentHalf * c
                                                    : p.part_out + slot_row * kDLatent + kDLatentHalf * c;
                for (int d = 0; d < kDLatentHalf; d += 4)
                    *reinterpret_cast<float4*>(dst + d) = make_float4(0.f, 0.f, 0.f, 0.f);
                if (c == 0) {
                    if (seg0.kind == kOutFinal) p.lse[grow] = -INFINITY;
                    else p.part_lse[slot_row] = -INFINITY;
                }
            }
            release_early();
            return;
        }
    }

    // Sparse gather warps: lane l of gather warp w handles key 4 * gather_group0(w) + l
    // of every tile (lanes past the warp's keys none).  The slot values of the first
    // segment's first tiles are loaded before the set-up below.
    [[maybe_unused]] const bool gather_warp = kSparse && (warp == 0 || warp == kPvWarp || warp == kGatherWarp2);
    static_assert(kGatherWarp2 < kSoftmaxWarp0 && kPvWarp < kSoftmaxWarp0, "producer roles in warpgroup 0");
    [[maybe_unused]] const int gw = warp == 0 ? 0 : warp == kPvWarp ? 1 : 2;
    [[maybe_unused]] const int key0 = 4 * gather_group0(gw);
    [[maybe_unused]] const int nkeys = 4 * gather_group0(gw + 1) - key0;
    [[maybe_unused]] const int key = key0 + lane;
    // raw slot value of this lane's key in local tile jj of segment sg (a KV position, -1 for none)
    [[maybe_unused]] auto slot_raw = [&](const Seg& sg, int jj) -> int {
        if (jj >= sg.n || lane >= nkeys) return -1;
        int kind, base;
        sparse_segment(sg.t0 + jj, sg.nA, sg.nB, kind, base);
        if (kind == 2) return base + key < sg.T ? sg.P + base + key : -1;
        return base + key < p.topk
                   ? __ldg(p.topk_idx + static_cast<long long>(sg.qbase + kind) * p.topk + base + key)
                   : -1;
    };
    [[maybe_unused]] int pre_raw[3] = {-1, -1, -1};
    if constexpr (kSparse) {
        if (gather_warp) {
#pragma unroll
            for (int t = 0; t < 3; ++t) pre_raw[t] = slot_raw(seg0, t);
        }
    }

    // Softmax warps: the query copies of a segment (global -> shared), in two rounds
    // of 128 features per row through the warp's 8 KB of the staging buffer (which
    // nothing else uses then); the rows move into TMEM after each round.  Each
    // instruction copies two 256-byte row pieces (unit u of row i at u ^ (i & 15));
    // the rope half goes straight into its swizzled slot with the first round.  The
    // dense kernel starts the first segment's first round before its work item's
    // KV is known; the sparse one later, so that the copies do not delay the first
    // tile's slot and block-table lookups, which gate its first QK.
    auto issue_q_copies = [&](const Seg& sg, int h) {
        const uint32_t qbuf = smem_u32(smem + kOffStaging) + q4 * 8192;
        const uint32_t qrope = smem_u32(smem + kOffQRope);
        const long long row0 = static_cast<long long>(sg.qbase) * kHeads + q4 * 32;
        const uint8_t* lat =
            reinterpret_cast<const uint8_t*>(p.q_lat) + (row0 * kDLatent + kDLatentHalf * c) * 2 + 256 * h;
#pragma unroll 8
        for (int i = 0; i < 16; ++i) {
            const int row = 2 * i + (lane >> 4), u = lane & 15;
            cp_async_16(qbuf + row * 256 + ((u ^ (row & 15)) << 4), lat + static_cast<long long>(row) * kDLatent * 2 + 16 * u);
        }
        if (h == 0) {
            const uint8_t* rope = reinterpret_cast<const uint8_t*>(p.q_rope) + (row0 * kDRope + kDRopeHalf * c) * 2;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = 8 * i + (lane >> 2), u = lane & 3, rr = q4 * 32 + row;
                cp_async_16(qrope + rr * 64 + ((u ^ ((rr >> 1) & 3)) << 4),
                            rope + static_cast<long long>(row) * kDRope * 2 + 16 * u);
            }
        }
        cp_async_commit();
    };
    if (!kSparse && softmax_warp && tok_local < seg0.ntok && seg0.n > 0) issue_q_copies(seg0, 0);

    // ---- set-up of the sparse kernel ----
    if constexpr (kSparse) {
        // byte count of the first incoming partial (the first tile of the first segment with tiles)
        uint32_t first_bytes = kXBufBytes;
        if (threadIdx.x == 0) {
            Cursor cf = cu0;
            Seg sf = seg0;
            bool have = true;
            while (have && sf.n <= 0) have = next_segment<kSparse, kSched>(p, n_items, cf, sf);
            if (have) first_bytes = exchange_bytes(exchange_rows<kSparse>(sf, 0));
        }
        setup(first_bytes);
    }
    const uint32_t tmem = ctl->tmem_base;

    volatile int* abort_flag = &ctl->abort;
    const uint64_t lim = p.timeout_ns;
    const uint32_t stage0 = smem_u32(smem + kOffStages);
    const uint32_t qrope_addr = smem_u32(smem + kOffQRope);

    // The roles below walk the same segments; tile i of the CTA's whole stream
    // (all segments) uses KV stage i % kStages and P barriers i & 1.  Each
    // warpgroup's branch starts with its register reallocation: warpgroup 1 (softmax)
    // takes the registers that warpgroups 0 and 2 give back.
    if (warp < kSoftmaxWarp0) {
        setmaxnreg_dec<kRegsOther>();
        if (warp == 0 || gather_warp) {
            // ================= TMA producer(s) =================
            // Dense: warp 0 loads one 64-row box per chunk of a tile.  Sparse: three
            // gather warps own 24, 20 and 20 keys of every tile (TMA instructions
            // issued by the lanes of one warp are serialised, so more warps shorten
            // the issue time).  Lane l looks up the cache row of the warp's key l;
            // lane g then loads the warp's keys 4g .. 4g + 3 with four-row gathers
            // (one box row per key), and each warp posts its share of the tile's bytes
            // on the stage barrier, so a gathered tile completes exactly like a dense one.  Empty
            // slots name a row past the end of the cache and read as zeros.  The
            // lookups run ahead of the copies: before tile jj waits for its stage,
            // the row of tile jj + 1 is completed and prefetched into L2, and the
            // block-table entry of tile jj + 2 and the slot value of tile jj + 3 are
            // loaded; each loaded value is first used one tile later.
            const uint64_t policy = l2_policy_evict_last();
            bool ok = true;
            int issued = 0;   // tiles issued into the ring
            Cursor cu = cu0;
            Seg sg = seg0;
            for (bool have = true, first = true; have && ok;
                 have = next_segment<kSparse, kSched>(p, n_items, cu, sg), first = false) {
                const int n = sg.n;
                if (n <= 0) continue;
                // checked position of a raw slot value of tile jt (slot positions the check
                // kernel rejected, >= P, are dropped); its block-table load is issued, not waited on
                [[maybe_unused]] auto translate = [&](int jt, int raw, int& tpos, int& page) {
                    int kind, base;
                    sparse_segment(sg.t0 + jt, sg.nA, sg.nB, kind, base);
                    tpos = (raw < 0 || (kind != 2 && raw >= sg.P)) ? -1 : raw;
                    page = tpos >= 0 ? __ldg(p.block_table + static_cast<long long>(sg.b) * p.max_pages + tpos / p.page_size)
                                     : -1;
                };
                // cache row from a checked position and its (landed) block-table entry
                [[maybe_unused]] auto row_of = [&](int tpos, int page) -> int {
                    if (tpos < 0) return -1;
                    if (page < 0 || page >= p.num_pages) {
                        raise_status(p.status, kStatusBadBlock);
                        return -1;
                    }
                    return page * p.page_size + tpos % p.page_size;
                };
                // this CTA's 576 bytes of a row span five 128-byte lines
                [[maybe_unused]] auto prefetch_row = [&](int row) {
                    if (row < 0) return;
                    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.kv) + static_cast<long long>(row) * (kDqk * 2);
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) prefetch_l2(src + kDLatentHalf * 2 * c + 128 * ch);
                    prefetch_l2(src + kDLatent * 2 + kDRopeHalf * 2 * c);
                };
                [[maybe_unused]] int raw = -1;   // slot value (tile jj + 3)
                [[maybe_unused]] int tpos = -1;  // checked position (tile jj + 2) ...
                [[maybe_unused]] int page = -1;  // ... and its block-table entry, in flight
                [[maybe_unused]] int cur = -1;   // cache row of tile jj, -1 for an empty slot
                [[maybe_unused]] const int oob_row = p.num_pages * p.page_size;
                [[maybe_unused]] int nxt = -1;   // cache row of tile jj + 1
                // dense: the block-table entry of the next tile, loaded one tile ahead so that
                // a freed stage is refilled without a round trip to the table
                [[maybe_unused]] int pg_next = -1;
                [[maybe_unused]] auto page_entry = [&](int jt) {
                    return __ldg(p.block_table + static_cast<long long>(sg.b) * p.max_pages +
                                 (sg.t0 + jt) * kBlockN / p.page_size);
                };
                if constexpr (!kSparse) {
                    if (lane == 0) pg_next = page_entry(0);
                }
                if constexpr (kSparse) {
                    // the first segment's slot values of tiles 0..2 were loaded before the
                    // set-up; the block-table entries of tiles 0 and 1 are one more round trip
                    if (!first) {
#pragma unroll
                        for (int t = 0; t < 3; ++t) pre_raw[t] = slot_raw(sg, t);
                    }
                    raw = pre_raw[2];
                    int tpos0, page0;
                    translate(0, pre_raw[0], tpos0, page0);
                    translate(1, pre_raw[1], tpos, page);
                    cur = row_of(tpos0, page0);
                    prefetch_row(cur);
                }
                for (int jj = 0; jj < n && ok; ++jj) {
                    const int gi = issued;
                    const int st = gi % kStages;
                    [[maybe_unused]] const int pg = pg_next;
                    if constexpr (!kSparse) {
                        if (lane == 0 && jj + 1 < n) pg_next = page_entry(jj + 1);
                    }
                    if constexpr (kSparse) {
                        if (jj + 1 < n) {
                            nxt = row_of(tpos, page);
                            prefetch_row(nxt);
                        }
                        if (jj + 2 < n) {
                            translate(jj + 2, raw, tpos, page);
                            raw = slot_raw(sg, jj + 3);
                        }
                    }
                    if (gi >= kStages) {
                        ok = __all_sync(0xffffffffu, mbar_wait(&ctl->kv_empty[st], ((gi / kStages) - 1) & 1, abort_flag, lim));
                        if (!ok) break;
                    }
                    uint8_t* dst = smem + kOffStages + st * kStageBytes;
                    if constexpr (kSparse) {
                        const uint32_t mask = __ballot_sync(0xffffffffu, cur >= 0);
                        int y[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int v = __shfl_sync(0xffffffffu, cur, (4 * lane + t) & 31);
                            y[t] = v >= 0 ? v : oob_row;
                        }
                        if (lane == 0) {
                            ctl->slot_mask[st][gw] = mask;
                            // this warp's share of the stage, 576 bytes per key; releases the mask with the tile
                            mbar_arrive_expect_tx(&ctl->kv_full[st], static_cast<uint32_t>(nkeys) * (kStageBytes / kBlockN));
                        }
                        __syncwarp();
                        if (lane < nkeys / 4) {
                            const int g = key0 / 4 + lane;  // keys 4g .. 4g + 3
#pragma unroll
                            for (int ch = 0; ch < 4; ++ch)
                                tma_gather4(dst + ch * kChunkBytes + 4 * g * 128, &map_lat, &ctl->kv_full[st],
                                            kDLatentHalf * static_cast<int>(c) + 64 * ch, y[0], y[1], y[2], y[3], policy);
                            tma_gather4(dst + 4 * kChunkBytes + 4 * g * 64, &map_rope, &ctl->kv_full[st],
                                        kDLatent + kDRopeHalf * static_cast<int>(c), y[0], y[1], y[2], y[3], policy);
                        }
                        cur = nxt;
                        ++issued;
                        __syncwarp();
                    } else {
                        const int kpos = (sg.t0 + jj) * kBlockN;
                        if (lane == 0) {
                            if (pg < 0 || pg >= p.num_pages) raise_status(p.status, kStatusBadBlock);
                            // out-of-range pages read as zeros (TMA out-of-bounds fill); the status reports them
                            const int row = pg * p.page_size + (kpos % p.page_size);
                            mbar_arrive_expect_tx(&ctl->kv_full[st], kStageBytes);
                            for (int ch = 0; ch < 4; ++ch)
                                tma_load_2d(dst + ch * kChunkBytes, &map_lat, &ctl->kv_full[st],
                                            kDLatentHalf * static_cast<int>(c) + 64 * ch, row, policy);
                            tma_load_2d(dst + 4 * kChunkBytes, &map_rope, &ctl->kv_full[st],
                                        kDLatent + kDRopeHalf * static_cast<int>(c), row, policy);
                        }
                        ++issued;
                        __syncwarp();
                        if (kpos + kBlockN > sg.L) {
                            // Last, partial tile: zero the rows past seq_len so that masked
                            // keys multiply finite values in PV.
                            ok = __all_sync(0xffffffffu, mbar_wait(&ctl->kv_full[st], (gi / kStages) & 1, abort_flag, lim));
                            if (!ok) break;
                            const int kvalid = sg.L - kpos;
                            uint8_t* base = smem + kOffStages + st * kStageBytes;
                            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                            for (int rr = kvalid + lane / 8; rr < kBlockN; rr += 4) {
                                const int u = lane % 8;  // 16-byte unit of the row
                                for (int ch = 0; ch < 4; ++ch)
                                    *reinterpret_cast<float4*>(base + ch * kChunkBytes + rr * 128 + u * 16) = z;
                                if (u < 4) *reinterpret_cast<float4*>(base + 4 * kChunkBytes + rr * 64 + u * 16) = z;
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&ctl->kv_fixed[st]);
                        }
                    }
                }
            }
            if (!ok) {
                if (lane == 0) raise_status(p.status, kStatusTimeout);
                *abort_flag = 1;
            }
            // Do not leave the CTA with bulk copies in flight.
            const int zero = 0;
            for (int st = 0; st < kStages && st < issued; ++st) {
                const int last = st + ((issued - 1 - st) / kStages) * kStages;  // last tile issued into stage st
                mbar_wait(&ctl->kv_full[st], (last / kStages) & 1, &zero, lim);
            }
        } else if (warp == 1) {
            // ================= QK issuer (sparse: also PV) =================
            const uint32_t idesc_qk = idesc_bf16(128, kBlockN, false, false);
            const uint64_t aq_rope = smem_desc(qrope_addr, 16, 512, kSwizzle64B);
            // Sparse: the PV warp gathers KV rows, so this warp issues PV of tile gi (the
            // segment's i-th) once its P is in TMEM, two tiles behind QK (P of tile gi is
            // ready before the S columns are free for tile gi + 2, so the wait does not
            // hold QK back), and the segment's last two after its last QK.  Returns false
            // if the wait ran out.
            [[maybe_unused]] auto issue_pv = [&](int gi, int i) -> bool {
                const int x = gi & 1;
                const int st = gi % kStages;
                if (!__all_sync(0xffffffffu, mbar_wait(&ctl->p_full[x], (gi >> 1) & 1, abort_flag, lim))) return false;
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t idesc_pv = idesc_bf16(128, kDLatentHalf, false, true);
                    const int lo = *reinterpret_cast<volatile int*>(&ctl->lo_flag[x]);
                    const uint64_t bv = smem_desc(stage0 + st * kStageBytes, kChunkBytes, 1024, kSwizzle128B);
#pragma unroll
                    for (int kk = 0; kk < kBlockN / 16; ++kk)
                        mma_ts(tmem + kTmO, tmem + kTmP + 8 * kk, desc_advance(bv, kk * 2048), idesc_pv,
                               (i > 0 || kk > 0) ? 1u : 0u);
                    if (lo) {
#pragma unroll
                        for (int kk = 0; kk < kBlockN / 16; ++kk)
                            mma_ts(tmem + kTmO, tmem + kTmPLo + 8 * kk, desc_advance(bv, kk * 2048), idesc_pv, 1u);
                    }
                    mma_commit(&ctl->pv_done[x]);
                    mma_commit(&ctl->kv_empty[st]);
                }
                __syncwarp();
                return true;
            };
            bool ok = true;
            int g = 0;              // tiles of the earlier segments
            int segs = 0;           // segments with tiles so far (phases of q_ready)
            uint32_t fixpar = 0;    // bit st: parity of the next phase of kv_fixed[st]
            Cursor cu = cu0;
            Seg sg = seg0;
            for (bool have = true; have && ok; have = next_segment<kSparse, kSched>(p, n_items, cu, sg)) {
                const int n = sg.n;
                if (n <= 0) continue;
                ok = __all_sync(0xffffffffu, mbar_wait(&ctl->q_ready, segs & 1, abort_flag, lim));
                ++segs;
                if (!ok) break;
                tc_fence_after();
                for (int jj = 0; jj < n; ++jj) {
                    const int gi = g + jj;
                    const int st = gi % kStages;
                    const bool tail = !kSparse && (sg.t0 + jj) * kBlockN + kBlockN > sg.L;
                    const bool inject = fault_kind() == 1 && sg.item == 0 && sg.split == 0 && c == 0 && jj == 1;
                    if (inject) {
                        ok = mbar_wait(&ctl->never, 0, abort_flag, lim);
                    } else if (tail) {
                        ok = mbar_wait(&ctl->kv_fixed[st], (fixpar >> st) & 1u, abort_flag, lim);
                        fixpar ^= 1u << st;
                    } else {
                        ok = mbar_wait(&ctl->kv_full[st], (gi / kStages) & 1, abort_flag, lim);
                    }
                    // the S columns held tile gi - 1; the softmax threads have read them out
                    if (ok && gi >= 1) ok = mbar_wait(&ctl->s_free, (gi - 1) & 1, abort_flag, lim);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t sb = stage0 + st * kStageBytes;
                        const uint32_t dS = tmem + kTmS;
                        // one base descriptor per operand; the k-steps add constant byte offsets
                        const uint64_t bk = smem_desc(sb, 16, 1024, kSwizzle128B);
                        const uint64_t br = smem_desc(sb + 4 * kChunkBytes, 16, 512, kSwizzle64B);
#pragma unroll
                        for (int k = 0; k < kDLatentHalf / 16; ++k)
                            mma_ts(dS, tmem + kTmQ + 8 * k, desc_advance(bk, (k >> 2) * kChunkBytes + (k & 3) * 32),
                                   idesc_qk, k > 0 ? 1u : 0u);
#pragma unroll
                        for (int k = 0; k < kDRopeHalf / 16; ++k)
                            mma_ss(dS, desc_advance(aq_rope, k * 32), desc_advance(br, k * 32), idesc_qk, 1u);
                        mma_commit(&ctl->s_full);
                    }
                    __syncwarp();
                    if constexpr (kSparse) {
                        if (jj > 1 && !issue_pv(gi - 2, jj - 2)) {
                            ok = false;
                            break;
                        }
                    }
                }
                if constexpr (kSparse) {
                    for (int i = n > 1 ? n - 2 : 0; i < n && ok; ++i) ok = issue_pv(g + i, i);
                }
                g += n;
            }
            if (!ok) {
                if (lane == 0) raise_status(p.status, kStatusTimeout);
                *abort_flag = 1;
            }
            // Wait until every MMA issued by this warp has finished before TMEM is released.
            const int zero = 0;
            if (lane == 0) mma_commit(&ctl->drain_qk);
            __syncwarp();
            mbar_wait(&ctl->drain_qk, 0, &zero, lim);
        } else if (warp == kPvWarp) {
            // ================= PV issuer: O[:, half c] += P * V (P in TMEM) =================
            const uint32_t idesc_pv = idesc_bf16(128, kDLatentHalf, false, true);
            bool ok = true;
            int g = 0;
            Cursor cu = cu0;
            Seg sg = seg0;
            for (bool have = true; have && ok; have = next_segment<kSparse, kSched>(p, n_items, cu, sg)) {
                const int n = sg.n;
                if (n <= 0) continue;
                for (int i = 0; i < n && ok; ++i) {
                    const int gi = g + i;
                    const int x = gi & 1;
                    const int st = gi % kStages;
                    ok = __all_sync(0xffffffffu, mbar_wait(&ctl->p_full[x], (gi >> 1) & 1, abort_flag, lim));
                    if (!ok) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const int lo = *reinterpret_cast<volatile int*>(&ctl->lo_flag[x]);
                        const uint64_t bv = smem_desc(stage0 + st * kStageBytes, kChunkBytes, 1024, kSwizzle128B);
#pragma unroll
                        for (int kk = 0; kk < kBlockN / 16; ++kk)
                            mma_ts(tmem + kTmO, tmem + kTmP + 8 * kk, desc_advance(bv, kk * 2048), idesc_pv,
                                   (i > 0 || kk > 0) ? 1u : 0u);
                        if (lo) {
#pragma unroll
                            for (int kk = 0; kk < kBlockN / 16; ++kk)
                                mma_ts(tmem + kTmO, tmem + kTmPLo + 8 * kk, desc_advance(bv, kk * 2048), idesc_pv, 1u);
                        }
                        mma_commit(&ctl->pv_done[x]);
                        mma_commit(&ctl->kv_empty[st]);
                    }
                    __syncwarp();
                }
                g += n;
            }
            if (!ok) {
                if (lane == 0) raise_status(p.status, kStatusTimeout);
                *abort_flag = 1;
            }
            const int zero = 0;
            if (lane == 0) mma_commit(&ctl->drain_pv);
            __syncwarp();
            mbar_wait(&ctl->drain_pv, 0, &zero, lim);
        }
    } else if (softmax_warp) {
        setmaxnreg_inc<kRegsSoftmax>();
        // ================= softmax / epilogue (thread = row) =================
        const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
        const uint32_t trow = tmem + lane_base;
        const uint32_t xbuf_local = smem_u32(smem + kOffXBuf);
        [[maybe_unused]] const uint32_t vis_addr = smem_u32(smem + kOffVis) + r * 16;   // this row's tail-tile masks
        const uint32_t stg_local = smem_u32(smem + kOffStaging);
        const uint32_t rowbase = stg_local + r * (kBlockN * 4);       // this row in the staging buffer
        const uint32_t peerbase = xbuf_local + r * (kBlockN * 4);     // this row in the receive buffer
        const uint32_t qbuf = stg_local + q4 * 8192;                  // this warp's 8 KB of the staging buffer (q)
        const uint32_t ebuf = stg_local + q4 * 4096;                  // this warp's 4 KB output tile
        const uint32_t mbuf = stg_local + 16384 + q4 * 4096;          // persistent merge: other pieces' rows
        int posted = 1;    // incoming partials whose byte count is posted (thread r == 0)
        int consumed = 0;  // incoming partials waited for (thread r == 0)
        bool ok = true;
        int g = 0;         // tiles of the earlier segments (sent and received partials)
        Cursor cu = cu0;
        Seg sg = seg0;


        // ---- persistent: merge of an item cut between CTA pairs ----
        // The pieces of item sg.item are the non-empty shares of pairs q_first,
        // q_first + 1, ... that start before the item's end; piece of pair q has
        // partial slot 2q (the first segment of the pair) or 2q + 1 (its last).
        // Per CTA half, the first pieces to finish write their normalised partial
        // and lse and count themselves written; the last to arrive waits for the
        // others, then sums w_k * o_k over the pieces in piece order (w_k from
        // the lse of all pieces) into TMEM columns [256, 512), free in an
        // epilogue, reading the other pieces' rows through the staging and P
        // buffers (16 KB per warp, half a row at a time), and writes the rows.
        // own(part, v): this piece's normalised columns; sent: partials this CTA
        // has shipped so far (the staging buffer is reused once the last landed).
        // Every term is rounded the same way whichever piece merges (explicit
        // fused multiply-adds), so the result does not depend on arrival order.
        auto piece_merge = [&](auto&& own, float lse_own, int sent) {
            const bool row_valid = tok_local < sg.ntok;
            const long long grow = static_cast<long long>(sg.qbase + tok_local) * kHeads + head;
            const long long O = __ldg(p.woff + sg.item), E = __ldg(p.woff + sg.item + 1);
            const int q_first = __ldg(p.item_first_pair + sg.item);
            int np = 0;
            for (int q = q_first; q < p.pairs; ++q) {
                const long long b0 = __ldg(p.pair_begin + q);
                if (b0 >= E) break;
                np += __ldg(p.pair_begin + q + 1) > b0 ? 1 : 0;
            }
            auto slot_of = [&](int q) { return 2 * q + (__ldg(p.pair_begin + q) >= O ? 0 : 1); };
            int32_t* cnt = p.merge_cnt + (sg.item * 2 + static_cast<int>(c)) * 2;
            named_bar_sync(4, kSoftmaxThreads);
            if (r == 0) ctl->merge_role = atomicAdd(cnt, 1);
            named_bar_sync(4, kSoftmaxThreads);
            const int role = *reinterpret_cast<volatile int*>(&ctl->merge_role);
            if (role < np - 1) {
                const int slot = slot_of(pair);
                float* wdst = p.part_out + (static_cast<long long>(slot) * kRows + q4 * 32) * kDLatent + kDLatentHalf * c;
                for (int part = 0; part < kDLatentHalf / 32; ++part) {
                    float v[32];
                    own(part, v);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        st_shared_v4(ebuf + lane * 128 + ((u ^ (lane & 7)) << 4), v[4 * u], v[4 * u + 1],
                                     v[4 * u + 2], v[4 * u + 3]);
                    __syncwarp();
                    if (row_valid) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int row = 4 * i + (lane >> 3), u = lane & 7;
                            *reinterpret_cast<float4*>(wdst + static_cast<long long>(row) * kDLatent + 32 * part + 4 * u) =
                                ld_shared_v4(ebuf + row * 128 + ((u ^ (row & 7)) << 4));
                        }
                    }
                    __syncwarp();
                }
                if (row_valid) p.part_lse[(static_cast<long long>(slot) * 2 + c) * kRows + r] = lse_own;
                __threadfence();
                named_bar_sync(4, kSoftmaxThreads);
                const bool skip_mark = fault_kind() == 4 && c == 0;
                if (r == 0 && !skip_mark) atomicAdd(cnt + 1, 1);
                return;
            }
            if (r == 0) {
                const uint64_t t0 = globaltimer_ns();
                while (atomicAdd(cnt + 1, 0) < np - 1) {
                    if (globaltimer_ns() - t0 > p.timeout_ns) {
                        raise_status(p.status, kStatusTimeout);
                        break;
                    }
                    __nanosleep(100);
                }
            }
            named_bar_sync(4, kSoftmaxThreads);
            __threadfence();
            // lse of the merged row: log-sum-exp over the pieces' lse
            auto lse_of = [&](int q) -> float {
                if (q == pair) return lse_own;
                return row_valid ? __ldcg(p.part_lse + (static_cast<long long>(slot_of(q)) * 2 + c) * kRows + r)
                                 : -INFINITY;
            };
            float m = -INFINITY;
            for (int q = q_first, k = 0; k < np; ++q) {
                if (__ldg(p.pair_begin + q + 1) <= __ldg(p.pair_begin + q)) continue;
                m = fmaxf(m, lse_of(q));
                ++k;
            }
            float lse_tot = -INFINITY;
            if (m != -INFINITY) {
                float sum = 0.f;
                for (int q = q_first, k = 0; k < np; ++q) {
                    if (__ldg(p.pair_begin + q + 1) <= __ldg(p.pair_begin + q)) continue;
                    const float lk = lse_of(q);
                    sum += lk == -INFINITY ? 0.f : __expf(lk - m);
                    ++k;
                }
                lse_tot = m + __logf(sum);
            }
            // the staging buffer is the source of this CTA's last partial-score copy until it landed
            if (sent > 0) mbar_wait<true>(&ctl->stg_free, (sent - 1) & 1, abort_flag, lim);
            for (int q = q_first, k = 0; k < np; ++q) {
                if (__ldg(p.pair_begin + q + 1) <= __ldg(p.pair_begin + q)) continue;
                const float lk = lse_of(q);
                const float w = (lk == -INFINITY || lse_tot == -INFINITY) ? 0.f : __expf(lk - lse_tot);
                if (row_valid) {   // warp-uniform: a warp's 32 rows belong to one token
                    if (q == pair) {
                        for (int part = 0; part < kDLatentHalf / 32; ++part) {
                            float v[32];
                            own(part, v);
                            uint32_t a[32];
                            if (k > 0) {
                                tmem_ld32(trow + kTmAcc + 32 * part, a);
                                tmem_wait_ld();
                            }
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                a[e] = __float_as_uint(k > 0 ? __fmaf_rn(w, v[e], __uint_as_float(a[e])) : __fmul_rn(w, v[e]));
                            tmem_st32(trow + kTmAcc + 32 * part, a);
                        }
                    } else {
                        const float* src = p.part_out + (static_cast<long long>(slot_of(q)) * kRows + q4 * 32) * kDLatent +
                                           kDLatentHalf * c;
                        for (int part = 0; part < kDLatentHalf / 32; ++part) {
                            // 32 rows x 32 columns: unit u of row i at u ^ (i & 7)
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int row = 4 * i + (lane >> 3), u = lane & 7;
                                cp_async_16(mbuf + row * 128 + ((u ^ (row & 7)) << 4),
                                            src + static_cast<long long>(row) * kDLatent + 32 * part + 4 * u);
                            }
                            cp_async_commit();
                            cp_async_wait<0>();
                            __syncwarp();
                            {
                                uint32_t a[32];
                                if (k > 0) {
                                    tmem_ld32(trow + kTmAcc + 32 * part, a);
                                    tmem_wait_ld();
                                }
#pragma unroll
                                for (int u = 0; u < 8; ++u) {
                                    const float4 t = ld_shared_v4(mbuf + lane * 128 + ((u ^ (lane & 7)) << 4));
                                    const float o4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const int idx = 4 * u + e;
                                        a[idx] = __float_as_uint(k > 0 ? __fmaf_rn(w, o4[e], __uint_as_float(a[idx]))
                                                                       : __fmul_rn(w, o4[e]));
                                    }
                                }
                                tmem_st32(trow + kTmAcc + 32 * part, a);
                            }
                            __syncwarp();
                        }
                    }
                    tmem_wait_st();
                }
                ++k;
            }
            // the merged rows leave through the warp's 4 KB tile in whole 128-byte lines
            named_bar_sync(4, kSoftmaxThreads);
            if (row_valid) {
                float* wdst = p.out + (grow - lane) * kDLatent + kDLatentHalf * c;
                for (int part = 0; part < kDLatentHalf / 32; ++part) {
                    uint32_t a[32];
                    tmem_ld32(trow + kTmAcc + 32 * part, a);
                    tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        st_shared_v4(ebuf + lane * 128 + ((u ^ (lane & 7)) << 4), __uint_as_float(a[4 * u]),
                                     __uint_as_float(a[4 * u + 1]), __uint_as_float(a[4 * u + 2]),
                                     __uint_as_float(a[4 * u + 3]));
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int row = 4 * i + (lane >> 3), u = lane & 7;
                        *reinterpret_cast<float4*>(wdst + static_cast<long long>(row) * kDLatent + 32 * part + 4 * u) =
                            ld_shared_v4(ebuf + row * 128 + ((u ^ (row & 7)) << 4));
                    }
                    __syncwarp();
                }
                if (c == 0) p.lse[grow] = lse_tot;
            }
        };

        for (bool have = true, first = true; have && ok;
             have = next_segment<kSparse, kSched>(p, n_items, cu, sg), first = false) {
            const int n = sg.n;
            const bool row_valid = tok_local < sg.ntok;
            const int qidx = sg.qbase + tok_local;
            const long long grow = static_cast<long long>(qidx) * kHeads + head;  // global output row
            float m_use = -INFINITY;
            float l = 0.f;
            if (n > 0) {
                // Does a later segment of this pair have tiles?  Its first partial then
                // follows this segment's last one, and its byte count is posted in time.
                bool more = false;
                uint32_t more_bytes = kXBufBytes;   // size of that first partial
                if constexpr (kPersistent) {
                    Cursor c2 = cu;
                    Seg s2;
                    while (next_segment<kSparse, kSched>(p, n_items, c2, s2))
                        if (s2.n > 0) {
                            more = true;
                            more_bytes = exchange_bytes(exchange_rows<kSparse>(s2, 0));
                            break;
                        }
                }
                // ---- q of the segment -> TMEM columns [kTmQ, kTmQ + 128), rope half -> shared memory ----
                // The warp's async copies land in its 8 KB of the staging buffer, half a
                // row at a time; then the thread of each row moves that half into TMEM.
                // A warp's rows belong to one token, so row_valid is warp-uniform; rows
                // of a missing second token are zeros.  A later segment reuses the
                // staging buffer once this CTA's last partial-score copy has landed;
                // the previous segment's QK and PV are complete by then.
                if (g > 0) {
                    const bool sok = ok && mbar_wait<true>(&ctl->stg_free, (g - 1) & 1, abort_flag, lim);
                    ok = named_bar_and(4, kSoftmaxThreads, sok);
                    if (!ok) break;
                }
                for (int h = 0; h < 2; ++h) {
                    if (row_valid) {
                        if (h == 1 || kSparse || !first) issue_q_copies(sg, h);
                        cp_async_wait<0>();
                    } else if (h == 0) {
                        for (int u = 0; u < 4; ++u)
                            st_shared_v4(qrope_addr + r * 64 + ((u ^ ((r >> 1) & 3)) << 4), 0.f, 0.f, 0.f, 0.f);
                    }
                    __syncwarp();
                    for (int pp = 0; pp < 2; ++pp) {
                        uint32_t v[32];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const float4 w = row_valid
                                                 ? ld_shared_v4(qbuf + lane * 256 + (((8 * pp + u) ^ (lane & 15)) << 4))
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                            v[4 * u + 0] = __float_as_uint(w.x);
                            v[4 * u + 1] = __float_as_uint(w.y);
                            v[4 * u + 2] = __float_as_uint(w.z);
                            v[4 * u + 3] = __float_as_uint(w.w);
                        }
                        tmem_st32(trow + kTmQ + 32 * (2 * h + pp), v);
                    }
                    __syncwarp();   // this half is read out before the next one lands
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&ctl->q_ready);

                const uint64_t anc = row_valid ? p.anc[qidx] : 0ull;
                // Dense: the KV tiles tmask and tmask + 1 (at most 64 tree tokens) reach the
                // draft tokens.  Key k of tile tmask is a prefix key (k < a) or tree token
                // k - a; key k of the next tile is tree token k + 64 - a.  Visible: the prefix
                // and the row's ancestors and itself.  Taken once per segment, so the tile
                // loop only selects.
                [[maybe_unused]] const int tmask = sg.P / kBlockN;
                if constexpr (!kSparse) {
                    const int a = sg.P - tmask * kBlockN;
                    const uint64_t vis_first = (a > 0 ? (1ull << a) - 1ull : 0ull) | (anc << a);
                    const uint64_t vis_second = a > 0 ? anc >> (kBlockN - a) : 0ull;
                    st_shared_u64x2(vis_addr, vis_first, vis_second);   // kept out of the registers of the tile loop
                }
                for (int jj = 0; jj < n; ++jj) {
                    const int gi = g + jj;
                    const int x = gi & 1;
                    // ---- A/B: full scores = own partial (staging) + the peer's (receive buffer) ----
                    if (ok) ok = mbar_wait(&ctl->staged, gi & 1, abort_flag, lim);
                    if (ok) ok = mbar_wait<true>(&ctl->x_full, gi & 1, abort_flag, lim);
                    float s[kBlockN];
                    if (ok) {
                        if (r == 0) {
                            ++consumed;
                            mbar_arrive_remote_relaxed(&ctl->stg_free, peer);  // our staging landed: peer may reuse its own
                        }
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const uint32_t sw = (u ^ (r & 7)) << 4;
                            const float4 a = ld_shared_v4(rowbase + sw);
                            const float4 v = ld_shared_v4(peerbase + sw);
                            s[4 * u] = a.x + v.x;
                            s[4 * u + 1] = a.y + v.y;
                            s[4 * u + 2] = a.z + v.z;
                            s[4 * u + 3] = a.w + v.w;
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < kBlockN; ++k) s[k] = 0.f;
                    }
                    // this warp's rows of the staging buffer are read: its exchange warp may stage the next partial
                    __syncwarp();
                    if (ok && lane == 0) mbar_arrive(&ctl->stg_read[q4]);
                    // the receive buffer has been read by all 128 threads: let the peer send the next tile
                    named_bar_sync(2, kSoftmaxThreads);
                    if (r == 0 && ok) {
                        if (jj + 1 < n || more) {
                            mbar_arrive_expect_tx(&ctl->x_full, jj + 1 < n ? exchange_bytes(exchange_rows<kSparse>(sg, jj + 1))
                                                                           : more_bytes);
                            ++posted;
                        }
                        mbar_arrive_remote_relaxed(&ctl->x_empty, peer);
                    }
                    // ---- D: this tile's softmax ----
                    // tree mask (tiles that reach the draft tokens only).  Scores stay unscaled here:
                    // the scale is positive, so the row max can be taken on raw scores and the scale
                    // folded into the exponent's FMA below.
                    uint64_t vis = ~0ull;    // bit k: key k of the tile is visible to this row
                    bool masked = kSparse;
                    if constexpr (kSparse) {
                        int kind, base;
                        sparse_segment(sg.t0 + jj, sg.nA, sg.nB, kind, base);
                        if (kind == 2) {
                            vis = base == 0 ? anc : 0ull;  // at most 64 tree tokens: one tree tile
                        } else {
                            // the slot mask was written before the stage was released to QK
                            const int st = gi % kStages;
                            if (ok) ok = mbar_wait(&ctl->kv_full[st], (gi / kStages) & 1, abort_flag, lim);
                            const volatile uint32_t* sm = ctl->slot_mask[st];
                            vis = kind == tok_local ? static_cast<uint64_t>(sm[0]) |
                                                          (static_cast<uint64_t>(sm[1]) << (4 * gather_group0(1))) |
                                                          (static_cast<uint64_t>(sm[2]) << (4 * gather_group0(2)))
                                                    : 0ull;
                        }
                    } else {
                        const int tt = sg.t0 + jj;
                        masked = tt >= tmask;
                        if (masked) vis = ld_shared_u64(vis_addr + (tt == tmask ? 0u : 8u));
                    }
                    // one compact select per score: this code also runs on a tile's first pass
                    if (masked) {
#pragma unroll
                        for (int k = 0; k < kBlockN; ++k) s[k] = ((vis >> k) & 1ull) ? s[k] : -INFINITY;
                    }
                    // tree reductions (8 independent chains) keep the dependent latency short
                    float mx[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) mx[k] = s[k];
#pragma unroll
                    for (int k = 8; k < kBlockN; ++k) mx[k & 7] = fmaxf(mx[k & 7], s[k]);
                    const float mt_raw = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                    const float mt = mt_raw == -INFINITY ? -INFINITY : mt_raw * p.scale_log2;  // log2 units
                    // ---- lazy online-softmax rescale (warp-uniform TMEM traffic) ----
                    const bool grow_max = ok && mt > m_use + kLazyRescaleLog2;
                    float alpha = 1.f;
                    if (grow_max) {
                        alpha = ex2_approx(m_use - mt);  // 0 when m_use is -inf
                        m_use = mt;
                        l *= alpha;
                    }
                    ok = __all_sync(0xffffffffu, ok);
                    // PV of the previous tile must be done before O is rescaled and before its
                    // P columns are overwritten (it normally finished long ago; the previous
                    // segment's last PV was waited for in its epilogue)
                    if (ok && jj > 0)
                        ok = __all_sync(0xffffffffu, mbar_wait(&ctl->pv_done[(gi - 1) & 1], ((gi - 1) >> 1) & 1,
                                                               abort_flag, lim));
                    if (ok && jj > 0 && __any_sync(0xffffffffu, grow_max)) {
                        tc_fence_after();
                        for (int part = 0; part < kDLatentHalf / 32; ++part) {
                            uint32_t o[32];
                            tmem_ld32(trow + kTmO + 32 * part, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                            tmem_st32(trow + kTmO + 32 * part, o);
                        }
                        tmem_wait_st();
                    }
                    // ---- probabilities: p = 2^(s * scale * log2 e - m), one FMA + ex2 each ----
                    const bool live = m_use != -INFINITY;
                    const float neg_m = -m_use;
                    float ps[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) ps[k] = 0.f;
                    if (live) {
#pragma unroll
                        for (int k = 0; k < kBlockN; ++k) {
                            s[k] = ex2_approx(fmaf(s[k], p.scale_log2, neg_m));
                            ps[k & 7] += s[k];
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < kBlockN; ++k) s[k] = 0.f;
                    }
                    const float psum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
                    const float pmax = live ? ex2_approx(mt - m_use) : 0.f;  // the tile's largest p
                    // One named barrier decides, uniformly for the 128 threads, whether to stop
                    // (bit 1) and whether this tile needs the low part of P (bit 0).
                    volatile int* flags = &ctl->tile_flags[gi % 3];
                    const int mine = (ok ? 0 : 2) | ((pmax > kLowPartShare * (l + psum)) ? 1 : 0);
                    if (mine) atomicOr(const_cast<int*>(flags), mine);
                    named_bar_sync(1, kSoftmaxThreads);
                    const int tf = *flags;
                    if (tf & 2) {
                        ok = false;
                        break;
                    }
                    const bool need_lo = tf & 1;
                    if (r == 0) {
                        ctl->tile_flags[(gi + 2) % 3] = 0;  // read by everyone before this barrier; next used by tile gi + 2
                        ctl->lo_flag[x] = need_lo ? 1 : 0;
                    }
                    // ---- P -> TMEM: keys 2k and 2k + 1 of the tile as the bf16 pair in column k of
                    // this row (the A operand of PV), the low part in the next 32 columns ----
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {   // 16 columns (32 keys) at a time
                        uint32_t ph[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k) ph[k] = pack_bf16x2(s[32 * hh + 2 * k], s[32 * hh + 2 * k + 1]);
                        tmem_st16(trow + kTmP + 16 * hh, ph);
                        if (need_lo) {
                            uint32_t pl[16];
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                pl[k] = pack_bf16x2(s[32 * hh + 2 * k] - bf16lo_to_f32(ph[k]),
                                                    s[32 * hh + 2 * k + 1] - bf16hi_to_f32(ph[k]));
                            tmem_st16(trow + kTmPLo + 16 * hh, pl);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    // The normaliser uses the fp32 weights.  Without the low part the bf16
                    // weights that PV sees differ from them by unbiased rounding of at most
                    // 2^-9 each, on tiles where no weight exceeds 1/16 of the row's mass.
                    l += psum;
                    mbar_arrive(&ctl->p_full[x]);   // the PV issuer (sparse: the QK warp) may go
                }
                // ---- epilogue: the segment's last PV ----
                if (ok) ok = mbar_wait(&ctl->pv_done[(g + n - 1) & 1], ((g + n - 1) >> 1) & 1, abort_flag, lim);
                // the staging buffer, the epilogue's scratch, was the source of the CTA's last
                // partial-score copy: wait until it has landed
                if (ok) ok = mbar_wait<true>(&ctl->stg_free, (g + n - 1) & 1, abort_flag, lim);
            }
            // one decision for all 128 softmax threads (the in-kernel merges and the next
            // segment synchronise them)
            if constexpr (kSched == kSchedPlain) ok = __all_sync(0xffffffffu, ok);
            else ok = named_bar_and(4, kSoftmaxThreads, ok);
            if (!ok) break;
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const float lse_v = (l > 0.f ? m_use + log2f(l) : -INFINITY) * 0.6931471805599453f;
            // this segment's normalised columns 32 part .. 32 part + 31 of the thread's row
            auto own = [&](int part, float* v) {
                if (n > 0) {
                    uint32_t o[32];
                    tmem_ld32(trow + kTmO + 32 * part, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = __fmul_rn(__uint_as_float(o[k]), inv_l);
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = 0.f;
                }
            };
            if constexpr (kSched == kSchedMerge) {
                if (sg.kind == kOutTwoSplit) {
                    two_split_merge(sg, own, lse_v);
                    g += n;
                    continue;
                }
            }
            if constexpr (kPersistent) {
                if (sg.kind == kOutPiece) {
                    piece_merge(own, lse_v, g + n);
                    g += n;
                    continue;
                }
            }
            {
                const long long slot_row = static_cast<long long>(sg.split - p.split_base) * out_rows + grow;
                float* dst = sg.kind == kOutFinal ? p.out + grow * kDLatent + kDLatentHalf * c
                                                  : p.part_out + slot_row * kDLatent + kDLatentHalf * c;
                // The rows go out through shared memory so that every store instruction
                // writes whole 128-byte lines: the thread of a row puts 32 of its values
                // into the warp's 4 KB tile (swizzled), then each lane stores 16 bytes of
                // one of four rows.  The staging buffer is free here (its last copy landed).  A warp's
                // 32 rows belong to one token, so row_valid is warp-uniform.
                float* wdst = dst - static_cast<long long>(lane) * kDLatent;   // the warp's first row
                for (int part = 0; part < kDLatentHalf / 32; ++part) {
                    float v[32];
                    own(part, v);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        st_shared_v4(ebuf + lane * 128 + ((u ^ (lane & 7)) << 4), v[4 * u], v[4 * u + 1],
                                     v[4 * u + 2], v[4 * u + 3]);
                    __syncwarp();
                    if (row_valid) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int row = 4 * i + (lane >> 3), u = lane & 7;
                            const float4 v4 = ld_shared_v4(ebuf + row * 128 + ((u ^ (row & 7)) << 4));
                            *reinterpret_cast<float4*>(wdst + static_cast<long long>(row) * kDLatent + 32 * part + 4 * u) = v4;
                        }
                    }
                    __syncwarp();
                }
                if (row_valid && c == 0) {
                    if (sg.kind == kOutFinal) p.lse[grow] = lse_v;
                    else p.part_lse[slot_row] = lse_v;
                }
            }
            g += n;
        }
        if (!ok) {
            if (r == 0) {
                raise_status(p.status, kStatusTimeout);
                // do not leave while the peer's bulk copies may still land in this CTA
                const int zero = 0;
                for (int t = consumed; t < posted; ++t) mbar_wait<true>(&ctl->x_full, t & 1, &zero, lim);
            }
            *abort_flag = 1;
        }

    } else if (stager_warp) {
        setmaxnreg_dec<kRegsOther>();
        // ================= exchange: S (TMEM) -> staging -> the peer's receive buffer =================
        // Step C of every tile t of the CTA's stream, off the softmax threads' path.  Exchange
        // warp w owns rows [32w, 32w + 32).  As soon as QK(t) is in TMEM and its rows of the
        // staging buffer are free (the peer has received partial t - 1 and softmax warp w has
        // read them), the thread of each row copies its 64 partial scores into the staging
        // buffer; the four warps then meet, and one thread sends the tile to the peer once
        // the peer has read partial t - 1, and marks it staged.
        const uint32_t trow = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
        const uint32_t stg_local = smem_u32(smem + kOffStaging);
        const uint32_t xbuf_peer = mapa(smem_u32(smem + kOffXBuf), peer);
        const uint32_t xfull_peer = mapa(smem_u32(&ctl->x_full), peer);
        const uint32_t rowbase = stg_local + r * (kBlockN * 4);       // this row in the staging buffer
        const int sr = static_cast<int>(threadIdx.x) - kStagerWarp0 * 32;   // 0 .. 127
        bool ok = true;
        int g = 0;
        Cursor cu = cu0;
        Seg sg = seg0;
        for (bool have = true; have && ok; have = next_segment<kSparse, kSched>(p, n_items, cu, sg)) {
            const int n = sg.n;
            if (n <= 0) continue;
            for (int jj = 0; jj < n; ++jj) {
                const int t = g + jj;
                // each warp stages its 32 rows as soon as its softmax warp has read them;
                // the four warps meet once, before the copy
                bool w = mbar_wait(&ctl->s_full, t & 1, abort_flag, lim);
                if (w && t >= 1) w = mbar_wait<true>(&ctl->stg_free, (t - 1) & 1, abort_flag, lim);
                if (w && t >= 1) w = mbar_wait(&ctl->stg_read[q4], (t - 1) & 1, abort_flag, lim);
                w = __all_sync(0xffffffffu, w);   // the TMEM loads are warp-wide
                if (w) {
                    tc_fence_after();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t a[32];
                        tmem_ld32(trow + kTmS + 32 * hh, a);
                        tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int uu = 8 * hh + u;
                            st_shared_v4(rowbase + ((uu ^ (r & 7)) << 4), __uint_as_float(a[4 * u]),
                                         __uint_as_float(a[4 * u + 1]), __uint_as_float(a[4 * u + 2]),
                                         __uint_as_float(a[4 * u + 3]));
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(&ctl->s_free);  // the S columns may take the next QK
                    fence_proxy_async_smem();
                }
                ok = named_bar_and(7, kSoftmaxThreads, w);
                if (!ok) break;
                if (sr == 0) {
                    // the peer has read the partial this CTA sent before (its receive buffer is free)
                    bool sent = t < 1 || mbar_wait<true>(&ctl->x_empty, (t - 1) & 1, abort_flag, lim);
                    const bool skip_send = fault_kind() == 3 && sg.item == 0 && sg.split == 0 && c == 0 && t == 1;
                    const int rows = exchange_rows<kSparse>(sg, jj);
                    const uint32_t off = rows < 0 ? 0u : static_cast<uint32_t>(rows) * (kXBufBytes / 2);
                    if (sent && !skip_send)
                        bulk_copy_to_peer(xbuf_peer + off, stg_local + off, exchange_bytes(rows), xfull_peer);
                    mbar_arrive(&ctl->staged);
                    if (!sent) {
                        raise_status(p.status, kStatusTimeout);
                        *abort_flag = 1;
                    }
                }
            }
            g += n;
        }
        if (!ok) {
            if (sr == 0) raise_status(p.status, kStatusTimeout);
            *abort_flag = 1;
        }
    }

    // ---- tear-down ----
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    cluster_sync();  // the peer may still be writing to this CTA's shared memory until here
}

}  // namespace mla
