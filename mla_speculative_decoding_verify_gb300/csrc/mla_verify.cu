// Host side of the C ABI declared in include/mla_verify.h: argument checks,
// per-device set-up, TMA descriptor encoding, the split heuristic, workspace
// layout and the launches (prep -> verify -> combine) on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>
#include <algorithm>
#include <functional>
#include <queue>
#include <vector>
#include <new>

#include "mla_verify.h"
#include "combine_kernel.cuh"
#include "kv_ops_kernel.cuh"
#include "prep_kernel.cuh"
#include "verify_kernel.cuh"

namespace mla_internal {
void noalloc_forget_device(int dev);   // mla_verify_noalloc.cu
}

namespace {

constexpr int kMaxDevices = 64;
#ifdef MLA_FAULT_INJECTION
constexpr uint64_t kDefaultTimeoutNs = 5000000ull;      // test build: 5 ms per pipeline wait
#else
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;  // 1 s per pipeline wait
#endif

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int pairs = 0;   // CTA pairs of the verify kernel that fit on the device at once
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
cudaEvent_t g_prof_begin = nullptr, g_prof_end = nullptr;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

// Workspace layout shared by the size query and the launch.
struct Layout {
    size_t status, item_count, q_off, req_state, order, item_off, anc, items, part_out, part_lse, tok_req, merge_cnt,
        tail_k, woff, pair_begin, pair_item, item_first_pair, rounds, total;
    int max_items;
};

// One split chosen automatically: the work items of the last, partial round of
// CTA pairs (rem = items mod pairs, when at most half the pairs) are cut in
// two and merged in the kernel, so that their halves run side by side and the
// last round ends about twice as early.  The prep kernel picks rem from the
// exact item count; the host fixes the cap (half the pairs: the grid's extra
// units and the partial buffers) and the cut, which balances the two halves,
// the second of which also carries the merge (merge_tiles, in KV tiles of the
// variant).  Items of fewer than 12 tiles are not cut (measured on a 5-tile
// item: the merge cost more than the halves saved).  cap = 0: no cutting.
struct TailPlan {
    int cap = 0, share = 0;
};

TailPlan tail_plan(int tiles, int pairs, double merge_tiles) {
    TailPlan t;
    if (tiles < 12 || pairs < 2) return t;   // short items: the merge costs more than it saves
    const int a = std::clamp(static_cast<int>(std::lround((tiles + merge_tiles) / 2.0)), (tiles + 1) / 2, tiles - 1);
    t.cap = pairs / 2;
    t.share = std::clamp((a * 1024 + tiles / 2) / tiles, 1, 1023);
    return t;
}

// sched_pairs > 0: the persistent schedule on that many CTA pairs (num_splits is then 1 and tail_cap 0).
Layout make_layout(int batch, int total_q, int num_splits, bool sparse = false, int tail_cap = 0, int sched_pairs = 0) {
    Layout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    L.max_items = (total_q + batch) / 2 + 1;
    L.status = take(sizeof(int));
    L.item_count = take(sizeof(int));
    L.q_off = take(sizeof(int32_t) * (batch + 1));
    L.req_state = take(sizeof(int32_t) * batch);
    L.order = take(sizeof(int32_t) * batch);
    L.item_off = take(sizeof(int32_t) * (batch + 1));
    L.anc = take(sizeof(uint64_t) * (total_q > 0 ? total_q : 1));
    L.items = take(sizeof(int2) * L.max_items);
    const size_t rows = static_cast<size_t>(total_q) * MLA_NUM_HEADS;
    L.part_out = L.part_lse = L.merge_cnt = L.tail_k = 0;
    L.woff = L.pair_begin = L.pair_item = L.item_first_pair = L.rounds = 0;
    if (sched_pairs > 0) {
        // pieces of items cut between pairs: slots 2q (first segment of pair q) and 2q + 1 (its last)
        const size_t slots = 2 * static_cast<size_t>(sched_pairs);
        L.part_out = take(sizeof(float) * slots * mla::kRows * MLA_D_LATENT);
        L.part_lse = take(sizeof(float) * slots * 2 * mla::kRows);
        L.merge_cnt = take(sizeof(int32_t) * 4 * static_cast<size_t>(L.max_items));
        L.woff = take(sizeof(long long) * (static_cast<size_t>(L.max_items) + 1));
        L.pair_begin = take(sizeof(long long) * (static_cast<size_t>(sched_pairs) + 1));
        L.pair_item = take(sizeof(int32_t) * (static_cast<size_t>(sched_pairs) + 1));
        L.item_first_pair = take(sizeof(int32_t) * static_cast<size_t>(L.max_items));
        L.rounds = take(sizeof(int32_t));
    } else if (num_splits > 1) {
        L.part_out = take(sizeof(float) * rows * MLA_D_LATENT * num_splits);
        // two splits are merged in the verify kernel: lse per CTA half, and per-tile counters
        L.part_lse = take(sizeof(float) * rows * num_splits * (num_splits == 2 ? 2 : 1));
        L.merge_cnt = num_splits == 2 ? take(sizeof(int32_t) * 4 * static_cast<size_t>(L.max_items)) : 0;
    } else if (tail_cap > 0) {
        // cut tail items: partials of up to tail_cap row tiles, compact, two splits
        const size_t prows = static_cast<size_t>(tail_cap) * mla::kRows;
        L.part_out = take(sizeof(float) * prows * MLA_D_LATENT * 2);
        L.part_lse = take(sizeof(float) * prows * 2 * 2);
        L.merge_cnt = take(sizeof(int32_t) * 4 * static_cast<size_t>(L.max_items));
        L.tail_k = take(sizeof(int32_t));
    }
    L.tok_req = sparse ? take(sizeof(int32_t) * (total_q > 0 ? total_q : 1)) : 0;
    L.total = off;
    return L;
}

int sm_count_of_current() {
    const int d = current_device();
    if (d >= 0 && d < kMaxDevices && g_dev[d].ready) return g_dev[d].sm_count;
    int n = 0;
    if (d >= 0 && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) == cudaSuccess && n > 0) return n;
    return 152;
}

constexpr double kUnitOverheadTiles = 6.0;  // per work unit: q load, pipeline fill, epilogue
constexpr double kMergeTiles = 6.0;         // extra for a second-split unit: the in-kernel merge

// Model of the verify time (in KV-tile units of one CTA pair) for `splits`
// splits: whole waves of (request, row tile, split) units over the SMs,
// a fixed per-unit cost, and the combine pass when split.
double model_time(long long units_per_split, int tiles, int splits, int pairs, long long rows) {
    const double kTileSeconds = 1.1e-6;     // one 64-key tile of 128 rows on a CTA pair
    const double kCombineBytesPerSecond = 5.0e12;
    const long long units = units_per_split * splits;
    const long long waves = (units + pairs - 1) / pairs;
    const double per_unit = std::ceil(static_cast<double>(tiles) / splits) + kUnitOverheadTiles;
    double t = static_cast<double>(waves) * per_unit;
    if (splits == 1 && units >= pairs) {
        // the automatic single split cuts the items of a partial last round in two
        // (tail_plan): that round takes about half an item plus the merge.  With no
        // full round before it the cut is a two-way split with a plainer share, and
        // the two-split estimate below is the better guide (measured: 4 x 4096 x 16
        // runs 2% faster on two splits).
        const TailPlan tp = tail_plan(tiles, pairs, kMergeTiles);
        const long long rem = units % pairs;
        if (tp.cap > 0 && rem > 0 && rem <= tp.cap)
            t = static_cast<double>(units / pairs) * per_unit +
                std::ceil((tiles + kMergeTiles) / 2.0) + kUnitOverheadTiles;
    }
    if (splits > 1) t += (static_cast<double>(rows) * splits * 2048.0 / kCombineBytesPerSecond) / kTileSeconds;
    return t;
}

// Work items of a launch (row tiles of two tree tokens), bounded from the sizes.
long long items_bound_of(int batch, int total_q, int max_tree) {
    return std::min<long long>(static_cast<long long>(batch) * ((max_tree + 1) / 2),
                               (static_cast<long long>(total_q) + batch) / 2);
}

// With two splits: the first split's share of a work item's tiles, in 1/1024.
// The CTAs of a launch start in grid order, every first split before any
// second one.  A greedy list-scheduling model of that order over the CTA pairs
// (a unit costs its tiles plus kUnitOverheadTiles) picks the cut whose rounds
// end most evenly: a long first part, and a short second part that fills the
// last round.  A second-split unit also carries the merge (kMergeTiles, fitted
// to a sweep of the share on a 16 x 16384-token batch, where the model's best
// cut matched the measured one).  Past eight rounds the tail is small and the
// halves are kept.
// The last answer is cached (a serving loop repeats its shapes).
int first_split_share(long long items, int tiles, int pairs) {
    if (items <= 0 || tiles < 2 || pairs <= 0 || 2 * items > 8LL * pairs) return 0;
    static std::mutex mu;
    static long long c_items = -1;
    static int c_tiles = -1, c_pairs = -1, c_share = 0;
    {
        std::lock_guard<std::mutex> g(mu);
        if (c_items == items && c_tiles == tiles && c_pairs == pairs) return c_share;
    }
    const double o = kUnitOverheadTiles;
    auto span = [&](int a) {
        std::priority_queue<double, std::vector<double>, std::greater<double>> q;
        for (int i = 0; i < pairs; ++i) q.push(0.0);
        auto put = [&](double w) {
            const double t = q.top();
            q.pop();
            q.push(t + w);
        };
        for (long long i = 0; i < items; ++i) put(a + o);
        for (long long i = 0; i < items; ++i) put(tiles - a + o + kMergeTiles);
        double m = 0.0;
        while (!q.empty()) {
            m = std::max(m, q.top());
            q.pop();
        }
        return m;
    };
    const int half = (tiles + 1) / 2;
    int best_a = half;
    double best = span(half);
    const int step = std::max(1, tiles / 64);
    for (int a = half + step; a < tiles; a += step) {
        const double m = span(a);
        if (m < best - 1e-9) {
            best = m;
            best_a = a;
        }
    }
    const int share = best_a == half ? 0 : std::clamp((best_a * 1024 + tiles / 2) / tiles, 1, 1023);
    std::lock_guard<std::mutex> g(mu);
    c_items = items;
    c_tiles = tiles;
    c_pairs = pairs;
    c_share = share;
    return share;
}

int persistent_pairs();

// Whole-item rounds of the persistent schedule for `items` work items on `pairs`
// CTA pairs (the prep kernel's rule: a last round of fewer than pairs / 4 items
// joins the round before, so that its items are not cut into many small pieces).
long long persistent_rounds(long long items, int pairs) {
    long long r = items / pairs;
    if (r > 0 && items - r * pairs < pairs / 4) --r;
    return r;
}

// Model of the persistent schedule's time, in the units of model_time: whole-item
// rounds, then the rest shared evenly over the pairs with one more segment and a
// merge per pair, every tile kPersistentTileCost times as long as on the per-unit
// grid.  Whole rounds of 24 x 16384-token requests measured 2.3 % slower (2.518
// against 2.462 ms: the persistent variant has no registers to spare for the
// four-stage pipeline and spills a little); 8 % is fitted to a sweep of eleven
// uniform shapes, on which the model then picks the faster schedule every time
// (persistent only for 12 x 8192 x 16: 0.3666 against 0.3707 ms).
constexpr double kPersistentTileCost = 1.08;

double persistent_model_time(long long items, int tiles, int pairs) {
    const long long rounds = persistent_rounds(items, pairs);
    const long long rest = items - rounds * pairs;
    double t = static_cast<double>(rounds) * (tiles + kUnitOverheadTiles);
    if (rest > 0) t += static_cast<double>(rest) * tiles / pairs + kUnitOverheadTiles + kMergeTiles;
    return kPersistentTileCost * t;
}

// Split count for requests of up to `tiles` KV tiles per row tile, or 0 for the
// persistent schedule.  Sizes are bounds (the host never reads device data), so
// the model takes every item as `tiles` long.  The persistent schedule is taken
// only when every request has max_tree tree tokens (total_q = batch x max_tree:
// then the item count is exact, and the rounds the model counts are the real
// ones), with at least one round of whole items (with none, pairs stream one
// request's KV at different offsets and lose its reuse in L2; measured 1-3 %
// slower), and when the model puts it at least 5 % ahead.
constexpr double kPersistentMargin = 0.95;

int choose_splits_tiles(int batch, int total_q, int max_tree, int tiles) {
    const long long items_bound = items_bound_of(batch, total_q, max_tree);
    const int pairs = sm_count_of_current() / 2;
    const long long rows = static_cast<long long>(total_q) * MLA_NUM_HEADS;
    const int max_s = std::max(1, std::min(MLA_MAX_SPLITS, tiles / 16));
    int best = 1;
    double best_t = model_time(items_bound, tiles, 1, pairs, rows);
    for (int s = 2; s <= max_s; ++s) {
        const double t = model_time(items_bound, tiles, s, pairs, rows);
        if (t < best_t * 0.97) {  // prefer fewer splits unless clearly faster
            best_t = t;
            best = s;
        }
    }
    const int pp = persistent_pairs();
    const bool exact = static_cast<long long>(batch) * max_tree == total_q;
    if (exact && persistent_rounds(items_bound, pp) >= 1 &&
        persistent_model_time(items_bound, tiles, pp) < kPersistentMargin * best_t)
        return 0;
    if (items_bound > 0 && 3 * items_bound <= pairs) {
        // Latency regime: three or more splits still fit in one wave, so a launch
        // takes as long as one unit's chain of dependent tiles plus the merge: the
        // combine kernel for three splits or more, the in-kernel merge for two
        // (whose variant's longer code costs a small launch more).  Measured step
        // device times (us) against the choice: 1 x 256 x 8: 29.3 on one split, 31.4
        // on two, 26.2 on three and five (5 chosen); 1 x 2048 x 8: 89.2 / 64.1 / 34.4
        // on 1 / 2 / 9; 4 x 512 x 8: 38.6 / 38.5 / 30.4 on 1 / 2 / 3 (3 chosen).
        const double kTileLatency = 2.1e-6, kMergeFixed = 8.5e-6, kCombineFixed = 4.5e-6;
        // per row and split: the fp32 partial written and read back, and q loaded again
        const double kRowSplitBytes = 2048.0 + 2048.0 + 1152.0, kBytesPerSecond = 5.0e12;
        const long long fit = std::min<long long>(pairs / items_bound, std::min(MLA_MAX_SPLITS, tiles));
        double t_best = 0.0;
        int s_best = 1;
        for (int s = 1; s <= std::max<long long>(1, fit); ++s) {
            const double t = std::ceil(static_cast<double>(tiles) / s) * kTileLatency +
                             (s == 1 ? 0.0
                              : s == 2 ? kMergeFixed
                                       : kCombineFixed + static_cast<double>(rows) * s * kRowSplitBytes / kBytesPerSecond);
            if (s == 1 || t < t_best) {
                t_best = t;
                s_best = s;
            }
        }
        return s_best;
    }
    return best;
}

int choose_splits(int batch, int total_q, int max_tree, int max_seq_len) {
    return choose_splits_tiles(batch, total_q, max_tree, (max_seq_len + mla::kBlockN - 1) / mla::kBlockN);
}

// KV tiles of a sparse row tile: two tokens' slot lists, then the tree keys.
int sparse_tiles(int topk) { return 2 * ((topk + mla::kBlockN - 1) / mla::kBlockN) + 1; }

// Persistent schedule: a share is moved to an item boundary rather than leave a
// piece of fewer tiles than this (a piece costs a q load, a pipeline fill and a merge).
constexpr int kMinPieceTiles = 4;

// CTA pairs of the persistent schedule: every pair of the device, whatever the
// sizes (the shares are cut from the exact work on the device; a pair whose share
// is empty exits at once).  The partition, and so the result, then depends only on
// the requests, not on the buffer sizes a graph was captured for.
int persistent_pairs() {
    const int d = current_device();
    if (d >= 0 && d < kMaxDevices && g_dev[d].ready && g_dev[d].pairs > 0) return g_dev[d].pairs;
    return std::max(1, sm_count_of_current() / 2);
}

// Tail cut of a launch whose split count was chosen automatically as one (an
// explicit request is taken as it is).  `tiles` = KV tiles of a work item.
TailPlan launch_tail_plan(bool sparse, int tiles, int requested, int splits) {
    if (requested != 0 || splits != 1) return TailPlan{};
    return tail_plan(tiles, sm_count_of_current() / 2, sparse ? 2.0 : kMergeTiles);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Maps over the cache as a [rows, 576] bf16 tensor: 64-dim latent chunks (128B
// swizzle) and 32-dim rope halves (64B swizzle).  box_rows is 64 for a dense
// tile and 1 for the sparse variant's four-row gathers.
int encode_maps(const void* kv_cache, long long rows, unsigned box_rows, CUtensorMap* lat, CUtensorMap* rope) {
    if (!g_encode) return MLA_ERR_NOT_INITIALIZED;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(MLA_D_LATENT + MLA_D_ROPE), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>((MLA_D_LATENT + MLA_D_ROPE) * 2)};
    const cuuint32_t box_lat[2] = {64, box_rows};
    const cuuint32_t box_rope[2] = {static_cast<cuuint32_t>(mla::kDRopeHalf), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r1 = g_encode(lat, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv_cache), dims, strides,
                           box_lat, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    CUresult r2 = g_encode(rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv_cache), dims, strides,
                           box_rope, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return (r1 == CUDA_SUCCESS && r2 == CUDA_SUCCESS) ? MLA_OK : MLA_ERR_CUDA;
}

// Launch as a programmatic dependent of the previous kernel in the stream: the
// grid may start while that one finishes and waits (griddepcontrol.wait) before
// reading its results, which hides the launch latency between the step's kernels.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

int launch_combine(const float* part_out, const float* part_lse, int num_splits, long long rows, float* out,
                   float* lse, cudaStream_t stream) {
    if (rows == 0) return MLA_OK;
    const long long blocks = (rows + mla::kCombineWarps - 1) / mla::kCombineWarps;
    const cudaError_t e = launch_dependent(mla::mla_combine_kernel, dim3(static_cast<unsigned>(blocks)),
                                           dim3(mla::kCombineWarps * 32), 0, stream, part_out, part_lse, num_splits,
                                           rows, out, lse);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

extern "C" {

int mla_version(void) { return 100; }

const char* mla_error_string(int status) {
    switch (status) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARG: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported shape";
        case MLA_ERR_WORKSPACE: return "workspace missing or too small";
        case MLA_ERR_CUDA: return "CUDA error";
        case MLA_ERR_TIMEOUT: return "device-side wait timed out";
        case MLA_ERR_BAD_TREE: return "invalid draft tree or lengths";
        case MLA_ERR_BAD_BLOCK: return "block-table entry out of range";
        case MLA_ERR_NOT_INITIALIZED: return "mla_init has not run on this device";
        case MLA_ERR_BAD_INDEX: return "a top-k slot is neither -1 nor a prefix position";
        default: return "unknown status";
    }
}

int mla_init(int device) {
    if (device < 0 || device >= kMaxDevices) return MLA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (cudaSetDevice(device) != cudaSuccess) return MLA_ERR_CUDA;
    // Every call sets the device up again (cheap): after cudaDeviceReset the
    // device has a new context, without the kernels' attributes of the old one.
    mla_internal::noalloc_forget_device(device);
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MLA_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return MLA_ERR_UNSUPPORTED;  // built for sm_103a only
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return MLA_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (cudaFuncSetAttribute(mla::mla_tree_accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(mla::kAcceptSmemBytes)) != cudaSuccess)
        return MLA_ERR_CUDA;
    for (const void* fn : {reinterpret_cast<const void*>(mla::mla_verify_kernel<false, mla::kSchedPlain>),
                           reinterpret_cast<const void*>(mla::mla_verify_kernel<false, mla::kSchedMerge>),
                           reinterpret_cast<const void*>(mla::mla_verify_kernel<false, mla::kSchedPersistent>),
                           reinterpret_cast<const void*>(mla::mla_verify_kernel<true, mla::kSchedPlain>),
                           reinterpret_cast<const void*>(mla::mla_verify_kernel<true, mla::kSchedMerge>),
                           reinterpret_cast<const void*>(mla::mla_verify_kernel<true, mla::kSchedPersistent>)})
    {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(mla::kSmemBytes)) !=
            cudaSuccess)
            return MLA_ERR_CUDA;
        // The warpgroups' register shares must fit in what the block is launched with,
        // or the softmax warps' setmaxnreg.inc would never complete: refuse to run.
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return MLA_ERR_CUDA;
        if (static_cast<long long>(fa.numRegs) * mla::kThreads <
            128LL * mla::kRegsSoftmax + 256LL * mla::kRegsOther)
            return MLA_ERR_UNSUPPORTED;
    }
    g_dev[device].sm_count = prop.multiProcessorCount;
    // 2-CTA clusters of the verify kernel resident at once (one CTA per SM; the
    // placement of clusters may leave SMs out), the grid of the persistent schedule
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2u * static_cast<unsigned>(std::max(1, prop.multiProcessorCount / 2)));
        cfg.blockDim = dim3(mla::kThreadsSparse);
        cfg.dynamicSmemBytes = mla::kSmemBytes;
        int clusters = 0;
        const cudaError_t e = cudaOccupancyMaxActiveClusters(
            &clusters, reinterpret_cast<const void*>(mla::mla_verify_kernel<true, mla::kSchedPersistent>), &cfg);
        if (e != cudaSuccess) cudaGetLastError();   // not fatal: fall back to half the SMs
        const int half = std::max(1, prop.multiProcessorCount / 2);
        g_dev[device].pairs = (e == cudaSuccess && clusters > 0) ? std::min(clusters, half) : half;
    }
    g_dev[device].ready = true;
    return MLA_OK;
}

int mla_verify_num_splits(int batch, int total_q, int max_tree, int max_seq_len, int num_heads, int requested) {
    if (batch < 0 || total_q < 0 || max_tree < 0 || max_seq_len < 0 || requested < MLA_SPLITS_PERSISTENT)
        return -MLA_ERR_INVALID_ARG;
    if (num_heads != MLA_NUM_HEADS) return -MLA_ERR_UNSUPPORTED;
    if (requested == MLA_SPLITS_PERSISTENT) return 0;
    if (requested > 0) return std::min(requested, MLA_MAX_SPLITS);
    return choose_splits(batch, total_q, max_tree, max_seq_len);
}

size_t mla_verify_workspace_size(int batch, int total_q, int max_tree, int max_seq_len, int num_heads,
                                 int num_splits) {
    const int s = mla_verify_num_splits(batch, total_q, max_tree, max_seq_len, num_heads, num_splits);
    if (s < 0) return 0;
    const int tiles = (max_seq_len + mla::kBlockN - 1) / mla::kBlockN;
    if (s == 0) return make_layout(batch, total_q, 1, false, 0, persistent_pairs()).total;
    const TailPlan tp = launch_tail_plan(false, tiles, num_splits, s);
    return make_layout(batch, total_q, s, false, tp.cap).total;
}

// Both entry points: topk == 0 is the dense verify, topk > 0 the sparse variant.
static int verify_impl(const void* q_lat, const void* q_rope, const void* kv_cache, const int32_t* block_table,
                       const int32_t* seq_lens, const int32_t* tree_parent, const int32_t* n_tree, float scale,
                       float* out, float* lse, cudaStream_t stream, int batch, int total_q, int max_tree,
                       int max_seq_len, int num_heads, int page_size, int num_pages, int max_pages_per_seq,
                       int num_splits, void* workspace, size_t workspace_bytes, const int32_t* topk_idx,
                       int topk, bool graph_capture = false, int split_begin = 0, int split_count = 0) {
    // split_count > 0: compute only splits split_begin .. split_begin + split_count - 1 of
    // num_splits, each one's partial into out / lse viewed as [split_count, rows, 512] / [split_count, rows]
    const bool range = split_count > 0;
    if (range && (topk > 0 || num_splits < 1 || split_begin < 0 || split_begin + split_count > num_splits))
        return num_splits > MLA_MAX_SPLITS ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
    // ---- host-checkable arguments ----
    if (batch < 0 || total_q < 0 || max_tree < 0 || max_seq_len < 0 || num_pages < 0 || max_pages_per_seq < 0 ||
        num_splits < MLA_SPLITS_PERSISTENT || page_size <= 0 || !std::isfinite(scale) || !(scale > 0.f))
        return MLA_ERR_INVALID_ARG;
    if (num_heads != MLA_NUM_HEADS || page_size % mla::kBlockN != 0 || max_tree > MLA_MAX_TREE ||
        num_splits > MLA_MAX_SPLITS)
        return MLA_ERR_UNSUPPORTED;
    if (static_cast<long long>(num_pages) * page_size > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
    if (batch == 0 || total_q == 0) return MLA_OK;  // nothing to compute
    if (!q_lat || !q_rope || !kv_cache || !block_table || !seq_lens || !tree_parent || !n_tree || !out || !lse)
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_lat) || !aligned16(q_rope) || !aligned16(kv_cache) || !aligned16(out) || !aligned16(lse))
        return MLA_ERR_INVALID_ARG;
    if (num_pages == 0 || max_pages_per_seq == 0) return MLA_ERR_INVALID_ARG;
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices || !g_dev[dev].ready) return MLA_ERR_NOT_INITIALIZED;
    const int resolved = topk > 0 ? mla_verify_sparse_num_splits(batch, total_q, max_tree, topk, num_heads, num_splits)
                                  : mla_verify_num_splits(batch, total_q, max_tree, max_seq_len, num_heads, num_splits);
    if (resolved < 0) return MLA_ERR_INVALID_ARG;
    const bool persistent = resolved == 0 && !range;   // 0: the persistent schedule
    if (resolved == 0 && range) return MLA_ERR_INVALID_ARG;
    const int splits = persistent ? 1 : resolved;
    const int item_tiles = topk > 0 ? sparse_tiles(topk) : (max_seq_len + mla::kBlockN - 1) / mla::kBlockN;
    const int sched_pairs = persistent ? persistent_pairs() : 0;
    const TailPlan tail = (range || persistent) ? TailPlan{} : launch_tail_plan(topk > 0, item_tiles, num_splits, splits);
    // a range of splits writes its partials to the caller's buffers: no partials in the workspace
    const Layout lay = make_layout(batch, total_q, range ? 1 : splits, topk > 0, tail.cap, sched_pairs);
    if (!workspace || workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MLA_ERR_WORKSPACE;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* status = reinterpret_cast<int*>(ws + lay.status);
    int32_t* item_count = reinterpret_cast<int32_t*>(ws + lay.item_count);
    int32_t* q_off = reinterpret_cast<int32_t*>(ws + lay.q_off);
    int32_t* req_state = reinterpret_cast<int32_t*>(ws + lay.req_state);
    uint64_t* anc = reinterpret_cast<uint64_t*>(ws + lay.anc);
    int2* items = reinterpret_cast<int2*>(ws + lay.items);
    const bool ws_parts = splits > 1 || tail.cap > 0 || persistent;
    float* part_out = range ? out : ws_parts ? reinterpret_cast<float*>(ws + lay.part_out) : nullptr;
    float* part_lse = range ? lse : ws_parts ? reinterpret_cast<float*>(ws + lay.part_lse) : nullptr;
    int32_t* tail_k = tail.cap > 0 ? reinterpret_cast<int32_t*>(ws + lay.tail_k) : nullptr;

    CUtensorMap map_lat, map_rope;
    const int enc = encode_maps(kv_cache, static_cast<long long>(num_pages) * page_size,
                                topk > 0 ? 1u : static_cast<unsigned>(mla::kBlockN), &map_lat, &map_rope);
    if (enc != MLA_OK) return enc;

    // ---- prep: offsets, ancestor bit sets, validation, work list ----
    mla::PrepParams pp{};
    pp.block_table = block_table;
    pp.seq_lens = seq_lens;
    pp.tree_parent = tree_parent;
    pp.n_tree = n_tree;
    pp.q_off = q_off;
    pp.req_state = req_state;
    pp.order = reinterpret_cast<int32_t*>(ws + lay.order);
    pp.item_off = reinterpret_cast<int32_t*>(ws + lay.item_off);
    pp.anc = anc;
    pp.items = items;
    pp.item_count = item_count;
    pp.status = status;
    pp.batch = batch;
    pp.total_q = total_q;
    pp.page_size = page_size;
    pp.max_pages = max_pages_per_seq;
    pp.num_pages = num_pages;
    pp.max_items = lay.max_items;
    pp.tok_req = topk > 0 ? reinterpret_cast<int32_t*>(ws + lay.tok_req) : nullptr;
    pp.allow_unused_rows = graph_capture ? 1 : 0;
    int32_t* merge_cnt = !range && (splits == 2 || tail.cap > 0 || persistent)
                             ? reinterpret_cast<int32_t*>(ws + lay.merge_cnt)
                             : nullptr;
    pp.tail_k = tail_k;
    pp.tail_cap = tail.cap;
    pp.pairs = sm_count_of_current() / 2;
    pp.zero_words = merge_cnt;
    pp.zero_count = merge_cnt ? 4 * lay.max_items : 0;
    long long* woff = persistent ? reinterpret_cast<long long*>(ws + lay.woff) : nullptr;
    long long* pair_begin = persistent ? reinterpret_cast<long long*>(ws + lay.pair_begin) : nullptr;
    int32_t* pair_item = persistent ? reinterpret_cast<int32_t*>(ws + lay.pair_item) : nullptr;
    int32_t* item_first_pair = persistent ? reinterpret_cast<int32_t*>(ws + lay.item_first_pair) : nullptr;
    int32_t* rounds = persistent ? reinterpret_cast<int32_t*>(ws + lay.rounds) : nullptr;
    pp.rounds = rounds;
    pp.woff = woff;
    pp.pair_begin = pair_begin;
    pp.pair_item = pair_item;
    pp.item_first_pair = item_first_pair;
    pp.sched_pairs = sched_pairs;
    pp.min_piece = kMinPieceTiles;
    pp.topk = topk;
    mla::mla_prep_kernel<<<1, mla::kPrepThreads, 0, stream>>>(pp);
    if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
    if (topk > 0) {
        const long long entries = static_cast<long long>(total_q) * topk;
        const long long want = (entries + 4LL * mla::kCheckThreads - 1) / (4LL * mla::kCheckThreads);
        const unsigned blocks =
            static_cast<unsigned>(std::max(1LL, std::min<long long>(want, 4LL * sm_count_of_current())));
        if (launch_dependent(mla::mla_topk_check_kernel, dim3(blocks), dim3(mla::kCheckThreads), 0, stream, topk_idx,
                             topk, entries, pp.tok_req, seq_lens, n_tree, batch, req_state, status) != cudaSuccess)
            return MLA_ERR_CUDA;
    }

    // ---- fused verify attention ----
    mla::VerifyParams vp{};
    vp.q_lat = static_cast<const uint16_t*>(q_lat);
    vp.q_rope = static_cast<const uint16_t*>(q_rope);
    vp.block_table = block_table;
    vp.seq_lens = seq_lens;
    vp.n_tree = n_tree;
    vp.q_off = q_off;
    vp.anc = anc;
    vp.req_state = req_state;
    vp.items = items;
    vp.item_count = item_count;
    vp.status = status;
    vp.out = out;
    vp.lse = lse;
    vp.part_out = part_out;
    vp.part_lse = part_lse;
    vp.batch = batch;
    vp.total_q = total_q;
    vp.page_size = page_size;
    vp.max_pages = max_pages_per_seq;
    vp.num_pages = num_pages;
    vp.num_splits = splits;
    vp.split_share = splits == 2 && !range ? first_split_share(items_bound_of(batch, total_q, max_tree), item_tiles,
                                                               sm_count_of_current() / 2)
                                           : 0;   // a range of splits uses equal shares
    vp.split_base = range ? split_begin : 0;
    vp.tail_cap = tail.cap;
    vp.tail_share = tail.share;
    vp.tail_k = tail_k;
    vp.max_items = lay.max_items;
    vp.scale_log2 = scale * 1.4426950408889634f;
    vp.timeout_ns = kDefaultTimeoutNs;
    vp.topk_idx = topk_idx;
    vp.topk = topk;
    vp.kv = static_cast<const uint16_t*>(kv_cache);
    vp.merge_cnt = merge_cnt;
    vp.woff = woff;
    vp.pair_begin = pair_begin;
    vp.pair_item = pair_item;
    vp.item_first_pair = item_first_pair;
    vp.rounds = rounds;
    vp.pairs = sched_pairs;
    const dim3 grid(2u * static_cast<unsigned>(persistent ? sched_pairs : lay.max_items + tail.cap),
                    static_cast<unsigned>(range ? split_count : splits), 1u);
    const bool prof = !graph_capture && g_prof_begin && g_prof_end;
    if (prof && cudaEventRecord(g_prof_begin, stream) != cudaSuccess) return MLA_ERR_CUDA;
    const int sched = persistent ? mla::kSchedPersistent : merge_cnt != nullptr ? mla::kSchedMerge : mla::kSchedPlain;
    auto* kernel = topk > 0 ? (sched == mla::kSchedPersistent ? mla::mla_verify_kernel<true, mla::kSchedPersistent>
                               : sched == mla::kSchedMerge    ? mla::mla_verify_kernel<true, mla::kSchedMerge>
                                                              : mla::mla_verify_kernel<true, mla::kSchedPlain>)
                            : (sched == mla::kSchedPersistent ? mla::mla_verify_kernel<false, mla::kSchedPersistent>
                               : sched == mla::kSchedMerge    ? mla::mla_verify_kernel<false, mla::kSchedMerge>
                                                              : mla::mla_verify_kernel<false, mla::kSchedPlain>);
    if (launch_dependent(kernel, grid, dim3(topk > 0 ? mla::kThreadsSparse : mla::kThreads), mla::kSmemBytes, stream,
                         vp, map_lat, map_rope) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (prof && cudaEventRecord(g_prof_end, stream) != cudaSuccess) return MLA_ERR_CUDA;

    // ---- merge of the split partials (two splits are merged inside the verify kernel) ----
    if (range) return MLA_OK;   // the caller merges the partials of all splits (mla_split_combine)
    if (splits > 2)
        return launch_combine(part_out, part_lse, splits, static_cast<long long>(total_q) * MLA_NUM_HEADS, out, lse,
                              stream);
    return MLA_OK;
}

int mla_verify_attn(const void* q_lat, const void* q_rope, const void* kv_cache, const int32_t* block_table,
                    const int32_t* seq_lens, const int32_t* tree_parent, const int32_t* n_tree, float scale,
                    float* out, float* lse, cudaStream_t stream, int batch, int total_q, int max_tree,
                    int max_seq_len, int num_heads, int page_size, int num_pages, int max_pages_per_seq,
                    int num_splits, void* workspace, size_t workspace_bytes) {
    return verify_impl(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree, scale, out, lse, stream,
                       batch, total_q, max_tree, max_seq_len, num_heads, page_size, num_pages, max_pages_per_seq,
                       num_splits, workspace, workspace_bytes, nullptr, 0);
}

int mla_verify_attn_split_range(const void* q_lat, const void* q_rope, const void* kv_cache,
                                const int32_t* block_table, const int32_t* seq_lens, const int32_t* tree_parent,
                                const int32_t* n_tree, float scale, float* part_out, float* part_lse,
                                cudaStream_t stream, int batch, int total_q, int max_tree, int max_seq_len,
                                int num_heads, int page_size, int num_pages, int max_pages_per_seq, int num_splits,
                                int split_begin, int split_count, void* workspace, size_t workspace_bytes) {
    if (split_count < 1) return MLA_ERR_INVALID_ARG;
    return verify_impl(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree, scale, part_out, part_lse,
                       stream, batch, total_q, max_tree, max_seq_len, num_heads, page_size, num_pages,
                       max_pages_per_seq, num_splits, workspace, workspace_bytes, nullptr, 0, false, split_begin,
                       split_count);
}

int mla_verify_sparse_num_splits(int batch, int total_q, int max_tree, int topk, int num_heads, int requested) {
    if (batch < 0 || total_q < 0 || max_tree < 0 || requested < MLA_SPLITS_PERSISTENT || topk < 1)
        return -MLA_ERR_INVALID_ARG;
    if (num_heads != MLA_NUM_HEADS || topk > MLA_MAX_TOPK) return -MLA_ERR_UNSUPPORTED;
    if (requested == MLA_SPLITS_PERSISTENT) return 0;
    if (requested > 0) return std::min(requested, MLA_MAX_SPLITS);
    return choose_splits_tiles(batch, total_q, max_tree, sparse_tiles(topk));
}

size_t mla_verify_sparse_workspace_size(int batch, int total_q, int max_tree, int topk, int num_heads,
                                        int num_splits) {
    const int s = mla_verify_sparse_num_splits(batch, total_q, max_tree, topk, num_heads, num_splits);
    if (s < 0) return 0;
    if (s == 0)
        return make_layout(batch, total_q, 1, true, 0, persistent_pairs()).total;
    const TailPlan tp = launch_tail_plan(true, sparse_tiles(topk), num_splits, s);
    return make_layout(batch, total_q, s, true, tp.cap).total;
}

int mla_verify_sparse_attn(const void* q_lat, const void* q_rope, const void* kv_cache, const int32_t* block_table,
                           const int32_t* seq_lens, const int32_t* tree_parent, const int32_t* n_tree,
                           const int32_t* topk_idx, int topk, float scale, float* out, float* lse,
                           cudaStream_t stream, int batch, int total_q, int max_tree, int max_seq_len, int num_heads,
                           int page_size, int num_pages, int max_pages_per_seq, int num_splits, void* workspace,
                           size_t workspace_bytes) {
    if (topk < 1) return MLA_ERR_INVALID_ARG;
    if (topk > MLA_MAX_TOPK) return MLA_ERR_UNSUPPORTED;
    if (batch > 0 && total_q > 0 && !topk_idx) return MLA_ERR_INVALID_ARG;
    return verify_impl(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree, scale, out, lse, stream,
                       batch, total_q, max_tree, max_seq_len, num_heads, page_size, num_pages, max_pages_per_seq,
                       num_splits, workspace, workspace_bytes, topk_idx, topk);
}

int mla_split_combine(const float* part_out, const float* part_lse, int num_splits, int rows, float* out, float* lse,
                      cudaStream_t stream) {
    if (num_splits < 1 || num_splits > MLA_MAX_SPLITS || rows < 0) return MLA_ERR_INVALID_ARG;
    if (rows == 0) return MLA_OK;
    if (!part_out || !part_lse || !out || !lse) return MLA_ERR_INVALID_ARG;
    if (!aligned16(part_out) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
    return launch_combine(part_out, part_lse, num_splits, rows, out, lse, stream);
}

int mla_set_profile_events(cudaEvent_t begin, cudaEvent_t end) {
    if ((begin == nullptr) != (end == nullptr)) return MLA_ERR_INVALID_ARG;
    g_prof_begin = begin;
    g_prof_end = end;
    return MLA_OK;
}

// Shared argument checks of the two paged-cache steps; fills the common parameters.
static int kv_op_setup(void* kv_cache, const int32_t* block_table, const int32_t* seq_lens, const int32_t* n_tree,
                       int batch, int total_q, int page_size, int num_pages, int max_pages_per_seq, void* workspace,
                       size_t workspace_bytes, mla::KvOpParams* kp) {
    if (batch < 0 || total_q < 0 || page_size <= 0 || num_pages < 0 || max_pages_per_seq < 0)
        return MLA_ERR_INVALID_ARG;
    if (static_cast<long long>(num_pages) * page_size > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < sizeof(int) || (reinterpret_cast<uintptr_t>(workspace) & 3u))
        return MLA_ERR_WORKSPACE;
    if (batch > 0 && (!kv_cache || !block_table || !seq_lens || !n_tree || num_pages == 0 || max_pages_per_seq == 0))
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(kv_cache)) return MLA_ERR_INVALID_ARG;
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices || !g_dev[dev].ready) return MLA_ERR_NOT_INITIALIZED;
    *kp = mla::KvOpParams{};
    kp->cache = static_cast<uint4*>(kv_cache);
    kp->block_table = block_table;
    kp->seq_lens = seq_lens;
    kp->n_tree = n_tree;
    kp->status = static_cast<int*>(workspace);
    kp->batch = batch;
    kp->total_q = total_q;
    kp->page_size = page_size;
    kp->max_pages = max_pages_per_seq;
    kp->num_pages = num_pages;
    return MLA_OK;
}

size_t mla_tree_kv_workspace_size(void) { return 256; }

int mla_tree_kv_append(const void* tree_kv, void* kv_cache, const int32_t* block_table, const int32_t* seq_lens,
                       const int32_t* n_tree, cudaStream_t stream, int batch, int total_q, int page_size,
                       int num_pages, int max_pages_per_seq, void* workspace, size_t workspace_bytes) {
    mla::KvOpParams kp;
    const int rc = kv_op_setup(kv_cache, block_table, seq_lens, n_tree, batch, total_q, page_size, num_pages,
                               max_pages_per_seq, workspace, workspace_bytes, &kp);
    if (rc != MLA_OK) return rc;
    if (batch > 0 && total_q > 0 && (!tree_kv || !aligned16(tree_kv))) return MLA_ERR_INVALID_ARG;
    kp.tree_kv = static_cast<const uint4*>(tree_kv);
    if (cudaMemsetAsync(workspace, 0, sizeof(int), stream) != cudaSuccess) return MLA_ERR_CUDA;
    if (batch == 0) return MLA_OK;
    mla::mla_tree_append_kernel<<<batch, mla::kKvOpThreads, 0, stream>>>(kp);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_tree_kv_accept(void* kv_cache, const int32_t* block_table, const int32_t* seq_lens, const int32_t* n_tree,
                       const int32_t* tree_parent, const int32_t* accept_len, const int32_t* accept_idx,
                       int32_t* new_seq_lens, cudaStream_t stream, int batch, int total_q, int page_size,
                       int num_pages, int max_pages_per_seq, void* workspace, size_t workspace_bytes) {
    mla::KvOpParams kp;
    const int rc = kv_op_setup(kv_cache, block_table, seq_lens, n_tree, batch, total_q, page_size, num_pages,
                               max_pages_per_seq, workspace, workspace_bytes, &kp);
    if (rc != MLA_OK) return rc;
    if (batch > 0 && (!accept_len || !new_seq_lens || (total_q > 0 && (!tree_parent || !accept_idx))))
        return MLA_ERR_INVALID_ARG;
    kp.tree_parent = tree_parent;
    kp.accept_len = accept_len;
    kp.accept_idx = accept_idx;
    kp.new_seq_lens = new_seq_lens;
    if (cudaMemsetAsync(workspace, 0, sizeof(int), stream) != cudaSuccess) return MLA_ERR_CUDA;
    if (batch == 0) return MLA_OK;
    mla::mla_tree_accept_kernel<<<batch, mla::kKvOpThreads, mla::kAcceptSmemBytes, stream>>>(kp);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_read_status(const void* workspace, int* device_status) {
    if (!workspace || !device_status) return MLA_ERR_INVALID_ARG;
    int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
    *device_status = v;
    return MLA_OK;
}

// ---------------------------------------------------------------- graph replay

struct mla_verify_graph {
    cudaGraphExec_t exec = nullptr;
    int device = -1;
    int max_batch = 0;
    int32_t* seq_lens = nullptr;
    int32_t* n_tree = nullptr;
};

int mla_verify_graph_create(const void* q_lat, const void* q_rope, const void* kv_cache, const int32_t* block_table,
                            int32_t* seq_lens, const int32_t* tree_parent, int32_t* n_tree, const int32_t* topk_idx,
                            int topk, float scale, float* out, float* lse, int max_batch, int max_total_q,
                            int max_tree, int max_seq_len, int num_heads, int page_size, int num_pages,
                            int max_pages_per_seq, int num_splits, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream, mla_verify_graph** graph) {
    if (!graph) return MLA_ERR_INVALID_ARG;
    *graph = nullptr;
    if (max_batch <= 0 || max_total_q <= 0 || !seq_lens || !n_tree || topk < 0) return MLA_ERR_INVALID_ARG;
    if (topk > MLA_MAX_TOPK) return MLA_ERR_UNSUPPORTED;
    if (topk > 0 && !topk_idx) return MLA_ERR_INVALID_ARG;
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices || !g_dev[dev].ready) return MLA_ERR_NOT_INITIALIZED;
    // the legacy and per-thread default streams cannot be captured: use a private one
    cudaStream_t cap = stream, own = nullptr;
    if (stream == nullptr || stream == cudaStreamLegacy || stream == cudaStreamPerThread) {
        if (cudaStreamCreateWithFlags(&own, cudaStreamNonBlocking) != cudaSuccess) return MLA_ERR_CUDA;
        cap = own;
    }
    cudaGraph_t def = nullptr;
    int rc = MLA_OK;
    if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        rc = MLA_ERR_CUDA;
    } else {
        rc = verify_impl(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree, scale, out, lse, cap,
                         max_batch, max_total_q, max_tree, max_seq_len, num_heads, page_size, num_pages,
                         max_pages_per_seq, num_splits, workspace, workspace_bytes, topk > 0 ? topk_idx : nullptr,
                         topk, true);
        const cudaError_t e = cudaStreamEndCapture(cap, &def);
        if (rc == MLA_OK && e != cudaSuccess) rc = MLA_ERR_CUDA;
    }
    cudaGraphExec_t exec = nullptr;
    if (rc == MLA_OK && cudaGraphInstantiate(&exec, def, 0) != cudaSuccess) rc = MLA_ERR_CUDA;
    if (def) cudaGraphDestroy(def);
    if (own) cudaStreamDestroy(own);
    mla_verify_graph* g = rc == MLA_OK ? new (std::nothrow) mla_verify_graph : nullptr;
    if (rc == MLA_OK && !g) rc = MLA_ERR_CUDA;
    if (rc != MLA_OK) {
        if (exec) cudaGraphExecDestroy(exec);
        return rc;
    }
    g->exec = exec;
    g->device = dev;
    g->max_batch = max_batch;
    g->seq_lens = seq_lens;
    g->n_tree = n_tree;
    *graph = g;
    return MLA_OK;
}

int mla_verify_graph_launch(mla_verify_graph* graph, int batch, cudaStream_t stream) {
    if (!graph || !graph->exec || batch < 0 || batch > graph->max_batch) return MLA_ERR_INVALID_ARG;
    if (current_device() != graph->device) return MLA_ERR_INVALID_ARG;
    if (batch < graph->max_batch) {
        // requests past `batch` become empty: no tree tokens, no keys, no work items
        const size_t bytes = sizeof(int32_t) * static_cast<size_t>(graph->max_batch - batch);
        if (cudaMemsetAsync(graph->n_tree + batch, 0, bytes, stream) != cudaSuccess ||
            cudaMemsetAsync(graph->seq_lens + batch, 0, bytes, stream) != cudaSuccess)
            return MLA_ERR_CUDA;
    }
    return cudaGraphLaunch(graph->exec, stream) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_verify_graph_destroy(mla_verify_graph* graph) {
    if (!graph) return MLA_OK;
    if (graph->exec && cudaGraphExecDestroy(graph->exec) != cudaSuccess) {
        delete graph;
        return MLA_ERR_CUDA;
    }
    delete graph;
    return MLA_OK;
}

}  // extern "C"


#ifdef MLA_FAULT_INJECTION
// Test build only (not part of the shipped library's interface): choose the
// fault the verify kernel injects from now on (0 = none; see verify_kernel.cuh).
extern "C" int mla_debug_set_fault(int kind) {
    return cudaMemcpyToSymbol(mla::g_fault_kind, &kind, sizeof(int)) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
#endif
