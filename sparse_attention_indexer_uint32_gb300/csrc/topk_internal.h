// topk_internal.h -- launch parameters, workspace layout and shared-memory
// layout shared by the host dispatcher and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace topkidx {

constexpr int kBins = 2048;             // bins per histogram round (11 bits)
constexpr int kBinBits = 11;
constexpr int kBinsX = kBins + 64;      // + control slots carried through cluster merges
constexpr int kSlotOverflow = kBins;    // merged slot: some block's candidate buffer overflowed
constexpr int kFinish = 32;             // a warp-wide compare-and-swap sort finishes <= 32 candidates
constexpr int kMaxSamples = 2048;       // gate samples per row (held 2048 / threads per thread)
constexpr int kItemsMax = 256;          // work items staged in shared memory per window
// The warp-per-row kernel (short rows in large batches).
constexpr int kWarpThreads = 256;       // 8 warps per block, one row each at a time
constexpr uint32_t kWarpCap = 1536;     // candidate buffer entries per warp
constexpr uint32_t kWarpMaxLen = 16384; // longest row it takes (16-bit positions, 2 KB tie bitmap)
constexpr int32_t kWarpMaxK = 512;      // largest k it takes (the buffer holds about 3k gated elements)
constexpr int kMaxK = 2048;
// Bounded device waits: the default limit of a wait for a bulk copy, and the
// limit of the drain that a block which gave up runs before it exits (its own
// copies still in flight must land first, whatever the caller's limit).
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 2000000000ull;
constexpr int kMaxCluster = 16;
constexpr int kSlotRankMin = kBins + 1;                   // + rank: a block's smallest key in a round's range
constexpr int kSlotRankMax = kSlotRankMin + kMaxCluster;  // + rank: its largest
static_assert(kSlotRankMax + kMaxCluster <= kBinsX, "rank slots fit the histogram padding");

// Workspace written by the plan kernel.
constexpr uint32_t kPlanMagic = 0x544f504bu;  // "TOPK"
struct PlanHeader {
    uint32_t magic;
    int32_t batch;
    int32_t max_seq_len;
    int32_t long_threshold;
    int32_t n_long;
    int32_t n_short;
    uint32_t flags;
    int32_t identity;  // 1: every row has the same class and length bucket, so the
                       // one non-empty list is rows 0..batch-1 in order (not written)
    int32_t reserved[8];
};
static_assert(sizeof(PlanHeader) == 64, "plan header is 64 bytes");

// The segment-split path (topk_split.cu): a batch of up to kSplitMaxRows
// rows is cut into segments that a persistent grid streams; each row's gated
// candidates are collected in the workspace, and the block that finishes a
// row's last segment resolves the row.
constexpr int32_t kSplitMaxRows = 128;     // rows of one split launch (the whole batch)
constexpr uint32_t kSplitCap = 8192;       // candidate entries per row (64-bit composites)
constexpr int32_t kSplitMaxUnits = 16384;  // segments of one launch
constexpr int kSplitThreads = 512;         // threads per block of the streaming kernel
constexpr int kSplitGateThreads = 512;     // threads per block of the gate kernel (one row each)
constexpr int kSplitMaxSamples = 8192;     // gate samples per row

// Per-row state of the split path, rewritten by the gate kernel every call.
struct SplitRow {
    uint32_t lo;      // gate key: elements with key > lo are candidates, key == lo are counted
    uint32_t n_gt;    // candidates reserved (may run past kSplitCap: overflow)
    uint32_t n_eq;    // elements with key == lo
    uint32_t done;    // segments finished
    int32_t len;      // clamped seq_len
    int32_t nunits;   // segments of the row (0: the gate kernel wrote the row)
    int32_t pad[2];
};
static_assert(sizeof(SplitRow) == 32, "split row state is 32 bytes");
struct SplitHeader {
    uint32_t next_unit;    // segments handed out so far
    uint32_t total_units;  // segments of the launch
    uint32_t pad[14];
};
static_assert(sizeof(SplitHeader) == 64, "split header is 64 bytes");

__host__ __device__ constexpr size_t round256(size_t b) { return (b + 255) / 256 * 256; }
__host__ __device__ constexpr int32_t split_rows_of(int32_t batch) {
    return batch < kSplitMaxRows ? batch : kSplitMaxRows;
}
// The plan's own part: header + the two row lists.
__host__ __device__ constexpr size_t plan_core_bytes(int32_t batch) {
    return round256(sizeof(PlanHeader) + 2 * sizeof(int32_t) * static_cast<size_t>(batch));
}
// The split path's fixed part (header, row states, segment starts, per-segment
// tie counts), then kSplitCap candidates per row.
__host__ __device__ constexpr size_t split_fixed_bytes(int32_t rows) {
    return round256(sizeof(SplitHeader) + sizeof(SplitRow) * static_cast<size_t>(rows) +
                    sizeof(int32_t) * static_cast<size_t>(rows + 1) +
                    sizeof(uint32_t) * static_cast<size_t>(kSplitMaxUnits));
}
__host__ __device__ constexpr size_t split_bytes(int32_t batch) {
    return split_fixed_bytes(split_rows_of(batch)) +
           sizeof(uint64_t) * static_cast<size_t>(kSplitCap) * static_cast<size_t>(split_rows_of(batch));
}
__host__ __device__ constexpr size_t plan_bytes(int32_t batch) {
    return batch < 1 ? 0 : plan_core_bytes(batch) + split_bytes(batch);
}
struct SplitRegion {
    SplitHeader* hdr;
    SplitRow* rows;
    int32_t* unit_start;  // [rows + 1]: first segment of each row, then the total
    uint32_t* unit_ties;  // [kSplitMaxUnits]: elements with key == lo per segment
    uint64_t* cand;       // [rows][kSplitCap]: (key << 32) | ~position
};
__host__ __device__ inline SplitRegion split_region(void* ws, int32_t batch) {
    const int32_t rows = split_rows_of(batch);
    char* b = static_cast<char*>(ws) + plan_core_bytes(batch);
    SplitRegion r;
    r.hdr = reinterpret_cast<SplitHeader*>(b);
    r.rows = reinterpret_cast<SplitRow*>(b + sizeof(SplitHeader));
    r.unit_start = reinterpret_cast<int32_t*>(b + sizeof(SplitHeader) + sizeof(SplitRow) * rows);
    r.unit_ties = reinterpret_cast<uint32_t*>(b + sizeof(SplitHeader) + sizeof(SplitRow) * rows +
                                              sizeof(int32_t) * (rows + 1));
    r.cand = reinterpret_cast<uint64_t*>(b + split_fixed_bytes(rows));
    return r;
}
__host__ __device__ inline int32_t* plan_long_list(void* ws) {
    return reinterpret_cast<int32_t*>(static_cast<char*>(ws) + sizeof(PlanHeader));
}
__host__ __device__ inline int32_t* plan_short_list(void* ws, int32_t batch) {
    return plan_long_list(ws) + batch;
}

// Parameters of the select kernel (one block, or one cluster, per row).
struct SelectParams {
    const float* scores;
    int64_t row_stride;
    const int32_t* seq_lens;
    int32_t batch;
    int32_t max_seq_len;
    const int32_t* page_table;
    int64_t pt_stride;
    int32_t log2_page;
    int32_t k;
    int32_t* out;
    int32_t* raw_out;
    const int32_t* items;     // row ids of this kernel's work list (nullptr: rows 0..n-1)
    const int32_t* n_items_dev;  // device count of items (nullptr: n_items_host)
    int32_t n_items_host;
    const int32_t* items2;    // optional second list, taken after the first (nullptr: none)
    const int32_t* n_items2_dev;
    const PlanHeader* plan;   // the planned workspace (checked against batch / max_seq_len)
    uint32_t* flags;          // device flag word (TOPK_FLAG_*)
    int32_t tile;             // floats per bulk copy, multiple of 4
    int32_t stages;           // bulk-copy ring depth
    int32_t cap;              // candidate buffer entries per block
    int32_t samples;          // gate samples per row
    float gate_fill;          // share of the candidate buffer the gate aims to fill
    int32_t gate_refresh;     // single block, 256 threads: tighten the gate every this many copies (0: never)
    int32_t force_two_pass;
    int32_t disable_gate;
    uint64_t timeout_ns;
};

// What a select kernel reads of the plan before its first row: the header
// check and the two work-list counts.  Every field is loaded before any is
// tested, so the loads go out together (one trip to memory at the kernel's
// start instead of two dependent ones).
struct PlanView {
    bool ok;          // the plan belongs to this batch (or there is none)
    bool identity;    // item i is row i (the plan wrote no lists)
    int32_t n_first;  // items taken from `items`
    int32_t n_items;  // n_first + items taken from `items2`
};

#ifdef __CUDACC__
__device__ __forceinline__ PlanView read_plan(const SelectParams& p) {
    uint32_t magic = kPlanMagic;
    int32_t batch = p.batch, max_len = p.max_seq_len, identity = 0;
    if (p.plan) {
        magic = p.plan->magic;
        batch = p.plan->batch;
        max_len = p.plan->max_seq_len;
        identity = p.plan->identity;
    }
    const int32_t a = p.n_items_dev ? *p.n_items_dev : p.n_items_host;
    const int32_t b = p.items2 ? *p.n_items2_dev : 0;
    PlanView v;
    v.ok = magic == kPlanMagic && batch == p.batch && max_len == p.max_seq_len;
    v.identity = p.plan != nullptr && identity != 0;
    v.n_first = min(a, p.batch);
    const int32_t n_second = p.items2 ? min(b, p.batch - v.n_first) : 0;
    v.n_items = v.n_first + max(n_second, 0);
    return v;
}
#endif

// Parameters of the two kernels of the segment-split path.
struct SplitParams {
    const float* scores;
    int64_t row_stride;
    const int32_t* seq_lens;
    int32_t batch;            // <= kSplitMaxRows; rows 0..batch-1 in order
    int32_t max_seq_len;
    const int32_t* page_table;
    int64_t pt_stride;
    int32_t log2_page;
    int32_t k;
    int32_t* out;
    int32_t* raw_out;
    const PlanHeader* plan;
    uint32_t* flags;
    SplitRegion ws;
    int32_t seg;              // elements per segment: a power of two, 4096..1048576
    int32_t samples;          // gate samples per row, <= kSplitMaxSamples
    int32_t full_resolve;     // 1: every row is resolved by the full-row path (tests)
    int32_t disable_gate;     // 1: gate key 0 (every element is a candidate)
};

struct __align__(16) Control {
    uint32_t ncand;       // candidates pushed in the current pass
    uint32_t nemit;       // entries in the local emit list
    uint32_t nfin;        // entries in the finish list
    uint32_t smax;        // largest sample key
    uint32_t res_bin, res_above, res_count, res_total;  // result of the last histogram scan
    uint32_t rank_eq[kMaxCluster];   // per-rank copies of the threshold key (tie quotas)
    uint32_t err;
    uint32_t res_local;   // the local (un-merged) count of the bin found by the last scan
    uint32_t win_tiles;   // bulk-copy tiles in the current window of work items
    uint32_t out_cursor[2];  // rank 0 of a cluster: output slots handed out, by row parity
    uint32_t out_base;       // this block's first output slot of the current row
    uint32_t tkey;           // gate refresh: the tightened gate key of the current row (0: none yet)
    uint32_t pad;
    uint32_t rnd_min[2], rnd_max[2], rnd_cnt[2];  // a cluster round's in-range key min/max/count, by parity
    uint32_t pad2[2];
};

struct Layout {
    uint32_t ring, hist_a, hist_b, hist_m, cand_key, cand_idx, emit, fin_key, fin_idx, warp_tot, ctl;
    uint32_t items_row, items_len, items_tiles, items_tile_start, claim, mbar, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline Layout make_layout(int cluster, int tile, int stages, int cap, int k) {
    Layout l;
    uint32_t o = 0;
    l.ring = o;
    o = align_up(o + static_cast<uint32_t>(stages) * tile * 4u, 128);
    l.hist_a = o;
    o += kBinsX * 4u;
    l.hist_b = o;
    o += kBinsX * 4u;
    l.hist_m = o;
    o += cluster > 1 ? kBinsX * 4u : 0u;
    l.cand_key = o;
    o += static_cast<uint32_t>(cap) * 4u;
    l.cand_idx = o;
    o += static_cast<uint32_t>(cap) * 4u;
    l.emit = o;
    o += align_up(static_cast<uint32_t>(k), 4) * 4u;
    l.fin_key = o;
    o += kFinish * 4u;
    l.fin_idx = o;
    o += kFinish * 4u;
    l.warp_tot = o;
    o += 32 * 4u;
    l.ctl = o;
    o += align_up(sizeof(Control), 16);
    l.items_row = o;
    o += kItemsMax * 4u;
    l.items_len = o;
    o += kItemsMax * 4u;
    l.items_tiles = o;
    o += kItemsMax * 4u;
    l.items_tile_start = o;
    o += kItemsMax * 4u;
    l.claim = o;
    o += align_up(static_cast<uint32_t>(stages), 4) * 4u;
    l.mbar = align_up(o, 8);
    o = l.mbar + 2u * stages * 8u;
    l.total = align_up(o, 128);
    return l;
}

// The warp-specialised single-block kernel (topk_stream.cu): 8 streaming
// warps run pass 1 of row q while 4 or 8 resolving warps finish row q - 1
// and compute the gate of row q + 1, with two candidate-buffer / histogram
// sets.
constexpr int kStreamWarps = 8;
constexpr int kStreamItemsMax = 32;     // work items per window of the warp-specialised kernel
constexpr int32_t kStreamMaxLen = 65536;  // longest row it takes (16-bit candidate positions)

struct __align__(16) SetControl {
    uint32_t ncand[2];  // candidates in set b (pass 1, or a collect pass)
    uint32_t lo[2];     // gate key of the row held by set b
    uint32_t shift[2];  // bin shift of set b's first histogram
    uint32_t ncand_seen; // the resolving warps' snapshot of the row's candidate count
    uint32_t pad;
};

struct StreamLayout {
    uint32_t ring, hist[2], cand_key[2], cand_idx[2], emit, fin_key, fin_idx, warp_tot, ctl, sctl;
    uint32_t items_row, items_len, items_tiles, items_tile_start, claim, mbar, total;
};

__host__ __device__ inline StreamLayout make_stream_layout(int tile, int stages, int cap, int k) {
    StreamLayout l;
    uint32_t o = 0;
    l.ring = o;
    o = align_up(o + static_cast<uint32_t>(stages) * tile * 4u, 128);
    for (int b = 0; b < 2; ++b) {  // no cluster-merge slots: kBins bins
        l.hist[b] = o;
        o += kBins * 4u;
    }
    for (int b = 0; b < 2; ++b) {  // 32-bit keys, 16-bit positions
        l.cand_key[b] = o;
        o += static_cast<uint32_t>(cap) * 4u;
        l.cand_idx[b] = o;
        o += align_up(static_cast<uint32_t>(cap) * 2u, 16);
    }
    l.emit = o;
    o += align_up(static_cast<uint32_t>(k), 4) * 4u;
    l.fin_key = o;
    o += kFinish * 4u;
    l.fin_idx = o;
    o += kFinish * 4u;
    l.warp_tot = o;
    o += 32 * 4u;
    l.ctl = o;
    o += align_up(sizeof(Control), 16);
    l.sctl = o;
    o += align_up(sizeof(SetControl), 16);
    l.items_row = o;
    o += kStreamItemsMax * 4u;
    l.items_len = o;
    o += kStreamItemsMax * 4u;
    l.items_tiles = o;
    o += kStreamItemsMax * 4u;
    l.items_tile_start = o;
    o += kStreamItemsMax * 4u;
    l.claim = o;
    o += align_up(static_cast<uint32_t>(stages), 4) * 4u;
    l.mbar = align_up(o, 8);
    o = l.mbar + (2u * stages + 4u) * 8u;  // full[stages], empty[stages], ready[2], done[2]
    l.total = align_up(o, 128);
    return l;
}

// Host-side launchers (defined in topk_kernels.cu).
cudaError_t launch_plan(const int32_t* seq_lens, int32_t batch, int32_t max_seq_len, int32_t long_threshold,
                        void* workspace, cudaStream_t stream);
// threads: 256 or 512 per block when cluster == 1; 512 for clusters.
cudaError_t launch_select(const SelectParams& p, int cluster, int threads, int grid_units, size_t smem,
                          cudaStream_t stream);
cudaError_t select_occupancy(int cluster, int threads, size_t smem, int* units_out);
cudaError_t launch_page_transform(const int32_t* raw, int32_t batch, int32_t k, const int32_t* page_table,
                                  int64_t pt_stride, int32_t log2_page, int32_t* out, cudaStream_t stream);
cudaError_t launch_key_map(const float* x, int64_t n, uint32_t* keys, cudaStream_t stream);
// programmatic: launched with programmatic stream serialization (its blocks
// are placed while the plan finishes).
cudaError_t launch_warp_select(const SelectParams& p, int grid, bool programmatic, cudaStream_t stream);
// The warp-specialised single-block kernel (topk_stream.cu).
// resolve_warps: 4 (two blocks per SM) or 8 (one block per SM).
cudaError_t launch_stream_select(const SelectParams& p, int resolve_warps, int grid, size_t smem,
                                 cudaStream_t stream);
cudaError_t stream_select_occupancy(int resolve_warps, size_t smem, int* units_out);
cudaError_t warp_select_occupancy(int* units_out);
size_t warp_select_smem_bytes();
// The segment-split path (topk_split.cu): the gate kernel (one block per
// row), then the persistent streaming kernel on `grid` blocks.
cudaError_t launch_split(const SplitParams& p, int grid, cudaStream_t stream);
cudaError_t split_occupancy(int* blocks_out);

}  // namespace topkidx
