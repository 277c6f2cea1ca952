// topkidx_api.cu -- the C ABI declared in include/topkidx.h: argument checks,
// the path split chosen by the plan, launch sizing and error mapping.  All
// compute runs in the kernels of topk_kernels.cu; there is no host fallback.

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "topk_internal.h"
#include "topkidx.h"

using namespace topkidx;

namespace {

std::mutex g_mutex;
thread_local char g_last_error[256] = "";

// Records a failed CUDA call for topk_last_error_string() and resets the
// runtime's per-thread error state, so a rejected launch does not surface
// later in an unrelated caller's cudaGetLastError().
topk_status_t cuda_fail(cudaError_t e, const char* where) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
    (void)cudaGetLastError();
    return TOPK_ECUDA;
}

// Dispatch defaults, from a sweep of batch x seq_len x k on GB300 (every path
// timed, plan + transform replayed from a graph, L2 flushed; the table is in
// the design notes).  Long rows (one cluster per row): above 16K for batches
// of up to 16 rows, above 64K up to 64 rows, above 128K for larger batches
// -- the batch-dependent floor of SGLang PR #26788 (commits "Fuse the
// cluster/non-cluster split for small batch" and its later floor change)
// with the seq-dependent cap of the same PR expressed as a third tier: at
// batch 128 x 128K one block per row is 1.3-1.8x faster than clusters, at
// 256K clusters win at every batch.  From 1024 rows on, short rows (<= 16K,
// k <= 512) go to the warp-per-row kernel (1.2-1.6x), and from 384 rows on,
// mid rows (16K..64K, k <= 624) to the warp-specialised kernel (1.05-1.2x).
topk_tuning_t g_tuning = {16384, 65536, 16, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 131072, 64, 1024, 384, 0, 0, 0};

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

int log2_exact(int64_t x) {
    int r = 0;
    while ((int64_t{1} << r) < x) ++r;
    return r;
}

topk_status_t check_device() {
    int dev = 0;
    const cudaError_t ge = cudaGetDevice(&dev);
    if (ge != cudaSuccess) return cuda_fail(ge, "cudaGetDevice");
    static std::map<int, topk_status_t> known;
    std::lock_guard<std::mutex> lock(g_mutex);
    auto it = known.find(dev);
    if (it != known.end()) return it->second;
    int major = 0, minor = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    const topk_status_t st = (major == 10 && minor == 3) ? TOPK_OK : TOPK_EDEVICE;
    known[dev] = st;
    return st;
}

int32_t long_threshold(const topk_tuning_t& t, int32_t batch) {
    if (batch <= t.small_batch_max) return t.long_threshold_small_batch;
    return batch <= t.large_batch_min ? t.long_threshold : t.long_threshold_large_batch;
}

struct PathConfig {
    int cluster;
    int threads;
    int tile;
    int stages;
    int cap;
    int samples;
    float gate_fill;
    size_t smem;
};

int sm_count() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

// Launch shape of the select kernel.  Larger bulk copies cost less per byte
// (the per-copy work of a warp is amortised over more elements), within the
// shared memory that keeps two or three blocks per SM.  Single blocks: a
// candidate buffer of 4k entries (>= 2048; >= 3072 for rows over 16K).
// Clusters: a k-entry buffer (>= 2048).
topk_status_t resident_units(int cluster, int threads, size_t smem, int* units);

// Gated elements per block of a C-block cluster at the gate's sampling floor:
// r = E + 4 sqrt(E) + 4 of M samples (E = M k / L) stands for r L / M
// elements of a row of L.
double floor_per_block(int cluster, int32_t k, int32_t max_seq_len, int samples) {
    const double L = static_cast<double>(max_seq_len);
    const double M = std::min(static_cast<double>(samples), L);
    const double E = M * static_cast<double>(std::min(k, max_seq_len)) / L;
    return (E + 4.0 * std::sqrt(E) + 4.0) * L / M / cluster;
}

// grow_buffer = false: the cluster buffer before it is sized to the gate's
// sampling floor (the dispatch's cluster-size floor reasons on that one).
PathConfig path_config(int cluster, int32_t k, int32_t batch, int32_t max_seq_len, const topk_tuning_t& t,
                       bool grow_buffer = true) {
    PathConfig c;
    c.cluster = cluster;
    const bool few_rows = cluster > 1 && static_cast<int64_t>(batch) * cluster * 2 <= sm_count();
    // floats per bulk copy and ring depth: single blocks 2 x 32 KB on rows over
    // 16K (2 x 16 KB below, three blocks per SM); clusters of few rows 5 x 32 KB
    // (one 512-thread block per SM), else 2 x 24 KB (two 256-thread blocks per
    // SM).  The select kernel is compiled for 2, 4, 6 or 8 float4s per thread
    // per copy: 256 threads take 8, 16, 24 or 32 KB copies, 512 threads 16 or 32 KB.
    if (cluster == 1) {
        c.tile = max_seq_len > 16384 ? 8192 : 4096;
        c.stages = 2;
    } else {
        c.tile = few_rows ? 8192 : 6144;
        c.stages = few_rows ? 5 : 2;
    }
    // Threads per block: single blocks 256 (three blocks per SM on short
    // rows), or 512 on long rows when asked; clusters 512 when few rows pull
    // 32 KB copies, else 256 (more float4s per thread per copy).
    if (cluster == 1)
        c.threads = (t.single_block_threads == 512 && c.tile == 8192) ? 512 : 256;
    else
        c.threads = few_rows ? 512 : 256;
    if (cluster == 1) {
        // Explicit single-block copy size (taken only where the kernel is
        // compiled for it: 2, 4, 6 or 8 float4s per thread at 256 threads,
        // 2 or 4 at 512) and ring depth.
        const int tile = t.single_block_copy_bytes / 4;
        const int v = tile / (4 * c.threads);
        if (tile > 0 && v * 4 * c.threads == tile && (v == 2 || v == 4 || (c.threads == 256 && (v == 6 || v == 8))))
            c.tile = tile;
        if (t.single_block_stages > 0) c.stages = t.single_block_stages;
    }
    int cap = t.candidate_capacity;
    if (cap == 0) {
        cap = cluster == 1 ? 4 * k : k;
        if (cap < 2048) cap = 2048;
        // Long single-block rows: the gate count of a row spreads by about
        // 1/sqrt(rank) around its aim, and a row past the buffer re-reads its
        // scores; 3072 entries hold the high draws while two blocks still fit
        // on an SM at k = 512.
        if (cluster == 1 && max_seq_len > 16384 && cap < 3072) cap = 3072;
        if (cap > 16384) cap = 16384;
        cap = (cap + 63) / 64 * 64;
    }
    c.cap = cap;
    c.gate_fill = t.gate_fill_percent > 0 ? 0.01f * static_cast<float>(t.gate_fill_percent) : 0.4f;
    int samples = t.samples;
    if (samples == 0 || samples > kMaxSamples) samples = kMaxSamples;
    c.samples = samples;
    c.smem = make_layout(cluster, c.tile, c.stages, c.cap, k).total;
    if (cluster > 1 && t.candidate_capacity == 0 && grow_buffer) {
        // The gate's count spreads with its sampled rank r (about 1/sqrt(r)
        // of the count, the same way in every block of the row), and a block
        // whose buffer overflows sends its cluster's row through re-reads of
        // the slices, tens of microseconds.  Where the sampling floor alone
        // fills a block's buffer past 40 %, the buffer grows toward that
        // share, within the shared memory left at the same blocks per SM
        // (3-block clusters on 256K rows at k = 1024 gate about 1024
        // elements per block: with 2048 entries one row in a few hundred
        // overflowed, and a batch of 190 such rows took 126 us instead of 65).
        const double per_block = floor_per_block(cluster, k, max_seq_len, samples);
        if (per_block > 0.4 * c.cap) {
            int dev = 0, optin = 0, per_sm = 0, reserved = 0, base = 0;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
            cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
            cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
            const int blocks = std::max(1, per_sm / (static_cast<int>(c.smem) + reserved));
            const int budget = std::min(optin, per_sm / blocks - reserved);
            int want = std::min(16384, static_cast<int>(std::ceil(per_block / 0.4 / 64.0)) * 64);
            while (want > c.cap && make_layout(cluster, c.tile, c.stages, want, k).total > static_cast<uint32_t>(budget))
                want -= 64;
            if (want > c.cap && resident_units(cluster, c.threads, c.smem, &base) == TOPK_OK) {
                const size_t grown = make_layout(cluster, c.tile, c.stages, want, k).total;
                int units = 0;
                if (resident_units(cluster, c.threads, grown, &units) == TOPK_OK && units >= base) {
                    c.cap = want;
                    c.smem = grown;
                }
            }
        }
    }
    if (cluster == 16 && t.candidate_capacity == 0) {
        // The largest cluster on rows so long that the gate's sampling floor
        // would fill a block's buffer past 80 % even so: a larger buffer,
        // paid for with ring stages (1 x 16M, k = 2048: 57K gated, 3.6K per
        // block).
        const double per_block = floor_per_block(cluster, k, max_seq_len, samples);
        if (per_block > 0.8 * c.cap) {
            int dev = 0, optin = 0;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
            int want = static_cast<int>(std::ceil(per_block / 0.6 / 64.0)) * 64;
            want = std::min(want, 16384);
            int stages = c.stages;
            while (stages > 2 && make_layout(cluster, c.tile, stages, want, k).total > static_cast<uint32_t>(optin))
                --stages;
            while (want > c.cap && make_layout(cluster, c.tile, stages, want, k).total > static_cast<uint32_t>(optin))
                want -= 64;
            if (want > c.cap) {
                c.cap = want;
                c.stages = stages;
                c.smem = make_layout(cluster, c.tile, c.stages, c.cap, k).total;
            }
        }
    }
    return c;
}

// Resident units (blocks, or clusters) of the select kernel for a launch shape.
topk_status_t resident_units(int cluster, int threads, size_t smem, int* units) {
    static std::map<std::pair<int, size_t>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_pair((threads * 64 + cluster) * 64 + dev, smem);
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *units = it->second;
            return TOPK_OK;
        }
    }
    int u = 0;
    const cudaError_t e = select_occupancy(cluster, threads, smem, &u);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    if (u <= 0) {
        snprintf(g_last_error, sizeof(g_last_error), "select kernel (cluster %d, %zu B smem) cannot be resident",
                 cluster, smem);
        return TOPK_ECUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    cache[key] = u;
    *units = u;
    return TOPK_OK;
}

// Resident blocks of the segment-split streaming kernel on the current device.
topk_status_t resident_split_units(int* units) {
    static std::map<int, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        auto it = cache.find(dev);
        if (it != cache.end()) {
            *units = it->second;
            return TOPK_OK;
        }
    }
    int u = 0;
    const cudaError_t e = split_occupancy(&u);
    if (e != cudaSuccess) return cuda_fail(e, "split select occupancy query");
    if (u <= 0) {
        snprintf(g_last_error, sizeof(g_last_error), "split select kernel cannot be resident");
        return TOPK_ECUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    cache[dev] = u;
    *units = u;
    return TOPK_OK;
}

// Elements per segment of the split path: about four segments per resident
// block over the batch's upper bound of elements (batch x max_seq_len),
// 4096..32768, doubled while the segment list would not fit; 0 when no size
// up to 1M elements fits.
int32_t split_segment(int32_t batch, int32_t max_seq_len, const topk_tuning_t& t, int units) {
    int64_t seg = t.split_segment;
    if (seg == 0) {
        const int64_t est = static_cast<int64_t>(batch) * max_seq_len / (4 * static_cast<int64_t>(units));
        seg = 4096;
        while (seg < est && seg < 32768) seg <<= 1;
    }
    while (static_cast<int64_t>(batch) * ((static_cast<int64_t>(max_seq_len) + seg - 1) / seg) > kSplitMaxUnits &&
           seg <= (1 << 20))
        seg <<= 1;
    return seg <= (1 << 20) ? static_cast<int32_t>(seg) : 0;
}

// Whether a row of max_seq_len keeps the split path's per-row candidate
// buffer (kSplitCap) at most 80 % full at its gate's sampling floor (about
// (E + 4 sqrt(E) + 4) L / M gated elements, E = M k / L): rows up to about 2M
// tokens at k = 2048.  Longer rows would overflow it into the one-block
// full-row resolve (8 x 4M: 2.2 ms against 65 us on the cluster path).
bool split_fits(int32_t max_seq_len, int32_t k, const topk_tuning_t& t) {
    const double L = static_cast<double>(max_seq_len);
    if (L <= 0.0) return true;
    const double M = std::min(L, static_cast<double>(t.samples > 0 ? t.samples : kSplitMaxSamples));
    const double E = M * static_cast<double>(k) / L;
    return (E + 4.0 * std::sqrt(E) + 4.0) * L / M <= 0.8 * kSplitCap;
}

// Resident blocks of the warp-per-row kernel on the current device.
topk_status_t resident_warp_units(int* units) {
    static std::map<int, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        auto it = cache.find(dev);
        if (it != cache.end()) {
            *units = it->second;
            return TOPK_OK;
        }
    }
    int u = 0;
    const cudaError_t e = warp_select_occupancy(&u);
    if (e != cudaSuccess) return cuda_fail(e, "warp select occupancy query");
    if (u <= 0) {
        snprintf(g_last_error, sizeof(g_last_error), "warp select kernel cannot be resident");
        return TOPK_ECUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    cache[dev] = u;
    *units = u;
    return TOPK_OK;
}

// Launch shapes of the warp-specialised single-block kernel.  Two candidate
// buffers of max(2496, 4k) entries (shape 2) or max(3072, 4k) (shape 3), of
// 6 bytes each (rows of up to 65536).
//  - shape 2: 4 resolving warps, 32 KB copies in a two-stage ring: about
//    112.5 KB of shared memory at k <= 624, two blocks per SM;
//  - shape 3: 8 resolving warps, 32 KB copies in a ring as deep as the
//    shared memory allows (up to four stages), one block per SM.
struct StreamConfig {
    int resolve_warps, tile, stages, cap, samples;
    float gate_fill;
    size_t smem;
};

StreamConfig stream_config(int shape, int32_t k, const topk_tuning_t& t) {
    StreamConfig c;
    c.resolve_warps = shape == 3 ? 8 : 4;
    c.tile = 8192;
    int cap = t.candidate_capacity;
    if (cap == 0) {
        cap = std::max(shape == 3 ? 3072 : 2496, 4 * k);
        if (cap > 16384) cap = 16384;
        cap = (cap + 63) / 64 * 64;
    }
    c.cap = cap;
    int samples = t.samples;
    if (samples == 0 || samples > kMaxSamples) samples = kMaxSamples;
    c.samples = samples;
    c.gate_fill = t.gate_fill_percent > 0 ? 0.01f * static_cast<float>(t.gate_fill_percent) : 0.4f;
    c.stages = 2;
    // Explicit copy size and ring depth (a copy is 2, 4, 6 or 8 float4s per
    // streaming thread).
    const int tile = t.single_block_copy_bytes / 4;
    const int v = tile / (4 * 32 * kStreamWarps);
    if (tile > 0 && v * 4 * 32 * kStreamWarps == tile && (v == 2 || v == 4 || v == 6 || v == 7 || v == 8))
        c.tile = tile;
    if (t.single_block_stages > 0) c.stages = t.single_block_stages;
    if (shape == 3 && t.single_block_stages == 0) {
        int dev = 0, optin = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        while (c.stages < 4 && make_stream_layout(c.tile, c.stages + 1, c.cap, k).total <= static_cast<uint32_t>(optin))
            ++c.stages;
    }
    c.smem = make_stream_layout(c.tile, c.stages, c.cap, k).total;
    return c;
}

topk_status_t resident_stream_units(int resolve_warps, size_t smem, int* units) {
    static std::map<std::pair<int, size_t>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_pair(dev * 16 + resolve_warps, smem);
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *units = it->second;
            return TOPK_OK;
        }
    }
    int u = 0;
    const cudaError_t e = stream_select_occupancy(resolve_warps, smem, &u);
    if (e != cudaSuccess) return cuda_fail(e, "stream select occupancy query");
    if (u <= 0) {
        snprintf(g_last_error, sizeof(g_last_error), "stream select kernel (%zu B smem) cannot be resident", smem);
        return TOPK_ECUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    cache[key] = u;
    *units = u;
    return TOPK_OK;
}

// The kernels one topk_transform call launches.  Long rows go to the cluster
// kernel.  Blocks per row (cluster_size 0): 16 while the rows take at most
// one SM per block that way, 8 while every row gets a resident cluster at
// once, else 3 or 4 (raised when the sampled gate's floor would crowd the
// clusters' candidate buffers).  When the whole batch fits in two
// waves of those clusters (four of automatic 3-block ones), the short rows
// are handed to the cluster kernel as well (after the long ones), so that no
// second launch runs after it.
struct Dispatch {
    bool launch_long = false;
    bool fold_short = false;
    PathConfig cl = {};
    int cl_units = 0;
    bool split = false;   // the segment-split path takes the whole batch
    int32_t split_seg = 0;
    int split_units = 0;
};

topk_status_t decide_dispatch(int32_t batch, int32_t max_seq_len, int32_t k, const topk_tuning_t& t, Dispatch* d) {
    *d = Dispatch();
    d->launch_long = max_seq_len > long_threshold(t, batch);
    // The segment-split path, when asked for and the batch fits one split
    // launch.  The automatic dispatch does not take it: on GB300 the cluster
    // kernel was faster on every long-row shape timed (1 / 8 / 32 x 1M,
    // k = 2048; 128 ragged rows up to 256K, k = 1024), because each segment
    // ends in a block barrier and a fenced count, and the gate is a kernel of
    // its own.
    if (batch <= kSplitMaxRows && t.split_rows == 1 && split_fits(max_seq_len, k, t)) {
        const topk_status_t r = resident_split_units(&d->split_units);
        if (r != TOPK_OK) return r;
        d->split_seg = split_segment(batch, max_seq_len, t, d->split_units);
        if (d->split_seg > 0) {
            d->split = true;
            return TOPK_OK;
        }
    }
    if (!d->launch_long) return TOPK_OK;
    int cluster = t.cluster_size;
    if (cluster == 0) {
        // 16 blocks per row for up to 4 rows; then 4 for rows of at most 64K
        // (8 blocks would give each block 8K elements or fewer: 16 x 64K takes
        // 25.3 us with 8-block clusters and 21.5 us with 4-block ones, and 4 is
        // no slower at 4 or 8 rows); else 8 while every row gets a resident
        // 8-block cluster at once, else 4 (the sweep: 8 beats 16 from 8 rows
        // on, 4 beats 8 once the rows exceed one wave of 8-block clusters).
        if (batch <= 4 && static_cast<int64_t>(batch) * 16 <= sm_count()) {
            cluster = 16;
        } else if (max_seq_len <= 65536) {
            cluster = 4;
        } else {
            const PathConfig c8 = path_config(8, k, batch, max_seq_len, t);
            int u8 = 0;
            const topk_status_t r = resident_units(8, c8.threads, c8.smem, &u8);
            if (r != TOPK_OK) return r;
            if (batch <= u8) {
                cluster = 8;
            } else {
                // 3 blocks per row where 4-block clusters would give some
                // cluster two rows, up to four waves of 3-block clusters in
                // one launch: the ragged mix of 128 rows up to 256K took
                // 46.2 vs 48.2 us, 150 bf16 rows of U[1K, 256K] 52.3 vs 85.1,
                // 300 of them 79.0 vs 94.4, 256 rows of 256K 90.2 vs 101.5;
                // rows of one length that fill one wave of 4-block clusters
                // and a part of the next lose (128 x 256K: 60.5 vs 54.4).
                // Only where a 3-block buffer holds the gate's sampling floor
                // at 40 %.
                const PathConfig c4 = path_config(4, k, batch, max_seq_len, t);
                const PathConfig c3 = path_config(3, k, batch, max_seq_len, t);
                int u4 = 0, u3 = 0;
                topk_status_t r2 = resident_units(4, c4.threads, c4.smem, &u4);
                if (r2 == TOPK_OK) r2 = resident_units(3, c3.threads, c3.smem, &u3);
                if (r2 != TOPK_OK) return r2;
                const bool fits = floor_per_block(3, k, max_seq_len, c3.samples) <= 0.4 * c3.cap;
                cluster = (fits && batch > u4 && batch <= 4 * u3) ? 3 : 4;
            }
        }
    }
    if (t.cluster_size == 0) {
        // At least enough blocks that a row of max_seq_len fills each block's
        // candidate buffer to at most 80 % at the gate's sampling floor: about
        // r_safe = E + 4 sqrt(E) + 4 of M samples are gated, E = M k / L, so a
        // row gates about r_safe * L / M elements.  Without it, 2 x 1M rows
        // with k = 2048 in a batch of 64 took 4-block clusters whose buffers
        // overflowed (233 us; 40 us with 8 blocks), and a 4M row among 16 rows
        // 8-block ones (438 us; 58 us with 16 blocks).  At 73 % (1M rows,
        // k = 1024, 4 blocks) the buffers hold: 58 us against 67 us with 8.
        const double L = static_cast<double>(max_seq_len);
        const double M = static_cast<double>(t.samples > 0 && t.samples < kMaxSamples ? t.samples : kMaxSamples);
        const double E = M * static_cast<double>(k) / L;
        const double gated = (E + 4.0 * std::sqrt(E) + 4.0) * L / M;
        const double cap = static_cast<double>(path_config(cluster, k, batch, max_seq_len, t, false).cap);
        while (cluster < 16 && gated / cluster > 0.8 * cap) cluster = cluster == 3 ? 4 : 2 * cluster;
    }
    d->cl = path_config(cluster, k, batch, max_seq_len, t);
    const topk_status_t r = resident_units(d->cl.cluster, d->cl.threads, d->cl.smem, &d->cl_units);
    if (r != TOPK_OK) return r;
    // Short rows join the cluster launch while the batch is at most two waves
    // of clusters (four of the automatic 3-block ones): one launch instead of
    // a second one after it.
    d->fold_short = static_cast<int64_t>(batch) <= (d->cl.cluster == 3 && t.cluster_size == 0 ? 4 : 2) *
                                                       static_cast<int64_t>(d->cl_units);
    return TOPK_OK;
}

}  // namespace

extern "C" {

size_t topk_plan_workspace_bytes(int32_t batch) { return plan_bytes(batch); }

const char* topk_last_error_string(void) { return g_last_error; }

const char* topk_status_string(topk_status_t status) {
    switch (status) {
        case TOPK_OK: return "ok";
        case TOPK_EINVAL: return "invalid argument";
        case TOPK_EALIGN: return "misaligned pointer or stride";
        case TOPK_ECUDA: return "CUDA error";
        case TOPK_ENOSPACE: return "workspace too small";
        case TOPK_EDEVICE: return "device is not an sm_103 GPU";
    }
    return "unknown status";
}

topk_status_t topk_get_tuning(topk_tuning_t* tuning_host) {
    if (!tuning_host) return TOPK_EINVAL;
    std::lock_guard<std::mutex> lock(g_mutex);
    *tuning_host = g_tuning;
    return TOPK_OK;
}

topk_status_t topk_set_tuning(const topk_tuning_t* t) {
    if (!t) return TOPK_EINVAL;
    if (t->long_threshold_small_batch < 0 || t->long_threshold < 0 || t->small_batch_max < 0 ||
        t->long_threshold_large_batch < 0 || t->large_batch_min < 0 || t->warp_batch_min < 0 ||
        t->stream_batch_min < 0)
        return TOPK_EINVAL;
    if (t->cluster_size != 0 && t->cluster_size != 2 && t->cluster_size != 3 && t->cluster_size != 4 &&
        t->cluster_size != 8 &&
        t->cluster_size != 16)
        return TOPK_EINVAL;
    if (t->candidate_capacity != 0 &&
        (t->candidate_capacity < 2048 || t->candidate_capacity > 16384 || t->candidate_capacity % 64 != 0))
        return TOPK_EINVAL;
    if (t->samples != 0 && (t->samples < 32 || t->samples > kMaxSamples || t->samples % 32 != 0))
        return TOPK_EINVAL;
    if (t->gate_fill_percent < 0 || t->gate_fill_percent > 100) return TOPK_EINVAL;
    if (t->single_block_threads != 0 && t->single_block_threads != 256 && t->single_block_threads != 512)
        return TOPK_EINVAL;
    if (t->single_block_copy_bytes != 0 && t->single_block_copy_bytes != 8192 &&
        t->single_block_copy_bytes != 16384 && t->single_block_copy_bytes != 24576 &&
        t->single_block_copy_bytes != 32768)
        return TOPK_EINVAL;
    if (t->single_block_stages != 0 && (t->single_block_stages < 2 || t->single_block_stages > 8)) return TOPK_EINVAL;
    if (t->gate_refresh_tiles < 0 || t->gate_refresh_tiles > 64) return TOPK_EINVAL;
    if (t->warp_rows < 0 || t->warp_rows > 2) return TOPK_EINVAL;
    if (t->wait_limit_us < 0 || t->wait_limit_us > 60000000) return TOPK_EINVAL;
    if (t->single_block_kernel < 0 || t->single_block_kernel > 3) return TOPK_EINVAL;
    if (t->split_rows < 0 || t->split_rows > 2) return TOPK_EINVAL;
    if (t->split_segment != 0 && (!is_pow2(t->split_segment) || t->split_segment < 4096 ||
                                  t->split_segment > (1 << 20)))
        return TOPK_EINVAL;
    if (t->split_full_resolve < 0 || t->split_full_resolve > 1) return TOPK_EINVAL;
    std::lock_guard<std::mutex> lock(g_mutex);
    g_tuning = *t;
    return TOPK_OK;
}

topk_status_t topk_plan(const int32_t* seq_lens, int32_t batch, int32_t max_seq_len, void* workspace,
                        size_t workspace_bytes, topk_stream_t stream) {
    if (!seq_lens || !workspace || batch < 1 || max_seq_len < 0) return TOPK_EINVAL;
    if (workspace_bytes < plan_bytes(batch)) return TOPK_ENOSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0 || reinterpret_cast<uintptr_t>(seq_lens) % 4 != 0)
        return TOPK_EALIGN;
    const topk_status_t dev = check_device();
    if (dev != TOPK_OK) return dev;
    topk_tuning_t t;
    topk_get_tuning(&t);
    const cudaError_t e = launch_plan(seq_lens, batch, max_seq_len, long_threshold(t, batch), workspace,
                                      reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "plan launch");
    return TOPK_OK;
}

topk_status_t topk_transform(const float* scores, int64_t row_stride, const int32_t* seq_lens, int32_t batch,
                             int32_t max_seq_len, const int32_t* page_table, int64_t page_table_stride,
                             int32_t page_size, int32_t k, int32_t* out_indices, int32_t* out_raw_indices_or_null,
                             void* workspace, topk_stream_t stream) {
    if (!scores || !seq_lens || !page_table || !out_indices || !workspace) return TOPK_EINVAL;
    if (batch < 1 || max_seq_len < 0 || k < 1 || k > kMaxK) return TOPK_EINVAL;
    if (!is_pow2(page_size) || page_size > (1 << 30)) return TOPK_EINVAL;
    if (row_stride < max_seq_len || row_stride < 1) return TOPK_EINVAL;
    if (page_table_stride < (static_cast<int64_t>(max_seq_len) + page_size - 1) / page_size || page_table_stride < 1)
        return TOPK_EINVAL;
    if (reinterpret_cast<uintptr_t>(scores) % 16 != 0 || row_stride % 4 != 0) return TOPK_EALIGN;
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return TOPK_EALIGN;
    if (reinterpret_cast<uintptr_t>(seq_lens) % 4 || reinterpret_cast<uintptr_t>(page_table) % 4 ||
        reinterpret_cast<uintptr_t>(out_indices) % 4 || reinterpret_cast<uintptr_t>(out_raw_indices_or_null) % 4)
        return TOPK_EALIGN;
    const topk_status_t dev = check_device();
    if (dev != TOPK_OK) return dev;

    topk_tuning_t t;
    topk_get_tuning(&t);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    auto* hdr = static_cast<PlanHeader*>(workspace);

    SelectParams p = {};
    p.scores = scores;
    p.row_stride = row_stride;
    p.seq_lens = seq_lens;
    p.batch = batch;
    p.max_seq_len = max_seq_len;
    p.page_table = page_table;
    p.pt_stride = page_table_stride;
    p.log2_page = log2_exact(page_size);
    p.k = k;
    p.out = out_indices;
    p.raw_out = out_raw_indices_or_null;
    p.plan = hdr;
    p.flags = &hdr->flags;
    p.force_two_pass = t.force_two_pass;
    p.disable_gate = t.disable_gate;
    p.timeout_ns = t.wait_limit_us > 0 ? 1000ull * static_cast<uint64_t>(t.wait_limit_us) : kDefaultWaitLimitNs;

    Dispatch d;
    {
        const topk_status_t r = decide_dispatch(batch, max_seq_len, k, t, &d);
        if (r != TOPK_OK) return r;
    }
    if (d.split) {
        SplitParams q = {};
        q.scores = scores;
        q.row_stride = row_stride;
        q.seq_lens = seq_lens;
        q.batch = batch;
        q.max_seq_len = max_seq_len;
        q.page_table = page_table;
        q.pt_stride = page_table_stride;
        q.log2_page = p.log2_page;
        q.k = k;
        q.out = out_indices;
        q.raw_out = out_raw_indices_or_null;
        q.plan = hdr;
        q.flags = &hdr->flags;
        q.ws = split_region(workspace, batch);
        q.seg = d.split_seg;
        q.samples = t.samples > 0 ? t.samples : kSplitMaxSamples;
        q.full_resolve = t.split_full_resolve;
        q.disable_gate = t.disable_gate;
        const cudaError_t e = launch_split(q, d.split_units, st);
        if (e != cudaSuccess) return cuda_fail(e, "split select launch");
        return TOPK_OK;
    }
    const bool launch_long = d.launch_long;
    const bool fold_short = d.fold_short;
    const PathConfig& cl = d.cl;
    const int cl_units = d.cl_units;
    // Short rows in a wide batch (or when asked for): the warp-per-row kernel
    // takes every row.
    const bool warp_fits = !launch_long && !fold_short && max_seq_len <= static_cast<int32_t>(kWarpMaxLen) &&
                           k <= kWarpMaxK;
    const bool warp_ok = warp_fits && (t.warp_rows == 1 || (t.warp_rows == 0 && batch >= t.warp_batch_min));
    if (warp_ok) {
        int warp_units = 0;
        {
            const topk_status_t r = resident_warp_units(&warp_units);
            if (r != TOPK_OK) return r;
        }
        SelectParams q = p;
        q.items = plan_short_list(workspace, batch);
        q.n_items_dev = &hdr->n_short;
        q.items2 = plan_long_list(workspace);
        q.n_items2_dev = &hdr->n_long;
        q.gate_fill = t.gate_fill_percent > 0 ? 0.01f * static_cast<float>(t.gate_fill_percent) : 0.4f;
        const int warps_per_block = kWarpThreads / 32;
        const int grid = std::min(warp_units, (batch + warps_per_block - 1) / warps_per_block);
        // A programmatic launch places the blocks while the plan finishes; on
        // GB300 that gains about 1 us when the grid leaves slots free, and
        // costs about 8 us (8192 x 8192 rows) when it fills every slot of the
        // GPU: then it is launched plainly, after the plan.
        const cudaError_t e = launch_warp_select(q, grid, grid < warp_units, st);
        if (e != cudaSuccess) return cuda_fail(e, "warp select launch");
        return TOPK_OK;
    }
    // The warp-specialised single-block kernel: forced, or automatic for rows
    // over 16K when two of its blocks fit on an SM (and no option of the
    // single-role kernel is asked for).
    bool use_stream = false;
    StreamConfig sc = {};
    int stream_units = 0;
    if (!fold_short && t.single_block_kernel != 1) {
        const bool classic_knobs = t.gate_refresh_tiles != 0 || t.single_block_threads != 0 ||
                                   t.single_block_copy_bytes != 0 || t.single_block_stages != 0;
        // The longest row the single-block launch takes (the short list only,
        // when a cluster launch takes the long rows); the warp-specialised
        // kernel keeps 16-bit positions, so it takes rows of up to 65536.
        const int32_t longest = launch_long ? std::min(max_seq_len, long_threshold(t, batch)) : max_seq_len;
        int shape = longest <= kStreamMaxLen ? t.single_block_kernel : 1;
        const bool auto_fit = shape == 0 && !classic_knobs && longest > 16384 && batch >= t.stream_batch_min;
        if (auto_fit) shape = 2;
        if (shape >= 2) {
            sc = stream_config(shape, k, t);
            const topk_status_t r = resident_stream_units(sc.resolve_warps, sc.smem, &stream_units);
            if (r != TOPK_OK) return r;
            // automatic only where two blocks fit on an SM (k <= 640)
            use_stream = !auto_fit || stream_units >= 2 * sm_count();
        }
    }
    if (use_stream) {
        SelectParams q = p;
        q.items = plan_short_list(workspace, batch);
        q.n_items_dev = &hdr->n_short;
        if (!launch_long) {
            q.items2 = plan_long_list(workspace);
            q.n_items2_dev = &hdr->n_long;
        }
        q.tile = sc.tile;
        q.stages = sc.stages;
        q.gate_refresh = 0;
        q.cap = sc.cap;
        q.samples = sc.samples;
        q.gate_fill = sc.gate_fill;
        // Every resident block (not the fewest blocks with equal shares): the
        // blocks that end up with one row fewer finish early and leave the
        // others more of the memory bandwidth (384 x 32K: 27.4 vs 29.2 us;
        // 1024 x 64K: 70.0 vs 72.9 us; 2048 x 64K unchanged).
        const int grid = std::min(stream_units, batch);
        const cudaError_t e = launch_stream_select(q, sc.resolve_warps, grid, sc.smem, st);
        if (e != cudaSuccess) return cuda_fail(e, "stream select launch");
    } else if (!fold_short) {
        // The single-block kernel goes first: at small batch it usually has no
        // rows and ends as soon as the plan does, and a cluster kernel, placed
        // on the GPU meanwhile (programmatic launch), starts right after it.
        const PathConfig c = path_config(1, k, batch, max_seq_len, t);
        int units = 0;
        const topk_status_t r = resident_units(1, c.threads, c.smem, &units);
        if (r != TOPK_OK) return r;
        SelectParams q = p;
        q.items = plan_short_list(workspace, batch);
        q.n_items_dev = &hdr->n_short;
        if (!launch_long) {  // rows the plan called long (if any) are taken here too
            q.items2 = plan_long_list(workspace);
            q.n_items2_dev = &hdr->n_long;
        }
        q.tile = c.tile;
        q.stages = c.stages;
        q.gate_refresh = c.threads == 256 ? t.gate_refresh_tiles : 0;
        q.cap = c.cap;
        q.samples = c.samples;
        q.gate_fill = c.gate_fill;
        // Equal shares: the fewest blocks that still give every block the
        // same number of rows when all rows are short.
        const int per_unit = (batch + units - 1) / units;
        const int grid = (batch + per_unit - 1) / per_unit;
        const cudaError_t e = launch_select(q, 1, c.threads, grid, c.smem, st);
        if (e != cudaSuccess) return cuda_fail(e, "select launch");
    }
    if (launch_long) {
        SelectParams q = p;
        q.items = plan_long_list(workspace);
        q.n_items_dev = &hdr->n_long;
        if (fold_short) {
            q.items2 = plan_short_list(workspace, batch);
            q.n_items2_dev = &hdr->n_short;
        }
        q.tile = cl.tile;
        q.stages = cl.stages;
        q.gate_refresh = 0;
        q.cap = cl.cap;
        q.samples = cl.samples;
        q.gate_fill = cl.gate_fill;
        const int grid = batch < cl_units ? batch : cl_units;
        const cudaError_t e = launch_select(q, cl.cluster, cl.threads, grid, cl.smem, st);
        if (e != cudaSuccess) return cuda_fail(e, "long-row select launch");
    }
    return TOPK_OK;
}

int32_t topk_transform_launches(int32_t batch, int32_t max_seq_len, int32_t k) {
    if (batch < 1 || max_seq_len < 0 || k < 1 || k > kMaxK) return TOPK_EINVAL;
    const topk_status_t dev = check_device();
    if (dev != TOPK_OK) return dev;
    topk_tuning_t t;
    topk_get_tuning(&t);
    Dispatch d;
    const topk_status_t r = decide_dispatch(batch, max_seq_len, k, t, &d);
    if (r != TOPK_OK) return r;
    if (d.split) return 2;  // the gate kernel and the streaming kernel
    return (d.fold_short ? 0 : 1) + (d.launch_long ? 1 : 0);
}

topk_status_t topk_page_transform(const int32_t* raw_indices, int32_t batch, int32_t k, const int32_t* page_table,
                                  int64_t page_table_stride, int32_t page_size, int32_t* out_indices,
                                  topk_stream_t stream) {
    if (!raw_indices || !page_table || !out_indices || batch < 1 || k < 1 || page_table_stride < 1)
        return TOPK_EINVAL;
    if (!is_pow2(page_size) || page_size > (1 << 30)) return TOPK_EINVAL;
    if (reinterpret_cast<uintptr_t>(raw_indices) % 4 || reinterpret_cast<uintptr_t>(page_table) % 4 ||
        reinterpret_cast<uintptr_t>(out_indices) % 4)
        return TOPK_EALIGN;
    const topk_status_t dev = check_device();
    if (dev != TOPK_OK) return dev;
    const cudaError_t e = launch_page_transform(raw_indices, batch, k, page_table, page_table_stride,
                                                log2_exact(page_size), out_indices,
                                                reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "page transform launch");
    return TOPK_OK;
}

topk_status_t topk_key_map(const float* x, int64_t n, uint32_t* keys, topk_stream_t stream) {
    if (n < 0 || (n > 0 && (!x || !keys))) return TOPK_EINVAL;
    if (reinterpret_cast<uintptr_t>(x) % 4 || reinterpret_cast<uintptr_t>(keys) % 4) return TOPK_EALIGN;
    const topk_status_t dev = check_device();
    if (dev != TOPK_OK) return dev;
    const cudaError_t e = launch_key_map(x, n, keys, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "key map launch");
    return TOPK_OK;
}

topk_status_t topk_read_flags(void* workspace, uint32_t* flags_host, int32_t clear, topk_stream_t stream) {
    if (!workspace || !flags_host) return TOPK_EINVAL;
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return TOPK_EALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    auto* hdr = static_cast<PlanHeader*>(workspace);
    cudaError_t e = cudaMemcpyAsync(flags_host, &hdr->flags, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e, "flag copy");
    if (clear && (e = cudaMemsetAsync(&hdr->flags, 0, sizeof(uint32_t), st)) != cudaSuccess)
        return cuda_fail(e, "flag reset");
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "stream synchronize");
    return TOPK_OK;
}

}  // extern "C"
