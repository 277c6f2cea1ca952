// select_common.cuh -- device helpers shared by the select kernels: warp
// scans and sorts, shared-memory list reservations, the histogram scan, the
// cluster histogram merge, the page-table map and the gate sample positions.
#pragma once

#include <cstddef>
#include <cstdint>

#include "ptx.cuh"
#include "topk_internal.h"

namespace topkidx {
namespace detail {

constexpr uint32_t kFull = 0xffffffffu;

__device__ __forceinline__ int bit_length(uint32_t x) { return 32 - __clz(x); }

__host__ __device__ __forceinline__ uint64_t min_u64(uint64_t a, uint64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t min_i64(int64_t a, int64_t b) { return a < b ? a : b; }

// Shift that maps the key span [0, span] onto at most kBins bins.
__device__ __forceinline__ int shift_for_span(uint32_t span) {
    const int b = bit_length(span);
    return b > kBinBits ? b - kBinBits : 0;
}

__device__ __forceinline__ uint32_t warp_inclusive_sum(uint32_t v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Exclusive prefix sum and total over the warp of small per-lane counts
// (0..32), from bit-plane ballots: no dependent shuffle chain.  Only the
// planes up to the warp's largest count are taken (one or two when the gate
// is sparse).
struct WarpPrefix {
    uint32_t excl, total;
};
__device__ __forceinline__ WarpPrefix warp_prefix_small(uint32_t cnt, int lane) {
    const uint32_t lt = (1u << lane) - 1u;
    WarpPrefix r{0u, 0u};
    const int planes = 32 - __clz(__reduce_max_sync(kFull, cnt));
#pragma unroll
    for (int b = 0; b < 6; ++b) {
        if (b < planes) {
            const uint32_t bal = __ballot_sync(kFull, (cnt >> b) & 1u);
            r.excl += static_cast<uint32_t>(__popc(bal & lt)) << b;
            r.total += static_cast<uint32_t>(__popc(bal)) << b;
        }
    }
    return r;
}

// Warp-wide bitonic compare-and-swap sort, largest value to lane 0
// (DistRadixTopK README, "Distributed Radix Sort via NoC", last point: once
// the residual is down to a handful of candidates a CAS sort finishes it).
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint64_t o = __shfl_xor_sync(kFull, v, j);
            const bool lower = (lane & j) == 0;
            const bool desc_seg = (lane & k) == 0;
            const bool take_max = (lower == desc_seg);
            v = take_max ? (v > o ? v : o) : (v < o ? v : o);
        }
    }
    return v;
}

// Reserves consecutive slots of a shared-memory list for the lanes whose
// `flag` is set, with a single atomic per warp, and returns this lane's slot
// (meaningful only where `flag`).  Every lane of the warp must call it.
__device__ __forceinline__ uint32_t warp_reserve(uint32_t counter, bool flag, int lane) {
    const uint32_t m = __ballot_sync(kFull, flag);
    if (m == 0u) return 0u;
    const int leader = __ffs(m) - 1;
    uint32_t base = 0;
    if (lane == leader) base = ptx::atom_add_s(counter, static_cast<uint32_t>(__popc(m)));
    base = __shfl_sync(kFull, base, leader);
    return base + static_cast<uint32_t>(__popc(m & ((1u << lane) - 1u)));
}

// Reserves `n` consecutive slots per lane (lane order) with a single atomic
// per warp; returns this lane's first slot.  Every lane must call it.
__device__ __forceinline__ uint32_t warp_reserve_n(uint32_t counter, uint32_t n, int lane) {
    const uint32_t incl = warp_inclusive_sum(n, lane);
    const uint32_t total = __shfl_sync(kFull, incl, 31);
    uint32_t base = 0;
    if (lane == 31 && total != 0u) base = ptx::atom_add_s(counter, total);
    base = __shfl_sync(kFull, base, 31);
    return base + incl - n;
}

__device__ __forceinline__ int32_t page_map(const int32_t* pt_row, int32_t log2_page, int32_t raw) {
    if (raw < 0) return -1;
    const uint32_t page = static_cast<uint32_t>(__ldg(pt_row + (raw >> log2_page)));
    const uint32_t mask = (1u << log2_page) - 1u;
    return static_cast<int32_t>((page << log2_page) + (static_cast<uint32_t>(raw) & mask));
}

// Writes n results of a row: slot dst0 + q gets position src(q) (or -1) in
// raw_row and its page-table mapping in out_row.  Four entries per thread are
// in flight: their page-table loads are all issued before any store.
template <int NT, typename Src>
__device__ __forceinline__ void write_results(int32_t* out_row, int32_t* raw_row, const int32_t* pt_row,
                                              int32_t log2_page, uint32_t n, uint32_t dst0, uint32_t tid, Src src) {
    for (uint32_t q0 = tid; q0 < n; q0 += 4u * NT) {
        int32_t r[4], v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t q = q0 + u * NT;
            r[u] = q < n ? src(q) : -1;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = page_map(pt_row, log2_page, r[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t q = q0 + u * NT;
            if (q < n) {
                out_row[dst0 + q] = v[u];
                if (raw_row) raw_row[dst0 + q] = r[u];
            }
        }
    }
}

// Barrier of the whole block (the default group of the helpers below).
struct BlockSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// Barrier of a named group of threads (bar.sync id, count): `count` threads,
// a multiple of 32, all of which must call it.
template <int kId, int kCount>
struct GroupSync {
    __device__ __forceinline__ void operator()() const {
        asm volatile("bar.sync %0, %1;" ::"n"(kId), "n"(kCount) : "memory");
    }
};

struct ScanResult {
    uint32_t bin, above, count, total;
    uint32_t local;  // this block's own count in `bin` (differs from `count` only in a cluster)
};

// 32-bit shared-window addresses of the block's shared-memory regions.
struct Smem {
    uint32_t ring, hist_a, hist_b, hist_m, cand_key, cand_idx, emit, fin_key, fin_idx, warp_tot, ctl;
    uint32_t it_row, it_len, it_tiles, it_tile_start, claim;
    uint32_t* claim_ptr;
    uint64_t* full;
    uint64_t* empty;
    Control* ctl_ptr;
};

// Addresses of Control fields.
#define CTL(s, field) ((s).ctl + static_cast<uint32_t>(offsetof(Control, field)))

// Clears N (default: the histogram with its cluster-merge slots) counters.
template <int NT, int N = kBinsX>
__device__ __forceinline__ void clear_hist(uint32_t h, int tid) {
    static_assert(N % 4 == 0, "whole uint4s");
    for (int i = tid * 4; i < N; i += NT * 4) ptx::sts_u4(h + 4u * i, make_uint4(0, 0, 0, 0));
}

// Finds, in a histogram whose bins are ordered by key, the bin where the
// count of elements taken from the top reaches `need`: returns that bin, the
// count in the bins above it, its own count and the histogram total.  If the
// total is below `need`, bin is 0xffffffff.  Every thread of the block must
// call it; it contains two barriers of the group (`sync`: the whole block by
// default) and reads `h` before the first.
// `h_local` (0: same as `h`) is the block's own histogram, whose count of
// the found bin is returned as `local`.
template <int NT, typename Sync = BlockSync>
__device__ __forceinline__ ScanResult scan_find(const Smem& s, uint32_t h, uint32_t need, int tid,
                                                uint32_t h_local = 0, Sync sync = Sync()) {
    constexpr int BPT = kBins / NT;
    static_assert(BPT % 4 == 0 && BPT >= 4, "bins per thread");
    const int lane = tid & 31, warp = tid >> 5;
    const int base = kBins - (tid + 1) * BPT;  // thread 0 owns the top bins
    uint32_t v[BPT];
#pragma unroll
    for (int i = 0; i < BPT; i += 4) {
        const uint4 q = ptx::lds_u4(h + 4u * (base + i));
        v[i] = q.x;
        v[i + 1] = q.y;
        v[i + 2] = q.z;
        v[i + 3] = q.w;
    }
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) sum += v[i];
    const uint32_t incl = warp_inclusive_sum(sum, lane);
    if (lane == 31) ptx::sts_u32(s.warp_tot + 4u * warp, incl);
    if (tid == 0) ptx::sts_u32(CTL(s, res_bin), 0xffffffffu);
    sync();
    uint32_t pre = 0, total = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; w += 4) {
        const uint4 t = ptx::lds_u4(s.warp_tot + 4u * w);
        const uint32_t ts[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            pre += (w + u < warp) ? ts[u] : 0u;
            total += ts[u];
        }
    }
    const uint32_t excl = pre + incl - sum;
    if (need > excl && need <= excl + sum) {
        uint32_t acc = excl;
#pragma unroll
        for (int i = BPT - 1; i >= 0; --i) {
            if (acc + v[i] >= need) {
                ptx::sts_u32(CTL(s, res_bin), static_cast<uint32_t>(base + i));
                ptx::sts_u32(CTL(s, res_above), acc);
                ptx::sts_u32(CTL(s, res_count), v[i]);
                ptx::sts_u32(CTL(s, res_local), h_local ? ptx::lds_u32(h_local + 4u * (base + i)) : v[i]);
                break;
            }
            acc += v[i];
        }
    }
    sync();
    ScanResult r;
    r.bin = ptx::lds_u32(CTL(s, res_bin));
    r.above = ptx::lds_u32(CTL(s, res_above));
    r.count = ptx::lds_u32(CTL(s, res_count));
    r.local = ptx::lds_u32(CTL(s, res_local));
    r.total = total;
    return r;
}

// Sums the histograms of all blocks of the cluster (DistRadixTopK README,
// "Distributed Radix Sort via NoC", first point: per-block histograms are
// accumulated over the on-chip network, then prefix-summed).  Rank r reduces
// slots [r*chunk, (r+1)*chunk) over every rank's `h_local` and broadcasts the
// sums into every rank's merged histogram: a reduce-scatter followed by an
// all-gather, both through distributed shared memory.  The caller must have
// finished writing `h_local` (all threads reach the first cluster barrier).
template <int NT, int C>
__device__ __forceinline__ void cluster_merge(const Smem& s, uint32_t h_local, uint32_t rank, int tid) {
    ptx::cluster_sync();
    constexpr int chunk = kBinsX / C;
    static_assert(chunk % 4 == 0, "merge chunk must be whole uint4s");
    const uint32_t lbase = h_local + rank * chunk * 4u;
    const uint32_t mbase = s.hist_m + rank * chunk * 4u;
    for (int i = tid * 4; i < chunk; i += NT * 4) {
        uint4 acc = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int q = 0; q < C; ++q) {
            const uint4 v = ptx::ld_cluster_v4(ptx::map_rank(lbase + i * 4u, q));
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
#pragma unroll
        for (int q = 0; q < C; ++q) ptx::st_cluster_v4(ptx::map_rank(mbase + i * 4u, q), acc);
    }
    ptx::cluster_sync();
}

// Position of gate sample i of a row of length L with M samples: every
// position when the row is short, otherwise 32-wide contiguous segments (one
// coalesced 128-byte read per warp) whose starts follow a golden-ratio
// sequence, so that the segments do not alias with periodic score patterns.
__device__ __forceinline__ uint32_t sample_pos(uint32_t i, uint32_t L, uint32_t M) {
    if (L <= M) return i;
    const uint32_t seg = i >> 5;
    const uint64_t frac = static_cast<uint64_t>(seg * 0x9E3779B9u);
    const uint32_t start = static_cast<uint32_t>((frac * static_cast<uint64_t>(L - 31u)) >> 32) & ~3u;
    return start + (i & 31u);
}

// Work items of a persistent grid of `nunits` units (blocks, or clusters):
// in round r, unit u takes item u + r * nunits when r is even and
// (r + 1) * nunits - 1 - u when r is odd -- a boustrophedon over the plan's
// longest-first list, so that a unit which took one of the longest rows in
// one round takes one of the shortest in the next.
__host__ __device__ __forceinline__ int32_t snake_item(int32_t unit, int32_t round, int32_t nunits) {
    return (round & 1) ? (round + 1) * nunits - 1 - unit : unit + round * nunits;
}

// Items unit u takes out of n_items under snake_item.
__host__ __device__ __forceinline__ int32_t snake_count(int32_t unit, int32_t n_items, int32_t nunits) {
    const int32_t full = n_items / nunits, rem = n_items - full * nunits;
    if (rem == 0) return full;
    const bool covered = (full & 1) ? (unit >= nunits - rem) : (unit < rem);
    return full + (covered ? 1 : 0);
}

}  // namespace detail
}  // namespace topkidx
