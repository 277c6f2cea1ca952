// topk_split.cu -- the segment-split select path, for batches of up to
// kSplitMaxRows rows: every row is cut into fixed-size segments, the segments
// of all rows are handed out one at a time to a persistent grid of blocks (so
// that every SM streams, whatever the mix of row lengths), and the block that
// finishes a row's last segment resolves that row.
//
// Method (SGLang PR #26788 "[JIT Kernel] DeepSeek-V4 DSA indexer: faster
// top-k + page-table transform (runtime k <= 2048)" and the DistRadixTopK
// README "Ultra Low Latency Distributed Radix TopK Indexer Via NoC"):
// order-preserving uint32 keys, a sampled lower bound on the k-th key that
// keeps all but a few thousand elements of a row out of the selection, radix
// rounds over the survivors, the last few finished by a warp sort, ties to
// the smaller position, and the gather through the page table.  The pages
// spread one long row over the blocks of a thread-block cluster, which merge
// their histograms through distributed shared memory; here a row's gated
// elements go to a per-row buffer in the workspace (through L2) instead, so
// that a row can take any number of blocks, and a batch of rows of mixed
// lengths keeps every SM streaming until its last segment.
//
// Kernel 1, the gate (one block per row): up to `samples` scores at the gate
// sample positions give lo, a lower bound on the row's k-th key (the
// sample's r-th largest key, r = E + 4 sqrt(E) + 4 with E the expected
// number of samples among the row's top k, cut to its top 22 bits).  Rows
// with seq_len <= k are written here.  Block 0 also lays out the segment
// list (an exclusive prefix of the rows' segment counts) and resets the
// hand-out counter; every block resets its row's counters.
//
// Kernel 2 (persistent; a block claims segments from a global counter):
//  1. Stream.  A block streams its segment with 16-byte loads, two steps in
//     flight; the segment one round ahead (this one's index plus the grid
//     size) is brought into L2 by a bulk prefetch.  A thread whose 16 values
//     all lie below the gate float skips them after one compare; otherwise
//     ties with lo are counted and keys above lo are staged, as 64-bit
//     composites (key << 32 | ~position), in the warp's part of shared
//     memory.  At the end of the segment each warp copies its staged
//     composites to the row's candidate buffer with one reservation; the
//     block fences its stores and counts the segment done for its row.
//  2. Resolve (the block whose segment completed the row):
//     a. k <= n_gt <= capacity: the candidates are loaded into shared memory
//        and the k largest composites found by 11-bit radix rounds over the
//        composite range, the last <= 32 finished by a warp sort.  Distinct
//        composites order the elements by key and then by smaller position,
//        so ties need no step of their own.
//     b. n_gt < k <= n_gt + n_eq: every candidate is taken; the rest are the
//        smallest positions whose key equals lo, collected in position order
//        from the segments whose tie count is non-zero (re-read from memory:
//        the first segment or two of a flat row).
//     c. otherwise (the gate was above the k-th key, or the buffer
//        overflowed): radix rounds over the composites of the whole row, read
//        from memory, until the threshold range fits in shared memory; then
//        the rounds of case a on it.
//  3. Emit + transform: the k positions go through the page table into out
//     (and raw_out).

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "keys.cuh"
#include "ptx.cuh"
#include "select_common.cuh"
#include "topk_internal.h"
#include "topkidx.h"

namespace topkidx {
namespace {

using namespace detail;

constexpr int kGT = kSplitGateThreads;
constexpr int kST = kSplitThreads;
constexpr uint32_t kStepVec = 4;  // float4s per thread per streaming step

// Dynamic shared memory of the streaming kernel.
constexpr uint32_t kSmCand = 0;                                  // u64 [kSplitCap]
constexpr uint32_t kSmHist = kSmCand + kSplitCap * 8u;          // u32 [kBins]
constexpr uint32_t kSmEmit = kSmHist + kBins * 4u;              // u32 [kMaxK]
constexpr uint32_t kSmFin = kSmEmit + kMaxK * 4u;               // u64 [kFinish]
constexpr uint32_t kSmUstart = kSmFin + kFinish * 8u;           // i32 [kSplitMaxRows + 1]
constexpr uint32_t kSmRowLen = kSmUstart + ((kSplitMaxRows + 1) * 4u + 15u) / 16u * 16u;  // u32 [kSplitMaxRows]
constexpr uint32_t kSmRowLo = kSmRowLen + kSplitMaxRows * 4u;   // u32 [kSplitMaxRows]
constexpr uint32_t kSmRowUnits = kSmRowLo + kSplitMaxRows * 4u; // u32 [kSplitMaxRows]
constexpr uint32_t kSmBytes = kSmRowUnits + kSplitMaxRows * 4u;

__device__ __forceinline__ int32_t clamped_len(const SplitParams& p, int32_t row, bool flag) {
    int32_t L = p.seq_lens[row];
    if (L < 0) {
        if (flag) atomicOr(p.flags, TOPK_FLAG_SEQ_NEGATIVE);
        L = 0;
    } else if (L > p.max_seq_len) {
        if (flag) atomicOr(p.flags, TOPK_FLAG_SEQ_CLAMPED);
        L = p.max_seq_len;
    }
    return L;
}

__device__ __forceinline__ uint32_t segments_of(int32_t L, const SplitParams& p) {
    return L > p.k ? (static_cast<uint32_t>(L) + static_cast<uint32_t>(p.seg) - 1u) / static_cast<uint32_t>(p.seg)
                   : 0u;
}

__device__ __forceinline__ bool plan_mismatch(const SplitParams& p) {
    return p.plan &&
           (p.plan->magic != kPlanMagic || p.plan->batch != p.batch || p.plan->max_seq_len != p.max_seq_len);
}

__device__ __forceinline__ uint64_t composite(uint32_t key, uint32_t pos) {
    return (static_cast<uint64_t>(key) << 32) | static_cast<uint64_t>(~pos);
}

// Shift that maps the span [0, span] of 64-bit values onto at most kBins bins.
__device__ __forceinline__ int shift_for_span64(uint64_t span) {
    const int b = 64 - __clzll(static_cast<long long>(span));
    return b > kBinBits ? b - kBinBits : 0;
}

// ------------------------------------------------------------------ gate
__global__ void __launch_bounds__(kGT, 1) split_gate_kernel(const SplitParams p) {
    __shared__ __align__(16) uint32_t hist[kBins];
    __shared__ __align__(16) uint32_t skey[kSplitMaxSamples];
    __shared__ __align__(16) uint32_t warp_tot[32];
    __shared__ __align__(16) Control ctl;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    Smem s = {};
    s.warp_tot = ptx::smem_addr(warp_tot);
    s.ctl = ptx::smem_addr(&ctl);
    const uint32_t h = ptx::smem_addr(hist);
    clear_hist<kGT, kBins>(h, tid);
    // The streaming kernel may be placed now: it waits for this grid to
    // complete before it reads anything.
    ptx::launch_dependents();
    ptx::grid_dependency_wait();
    if (plan_mismatch(p)) {
        if (blockIdx.x == 0 && tid == 0) atomicOr(p.flags, TOPK_FLAG_PLAN_MISMATCH);
        return;
    }
    if (blockIdx.x == 0) {
        // The segment list: first segment of each row (batch <= kGT threads).
        const uint32_t n = tid < p.batch ? segments_of(clamped_len(p, tid, false), p) : 0u;
        const uint32_t incl = warp_inclusive_sum(n, lane);
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        uint32_t pre = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kGT / 32; ++w) {
            const uint32_t t = warp_tot[w];
            pre += w < warp ? t : 0u;
            total += t;
        }
        if (tid < p.batch) p.ws.unit_start[tid] = static_cast<int32_t>(pre + incl - n);
        if (tid == 0) {
            // The host sizes the segments so that the list fits; a list that
            // does not is cut (its rows stay unwritten) and flagged.
            if (total > static_cast<uint32_t>(kSplitMaxUnits)) atomicOr(p.flags, TOPK_FLAG_INTERNAL);
            const uint32_t tot = min(total, static_cast<uint32_t>(kSplitMaxUnits));
            p.ws.unit_start[p.batch] = static_cast<int32_t>(tot);
            p.ws.hdr->next_unit = 0u;
            p.ws.hdr->total_units = tot;
        }
        __syncthreads();  // warp_tot is reused below
    }

    const int32_t row = static_cast<int32_t>(blockIdx.x);
    const int32_t L = clamped_len(p, row, tid == 0);
    const uint32_t K = static_cast<uint32_t>(p.k);
    SplitRow* rs = p.ws.rows + row;
    if (L <= p.k) {  // every position is selected: written here, no segments
        int32_t* out_row = p.out + static_cast<int64_t>(row) * p.k;
        int32_t* raw_row = p.raw_out ? p.raw_out + static_cast<int64_t>(row) * p.k : nullptr;
        const int32_t* pt_row = p.page_table + static_cast<int64_t>(row) * p.pt_stride;
        write_results<kGT>(out_row, raw_row, pt_row, p.log2_page, K, 0u, static_cast<uint32_t>(tid),
                           [&](uint32_t q) { return q < static_cast<uint32_t>(L) ? static_cast<int32_t>(q) : -1; });
        if (tid == 0) {
            rs->lo = 0u;
            rs->n_gt = 0u;
            rs->n_eq = 0u;
            rs->done = 0u;
            rs->len = L;
            rs->nunits = 0;
        }
        return;
    }

    const float* rowp = p.scores + static_cast<int64_t>(row) * p.row_stride;
    const uint32_t M = min(static_cast<uint32_t>(p.samples), static_cast<uint32_t>(L));
    const float E = static_cast<float>(M) * static_cast<float>(K) / static_cast<float>(L);
    const float r_f = ceilf(E + 4.0f * sqrtf(E) + 4.0f);
    uint32_t lo = 0u;  // 0: every element is a candidate
    if (!p.disable_gate && r_f < static_cast<float>(M)) {
        const uint32_t r = static_cast<uint32_t>(r_f);
        // Every sample load is issued before any is used: one memory latency.
        constexpr int kPer = kSplitMaxSamples / kGT;
        float x[kPer];
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const uint32_t i = static_cast<uint32_t>(q * kGT + tid);
            x[q] = i < M ? __ldg(rowp + sample_pos(i, static_cast<uint32_t>(L), M)) : 0.0f;
        }
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const uint32_t i = static_cast<uint32_t>(q * kGT + tid);
            if (i < M) {
                const uint32_t key = score_key(x[q]);
                skey[i] = key;
                ptx::red_add_s(h + 4u * (key >> (32 - kBinBits)), 1u);
            }
        }
        __syncthreads();
        const ScanResult g = scan_find<kGT>(s, h, r, tid);
        lo = g.bin << (32 - kBinBits);
        if (g.above + g.count > r + r / 4u + 4u && g.count > 1u) {
            // Refine inside the coarse bin on the next 11 bits.
            clear_hist<kGT, kBins>(h, tid);
            __syncthreads();
            for (uint32_t i = static_cast<uint32_t>(tid); i < M; i += kGT) {
                const uint32_t key = skey[i];
                if ((key >> (32 - kBinBits)) == g.bin)
                    ptx::red_add_s(h + 4u * ((key >> (32 - 2 * kBinBits)) & (kBins - 1)), 1u);
            }
            __syncthreads();
            const ScanResult g2 = scan_find<kGT>(s, h, r - g.above, tid);
            lo |= g2.bin << (32 - 2 * kBinBits);
        }
    }
    if (tid == 0) {
        rs->lo = lo;
        rs->n_gt = 0u;
        rs->n_eq = 0u;
        rs->done = 0u;
        rs->len = L;
        rs->nunits = static_cast<int32_t>(segments_of(L, p));
    }
}

// ------------------------------------------------------- stream + resolve
__global__ void __launch_bounds__(kST, 2) split_select_kernel(const SplitParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ __align__(16) uint32_t warp_tot[32];
    __shared__ __align__(16) Control ctl;
    __shared__ unsigned long long s_vmax;
    __shared__ uint32_t s_cur, s_eq, s_t, s_e;
    __shared__ int32_t s_res;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t base = ptx::smem_addr(smem_raw);
    Smem s = {};
    s.warp_tot = ptx::smem_addr(warp_tot);
    s.ctl = ptx::smem_addr(&ctl);
    const uint32_t sh_hist = base + kSmHist;
    const uint32_t sh_emit = base + kSmEmit;
    uint64_t* cand_s = reinterpret_cast<uint64_t*>(smem_raw + kSmCand);
    uint64_t* fin_s = reinterpret_cast<uint64_t*>(smem_raw + kSmFin);
    int32_t* ustart = reinterpret_cast<int32_t*>(smem_raw + kSmUstart);
    uint32_t* row_len = reinterpret_cast<uint32_t*>(smem_raw + kSmRowLen);
    uint32_t* row_lo = reinterpret_cast<uint32_t*>(smem_raw + kSmRowLo);
    uint32_t* row_nunits = reinterpret_cast<uint32_t*>(smem_raw + kSmRowUnits);
    const uint32_t K = static_cast<uint32_t>(p.k);
    const uint32_t seg = static_cast<uint32_t>(p.seg);
    // While a segment streams, the candidate area holds each warp's staged
    // candidates (kWarpStage entries per warp); a resolve reuses it whole.
    __shared__ uint32_t s_wcnt[kST / 32];
    constexpr uint32_t kWarpStage = kSplitCap / (kST / 32);
    uint64_t* stage = cand_s + static_cast<uint32_t>(warp) * kWarpStage;
    const uint32_t wcnt_addr = ptx::smem_addr(&s_wcnt[warp]);

    clear_hist<kST, kBins>(sh_hist, tid);
    if (lane == 0) s_wcnt[warp] = 0u;
    if (tid == 0) {
        ctl.err = 0u;
        s_eq = 0u;
    }
    // Every global access comes after this point: the gate grid has completed.
    ptx::grid_dependency_wait();
    if (plan_mismatch(p)) return;  // flagged by the gate kernel
    for (int i = tid; i <= p.batch; i += kST) ustart[i] = p.ws.unit_start[i];
    for (int i = tid; i < p.batch; i += kST) {  // the gate kernel's row states, read once
        row_len[i] = static_cast<uint32_t>(p.ws.rows[i].len);
        row_lo[i] = p.ws.rows[i].lo;
        row_nunits[i] = static_cast<uint32_t>(p.ws.rows[i].nunits);
    }

    auto set_err = [&](uint32_t f) { atomicOr(&ctl.err, f); };
    // Appends `pos` to the emit list for the lanes with `flag` (every lane
    // of the warp calls it).
    auto emit_lanes = [&](bool flag, uint32_t pos) {
        const uint32_t slot = warp_reserve(CTL(s, nemit), flag, lane);
        if (flag) {
            if (slot < K)
                ptx::sts_u32(sh_emit + 4u * slot, pos);
            else
                set_err(TOPK_FLAG_INTERNAL);
        }
    };

    // The `need` largest of the n distinct composites in cand_s, all of them
    // in [r_lo, r_hi]: radix rounds until the range holds <= kFinish, then a
    // warp sort.  Every thread calls it; it ends with a barrier.
    auto select_smem = [&](uint32_t n, uint64_t r_lo, uint64_t r_hi, uint32_t need) {
        uint32_t cnt = n;
        for (int round = 0; cnt > static_cast<uint32_t>(kFinish); ++round) {
            if (round >= 8) {  // cannot happen: each round narrows a 64-bit range by 11 bits
                set_err(TOPK_FLAG_INTERNAL);
                break;
            }
            const int sh = shift_for_span64(r_hi - r_lo);
            for (uint32_t i = static_cast<uint32_t>(tid); i < n; i += kST) {
                const uint64_t v = cand_s[i];
                if (v >= r_lo && v <= r_hi)
                    ptx::red_add_s(sh_hist + 4u * static_cast<uint32_t>((v - r_lo) >> sh), 1u);
            }
            __syncthreads();
            const ScanResult sr = scan_find<kST>(s, sh_hist, need, tid);
            clear_hist<kST, kBins>(sh_hist, tid);
            if (sr.bin >= static_cast<uint32_t>(kBins)) {  // cannot happen: the range holds >= need
                set_err(TOPK_FLAG_INTERNAL);
                __syncthreads();
                break;
            }
            need -= sr.above;
            const uint64_t nlo = r_lo + (static_cast<uint64_t>(sr.bin) << sh);
            const uint64_t width = (1ull << sh) - 1ull;
            r_hi = (r_hi - nlo <= width) ? r_hi : nlo + width;
            r_lo = nlo;
            cnt = sr.count;
            __syncthreads();  // the histogram is clear before the next round adds to it
        }
        if (tid == 0) ptx::sts_u32(CTL(s, nfin), 0u);
        __syncthreads();
        for (uint32_t i0 = 0; i0 < n; i0 += kST) {
            const uint32_t i = i0 + static_cast<uint32_t>(tid);
            const uint64_t v = i < n ? cand_s[i] : 0ull;
            emit_lanes(i < n && v > r_hi, ~static_cast<uint32_t>(v));
            const bool inr = i < n && v >= r_lo && v <= r_hi;
            const uint32_t slot = warp_reserve(CTL(s, nfin), inr, lane);
            if (inr && slot < static_cast<uint32_t>(kFinish)) fin_s[slot] = v;
        }
        __syncthreads();
        if (warp == 0) {
            const uint32_t nf = min(ptx::lds_u32(CTL(s, nfin)), static_cast<uint32_t>(kFinish));
            uint64_t v = static_cast<uint32_t>(lane) < nf ? fin_s[lane] : 0ull;
            v = warp_sort_desc(v, lane);
            emit_lanes(static_cast<uint32_t>(lane) < need && static_cast<uint32_t>(lane) < nf, ~static_cast<uint32_t>(v));
            if (lane == 0 && nf < need) set_err(TOPK_FLAG_INTERNAL);
        }
        __syncthreads();
    };

    // Emits, in position order, the first `need` elements of src[0, n) whose
    // key is X (positions off + i); returns how many it emitted.
    auto collect_eq = [&](const float* src, uint32_t off, uint32_t n, uint32_t X, uint32_t need) -> uint32_t {
        const float4* s4 = reinterpret_cast<const float4*>(src);
        const uint32_t nv = (n + 3u) >> 2;
        uint32_t taken = 0;
        for (uint32_t v0 = 0; v0 < nv && taken < need; v0 += kST) {
            const uint32_t v = v0 + static_cast<uint32_t>(tid);
            const float4 x = v < nv ? __ldcg(s4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float xs[4] = {x.x, x.y, x.z, x.w};
            uint32_t m = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (v < nv && 4u * v + c < n && score_key(xs[c]) == X) m |= 1u << c;
            const uint32_t cnt = __popc(m);
            const uint32_t incl = warp_inclusive_sum(cnt, lane);
            if (lane == 31) warp_tot[warp] = incl;
            __syncthreads();
            uint32_t pre = 0, tot = 0;
#pragma unroll
            for (int w = 0; w < kST / 32; ++w) {
                const uint32_t t = warp_tot[w];
                pre += w < warp ? t : 0u;
                tot += t;
            }
            uint32_t slot = taken + pre + incl - cnt;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if ((m >> c) & 1u) {
                    if (slot < need) {
                        const uint32_t e = ptx::atom_add_s(CTL(s, nemit), 1u);
                        if (e < K)
                            ptx::sts_u32(sh_emit + 4u * e, off + 4u * v + c);
                        else
                            set_err(TOPK_FLAG_INTERNAL);
                    }
                    ++slot;
                }
            }
            taken += tot;
            __syncthreads();  // warp_tot is rewritten by the next step
        }
        return min(taken, need);
    };

    // Case c: the k largest composites of the whole row, from memory.
    auto full_row = [&](const float* rowp, uint32_t L, uint32_t need) {
        const float4* r4 = reinterpret_cast<const float4*>(rowp);
        const uint32_t nv = (L + 3u) >> 2;
        uint64_t r_lo = 0ull, r_hi = ~0ull;
        uint32_t cnt = L;
        for (int round = 0; cnt > kSplitCap; ++round) {
            if (round >= 8) {
                set_err(TOPK_FLAG_INTERNAL);
                break;
            }
            const int sh = shift_for_span64(r_hi - r_lo);
            for (uint32_t v0 = 0; v0 < nv; v0 += kStepVec * kST) {
                float4 x[kStepVec];
#pragma unroll
                for (uint32_t q = 0; q < kStepVec; ++q) {
                    const uint32_t v = v0 + q * kST + static_cast<uint32_t>(tid);
                    x[q] = v < nv ? __ldg(r4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (uint32_t q = 0; q < kStepVec; ++q) {
                    const uint32_t v = v0 + q * kST + static_cast<uint32_t>(tid);
                    const float xs[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
#pragma unroll
                    for (uint32_t c = 0; c < 4; ++c) {
                        const uint32_t idx = 4u * v + c;
                        if (v < nv && idx < L) {
                            const uint64_t w = composite(score_key(xs[c]), idx);
                            if (w >= r_lo && w <= r_hi)
                                ptx::red_add_s(sh_hist + 4u * static_cast<uint32_t>((w - r_lo) >> sh), 1u);
                        }
                    }
                }
            }
            __syncthreads();
            const ScanResult sr = scan_find<kST>(s, sh_hist, need, tid);
            clear_hist<kST, kBins>(sh_hist, tid);
            if (sr.bin >= static_cast<uint32_t>(kBins)) {
                set_err(TOPK_FLAG_INTERNAL);
                __syncthreads();
                break;
            }
            need -= sr.above;
            const uint64_t nlo = r_lo + (static_cast<uint64_t>(sr.bin) << sh);
            const uint64_t width = (1ull << sh) - 1ull;
            r_hi = (r_hi - nlo <= width) ? r_hi : nlo + width;
            r_lo = nlo;
            cnt = sr.count;
            __syncthreads();
        }
        // Collect: above the range -> emitted; inside -> the shared buffer.
        if (tid == 0) ptx::sts_u32(CTL(s, ncand), 0u);
        __syncthreads();
        for (uint32_t v0 = 0; v0 < nv; v0 += kStepVec * kST) {
            float4 x[kStepVec];
#pragma unroll
            for (uint32_t q = 0; q < kStepVec; ++q) {
                const uint32_t v = v0 + q * kST + static_cast<uint32_t>(tid);
                x[q] = v < nv ? __ldg(r4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (uint32_t q = 0; q < kStepVec; ++q) {
                const uint32_t v = v0 + q * kST + static_cast<uint32_t>(tid);
                const float xs[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
#pragma unroll
                for (uint32_t c = 0; c < 4; ++c) {
                    const uint32_t idx = 4u * v + c;
                    const bool live = v < nv && idx < L;
                    const uint64_t w = composite(score_key(xs[c]), idx);
                    emit_lanes(live && w > r_hi, idx);
                    const bool inr = live && w >= r_lo && w <= r_hi;
                    const uint32_t slot = warp_reserve(CTL(s, ncand), inr, lane);
                    if (inr) {
                        if (slot < kSplitCap)
                            cand_s[slot] = w;
                        else
                            set_err(TOPK_FLAG_INTERNAL);
                    }
                }
            }
        }
        __syncthreads();
        select_smem(min(ptx::lds_u32(CTL(s, ncand)), kSplitCap), r_lo, r_hi, need);
    };

    auto resolve = [&](int32_t row) {
        const SplitRow* rs = p.ws.rows + row;
        const uint32_t L = static_cast<uint32_t>(rs->len);  // > k: shorter rows have no segments
        const uint32_t lo = rs->lo;
        const float* rowp = p.scores + static_cast<int64_t>(row) * p.row_stride;
        const uint64_t* cand_g = p.ws.cand + static_cast<size_t>(row) * kSplitCap;
        // The row's counts, read once and shared: every branch below that
        // holds a barrier depends on them, so all threads must see one value.
        if (tid == 0) {
            ptx::sts_u32(CTL(s, nemit), 0u);
            s_vmax = 0ull;
            s_t = __ldcg(&rs->n_gt);
            s_e = __ldcg(&rs->n_eq);
        }
        __syncthreads();
        const uint32_t T = s_t;
        const uint32_t E = s_e;
        if (!p.full_resolve && T <= kSplitCap && T >= K) {
            // a. the k largest of the candidates
            // Every load of the buffer is issued before any is used (T <=
            // kSplitCap = 16 per thread): one round trip to L2.
            constexpr uint32_t kPer = kSplitCap / kST;
            unsigned long long vmax = 0ull;
            unsigned long long v[kPer];
#pragma unroll
            for (uint32_t q = 0; q < kPer; ++q) {
                const uint32_t i = q * kST + static_cast<uint32_t>(tid);
                v[q] = i < T ? __ldcg(reinterpret_cast<const unsigned long long*>(cand_g) + i) : 0ull;
            }
#pragma unroll
            for (uint32_t q = 0; q < kPer; ++q) {
                const uint32_t i = q * kST + static_cast<uint32_t>(tid);
                if (i < T) cand_s[i] = v[q];
                vmax = v[q] > vmax ? v[q] : vmax;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long t = __shfl_xor_sync(kFull, vmax, o);
                vmax = t > vmax ? t : vmax;
            }
            if (lane == 0) atomicMax(&s_vmax, vmax);
            __syncthreads();
            // every candidate's key is above lo, so its composite is at least (lo + 1) << 32
            select_smem(T, (static_cast<uint64_t>(lo) + 1ull) << 32, s_vmax, K);
        } else if (!p.full_resolve && T <= kSplitCap && static_cast<uint64_t>(T) + E >= K) {
            // b. every candidate, then the smallest positions of key lo
            // T < k <= kMaxK: at most kMaxK / kST loads per thread, all issued first.
            constexpr uint32_t kPerB = kMaxK / kST;
            unsigned long long v[kPerB];
#pragma unroll
            for (uint32_t q = 0; q < kPerB; ++q) {
                const uint32_t i = q * kST + static_cast<uint32_t>(tid);
                v[q] = i < T ? __ldcg(reinterpret_cast<const unsigned long long*>(cand_g) + i) : 0ull;
            }
#pragma unroll
            for (uint32_t q = 0; q < kPerB; ++q) {
                const uint32_t i = q * kST + static_cast<uint32_t>(tid);
                emit_lanes(i < T, ~static_cast<uint32_t>(v[q]));
            }
            __syncthreads();
            uint32_t need = K - T;
            const int32_t u0 = ustart[row];
            const int32_t nunits = rs->nunits;
            for (int32_t j = 0; j < nunits && need > 0u; ++j) {
                if (tid == 0) s_e = __ldcg(p.ws.unit_ties + u0 + j);
                __syncthreads();
                const uint32_t e = s_e;
                __syncthreads();  // read by all before thread 0 writes the next one
                if (e == 0u) continue;
                const uint32_t off = static_cast<uint32_t>(j) * seg;
                need -= collect_eq(rowp + off, off, min(seg, L - off), lo, need);
            }
            if (tid == 0 && need != 0u) set_err(TOPK_FLAG_INTERNAL);
            __syncthreads();
        } else {
            // c. the gate was above the k-th key, or the buffer overflowed
            full_row(rowp, L, K);
        }
        const uint32_t ne = ptx::lds_u32(CTL(s, nemit));
        if (tid == 0 && ne != K) set_err(TOPK_FLAG_INTERNAL);
        int32_t* out_row = p.out + static_cast<int64_t>(row) * p.k;
        int32_t* raw_row = p.raw_out ? p.raw_out + static_cast<int64_t>(row) * p.k : nullptr;
        const int32_t* pt_row = p.page_table + static_cast<int64_t>(row) * p.pt_stride;
        write_results<kST>(out_row, raw_row, pt_row, p.log2_page, K, 0u, static_cast<uint32_t>(tid),
                           [&](uint32_t q) -> int32_t {
                               return q < ne ? static_cast<int32_t>(ptx::lds_u32(sh_emit + 4u * q)) : -1;
                           });
        __syncthreads();  // the emit list and the buffers are free again
    };

    // Segment u: its row, its offset in the row and its length.
    auto locate = [&](uint32_t u, int32_t& row, uint32_t& off, uint32_t& n) {
        int32_t a = 0, b = p.batch - 1;  // the last row whose first segment is <= u
        while (a < b) {
            const int32_t mid = (a + b + 1) >> 1;
            if (static_cast<uint32_t>(ustart[mid]) <= u)
                a = mid;
            else
                b = mid - 1;
        }
        row = a;
        off = (u - static_cast<uint32_t>(ustart[a])) * seg;
        n = min(seg, row_len[a] - off);
    };
    auto prefetch_segment = [&](uint32_t u) {
        int32_t row;
        uint32_t off, n;
        locate(u, row, off, n);
        ptx::bulk_prefetch_l2(p.scores + static_cast<int64_t>(row) * p.row_stride + off, ((n + 3u) & ~3u) * 4u);
    };

    __syncthreads();  // ustart is loaded
    const uint32_t total = static_cast<uint32_t>(ustart[p.batch]);
    // Thread 0 claims the block's next segment while the current one
    // streams (its atomic is in flight meanwhile).  Segments are handed out
    // in order, so the one a block will claim about one round from now is
    // near u + gridDim.x: that one is prefetched into L2 when segment u starts.
    uint32_t nxt = 0u;
    const uint32_t G = gridDim.x;
    if (tid == 0) {
        const uint32_t cur = atomicAdd(&p.ws.hdr->next_unit, 1u);
        s_cur = cur;
        if (cur < total) prefetch_segment(cur);
    }
    __syncthreads();
    for (;;) {
        const uint32_t cur = s_cur;
        if (cur >= total) break;
        if (tid == 0) {
            if (cur + G < total) prefetch_segment(cur + G);
            nxt = atomicAdd(&p.ws.hdr->next_unit, 1u);
        }
        int32_t row;
        uint32_t off, n;
        locate(cur, row, off, n);
        const uint32_t lo = row_lo[row];
        const float4* src4 = reinterpret_cast<const float4*>(p.scores + static_cast<int64_t>(row) * p.row_stride + off);
        uint64_t* cand_g = p.ws.cand + static_cast<size_t>(row) * kSplitCap;
        uint32_t* n_gt = &p.ws.rows[row].n_gt;
        const uint32_t nv = (n + 3u) >> 2;  // the last float4 may run into the row's padding
        uint32_t eq = 0u;
        // The float of the gate key: key(x) >= lo <=> !(x < f_lo) and
        // key(x) == lo <=> x == f_lo for every non-NaN x; NaNs pass the first
        // compare (lo == 0 gives a NaN f_lo, so that everything passes).  A
        // thread first compares the NaN-propagating max of its 16 values;
        // only where that passes are the values tested one by one: ties are
        // counted, and the others are keyed exactly and, when above lo,
        // appended to the warp's staging area in shared memory.
        const float f_lo = key_float(lo);
        auto step = [&](const float4 (&x)[kStepVec], uint32_t c4) {
            float mq[kStepVec];
#pragma unroll
            for (uint32_t q = 0; q < kStepVec; ++q)
                mq[q] = ptx::fmax_nan(ptx::fmax_nan(x[q].x, x[q].y), ptx::fmax_nan(x[q].z, x[q].w));
            const float m = ptx::fmax_nan(ptx::fmax_nan(mq[0], mq[1]), ptx::fmax_nan(mq[2], mq[3]));
            if (m < f_lo) return;  // every value below the gate (m is a NaN if any value is)
            const uint32_t e_base = 4u * (c4 + static_cast<uint32_t>(tid));
#pragma unroll
            for (uint32_t q = 0; q < kStepVec; ++q) {
                if (mq[q] < f_lo) continue;  // this float4 holds nothing at or above the gate
                const uint32_t e0 = e_base + 4u * q * kST;
                const float xs[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
#pragma unroll
                for (uint32_t c = 0; c < 4; ++c) {
                    if (xs[c] < f_lo || e0 + c >= n) continue;
                    if (xs[c] == f_lo) {  // a tie with the gate key
                        ++eq;
                        continue;
                    }
                    const uint32_t key = score_key(xs[c]);
                    if (key > lo) {
                        const uint32_t slot = ptx::atom_add_s(wcnt_addr, 1u);
                        if (slot < kWarpStage) stage[slot] = composite(key, off + e0 + c);
                    } else if (key == lo) {  // f_lo is a NaN: ties are found by key
                        ++eq;
                    }
                }
            }
        };
        auto load = [&](float4 (&x)[kStepVec], uint32_t c4) {
#pragma unroll
            for (uint32_t q = 0; q < kStepVec; ++q) {
                const uint32_t v = c4 + q * kST + static_cast<uint32_t>(tid);
                x[q] = v < nv ? __ldcs(src4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        };
        // Two steps of loads in flight: the next step's loads are issued
        // before the current step is tested.
        constexpr uint32_t kStep = kStepVec * kST;  // float4s per step
        float4 xa[kStepVec], xb[kStepVec];
        load(xa, 0u);
        for (uint32_t c4 = 0; c4 < nv; c4 += 2u * kStep) {
            if (c4 + kStep < nv) load(xb, c4 + kStep);
            step(xa, c4);
            if (c4 + kStep >= nv) break;
            if (c4 + 2u * kStep < nv) load(xa, c4 + 2u * kStep);
            step(xb, c4 + kStep);
        }
        // The warp's staged candidates go to the row's buffer: one
        // reservation per warp and segment.  A warp whose staging area ran
        // full reserves past the buffer's capacity as well, so that the row
        // takes the full-row resolve.
        __syncwarp();
        {
            uint32_t wc = lane == 0 ? ptx::lds_u32(wcnt_addr) : 0u;
            wc = __shfl_sync(kFull, wc, 0);
            if (wc != 0u) {
                const uint32_t ns = min(wc, kWarpStage);
                uint32_t gb = 0u;
                if (lane == 0) {
                    gb = atomicAdd(n_gt, wc > kWarpStage ? ns + kSplitCap + 1u : ns);
                    ptx::sts_u32(wcnt_addr, 0u);
                }
                gb = __shfl_sync(kFull, gb, 0);
                for (uint32_t i = static_cast<uint32_t>(lane); i < ns; i += 32u)
                    if (gb + i < kSplitCap) cand_g[gb + i] = stage[i];
            }
        }
        eq = __reduce_add_sync(kFull, eq);
        if (lane == 0 && eq != 0u) atomicAdd(&s_eq, eq);
        __threadfence();  // this thread's candidate stores, before the segment counts as done
        __syncthreads();
        if (tid == 0) {
            const uint32_t e = s_eq;
            s_eq = 0u;
            p.ws.unit_ties[cur] = e;
            if (e != 0u) atomicAdd(&p.ws.rows[row].n_eq, e);
            __threadfence();
            const uint32_t d = atomicAdd(&p.ws.rows[row].done, 1u);
            const bool last = d + 1u == row_nunits[row];
            if (last) __threadfence();  // the other blocks' stores, before this block reads them
            s_res = last ? row : -1;
            s_cur = nxt;
        }
        __syncthreads();
        if (s_res >= 0) resolve(s_res);
    }
    if (tid == 0 && ctl.err != 0u) atomicOr(p.flags, ctl.err);
    // Dependents may start once every block has written its rows.
    __syncthreads();
    __threadfence();
    ptx::launch_dependents();
}

template <typename... Args>
cudaError_t launch_pdl(void (*kern)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
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
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t ensure_split_attributes() {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(split_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmBytes));
    if (e != cudaSuccess) return e;
    done.fetch_or(bit, std::memory_order_release);
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_split(const SplitParams& p, int grid, cudaStream_t stream) {
    cudaError_t e = ensure_split_attributes();
    if (e != cudaSuccess) return e;
    e = launch_pdl(split_gate_kernel, dim3(p.batch), dim3(kGT), 0, stream, p);
    if (e != cudaSuccess) return e;
    return launch_pdl(split_select_kernel, dim3(grid), dim3(kST), kSmBytes, stream, p);
}

cudaError_t split_occupancy(int* blocks_out) {
    cudaError_t e = ensure_split_attributes();
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, split_select_kernel, kST, kSmBytes);
    if (e != cudaSuccess) return e;
    *blocks_out = per_sm * sms;
    return cudaSuccess;
}

}  // namespace topkidx
