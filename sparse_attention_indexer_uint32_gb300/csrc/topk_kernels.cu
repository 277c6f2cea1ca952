// topk_kernels.cu -- sm_103a kernels of the indexer top-k + page-table
// transform: the row-select kernel (one block, or one thread-block cluster,
// per row), the plan kernel, the stand-alone page transform and the key map.
//
// Method (SGLang PR #26788 "[JIT Kernel] DeepSeek-V4 DSA indexer: faster
// top-k + page-table transform (runtime k <= 2048)" and the DistRadixTopK
// README "Ultra Low Latency Distributed Radix TopK Indexer Via NoC"): scores
// are mapped to order-preserving uint32 keys, a radix histogram over the keys
// finds the bin that holds the k-th largest key, later rounds refine that bin
// over a shrinking candidate set, the last <= 32 candidates are finished by a
// warp compare-and-swap sort, and a separate pass gathers the selected
// positions through the page table.  Long rows are split over a cluster whose
// blocks merge their histograms through distributed shared memory.
//
// GB300 choices (see the block comment above select_kernel): the row is
// streamed once by the bulk-copy (TMA) engine into a shared-memory ring that
// runs ahead across rows; a sampled gate keeps all but ~2k elements of a row
// away from the histogram atomics; the gated elements are kept on chip, so a
// second read of the row is only needed when they do not fit.

#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <type_traits>

#include "keys.cuh"
#include "ptx.cuh"
#include "select_common.cuh"
#include "topk_internal.h"
#include "topkidx.h"

namespace topkidx {
using namespace detail;

// ============================================================================
// select_kernel<NT, C>: NT threads per block, C blocks per row (C == 1: one
// block per row; C > 1: a thread-block cluster per row, each block owning a
// contiguous slice of the row, rank order == position order).
//
// Per row:
//  1. Gate.  Up to `samples` scores of the row are read (prefetched while the
//     previous row is processed).  Their keys give a lower bound `lo`: the
//     sample's r-th largest key (an 11-bit sample histogram, refined on the
//     next 11 bits when its bin is crowded), r = max(E + 4 sqrt(E) + 4, the
//     rank expected to fill a set share of the candidate buffer), E the
//     expected number of samples in the top k.  The bin width of the row's
//     histogram is chosen so that [lo, sample max] covers about 1024 of the
//     2048 bins (the "linear mapping" of the DistRadixTopK README: bins spread
//     over the range where the threshold lies, so few elements share its bin).
//  2. Pass 1 streams the slice through the bulk-copy ring.  Each thread tests
//     its float4s against the float of `lo` (one compare per element); each
//     warp reserves buffer slots for its gated elements with one atomic per
//     copy, and the gated elements are keyed exactly, counted in the
//     histogram and pushed (key, position) into the candidate buffer in
//     shared memory.  In a cluster the histograms are merged through
//     distributed shared memory.
//  3. Resolve.  Scanning the merged histogram from the top gives the bin of
//     the k-th key; later 11-bit rounds histogram only the candidates inside
//     that bin, until either the bin is a single key or it holds <= 32
//     candidates, which a warp sort finishes (ties by smaller position).
//     When the buffer overflowed (or the gate was too tight) the rounds
//     re-read the slice from memory instead, and once the threshold bin fits
//     a collect pass fills the buffer with it: the two-pass streaming path.
//     A single threshold key tied by many elements takes the smallest
//     positions: per-rank quotas in rank order, then a selection on position.
//  4. Emit + transform.  Selected positions go to a shared-memory list; after
//     a barrier the page-table gather writes out (and raw_out) coalesced,
//     padding with -1 (PR #26788, commit "Dynamic dispatch via the plan's
//     cluster_threshold": the transform is a separate pass).
// ============================================================================
template <int NT, int C, bool kRefresh = false>
__global__ void __launch_bounds__(NT, NT == 256 ? 3 : 2) select_kernel(const SelectParams p) {
    static_assert(!kRefresh || C == 1, "the gate refresh counts a whole row in one block");
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const Layout lay = make_layout(C, p.tile, p.stages, p.cap, p.k);
    const uint32_t sbase = ptx::smem_addr(smem_raw);
    Smem s;
    s.ring = sbase + lay.ring;
    s.hist_a = sbase + lay.hist_a;
    s.hist_b = sbase + lay.hist_b;
    s.hist_m = sbase + lay.hist_m;
    s.cand_key = sbase + lay.cand_key;
    s.cand_idx = sbase + lay.cand_idx;
    s.emit = sbase + lay.emit;
    s.fin_key = sbase + lay.fin_key;
    s.fin_idx = sbase + lay.fin_idx;
    s.warp_tot = sbase + lay.warp_tot;
    s.ctl = sbase + lay.ctl;
    s.it_row = sbase + lay.items_row;
    s.it_len = sbase + lay.items_len;
    s.it_tiles = sbase + lay.items_tiles;
    s.it_tile_start = sbase + lay.items_tile_start;
    s.claim = sbase + lay.claim;
    s.claim_ptr = reinterpret_cast<uint32_t*>(smem_raw + lay.claim);
    s.full = reinterpret_cast<uint64_t*>(smem_raw + lay.mbar);
    s.empty = s.full + p.stages;
    s.ctl_ptr = reinterpret_cast<Control*>(smem_raw + lay.ctl);

    constexpr int kSamplesPerThread = kMaxSamples / NT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = (C > 1) ? ptx::cluster_ctarank() : 0u;
    const uint32_t unit = (C > 1) ? ptx::cluster_id_x() : blockIdx.x;
    const uint32_t nunits = (C > 1) ? ptx::cluster_count_x() : gridDim.x;
    const uint32_t stages = static_cast<uint32_t>(p.stages);

    // ---------------------------------------------------------------- init
    // Shared memory only: with a programmatic launch this overlaps the tail
    // of the kernel before (the plan), whose results are read after the wait.
    if (tid == 0) {
        for (uint32_t i = 0; i < stages; ++i) {
            ptx::mbar_init(&s.full[i], 1);
            ptx::mbar_init(&s.empty[i], NT / 32);
        }
        ptx::fence_mbarrier_init();
        ptx::sts_u32(CTL(s, ncand), 0);
        ptx::sts_u32(CTL(s, nemit), 0);
        ptx::sts_u32(CTL(s, nfin), 0);
        ptx::sts_u32(CTL(s, smax), 0);
        ptx::sts_u32(CTL(s, err), 0);
        ptx::sts_u32(CTL(s, out_cursor[0]), 0);
        ptx::sts_u32(CTL(s, out_cursor[1]), 0);
        for (uint32_t i = 0; i < stages; ++i) ptx::sts_u32(s.claim + 4u * i, 0xffffffffu);
    }
    clear_hist<NT>(s.hist_a, tid);
    clear_hist<NT>(s.hist_b, tid);
    __syncthreads();
    // The cluster's start barrier is split: this block arrives now and waits
    // just before its first access to another block's shared memory (the
    // first histogram merge), so that the wait overlaps the prologue, the gate
    // and pass 1.  Every block of the cluster is running before any DSMEM
    // access.  (Block-uniform: every path to an exit goes through it.)
    bool cl_arrived = false;
    if (C > 1) {
        ptx::cluster_arrive();
        cl_arrived = true;
    }
    auto cluster_ready = [&]() {
        if (C > 1 && cl_arrived) {
            ptx::cluster_wait();
            cl_arrived = false;
        }
    };
    // Every global access of this kernel comes after this point: the
    // preceding grid in the stream has completed and its writes are visible.
    ptx::grid_dependency_wait();

    const PlanView pv = read_plan(p);
    if (!pv.ok) {
        if (tid == 0 && rank == 0 && unit == 0) atomicOr(p.flags, TOPK_FLAG_PLAN_MISMATCH);
        cluster_ready();
        return;  // same for every block of a cluster
    }
    const int32_t n_first = pv.n_first;
    const bool identity = pv.identity;  // the plan wrote no lists: item i is row i
    const int32_t n_items = pv.n_items;
    const int32_t my_items = snake_count(static_cast<int32_t>(unit), n_items, static_cast<int32_t>(nunits));
    if (my_items <= 0) {
        cluster_ready();
        return;  // same for every block of a cluster
    }

    const uint32_t K = static_cast<uint32_t>(p.k);
    const uint32_t cap = static_cast<uint32_t>(p.cap);
    const uint32_t tile = static_cast<uint32_t>(p.tile);  // a multiple of 4 * NT floats, <= 4 * 8 * NT
    const uint32_t vec_per_tile = tile / (4u * NT);       // float4s per thread per bulk-copy tile

    const uint64_t policy = ptx::l2_policy_evict_first();
    const uint32_t m_max = static_cast<uint32_t>(p.samples);
    auto set_err = [&](uint32_t f) { atomicOr(&s.ctl_ptr->err, f); };

    // Consumer tile sequence number (the same in every thread); tile t of the
    // sequence lives in ring stage t % stages (kept as cst) and belongs to
    // ring round t / stages (cround), whose parity its wait takes.
    uint32_t cseq = 0, cst = 0, cround = 0;
    // Cluster rows that reached the output step, and (rank 0, thread 0) the
    // last such row's k: row e takes its output slots from rank 0's
    // out_cursor[e & 1], which rank 0 checks and clears after the next row's
    // histogram merge (every rank is past row e's output by then).
    uint32_t erow = 0, prev_kp = 0;

    auto slice_of = [&](int32_t L, uint32_t& s0, uint32_t& s1) {
        const uint32_t chunk = ((static_cast<uint32_t>(L) + C - 1) / C + 3u) & ~3u;
        s0 = min(static_cast<uint32_t>(L), rank * chunk);
        s1 = min(static_cast<uint32_t>(L), s0 + chunk);
    };

    for (int32_t w0 = 0; w0 < my_items; w0 += kItemsMax) {
        const int32_t nw = min(kItemsMax, my_items - w0);
        for (int32_t i = tid; i < nw; i += NT) {
            const int32_t it = snake_item(static_cast<int32_t>(unit), w0 + i, static_cast<int32_t>(nunits));
            const int32_t row = identity ? (it < n_first ? it : it - n_first)
                                         : (it < n_first ? (p.items ? p.items[it] : it) : p.items2[it - n_first]);
            int32_t L = -1;
            uint32_t nt = 0;
            if (row < 0 || row >= p.batch) {  // a list that does not belong to this batch
                atomicOr(p.flags, TOPK_FLAG_PLAN_MISMATCH);
            } else {
                L = p.seq_lens[row];
                if (L < 0) {
                    atomicOr(p.flags, TOPK_FLAG_SEQ_NEGATIVE);
                    L = 0;
                } else if (L > p.max_seq_len) {
                    atomicOr(p.flags, TOPK_FLAG_SEQ_CLAMPED);
                    L = p.max_seq_len;
                }
                if (L > p.k) {  // rows with L <= k need no select, hence no tiles
                    uint32_t s0, s1;
                    slice_of(L, s0, s1);
                    if (s1 > s0) nt = ((((s1 + 3u) & ~3u) - s0) + tile - 1) / tile;
                }
            }
            ptx::sts_u32(s.it_row + 4u * i, static_cast<uint32_t>(row < 0 || row >= p.batch ? 0 : row));
            ptx::sts_u32(s.it_len + 4u * i, static_cast<uint32_t>(L));
            ptx::sts_u32(s.it_tiles + 4u * i, nt);
        }
        __syncthreads();
        // Tile sequence of this window: exclusive prefix of the items' tile counts.
        if (tid == 0) {
            uint32_t run = 0;
            for (int32_t i = 0; i < nw; ++i) {
                ptx::sts_u32(s.it_tile_start + 4u * i, run);
                run += ptx::lds_u32(s.it_tiles + 4u * i);
            }
            ptx::sts_u32(CTL(s, win_tiles), run);
        }
        __syncthreads();
        const uint32_t win_base = cseq;
        const uint32_t win_end = win_base + ptx::lds_u32(CTL(s, win_tiles));

        // Source address and byte count of window tile `t` (global sequence number).
        auto tile_src = [&](uint32_t t, uint32_t& bytes) -> const float* {
            const uint32_t qw = t - win_base;
            int32_t lo_i = 0, hi_i = nw - 1;  // largest item whose first tile is <= qw
            while (lo_i < hi_i) {
                const int32_t mid = (lo_i + hi_i + 1) >> 1;
                if (ptx::lds_u32(s.it_tile_start + 4u * mid) <= qw)
                    lo_i = mid;
                else
                    hi_i = mid - 1;
            }
            const uint32_t tile_in_item = qw - ptx::lds_u32(s.it_tile_start + 4u * lo_i);
            const int32_t L = static_cast<int32_t>(ptx::lds_u32(s.it_len + 4u * lo_i));
            uint32_t t0, t1;
            slice_of(L, t0, t1);
            const uint32_t n4 = ((t1 + 3u) & ~3u) - t0;
            const uint32_t off = tile_in_item * tile;
            const uint32_t elems = min(tile, n4 - off);
            const int32_t prow = static_cast<int32_t>(ptx::lds_u32(s.it_row + 4u * lo_i));
            bytes = elems * 4u;
            return p.scores + static_cast<int64_t>(prow) * p.row_stride + t0 + off;
        };
        // Issues the bulk copy of window tile `t` into its stage st = t % stages.
        auto issue_tile = [&](uint32_t t, uint32_t st) {
            uint32_t bytes;
            const float* src = tile_src(t, bytes);
            ptx::mbar_arrive_expect_tx(&s.full[st], bytes);
            ptx::bulk_copy_g2s_addr(s.ring + st * tile * 4u, src, bytes, &s.full[st], policy);
        };
        // Initial fill: the stages are all free at a window boundary.  A block
        // whose wait gave up issues no more copies (a stage it gave up on may
        // still be receiving its copy).
        // Lane i of warp 0 issues the copy of stage i, so the first copies go
        // out together.
        if (warp == 0 && static_cast<uint32_t>(lane) < stages &&
            (ptx::lds_u32(CTL(s, err)) & TOPK_FLAG_TIMEOUT) == 0u) {
            const uint32_t t = win_base + static_cast<uint32_t>(lane);
            if (t < win_end) {
                ptx::sts_u32(s.claim + 4u * (t % stages), t / stages);
                issue_tile(t, t % stages);
            }
        }
        // Called by lane 0 of every warp after it released tile t: the warp
        // whose release completed the stage refills it with tile t + stages
        // (one claim per stage and round), so the ring is refilled as soon as
        // the slowest warp is done, not when a designated producer gets to it.
        // (st, r: the stage and ring round of tile t.)
        // A warp that gave up waiting for a stage's copy records the timeout
        // before it releases the stage, so the refill sees the flag and leaves
        // the stage alone: at most one copy is ever in flight per stage.
        auto refill_after = [&](uint32_t t, uint32_t st, uint32_t r) {
            const uint32_t next = t + stages;
            if (next >= win_end) return;
            if (!ptx::mbar_test_wait(&s.empty[st], r & 1u)) return;
            if (ptx::lds_u32(CTL(s, err)) & TOPK_FLAG_TIMEOUT) return;
            if (atomicCAS(&s.claim_ptr[st], r, r + 1u) != r) return;
            issue_tile(next, st);
        };

        // Samples per row: 1024 for rows up to 16K, more for longer rows.
        auto samples_for = [&](uint32_t L) -> uint32_t {
            const uint32_t m = L <= 16384u ? min(m_max, 1024u) : m_max;
            return min(m, L);
        };
        // Gate samples of the next non-trivial row are loaded one row ahead.
        float smp[kSamplesPerThread];
        auto load_samples = [&](int32_t j) {
#pragma unroll
            for (int q = 0; q < kSamplesPerThread; ++q) smp[q] = 0.0f;
            if (j >= nw) return;
            const int32_t L = static_cast<int32_t>(ptx::lds_u32(s.it_len + 4u * j));
            if (L <= p.k) return;
            const uint32_t M = samples_for(static_cast<uint32_t>(L));
            const float* rowp =
                p.scores + static_cast<int64_t>(ptx::lds_u32(s.it_row + 4u * j)) * p.row_stride;
#pragma unroll
            for (int q = 0; q < kSamplesPerThread; ++q) {
                const uint32_t i = static_cast<uint32_t>(q * NT + tid);
                if (i < M) smp[q] = __ldg(rowp + sample_pos(i, static_cast<uint32_t>(L), M));
            }
        };
        load_samples(0);

        for (int32_t j = 0; j < nw; ++j) {
            const int32_t row = static_cast<int32_t>(ptx::lds_u32(s.it_row + 4u * j));
            const int32_t L = static_cast<int32_t>(ptx::lds_u32(s.it_len + 4u * j));
            if (L < 0) {  // rejected item: nothing to write
                load_samples(j + 1);
                continue;
            }
            const uint32_t Kp = min(K, static_cast<uint32_t>(L));
            int32_t* out_row = p.out + static_cast<int64_t>(row) * p.k;
            int32_t* raw_row = p.raw_out ? p.raw_out + static_cast<int64_t>(row) * p.k : nullptr;
            const int32_t* pt_row = p.page_table + static_cast<int64_t>(row) * p.pt_stride;

            if (static_cast<uint32_t>(L) <= K) {
                // Every position is selected (seq_len <= k): no select at all.
                if (rank == 0)
                    write_results<NT>(out_row, raw_row, pt_row, p.log2_page, K, 0u, tid, [&](uint32_t q) {
                        return q < static_cast<uint32_t>(L) ? static_cast<int32_t>(q) : -1;
                    });
                load_samples(j + 1);
                continue;
            }

            uint32_t s0, s1;
            slice_of(L, s0, s1);
            {
                // Pull this slice's page-table entries into L2 now, so that the
                // final gather finds them there.  Skipped when the slice spans
                // far more pages than results (small pages).
                const uint32_t pg0 = s0 >> p.log2_page;
                const uint32_t npg = s1 > s0 ? ((s1 - 1u) >> p.log2_page) - pg0 + 1u : 0u;
                if (npg > 0u && npg <= 8u * K)
                    for (uint32_t e = 32u * tid; e < npg + 31u; e += 32u * NT)
                        ptx::prefetch_l2(pt_row + pg0 + min(e, npg - 1u));
            }
            const uint32_t ntiles = ptx::lds_u32(s.it_tiles + 4u * j);
            const float* row_ptr = p.scores + static_cast<int64_t>(row) * p.row_stride;

            if (tid == 0) {
                ptx::sts_u32(CTL(s, ncand), 0);
                ptx::sts_u32(CTL(s, nemit), 0);
                ptx::sts_u32(CTL(s, nfin), 0);
                ptx::sts_u32(CTL(s, smax), 0);
                if (kRefresh) ptx::sts_u32(CTL(s, tkey), 0);
                if (C > 1) {  // both parities: the first buffered round may be an odd one
                    ptx::sts_u32(CTL(s, rnd_min[0]), 0xffffffffu);
                    ptx::sts_u32(CTL(s, rnd_max[0]), 0u);
                    ptx::sts_u32(CTL(s, rnd_cnt[0]), 0u);
                    ptx::sts_u32(CTL(s, rnd_min[1]), 0xffffffffu);
                    ptx::sts_u32(CTL(s, rnd_max[1]), 0u);
                    ptx::sts_u32(CTL(s, rnd_cnt[1]), 0u);
                }
            }
            __syncthreads();

            // ------------------------------------------------------ 1. gate
            uint32_t lo = 0;
            int shift = 32 - kBinBits;
            {
                // r = the sample rank used as the gate.  E samples are expected in the
                // row's top k; r = E + 4 sqrt(E) + 4 keeps the chance that fewer than k
                // elements pass the gate small (that case is detected and recounted),
                // and r is raised to aim at a share (p.gate_fill) of the on-chip
                // candidate capacity, which lowers the chance of a recount further.
                const uint32_t M = samples_for(static_cast<uint32_t>(L));
                const float E = static_cast<float>(M) * static_cast<float>(Kp) / static_cast<float>(L);
                const float r_safe = ceilf(E + 4.0f * sqrtf(E) + 4.0f);
                const float r_fill = floorf(p.gate_fill * static_cast<float>(cap) * C * static_cast<float>(M) /
                                            static_cast<float>(L));
                const float r_f = fmaxf(r_safe, r_fill);
                if (!p.disable_gate && r_f < static_cast<float>(M)) {
                    const uint32_t r = static_cast<uint32_t>(r_f);
                    uint32_t keys[kSamplesPerThread];
                    uint32_t kmax = 0;
#pragma unroll
                    for (int q = 0; q < kSamplesPerThread; ++q) {
                        const uint32_t i = static_cast<uint32_t>(q * NT + tid);
                        keys[q] = score_key(smp[q]);
                        if (i < M) {
                            ptx::red_add_s(s.hist_a + 4u * (keys[q] >> (32 - kBinBits)), 1u);
                            kmax = max(kmax, keys[q]);
                        }
                    }
                    kmax = __reduce_max_sync(kFull, kmax);
                    if (lane == 0) atomicMax(&s.ctl_ptr->smax, kmax);
                    __syncthreads();
                    const ScanResult g = scan_find<NT>(s, s.hist_a, r, tid);
                    lo = g.bin << (32 - kBinBits);
                    if (g.above + g.count > r + r / 4u + 4u && g.count > 1u) {
                        // Refine inside the coarse bin on the next 11 bits.
#pragma unroll
                        for (int q = 0; q < kSamplesPerThread; ++q) {
                            const uint32_t i = static_cast<uint32_t>(q * NT + tid);
                            if (i < M && (keys[q] >> (32 - kBinBits)) == g.bin)
                                ptx::red_add_s(s.hist_b + 4u * ((keys[q] >> (32 - 2 * kBinBits)) & (kBins - 1)), 1u);
                        }
                        __syncthreads();
                        const ScanResult g2 = scan_find<NT>(s, s.hist_b, r - g.above, tid);
                        lo |= g2.bin << (32 - 2 * kBinBits);
                        clear_hist<NT>(s.hist_b, tid);
                    }
                    clear_hist<NT>(s.hist_a, tid);
                    const uint32_t smax = ptx::lds_u32(CTL(s, smax));
                    const int b = bit_length(smax - lo);
                    shift = b > kBinBits - 1 ? b - (kBinBits - 1) : 0;
                    __syncthreads();
                }
            }
            load_samples(j + 1);
            // The float at the bottom of the gate: key(x) >= lo <=> !(x < f_lo) for
            // every non-NaN x (the inverse of the key map; lo = 0 gives a NaN,
            // so that everything passes).
            const float f_lo = key_float(lo);

            // ------------------------------------------------- 2. pass 1
            const bool buffering = !p.force_two_pass;
            // The tile loop, compiled for V float4s per thread per tile (the
            // tile and block sizes in use give V = 2, 4, 6 or 8).
            auto pass1 = [&](auto v_tag) {
                constexpr int V = decltype(v_tag)::value;
                for (uint32_t t = 0; t < ntiles; ++t) {
                    const uint32_t st = cst;
                    const bool gave_up = (ptx::lds_u32(CTL(s, err)) & TOPK_FLAG_TIMEOUT) != 0u;
                    if (!gave_up && !ptx::mbar_wait_bounded(&s.full[st], cround & 1u, p.timeout_ns))
                        set_err(TOPK_FLAG_TIMEOUT);
                    const uint32_t off = t * tile;
                    const uint32_t ring_st = s.ring + st * tile * 4u;
                    const uint32_t base_idx = s0 + off;
                    // Each thread tests float4s v = q * NT + tid of the tile against the
                    // gate into a bitmask with one float compare per element: with f_lo
                    // the float whose key is lo, !(x < f_lo) holds for every x with
                    // key(x) >= lo, and also for NaNs (and everything, if f_lo is a NaN).
                    // One warp-wide reservation per tile; only the gated elements, a
                    // small fraction, are re-read, keyed exactly, counted in the
                    // histogram and buffered.  A false positive (a NaN under the gate)
                    // fills its reserved slot with key 0, which no later step selects.
                    const uint32_t lim = min(s1 - base_idx, tile);  // valid elements in this tile
                    // The gate float of this copy: f_lo, or the tightened gate once a
                    // refresh has raised it (read once per warp and copy).
                    float f_gate = f_lo;
                    if constexpr (kRefresh) {
                        const uint32_t tk = ptx::lds_u32(CTL(s, tkey));
                        if (tk > lo) f_gate = key_float(tk);
                    }
                    uint32_t gmask = 0;
                    {
                        float4 x[V];  // this thread's float4s of the tile (a ragged tail is masked)
#pragma unroll
                        for (int q = 0; q < V; ++q) x[q] = ptx::lds_f4(ring_st + 16u * (q * NT + tid));
#pragma unroll
                        for (int q = 0; q < V; ++q)
                            gmask |= ((x[q].x < f_gate ? 0u : 1u) | (x[q].y < f_gate ? 0u : 2u) |
                                      (x[q].z < f_gate ? 0u : 4u) | (x[q].w < f_gate ? 0u : 8u))
                                     << (4 * q);
                    }
                    if (lim != tile) {
#pragma unroll
                        for (int q = 0; q < V; ++q) {
                            const uint32_t e0 = 4u * (q * NT + tid);
                            const uint32_t valid =
                                e0 + 4u <= lim ? 15u : (e0 >= lim ? 0u : (1u << (lim - e0)) - 1u);
                            gmask &= ~((15u & ~valid) << (4 * q));
                        }
                    }
                    // Gated elements: each lane keys its own gated elements exactly
                    // (re-read from the stage), counts them in the histogram and
                    // writes (key, position) into its reserved slots.  When the buffer
                    // is full (or not used) each lane counts its own elements instead.
                    const uint32_t cnt = __popc(gmask);
                    const WarpPrefix wp = warp_prefix_small(cnt, lane);
                    const uint32_t total = wp.total;
                    uint32_t wbase = 0;
                    if (buffering && lane == 0 && total != 0u) wbase = ptx::atom_add_s(CTL(s, ncand), total);
                    wbase = __shfl_sync(kFull, wbase, 0);
                    if (buffering && wbase + total <= cap) {
                        uint32_t slot = wbase + wp.excl;
                        while (gmask) {
                            const int e = __ffs(gmask) - 1;
                            gmask &= gmask - 1u;
                            const uint32_t idx_in_tile = 4u * (static_cast<uint32_t>(e >> 2) * NT + tid) + (e & 3);
                            const uint32_t key = score_key(__uint_as_float(ptx::lds_u32(ring_st + 4u * idx_in_tile)));
                            const bool pass = key >= lo;
                            if (pass)
                                ptx::red_add_s(s.hist_a + 4u * min((key - lo) >> shift, static_cast<uint32_t>(kBins - 1)),
                                               1u);
                            ptx::sts_u32(s.cand_key + 4u * slot, pass ? key : 0u);
                            ptx::sts_u32(s.cand_idx + 4u * slot, base_idx + idx_in_tile);
                            ++slot;
                        }
                    } else {
                        // Each lane counts its own gated elements (their float4s read
                        // again, straight-line); runs of one bin take one atomic (a
                        // flat row puts every element in the same bin).
                        // In a cluster (rows long enough to be split), elements equal
                        // to the gate float (key == lo, bin 0: a flat or top-tied row)
                        // are only counted, without keying.
                        uint32_t run_bin = 0u, run_n = 0u, n_lo = 0u;
                        auto count = [&](bool gated, float v) {
                            if constexpr (C > 1) {
                                if (gated && v == f_lo) {
                                    ++n_lo;
                                    return;
                                }
                            }
                            const uint32_t key = score_key(v);
                            if (gated && key >= lo) {
                                const uint32_t bin = min((key - lo) >> shift, static_cast<uint32_t>(kBins - 1));
                                if (bin != run_bin && run_n) {
                                    ptx::red_add_s(s.hist_a + 4u * run_bin, run_n);
                                    run_n = 0u;
                                }
                                run_bin = bin;
                                ++run_n;
                            }
                        };
#pragma unroll
                        for (int q = 0; q < V; ++q) {
                            if ((gmask >> (4 * q)) & 15u) {
                                const float4 y = ptx::lds_f4(ring_st + 16u * (q * NT + tid));
                                count((gmask >> (4 * q)) & 1u, y.x);
                                count((gmask >> (4 * q + 1)) & 1u, y.y);
                                count((gmask >> (4 * q + 2)) & 1u, y.z);
                                count((gmask >> (4 * q + 3)) & 1u, y.w);
                            }
                        }
                        if (run_n) ptx::red_add_s(s.hist_a + 4u * run_bin, run_n);
                        if (C > 1 && n_lo) ptx::red_add_s(s.hist_a, n_lo);
                    }
                    __syncwarp();
                    if (lane == 0) {
                        ptx::mbar_arrive(&s.empty[st]);
                        refill_after(cseq, st, cround);
                    }
                    if constexpr (kRefresh) {
                        // Gate refresh (SGLang PR #32094, "[DSA] Add LiteTopk fused
                        // indexer top-k prefill path for SM100", the threshold-refresh
                        // step of "Background: how LiteTopk replaces the dense top-k"
                        // and the recall argument of its summary): every
                        // gate_refresh copies one warp, taking turns, walks the live
                        // histogram from the top to the lowest bin b with at least Kp
                        // counted elements at or above it.  Those elements are real
                        // elements of the row with keys >= lo + (b << shift), so the
                        // row's Kp-th key is at least that: the gate may rise to it
                        // and no top-k element is lost.  Counts still being added make
                        // the walk undercount, which only lowers b (a looser gate).
                        const uint32_t R = static_cast<uint32_t>(p.gate_refresh);
                        if ((t + 1u) % R == 0u && static_cast<uint32_t>(warp) == ((t + 1u) / R) % (NT / 32u)) {
                            const uint32_t top = static_cast<uint32_t>(kBins) - 64u * (static_cast<uint32_t>(lane) + 1u);
                            uint32_t sum = 0;
#pragma unroll
                            for (int i = 0; i < 64; i += 4) {
                                const uint4 q4 = ptx::lds_u4(s.hist_a + 4u * (top + i));
                                sum += q4.x + q4.y + q4.z + q4.w;
                            }
                            const uint32_t incl = warp_inclusive_sum(sum, lane);  // lane 0 holds the top bins
                            const uint32_t reach = __ballot_sync(kFull, incl >= Kp);
                            if (reach != 0u && lane == __ffs(reach) - 1) {
                                uint32_t acc = incl - sum;
                                uint32_t b = top;
                                for (int i = 63; i >= 0; --i) {
                                    acc += ptx::lds_u32(s.hist_a + 4u * (top + i));
                                    if (acc >= Kp) {
                                        b = top + static_cast<uint32_t>(i);
                                        break;
                                    }
                                }
                                const uint64_t nk = static_cast<uint64_t>(lo) + (static_cast<uint64_t>(b) << shift);
                                if (nk > lo && nk <= 0xffffffffull) atomicMax(&s.ctl_ptr->tkey, static_cast<uint32_t>(nk));
                            }
                        }
                    }
                    ++cseq;
                    if (++cst == stages) {
                        cst = 0;
                        ++cround;
                    }
                }
            };
            if (NT == 256) {
                if (vec_per_tile == 8u)
                    pass1(std::integral_constant<int, 8>{});
                else if (vec_per_tile == 6u)
                    pass1(std::integral_constant<int, 6>{});
                else if (vec_per_tile == 4u)
                    pass1(std::integral_constant<int, 4>{});
                else
                    pass1(std::integral_constant<int, 2>{});
            } else {
                if (vec_per_tile == 4u)
                    pass1(std::integral_constant<int, 4>{});
                else
                    pass1(std::integral_constant<int, 2>{});
            }
            __syncthreads();

            const uint32_t local_ovf = (!buffering || ptx::lds_u32(CTL(s, ncand)) > cap) ? 1u : 0u;
            uint32_t hm = s.hist_a;
            if (C > 1) {
                if (tid == 0) ptx::sts_u32(s.hist_a + 4u * kSlotOverflow, local_ovf);
                cluster_ready();
                cluster_merge<NT, C>(s, s.hist_a, rank, tid);
                hm = s.hist_m;
                if (rank == 0 && tid == 0) {
                    const uint32_t a = CTL(s, out_cursor[0]) + 4u * ((erow + 1u) & 1u);
                    if (erow > 0u && ptx::lds_u32(a) != prev_kp) set_err(TOPK_FLAG_INTERNAL);
                    ptx::sts_u32(a, 0u);
                }
            }
            const bool overflow = (C > 1) ? (ptx::lds_u32(hm + 4u * kSlotOverflow) != 0u) : (local_ovf != 0u);
            ScanResult sr = scan_find<NT>(s, hm, Kp, tid, s.hist_a);

            // ----------------------------------------------------- 3. resolve
            uint32_t r_lo, r_hi, G, cnt, local_cnt = 0;
            bool stream_mode;
            if (sr.total < Kp || sr.bin >= static_cast<uint32_t>(kBins)) {
                // The gate was tighter than the k-th key: recount everything.
                r_lo = 0;
                r_hi = 0xffffffffu;
                G = 0;
                cnt = 0xffffffffu;
                stream_mode = true;
            } else {
                G = sr.above;
                const uint64_t b = sr.bin;
                r_lo = static_cast<uint32_t>(lo + (b << shift));
                r_hi = (sr.bin == kBins - 1)
                           ? 0xffffffffu
                           : static_cast<uint32_t>(min_u64(0xffffffffull, lo + ((b + 1) << shift) - 1));
                cnt = sr.count;
                stream_mode = overflow;
                local_cnt = sr.local;
            }
            clear_hist<NT>(s.hist_a, tid);
            uint32_t h_next = s.hist_b;
            uint32_t h_other = s.hist_a;

            const uint32_t n4_slice = (s1 > s0) ? ((s1 + 3u) & ~3u) - s0 : 0u;
            const uint32_t nvec_slice = n4_slice >> 2;
            const float4* slice4 = reinterpret_cast<const float4*>(row_ptr + s0);

            // Appends `idx` to the emit list for the lanes with `flag`; every lane
            // of the warp must call it.
            auto emit_warp = [&](bool flag, uint32_t idx) {
                const uint32_t slot = warp_reserve(CTL(s, nemit), flag, lane);
                if (flag) {
                    if (slot < K)
                        ptx::sts_u32(s.emit + 4u * slot, idx);
                    else
                        set_err(TOPK_FLAG_INTERNAL);
                }
            };
            // Emits the positions of the buffer entries that satisfy `take(key)`:
            // each thread reads 4 entries per step, one warp-wide reservation per
            // step.
            auto emit_from_buffer = [&](uint32_t nc, auto take) {
                for (uint32_t i0 = 0; i0 < nc; i0 += 4u * NT) {
                    uint32_t pos[4];
                    uint32_t m = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t i = i0 + q * NT + tid;
                        const bool in = i < nc;
                        const uint32_t key = in ? ptx::lds_u32(s.cand_key + 4u * i) : 0u;
                        pos[q] = in ? ptx::lds_u32(s.cand_idx + 4u * i) : 0u;
                        if (in && take(key)) m |= 1u << q;
                    }
                    uint32_t slot = warp_reserve_n(CTL(s, nemit), __popc(m), lane);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (m >> q & 1u) {
                            if (slot < K)
                                ptx::sts_u32(s.emit + 4u * slot, pos[q]);
                            else
                                set_err(TOPK_FLAG_INTERNAL);
                            ++slot;
                        }
                    }
                }
            };

            for (int round = 0;; ++round) {
                if (round > 8) {
                    set_err(TOPK_FLAG_INTERNAL);
                    break;
                }
                if (r_lo == r_hi) break;
                if (!stream_mode && cnt <= static_cast<uint32_t>(kFinish)) break;
                if (stream_mode && cnt <= cap) {
                    // Collect pass: emit everything above the bin, keep the bin.
                    __syncthreads();
                    if (tid == 0) ptx::sts_u32(CTL(s, ncand), 0);
                    __syncthreads();
                    // Four vectors in flight per lane: these re-reads are latency-bound.
                    for (uint32_t v0 = warp * 32u; v0 < nvec_slice; v0 += 4u * NT) {
                        float4 xv[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint32_t v = v0 + u * NT + lane;
                            xv[u] = v < nvec_slice ? __ldg(slice4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint32_t v = v0 + u * NT + lane;
                            const bool in = v < nvec_slice;
                            const float xs[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const uint32_t idx = s0 + 4u * v + c;
                                const uint32_t key = score_key(xs[c]);
                                const bool live = in && idx < s1;
                                emit_warp(live && key > r_hi, idx);
                                const bool keep = live && key >= r_lo && key <= r_hi;
                                const uint32_t slot = warp_reserve(CTL(s, ncand), keep, lane);
                                if (keep) {
                                    if (slot < cap) {
                                        ptx::sts_u32(s.cand_key + 4u * slot, key);
                                        ptx::sts_u32(s.cand_idx + 4u * slot, idx);
                                    } else {
                                        set_err(TOPK_FLAG_INTERNAL);
                                    }
                                }
                            }
                        }
                    }
                    __syncthreads();
                    stream_mode = false;
                    continue;
                }
                // One more 11-bit round over [r_lo, r_hi].
                const int sh = shift_for_span(r_hi - r_lo);
                const uint32_t par = static_cast<uint32_t>(round) & 1u;
                if (!stream_mode) {
                    const uint32_t nc = min(ptx::lds_u32(CTL(s, ncand)), cap);  // never past the buffer
                    uint32_t kmin = 0xffffffffu, kmax = 0u, kcnt = 0u;
                    for (uint32_t i = tid; i < nc; i += NT) {
                        const uint32_t key = ptx::lds_u32(s.cand_key + 4u * i);
                        if (key >= r_lo && key <= r_hi) {
                            ptx::red_add_s(h_next + 4u * ((key - r_lo) >> sh), 1u);
                            if constexpr (C > 1) {
                                kmin = min(kmin, key);
                                kmax = max(kmax, key);
                                ++kcnt;
                            }
                        }
                    }
                    if constexpr (C > 1) {
                        // The range's smallest and largest key over the cluster (each
                        // block's pair rides in its own slots of the merged histogram):
                        // when they are equal, the range is one key and the rounds end.
                        kmin = __reduce_min_sync(kFull, kmin);
                        kmax = __reduce_max_sync(kFull, kmax);
                        kcnt = __reduce_add_sync(kFull, kcnt);
                        if (lane == 0) {
                            atomicMin(&s.ctl_ptr->rnd_min[par], kmin);
                            atomicMax(&s.ctl_ptr->rnd_max[par], kmax);
                            atomicAdd(&s.ctl_ptr->rnd_cnt[par], kcnt);
                        }
                    }
                } else {
                    for (uint32_t v0 = tid; v0 < nvec_slice; v0 += 4u * NT) {
                        float4 xv[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint32_t v = v0 + u * NT;
                            xv[u] = v < nvec_slice ? __ldg(slice4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                        uint32_t run_bin = 0u, run_n = 0u;  // runs of one bin: one atomic
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint32_t v = v0 + u * NT;
                            const float xs[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const uint32_t idx = s0 + 4u * v + c;
                                const uint32_t key = score_key(xs[c]);
                                if (v < nvec_slice && idx < s1 && key >= r_lo && key <= r_hi) {
                                    const uint32_t bin = (key - r_lo) >> sh;
                                    if (bin != run_bin && run_n) {
                                        ptx::red_add_s(h_next + 4u * run_bin, run_n);
                                        run_n = 0u;
                                    }
                                    run_bin = bin;
                                    ++run_n;
                                }
                            }
                        }
                        if (run_n) ptx::red_add_s(h_next + 4u * run_bin, run_n);
                    }
                }
                __syncthreads();
                uint32_t hr = h_next;
                if (C > 1) {
                    if (!stream_mode && tid == 0) {
                        ptx::sts_u32(h_next + 4u * (kSlotRankMin + rank), ptx::lds_u32(CTL(s, rnd_min[0]) + 4u * par));
                        ptx::sts_u32(h_next + 4u * (kSlotRankMax + rank), ptx::lds_u32(CTL(s, rnd_max[0]) + 4u * par));
                        ptx::sts_u32(CTL(s, rnd_min[0]) + 4u * (par ^ 1u), 0xffffffffu);  // the next round's fields
                        ptx::sts_u32(CTL(s, rnd_max[0]) + 4u * (par ^ 1u), 0u);
                        ptx::sts_u32(CTL(s, rnd_cnt[0]) + 4u * (par ^ 1u), 0u);
                    }
                    cluster_merge<NT, C>(s, h_next, rank, tid);
                    hr = s.hist_m;
                    if (!stream_mode) {
                        uint32_t gmin = 0xffffffffu, gmax = 0u;
                        for (uint32_t q = 0; q < static_cast<uint32_t>(C); ++q) {
                            gmin = min(gmin, ptx::lds_u32(hr + 4u * (kSlotRankMin + q)));
                            gmax = max(gmax, ptx::lds_u32(hr + 4u * (kSlotRankMax + q)));
                        }
                        if (gmin == gmax) {  // one key left in the range (cluster-uniform)
                            local_cnt = ptx::lds_u32(CTL(s, rnd_cnt[0]) + 4u * par);
                            r_lo = gmin;
                            r_hi = gmin;
                            clear_hist<NT>(h_next, tid);
                            break;
                        }
                    }
                }
                sr = scan_find<NT>(s, hr, Kp - G, tid, h_next);
                if (sr.bin >= static_cast<uint32_t>(kBins)) {  // cannot happen: the bin holds >= need
                    set_err(TOPK_FLAG_INTERNAL);
                    clear_hist<NT>(h_next, tid);
                    break;
                }
                local_cnt = sr.local;
                G += sr.above;
                const uint64_t b = sr.bin;
                const uint32_t nlo = static_cast<uint32_t>(r_lo + (b << sh));
                const uint32_t nhi = static_cast<uint32_t>(min_u64(r_hi, r_lo + ((b + 1) << sh) - 1));
                r_lo = nlo;
                r_hi = nhi;
                cnt = sr.count;
                clear_hist<NT>(h_next, tid);
                const uint32_t t = h_next;
                h_next = h_other;
                h_other = t;
            }
            __syncthreads();

            const uint32_t need = Kp - G;
            if (r_lo == r_hi) {
                // ---- a single threshold key T; `need` of its `cnt` copies are taken
                const uint32_t T = r_lo;
                uint32_t quota = need;
                if (C > 1) {
                    if (tid < C) ptx::st_cluster_u32(ptx::map_rank(CTL(s, rank_eq) + 4u * rank, tid), local_cnt);
                    ptx::cluster_sync();
                    uint32_t before = 0;
                    for (uint32_t q = 0; q < rank; ++q) before += ptx::lds_u32(CTL(s, rank_eq) + 4u * q);
                    quota = need > before ? min(need - before, local_cnt) : 0u;
                }
                const bool all_eq = (quota == local_cnt);
                if (!stream_mode) {
                    const uint32_t nc = min(ptx::lds_u32(CTL(s, ncand)), cap);  // never past the buffer
                    emit_from_buffer(nc, [&](uint32_t key) { return key > T || (all_eq && key == T); });
                    if (!all_eq && quota > 0) {
                        // The `quota` smallest positions among this block's copies of T:
                        // rounds on v = ~position (larger v = smaller position).
                        uint32_t v_lo = ~(s1 - 1u), v_hi = ~s0, v_g = 0, v_cnt = local_cnt;
                        for (int vr = 0; vr < 6; ++vr) {
                            if (v_lo == v_hi || v_cnt <= static_cast<uint32_t>(kFinish)) break;
                            const int sh = shift_for_span(v_hi - v_lo);
                            for (uint32_t i = tid; i < nc; i += NT) {
                                const uint32_t v = ~ptx::lds_u32(s.cand_idx + 4u * i);
                                if (ptx::lds_u32(s.cand_key + 4u * i) == T && v >= v_lo && v <= v_hi)
                                    ptx::red_add_s(h_next + 4u * ((v - v_lo) >> sh), 1u);
                            }
                            __syncthreads();
                            const ScanResult vs = scan_find<NT>(s, h_next, quota - v_g, tid);
                            v_g += vs.above;
                            const uint64_t b = vs.bin;
                            const uint32_t nlo = static_cast<uint32_t>(v_lo + (b << sh));
                            const uint32_t nhi = static_cast<uint32_t>(min_u64(v_hi, v_lo + ((b + 1) << sh) - 1));
                            v_lo = nlo;
                            v_hi = nhi;
                            v_cnt = vs.count;
                            clear_hist<NT>(h_next, tid);
                            __syncthreads();
                        }
                        // Above the final range: taken.  Inside it: a warp sort picks the rest.
                        if (tid == 0) ptx::sts_u32(CTL(s, nfin), 0);
                        __syncthreads();
                        for (uint32_t i0 = warp * 32u; i0 < nc; i0 += NT) {
                            const uint32_t i = i0 + lane;
                            const bool eq = i < nc && ptx::lds_u32(s.cand_key + 4u * i) == T;
                            const uint32_t pos = eq ? ptx::lds_u32(s.cand_idx + 4u * i) : 0u;
                            const uint32_t v = ~pos;
                            emit_warp(eq && v > v_hi, pos);
                            const bool fin = eq && v >= v_lo && v <= v_hi;
                            const uint32_t slot = warp_reserve(CTL(s, nfin), fin, lane);
                            if (fin) {
                                if (slot < static_cast<uint32_t>(kFinish)) {
                                    ptx::sts_u32(s.fin_key + 4u * slot, v);
                                    ptx::sts_u32(s.fin_idx + 4u * slot, pos);
                                } else {
                                    set_err(TOPK_FLAG_INTERNAL);
                                }
                            }
                        }
                        __syncthreads();
                        if (warp == 0) {
                            const uint32_t nf = min(ptx::lds_u32(CTL(s, nfin)), static_cast<uint32_t>(kFinish));
                            const uint64_t e = lane < static_cast<int>(nf)
                                                   ? (static_cast<uint64_t>(ptx::lds_u32(s.fin_key + 4u * lane)) << 32) | 1ull
                                                   : 0ull;
                            const uint64_t srt = warp_sort_desc(e, lane);
                            const uint32_t take = quota - v_g;
                            emit_warp(static_cast<uint32_t>(lane) < take && srt != 0ull,
                                      ~static_cast<uint32_t>(srt >> 32));
                        }
                    }
                } else {
                    // Final streaming pass: > T is taken; copies of T up to the quota,
                    // in position order when only some of them are taken.
                    // With nothing above T anywhere (G == 0: a flat or top-tied row),
                    // a block that takes no copies skips the pass, and one that takes
                    // some stops as soon as its quota is met.
                    const bool ordered = (!all_eq && quota > 0);
                    const bool none_above = (G == 0u);
                    const uint32_t vend = (none_above && !all_eq && quota == 0u) ? 0u : nvec_slice;
                    uint32_t running = 0;
                    for (uint32_t vb = 0; vb < vend; vb += NT) {
                        if (none_above && ordered && running >= quota) break;  // block-uniform
                        const uint32_t v = vb + tid;
                        uint32_t eqm = 0;
                        const bool in = v < nvec_slice;
                        const float4 x = in ? __ldg(slice4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint32_t idx = s0 + 4u * v + c;
                            const uint32_t key = score_key(xs[c]);
                            const bool live = in && idx < s1;
                            emit_warp(live && key > T, idx);
                            if (live && key == T) eqm |= 1u << c;
                        }
                        if (!ordered) {
#pragma unroll
                            for (int c = 0; c < 4; ++c) emit_warp(all_eq && (eqm >> c & 1u), s0 + 4u * v + c);
                            continue;
                        }
                        const uint32_t n_eq = __popc(eqm);
                        const uint32_t incl = warp_inclusive_sum(n_eq, lane);
                        if (lane == 31) ptx::sts_u32(s.warp_tot + 4u * warp, incl);
                        __syncthreads();
                        uint32_t pre = 0, tot = 0;
                        for (int w = 0; w < NT / 32; ++w) {
                            const uint32_t t = ptx::lds_u32(s.warp_tot + 4u * w);
                            pre += (w < warp) ? t : 0u;
                            tot += t;
                        }
                        uint32_t r0 = running + pre + incl - n_eq;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const bool e = (eqm >> c & 1u) != 0u;
                            emit_warp(e && r0 < quota, s0 + 4u * v + c);
                            r0 += e ? 1u : 0u;
                        }
                        running += tot;
                        __syncthreads();
                    }
                }
            } else {
                // ---- <= 32 candidates in [r_lo, r_hi]: warp compare-and-swap finish
                // One pass over the buffer: entries above the range are emitted,
                // entries inside it go to the finish list (of rank 0 in a cluster),
                // or are emitted too when all of them are taken (need == count: no
                // sort and no barrier).
                const bool take_range = need >= cnt;
                const uint32_t nc = min(ptx::lds_u32(CTL(s, ncand)), cap);  // never past the buffer
                for (uint32_t i0 = 0; i0 < nc; i0 += 4u * NT) {
                    uint32_t key[4], pos[4];
                    uint32_t m = 0, f = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t i = i0 + q * NT + tid;
                        const bool in = i < nc;
                        key[q] = in ? ptx::lds_u32(s.cand_key + 4u * i) : 0u;
                        pos[q] = in ? ptx::lds_u32(s.cand_idx + 4u * i) : 0u;
                        const bool in_range = in && key[q] >= r_lo && key[q] <= r_hi;
                        if ((in && key[q] > r_hi) || (take_range && in_range)) m |= 1u << q;
                        if (!take_range && in_range) f |= 1u << q;
                    }
                    uint32_t slot = warp_reserve_n(CTL(s, nemit), __popc(m), lane);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (m >> q & 1u) {
                            if (slot < K)
                                ptx::sts_u32(s.emit + 4u * slot, pos[q]);
                            else
                                set_err(TOPK_FLAG_INTERNAL);
                            ++slot;
                        }
                        if (f >> q & 1u) {
                            if (C > 1) {
                                const uint32_t fs = ptx::atom_add_cluster_u32(ptx::map_rank(CTL(s, nfin), 0), 1u);
                                if (fs < static_cast<uint32_t>(kFinish)) {
                                    ptx::st_cluster_u32(ptx::map_rank(s.fin_key + fs * 4u, 0), key[q]);
                                    ptx::st_cluster_u32(ptx::map_rank(s.fin_idx + fs * 4u, 0), pos[q]);
                                } else {
                                    set_err(TOPK_FLAG_INTERNAL);
                                }
                            } else {
                                const uint32_t fs = ptx::atom_add_s(CTL(s, nfin), 1u);
                                if (fs < static_cast<uint32_t>(kFinish)) {
                                    ptx::sts_u32(s.fin_key + 4u * fs, key[q]);
                                    ptx::sts_u32(s.fin_idx + 4u * fs, pos[q]);
                                } else {
                                    set_err(TOPK_FLAG_INTERNAL);
                                }
                            }
                        }
                    }
                }
                if (!take_range) {
                    if (C > 1)
                        ptx::cluster_sync();
                    else
                        __syncthreads();
                }
                if (!take_range && rank == 0 && warp == 0) {
                    const uint32_t nf = min(ptx::lds_u32(CTL(s, nfin)), static_cast<uint32_t>(kFinish));
                    const uint64_t e =
                        lane < static_cast<int>(nf)
                            ? (static_cast<uint64_t>(ptx::lds_u32(s.fin_key + 4u * lane)) << 32) |
                                  (~ptx::lds_u32(s.fin_idx + 4u * lane))
                            : 0ull;
                    const uint64_t srt = warp_sort_desc(e, lane);
                    emit_warp(static_cast<uint32_t>(lane) < need && srt != 0ull,
                              ~static_cast<uint32_t>(srt & 0xffffffffull));
                }
            }
            __syncthreads();

            // ------------------------------------------- 4. transform + write
            const uint32_t nemit = min(ptx::lds_u32(CTL(s, nemit)), K);
            if (C == 1) {
                if (nemit != Kp && tid == 0) set_err(TOPK_FLAG_INTERNAL);
                write_results<NT>(out_row, raw_row, pt_row, p.log2_page, K, 0u, tid, [&](uint32_t q) {
                    return q < nemit ? static_cast<int32_t>(ptx::lds_u32(s.emit + 4u * q)) : -1;
                });
            } else {
                // Output slots come from one atomic on rank 0's cursor (no
                // cluster barrier); all ranks together emit exactly Kp.
                if (tid == 0)
                    ptx::sts_u32(CTL(s, out_base),
                                 ptx::atom_add_cluster_u32(
                                     ptx::map_rank(CTL(s, out_cursor[0]) + 4u * (erow & 1u), 0), nemit));
                __syncthreads();
                const uint32_t before = ptx::lds_u32(CTL(s, out_base));
                if (tid == 0 && before + nemit > Kp) set_err(TOPK_FLAG_INTERNAL);
                const uint32_t n_own = before < Kp ? min(nemit, Kp - before) : 0u;
                write_results<NT>(out_row, raw_row, pt_row, p.log2_page, n_own, before, tid, [&](uint32_t q) {
                    return static_cast<int32_t>(ptx::lds_u32(s.emit + 4u * q));
                });
                if (rank == 0) {
                    for (uint32_t q = Kp + tid; q < K; q += NT) {
                        out_row[q] = -1;
                        if (raw_row) raw_row[q] = -1;
                    }
                }
                if (tid == 0) prev_kp = Kp;
                ++erow;
            }
            __syncthreads();
        }
        __syncthreads();
    }

    // Drain: every issued tile was consumed unless a wait gave up; then the
    // last copy of each stage is waited for before the block exits, with the
    // drain's own limit (not the caller's wait limit, which may be short).
    if (tid == 0 && (ptx::lds_u32(CTL(s, err)) & TOPK_FLAG_TIMEOUT)) {
        for (uint32_t st = 0; st < stages; ++st) {
            const uint32_t r = ptx::lds_u32(s.claim + 4u * st);
            if (r != 0xffffffffu) ptx::mbar_wait_bounded(&s.full[st], r & 1u, kDrainLimitNs);
        }
    }
    if (C > 1) {
        cluster_ready();
        ptx::cluster_sync();  // no block leaves while others may still address its shared memory
        // every rank is past its last output: rank 0 checks the last row's slot count
        if (rank == 0 && tid == 0 && erow > 0u &&
            ptx::lds_u32(CTL(s, out_cursor[0]) + 4u * ((erow - 1u) & 1u)) != prev_kp)
            set_err(TOPK_FLAG_INTERNAL);
    }
    if (tid == 0) {
        const uint32_t err = ptx::lds_u32(CTL(s, err));
        if (err) atomicOr(p.flags, err);
    }
    // Every output store of this block has been issued: a kernel launched
    // after this one with programmatic serialization may be placed now (SGLang
    // PR #26788, commit log: the dependents are triggered only after the full
    // output is written).  It still waits for this grid's completion before
    // reading the output.
    __syncthreads();
    __threadfence();
    ptx::launch_dependents();
}

namespace {

__device__ __forceinline__ int length_bucket(int32_t L) {
    if (L <= 0) return 0;
    const int bl = bit_length(static_cast<uint32_t>(L));
    if (bl < 2) return 2 * bl;
    return 2 * bl + ((L >> (bl - 2)) & 1);
}

// Plan (PR #26788, commit "Replace the per-element cluster launch ...": the
// plan compacts the long items into a work list).  One block: every row is
// classified long (clamped seq_len > threshold) or short, and each class is
// written as a list ordered by half-octave length bucket, longest first, so
// that the persistent kernels hand out the longest rows first.  Lengths are
// loaded into registers up front (no dependent load chain), and a thread's
// run of rows with one (class, bucket) takes one atomic.
constexpr int kPlanPerThread = 16;  // rows held in registers per thread in one sweep
constexpr int kPlanKeys = 128;      // 2 classes x 64 length buckets

__device__ __forceinline__ int32_t clamp_len(int32_t L, int32_t max_seq_len, uint32_t* flags) {
    if (L < 0) {
        *flags |= TOPK_FLAG_SEQ_NEGATIVE;
        return 0;
    }
    if (L > max_seq_len) {
        *flags |= TOPK_FLAG_SEQ_CLAMPED;
        return max_seq_len;
    }
    return L;
}

// Each row gets the key (class, bucket): long rows (L > threshold) take keys
// 64..127, short rows 0..63, longer buckets higher.  The lists are written in
// descending key order, so position = (rows with a higher key) + (rows with
// the same key counted before it).  Counts are kept per warp (no contention
// between warps) and turned into per-warp starting offsets by one block-wide
// exclusive scan over (key descending, warp ascending).
// PT threads (256 for batches of up to 4096 rows, 512 up to 8192, 1024
// above: fewer warps make the block barriers of a small batch cheaper).
template <int PT>
__global__ void __launch_bounds__(PT) plan_kernel(const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                                  int32_t threshold, void* ws) {
    constexpr int kPlanThreads = PT;
    constexpr int kPlanWarps = PT / 32;
    constexpr int kLanesPerKey = kPlanWarps / 4;  // a key's kPlanWarps counters, 4 per lane
    static_assert(kPlanWarps >= 4 && kPlanKeys * kPlanWarps == 4 * PT, "four scan entries per thread, one key");
    __shared__ uint32_t cnt[kPlanKeys][kPlanWarps];  // per-warp counts, then per-warp cursors
    __shared__ uint32_t warp_sum[kPlanWarps];
    __shared__ uint32_t flags_s;
    __shared__ uint32_t uniform_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // The select kernel that follows waits for this grid's completion before
    // reading the lists, so it may be placed on the GPU right away.
    ptx::launch_dependents();
    int32_t* lists[2] = {plan_short_list(ws, batch), plan_long_list(ws)};
    uint32_t flags = 0;
    if (tid == 0) {
        flags_s = 0;
        uniform_s = 0;
    }
    // A batch that fits one sweep and whose rows all share one key needs no
    // lists: the order is the identity, which the header says instead.
    const bool one_sweep = batch <= kPlanThreads * kPlanPerThread;
    uint32_t n_long_total = 0;
    for (int32_t base = 0; base < batch; base += kPlanThreads * kPlanPerThread) {
        uint32_t* c = &cnt[0][0];
        for (int i = tid; i < kPlanKeys * kPlanWarps; i += kPlanThreads) c[i] = 0;
        __syncthreads();
        // All loads are issued before any is used (indices clamped into the
        // batch rather than branched around), so their latencies overlap.
        int32_t len[kPlanPerThread];
#pragma unroll
        for (int q = 0; q < kPlanPerThread; ++q)
            len[q] = __ldg(seq_lens + min(base + q * kPlanThreads + tid, batch - 1));
        uint32_t key[kPlanPerThread];
#pragma unroll
        for (int q = 0; q < kPlanPerThread; ++q) {
            const int32_t b = base + q * kPlanThreads + tid;
            key[q] = 0xffffffffu;
            if (b < batch) {
                const int32_t L = clamp_len(len[q], max_seq_len, &flags);
                key[q] = static_cast<uint32_t>((L > threshold ? 64 : 0) + length_bucket(L));
            }
        }
        // Runs of equal keys within a thread's rows take one atomic each (rows
        // of a batch often share a length, and so every lane of a warp would
        // otherwise hit the same counter for every row).
        {
            uint32_t run_key = key[0], run_len = 0;
#pragma unroll
            for (int q = 0; q < kPlanPerThread; ++q) {
                if (key[q] != run_key) {
                    if (run_key != 0xffffffffu && run_len) atomicAdd(&cnt[run_key][warp], run_len);
                    run_key = key[q];
                    run_len = 0;
                }
                ++run_len;
            }
            if (run_key != 0xffffffffu && run_len) atomicAdd(&cnt[run_key][warp], run_len);
        }
        __syncthreads();
        // Exclusive scan over entries e = 0..4 PT - 1 ordered (key desc, warp
        // asc): thread t owns entries 4t..4t+3, which share one key.
        const uint32_t k = kPlanKeys - 1 - (4 * tid) / kPlanWarps;
        const int w0 = (4 * tid) % kPlanWarps;
        uint32_t v[4], sum = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            v[u] = cnt[k][w0 + u];
            sum += v[u];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) warp_sum[warp] = incl;
        {
            // the kLanesPerKey lanes that own one key hold its whole count
            uint32_t key_total = sum;
#pragma unroll
            for (int o = 1; o < kLanesPerKey; o <<= 1) key_total += __shfl_xor_sync(kFull, key_total, o);
            if (one_sweep && (lane & (kLanesPerKey - 1)) == 0 && key_total == static_cast<uint32_t>(batch))
                uniform_s = 1;
        }
        __syncthreads();
        uint32_t pre = 0, n_long = 0;
        for (int w = 0; w < kPlanWarps; ++w) {
            const uint32_t t = warp_sum[w];
            pre += (w < warp) ? t : 0u;
            n_long += (w < kPlanWarps / 2) ? t : 0u;  // keys 64..127 are the first half of the order
        }
        uint32_t run = pre + incl - sum;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            cnt[k][w0 + u] = run;
            run += v[u];
        }
        __syncthreads();
        if (!uniform_s) {
            // Same runs: one atomic reserves a run's positions (run lengths are
            // counted backwards first).
            uint32_t rl[kPlanPerThread];
#pragma unroll
            for (int q = kPlanPerThread - 1; q >= 0; --q)
                rl[q] = (q + 1 < kPlanPerThread && key[q + 1] == key[q]) ? rl[q + 1] + 1u : 1u;
            uint32_t pos = 0;
#pragma unroll
            for (int q = 0; q < kPlanPerThread; ++q) {
                if (key[q] == 0xffffffffu) continue;
                if (q == 0 || key[q] != key[q - 1]) pos = atomicAdd(&cnt[key[q]][warp], rl[q]);
                const int32_t b = base + q * kPlanThreads + tid;
                if (key[q] >= 64u)
                    lists[1][n_long_total + pos] = b;
                else
                    lists[0][(static_cast<uint32_t>(base) - n_long_total) + (pos - n_long)] = b;
                ++pos;
            }
        }
        n_long_total += n_long;
        __syncthreads();
    }
    if (flags) atomicOr(&flags_s, flags);
    __syncthreads();
    if (tid == 0) {
        PlanHeader* h = static_cast<PlanHeader*>(ws);
        h->magic = kPlanMagic;
        h->batch = batch;
        h->max_seq_len = max_seq_len;
        h->long_threshold = threshold;
        h->n_long = static_cast<int32_t>(n_long_total);
        h->n_short = batch - static_cast<int32_t>(n_long_total);
        h->flags = flags_s;
        h->identity = uniform_s ? 1 : 0;
    }
}

// The stand-alone gather pass.  It is launched with programmatic stream
// serialization, so that it can be placed while the select kernel that wrote
// `raw` finishes (the select kernels trigger their dependents after their
// last output store); it waits for that grid before reading anything.
__global__ void page_transform_kernel(const int32_t* raw, int32_t batch, int32_t k, const int32_t* page_table,
                                      int64_t pt_stride, int32_t log2_page, int32_t* out) {
    ptx::grid_dependency_wait();
    const int64_t n = static_cast<int64_t>(batch) * k;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = i / k;
        out[i] = page_map(page_table + b * pt_stride, log2_page, raw[i]);
    }
    __syncthreads();
    __threadfence();
    ptx::launch_dependents();
}

__global__ void key_map_kernel(const float* x, int64_t n, uint32_t* keys) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        keys[i] = score_key(x[i]);
}

// Raises the kernel's dynamic shared-memory limit to the device's opt-in
// maximum (and allows 16-block clusters) once per device.  The limit is only
// a ceiling, so every launch below it stays valid whatever its size.
template <int NT, int C, bool R = false>
cudaError_t ensure_attributes() {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(select_kernel<NT, C, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e != cudaSuccess) return e;
    if (C > 8) {
        e = cudaFuncSetAttribute(select_kernel<NT, C, R>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    done.fetch_or(bit, std::memory_order_release);
    return cudaSuccess;
}

template <int NT, int C, bool R = false>
cudaError_t launch_select_t(const SelectParams& p, int grid_units, size_t smem, cudaStream_t stream) {
    cudaError_t e = ensure_attributes<NT, C, R>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid_units * C));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    // Programmatic serialization: the blocks are placed and initialise their
    // shared memory while the previous kernel (the plan) finishes; the kernel
    // waits for it before its first global access.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (C > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = C;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, select_kernel<NT, C, R>, p);
}

template <int NT, int C>
cudaError_t occupancy_t(size_t smem, int* units) {
    auto kern = select_kernel<NT, C>;
    cudaError_t e = ensure_attributes<NT, C>();
    if (e != cudaSuccess) return e;
    if (C == 1) {
        int per_sm = 0, dev = 0, sms = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
        if (e != cudaSuccess) return e;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        *units = per_sm * sms;
        return cudaSuccess;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C * 64);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    *units = clusters;
    return cudaSuccess;
}

template <typename... Args>
cudaError_t launch_plain(void (*kern)(Args...), dim3 grid, dim3 block, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The same with programmatic stream serialization: the kernel may start
// before the previous grid in the stream completes, and must wait for it
// (griddepcontrol.wait) before its first global access.
template <typename... Args>
cudaError_t launch_dependent(void (*kern)(Args...), dim3 grid, dim3 block, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int C>
cudaError_t launch_select_c(const SelectParams& p, int threads, int grid_units, size_t smem, cudaStream_t stream) {
    return threads == 512 ? launch_select_t<512, C>(p, grid_units, smem, stream)
                          : launch_select_t<256, C>(p, grid_units, smem, stream);
}
template <int C>
cudaError_t occupancy_c(int threads, size_t smem, int* units_out) {
    return threads == 512 ? occupancy_t<512, C>(smem, units_out) : occupancy_t<256, C>(smem, units_out);
}

}  // namespace

cudaError_t launch_select(const SelectParams& p, int cluster, int threads, int grid_units, size_t smem,
                          cudaStream_t stream) {
    if (cluster == 1 && threads == 256 && p.gate_refresh > 0)
        return launch_select_t<256, 1, true>(p, grid_units, smem, stream);
    switch (cluster) {
        case 1: return launch_select_c<1>(p, threads, grid_units, smem, stream);
        case 2: return launch_select_c<2>(p, threads, grid_units, smem, stream);
        case 3: return launch_select_c<3>(p, threads, grid_units, smem, stream);
        case 4: return launch_select_c<4>(p, threads, grid_units, smem, stream);
        case 8: return launch_select_c<8>(p, threads, grid_units, smem, stream);
        case 16: return launch_select_c<16>(p, threads, grid_units, smem, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t select_occupancy(int cluster, int threads, size_t smem, int* units_out) {
    switch (cluster) {
        case 1: return occupancy_c<1>(threads, smem, units_out);
        case 2: return occupancy_c<2>(threads, smem, units_out);
        case 3: return occupancy_c<3>(threads, smem, units_out);
        case 4: return occupancy_c<4>(threads, smem, units_out);
        case 8: return occupancy_c<8>(threads, smem, units_out);
        case 16: return occupancy_c<16>(threads, smem, units_out);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_plan(const int32_t* seq_lens, int32_t batch, int32_t max_seq_len, int32_t long_threshold,
                        void* workspace, cudaStream_t stream) {
    if (batch <= 256 * kPlanPerThread)
        return launch_plain(plan_kernel<256>, dim3(1), dim3(256), stream, seq_lens, batch, max_seq_len,
                            long_threshold, workspace);
    if (batch <= 512 * kPlanPerThread)
        return launch_plain(plan_kernel<512>, dim3(1), dim3(512), stream, seq_lens, batch, max_seq_len,
                            long_threshold, workspace);
    return launch_plain(plan_kernel<1024>, dim3(1), dim3(1024), stream, seq_lens, batch, max_seq_len, long_threshold,
                        workspace);
}

cudaError_t launch_page_transform(const int32_t* raw, int32_t batch, int32_t k, const int32_t* page_table,
                                  int64_t pt_stride, int32_t log2_page, int32_t* out, cudaStream_t stream) {
    const int64_t n = static_cast<int64_t>(batch) * k;
    const int blocks = static_cast<int>(min_i64((n + 255) / 256, 152 * 8));
    return launch_dependent(page_transform_kernel, dim3(blocks), dim3(256), stream, raw, batch, k, page_table,
                            pt_stride, log2_page, out);
}

cudaError_t launch_key_map(const float* x, int64_t n, uint32_t* keys, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const int blocks = static_cast<int>(min_i64((n + 255) / 256, 152 * 16));
    return launch_plain(key_map_kernel, dim3(blocks), dim3(256), stream, x, n, keys);
}

}  // namespace topkidx
