// topk_stream.cu -- the warp-specialised single-block select kernel.
//
// It computes what select_kernel<NT, 1> computes (SGLang PR #26788 "[JIT
// Kernel] DeepSeek-V4 DSA indexer: faster top-k + page-table transform
// (runtime k <= 2048)": per-row top-k over order-preserving keys, fused with
// the page-table transform; ties at the k-th key go to the smaller position),
// one block per row, but it splits the block's warps by role so that the
// row's stream from HBM never waits for the row's fixed steps:
//
//  * 8 streaming warps run pass 1 only: every row's tiles come through the
//    bulk-copy ring; each element is tested against the row's gate, and the
//    ones that pass are keyed, counted in the row's 2048-bin histogram and
//    kept (32-bit key, 16-bit position: rows of up to 65536) in the row's
//    candidate buffer.
//  * 4 resolving warps do the rest, one row behind: the histogram scan, the
//    refinement rounds over the candidate buffer, the finish of the last <= 32
//    candidates, the page-table gather and the output; then the sampled gate
//    of the row two slots ahead, in the histogram they just freed.
//
// Two (histogram, candidate buffer) sets alternate between rows, so the
// streaming warps fill one while the resolving warps drain the other.  Two
// mbarrier pairs hand a set over: `done[b]` (8 streaming warps arrive: pass 1
// of the set's row is complete) and `ready[b]` (one resolving thread arrives:
// the gate of the set's next row is published and the set is clear).  For
// row slot q (the q-th row of the block that needs a select) the set is
// q & 1 and the phase q >> 1; neither barrier can run a phase ahead of its
// waiter, because each side needs the other's previous hand-over first.
//
// The algorithm of every step is the one of select_kernel (topk_kernels.cu);
// the resolving warps use a single histogram per set (a barrier more per
// refinement round).  Rows that overflow the candidate buffer, or whose gate
// was tighter than the k-th key, are resolved by re-reading the row with
// plain loads in the resolving warps (the two-pass streaming path).

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

namespace {

constexpr int kST = 32 * kStreamWarps;  // streaming threads

#define SCTL(base, field) ((base) + static_cast<uint32_t>(offsetof(SetControl, field)))

}  // namespace

// RW resolving warps: 4 (two blocks per SM, a two-stage ring) or 8 (one
// block per SM, a deeper ring).
template <int RW>
__global__ void __launch_bounds__(32 * (kStreamWarps + RW), RW == 4 ? 2 : 1) stream_select_kernel(const SelectParams p) {
    constexpr int kRT = 32 * RW;                      // resolving threads
    constexpr int kThreads = kST + kRT;
    constexpr int kRSamples = kMaxSamples / kRT;      // gate samples per resolving thread
    static_assert(kRSamples % 4 == 0, "gate samples are loaded as float4s");
    using RSync = GroupSync<1, kRT>;                  // barrier of the resolving warps only
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const StreamLayout lay = make_stream_layout(p.tile, p.stages, p.cap, p.k);
    const uint32_t sbase = ptx::smem_addr(smem_raw);
    const uint32_t ring = sbase + lay.ring;
    // Per-set regions at a fixed stride (addresses computed, not indexed, so
    // that nothing of the set choice lives in local memory).
    const uint32_t hist0 = sbase + lay.hist[0], hist_stride = lay.hist[1] - lay.hist[0];
    const uint32_t ckey0 = sbase + lay.cand_key[0], cidx0 = sbase + lay.cand_idx[0];
    const uint32_t cand_stride = lay.cand_key[1] - lay.cand_key[0];
    auto hist_of = [&](uint32_t b) { return hist0 + b * hist_stride; };
    auto ckey_of = [&](uint32_t b) { return ckey0 + b * cand_stride; };
    auto cidx_of = [&](uint32_t b) { return cidx0 + b * cand_stride; };
    const uint32_t sctl = sbase + lay.sctl;
    const uint32_t it_row = sbase + lay.items_row, it_len = sbase + lay.items_len;
    const uint32_t it_tiles = sbase + lay.items_tiles, it_tile_start = sbase + lay.items_tile_start;
    const uint32_t claim = sbase + lay.claim;
    uint32_t* claim_ptr = reinterpret_cast<uint32_t*>(smem_raw + lay.claim);
    const uint32_t stages = static_cast<uint32_t>(p.stages);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + lay.mbar);
    uint64_t* empty = full + stages;
    uint64_t* ready = empty + stages;
    uint64_t* done = ready + 2;
    Control* ctl_ptr = reinterpret_cast<Control*>(smem_raw + lay.ctl);
    // The resolving warps' view for the shared helpers (histogram and buffer
    // fields are set per row to the row's set).
    Smem s = {};
    s.emit = sbase + lay.emit;
    s.fin_key = sbase + lay.fin_key;
    s.fin_idx = sbase + lay.fin_idx;
    s.warp_tot = sbase + lay.warp_tot;
    s.ctl = sbase + lay.ctl;
    s.ctl_ptr = ctl_ptr;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool streaming = tid < kST;
    const int rtid = tid - kST;      // resolving-thread index (valid when !streaming)
    const int rwarp = rtid >> 5;

    if (tid == 0) {
        for (uint32_t i = 0; i < stages; ++i) {
            ptx::mbar_init(&full[i], 1);
            ptx::mbar_init(&empty[i], kStreamWarps);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&ready[b], 1);
            ptx::mbar_init(&done[b], kStreamWarps);
        }
        ptx::fence_mbarrier_init();
        ptx::sts_u32(CTL(s, err), 0);
        for (int b = 0; b < 2; ++b) ptx::sts_u32(SCTL(sctl, ncand) + 4u * b, 0);
        for (uint32_t i = 0; i < stages; ++i) ptx::sts_u32(claim + 4u * i, 0xffffffffu);
    }
    clear_hist<kThreads, kBins>(hist_of(0), tid);
    clear_hist<kThreads, kBins>(hist_of(1), tid);
    __syncthreads();
    // Every global access of this kernel comes after this point.
    ptx::grid_dependency_wait();

    const PlanView pv = read_plan(p);
    if (!pv.ok) {
        if (tid == 0 && blockIdx.x == 0) atomicOr(p.flags, TOPK_FLAG_PLAN_MISMATCH);
        return;
    }
    const int32_t n_first = pv.n_first;
    const bool identity = pv.identity;
    const int32_t n_items = pv.n_items;
    const int32_t unit = static_cast<int32_t>(blockIdx.x), nunits = static_cast<int32_t>(gridDim.x);
    const int32_t my_items = snake_count(unit, n_items, nunits);
    if (my_items <= 0) return;

    const uint32_t K = static_cast<uint32_t>(p.k);
    const uint32_t cap = static_cast<uint32_t>(p.cap);
    const uint32_t tile = static_cast<uint32_t>(p.tile);
    const uint32_t vec_per_tile = tile / (4u * kST);
    const uint64_t policy = ptx::l2_policy_evict_first();
    const bool buffering = !p.force_two_pass;
    auto set_err = [&](uint32_t f) { atomicOr(&ctl_ptr->err, f); };
    auto timed_out = [&]() { return (ptx::lds_u32(CTL(s, err)) & TOPK_FLAG_TIMEOUT) != 0u; };
    // Waits of the hand-over barriers: bounded, a time-out is recorded and the
    // caller carries on (the call's output is then void).
    auto handover_wait = [&](uint64_t* bar, uint32_t parity) {
        if (!timed_out() && !ptx::mbar_wait_bounded(bar, parity, p.timeout_ns)) set_err(TOPK_FLAG_TIMEOUT);
    };

    // Streaming-side ring bookkeeping (the same in every streaming thread).
    uint32_t cseq = 0, cst = 0, cround = 0;
    // Row slots handed out so far (both roles count the rows that need a select alike).
    uint32_t qslot = 0;

    for (int32_t w0 = 0; w0 < my_items; w0 += kStreamItemsMax) {
        const int32_t nw = min(kStreamItemsMax, my_items - w0);
        for (int32_t i = tid; i < nw; i += kThreads) {
            const int32_t it = snake_item(unit, w0 + i, nunits);
            const int32_t row = identity ? (it < n_first ? it : it - n_first)
                                         : (it < n_first ? (p.items ? p.items[it] : it) : p.items2[it - n_first]);
            int32_t L = -1;
            uint32_t nt = 0;
            if (row < 0 || row >= p.batch) {
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
                if (L > p.k) nt = ((static_cast<uint32_t>(L) + 3u) / 4u * 4u + tile - 1u) / tile;
            }
            ptx::sts_u32(it_row + 4u * i, static_cast<uint32_t>(row < 0 || row >= p.batch ? 0 : row));
            ptx::sts_u32(it_len + 4u * i, static_cast<uint32_t>(L));
            ptx::sts_u32(it_tiles + 4u * i, nt);
        }
        __syncthreads();
        if (tid == 0) {
            uint32_t run = 0;
            for (int32_t i = 0; i < nw; ++i) {
                ptx::sts_u32(it_tile_start + 4u * i, run);
                run += ptx::lds_u32(it_tiles + 4u * i);
            }
            ptx::sts_u32(CTL(s, win_tiles), run);
        }
        __syncthreads();
        const uint32_t win_base = cseq;
        const uint32_t win_end = win_base + ptx::lds_u32(CTL(s, win_tiles));

        auto tile_src = [&](uint32_t t, uint32_t& bytes) -> const float* {
            const uint32_t qw = t - win_base;
            int32_t lo_i = 0, hi_i = nw - 1;  // largest item whose first tile is <= qw
            while (lo_i < hi_i) {
                const int32_t mid = (lo_i + hi_i + 1) >> 1;
                if (ptx::lds_u32(it_tile_start + 4u * mid) <= qw)
                    lo_i = mid;
                else
                    hi_i = mid - 1;
            }
            const uint32_t tile_in_item = qw - ptx::lds_u32(it_tile_start + 4u * lo_i);
            const uint32_t L = ptx::lds_u32(it_len + 4u * lo_i);
            const uint32_t n4 = (L + 3u) & ~3u;
            const uint32_t off = tile_in_item * tile;
            bytes = min(tile, n4 - off) * 4u;
            return p.scores + static_cast<int64_t>(ptx::lds_u32(it_row + 4u * lo_i)) * p.row_stride + off;
        };
        auto issue_tile = [&](uint32_t t, uint32_t st) {
            uint32_t bytes;
            const float* src = tile_src(t, bytes);
            ptx::mbar_arrive_expect_tx(&full[st], bytes);
            ptx::bulk_copy_g2s_addr(ring + st * tile * 4u, src, bytes, &full[st], policy);
        };
        if (tid == 0 && !timed_out()) {
            for (uint32_t t = win_base; t < win_end && t < win_base + stages; ++t) {
                ptx::sts_u32(claim + 4u * (t % stages), t / stages);
                issue_tile(t, t % stages);
            }
        }

        if (streaming) {
            // ================================================ streaming warps
            // The warp whose release completes a stage's empty phase refills it
            // (one claim per stage and round), unless the block gave up a wait.
            auto refill_after = [&](uint32_t t, uint32_t st, uint32_t r) {
                const uint32_t next = t + stages;
                if (next >= win_end) return;
                if (!ptx::mbar_test_wait(&empty[st], r & 1u)) return;
                if (timed_out()) return;
                if (atomicCAS(&claim_ptr[st], r, r + 1u) != r) return;
                issue_tile(next, st);
            };
            for (int32_t j = 0; j < nw; ++j) {
                const uint32_t ntiles = ptx::lds_u32(it_tiles + 4u * j);
                if (ntiles == 0u) continue;
                const uint32_t b = qslot & 1u;
                handover_wait(&ready[b], (qslot >> 1) & 1u);
                const uint32_t L = ptx::lds_u32(it_len + 4u * j);
                const uint32_t lo = ptx::lds_u32(SCTL(sctl, lo) + 4u * b);
                const int shift = static_cast<int>(ptx::lds_u32(SCTL(sctl, shift) + 4u * b));
                const float f_lo = key_float(lo);
                const uint32_t hs = hist_of(b), ck = ckey_of(b), ci = cidx_of(b);
                const uint32_t ncand_addr = SCTL(sctl, ncand) + 4u * b;
                {
                    // The row's page-table lines into L2 for the resolving warps'
                    // gather (skipped when the row spans far more pages than results).
                    const int32_t* pt_row =
                        p.page_table + static_cast<int64_t>(ptx::lds_u32(it_row + 4u * j)) * p.pt_stride;
                    const uint32_t npg = ((L - 1u) >> p.log2_page) + 1u;
                    if (npg <= 8u * K)
                        for (uint32_t e = 32u * tid; e < npg + 31u; e += 32u * kST)
                            ptx::prefetch_l2(pt_row + min(e, npg - 1u));
                }
                auto pass1 = [&](auto v_tag) {
                    constexpr int V = decltype(v_tag)::value;
                    for (uint32_t t = 0; t < ntiles; ++t) {
                        const uint32_t st = cst;
                        if (!timed_out() && !ptx::mbar_wait_bounded(&full[st], cround & 1u, p.timeout_ns))
                            set_err(TOPK_FLAG_TIMEOUT);
                        const uint32_t base_idx = t * tile;
                        const uint32_t ring_st = ring + st * tile * 4u;
                        const uint32_t lim = min(L - base_idx, tile);
                        uint32_t gmask = 0;
                        {
                            float4 x[V];
#pragma unroll
                            for (int q = 0; q < V; ++q) x[q] = ptx::lds_f4(ring_st + 16u * (q * kST + tid));
#pragma unroll
                            for (int q = 0; q < V; ++q)
                                gmask |= ((x[q].x < f_lo ? 0u : 1u) | (x[q].y < f_lo ? 0u : 2u) |
                                          (x[q].z < f_lo ? 0u : 4u) | (x[q].w < f_lo ? 0u : 8u))
                                         << (4 * q);
                        }
                        if (lim != tile) {
#pragma unroll
                            for (int q = 0; q < V; ++q) {
                                const uint32_t e0 = 4u * (q * kST + tid);
                                const uint32_t valid =
                                    e0 + 4u <= lim ? 15u : (e0 >= lim ? 0u : (1u << (lim - e0)) - 1u);
                                gmask &= ~((15u & ~valid) << (4 * q));
                            }
                        }
                        const uint32_t cnt = __popc(gmask);
                        const WarpPrefix wp = warp_prefix_small(cnt, lane);
                        uint32_t wbase = 0;
                        if (buffering && lane == 0 && wp.total != 0u) wbase = ptx::atom_add_s(ncand_addr, wp.total);
                        wbase = __shfl_sync(kFull, wbase, 0);
                        if (buffering && wbase + wp.total <= cap) {
                            uint32_t slot = wbase + wp.excl;
                            while (gmask) {
                                const int e = __ffs(gmask) - 1;
                                gmask &= gmask - 1u;
                                const uint32_t idx_in_tile =
                                    4u * (static_cast<uint32_t>(e >> 2) * kST + tid) + (e & 3);
                                const uint32_t key =
                                    score_key(__uint_as_float(ptx::lds_u32(ring_st + 4u * idx_in_tile)));
                                const bool pass = key >= lo;
                                if (pass)
                                    ptx::red_add_s(
                                        hs + 4u * min((key - lo) >> shift, static_cast<uint32_t>(kBins - 1)), 1u);
                                ptx::sts_u32(ck + 4u * slot, pass ? key : 0u);
                                ptx::sts_u16(ci + 2u * slot, base_idx + idx_in_tile);
                                ++slot;
                            }
                        } else {
                            // Buffer full (or not used): count only; runs of one bin take one atomic.
                            uint32_t run_bin = 0u, run_n = 0u;
                            auto count = [&](bool gated, float v) {
                                const uint32_t key = score_key(v);
                                if (gated && key >= lo) {
                                    const uint32_t bin = min((key - lo) >> shift, static_cast<uint32_t>(kBins - 1));
                                    if (bin != run_bin && run_n) {
                                        ptx::red_add_s(hs + 4u * run_bin, run_n);
                                        run_n = 0u;
                                    }
                                    run_bin = bin;
                                    ++run_n;
                                }
                            };
#pragma unroll
                            for (int q = 0; q < V; ++q) {
                                if ((gmask >> (4 * q)) & 15u) {
                                    const float4 y = ptx::lds_f4(ring_st + 16u * (q * kST + tid));
                                    count((gmask >> (4 * q)) & 1u, y.x);
                                    count((gmask >> (4 * q + 1)) & 1u, y.y);
                                    count((gmask >> (4 * q + 2)) & 1u, y.z);
                                    count((gmask >> (4 * q + 3)) & 1u, y.w);
                                }
                            }
                            if (run_n) ptx::red_add_s(hs + 4u * run_bin, run_n);
                        }
                        __syncwarp();
                        if (lane == 0) {
                            ptx::mbar_arrive(&empty[st]);
                            refill_after(cseq, st, cround);
                        }
                        ++cseq;
                        if (++cst == stages) {
                            cst = 0;
                            ++cround;
                        }
                    }
                };
                if (vec_per_tile == 8u)
                    pass1(std::integral_constant<int, 8>{});
                else if (vec_per_tile == 7u)
                    pass1(std::integral_constant<int, 7>{});
                else if (vec_per_tile == 6u)
                    pass1(std::integral_constant<int, 6>{});
                else if (vec_per_tile == 4u)
                    pass1(std::integral_constant<int, 4>{});
                else
                    pass1(std::integral_constant<int, 2>{});
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&done[b]);
                ++qslot;
            }
        } else {
            // ================================================ resolving warps
            const RSync rsync;
            // The gate of item j, computed into set b's histogram (clear on
            // entry and on exit) and published with set b: after SGLang PR
            // #32094 "[DSA] Add LiteTopk fused indexer top-k prefill path for
            // SM100" ("Summary": a recall-safe gate) applied to precomputed
            // scores, with the bins spread over [gate, sample max] as in the
            // DistRadixTopK README's "linear mapping".
            auto samples_for = [&](uint32_t L) -> uint32_t {
                const uint32_t m = L <= 16384u ? min(static_cast<uint32_t>(p.samples), 1024u)
                                               : static_cast<uint32_t>(p.samples);
                return min(m, L);
            };
            auto publish_gate = [&](int32_t j, uint32_t b) {
                const uint32_t hs = hist_of(b);
                const uint32_t L = ptx::lds_u32(it_len + 4u * j);
                const uint32_t Kp = min(K, L);
                const uint32_t M = samples_for(L);
                uint32_t lo = 0;
                int shift = 32 - kBinBits;
                const float E = static_cast<float>(M) * static_cast<float>(Kp) / static_cast<float>(L);
                const float r_safe = ceilf(E + 4.0f * sqrtf(E) + 4.0f);
                const float r_fill =
                    floorf(p.gate_fill * static_cast<float>(cap) * static_cast<float>(M) / static_cast<float>(L));
                const float r_f = fmaxf(r_safe, r_fill);
                if (!p.disable_gate && r_f < static_cast<float>(M)) {
                    const uint32_t r = static_cast<uint32_t>(r_f);
                    const float* rowp =
                        p.scores + static_cast<int64_t>(ptx::lds_u32(it_row + 4u * j)) * p.row_stride;
                    // The samples come in 32-float segments: a thread loads float4
                    // f = q * 128 + rtid, part f & 7 of segment f >> 3 (16-byte
                    // loads, all issued before any is used).
                    uint32_t keys[kRSamples];
                    uint32_t valid = 0;  // bit 4q + c: keys[4q + c] is a sample
                    uint32_t kmax = 0;
                    if (rtid == 0) ptx::sts_u32(CTL(s, smax), 0);
                    {
                        float4 sv[kRSamples / 4];
#pragma unroll
                        for (int q = 0; q < kRSamples / 4; ++q) {
                            const uint32_t f = static_cast<uint32_t>(q * kRT + rtid);
                            const uint32_t i0 = (f >> 3) * 32u + (f & 7u) * 4u;  // first sample of the float4
                            sv[q] = i0 < M ? __ldg(reinterpret_cast<const float4*>(
                                                 rowp + sample_pos((f >> 3) * 32u, L, M) + (f & 7u) * 4u))
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                            const uint32_t vq = i0 + 4u <= M ? 15u : (i0 >= M ? 0u : (1u << (M - i0)) - 1u);
                            valid |= vq << (4 * q);
                        }
#pragma unroll
                        for (int q = 0; q < kRSamples / 4; ++q) {
                            keys[4 * q] = score_key(sv[q].x);
                            keys[4 * q + 1] = score_key(sv[q].y);
                            keys[4 * q + 2] = score_key(sv[q].z);
                            keys[4 * q + 3] = score_key(sv[q].w);
                        }
                    }
                    rsync();
#pragma unroll
                    for (int q = 0; q < kRSamples; ++q) {
                        if ((valid >> q) & 1u) {
                            ptx::red_add_s(hs + 4u * (keys[q] >> (32 - kBinBits)), 1u);
                            kmax = max(kmax, keys[q]);
                        }
                    }
                    kmax = __reduce_max_sync(kFull, kmax);
                    if (lane == 0) atomicMax(&ctl_ptr->smax, kmax);
                    rsync();
                    const ScanResult g = scan_find<kRT>(s, hs, r, rtid, 0, rsync);
                    lo = g.bin << (32 - kBinBits);
                    if (g.above + g.count > r + r / 4u + 4u && g.count > 1u) {
                        // Refine inside the coarse bin on the next 11 bits.
                        clear_hist<kRT, kBins>(hs, rtid);
                        rsync();
#pragma unroll
                        for (int q = 0; q < kRSamples; ++q) {
                            if (((valid >> q) & 1u) && (keys[q] >> (32 - kBinBits)) == g.bin)
                                ptx::red_add_s(hs + 4u * ((keys[q] >> (32 - 2 * kBinBits)) & (kBins - 1)), 1u);
                        }
                        rsync();
                        const ScanResult g2 = scan_find<kRT>(s, hs, r - g.above, rtid, 0, rsync);
                        lo |= g2.bin << (32 - 2 * kBinBits);
                    }
                    const uint32_t smax = ptx::lds_u32(CTL(s, smax));
                    const int bl = bit_length(smax - lo);
                    shift = bl > kBinBits - 1 ? bl - (kBinBits - 1) : 0;
                    clear_hist<kRT, kBins>(hs, rtid);
                }
                if (rtid == 0) {
                    ptx::sts_u32(SCTL(sctl, lo) + 4u * b, lo);
                    ptx::sts_u32(SCTL(sctl, shift) + 4u * b, static_cast<uint32_t>(shift));
                    ptx::sts_u32(SCTL(sctl, ncand) + 4u * b, 0u);
                }
                rsync();
                if (rtid == 0) ptx::mbar_arrive(&ready[b]);
            };
            // The item of the n-th row slot after item j (-1: none in this window).
            auto nth_select_item = [&](int32_t j, int n) -> int32_t {
                for (int32_t i = j + 1; i < nw; ++i)
                    if (ptx::lds_u32(it_tiles + 4u * i) != 0u && --n == 0) return i;
                return -1;
            };

            // The first two rows of the window get their gates now.
            {
                const int32_t j0 = nth_select_item(-1, 1);
                const int32_t j1 = j0 >= 0 ? nth_select_item(j0, 1) : -1;
                if (j0 >= 0) publish_gate(j0, qslot & 1u);
                if (j1 >= 0) publish_gate(j1, (qslot + 1u) & 1u);
            }
            for (int32_t j = 0; j < nw; ++j) {
                const int32_t row = static_cast<int32_t>(ptx::lds_u32(it_row + 4u * j));
                const int32_t Ls = static_cast<int32_t>(ptx::lds_u32(it_len + 4u * j));
                if (Ls < 0) continue;  // rejected item: nothing to write
                const uint32_t L = static_cast<uint32_t>(Ls);
                const uint32_t Kp = min(K, L);
                int32_t* out_row = p.out + static_cast<int64_t>(row) * p.k;
                int32_t* raw_row = p.raw_out ? p.raw_out + static_cast<int64_t>(row) * p.k : nullptr;
                const int32_t* pt_row = p.page_table + static_cast<int64_t>(row) * p.pt_stride;
                if (ptx::lds_u32(it_tiles + 4u * j) == 0u) {
                    // Every position is selected (seq_len <= k): no select at all.
                    write_results<kRT>(out_row, raw_row, pt_row, p.log2_page, K, 0u, rtid, [&](uint32_t q) {
                        return q < L ? static_cast<int32_t>(q) : -1;
                    });
                    continue;
                }
                const uint32_t b = qslot & 1u;
                const int32_t j_next = nth_select_item(j, 2);  // the row whose gate set b takes next
                if (rtid == 0) {
                    ptx::sts_u32(CTL(s, nemit), 0);
                    ptx::sts_u32(CTL(s, nfin), 0);
                }
                handover_wait(&done[b], (qslot >> 1) & 1u);
                // Every decision of the resolving warps must be the same in all
                // of them (they meet at group barriers): the candidate count is
                // read once and shared.  (After a hand-over wait gave up, the
                // streaming warps may still be adding to it.)
                if (rtid == 0) ptx::sts_u32(SCTL(sctl, ncand_seen), ptx::lds_u32(SCTL(sctl, ncand) + 4u * b));
                rsync();

                // -------------------------------------------------- resolve
                const uint32_t hs = hist_of(b), ck = ckey_of(b), ci = cidx_of(b);
                const uint32_t ncand_addr = SCTL(sctl, ncand) + 4u * b;
                const uint32_t lo = ptx::lds_u32(SCTL(sctl, lo) + 4u * b);
                const int shift = static_cast<int>(ptx::lds_u32(SCTL(sctl, shift) + 4u * b));
                const bool overflow = !buffering || ptx::lds_u32(SCTL(sctl, ncand_seen)) > cap;
                const float* row_ptr = p.scores + static_cast<int64_t>(row) * p.row_stride;
                const float4* row4 = reinterpret_cast<const float4*>(row_ptr);
                const uint32_t nvec = (L + 3u) >> 2;
                s.hist_a = hs;
                s.cand_key = ck;
                s.cand_idx = ci;

                ScanResult sr = scan_find<kRT>(s, hs, Kp, rtid, 0, rsync);
                uint32_t r_lo, r_hi, G, cnt;
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
                    const uint64_t bb = sr.bin;
                    r_lo = static_cast<uint32_t>(lo + (bb << shift));
                    r_hi = (sr.bin == kBins - 1)
                               ? 0xffffffffu
                               : static_cast<uint32_t>(min_u64(0xffffffffull, lo + ((bb + 1) << shift) - 1));
                    cnt = sr.count;
                    stream_mode = overflow;
                }
                clear_hist<kRT, kBins>(hs, rtid);
                rsync();

                // The set's candidate count, the same in every resolving thread
                // (loops that hold warp-wide ballots and shuffles take it as
                // their bound; capped at the buffer).  Every resolving thread
                // must call it.
                auto group_count = [&]() -> uint32_t {
                    rsync();
                    if (rtid == 0) ptx::sts_u32(SCTL(sctl, ncand_seen), min(ptx::lds_u32(ncand_addr), cap));
                    rsync();
                    return ptx::lds_u32(SCTL(sctl, ncand_seen));
                };
                auto emit_warp = [&](bool flag, uint32_t idx) {
                    const uint32_t slot = warp_reserve(CTL(s, nemit), flag, lane);
                    if (flag) {
                        if (slot < K)
                            ptx::sts_u32(s.emit + 4u * slot, idx);
                        else
                            set_err(TOPK_FLAG_INTERNAL);
                    }
                };
                auto emit_from_buffer = [&](uint32_t nc, auto take) {
                    for (uint32_t i0 = 0; i0 < nc; i0 += 4u * kRT) {
                        uint32_t pos[4];
                        uint32_t m = 0;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t i = i0 + q * kRT + rtid;
                            const bool in = i < nc;
                            const uint32_t key = in ? ptx::lds_u32(ck + 4u * i) : 0u;
                            pos[q] = in ? ptx::lds_u16(ci + 2u * i) : 0u;
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
                        // Collect pass: emit everything above the range, keep the range.
                        if (rtid == 0) ptx::sts_u32(ncand_addr, 0);
                        rsync();
                        for (uint32_t v0 = rwarp * 32u; v0 < nvec; v0 += 4u * kRT) {
                            float4 xv[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const uint32_t v = v0 + u * kRT + lane;
                                xv[u] = v < nvec ? __ldg(row4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const uint32_t v = v0 + u * kRT + lane;
                                const bool in = v < nvec;
                                const float xs[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    const uint32_t idx = 4u * v + c;
                                    const uint32_t key = score_key(xs[c]);
                                    const bool live = in && idx < L;
                                    emit_warp(live && key > r_hi, idx);
                                    const bool keep = live && key >= r_lo && key <= r_hi;
                                    const uint32_t slot = warp_reserve(ncand_addr, keep, lane);
                                    if (keep) {
                                        if (slot < cap) {
                                            ptx::sts_u32(ck + 4u * slot, key);
                                            ptx::sts_u16(ci + 2u * slot, idx);
                                        } else {
                                            set_err(TOPK_FLAG_INTERNAL);
                                        }
                                    }
                                }
                            }
                        }
                        rsync();
                        stream_mode = false;
                        continue;
                    }
                    // One more 11-bit round over [r_lo, r_hi].
                    const int sh = shift_for_span(r_hi - r_lo);
                    if (!stream_mode) {
                        const uint32_t nc = group_count();
                        for (uint32_t i = rtid; i < nc; i += kRT) {
                            const uint32_t key = ptx::lds_u32(ck + 4u * i);
                            if (key >= r_lo && key <= r_hi) ptx::red_add_s(hs + 4u * ((key - r_lo) >> sh), 1u);
                        }
                    } else {
                        for (uint32_t v0 = rtid; v0 < nvec; v0 += 4u * kRT) {
                            float4 xv[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const uint32_t v = v0 + u * kRT;
                                xv[u] = v < nvec ? __ldg(row4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                            uint32_t run_bin = 0u, run_n = 0u;
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const uint32_t v = v0 + u * kRT;
                                const float xs[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    const uint32_t idx = 4u * v + c;
                                    const uint32_t key = score_key(xs[c]);
                                    if (v < nvec && idx < L && key >= r_lo && key <= r_hi) {
                                        const uint32_t bin = (key - r_lo) >> sh;
                                        if (bin != run_bin && run_n) {
                                            ptx::red_add_s(hs + 4u * run_bin, run_n);
                                            run_n = 0u;
                                        }
                                        run_bin = bin;
                                        ++run_n;
                                    }
                                }
                            }
                            if (run_n) ptx::red_add_s(hs + 4u * run_bin, run_n);
                        }
                    }
                    rsync();
                    sr = scan_find<kRT>(s, hs, Kp - G, rtid, 0, rsync);
                    if (sr.bin >= static_cast<uint32_t>(kBins)) {  // cannot happen: the range holds >= need
                        set_err(TOPK_FLAG_INTERNAL);
                        clear_hist<kRT, kBins>(hs, rtid);
                        rsync();
                        break;
                    }
                    G += sr.above;
                    const uint64_t bb = sr.bin;
                    const uint32_t nlo = static_cast<uint32_t>(r_lo + (bb << sh));
                    const uint32_t nhi = static_cast<uint32_t>(min_u64(r_hi, r_lo + ((bb + 1) << sh) - 1));
                    r_lo = nlo;
                    r_hi = nhi;
                    cnt = sr.count;
                    clear_hist<kRT, kBins>(hs, rtid);
                    rsync();
                }
                rsync();

                const uint32_t need = Kp - G;
                if (r_lo == r_hi) {
                    // ---- a single threshold key T; `need` of its `cnt` copies are taken
                    const uint32_t T = r_lo;
                    const uint32_t quota = need;
                    const bool all_eq = (quota == cnt);
                    if (!stream_mode) {
                        const uint32_t nc = group_count();
                        emit_from_buffer(nc, [&](uint32_t key) { return key > T || (all_eq && key == T); });
                        if (!all_eq && quota > 0) {
                            // The `quota` smallest positions among the copies of T:
                            // rounds on v = ~position (larger v = smaller position).
                            uint32_t v_lo = ~(L - 1u), v_hi = ~0u, v_g = 0, v_cnt = cnt;
                            for (int vr = 0; vr < 6; ++vr) {
                                if (v_lo == v_hi || v_cnt <= static_cast<uint32_t>(kFinish)) break;
                                const int sh = shift_for_span(v_hi - v_lo);
                                for (uint32_t i = rtid; i < nc; i += kRT) {
                                    const uint32_t v = ~ptx::lds_u16(ci + 2u * i);
                                    if (ptx::lds_u32(ck + 4u * i) == T && v >= v_lo && v <= v_hi)
                                        ptx::red_add_s(hs + 4u * ((v - v_lo) >> sh), 1u);
                                }
                                rsync();
                                const ScanResult vs = scan_find<kRT>(s, hs, quota - v_g, rtid, 0, rsync);
                                v_g += vs.above;
                                const uint64_t bb = vs.bin;
                                const uint32_t nlo = static_cast<uint32_t>(v_lo + (bb << sh));
                                const uint32_t nhi = static_cast<uint32_t>(min_u64(v_hi, v_lo + ((bb + 1) << sh) - 1));
                                v_lo = nlo;
                                v_hi = nhi;
                                v_cnt = vs.count;
                                clear_hist<kRT, kBins>(hs, rtid);
                                rsync();
                            }
                            if (rtid == 0) ptx::sts_u32(CTL(s, nfin), 0);
                            rsync();
                            for (uint32_t i0 = rwarp * 32u; i0 < nc; i0 += kRT) {
                                const uint32_t i = i0 + lane;
                                const bool eq = i < nc && ptx::lds_u32(ck + 4u * i) == T;
                                const uint32_t pos = eq ? ptx::lds_u16(ci + 2u * i) : 0u;
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
                            rsync();
                            if (rwarp == 0) {
                                const uint32_t nf = min(ptx::lds_u32(CTL(s, nfin)), static_cast<uint32_t>(kFinish));
                                const uint64_t e =
                                    lane < static_cast<int>(nf)
                                        ? (static_cast<uint64_t>(ptx::lds_u32(s.fin_key + 4u * lane)) << 32) | 1ull
                                        : 0ull;
                                const uint64_t srt = warp_sort_desc(e, lane);
                                const uint32_t take = quota - v_g;
                                emit_warp(static_cast<uint32_t>(lane) < take && srt != 0ull,
                                          ~static_cast<uint32_t>(srt >> 32));
                            }
                        }
                    } else {
                        // Final streaming pass: > T is taken; copies of T up to the
                        // quota, in position order when only some of them are taken.
                        const bool ordered = (!all_eq && quota > 0);
                        const bool none_above = (G == 0u);
                        const uint32_t vend = (none_above && !all_eq && quota == 0u) ? 0u : nvec;
                        uint32_t running = 0;
                        for (uint32_t vb = 0; vb < vend; vb += kRT) {
                            if (none_above && ordered && running >= quota) break;  // group-uniform
                            const uint32_t v = vb + rtid;
                            uint32_t eqm = 0;
                            const bool in = v < nvec;
                            const float4 x = in ? __ldg(row4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                            const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const uint32_t idx = 4u * v + c;
                                const uint32_t key = score_key(xs[c]);
                                const bool live = in && idx < L;
                                emit_warp(live && key > T, idx);
                                if (live && key == T) eqm |= 1u << c;
                            }
                            if (!ordered) {
#pragma unroll
                                for (int c = 0; c < 4; ++c) emit_warp(all_eq && (eqm >> c & 1u), 4u * v + c);
                                continue;
                            }
                            const uint32_t n_eq = __popc(eqm);
                            const uint32_t incl = warp_inclusive_sum(n_eq, lane);
                            if (lane == 31) ptx::sts_u32(s.warp_tot + 4u * rwarp, incl);
                            rsync();
                            uint32_t pre = 0, tot = 0;
                            for (int w = 0; w < RW; ++w) {
                                const uint32_t t = ptx::lds_u32(s.warp_tot + 4u * w);
                                pre += (w < rwarp) ? t : 0u;
                                tot += t;
                            }
                            uint32_t r0 = running + pre + incl - n_eq;
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const bool e = (eqm >> c & 1u) != 0u;
                                emit_warp(e && r0 < quota, 4u * v + c);
                                r0 += e ? 1u : 0u;
                            }
                            running += tot;
                            rsync();
                        }
                    }
                } else {
                    // ---- <= 32 candidates in [r_lo, r_hi]: warp compare-and-swap finish
                    const bool take_range = need >= cnt;
                    const uint32_t nc = group_count();
                    for (uint32_t i0 = 0; i0 < nc; i0 += 4u * kRT) {
                        uint32_t key[4], pos[4];
                        uint32_t m = 0, f = 0;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t i = i0 + q * kRT + rtid;
                            const bool in = i < nc;
                            key[q] = in ? ptx::lds_u32(ck + 4u * i) : 0u;
                            pos[q] = in ? ptx::lds_u16(ci + 2u * i) : 0u;
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
                    if (!take_range) {
                        rsync();
                        if (rwarp == 0) {
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
                }
                rsync();

                // ------------------------------------------- transform + write
                const uint32_t nemit = min(ptx::lds_u32(CTL(s, nemit)), K);
                if (nemit != Kp && rtid == 0) set_err(TOPK_FLAG_INTERNAL);
                write_results<kRT>(out_row, raw_row, pt_row, p.log2_page, K, 0u, rtid, [&](uint32_t q) {
                    return q < nemit ? static_cast<int32_t>(ptx::lds_u32(s.emit + 4u * q)) : -1;
                });
                // Set b is free: it takes the gate of the row two slots ahead.
                if (j_next >= 0) publish_gate(j_next, b);
                ++qslot;
            }
        }
        __syncthreads();
    }

    // Drain: every issued tile was consumed unless a wait gave up; then the
    // last copy of each stage is waited for, with the drain's own limit.
    if (tid == 0 && timed_out()) {
        for (uint32_t st = 0; st < stages; ++st) {
            const uint32_t r = ptx::lds_u32(claim + 4u * st);
            if (r != 0xffffffffu) ptx::mbar_wait_bounded(&full[st], r & 1u, kDrainLimitNs);
        }
    }
    if (tid == 0) {
        const uint32_t err = ptx::lds_u32(CTL(s, err));
        if (err) atomicOr(p.flags, err);
    }
    // Every output store of this block has been issued: dependents may be placed.
    __syncthreads();
    __threadfence();
    ptx::launch_dependents();
}

namespace {

template <int RW>
cudaError_t stream_attributes() {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(stream_select_kernel<RW>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit, std::memory_order_release);
    return cudaSuccess;
}

template <int RW>
cudaError_t launch_stream_t(const SelectParams& p, int grid, size_t smem, cudaStream_t stream) {
    const cudaError_t ea = stream_attributes<RW>();
    if (ea != cudaSuccess) return ea;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(32 * (kStreamWarps + RW));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stream_select_kernel<RW>, p);
}

template <int RW>
cudaError_t stream_occupancy_t(size_t smem, int* units_out) {
    cudaError_t e = stream_attributes<RW>();
    if (e != cudaSuccess) return e;
    int per_sm = 0, dev = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stream_select_kernel<RW>, 32 * (kStreamWarps + RW),
                                                      smem);
    if (e != cudaSuccess) return e;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    *units_out = per_sm * sms;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_stream_select(const SelectParams& p, int resolve_warps, int grid, size_t smem,
                                 cudaStream_t stream) {
    return resolve_warps == 8 ? launch_stream_t<8>(p, grid, smem, stream) : launch_stream_t<4>(p, grid, smem, stream);
}

cudaError_t stream_select_occupancy(int resolve_warps, size_t smem, int* units_out) {
    return resolve_warps == 8 ? stream_occupancy_t<8>(smem, units_out) : stream_occupancy_t<4>(smem, units_out);
}

}  // namespace topkidx
