// topk_warp.cu -- the warp-per-row select kernel for short rows (seq_len up
// to 16384, k up to 512), chosen with the warp_rows tuning knob.
//
// It computes what select_kernel computes (SGLang PR #26788 "[JIT Kernel]
// DeepSeek-V4 DSA indexer: faster top-k + page-table transform (runtime k <=
// 2048)": per-row top-k over order-preserving keys fused with the page-table
// transform; ties at the k-th key go to the smaller position), but one warp
// owns a row from the gate to the output.  No block barrier and no shared
// atomic on a block-wide buffer sits on the path, and a block of 8 warps
// has 8 rows in flight instead of one, so the per-row fixed steps of one row
// overlap the streaming of the others.
//
// Per row:
//  1. Gate: 1024 samples (32-wide contiguous segments at golden-ratio starts)
//     give the r-th largest sample key by an 8-bit-digit radix select in the
//     warp's 256-bin histogram (r from the same sampling bound as the block
//     kernel); lo = the lower edge of that digit's bin.
//  2. Pass 1: the row is read with 16-byte loads, 1024 floats per warp step,
//     the next step's loads in flight while the current one is tested.  The
//     elements that pass the gate are keyed and stored, with their 16-bit
//     positions, in the warp's candidate buffer (a warp prefix of per-lane
//     counts gives the slots; no atomics).
//  3. Resolve: 8-bit radix rounds over the buffer narrow the range that
//     holds the k-th key until it is one key or holds at most 32 entries.
//  4. Output: entries above the range are written straight to out/raw_out
//     through the page table; the last <= 32 are ranked in the warp; copies
//     of a single threshold key are taken in position order through a
//     position bitmap.
//  If the gate passed fewer than k elements or more than the buffer holds,
//  the row is resolved by radix rounds over re-reads of the row instead,
//  with a collect pass once the threshold range fits the buffer.

#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>

#include "keys.cuh"
#include "ptx.cuh"
#include "topk_internal.h"
#include "topkidx.h"

namespace topkidx {
namespace {

constexpr uint32_t kWFull = 0xffffffffu;
constexpr int kWBins = 256;                    // 8-bit digits
constexpr int kWSamples = 1024;                // gate samples per row (32 per lane)
constexpr int kWVec = 8;                       // float4s per lane per step (1024 floats per warp step)
constexpr uint32_t kWStep = 32u * kWVec;       // float4s per warp step

// Per-warp shared memory.
struct WarpSmem {
    uint32_t key[kWarpCap];
    uint16_t pos[kWarpCap];
    uint32_t hist[kWBins];
    uint32_t ties[kWarpMaxLen / 32];  // position bitmap of the copies of a threshold key
    uint16_t sel[kWarpMaxK];          // the selected positions of the current row, by output slot
};
static_assert(sizeof(WarpSmem) % 16 == 0, "per-warp regions stay 16-byte aligned");

__device__ __forceinline__ int wbits(uint32_t x) { return 32 - __clz(x); }

// Shift that maps the key span [0, span] onto at most 256 bins.
__device__ __forceinline__ int wshift(uint32_t span) {
    const int b = wbits(span);
    return b > 8 ? b - 8 : 0;
}

__device__ __forceinline__ uint32_t wsum_incl(uint32_t v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(kWFull, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

__device__ __forceinline__ int32_t wpage(const int32_t* pt_row, int32_t log2_page, int32_t raw) {
    if (raw < 0) return -1;
    const uint32_t page = static_cast<uint32_t>(__ldg(pt_row + (raw >> log2_page)));
    return static_cast<int32_t>((page << log2_page) + (static_cast<uint32_t>(raw) & ((1u << log2_page) - 1u)));
}

// First position of gate sample segment `seg` (32 floats each) of a row of
// length L with M samples: consecutive segments when the row is short (every
// position is a sample), else golden-ratio starts as in the block kernel.
// Always a multiple of 4.
__device__ __forceinline__ uint32_t wsegment(uint32_t seg, uint32_t L, uint32_t M) {
    if (L <= M) return 32u * seg;
    const uint64_t frac = static_cast<uint64_t>(seg * 0x9E3779B9u);
    return static_cast<uint32_t>((frac * static_cast<uint64_t>(L - 31u)) >> 32) & ~3u;
}

struct Pick {
    uint32_t bin, above, count, total;
};

// Finds, in the warp's histogram (bin 255 = largest keys), the bin where the
// count from the top reaches `need`; clears the histogram.  bin = 256 if the
// total is below `need`.  Every lane must call it.
__device__ __forceinline__ Pick wpick(uint32_t* hist, uint32_t need, int lane) {
    const int base = kWBins - 8 * (lane + 1);  // lane 0 owns the top 8 bins
    const uint4 a = *reinterpret_cast<const uint4*>(hist + base);
    const uint4 b = *reinterpret_cast<const uint4*>(hist + base + 4);
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += v[i];
    const uint32_t incl = wsum_incl(sum, lane);
    const uint32_t total = __shfl_sync(kWFull, incl, 31);
    const uint32_t reach = __ballot_sync(kWFull, incl >= need);
    Pick r{256u, 0u, 0u, total};
    uint32_t pb = 0, pa = 0, pc = 0;
    if (reach != 0u && lane == __ffs(reach) - 1) {
        uint32_t acc = incl - sum;
#pragma unroll
        for (int i = 7; i >= 0; --i) {
            if (acc + v[i] >= need && pc == 0u && v[i] != 0u) {
                pb = static_cast<uint32_t>(base + i);
                pa = acc;
                pc = v[i];
            }
            acc += v[i];
        }
    }
    if (reach != 0u) {
        const int src = __ffs(reach) - 1;
        r.bin = __shfl_sync(kWFull, pb, src);
        r.above = __shfl_sync(kWFull, pa, src);
        r.count = __shfl_sync(kWFull, pc, src);
    }
    *reinterpret_cast<uint4*>(hist + base) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(hist + base + 4) = make_uint4(0, 0, 0, 0);
    __syncwarp();
    return r;
}

// Rank of this lane's value among lanes 0..n-1 (values distinct).
__device__ __forceinline__ uint32_t wrank(uint64_t v, uint32_t n) {
    uint32_t r = 0;
    for (uint32_t j = 0; j < n; ++j) r += (__shfl_sync(kWFull, v, static_cast<int>(j)) > v) ? 1u : 0u;
    return r;
}

__global__ void __launch_bounds__(kWarpThreads, 2) warp_select_kernel(const SelectParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    WarpSmem& ws = reinterpret_cast<WarpSmem*>(smem_raw)[warp];
    const uint32_t lt = (1u << lane) - 1u;

    for (int i = lane; i < kWBins; i += 32) ws.hist[i] = 0u;
    for (int i = lane; i < static_cast<int>(kWarpMaxLen / 32); i += 32) ws.ties[i] = 0u;
    __syncwarp();
    // Every global access comes after this point (programmatic launch).
    ptx::grid_dependency_wait();

    const PlanView pv = read_plan(p);
    if (!pv.ok) {
        if (tid == 0 && blockIdx.x == 0) atomicOr(p.flags, TOPK_FLAG_PLAN_MISMATCH);
        return;
    }
    const int32_t n_first = pv.n_first;
    const bool identity = pv.identity;
    const int32_t n_items = pv.n_items;
    const int32_t gw = static_cast<int32_t>(blockIdx.x) * (kWarpThreads / 32) + warp;
    const int32_t nwarps = static_cast<int32_t>(gridDim.x) * (kWarpThreads / 32);
    const uint32_t K = static_cast<uint32_t>(p.k);
    uint32_t err = 0;  // this warp's TOPK_FLAG_* bits (lane 0)

    for (int32_t it = gw; it < n_items; it += nwarps) {
        const int32_t row = identity ? (it < n_first ? it : it - n_first)
                                     : (it < n_first ? (p.items ? p.items[it] : it) : p.items2[it - n_first]);
        if (row < 0 || row >= p.batch) {
            err |= TOPK_FLAG_PLAN_MISMATCH;
            continue;
        }
        int32_t Ls = p.seq_lens[row];
        if (Ls < 0) {
            err |= TOPK_FLAG_SEQ_NEGATIVE;
            Ls = 0;
        } else if (Ls > p.max_seq_len) {
            err |= TOPK_FLAG_SEQ_CLAMPED;
            Ls = p.max_seq_len;
        }
        const uint32_t L = static_cast<uint32_t>(Ls);
        const uint32_t Kp = min(K, L);
        int32_t* out_row = p.out + static_cast<int64_t>(row) * p.k;
        int32_t* raw_row = p.raw_out ? p.raw_out + static_cast<int64_t>(row) * p.k : nullptr;
        const int32_t* pt_row = p.page_table + static_cast<int64_t>(row) * p.pt_stride;
        const float* row_ptr = p.scores + static_cast<int64_t>(row) * p.row_stride;
        const float4* row4 = reinterpret_cast<const float4*>(row_ptr);

        if (L <= K) {  // every position is selected
            for (uint32_t q = lane; q < K; q += 32u) {
                const int32_t r = q < L ? static_cast<int32_t>(q) : -1;
                out_row[q] = wpage(pt_row, p.log2_page, r);
                if (raw_row) raw_row[q] = r;
            }
            continue;
        }
        if (L > kWarpMaxLen) {  // not this kernel's row (the dispatch never sends one)
            err |= TOPK_FLAG_INTERNAL;
            continue;
        }
        {
            // Pull the row's page-table entries into L2 now, so that the output
            // gathers find them there (skipped when the row spans far more
            // pages than it selects).
            const uint32_t npg = ((L - 1u) >> p.log2_page) + 1u;
            if (npg <= 8u * K)
                for (uint32_t e = 32u * static_cast<uint32_t>(lane); e < npg + 31u; e += 32u * 32u)
                    ptx::prefetch_l2(pt_row + min(e, npg - 1u));
        }
        for (uint32_t q = Kp + lane; q < K; q += 32u) {  // slots past Kp
            out_row[q] = -1;
            if (raw_row) raw_row[q] = -1;
        }

        // Selection: every lane calls it; lanes with `take` put `pos` in the
        // next free slots of the selection list (in lane order).  The list is
        // written out, through the page table, once the row is resolved.
        uint32_t ocnt = 0;
        auto emit = [&](bool take, uint32_t pos) {
            const uint32_t m = __ballot_sync(kWFull, take);
            if (take) {
                const uint32_t slot = ocnt + static_cast<uint32_t>(__popc(m & lt));
                if (slot < Kp)
                    ws.sel[slot] = static_cast<uint16_t>(pos);
                else
                    err |= TOPK_FLAG_INTERNAL;
            }
            ocnt += static_cast<uint32_t>(__popc(m));
        };
        const uint32_t nvec = (L + 3u) >> 2;           // float4s covering [0, L)
        const uint32_t nsteps = (nvec + kWStep - 1u) / kWStep;

        // ------------------------------------------------------- 1. gate
        uint32_t lo = 0;
        const uint32_t M = min(static_cast<uint32_t>(kWSamples), L);
        {
            const float E = static_cast<float>(M) * static_cast<float>(Kp) / static_cast<float>(L);
            const float r_safe = ceilf(E + 4.0f * sqrtf(E) + 4.0f);
            const float r_fill = floorf(p.gate_fill * static_cast<float>(kWarpCap) * static_cast<float>(M) /
                                        static_cast<float>(L));
            const float r_f = fmaxf(r_safe, r_fill);
            if (!p.disable_gate && r_f < static_cast<float>(M)) {
                const uint32_t r = static_cast<uint32_t>(r_f);
                // 32 segments of 32 floats; lane l reads float4 (l & 7) of
                // segments 4j + (l >> 3): 8 independent 16-byte loads a lane.
                uint32_t keys[kWSamples / 32];
                uint32_t smask = 0;  // bit 4j + c: keys[4j + c] is a sample
                {
                    float4 sx[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t e0 = wsegment(static_cast<uint32_t>(4 * j + (lane >> 3)), L, M) +
                                            4u * static_cast<uint32_t>(lane & 7);
                        sx[j] = e0 < L ? __ldg(reinterpret_cast<const float4*>(row_ptr + e0))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                        const uint32_t valid = e0 + 4u <= L ? 15u : (e0 >= L ? 0u : (1u << (L - e0)) - 1u);
                        smask |= valid << (4 * j);
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        keys[4 * j] = score_key(sx[j].x);
                        keys[4 * j + 1] = score_key(sx[j].y);
                        keys[4 * j + 2] = score_key(sx[j].z);
                        keys[4 * j + 3] = score_key(sx[j].w);
                    }
                }
                uint32_t prefix = 0, pmask = 0, above = 0;
                for (int d = 0; d < 4; ++d) {
                    const int sh = 24 - 8 * d;
#pragma unroll
                    for (int j = 0; j < kWSamples / 32; ++j)
                        if ((smask >> j & 1u) && (keys[j] & pmask) == prefix)
                            atomicAdd(&ws.hist[(keys[j] >> sh) & 255u], 1u);
                    __syncwarp();
                    const Pick pk = wpick(ws.hist, r - above, lane);
                    if (pk.bin >= static_cast<uint32_t>(kWBins)) break;  // cannot happen: r < M
                    prefix |= pk.bin << sh;
                    pmask |= 255u << sh;
                    above += pk.above;
                    lo = prefix;
                    if (above + pk.count <= r + r / 4u + 4u) break;
                }
            }
        }
        const float f_lo = key_float(lo);

        // ------------------------------------------------------ 2. pass 1
        // Each step tests 32 floats per lane against the gate and appends the
        // ones that pass, as raw bits with their positions, to the warp's
        // buffer (slots from a warp prefix of the lane counts).  Keying is left
        // to one sweep over the compacted buffer afterwards, so the per-element
        // work here is a compare and, for the few that pass, two stores.  Only
        // the last step of a row is masked to the row's end, and the two
        // register buffers alternate, so the next step's loads are always in
        // flight while a step is tested.
        uint32_t wcnt = 0, kmax = 0;
        const bool buffering = !p.force_two_pass;
        if (buffering) {
            float4 xa[kWVec], xb[kWVec];
            auto load = [&](float4* x, uint32_t step) {
#pragma unroll
                for (int q = 0; q < kWVec; ++q) {
                    const uint32_t v = step * kWStep + static_cast<uint32_t>(q * 32 + lane);
                    x[q] = v < nvec ? __ldcs(row4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            };
            auto test = [&](const float4* x, uint32_t step) {
                uint32_t gmask = 0;
#pragma unroll
                for (int q = 0; q < kWVec; ++q)
                    gmask |= ((x[q].x < f_lo ? 0u : 1u) | (x[q].y < f_lo ? 0u : 2u) | (x[q].z < f_lo ? 0u : 4u) |
                              (x[q].w < f_lo ? 0u : 8u))
                             << (4 * q);
                if ((step + 1u) * 4u * kWStep > L) {  // the row ends inside this step
#pragma unroll
                    for (int q = 0; q < kWVec; ++q) {
                        const uint32_t e0 = 4u * (step * kWStep + static_cast<uint32_t>(q * 32 + lane));
                        const uint32_t valid = e0 + 4u <= L ? 15u : (e0 >= L ? 0u : (1u << (L - e0)) - 1u);
                        gmask &= ~((15u & ~valid) << (4 * q));
                    }
                }
                const uint32_t cnt = static_cast<uint32_t>(__popc(gmask));
                const uint32_t incl = wsum_incl(cnt, lane);
                uint32_t slot = wcnt + incl - cnt;
                wcnt += __shfl_sync(kWFull, incl, 31);
                if (__any_sync(kWFull, gmask != 0u)) {
#pragma unroll
                    for (int q = 0; q < kWVec; ++q) {
                        const uint32_t p0 = 4u * (step * kWStep + static_cast<uint32_t>(q * 32 + lane));
                        const float xs[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint32_t t = (gmask >> (4 * q + c)) & 1u;
                            if (t != 0u && slot < kWarpCap) {
                                ws.key[slot] = __float_as_uint(xs[c]);
                                ws.pos[slot] = static_cast<uint16_t>(p0 + c);
                            }
                            slot += t;
                        }
                    }
                }
            };
            load(xa, 0u);
            for (uint32_t step = 0; step < nsteps; step += 2u) {
                if (step + 1u < nsteps) load(xb, step + 1u);
                test(xa, step);
                if (step + 2u < nsteps) load(xa, step + 2u);
                if (step + 1u < nsteps) test(xb, step + 1u);
            }
            __syncwarp();
            {
                // The warp's next row: its gate samples into L2 now (one 128-byte
                // segment per lane), so that its gate does not wait on DRAM behind
                // the stream; the row streams above use evict-first loads, which
                // leave these lines (and the page-table lines) in L2.
                const int32_t itn = it + nwarps;
                if (itn < n_items) {
                    const int32_t rown =
                        identity ? (itn < n_first ? itn : itn - n_first)
                                 : (itn < n_first ? (p.items ? p.items[itn] : itn) : p.items2[itn - n_first]);
                    if (rown >= 0 && rown < p.batch) {
                        const int32_t Ln = min(max(p.seq_lens[rown], 0), p.max_seq_len);
                        const uint32_t Mn = min(static_cast<uint32_t>(kWSamples), static_cast<uint32_t>(Ln));
                        if (Ln > p.k && 32u * static_cast<uint32_t>(lane) < Mn)
                            ptx::prefetch_l2(p.scores + static_cast<int64_t>(rown) * p.row_stride +
                                             wsegment(static_cast<uint32_t>(lane), static_cast<uint32_t>(Ln), Mn));
                    }
                }
            }
            if (wcnt <= kWarpCap) {
                // Key the buffered elements.  An element that passed the float
                // compare but whose key is below the gate can only be a NaN; it
                // gets key 0, which no later step selects.
#pragma unroll 4
                for (uint32_t i = lane; i < wcnt; i += 32u) {
                    const uint32_t key = score_key(__uint_as_float(ws.key[i]));
                    const uint32_t kept = key >= lo ? key : 0u;
                    ws.key[i] = kept;
                    kmax = max(kmax, kept);
                }
                kmax = __reduce_max_sync(kWFull, kmax);
            }
            __syncwarp();
        }

        // ------------------------------------------- 3./4. resolve + output
        uint32_t r_lo = lo, r_hi = kmax, G = 0, cnt = 0;
        bool from_buffer = buffering && wcnt <= kWarpCap;
        // Key-0 entries of a buffer filled by pass 1 under a gate (lo > 0) are
        // fillers for NaNs that passed the float test; in a buffer filled by
        // the collect pass, or with no gate, key 0 is a real key.
        bool fillers = lo != 0u;
        uint32_t nbuf = from_buffer ? wcnt : 0u;
        if (from_buffer) {
            // First round over the buffer: if fewer than Kp keys passed the
            // gate, it was too tight and the row is read again.
            uint32_t total = 0;
            for (int round = 0; round < 6; ++round) {
                if (round > 0 && (r_lo == r_hi || cnt <= 32u)) break;
                const int sh = wshift(r_hi - r_lo);
                for (uint32_t i0 = 0; i0 < nbuf; i0 += 4u * 32u) {
                    uint32_t kk[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t i = i0 + 32u * u + static_cast<uint32_t>(lane);
                        kk[u] = i < nbuf ? ws.key[i] : 0u;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t i = i0 + 32u * u + static_cast<uint32_t>(lane);
                        if (i < nbuf && kk[u] >= r_lo && kk[u] <= r_hi && (kk[u] != 0u || !fillers))
                            atomicAdd(&ws.hist[(kk[u] - r_lo) >> sh], 1u);
                    }
                }
                __syncwarp();
                const Pick pk = wpick(ws.hist, Kp - G, lane);
                if (round == 0) total = pk.total;
                if (pk.bin >= static_cast<uint32_t>(kWBins)) break;
                G += pk.above;
                const uint32_t nlo = r_lo + (pk.bin << sh);
                const uint32_t nhi = static_cast<uint32_t>(
                    min(static_cast<uint64_t>(r_hi), static_cast<uint64_t>(r_lo) + ((static_cast<uint64_t>(pk.bin) + 1u) << sh) - 1u));
                r_lo = nlo;
                r_hi = nhi;
                cnt = pk.count;
            }
            // The row is read again when the buffer's counted keys are fewer
            // than Kp (the gate was tighter than the k-th key), or when the
            // rounds ended with more than 32 entries still in a range of
            // several keys.
            if (total < Kp || (cnt > 32u && r_lo != r_hi)) from_buffer = false;
        }
        if (!from_buffer) {
            // ---- radix rounds over re-reads of the row; a collect pass fills
            // the buffer once the threshold range fits it.
            r_lo = 0u;
            r_hi = 0xffffffffu;
            G = 0u;
            cnt = L;
            for (int round = 0; round < 6 && r_lo != r_hi && cnt > kWarpCap; ++round) {
                const int sh = wshift(r_hi - r_lo);
                for (uint32_t v0 = 0; v0 < nvec; v0 += 32u) {
                    const uint32_t v = v0 + static_cast<uint32_t>(lane);
                    if (v < nvec) {
                        const float4 x = __ldg(row4 + v);
                        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint32_t key = score_key(xs[c]);
                            if (4u * v + c < L && key >= r_lo && key <= r_hi)
                                atomicAdd(&ws.hist[(key - r_lo) >> sh], 1u);
                        }
                    }
                }
                __syncwarp();
                const Pick pk = wpick(ws.hist, Kp - G, lane);
                if (pk.bin >= static_cast<uint32_t>(kWBins)) {  // cannot happen: the range holds >= Kp - G
                    err |= TOPK_FLAG_INTERNAL;
                    break;
                }
                G += pk.above;
                const uint32_t nlo = r_lo + (pk.bin << sh);
                const uint32_t nhi = static_cast<uint32_t>(
                    min(static_cast<uint64_t>(r_hi), static_cast<uint64_t>(r_lo) + ((static_cast<uint64_t>(pk.bin) + 1u) << sh) - 1u));
                r_lo = nlo;
                r_hi = nhi;
                cnt = pk.count;
            }
            if (cnt <= kWarpCap && r_lo != r_hi) {
                // Collect: above the range is taken; the range goes to the buffer.
                nbuf = 0;
                for (uint32_t v0 = 0; v0 < nvec; v0 += 32u) {
                    const uint32_t v = v0 + static_cast<uint32_t>(lane);
                    const float4 x = v < nvec ? __ldg(row4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t idx = 4u * v + c;
                        const uint32_t key = score_key(xs[c]);
                        const bool live = v < nvec && idx < L;
                        emit(live && key > r_hi, idx);
                        const bool keep = live && key >= r_lo && key <= r_hi;
                        const uint32_t m = __ballot_sync(kWFull, keep);
                        if (keep) {
                            const uint32_t s = nbuf + static_cast<uint32_t>(__popc(m & lt));
                            if (s < kWarpCap) {
                                ws.key[s] = key;
                                ws.pos[s] = static_cast<uint16_t>(idx);
                            } else {
                                err |= TOPK_FLAG_INTERNAL;
                            }
                        }
                        nbuf += static_cast<uint32_t>(__popc(m));
                    }
                }
                __syncwarp();
                nbuf = min(nbuf, kWarpCap);
                G = ocnt;  // taken so far
                // Rounds over the buffer until one key or <= 32 entries.
                for (int round = 0; round < 6 && r_lo != r_hi && cnt > 32u; ++round) {
                    const int sh = wshift(r_hi - r_lo);
                    for (uint32_t i0 = 0; i0 < nbuf; i0 += 4u * 32u) {
                        uint32_t kk[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint32_t i = i0 + 32u * u + static_cast<uint32_t>(lane);
                            kk[u] = i < nbuf ? ws.key[i] : 0u;
                        }
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint32_t i = i0 + 32u * u + static_cast<uint32_t>(lane);
                            if (i < nbuf && kk[u] >= r_lo && kk[u] <= r_hi) atomicAdd(&ws.hist[(kk[u] - r_lo) >> sh], 1u);
                        }
                    }
                    __syncwarp();
                    const Pick pk = wpick(ws.hist, Kp - G, lane);
                    if (pk.bin >= static_cast<uint32_t>(kWBins)) {
                        err |= TOPK_FLAG_INTERNAL;
                        break;
                    }
                    G += pk.above;
                    const uint32_t nlo = r_lo + (pk.bin << sh);
                    const uint32_t nhi = static_cast<uint32_t>(min(
                        static_cast<uint64_t>(r_hi), static_cast<uint64_t>(r_lo) + ((static_cast<uint64_t>(pk.bin) + 1u) << sh) - 1u));
                    r_lo = nlo;
                    r_hi = nhi;
                    cnt = pk.count;
                }
                from_buffer = true;
                fillers = false;
                // The buffer holds only the collected range: nothing above it
                // is left to take from it, and G counts what was taken.
            }
        }

        const uint32_t need = Kp - G;
        if (r_lo == r_hi) {
            // ---- a single threshold key T: above T is taken; `need` of its
            // copies, the smallest positions first (a position bitmap).
            const uint32_t T = r_lo;
            if (from_buffer) {
                for (uint32_t i0 = 0; i0 < nbuf; i0 += 4u * 32u) {
                    uint32_t kk[4], pp[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t i = i0 + 32u * u + static_cast<uint32_t>(lane);
                        kk[u] = i < nbuf ? ws.key[i] : 0u;
                        pp[u] = i < nbuf ? ws.pos[i] : 0u;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t i = i0 + 32u * u + static_cast<uint32_t>(lane);
                        emit(i < nbuf && kk[u] > T, pp[u]);
                        if (i < nbuf && kk[u] == T && (kk[u] != 0u || !fillers))
                            atomicOr(&ws.ties[pp[u] >> 5], 1u << (pp[u] & 31u));
                    }
                }
            } else {
                for (uint32_t v0 = 0; v0 < nvec; v0 += 32u) {
                    const uint32_t v = v0 + static_cast<uint32_t>(lane);
                    const float4 x = v < nvec ? __ldg(row4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t idx = 4u * v + c;
                        const uint32_t key = score_key(xs[c]);
                        const bool live = v < nvec && idx < L;
                        emit(live && key > T, idx);
                        if (live && key == T) atomicOr(&ws.ties[idx >> 5], 1u << (idx & 31u));
                    }
                }
            }
            __syncwarp();
            // Lane l owns bitmap words [l * wpl, (l + 1) * wpl).
            const uint32_t words = (L + 31u) >> 5;
            const uint32_t wpl = (words + 31u) >> 5;
            uint32_t mine = 0;
            for (uint32_t w = 0; w < wpl; ++w) {
                const uint32_t wi = static_cast<uint32_t>(lane) * wpl + w;
                if (wi < words) mine += static_cast<uint32_t>(__popc(ws.ties[wi]));
            }
            const uint32_t incl = wsum_incl(mine, lane);
            uint32_t rank = incl - mine;                      // copies before this lane's words
            uint32_t slot = ocnt + min(rank, need);           // their output slots come first
            for (uint32_t w = 0; w < wpl; ++w) {
                const uint32_t wi = static_cast<uint32_t>(lane) * wpl + w;
                if (wi >= words) break;
                uint32_t bits = ws.ties[wi];
                ws.ties[wi] = 0u;
                while (bits) {
                    const uint32_t b = static_cast<uint32_t>(__ffs(bits) - 1);
                    bits &= bits - 1u;
                    if (rank < need) {
                        if (slot < Kp)
                            ws.sel[slot] = static_cast<uint16_t>(wi * 32u + b);
                        else
                            err |= TOPK_FLAG_INTERNAL;
                        ++slot;
                    }
                    ++rank;
                }
            }
            const uint32_t copies = __shfl_sync(kWFull, incl, 31);
            if (copies < need) err |= TOPK_FLAG_INTERNAL;
            ocnt += min(copies, need);
            __syncwarp();
        } else {
            // ---- at most 32 entries in [r_lo, r_hi] (from the buffer): above
            // the range is taken; the range's entries are ranked in the warp.
            uint32_t nf = 0;
            for (uint32_t i0 = 0; i0 < nbuf; i0 += 4u * 32u) {
                // Four chunks' entries are loaded before any is used.
                uint32_t kk[4], pp[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t i = i0 + 32u * u + static_cast<uint32_t>(lane);
                    kk[u] = i < nbuf ? ws.key[i] : 0u;
                    pp[u] = i < nbuf ? ws.pos[i] : 0u;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t i = i0 + 32u * u + static_cast<uint32_t>(lane);
                    const uint32_t key = kk[u], pos = pp[u];
                    const bool live = i < nbuf && (key != 0u || !fillers);
                    emit(live && key > r_hi, pos);
                    const bool in = live && key >= r_lo && key <= r_hi;
                    const uint32_t m = __ballot_sync(kWFull, in);
                    if (in) {
                        const uint32_t s = nf + static_cast<uint32_t>(__popc(m & lt));
                        if (s < 32u) {
                            ws.hist[s] = key;
                            ws.hist[32u + s] = pos;
                        } else {
                            err |= TOPK_FLAG_INTERNAL;
                        }
                    }
                    nf += static_cast<uint32_t>(__popc(m));
                }
            }
            __syncwarp();
            nf = min(nf, 32u);
            const bool mine = static_cast<uint32_t>(lane) < nf;
            const uint32_t fpos = mine ? ws.hist[32 + lane] : 0u;
            const uint64_t e = mine ? (static_cast<uint64_t>(ws.hist[lane]) << 32) | (~fpos & 0xffffffffu) : 0ull;
            const uint32_t rk = wrank(e, nf);  // every lane takes part
            __syncwarp();
            ws.hist[lane] = 0u;
            ws.hist[32 + lane] = 0u;
            __syncwarp();
            emit(mine && rk < need, fpos);
        }
        if (ocnt != Kp) err |= TOPK_FLAG_INTERNAL;
        // Output: 8 slots per lane at a time, their page-table loads issued
        // before any store.
        __syncwarp();
        for (uint32_t q0 = lane; q0 < Kp; q0 += 8u * 32u) {
            int32_t r[8], v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t q = q0 + 32u * u;
                r[u] = q < Kp ? static_cast<int32_t>(ws.sel[q]) : -1;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = wpage(pt_row, p.log2_page, r[u]);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t q = q0 + 32u * u;
                if (q < Kp) {
                    out_row[q] = v[u];
                    if (raw_row) raw_row[q] = r[u];
                }
            }
        }
        __syncwarp();
    }
    err = __reduce_or_sync(kWFull, err);
    if (lane == 0 && err) atomicOr(p.flags, err);
    // Every output store of the block has been issued: a kernel launched after
    // this one with programmatic serialization may be placed now (it still
    // waits for this grid's completion before it reads the output).
    __syncthreads();
    __threadfence();
    ptx::launch_dependents();
}

}  // namespace

// Sets the kernel's shared-memory attribute once per device.
cudaError_t warp_attributes(size_t smem) {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(warp_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    done.fetch_or(bit, std::memory_order_release);
    return cudaSuccess;
}

cudaError_t launch_warp_select(const SelectParams& p, int grid, bool programmatic, cudaStream_t stream) {
    const size_t smem = warp_select_smem_bytes();
    const cudaError_t ea = warp_attributes(smem);
    if (ea != cudaSuccess) return ea;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kWarpThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = programmatic ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, warp_select_kernel, p);
}

cudaError_t warp_select_occupancy(int* units_out) {
    const size_t smem = warp_select_smem_bytes();
    cudaError_t e = warp_attributes(smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0, dev = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, warp_select_kernel, kWarpThreads, smem);
    if (e != cudaSuccess) return e;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    *units_out = per_sm * sms;
    return cudaSuccess;
}

size_t warp_select_smem_bytes() { return sizeof(WarpSmem) * (kWarpThreads / 32); }

}  // namespace topkidx
