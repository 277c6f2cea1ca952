/*
 * topkidx.h -- C ABI of the GB300 (sm_103a) top-k + page-table transform
 * library for sparse-attention indexers.
 *
 * The operation (SGLang PR #26788 "[JIT Kernel] DeepSeek-V4 DSA indexer:
 * faster top-k + page-table transform (runtime k <= 2048)", sections
 * "Motivation" and "Feature"): for each row b of an fp32 score matrix, select
 * the k positions with the largest scores among the first seq_lens[b]
 * entries and emit
 *
 *     out[b][j] = page_table[b][idx / page_size] * page_size + idx % page_size
 *
 * for the selected positions idx, with -1 in the slots past min(k, seq_len).
 * k is a runtime value in [1, 2048]; page_size is a power of two.
 *
 * Conventions for every entry point below:
 *   - Pointers named *_host are host memory; every other pointer is device
 *     memory on the current CUDA device, owned by the caller.  The library
 *     never allocates, frees or retains caller memory.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns without waiting for it, except topk_read_flags.
 *   - A non-OK status means nothing was enqueued (argument errors are found
 *     on the host before any launch), except TOPK_ECUDA, which reports a
 *     failed launch.
 *   - Every kernel is hand-written CUDA for sm_103a; there is no CPU
 *     fallback.  On any other device the calls return TOPK_EDEVICE.
 *   - Ties at the k-th score go to the smaller position, -0.0 equals +0.0,
 *     -inf is an ordinary score; a NaN with the sign bit clear ranks above
 *     +inf and one with the sign bit set below -inf.  The selected set is
 *     therefore unique.  Slot order within a row is unspecified.
 */
#ifndef TOPKIDX_H
#define TOPKIDX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st* topk_stream_t;

typedef enum {
    TOPK_OK = 0,
    TOPK_EINVAL = -1,   /* an argument is out of range or inconsistent      */
    TOPK_EALIGN = -2,   /* a pointer or stride breaks an alignment rule      */
    TOPK_ECUDA = -3,    /* a CUDA runtime call or launch failed              */
    TOPK_ENOSPACE = -4, /* the workspace is smaller than required            */
    TOPK_EDEVICE = -5   /* the current device is not an sm_103 GPU           */
} topk_status_t;

/* Bits of the device-side flag word kept in the workspace (topk_read_flags). */
#define TOPK_FLAG_SEQ_CLAMPED 0x1u   /* a seq_len above max_seq_len was clamped      */
#define TOPK_FLAG_SEQ_NEGATIVE 0x2u  /* a negative seq_len was treated as 0         */
#define TOPK_FLAG_PLAN_MISMATCH 0x4u /* transform batch/max_seq_len differ from plan */
#define TOPK_FLAG_TIMEOUT 0x8u       /* a bounded device wait gave up (output void)  */
#define TOPK_FLAG_INTERNAL 0x10u     /* an internal consistency check failed        */

/*
 * Bytes of device workspace that topk_plan needs for `batch` rows (the plan's
 * work lists, after SGLang PR #26788, commit "Replace the per-element cluster
 * launch ... with a FIXED persistent pool": a compacted list of long items,
 * plus a list of the other rows and a flag word; then the state and the
 * candidate buffers of the opt-in segment-split path for the first 128 rows,
 * 64 KB per row plus 70 KB: about 8.5 MB from 128 rows on).  Returns 0 for
 * batch < 1.
 */
size_t topk_plan_workspace_bytes(int32_t batch);

/*
 * Plan step (PR #26788, commits "Dynamic dispatch via the plan's
 * cluster_threshold" and "Fuse the cluster/non-cluster split for small
 * batch"): reads seq_lens on the device and splits the rows into a list of
 * long rows (seq_len > the long-row threshold, processed by one thread-block
 * cluster per row) and a list of the other rows (one thread block per row),
 * each ordered from longest to shortest.  The plan depends only on seq_lens,
 * batch and max_seq_len, not on k, and can be reused by every
 * topk_transform call with the same seq_lens contents.
 *
 *   seq_lens          device int32[batch]; negative values count as 0,
 *                     values above max_seq_len are clamped (both flagged).
 *   batch             >= 1.
 *   max_seq_len       >= 0, the largest seq_len the caller will pass.
 *   workspace         device memory of at least workspace_bytes >=
 *                     topk_plan_workspace_bytes(batch), 16-byte aligned,
 *                     owned by the caller, valid until the next topk_plan on
 *                     it.  The flag word is reset by this call.
 * Errors: TOPK_EINVAL (batch < 1, max_seq_len < 0, null pointer),
 *         TOPK_ENOSPACE, TOPK_EALIGN, TOPK_EDEVICE, TOPK_ECUDA.
 */
topk_status_t topk_plan(const int32_t* seq_lens, int32_t batch, int32_t max_seq_len, void* workspace,
                        size_t workspace_bytes, topk_stream_t stream);

/*
 * Top-k selection fused with the page-table transform (PR #26788, "Feature":
 * runtime k, ragged per-row seq_lens, power-of-two page size, optional raw
 * index output).  The rows are processed by the kernels the plan assigns:
 * long rows by a cluster of thread blocks that merge their radix histograms
 * through distributed shared memory, the others by one block each (or, when
 * the whole batch fits in two waves of clusters, by the cluster kernel too,
 * after the long rows); both stream the row once from HBM in the common
 * case.
 *
 *   scores            device float[batch][row_stride]; row b is valid in
 *                     [0, seq_lens[b]).  16-byte aligned.  Entries up to the
 *                     next multiple of 4 past seq_len may be read (never
 *                     past the row stride) and do not affect the result.
 *   row_stride        floats between rows; a multiple of 4, >= max_seq_len.
 *   seq_lens          device int32[batch]; the same contents that were
 *                     planned (the kernels read it again; a row whose length
 *                     changed is still computed correctly, only its path
 *                     assignment may be suboptimal).
 *   batch, max_seq_len  the values given to topk_plan for this workspace.
 *   page_table        device int32[batch][page_table_stride]; row b maps
 *                     page p of row b to a page id.  Only the entries of
 *                     selected positions are read; values are used as they
 *                     are (the product is computed modulo 2^32).
 *   page_table_stride int32 entries between page-table rows;
 *                     >= ceil(max_seq_len / page_size).
 *   page_size         power of two, 1 <= page_size <= 2^30.
 *   k                 1 <= k <= 2048.
 *   out_indices       device int32[batch][k] (written in full).
 *   out_raw_indices_or_null  device int32[batch][k] or NULL: the selected
 *                     positions before the transform, slot-aligned with
 *                     out_indices (-1 in the same padded slots).
 *   workspace         the planned workspace; its flag word may be updated.
 * Errors: TOPK_EINVAL, TOPK_EALIGN, TOPK_EDEVICE, TOPK_ECUDA.
 */
topk_status_t topk_transform(const float* scores, int64_t row_stride, const int32_t* seq_lens, int32_t batch,
                             int32_t max_seq_len, const int32_t* page_table, int64_t page_table_stride,
                             int32_t page_size, int32_t k, int32_t* out_indices,
                             int32_t* out_raw_indices_or_null, void* workspace, topk_stream_t stream);

/*
 * Number of kernels one topk_transform call with these arguments enqueues
 * under the current tuning (1 or 2), or a negative topk_status_t
 * (TOPK_EINVAL, TOPK_EDEVICE, TOPK_ECUDA).  Enqueues nothing.
 */
int32_t topk_transform_launches(int32_t batch, int32_t max_seq_len, int32_t k);

/*
 * The gather-and-transform pass on its own (PR #26788, commit "Dynamic
 * dispatch via the plan's cluster_threshold": the page-table transform runs
 * as a separate pass after the raw indices are complete).  For every slot:
 * out[b][j] = raw[b][j] < 0 ? -1 : page_table[b][raw / page_size] *
 * page_size + raw % page_size.  raw values must be < page_table_stride *
 * page_size (not checked).
 *   raw_indices  device int32[batch][k]; out_indices device int32[batch][k]
 *   (may alias raw_indices).  batch >= 1, 1 <= k.
 */
topk_status_t topk_page_transform(const int32_t* raw_indices, int32_t batch, int32_t k,
                                  const int32_t* page_table, int64_t page_table_stride, int32_t page_size,
                                  int32_t* out_indices, topk_stream_t stream);

/*
 * The order-preserving fp32 -> uint32 key map used by every select kernel
 * (DistRadixTopK README "Ultra Low Latency Distributed Radix TopK Indexer Via
 * NoC", second point of "Distributed Radix Sort via NoC": a bin map under
 * which a larger bin implies a larger score).  keys[i] = key(x[i]) with
 * x > y => key(x) > key(y) and x == y => key(x) == key(y) (-0.0 and +0.0 map
 * to one key); NaNs are placed as described above.  n >= 0; x and keys are
 * device arrays of n elements.
 */
topk_status_t topk_key_map(const float* x, int64_t n, uint32_t* keys, topk_stream_t stream);

/*
 * Copies the workspace's TOPK_FLAG_* word to *flags_host after all work
 * enqueued on `stream` so far has finished (this call synchronises the
 * stream).  clear != 0 resets the word afterwards.
 */
topk_status_t topk_read_flags(void* workspace, uint32_t* flags_host, int32_t clear, topk_stream_t stream);

/*
 * Allocation-free variant of topk_plan + topk_transform (the pages have no
 * counterpart; this is a convenience of this library).
 *
 * For callers that cannot allocate device memory -- for example a plugin or
 * an allocator-managed runtime that only hands out its inputs and outputs and
 * must not call cudaMalloc behind its allocator's back -- this call keeps the
 * plan's work lists in a fixed device array owned by the library instead of
 * a caller workspace.  Every GPU that loads the library holds that array
 * (topk_plan_workspace_bytes(TOPK_NOALLOC_MAX_BATCH), about 8.6 MB) until the
 * process exits.  Arguments and outputs are those
 * of topk_transform; the caller still passes scores, seq_lens, the page table
 * and the output buffers.
 *
 *   - batch must be <= TOPK_NOALLOC_MAX_BATCH; larger batches return
 *     TOPK_ENOSPACE and enqueue nothing (use topk_plan + topk_transform with
 *     a caller workspace instead).
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.  The address is kept for the life of the process, so
 *     do not call this entry point again on a device after cudaDeviceReset
 *     on it (the reset unloads the array; use topk_plan + topk_transform).
 *   - Every call on a device shares the one array and leaves its contents in
 *     it.  Calls whose work can overlap on the GPU (two streams, or two host
 *     threads, at once) race on it: serialise them.
 *   - The array's flag word is not exposed; use topk_plan + topk_transform +
 *     topk_read_flags when the clamp/timeout flags are needed.
 *   - No cudaMalloc, cudaFree or other allocating call is made.
 */
#define TOPK_NOALLOC_MAX_BATCH 16384
topk_status_t topk_transform_noalloc(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                                     int32_t batch, int32_t max_seq_len, const int32_t* page_table,
                                     int64_t page_table_stride, int32_t page_size, int32_t k,
                                     int32_t* out_indices, int32_t* out_raw_indices_or_null, topk_stream_t stream);

/* Static, human-readable name of a status code. */
const char* topk_status_string(topk_status_t status);

/*
 * Text of the last CUDA failure that made a call on this host thread return
 * TOPK_ECUDA ("" if none): the failing step and the runtime's error name and
 * message.  The library resets the CUDA runtime's per-thread error state
 * after such a failure, so it does not resurface in the caller's own
 * cudaGetLastError().  The pointer stays valid for the thread's lifetime.
 */
const char* topk_last_error_string(void);

/*
 * Dispatch knobs.  Defaults are the GB300 settings; tests use the overrides
 * to drive every path.  The values are process-wide and take effect for
 * calls made after topk_set_tuning returns; do not change them while another
 * host thread is enqueuing topk_transform.
 */
typedef struct {
    int32_t long_threshold_small_batch; /* long row if seq_len > this, batch <= small_batch_max
                                           (16384)                                               */
    int32_t long_threshold;             /* long row if seq_len > this, batch <= large_batch_min
                                           (65536)                                               */
    int32_t small_batch_max;            /* (16)                                                  */
    int32_t cluster_size;               /* blocks per long row: 2, 3, 4, 8 or 16; 0: automatic
                                           (16 for up to 4 rows; else 4 for rows of at most 64K;
                                           else 8 while every row gets a resident 8-block cluster;
                                           else 3 when 4-block clusters would take two rows on
                                           some cluster, the batch is at most four waves of
                                           3-block ones and a 3-block buffer holds the gate's
                                           sampling floor at 40 %; else 4; then raised (3 to 4,
                                           then doubled) while a row of max_seq_len would fill a
                                           buffer of max(k, 2048) past 80 % at that floor)       */
    int32_t force_two_pass;             /* 1: no candidate buffering in the first pass, so every
                                           row takes the two-pass streaming path                  */
    int32_t disable_gate;               /* 1: the first pass counts every element (no sample gate) */
    int32_t candidate_capacity;         /* 0: automatic (single blocks 4k, at least 2048, 3072
                                           on rows over 16K; clusters max(k, 2048), grown toward
                                           2.5 times the gate's sampling floor per block where the
                                           shared memory at the same blocks per SM allows); else
                                           candidates per block, 2048..16384, a multiple of 64    */
    int32_t samples;                    /* 0: automatic; else at most this many gate samples per
                                           row, 32..2048, a multiple of 32                       */
    int32_t gate_fill_percent;          /* 0: automatic; else 1..100: the gate is loosened until it
                                           is expected to pass this share of the candidate buffer
                                           (never tighter than the sampling bound needs)         */
    int32_t single_block_threads;       /* 0: automatic; 256 or 512: threads per block of the
                                           single-block kernel on rows longer than 16K            */
    int32_t single_block_copy_bytes;    /* 0: automatic; 8192, 16384, 24576 or 32768: bytes per bulk
                                           copy of the single-block kernel (taken where its block
                                           size is compiled for that copy: 256 threads all four,
                                           512 threads 16384 and 32768)                           */
    int32_t single_block_stages;        /* 0: automatic; 2..8: bulk copies in flight per block of
                                           the single-block kernel (its shared-memory ring depth) */
    int32_t gate_refresh_tiles;         /* 0: off; 1..64: the 256-thread single-block kernel
                                           tightens a row's gate every this many bulk copies from
                                           the counts of its histogram so far (a monotone gate that
                                           never drops a top-k element); other kernels ignore it  */
    int32_t warp_rows;                  /* the warp-per-row kernel (one warp per row) for batches
                                           whose rows are all at most 16384 long, with k <= 512:
                                           0: automatic (from warp_batch_min rows on); 1: always;
                                           2: never                                              */
    int32_t wait_limit_us;              /* 0: 2 s; else 1..60000000: how long a select block waits
                                           for one bulk copy of scores before it gives up, sets
                                           TOPK_FLAG_TIMEOUT (the call's output is then void) and
                                           stops issuing copies; the call still returns, and the
                                           block waits for its copies in flight before it exits  */
    int32_t single_block_kernel;        /* 0: automatic (shape 2 for rows of 16K..64K from
                                           stream_batch_min rows on, when two blocks fit an SM);
                                           1: the single-role kernel; 2 / 3: the warp-specialised
                                           kernel, in which 8 warps stream row q while other warps
                                           finish row q - 1: 2 = 4 finishing warps, a 2 x 32 KB
                                           ring, two blocks per SM (k <= 624); 3 = 8 finishing
                                           warps, up to 4 x 32 KB, one block per SM.  It takes
                                           rows of up to 65536; longer ones use the single-role
                                           kernel whatever this field says                       */
    int32_t long_threshold_large_batch; /* long row if seq_len > this, batch > large_batch_min
                                           (131072)                                              */
    int32_t large_batch_min;            /* (64)                                                  */
    int32_t warp_batch_min;             /* batch from which the automatic dispatch takes the
                                           warp-per-row kernel (1024)                            */
    int32_t stream_batch_min;           /* batch from which the automatic dispatch takes the
                                           warp-specialised kernel (384)                         */
    int32_t split_rows;                 /* the segment-split path (the rows of the whole batch
                                           cut into segments that every SM streams; the block
                                           that finishes a row's last segment resolves it), for
                                           batches of up to 128 rows whose longest row keeps its
                                           gated candidates within the path's per-row buffer
                                           (about 2M tokens at k = 2048): 1: always; 0
                                           (automatic) and 2: never.  On GB300 it is faster on
                                           batches that mix a few very long rows with short ones
                                           (1 x 1M + 63 x 4K, k = 2048: 33 vs 39 us; 4 x 1M +
                                           124 x 8K, k = 1024: 34 vs 58 us) and slower on batches
                                           of similar lengths (8 x 1M: 47 vs 33 us; 128 ragged
                                           rows up to 256K: 63 vs 49 us); the host does not see
                                           the lengths, so the caller chooses                    */
    int32_t split_segment;              /* 0: automatic; else a power of two, 4096..1048576:
                                           elements per segment of the split path (raised where
                                           the batch would need more than 16384 segments)        */
    int32_t split_full_resolve;         /* 1: the split path resolves every row from a full
                                           re-read of the row (the path it otherwise takes only
                                           when a row's gate misses); for tests                  */
} topk_tuning_t;

topk_status_t topk_get_tuning(topk_tuning_t* tuning_host);
topk_status_t topk_set_tuning(const topk_tuning_t* tuning_host);

#ifdef __cplusplus
}
#endif

#endif /* TOPKIDX_H */
