/*
 * opw.h -- C ABI of the tile-centric AllGather->GEMM / GEMM->ReduceScatter
 * overlap library for NVIDIA GB300 (sm_103a).
 *
 * The operations follow "Triton-distributed Semantics" (sections
 * "Producer-Consumer Model", "Signal-Based Synchronization", "Symmetric
 * Memory Model", "AllGather and GEMM Overlapping", "GEMM and ReduceScatter
 * Overlapping", "Threadblock Swizzling", "Token-Based Data Dependency") and
 * "Distributed Architecture Design" (section 2.3 SignalOp, section 5 symmetric
 * heap, section 6 signal/wait mechanisms).  The epoch carried by every signal
 * follows the put_signal / wait_signal(flag, epoch) contract of the Aboleth
 * README ("Tier 1" device library).
 *
 * All R ranks are LOGICAL ranks on one GPU: each rank owns one slice of a
 * single device allocation (the "heap"), and an offset table stands in for
 * the peer mappings of a real symmetric heap.
 *
 * Conventions
 *   - Pointers named *_dev are device pointers; everything else is host.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *   - Matrices are row-major bf16 (IEEE binary32 upper half), element
 *     (i, j) of an [rows, cols] matrix at byte offset 2*(i*cols + j).
 *   - Every call that takes a stream is asynchronous: argument errors are
 *     returned at once; errors found on the device (a wait that timed out, a
 *     flag protocol violation) are latched in the signal object's status
 *     word and returned by opw_status_sync().  Once a device error is
 *     latched, later launches on that signal object do no work until
 *     opw_signal_reset().
 *   - No function throws, prints or aborts.  No function allocates memory
 *     except opw_signal_alloc().
 *   - The caller owns every buffer it passes and keeps it alive until the
 *     stream has executed the call.  The library owns only opw_signal.
 */
#ifndef OPW_H
#define OPW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OPW_ABI_VERSION 2
#define OPW_MAX_RANKS 8

/* ---------------------------------------------------------------- status */

typedef int32_t opw_status;
#define OPW_OK                    0
#define OPW_ERR_INVALID_ARG       1  /* NULL pointer, bad enum, R out of range, too few slots */
#define OPW_ERR_UNSUPPORTED_SHAPE 2  /* a size is not a multiple of the flag tile, or <= 0 */
#define OPW_ERR_MISALIGNED        3  /* a pointer or offset is not 16-byte aligned (TMA rule) */
#define OPW_ERR_BAD_EPOCH         4  /* epoch is not the next one for this signal object */
#define OPW_ERR_CUDA              5  /* a CUDA runtime/driver call failed */
#define OPW_ERR_TIMEOUT           6  /* a device-side wait ran past opts.timeout_ns */
#define OPW_ERR_FLAG_PROTOCOL     7  /* a flag held a value other than the epoch it should */
#define OPW_ERR_NOT_READY         8  /* the signal object has a latched device error; reset it */

/* Human-readable name of a status code (static storage, never NULL). */
const char* opw_status_str(opw_status s);

/* OPW_ABI_VERSION of the loaded library. */
int32_t opw_abi_version(void);

/* ---------------------------------------------------------------- signals */

/*
 * A signal object: an array of int64 flags in device memory ("Signal-Based
 * Synchronization": one signal per tile), the host-side epoch counter, and a
 * device status word.  A flag holds the last epoch published for its tile
 * (SignalOp SET, "Distributed Architecture Design" 2.3); a waiter spins until
 * flag >= epoch (the GE predicate of section 6.3).  Waiting never modifies a
 * flag (non-consuming wait, section 6.3); only opw_signal_reset() writes
 * flags back to 0, so the reset is the one step that must be ordered against
 * the launches (section 6.3).  Flags are
 * dense (8 bytes apart): on GB300 the L2 is the coherence point for
 * .gpu-scope release/acquire, so the 64-byte slot stride that section 4.2
 * needs on Ascend buys nothing here.
 */
typedef struct opw_signal opw_signal;

/*
 * Allocate a signal object with `num_slots` flags (>= 1), all 0, epoch 0.
 * The zeroing is enqueued on `stream`.  On success *out owns device memory
 * until opw_signal_free().  Errors: INVALID_ARG (out NULL, num_slots < 1),
 * CUDA (allocation failed; *out is left NULL).
 */
opw_status opw_signal_alloc(opw_signal** out, int64_t num_slots, void* stream);

/*
 * Enqueue on `stream`: every flag := 0, the device status word := OK, the
 * internal counters := 0; and set the host epoch counter to 0, so the next
 * epoch is 1.  The caller must not have launches on this object in flight
 * on other streams.  Errors: INVALID_ARG (NULL), CUDA.
 *
 * CUDA graphs: a launch takes its epoch and claim bases from the host, so a
 * captured launch replays the same ones.  Capture this reset and then the
 * launch at epoch 1 (after one call outside any capture, which sets up the
 * library's per-device state): every replay zeroes the flags and publishes
 * epoch 1 again.  A whole tensor-parallel step (opw_ag_gemm, then
 * opw_gemm_rs, each behind the reset of its own signal object) replays
 * this way.
 */
opw_status opw_signal_reset(opw_signal* sig, void* stream);

/* Free a signal object (synchronises the device first).  NULL is a no-op. */
opw_status opw_signal_free(opw_signal* sig);

/* *epoch := last epoch published on this object + 1 (the value the next
 * fused or producer-only launch must pass).  Errors: INVALID_ARG. */
opw_status opw_signal_next_epoch(const opw_signal* sig, uint64_t* epoch);

/* Device pointer to the flag array and its length (for read-back checks).
 * Errors: INVALID_ARG. */
opw_status opw_signal_flags(const opw_signal* sig, int64_t** flags_dev, int64_t* num_slots);

/*
 * Synchronise `stream`, then read and return the device status word.  If a
 * device-side error was latched, *rank / *tile (either may be NULL) receive
 * the logical rank and flag slot the failing wait was on (-1 if none).
 * The latched error stays until opw_signal_reset().  Every device-side wait
 * on a signal ("Distributed Architecture Design" 6.3, wait until the signal
 * satisfies its predicate) is bounded by opts.timeout_ns; a wait that runs
 * out is reported here instead of hanging.
 */
opw_status opw_status_sync(opw_signal* sig, void* stream, int32_t* rank, int32_t* tile);

/* ---------------------------------------------------------------- heap */

/*
 * Logical symmetric heap ("Distributed Architecture Design" 5.3): rank r's
 * slice starts at heap_dev + rank_off[r].  A symmetric object at offset `off`
 * is at heap_dev + rank_off[r] + off on rank r, which is symm_at(ptr, r) =
 * ptr - heap_base[self] + heap_base[r] with heap_base[r] = heap_dev +
 * rank_off[r].  rank_off is a HOST array of R entries, read during the call
 * only; entries need not be increasing (a permuted table is allowed) and
 * must be multiples of 16.
 */
typedef struct {
    void* heap_dev;
    const int64_t* rank_off;
    int32_t R;          /* 1 .. OPW_MAX_RANKS */
    int32_t reserved;   /* must be 0 */
} opw_symm;

/* ---------------------------------------------------------------- options */

#define OPW_SYNC_OVERLAP 0   /* per-tile flags: consumers start as tiles land */
#define OPW_SYNC_SERIAL  1   /* consumers wait until EVERY tile is published
                                (the debugging step of "Triton-distributed
                                Semantics", Best Practices 8: rule out the
                                fine-grained synchronisation first) */
#define OPW_SYNC_CHECKED 2   /* as OVERLAP, but every publish is an atomic exchange
                                that must find epoch-1 in the slot (with
                                OPW_SIGNAL_ROW_ADD: a fetch-add that must find a
                                count of this epoch's window), so each slot is
                                published exactly once per epoch; otherwise the
                                launch stops with OPW_ERR_FLAG_PROTOCOL (rank, slot).
                                AG-GEMM and GEMM-RS.  Every launch on the signal
                                object since its last reset must have covered the
                                same slots (same R and tile geometry): slots an
                                earlier launch did not publish hold older epochs. */

/* Both schedules walk one order of the 256 x TN output tiles (TN = the pair
 * tile width of the launch, 256 or 512; see opw_ag_tile_n): pair rows in
 * groups (8 when B is over 64 MiB, else 1), the column index outermost in a
 * group and running backwards in every second group; rows renamed so that the
 * PE the GPU plays (opts.local_rank, rank 0 when -1) starts on its own rows,
 * then the other ranks' rows in publish order: with the default ring publish
 * order that is "Threadblock Swizzling"'s pid_m = (pid_m + rank *
 * tiles_per_pe) % total_tiles with tiles_per_pe = M_r / 256. */
#define OPW_SCHED_READY   0  /* dynamic (default): CTA pairs claim positions of
                                that order from a device counter, so every
                                consumer starts on the tiles that are ready
                                first */
#define OPW_SCHED_SWIZZLE 1  /* static: CTA pair c takes positions c, c + G,
                                c + 2G, ... of that order (G pairs) */

#define OPW_ROLE_FUSED    0  /* producer warps and consumer warps together */
#define OPW_ROLE_PRODUCER 1  /* only the gather + publish (for overlap timing) */
#define OPW_ROLE_CONSUMER 2  /* only wait + GEMM; the epoch must already be
                                published by an earlier producer launch */

#define OPW_SIGNAL_TILE_SET 0  /* one flag per flag tile, SET to the epoch (default) */
#define OPW_SIGNAL_ROW_ADD  1  /* one counter per flag row (rank r, row tile mt):
                                  the producer ADDs 1 per published k-tile
                                  (SignalOp ADD, "Distributed Architecture Design"
                                  2.3); a consumer starts on the row only when the
                                  counter reaches epoch * K/ft, i.e. every k-tile of
                                  the row is in (signals shared by tiles that are
                                  always used together, Best Practices 4).
                                  Counters are cumulative, so a
                                  signal object must keep one mode and one K/ft
                                  between resets. */

#define OPW_FAULT_NONE        0
#define OPW_FAULT_DROP_TILE   1  /* the producer never publishes flag slot fault_arg */
#define OPW_FAULT_STALE_EPOCH 2  /* the producer publishes epoch-1 into slot fault_arg */

typedef struct {
    uint64_t timeout_ns;          /* bound on every device-side wait; 0 = 2e9 (2 s) */
    int32_t sync_mode;            /* OPW_SYNC_* */
    int32_t schedule;             /* OPW_SCHED_* */
    int32_t role;                 /* OPW_ROLE_* */
    int32_t num_ctas;             /* persistent grid size; 0 = one CTA per SM.  AG-GEMM
                                     and GEMM-RS run CTAs in pairs (clusters of 2): the
                                     count is rounded down to an even number, at least 2,
                                     and capped at the pairs that can be resident. */
    const int32_t* publish_perm;  /* host [R] or NULL: rank publish_perm[i] is published
                                     i-th, and none of its tiles before every tile of
                                     rank publish_perm[i-1] is published.  NULL: ranks
                                     in ring order after local_rank (local_rank + 1,
                                     + 2, ...), the local rank's own shard last. */
    const uint32_t* delay_ns;     /* host [R] or NULL: no copy of rank r starts earlier
                                     than delay_ns[r] after its CTA started */
    uint64_t* trace_dev;          /* device [opw_ag_trace_words()] or NULL; see below */
    int32_t fault_kind;           /* OPW_FAULT_* (fault injection on the host-chosen slot) */
    int32_t fault_arg;
    int32_t signal_mode;          /* OPW_SIGNAL_* (AG-GEMM only) */
    int32_t local_rank;           /* AG-GEMM: the logical rank the consumer plays, whose own
                                     shard is local (default 0); -1: none.  Other calls
                                     accept 0 or -1 and ignore it.  See opw_ag_gemm. */
    int32_t tile_n;               /* AG-GEMM: output columns of a pair tile, 256 or 512;
                                     0 (default) = the library's choice for the shape and
                                     grid (opw_ag_tile_n).  Other calls require 0. */
} opw_opts;

/* Fill *o with the defaults (all fields 0 / NULL). */
void opw_opts_default(opw_opts* o);

/* ---------------------------------------------------------------- AG-GEMM */

/*
 * Sizing of the signal object for AG-GEMM ("Signal-Based Synchronization":
 * one signal per tile; "AllGather and GEMM Overlapping" step 2, a signal
 * after each tile transfer).  Flag tile (square, in elements) used for
 * shapes (M_r, K): 128 when both are multiples of 128, else 64.  Flag slot
 * of tile (r, mt, kt): (r * (M_r/ft) + mt) * (K/ft) + kt.  Returns the slot
 * count, or -1 for invalid sizes.
 */
int64_t opw_ag_flag_tile(int64_t M_r, int64_t K);
int64_t opw_ag_num_flags(int32_t R, int64_t M_r, int64_t K);

/* Counters needed with OPW_SIGNAL_ROW_ADD: R * (M_r/ft); counter of flag row
 * (r, mt) is slot r * (M_r/ft) + mt.  -1 for invalid sizes. */
int64_t opw_ag_num_row_counters(int32_t R, int64_t M_r, int64_t K);

/*
 * Trace of an AG-GEMM launch: the order checks of "Best Practices" 6
 * (profile the overlap and the synchronization).  Layout (uint64 words),
 * written only when opts.trace_dev != NULL:
 *   [0, F)            publish time (%globaltimer ns) of each flag slot
 *   [F, 2F)           earliest time a consumer's acquire of the slot
 *                     succeeded (atomicMin; the caller fills this range
 *                     with all-ones bits before the launch)
 *   [2F, 2F+T)        per 256 x TN output tile q = (row / 256) * ceil(N/TN)
 *                     + col / TN: (pair << 32) | visit position, where
 *                     pair c is the CTA pair 2c, 2c+1
 *   [2F+T, 2F+2T)     per output tile: time its pair's scheduler claimed it
 *                     (before its first flag acquire)
 *   [2F+2T, 2F+2T+G)  per CTA: start time
 * with F = opw_ag_num_flags(), T = ceil(M/256)*ceil(N/TN), TN the launch's
 * pair tile width (opw_ag_tile_n), G = grid size (at most OPW_TRACE_MAX_CTAS
 * words are reserved).  opw_ag_trace_words() sizes the buffer for TN = 256,
 * which also covers TN = 512.
 */
#define OPW_TRACE_MAX_CTAS 1024
int64_t opw_ag_trace_words(int32_t R, int64_t M_r, int64_t N, int64_t K);

/*
 * Output columns TN of the pair tiles an opw_ag_gemm (or opw_ag_gemm_noalloc)
 * launch with these sizes and options uses on the current device: opts->tile_n
 * when it is set, else the library's choice.  A 256 x 512 pair tile reads a
 * quarter less operand data from L2 per FLOP than a 256 x 256 one (a lower
 * on-chip power draw, so a higher clock under the power cap), but holds its
 * one 512-column TMEM accumulator through the epilogue; the library takes it
 * when its whole waves of tiles, at 1.93 times the time of a 256-wide wave,
 * are shorter than the 256-wide waves.  This refines the pages' consumer
 * program, which owns one output tile ("AllGather and GEMM Overlapping"), with no
 * change to the results: every output element sums the same products in the
 * same order.  Returns 256, 512, or -1 (invalid arguments, or no CUDA device
 * to size the grid for when opts->tile_n is 0).  opts may be NULL.
 */
int32_t opw_ag_tile_n(int32_t R, int64_t M_r, int64_t N, const opw_opts* opts);

/*
 * AllGather -> GEMM ("AllGather and GEMM Overlapping"):
 *   G = concat(A_0, ..., A_{R-1})  along rows        (the AllGather)
 *   C = G * B                       fp32 accumulate, bf16 round-to-nearest-even
 *
 *   symm    : logical heap; A_r = [M_r, K] bf16 at heap_dev + rank_off[r] + a_off.
 *   B_dev   : [K, N] bf16.
 *   G_dev   : [R*M_r, K] bf16 gathered buffer, written by the producer warps.
 *   C_dev   : [R*M_r, N] bf16 output.
 *   sig     : at least opw_ag_num_flags(R, M_r, K) slots
 *             (opw_ag_num_row_counters with OPW_SIGNAL_ROW_ADD).
 *   epoch   : opw_signal_next_epoch() for FUSED / PRODUCER roles; for the
 *             CONSUMER role, the epoch an earlier PRODUCER launch published.
 *   opts    : NULL = defaults.
 *
 * Producer warps copy each flag tile of each A_r into G with TMA, wait for the
 * copy to complete, then publish flags[slot] = epoch with a .gpu release.
 * The GPU plays the consumer of rank opts.local_rank (default 0): that rank's
 * own shard is local, so consumers read its rows in place from A_local and
 * never wait on its flags, and they take its tiles first.  Its tiles are still
 * copied into G (after every other rank's) and published.  With local_rank =
 * -1 every tile is read from G after its flag.
 * Consumers, in CTA pairs working on 256 x TN output tiles (opw_ag_tile_n),
 * acquire each flag (>= epoch) before their TMA loads read that tile of G,
 * then run tcgen05 cta_group::2 MMAs with TMEM accumulators.  After the launch every flag slot
 * holds `epoch` and G is bit-identical to the concatenation.
 *
 * Producer warps claim flag tiles from a device counter in publish order, so
 * every flag is published by CTAs that are running: the launch (clusters of 2,
 * one CTA per SM) needs no co-residency guarantee, and profilers can replay it.
 *
 * Shapes: M_r, K multiples of 64 (flag tile 64) or 128; N a multiple of 8;
 * R*M_r, N, K <= 2^31.  Alignment: heap_dev, B_dev, G_dev, C_dev, a_off and
 * rank_off[] multiples of 16 bytes.  G and C must not overlap any A_r or B.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, BAD_EPOCH, NOT_READY,
 * CUDA (launch failure).  Device errors (TIMEOUT, FLAG_PROTOCOL) surface at
 * opw_status_sync().
 */
opw_status opw_ag_gemm(const opw_symm* symm, size_t a_off, int64_t M_r, int64_t N, int64_t K,
                       const void* B_dev, void* G_dev, void* C_dev, opw_signal* sig,
                       uint64_t epoch, const opw_opts* opts, void* stream);

/* ------------------------------------------- AG-GEMM without allocation */

/*
 * The pages have no counterpart to this call: it exists for callers that
 * cannot allocate device memory.  opw_ag_gemm needs a signal object, and
 * opw_signal_alloc calls cudaMalloc.  Some callers cannot: code that runs
 * inside a framework owning all device memory through its own pool (a raw
 * allocation bypasses its accounting or fails against its cap), and
 * latency-critical serving loops that cannot take cudaMalloc's implicit
 * device synchronisation.  This variant computes the same G and C as
 * opw_ag_gemm and calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Scratch: the per-tile flags and counters live in one fixed array compiled
 * into the library, sized for OPW_NOALLOC_MAX_FLAGS flag tiles (about
 * 512 KiB).  Every GPU that loads the library holds it until the process
 * exits.  A call whose opw_ag_num_flags(R, M_r, K) exceeds the maximum is
 * rejected with OPW_ERR_UNSUPPORTED_SHAPE before anything is launched.
 *
 * Sharing: every call on a device uses the same array.  Each call clears the
 * flags and counters it needs (and *status_dev) on `stream`, then publishes
 * epoch 1.  Calls that overlap on the GPU (other streams, other threads)
 * therefore race and give wrong results: serialise them.
 *
 * Set-up: the first call on a device, with that device current, looks up
 * the array's device address and keeps it for the life of the process.  Make
 * that first call before any stream capture.  After it, a call can be
 * captured in a CUDA graph: it launches the same two kernels (clear, then
 * AG-GEMM) with the same arguments every time, so replaying the graph
 * recomputes G and C from whatever the captured buffers then hold.  cudaDeviceReset() (or anything
 * else that destroys the device's primary context) invalidates the kept
 * address: do not call this entry point on that device afterwards.
 *
 * Every buffer (the heap, B_dev, G_dev, C_dev, status_dev) must be memory of
 * the current device; otherwise the call returns OPW_ERR_INVALID_ARG before
 * launching anything.
 *
 *   status_dev : device int32[4], 16-byte aligned, written by the call:
 *                [0] status (OPW_OK or a device-side error such as
 *                OPW_ERR_TIMEOUT), [1] rank, [2] flag slot.  The caller reads
 *                it after synchronising the stream.
 *   opts       : as for opw_ag_gemm, except role must be OPW_ROLE_FUSED.
 * All other arguments, shapes, alignment rules and errors are those of
 * opw_ag_gemm (there is no signal object and no epoch argument).
 */
#define OPW_NOALLOC_MAX_FLAGS 65536
opw_status opw_ag_gemm_noalloc(const opw_symm* symm, size_t a_off, int64_t M_r, int64_t N,
                               int64_t K, const void* B_dev, void* G_dev, void* C_dev,
                               int32_t* status_dev, const opw_opts* opts, void* stream);

/* ---------------------------------------------------------------- GEMM-RS */

/* Flag slots for GEMM-RS outputs ("GEMM and ReduceScatter Overlapping" step
 * 2, a signal after each tile is computed): 128x128 tiles of each rank's
 * [M/R, N] block, slot (j * (M/R/128) + mt) * ceil(N/128) + nt.  -1 if
 * invalid. */
int64_t opw_rs_num_flags(int32_t R, int64_t M, int64_t N);

/*
 * GEMM -> ReduceScatter ("GEMM and ReduceScatter Overlapping"):
 *   P_r   = A_r * B_r                  (fresh fp32 TMEM accumulator per rank)
 *   S     = (((0 + P_0) + P_1) + ...)  fp32 adds in rank order 0..R-1
 *   out_j = bf16_rne(rows [j*M/R, (j+1)*M/R) of S), stored in rank j's slice
 *
 *   A_r   = [M, K_r] bf16 at heap_dev + rank_off[r] + a_off
 *   B_r   = [K_r, N] bf16 at heap_dev + rank_off[r] + b_off
 *   out_j = [M/R, N] bf16 at heap_dev + rank_off[j] + out_off
 *
 * CTA pairs work on 256x256 output tiles.  The pair's MMA (tcgen05
 * cta_group::2) produces partial tiles into a double-buffered TMEM
 * accumulator and signals each on an on-chip barrier; the reduction warps of
 * both CTAs add them in rank order as they land, write each finished row
 * block to its rank, and publish flags[slot] = epoch (.gpu release) per
 * 128x128 output tile.
 *
 * Roles (opts->role), for timing the two legs apart:
 *   OPW_ROLE_FUSED    the whole path (default).
 *   OPW_ROLE_PRODUCER the GEMM leg alone: loads, MMAs and the rank-order
 *                     sums; no output is stored, no flag is published, and
 *                     `epoch` (which must still be the next epoch) is not
 *                     used up.
 *   OPW_ROLE_CONSUMER the scatter leg alone: no loads and no MMAs, so S is 0;
 *                     every output tile is stored as bf16 zeros in its
 *                     rank's block and its flag published with `epoch`.
 *
 * Shapes: M a multiple of 128*R; K_r and N multiples of 8 (a ragged last
 * k-block or column tile is zero-filled by TMA and not stored).
 * Alignment and errors as for opw_ag_gemm.  `opts` fields used: timeout_ns,
 * num_ctas, role, sync_mode (OVERLAP or CHECKED), trace_dev, fault_kind
 * (NONE, or DROP_TILE: flag slot fault_arg is never published); the others
 * must be defaults.  With trace_dev (device, 2 * opw_rs_num_flags() uint64
 * words) word `slot` receives the %globaltimer time at which the slot was
 * published, and word F + slot the time the receiving side of
 * opw_gemm_rs_consume acquired it.
 */
opw_status opw_gemm_rs(const opw_symm* symm, size_t a_off, size_t b_off, size_t out_off,
                       int64_t M, int64_t N, int64_t K_r, opw_signal* sig, uint64_t epoch,
                       const opw_opts* opts, void* stream);

/*
 * GEMM -> ReduceScatter with the receiving side in the same launch
 * ("GEMM and ReduceScatter Overlapping", step 3: the consumer waits for
 * tiles as they are published).  Computes exactly what opw_gemm_rs computes,
 * and in addition, for every 128x128 output tile of every rank's block, a
 * warp on another SM than the one that stored the tile acquires the tile's
 * flag (>= epoch, a bounded wait) and only then copies the tile from out_j
 * into recv_dev.  Afterwards recv_dev [M, N] bf16 (row i of S at row i)
 * equals the concatenation out_0, ..., out_{R-1} bit for bit.
 *
 *   recv_dev : device, [M, N] bf16, 16-byte aligned, must not overlap the
 *              heap's A_r, B_r or out_j; written only after each tile's flag
 *              is acquired.
 * opts->role must be OPW_ROLE_FUSED.  A flag that never comes (fault_kind
 * DROP_TILE) makes the receiving wait run out: OPW_ERR_TIMEOUT with the
 * rank and slot, latched in the signal object.  Other arguments and errors
 * as for opw_gemm_rs; recv_dev NULL is INVALID_ARG.
 */
opw_status opw_gemm_rs_consume(const opw_symm* symm, size_t a_off, size_t b_off, size_t out_off,
                               int64_t M, int64_t N, int64_t K_r, void* recv_dev, opw_signal* sig,
                               uint64_t epoch, const opw_opts* opts, void* stream);

/* ---------------------------------------------------------- ring AllReduce */

/*
 * Tile-centric ring AllReduce over the R logical ranks ("Triton-distributed
 * Semantics", "Example: Ring AllReduce with Overlap").  Rank r holds n fp32
 * values at heap_dev + rank_off[r] + data_off, viewed as R chunks of n/R.
 * Reduce-scatter: chunk c's partial starts at rank c and visits ranks c+1,
 * c+2, ... (mod R), each adding its own copy (reduced = local + incoming,
 * binary32, round to nearest); all-gather: the finished chunks go around the
 * ring once more.  On return every rank's out_off holds the same n values.
 *
 * Each chunk is cut into pieces of 1024 values that move independently; the
 * piece arriving at rank r in ring step g sits in r's receive area at
 * recv_off + 4*(g*n/R + piece offset) and is announced by flag slot
 * (r*(2R-2) + g)*P + piece, P = ceil((n/R)/1024), set to the epoch with a
 * .gpu release; the receiver acquires it (>= epoch) before reading.
 *
 *   data_off : n fp32 per rank (input, not modified)
 *   recv_off : opw_ring_recv_bytes(R, n) bytes per rank (scratch owned by the
 *              caller; contents are overwritten)
 *   out_off  : n fp32 per rank (output); must not overlap data or recv
 *   sig      : at least opw_ring_num_flags(R, n) slots; epoch = next epoch
 *   opts     : NULL or defaults except timeout_ns / num_ctas
 * Shapes: n a multiple of 4*R.  Offsets and rank_off[] multiples of 16.
 * Errors as for opw_ag_gemm.
 */
int64_t opw_ring_num_flags(int32_t R, int64_t n);
int64_t opw_ring_recv_bytes(int32_t R, int64_t n);
opw_status opw_ring_allreduce(const opw_symm* symm, size_t data_off, size_t recv_off,
                              size_t out_off, int64_t n, opw_signal* sig, uint64_t epoch,
                              const opw_opts* opts, void* stream);

/* -------------------------------------------------------------- all-to-all */

/*
 * All-to-all over the R logical ranks with put + signal + epoch (Aboleth
 * README, Tier-2 all-to-all): rank r's send buffer holds R slices of
 * bytes_per_peer bytes at heap_dev + rank_off[r] + send_off; afterwards
 * rank j's receive buffer (recv_off, R slices) holds at slot r the slice j of
 * rank r's send buffer.  Slices move in 32 KiB pieces; each piece sent to a
 * peer is announced by flag slot (j*R + r)*P + piece = epoch (.gpu release),
 * P = ceil(bytes_per_peer / 32768), and every receiver acquires all of its
 * incoming flags (>= epoch) before the call completes.  The rank's own slice
 * is copied without a flag.
 *
 *   sig  : at least opw_alltoall_num_flags(R, bytes_per_peer) slots; epoch =
 *          next epoch.   opts: NULL or defaults except timeout_ns / num_ctas.
 * Shapes: bytes_per_peer a multiple of 16.  Offsets and rank_off[] multiples
 * of 16; send and receive buffers must not overlap.  Errors as opw_ag_gemm.
 */
int64_t opw_alltoall_num_flags(int32_t R, int64_t bytes_per_peer);
opw_status opw_alltoall(const opw_symm* symm, size_t send_off, size_t recv_off,
                        int64_t bytes_per_peer, opw_signal* sig, uint64_t epoch,
                        const opw_opts* opts, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* OPW_H */
