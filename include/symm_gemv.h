/*
 * symm_gemv.h -- C ABI of the GB300 symmetric-slot GEMV + one-shot all-reduce.
 *
 * The library computes the row-parallel (tensor-parallel) linear layer
 *
 *     y = sum_{r=0}^{R-1} W_r x_r
 *
 * in one fused CUDA kernel: each rank's partial product is published as soon
 * as its row tile is done and the last contributor of a tile sums all ranks'
 * partials in fixed rank order and stores the bf16 result into every rank's
 * output slot.  The R ranks are R "symmetric slots" of one HBM allocation on
 * one GPU: the same offset in every slot names the same tensor of each rank,
 * the way a symmetric-memory handle's per-peer buffer pointers do.
 *
 * Sources for the semantics (page titles and sections):
 *  - "PyTorch Symmetric Memory" documentation: symmetric allocation
 *    (`empty`), `rendezvous` and the handle's buffer / signal-pad pointers
 *    ("Hello World", "Write your own kernel", API reference); the signal pad
 *    whose size scales with launched blocks and world size
 *    (`set_signal_pad_size`); op reference `one_shot_all_reduce` (sum only);
 *    the warning that all symmetric-memory collectives of a group must run on
 *    one CUDA stream; the "higher-precision reduction" note (bf16 in, fp32
 *    accumulate, bf16 out).
 *  - "PyTorch Symmetric Memory: A New Programming Paradigm for Distributed
 *    AI" (talk): the one-shot all-reduce -- every rank loads the block of every
 *    rank and reduces locally.
 *  - "Overlapping Collective Communication with Dependent Computation in
 *    Distributed Machine Learning using GPU-Initiated Intra-Kernel
 *    Networking" (summary of "Optimizing Distributed ML Communication with
 *    Fused Computation-Collective Operations"), Abstract: the fused GEMV +
 *    AllReduce operator, partials pushed as soon as each share is computed,
 *    zero-copy writes into peer memory, communication-aware workgroup
 *    scheduling.
 *  - "Bay.Area.AI: Tensor and 2D Parallelism" (talk): column-wise then
 *    row-wise sharding, which ends in exactly one all-reduce.
 *
 * Conventions for every call:
 *  - Returns SYMM_OK (0) or a negative SYMM_E* code; never aborts.  On error
 *    symm_last_error() describes the failure (thread-local string).
 *  - "Symmetric pointer": a device address inside SLOT 0's user region.  Rank
 *    r's instance is that address + r * stride (stride from symm_rendezvous).
 *  - Tensors are bf16, row-major, 16-byte aligned.
 *  - Calls that take a stream only enqueue work and return; device-side
 *    protocol errors are latched in the handle's status word (symm_status).
 *  - All calls on one handle must be issued on ONE stream (or streams the
 *    caller serialises): the per-tile counters and flags of the signal pad
 *    are shared by every launch on the handle.  Overlapping launches on the
 *    same handle are detected (SYMM_EPROTO in symm_status) rather than hung:
 *    no kernel in this library waits on another CTA.
 *  - A handle's host-side state (options, the output range of the last call,
 *    packed-weight registrations, cached tensor maps) is not locked: use a
 *    handle from one host thread at a time.  Different handles are
 *    independent.
 *  - Device memory ownership: the library owns what symm_alloc allocates
 *    (backing == NULL) and frees it in symm_free; borrowed backing memory
 *    stays the caller's and must outlive the handle.
 *  - CUDA graphs: every call on a handle may be captured into a CUDA graph
 *    and the graph replayed any number of times ("PyTorch Symmetric Memory" docs:
 *    the signal-pad synchronisation primitives are CUDA-graph compatible).
 *    The fused calls keep their whole protocol state in the signal pad: the
 *    launch epoch (advanced on the device by the last tile's reducer), the
 *    per-tile arrival counters and the work counters are back at zero when a
 *    launch ends, so a launch depends on no host-side state and eager calls
 *    of any geometry may run on the handle between replays.  Make one eager
 *    call of each kind before capturing it, so that one-time set-up (kernel
 *    attributes) happens outside the capture.
 *  - After a launch in which a CTA gave up (a bounded wait ran out, latched
 *    in the status word), the epoch is not advanced and the results of later
 *    fused calls are undefined until symm_status has reported the error and
 *    reset the signal pad.
 */
#ifndef SYMM_GEMV_H
#define SYMM_GEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque handle: R slots carved from one device allocation. */
typedef struct symm_handle symm_handle_t;

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *symm_stream_t;

enum {
    SYMM_OK = 0,
    SYMM_EINVAL = -1,   /* bad argument: count, size, alignment, pointer outside slot 0 */
    SYMM_ENOMEM = -2,   /* device allocation failed or backing too small */
    SYMM_ECUDA = -3,    /* a CUDA runtime call failed (message names it) */
    SYMM_ERANGE = -4,   /* the problem exceeds the handle's scratch or signal-pad capacity */
    SYMM_EPROTO = -5,   /* device protocol error: stale or missing tile flag, bad ticket */
    SYMM_ECORRUPT = -6  /* a guard band around a region was overwritten */
};

/* Largest rank count and batch width the kernels accept. */
#define SYMM_MAX_RANKS 64
#define SYMM_MAX_BATCH 16

/*
 * symm_layout -- the slot stride and total bytes symm_alloc needs for these
 * sizes, so a caller can provide (borrow) the backing memory itself.
 *   R                 ranks, 1..SYMM_MAX_RANKS
 *   slot_bytes        user region per slot (W_r, x_r, y, all-reduce in/out)
 *   scratch_bytes     fp32 partial-product region per slot (>= 4*B*N for a
 *                     gemv_all_reduce of batch B and N rows; 0 if unused)
 *   signal_pad_bytes  per-slot signal pad; holds one flag and one counter per
 *                     row tile (PyTorch Symmetric Memory docs,
 *                     set_signal_pad_size: size proportional to launched
 *                     blocks and world size); >= 4096
 * Writes *stride_out and *total_bytes_out.  Host only; no device work.
 */
int symm_layout(int R, size_t slot_bytes, size_t scratch_bytes, size_t signal_pad_bytes,
                size_t *stride_out, size_t *total_bytes_out);

/*
 * symm_alloc -- carve R symmetric slots out of one device allocation
 * (PyTorch Symmetric Memory docs, API reference `empty`: host-synchronous,
 * meant for initialisation, allocate once and reuse).
 *   backing, backing_bytes  NULL/0: the library cudaMalloc's the memory on the
 *       current device and owns it.  Otherwise a device pointer the caller
 *       owns (256-byte aligned, >= total bytes from symm_layout); the library
 *       borrows it until symm_free.
 *   out  receives the handle.
 * Zeroes every slot's scratch region and signal pad and fills the guard bands,
 * then synchronises the device.  Errors: SYMM_EINVAL (R outside 1..64,
 * slot_bytes == 0, pad < 4096, misaligned or undersized backing),
 * SYMM_ENOMEM, SYMM_ECUDA.
 */
int symm_alloc(int R, size_t slot_bytes, size_t scratch_bytes, size_t signal_pad_bytes,
               void *backing, size_t backing_bytes, symm_handle_t **out);

/*
 * symm_mp_alloc / symm_mp_import -- a handle whose R ranks are R processes
 * (on one GPU or several GPUs of one node), the symmetric memory of the
 * "PyTorch Symmetric Memory" docs ("Hello World": every rank allocates its
 * symmetric buffer, `rendezvous` exchanges the handles, after which each rank
 * holds its peers' buffer and signal-pad pointers).
 *
 * symm_mp_alloc allocates THIS process's slot (rank `rank` of R; sizes as for
 * symm_alloc, identical on every rank) as a CUDA virtual-memory allocation
 * on the current device, reserves one address range for all R slots and maps
 * the own slot at base + rank * stride.  It returns the handle and, in
 * *fd_out, a POSIX file descriptor of the allocation: the caller sends it to
 * every other rank's process (over a Unix-domain socket, as the binding's
 * multiproc.exchange_fds does) and closes it once they have it.  Host-
 * synchronous.  Errors: SYMM_EINVAL, SYMM_ENOMEM, SYMM_ECUDA.
 *
 * symm_mp_import maps rank `peer`'s slot, from the descriptor this process
 * received, at base + peer * stride.  The caller may close fd afterwards.
 * Once every peer is imported, symm_rendezvous returns all R slot pointers
 * and every symmetric pointer addresses rank r's instance at + r * stride, in
 * every process alike.  The allocations stay mapped until symm_free, also
 * after a peer's process has exited.
 *
 * On such a handle each process launches its own rank's share of a call:
 *  - gemv_all_reduce / gemv_reduce_scatter (paths 1 and 4): this process
 *    computes the units of its rank and publishes their partials; whichever
 *    process's CTA arrives last at a tile sums every rank's partials (loads
 *    from the peers' slots) and stores the result into every rank's y
 *    (stores into the peers' slots).  No kernel waits on another process.
 *  - one_shot_all_reduce: this process reads every rank's input and writes
 *    its own rank's output.
 *  - symm_pack_w packs the own rank's weight.
 * The other collectives, the bias + RMSNorm form and SYMM_OPT_UNFUSED return
 * SYMM_EINVAL.  Every rank must issue the same sequence of calls, and the
 * caller must order them across processes the way one stream orders them on
 * one handle: a call's inputs written in every process before any process
 * launches it, and every process's launch of a call finished before any
 * launches the next (e.g. stream synchronisation and a process-group barrier
 * between calls).  A rank that skips a call (or leaves) leaves the others'
 * tiles unreduced, and nothing waits for it.  Each process's symm_status,
 * called after such a barrier, reports SYMM_EPROTO naming that rank: it
 * compares the ranks' launch counts (every rank's epoch word) besides its own
 * status words, where its kernels latch stale flags and tickets out of range
 * found in later calls.  It resets its own slot's status words and pad (rank
 * 0's holds the shared tile counters) but keeps the process's launch count,
 * so the ranks' counts stay comparable whatever order they reset in; after an
 * error every rank calls it, after a barrier.
 * symm_check_guards checks the own slot.  No counterpart on the pages beyond
 * the symmetric-memory semantics above.
 */
int symm_mp_alloc(int R, int rank, size_t slot_bytes, size_t scratch_bytes, size_t signal_pad_bytes,
                  symm_handle_t **out, int *fd_out);
int symm_mp_import(symm_handle_t *h, int peer, int fd);

/*
 * symm_rendezvous -- the per-rank pointer tables of the handle (PyTorch
 * Symmetric Memory docs, `rendezvous` and the handle's `buffer_ptrs` /
 * `signal_pad_ptrs`).  Host only, not stream-ordered, not capturable; later
 * calls return the same values.  No multicast pointer exists.
 *   slot_ptrs        [R] out: device address of each rank's user region
 *                    (NULL to skip)
 *   signal_pad_ptrs  [R] out: device address of each rank's signal pad
 *                    (NULL to skip)
 *   stride_out       out: bytes between consecutive slots (NULL to skip)
 * The pointers are borrowed; valid until symm_free.
 */
int symm_rendezvous(symm_handle_t *h, void **slot_ptrs, void **signal_pad_ptrs,
                    size_t *stride_out);

/*
 * one_shot_all_reduce -- out_s[i] = bf16_rne( sum_{r=0}^{R-1} in_r[i] ) for
 * every rank s, the sum taken in fp32 in rank order 0..R-1 (PyTorch Symmetric
 * Memory docs, op reference `one_shot_all_reduce`, reduce op "sum"; the
 * symmetric-memory talk's one-shot algorithm: each rank reads every rank's
 * block and reduces locally; "higher-precision reduction": fp32 accumulate).
 *   in, out  symmetric bf16 pointers (slot 0), 16-byte aligned; n elements
 *            must fit in the user region.  in == out (in place) is allowed:
 *            each element is read in all slots before it is written.  Partial
 *            overlap of in and out is rejected.
 *   R        must equal the handle's rank count.
 *   n        elements per rank; 0 is a no-op.
 * Every slot's out receives identical bits.  Errors: SYMM_EINVAL, SYMM_ECUDA.
 */
int one_shot_all_reduce(symm_handle_t *h, const void *in, void *out, int R, size_t n,
                        symm_stream_t stream);

/*
 * gemv_all_reduce -- the fused row-parallel GEMV + one-shot all-reduce
 * ("Overlapping Collective Communication with Dependent Computation ...",
 * Abstract, the GEMV + AllReduce fused operator; "Bay.Area.AI: Tensor and 2D
 * Parallelism", row-wise sharded linear ending in one all-reduce):
 *
 *     y_s[b][n] = bf16_rne( sum_{r=0}^{R-1} sum_{k<K/R} W_r[n][k] x_r[b][k] )
 *
 * for every rank s, fp32 accumulation, ranks summed in order 0..R-1.
 *   W_r  symmetric bf16 pointer; rank r's N x (K/R) row-major column block,
 *        or a packed weight of this N and K made by symm_pack_w (the same
 *        values in the layout the fused kernel streams fastest; the call's
 *        results are bitwise those of the row-major form).
 *   x_r  symmetric bf16 pointer; rank r's B x (K/R) row-major activations.
 *   y    symmetric bf16 pointer; B x N row-major output, written in every slot.
 *   R    must equal the handle's rank count.
 *   N    output rows (>= 0).   K  TOTAL reduction length: K % R == 0 and
 *        (K/R) % 8 == 0 (rows are read in 16-byte vectors).  K == 0 writes +0.
 *   B    batch columns, 0..SYMM_MAX_BATCH.  N == 0 or B == 0 is a no-op.
 * Requirements: W_r, x_r, y 16-byte aligned inside slot 0's user region; y
 * must not overlap W_r or x_r; 4*B*N <= scratch bytes per slot; the number of
 * row tiles fits the signal pad (else SYMM_ERANGE).
 * Results are deterministic (fixed intra-tile and rank order) and bitwise
 * identical across the R output slots.  Errors: SYMM_EINVAL, SYMM_ERANGE,
 * SYMM_ECUDA; device-side protocol errors via symm_status.
 */
int gemv_all_reduce(symm_handle_t *h, const void *W_r, const void *x_r, void *y, int R, int N,
                    int K, int B, symm_stream_t stream);

/*
 * symm_status -- synchronise `stream`, read the device status word, clear it.
 * (The library's counterpart of a collective watchdog's error report: the
 * "Bay.Area.AI: Tensor and 2D Parallelism" talk describes a watchdog that
 * catches hung collectives and a desync report; here no kernel ever waits, so
 * a protocol violation is recorded and reported instead of hanging.)
 *   code  out: SYMM_OK, or SYMM_EPROTO when a launch found a stale or missing
 *         tile flag or an out-of-range arrival ticket (e.g. two launches on
 *         the handle overlapped on different streams).
 *   rank, tile  out: where it was detected (-1 if none).
 * After an error the signal pad's flags, counters and launch epoch are reset
 * so the handle is usable again (a multi-process handle keeps the epoch, its
 * launch count).  Returns SYMM_OK if the status could be read (whatever
 * `code` says), SYMM_ECUDA otherwise.
 */
int symm_status(symm_handle_t *h, symm_stream_t stream, int *code, int *rank, int *tile);

/*
 * symm_copy_to_slots / symm_copy_from_slots -- stage per-rank data between a
 * contiguous buffer and the symmetric slots in one strided copy (the
 * rendezvous handle's per-peer buffers addressed the same way: rank r's
 * instance of a symmetric pointer p is p + r * stride).  A convenience of
 * this library for feeding the calls above from host memory; the source
 * pages have no counterpart.
 *   to_slots:   dst symmetric pointer; src holds nranks consecutive blocks of
 *               bytes_per_rank; block r goes to dst + r * stride.
 *   from_slots: src symmetric pointer; block r of dst receives
 *               src + r * stride.
 *   The contiguous side may be host memory (pinned for an asynchronous copy)
 *   or device memory.  nranks 0..R; 0 bytes or 0 ranks is a no-op.
 *   Device memory and pinned host memory the GPU addresses at the same
 *   pointer (every pinned allocation on this platform) are copied by a
 *   kernel -- the SMs read or write the host buffer over the CPU-GPU link --
 *   which, like the other calls, chains with its neighbours on the stream
 *   (SYMM_OPT_CHAIN); other host memory, or SYMM_OPT_COPY_ENGINE = 1, takes
 *   one strided copy-engine copy.
 * Stream-ordered; returns after enqueueing.  Errors: SYMM_EINVAL (NULL
 * pointer, nranks out of range, the symmetric side outside slot 0's user
 * region), SYMM_ECUDA.
 */
int symm_copy_to_slots(symm_handle_t *h, void *dst, const void *src, size_t bytes_per_rank, int nranks,
                       symm_stream_t stream);
int symm_copy_from_slots(symm_handle_t *h, void *dst, const void *src, size_t bytes_per_rank, int nranks,
                         symm_stream_t stream);

/*
 * Packed weights -- a second layout for the W_r of the fused calls
 * (gemv_all_reduce, gemv_reduce_scatter, gemv_all_reduce_bias_rmsnorm), made
 * once when the weights are loaded.  The pages fix no layout for the weight
 * shards; this one lets the fused kernel stream each 128-row x 64-column
 * block of W_r as one contiguous 16 KB read instead of 128 rows of 128 bytes
 * (the bytes read per call are the same; measured 1-5 % faster from about 60 MB of W up, and
 * 0.5-2 % slower on a 34 MB one).
 *
 * symm_packed_w_bytes -- bytes per slot of the packed form of an N x (K/R)
 * W_r: (ceil(N/128) * ceil((K/R)/64) + 1) * 16384.  Same K, R rules as
 * gemv_all_reduce.  Errors: SYMM_EINVAL.
 *
 * symm_pack_w -- for every slot r, writes the packed form of the row-major
 * W_r (+ r * stride) into Wp (+ r * stride) and registers Wp with the handle
 * for this N and K.  Layout: block (t, j) covers rows 128t.. and columns
 * 64j.. and sits at byte (t * ceil((K/R)/64) + j) * 16384; inside it, row i
 * starts at i * 128 and its 16-byte chunk c (elements 8c..8c+7) is stored at
 * chunk position c XOR (i mod 8); rows past N and columns past K/R are zero;
 * one all-zero block follows the last.
 *   W_r, Wp  symmetric pointers, 16-byte aligned inside slot 0's user region;
 *            they must not overlap; W_r must not itself be a packed weight.
 * A fused call whose W_r equals a registered Wp reads it packed; it must use
 * the same N and K (else SYMM_EINVAL) and runs on the persistent kernel
 * (SYMM_OPT_GEMV_PATH 0 or 4, else SYMM_EINVAL).  The registration ends with
 * symm_release_w, with a later symm_pack_w whose Wp range overlaps it, or with
 * symm_free; writing other data into Wp does not end it.
 * Stream-ordered (the W_r it reads may be written by earlier work on the
 * stream); returns after enqueueing.  Errors: SYMM_EINVAL, SYMM_ECUDA.
 *
 * symm_release_w -- forget the packed weight registered at Wp (its bytes are
 * untouched; a later fused call with W_r == Wp reads them row-major).
 * Errors: SYMM_EINVAL (no packed weight registered at Wp).
 */
int symm_packed_w_bytes(int R, int N, int K, size_t *bytes_out);
int symm_pack_w(symm_handle_t *h, const void *W_r, void *Wp, int R, int N, int K, symm_stream_t stream);
int symm_release_w(symm_handle_t *h, const void *Wp);

/*
 * symm_check_guards -- verify the guard bands around every slot's user
 * region, scratch region and signal pad (synchronises the device).
 * Returns SYMM_OK, or SYMM_ECORRUPT with *bad_rank / *bad_band set
 * (band 0: after the user region, 1: after scratch, 2: after the pad).
 */
int symm_check_guards(symm_handle_t *h, int *bad_rank, int *bad_band);

/*
 * gemv_reduce_scatter -- the fused row-parallel layer ending in a
 * reduce-scatter instead of an all-reduce: the sequence-parallel form
 * ("Bay.Area.AI: Tensor and 2D Parallelism", sequence-parallel passage: the
 * activations are sharded along the sequence, and after the row-wise sharded
 * linear one reduce-scatter returns each rank its own tokens of the sum).
 * With y_full = bf16_rne( sum_r W_r x_r ) (B x N, as gemv_all_reduce computes
 * it), rank s receives batch rows [s*B/R, (s+1)*B/R):
 *
 *     y_s[i][n] = y_full[s*B/R + i][n]      i < B/R
 *
 *   y  symmetric bf16 pointer; (B/R) x N row-major per slot.
 * B % R == 0 is required (else SYMM_EINVAL); every other argument, layout,
 * requirement and error as for gemv_all_reduce.  Bitwise equal to the rows of
 * gemv_all_reduce's result for the same inputs and options.
 */
int gemv_reduce_scatter(symm_handle_t *h, const void *W_r, const void *x_r, void *y, int R, int N, int K,
                        int B, symm_stream_t stream);

/*
 * gemv_all_reduce_bias_rmsnorm -- the fused layer followed by a bias and RMS
 * normalisation of each batch row's N outputs (the all-reduce + bias + RMSNorm
 * kernel of the "PyTorch Symmetric Memory" talk, fused-kernel segment,
 * applied to the fused GEMV):
 *
 *     z[b][n]   = sum_r (W_r x_r)[b][n] + bias[n]                 (fp32)
 *     y_s[b][n] = bf16_rne( z[b][n] / sqrt(mean_n z[b][n]^2 + eps) * gamma[n] )
 *
 * for every rank s.  The tile reducers store z (fp32) at the top of slot 0's
 * scratch region instead of y; a second kernel (one thread-block cluster per
 * batch row) normalises.  It is launched right after the GEMV on the same
 * stream, as a programmatic dependent unless SYMM_OPT_NORM_PDL is 0.
 *   bias, gamma  symmetric bf16 pointers to N elements (slot 0's copy is
 *                read), 16-byte aligned; NULL means zeros / ones.
 *   eps          >= 0, finite.
 * Requirements beyond gemv_all_reduce: N % 8 == 0, N <= 65536, and the
 * scratch region holds the partials plus 4*B*N bytes of z (else
 * SYMM_ERANGE).  Errors: SYMM_EINVAL, SYMM_ERANGE, SYMM_ECUDA.
 */
int gemv_all_reduce_bias_rmsnorm(symm_handle_t *h, const void *W_r, const void *x_r, const void *bias,
                                 const void *gamma, void *y, int R, int N, int K, int B, float eps,
                                 symm_stream_t stream);

/*
 * reduce_scatter -- out_s[j] = bf16_rne( sum_{r=0}^{R-1} in_r[s*n/R + j] ),
 * j < n/R, for every rank s: each rank keeps its own block of the summed flat
 * tensor ("Bay.Area.AI: Tensor and 2D Parallelism", sequence-parallel
 * passage; the reduce-scatter of the PyTorch Symmetric Memory docs' NCCL
 * symmetric-kernel list).  fp32 accumulation in rank order.
 *   in   symmetric bf16 pointer, n elements; out  symmetric, n/R elements.
 *   n % R == 0; in and out must not overlap; 16-byte aligned.
 * Errors: SYMM_EINVAL, SYMM_ECUDA.
 */
int reduce_scatter(symm_handle_t *h, const void *in, void *out, int R, size_t n, symm_stream_t stream);

/*
 * two_shot_all_reduce -- the same result as one_shot_all_reduce, bit for bit,
 * computed in two phases (PyTorch Symmetric Memory docs, op reference
 * `two_shot_all_reduce_`): rank s reduces only its block of elements
 * [s*c, (s+1)*c) (c = ceil(n/R) rounded up to 8) into its own out, then every
 * rank gathers the other blocks from their owners.  The two phases are two
 * launches on `stream` (stream order is the barrier between them).  in == out
 * (in place, as the docs' op) is allowed; other arguments as for
 * one_shot_all_reduce.
 */
int two_shot_all_reduce(symm_handle_t *h, const void *in, void *out, int R, size_t n, symm_stream_t stream);

/*
 * all_reduce_bias_rmsnorm -- the all-reduce + bias + RMSNorm kernel of the
 * "PyTorch Symmetric Memory" talk (fused-kernel segment: the bias is added in
 * the reduction's element-wise loop and the RMS normalisation follows in the
 * same launch).  For each of `rows` rows of H elements and every rank s:
 *
 *     z[h]    = (sum_{r=0}^{R-1} in_r[h]) + bias[h]               (fp32)
 *     out_s[h] = bf16_rne( z[h] / sqrt(mean_h z[h]^2 + eps) * gamma[h] )
 *
 *   in, out      symmetric bf16 pointers, rows x H row-major; in == out is
 *                allowed, partial overlap is not.
 *   bias, gamma  symmetric bf16 pointers to H elements or NULL (zeros / ones).
 *   rows 0..65535; H % 8 == 0, 8 <= H <= 65536; eps >= 0 finite.
 * One thread-block cluster per row.  Errors: SYMM_EINVAL, SYMM_ECUDA.
 */
int all_reduce_bias_rmsnorm(symm_handle_t *h, const void *in, const void *bias, const void *gamma, void *out,
                            int R, int rows, int H, float eps, symm_stream_t stream);

/*
 * tile_reduce -- sum a 2-D tile over all ranks into the root's output tile
 * (PyTorch Symmetric Memory docs, op reference `tile_reduce`, reduce op
 * "sum"; the talk's tile-communication segment):
 *
 *     out_root[a][c] = bf16_rne( sum_{r=0}^{R-1} in_r[a][c] )   a < rows, c < cols
 *
 * where element (a, c) of a tile is at tile + (a * ld + c) * 2 bytes, i.e. a
 * rows x cols block of a row-major tensor with leading dimension ld
 * (elements), not contiguous.  Only the root's output tile is written.
 *   in_tile, out_tile  symmetric bf16 pointers (2-byte aligned; rows whose
 *                      starts are all 16-byte aligned use 16-byte loads);
 *                      they must not overlap.
 *   ld_in, ld_out >= cols.  rows == 0 or cols == 0 is a no-op.
 * Errors: SYMM_EINVAL, SYMM_ECUDA.
 */
int tile_reduce(symm_handle_t *h, const void *in_tile, void *out_tile, int root, int rows, int cols,
                long long ld_in, long long ld_out, symm_stream_t stream);

/*
 * multi_root_tile_reduce -- several tiles at once, tile i summed over all
 * ranks into the output tile of rank roots[i] (PyTorch Symmetric Memory docs,
 * op reference `multi_root_tile_reduce`: no rank is root of two tiles).  All
 * tiles have the same shape and leading dimension; the output tile is the
 * same symmetric address for every root.  One launch.
 *   in_tiles [ntiles] host array of symmetric pointers; roots [ntiles] host
 *   array of distinct ranks; 1 <= ntiles <= R.  Otherwise as tile_reduce.
 */
int multi_root_tile_reduce(symm_handle_t *h, const void *const *in_tiles, void *out_tile, const int *roots,
                           int ntiles, int rows, int cols, long long ld_in, long long ld_out,
                           symm_stream_t stream);

/* Per-handle options.  The kernel choice is automatic by default; the
 * others exist for tests and measurements. */
enum {
    SYMM_OPT_GEMV_PATH = 1,   /* 0 auto: 4 when K > 0 and W_r of all ranks is over 24 MB or B > 4; else 5
                                 when R <= 8, B <= 4 and its CTAs (R x ceil(N / 16)) times B are at most
                                 512, else 4; 1 where 5 cannot run (R > 8, a multi-process handle) and
                                 for K = 0.  1 CUDA-core kernel, one CTA per (row
                                 tile, rank); 4 persistent kernel drawing (tile, rank) units from a work
                                 counter; 5 cluster kernel for small layers, one thread-block cluster of R
                                 CTAs per 16-row tile, the partials exchanged through distributed shared
                                 memory (R <= 8, B <= 4, else SYMM_EINVAL; it uses no scratch and no
                                 signal pad).  2 and 3 (a tensor-core kernel per tile and a static
                                 stream-K partition) were retired: neither won on any shape measured;
                                 they return SYMM_EINVAL */
    SYMM_OPT_TILE_ORDER = 2,  /* 0 natural CTA order, 1 reversed (tests arrival-order independence; the
                                 cluster epilogue, which has no arrival order, ignores it) */
    SYMM_OPT_SK_SLABS = 3,    /* path 4: 64-column slabs per pipeline stage, 0 auto (2), 1..4 (the
                                 instantiated pipelines: 1, 2, 4 slabs at 1 CTA per SM; 1, 2, 3 at 2; 1 at 3) */
    SYMM_OPT_SK_ENGINE = 4,   /* path 4: -1 auto or 0, both the tcgen05 engine; 1 (a CUDA-core engine) was
                                 retired, having won on no shape measured, and returns SYMM_EINVAL */
    SYMM_OPT_SK_CTAS_PER_SM = 5, /* path 4: CTAs per SM the ring is sized for, 0 auto (2), 1..3 (the ring
                                 shrinks).  By its registers the kernel holds fewer CTAs per SM than 3:
                                 at 3 the grid runs in two waves, correctly but slower */
    SYMM_OPT_SK_GRID = 6,     /* path 4: persistent grid, 0 auto (CTAs per SM x SMs) or a CTA count */
    SYMM_OPT_DYN_SPLITS = 7,  /* persistent kernel: K splits per (tile, rank), 0 auto, 1..16 */
    SYMM_OPT_NORM_PDL = 8,    /* gemv_all_reduce_bias_rmsnorm: 1 (default) launches the RMSNorm stage as a
                                 programmatic dependent of the GEMV so its launch overlaps the GEMV's
                                 tail; 0 plain stream order */
    SYMM_OPT_CHAIN = 9,       /* 1 (default): every kernel of this library is launched as a programmatic
                                 dependent of the previous kernel on the stream, so back-to-back calls
                                 overlap one call's start-up with the previous call's end; each lets its
                                 successor be scheduled early.  A chained kernel reads nothing before its
                                 predecessor has finished, with two exceptions: the persistent fused
                                 kernel (path 4) loads a packed weight (symm_pack_w) for its first stages
                                 early (a row-major W_r is loaded after the wait, like x), and the
                                 standalone all-reduce + bias + RMSNorm loads gamma and bias early.  Such
                                 a call is launched in plain stream order when those operands overlap
                                 the output of the last call on the same handle (any call, symm_pack_w
                                 included).  A packed weight is written by symm_pack_w only; gamma and
                                 bias must not be written by any other kernel launched just before the
                                 call on the stream.  0: plain stream order always */
    SYMM_OPT_AR_CTAS_PER_SM = 10, /* one_shot_all_reduce (per-thread kernel), two_shot_all_reduce,
                                 reduce_scatter: grid cap in CTAs (256 threads) per SM, grid-stride beyond
                                 it; 0 auto (16) */
    SYMM_OPT_AR_KERNEL = 11,  /* one_shot_all_reduce: 0 auto (= 1), 1 per-thread 16-byte loads and
                                 stores, 2 staged: each CTA reduces a contiguous range chunk by chunk in
                                 shared memory, moved in and out by bulk (TMA) copies (measured slower
                                 than 1 from 0.5 MB per rank up) */
    SYMM_OPT_COPY_ENGINE = 12, /* symm_copy_to_slots / from_slots: 0 (default) copy with a kernel when the
                                 contiguous side is device memory or pinned host memory mapped at the same
                                 address (a link in the chain of programmatic dependent launches, see
                                 SYMM_OPT_CHAIN), else with the copy engine; 1 always the copy engine */
    SYMM_OPT_UNFUSED = 13,    /* gemv_all_reduce only, for measuring what fusion buys: 1 runs the call
                                 unfused, as two kernels -- the persistent GEMV (path 4) storing every
                                 rank's fp32 partials, then a separate all-reduce kernel that sums them in
                                 the fused reducer's order and stores bf16 into every slot (the same
                                 bits as the fused call); 0 (default) fused.  The other forms, path 1
                                 and K == 0 return SYMM_EINVAL while it is set */
    SYMM_OPT_DYN_CLUSTER = 14 /* path 4, the end of a launch: -1 auto (default), 0 off, 1 on.  On: the
                                 launch is a grid of thread-block clusters of R CTAs, one (row tile, rank)
                                 unit per CTA, the R units of a tile in one cluster; each CTA keeps its
                                 fp32 partial in its own shared memory, and after a cluster barrier every
                                 CTA sums its share of the tile over the R partials (read through
                                 distributed shared memory, rank order, the same bits as the global-memory
                                 protocol) and stores it.  With K splits (SYMM_OPT_DYN_SPLITS, honoured
                                 when it is forced on) a cluster holds the R x splits units of a tile.  It
                                 needs 2 CTAs per SM, R x splits <= 8, the fused
                                 form, a single-process handle and a device that can hold such a cluster
                                 (else 1 returns SYMM_EINVAL).  Auto, where those hold: for R <= 4 whose
                                 (tile, rank) units fill at most half of the persistent grid, it splits
                                 K inside the clusters (R x splits <= 8) as far as one wave holds (with
                                 SYMM_OPT_DYN_SPLITS unset; R = 1 too, the splits then being the
                                 cluster); otherwise, for R >= 2 without K splits, it turns it on when
                                 the units fit the grid in one wave (nothing would be drawn) or are long
                                 (K/R >= 3072, 768 KB of W per unit), when the hardware's scheduling of
                                 whole clusters beats drawing single units */
};
int symm_set_option(symm_handle_t *h, int option, int value);

/* Capacities of the handle: ranks, user/scratch/pad bytes per slot, and the
 * number of row tiles the signal pad can hold. */
typedef struct {
    int R;
    int device;
    size_t stride, slot_bytes, scratch_bytes, signal_pad_bytes;
    int max_tiles;
} symm_info_t;
int symm_info(symm_handle_t *h, symm_info_t *info);

/* The kernel and launch geometry gemv_all_reduce would use for (N, K, B) on
 * this handle with a row-major W_r, without launching anything (SYMM_EINVAL /
 * SYMM_ERANGE exactly as the call would return them).  A call on a packed
 * weight (symm_pack_w) runs path 4 with the plan reported while
 * SYMM_OPT_GEMV_PATH is 4.
 *   path           1 CUDA-core per tile, 4 persistent dynamic, 5 cluster per tile
 *   engine         path 4 compute engine: 0 (tcgen05)
 *   slabs          path 4: 64-column slabs per pipeline stage
 *   rows_per_tile  output rows per tile; tiles = ceil(N / rows_per_tile)
 *   splits         K-splits per rank (path 4)
 *   grid           CTAs launched
 *   parts_max      1 (kept for layout compatibility)
 *   kblocks        path 4: K blocks per (tile, rank)
 *   ctas_per_sm    path 4: resident CTAs per SM the ring is sized for
 *   cluster        CTAs per thread-block cluster: R on path 5 and for path 4's
 *                  cluster epilogue (SYMM_OPT_DYN_CLUSTER), else 0 */
typedef struct {
    int path, engine, slabs, rows_per_tile, tiles, splits, grid, parts_max, kblocks, ctas_per_sm, cluster;
} symm_gemv_plan_t;
int symm_gemv_plan(symm_handle_t *h, int N, int K, int B, symm_gemv_plan_t *out);

/*
 * gemv_all_reduce_noalloc -- the fused GEMV + one-shot all-reduce for callers
 * that cannot allocate device memory: code whose device memory is owned by
 * another allocator (a framework's caching allocator, a serving process with
 * a fixed memory budget), or that runs on a hot path where cudaMalloc's
 * implicit synchronisation is not allowed.  Such a caller cannot create a
 * handle, because symm_alloc allocates.
 *
 * The source pages have no counterpart of this call; it is an addition of
 * this library.
 *
 * Same result as gemv_all_reduce (y_s = bf16_rne(sum_r W_r x_r), fp32
 * accumulation, ranks summed in order 0..R-1, every rank's y written), on
 * tensors the caller owns: rank r's W_r, x_r and y are at W_r + r * stride,
 * x_r + r * stride and y + r * stride (bytes).  Layouts as for
 * gemv_all_reduce; pointers and stride 16-byte aligned; no instance of y may
 * overlap an instance of W_r or x_r.  R in 1..64, B in 0..16, K % R == 0,
 * (K/R) % 8 == 0; N == 0 or B == 0 is a no-op.
 *
 * Working memory: a fixed 16 MiB device array inside this library (present
 * on every GPU that loads the library until the process exits).  It holds the
 * fp32 partials of all ranks (4 * R * B * N bytes, rounded up to 256) plus one
 * 4-byte counter per row tile; larger problems return SYMM_ERANGE.  No
 * cudaMalloc, cudaFree or allocating library call is made.
 *
 * Every call on a device shares that array and it keeps the last call's
 * contents (the counters are cleared by a stream-ordered memset at the start
 * of each call).  Calls that overlap on the GPU race on the array: issue them
 * on one stream.  The first call on each device, with that device current,
 * looks up the array's address (cudaGetSymbolAddress); make that first call
 * before any stream capture.
 *
 * Returns SYMM_OK after enqueueing, SYMM_EINVAL, SYMM_ERANGE or SYMM_ECUDA.
 */
int gemv_all_reduce_noalloc(const void *W_r, const void *x_r, void *y, size_t stride, int R, int N, int K,
                            int B, symm_stream_t stream);

/*
 * symm_set_timeline -- diagnostics: register a device buffer that the
 * kernels of later calls on this handle fill with per-CTA %globaltimer
 * stamps at their phase boundaries (one row of 16 unsigned 64-bit words per
 * CTA, row = the CTA's linear index; which slot holds which phase is listed
 * in each kernel's source).  Only the timeline build of this library
 * (-DSYMM_TIMELINE) writes stamps; the product build returns SYMM_EINVAL for a
 * non-NULL buffer.  CTAs whose row does not fit in `bytes` write nothing.
 * buf == NULL (or bytes == 0) switches the timeline off.  The buffer is
 * borrowed: it must stay valid while calls that may write it run.  No counterpart on the pages.
 */
int symm_set_timeline(symm_handle_t *h, void *buf, size_t bytes);

/* Release the handle; frees owned memory (synchronises the device first). */
int symm_free(symm_handle_t *h);

/* Last error message of the calling thread ("" if none). */
const char *symm_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SYMM_GEMV_H */
