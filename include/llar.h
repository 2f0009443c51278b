/*
 * llar: low-latency sum AllReduce over N virtual ranks on one GPU.
 *
 * C ABI. Every argument is a plain pointer, size or integer; no framework
 * types cross this boundary. A `stream` argument is a cudaStream_t passed
 * as `void*` (NULL = the legacy default stream).
 *
 * The operation, from the pages this library restates:
 *  - AllReduce: afterwards every rank holds the complete aggregated result
 *    ("zcube network architecture for LLM inference", collectives table,
 *    All-Reduce row); in tensor parallelism the aggregation is the sum of
 *    the ranks' partial outputs (same page, "Why does Tensor Parallel
 *    affect every token").
 *  - One-shot, or two-shot = ReduceScatter then AllGather ("Every
 *    Microsecond Matters: Achieving Near Speed-of-Light Latency in GPU
 *    Collectives", summary page, technique 4).
 *  - Signalling without a global memory barrier (same page, techniques
 *    1-4: LL flag-in-data, sentinel, bidirectional double buffering,
 *    two-shot LL128 atomics).
 *
 * Virtual ranks: rank r is a group of CTAs of one persistent kernel, with
 * its own input, output and staging buffers in device memory; ranks signal
 * each other through L2 with relaxed/acquire/release loads, stores and
 * reductions at GPU scope.
 *
 * Numerics: every fixed-order protocol (LL, SENTINEL, FIXED_*) adds the
 * ranks in order 0..N-1 in float32 and rounds once (roundTiesToEven) to the
 * element type, so its result is bit-identical to that definition.
 * LL128_ATOMIC adds with floating-point atomics in the element type in
 * arrival order; its result is not deterministic (technique 4 says so).
 * Its bound: per element, |result - rank-order sum| <= (N-1) ulp of the
 * element type at sum_r |x_r|, with two limits:
 *  - float32: the GPU's float32 atomic add reads a subnormal operand as
 *    zero and returns zero for a subnormal result, so on subnormal data the
 *    error can grow by up to 2 N 2^-126 (an all-subnormal column sums to
 *    +0); fp16 and bf16 use the non-flushing (.noftz) atomics;
 *  - fp16 / bf16: every partial sum is rounded in the element type, so the
 *    bound holds while sum_r |x_r| <= max - N ulp(max) / 2 (fp16 at 8
 *    ranks: 65376); beyond it, with cancelling values, a partial sum can
 *    overflow to an infinity where the float32 sum is finite (in the
 *    arrival orders that add same-signed values first).
 *
 * Errors: calls return an llar_status_t. Invalid arguments are rejected
 * before any device work. Every device-side wait is bounded by a timeout
 * (llar_set_timeout_ns); a wait that runs out records LLAR_ERR_TIMEOUT
 * with the rank, CTA and epoch in a status word, the kernel returns, and
 * every later call reports LLAR_ERR_TIMEOUT until llar_reset().
 *
 * Concurrency: one process-global context. Calls on it must be ordered
 * (one stream, or streams ordered by events): two of its kernels running
 * at once would share staging and race.
 */
#ifndef LLAR_H
#define LLAR_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { LLAR_F32 = 0, LLAR_F16 = 1, LLAR_BF16 = 2 } llar_dtype_t;

typedef enum {
  LLAR_PROTO_AUTO = 0,          /* measured choice per call kind, rank count and size:
                                   llar_select_protocol (and _iters, _segment, _host);
                                   a nondeterministic protocol only after
                                   llar_set_auto_nondeterministic(1) */
  LLAR_PROTO_LL = 1,            /* one-shot, 8 B data + 8 B flag per 16 B line (technique 1) */
  LLAR_PROTO_SENTINEL = 2,      /* one-shot, -NaN prefilled staging, chunked and
                                   double-buffered with implicit credits (techniques 2, 3) */
  LLAR_PROTO_LL128_ATOMIC = 3,  /* two-shot, atomic ReduceScatter into 128 B lines with a
                                   count flag, LL AllGather (technique 4); nondeterministic */
  LLAR_PROTO_FIXED_ONESHOT = 4, /* one-shot, every rank reads all inputs directly */
  LLAR_PROTO_FIXED_TWOSHOT = 5, /* two-shot, owner of each segment reads all inputs
                                   directly and writes every rank's output */
  LLAR_PROTO_LL128_DIRECT = 6   /* two-shot as LL128_ATOMIC, but every rank reads the
                                   reduced data straight from the owners' 128 B lines once
                                   their count reads N (three line slots in turn) instead
                                   of an LL AllGather; nondeterministic, same bound */
} llar_proto_t;

typedef enum {
  LLAR_OK = 0,
  LLAR_ERR_INVALID = 1,     /* bad argument (null/misaligned pointer, aliasing, bad rank count) */
  LLAR_ERR_NOT_INIT = 2,    /* no context (llar_init not called, or destroyed) */
  LLAR_ERR_TOO_LARGE = 3,   /* count * element size exceeds the staging sized at init */
  LLAR_ERR_UNSUPPORTED = 4, /* dtype/protocol/mode combination not provided */
  LLAR_ERR_OCCUPANCY = 5,   /* the N x G CTAs cannot all be resident at once */
  LLAR_ERR_CUDA = 6,        /* a CUDA runtime call failed (no device, out of memory, ...) */
  LLAR_ERR_TIMEOUT = 7      /* a device-side wait ran out; see llar_get_status */
} llar_status_t;

typedef enum {
  LLAR_INJECT_NONE = 0,
  LLAR_INJECT_SKIP_PUSH = 1, /* the chosen rank never sends: its peers' waits run out */
  LLAR_INJECT_POISON = 2,    /* the chosen rank sends lines whose signal never completes */
  LLAR_INJECT_DELAY = 3      /* the chosen rank sleeps ~20 us before each send; results stay exact */
} llar_inject_t;

/* Create the context: `nranks` virtual ranks (2..8), element type `dtype`
 * (llar_dtype_t), messages up to `max_bytes` per rank. Allocates and
 * initialises all staging (LL lines zeroed, sentinel slots filled with the
 * all-ones -NaN pattern, LL128 lines zeroed), the epoch counter and the
 * status word, and chooses the LL placement (llar_ll_placement). Tuning
 * variables of the environment (LLAR_CTAS_PER_RANK, LLAR_THREADS,
 * LLAR_CLUSTER, LLAR_BULK, LLAR_BULK_MIN_BYTES, LLAR_PDL, LLAR_COOP,
 * LLAR_SPREAD_SMEM, LLAR_CHUNK_BYTES, LLAR_LL_MAX_BYTES,
 * LLAR_LL128_MAX_BYTES, LLAR_LOG, LLAR_TUNE) are read
 * here: each context sees the environment as it is at its init, an unset
 * variable meaning the built-in default. LLAR_COOP=0 launches the kernels
 * whose CTAs wait on each other without the cooperative attribute: cheaper
 * per call outside CUDA graphs (8 x 16 KiB bf16 LL queued from C: 5.0 ->
 * 3.1 us of GPU time a call; in a graph no gain), the grid still sized to
 * fit the GPU at once;
 * but the launch is then not held back while other kernels occupy SMs, so
 * its waits can run out (LLAR_ERR_TIMEOUT) if the library's launches
 * overlap other kernels. Default 1 (cooperative). Returns LLAR_ERR_INVALID for a
 * second init without llar_destroy, LLAR_ERR_CUDA if no device or memory
 * is available. */
int llar_init(int nranks, int dtype, size_t max_bytes);

/* Free everything llar_init allocated. Synchronises the device first. */
int llar_destroy(void);

/* One AllReduce. in[r] / out[r] (host arrays of N device pointers, copied
 * at call time) are rank r's input and output, each `count` elements,
 * 16-byte aligned, owned by the caller. out[r] must not alias any in[q].
 * On return the work is queued on `stream`; out[r] holds the sum of all
 * in[q] once the stream reaches it. count == 0 is a no-op. protocol: an
 * llar_proto_t; LLAR_PROTO_AUTO follows llar_select_protocol. */
int llar_allreduce(const void* const* in, void* const* out, size_t count,
                   int protocol, void* stream);

/* `iters` AllReduces back to back inside ONE persistent launch, with no
 * barrier between iterations (technique 3). Iteration e writes
 * out[r] + e*out_stride_elems. Its input is in[r] + e*in_stride_elems, or,
 * when chain_scale != 0 (a chain of dependent AllReduces, as across the
 * layers of one decode step), in[r] for e == 0 and afterwards
 * roundTiesToEven(chain_scale * output of e-1), kept in library memory.
 * The output of iteration e is identical to llar_allreduce on that input.
 * LLAR_PROTO_AUTO follows llar_select_protocol_iters. */
int llar_allreduce_iters(const void* const* in, void* const* out, size_t count,
                         int protocol, int iters, size_t in_stride_elems,
                         size_t out_stride_elems, float chain_scale, void* stream);

/* ReduceScatter, the first half of the two-shot AllReduce ("zcube network
 * architecture for LLM inference", collectives table, Reduce-Scatter row:
 * after it each rank keeps one reduced segment). Segment s of the
 * count-element vector is [s*S, min(count, (s+1)*S)), S = ceil(count/N).
 * in[r]: count elements; out[r]: the S (or fewer) elements of segment r,
 * = sum over q of in[q][segment r], added in rank order in float32 and
 * rounded once. protocol: LLAR_PROTO_LL (flag-in-data lines),
 * LLAR_PROTO_SENTINEL (raw vectors into all-ones slots; a segment must fit
 * one sentinel chunk, else LLAR_ERR_TOO_LARGE), LLAR_PROTO_FIXED_ONESHOT
 * (direct reads), LLAR_PROTO_LL128_ATOMIC (technique 4's atomic
 * reductions into 128-byte lines with a count flag: element-type
 * additions in arrival order, within (N-1) ulp of the sum of |x|) or
 * LLAR_PROTO_AUTO (llar_select_protocol_segment); others give
 * LLAR_ERR_UNSUPPORTED. One collective per launch. */
int llar_reduce_scatter(const void* const* in, void* const* out, size_t count,
                        int protocol, void* stream);

/* AllGather, the second half of the two-shot AllReduce (same table,
 * All-Gather row: each rank collects every rank's segment). in[r]: segment
 * r of a count-element vector (segments as for llar_reduce_scatter);
 * out[r]: all count elements, segment q at offset q*S. Protocols as for
 * llar_reduce_scatter except LLAR_PROTO_LL128_ATOMIC (nothing is added in
 * an AllGather: LLAR_ERR_UNSUPPORTED). With LLAR_PROTO_FIXED_ONESHOT
 * rank r's CTAs copy segment r into every output (16-byte vectors when
 * S * element size is a multiple of 16, elements otherwise). */
int llar_all_gather(const void* const* in, void* const* out, size_t count,
                    int protocol, void* stream);

/* Point-to-point transfers between virtual ranks (a pipeline-parallel
 * stage hand-off; "Every Microsecond Matters", summary page: the LL and
 * sentinel signalling, double-buffered). Rank r sends `count` elements of
 * the context's type from send[r] to rank dst[r] (dst: host array of N
 * ints, -1 = rank r sends nothing; dst[r] != r; every rank receives from at
 * most one sender) into recv[dst[r]]. `iters` >= 1 transfers run back to
 * back in one launch; transfer e reads send[r] + e*send_stride and writes
 * recv[q] + e*recv_stride (strides in elements, 16-byte multiples; 0 =
 * the same buffers). The receiver of each CTA's share acknowledges it
 * after consuming it, and the sender waits for that before reusing the
 * slot two transfers later (a one-way flow has no returning data to act
 * as the credit). protocol: LLAR_PROTO_LL (count * elem <= the LL
 * capacity, 1 MiB by default), LLAR_PROTO_SENTINEL (chunked; data must not
 * contain the all-ones element pattern), LLAR_PROTO_FIXED_ONESHOT (direct
 * reads: the receiver's CTAs copy the sender's buffer, made ready by
 * stream order; nothing is signalled) or LLAR_PROTO_AUTO (the direct
 * copy: measured faster than LL and the sentinel at every size from 512 B
 * to 8 MiB, 2 to 8 ranks, one GPU). Pointers of ranks that neither send (send) nor receive (recv)
 * may be NULL; the others are device pointers, 16-byte aligned, and no
 * receive span overlaps a send span or another receive span. The result
 * is a bit copy. Asynchronous; status codes as llar_allreduce. */
int llar_sendrecv(const void* const* send, void* const* recv, const int* dst, size_t count,
                  int protocol, int iters, size_t send_stride, size_t recv_stride, void* stream);

/* One AllReduce on HOST buffers: in_host and out_host are [N][count]
 * contiguous arrays in host memory. If both are page-locked and
 * device-addressable (cudaHostAlloc / cudaHostRegister memory under
 * unified addressing) and count * element size is a multiple of 16, the
 * kernel reads the inputs and writes the outputs across the bus directly
 * (one launch, no staging copies); there LLAR_PROTO_AUTO follows
 * llar_select_protocol_host, not llar_select_protocol. Otherwise the call
 * copies in, runs and copies out on `stream` through device buffers the
 * library allocates on first use. Returns once the work is queued
 * (synchronise the stream before reading out_host). */
int llar_allreduce_host(const void* in_host, void* out_host, size_t count,
                        int protocol, void* stream);

/* Register a page-locked host buffer that the device can address (from
 * cudaHostAlloc, or torch's pin_memory) of `bytes` bytes with the context:
 * llar_allreduce_host calls whose input and output each lie inside a
 * registered buffer take its device address from this table instead of
 * querying the pointers' attributes on every call. (No page describes it;
 * it trims the host cost of the host-buffer entry.) The caller must
 * unregister a buffer before freeing it: a freed and reused address left in
 * the table would hand the kernel memory it cannot reach. At most 64
 * buffers, none overlapping another. LLAR_ERR_NOT_INIT without a context
 * (llar_destroy drops the table); LLAR_ERR_INVALID for NULL, zero bytes, an
 * overlap, a full table, or memory that is not page-locked and
 * device-addressable. Synchronous; no device work. */
int llar_host_register(const void* ptr, size_t bytes);

/* Remove the buffer registered at `ptr` (the address given to
 * llar_host_register). LLAR_ERR_INVALID if none is; LLAR_ERR_NOT_INIT
 * without a context. */
int llar_host_unregister(const void* ptr);

/* The status word written by the device: LLAR_OK, or LLAR_ERR_TIMEOUT with
 * the virtual rank, CTA and epoch of the first wait that ran out. Any
 * pointer may be NULL. Reads the word without synchronising. */
int llar_get_status(int* rank, int* cta, unsigned long long* epoch);

/* Refill sentinel staging, zero LL and LL128 staging and the abort flag,
 * clear the status word; epochs keep counting. Synchronises the device. */
int llar_reset(void* stream);

/* Bound on every device-side wait, in nanoseconds (default 1e9). */
void llar_set_timeout_ns(unsigned long long ns);

/* Force CTAs per rank and threads per CTA for later launches (0 = choose
 * automatically). threads must be a multiple of 32, at most 512. */
int llar_set_launch(int ctas_per_rank, int threads);

/* Sentinel chunk size in bytes per rank (multiple of 16, at most 64 KiB;
 * default 64 KiB): each call moves ceil(bytes / chunk) chunks through the
 * two staging slots of every peer (technique 3). */
int llar_set_sentinel_chunk(size_t bytes);

/* Host-controlled fault injection on virtual rank `rank` (llar_inject_t);
 * LLAR_INJECT_NONE switches it off. No GPU fault is ever raised: the
 * affected waits end through their timeout. */
int llar_debug_inject(int rank, int mode);

/* Speed-of-light latency of one AllReduce on this GPU, measured as the
 * pages define it ("Every Microsecond Matters", summary page, the
 * speed-of-light paragraph: 2 x L2 round trip + one remote write).
 * l2_rt_us: median dependent-load latency of a pointer chase over a 16 MB
 * buffer resident in L2, one chasing thread per SM; write_us: half the
 * median round trip of a store-to-observe ping-pong between CTA pairs on
 * different SMs; sol_us = 2 * l2_rt_us + write_us. Needs llar_init. */
int llar_sol_probe(double* l2_rt_us, double* write_us, double* sol_us);

/* The same bound over the rank CTAs a launch actually places, at the
 * worst pair. A probe grid shaped like the most recent AllReduce launch
 * (N x G blocks, its threads, shared memory, cluster and cooperative
 * attributes) records the SM of every block; block c of every two ranks
 * (the blocks that exchange data) ping-pong in rounds of disjoint pairs.
 * l2_rt_us: the slowest pointer-chase latency (as in llar_sol_probe) among
 * the SMs that hold the blocks; write_us: half the slowest pair's round
 * trip; sol_us = 2 * l2_rt_us + write_us; npairs: pairs measured. Needs
 * llar_init and an AllReduce launched since (LLAR_ERR_INVALID otherwise).
 * Synchronises the device. */
int llar_sol_probe_placed(double* l2_rt_us, double* write_us, double* sol_us, int* npairs);

/* LL placement chosen for this context (diagnostic; no page describes
 * it): *clustered = 1 if LL launches of 16 or more AllReduces of up to
 * 16 KiB per rank (the size timed) run in clusters of N blocks (the CTAs
 * that exchange a word range on one GPC), 0 if not. llar_init times both
 * on this GPU (a few hundred 16 KiB AllReduces each, a few milliseconds)
 * and keeps clusters only if they are at least 3 % faster: which placement
 * is faster differs between GPUs of the same model. LLAR_TUNE=0, or a fault injection (llar_debug_inject)
 * active at llar_init, skips the timing (no clusters); LLAR_CLUSTER = 0 or
 * 2 forces it. Results are identical either way. */
int llar_ll_placement(int* clustered);

/* The speed-of-light bound itself (host only): 2 * l2_rt_us + write_us. */
double llar_sol_bound_us(double l2_rt_us, double write_us);

/* The raw measurements behind llar_sol_probe. Arrays hold at least 256
 * (chase) and 128 (pairs) entries. chase_ns[i]: ns per dependent load of
 * the chasing thread on SM chase_smid[i]; rt_ns[k]: ns per round trip of
 * pair k between SMs smid_a[k] and smid_b[k] (0 if its wait ran out). */
int llar_sol_probe_detail(double* chase_ns, int* chase_smid, int* nchase, double* rt_ns,
                          int* smid_a, int* smid_b, int* npairs);

/* Location of a protocol's staging (for state checks): base device
 * pointer, bytes between consecutive ranks' regions, and bytes used per
 * rank. For LLAR_PROTO_LL128_ATOMIC this is the line staging only. */
int llar_staging(int protocol, void** dev_ptr, size_t* rank_stride_bytes,
                 size_t* rank_bytes);

/* Host-only layout query (no device needed): bytes per signalling line,
 * data elements per line, and staging bytes per rank that `protocol`
 * needs for `count` elements of `dtype` over `nranks` ranks. */
int llar_layout(int protocol, int dtype, int nranks, size_t count,
                size_t* line_bytes, size_t* payload_elems_per_line,
                size_t* staging_bytes_per_rank);

/* The protocol LLAR_PROTO_AUTO picks for one AllReduce (llar_allreduce) of
 * this rank count and size (host-only). Measured per rank count on a B300
 * (graph-replayed single calls): a single call pays LL's cooperative
 * launch and epoch exchange, which the direct-read one-shot does not, so
 * the one-shot takes small messages with 2, 3, 5 and 6 ranks, LL those up
 * to 64 KiB per rank with 4 ranks and up to 32 KiB with 7-8; the one-shot
 * then runs up to 1 MiB (2-3 ranks), 256 KiB (4), 128 KiB (5), 64 KiB (6),
 * and the direct-read two-shot above, streamed through shared memory with
 * TMA bulk copies from 1 MiB (3-4 ranks), 512 KiB (5) or 32 KiB (6-8),
 * never for 2. LLAR_PROTO (environment) forces a protocol. */
int llar_select_protocol(int nranks, int dtype, size_t count);

/* The protocol LLAR_PROTO_AUTO picks for llar_allreduce_iters (host-only;
 * with the default 1 MiB LL capacity, the context's own in a call). With
 * iters == 1, llar_select_protocol. A chain (`chained` != 0) takes LL up to
 * the LL capacity, with 7-8 ranks up to 512 KiB per rank, and the
 * direct-read two-shot beyond (8 x 64 KiB bf16 chained: LL 1.41 us per
 * AllReduce against 11.7 for the two-shot); independent AllReduces back
 * to back take LL up to 256 KiB per rank (2 ranks), 128 KiB (3-4), 64 KiB
 * (5-8), the one-shot up to 1 MiB (2-3), 512 KiB (4), 256 KiB (5), and the
 * two-shot above.
 * Deterministic protocols only, unless `nondeterministic` != 0 (what
 * llar_set_auto_nondeterministic(1) gives a context): then chains take the
 * LL128 direct form where it measured fastest, 5-8 ranks at 512 KiB per
 * rank, 8 ranks from 256 KiB, 5-6 ranks above 512 KiB (8 x 256 KiB bf16
 * chained: 4.2 us per AllReduce against 5.6 for LL, 11.9 for the
 * two-shot). LLAR_PROTO (environment) forces a protocol. LLAR_PROTO_AUTO
 * for invalid arguments. */
int llar_select_protocol_iters(int nranks, int dtype, size_t count, int iters, int chained,
                               int nondeterministic);

/* Let LLAR_PROTO_AUTO pick the LL128 direct protocol where it measured
 * fastest (llar_select_protocol_iters with nondeterministic = 1): its
 * atomic additions make the result depend on arrival order, within the
 * (N-1)-ulp bound of the LL128 protocols instead of bit-exact. allow: 0
 * (the default at llar_init) or 1; LLAR_ERR_NOT_INIT without a context,
 * LLAR_ERR_INVALID otherwise. (The pages name the atomic protocol's
 * nondeterminism; the switch is this library's.) */
int llar_set_auto_nondeterministic(int allow);

/* The protocol LLAR_PROTO_AUTO picks for llar_reduce_scatter
 * (reduce_scatter != 0) or llar_all_gather of `count` elements (host-only).
 * Measured per rank count on a B300 (one call per launch, 2..8 ranks,
 * 1 KiB .. 64 MiB): the direct copies (LLAR_PROTO_FIXED_ONESHOT) at every
 * size for both (8 x 16 KiB bf16: ReduceScatter 1.7 us against 4.0 for
 * LL, AllGather 1.6 against 2.7). LLAR_PROTO (environment) forces a
 * protocol.
 * LLAR_PROTO_AUTO for an invalid rank count or dtype. */
int llar_select_protocol_segment(int reduce_scatter, int nranks, int dtype, size_t count);

/* The protocol LLAR_PROTO_AUTO picks when llar_allreduce_host reads and
 * writes host memory directly (host-only). (No page describes it.) The
 * bus sets the cost there: LL up to 4 KiB per rank (a single call answers
 * ~1 us sooner), the direct-read two-shot above (8 x 16 KiB bf16: 7.1-7.4
 * us per call back to back against 8.3-10.1 for LL). LLAR_PROTO
 * (environment) forces a protocol. LLAR_PROTO_AUTO for an invalid rank
 * count or dtype. */
int llar_select_protocol_host(int nranks, int dtype, size_t count);

/* Epoch the next launch will use for its first AllReduce; strictly
 * increasing, never reset. The counter lives in device memory (each launch
 * advances it when its last CTA finishes), so launches captured in a CUDA
 * graph get fresh epochs on every replay. Synchronises the device to read it. */
unsigned long long llar_epoch(void);

/* Launch shape of the most recent launch of this context (llar_init clears
 * it): protocol used, CTAs per rank, threads per CTA, iterations. Any
 * pointer may be NULL. */
int llar_last_launch(int* protocol, int* ctas_per_rank, int* threads, int* iters);

/* Diagnostic, host arithmetic only (no GPU work, no llar_init needed; no
 * page describes it: it exposes the launch-shape rule to tests). The shape
 * (CTAs per rank, threads per CTA) the runtime picks for a call of `count`
 * elements per rank with `nranks` ranks (2..8), element type `dtype` and
 * `protocol` (LLAR_PROTO_LL .. LLAR_PROTO_LL128_DIRECT, not AUTO), for
 * `chained` = 0: several AllReduces in one launch without a chain, 1: a
 * chain (llar_allreduce_iters with a chain scale), 2: one AllReduce per
 * launch (llar_allreduce; the fixed-order paths take a shape of their own
 * there),
 * on a GPU with `sms` SMs and sentinel chunks of `chunk_bytes` (16 ..
 * 65536, a multiple of 16). It is the shape before a launch applies the
 * GPU's residency limit (fewer CTAs per rank when not all can be resident)
 * and before an unchained fixed two-shot at or above its TMA threshold
 * switches to the TMA kernel's own shape; a shape forced with
 * llar_set_launch is reported as forced. Either pointer may be NULL.
 * LLAR_ERR_INVALID for arguments out of range. */
int llar_debug_launch_shape(int nranks, int dtype, size_t count, int protocol, int chained, int sms,
                            size_t chunk_bytes, int* ctas_per_rank, int* threads);

/* One LL AllReduce that allocates nothing: no cudaMalloc, no cudaFree and
 * no allocating library routine, before or during the call, and no
 * llar_init needed. (No page describes this entry point; it exists for
 * callers whose device memory is all owned by a caching allocator or a
 * fixed budget, e.g. an inference-server plugin, and for latency-critical
 * paths where cudaMalloc's implicit device synchronisation is not
 * acceptable.) The LL staging lives in a fixed 1 MiB + 512 B device array
 * inside this library, held by every GPU that loads it until the process
 * exits. in[r] / out[r] are as for llar_allreduce; nranks 2..8; dtype an
 * llar_dtype_t; count * element size must be at most 32 KiB per rank,
 * else LLAR_ERR_TOO_LARGE. The first call on a device resolves the array's
 * device address (cudaGetSymbolAddress), so make that first call before
 * any stream capture. Every call shares the array: calls that overlap on
 * the GPU (other streams, other threads) race and must be avoided; calls
 * in one stream are safe. Each call uses a fresh epoch, so no clearing is
 * needed between calls. Device waits are bounded by llar_set_timeout_ns
 * and honour llar_debug_inject, as the context's launches do. A wait that
 * runs out sets an abort word in the array, and the call's outputs are
 * invalid. The host learns of it only later: the first call made while
 * `stream` is idle (cudaStreamQuery, then a 4-byte device-to-host copy and
 * a stream synchronisation, paid by every call on an idle stream) returns
 * LLAR_ERR_TIMEOUT once, clears the word and launches nothing; the next
 * call works normally. Calls queued while the stream was still busy
 * (between the call whose wait ran out and the one that reports it) find
 * the abort word set, give up their waits at once, return LLAR_OK and
 * also leave invalid outputs. No check is made while `stream` is being
 * captured. */
int llar_allreduce_noalloc(const void* const* in, void* const* out, size_t count,
                           int nranks, int dtype, void* stream);

/* Poll counts (diagnostic; no page describes it). In the poll-counting
 * build of this library (libllar_polls.so, compiled with LLAR_POLL_STATS:
 * python -m tp_allreduce_persistent_b300.build --poll-stats) the library's
 * own AllReduce kernels count their polling: stats[0] thread polling rounds
 * (one round loads every line the thread still awaits), stats[1] line loads
 * issued in those rounds, stats[2] bounded waits started, stats[3] lines
 * those waits awaited. stats[1] / stats[3] is the loads per awaited line (1
 * = every line was there at its first load); stats[0] / stats[2] the rounds
 * per wait. The counters add up across launches; reset != 0 zeroes them
 * after the read. Synchronises the device. The regular build returns
 * LLAR_ERR_UNSUPPORTED; timings of the counting build are not the
 * library's. */
int llar_debug_poll_stats(unsigned long long* stats, int reset);

/* Static description of a status code. */
const char* llar_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* LLAR_H */
