/*
 * llar LL buffer: the signalling primitives of the low-latency collectives,
 * packaged for kernels written by the user ("Every Microsecond Matters:
 * Achieving Near Speed-of-Light Latency in GPU Collectives", summary page:
 * the four techniques are offered as a low-level buffer API for custom
 * kernels).
 *
 * This header is the host half, plain C: a descriptor that the host
 * creates once and then passes BY VALUE to any kernel, and the calls that
 * create, inspect, reset and destroy it. The device half, the
 * `__device__` primitives that act on the descriptor, is the header-only
 * `llar_llbuffer.cuh`, which a user .cu file includes.
 *
 * A descriptor owns, for N virtual ranks (2..8) and a payload of up to
 * `bytes` bytes per rank per exchange:
 *  - LL lines (technique 1): rank q publishes 8-byte word w of exchange
 *    epoch E as one 16-byte line {word, E} at
 *      ll + q*ll_rank_stride + (E & 1)*ll_slot_stride + 16*w,
 *    w < ll_words, which is at least ceil(bytes / 8) and also covers 16
 *    words for every LL128 line of every owner (an LL AllGather of the
 *    reduced lines). Lines are never reset: epochs grow.
 *  - sentinel vectors (technique 2): the 16-byte vector v that source q
 *    sends to receiver d in slot s lives at
 *      sen + d*sen_rank_stride + s*sen_slot_stride + q*sen_src_stride + 16*v,
 *    v < sen_vecs = ceil(bytes / 16). Every byte starts as 0xFF (the
 *    all-ones -NaN pattern, in every element type) and the receiver writes
 *    it back after reading.
 *  - LL128 lines (technique 4): 128-byte line l of owner o in slot s at
 *      ll128 + o*ll128_rank_stride + s*ll128_slot_stride + 128*l,
 *    l < ll128_lines (enough for a segment of ceil(bytes / N) bytes at 124
 *    payload bytes per line, plus one). Element 0 of each line is its
 *    count flag. Lines start at zero and the owner zeroes them after use.
 *  - an epoch counter, a completion counter and an abort word in device
 *    memory, and a status record in mapped host memory.
 * Slots alternate with the exchange epoch (E & 1): technique 3's double
 * buffering; the credit rule that makes slot reuse safe is the user
 * kernel's duty (the primitives' comments state it).
 *
 * Concurrency: kernels that use one descriptor must not run at the same
 * time. Every wait in the device primitives is bounded by timeout_ns; a
 * wait that runs out records LLAR_ERR_TIMEOUT (llar.h) with the rank and
 * epoch, sets the abort word so that every other wait gives up at once,
 * and returns false. The descriptor stays unusable (every primitive wait
 * fails at once) until llar_llbuffer_reset().
 */
#ifndef LLAR_LLBUFFER_H
#define LLAR_LLBUFFER_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Error record; the device writes it, the host reads it (mapped memory). */
typedef struct llar_llbuffer_status {
  unsigned code;              /* 0, or LLAR_ERR_TIMEOUT (7) */
  int rank;                   /* virtual rank whose wait ran out */
  unsigned long long epoch;   /* epoch it waited for */
} llar_llbuffer_status;

typedef struct llar_llbuffer {
  int nranks;                       /* 2..8 */
  int reserved;
  size_t bytes;                     /* payload capacity per rank per exchange */
  unsigned long long timeout_ns;    /* bound of every primitive wait */
  /* LL lines */
  void* ll;
  size_t ll_rank_stride, ll_slot_stride, ll_words;
  /* sentinel vectors */
  void* sen;
  size_t sen_rank_stride, sen_slot_stride, sen_src_stride, sen_vecs;
  /* LL128 lines */
  void* ll128;
  size_t ll128_rank_stride, ll128_slot_stride, ll128_lines;
  /* device control words */
  unsigned long long* epoch;        /* exchanges completed so far */
  unsigned* done_count;             /* CTAs that finished the current launch */
  unsigned* abort_word;             /* nonzero after a timeout */
  llar_llbuffer_status* status;     /* device address of the mapped record */
  llar_llbuffer_status* status_host;/* host address of the same record */
} llar_llbuffer;

/* Allocate and initialise a descriptor for `nranks` (2..8) virtual ranks
 * and `bytes` (1 .. 1 GiB) payload bytes per rank per exchange. Fills *out.
 * Needs no llar_init(). Returns LLAR_OK, LLAR_ERR_INVALID (bad arguments,
 * out NULL) or LLAR_ERR_CUDA (allocation failed; nothing is left
 * allocated). Synchronous. */
int llar_llbuffer_create(int nranks, size_t bytes, llar_llbuffer* out);

/* Free everything `b` owns and zero *b. The caller guarantees that no
 * kernel using it is still running. LLAR_ERR_INVALID for NULL or a
 * descriptor that was never created. Synchronous. */
int llar_llbuffer_destroy(llar_llbuffer* b);

/* Status of the descriptor: LLAR_OK, or LLAR_ERR_TIMEOUT with *rank and
 * *epoch (either pointer may be NULL). Reads host memory only: a timeout
 * of a kernel still running may not be visible yet. */
int llar_llbuffer_get_status(const llar_llbuffer* b, int* rank, unsigned long long* epoch);

/* After a timeout: on `stream`, refill the sentinel vectors with 0xFF,
 * zero the LL128 lines, clear the abort word, then synchronise the stream
 * and clear the status record. Epochs keep growing, so stale LL lines
 * never match a later epoch. */
int llar_llbuffer_reset(llar_llbuffer* b, void* stream);

/* Set the bound of every primitive wait (nanoseconds, > 0) in *b; kernels
 * launched afterwards with the updated descriptor use it. */
int llar_llbuffer_set_timeout_ns(llar_llbuffer* b, unsigned long long ns);

/* Exchanges completed so far: the device epoch counter (every launch of a
 * kernel that called llb::end(b, n[, E]) added n). Synchronises the
 * device. */
int llar_llbuffer_epoch(const llar_llbuffer* b, unsigned long long* epoch);

/* Diagnostic: one thread of one CTA waits (llb::ll_wait) as rank `rank`
 * for word `word` of rank `src` to carry epoch `epoch`. A wait for an
 * epoch that no kernel publishes ends after timeout_ns with
 * LLAR_ERR_TIMEOUT recorded for (rank, epoch), which exercises the
 * timeout and reset path without any fault. Asynchronous on `stream`. */
int llar_llbuffer_probe_wait(const llar_llbuffer* b, int rank, int src, unsigned long long epoch,
                             size_t word, void* stream);

/* ---- kernels built only from the device primitives of llar_llbuffer.cuh
 *
 * An AllReduce of `count` elements per rank (in[r], out[r]: device
 * pointers, 16-byte aligned, out not overlapping any input; count * elem
 * <= b->bytes) using one of LLAR_PROTO_LL, LLAR_PROTO_SENTINEL (fixed
 * rank order, bit-identical to the float32 rank-order sum rounded once)
 * or LLAR_PROTO_LL128_ATOMIC (atomic, within (N-1) ulp of sum |x|).
 * `iters` >= 1 repeats it on the same buffers back to back inside one
 * persistent launch (for latency measurement; every iteration computes
 * the same result). Sentinel inputs must not contain the all-ones
 * element pattern. Asynchronous on `stream`; returns LLAR_ERR_INVALID,
 * LLAR_ERR_TOO_LARGE, LLAR_ERR_UNSUPPORTED (protocol), LLAR_ERR_TIMEOUT
 * (status already set), LLAR_ERR_OCCUPANCY or LLAR_ERR_CUDA. */
int llar_llbuffer_allreduce(const llar_llbuffer* b, const void* const* in, void* const* out,
                            size_t count, int dtype, int protocol, int iters, void* stream);

/* Tensor-parallel row-parallel linear layer with its AllReduce fused into
 * the epilogue ("zcube network architecture for LLM inference", section
 * "Why does Tensor Parallel affect every token": every layer ends in the
 * sum of the ranks' partial outputs):
 *   out[q][m][h] = sum over r = 0..N-1 (in that order) of p_r[m][h],
 *   p_r[m][h]    = round_dtype( sum over k = 0..K-1 of x[r][m][k] * w[r][k][h] ),
 * x[r]: M x K, w[r]: K x H, out[q]: M x H, all row-major `dtype`, N =
 * b->nranks. Dot products accumulate in float32 with fused multiply-adds
 * (K split across warps, the slices added in order; for fp16/bf16 every
 * product is exact in float32), the rank sum in float32 with one
 * rounding. Up to 4 rows (and for fp32) the dot products run on CUDA
 * cores; for fp16/bf16 with more rows on the tensor cores (mma.sync,
 * float32 accumulation in an order and rounding of their own: within the
 * same float32 error bound with 2^-23 per addition). The partial p_r never goes to memory: the GEMV epilogue
 * publishes it as LL lines and every rank reduces the lines it polls.
 * Limits: 1 <= M <= 16, 1 <= K, H >= 8, H % 8 == 0, M*H*elem <= b->bytes,
 * M*K*elem <= 96 KiB; pointers 16-byte aligned. Asynchronous on `stream`;
 * status codes as llar_llbuffer_allreduce. */
int llar_fused_linear_allreduce(const llar_llbuffer* b, const void* const* x, const void* const* w,
                                void* const* out, int m, int k, int h, int dtype, void* stream);

/* The GEMV half alone (the unfused pipeline's first launch): p[r] = the
 * rounded partial p_r above, for r < nranks, same arithmetic. Pair it with
 * llar_allreduce or llar_llbuffer_allreduce over p to get the unfused
 * layer. Same limits (without the b->bytes one). */
int llar_linear_partials(const void* const* x, const void* const* w, void* const* p, int nranks,
                         int m, int k, int h, int dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LLAR_LLBUFFER_H */
