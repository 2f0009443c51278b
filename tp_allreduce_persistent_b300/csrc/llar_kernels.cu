// Persistent AllReduce kernels over N virtual ranks, and the speed-of-light
// probes. One launch = N x G CTAs; CTAs [r*G, (r+1)*G) are virtual rank r.
// CTA c of rank r pairs with CTA c of every peer: all of them cover the same
// element range, and every element position is always handled by the same
// thread index, so a thread's program order carries the credit rule of the
// double-buffered protocols ("Every Microsecond Matters: Achieving Near
// Speed-of-Light Latency in GPU Collectives", summary page, technique 3:
// receiving a chunk from a peer is the permission to send it the next one).
// No kernel contains a grid-wide barrier; the only waits are per-line polls
// (techniques 1, 2, 4) and, on the fixed-order chained paths, per-CTA-pair
// epoch flags.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "llar.h"
#include "llar_device.cuh"

namespace llar {

// ----------------------------------------------------------- shared helpers
template <int DT>
__device__ __forceinline__ const char* rank_input(const Params& p, int q, int e) {
  if (p.chain)
    return e == 0 ? p.in[q] : p.chainbuf + (size_t)q * p.chain_stride + (size_t)(e & 1) * p.chain_slot_bytes;
  return p.in[q] + (size_t)e * p.in_stride * Fmt<DT>::kBytes;
}
template <int DT>
__device__ __forceinline__ char* rank_output(const Params& p, int q, int e) {
  return p.out[q] + (size_t)e * p.out_stride * Fmt<DT>::kBytes;
}
__device__ __forceinline__ char* chain_next_buf(const Params& p, int q, int e) {
  return p.chainbuf + (size_t)q * p.chain_stride + (size_t)((e + 1) & 1) * p.chain_slot_bytes;
}

// 8-byte word w (elements [w*PER8, (w+1)*PER8)) of a rank buffer; a word
// that runs past `count` is read element by element, the rest as zeros.
template <int DT>
__device__ __forceinline__ u64 load_word8(const char* base, size_t w, size_t count) {
  constexpr int PER8 = 8 / Fmt<DT>::kBytes;
  if ((w + 1) * PER8 <= count) return *reinterpret_cast<const u64*>(base + w * 8);
  unsigned x[2];
  load_words_tail<DT, 2>(base, w * PER8, count, x);
  return (u64)x[0] | ((u64)x[1] << 32);
}
template <int DT>
__device__ __forceinline__ void store_word8(char* base, size_t w, size_t count, u64 v) {
  constexpr int PER8 = 8 / Fmt<DT>::kBytes;
  if ((w + 1) * PER8 <= count) {
    *reinterpret_cast<u64*>(base + w * 8) = v;
    return;
  }
  unsigned x[2] = {(unsigned)v, (unsigned)(v >> 32)};
  store_words_tail<DT, 2>(base, w * PER8, count, x);
}
template <int DT>
__device__ __forceinline__ uint4 load_vec16(const char* base, size_t v, size_t count, bool stream) {
  constexpr int PER16 = 16 / Fmt<DT>::kBytes;
  if ((v + 1) * PER16 <= count) return stream ? ld_stream_v4(base + v * 16) : ld_cg_v4(base + v * 16);
  unsigned x[4];
  load_words_tail<DT, 4>(base, v * PER16, count, x);
  return make_uint4(x[0], x[1], x[2], x[3]);
}
template <int DT>
__device__ __forceinline__ void store_vec16(char* base, size_t v, size_t count, uint4 val) {
  constexpr int PER16 = 16 / Fmt<DT>::kBytes;
  if ((v + 1) * PER16 <= count) {
    st_v4(base + v * 16, val);
    return;
  }
  unsigned x[4] = {val.x, val.y, val.z, val.w};
  store_words_tail<DT, 4>(base, v * PER16, count, x);
}

__device__ __forceinline__ uint4 u4(const unsigned* w) { return make_uint4(w[0], w[1], w[2], w[3]); }

// Block b is CTA c = b / N of virtual rank r = b % N: the N CTAs that serve
// the same range c of every rank are consecutive, so a launch with a
// cluster of N blocks puts each such group on one GPC.
__device__ __forceinline__ int rank_of_block(const Params& p) { return blockIdx.x % p.nranks; }
__device__ __forceinline__ int cta_of_block(const Params& p) { return blockIdx.x / p.nranks; }

// Epochs live in device memory, so a launch captured in a CUDA graph and
// replayed still gets fresh epochs: every CTA reads the counter when it
// starts (iteration e of the launch uses counter + 1 + e), and the last CTA
// to finish, which knows that every CTA has read it, advances it by the
// launch's iteration count. A CTA's read has completed (its value is in
// use) before the CTA counts itself finished, and the next launch is
// stream-ordered after this one, so relaxed atomics suffice: no fence.
// Measured per launch on B300 (128 CTAs, cooperative, graph replay): the
// fenced version cost 1.7 us over a bare launch, the relaxed one 1.0 us.
// A launch made as a programmatic dependent of the previous kernel in the
// stream (p.pdl) may be scheduled before that kernel ends; griddepcontrol
// .wait holds it until the previous kernel has completed and its memory
// is visible (a no-op otherwise), and launch_dependents lets the next
// launch be scheduled early in turn.
__device__ __forceinline__ u64 launch_epoch(const Params& p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const u64 e = *reinterpret_cast<volatile const u64*>(p.epoch_dev) + 1;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  return e;
}
// `counted`: whether this CTA takes part in the count; `participants`: how
// many do. Every CTA may take part; a kernel in which rank 0's CTA c
// consumes, in its last iteration, data that every CTA of column c produced
// after reading the counter may count rank 0's CTAs alone (G atomics on
// the counter word instead of N x G).
// `epoch0` is what launch_epoch returned: the counter every CTA read is
// epoch0 - 1, and only the last CTA to count writes it, so the new value
// needs no second read of the counter (a round trip at the end of every
// launch: 8 x 16 KiB bf16 LL, one AllReduce per launch replayed from a
// graph, 2.79 -> 2.46 us per launch).
__device__ __forceinline__ void finish_launch(const Params& p, u64 epoch0, bool counted, unsigned participants) {
  __syncthreads();
  if (threadIdx.x == 0 && counted) {
    if (atomicAdd(p.done_count, 1u) == participants - 1) {
      *reinterpret_cast<volatile unsigned*>(p.done_count) = 0u;
      *reinterpret_cast<volatile u64*>(p.epoch_dev) = epoch0 - 1 + (u64)p.iters;
    }
  }
}
__device__ __forceinline__ void finish_launch(const Params& p, u64 epoch0) {
  finish_launch(p, epoch0, true, gridDim.x);
}

// One thread per unit (an 8-byte LL word or a 16-byte sentinel vector):
// the thread sends its unit of my data (LL: publishes it once in my own
// staging; sentinel: pushes it into every peer's slot), polls the unit of
// every peer, adds the N values in rank order and stores the result. The
// kernels are instantiated per N, so the peer loops unroll without guards.
// A warp's store, and a warp's poll of one source, cover 32 consecutive
// units.

// float32 values of the elements of a 32-bit word
template <int DT>
__device__ __forceinline__ void unpack2(unsigned w, float& a, float& b) {
  if (DT == 2) {  // bf16: the value is the upper half of a float32
    a = __uint_as_float(w << 16);
    b = __uint_as_float(w & 0xFFFF0000u);
  } else if (DT == 1) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    a = f.x;
    b = f.y;
  }
}
// two float32 values rounded (roundTiesToEven) into one 32-bit word
template <int DT>
__device__ __forceinline__ unsigned pack2(float a, float b) {
  if (DT == 2) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const unsigned*>(&h);
  }
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const unsigned*>(&h);
}

// acc (n32*PER32 floats) = values of the words of `w`, or += them
template <int DT, int NW>
__device__ __forceinline__ void acc_words(float* acc, const unsigned* w, bool first) {
#pragma unroll
  for (int k = 0; k < NW; ++k) {
    if (DT == 0) {
      const float f = __uint_as_float(w[k]);
      acc[k] = first ? f : __fadd_rn(acc[k], f);
    } else {
      float a, b;
      unpack2<DT>(w[k], a, b);
      acc[2 * k] = first ? a : __fadd_rn(acc[2 * k], a);
      acc[2 * k + 1] = first ? b : __fadd_rn(acc[2 * k + 1], b);
    }
  }
}
template <int DT, int NW>
__device__ __forceinline__ void round_words(const float* acc, unsigned* w) {
#pragma unroll
  for (int k = 0; k < NW; ++k) w[k] = (DT == 0) ? __float_as_uint(acc[k]) : pack2<DT>(acc[2 * k], acc[2 * k + 1]);
}
template <int DT, int NW>
__device__ __forceinline__ void chain_words_fast(const float* acc, const unsigned* y, unsigned* nx, float scale) {
  // next input = roundTiesToEven(scale * y), y being the rounded output
  float t[NW * 2];
  acc_words<DT, NW>(t, y, true);
  (void)acc;
#pragma unroll
  for (int k = 0; k < NW * (DT == 0 ? 1 : 2); ++k) t[k] = __fmul_rn(scale, t[k]);
  round_words<DT, NW>(t, nx);
}

// ============================================================ LL one-shot
// Technique 1: each 8 bytes of data leave with an 8-byte flag (the epoch of
// this AllReduce) as one 16-byte store; the reader polls that 16-byte line
// until the flag equals the epoch, so no separate signal and no barrier is
// needed, and epochs only grow, so lines never need a reset. On one GPU a
// store into the reader's staging and a load of the writer's staging both
// travel to the same L2, so each rank publishes its lines once, in its own
// staging [epoch & 1][word], and every peer reads them there (one store per
// word instead of N-1). Credit (technique 3): the owner of word w of rank r
// rewrites slot (E & 1) at epoch E + 2 only after it read word w of epoch
// E + 1 from every peer, and each peer's owner of word w published that
// only after reading my epoch-E word w.
//
// The kernel is written with the public device primitives of the LL buffer
// API (llar_llbuffer.cuh) over a descriptor view of this context's LL
// staging; measured on B300 this form is also the fastest (8 ranks x 16 KiB
// bf16: 0.65 us per AllReduce against 0.71 for the earlier hand-rolled
// loop).
template <int DT> struct ElemOf;
template <> struct ElemOf<0> { typedef float T; };
template <> struct ElemOf<1> { typedef __half T; };
template <> struct ElemOf<2> { typedef __nv_bfloat16 T; };

// the context's LL staging as an LL buffer descriptor (only the fields the
// LL primitives and the bounded waits read)
__device__ __forceinline__ llar_llbuffer ll_view(const Params& p, int n) {
  llar_llbuffer b = {};
  b.nranks = n;
  b.timeout_ns = p.timeout_ns;
  b.ll = p.ll;
  b.ll_rank_stride = p.ll_stride;
  b.ll_slot_stride = p.ll_slot_words * (size_t)kLLLine;
  b.abort_word = p.abort_flag;
  b.status = reinterpret_cast<llar_llbuffer_status*>(p.status);
  return b;
}

// MODE 0: the same buffers every iteration, no fault injection (the fast
// instance: per-iteration pointer arithmetic costs about 95 ns per
// AllReduce here); 1: strided inputs/outputs and fault injection; 2: the
// chain (the next input is computed from the output), as 1.
template <int DT, int N, int MODE>
__global__ void __launch_bounds__(kMaxThreads) k_ll(const Params p) {
  typedef typename ElemOf<DT>::T T;
  constexpr bool CHAIN = MODE == 2, GENERAL = MODE != 0;
  const llar_llbuffer b = ll_view(p, N);
  const u64 E0 = launch_epoch(p);
  const int r = blockIdx.x % N, c = blockIdx.x / N;
  const size_t W = (p.count * Fmt<DT>::kBytes + 7) / 8;  // 8-byte words per rank
  const size_t per = (W + p.G - 1) / p.G;
  const size_t w0 = min(W, (size_t)c * per), w1 = min(W, w0 + per);
  const bool injected = GENERAL && p.inject_rank == r;
  const bool skip = injected && p.inject_mode == LLAR_INJECT_SKIP_;
  const bool poison = injected && p.inject_mode == LLAR_INJECT_POISON_;
  auto publish = [&](u64 E, size_t w, u64 x) {
    if (skip) return;
    if (poison) llb::st_relaxed_b128(llb::ll_line(b, r, E, w), x, E + 2);
    else llb::ll_put(b, r, E, w, x);
  };

  // AllReduce 0's lines go out first; afterwards each word's line for
  // AllReduce e+1 goes out as soon as that word of AllReduce e has been
  // received from every peer (technique 3: receiving is the permission to
  // send the next one), before the reduction of e is computed.
  if (injected && p.inject_mode == LLAR_INJECT_DELAY_) injected_delay();
  for (size_t w = w0 + threadIdx.x; w < w1; w += blockDim.x) publish(E0, w, load_word8<DT>(p.in[r], w, p.count));
  bool ok = true;
  for (int e = 0; e < p.iters && ok; ++e) {
    const u64 E = E0 + (u64)e;
    const bool more = e + 1 < p.iters;
    const char* in = GENERAL ? rank_input<DT>(p, r, e) : p.in[r];
    const char* in_next = (GENERAL && !CHAIN && more) ? rank_input<DT>(p, r, e + 1) : in;
    char* out = GENERAL ? rank_output<DT>(p, r, e) : p.out[r];
    if (e > 0 && injected && p.inject_mode == LLAR_INJECT_DELAY_) injected_delay();
    for (size_t w = w0 + threadIdx.x; w < w1; w += blockDim.x) {
      u64 d[N];
      d[r] = load_word8<DT>(in, w, p.count);
      // the next input's word is loaded before the poll, so that its line
      // leaves right after the poll succeeds
      const u64 nxt = (GENERAL && !CHAIN && in_next != in) ? load_word8<DT>(in_next, w, p.count) : d[r];
      if (!llb::ll_wait_peers<N>(b, r, E, w, d)) {
        ok = false;
        break;
      }
      if (!CHAIN && more) publish(E + 1, w, nxt);
      const u64 y = llb::sum_words<T, N>(d);  // rank order, float32, one rounding
      if (CHAIN && more) {
        const unsigned y2[2] = {(unsigned)y, (unsigned)(y >> 32)};
        unsigned nx[2];
        chain_words<DT, 2>(y2, nx, p.chain_scale);
        const u64 nw = (u64)nx[0] | ((u64)nx[1] << 32);
        publish(E + 1, w, nw);  // the next input is known now: send it before storing
        store_word8<DT>(chain_next_buf(p, r, e), w, p.count, nw);
      }
      store_word8<DT>(out, w, p.count, y);
    }
  }
  // every thread of rank 0's CTA c read, in the last iteration, a line that
  // the same thread of each peer CTA c published after reading the counter
  // (peer threads without words do nothing with it)
  finish_launch(p, E0, r == 0, (unsigned)p.G);
}

// ====================================================== sentinel one-shot
// Technique 2 with technique 3's chunking: staging slot
// [seq & 1][source][vector] is prefilled with the all-ones (-NaN) pattern;
// the owner of vector j pushes my raw 16-byte vector to every peer, polls
// the vector every peer sent until none of its elements is the sentinel,
// and writes the sentinel back (the reset). Chunk seq+1 is pushed to peer q
// only after chunk seq was received from peer q, so peer q's slot
// (seq+1) & 1 for me was consumed and reset in its chunk seq-1 by the
// owner of the same vector; a fence orders that reset before the owner's
// next push.
template <int DT, int N, bool CHAIN, bool INJ>
__device__ __forceinline__ void body_sentinel(const Params& p, const u64 epoch0) {
  constexpr int EB = Fmt<DT>::kBytes;
  constexpr int PER16 = 16 / EB;
  const int r = rank_of_block(p);
  const int c = cta_of_block(p);
  const unsigned NV = (unsigned)((p.count + PER16 - 1) / PER16);
  const bool full = (p.count % PER16) == 0;  // no partial vector at the end
  const unsigned CV = (unsigned)p.sen_chunk_vecs;
  const unsigned nchunks = (NV + CV - 1) / CV;
  // the CTAs split the part of a chunk the message uses (a message shorter
  // than the chunk would otherwise land on the first CTAs only)
  const unsigned CU = min(CV, NV);
  const unsigned per = (CU + p.G - 1) / p.G;
  const unsigned j0 = min(CU, (unsigned)c * per);
  const unsigned j1 = min(CU, j0 + per);
  const size_t src_stride = (size_t)CV * 16;
  const size_t slot_stride = (size_t)N * src_stride;
  const bool injected = INJ && (p.inject_rank == r);
  const bool skip = injected && p.inject_mode == LLAR_INJECT_SKIP_;
  const bool poison = injected && p.inject_mode == LLAR_INJECT_POISON_;
  const uint4 ones = make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
  char* to[N];    // my slots in peer q's staging
  char* from[N];  // peer q's slots in my staging
#pragma unroll
  for (int q = 0; q < N; ++q) {
    to[q] = p.sen + (size_t)q * p.sen_stride + (size_t)r * src_stride;
    from[q] = p.sen + (size_t)r * p.sen_stride + (size_t)q * src_stride;
  }
  const unsigned others = ((1u << N) - 1u) & ~(1u << r);
  constexpr bool EARLY = N <= kSenEarlyMaxN;
  auto input = [&](int e) -> const char* {
    return CHAIN ? rank_input<DT>(p, r, e) : p.in[r] + (size_t)e * p.in_stride * EB;
  };
  auto load = [&](const char* src, unsigned v) -> uint4 {
    if (poison) return ones;
    if (full || v + 1 < NV) return CHAIN ? ld_cg_v4(src + (size_t)v * 16) : ld_stream_v4(src + (size_t)v * 16);
    return load_vec16<DT>(src, v, p.count, !CHAIN);
  };
  auto load_cg = [&](const char* src, unsigned v) -> uint4 {
    if (poison) return ones;
    if (full || v + 1 < NV) return ld_cg_v4(src + (size_t)v * 16);
    return load_vec16<DT>(src, v, p.count, false);
  };
  // Push my vector j of chunk sequence number sq into every peer's slot
  // sq & 1. Credit (technique 3): peer q consumed and reset my vector j of
  // sq - 2 before it pushed its vector j of sq - 1, which I have received.
  // A vector index that had no vector in sq - 1 (beyond a partial last
  // chunk) has no such credit: it waits until the cell reads all-ones,
  // which after my own earlier write there can only be q's reset. False on
  // timeout.
  auto push = [&](unsigned long long sq, unsigned j, uint4 x, bool no_credit, u64 E) -> bool {
    if (skip) return true;
    const size_t off = (size_t)(sq & 1) * slot_stride + (size_t)j * 16;
#pragma unroll
    for (int q = 0; q < N; ++q) {
      if (q == r) continue;
      char* cell = to[q] + off;
      if (no_credit && sq >= 2) {
        Waiter wt;
        while (!is_all_ones(ld_relaxed_v4(cell)))
          if (wt.expired(p)) {
            report_timeout(p, r, c, E);
            return false;
          }
      }
      st_relaxed_v4(cell, x);
    }
    return true;
  };

  // PUBLISH-ONCE (at least kSenPubMinN ranks, at most one vector per thread
  // and chunk). As in the LL one-shot, each rank writes its vector j of
  // chunk t once, into its own ring of S = kSenPubSlots slots (slot t % S,
  // all-ones when idle), and every peer polls it there until no element is
  // the sentinel. On one GPU a peer's load and a store into the peer's
  // staging meet in the same L2, so one store replaces N - 1 pushes
  // (measured with the pushes: 7 stores took 0.45 us of a 1.66 us step).
  // The owner resets its slot D = 2F steps later (F = kSenFencePeriod), runs
  // a fence every F steps, and S = 4F. Step t: fence if t is a positive
  // multiple of F; publish chunk t; reset chunk t - D; store the output of
  // chunk t - 1; load the next step's input; poll chunk t from every peer;
  // reduce into registers. Credit (technique 3): (1) no reset before every
  // reader has read: reader q polled my chunk u in its step u, fenced at
  // g = the first multiple of F after u, and published chunk g (or g + 1,
  // the steps without a vector being isolated); I received that before my
  // fence at g + F <= u + D, which precedes my reset of u. (2) no stale read
  // after reuse: my reset of chunk u - S, in step u - S + D = u - 2F,
  // precedes my fence f <= u - F and my publication of chunk f (or f + 1);
  // q received that before its fence at f + F <= u, which precedes its poll
  // of chunk u. At the end of the launch each thread publishes the launch's
  // last epoch in a tail word (after a fence), waits for its peers' tail
  // words, fences and resets the slots still holding data, so the next
  // launch finds every slot all-ones. That tail costs about one round trip
  // and two fences per launch (8 ranks x 16 KiB bf16, one AllReduce per
  // launch: 3.7 us on the push path, 5.4 us published once), so launches of
  // fewer than kSenPubMinSteps chunks take the push path below.
  if (N >= kSenPubMinN && per <= blockDim.x && (unsigned)p.iters * nchunks >= (unsigned)kSenPubMinSteps) {
    const unsigned j = j0 + threadIdx.x;
    if (j >= j1) return;
    constexpr unsigned S = (unsigned)kSenPubSlots, F = (unsigned)kSenFencePeriod, D = 2 * F;
    static_assert(S == 4 * F && F >= 2, "the credit chain needs S = 4F slots and F >= 2");
    static_assert(2 * F < 32, "the history mask keeps the last 2F steps");
    const size_t ring = (size_t)CV * 16;  // bytes per slot
    char* const col = p.sen + (size_t)j * 16;  // vector j's cell in slot 0 of rank 0's ring
    auto cell = [&](int q, size_t slot_off) -> char* { return col + (size_t)q * p.sen_stride + slot_off; };
    auto tail_word = [&](int q) -> u64* {
      return reinterpret_cast<u64*>(p.sen + (size_t)q * p.sen_stride + (size_t)S * kSenMaxChunkBytes) + j;
    };
    unsigned hist = 0;  // bit i: step t - i had vector j (after this step's bit is shifted in)
    bool lag = false;  // step t - 1 had my vector j: its output is still to be stored
    char* lag_dst = nullptr;
    char* lag_chain = nullptr;
    unsigned lag_v = 0;
    uint4 lag_y = ones, lag_nx = ones;
    auto store_lagged = [&]() {
      if (!lag) return;
      if (full || lag_v + 1 < NV) st_v4(lag_dst + (size_t)lag_v * 16, lag_y);
      else store_vec16<DT>(lag_dst, lag_v, p.count, lag_y);
      if (CHAIN) store_vec16<DT>(lag_chain, lag_v, p.count, lag_nx);
      lag = false;
    };
    // the chunk received last, reduced only after the next chunk has been
    // published (the reduction is register work: the order of the memory
    // operations, and so the credit argument, is unchanged)
    bool pending = false;
    uint4 pd[N];
    uint4 p_own = ones;
    char* p_dst = nullptr;
    unsigned p_v = 0;
    int p_e = 0;
    auto reduce_pending = [&]() {
      if (!pending) return;
      float acc[PER16];
#pragma unroll
      for (int q = 0; q < N; ++q) {
        const uint4 vq = (q == r) ? p_own : pd[q];
        const unsigned w4[4] = {vq.x, vq.y, vq.z, vq.w};
        acc_words<DT, 4>(acc, w4, q == 0);
      }
      unsigned y[4];
      round_words<DT, 4>(acc, y);
      lag_y = u4(y);
      if (CHAIN) {
        unsigned nx[4];
        chain_words_fast<DT, 4>(acc, y, nx, p.chain_scale);
        lag_nx = u4(nx);
        lag_chain = chain_next_buf(p, r, p_e);
      }
      lag = true;
      lag_dst = p_dst;
      lag_v = p_v;
      pending = false;
    };
    // The next step's input is loaded before this step's poll, with
    // L2-coherent (.cg) loads: through the non-coherent read-only path the
    // inputs took 2.5x longer per AllReduce here (8 ranks x 64 KiB fp16 in
    // 8 KiB chunks: 25.3 against 10.4 us on one box; the push path below
    // does not gain from .cg). A chain's next inputs are its own outputs of
    // the previous iteration: loading them ahead measured slower (C5 chain,
    // 8 ranks: 14.0 against 11.5 us per AllReduce), so a chain loads them
    // at the publication.
    const bool ahead = !CHAIN;
    bool have_next = false;
    uint4 next_own = ones;
    unsigned t = 0;
    size_t slot_off = 0;                          // (t % S) * ring
    size_t reset_off = (size_t)(S - D) * ring;    // ((t - D) % S) * ring
    auto advance = [&](size_t off) { return off + ring == (size_t)S * ring ? (size_t)0 : off + ring; };
    u64 E = epoch0;
    for (int e = 0; e < p.iters; ++e) {
      E = epoch0 + (u64)e;
      const char* src = input(e);
      char* dst = rank_output<DT>(p, r, e);
      for (unsigned k = 0; k < nchunks; ++k, ++t, slot_off = advance(slot_off), reset_off = advance(reset_off)) {
        if (injected && p.inject_mode == LLAR_INJECT_DELAY_) injected_delay();
        // a chain reduces first: with one chunk per iteration its next input is
        // that reduction's output, and otherwise the input load of the
        // publication below then overlaps the reduction (C5 chain, 8 ranks:
        // 11.5 against 13.0 us per AllReduce reducing after the publication)
        if (CHAIN) reduce_pending();
        if (t > 0 && t % F == 0) fence_gpu();
        const unsigned v = k * CV + j;
        const bool has = v < NV;
        hist = (hist << 1) | (has ? 1u : 0u);
        uint4 own = ones;
        if (has) {
          own = have_next ? next_own
                          : ((CHAIN && e > 0 && nchunks == 1) ? (poison ? ones : lag_nx) : load_cg(src, v));
          // one 128-bit access: a poller sees all of it or none of it
          if (!skip)
            st_relaxed_b128(cell(r, slot_off), (u64)own.x | ((u64)own.y << 32), (u64)own.z | ((u64)own.w << 32));
        }
        reduce_pending();
        if (t >= D && ((hist >> D) & 1u) && !skip) st_relaxed_v4(cell(r, reset_off), ones);
        store_lagged();
        have_next = false;
        if (ahead) {
          const bool wrap = k + 1 == nchunks;
          const unsigned nv = (wrap ? 0u : k + 1) * CV + j;
          if ((!wrap || e + 1 < p.iters) && nv < NV) {
            next_own = load_cg(wrap ? input(e + 1) : src, nv);
            have_next = true;
          }
        }
        if (!has) continue;
        uint4 d[N];
        unsigned pend = others;
        Waiter wt;
        // each vector is read as one 128-bit access (published as one): it
        // is either still all-ones or entirely the new data, which holds no
        // all-ones element, so one test of all 128 bits replaces a test of
        // every element
        for (bool first_round = true;; first_round = false) {
          LLB_ON_POLL_ROUND(first_round, pend);
          u64 lo[N], hi[N];
#pragma unroll
          for (int q = 0; q < N; ++q)
            if ((pend >> q) & 1u) ld_relaxed_b128(cell(q, slot_off), lo[q], hi[q]);
#pragma unroll
          for (int q = 0; q < N; ++q)
            if (((pend >> q) & 1u) && (lo[q] & hi[q]) != ~0ull) {
              d[q] = make_uint4((unsigned)lo[q], (unsigned)(lo[q] >> 32), (unsigned)hi[q], (unsigned)(hi[q] >> 32));
              pend &= ~(1u << q);
            }
          if (pend == 0u) break;
          if (wt.expired(p)) {
            report_timeout(p, r, c, E);
            return;
          }
        }
#pragma unroll
        for (int q = 0; q < N; ++q) pd[q] = d[q];
        p_own = own;
        p_dst = dst;
        p_v = v;
        p_e = e;
        pending = true;
      }
    }
    reduce_pending();
    store_lagged();
    // tail: every peer has read my last chunks once it publishes the last
    // epoch in its tail word, which it does after a fence that follows
    // its polls; then my remaining slots can be reset
    if (skip) return;
    fence_gpu();
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" :: "l"(tail_word(r)), "l"(E) : "memory");
    unsigned pend = others;
    Waiter wt;
    for (bool first_round = true;; first_round = false) {
      LLB_ON_POLL_ROUND(first_round, pend);
#pragma unroll
      for (int q = 0; q < N; ++q)
        if (((pend >> q) & 1u) && ld_relaxed_u64(tail_word(q)) == E) pend &= ~(1u << q);
      if (pend == 0u) break;
      if (wt.expired(p)) {
        report_timeout(p, r, c, E);
        return;
      }
    }
    fence_gpu();
    // chunks t - 1, t - 2, ..., t - D (those that exist), newest first
    size_t off = slot_off;
    for (unsigned i = 0; i < D && i < t; ++i) {
      off = off == 0 ? (size_t)(S - 1) * ring : off - ring;
      if ((hist >> i) & 1u) st_relaxed_v4(cell(r, off), ones);
    }
    return;
  }

  // EARLY (up to 4 ranks): chunk 0 of the first iteration goes out first;
  // afterwards the next chunk's vector j goes out as soon as vector j of
  // this chunk has arrived from every peer and been reset (a fence orders
  // those resets before the push), before this chunk's reduction
  // (technique 3, as in LL); in a chain the next iteration's input is this
  // iteration's output, so its first chunk goes out after the iteration.
  // With more ranks the fence would wait for N - 1 resets just issued;
  // there every chunk is pushed at its start, after a fence that finds the
  // previous chunk's resets landed (measured, 8 ranks: 64 KiB in 8 KiB
  // chunks 15.7 us with this order, 20.0 us with early push; 4 ranks x
  // 16 KiB: 1.57 vs 1.49 us).
  if (injected && p.inject_mode == LLAR_INJECT_DELAY_) injected_delay();
  if (EARLY)
    for (unsigned j = j0 + threadIdx.x; j < j1; j += blockDim.x)
      if (j < NV && !push(0, j, load(input(0), j), false, epoch0)) return;
  unsigned long long seq = 0;
  for (int e = 0; e < p.iters; ++e) {
    const u64 E = epoch0 + (u64)e;
    const char* src = input(e);
    char* dst = rank_output<DT>(p, r, e);
    for (unsigned k = 0; k < nchunks; ++k, ++seq) {
      const size_t slot_off = (size_t)(seq & 1) * slot_stride;
      if (seq > 0 && injected && p.inject_mode == LLAR_INJECT_DELAY_) injected_delay();
      if (!EARLY) {
        if (seq > 0) fence_gpu();  // my resets of the previous chunk before this chunk's pushes
        const unsigned kprev = k > 0 ? k - 1 : nchunks - 1;
        for (unsigned j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
          const unsigned v = k * CV + j;
          if (v >= NV) break;
          if (!push(seq, j, load(src, v), kprev * CV + j >= NV, E)) return;
        }
      }
      const bool last = k + 1 == nchunks;
      const bool has_next = EARLY && (!last || (!CHAIN && e + 1 < p.iters));
      const unsigned nk = last ? 0u : k + 1;                       // next chunk
      const char* nsrc = (has_next && last) ? input(e + 1) : src;  // its input
      for (unsigned j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
        const unsigned v = k * CV + j;
        const bool next_has = has_next && nk * CV + j < NV;
        if (v >= NV) {  // no vector here (partial last chunk): push the next one without credit
          if (next_has) {
            fence_gpu();
            if (!push(seq + 1, j, load(nsrc, nk * CV + j), true, E)) return;
          }
          continue;
        }
        const size_t off = slot_off + (size_t)j * 16;
        const uint4 own = load(src, v);
        uint4 d[N];
        unsigned pend = others;
        unsigned spins = 0;
        u64 deadline = 0;
        for (bool first_round = true;; first_round = false) {
          LLB_ON_POLL_ROUND(first_round, pend);
          uint4 t[N];
#pragma unroll
          for (int q = 0; q < N; ++q)
            if ((pend >> q) & 1u) t[q] = ld_relaxed_v4(from[q] + off);
#pragma unroll
          for (int q = 0; q < N; ++q)
            if (((pend >> q) & 1u) && !has_sentinel<DT>(t[q])) {
              d[q] = t[q];
              pend &= ~(1u << q);
              // reset for the next use of this slot as soon as the vector is
              // in: the resets of early peers land while the others are awaited
              st_relaxed_v4(from[q] + off, ones);
            }
          if (pend == 0u) break;
          if ((++spins & 63u) == 0u) {
            const u64 now = globaltimer_ns();
            if (deadline == 0) deadline = now + p.timeout_ns;
            if (now > deadline || ld_relaxed_u32(p.abort_flag) != 0) {
              report_timeout(p, r, c, E);
              return;  // no barrier inside this body: every exit is per thread
            }
          }
        }
        if (next_has) {
          fence_gpu();  // the resets before the next push
          if (!push(seq + 1, j, load(nsrc, nk * CV + j), false, E)) return;
        }
        float acc[PER16];
#pragma unroll
        for (int q = 0; q < N; ++q) {
          const uint4 vq = (q == r) ? own : d[q];
          const unsigned w4[4] = {vq.x, vq.y, vq.z, vq.w};
          acc_words<DT, 4>(acc, w4, q == 0);
        }
        unsigned y[4];
        round_words<DT, 4>(acc, y);
        if (full || v + 1 < NV) st_v4(dst + (size_t)v * 16, u4(y));
        else store_vec16<DT>(dst, v, p.count, u4(y));
        if (CHAIN) {
          unsigned nx[4];
          chain_words_fast<DT, 4>(acc, y, nx, p.chain_scale);
          store_vec16<DT>(chain_next_buf(p, r, e), v, p.count, u4(nx));
        }
      }
    }
    // a chain's next iteration: its chunk 0 (this thread's own chain values)
    if (EARLY && CHAIN && e + 1 < p.iters) {
      const char* nsrc = input(e + 1);
      for (unsigned j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
        if (j >= NV) continue;
        const bool no_credit = (nchunks - 1) * CV + j >= NV;  // no vector j in the last chunk
        fence_gpu();
        if (!push(seq, j, load(nsrc, j), no_credit, E)) return;
      }
    }
  }
}

template <int DT, int N, bool CHAIN, bool INJ>
__global__ void __launch_bounds__(kMaxThreads) k_sentinel(const Params p) {
  const u64 epoch0 = launch_epoch(p);
  body_sentinel<DT, N, CHAIN, INJ>(p, epoch0);
  // rank 0's thread j took, in the last chunk it handled, the vector that
  // thread j of each peer CTA pushed after reading the counter
  finish_launch(p, epoch0, rank_of_block(p) == 0, (unsigned)p.G);
}

// ======================================================= LL128 two-shot
// Technique 4. Rank s owns segment s (ceil(count/N) elements). A segment
// is carried in 128-byte lines of 8 lanes x 16 bytes; element 0 of lane 0
// is the line's count flag, the other 128/e - 1 elements are data. Every
// rank adds its data of segment s into owner s's line with vector
// reductions in the element type; after a fence, lane 0 adds 1 to the
// flag. When the owner's flag reads N, every contribution is in. The owner
// publishes its reduced lines once, as LL lines in its own staging, which
// every peer polls (AllGather), and zeroes its lines for their next use
// (epoch + 2).
template <int DT>
__device__ __forceinline__ void red_add_v4(void* a, const unsigned* w) {
  if (DT == 0)
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                 :: "l"(a), "f"(__uint_as_float(w[0])), "f"(__uint_as_float(w[1])),
                    "f"(__uint_as_float(w[2])), "f"(__uint_as_float(w[3])) : "memory");
  else if (DT == 1)
    asm volatile("red.relaxed.gpu.global.add.noftz.v4.f16x2 [%0], {%1, %2, %3, %4};"
                 :: "l"(a), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
  else
    asm volatile("red.relaxed.gpu.global.add.noftz.v4.bf16x2 [%0], {%1, %2, %3, %4};"
                 :: "l"(a), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
}
// Count one contribution on a line's flag (element 0). For 16-bit types
// the packed pair {one, -0} is added to the flag's 32-bit word: adding -0
// leaves the neighbouring data element unchanged (x + -0 = x for every x,
// +0 and -0 included, under roundTiesToEven), and the packed reduction is
// a single native operation where the scalar 16-bit one measured 0.7-2.5
// us per issue on B300 (8 ranks, 16 KiB bf16: 5.8 -> see the bench).
template <int DT>
__device__ __forceinline__ void red_add_flag(void* a, unsigned one_bits) {
  if (DT == 0) {
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;"
                 :: "l"(a), "f"(__uint_as_float(one_bits)) : "memory");
  } else {
    const unsigned pair = (one_bits & 0xFFFFu) | (0x8000u << 16);
    if (DT == 1)
      asm volatile("red.relaxed.gpu.global.add.noftz.f16x2 [%0], %1;" :: "l"(a), "r"(pair) : "memory");
    else
      asm volatile("red.relaxed.gpu.global.add.noftz.bf16x2 [%0], %1;" :: "l"(a), "r"(pair) : "memory");
  }
}

// A lane of LL128 line l of segment s carries the V elements at segment
// positions l*P + j*V - 1 + k (k < V; lane 0's k = 0 is the flag): a window
// of 16 bytes that starts one element before a lane boundary, so for
// 63-element (31-element) lines its alignment to the 16-byte vectors of the
// message rotates from line to line. Inside the message the window is read
// with two aligned 16-byte loads and shifted into place, and written with
// at most five naturally aligned stores; windows that reach past the
// segment or the message (or start before it) take elements one by one.
// ll128_window returns false there; ll128_first is the window's first
// element index in the message.
template <int DT>
__device__ __forceinline__ bool ll128_window(size_t count, size_t seg, int s, size_t l, int j, size_t& first) {
  constexpr int V = 16 / Fmt<DT>::kBytes;
  constexpr int P = 128 / Fmt<DT>::kBytes - 1;
  const size_t sl0 = l * P + (size_t)j * V;  // segment position of element k = 1
  const size_t base = (size_t)s * seg;
  const size_t lim = min(seg, count - min(count, base));  // elements of segment s
  first = base + sl0 - 1;
  return sl0 + V - 1 <= lim && base + sl0 >= 1;
}
// the V elements at `first` as 4 packed words, for an in-message window
// whose two covering vectors lie inside the buffer (`nbytes` long)
template <int DT>
__device__ __forceinline__ bool ll128_gather_fast(const char* src, size_t first, size_t nbytes, unsigned w[4]) {
  const size_t off = first * Fmt<DT>::kBytes;
  const size_t vb = off & ~(size_t)15;
  const unsigned h = (unsigned)(off & 15) >> 1;  // 16-bit halves into the vector
  if (h != 0 && vb + 32 > nbytes) return false;
  const uint4 a = *reinterpret_cast<const uint4*>(src + vb);
  const uint4 b = h ? *reinterpret_cast<const uint4*>(src + vb + 16) : make_uint4(0, 0, 0, 0);
  unsigned x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  if (h & 4) {
#pragma unroll
    for (int i = 0; i < 6; ++i) x[i] = x[i + 2];
  }
  if (h & 2) {
#pragma unroll
    for (int i = 0; i < 5; ++i) x[i] = x[i + 1];
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = (h & 1) ? __byte_perm(x[i], x[i + 1], 0x5432) : x[i];
  return true;
}
// store the window's elements (all V, or V-1 without element 0 for lane 0)
template <int DT>
__device__ __forceinline__ void ll128_scatter_fast(char* dst, size_t first, bool skip0, const unsigned w[4]) {
  char* b = dst + first * Fmt<DT>::kBytes;
  if (Fmt<DT>::kBytes == 4) {
    if (!skip0 && (first & 3) == 0) {
      *reinterpret_cast<uint4*>(b) = make_uint4(w[0], w[1], w[2], w[3]);
      return;
    }
    if (!skip0) *reinterpret_cast<unsigned*>(b) = w[0];
#pragma unroll
    for (int i = 1; i < 4; ++i) *reinterpret_cast<unsigned*>(b + 4 * i) = w[i];
    return;
  }
  if (!skip0 && (first & 7) == 0) {
    *reinterpret_cast<uint4*>(b) = make_uint4(w[0], w[1], w[2], w[3]);
  } else if ((first & 1) == 0) {
    if (skip0) *reinterpret_cast<unsigned short*>(b + 2) = (unsigned short)(w[0] >> 16);
    else *reinterpret_cast<unsigned*>(b) = w[0];
#pragma unroll
    for (int i = 1; i < 4; ++i) *reinterpret_cast<unsigned*>(b + 4 * i) = w[i];
  } else {
    if (!skip0) *reinterpret_cast<unsigned short*>(b) = (unsigned short)w[0];
#pragma unroll
    for (int i = 0; i < 3; ++i) *reinterpret_cast<unsigned*>(b + 2 + 4 * i) = __byte_perm(w[i], w[i + 1], 0x5432);
    *reinterpret_cast<unsigned short*>(b + 14) = (unsigned short)(w[3] >> 16);
  }
}
// element by element (windows at the edges of a segment or the message)
template <int DT>
__device__ __forceinline__ bool ll128_gather_slow(const char* src, size_t count, size_t seg, int s, size_t l, int j,
                                                  unsigned w[4]) {
  constexpr int EB = Fmt<DT>::kBytes;
  constexpr int V = 16 / EB;
  constexpr int P = 128 / EB - 1;
  bool any = false;
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int pos = j * V + k;
    const size_t sl = l * P + (size_t)pos - 1;
    const size_t g = (size_t)s * seg + sl;
    unsigned b = 0;
    if (pos >= 1 && sl < seg && g < count) {
      b = Fmt<DT>::load(src, g);
      any = true;
    }
    const int word = (k * EB) / 4, sub = (EB == 4) ? 0 : (k & 1);
    if (EB == 4) w[word] = b;
    else w[word] = sub ? (w[word] | (b << 16)) : b;
  }
  return any;
}
template <int DT>
__device__ __forceinline__ void ll128_scatter_slow(char* dst, size_t dst_off, size_t count, size_t seg, int s, size_t l,
                                                   int j, const unsigned w[4]) {
  constexpr int EB = Fmt<DT>::kBytes;
  constexpr int V = 16 / EB;
  constexpr int P = 128 / EB - 1;
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int pos = j * V + k;
    const size_t sl = l * P + (size_t)pos - 1;
    const size_t g = (size_t)s * seg + sl;
    if (pos >= 1 && sl < seg && g < count)
      Fmt<DT>::store(dst, g - dst_off, word_elem<DT>(w[(k * EB) / 4], (EB == 4) ? 0 : (k & 1)));
  }
}
// lane j of line l of segment s: gather my input (zero where no element)
template <int DT>
__device__ __forceinline__ bool ll128_gather(const char* src, size_t count, size_t seg, int s, size_t l, int j,
                                             unsigned w[4]) {
  size_t first;
  if (ll128_window<DT>(count, seg, s, l, j, first) &&
      ll128_gather_fast<DT>(src, first, count * Fmt<DT>::kBytes, w)) {
    if (j == 0) w[0] &= (Fmt<DT>::kBytes == 4) ? 0u : 0xFFFF0000u;  // the flag's element
    return true;
  }
  return ll128_gather_slow<DT>(src, count, seg, s, l, j, w);
}
// store lane j of line l of segment s; message element g goes to dst
// element g - dst_off (0: a whole-message output; s * seg: a segment output)
template <int DT>
__device__ __forceinline__ void ll128_scatter(char* dst, size_t dst_off, size_t count, size_t seg, int s, size_t l,
                                              int j, const unsigned w[4]) {
  size_t first;
  if (ll128_window<DT>(count, seg, s, l, j, first) && first >= dst_off)
    ll128_scatter_fast<DT>(dst, first - dst_off, j == 0, w);
  else ll128_scatter_slow<DT>(dst, dst_off, count, seg, s, l, j, w);
}

template <int DT>
__device__ __forceinline__ void body_ll128(const Params& p, const u64 epoch0) {
  constexpr int EB = Fmt<DT>::kBytes;
  constexpr int EL = 128 / EB;  // elements per line
  constexpr int P = EL - 1;     // data elements per line
  const int N = p.nranks;
  const int r = rank_of_block(p);
  const int c = cta_of_block(p);
  const size_t count = p.count;
  const size_t seg = (count + N - 1) / N;
  const size_t L = (seg + P - 1) / P;
  const size_t Lc = (L + p.G - 1) / p.G;
  const size_t l0 = min(L, (size_t)c * Lc);
  const size_t nl = min(L, l0 + Lc) - l0;
  // items of this CTA: (segment, line, lane), lane fastest; fewer than
  // 2^32 (LL128 messages are at most 1 GiB per rank: a segment of at most
  // 2^28 elements has under 2^23 lines)
  const unsigned per_seg = (unsigned)(nl * kLL128Lanes);
  const unsigned items = (unsigned)N * per_seg;
  const unsigned T = blockDim.x;
  const unsigned one_bits = Fmt<DT>::from_f(1.0f);
  const unsigned n_bits = Fmt<DT>::from_f((float)N);
  const unsigned flag_mask = (EB == 4) ? 0xFFFFFFFFu : 0xFFFFu;
  const bool injected = (p.inject_rank == r);
  const bool skip = injected && p.inject_mode == LLAR_INJECT_SKIP_;
  const bool poison = injected && p.inject_mode == LLAR_INJECT_POISON_;
  const size_t line_slot = p.l128_lines * (size_t)kLL128Line;
  // AllGather lines are published once, in the owner's own staging
  // [slot][line][lane]; every peer polls them there (as the LL one-shot:
  // on one GPU a peer's load and a push into the peer's staging meet in
  // the same L2, and one store replaces N-1)
  const size_t ag_slot = p.l128_lines * (size_t)kAgLineBytes;
  char* const my_lines = p.l128 + (size_t)r * p.l128_stride;
  char* const my_ag = p.l128ag + (size_t)r * p.l128ag_stride;
  bool failed = false;

  for (int e = 0; e < p.iters; ++e) {
    const u64 E = epoch0 + (u64)e;
    const int slot = (int)(E & 1);
    const char* src = rank_input<DT>(p, r, e);
    char* dst = rank_output<DT>(p, r, e);
    if (injected && p.inject_mode == LLAR_INJECT_DELAY_) injected_delay();

    // ---- ReduceScatter: add my data into every owner's lines
    if (!skip) {
      for (unsigned i = threadIdx.x; i < items; i += T) {
        const int s = (int)(i / per_seg);
        const unsigned rem = i - (unsigned)s * per_seg;
        const size_t l = l0 + rem / kLL128Lanes;
        const int j = (int)(rem % kLL128Lanes);
        unsigned w[4];
        if (ll128_gather<DT>(src, count, seg, s, l, j, w))
          red_add_v4<DT>(p.l128 + (size_t)s * p.l128_stride + slot * line_slot + l * kLL128Line + j * 16, w);
      }
    }
    __syncwarp();
    fence_gpu();  // every data reduction of this warp before its flags
    if (!skip) {
      for (unsigned i = threadIdx.x; i < items; i += T) {
        if ((i % kLL128Lanes) != 0) continue;
        const int s = (int)(i / per_seg);
        const size_t l = l0 + (i - (unsigned)s * per_seg) / kLL128Lanes;
        red_add_flag<DT>(p.l128 + (size_t)s * p.l128_stride + slot * line_slot + l * kLL128Line,
                         poison ? 0u : one_bits);
      }
    }

    // ---- owner: wait for count N, read, AllGather as LL lines, zero
    for (unsigned base = 0; base < items; base += T) {
      const unsigned i = base + threadIdx.x;
      int s = -1;
      size_t l = 0;
      int j = 0;
      if (i < items) {
        s = (int)(i / per_seg);
        const unsigned rem = i - (unsigned)s * per_seg;
        l = l0 + rem / kLL128Lanes;
        j = (int)(rem % kLL128Lanes);
      }
      const bool own = (s == r);
      char* line = my_lines + slot * line_slot + l * kLL128Line;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (own) {
        if (!failed) {
          Waiter wt;
          for (bool first_round = true;; first_round = false) {
            LLB_ON_POLL_ROUND(first_round, 1u);
            if ((ld_acquire_u32(line) & flag_mask) == n_bits) break;
            if (wt.expired(p)) {
              report_timeout(p, r, c, E);
              failed = true;
              break;
            }
          }
        }
        v = ld_relaxed_v4(line + j * 16);
      }
      __syncwarp();  // all 8 lanes have read the flag and their data before any zeroing
      if (own) {
        const unsigned w[4] = {v.x, v.y, v.z, v.w};
        ll128_scatter<DT>(dst, 0, count, seg, r, l, j, w);
        if (p.chain) {
          unsigned nx[4];
          chain_words<DT, 4>(w, nx, p.chain_scale);
          ll128_scatter<DT>(chain_next_buf(p, r, e), 0, count, seg, r, l, j, nx);
        }
        if (!skip) {
          const u64 lo = (u64)v.x | ((u64)v.y << 32);
          const u64 hi = (u64)v.z | ((u64)v.w << 32);
          const u64 flag = poison ? E + 2 : E;
          char* ag = my_ag + slot * ag_slot + l * kAgLineBytes + j * 32;
          st_relaxed_b128(ag, lo, flag);
          st_relaxed_b128(ag + 16, hi, flag);
        }
        st_relaxed_v4(line + j * 16, make_uint4(0, 0, 0, 0));
      }
    }

    // ---- AllGather receive: poll the owners' LL lines, write my output
    for (unsigned i = threadIdx.x; i < items; i += T) {
      const int s = (int)(i / per_seg);
      if (s == r) continue;
      const unsigned rem = i - (unsigned)s * per_seg;
      const size_t l = l0 + rem / kLL128Lanes;
      const int j = (int)(rem % kLL128Lanes);
      const char* ag = p.l128ag + (size_t)s * p.l128ag_stride + slot * ag_slot + l * kAgLineBytes + j * 32;
      u64 lo = 0, hi = 0;
      if (!failed) {
        Waiter wt;
        bool got0 = false, got1 = false;
        for (bool first_round = true;; first_round = false) {
          LLB_ON_POLL_ROUND(first_round, (got0 ? 0u : 1u) | (got1 ? 0u : 2u));
          u64 a0, f0, a1, f1;
          if (!got0) ld_relaxed_b128(ag, a0, f0);
          if (!got1) ld_relaxed_b128(ag + 16, a1, f1);
          if (!got0 && f0 == E) { lo = a0; got0 = true; }
          if (!got1 && f1 == E) { hi = a1; got1 = true; }
          if (got0 && got1) break;
          if (wt.expired(p)) {
            report_timeout(p, r, c, E);
            failed = true;
            break;
          }
        }
      }
      const unsigned w[4] = {(unsigned)lo, (unsigned)(lo >> 32), (unsigned)hi, (unsigned)(hi >> 32)};
      ll128_scatter<DT>(dst, 0, count, seg, s, l, j, w);
      if (p.chain) {
        unsigned nx[4];
        chain_words<DT, 4>(w, nx, p.chain_scale);
        ll128_scatter<DT>(chain_next_buf(p, r, e), 0, count, seg, s, l, j, nx);
      }
    }
    if (__any_sync(0xFFFFFFFFu, failed)) return;
  }
}

// Technique 4 with the AllGather read straight from the owners' lines (a
// variant beside the pages' LL AllGather): the ReduceScatter is the same
// (data reductions into owner s's line, a fence, the count), but instead of
// the owner reading its lines and publishing them again as LL lines, every
// rank polls each owner's line until the count reads N (acquire) and reads
// the reduced data there. That removes one store -> load hop and the LL
// copy of every segment. Lines then stay read for an AllReduce after their
// count completes, so each owner keeps three slots in turn: sequence
// number s (a per-context counter of these AllReduces, advanced like the
// epoch) uses slot s % 3, and when the owner sees the count of its line in
// slot s % 3 reach N it zeroes the same line in slot (s - 1) % 3. That is
// safe: each contributor added to slot s % 3 after (program order, then the
// fence before its count) it had read every line of s - 1. The zeroed slot
// is next used by s + 2, whose additions each contributor makes only after
// it saw the count N of s + 1 on that owner's line, which includes the
// owner's own count, added after a fence that follows the zeroing. After a
// launch only the last slot holds data, in the lines that launch used (its
// line count is kept beside the sequence counter); the next launch's first
// AllReduce zeroes all of them at once (the launch boundary orders every
// read of that slot before), since its own, possibly fewer, lines would
// leave the rest.
template <int DT>
__device__ __forceinline__ void body_ll128d(const Params& p, const u64 epoch0, const u64 seq0,
                                            const size_t lines_prev) {
  constexpr int EB = Fmt<DT>::kBytes;
  constexpr int EL = 128 / EB;  // elements per line
  constexpr int P = EL - 1;     // data elements per line
  const int N = p.nranks;
  const int r = rank_of_block(p);
  const int c = cta_of_block(p);
  const size_t count = p.count;
  const size_t seg = (count + N - 1) / N;
  const size_t L = (seg + P - 1) / P;
  const size_t Lc = (L + p.G - 1) / p.G;
  const size_t l0 = min(L, (size_t)c * Lc);
  const size_t nl = min(L, l0 + Lc) - l0;
  const unsigned per_seg = (unsigned)(nl * kLL128Lanes);  // fewer than 2^32 items, as in body_ll128
  const unsigned items = (unsigned)N * per_seg;
  const unsigned T = blockDim.x;
  const unsigned one_bits = Fmt<DT>::from_f(1.0f);
  const unsigned n_bits = Fmt<DT>::from_f((float)N);
  const unsigned flag_mask = (EB == 4) ? 0xFFFFFFFFu : 0xFFFFu;
  const bool injected = (p.inject_rank == r);
  const bool skip = injected && p.inject_mode == LLAR_INJECT_SKIP_;
  const bool poison = injected && p.inject_mode == LLAR_INJECT_POISON_;
  const size_t line_slot = p.l128_lines * (size_t)kLL128Line;
  char* const my_lines = p.l128d + (size_t)r * p.l128d_stride;
  bool failed = false;
  {
    // the previous launch's last slot, every line it used, my segment:
    // this CTA's share of (line, lane) items
    const size_t Lp = min(lines_prev, (size_t)p.l128_lines);
    const size_t Lpc = (Lp + p.G - 1) / p.G;
    const size_t lp0 = min(Lp, (size_t)c * Lpc), lp1 = min(Lp, lp0 + Lpc);
    char* const last = my_lines + (size_t)(seq0 % 3) * line_slot;
    for (size_t i = lp0 * kLL128Lanes + threadIdx.x; i < lp1 * kLL128Lanes; i += T)
      st_relaxed_v4(last + i * 16, make_uint4(0, 0, 0, 0));
  }

  for (int e = 0; e < p.iters; ++e) {
    const u64 E = epoch0 + (u64)e;
    const u64 sq = seq0 + 1 + (u64)e;
    const size_t slot = (size_t)(sq % 3), prev = (size_t)((sq + 2) % 3);
    const char* src = rank_input<DT>(p, r, e);
    char* dst = rank_output<DT>(p, r, e);
    if (injected && p.inject_mode == LLAR_INJECT_DELAY_) injected_delay();

    // ---- ReduceScatter: add my data into every owner's lines
    if (!skip) {
      for (unsigned i = threadIdx.x; i < items; i += T) {
        const int s = (int)(i / per_seg);
        const unsigned rem = i - (unsigned)s * per_seg;
        const size_t l = l0 + rem / kLL128Lanes;
        const int j = (int)(rem % kLL128Lanes);
        unsigned w[4];
        if (ll128_gather<DT>(src, count, seg, s, l, j, w))
          red_add_v4<DT>(p.l128d + (size_t)s * p.l128d_stride + slot * line_slot + l * kLL128Line + j * 16, w);
      }
    }
    __syncwarp();
    fence_gpu();  // every data reduction (and zeroing) of this warp before its counts
    if (!skip) {
      for (unsigned i = threadIdx.x; i < items; i += T) {
        if ((i % kLL128Lanes) != 0) continue;
        const int s = (int)(i / per_seg);
        const size_t l = l0 + (i - (unsigned)s * per_seg) / kLL128Lanes;
        red_add_flag<DT>(p.l128d + (size_t)s * p.l128d_stride + slot * line_slot + l * kLL128Line,
                         poison ? 0u : one_bits);
      }
    }

    // ---- AllGather: every owner's line, once its count reads N
    for (unsigned i = threadIdx.x; i < items; i += T) {
      const int s = (int)(i / per_seg);
      const unsigned rem = i - (unsigned)s * per_seg;
      const size_t l = l0 + rem / kLL128Lanes;
      const int j = (int)(rem % kLL128Lanes);
      const char* line = p.l128d + (size_t)s * p.l128d_stride + slot * line_slot + l * kLL128Line;
      if (!failed) {
        Waiter wt;
        for (bool first_round = true;; first_round = false) {
          LLB_ON_POLL_ROUND(first_round, 1u);
          if ((ld_acquire_u32(line) & flag_mask) == n_bits) break;
          if (wt.expired(p)) {
            report_timeout(p, r, c, E);
            failed = true;
            break;
          }
        }
      }
      if (failed) continue;
      const uint4 v = ld_relaxed_v4(line + j * 16);
      const unsigned w[4] = {v.x, v.y, v.z, v.w};
      ll128_scatter<DT>(dst, 0, count, seg, s, l, j, w);
      if (p.chain) {
        unsigned nx[4];
        chain_words<DT, 4>(w, nx, p.chain_scale);
        ll128_scatter<DT>(chain_next_buf(p, r, e), 0, count, seg, s, l, j, nx);
      }
      // the owner: every contributor has read this line's previous slot
      if (s == r) st_relaxed_v4(my_lines + prev * line_slot + l * kLL128Line + j * 16, make_uint4(0, 0, 0, 0));
    }
    if (__any_sync(0xFFFFFFFFu, failed)) return;
  }
}

template <int DT>
__global__ void __launch_bounds__(kMaxThreads) k_ll128d(const Params p) {
  const u64 epoch0 = launch_epoch(p);
  const u64 seq0 = *reinterpret_cast<volatile const u64*>(p.l128d_seq);
  const u64 lines_prev = *reinterpret_cast<volatile const u64*>(p.l128d_seq + 1);
  body_ll128d<DT>(p, epoch0, seq0, (size_t)lines_prev);
  // as k_ll128: rank 0's CTA c waited for every contribution to every line
  // of its range, each made after its CTA read both counters; the last of
  // rank 0's CTAs advances the sequence counter with the epoch
  __syncthreads();
  if (threadIdx.x == 0 && rank_of_block(p) == 0) {
    if (atomicAdd(p.done_count, 1u) == (unsigned)p.G - 1) {
      *reinterpret_cast<volatile unsigned*>(p.done_count) = 0u;
      *reinterpret_cast<volatile u64*>(p.epoch_dev) = epoch0 - 1 + (u64)p.iters;
      volatile u64* sp = p.l128d_seq;
      *sp = seq0 + (u64)p.iters;
      // the lines of every segment this launch used (the same in every AllReduce)
      const size_t seg = (p.count + p.nranks - 1) / p.nranks;
      sp[1] = (u64)((seg + (128 / Fmt<DT>::kBytes - 1) - 1) / (128 / Fmt<DT>::kBytes - 1));
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kMaxThreads) k_ll128(const Params p) {
  const u64 epoch0 = launch_epoch(p);
  body_ll128<DT>(p, epoch0);
  // rank 0's CTA c waited for every contribution to its own lines and for
  // every other owner's AllGather lines of its range, which each owner sent
  // only after all contributions to them: every working thread of column c
  // had read the counter
  finish_launch(p, epoch0, rank_of_block(p) == 0, (unsigned)p.G);
}

// ==================================================== fixed-order paths
// Deterministic direct-read variants: the reader loads every rank's input
// itself, adds in rank order 0..N-1 in float32 and rounds once. Inputs of a
// launch are complete when it starts (stream order), so without a chain no
// flag is needed. In a chain, the next input of rank q is written by rank q
// into its double-buffered chain slot, and CTA c publishes epoch flags for
// its range: ready[q][c] (input of epoch E is in place, and q's reads of
// epoch E-1 are done) and, for the two-shot, done[s][c] (owner s wrote
// segment s, range c, of every output for epoch E).
__device__ __forceinline__ unsigned long long* flag_ptr(const Params& p, int rank, int cta, int kind) {
  return p.flags + ((size_t)rank * p.flags_gmax + cta) * kFlagKinds + kind;
}

// Thread 0 waits until flag[q][c][kind] >= want for every q != skip_rank;
// the result is shared with the CTA through a barrier. Returns false on timeout.
// Lane q of the first warp waits for rank q's flag, so the N - 1 waits run
// side by side: one round trip once the flags are set, where one thread
// polling them in turn paid one per rank (8 ranks, bf16, chained, us per
// AllReduce: two-shot 15.0 -> 11.7 at 64 KiB, one-shot 6.1 -> 4.5 at
// 16 KiB).
__device__ __forceinline__ bool wait_flags(const Params& p, int skip_rank, int c, int kind, u64 want,
                                           int my_rank, u64 E, int* s_fail) {
  if (threadIdx.x < 32) {
    const int q = (int)threadIdx.x;
    int fail = 0;
    if (q < p.nranks && q != skip_rank) {
      Waiter wt;
      while (ld_acquire_u64(flag_ptr(p, q, c, kind)) < want) {
        if (wt.expired(p)) {
          report_timeout(p, my_rank, c, E);
          fail = 1;
          break;
        }
      }
    }
    fail = __any_sync(0xFFFFFFFFu, fail);
    if (q == 0) *s_fail = fail;
  }
  __syncthreads();
  return *s_fail == 0;
}
__device__ __forceinline__ void publish_flag(const Params& p, int rank, int c, int kind, u64 value) {
  __syncthreads();
  if (p.inject_rank == rank && p.inject_mode == LLAR_INJECT_SKIP_) return;  // a rank that never signals
  if (p.inject_rank == rank && p.inject_mode == LLAR_INJECT_DELAY_ && threadIdx.x == 0) injected_delay();
  if (threadIdx.x == 0) {
    fence_gpu();
    st_relaxed_u64(flag_ptr(p, rank, c, kind), value);
  }
}

// Sum of vector v over all ranks' inputs of iteration e, rank order,
// float32, one rounding. `full` vectors are loaded whole; the last vector of
// a ragged message element by element.
// Sum of the 16-byte vectors x[0..N) element by element: rank order,
// float32, one rounding.
template <int DT>
__device__ __forceinline__ uint4 add_in_rank_order(const uint4 (&x)[kMaxRanks], int N) {
  constexpr int PER16 = 16 / Fmt<DT>::kBytes;
  float acc[PER16];
  {
    const unsigned w4[4] = {x[0].x, x[0].y, x[0].z, x[0].w};
    init_acc<DT, 4>(acc, w4);
  }
#pragma unroll
  for (int q = 1; q < kMaxRanks; ++q)
    if (q < N) {
      const unsigned w4[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
      accumulate<DT, 4>(acc, w4);
    }
  unsigned y[4];
  pack_acc<DT, 4>(acc, y);
  return u4(y);
}

// Sum of vector v over all ranks' inputs of iteration e, rank order,
// float32, one rounding. `full` vectors are loaded whole; the last vector of
// a ragged message element by element.
template <int DT>
__device__ __forceinline__ uint4 sum_ranks_vec(const Params& p, int e, size_t v, bool stream) {
  const int N = p.nranks;
  uint4 x[kMaxRanks];
#pragma unroll
  for (int q = 0; q < kMaxRanks; ++q)
    if (q < N) x[q] = load_vec16<DT>(rank_input<DT>(p, q, e), v, p.count, stream);
  return add_in_rank_order<DT>(x, N);
}

// Reduce vectors [v0, v1) of iteration e and store the result to rank
// `only`'s output (one-shot) or, with only < 0, to every rank's output
// (two-shot AllGather by direct writes). Full vectors go through an
// unrolled loop that keeps 2N 16-byte loads in flight per thread.
template <int DT>
__device__ __forceinline__ void reduce_range(const Params& p, int e, size_t v0, size_t v1, bool stream,
                                             int only) {
  constexpr int PER16 = 16 / Fmt<DT>::kBytes;
  const int N = p.nranks;
  const size_t T = blockDim.x;
  const size_t nfull = p.count / PER16;
  const size_t h1 = v1 < nfull ? v1 : nfull;
  size_t v = v0 + threadIdx.x;
  for (; v + T < h1; v += 2 * T) {
    const uint4 ya = sum_ranks_vec<DT>(p, e, v, stream);
    const uint4 yb = sum_ranks_vec<DT>(p, e, v + T, stream);
    if (only >= 0) {
      char* o = rank_output<DT>(p, only, e);
      st_v4(o + v * 16, ya);
      st_v4(o + (v + T) * 16, yb);
    } else {
#pragma unroll
      for (int q = 0; q < kMaxRanks; ++q)
        if (q < N) {
          char* o = rank_output<DT>(p, q, e);
          st_v4(o + v * 16, ya);
          st_v4(o + (v + T) * 16, yb);
        }
    }
  }
  for (; v < v1; v += T) {
    const uint4 y = sum_ranks_vec<DT>(p, e, v, stream);
#pragma unroll
    for (int q = 0; q < kMaxRanks; ++q)
      if (q < N && (only < 0 || q == only)) store_vec16<DT>(rank_output<DT>(p, q, e), v, p.count, y);
  }
}

template <int DT>
__device__ __forceinline__ void chain_range(const Params& p, int r, int e, size_t v0, size_t v1) {
  const char* y_src = rank_output<DT>(p, r, e);
  char* nxt = chain_next_buf(p, r, e);
  for (size_t v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
    const uint4 y = load_vec16<DT>(y_src, v, p.count, false);
    const unsigned w4[4] = {y.x, y.y, y.z, y.w};
    unsigned nx[4];
    chain_words<DT, 4>(w4, nx, p.chain_scale);
    store_vec16<DT>(nxt, v, p.count, u4(nx));
  }
}

template <int DT>
__device__ __forceinline__ void body_fixed_oneshot(const Params& p, const u64 epoch0) {
  constexpr int PER16 = 16 / Fmt<DT>::kBytes;
  __shared__ int s_fail;
  const int r = rank_of_block(p);
  const int c = cta_of_block(p);
  const size_t NV = (p.count + PER16 - 1) / PER16;
  const size_t per = (NV + p.G - 1) / p.G;
  const size_t v0 = min(NV, (size_t)c * per);
  const size_t v1 = min(NV, v0 + per);
  for (int e = 0; e < p.iters; ++e) {
    const u64 E = epoch0 + (u64)e;
    if (p.chain && e > 0 && !wait_flags(p, r, c, 0, E, r, E, &s_fail)) return;
    reduce_range<DT>(p, e, v0, v1, !p.chain || e == 0, r);
    if (p.chain) {
      // my own output was written by this CTA: the barrier in publish_flag
      // is not needed for it, each thread re-reads what it stored
      chain_range<DT>(p, r, e, v0, v1);
      publish_flag(p, r, c, 0, E + 1);
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kMaxThreads) k_fixed_oneshot(const Params p) {
  const u64 epoch0 = launch_epoch(p);
  body_fixed_oneshot<DT>(p, epoch0);
  finish_launch(p, epoch0);
}

// Two-shot: rank s owns vectors [s*ceil(NV/N), ...) of the message; CTA c
// of every rank covers sub-range c of every segment.
template <int DT>
__device__ __forceinline__ void body_fixed_twoshot(const Params& p, const u64 epoch0) {
  constexpr int PER16 = 16 / Fmt<DT>::kBytes;
  __shared__ int s_fail;
  const int N = p.nranks;
  const int r = rank_of_block(p);
  const int c = cta_of_block(p);
  const size_t NV = (p.count + PER16 - 1) / PER16;
  const size_t segv = (NV + N - 1) / N;
  const size_t per = (segv + p.G - 1) / p.G;
  auto sub = [&](int s, size_t& v0, size_t& v1) {
    const size_t sbeg = min(NV, (size_t)s * segv);
    const size_t send = min(NV, sbeg + segv);
    v0 = min(send, sbeg + (size_t)c * per);
    v1 = min(send, v0 + per);
  };
  for (int e = 0; e < p.iters; ++e) {
    const u64 E = epoch0 + (u64)e;
    // phase 1, owner of segment r: reduce sub-range c, write it to every rank
    if (p.chain && e > 0 && !wait_flags(p, r, c, 0, E, r, E, &s_fail)) return;
    size_t v0, v1;
    sub(r, v0, v1);
    reduce_range<DT>(p, e, v0, v1, !p.chain || e == 0, -1);
    if (!p.chain) continue;
    publish_flag(p, r, c, 1, E);
    if (e + 1 == p.iters) continue;  // no next input after the last step
    // phase 2, rank r: once every owner wrote sub-range c of its segment
    // into my output, compute my next input there
    if (!wait_flags(p, r, c, 1, E, r, E, &s_fail)) return;
    for (int s = 0; s < N; ++s) {
      sub(s, v0, v1);
      chain_range<DT>(p, r, e, v0, v1);
    }
    publish_flag(p, r, c, 0, E + 1);
  }
}

template <int DT>
__global__ void __launch_bounds__(kMaxThreads) k_fixed_twoshot(const Params p) {
  const u64 epoch0 = launch_epoch(p);
  body_fixed_twoshot<DT>(p, epoch0);
  finish_launch(p, epoch0);
}

// Large two-shot without a chain: the owner's CTAs stream their sub-range
// through shared memory with TMA bulk copies. Stage k of a kBulkStages-deep
// ring holds one tile (kBulkTileBytes) of every rank's input, filled by one
// thread with N cp.async.bulk copies that complete on the stage's mbarrier.
// All threads wait for the stage, add the N tiles in rank order (float32,
// one rounding) and store the result to every rank's output; after a CTA
// barrier the same thread refills the stage with the tile kBulkStages
// further on. Tiles of every iteration form one sequence, so the ring keeps
// running across iterations. Measured at 8 x 64 MiB bf16: one stage of
// 20 KiB tiles (160 KiB of shared memory, one CTA per SM) beats deeper
// rings (3 x 8 KiB: 5.4 TB/s, 2 x 8 KiB: 5.8, 1 x 20 KiB: 5.9): with more
// reads in flight the writes of the same kernel lose DRAM time.
#ifndef LLAR_BULK_STAGES
#define LLAR_BULK_STAGES 1
#endif
#ifndef LLAR_BULK_TILE
#define LLAR_BULK_TILE 20480
#endif
#ifndef LLAR_BULK_CS
#define LLAR_BULK_CS 0
#endif
constexpr int kBulkStages = LLAR_BULK_STAGES;
constexpr int kBulkTileBytes = LLAR_BULK_TILE;

template <int DT>
__device__ __forceinline__ void body_fixed_twoshot_bulk(const Params& p, const u64 epoch0) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int PER16 = 16 / Fmt<DT>::kBytes;
  constexpr unsigned TV = kBulkTileBytes / 16;  // vectors per tile
  const int N = p.nranks;
  const int r = rank_of_block(p);
  const int c = cta_of_block(p);
  const size_t NV = (p.count + PER16 - 1) / PER16;
  const size_t nfull = p.count / PER16;
  const size_t segv = (NV + N - 1) / N;
  const size_t per = (segv + p.G - 1) / p.G;
  const size_t sbeg = min(NV, (size_t)r * segv);
  const size_t send = min(NV, sbeg + segv);
  const size_t v0 = min(send, sbeg + (size_t)c * per);
  const size_t v1 = min(send, v0 + per);
  const size_t v1f = min(v1, nfull);  // full vectors go through the ring
  const size_t span = v1f > v0 ? v1f - v0 : 0;
  const unsigned tiles = (unsigned)((span + TV - 1) / TV);
  const unsigned long long total = (unsigned long long)tiles * p.iters;
  const size_t stage_bytes = (size_t)N * kBulkTileBytes;
  const unsigned base = smem_addr(smem);
  const unsigned bars = base + (unsigned)(kBulkStages * stage_bytes);
  (void)epoch0;

  if (threadIdx.x == 0) {
    for (int k = 0; k < kBulkStages; ++k) mbar_init(bars + 8 * k, 1);
    fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](unsigned long long g) {
    const int e = (int)(g / tiles);
    const unsigned t = (unsigned)(g % tiles);
    const int k = (int)(g % kBulkStages);
    const size_t vb = v0 + (size_t)t * TV;
    const unsigned nv = (unsigned)min((size_t)TV, v1f - vb);
    mbar_arrive_expect_tx(bars + 8 * k, nv * 16u * (unsigned)N);
    for (int q = 0; q < N; ++q)
      bulk_load(base + (unsigned)(k * stage_bytes + (size_t)q * kBulkTileBytes),
                rank_input<DT>(p, q, e) + vb * 16, nv * 16u, bars + 8 * k);
  };
  if (threadIdx.x == 0)
    for (unsigned long long g = 0; g < total && g < (unsigned long long)kBulkStages; ++g) issue(g);

  bool failed = false;
  for (unsigned long long g = 0; g < total; ++g) {
    const int e = (int)(g / tiles);
    const unsigned t = (unsigned)(g % tiles);
    const int k = (int)(g % kBulkStages);
    const unsigned parity = (unsigned)((g / kBulkStages) & 1u);
    const size_t vb = v0 + (size_t)t * TV;
    const unsigned nv = (unsigned)min((size_t)TV, v1f - vb);
    if (!failed) {
      unsigned spins = 0;
      u64 deadline = 0;
      while (!mbar_try_wait(bars + 8 * k, parity)) {
        if ((++spins & 1023u) == 0u) {
          const u64 now = globaltimer_ns();
          if (deadline == 0) deadline = now + p.timeout_ns;
          if (now > deadline) {
            report_timeout(p, r, c, epoch0 + (u64)e);
            failed = true;
            break;
          }
        }
      }
    }
    const unsigned sb = base + (unsigned)(k * stage_bytes);
    for (unsigned v = threadIdx.x; v < nv; v += blockDim.x) {
      float acc[PER16];
      for (int q = 0; q < N; ++q) {
        const uint4 x = ld_shared_v4(sb + (unsigned)q * kBulkTileBytes + v * 16u);
        const unsigned w4[4] = {x.x, x.y, x.z, x.w};
        acc_words<DT, 4>(acc, w4, q == 0);
      }
      unsigned y[4];
      round_words<DT, 4>(acc, y);
      const uint4 yv = u4(y);
      if (LLAR_BULK_CS)
        for (int q = 0; q < N; ++q) st_cs_v4(rank_output<DT>(p, q, e) + (vb + v) * 16, yv);
      else
        for (int q = 0; q < N; ++q) st_v4(rank_output<DT>(p, q, e) + (vb + v) * 16, yv);
    }
    __syncthreads();  // every thread is done with stage k
    if (threadIdx.x == 0 && !failed && g + kBulkStages < total) issue(g + kBulkStages);
  }
  // the ragged last vector of the message, if it falls in my range
  if (v0 <= nfull && nfull < v1 && nfull < NV && threadIdx.x == 0)
    for (int e = 0; e < p.iters; ++e) {
      const uint4 y = sum_ranks_vec<DT>(p, e, v1f, true);
      for (int q = 0; q < N; ++q) store_vec16<DT>(rank_output<DT>(p, q, e), v1f, p.count, y);
    }
}

template <int DT>
__global__ void __launch_bounds__(kMaxThreads) k_fixed_twoshot_bulk(const Params p) {
  const u64 epoch0 = launch_epoch(p);
  body_fixed_twoshot_bulk<DT>(p, epoch0);
  finish_launch(p, epoch0);
}

// ============================================ ReduceScatter / AllGather
// The two halves of the two-shot AllReduce as collectives of their own
// ("zcube network architecture for LLM inference", collectives table, rows
// Reduce-Scatter and All-Gather; "Every Microsecond Matters", technique 4).
// Segment s of a count-element vector is [s*S, min(count, (s+1)*S)) with
// S = ceil(count/N). One collective per launch: the launch boundary orders
// every reuse of staging, so no credits are needed inside.
__device__ __forceinline__ void segment_of(size_t count, int N, int s, size_t& lo, size_t& hi) {
  const size_t per = (count + N - 1) / N;
  lo = min(count, (size_t)s * per);
  hi = min(count, lo + per);
}

// ReduceScatter over LL lines: every rank publishes all its words once;
// owner r polls the words of segment r from every peer, adds in rank order
// and stores segment r to out[r].
template <int DT, int N>
__device__ __forceinline__ void body_rs_ll(const Params& p, const u64 E) {
  constexpr int EB = Fmt<DT>::kBytes;
  constexpr int PER8 = 8 / EB;
  const int r = rank_of_block(p);
  const int c = cta_of_block(p);
  const size_t count = p.count;
  const size_t W = (count + PER8 - 1) / PER8;
  char* const mine = p.ll + (size_t)r * p.ll_stride + (size_t)(E & 1) * p.ll_slot_words * kLLLine;
  const bool skip = p.inject_rank == r && p.inject_mode == LLAR_INJECT_SKIP_;
  const u64 flag = (p.inject_rank == r && p.inject_mode == LLAR_INJECT_POISON_) ? E + 2 : E;
  if (p.inject_rank == r && p.inject_mode == LLAR_INJECT_DELAY_) injected_delay();
  const char* src = p.in[r];
  {
    const size_t per = (W + p.G - 1) / p.G;
    const size_t a = min(W, (size_t)c * per), b = min(W, a + per);
    if (!skip)
      for (size_t w = a + threadIdx.x; w < b; w += blockDim.x)
        st_relaxed_b128(mine + w * kLLLine, load_word8<DT>(src, w, count), flag);
  }
  size_t lo, hi;
  segment_of(count, N, r, lo, hi);
  if (lo >= hi) return;
  const size_t wa = lo / PER8, wb = (hi + PER8 - 1) / PER8;
  const size_t per = (wb - wa + p.G - 1) / p.G;
  const size_t a = min(wb, wa + (size_t)c * per), b = min(wb, a + per);
  char* dst = p.out[r];
  for (size_t w = a + threadIdx.x; w < b; w += blockDim.x) {
    const size_t off = (size_t)(E & 1) * p.ll_slot_words * kLLLine + w * kLLLine;
    u64 d[N];
    unsigned pend = ((1u << N) - 1u) & ~(1u << r);
    unsigned spins = 0;
    u64 deadline = 0;
    while (pend) {
      u64 l[N], h[N];
#pragma unroll
      for (int q = 0; q < N; ++q)
        if ((pend >> q) & 1u) ld_relaxed_b128(p.ll + (size_t)q * p.ll_stride + off, l[q], h[q]);
#pragma unroll
      for (int q = 0; q < N; ++q)
        if (((pend >> q) & 1u) && h[q] == E) {
          d[q] = l[q];
          pend &= ~(1u << q);
        }
      if (pend && (++spins & 63u) == 0u) {
        const u64 now = globaltimer_ns();
        if (deadline == 0) deadline = now + p.timeout_ns;
        if (now > deadline || ld_relaxed_u32(p.abort_flag) != 0) {
          report_timeout(p, r, c, E);
          return;
        }
      }
    }
    const u64 own = load_word8<DT>(src, w, count);
    float acc[PER8];
#pragma unroll
    for (int q = 0; q < N; ++q) {
      const u64 v = (q == r) ? own : d[q];
      const unsigned w2[2] = {(unsigned)v, (unsigned)(v >> 32)};
      acc_words<DT, 2>(acc, w2, q == 0);
    }
    unsigned y[2];
    round_words<DT, 2>(acc, y);
#pragma unroll
    for (int k = 0; k < PER8; ++k) {
      const size_t g = w * PER8 + k;
      if (g >= lo && g < hi) Fmt<DT>::store(dst, g - lo, word_elem<DT>(y[(k * EB) / 4], (EB == 4) ? 0 : (k & 1)));
    }
  }
}

// AllGather over LL lines: rank r publishes the words of its segment
// (in[r] holds that segment only); every rank polls every peer's words and
// places them at the segment's offset in its output.
template <int DT, int N>
__device__ __forceinline__ void body_ag_ll(const Params& p, const u64 E) {
  constexpr int EB = Fmt<DT>::kBytes;
  constexpr int PER8 = 8 / EB;
  const int r = rank_of_block(p);
  const int c = cta_of_block(p);
  const size_t count = p.count;
  const size_t S = (count + N - 1) / N;
  const size_t WS = (S + PER8 - 1) / PER8;  // words of the longest segment
  const size_t slot_off = (size_t)(E & 1) * p.ll_slot_words * kLLLine;
  const bool skip = p.inject_rank == r && p.inject_mode == LLAR_INJECT_SKIP_;
  const u64 flag = (p.inject_rank == r && p.inject_mode == LLAR_INJECT_POISON_) ? E + 2 : E;
  if (p.inject_rank == r && p.inject_mode == LLAR_INJECT_DELAY_) injected_delay();
  size_t lo, hi;
  segment_of(count, N, r, lo, hi);
  const size_t my_len = hi - lo;
  const size_t my_words = (my_len + PER8 - 1) / PER8;
  {
    const size_t per = (my_words + p.G - 1) / p.G;
    const size_t a = min(my_words, (size_t)c * per), b = min(my_words, a + per);
    char* mine = p.ll + (size_t)r * p.ll_stride + slot_off;
    if (!skip)
      for (size_t w = a + threadIdx.x; w < b; w += blockDim.x)
        st_relaxed_b128(mine + w * kLLLine, load_word8<DT>(p.in[r], w, my_len), flag);
  }
  // items: (segment q, word w) for all q, split over my CTAs
  const size_t items = (size_t)N * WS;
  const size_t per = (items + p.G - 1) / p.G;
  const size_t a = min(items, (size_t)c * per), b = min(items, a + per);
  char* dst = p.out[r];
  for (size_t i = a + threadIdx.x; i < b; i += blockDim.x) {
    const int q = (int)(i / WS);
    const size_t w = i - (size_t)q * WS;
    size_t qlo, qhi;
    segment_of(count, N, q, qlo, qhi);
    if (w * PER8 >= qhi - qlo) continue;
    u64 v;
    if (q == r) {
      v = load_word8<DT>(p.in[r], w, my_len);
    } else {
      const char* line = p.ll + (size_t)q * p.ll_stride + slot_off + w * kLLLine;
      unsigned spins = 0;
      u64 deadline = 0;
      while (true) {
        u64 hv;
        ld_relaxed_b128(line, v, hv);
        if (hv == E) break;
        if ((++spins & 63u) == 0u) {
          const u64 now = globaltimer_ns();
          if (deadline == 0) deadline = now + p.timeout_ns;
          if (now > deadline || ld_relaxed_u32(p.abort_flag) != 0) {
            report_timeout(p, r, c, E);
            return;
          }
        }
      }
    }
    const unsigned y[2] = {(unsigned)v, (unsigned)(v >> 32)};
#pragma unroll
    for (int k = 0; k < PER8; ++k) {
      const size_t g = qlo + w * PER8 + k;
      if (g < qhi) Fmt<DT>::store(dst, g, word_elem<DT>(y[(k * EB) / 4], (EB == 4) ? 0 : (k & 1)));
    }
  }
}

// Fixed-order ReduceScatter by direct reads: owner r reads segment r of
// every rank's input, adds in rank order, stores to out[r].
template <int DT>
__device__ __forceinline__ void body_rs_fixed(const Params& p, const u64 E) {
  (void)E;
  constexpr int EB = Fmt<DT>::kBytes, PER16 = 16 / EB;
  const int N = p.nranks;
  const int r = rank_of_block(p);
  const int c = cta_of_block(p);
  size_t lo, hi;
  segment_of(p.count, N, r, lo, hi);
  const size_t stride = (size_t)p.G * blockDim.x;
  char* dst = p.out[r];
  if ((((p.count + N - 1) / N) * EB) % 16 == 0 && p.count * EB > kRsVectorMinBytes) {
    // every segment starts on a 16-byte boundary: one vector per item, the N
    // loads of an item in flight together. The test is the same for all
    // ranks: with segments of ragged length, a vector path for the ranks
    // whose segment happens to start aligned made the launch slower (bf16,
    // 5 and 7 ranks x 1 .. 256 KiB: 2.9-3.9 against 1.5-2.6 us). Up to
    // kRsVectorMinBytes per rank one element per thread is faster (more
    // threads share the work: 8 x 16 KiB bf16 1.70 against 1.80 us, 8 x
    // 1 KiB 1.57 against 1.84; from 256 KiB the vectors win, 8 x 1 MiB
    // 2.56 against 3.85)
    const size_t len = hi - lo, nv = (len + PER16 - 1) / PER16;
    for (size_t j = (size_t)c * blockDim.x + threadIdx.x; j < nv; j += stride) {
      uint4 x[kMaxRanks];
#pragma unroll
      for (int q = 0; q < kMaxRanks; ++q)
        if (q < N) x[q] = load_vec16<DT>(p.in[q] + lo * EB, j, len, true);
      store_vec16<DT>(dst, j, len, add_in_rank_order<DT>(x, N));
    }
    return;
  }
  for (size_t g = lo + (size_t)c * blockDim.x + threadIdx.x; g < hi; g += stride) {
    unsigned x[kMaxRanks];
#pragma unroll
    for (int q = 0; q < kMaxRanks; ++q)
      if (q < N) x[q] = Fmt<DT>::load(p.in[q], g);
    float acc = Fmt<DT>::to_f(x[0]);
#pragma unroll
    for (int q = 1; q < kMaxRanks; ++q)
      if (q < N) acc = __fadd_rn(acc, Fmt<DT>::to_f(x[q]));
    Fmt<DT>::store(dst, g - lo, Fmt<DT>::from_f(acc));
  }
}

// Fixed AllGather by direct copies: rank r's CTAs read segment r once and
// store it to every rank's output (as the two-shot's owner does), so each
// input byte is read once; in 16-byte vectors when segments are a whole
// number of them long, element by element otherwise. Measured on a B300
// (bf16, 2..8 ranks, 16 KiB .. 64 MiB per rank) this beat every rank
// reading all N segments into its own output at all but the smallest size
// (8 x 1 MiB: 2.75 against 3.95 us; 8 x 64 MiB: 107 against 134).
template <int DT>
__device__ __forceinline__ void body_ag_fixed(const Params& p, const u64 E) {
  (void)E;
  constexpr int EB = Fmt<DT>::kBytes, PER16 = 16 / EB;
  const int N = p.nranks;
  const int r = rank_of_block(p);
  const int c = cta_of_block(p);
  const size_t stride = (size_t)p.G * blockDim.x;
  const size_t per = (p.count + N - 1) / N;
  size_t lo, hi;
  segment_of(p.count, N, r, lo, hi);
  if ((per * EB) % 16 == 0) {
    const size_t len = hi - lo, nv = (len + PER16 - 1) / PER16;
    for (size_t j = (size_t)c * blockDim.x + threadIdx.x; j < nv; j += stride) {
      const uint4 v = load_vec16<DT>(p.in[r], j, len, true);
#pragma unroll
      for (int q = 0; q < kMaxRanks; ++q)
        if (q < N) store_vec16<DT>(p.out[q] + lo * EB, j, len, v);
    }
    return;
  }
  for (size_t g = lo + (size_t)c * blockDim.x + threadIdx.x; g < hi; g += stride) {
    const unsigned v = Fmt<DT>::load(p.in[r], g - lo);
#pragma unroll
    for (int q = 0; q < kMaxRanks; ++q)
      if (q < N) Fmt<DT>::store(p.out[q], g, v);
  }
}

// Element i of segment s of a rank buffer, as raw bits (0 past the end).
template <int DT>
__device__ __forceinline__ unsigned seg_elem(const char* base, size_t lo, size_t len, size_t i) {
  return i < len ? Fmt<DT>::load(base, lo + i) : 0u;
}
// 16-byte vector j of a segment [lo, lo + len) of a buffer: elements
// [j * PER16, (j + 1) * PER16), zero past the end; one vector load when the
// segment starts on a 16-byte boundary and the vector is whole.
template <int DT>
__device__ __forceinline__ uint4 seg_vec(const char* base, size_t lo, size_t len, size_t j) {
  constexpr int PER16 = 16 / Fmt<DT>::kBytes;
  const size_t first = j * PER16;
  if ((lo * Fmt<DT>::kBytes) % 16 == 0 && first + PER16 <= len)
    return ld_stream_v4(base + (lo + first) * Fmt<DT>::kBytes);
  unsigned w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int k = 0; k < PER16; ++k) {
    const unsigned b = seg_elem<DT>(base, lo, len, first + k);
    const int word = (k * Fmt<DT>::kBytes) / 4;
    w[word] = Fmt<DT>::kBytes == 4 ? b : word_set<DT>(w[word], k & 1, b);
  }
  return u4(w);
}
template <int DT>
__device__ __forceinline__ void seg_store(char* base, size_t lo, size_t len, size_t j, uint4 v) {
  constexpr int PER16 = 16 / Fmt<DT>::kBytes;
  const size_t first = j * PER16;
  if ((lo * Fmt<DT>::kBytes) % 16 == 0 && first + PER16 <= len) {
    st_v4(base + (lo + first) * Fmt<DT>::kBytes, v);
    return;
  }
  const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < PER16; ++k)
    if (first + k < len)
      Fmt<DT>::store(base, lo + first + k, word_elem<DT>(w[(k * Fmt<DT>::kBytes) / 4], Fmt<DT>::kBytes == 4 ? 0 : (k & 1)));
}

// ReduceScatter over LL128 lines (technique 4's first half): every rank
// adds its part of segment s into owner s's lines with vector reductions
// in the element type, then, after a fence, counts itself on each line;
// owner r waits for count N, writes its segment and zeroes the lines.
// Atomic: the order of the additions is not fixed.
template <int DT>
__device__ __forceinline__ void body_rs_ll128(const Params& p, const u64 E) {
  constexpr int EB = Fmt<DT>::kBytes;
  constexpr int P = 128 / EB - 1;
  const int N = p.nranks;
  const int r = rank_of_block(p);
  const int c = cta_of_block(p);
  const size_t count = p.count;
  const size_t seg = (count + N - 1) / N;
  const size_t L = (seg + P - 1) / P;
  const size_t Lc = (L + p.G - 1) / p.G;
  const size_t l0 = min(L, (size_t)c * Lc);
  const size_t nl = min(L, l0 + Lc) - l0;
  const unsigned per_seg = (unsigned)(nl * kLL128Lanes);  // fewer than 2^32 items, as in body_ll128
  const unsigned items = (unsigned)N * per_seg;
  const unsigned T = blockDim.x;
  const int slot = (int)(E & 1);
  const size_t line_slot = p.l128_lines * (size_t)kLL128Line;
  const unsigned one_bits = Fmt<DT>::from_f(1.0f);
  const unsigned n_bits = Fmt<DT>::from_f((float)N);
  const unsigned flag_mask = (EB == 4) ? 0xFFFFFFFFu : 0xFFFFu;
  const bool skip = p.inject_rank == r && p.inject_mode == LLAR_INJECT_SKIP_;
  const char* src = p.in[r];
  if (!skip)
    for (unsigned i = threadIdx.x; i < items; i += T) {
      const int s = (int)(i / per_seg);
      const unsigned rem = i - (unsigned)s * per_seg;
      const size_t l = l0 + rem / kLL128Lanes;
      const int j = (int)(rem % kLL128Lanes);
      unsigned w[4];
      if (ll128_gather<DT>(src, count, seg, s, l, j, w))
        red_add_v4<DT>(p.l128 + (size_t)s * p.l128_stride + slot * line_slot + l * kLL128Line + j * 16, w);
    }
  __syncwarp();
  fence_gpu();  // every data reduction of this warp before its counts
  if (!skip)
    for (unsigned i = threadIdx.x; i < items; i += T) {
      if ((i % kLL128Lanes) != 0) continue;
      const int s = (int)(i / per_seg);
      const size_t l = l0 + (i - (unsigned)s * per_seg) / kLL128Lanes;
      red_add_flag<DT>(p.l128 + (size_t)s * p.l128_stride + slot * line_slot + l * kLL128Line, one_bits);
    }
  // owner r: my lines [l0, l0 + nl), 8 lanes each; out[r] holds segment r
  const size_t lo = min(count, (size_t)r * seg);
  char* const my_lines = p.l128 + (size_t)r * p.l128_stride + slot * line_slot;
  bool failed = false;
  const unsigned mine = per_seg;
  for (unsigned base = 0; base < mine; base += T) {  // warp-uniform trip count
    const unsigned i = base + threadIdx.x;
    const bool active = i < mine;
    const size_t l = l0 + i / kLL128Lanes;
    const int j = (int)(i % kLL128Lanes);
    char* line = my_lines + l * kLL128Line;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (active && !failed) {
      Waiter wt;
      while ((ld_acquire_u32(line) & flag_mask) != n_bits)
        if (wt.expired(p)) {
          report_timeout(p, r, c, E);
          failed = true;
          break;
        }
      if (!failed) v = ld_relaxed_v4(line + j * 16);
    }
    __syncwarp();  // all lanes of the line have read before any zeroing
    if (active && !failed) {
      st_relaxed_v4(line + j * 16, make_uint4(0, 0, 0, 0));
      const unsigned w[4] = {v.x, v.y, v.z, v.w};
      ll128_scatter<DT>(p.out[r], lo, count, seg, r, l, j, w);
    }
  }
}

// ReduceScatter and AllGather over sentinel slots, one chunk per launch
// (the host checks that a segment fits a chunk; the launch boundary orders
// slot reuse): vector j of a segment travels raw into the receiver's slot
// [0][sender][j], which holds the all-ones pattern until it lands; the
// receiver polls until no element is the pattern, then writes the pattern
// back.
template <int DT, int N>
__device__ __forceinline__ bool sen_take(const Params& p, char* cell, int r, int c, u64 E, uint4& x) {
  Waiter wt;
  while (true) {
    x = ld_relaxed_v4(cell);
    if (!has_sentinel<DT>(x)) break;
    if (wt.expired(p)) {
      report_timeout(p, r, c, E);
      return false;
    }
  }
  st_relaxed_v4(cell, make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu));
  return true;
}

template <int DT, int N>
__device__ __forceinline__ void body_rs_sentinel(const Params& p, const u64 E) {
  const int r = rank_of_block(p);
  const int c = cta_of_block(p);
  const size_t count = p.count;
  const size_t S = (count + N - 1) / N;
  const size_t VS = (S * Fmt<DT>::kBytes + 15) / 16;  // vectors of the longest segment
  const size_t per = (VS + p.G - 1) / p.G;
  const size_t j0 = min(VS, (size_t)c * per), j1 = min(VS, j0 + per);
  const size_t src_stride = (size_t)p.sen_chunk_vecs * 16;
  const bool skip = p.inject_rank == r && p.inject_mode == LLAR_INJECT_SKIP_;
  for (size_t j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
    if (!skip)
#pragma unroll
      for (int s = 0; s < N; ++s) {
        if (s == r) continue;
        size_t lo, hi;
        segment_of(count, N, s, lo, hi);
        if (j * 16 >= (hi - lo) * Fmt<DT>::kBytes) continue;
        st_relaxed_v4(p.sen + (size_t)s * p.sen_stride + (size_t)r * src_stride + j * 16,
                      seg_vec<DT>(p.in[r], lo, hi - lo, j));
      }
  }
  size_t lo, hi;
  segment_of(count, N, r, lo, hi);
  const size_t len = hi - lo;
  for (size_t j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
    if (j * 16 >= len * Fmt<DT>::kBytes) break;
    float acc[16 / Fmt<DT>::kBytes];
#pragma unroll
    for (int q = 0; q < N; ++q) {
      uint4 x;
      if (q == r) x = seg_vec<DT>(p.in[r], lo, len, j);
      else if (!sen_take<DT, N>(p, p.sen + (size_t)r * p.sen_stride + (size_t)q * src_stride + j * 16, r, c, E, x))
        return;
      const unsigned w4[4] = {x.x, x.y, x.z, x.w};
      acc_words<DT, 4>(acc, w4, q == 0);
    }
    unsigned y[4];
    round_words<DT, 4>(acc, y);
    seg_store<DT>(p.out[r], 0, len, j, u4(y));
  }
}

template <int DT, int N>
__device__ __forceinline__ void body_ag_sentinel(const Params& p, const u64 E) {
  const int r = rank_of_block(p);
  const int c = cta_of_block(p);
  const size_t count = p.count;
  const size_t S = (count + N - 1) / N;
  const size_t VS = (S * Fmt<DT>::kBytes + 15) / 16;
  const size_t per = (VS + p.G - 1) / p.G;
  const size_t j0 = min(VS, (size_t)c * per), j1 = min(VS, j0 + per);
  const size_t src_stride = (size_t)p.sen_chunk_vecs * 16;
  const bool skip = p.inject_rank == r && p.inject_mode == LLAR_INJECT_SKIP_;
  size_t lo, hi;
  segment_of(count, N, r, lo, hi);
  const size_t len = hi - lo;
  for (size_t j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
    if (j * 16 >= len * Fmt<DT>::kBytes) break;
    const uint4 x = seg_vec<DT>(p.in[r], 0, len, j);
    if (!skip)
#pragma unroll
      for (int q = 0; q < N; ++q)
        if (q != r) st_relaxed_v4(p.sen + (size_t)q * p.sen_stride + (size_t)r * src_stride + j * 16, x);
    seg_store<DT>(p.out[r], lo, len, j, x);
  }
  for (size_t j = j0 + threadIdx.x; j < j1; j += blockDim.x)
#pragma unroll
    for (int q = 0; q < N; ++q) {
      if (q == r) continue;
      size_t qlo, qhi;
      segment_of(count, N, q, qlo, qhi);
      if (j * 16 >= (qhi - qlo) * Fmt<DT>::kBytes) continue;
      uint4 x;
      if (!sen_take<DT, N>(p, p.sen + (size_t)r * p.sen_stride + (size_t)q * src_stride + j * 16, r, c, E, x))
        return;
      seg_store<DT>(p.out[r], qlo, qhi - qlo, j, x);
    }
}

template <int DT>
__global__ void __launch_bounds__(kMaxThreads) k_rs_ll128(const Params p) {
  const u64 epoch0 = launch_epoch(p);
  body_rs_ll128<DT>(p, epoch0);
  finish_launch(p, epoch0);
}
template <int DT, int N>
__global__ void __launch_bounds__(kMaxThreads) k_rs_sentinel(const Params p) {
  const u64 epoch0 = launch_epoch(p);
  body_rs_sentinel<DT, N>(p, epoch0);
  finish_launch(p, epoch0);
}
template <int DT, int N>
__global__ void __launch_bounds__(kMaxThreads) k_ag_sentinel(const Params p) {
  const u64 epoch0 = launch_epoch(p);
  body_ag_sentinel<DT, N>(p, epoch0);
  finish_launch(p, epoch0);
}

template <int DT, int N>
__global__ void __launch_bounds__(kMaxThreads) k_rs_ll(const Params p) {
  const u64 epoch0 = launch_epoch(p);
  body_rs_ll<DT, N>(p, epoch0);
  finish_launch(p, epoch0);
}
template <int DT, int N>
__global__ void __launch_bounds__(kMaxThreads) k_ag_ll(const Params p) {
  const u64 epoch0 = launch_epoch(p);
  body_ag_ll<DT, N>(p, epoch0);
  finish_launch(p, epoch0);
}
template <int DT>
__global__ void __launch_bounds__(kMaxThreads) k_rs_fixed(const Params p) {
  const u64 epoch0 = launch_epoch(p);
  body_rs_fixed<DT>(p, epoch0);
  finish_launch(p, epoch0);
}
template <int DT>
__global__ void __launch_bounds__(kMaxThreads) k_ag_fixed(const Params p) {
  const u64 epoch0 = launch_epoch(p);
  body_ag_fixed<DT>(p, epoch0);
  finish_launch(p, epoch0);
}

// ========================================================= point to point
// A pipeline-parallel stage hand-off between virtual ranks: rank r sends
// its buffer to rank peer_dst[r] and receives from peer_src[r] ("Every
// Microsecond Matters", summary page: the same LL and sentinel signalling,
// double-buffered). CTA c of every rank covers the same share of the
// message. A one-directional flow carries no returning data that could
// act as technique 3's implicit credit, so the receiving CTA publishes an
// explicit acknowledgement after it has consumed (and, for the sentinel,
// reset) its share of a transfer; the sending CTA waits for it before it
// reuses that slot two transfers later. Acknowledgement values are
// (epoch << 24) + chunk, monotone across launches, in their own flag kind.
__device__ __forceinline__ u64 ack_value(u64 E, unsigned chunk) { return (E << 24) + chunk; }

// Thread 0 waits until rank q's CTA c acknowledged `want`; CTA-uniform result.
__device__ __forceinline__ bool wait_ack(const Params& p, int q, int c, u64 want, int me, u64 E) {
  int fail = 0;
  if (threadIdx.x == 0) {
    Waiter wt;
    while (ld_acquire_u64(flag_ptr(p, q, c, kFlagAck)) < want)
      if (wt.expired(p)) {
        report_timeout(p, me, c, E);
        fail = 1;
        break;
      }
  }
  return !__syncthreads_or(fail);
}
// After a CTA-wide barrier: thread 0 releases the CTA's reads and resets.
__device__ __forceinline__ void post_ack(const Params& p, int me, int c, u64 value) {
  if (threadIdx.x == 0) {
    fence_gpu();
    st_relaxed_u64(flag_ptr(p, me, c, kFlagAck), value);
  }
}

// LL: rank r publishes its words in its own staging (slot E & 1) as in the
// one-shot; the receiver polls the sender's lines. Slot E & 1 held epoch
// E - 2, so the sender first waits for the receiver's acknowledgement of it.
// Point to point by direct reads (the fixed-order protocols' way): the
// receiver's CTAs copy the sender's buffer, which stream order has made
// ready, 16 bytes a thread; transfers of one launch are independent, so
// nothing is signalled. Block b copies its share of rank b % N's transfer.
template <int DT>
__global__ void __launch_bounds__(kMaxThreads) k_p2p_copy(const Params p) {
  const u64 E0 = launch_epoch(p);
  const int r = rank_of_block(p), c = cta_of_block(p);
  const int q = p.peer_dst[r];
  if (q >= 0) {
    constexpr int EB = Fmt<DT>::kBytes;
    const size_t nbytes = p.count * EB;
    const size_t NV = nbytes / 16;                    // whole vectors
    const size_t total = (size_t)p.G * blockDim.x;    // this rank's threads
    const size_t t0 = (size_t)c * blockDim.x + threadIdx.x;
    for (int e = 0; e < p.iters; ++e) {
      const char* src = p.in[r] + (size_t)e * p.in_stride * EB;
      char* dst = p.out[q] + (size_t)e * p.out_stride * EB;
      for (size_t v = t0; v < NV; v += total) st_v4(dst + v * 16, ld_stream_v4(src + v * 16));
      for (size_t i = NV * 16 / EB + t0; i < p.count; i += total) Fmt<DT>::store(dst, i, Fmt<DT>::load(src, i));
    }
  }
  finish_launch(p, E0);
}

template <int DT>
__global__ void __launch_bounds__(kMaxThreads) k_p2p_ll(const Params p) {
  const u64 E0 = launch_epoch(p);
  const int r = blockIdx.x % p.nranks, c = blockIdx.x / p.nranks;
  // an injected silent rank neither sends nor acknowledges
  const bool silent = p.inject_rank == r && p.inject_mode == LLAR_INJECT_SKIP_;
  const int dst = silent ? -1 : p.peer_dst[r], src = p.peer_src[r];
  const size_t W = (p.count * Fmt<DT>::kBytes + 7) / 8;
  const size_t per = (W + p.G - 1) / p.G;
  const size_t w0 = min(W, (size_t)c * per), w1 = min(W, w0 + per);
  const size_t slot_stride = p.ll_slot_words * (size_t)kLLLine;
  char* const mine = p.ll + (size_t)r * p.ll_stride;
  const char* const from = p.ll + (size_t)(src < 0 ? 0 : src) * p.ll_stride;
  bool ok = true;
  u64 unacked = 0;  // epoch received but not yet acknowledged (0: none)
  for (int e = 0; e < p.iters && ok; ++e) {
    const u64 E = E0 + (u64)e;
    const size_t slot = (size_t)(E & 1) * slot_stride;
    if (dst >= 0) {
      if (e >= 2) ok = wait_ack(p, dst, c, ack_value(E - 2, 0), r, E);
      if (ok) {
        const char* in = rank_input<DT>(p, r, e);
        for (size_t w = w0 + threadIdx.x; w < w1; w += blockDim.x)
          st_relaxed_b128(mine + slot + w * kLLLine, load_word8<DT>(in, w, p.count), E);
      }
    }
    // the previous transfer's acknowledgement goes out after this one's
    // send (its sender needs it only before sending the next transfer):
    // thread 0's fence is then off the path from receiving to sending
    if (unacked && ok) {
      post_ack(p, r, c, ack_value(unacked, 0));
      unacked = 0;
    }
    if (src >= 0 && ok) {
      char* out = rank_output<DT>(p, r, e);
      bool mine_ok = true;
      for (size_t w = w0 + threadIdx.x; w < w1 && mine_ok; w += blockDim.x) {
        Waiter wt;
        u64 lo, hi;
        while (true) {
          ld_relaxed_b128(from + slot + w * kLLLine, lo, hi);
          if (hi == E) break;
          if (wt.expired(p)) {
            report_timeout(p, r, c, E);
            mine_ok = false;
            break;
          }
        }
        if (mine_ok) store_word8<DT>(out, w, p.count, lo);
      }
      ok = !__syncthreads_or(!mine_ok);
      if (ok && !silent) unacked = E;
    }
  }
  finish_launch(p, E0);
}

// Sentinel: the sender pushes raw 16-byte vectors into the receiver's slot
// [seq & 1][sender][vector] (all-ones when idle); the receiver polls until
// no element is the all-ones pattern, stores the vector and resets the
// slot. Messages longer than a chunk go in chunks, seq numbering them
// within the launch; slot seq & 1 was last used by seq - 2.
template <int DT>
__global__ void __launch_bounds__(kMaxThreads) k_p2p_sentinel(const Params p) {
  const u64 E0 = launch_epoch(p);
  const int N = p.nranks;
  const int r = blockIdx.x % N, c = blockIdx.x / N;
  const bool silent = p.inject_rank == r && p.inject_mode == LLAR_INJECT_SKIP_;
  const int dst = silent ? -1 : p.peer_dst[r], src = p.peer_src[r];
  const size_t NV = (p.count * Fmt<DT>::kBytes + 15) / 16;
  const unsigned CV = (unsigned)p.sen_chunk_vecs;
  const unsigned nchunks = (unsigned)((NV + CV - 1) / CV);
  const unsigned CU = (unsigned)min((size_t)CV, NV);  // vectors of a chunk the message uses
  const unsigned per = (CU + p.G - 1) / p.G;
  const unsigned j0 = min(CU, (unsigned)c * per), j1 = min(CU, j0 + per);
  const size_t src_stride = (size_t)CV * 16;
  const size_t slot_stride = (size_t)N * src_stride;
  const uint4 ones = make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
  char* const to = p.sen + (size_t)(dst < 0 ? 0 : dst) * p.sen_stride + (size_t)r * src_stride;
  char* const box = p.sen + (size_t)r * p.sen_stride + (size_t)(src < 0 ? 0 : src) * src_stride;
  bool ok = true;
  for (int e = 0; e < p.iters && ok; ++e) {
    const u64 E = E0 + (u64)e;
    const char* in = rank_input<DT>(p, r, e);
    char* out = rank_output<DT>(p, r, e);
    for (unsigned k = 0; k < nchunks && ok; ++k) {
      const size_t seq = (size_t)e * nchunks + k;
      const size_t slot = (seq & 1) * slot_stride;
      if (dst >= 0) {
        if (seq >= 2) {
          const size_t prev = seq - 2;
          ok = wait_ack(p, dst, c, ack_value(E0 + prev / nchunks, (unsigned)(prev % nchunks)), r, E);
        }
        if (ok)
          for (unsigned j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
            const size_t v = (size_t)k * CV + j;
            if (v < NV) st_relaxed_v4(to + slot + (size_t)j * 16, load_vec16<DT>(in, v, p.count, false));
          }
      }
      if (src >= 0 && ok) {
        bool mine_ok = true;
        for (unsigned j = j0 + threadIdx.x; j < j1 && mine_ok; j += blockDim.x) {
          const size_t v = (size_t)k * CV + j;
          if (v >= NV) continue;
          char* cell = box + slot + (size_t)j * 16;
          Waiter wt;
          uint4 x;
          while (true) {
            x = ld_relaxed_v4(cell);
            if (!has_sentinel<DT>(x)) break;
            if (wt.expired(p)) {
              report_timeout(p, r, c, E);
              mine_ok = false;
              break;
            }
          }
          if (mine_ok) {
            st_relaxed_v4(cell, ones);
            store_vec16<DT>(out, v, p.count, x);
          }
        }
        ok = !__syncthreads_or(!mine_ok);
        if (ok && !silent) post_ack(p, r, c, ack_value(E, k));
      }
    }
  }
  finish_launch(p, E0);
}

// ============================================================ launchers
// Launch N x G blocks: cooperative when CTAs wait on each other (the
// runtime refuses a grid that cannot be fully resident and starts it only
// when it is), unless p.no_coop; in clusters of N blocks (one CTA of every
// rank for the same range, on one GPC) when p.clustered is set.
static cudaLaunchConfig_t launch_config(const Params& p, int threads, cudaStream_t s, bool coop,
                                        cudaLaunchAttribute* at) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nranks * p.G);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = p.spread_smem;
  cfg.stream = s;
  int na = 0;
  if (coop && !p.no_coop) {
    at[na].id = cudaLaunchAttributeCooperative;
    at[na].val.cooperative = 1;
    ++na;
  }
  if (p.pdl) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.clustered) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = p.nranks;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  return cfg;
}
static cudaError_t launch_kernel(const void* k, const Params& p, int threads, cudaStream_t s, bool coop) {
  if (p.spread_smem > 0) {
    const cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, p.spread_smem);
    if (err != cudaSuccess) return err;
  }
  cudaLaunchAttribute at[3];
  cudaLaunchConfig_t cfg = launch_config(p, threads, s, coop, at);
  void* args[] = {const_cast<Params*>(&p)};
  return cudaLaunchKernelExC(&cfg, k, args);
}

#define LLAR_DISPATCH(KERNEL, COOP)                                                        \
  switch (dtype) {                                                                         \
    case 0: return launch_kernel((const void*)KERNEL<0>, p, threads, s, (COOP));           \
    case 1: return launch_kernel((const void*)KERNEL<1>, p, threads, s, (COOP));           \
    case 2: return launch_kernel((const void*)KERNEL<2>, p, threads, s, (COOP));           \
    default: return cudaErrorInvalidValue;                                                 \
  }

// INJ: fault injection armed; strided: inputs or outputs move per iteration
template <int DT, int N, bool INJ>
static const void* one_shot_kernel(int proto, bool chain, bool strided) {
  if (proto == 1)
    return chain ? (const void*)k_ll<DT, N, 2>
                 : (INJ || strided) ? (const void*)k_ll<DT, N, 1> : (const void*)k_ll<DT, N, 0>;
  return chain ? (const void*)k_sentinel<DT, N, true, INJ> : (const void*)k_sentinel<DT, N, false, INJ>;
}
template <int DT, bool INJ>
static const void* one_shot_kernel_n(int proto, int n, bool chain, bool strided) {
  switch (n) {
    case 2: return one_shot_kernel<DT, 2, INJ>(proto, chain, strided);
    case 3: return one_shot_kernel<DT, 3, INJ>(proto, chain, strided);
    case 4: return one_shot_kernel<DT, 4, INJ>(proto, chain, strided);
    case 5: return one_shot_kernel<DT, 5, INJ>(proto, chain, strided);
    case 6: return one_shot_kernel<DT, 6, INJ>(proto, chain, strided);
    case 7: return one_shot_kernel<DT, 7, INJ>(proto, chain, strided);
    case 8: return one_shot_kernel<DT, 8, INJ>(proto, chain, strided);
    default: return nullptr;
  }
}
template <bool INJ>
static const void* one_shot_kernel_inj(int proto, int dtype, int n, bool chain, bool strided) {
  return dtype == 0   ? one_shot_kernel_n<0, INJ>(proto, n, chain, strided)
         : dtype == 1 ? one_shot_kernel_n<1, INJ>(proto, n, chain, strided)
                      : one_shot_kernel_n<2, INJ>(proto, n, chain, strided);
}
static const void* one_shot_kernel_for(int proto, int dtype, int n, bool chain, bool inject = false,
                                       bool strided = false) {
  return inject ? one_shot_kernel_inj<true>(proto, dtype, n, chain, strided)
                : one_shot_kernel_inj<false>(proto, dtype, n, chain, strided);
}
static bool injection_armed(const Params& p) { return p.inject_rank >= 0 && p.inject_mode != 0; }
static cudaError_t launch_one_shot(int proto, int dtype, const Params& p, int threads, cudaStream_t s) {
  const void* k = one_shot_kernel_for(proto, dtype, p.nranks, p.chain != 0, injection_armed(p),
                                      p.in_stride != 0 || p.out_stride != 0);
  if (!k) return cudaErrorInvalidValue;
  return launch_kernel(k, p, threads, s, true);
}
template <int DT>
static const void* segment_kernel(int which, int n) {
  // which: 0 = ReduceScatter LL, 1 = AllGather LL, 2 = ReduceScatter fixed,
  // 3 = AllGather fixed, 4 = ReduceScatter LL128, 5 = ReduceScatter
  // sentinel, 6 = AllGather sentinel
  if (which == 2) return (const void*)k_rs_fixed<DT>;
  if (which == 3) return (const void*)k_ag_fixed<DT>;
  if (which == 4) return (const void*)k_rs_ll128<DT>;
  switch (n) {
#define LLAR_SEG_CASE(NN)                                                                       \
    case NN:                                                                                    \
      return which == 0   ? (const void*)k_rs_ll<DT, NN>                                        \
             : which == 1 ? (const void*)k_ag_ll<DT, NN>                                        \
             : which == 5 ? (const void*)k_rs_sentinel<DT, NN> : (const void*)k_ag_sentinel<DT, NN>;
    LLAR_SEG_CASE(2) LLAR_SEG_CASE(3) LLAR_SEG_CASE(4) LLAR_SEG_CASE(5)
    LLAR_SEG_CASE(6) LLAR_SEG_CASE(7) LLAR_SEG_CASE(8)
#undef LLAR_SEG_CASE
    default: return nullptr;
  }
}
const void* segment_kernel_for(int which, int dtype, int n) {
  return dtype == 0 ? segment_kernel<0>(which, n) : dtype == 1 ? segment_kernel<1>(which, n) : segment_kernel<2>(which, n);
}
cudaError_t launch_segment(int which, int dtype, const Params& p, int threads, cudaStream_t s) {
  const void* k = segment_kernel_for(which, dtype, p.nranks);
  if (!k) return cudaErrorInvalidValue;
  return launch_kernel(k, p, threads, s, which != 2 && which != 3);  // the direct-read ones never wait
}
int max_resident_segment_ctas(int which, int dtype, int nranks, int threads) {
  const void* k = segment_kernel_for(which, dtype, nranks);
  int per_sm = 0, dev = 0, sms = 0;
  if (!k || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, 0) != cudaSuccess) return 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return per_sm * sms;
}

cudaError_t launch_ll(int dtype, const Params& p, int threads, cudaStream_t s) {
  return launch_one_shot(1, dtype, p, threads, s);
}
cudaError_t launch_sentinel(int dtype, const Params& p, int threads, cudaStream_t s) {
  return launch_one_shot(2, dtype, p, threads, s);
}
cudaError_t launch_ll128(int dtype, const Params& p, int threads, cudaStream_t s) {
  LLAR_DISPATCH(k_ll128, true)
}
cudaError_t launch_ll128d(int dtype, const Params& p, int threads, cudaStream_t s) {
  LLAR_DISPATCH(k_ll128d, true)
}
cudaError_t launch_fixed_oneshot(int dtype, const Params& p, int threads, cudaStream_t s) {
  LLAR_DISPATCH(k_fixed_oneshot, p.chain != 0)
}
cudaError_t launch_fixed_twoshot(int dtype, const Params& p, int threads, cudaStream_t s) {
  LLAR_DISPATCH(k_fixed_twoshot, p.chain != 0)
}

size_t bulk_smem_bytes(int nranks) { return (size_t)kBulkStages * nranks * kBulkTileBytes + 8 * kBulkStages; }
size_t bulk_tile_vectors() { return kBulkTileBytes / 16; }

static const void* p2p_kernel(int proto, int dtype) {
  if (proto == 4)
    return dtype == 0 ? (const void*)k_p2p_copy<0> : dtype == 1 ? (const void*)k_p2p_copy<1> : (const void*)k_p2p_copy<2>;
  if (proto == 1)
    return dtype == 0 ? (const void*)k_p2p_ll<0> : dtype == 1 ? (const void*)k_p2p_ll<1> : (const void*)k_p2p_ll<2>;
  return dtype == 0 ? (const void*)k_p2p_sentinel<0>
                    : dtype == 1 ? (const void*)k_p2p_sentinel<1> : (const void*)k_p2p_sentinel<2>;
}
cudaError_t launch_p2p(int proto, int dtype, const Params& p, int threads, cudaStream_t s) {
  // the direct copy waits on nothing: no co-residency needed
  return launch_kernel(p2p_kernel(proto, dtype), p, threads, s, proto != 4);
}
int max_resident_p2p_ctas(int proto, int dtype, int threads) {
  int per = 0, sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, p2p_kernel(proto, dtype), threads, 0) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return per * sms;
}

cudaError_t launch_fixed_twoshot_bulk(int dtype, const Params& p, int threads, cudaStream_t s) {
  const void* k = dtype == 0 ? (const void*)k_fixed_twoshot_bulk<0>
                  : dtype == 1 ? (const void*)k_fixed_twoshot_bulk<1> : (const void*)k_fixed_twoshot_bulk<2>;
  const int smem = (int)bulk_smem_bytes(p.nranks);
  cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute at[3];  // cooperative, programmatic dependency, cluster
  cudaLaunchConfig_t cfg = launch_config(p, threads, s, false, at);
  cfg.dynamicSmemBytes = smem;
  void* args[] = {const_cast<Params*>(&p)};
  return cudaLaunchKernelExC(&cfg, k, args);
}

template <int DT>
static const void* kernel_for(int proto) {
  switch (proto) {
    case 3: return (const void*)k_ll128<DT>;
    case 6: return (const void*)k_ll128d<DT>;
    case 4: return (const void*)k_fixed_oneshot<DT>;
    case 5: return (const void*)k_fixed_twoshot<DT>;
    default: return nullptr;
  }
}

int max_resident_ctas(int proto, int dtype, int nranks, int threads, bool clustered, int spread_smem) {
  const void* k = (proto == 1 || proto == 2) ? one_shot_kernel_for(proto, dtype, nranks, false)
                  : dtype == 0 ? kernel_for<0>(proto) : dtype == 1 ? kernel_for<1>(proto) : kernel_for<2>(proto);
  if (!k) return 0;
  if (clustered) {
    // how many clusters of nranks blocks fit at once, times the cluster size
    Params p;
    memset(&p, 0, sizeof(p));
    p.nranks = nranks;
    p.G = 1;
    p.clustered = 1;
    p.spread_smem = spread_smem;
    if (spread_smem > 0 && cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, spread_smem) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cudaLaunchAttribute at[3];  // cooperative, programmatic dependency, cluster
    cudaLaunchConfig_t cfg = launch_config(p, threads, 0, false, at);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, k, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return clusters * nranks;
  }
  int per_sm = 0, dev = 0, sms = 0;
  if (spread_smem > 0 && cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, spread_smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, spread_smem) != cudaSuccess) return 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return per_sm * sms;
}

// ======================================================= speed-of-light
// Pointer chase: buf holds, at word 32*i (one 128-byte line per entry), the
// index of the next line of one random cycle. One thread per block walks
// `hops` dependent GPU-scope loads (served by L2, never by L1) after an
// equal warm-up walk. The dynamic shared memory request keeps blocks on
// distinct SMs.
__global__ void k_sol_chase(const unsigned* buf, unsigned nlines, int hops, unsigned long long* ns,
                            int* smid, unsigned* sink) {
  extern __shared__ char pad[];
  if (threadIdx.x != 0) return;
  unsigned cur = (unsigned)(((unsigned long long)blockIdx.x * nlines) / gridDim.x);
  for (int i = 0; i < hops; ++i) cur = ld_relaxed_u32(buf + (size_t)cur * 32);
  const u64 t0 = globaltimer_ns();
  for (int i = 0; i < hops; ++i) cur = ld_relaxed_u32(buf + (size_t)cur * 32);
  const u64 t1 = globaltimer_ns();
  unsigned id;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(id));
  ns[blockIdx.x] = t1 - t0;
  smid[blockIdx.x] = (int)id;
  sink[blockIdx.x] = cur;
  (void)pad;
}

// Ping-pong: blocks 2k (A) and 2k+1 (B) share two flags on separate lines.
// A stores i into B's flag and waits to see i in its own; B waits for i and
// answers. One round trip = two store-to-observe latencies. Waits are
// bounded by the timeout and by the abort word.
__global__ void k_sol_pingpong(unsigned* flags, int rounds, unsigned long long* ns, int* smid,
                               unsigned* abort_flag, unsigned long long timeout_ns) {
  extern __shared__ char pad[];
  if (threadIdx.x != 0) return;
  const int pair = blockIdx.x / 2;
  const bool a_side = (blockIdx.x & 1) == 0;
  unsigned* to_a = flags + (size_t)pair * 64;
  unsigned* to_b = to_a + 32;
  unsigned id;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(id));
  smid[blockIdx.x] = (int)id;
  const u64 start = globaltimer_ns();
  const u64 deadline = start + timeout_ns;
  bool ok = true;
  for (int i = 1; i <= rounds && ok; ++i) {
    if (a_side) asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" :: "l"(to_b), "r"((unsigned)i) : "memory");
    const unsigned* watch = a_side ? to_a : to_b;
    unsigned spins = 0;
    while (ld_relaxed_u32(watch) != (unsigned)i) {
      if ((++spins & 1023u) == 0 && (globaltimer_ns() > deadline || ld_relaxed_u32(abort_flag) != 0)) {
        atomicExch(abort_flag, 7u);
        ok = false;
        break;
      }
    }
    if (!a_side && ok)
      asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" :: "l"(to_a), "r"((unsigned)i) : "memory");
  }
  const u64 end = globaltimer_ns();
  if (a_side) ns[pair] = ok ? end - start : 0ull;
  (void)pad;
}

static int sol_pad_bytes() {
  int dev = 0, smem = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  return smem / 2 + 1024;  // more than half an SM's shared memory: one block per SM
}

cudaError_t run_sol(SolResult* res, unsigned long long timeout_ns) {
  cudaError_t err;
  int dev = 0, sms = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
  const int pad = sol_pad_bytes();

  // one random cycle over the lines of a 16 MiB buffer (Sattolo's shuffle)
  const unsigned nlines = (16u << 20) / 128u;
  std::vector<unsigned> next(nlines), host((size_t)nlines * 32u, 0u);
  for (unsigned i = 0; i < nlines; ++i) next[i] = i;
  unsigned long long rng = 0x9E3779B97F4A7C15ull;
  for (unsigned i = nlines - 1; i > 0; --i) {
    rng ^= rng << 13; rng ^= rng >> 7; rng ^= rng << 17;
    const unsigned j = (unsigned)(rng % i);
    const unsigned t = next[i]; next[i] = next[j]; next[j] = t;
  }
  for (unsigned i = 0; i < nlines; ++i) host[(size_t)i * 32u] = next[i];

  const int blocks = sms < kSolMaxBlocks ? sms : kSolMaxBlocks;
  const int pairs = blocks / 2;
  const int hops = 20000, rounds = 20000;
  unsigned *buf = nullptr, *sink = nullptr, *flags = nullptr, *abort_flag = nullptr;
  unsigned long long* ns = nullptr;
  int* smid = nullptr;
  std::vector<unsigned long long> h_ns(blocks);
  std::vector<int> h_smid(blocks);
#define LLAR_TRY(x) do { if ((err = (x)) != cudaSuccess) goto done; } while (0)
  LLAR_TRY(cudaMalloc(&buf, host.size() * sizeof(unsigned)));
  LLAR_TRY(cudaMalloc(&sink, blocks * sizeof(unsigned)));
  LLAR_TRY(cudaMalloc(&ns, blocks * sizeof(unsigned long long)));
  LLAR_TRY(cudaMalloc(&smid, blocks * sizeof(int)));
  LLAR_TRY(cudaMalloc(&flags, (size_t)pairs * 64 * sizeof(unsigned)));
  LLAR_TRY(cudaMalloc(&abort_flag, sizeof(unsigned)));
  LLAR_TRY(cudaMemset(abort_flag, 0, sizeof(unsigned)));
  LLAR_TRY(cudaMemcpy(buf, host.data(), host.size() * sizeof(unsigned), cudaMemcpyHostToDevice));
  LLAR_TRY(cudaFuncSetAttribute(k_sol_chase, cudaFuncAttributeMaxDynamicSharedMemorySize, pad));
  LLAR_TRY(cudaFuncSetAttribute(k_sol_pingpong, cudaFuncAttributeMaxDynamicSharedMemorySize, pad));
  k_sol_chase<<<blocks, 32, pad>>>(buf, nlines, hops, ns, smid, sink);
  LLAR_TRY(cudaGetLastError());
  LLAR_TRY(cudaDeviceSynchronize());
  LLAR_TRY(cudaMemcpy(h_ns.data(), ns, blocks * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
  LLAR_TRY(cudaMemcpy(h_smid.data(), smid, blocks * sizeof(int), cudaMemcpyDeviceToHost));
  res->nchase = blocks;
  for (int b = 0; b < blocks; ++b) {
    res->chase_ns[b] = (double)h_ns[b] / hops;
    res->chase_smid[b] = h_smid[b];
  }
  LLAR_TRY(cudaMemset(flags, 0, (size_t)pairs * 64 * sizeof(unsigned)));
  LLAR_TRY(cudaMemset(ns, 0, blocks * sizeof(unsigned long long)));
  {
    int rounds_arg = rounds;
    void* args[] = {&flags, &rounds_arg, &ns, &smid, &abort_flag, &timeout_ns};
    LLAR_TRY(cudaLaunchCooperativeKernel((const void*)k_sol_pingpong, dim3(2 * pairs), dim3(32), args, pad, 0));
  }
  LLAR_TRY(cudaDeviceSynchronize());
  LLAR_TRY(cudaMemcpy(h_ns.data(), ns, pairs * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
  LLAR_TRY(cudaMemcpy(h_smid.data(), smid, 2 * pairs * sizeof(int), cudaMemcpyDeviceToHost));
  res->npairs = pairs;
  for (int k = 0; k < pairs; ++k) {
    res->rt_ns[k] = (double)h_ns[k] / rounds;  // 0 if that pair's wait ran out
    res->smid_a[k] = h_smid[2 * k];
    res->smid_b[k] = h_smid[2 * k + 1];
  }
#undef LLAR_TRY
done:
  cudaFree(buf);
  cudaFree(sink);
  cudaFree(ns);
  cudaFree(smid);
  cudaFree(flags);
  cudaFree(abort_flag);
  return err;
}

// Speed of light over the CTAs a launch places. A grid of the launch's
// shape (N x G blocks, its threads, dynamic shared memory, cluster and
// cooperative attributes) records each block's SM; then block c of rank r
// ping-pongs with block c of every other rank q (the blocks that exchange
// data), in rounds of disjoint pairs (round-robin schedule over the ranks
// plus a bye when N is odd). rt_ns[(c * M + k) * P + min(r, q)] receives
// the pair's ns per round trip in round k (0 for a bye or a wait that ran
// out). Waits are bounded by the timeout and the abort word.
__global__ void k_sol_placed(int nranks, int reps, unsigned* flags, int* smid, unsigned long long* rt_ns,
                             unsigned* abort_flag, unsigned long long timeout_ns) {
  extern __shared__ char pad[];
  if (threadIdx.x != 0) return;
  const int r = blockIdx.x % nranks, c = blockIdx.x / nranks;
  unsigned id;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(id));
  smid[blockIdx.x] = (int)id;
  const int P = nranks + (nranks & 1);  // players, with a bye for odd N
  const int M = P - 1;                  // rounds
  u64 deadline = 0;
  auto wait_for = [&](const unsigned* w, unsigned v) -> bool {
    unsigned spins = 0;
    while (ld_relaxed_u32(w) != v)
      if ((++spins & 1023u) == 0 && (globaltimer_ns() > deadline || ld_relaxed_u32(abort_flag) != 0)) {
        atomicExch(abort_flag, 7u);
        return false;
      }
    return true;
  };
  for (int k = 0; k < M; ++k) {
    int q;
    if (r == M) {
      q = k;
    } else {
      q = ((2 * k - r) % M + M) % M;
      if (q == r) q = M;
    }
    if (q >= nranks) continue;  // bye
    deadline = globaltimer_ns() + timeout_ns;  // each round's waits have the full bound
    const int lo = r < q ? r : q;
    const size_t pair = ((size_t)c * M + k) * P + lo;
    unsigned* to_a = flags + pair * 64;
    unsigned* to_b = to_a + 32;
    if (r == lo) {  // A: handshake 1, then reps timed round trips
      asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" :: "l"(to_b), "r"(1u) : "memory");
      if (!wait_for(to_a, 1u)) return;
      const u64 t0 = globaltimer_ns();
      for (int i = 2; i <= reps + 1; ++i) {
        asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" :: "l"(to_b), "r"((unsigned)i) : "memory");
        if (!wait_for(to_a, (unsigned)i)) return;
      }
      rt_ns[pair] = (globaltimer_ns() - t0) / (u64)reps;
    } else {  // B: answer every value
      for (int i = 1; i <= reps + 1; ++i) {
        if (!wait_for(to_b, (unsigned)i)) return;
        asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" :: "l"(to_a), "r"((unsigned)i) : "memory");
      }
    }
  }
  (void)pad;
}

cudaError_t run_sol_placed(int nranks, int G, int threads, int clustered, int spread_smem,
                           unsigned long long timeout_ns, SolPlaced* out) {
  cudaError_t err;
  SolResult chase;
  if ((err = run_sol(&chase, timeout_ns)) != cudaSuccess) return err;
  const int P = nranks + (nranks & 1), M = P - 1, blocks = nranks * G;
  const size_t npair_slots = (size_t)G * M * P;
  const int reps = 2000;
  unsigned *flags = nullptr, *abort_flag = nullptr;
  int* smid = nullptr;
  unsigned long long* rt = nullptr;
  std::vector<int> h_smid(blocks);
  std::vector<unsigned long long> h_rt(npair_slots);
#define LLAR_TRY(x) do { if ((err = (x)) != cudaSuccess) goto done; } while (0)
  LLAR_TRY(cudaMalloc(&flags, npair_slots * 64 * sizeof(unsigned)));
  LLAR_TRY(cudaMalloc(&abort_flag, sizeof(unsigned)));
  LLAR_TRY(cudaMalloc(&smid, blocks * sizeof(int)));
  LLAR_TRY(cudaMalloc(&rt, npair_slots * sizeof(unsigned long long)));
  LLAR_TRY(cudaMemset(flags, 0, npair_slots * 64 * sizeof(unsigned)));
  LLAR_TRY(cudaMemset(abort_flag, 0, sizeof(unsigned)));
  LLAR_TRY(cudaMemset(rt, 0, npair_slots * sizeof(unsigned long long)));
  if (spread_smem > 0)
    LLAR_TRY(cudaFuncSetAttribute(k_sol_placed, cudaFuncAttributeMaxDynamicSharedMemorySize, spread_smem));
  {
    Params shape;
    memset(&shape, 0, sizeof(shape));
    shape.nranks = nranks;
    shape.G = G;
    shape.clustered = clustered;
    shape.spread_smem = spread_smem;
    cudaLaunchAttribute at[3];
    cudaLaunchConfig_t cfg = launch_config(shape, threads, 0, true, at);
    int n_arg = nranks, reps_arg = reps;
    void* args[] = {&n_arg, &reps_arg, &flags, &smid, &rt, &abort_flag, &timeout_ns};
    LLAR_TRY(cudaLaunchKernelExC(&cfg, (const void*)k_sol_placed, args));
  }
  LLAR_TRY(cudaDeviceSynchronize());
  LLAR_TRY(cudaMemcpy(h_smid.data(), smid, blocks * sizeof(int), cudaMemcpyDeviceToHost));
  LLAR_TRY(cudaMemcpy(h_rt.data(), rt, npair_slots * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
  {
    // the slowest chase among the SMs that hold rank CTAs
    double worst_chase = 0.0;
    for (int b = 0; b < blocks; ++b)
      for (int i = 0; i < chase.nchase; ++i)
        if (chase.chase_smid[i] == h_smid[b] && chase.chase_ns[i] > worst_chase) worst_chase = chase.chase_ns[i];
    std::vector<double> rts;
    for (size_t i = 0; i < npair_slots; ++i)
      if (h_rt[i] > 0) rts.push_back((double)h_rt[i]);
    out->npairs = (int)rts.size();
    out->chase_worst_ns = worst_chase;
    out->rt_worst_ns = 0.0;
    out->rt_median_ns = 0.0;
    if (!rts.empty()) {
      std::sort(rts.begin(), rts.end());
      out->rt_worst_ns = rts.back();
      out->rt_median_ns = rts[rts.size() / 2];
    }
    out->distinct_sms = 0;
    std::vector<int> sorted_sm(h_smid);
    std::sort(sorted_sm.begin(), sorted_sm.end());
    out->distinct_sms = (int)(std::unique(sorted_sm.begin(), sorted_sm.end()) - sorted_sm.begin());
  }
#undef LLAR_TRY
done:
  cudaFree(flags);
  cudaFree(abort_flag);
  cudaFree(smid);
  cudaFree(rt);
  return err;
}

}  // namespace llar

// ==================================================== allocation-free LL
// Some callers cannot allocate device memory at the point where they need
// an AllReduce: code whose device memory is owned entirely by a caching
// allocator or a fixed memory budget (an inference server plugin, a
// framework pool that forbids raw cudaMalloc), or latency-critical paths
// where cudaMalloc's implicit device synchronisation is not acceptable.
// For them, llar_allreduce_noalloc runs the LL kernel above with its
// staging in the fixed-size device array below instead of llar_init's
// allocation. The array exists once per device for the life of the process.
using namespace llar;
namespace {

constexpr size_t kNoAllocMaxBytes = 32u << 10;                   // per rank
constexpr size_t kNoAllocWords = kNoAllocMaxBytes / 8;           // LL words per rank
constexpr size_t kNoAllocRankBytes = 2 * kNoAllocWords * kLLLine;  // two slots of lines
constexpr size_t kNoAllocHeader = 512;                           // abort word + status
constexpr size_t kNoAllocBytes = kNoAllocHeader + kMaxRanks * kNoAllocRankBytes;
constexpr int kNoAllocMaxDevices = 64;

// header: [0, 4) abort word, [64, 68) CTAs finished, [128, 136) epoch,
// [256, 256 + sizeof(DevStatus)) status; then
// rank r's LL lines [slot][word] at kNoAllocHeader + r * kNoAllocRankBytes.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

struct NoAllocDevice {
  bool ready = false;
  char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int sms = 0;
  int cap[3][kMaxRanks + 1] = {};  // resident-CTA capacity per (dtype, ranks), queried once
};
NoAllocDevice g_noalloc[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

}  // namespace

extern "C" int llar_allreduce_noalloc(const void* const* in, void* const* out, size_t count,
                                      int nranks, int dtype, void* stream) {
  if (nranks < 2 || nranks > kMaxRanks || dtype < 0 || dtype > 2) return LLAR_ERR_INVALID;
  if (!in || !out) return LLAR_ERR_INVALID;
  const size_t esize = dtype == 0 ? 4 : 2;
  const size_t bytes = count * esize;
  if (bytes > kNoAllocMaxBytes) return LLAR_ERR_TOO_LARGE;
  for (int r = 0; r < nranks; ++r) {
    if (!in[r] || !out[r] || (((uintptr_t)in[r] | (uintptr_t)out[r]) & 15u)) return LLAR_ERR_INVALID;
    for (int q = 0; q < nranks; ++q) {
      const uintptr_t o0 = (uintptr_t)out[r], i0 = (uintptr_t)in[q];
      if (o0 < i0 + bytes && i0 < o0 + bytes) return LLAR_ERR_INVALID;
      const uintptr_t p0 = (uintptr_t)out[q];
      if (q != r && o0 < p0 + bytes && p0 < o0 + bytes) return LLAR_ERR_INVALID;
    }
  }
  if (count == 0) return LLAR_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
    cudaGetLastError();
    return LLAR_ERR_CUDA;
  }
  NoAllocDevice& d = g_noalloc[dev];
  if (!d.ready) {
    // first call on this device: resolve the array's device address (the
    // host-side name is only a stand-in) and the SM count
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return LLAR_ERR_CUDA;
    }
    d.scratch = static_cast<char*>(ptr);
    d.ready = true;
  }
  // a wait that ran out in an earlier call is reported once that call has
  // drained from the stream; the word is then cleared. A stream that is
  // being captured must not be queried (the query would invalidate the
  // capture), so the check waits for a later call there.
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &capture) != cudaSuccess) {
    cudaGetLastError();
    capture = cudaStreamCaptureStatusActive;  // unknown: treat as capturing, skip the check
  }
  if (capture == cudaStreamCaptureStatusNone && cudaStreamQuery(s) == cudaSuccess) {
    unsigned word = 0;
    if (cudaMemcpyAsync(&word, d.scratch, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
      cudaGetLastError();
      return LLAR_ERR_CUDA;
    }
    if (word != 0) {
      cudaMemsetAsync(d.scratch, 0, 4, s);          // abort word
      cudaMemsetAsync(d.scratch + 256, 0, 256, s);  // status
      return LLAR_ERR_TIMEOUT;
    }
  } else if (capture == cudaStreamCaptureStatusNone) {
    cudaGetLastError();  // cudaErrorNotReady: still busy, check on a later call
  }

  Params p;
  memset(&p, 0, sizeof(p));
  for (int r = 0; r < nranks; ++r) {
    p.in[r] = static_cast<const char*>(in[r]);
    p.out[r] = static_cast<char*>(out[r]);
  }
  p.count = count;
  p.nranks = nranks;
  p.iters = 1;
  p.epoch_dev = reinterpret_cast<unsigned long long*>(d.scratch + 128);
  p.done_count = reinterpret_cast<unsigned*>(d.scratch + 64);
  p.ll = d.scratch + kNoAllocHeader;
  p.ll_stride = kNoAllocRankBytes;
  p.ll_slot_words = kNoAllocWords;
  fault_settings(&p.timeout_ns, &p.inject_rank, &p.inject_mode);  // as llar_set_timeout_ns / llar_debug_inject
  if (p.inject_rank >= nranks) p.inject_rank = -1;
  p.abort_flag = reinterpret_cast<unsigned*>(d.scratch);
  p.status = reinterpret_cast<DevStatus*>(d.scratch + 256);
  const size_t words = (bytes + 7) / 8;
  const int threads = 128;
  int G = (int)((words + threads - 1) / threads);
  G = G < 1 ? 1 : G;
  const int one_per_sm = d.sms / nranks > 0 ? d.sms / nranks : 1;
  G = G > one_per_sm ? one_per_sm : G;
  p.clustered = 0;  // the LL kernel runs faster with its CTAs spread over the GPU
  int& cap = d.cap[dtype][nranks];  // an occupancy query costs microseconds: once per shape
  if (cap <= 0) cap = max_resident_ctas(1, dtype, nranks, threads, false, 0);
  if (cap <= 0) return LLAR_ERR_CUDA;
  if (nranks * G > cap) G = cap / nranks > 0 ? cap / nranks : 1;
  p.G = G;
  const cudaError_t err = launch_ll(dtype, p, threads, s);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return err == cudaErrorCooperativeLaunchTooLarge ? LLAR_ERR_OCCUPANCY : LLAR_ERR_CUDA;
  }
  return LLAR_OK;
}

// =================================================== poll statistics
extern "C" int llar_debug_poll_stats(unsigned long long* stats, int reset) {
#ifdef LLAR_POLL_STATS
  if (!stats) return LLAR_ERR_INVALID;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpyFromSymbol(stats, g_llar_poll_stats, sizeof(g_llar_poll_stats)) != cudaSuccess) {
    cudaGetLastError();
    return LLAR_ERR_CUDA;
  }
  if (reset) {
    const unsigned long long zero[4] = {0, 0, 0, 0};
    if (cudaMemcpyToSymbol(g_llar_poll_stats, zero, sizeof(zero)) != cudaSuccess) {
      cudaGetLastError();
      return LLAR_ERR_CUDA;
    }
  }
  return LLAR_OK;
#else
  (void)stats;
  (void)reset;
  return LLAR_ERR_UNSUPPORTED;
#endif
}
