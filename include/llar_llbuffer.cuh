// llar LL buffer, device half: header-only __device__ primitives that act on
// an llar_llbuffer descriptor (llar_llbuffer.h), for user kernels that
// exchange data between virtual ranks without a global memory barrier
// ("Every Microsecond Matters: Achieving Near Speed-of-Light Latency in GPU
// Collectives", summary page, techniques 1-4, packaged as a low-level buffer
// API for custom kernels).
//
// Model. A virtual rank is a set of CTAs of one launch; ranks exchange data
// through the descriptor's staging in device memory, signalling with GPU-
// scope relaxed/acquire loads, stores and reductions that meet in L2. Every
// CTA that waits on another must be resident at the same time as it:
// launch such a kernel cooperatively (cudaLaunchAttributeCooperative) or
// size the grid to the occupancy.
//
// Epochs. An exchange is named by a 64-bit epoch E that every rank agrees
// on. llb::begin() returns the first epoch of a launch (the descriptor's
// device counter + 1, so a launch replayed from a CUDA graph still gets
// fresh epochs); a launch that used `n` epochs calls llb::end(b, n, E) in
// every thread of every CTA as its last step, E being what begin() returned
// (llb::end(b, n) does the same but reads the counter once more).
//
// Waits. Every wait is bounded by b.timeout_ns. A wait that runs out
// records the rank and epoch (llar_llbuffer_get_status on the host), raises
// the abort word (every other wait then gives up at once) and returns false;
// the caller should leave the kernel.
//
// Memory-model notes (PTX memory consistency model): signalling accesses
// are .relaxed.gpu (morally strong, served by L2); fence_gpu() followed by a
// signalling store is a release; a consumer that reads other locations
// after a flag reads the flag with ld.acquire.gpu.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "llar_llbuffer.h"

// Diagnostic hook: every bounded wait below calls it once per polling
// round, with `first` (the wait's first round) and `pending` (one bit per
// line still awaited; its population count is the loads the round issues).
// It expands to nothing unless the includer defines LLB_ON_POLL_ROUND
// before including this header (the library's poll-counting build does).
#ifndef LLB_ON_POLL_ROUND
__device__ __forceinline__ void llb_poll_round_unused(bool, unsigned) {}
#define LLB_ON_POLL_ROUND(first, pending) llb_poll_round_unused((first), (pending))
#endif

namespace llb {

typedef unsigned long long u64;

// ------------------------------------------------------------------- PTX
__device__ __forceinline__ u64 globaltimer_ns() {
  u64 t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// one single 16-byte access (.b128): an LL line {8 bytes data, 8 bytes flag}
__device__ __forceinline__ void st_relaxed_b128(void* p, u64 lo, u64 hi) {
  asm volatile("{\n .reg .b128 t;\n mov.b128 t, {%1, %2};\n st.relaxed.gpu.global.b128 [%0], t;\n}"
               :: "l"(p), "l"(lo), "l"(hi) : "memory");
}
__device__ __forceinline__ void ld_relaxed_b128(const void* p, u64& lo, u64& hi) {
  asm volatile("{\n .reg .b128 t;\n ld.relaxed.gpu.global.b128 t, [%2];\n mov.b128 {%0, %1}, t;\n}"
               : "=l"(lo), "=l"(hi) : "l"(p) : "memory");
}
// 16-byte vector of four single-copy-atomic 32-bit parts
__device__ __forceinline__ void st_relaxed_v4(void* p, uint4 v) {
  asm volatile("st.relaxed.gpu.global.v4.b32 [%0], {%1, %2, %3, %4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ uint4 ld_relaxed_v4(const void* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_acquire_u32(const void* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_relaxed_u32(const void* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// --------------------------------------------------------- element types
// Elem<T>: raw bits <-> float32 and the vector reductions of one type.
// Conversions to T round to nearest even.
template <typename T> struct Elem;

template <> struct Elem<float> {
  static constexpr int kBytes = 4;
  static constexpr unsigned kMask = 0xFFFFFFFFu;
  __device__ static __forceinline__ float to_f(unsigned b) { return __uint_as_float(b); }
  __device__ static __forceinline__ unsigned from_f(float f) { return __float_as_uint(f); }
  __device__ static __forceinline__ void red_v4(void* a, uint4 w) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                 :: "l"(a), "f"(__uint_as_float(w.x)), "f"(__uint_as_float(w.y)),
                    "f"(__uint_as_float(w.z)), "f"(__uint_as_float(w.w)) : "memory");
  }
  __device__ static __forceinline__ void red_one(void* a) {
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" :: "l"(a), "f"(1.0f) : "memory");
  }
};
template <> struct Elem<__half> {
  static constexpr int kBytes = 2;
  static constexpr unsigned kMask = 0xFFFFu;
  __device__ static __forceinline__ float to_f(unsigned b) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
  }
  __device__ static __forceinline__ unsigned from_f(float f) { return __half_as_ushort(__float2half_rn(f)); }
  __device__ static __forceinline__ void red_v4(void* a, uint4 w) {
    asm volatile("red.relaxed.gpu.global.add.noftz.v4.f16x2 [%0], {%1, %2, %3, %4};"
                 :: "l"(a), "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w) : "memory");
  }
  // {1, -0} on the flag's 32-bit word: -0 leaves the next element as it is
  __device__ static __forceinline__ void red_one(void* a) {
    const unsigned pair = 0x3C00u | (0x8000u << 16);
    asm volatile("red.relaxed.gpu.global.add.noftz.f16x2 [%0], %1;" :: "l"(a), "r"(pair) : "memory");
  }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static constexpr unsigned kMask = 0xFFFFu;
  __device__ static __forceinline__ float to_f(unsigned b) { return __uint_as_float(b << 16); }
  __device__ static __forceinline__ unsigned from_f(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
  }
  __device__ static __forceinline__ void red_v4(void* a, uint4 w) {
    asm volatile("red.relaxed.gpu.global.add.noftz.v4.bf16x2 [%0], {%1, %2, %3, %4};"
                 :: "l"(a), "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w) : "memory");
  }
  __device__ static __forceinline__ void red_one(void* a) {
    const unsigned pair = 0x3F80u | (0x8000u << 16);
    asm volatile("red.relaxed.gpu.global.add.noftz.bf16x2 [%0], %1;" :: "l"(a), "r"(pair) : "memory");
  }
};

// element i of a little-endian packed group of 32-bit words
template <typename T>
__device__ __forceinline__ unsigned elem_get(const unsigned* w, int i) {
  if (Elem<T>::kBytes == 4) return w[i];
  return (w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
}
template <typename T>
__device__ __forceinline__ void elem_set(unsigned* w, int i, unsigned bits) {
  if (Elem<T>::kBytes == 4) {
    w[i] = bits;
  } else {
    const int sh = 16 * (i & 1);
    w[i >> 1] = (w[i >> 1] & ~(0xFFFFu << sh)) | (bits << sh);
  }
}

// ------------------------------------------------------------ bounded waits
// Counts polls; every 32nd poll reads %globaltimer (the deadline starts at
// the first reading, so short waits never read the clock) and the abort
// word. expired() == true: give up.
struct Wait {
  u64 deadline = 0;
  unsigned spins = 0;
  __device__ __forceinline__ bool expired(const llar_llbuffer& b) {
    if ((++spins & 31u) != 0) return false;
    const u64 now = globaltimer_ns();
    if (deadline == 0) deadline = now + b.timeout_ns;
    return now > deadline || ld_relaxed_u32(b.abort_word) != 0;
  }
};

// Record a timeout of `rank` waiting for epoch E; the first one wins. Kept
// out of line (it is cold); internal linkage, so that any number of
// translation units of one program may include this header.
static __device__ __noinline__ void fail(const llar_llbuffer& b, int rank, u64 E) {
  if (atomicCAS(b.abort_word, 0u, 7u) == 0u) {
    volatile llar_llbuffer_status* st = b.status;
    st->rank = rank;
    st->epoch = E;
    __threadfence_system();
    st->code = 7u;
    __threadfence_system();
  }
}
__device__ __forceinline__ bool aborted(const llar_llbuffer& b) { return ld_relaxed_u32(b.abort_word) != 0; }

// ---------------------------------------------------------------- epochs
// When the kernel was launched as a programmatic dependent of the previous
// kernel in its stream, begin() first waits for that kernel to complete
// (griddepcontrol.wait; a no-op otherwise), then lets the next launch be
// scheduled early.
__device__ __forceinline__ u64 begin(const llar_llbuffer& b) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const u64 e = *reinterpret_cast<volatile const u64*>(b.epoch) + 1;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  return e;
}
// Every thread of every CTA, once, as the launch's last step: the last CTA
// to get here (all CTAs have read the counter by then: each read completed
// before its CTA counted itself) advances it by n. The next launch is
// stream-ordered after this one, so relaxed atomics suffice.
__device__ __forceinline__ void end(const llar_llbuffer& b, unsigned n) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned total = gridDim.x * gridDim.y * gridDim.z;
    if (atomicAdd(b.done_count, 1u) == total - 1) {
      *reinterpret_cast<volatile unsigned*>(b.done_count) = 0u;
      volatile u64* ep = b.epoch;
      *ep = *ep + (u64)n;
    }
  }
}
// The same with `first`, the value begin() returned: the counter every CTA
// read is first - 1 and nobody has written it since, so the last CTA
// writes first - 1 + n without reading it again (one round trip less at
// the end of the launch).
__device__ __forceinline__ void end(const llar_llbuffer& b, unsigned n, u64 first) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned total = gridDim.x * gridDim.y * gridDim.z;
    if (atomicAdd(b.done_count, 1u) == total - 1) {
      *reinterpret_cast<volatile unsigned*>(b.done_count) = 0u;
      *reinterpret_cast<volatile u64*>(b.epoch) = first - 1 + (u64)n;
    }
  }
}

// ================================================================ LL lines
// Technique 1: 8 bytes of data travel with an 8-byte flag (the epoch) in one
// 16-byte store, so a reader that sees the flag has the data; lines need no
// reset because epochs only grow. Rank q publishes word w of epoch E once,
// in its own staging; any rank may read it there.
//
// Credit rule (technique 3): rank q may publish word w for epoch E + 2 (same
// slot as E) only after every reader of word w at epoch E has read it. The
// usual way: each rank reads word w of epoch E + 1 from every peer before
// publishing w for E + 2, and every peer published E + 1 only after reading
// q's epoch-E line.
__device__ __forceinline__ char* ll_line(const llar_llbuffer& b, int q, u64 E, size_t w) {
  return static_cast<char*>(b.ll) + (size_t)q * b.ll_rank_stride + (size_t)(E & 1) * b.ll_slot_stride + w * 16;
}
__device__ __forceinline__ void ll_put(const llar_llbuffer& b, int q, u64 E, size_t w, u64 data) {
  st_relaxed_b128(ll_line(b, q, E, w), data, E);
}
// One poll of q's word w: true (and *data) if it carries epoch E.
__device__ __forceinline__ bool ll_try(const llar_llbuffer& b, int q, u64 E, size_t w, u64& data) {
  u64 lo, hi;
  ld_relaxed_b128(ll_line(b, q, E, w), lo, hi);
  data = lo;
  return hi == E;
}
// Poll q's word w until it carries epoch E; `me` is the rank reported on
// timeout. False on timeout or abort.
__device__ __forceinline__ bool ll_wait(const llar_llbuffer& b, int me, int q, u64 E, size_t w, u64& data) {
  Wait wt;
  for (bool first = true;; first = false) {
    LLB_ON_POLL_ROUND(first, 1u);
    if (ll_try(b, q, E, w, data)) return true;
    if (wt.expired(b)) {
      fail(b, me, E);
      return false;
    }
  }
}
// Poll word w of every rank but `me` at once (one load per pending rank per
// round); d[q] receives rank q's word, d[me] is left alone.
template <int N>
__device__ __forceinline__ bool ll_wait_peers(const llar_llbuffer& b, int me, u64 E, size_t w, u64 (&d)[N]) {
  unsigned pend = ((1u << N) - 1u) & ~(1u << me);
  Wait wt;
  for (bool first = true;; first = false) {
    LLB_ON_POLL_ROUND(first, pend);
    u64 lo[N], hi[N];
#pragma unroll
    for (int q = 0; q < N; ++q)
      if ((pend >> q) & 1u) ld_relaxed_b128(ll_line(b, q, E, w), lo[q], hi[q]);
#pragma unroll
    for (int q = 0; q < N; ++q)
      if (((pend >> q) & 1u) && hi[q] == E) {
        d[q] = lo[q];
        pend &= ~(1u << q);
      }
    if (pend == 0u) return true;
    if (wt.expired(b)) {
      fail(b, me, E);
      return false;
    }
  }
}
// Rank-order sum of N packed 8-byte words of T: float32 accumulation of
// ranks 0, 1, ..., N-1, one roundTiesToEven to T per element.
template <typename T, int N>
__device__ __forceinline__ u64 sum_words(const u64 (&d)[N]) {
  constexpr int PER = 8 / Elem<T>::kBytes;
  float acc[PER];
#pragma unroll
  for (int q = 0; q < N; ++q) {
    const unsigned w2[2] = {(unsigned)d[q], (unsigned)(d[q] >> 32)};
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const float v = Elem<T>::to_f(elem_get<T>(w2, i));
      acc[i] = (q == 0) ? v : __fadd_rn(acc[i], v);
    }
  }
  unsigned y[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < PER; ++i) elem_set<T>(y, i, Elem<T>::from_f(acc[i]));
  return (u64)y[0] | ((u64)y[1] << 32);
}
// The same two steps for a rank count known only at run time (b.nranks):
// d has room for the largest count (8 ranks).
__device__ __forceinline__ bool ll_wait_ranks(const llar_llbuffer& b, int me, u64 E, size_t w, u64 (&d)[8]) {
  unsigned pend = ((1u << b.nranks) - 1u) & ~(1u << me);
  Wait wt;
  for (bool first = true;; first = false) {
    LLB_ON_POLL_ROUND(first, pend);
    u64 lo[8], hi[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if ((pend >> q) & 1u) ld_relaxed_b128(ll_line(b, q, E, w), lo[q], hi[q]);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (((pend >> q) & 1u) && hi[q] == E) {
        d[q] = lo[q];
        pend &= ~(1u << q);
      }
    if (pend == 0u) return true;
    if (wt.expired(b)) {
      fail(b, me, E);
      return false;
    }
  }
}
template <typename T>
__device__ __forceinline__ u64 sum_words_ranks(const u64 (&d)[8], int n) {
  constexpr int PER = 8 / Elem<T>::kBytes;
  float acc[PER];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (q >= n) break;
    const unsigned w2[2] = {(unsigned)d[q], (unsigned)(d[q] >> 32)};
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const float v = Elem<T>::to_f(elem_get<T>(w2, i));
      acc[i] = (q == 0) ? v : __fadd_rn(acc[i], v);
    }
  }
  unsigned y[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < PER; ++i) elem_set<T>(y, i, Elem<T>::from_f(acc[i]));
  return (u64)y[0] | ((u64)y[1] << 32);
}

// One word of a one-shot AllReduce: publish mine, poll every peer's, sum in
// rank order. The thread that handles word w must handle it at every epoch
// (that carries the credit rule above).
template <typename T, int N>
__device__ __forceinline__ bool ll_allreduce_word(const llar_llbuffer& b, int me, u64 E, size_t w, u64 mine, u64& y) {
  u64 d[N];
  ll_put(b, me, E, w, mine);
  d[me] = mine;
  if (!ll_wait_peers<N>(b, me, E, w, d)) return false;
  y = sum_words<T, N>(d);
  return true;
}

// ========================================================= sentinel vectors
// Technique 2: the receiver's slot holds the all-ones pattern (-NaN in
// every element type) until data lands; the receiver polls until no element
// is all-ones, takes the vector and writes the pattern back. Data that
// contains the pattern cannot be sent this way.
//
// Credit rule (technique 3): source q may write slot s of receiver d again
// (two exchanges later) only after receiving, from d, an exchange that d
// sent after resetting that slot; d must fence_gpu() between the reset and
// that send. With one exchange per epoch in both directions: at the start
// of each exchange every thread calls fence_gpu(), then sends, then waits.
__device__ __forceinline__ char* sen_vec(const llar_llbuffer& b, int d, int s, int q, size_t v) {
  return static_cast<char*>(b.sen) + (size_t)d * b.sen_rank_stride + (size_t)s * b.sen_slot_stride +
         (size_t)q * b.sen_src_stride + v * 16;
}
// source q -> receiver d, slot s, vector v
__device__ __forceinline__ void sen_put(const llar_llbuffer& b, int d, int q, int s, size_t v, uint4 x) {
  st_relaxed_v4(sen_vec(b, d, s, q, v), x);
}
template <typename T>
__device__ __forceinline__ bool has_pattern(uint4 v) {
  const unsigned w[4] = {v.x, v.y, v.z, v.w};
  bool any = false;
#pragma unroll
  for (int i = 0; i < 16 / Elem<T>::kBytes; ++i) any |= elem_get<T>(w, i) == Elem<T>::kMask;
  return any;
}
// Receiver d takes vector v from source q in slot s (E: epoch reported on
// timeout) and resets it. False on timeout or abort.
template <typename T>
__device__ __forceinline__ bool sen_take(const llar_llbuffer& b, int d, int q, int s, size_t v, u64 E, uint4& x) {
  char* p = sen_vec(b, d, s, q, v);
  Wait wt;
  for (bool first = true;; first = false) {
    LLB_ON_POLL_ROUND(first, 1u);
    x = ld_relaxed_v4(p);
    if (!has_pattern<T>(x)) break;
    if (wt.expired(b)) {
      fail(b, d, E);
      return false;
    }
  }
  st_relaxed_v4(p, make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu));
  return true;
}
// Receiver d takes vector v of slot s from every source but itself at once
// (one load per pending source per round, so the waits overlap), resetting
// each slot as its vector arrives; x[q] receives source q's vector, x[d] is
// left alone. False on timeout or abort.
template <typename T, int N>
__device__ __forceinline__ bool sen_take_peers(const llar_llbuffer& b, int d, int s, size_t v, u64 E, uint4 (&x)[N]) {
  const uint4 ones = make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
  unsigned pend = ((1u << N) - 1u) & ~(1u << d);
  Wait wt;
  for (bool first = true;; first = false) {
    LLB_ON_POLL_ROUND(first, pend);
    uint4 t[N];
#pragma unroll
    for (int q = 0; q < N; ++q)
      if ((pend >> q) & 1u) t[q] = ld_relaxed_v4(sen_vec(b, d, s, q, v));
#pragma unroll
    for (int q = 0; q < N; ++q)
      if (((pend >> q) & 1u) && !has_pattern<T>(t[q])) {
        x[q] = t[q];
        pend &= ~(1u << q);
        st_relaxed_v4(sen_vec(b, d, s, q, v), ones);
      }
    if (pend == 0u) return true;
    if (wt.expired(b)) {
      fail(b, d, E);
      return false;
    }
  }
}

// ============================================================ LL128 lines
// Technique 4: a 128-byte line is 8 lanes x 16 bytes; element 0 of lane 0
// counts the contributions, the other 128/sizeof(T) - 1 elements carry data.
// Every contributor adds its data into the owner's line with vector
// reductions in T, then (after a fence) adds 1 to the count; when the count
// reads N every contribution is in. Additions in T happen in arrival order:
// the result is not deterministic.
//
// Lines are handled by groups of 8 consecutive lanes of a warp (lane & 7 is
// the lane of the line), and every primitive here is called by all 32 lanes
// of the warp together (a lane without a line passes active = false).
//
// Reuse (technique 3): the owner zeroes the line in ll128_take; a
// contributor may add into the same slot again (two epochs later) only
// after observing something the owner wrote after a fence_gpu() that
// followed that zeroing (ll128_add of the owner's next epoch contains such
// a fence, so the owner's LL AllGather lines of epoch E + 1 qualify).
template <typename T>
__device__ __forceinline__ constexpr int ll128_payload() { return 128 / Elem<T>::kBytes - 1; }

__device__ __forceinline__ char* ll128_line(const llar_llbuffer& b, int o, int s, size_t l) {
  return static_cast<char*>(b.ll128) + (size_t)o * b.ll128_rank_stride + (size_t)s * b.ll128_slot_stride + l * 128;
}
// Lane `lane` (0..7) of line l of a segment `seg` (seg_len elements): the
// 16 bytes the line carries there; element 0 of lane 0 (the count) and
// elements past the end read as zero.
template <typename T>
__device__ __forceinline__ uint4 ll128_pack(const T* seg, size_t seg_len, size_t l, int lane) {
  constexpr int V = 16 / Elem<T>::kBytes;
  unsigned w[4] = {0u, 0u, 0u, 0u};
  const unsigned short* s16 = reinterpret_cast<const unsigned short*>(seg);
  const unsigned* s32 = reinterpret_cast<const unsigned*>(seg);
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int pos = lane * V + k;
    const size_t i = l * ll128_payload<T>() + (size_t)pos - 1;
    if (pos >= 1 && i < seg_len) elem_set<T>(w, k, Elem<T>::kBytes == 4 ? s32[i] : s16[i]);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
// The inverse: store the data elements of lane `lane` of line l.
template <typename T>
__device__ __forceinline__ void ll128_unpack(T* seg, size_t seg_len, size_t l, int lane, uint4 v) {
  constexpr int V = 16 / Elem<T>::kBytes;
  const unsigned w[4] = {v.x, v.y, v.z, v.w};
  unsigned short* s16 = reinterpret_cast<unsigned short*>(seg);
  unsigned* s32 = reinterpret_cast<unsigned*>(seg);
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int pos = lane * V + k;
    const size_t i = l * ll128_payload<T>() + (size_t)pos - 1;
    if (pos >= 1 && i < seg_len) {
      if (Elem<T>::kBytes == 4) s32[i] = elem_get<T>(w, k);
      else s16[i] = (unsigned short)elem_get<T>(w, k);
    }
  }
}
// Add my lane data (from ll128_pack) into owner o's line l of slot s, then
// count the contribution. All 32 lanes call; active = false skips a lane.
template <typename T>
__device__ __forceinline__ void ll128_add(const llar_llbuffer& b, int o, int s, size_t l, int lane, uint4 data,
                                          bool active) {
  char* line = ll128_line(b, o, s, l);
  if (active && (data.x | data.y | data.z | data.w)) Elem<T>::red_v4(line + lane * 16, data);
  __syncwarp();
  fence_gpu();  // every data reduction of the warp before any count
  if (active && lane == 0) Elem<T>::red_one(line);
}
// Owner o: wait until line l of slot s counts N contributions, return my
// lane's 16 bytes (lane 0's element 0 holds the count) and zero the line.
// All 32 lanes call; active = false skips a lane. E: epoch reported on
// timeout. False on timeout or abort.
template <typename T>
__device__ __forceinline__ bool ll128_take(const llar_llbuffer& b, int o, int s, size_t l, int lane, u64 E,
                                           bool active, uint4& data) {
  char* line = ll128_line(b, o, s, l);
  const unsigned want = Elem<T>::from_f((float)b.nranks);
  bool ok = true;
  data = make_uint4(0u, 0u, 0u, 0u);
  if (active) {
    Wait wt;
    for (bool first = true;; first = false) {
      LLB_ON_POLL_ROUND(first, 1u);
      if ((ld_acquire_u32(line) & Elem<T>::kMask) == want) break;
      if (wt.expired(b)) {
        fail(b, o, E);
        ok = false;
        break;
      }
    }
    if (ok) data = ld_relaxed_v4(line + lane * 16);
  }
  __syncwarp();  // every lane has its data before any lane zeroes
  if (active && ok) st_relaxed_v4(line + lane * 16, make_uint4(0u, 0u, 0u, 0u));
  return ok;
}

}  // namespace llb
