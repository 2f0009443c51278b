// Device-side building blocks: GPU-scope loads/stores/reductions in inline
// PTX, element formats, bounded waits and error reporting.
//
// Memory-model notes (PTX ISA memory consistency model):
//  * Signalling loads and stores are .relaxed.gpu: they are morally strong,
//    go to L2 (not the non-coherent L1), and never form a data race.
//  * A producer that must make earlier writes (a reset of a sentinel slot,
//    zeroing of an LL128 line, data reductions before a count flag) visible
//    before a later signal issues fence.acq_rel.gpu between them: fence
//    followed by a strong write is a release pattern.
//  * A consumer's completed poll (a relaxed load whose value was tested)
//    gates its later stores through a control dependency; stores are not
//    issued before the branch on the loaded value resolves. Where a consumer
//    reads *other* locations after seeing a flag (LL128 count flag, fixed
//    path ready flags) the flag load is ld.acquire.gpu.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "llar_internal.h"

#ifdef LLAR_POLL_STATS
// Poll-counting build (diagnostic, a separate library): per warp and
// polling round, the lowest active lane adds the active lanes (thread
// rounds), the lines they load, the waits whose first round this is and
// the lines those waits await. One reduction per warp and round, issued
// without waiting for its result.
static __device__ unsigned long long g_llar_poll_stats[4];
static __device__ __forceinline__ void llar_poll_stat(bool first, unsigned pending) {
  const unsigned m = __activemask();
  const unsigned loads = __reduce_add_sync(m, (unsigned)__popc(pending));
  const unsigned starts = __popc(__ballot_sync(m, first));
  const unsigned awaited = __reduce_add_sync(m, first ? (unsigned)__popc(pending) : 0u);
  if ((int)(threadIdx.x & 31u) == __ffs(m) - 1) {
    atomicAdd(&g_llar_poll_stats[0], (unsigned long long)__popc(m));
    atomicAdd(&g_llar_poll_stats[1], (unsigned long long)loads);
    if (starts) {
      atomicAdd(&g_llar_poll_stats[2], (unsigned long long)starts);
      atomicAdd(&g_llar_poll_stats[3], (unsigned long long)awaited);
    }
  }
}
#define LLB_ON_POLL_ROUND(first, pending) llar_poll_stat((first), (pending))
#endif

#include "llar_llbuffer.cuh"

namespace llar {

typedef unsigned long long u64;

// ------------------------------------------------------------------ PTX
// The signalling accesses shared with the public device primitives.
using llb::fence_gpu;
using llb::globaltimer_ns;
using llb::ld_acquire_u32;
using llb::ld_relaxed_b128;
using llb::ld_relaxed_u32;
using llb::ld_relaxed_v4;
using llb::st_relaxed_b128;
using llb::st_relaxed_v4;

__device__ __forceinline__ u64 ld_relaxed_u64(const void* p) {
  u64 v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ u64 ld_acquire_u64(const void* p) {
  u64 v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(void* p, u64 v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

// read-only streaming load (inputs that no one writes during the launch)
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
// L2-coherent load (data another CTA wrote during this launch)
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
// streaming store: the line is not expected to be reused from L2
__device__ __forceinline__ void st_cs_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// ----------------------------------------------- TMA bulk copy + mbarrier
__device__ __forceinline__ unsigned smem_addr(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
// make initialised barriers visible to the async (bulk copy) proxy
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16)
// completing `bytes` transactions on barrier `bar`
__device__ __forceinline__ void bulk_load(unsigned dst, const void* src, unsigned bytes, unsigned bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(unsigned a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}

// --------------------------------------------------------- element formats
// DT: 0 = fp32, 1 = fp16, 2 = bf16 (llar_dtype_t values).
template <int DT> struct Fmt;

template <> struct Fmt<0> {
  static constexpr int kBytes = 4;
  static constexpr unsigned kSentinel = 0xFFFFFFFFu;
  __device__ static __forceinline__ float to_f(unsigned b) { return __uint_as_float(b); }
  __device__ static __forceinline__ unsigned from_f(float f) { return __float_as_uint(f); }
  __device__ static __forceinline__ unsigned load(const char* base, size_t i) {
    return *reinterpret_cast<const unsigned*>(base + i * 4);
  }
  __device__ static __forceinline__ void store(char* base, size_t i, unsigned b) {
    *reinterpret_cast<unsigned*>(base + i * 4) = b;
  }
};
template <> struct Fmt<1> {
  static constexpr int kBytes = 2;
  static constexpr unsigned kSentinel = 0xFFFFu;
  __device__ static __forceinline__ float to_f(unsigned b) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
  }
  __device__ static __forceinline__ unsigned from_f(float f) {
    return __half_as_ushort(__float2half_rn(f));
  }
  __device__ static __forceinline__ unsigned load(const char* base, size_t i) {
    return *reinterpret_cast<const unsigned short*>(base + i * 2);
  }
  __device__ static __forceinline__ void store(char* base, size_t i, unsigned b) {
    *reinterpret_cast<unsigned short*>(base + i * 2) = static_cast<unsigned short>(b);
  }
};
template <> struct Fmt<2> {
  static constexpr int kBytes = 2;
  static constexpr unsigned kSentinel = 0xFFFFu;
  __device__ static __forceinline__ float to_f(unsigned b) { return __uint_as_float(b << 16); }
  __device__ static __forceinline__ unsigned from_f(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
  }
  __device__ static __forceinline__ unsigned load(const char* base, size_t i) {
    return *reinterpret_cast<const unsigned short*>(base + i * 2);
  }
  __device__ static __forceinline__ void store(char* base, size_t i, unsigned b) {
    *reinterpret_cast<unsigned short*>(base + i * 2) = static_cast<unsigned short>(b);
  }
};

// Elements of a 32-bit word: element k of word w (little endian).
template <int DT>
__device__ __forceinline__ unsigned word_elem(unsigned w, int k) {
  if (Fmt<DT>::kBytes == 4) return w;
  return (w >> (16 * k)) & 0xFFFFu;
}
template <int DT>
__device__ __forceinline__ unsigned word_set(unsigned w, int k, unsigned e) {
  if (Fmt<DT>::kBytes == 4) return e;
  const unsigned sh = 16 * k;
  return (w & ~(0xFFFFu << sh)) | (e << sh);
}

// acc[i] += value of element i of a packed group of 32-bit words
template <int DT, int NW>
__device__ __forceinline__ void accumulate(float* acc, const unsigned* w) {
  constexpr int PER = 4 / Fmt<DT>::kBytes;
#pragma unroll
  for (int i = 0; i < NW; ++i)
#pragma unroll
    for (int k = 0; k < PER; ++k)
      acc[i * PER + k] = __fadd_rn(acc[i * PER + k], Fmt<DT>::to_f(word_elem<DT>(w[i], k)));
}
template <int DT, int NW>
__device__ __forceinline__ void init_acc(float* acc, const unsigned* w) {
  constexpr int PER = 4 / Fmt<DT>::kBytes;
#pragma unroll
  for (int i = 0; i < NW; ++i)
#pragma unroll
    for (int k = 0; k < PER; ++k) acc[i * PER + k] = Fmt<DT>::to_f(word_elem<DT>(w[i], k));
}
// round every accumulator once (roundTiesToEven) and pack into words
template <int DT, int NW>
__device__ __forceinline__ void pack_acc(const float* acc, unsigned* w) {
  constexpr int PER = 4 / Fmt<DT>::kBytes;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    unsigned x = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) x = word_set<DT>(x, k, Fmt<DT>::from_f(acc[i * PER + k]));
    w[i] = x;
  }
}
// next input of a chain: roundTiesToEven(scale * y), product in float32
template <int DT, int NW>
__device__ __forceinline__ void chain_words(const unsigned* y, unsigned* nx, float scale) {
  constexpr int PER = 4 / Fmt<DT>::kBytes;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    unsigned x = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k)
      x = word_set<DT>(x, k, Fmt<DT>::from_f(__fmul_rn(scale, Fmt<DT>::to_f(word_elem<DT>(y[i], k)))));
    nx[i] = x;
  }
}

__device__ __forceinline__ bool is_all_ones(uint4 v) { return (v.x & v.y & v.z & v.w) == 0xFFFFFFFFu; }

// True if any element of the 16-byte vector is the sentinel pattern.
template <int DT>
__device__ __forceinline__ bool has_sentinel(uint4 v) {
  if (Fmt<DT>::kBytes == 4)
    return v.x == 0xFFFFFFFFu || v.y == 0xFFFFFFFFu || v.z == 0xFFFFFFFFu || v.w == 0xFFFFFFFFu;
  auto h = [](unsigned w) {
    return ((w & 0xFFFFu) == 0xFFFFu) || ((w >> 16) == 0xFFFFu);
  };
  return h(v.x) || h(v.y) || h(v.z) || h(v.w);
}

// Load n32 32-bit words of a vector that may run past `count` elements:
// words (and elements) at or beyond the end read as zero.
template <int DT, int NW>
__device__ __forceinline__ void load_words_tail(const char* base, size_t first_elem, size_t count,
                                                unsigned* w) {
  constexpr int PER = 4 / Fmt<DT>::kBytes;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    unsigned x = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const size_t g = first_elem + i * PER + k;
      if (g < count) x = word_set<DT>(x, k, Fmt<DT>::load(base, g));
    }
    w[i] = x;
  }
}
template <int DT, int NW>
__device__ __forceinline__ void store_words_tail(char* base, size_t first_elem, size_t count,
                                                 const unsigned* w) {
  constexpr int PER = 4 / Fmt<DT>::kBytes;
#pragma unroll
  for (int i = 0; i < NW; ++i)
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const size_t g = first_elem + i * PER + k;
      if (g < count) Fmt<DT>::store(base, g, word_elem<DT>(w[i], k));
    }
}

// ------------------------------------------------------------ bounded waits
// Counts polls; every 32nd poll it reads %globaltimer (the deadline is set
// on the first reading, so short waits never read the clock) and the
// launch-wide abort word. expired() == true means: give up.
struct Waiter {
  u64 deadline = 0;
  unsigned spins = 0;
  __device__ __forceinline__ bool expired(const Params& p) {
    if ((++spins & 31u) != 0) return false;
    const u64 now = globaltimer_ns();
    if (deadline == 0) deadline = now + p.timeout_ns;
    if (now > deadline) return true;
    return ld_relaxed_u32(p.abort_flag) != 0;
  }
};

// First failing wait wins the device word and fills the host-visible status.
__device__ __noinline__ void report_timeout(const Params& p, int rank, int cta, u64 epoch) {
  if (atomicCAS(p.abort_flag, 0u, 7u) == 0u) {
    volatile DevStatus* st = p.status;
    st->rank = rank;
    st->cta = cta;
    st->epoch = epoch;
    __threadfence_system();
    st->code = 7u;
    __threadfence_system();
  }
}

__device__ __forceinline__ bool aborted(const Params& p) {
  return ld_relaxed_u32(p.abort_flag) != 0;
}

// Injected sleep of the DELAY fault mode (about 20 us, bounded).
__device__ __forceinline__ void injected_delay() {
  for (int i = 0; i < 20; ++i) __nanosleep(1000);
}

}  // namespace llar
