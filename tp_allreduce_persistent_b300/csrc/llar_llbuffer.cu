// The LL buffer API: host calls of llar_llbuffer.h, and the library kernels
// that are written ONLY against the public device primitives of
// llar_llbuffer.cuh (no internal header reaches their device code), as a
// user's custom kernel would be: one-shot LL and sentinel AllReduces, the
// two-shot LL128 atomic AllReduce, and a tensor-parallel row-parallel
// linear layer (GEMV) whose epilogue is the LL AllReduce ("Every
// Microsecond Matters: Achieving Near Speed-of-Light Latency in GPU
// Collectives", summary page: the four techniques packaged as a buffer API
// for custom kernels).
//
// Virtual ranks as everywhere in this library: block b is CTA b / N of rank
// b % N, and CTA c of every rank covers the same share of the data, so the
// thread that handles a word or line of one rank handles the same word or
// line at every epoch and on every rank (this carries the credit rules).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "llar.h"
#include "llar_llbuffer.cuh"
#include "llar_llbuffer.h"

namespace {

using llb::u64;
constexpr int kMaxN = 8;
constexpr size_t kMaxBytes = size_t(1) << 30;
constexpr int kLinearMaxM = 16;
constexpr size_t kLinearMaxXBytes = 96 * 1024;
constexpr int kLinearThreads = 256;  // 8 warps split K
constexpr int kLinearWarps = kLinearThreads / 32;

struct Ptrs {
  const char* in[kMaxN];
  char* out[kMaxN];
};

// ------------------------------------------------------ tail-safe access
// Word w of 8 bytes (vector v of 16 bytes) of a buffer of `nbytes` bytes:
// bytes past the end read as zero and are not written.
__device__ __forceinline__ u64 load_word(const char* base, size_t w, size_t nbytes) {
  const size_t off = w * 8;
  if (off + 8 <= nbytes) return *reinterpret_cast<const u64*>(base + off);
  u64 v = 0;
  for (size_t i = off; i < nbytes; ++i) v |= (u64)(unsigned char)base[i] << (8 * (i - off));
  return v;
}
__device__ __forceinline__ void store_word(char* base, size_t w, size_t nbytes, u64 v) {
  const size_t off = w * 8;
  if (off + 8 <= nbytes) {
    *reinterpret_cast<u64*>(base + off) = v;
    return;
  }
  for (size_t i = off; i < nbytes; ++i) base[i] = (char)(v >> (8 * (i - off)));
}
__device__ __forceinline__ uint4 load_vec(const char* base, size_t v, size_t nbytes) {
  const size_t off = v * 16;
  if (off + 16 <= nbytes) return *reinterpret_cast<const uint4*>(base + off);
  const u64 lo = load_word(base, 2 * v, nbytes), hi = load_word(base, 2 * v + 1, nbytes);
  return make_uint4((unsigned)lo, (unsigned)(lo >> 32), (unsigned)hi, (unsigned)(hi >> 32));
}
__device__ __forceinline__ void store_vec(char* base, size_t v, size_t nbytes, uint4 x) {
  const size_t off = v * 16;
  if (off + 16 <= nbytes) {
    *reinterpret_cast<uint4*>(base + off) = x;
    return;
  }
  store_word(base, 2 * v, nbytes, (u64)x.x | ((u64)x.y << 32));
  store_word(base, 2 * v + 1, nbytes, (u64)x.z | ((u64)x.w << 32));
}

// share [lo, hi) of `units` for CTA c of G
__device__ __forceinline__ void share(size_t units, int c, int G, size_t& lo, size_t& hi) {
  const size_t per = (units + G - 1) / G;
  lo = min(units, (size_t)c * per);
  hi = min(units, lo + per);
}

// ========================================================== LL one-shot
// Each thread owns LL words; iteration e+1's line (same input) goes out as
// soon as iteration e's word arrived from every peer (credit rule: my next
// publication of this word's slot waits for every peer's line of the
// following epoch).
template <typename T, int N>
__global__ void __launch_bounds__(512) kb_ll(const llar_llbuffer b, const Ptrs io, size_t nbytes, int iters, int G) {
  const u64 E0 = llb::begin(b);
  const int r = blockIdx.x % N, c = blockIdx.x / N;
  size_t w0, w1;
  share((nbytes + 7) / 8, c, G, w0, w1);
  for (size_t w = w0 + threadIdx.x; w < w1; w += blockDim.x) llb::ll_put(b, r, E0, w, load_word(io.in[r], w, nbytes));
  bool ok = true;
  for (int e = 0; e < iters && ok; ++e) {
    const u64 E = E0 + (u64)e;
    for (size_t w = w0 + threadIdx.x; w < w1; w += blockDim.x) {
      u64 d[N];
      d[r] = load_word(io.in[r], w, nbytes);
      if (!llb::ll_wait_peers<N>(b, r, E, w, d)) {
        ok = false;
        break;
      }
      if (e + 1 < iters) llb::ll_put(b, r, E + 1, w, d[r]);
      store_word(io.out[r], w, nbytes, llb::sum_words<T, N>(d));
    }
  }
  llb::end(b, (unsigned)iters, E0);
}

// ====================================================== sentinel one-shot
// One exchange per epoch in slot E & 1; a fence at its start releases this
// thread's resets of the previous exchange before its new sends.
template <typename T, int N>
__global__ void __launch_bounds__(512) kb_sentinel(const llar_llbuffer b, const Ptrs io, size_t nbytes, int iters,
                                                   int G) {
  const u64 E0 = llb::begin(b);
  const int r = blockIdx.x % N, c = blockIdx.x / N;
  constexpr int PER = 16 / llb::Elem<T>::kBytes;
  size_t v0, v1;
  share((nbytes + 15) / 16, c, G, v0, v1);
  bool ok = true;
  for (int e = 0; e < iters && ok; ++e) {
    const u64 E = E0 + (u64)e;
    const int s = (int)(E & 1);
    llb::fence_gpu();
    for (size_t v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
      const uint4 x = load_vec(io.in[r], v, nbytes);
#pragma unroll
      for (int q = 0; q < N; ++q)
        if (q != r) llb::sen_put(b, q, r, s, v, x);
    }
    for (size_t v = v0 + threadIdx.x; v < v1 && ok; v += blockDim.x) {
      const uint4 own = load_vec(io.in[r], v, nbytes);
      uint4 x[N];
      if (!llb::sen_take_peers<T, N>(b, r, s, v, E, x)) {
        ok = false;
        break;
      }
      float acc[PER];
#pragma unroll
      for (int q = 0; q < N; ++q) {
        const uint4 xq = q == r ? own : x[q];
        const unsigned w[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const float f = llb::Elem<T>::to_f(llb::elem_get<T>(w, i));
          acc[i] = (q == 0) ? f : __fadd_rn(acc[i], f);
        }
      }
      unsigned y[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int i = 0; i < PER; ++i) llb::elem_set<T>(y, i, llb::Elem<T>::from_f(acc[i]));
      store_vec(io.out[r], v, nbytes, make_uint4(y[0], y[1], y[2], y[3]));
    }
  }
  llb::end(b, (unsigned)iters, E0);
}

// ======================================================= LL128 two-shot
// Rank s owns segment s (ceil(count / N) elements) in LL128 lines. Item i
// of a CTA is (segment s, line l, lane j) with i & 7 == j, so the 8 lanes
// of a line are 8 consecutive lanes of one warp. ReduceScatter: ll128_add
// into every owner's line. Owner: ll128_take, write my output, publish the
// lane as two LL words (AllGather). Everyone: poll the other owners' words.
template <typename T, int N>
__global__ void __launch_bounds__(512) kb_ll128(const llar_llbuffer b, const Ptrs io, size_t count, int iters,
                                                int G) {
  const u64 E0 = llb::begin(b);
  const int r = blockIdx.x % N, c = blockIdx.x / N;
  constexpr int P = llb::ll128_payload<T>();
  const size_t seg = (count + N - 1) / N;
  auto seg_len = [&](int s) -> size_t {
    const size_t lo = min(count, (size_t)s * seg);
    return min(count, lo + seg) - lo;
  };
  const size_t L = (seg + P - 1) / P;
  size_t l0, l1;
  share(L, c, G, l0, l1);
  const size_t nl = l1 - l0;
  const size_t items = (size_t)N * nl * 8;
  const size_t T_ = blockDim.x;
  const T* in = reinterpret_cast<const T*>(io.in[r]);
  T* out = reinterpret_cast<T*>(io.out[r]);
  bool ok = true;
  for (int e = 0; e < iters && ok; ++e) {
    const u64 E = E0 + (u64)e;
    const int slot = (int)(E & 1);
    // ReduceScatter
    for (size_t base = 0; base < items; base += T_) {
      const size_t i = base + threadIdx.x;
      const bool active = i < items;
      const int s = active ? (int)(i / (nl * 8)) : 0;
      const size_t l = active ? l0 + (i % (nl * 8)) / 8 : 0;
      const int j = (int)(i & 7);
      const uint4 d = active ? llb::ll128_pack<T>(in + (size_t)s * seg, seg_len(s), l, j) : make_uint4(0, 0, 0, 0);
      llb::ll128_add<T>(b, s, slot, l, j, d, active);
    }
    // owner: take my lines, keep them, send them
    const size_t mine = nl * 8;
    for (size_t base = 0; base < mine; base += T_) {
      const size_t i = base + threadIdx.x;
      const bool active = i < mine;
      const size_t l = l0 + i / 8;
      const int j = (int)(i & 7);
      uint4 d;
      if (!llb::ll128_take<T>(b, r, slot, l, j, E, active, d)) ok = false;
      if (active && ok) {
        llb::ll128_unpack<T>(out + (size_t)r * seg, seg_len(r), l, j, d);
        llb::ll_put(b, r, E, (l * 8 + j) * 2, (u64)d.x | ((u64)d.y << 32));
        llb::ll_put(b, r, E, (l * 8 + j) * 2 + 1, (u64)d.z | ((u64)d.w << 32));
      }
    }
    if (__syncthreads_or(!ok)) break;
    // AllGather receive
    for (size_t i = threadIdx.x; i < items && ok; i += T_) {
      const int s = (int)(i / (nl * 8));
      if (s == r) continue;
      const size_t l = l0 + (i % (nl * 8)) / 8;
      const int j = (int)(i & 7);
      // the lane's two words, polled in the same round
      u64 lo = 0, hi = 0;
      bool got_lo = false, got_hi = false;
      llb::Wait wt;
      while (!(got_lo && got_hi)) {
        if (!got_lo) got_lo = llb::ll_try(b, s, E, (l * 8 + j) * 2, lo);
        if (!got_hi) got_hi = llb::ll_try(b, s, E, (l * 8 + j) * 2 + 1, hi);
        if (!(got_lo && got_hi) && wt.expired(b)) {
          llb::fail(b, r, E);
          ok = false;
          break;
        }
      }
      if (!ok) break;
      llb::ll128_unpack<T>(out + (size_t)s * seg, seg_len(s), l, j,
                           make_uint4((unsigned)lo, (unsigned)(lo >> 32), (unsigned)hi, (unsigned)(hi >> 32)));
    }
    if (__syncthreads_or(!ok)) break;
  }
  llb::end(b, (unsigned)iters, E0);
}

// ================================================= fused linear + AllReduce
// CTA tile: 32 lanes x LW bytes of output columns (LW / sizeof(T) columns a
// lane) for all M rows. The 8 warps split K into contiguous slices; a lane
// streams its columns of w row by row (UNROLL rows in flight) and keeps
// float32 sums for every row of x (fused multiply-add, one rounding per
// term; for fp16/bf16 operands the product is exact in float32). The
// slices are added in warp order through shared memory and rounded to T.
// Fused: phase 1 publishes each (row, LL word) of the partial as an LL line
// for every tile of the CTA; phase 2 polls every rank's line of those words
// and adds them in rank order (the AllReduce), so a rank's GEMV never waits
// for another's. Unfused (FUSE = false): the rounded partial goes to memory.
// MT is M rounded up to a power of two (registers scale with it).
struct LinearArgs {
  const char* x[kMaxN];
  const char* w[kMaxN];
  char* out[kMaxN];
  int n, m, k, h;
};

template <typename T>
__device__ __forceinline__ float elem_f(const T* p, size_t i) {
  if (llb::Elem<T>::kBytes == 4) return llb::Elem<T>::to_f(reinterpret_cast<const unsigned*>(p)[i]);
  return llb::Elem<T>::to_f(reinterpret_cast<const unsigned short*>(p)[i]);
}

// float32 values of elements (2i, 2i + 1) of a packed group of words, as
// one 64-bit pair (element 2i in the low half)
template <typename T>
__device__ __forceinline__ u64 pair_of(const unsigned* v, int i) {
  if (llb::Elem<T>::kBytes == 4) return (u64)v[2 * i] | ((u64)v[2 * i + 1] << 32);
  const unsigned w = v[i];
  const float lo = llb::Elem<T>::to_f(w & 0xFFFFu), hi = llb::Elem<T>::to_f(w >> 16);
  return (u64)__float_as_uint(lo) | ((u64)__float_as_uint(hi) << 32);
}
// the MT activations of one k from shared memory, in 16-, 8-, 4- or 2-byte loads
template <int XROW>
__device__ __forceinline__ void load_xrow(const unsigned char* p, unsigned (&w)[(XROW + 3) / 4]) {
  if (XROW >= 16) {
#pragma unroll
    for (int i = 0; i < XROW / 16; ++i) {
      const uint4 v = reinterpret_cast<const uint4*>(p)[i];
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
  } else if (XROW == 8) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x;
    w[1] = v.y;
  } else if (XROW == 4) {
    w[0] = *reinterpret_cast<const unsigned*>(p);
  } else {
    w[0] = *reinterpret_cast<const unsigned short*>(p);
  }
}
// acc (two float32 lanes) += x * w lane by lane, one rounding per lane
__device__ __forceinline__ void fma2(u64& acc, u64 x, u64 w) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(x), "l"(w));
}

template <int LW>
__device__ __forceinline__ void load_lane(const char* p, unsigned (&v)[LW / 4]) {
  if (LW == 16) {
    const uint4 q = __ldcs(reinterpret_cast<const uint4*>(p));
    v[0] = q.x;
    v[1] = q.y;
    v[2] = q.z;
    v[3] = q.w;
  } else {
    const uint2 q = __ldcs(reinterpret_cast<const uint2*>(p));
    v[0] = q.x;
    v[1] = q.y;
  }
}

template <typename T, int MT, int LW, bool FUSE>
__global__ void __launch_bounds__(kLinearThreads, 2) kb_linear(const llar_llbuffer b, const LinearArgs a, int G) {
  constexpr int EB = llb::Elem<T>::kBytes;
  constexpr int VEC = LW / EB;       // columns per lane
  constexpr int COLS = 32 * VEC;     // columns per tile
  constexpr int WPL = LW / 8;        // LL words per lane per row
  constexpr int UNROLL = (MT <= 2 && LW == 16) ? 16 : 8;  // weight rows in flight per lane
  extern __shared__ __align__(16) unsigned char smem[];
  const u64 E = FUSE ? llb::begin(b) : 0;
  // block b is CTA b / N of rank b % N, as everywhere
  const int n = a.n;
  const int rank = (int)(blockIdx.x % n), cta = (int)(blockIdx.x / n);
  const int M = a.m, K = a.k, H = a.h;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // x staged transposed, [k][MT] with rows M..MT-1 zero: the activations
  // of one k for every row come in one or two vector loads
  unsigned char* xs = smem;
  constexpr int XROW = MT * EB;  // bytes per k
  const size_t xbytes = ((size_t)K * XROW + 15) & ~size_t(15);
  float* part = reinterpret_cast<float*>(smem + xbytes);  // [warp][m][COLS]
  const T* x = reinterpret_cast<const T*>(a.x[rank]);
  const char* w = a.w[rank];
  char* out = a.out[rank];
  constexpr int PV = 16 / EB;  // elements per 16-byte load
  if (K % PV == 0) {  // rows of x start on 16-byte boundaries: 16-byte loads, scattered to [k][MT]
    const int rowv = K / PV;
    for (int i = threadIdx.x; i < MT * rowv; i += blockDim.x) {
      const int m = i / rowv, j = i % rowv;
      const uint4 v = m < M ? *reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(x) +
                                                              ((size_t)m * K + (size_t)j * PV) * EB)
                            : make_uint4(0, 0, 0, 0);
      const unsigned w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < PV; ++u) {
        const size_t kk = (size_t)j * PV + u;
        if (EB == 4) reinterpret_cast<unsigned*>(xs)[kk * MT + m] = w4[u];
        else reinterpret_cast<unsigned short*>(xs)[kk * MT + m] = (unsigned short)llb::elem_get<T>(w4, u);
      }
    }
  } else {
    for (size_t i = threadIdx.x; i < (size_t)K * MT; i += blockDim.x) {
      const size_t kk = i / MT, m = i % MT;
      const unsigned b = m < (size_t)M ? (EB == 4 ? reinterpret_cast<const unsigned*>(x)[m * K + kk]
                                                  : reinterpret_cast<const unsigned short*>(x)[m * K + kk])
                                       : 0u;
      if (EB == 4) reinterpret_cast<unsigned*>(xs)[i] = b;
      else reinterpret_cast<unsigned short*>(xs)[i] = (unsigned short)b;
    }
  }
  __syncthreads();
  const int tiles = (H + COLS - 1) / COLS;
  const int words_per_row = H / (8 / EB);
  const int kc = (K + kLinearWarps - 1) / kLinearWarps;
  const int k0 = min(K, warp * kc), k1 = min(K, k0 + kc);
  const size_t row_bytes = (size_t)H * EB;

  // ---- phase 1: GEMV of every tile of this CTA
  for (int t = cta; t < tiles; t += G) {
    const int col = t * COLS + lane * VEC;  // first column of my lane
    // accumulators in float32 pairs (columns i, i + 1), updated with the
    // packed two-lane fused multiply-add: each lane rounds once, exactly as
    // a scalar fmaf, at half the instructions
    u64 acc[MT][VEC / 2];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int i = 0; i < VEC / 2; ++i) acc[m][i] = 0ull;
    if (col < H) {
      const char* wp = w + (size_t)col * EB;
      auto fma_row = [&](const unsigned (&v)[LW / 4], int kk) {
        u64 wpair[VEC / 2];  // float32 values of columns (2i, 2i + 1)
#pragma unroll
        for (int i = 0; i < VEC / 2; ++i) wpair[i] = pair_of<T>(v, i);
        unsigned xw[(XROW + 3) / 4];
        load_xrow<XROW>(xs + (size_t)kk * XROW, xw);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < M) {
            const unsigned xb = __float_as_uint(llb::Elem<T>::to_f(llb::elem_get<T>(xw, m)));
            const u64 xx = ((u64)xb << 32) | xb;
#pragma unroll
            for (int i = 0; i < VEC / 2; ++i) fma2(acc[m][i], xx, wpair[i]);
          }
        }
      };
      int kk = k0;
      for (; kk + UNROLL <= k1; kk += UNROLL) {
        unsigned v[UNROLL][LW / 4];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) load_lane<LW>(wp + (size_t)(kk + u) * row_bytes, v[u]);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) fma_row(v[u], kk + u);
      }
      for (; kk < k1; ++kk) {
        unsigned v[LW / 4];
        load_lane<LW>(wp + (size_t)kk * row_bytes, v);
        fma_row(v, kk);
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
      if (m < M)
#pragma unroll
        for (int i = 0; i < VEC / 2; ++i) {
          float* d = &part[((size_t)warp * M + m) * COLS + lane * VEC + 2 * i];
          d[0] = __uint_as_float((unsigned)acc[m][i]);
          d[1] = __uint_as_float((unsigned)(acc[m][i] >> 32));
        }
    __syncthreads();
    // (row, word) pairs of the tile: slices in warp order, round, publish
    for (int p = threadIdx.x; p < M * 32 * WPL; p += blockDim.x) {
      const int m = p / (32 * WPL), j = p % (32 * WPL);  // j: LL word within the tile
      const int wc = t * COLS + j * (8 / EB);
      if (wc >= H) continue;
      float s8[8 / EB];
#pragma unroll
      for (int i = 0; i < 8 / EB; ++i) {
        const size_t o = (size_t)m * COLS + j * (8 / EB) + i;
        s8[i] = part[o];
        for (int q = 1; q < kLinearWarps; ++q) s8[i] = __fadd_rn(s8[i], part[(size_t)q * M * COLS + o]);
      }
      unsigned y2[2] = {0u, 0u};
#pragma unroll
      for (int i = 0; i < 8 / EB; ++i) llb::elem_set<T>(y2, i, llb::Elem<T>::from_f(s8[i]));
      const u64 mine = (u64)y2[0] | ((u64)y2[1] << 32);
      const size_t wid = (size_t)m * words_per_row + wc / (8 / EB);
      if (FUSE) llb::ll_put(b, rank, E, wid, mine);
      else *reinterpret_cast<u64*>(out + wid * 8) = mine;
    }
    __syncthreads();  // part is rewritten by the next tile
  }

  // ---- phase 2 (fused): the AllReduce of every word this CTA published
  if (FUSE) {
    bool ok = true;
    for (int t = cta; t < tiles && ok; t += G)
      for (int p = threadIdx.x; p < M * 32 * WPL; p += blockDim.x) {
        const int m = p / (32 * WPL), j = p % (32 * WPL);
        const int wc = t * COLS + j * (8 / EB);
        if (wc >= H) continue;
        const size_t wid = (size_t)m * words_per_row + wc / (8 / EB);
        u64 d[8];
        llb::ll_try(b, rank, E, wid, d[rank]);  // my own line, written by this thread
        if (!llb::ll_wait_ranks(b, rank, E, wid, d)) {
          ok = false;
          break;
        }
        *reinterpret_cast<u64*>(out + wid * 8) = llb::sum_words_ranks<T>(d, n);
      }
    llb::end(b, 1u, E);
  }
}

// ---------------------------------------------- tensor-core variant (M <= 16)
// For 16-bit types and more than 4 rows the FMA rate bounds the kernel
// above, so the same layer runs on the tensor cores: mma.sync m16n8k16
// (fp16/bf16 operands, float32 accumulators), the rows of x padded to 16.
// Each warp owns 32 output columns over the whole of K (no cross-warp
// reduction): it streams its weight rows with coalesced 16-byte cp.async
// copies into a warp-private ring of kTcStages shared tiles [16 k][32
// columns] (80-byte pitch: the rows of an ldmatrix land in distinct
// banks), from which ldmatrix.trans builds the B fragments; x sits in shared memory as [16 rows][Kp] (Kp = K rounded up
// to 16, pitch 2 Kp + 16 bytes, zero beyond K and beyond M). The
// accumulators become LL words (4 consecutive columns of a row) through
// one shuffle between neighbouring lanes; the epilogue is the LL
// AllReduce as in kb_linear. The tensor cores sum the 16 products of a
// step in an order of their own.
constexpr int kTcWarps = 8;
constexpr int kTcCols = 32 * kTcWarps;  // columns per CTA tile
constexpr int kTcPitch = 80;            // bytes per row of a warp's weight tile
constexpr int kTcTile = 16 * kTcPitch;  // one buffer
constexpr int kTcStages = 6;            // k-steps of weights in flight per warp (cp.async ring)

__device__ __forceinline__ void ldsm_x4(unsigned addr, unsigned (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(unsigned addr, unsigned (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], const unsigned (&a)[4], unsigned b0, unsigned b1) {
  if constexpr (std::is_same<T, __half>::value)
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <typename T, bool FUSE>
__global__ void __launch_bounds__(32 * kTcWarps, 2) kb_linear_tc(const llar_llbuffer b, const LinearArgs a, int G) {
  extern __shared__ __align__(16) unsigned char smem[];
  const u64 E = FUSE ? llb::begin(b) : 0;
  const int n = a.n;
  const int rank = (int)(blockIdx.x % n), cta = (int)(blockIdx.x / n);
  const int M = a.m, K = a.k, H = a.h;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int Kp = (K + 15) & ~15;
  const int xpitch = 2 * Kp + 16;
  unsigned char* xs = smem;                                               // [16][Kp]
  unsigned char* wt = smem + 16 * xpitch + warp * kTcStages * kTcTile;    // my ring
  const unsigned short* x = reinterpret_cast<const unsigned short*>(a.x[rank]);
  const char* w = a.w[rank];
  char* out = a.out[rank];
  if (K % 8 == 0) {  // rows of x start on 16-byte boundaries: 16-byte loads
    const int kv = Kp / 8, rowv = K / 8;
    for (int i = threadIdx.x; i < 16 * kv; i += blockDim.x) {
      const int m = i / kv, j = i % kv;
      const uint4 v = (m < M && j < rowv) ? *reinterpret_cast<const uint4*>(x + (size_t)m * K + (size_t)j * 8)
                                          : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(xs + m * xpitch + j * 16) = v;
    }
  } else {
    for (int i = threadIdx.x; i < 16 * Kp; i += blockDim.x) {
      const int m = i / Kp, kk = i % Kp;
      reinterpret_cast<unsigned short*>(xs + m * xpitch)[kk] = (m < M && kk < K) ? x[(size_t)m * K + kk] : 0;
    }
  }
  __syncthreads();
  const int tiles = (H + kTcCols - 1) / kTcCols;
  const int steps = Kp / 16;
  const size_t row_bytes = (size_t)H * 2;
  const int words_per_row = H / 4;
  const int g = lane >> 2, q = lane & 3;
  // my two 16-byte chunks of a k-step: rows id / 4, column chunks id % 4
  const int id0 = lane, id1 = lane + 32;
  const unsigned wt_s = (unsigned)__cvta_generic_to_shared(wt);
  const unsigned xs_s = (unsigned)__cvta_generic_to_shared(xs);
  // ldmatrix row addresses: A (x) rows (mi & 1) * 8 + l % 8, k half mi >> 1;
  // B (weights) k rows (mi & 1) * 8 + l % 8, column block mi >> 1
  const int mi = lane >> 3, li = lane & 7;
  const unsigned a_row = xs_s + (unsigned)(((mi & 1) * 8 + li) * xpitch + (mi >> 1) * 16);
  const unsigned b_row = (unsigned)(((mi & 1) * 8 + li) * kTcPitch + (mi >> 1) * 16);

  u64 own[4] = {0, 0, 0, 0};  // my published words of my last tile (nb = 0..3)
  for (int t = cta; t < tiles; t += G) {
    const int c0 = t * kTcCols + warp * 32;  // my first column
    // my two 16-byte chunks of k-step st into ring slot st % kTcStages;
    // chunks past K or H are zero-filled (source size 0)
    auto issue = [&](int st) {
      if (st < steps) {
        const unsigned slot = wt_s + (unsigned)((st % kTcStages) * kTcTile);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int id = h2 ? id1 : id0;
          const int row = st * 16 + id / 4, col = c0 + (id % 4) * 8;
          const bool in = row < K && col < H;
          const char* src = in ? w + (size_t)row * row_bytes + (size_t)col * 2 : w;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                       :: "r"(slot + (unsigned)((id / 4) * kTcPitch + (id % 4) * 16)), "l"(src), "r"(in ? 16 : 0)
                       : "memory");
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");  // one group per step, even if empty
    };
    float d[4][4];
#pragma unroll
    for (int nb = 0; nb < 4; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) d[nb][i] = 0.0f;
#pragma unroll
    for (int i = 0; i < kTcStages - 1; ++i) issue(i);
    for (int st = 0; st < steps; ++st) {
      issue(st + kTcStages - 1);
      asm volatile("cp.async.wait_group %0;" :: "n"(kTcStages - 1) : "memory");  // step st is in
      __syncwarp();  // ... for every lane's copies
      unsigned af[4], bf0[4], bf1[4];
      ldsm_x4(a_row + (unsigned)(st * 32), af);
      const unsigned bs = wt_s + (unsigned)((st % kTcStages) * kTcTile);
      ldsm_x4_trans(bs + b_row, bf0);       // column blocks 0, 1
      ldsm_x4_trans(bs + b_row + 32, bf1);  // column blocks 2, 3
      mma16816<T>(d[0], af, bf0[0], bf0[1]);
      mma16816<T>(d[1], af, bf0[2], bf0[3]);
      mma16816<T>(d[2], af, bf1[0], bf1[1]);
      mma16816<T>(d[3], af, bf1[2], bf1[3]);
      __syncwarp();  // every lane has read this slot before it is refilled
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // accumulators -> LL words: lane (g, q) holds columns 2q, 2q + 1 of rows
    // g and g + 8 in each column block; an even q takes its neighbour's pair
    // of row g (4 columns of row g), an odd q gives its row-(g + 8) pair to
    // its neighbour and takes theirs (4 columns of row g + 8)
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      const float o0 = __shfl_xor_sync(0xFFFFFFFFu, (q & 1) ? d[nb][0] : d[nb][2], 1);
      const float o1 = __shfl_xor_sync(0xFFFFFFFFu, (q & 1) ? d[nb][1] : d[nb][3], 1);
      float v[4];
      int row;
      if (!(q & 1)) {
        row = g;
        v[0] = d[nb][0]; v[1] = d[nb][1]; v[2] = o0; v[3] = o1;
      } else {
        row = g + 8;
        v[0] = o0; v[1] = o1; v[2] = d[nb][2]; v[3] = d[nb][3];
      }
      const int col = c0 + nb * 8 + 2 * (q & ~1);
      if (row < M && col < H) {
        unsigned y2[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 4; ++i) llb::elem_set<T>(y2, i, llb::Elem<T>::from_f(v[i]));
        const u64 mine = (u64)y2[0] | ((u64)y2[1] << 32);
        const size_t wid = (size_t)row * words_per_row + col / 4;
        own[nb] = mine;
        if (FUSE) llb::ll_put(b, rank, E, wid, mine);
        else *reinterpret_cast<u64*>(out + wid * 8) = mine;
      }
    }
  }
  if (FUSE) {
    // The LL AllReduce of my words, two per polling round (their 2(N-1)
    // peer lines in flight together). Lanes q and q ^ 1 share rows g and
    // g + 8 of column blocks 0-3: the even lane takes blocks 0, 1 and the
    // odd lane blocks 2, 3 of both rows, so up to 8 rows take one round.
    // My own word comes from registers (mine, or my neighbour's by a
    // shuffle) for my last tile, from my line for earlier ones.
    const bool odd = (q & 1) != 0;
    const int nbA = odd ? 2 : 0;  // my two column blocks nbA, nbA + 1
    u64 nbr[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) nbr[k] = __shfl_xor_sync(0xFFFFFFFFu, own[k], 1);
    const u64 myA = odd ? own[2] : own[0], myB = odd ? own[3] : own[1];
    const u64 nbrA = odd ? nbr[2] : nbr[0], nbrB = odd ? nbr[3] : nbr[1];
    bool ok = true;
    for (int t = cta; t < tiles && ok; t += G) {
      const int c0 = t * kTcCols + warp * 32;
      const bool last = t + G >= tiles;
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // row g, then row g + 8
        const int row = g + 8 * half;
        const bool held = (int)odd == half;  // my lane published this row's words
        size_t wid[2];
        u64 dd[2][8];
        unsigned pend = 0;  // bit 8u + q: word u of rank q not yet in
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int col = c0 + (nbA + u) * 8 + 2 * (q & ~1);
          wid[u] = (size_t)row * words_per_row + col / 4;
          if (row < M && col < H) {
            u64 mine = held ? (u ? myB : myA) : (u ? nbrB : nbrA);
            if (!last) llb::ll_try(b, rank, E, wid[u], mine);  // my rank's line
#pragma unroll
            for (int r2 = 0; r2 < 8; ++r2)  // constant indices: dd stays in registers
              if (r2 == rank) dd[u][r2] = mine;
            pend |= (((1u << n) - 1u) & ~(1u << rank)) << (8 * u);
          }
        }
        const unsigned valid = pend;
        llb::Wait wt;
        while (pend != 0u) {
          u64 lo[16], hi[16];
#pragma unroll
          for (int h2 = 0; h2 < 16; ++h2)
            if ((pend >> h2) & 1u) llb::ld_relaxed_b128(llb::ll_line(b, h2 & 7, E, wid[h2 >> 3]), lo[h2], hi[h2]);
#pragma unroll
          for (int h2 = 0; h2 < 16; ++h2)
            if (((pend >> h2) & 1u) && hi[h2] == E) {
              dd[h2 >> 3][h2 & 7] = lo[h2];
              pend &= ~(1u << h2);
            }
          if (pend != 0u && wt.expired(b)) {
            llb::fail(b, rank, E);
            ok = false;
            break;
          }
        }
        if (!ok) break;
#pragma unroll
        for (int u = 0; u < 2; ++u)
          if ((valid >> (8 * u)) & 0xFFu) *reinterpret_cast<u64*>(out + wid[u] * 8) = llb::sum_words_ranks<T>(dd[u], n);
      }
    }
    llb::end(b, 1u, E);
  }
}

// one bounded wait for one LL word (diagnostic entry point)
__global__ void kb_probe_wait(const llar_llbuffer b, int rank, int src, u64 E, size_t w) {
  if (threadIdx.x == 0) {
    u64 d;
    llb::ll_wait(b, rank, src, E, w, d);
  }
}

// ------------------------------------------------------------- host side
int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return LLAR_OK;
  cudaGetLastError();
  return e == cudaErrorCooperativeLaunchTooLarge ? LLAR_ERR_OCCUPANCY : LLAR_ERR_CUDA;
}

size_t elem_bytes(int dtype) { return dtype == LLAR_F32 ? 4 : 2; }

bool valid(const llar_llbuffer* b) {
  return b && b->nranks >= 2 && b->nranks <= kMaxN && b->ll && b->sen && b->ll128 && b->epoch && b->status_host;
}

// CTAs of `kernel` resident per SM (cached per kernel and shape)
int resident_per_sm(const void* kernel, int threads, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, size_t>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(kernel, threads, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int per = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    per = 0;
  }
  cache[key] = per;
  return per;
}
int sm_count() {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  return sms;
}

// Cooperative (CTAs wait on one another), and a programmatic dependent of
// the previous kernel in the stream: llb::begin() waits for it.
cudaError_t launch_coop(const void* kernel, int blocks, int threads, size_t smem, cudaStream_t s, void** args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelExC(&cfg, kernel, args);
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const char* x = static_cast<const char*>(a);
  const char* y = static_cast<const char*>(b);
  return x < y + nb && y < x + na;
}

// instantiation of KERNEL<..., n, ...> for n = 2..8
#define LLB_PICK_N(INST)                 \
  switch (n) {                           \
    case 2: return (const void*)INST(2); \
    case 3: return (const void*)INST(3); \
    case 4: return (const void*)INST(4); \
    case 5: return (const void*)INST(5); \
    case 6: return (const void*)INST(6); \
    case 7: return (const void*)INST(7); \
    case 8: return (const void*)INST(8); \
  }                                      \
  return nullptr;

template <typename T>
const void* allreduce_kernel(int proto, int n) {
#define LLB_LL(N) kb_ll<T, N>
#define LLB_SEN(N) kb_sentinel<T, N>
#define LLB_L128(N) kb_ll128<T, N>
  if (proto == LLAR_PROTO_LL) { LLB_PICK_N(LLB_LL) }
  if (proto == LLAR_PROTO_SENTINEL) { LLB_PICK_N(LLB_SEN) }
  if (proto == LLAR_PROTO_LL128_ATOMIC) { LLB_PICK_N(LLB_L128) }
  return nullptr;
#undef LLB_LL
#undef LLB_SEN
#undef LLB_L128
}
#undef LLB_PICK_N
// kb_linear instance for the element type, M (rounded up to 1, 2, 4, 8,
// 16; 16-byte lanes up to 4 rows, 8-byte lanes above, to bound registers)
template <typename T, bool FUSE>
const void* linear_kernel(int m) {
  if (m <= 1) return (const void*)kb_linear<T, 1, 16, FUSE>;
  if (m <= 2) return (const void*)kb_linear<T, 2, 16, FUSE>;
  if (m <= 4) return (const void*)kb_linear<T, 4, 16, FUSE>;
  if (m <= 8) return (const void*)kb_linear<T, 8, 16, FUSE>;
  return (const void*)kb_linear<T, 16, 8, FUSE>;
}
template <bool FUSE>
const void* linear_tc_kernel_for(int dtype) {
  return dtype == LLAR_F16 ? (const void*)kb_linear_tc<__half, FUSE> : (const void*)kb_linear_tc<__nv_bfloat16, FUSE>;
}
// shared memory of the tensor-core variant: x [16][Kp] and a warp's ring
size_t linear_tc_smem(int k) {
  const size_t kp = ((size_t)k + 15) & ~size_t(15);
  return 16 * (2 * kp + 16) + (size_t)kTcWarps * kTcStages * kTcTile;
}
template <bool FUSE>
const void* linear_kernel_for(int dtype, int m) {
  if (dtype == LLAR_F32) return linear_kernel<float, FUSE>(m);
  if (dtype == LLAR_F16) return linear_kernel<__half, FUSE>(m);
  return linear_kernel<__nv_bfloat16, FUSE>(m);
}
int linear_lane_bytes(int m) { return m <= 8 ? 16 : 8; }
int linear_rows(int m) { return m <= 1 ? 1 : m <= 2 ? 2 : m <= 4 ? 4 : m <= 8 ? 8 : 16; }

int linear_launch(const llar_llbuffer* b, const void* const* x, const void* const* w, void* const* out, int n,
                  int m, int k, int h, int dtype, bool fuse, void* stream) {
  if (dtype < LLAR_F32 || dtype > LLAR_BF16 || !x || !w || !out) return LLAR_ERR_INVALID;
  if (n < 2 || n > kMaxN || m < 1 || m > kLinearMaxM || k < 1 || h < 8 || h % 8) return LLAR_ERR_INVALID;
  const size_t e = elem_bytes(dtype);
  const size_t xbytes = (size_t)m * k * e, obytes = (size_t)m * h * e, wbytes = (size_t)k * h * e;
  if (xbytes > kLinearMaxXBytes) return LLAR_ERR_TOO_LARGE;
  if (fuse && obytes > b->bytes) return LLAR_ERR_TOO_LARGE;
  for (int r = 0; r < n; ++r) {
    if (!x[r] || !w[r] || !out[r] || (((uintptr_t)x[r] | (uintptr_t)w[r] | (uintptr_t)out[r]) & 15u))
      return LLAR_ERR_INVALID;
    for (int q = 0; q < n; ++q)
      if (overlaps(out[r], obytes, x[q], xbytes) || overlaps(out[r], obytes, w[q], wbytes) ||
          (q != r && overlaps(out[r], obytes, out[q], obytes)))
        return LLAR_ERR_INVALID;
  }
  if (fuse && b->status_host->code != 0) return LLAR_ERR_TIMEOUT;
  LinearArgs a = {};
  for (int r = 0; r < n; ++r) {
    a.x[r] = static_cast<const char*>(x[r]);
    a.w[r] = static_cast<const char*>(w[r]);
    a.out[r] = static_cast<char*>(out[r]);
  }
  a.n = n;
  a.m = m;
  a.k = k;
  a.h = h;
  // 16-bit types with more than 4 rows: the tensor-core variant, when its
  // shared memory fits (measured: the FMA rate bounds the CUDA-core one)
  const bool tc = e == 2 && m > 4 && linear_tc_smem(k) <= (200u << 10) && !std::getenv("LLAR_LINEAR_NO_TC");
  const int cols = tc ? kTcCols : 32 * linear_lane_bytes(m) / (int)e;
  const int tiles = (h + cols - 1) / cols;
  const size_t smem = tc ? linear_tc_smem(k)
                         : (((size_t)k * linear_rows(m) * e + 15) & ~size_t(15)) + (size_t)kLinearWarps * m * cols * 4;
  if (smem > (227u << 10)) return LLAR_ERR_TOO_LARGE;  // not reached within the documented limits
  const void* kern = tc ? (fuse ? linear_tc_kernel_for<true>(dtype) : linear_tc_kernel_for<false>(dtype))
                        : (fuse ? linear_kernel_for<true>(dtype, m) : linear_kernel_for<false>(dtype, m));
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return cuda_status(err);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  llar_llbuffer bb = fuse ? *b : llar_llbuffer{};
  if (!fuse) {
    // one CTA per (rank, tile); no CTA waits on another
    int G = tiles;
    void* args[] = {&bb, &a, &G};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n * tiles);
    cfg.blockDim = dim3(kLinearThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cuda_status(cudaLaunchKernelExC(&cfg, kern, args));
  }
  // fused: CTAs wait on their peers, so all must be resident (cooperative)
  const int per_sm = resident_per_sm(kern, kLinearThreads, smem);
  if (per_sm < 1) return LLAR_ERR_OCCUPANCY;
  int G = std::max(1, std::min(tiles, per_sm * sm_count() / n));
  void* args[] = {&bb, &a, &G};
  return cuda_status(launch_coop(kern, n * G, kLinearThreads, smem, s, args));
}

}  // namespace

extern "C" {

int llar_llbuffer_create(int nranks, size_t bytes, llar_llbuffer* out) {
  if (!out || nranks < 2 || nranks > kMaxN || bytes == 0 || bytes > kMaxBytes) return LLAR_ERR_INVALID;
  llar_llbuffer b = {};
  b.nranks = nranks;
  b.bytes = bytes;
  b.timeout_ns = 1000000000ull;
  if (const char* v = std::getenv("LLAR_TIMEOUT_NS")) {
    const unsigned long long t = std::strtoull(v, nullptr, 10);
    if (t) b.timeout_ns = t;
  }
  auto up = [](size_t v, size_t a) { return (v + a - 1) / a * a; };
  b.ll128_lines = (bytes / nranks + 4) / 124 + 2;
  b.ll_words = std::max((bytes + 7) / 8, (size_t)16 * nranks * b.ll128_lines);
  b.ll_slot_stride = up(b.ll_words * 16, 256);
  b.ll_rank_stride = 2 * b.ll_slot_stride;
  b.sen_vecs = (bytes + 15) / 16;
  b.sen_src_stride = up(b.sen_vecs * 16, 256);
  b.sen_slot_stride = (size_t)nranks * b.sen_src_stride;
  b.sen_rank_stride = 2 * b.sen_slot_stride;
  b.ll128_slot_stride = up(b.ll128_lines * 128, 256);
  b.ll128_rank_stride = 2 * b.ll128_slot_stride;
  const size_t ll_bytes = nranks * b.ll_rank_stride, sen_bytes = nranks * b.sen_rank_stride,
               l128_bytes = nranks * b.ll128_rank_stride, ctl_bytes = 256;
  char* dev = nullptr;
  void* host = nullptr;
  const size_t total = ll_bytes + sen_bytes + l128_bytes + ctl_bytes;
  if (cudaMalloc(&dev, total) != cudaSuccess) {
    cudaGetLastError();
    return LLAR_ERR_CUDA;
  }
  if (cudaHostAlloc(&host, sizeof(llar_llbuffer_status), cudaHostAllocMapped) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(dev);
    return LLAR_ERR_CUDA;
  }
  void* host_dev = nullptr;
  cudaError_t err = cudaHostGetDevicePointer(&host_dev, host, 0);
  // LL lines and control words start at zero (epoch 0 is never used by a
  // kernel: llb::begin returns counter + 1); sentinel vectors all ones
  if (err == cudaSuccess) err = cudaMemset(dev, 0, ll_bytes);
  if (err == cudaSuccess) err = cudaMemset(dev + ll_bytes, 0xFF, sen_bytes);
  if (err == cudaSuccess) err = cudaMemset(dev + ll_bytes + sen_bytes, 0, l128_bytes + ctl_bytes);
  if (err == cudaSuccess) err = cudaDeviceSynchronize();
  if (err != cudaSuccess) {
    cudaGetLastError();
    cudaFreeHost(host);
    cudaFree(dev);
    return LLAR_ERR_CUDA;
  }
  std::memset(host, 0, sizeof(llar_llbuffer_status));
  b.ll = dev;
  b.sen = dev + ll_bytes;
  b.ll128 = dev + ll_bytes + sen_bytes;
  char* ctl = dev + ll_bytes + sen_bytes + l128_bytes;
  b.epoch = reinterpret_cast<unsigned long long*>(ctl);
  b.done_count = reinterpret_cast<unsigned*>(ctl + 64);
  b.abort_word = reinterpret_cast<unsigned*>(ctl + 128);
  b.status = static_cast<llar_llbuffer_status*>(host_dev);
  b.status_host = static_cast<llar_llbuffer_status*>(host);
  *out = b;
  return LLAR_OK;
}

int llar_llbuffer_destroy(llar_llbuffer* b) {
  if (!valid(b)) return LLAR_ERR_INVALID;
  cudaFree(b->ll);
  cudaFreeHost(b->status_host);
  std::memset(b, 0, sizeof(*b));
  return LLAR_OK;
}

int llar_llbuffer_get_status(const llar_llbuffer* b, int* rank, unsigned long long* epoch) {
  if (!valid(b)) return LLAR_ERR_INVALID;
  volatile const llar_llbuffer_status* st = b->status_host;
  const unsigned code = st->code;
  if (rank) *rank = code ? st->rank : -1;
  if (epoch) *epoch = code ? st->epoch : 0ull;
  return code ? (int)code : LLAR_OK;
}

int llar_llbuffer_reset(llar_llbuffer* b, void* stream) {
  if (!valid(b)) return LLAR_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t sen_bytes = (size_t)b->nranks * b->sen_rank_stride;
  const size_t l128_bytes = (size_t)b->nranks * b->ll128_rank_stride;
  cudaError_t err = cudaMemsetAsync(b->sen, 0xFF, sen_bytes, s);
  if (err == cudaSuccess) err = cudaMemsetAsync(b->ll128, 0, l128_bytes, s);
  if (err == cudaSuccess) err = cudaMemsetAsync(b->done_count, 0, sizeof(unsigned), s);
  if (err == cudaSuccess) err = cudaMemsetAsync(b->abort_word, 0, sizeof(unsigned), s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  if (err != cudaSuccess) return cuda_status(err);
  std::memset(b->status_host, 0, sizeof(llar_llbuffer_status));
  return LLAR_OK;
}

int llar_llbuffer_set_timeout_ns(llar_llbuffer* b, unsigned long long ns) {
  if (!valid(b) || ns == 0) return LLAR_ERR_INVALID;
  b->timeout_ns = ns;
  return LLAR_OK;
}

int llar_llbuffer_epoch(const llar_llbuffer* b, unsigned long long* epoch) {
  if (!valid(b) || !epoch) return LLAR_ERR_INVALID;
  cudaError_t err = cudaDeviceSynchronize();
  if (err == cudaSuccess) err = cudaMemcpy(epoch, b->epoch, sizeof(*epoch), cudaMemcpyDeviceToHost);
  return cuda_status(err);
}

int llar_llbuffer_probe_wait(const llar_llbuffer* b, int rank, int src, unsigned long long epoch, size_t word,
                             void* stream) {
  if (!valid(b) || rank < 0 || rank >= b->nranks || src < 0 || src >= b->nranks || word >= b->ll_words)
    return LLAR_ERR_INVALID;
  kb_probe_wait<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(*b, rank, src, epoch, word);
  return cuda_status(cudaGetLastError());
}

int llar_llbuffer_allreduce(const llar_llbuffer* b, const void* const* in, void* const* out, size_t count,
                            int dtype, int protocol, int iters, void* stream) {
  if (!valid(b) || !in || !out || iters < 1) return LLAR_ERR_INVALID;
  if (dtype < LLAR_F32 || dtype > LLAR_BF16) return LLAR_ERR_INVALID;
  if (protocol != LLAR_PROTO_LL && protocol != LLAR_PROTO_SENTINEL && protocol != LLAR_PROTO_LL128_ATOMIC)
    return LLAR_ERR_UNSUPPORTED;
  const int n = b->nranks;
  const size_t e = elem_bytes(dtype);
  if (count > b->bytes / e) return LLAR_ERR_TOO_LARGE;
  const size_t nbytes = count * e;
  Ptrs io = {};
  for (int r = 0; r < n; ++r) {
    if (!in[r] || !out[r] || (((uintptr_t)in[r] | (uintptr_t)out[r]) & 15u)) return LLAR_ERR_INVALID;
    for (int q = 0; q < n; ++q)
      if (overlaps(out[r], nbytes, in[q], nbytes) || (q != r && overlaps(out[r], nbytes, out[q], nbytes)))
        return LLAR_ERR_INVALID;
    io.in[r] = static_cast<const char*>(in[r]);
    io.out[r] = static_cast<char*>(out[r]);
  }
  if (b->status_host->code != 0) return LLAR_ERR_TIMEOUT;
  if (count == 0) return LLAR_OK;
  const void* kern = dtype == LLAR_F32   ? allreduce_kernel<float>(protocol, n)
                     : dtype == LLAR_F16 ? allreduce_kernel<__half>(protocol, n)
                                         : allreduce_kernel<__nv_bfloat16>(protocol, n);
  // units per CTA: LL 8-byte words, sentinel 16-byte vectors, LL128 lines
  // (8 lanes x N segments per line); threads and CTAs per rank as the
  // library's own kernels of the same protocol pick them
  size_t units;
  int threads;
  if (protocol == LLAR_PROTO_LL) {
    units = (nbytes + 7) / 8;
    threads = 128;
  } else if (protocol == LLAR_PROTO_SENTINEL) {
    units = (nbytes + 15) / 16;
    threads = 64;
  } else {
    const size_t P = 128 / e - 1;
    units = ((count + n - 1) / n + P - 1) / P * 8 * n;
    threads = 256;
  }
  const int per_sm = resident_per_sm(kern, threads, 0);
  if (per_sm < 1) return LLAR_ERR_OCCUPANCY;
  const size_t max_g = (size_t)per_sm * sm_count() / n;
  size_t G = std::min(max_g, std::max<size_t>(1, (units + threads - 1) / threads));
  if (protocol == LLAR_PROTO_LL128_ATOMIC) G = std::min(G, std::max<size_t>(1, units / (8 * n)));
  if (G < 1) return LLAR_ERR_OCCUPANCY;
  llar_llbuffer bb = *b;
  int Gi = (int)G;
  size_t arg3 = protocol == LLAR_PROTO_LL128_ATOMIC ? count : nbytes;
  void* args[] = {&bb, &io, &arg3, &iters, &Gi};
  return cuda_status(launch_coop(kern, n * Gi, threads, 0, static_cast<cudaStream_t>(stream), args));
}

int llar_fused_linear_allreduce(const llar_llbuffer* b, const void* const* x, const void* const* w,
                                void* const* out, int m, int k, int h, int dtype, void* stream) {
  if (!valid(b)) return LLAR_ERR_INVALID;
  return linear_launch(b, x, w, out, b->nranks, m, k, h, dtype, true, stream);
}

int llar_linear_partials(const void* const* x, const void* const* w, void* const* p, int nranks, int m, int k,
                         int h, int dtype, void* stream) {
  return linear_launch(nullptr, x, w, p, nranks, m, k, h, dtype, false, stream);
}

}  // extern "C"
