// Host runtime of the C ABI declared in include/llar.h: the process-global
// context, staging layout and initialisation, argument checks, launch-shape
// choice, epochs, status word, and the speed-of-light probe.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "llar.h"
#include "llar_internal.h"

namespace {

using llar::Params;

constexpr size_t kAlign = 256;
constexpr size_t kDefaultLLCap = 1u << 20;      // LL messages up to 1 MiB per rank
constexpr size_t kDefaultLL128Cap = 64u << 20;  // LL128 messages up to 64 MiB per rank
constexpr size_t kMaxLL128Cap = size_t(1) << 30;  // the LL128 kernels index a CTA's items in 32 bits
constexpr size_t kMaxHostRegs = 64;               // registered host buffers per context
constexpr size_t kDefaultChunk = 64u << 10;     // sentinel chunk per rank: every chunk costs a round trip and a fence
constexpr size_t kMaxChunk = 64u << 10;         // largest sentinel chunk
constexpr int kFlagsGmax = 1024;                // CTAs per rank the chain flags can address
constexpr int kLLTuneMinIters = 16;             // LL launches the calibrated placement applies to

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
size_t elem_bytes(int dtype) { return dtype == LLAR_F32 ? 4 : 2; }

size_t env_size(const char* name, size_t dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  return (size_t)std::strtoull(v, nullptr, 0);
}

struct Ctx {
  int n = 0, dtype = 0, dev = 0, sms = 0;
  size_t max_bytes = 0, esize = 0;
  size_t ll_cap = 0, ll128_cap = 0, chunk_bytes = kDefaultChunk;
  char* base = nullptr;
  size_t total = 0;
  // regions
  size_t ll_off = 0, ll_stride = 0, ll_words = 0;
  size_t sen_off = 0, sen_stride = 0;
  size_t l128_off = 0, l128_stride = 0, l128_lines = 0;
  size_t ag_off = 0, ag_stride = 0;
  size_t l128d_off = 0, l128d_stride = 0;  // [3 slots][lines][128 B] of LLAR_PROTO_LL128_DIRECT
  size_t chain_off = 0, chain_stride = 0, chain_slot = 0;
  size_t flags_off = 0, abort_off = 0;
  llar::DevStatus* status_host = nullptr;
  llar::DevStatus* status_dev = nullptr;
  // host-API staging
  char* io = nullptr;
  size_t io_stride = 0;
  // host buffers registered by the caller: host range -> device address
  struct HostReg {
    const char* host;
    size_t bytes;
    char* dev;
  };
  std::vector<HostReg> host_regs;
  // resident-CTA capacity per (protocol, chain, threads, clustered): the
  // occupancy queries cost microseconds, so each is made once
  std::map<long long, int> capacity;
  // LL launches of many AllReduces in clusters of N blocks (chosen by
  // calibrate_ll on this GPU)
  int auto_atomic = 0;      // AUTO may take the (nondeterministic) LL128 direct form
  int ll_cluster = 0;       // LL launches of many AllReduces up to ll_cal_bytes run in clusters
  size_t ll_cal_bytes = 0;  // bytes per rank the placement was timed at
};

std::mutex g_mu;
Ctx* g = nullptr;
unsigned long long g_timeout_ns = 1000000000ull;
int g_force_G = 0, g_force_T = 0;
int g_cluster = 1, g_log = 0, g_bulk = 1, g_spread = 0, g_pdl = 1;  // LLAR_PDL=0: plain stream order
// LLAR_COOP=0: waiting kernels launch without the cooperative attribute.
// Measured on a B300 (8 x 16 KiB bf16 LL, one AllReduce per call, calls
// queued back to back from C): 4.0 -> 2.5 us of host time and 5.0 -> 3.1 us
// of GPU time per call; from Python 8.5 -> 7.7 us (host-bound); replayed
// from a CUDA graph no gain (2.50 -> 2.65 us), so the cooperative launch
// stays the default. The grid is still sized by the same residency check
// (it fits the GPU at once), but nothing holds the launch back while other
// kernels occupy SMs: rank CTAs that start then wait for the rest, and a
// wait that outlasts the timeout fails with LLAR_ERR_TIMEOUT. For callers
// whose library launches overlap no other kernels.
int g_no_coop = 0;
size_t g_bulk_min_bytes = 0;  // LLAR_BULK_MIN_BYTES: TMA two-shot threshold for every N (0: per N)
int g_inject_rank = -1, g_inject_mode = 0;
int g_last_proto = 0, g_last_G = 0, g_last_T = 0, g_last_iters = 0;
int g_last_clustered = 0, g_last_spread = 0;  // of the last AllReduce launch

// no error recorded; cta -1 until a wait that records its CTA runs out
void clear_status(llar::DevStatus* st) {
  std::memset(st, 0, sizeof(*st));
  st->cta = -1;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return LLAR_OK;
  if (e == cudaErrorCooperativeLaunchTooLarge) return LLAR_ERR_OCCUPANCY;
  return LLAR_ERR_CUDA;
}

// Chunk-sized slots per rank region the sentinel one-shot keeps all-ones
// between launches: the publish-once ring, or two slots per peer on the
// push path (forced launch shapes); the publish-once tail words follow at
// kSenPubSlots * kSenMaxChunkBytes.
size_t sen_slots(int n) { return std::max<size_t>(llar::kSenPubSlots, 2 * (size_t)n); }
size_t sen_region_bytes(int n) {
  static_assert(llar::kSenMaxChunkBytes == kMaxChunk, "one largest chunk");
  return std::max<size_t>(llar::kSenPubSlots, 2 * (size_t)n) * kMaxChunk + (kMaxChunk / 16) * 8;
}

size_t ll128_payload(int dtype) { return 128 / elem_bytes(dtype) - 1; }
size_t ll128_lines_for(size_t count, int n, int dtype) {
  const size_t seg = (count + n - 1) / n;
  const size_t pl = ll128_payload(dtype);
  return (seg + pl - 1) / pl;
}

bool valid_dtype(int d) { return d == LLAR_F32 || d == LLAR_F16 || d == LLAR_BF16; }
bool valid_proto(int p) { return p >= LLAR_PROTO_AUTO && p <= LLAR_PROTO_LL128_DIRECT; }
// the two-shot LL128 atomic protocols: the pages' LL AllGather, or reads from the owners' lines
bool is_ll128(int p) { return p == LLAR_PROTO_LL128_ATOMIC || p == LLAR_PROTO_LL128_DIRECT; }

// AUTO for AllReduces back to back in one launch, per rank count.
// Measured on a B300 (bf16, 2 KiB .. 4 MiB per rank): LL is fastest up to
// ll_max, the direct-read one-shot up to oneshot_max, the direct-read
// two-shot above, streamed through shared memory with TMA bulk copies
// from bulk_min (with 6 or more ranks already from 32 KiB: 3.3 us against
// 3.5-6.2 us for the other paths at 64 KiB). bulk_min holds for every call.
struct AutoRule {
  size_t ll_max, oneshot_max, bulk_min;
};
AutoRule auto_rule(int n) {
  constexpr size_t K = 1024, M = 1024 * 1024, kNever = ~size_t(0);
  switch (n) {
    case 2: return {256 * K, 1 * M, kNever};
    case 3: return {128 * K, 1 * M, 1 * M};
    case 4: return {128 * K, 512 * K, 1 * M};
    case 5: return {64 * K, 256 * K, 512 * K};
    default: return {32 * K, 32 * K, 32 * K};
  }
}
// AUTO for one AllReduce per launch (llar_allreduce), per rank count.
// Measured on a B300 (bf16, graph-replayed single calls, 8 KiB .. 2 MiB
// per rank), with the fixed-order paths' single-call shape (one vector a
// thread): a single call pays the cooperative launch and the epoch
// exchange of LL, which the direct-read one-shot (no co-residency, nothing
// signalled) does not, so the one-shot wins small messages with 2, 3, 5
// and 6 ranks (2 x 16 KiB: 2.22 against 2.47 us; 6 x 16 KiB: 2.71 against
// 2.91), while LL keeps them with 4 ranks (up to 64 KiB, by ~0.1 us) and
// 7-8 ranks (8 x 16 KiB: 2.59 against 2.96, up to 32 KiB); the two-shot
// takes over from 512 KiB (4 ranks), 256 KiB (5), 128 KiB (6), 64 KiB
// (7-8) and above 1 MiB (2-3).
AutoRule auto_rule_single(int n) {
  constexpr size_t K = 1024, M = 1024 * 1024;
  const size_t bulk = auto_rule(n).bulk_min;
  switch (n) {
    case 2: return {0, 1 * M, bulk};
    case 3: return {0, 1 * M, bulk};
    case 4: return {64 * K, 256 * K, bulk};
    case 5: return {0, 128 * K, bulk};
    case 6: return {0, 64 * K, bulk};
    default: return {32 * K, 32 * K, bulk};
  }
}
size_t bulk_min_bytes(int n) {
  return g_bulk_min_bytes ? g_bulk_min_bytes : auto_rule(n).bulk_min;
}

int forced_protocol() {
  const char* force = std::getenv("LLAR_PROTO");
  if (force && *force) {
    const int f = std::atoi(force);
    if (f >= LLAR_PROTO_LL && f <= LLAR_PROTO_LL128_DIRECT) return f;
  }
  return LLAR_PROTO_AUTO;
}

int select_by(const AutoRule& rule, size_t bytes) {
  if (bytes <= rule.ll_max) return LLAR_PROTO_LL;
  if (bytes <= rule.oneshot_max) return LLAR_PROTO_FIXED_ONESHOT;
  return LLAR_PROTO_FIXED_TWOSHOT;
}
// one AllReduce per launch
int select_protocol(int n, int dtype, size_t count) {
  if (const int f = forced_protocol()) return f;
  return select_by(auto_rule_single(n), count * elem_bytes(dtype));
}

// AUTO for a persistent launch of `iters` > 1 AllReduces. Measured on a
// B300 (bf16, 2/4/8 ranks, 16 KiB .. 1 MiB per rank, us per AllReduce):
// * chains (each input = scale x the previous output): LL is the fastest
//   deterministic path nearly everywhere, by far (8 x 64 KiB: 1.41 against
//   11.7 for the two-shot, whose chained form pays two flag rounds per
//   step), except 7-8 ranks at 1 MiB (8 ranks: two-shot 13.3 against LL
//   19.9). The LL128 direct form is faster still at 8 ranks from 256 KiB
//   (4.2 against 5.6) but its atomic sums are not bit-reproducible, so
//   AUTO leaves it to the caller;
// * independent AllReduces back to back: auto_rule, except that LL stays
//   ahead up to 64 KiB with 6-8 ranks (8 x 64 KiB: 1.22 against 1.67).
// LL only up to the context's LL capacity (ll_cap).
// With `atomic` (llar_set_auto_nondeterministic), chains also take the LL128
// direct form where it measured fastest of all (bf16 and fp32): 5-8 ranks
// at 512 KiB, 8 ranks from 256 KiB, 5-6 ranks above 512 KiB (5 x 1 MiB
// bf16: 9.6 against LL 12.5); 7-8 ranks above 512 KiB keep the two-shot.
int select_protocol_iters(int n, int dtype, size_t count, int iters, bool chain, size_t ll_cap,
                          bool atomic = false, size_t ll128_cap = kDefaultLL128Cap) {
  if (const int f = forced_protocol()) return f;
  const size_t bytes = count * elem_bytes(dtype);
  constexpr size_t K = 1024;
  if (atomic && iters > 1 && chain && n >= 5 && bytes <= ll128_cap &&
      (bytes >= 512 * K || (n == 8 && bytes >= 256 * K)) && (n <= 6 || bytes <= 512 * K))
    return LLAR_PROTO_LL128_DIRECT;
  if (iters > 1 && chain && bytes <= ll_cap && (n <= 6 || bytes <= (512u << 10))) return LLAR_PROTO_LL;
  if (iters > 1 && chain) return LLAR_PROTO_FIXED_TWOSHOT;
  if (iters > 1 && n >= 6 && bytes <= std::min<size_t>(ll_cap, 64u << 10)) return LLAR_PROTO_LL;
  if (iters > 1) return select_by(auto_rule(n), bytes);
  return select_protocol(n, dtype, count);
}

// AUTO when the inputs and outputs are host memory that the kernel reads
// and writes across the bus (the host-buffer entry's direct path). The bus
// sets the cost there, and every path moves the same bytes across it; what
// differs is how many reads are in flight and when the writes start.
// Measured on a B300 (bf16, pinned registered buffers, 2..8 ranks, 64 B ..
// 1 MiB per rank): LL answers a single call ~1 us sooner up to a few KiB
// per rank (13.0-13.3 against 14.0-14.2 us, idle GPU); from 16 KiB the
// direct-read two-shot is fastest or within a few percent (8 x 16 KiB:
// 7.1-7.4 us back to back against 8.3-10.1 for LL; 4 x 1 MiB: 128 us
// against 170), except 8 ranks from 256 KiB, where a sentinel launch with
// 16 KiB chunks is ~10-25 % faster (the chunk is the caller's setting, so
// AUTO does not take it).
int select_protocol_host(int n, int dtype, size_t count) {
  if (const int f = forced_protocol()) return f;
  (void)n;
  return count * elem_bytes(dtype) <= 4096 ? LLAR_PROTO_LL : LLAR_PROTO_FIXED_TWOSHOT;
}

// CTAs per rank and threads per CTA for one launch.
// `single`: one AllReduce per launch (llar_allreduce), not a persistent loop.
void choose_shape(const Ctx& c, int proto, size_t count, int chain, int* G, int* T, bool single = false) {
  const int n = c.n;
  const size_t e = c.esize;
  const int one_per_sm = std::max(1, c.sms / n);
  size_t units = 0;  // independent work items per rank
  int t = 128;
  switch (proto) {
    case LLAR_PROTO_LL: units = (count * e + 7) / 8; break;
    case LLAR_PROTO_SENTINEL: units = std::min(c.chunk_bytes, round_up(count * e, 16)) / 16; break;
    case LLAR_PROTO_LL128_ATOMIC:
    case LLAR_PROTO_LL128_DIRECT: units = ll128_lines_for(count, n, c.dtype) * n * llar::kLL128Lanes; break;
    default: units = (count * e + 15) / 16; break;
  }
  int g = 1;
  if (proto == LLAR_PROTO_FIXED_TWOSHOT || proto == LLAR_PROTO_FIXED_ONESHOT) {
    t = 256;
    const bool two = proto == LLAR_PROTO_FIXED_TWOSHOT;
    const size_t per_rank = two ? (units + n - 1) / n : units;
    // A single call is latency-bound up to mid sizes: one vector a thread
    // in CTAs of 128 threads. Measured, one call per launch (graph replay,
    // bf16): one-shot 4 x 64 KiB 3.07 -> 2.55 us, 8 x 16 KiB 4.14 -> 3.03;
    // two-shot (without TMA) 4 x 256 KiB 3.93 -> 3.05. Not where the
    // one-shot's N reads of the message grow large (8 x 256 KiB: 4.71 ->
    // 6.06, slower) or a two-shot segment passes 512 KiB (not measured).
    if (single && !chain && (two ? per_rank <= 32768 : per_rank * (size_t)n <= 65536)) {
      t = 128;
      g = (int)std::min<size_t>(std::max<size_t>((per_rank + t - 1) / t, 1),
                                (size_t)std::max(1, (c.sms * 8) / n));
    } else {
      const size_t want = (per_rank + 2 * t - 1) / (2 * t);
      const int cap = chain ? one_per_sm : std::max(1, (c.sms * 4) / n);
      g = (int)std::min<size_t>(std::max<size_t>(want, 1), (size_t)cap);
    }
  } else if (proto == LLAR_PROTO_SENTINEL) {
    // every vector costs N-1 pushes, polls and resets plus a fence per
    // chunk: spread the chunk thinly over as many SMs as possible (measured,
    // 8 ranks x 2 KiB: 2 CTAs of 64 threads per rank 4.1 us, 16 of 32
    // threads 2.9 us)
    t = units <= 512 ? 32 : 64;
    const size_t want = std::max<size_t>((units + t - 1) / t, 16);
    g = (int)std::min<size_t>(want, (size_t)std::max(1, 2 * c.sms / n));
    if (want > (size_t)g) t = (int)std::min<size_t>(llar::kMaxThreads, round_up((units + g - 1) / g, 32));
  } else if (is_ll128(proto) && units > (size_t)one_per_sm * llar::kMaxThreads) {
    // more (segment, line, lane) items than one CTA of 512 threads per SM
    // covers: as many resident CTAs of 256 threads as fit (the capacity
    // check clamps G); 8 ranks x 1 MiB bf16, one call: 23.1 -> 20.9 us
    t = 256;
    g = (int)std::max<size_t>(1, (units + t - 1) / t);
  } else {
    const size_t want = (units + t - 1) / t;
    if (want <= (size_t)one_per_sm) {
      g = (int)std::max<size_t>(want, 1);
    } else {
      g = one_per_sm;
      const size_t per_cta = (units + g - 1) / g;
      t = (int)std::min<size_t>(llar::kMaxThreads, round_up(per_cta, 32));
    }
    if (is_ll128(proto)) {
      // a CTA takes whole lines, ceil(L / g) of every segment: threads for
      // all of its items in one pass (8 ranks x 128 KiB bf16 chain: 480
      // threads left 32 of 512 items for a second pass, 5.17 us per layer;
      // 512 threads 4.18 us)
      const size_t lines = units / ((size_t)n * llar::kLL128Lanes);
      const size_t items = (lines + g - 1) / g * (size_t)n * llar::kLL128Lanes;
      t = (int)std::min<size_t>(llar::kMaxThreads, round_up(items, 32));
    }
  }
  if (g_force_G > 0) g = g_force_G;
  if (g_force_T > 0) t = g_force_T;
  g = std::min(g, kFlagsGmax);
  *G = g;
  *T = t;
}

// Pointers non-null and 16-byte aligned; no output overlaps an input or
// another output. Spans are per rank, in bytes.
int check_ptrs_spans(const void* const* in, void* const* out, int n, const size_t* in_span,
                     const size_t* out_span) {
  if (!in || !out) return LLAR_ERR_INVALID;
  for (int r = 0; r < n; ++r) {
    if (!in[r] || !out[r]) return LLAR_ERR_INVALID;
    if (((uintptr_t)in[r] | (uintptr_t)out[r]) & 15u) return LLAR_ERR_INVALID;
  }
  for (int r = 0; r < n; ++r) {
    const uintptr_t o0 = (uintptr_t)out[r], o1 = o0 + out_span[r];
    for (int q = 0; q < n; ++q) {
      const uintptr_t i0 = (uintptr_t)in[q], i1 = i0 + in_span[q];
      if (o0 < i1 && i0 < o1) return LLAR_ERR_INVALID;  // output overlaps an input
      if (q != r) {
        const uintptr_t p0 = (uintptr_t)out[q], p1 = p0 + out_span[q];
        if (o0 < p1 && p0 < o1) return LLAR_ERR_INVALID;  // two outputs overlap
      }
    }
  }
  return LLAR_OK;
}
int check_ptrs(const void* const* in, void* const* out, int n, size_t in_span, size_t out_span) {
  size_t is[llar::kMaxRanks], os[llar::kMaxRanks];
  for (int r = 0; r < n; ++r) {
    is[r] = in_span;
    os[r] = out_span;
  }
  return check_ptrs_spans(in, out, n, is, os);
}

// Pointers, sizes, staging bases, status and injection settings shared by
// every launch of the context.
void fill_params(Ctx& c, Params& p, const void* const* in, void* const* out, size_t count) {
  std::memset(&p, 0, sizeof(p));
  for (int r = 0; r < c.n; ++r) {
    p.in[r] = static_cast<const char*>(in[r]);
    p.out[r] = static_cast<char*>(out[r]);
  }
  p.count = count;
  p.nranks = c.n;
  p.iters = 1;
  p.epoch_dev = reinterpret_cast<unsigned long long*>(c.base + c.abort_off + 128);
  p.done_count = reinterpret_cast<unsigned*>(c.base + c.abort_off + 64);
  p.ll = c.base + c.ll_off;
  p.ll_stride = c.ll_stride;
  p.ll_slot_words = c.ll_words;
  p.sen = c.base + c.sen_off;
  p.sen_stride = c.sen_stride;
  p.sen_chunk_vecs = (int)(c.chunk_bytes / 16);
  p.l128 = c.base + c.l128_off;
  p.l128_stride = c.l128_stride;
  p.l128ag = c.base + c.ag_off;
  p.l128ag_stride = c.ag_stride;
  p.l128_lines = c.l128_lines;
  p.l128d = c.base + c.l128d_off;
  p.l128d_stride = c.l128d_stride;
  p.l128d_seq = reinterpret_cast<unsigned long long*>(c.base + c.abort_off + 192);
  p.chainbuf = c.base + c.chain_off;
  p.chain_stride = c.chain_stride;
  p.chain_slot_bytes = c.chain_slot;
  p.flags = reinterpret_cast<unsigned long long*>(c.base + c.flags_off);
  p.flags_gmax = kFlagsGmax;
  p.timeout_ns = g_timeout_ns;
  p.inject_rank = g_inject_rank;
  p.inject_mode = g_inject_mode;
  p.abort_flag = reinterpret_cast<unsigned*>(c.base + c.abort_off);
  p.status = c.status_dev;
  p.pdl = g_pdl;
  p.no_coop = g_no_coop;
}

// AUTO for the standalone halves. Measured on a B300 (bf16, one call per
// launch replayed from a graph, 2..8 ranks, 1 KiB .. 64 MiB per rank,
// segments of whole 16-byte vectors and ragged ones): the direct copies are
// the fastest at every point, ReduceScatter (8 x 16 KiB: 1.7 us against
// 4.0 for LL and 3.8 for LL128) and AllGather (8 x 16 KiB: 1.6 against 2.7
// for LL; ragged segments, 7 ranks x 16 KiB: 1.5 against 2.8).
int select_segment_protocol(bool rs, int n, size_t count, size_t e) {
  (void)rs;
  (void)n;
  (void)count;
  (void)e;
  if (const int f = forced_protocol()) return f;
  return LLAR_PROTO_FIXED_ONESHOT;
}

// ReduceScatter (rs) or AllGather over segments of a count-element vector.
int run_segment(bool rs, const void* const* in, void* const* out, size_t count, int proto, cudaStream_t stream) {
  if (!g) return LLAR_ERR_NOT_INIT;
  Ctx& c = *g;
  const size_t e = c.esize;
  const size_t bytes = count * e;
  const size_t seg_bytes = (count + c.n - 1) / c.n * e;
  if (proto == LLAR_PROTO_AUTO) proto = select_segment_protocol(rs, c.n, count, e);
  // AllGather adds nothing, so the atomic LL128 protocol has no AllGather
  // of its own (its second half is LL)
  const bool ok_proto = proto == LLAR_PROTO_LL || proto == LLAR_PROTO_FIXED_ONESHOT ||
                        proto == LLAR_PROTO_SENTINEL || (rs && proto == LLAR_PROTO_LL128_ATOMIC);
  if (!ok_proto) return LLAR_ERR_UNSUPPORTED;
  if (bytes > c.max_bytes) return LLAR_ERR_TOO_LARGE;
  if (proto == LLAR_PROTO_LL && bytes > c.ll_cap) return LLAR_ERR_TOO_LARGE;
  if (proto == LLAR_PROTO_LL128_ATOMIC && bytes > c.ll128_cap) return LLAR_ERR_TOO_LARGE;
  // the sentinel variants move every segment in one chunk
  if (proto == LLAR_PROTO_SENTINEL && round_up(seg_bytes, 16) > c.chunk_bytes) return LLAR_ERR_TOO_LARGE;
  size_t full[llar::kMaxRanks], seg[llar::kMaxRanks];
  for (int r = 0; r < c.n; ++r) {
    const size_t per = (count + c.n - 1) / c.n;
    const size_t lo = std::min(count, (size_t)r * per), hi = std::min(count, lo + per);
    full[r] = bytes;
    seg[r] = (hi - lo) * e;
  }
  const int st = check_ptrs_spans(in, out, c.n, rs ? full : seg, rs ? seg : full);
  if (st != LLAR_OK) return st;
  if (c.status_host->code != 0) return LLAR_ERR_TIMEOUT;
  if (count == 0) return LLAR_OK;
  Params p;
  fill_params(c, p, in, out, count);
  int which;
  switch (proto) {
    case LLAR_PROTO_LL: which = rs ? 0 : 1; break;
    case LLAR_PROTO_LL128_ATOMIC: which = 4; break;
    case LLAR_PROTO_SENTINEL: which = rs ? 5 : 6; break;
    default: which = rs ? 2 : 3; break;
  }
  int T = proto == LLAR_PROTO_LL ? 128 : 256;
  bool two_per_sm = false;
  size_t units;
  if (proto == LLAR_PROTO_LL) {
    const size_t words = (bytes + 7) / 8, seg_words = (seg_bytes + 7) / 8;
    units = rs ? std::max(words, seg_words) : seg_words * c.n;
  } else if (proto == LLAR_PROTO_LL128_ATOMIC) {
    units = ll128_lines_for(count, c.n, c.dtype) * c.n * llar::kLL128Lanes;  // (segment, line, lane) items
  } else if (proto == LLAR_PROTO_SENTINEL) {
    units = round_up(seg_bytes, 16) / 16;  // one thread per vector of a segment, thin CTAs
    T = units <= 512 ? 32 : 64;
  } else if (seg_bytes % 16 == 0 && rs && bytes > llar::kRsVectorMinBytes) {
    // segments of whole 16-byte vectors: one vector per thread in 128-thread
    // CTAs while the grid holds them (the single-call shape of the fixed
    // AllReduce); beyond that 512-thread CTAs that loop, two per SM over all
    // ranks. Measured on a B300 (bf16, 2..8 ranks, 256 KiB .. 64 MiB per
    // rank, CTAs of 32..512 threads, 1..4 vectors a thread): 8 x 4 MiB took
    // 4.8 us against 6.0 with four CTAs per SM
    units = seg_bytes / 16;
    T = units <= (size_t)128 * (4 * c.sms / c.n) ? 128 : 512;
    two_per_sm = T == 512;
  } else if (seg_bytes % 16 == 0 && !rs) {
    // the AllGather's owners store every vector N times: threads over all
    // ranks up to 512 per SM (up to 8 MiB per rank) or 512 x 8 / N per SM
    // (larger), in 128-thread CTAs up to 8192 a rank, 256-thread ones
    // beyond. Measured on a B300 (bf16, 2..8 ranks, 1 KiB .. 64 MiB per
    // rank, 1..592 CTAs of 128..512 threads): the fastest shapes at each
    // point had about these thread counts (8 x 64 MiB: 102 us with 64 x 128
    // threads a rank, 109 with 74 x 512)
    const size_t per_sm = bytes <= (8u << 20) ? 512 : 4096 / c.n;
    units = std::min<size_t>(seg_bytes / 16, std::max<size_t>(1, per_sm * c.sms / c.n));
    T = units <= 8192 ? 128 : 256;
  } else {
    // one element per thread (ReduceScatter: small or ragged segments;
    // AllGather: ragged ones, each element stored N times by its owner)
    units = seg_bytes / e;
  }
  int G = (int)std::max<size_t>(1, (units + T - 1) / T);
  if (proto == LLAR_PROTO_SENTINEL) G = std::max(G, 16);
  const bool waits = proto != LLAR_PROTO_FIXED_ONESHOT;
  int cap = waits || two_per_sm ? llar::max_resident_segment_ctas(which, c.dtype, c.n, T) : 4 * c.sms;
  if (two_per_sm) cap = std::min(cap, 2 * c.sms);
  if (cap <= 0) return LLAR_ERR_CUDA;
  G = std::min(G, std::max(1, cap / c.n));
  if (g_force_G > 0) G = g_force_G;
  if (g_force_T > 0) T = g_force_T;
  p.G = G;
  const cudaError_t err = llar::launch_segment(which, c.dtype, p, T, stream);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return cuda_status(err);
  }
  g_last_proto = proto;
  g_last_G = G;
  g_last_T = T;
  g_last_iters = 1;
  return LLAR_OK;
}

// Point-to-point transfers: rank r sends to dst[r] (-1: nothing).
int run_p2p(const void* const* send, void* const* recv, const int* dst, size_t count, int proto, int iters,
            size_t send_stride, size_t recv_stride, cudaStream_t stream) {
  if (!g) return LLAR_ERR_NOT_INIT;
  Ctx& c = *g;
  if (!send || !recv || !dst || iters < 1) return LLAR_ERR_INVALID;
  const size_t e = c.esize;
  const size_t bytes = count * e;
  if ((send_stride * e) % 16 || (recv_stride * e) % 16) return LLAR_ERR_INVALID;
  int src[llar::kMaxRanks];
  for (int r = 0; r < c.n; ++r) src[r] = -1;
  for (int r = 0; r < c.n; ++r) {
    const int d = dst[r];
    if (d < -1 || d >= c.n || d == r) return LLAR_ERR_INVALID;
    if (d >= 0) {
      if (src[d] >= 0) return LLAR_ERR_INVALID;  // a rank receives from one sender at most
      src[d] = r;
    }
  }
  // AUTO: the direct copy. Measured on a B300 (bf16, a pair and an 8-rank
  // ring, 512 B .. 8 MiB, one call per launch replayed from a graph / 50 per
  // launch): it is ahead of LL and the sentinel at every size (512 B: 1.46
  // against LL 2.20 us a call; 1 MiB: 2.0 against 4.2; 8 MiB: 5.2 against the
  // sentinel's 231), since stream order already makes the sender's buffer
  // ready and nothing has to be signalled between the virtual ranks
  if (proto == LLAR_PROTO_AUTO) proto = LLAR_PROTO_FIXED_ONESHOT;
  if (proto != LLAR_PROTO_LL && proto != LLAR_PROTO_SENTINEL && proto != LLAR_PROTO_FIXED_ONESHOT)
    return LLAR_ERR_UNSUPPORTED;
  if (bytes > c.max_bytes) return LLAR_ERR_TOO_LARGE;
  if (proto == LLAR_PROTO_LL && bytes > c.ll_cap) return LLAR_ERR_TOO_LARGE;
  // participating buffers: 16-byte aligned, no receive span overlapping a
  // send span or another receive span
  const size_t sspan = (size_t)(iters - 1) * send_stride * e + bytes;
  const size_t rspan = (size_t)(iters - 1) * recv_stride * e + bytes;
  for (int r = 0; r < c.n; ++r) {
    if (dst[r] >= 0 && (!send[r] || ((uintptr_t)send[r] & 15u))) return LLAR_ERR_INVALID;
    if (src[r] >= 0 && (!recv[r] || ((uintptr_t)recv[r] & 15u))) return LLAR_ERR_INVALID;
  }
  for (int r = 0; r < c.n; ++r) {
    if (src[r] < 0) continue;
    const uintptr_t o0 = (uintptr_t)recv[r], o1 = o0 + rspan;
    for (int q = 0; q < c.n; ++q) {
      if (dst[q] >= 0) {
        const uintptr_t i0 = (uintptr_t)send[q], i1 = i0 + sspan;
        if (o0 < i1 && i0 < o1) return LLAR_ERR_INVALID;
      }
      if (q != r && src[q] >= 0) {
        const uintptr_t p0 = (uintptr_t)recv[q], p1 = p0 + rspan;
        if (o0 < p1 && p0 < o1) return LLAR_ERR_INVALID;
      }
    }
  }
  if (c.status_host->code != 0) return LLAR_ERR_TIMEOUT;
  if (count == 0) return LLAR_OK;
  Params p;
  const void* ins[llar::kMaxRanks];
  void* outs[llar::kMaxRanks];
  for (int r = 0; r < c.n; ++r) {
    ins[r] = dst[r] >= 0 ? send[r] : nullptr;
    outs[r] = src[r] >= 0 ? recv[r] : nullptr;
  }
  fill_params(c, p, ins, outs, count);
  for (int r = 0; r < c.n; ++r) {
    p.peer_dst[r] = dst[r];
    p.peer_src[r] = src[r];
  }
  p.iters = iters;
  p.in_stride = send_stride;
  p.out_stride = recv_stride;
  // units of CTA work: LL 8-byte words; sentinel 16-byte vectors of a chunk;
  // the direct copy 16-byte vectors, two a thread, up to four CTAs an SM
  int T;
  size_t units;
  if (proto == LLAR_PROTO_LL) {
    T = 128;
    units = (bytes + 7) / 8;
  } else if (proto == LLAR_PROTO_FIXED_ONESHOT) {
    T = 256;
    units = (bytes + 15) / 16;
  } else {
    T = 64;
    units = std::min(c.chunk_bytes, round_up(bytes, 16)) / 16;
  }
  int G = (int)std::max<size_t>(1, (units + T - 1) / T);
  if (proto == LLAR_PROTO_FIXED_ONESHOT)
    G = (int)std::min<size_t>(std::max<size_t>(1, (units + 2 * T - 1) / (2 * T)), std::max(1, 4 * c.sms / c.n));
  if (proto != LLAR_PROTO_FIXED_ONESHOT) {  // CTAs that wait on one another must all be resident
    const int cap = llar::max_resident_p2p_ctas(proto, c.dtype, T);
    if (cap <= 0) return LLAR_ERR_CUDA;
    G = std::min(G, std::max(1, cap / c.n));
    if (g_force_G > 0) G = g_force_G;
    if (g_force_T > 0) T = g_force_T;
    if (G * c.n > cap) return LLAR_ERR_OCCUPANCY;
  } else {
    if (g_force_G > 0) G = g_force_G;
    if (g_force_T > 0) T = g_force_T;
  }
  G = std::min(G, kFlagsGmax);
  p.G = G;
  const cudaError_t err = llar::launch_p2p(proto, c.dtype, p, T, stream);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return cuda_status(err);
  }
  g_last_proto = proto;
  g_last_G = G;
  g_last_T = T;
  g_last_iters = iters;
  return LLAR_OK;
}

int run(const void* const* in, void* const* out, size_t count, int proto, int iters,
        size_t in_stride, size_t out_stride, float chain_scale, cudaStream_t stream) {
  if (!g) return LLAR_ERR_NOT_INIT;
  Ctx& c = *g;
  if (!valid_proto(proto) || iters < 1) return LLAR_ERR_INVALID;
  const size_t e = c.esize;
  const int chain = chain_scale != 0.0f;
  if (chain) in_stride = 0;
  if ((in_stride * e) % 16 || (out_stride * e) % 16) return LLAR_ERR_INVALID;
  const size_t bytes = count * e;
  const size_t in_span = (size_t)(iters - 1) * in_stride * e + bytes;
  const size_t out_span = (size_t)(iters - 1) * out_stride * e + bytes;
  if (proto == LLAR_PROTO_AUTO)
    proto = select_protocol_iters(c.n, c.dtype, count, iters, chain, c.ll_cap, c.auto_atomic != 0, c.ll128_cap);
  if (bytes > c.max_bytes) return LLAR_ERR_TOO_LARGE;
  if (proto == LLAR_PROTO_LL && bytes > c.ll_cap) return LLAR_ERR_TOO_LARGE;
  if (is_ll128(proto) && bytes > c.ll128_cap) return LLAR_ERR_TOO_LARGE;
  int st = check_ptrs(in, out, c.n, in_span, out_span);
  if (st != LLAR_OK) return st;
  if (c.status_host->code != 0) return LLAR_ERR_TIMEOUT;
  if (count == 0) return LLAR_OK;

  Params p;
  fill_params(c, p, in, out, count);
  p.iters = iters;
  p.chain = chain;
  p.chain_scale = chain_scale;
  p.in_stride = in_stride;
  p.out_stride = out_stride;

  int G = 1, T = 128;
  choose_shape(c, proto, count, chain, &G, &T, iters == 1);
  const bool coop = proto == LLAR_PROTO_LL || proto == LLAR_PROTO_SENTINEL ||
                    is_ll128(proto) || chain;
  // Thread-block clusters put the N CTAs that serve one range on one GPC.
  // Measured on B300 (8 ranks, bf16, CTAs per rank as chosen above): they
  // help the sentinel protocol (64 KiB in 8 KiB chunks: 18.0 -> 15.1 us)
  // and the chained fixed-order paths (two-shot, 128 KiB: 16.3 -> 14.9 us),
  // and hurt LL (16 KiB: 0.79 -> 0.87 us) and LL128 (1 MiB: 21 -> 31 us).
  // LLAR_CLUSTER: 0 never, 1 per protocol (default), 2 always.
  const bool cluster_helps = proto == LLAR_PROTO_SENTINEL || proto == LLAR_PROTO_FIXED_ONESHOT ||
                             proto == LLAR_PROTO_FIXED_TWOSHOT ||
                             (proto == LLAR_PROTO_LL && c.ll_cluster && iters >= kLLTuneMinIters &&
                              count * e <= c.ll_cal_bytes);
  p.clustered = (coop && (g_cluster == 2 || (g_cluster == 1 && cluster_helps))) ? 1 : 0;
  p.spread_smem = (coop && (proto == LLAR_PROTO_LL || proto == LLAR_PROTO_SENTINEL)) ? g_spread : 0;
  if (coop) {
    auto capacity = [&](bool clustered) {
      const long long key = ((long long)proto * 2 + chain) * 4096 * 2 + (long long)T * 2 + (clustered ? 1 : 0);
      auto it = c.capacity.find(key);
      if (it != c.capacity.end()) return it->second;
      const int v = llar::max_resident_ctas(proto, c.dtype, c.n, T, clustered, p.spread_smem);
      c.capacity[key] = v;
      return v;
    };
    int cap = capacity(p.clustered != 0);
    if (cap <= 0 && p.clustered) {
      p.clustered = 0;
      cap = capacity(false);
    }
    if (cap <= 0) return LLAR_ERR_CUDA;
    if (c.n * G > cap) {
      if (g_force_G > 0) return LLAR_ERR_OCCUPANCY;
      G = std::max(1, cap / c.n);
    }
  }
  p.G = G;
  if (g_log)
    std::fprintf(stderr, "llar: protocol %d, %d ranks x %d CTAs x %d threads, clustered %d, iters %d, count %zu\n",
                 proto, c.n, G, T, p.clustered, iters, count);
  cudaError_t err;
  switch (proto) {
    case LLAR_PROTO_LL: err = llar::launch_ll(c.dtype, p, T, stream); break;
    case LLAR_PROTO_SENTINEL: err = llar::launch_sentinel(c.dtype, p, T, stream); break;
    case LLAR_PROTO_LL128_ATOMIC: err = llar::launch_ll128(c.dtype, p, T, stream); break;
    case LLAR_PROTO_LL128_DIRECT: err = llar::launch_ll128d(c.dtype, p, T, stream); break;
    case LLAR_PROTO_FIXED_ONESHOT: err = llar::launch_fixed_oneshot(c.dtype, p, T, stream); break;
    default:
      if (!chain && g_bulk && bytes >= bulk_min_bytes(c.n) && g_force_G == 0) {
        // as many CTAs as the ring's shared memory lets each SM hold
        const int per_sm = std::max(1, (int)((227u << 10) / llar::bulk_smem_bytes(c.n)));
        p.G = std::max(1, per_sm * c.sms / c.n);
        T = (int)std::min<size_t>(llar::kMaxThreads, std::max<size_t>(128, llar::bulk_tile_vectors()));
        G = p.G;
        err = llar::launch_fixed_twoshot_bulk(c.dtype, p, T, stream);
      } else {
        err = llar::launch_fixed_twoshot(c.dtype, p, T, stream);
      }
      break;
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return cuda_status(err);
  }
  g_last_proto = proto;
  g_last_G = G;
  g_last_T = T;
  g_last_iters = iters;
  g_last_clustered = p.clustered;
  g_last_spread = p.spread_smem;
  return LLAR_OK;
}

int fill_staging(Ctx& c, cudaStream_t s) {
  cudaError_t err = cudaSuccess;
  auto ok = [&](cudaError_t x) { if (err == cudaSuccess) err = x; };
  ok(cudaMemsetAsync(c.base + c.ll_off, 0, c.ll_stride * c.n, s));
  ok(cudaMemsetAsync(c.base + c.sen_off, 0xFF, c.sen_stride * c.n, s));
  ok(cudaMemsetAsync(c.base + c.l128_off, 0, c.l128_stride * c.n, s));
  ok(cudaMemsetAsync(c.base + c.ag_off, 0, c.ag_stride * c.n, s));
  ok(cudaMemsetAsync(c.base + c.l128d_off, 0, c.l128d_stride * c.n, s));
  ok(cudaMemsetAsync(c.base + c.abort_off + 192, 0, 16, s));  // direct LL128 sequence and last line count
  ok(cudaMemsetAsync(c.base + c.flags_off, 0, (size_t)c.n * kFlagsGmax * llar::kFlagKinds * 8, s));
  // abort word only: the epoch counter at +128 keeps counting across resets
  ok(cudaMemsetAsync(c.base + c.abort_off, 0, 4, s));
  ok(cudaStreamSynchronize(s));
  clear_status(c.status_host);
  return cuda_status(err);
}

}  // namespace

// LL placement. Launched in clusters of N blocks, the N CTAs that exchange
// each word range sit on one GPC; whether that is faster depends on the
// GPU. Measured on B300s, 8 ranks x 16 KiB bf16 back to back: without
// clusters 0.65 us per AllReduce on some GPUs and 0.84-0.85 on others,
// with clusters 0.72-0.73 on both (dependent chains 0.81 / 0.97 against
// 0.93). llar_init times both here, on this GPU (300 AllReduces of up to
// 16 KiB per rank, twice each), and keeps clusters for LL launches of
// many AllReduces no larger than that if they are at least 3 % faster
// (larger messages stay unclustered: 4 ranks x 128 KiB bf16 chained took
// 1.60 us per AllReduce in clusters against 1.21 without, on a GPU where
// 16 KiB ran faster in them). LLAR_TUNE=0 skips it;
// LLAR_CLUSTER (0 or 2) forces either way. Results are identical either
// way (the sums are fixed-order); only the timing differs.
static void calibrate_ll(Ctx& c) {
  c.ll_cluster = 0;
  // injected faults would time the injection (or wait out its timeouts)
  if (env_size("LLAR_TUNE", 1) == 0 || g_cluster != 1 || g_inject_mode != LLAR_INJECT_NONE) return;
  const size_t bytes = std::min<size_t>(std::min(c.max_bytes, c.ll_cap), 16u << 10) / 16 * 16;
  const size_t count = bytes / c.esize;
  if (count == 0) return;
  c.ll_cal_bytes = bytes;
  char* buf = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaStream_t st = nullptr;  // a stream of its own: no implicit wait on the caller's other streams
  if (cudaMalloc(&buf, 2 * (size_t)c.n * bytes) != cudaSuccess || cudaMemset(buf, 0, 2 * (size_t)c.n * bytes) != cudaSuccess ||
      cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess ||
      cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    if (buf) cudaFree(buf);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (st) cudaStreamDestroy(st);
    return;
  }
  const void* in[llar::kMaxRanks];
  void* out[llar::kMaxRanks];
  for (int r = 0; r < c.n; ++r) {
    in[r] = buf + (size_t)r * bytes;
    out[r] = buf + (size_t)(c.n + r) * bytes;
  }
  float best[2] = {1e30f, 1e30f};
  bool ok = true;
  for (int rep = 0; rep < 3 && ok; ++rep) {
    for (int pref = 0; pref < 2 && ok; ++pref) {
      c.ll_cluster = pref;
      ok = cudaEventRecord(e0, st) == cudaSuccess &&
           run(in, out, count, LLAR_PROTO_LL, 300, 0, 0, 0.0f, st) == LLAR_OK &&
           cudaEventRecord(e1, st) == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess;
      float ms = 0.f;
      if (ok && rep > 0 && cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess) best[pref] = std::min(best[pref], ms);
    }
  }
  cudaGetLastError();
  c.ll_cluster = (ok && c.status_host->code == 0 && best[1] < 0.97f * best[0]) ? 1 : 0;
  if (g_log)
    std::fprintf(stderr, "llar: LL placement %s (%.3f ms unclustered, %.3f ms clustered, 300 AllReduces)\n",
                 c.ll_cluster ? "clustered" : "unclustered", best[0], best[1]);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaStreamDestroy(st);
  cudaFree(buf);
  if (c.status_host->code != 0) fill_staging(c, 0);  // a wait ran out: start the context clean
}

namespace llar {
void fault_settings(unsigned long long* timeout_ns, int* inject_rank, int* inject_mode) {
  std::lock_guard<std::mutex> lk(g_mu);
  *timeout_ns = g_timeout_ns;
  *inject_rank = g_inject_rank;
  *inject_mode = g_inject_mode;
}
}  // namespace llar

extern "C" {

int llar_init(int nranks, int dtype, size_t max_bytes) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g) return LLAR_ERR_INVALID;
  // the last-launch record belongs to the context
  g_last_proto = g_last_G = g_last_T = g_last_iters = g_last_clustered = g_last_spread = 0;
  if (nranks < 2 || nranks > llar::kMaxRanks || !valid_dtype(dtype) || max_bytes == 0)
    return LLAR_ERR_INVALID;
  Ctx* c = new Ctx();
  c->n = nranks;
  c->dtype = dtype;
  c->esize = elem_bytes(dtype);
  c->max_bytes = round_up(max_bytes, 16);
  c->ll_cap = std::min(c->max_bytes, round_up(env_size("LLAR_LL_MAX_BYTES", kDefaultLLCap), 16));
  c->ll128_cap = std::min(c->max_bytes,
                           std::min(kMaxLL128Cap, round_up(env_size("LLAR_LL128_MAX_BYTES", kDefaultLL128Cap), 16)));
  c->chunk_bytes = round_up(std::min(env_size("LLAR_CHUNK_BYTES", kDefaultChunk), kMaxChunk), 16);
  g_timeout_ns = env_size("LLAR_TIMEOUT_NS", g_timeout_ns);
  // tuning knobs: each context takes the environment as it is at its
  // llar_init (an unset variable means the built-in default)
  g_force_G = (int)env_size("LLAR_CTAS_PER_RANK", 0);
  g_force_T = (int)env_size("LLAR_THREADS", 0);
  // the same limits as llar_set_launch: whole warps, at most the kernels' bound
  if (g_force_G < 0 || g_force_G > kFlagsGmax) g_force_G = 0;
  if (g_force_T < 0 || g_force_T % 32 || g_force_T > llar::kMaxThreads) g_force_T = 0;
  g_cluster = (int)env_size("LLAR_CLUSTER", 1);
  g_log = (int)env_size("LLAR_LOG", 0);
  g_bulk = (int)env_size("LLAR_BULK", 1);
  g_pdl = (int)env_size("LLAR_PDL", 1);
  g_no_coop = env_size("LLAR_COOP", 1) == 0 ? 1 : 0;
  g_bulk_min_bytes = env_size("LLAR_BULK_MIN_BYTES", 0);
  g_spread = (int)env_size("LLAR_SPREAD_SMEM", 0);

  cudaError_t err = cudaGetDevice(&c->dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&c->sms, cudaDevAttrMultiProcessorCount, c->dev);
  if (err != cudaSuccess) {
    cudaGetLastError();
    delete c;
    return LLAR_ERR_CUDA;
  }
  const int n = nranks;
  size_t off = 0;
  auto region = [&](size_t per_rank, size_t* o, size_t* stride) {
    *stride = round_up(std::max<size_t>(per_rank, 16), kAlign);
    *o = off;
    off += *stride * n;
  };
  c->ll_words = (c->ll_cap + 7) / 8;
  region(2 * c->ll_words * llar::kLLLine, &c->ll_off, &c->ll_stride);  // [slot][word] published lines
  region(sen_region_bytes(n), &c->sen_off, &c->sen_stride);
  c->l128_lines = ll128_lines_for(c->ll128_cap / c->esize, n, dtype);
  region(2 * c->l128_lines * llar::kLL128Line, &c->l128_off, &c->l128_stride);
  region(2 * c->l128_lines * llar::kAgLineBytes, &c->ag_off, &c->ag_stride);
  region(3 * c->l128_lines * llar::kLL128Line, &c->l128d_off, &c->l128d_stride);
  c->chain_slot = round_up(c->max_bytes, kAlign);
  region(2 * c->chain_slot, &c->chain_off, &c->chain_stride);
  c->flags_off = off;
  off += round_up((size_t)n * kFlagsGmax * llar::kFlagKinds * 8, kAlign);
  c->abort_off = off;
  off += kAlign;
  c->total = off;
  err = cudaMalloc(&c->base, c->total);
  if (err == cudaSuccess) err = cudaHostAlloc(&c->status_host, sizeof(llar::DevStatus), cudaHostAllocMapped);
  if (err == cudaSuccess) err = cudaHostGetDevicePointer((void**)&c->status_dev, c->status_host, 0);
  if (err != cudaSuccess) {
    cudaGetLastError();
    if (c->base) cudaFree(c->base);
    if (c->status_host) cudaFreeHost(c->status_host);
    delete c;
    return LLAR_ERR_CUDA;
  }
  if (cudaMemset(c->base + c->abort_off, 0, kAlign) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(c->base);
    cudaFreeHost(c->status_host);
    delete c;
    return LLAR_ERR_CUDA;
  }
  const int st = fill_staging(*c, 0);
  if (st != LLAR_OK) {
    cudaFree(c->base);
    cudaFreeHost(c->status_host);
    delete c;
    return st;
  }
  g = c;
  calibrate_ll(*c);
  g_last_proto = g_last_G = g_last_T = g_last_iters = g_last_clustered = g_last_spread = 0;  // the user's launches only
  return LLAR_OK;
}

int llar_destroy(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g) return LLAR_ERR_NOT_INIT;
  cudaError_t err = cudaDeviceSynchronize();
  cudaFree(g->base);
  if (g->io) cudaFree(g->io);
  cudaFreeHost(g->status_host);
  delete g;
  g = nullptr;
  return cuda_status(err);
}

int llar_allreduce(const void* const* in, void* const* out, size_t count, int protocol, void* stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  return run(in, out, count, protocol, 1, 0, 0, 0.0f, static_cast<cudaStream_t>(stream));
}

int llar_allreduce_iters(const void* const* in, void* const* out, size_t count, int protocol, int iters,
                         size_t in_stride_elems, size_t out_stride_elems, float chain_scale, void* stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  return run(in, out, count, protocol, iters, in_stride_elems, out_stride_elems, chain_scale,
             static_cast<cudaStream_t>(stream));
}

int llar_reduce_scatter(const void* const* in, void* const* out, size_t count, int protocol, void* stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  return run_segment(true, in, out, count, protocol, static_cast<cudaStream_t>(stream));
}

int llar_all_gather(const void* const* in, void* const* out, size_t count, int protocol, void* stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  return run_segment(false, in, out, count, protocol, static_cast<cudaStream_t>(stream));
}

int llar_sendrecv(const void* const* send, void* const* recv, const int* dst, size_t count, int protocol, int iters,
                  size_t send_stride, size_t recv_stride, void* stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  return run_p2p(send, recv, dst, count, protocol, iters, send_stride, recv_stride,
                 static_cast<cudaStream_t>(stream));
}

int llar_allreduce_host(const void* in_host, void* out_host, size_t count, int protocol, void* stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g) return LLAR_ERR_NOT_INIT;
  if (!in_host || !out_host) return LLAR_ERR_INVALID;
  Ctx& c = *g;
  const size_t bytes = count * c.esize;
  if (bytes > c.max_bytes) return LLAR_ERR_TOO_LARGE;
  if (c.status_host->code != 0) return LLAR_ERR_TIMEOUT;
  if (count == 0) return LLAR_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Pinned host buffers that the device can address (page-locked memory
  // under unified addressing): the kernel reads the inputs and writes the
  // outputs across the bus itself, one launch and no staging copies.
  // Measured against one DMA each way (or DMA in, zero-copy out), this is
  // the fastest of the three for the small messages this entry serves.
  if (bytes % 16 == 0) {
    // registered buffers: device addresses without per-call queries
    auto registered = [&](const void* p, size_t len) -> char* {
      const uintptr_t q = (uintptr_t)p;
      for (const auto& h : c.host_regs) {
        const uintptr_t h0 = (uintptr_t)h.host;
        if (q >= h0 && len <= h.bytes && q - h0 <= h.bytes - len) return h.dev + (q - h0);
      }
      return nullptr;
    };
    const int proto = protocol == LLAR_PROTO_AUTO ? select_protocol_host(c.n, c.dtype, count) : protocol;
    char* rin = registered(in_host, bytes * c.n);
    char* rout = registered(out_host, bytes * c.n);
    if (rin && rout && ((((uintptr_t)rin) | ((uintptr_t)rout)) & 15u) == 0) {
      const void* ins[llar::kMaxRanks];
      void* outs[llar::kMaxRanks];
      for (int r = 0; r < c.n; ++r) {
        ins[r] = rin + r * bytes;
        outs[r] = rout + r * bytes;
      }
      return run(ins, outs, count, proto, 1, 0, 0, 0.0f, s);
    }
    cudaPointerAttributes ai, ao;
    if (cudaPointerGetAttributes(&ai, in_host) == cudaSuccess && cudaPointerGetAttributes(&ao, out_host) == cudaSuccess &&
        ai.type == cudaMemoryTypeHost && ao.type == cudaMemoryTypeHost && ai.devicePointer && ao.devicePointer &&
        ((((uintptr_t)ai.devicePointer) | ((uintptr_t)ao.devicePointer)) & 15u) == 0) {
      const void* ins[llar::kMaxRanks];
      void* outs[llar::kMaxRanks];
      for (int r = 0; r < c.n; ++r) {
        ins[r] = static_cast<const char*>(ai.devicePointer) + r * bytes;
        outs[r] = static_cast<char*>(ao.devicePointer) + r * bytes;
      }
      return run(ins, outs, count, proto, 1, 0, 0, 0.0f, s);
    }
    cudaGetLastError();  // pageable memory: not an error, take the copy path
  }
  if (!c.io) {
    c.io_stride = round_up(c.max_bytes, kAlign);
    if (cudaMalloc(&c.io, 2 * c.io_stride * c.n) != cudaSuccess) {
      cudaGetLastError();
      c.io = nullptr;
      return LLAR_ERR_CUDA;
    }
  }
  char* din = c.io;
  char* dout = c.io + c.io_stride * c.n;
  const bool rows16 = bytes % 16 == 0;
  // Rows that are 16-byte multiples go in one 1-D copy each way (contiguous
  // staging rows keep every rank's pointer 16-byte aligned).
  const size_t dstride = rows16 ? bytes : c.io_stride;
  cudaError_t err = rows16 ? cudaMemcpyAsync(din, in_host, bytes * c.n, cudaMemcpyHostToDevice, s)
                           : cudaMemcpy2DAsync(din, c.io_stride, in_host, bytes, bytes, c.n, cudaMemcpyHostToDevice, s);
  if (err != cudaSuccess) return cuda_status(err);
  const void* ins[llar::kMaxRanks];
  void* outs[llar::kMaxRanks];
  for (int r = 0; r < c.n; ++r) {
    ins[r] = din + r * dstride;
    outs[r] = dout + r * dstride;
  }
  const int st = run(ins, outs, count, protocol, 1, 0, 0, 0.0f, s);
  if (st != LLAR_OK) return st;
  err = rows16 ? cudaMemcpyAsync(out_host, dout, bytes * c.n, cudaMemcpyDeviceToHost, s)
               : cudaMemcpy2DAsync(out_host, bytes, dout, c.io_stride, bytes, c.n, cudaMemcpyDeviceToHost, s);
  return cuda_status(err);
}

int llar_host_register(const void* ptr, size_t bytes) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g) return LLAR_ERR_NOT_INIT;
  if (!ptr || bytes == 0) return LLAR_ERR_INVALID;
  Ctx& c = *g;
  if (c.host_regs.size() >= kMaxHostRegs) return LLAR_ERR_INVALID;
  const uintptr_t q = (uintptr_t)ptr;
  for (const auto& h : c.host_regs)
    if (q < (uintptr_t)h.host + h.bytes && (uintptr_t)h.host < q + bytes) return LLAR_ERR_INVALID;  // overlap
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess || a.type != cudaMemoryTypeHost || !a.devicePointer) {
    cudaGetLastError();
    return LLAR_ERR_INVALID;  // not page-locked memory the device can address
  }
  c.host_regs.push_back({static_cast<const char*>(ptr), bytes, static_cast<char*>(a.devicePointer)});
  return LLAR_OK;
}

int llar_host_unregister(const void* ptr) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g) return LLAR_ERR_NOT_INIT;
  auto& regs = g->host_regs;
  for (size_t i = 0; i < regs.size(); ++i)
    if (regs[i].host == static_cast<const char*>(ptr)) {
      regs.erase(regs.begin() + (long)i);
      return LLAR_OK;
    }
  return LLAR_ERR_INVALID;
}

int llar_get_status(int* rank, int* cta, unsigned long long* epoch) {
  if (!g) return LLAR_ERR_NOT_INIT;
  volatile llar::DevStatus* st = g->status_host;
  const unsigned code = st->code;
  if (rank) *rank = code ? st->rank : -1;
  if (cta) *cta = code ? st->cta : -1;
  if (epoch) *epoch = code ? st->epoch : 0ull;
  return (int)code;
}

int llar_reset(void* stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g) return LLAR_ERR_NOT_INIT;
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return cuda_status(err);
  return fill_staging(*g, static_cast<cudaStream_t>(stream));
}

void llar_set_timeout_ns(unsigned long long ns) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_timeout_ns = ns ? ns : 1;
}

int llar_set_launch(int ctas_per_rank, int threads) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (ctas_per_rank < 0 || ctas_per_rank > kFlagsGmax) return LLAR_ERR_INVALID;
  if (threads < 0 || threads > llar::kMaxThreads || threads % 32) return LLAR_ERR_INVALID;
  g_force_G = ctas_per_rank;
  g_force_T = threads;
  return LLAR_OK;
}

int llar_set_sentinel_chunk(size_t bytes) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g) return LLAR_ERR_NOT_INIT;
  if (bytes == 0 || bytes % 16 || bytes > kMaxChunk) return LLAR_ERR_INVALID;
  g->chunk_bytes = bytes;
  return LLAR_OK;
}

int llar_debug_inject(int rank, int mode) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (mode < LLAR_INJECT_NONE || mode > LLAR_INJECT_DELAY) return LLAR_ERR_INVALID;
  if (mode != LLAR_INJECT_NONE && (rank < 0 || rank >= llar::kMaxRanks)) return LLAR_ERR_INVALID;
  g_inject_rank = mode == LLAR_INJECT_NONE ? -1 : rank;
  g_inject_mode = mode;
  return LLAR_OK;
}

int llar_sol_probe_detail(double* chase_ns, int* chase_smid, int* nchase, double* rt_ns, int* smid_a,
                          int* smid_b, int* npairs) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g) return LLAR_ERR_NOT_INIT;
  std::vector<llar::SolResult> res(1);
  cudaError_t err = llar::run_sol(res.data(), g_timeout_ns);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return cuda_status(err);
  }
  const llar::SolResult& r = res[0];
  for (int i = 0; i < r.nchase; ++i) {
    if (chase_ns) chase_ns[i] = r.chase_ns[i];
    if (chase_smid) chase_smid[i] = r.chase_smid[i];
  }
  for (int i = 0; i < r.npairs; ++i) {
    if (rt_ns) rt_ns[i] = r.rt_ns[i];
    if (smid_a) smid_a[i] = r.smid_a[i];
    if (smid_b) smid_b[i] = r.smid_b[i];
  }
  if (nchase) *nchase = r.nchase;
  if (npairs) *npairs = r.npairs;
  for (int i = 0; i < r.npairs; ++i)
    if (r.rt_ns[i] <= 0.0) return LLAR_ERR_TIMEOUT;  // that pair's wait ran out
  return LLAR_OK;
}

static double median(std::vector<double> v) {
  if (v.empty()) return 0.0;
  std::sort(v.begin(), v.end());
  const size_t m = v.size() / 2;
  return v.size() % 2 ? v[m] : 0.5 * (v[m - 1] + v[m]);
}

double llar_sol_bound_us(double l2_rt_us, double write_us) { return 2.0 * l2_rt_us + write_us; }

int llar_sol_probe(double* l2_rt_us, double* write_us, double* sol_us) {
  std::vector<double> chase(llar::kSolMaxBlocks), rt(llar::kSolMaxBlocks / 2);
  int nchase = 0, npairs = 0;
  const int st = llar_sol_probe_detail(chase.data(), nullptr, &nchase, rt.data(), nullptr, nullptr, &npairs);
  if (st != LLAR_OK) return st;
  chase.resize(nchase);
  std::vector<double> ok;
  for (int i = 0; i < npairs; ++i)
    if (rt[i] > 0) ok.push_back(rt[i]);
  if (ok.empty() || chase.empty()) return LLAR_ERR_TIMEOUT;
  const double l2 = median(chase) * 1e-3;
  const double wr = 0.5 * median(ok) * 1e-3;
  if (l2_rt_us) *l2_rt_us = l2;
  if (write_us) *write_us = wr;
  if (sol_us) *sol_us = llar_sol_bound_us(l2, wr);
  return LLAR_OK;
}

int llar_ll_placement(int* clustered) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g) return LLAR_ERR_NOT_INIT;
  if (clustered) *clustered = (g_cluster == 2 || (g_cluster == 1 && g->ll_cluster)) ? 1 : 0;
  return LLAR_OK;
}

int llar_sol_probe_placed(double* l2_rt_us, double* write_us, double* sol_us, int* npairs) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g) return LLAR_ERR_NOT_INIT;
  if (g_last_G <= 0 || g_last_T <= 0) return LLAR_ERR_INVALID;  // no AllReduce launched yet
  llar::SolPlaced res;
  const cudaError_t err = llar::run_sol_placed(g->n, g_last_G, g_last_T, g_last_clustered, g_last_spread,
                                               g_timeout_ns, &res);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return cuda_status(err);
  }
  if (res.npairs == 0 || res.chase_worst_ns <= 0.0) return LLAR_ERR_TIMEOUT;
  const double l2 = res.chase_worst_ns * 1e-3;
  const double wr = 0.5 * res.rt_worst_ns * 1e-3;
  if (l2_rt_us) *l2_rt_us = l2;
  if (write_us) *write_us = wr;
  if (sol_us) *sol_us = llar_sol_bound_us(l2, wr);
  if (npairs) *npairs = res.npairs;
  return LLAR_OK;
}

int llar_staging(int protocol, void** dev_ptr, size_t* rank_stride_bytes, size_t* rank_bytes) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g) return LLAR_ERR_NOT_INIT;
  const Ctx& c = *g;
  size_t off = 0, stride = 0, used = 0;
  switch (protocol) {
    case LLAR_PROTO_LL: off = c.ll_off; stride = c.ll_stride; used = 2 * c.ll_words * llar::kLLLine; break;
    case LLAR_PROTO_SENTINEL: off = c.sen_off; stride = c.sen_stride; used = sen_slots(c.n) * c.chunk_bytes; break;
    case LLAR_PROTO_LL128_ATOMIC: off = c.l128_off; stride = c.l128_stride; used = 2 * c.l128_lines * llar::kLL128Line; break;
    case LLAR_PROTO_LL128_DIRECT: off = c.l128d_off; stride = c.l128d_stride; used = 3 * c.l128_lines * llar::kLL128Line; break;
    default: return LLAR_ERR_UNSUPPORTED;
  }
  if (dev_ptr) *dev_ptr = c.base + off;
  if (rank_stride_bytes) *rank_stride_bytes = stride;
  if (rank_bytes) *rank_bytes = used;
  return LLAR_OK;
}

int llar_layout(int protocol, int dtype, int nranks, size_t count, size_t* line_bytes,
                size_t* payload_elems_per_line, size_t* staging_bytes_per_rank) {
  if (!valid_dtype(dtype) || nranks < 2 || nranks > llar::kMaxRanks || !valid_proto(protocol))
    return LLAR_ERR_INVALID;
  if (protocol == LLAR_PROTO_AUTO) protocol = select_protocol(nranks, dtype, count);
  const size_t e = elem_bytes(dtype);
  size_t lb = 16, pl = 16 / e, st = 0;
  switch (protocol) {
    case LLAR_PROTO_LL:
      pl = 8 / e;
      st = 2 * ((count * e + 7) / 8) * llar::kLLLine;  // two slots of the rank's published lines
      break;
    case LLAR_PROTO_SENTINEL: {
      const size_t chunk = g ? g->chunk_bytes : kDefaultChunk;
      // the publish-once ring of kSenPubSlots chunks and a tail word per vector
      st = nranks >= llar::kSenPubMinN ? (size_t)llar::kSenPubSlots * chunk + chunk / 16 * 8
                                       : 2 * (size_t)nranks * chunk;
      break;
    }
    case LLAR_PROTO_LL128_ATOMIC:
    case LLAR_PROTO_LL128_DIRECT:
      lb = llar::kLL128Line;
      pl = ll128_payload(dtype);
      // two slots (LL AllGather) or three (AllGather read from the lines)
      st = (protocol == LLAR_PROTO_LL128_DIRECT ? 3 : 2) * ll128_lines_for(count, nranks, dtype) * llar::kLL128Line;
      break;
    default: st = 0; break;
  }
  if (line_bytes) *line_bytes = lb;
  if (payload_elems_per_line) *payload_elems_per_line = pl;
  if (staging_bytes_per_rank) *staging_bytes_per_rank = st;
  return LLAR_OK;
}

int llar_select_protocol(int nranks, int dtype, size_t count) {
  if (!valid_dtype(dtype) || nranks < 2 || nranks > llar::kMaxRanks) return LLAR_PROTO_AUTO;
  return select_protocol(nranks, dtype, count);
}

int llar_select_protocol_iters(int nranks, int dtype, size_t count, int iters, int chained, int nondeterministic) {
  if (!valid_dtype(dtype) || nranks < 2 || nranks > llar::kMaxRanks || iters < 1) return LLAR_PROTO_AUTO;
  return select_protocol_iters(nranks, dtype, count, iters, chained != 0, kDefaultLLCap, nondeterministic != 0);
}

int llar_set_auto_nondeterministic(int allow) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g) return LLAR_ERR_NOT_INIT;
  if (allow != 0 && allow != 1) return LLAR_ERR_INVALID;
  g->auto_atomic = allow;
  return LLAR_OK;
}

int llar_select_protocol_segment(int reduce_scatter, int nranks, int dtype, size_t count) {
  if (!valid_dtype(dtype) || nranks < 2 || nranks > llar::kMaxRanks) return LLAR_PROTO_AUTO;
  return select_segment_protocol(reduce_scatter != 0, nranks, count, elem_bytes(dtype));
}

int llar_select_protocol_host(int nranks, int dtype, size_t count) {
  if (!valid_dtype(dtype) || nranks < 2 || nranks > llar::kMaxRanks) return LLAR_PROTO_AUTO;
  return select_protocol_host(nranks, dtype, count);
}

unsigned long long llar_epoch(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g) return 0ull;
  unsigned long long done = 0;  // epochs used so far, kept on the device
  if (cudaMemcpy(&done, g->base + g->abort_off + 128, sizeof(done), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return 0ull;
  }
  return done + 1;
}

int llar_last_launch(int* protocol, int* ctas_per_rank, int* threads, int* iters) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (protocol) *protocol = g_last_proto;
  if (ctas_per_rank) *ctas_per_rank = g_last_G;
  if (threads) *threads = g_last_T;
  if (iters) *iters = g_last_iters;
  return LLAR_OK;
}

int llar_debug_launch_shape(int nranks, int dtype, size_t count, int protocol, int chained, int sms,
                            size_t chunk_bytes, int* ctas_per_rank, int* threads) {
  if (nranks < 2 || nranks > llar::kMaxRanks || !valid_dtype(dtype) || count == 0 || sms < 1) return LLAR_ERR_INVALID;
  if (protocol < LLAR_PROTO_LL || protocol > LLAR_PROTO_LL128_DIRECT) return LLAR_ERR_INVALID;
  if (chunk_bytes == 0 || chunk_bytes % 16 || chunk_bytes > kMaxChunk) return LLAR_ERR_INVALID;
  Ctx c;  // host arithmetic only: no device memory behind it
  c.n = nranks;
  c.dtype = dtype;
  c.esize = elem_bytes(dtype);
  c.sms = sms;
  c.chunk_bytes = chunk_bytes;
  int G = 1, T = 128;
  {
    std::lock_guard<std::mutex> lk(g_mu);  // a shape forced by llar_set_launch is read under the lock
    choose_shape(c, protocol, count, chained == 1 ? 1 : 0, &G, &T, chained == 2);
  }
  if (ctas_per_rank) *ctas_per_rank = G;
  if (threads) *threads = T;
  return LLAR_OK;
}

const char* llar_strerror(int status) {
  switch (status) {
    case LLAR_OK: return "ok";
    case LLAR_ERR_INVALID: return "invalid argument";
    case LLAR_ERR_NOT_INIT: return "llar_init has not been called";
    case LLAR_ERR_TOO_LARGE: return "message larger than the staging sized at init";
    case LLAR_ERR_UNSUPPORTED: return "unsupported dtype, protocol or mode";
    case LLAR_ERR_OCCUPANCY: return "the persistent grid cannot be fully resident";
    case LLAR_ERR_CUDA: return "CUDA runtime error";
    case LLAR_ERR_TIMEOUT: return "a device-side wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"
