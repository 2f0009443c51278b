// Internal types shared by the host runtime (llar_runtime.cu) and the
// kernels (llar_kernels.cu). Not part of the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "llar_llbuffer.h"

namespace llar {

constexpr int kMaxRanks = 8;
constexpr int kMaxThreads = 512;   // threads per CTA, upper bound of every kernel
constexpr size_t kRsVectorMinBytes = 64u << 10;  // fixed ReduceScatter: 16-byte vectors above this
                                                 // many bytes per rank, one element a thread up to it
constexpr int kLL128Line = 128;    // bytes per LL128 line
constexpr int kLL128Lanes = 8;     // 16-byte lanes (threads) per line
constexpr int kLLLine = 16;        // bytes per LL line: 8 data + 8 flag
constexpr int kAgLineBytes = 256;  // one LL128 line published again as 16 LL lines
// Sentinel one-shot. From kSenPubMinN ranks (with at most one vector per
// thread and chunk, and at least kSenPubMinSteps chunks in the launch) each
// rank publishes its chunks once in its own ring of
// kSenPubSlots = 4 kSenFencePeriod slots, fences every kSenFencePeriod
// chunks and resets a slot 2 kSenFencePeriod chunks after publishing it;
// its tail words (one u64 per vector of a chunk) follow the ring at
// kSenPubSlots * kSenMaxChunkBytes. Otherwise chunks are pushed into two
// slots per peer at the receivers, with the next chunk pushed as soon as
// this one has arrived for up to kSenEarlyMaxN ranks.
#ifndef LLAR_SEN_EARLY_MAX_N
#define LLAR_SEN_EARLY_MAX_N 4
#endif
#ifndef LLAR_SEN_PUB_MIN_N
#define LLAR_SEN_PUB_MIN_N 2
#endif
#ifndef LLAR_SEN_FENCE_PERIOD
#define LLAR_SEN_FENCE_PERIOD 8  // measured against 4: 8 ranks x 64 KiB fp16 in 8 KiB chunks 10.4 -> 10.0 us
#endif
#ifndef LLAR_SEN_PUB_MIN_STEPS
#define LLAR_SEN_PUB_MIN_STEPS 4
#endif
constexpr int kSenEarlyMaxN = LLAR_SEN_EARLY_MAX_N;
constexpr int kSenPubMinN = LLAR_SEN_PUB_MIN_N;
constexpr int kSenFencePeriod = LLAR_SEN_FENCE_PERIOD;
constexpr int kSenPubMinSteps = LLAR_SEN_PUB_MIN_STEPS;  // chunks per launch (iterations x chunks)
constexpr int kSenPubSlots = 4 * kSenFencePeriod;
constexpr size_t kSenMaxChunkBytes = 64u << 10;  // largest sentinel chunk per rank
// per (rank, CTA) signal words: 0 ready and 1 done epochs of the fixed-order
// chains, 2 consumption acknowledgements of point-to-point transfers
constexpr int kFlagKinds = 3;
constexpr int kFlagAck = 2;

// fault-injection modes (values of llar_inject_t)
constexpr int LLAR_INJECT_SKIP_ = 1;
constexpr int LLAR_INJECT_POISON_ = 2;
constexpr int LLAR_INJECT_DELAY_ = 3;

// Written by the first device wait that runs out; lives in mapped host
// memory so the host can read it without a device synchronisation. Its
// first three fields are an llar_llbuffer_status, so that the public device
// primitives (which record code, rank and epoch) can report into it; they
// leave `cta` as the host set it (-1: not recorded).
struct DevStatus {
  unsigned int code;  // 0 = ok, else an llar_status_t
  int rank;
  unsigned long long epoch;
  int cta;
  int pad;
};
static_assert(offsetof(DevStatus, code) == offsetof(llar_llbuffer_status, code) &&
                  offsetof(DevStatus, rank) == offsetof(llar_llbuffer_status, rank) &&
                  offsetof(DevStatus, epoch) == offsetof(llar_llbuffer_status, epoch),
              "DevStatus must start with an llar_llbuffer_status");

// Everything a launch needs. Passed by value as the kernel parameter.
struct Params {
  const char* in[kMaxRanks];  // rank inputs (iteration 0 / base)
  char* out[kMaxRanks];       // rank outputs (iteration 0 / base)
  size_t count;               // elements per rank
  int nranks;
  int G;                      // CTAs per rank
  int clustered;              // launch in clusters of nranks blocks (one CTA per rank, same range)
  int spread_smem;            // dynamic shared memory reserved only to keep one CTA per SM
  int pdl;                    // launch as a programmatic dependent of the previous kernel
  int no_coop;                // 1: waiting kernels launch without the cooperative attribute
                              // (the grid is still sized to fit the GPU at once)
  int iters;
  int chain;                  // 1: next input = RNE(chain_scale * output)
  float chain_scale;
  size_t in_stride;           // elements between iterations' inputs
  size_t out_stride;          // elements between iterations' outputs
  unsigned long long* epoch_dev;  // device epoch counter: iteration e uses *epoch_dev + 1 + e
  unsigned int* done_count;       // CTAs of this launch that finished (last one advances the epoch)

  // staging regions (device memory), rank r's region at base + r * stride
  char* ll;            size_t ll_stride;        // [2][N][W][16]
  size_t ll_slot_words;                         // W for this launch's layout (max words)
  char* sen;           size_t sen_stride;       // [2][N][CV][16]
  int sen_chunk_vecs;                           // CV: 16-byte vectors per chunk
  char* l128;          size_t l128_stride;      // [2][L][128]
  char* l128ag;        size_t l128ag_stride;    // [2][L][256]: the owner's published AllGather lines
  size_t l128_lines;                            // L: lines per slot
  char* l128d;         size_t l128d_stride;     // [3][L][128]: lines of the direct-AllGather variant
  unsigned long long* l128d_seq;                // [0] its AllReduces so far (slot = sequence % 3),
                                                // [1] lines per segment of its last launch
  char* chainbuf;      size_t chain_stride;     // [2][max_bytes] per rank
  size_t chain_slot_bytes;
  unsigned long long* flags;                    // [N][Gmax][kFlagKinds] signal words
  int flags_gmax;

  int peer_dst[kMaxRanks];  // point to point: rank r sends to peer_dst[r] (-1: none)
  int peer_src[kMaxRanks];  // and receives from peer_src[r] (-1: none)

  unsigned long long timeout_ns;
  int inject_rank;
  int inject_mode;
  unsigned int* abort_flag;  // device memory
  DevStatus* status;         // mapped host memory (device pointer)
};

// Process-wide wait bound (llar_set_timeout_ns) and fault injection
// (llar_debug_inject), for launches made outside the context (defined in
// llar_runtime.cu).
void fault_settings(unsigned long long* timeout_ns, int* inject_rank, int* inject_mode);

// Launchers, defined in llar_kernels.cu. Return a cudaError_t.
cudaError_t launch_ll(int dtype, const Params& p, int threads, cudaStream_t s);
cudaError_t launch_sentinel(int dtype, const Params& p, int threads, cudaStream_t s);
cudaError_t launch_ll128(int dtype, const Params& p, int threads, cudaStream_t s);
cudaError_t launch_ll128d(int dtype, const Params& p, int threads, cudaStream_t s);
cudaError_t launch_fixed_oneshot(int dtype, const Params& p, int threads, cudaStream_t s);
cudaError_t launch_fixed_twoshot(int dtype, const Params& p, int threads, cudaStream_t s);
// ReduceScatter / AllGather: which = 0 RS over LL, 1 AG over LL, 2 RS fixed,
// 3 AG fixed (one collective per launch)
cudaError_t launch_segment(int which, int dtype, const Params& p, int threads, cudaStream_t s);
int max_resident_segment_ctas(int which, int dtype, int nranks, int threads);
// point-to-point transfers (proto LLAR_PROTO_LL or LLAR_PROTO_SENTINEL)
cudaError_t launch_p2p(int proto, int dtype, const Params& p, int threads, cudaStream_t s);
int max_resident_p2p_ctas(int proto, int dtype, int threads);
// TMA bulk-copy variant of the fixed two-shot (no chain), one CTA per SM
cudaError_t launch_fixed_twoshot_bulk(int dtype, const Params& p, int threads, cudaStream_t s);
size_t bulk_smem_bytes(int nranks);
size_t bulk_tile_vectors();  // 16-byte vectors per rank tile of the bulk ring

// Largest number of CTAs of the kernel for (proto, dtype, nranks) that can
// be resident at once with `threads` threads each, in clusters of nranks
// blocks if `clustered` (0 on error).
int max_resident_ctas(int proto, int dtype, int nranks, int threads, bool clustered, int spread_smem);

// Speed-of-light probes: per-SM pointer-chase latency (ns per dependent
// L2 load) and per-pair ping-pong round trips (ns per store-observe-reply).
constexpr int kSolMaxBlocks = 256;
struct SolResult {
  int nchase;
  double chase_ns[kSolMaxBlocks];
  int chase_smid[kSolMaxBlocks];
  int npairs;
  double rt_ns[kSolMaxBlocks / 2];
  int smid_a[kSolMaxBlocks / 2];
  int smid_b[kSolMaxBlocks / 2];
};
// The probes use their own abort word, never the context's.
cudaError_t run_sol(SolResult* res, unsigned long long timeout_ns);
// The same two measurements over the CTAs of a launch of the given shape:
// the slowest chase among the SMs holding its blocks, and the round trips
// of every pair of blocks that exchange data (block c of two ranks).
struct SolPlaced {
  int npairs;
  int distinct_sms;
  double chase_worst_ns;
  double rt_worst_ns;
  double rt_median_ns;
};
cudaError_t run_sol_placed(int nranks, int G, int threads, int clustered, int spread_smem,
                           unsigned long long timeout_ns, SolPlaced* out);

}  // namespace llar
