// Device code of the fused all-gather matmul and of its barrier baseline.
//
// The design keeps the protocol of "Fused all-gather+GEMM HBM-buffer kernel
// for iris.ops" (ROCm/iris #346, section "New kernel") -- A tiles are staged
// into an HBM buffer, per-tile ready flags are published, GEMM workers wait on
// the flags and compute tiles as soon as their rows are staged -- and maps it
// onto persistent sm_103a CTA pairs (clusters of two; one CTA per SM) with
// specialised warps:
//
//   warp 0      A loads.  Barrier GEMM: the A issuer.  Fused: the A loader,
//               which issues each chunk's loads from the descriptor the
//               protocol warp (warp 7) wrote for it.
//   warp 1      MMA issuer (the pair's even CTA): tcgen05.mma.cta_group::2
//               256 x 256 x 16 (bf16/fp16; FP8 E4M3: x 32) with fp32
//               accumulation into one of two TMEM accumulators.
//   warps 2-5   epilogue: tcgen05.ld, (FP8: x scale) + fp32 bias, round to
//               16 bits, 128-byte-swizzled shared memory, TMA store.
//   warp 6      B loader: b's k-blocks in the chunk order of the A loads.
//   warp 7      protocol (fused only): the ready-flag protocol, a few chunks
//               ahead of the A loader.  Every (row block, k-group) chunk has
//               an owner: the column block whose tile starts its k-loop there
//               (tiles of one row block start at evenly spread k-groups).  The
//               owner has the chunk staged (a tile ahead, where it can) and
//               loads it; the other tiles of the row block follow: they wait
//               on the chunk's ready flag (read one chunk ahead) and load the
//               staged copy.  Chunks of the local shard are read straight
//               from it and never waited on.  Flag reads, waits, take-overs
//               and hand-offs all happen here, so none of them delays a load.
//               When A is small this warp first asks L2 for the CTA's share of
//               the shards.
//   warps 8-11  copiers (fused only), off the MMA pipeline.  The protocol
//               warp hands a chunk's record to them through a ring in shared
//               memory; they copy the chunk's boxes (spread over the four
//               warps) from its shard into a_gathered (the k-contiguous
//               staging) -- and, for the m-contiguous layout, transposed into
//               the [K, M] staging, which is what followers then read -- with
//               16-byte global loads and stores, and the last of them to
//               finish publishes the chunk.  The first copier starts as the
//               register fetcher: it copies the chunks that TMA cannot load
//               from a single shard (a row block straddling shards whose row
//               count is not a multiple of 8) and publishes them.
//
// Each staged box is therefore read from its shard once, and no atomic sits
// on the load path.  If a follower finds a chunk unpublished while its owner
// tile has not started yet (its CTA is still busy with an earlier tile, or the
// grid is small), it takes the chunk over: one atom.max decides between
// competing followers, and the winner loads, stages and publishes it.  A chunk
// staged twice (owner and taker) is harmless: both write identical bytes and
// publish the same value, and each publishes only after all of its own writes.
//
// Fetch prologue: when a k-contiguous call takes at most three waves and the
// last is partial, the CTAs with one tile fewer first copy all of A (their
// copier and epilogue warps, chunk by chunk in k-group order) and publish it;
// no tile owns a chunk then, every tile runs k ascending and waits on flags.
//
// Flags are 64-bit.  A call with epoch e uses base = e << 20: a flag below base
// is untouched by this call, base means taken over, base + boxes means
// published (ready).  Nothing is cleared between calls.  Every wait is bounded
// by a time limit; on expiry the kernel records an error word and finishes
// without hanging.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace agmm {

constexpr int kBM = 128;  // rows of an output tile (TMEM lanes)
constexpr int kBN = 256;  // columns of an output tile (TMEM columns per accumulator)
constexpr int kBK = 64;   // K per stage: 64 x 16 bit = one 128-byte swizzle row
constexpr int kUmmaK = 16;
constexpr int kAStageBytes = kBM * kBK * 2;  // 16 KB
constexpr int kMnChunkBytes = 64 * kBK * 2;  // one 64-wide MN chunk of an MN-major operand (8 KB)
constexpr int kEpiWarps = 4;
constexpr int kEpiRows = 32;                           // rows per epilogue warp
constexpr int kEpiCols = 64;                           // columns per store box (128 bytes)
constexpr int kEpiBufBytes = kEpiRows * kEpiCols * 2;  // 4 KB
constexpr int kEpiBufs = 2;
constexpr int kTmemCols = 2 * kBN;
constexpr int kCopyWarps = 4;  // fused kernel: warps copying staged chunks
constexpr int kProWarps = kCopyWarps + kEpiWarps;  // warps of the fetch prologue
constexpr int kMaxShards = 16;
constexpr int kFlagShift = 20;      // flag base = epoch << 20; boxes per chunk < 2^20

// Kernel variants: barrier-path GEMM (A from a_gathered or the [K, M] staging)
// and the fused kernel, each for both staging layouts.
enum Mode : int { kGemmK = 0, kGemmM = 1, kFusedK = 2, kFusedM = 3 };

__host__ __device__ constexpr bool mode_fused(int m) { return m >= kFusedK; }
__host__ __device__ constexpr bool mode_layout_m(int m) { return m == kGemmM || m == kFusedM; }
// Warp roles: 0 A loads, 1 MMA (pair: the even CTA's), 2..5 epilogue, 6 B
// loads; fused: 7 the ready-flag protocol, 8..11 copiers (8 also the register
// fetcher).
constexpr int kBWarp = 2 + kEpiWarps;
constexpr int kProtoWarp = 3 + kEpiWarps;
constexpr int kCopyWarp0 = 4 + kEpiWarps;
__host__ __device__ constexpr int mode_threads(int m) {
  return 32 * (3 + kEpiWarps + (mode_fused(m) ? 1 + kCopyWarps : 0));
}

// Bits of a stage's record (read by the MMA warp once the stage is full) and
// of a chunk record handed to the copiers.
constexpr uint32_t kInfoStage = 1u;    // chunk: to be written into a_gathered
constexpr uint32_t kInfoPublish = 2u;  // chunk: ... and published once written
constexpr uint32_t kInfoAmn = 4u;      // stage: the A box in shared memory is MN-major
constexpr uint32_t kInfoEnd = 8u;      // chunk record: no more chunks, the copiers leave

// Chunk records handed from the protocol warp to the copiers:
// {bits, mb, first k-block, boxes, flag index, box sequence index, done count, -}.
constexpr int kRing = 8;
constexpr int kRingWords = 8;

// Chunk descriptors handed from the protocol warp to the A loader (fused):
// {kind bits | bits << 8, row block, k-group | boxes << 16, first shard}.
constexpr int kDRing = 4;
constexpr uint32_t kDescDirect = 1u;    // load from a shard (else from the staging)
constexpr uint32_t kDescOneShard = 2u;  // ... from one shard map (else row groups across shards)
constexpr uint32_t kDescFence = 4u;     // staged data behind a flag: proxy fence before the loads
constexpr uint32_t kDescEnd = 8u;       // no more chunks

// Pipeline shape.  One CTA per output tile (kPair = false): 4 stages of A
// (128 x 64) + B (64 x 256).  A CTA pair per 256 x 256 tile (kPair = true):
// each CTA stages its own 128 rows of A and half of B's 256 columns, so a
// stage is 32 KB and 6 of them fit, half again as much latency cover.
template <bool kPair>
struct Pipe {
  static constexpr int kStages = kPair ? 6 : 4;
  static constexpr int kBCols = kPair ? kBN / 2 : kBN;  // B columns staged by this CTA
  static constexpr int kBStageBytes = kBCols * kBK * 2;
  static constexpr int kStageBytes = kAStageBytes + kBStageBytes;
  static constexpr int kData = kStages * kStageBytes + kEpiWarps * kEpiBufs * kEpiBufBytes;
  // full, empty [kStages]; tmem_full, tmem_empty [2]; drain; rfull, rfree
  // [kRing]; pro (fetch prologue done); dfull, dfree [kDRing]
  static constexpr int kBars = 2 * kStages + 4 + 1 + 2 * kRing + 1 + 2 * kDRing;
  // (+ the chunk descriptors, the protocol's progress word, the TMEM address and
  // the abort word)
  static constexpr int kSmemBytes = 1024 + kData + 8 * kBars + 4 * kStages +
                                    4 * kRing * kRingWords + 16 * kDRing + 16 + 64;
  static_assert(kSmemBytes <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
};

// Error codes written to the device error word (match ag_status).
constexpr uint32_t kErrTimeout = 4;
constexpr uint32_t kErrBounds = 8;  // AGMM_DEBUG builds: info = site << 24 | index
// Sites of a bounds violation (AGMM_DEBUG builds).
constexpr uint32_t kDbgFlag = 1, kDbgStarted = 2, kDbgShardRow = 3, kDbgGathered = 4,
                   kDbgStaging = 5, kDbgTile = 6;
// Sites reported with a pipeline timeout (ready-flag timeouts report the flag index).
constexpr uint32_t kSiteEmpty = 0xF00001, kSiteFull = 0xF00002, kSiteTmemEmpty = 0xF00003,
                   kSiteTmemFull = 0xF00004, kSiteRing = 0xF00005, kSiteCopy = 0xF00006,
                   kSitePro = 0xF00007, kSiteDesc = 0xF00008;

// Trace roles (see include/agmm.h).
constexpr uint32_t kTraceClaim = 1, kTraceWait = 2, kTraceTile = 3, kTraceGather = 4,
                   kTraceRegFetch = 5, kTraceIssue = 6;

struct GemmParams {
  CUtensorMap tm_a;                    // a_gathered [M, K]: box {64, 128}, 128B swizzle
  CUtensorMap tm_a_mk;                 // staging [K, M]: box {64, 64}, 128B swizzle
  CUtensorMap tm_b;                    // b [K, N]: box {64, 64}, 128B swizzle (MN-major B)
  CUtensorMap tm_out;                  // out [M, N]: box {64, 32}, 128B swizzle (store)
  CUtensorMap tm_shard[kMaxShards];    // shard r [m_per_shard, K]: box {64, 128}
  CUtensorMap tm_shard8[kMaxShards];   // shard r: box {64, 2^sh_log2} (row blocks straddling shards)
  const uint16_t* shards[kMaxShards];
  uint16_t* a_gathered;
  uint16_t* staging_mk;
  const float* bias;
  uint64_t* flags;          // [num_mb * G]
  uint64_t* started;        // [num_tiles]: epoch once the tile's protocol began it
  unsigned long long* err;  // [2]: epoch of newest error, code << 32 | info
  uint64_t* trace;
  int64_t trace_words;
  uint64_t epoch;
  uint64_t fbase;           // epoch << kFlagShift
  int64_t timeout_ns;       // one ready-flag wait
  int64_t pipe_timeout_ns;  // one pipeline (mbarrier) wait
  int M, N, K, D, mps, rank;
  int num_mb, num_nb, num_kb, num_tiles;
  int pair;                 // 1: CTA pairs, tile slot t = 2 * pair tile + CTA rank
  int sched_mb;             // rows of the schedule: num_mb, or pairs of row blocks
  int kpf, G;               // k-blocks per flag, flags per row block
  int mb_start;             // first row block of the schedule (ring order)
  int ng;                   // column blocks per schedule pass
  int w0;                   // column blocks of the first pass (they own the chunks)
  int sh_log2;              // log2 of the rows of a tm_shard8 box (3..6; divides m_per_shard)
  int seg_blocks;           // barrier GEMM over row segments (0: off): tm_a / tm_out are 3-D
  int seg_rows;             // [.., seg_rows, segments]; row block mb = segment mb / seg_blocks
  int fp16;                 // 1: fp16, 0: bf16 (the output's type for FP8 inputs)
  float scale_ab;           // FP8 inputs: scale_a * scale_b, applied to the fp32 sum
  int inject_skip_flag;     // this flag index is never published (fault injection)
  int pro_cta0;             // fetch prologue: CTAs from this index stage every chunk first (-1: off)
  int k_asc;                // 1: every tile visits its k-groups in ascending order
  int local_direct;         // 1 (fused m-contiguous pairs): pairs wholly in the local shard read it
                            // K-major, unstaged
  int stage_from;           // staging ahead starts at this position of the current tile's k-loop
  int l2_prefetch;          // 1: each CTA prefetches its share of the shards into L2 at the start
  int64_t inject_delay_ns;  // stress testing: publishers wait up to this long before a release
  int64_t flag_words;       // bounds of flags / started (checked in AGMM_DEBUG builds only)
  int64_t started_words;
};

struct GatherParams {
  const uint16_t* shards[kMaxShards];
  uint16_t* a_gathered;
  uint16_t* staging_mk;     // [K, M] or null
  int64_t vec_per_shard;    // 16-byte vectors per shard
  int M, K, mps;
  int row0, row1;           // agmm_gather_kernel copies gathered rows [row0, row1) ...
  int loc0, loc1;           // ... that are also local rows [loc0, loc1) of their shard
  uint64_t* trace;
  int64_t trace_words;
};

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ void record_error(const unsigned long long* err_c, uint64_t epoch,
                                             uint32_t code, uint32_t info) {
  unsigned long long* err = const_cast<unsigned long long*>(err_c);
  unsigned long long prev = atomicMax(err, (unsigned long long)epoch);
  if (prev < epoch) {
    atomicExch(err + 1, ((unsigned long long)code << 32) | info);
    __threadfence();
  }
}

// Bounds check of the bounds-checked build (-DAGMM_DEBUG, libagmm_debug.so):
// false when `ok` does not hold, after recording AG_ERR_BOUNDS with the site
// and the low 24 bits of the index; the caller then skips the access.  The
// release build compiles it to `true`.
__device__ __forceinline__ bool dbg_ok(const GemmParams& p, bool ok, uint32_t site, int64_t idx) {
#ifdef AGMM_DEBUG
  if (!ok) {
    record_error(p.err, p.epoch, kErrBounds, (site << 24) | ((uint32_t)idx & 0xFFFFFFu));
    return false;
  }
#else
  (void)p, (void)ok, (void)site, (void)idx;
#endif
  return true;
}

__device__ __forceinline__ bool flag_ok(const GemmParams& p, int64_t idx) {
  return dbg_ok(p, idx >= 0 && idx < p.flag_words, kDbgFlag, idx);
}

// Stress testing (ag_options.inject_delay_ns): a publisher waits a
// pseudo-random 0 .. inject_delay_ns (a hash of the flag index and the call's
// epoch) between its copies and the release store that publishes them, so
// that readers meet publishers late and in shuffled order.  The wait is
// bounded by time and by an iteration count.
__device__ __forceinline__ void inject_delay(const GemmParams& p, int flag_idx) {
  if (p.inject_delay_ns <= 0) return;
  uint32_t h = (uint32_t)flag_idx * 0x9E3779B1u ^ (uint32_t)p.epoch * 0x85EBCA77u;
  h ^= h >> 15;
  h *= 0xC2B2AE3Du;
  h ^= h >> 13;
  const uint64_t d = (uint64_t)p.inject_delay_ns * (h & 1023u) / 1023u;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 26) && globaltimer_ns() - t0 < d; ++it) {
  }
}

__device__ __forceinline__ bool error_this_call(const GemmParams& p) {
  return ld_relaxed_gpu(reinterpret_cast<const uint64_t*>(p.err)) == p.epoch;
}

__device__ __forceinline__ void trace_rec(uint64_t* tr, int64_t words, uint32_t role, uint32_t a,
                                          uint32_t b, uint64_t t0, uint64_t t1) {
  unsigned long long i = atomicAdd(reinterpret_cast<unsigned long long*>(tr), 1ull);
  int64_t w = 1 + 4 * (int64_t)i;
  if (w + 4 > words) return;
  tr[w] = t0;
  tr[w + 1] = t1;
  tr[w + 2] = ((uint64_t)role << 56) | ((uint64_t)(blockIdx.x & 0xFFFFu) << 40) |
              ((uint64_t)(a & 0xFFFFFu) << 20) | (uint64_t)(b & 0xFFFFFu);
  tr[w + 3] = 0;
}

// Persistent schedule: tile t -> (row block, column block).  Column blocks
// are taken in groups of ng: a pass sweeps every row block over one group, so
// only that group's columns of b need to stay in L2 during the pass (A is read
// once per group).  Within a pass, row blocks are visited in ring order
// starting at mb_start (the local shard's first block for the fused kernel),
// the group's column blocks of one row block consecutively, so concurrently
// running CTAs share A rows in L2.
__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& mb, int& nb) {
  // With CTA pairs a schedule row is a pair of row blocks and slot t belongs
  // to CTA rank t & 1 of the pair that takes pair tile t >> 1 (the grid is
  // even, so a CTA's slots all have its rank).  Row block num_mb (the second
  // half of a last, odd pair) lies past M: its loads read zeros, its stores
  // are skipped.
  const int u = t >> p.pair;
  const int per_pass = p.sched_mb * p.ng;
  const int gq = u / per_pass;
  const int g0 = gq * p.ng;
  const int width = min(p.ng, p.num_nb - g0);
  const int r = u - gq * per_pass;
  const int pos = r / width;
  nb = g0 + (r - pos * width);
  int ms = p.mb_start + pos;
  if (ms >= p.sched_mb) ms -= p.sched_mb;
  mb = p.pair ? 2 * ms + (t & 1) : ms;
}

__device__ __forceinline__ int my_tile_count(const GemmParams& p) {
  return p.num_tiles > (int)blockIdx.x ? (p.num_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1
                                       : 0;
}

// How a row block's A rows can be fetched.
// kEmpty: the second row block of a last, odd CTA pair (rows past M).
enum BlockKind : int { kLocal = 0, kDirect = 1, kRegFetch = 2, kEmpty = 3 };

// Local: every row lies in the local shard.  Direct: one shard holds every
// row, or the block straddles shards at multiples of 8 rows (8-row TMA boxes).
// Otherwise the register fetcher stages it.
__device__ __forceinline__ int block_kind(const GemmParams& p, int mb) {
  const int lo = mb * kBM;
  const int hi = min(lo + kBM, p.M);
  if (lo >= p.rank * p.mps && hi <= (p.rank + 1) * p.mps) return kLocal;
  if (lo / p.mps == (hi - 1) / p.mps || (p.mps & 7) == 0) return kDirect;
  return kRegFetch;
}

// First k-group of every tile in column block nb: the column blocks of a row
// block start evenly spread over its k-groups.
__device__ __forceinline__ int chunk_start(const GemmParams& p, int nb) {
  // nb * G < 2^31: num_mb * G and num_tiles are bounded
  return nb < p.w0 ? (nb * p.G) / p.w0 : 0;
}

// End of the window owned by column block nb (empty outside the first group).
__device__ __forceinline__ int chunk_end(const GemmParams& p, int nb) {
  return nb < p.w0 ? ((nb + 1) * p.G) / p.w0 : 0;
}

// k-group visited at position i of a tile whose owned window is [ws, we): the
// window first, then every other k-group in ascending order.  After the short
// owner phase the tiles of a row block walk k in step again (they share A
// k-slices in L2), and by then every window has been published.
__device__ __forceinline__ int chunk_at(int i, int ws, int we) {
  const int wlen = we - ws;
  if (i < wlen) return ws + i;
  const int j = i - wlen;
  return j < ws ? j : j + wlen;
}

// k-group visited at position i of a tile: k ascending when the launch plan
// says so (p.k_asc: calls of four or more waves, where a CTA's next window is
// staged while it works on the current tile, so every tile of a row block can
// read A in the same order as its neighbours and the barrier GEMM, sharing
// each k-slice in L2), else the owned window first (chunk_at).
__device__ __forceinline__ int order_at(const GemmParams& p, int i, int ws, int we) {
  return p.k_asc ? i : chunk_at(i, ws, we);
}

// The column block whose tiles own k-group g: the nb < w0 with
// chunk_start(nb) <= g < chunk_end(nb).
__device__ __forceinline__ int owner_nb(const GemmParams& p, int g) {
  return ((g + 1) * p.w0 + p.G - 1) / p.G - 1;
}

// Schedule index of tile (mb, nb) (inverse of tile_coords).
__device__ __forceinline__ int tile_index(const GemmParams& p, int mb, int nb) {
  int pos = (mb >> p.pair) - p.mb_start;
  if (pos < 0) pos += p.sched_mb;
  const int gq = nb / p.ng;
  const int g0 = gq * p.ng;
  const int width = min(p.ng, p.num_nb - g0);
  const int u = gq * p.sched_mb * p.ng + pos * width + (nb - g0);
  return p.pair ? 2 * u + (mb & 1) : u;
}

__device__ __forceinline__ int chunk_boxes(const GemmParams& p, int g) {
  return min(p.kpf, p.num_kb - g * p.kpf);
}

// Per-tile facts the chunk loop needs for every chunk, computed once per tile.
struct TileCtx {
  int mb, nb;
  int sd, sy;      // segmented barrier GEMM: segment and first row of the block in it
  int kind;        // BlockKind (kDirect for the barrier-path GEMM)
  int r0;          // shard holding the block's first row
  bool one_shard;  // every row of the block lies in shard r0
  int ws, we;      // owned window of k-groups [ws, we); ws is also the k-loop start
  bool pair_local; // CTA pairs with p.local_direct: every row of the pair's two blocks is in
                   // the local shard (or past M), so the pair reads A straight from the
                   // shard, even with the m-contiguous staging
  __device__ __forceinline__ bool owns(int g) const { return g >= ws && g < we; }
};

template <bool kFused>
__device__ __forceinline__ void tile_ctx(const GemmParams& p, int t, TileCtx& c) {
  tile_coords(p, t, c.mb, c.nb);
  if (!dbg_ok(p, c.mb >= 0 && c.mb < p.num_mb + p.pair && c.nb >= 0 && c.nb < p.num_nb, kDbgTile,
              t))
    c.mb = p.num_mb + p.pair;  // (bounds-checked build) treated as rows past M
  // Fused: the owned window first (chunk_at).  The barrier GEMM has nothing
  // to own and runs k in ascending order, which keeps the tiles of a row
  // block reading the same A k-block at about the same time.
  c.ws = kFused ? chunk_start(p, c.nb) : 0;
  c.we = kFused ? chunk_end(p, c.nb) : 0;
  if (!kFused && p.seg_blocks) {
    c.sd = c.mb / p.seg_blocks;
    c.sy = (c.mb - c.sd * p.seg_blocks) * kBM;
  }
  c.pair_local = false;
  if (kFused && p.pair && p.local_direct) {
    const int m0 = c.mb & ~1;
    const int k1 = m0 + 1 < p.num_mb ? block_kind(p, m0 + 1) : (int)kEmpty;
    c.pair_local = m0 < p.num_mb && block_kind(p, m0) == kLocal && (k1 == kLocal || k1 == kEmpty);
  }
  if (c.mb >= p.num_mb) {
    c.kind = kEmpty;
    c.r0 = 0;
    c.one_shard = true;
    return;
  }
  c.kind = kFused ? block_kind(p, c.mb) : kDirect;
  const int lo = c.mb * kBM, hi = min(lo + kBM, p.M);
  c.r0 = lo / p.mps;
  c.one_shard = (hi - 1) / p.mps == c.r0;
}

// Bounded mbarrier wait.  Returns false (after flagging the CTA abort word and
// recording an error) when the phase does not complete in time.
// kCluster: acquire at cluster scope (the barrier takes arrivals from the peer CTA).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(const GemmParams& p, uint64_t* bar, uint32_t parity,
                                         volatile int* abort_flag, uint32_t site) {
  auto test = [&]() {
    return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (test()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (test()) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > (uint64_t)p.pipe_timeout_ns || it > (1u << 28)) {
        *abort_flag = 1;
        record_error(p.err, p.epoch, kErrTimeout, site);
        return false;
      }
    }
  }
}

// Issuer side of the hand-off: writes a chunk record into a ring slot and
// arrives on the slot's rfull barrier (the arrive releases the record).
__device__ __forceinline__ void hand_chunk(uint32_t* rec, uint64_t* rfull_bar, uint32_t bits,
                                           int mb, int g, int nbox, int flag_idx, int seq,
                                           const GemmParams& p) {
  rec[0] = bits;
  rec[1] = (uint32_t)mb;
  rec[2] = (uint32_t)(g * p.kpf);
  rec[3] = (uint32_t)nbox;
  rec[4] = (uint32_t)flag_idx;
  rec[5] = (uint32_t)seq;
  rec[6] = 0u;  // done count
  mbar_arrive(rfull_bar);
}

// Copier side of the hand-off: waits for phase `n` of a ring slot's `rfull`
// barrier (the protocol warp's n-th record in that slot).  False on abort or
// timeout.  Copiers may idle for as long as their CTA has nothing to stage,
// so the time limit restarts whenever the protocol warp makes progress (`iseq`).
__device__ __forceinline__ bool wait_handoff(const GemmParams& p, uint64_t* bar, uint32_t n,
                                             volatile uint32_t* iseq, volatile int* abort_flag) {
  const uint32_t parity = n & 1u;
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  uint32_t seen = *iseq;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      const uint32_t now_seq = *iseq;
      const uint64_t now = globaltimer_ns();
      if (now_seq != seen) {
        seen = now_seq;
        t0 = now;
      } else if (now - t0 > (uint64_t)p.pipe_timeout_ns) {
        *abort_flag = 1;
        record_error(p.err, p.epoch, kErrTimeout, kSiteCopy);
        return false;
      }
    }
  }
}

// Follower wait on a chunk: bounded acquire-polling until flag >= target.
// When the flag is still untouched and the owner tile (owner_tile >= 0) has
// not started, try to take the chunk over (atom.max to base); returns true if
// this caller won it (it must then load, stage and publish the chunk).  On
// expiry (or once another wait of this call has expired) it records the error
// and returns false; the caller then proceeds, so the pipeline always drains.
__device__ __forceinline__ bool wait_or_take(const GemmParams& p, int flag_idx, uint64_t target,
                                             int owner_tile) {
  if (!flag_ok(p, flag_idx)) return false;
  if (owner_tile >= 0 && !dbg_ok(p, owner_tile < p.started_words, kDbgStarted, owner_tile))
    owner_tile = -1;
  uint64_t* f = p.flags + flag_idx;
  const uint64_t t0 = globaltimer_ns();
  // Once the owner tile is seen started it stays started for this call, so
  // its word is no longer read; while it is read, both loads are in flight at
  // once.  Polls are relaxed: one acquire fence follows the poll that sees
  // the chunk published.
  bool owner_started = owner_tile < 0;
  for (uint32_t it = 0;; ++it) {
    const uint64_t v = ld_relaxed_gpu(f);
    const uint64_t st = owner_started ? p.epoch : ld_relaxed_gpu(p.started + owner_tile);
    if (v >= target) {
      fence_acquire_gpu();
      return false;
    }
    if (st == p.epoch) {
      owner_started = true;
    } else if (v < p.fbase && atom_max_relaxed_gpu(f, p.fbase) < p.fbase) {
      return true;
    }
    __nanosleep(64);
    if ((it & 15u) == 15u) {
      if (error_this_call(p)) return false;
      if (globaltimer_ns() - t0 > (uint64_t)p.timeout_ns || it > (1u << 26)) {
        record_error(p.err, p.epoch, kErrTimeout, (uint32_t)flag_idx & 0xFFFFFFu);
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t u4_get(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// 8x8 transpose of 16-bit values held as 8 rows of 16 bytes: column c of the
// input becomes vector c of the output (word w holds rows 2w, 2w+1).
__device__ __forceinline__ uint4 transpose_col(const uint4 (&v)[8], int c) {
  const uint32_t sel = (c & 1) ? 0x7632u : 0x5410u;
  uint4 o;
  o.x = __byte_perm(u4_get(v[0], c >> 1), u4_get(v[1], c >> 1), sel);
  o.y = __byte_perm(u4_get(v[2], c >> 1), u4_get(v[3], c >> 1), sel);
  o.z = __byte_perm(u4_get(v[4], c >> 1), u4_get(v[5], c >> 1), sel);
  o.w = __byte_perm(u4_get(v[6], c >> 1), u4_get(v[7], c >> 1), sel);
  return o;
}

__device__ __forceinline__ const uint16_t* shard_row(const uint16_t* const* shards, int mps, int K,
                                                     int grow) {
  int s = grow / mps;
  int lr = grow - s * mps;
  return shards[s] + (int64_t)lr * K;
}

// Fetch prologue: copy box kb (64 columns) of row block mb from the shards
// into a_gathered, one warp per box.  Lane = (row-group quarter, 16-byte
// column chunk): four 8-row groups per lane, all 32 loads in flight before
// the first store.  Needs m_per_shard % 8 == 0 (no 8-row group straddles).
__device__ __forceinline__ void prologue_copy_box(const GemmParams& p, int mb, int kb, int lane) {
  const int k = kb * kBK + (lane & 7) * 8;
  if (k >= p.K) return;  // K % 8 == 0: a column chunk is all in or all out
  uint4 v[4][8];
  int m[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    m[h] = mb * kBM + (4 * h + (lane >> 3)) * 8;
    const int nrow = min(8, p.M - m[h]);
    if (nrow > 0 && dbg_ok(p, m[h] >= 0 && k + 8 <= p.K, kDbgShardRow, m[h])) {
      const uint16_t* src = shard_row(p.shards, p.mps, p.K, m[h]) + k;
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r < nrow) v[h][r] = ld_stream_v4(src + (int64_t)r * p.K);
    }
  }
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const int nrow = min(8, p.M - m[h]);
    if (!dbg_ok(p, m[h] >= 0 && k + 8 <= p.K, kDbgGathered, m[h])) continue;
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < nrow) st_v4(p.a_gathered + (int64_t)(m[h] + r) * p.K + k, v[h][r]);
  }
}

// Fetch prologue (calls whose last wave is partial; p.pro_cta0 >= 0): the
// CTAs with one tile fewer than the others stage every chunk of A before
// their own tiles, k-group by k-group (the order in which the tiles read
// them), chunk c by prologue CTA c mod (their number).  The copier and the
// epilogue warps (pw = 0 .. kProWarps - 1) split a chunk's boxes; once all of
// them are through (named barrier 1), one thread publishes it.  Nothing here
// waits on another CTA, so every chunk is published whatever the pipelines
// do.  Every one of those warps then arrives on pro_bar (all CTAs).
__device__ __forceinline__ void fetch_prologue(const GemmParams& p, int pw, int lane,
                                               uint64_t* pro_bar) {
  if (p.pro_cta0 >= 0 && (int)blockIdx.x >= p.pro_cta0) {
    const int nf = (int)gridDim.x - p.pro_cta0;
    const int total = p.num_mb * p.G;
    for (int c = (int)blockIdx.x - p.pro_cta0; c < total; c += nf) {
      const uint64_t t0 = p.trace ? globaltimer_ns() : 0;
      const int g = c / p.num_mb;
      const int mb = c - g * p.num_mb;
      const int nbox = chunk_boxes(p, g);
      for (int j = pw; j < nbox; j += kProWarps) prologue_copy_box(p, mb, g * p.kpf + j, lane);
      __threadfence();
      fence_proxy_async_global();
      named_bar_sync(1, kProWarps * 32);
      if (pw == 0 && lane == 0) {
        const int flag_idx = mb * p.G + g;
        if (flag_idx != p.inject_skip_flag && flag_ok(p, flag_idx)) {
          inject_delay(p, flag_idx);
          st_release_gpu(p.flags + flag_idx, p.fbase + (uint64_t)nbox);
        }
        if (p.trace) trace_rec(p.trace, p.trace_words, kTraceGather, mb, g, t0, globaltimer_ns());
      }
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(pro_bar);
}

// ------------------------------------------------------------------ register fetcher

// Stage one chunk of a row block TMA cannot load from the shards (it straddles
// shards at a row offset that is not a multiple of 8).  k-contiguous: copy into
// a_gathered.  m-contiguous: also write it transposed into the [K, M] staging.
__device__ __noinline__ void regfetch_chunk(const GemmParams& p, int mb, int g, int lane,
                                            bool layout_m) {
  const int row0 = mb * kBM;
  const int rows = min(kBM, p.M - row0);
  const int c0 = g * p.kpf * kBK;
  const int cols = min(p.kpf * kBK, p.K - c0);
  if (!layout_m) {
    const int nv = cols >> 3;  // 16-byte vectors per row
    const int total = rows * nv;
    constexpr int U = 8;
    for (int base = 0; base < total; base += 32 * U) {
      uint4 v[U];
      int64_t dst[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int idx = base + u * 32 + lane;
        dst[u] = -1;
        if (idx < total) {
          const int r = idx / nv;
          const int cv = idx - r * nv;
          if (dbg_ok(p, row0 + r < p.M && c0 + cv * 8 + 8 <= p.K, kDbgShardRow, row0 + r)) {
            v[u] = ld_stream_v4(shard_row(p.shards, p.mps, p.K, row0 + r) + c0 + cv * 8);
            dst[u] = (int64_t)(row0 + r) * p.K + c0 + cv * 8;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (dst[u] >= 0) st_v4(p.a_gathered + dst[u], v[u]);
    }
    return;
  }
  // rows is a multiple of 8 here (M % 8 == 0 for the m-contiguous layout).
  const int nrg = rows >> 3, ncg = cols >> 3;
  const int total = nrg * ncg;
  for (int idx = lane; idx < total; idx += 32) {
    const int rg = idx % nrg, cg = idx / nrg;
    const int col = c0 + cg * 8;
    if (!dbg_ok(p, row0 + rg * 8 + 8 <= p.M && col + 8 <= p.K, kDbgStaging, row0 + rg * 8))
      continue;
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      v[i] = ld_stream_v4(shard_row(p.shards, p.mps, p.K, row0 + rg * 8 + i) + col);
#pragma unroll
    for (int i = 0; i < 8; ++i) st_v4(p.a_gathered + (int64_t)(row0 + rg * 8 + i) * p.K + col, v[i]);
#pragma unroll
    for (int c = 0; c < 8; ++c)
      st_v4(p.staging_mk + (int64_t)(col + c) * p.M + row0 + rg * 8, transpose_col(v, c));
  }
}

__device__ __forceinline__ void regfetch_loop(const GemmParams& p, int lane, bool layout_m) {
  int last_mb = -1;
  for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
    int mb, nb;
    tile_coords(p, t, mb, nb);
    if (mb == last_mb || mb >= p.num_mb || block_kind(p, mb) != kRegFetch) continue;
    last_mb = mb;
    for (int g = 0; g < p.G; ++g) {
      const int idx = mb * p.G + g;
      uint64_t* f = p.flags + idx;
      int won = 0;
      if (lane == 0 && flag_ok(p, idx)) {
        const uint64_t v = ld_relaxed_gpu(f);
        if (v < p.fbase)
          won = atomicCAS(reinterpret_cast<unsigned long long*>(f), (unsigned long long)v,
                          (unsigned long long)p.fbase) == v;
      }
      won = __shfl_sync(0xffffffffu, won, 0);
      if (!won) continue;
      const uint64_t t0 = p.trace ? globaltimer_ns() : 0;
      regfetch_chunk(p, mb, g, lane, layout_m);
      __threadfence();
      fence_proxy_async_global();
      __syncwarp();
      if (lane == 0) {
        if (idx != p.inject_skip_flag) {
          inject_delay(p, idx);
          red_release_add_gpu(f, (uint64_t)chunk_boxes(p, g));
        }
        if (p.trace) trace_rec(p.trace, p.trace_words, kTraceRegFetch, mb, g, t0, globaltimer_ns());
      }
    }
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int fp16) {
  if (fp16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// A stage's tiled loads: counted on this CTA's `full` barrier, or (CTA pair)
// on the leader's, whose shared::cluster address is bar_c.
template <bool kPair>
__device__ __forceinline__ void stage_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                              uint32_t bar_c, int32_t x, int32_t y) {
  if constexpr (kPair)
    tma_load_2d_pair(dst, m, bar_c, x, y);
  else
    tma_load_2d(dst, m, bar, x, y);
}

template <bool kPair>
__device__ __forceinline__ void stage_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                              uint32_t bar_c, int32_t x, int32_t y, int32_t z) {
  if constexpr (kPair)
    tma_load_3d_pair(dst, m, bar_c, x, y, z);
  else
    tma_load_3d(dst, m, bar, x, y, z);
}

// After an abort: let this thread's issued loads land before the CTA (and
// its shared memory) goes away.  Waits on the stages' `full` phases, bounded;
// the pair's peer cannot observe its loads (they count on the leader's
// barriers) and waits a fixed 200 us instead, far above a load's latency.
template <bool kPair>
__device__ __forceinline__ void drain_loads(uint64_t* full, uint32_t issued_mask,
                                            uint32_t issued_parity, uint32_t rank) {
  if (kPair && rank != 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) {
    }
    return;
  }
  constexpr int kStages = Pipe<kPair>::kStages;
  for (int s = 0; s < kStages; ++s)
    if (issued_mask & (1u << s)) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&full[s], (issued_parity >> s) & 1u) &&
             globaltimer_ns() - t0 < 1000000000ull) {
      }
    }
}

// The A side of the stage ring, as the thread that loads A sees it.
struct ARing {
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued_mask = 0, issued_parity = 0;  // for drain_loads after an abort
};

// One chunk's A loads: `nbox` k-blocks from k-block `kb0` of row block `mb`,
// each into the next stage of the ring once the MMA has freed it; `bits`
// goes to the stage record.  One loop per kind of A box (shard map, shard row
// groups, [K, M] staging, segmented or plain gathered map), so that nothing in
// the per-stage path branches on the chunk's kind: the loading thread's time
// per stage bounds how far ahead of the MMA it keeps the ring.  False on
// abort or timeout.
template <bool kPair, bool kFused, bool kLayoutM>
__device__ __forceinline__ bool a_chunk_loads(const GemmParams& p, ARing& ar, uint8_t* smem,
                                              uint64_t* full, uint64_t* empty, uint32_t* info,
                                              uint32_t full_c, uint32_t rank,
                                              volatile int* abort_flag, uint32_t bits,
                                              bool direct, bool one_shard, int r0, int mb,
                                              int kb0, int nbox, int sy, int sd) {
  constexpr int kStages = Pipe<kPair>::kStages;
  constexpr int kStageBytes = Pipe<kPair>::kStageBytes;
  bool ok = true;
  auto stage_loop = [&](auto&& load_a) {
    for (int j = 0; j < nbox; ++j) {
      if (!wait_bar(p, &empty[ar.stage], ar.phase ^ 1u, abort_flag, kSiteEmpty)) {
        ok = false;
        return;
      }
      info[ar.stage] = bits;
      uint8_t* a_dst = smem + ar.stage * kStageBytes;
      const uint32_t bar_c = full_c + 8u * (uint32_t)ar.stage;
      if (!kPair || rank == 0)
        mbar_arrive_expect_tx(&full[ar.stage], kPair ? 2 * kAStageBytes : kAStageBytes);
      load_a(a_dst, &full[ar.stage], bar_c, (kb0 + j) * kBK);
      ar.issued_mask |= 1u << ar.stage;
      ar.issued_parity = (ar.issued_parity & ~(1u << ar.stage)) | (ar.phase << ar.stage);
      if (++ar.stage == kStages) {
        ar.stage = 0;
        ar.phase ^= 1u;
      }
    }
  };
  if (direct && one_shard) {
    const CUtensorMap* m = &p.tm_shard[r0];
    const int y = mb * kBM - r0 * p.mps;
    stage_loop([&](uint8_t* a_dst, uint64_t* fb, uint32_t bar_c, int x) {
      stage_load_2d<kPair>(a_dst, m, fb, bar_c, x, y);
    });
  } else if (direct) {
    // Walk the row groups (2^sh_log2 rows, which divides both 128 and
    // m_per_shard, so no group straddles a boundary) across the shards
    // without a division per group.  Past the last shard the row stays out of
    // range: TMA zero-fills it.
    stage_loop([&](uint8_t* a_dst, uint64_t* fb, uint32_t bar_c, int x) {
      const int h = 1 << p.sh_log2;
      int r = r0, lr = mb * kBM - r0 * p.mps;
#pragma unroll 1
      for (int q = 0; q < (kBM >> p.sh_log2); ++q) {
        stage_load_2d<kPair>(a_dst + q * h * 128, &p.tm_shard8[r], fb, bar_c, x, lr);
        lr += h;
        if (lr >= p.mps && r < p.D - 1) {
          lr -= p.mps;
          ++r;
        }
      }
    });
  } else if (kLayoutM) {
    stage_loop([&](uint8_t* a_dst, uint64_t* fb, uint32_t bar_c, int x) {
      stage_load_2d<kPair>(a_dst, &p.tm_a_mk, fb, bar_c, mb * kBM, x);
      stage_load_2d<kPair>(a_dst + kMnChunkBytes, &p.tm_a_mk, fb, bar_c, mb * kBM + 64, x);
    });
  } else if (!kFused && p.seg_blocks) {
    stage_loop([&](uint8_t* a_dst, uint64_t* fb, uint32_t bar_c, int x) {
      stage_load_3d<kPair>(a_dst, &p.tm_a, fb, bar_c, x, sy, sd);
    });
  } else {
    stage_loop([&](uint8_t* a_dst, uint64_t* fb, uint32_t bar_c, int x) {
      stage_load_2d<kPair>(a_dst, &p.tm_a, fb, bar_c, x, mb * kBM);
    });
  }
  return ok;
}

// ------------------------------------------------------------------ the kernel

// kPair: launched in clusters of two CTAs; the even CTA (rank 0, the leader)
// issues tcgen05.mma.cta_group::2 for the pair's 256 x 256 tile.  Both CTAs
// load their own 128 rows of A and half of B's columns into their own shared
// memory, but every load of the pair counts its bytes on the LEADER's `full`
// barrier (cta_group::2 loads), whose two arrivals (the leader's A and B
// loaders) expect the bytes of both CTAs; the peer's `full` barriers are
// unused.  A stage of the peer is refilled only after the MMA commit that
// frees it (multicast to both CTAs' `empty`), which follows the completion of
// the leader's phase, so no load of a new phase can land in an old one.
// kF8: A and b are FP8 E4M3 (kind::f8f6f4 MMAs), b given K-major ([N, K]),
// out bf16 scaled by scale_ab.  All data movement treats a row of K bytes as
// K/2 16-bit words, so p.K, the boxes, the flags and the copiers are those of
// a 16-bit problem with half the columns; only the MMA, B's major-ness and
// the epilogue differ.  k-contiguous layout only.
template <int kMode, bool kPair, bool kF8>
__global__ void __launch_bounds__(mode_threads(kMode), 1)
    agmm_gemm_kernel(const __grid_constant__ GemmParams p) {
  static_assert(!kF8 || !mode_layout_m(kMode), "FP8 runs with the k-contiguous layout only");
  using P = Pipe<kPair>;
  constexpr int kStages = P::kStages;
  constexpr int kStageBytes = P::kStageBytes;
  constexpr bool kFused = mode_fused(kMode);
  constexpr bool kLayoutM = mode_layout_m(kMode);
  // Fused m-contiguous on CTA pairs: every A tile is read from the [K, M]
  // staging (MN-major) -- the owner's window and local rows included, once
  // published -- because one pair MMA reads both CTAs' A with one major-ness;
  // except in pairs whose rows all lie in the local shard (TileCtx::pair_local):
  // both CTAs read those K-major from the shard, nobody waits for them, and
  // their chunks go to a_gathered only (no reader needs them transposed).
  constexpr bool kAllStaged = kFused && kLayoutM && kPair;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* epi_smem = smem + kStages * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P::kData);
  uint64_t* full = bars;                     // [kStages] TMA landed
  uint64_t* empty = bars + kStages;          // [kStages] the MMAs reading the stage are done
  uint64_t* tmem_full = bars + 2 * kStages;  // [2] accumulator ready
  uint64_t* tmem_empty = tmem_full + 2;      // [2] accumulator drained
  uint64_t* drain = tmem_empty + 2;          // [1] final MMA drain
  uint64_t* rfull = drain + 1;               // [kRing] fused: chunk record written
  uint64_t* rfree = rfull + kRing;           // [kRing] fused: every copier is done with it
  uint64_t* pro_bar = rfree + kRing;         // [1] fused: this CTA's fetch prologue is done
  uint64_t* dfull = pro_bar + 1;             // [kDRing] fused: chunk descriptor written
  uint64_t* dfree = dfull + kDRing;          // [kDRing] fused: the A loader has read it
  uint32_t* info = reinterpret_cast<uint32_t*>(dfree + kDRing);  // [kStages]
  uint32_t* ring = info + kStages;                // [kRing][kRingWords] chunk records
  uint32_t* dring = ring + kRing * kRingWords;    // [kDRing][4] chunk descriptors
  volatile uint32_t* iseq = dring + kDRing * 4;   // protocol progress (boxes), a liveness signal
  uint32_t* tmem_slot = dring + kDRing * 4 + 1;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int my_tiles = my_tile_count(p);
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 2);  // the A and the B loader (pair: the leader's, for both CTAs' bytes)
      mbar_init(&empty[s], 1);  // the MMA commit (pair: multicast to both CTAs)
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&rfull[r], 1);
      mbar_init(&rfree[r], kCopyWarps);
    }
    mbar_init(pro_bar, kProWarps);
    for (int d = 0; d < kDRing; ++d) {
      mbar_init(&dfull[d], 1);
      mbar_init(&dfree[d], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      // one arrive per epilogue warp (pair: the leader's barrier takes both CTAs')
      mbar_init(&tmem_empty[b], kEpiWarps * (kPair ? 2 : 1));
    }
    mbar_init(drain, 1);
    *iseq = 0;
    *abort_flag = 0;
    fence_mbarrier_init();
    prefetch_tensormap(&p.tm_a);
    prefetch_tensormap(&p.tm_b);
    prefetch_tensormap(&p.tm_out);
    if (kLayoutM) prefetch_tensormap(&p.tm_a_mk);
  }
  if (warp == 1) {
    tmem_alloc<kPair>(tmem_slot, kTmemCols);
    tmem_relinquish_alloc_permit<kPair>();
  }
  tcgen05_fence_before_sync();
  __syncthreads();
  // Pair: both CTAs' barriers are initialised before either signals the other's.
  if (kPair) cluster_sync();
  tcgen05_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // Pair: the leader's `full` barriers, where both CTAs' loads count their bytes.
  const uint32_t full_c = kPair ? mapa_shared(smem_u32(&full[0]), 0) : 0u;

  if (warp == (kFused ? kProtoWarp : 0)) {
    // ---------------------------------------------------------- A issuer / protocol
    // The barrier GEMM's warp 0 issues its A loads here.  In the fused kernel
    // this warp runs the ready-flag protocol and hands each chunk's decision
    // to the A loader (warp 0) as a descriptor, so that flag reads, waits,
    // fences and hand-offs never delay a load.
    if (kFused && p.l2_prefetch) {
      // Small A (the host's choice): every CTA first asks L2 for its share of
      // the shards' rows, so that the owners' and copiers' first reads of A
      // hit L2, as the GEMM's do after the barrier path's gather.  Pieces of
      // 32 KB, in bounds of each shard, 16-byte aligned (K % 8 == 0).
      const int rows_per = (p.M + (int)gridDim.x - 1) / (int)gridDim.x;
      int r0 = min(p.M, (int)blockIdx.x * rows_per);
      const int r1 = min(p.M, r0 + rows_per);
      while (r0 < r1) {
        const int s = r0 / p.mps;
        const int lr = r0 - s * p.mps;
        const int n = min(r1 - r0, p.mps - lr);
        const char* base = reinterpret_cast<const char*>(p.shards[s] + (int64_t)lr * p.K);
        const int64_t bytes = (int64_t)n * p.K * 2;
        for (int64_t off = (int64_t)lane * 32768; off < bytes; off += 32 * 32768)
          prefetch_l2_bulk(base + off, (uint32_t)(bytes - off < 32768 ? bytes - off : 32768));
        r0 += n;
      }
    }
    if (lane == 0) {
      ARing ar;             // barrier GEMM: the A loads issued here
      bool aborted = false;
      int seq = 0;          // boxes so far (fused: handed to the A loader)
      int rslot = 0;        // fused: next ring slot for a chunk record
      uint32_t rphase = 0;  // ... and the parity of its use
      // Chunk cursor over this CTA's (tile, k-group) sequence.  Tile (mb, nb)
      // owns the window [chunk_start(nb), chunk_start(nb + 1)) and visits it
      // first (chunk_at).  Everything that needs a
      // division is computed once per tile; a chunk costs a few adds.  A
      // follower's flag is read one chunk ahead, so its latency overlaps the
      // current chunk's loads.
      //
      // Staging ahead (fused): while it works on a tile, the protocol hands the
      // window of its next tile (nxt) to the copiers, one chunk per chunk it
      // issues and only when a ring slot is free at once, so that tile's
      // followers in other CTAs find those chunks published early.  `pre`
      // counts the chunks of nxt handed so far (window order), `cur_pre`
      // those of the current tile, which it then loads without staging.  The
      // hand-off starts at position p.stage_from of the current tile (the
      // plan sets it three quarters through for calls of four or more waves), so
      // the staged copy is still in L2 when the next wave reads it.  The
      // next tile is marked started only once its whole window is handed:
      // until then a follower may still take its chunks over, as for any
      // tile that has not started.
      TileCtx cur, nxt;
      int t = blockIdx.x, gi = 0;
      int pre = 0, cur_pre = 0;
      uint64_t cur_peek = 0;
      int dslot = 0;        // fused: next descriptor slot
      uint32_t dphase = 0;  // ... and the parity of its use
      if (t < p.num_tiles) {
        tile_ctx<kFused>(p, t, cur);
        const int g0 = order_at(p, 0, cur.ws, cur.we);
        if ((kAllStaged && !cur.pair_local)
                ? cur.kind != kEmpty
                : (cur.kind != kLocal && cur.kind != kEmpty && !cur.owns(g0)))
          if (flag_ok(p, cur.mb * p.G + g0)) cur_peek = ld_relaxed_gpu(p.flags + cur.mb * p.G + g0);
        if (t + (int)gridDim.x < p.num_tiles) tile_ctx<kFused>(p, t + gridDim.x, nxt);
      }
      const int last_nbox = chunk_boxes(p, p.G - 1);
      // A CTA that runs the fetch prologue loads nothing (A here, B in the B
      // loader) before it is through (the copies have the SM to themselves).
      if (kFused && !kLayoutM && p.pro_cta0 >= 0 && (int)blockIdx.x >= p.pro_cta0 &&
          !wait_bar(p, pro_bar, 0u, abort_flag, kSitePro))
        aborted = true;
      while (t < p.num_tiles && !aborted) {
        const uint64_t t_chunk = p.trace ? globaltimer_ns() : 0;
        if (kFused && gi == 0) {
          // Before any load of the tile: hand the rest of its owned window to
          // the copiers, then mark the tile started.  A follower waits
          // (instead of taking a chunk over) only on a started owner, and
          // handed chunks are published whatever this CTA's pipeline does --
          // with CTA pairs that pipeline also waits on the partner CTA.
          if (cur.kind == kLocal || cur.kind == kDirect) {
            const uint32_t wbits =
                (cur.kind == kDirect || (kAllStaged && !cur.pair_local)) ? (kInfoStage | kInfoPublish)
                                                                         : kInfoStage;
            for (int wg = cur.ws + cur_pre; wg < cur.we; ++wg) {
              if (!wait_bar(p, &rfree[rslot], rphase ^ 1u, abort_flag, kSiteRing)) {
                aborted = true;
                break;
              }
              hand_chunk(ring + rslot * kRingWords, &rfull[rslot], wbits, cur.mb, wg,
                         chunk_boxes(p, wg), cur.mb * p.G + wg, seq, p);
              if (p.trace) {
                const uint64_t now = globaltimer_ns();
                trace_rec(p.trace, p.trace_words, kTraceClaim, cur.mb, wg, now, now);
              }
              if (++rslot == kRing) {
                rslot = 0;
                rphase ^= 1u;
              }
            }
            if (aborted) break;
          }
          if (dbg_ok(p, t < p.started_words, kDbgStarted, t)) st_relaxed_gpu(p.started + t, p.epoch);
        }
        const int g = order_at(p, gi, cur.ws, cur.we);
        const int mb = cur.mb;
        const int flag_idx = mb * p.G + g;
        const int nbox = g == p.G - 1 ? last_nbox : p.kpf;
        const int kind = cur.kind;
        bool direct = false;  // A straight from a shard (else from the staging)
        bool need_fence = false;
        uint32_t bits = 0;
        if (kFused) {
          // A window chunk staged ahead is read like a follower's: from the
          // staging its copiers wrote a tile ago (still in L2), not again from
          // the shard.
          // (Owned chunks were handed to the copiers at the tile start.)
          const bool staged_ahead = cur.owns(g) && g - cur.ws < cur_pre;
          if (kind == kLocal && (!kAllStaged || cur.pair_local)) {
            direct = true;
          } else if (kind == kEmpty) {
            // rows past M: the gathered copy's maps read zeros there
          } else if (kind == kDirect && cur.owns(g) && !staged_ahead && !kAllStaged) {
            direct = true;
          } else {
            const uint64_t target = p.fbase + (uint64_t)nbox;
            if (cur_peek >= target) {
              fence_acquire_gpu();  // the relaxed read saw it published: make it an acquire
            } else {
              const uint64_t t0 = p.trace ? globaltimer_ns() : 0;
              // (with the fetch prologue nobody owns a chunk: wait only)
              const int owner_tile =
                  p.pro_cta0 < 0 && (kind == kDirect || (kAllStaged && kind == kLocal))
                      ? tile_index(p, mb, owner_nb(p, g)) : -1;
              if (wait_or_take(p, flag_idx, target, owner_tile)) {
                if constexpr (kAllStaged) {
                  // Taken over: have it staged here, then read it like anyone else.
                  if (!wait_bar(p, &rfree[rslot], rphase ^ 1u, abort_flag, kSiteRing)) {
                    aborted = true;
                    break;
                  }
                  hand_chunk(ring + rslot * kRingWords, &rfull[rslot], kInfoStage | kInfoPublish,
                             mb, g, nbox, flag_idx, seq, p);
                  if (++rslot == kRing) {
                    rslot = 0;
                    rphase ^= 1u;
                  }
                  if (p.trace) {
                    const uint64_t now = globaltimer_ns();
                    trace_rec(p.trace, p.trace_words, kTraceClaim, mb, g, now, now);
                  }
                  wait_or_take(p, flag_idx, target, -1);
                } else {
                  direct = true;
                  bits = kInfoStage | kInfoPublish;
                }
              }
              if (p.trace) trace_rec(p.trace, p.trace_words, kTraceWait, mb, g, t0, globaltimer_ns());
            }
            // The loader orders this acquire before its TMA loads of the
            // staged data with a proxy fence.
            need_fence = !direct;
          }
          if ((bits & kInfoStage) && p.trace) {
            const uint64_t now = globaltimer_ns();
            trace_rec(p.trace, p.trace_words, kTraceClaim, mb, g, now, now);
          }
        }
        if (kFused && (bits & kInfoStage)) {
          // A chunk taken over: hand it to the copiers.
          if (!wait_bar(p, &rfree[rslot], rphase ^ 1u, abort_flag, kSiteRing)) {
            aborted = true;
            break;
          }
          hand_chunk(ring + rslot * kRingWords, &rfull[rslot], bits, mb, g, nbox, flag_idx, seq, p);
          if (++rslot == kRing) {
            rslot = 0;
            rphase ^= 1u;
          }
        }
        if (!direct && kLayoutM) bits |= kInfoAmn;

        // Next chunk in sequence.  Only a follower chunk reads its flag; owner
        // and local chunks never touch it, so the protocol never stalls on a
        // load it does not need.
        int nt = t, ngi = gi + 1;
        bool new_tile = false;
        if (ngi == p.G) {
          ngi = 0;
          nt += gridDim.x;
          new_tile = true;
        }
        // (scalar selects, not a reference: the cursor must stay in registers)
        const int n_mb = new_tile ? nxt.mb : cur.mb;
        const int n_kind = new_tile ? nxt.kind : cur.kind;
        const int n_ws = new_tile ? nxt.ws : cur.ws;
        const int n_we = new_tile ? nxt.we : cur.we;
        const bool n_pl = new_tile ? nxt.pair_local : cur.pair_local;
        // (staging ahead does not run on a tile's last chunk, so pre is final here)
        const int n_pre = new_tile ? pre : cur_pre;
        uint64_t nxt_peek = 0;
        bool nxt_follow = false;
        if (kFused && nt < p.num_tiles) {
          const int ng = order_at(p, ngi, n_ws, n_we);
          nxt_follow = (kAllStaged && !n_pl)
                           ? n_kind != kEmpty
                           : (n_kind != kLocal && n_kind != kEmpty &&
                                     !(n_kind == kDirect && ng >= n_ws && ng < n_we &&
                                       ng - n_ws >= n_pre));
          if (nxt_follow && flag_ok(p, n_mb * p.G + ng))
            nxt_peek = ld_relaxed_gpu(p.flags + n_mb * p.G + ng);
        }

        if constexpr (kFused) {
          // Hand the chunk to the A loader (warp 0).
          if (!wait_bar(p, &dfree[dslot], dphase ^ 1u, abort_flag, kSiteDesc)) {
            aborted = true;
            break;
          }
          uint32_t* d = dring + dslot * 4;
          d[0] = (direct ? kDescDirect : 0u) | (cur.one_shard ? kDescOneShard : 0u) |
                 (need_fence ? kDescFence : 0u) | (bits << 8);
          d[1] = (uint32_t)mb;
          d[2] = (uint32_t)g | ((uint32_t)nbox << 16);
          d[3] = (uint32_t)cur.r0;
          mbar_arrive(&dfull[dslot]);  // (release: the loader reads the record after its wait)
          if (++dslot == kDRing) {
            dslot = 0;
            dphase ^= 1u;
          }
          seq += nbox;
        } else {
          if (!a_chunk_loads<kPair, kFused, kLayoutM>(p, ar, smem, full, empty, info, full_c, rank,
                                                       abort_flag, bits, direct, cur.one_shard,
                                                       cur.r0, mb, g * p.kpf, nbox, cur.sy,
                                                       cur.sd)) {
            aborted = true;
            break;
          }
          seq += nbox;
        }
        if (p.trace)  // b: k-group | 1 << 16 if loaded from a shard | 2 << 16 if staged here
          trace_rec(p.trace, p.trace_words, kTraceIssue, mb,
                    (uint32_t)g | (direct ? 1u << 16 : 0u) | ((bits & kInfoStage) ? 2u << 16 : 0u),
                    t_chunk, globaltimer_ns());
        if (kFused && !new_tile && t + (int)gridDim.x < p.num_tiles &&
            (nxt.kind == kLocal || nxt.kind == kDirect) && pre < nxt.we - nxt.ws &&
            gi >= p.stage_from &&
            mbar_test_wait(&rfree[rslot], rphase ^ 1u)) {
          // Stage ahead: one chunk of the next tile's window.
          const int pg = nxt.ws + pre;
          hand_chunk(ring + rslot * kRingWords, &rfull[rslot],
                     kInfoStage | ((nxt.kind == kDirect || (kAllStaged && !nxt.pair_local))
                                       ? kInfoPublish : 0u), nxt.mb, pg,
                     chunk_boxes(p, pg), nxt.mb * p.G + pg, seq, p);
          if (p.trace) {
            const uint64_t now = globaltimer_ns();
            trace_rec(p.trace, p.trace_words, kTraceClaim, nxt.mb, pg, now, now);
          }
          if (++rslot == kRing) {
            rslot = 0;
            rphase ^= 1u;
          }
          if (++pre == nxt.we - nxt.ws &&
              dbg_ok(p, t + (int)gridDim.x < p.started_words, kDbgStarted, t + (int)gridDim.x))
            st_relaxed_gpu(p.started + t + gridDim.x, p.epoch);
        }
        t = nt;
        gi = ngi;
        if (new_tile) {
          cur = nxt;
          cur_pre = pre;
          pre = 0;
          if (t + (int)gridDim.x < p.num_tiles) tile_ctx<kFused>(p, t + gridDim.x, nxt);
        }
        if (nxt_follow) cur_peek = nxt_peek;
        if (kFused) *iseq = (uint32_t)seq;
      }
      if constexpr (kFused) {
        // End of stream, for the A loader and for the copiers (if a slot does
        // not free, the abort flag is set and they leave on it).
        if (wait_bar(p, &dfree[dslot], dphase ^ 1u, abort_flag, kSiteDesc)) {
          dring[dslot * 4] = kDescEnd;
          mbar_arrive(&dfull[dslot]);
        }
        if (wait_bar(p, &rfree[rslot], rphase ^ 1u, abort_flag, kSiteRing)) {
          ring[rslot * kRingWords] = kInfoEnd;
          mbar_arrive(&rfull[rslot]);
        }
      } else {
        if (aborted || *abort_flag) drain_loads<kPair>(full, ar.issued_mask, ar.issued_parity, rank);
      }
    }
    __syncwarp();
  } else if (kFused && warp == 0) {
    // ---------------------------------------------------------- A loader (fused)
    // Takes the protocol warp's chunk descriptors in order and issues each
    // chunk's A loads.  A descriptor marked kDescFence follows the protocol
    // warp's acquire of the chunk's ready flag; the descriptor barrier carries
    // that acquire here (release/acquire at CTA scope), and the proxy fence
    // then orders it before the TMA loads of the staged data.
    if (lane == 0) {
      ARing ar;
      bool aborted = false;
      int dslot = 0;
      uint32_t dphase = 0;
      for (;;) {
        if (!wait_bar(p, &dfull[dslot], dphase, abort_flag, kSiteDesc)) {
          aborted = true;
          break;
        }
        const uint32_t* d = dring + dslot * 4;
        const uint32_t d0 = d[0], d1 = d[1], d2 = d[2], d3 = d[3];
        mbar_arrive(&dfree[dslot]);
        if (++dslot == kDRing) {
          dslot = 0;
          dphase ^= 1u;
        }
        if (d0 & kDescEnd) break;
        if (d0 & kDescFence) fence_proxy_async_global();
        const int mb = (int)d1, g = (int)(d2 & 0xFFFFu), nbox = (int)(d2 >> 16);
        if (!a_chunk_loads<kPair, kFused, kLayoutM>(p, ar, smem, full, empty, info, full_c, rank,
                                                     abort_flag, d0 >> 8, (d0 & kDescDirect) != 0,
                                                     (d0 & kDescOneShard) != 0, (int)d3, mb,
                                                     g * p.kpf, nbox, 0, 0)) {
          aborted = true;
          break;
        }
      }
      if (aborted || *abort_flag) drain_loads<kPair>(full, ar.issued_mask, ar.issued_parity, rank);
    }
    __syncwarp();
  } else if (warp == 1 && kPair && rank != 0) {
    // ---------------------------------------------------------- pair peer
    // Nothing to do: the leader issues the pair's MMAs, and this CTA's loads
    // count their bytes on the leader's barriers themselves.
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs this loop in step (waits are voted, so every lane
    // takes the same branch); one elected lane issues each MMA and commit.
    {
      const uint32_t ab_bf16 = p.fp16 ? 0u : 1u;
      constexpr uint32_t kM = kPair ? 2 * kBM : kBM;
      const uint32_t idesc_k = kF8 ? idesc_e4m3_f32(kM, kBN) : idesc_f16_f32(ab_bf16, 0, 1, kM, kBN);
      const uint32_t idesc_mn = idesc_f16_f32(ab_bf16, 1, 1, kM, kBN);
      // A's major-ness: K-major for the k-contiguous layout, MN-major for the
      // [K, M] staging.  The single-CTA fused m-contiguous kernel mixes the two
      // per chunk (shard rows K-major) and reads it from the stage record; the
      // pair kernel decides per tile (K-major only for pairs wholly in the
      // local shard), so its loop reads no shared memory for it.
      constexpr int kAMajor = !kLayoutM ? 0 : (kFused && !kPair) ? 2 : 1;
      bool aborted = false;
      int stage = 0;
      uint32_t phase = 0;
      // The MMA issue queue is shallow: whatever this warp waits on between
      // two stages' MMAs idles the tensor pipe.  So the next stage's barrier
      // is tested (without blocking) right after this stage's MMAs and commit
      // are issued -- its latency then overlaps the queued MMAs -- and a
      // blocking wait happens only when that stage had not landed yet.  A
      // completed phase stays completed until the stage is refilled, which
      // needs this warp's commit, so a positive test also holds across a
      // tile boundary.
      bool ready = false;  // stage `stage` (phase `phase`) is known to have landed
      const int total = my_tiles * p.num_kb;
      int done = 0;
      for (int j = 0; j < my_tiles && !aborted; ++j) {
        const int buf = j & 1;
        const uint32_t use = (uint32_t)(j >> 1);
        bool tile_mn = kAMajor == 1;
        if constexpr (kAllStaged) {
          if (p.local_direct) {
            TileCtx tc;
            tile_ctx<true>(p, blockIdx.x + j * gridDim.x, tc);
            tile_mn = !tc.pair_local;
          }
        }
        if (!__all_sync(0xffffffffu, wait_bar<kPair>(p, &tmem_empty[buf], (use & 1u) ^ 1u,
                                                     abort_flag, kSiteTmemEmpty))) {
          aborted = true;
          break;
        }
        tcgen05_fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kBN);
        for (int kb = 0; kb < p.num_kb; ++kb, ++done) {
          if (!ready &&
              !__all_sync(0xffffffffu, wait_bar(p, &full[stage], phase, abort_flag, kSiteFull))) {
            aborted = true;
            break;
          }
          tcgen05_fence_after_sync();
          const int s1 = stage + 1 == kStages ? 0 : stage + 1;
          const uint32_t ph1 = stage + 1 == kStages ? phase ^ 1u : phase;
          const bool more = done + 1 < total;
          const bool a_mn = kAMajor == 2 ? (info[stage] & kInfoAmn) != 0 : tile_mn;
          const uint32_t idesc = a_mn ? idesc_mn : idesc_k;
          const uint32_t a_addr = smem_u32(smem + stage * kStageBytes);
          const uint32_t b_addr = a_addr + kAStageBytes;
          const uint64_t a_desc0 = a_mn ? smem_desc_sw128(a_addr, kMnChunkBytes, 1024)
                                        : smem_desc_sw128(a_addr, 16, 1024);
          const uint64_t b_desc0 = kF8 ? smem_desc_sw128(b_addr, 16, 1024)
                                       : smem_desc_sw128(b_addr, kMnChunkBytes, 1024);
          // Each k-slice of 16 elements moves a descriptor's start address by
          // 32 bytes (K-major: inside the swizzle row) or 2048 bytes (MN-major:
          // two 1024-byte groups of 8 k-rows), i.e. its address field
          // (address >> 4, 14 bits, no carry within the stage) by 2 or 128:
          // one add per MMA instead of rebuilding the descriptor.
          const uint64_t a_step = a_mn ? 128u : 2u;
          constexpr uint64_t b_step = kF8 ? 2u : 128u;
#pragma unroll
          for (int ks = 0; ks < kBK / kUmmaK; ++ks) {
            const uint64_t a_desc = a_desc0 + a_step * ks;
            const uint64_t b_desc = b_desc0 + b_step * ks;
            const uint32_t acc = (kb | ks) != 0 ? 1u : 0u;
            if constexpr (kF8 && kPair)
              umma_f8_pair(d_tmem, a_desc, b_desc, idesc, acc);
            else if constexpr (kF8)
              umma_f8(d_tmem, a_desc, b_desc, idesc, acc);
            else if constexpr (kPair)
              umma_f16_pair(d_tmem, a_desc, b_desc, idesc, acc);
            else
              umma_f16(d_tmem, a_desc, b_desc, idesc, acc);
          }
          if constexpr (kPair)
            umma_commit_pair_mc(&empty[stage], 3);  // frees the stage in both CTAs
          else
            umma_commit(&empty[stage]);
          const bool t_full = __all_sync(0xffffffffu, more && mbar_test_wait(&full[s1], ph1));
          stage = s1;
          phase = ph1;
          ready = t_full;
        }
        if (aborted) break;
        if constexpr (kPair)
          umma_commit_pair_mc(&tmem_full[buf], 3);
        else
          umma_commit(&tmem_full[buf]);
      }
      // All MMAs issued by this warp complete before TMEM is released.
      if constexpr (kPair)
        umma_commit_pair(drain);
      else
        umma_commit(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < 1000000000ull) {
      }
    }
    __syncwarp();
  } else if (warp < 2 + kEpiWarps) {
    // ---------------------------------------------------------- epilogue
    // (fetch prologue first: these warps have nothing to drain before it ends)
    if constexpr (kFused && !kLayoutM) fetch_prologue(p, kCopyWarps + warp - 2, lane, pro_bar);
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint8_t* my_bufs = epi_smem + (warp - 2) * kEpiBufs * kEpiBufBytes;
    const uint32_t my_bufs_u32 = smem_u32(my_bufs);
    int chunk_count = 0;
    for (int j = 0; j < my_tiles; ++j) {
      int mb, nb;
      tile_coords(p, blockIdx.x + j * gridDim.x, mb, nb);
      const int buf = j & 1;
      const uint32_t use = (uint32_t)(j >> 1);
      // Every lane waits; the vote keeps the warp converged for tcgen05.ld.
      const bool ok = wait_bar(p, &tmem_full[buf], use & 1u, abort_flag, kSiteTmemFull);
      if (!__all_sync(0xffffffffu, ok)) break;
      tcgen05_fence_after_sync();
      const uint64_t t0 = p.trace ? globaltimer_ns() : 0;
      int m0 = mb * kBM + q * kEpiRows, sd = 0, m_end = p.M;
      if (!kFused && p.seg_blocks) {  // segmented: rows within segment sd
        sd = mb / p.seg_blocks;
        m0 = (mb - sd * p.seg_blocks) * kBM + q * kEpiRows;
        m_end = sd < p.D ? p.seg_rows : 0;  // (a pair's half past the last segment)
      }
      const int n_tile = nb * kBN;
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kBN);
#pragma unroll 1
      for (int c = 0; c < kBN / kEpiCols; ++c) {
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(t_row + c * kEpiCols, r0);
        tmem_ld_32x32b_x32(t_row + c * kEpiCols + 32, r1);
        tmem_ld_wait();
        if (c == kBN / kEpiCols - 1) {
          // This warp has read its lanes of the accumulator (pair: the peer's
          // warps arrive on the leader's barrier).
          tcgen05_fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            if (kPair && rank != 0)
              mbar_arrive_remote(mapa_shared(smem_u32(&tmem_empty[buf]), 0));
            else
              mbar_arrive(&tmem_empty[buf]);
          }
        }
        const int n0 = n_tile + c * kEpiCols;
        uint32_t packed[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float v0 = __uint_as_float(r0[2 * i]), v1 = __uint_as_float(r0[2 * i + 1]);
          float w0 = __uint_as_float(r1[2 * i]), w1 = __uint_as_float(r1[2 * i + 1]);
          if constexpr (kF8) {
            v0 *= p.scale_ab;
            v1 *= p.scale_ab;
            w0 *= p.scale_ab;
            w1 *= p.scale_ab;
          }
          if (p.bias) {
            const int na = n0 + 2 * i, nb2 = n0 + 32 + 2 * i;
            v0 += na < p.N ? __ldg(p.bias + na) : 0.f;
            v1 += na + 1 < p.N ? __ldg(p.bias + na + 1) : 0.f;
            w0 += nb2 < p.N ? __ldg(p.bias + nb2) : 0.f;
            w1 += nb2 + 1 < p.N ? __ldg(p.bias + nb2 + 1) : 0.f;
          }
          packed[i] = pack2(v0, v1, p.fp16);
          packed[16 + i] = pack2(w0, w1, p.fp16);
        }
        const bool store = (m0 < m_end) && (n0 < p.N);
        const int eb = chunk_count & 1;
        if (lane == 0) bulk_wait_group_read<kEpiBufs - 1>();
        __syncwarp();
        const uint32_t row_addr = my_bufs_u32 + eb * kEpiBufBytes + lane * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          st_shared_v4(row_addr + ((ch ^ (lane & 7)) << 4), packed[4 * ch], packed[4 * ch + 1],
                       packed[4 * ch + 2], packed[4 * ch + 3]);
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0 && store) {
          if (!kFused && p.seg_blocks)
            tma_store_3d(&p.tm_out, my_bufs + eb * kEpiBufBytes, n0, m0, sd);
          else
            tma_store_2d(&p.tm_out, my_bufs + eb * kEpiBufBytes, n0, m0);
        }
        if (lane == 0) bulk_commit_group();
        ++chunk_count;
      }
      if (p.trace && lane == 0 && q == 0)
        trace_rec(p.trace, p.trace_words, kTraceTile, mb, nb, t0, globaltimer_ns());
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  } else if (warp == kBWarp) {
    // ---------------------------------------------------------- B loader
    // The tile's B k-blocks in the order of its A chunks (owned window first):
    // one thread issuing both operands' loads could not keep up with the
    // tensor pipe.  Each loader arrives on `full` for its own bytes.
    if (lane == 0) {
      uint32_t issued_mask = 0, issued_parity = 0;
      bool aborted = false;
      int stage = 0;
      uint32_t phase = 0;
      if (kFused && !kLayoutM && p.pro_cta0 >= 0 && (int)blockIdx.x >= p.pro_cta0 &&
          !wait_bar(p, pro_bar, 0u, abort_flag, kSitePro))
        aborted = true;
      for (int t = blockIdx.x; t < p.num_tiles && !aborted; t += gridDim.x) {
        int mb, nb;
        tile_coords(p, t, mb, nb);
        const int ws = kFused ? chunk_start(p, nb) : 0;
        const int we = kFused ? chunk_end(p, nb) : 0;
        const int n0 = nb * kBN + (int)rank * P::kBCols;  // this CTA's columns (pair: the rank's half)
        for (int gi = 0; gi < p.G && !aborted; ++gi) {
          const int g = order_at(p, gi, ws, we);
          const int nbox = chunk_boxes(p, g);
          for (int j = 0; j < nbox; ++j) {
            const int kb = g * p.kpf + j;
            if (!wait_bar(p, &empty[stage], phase ^ 1u, abort_flag, kSiteEmpty)) {
              aborted = true;
              break;
            }
            uint8_t* b_dst = smem + stage * kStageBytes + kAStageBytes;
            const uint32_t bar_c = full_c + 8u * (uint32_t)stage;
            if (!kPair || rank == 0)
              mbar_arrive_expect_tx(&full[stage], kPair ? 2 * P::kBStageBytes : P::kBStageBytes);
            if constexpr (kF8) {
              // [N, K] rows: one box of this CTA's columns x 128 bytes of K
              stage_load_2d<kPair>(b_dst, &p.tm_b, &full[stage], bar_c, kb * kBK, n0);
            } else {
#pragma unroll
              for (int q = 0; q < P::kBCols / 64; ++q)
                stage_load_2d<kPair>(b_dst + q * kMnChunkBytes, &p.tm_b, &full[stage], bar_c,
                                     n0 + q * 64, kb * kBK);
            }
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (aborted || *abort_flag) drain_loads<kPair>(full, issued_mask, issued_parity, rank);
    }
    __syncwarp();
  } else if (kFused) {
    // ---------------------------------------------------------- copiers
    // Take the protocol warp's chunk records in order.  Box j of a chunk
    // whose first box has sequence index q goes to warp (q + j) % kCopyWarps,
    // so the boxes of consecutive chunks spread evenly over the warps.  A box is
    // copied in 8-row groups: lane = (row group, 16-byte column chunk), 8 rows
    // of 16 bytes per lane, two groups (16 loads) in flight; for the
    // m-contiguous layout a published box is also written transposed (8x8
    // register transposes) into the [K, M] staging.  Each warp that copied
    // boxes of a chunk then adds one to the record's done count (acq_rel, CTA
    // scope); the one that completes it publishes the chunk (release, GPU
    // scope), so the flag follows every copier's writes.
    const int w = warp - kCopyWarp0;
    if constexpr (!kLayoutM) fetch_prologue(p, w, lane, pro_bar);
    // The first copier also runs the register fetcher first: it copies the
    // chunks that TMA cannot load from a single shard (row blocks straddling
    // shards whose row count is not a multiple of 8) and publishes them; it
    // waits on nobody, so every such chunk is published whatever else runs.
    if (w == 0) regfetch_loop(p, lane, kLayoutM);
    const int ch = lane & 7;  // 16-byte column chunk of a 128-byte box row
    for (uint32_t n = 0;; ++n) {
      const int slot = (int)(n % kRing);
      const bool got = wait_handoff(p, &rfull[slot], n / kRing, iseq, abort_flag);
      if (!__all_sync(0xffffffffu, got)) break;
      uint32_t* rec = ring + slot * kRingWords;
      const uint32_t bits = rec[0];
      if (bits & kInfoEnd) break;
      const int mb = (int)rec[1], kb0 = (int)rec[2], nbox = (int)rec[3], flag_idx = (int)rec[4];
      const int q = (int)rec[5];
      const int j0 = (w - q % kCopyWarps + kCopyWarps) % kCopyWarps;
      const bool publish_m = kLayoutM && (bits & kInfoPublish);
      const int row0 = mb * kBM;
      for (int j = j0; j < nbox; j += kCopyWarps) {
        const int k = (kb0 + j) * kBK + ch * 8;
        if (k >= p.K) continue;  // K % 8 == 0: a column chunk is all in or all out
#pragma unroll 1
        for (int b = 0; b < 4; b += 2) {
          uint4 v[2][8];
          int m[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // Row group rg = 8 consecutive rows; with m_per_shard % 8 == 0 (or
            // a row block inside one shard) the group is inside one shard.
            m[h] = row0 + (4 * (b + h) + (lane >> 3)) * 8;
            const int nrow = min(8, p.M - m[h]);
            if (nrow > 0 && dbg_ok(p, m[h] >= 0, kDbgShardRow, m[h])) {
              const uint16_t* src = shard_row(p.shards, p.mps, p.K, m[h]) + k;
#pragma unroll
              for (int r = 0; r < 8; ++r)
                if (r < nrow) v[h][r] = ld_stream_v4(src + (int64_t)r * p.K);
            }
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int nrow = min(8, p.M - m[h]);
            if (!dbg_ok(p, m[h] >= 0 && k + 8 <= p.K, kDbgGathered, m[h])) continue;
#pragma unroll
            for (int r = 0; r < 8; ++r)
              if (r < nrow) st_v4(p.a_gathered + (int64_t)(m[h] + r) * p.K + k, v[h][r]);
            if (publish_m && nrow == 8 &&
                dbg_ok(p, m[h] + 8 <= p.M, kDbgStaging, m[h])) {  // M % 8 == 0 for this layout
#pragma unroll
              for (int c = 0; c < 8; ++c)
                st_v4(p.staging_mk + (int64_t)(k + c) * p.M + m[h], transpose_col(v[h], c));
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        if ((bits & kInfoPublish) && j0 < nbox) {
          const uint32_t done = atom_add_acq_rel_cta_shared(smem_u32(rec + 6), 1u) + 1u;
          if (done == (uint32_t)min(nbox, kCopyWarps) && flag_idx != p.inject_skip_flag &&
              flag_ok(p, flag_idx)) {
            inject_delay(p, flag_idx);
            st_release_gpu(p.flags + flag_idx, p.fbase + (uint64_t)nbox);
          }
        }
        mbar_arrive(&rfree[slot]);
      }
      __syncwarp();
    }
    __syncwarp();
  }

  tcgen05_fence_before_sync();
  __syncthreads();
  // Pair: neither CTA leaves (or frees TMEM) while the other may still signal
  // its barriers or the leader's MMAs may still write its TMEM.
  if (kPair) cluster_sync();
  tcgen05_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc<kPair>(tmem_base, kTmemCols);
  }
}

// Barrier-path gather: shard r is copied to rows [r*m_per_shard, ...) of
// a_gathered, restricted to gathered rows [row0, row1) and to local rows
// [loc0, loc1) of each shard (everything for the barrier baseline; for the
// chunked pipeline, chunk s's sub-block of every shard).  What a shard
// contributes is one contiguous block, so this is at most D flat copies;
// blockIdx.y selects the shard.
__global__ void __launch_bounds__(256) agmm_gather_kernel(const __grid_constant__ GatherParams gp) {
  const uint64_t t0 = gp.trace ? globaltimer_ns() : 0;
  const int s = blockIdx.y;
  const int64_t lo = max(max(0, gp.row0 - s * gp.mps), gp.loc0);
  const int64_t hi = min(min(gp.mps, gp.row1 - s * gp.mps), gp.loc1);
  if (hi <= lo) return;
  const int64_t vk = gp.K / 8;  // 16-byte vectors per row (K % 8 == 0)
  const uint4* src = reinterpret_cast<const uint4*>(gp.shards[s]) + lo * vk;
  uint4* dst = reinterpret_cast<uint4*>(gp.a_gathered) + ((int64_t)s * gp.mps + lo) * vk;
  const int64_t n = (hi - lo) * vk;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  constexpr int U = 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i + u * stride < n) v[u] = ld_stream_v4(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i + u * stride < n) st_v4(dst + i + u * stride, v[u]);
  }
  if (gp.trace && threadIdx.x == 0)
    trace_rec(gp.trace, gp.trace_words, kTraceGather, blockIdx.x + blockIdx.y * gridDim.x, 0, t0,
              globaltimer_ns());
}

// Barrier-path gather for the m-contiguous layout: a_gathered plus the [K, M]
// staging.  Thread -> one 8x8 block (8 rows x 8 columns); a warp covers 16
// consecutive row groups of two column groups so the transposed stores run
// along M.
__global__ void __launch_bounds__(256) agmm_gather_mk_kernel(const __grid_constant__ GatherParams gp) {
  const uint64_t t0 = gp.trace ? globaltimer_ns() : 0;
  const int nrg = gp.M >> 3, ncg = gp.K >> 3;
  const int64_t row_blocks = (nrg + 15) / 16, col_pairs = (ncg + 1) / 2;
  const int64_t total = row_blocks * col_pairs * 32;  // one thread per (16 x 2)-block slot
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t wi = idx >> 5;
    const int lane = (int)(idx & 31);
    const int64_t cp = wi / row_blocks;
    const int rg = (int)((wi - cp * row_blocks) * 16 + (lane & 15));
    const int cg = (int)(cp * 2 + (lane >> 4));
    if (rg >= nrg || cg >= ncg) continue;
    const int col = cg * 8;
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = ld_stream_v4(shard_row(gp.shards, gp.mps, gp.K, rg * 8 + i) + col);
#pragma unroll
    for (int i = 0; i < 8; ++i) st_v4(gp.a_gathered + (int64_t)(rg * 8 + i) * gp.K + col, v[i]);
#pragma unroll
    for (int c = 0; c < 8; ++c)
      st_v4(gp.staging_mk + (int64_t)(col + c) * gp.M + rg * 8, transpose_col(v, c));
  }
  if (gp.trace && threadIdx.x == 0)
    trace_rec(gp.trace, gp.trace_words, kTraceGather, blockIdx.x, 0, t0, globaltimer_ns());
}

}  // namespace agmm
