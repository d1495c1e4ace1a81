// Host side of libagmm: argument validation, workspace and epoch management,
// TMA tensor-map encoding and the kernel launches behind the C ABI declared in
// include/agmm.h.  Everything the operation computes runs in the kernels of
// kernels.cuh; this file only prepares and enqueues them.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "agmm.h"
#include "kernels.cuh"

using namespace agmm;

static_assert(AG_MAX_SHARDS == kMaxShards, "header and kernel shard limits differ");

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kDefaultTimeoutNs = 2000000000LL;
// Automatic flag granularity (k-blocks per flag), measured over the cube sweep
// and the Iris shapes.  When every tile fits in one wave of the grid, the
// followers wait on owners that all start together: K-blocks per column
// block, clamped to [4, 8] (one-wave cubes: 4; M=1024 with 128 K-blocks: 8).
// Otherwise 8 for the k-contiguous layout and 16 for the m-contiguous one
// (fewer flags: fewer waits, fences and copier hand-offs per tile; the
// owners' longer first chunks are covered by staging ahead).
constexpr int kAutoKpfOneWave = 4, kAutoKpfOneWaveMax = 8, kAutoKpfK = 8, kAutoKpfM = 16;
// A up to 12 MB is prefetched into L2 at the start of a fused call.  Measured
// (means, L2 flushed): cube_640 -0.8 us, cube_1024 -0.6 us, cube_2432 -1.1 us;
// at 16-34 MB (cube_2944, M=1024, cube_4096) it cost 0.7-2.6 us.
constexpr int64_t kL2PrefetchMaxBytes = 12ll << 20;

// log2 of the row count of the boxes that load a row block straddling shards:
// the largest of 64, 32, 16, 8 rows dividing m_per_shard (3 if none does; such
// blocks are then copied by the register fetcher instead).
int straddle_log2(int m_per_shard) {
  for (int l = 6; l > 3; --l)
    if (m_per_shard % (1 << l) == 0) return l;
  return 3;
}

// Granularity the workspace is sized for when k_per_flag is automatic: the
// finest automatic choice, so the flags fit whichever one a launch makes.
int sizing_k_per_flag(int num_kb) { return std::max(1, std::min(kAutoKpfOneWave, num_kb)); }

int auto_k_per_flag(int num_kb, int num_nb, bool one_wave, bool layout_m) {
  const int k = one_wave ? std::min(kAutoKpfOneWaveMax,
                                    std::max(kAutoKpfOneWave, num_kb / std::max(1, num_nb)))
                         : (layout_m ? kAutoKpfM : kAutoKpfK);
  return std::max(1, std::min(k, num_kb));
}

thread_local char t_cuda_msg[320] = "no CUDA error recorded on this thread";

int cuda_fail(cudaError_t e, const char* what) {
  snprintf(t_cuda_msg, sizeof t_cuda_msg, "%s failed: %s (%s)", what, cudaGetErrorName(e),
           cudaGetErrorString(e));
  return AG_ERR_CUDA;
}

#define AG_CK(call)                                     \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Library-owned state, one per device.
struct DevState {
  bool init = false;
  bool supported = false;
  int sms = 0;
  int pair_clusters = 0;  // CTA pairs of the pair kernels that fit on the GPU at once
  unsigned long long* err = nullptr;  // [2] device error word
  // chunked pipeline: its streams and fork/join events (created on first use)
  static constexpr int kChunkStreams = 4;
  bool chunk_init = false;
  cudaStream_t cstream[kChunkStreams] = {};
  cudaEvent_t fork_ev = nullptr, join_ev[kChunkStreams] = {};
  uint64_t* flags = nullptr;
  size_t flags_cap = 0;  // words
  uint16_t* staging = nullptr;
  size_t staging_cap = 0;  // elements
  uint64_t reported_epoch = 0;
  // Overlap detection on the library workspace: the stream of the last call
  // that used it and an event recorded on that stream after the call.
  cudaEvent_t ws_done = nullptr;
  cudaStream_t ws_stream = nullptr;
  bool ws_used = false;
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];
// One epoch counter for the whole process: flags in any workspace on any
// device compare against it, so a workspace never needs clearing between calls.
std::atomic<uint64_t> g_epoch{0};

struct Shape {
  int D, mps, K, N;
  int64_t M;
  int num_mb, num_nb, num_kb, kpf, G;
};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
  uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bn && y < x + an;
}

// Tile options: only the compiled shapes.  128-row tiles run on single CTAs
// with 4 stages, 256-row tiles on CTA pairs with 6 (Pipe<>), both 256 columns
// wide, 64 16-bit elements (128 FP8 bytes) per stage, 4 copier warps.
constexpr int kStagesSingle = 4, kStagesPair = 6;
constexpr int kSingleMaxKb = 32;  // automatic single CTAs: K up to 32 k-blocks, one wave
static_assert(Pipe<false>::kStages == kStagesSingle && Pipe<true>::kStages == kStagesPair,
              "tile options and compiled pipelines differ");
int check_tile_options(const ag_options& o) {
  if (o.block_m < 0 || o.block_n < 0 || o.block_k < 0 || o.stages < 0 || o.producer_warps < 0)
    return AG_ERR_INVALID_ARG;
  const int bk = o.dtype == AG_DTYPE_FP8_E4M3 ? 2 * kBK : kBK;
  if ((o.block_m && o.block_m != kBM && o.block_m != 2 * kBM) || (o.block_n && o.block_n != kBN) ||
      (o.block_k && o.block_k != bk) || (o.producer_warps && o.producer_warps != kCopyWarps))
    return AG_ERR_UNSUPPORTED;
  if (o.stages && o.stages != kStagesSingle && o.stages != kStagesPair) return AG_ERR_UNSUPPORTED;
  if (o.stages && o.block_m &&
      (o.stages == kStagesPair) != (o.block_m == 2 * kBM))
    return AG_ERR_UNSUPPORTED;
  return AG_OK;
}

// Sizes and options (no pointers, no CUDA call).  Fills `sh`.
int shape_of(int D, int m_per_shard, int K, int N, const ag_options& o, Shape* sh) {
  if (D < 1 || m_per_shard < 1 || K < 8 || N < 8) return AG_ERR_INVALID_ARG;
  if (K % 8 || N % 8) return AG_ERR_INVALID_ARG;
  if (D > AG_MAX_SHARDS) return AG_ERR_UNSUPPORTED;
  const int64_t M = (int64_t)D * m_per_shard;
  if (M > INT32_MAX) return AG_ERR_INVALID_ARG;
  if (o.dtype != AG_DTYPE_BF16 && o.dtype != AG_DTYPE_FP16 && o.dtype != AG_DTYPE_FP8_E4M3)
    return AG_ERR_INVALID_ARG;
  if (o.dtype == AG_DTYPE_FP8_E4M3) {
    if (!std::isfinite(o.scale_a) || !std::isfinite(o.scale_b)) return AG_ERR_INVALID_ARG;
    if (o.layout != AG_LAYOUT_K_CONTIGUOUS) return AG_ERR_UNSUPPORTED;
  }
  if (o.layout != AG_LAYOUT_K_CONTIGUOUS && o.layout != AG_LAYOUT_M_CONTIGUOUS)
    return AG_ERR_INVALID_ARG;
  if (o.rank < 0 || o.rank >= D) return AG_ERR_INVALID_ARG;
  if (o.k_per_flag < 0 || o.k_per_flag > 65536 || o.num_sms < 0 || o.timeout_ns < 0 ||
      o.trace_words < 0 || o.workspace_bytes < 0)
    return AG_ERR_INVALID_ARG;
  if (o.trace && (o.trace_words < 1 || !aligned(o.trace, 8))) return AG_ERR_INVALID_ARG;
  if (o.inject_delay_ns < 0 ||
      o.inject_delay_ns > (o.timeout_ns ? o.timeout_ns : kDefaultTimeoutNs) / 16)
    return AG_ERR_INVALID_ARG;
  if (int st = check_tile_options(o)) return st;
  if (o.layout == AG_LAYOUT_M_CONTIGUOUS && (M % 8)) return AG_ERR_UNSUPPORTED;
  sh->D = D;
  sh->mps = m_per_shard;
  sh->K = K;
  sh->N = N;
  sh->M = M;
  sh->num_mb = (int)((M + kBM - 1) / kBM);
  sh->num_nb = (N + kBN - 1) / kBN;
  sh->num_kb = (K + kBK - 1) / kBK;
  sh->kpf = o.k_per_flag ? o.k_per_flag : sizing_k_per_flag(sh->num_kb);
  sh->G = (sh->num_kb + sh->kpf - 1) / sh->kpf;
  if ((int64_t)sh->num_mb * sh->num_nb > INT32_MAX || (int64_t)sh->num_mb * sh->G > 0xFFFFFF)
    return AG_ERR_UNSUPPORTED;
  return AG_OK;
}

// Validation that needs no CUDA call.  Fills `sh`.
int validate(const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
             const void* bias, void* a_gathered, void* out, const ag_options& o, bool fused,
             Shape* sh) {
  (void)fused;
  if (!a_shards || !b || !a_gathered || !out) return AG_ERR_INVALID_ARG;
  int st = shape_of(D, m_per_shard, K, N, o, sh);
  if (st != AG_OK) return st;
  const int64_t M = sh->M;
  if (!aligned(b, 16) || !aligned(a_gathered, 16) || !aligned(out, 16)) return AG_ERR_INVALID_ARG;
  if (bias && !aligned(bias, 4)) return AG_ERR_INVALID_ARG;
  const size_t shard_bytes = (size_t)m_per_shard * K * 2;
  const size_t ag_bytes = (size_t)M * K * 2, out_bytes = (size_t)M * N * 2;
  const size_t b_bytes = (size_t)K * N * 2, bias_bytes = (size_t)N * 4;
  for (int r = 0; r < D; ++r) {
    if (!a_shards[r] || !aligned(a_shards[r], 16)) return AG_ERR_INVALID_ARG;
    if (overlaps(a_shards[r], shard_bytes, a_gathered, ag_bytes) ||
        overlaps(a_shards[r], shard_bytes, out, out_bytes))
      return AG_ERR_INVALID_ARG;
  }
  if (overlaps(a_gathered, ag_bytes, out, out_bytes) || overlaps(b, b_bytes, a_gathered, ag_bytes) ||
      overlaps(b, b_bytes, out, out_bytes))
    return AG_ERR_INVALID_ARG;
  if (bias && (overlaps(bias, bias_bytes, a_gathered, ag_bytes) ||
               overlaps(bias, bias_bytes, out, out_bytes)))
    return AG_ERR_INVALID_ARG;
  return AG_OK;
}

size_t round_kib(size_t n) { return (n + 1023) & ~size_t(1023); }

// Column blocks per schedule pass (see tile_coords).  A grid that runs every
// tile in one wave gains nothing from passes; otherwise a pass keeps its
// slice of b (K x 256 columns x 2 bytes per column block) near 32 MB so it
// stays in L2 while A streams past.  Measured at N=3584, K=8192 (8 of 14
// column blocks per pass): at M=16384 it ties one pass and beats 4 or 7 per
// pass (7 costs the m-contiguous kernel 6%); at M=4096 m-contiguous it beats
// one pass by 5%.
int schedule_group(const Shape& s, int sms) {
  if ((int64_t)s.num_mb * s.num_nb <= sms) return s.num_nb;
  const int64_t slice = (int64_t)s.K * kBN * 2;
  const int ng = (int)std::max<int64_t>(1, (32ll << 20) / slice);
  return std::min(ng, s.num_nb);
}

// Fused-path metadata: ready flags [num_mb * G], then the per-tile started
// words [num_mb * num_nb]; both 8 bytes each.
size_t flags_region(const Shape& s) { return round_kib((size_t)s.num_mb * s.G * 8); }
// Flags, then one "started" word per tile slot (CTA pairs: an odd row-block
// count adds a slot per column block).
size_t flags_bytes(const Shape& s) {
  return flags_region(s) + round_kib((size_t)(s.num_mb + 1) * s.num_nb * 8);
}

// Device pointers must be device (or managed) memory of the current device:
// a host pointer handed to a kernel would fault.
int check_device_ptr(const void* p, int dev) {
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return AG_ERR_INVALID_ARG;
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return AG_ERR_INVALID_ARG;
  if (at.type == cudaMemoryTypeDevice && at.device != dev) return AG_ERR_INVALID_ARG;
  return AG_OK;
}

// Number of CTA pairs of the pair kernels that can be resident at once (0 if
// a cluster launch is not possible).  A cluster's two CTAs need two free SMs
// of one GPC; with 1 CTA per SM not every SM pairs up, and a persistent grid
// larger than what fits at once would leave the extra clusters for a second
// wave.  Allocates nothing.
int query_pair_clusters(int sms, int* clusters) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sms & ~1));
  cfg.blockDim = dim3((unsigned)mode_threads(kFusedK));
  cfg.dynamicSmemBytes = Pipe<true>::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  *clusters = 0;
  AG_CK(cudaOccupancyMaxActiveClusters(clusters, agmm_gemm_kernel<kFusedK, true, false>, &cfg));
  return AG_OK;
}

int device_init(DevState& ds, int dev) {
  if (ds.init) return ds.supported ? AG_OK : AG_ERR_UNSUPPORTED;
  int major = 0, minor = 0, sms = 0;
  AG_CK(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
  AG_CK(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
  AG_CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  ds.sms = sms;
  // The kernels are built for sm_103a only; a missing image is "unsupported".
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, agmm_gemm_kernel<kFusedK, false, false>) != cudaSuccess || major != 10) {
    cudaGetLastError();
    ds.init = true;
    ds.supported = false;
    return AG_ERR_UNSUPPORTED;
  }
  constexpr int kSmem1 = Pipe<false>::kSmemBytes, kSmem2 = Pipe<true>::kSmemBytes;
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kGemmK, false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem1));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kGemmM, false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem1));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kFusedK, false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem1));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kFusedM, false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem1));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kGemmK, true, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem2));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kGemmM, true, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem2));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kFusedK, true, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem2));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kFusedM, true, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem2));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kGemmK, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem1));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kFusedK, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem1));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kGemmK, true, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem2));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kFusedK, true, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem2));
  if (int st = query_pair_clusters(sms, &ds.pair_clusters)) return st;
  AG_CK(cudaEventCreateWithFlags(&ds.ws_done, cudaEventDisableTiming));
  AG_CK(cudaMalloc(&ds.err, 2 * sizeof(unsigned long long)));
  AG_CK(cudaMemset(ds.err, 0, 2 * sizeof(unsigned long long)));
  ds.init = true;
  ds.supported = true;
  return AG_OK;
}

// A call about to use the library workspace on `stream`: AG_ERR_BUSY while
// the last call that used it was made on another stream and has not finished
// (its event has not completed).  Same-stream calls are ordered by the stream.
// While `stream` is being captured nothing runs, so nothing is checked or
// recorded.
bool capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return cs != cudaStreamCaptureStatusNone;
}

int check_busy(DevState& ds, cudaStream_t stream) {
  if (!ds.ws_used || ds.ws_stream == stream || capturing(stream)) return AG_OK;
  const cudaError_t q = cudaEventQuery(ds.ws_done);
  if (q == cudaErrorNotReady) {
    cudaGetLastError();
    return AG_ERR_BUSY;
  }
  if (q != cudaSuccess) return cuda_fail(q, "cudaEventQuery (workspace in use?)");
  return AG_OK;
}

// After a successful launch that used the library workspace.
int mark_busy(DevState& ds, cudaStream_t stream) {
  if (capturing(stream)) return AG_OK;
  AG_CK(cudaEventRecord(ds.ws_done, stream));
  ds.ws_stream = stream;
  ds.ws_used = true;
  return AG_OK;
}

int grow_workspace(DevState& ds, const Shape& s, bool need_flags, bool need_staging,
                   cudaStream_t stream) {
  const size_t words = need_flags ? flags_bytes(s) / 8 : 0;
  const size_t stage_elems = need_staging ? (size_t)s.K * s.M : 0;
  if (words > ds.flags_cap || stage_elems > ds.staging_cap) {
    // Older calls may still use the old buffers.
    AG_CK(cudaDeviceSynchronize());
  }
  if (words > ds.flags_cap) {
    if (ds.flags) AG_CK(cudaFree(ds.flags));
    ds.flags = nullptr;
    ds.flags_cap = 0;
    AG_CK(cudaMalloc(&ds.flags, words * 8));
    AG_CK(cudaMemsetAsync(ds.flags, 0, words * 8, stream));
    ds.flags_cap = words;
  }
  if (stage_elems > ds.staging_cap) {
    if (ds.staging) AG_CK(cudaFree(ds.staging));
    ds.staging = nullptr;
    ds.staging_cap = 0;
    AG_CK(cudaMalloc(&ds.staging, stage_elems * 2));
    ds.staging_cap = stage_elems;
  }
  return AG_OK;
}

// The launch plan shared by every entry point: CTA pairs (256 x 256 tiles)
// whenever two SMs are allowed, unless the tile options ask for 128-row
// tiles; the schedule; the automatic k_per_flag (the workspace is sized for
// s.G, which is >= the automatic choice's G).  Fills the schedule fields of p
// and *grid (CTAs; even for pairs).  The options were checked by
// check_tile_options; 256-row tiles on a grid without a CTA pair are
// AG_ERR_UNSUPPORTED.
int plan_launch(GemmParams& p, const Shape& s, int cap, int pair_clusters, bool fused,
                bool layout_m, const ag_options& o, int* grid) {
  const int k_per_flag = o.k_per_flag, rank = o.rank;
  const bool want_single = o.block_m == kBM || o.stages == kStagesSingle;
  const bool want_pair = o.block_m == 2 * kBM || o.stages == kStagesPair;
  const bool can_pair = cap >= 2 && pair_clusters >= 1;
  if (want_pair && !can_pair) return AG_ERR_UNSUPPORTED;
  // Automatic tile shape: CTA pairs, except for short calls -- K of at most
  // kSingleMaxKb k-blocks with every 128-row tile in one wave of the grid --
  // which run on single CTAs: there the start-up of a cluster launch weighs
  // more than the pair's halved B traffic.  Measured (means, L2 flushed), on
  // the one-wave cubes n = 256 ... 2048 single CTAs were 1.5-2 us faster for
  // the fused call and the barrier GEMM alike (cube_1024: fused 21.3 -> 19.6,
  // barrier 22.0 -> 19.9 us); at M=1024 N=3584 K=8192 (one wave either way)
  // pairs stayed faster (fused 57.7 vs 62.3 us).
  const bool short_one_wave =
      s.num_kb <= kSingleMaxKb && (int64_t)s.num_mb * s.num_nb <= (int64_t)cap;
  const bool pair = can_pair && !want_single && (want_pair || !short_one_wave);
  Shape sched = s;
  sched.num_mb = pair ? (s.num_mb + 1) / 2 : s.num_mb;
  const int units = pair ? std::min(cap / 2, pair_clusters) : cap;  // CTAs, or CTA pairs
  p.pair = pair ? 1 : 0;
  p.sched_mb = sched.num_mb;
  p.num_tiles = (sched.num_mb * s.num_nb) << p.pair;
  p.kpf = k_per_flag ? s.kpf
                     : auto_k_per_flag(s.num_kb, s.num_nb,
                                       (int64_t)sched.num_mb * s.num_nb <= units, layout_m);
  p.G = (s.num_kb + p.kpf - 1) / p.kpf;
  // schedule rows start at the local shard (pairs: the pair holding its first block)
  p.mb_start = fused ? (int)(((int64_t)rank * s.mps) / kBM) >> p.pair : 0;
  p.ng = schedule_group(sched, units);
  p.w0 = std::min(p.ng, s.num_nb);
  const int tiles = sched.num_mb * s.num_nb;  // tiles (pairs: pair tiles), one unit each
  const int grid_units = std::max(1, std::min(units, tiles));
  p.pro_cta0 = -1;  // fetch prologue off unless chosen below
  // A small enough to be read from L2 soon after the start: the fused kernel
  // asks L2 for all of it first (the protocol warp, before its first chunk).
  p.l2_prefetch = fused && s.M * (int64_t)s.num_kb * kBK * 2 <= kL2PrefetchMaxBytes ? 1 : 0;
  // Fetch prologue.  When a k-contiguous fused call takes two or three waves
  // and the last one is partial, the units with one tile fewer than the rest
  // have a tile's time to spare: their copier and epilogue warps stage all of
  // A first (about 256 KB per CTA at most), in k-group order with ready
  // flags, while the other units start their tiles and wait on those flags.
  // No tile owns a window then (w0 = 0: k ascending, as in the barrier GEMM).
  // m_per_shard % 8 == 0 keeps the register fetcher, which publishes its own
  // chunks, out of it.  Measured on the cube workloads that qualify (n = 2176
  // ... 3328, D = 8): the owner protocol's first wave waited about 8 us for
  // chunks copied beside the GEMM's own loads.
  if (fused && !layout_m && (s.mps % 8) == 0 && tiles > grid_units &&
      tiles % grid_units != 0 && tiles <= 3 * grid_units) {
    const int fetch_ctas = (grid_units - tiles % grid_units) << p.pair;
    const int64_t a_bytes = s.M * (int64_t)s.num_kb * kBK * 2;
    if (fetch_ctas >= 16 && a_bytes <= (int64_t)fetch_ctas * (256 << 10)) {
      p.pro_cta0 = (tiles % grid_units) << p.pair;
      p.w0 = 0;
    }
  }
  // Calls of four or more waves: every tile runs k ascending (the tiles of a
  // row block then read each A k-slice at about the same time, as in the
  // barrier GEMM, and share it in L2), and a CTA hands its next tile's
  // window to the copiers only late in the current tile -- from three
  // quarters of its k-groups, counted where the protocol warp is, a few
  // chunks ahead of the loads -- so that staged chunks are still in L2 when
  // the next wave reads them.  Measured at M=16384 N=3584 K=8192 (ncu, per
  // fused launch, hand-off from half-way with the protocol still in the
  // loading thread): DRAM reads 1293 -> 1069 MB, 589 -> 579 us; interleaved
  // timing 609 -> 601 us.  With the protocol warp, three quarters instead of
  // half: -3 us, FP8 -4 us; the m-contiguous staging, which gained nothing
  // from a later hand-off while the protocol ran in the loading thread, now
  // gains 4.5 us.  On one to three waves ascending order cost 2-7 us (the
  // first wave waits on the owners' copiers) and the later hand-off 2 us at
  // cube 4096: those keep the owned window first and hand off at once (with
  // the protocol warp, ascending order from three waves on still cost 4 us
  // at cube 3968 and 8 us with FP8 at cube 4096).  The order depends on the
  // shape only, so every rank and both layouts of a call get the same
  // per-tile order (and, with k ascending, the barrier GEMM's results bit
  // for bit).
  if (fused && p.w0 > 0 && tiles >= 4 * grid_units) {
    p.k_asc = 1;
    p.stage_from = (3 * p.G) / 4;
    // m-contiguous on CTA pairs: pairs whose rows all lie in the local shard
    // read them K-major from the shard instead of MN-major from the [K, M]
    // staging, so those chunks are neither written transposed nor waited on.
    // Measured at M=16384 (interleaved): 641.7 -> 627.4 us; at M=4096 (three
    // waves) it cost 4 us, so it goes with the four-wave plan.
    if (layout_m && p.pair) p.local_direct = 1;
  }
  p.flag_words = (int64_t)s.num_mb * p.G;
  p.started_words = p.num_tiles;
  *grid = grid_units << p.pair;
  return AG_OK;
}

// A 3-D view of D equal row segments, `rows` x `inner` each, `seg_stride`
// rows apart: dims {inner, rows, D}; box {box_inner, box_rows, 1}; 128-byte
// swizzle.  Not cached (the chunked pipeline encodes one per chunk).
int make_map3(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t D,
              uint64_t seg_stride, uint32_t box_inner, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) {
    snprintf(t_cuda_msg, sizeof t_cuda_msg, "cuTensorMapEncodeTiled entry point unavailable");
    return AG_ERR_CUDA;
  }
  cuuint64_t dims[3] = {inner, rows, D};
  cuuint64_t strides[2] = {inner * 2, seg_stride * inner * 2};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(t_cuda_msg, sizeof t_cuda_msg, "cuTensorMapEncodeTiled (3-D) failed (CUresult %d)",
             (int)r);
    return AG_ERR_CUDA;
  }
  return AG_OK;
}

// pair: clusters of two CTAs (grid even), the kernel's CTA-pair variant.
template <int kMode, bool kPair, bool kF8 = false>
int launch(int grid, cudaStream_t stream, const GemmParams& p, const char* what) {
  auto k = agmm_gemm_kernel<kMode, kPair, kF8>;
  cudaError_t e;
  if constexpr (kPair) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)mode_threads(kMode));
    cfg.dynamicSmemBytes = Pipe<true>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k, p);
    if (e == cudaSuccess) e = cudaGetLastError();
  } else {
    k<<<grid, mode_threads(kMode), Pipe<false>::kSmemBytes, stream>>>(p);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? AG_OK : cuda_fail(e, what);
}

// Encoded tensor maps, keyed by everything that goes into one (the address,
// the 2-D extent, the box).  Callers usually pass the same buffers call after
// call, and encoding is host work that would otherwise sit in front of every
// launch.  A map holds only an address and a shape, so a cached entry stays
// valid for any buffer later allocated at that address with that shape.
// Guarded by g_mu (make_map runs under it); cleared when it grows large.
struct MapKey {
  uintptr_t base;
  uint64_t inner, outer;
  uint32_t box_inner, box_outer;
  bool operator==(const MapKey& o) const {
    return base == o.base && inner == o.inner && outer == o.outer && box_inner == o.box_inner &&
           box_outer == o.box_outer;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = k.base * 0x9E3779B97F4A7C15ull;
    h ^= (k.inner + 0x632BE59BD9B4E019ull + (h << 6) + (h >> 2));
    h ^= (k.outer + 0x94D049BB133111EBull + (h << 6) + (h >> 2));
    h ^= ((uint64_t)k.box_inner << 32 | k.box_outer) + (h << 6) + (h >> 2);
    return (size_t)h;
  }
};
constexpr size_t kMapCacheMax = 1024;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

int make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
             uint32_t box_outer) {
  const MapKey key{reinterpret_cast<uintptr_t>(base), inner, outer, box_inner, box_outer};
  auto hit = g_maps.find(key);
  if (hit != g_maps.end()) {
    *m = hit->second;
    return AG_OK;
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) {
    snprintf(t_cuda_msg, sizeof t_cuda_msg, "cuTensorMapEncodeTiled entry point unavailable");
    return AG_ERR_CUDA;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(t_cuda_msg, sizeof t_cuda_msg, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return AG_ERR_CUDA;
  }
  if (g_maps.size() >= kMapCacheMax) g_maps.clear();
  g_maps.emplace(key, *m);
  return AG_OK;
}

int run(bool fused, const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
        const void* bias, void* a_gathered, void* out, cudaStream_t stream,
        const ag_options* opt_in) {
  ag_options o;
  ag_options_default(&o);
  if (opt_in) o = *opt_in;
  // FP8: a row of K bytes is moved as K/2 16-bit words, so from here on K
  // counts those words (shapes, maps, flags, copies); only b's map, the MMA
  // and the epilogue know the elements are 8-bit.
  const bool fp8 = o.dtype == AG_DTYPE_FP8_E4M3;
  if (fp8) {
    if (K < 16 || K % 16) return AG_ERR_INVALID_ARG;
    K /= 2;
  }
  Shape s;
  int st = validate(a_shards, D, m_per_shard, K, b, N, bias, a_gathered, out, o, fused, &s);
  if (st != AG_OK) return st;

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  AG_CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return AG_ERR_UNSUPPORTED;
  DevState& ds = g_dev[dev];
  st = device_init(ds, dev);
  if (st != AG_OK) return st;

  for (int r = 0; r < D; ++r)
    if ((st = check_device_ptr(a_shards[r], dev)) != AG_OK) return st;
  if ((st = check_device_ptr(b, dev)) != AG_OK || (st = check_device_ptr(a_gathered, dev)) != AG_OK ||
      (st = check_device_ptr(out, dev)) != AG_OK)
    return st;
  if (bias && (st = check_device_ptr(bias, dev)) != AG_OK) return st;
  if (o.trace && (st = check_device_ptr(o.trace, dev)) != AG_OK) return st;

  const bool layout_m = o.layout == AG_LAYOUT_M_CONTIGUOUS;
  const int cap = o.num_sms ? std::min(o.num_sms, ds.sms) : ds.sms;
  // The launch plan first: it can still refuse the tile options, and nothing
  // may be enqueued before every check has passed.
  GemmParams p;
  memset(&p, 0, sizeof p);
  p.M = (int)s.M;
  p.N = N;
  p.K = K;
  p.D = D;
  p.mps = m_per_shard;
  p.rank = fused ? o.rank : 0;
  p.num_mb = s.num_mb;
  p.num_nb = s.num_nb;
  p.num_kb = s.num_kb;
  int grid = 0;
  if ((st = plan_launch(p, s, cap, ds.pair_clusters, fused, layout_m, o, &grid)) != AG_OK)
    return st;

  // Workspace: flags (fused) and the [K, M] staging (m-contiguous layout).
  uint64_t* flags = nullptr;
  uint16_t* staging = nullptr;
  bool library_ws = false;
  if (fused && o.workspace) {
    const size_t need = flags_bytes(s) + (layout_m ? (size_t)s.K * s.M * 2 : 0);
    if ((size_t)o.workspace_bytes < need) return AG_ERR_WORKSPACE;
    if (!aligned(o.workspace, 256)) return AG_ERR_INVALID_ARG;
    if ((st = check_device_ptr(o.workspace, dev)) != AG_OK) return st;
    flags = static_cast<uint64_t*>(o.workspace);
    staging = layout_m ? reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(o.workspace) +
                                                     flags_bytes(s))
                       : nullptr;
  } else if (fused || layout_m) {
    library_ws = true;
    if ((st = check_busy(ds, stream)) != AG_OK) return st;
    if ((st = grow_workspace(ds, s, fused, layout_m, stream)) != AG_OK) return st;
    flags = fused ? ds.flags : nullptr;
    staging = layout_m ? ds.staging : nullptr;
  }

  if ((st = make_map(&p.tm_a, a_gathered, (uint64_t)K, (uint64_t)s.M, kBK, kBM)) != AG_OK) return st;
  const bool pair = p.pair != 0;
  if (fp8) {
    // b is [N, K] (K-major): boxes of this CTA's b columns (pair: 128 of the
    // tile's 256) x 128 bytes of K.
    if ((st = make_map(&p.tm_b, b, (uint64_t)K, (uint64_t)N, kBK, pair ? kBN / 2 : kBN)) != AG_OK)
      return st;
  } else if ((st = make_map(&p.tm_b, b, (uint64_t)N, (uint64_t)K, 64, kBK)) != AG_OK) {
    return st;
  }
  if ((st = make_map(&p.tm_out, out, (uint64_t)N, (uint64_t)s.M, kEpiCols, kEpiRows)) != AG_OK)
    return st;
  if (layout_m &&
      (st = make_map(&p.tm_a_mk, staging, (uint64_t)s.M, (uint64_t)K, 64, kBK)) != AG_OK)
    return st;
  if (fused) {
    // Row blocks that straddle shards are loaded in boxes of 2^sh_log2 rows
    // (the largest of 64, 32, 16, 8 that divides m_per_shard) when the shard
    // boundaries fall on multiples of 8 rows.
    const bool straddle8 = D > 1 && (m_per_shard % kBM) != 0 && (m_per_shard % 8) == 0;
    p.sh_log2 = straddle_log2(m_per_shard);
    for (int r = 0; r < D; ++r) {
      if ((st = make_map(&p.tm_shard[r], a_shards[r], (uint64_t)K, (uint64_t)m_per_shard, kBK,
                         kBM)) != AG_OK)
        return st;
      if (straddle8 && (st = make_map(&p.tm_shard8[r], a_shards[r], (uint64_t)K,
                                      (uint64_t)m_per_shard, kBK, 1u << p.sh_log2)) != AG_OK)
        return st;
    }
  }

  const uint64_t epoch = g_epoch.fetch_add(1) + 1;
  const int64_t timeout = o.timeout_ns ? o.timeout_ns : kDefaultTimeoutNs;
  for (int r = 0; r < D; ++r) p.shards[r] = static_cast<const uint16_t*>(a_shards[r]);
  p.a_gathered = static_cast<uint16_t*>(a_gathered);
  p.staging_mk = staging;
  p.bias = static_cast<const float*>(bias);
  p.flags = flags;
  p.started = flags ? flags + flags_region(s) / 8 : nullptr;
  p.err = ds.err;
  p.trace = o.trace;
  p.trace_words = o.trace_words;
  p.epoch = epoch;
  p.fbase = epoch << kFlagShift;
  p.timeout_ns = timeout;
  p.pipe_timeout_ns = 4 * timeout + 2000000000LL;
  p.inject_delay_ns = fused ? o.inject_delay_ns : 0;
  p.fp16 = o.dtype == AG_DTYPE_FP16 ? 1 : 0;  // FP8 writes bf16
  p.inject_skip_flag = fused ? o.inject_skip_flag : -1;
  if (fp8) p.scale_ab = o.scale_a * o.scale_b;

  if (!fused) {
    GatherParams gp;
    memset(&gp, 0, sizeof gp);
    for (int r = 0; r < D; ++r) gp.shards[r] = static_cast<const uint16_t*>(a_shards[r]);
    gp.a_gathered = static_cast<uint16_t*>(a_gathered);
    gp.staging_mk = staging;
    gp.vec_per_shard = (int64_t)m_per_shard * K / 8;
    gp.M = (int)s.M;
    gp.K = K;
    gp.mps = m_per_shard;
    gp.row0 = 0;
    gp.row1 = (int)s.M;
    gp.loc0 = 0;
    gp.loc1 = m_per_shard;
    gp.trace = o.trace;
    gp.trace_words = o.trace_words;
    if (layout_m) {
      const int64_t slots = ((s.M / 8 + 15) / 16) * ((K / 8 + 1) / 2) * 32;
      const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(ds.sms * 8, (slots + 255) / 256));
      agmm_gather_mk_kernel<<<blocks, 256, 0, stream>>>(gp);
    } else {
      const int64_t per_shard_blocks = (gp.vec_per_shard + 255) / 256;
      const int gx = (int)std::max<int64_t>(
          1, std::min<int64_t>((ds.sms * 4 + D - 1) / D, per_shard_blocks));
      agmm_gather_kernel<<<dim3(gx, D), 256, 0, stream>>>(gp);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "gather kernel launch");
  }

  if (fp8 && fused)
    st = pair ? launch<kFusedK, true, true>(grid, stream, p, "fused kernel (fp8)")
              : launch<kFusedK, false, true>(grid, stream, p, "fused kernel (fp8)");
  else if (fp8)
    st = pair ? launch<kGemmK, true, true>(grid, stream, p, "gemm kernel (fp8)")
              : launch<kGemmK, false, true>(grid, stream, p, "gemm kernel (fp8)");
  else if (fused && layout_m)
    st = pair ? launch<kFusedM, true>(grid, stream, p, "fused kernel")
              : launch<kFusedM, false>(grid, stream, p, "fused kernel");
  else if (fused)
    st = pair ? launch<kFusedK, true>(grid, stream, p, "fused kernel")
              : launch<kFusedK, false>(grid, stream, p, "fused kernel");
  else if (layout_m)
    st = pair ? launch<kGemmM, true>(grid, stream, p, "gemm kernel")
              : launch<kGemmM, false>(grid, stream, p, "gemm kernel");
  else
    st = pair ? launch<kGemmK, true>(grid, stream, p, "gemm kernel")
              : launch<kGemmK, false>(grid, stream, p, "gemm kernel");
  if (st == AG_OK && library_ws) st = mark_busy(ds, stream);
  return st;
}

}  // namespace

namespace {

// ---------------------------------------------------------------------------
// The chunked pipeline: the third way to run the operation, between the
// barrier (one gather, then one GEMM) and the fused kernel (tile-level flags).
// A is taken as [S, D, m/S, K] (S chunks, D shards): chunk s is the s-th
// sub-block of every shard, local rows [s*m/S, (s+1)*m/S).  For each chunk,
// round-robin over four streams: gather the chunk (every shard contributes),
// then multiply its D row segments in one launch of the barrier GEMM core
// (k ascending).  The caller's stream forks to the chunk streams and joins
// back.

// One barrier-core GEMM over D row segments of a_gathered -- rows
// [d*m_per_shard + lo, d*m_per_shard + hi) for every d -- into the same rows
// of out: A and out as 3-D views {K or N, hi - lo, D}, each segment padded to
// whole row blocks (rows past a segment's end load as zeros and are not
// stored).
int gemm_segments(DevState& ds, const Shape& s, int lo, int hi, const void* a_gathered,
                  const void* b, const void* bias, void* out, int cap, const ag_options& o,
                  uint64_t epoch, int64_t timeout, cudaStream_t stream) {
  const int seg_rows = hi - lo;
  const int seg_blocks = (seg_rows + kBM - 1) / kBM;
  Shape sc = s;
  sc.num_mb = s.D * seg_blocks;
  sc.M = (int64_t)sc.num_mb * kBM;
  const uint16_t* a_base = static_cast<const uint16_t*>(a_gathered) + (int64_t)lo * s.K;
  uint16_t* out_base = static_cast<uint16_t*>(out) + (int64_t)lo * s.N;
  GemmParams p;
  memset(&p, 0, sizeof p);
  int st;
  if ((st = make_map3(&p.tm_a, a_base, (uint64_t)s.K, (uint64_t)seg_rows, (uint64_t)s.D,
                      (uint64_t)s.mps, kBK, kBM)) != AG_OK)
    return st;
  const bool fp8 = o.dtype == AG_DTYPE_FP8_E4M3;  // s.K counts 16-bit words (see run)
  if (!fp8 && (st = make_map(&p.tm_b, b, (uint64_t)s.N, (uint64_t)s.K, 64, kBK)) != AG_OK) return st;
  if ((st = make_map3(&p.tm_out, out_base, (uint64_t)s.N, (uint64_t)seg_rows, (uint64_t)s.D,
                      (uint64_t)s.mps, kEpiCols, kEpiRows)) != AG_OK)
    return st;
  p.a_gathered = const_cast<uint16_t*>(a_base);
  p.bias = static_cast<const float*>(bias);
  p.err = ds.err;
  p.epoch = epoch;
  p.fbase = epoch << kFlagShift;
  p.timeout_ns = timeout;
  p.pipe_timeout_ns = 4 * timeout + 2000000000LL;
  p.M = (int)sc.M;
  p.N = s.N;
  p.K = s.K;
  p.D = s.D;
  p.mps = (int)sc.M;
  p.num_mb = sc.num_mb;
  p.num_nb = sc.num_nb;
  p.num_kb = sc.num_kb;
  p.sh_log2 = 3;
  p.seg_blocks = seg_blocks;
  p.seg_rows = seg_rows;
  p.fp16 = o.dtype == AG_DTYPE_FP16 ? 1 : 0;
  p.inject_skip_flag = -1;
  int grid = 0;
  if ((st = plan_launch(p, sc, cap, ds.pair_clusters, false, false, o, &grid)) != AG_OK) return st;
  if (fp8) {
    if ((st = make_map(&p.tm_b, b, (uint64_t)s.K, (uint64_t)s.N, kBK, p.pair ? kBN / 2 : kBN)) !=
        AG_OK)
      return st;
    p.scale_ab = o.scale_a * o.scale_b;
    return p.pair ? launch<kGemmK, true, true>(grid, stream, p, "gemm kernel (chunk, fp8)")
                  : launch<kGemmK, false, true>(grid, stream, p, "gemm kernel (chunk, fp8)");
  }
  return p.pair ? launch<kGemmK, true>(grid, stream, p, "gemm kernel (chunk)")
                : launch<kGemmK, false>(grid, stream, p, "gemm kernel (chunk)");
}

int run_chunked(const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
                const void* bias, void* a_gathered, void* out, cudaStream_t stream,
                const ag_options* opt_in, int chunks) {
  ag_options o;
  ag_options_default(&o);
  if (opt_in) o = *opt_in;
  if (o.dtype == AG_DTYPE_FP8_E4M3) {  // moved as K/2 16-bit words, as in run()
    if (K < 16 || K % 16) return AG_ERR_INVALID_ARG;
    K /= 2;
  }
  Shape s;
  int st = validate(a_shards, D, m_per_shard, K, b, N, bias, a_gathered, out, o, false, &s);
  if (st != AG_OK) return st;
  if (chunks < 1 || chunks > 4096) return AG_ERR_INVALID_ARG;
  if (o.layout != AG_LAYOUT_K_CONTIGUOUS) return AG_ERR_UNSUPPORTED;

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  AG_CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return AG_ERR_UNSUPPORTED;
  DevState& ds = g_dev[dev];
  if ((st = device_init(ds, dev)) != AG_OK) return st;
  for (int r = 0; r < D; ++r)
    if ((st = check_device_ptr(a_shards[r], dev)) != AG_OK) return st;
  if ((st = check_device_ptr(b, dev)) != AG_OK || (st = check_device_ptr(a_gathered, dev)) != AG_OK ||
      (st = check_device_ptr(out, dev)) != AG_OK)
    return st;
  if (bias && (st = check_device_ptr(bias, dev)) != AG_OK) return st;
  if (!ds.chunk_init) {
    for (int i = 0; i < DevState::kChunkStreams; ++i) {
      AG_CK(cudaStreamCreateWithFlags(&ds.cstream[i], cudaStreamNonBlocking));
      AG_CK(cudaEventCreateWithFlags(&ds.join_ev[i], cudaEventDisableTiming));
    }
    AG_CK(cudaEventCreateWithFlags(&ds.fork_ev, cudaEventDisableTiming));
    ds.chunk_init = true;
  }

  const uint64_t epoch = g_epoch.fetch_add(1) + 1;
  const int64_t timeout = o.timeout_ns ? o.timeout_ns : kDefaultTimeoutNs;
  const int cap = o.num_sms ? std::min(o.num_sms, ds.sms) : ds.sms;
  // Sub-blocks shorter than a 128-row tile would be padded to one (wasted
  // MMA work), so S is at most m_per_shard / 128 (at least 1).
  const int S = std::max(1, std::min(chunks, m_per_shard / kBM));
  const int used = std::min(S, DevState::kChunkStreams);
  AG_CK(cudaEventRecord(ds.fork_ev, stream));
  for (int i = 0; i < used; ++i) AG_CK(cudaStreamWaitEvent(ds.cstream[i], ds.fork_ev, 0));

  for (int c = 0; c < S; ++c) {
    cudaStream_t cs = ds.cstream[c % DevState::kChunkStreams];
    const int lo = (int)((int64_t)c * m_per_shard / S);
    const int hi = (int)((int64_t)(c + 1) * m_per_shard / S);
    GatherParams gp;
    memset(&gp, 0, sizeof gp);
    for (int r = 0; r < D; ++r) gp.shards[r] = static_cast<const uint16_t*>(a_shards[r]);
    gp.a_gathered = static_cast<uint16_t*>(a_gathered);
    gp.vec_per_shard = (int64_t)m_per_shard * K / 8;
    gp.M = (int)s.M;
    gp.K = K;
    gp.mps = m_per_shard;
    gp.row0 = 0;
    gp.row1 = (int)s.M;
    gp.loc0 = lo;
    gp.loc1 = hi;
    const int64_t blocks = ((int64_t)(hi - lo) * K / 8 + 255) / 256;
    const int gx = (int)std::max<int64_t>(1, std::min<int64_t>((ds.sms * 4 + D - 1) / D, blocks));
    agmm_gather_kernel<<<dim3(gx, D), 256, 0, cs>>>(gp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "gather kernel launch (chunk)");
    if ((st = gemm_segments(ds, s, lo, hi, a_gathered, b, bias, out, cap, o, epoch, timeout, cs)) !=
        AG_OK)
      return st;
  }
  for (int i = 0; i < used; ++i) {
    AG_CK(cudaEventRecord(ds.join_ev[i], ds.cstream[i]));
    AG_CK(cudaStreamWaitEvent(stream, ds.join_ev[i], 0));
  }
  return AG_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// ag_matmul_noalloc: the fused kernel with its scratch in a fixed device array
// (for callers that cannot allocate device memory; see include/agmm.h).

namespace {

constexpr size_t kNoAllocErrBytes = 256;  // error word at the front, 256-byte aligned rest

// Scratch of ag_matmul_noalloc: [error word | ready flags | per-tile words].
// Zero at module load; every call of every stream on this device shares it.
static __device__ __align__(256) uint8_t g_noalloc_scratch[AG_NOALLOC_SCRATCH_BYTES];

struct NoAllocState {
  bool init = false;
  bool supported = false;
  int sms = 0;
  int pair_clusters = 0;
  uint8_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  uint64_t reported_epoch = 0;
};
NoAllocState g_noalloc[kMaxDevices];

// Once per device, with that device current: check the device, set the fused
// kernel's shared-memory limit and look up the array's device address (the
// host-side name of a __device__ array is only a stand-in, never a device
// pointer).  Allocates nothing.
int noalloc_setup(NoAllocState& ns, int dev) {
  if (ns.init) return ns.supported ? AG_OK : AG_ERR_UNSUPPORTED;
  int major = 0, sms = 0;
  AG_CK(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
  AG_CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, agmm_gemm_kernel<kFusedK, false, false>) != cudaSuccess || major != 10) {
    cudaGetLastError();
    ns.init = true;
    ns.supported = false;
    return AG_ERR_UNSUPPORTED;
  }
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kFusedK, false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Pipe<false>::kSmemBytes));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kFusedK, true, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Pipe<true>::kSmemBytes));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kFusedK, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Pipe<false>::kSmemBytes));
  AG_CK(cudaFuncSetAttribute(agmm_gemm_kernel<kFusedK, true, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Pipe<true>::kSmemBytes));
  if (int st = query_pair_clusters(sms, &ns.pair_clusters)) return st;
  void* ptr = nullptr;
  AG_CK(cudaGetSymbolAddress(&ptr, g_noalloc_scratch));
  if (!ptr || !aligned(ptr, 256)) {
    snprintf(t_cuda_msg, sizeof t_cuda_msg, "scratch array has no usable device address");
    return AG_ERR_CUDA;
  }
  ns.sms = sms;
  ns.scratch = static_cast<uint8_t*>(ptr);
  ns.init = true;
  ns.supported = true;
  return AG_OK;
}

int run_noalloc(const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
                const void* bias, void* a_gathered, void* out, cudaStream_t stream,
                const ag_options* opt_in) {
  ag_options o;
  ag_options_default(&o);
  if (opt_in) o = *opt_in;
  if (o.workspace) return AG_ERR_INVALID_ARG;  // the scratch is fixed
  if (o.layout != AG_LAYOUT_K_CONTIGUOUS) return AG_ERR_UNSUPPORTED;
  const bool fp8 = o.dtype == AG_DTYPE_FP8_E4M3;
  if (fp8) {  // moved as K/2 16-bit words, as in run()
    if (K < 16 || K % 16) return AG_ERR_INVALID_ARG;
    K /= 2;
  }
  Shape s;
  int st = validate(a_shards, D, m_per_shard, K, b, N, bias, a_gathered, out, o, true, &s);
  if (st != AG_OK) return st;
  if (kNoAllocErrBytes + flags_bytes(s) > (size_t)AG_NOALLOC_SCRATCH_BYTES) return AG_ERR_TOO_LARGE;

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  AG_CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return AG_ERR_UNSUPPORTED;
  NoAllocState& ns = g_noalloc[dev];
  if ((st = noalloc_setup(ns, dev)) != AG_OK) return st;
  for (int r = 0; r < D; ++r)
    if ((st = check_device_ptr(a_shards[r], dev)) != AG_OK) return st;
  if ((st = check_device_ptr(b, dev)) != AG_OK || (st = check_device_ptr(a_gathered, dev)) != AG_OK ||
      (st = check_device_ptr(out, dev)) != AG_OK)
    return st;
  if (bias && (st = check_device_ptr(bias, dev)) != AG_OK) return st;
  if (o.trace && (st = check_device_ptr(o.trace, dev)) != AG_OK) return st;

  GemmParams p;
  memset(&p, 0, sizeof p);
  if ((st = make_map(&p.tm_a, a_gathered, (uint64_t)K, (uint64_t)s.M, kBK, kBM)) != AG_OK) return st;
  if (!fp8 && (st = make_map(&p.tm_b, b, (uint64_t)N, (uint64_t)K, 64, kBK)) != AG_OK) return st;
  if ((st = make_map(&p.tm_out, out, (uint64_t)N, (uint64_t)s.M, kEpiCols, kEpiRows)) != AG_OK)
    return st;
  const bool straddle8 = D > 1 && (m_per_shard % kBM) != 0 && (m_per_shard % 8) == 0;
  p.sh_log2 = straddle_log2(m_per_shard);
  for (int r = 0; r < D; ++r) {
    if ((st = make_map(&p.tm_shard[r], a_shards[r], (uint64_t)K, (uint64_t)m_per_shard, kBK,
                       kBM)) != AG_OK)
      return st;
    if (straddle8 && (st = make_map(&p.tm_shard8[r], a_shards[r], (uint64_t)K,
                                    (uint64_t)m_per_shard, kBK, 1u << p.sh_log2)) != AG_OK)
      return st;
  }
  const uint64_t epoch = g_epoch.fetch_add(1) + 1;
  const int64_t timeout = o.timeout_ns ? o.timeout_ns : kDefaultTimeoutNs;
  uint64_t* flags = reinterpret_cast<uint64_t*>(ns.scratch + kNoAllocErrBytes);
  for (int r = 0; r < D; ++r) p.shards[r] = static_cast<const uint16_t*>(a_shards[r]);
  p.a_gathered = static_cast<uint16_t*>(a_gathered);
  p.staging_mk = nullptr;
  p.bias = static_cast<const float*>(bias);
  p.flags = flags;
  p.started = flags + flags_region(s) / 8;
  p.err = reinterpret_cast<unsigned long long*>(ns.scratch);
  p.trace = o.trace;
  p.trace_words = o.trace_words;
  p.epoch = epoch;
  p.fbase = epoch << kFlagShift;
  p.timeout_ns = timeout;
  p.pipe_timeout_ns = 4 * timeout + 2000000000LL;
  p.M = (int)s.M;
  p.N = N;
  p.K = K;
  p.D = D;
  p.mps = m_per_shard;
  p.rank = o.rank;
  p.num_mb = s.num_mb;
  p.num_nb = s.num_nb;
  p.num_kb = s.num_kb;
  const int cap = o.num_sms ? std::min(o.num_sms, ns.sms) : ns.sms;
  int grid = 0;
  if ((st = plan_launch(p, s, cap, ns.pair_clusters, true, false, o, &grid)) != AG_OK) return st;
  p.inject_delay_ns = o.inject_delay_ns;
  p.fp16 = o.dtype == AG_DTYPE_FP16 ? 1 : 0;
  p.inject_skip_flag = o.inject_skip_flag;
  if (fp8) {
    if ((st = make_map(&p.tm_b, b, (uint64_t)K, (uint64_t)N, kBK, p.pair ? kBN / 2 : kBN)) !=
        AG_OK)
      return st;
    p.scale_ab = o.scale_a * o.scale_b;
    return p.pair ? launch<kFusedK, true, true>(grid, stream, p, "fused kernel (no-alloc, fp8)")
                  : launch<kFusedK, false, true>(grid, stream, p, "fused kernel (no-alloc, fp8)");
  }
  return p.pair ? launch<kFusedK, true>(grid, stream, p, "fused kernel (no-alloc)")
                : launch<kFusedK, false>(grid, stream, p, "fused kernel (no-alloc)");
}

}  // namespace

extern "C" {

void ag_options_default(ag_options* opt) {
  if (!opt) return;
  memset(opt, 0, sizeof *opt);
  opt->dtype = AG_DTYPE_BF16;
  opt->layout = AG_LAYOUT_K_CONTIGUOUS;
  opt->rank = 0;
  opt->k_per_flag = 0;  // automatic
  opt->num_sms = 0;
  opt->inject_skip_flag = -1;
  opt->timeout_ns = kDefaultTimeoutNs;
  opt->scale_a = 1.0f;
  opt->scale_b = 1.0f;
}

int ag_matmul(const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
              const void* bias_or_null, void* a_gathered, void* out, cudaStream_t stream) {
  return run(true, a_shards, D, m_per_shard, K, b, N, bias_or_null, a_gathered, out, stream,
             nullptr);
}

int ag_then_matmul(const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
                   const void* bias_or_null, void* a_gathered, void* out, cudaStream_t stream) {
  return run(false, a_shards, D, m_per_shard, K, b, N, bias_or_null, a_gathered, out, stream,
             nullptr);
}

int ag_matmul_ex(const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
                 const void* bias_or_null, void* a_gathered, void* out, cudaStream_t stream,
                 const ag_options* opt) {
  return run(true, a_shards, D, m_per_shard, K, b, N, bias_or_null, a_gathered, out, stream, opt);
}

int ag_then_matmul_ex(const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
                      const void* bias_or_null, void* a_gathered, void* out, cudaStream_t stream,
                      const ag_options* opt) {
  return run(false, a_shards, D, m_per_shard, K, b, N, bias_or_null, a_gathered, out, stream, opt);
}

int ag_chunked_matmul_ex(const void** a_shards, int D, int m_per_shard, int K, const void* b,
                         int N, const void* bias_or_null, void* a_gathered, void* out,
                         cudaStream_t stream, const ag_options* opt, int chunks) {
  return run_chunked(a_shards, D, m_per_shard, K, b, N, bias_or_null, a_gathered, out, stream,
                     opt, chunks);
}

size_t ag_workspace_size(int D, int m_per_shard, int K, int N, const ag_options* opt) {
  ag_options o;
  ag_options_default(&o);
  if (opt) o = *opt;
  if (o.dtype == AG_DTYPE_FP8_E4M3) {  // sized like the 16-bit problem with K/2 columns
    if (K % 16) return 0;
    K /= 2;
  }
  if (D < 1 || D > AG_MAX_SHARDS || m_per_shard < 1 || K < 8 || N < 8 || K % 8 || N % 8 ||
      o.k_per_flag < 0)
    return 0;
  const int64_t M = (int64_t)D * m_per_shard;
  if (M > INT32_MAX) return 0;
  Shape s;
  s.M = M;
  s.K = K;
  s.N = N;
  s.num_mb = (int)((M + kBM - 1) / kBM);
  s.num_nb = (N + kBN - 1) / kBN;
  s.num_kb = (K + kBK - 1) / kBK;
  s.kpf = o.k_per_flag ? o.k_per_flag : sizing_k_per_flag(s.num_kb);
  s.G = (s.num_kb + s.kpf - 1) / s.kpf;
  return flags_bytes(s) + (o.layout == AG_LAYOUT_M_CONTIGUOUS ? (size_t)K * M * 2 : 0);
}

int ag_get_device_error(cudaStream_t stream, int* code, int* info) {
  if (code) *code = AG_OK;
  if (info) *info = 0;
  int dev = 0;
  AG_CK(cudaGetDevice(&dev));
  AG_CK(cudaStreamSynchronize(stream));
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev < 0 || dev >= kMaxDevices) return AG_OK;
  // Both error words carry epochs of the one process-wide counter, so the
  // later call's error is the one with the larger epoch; the other word keeps
  // its error for the next report.
  unsigned long long lib[2] = {0, 0}, na[2] = {0, 0};
  DevState& ds = g_dev[dev];
  NoAllocState& ns = g_noalloc[dev];
  if (ds.err) AG_CK(cudaMemcpy(lib, ds.err, sizeof lib, cudaMemcpyDeviceToHost));
  if (ns.scratch) AG_CK(cudaMemcpy(na, ns.scratch, sizeof na, cudaMemcpyDeviceToHost));
  const bool lib_new = lib[0] > ds.reported_epoch, na_new = na[0] > ns.reported_epoch;
  const unsigned long long* w = nullptr;
  if (lib_new && (!na_new || lib[0] > na[0])) {
    ds.reported_epoch = lib[0];
    w = lib;
  } else if (na_new) {
    ns.reported_epoch = na[0];
    w = na;
  }
  if (w) {
    if (code) *code = (int)(w[1] >> 32);
    if (info) *info = (int)(w[1] & 0xFFFFFFFFull);
  }
  return AG_OK;
}

int ag_release_workspace(void) {
  int dev = 0;
  AG_CK(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev < 0 || dev >= kMaxDevices) return AG_OK;
  DevState& ds = g_dev[dev];
  if (!ds.flags && !ds.staging) return AG_OK;
  AG_CK(cudaDeviceSynchronize());
  if (ds.flags) AG_CK(cudaFree(ds.flags));
  if (ds.staging) AG_CK(cudaFree(ds.staging));
  ds.flags = nullptr;
  ds.staging = nullptr;
  ds.flags_cap = ds.staging_cap = 0;
  return AG_OK;
}

const char* ag_status_string(int status) {
  switch (status) {
    case AG_OK: return "ok";
    case AG_ERR_INVALID_ARG: return "invalid argument";
    case AG_ERR_UNSUPPORTED: return "unsupported by the library or the device";
    case AG_ERR_CUDA: return t_cuda_msg;
    case AG_ERR_TIMEOUT: return "device-side wait timed out";
    case AG_ERR_WORKSPACE: return "caller workspace too small";
    case AG_ERR_TOO_LARGE: return "problem needs more than the fixed no-alloc scratch";
    case AG_ERR_BUSY: return "library workspace in use by an unfinished call on another stream";
    case AG_ERR_BOUNDS: return "device-side index outside its buffer (bounds-checked build)";
    default: return "unknown status";
  }
}

int ag_matmul_noalloc(const void** a_shards, int D, int m_per_shard, int K, const void* b, int N,
                      const void* bias_or_null, void* a_gathered, void* out,
                      cudaStream_t stream, const ag_options* opt) {
  return run_noalloc(a_shards, D, m_per_shard, K, b, N, bias_or_null, a_gathered, out, stream,
                     opt);
}

int ag_plan_fused(int D, int m_per_shard, int K, int N, const ag_options* opt_in, int sms,
                  int pair_clusters, ag_plan* plan) {
  if (!plan || sms < 1 || pair_clusters < 0) return AG_ERR_INVALID_ARG;
  ag_options o;
  ag_options_default(&o);
  if (opt_in) o = *opt_in;
  if (o.dtype == AG_DTYPE_FP8_E4M3) {  // 16-bit words, as the calls count them
    if (K < 16 || K % 16) return AG_ERR_INVALID_ARG;
    K /= 2;
  }
  Shape s;
  const int st = shape_of(D, m_per_shard, K, N, o, &s);
  if (st != AG_OK) return st;
  GemmParams p;
  memset(&p, 0, sizeof p);
  const int cap = o.num_sms ? std::min(o.num_sms, sms) : sms;
  int grid = 0;
  const int pst =
      plan_launch(p, s, cap, pair_clusters, true, o.layout == AG_LAYOUT_M_CONTIGUOUS, o, &grid);
  if (pst != AG_OK) return pst;
  plan->grid = grid;
  plan->k_ascending = p.k_asc;
  plan->block_m = p.pair ? 2 * kBM : kBM;
  plan->stages = p.pair ? kStagesPair : kStagesSingle;
  plan->cta_pairs = p.pair;
  plan->tiles = p.num_tiles >> p.pair;
  plan->k_per_flag = p.kpf;
  plan->prologue_cta0 = p.pro_cta0;
  plan->l2_prefetch = p.l2_prefetch;
  return AG_OK;
}

int ag_num_sms(void) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return sms;
}

}  // extern "C"
