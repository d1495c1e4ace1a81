// Device code of the fused all-gather matmul and of its barrier baseline.
//
// The design follows "Fused all-gather+GEMM HBM-buffer kernel for iris.ops"
// (ROCm/iris #346, section "New kernel"): fetchers copy A tiles into an HBM
// staging buffer and publish per-tile ready flags; GEMM workers wait on the
// flags and compute tiles as they arrive.  On sm_103a both roles live in one
// persistent CTA per SM as specialised warps:
//
//   warp 0      TMA issuer: waits for a tile's ready flag (or takes the local
//               shard directly), then streams A and B k-blocks into a 4-stage
//               shared-memory ring with cp.async.bulk.tensor.
//   warp 1      MMA issuer: tcgen05.mma 128x256x16 (bf16/fp16 in, fp32 out)
//               into one of two TMEM accumulators (2 x 256 columns).
//   warps 2-5   epilogue: tcgen05.ld, + fp32 bias, round to 16 bits,
//               128-byte-swizzled shared memory, TMA store of the out tile.
//   warps 6-7   fetchers (fused kernel only): claim (row block, k-group)
//               chunks with a CAS on the chunk's flag, copy them from the
//               shards into a_gathered (and, for the m-contiguous layout,
//               transposed into the [K, M] staging), then release the flag.
//
// Flags are 64-bit and epoch-valued: for a call with epoch e, a flag below
// 2e-1 is untouched, 2e-1 is claimed and 2e is ready; nothing needs clearing
// between calls.  Every wait is bounded by a time limit; on expiry the kernel
// records an error word and finishes without hanging.
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
constexpr int kStages = 4;
constexpr int kAStageBytes = kBM * kBK * 2;  // 16 KB
constexpr int kBStageBytes = kBN * kBK * 2;  // 32 KB
constexpr int kStageBytes = kAStageBytes + kBStageBytes;
constexpr int kMnChunkBytes = 64 * kBK * 2;  // one 64-wide MN chunk of an MN-major operand (8 KB)
constexpr int kEpiWarps = 4;
constexpr int kEpiRows = 32;                          // rows per epilogue warp
constexpr int kEpiCols = 64;                          // columns per store box (128 bytes)
constexpr int kEpiBufBytes = kEpiRows * kEpiCols * 2;  // 4 KB
constexpr int kEpiBufs = 2;
constexpr int kTmemCols = 2 * kBN;
constexpr int kFetchWarps = 2;
constexpr int kGemmThreads = 32 * (2 + kEpiWarps);
constexpr int kFusedThreads = kGemmThreads + 32 * kFetchWarps;
constexpr int kMaxShards = 64;
constexpr int kNumBars = 2 * kStages + 4 + 1;
constexpr int kSmemData = kStages * kStageBytes + kEpiWarps * kEpiBufs * kEpiBufBytes;
constexpr int kSmemBytes = 1024 + kSmemData + 8 * kNumBars + 64;
static_assert(kSmemBytes <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");

// Error codes written to the device error word (match ag_status).
constexpr uint32_t kErrTimeout = 4;
// Sites reported with a pipeline timeout (ready-flag timeouts report the flag index).
constexpr uint32_t kSiteEmpty = 0xF00001, kSiteFull = 0xF00002, kSiteTmemEmpty = 0xF00003,
                   kSiteTmemFull = 0xF00004, kSiteDrain = 0xF00005;

struct GemmParams {
  CUtensorMap tm_a;      // a_gathered [M, K]: box {64, 128}, 128B swizzle (K-major A)
  CUtensorMap tm_a_mk;   // staging [K, M]: box {64, 64}, 128B swizzle (MN-major A)
  CUtensorMap tm_local;  // local shard [m_per_shard, K]: box {64, 128}
  CUtensorMap tm_b;      // b [K, N]: box {64, 64}, 128B swizzle (MN-major B)
  CUtensorMap tm_out;    // out [M, N]: box {64, 32}, 128B swizzle (store)
  const uint16_t* shards[kMaxShards];
  uint16_t* a_gathered;
  uint16_t* staging_mk;
  const float* bias;
  uint64_t* flags;              // [num_mb * G]
  unsigned long long* err;      // [2]: epoch of newest error, code << 32 | info
  uint64_t* trace;
  int64_t trace_words;
  uint64_t epoch;
  int64_t timeout_ns;           // one ready-flag wait
  int64_t pipe_timeout_ns;      // one pipeline (mbarrier) wait
  int M, N, K, D, mps, rank;
  int num_mb, num_nb, num_kb, num_tiles;
  int kpf, G;                   // k-blocks per flag, flags per row block
  int mb_start;                 // first row block of the schedule (ring order)
  int layout_m;                 // 1: A is read MN-major from the [K, M] staging
  int fp16;                     // 1: fp16, 0: bf16
  int inject_skip_flag;
};

struct GatherParams {
  const uint16_t* shards[kMaxShards];
  uint16_t* a_gathered;
  int64_t vec_per_shard;  // 16-byte vectors per shard
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

// Persistent schedule: tile t -> (row block, column block).  Row blocks are
// visited in ring order starting at mb_start (the local shard's first block
// for the fused kernel), all column blocks of one row block consecutively, so
// concurrently running CTAs share A rows in L2 and sweep b.
__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& mb, int& nb) {
  int pos = t / p.num_nb;
  nb = t - pos * p.num_nb;
  mb = p.mb_start + pos;
  if (mb >= p.num_mb) mb -= p.num_mb;
}

// A row block is "local" when every row it holds lies in the local shard.
__device__ __forceinline__ bool block_is_local(const GemmParams& p, int mb) {
  int lo = mb * kBM;
  int hi = min(lo + kBM, p.M);
  return lo >= p.rank * p.mps && hi <= (p.rank + 1) * p.mps;
}

// Bounded mbarrier wait.  Returns false (after flagging the CTA abort word and
// recording an error) when the phase does not complete in time.
__device__ __forceinline__ bool wait_bar(const GemmParams& p, uint64_t* bar, uint32_t parity,
                                         volatile int* abort_flag, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
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

// Bounded acquire-wait on a ready flag.  On expiry (or once another wait of
// this call has expired) it records the error and returns false; the caller
// then proceeds, so the pipeline always drains.
__device__ __forceinline__ bool wait_ready(const GemmParams& p, int flag_idx) {
  const uint64_t ready = 2 * p.epoch;
  const uint64_t* f = p.flags + flag_idx;
  if (ld_acquire_gpu(f) >= ready) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t ns = 32;
  for (uint32_t it = 1;; ++it) {
    __nanosleep(ns);
    if (ns < 256) ns <<= 1;
    if (ld_acquire_gpu(f) >= ready) return true;
    if ((it & 15u) == 0) {
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

__device__ __forceinline__ const uint16_t* shard_row(const GemmParams& p, int grow) {
  int s = grow / p.mps;
  int lr = grow - s * p.mps;
  return p.shards[s] + (int64_t)lr * p.K;
}

// Copy one chunk (row block mb, k-group g) from the shards into a_gathered.
__device__ __noinline__ void fetch_chunk_k(const GemmParams& p, int mb, int g, int lane) {
  const int row0 = mb * kBM;
  const int rows = min(kBM, p.M - row0);
  const int c0 = g * p.kpf * kBK;
  const int nv = min(p.kpf * kBK, p.K - c0) >> 3;  // 16-byte vectors per row
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
        v[u] = ld_stream_v4(shard_row(p, row0 + r) + c0 + cv * 8);
        dst[u] = (int64_t)(row0 + r) * p.K + c0 + cv * 8;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (dst[u] >= 0) st_v4(p.a_gathered + dst[u], v[u]);
  }
}

// m-contiguous layout: the same chunk, written both to a_gathered ([M, K]) and
// transposed into the [K, M] staging.  Each lane moves an 8x8 block: 8 row
// loads of 16 bytes, an in-register transpose with byte permutes, 8 column
// stores of 16 bytes.  Consecutive lanes take consecutive row groups so the
// transposed stores are contiguous along M.
__device__ __noinline__ void fetch_chunk_m(const GemmParams& p, int mb, int g, int lane) {
  const int row0 = mb * kBM;
  const int rows = min(kBM, p.M - row0);  // a multiple of 8 (M % 8 == 0)
  const int c0 = g * p.kpf * kBK;
  const int cols = min(p.kpf * kBK, p.K - c0);
  const int nrg = rows >> 3, ncg = cols >> 3;
  const int total = nrg * ncg;
  for (int idx = lane; idx < total; idx += 32) {
    const int rg = idx % nrg, cg = idx / nrg;
    const int col = c0 + cg * 8;
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = ld_stream_v4(shard_row(p, row0 + rg * 8 + i) + col);
#pragma unroll
    for (int i = 0; i < 8; ++i) st_v4(p.a_gathered + (int64_t)(row0 + rg * 8 + i) * p.K + col, v[i]);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t sel = (c & 1) ? 0x7632u : 0x5410u;
      uint4 o;
      o.x = __byte_perm(u4_get(v[0], c >> 1), u4_get(v[1], c >> 1), sel);
      o.y = __byte_perm(u4_get(v[2], c >> 1), u4_get(v[3], c >> 1), sel);
      o.z = __byte_perm(u4_get(v[4], c >> 1), u4_get(v[5], c >> 1), sel);
      o.w = __byte_perm(u4_get(v[6], c >> 1), u4_get(v[7], c >> 1), sel);
      st_v4(p.staging_mk + (int64_t)(col + c) * p.M + row0 + rg * 8, o);
    }
  }
}

// Fetcher warp: walk this CTA's tiles (non-local row blocks first, then the
// local ones, which nobody waits for but a_gathered must still receive), claim
// each still-untouched chunk, copy it, publish it.
__device__ __forceinline__ void fetch_loop(const GemmParams& p, int lane) {
  const uint64_t claimed = 2 * p.epoch - 1, ready = 2 * p.epoch;
  for (int pass = 0; pass < 2; ++pass) {
    int last_mb = -1;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(p, t, mb, nb);
      if (mb == last_mb) continue;
      last_mb = mb;
      if (block_is_local(p, mb) != (pass == 1)) continue;
      for (int g = 0; g < p.G; ++g) {
        const int idx = mb * p.G + g;
        uint64_t* f = p.flags + idx;
        int won = 0;
        if (lane == 0) {
          const uint64_t v = ld_relaxed_gpu(f);
          if (v < claimed)
            won = atomicCAS(reinterpret_cast<unsigned long long*>(f), (unsigned long long)v,
                            (unsigned long long)claimed) == v;
        }
        won = __shfl_sync(0xffffffffu, won, 0);
        if (!won) continue;
        const uint64_t t0 = p.trace ? globaltimer_ns() : 0;
        if (p.layout_m)
          fetch_chunk_m(p, mb, g, lane);
        else
          fetch_chunk_k(p, mb, g, lane);
        __threadfence();
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) {
          if (idx != p.inject_skip_flag) st_release_gpu(f, ready);
          if (p.trace) trace_rec(p.trace, p.trace_words, 1, mb, g, t0, globaltimer_ns());
        }
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

// ------------------------------------------------------------------ the kernel

template <bool kFused>
__global__ void __launch_bounds__(kFused ? kFusedThreads : kGemmThreads, 1)
    agmm_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* epi_smem = smem + kStages * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSmemData);
  uint64_t* full = bars;                    // [kStages] TMA landed
  uint64_t* empty = bars + kStages;         // [kStages] MMAs done reading
  uint64_t* tmem_full = bars + 2 * kStages; // [2] accumulator ready
  uint64_t* tmem_empty = tmem_full + 2;     // [2] accumulator drained
  uint64_t* drain = tmem_empty + 2;         // [1] final MMA drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], 32 * kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    prefetch_tensormap(&p.tm_a);
    prefetch_tensormap(&p.tm_b);
    prefetch_tensormap(&p.tm_out);
    if (kFused) {
      prefetch_tensormap(&p.tm_local);
      if (p.layout_m) prefetch_tensormap(&p.tm_a_mk);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tcgen05_fence_before_sync();
  __syncthreads();
  tcgen05_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  // Parity of the newest TMA load issued into each stage (drained on abort).
  uint32_t issued_mask = 0, issued_parity = 0;
  bool aborted = false;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < p.num_tiles && !aborted; t += gridDim.x) {
        int mb, nb;
        tile_coords(p, t, mb, nb);
        const bool local = kFused && block_is_local(p, mb);
        const bool a_mn = kFused && p.layout_m && !local;
        int last_g = -1;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!wait_bar(p, &empty[stage], phase ^ 1u, abort_flag, kSiteEmpty)) {
            aborted = true;
            break;
          }
          if (kFused && !local) {
            const int g = kb / p.kpf;
            if (g != last_g) {
              const uint64_t t0 = p.trace ? globaltimer_ns() : 0;
              wait_ready(p, mb * p.G + g);
              fence_proxy_async_global();
              if (p.trace) trace_rec(p.trace, p.trace_words, 2, mb, g, t0, globaltimer_ns());
              last_g = g;
            }
          }
          uint8_t* a_dst = smem + stage * kStageBytes;
          uint8_t* b_dst = a_dst + kAStageBytes;
          mbar_arrive_expect_tx(&full[stage], kStageBytes);
          if (local) {
            tma_load_2d(a_dst, &p.tm_local, &full[stage], kb * kBK, mb * kBM - p.rank * p.mps);
          } else if (a_mn) {
            tma_load_2d(a_dst, &p.tm_a_mk, &full[stage], mb * kBM, kb * kBK);
            tma_load_2d(a_dst + kMnChunkBytes, &p.tm_a_mk, &full[stage], mb * kBM + 64, kb * kBK);
          } else {
            tma_load_2d(a_dst, &p.tm_a, &full[stage], kb * kBK, mb * kBM);
          }
#pragma unroll
          for (int j = 0; j < kBN / 64; ++j)
            tma_load_2d(b_dst + j * kMnChunkBytes, &p.tm_b, &full[stage], nb * kBN + j * 64,
                        kb * kBK);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (aborted || *abort_flag) {
        // Let every issued load land before shared memory is released.
        for (int s = 0; s < kStages; ++s)
          if (issued_mask & (1u << s)) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&full[s], (issued_parity >> s) & 1u) &&
                   globaltimer_ns() - t0 < 1000000000ull) {
            }
          }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t ab_bf16 = p.fp16 ? 0u : 1u;
      const uint32_t idesc_k = idesc_f16_f32(ab_bf16, 0, 1, kBM, kBN);
      const uint32_t idesc_mn = idesc_f16_f32(ab_bf16, 1, 1, kBM, kBN);
      int stage = 0;
      uint32_t phase = 0;
      int j = 0;
      for (int t = blockIdx.x; t < p.num_tiles && !aborted; t += gridDim.x, ++j) {
        int mb, nb;
        tile_coords(p, t, mb, nb);
        const bool local = kFused && block_is_local(p, mb);
        const bool a_mn = kFused && p.layout_m && !local;
        const uint32_t idesc = a_mn ? idesc_mn : idesc_k;
        const int buf = j & 1;
        const uint32_t use = (uint32_t)(j >> 1);
        if (!wait_bar(p, &tmem_empty[buf], (use & 1u) ^ 1u, abort_flag, kSiteTmemEmpty)) {
          aborted = true;
          break;
        }
        tcgen05_fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kBN);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!wait_bar(p, &full[stage], phase, abort_flag, kSiteFull)) {
            aborted = true;
            break;
          }
          tcgen05_fence_after_sync();
          const uint32_t a_addr = smem_u32(smem + stage * kStageBytes);
          const uint32_t b_addr = a_addr + kAStageBytes;
#pragma unroll
          for (int ks = 0; ks < kBK / kUmmaK; ++ks) {
            // K-major A: advance 16 elements (32 bytes) inside the swizzle row.
            // MN-major A/B: advance 16 k-rows (2 x 1024-byte groups).
            const uint64_t a_desc =
                a_mn ? smem_desc_sw128(a_addr + ks * 2048, kMnChunkBytes, 1024)
                     : smem_desc_sw128(a_addr + ks * 32, 16, 1024);
            const uint64_t b_desc = smem_desc_sw128(b_addr + ks * 2048, kMnChunkBytes, 1024);
            umma_f16(d_tmem, a_desc, b_desc, idesc, (kb | ks) != 0 ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (aborted) break;
        umma_commit(&tmem_full[buf]);
      }
      // All MMAs issued by this thread complete before TMEM is released.
      umma_commit(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < 1000000000ull) {
      }
    }
    __syncwarp();
  } else if (warp < 2 + kEpiWarps) {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint8_t* my_bufs = epi_smem + (warp - 2) * kEpiBufs * kEpiBufBytes;
    const uint32_t my_bufs_u32 = smem_u32(my_bufs);
    int j = 0;
    int chunk_count = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++j) {
      int mb, nb;
      tile_coords(p, t, mb, nb);
      const int buf = j & 1;
      const uint32_t use = (uint32_t)(j >> 1);
      // Every lane waits; the vote keeps the warp converged for tcgen05.ld.
      const bool ok = wait_bar(p, &tmem_full[buf], use & 1u, abort_flag, kSiteTmemFull);
      if (!__all_sync(0xffffffffu, ok)) break;
      tcgen05_fence_after_sync();
      const uint64_t t0 = p.trace ? globaltimer_ns() : 0;
      const int m0 = mb * kBM + q * kEpiRows;
      const int n_tile = nb * kBN;
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kBN);
#pragma unroll 1
      for (int c = 0; c < kBN / kEpiCols; ++c) {
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(t_row + c * kEpiCols, r0);
        tmem_ld_32x32b_x32(t_row + c * kEpiCols + 32, r1);
        tmem_ld_wait();
        if (c == kBN / kEpiCols - 1) {
          tcgen05_fence_before_sync();
          mbar_arrive(&tmem_empty[buf]);
        }
        const int n0 = n_tile + c * kEpiCols;
        uint32_t packed[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float v0 = __uint_as_float(r0[2 * i]), v1 = __uint_as_float(r0[2 * i + 1]);
          float w0 = __uint_as_float(r1[2 * i]), w1 = __uint_as_float(r1[2 * i + 1]);
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
        const bool store = (m0 < p.M) && (n0 < p.N);
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
          tma_store_2d(&p.tm_out, my_bufs + eb * kEpiBufBytes, n0, m0);
        }
        if (lane == 0) bulk_commit_group();
        ++chunk_count;
      }
      if (p.trace && lane == 0 && q == 0)
        trace_rec(p.trace, p.trace_words, 3, mb, nb, t0, globaltimer_ns());
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  } else if (kFused) {
    // ---------------------------------------------------------- fetchers
    fetch_loop(p, lane);
    __syncwarp();
  }

  tcgen05_fence_before_sync();
  __syncthreads();
  tcgen05_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Barrier-path gather: shard r is copied to rows [r*m_per_shard, ...) of
// a_gathered.  Each shard is one contiguous block, so this is D flat copies;
// blockIdx.y selects the shard.
__global__ void __launch_bounds__(256) agmm_gather_kernel(const __grid_constant__ GatherParams gp) {
  const uint64_t t0 = gp.trace ? globaltimer_ns() : 0;
  const int s = blockIdx.y;
  const uint4* src = reinterpret_cast<const uint4*>(gp.shards[s]);
  uint4* dst = reinterpret_cast<uint4*>(gp.a_gathered) + (int64_t)s * gp.vec_per_shard;
  const int64_t n = gp.vec_per_shard;
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
  if (gp.trace && threadIdx.x == 0) {
    __syncwarp(1u);
    trace_rec(gp.trace, gp.trace_words, 4, blockIdx.x + blockIdx.y * gridDim.x, 0, t0,
              globaltimer_ns());
  }
}

}  // namespace agmm
