// Tensor-core LR-cache build: L = X . A_cat on tcgen05 (TMEM accumulators).
//
// LRAgent technical summary (gist.science), Metodologia section 2 (BaseShared:
// the LR cache holds the LoRA down-projection X.A_i at width r); PReCache
// abstract (PreLRShared: every agent's LR cache built in one pass over the
// context).  All agents' down-projections sit side by side in
// A_cat = [A_1|...|A_A] ([d_model, A*r], row-major), so one GEMM reads each row
// of X once and writes every agent's r columns: L[t, :] = X[t, :] . A_cat.
//
// A_cat is consumed as it is stored: TMA copies boxes of 64 K-rows x 64
// columns (128-byte swizzle) and the MMA reads them as an MN-major B operand,
// so no caller has to transpose the weights.
//
// One CTA per (128-row tile of X, column tile of <= 512 columns): the tile's
// columns are accumulated in tensor memory (fp32, 128 lanes):
//   warp 0     TMA producer: X tile [128 x 64] and the column tile's A_cat
//              boxes per k-step into a ring of shared-memory stages;
//   warp 1     allocates TMEM; lane 0 issues tcgen05.mma (M = 128, N split in
//              chunks of <= 256 columns, K = 16 per instruction) and
//              tcgen05.commit to release each stage and, at the end, to
//              publish the accumulator;
//   warps 2-5  epilogue: tcgen05.ld of their 32-lane quarter, fp32 -> bf16,
//              stores to L.
// Short inputs (a few row tiles) would leave most SMs idle, so the plan may
// split d_model over a thread-block cluster of S CTAs: each accumulates its
// share of the k-steps, writes its fp32 partial tile into its own shared
// memory, and after a cluster barrier CTA j of the cluster sums rows
// [j*128/S, (j+1)*128/S) of all S partials through distributed shared memory
// in rank order (deterministic) and stores them as bf16.
// Every wait is bounded; on a timeout the CTA records the error, waits
// (bounded) for its copies and MMAs in flight, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>

#include "../../include/flash_lora_attn.h"
#include "fla_common.cuh"
#include "ptx.cuh"

namespace fla {
namespace bld {

constexpr int kBM = 128;                 // rows of X per CTA (MMA M)
constexpr int kBK = 64;                  // K per stage: one 128-byte swizzle row of bf16
constexpr int kBoxN = 64;                // A_cat columns per TMA box (128 bytes)
constexpr int kBoxBytes = kBK * 128;     // one A_cat box: 64 K-rows x 128 bytes
constexpr int kThreads = 192;            // 6 warps
constexpr int kSmemBudget = 220 * 1024;
constexpr int kMaxSplit = 16;
constexpr int kMaxTileCols = 512;        // TMEM columns

constexpr int kMaxSegments = 3;

// Columns [seg_begin(s), seg_end[s]) of the product go to out[s] (row stride
// ld[s], column 0 = the segment's first column); segment ends are multiples of 32.
struct Params {
  __nv_bfloat16 *out[kMaxSegments];
  int64_t ld[kMaxSegments];
  int32_t seg_end[kMaxSegments];
  int32_t n_seg;
  int64_t n;
  int32_t K;                 // d_model
  int32_t N;                 // columns of the product (= seg_end[n_seg - 1])
  int32_t tile_boxes;        // 64-column boxes per column tile (<= 8)
  int32_t n_ntiles;          // column tiles
  int32_t stages;
  int32_t split;             // CTAs per cluster along d_model (1: no split)
  int32_t ksteps;            // k-steps per CTA
  int32_t red_pitch;         // floats per row of the split-K partial tile
  uint32_t tmem_cols;
};

// Destination of 4 (or more, within one segment) consecutive product columns
// starting at column c of row `row`.
__device__ __forceinline__ __nv_bfloat16 *out_ptr(const Params &p, int64_t row, int c) {
  // constant indices only, so the parameter arrays stay in the constant bank
  const bool s1 = p.n_seg > 1 && c >= p.seg_end[0];
  const bool s2 = p.n_seg > 2 && c >= p.seg_end[1];
  __nv_bfloat16 *base = s2 ? p.out[2] : (s1 ? p.out[1] : p.out[0]);
  const int64_t ld = s2 ? p.ld[2] : (s1 ? p.ld[1] : p.ld[0]);
  const int begin = s2 ? p.seg_end[1] : (s1 ? p.seg_end[0] : 0);
  return base + row * ld + (c - begin);
}

__global__ void __launch_bounds__(kThreads, 1)
build_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmA, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int a_bytes = kBM * kBK * 2;
  const int stage_bytes = a_bytes + p.tile_boxes * kBoxBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.stages * stage_bytes);
  // bars: full[stages] | empty[stages] | acc_full | drain
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tile = blockIdx.x / p.split;
  const int kslice = blockIdx.x % p.split;  // = rank in the cluster (cluster dims (split, 1, 1))
  const int nt = (int)(tile % p.n_ntiles);
  const int64_t m0 = (tile / p.n_ntiles) * kBM;
  const int c0 = nt * p.tile_boxes * kBoxN;  // first product column of this CTA
  // boxes of this tile (the last tile may be narrower), split into <= 2 MMA
  // chunks of <= 4 boxes (256 columns)
  const int n_boxes = min(p.tile_boxes, ((p.N + kBoxN - 1) / kBoxN) - nt * p.tile_boxes);
  const int chunk0 = n_boxes <= 4 ? n_boxes : (n_boxes + 1) / 2;
  const int chunk1 = n_boxes - chunk0;
  const int load_bytes = a_bytes + n_boxes * kBoxBytes;
  const int n_k = p.ksteps;
  const int kt0 = kslice * p.ksteps;
  const uint32_t full0 = ptx::smem_u32(&bars[0]);
  const uint32_t empty0 = ptx::smem_u32(&bars[p.stages]);
  const uint32_t acc_full = ptx::smem_u32(&bars[2 * p.stages]);
  const uint32_t drain = ptx::smem_u32(&bars[2 * p.stages + 1]);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < p.stages; ++s) {
      ptx::mbar_init(full0 + 8 * s, 1);
      ptx::mbar_init(empty0 + 8 * s, 1);
    }
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(drain, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&s_tmem), p.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      ptx::prefetch_tmap(&tmX);
      ptx::prefetch_tmap(&tmA);
      int issued = 0;
      for (int kt = 0; kt < n_k; ++kt) {
        const int s = kt % p.stages;
        if (kt >= p.stages && !ptx::mbar_wait(empty0 + 8 * s, ((kt / p.stages) & 1) ^ 1)) {
          set_device_error(kErrBuildEmptyWait);
          s_abort = 1;
          break;
        }
        if (*(volatile int *)&s_abort) break;
        const uint32_t fb = full0 + 8 * s;
        ptx::mbar_arrive_expect_tx(fb, load_bytes);
        const uint32_t sa = ptx::smem_u32(smem + s * stage_bytes);
        const int k = (kt0 + kt) * kBK;
        ptx::tma_load_2d(sa, &tmX, k, (int32_t)m0, fb);
        // boxes past column N are filled with zeros by the copy (their MMA
        // columns are never stored)
        for (int b = 0; b < n_boxes; ++b)
          ptx::tma_load_2d(sa + a_bytes + b * kBoxBytes, &tmA, c0 + b * kBoxN, k, fb);
        ++issued;
      }
      // leave no copy in flight
      for (int k = 0; k < p.stages && k < issued; ++k) {
        const int kt = issued - 1 - k;
        ptx::mbar_wait(full0 + 8 * (kt % p.stages), (kt / p.stages) & 1);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      const uint32_t idesc0 = ptx::idesc_bf16_f32(kBM, chunk0 * kBoxN) | (1u << 16);  // B MN-major
      const uint32_t idesc1 = ptx::idesc_bf16_f32(kBM, (chunk1 > 0 ? chunk1 : 1) * kBoxN) | (1u << 16);
      const uint64_t d_a = ptx::smem_desc_k128(ptx::smem_u32(smem));
      const uint64_t d_b = ptx::smem_desc_mn128(ptx::smem_u32(smem) + a_bytes, kBoxBytes);
      bool ok = true;
      for (int kt = 0; kt < n_k; ++kt) {
        const int s = kt % p.stages;
        if (!ptx::mbar_wait(full0 + 8 * s, (kt / p.stages) & 1)) {
          set_device_error(kErrBuildFullWait);
          s_abort = 1;
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint64_t da = ptx::desc_advance(d_a, s * stage_bytes);
        const uint64_t db = ptx::desc_advance(d_b, s * stage_bytes);
#pragma unroll
        for (int k16 = 0; k16 < kBK / 16; ++k16) {
          const uint32_t acc = (kt > 0 || k16 > 0) ? 1u : 0u;
          // A: 16 K-columns = 32 bytes further along each swizzled row;
          // B: 16 K-rows = two 1024-byte swizzle atoms further on
          ptx::tc_mma_f16(tmem, ptx::desc_advance(da, k16 * 32), ptx::desc_advance(db, k16 * 2048), idesc0, acc);
          if (chunk1 > 0)
            ptx::tc_mma_f16(tmem + chunk0 * kBoxN, ptx::desc_advance(da, k16 * 32),
                            ptx::desc_advance(db, chunk0 * kBoxBytes + k16 * 2048), idesc1, acc);
        }
        ptx::tc_commit(empty0 + 8 * s);  // stage s is free once these MMAs have read it
      }
      // accumulator complete (or, after an abort, every issued MMA retired)
      ptx::tc_commit(ok ? acc_full : drain);
      if (!ok) ptx::mbar_wait(drain, 0);
    }
  } else {
    // ======================= epilogue (warps 2..5) =======================
    const int quarter = warp & 3;  // TMEM lanes [32*quarter, 32*quarter + 32)
    const int rloc = quarter * 32 + lane;
    const int64_t row = m0 + rloc;
    bool ready = false;
    // the accumulator arrives after the whole K loop: poll with a bound, but
    // stop early if the CTA aborted
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      if (ptx::mbar_try_wait(acc_full, 0)) { ready = true; break; }
      if (*(volatile int *)&s_abort) break;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        set_device_error(kErrBuildAccWait);
        s_abort = 1;
        break;
      }
    }
    if (ready) {
      ptx::tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
      const int ncols = min(p.tile_boxes * kBoxN, p.N - c0);  // multiple of 32
      // split-K: the fp32 partial goes to this CTA's own shared memory (the
      // stage ring is idle: every MMA, hence every copy, has completed)
      float *red = reinterpret_cast<float *>(smem) + (size_t)rloc * p.red_pitch;
      for (int c = 0; c < ncols; c += 32) {
        uint32_t v[32];
        ptx::tmem_ld32(tl + c, v);
        ptx::tmem_ld_wait();
        if (p.split > 1) {
          float4 *dst = reinterpret_cast<float4 *>(red + c);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        } else if (row < p.n) {
          uint4 out[4];
          uint32_t *o = reinterpret_cast<uint32_t *>(out);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            o[i] = ptx::pack_bf16(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          uint4 *dst = reinterpret_cast<uint4 *>(out_ptr(p, row, c0 + c));  // 32 columns, one segment
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = out[i];
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) ptx::tmem_dealloc(tmem, p.tmem_cols);
  if (p.split == 1) return;

  // ======================= split-K: sum the cluster's partial tiles =======================
  // Two cluster barriers, each reached by every thread of every CTA of the
  // cluster exactly once and only through bounded waits: the first publishes
  // the partial tiles (release / acquire at cluster scope), the second keeps
  // each CTA's shared memory alive until every peer has read it.  A CTA that
  // aborted still takes part (its error is recorded; the outputs are then
  // undefined).
  ptx::cluster_sync_all();
  {
    const int rows = kBM / p.split;
    const int r0 = kslice * rows;
    const int ncols = min(p.tile_boxes * kBoxN, p.N - c0);
    const int c4n = ncols / 4;
    const uint32_t red_local = ptx::smem_u32(smem);
    for (int e = threadIdx.x; e < rows * c4n; e += kThreads) {
      const int rr = e / c4n, c4 = e - rr * c4n;
      const int rloc = r0 + rr;
      const uint32_t off = (uint32_t)(rloc * p.red_pitch + c4 * 4) * 4u;
      // every peer's load in flight at once, then the sum in rank order (the
      // same result whichever CTA finished first)
      float4 v[kMaxSplit];
#pragma unroll
      for (int q = 0; q < kMaxSplit; ++q)
        if (q < p.split) v[q] = ptx::ld_cluster_f4(ptx::mapa_cluster(red_local + off, (uint32_t)q));
      float4 acc = v[0];
#pragma unroll
      for (int q = 1; q < kMaxSplit; ++q)
        if (q < p.split) {
          acc.x += v[q].x; acc.y += v[q].y; acc.z += v[q].z; acc.w += v[q].w;
        }
      const int64_t row = m0 + rloc;
      if (row < p.n)
        *reinterpret_cast<uint2 *>(out_ptr(p, row, c0 + c4 * 4)) =
            make_uint2(ptx::pack_bf16(acc.x, acc.y), ptx::pack_bf16(acc.z, acc.w));
    }
  }
  ptx::cluster_sync_all();
}

// ---------------------------------------------------------------------------
// The same GEMM on CTA pairs (cluster of 2, tcgen05 cta_group::2): a pair owns
// 256 rows of X (128 per CTA) and a column tile; each MMA chunk (128 or 256
// columns) is split into column halves, one in each CTA's shared memory, so a
// CTA copies only half of the tile's W boxes per k-step and the W bytes each
// SM loads per MMA flop halve.  The even CTA issues every MMA and commits the
// stage releases and the finished accumulator to both CTAs; both CTAs' copies
// count on the even CTA's full barriers.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
build_tc2_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmA, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int a_bytes = kBM * kBK * 2;
  const int stage_bytes = a_bytes + (p.tile_boxes / 2) * kBoxBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.stages * stage_bytes);
  // bars: full[stages] | empty[stages] | acc_full | drain
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();  // 0: the CTA that issues the MMAs
  const int64_t pair_tile = blockIdx.x / 2;
  const int nt = (int)(pair_tile % p.n_ntiles);
  const int64_t m0 = (pair_tile / p.n_ntiles) * (2 * kBM) + rank * kBM;  // this CTA's rows
  const int c0 = nt * p.tile_boxes * kBoxN;
  // boxes of this tile, rounded up to an even count (zero-filled past N);
  // MMA chunk 0 takes up to 4 of them (256 columns), chunk 1 the rest
  int nb = min(p.tile_boxes, (p.N + kBoxN - 1) / kBoxN - nt * p.tile_boxes);
  nb = (nb + 1) & ~1;
  const int chunk0 = min(4, nb), chunk1 = nb - chunk0;
  const int load_bytes = a_bytes + (nb / 2) * kBoxBytes;  // this CTA's copies per k-step
  const int n_k = p.ksteps;
  const uint32_t full0 = ptx::smem_u32(&bars[0]);
  const uint32_t empty0 = ptx::smem_u32(&bars[p.stages]);
  const uint32_t acc_full = ptx::smem_u32(&bars[2 * p.stages]);
  const uint32_t drain = ptx::smem_u32(&bars[2 * p.stages + 1]);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < p.stages; ++s) {
      ptx::mbar_init(full0 + 8 * s, 1);
      ptx::mbar_init(empty0 + 8 * s, 1);
    }
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(drain, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(&s_tmem), p.tmem_cols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  // the peer signals this CTA's barriers: both initialisations first
  ptx::cluster_sync_all();
  ptx::tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t lead_full0 = ptx::mapa_cluster(full0, 0);

  if (warp == 0) {
    // ======================= TMA producer (both CTAs) =======================
    if (lane == 0) {
      ptx::prefetch_tmap(&tmX);
      ptx::prefetch_tmap(&tmA);
      int issued = 0;
      for (int kt = 0; kt < n_k; ++kt) {
        const int s = kt % p.stages;
        if (kt >= p.stages && !ptx::mbar_wait_cluster(empty0 + 8 * s, ((kt / p.stages) & 1) ^ 1)) {
          set_device_error(kErrBuildEmptyWait);
          s_abort = 1;
          break;
        }
        if (*(volatile int *)&s_abort) break;
        const uint32_t fb = lead_full0 + 8 * s;  // the even CTA's full barrier counts both CTAs' bytes
        if (rank == 0) ptx::mbar_arrive_expect_tx(full0 + 8 * s, 2 * load_bytes);
        const uint32_t sa = ptx::smem_u32(smem + s * stage_bytes);
        const int k = kt * kBK;
        ptx::tma_load_2d_pair(sa, &tmX, k, (int32_t)m0, fb);
        // this CTA's column half of each chunk
        for (int b = 0; b < chunk0 / 2; ++b)
          ptx::tma_load_2d_pair(sa + a_bytes + b * kBoxBytes, &tmA, c0 + (rank * (chunk0 / 2) + b) * kBoxN, k, fb);
        for (int b = 0; b < chunk1 / 2; ++b)
          ptx::tma_load_2d_pair(sa + a_bytes + (chunk0 / 2 + b) * kBoxBytes, &tmA,
                                c0 + (chunk0 + rank * (chunk1 / 2) + b) * kBoxN, k, fb);
        ++issued;
      }
      // the even CTA's full barriers also count the peer's copies: leave none in flight
      if (rank == 0)
        for (int k = 0; k < p.stages && k < issued; ++k) {
          const int kt = issued - 1 - k;
          ptx::mbar_wait_cluster(full0 + 8 * (kt % p.stages), (kt / p.stages) & 1);
        }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer (even CTA) =======================
    if (lane == 0 && rank == 0) {
      const uint32_t idesc0 = ptx::idesc_bf16_f32(2 * kBM, chunk0 * kBoxN) | (1u << 16);  // B MN-major
      const uint32_t idesc1 = ptx::idesc_bf16_f32(2 * kBM, (chunk1 > 0 ? chunk1 : 2) * kBoxN) | (1u << 16);
      const uint64_t d_a = ptx::smem_desc_k128(ptx::smem_u32(smem));
      const uint64_t d_b = ptx::smem_desc_mn128(ptx::smem_u32(smem) + a_bytes, kBoxBytes);
      const uint32_t empty_peer0 = ptx::mapa_cluster(empty0, 1);
      const uint32_t empty_own0 = ptx::mapa_cluster(empty0, 0);
      bool ok = true;
      for (int kt = 0; kt < n_k; ++kt) {
        const int s = kt % p.stages;
        if (!ptx::mbar_wait_cluster(full0 + 8 * s, (kt / p.stages) & 1)) {
          set_device_error(kErrBuildFullWait);
          s_abort = 1;
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint64_t da = ptx::desc_advance(d_a, s * stage_bytes);
        const uint64_t db = ptx::desc_advance(d_b, s * stage_bytes);
#pragma unroll
        for (int k16 = 0; k16 < kBK / 16; ++k16) {
          const uint32_t acc = (kt > 0 || k16 > 0) ? 1u : 0u;
          ptx::tc_mma_f16_pair(tmem, ptx::desc_advance(da, k16 * 32), ptx::desc_advance(db, k16 * 2048), idesc0, acc);
          if (chunk1 > 0)
            ptx::tc_mma_f16_pair(tmem + chunk0 * kBoxN, ptx::desc_advance(da, k16 * 32),
                                 ptx::desc_advance(db, (chunk0 / 2) * kBoxBytes + k16 * 2048), idesc1, acc);
        }
        // stage s is free in both CTAs once these MMAs have read it
        ptx::tc_commit_pair(empty_own0 + 8 * s);
        ptx::tc_commit_pair(empty_peer0 + 8 * s);
      }
      if (ok) {
        ptx::tc_commit_pair(ptx::mapa_cluster(acc_full, 0));
        ptx::tc_commit_pair(ptx::mapa_cluster(acc_full, 1));
      } else {
        ptx::tc_commit_pair(ptx::mapa_cluster(drain, 0));
        ptx::mbar_wait(drain, 0);
      }
    }
  } else {
    // ======================= epilogue (warps 2..5, both CTAs) =======================
    const int quarter = warp & 3;  // TMEM lanes [32*quarter, 32*quarter + 32)
    const int64_t row = m0 + quarter * 32 + lane;
    bool ready = false;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      if (ptx::mbar_try_wait_cluster(acc_full, 0)) { ready = true; break; }
      if (*(volatile int *)&s_abort) break;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        set_device_error(kErrBuildAccWait);
        s_abort = 1;
        break;
      }
    }
    if (ready) {
      ptx::tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
      const int ncols = min(nb * kBoxN, p.N - c0);  // multiple of 32
      for (int c = 0; c < ncols; c += 32) {
        uint32_t v[32];
        ptx::tmem_ld32(tl + c, v);
        ptx::tmem_ld_wait();
        if (row < p.n) {
          uint4 out[4];
          uint32_t *o = reinterpret_cast<uint32_t *>(out);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            o[i] = ptx::pack_bf16(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          uint4 *dst = reinterpret_cast<uint4 *>(out_ptr(p, row, c0 + c));  // 32 columns, one segment
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = out[i];
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  // neither CTA frees the pair's TMEM (or leaves) while the other still works
  ptx::cluster_sync_all();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem, p.tmem_cols);
}

}  // namespace bld

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
inline const char *&build_tc_err() {
  static thread_local const char *e = "";
  return e;
}
inline const char *build_tc_last_error() { return build_tc_err(); }

struct BuildPlan {
  int tile_boxes, n_ntiles, stages, smem_bytes, split, ksteps, red_pitch;
  uint32_t tmem_cols;
  bool ok;
};

inline int build_smem_bytes(int stages, int stage) { return stages * stage + (2 * stages + 2) * 8 + 1024; }

// Plan for column tiles of `bpt` boxes (64 columns each) and a split of d_model
// over `split` CTAs; ok = false when it does not fit shared memory.
inline BuildPlan build_tc_plan_for(int d_model, int n_cols, int bpt, int split) {
  BuildPlan pl{};
  pl.ok = false;
  const int boxes = (n_cols + bld::kBoxN - 1) / bld::kBoxN;
  const int nk = d_model / bld::kBK;
  if (bpt < 1 || bpt > 8 || nk % split != 0) return pl;
  pl.tile_boxes = std::min(bpt, boxes);
  pl.n_ntiles = (boxes + pl.tile_boxes - 1) / pl.tile_boxes;
  pl.split = split;
  pl.ksteps = nk / split;
  pl.red_pitch = pl.tile_boxes * bld::kBoxN + 4;
  const int stage = bld::kBM * bld::kBK * 2 + pl.tile_boxes * bld::kBoxBytes;
  int st = (bld::kSmemBudget - 1024 - 128) / stage;
  st = std::min(st, 8);
  if (split > 1) {
    // no more stages than k-steps, but room for the fp32 partial tile
    st = std::min(st, std::max(2, pl.ksteps));
    while (st * stage < bld::kBM * pl.red_pitch * 4) ++st;
  }
  if (st < 2 || build_smem_bytes(st, stage) > 227 * 1024) return pl;
  pl.stages = st;
  pl.smem_bytes = build_smem_bytes(st, stage);
  uint32_t cols = 32;
  while ((int)cols < pl.tile_boxes * bld::kBoxN) cols <<= 1;
  pl.tmem_cols = cols;
  pl.ok = true;
  return pl;
}

// Widest balanced tiles (<= 8 boxes = 512 TMEM columns), no split.
inline BuildPlan build_tc_shape_plan(int d_model, int n_cols) {
  BuildPlan pl{};
  pl.ok = false;
  if (d_model < bld::kBK || d_model % bld::kBK != 0 || n_cols % 32 != 0 || n_cols < 32) return pl;
  const int boxes = (n_cols + bld::kBoxN - 1) / bld::kBoxN;
  const int nt = (boxes + 7) / 8;
  return build_tc_plan_for(d_model, n_cols, (boxes + nt - 1) / nt, 1);
}

// Full plan for n rows on `sms` SMs.  When the widest tiles cover less than
// half the GPU, narrower tiles (<= 4 boxes) and a split of d_model over a
// cluster of up to max_split CTAs are considered; the plan that puts the
// most CTAs on the SMs (at most one wave) wins, the larger split on ties.
inline BuildPlan build_tc_plan(int64_t n, int d_model, int n_cols, int sms, int max_split) {
  BuildPlan best = build_tc_shape_plan(d_model, n_cols);
  if (!best.ok || n <= 0) return best;
  const int64_t m_tiles = (n + bld::kBM - 1) / bld::kBM;
  if (m_tiles * best.n_ntiles * 2 > sms) return best;
  const int boxes = (n_cols + bld::kBoxN - 1) / bld::kBoxN;
  int64_t best_ctas = m_tiles * best.n_ntiles;
  const int narrow_nt = (boxes + 3) / 4;
  const int bpts[2] = {best.tile_boxes, (boxes + narrow_nt - 1) / narrow_nt};
  for (int bpt : bpts)
    for (int sp = max_split; sp >= 2; sp >>= 1) {
      const BuildPlan c = build_tc_plan_for(d_model, n_cols, bpt, sp);
      if (!c.ok) continue;
      const int64_t ctas = m_tiles * c.n_ntiles * sp;
      if (ctas > sms) continue;
      if (ctas > best_ctas) {
        best = c;
        best_ctas = ctas;
      }
    }
  return best;
}

// Plan of the CTA-pair kernel: column tiles of an even number of boxes (<= 8;
// a tile whose box count is odd copies one zero-filled box past column N), each
// CTA holding half of every tile's boxes per stage.
inline BuildPlan build_tc2_plan(int d_model, int n_cols) {
  BuildPlan pl{};
  pl.ok = false;
  if (d_model < bld::kBK || d_model % bld::kBK != 0 || n_cols % 32 != 0 || n_cols < 32) return pl;
  const int boxes = (n_cols + bld::kBoxN - 1) / bld::kBoxN;
  const int nt = (boxes + 7) / 8;
  int bpt = (boxes + nt - 1) / nt;
  bpt = (bpt + 1) & ~1;
  pl.tile_boxes = bpt;
  pl.n_ntiles = (boxes + bpt - 1) / bpt;
  pl.split = 1;
  pl.ksteps = d_model / bld::kBK;
  pl.red_pitch = 0;
  const int stage = bld::kBM * bld::kBK * 2 + (bpt / 2) * bld::kBoxBytes;
  const int st = std::min((bld::kSmemBudget - 1024 - 128) / stage, 8);
  if (st < 2 || build_smem_bytes(st, stage) > 227 * 1024) return pl;
  pl.stages = st;
  pl.smem_bytes = build_smem_bytes(st, stage);
  uint32_t cols = 32;
  while ((int)cols < bpt * bld::kBoxN) cols <<= 1;
  pl.tmem_cols = cols;
  pl.ok = true;
  return pl;
}

// Largest cluster (16, else 8) of this kernel that the device can place with
// `smem` bytes per CTA; cached per device and shared-memory size.
inline int build_max_cluster(int smem) {
  static std::mutex mu;
  static int cached_smem[kMaxDevices], cached_val[kMaxDevices];
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(mu);
  if (cached_val[dev] > 0 && cached_smem[dev] == smem) return cached_val[dev];
  int best = 8;
  const void *fn = reinterpret_cast<const void *>(bld::build_tc_kernel);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
      ensure_dynamic_smem(fn, smem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16);
    cfg.blockDim = dim3(bld::kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 16;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int nclu = 0;
    if (cudaOccupancyMaxActiveClusters(&nclu, bld::build_tc_kernel, &cfg) == cudaSuccess && nclu >= 1) best = 16;
  }
  cudaGetLastError();  // a refused query leaves no sticky error
  cached_smem[dev] = smem;
  cached_val[dev] = best;
  return best;
}

// One output segment of the product: `cols` columns written to `ptr` with row stride `ld`.
struct BuildSegment {
  void *ptr;
  int64_t ld;
  int32_t cols;
};

inline bool build_tc_supported(const void *X, int64_t ldx, const void *W, const BuildSegment *seg, int n_seg,
                               int d_model, int dtype) {
  auto al16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  if (dtype != FLA_BF16 || !al16(X) || !al16(W) || ldx % 8 != 0 || n_seg < 1 || n_seg > bld::kMaxSegments)
    return false;
  int n_cols = 0;
  for (int i = 0; i < n_seg; ++i) {
    if (!al16(seg[i].ptr) || seg[i].ld % 8 != 0 || seg[i].cols % 32 != 0 || seg[i].cols < 32) return false;
    n_cols += seg[i].cols;
  }
  return build_tc_shape_plan(d_model, n_cols).ok;
}

// out = X . W, W = [d_model rows, sum of the segments' columns], dense row-major,
// the product's columns written segment by segment.
inline fla_status build_tc_launch(const void *X, int64_t ldx, const void *W, const BuildSegment *seg, int n_seg,
                                  int64_t n, int d_model, cudaStream_t s) {
  int n_cols = 0;
  for (int i = 0; i < n_seg; ++i) n_cols += seg[i].cols;
  const int sms = device_sm_count();
  BuildPlan pl = build_tc_plan(n, d_model, n_cols, sms, 8);
  if (!pl.ok) {
    build_tc_err() = "shape outside the tensor-core build kernel";
    return FLA_ERR_UNSUPPORTED;
  }
  {  // a 16-CTA cluster where the device can place one and it covers more SMs
    const BuildPlan p16 = build_tc_plan(n, d_model, n_cols, sms, 16);
    if (p16.split == 16 && build_max_cluster(p16.smem_bytes) >= 16) pl = p16;
  }
  // Without a split of d_model the rows fill the GPU: CTA pairs (256 rows,
  // half of the W boxes per CTA) do the same work with half the W copies.
  bool pair = false;
  if (pl.split == 1 && n > bld::kBM) {
    const BuildPlan p2 = build_tc2_plan(d_model, n_cols);
    if (p2.ok) {
      pl = p2;
      pair = true;
    }
  }
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) {
    build_tc_err() = "cuTensorMapEncodeTiled is not available from the driver";
    return FLA_ERR_CUDA;
  }
  CUtensorMap mX, mW;
  const cuuint32_t es[2] = {1, 1};
  {
    const cuuint64_t dims[2] = {(cuuint64_t)d_model, (cuuint64_t)n};
    const cuuint64_t strides[1] = {(cuuint64_t)ldx * 2};
    const cuuint32_t box[2] = {(cuuint32_t)bld::kBK, (cuuint32_t)bld::kBM};
    if (enc(&mX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(X), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      build_tc_err() = "encoding the X tensor map failed";
      return FLA_ERR_CUDA;
    }
  }
  {
    // W [d_model rows, n_cols columns], row-major: boxes of 64 columns x 64 rows
    const cuuint64_t dims[2] = {(cuuint64_t)n_cols, (cuuint64_t)d_model};
    const cuuint64_t strides[1] = {(cuuint64_t)n_cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)bld::kBoxN, (cuuint32_t)bld::kBK};
    if (enc(&mW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(W), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      build_tc_err() = "encoding the weight tensor map failed";
      return FLA_ERR_CUDA;
    }
  }
  bld::Params prm{};
  int end = 0;
  for (int i = 0; i < n_seg; ++i) {
    prm.out[i] = reinterpret_cast<__nv_bfloat16 *>(seg[i].ptr);
    prm.ld[i] = seg[i].ld;
    end += seg[i].cols;
    prm.seg_end[i] = end;
  }
  prm.n_seg = n_seg;
  prm.n = n;
  prm.K = d_model;
  prm.N = n_cols;
  prm.tile_boxes = pl.tile_boxes;
  prm.n_ntiles = pl.n_ntiles;
  prm.stages = pl.stages;
  prm.split = pl.split;
  prm.ksteps = pl.ksteps;
  prm.red_pitch = pl.red_pitch;
  prm.tmem_cols = pl.tmem_cols;
  const void *fn = pair ? reinterpret_cast<const void *>(bld::build_tc2_kernel)
                        : reinterpret_cast<const void *>(bld::build_tc_kernel);
  cudaError_t e = ensure_dynamic_smem(fn, pl.smem_bytes);
  if (e != cudaSuccess) {
    build_tc_err() = cudaGetErrorString(e);
    return FLA_ERR_CUDA;
  }
  const int64_t grid = pair ? (n + 2 * bld::kBM - 1) / (2 * bld::kBM) * pl.n_ntiles * 2
                            : (n + bld::kBM - 1) / bld::kBM * pl.n_ntiles * pl.split;
  if (grid > 0x7fffffffLL) {
    build_tc_err() = "n_tokens too large";
    return FLA_ERR_UNSUPPORTED;
  }
  if (pair) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(bld::kThreads);
    cfg.dynamicSmemBytes = pl.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, bld::build_tc2_kernel, mX, mW, prm);
    if (e != cudaSuccess) {
      build_tc_err() = cudaGetErrorString(e);
      return FLA_ERR_CUDA;
    }
    return FLA_OK;
  }
  if (pl.split == 1) {
    bld::build_tc_kernel<<<(unsigned)grid, bld::kThreads, pl.smem_bytes, s>>>(mX, mW, prm);
    return FLA_OK;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(bld::kThreads);
  cfg.dynamicSmemBytes = pl.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)pl.split;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, bld::build_tc_kernel, mX, mW, prm);
  if (e != cudaSuccess) {
    build_tc_err() = cudaGetErrorString(e);
    return FLA_ERR_CUDA;
  }
  return FLA_OK;
}

}  // namespace fla
