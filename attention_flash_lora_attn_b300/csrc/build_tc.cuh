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
// memory, and CTA j of the cluster sums rows [j*128/S, (j+1)*128/S) of all S
// partials through distributed shared memory in rank order (deterministic)
// and stores them as bf16.
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

struct Params {
  __nv_bfloat16 *L;
  int64_t ldl, n;
  int32_t K;                 // d_model
  int32_t N;                 // columns of L (A * r)
  int32_t n_tile;            // columns per CTA (multiple of 64)
  int32_t n_ntiles;          // column tiles
  int32_t n_chunks;          // MMAs per k16 step (each <= 256 columns)
  int32_t chunk_boxes[2];    // 64-column boxes per MMA chunk
  int32_t stages;
  int32_t split;             // CTAs per cluster along d_model (1: no split)
  int32_t ksteps;            // k-steps per CTA
  int32_t red_pitch;         // floats per row of the split-K partial tile
  uint32_t tmem_cols;
};

__global__ void __launch_bounds__(kThreads, 1)
build_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmA, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int n_boxes = p.n_tile / kBoxN;
  const int a_bytes = kBM * kBK * 2;
  const int stage_bytes = a_bytes + n_boxes * kBoxBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.stages * stage_bytes);
  // bars: full[stages] | empty[stages] | acc_full | drain | red_ready | red_done
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tile = blockIdx.x / p.split;
  const int kslice = blockIdx.x % p.split;  // = rank in the cluster (cluster dims (split, 1, 1))
  const int nt = (int)(tile % p.n_ntiles);
  const int64_t m0 = (tile / p.n_ntiles) * kBM;
  const int c0 = nt * p.n_tile;             // first column of L this CTA produces
  const int n_k = p.ksteps;
  const int kt0 = kslice * p.ksteps;
  const uint32_t full0 = ptx::smem_u32(&bars[0]);
  const uint32_t empty0 = ptx::smem_u32(&bars[p.stages]);
  const uint32_t acc_full = ptx::smem_u32(&bars[2 * p.stages]);
  const uint32_t drain = ptx::smem_u32(&bars[2 * p.stages + 1]);
  const uint32_t red_ready = ptx::smem_u32(&bars[2 * p.stages + 2]);
  const uint32_t red_done = ptx::smem_u32(&bars[2 * p.stages + 3]);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < p.stages; ++s) {
      ptx::mbar_init(full0 + 8 * s, 1);
      ptx::mbar_init(empty0 + 8 * s, 1);
    }
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(red_ready, p.split);  // one arrival per CTA of the cluster
    ptx::mbar_init(red_done, p.split);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&s_tmem), p.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // peers arrive on this CTA's barriers later: their initialisation must be
  // visible cluster-wide first (every CTA of a cluster is co-resident)
  if (p.split > 1) ptx::cluster_sync_all();
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
        ptx::mbar_arrive_expect_tx(fb, stage_bytes);
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
      const uint32_t idesc0 = ptx::idesc_bf16_f32(kBM, p.chunk_boxes[0] * kBoxN) | (1u << 16);  // B MN-major
      const uint32_t idesc1 = ptx::idesc_bf16_f32(kBM, p.chunk_boxes[1] * kBoxN) | (1u << 16);
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
          if (p.n_chunks > 1)
            ptx::tc_mma_f16(tmem + p.chunk_boxes[0] * kBoxN, ptx::desc_advance(da, k16 * 32),
                            ptx::desc_advance(db, p.chunk_boxes[0] * kBoxBytes + k16 * 2048), idesc1, acc);
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
      const int ncols = min(p.n_tile, p.N - c0);  // multiple of 32
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
          uint4 *dst = reinterpret_cast<uint4 *>(p.L + row * p.ldl + c0 + c);
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
  const uint32_t rank = (uint32_t)kslice;
  if (threadIdx.x == 0 && !*(volatile int *)&s_abort) {
    ptx::fence_acq_rel_cluster();  // this CTA's partial (written before the barrier above) first
    for (int s = 0; s < p.split; ++s) ptx::mbar_arrive_cluster(ptx::mapa_cluster(red_ready, (uint32_t)s));
  }
  // every CTA's partial is complete once all of them have arrived here; an
  // aborted peer never arrives and this wait runs out instead
  const bool have_all = !*(volatile int *)&s_abort && ptx::mbar_wait_cluster(red_ready, 0);
  if (!have_all && threadIdx.x == 0 && !*(volatile int *)&s_abort) set_device_error(kErrBuildClusterWait);
  if (have_all) {
    const int rows = kBM / p.split;
    const int r0 = (int)rank * rows;
    const int ncols = min(p.n_tile, p.N - c0);
    const int c4n = ncols / 4;
    const uint32_t red_local = ptx::smem_u32(smem);
    for (int e = threadIdx.x; e < rows * c4n; e += kThreads) {
      const int rr = e / c4n, c4 = e - rr * c4n;
      const int rloc = r0 + rr;
      const uint32_t off = (uint32_t)(rloc * p.red_pitch + c4 * 4) * 4u;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < p.split; ++s) {  // rank order: the same sum whichever CTA finishes first
        const float4 v = ptx::ld_cluster_f4(ptx::mapa_cluster(red_local + off, (uint32_t)s));
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      const int64_t row = m0 + rloc;
      if (row < p.n)
        *reinterpret_cast<uint2 *>(p.L + row * p.ldl + c0 + c4 * 4) =
            make_uint2(ptx::pack_bf16(acc.x, acc.y), ptx::pack_bf16(acc.z, acc.w));
    }
  }
  __syncthreads();
  // this CTA's partial must stay in place until every peer has read it
  if (threadIdx.x == 0) {
    if (have_all)
      for (int s = 0; s < p.split; ++s) ptx::mbar_arrive_cluster(ptx::mapa_cluster(red_done, (uint32_t)s));
    if (!ptx::mbar_wait_cluster(red_done, 0)) set_device_error(kErrBuildClusterWait);
  }
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
  int n_tile, n_ntiles, n_chunks, chunk_boxes[2];
  int stages, smem_bytes, split, ksteps, red_pitch;
  uint32_t tmem_cols;
  bool ok;
};

// Shape part of the plan (independent of the number of rows).
inline BuildPlan build_tc_shape_plan(int d_model, int n_cols) {
  BuildPlan pl{};
  pl.ok = false;
  if (d_model < bld::kBK || d_model % bld::kBK != 0 || n_cols % 32 != 0 || n_cols < 32) return pl;
  pl.n_ntiles = (n_cols + bld::kMaxTileCols - 1) / bld::kMaxTileCols;
  const int per = (n_cols + pl.n_ntiles - 1) / pl.n_ntiles;
  pl.n_tile = (per + bld::kBoxN - 1) / bld::kBoxN * bld::kBoxN;
  const int boxes = pl.n_tile / bld::kBoxN;
  pl.n_chunks = (boxes + 3) / 4;  // <= 256 columns per MMA
  pl.chunk_boxes[0] = (boxes + pl.n_chunks - 1) / pl.n_chunks;
  pl.chunk_boxes[1] = boxes - pl.chunk_boxes[0];
  if (pl.n_chunks > 2 || pl.chunk_boxes[0] > 4 || pl.chunk_boxes[1] > 4) return pl;
  if (pl.n_chunks == 1) pl.chunk_boxes[1] = pl.chunk_boxes[0];  // unused, keeps the descriptor valid
  const int stage = bld::kBM * bld::kBK * 2 + boxes * bld::kBoxBytes;
  int stages = (bld::kSmemBudget - 1024 - 64) / stage;
  if (stages > 8) stages = 8;
  if (stages < 2) return pl;
  pl.stages = stages;
  uint32_t cols = 32;
  while ((int)cols < pl.n_tile) cols <<= 1;
  pl.tmem_cols = cols;
  pl.split = 1;
  pl.ksteps = d_model / bld::kBK;
  pl.red_pitch = pl.n_tile + 4;
  pl.smem_bytes = stages * stage + 6 * 8 + (2 * stages) * 8 + 1024;
  pl.ok = true;
  return pl;
}

// Full plan for n rows on `sms` SMs: when the tiles cover less than half the
// GPU, d_model is split over a cluster of up to max_split CTAs (k-steps divide
// evenly; the fp32 partial tile must fit the stage ring).
inline BuildPlan build_tc_plan(int64_t n, int d_model, int n_cols, int sms, int max_split) {
  BuildPlan pl = build_tc_shape_plan(d_model, n_cols);
  if (!pl.ok || n <= 0) return pl;
  const int64_t tiles = (n + bld::kBM - 1) / bld::kBM * pl.n_ntiles;
  const int nk = d_model / bld::kBK;
  const int stage = bld::kBM * bld::kBK * 2 + (pl.n_tile / bld::kBoxN) * bld::kBoxBytes;
  const int red_bytes = bld::kBM * pl.red_pitch * 4;
  if (tiles * 2 <= sms) {
    for (int s = max_split; s >= 2; s >>= 1) {
      if (tiles * s > sms || nk % s != 0) continue;
      int st = std::min(8, std::max(2, nk / s));  // no more stages than k-steps
      while (st * stage < red_bytes) ++st;
      if (st * stage + 6 * 8 + 2 * st * 8 + 1024 > 227 * 1024) continue;
      pl.split = s;
      pl.ksteps = nk / s;
      pl.stages = st;
      pl.smem_bytes = st * stage + 6 * 8 + 2 * st * 8 + 1024;
      break;
    }
  }
  return pl;
}

inline bool build_tc_supported(const void *X, int64_t ldx, const void *A_cat, const void *L, int64_t ldl,
                               int d_model, int n_cols, int dtype) {
  auto al16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  return dtype == FLA_BF16 && al16(X) && al16(A_cat) && al16(L) && ldx % 8 == 0 && ldl % 8 == 0 &&
         build_tc_shape_plan(d_model, n_cols).ok;
}

// Largest cluster (16, else 8) of this kernel that the device can place with
// `smem` bytes per CTA; cached per device and shared-memory size.
inline int build_max_cluster(int smem) {
  static std::mutex mu;
  static int cached_dev[kMaxDevices], cached_smem[kMaxDevices], cached_val[kMaxDevices];
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(mu);
  if (cached_smem[dev] == smem && cached_val[dev] > 0 && cached_dev[dev] == dev + 1) return cached_val[dev];
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
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, bld::build_tc_kernel, &cfg) == cudaSuccess && n >= 1) best = 16;
  }
  cudaGetLastError();  // a refused query leaves no sticky error
  cached_dev[dev] = dev + 1;
  cached_smem[dev] = smem;
  cached_val[dev] = best;
  return best;
}

inline fla_status build_tc_launch(const void *X, int64_t ldx, const void *A_cat, void *L, int64_t ldl, int64_t n,
                                  int d_model, int n_cols, cudaStream_t s) {
  BuildPlan pl = build_tc_plan(n, d_model, n_cols, device_sm_count(), 8);
  if (!pl.ok) {
    build_tc_err() = "shape outside the tensor-core build kernel";
    return FLA_ERR_UNSUPPORTED;
  }
  if (pl.split == 8) {  // try a 16-CTA cluster where the device can place one
    const BuildPlan p16 = build_tc_plan(n, d_model, n_cols, device_sm_count(), 16);
    if (p16.split == 16 && build_max_cluster(p16.smem_bytes) >= 16) pl = p16;
  }
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) {
    build_tc_err() = "cuTensorMapEncodeTiled is not available from the driver";
    return FLA_ERR_CUDA;
  }
  CUtensorMap mX, mA;
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
    // A_cat [d_model rows, n_cols columns], row-major: boxes of 64 columns x 64 rows
    const cuuint64_t dims[2] = {(cuuint64_t)n_cols, (cuuint64_t)d_model};
    const cuuint64_t strides[1] = {(cuuint64_t)n_cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)bld::kBoxN, (cuuint32_t)bld::kBK};
    if (enc(&mA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(A_cat), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      build_tc_err() = "encoding the A_cat tensor map failed";
      return FLA_ERR_CUDA;
    }
  }
  bld::Params prm{};
  prm.L = reinterpret_cast<__nv_bfloat16 *>(L);
  prm.ldl = ldl;
  prm.n = n;
  prm.K = d_model;
  prm.N = n_cols;
  prm.n_tile = pl.n_tile;
  prm.n_ntiles = pl.n_ntiles;
  prm.n_chunks = pl.n_chunks;
  prm.chunk_boxes[0] = pl.chunk_boxes[0];
  prm.chunk_boxes[1] = pl.chunk_boxes[1];
  prm.stages = pl.stages;
  prm.split = pl.split;
  prm.ksteps = pl.ksteps;
  prm.red_pitch = pl.red_pitch;
  prm.tmem_cols = pl.tmem_cols;
  const void *fn = reinterpret_cast<const void *>(bld::build_tc_kernel);
  cudaError_t e = ensure_dynamic_smem(fn, pl.smem_bytes);
  if (e != cudaSuccess) {
    build_tc_err() = cudaGetErrorString(e);
    return FLA_ERR_CUDA;
  }
  const int64_t grid = (n + bld::kBM - 1) / bld::kBM * pl.n_ntiles * pl.split;
  if (grid > 0x7fffffffLL) {
    build_tc_err() = "n_tokens too large";
    return FLA_ERR_UNSUPPORTED;
  }
  if (pl.split == 1) {
    bld::build_tc_kernel<<<(unsigned)grid, bld::kThreads, pl.smem_bytes, s>>>(mX, mA, prm);
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
  e = cudaLaunchKernelEx(&cfg, bld::build_tc_kernel, mX, mA, prm);
  if (e != cudaSuccess) {
    build_tc_err() = cudaGetErrorString(e);
    return FLA_ERR_CUDA;
  }
  return FLA_OK;
}

}  // namespace fla
