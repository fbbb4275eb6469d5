// Tensor-core LR-cache build: L = X . A_cat on tcgen05 (TMEM accumulators).
//
// LRAgent technical summary (gist.science), Metodologia section 2 (BaseShared:
// the LR cache holds the LoRA down-projection X.A_i at width r); PReCache
// abstract (PreLRShared: every agent's LR cache built in one pass over the
// context).  All agents' down-projections are stacked, A_t = [A_1|...|A_A]^T
// ([A*r, d_model], K-major), so one GEMM reads each row of X once and writes
// every agent's r columns: L[t, :] = X[t, :] . A_t^T.
//
// One CTA per 128-row tile of X, all N = A*r columns (<= 512) accumulated in
// tensor memory (N fp32 columns x 128 lanes):
//   warp 0     TMA producer: X tile [128 x 64] and A_t tile [N x 64] per k-step
//              (128-byte swizzle) into a ring of shared-memory stages;
//   warp 1     allocates TMEM; lane 0 issues tcgen05.mma (M = 128, N split in
//              chunks of <= 256, K = 16 per instruction) and tcgen05.commit to
//              release each stage and, at the end, to publish the accumulator;
//   warps 2-5  epilogue: tcgen05.ld of their 32-lane quarter, fp32 -> bf16,
//              stores to L.
// Every wait is bounded; on a timeout the CTA records the error, waits
// (bounded) for its copies and MMAs in flight, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>

#include "../../include/flash_lora_attn.h"
#include "fla_common.cuh"
#include "ptx.cuh"

namespace fla {
namespace bld {

constexpr int kBM = 128;       // rows of X per CTA (MMA M)
constexpr int kBK = 64;        // K per stage: one 128-byte swizzle row of bf16
constexpr int kThreads = 192;  // 6 warps
constexpr int kSmemBudget = 220 * 1024;

struct Params {
  __nv_bfloat16 *L;
  int64_t ldl, n;
  int32_t K;        // d_model
  int32_t N;        // columns of L (A * r)
  int32_t n_chunks; // MMA N split: chunk = N / n_chunks (multiple of 16, <= 256)
  int32_t stages;
  uint32_t tmem_cols;
};

__global__ void __launch_bounds__(kThreads, 1)
build_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmA, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int a_bytes = kBM * kBK * 2;
  const int b_bytes = p.N * kBK * 2;
  const int stage_bytes = a_bytes + b_bytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.stages * stage_bytes);
  // bars: full[stages] | empty[stages] | acc_full | drain
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m0 = (int64_t)blockIdx.x * kBM;
  const int n_k = p.K / kBK;
  const int chunk = p.N / p.n_chunks;
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
        ptx::mbar_arrive_expect_tx(fb, stage_bytes);
        const uint32_t sa = ptx::smem_u32(smem + s * stage_bytes);
        ptx::tma_load_2d(sa, &tmX, kt * kBK, (int32_t)m0, fb);
        for (int c = 0; c < p.n_chunks; ++c)
          ptx::tma_load_2d(sa + a_bytes + c * chunk * 128, &tmA, kt * kBK, c * chunk, fb);
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
      const uint32_t idesc = ptx::idesc_bf16_f32(kBM, chunk);
      const uint64_t d_smem = ptx::smem_desc_k128(ptx::smem_u32(smem));
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
        const uint64_t da = ptx::desc_advance(d_smem, s * stage_bytes);
        const uint64_t db = ptx::desc_advance(da, a_bytes);
#pragma unroll
        for (int k16 = 0; k16 < kBK / 16; ++k16) {
          const uint32_t acc = (kt > 0 || k16 > 0) ? 1u : 0u;
          for (int c = 0; c < p.n_chunks; ++c)
            ptx::tc_mma_f16(tmem + c * chunk, ptx::desc_advance(da, k16 * 32),
                            ptx::desc_advance(db, c * chunk * 128 + k16 * 32), idesc, acc);
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
    const int64_t row = m0 + quarter * 32 + lane;
    bool ready = false;
    // the accumulator arrives after the whole K loop: poll with a bound, but
    // stop early if the CTA aborted
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      if (ptx::mbar_try_wait(acc_full, 0)) { ready = true; break; }
      if (*(volatile int *)&s_abort) break;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        set_device_error(kErrBuildAccWait);
        break;
      }
    }
    if (ready) {
      ptx::tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
      for (int c0 = 0; c0 < p.N; c0 += 32) {
        uint32_t v[32];
        ptx::tmem_ld32(tl + c0, v);
        ptx::tmem_ld_wait();
        if (row < p.n) {
          uint4 out[4];
          uint32_t *o = reinterpret_cast<uint32_t *>(out);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            o[i] = ptx::pack_bf16(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          uint4 *dst = reinterpret_cast<uint4 *>(p.L + row * p.ldl + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = out[i];
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) ptx::tmem_dealloc(tmem, p.tmem_cols);
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
  int n_chunks, stages, smem_bytes;
  uint32_t tmem_cols;
  bool ok;
};

inline BuildPlan build_tc_plan(int d_model, int n_cols) {
  BuildPlan pl{};
  pl.ok = false;
  if (d_model % bld::kBK != 0 || n_cols % 32 != 0 || n_cols > 512 || n_cols < 32) return pl;
  int nc = (n_cols + 255) / 256;
  while (nc <= n_cols / 16 && (n_cols % nc != 0 || (n_cols / nc) % 16 != 0)) ++nc;
  if (n_cols % nc != 0 || (n_cols / nc) % 16 != 0 || n_cols / nc > 256) return pl;
  const int stage = (bld::kBM + n_cols) * bld::kBK * 2;
  int stages = (bld::kSmemBudget - 1024 - 64) / stage;
  if (stages > 8) stages = 8;
  if (stages < 2) return pl;
  uint32_t cols = 32;
  while ((int)cols < n_cols) cols <<= 1;
  pl.n_chunks = nc;
  pl.stages = stages;
  pl.smem_bytes = stages * stage + (2 * stages + 2) * 8 + 1024;
  pl.tmem_cols = cols;
  pl.ok = true;
  return pl;
}

inline bool build_tc_supported(const void *X, int64_t ldx, const void *A_t, const void *L, int64_t ldl, int d_model,
                               int n_cols, int dtype) {
  auto al16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  return dtype == FLA_BF16 && al16(X) && al16(A_t) && al16(L) && ldx % 8 == 0 && ldl % 8 == 0 &&
         build_tc_plan(d_model, n_cols).ok;
}

inline fla_status build_tc_launch(const void *X, int64_t ldx, const void *A_t, void *L, int64_t ldl, int64_t n,
                                  int d_model, int n_cols, cudaStream_t s) {
  const BuildPlan pl = build_tc_plan(d_model, n_cols);
  if (!pl.ok) {
    build_tc_err() = "shape outside the tensor-core build kernel";
    return FLA_ERR_UNSUPPORTED;
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
    const cuuint64_t dims[2] = {(cuuint64_t)d_model, (cuuint64_t)n_cols};
    const cuuint64_t strides[1] = {(cuuint64_t)d_model * 2};
    const cuuint32_t box[2] = {(cuuint32_t)bld::kBK, (cuuint32_t)(n_cols / pl.n_chunks)};
    if (enc(&mA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(A_t), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      build_tc_err() = "encoding the A_t tensor map failed";
      return FLA_ERR_CUDA;
    }
  }
  bld::Params prm{};
  prm.L = reinterpret_cast<__nv_bfloat16 *>(L);
  prm.ldl = ldl;
  prm.n = n;
  prm.K = d_model;
  prm.N = n_cols;
  prm.n_chunks = pl.n_chunks;
  prm.stages = pl.stages;
  prm.tmem_cols = pl.tmem_cols;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(bld::build_tc_kernel), pl.smem_bytes);
  if (e != cudaSuccess) {
    build_tc_err() = cudaGetErrorString(e);
    return FLA_ERR_CUDA;
  }
  const int64_t grid = (n + bld::kBM - 1) / bld::kBM;
  if (grid > 0x7fffffffLL) {
    build_tc_err() = "n_tokens too large";
    return FLA_ERR_UNSUPPORTED;
  }
  bld::build_tc_kernel<<<(unsigned)grid, bld::kThreads, pl.smem_bytes, s>>>(mX, mA, prm);
  return FLA_OK;
}

}  // namespace fla
