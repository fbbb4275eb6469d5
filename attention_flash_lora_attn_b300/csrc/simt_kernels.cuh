// CUDA-core (SIMT) kernels: every supported shape, fp32 or bf16 storage.
//
// These are the general kernels of the library: they handle the shapes the
// tensor-core kernels do not (any head_dim <= 256 that is a multiple of 4, any
// rank <= 256, fp32 storage) and serve as the second GPU implementation the
// tests compare the tensor-core kernels with.
//
// Attention (decode and prefill), one CTA per query row:
//   LRAgent technical summary, Metodologia section 3 (Flash-LoRA-Attention):
//   the row's output is P.V_base + (P.L_a).B_a.  Four warps stream disjoint
//   token subsets with an online softmax (running max m, running sum l), each
//   lane holding d/32 entries of the d-wide P.V_base accumulator and r/32
//   entries of the r-wide P.L_a accumulator; the warps are merged in shared
//   memory and B_a's head slice is applied once in the epilogue.
#pragma once

#include "fla_common.cuh"

namespace fla {

constexpr int kSimtMaxD = 256;
constexpr int kSimtMaxR = 256;
constexpr int kSimtWarps = 4;

struct SimtAttnParams {
  const void *Q, *K, *V, *L, *B;
  float *O;
  const int32_t *offsets;  // decode: [n_req+1]; prefill: unused
  int64_t l_row_stride, l_agent_stride;
  int64_t n0;              // prefill: cached tokens before the chunk
  int32_t n_agents, hq, hkv, d, r;
  int32_t n_req, chunk;    // decode: n_req; prefill: chunk
  int32_t prefill;         // 0 = decode rows [q][a][j]; 1 = prefill rows [a][p][j]
  float scale;
};

template <typename T>
__global__ void __launch_bounds__(kSimtWarps * 32)
simt_attn_kernel(const SimtAttnParams p) {
  const int row = blockIdx.x;
  const int j = row % p.hq;
  const int G = p.hq / p.hkv;
  const int h = j / G;
  int a;
  int64_t t0, nvis;
  if (p.prefill) {
    const int pos = (row / p.hq) % p.chunk;
    a = row / (p.hq * p.chunk);
    t0 = 0;
    nvis = p.n0 + pos + 1;  // causal: keys 0 .. n0+pos inclusive
  } else {
    const int q = row / (p.hq * p.n_agents);
    a = (row / p.hq) % p.n_agents;
    t0 = p.offsets[q];
    nvis = (int64_t)p.offsets[q + 1] - t0;
  }

  __shared__ float q_s[kSimtMaxD];
  __shared__ float accv_s[kSimtWarps][kSimtMaxD];
  __shared__ float accl_s[kSimtWarps][kSimtMaxR];
  __shared__ float m_s[kSimtWarps], l_s[kSimtWarps];

  const T *Q = reinterpret_cast<const T *>(p.Q);
  const T *K = reinterpret_cast<const T *>(p.K);
  const T *V = reinterpret_cast<const T *>(p.V);
  const T *L = reinterpret_cast<const T *>(p.L);
  const T *B = reinterpret_cast<const T *>(p.B);
  const int d = p.d, r = p.r;
  for (int i = threadIdx.x; i < d; i += blockDim.x) q_s[i] = to_f32(Q[(int64_t)row * d + i]);
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float accv[kSimtMaxD / 32], accl[kSimtMaxR / 32];
#pragma unroll
  for (int i = 0; i < kSimtMaxD / 32; ++i) accv[i] = 0.f;
#pragma unroll
  for (int i = 0; i < kSimtMaxR / 32; ++i) accl[i] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int64_t kv_row = (int64_t)p.hkv * d;
  const int64_t lcol0 = (int64_t)a * p.l_agent_stride;

  for (int64_t t = warp; t < nvis; t += kSimtWarps) {
    const int64_t tok = t0 + t;
    const T *krow = K + tok * kv_row + (int64_t)h * d;
    float part = 0.f;
    for (int i = lane; i < d; i += 32) part += q_s[i] * to_f32(krow[i]);
    const float s = warp_sum(part) * p.scale;
    const float m_new = fmaxf(m, s);
    const float corr = expf(m - m_new);  // 0 when m == -inf
    const float pt = expf(s - m_new);
    l = l * corr + pt;
    m = m_new;
    const T *vrow = V + tok * kv_row + (int64_t)h * d;
#pragma unroll
    for (int i = 0; i < kSimtMaxD / 32; ++i) {
      const int c = lane + 32 * i;
      if (c < d) accv[i] = accv[i] * corr + pt * to_f32(vrow[c]);
    }
    const T *lrow = L + tok * p.l_row_stride + lcol0;
#pragma unroll
    for (int i = 0; i < kSimtMaxR / 32; ++i) {
      const int c = lane + 32 * i;
      if (c < r) accl[i] = accl[i] * corr + pt * to_f32(lrow[c]);
    }
  }

  // merge the warps' partial softmax states
#pragma unroll
  for (int i = 0; i < kSimtMaxD / 32; ++i) {
    const int c = lane + 32 * i;
    if (c < d) accv_s[warp][c] = accv[i];
  }
#pragma unroll
  for (int i = 0; i < kSimtMaxR / 32; ++i) {
    const int c = lane + 32 * i;
    if (c < r) accl_s[warp][c] = accl[i];
  }
  if (lane == 0) {
    m_s[warp] = m;
    l_s[warp] = l;
  }
  __syncthreads();

  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kSimtWarps; ++w) M = fmaxf(M, m_s[w]);
  float wgt[kSimtWarps];
  float Lsum = 0.f;
#pragma unroll
  for (int w = 0; w < kSimtWarps; ++w) {
    wgt[w] = (m_s[w] == -INFINITY) ? 0.f : expf(m_s[w] - M);
    Lsum += wgt[w] * l_s[w];
  }
  // merged P.L_a (r wide), then O = (merged P.V_base + (P.L_a).B_a) / l
  __shared__ float pl_s[kSimtMaxR];
  for (int c = threadIdx.x; c < r; c += blockDim.x) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kSimtWarps; ++w) v += wgt[w] * accl_s[w][c];
    pl_s[c] = v;
  }
  __syncthreads();
  const float inv = (nvis > 0) ? 1.f / Lsum : 0.f;
  const T *Ba = B + (int64_t)a * r * ((int64_t)p.hkv * d) + (int64_t)h * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kSimtWarps; ++w) v += wgt[w] * accv_s[w][c];
    float lora = 0.f;
    for (int k = 0; k < r; ++k) lora += pl_s[k] * to_f32(Ba[(int64_t)k * p.hkv * d + c]);
    p.O[(int64_t)row * d + c] = (nvis > 0) ? (v + lora) * inv : 0.f;
  }
}

// ---------------------------------------------------------------------------
// LR-cache build on CUDA cores: L[t, c] = sum_k X[t, k] * A_cat[k, c].
// 64x64 output tile per CTA, 256 threads with a 4x4 register tile each,
// k-steps of 16 staged in shared memory.  fp32 accumulation.
// ---------------------------------------------------------------------------
struct SimtBuildParams {
  const void *X, *A;  // A: the first of N columns of a row-major weight matrix with row stride lda
  void *L;
  int64_t ldx, ldl, n;
  int32_t D, N;
  int64_t lda;
};

template <typename T>
__global__ void __launch_bounds__(256) simt_build_kernel(const SimtBuildParams p) {
  __shared__ float xs[16][64 + 1];
  __shared__ float as[16][64 + 1];
  const T *X = reinterpret_cast<const T *>(p.X);
  const T *Ac = reinterpret_cast<const T *>(p.A);
  T *L = reinterpret_cast<T *>(p.L);
  const int64_t row0 = (int64_t)blockIdx.x * 64;
  const int col0 = blockIdx.y * 64;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < p.D; k0 += 16) {
    for (int e = threadIdx.x; e < 64 * 16; e += 256) {
      const int rr = e / 16, kk = e % 16;
      const int64_t gr = row0 + rr;
      const int gk = k0 + kk;
      xs[kk][rr] = (gr < p.n && gk < p.D) ? to_f32(X[gr * p.ldx + gk]) : 0.f;
      // A_cat rows are contiguous along the columns: consecutive threads read consecutive columns
      const int ak = e / 64, ac = e % 64;
      const int gc = col0 + ac, gka = k0 + ak;
      as[ak][ac] = (gc < p.N && gka < p.D) ? to_f32(Ac[(int64_t)gka * p.lda + gc]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float xv[4], av[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = as[kk][tx * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(xv[i], av[jj], acc[i][jj]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gr = row0 + ty * 4 + i;
    if (gr >= p.n) continue;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int gc = col0 + tx * 4 + jj;
      if (gc < p.N) L[gr * p.ldl + gc] = from_f32<T>(acc[i][jj]);
    }
  }
}

}  // namespace fla
