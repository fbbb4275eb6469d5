// Materialised value cache of every agent, V_i = V_base + L_i . B_i.
//
// LRAgent technical summary (gist.science), Metodologia section 1: an agent's
// value cache is the shared base part plus the adapter output; section 3
// (Problema): reconstructing that sum at full width for every agent is the
// cost Flash-LoRA-Attention removes.  These kernels perform exactly that
// reconstruction.  They are the first half of the naive-materialisation
// baseline the reordered decode is measured against (the second half is plain
// attention over each V_i); no attention path of the library calls them.
//
// Two forms.  bf16 storage with head_dim 64 / 128 and r % 16 == 0 runs the
// expansion as what it is, a GEMM [tokens, r] x [r, d] per agent and head plus
// V_base, on warp-level mma.sync; every other shape uses a CUDA-core kernel.
// Both give one CTA a range of token rows of one kv head (sized on the host
// for about four CTAs per SM), stage the head's columns of B for a group of
// agents in shared memory once, and then walk the rows with no further
// barrier.  fp32 accumulation, one rounding to the storage type per value.
// HBM traffic per call: V_base and L read once per agent group, A x V_base
// written; B is re-read from L2 by every CTA.
#pragma once

#include <cuda_bf16.h>

#include "fla_common.cuh"
#include "ptx.cuh"

namespace fla {

constexpr int kExpThreads = 256;
constexpr int kExpMmaWarps = 4;
constexpr int kExpMaxSmem = 96 * 1024;  // B of one agent group

struct ExpandParams {
  const void *V;
  const void *L;
  const void *B;
  void *Vout;
  int64_t n_tokens, l_row_stride, l_agent_stride;
  int32_t A, hkv, d, r;
  int32_t rows_per_cta, agents_per_group;
};

template <typename T>
__device__ __forceinline__ void load8(const T *src, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<float>(const float *src, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4 *>(src), b = *reinterpret_cast<const float4 *>(src + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *src, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4 *>(src);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <typename T>
__device__ __forceinline__ void store8(T *dst, const float (&v)[8]);
template <>
__device__ __forceinline__ void store8<float>(float *dst, const float (&v)[8]) {
  *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4 *>(dst + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16 *dst, const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = ptx::pack_bf16(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}

// CUDA-core form: each thread owns 8 consecutive columns of two token rows at
// a time, reads the rows' r values of L_a through the read-only cache (shared
// by the threads of a row) and B_a from shared memory (fp32).
template <typename T>
__global__ void __launch_bounds__(kExpThreads, 3) lora_value_expand_kernel(const ExpandParams p) {
  extern __shared__ __align__(16) float exp_smem[];  // [agent of group][r][d]: B_a[:, head*d : (head+1)*d]
  const int head = blockIdx.y;
  const int64_t t_begin = (int64_t)blockIdx.x * p.rows_per_cta;
  const int64_t t_end = t_begin + p.rows_per_cta < p.n_tokens ? t_begin + p.rows_per_cta : p.n_tokens;
  const int d = p.d, r = p.r;
  const int64_t row_elems = (int64_t)p.hkv * d;  // elements per token of V_base / V_i
  const int cg = d / 8;              // 8-column groups per token row (1..32)
  const int tpp = kExpThreads / cg;  // token rows per pass (>= 8)
  const int my_cg = threadIdx.x % cg, my_row = threadIdx.x / cg;
  const bool active = my_row < tpp;
  const T *V = reinterpret_cast<const T *>(p.V);
  const T *L = reinterpret_cast<const T *>(p.L);
  const T *B = reinterpret_cast<const T *>(p.B);
  T *Vo = reinterpret_cast<T *>(p.Vout);
  const int64_t col0 = (int64_t)head * d + my_cg * 8;

  for (int a0 = 0; a0 < p.A; a0 += p.agents_per_group) {
    const int ng = p.A - a0 < p.agents_per_group ? p.A - a0 : p.agents_per_group;
    __syncthreads();  // the previous group's B is no longer read
    for (int e = threadIdx.x; e < ng * r * d; e += kExpThreads) {
      const int ak = e / d, c = e - ak * d;  // ak = agent-in-group * r + k
      exp_smem[e] = to_f32<T>(B[((int64_t)a0 * r + ak) * row_elems + (int64_t)head * d + c]);
    }
    __syncthreads();
    if (!active) continue;
    for (int64_t row = t_begin + my_row; row < t_end; row += 2 * tpp) {
      const int64_t row2 = row + tpp;
      const bool has2 = row2 < t_end;
      float v0[8], v1[8];
      load8<T>(V + row * row_elems + col0, v0);
      if (has2) {
        load8<T>(V + row2 * row_elems + col0, v1);
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) v1[c] = 0.f;
      }
      for (int ai = 0; ai < ng; ++ai) {
        const int a = a0 + ai;
        const T *l0 = L + row * p.l_row_stride + a * p.l_agent_stride;
        const T *l1 = L + (has2 ? row2 : row) * p.l_row_stride + a * p.l_agent_stride;
        const float *bs = exp_smem + (int64_t)ai * r * d + my_cg * 8;
        float acc0[8], acc1[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          acc0[c] = v0[c];
          acc1[c] = v1[c];
        }
#pragma unroll 4
        for (int k = 0; k < r; ++k) {
          const float la = to_f32<T>(__ldg(l0 + k)), lb = to_f32<T>(__ldg(l1 + k));
          const float4 b0 = *reinterpret_cast<const float4 *>(bs + k * d);
          const float4 b1 = *reinterpret_cast<const float4 *>(bs + k * d + 4);
          acc0[0] = fmaf(la, b0.x, acc0[0]); acc0[1] = fmaf(la, b0.y, acc0[1]);
          acc0[2] = fmaf(la, b0.z, acc0[2]); acc0[3] = fmaf(la, b0.w, acc0[3]);
          acc0[4] = fmaf(la, b1.x, acc0[4]); acc0[5] = fmaf(la, b1.y, acc0[5]);
          acc0[6] = fmaf(la, b1.z, acc0[6]); acc0[7] = fmaf(la, b1.w, acc0[7]);
          acc1[0] = fmaf(lb, b0.x, acc1[0]); acc1[1] = fmaf(lb, b0.y, acc1[1]);
          acc1[2] = fmaf(lb, b0.z, acc1[2]); acc1[3] = fmaf(lb, b0.w, acc1[3]);
          acc1[4] = fmaf(lb, b1.x, acc1[4]); acc1[5] = fmaf(lb, b1.y, acc1[5]);
          acc1[6] = fmaf(lb, b1.z, acc1[6]); acc1[7] = fmaf(lb, b1.w, acc1[7]);
        }
        store8<T>(Vo + ((int64_t)a * p.n_tokens + row) * row_elems + col0, acc0);
        if (has2) store8<T>(Vo + ((int64_t)a * p.n_tokens + row2) * row_elems + col0, acc1);
      }
    }
  }
}

// Tensor-core form (bf16, head_dim 64 or 128, r % 16 == 0): each warp runs
// mma.sync m16n8k16 over 16 tokens and the head's d columns.  A = the tokens'
// L_a values (fragments loaded from global as bf16 pairs), B = B_a's head
// columns pre-packed once per CTA into fragment order in shared memory, C
// initialised with V_base (kept as packed bf16 across the agents) and rounded
// to bf16 on the way out.
template <int D>
__global__ void __launch_bounds__(kExpMmaWarps * 32, 3) lora_value_expand_mma_kernel(const ExpandParams p) {
  constexpr int NT = D / 8;  // n-tiles of the head
  extern __shared__ __align__(16) uint2 exp_frag[];  // [agent of group][k-step][n-tile][lane]
  const int head = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int KS = p.r / 16;
  const int64_t t_begin = (int64_t)blockIdx.x * p.rows_per_cta;
  const int64_t t_end = t_begin + p.rows_per_cta < p.n_tokens ? t_begin + p.rows_per_cta : p.n_tokens;
  const int64_t row_elems = (int64_t)p.hkv * D;
  const __nv_bfloat16 *V = reinterpret_cast<const __nv_bfloat16 *>(p.V);
  const __nv_bfloat16 *L = reinterpret_cast<const __nv_bfloat16 *>(p.L);
  const uint16_t *B = reinterpret_cast<const uint16_t *>(p.B);
  __nv_bfloat16 *Vo = reinterpret_cast<__nv_bfloat16 *>(p.Vout);
  const int64_t col_base = (int64_t)head * D + 2 * t4;

  for (int a0 = 0; a0 < p.A; a0 += p.agents_per_group) {
    const int ng = p.A - a0 < p.agents_per_group ? p.A - a0 : p.agents_per_group;
    __syncthreads();  // the previous group's fragments are no longer read
    for (int e = threadIdx.x; e < ng * KS * NT * 32; e += kExpMmaWarps * 32) {
      const int ln = e & 31, nt = (e >> 5) % NT, aks = (e >> 5) / NT;  // aks = agent-in-group * KS + k-step
      const int ai = aks / KS, ks = aks - ai * KS;
      const int n = head * D + nt * 8 + (ln >> 2), k0 = ks * 16 + 2 * (ln & 3);
      const uint16_t *bb = B + ((int64_t)(a0 + ai) * p.r + k0) * row_elems + n;
      exp_frag[e] = make_uint2((uint32_t)bb[0] | ((uint32_t)bb[row_elems] << 16),
                               (uint32_t)bb[8 * row_elems] | ((uint32_t)bb[9 * row_elems] << 16));
    }
    __syncthreads();
    for (int64_t t0 = t_begin + warp * 16; t0 < t_end; t0 += kExpMmaWarps * 16) {
      const int64_t r0 = t0 + g, r1 = t0 + g + 8;
      const bool ok0 = r0 < t_end, ok1 = r1 < t_end;
      uint32_t v[NT][2];  // V_base as bf16 pairs: [0] row g, [1] row g + 8
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        v[nt][0] = ok0 ? *reinterpret_cast<const uint32_t *>(V + r0 * row_elems + col_base + nt * 8) : 0u;
        v[nt][1] = ok1 ? *reinterpret_cast<const uint32_t *>(V + r1 * row_elems + col_base + nt * 8) : 0u;
      }
      for (int ai = 0; ai < ng; ++ai) {
        const int a = a0 + ai;
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          acc[nt][0] = __uint_as_float(v[nt][0] << 16);
          acc[nt][1] = __uint_as_float(v[nt][0] & 0xFFFF0000u);
          acc[nt][2] = __uint_as_float(v[nt][1] << 16);
          acc[nt][3] = __uint_as_float(v[nt][1] & 0xFFFF0000u);
        }
        const __nv_bfloat16 *l0 = L + r0 * p.l_row_stride + a * p.l_agent_stride + 2 * t4;
        const __nv_bfloat16 *l1 = L + r1 * p.l_row_stride + a * p.l_agent_stride + 2 * t4;
        const uint2 *fr = exp_frag + (int64_t)ai * KS * NT * 32 + lane;
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t af[4];
          af[0] = ok0 ? *reinterpret_cast<const uint32_t *>(l0 + ks * 16) : 0u;
          af[1] = ok1 ? *reinterpret_cast<const uint32_t *>(l1 + ks * 16) : 0u;
          af[2] = ok0 ? *reinterpret_cast<const uint32_t *>(l0 + ks * 16 + 8) : 0u;
          af[3] = ok1 ? *reinterpret_cast<const uint32_t *>(l1 + ks * 16 + 8) : 0u;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint2 b = fr[(ks * NT + nt) * 32];
            ptx::mma_bf16(acc[nt], af, b.x, b.y);
          }
        }
        __nv_bfloat16 *o0 = Vo + ((int64_t)a * p.n_tokens + r0) * row_elems + col_base;
        __nv_bfloat16 *o1 = Vo + ((int64_t)a * p.n_tokens + r1) * row_elems + col_base;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (ok0) *reinterpret_cast<uint32_t *>(o0 + nt * 8) = ptx::pack_bf16(acc[nt][0], acc[nt][1]);
          if (ok1) *reinterpret_cast<uint32_t *>(o1 + nt * 8) = ptx::pack_bf16(acc[nt][2], acc[nt][3]);
        }
      }
    }
  }
}

// Agents whose B columns of one head fit the shared-memory budget together
// (bytes per agent: r * d * 4 for the CUDA-core form, r * d * 2 packed for the
// mma.sync form); 0 when not even one fits.
inline int expand_agents_per_group(int A, int r, int d, bool mma) {
  const size_t per = (size_t)r * d * (mma ? 2 : 4);
  const int g = (int)(kExpMaxSmem / per);
  return g < A ? g : A;
}

// Token rows per CTA: about four CTAs per SM over the whole grid, 64..4096 rows.
inline int expand_rows_per_cta(int64_t n_tokens, int hkv, int sms) {
  const int64_t ctas = 4LL * sms;
  int64_t rows = (n_tokens * hkv + ctas - 1) / ctas;
  rows = (rows + 63) / 64 * 64;
  if (rows < 64) rows = 64;
  if (rows > 4096) rows = 4096;
  return (int)rows;
}

}  // namespace fla
