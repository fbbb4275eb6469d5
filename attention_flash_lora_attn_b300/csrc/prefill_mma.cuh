// Tensor-core chunked causal prefill (mma.sync): Flash-LoRA-Attention for the
// `chunk` new tokens of every agent over a shared context of n0 tokens.
//
// LRAgent technical summary (gist.science), Metodologia section 3: the
// output is P.V_base + (P.L_a).B_a with B_a applied once per query block;
// section 2 (BaseShared): K_base / V_base shared by every agent, so one CTA
// serves all agents' queries of a kv head from one read of each K/V tile.
// The query at chunk position p (absolute position n0 + p) sees keys
// 0 .. n0 + p.
//
// One CTA per (kv head h, block of QB consecutive chunk positions).  Its
// query rows are (agent a, q head g of the group, position pi), row =
// (a*G + g)*QB + pi, at most 128 rows = 8 tiles of 16; warp w owns row tile w.
// Key tiles of 64 tokens (K, V and the L columns of every agent) stream
// through a TMA ring; lane 0 of warp 0 refills a stage once all warps have
// released it.  Per tile each warp computes S = Q.K^T (16 x 64), the online
// softmax in registers, P.V_base and P.L_window with mma.sync m16n8k16; only
// tiles that reach the chunk apply the causal mask.  After the last tile each
// warp adds (P.L_a).B_a (bf16 high/low split) and writes its rows of O.
#pragma once

#include <cuda_bf16.h>

#include "../../include/flash_lora_attn.h"
#include "decode_tc.cuh"
#include "fla_common.cuh"
#include "ptx.cuh"

namespace fla {
namespace pre {

constexpr int kT = 64;          // keys per stage (each warp processes all of them)
constexpr int kMaxRows = 128;   // query rows per CTA
constexpr int kSmemBudget = 224 * 1024;

struct Params {
  const __nv_bfloat16 *Q, *B;
  float *O;
  int64_t n0;
  int32_t chunk, A, hq, hkv, G, r, QB, rows, rpa;  // rpa: rows per agent = G * QB
  int32_t l_agent_stride, l_width, l_box_cols, l_swz_bytes;
  int32_t stages, bs_bytes;
  float scale_log2;
};

template <int D, int MT, int NLT>
__global__ void __launch_bounds__(MT * 32, 1)
prefill_mma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmB,
                   const Params p) {
  constexpr int T = kT;
  constexpr int kNT = MT * 32;
  constexpr int kQPitch = D * 2 + 16;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int k_bytes = T * D * 2;
  const int stage_bytes = 2 * k_bytes + T * p.l_width * 2;
  uint8_t *bsm = smem + p.stages * stage_bytes;  // B slices [A][r][D] (16-row x 64-col boxes)
  uint8_t *q_smem = bsm + p.bs_bytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(q_smem + MT * 16 * kQPitch);
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x % p.hkv;
  const int qb = blockIdx.x / p.hkv;
  const int p0 = qb * p.QB;                                   // first chunk position of the block
  const int64_t n_keys = p.n0 + min(p.chunk, p0 + p.QB);     // keys any row of the block sees
  const int n_tiles = (int)((n_keys + T - 1) / T);
  const int64_t causal_from = p.n0 + p0;                      // keys >= this need the per-row mask
  const uint32_t full0 = ptx::smem_u32(&bars[0]);
  const uint32_t empty0 = ptx::smem_u32(&bars[p.stages]);
  const uint32_t bar_b = ptx::smem_u32(&bars[2 * p.stages]);
  const int n_lbox = p.l_width / p.l_box_cols;
  const int lbox_bytes = T * p.l_swz_bytes;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < p.stages; ++s) {
      ptx::mbar_init(full0 + 8 * s, 1);
      ptx::mbar_init(empty0 + 8 * s, MT);
    }
    ptx::mbar_init(bar_b, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();

  auto issue_tile = [&](int it) {
    const int st = it % p.stages;
    const uint32_t fb = full0 + 8 * st;
    ptx::mbar_arrive_expect_tx(fb, stage_bytes);
    const uint32_t sbase = ptx::smem_u32(smem + st * stage_bytes);
    const int tok = it * T;
#pragma unroll
    for (int b = 0; b < D / 64; ++b) {
      ptx::tma_load_3d(sbase + b * T * 128, &tmK, b * 64, head, tok, fb);
      ptx::tma_load_3d(sbase + k_bytes + b * T * 128, &tmV, b * 64, head, tok, fb);
    }
    for (int b = 0; b < n_lbox; ++b)
      ptx::tma_load_2d(sbase + 2 * k_bytes + b * lbox_bytes, &tmL, b * p.l_box_cols, tok, fb);
  };
  const bool producer = (threadIdx.x == 0);
  int last_issued = -1;
  if (producer) {
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
    ptx::prefetch_tmap(&tmL);
    for (int it = 0; it < p.stages && it < n_tiles; ++it) {
      issue_tile(it);
      last_issued = it;
    }
    ptx::mbar_arrive_expect_tx(bar_b, p.bs_bytes);
    for (int kc = 0; kc < p.A * p.r / 16; ++kc)
#pragma unroll
      for (int b = 0; b < D / 64; ++b)
        ptx::tma_load_2d(ptx::smem_u32(bsm) + (kc * (D / 64) + b) * 2048, &tmB, head * D + b * 64, kc * 16, bar_b);
  }

  // Q rows of this block into shared memory (zero rows beyond the valid ones)
  for (int e = threadIdx.x; e < MT * 16 * (D / 8); e += kNT) {
    const int row = e / (D / 8), c8 = e % (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < p.rows) {
      const int a = row / p.rpa, g = (row / p.QB) % p.G, pi = row % p.QB;
      const int pos = p0 + pi;
      if (pos < p.chunk)
        v = *reinterpret_cast<const uint4 *>(p.Q + (((int64_t)a * p.chunk + pos) * p.hq + head * p.G + g) * D +
                                             c8 * 8);
    }
    *reinterpret_cast<uint4 *>(q_smem + row * kQPitch + c8 * 16) = v;
  }
  __syncthreads();
  const int g8 = lane >> 2, t4 = lane & 3;
  uint32_t qf[D / 16][4];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int row = warp * 16 + (lane & 15);
    const int col = kk * 16 + (lane >> 4) * 8;
    ptx::ldsm_x4(ptx::smem_u32(q_smem + row * kQPitch + col * 2), qf[kk]);
  }

  // this warp's rows, their agents and causal limits (keys visible: < lim)
  const int row_lo = warp * 16;
  const int row0 = row_lo + g8, row1 = row_lo + g8 + 8;
  const int64_t lim0 = p.n0 + p0 + (row0 % p.QB) + 1;
  const int64_t lim1 = p.n0 + p0 + (row1 % p.QB) + 1;
  const int row_hi = min(p.rows, row_lo + 16) - 1;
  const int a_lo = row_lo / p.rpa;
  const int a_hi = row_hi >= row_lo ? row_hi / p.rpa : a_lo;
  const int c_lo = a_lo * p.l_agent_stride;
  const int win = (a_hi - a_lo) * p.l_agent_stride + p.r;

  float acc_v[D / 8][4];
  float acc_l[NLT][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) acc_v[i][0] = acc_v[i][1] = acc_v[i][2] = acc_v[i][3] = 0.f;
#pragma unroll
  for (int i = 0; i < NLT; ++i) acc_l[i][0] = acc_l[i][1] = acc_l[i][2] = acc_l[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float sl2 = p.scale_log2;
  bool aborted = false;

  for (int it = 0; it < n_tiles; ++it) {
    const int st = it % p.stages;
    if (!ptx::mbar_wait(full0 + 8 * st, (it / p.stages) & 1)) {
      set_device_error(kErrPrefillWait);
      aborted = true;
      break;
    }
    const uint32_t aK = ptx::smem_u32(smem + st * stage_bytes);
    const uint32_t aV = aK + k_bytes;
    const uint32_t aL = aK + 2 * k_bytes;
    const int64_t tile0 = (int64_t)it * T;

    // ---- S = Q . K^T  (16 rows x 64 keys)
    float s[T / 8][4];
#pragma unroll
    for (int i = 0; i < T / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < T / 16; ++np) {
        const int mi = lane >> 3, ri = lane & 7;
        const int tok = np * 16 + (mi >> 1) * 8 + ri;
        const int c16 = kk * 2 + (mi & 1);
        const uint32_t addr = aK + (c16 >> 3) * (T * 128) + tok * 128 + (dec::swz_chunk(c16 & 7, tok, 128) << 4);
        uint32_t kb[4];
        ptx::ldsm_x4(addr, kb);
        ptx::mma_bf16(s[2 * np], qf[kk], kb[0], kb[1]);
        ptx::mma_bf16(s[2 * np + 1], qf[kk], kb[2], kb[3]);
      }
    }
    // ---- causal mask on the tiles that reach the chunk (and the key tail)
    if (tile0 + T > causal_from) {
#pragma unroll
      for (int nt = 0; nt < T / 8; ++nt) {
        const int64_t t = tile0 + nt * 8 + 2 * t4;
        if (t >= lim0) s[nt][0] = -INFINITY;
        if (t + 1 >= lim0) s[nt][1] = -INFINITY;
        if (t >= lim1) s[nt][2] = -INFINITY;
        if (t + 1 >= lim1) s[nt][3] = -INFINITY;
      }
    }
    // ---- online softmax (log2 domain)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < T / 8; ++nt) {
      s[nt][0] *= sl2; s[nt][1] *= sl2; s[nt][2] *= sl2; s[nt][3] *= sl2;
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float ref0 = (mn0 == -INFINITY) ? 0.f : mn0;
    const float ref1 = (mn1 == -INFINITY) ? 0.f : mn1;
    const float corr0 = ptx::ex2(m0 - ref0), corr1 = ptx::ex2(m1 - ref1);
    m0 = mn0;
    m1 = mn1;
    uint32_t pa[T / 16][4];
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < T / 8; ++nt) {
      const float q0 = ptx::ex2(s[nt][0] - ref0), q1 = ptx::ex2(s[nt][1] - ref0);
      const float q2 = ptx::ex2(s[nt][2] - ref1), q3 = ptx::ex2(s[nt][3] - ref1);
      rs0 += q0 + q1;
      rs1 += q2 + q3;
      pa[nt >> 1][(nt & 1) * 2 + 0] = ptx::pack_bf16(q0, q1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = ptx::pack_bf16(q2, q3);
    }
    l0 = l0 * corr0 + rs0;
    l1 = l1 * corr1 + rs1;
    if (__any_sync(0xffffffffu, corr0 != 1.f || corr1 != 1.f)) {
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        acc_v[i][0] *= corr0; acc_v[i][1] *= corr0; acc_v[i][2] *= corr1; acc_v[i][3] *= corr1;
      }
#pragma unroll
      for (int i = 0; i < NLT; ++i) {
        acc_l[i][0] *= corr0; acc_l[i][1] *= corr0; acc_l[i][2] *= corr1; acc_l[i][3] *= corr1;
      }
    }
    // ---- acc_v += P . V_base ; acc_l += P . L_window
#pragma unroll
    for (int ks = 0; ks < T / 16; ++ks) {
      const int mi = lane >> 3, ri = lane & 7;
      const int tok = ks * 16 + (mi & 1) * 8 + ri;
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int c16 = dp * 2 + (mi >> 1);
        const uint32_t addr = aV + (c16 >> 3) * (T * 128) + tok * 128 + (dec::swz_chunk(c16 & 7, tok, 128) << 4);
        uint32_t vb[4];
        ptx::ldsm_x4_t(addr, vb);
        ptx::mma_bf16(acc_v[2 * dp], pa[ks], vb[0], vb[1]);
        ptx::mma_bf16(acc_v[2 * dp + 1], pa[ks], vb[2], vb[3]);
      }
#pragma unroll
      for (int lp = 0; lp < NLT / 2; ++lp) {
        if (lp * 16 >= win) break;  // warp-uniform
        int c8 = (c_lo >> 3) + lp * 2 + (mi >> 1);
        if (c8 * 8 >= p.l_width) c8 = 0;  // chunk past the tile: read a valid one, unused
        const int cb = c8 * 8;
        const int box = cb / p.l_box_cols;
        const int chunk = (cb % p.l_box_cols) >> 3;
        const uint32_t addr = aL + box * lbox_bytes + tok * p.l_swz_bytes +
                              (dec::swz_chunk(chunk, tok, p.l_swz_bytes) << 4);
        uint32_t lb[4];
        ptx::ldsm_x4_t(addr, lb);
        ptx::mma_bf16(acc_l[2 * lp], pa[ks], lb[0], lb[1]);
        if (lp * 16 + 8 < win) ptx::mma_bf16(acc_l[2 * lp + 1], pa[ks], lb[2], lb[3]);
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(empty0 + 8 * st);
    if (producer && it + p.stages < n_tiles) {
      if (!ptx::mbar_wait(empty0 + 8 * st, (it / p.stages) & 1)) {
        set_device_error(kErrPrefillWait);
        aborted = true;
        break;
      }
      issue_tile(it + p.stages);
      last_issued = it + p.stages;
    }
  }
  if (aborted) s_abort = 1;
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  __syncthreads();
  if (s_abort) {
    if (producer) {
      for (int it = last_issued; it >= 0 && it > last_issued - p.stages; --it)
        ptx::mbar_wait(full0 + 8 * (it % p.stages), (it / p.stages) & 1);
      ptx::mbar_wait(bar_b, 0);
    }
    return;
  }
  if (!ptx::mbar_wait(bar_b, 0)) {
    set_device_error(kErrPrefillWait);
    return;  // the only copy in flight is the one that never completed
  }

  // ---- acc_v += (P.L_a) . B_a for this warp's rows (K = window columns of agent a)
  {
    const int ag0 = row0 < p.rows ? row0 / p.rpa : -1;
    const int ag1 = row1 < p.rows ? row1 / p.rpa : -1;
#pragma unroll
    for (int ks = 0; ks < NLT / 2; ++ks) {
      if (ks * 16 >= win) break;  // warp-uniform
      for (int a = a_lo; a <= a_hi; ++a) {
        const int blk = a * p.l_agent_stride - c_lo;
        if (ks * 16 < blk || ks * 16 >= blk + p.r) continue;
        const int kb = ks * 16 - blk;
        const bool own0 = (ag0 == a), own1 = (ag1 == a);
        uint32_t ah[4], al[4];
        ah[0] = dec::pack_hi_lo(own0 ? acc_l[2 * ks][0] : 0.f, own0 ? acc_l[2 * ks][1] : 0.f, al[0]);
        ah[1] = dec::pack_hi_lo(own1 ? acc_l[2 * ks][2] : 0.f, own1 ? acc_l[2 * ks][3] : 0.f, al[1]);
        ah[2] = dec::pack_hi_lo(own0 ? acc_l[2 * ks + 1][0] : 0.f, own0 ? acc_l[2 * ks + 1][1] : 0.f, al[2]);
        ah[3] = dec::pack_hi_lo(own1 ? acc_l[2 * ks + 1][2] : 0.f, own1 ? acc_l[2 * ks + 1][3] : 0.f, al[3]);
        const int mi = lane >> 3, ri = lane & 7;
        const int rr = (mi & 1) * 8 + ri;
        const int kc = (a * p.r + kb) >> 4;
        const uint32_t bbox = ptx::smem_u32(bsm) + kc * (D / 64) * 2048 + rr * 128;
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          const int c16 = dp * 2 + (mi >> 1);
          uint32_t bb[4];
          ptx::ldsm_x4_t(bbox + (c16 >> 3) * 2048 + (dec::swz_chunk(c16 & 7, rr, 128) << 4), bb);
          ptx::mma_bf16(acc_v[2 * dp], ah, bb[0], bb[1]);
          ptx::mma_bf16(acc_v[2 * dp + 1], ah, bb[2], bb[3]);
          ptx::mma_bf16(acc_v[2 * dp], al, bb[0], bb[1]);
          ptx::mma_bf16(acc_v[2 * dp + 1], al, bb[2], bb[3]);
        }
      }
    }
  }

  // ---- O = (P.V_base + (P.L_a).B_a) / l, straight from the fragments
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int row = h2 ? row1 : row0;
    if (row >= p.rows) continue;
    const int a = row / p.rpa, g = (row / p.QB) % p.G, pos = p0 + row % p.QB;
    if (pos >= p.chunk) continue;
    float *o = p.O + (((int64_t)a * p.chunk + pos) * p.hq + head * p.G + g) * D;
    const float inv = h2 ? inv1 : inv0;
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
      *reinterpret_cast<float2 *>(o + i * 8 + 2 * t4) =
          make_float2(acc_v[i][2 * h2] * inv, acc_v[i][2 * h2 + 1] * inv);
  }
}

}  // namespace pre

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
inline const char *&prefill_tc_err() {
  static thread_local const char *e = "";
  return e;
}
inline const char *prefill_tc_last_error() { return prefill_tc_err(); }

struct PrefillPlan {
  int D, MT, NLT, QB, rows, l_width, l_box_cols, l_swz, stages, smem_bytes, bs_bytes;
  bool ok;
};

inline PrefillPlan prefill_tc_plan(const fla_attn_dims &d) {
  PrefillPlan pl{};
  pl.ok = false;
  if (d.dtype != FLA_BF16) return pl;
  if (d.head_dim != 64 && d.head_dim != 128) return pl;
  if (d.rank % 16 != 0 || d.rank > 64) return pl;
  if (d.l_agent_stride != 0 && d.l_agent_stride != d.rank) return pl;
  const int D = d.head_dim, r = d.rank, G = d.hq / d.hkv;
  const auto instanced = [D](int mt) { return D == 128 ? (mt >= 1 && mt <= 8) : (mt == 1 || mt == 2 || mt == 4 || mt == 8); };
  const int ag = d.n_agents * G;  // rows per chunk position
  if (ag > pre::kMaxRows) return pl;
  int QB = 1;
  while (ag * QB * 2 <= pre::kMaxRows) QB *= 2;
  while (QB > 1 && !instanced((ag * QB + 15) / 16)) QB /= 2;
  const int rows = ag * QB;
  const int MT = (rows + 15) / 16;
  if (!instanced(MT)) return pl;
  const int rpa = G * QB;
  int wmax = 0;
  for (int mt = 0; mt < MT; ++mt) {
    const int lo = mt * 16, hi = std::min(rows, lo + 16) - 1;
    wmax = std::max(wmax, (hi / rpa - lo / rpa) * (int)d.l_agent_stride + r);
  }
  if (wmax > 64) return pl;
  const int l_width = d.l_agent_stride == 0 ? r : d.n_agents * r;
  int swz = 0;
  if ((l_width * 2) % 128 == 0) swz = 128;
  else if ((l_width * 2) % 64 == 0) swz = 64;
  else if ((l_width * 2) % 32 == 0) swz = 32;
  else return pl;
  const int stage = 2 * pre::kT * D * 2 + pre::kT * l_width * 2;
  const int bs_bytes = d.n_agents * r * D * 2;
  const int fixed = MT * 16 * (D * 2 + 16) + bs_bytes + 64 * 8 + 1024;
  int stages = (pre::kSmemBudget - fixed) / stage;
  if (stages > 6) stages = 6;
  if (stages < 2) return pl;
  pl.D = D; pl.MT = MT; pl.NLT = 8; pl.QB = QB; pl.rows = rows;
  pl.l_width = l_width; pl.l_box_cols = swz / 2; pl.l_swz = swz;
  pl.stages = stages; pl.bs_bytes = bs_bytes;
  pl.smem_bytes = stages * stage + fixed + (2 * stages + 1) * 8;
  if (pl.smem_bytes > 227 * 1024) return pl;
  pl.ok = true;
  return pl;
}

inline bool prefill_tc_shape_supported(const fla_attn_dims &d) { return prefill_tc_plan(d).ok; }

inline fla_status prefill_tc_launch(const fla_attn_dims &d, float scale, const void *Q, const void *K,
                                    const void *V, const void *L, const void *B, int64_t n0, int chunk, float *O,
                                    cudaStream_t s) {
  const PrefillPlan pl = prefill_tc_plan(d);
  if (!pl.ok) {
    prefill_tc_err() = "shape outside the tensor-core prefill kernel";
    return FLA_ERR_UNSUPPORTED;
  }
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) {
    prefill_tc_err() = "cuTensorMapEncodeTiled is not available from the driver";
    return FLA_ERR_CUDA;
  }
  const int64_t n_total = n0 + chunk;
  CUtensorMap mK, mV, mL, mB;
  const cuuint32_t es[3] = {1, 1, 1};
  {
    const cuuint64_t dims[3] = {(cuuint64_t)d.head_dim, (cuuint64_t)d.hkv, (cuuint64_t)n_total};
    const cuuint64_t strides[2] = {(cuuint64_t)d.head_dim * 2, (cuuint64_t)d.hkv * d.head_dim * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)pre::kT};
    if (enc(&mK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(K), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&mV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(V), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      prefill_tc_err() = "encoding the K/V tensor maps failed";
      return FLA_ERR_CUDA;
    }
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)pl.l_width, (cuuint64_t)n_total};
    const cuuint64_t strides[1] = {(cuuint64_t)d.l_row_stride * 2};
    const cuuint32_t box[2] = {(cuuint32_t)pl.l_box_cols, (cuuint32_t)pre::kT};
    if (enc(&mL, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(L), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_enum(pl.l_swz), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      prefill_tc_err() = "encoding the L tensor map failed";
      return FLA_ERR_CUDA;
    }
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)d.hkv * d.head_dim, (cuuint64_t)d.n_agents * d.rank};
    const cuuint64_t strides[1] = {(cuuint64_t)d.hkv * d.head_dim * 2};
    const cuuint32_t box[2] = {64, 16};
    if (enc(&mB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(B), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      prefill_tc_err() = "encoding the B tensor map failed";
      return FLA_ERR_CUDA;
    }
  }
  pre::Params prm{};
  prm.Q = reinterpret_cast<const __nv_bfloat16 *>(Q);
  prm.B = reinterpret_cast<const __nv_bfloat16 *>(B);
  prm.O = O;
  prm.n0 = n0;
  prm.chunk = chunk;
  prm.A = d.n_agents; prm.hq = d.hq; prm.hkv = d.hkv; prm.G = d.hq / d.hkv; prm.r = d.rank;
  prm.QB = pl.QB; prm.rows = pl.rows; prm.rpa = prm.G * pl.QB;
  prm.l_agent_stride = (int)d.l_agent_stride; prm.l_width = pl.l_width; prm.l_box_cols = pl.l_box_cols;
  prm.l_swz_bytes = pl.l_swz;
  prm.stages = pl.stages; prm.bs_bytes = pl.bs_bytes;
  prm.scale_log2 = scale * 1.4426950408889634f;
  const int64_t grid64 = (int64_t)d.hkv * ((chunk + pl.QB - 1) / pl.QB);
  if (grid64 > 0x7fffffffLL) {
    prefill_tc_err() = "chunk too large";
    return FLA_ERR_UNSUPPORTED;
  }
  // heavy query blocks (most keys) first: the last blocks of the chunk see the most context
  cudaError_t e = cudaSuccess;
#define FLA_PRE_CASE(DD, MM)                                                                              \
  if (pl.D == DD && pl.MT == MM) {                                                                        \
    auto kern = pre::prefill_mma_kernel<DD, MM, 8>;                                                       \
    e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), pl.smem_bytes);                        \
    if (e == cudaSuccess) kern<<<(unsigned)grid64, MM * 32, pl.smem_bytes, s>>>(mK, mV, mL, mB, prm);     \
    if (e != cudaSuccess) {                                                                               \
      prefill_tc_err() = cudaGetErrorString(e);                                                           \
      return FLA_ERR_CUDA;                                                                                \
    }                                                                                                     \
    return FLA_OK;                                                                                        \
  }
  FLA_PRE_CASE(128, 8) FLA_PRE_CASE(128, 7) FLA_PRE_CASE(128, 6) FLA_PRE_CASE(128, 5)
  FLA_PRE_CASE(128, 4) FLA_PRE_CASE(128, 3) FLA_PRE_CASE(128, 2) FLA_PRE_CASE(128, 1)
  FLA_PRE_CASE(64, 8) FLA_PRE_CASE(64, 4) FLA_PRE_CASE(64, 2) FLA_PRE_CASE(64, 1)
#undef FLA_PRE_CASE
  prefill_tc_err() = "no kernel instance for this plan";
  return FLA_ERR_UNSUPPORTED;
}

}  // namespace fla
