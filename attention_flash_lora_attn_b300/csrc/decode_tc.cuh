// Tensor-core decode kernel: Flash-LoRA-Attention over a shared base cache.
//
// LRAgent technical summary (gist.science), Metodologia section 3: the output
// is computed as P.V_base + (P.L_a).B_a, so the r-wide P.L_a accumulates in the
// same pass as the d-wide P.V_base and B_a is applied once per query, after
// the token loop.  Section 2 (BaseShared): K_base / V_base are one cache
// shared by every agent, so all agents' query rows of a kv head are served
// from one read of each K/V tile (like the query heads of a GQA group).
//
// Work decomposition.  A work item is (request q, kv head h, unit u): a
// contiguous range of at most `unit_tokens` tokens of request q.  One CTA per
// work item; the CTA index is unit * hkv + h so the kv heads of the same token
// range run side by side and share the L tile through L2 (map_unit gives the
// unit order).
//
// Inside a CTA (SG x MT x TG warps, no dedicated producer warp):
//   * the A*G query rows of kv head h (agent-major: row = a*G + g) are cut into
//     MT tiles of 16 rows; warp (sg, mt, tg) owns row tile mt and token slice
//     tg (16 tokens) of the stages of T = 16*TG tokens that warp group sg
//     consumes (tile i belongs to group i % SG);
//   * lane 0 of each group's first warp streams that group's token tiles with
//     TMA into a ring of shared-memory stages (K tile, V tile, and the L tile
//     holding every agent's r columns; 128/64/32-byte swizzle) guarded by
//     full/empty mbarriers, and refills a stage as soon as every warp of the
//     group has released it;
//   * S = Q.K^T, P.V_base and P.L_window run on mma.sync m16n8k16 (bf16 in,
//     fp32 accumulate); the online-softmax state (running max m, running sum
//     l) and both accumulators stay in registers, row reductions use quad
//     shuffles; the rescale is skipped when no running max moved;
//   * after the loop each warp adds (P.L_a).B_a to its P.V_base accumulator
//     with mma.sync, the r-wide P.L_a split into a bf16 high and low part so
//     the product keeps ~16 mantissa bits, rows masked to their own agent;
//   * the SG*TG token slices are merged in shared memory; a CTA that is the only
//     unit of its (q, h) writes O, otherwise it writes its partial
//     (m, l, d-wide accumulator) to the workspace;
//   * the merge kernel, launched right behind with programmatic dependent
//     launch (it waits on the grid dependency, no flag polling), combines the
//     partials of every (q, h) in unit order (deterministic) and writes O: one
//     warp per query row, every unit's load in flight at once.
#pragma once

#include <cuda_bf16.h>

#include <algorithm>

#include "../../include/flash_lora_attn.h"
#include "fla_common.cuh"
#include "ptx.cuh"

namespace fla {
namespace dec {

constexpr int kMaxRows = 64;         // A*G query rows per kv head (MT <= 4)
constexpr int kMaxUnitsPerPair = 128;
constexpr int kSmemBudget = 224 * 1024;
constexpr int kTW = 16;              // tokens per warp per stage

struct Params {
  const __nv_bfloat16 *Q, *B;
  float *O;
  const int32_t *offsets;
  float *partials;
  int2 *pair_info;         // per (q, head): first global unit, unit count (for the merge kernel)
  int32_t n_req, A, hq, hkv, G, r, rows;
  int32_t l_agent_stride;  // 0 or r
  int32_t l_width;         // columns of L held per token in shared memory
  int32_t l_box_cols;      // columns per L TMA box (16, 32 or 64)
  int32_t l_swz_bytes;     // 32, 64 or 128
  int32_t unit_tokens;
  int32_t stages;
  int32_t bs_dedicated;    // 1: B slices prefetched into their own region at kernel start
  int32_t single_len;      // n_req == 1: tokens of the request (no offsets scan); else -1
  int32_t part_stride;     // floats per unit partial in the workspace (multiple of 4)
  float scale_log2;        // softmax scale * log2(e)
};

// Shared-memory geometry of one pipeline stage.
struct StageGeom {
  int T, D, l_width, l_swz;
  __host__ __device__ int k_bytes() const { return T * D * 2; }
  __host__ __device__ int l_bytes() const { return T * l_width * 2; }
  __host__ __device__ int stage_bytes() const { return 2 * k_bytes() + l_bytes(); }
};

__device__ __forceinline__ int swz_chunk(int chunk, int row, int row_bytes) {
  // TMA swizzle: the 16-byte chunk index within a row_bytes span is XORed
  // with address bits 7.. of the row start (128B: 3 bits, 64B: 2, 32B: 1).
  return chunk ^ (((row * row_bytes) >> 7) & (row_bytes / 16 - 1));
}

// D: head_dim; MT: 16-row tiles; TG: token slices (warps) per row tile and
// stage; NLT: 8-column n-tiles of the L window; SG: warp groups taking
// alternate stages.
template <int D, int MT, int TG, int NLT, int SG>
struct Cfg {
  static constexpr int TW = kTW;
  static constexpr int T = TG * TW;
  static constexpr int kGroupWarps = MT * TG;
  static constexpr int kWarps = kGroupWarps * SG;
  static constexpr int kSlices = TG * SG;  // warps sharing one row tile
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kRowsPad = MT * 16;
  static constexpr int kQPitch = D * 2 + 16;  // bytes per Q row in shared memory
};

// Floats of the slice-merge exchange (aliased onto the stage ring after the
// token loop): every warp's fragments and running max / sum, then the merged
// max and sum of each row tile.
__host__ __device__ constexpr int merge_exchange_floats(int D, int MT, int TG, int NLT, int SG) {
  return MT * TG * SG * ((D / 8) * 4 + NLT * 4 + 4) * 32 + MT * 4 * 32;
}

__device__ __forceinline__ uint32_t pack_hi_lo(float x0, float x1, uint32_t &lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
  lo = ptx::pack_bf16(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
  return (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
}

// Maps a CTA's unit index (its position in the launch order) to s_info:
// [0] request q, [1] unit u of q, [2] units of q, [3] first token, [4] token
// count, [6] partial-record slot.  Returns whether the unit exists.  Run by one
// whole warp.  A request of length len has nu = max(1, ceil(len / U)) units;
// the slots of its units are contiguous (request-major), which is how the
// merge kernel finds them.
// Launch order (several requests): first every unit but the last of each
// request (all exactly U tokens, request order), then the last units, the
// larger first (a warp sort within each group of 32 requests), so the
// remainders fill the final wave and the grid ends on its shortest units.
__device__ __forceinline__ int map_unit(int unit_global, int U, int single_len, const int32_t *offsets, int n_req,
                                        int *s_info) {
  const int lane = threadIdx.x & 31;
  if (single_len >= 0) {  // one request: its length is known, no scan
    const int len = single_len;
    const int nu = len > 0 ? (len + U - 1) / U : 1;
    const int found = unit_global < nu;
    if (found && lane == 0) {
      s_info[0] = 0;
      s_info[1] = unit_global;
      s_info[2] = nu;
      s_info[3] = unit_global * U;
      s_info[4] = len > 0 ? min(U, len - unit_global * U) : 0;
      s_info[6] = unit_global;
    }
    return found;
  }
  auto units_of = [&](int q, int &len) {
    len = offsets[q + 1] - offsets[q];
    return len > 0 ? (len + U - 1) / U : 1;
  };
  // ---- pass 1: full units (all but each request's last), request order
  int base_f = 0, base_n = 0;
  for (int q0 = 0; q0 < n_req; q0 += 32) {
    const int q = q0 + lane;
    int len = 0, nu = 0;
    if (q < n_req) nu = units_of(q, len);
    const int f = q < n_req ? nu - 1 : 0;
    int incl_f = f, incl_n = nu;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int vf = __shfl_up_sync(0xffffffffu, incl_f, o), vn = __shfl_up_sync(0xffffffffu, incl_n, o);
      if (lane >= o) {
        incl_f += vf;
        incl_n += vn;
      }
    }
    const int excl_f = base_f + incl_f - f, excl_n = base_n + incl_n - nu;
    const bool mine = (q < n_req) && unit_global >= excl_f && unit_global < excl_f + f;
    if (__ballot_sync(0xffffffffu, mine)) {
      if (mine) {
        const int u = unit_global - excl_f;
        s_info[0] = q;
        s_info[1] = u;
        s_info[2] = nu;
        s_info[3] = offsets[q] + u * U;
        s_info[4] = U;
        s_info[6] = excl_n + u;
      }
      return 1;
    }
    base_f += __shfl_sync(0xffffffffu, incl_f, 31);
    base_n += __shfl_sync(0xffffffffu, incl_n, 31);
  }
  // ---- pass 2: the last unit of every request, larger first within each group of 32
  const int k = unit_global - base_f;
  if (k >= n_req) return 0;  // grid slack
  const int grp = k / 32, rank = k % 32;
  int slot_base = 0;  // units of the requests before this group
  for (int q0 = 0; q0 < grp * 32; q0 += 32) {
    int len, nu = 0;
    if (q0 + lane < n_req) nu = units_of(q0 + lane, len);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nu += __shfl_xor_sync(0xffffffffu, nu, o);
    slot_base += nu;
  }
  const int q = grp * 32 + lane;
  int len = 0, nu = 0, size = -1;
  if (q < n_req) {
    nu = units_of(q, len);
    size = len - (nu - 1) * U;  // 0 for an empty request
  }
  int incl_n = nu;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl_n, o);
    if (lane >= o) incl_n += v;
  }
  const int slot_last = slot_base + incl_n - 1;  // slot of this request's last unit
  // bitonic sort of (size, request) keys, descending size, ascending request on ties
  unsigned long long key = ((unsigned long long)(uint32_t)(size + 1) << 32) | (uint32_t)(0xffffffffu - (uint32_t)q);
#pragma unroll
  for (int k2 = 2; k2 <= 32; k2 <<= 1)
#pragma unroll
    for (int j = k2 >> 1; j > 0; j >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, j);
      const bool desc = (lane & k2) == 0 || k2 == 32;
      const bool lower = (lane & j) == 0;
      key = (desc == lower) ? (key > other ? key : other) : (key < other ? key : other);
    }
  const unsigned long long pick = __shfl_sync(0xffffffffu, key, rank);
  const int qs = (int)(0xffffffffu - (uint32_t)(pick & 0xffffffffull));
  const int src = qs - grp * 32;
  const int nus = __shfl_sync(0xffffffffu, nu, src);
  const int sizes = __shfl_sync(0xffffffffu, size, src);
  const int slots = __shfl_sync(0xffffffffu, slot_last, src);
  if (lane == 0) {
    s_info[0] = qs;
    s_info[1] = nus - 1;
    s_info[2] = nus;
    s_info[3] = offsets[qs] + (nus - 1) * U;
    s_info[4] = sizes;
    s_info[6] = slots;
  }
  return 1;
}

template <int D, int MT, int TG, int NLT, int SG>
__global__ void __launch_bounds__(Cfg<D, MT, TG, NLT, SG>::kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmB,
                 const Params p) {
  using C = Cfg<D, MT, TG, NLT, SG>;
  constexpr int TW = C::TW;
  constexpr int T = C::T;
  constexpr int kNT = C::kThreads;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const StageGeom geo{T, D, p.l_width, p.l_swz_bytes};
  const int stage_bytes = geo.stage_bytes();
  const int bs_bytes = p.A * p.r * D * 2;
  uint8_t *bsm = smem + p.stages * stage_bytes;  // dedicated B region (when bs_dedicated)
  uint8_t *q_smem = bsm + (p.bs_dedicated ? bs_bytes : 0);
  uint64_t *bars = reinterpret_cast<uint64_t *>(q_smem + C::kRowsPad * C::kQPitch);
  // bars: full[stages] | empty[stages] | B loaded | merge batch
  __shared__ int s_info[8];   // q, unit, n_units, token begin, token count, found
  __shared__ int s_flag[1];   // abort
  __shared__ int s_last_issue[8];  // last tile copied into each stage (drained on an abort)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x % p.hkv;
  const int unit_global = blockIdx.x / p.hkv;
  // Launched with programmatic dependent launch: the CTA may start while the
  // previous kernel of the stream (this library's merge or decode kernel)
  // drains.  The token loop reads only this call's inputs, which that kernel
  // does not write; griddepcontrol.wait runs before this CTA's first global
  // write (pair_info, partials, O: the previous call's merge reads the
  // workspace), so the loop overlaps the previous call's tail.

  // ---- map unit_global -> (request, unit) with a warp-parallel scan
  if (warp == 0) {
    const int found = map_unit(unit_global, p.unit_tokens, p.single_len, p.offsets, p.n_req, s_info);
    if (lane == 0) {
      s_info[5] = found;
      s_flag[0] = 0;
      for (int s = 0; s < 8; ++s) s_last_issue[s] = -1;
      for (int s = 0; s < p.stages; ++s) {
        ptx::mbar_init(ptx::smem_u32(&bars[s]), 1);                   // full: one arrive + tx bytes
        ptx::mbar_init(ptx::smem_u32(&bars[p.stages + s]), C::kGroupWarps);  // empty: one arrive per warp of the group
      }
      ptx::mbar_init(ptx::smem_u32(&bars[2 * p.stages]), 1);      // B slices loaded
      ptx::mbar_init(ptx::smem_u32(&bars[2 * p.stages + 1]), 1);  // merge batch loaded
      ptx::fence_mbar_init();
    }
  }
  __syncthreads();
  // the merge kernel behind this one may be scheduled now; it still waits for
  // this grid to finish before reading the partials
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!s_info[5]) return;  // grid slack beyond the last unit
  const int q = s_info[0], unit = s_info[1], n_units = s_info[2];
  const int tok_begin = s_info[3], n_tok = s_info[4], slot = s_info[6];
  // every (q, head) tells the merge kernel where its units start and how many
  // there are (the workspace is not initialised; single-unit pairs are skipped)
  const int n_tiles = (n_tok + T - 1) / T;
  const uint32_t bar_full0 = ptx::smem_u32(&bars[0]);
  const uint32_t bar_empty0 = ptx::smem_u32(&bars[p.stages]);
  const int grp = warp / C::kGroupWarps;  // warp group: consumes tiles grp, grp + SG, ...
  const bool producer = (threadIdx.x == grp * C::kGroupWarps * 32);
  const int n_lbox = p.l_width / p.l_box_cols;
  const int lbox_bytes = T * p.l_swz_bytes;

  auto issue_tile = [&](int it) {
    const int st = it % p.stages;
    s_last_issue[st] = it;
    const uint32_t fb = bar_full0 + 8 * st;
    ptx::mbar_arrive_expect_tx(fb, stage_bytes);
    const uint32_t sbase = ptx::smem_u32(smem + st * stage_bytes);
    const int tok = tok_begin + it * T;
#pragma unroll
    for (int b = 0; b < D / 64; ++b) {
      ptx::tma_load_3d(sbase + b * T * 128, &tmK, b * 64, head, tok, fb);
      ptx::tma_load_3d(sbase + geo.k_bytes() + b * T * 128, &tmV, b * 64, head, tok, fb);
    }
    for (int b = 0; b < n_lbox; ++b)
      ptx::tma_load_2d(sbase + 2 * geo.k_bytes() + b * lbox_bytes, &tmL, b * p.l_box_cols, tok, fb);
  };
  // B_a[:, h*d:(h+1)*d] of every agent: boxes of 16 rows x 64 columns, 128B swizzle
  const uint32_t bar_b = ptx::smem_u32(&bars[2 * p.stages]);
  auto issue_B = [&](uint32_t dst) {
    ptx::mbar_arrive_expect_tx(bar_b, bs_bytes);
    for (int kc = 0; kc < p.A * p.r / 16; ++kc)
#pragma unroll
      for (int b = 0; b < D / 64; ++b)
        ptx::tma_load_2d(dst + (kc * (D / 64) + b) * 2048, &tmB, head * D + b * 64, kc * 16, bar_b);
  };
  // Q rows of this kv head (zero rows beyond A*G): the global loads are issued
  // before the stage ring's copies so they are not queued behind them
  constexpr int kQChunks = C::kRowsPad * (D / 8);
  constexpr int kQPerThread = (kQChunks + kNT - 1) / kNT;
  uint4 qv[kQPerThread];
#pragma unroll
  for (int i = 0; i < kQPerThread; ++i) {
    const int e = threadIdx.x + i * kNT;
    const int row = e / (D / 8), c8 = e % (D / 8);
    qv[i] = make_uint4(0, 0, 0, 0);
    if (e < kQChunks && row < p.rows) {
      const int a = row / p.G, j = head * p.G + row % p.G;
      qv[i] = *reinterpret_cast<const uint4 *>(p.Q + (((int64_t)q * p.A + a) * p.hq + j) * D + c8 * 8);
    }
  }
  if (producer) {
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
    ptx::prefetch_tmap(&tmL);
    for (int it = grp; it < p.stages && it < n_tiles; it += SG) {
      issue_tile(it);
    }
    // B is applied here only when this CTA is the only unit of its (q, head);
    // otherwise the merge kernel applies it once after combining the units
    if (p.bs_dedicated && grp == 0 && n_units == 1) issue_B(ptx::smem_u32(bsm));
  }

  const int mt = (warp % C::kGroupWarps) / TG, tg = warp % TG;
  const int g = lane >> 2, t4 = lane & 3;

#pragma unroll
  for (int i = 0; i < kQPerThread; ++i) {
    const int e = threadIdx.x + i * kNT;
    if (e < kQChunks)
      *reinterpret_cast<uint4 *>(q_smem + (e / (D / 8)) * C::kQPitch + (e % (D / 8)) * 16) = qv[i];
  }
  __syncthreads();
  uint32_t qf[D / 16][4];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int row = mt * 16 + (lane & 15);
    const int col = kk * 16 + (lane >> 4) * 8;
    ptx::ldsm_x4(ptx::smem_u32(q_smem + row * C::kQPitch + col * 2), qf[kk]);
  }

  // L column window of this row tile: agents a_lo..a_hi of rows [16mt, 16mt+16)
  const int row_lo = mt * 16;
  const int row_hi = min(p.rows, row_lo + 16) - 1;
  const int a_lo = row_lo / p.G;
  const int a_hi = row_hi >= row_lo ? row_hi / p.G : a_lo;
  const int c_lo = a_lo * p.l_agent_stride;
  const int win = (a_hi - a_lo) * p.l_agent_stride + p.r;  // columns actually used

  float acc_v[D / 8][4];
  float acc_l[NLT][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) acc_v[i][0] = acc_v[i][1] = acc_v[i][2] = acc_v[i][3] = 0.f;
#pragma unroll
  for (int i = 0; i < NLT; ++i) acc_l[i][0] = acc_l[i][1] = acc_l[i][2] = acc_l[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float sl2 = p.scale_log2;
  bool aborted = false;

  for (int it = grp; it < n_tiles; it += SG) {
    const int st = it % p.stages;
    if (!ptx::mbar_wait(bar_full0 + 8 * st, (it / p.stages) & 1)) {
      set_device_error(kErrDecodeFullWait);
      aborted = true;
      break;
    }
    const uint32_t aK = ptx::smem_u32(smem + st * stage_bytes);
    const uint32_t aV = aK + geo.k_bytes();
    const uint32_t aL = aK + 2 * geo.k_bytes();
    const int tok0 = tg * TW;  // first token of this warp's slice within the tile

    // ---- S = Q . K^T  (16 rows x TW tokens)
    float s[TW / 8][4];
#pragma unroll
    for (int i = 0; i < TW / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < TW / 16; ++np) {
        const int mi = lane >> 3, ri = lane & 7;
        const int tok = tok0 + np * 16 + (mi >> 1) * 8 + ri;
        const int c16 = kk * 2 + (mi & 1);
        const uint32_t addr = aK + (c16 >> 3) * (T * 128) + tok * 128 + (swz_chunk(c16 & 7, tok, 128) << 4);
        uint32_t kb[4];
        ptx::ldsm_x4(addr, kb);
        ptx::mma_bf16(s[2 * np], qf[kk], kb[0], kb[1]);
        ptx::mma_bf16(s[2 * np + 1], qf[kk], kb[2], kb[3]);
      }
    }
    // ---- mask tokens past the end of this unit (last tile only)
    const int valid = n_tok - it * T - tok0;  // tokens of this slice that exist
    if (valid < TW) {
#pragma unroll
      for (int nt = 0; nt < TW / 8; ++nt) {
        const int c = nt * 8 + 2 * t4;
        if (c >= valid) { s[nt][0] = -INFINITY; s[nt][2] = -INFINITY; }
        if (c + 1 >= valid) { s[nt][1] = -INFINITY; s[nt][3] = -INFINITY; }
      }
    }
    // ---- online softmax (log2 domain)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < TW / 8; ++nt) {
      s[nt][0] *= sl2; s[nt][1] *= sl2; s[nt][2] *= sl2; s[nt][3] *= sl2;
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    // reference points: finite even when every score so far is masked
    const float ref0 = (mn0 == -INFINITY) ? 0.f : mn0;
    const float ref1 = (mn1 == -INFINITY) ? 0.f : mn1;
    const float corr0 = ptx::ex2(m0 - ref0), corr1 = ptx::ex2(m1 - ref1);
    m0 = mn0;
    m1 = mn1;
    uint32_t pa[TW / 16][4];
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < TW / 8; ++nt) {
      const float p0 = ptx::ex2(s[nt][0] - ref0), p1 = ptx::ex2(s[nt][1] - ref0);
      const float p2 = ptx::ex2(s[nt][2] - ref1), p3 = ptx::ex2(s[nt][3] - ref1);
      rs0 += p0 + p1;
      rs1 += p2 + p3;
      pa[nt >> 1][(nt & 1) * 2 + 0] = ptx::pack_bf16(p0, p1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = ptx::pack_bf16(p2, p3);
    }
    l0 = l0 * corr0 + rs0;
    l1 = l1 * corr1 + rs1;
    // rescale only when some row's running max moved (rare after the first tiles)
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
    for (int ks = 0; ks < TW / 16; ++ks) {
      const int mi = lane >> 3, ri = lane & 7;
      const int tok = tok0 + ks * 16 + (mi & 1) * 8 + ri;
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int c16 = dp * 2 + (mi >> 1);
        const uint32_t addr = aV + (c16 >> 3) * (T * 128) + tok * 128 + (swz_chunk(c16 & 7, tok, 128) << 4);
        uint32_t vb[4];
        ptx::ldsm_x4_t(addr, vb);
        ptx::mma_bf16(acc_v[2 * dp], pa[ks], vb[0], vb[1]);
        ptx::mma_bf16(acc_v[2 * dp + 1], pa[ks], vb[2], vb[3]);
      }
#pragma unroll
      for (int lp = 0; lp < NLT / 2; ++lp) {
        if (lp * 16 >= win) break;  // warp-uniform
        int c8 = (c_lo >> 3) + lp * 2 + (mi >> 1);  // 8-column chunk within the L row
        if (c8 * 8 >= p.l_width) c8 = 0;            // chunk past the tile: read a valid one, unused
        const int cb = c8 * 8;
        const int box = cb / p.l_box_cols;
        const int chunk = (cb % p.l_box_cols) >> 3;
        const uint32_t addr = aL + box * lbox_bytes + tok * p.l_swz_bytes +
                              (swz_chunk(chunk, tok, p.l_swz_bytes) << 4);
        uint32_t lb[4];
        ptx::ldsm_x4_t(addr, lb);
        ptx::mma_bf16(acc_l[2 * lp], pa[ks], lb[0], lb[1]);
        if (lp * 16 + 8 < win) ptx::mma_bf16(acc_l[2 * lp + 1], pa[ks], lb[2], lb[3]);
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar_empty0 + 8 * st);
    // ---- refill: once every warp of the group has released this stage, load
    //      tile it + stages into it (with an odd stage count that tile belongs
    //      to the other group, whose warps wait on this stage's full barrier)
    if (producer && it + p.stages < n_tiles) {
      if (!ptx::mbar_wait(bar_empty0 + 8 * st, (it / p.stages) & 1)) {
        set_device_error(kErrDecodeEmptyWait);
        aborted = true;
        break;
      }
      issue_tile(it + p.stages);
    }
  }
  if (aborted) s_flag[0] = 1;

  // ---- row sums across the quad
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  __syncthreads();
  if (s_flag[0]) {
    // Do not leave while copies are in flight: wait (bounded) for the last
    // load issued into each stage.
    if (threadIdx.x == 0) {
      for (int st = 0; st < p.stages; ++st) {
        const int it = s_last_issue[st];
        if (it >= 0) ptx::mbar_wait(bar_full0 + 8 * st, (it / p.stages) & 1);
      }
    }
    if (producer && p.bs_dedicated && grp == 0 && n_units == 1) ptx::mbar_wait(bar_b, 0);
    return;
  }
  // Every issued tile was waited on by every warp, so no TMA write is pending:
  // the stage ring is reused below.

  // ---- merge the SG*TG token slices of each row tile in one pass: every warp
  //      publishes its fragments into the free ring (one float4 per n-tile and
  //      lane, thread-linear, conflict-free); after one barrier each warp
  //      combines a strided share of the n-tiles over all slices of its row
  //      tile.  A CTA that is one of several units of its (q, head) stores the
  //      result straight into its partial record ([rows][D + r] (P.V_base |
  //      own agent's P.L_a) | m[rows] | l[rows]); the only unit of a context
  //      writes it into the slot of the tile's slice 0 (and the tile's running
  //      max and row sum into a small table) for the B epilogue below.
  const bool single = (n_units == 1);
  const int W = D + p.r;
  float *part = p.partials + ((int64_t)slot * p.hkv + head) * p.part_stride;
  if (!single) {
    // the first global write: the previous grid of the stream (this library's
    // merge, which reads the workspace) must have finished
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (unit == 0 && threadIdx.x == 0) p.pair_info[q * p.hkv + head] = make_int2(slot - unit, n_units);
  }
  constexpr int NS = C::kSlices;
  constexpr int NQ = D / 8 + NLT;  // float4 groups per lane: acc_v n-tiles | acc_l n-tiles
  constexpr int NV4 = NQ + 1;      // + (m0, m1, l0, l1)
  static_assert(NQ % NS == 0, "slices must divide the n-tile count");
  const int kslice = grp * TG + tg;  // this warp's slice within its row tile
  float4 *xch = reinterpret_cast<float4 *>(smem);  // [warp][NV4][32 lanes]
  float4 *mlx = xch + C::kWarps * NV4 * 32;        // [row tile][32 lanes]: merged (M0, M1, L0, L1)
  auto slice_warp = [&](int k) { return (k / TG) * C::kGroupWarps + mt * TG + (k % TG); };
  {
    float4 *dst = xch + warp * NV4 * 32 + lane;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) dst[i * 32] = make_float4(acc_v[i][0], acc_v[i][1], acc_v[i][2], acc_v[i][3]);
#pragma unroll
    for (int i = 0; i < NLT; ++i)
      dst[(D / 8 + i) * 32] = make_float4(acc_l[i][0], acc_l[i][1], acc_l[i][2], acc_l[i][3]);
    dst[NQ * 32] = make_float4(m0, m1, l0, l1);
  }
  __syncthreads();
  {
    float f0[NS], f1[NS];
    float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      const float4 ml = xch[(slice_warp(k) * NV4 + NQ) * 32 + lane];
      f0[k] = ml.x;
      f1[k] = ml.y;
      M0 = fmaxf(M0, ml.x);
      M1 = fmaxf(M1, ml.y);
    }
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      f0[k] = (f0[k] == -INFINITY) ? 0.f : ptx::ex2(f0[k] - M0);
      f1[k] = (f1[k] == -INFINITY) ? 0.f : ptx::ex2(f1[k] - M1);
    }
    const int r0 = row_lo + g, r1 = row_lo + g + 8;  // this lane's rows (x, y: r0; z, w: r1)
    // own agent's first column within the tile's L window, per row
    const int blk0 = (r0 / p.G - a_lo) * p.l_agent_stride, blk1 = (r1 / p.G - a_lo) * p.l_agent_stride;
#pragma unroll
    for (int jj = 0; jj < NQ / NS; ++jj) {
      const int i = jj * NS + kslice;  // fragment elements x, y: row g; z, w: row g + 8
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        const float4 v = xch[(slice_warp(k) * NV4 + i) * 32 + lane];
        acc.x = fmaf(f0[k], v.x, acc.x);
        acc.y = fmaf(f0[k], v.y, acc.y);
        acc.z = fmaf(f1[k], v.z, acc.z);
        acc.w = fmaf(f1[k], v.w, acc.w);
      }
      if (single) {
        xch[(slice_warp(0) * NV4 + i) * 32 + lane] = acc;  // n-tile i is read and written by this warp alone
      } else if (i < D / 8) {
        const int col = i * 8 + 2 * t4;
        if (r0 < p.rows) *reinterpret_cast<float2 *>(part + r0 * W + col) = make_float2(acc.x, acc.y);
        if (r1 < p.rows) *reinterpret_cast<float2 *>(part + r1 * W + col) = make_float2(acc.z, acc.w);
      } else {
        const int cc = (i - D / 8) * 8 + 2 * t4;  // window column (cc, cc + 1 share an agent: r is even)
        if (r0 < p.rows && cc >= blk0 && cc < blk0 + p.r)
          *reinterpret_cast<float2 *>(part + r0 * W + D + cc - blk0) = make_float2(acc.x, acc.y);
        if (r1 < p.rows && cc >= blk1 && cc < blk1 + p.r)
          *reinterpret_cast<float2 *>(part + r1 * W + D + cc - blk1) = make_float2(acc.z, acc.w);
      }
    }
    if (kslice == 0) {
      float L0 = 0.f, L1 = 0.f;
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        const float4 ml = xch[(slice_warp(k) * NV4 + NQ) * 32 + lane];
        L0 = fmaf(f0[k], ml.z, L0);
        L1 = fmaf(f1[k], ml.w, L1);
      }
      if (single) {
        mlx[mt * 32 + lane] = make_float4(M0, M1, L0, L1);
      } else if (t4 == 0) {
        if (r0 < p.rows) {
          part[p.rows * W + r0] = M0;
          part[p.rows * W + p.rows + r0] = L0;
        }
        if (r1 < p.rows) {
          part[p.rows * W + r1] = M1;
          part[p.rows * W + p.rows + r1] = L1;
        }
      }
    }
  }
  if (!single) return;  // the partial record is complete
  __syncthreads();

  // ---- the only unit of its context: (P.L_a).B_a and O, in this CTA
  const int row0 = row_lo + g, row1 = row_lo + g + 8;
  if (kslice == 0) {
    const float4 *src = xch + warp * NV4 * 32 + lane;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      const float4 v = src[i * 32];
      acc_v[i][0] = v.x; acc_v[i][1] = v.y; acc_v[i][2] = v.z; acc_v[i][3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < NLT; ++i) {
      const float4 v = src[(D / 8 + i) * 32];
      acc_l[i][0] = v.x; acc_l[i][1] = v.y; acc_l[i][2] = v.z; acc_l[i][3] = v.w;
    }
    const float4 ml = mlx[mt * 32 + lane];
    l0 = ml.z;
    l1 = ml.w;
  }
  if (!p.bs_dedicated) {
    // the B slices are staged in the ring the fragments were just read from
    ptx::fence_proxy_async_smem();
    __syncthreads();
  }
  // ---- B slices: prefetched at the start, or loaded now into the free ring
  uint8_t *bs = p.bs_dedicated ? bsm : smem;
  if (!p.bs_dedicated && threadIdx.x == 0) issue_B(ptx::smem_u32(bs));
  if (!ptx::mbar_wait(bar_b, 0)) {
    set_device_error(kErrDecodeFullWait);
    return;  // the only copy in flight is the one that never completed
  }
  if (kslice != 0) return;
  // ---- acc_v += (P.L_a) . B_a for this warp's rows (K = window columns of agent a)
  {
    const int ag0 = row0 < p.rows ? row0 / p.G : -1;
    const int ag1 = row1 < p.rows ? row1 / p.G : -1;
#pragma unroll
    for (int ks = 0; ks < NLT / 2; ++ks) {
      if (ks * 16 >= win) break;  // warp-uniform
      for (int a = a_lo; a <= a_hi; ++a) {
        const int blk = a * p.l_agent_stride - c_lo;          // agent a's first window column
        if (ks * 16 < blk || ks * 16 >= blk + p.r) continue;  // this k-step is not agent a's
        const int kb = ks * 16 - blk;                          // first row of B_a for this k-step
        const bool own0 = (ag0 == a), own1 = (ag1 == a);
        uint32_t ah[4], al[4];
        ah[0] = pack_hi_lo(own0 ? acc_l[2 * ks][0] : 0.f, own0 ? acc_l[2 * ks][1] : 0.f, al[0]);
        ah[1] = pack_hi_lo(own1 ? acc_l[2 * ks][2] : 0.f, own1 ? acc_l[2 * ks][3] : 0.f, al[1]);
        ah[2] = pack_hi_lo(own0 ? acc_l[2 * ks + 1][0] : 0.f, own0 ? acc_l[2 * ks + 1][1] : 0.f, al[2]);
        ah[3] = pack_hi_lo(own1 ? acc_l[2 * ks + 1][2] : 0.f, own1 ? acc_l[2 * ks + 1][3] : 0.f, al[3]);
        const int mi = lane >> 3, ri = lane & 7;
        const int rr = (mi & 1) * 8 + ri;                 // row within the 16-row box
        const int kc = (a * p.r + kb) >> 4;               // 16-row box index
        const uint32_t bbox = ptx::smem_u32(bs) + kc * (D / 64) * 2048 + rr * 128;
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          const int c16 = dp * 2 + (mi >> 1);
          uint32_t bb[4];
          ptx::ldsm_x4_t(bbox + (c16 >> 3) * 2048 + (swz_chunk(c16 & 7, rr, 128) << 4), bb);
          ptx::mma_bf16(acc_v[2 * dp], ah, bb[0], bb[1]);
          ptx::mma_bf16(acc_v[2 * dp + 1], ah, bb[2], bb[3]);
          ptx::mma_bf16(acc_v[2 * dp], al, bb[0], bb[1]);
          ptx::mma_bf16(acc_v[2 * dp + 1], al, bb[2], bb[3]);
        }
      }
    }
  }
  // ---- O = (P.V_base + (P.L_a).B_a) / l, straight from the fragments
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (unit == 0 && threadIdx.x == 0) p.pair_info[q * p.hkv + head] = make_int2(slot - unit, n_units);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int row = h2 ? row1 : row0;
    if (row >= p.rows) continue;
    const int a = row / p.G, j = head * p.G + row % p.G;
    float *o = p.O + (((int64_t)q * p.A + a) * p.hq + j) * D;
    const float inv = h2 ? inv1 : inv0;
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
      *reinterpret_cast<float2 *>(o + i * 8 + 2 * t4) =
          make_float2(acc_v[i][2 * h2] * inv, acc_v[i][2 * h2 + 1] * inv);
  }
}

// ---------------------------------------------------------------------------
// Split merge and B epilogue.  For every (q, head) whose context was split
// into units u with partials (m_u, l_u, acc_u = P_u.V_base, pl_u = P_u.L_a):
//   w_u = 2^(m_u - max_u m_u)          (log2-domain running maxima)
//   O   = (sum_u w_u acc_u + (sum_u w_u pl_u) . B_a[:, h*d:(h+1)*d]) / sum_u w_u l_u
// units combined in order (deterministic).  Two geometries: one warp per
// query row (32 rows per CTA) when the merge fits on the SMs the decode grid
// leaves idle or the rows have few units; four warps per row otherwise
// (units split by index and combined in shared memory in fixed order, the
// agent's B slice staged before the wait; one row per CTA, so the merge
// spreads over every SM).  Launched with programmatic dependent
// launch right behind the decode kernel; griddepcontrol.wait returns once the
// decode grid has completed and its writes are visible.  The next decode may
// start its token loop while this decode's tail and this kernel run.
// ---------------------------------------------------------------------------

struct MergeParams {
  const float *partials;
  const int2 *pair_info;
  const __nv_bfloat16 *B;
  float *O;
  int32_t n_req, A, hq, hkv, G, r, rows, part_stride, unit_tokens, single_len;
  int32_t merge_single;  // 1: single-unit pairs have a partial too (finish them here)
};

// Two warps per query row (kMergeLaneWarps / 2 rows per CTA), at most 128
// registers a thread.  Each warp combines half of the row's units, CH units
// per round of loads; the second half is folded into the first through shared
// memory (first half first: a fixed order).  The first warp of a row loads the
// first RB rows of its B slice into registers before the wait, so once the
// decode grid ends only the partials' loads and the combine remain.  A
// single-request decode leaves enough SMs idle for every merge warp (see
// decode_unit_tokens), so the whole merge grid is resident early and the next
// decode can launch behind it.
constexpr int kMergeLaneWarps = 8;
static_assert(kMergeLaneWarps / 2 <= 4, "one named barrier (ids 1..4) per row of a CTA");

template <int D>
__global__ void __launch_bounds__(kMergeLaneWarps * 32, 2) decode_merge_lane_kernel(const MergeParams p) {
  constexpr int CPL = D / 32;  // accumulator columns per lane
  constexpr int RB = 16;       // rows of B held in registers from before the wait
  constexpr int CH = 8;        // units loaded per round
  __shared__ float xw[kMergeLaneWarps / 2][CPL + 4][32];  // the second warp's state, per row
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rl = warp >> 1, half = warp & 1;
  const int gr = blockIdx.x * (kMergeLaneWarps / 2) + rl;
  // the next decode may be scheduled now (see decode_merge_row_kernel)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (gr >= p.n_req * p.hkv * p.rows) return;  // both warps of the row
  const int pair = gr / p.rows, row = gr - pair * p.rows;
  const int q = pair / p.hkv, head = pair - q * p.hkv;
  const int a = row / p.G, j = head * p.G + row % p.G;
  // B_a[:, h*d:(h+1)*d] is an input: this lane's columns of its first RB rows
  const __nv_bfloat16 *bcol = p.B + (int64_t)a * p.r * p.hkv * D + head * D + lane * CPL;
  const int64_t bstride = (int64_t)p.hkv * D;
  uint32_t bpre[RB][CPL / 2];
#pragma unroll
  for (int i = 0; i < RB; ++i) {
    if (half == 0 && i < p.r) {
      if constexpr (CPL == 4) {
        const uint2 t = __ldg(reinterpret_cast<const uint2 *>(bcol + i * bstride));
        bpre[i][0] = t.x;
        bpre[i][1] = t.y;
      } else {
        bpre[i][0] = __ldg(reinterpret_cast<const uint32_t *>(bcol + i * bstride));
      }
    } else {
#pragma unroll
      for (int c = 0; c < CPL / 2; ++c) bpre[i][c] = 0u;
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int ug0, nu;
  if (p.single_len >= 0) {
    ug0 = 0;
    nu = p.single_len > 0 ? (p.single_len + p.unit_tokens - 1) / p.unit_tokens : 1;
  } else {
    const int2 info = __ldcg(p.pair_info + pair);
    ug0 = info.x;
    nu = info.y;
  }
  if (nu <= 1 && !p.merge_single) return;  // written directly by the decode kernel (both warps)
  const int W = D + p.r;
  const int64_t ustride = (int64_t)p.hkv * p.part_stride;
  const float *base = p.partials + ((int64_t)ug0 * p.hkv + head) * p.part_stride;
  const int nh = (nu + 1) / 2;
  const int ub = half ? nh : 0, ue = half ? nu : nh;  // this warp's units
  float M = -INFINITY, lsum = 0.f, acc[CPL], pl[2] = {0.f, 0.f};
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
  for (int u0 = ub; u0 < ue; u0 += CH) {
    float mu[CH], lu[CH], v[CH][CPL], a2[CH][2];
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int u = min(u0 + k, ue - 1);
      const float *src = base + u * ustride;
      mu[k] = __ldcg(src + p.rows * W + row);
      lu[k] = __ldcg(src + p.rows * W + p.rows + row);
      if constexpr (CPL == 4) {
        const float4 t = __ldcg(reinterpret_cast<const float4 *>(src + row * W) + lane);
        v[k][0] = t.x; v[k][1] = t.y; v[k][2] = t.z; v[k][3] = t.w;
      } else {
#pragma unroll
        for (int c = 0; c < CPL; ++c) v[k][c] = __ldcg(src + row * W + lane * CPL + c);
      }
      a2[k][0] = lane < p.r ? __ldcg(src + row * W + D + lane) : 0.f;
      a2[k][1] = lane + 32 < p.r ? __ldcg(src + row * W + D + 32 + lane) : 0.f;
    }
    float Mc = M;
#pragma unroll
    for (int k = 0; k < CH; ++k)
      if (u0 + k < ue) Mc = fmaxf(Mc, mu[k]);
    const float sc = (M == -INFINITY) ? 0.f : ptx::ex2(M - Mc);
    M = Mc;
    lsum *= sc;
    pl[0] *= sc;
    pl[1] *= sc;
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] *= sc;
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      if (u0 + k < ue) {
        const float w = (mu[k] == -INFINITY) ? 0.f : ptx::ex2(mu[k] - M);
        lsum += w * lu[k];
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[c] += w * v[k][c];
        pl[0] += w * a2[k][0];
        pl[1] += w * a2[k][1];
      }
    }
  }
  // fold the second half into the first
  if (half) {
    xw[rl][0][lane] = M;
    xw[rl][1][lane] = lsum;
    xw[rl][2][lane] = pl[0];
    xw[rl][3][lane] = pl[1];
#pragma unroll
    for (int c = 0; c < CPL; ++c) xw[rl][4 + c][lane] = acc[c];
  }
  // the row's two warps (constant barrier ids keep the CTA's barrier count low)
  switch (rl) {
    case 0: asm volatile("bar.sync 1, 64;" ::: "memory"); break;
    case 1: asm volatile("bar.sync 2, 64;" ::: "memory"); break;
    case 2: asm volatile("bar.sync 3, 64;" ::: "memory"); break;
    default: asm volatile("bar.sync 4, 64;" ::: "memory"); break;
  }
  if (half) return;
  {
    const float M1 = xw[rl][0][lane];
    const float Mt = fmaxf(M, M1);
    const float w0 = (M == -INFINITY) ? 0.f : ptx::ex2(M - Mt);
    const float w1 = (M1 == -INFINITY) ? 0.f : ptx::ex2(M1 - Mt);
    lsum = w0 * lsum + w1 * xw[rl][1][lane];
    pl[0] = w0 * pl[0] + w1 * xw[rl][2][lane];
    pl[1] = w0 * pl[1] + w1 * xw[rl][3][lane];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = w0 * acc[c] + w1 * xw[rl][4 + c][lane];
  }
  // (sum_u w_u pl_u) . B_a[:, h*d:(h+1)*d]: lane k holds pl[k] (and pl[k + 32] when r > 32)
  float lora[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) lora[c] = 0.f;
#pragma unroll
  for (int i = 0; i < RB; ++i) {
    const float plk = __shfl_sync(0xffffffffu, pl[0], i);
    if (i < p.r) {
#pragma unroll
      for (int c = 0; c < CPL / 2; ++c) {
        lora[2 * c] += plk * __uint_as_float(bpre[i][c] << 16);
        lora[2 * c + 1] += plk * __uint_as_float(bpre[i][c] & 0xffff0000u);
      }
    }
  }
  // the remaining rows of B (ranks above RB), eight in flight at a time
  constexpr int KB = 8;
  for (int k0 = RB; k0 < p.r; k0 += KB) {
    uint32_t bv[KB][CPL / 2];
#pragma unroll
    for (int i = 0; i < KB; ++i) {
      const int k = min(k0 + i, p.r - 1);
      if constexpr (CPL == 4) {
        const uint2 t = __ldg(reinterpret_cast<const uint2 *>(bcol + k * bstride));
        bv[i][0] = t.x;
        bv[i][1] = t.y;
      } else {
        bv[i][0] = __ldg(reinterpret_cast<const uint32_t *>(bcol + k * bstride));
      }
    }
#pragma unroll
    for (int i = 0; i < KB; ++i) {
      const int k = k0 + i;
      const float plk = __shfl_sync(0xffffffffu, k < 32 ? pl[0] : pl[1], k & 31);
      if (k < p.r) {
#pragma unroll
        for (int c = 0; c < CPL / 2; ++c) {
          lora[2 * c] += plk * __uint_as_float(bv[i][c] << 16);
          lora[2 * c + 1] += plk * __uint_as_float(bv[i][c] & 0xffff0000u);
        }
      }
    }
  }
  float *out = p.O + (((int64_t)q * p.A + a) * p.hq + j) * D + lane * CPL;
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  if constexpr (CPL == 4) {
    *reinterpret_cast<float4 *>(out) =
        make_float4((acc[0] + lora[0]) * inv, (acc[1] + lora[1]) * inv, (acc[2] + lora[2]) * inv,
                    (acc[3] + lora[3]) * inv);
  } else {
#pragma unroll
    for (int c = 0; c < CPL; ++c) out[c] = (acc[c] + lora[c]) * inv;
  }
}

// Four warps per query row, one row per CTA (the geometry for rows with many
// units): this row's B_a slice is staged in shared memory before the wait, and
// the rank is applied by one warp after a fixed-order combine.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_row_kernel(const MergeParams p) {
  extern __shared__ __align__(16) uint8_t msm[];
  constexpr int CPL = D / 32;  // accumulator columns per lane
  __nv_bfloat16 *Bs = reinterpret_cast<__nv_bfloat16 *>(msm);  // [r][D] of this row's agent
  float *red = reinterpret_cast<float *>(msm + (size_t)p.r * D * 2);  // [4 warps][32 lanes][CPL + 4]
  const int pair = blockIdx.x;
  const int q = pair / p.hkv, head = pair % p.hkv;
  const int row = blockIdx.y;
  const int a = row / p.G, j = head * p.G + row % p.G;
  const int r = p.r;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // B_a[:, h*d:(h+1)*d] is an input: stage it before waiting on the decode grid
  for (int e = threadIdx.x; e < r * (D / 8); e += 128) {
    const int k = e / (D / 8), c8 = e - k * (D / 8);
    reinterpret_cast<uint4 *>(Bs)[e] =
        *reinterpret_cast<const uint4 *>(p.B + ((int64_t)(a * r + k) * p.hkv + head) * D + c8 * 8);
  }
  // The next decode may be scheduled as soon as every CTA of this grid is
  // resident: its token loop reads only its own inputs and it waits for this
  // grid before its first global write.  Every grid waited on is then fully
  // resident (a dependent launches only once all CTAs of its primary have
  // issued this instruction), so the chain decode -> merge -> decode cannot
  // deadlock on SM space.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int ug0, nu;
  if (p.single_len >= 0) {
    ug0 = 0;
    nu = p.single_len > 0 ? (p.single_len + p.unit_tokens - 1) / p.unit_tokens : 1;
  } else {
    const int2 info = __ldcg(p.pair_info + pair);
    ug0 = info.x;
    nu = info.y;
  }
  if (nu <= 1 && !p.merge_single) return;  // written directly by the decode kernel (uniform over the CTA)
  const int W = D + r;
  const int64_t ustride = (int64_t)p.hkv * p.part_stride;
  const float *base = p.partials + ((int64_t)ug0 * p.hkv + head) * p.part_stride;
  // warp w combines units w, w + 4, ... ; eight of them in flight per step
  float M = -INFINITY, lsum = 0.f, acc[CPL], pl[2] = {0.f, 0.f};
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
  constexpr int CH = 8;
  for (int u0 = warp; u0 < nu; u0 += 4 * CH) {
    float mu[CH], lu[CH], v[CH][CPL], a2[CH][2];
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int u = min(u0 + 4 * k, nu - 1);
      const float *src = base + u * ustride;
      mu[k] = __ldcg(src + p.rows * W + row);
      lu[k] = __ldcg(src + p.rows * W + p.rows + row);
      if constexpr (CPL == 4) {
        const float4 t = __ldcg(reinterpret_cast<const float4 *>(src + row * W) + lane);
        v[k][0] = t.x; v[k][1] = t.y; v[k][2] = t.z; v[k][3] = t.w;
      } else {
#pragma unroll
        for (int c = 0; c < CPL; ++c) v[k][c] = __ldcg(src + row * W + lane * CPL + c);
      }
      a2[k][0] = lane < r ? __ldcg(src + row * W + D + lane) : 0.f;
      a2[k][1] = lane + 32 < r ? __ldcg(src + row * W + D + 32 + lane) : 0.f;
    }
    float Mc = M;
#pragma unroll
    for (int k = 0; k < CH; ++k)
      if (u0 + 4 * k < nu) Mc = fmaxf(Mc, mu[k]);
    const float sc = (M == -INFINITY) ? 0.f : ptx::ex2(M - Mc);
    M = Mc;
    lsum *= sc;
    pl[0] *= sc;
    pl[1] *= sc;
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] *= sc;
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      if (u0 + 4 * k < nu) {
        const float w = (mu[k] == -INFINITY) ? 0.f : ptx::ex2(mu[k] - M);
        lsum += w * lu[k];
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[c] += w * v[k][c];
        pl[0] += w * a2[k][0];
        pl[1] += w * a2[k][1];
      }
    }
  }
  // combine the four warps (fixed order: deterministic)
  float *my = red + (warp * 32 + lane) * (CPL + 4);
  my[0] = M;
  my[1] = lsum;
  my[2] = pl[0];
  my[3] = pl[1];
#pragma unroll
  for (int c = 0; c < CPL; ++c) my[4 + c] = acc[c];
  __syncthreads();
  if (warp != 0) return;
  float Mt = -INFINITY;
#pragma unroll
  for (int w = 0; w < 4; ++w) Mt = fmaxf(Mt, red[(w * 32 + lane) * (CPL + 4)]);
  float ls = 0.f, plt[2] = {0.f, 0.f}, at[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) at[c] = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float *o = red + (w * 32 + lane) * (CPL + 4);
    const float wt = (o[0] == -INFINITY) ? 0.f : ptx::ex2(o[0] - Mt);
    ls += wt * o[1];
    plt[0] += wt * o[2];
    plt[1] += wt * o[3];
#pragma unroll
    for (int c = 0; c < CPL; ++c) at[c] += wt * o[4 + c];
  }
  // (sum_u w_u pl_u) . B_a: lane k holds pl[k] (and pl[k + 32] when r > 32)
  float lora[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) lora[c] = 0.f;
  const __nv_bfloat16 *bs = Bs + lane * CPL;
  for (int k = 0; k < r; ++k) {
    const float plk = __shfl_sync(0xffffffffu, k < 32 ? plt[0] : plt[1], k & 31);
#pragma unroll
    for (int c = 0; c < CPL; ++c) lora[c] += plk * __bfloat162float(bs[k * D + c]);
  }
  float *out = p.O + (((int64_t)q * p.A + a) * p.hq + j) * D + lane * CPL;
  const float inv = ls > 0.f ? 1.f / ls : 0.f;
#pragma unroll
  for (int c = 0; c < CPL; ++c) out[c] = (at[c] + lora[c]) * inv;
}

}  // namespace dec

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
inline const char *&decode_tc_err() {
  static thread_local const char *e = "";
  return e;
}
inline const char *decode_tc_last_error() { return decode_tc_err(); }
inline const char *decode_tc_limits() {
  return "bf16; head_dim 64 or 128; rank % 16 == 0 and <= 64; l_agent_stride 0 or rank; n_agents*hq/hkv <= 64; "
         "L window per 16-row tile <= 128 columns; loaded L width % 16 == 0; 16-byte aligned pointers; "
         "l_row_stride % 8 == 0";
}

struct DecodePlan {
  int D, MT, TG, NLT, SG;
  int rows, l_width, l_box_cols, l_swz;
  int T, stages, smem_bytes, part_stride, bs_dedicated;
  bool ok;
};

// two_per_sm: a single-row-tile shape may use one warp group and at most
// kTwoPerSmBudget bytes of shared memory, so two CTAs share an SM (a CTA's
// setup, first loads and epilogue then overlap its neighbour's token loop);
// this pays off when the grid spans several waves.
constexpr int kTwoPerSmBudget = 110 * 1024;

inline DecodePlan decode_tc_plan(const fla_attn_dims &d, bool two_per_sm = false) {
  DecodePlan pl{};
  pl.ok = false;
  if (d.dtype != FLA_BF16) return pl;
  if (d.head_dim != 64 && d.head_dim != 128) return pl;
  if (d.rank % 16 != 0 || d.rank > 64) return pl;
  if (d.l_agent_stride != 0 && d.l_agent_stride != d.rank) return pl;
  const int D = d.head_dim, r = d.rank;
  const int G = d.hq / d.hkv;
  const int rows = d.n_agents * G;
  if (rows > dec::kMaxRows) return pl;
  const int MT = (rows + 15) / 16;
  // widest L window over the row tiles
  int wmax = 0;
  for (int mt = 0; mt < MT; ++mt) {
    const int lo = mt * 16, hi = std::min(rows, lo + 16) - 1;
    const int w = (hi / G - lo / G) * (int)d.l_agent_stride + r;
    wmax = std::max(wmax, w);
  }
  if (wmax > 128) return pl;
  const int NLT = wmax <= 64 ? 8 : 16;
  const int l_width = d.l_agent_stride == 0 ? r : d.n_agents * r;
  int swz = 0;
  if ((l_width * 2) % 128 == 0) swz = 128;
  else if ((l_width * 2) % 64 == 0) swz = 64;
  else if ((l_width * 2) % 32 == 0) swz = 32;
  else return pl;
  // eight warps (two per scheduler) where the row tiles allow it; a single row
  // tile uses two warp groups on alternate 64-token stages (more, smaller
  // stages in flight than one group of eight on 128-token stages), or one
  // group of four in the two-CTAs-per-SM layout
  const bool two = two_per_sm && MT == 1;
  const int TG = MT <= 2 ? 4 : 2;
  const int SG = (MT == 1 && !two) ? 2 : 1;
  const int budget = two ? kTwoPerSmBudget : dec::kSmemBudget;
  const int T = TG * dec::kTW;
  const int stage = 2 * T * D * 2 + T * l_width * 2;
  const int q_bytes = MT * 16 * (D * 2 + 16);
  // the slice-merge exchange is aliased onto the stage ring after the main loop
  const int bs_bytes = d.n_agents * r * D * 2;
  const int ring_min = std::max(dec::merge_exchange_floats(D, MT, TG, NLT, SG) * 4, 2 * stage);
  const int fixed = q_bytes + (2 * 8 + 2) * 8 + 1024;
  // B slices (needed in this kernel only by single-unit contexts) get their own
  // region, prefetched at kernel start, when that costs no stage; otherwise
  // they are loaded into the ring after the token loop
  auto fit = [&](bool ded, int &st, int &smem) {
    st = (budget - fixed - (ded ? bs_bytes : 0)) / stage;
    if (st > 8) st = 8;
    // a multiple of the warp groups: an odd count was measured no faster (the
    // token loop is bound by the memory system's latency under load, which
    // grows with the bytes in flight)
    st -= st % SG;
    if (st < 2) st = 2;
    while (st * stage < std::max(ring_min, ded ? 0 : bs_bytes)) st += SG;
    smem = st * stage + (ded ? bs_bytes : 0) + fixed;
    return smem <= (two ? kTwoPerSmBudget : 227 * 1024);
  };
  int st_plain, sm_plain, st_ded, sm_ded;
  const bool ok_plain = fit(false, st_plain, sm_plain);
  const bool ok_ded = fit(true, st_ded, sm_ded);
  int bs_dedicated, stages;
  if (ok_ded && (st_ded >= st_plain || !ok_plain)) {
    bs_dedicated = 1;
    stages = st_ded;
    pl.smem_bytes = sm_ded;
  } else if (ok_plain) {
    bs_dedicated = 0;
    stages = st_plain;
    pl.smem_bytes = sm_plain;
  } else {
    return pl;
  }
  pl.bs_dedicated = bs_dedicated;
  pl.D = D; pl.MT = MT; pl.TG = TG; pl.NLT = NLT; pl.SG = SG;
  pl.rows = rows; pl.l_width = l_width; pl.l_box_cols = swz / 2; pl.l_swz = swz;
  pl.T = T; pl.stages = stages;
  pl.part_stride = (rows * (D + r + 2) + 3) & ~3;
  pl.ok = true;
  return pl;
}

inline bool decode_tc_shape_supported(const fla_attn_dims &d) { return decode_tc_plan(d).ok; }

// SMs a single-request decode leaves idle for the merge grid behind it: one
// per 16 merge warps (two warps per query row, at most 128 registers a thread).
inline int decode_merge_reserve_sms(int hkv, int rows) { return (2 * hkv * rows + 15) / 16; }

// Tokens per work unit.  Single request: split every kv head's context into
// floor((SMs - merge SMs) / hkv) units, so one wave covers the GPU and the
// merge's warps find room on the SMs left over (rows = 0: no reservation).
// Several requests: aim at about four units per SM so the block scheduler
// balances ragged lengths.
inline int64_t decode_unit_tokens(int n_req, int64_t total_tokens, int hkv, int rows = 0) {
  const int sms = device_sm_count();
  int64_t U;
  if (n_req == 1) {
    const int avail = std::max(hkv, sms - (rows > 0 ? decode_merge_reserve_sms(hkv, rows) : 0));
    const int per_head = std::max(1, avail / hkv);
    U = (total_tokens + per_head - 1) / per_head;
  } else {
    const int64_t target_units = (int64_t)sms * 4;
    U = (total_tokens * hkv + target_units - 1) / target_units;
  }
  // at most kMaxUnitsPerPair units per (request, head)
  U = std::max<int64_t>(U, (total_tokens + dec::kMaxUnitsPerPair - 1) / dec::kMaxUnitsPerPair);
  U = std::max<int64_t>(U, 32);
  U = (U + 63) / 64 * 64;  // whole 64-token tiles: no unit ends on a nearly empty tile
  return U;
}

inline int64_t decode_max_units(int n_req, int64_t total_tokens, int64_t U) {
  return total_tokens / U + n_req;
}

inline size_t decode_tc_workspace_bytes(const fla_attn_dims &d, int n_req, int64_t total_tokens) {
  const DecodePlan pl = decode_tc_plan(d);
  if (!pl.ok || n_req <= 0) return 0;
  const int64_t U = decode_unit_tokens(n_req, std::max<int64_t>(total_tokens, 1), d.hkv, pl.rows);
  const int64_t units = decode_max_units(n_req, total_tokens, U);
  const size_t info = ((size_t)n_req * d.hkv * sizeof(int2) + 255) / 256 * 256;
  const size_t part = (size_t)units * d.hkv * pl.part_stride * 4;
  return info + part;
}

typedef CUresult (*PFN_encodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                    CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                    CUtensorMapFloatOOBfill);

inline PFN_encodeTiled get_encode_tiled() {
  static PFN_encodeTiled fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(p);
  }
  return fn;
}

inline CUtensorMapSwizzle swizzle_enum(int bytes) {
  return bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                      : bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
}

// Merge-kernel geometry: one warp per query row (kMergeLaneWarps rows per CTA),
// or, for rows with many units (or when the caller asks for it), four warps
// per row in one CTA each.
constexpr int kLaneMaxUnits = 32;

// Launches the merge kernel behind a decode kernel (programmatic dependent launch).
// nu_bound: an upper bound on the units of any (request, head) pair.
template <int D>
inline cudaError_t launch_merge(const dec::MergeParams &mp, int64_t nu_bound, bool prefer_rows, cudaStream_t s) {
  const int64_t total = (int64_t)mp.n_req * mp.hkv * mp.rows;
  const bool lane = !prefer_rows && nu_bound <= kLaneMaxUnits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = lane ? dim3((unsigned)((total + dec::kMergeLaneWarps / 2 - 1) / (dec::kMergeLaneWarps / 2)))
                     : dim3((unsigned)(mp.n_req * mp.hkv), (unsigned)mp.rows);
  cfg.blockDim = dim3(lane ? dec::kMergeLaneWarps * 32 : 4 * 32);
  // the four-warp kernel: this row's B slice plus the cross-warp combine buffer
  cfg.dynamicSmemBytes = lane ? 0 : (size_t)mp.r * D * 2 + 4 * 32 * (D / 32 + 4) * 4;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (lane) return cudaLaunchKernelEx(&cfg, dec::decode_merge_lane_kernel<D>, mp);
  if (cfg.dynamicSmemBytes > 48 * 1024) {
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(dec::decode_merge_row_kernel<D>),
                                              (int)cfg.dynamicSmemBytes);
    if (e != cudaSuccess) return e;
  }
  return cudaLaunchKernelEx(&cfg, dec::decode_merge_row_kernel<D>, mp);
}

// Upper bound on the units of one (request, head) pair.
inline int64_t decode_units_bound(int64_t total_tokens, int64_t U) {
  return std::max<int64_t>(1, std::min<int64_t>(dec::kMaxUnitsPerPair, (total_tokens + U - 1) / U));
}

template <int D, int MT, int TG, int NLT, int SG>
inline fla_status decode_tc_run(const DecodePlan &pl, const CUtensorMap &mK, const CUtensorMap &mV,
                                const CUtensorMap &mL, const CUtensorMap &mB, const dec::Params &prm, unsigned grid,
                                bool need_merge, int64_t nu_bound, cudaStream_t s) {
  auto kern = dec::decode_tc_kernel<D, MT, TG, NLT, SG>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), pl.smem_bytes);
  if (e != cudaSuccess) {
    decode_tc_err() = cudaGetErrorString(e);
    return FLA_ERR_CUDA;
  }
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(dec::Cfg<D, MT, TG, NLT, SG>::kThreads);
    cfg.dynamicSmemBytes = pl.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mK, mV, mL, mB, prm);
    if (e != cudaSuccess) {
      decode_tc_err() = cudaGetErrorString(e);
      return FLA_ERR_CUDA;
    }
  }
  if (!need_merge) return FLA_OK;
  dec::MergeParams mp{};
  mp.partials = prm.partials;
  mp.pair_info = prm.pair_info;
  mp.B = prm.B;
  mp.O = prm.O;
  mp.n_req = prm.n_req; mp.A = prm.A; mp.hq = prm.hq; mp.hkv = prm.hkv; mp.G = prm.G; mp.rows = prm.rows;
  mp.r = prm.r;
  mp.part_stride = prm.part_stride; mp.unit_tokens = prm.unit_tokens; mp.single_len = prm.single_len;
  e = launch_merge<D>(mp, nu_bound, false, s);
  if (e != cudaSuccess) {
    decode_tc_err() = cudaGetErrorString(e);
    return FLA_ERR_CUDA;
  }
  return FLA_OK;
}

inline fla_status decode_tc_launch(const fla_attn_dims &d, float scale, const void *Q, const void *K,
                                   const void *V, const void *L, const void *B, const int32_t *offsets,
                                   int n_req, int64_t total_tokens, float *O, void *workspace,
                                   cudaStream_t s) {
  DecodePlan pl = decode_tc_plan(d);
  if (!pl.ok) {
    decode_tc_err() = "shape outside the tensor-core decode kernel";
    return FLA_ERR_UNSUPPORTED;
  }
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) {
    decode_tc_err() = "cuTensorMapEncodeTiled is not available from the driver";
    return FLA_ERR_CUDA;
  }
  const int64_t U = decode_unit_tokens(n_req, total_tokens, d.hkv, pl.rows);
  const int64_t units = decode_max_units(n_req, total_tokens, U);
  if (units * d.hkv > 2 * (int64_t)device_sm_count()) {
    // several waves of CTAs: two per SM where the shape allows
    const DecodePlan two = decode_tc_plan(d, true);
    if (two.ok && two.SG == 1 && two.MT == 1) pl = two;
  }
  CUtensorMap mK, mV, mL, mB;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)d.head_dim, (cuuint64_t)d.hkv, (cuuint64_t)total_tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)d.head_dim * 2, (cuuint64_t)d.hkv * d.head_dim * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)pl.T};
    const cuuint32_t es[3] = {1, 1, 1};
    CUresult r1 = enc(&mK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(K), dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    CUresult r2 = enc(&mV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(V), dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS) {
      decode_tc_err() = "encoding the K/V tensor maps failed";
      return FLA_ERR_CUDA;
    }
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)pl.l_width, (cuuint64_t)total_tokens};
    const cuuint64_t strides[1] = {(cuuint64_t)d.l_row_stride * 2};
    const cuuint32_t box[2] = {(cuuint32_t)pl.l_box_cols, (cuuint32_t)pl.T};
    const cuuint32_t es[2] = {1, 1};
    CUresult r3 = enc(&mL, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(L), dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_enum(pl.l_swz), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r3 != CUDA_SUCCESS) {
      decode_tc_err() = "encoding the L tensor map failed";
      return FLA_ERR_CUDA;
    }
  }
  {
    // B viewed as [A*r rows, hkv*d columns]; boxes of 16 rows x 64 columns
    const cuuint64_t dims[2] = {(cuuint64_t)d.hkv * d.head_dim, (cuuint64_t)d.n_agents * d.rank};
    const cuuint64_t strides[1] = {(cuuint64_t)d.hkv * d.head_dim * 2};
    const cuuint32_t box[2] = {64, 16};
    const cuuint32_t es[2] = {1, 1};
    CUresult r4 = enc(&mB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(B), dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r4 != CUDA_SUCCESS) {
      decode_tc_err() = "encoding the B tensor map failed";
      return FLA_ERR_CUDA;
    }
  }
  dec::Params prm{};
  prm.Q = reinterpret_cast<const __nv_bfloat16 *>(Q);
  prm.B = reinterpret_cast<const __nv_bfloat16 *>(B);
  prm.O = O;
  prm.offsets = offsets;
  const size_t info = ((size_t)n_req * d.hkv * sizeof(int2) + 255) / 256 * 256;
  prm.pair_info = reinterpret_cast<int2 *>(workspace);
  prm.partials = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + info);
  prm.n_req = n_req; prm.A = d.n_agents; prm.hq = d.hq; prm.hkv = d.hkv; prm.G = d.hq / d.hkv;
  prm.r = d.rank; prm.rows = pl.rows; prm.l_agent_stride = (int)d.l_agent_stride;
  prm.l_width = pl.l_width; prm.l_box_cols = pl.l_box_cols; prm.l_swz_bytes = pl.l_swz;
  prm.unit_tokens = (int)U; prm.stages = pl.stages;
  prm.bs_dedicated = pl.bs_dedicated; prm.part_stride = pl.part_stride;
  prm.single_len = n_req == 1 ? (int)total_tokens : -1;
  prm.scale_log2 = scale * 1.4426950408889634f;
  const int64_t grid64 = units * d.hkv;
  if (grid64 > 0x7fffffffLL) {
    decode_tc_err() = "too many work units";
    return FLA_ERR_UNSUPPORTED;
  }
  const unsigned grid = (unsigned)grid64;
  // the merge kernel is needed unless the only request fits in one unit
  const bool need_merge = !(n_req == 1 && total_tokens <= U);
#define FLA_DEC_CASE(DD, MM, TT, NN, GG)                                                    \
  if (pl.D == DD && pl.MT == MM && pl.TG == TT && pl.NLT == NN && pl.SG == GG)              \
    return decode_tc_run<DD, MM, TT, NN, GG>(pl, mK, mV, mL, mB, prm, grid, need_merge,          \
                                             decode_units_bound(total_tokens, U), s);
  FLA_DEC_CASE(128, 1, 4, 8, 2) FLA_DEC_CASE(128, 1, 4, 16, 2)
  FLA_DEC_CASE(128, 1, 4, 8, 1) FLA_DEC_CASE(128, 1, 4, 16, 1)
  FLA_DEC_CASE(128, 2, 4, 8, 1) FLA_DEC_CASE(128, 2, 4, 16, 1)
  FLA_DEC_CASE(128, 3, 2, 8, 1) FLA_DEC_CASE(128, 3, 2, 16, 1)
  FLA_DEC_CASE(128, 4, 2, 8, 1) FLA_DEC_CASE(128, 4, 2, 16, 1)
  FLA_DEC_CASE(64, 1, 4, 8, 2) FLA_DEC_CASE(64, 1, 4, 16, 2)
  FLA_DEC_CASE(64, 1, 4, 8, 1) FLA_DEC_CASE(64, 1, 4, 16, 1)
  FLA_DEC_CASE(64, 2, 4, 8, 1) FLA_DEC_CASE(64, 2, 4, 16, 1)
  FLA_DEC_CASE(64, 3, 2, 8, 1) FLA_DEC_CASE(64, 3, 2, 16, 1)
  FLA_DEC_CASE(64, 4, 2, 8, 1) FLA_DEC_CASE(64, 4, 2, 16, 1)
#undef FLA_DEC_CASE
  decode_tc_err() = "no kernel instance for this plan";
  return FLA_ERR_UNSUPPORTED;
}

}  // namespace fla
