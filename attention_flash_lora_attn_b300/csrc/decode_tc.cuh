// Tensor-core decode kernel: Flash-LoRA-Attention over a shared base cache.
//
// LRAgent technical summary (gist.science), Metodologia section 3: the output
// is computed as P.V_base + (P.L_a).B_a, so the r-wide P.L_a accumulates in the
// same pass as the d-wide P.V_base and B_a is applied once per query at the
// end.  Section 2 (BaseShared): K_base / V_base are one cache shared by every
// agent, so all agents' query rows of a kv head are served from one read of
// each K/V tile (like query heads of a GQA group).
//
// Work decomposition.  A work item is (request q, kv head h, unit u): a
// contiguous range of at most `unit_tokens` tokens of request q.  One CTA per
// work item; the CTA index is unit_global * hkv + h so the kv heads of the same
// token range run side by side and share the L tile through L2.
//
// Inside a CTA:
//   * one producer warp streams token tiles of T tokens with TMA into a ring of
//     STAGES shared-memory stages (K tile, V tile and the L tile holding every
//     agent's r columns), 128/64/32-byte swizzled, mbarrier full/empty ring;
//   * MT x TG consumer warps: the A*G query rows of kv head h (agent-major:
//     row = a*G + g) are cut into MT tiles of 16 rows; warp (mt, tg) owns row
//     tile mt and a 32-token slice tg of every stage.  S = Q.K^T, P.V_base and
//     P.L_window run on mma.sync m16n8k16 (bf16 in, fp32 accumulate); the online
//     softmax state (running max m, running sum l) and both accumulators stay
//     in registers, reductions over the 4 lanes of a row quad use shuffles;
//   * the TG token slices are merged in shared memory; a CTA that is the only
//     unit of its (q, h) applies B and writes O, otherwise it writes its
//     partial (m, l, P.V_base, own-agent P.L_a) to the workspace and the last
//     CTA to arrive (atomic ticket, no waiting) merges all units of (q, h) in
//     unit order (deterministic), applies B_a's head slice and writes O.
#pragma once

#include <cuda_bf16.h>

#include <algorithm>

#include "../../include/flash_lora_attn.h"
#include "fla_common.cuh"
#include "ptx.cuh"

namespace fla {
namespace dec {

constexpr int kTW = 32;             // tokens per consumer warp per stage
constexpr int kMaxRows = 64;        // A*G query rows per kv head (MT <= 4)
constexpr int kMaxUnitsPerPair = 512;
constexpr int kSmemBudget = 200 * 1024;

struct Params {
  const __nv_bfloat16 *Q, *B;
  float *O;
  const int32_t *offsets;
  float *partials;
  uint32_t *tickets;
  int32_t n_req, A, hq, hkv, G, r, rows;
  int32_t l_agent_stride;  // 0 or r
  int32_t l_width;         // columns of L held per token in shared memory
  int32_t l_box_cols;      // columns per L TMA box (16, 32 or 64)
  int32_t l_swz_bytes;     // 32, 64 or 128
  int32_t unit_tokens;
  int32_t stages;
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

template <int D, int MT, int TG, int NLT>
struct Cfg {
  static constexpr int T = TG * kTW;
  static constexpr int kConsumerWarps = MT * TG;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int kRowsPad = MT * 16;
  static constexpr int kQPitch = D * 2 + 16;  // bytes per Q row in shared memory
  static constexpr int kLwin = NLT * 8;       // L window columns per row tile
  // per-warp merge scratch: 16 rows x (D + kLwin) accumulators + m + l
  static constexpr int kScratchFloats = 16 * (D + kLwin + 2);
};

template <int D, int MT, int TG, int NLT>
__global__ void __launch_bounds__(Cfg<D, MT, TG, NLT>::kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmL, const Params p) {
  using C = Cfg<D, MT, TG, NLT>;
  constexpr int T = C::T;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const StageGeom geo{T, D, p.l_width, p.l_swz_bytes};
  const int stage_bytes = geo.stage_bytes();
  uint8_t *q_smem = smem + p.stages * stage_bytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(q_smem + C::kRowsPad * C::kQPitch);
  __shared__ int s_info[8];   // q, unit, n_units, token begin, token count, valid
  __shared__ int s_flag[2];   // [0] abort, [1] last-arrival

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x % p.hkv;
  const int unit_global = blockIdx.x / p.hkv;

  // ---- map unit_global -> (request, unit) with a warp-parallel scan
  if (warp == 0) {
    int base = 0, found = 0;
    const int U = p.unit_tokens;
    for (int q0 = 0; q0 < p.n_req && !found; q0 += 32) {
      const int q = q0 + lane;
      int len = 0, nu = 0;
      if (q < p.n_req) {
        len = p.offsets[q + 1] - p.offsets[q];
        nu = len > 0 ? (len + U - 1) / U : 1;
      }
      int incl = nu;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int excl = base + incl - nu;
      const bool mine = (q < p.n_req) && unit_global >= excl && unit_global < excl + nu;
      const unsigned m = __ballot_sync(0xffffffffu, mine);
      if (m) {
        found = 1;
        if (mine) {
          const int u = unit_global - excl;
          const int tb = p.offsets[q] + u * U;
          s_info[0] = q;
          s_info[1] = u;
          s_info[2] = nu;
          s_info[3] = tb;
          s_info[4] = len > 0 ? min(U, len - u * U) : 0;
        }
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      s_info[5] = found;
      s_flag[0] = 0;
      s_flag[1] = 0;
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars[s]), 1);                         // full: producer arrive + tx
      ptx::mbar_init(ptx::smem_u32(&bars[p.stages + s]), C::kConsumerWarps);  // empty
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (!s_info[5]) return;  // grid slack beyond the last unit
  const int q = s_info[0], unit = s_info[1], n_units = s_info[2];
  const int tok_begin = s_info[3], n_tok = s_info[4];
  const int n_tiles = (n_tok + T - 1) / T;
  const uint32_t bar_full0 = ptx::smem_u32(&bars[0]);
  const uint32_t bar_empty0 = ptx::smem_u32(&bars[p.stages]);

  if (warp == C::kConsumerWarps) {
    // ======================= producer warp =======================
    if (lane == 0) {
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      ptx::prefetch_tmap(&tmL);
      const int n_lbox = p.l_width / p.l_box_cols;
      const int lbox_bytes = T * p.l_swz_bytes;
      int issued = 0;
      for (int it = 0; it < n_tiles; ++it) {
        const int st = it % p.stages;
        const uint32_t ph = (it / p.stages) & 1;
        if (it >= p.stages) {
          if (!ptx::mbar_wait(bar_empty0 + 8 * st, ph ^ 1)) {
            set_device_error(kErrDecodeEmptyWait);
            s_flag[0] = 1;
            break;
          }
        }
        if (*(volatile int *)&s_flag[0]) break;
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
        ++issued;
      }
      // Do not leave while copies are in flight: wait (bounded) for the last
      // load issued into each stage.
      for (int k = 0; k < p.stages && k < issued; ++k) {
        const int it = issued - 1 - k;
        const int st = it % p.stages;
        if (!ptx::mbar_wait(bar_full0 + 8 * st, (it / p.stages) & 1)) set_device_error(kErrDecodeFullWait);
      }
    }
    return;  // the producer takes no part in the epilogue
  }

  // ======================= consumer warps =======================
  constexpr int kConsumerThreads = C::kConsumerWarps * 32;
  const int mt = warp / TG, tg = warp % TG;
  const int g = lane >> 2, t4 = lane & 3;

  // Q rows of this kv head into shared memory (zero rows beyond A*G).
  for (int e = threadIdx.x; e < C::kRowsPad * (D / 8); e += kConsumerThreads) {
    const int row = e / (D / 8), c8 = e % (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < p.rows) {
      const int a = row / p.G, j = head * p.G + row % p.G;
      v = *reinterpret_cast<const uint4 *>(p.Q + (((int64_t)q * p.A + a) * p.hq + j) * D + c8 * 8);
    }
    *reinterpret_cast<uint4 *>(q_smem + row * C::kQPitch + c8 * 16) = v;
  }
  ptx::named_bar_sync(1, kConsumerThreads);
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
  const int lbox_bytes = T * p.l_swz_bytes;
  const int lbox_cols = p.l_box_cols;

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
    if (!ptx::mbar_wait(bar_full0 + 8 * st, (it / p.stages) & 1)) {
      set_device_error(kErrDecodeFullWait);
      s_flag[0] = 1;
      aborted = true;
      break;
    }
    const uint8_t *sK = smem + st * stage_bytes;
    const uint8_t *sV = sK + geo.k_bytes();
    const uint8_t *sL = sK + 2 * geo.k_bytes();
    const uint32_t aK = ptx::smem_u32(sK), aV = ptx::smem_u32(sV), aL = ptx::smem_u32(sL);
    const int tok0 = tg * kTW;  // first token of this warp's slice within the tile

    // ---- S = Q . K^T  (16 rows x 32 tokens)
    float s[kTW / 8][4];
#pragma unroll
    for (int i = 0; i < kTW / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < kTW / 16; ++np) {
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
    if (valid < kTW) {
#pragma unroll
      for (int nt = 0; nt < kTW / 8; ++nt) {
        const int c = nt * 8 + 2 * t4;
        if (c >= valid) { s[nt][0] = -INFINITY; s[nt][2] = -INFINITY; }
        if (c + 1 >= valid) { s[nt][1] = -INFINITY; s[nt][3] = -INFINITY; }
      }
    }
    // ---- online softmax (log2 domain)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < kTW / 8; ++nt) {
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
    uint32_t pa[kTW / 16][4];
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < kTW / 8; ++nt) {
      const float p0 = ptx::ex2(s[nt][0] - ref0), p1 = ptx::ex2(s[nt][1] - ref0);
      const float p2 = ptx::ex2(s[nt][2] - ref1), p3 = ptx::ex2(s[nt][3] - ref1);
      rs0 += p0 + p1;
      rs1 += p2 + p3;
      pa[nt >> 1][(nt & 1) * 2 + 0] = ptx::pack_bf16(p0, p1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = ptx::pack_bf16(p2, p3);
    }
    l0 = l0 * corr0 + rs0;
    l1 = l1 * corr1 + rs1;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      acc_v[i][0] *= corr0; acc_v[i][1] *= corr0; acc_v[i][2] *= corr1; acc_v[i][3] *= corr1;
    }
#pragma unroll
    for (int i = 0; i < NLT; ++i) {
      acc_l[i][0] *= corr0; acc_l[i][1] *= corr0; acc_l[i][2] *= corr1; acc_l[i][3] *= corr1;
    }
    // ---- acc_v += P . V_base ; acc_l += P . L_window
#pragma unroll
    for (int ks = 0; ks < kTW / 16; ++ks) {
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
        const int box = cb / lbox_cols;
        const int chunk = (cb % lbox_cols) >> 3;
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
  }

  // ---- row sums across the quad
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // All consumers are past every full-barrier wait, so every TMA write into
  // the stage ring has landed: the ring is reused as merge scratch.
  ptx::named_bar_sync(1, kConsumerThreads);
  if (*(volatile int *)&s_flag[0] || aborted) return;

  float *scratch = reinterpret_cast<float *>(smem) + warp * C::kScratchFloats;
  // layout per warp: [16][D] acc_v | [16][kLwin] acc_l | [16] m | [16] l
  {
    float *sv = scratch, *sl = scratch + 16 * D, *sm = sl + 16 * C::kLwin, *ss = sm + 16;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      const int c = i * 8 + 2 * t4;
      sv[g * D + c] = acc_v[i][0];
      sv[g * D + c + 1] = acc_v[i][1];
      sv[(g + 8) * D + c] = acc_v[i][2];
      sv[(g + 8) * D + c + 1] = acc_v[i][3];
    }
#pragma unroll
    for (int i = 0; i < NLT; ++i) {
      const int c = i * 8 + 2 * t4;
      sl[g * C::kLwin + c] = acc_l[i][0];
      sl[g * C::kLwin + c + 1] = acc_l[i][1];
      sl[(g + 8) * C::kLwin + c] = acc_l[i][2];
      sl[(g + 8) * C::kLwin + c + 1] = acc_l[i][3];
    }
    if (t4 == 0) {
      sm[g] = m0; sm[g + 8] = m1;
      ss[g] = l0; ss[g + 8] = l1;
    }
  }
  ptx::named_bar_sync(1, kConsumerThreads);

  // ---- merge the TG token slices: combined state per valid row
  const int D_ = D, r = p.r;
  float *cmb = reinterpret_cast<float *>(smem) + C::kConsumerWarps * C::kScratchFloats;
  // layout: [rows][D] v | [rows][r] L(own agent) | [rows] m | [rows] l | [rows][TG] w
  float *cv = cmb, *cl = cv + p.rows * D_, *cm = cl + p.rows * r, *cs = cm + p.rows, *cw = cs + p.rows;
  for (int row = threadIdx.x; row < p.rows; row += kConsumerThreads) {
    const int rt = row / 16, rr = row % 16;
    float M = -INFINITY;
    for (int k = 0; k < TG; ++k) {
      const float *sc = reinterpret_cast<float *>(smem) + (rt * TG + k) * C::kScratchFloats;
      M = fmaxf(M, sc[16 * D + 16 * C::kLwin + rr]);
    }
    float lsum = 0.f;
    for (int k = 0; k < TG; ++k) {
      const float *sc = reinterpret_cast<float *>(smem) + (rt * TG + k) * C::kScratchFloats;
      const float mk = sc[16 * D + 16 * C::kLwin + rr];
      const float w = (mk == -INFINITY) ? 0.f : ptx::ex2(mk - M);
      cw[row * TG + k] = w;
      lsum += w * sc[16 * D + 16 * C::kLwin + 16 + rr];
    }
    cm[row] = M;
    cs[row] = lsum;
  }
  ptx::named_bar_sync(1, kConsumerThreads);
  for (int e = threadIdx.x; e < p.rows * (D_ + r); e += kConsumerThreads) {
    const int row = e / (D_ + r), c = e % (D_ + r);
    const int rt = row / 16, rr = row % 16;
    float v = 0.f;
    if (c < D_) {
      for (int k = 0; k < TG; ++k) {
        const float *sc = reinterpret_cast<float *>(smem) + (rt * TG + k) * C::kScratchFloats;
        v += cw[row * TG + k] * sc[rr * D + c];
      }
      cv[row * D_ + c] = v;
    } else {
      const int kcol = c - D_;
      const int a = row / p.G;
      const int wc = a * p.l_agent_stride - (rt * 16 / p.G) * p.l_agent_stride + kcol;  // window column
      for (int k = 0; k < TG; ++k) {
        const float *sc = reinterpret_cast<float *>(smem) + (rt * TG + k) * C::kScratchFloats;
        v += cw[row * TG + k] * sc[16 * D + rr * C::kLwin + wc];
      }
      cl[row * r + kcol] = v;
    }
  }
  ptx::named_bar_sync(1, kConsumerThreads);

  const int pair = q * p.hkv + head;
  const int part_floats = p.rows * (D_ + r + 2);
  if (n_units > 1) {
    // ---- publish this unit's partial; the last unit of (q, head) merges
    float *dst = p.partials + ((int64_t)unit_global * p.hkv + head) * part_floats;
    for (int e = threadIdx.x; e < part_floats; e += kConsumerThreads) dst[e] = cmb[e];
    __threadfence();
    ptx::named_bar_sync(1, kConsumerThreads);
    if (threadIdx.x == 0) {
      const uint32_t old = atomicAdd(&p.tickets[pair], 1u);
      s_flag[1] = (old == (uint32_t)(n_units - 1));
    }
    ptx::named_bar_sync(1, kConsumerThreads);
    if (!s_flag[1]) return;
    __threadfence();
    // weights per (row, unit) into the (now free) merge scratch
    const int ug0 = unit_global - unit;  // first unit of this request
    float *wts = reinterpret_cast<float *>(smem);
    float *msum = wts + p.rows * n_units;
    for (int row = threadIdx.x; row < p.rows; row += kConsumerThreads) {
      float M = -INFINITY;
      for (int u = 0; u < n_units; ++u) {
        const float *src = p.partials + ((int64_t)(ug0 + u) * p.hkv + head) * part_floats;
        M = fmaxf(M, __ldcg(src + p.rows * (D_ + r) + row));
      }
      float lsum = 0.f;
      for (int u = 0; u < n_units; ++u) {
        const float *src = p.partials + ((int64_t)(ug0 + u) * p.hkv + head) * part_floats;
        const float mu = __ldcg(src + p.rows * (D_ + r) + row);
        const float w = (mu == -INFINITY) ? 0.f : ptx::ex2(mu - M);
        wts[row * n_units + u] = w;
        lsum += w * __ldcg(src + p.rows * (D_ + r) + p.rows + row);
      }
      msum[row] = lsum;
    }
    ptx::named_bar_sync(1, kConsumerThreads);
    float *cv2 = msum + p.rows;  // merged [rows][D] v | [rows][r] L
    for (int e = threadIdx.x; e < p.rows * (D_ + r); e += kConsumerThreads) {
      const int row = (e < p.rows * D_) ? e / D_ : (e - p.rows * D_) / r;
      float v = 0.f;
      for (int u = 0; u < n_units; ++u) {
        const float *src = p.partials + ((int64_t)(ug0 + u) * p.hkv + head) * part_floats;
        v += wts[row * n_units + u] * __ldcg(src + e);
      }
      cv2[e] = v;
    }
    if (threadIdx.x == 0) p.tickets[pair] = 0;  // leave the workspace zeroed for the next call
    ptx::named_bar_sync(1, kConsumerThreads);
    cv = cv2;
    cl = cv2 + p.rows * D_;
    cs = msum;
  }

  // ---- epilogue: O = (P.V_base + (P.L_a) . B_a[:, h*d:(h+1)*d]) / l
  const int64_t bstride = (int64_t)p.hkv * D_;
  for (int e = threadIdx.x; e < p.rows * D_; e += kConsumerThreads) {
    const int row = e / D_, c = e % D_;
    const int a = row / p.G, j = head * p.G + row % p.G;
    const float lsum = cs[row];
    float o = 0.f;
    if (lsum > 0.f) {
      const __nv_bfloat16 *Bc = p.B + (int64_t)a * r * bstride + (int64_t)head * D_ + c;
      float lora = 0.f;
      for (int k = 0; k < r; ++k) lora += cl[row * r + k] * __bfloat162float(Bc[(int64_t)k * bstride]);
      o = (cv[row * D_ + c] + lora) / lsum;
    }
    p.O[(((int64_t)q * p.A + a) * p.hq + j) * D_ + c] = o;
  }
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
  return "bf16; head_dim 64 or 128; rank % 8 == 0; l_agent_stride 0 or rank; n_agents*hq/hkv <= 64; "
         "L window per 16-row tile <= 128 columns; loaded L width % 16 == 0; 16-byte aligned pointers; "
         "l_row_stride % 8 == 0";
}

struct DecodePlan {
  int D, MT, TG, NLT;
  int rows, l_width, l_box_cols, l_swz;
  int T, stages, smem_bytes;
  bool ok;
};

inline DecodePlan decode_tc_plan(const fla_attn_dims &d) {
  DecodePlan pl{};
  pl.ok = false;
  if (d.dtype != FLA_BF16) return pl;
  if (d.head_dim != 64 && d.head_dim != 128) return pl;
  if (d.rank % 8 != 0 || d.rank > 128) return pl;
  if (d.l_agent_stride != 0 && d.l_agent_stride != d.rank) return pl;
  const int G = d.hq / d.hkv;
  const int rows = d.n_agents * G;
  if (rows > dec::kMaxRows) return pl;
  const int MT = (rows + 15) / 16;
  // widest L window over the row tiles
  int wmax = 0;
  for (int mt = 0; mt < MT; ++mt) {
    const int lo = mt * 16, hi = std::min(rows, lo + 16) - 1;
    const int w = (hi / G - lo / G) * (int)d.l_agent_stride + d.rank;
    wmax = std::max(wmax, w);
  }
  if (wmax > 128) return pl;
  const int NLT = wmax <= 64 ? 8 : 16;
  const int l_width = d.l_agent_stride == 0 ? d.rank : d.n_agents * d.rank;
  int swz = 0;
  if ((l_width * 2) % 128 == 0) swz = 128;
  else if ((l_width * 2) % 64 == 0) swz = 64;
  else if ((l_width * 2) % 32 == 0) swz = 32;
  else return pl;
  const int TG = MT == 1 ? 4 : (MT == 4 ? 1 : 2);
  const int T = TG * dec::kTW;
  const int stage = 2 * T * d.head_dim * 2 + T * l_width * 2;
  const int q_bytes = MT * 16 * (d.head_dim * 2 + 16);
  // merge scratch (aliases the stage ring) must fit into the ring
  const int scratch_tg = (MT * TG * 16 * (d.head_dim + NLT * 8 + 2) + rows * (d.head_dim + d.rank + 2 + TG)) * 4;
  // the last unit's merge: weights [rows][units] + sums [rows] + merged [rows][D + r]
  const int scratch_units = rows * (dec::kMaxUnitsPerPair + 1 + d.head_dim + d.rank) * 4;
  const int scratch = std::max(scratch_tg, scratch_units);
  int stages = (dec::kSmemBudget - q_bytes - 1024 - 256) / stage;
  if (stages > 8) stages = 8;
  while (stages >= 2 && stages * stage < scratch) ++stages;
  if (stages < 2) return pl;
  pl.smem_bytes = stages * stage + q_bytes + 2 * stages * 8 + 1024;
  if (pl.smem_bytes > 227 * 1024) return pl;
  pl.D = d.head_dim; pl.MT = MT; pl.TG = TG; pl.NLT = NLT;
  pl.rows = rows; pl.l_width = l_width; pl.l_box_cols = swz / 2; pl.l_swz = swz;
  pl.T = T; pl.stages = stages;
  pl.ok = true;
  return pl;
}

inline bool decode_tc_shape_supported(const fla_attn_dims &d) { return decode_tc_plan(d).ok; }

inline int device_sm_count() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

// Tokens per work unit.  Single request: split every kv head's context into
// floor(SMs / hkv) units so one wave covers the GPU.  Several requests: aim at
// about four units per SM so the block scheduler balances ragged lengths.
inline int64_t decode_unit_tokens(int n_req, int64_t total_tokens, int hkv) {
  const int sms = device_sm_count();
  int64_t U;
  if (n_req == 1) {
    const int per_head = std::max(1, sms / hkv);
    U = (total_tokens + per_head - 1) / per_head;
  } else {
    const int64_t target_units = (int64_t)sms * 4;
    U = (total_tokens * hkv + target_units - 1) / target_units;
  }
  // at most kMaxUnitsPerPair units per (request, head)
  U = std::max<int64_t>(U, (total_tokens + dec::kMaxUnitsPerPair - 1) / dec::kMaxUnitsPerPair);
  U = std::max<int64_t>(U, 32);
  U = (U + 15) / 16 * 16;
  return U;
}

inline int64_t decode_max_units(int n_req, int64_t total_tokens, int64_t U) {
  return total_tokens / U + n_req;
}

inline size_t decode_tc_workspace_bytes(const fla_attn_dims &d, int n_req, int64_t total_tokens) {
  const DecodePlan pl = decode_tc_plan(d);
  if (!pl.ok || n_req <= 0) return 0;
  const int64_t U = decode_unit_tokens(n_req, std::max<int64_t>(total_tokens, 1), d.hkv);
  const int64_t units = decode_max_units(n_req, total_tokens, U);
  const size_t tickets = ((size_t)n_req * d.hkv * 4 + 255) / 256 * 256;
  const size_t part = (size_t)units * d.hkv * pl.rows * (d.head_dim + d.rank + 2) * 4;
  return tickets + part;
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

template <int D, int MT, int TG, int NLT>
inline fla_status decode_tc_run(const DecodePlan &pl, const CUtensorMap &mK, const CUtensorMap &mV,
                                const CUtensorMap &mL, const dec::Params &prm, unsigned grid, cudaStream_t s) {
  auto kern = dec::decode_tc_kernel<D, MT, TG, NLT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem_bytes);
  if (e != cudaSuccess) {
    decode_tc_err() = cudaGetErrorString(e);
    return FLA_ERR_CUDA;
  }
  kern<<<grid, dec::Cfg<D, MT, TG, NLT>::kThreads, pl.smem_bytes, s>>>(mK, mV, mL, prm);
  return FLA_OK;
}

inline fla_status decode_tc_launch(const fla_attn_dims &d, float scale, const void *Q, const void *K,
                                   const void *V, const void *L, const void *B, const int32_t *offsets,
                                   int n_req, int64_t total_tokens, float *O, void *workspace,
                                   cudaStream_t s) {
  const DecodePlan pl = decode_tc_plan(d);
  if (!pl.ok) {
    decode_tc_err() = "shape outside the tensor-core decode kernel";
    return FLA_ERR_UNSUPPORTED;
  }
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) {
    decode_tc_err() = "cuTensorMapEncodeTiled is not available from the driver";
    return FLA_ERR_CUDA;
  }
  const int64_t U = decode_unit_tokens(n_req, total_tokens, d.hkv);
  const int64_t units = decode_max_units(n_req, total_tokens, U);
  CUtensorMap mK, mV, mL;
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
  dec::Params prm{};
  prm.Q = reinterpret_cast<const __nv_bfloat16 *>(Q);
  prm.B = reinterpret_cast<const __nv_bfloat16 *>(B);
  prm.O = O;
  prm.offsets = offsets;
  const size_t tickets = ((size_t)n_req * d.hkv * 4 + 255) / 256 * 256;
  prm.tickets = reinterpret_cast<uint32_t *>(workspace);
  prm.partials = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + tickets);
  prm.n_req = n_req; prm.A = d.n_agents; prm.hq = d.hq; prm.hkv = d.hkv; prm.G = d.hq / d.hkv;
  prm.r = d.rank; prm.rows = pl.rows; prm.l_agent_stride = (int)d.l_agent_stride;
  prm.l_width = pl.l_width; prm.l_box_cols = pl.l_box_cols; prm.l_swz_bytes = pl.l_swz;
  prm.unit_tokens = (int)U; prm.stages = pl.stages;
  prm.scale_log2 = scale * 1.4426950408889634f;
  const int64_t grid64 = units * d.hkv;
  if (grid64 > 0x7fffffffLL) {
    decode_tc_err() = "too many work units";
    return FLA_ERR_UNSUPPORTED;
  }
  const unsigned grid = (unsigned)grid64;
#define FLA_DEC_CASE(DD, MM, TT, NN)                                                     \
  if (pl.D == DD && pl.MT == MM && pl.TG == TT && pl.NLT == NN)                          \
    return decode_tc_run<DD, MM, TT, NN>(pl, mK, mV, mL, prm, grid, s);
  FLA_DEC_CASE(128, 1, 4, 8) FLA_DEC_CASE(128, 1, 4, 16)
  FLA_DEC_CASE(128, 2, 2, 8) FLA_DEC_CASE(128, 2, 2, 16)
  FLA_DEC_CASE(128, 3, 2, 8) FLA_DEC_CASE(128, 3, 2, 16)
  FLA_DEC_CASE(128, 4, 1, 8) FLA_DEC_CASE(128, 4, 1, 16)
  FLA_DEC_CASE(64, 1, 4, 8) FLA_DEC_CASE(64, 1, 4, 16)
  FLA_DEC_CASE(64, 2, 2, 8) FLA_DEC_CASE(64, 2, 2, 16)
  FLA_DEC_CASE(64, 3, 2, 8) FLA_DEC_CASE(64, 3, 2, 16)
  FLA_DEC_CASE(64, 4, 1, 8) FLA_DEC_CASE(64, 4, 1, 16)
#undef FLA_DEC_CASE
  decode_tc_err() = "no kernel instance for this plan";
  return FLA_ERR_UNSUPPORTED;
}

}  // namespace fla
