// 5th-generation tensor-core (tcgen05 + TMEM) chunked causal prefill:
// Flash-LoRA-Attention for the `chunk` new tokens of every agent over a
// shared context of n0 tokens.
//
// LRAgent technical summary (gist.science), Metodologia section 3: the output
// is P.V_base + (P.L_a).B_a, with B_a applied once per query block after the
// key loop; section 2 (BaseShared): K_base / V_base are shared by every
// agent, so one CTA serves all agents' queries of a kv head from one read of
// each K / V tile.  The query at chunk position p (absolute position n0 + p)
// sees keys 0 .. n0 + p.
//
// One CTA per (kv head, block of QB consecutive chunk positions); its 128
// query rows are row = (a*QB + pi)*G + g (agent a, position pi, q head g of
// the group), zero rows past the valid ones.  Per key tile of 128 tokens:
//   S_j  = Q . K_j^T                 tcgen05.mma, A = Q (smem), B = K_j (smem),
//                                    accumulator in TMEM (two S buffers)
//   P_j  = exp2(S_j*scale - m)       4 softmax warps, one TMEM lane (query
//                                    row) per thread; P_j (bf16) goes back
//                                    into TMEM
//   [O | OL] += P_j . [V_j | L_j]    one tcgen05.mma, A = P_j (TMEM),
//                                    B = V_j and the L columns of every agent
//                                    stacked along N (MN-major, smem)
// The running max m is only raised (and O, OL rescaled in TMEM) when a tile's
// max exceeds it by more than 2^8, so the rescale is rare; the result is the
// same softmax up to rounding.  After the last tile one more tcgen05.mma adds
// (P.L_a).B_a: A = the OL row of each query restricted to its own agent's
// columns (bf16 high + low parts, K = 2*A*r), B = [B_cat; B_cat] of the head.
//
// Warp roles: warp 0 lane 0 issues the K ring's TMA copies (then B), warp 6
// lane 0 the V|L ring's; warp 1 owns the TMEM allocation and lane 0 issues
// every MMA; warps 2..5 run the softmax and the epilogue.  Every wait is bounded; on a timeout the kernel records the
// error, drains its own copies and MMAs, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>

#include "../../include/flash_lora_attn.h"
#include "decode_tc.cuh"
#include "fla_common.cuh"
#include "ptx.cuh"

namespace fla {
namespace ptc {

constexpr int kT = 128;          // keys per tile
constexpr int kM = 128;          // query rows per CTA (MMA M)
constexpr int kThreads = 224;    // 7 warps
constexpr int kVWarp = 6;        // the V|L producer warp
constexpr int kBoxBytes = 128 * 128;  // one 64-column box of a 128-row tile
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP = 448;  // TMEM columns
constexpr float kRescaleLog2 = 8.f;  // raise the running max only past 2^8
constexpr int kMaxRing = 4;

struct Params {
  const __nv_bfloat16 *Q;
  float *O;
  int64_t n0;
  int32_t chunk, A, hq, hkv, G, r, QB, rows, rpa;  // rpa: rows per agent = QB * G
  int32_t l_agent_stride;
  int32_t nk, nv;  // depths of the K ring and of the V|L ring
  float scale_log2;
};

__device__ __forceinline__ bool wait_ab(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  return ptx::mbar_wait_or_abort(bar, parity, abort_flag, kErrPrefillWait);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmB,
                  const Params p) {
  constexpr int kQBytes = kM * D * 2;
  constexpr int kKBytes = kT * D * 2;
  constexpr int kVLBytes = kT * (D + 64) * 2;
  constexpr uint32_t kColOL = kColO + D;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *q_s = smem;
  uint8_t *k_s = smem + kQBytes;
  uint8_t *vl_s = k_s + p.nk * kKBytes;
  __shared__ __align__(8) uint64_t bars[4 * kMaxRing + 8];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x % p.hkv;
  const int n_qb = (int)(gridDim.x / p.hkv);
  const int qb = n_qb - 1 - (int)(blockIdx.x / p.hkv);  // late chunk blocks (most keys) first
  const int p0 = qb * p.QB;
  const int64_t n_keys = p.n0 + min(p.chunk, p0 + p.QB);
  const int n = (int)((n_keys + kT - 1) / kT);
  const int64_t causal_from = p.n0 + p0;  // keys >= this need the per-row mask

  const uint32_t bar0 = ptx::smem_u32(bars);
  auto kf = [&](int s) { return bar0 + 8u * s; };
  auto ke = [&](int s) { return bar0 + 8u * (kMaxRing + s); };
  auto vf = [&](int s) { return bar0 + 8u * (2 * kMaxRing + s); };
  auto ve = [&](int s) { return bar0 + 8u * (3 * kMaxRing + s); };
  auto sfull = [&](int b) { return bar0 + 8u * (4 * kMaxRing + b); };
  auto sfree = [&](int b) { return bar0 + 8u * (4 * kMaxRing + 2 + b); };
  const uint32_t pfull = bar0 + 8u * (4 * kMaxRing + 4);
  const uint32_t pvdone = bar0 + 8u * (4 * kMaxRing + 5);
  const uint32_t bfull = bar0 + 8u * (4 * kMaxRing + 6);
  const uint32_t drain = bar0 + 8u * (4 * kMaxRing + 7);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < p.nk; ++s) {
      ptx::mbar_init(kf(s), 1);
      ptx::mbar_init(ke(s), 1);
    }
    for (int s = 0; s < p.nv; ++s) {
      ptx::mbar_init(vf(s), 1);
      ptx::mbar_init(ve(s), 1);
    }
    ptx::mbar_init(sfull(0), 1);
    ptx::mbar_init(sfull(1), 1);
    ptx::mbar_init(sfree(0), 4);
    ptx::mbar_init(sfree(1), 4);
    ptx::mbar_init(pfull, 4);
    ptx::mbar_init(pvdone, 1);
    ptx::mbar_init(bfull, 1);
    ptx::mbar_init(drain, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&s_tmem), 512);
    ptx::tmem_relinquish();
  }
  // Q rows of the block into the K-major 128-byte-swizzled layout the MMA reads
  for (int e = threadIdx.x; e < kM * (D / 8); e += kThreads) {
    const int row = e / (D / 8), c8 = e % (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < p.rows) {
      const int a = row / p.rpa, pi = (row / p.G) % p.QB, g = row % p.G;
      const int pos = p0 + pi;
      if (pos < p.chunk)
        v = *reinterpret_cast<const uint4 *>(p.Q + (((int64_t)a * p.chunk + pos) * p.hq + head * p.G + g) * D +
                                             c8 * 8);
    }
    *reinterpret_cast<uint4 *>(q_s + (c8 >> 3) * kBoxBytes + row * 128 + (((c8 & 7) ^ (row & 7)) << 4)) = v;
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool ok = true;

  if (warp == 0 || warp == kVWarp) {
    // ------------------------------------------------------------ TMA producers:
    // warp 0 streams the K ring (then B_cat), warp kVWarp the V|L ring, so
    // neither ring waits behind the other's free slots
    int k_issued = 0, v_issued = 0;
    bool b_issued = false;
    if (lane == 0 && warp == 0) {
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmB);
      for (int j = 0; ok && j < n; ++j) {
        const int st = j % p.nk;
        if (j >= p.nk && !wait_ab(ke(st), ((j / p.nk) - 1) & 1, &s_abort)) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(kf(st), kKBytes);
        const uint32_t dst = ptx::smem_u32(k_s + st * kKBytes);
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
          ptx::tma_load_3d(dst + b * kBoxBytes, &tmK, b * 64, head, j * kT, kf(st));
        k_issued = j + 1;
      }
      // B_cat rows of this head for the epilogue GEMM, into the K ring once
      // the last S MMA (hence every S MMA) has finished with it
      if (ok) ok = wait_ab(ke((n - 1) % p.nk), ((n - 1) / p.nk) & 1, &s_abort);
      if (ok) {
        ptx::mbar_arrive_expect_tx(bfull, 64 * D * 2);
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
          ptx::tma_load_2d(ptx::smem_u32(k_s) + b * (64 * 128), &tmB, head * D + b * 64, 0, bfull);
        b_issued = true;
      }
      if (!ok) s_abort = 1;
    }
    if (lane == 0 && warp == kVWarp) {
      ptx::prefetch_tmap(&tmV);
      ptx::prefetch_tmap(&tmL);
      for (int j = 0; ok && j < n; ++j) {
        const int st = j % p.nv;
        if (j >= p.nv && !wait_ab(ve(st), ((j / p.nv) - 1) & 1, &s_abort)) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(vf(st), kVLBytes);
        const uint32_t dst = ptx::smem_u32(vl_s + st * kVLBytes);
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
          ptx::tma_load_3d(dst + b * kBoxBytes, &tmV, b * 64, head, j * kT, vf(st));
        ptx::tma_load_2d(dst + (D / 64) * kBoxBytes, &tmL, 0, j * kT, vf(st));
        v_issued = j + 1;
      }
      if (!ok) s_abort = 1;
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (s_abort && lane == 0) {
      // wait for this warp's own copies still in flight: the latest load of each stage
      for (int j = max(0, k_issued - p.nk); j < k_issued; ++j) ptx::mbar_wait(kf(j % p.nk), (j / p.nk) & 1);
      for (int j = max(0, v_issued - p.nv); j < v_issued; ++j) ptx::mbar_wait(vf(j % p.nv), (j / p.nv) & 1);
      if (b_issued) ptx::mbar_wait(bfull, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    bool issued_any = false;
    if (lane == 0) {
      const uint32_t idesc_s = ptx::idesc_bf16_f32(kM, kT);
      const uint32_t idesc_pv = ptx::idesc_bf16_f32(kM, D + 64) | (1u << 16);  // B (V|L) MN-major
      const uint32_t idesc_ep = ptx::idesc_bf16_f32(kM, D) | (1u << 16);       // B (B_cat) MN-major
      const uint64_t d_q = ptx::smem_desc_k128(ptx::smem_u32(q_s));
      const uint64_t d_k = ptx::smem_desc_k128(ptx::smem_u32(k_s));
      const uint64_t d_vl = ptx::smem_desc_mn128(ptx::smem_u32(vl_s), kBoxBytes);
      auto issue_s = [&](int j) -> bool {
        const int st = j % p.nk, b = j & 1;
        if (!wait_ab(kf(st), (j / p.nk) & 1, &s_abort)) return false;
        if (j >= 2 && !wait_ab(sfree(b), ((j >> 1) - 1) & 1, &s_abort)) return false;
        ptx::tc_fence_after();
        const uint64_t dk = ptx::desc_advance(d_k, st * kKBytes);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kBoxBytes + (ks & 3) * 32;
          ptx::tc_mma_f16(tmem + (b ? kColS1 : kColS0), ptx::desc_advance(d_q, off), ptx::desc_advance(dk, off),
                          idesc_s, ks > 0 ? 1u : 0u);
        }
        issued_any = true;
        ptx::tc_commit(ke(st));
        ptx::tc_commit(sfull(b));
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        const int st = j % p.nv;
        if (!wait_ab(pfull, j & 1, &s_abort)) return false;
        if (!wait_ab(vf(st), (j / p.nv) & 1, &s_abort)) return false;
        ptx::tc_fence_after();
        const uint64_t dv = ptx::desc_advance(d_vl, st * kVLBytes);
#pragma unroll
        for (int ks = 0; ks < kT / 16; ++ks)
          ptx::tc_mma_f16_ts(tmem + kColO, tmem + kColP + ks * 8, ptx::desc_advance(dv, ks * 16 * 128), idesc_pv,
                             (j > 0 || ks > 0) ? 1u : 0u);
        ptx::tc_commit(ve(st));
        ptx::tc_commit(pvdone);
        return true;
      };
      ok = issue_s(0);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) ok = issue_s(j + 1);
        if (ok) ok = issue_pv(j);
      }
      // O += [OL_hi | OL_lo] . [B_cat ; B_cat]   (K = 2 x 64)
      if (ok) ok = wait_ab(pfull, n & 1, &s_abort);
      if (ok) ok = wait_ab(bfull, 0, &s_abort);
      if (ok) {
        ptx::tc_fence_after();
        const uint64_t dbb = ptx::smem_desc_mn128(ptx::smem_u32(k_s), 64 * 128);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          ptx::tc_mma_f16_ts(tmem + kColO, tmem + kColP + ks * 8, ptx::desc_advance(dbb, (ks & 3) * 16 * 128), idesc_ep,
                             1u);
        ptx::tc_commit(pvdone);
      }
      if (!ok) s_abort = 1;
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (s_abort && lane == 0 && issued_any) {
      ptx::tc_commit(drain);  // completes once every MMA this thread issued has finished
      ptx::mbar_wait(drain, 0);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ softmax + epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int a = -1, pos = 0, g = 0;
    int64_t lim = INT64_MAX;  // keys < lim are visible to this row
    if (row < p.rows) {
      a = row / p.rpa;
      pos = p0 + (row / p.G) % p.QB;
      g = row % p.G;
      if (pos < p.chunk) lim = p.n0 + pos + 1;
      else a = -1;
    }
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    for (int j = 0; ok && j < n; ++j) {
      const int b = j & 1;
      if (!__all_sync(0xffffffffu, wait_ab(sfull(b), (j >> 1) & 1, &s_abort))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t s_col = tmem + lane_base + (b ? kColS1 : kColS0);
      uint32_t sv[kT];
      auto sv32 = [&](int c) -> uint32_t(&)[32] { return *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]); };
      const int64_t tile0 = (int64_t)j * kT;
      const bool masked = tile0 + kT > causal_from;
      const int64_t rel = lim - tile0;  // keys i >= rel of this tile are masked for this row
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      float rsum[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[kT / 2];
      // mask + running column max of keys [h*64, h*64 + 64)
      auto mask_max = [&](int h) {
        if (masked) {  // only the tiles that reach the chunk
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (64 * h + i >= rel) sv[64 * h + i] = 0xff800000u;  // -inf
        }
#pragma unroll
        for (int i = 0; i < 64; ++i) mx[i & 3] = fmaxf(mx[i & 3], __uint_as_float(sv[64 * h + i]));
      };
      // P = exp2(S*scale - moff) for keys [h*64, h*64 + 64), packed bf16 pairs
      auto exps = [&](int h, float moff) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float e0 = ptx::ex2(fmaf(__uint_as_float(sv[64 * h + 2 * i]), sl2, -moff));
          const float e1 = ptx::ex2(fmaf(__uint_as_float(sv[64 * h + 2 * i + 1]), sl2, -moff));
          rsum[i & 3] += e0;
          rsum[(i + 2) & 3] += e1;
          pk[32 * h + i] = ptx::pack_bf16(e0, e1);
        }
      };
      auto load_half = [&](int h) {
        ptx::tmem_ld32(s_col + 64 * h, sv32(2 * h));
        ptx::tmem_ld32(s_col + 64 * h + 32, sv32(2 * h + 1));
      };
      auto land_half = [&](int h) {
        ptx::tmem_ld_wait();
        ptx::reg_fence32(sv32(2 * h));
        ptx::reg_fence32(sv32(2 * h + 1));
      };
      auto release_s = [&]() {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(sfree(b));
      };
      bool waited = false;
      load_half(0);
      land_half(0);
      load_half(1);  // the second half lands while the first is processed
      if (j == 0) {
        mask_max(0);
        land_half(1);
        release_s();
        mask_max(1);
        m_used = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
        const float moff = (m_used == -INFINITY) ? 0.f : m_used;
        exps(0, moff);
        exps(1, moff);
      } else {
        // past the first tile the exponentials use the running max
        // speculatively: it only moves when this tile's max exceeds it by 2^8
        mask_max(0);
        exps(0, m_used);
        land_half(1);
        release_s();
        mask_max(1);
        exps(1, m_used);
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
        const bool need = mt > m_used + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          // rescale O and OL of the rows whose max moved: PV_{j-1} must have finished
          if (!__all_sync(0xffffffffu, wait_ab(pvdone, (j - 1) & 1, &s_abort))) {
            ok = false;
            break;
          }
          waited = true;
          ptx::tc_fence_after();
          const float f = need ? ptx::ex2(m_used - mt) : 1.f;
          if (need) {
            m_used = mt;
            l *= f;
          }
#pragma unroll
          for (int c = 0; c < (D + 64) / 32; ++c) {
            uint32_t ov[32];
            ptx::tmem_ld32(tmem + lane_base + kColO + c * 32, ov);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
            ptx::tmem_st32(tmem + lane_base + kColO + c * 32, ov);
          }
          ptx::tmem_st_wait();
          // recompute P with the new max from S_j, still intact in TMEM: the
          // MMA thread issues S_{j+2} into this buffer only after PV_j, which
          // waits for P_j
          load_half(0);
          load_half(1);
          land_half(1);
          ptx::reg_fence32(sv32(0));
          ptx::reg_fence32(sv32(1));
          rsum[0] = rsum[1] = rsum[2] = rsum[3] = 0.f;
          mask_max(0);
          mask_max(1);
          exps(0, m_used);
          exps(1, m_used);
        }
      }
      l += (rsum[0] + rsum[1]) + (rsum[2] + rsum[3]);
      if (j > 0 && !waited) {
        // the P buffer is free once PV_{j-1} has finished reading it
        if (!__all_sync(0xffffffffu, wait_ab(pvdone, (j - 1) & 1, &s_abort))) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
      }
      ptx::tmem_st32(tmem + lane_base + kColP, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      ptx::tmem_st32(tmem + lane_base + kColP + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(pfull);
    }
    // ---- epilogue: A operand of the B GEMM = OL restricted to the row's agent
    if (ok) ok = __all_sync(0xffffffffu, wait_ab(pvdone, (n - 1) & 1, &s_abort));
    if (ok) {
      ptx::tc_fence_after();
      uint32_t olr[64];
      ptx::tmem_ld32(tmem + lane_base + kColOL, *reinterpret_cast<uint32_t(*)[32]>(&olr[0]));
      ptx::tmem_ld32(tmem + lane_base + kColOL + 32, *reinterpret_cast<uint32_t(*)[32]>(&olr[32]));
      ptx::tmem_ld_wait();
      ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&olr[0]));
      ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&olr[32]));
      // own-row staging in the (now idle) V|L ring, [column][row]: lets the
      // agent's window be indexed at run time
      float *olT = reinterpret_cast<float *>(vl_s);
#pragma unroll
      for (int c = 0; c < 64; ++c) olT[c * kM + row] = __uint_as_float(olr[c]);
      const int ar = p.A * p.r;
      const int base_k = a * p.r, base_c = a * p.l_agent_stride;
      uint32_t hi[32], lo[32];
#pragma unroll
      for (int kk = 0; kk < 32; ++kk) {
        float v[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int k = 2 * kk + h;
          v[h] = 0.f;
          if (a >= 0 && k < ar && k >= base_k && k < base_k + p.r) v[h] = olT[(base_c + k - base_k) * kM + row];
        }
        hi[kk] = ptx::pack_bf16(v[0], v[1]);
        const float h0 = __uint_as_float(hi[kk] << 16), h1 = __uint_as_float(hi[kk] & 0xffff0000u);
        lo[kk] = ptx::pack_bf16(v[0] - h0, v[1] - h1);
      }
      ptx::tmem_st32(tmem + lane_base + kColP, hi);
      ptx::tmem_st32(tmem + lane_base + kColP + 32, lo);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(pfull);
      ok = __all_sync(0xffffffffu, wait_ab(pvdone, n & 1, &s_abort));
    }
    if (ok) {
      ptx::tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float *orow = a >= 0 ? p.O + (((int64_t)a * p.chunk + pos) * p.hq + head * p.G + g) * D : nullptr;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        ptx::tmem_ld32(tmem + lane_base + kColO + c * 32, ov);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(ov);
        if (orow) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4 *>(orow + c * 32 + 4 * i) =
                make_float4(__uint_as_float(ov[4 * i]) * inv, __uint_as_float(ov[4 * i + 1]) * inv,
                            __uint_as_float(ov[4 * i + 2]) * inv, __uint_as_float(ov[4 * i + 3]) * inv);
        }
      }
    }
    if (!ok) s_abort = 1;
    ptx::tc_fence_before();
    __syncthreads();
  }
  // every role has passed the barrier above (and drained on abort)
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace ptc

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
inline const char *&prefill_tcgen05_err() {
  static thread_local const char *e = "";
  return e;
}
inline const char *prefill_tcgen05_last_error() { return prefill_tcgen05_err(); }

struct PrefillTcgen05Plan {
  int D, QB, rows, l_width, nk, nv, smem_bytes;
  bool ok;
};

inline PrefillTcgen05Plan prefill_tcgen05_plan(const fla_attn_dims &d, int chunk) {
  PrefillTcgen05Plan pl{};
  pl.ok = false;
  if (d.dtype != FLA_BF16) return pl;
  if (d.head_dim != 64 && d.head_dim != 128) return pl;
  if (d.l_agent_stride != 0 && d.l_agent_stride != d.rank) return pl;
  const int D = d.head_dim, G = d.hq / d.hkv;
  const int l_width = d.l_agent_stride == 0 ? d.rank : d.n_agents * d.rank;
  if (l_width > 64 || d.n_agents * d.rank > 64) return pl;  // OL and the B GEMM's K fit one 64-column box
  const int ag = d.n_agents * G;  // query rows per chunk position
  if (ag > ptc::kM) return pl;
  int QB = 1;
  while (ag * QB * 2 <= ptc::kM && QB < chunk) QB *= 2;
  const int q_bytes = ptc::kM * D * 2, k_bytes = ptc::kT * D * 2, vl_bytes = ptc::kT * (D + 64) * 2;
  const int budget = 227 * 1024 - 1024 /* alignment */ - 1024 /* static shared */;
  int nk = 0, nv = 0;
  const int cand[][2] = {{4, 3}, {3, 3}, {3, 2}, {2, 2}};
  for (const auto &c : cand)
    if (q_bytes + c[0] * k_bytes + c[1] * vl_bytes <= budget) {
      nk = c[0];
      nv = c[1];
      break;
    }
  if (nk == 0) return pl;
  pl.D = D; pl.QB = QB; pl.rows = ag * QB; pl.l_width = l_width; pl.nk = nk; pl.nv = nv;
  pl.smem_bytes = q_bytes + nk * k_bytes + nv * vl_bytes + 1024;
  pl.ok = true;
  return pl;
}

inline fla_status prefill_tcgen05_launch(const fla_attn_dims &d, float scale, const void *Q, const void *K,
                                         const void *V, const void *L, const void *B, int64_t n0, int chunk, float *O,
                                         cudaStream_t s) {
  const PrefillTcgen05Plan pl = prefill_tcgen05_plan(d, chunk);
  if (!pl.ok) {
    prefill_tcgen05_err() = "shape outside the tcgen05 prefill kernel";
    return FLA_ERR_UNSUPPORTED;
  }
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) {
    prefill_tcgen05_err() = "cuTensorMapEncodeTiled is not available from the driver";
    return FLA_ERR_CUDA;
  }
  const int64_t n_total = n0 + chunk;
  CUtensorMap mK, mV, mL, mB;
  const cuuint32_t es[3] = {1, 1, 1};
  {
    const cuuint64_t dims[3] = {(cuuint64_t)d.head_dim, (cuuint64_t)d.hkv, (cuuint64_t)n_total};
    const cuuint64_t strides[2] = {(cuuint64_t)d.head_dim * 2, (cuuint64_t)d.hkv * d.head_dim * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)ptc::kT};
    if (enc(&mK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(K), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&mV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(V), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      prefill_tcgen05_err() = "encoding the K/V tensor maps failed";
      return FLA_ERR_CUDA;
    }
  }
  {
    // one 64-column box per tile; columns past l_width read as zeros
    const cuuint64_t dims[2] = {(cuuint64_t)pl.l_width, (cuuint64_t)n_total};
    const cuuint64_t strides[1] = {(cuuint64_t)d.l_row_stride * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)ptc::kT};
    if (enc(&mL, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(L), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      prefill_tcgen05_err() = "encoding the L tensor map failed";
      return FLA_ERR_CUDA;
    }
  }
  {
    // B_cat [A*r rows][hkv*D cols]; rows past A*r read as zeros
    const cuuint64_t dims[2] = {(cuuint64_t)d.hkv * d.head_dim, (cuuint64_t)d.n_agents * d.rank};
    const cuuint64_t strides[1] = {(cuuint64_t)d.hkv * d.head_dim * 2};
    const cuuint32_t box[2] = {64, 64};
    if (enc(&mB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(B), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      prefill_tcgen05_err() = "encoding the B tensor map failed";
      return FLA_ERR_CUDA;
    }
  }
  ptc::Params prm{};
  prm.Q = reinterpret_cast<const __nv_bfloat16 *>(Q);
  prm.O = O;
  prm.n0 = n0;
  prm.chunk = chunk;
  prm.A = d.n_agents; prm.hq = d.hq; prm.hkv = d.hkv; prm.G = d.hq / d.hkv; prm.r = d.rank;
  prm.QB = pl.QB; prm.rows = pl.rows; prm.rpa = prm.G * pl.QB;
  prm.l_agent_stride = (int)d.l_agent_stride;
  prm.nk = pl.nk; prm.nv = pl.nv;
  prm.scale_log2 = scale * 1.4426950408889634f;
  const int64_t grid64 = (int64_t)d.hkv * ((chunk + pl.QB - 1) / pl.QB);
  if (grid64 > 0x7fffffffLL || n_total > 0x7fffffffLL) {
    prefill_tcgen05_err() = "chunk or context too large";
    return FLA_ERR_UNSUPPORTED;
  }
  cudaError_t e = cudaSuccess;
#define FLA_PTC_CASE(DD)                                                                          \
  if (pl.D == DD) {                                                                               \
    auto kern = ptc::prefill_tc_kernel<DD>;                                                       \
    e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), pl.smem_bytes);                \
    if (e == cudaSuccess) kern<<<(unsigned)grid64, ptc::kThreads, pl.smem_bytes, s>>>(mK, mV, mL, mB, prm); \
    if (e != cudaSuccess) {                                                                       \
      prefill_tcgen05_err() = cudaGetErrorString(e);                                              \
      return FLA_ERR_CUDA;                                                                        \
    }                                                                                             \
    return FLA_OK;                                                                                \
  }
  FLA_PTC_CASE(128) FLA_PTC_CASE(64)
#undef FLA_PTC_CASE
  prefill_tcgen05_err() = "no kernel instance for this plan";
  return FLA_ERR_UNSUPPORTED;
}

}  // namespace fla
