// 5th-generation tensor-core (tcgen05 + TMEM) chunked causal prefill on CTA
// pairs (cta_group::2): Flash-LoRA-Attention for the `chunk` new tokens of
// every agent over a shared context of n0 tokens.
//
// LRAgent technical summary (gist.science), Metodologia section 3: the output
// is P.V_base + (P.L_a).B_a, with B_a applied once per query after the key
// loop; section 2 (BaseShared): K_base / V_base are shared by every agent, so
// one CTA serves all agents' queries of a kv head from one read of each K / V
// tile.  The query at chunk position p (absolute position n0 + p) sees keys
// 0 .. n0 + p.
//
// A CTA holds 128 query rows of one kv head, row = (a*QB + pi)*G + g (agent a,
// position pi of a block of QB consecutive chunk positions, q head g of the
// group), zero rows past the valid ones.  Two CTAs of a cluster (two
// consecutive position blocks) share every key tile: each tcgen05.mma of the
// pair covers their 256 rows, so each CTA copies only half of every operand
// tile.  Per key tile of T keys (T = 96 for d = 128, 128 for d = 64):
//   S_j       = Q . K_j^T            M = 256, N = T: each CTA holds T/2 keys of K_j
//   [O | OL] += P_j . [V_j | L_j]     N = d + 64: each CTA holds half of the
//                                     columns as 32-column groups (64-byte
//                                     swizzle): the even CTA the first
//                                     (d + 64) / 2 columns of [V_j | L_j], the
//                                     odd CTA the rest, so O and OL come out
//                                     as contiguous TMEM columns
//   O        += OL_a . B_a            N = d, after the last tile: A = the OL row
//                                     of each query restricted to its own
//                                     agent's columns (bf16 high + low parts,
//                                     K = 2 x 64), B = [B_cat; B_cat], each CTA
//                                     holding d/2 columns of the head's B_cat
// Four softmax warps per CTA own one TMEM lane (query row) per thread.  P_j
// (bf16) overwrites the first T/2 columns of S_j in tensor memory and is the A
// operand of its P.V MMA.  Three S buffers (with O and OL: 3T + d + 64 <= 512
// TMEM columns) let S_{j+2} be computed while the softmax warps work on tile
// j: the softmax of tile j+1 never waits for anything of tile j.  The running
// max m is only raised (and O, OL rescaled in TMEM) when a tile's max exceeds
// it by more than 2^8, so the rescale is rare; the result is the same softmax
// up to rounding.
//
// In the even CTA, lane 0 of warp 1 issues the S MMAs and lane 0 of warp 7
// the P.V MMAs (and the B GEMM): an issuing thread stalls while the tensor
// core's queue is full, so one thread per stream keeps both streams fed while
// the other waits.  S_j reuses the buffer of P_{j-3} once PV_{j-3} has
// completed.  Warp 0 lane 0 of each CTA issues its K copies (then B_cat),
// warp 6 lane 0 its [V | L] copies; both CTAs' copies count on the even CTA's
// full barriers.  Each MMA group is committed to both CTAs' barriers with one
// multicast commit (stage releases, S ready, PV done); the softmax warps of
// both CTAs arrive on the even CTA's P-ready barriers.  Every wait is bounded;
// on a timeout a CTA records the error and unwinds, the even CTA drains its
// MMAs, and both leave through a cluster barrier before the tensor memory is
// freed.
#pragma once

#include <cuda_bf16.h>

#include "../../include/flash_lora_attn.h"
#include "fla_common.cuh"
#include "decode_tc.cuh"
#include "ptx.cuh"

namespace fla {
namespace ptp {

constexpr int kM = 128;          // query rows per CTA
constexpr int kThreads = 256;    // 8 warps
constexpr int kVWarp = 6;         // V|L producer (warp 0: K producer, 1: S MMAs, 2-5: softmax)
constexpr int kPVWarp = 7;        // P.V MMAs
constexpr int kQBox = 128 * 128;  // one 64-column box of the 128-row Q block
constexpr int kNBuf = 3;          // S (and P) buffers in TMEM
constexpr float kRescaleLog2 = 8.f;
constexpr int kMaxRing = 6;

struct Params {
  const __nv_bfloat16 *Q;
  float *O;
  int64_t n0;
  int32_t chunk, A, hq, hkv, G, r, QB, rows, rpa;  // rpa: rows per agent = QB * G
  int32_t l_agent_stride;
  int32_t nk, nv;  // depths of the K ring and of the [V | L] ring
  float scale_log2;
  // Work items, in launch order: n_full pairs that run their whole key range,
  // then n_split pairs run as two items each, one per half of their key tiles,
  // whose unnormalised rows go to `part` (see PrefillPartRecord below)
  int32_t n_qbp, n_full, n_split;
  float *part;
};

// A half-range item's record of one query row: O and OL accumulated against
// the running max m (log2 units of scaled scores), the row sum l against the
// same max.  Records: [split pair][half][CTA rank][row], floats.
template <int D>
struct PartRec {
  static constexpr int kFloats = D + 64 + 4;  // O[D], OL[64], m, l, 2 pad (16-byte aligned records)
};

template <int D>
struct Shape {
  static constexpr int T = D == 128 ? 96 : 128;  // keys per tile
  static constexpr uint32_t kColO = kNBuf * T;    // O, then OL at kColO + D
  static_assert(kColO + D + 64 <= 512, "tensor memory columns");
};

__device__ __forceinline__ bool wait_ab(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  return ptx::mbar_wait_cluster_or_abort(bar, parity, abort_flag, kErrPrefillWait);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_pair_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmB,
                    const Params p) {
  constexpr int kT = Shape<D>::T;
  constexpr int NC = kT / 32;                  // 32-column chunks of an S row
  constexpr uint32_t kColO = Shape<D>::kColO;
  constexpr uint32_t kColOL = kColO + D;
  constexpr uint32_t kColE = 0;                // epilogue A operand, in S buffer 0 after the loop
  constexpr int VH = D / 2;                    // B_cat columns held by each CTA
  constexpr uint32_t kBRow = VH * 2;           // bytes per row of that half: 128 or 64
  constexpr int kQBytes = kM * D * 2;
  constexpr int kKBox = (kT / 2) * 128;        // one 64-column box of this CTA's T/2 keys
  constexpr int kKBytes = (kT / 2) * D * 2;
  constexpr int kGroups = (D + 64) / 64;       // 32-column groups of [V | L] per CTA: 3 or 2
  constexpr int kGroupBytes = kT * 64;         // T keys x 32 columns
  constexpr int kVLBytes = kGroups * kGroupBytes;
  constexpr int kBBytes = 64 * VH * 2;         // this CTA's half of the head's B_cat rows
  static_assert(kVLBytes * 2 >= 64 * kM * 4, "the epilogue stages OL in the V|L ring");
  static_assert(kBBytes <= kKBytes, "B_cat goes into one K stage");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *q_s = smem;
  uint8_t *k_s = smem + kQBytes;
  uint8_t *vl_s = k_s + p.nk * kKBytes;
  __shared__ __align__(8) uint64_t bars[4 * kMaxRing + 3 * kNBuf + 3];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();  // 0: the CTA that issues the MMAs
  const int item = (int)(blockIdx.x >> 1);
  int pr = item, part_half = -1;  // -1: the whole key range
  if (item >= p.n_full) {
    pr = p.n_full + (item - p.n_full) / 2;
    part_half = (item - p.n_full) & 1;
  }
  const int head = pr % p.hkv;
  const int qbp = p.n_qbp - 1 - pr / p.hkv;  // late chunk blocks (most keys) first
  const int p0 = (2 * qbp + (int)rank) * p.QB;
  // both CTAs run the tiles of the pair's later block; the earlier block's
  // rows see the extra keys masked
  const int64_t n_keys = p.n0 + min(p.chunk, (2 * qbp + 2) * p.QB);
  const int n_all = (int)((n_keys + kT - 1) / kT);
  // this item's key tiles [tb, tb + n)
  const int tb = part_half == 1 ? n_all / 2 : 0;
  const int n = part_half < 0 ? n_all : (part_half == 0 ? n_all / 2 : n_all - n_all / 2);
  const bool full = part_half < 0;
  const int64_t causal_from = p.n0 + p0;

  const uint32_t bar0 = ptx::smem_u32(bars);
  auto kf = [&](int s) { return bar0 + 8u * s; };
  auto ke = [&](int s) { return bar0 + 8u * (kMaxRing + s); };
  auto vf = [&](int s) { return bar0 + 8u * (2 * kMaxRing + s); };
  auto ve = [&](int s) { return bar0 + 8u * (3 * kMaxRing + s); };
  auto sfull = [&](int b) { return bar0 + 8u * (4 * kMaxRing + b); };
  auto pfull = [&](int b) { return bar0 + 8u * (4 * kMaxRing + kNBuf + b); };
  auto pvdone = [&](int b) { return bar0 + 8u * (4 * kMaxRing + 2 * kNBuf + b); };
  const uint32_t bfull = bar0 + 8u * (4 * kMaxRing + 3 * kNBuf);
  auto drain = [&](int w) { return bar0 + 8u * (4 * kMaxRing + 3 * kNBuf + 1 + w); };  // per issuing thread
  // the even CTA's copy of a barrier
  auto lead = [&](uint32_t a) { return ptx::mapa_cluster(a, 0); };

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
    for (int b = 0; b < kNBuf; ++b) {
      ptx::mbar_init(sfull(b), 1);
      ptx::mbar_init(pfull(b), 8);  // 4 softmax warps in each CTA
      ptx::mbar_init(pvdone(b), 1);
    }
    ptx::mbar_init(bfull, 1);
    ptx::mbar_init(drain(0), 1);
    ptx::mbar_init(drain(1), 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(&s_tmem), 512);
    ptx::tmem_relinquish_pair();
  }
  // Q rows of this CTA's block into the K-major 128-byte-swizzled layout the MMA reads
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
    *reinterpret_cast<uint4 *>(q_s + (c8 >> 3) * kQBox + row * 128 + (((c8 & 7) ^ (row & 7)) << 4)) = v;
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  // the peer arrives on this CTA's barriers and its MMAs read this CTA's Q:
  // both CTAs initialised and staged before anything is issued
  ptx::cluster_sync_all();
  ptx::tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool ok = true;

  if (warp == 0 || warp == kVWarp) {
    // ------------------------------------------------------------ TMA producers (both CTAs)
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
        if (rank == 0) ptx::mbar_arrive_expect_tx(kf(st), 2 * kKBytes);
        const uint32_t dst = ptx::smem_u32(k_s + st * kKBytes);
        const uint32_t fb = lead(kf(st));
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
          ptx::tma_load_3d_pair(dst + b * kKBox, &tmK, b * 64, head, (tb + j) * kT + (int)rank * (kT / 2), fb);
        k_issued = j + 1;
      }
      // this CTA's half of the head's B_cat rows, into the K ring once the
      // last S MMA (hence every S MMA) has finished with it
      if (ok && full) ok = wait_ab(ke((n - 1) % p.nk), ((n - 1) / p.nk) & 1, &s_abort);
      if (ok && full) {
        if (rank == 0) ptx::mbar_arrive_expect_tx(bfull, 2 * kBBytes);
        ptx::tma_load_2d_pair(ptx::smem_u32(k_s), &tmB, head * D + (int)rank * VH, 0, lead(bfull));
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
        if (rank == 0) ptx::mbar_arrive_expect_tx(vf(st), 2 * kVLBytes);
        const uint32_t dst = ptx::smem_u32(vl_s + st * kVLBytes);
        const uint32_t fb = lead(vf(st));
#pragma unroll
        for (int gi = 0; gi < kGroups; ++gi) {
          const int g = (int)rank * kGroups + gi;  // group of [V | L]
          if (g < D / 32)
            ptx::tma_load_3d_pair(dst + gi * kGroupBytes, &tmV, 32 * g, head, (tb + j) * kT, fb);
          else
            ptx::tma_load_2d_pair(dst + gi * kGroupBytes, &tmL, 32 * (g - D / 32), (tb + j) * kT, fb);
        }
        v_issued = j + 1;
      }
      if (!ok) s_abort = 1;
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (s_abort && lane == 0 && rank == 0) {
      // the even CTA's full barriers count both CTAs' copies: wait (bounded)
      // for the latest phase of each stage
      for (int j = max(0, k_issued - p.nk); j < k_issued; ++j) ptx::mbar_wait_cluster(kf(j % p.nk), (j / p.nk) & 1);
      for (int j = max(0, v_issued - p.nv); j < v_issued; ++j) ptx::mbar_wait_cluster(vf(j % p.nv), (j / p.nv) & 1);
      if (b_issued) ptx::mbar_wait_cluster(bfull, 0);
    }
  } else if (warp == 1 || warp == kPVWarp) {
    // ------------------------------------------------------------ MMA issuers (even CTA)
    bool issued_any = false;
    // one arrival on the barrier at the same offset in both CTAs
    auto commit_both = [&](uint32_t bar) { ptx::tc_commit_pair_mc(bar, 0x3); };
    if (lane == 0 && rank == 0 && warp == 1) {
      // S_j = Q . K_j^T into buffer j % 3
      const uint32_t idesc_s = ptx::idesc_bf16_f32(2 * kM, kT);
      const uint64_t d_q = ptx::smem_desc_k128(ptx::smem_u32(q_s));
      const uint64_t d_k = ptx::smem_desc_k128(ptx::smem_u32(k_s));
      for (int j = 0; ok && j < n; ++j) {
        const int st = j % p.nk, b = j % kNBuf;
        if (!wait_ab(kf(st), (j / p.nk) & 1, &s_abort)) { ok = false; break; }
        // the buffer's P_{j-3} has been read: PV_{j-3} has completed (its
        // barrier's previous phase, PV_{j-6}, was waited for three tiles ago)
        if (j >= kNBuf && !wait_ab(pvdone(b), ((j - kNBuf) / kNBuf) & 1, &s_abort)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint64_t dk = ptx::desc_advance(d_k, st * kKBytes);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ptx::tc_mma_f16_pair(tmem + b * kT, ptx::desc_advance(d_q, (ks >> 2) * kQBox + (ks & 3) * 32),
                               ptx::desc_advance(dk, (ks >> 2) * kKBox + (ks & 3) * 32), idesc_s, ks > 0 ? 1u : 0u);
        issued_any = true;
        commit_both(ke(st));
        commit_both(sfull(b));
      }
      if (!ok) s_abort = 1;
    }
    if (lane == 0 && rank == 0 && warp == kPVWarp) {
      // [O | OL] += P_j . [V_j | L_j], then the B GEMM
      const uint32_t idesc_pv = ptx::idesc_bf16_f32(2 * kM, D + 64) | (1u << 16);  // B MN-major
      const uint32_t idesc_ep = ptx::idesc_bf16_f32(2 * kM, D) | (1u << 16);
      const uint64_t d_vl = ptx::smem_desc_mn64(ptx::smem_u32(vl_s), kGroupBytes);
      for (int j = 0; ok && j < n; ++j) {
        const int st = j % p.nv, b = j % kNBuf;
        // the V|L stage is normally in long before P_j: wait for it first
        if (!wait_ab(vf(st), (j / p.nv) & 1, &s_abort)) { ok = false; break; }
        if (!wait_ab(pfull(b), (j / kNBuf) & 1, &s_abort)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint64_t dvl = ptx::desc_advance(d_vl, st * kVLBytes);
#pragma unroll
        for (int ks = 0; ks < kT / 16; ++ks)
          // 16 keys further on: 16 rows of 64 bytes in every group
          ptx::tc_mma_f16_ts_pair(tmem + kColO, tmem + b * kT + ks * 8, ptx::desc_advance(dvl, ks * 16 * 64),
                                  idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
        issued_any = true;
        commit_both(ve(st));
        commit_both(pvdone(b));
      }
      // O += [OL_hi | OL_lo] . [B_cat ; B_cat]   (K = 2 x 64), signalled as "tile n"
      // (a half-range item leaves its rows unnormalised to the merge kernel)
      if (ok && full) ok = wait_ab(pfull(n % kNBuf), (n / kNBuf) & 1, &s_abort);
      if (ok && full) ok = wait_ab(bfull, 0, &s_abort);
      if (ok && full) {
        ptx::tc_fence_after();
        const uint32_t kb = ptx::smem_u32(k_s);
        const uint64_t dbb = VH == 64 ? ptx::smem_desc_mn128(kb, kBBytes) : ptx::smem_desc_mn64(kb, kBBytes);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          ptx::tc_mma_f16_ts_pair(tmem + kColO, tmem + kColE + ks * 8, ptx::desc_advance(dbb, (ks & 3) * 16 * kBRow),
                                  idesc_ep, 1u);
        commit_both(pvdone(n % kNBuf));
      }
      if (!ok) s_abort = 1;
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (s_abort && lane == 0 && rank == 0 && issued_any) {
      const uint32_t dr = drain(warp == 1 ? 0 : 1);
      ptx::tc_commit_pair(lead(dr));  // completes once every MMA this thread issued has finished
      ptx::mbar_wait_cluster(dr, 0);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ softmax + epilogue (both CTAs, own rows)
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
    // Waits for PV_i to have finished.  pvdone(i % 3) completes once per PV
    // of that buffer; PV_{i-3} has finished whenever this is called (S_i,
    // issued after PV_{i-3} completed, has been seen), so the parity names
    // PV_i alone.
    auto wait_pv = [&](int i) -> bool {
      return __all_sync(0xffffffffu, wait_ab(pvdone(i % kNBuf), (i / kNBuf) & 1, &s_abort));
    };
    for (int j = 0; ok && j < n; ++j) {
      const int b = j % kNBuf;
      if (!__all_sync(0xffffffffu, wait_ab(sfull(b), (j / kNBuf) & 1, &s_abort))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t s_col = tmem + lane_base + b * kT;
      uint32_t sv[kT];
#pragma unroll
      for (int c = 0; c < NC; ++c) ptx::tmem_ld32(s_col + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]));
      ptx::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < NC; ++c) ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]));
      const int64_t tile0 = (int64_t)(tb + j) * kT;
      if (tile0 + kT > causal_from) {  // only the tiles that reach the chunk
        const int64_t rel = lim - tile0;  // keys i >= rel of this tile are masked for this row
#pragma unroll
        for (int i = 0; i < kT; ++i)
          if (i >= rel) sv[i] = 0xff800000u;  // -inf
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < kT; ++i) mx[i & 3] = fmaxf(mx[i & 3], __uint_as_float(sv[i]));
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
      if (j == 0) {
        m_used = mt;
      } else {
        // the running max only moves when this tile's max exceeds it by 2^8
        const bool need = mt > m_used + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          // rescale O and OL of the rows whose max moved, once PV_{j-1} has
          // finished (PV_j waits for P_j)
          if (!wait_pv(j - 1)) {
            ok = false;
            break;
          }
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
        }
      }
      const float moff = (m_used == -INFINITY) ? 0.f : m_used;
      float rsum[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[kT / 2];
#pragma unroll
      for (int i = 0; i < kT / 2; ++i) {
        const float e0 = ptx::ex2(fmaf(__uint_as_float(sv[2 * i]), sl2, -moff));
        const float e1 = ptx::ex2(fmaf(__uint_as_float(sv[2 * i + 1]), sl2, -moff));
        pk[i] = ptx::pack_bf16(e0, e1);
        // the normaliser sums the bf16 probabilities the MMA multiplies, so the
        // weights of each output row sum to one up to fp32 rounding
        rsum[i & 3] += __uint_as_float(pk[i] << 16);
        rsum[(i + 2) & 3] += __uint_as_float(pk[i] & 0xffff0000u);
      }
      l += (rsum[0] + rsum[1]) + (rsum[2] + rsum[3]);
      // P_j over the first T/2 columns of its own S buffer: nothing else reads
      // or writes that buffer until PV_j
#pragma unroll
      for (int c = 0; c < kT / 64; ++c) ptx::tmem_st32(s_col + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&pk[32 * c]));
      if constexpr ((kT / 2) % 32 != 0) ptx::tmem_st16(s_col + 32 * (kT / 64), &pk[32 * (kT / 64)]);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster_relaxed(lead(pfull(b)));
    }
    // ---- epilogue: A operand of the B GEMM = OL restricted to the row's agent
    if (ok) ok = wait_pv(n - 1);  // every P.V MMA has finished
    if (ok && !full) {
      // half-range item: this row's O and OL against m_used, then m_used and l
      ptx::tc_fence_after();
      float *rec = p.part + ((((int64_t)(pr - p.n_full) * 2 + part_half) * 2 + rank) * kM + row) *
                                PartRec<D>::kFloats;
#pragma unroll
      for (int c = 0; c < (D + 64) / 32; ++c) {
        uint32_t ov[32];
        ptx::tmem_ld32(tmem + lane_base + kColO + c * 32, ov);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(ov);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<float4 *>(rec + c * 32 + 4 * i) =
              make_float4(__uint_as_float(ov[4 * i]), __uint_as_float(ov[4 * i + 1]), __uint_as_float(ov[4 * i + 2]),
                          __uint_as_float(ov[4 * i + 3]));
      }
      *reinterpret_cast<float4 *>(rec + D + 64) = make_float4(m_used, l, 0.f, 0.f);
    }
    if (ok && full) {
      ptx::tc_fence_after();
      uint32_t olr[64];
      ptx::tmem_ld32(tmem + lane_base + kColOL, *reinterpret_cast<uint32_t(*)[32]>(&olr[0]));
      ptx::tmem_ld32(tmem + lane_base + kColOL + 32, *reinterpret_cast<uint32_t(*)[32]>(&olr[32]));
      ptx::tmem_ld_wait();
      ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&olr[0]));
      ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&olr[32]));
      // own-row staging in this CTA's (now idle) V|L ring, [column][row]
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
      ptx::tmem_st32(tmem + lane_base + kColE, hi);
      ptx::tmem_st32(tmem + lane_base + kColE + 32, lo);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster_relaxed(lead(pfull(n % kNBuf)));
      ok = wait_pv(n);  // the B GEMM, committed as "tile n"
    }
    if (ok && full) {
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
  // every role has passed the barrier above (and drained on abort); neither
  // CTA frees the pair's tensor memory (or exits) while the other still works
  __syncthreads();
  ptx::cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, 512);
  }
}

// Merge of a split pair's two half-range items (LRAgent technical summary,
// Metodologia section 3: O = (P.V_base + (P.L_a).B_a) / l over all keys).
// Per query row the two records are combined as online softmax combines two
// blocks (each scaled by 2^(m_half - m), m the larger running max), OL is
// restricted to the row's agent and multiplied by B_a in fp32, and O is
// written.  One warp per row; lanes over the output columns.
template <int D>
__global__ void __launch_bounds__(256) prefill_merge_kernel(const Params p, const __nv_bfloat16 *__restrict__ B) {
  constexpr int RF = PartRec<D>::kFloats;
  __shared__ float s_ol[8][64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * 8 + warp;  // [split pair][CTA rank][row]
  if (gw >= (int64_t)p.n_split * 2 * kM) return;
  const int sp = (int)(gw / (2 * kM)), rank = (int)((gw / kM) & 1), row = (int)(gw % kM);
  const int pr = p.n_full + sp;
  const int head = pr % p.hkv, qbp = p.n_qbp - 1 - pr / p.hkv;
  if (row >= p.rows) return;
  const int a = row / p.rpa, pos = (2 * qbp + rank) * p.QB + (row / p.G) % p.QB, g = row % p.G;
  if (pos >= p.chunk) return;
  const float *r0 = p.part + ((((int64_t)sp * 2 + 0) * 2 + rank) * kM + row) * RF;
  const float *r1 = p.part + ((((int64_t)sp * 2 + 1) * 2 + rank) * kM + row) * RF;
  const float m0 = r0[D + 64], l0 = r0[D + 65], m1 = r1[D + 64], l1 = r1[D + 65];
  const float m = fmaxf(m0, m1);
  const float w0 = m0 == -INFINITY ? 0.f : exp2f(m0 - m);
  const float w1 = m1 == -INFINITY ? 0.f : exp2f(m1 - m);
  const float lt = w0 * l0 + w1 * l1;
  const float inv = lt > 0.f ? 1.f / lt : 0.f;
  for (int c = lane; c < 64; c += 32) s_ol[warp][c] = (w0 * r0[D + c] + w1 * r1[D + c]) * inv;
  __syncwarp();
  const int base_k = a * p.r, base_c = a * p.l_agent_stride;
  const int64_t ldb = (int64_t)p.hkv * D;
  const __nv_bfloat16 *bh = B + (int64_t)base_k * ldb + head * D;
  float *orow = p.O + (((int64_t)a * p.chunk + pos) * p.hq + head * p.G + g) * D;
  for (int d = lane; d < D; d += 32) {
    float o = (w0 * r0[d] + w1 * r1[d]) * inv;
    for (int k = 0; k < p.r; ++k) o = fmaf(s_ol[warp][base_c + k], __bfloat162float(bh[(int64_t)k * ldb + d]), o);
    orow[d] = o;
  }
}

}  // namespace ptp

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
inline const char *&prefill_tcgen05_err() {
  static thread_local const char *e = "";
  return e;
}
inline const char *prefill_tcgen05_last_error() { return prefill_tcgen05_err(); }

struct PrefillTcgen05Plan {
  int D, QB, rows, l_width, T, nk, nv, smem_bytes, n_qbp;
  int n_full, n_split;   // work items: whole-range pairs, pairs split over two items
  size_t part_bytes;     // workspace the split pairs' row records need
  bool ok;
};

// Shape limits, query block, tile and ring depths of the tcgen05 prefill.
inline PrefillTcgen05Plan prefill_tcgen05_plan(const fla_attn_dims &d, int chunk, int64_t n0) {
  PrefillTcgen05Plan pl{};
  pl.ok = false;
  if (d.dtype != FLA_BF16) return pl;
  if (d.head_dim != 64 && d.head_dim != 128) return pl;
  if (d.l_agent_stride != 0 && d.l_agent_stride != d.rank) return pl;
  const int D = d.head_dim, G = d.hq / d.hkv;
  const int l_width = d.l_agent_stride == 0 ? d.rank : d.n_agents * d.rank;
  if (l_width > 64 || d.n_agents * d.rank > 64) return pl;  // OL and the B GEMM's K fit one 64-column box
  const int ag = d.n_agents * G;  // query rows per chunk position
  if (ag > ptp::kM) return pl;
  int QB = 1;
  while (ag * QB * 2 <= ptp::kM && QB < chunk) QB *= 2;
  pl.D = D;
  pl.QB = QB;
  pl.rows = ag * QB;
  pl.l_width = l_width;
  pl.T = D == 128 ? ptp::Shape<128>::T : ptp::Shape<64>::T;
  const int q_bytes = ptp::kM * D * 2, k_bytes = (pl.T / 2) * D * 2, vl_bytes = (D + 64) / 64 * pl.T * 64;
  const int budget = 227 * 1024 - 1024 /* alignment */ - 1024 /* static shared */;
  for (int depth = ptp::kMaxRing; depth >= 2; --depth)
    if (q_bytes + depth * (k_bytes + vl_bytes) <= budget) {
      pl.nk = pl.nv = depth;
      break;
    }
  if (pl.nk == 0) return pl;
  pl.smem_bytes = q_bytes + pl.nk * k_bytes + pl.nv * vl_bytes + 1024;
  const int n_qb = (chunk + QB - 1) / QB;
  pl.n_qbp = (n_qb + 1) / 2;
  // The pairs of a last, partly filled wave run as two half-range items each
  // (merged afterwards), so that wave ends about halfway; with fewer pairs
  // than half the pair slots, every pair is split.  Only pairs of at least two
  // key tiles split; the last pairs of the launch order have the fewest keys.
  const int64_t pairs = (int64_t)d.hkv * pl.n_qbp;
  const int slots = device_sm_count() / 2;
  const int64_t min_tiles = (n0 + std::min(chunk, 2 * QB) + pl.T - 1) / pl.T;
  int64_t n_split = 0;
  if (min_tiles >= 2 && slots > 0) {
    if (2 * pairs <= slots) n_split = pairs;
    else if (pairs % slots != 0 && 2 * (pairs % slots) <= slots) n_split = pairs % slots;
  }
  pl.n_split = (int)n_split;
  pl.n_full = (int)(pairs - n_split);
  pl.part_bytes = (size_t)n_split * 2 * 2 * ptp::kM * (D == 128 ? ptp::PartRec<128>::kFloats : ptp::PartRec<64>::kFloats) * 4;
  pl.ok = true;
  return pl;
}

inline fla_status prefill_tcgen05_launch(const fla_attn_dims &d, float scale, const void *Q, const void *K,
                                         const void *V, const void *L, const void *B, int64_t n0, int chunk, float *O,
                                         void *workspace, size_t workspace_bytes, cudaStream_t s) {
  PrefillTcgen05Plan pl = prefill_tcgen05_plan(d, chunk, n0);
  if (pl.ok && pl.n_split > 0 &&
      (workspace == nullptr || workspace_bytes < pl.part_bytes || (reinterpret_cast<uintptr_t>(workspace) & 15u))) {
    // no room for the split pairs' records: every pair runs its whole range
    pl.n_full += pl.n_split;
    pl.n_split = 0;
  }
  if (!pl.ok) {
    prefill_tcgen05_err() = "shape outside the tcgen05 prefill kernel";
    return FLA_ERR_UNSUPPORTED;
  }
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) {
    prefill_tcgen05_err() = "cuTensorMapEncodeTiled is not available from the driver";
    return FLA_ERR_CUDA;
  }
  const int D = pl.D, VH = D / 2;
  const int64_t n_total = n0 + chunk;
  CUtensorMap mK, mV, mL, mB;
  const cuuint32_t es[3] = {1, 1, 1};
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)d.hkv, (cuuint64_t)n_total};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)d.hkv * D * 2};
    const cuuint32_t kbox[3] = {64, 1, (cuuint32_t)(pl.T / 2)};  // this CTA's half of a tile's keys
    const cuuint32_t vbox[3] = {32, 1, (cuuint32_t)pl.T};        // one 32-column group
    if (enc(&mK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(K), dims, strides, kbox, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&mV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(V), dims, strides, vbox, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      prefill_tcgen05_err() = "encoding the K/V tensor maps failed";
      return FLA_ERR_CUDA;
    }
  }
  {
    // 32-column groups (64-byte swizzle); columns past l_width read as zeros
    const cuuint64_t dims[2] = {(cuuint64_t)pl.l_width, (cuuint64_t)n_total};
    const cuuint64_t strides[1] = {(cuuint64_t)d.l_row_stride * 2};
    const cuuint32_t box[2] = {32, (cuuint32_t)pl.T};
    if (enc(&mL, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(L), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      prefill_tcgen05_err() = "encoding the L tensor map failed";
      return FLA_ERR_CUDA;
    }
  }
  {
    // B_cat [A*r rows][hkv*D cols]: D/2 columns per CTA; rows past A*r read as zeros
    const cuuint64_t dims[2] = {(cuuint64_t)d.hkv * D, (cuuint64_t)d.n_agents * d.rank};
    const cuuint64_t strides[1] = {(cuuint64_t)d.hkv * D * 2};
    const cuuint32_t box[2] = {(cuuint32_t)VH, 64};
    if (enc(&mB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(B), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, VH == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      prefill_tcgen05_err() = "encoding the B tensor map failed";
      return FLA_ERR_CUDA;
    }
  }
  ptp::Params prm{};
  prm.Q = reinterpret_cast<const __nv_bfloat16 *>(Q);
  prm.O = O;
  prm.n0 = n0;
  prm.chunk = chunk;
  prm.A = d.n_agents; prm.hq = d.hq; prm.hkv = d.hkv; prm.G = d.hq / d.hkv; prm.r = d.rank;
  prm.QB = pl.QB; prm.rows = pl.rows; prm.rpa = prm.G * pl.QB;
  prm.l_agent_stride = (int)d.l_agent_stride;
  prm.nk = pl.nk; prm.nv = pl.nv;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.n_qbp = pl.n_qbp;
  prm.n_full = pl.n_full;
  prm.n_split = pl.n_split;
  prm.part = reinterpret_cast<float *>(workspace);
  const int64_t grid64 = 2LL * (pl.n_full + 2LL * pl.n_split);
  if (grid64 > 0x7fffffffLL || n_total > 0x7fffffffLL) {
    prefill_tcgen05_err() = "chunk or context too large";
    return FLA_ERR_UNSUPPORTED;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid64);
  cfg.blockDim = dim3(ptp::kThreads);
  cfg.dynamicSmemBytes = pl.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaSuccess;
  const unsigned merge_blocks = (unsigned)((2LL * ptp::kM * pl.n_split + 7) / 8);  // one warp per row
#define FLA_PTP_CASE(DD)                                                                                \
  if (D == DD) {                                                                                        \
    auto kern = ptp::prefill_pair_kernel<DD>;                                                           \
    e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), pl.smem_bytes);                      \
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, kern, mK, mV, mL, mB, prm);                     \
    if (e == cudaSuccess && pl.n_split > 0) {                                                           \
      ptp::prefill_merge_kernel<DD><<<merge_blocks, 256, 0, s>>>(prm, reinterpret_cast<const __nv_bfloat16 *>(B)); \
      e = cudaGetLastError();                                                                           \
    }                                                                                                   \
    if (e != cudaSuccess) {                                                                             \
      prefill_tcgen05_err() = cudaGetErrorString(e);                                                    \
      return FLA_ERR_CUDA;                                                                              \
    }                                                                                                   \
    return FLA_OK;                                                                                      \
  }
  FLA_PTP_CASE(128) FLA_PTP_CASE(64)
#undef FLA_PTP_CASE
  prefill_tcgen05_err() = "no kernel instance for this plan";
  return FLA_ERR_UNSUPPORTED;
}

}  // namespace fla
