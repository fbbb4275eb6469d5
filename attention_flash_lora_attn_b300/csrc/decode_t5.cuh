// 5th-generation tensor-core (tcgen05 + TMEM) decode: Flash-LoRA-Attention
// over a shared base cache, one query token per agent and request.
//
// LRAgent technical summary (gist.science), Metodologia section 3: the output
// is P.V_base + (P.L_a).B_a, the r-wide P.L_a accumulated in the same pass as
// P.V_base and B_a applied once per query after the token loop; section 2
// (BaseShared): every agent's query rows of a kv head are served from one
// read of each K / V tile.
//
// Work items are the (request, kv head, unit) triples of the mma.sync decode
// kernel (decode_tc.cuh), with units a multiple of 128 tokens, and each CTA
// writes that kernel's partial record ([rows][d + r] | m | l), so the same
// merge kernel combines the units and applies B.  Inside a CTA the roles of
// P and S are transposed so the per-row LoRA width never has to fit TMEM
// next to the d-wide accumulator of every row:
//   S^T  = K_tile . Q^T        M = 128 keys (one TMEM lane per key),
//                              N = 64 query rows (A*G of them real)
//   O^T += V_tile^T . P^T      M = d = 128, K = keys: V as an MN-major A
//   OL^T+= L_tile^T . P^T      M = 128 L columns per MMA (a chunk of the
//                              agents' r-column blocks), N = only the query
//                              rows of the agents owning those columns (the
//                              P^T operand starts at the chunk's first row),
//                              so each chunk costs a few TMEM columns
//   l                          row sums: each softmax thread adds its key's P
//                              values into its own TMEM lane (64 columns, one
//                              per query row); the 128 lanes are summed once,
//                              after the last tile
// P^T (bf16, key-major rows of 64 query rows) is written by the four softmax
// warps to shared memory as an MN-major B operand.  The running max per query
// row lives in shared memory; exponentials use it speculatively and the CTA
// votes once per tile on whether any row's max rose by more than 2^8, in which
// case (rarely, and on the first tile) the row maxima are reduced across the
// 128 keys, O^T, OL^T and the per-lane row sums are rescaled in TMEM and P
// is recomputed.
//
// Warp roles: warp 0 lane 0 streams the K ring (128-token tiles), warp 6
// lane 0 the V|L ring (64-token halves); warp 1 owns TMEM and lane 0 issues
// every MMA; warps 2..5 run the softmax and write the partial record.  Every
// wait is bounded; a timeout records the error, drains this CTA's copies and
// MMAs, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>

#include "../../include/flash_lora_attn.h"
#include "decode_tc.cuh"
#include "fla_common.cuh"
#include "ptx.cuh"

namespace fla {
namespace dt5 {

constexpr int D = 128;            // head_dim
constexpr int kKeys = 128;        // keys per tile (M of S^T)
constexpr int kHalf = 64;         // keys per V|L stage
constexpr int kN = 64;            // query rows per CTA (N), A*G <= 64 real
constexpr int kThreads = 224;     // 7 warps
constexpr int kVWarp = 6;
constexpr int kMaxRing = 8;
constexpr int kMaxLChunks = 4;    // L columns per tile <= 4 x 128
constexpr uint32_t kColS0 = 0, kColS1 = 64, kColO = 128, kColLs = 192, kColOL = 256;
constexpr float kRescaleLog2 = 8.f;
constexpr int kQBytes = kN * D * 2;        // 16 KB
constexpr int kPBytes = kKeys * kN * 2;    // 16 KB
constexpr int kKBytes = kKeys * D * 2;     // 32 KB
constexpr int kVBytes = kHalf * D * 2;     // 16 KB
constexpr int kLBoxBytes = kHalf * 128;    // one 64-column L box of a half tile

struct Params {
  const __nv_bfloat16 *Q;
  const int32_t *offsets;
  float *partials;
  int2 *pair_info;
  int32_t n_req, A, hq, hkv, G, r, rows;
  int32_t l_agent_stride, l_width, n_lbox, n_lchunk;
  int32_t unit_tokens, single_len, part_stride;
  int32_t nk, nv, vl_bytes;
  // OL^T chunk c: query rows [ol_row0[c], ol_row0[c] + ol_rows[c]) (a multiple
  // of 8, a multiple of 16) accumulated in TMEM columns kColOL + ol_col[c] + i
  int32_t ol_row0[kMaxLChunks], ol_rows[kMaxLChunks], ol_col[kMaxLChunks];
  float scale_log2;
};

__device__ __forceinline__ bool wait_ab(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  return ptx::mbar_wait_or_abort(bar, parity, abort_flag, kErrDecodeT5Wait);
}

__global__ void __launch_bounds__(kThreads, 1)
decode_t5_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmL, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *q_s = smem;
  uint8_t *p_s = q_s + kQBytes;
  uint8_t *k_s = p_s + kPBytes;
  uint8_t *vl_s = k_s + p.nk * kKBytes;
  __shared__ __align__(8) uint64_t bars[4 * kMaxRing + 10];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int s_info[8];
  __shared__ int s_vote[2][4];
  // per-warp row maxima of a rescale tile; one buffer suffices: a second
  // rescale starts only after the next tile's vote, which every warp reaches
  // after reading this one
  __shared__ __align__(16) float s_red[4][kN];
  __shared__ __align__(16) float s_m[2][kN];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x % p.hkv;
  const int unit_global = blockIdx.x / p.hkv;
  const uint32_t bar0 = ptx::smem_u32(bars);
  auto kf = [&](int s) { return bar0 + 8u * s; };
  auto ke = [&](int s) { return bar0 + 8u * (kMaxRing + s); };
  auto vf = [&](int s) { return bar0 + 8u * (2 * kMaxRing + s); };
  auto ve = [&](int s) { return bar0 + 8u * (3 * kMaxRing + s); };
  auto sfull = [&](int b) { return bar0 + 8u * (4 * kMaxRing + b); };
  auto sfree = [&](int b) { return bar0 + 8u * (4 * kMaxRing + 2 + b); };
  const uint32_t pfull = bar0 + 8u * (4 * kMaxRing + 4);
  const uint32_t pvdone = bar0 + 8u * (4 * kMaxRing + 5);
  const uint32_t vote = bar0 + 8u * (4 * kMaxRing + 6);
  const uint32_t red = bar0 + 8u * (4 * kMaxRing + 7);
  const uint32_t drain = bar0 + 8u * (4 * kMaxRing + 8);

  // Launched with programmatic dependent launch: the token loop reads only
  // this call's inputs, so it may overlap the previous kernel of the stream
  // (this library's merge kernel, which reads the workspace);
  // griddepcontrol.wait runs before this CTA's first global write.
  if (warp == 0) {
    const int found = dec::map_unit(unit_global, p.unit_tokens, p.single_len, p.offsets, p.n_req, s_info);
    if (lane == 0) s_info[5] = found;
  }
  if (threadIdx.x == 32) {
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
    ptx::mbar_init(vote, 4);
    ptx::mbar_init(red, 4);
    ptx::mbar_init(drain, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  // the merge kernel behind this one may be scheduled now; it still waits for
  // this grid to finish before reading the partials
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!s_info[5]) return;  // grid slack beyond the last unit (uniform over the CTA)
  const int qreq = s_info[0], unit = s_info[1], n_units = s_info[2];
  const int tok_begin = s_info[3], n_tok = s_info[4], slot = s_info[6];
  const int n = (n_tok + kKeys - 1) / kKeys;  // 128-token tiles of this unit
  // The kv heads of a unit share its L rows.  Head h visits the unit's tiles
  // starting at tile h, so one head pulls each L tile from HBM and the others
  // read it from L2 a tile later instead of all waiting on the same miss (the
  // online softmax is order-independent).
  const int rot = n > 0 ? head % n : 0;
  auto key_tile = [&](int j) { const int t = j + rot; return t >= n ? t - n : t; };

  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&s_tmem), 512);
    ptx::tmem_relinquish();
  }
  // Q rows (n = a*G + g) into the K-major 128-byte-swizzled layout
  for (int e = threadIdx.x; e < kN * (D / 8); e += kThreads) {
    const int row = e / (D / 8), c8 = e % (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < p.rows) {
      const int a = row / p.G, g = row % p.G;
      v = *reinterpret_cast<const uint4 *>(p.Q + (((int64_t)qreq * p.A + a) * p.hq + head * p.G + g) * D + c8 * 8);
    }
    *reinterpret_cast<uint4 *>(q_s + (c8 >> 3) * (kN * 128) + row * 128 + (((c8 & 7) ^ (row & 7)) << 4)) = v;
  }
  if (threadIdx.x < kN) s_m[0][threadIdx.x] = threadIdx.x < p.rows ? -INFINITY : 0.f;
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool ok = true;

  if (warp == 0 || warp == kVWarp) {
    // ------------------------------------------------------------ TMA producers
    int k_issued = 0, v_issued = 0;
    if (lane == 0 && warp == 0) {
      ptx::prefetch_tmap(&tmK);
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
          ptx::tma_load_3d(dst + b * (kKeys * 128), &tmK, b * 64, head, tok_begin + key_tile(j) * kKeys, kf(st));
        k_issued = j + 1;
      }
      if (!ok) s_abort = 1;
    }
    if (lane == 0 && warp == kVWarp) {
      ptx::prefetch_tmap(&tmV);
      ptx::prefetch_tmap(&tmL);
      const uint32_t bytes = kVBytes + p.n_lbox * kLBoxBytes;
      for (int v = 0; ok && v < 2 * n; ++v) {
        const int st = v % p.nv;
        if (v >= p.nv && !wait_ab(ve(st), ((v / p.nv) - 1) & 1, &s_abort)) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(vf(st), bytes);
        const uint32_t dst = ptx::smem_u32(vl_s + st * p.vl_bytes);
        const int tok = tok_begin + key_tile(v >> 1) * kKeys + (v & 1) * kHalf;
#pragma unroll
        for (int b = 0; b < D / 64; ++b) ptx::tma_load_3d(dst + b * kLBoxBytes, &tmV, b * 64, head, tok, vf(st));
        for (int b = 0; b < p.n_lbox; ++b) ptx::tma_load_2d(dst + kVBytes + b * kLBoxBytes, &tmL, b * 64, tok, vf(st));
        v_issued = v + 1;
      }
      if (!ok) s_abort = 1;
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (s_abort && lane == 0) {
      for (int j = max(0, k_issued - p.nk); j < k_issued; ++j) ptx::mbar_wait(kf(j % p.nk), (j / p.nk) & 1);
      for (int v = max(0, v_issued - p.nv); v < v_issued; ++v) ptx::mbar_wait(vf(v % p.nv), (v / p.nv) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    bool issued_any = false;
    if (lane == 0) {
      const uint32_t idesc_s = ptx::idesc_bf16_f32(kKeys, kN);                           // K, Q: K-major
      const uint32_t idesc_v = ptx::idesc_bf16_f32(kKeys, kN) | (1u << 15) | (1u << 16);  // V/L and P: MN-major
      uint32_t idesc_ol[kMaxLChunks];
#pragma unroll
      for (int c = 0; c < kMaxLChunks; ++c)
        idesc_ol[c] = ptx::idesc_bf16_f32(kKeys, c < p.n_lchunk ? p.ol_rows[c] : 16) | (1u << 15) | (1u << 16);
      const uint64_t d_q = ptx::smem_desc_k128(ptx::smem_u32(q_s));
      const uint64_t d_k = ptx::smem_desc_k128(ptx::smem_u32(k_s));
      const uint64_t d_p = ptx::smem_desc_mn128(ptx::smem_u32(p_s), 8192);
      const uint64_t d_vl = ptx::smem_desc_mn128(ptx::smem_u32(vl_s), kLBoxBytes);
      auto issue_s = [&](int j) -> bool {
        const int st = j % p.nk, b = j & 1;
        if (!wait_ab(kf(st), (j / p.nk) & 1, &s_abort)) return false;
        if (j >= 2 && !wait_ab(sfree(b), ((j >> 1) - 1) & 1, &s_abort)) return false;
        ptx::tc_fence_after();
        const uint64_t dk = ptx::desc_advance(d_k, st * kKBytes);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t col = (ks & 3) * 32;
          ptx::tc_mma_f16(tmem + (b ? kColS1 : kColS0), ptx::desc_advance(dk, (ks >> 2) * (kKeys * 128) + col),
                          ptx::desc_advance(d_q, (ks >> 2) * (kN * 128) + col), idesc_s, ks > 0 ? 1u : 0u);
        }
        issued_any = true;
        ptx::tc_commit(ke(st));
        ptx::tc_commit(sfull(b));
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        if (!wait_ab(pfull, j & 1, &s_abort)) return false;
        for (int h = 0; h < 2; ++h) {
          const int v = 2 * j + h, st = v % p.nv;
          if (!wait_ab(vf(st), (v / p.nv) & 1, &s_abort)) return false;
          ptx::tc_fence_after();
          const uint64_t dv = ptx::desc_advance(d_vl, st * p.vl_bytes);
          const uint64_t dl = ptx::desc_advance(dv, kVBytes);
#pragma unroll
          for (int ks = 0; ks < kHalf / 16; ++ks) {
            const uint32_t acc = (j > 0 || h > 0 || ks > 0) ? 1u : 0u;
            const uint64_t bP = ptx::desc_advance(d_p, (h * kHalf + ks * 16) * 128);
            ptx::tc_mma_f16(tmem + kColO, ptx::desc_advance(dv, ks * 2048), bP, idesc_v, acc);
#pragma unroll
            for (int c = 0; c < kMaxLChunks; ++c)
              if (c < p.n_lchunk)  // P^T from the chunk's first query row: 2 bytes a row within each key's 128
                ptx::tc_mma_f16(tmem + kColOL + p.ol_col[c], ptx::desc_advance(dl, c * 2 * kLBoxBytes + ks * 2048),
                                ptx::desc_advance(bP, p.ol_row0[c] * 2), idesc_ol[c], acc);
          }
          ptx::tc_commit(ve(st));
        }
        ptx::tc_commit(pvdone);
        return true;
      };
      if (n > 0) ok = issue_s(0);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) ok = issue_s(j + 1);
        if (ok) ok = issue_pv(j);
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
    // ------------------------------------------------------------ softmax + partial record
    const int q = warp & 3;
    const int key = q * 32 + lane;  // this thread's TMEM lane: key of S^T, d of O^T, L column of OL^T
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const float sl2 = p.scale_log2;
    // running max per query row (log2 domain): s_m[n_resc & 1], rewritten only
    // on a rescale, into the other buffer (read by every thread, written by key 0)
    int n_resc = 0;
    for (int j = 0; ok && j < n; ++j) {
      const int b = j & 1;
      const float *m_cur = s_m[n_resc & 1];
      if (!__all_sync(0xffffffffu, wait_ab(sfull(b), (j >> 1) & 1, &s_abort))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t sv[kN];
      ptx::tmem_ld32(tmem + lane_base + (b ? kColS1 : kColS0), *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      ptx::tmem_ld32(tmem + lane_base + (b ? kColS1 : kColS0) + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      ptx::tmem_ld_wait();
      ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sfree(b));
      const bool key_ok = key_tile(j) * kKeys + key < n_tok;
      // P with the running max, speculatively: a row whose max rose by more
      // than 2^8 (every row on the first tile) flags a rescale
      uint32_t pk[kN / 2];
      bool flag = false;
#pragma unroll
      for (int i = 0; i < kN / 2; ++i) {
        const float2 m2 = *reinterpret_cast<const float2 *>(m_cur + 2 * i);
        const float x0 = key_ok ? fmaf(__uint_as_float(sv[2 * i]), sl2, -m2.x) : -INFINITY;
        const float x1 = key_ok ? fmaf(__uint_as_float(sv[2 * i + 1]), sl2, -m2.y) : -INFINITY;
        flag |= (x0 > kRescaleLog2) | (x1 > kRescaleLog2);
        pk[i] = ptx::pack_bf16(ptx::ex2(x0), ptx::ex2(x1));
      }
      {
        const int any = __any_sync(0xffffffffu, flag) ? 1 : 0;
        if (lane == 0) {
          s_vote[b][q] = any;
          ptx::mbar_arrive(vote);
        }
        if (!__all_sync(0xffffffffu, wait_ab(vote, j & 1, &s_abort))) {
          ok = false;
          break;
        }
      }
      bool waited = false;
      if (s_vote[b][0] | s_vote[b][1] | s_vote[b][2] | s_vote[b][3]) {
        // row maxima of this tile over all 128 keys
        const int rb = n_resc & 1;
#pragma unroll
        for (int c = 0; c < kN; ++c) {
          float v = key_ok ? __uint_as_float(sv[c]) : -INFINITY;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
          if (lane == 0) s_red[q][c] = v;
        }
        if (lane == 0) ptx::mbar_arrive(red);
        if (!__all_sync(0xffffffffu, wait_ab(red, rb, &s_abort))) {  // phase = rescale count parity
          ok = false;
          break;
        }
        // new running max: raised only where this tile's max exceeds it by 2^8
        auto m_new = [&](int c) {
          const float tm =
              fmaxf(fmaxf(s_red[0][c], s_red[1][c]), fmaxf(s_red[2][c], s_red[3][c])) * sl2;
          return (c < p.rows && tm > m_cur[c] + kRescaleLog2) ? tm : m_cur[c];
        };
        float f[kN];
#pragma unroll
        for (int c = 0; c < kN; ++c) {
          const float mn = m_new(c);
          f[c] = (m_cur[c] == -INFINITY) ? 0.f : ptx::ex2(m_cur[c] - mn);
          if (key == 0) s_m[rb ^ 1][c] = mn;
        }
        if (j > 0) {
          // O^T, l and OL^T hold PV_0..PV_{j-1}: rescale their columns once PV_{j-1} is done
          if (!__all_sync(0xffffffffu, wait_ab(pvdone, (j - 1) & 1, &s_abort))) {
            ok = false;
            break;
          }
          waited = true;
          ptx::tc_fence_after();
          for (int reg = 0; reg < 2; ++reg) {
            const uint32_t col = reg == 0 ? kColO : kColLs;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t ov[32];
              ptx::tmem_ld32(tmem + lane_base + col + hh * 32, ov);
              ptx::tmem_ld_wait();
              ptx::reg_fence32(ov);
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f[hh * 32 + i]);
              ptx::tmem_st32(tmem + lane_base + col + hh * 32, ov);
            }
          }
          // OL^T chunks: column i of chunk c holds row ol_row0[c] + i; chunks
          // are scaled one after another (a 32-column load may reach into the
          // next chunk, whose values are written back unchanged first)
          for (int c = 0; c < p.n_lchunk; ++c) {
            const int r0 = p.ol_row0[c], nr = p.ol_rows[c];
            for (int hh = 0; hh * 32 < nr; ++hh) {
              uint32_t ov[32];
              ptx::tmem_st_wait();
              ptx::tmem_ld32(tmem + lane_base + kColOL + p.ol_col[c] + hh * 32, ov);
              ptx::tmem_ld_wait();
              ptx::reg_fence32(ov);
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int row = r0 + hh * 32 + i;
                if (hh * 32 + i < nr) {
                  const float mc = m_cur[row];
                  const float fr = (mc == -INFINITY) ? 0.f : ptx::ex2(mc - m_new(row));
                  ov[i] = __float_as_uint(__uint_as_float(ov[i]) * fr);
                }
              }
              ptx::tmem_st32(tmem + lane_base + kColOL + p.ol_col[c] + hh * 32, ov);
            }
          }
          ptx::tmem_st_wait();
        }
#pragma unroll
        for (int i = 0; i < kN / 2; ++i) {
          const float x0 = key_ok ? fmaf(__uint_as_float(sv[2 * i]), sl2, -m_new(2 * i)) : -INFINITY;
          const float x1 = key_ok ? fmaf(__uint_as_float(sv[2 * i + 1]), sl2, -m_new(2 * i + 1)) : -INFINITY;
          pk[i] = ptx::pack_bf16(ptx::ex2(x0), ptx::ex2(x1));
        }
        ++n_resc;  // the other buffer is current from the next tile on (published by the next vote)
      }
      if (j > 0 && !waited) {
        // the P buffer is free once PV_{j-1} has finished reading it
        if (!__all_sync(0xffffffffu, wait_ab(pvdone, (j - 1) & 1, &s_abort))) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
      }
      // P^T row of this key: 64 query rows, MN-major 128-byte swizzle
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4 *>(p_s + key * 128 + ((c ^ (key & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(pfull);
      // row sums of this key's lane: the same bf16 P values the MMAs use
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t lv[32];
        if (j > 0) {
          ptx::tmem_ld32(tmem + lane_base + kColLs + hh * 32, lv);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(lv);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t w = pk[hh * 16 + i];
          const float p0 = __uint_as_float(w << 16), p1 = __uint_as_float(w & 0xFFFF0000u);
          lv[2 * i] = __float_as_uint(j > 0 ? __uint_as_float(lv[2 * i]) + p0 : p0);
          lv[2 * i + 1] = __float_as_uint(j > 0 ? __uint_as_float(lv[2 * i + 1]) + p1 : p1);
        }
        ptx::tmem_st32(tmem + lane_base + kColLs + hh * 32, lv);
      }
      ptx::tmem_st_wait();
    }
    // ---- partial record: [rows][d + r] (O | own agent's OL) | m[rows] | l[rows]
    if (ok && n > 0) ok = __all_sync(0xffffffffu, wait_ab(pvdone, (n - 1) & 1, &s_abort));
    // row sums: reduce-scatter each warp's 32 lanes (lane L ends with rows 2L,
    // 2L+1), then add the four warps' shares through the P buffer, which the
    // completed last P.V MMAs no longer read.  Every softmax warp reaches the
    // named barrier once, whatever its ok.
    float *lred = reinterpret_cast<float *>(p_s);  // [4 warps][64 rows]
    if (ok && n > 0) {
      uint32_t lw[kN];
      ptx::tmem_ld32(tmem + lane_base + kColLs, *reinterpret_cast<uint32_t(*)[32]>(&lw[0]));
      ptx::tmem_ld32(tmem + lane_base + kColLs + 32, *reinterpret_cast<uint32_t(*)[32]>(&lw[32]));
      ptx::tmem_ld_wait();
      ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&lw[0]));
      ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&lw[32]));
      float lv[kN];
#pragma unroll
      for (int c = 0; c < kN; ++c) lv[c] = __uint_as_float(lw[c]);
#pragma unroll
      for (int o = 16, nh = kN / 2; o >= 1; o >>= 1, nh >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < nh; ++i) {
          const float send = upper ? lv[i] : lv[i + nh];
          const float keep = upper ? lv[i + nh] : lv[i];
          lv[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      lred[q * kN + 2 * lane] = lv[0];
      lred[q * kN + 2 * lane + 1] = lv[1];
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (unit == 0 && key == 0) p.pair_info[qreq * p.hkv + head] = make_int2(slot - unit, n_units);
    if (ok) {
      const int W = D + p.r;
      float *part = p.partials + ((int64_t)slot * p.hkv + head) * p.part_stride;
      if (n > 0) {
        ptx::tc_fence_after();
        uint32_t ov[kN];
        ptx::tmem_ld32(tmem + lane_base + kColO, *reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
        ptx::tmem_ld32(tmem + lane_base + kColO + 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
        ptx::tmem_ld_wait();
        ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
        ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
#pragma unroll
        for (int c = 0; c < kN; ++c)
          if (c < p.rows) part[c * W + key] = __uint_as_float(ov[c]);
        for (int ch = 0; ch < p.n_lchunk; ++ch) {
          // columns kColOL + ol_col[ch] + i hold rows ol_row0[ch] + i (the
          // loads may reach into the next chunk, whose columns are not used here)
          ptx::tmem_ld32(tmem + lane_base + kColOL + p.ol_col[ch], *reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
          ptx::tmem_ld32(tmem + lane_base + kColOL + p.ol_col[ch] + 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
          ptx::tmem_ld_wait();
          ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
          ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
          const int col = ch * kKeys + key;  // L column held by this lane
          const int r0 = p.ol_row0[ch], nr = p.ol_rows[ch];
          if (col < p.l_width) {
#pragma unroll
            for (int i = 0; i < kN; ++i) {
              const int c = r0 + i;
              if (i >= nr || c >= p.rows) break;
              const int lo = (c / p.G) * p.l_agent_stride;
              if (col >= lo && col < lo + p.r) part[c * W + D + col - lo] = __uint_as_float(ov[i]);
            }
          }
        }
        if (key < p.rows) {
          part[p.rows * W + key] = s_m[n_resc & 1][key];
          part[p.rows * W + p.rows + key] = (lred[key] + lred[kN + key]) + (lred[2 * kN + key] + lred[3 * kN + key]);
        }
      } else {
        // empty unit (an empty request): zero accumulators, m = -inf, l = 0
        for (int e = key; e < p.rows * W; e += kKeys) part[e] = 0.f;
        for (int c = key; c < p.rows; c += kKeys) {
          part[p.rows * W + c] = -INFINITY;
          part[p.rows * W + p.rows + c] = 0.f;
        }
      }
    }
    if (!ok) s_abort = 1;
    ptx::tc_fence_before();
    __syncthreads();
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace dt5

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct DecodeT5Plan {
  int rows, l_width, n_lbox, n_lchunk, nk, nv, vl_bytes, smem_bytes, part_stride;
  int ol_row0[dt5::kMaxLChunks], ol_rows[dt5::kMaxLChunks], ol_col[dt5::kMaxLChunks];
  bool ok;
};

inline DecodeT5Plan decode_t5_plan(const fla_attn_dims &d) {
  DecodeT5Plan pl{};
  pl.ok = false;
  if (d.dtype != FLA_BF16 || d.head_dim != dt5::D) return pl;
  if (d.rank > 64) return pl;  // the merge kernel holds up to 64 LoRA columns per row
  if (d.l_agent_stride != 0 && d.l_agent_stride != d.rank) return pl;
  const int G = d.hq / d.hkv, rows = d.n_agents * G;
  if (rows > dt5::kN) return pl;
  const int l_width = d.l_agent_stride == 0 ? d.rank : d.n_agents * d.rank;
  const int n_lbox = (l_width + 63) / 64;
  const int n_lchunk = (n_lbox + 1) / 2;
  if (n_lchunk > dt5::kMaxLChunks) return pl;
  // a stage holds V and the n_lbox loaded L boxes; when n_lbox is odd the
  // last chunk's MMA also reads one box past the stage (rows of OL^T that are
  // never used), so the ring gets one spare box at its end
  const int vl_bytes = dt5::kVBytes + n_lbox * dt5::kLBoxBytes;
  const int spare = (n_lbox & 1) ? dt5::kLBoxBytes : 0;
  const int budget = 227 * 1024 - 1024 /* alignment */ - 3072 /* static shared */;
  const int fixed = dt5::kQBytes + dt5::kPBytes;
  int nk = 2, nv = (budget - fixed - nk * dt5::kKBytes - spare) / vl_bytes;
  if (nv > 6) nv = 6;
  if (nv < 2) return pl;
  if (nv >= 5 && fixed + 3 * dt5::kKBytes + (nv - 1) * vl_bytes + spare <= budget) {
    nk = 3;
    nv -= 1;
  }
  // OL^T chunk c (L columns [128c, 128c + 128)) only needs the query rows of
  // the agents whose blocks it holds: rows [a_lo*G, (a_hi+1)*G), widened to a
  // start on a multiple of 8 rows (16-byte operand offset) and a multiple of
  // 16 rows (the MMA's N), inside the 64 rows of P^T
  int col = 0;
  for (int c = 0; c < n_lchunk; ++c) {
    int lo_row = 0, hi_row = rows;
    if (d.l_agent_stride != 0) {
      const int a_lo = (c * dt5::kKeys) / d.rank;
      const int a_hi = std::min(d.n_agents - 1, (c * dt5::kKeys + dt5::kKeys - 1) / d.rank);
      lo_row = a_lo * G;
      hi_row = std::min(rows, (a_hi + 1) * G);
    }
    int r0 = lo_row / 8 * 8;
    int nr = (hi_row - r0 + 15) / 16 * 16;
    if (nr < 16) nr = 16;
    if (r0 + nr > dt5::kN) r0 = dt5::kN - nr;  // still covers [lo_row, hi_row)
    pl.ol_row0[c] = r0;
    pl.ol_rows[c] = nr;
    pl.ol_col[c] = col;
    col += nr;
  }
  pl.rows = rows; pl.l_width = l_width; pl.n_lbox = n_lbox; pl.n_lchunk = n_lchunk;
  pl.nk = nk; pl.nv = nv; pl.vl_bytes = vl_bytes;
  pl.smem_bytes = fixed + nk * dt5::kKBytes + nv * vl_bytes + spare + 1024;
  pl.part_stride = (rows * (dt5::D + d.rank + 2) + 3) & ~3;
  pl.ok = true;
  return pl;
}

inline bool decode_t5_shape_supported(const fla_attn_dims &d) { return decode_t5_plan(d).ok; }

inline int64_t decode_t5_unit_tokens(int n_req, int64_t total_tokens, int hkv) {
  const int64_t U = decode_unit_tokens(n_req, std::max<int64_t>(total_tokens, 1), hkv);
  return (U + dt5::kKeys - 1) / dt5::kKeys * dt5::kKeys;
}

inline size_t decode_t5_workspace_bytes(const fla_attn_dims &d, int n_req, int64_t total_tokens) {
  const DecodeT5Plan pl = decode_t5_plan(d);
  if (!pl.ok || n_req <= 0) return 0;
  const int64_t U = decode_t5_unit_tokens(n_req, total_tokens, d.hkv);
  const int64_t units = decode_max_units(n_req, total_tokens, U);
  const size_t info = ((size_t)n_req * d.hkv * sizeof(int2) + 255) / 256 * 256;
  return info + (size_t)units * d.hkv * pl.part_stride * 4;
}

inline fla_status decode_t5_launch(const fla_attn_dims &d, float scale, const void *Q, const void *K, const void *V,
                                   const void *L, const void *B, const int32_t *offsets, int n_req,
                                   int64_t total_tokens, float *O, void *workspace, cudaStream_t s) {
  const DecodeT5Plan pl = decode_t5_plan(d);
  if (!pl.ok) {
    decode_tc_err() = "shape outside the tcgen05 decode kernel";
    return FLA_ERR_UNSUPPORTED;
  }
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) {
    decode_tc_err() = "cuTensorMapEncodeTiled is not available from the driver";
    return FLA_ERR_CUDA;
  }
  const int64_t U = decode_t5_unit_tokens(n_req, total_tokens, d.hkv);
  const int64_t units = decode_max_units(n_req, total_tokens, U);
  const int64_t n_rows = std::max<int64_t>(total_tokens, 1);
  CUtensorMap mK, mV, mL;
  const cuuint32_t es[3] = {1, 1, 1};
  {
    const cuuint64_t dims[3] = {(cuuint64_t)dt5::D, (cuuint64_t)d.hkv, (cuuint64_t)n_rows};
    const cuuint64_t strides[2] = {(cuuint64_t)dt5::D * 2, (cuuint64_t)d.hkv * dt5::D * 2};
    const cuuint32_t box_k[3] = {64, 1, (cuuint32_t)dt5::kKeys};
    const cuuint32_t box_v[3] = {64, 1, (cuuint32_t)dt5::kHalf};
    if (enc(&mK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(K), dims, strides, box_k, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&mV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(V), dims, strides, box_v, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      decode_tc_err() = "encoding the K/V tensor maps failed";
      return FLA_ERR_CUDA;
    }
  }
  {
    // 64-column boxes; columns past l_width read as zeros
    const cuuint64_t dims[2] = {(cuuint64_t)pl.l_width, (cuuint64_t)n_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)d.l_row_stride * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)dt5::kHalf};
    if (enc(&mL, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(L), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      decode_tc_err() = "encoding the L tensor map failed";
      return FLA_ERR_CUDA;
    }
  }
  dt5::Params prm{};
  prm.Q = reinterpret_cast<const __nv_bfloat16 *>(Q);
  prm.offsets = offsets;
  const size_t info = ((size_t)n_req * d.hkv * sizeof(int2) + 255) / 256 * 256;
  prm.pair_info = reinterpret_cast<int2 *>(workspace);
  prm.partials = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + info);
  prm.n_req = n_req; prm.A = d.n_agents; prm.hq = d.hq; prm.hkv = d.hkv; prm.G = d.hq / d.hkv;
  prm.r = d.rank; prm.rows = pl.rows;
  prm.l_agent_stride = (int)d.l_agent_stride; prm.l_width = pl.l_width;
  prm.n_lbox = pl.n_lbox; prm.n_lchunk = pl.n_lchunk;
  prm.unit_tokens = (int)U;
  prm.single_len = n_req == 1 ? (int)total_tokens : -1;
  prm.part_stride = pl.part_stride;
  prm.nk = pl.nk; prm.nv = pl.nv; prm.vl_bytes = pl.vl_bytes;
  for (int c = 0; c < dt5::kMaxLChunks; ++c) {
    prm.ol_row0[c] = c < pl.n_lchunk ? pl.ol_row0[c] : 0;
    prm.ol_rows[c] = c < pl.n_lchunk ? pl.ol_rows[c] : 16;
    prm.ol_col[c] = c < pl.n_lchunk ? pl.ol_col[c] : 0;
  }
  prm.scale_log2 = scale * 1.4426950408889634f;
  const int64_t grid64 = units * d.hkv;
  if (grid64 > 0x7fffffffLL) {
    decode_tc_err() = "too many work units";
    return FLA_ERR_UNSUPPORTED;
  }
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(dt5::decode_t5_kernel), pl.smem_bytes);
  if (e != cudaSuccess) {
    decode_tc_err() = cudaGetErrorString(e);
    return FLA_ERR_CUDA;
  }
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid64);
    cfg.blockDim = dim3(dt5::kThreads);
    cfg.dynamicSmemBytes = pl.smem_bytes;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, dt5::decode_t5_kernel, mK, mV, mL, prm);
    if (e != cudaSuccess) {
      decode_tc_err() = cudaGetErrorString(e);
      return FLA_ERR_CUDA;
    }
  }
  // every pair (even a single-unit one) is finished by the merge kernel
  dec::MergeParams mp{};
  mp.partials = prm.partials;
  mp.pair_info = prm.pair_info;
  mp.B = reinterpret_cast<const __nv_bfloat16 *>(B);
  mp.O = O;
  mp.n_req = n_req; mp.A = d.n_agents; mp.hq = d.hq; mp.hkv = d.hkv; mp.G = prm.G; mp.rows = pl.rows;
  mp.r = d.rank;
  mp.part_stride = pl.part_stride; mp.unit_tokens = (int)U; mp.single_len = prm.single_len;
  mp.merge_single = 1;
  e = launch_merge<dt5::D>(mp, decode_units_bound(total_tokens, U), true, s);
  if (e != cudaSuccess) {
    decode_tc_err() = cudaGetErrorString(e);
    return FLA_ERR_CUDA;
  }
  return FLA_OK;
}

}  // namespace fla
