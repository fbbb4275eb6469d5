// Host side of the C ABI declared in include/flash_lora_attn.h.
//
// Validation happens here, before anything is enqueued; each entry point then
// picks a kernel family (tensor-core or SIMT) and launches on the caller's
// stream.  The library allocates no memory and keeps no per-call state.
//
// Unity build: every kernel family is a header included below, so the whole
// library is one translation unit with one device error word.
#include <algorithm>
#include <cmath>
#include <mutex>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/flash_lora_attn.h"
#include "fla_common.cuh"
#include "simt_kernels.cuh"
#include "decode_tc.cuh"
#include "decode_t5.cuh"
#include "build_tc.cuh"
#include "prefill_mma.cuh"
#include "prefill_tc.cuh"
#include "expand.cuh"

namespace {

thread_local std::string g_last_error;

fla_status fail(fla_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

fla_status ok() { return FLA_OK; }

fla_status check_launch(const char *what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FLA_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return FLA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


// Checks shared by decode and prefill.  Fills `scale`.
fla_status check_dims(const fla_attn_dims *d, float *scale) {
  if (!d) return fail(FLA_ERR_INVALID_ARG, "dims is NULL");
  if (d->n_agents < 1) return fail(FLA_ERR_INVALID_ARG, "n_agents must be >= 1 (got %d)", d->n_agents);
  if (d->hq < 1 || d->hkv < 1) return fail(FLA_ERR_INVALID_ARG, "hq and hkv must be >= 1");
  if (d->hq % d->hkv != 0)
    return fail(FLA_ERR_INVALID_ARG, "hq (%d) must be a multiple of hkv (%d)", d->hq, d->hkv);
  if (d->head_dim < 1 || d->head_dim > fla::kSimtMaxD || d->head_dim % 4 != 0)
    return fail(FLA_ERR_UNSUPPORTED, "head_dim %d: must be a multiple of 4 in [4, 256]", d->head_dim);
  if (d->rank < 1 || d->rank > fla::kSimtMaxR)
    return fail(FLA_ERR_UNSUPPORTED, "rank %d: must be in [1, 256]", d->rank);
  if (d->dtype != FLA_F32 && d->dtype != FLA_BF16)
    return fail(FLA_ERR_INVALID_ARG, "dtype %d is not FLA_F32 or FLA_BF16", d->dtype);
  if (d->kernel < FLA_KERNEL_AUTO || d->kernel > FLA_KERNEL_TCGEN05)
    return fail(FLA_ERR_INVALID_ARG, "kernel %d is not a fla_kernel", d->kernel);
  if (d->l_agent_stride < 0) return fail(FLA_ERR_INVALID_ARG, "l_agent_stride must be >= 0");
  const int64_t need = (int64_t)(d->n_agents - 1) * d->l_agent_stride + d->rank;
  if (d->l_row_stride < need)
    return fail(FLA_ERR_INVALID_ARG, "l_row_stride %lld is smaller than the %lld columns the agents read",
                (long long)d->l_row_stride, (long long)need);
  if (d->l_agent_stride != 0 && d->l_agent_stride < d->rank)
    return fail(FLA_ERR_INVALID_ARG, "l_agent_stride must be 0 (shared LR cache) or >= rank");
  *scale = d->softmax_scale > 0.f ? d->softmax_scale : 1.0f / std::sqrt((float)d->head_dim);
  return FLA_OK;
}

// out = X . W over the column segments seg[0..n_seg) of W (row-major, the
// segments' columns side by side): the tcgen05 GEMM reads each tile of X once
// for every segment; the CUDA-core fallback runs one launch per segment.
fla_status run_projection(const char *what, const void *X, int64_t ldx, const void *W, const fla::BuildSegment *seg,
                          int n_seg, int64_t n_tokens, int32_t d_model, int32_t dtype, int32_t kernel,
                          cudaStream_t s) {
  if (kernel == FLA_KERNEL_MMA_SYNC)
    return fail(FLA_ERR_UNSUPPORTED, "%s has no mma.sync kernel (use TENSOR or TCGEN05)", what);
  const bool tc_ok = fla::build_tc_supported(X, ldx, W, seg, n_seg, d_model, dtype);
  if ((kernel == FLA_KERNEL_TENSOR || kernel == FLA_KERNEL_TCGEN05) && !tc_ok)
    return fail(FLA_ERR_UNSUPPORTED, "%s: shape/alignment outside the tensor-core kernel (needs bf16, "
                "d_model %% 64 == 0, every output width %% 32 == 0, 16-byte alignment, row strides multiples of 8)",
                what);
  if (tc_ok && kernel != FLA_KERNEL_SIMT) {
    const fla_status st = fla::build_tc_launch(X, ldx, W, seg, n_seg, n_tokens, d_model, s);
    if (st != FLA_OK) return fail(st, "%s (tensor): %s", what, fla::build_tc_last_error());
    return check_launch(what);
  }
  int64_t lda = 0;
  for (int i = 0; i < n_seg; ++i) lda += seg[i].cols;
  const size_t esize = dtype == FLA_F32 ? 4 : 2;
  int64_t col = 0;
  for (int i = 0; i < n_seg; ++i) {
    fla::SimtBuildParams p{X, static_cast<const uint8_t *>(W) + col * esize, seg[i].ptr, ldx, seg[i].ld,
                           n_tokens, d_model, seg[i].cols, lda};
    col += seg[i].cols;
    if ((n_tokens + 63) / 64 > 0x7fffffffLL || (seg[i].cols + 63) / 64 > 65535)
      return fail(FLA_ERR_UNSUPPORTED, "%s: n_tokens or the output width too large", what);
    dim3 grid((unsigned)((n_tokens + 63) / 64), (unsigned)((seg[i].cols + 63) / 64));
    if (dtype == FLA_F32)
      fla::simt_build_kernel<float><<<grid, 256, 0, s>>>(p);
    else
      fla::simt_build_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(p);
  }
  return check_launch(what);
}

template <typename T>
void launch_simt_attn(const fla::SimtAttnParams &p, int64_t rows, cudaStream_t s) {
  fla::simt_attn_kernel<T><<<(unsigned)rows, fla::kSimtWarps * 32, 0, s>>>(p);
}

// The bounded-wait path every pipeline kernel relies on, run on purpose:
// warp 0 waits on an mbarrier no one arrives on, with a limit of limit_ns; on
// timeout the helper records kErrSelfTestWait and raises the CTA's abort flag.
// Warp 1 waits on a second such barrier with the kernels' 2 s limit and must
// leave through the abort flag instead.  out[0] = 1 if warp 0's wait ran out,
// out[1] = 1 if warp 1 left on the abort flag, out[2] = warp 0's wait in ns.
__global__ void selftest_bounded_wait_kernel(uint64_t limit_ns, unsigned long long *out) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ volatile int s_abort;
  const uint32_t b0 = fla::ptx::smem_u32(&bars[0]), b1 = fla::ptx::smem_u32(&bars[1]);
  if (threadIdx.x == 0) {
    s_abort = 0;
    fla::ptx::mbar_init(b0, 1);
    fla::ptx::mbar_init(b1, 1);
    fla::ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = fla::globaltimer_ns();
    const bool ok = fla::ptx::mbar_wait_or_abort(b0, 0, &s_abort, fla::kErrSelfTestWait, limit_ns);
    out[0] = ok ? 0ull : 1ull;
    out[2] = fla::globaltimer_ns() - t0;
  } else if (threadIdx.x == 32) {
    const bool ok = fla::ptx::mbar_wait_or_abort(b1, 0, &s_abort, fla::kErrSelfTestWait);
    out[1] = (!ok && s_abort) ? 1ull : 0ull;
  }
}

}  // namespace

extern "C" {

const char *fla_version(void) { return "0.1.0"; }

const char *fla_status_string(fla_status s) {
  switch (s) {
    case FLA_OK: return "FLA_OK";
    case FLA_ERR_INVALID_ARG: return "FLA_ERR_INVALID_ARG";
    case FLA_ERR_UNSUPPORTED: return "FLA_ERR_UNSUPPORTED";
    case FLA_ERR_WORKSPACE: return "FLA_ERR_WORKSPACE";
    case FLA_ERR_CUDA: return "FLA_ERR_CUDA";
    case FLA_ERR_DEVICE_TIMEOUT: return "FLA_ERR_DEVICE_TIMEOUT";
  }
  return "FLA_ERR_UNKNOWN";
}

const char *fla_last_error(void) { return g_last_error.c_str(); }

fla_status fla_selftest_bounded_wait(uint64_t limit_ns, unsigned long long *out, fla_stream_t stream) {
  g_last_error.clear();
  if (!out) return fail(FLA_ERR_INVALID_ARG, "out is NULL");
  if (limit_ns == 0 || limit_ns > fla::kWaitLimitNs)
    return fail(FLA_ERR_INVALID_ARG, "limit_ns must be in (0, %llu]", (unsigned long long)fla::kWaitLimitNs);
  selftest_bounded_wait_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, out);
  return check_launch("fla_selftest_bounded_wait");
}

fla_status fla_device_error(uint32_t *code) {
  if (!code) return fail(FLA_ERR_INVALID_ARG, "code is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(FLA_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
  uint32_t v = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&v, fla::g_device_error, sizeof(v));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(fla::g_device_error, &zero, sizeof(zero));
  if (e != cudaSuccess) return fail(FLA_ERR_CUDA, "reading the device error word: %s", cudaGetErrorString(e));
  *code = v;
  return FLA_OK;
}

// ---------------------------------------------------------------------------
fla_status lr_cache_build(const void *X, int64_t ldx, const void *A_cat, void *L, int64_t ldl,
                          int64_t n_tokens, int32_t d_model, int32_t n_agents, int32_t rank, int32_t dtype,
                          int32_t kernel, fla_stream_t stream) {
  g_last_error.clear();
  if (n_tokens < 0 || d_model < 1 || n_agents < 1 || rank < 1)
    return fail(FLA_ERR_INVALID_ARG, "n_tokens must be >= 0; d_model, n_agents and rank >= 1");
  const int64_t n_cols64 = (int64_t)n_agents * rank;
  if (n_cols64 > INT32_MAX) return fail(FLA_ERR_INVALID_ARG, "n_agents * rank overflows int32");
  const int32_t n_cols = (int32_t)n_cols64;
  if (dtype != FLA_F32 && dtype != FLA_BF16) return fail(FLA_ERR_INVALID_ARG, "bad dtype %d", dtype);
  if (kernel < FLA_KERNEL_AUTO || kernel > FLA_KERNEL_TCGEN05)
    return fail(FLA_ERR_INVALID_ARG, "kernel %d is not a fla_kernel", kernel);
  if (ldx < d_model) return fail(FLA_ERR_INVALID_ARG, "ldx (%lld) < d_model (%d)", (long long)ldx, d_model);
  if (ldl < n_cols)
    return fail(FLA_ERR_INVALID_ARG, "ldl (%lld) < n_agents * rank (%d)", (long long)ldl, n_cols);
  if (n_tokens == 0) return ok();
  if (!X || !A_cat || !L) return fail(FLA_ERR_INVALID_ARG, "X, A_cat and L must be non-NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  const fla::BuildSegment seg{L, ldl, n_cols};
  return run_projection("lr_cache_build", X, ldx, A_cat, &seg, 1, n_tokens, d_model, dtype, kernel, s);
}

// ---------------------------------------------------------------------------
fla_status rebase_kv_lr_build(const void *X, int64_t ldx, const void *W_cat, void *K_base, void *V_base, void *L,
                              int64_t ldl, int64_t n_tokens, int32_t d_model, int32_t hkv, int32_t head_dim,
                              int32_t n_agents, int32_t rank, int32_t dtype, int32_t kernel, fla_stream_t stream) {
  g_last_error.clear();
  if (n_tokens < 0 || d_model < 1 || hkv < 1 || head_dim < 1 || n_agents < 1 || rank < 1)
    return fail(FLA_ERR_INVALID_ARG, "n_tokens must be >= 0; d_model, hkv, head_dim, n_agents and rank >= 1");
  const int64_t kv64 = (int64_t)hkv * head_dim, lr64 = (int64_t)n_agents * rank;
  if (2 * kv64 + lr64 > INT32_MAX) return fail(FLA_ERR_INVALID_ARG, "the projection width overflows int32");
  if (dtype != FLA_F32 && dtype != FLA_BF16) return fail(FLA_ERR_INVALID_ARG, "bad dtype %d", dtype);
  if (kernel < FLA_KERNEL_AUTO || kernel > FLA_KERNEL_TCGEN05)
    return fail(FLA_ERR_INVALID_ARG, "kernel %d is not a fla_kernel", kernel);
  if (ldx < d_model) return fail(FLA_ERR_INVALID_ARG, "ldx (%lld) < d_model (%d)", (long long)ldx, d_model);
  if (ldl < lr64)
    return fail(FLA_ERR_INVALID_ARG, "ldl (%lld) < n_agents * rank (%lld)", (long long)ldl, (long long)lr64);
  if (n_tokens == 0) return ok();
  if (!X || !W_cat || !K_base || !V_base || !L)
    return fail(FLA_ERR_INVALID_ARG, "X, W_cat, K_base, V_base and L must be non-NULL");
  const fla::BuildSegment seg[3] = {{K_base, kv64, (int32_t)kv64}, {V_base, kv64, (int32_t)kv64},
                                    {L, ldl, (int32_t)lr64}};
  return run_projection("rebase_kv_lr_build", X, ldx, W_cat, seg, 3, n_tokens, d_model, dtype, kernel,
                        reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
size_t flash_lora_attn_decode_workspace_size(const fla_attn_dims *dims, int32_t n_req,
                                             int64_t total_tokens) {
  float scale = 0.f;
  if (check_dims(dims, &scale) != FLA_OK || n_req < 0 || total_tokens < 0) return 0;
  if (dims->kernel == FLA_KERNEL_SIMT) return 0;
  size_t need = 0;
  if (dims->kernel != FLA_KERNEL_TCGEN05 && fla::decode_tc_shape_supported(*dims))
    need = fla::decode_tc_workspace_bytes(*dims, n_req, total_tokens);
  if (dims->kernel != FLA_KERNEL_MMA_SYNC && fla::decode_t5_shape_supported(*dims))
    need = std::max(need, fla::decode_t5_workspace_bytes(*dims, n_req, total_tokens));
  return need;
}

// The tcgen05 decode kernel is chosen over the mma.sync one for these shapes
// (AUTO and TENSOR): groups of query rows large enough that the mma.sync
// kernel becomes compute-latency bound.
static bool prefer_tcgen05_decode(const fla_attn_dims &d) {
  return d.n_agents * (d.hq / d.hkv) > 16;
}

fla_status flash_lora_attn_decode(const fla_attn_dims *dims, const void *Q, const void *K_base,
                                  const void *V_base, const void *L, const void *B,
                                  const int32_t *offsets, int32_t n_req, int64_t total_tokens,
                                  float *O, void *workspace, size_t workspace_bytes,
                                  fla_stream_t stream) {
  g_last_error.clear();
  float scale = 0.f;
  fla_status st = check_dims(dims, &scale);
  if (st != FLA_OK) return st;
  if (n_req < 0 || total_tokens < 0) return fail(FLA_ERR_INVALID_ARG, "n_req and total_tokens must be >= 0");
  if (n_req == 0) return ok();
  if (!Q || !B || !offsets || !O) return fail(FLA_ERR_INVALID_ARG, "Q, B, offsets and O must be non-NULL");
  if (total_tokens > 0 && (!K_base || !V_base || !L))
    return fail(FLA_ERR_INVALID_ARG, "K_base, V_base and L must be non-NULL when total_tokens > 0");
  if (total_tokens > INT32_MAX) return fail(FLA_ERR_UNSUPPORTED, "total_tokens must fit in int32 (offsets are int32)");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  const bool align_tc = aligned16(Q) && aligned16(K_base) && aligned16(V_base) && aligned16(L) &&
                        aligned16(B) && aligned16(O) && (dims->l_row_stride % 8 == 0);
  const bool t5 = align_tc && fla::decode_t5_shape_supported(*dims);
  const bool mma = align_tc && fla::decode_tc_shape_supported(*dims);
  const int32_t k = dims->kernel;
  if (k == FLA_KERNEL_TCGEN05 && !t5)
    return fail(FLA_ERR_UNSUPPORTED, "decode: shape/alignment outside the tcgen05 kernel (bf16; head_dim 128; "
                "n_agents*hq/hkv <= 64; rank <= 64; L width <= 512; l_agent_stride 0 or rank; 16-byte alignment)");
  if (k == FLA_KERNEL_MMA_SYNC && !mma)
    return fail(FLA_ERR_UNSUPPORTED, "decode: shape/alignment outside the mma.sync kernel (%s)",
                fla::decode_tc_limits());
  if (k == FLA_KERNEL_TENSOR && !mma && !t5)
    return fail(FLA_ERR_UNSUPPORTED, "decode: shape/alignment outside both tensor-core kernels (%s)",
                fla::decode_tc_limits());
  const bool use_t5 = t5 && total_tokens > 0 &&
                      (k == FLA_KERNEL_TCGEN05 ||
                       ((k == FLA_KERNEL_AUTO || k == FLA_KERNEL_TENSOR) && (!mma || prefer_tcgen05_decode(*dims))));
  if (use_t5) {
    const size_t need = fla::decode_t5_workspace_bytes(*dims, n_req, total_tokens);
    if (!workspace || workspace_bytes < need)
      return fail(FLA_ERR_WORKSPACE, "decode: workspace of %zu bytes required, %zu given", need,
                  workspace ? workspace_bytes : (size_t)0);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
      return fail(FLA_ERR_INVALID_ARG, "decode: workspace must be 256-byte aligned");
    st = fla::decode_t5_launch(*dims, scale, Q, K_base, V_base, L, B, offsets, n_req, total_tokens, O, workspace, s);
    if (st != FLA_OK) return fail(st, "decode (tcgen05): %s", fla::decode_tc_last_error());
    return check_launch("decode (tcgen05)");
  }
  const bool shape_tc = mma;
  if (shape_tc && k != FLA_KERNEL_SIMT && total_tokens > 0) {
    const size_t need = fla::decode_tc_workspace_bytes(*dims, n_req, total_tokens);
    if (need > 0 && (!workspace || workspace_bytes < need))
      return fail(FLA_ERR_WORKSPACE, "decode: workspace of %zu bytes required, %zu given", need,
                  workspace ? workspace_bytes : (size_t)0);
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return fail(FLA_ERR_INVALID_ARG, "decode: workspace must be 256-byte aligned");
    st = fla::decode_tc_launch(*dims, scale, Q, K_base, V_base, L, B, offsets, n_req, total_tokens, O,
                               workspace, s);
    if (st != FLA_OK) return fail(st, "decode (tensor): %s", fla::decode_tc_last_error());
    return check_launch("decode (tensor)");
  }

  fla::SimtAttnParams p{};
  p.Q = Q; p.K = K_base; p.V = V_base; p.L = L; p.B = B; p.O = O; p.offsets = offsets;
  p.l_row_stride = dims->l_row_stride; p.l_agent_stride = dims->l_agent_stride;
  p.n_agents = dims->n_agents; p.hq = dims->hq; p.hkv = dims->hkv; p.d = dims->head_dim;
  p.r = dims->rank; p.n_req = n_req; p.prefill = 0; p.scale = scale;
  const int64_t rows = (int64_t)n_req * dims->n_agents * dims->hq;
  if (rows > 0x7fffffffLL) return fail(FLA_ERR_UNSUPPORTED, "too many query rows");
  if (dims->dtype == FLA_F32) launch_simt_attn<float>(p, rows, s);
  else launch_simt_attn<__nv_bfloat16>(p, rows, s);
  return check_launch("decode (simt)");
}

// ---------------------------------------------------------------------------
size_t flash_lora_attn_prefill_workspace_size(const fla_attn_dims *dims, int32_t chunk, int64_t n0) {
  float scale = 0.f;
  if (!dims || check_dims(dims, &scale) != FLA_OK || chunk <= 0 || n0 < 0) return 0;
  if (dims->kernel == FLA_KERNEL_SIMT || dims->kernel == FLA_KERNEL_MMA_SYNC) return 0;
  const fla::PrefillTcgen05Plan pl = fla::prefill_tcgen05_plan(*dims, chunk, n0);
  return pl.ok ? pl.part_bytes : 0;
}

fla_status flash_lora_attn_prefill(const fla_attn_dims *dims, const void *Q, const void *K_base,
                                   const void *V_base, const void *L, const void *B, int64_t n0,
                                   int32_t chunk, float *O, void *workspace, size_t workspace_bytes,
                                   fla_stream_t stream) {
  g_last_error.clear();
  float scale = 0.f;
  fla_status st = check_dims(dims, &scale);
  if (st != FLA_OK) return st;
  if (n0 < 0 || chunk < 0) return fail(FLA_ERR_INVALID_ARG, "n0 and chunk must be >= 0");
  if (chunk == 0) return ok();
  if (!Q || !K_base || !V_base || !L || !B || !O)
    return fail(FLA_ERR_INVALID_ARG, "Q, K_base, V_base, L, B and O must be non-NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool align_tc = aligned16(Q) && aligned16(K_base) && aligned16(V_base) && aligned16(L) &&
                        aligned16(B) && aligned16(O) && (dims->l_row_stride % 8 == 0);
  const bool tc5 = align_tc && fla::prefill_tcgen05_plan(*dims, chunk, n0).ok;
  const bool mma = align_tc && fla::prefill_tc_shape_supported(*dims);
  const int32_t k = dims->kernel;
  if (k == FLA_KERNEL_TCGEN05 && !tc5)
    return fail(FLA_ERR_UNSUPPORTED, "prefill: shape/alignment outside the tcgen05 kernel (bf16; head_dim 64 or "
                "128; A*hq/hkv <= 128; L width and A*rank <= 64; l_agent_stride 0 or rank; 16-byte alignment)");
  if (k == FLA_KERNEL_MMA_SYNC && !mma)
    return fail(FLA_ERR_UNSUPPORTED, "prefill: shape/alignment outside the mma.sync kernel (bf16; head_dim 64 or "
                "128; rank %% 16 == 0 and <= 64; l_agent_stride 0 or rank; 16-byte alignment)");
  if (k == FLA_KERNEL_TENSOR && !tc5 && !mma)
    return fail(FLA_ERR_UNSUPPORTED, "prefill: shape/alignment outside both tensor-core kernels");
  if (tc5 && (k == FLA_KERNEL_AUTO || k == FLA_KERNEL_TENSOR || k == FLA_KERNEL_TCGEN05)) {
    st = fla::prefill_tcgen05_launch(*dims, scale, Q, K_base, V_base, L, B, n0, chunk, O, workspace, workspace_bytes,
                                     s);
    if (st != FLA_OK) return fail(st, "prefill (tcgen05): %s", fla::prefill_tcgen05_last_error());
    return check_launch("prefill (tcgen05)");
  }
  if (mma && k != FLA_KERNEL_SIMT) {
    st = fla::prefill_tc_launch(*dims, scale, Q, K_base, V_base, L, B, n0, chunk, O, s);
    if (st != FLA_OK) return fail(st, "prefill (mma.sync): %s", fla::prefill_tc_last_error());
    return check_launch("prefill (mma.sync)");
  }
  fla::SimtAttnParams p{};
  p.Q = Q; p.K = K_base; p.V = V_base; p.L = L; p.B = B; p.O = O; p.offsets = nullptr;
  p.l_row_stride = dims->l_row_stride; p.l_agent_stride = dims->l_agent_stride; p.n0 = n0;
  p.n_agents = dims->n_agents; p.hq = dims->hq; p.hkv = dims->hkv; p.d = dims->head_dim;
  p.r = dims->rank; p.chunk = chunk; p.prefill = 1; p.scale = scale;
  const int64_t rows = (int64_t)dims->n_agents * chunk * dims->hq;
  if (rows > 0x7fffffffLL) return fail(FLA_ERR_UNSUPPORTED, "too many query rows");
  if (dims->dtype == FLA_F32) launch_simt_attn<float>(p, rows, s);
  else launch_simt_attn<__nv_bfloat16>(p, rows, s);
  return check_launch("prefill (simt)");
}

// ---------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call the library: a
// serving loop that fixed its memory budget at start-up and must not grow it
// (cudaMalloc also synchronises the device, which a latency-bound decode loop
// cannot afford), or a plugin whose host framework owns every allocation and
// hands it no scratch buffer.  For them the split-context partials live in
// the fixed array below, part of the library image: every GPU that loads the
// library holds these 16 MiB until the process exits.
// ---------------------------------------------------------------------------
static constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB
static __device__ __align__(256) unsigned char fla_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kNoAllocMaxDevices] = {};
void *g_noalloc_ctx[kNoAllocMaxDevices] = {};  // context the cached address belongs to

typedef CUresult (*PFN_ctxGetCurrent)(CUcontext *);

// The current driver context (nullptr if it cannot be asked).  A device reset
// destroys the primary context and the next one maps the library image again,
// possibly elsewhere, so the cached address is only valid for its context.
void *current_context() {
  static PFN_ctxGetCurrent fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_ctxGetCurrent>(p);
  });
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of the scratch array on the current device.  In host code
// the array's name only stands in for the symbol, so the address is asked of
// the runtime once per device (and again after a device reset), with that
// device current, and cached.
fla_status noalloc_scratch(void **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FLA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(FLA_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  void *ctx = current_context();
  if (!g_noalloc_ptr[dev] || ctx != g_noalloc_ctx[dev] || !ctx) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, fla_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return fail(FLA_ERR_CUDA, "cudaGetSymbolAddress(scratch) on device %d: %s", dev, cudaGetErrorString(e));
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx[dev] = current_context();  // the lookup may have created the primary context
  }
  *out = g_noalloc_ptr[dev];
  return FLA_OK;
}
}  // namespace

fla_status flash_lora_attn_decode_noalloc(const fla_attn_dims *dims, const void *Q, const void *K_base,
                                          const void *V_base, const void *L, const void *B,
                                          const int32_t *offsets, int32_t n_req, int64_t total_tokens, float *O,
                                          fla_stream_t stream) {
  g_last_error.clear();
  if (!dims) return fail(FLA_ERR_INVALID_ARG, "dims is NULL");
  const size_t need = flash_lora_attn_decode_workspace_size(dims, n_req, total_tokens);
  if (need > kNoAllocScratchBytes)
    return fail(FLA_ERR_WORKSPACE,
                "decode_noalloc: this call needs %zu bytes of scratch, more than the fixed %zu-byte array; "
                "use flash_lora_attn_decode with a caller-provided workspace",
                need, kNoAllocScratchBytes);
  void *scratch = nullptr;
  if (need > 0) {
    const fla_status st = noalloc_scratch(&scratch);
    if (st != FLA_OK) return st;
  }
  return flash_lora_attn_decode(dims, Q, K_base, V_base, L, B, offsets, n_req, total_tokens, O, scratch,
                                need > 0 ? kNoAllocScratchBytes : 0, stream);
}

// ---------------------------------------------------------------------------
fla_status lora_value_expand(const fla_attn_dims *dims, const void *V_base, const void *L, const void *B,
                             int64_t n_tokens, void *V_out, fla_stream_t stream) {
  g_last_error.clear();
  float scale;
  fla_status st = check_dims(dims, &scale);
  if (st != FLA_OK) return st;
  if (n_tokens < 0) return fail(FLA_ERR_INVALID_ARG, "n_tokens must be >= 0");
  if (!B) return fail(FLA_ERR_INVALID_ARG, "B must be non-NULL");
  if (n_tokens == 0) return FLA_OK;
  if (!V_base || !L || !V_out) return fail(FLA_ERR_INVALID_ARG, "V_base, L and V_out must be non-NULL");
  const fla_attn_dims &d = *dims;
  if (d.head_dim % 8 != 0)
    return fail(FLA_ERR_UNSUPPORTED, "lora_value_expand: head_dim %d must be a multiple of 8", d.head_dim);
  if (!aligned16(V_base) || !aligned16(V_out))
    return fail(FLA_ERR_INVALID_ARG, "lora_value_expand: V_base and V_out must be 16-byte aligned");
  if (d.kernel == FLA_KERNEL_TCGEN05)
    return fail(FLA_ERR_UNSUPPORTED, "lora_value_expand has no tcgen05 kernel (use TENSOR or MMA_SYNC)");
  const bool mma_shape = d.dtype == FLA_BF16 && (d.head_dim == 64 || d.head_dim == 128) && d.rank % 16 == 0 &&
                         d.l_row_stride % 2 == 0 && d.l_agent_stride % 2 == 0 &&
                         (reinterpret_cast<uintptr_t>(L) & 3u) == 0;
  const bool use_mma = d.kernel != FLA_KERNEL_SIMT && mma_shape;
  if ((d.kernel == FLA_KERNEL_TENSOR || d.kernel == FLA_KERNEL_MMA_SYNC) && !use_mma)
    return fail(FLA_ERR_UNSUPPORTED, "lora_value_expand: shape outside the mma.sync kernel (bf16; head_dim 64 or "
                "128; rank %% 16 == 0; even L strides; 4-byte aligned L)");
  const int group = fla::expand_agents_per_group(d.n_agents, d.rank, d.head_dim, use_mma);
  if (group < 1)
    return fail(FLA_ERR_UNSUPPORTED, "lora_value_expand: rank %d x head_dim %d of B exceeds the %d-byte "
                "shared-memory budget", d.rank, d.head_dim, fla::kExpMaxSmem);
  const size_t smem = (size_t)group * d.rank * d.head_dim * (use_mma ? 2 : 4);
  const int rows = fla::expand_rows_per_cta(n_tokens, d.hkv, fla::device_sm_count());
  const int64_t tiles = (n_tokens + rows - 1) / rows;
  if (tiles > 0x7fffffffLL || d.hkv > 65535) return fail(FLA_ERR_UNSUPPORTED, "lora_value_expand: grid too large");
  fla::ExpandParams p{};
  p.V = V_base; p.L = L; p.B = B; p.Vout = V_out;
  p.n_tokens = n_tokens; p.l_row_stride = d.l_row_stride; p.l_agent_stride = d.l_agent_stride;
  p.A = d.n_agents; p.hkv = d.hkv; p.d = d.head_dim; p.r = d.rank;
  p.rows_per_cta = rows; p.agents_per_group = group;
  const dim3 grid((unsigned)tiles, (unsigned)d.hkv);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  auto launch = [&](const void *fn, auto kernel, int threads) {
    e = fla::ensure_dynamic_smem(fn, (int)smem);
    if (e == cudaSuccess) kernel<<<grid, threads, smem, s>>>(p);
  };
  if (use_mma && d.head_dim == 128)
    launch(reinterpret_cast<const void *>(fla::lora_value_expand_mma_kernel<128>),
           fla::lora_value_expand_mma_kernel<128>, fla::kExpMmaWarps * 32);
  else if (use_mma)
    launch(reinterpret_cast<const void *>(fla::lora_value_expand_mma_kernel<64>),
           fla::lora_value_expand_mma_kernel<64>, fla::kExpMmaWarps * 32);
  else if (d.dtype == FLA_BF16)
    launch(reinterpret_cast<const void *>(fla::lora_value_expand_kernel<__nv_bfloat16>),
           fla::lora_value_expand_kernel<__nv_bfloat16>, fla::kExpThreads);
  else
    launch(reinterpret_cast<const void *>(fla::lora_value_expand_kernel<float>), fla::lora_value_expand_kernel<float>,
           fla::kExpThreads);
  if (e != cudaSuccess) return fail(FLA_ERR_CUDA, "lora_value_expand: %s", cudaGetErrorString(e));
  return check_launch("lora_value_expand");
}

// ---------------------------------------------------------------------------
fla_status flash_lora_attn_decode_host_io(const fla_attn_dims *dims, const void *Q_host, void *Q_dev,
                                          const void *K_base, const void *V_base, const void *L, const void *B,
                                          const int32_t *offsets, int32_t n_req, int64_t total_tokens,
                                          float *O_dev, float *O_host, void *workspace, size_t workspace_bytes,
                                          fla_stream_t stream) {
  g_last_error.clear();
  if (!dims) return fail(FLA_ERR_INVALID_ARG, "dims is NULL");
  if (!Q_host || !Q_dev || !O_dev || !O_host)
    return fail(FLA_ERR_INVALID_ARG, "Q_host, Q_dev, O_dev and O_host must be non-NULL");
  if (n_req < 0) return fail(FLA_ERR_INVALID_ARG, "n_req must be >= 0");
  const size_t esize = dims->dtype == FLA_BF16 ? 2 : 4;
  const size_t elems = (size_t)n_req * dims->n_agents * dims->hq * dims->head_dim;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the shape checks shared with decode run before the copy; the decode's own
  // remaining checks run after it (documented: Q_dev may then hold the queries)
  float scale;
  fla_status st = check_dims(dims, &scale);
  if (st != FLA_OK) return st;
  if (elems == 0) return FLA_OK;
  cudaError_t e = cudaMemcpyAsync(Q_dev, Q_host, elems * esize, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return fail(FLA_ERR_CUDA, "decode_host_io: copying Q to the device: %s", cudaGetErrorString(e));
  st = flash_lora_attn_decode(dims, Q_dev, K_base, V_base, L, B, offsets, n_req, total_tokens, O_dev, workspace,
                              workspace_bytes, stream);
  if (st != FLA_OK) return st;
  e = cudaMemcpyAsync(O_host, O_dev, elems * sizeof(float), cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return fail(FLA_ERR_CUDA, "decode_host_io: copying O to the host: %s", cudaGetErrorString(e));
  return FLA_OK;
}

}  // extern "C"
