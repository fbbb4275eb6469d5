/*
 * flash_lora_attn.h - C ABI of the Flash-LoRA-Attention library (B300, sm_103a).
 *
 * The method (LRAgent technical summary, gist.science, "Metodologia"):
 *   - section 1 "Descomposicion de la Cache": an agent's value cache is a base
 *     part shared by all agents plus a LoRA adapter part, V_i = V_base + dV_i;
 *   - section 2, BaseShared: the adapter part is kept in low-rank form, the LR
 *     cache L_i = X . A_i of width r, expanded by the up-projection B_i only
 *     when needed; BaseLRShared: A is shared, so one LR cache serves all agents;
 *   - section 3 "Flash-LoRA-Attention": attention over the decomposed cache is
 *     evaluated as P.V_base + (P.L_i).B_i instead of P.(V_base + L_i.B_i), so
 *     L_i.B_i is never expanded to full width and B_i is applied once per query.
 * PReCache abstract (arxivdaily), PreLRShared: every agent's LR cache is built
 * when the shared context is first processed (lr_cache_build over all agents).
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers to caller-owned memory on the
 *     current CUDA device (the one exception: the Q_host / O_host buffers of
 *     flash_lora_attn_decode_host_io); the library never allocates, frees or
 *     keeps them.
 *   - Tensors are dense row-major unless a stride argument says otherwise.
 *   - Calls are enqueued on `stream` (NULL = the legacy default stream), are
 *     asynchronous and never synchronise the host.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns an error status and launches nothing.
 *   - Errors never cross the ABI as exceptions.  fla_last_error()
 *     returns a thread-local description of the last failure.
 *   - Device-side waits are bounded.  A kernel whose wait runs out sets a
 *     device error word and returns early (its outputs are then undefined);
 *     read and clear it with fla_device_error() after synchronising.
 *   - Storage dtype: FLA_BF16 (fp32 accumulation) or FLA_F32.  Attention
 *     outputs O are always fp32.
 */
#ifndef FLASH_LORA_ATTN_H_
#define FLASH_LORA_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FLA_API __attribute__((visibility("default")))
#else
#define FLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL selects the legacy default stream. */
typedef struct CUstream_st *fla_stream_t;

typedef enum {
  FLA_OK = 0,
  FLA_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned pointer, ... */
  FLA_ERR_UNSUPPORTED = 2,    /* valid but outside what the kernels implement */
  FLA_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required */
  FLA_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed (no device, launch error) */
  FLA_ERR_DEVICE_TIMEOUT = 5  /* reported by fla_device_error(): a bounded wait ran out */
} fla_status;

typedef enum { FLA_F32 = 0, FLA_BF16 = 1 } fla_dtype;

/* Kernel family.  AUTO picks the fastest kernel the shape allows.  SIMT
 * forces the CUDA-core kernels (every supported shape).  TENSOR uses a
 * tensor-core kernel (tcgen05 where the operation has one and the shape fits,
 * warp-level mma.sync otherwise) and fails with FLA_ERR_UNSUPPORTED when the
 * shape is outside every tensor-core kernel's limits.  MMA_SYNC and TCGEN05
 * pin the tensor-core generation: warp-level mma.sync (decode, prefill) or
 * tcgen05 with TMEM accumulators (LR-cache build, prefill); an operation
 * without a kernel of that generation returns FLA_ERR_UNSUPPORTED. */
typedef enum {
  FLA_KERNEL_AUTO = 0,
  FLA_KERNEL_SIMT = 1,
  FLA_KERNEL_TENSOR = 2,
  FLA_KERNEL_MMA_SYNC = 3,
  FLA_KERNEL_TCGEN05 = 4
} fla_kernel;

/* Shape of the attention problem (decode and prefill). */
typedef struct {
  int32_t n_agents;       /* A >= 1: agents sharing the base cache */
  int32_t hq;             /* query heads per agent, hq % hkv == 0 */
  int32_t hkv;            /* key/value heads; q head j reads kv head j / (hq/hkv) */
  int32_t head_dim;       /* d: 64 or 128 (tensor kernels); 1..256, multiple of 4 (SIMT) */
  int32_t rank;           /* r: LoRA rank, 1..256 */
  int32_t dtype;          /* fla_dtype of Q, K_base, V_base, L and B */
  int64_t l_row_stride;   /* elements between consecutive tokens of L */
  int64_t l_agent_stride; /* elements between agents' column blocks of L: r for
                             per-agent LR caches (BaseShared), 0 for one LR cache
                             shared by every agent (BaseLRShared) */
  float softmax_scale;    /* <= 0 selects 1/sqrt(head_dim) */
  int32_t kernel;         /* fla_kernel */
} fla_attn_dims;

/*
 * lr_cache_build - L = X . A_cat, i.e. L[t, c] = sum_k X[t, k] * A_cat[k, c]
 *
 * LRAgent summary, Metodologia section 2 (BaseShared: the LR cache stores the
 * LoRA down-projection X.A_i at width r); PReCache abstract (PreLRShared:
 * all agents' LR caches built in one pass over the context).
 *
 *   X        [n_tokens, d_model], row stride ldx elements    (input)
 *   A_cat    [d_model, n_agents * rank], dense row-major: the agents'
 *            down-projections side by side, A_cat = [A_1 | ... | A_A], agent i
 *            owning columns [i*rank, (i+1)*rank)               (input)
 *   L        [n_tokens, n_agents * rank] written with row stride ldl elements
 *            (output; column block i is agent i's LR cache L_i = X . A_i;
 *            other columns of a wider L are left untouched)
 *   dtype    storage type of X, A_cat and L; fp32 accumulation.
 *   kernel   fla_kernel.  The tensor-core (tcgen05) path needs bf16,
 *            d_model % 64 == 0, n_agents * rank % 32 == 0, 16-byte aligned
 *            pointers and ldx, ldl multiples of 8; wider products are tiled
 *            over 512-column tiles, and short inputs split d_model over a
 *            thread-block cluster.  SIMT covers every other shape.
 * Errors: FLA_ERR_INVALID_ARG for null pointers with n_tokens > 0, negative
 * sizes, n_agents or rank < 1, ldx < d_model or ldl < n_agents * rank.
 * n_tokens == 0 is a no-op.
 */
FLA_API fla_status lr_cache_build(const void *X, int64_t ldx, const void *A_cat, void *L, int64_t ldl,
                                  int64_t n_tokens, int32_t d_model, int32_t n_agents, int32_t rank,
                                  int32_t dtype, int32_t kernel, fla_stream_t stream);

/*
 * rebase_kv_lr_build - the shared base K/V caches and every agent's LR cache
 * from one pass over the hidden states:
 *   [K_base | V_base | L] = X . [W_k | W_v | A_cat]
 *
 * PReCache abstract (arxivdaily), ReBaseShared: the shared base cache is
 * rebuilt from adapter-free hidden states with the pretrained weights;
 * PreLRShared: each agent's LR cache is computed when the context is
 * processed.  LRAgent summary, Metodologia section 1: the base value cache
 * comes from the frozen pretrained projection.  One tensor-core GEMM reads
 * each tile of X once for all three outputs.  No rotary embedding is applied
 * to K_base (a caller that uses one applies it afterwards).
 *
 *   X        [n_tokens, d_model], row stride ldx elements        (input)
 *   W_cat    [d_model, 2*hkv*head_dim + n_agents*rank], dense row-major:
 *            the pretrained key projection W_k [d_model, hkv*head_dim], the
 *            value projection W_v (same shape) and A_cat = [A_1 | ... | A_A]
 *            side by side, in that order                         (input)
 *   K_base   [n_tokens, hkv, head_dim], dense                    (output)
 *   V_base   [n_tokens, hkv, head_dim], dense                    (output)
 *   L        [n_tokens, n_agents * rank], row stride ldl         (output)
 *   dtype, kernel as for lr_cache_build.  The tensor-core path needs bf16,
 *            d_model % 64 == 0, hkv*head_dim and n_agents*rank multiples of
 *            32, 16-byte aligned pointers, ldx and ldl multiples of 8.
 * Errors: FLA_ERR_INVALID_ARG for null pointers with n_tokens > 0, sizes < 1,
 * ldx < d_model or ldl < n_agents * rank.  n_tokens == 0 is a no-op.
 */
FLA_API fla_status rebase_kv_lr_build(const void *X, int64_t ldx, const void *W_cat, void *K_base, void *V_base,
                                      void *L, int64_t ldl, int64_t n_tokens, int32_t d_model, int32_t hkv,
                                      int32_t head_dim, int32_t n_agents, int32_t rank, int32_t dtype,
                                      int32_t kernel, fla_stream_t stream);

/*
 * flash_lora_attn_decode - one query token per agent per request.
 *
 * For request q, agent a, query head j (kv head h = j / (hq/hkv)) and the
 * tokens t of request q (offsets[q] <= t < offsets[q+1]):
 *   s_t = softmax_scale * <Q[q,a,j,:], K_base[t,h,:]>,  P = softmax_t(s)
 *   O[q,a,j,:] = sum_t P_t V_base[t,h,:] + (sum_t P_t L[t, a*l_agent_stride + (0..r-1)]) . B[a, :, h*d:(h+1)*d]
 * i.e. softmax(Q.K_base^T/sqrt(d)).(V_base + L_a.B_a) evaluated in the
 * reordered form of LRAgent section 3; L_a.B_a is never formed.  Every
 * agent's query rows for a kv head are served from one read of each K_base /
 * V_base tile.  A request with no tokens gets O = 0.
 *
 *   Q        [n_req, A, hq, d]                              (input)
 *   K_base   [total_tokens, hkv, d]  requests packed by offsets  (input)
 *   V_base   [total_tokens, hkv, d]                         (input)
 *   L        [total_tokens, l_row_stride]                   (input)
 *   B        [A, r, hkv*d]                                  (input)
 *   offsets  device int32 [n_req + 1], offsets[0] == 0, non-decreasing,
 *            offsets[n_req] == total_tokens                 (input)
 *   O        fp32 [n_req, A, hq, d]                         (output)
 *   workspace device scratch of at least
 *            flash_lora_attn_decode_workspace_size() bytes, 256-byte
 *            aligned, any initial contents.  It holds the per-unit partial
 *            results of long contexts between the decode kernel and the merge
 *            kernel the call enqueues behind it; calls that may overlap on the
 *            GPU must use different workspaces.
 * Ordering: the call's kernels are launched with programmatic dependent
 * launch, so when the previous work on the stream is this library's decode,
 * the new call starts reading Q, K_base, V_base, L, B and offsets while that
 * decode finishes.  Those inputs must not be the O or the workspace of the
 * decode call enqueued immediately before on the same stream (every other
 * producer, e.g. a PyTorch kernel, has completed first as usual).
 * Errors: INVALID_ARG (null pointer, hq % hkv, offsets layout on the host
 * side, strides), UNSUPPORTED (shape outside the selected kernel's limits),
 * WORKSPACE (too small), CUDA (launch failure).
 */
FLA_API size_t flash_lora_attn_decode_workspace_size(const fla_attn_dims *dims, int32_t n_req,
                                             int64_t total_tokens);
FLA_API fla_status flash_lora_attn_decode(const fla_attn_dims *dims, const void *Q, const void *K_base,
                                  const void *V_base, const void *L, const void *B,
                                  const int32_t *offsets, int32_t n_req, int64_t total_tokens,
                                  float *O, void *workspace, size_t workspace_bytes,
                                  fla_stream_t stream);

/*
 * flash_lora_attn_prefill - causal chunked prefill of `chunk` new tokens for
 * every agent over a shared context of n0 cached tokens.
 *
 * The query at chunk position p (absolute position n0 + p) sees keys
 * 0 .. n0 + p inclusive:
 *   O[a,p,j,:] = softmax over t <= n0+p of (scale <Q[a,p,j,:], K_base[t,h,:]>)
 *                applied to V_base[t,h,:] + L[t, a-block] . B[a, :, h*d:(h+1)*d]
 * evaluated as P.V_base + (P.L_a).B_a (B applied once per query block).
 *
 *   Q        [A, chunk, hq, d]                   (input)
 *   K_base   [n0 + chunk, hkv, d]                (input; the chunk's keys appended)
 *   V_base   [n0 + chunk, hkv, d]                (input)
 *   L        [n0 + chunk, l_row_stride]          (input; the chunk's rows built
 *                                                 by lr_cache_build beforehand)
 *   B        [A, r, hkv*d]                       (input)
 *   O        fp32 [A, chunk, hq, d]              (output)
 *   workspace flash_lora_attn_prefill_workspace_size() bytes, 16-byte aligned
 *            (may be 0 bytes / NULL when the size query returns 0).  The
 *            tcgen05 kernel uses it to run the CTA pairs of a last, partly
 *            filled wave as two half-range items whose row records a merge
 *            kernel combines; with a smaller or unaligned workspace it runs
 *            every pair over its whole key range instead (same results up to
 *            rounding, no error).  Calls on one stream may share it.
 * Kernels: tcgen05 (bf16; head_dim 64 or 128; A*(hq/hkv) <= 128; L width
 * (r, or A*r) <= 64 and A*r <= 64; l_agent_stride 0 or r); mma.sync (bf16;
 * head_dim 64 or 128; r % 16 == 0, r <= 64; l_agent_stride 0 or r); both need
 * 16-byte aligned pointers and l_row_stride % 8 == 0.  SIMT covers the rest.
 * Errors as for decode.
 */
FLA_API size_t flash_lora_attn_prefill_workspace_size(const fla_attn_dims *dims, int32_t chunk, int64_t n0);
FLA_API fla_status flash_lora_attn_prefill(const fla_attn_dims *dims, const void *Q, const void *K_base,
                                   const void *V_base, const void *L, const void *B, int64_t n0,
                                   int32_t chunk, float *O, void *workspace,
                                   size_t workspace_bytes, fla_stream_t stream);

/*
 * flash_lora_attn_decode_noalloc - flash_lora_attn_decode without a
 * caller-provided workspace.  The pages have no counterpart: this is a
 * library convenience, not part of the method.
 *
 * For callers that cannot allocate device memory at call time (a serving
 * loop whose memory budget is fixed at start-up, or a plugin whose host
 * framework owns every allocation and gives it no scratch buffer).  Same
 * arguments, layouts and results as flash_lora_attn_decode minus the
 * workspace; the partial results of split contexts go to a 16 MiB array that
 * is part of the library image (every GPU that loads the library holds it
 * until the process exits).
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.  The cache is keyed on the
 *     device's current context, so after cudaDeviceReset the next call looks
 *     the address up again (make that call outside a capture too).
 *   - Every call on a device shares the one array; it needs no zeroing (each
 *     call writes every scratch value before reading it) and keeps the last
 *     call's contents.  Calls on one device that may overlap on the GPU (for
 *     example on different streams) race on the array: serialise them, or
 *     use flash_lora_attn_decode with a workspace per stream.
 *   - Returns FLA_ERR_WORKSPACE when the call needs more scratch than the
 *     array holds (flash_lora_attn_decode_workspace_size() > 16 MiB).
 */
FLA_API fla_status flash_lora_attn_decode_noalloc(const fla_attn_dims *dims, const void *Q, const void *K_base,
                                                  const void *V_base, const void *L, const void *B,
                                                  const int32_t *offsets, int32_t n_req, int64_t total_tokens,
                                                  float *O, fla_stream_t stream);

/*
 * lora_value_expand - the materialised value cache of every agent:
 *   V_out[a, t, h, :] = V_base[t, h, :] + L[t, a*l_agent_stride + (0..r-1)] . B[a, :, h*d:(h+1)*d]
 *
 * LRAgent summary, Metodologia section 1 (V_i = V_base + L_i.B_i) and section
 * 3, Problema bullet: this full-width reconstruction for every agent is what
 * Flash-LoRA-Attention avoids.  It is provided as the first half of the
 * naive-materialisation baseline (plain attention over each V_i is the
 * second) that the reordered decode is measured against.  No decode or
 * prefill call uses it.
 *
 *   V_base  [n_tokens, hkv, d]                 (input)
 *   L       [n_tokens, l_row_stride]           (input)
 *   B       [A, r, hkv*d]                      (input)
 *   V_out   [A, n_tokens, hkv, d], same dtype  (output; agent-major)
 * Uses n_agents, hkv, head_dim, rank, dtype, l_row_stride, l_agent_stride and
 * kernel of `dims` (hq and softmax_scale are validated as for decode but not
 * used).  fp32 accumulation, one rounding to the storage dtype per value.
 * Kernels: mma.sync (bf16; head_dim 64 or 128; rank % 16 == 0; even
 * l_row_stride and l_agent_stride; L 4-byte aligned; rank x head_dim x 2
 * bytes at most 96 KiB); CUDA cores otherwise (head_dim % 8 == 0; rank x
 * head_dim x 4 bytes at most 96 KiB).  TCGEN05 is UNSUPPORTED.  V_base and
 * V_out must be 16-byte aligned.
 * Errors: INVALID_ARG (null pointer with n_tokens > 0, n_tokens < 0,
 * alignment, the dims checks of decode), UNSUPPORTED (shape outside the
 * selected kernel), CUDA (launch failure).  n_tokens == 0 is a no-op.
 */
FLA_API fla_status lora_value_expand(const fla_attn_dims *dims, const void *V_base, const void *L, const void *B,
                                     int64_t n_tokens, void *V_out, fla_stream_t stream);

/*
 * flash_lora_attn_decode_host_io - flash_lora_attn_decode for queries that
 * arrive in host memory and outputs that are wanted there: one call enqueues,
 * on `stream`, the copy Q_host -> Q_dev, the decode of Q_dev into O_dev and
 * the copy O_dev -> O_host.  A serving loop's step is then one library call.
 * The pages have no counterpart: this is a library convenience.
 *
 *   Q_host   host [n_req, A, hq, d] in dims->dtype; page-locked (pinned)
 *            memory keeps both copies asynchronous
 *   Q_dev    device buffer of the same size (the decode's Q)
 *   O_dev    device fp32 [n_req, A, hq, d] (the decode's O)
 *   O_host   host fp32 [n_req, A, hq, d], pinned as above; valid once the
 *            stream has reached the end of this call's work
 *   the other arguments as for flash_lora_attn_decode.
 * Allocates nothing; the copies are plain cudaMemcpyAsync calls.  The shape
 * checks shared with decode run before anything is enqueued; when a later
 * decode check fails, the Q copy has been enqueued (Q_dev is overwritten) but
 * no kernel is launched.  n_req == 0 is a no-op.
 * Errors: as for flash_lora_attn_decode, plus INVALID_ARG for a NULL host or
 * staging pointer and CUDA when a copy cannot be enqueued.
 */
FLA_API fla_status flash_lora_attn_decode_host_io(const fla_attn_dims *dims, const void *Q_host, void *Q_dev,
                                                  const void *K_base, const void *V_base, const void *L,
                                                  const void *B, const int32_t *offsets, int32_t n_req,
                                                  int64_t total_tokens, float *O_dev, float *O_host, void *workspace,
                                                  size_t workspace_bytes, fla_stream_t stream);

/* Human-readable name of a status code (static storage). */
FLA_API const char *fla_status_string(fla_status status);

/* Description of the last failure on the calling thread ("" if none). */
FLA_API const char *fla_last_error(void);

/* Reads, and resets to 0, the device error word of the current device.
 * Synchronises the device first.  Writes 0 (no error) or a nonzero code that
 * identifies the bounded wait that ran out; returns FLA_ERR_CUDA if the read
 * itself fails. */
FLA_API fla_status fla_device_error(uint32_t *code);

/* Self-test of the bounded waits (failure detection without a fault).
 *
 * Launches one CTA on `stream` whose warp 0 waits on an mbarrier that no one
 * arrives on, through the same bounded-wait helper every pipeline kernel uses,
 * with a limit of limit_ns nanoseconds; when it runs out the helper records
 * code 0x401 in the device error word and raises the CTA's abort flag.  Warp 1
 * waits on a second such barrier with the kernels' own 2 s limit and leaves
 * through that flag.  No fault, trap or hang: the CTA returns and the context
 * stays usable.
 *   limit_ns  (0, 2e9].
 *   out       device memory, 3 x uint64, written by the kernel: out[0] = 1 if
 *             warp 0's wait ran out, out[1] = 1 if warp 1 left on the abort
 *             flag, out[2] = warp 0's wait in nanoseconds.
 * Read (and clear) the code with fla_device_error() afterwards.  Errors:
 * INVALID_ARG (out NULL, limit out of range), CUDA (launch failure). */
FLA_API fla_status fla_selftest_bounded_wait(uint64_t limit_ns, unsigned long long *out, fla_stream_t stream);

/* Library version, e.g. "0.1.0". */
FLA_API const char *fla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FLASH_LORA_ATTN_H_ */
