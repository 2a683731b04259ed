/*
 * cpattn.h -- C ABI of libcpattn.so: the data-parallel hot path of
 * context-parallel attention (Ring, Ring Anything, Ulysses, Ulysses Anything
 * and their Unified composition) on one GB300.
 *
 * Sources (page title, section):
 *   [CP]   Diffusers "Context parallelism" guide: variants table, "Ring
 *          Attention", "Ulysses Attention", "Unified Attention", "Ring
 *          Anything Attention", "Ulysses Anything Attention".
 *   [API]  Diffusers "Parallelism" API page, ContextParallelConfig:
 *          ring_degree, ulysses_degree, convert_to_fp32, ring_anything,
 *          ulysses_anything.
 *   [PARA] ParaAttention README, "Run Unified Attention ... with
 *          torch.compile": scaled_dot_product_attention with no mask, no
 *          dropout, not causal, on [B, H, S, D] tensors chunked on dim -2.
 *   [CFG]  diffusers _modeling_parallel.py, ContextParallelConfig
 *          (__post_init__ validation).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Tensors are described by cpattn_tensor: a DEVICE pointer, a dtype, and
 *   shape/stride in ELEMENTS.  The innermost dimension must have stride 1;
 *   every other stride times the element size must be a multiple of 16 bytes,
 *   and the data pointer must be 16-byte aligned (CPATTN_ERR_LAYOUT).
 * - Ownership: the caller allocates every input, output and workspace buffer
 *   and keeps it alive until the stream has finished the call.  The library
 *   allocates no device memory and keeps no state between calls except one
 *   device error word (see cpattn_last_device_status) and the fixed
 *   workspace array of cpattn_ring_noalloc (part of the library's static
 *   device memory).  Descriptors are only read during the call.
 * - Asynchrony: every call is enqueued on `stream` (a cudaStream_t; NULL is the
 *   legacy default stream).  Argument errors are returned synchronously before
 *   anything is launched; a launch failure returns CPATTN_ERR_CUDA.  A wait
 *   inside a kernel that runs out of its time limit records CPATTN_ERR_TIMEOUT
 *   in the device error word, and the kernel returns.
 * - Scale: scale <= 0 or NaN selects 1/sqrt(D), the scaled_dot_product_attention
 *   default [PARA].
 * - Supported: head size D in {64, 128}, for bf16 inputs (tensor cores, bf16
 *   operands, fp32 accumulation) and fp32 inputs (tensor cores, tf32
 *   operands with Q K^T taken as three tf32 products of a high/low split,
 *   fp32 accumulation).  Anything else: CPATTN_ERR_UNSUPPORTED.  There is
 *   no CPU fallback.
 */
#ifndef CPATTN_H_
#define CPATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CPATTN_OK = 0,
  CPATTN_ERR_NULL = 1,          /* a required pointer is NULL */
  CPATTN_ERR_DTYPE = 2,         /* dtype not allowed for that argument */
  CPATTN_ERR_SHAPE = 3,         /* ranks or extents inconsistent */
  CPATTN_ERR_DIVISIBILITY = 4,  /* S % ring_degree or H % degree != 0 */
  CPATTN_ERR_LAYOUT = 5,        /* inner stride != 1, or not 16-byte aligned */
  CPATTN_ERR_UNSUPPORTED = 6,   /* valid, but outside what the kernels cover */
  CPATTN_ERR_WORKSPACE = 7,     /* workspace missing or too small */
  CPATTN_ERR_CUDA = 8,          /* a CUDA runtime call failed */
  CPATTN_ERR_TIMEOUT = 9,       /* a device-side wait ran out of time */
  CPATTN_ERR_BOUNDS = 10        /* a device-side bounds check failed (check builds only) */
} cpattn_status;

typedef enum { CPATTN_F32 = 0, CPATTN_BF16 = 1 } cpattn_dtype;

#define CPATTN_MAX_DIMS 5
#define CPATTN_MAX_RING_DEGREE 64

typedef struct {
  void* data;                        /* device pointer */
  int32_t dtype;                     /* cpattn_dtype */
  int32_t ndim;
  int64_t shape[CPATTN_MAX_DIMS];    /* elements */
  int64_t stride[CPATTN_MAX_DIMS];   /* elements */
} cpattn_tensor;

/*
 * cpattn_partial -- one ring step: attention of a query chunk against ONE K/V
 * chunk, emitting the partial output and its log-sum-exp ([CP] "Ring
 * Attention": each GPU computes attention against the K/V block it holds;
 * [API] convert_to_fp32: output and LSE kept in float32).
 *   q   [B, H, S_q, D]   bf16 or f32
 *   k,v [B, H, S_kv, D]  same dtype as q, S_kv >= 1
 *   out [B, H, S_q, D]   f32 (written):  softmax(scale q k^T) v
 *   lse [B, H, S_q]      f32 (written):  natural log of sum_j exp(scale q.k_j)
 * S_q = 0 (or B = 0, H = 0) is a no-op.  S_kv = 0 is CPATTN_ERR_SHAPE.
 */
cpattn_status cpattn_partial(const cpattn_tensor* q, const cpattn_tensor* k,
                             const cpattn_tensor* v, float scale,
                             cpattn_tensor* out, cpattn_tensor* lse,
                             void* stream);

/*
 * cpattn_merge -- LSE merge of two partials over disjoint key sets, in place
 * into (out_a, lse_a) ([API] convert_to_fp32: the ring's partials are kept
 * in fp32 while they are combined, for stability):
 *   lse = max(a, b) + log1p(exp(min(a, b) - max(a, b)))
 *   out = exp(a - lse) out_a + exp(b - lse) out_b
 * lse = -inf marks an empty partial; two empty partials give (0, -inf).
 *   out_a, out_b [B, H, S, D] f32;  lse_a, lse_b [B, H, S] f32.
 * out_a/lse_a may not overlap out_b/lse_b.
 */
cpattn_status cpattn_merge(cpattn_tensor* out_a, cpattn_tensor* lse_a,
                           const cpattn_tensor* out_b,
                           const cpattn_tensor* lse_b, void* stream);

/*
 * cpattn_ring_workspace_bytes -- bytes of device workspace cpattn_ring needs
 * for q [B, H, S_q, D] and this ring_degree: the running merged output and
 * its LSE in f32, S_q rounded up to a multiple of 128 rows:
 * B * H * ceil(S_q / 128) * 128 * (D + 1) * 4 bytes; 0 when ring_degree = 1.
 * The layout inside is private to the library.  Returns 0 for an invalid
 * descriptor.
 */
size_t cpattn_ring_workspace_bytes(const cpattn_tensor* q, int ring_degree);

/*
 * cpattn_ring -- the whole ring schedule simulated on one GPU ([CP] "Ring
 * Attention"): the keys are split into ring_degree chunks; every query tile
 * meets every chunk in order 0 .. R-1, each meeting emits (partial out, f32
 * LSE) and the partials are folded with the merge above.  All chunk loops and
 * merges run inside one kernel launch.
 *   ring_anything = 0: S_kv % ring_degree != 0 is CPATTN_ERR_DIVISIBILITY
 *     ([CP] variants table).
 *   ring_anything = 1: any S_kv >= ring_degree; the first S_kv % R chunks are
 *     one key longer ([CP] "Ring Anything Attention"; no mask exists here,
 *     as that variant requires).
 *   q [B, H, S_q, D], k, v [B, H, S_kv, D]: bf16 or f32, D = 64 or 128.
 *   out [B, H, S_q, D] same dtype as q (written); lse [B, H, S_q] f32.
 *   workspace: device buffer of at least cpattn_ring_workspace_bytes (16-byte
 *     aligned), may be NULL when ring_degree = 1; its contents on entry do
 *     not matter.
 *   1 <= ring_degree <= CPATTN_MAX_RING_DEGREE.
 */
cpattn_status cpattn_ring(const cpattn_tensor* q, const cpattn_tensor* k,
                          const cpattn_tensor* v, float scale, int ring_degree,
                          int ring_anything, cpattn_tensor* out,
                          cpattn_tensor* lse, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * cpattn_ring_causal -- cpattn_ring with causal masking, the is_causal of
 * scaled_dot_product_attention ([PARA] passes is_causal; SDPA's mask is
 * top-left aligned): query i attends keys j <= i only.  Every chunk's
 * partial covers the admissible keys of that chunk; a row with none gets the
 * empty partial (0, -inf), the identity of the merge, so the ring result is
 * causal attention over all keys.  Chunks wholly after a query tile are not
 * visited, and query tiles are scheduled heaviest first.  Arguments, layout,
 * workspace and errors as cpattn_ring.
 */
cpattn_status cpattn_ring_causal(const cpattn_tensor* q, const cpattn_tensor* k,
                                 const cpattn_tensor* v, float scale, int ring_degree,
                                 int ring_anything, cpattn_tensor* out,
                                 cpattn_tensor* lse, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * cpattn_ulysses_permute -- the Ulysses head regroup ([CP] "Ulysses
 * Attention": the all-to-all leaves each of G ranks every token for H/G
 * heads), on one GPU a bit-exact layout permute:
 *   dir = +1: x [B, S, H, D] -> y [G, B, S, H/G, D],
 *             y[g, b, s, hh, :] = x[b, s, g*H/G + hh, :]
 *   dir = -1: x [G, B, S, H/G, D] -> y [B, S, H, D] (the inverse map)
 * degree = G >= 1 with H % G == 0 (else CPATTN_ERR_DIVISIBILITY).  Any dtype
 * of this header (the copy moves bytes).  x and y must be contiguous and must
 * not overlap.
 */
cpattn_status cpattn_ulysses_permute(const cpattn_tensor* x, int degree,
                                     int dir, cpattn_tensor* y, void* stream);

/* Up to CPATTN_MAX_PERMUTE_BATCH regroups in one launch. */
#define CPATTN_MAX_PERMUTE_BATCH 4

/*
 * cpattn_ulysses_permute_batch -- cpattn_ulysses_permute of n tensors of one
 * shape and dtype in one launch (q, k and v each pass through the all-to-all
 * of [CP] "Ulysses Attention" before the per-group attention).
 *   x, y: arrays of n descriptors; pair i is regrouped x[i] -> y[i] exactly
 *   as cpattn_ulysses_permute does, 1 <= n <= CPATTN_MAX_PERMUTE_BATCH
 *   (else CPATTN_ERR_SHAPE).  Every pair must have the shapes and dtype of
 *   pair 0 (else CPATTN_ERR_SHAPE / CPATTN_ERR_DTYPE); no output may overlap
 *   any input or another output (CPATTN_ERR_LAYOUT).  Other errors as
 *   cpattn_ulysses_permute; on any error nothing is launched.
 */
cpattn_status cpattn_ulysses_permute_batch(int n, const cpattn_tensor* x, int degree,
                                           int dir, cpattn_tensor* y, void* stream);

/*
 * cpattn_ulysses_anything_permute -- the head regroup of Ulysses Anything
 * ([CP] "Ulysses Anything Attention", [API] ulysses_anything: Ulysses without
 * the rule that H divides by G).  Heads are dealt out as torch.tensor_split
 * does (G consecutive groups, the first H mod G of them one head longer);
 * every group gets hm = ceil(H/G) head slots so the exchange buffer has one
 * shape, and group g fills slots 0 .. h_g - 1:
 *   dir = +1: x [B, S, H, D] -> y [G, B, S, hm, D],
 *             y[g, b, s, j, :] = x[b, s, start_g + j, :] for j < h_g;
 *             padding slots of y are not written.
 *   dir = -1: x [G, B, S, hm, D] -> y [B, S, H, D] (the inverse map; padding
 *             slots of x are not read).
 * degree = G >= 1, any H >= 1 (groups past H hold no head).  Any dtype of
 * this header.  x and y must be contiguous and must not overlap.  On one GPU
 * every group keeps the whole sequence, so S needs no rule.
 */
cpattn_status cpattn_ulysses_anything_permute(const cpattn_tensor* x,
                                              int degree, int dir,
                                              cpattn_tensor* y, void* stream);

/*
 * cpattn_ulysses_anything_permute_batch -- cpattn_ulysses_anything_permute
 * of n tensors of one shape and dtype in one launch; arguments, pairing and
 * errors as cpattn_ulysses_permute_batch.
 */
cpattn_status cpattn_ulysses_anything_permute_batch(int n, const cpattn_tensor* x,
                                                    int degree, int dir,
                                                    cpattn_tensor* y, void* stream);

/*
 * cpattn_ulysses_anything_attention -- attention of every Ulysses Anything
 * group over its own heads and the whole sequence, all groups in one launch
 * ([CP] "Ulysses Anything Attention": ring_degree must be 1, so each group
 * runs plain attention).
 *   q, k, v, out [G, B, S, hm, D] in the layout cpattn_ulysses_anything_permute
 *     writes (any strides with inner stride 1, 16-byte multiples elsewhere
 *     and stride[0] = B * stride[1]); hm = ceil(heads / G).
 *   heads = H, the total head count (it fixes each group's h_g).
 *   is_causal: 0, or 1 for query i attending keys j <= i.
 *   out: same dtype as q; lse [G, B, hm, S] f32 (stride[0] = B * stride[1]).
 *   Padding slots j >= h_g of out and lse are not written.
 * Dtypes and head sizes as cpattn_ring; G * B <= 65535.
 */
cpattn_status cpattn_ulysses_anything_attention(const cpattn_tensor* q,
                                                const cpattn_tensor* k,
                                                const cpattn_tensor* v,
                                                float scale, int heads,
                                                int is_causal,
                                                cpattn_tensor* out,
                                                cpattn_tensor* lse,
                                                void* stream);

/*
 * cpattn_ring_noalloc -- cpattn_ring for callers that cannot allocate device
 * memory (a fixed device-memory budget, a memory pool that hands out no extra
 * buffers, a plugin that only receives its input and output pointers).  The
 * pages have no counterpart: it is an entry point of this library only.
 * Same arguments and results as cpattn_ring minus the workspace: the running
 * merged output and LSE live in a fixed array in the library's own device
 * memory, cpattn_ring_noalloc_max_workspace_bytes() bytes (64 MiB), which
 * every GPU that loads the library holds until the process exits.  A call
 * whose cpattn_ring_workspace_bytes() exceeds that returns
 * CPATTN_ERR_WORKSPACE (1 x 24 x 4608 x 128 fits; larger problems need
 * cpattn_ring).  The first call on a device looks the array's address up
 * (cudaGetSymbolAddress); make it before any stream capture.  All calls share
 * the array: calls whose kernels overlap on the GPU race on it.  Nothing is
 * allocated or freed by this call.
 */
cpattn_status cpattn_ring_noalloc(const cpattn_tensor* q, const cpattn_tensor* k,
                                  const cpattn_tensor* v, float scale, int ring_degree,
                                  int ring_anything, cpattn_tensor* out,
                                  cpattn_tensor* lse, void* stream);

/* Size of the fixed workspace array of cpattn_ring_noalloc, in bytes. */
size_t cpattn_ring_noalloc_max_workspace_bytes(void);

/* Human-readable name of a status code (static storage). */
const char* cpattn_status_string(cpattn_status status);

/*
 * cpattn_last_device_status -- synchronises `stream`, then reads and clears
 * the device error word that kernel-side waits set when they time out.
 * Returns CPATTN_OK, CPATTN_ERR_TIMEOUT, CPATTN_ERR_BOUNDS (check builds;
 * reported first when both happened), or CPATTN_ERR_CUDA if the
 * synchronisation itself failed.
 */
cpattn_status cpattn_last_device_status(void* stream);

/*
 * cpattn_set_wait_timeout_ns -- time limit of every kernel-side wait on an
 * mbarrier (default 2e9 ns).  Process-wide, read at each launch.
 */
void cpattn_set_wait_timeout_ns(uint64_t ns);

/*
 * Check builds.  The library can also be built with -DCPATTN_CHECK
 * (libcpattn_check.so; a debugging aid with the same ABI): every global
 * load and store of the kernels is then tested against the extent of the
 * buffer it belongs to (the bytes from the descriptor's data pointer to its
 * last element, or the workspace size); an access outside is skipped and
 * cpattn_last_device_status reports CPATTN_ERR_BOUNDS.  Nothing traps.
 * cpattn_is_check_build returns 1 in such a build, 0 otherwise.
 * cpattn_set_check_shrink (testing hook, process-wide, read at each call):
 * the extents of every OUTPUT (out, lse, the ring workspace, merge's
 * out_a/lse_a, a regroup's destination) are taken `bytes` smaller, so a
 * check build reports the writes to their last bytes and leaves those
 * bytes untouched; 0 (default) restores them.  No effect in normal builds.
 */
int cpattn_is_check_build(void);
void cpattn_set_check_shrink(int64_t bytes);

/*
 * cpattn_set_fault_injection -- testing hook for the failure path.  mode 1:
 * the TMA producer of every following attention launch issues no K/V
 * copies, so the consumers' bounded waits run out; each CTA then drains what
 * it has in flight, frees its TMEM and returns, and cpattn_last_device_status
 * reports CPATTN_ERR_TIMEOUT (outputs are not written).  mode 0 (default):
 * normal operation.  Process-wide, read at each launch.
 */
void cpattn_set_fault_injection(int mode);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H_ */
