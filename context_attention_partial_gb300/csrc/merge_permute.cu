// merge_permute.cu -- the two HBM-bound steps of the hot path.
//
// merge: LSE merge of two fp32 partials, in place into (o_a, lse_a)
//   (Diffusers "Parallelism" API, ContextParallelConfig convert_to_fp32:
//   each ring step's output and LSE are held in fp32 while they are
//   combined, to keep the combination stable; the formula follows from the
//   definition of LSE):
//     lse = max(a, b) + log1p(exp(min(a, b) - max(a, b)))
//     o   = exp(a - lse) o_a + exp(b - lse) o_b,   (0, -inf) if both empty.
//   One thread per 16-byte vector of a row; the D/4 threads of a row sit in
//   one warp, read both LSEs, synchronise, then one of them writes lse_a.
//
// permute: the Ulysses head regroup (Diffusers "Context parallelism",
//   "Ulysses Attention") as a layout copy between [B, S, H, D] and
//   [G, B, S, H/G, D].  Every (b, s, g) segment of H/G * D elements is
//   contiguous on both sides; threads walk the destination in order with
//   16-byte vectors (4 in flight per thread), or element by element when a
//   segment is not a whole number of vectors.
//   Ulysses Anything (Diffusers "Context parallelism", "Ulysses Anything
//   Attention"): H need not divide by G; groups take tensor_split head counts
//   and are padded to ceil(H/G) slots, which this copy neither writes nor
//   reads.  The unit is one head row (16-byte vectors when D bytes allow).
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"

namespace cpattn {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kPermuteThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
  const int vpr = p.head_dim / 4;                          // float4 per row
  const int64_t total = p.rows * vpr;
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31);
       base < total; base += stride) {
    const int64_t i = base + lane;
    const bool in = i < total;
    const int64_t r = in ? i / vpr : 0;
    const int cv = static_cast<int>(i - r * vpr);
    int64_t oa, ob, la, lb;
    if (p.dense) {
      oa = ob = r * p.head_dim + 4 * cv;
      la = lb = r;
    } else {
      const int64_t s = r % p.seq, bh = r / p.seq;
      const int64_t hh = bh % p.heads, bb = bh / p.heads;
      oa = bb * p.oa_s[0] + hh * p.oa_s[1] + s * p.oa_s[2] + 4 * cv;
      ob = bb * p.ob_s[0] + hh * p.ob_s[1] + s * p.ob_s[2] + 4 * cv;
      la = bb * p.la_s[0] + hh * p.la_s[1] + s * p.la_s[2];
      lb = bb * p.lb_s[0] + hh * p.lb_s[1] + s * p.lb_s[2];
    }
    float a = 0.f, b = 0.f;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
    if (in) {
      if (CPATTN_IN(p.la_span, p.l_a + la, 4, p.err)) a = p.l_a[la];
      if (CPATTN_IN(p.lb_span, p.l_b + lb, 4, p.err)) b = p.l_b[lb];
      if (CPATTN_IN(p.oa_span, p.o_a + oa, 16, p.err)) x = *reinterpret_cast<const float4*>(p.o_a + oa);
      if (CPATTN_IN(p.ob_span, p.o_b + ob, 16, p.err))
        y = __ldcs(reinterpret_cast<const float4*>(p.o_b + ob));
    }
    __syncwarp();   // every lane of the row has read lse_a before it is overwritten
    if (in) {
      float lse, wa, wb;
      if (a == -INFINITY && b == -INFINITY) {
        lse = -INFINITY;
        wa = wb = 0.f;
      } else {
        const float hi = fmaxf(a, b), lo = fminf(a, b);
        lse = hi + log1pf(expf(lo - hi));
        wa = expf(a - lse);
        wb = expf(b - lse);
      }
      const float4 o = make_float4(wa * x.x + wb * y.x, wa * x.y + wb * y.y,
                                   wa * x.z + wb * y.z, wa * x.w + wb * y.w);
      if (CPATTN_IN(p.oa_span, p.o_a + oa, 16, p.err)) __stcs(reinterpret_cast<float4*>(p.o_a + oa), o);
      if (cv == 0 && CPATTN_IN(p.la_span, p.l_a + la, 4, p.err)) p.l_a[la] = lse;
    }
  }
}

// Destination index -> source index of the same element (or vector).
//   unit: elements (or 16-byte vectors) per (b, s, g) segment.
//   dir +1: destination [G][B*S][unit], source [B*S][G][unit]
//   dir -1: destination [B*S][G][unit], source [G][B*S][unit]
template <typename Index>
__device__ __forceinline__ Index source_of(Index idx, Index unit, Index bs, Index g, int dir) {
  const Index w = idx % unit, seg = idx / unit;
  Index src_seg;
  if (dir > 0)
    src_seg = (seg % bs) * g + seg / bs;
  else
    src_seg = (seg % g) * bs + seg / g;
  return src_seg * unit + w;
}

// The tensors of one launch: grid row blockIdx.y (even regroup) or slice
// blockIdx.z (Ulysses Anything) selects one.
template <typename V>
struct PermutePtrs {
  const V* x[kMaxPermuteBatch];
  V* y[kMaxPermuteBatch];
  uint64_t x_bytes, y_bytes;   // extent of each x / y (CPATTN_CHECK builds)
  unsigned int* err;           // device error word
};

// Tensor t's pointers through fixed indices (the parameter block is not
// indexed at run time).
template <typename V>
__device__ __forceinline__ void permute_pick(const PermutePtrs<V>& p, unsigned t, const V*& x,
                                             V*& y) {
  static_assert(kMaxPermuteBatch == 4, "one select per tensor slot");
  x = t == 0 ? p.x[0] : t == 1 ? p.x[1] : t == 2 ? p.x[2] : p.x[3];
  y = t == 0 ? p.y[0] : t == 1 ? p.y[1] : t == 2 ? p.y[2] : p.y[3];
}

template <typename V, typename Index>
__global__ void __launch_bounds__(kPermuteThreads)
    permute_kernel(const PermutePtrs<V> ptrs, Index total, Index unit, Index bs, Index g,
                   int dir) {
  const V* x;
  V* y;
  permute_pick(ptrs, blockIdx.y, x, y);
  const Index stride = static_cast<Index>(gridDim.x) * blockDim.x;
  const Span xs{x, ptrs.x_bytes}, ys{y, ptrs.y_bytes};
  for (Index base = static_cast<Index>(blockIdx.x) * blockDim.x + threadIdx.x; base < total;
       base += stride * kUnroll) {
    V v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const Index idx = base + u * stride;
      const V* src = x + source_of<Index>(idx, unit, bs, g, dir);
      if (idx < total && CPATTN_IN(xs, src, sizeof(V), ptrs.err)) v[u] = __ldcs(src);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const Index idx = base + u * stride;
      if (idx < total && CPATTN_IN(ys, y + idx, sizeof(V), ptrs.err)) __stcs(y + idx, v[u]);
    }
  }
}

// Ulysses Anything regroup.  Grid row blockIdx.y is one head h of the
// [B, S, H, D] side; its group g and slot j follow from tensor_split (the
// first r = H mod G groups hold q + 1 heads, the others q) once per block.
// The block's threads then walk that head's B*S rows of `row` units
// (16-byte vectors or elements): unit w of token tok sits at
// (tok * H + h) * row + w on the flat side and at
// ((g * bs + tok) * hm + j) * row + w on the grouped side, whose groups are
// padded to hm = ceil(H/G) slots.
template <typename V, typename Index, bool POW2>
__global__ void __launch_bounds__(kPermuteThreads)
    permute_anything_kernel(const PermutePtrs<V> ptrs, Index per_head, Index row, int row_shift,
                            Index heads, Index hm, Index bs, Index q, Index r, int dir) {
  const V* x;
  V* y;
  permute_pick(ptrs, blockIdx.z, x, y);
  const Index h = blockIdx.y;
  const Index big = r * (q + 1);
  Index g, j;
  if (h < big) {
    g = h / (q + 1);
    j = h - g * (q + 1);
  } else {   // only reached when q > 0
    g = r + (h - big) / q;
    j = h - big - (g - r) * q;
  }
  const Span xs{x, ptrs.x_bytes}, ys{y, ptrs.y_bytes};
  const Index flat_base = h * row, flat_step = heads * row;
  const Index grouped_base = (g * bs * hm + j) * row, grouped_step = hm * row;
  const Index stride = static_cast<Index>(gridDim.x) * blockDim.x;
  for (Index base = static_cast<Index>(blockIdx.x) * blockDim.x + threadIdx.x; base < per_head;
       base += stride * kUnroll) {
    V v[kUnroll];
    Index src[kUnroll], dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const Index i = base + u * stride;
      const Index tok = POW2 ? (i >> row_shift) : (i / row);
      const Index w = i - tok * row;
      const Index flat = flat_base + tok * flat_step + w;
      const Index grouped = grouped_base + tok * grouped_step + w;
      src[u] = dir > 0 ? flat : grouped;
      dst[u] = dir > 0 ? grouped : flat;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (base + u * stride < per_head && CPATTN_IN(xs, x + src[u], sizeof(V), ptrs.err))
        v[u] = __ldcs(x + src[u]);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (base + u * stride < per_head && CPATTN_IN(ys, y + dst[u], sizeof(V), ptrs.err))
        __stcs(y + dst[u], v[u]);
  }
}

template <typename V>
PermutePtrs<V> permute_ptrs(const PermuteParams& p) {
  PermutePtrs<V> ptrs{};
  for (int i = 0; i < p.n; ++i) {
    ptrs.x[i] = static_cast<const V*>(p.x[i]);
    ptrs.y[i] = static_cast<V*>(p.y[i]);
  }
  ptrs.x_bytes = p.x_bytes;
  ptrs.y_bytes = p.y_bytes;
  ptrs.err = p.err;
  return ptrs;
}

template <typename V>
cudaError_t launch_permute_typed(const PermuteParams& p, int64_t total, int64_t unit,
                                 cudaStream_t stream) {
  const int64_t bs = p.batch * p.seq;
  const int64_t want = (total + kPermuteThreads * kUnroll - 1) / (kPermuteThreads * kUnroll);
  // about 32 blocks of 256 threads per SM in total (8 resident at a time),
  // shared by the tensors: the finer split evens out the tail of a batch
  // (three tensors: 29.8 us with 8, 27.0 us with 32; one tensor unchanged)
  const int64_t cap = (static_cast<int64_t>(sm_count()) * 32 + p.n - 1) / p.n;
  const int blocks = static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
  const dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(p.n));
  const PermutePtrs<V> ptrs = permute_ptrs<V>(p);
  if (total + static_cast<int64_t>(blocks) * kPermuteThreads * kUnroll < (int64_t(1) << 31))
    permute_kernel<V, uint32_t><<<grid, kPermuteThreads, 0, stream>>>(
        ptrs, static_cast<uint32_t>(total), static_cast<uint32_t>(unit),
        static_cast<uint32_t>(bs), static_cast<uint32_t>(p.degree), p.dir);
  else
    permute_kernel<V, uint64_t><<<grid, kPermuteThreads, 0, stream>>>(
        ptrs, static_cast<uint64_t>(total), static_cast<uint64_t>(unit),
        static_cast<uint64_t>(bs), static_cast<uint64_t>(p.degree), p.dir);
  return cudaGetLastError();
}

template <typename V, typename Index>
cudaError_t launch_permute_anything_index(const PermuteParams& p, int64_t per_head, int64_t row,
                                          dim3 grid, cudaStream_t stream) {
  const int64_t bs = p.batch * p.seq;
  const int64_t hm = (p.heads + p.degree - 1) / p.degree;
  const int64_t q = p.heads / p.degree, r = p.heads % p.degree;
  int shift = 0;
  while ((int64_t(1) << shift) < row) ++shift;
  const PermutePtrs<V> ptrs = permute_ptrs<V>(p);
  if ((int64_t(1) << shift) == row)
    permute_anything_kernel<V, Index, true><<<grid, kPermuteThreads, 0, stream>>>(
        ptrs, static_cast<Index>(per_head), static_cast<Index>(row), shift,
        static_cast<Index>(p.heads), static_cast<Index>(hm), static_cast<Index>(bs),
        static_cast<Index>(q), static_cast<Index>(r), p.dir);
  else
    permute_anything_kernel<V, Index, false><<<grid, kPermuteThreads, 0, stream>>>(
        ptrs, static_cast<Index>(per_head), static_cast<Index>(row), shift,
        static_cast<Index>(p.heads), static_cast<Index>(hm), static_cast<Index>(bs),
        static_cast<Index>(q), static_cast<Index>(r), p.dir);
  return cudaGetLastError();
}

template <typename V>
cudaError_t launch_permute_anything_typed(const PermuteParams& p, int64_t row,
                                          cudaStream_t stream) {
  const int64_t bs = p.batch * p.seq;
  const int64_t hm = (p.heads + p.degree - 1) / p.degree;
  const int64_t per_head = bs * row;   // units of one head
  // about 32 blocks of 256 threads per SM in total, spread over the heads
  // and the tensors (as for the even regroup)
  const int64_t cap = static_cast<int64_t>(sm_count()) * 32;
  int64_t bx = (cap + p.heads * p.n - 1) / (p.heads * p.n);
  const int64_t want = (per_head + kPermuteThreads * kUnroll - 1) / (kPermuteThreads * kUnroll);
  if (bx > want) bx = want;
  if (bx < 1) bx = 1;
  if (p.heads > 65535) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(p.heads),
                  static_cast<unsigned>(p.n));
  // largest index on either side, and the loop counter's reach
  const int64_t flat_total = bs * p.heads * row;
  const int64_t grouped_total = p.degree * bs * hm * row;
  const int64_t reach = per_head + bx * kPermuteThreads * kUnroll;
  const int64_t lim = int64_t(1) << 31;
  if (flat_total < lim && grouped_total < lim && reach < lim)
    return launch_permute_anything_index<V, uint32_t>(p, per_head, row, grid, stream);
  return launch_permute_anything_index<V, uint64_t>(p, per_head, row, grid, stream);
}

}  // namespace

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;   // GB300's count
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 152;
  return n;
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
  const int64_t total = p.rows * (p.head_dim / 4);
  if (total == 0) return cudaSuccess;
  const int64_t want = (total + kMergeThreads - 1) / kMergeThreads;
  // about 32 blocks of 256 threads per SM in total (8 resident at a time):
  // FLUX shape 28.7-29.0 us with 8, 27.3-27.4 us with 32
  const int64_t cap = static_cast<int64_t>(sm_count()) * 32;
  const int blocks = static_cast<int>(want < cap ? want : cap);
  merge_kernel<<<blocks, kMergeThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

// every tensor's base 16-byte aligned (the vector paths)
static bool all_aligned16(const PermuteParams& p) {
  for (int i = 0; i < p.n; ++i)
    if (reinterpret_cast<uintptr_t>(p.x[i]) % 16 != 0 || reinterpret_cast<uintptr_t>(p.y[i]) % 16 != 0)
      return false;
  return true;
}

cudaError_t launch_permute(const PermuteParams& p, cudaStream_t stream) {
  if (p.n < 1 || p.n > kMaxPermuteBatch) return cudaErrorInvalidValue;
  const int64_t seg_elems = (p.heads / p.degree) * p.head_dim;
  const int64_t total_elems = p.batch * p.seq * p.heads * p.head_dim;
  if (total_elems == 0) return cudaSuccess;
  const int64_t seg_bytes = seg_elems * p.elem_bytes;
  const bool vec = seg_bytes % 16 == 0 && all_aligned16(p);
  if (vec)
    return launch_permute_typed<uint4>(p, total_elems * p.elem_bytes / 16, seg_bytes / 16, stream);
  if (p.elem_bytes == 2)
    return launch_permute_typed<unsigned short>(p, total_elems, seg_elems, stream);
  if (p.elem_bytes == 4)
    return launch_permute_typed<unsigned int>(p, total_elems, seg_elems, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_permute_anything(const PermuteParams& p, cudaStream_t stream) {
  if (p.n < 1 || p.n > kMaxPermuteBatch) return cudaErrorInvalidValue;
  const int64_t total_elems = p.batch * p.seq * p.heads * p.head_dim;
  if (total_elems == 0) return cudaSuccess;
  const int64_t row_bytes = p.head_dim * p.elem_bytes;
  const bool vec = row_bytes % 16 == 0 && all_aligned16(p);
  if (vec) return launch_permute_anything_typed<uint4>(p, row_bytes / 16, stream);
  if (p.elem_bytes == 2) return launch_permute_anything_typed<unsigned short>(p, p.head_dim, stream);
  if (p.elem_bytes == 4) return launch_permute_anything_typed<unsigned int>(p, p.head_dim, stream);
  return cudaErrorInvalidValue;
}

}  // namespace cpattn
