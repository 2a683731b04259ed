// cpattn_api.cu -- the C ABI of libcpattn.so: argument validation, the ring
// chunk partition, TMA descriptor encoding and kernel dispatch.  Host code
// only; every step of the computation runs in the kernels.
//
// Validation rules (page title, section):
//   Diffusers "Context parallelism", variants table: Ring needs the sequence
//   length divisible by ring_degree, Ulysses needs the head count divisible
//   by ulysses_degree; "Ring Anything Attention" lifts the first rule and
//   takes no mask.  diffusers _modeling_parallel.py ContextParallelConfig:
//   degrees must be >= 1.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace {

using cpattn::InDtype;

std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<int> g_fault_skip_kv{0};
std::atomic<long long> g_check_shrink{0};   // testing: output extents shrunk by this many bytes

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

int elem_bytes(int32_t dtype) { return dtype == CPATTN_BF16 ? 2 : 4; }

bool dtype_known(int32_t dtype) { return dtype == CPATTN_F32 || dtype == CPATTN_BF16; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Inner stride 1; other strides of extent>1 dims are multiples of 16 bytes
// and non-negative; data 16-byte aligned.
bool layout_ok(const cpattn_tensor* t) {
  if (t->ndim < 1) return false;
  if (t->shape[t->ndim - 1] > 1 && t->stride[t->ndim - 1] != 1) return false;
  if (!aligned16(t->data)) return false;
  const int eb = elem_bytes(t->dtype);
  for (int i = 0; i < t->ndim - 1; ++i) {
    if (t->stride[i] < 0) return false;
    if (t->shape[i] > 1 && (t->stride[i] * eb) % 16 != 0) return false;
  }
  return true;
}

bool shape_ok(const cpattn_tensor* t, int ndim) {
  if (t->ndim != ndim) return false;
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0) return false;
  return true;
}

// Bytes from a tensor's data pointer to the end of its last element (0 if
// it has none), less `shrink` (the bounds-check testing hook).
uint64_t extent_bytes(const cpattn_tensor* t, long long shrink = 0) {
  int64_t last = 0;
  for (int i = 0; i < t->ndim; ++i) {
    if (t->shape[i] == 0) return 0;
    last += (t->shape[i] - 1) * t->stride[i];
  }
  const int64_t bytes = (last + 1) * elem_bytes(t->dtype) - shrink;
  return bytes > 0 ? static_cast<uint64_t>(bytes) : 0;
}

bool contiguous(const cpattn_tensor* t) {
  int64_t expect = 1;
  for (int i = t->ndim - 1; i >= 0; --i) {
    if (t->shape[i] > 1 && t->stride[i] != expect) return false;
    expect *= t->shape[i];
  }
  return true;
}

// Stride of a dimension as the TMA map sees it: dims of extent 1 get the
// dense stride so that every stride stays a positive multiple of 16 bytes.
int64_t tma_stride(const cpattn_tensor* t, int dim, int64_t dense) {
  return t->shape[dim] > 1 ? t->stride[dim] : dense;
}

// 4-D map over a [B, H, S, D] tensor: dims (D, S, H, B), box (128 bytes of D,
// box_rows rows, 1, 1), 128-byte swizzle, zero fill out of bounds.
cpattn_status make_tmap(CUtensorMap* m, const cpattn_tensor* t, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return CPATTN_ERR_CUDA;
  const int eb = elem_bytes(t->dtype);
  const int64_t B = t->shape[0], H = t->shape[1], S = t->shape[2], D = t->shape[3];
  const int64_t ss = tma_stride(t, 2, D);
  const int64_t sh = tma_stride(t, 1, ss * S);
  const int64_t sb = tma_stride(t, 0, sh * H);
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)(ss * eb), (cuuint64_t)(sh * eb),
                                 (cuuint64_t)(sb * eb)};
  const cuuint32_t box[4] = {(cuuint32_t)(128 / eb), (cuuint32_t)box_rows, 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUtensorMapDataType dt =
      t->dtype == CPATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const CUresult r = enc(m, dt, 4, t->data, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CPATTN_OK : CPATTN_ERR_CUDA;
}

// Key partition of the ring (plain: S/R each; Ring Anything: the first
// S mod R chunks one longer).
cpattn_status ring_partition(int64_t s_kv, int ring_degree, int ring_anything, int* start) {
  if (ring_degree < 1) return CPATTN_ERR_SHAPE;
  if (ring_degree > CPATTN_MAX_RING_DEGREE) return CPATTN_ERR_UNSUPPORTED;
  if (!ring_anything && s_kv % ring_degree != 0) return CPATTN_ERR_DIVISIBILITY;
  if (ring_anything && ring_degree > s_kv) return CPATTN_ERR_SHAPE;
  const int64_t len = s_kv / ring_degree, longer = s_kv % ring_degree;
  int64_t pos = 0;
  for (int c = 0; c < ring_degree; ++c) {
    start[c] = static_cast<int>(pos);
    pos += len + (c < longer ? 1 : 0);
  }
  start[ring_degree] = static_cast<int>(pos);
  return CPATTN_OK;
}

size_t workspace_bytes_for(int64_t B, int64_t H, int64_t S, int64_t D, int ring_degree) {
  if (ring_degree <= 1) return 0;
  // [B*H*ceil(S/128) query tiles][128 rows][D + 1] floats
  const int64_t rows = B * H * ((S + 127) / 128) * 128;
  return static_cast<size_t>(rows) * static_cast<size_t>(D + 1) * sizeof(float);
}

cpattn_status check_qkv(const cpattn_tensor* q, const cpattn_tensor* k, const cpattn_tensor* v) {
  if (!q || !k || !v) return CPATTN_ERR_NULL;
  if (!dtype_known(q->dtype) || k->dtype != q->dtype || v->dtype != q->dtype)
    return CPATTN_ERR_DTYPE;
  if (!shape_ok(q, 4) || !shape_ok(k, 4) || !shape_ok(v, 4)) return CPATTN_ERR_SHAPE;
  for (int i = 0; i < 4; ++i)
    if (k->shape[i] != v->shape[i]) return CPATTN_ERR_SHAPE;
  if (q->shape[0] != k->shape[0] || q->shape[1] != k->shape[1] || q->shape[3] != k->shape[3])
    return CPATTN_ERR_SHAPE;
  const bool empty_q = q->shape[0] == 0 || q->shape[1] == 0 || q->shape[2] == 0;
  if (!empty_q && k->shape[2] == 0) return CPATTN_ERR_SHAPE;
  if (!empty_q && (!q->data || !k->data || !v->data)) return CPATTN_ERR_NULL;
  return CPATTN_OK;
}

cpattn_status run_attention(const cpattn_tensor* q, const cpattn_tensor* k,
                            const cpattn_tensor* v, float scale, int ring_degree,
                            int ring_anything, cpattn_tensor* out, cpattn_tensor* lse,
                            void* workspace, size_t workspace_bytes, bool out_f32,
                            bool causal, cudaStream_t stream, int group_count = 0,
                            int group_heads = 0) {
  cpattn_status st = check_qkv(q, k, v);
  if (st != CPATTN_OK) return st;
  if (!out || !lse) return CPATTN_ERR_NULL;
  const int32_t want_out = out_f32 ? CPATTN_F32 : q->dtype;
  if (out->dtype != want_out || lse->dtype != CPATTN_F32) return CPATTN_ERR_DTYPE;
  if (!shape_ok(out, 4) || !shape_ok(lse, 3)) return CPATTN_ERR_SHAPE;
  for (int i = 0; i < 4; ++i)
    if (out->shape[i] != q->shape[i]) return CPATTN_ERR_SHAPE;
  for (int i = 0; i < 3; ++i)
    if (lse->shape[i] != q->shape[i]) return CPATTN_ERR_SHAPE;
  const int64_t B = q->shape[0], H = q->shape[1], S_q = q->shape[2], S_kv = k->shape[2],
                D = q->shape[3];
  int chunk_start[CPATTN_MAX_RING_DEGREE + 1];
  if (ring_degree < 1) return CPATTN_ERR_SHAPE;
  if (ring_degree > CPATTN_MAX_RING_DEGREE) return CPATTN_ERR_UNSUPPORTED;
  const bool empty_q = B == 0 || H == 0 || S_q == 0;
  if (!empty_q) {
    st = ring_partition(S_kv, ring_degree, ring_anything, chunk_start);
    if (st != CPATTN_OK) return st;
  } else if (!ring_anything && S_kv % ring_degree != 0) {
    return CPATTN_ERR_DIVISIBILITY;
  }
  const bool supported = D == 64 || D == 128;
  if (!supported) return CPATTN_ERR_UNSUPPORTED;
  if (B > 65535 || H > 65535 || S_q > (int64_t(1) << 30) || S_kv > (int64_t(1) << 30))
    return CPATTN_ERR_UNSUPPORTED;
  if (empty_q) return CPATTN_OK;
  if (!out->data || !lse->data) return CPATTN_ERR_NULL;
  if (!layout_ok(q) || !layout_ok(k) || !layout_ok(v) || !layout_ok(out)) return CPATTN_ERR_LAYOUT;
  if (lse->shape[2] > 1 && lse->stride[2] != 1) return CPATTN_ERR_LAYOUT;
  if ((reinterpret_cast<uintptr_t>(lse->data) & 3u) != 0) return CPATTN_ERR_LAYOUT;
  const size_t need = workspace_bytes_for(B, H, S_q, D, ring_degree);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
    return CPATTN_ERR_WORKSPACE;

  const InDtype dt = q->dtype == CPATTN_BF16 ? InDtype::BF16 : InDtype::F32;
  const int kv_rows = cpattn::attn_kv_tile_rows(dt, static_cast<int>(D));
  CUtensorMap tm_q, tm_k, tm_v;
  if ((st = make_tmap(&tm_q, q, 128)) != CPATTN_OK) return st;
  if ((st = make_tmap(&tm_k, k, kv_rows)) != CPATTN_OK) return st;
  if ((st = make_tmap(&tm_v, v, kv_rows)) != CPATTN_OK) return st;

  cpattn::AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.out = out->data;
  p.out_sb = out->stride[0];
  p.out_sh = out->stride[1];
  p.out_ss = out->stride[2];
  p.lse = static_cast<float*>(lse->data);
  p.lse_sb = lse->stride[0];
  p.lse_sh = lse->stride[1];
  p.lse_ss = lse->stride[2];
  if (need > 0) {
    p.ws_o = static_cast<float*>(workspace);
    p.ws_lse = p.ws_o + B * H * ((S_q + 127) / 128) * 128 * D;
  }
  const long long shrink = g_check_shrink.load();
  p.out_span = {out->data, extent_bytes(out, shrink)};
  p.lse_span = {lse->data, extent_bytes(lse, shrink)};
  p.ws_span = {workspace, need > static_cast<size_t>(shrink) ? need - shrink : 0};
  p.batch = static_cast<int>(B);
  p.heads = static_cast<int>(H);
  p.s_q = static_cast<int>(S_q);
  p.s_kv = static_cast<int>(S_kv);
  if (!(scale > 0.f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt(static_cast<float>(D));
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.ring_degree = ring_degree;
  p.out_f32 = out->dtype == CPATTN_F32 ? 1 : 0;
  p.timeout_ns = g_timeout_ns.load();
  p.fault_skip_kv = g_fault_skip_kv.load();
  p.causal = causal ? 1 : 0;
  p.group_count = group_count;
  p.group_heads = group_heads;
  for (int c = 0; c <= ring_degree; ++c) p.chunk_start[c] = chunk_start[c];
  p.n_tiles_all = 0;
  for (int c = 0; c < ring_degree; ++c)
    p.n_tiles_all += (chunk_start[c + 1] - chunk_start[c] + kv_rows - 1) / kv_rows;
  const cudaError_t e =
      cpattn::launch_attention(dt, static_cast<int>(D), tm_q, tm_k, tm_v, p, stream);
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

// One Ulysses regroup pair x -> y (even: [B,S,H,D] <-> [G,B,S,H/G,D];
// Ulysses Anything: [B,S,H,D] <-> [G,B,S,ceil(H/G),D]).  Fills dims with
// (B, S, H, D) and bytes with the sizes of x and y.
cpattn_status permute_pair_check(const cpattn_tensor* x, const cpattn_tensor* y, int degree,
                                 int dir, bool anything, int64_t* dims, uintptr_t* xbytes,
                                 uintptr_t* ybytes) {
  if (!x || !y) return CPATTN_ERR_NULL;
  if (!dtype_known(x->dtype) || y->dtype != x->dtype) return CPATTN_ERR_DTYPE;
  if (dir != 1 && dir != -1) return CPATTN_ERR_SHAPE;
  if (degree < 1) return CPATTN_ERR_SHAPE;
  const cpattn_tensor* flat = dir == 1 ? x : y;      // [B, S, H, D]
  const cpattn_tensor* grouped = dir == 1 ? y : x;   // [G, B, S, H/G or ceil(H/G), D]
  if (!shape_ok(flat, 4) || !shape_ok(grouped, 5)) return CPATTN_ERR_SHAPE;
  const int64_t B = flat->shape[0], S = flat->shape[1], H = flat->shape[2], D = flat->shape[3];
  if (!anything && H % degree != 0) return CPATTN_ERR_DIVISIBILITY;
  const int64_t hg = anything ? (H + degree - 1) / degree : H / degree;
  if (grouped->shape[0] != degree || grouped->shape[1] != B || grouped->shape[2] != S ||
      grouped->shape[3] != hg || grouped->shape[4] != D)
    return CPATTN_ERR_SHAPE;
  dims[0] = B;
  dims[1] = S;
  dims[2] = H;
  dims[3] = D;
  const int eb = elem_bytes(x->dtype);
  const uintptr_t flat_bytes = static_cast<uintptr_t>(B * S * H * D * eb);
  const uintptr_t grouped_bytes = static_cast<uintptr_t>(degree * B * S * hg * D * eb);
  *xbytes = dir == 1 ? flat_bytes : grouped_bytes;
  *ybytes = dir == 1 ? grouped_bytes : flat_bytes;
  if (B * S * H * D == 0) return CPATTN_OK;
  if (!x->data || !y->data) return CPATTN_ERR_NULL;
  if (!contiguous(x) || !contiguous(y)) return CPATTN_ERR_LAYOUT;
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x->data), ya = reinterpret_cast<uintptr_t>(y->data);
  if (xa % eb || ya % eb) return CPATTN_ERR_LAYOUT;
  return CPATTN_OK;
}

bool overlaps(const void* a, uintptr_t an, const void* b, uintptr_t bn) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bn && y < x + an;
}

// n regroups of one shape and dtype in one launch; no output may overlap
// any buffer of the call.
cpattn_status permute_batch(int n, const cpattn_tensor* x, int degree, int dir, cpattn_tensor* y,
                            bool anything, cudaStream_t stream) {
  if (n < 1 || n > cpattn::kMaxPermuteBatch) return CPATTN_ERR_SHAPE;
  if (!x || !y) return CPATTN_ERR_NULL;
  int64_t dims[4] = {0, 0, 0, 0};
  uintptr_t xb = 0, yb = 0;
  for (int i = 0; i < n; ++i) {
    int64_t d[4];
    uintptr_t xbi = 0, ybi = 0;
    const cpattn_status st = permute_pair_check(&x[i], &y[i], degree, dir, anything, d, &xbi, &ybi);
    if (st != CPATTN_OK) return st;
    if (i == 0) {
      for (int j = 0; j < 4; ++j) dims[j] = d[j];
      xb = xbi;
      yb = ybi;
    } else {
      if (x[i].dtype != x[0].dtype) return CPATTN_ERR_DTYPE;
      for (int j = 0; j < 4; ++j)
        if (d[j] != dims[j]) return CPATTN_ERR_SHAPE;
    }
  }
  if (dims[0] * dims[1] * dims[2] * dims[3] == 0) return CPATTN_OK;
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j)
      if (overlaps(y[i].data, yb, x[j].data, xb) || (i != j && overlaps(y[i].data, yb, y[j].data, yb)))
        return CPATTN_ERR_LAYOUT;
  cpattn::PermuteParams p;
  p.n = n;
  for (int i = 0; i < n; ++i) {
    p.x[i] = x[i].data;
    p.y[i] = y[i].data;
  }
  p.batch = dims[0];
  p.seq = dims[1];
  p.heads = dims[2];
  p.head_dim = dims[3];
  p.degree = degree;
  p.dir = dir;
  p.elem_bytes = elem_bytes(x[0].dtype);
  const long long shrink = g_check_shrink.load();
  p.x_bytes = xb;
  p.y_bytes = yb > static_cast<uintptr_t>(shrink) ? yb - shrink : 0;
  p.err = cpattn::device_error_word();
  const cudaError_t e =
      anything ? cpattn::launch_permute_anything(p, stream) : cpattn::launch_permute(p, stream);
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

cpattn_status cpattn_partial(const cpattn_tensor* q, const cpattn_tensor* k,
                             const cpattn_tensor* v, float scale, cpattn_tensor* out,
                             cpattn_tensor* lse, void* stream) {
  return run_attention(q, k, v, scale, 1, 0, out, lse, nullptr, 0, true, false,
                       static_cast<cudaStream_t>(stream));
}

cpattn_status cpattn_ring(const cpattn_tensor* q, const cpattn_tensor* k, const cpattn_tensor* v,
                          float scale, int ring_degree, int ring_anything, cpattn_tensor* out,
                          cpattn_tensor* lse, void* workspace, size_t workspace_bytes,
                          void* stream) {
  return run_attention(q, k, v, scale, ring_degree, ring_anything, out, lse, workspace,
                       workspace_bytes, false, false, static_cast<cudaStream_t>(stream));
}

cpattn_status cpattn_ring_causal(const cpattn_tensor* q, const cpattn_tensor* k,
                                 const cpattn_tensor* v, float scale, int ring_degree,
                                 int ring_anything, cpattn_tensor* out, cpattn_tensor* lse,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  return run_attention(q, k, v, scale, ring_degree, ring_anything, out, lse, workspace,
                       workspace_bytes, false, true, static_cast<cudaStream_t>(stream));
}

size_t cpattn_ring_workspace_bytes(const cpattn_tensor* q, int ring_degree) {
  if (!q || q->ndim != 4) return 0;
  for (int i = 0; i < 4; ++i)
    if (q->shape[i] < 0) return 0;
  return workspace_bytes_for(q->shape[0], q->shape[1], q->shape[2], q->shape[3], ring_degree);
}

cpattn_status cpattn_merge(cpattn_tensor* out_a, cpattn_tensor* lse_a, const cpattn_tensor* out_b,
                           const cpattn_tensor* lse_b, void* stream) {
  if (!out_a || !lse_a || !out_b || !lse_b) return CPATTN_ERR_NULL;
  if (out_a->dtype != CPATTN_F32 || out_b->dtype != CPATTN_F32 || lse_a->dtype != CPATTN_F32 ||
      lse_b->dtype != CPATTN_F32)
    return CPATTN_ERR_DTYPE;
  if (!shape_ok(out_a, 4) || !shape_ok(out_b, 4) || !shape_ok(lse_a, 3) || !shape_ok(lse_b, 3))
    return CPATTN_ERR_SHAPE;
  for (int i = 0; i < 4; ++i)
    if (out_a->shape[i] != out_b->shape[i]) return CPATTN_ERR_SHAPE;
  for (int i = 0; i < 3; ++i)
    if (lse_a->shape[i] != out_a->shape[i] || lse_b->shape[i] != out_a->shape[i])
      return CPATTN_ERR_SHAPE;
  const int64_t B = out_a->shape[0], H = out_a->shape[1], S = out_a->shape[2],
                D = out_a->shape[3];
  if (D != 4 && D != 8 && D != 16 && D != 32 && D != 64 && D != 128)
    return CPATTN_ERR_UNSUPPORTED;
  if (B > 65535 || H > 65535 || S > (int64_t(1) << 31)) return CPATTN_ERR_UNSUPPORTED;
  if (B * H * S == 0) return CPATTN_OK;
  if (!out_a->data || !lse_a->data || !out_b->data || !lse_b->data) return CPATTN_ERR_NULL;
  if (!layout_ok(out_a) || !layout_ok(out_b)) return CPATTN_ERR_LAYOUT;
  if ((lse_a->shape[2] > 1 && lse_a->stride[2] != 1) ||
      (lse_b->shape[2] > 1 && lse_b->stride[2] != 1))
    return CPATTN_ERR_LAYOUT;
  if ((reinterpret_cast<uintptr_t>(lse_a->data) & 3u) || (reinterpret_cast<uintptr_t>(lse_b->data) & 3u))
    return CPATTN_ERR_LAYOUT;
  cpattn::MergeParams p;
  p.o_a = static_cast<float*>(out_a->data);
  p.l_a = static_cast<float*>(lse_a->data);
  p.o_b = static_cast<const float*>(out_b->data);
  p.l_b = static_cast<const float*>(lse_b->data);
  p.rows = B * H * S;
  p.head_dim = static_cast<int>(D);
  p.heads = static_cast<int>(H);
  p.seq = static_cast<int>(S);
  for (int i = 0; i < 3; ++i) {
    p.oa_s[i] = out_a->stride[i];
    p.ob_s[i] = out_b->stride[i];
    p.la_s[i] = lse_a->stride[i];
    p.lb_s[i] = lse_b->stride[i];
  }
  p.dense = contiguous(out_a) && contiguous(out_b) && contiguous(lse_a) && contiguous(lse_b);
  const long long shrink = g_check_shrink.load();
  p.oa_span = {out_a->data, extent_bytes(out_a, shrink)};
  p.la_span = {lse_a->data, extent_bytes(lse_a, shrink)};
  p.ob_span = {out_b->data, extent_bytes(out_b)};
  p.lb_span = {lse_b->data, extent_bytes(lse_b)};
  p.err = cpattn::device_error_word();
  const cudaError_t e = cpattn::launch_merge(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

cpattn_status cpattn_ulysses_permute_batch(int n, const cpattn_tensor* x, int degree, int dir,
                                           cpattn_tensor* y, void* stream) {
  return permute_batch(n, x, degree, dir, y, false, static_cast<cudaStream_t>(stream));
}

cpattn_status cpattn_ulysses_permute(const cpattn_tensor* x, int degree, int dir, cpattn_tensor* y,
                                     void* stream) {
  return permute_batch(1, x, degree, dir, y, false, static_cast<cudaStream_t>(stream));
}

cpattn_status cpattn_ulysses_anything_permute_batch(int n, const cpattn_tensor* x, int degree,
                                                    int dir, cpattn_tensor* y, void* stream) {
  return permute_batch(n, x, degree, dir, y, true, static_cast<cudaStream_t>(stream));
}

cpattn_status cpattn_ulysses_anything_permute(const cpattn_tensor* x, int degree, int dir,
                                              cpattn_tensor* y, void* stream) {
  return permute_batch(1, x, degree, dir, y, true, static_cast<cudaStream_t>(stream));
}

cpattn_status cpattn_ulysses_anything_attention(const cpattn_tensor* q, const cpattn_tensor* k,
                                                const cpattn_tensor* v, float scale, int heads,
                                                int is_causal, cpattn_tensor* out,
                                                cpattn_tensor* lse, void* stream) {
  if (!q || !k || !v || !out || !lse) return CPATTN_ERR_NULL;
  const cpattn_tensor* five[4] = {q, k, v, out};
  for (const cpattn_tensor* t : five)
    if (!shape_ok(t, 5)) return CPATTN_ERR_SHAPE;
  if (!shape_ok(lse, 4)) return CPATTN_ERR_SHAPE;
  const int64_t G = q->shape[0], B = q->shape[1], S = q->shape[2], hm = q->shape[3];
  if (heads < 1 || G < 1 || hm != (heads + G - 1) / G) return CPATTN_ERR_SHAPE;
  for (const cpattn_tensor* t : five)
    for (int i = 0; i < 5; ++i)
      if (t->shape[i] != q->shape[i]) return CPATTN_ERR_SHAPE;
  if (lse->shape[0] != G || lse->shape[1] != B || lse->shape[2] != hm || lse->shape[3] != S)
    return CPATTN_ERR_SHAPE;
  // the (group, batch) axes merge into one batch axis of the 4-D view
  for (const cpattn_tensor* t : five)
    if (G > 1 && B > 0 && t->stride[0] != B * t->stride[1]) return CPATTN_ERR_LAYOUT;
  if (G > 1 && B > 0 && lse->stride[0] != B * lse->stride[1]) return CPATTN_ERR_LAYOUT;
  if (G * B > 65535) return CPATTN_ERR_UNSUPPORTED;
  // view [G*B, hm, S, D] (strides: batch, head, token, feature)
  auto view = [&](const cpattn_tensor* t) {
    cpattn_tensor w = *t;
    w.ndim = 4;
    w.shape[0] = G * B; w.shape[1] = hm; w.shape[2] = S; w.shape[3] = t->shape[4];
    w.stride[0] = t->stride[1]; w.stride[1] = t->stride[3]; w.stride[2] = t->stride[2];
    w.stride[3] = t->stride[4];
    w.stride[4] = 0; w.shape[4] = 0;
    return w;
  };
  cpattn_tensor vq = view(q), vk = view(k), vv = view(v), vo = view(out);
  cpattn_tensor vl = *lse;
  vl.ndim = 3;
  vl.shape[0] = G * B; vl.shape[1] = hm; vl.shape[2] = S;
  vl.stride[0] = lse->stride[1]; vl.stride[1] = lse->stride[2]; vl.stride[2] = lse->stride[3];
  vl.shape[3] = vl.shape[4] = 0; vl.stride[3] = vl.stride[4] = 0;
  return run_attention(&vq, &vk, &vv, scale, 1, 0, &vo, &vl, nullptr, 0, false, is_causal != 0,
                       static_cast<cudaStream_t>(stream), static_cast<int>(G), heads);
}

const char* cpattn_status_string(cpattn_status status) {
  switch (status) {
    case CPATTN_OK: return "ok";
    case CPATTN_ERR_NULL: return "null pointer";
    case CPATTN_ERR_DTYPE: return "dtype not allowed";
    case CPATTN_ERR_SHAPE: return "inconsistent shape";
    case CPATTN_ERR_DIVISIBILITY: return "length not divisible by the degree";
    case CPATTN_ERR_LAYOUT: return "layout: inner stride must be 1, strides and data 16-byte aligned";
    case CPATTN_ERR_UNSUPPORTED: return "unsupported size or head dimension";
    case CPATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case CPATTN_ERR_CUDA: return "CUDA runtime error";
    case CPATTN_ERR_TIMEOUT: return "device-side wait timed out";
    case CPATTN_ERR_BOUNDS: return "device-side bounds check failed (check build)";
  }
  return "unknown status";
}

cpattn_status cpattn_last_device_status(void* stream) {
  unsigned int v = 0;
  const cudaError_t e = cpattn::read_and_clear_device_error(&v, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return CPATTN_ERR_CUDA;
  if (v & cpattn::kErrBounds) return CPATTN_ERR_BOUNDS;
  return v ? CPATTN_ERR_TIMEOUT : CPATTN_OK;
}

void cpattn_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1); }

void cpattn_set_fault_injection(int mode) { g_fault_skip_kv.store(mode == 1 ? 1 : 0); }

void cpattn_set_check_shrink(int64_t bytes) { g_check_shrink.store(bytes > 0 ? bytes : 0); }

int cpattn_is_check_build(void) {
#ifdef CPATTN_CHECK
  return 1;
#else
  return 0;
#endif
}

}  // extern "C"
