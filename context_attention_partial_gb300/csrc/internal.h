// internal.h -- declarations shared by the translation units of libcpattn.so
// (not part of the public ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/cpattn.h"
#include "check.cuh"

namespace cpattn {

// Parameters of one attention launch (ring or single partial).
struct AttnParams {
  void* out;             // [B, H, S_q, D], f32 or the input dtype
  int64_t out_sb, out_sh, out_ss;
  float* lse;            // [B, H, S_q] f32
  int64_t lse_sb, lse_sh, lse_ss;
  // running merged partial (ring_degree > 1), per 128-row query tile t of
  // the B*H*ceil(S_q/128) tiles: ws_o f32 [t][D/4][128 rows][4] (a warp's
  // float4 accesses at one column group are 512 contiguous bytes), ws_lse
  // f32 [t][128 rows]
  float* ws_o;
  float* ws_lse;
  int batch, heads, s_q, s_kv;
  float scale_log2;      // softmax scale times log2(e)
  int ring_degree;
  int out_f32;           // 1: out is f32, 0: out has the input dtype (bf16)
  unsigned long long timeout_ns;
  int fault_skip_kv;     // testing: the producer issues no K/V loads
  int causal;            // 1: query i attends keys j <= i (is_causal)
  // Ulysses Anything: 0, or G when the batch axis is (group, batch) and the
  // head axis holds ceil(H/G) slots of which group g fills its first h_g
  // (tensor_split sizes of group_heads = H); padding slots are skipped
  int group_count;
  int group_heads;
  int n_tiles_all;       // key tiles over all chunks (the count without causal masking)
  int resident_ctas;     // CTAs in flight at once (one per SM; set at launch)
  int chunk_start[CPATTN_MAX_RING_DEGREE + 1];
  // extents of out, lse and the workspace (checked in CPATTN_CHECK builds)
  Span out_span, lse_span, ws_span;
};

enum class InDtype { F32, BF16 };

// Keys per K/V tile of the attention kernel for this input type and head
// size (the row count of the K and V tensor maps' boxes; query boxes have
// 128 rows).
int attn_kv_tile_rows(InDtype dt, int head_dim);

// Launches the attention kernel; tensor maps already encoded.
cudaError_t launch_attention(InDtype dt, int head_dim, const CUtensorMap& tm_q,
                             const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const AttnParams& p, cudaStream_t stream);

struct MergeParams {
  float* o_a;
  float* l_a;
  const float* o_b;
  const float* l_b;
  int64_t rows;          // B * H * S
  int head_dim;
  int heads, seq;        // for the strided index map
  int64_t oa_s[3], ob_s[3], la_s[3], lb_s[3];   // strides (b, h, s) in elements
  int dense;             // 1: all four tensors are dense row-major
  Span oa_span, ob_span, la_span, lb_span;   // (CPATTN_CHECK builds)
  unsigned int* err;     // device error word
};
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);

// Up to kMaxPermuteBatch tensors of one shape and dtype regrouped by one
// launch (tensor i: x[i] -> y[i]).
constexpr int kMaxPermuteBatch = CPATTN_MAX_PERMUTE_BATCH;
struct PermuteParams {
  int n;
  const void* x[kMaxPermuteBatch];
  void* y[kMaxPermuteBatch];
  int64_t batch, seq, heads, head_dim, degree;
  int dir;               // +1 forward, -1 inverse
  int elem_bytes;
  uint64_t x_bytes, y_bytes;   // extent of every x[i] / y[i] (CPATTN_CHECK builds)
  unsigned int* err;           // device error word
};
cudaError_t launch_permute(const PermuteParams& p, cudaStream_t stream);
// Ulysses Anything regroup between [B, S, H, D] and [G, B, S, ceil(H/G), D]
// (heads = H; H need not divide by G).
cudaError_t launch_permute_anything(const PermuteParams& p, cudaStream_t stream);

// Error word helpers (defined with the device symbol).
cudaError_t read_and_clear_device_error(unsigned int* value, cudaStream_t stream);
// Device address of the error word on the current device (nullptr on
// failure); looked up once per device.
unsigned int* device_error_word();

// SM count of the current device (152, GB300's, if it cannot be read).
int sm_count();

}  // namespace cpattn
