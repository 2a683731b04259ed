// attn_fwd.cu -- blockwise attention with in-kernel ring schedule for sm_103a.
//
// What it computes (page title, section):
//   Diffusers "Context parallelism", "Ring Attention": every query meets the
//   K/V block of every ring rank in turn; "Ring Anything Attention": the
//   blocks may be uneven.  Diffusers "Parallelism" API, ContextParallelConfig
//   convert_to_fp32: each step's output and LSE are kept in fp32 and merged.
//   One launch runs the whole ring for a tile of queries: for each chunk c
//   (in order 0 .. R-1) it computes the chunk's partial output o_c = O_c / l_c
//   and lse_c = m_c + ln l_c with an online softmax over the chunk's key
//   tiles, then folds (o_c, lse_c) into the running (o, lse) with
//     lse = max + log1p(exp(min - max)),  o = e^(lse_r - lse) o_r + e^(lse_c - lse) o_c.
//   With ring_degree = 1 it is a single partial (cpattn_partial).
//
// How (one CTA = two 128-row query tiles of one (batch, head) against
// 128-key K/V tiles; fp32 inputs at D = 128: one query tile against 64-key
// tiles, see Cfg; 12 warps):
//   warp 8      TMA producer: Q once, then K_j, V_j tiles through a
//               STAGES-deep shared-memory ring (128-byte swizzle); query
//               tiles are marked evict-first in L2, K/V tiles evict-last.
//   warp 9      MMA issuer (one thread): S_i = Q_i K_j^T into TMEM, then
//               O_i += P_i V_j with P_i read from TMEM (tcgen05.mma, fp32
//               accumulation), ping-ponging the two query tiles so the tensor
//               core works on one tile while the other tile's softmax runs.
//   warps 10-11 fp32 inputs only: transpose each V tile into a K-major copy
//               (the tf32 MMA kind takes no MN-major B operand) and split
//               each K tile into hi/lo parts; with one query tile per CTA
//               the otherwise idle warps 4-7 share that work.
//   warps 0-7   softmax, one warpgroup per query tile, one thread per query
//               row: S row from TMEM -> row max -> 2^(s*scale*log2e - m)
//               -> row sum, P (bf16, or fp32 rounded to the nearest tf32
//               for fp32 inputs) back into S's columns;
//               at each chunk end the normalised partial is merged in fp32
//               with the running result (held in a global fp32 workspace).
//   Three quarters through its key tiles, the producer also has the Q
//   tiles of the CTA one wave later (linear block order, one CTA per SM)
//   fetched into L2, so the next wave's start finds them there (bf16
//   launches; not for Ulysses Anything's padded head slots).
//   Without causal masking (bf16), once every K/V tile is in flight the
//   producer also bulk-copies the running result that the final merge
//   reads into shared memory (a spare region plus three released stages),
//   so the last epilogue reads it there instead of from global memory.
//   setmaxnreg moves registers from the control warpgroup (warps 8-11) to
//   the two softmax warpgroups.
//   TMEM (512 columns): S_0 | S_1 | O_0 | O_1, P written over S's first
//   columns.  bf16 at D = 64: S_0 | S_1 | O_0 | O_1 | P_0 | P_1, so a query
//   tile's next Q K^T goes out as soon as its softmax has loaded S, without
//   waiting for its P V (the softmax waits for that P V before it reads or
//   rescales O or writes P again).
//   The running max is only raised when it grows by more than 2^8 (exponent
//   8 in log2 units); between raises P values stay below 256, exact enough
//   for bf16/fp32 and far from overflow.  The O rescale that a raise needs
//   happens in TMEM, after the previous P V has completed.
#include <cuda_bf16.h>

#include <atomic>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"
#include "tmem_ops.cuh"

namespace cpattn {

// Device error word: bit flags of waits that ran out of time (and, in the
// bounds-checking build, of skipped out-of-extent accesses); read and
// cleared by the host after a stream synchronisation.
__device__ unsigned int g_cpattn_device_error = 0;

namespace {

constexpr int kBM = 128;          // query rows per tile (TMEM lanes)
constexpr int kThreads = 384;     // 3 warpgroups
constexpr int kWarpProducer = 8;  // warpgroup 2: producer, MMA, V transposer, spare
constexpr int kWarpMma = 9;
constexpr int kWarpTranspose = 10;
constexpr int kLaunchRegs = 168;  // registers per thread at launch (65536 / 384, rounded down to 8)
constexpr int kSoftmaxRegs = 208; // after setmaxnreg: 8 x 32 x 208 + 4 x 32 x 88 = 384 x 168
constexpr int kControlRegs = 88;
static_assert(2 * 4 * 32 * kSoftmaxRegs + 4 * 32 * kControlRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr float kLn2 = 0.693147180559945309f;
constexpr unsigned kErrWaitProducer = 1u, kErrWaitMma = 2u, kErrWaitSoftmax = 4u,
                   kErrWaitTranspose = 8u;

template <typename T, int D>
struct Cfg {
  static constexpr int ES = sizeof(T);
  static constexpr bool TF32 = (ES == 4);
  // query tiles per CTA and keys per K/V tile: two 128-row query tiles
  // against 128-key tiles, except for fp32 inputs with D = 128, whose tiles
  // fit shared memory and TMEM only as one query tile against 64-key tiles
  static constexpr int NT = (TF32 && D == 128) ? 1 : 2;
  static constexpr int BN = (TF32 && D == 128) ? 64 : 128;
  static constexpr int ROW_BYTES = D * ES;
  static constexpr int NKB = ROW_BYTES / 128;       // 128-byte column blocks per row
  static constexpr int BOX_COLS = 128 / ES;         // elements per column block
  static constexpr int Q_TILE_BYTES = kBM * ROW_BYTES;
  static constexpr int KV_TILE_BYTES = BN * ROW_BYTES;
  // fp32 inputs: the tf32 MMA kind takes no MN-major B operand, so V tiles
  // are transposed into K-major copies (rows = D, 128-byte blocks of 32
  // keys), double-buffered.  Q K^T runs as three tf32 products,
  // Q_hi K_hi + Q_hi K_lo + Q_lo K_hi (x = hi + lo, hi = x with its low 13
  // mantissa bits cleared), which keeps scores to about 2^-20 relative; Q_lo
  // sits in TMEM, K_lo in one shared-memory tile.
  static constexpr int VT_BUFS = TF32 ? 2 : 0;
  // fp32 inputs: warps that transpose V and split K (warps 10 and 11, plus
  // the second softmax warpgroup when it has no query tile)
  static constexpr int TP_WARPS = TF32 ? (NT == 1 ? 6 : 2) : 0;
  static constexpr int VT_TILE_BYTES = D * BN * ES;
  static constexpr int KLO_BYTES = TF32 ? KV_TILE_BYTES : 0;
  static constexpr int SMEM_BUDGET = (TF32 ? 226 : 220) * 1024;
  static constexpr int STAGES_FIT =
      (SMEM_BUDGET - NT * Q_TILE_BYTES - VT_BUFS * VT_TILE_BYTES - KLO_BYTES) / KV_TILE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  // bf16 without causal masking: the final merge's running state (fp32,
  // NT query tiles x D) is fetched into shared memory as 2 NT pieces of
  // one K/V tile's size each (half of D of one query tile): one into a
  // region of its own, the others into the stages released first once
  // every K/V tile is in flight
  static constexpr int WS_PIECE_BYTES = kBM * (D / 2) * 4;
  static constexpr int WSX_BYTES = TF32 ? 0 : WS_PIECE_BYTES;
  static constexpr int NUM_BARS =
      1 + 2 * STAGES + 3 * NT + 1 + 2 * VT_BUFS + (TF32 ? 3 : 0) + 4 * NT;
  static constexpr int SMEM_BYTES = 1024 + NT * Q_TILE_BYTES + STAGES * KV_TILE_BYTES +
                                    VT_BUFS * VT_TILE_BYTES + KLO_BYTES + WSX_BYTES +
                                    NUM_BARS * 8 + 16;
  static constexpr int KSTEP = 32 / ES;             // K elements per MMA (32 bytes)
  static constexpr int QK_STEPS = ROW_BYTES / 32;
  static constexpr int PV_STEPS = BN / KSTEP;
  static constexpr int P_COLS_PER_STEP = KSTEP * ES / 4;
  static constexpr uint32_t FMT = TF32 ? 2u : 1u;   // tf32 : bf16
  static constexpr uint32_t IDESC_QK = make_idesc(FMT, false, kBM, BN);
  static constexpr uint32_t IDESC_PV = make_idesc(FMT, !TF32, kBM, D);
  static constexpr int O_COL = NT * BN;
  static constexpr int QLO_COL = O_COL + NT * D;   // fp32 inputs: Q_lo of tile i at + i*D
  // bf16 at D = 64: TMEM has room for P apart from S (S0 S1 O0 O1 P0 P1 =
  // 128 + 128 + 64 + 64 + 64 + 64 columns), so a query tile's next Q K^T
  // need not wait for its P V; P of tile i at P_COL + i * BN / 2
  static constexpr bool SEP_P = !TF32 && D == 64;
  static constexpr int P_COL = O_COL + NT * D;
  static_assert(ROW_BYTES % 128 == 0, "rows must be whole 128-byte blocks");
  static_assert(O_COL + NT * D <= (int)kTmemCols, "TMEM budget");
  static_assert(!TF32 || QLO_COL + NT * D <= (int)kTmemCols, "tf32 TMEM budget");
  static_assert(!SEP_P || P_COL + NT * BN / 2 <= (int)kTmemCols, "separate-P TMEM budget");
  static_assert(TF32 || (NT == 2 && BN == 128), "the bf16 MMA schedule ping-pongs two tiles");
  static_assert(!TF32 || STAGES % 2 == 0, "fp32 inputs keep K tiles on even stages");
  static_assert(STAGES >= 2, "need at least two K/V stages");
  static_assert(TF32 || (WS_PIECE_BYTES == KV_TILE_BYTES && STAGES >= 2 * NT),
                "running-state pieces reuse K/V stages");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Byte offset of (row r, byte b of the row) in a tile stored as 128-byte
// column blocks of `rows` rows each, with the 128-byte swizzle (16-byte
// chunk index XOR row % 8), the layout TMA writes and tcgen05 reads.
__device__ __forceinline__ uint32_t sw128_offset(int r, int b, int rows) {
  return (b >> 7) * rows * 128 + r * 128 + ((((b >> 4) & 7) ^ (r & 7)) << 4) + (b & 15);
}

// The key tiles of chunk c this CTA visits: all of them, or with causal
// masking only those starting at or before `kmax`, the CTA's last query row.
template <int BN>
__device__ __forceinline__ int chunk_tiles(const AttnParams& p, int c, int kmax) {
  const int end = min(p.chunk_start[c + 1], kmax + 1);
  return end > p.chunk_start[c] ? ceil_div(end - p.chunk_start[c], BN) : 0;
}

// Walks the (chunk, tile) sequence shared by all roles; r_eff chunks (with
// causal masking the chunks past the CTA's last query row are empty for
// every row here, identities of the merge, and are not visited).
template <int BN>
struct TileWalk {
  int c = 0, t = 0, nt = 0, kmax = 0, r_eff = 0;
  __device__ void start(const AttnParams& p, int kmax_, int r_eff_) {
    c = 0;
    t = 0;
    kmax = kmax_;
    r_eff = r_eff_;
    nt = chunk_tiles<BN>(p, 0, kmax);
  }
  __device__ void next(const AttnParams& p) {
    if (++t == nt) {
      ++c;
      t = 0;
      if (c < r_eff) nt = chunk_tiles<BN>(p, c, kmax);
    }
  }
};

// Largest of the first `valid` scores of this thread's row; the others are
// set to -inf in place (keys past a chunk's end or, causal, after the row).
template <int N>
__device__ __forceinline__ float masked_row_max(uint32_t (&s)[N], int valid) {
#pragma unroll
  for (int i = 0; i < N; ++i)
    if (i >= valid) s[i] = f2u(-INFINITY);
  float mx[4] = {u2f(s[0]), u2f(s[1]), u2f(s[2]), u2f(s[3])};
#pragma unroll
  for (int i = 4; i < N; i += 8) {
    mx[0] = fmax3(mx[0], u2f(s[i + 0]), u2f(s[i + 1]));
    mx[1] = fmax3(mx[1], u2f(s[i + 2]), u2f(s[i + 3]));
    if (i + 4 < N) {
      mx[2] = fmax3(mx[2], u2f(s[i + 4]), u2f(s[i + 5]));
      mx[3] = fmax3(mx[3], u2f(s[i + 6]), u2f(s[i + 7]));
    }
  }
  return fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]);
}

// The running state's LSE of workspace row i (bounds-checked in
// CPATTN_CHECK builds).
__device__ __forceinline__ float ws_lse_at(const AttnParams& p, int64_t i) {
  return CPATTN_IN(p.ws_span, p.ws_lse + i, 4, &g_cpattn_device_error) ? p.ws_lse[i] : 0.f;
}

// Multiplies this thread's O row (TMEM) by `factor`.
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t tO, float factor) {
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t o[32];
    tmem_ld_x32(tO + c0, o);
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * factor);
    tmem_st_x32(tO + c0, o);
  }
  tmem_wait_st();
}

// End of chunk c for this thread's query row: emit the chunk's partial
// (o_c = O / l, lse_c = m ln2 + ln l) and fold it into the running result.
// PRE: the running state was prefetched into shared memory (pre0, pre1:
// byte offsets from sbase of the pieces holding D's first and second half,
// in the workspace tile's layout).
template <typename T, int D, bool PRE>
__device__ __forceinline__ void chunk_epilogue(const AttnParams& p, uint32_t tO, int c,
                                               int r_eff, float m_used, float l, int b, int h,
                                               int q_row, bool row_ok, int64_t tile_id,
                                               int tile_row, uint8_t* stage, float lse_run,
                                               const uint8_t* sbase, uint32_t pre0, uint32_t pre1) {
  const bool last = (c == r_eff - 1);
  // a row with no admissible key in the chunk (causal masking) emits the
  // empty partial (0, -inf): the identity of the merge below
  const bool empty = !(l > 0.f);
  const float inv_l = empty ? 0.f : 1.0f / l;
  const float lse_c = empty ? -INFINITY : (m_used + log2f(l)) * kLn2;
  // running merged state per 128-row query tile, laid out [D/4][kBM][4]:
  // the 32 lanes of a warp (32 consecutive rows) touch 512 contiguous bytes
  // with each float4 access
  float4* ws_tile = reinterpret_cast<float4*>(p.ws_o) + tile_id * (kBM * D / 4) + tile_row;
  float* ws_lse = p.ws_lse + tile_id * kBM + tile_row;
  float w_run = 0.f, w_c = 1.f, lse_new = lse_c;
  if (c > 0 && row_ok) {
    const float hi = fmaxf(lse_run, lse_c), lo = fminf(lse_run, lse_c);
    lse_new = hi + log1pf(expf(lo - hi));
    w_run = expf(lse_run - lse_new);
    w_c = expf(lse_c - lse_new);
  }
  // O columns per part: halves, or quarters when the running state comes
  // from shared memory (it is read in the same pass, so the part is smaller)
  // or when a row holds more than 64 fp32 values
  constexpr int NPARTS = (PRE || sizeof(T) * D > 256) ? 4 : 2;
  constexpr int HC = D / NPARTS;
  const int lane = tile_row % 32;
  // the final output goes through the warp's staging area when its element
  // has the input's size (bf16 -> bf16, f32 -> f32): 16-byte chunks per row
  const bool staged = (p.out_f32 != 0) == (sizeof(T) == 4);
  constexpr int kCPR = D * static_cast<int>(sizeof(T)) / 16;
#pragma unroll 1
  for (int part = 0; part < NPARTS; ++part) {
    uint32_t o[HC];
    __syncwarp();
    if constexpr (HC == 64)
      tmem_ld_x64(tO + part * HC, o);
    else if constexpr (HC == 32)
      tmem_ld_x32(tO + part * HC, o);
    else
      tmem_ld_x16(tO + part * HC, o);
    if (row_ok) {
      float4 v[HC / 4];
#pragma unroll
      for (int i = 0; i < HC / 4; ++i)   // partial output o_c
        v[i] = make_float4(u2f(o[4 * i]) * inv_l, u2f(o[4 * i + 1]) * inv_l,
                           u2f(o[4 * i + 2]) * inv_l, u2f(o[4 * i + 3]) * inv_l);
      float4* slot = ws_tile + part * (HC / 4) * kBM;
      if (c > 0) {
        // the running state: prefetched into shared memory (same layout as
        // the workspace tile, one piece per half of D) or read from the workspace
        auto fold = [&](int i, const float4& r) {
          v[i] = make_float4(w_run * r.x + w_c * v[i].x, w_run * r.y + w_c * v[i].y,
                             w_run * r.z + w_c * v[i].z, w_run * r.w + w_c * v[i].w);
        };
        if constexpr (PRE) {
          // shared-memory latency is short: each value is folded as it arrives
          constexpr int kPerPiece = NPARTS / 2;
          const float4* src =
              reinterpret_cast<const float4*>(sbase + (part < kPerPiece ? pre0 : pre1)) +
              (part % kPerPiece) * (HC / 4) * kBM + tile_row;
#pragma unroll
          for (int i = 0; i < HC / 4; ++i) fold(i, src[i * kBM]);
        } else {
          float4 r[HC / 4];
#pragma unroll
          for (int i = 0; i < HC / 4; ++i)
            r[i] = CPATTN_IN(p.ws_span, &slot[i * kBM], 16, &g_cpattn_device_error)
                       ? slot[i * kBM]
                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int i = 0; i < HC / 4; ++i) fold(i, r[i]);
        }
      }
      if (!last) {
#pragma unroll
        for (int i = 0; i < HC / 4; ++i)
          if (CPATTN_IN(p.ws_span, &slot[i * kBM], 16, &g_cpattn_device_error)) slot[i * kBM] = v[i];
      } else if (!staged) {
        // f32 output of bf16 inputs (a single partial): straight to memory
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + b * p.out_sb +
                                                h * p.out_sh + q_row * p.out_ss + part * HC);
#pragma unroll
        for (int i = 0; i < HC / 4; ++i)
          if (CPATTN_IN(p.out_span, &dst[i], 16, &g_cpattn_device_error)) dst[i] = v[i];
      } else {
        // final output: this lane's row into the warp's staging area
        // (16-byte chunks XOR-swizzled by row against bank conflicts)
        uint4* srow = reinterpret_cast<uint4*>(stage) + lane * kCPR;
        if constexpr (sizeof(T) == 4) {
#pragma unroll
          for (int i = 0; i < HC / 4; ++i) {
            const int c = part * (HC / 4) + i;
            srow[c ^ (lane % kCPR)] = make_uint4(f2u(v[i].x), f2u(v[i].y), f2u(v[i].z), f2u(v[i].w));
          }
        } else {
#pragma unroll
          for (int i = 0; i < HC / 8; ++i) {
            const int c = part * (HC / 8) + i;
            srow[c ^ (lane % kCPR)] =
                make_uint4(pack_bf16x2(v[2 * i].x, v[2 * i].y), pack_bf16x2(v[2 * i].z, v[2 * i].w),
                           pack_bf16x2(v[2 * i + 1].x, v[2 * i + 1].y),
                           pack_bf16x2(v[2 * i + 1].z, v[2 * i + 1].w));
          }
        }
      }
    }
  }
  if (last && staged) {
    // the warp's 32 rows leave the staging area as whole rows: half a warp
    // writes one row's bytes contiguously
    __syncwarp();
    const int row0 = q_row - lane;
    constexpr int64_t es = sizeof(T);
    uint8_t* out_base = static_cast<uint8_t*>(p.out) + (b * p.out_sb + h * p.out_sh) * es;
    const uint64_t pol_out = l2_policy_evict_first();   // not read again by this kernel
#pragma unroll
    for (int it = 0; it < kCPR; ++it) {
      const int idx = it * 32 + lane, r = idx / kCPR, c = idx % kCPR;
      if (row0 + r < p.s_q) {
        const uint4 val = reinterpret_cast<const uint4*>(stage)[r * kCPR + (c ^ (r % kCPR))];
        uint8_t* dst = out_base + (row0 + r) * p.out_ss * es + c * 16;
        if (CPATTN_IN(p.out_span, dst, 16, &g_cpattn_device_error))
          st_global_v4_hint(dst, val, pol_out);
      }
    }
  }
  if (row_ok) {
    if (last) {
      float* dst = p.lse + (b * p.lse_sb + h * p.lse_sh + q_row * p.lse_ss);
      if (CPATTN_IN(p.lse_span, dst, 4, &g_cpattn_device_error)) *dst = lse_new;
    } else if (CPATTN_IN(p.ws_span, ws_lse, 4, &g_cpattn_device_error)) {
      *ws_lse = lse_new;
    }
  }
  __syncwarp();
}

template <typename T, int D, bool CAUSAL, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ AttnParams p) {
  using C = Cfg<T, D>;
  // bf16 without causal masking prefetches the final merge's running state
  // (the causal kernel has no registers to spare for it)
  constexpr bool kPrefetchState = !C::TF32 && !CAUSAL;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

  const uint32_t sQ = smem_addr(smem);
  const uint32_t sKV = sQ + C::NT * C::Q_TILE_BYTES;
  const uint32_t sVt = sKV + C::STAGES * C::KV_TILE_BYTES;
  const uint32_t sKlo = sVt + C::VT_BUFS * C::VT_TILE_BYTES;
  const uint32_t sWsx = sKlo + C::KLO_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::NT * C::Q_TILE_BYTES +
                                               C::STAGES * C::KV_TILE_BYTES +
                                               C::VT_BUFS * C::VT_TILE_BYTES + C::KLO_BYTES +
                                               C::WSX_BYTES);
  const uint32_t bar0 = smem_addr(bars);
  const uint32_t BAR_Q = bar0;
  auto bar_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_empty = [&](int s) { return bar0 + 8u * (1 + C::STAGES + s); };
  auto bar_s = [&](int i) { return bar0 + 8u * (1 + 2 * C::STAGES + i); };
  auto bar_p = [&](int i) { return bar0 + 8u * (1 + 2 * C::STAGES + C::NT + i); };
  auto bar_o = [&](int i) { return bar0 + 8u * (1 + 2 * C::STAGES + 2 * C::NT + i); };
  const uint32_t BAR_DRAIN = bar0 + 8u * (1 + 2 * C::STAGES + 3 * C::NT);
  auto bar_vt_full = [&](int i) { return bar0 + 8u * (2 + 2 * C::STAGES + 3 * C::NT + i); };
  auto bar_vt_empty = [&](int i) {
    return bar0 + 8u * (2 + 2 * C::STAGES + 3 * C::NT + C::VT_BUFS + i);
  };
  const uint32_t BAR_QLO = bar0 + 8u * (2 + 2 * C::STAGES + 3 * C::NT + 2 * C::VT_BUFS);
  const uint32_t BAR_KLO_FULL = BAR_QLO + 8u;
  const uint32_t BAR_KLO_EMPTY = BAR_QLO + 16u;
  auto bar_ws = [&](int i) { return bar0 + 8u * (C::NUM_BARS - 2 * C::NT + i); };
  // bf16 at D = 64 (separate P): the softmax has S_j of tile i in registers;
  // P V_j of tile i has completed
  auto bar_sread = [&](int i) { return bar0 + 8u * (C::NUM_BARS - 4 * C::NT + i); };
  auto bar_pvdone = [&](int i) { return bar0 + 8u * (C::NUM_BARS - 3 * C::NT + i); };
  // the running state of query tile i is written and fenced for the bulk copy
  auto bar_ws_ready = [&](int i) { return bar0 + 8u * (C::NUM_BARS - C::NT + i); };
  // home of piece k of the final merge's running state (query tile k / 2,
  // half k % 2 of D) with n key tiles: the spare region, then the stages of
  // K/V loads 2n, 2n + 1, ..., whose previous tiles are released first
  // (as a byte offset from the Q tiles' start)
  auto ws_piece = [&](int k, int n) -> uint32_t {
    return k == 0 ? sWsx - sQ : sKV - sQ + ((2 * n + k - 1) % C::STAGES) * C::KV_TILE_BYTES;
  };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  // The warp index goes through a shuffle so that the compiler knows it is
  // the same for every lane of a warp: each role's code is then uniform,
  // which keeps the MMA warp's descriptors and loop state in uniform
  // registers (FLUX ring 209 -> 195 us).
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x / 32), 0);
  const int lane = threadIdx.x % 32;
  // causal: grid (H, B, query blocks), the heaviest query blocks first
  const int q_row0 =
      (CAUSAL ? static_cast<int>(gridDim.z - 1 - blockIdx.z) : static_cast<int>(blockIdx.x)) *
      (C::NT * kBM);
  const int h = CAUSAL ? blockIdx.x : blockIdx.y;
  const int b = CAUSAL ? blockIdx.y : blockIdx.z;
  if constexpr (GROUPED) {
    // Ulysses Anything: b = group * (batch / G) + batch index; head slots
    // past the group's own heads are padding (uniform per CTA, before any
    // barrier or TMEM allocation)
    const int g = b / (p.batch / p.group_count);
    const int hg = p.group_heads / p.group_count + (g < p.group_heads % p.group_count ? 1 : 0);
    if (h >= hg) return;
  }

  if (threadIdx.x == 0) {
    mbar_init(BAR_Q, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      // fp32 inputs: a K stage is released by the MMA and by the K_lo pass
      // (fp32 inputs: a K stage is released by the MMA and the transposing
      // warps, a V stage by the transposing warps)
      mbar_init(bar_empty(s), C::TF32 ? (s % 2 == 0 ? 1 + C::TP_WARPS : C::TP_WARPS) : 1);
    }
    for (int i = 0; i < C::NT; ++i) {
      mbar_init(bar_s(i), 1);
      mbar_init(bar_p(i), 4);   // one arrival per softmax warp
      mbar_init(bar_o(i), 1);
    }
    mbar_init(BAR_DRAIN, 1);
    for (int i = 0; i < C::NT; ++i) {
      mbar_init(bar_ws(i), 1);
      mbar_init(bar_ws_ready(i), 4);   // one arrival per softmax warp
      mbar_init(bar_sread(i), 4);      // one arrival per softmax warp
      mbar_init(bar_pvdone(i), 1);
    }
    for (int i = 0; i < C::VT_BUFS; ++i) {
      mbar_init(bar_vt_full(i), C::TP_WARPS);
      mbar_init(bar_vt_empty(i), 1);
    }
    if (C::TF32) {
      mbar_init(BAR_QLO, 4 * C::NT);   // one arrival per softmax warp
      mbar_init(BAR_KLO_FULL, C::TP_WARPS);
      mbar_init(BAR_KLO_EMPTY, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    // The Q tiles (and, bf16, the first K tile) are requested before the
    // block-wide barrier, so their latency overlaps the rest of the setup.
    mbar_arrive_expect_tx(BAR_Q, C::NT * C::Q_TILE_BYTES);
    const uint64_t pol_q = l2_policy_evict_first();
    for (int i = 0; i < C::NT; ++i)
      for (int kb = 0; kb < C::NKB; ++kb)
        tma_load_4d_hint(sQ + i * C::Q_TILE_BYTES + kb * kBM * 128, &tm_q, BAR_Q,
                         kb * C::BOX_COLS, q_row0 + i * kBM, h, b, pol_q);
    if (!C::TF32 && p.fault_skip_kv == 0) {
      mbar_arrive_expect_tx(bar_full(0), C::KV_TILE_BYTES);
      const uint64_t pol_kv = l2_policy_evict_last();
      for (int kb = 0; kb < C::NKB; ++kb)
        tma_load_4d_hint(sKV + kb * C::BN * 128, &tm_k, bar_full(0), kb * C::BOX_COLS,
                         p.chunk_start[0], h, b, pol_kv);
    }
  }
  if (warp == kWarpMma) tmem_alloc(smem_addr(tmem_holder), kTmemCols);
  if (warp == kWarpProducer && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // largest key index a row of this CTA may attend; chunks starting past it
  // are skipped (chunk 0 starts at key 0, so at least one chunk remains)
  // (INT_MAX - 1 without causal masking, so that kmax + 1 cannot overflow)
  const int kmax = CAUSAL ? min(q_row0 + C::NT * kBM, p.s_q) - 1 : 0x7ffffffe;
  int r_eff = p.ring_degree;
  int n_tiles = p.n_tiles_all;   // (computed by the host without causal masking)
  if (CAUSAL) {
    while (r_eff > 1 && p.chunk_start[r_eff - 1] > kmax) --r_eff;
    n_tiles = 0;
    for (int c = 0; c < r_eff; ++c) n_tiles += chunk_tiles<C::BN>(p, c, kmax);
  }

  // ------------------------------------------------------------ fp32 operand prep
  // K_j in place -> K_hi (low 13 mantissa bits cleared), K_lo = K - K_hi into
  // its own tile (same layout); V_j [keys x D] as TMA wrote it -> Vt [D x
  // keys] (values rounded to the nearest tf32: P V is a single tf32 product,
  // so this rounding and P's are its only error), K-major, swizzled.  Run by
  // warps 10 and 11, and with one query tile per CTA also by the idle second
  // softmax warpgroup: C::TP_WARPS warps in all, warp tw of them taking every
  // C::TP_WARPS-th group of 32 elements (one warp alone set the fp32 path's
  // pace).
  auto transpose_role = [&](int tw) {
    const int tl = tw * 32 + lane;
    constexpr int kStride = 32 * (C::TP_WARPS > 0 ? C::TP_WARPS : 1);
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int lk = 2 * j, sk = lk % C::STAGES;
      ok = mbar_wait(bar_full(sk), (lk / C::STAGES) & 1, abort_flag, p.timeout_ns,
                     &g_cpattn_device_error, kErrWaitTranspose);
      if (ok)
        ok = mbar_wait(BAR_KLO_EMPTY, (j & 1) ^ 1, abort_flag, p.timeout_ns,
                       &g_cpattn_device_error, kErrWaitTranspose);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      {
        uint32_t* kt = reinterpret_cast<uint32_t*>(smem + (sKV - sQ) + sk * C::KV_TILE_BYTES);
        uint32_t* klo = reinterpret_cast<uint32_t*>(smem + (sKlo - sQ));
        for (int e = tl; e < C::KV_TILE_BYTES / 4; e += kStride) {
          const uint32_t x = kt[e], hi = x & 0xFFFFE000u;
          kt[e] = hi;
          klo[e] = f2u(u2f(x) - u2f(hi));
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(BAR_KLO_FULL);
        mbar_arrive(bar_empty(sk));
      }
      const int lv = 2 * j + 1, sv = lv % C::STAGES;
      ok = mbar_wait(bar_full(sv), (lv / C::STAGES) & 1, abort_flag, p.timeout_ns,
                     &g_cpattn_device_error, kErrWaitTranspose);
      if (ok)
        ok = mbar_wait(bar_vt_empty(j & 1), ((j >> 1) & 1) ^ 1, abort_flag, p.timeout_ns,
                       &g_cpattn_device_error, kErrWaitTranspose);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const uint8_t* src = smem + (sKV - sQ) + sv * C::KV_TILE_BYTES;
      uint8_t* dst = smem + (sVt - sQ) + (j & 1) * C::VT_TILE_BYTES;
      for (int e = tl; e < C::BN * D; e += kStride) {
        const int key = e % C::BN, d = e / C::BN;
        const uint32_t v = *reinterpret_cast<const uint32_t*>(src + sw128_offset(key, d * 4, C::BN));
        *reinterpret_cast<uint32_t*>(dst + sw128_offset(d, key * 4, D)) = tf32_round_bits(v);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_vt_full(j & 1));
        mbar_arrive(bar_empty(sv));
      }
    }
    __syncwarp();
  };

  if (warp >= 8) {
    regs_decrease<kControlRegs>();
    // The producer and MMA warps run their schedules with all 32 lanes, so
    // every index, phase and descriptor stays warp-uniform; one elected lane
    // issues the TMA copies, the MMAs and the commits (a commit tracks the
    // MMAs of the thread that issues it).
    auto wait_all = [&](uint32_t bar, uint32_t parity, unsigned code) {
      const bool r = mbar_wait(bar, parity, abort_flag, p.timeout_ns, &g_cpattn_device_error, code);
      return __all_sync(0xffffffffu, r);
    };
    const bool leader = elect_one();
    if (warp == kWarpProducer) {
      // ---------------------------------------------------------- producer
      // (the Q tiles and bf16's K_0 were requested during the setup)
      int ld = 0;
      int ws_armed = 0;   // query tiles whose running-state pieces are in flight
      // fault injection (testing): no K/V copies, so every consumer's
      // bounded wait runs out and the CTA takes the abort path
      bool ok = p.fault_skip_kv == 0;
      TileWalk<C::BN> w;
      w.start(p, kmax, r_eff);
      if constexpr (!C::TF32) {
        // bf16: K_0 alone, then V_j and K_{j+1} as one pair on K_{j+1}'s
        // full barrier (V_{n-1} alone on its own), so the MMA warp waits
        // once per tile.  With an even stage count K always lands in an
        // even stage and V in an odd one.
        static_assert(C::STAGES % 2 == 0, "K/V pairing needs an even stage count");
        const uint64_t pol_kv = l2_policy_evict_last();
        auto load = [&](const CUtensorMap* tm, int stage, uint32_t bar, int key0) {
          for (int kb = 0; kb < C::NKB; ++kb)
            tma_load_4d_hint(sKV + stage * C::KV_TILE_BYTES + kb * C::BN * 128, tm, bar,
                             kb * C::BOX_COLS, key0, h, b, pol_kv);
        };
        if (ok) ld = 1;   // K_0
        for (int j = 0; j < n_tiles && ok; ++j) {
          // three quarters through, the Q tiles of the CTA that will start
          // one wave later (blocks are dispatched in linear order, one per
          // SM) are fetched into L2, while HBM is otherwise little used
          if (!GROUPED && j == (3 * n_tiles) / 4 && leader) {
            const int64_t ln =
                blockIdx.x +
                static_cast<int64_t>(gridDim.x) *
                    (blockIdx.y + static_cast<int64_t>(gridDim.y) * blockIdx.z) +
                p.resident_ctas;
            if (ln < static_cast<int64_t>(gridDim.x) * gridDim.y * gridDim.z) {
              const int xn = static_cast<int>(ln % gridDim.x);
              const int yn = static_cast<int>((ln / gridDim.x) % gridDim.y);
              const int zn = static_cast<int>(ln / (static_cast<int64_t>(gridDim.x) * gridDim.y));
              const int row0 = (CAUSAL ? static_cast<int>(gridDim.z) - 1 - zn : xn) * (C::NT * kBM);
              const int hn = CAUSAL ? xn : yn, bn = CAUSAL ? yn : zn;
              for (int i = 0; i < C::NT; ++i)
                if (row0 + i * kBM < p.s_q)
                  for (int kb = 0; kb < C::NKB; ++kb)
                    tma_prefetch_l2_4d(&tm_q, kb * C::BOX_COLS, row0 + i * kBM, hn, bn);
            }
          }
          const int key_v = p.chunk_start[w.c] + w.t * C::BN;
          w.next(p);
          const bool more = j + 1 < n_tiles;
          const int key_k = more ? p.chunk_start[w.c] + w.t * C::BN : 0;
          const int sv = ld % C::STAGES, sk = (ld + 1) % C::STAGES;
          ok = wait_all(bar_empty(sv), ((ld / C::STAGES) & 1) ^ 1, kErrWaitProducer);
          if (ok && more)
            ok = wait_all(bar_empty(sk), (((ld + 1) / C::STAGES) & 1) ^ 1, kErrWaitProducer);
          if (!ok) break;
          if (leader) {
            const uint32_t bar = more ? bar_full(sk) : bar_full(sv);
            mbar_arrive_expect_tx(bar, (more ? 2 : 1) * C::KV_TILE_BYTES);
            load(&tm_v, sv, bar, key_v);
            if (more) load(&tm_k, sk, bar, key_k);
          }
          __syncwarp();
          ld += more ? 2 : 1;
        }
        // the final merge's running state, once every K/V tile is in flight:
        // a query tile's two pieces are armed and issued together once both
        // of their homes are free, so an abort never leaves one half-armed
        if (kPrefetchState && ok && r_eff > 1) {
          const int64_t tile0 =
              (static_cast<int64_t>(b) * p.heads + h) * ((p.s_q + kBM - 1) / kBM) + q_row0 / kBM;
          for (int i = 0; i < C::NT && ok; ++i) {
            if (q_row0 + i * kBM >= p.s_q) break;   // no such query tile, no state
            ok = wait_all(bar_ws_ready(i), 0, kErrWaitProducer);
            for (int k = 2 * i; k < 2 * i + 2 && ok; ++k) {
              if (k == 0) continue;   // the spare region is always free
              const int x = ld + k - 1;
              ok = wait_all(bar_empty(x % C::STAGES), ((x / C::STAGES) & 1) ^ 1, kErrWaitProducer);
            }
            if (!ok) break;
            if (leader) {
              const char* src = reinterpret_cast<const char*>(p.ws_o) + (tile0 + i) * (kBM * D * 4);
              if (CPATTN_IN(p.ws_span, src, 2 * C::WS_PIECE_BYTES, &g_cpattn_device_error)) {
                mbar_arrive_expect_tx(bar_ws(i), 2 * C::WS_PIECE_BYTES);
                for (int k = 2 * i; k < 2 * i + 2; ++k)
                  bulk_load(sQ + ws_piece(k, n_tiles), src + (k % 2) * C::WS_PIECE_BYTES,
                            C::WS_PIECE_BYTES, bar_ws(i));
              } else {
                mbar_arrive(bar_ws(i));   // (reported; nothing copied)
              }
            }
            __syncwarp();
            ws_armed = i + 1;
          }
        }
      } else {
        // fp32 inputs: K_j and V_j each on their own stage barrier
        for (int j = 0; j < n_tiles && ok; ++j) {
          const int key0 = p.chunk_start[w.c] + w.t * C::BN;
          for (int which = 0; which < 2; ++which) {
            const int s = ld % C::STAGES;
            const uint32_t ph = (ld / C::STAGES) & 1;
            ok = wait_all(bar_empty(s), ph ^ 1, kErrWaitProducer);
            if (!ok) break;
            if (leader) {
              mbar_arrive_expect_tx(bar_full(s), C::KV_TILE_BYTES);
              const CUtensorMap* tm = which == 0 ? &tm_k : &tm_v;
              for (int kb = 0; kb < C::NKB; ++kb)
                tma_load_4d(sKV + s * C::KV_TILE_BYTES + kb * C::BN * 128, tm, bar_full(s),
                            kb * C::BOX_COLS, key0, h, b);
            }
            __syncwarp();
            ++ld;
          }
          w.next(p);
        }
      }
      if (!ok && leader) {
        // leave no copy in flight into this CTA's shared memory
        mbar_drain(BAR_Q, 0, p.timeout_ns);
        for (int x = ld > C::STAGES ? ld - C::STAGES : 0; x < ld; ++x) {
          if (C::TF32 || x % 2 == 0)
            mbar_drain(bar_full(x % C::STAGES), (x / C::STAGES) & 1, p.timeout_ns);
          else if (x + 1 >= ld)   // bf16: a V issued alone completes its own barrier once
            mbar_drain(bar_full(x % C::STAGES), 0, p.timeout_ns);
        }
      }
      // the running-state pieces land before this CTA's shared memory is released
      if (leader)
        for (int i = 0; i < ws_armed; ++i) mbar_drain(bar_ws(i), 0, p.timeout_ns);
      __syncwarp();
    } else if (warp == kWarpMma) {
      // ---------------------------------------------------------- MMA issuer
      // Descriptors are built once; an MMA's operands are a base plus a
      // compile-time offset (byte offset >> 4).
      const uint64_t q_desc = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t k_desc = smem_desc_sw128(sKV, 16, 1024);
      const uint64_t v_desc = smem_desc_sw128(sKV, C::BN * 128, 1024);
      const uint64_t vt_desc = C::TF32 ? smem_desc_sw128(sVt, 16, 1024) : 0;
      const uint64_t klo_desc = C::TF32 ? smem_desc_sw128(sKlo, 16, 1024) : 0;
      auto issue_qk = [&](int i, int stage) {
        const uint32_t d_tmem = tmem + i * C::BN;
        const uint64_t a0 = q_desc + static_cast<uint64_t>((i * C::Q_TILE_BYTES) >> 4);
        const uint64_t b0 = k_desc + static_cast<uint64_t>((stage * C::KV_TILE_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < C::QK_STEPS; ++kk) {
          const uint64_t off_a = ((kk / 4) * (kBM * 128) + (kk % 4) * 32) >> 4;
          const uint64_t off_b = ((kk / 4) * (C::BN * 128) + (kk % 4) * 32) >> 4;
          mma_ss<C::TF32>(d_tmem, a0 + off_a, b0 + off_b, C::IDESC_QK, kk > 0);
          if constexpr (C::TF32) {
            mma_ss<true>(d_tmem, a0 + off_a, klo_desc + off_b, C::IDESC_QK, 1u);
            mma_ts<true>(d_tmem, tmem + C::QLO_COL + i * D + kk * C::P_COLS_PER_STEP, b0 + off_b,
                         C::IDESC_QK, 1u);
          }
        }
      };
      // P (TMEM) x V: bf16 reads V as an MN-major operand straight from the
      // TMA tile; tf32 reads the transposed, K-major copy.
      auto issue_pv = [&](int i, uint64_t b0, uint32_t acc) {
        const uint32_t d_tmem = tmem + C::O_COL + i * D;
        const uint32_t a_tmem = tmem + i * C::BN;
#pragma unroll
        for (int kk = 0; kk < C::PV_STEPS; ++kk) {
          uint64_t off_b;
          if constexpr (C::TF32)
            off_b = ((kk / 4) * (D * 128) + (kk % 4) * 32) >> 4;
          else
            off_b = (kk * C::KSTEP * 128) >> 4;
          mma_ts<C::TF32>(d_tmem, a_tmem + kk * C::P_COLS_PER_STEP, b0 + off_b, C::IDESC_PV,
                          (kk > 0 || acc) ? 1u : 0u);
        }
      };
      bool ok = wait_all(BAR_Q, 0, kErrWaitMma);
      if (ok) ok = wait_all(bar_full(0), 0, kErrWaitMma);
      if (C::TF32 && ok) ok = wait_all(BAR_QLO, 0, kErrWaitMma);
      if (C::TF32 && ok) ok = wait_all(BAR_KLO_FULL, 0, kErrWaitMma);
      if (ok) {
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int i = 0; i < C::NT; ++i) {
            issue_qk(i, 0);
            mma_commit(bar_s(i));
          }
          mma_commit(bar_empty(0));
          if constexpr (C::TF32) mma_commit(BAR_KLO_EMPTY);
        }
        __syncwarp();
      }
      TileWalk<C::BN> w;
      w.start(p, kmax, r_eff);
      for (int j = 0; j < n_tiles && ok; ++j) {
        const uint32_t acc = w.t != 0 ? 1u : 0u;
        const int lv = 2 * j + 1, sv = lv % C::STAGES;
        const uint32_t phv = (lv / C::STAGES) & 1;
        const int lk = 2 * j + 2, sk = lk % C::STAGES;
        const uint32_t phk = (lk / C::STAGES) & 1;
        const bool more = j + 1 < n_tiles;
        if constexpr (C::SEP_P) {
          // bf16 at D = 64: P has TMEM of its own, so each query tile's
          // Q K_{j+1}^T goes out once its softmax has S_j in registers, and
          // P V_j once P_j is ready (V_j and K_{j+1} arrive together on
          // K_{j+1}'s barrier; the last V alone on its own).  Tile by tile
          // (Q K_{j+1}^T and P V_j of tile 0, then of tile 1) keeps the two
          // softmaxes half a period apart; both tiles' Q K first, then both
          // P V, let them run in step and was 7-9 % slower.
          const uint32_t kv_bar = more ? bar_full(sk) : bar_full(sv);
          const uint32_t kv_ph = more ? phk : 0u;
          const uint32_t hi = static_cast<uint32_t>(q_desc >> 32);
          const uint32_t vb = static_cast<uint32_t>(v_desc) + ((sv * C::KV_TILE_BYTES) >> 4);
          const uint32_t kb = static_cast<uint32_t>(k_desc) + ((sk * C::KV_TILE_BYTES) >> 4);
          uint32_t vd[C::PV_STEPS], kd[C::QK_STEPS], qd[C::QK_STEPS], pa[C::PV_STEPS];
#pragma unroll
          for (int kk = 0; kk < C::PV_STEPS; ++kk) {
            vd[kk] = vb + ((kk * C::KSTEP * 128) >> 4);
            pa[kk] = tmem + C::P_COL + kk * C::P_COLS_PER_STEP;
          }
#pragma unroll
          for (int kk = 0; kk < C::QK_STEPS; ++kk) {
            kd[kk] = kb + (((kk / 4) * (C::BN * 128) + (kk % 4) * 32) >> 4);
            qd[kk] = static_cast<uint32_t>(q_desc) + (((kk / 4) * (kBM * 128) + (kk % 4) * 32) >> 4);
          }
          ok = wait_all(kv_bar, kv_ph, kErrWaitMma);
          if (!ok) break;
          // per query tile: Q K_{j+1}^T once S_j is read, then P V_j
#pragma unroll
          for (int i = 0; i < C::NT; ++i) {
            if (more) {
              ok = wait_all(bar_sread(i), j & 1, kErrWaitMma);
              if (!ok) break;
              tc_fence_after();
              if (leader) {
                mma_group<C::QK_STEPS, true>(tmem + i * C::BN, qd, kd, hi, C::IDESC_QK, 0u);
                mma_commit(bar_s(i));
                if (i == C::NT - 1) mma_commit(bar_empty(sk));
              }
              __syncwarp();
#pragma unroll
              for (int kk = 0; kk < C::QK_STEPS; ++kk) qd[kk] += C::Q_TILE_BYTES >> 4;
            }
            ok = wait_all(bar_p(i), j & 1, kErrWaitMma);
            if (!ok) break;
            tc_fence_after();
            if (leader) {
              mma_group<C::PV_STEPS, false>(tmem + C::O_COL + i * D, pa, vd, hi, C::IDESC_PV, acc);
              mma_commit(bar_pvdone(i));
              if (i == C::NT - 1) mma_commit(bar_empty(sv));
              if (!more) mma_commit(bar_o(i));
            }
            __syncwarp();
#pragma unroll
            for (int kk = 0; kk < C::PV_STEPS; ++kk) pa[kk] += C::BN / 2;
          }
          if (!ok) break;
        } else if constexpr (!C::TF32) {
          // Every wait that does not depend on the softmax comes first and
          // all descriptors of both groups are built before P_0 is awaited,
          // so that once it is seen only the MMAs are left to issue: this
          // warp gets few issue slots beside the softmax warps of its SM
          // sub-partition, and the hardware MMA queue is only a few MMAs
          // deep, draining during any wait placed between MMAs.
          // V_j and K_{j+1} arrive together on K_{j+1}'s barrier; the last V
          // alone completes its own barrier's first phase
          const uint32_t kv_bar = more ? bar_full(sk) : bar_full(sv);
          const uint32_t kv_ph = more ? phk : 0u;
          // non-blocking probes first: their latency overlaps the descriptor
          // build; a barrier found incomplete is waited for afterwards
          const bool kv_now = mbar_test(kv_bar, kv_ph);
          const bool p0_now = mbar_test(bar_p(0), j & 1);
          // all descriptors share their high word; the low word holds the
          // start address (no carry: shared memory is below 256 KB)
          const uint32_t hi = static_cast<uint32_t>(q_desc >> 32);
          const uint32_t vb = static_cast<uint32_t>(v_desc) + ((sv * C::KV_TILE_BYTES) >> 4);
          const uint32_t kb = static_cast<uint32_t>(k_desc) + ((sk * C::KV_TILE_BYTES) >> 4);
          uint32_t vd[C::PV_STEPS], kd[C::QK_STEPS], qd[C::QK_STEPS], pa[C::PV_STEPS];
#pragma unroll
          for (int kk = 0; kk < C::PV_STEPS; ++kk) {
            vd[kk] = vb + ((kk * C::KSTEP * 128) >> 4);
            pa[kk] = tmem + kk * C::P_COLS_PER_STEP;
          }
#pragma unroll
          for (int kk = 0; kk < C::QK_STEPS; ++kk) {
            kd[kk] = kb + (((kk / 4) * (C::BN * 128) + (kk % 4) * 32) >> 4);
            qd[kk] = static_cast<uint32_t>(q_desc) + (((kk / 4) * (kBM * 128) + (kk % 4) * 32) >> 4);
          }
          ok = __all_sync(0xffffffffu, kv_now) || wait_all(kv_bar, kv_ph, kErrWaitMma);
          if (!ok) break;
          ok = __all_sync(0xffffffffu, p0_now) || wait_all(bar_p(0), j & 1, kErrWaitMma);
          if (!ok) break;
          // tile 1's P is probed now and waited for only if it was not yet
          // complete (a completed phase cannot advance before this warp's
          // next commit)
          const bool p1_now = mbar_test(bar_p(1), j & 1);
          tc_fence_after();
          if (leader) {
            mma_group<C::PV_STEPS, false>(tmem + C::O_COL, pa, vd, hi, C::IDESC_PV, acc);
            if (more) {
              mma_group<C::QK_STEPS, true>(tmem, qd, kd, hi, C::IDESC_QK, 0u);
              mma_commit(bar_s(0));
            } else {
              mma_commit(bar_o(0));
            }
          }
          __syncwarp();
          // query tile 1: P in the next S columns, Q in the next tile
#pragma unroll
          for (int kk = 0; kk < C::PV_STEPS; ++kk) pa[kk] += C::BN;
#pragma unroll
          for (int kk = 0; kk < C::QK_STEPS; ++kk) qd[kk] += C::Q_TILE_BYTES >> 4;
          ok = __all_sync(0xffffffffu, p1_now) || wait_all(bar_p(1), j & 1, kErrWaitMma);
          if (!ok) break;
          tc_fence_after();
          if (leader) {
            mma_group<C::PV_STEPS, false>(tmem + C::O_COL + D, pa, vd, hi, C::IDESC_PV, acc);
            mma_commit(bar_empty(sv));
            if (more) {
              mma_group<C::QK_STEPS, true>(tmem + C::BN, qd, kd, hi, C::IDESC_QK, 0u);
              mma_commit(bar_s(1));
              mma_commit(bar_empty(sk));
            } else {
              mma_commit(bar_o(1));
            }
          }
        } else {
          // fp32 inputs (3 MMAs per Q K step), query tile by query tile; the
          // first tile's group waits for everything it reads (P_0, the
          // transposed V_j, K_{j+1} and its low part) before its first MMA,
          // the last tile's group releases V_j's copy, K_{j+1} and K_lo
          const uint64_t v_base = vt_desc + static_cast<uint64_t>(((j & 1) * C::VT_TILE_BYTES) >> 4);
#pragma unroll
          for (int i = 0; i < C::NT && ok; ++i) {
            ok = wait_all(bar_p(i), j & 1, kErrWaitMma);
            if (ok && i == 0) ok = wait_all(bar_vt_full(j & 1), (j >> 1) & 1, kErrWaitMma);
            if (ok && i == 0 && more) ok = wait_all(bar_full(sk), phk, kErrWaitMma);
            if (ok && i == 0 && more) ok = wait_all(BAR_KLO_FULL, (j + 1) & 1, kErrWaitMma);
            if (!ok) break;
            tc_fence_after();
            if (leader) {
              const bool last_tile = i == C::NT - 1;
              issue_pv(i, v_base, acc);
              if (last_tile) mma_commit(bar_vt_empty(j & 1));
              if (more) {
                issue_qk(i, sk);
                mma_commit(bar_s(i));
                if (last_tile) {
                  mma_commit(bar_empty(sk));
                  mma_commit(BAR_KLO_EMPTY);
                }
              } else {
                mma_commit(bar_o(i));
              }
            }
            __syncwarp();
          }
          if (!ok) break;
        }
        __syncwarp();
        w.next(p);
      }
      if (!ok && leader) {
        // let every MMA already issued finish before TMEM is released
        mma_commit(BAR_DRAIN);
        mbar_drain(BAR_DRAIN, 0, p.timeout_ns);
      }
      __syncwarp();
    } else if (warp >= kWarpTranspose && warp < kWarpTranspose + 2 && C::TF32) {
      transpose_role(warp - kWarpTranspose);
    }
  } else if (C::TF32 && C::NT == 1 && warp >= 4 && warp < 8) {
    transpose_role(2 + warp - 4);
  } else if (warp / 4 < C::NT) {
    // ------------------------------------------------------------ softmax
    // (one warpgroup per query tile; with a single query tile per CTA, fp32
    // inputs at D = 128, the second warpgroup transposes V instead)
    regs_increase<kSoftmaxRegs>();
    const int wg = warp / 4;
    const int quarter = warp % 4;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + wg * C::BN;
    const uint32_t tO = tmem + lane_base + C::O_COL + wg * D;
    const int q_row = q_row0 + wg * kBM + quarter * 32 + lane;
    // this row's query tile in the running-state workspace, and its row there
    const int64_t tile_id = (static_cast<int64_t>(b) * p.heads + h) * ((p.s_q + kBM - 1) / kBM) +
                            q_row0 / kBM + wg;
    const int tile_row = quarter * 32 + lane;
    const bool row_ok = q_row < p.s_q;
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    if constexpr (C::TF32) {
      // this thread's Q row: Q_hi back in place, Q_lo into TMEM
      ok = mbar_wait(BAR_Q, 0, abort_flag, p.timeout_ns, &g_cpattn_device_error,
                     kErrWaitSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        uint8_t* qt = smem + wg * C::Q_TILE_BYTES;
        const int r = quarter * 32 + lane;
        uint32_t lo[D];
#pragma unroll
        for (int d = 0; d < D; ++d) {
          uint32_t* e = reinterpret_cast<uint32_t*>(qt + sw128_offset(r, d * 4, kBM));
          const uint32_t x = *e, hi = x & 0xFFFFE000u;
          *e = hi;
          lo[d] = f2u(u2f(x) - u2f(hi));
        }
        fence_proxy_async_smem();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 64)
          tmem_st_x64(tmem + lane_base + C::QLO_COL + wg * D + c0,
                      *reinterpret_cast<uint32_t(*)[64]>(&lo[c0]));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR_QLO);
      }
    }
    TileWalk<C::BN> w;
    w.start(p, kmax, r_eff);
    for (int j = 0; j < n_tiles && ok; ++j) {
      ok = mbar_wait(bar_s(wg), j & 1, abort_flag, p.timeout_ns, &g_cpattn_device_error,
                     kErrWaitSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // separate P: P V_{j-1} of this tile must have completed before O is
      // read or rescaled and before P is overwritten (waited for once)
      bool pv_done = !C::SEP_P || j == 0;
      if (C::SEP_P && !pv_done && w.t == 0 && w.c > 0) {
        ok = mbar_wait(bar_pvdone(wg), (j - 1) & 1, abort_flag, p.timeout_ns,
                       &g_cpattn_device_error, kErrWaitSoftmax);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        pv_done = true;
      }
      if (w.t == 0 && w.c > 0) {
        const float lse_run = (w.c > 1 && row_ok) ? ws_lse_at(p, tile_id * kBM + tile_row) : 0.f;
        chunk_epilogue<T, D, false>(p, tO, w.c - 1, r_eff, m_used, l, b, h, q_row, row_ok,
                                    tile_id, tile_row, nullptr, lse_run, nullptr, 0u, 0u);
      }

      // keys past the chunk's end, and with causal masking keys after this
      // row, are masked
      const int key0 = p.chunk_start[w.c] + w.t * C::BN;
      int valid = p.chunk_start[w.c + 1] - key0;
      if constexpr (CAUSAL) valid = min(valid, q_row + 1 - key0);
      const bool masked = CAUSAL ? __any_sync(0xffffffffu, valid < C::BN) : valid < C::BN;
      uint32_t s[C::BN];
      float row_max;
      if constexpr (C::BN == 128) {
        if (!masked) {
          // the TMEM load returns the row max as well (no max pass)
          tmem_ld_max_x128(tS, s, row_max);
        } else {
          tmem_ld_x128(tS, s);
          row_max = masked_row_max<C::BN>(s, valid);
        }
        if constexpr (C::SEP_P) {
          // S_j is in registers: Q K_{j+1}^T may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_sread(wg));
        }
      } else {
        tmem_ld_x64(tS, s);
        row_max = masked_row_max<C::BN>(s, masked ? valid : C::BN);
      }
      const float m_tile = row_max * sl2;
      float factor = 1.f;
      bool need = false;
      if (w.t == 0) {
        m_used = m_tile;
        l = 0.f;
      } else if (m_tile > m_used + kRescaleThreshold) {
        factor = ex2_approx(m_used - m_tile);
        m_used = m_tile;
        l *= factor;
        need = true;
      }
      if (__any_sync(0xffffffffu, need)) {
        if (C::SEP_P && !pv_done) {
          ok = mbar_wait(bar_pvdone(wg), (j - 1) & 1, abort_flag, p.timeout_ns,
                         &g_cpattn_device_error, kErrWaitSoftmax);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          pv_done = true;
        }
        rescale_o<D>(tO, factor);
      }

      // a row with every key so far masked keeps m = -inf; its P stays 0
      const float neg_m = (CAUSAL && m_used == -INFINITY) ? 0.f : -m_used;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < C::BN / 2; ++i) {
        float x0, x1;
        ffma2(x0, x1, u2f(s[2 * i]), u2f(s[2 * i + 1]), sl2, sl2, neg_m, neg_m);
        const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
        const int a = 2 * (i & 1);
        fadd2(acc[a], acc[a + 1], acc[a], acc[a + 1], e0, e1);
        if constexpr (C::TF32) {
          // P V reads P as tf32: rounded to nearest here (unbiased; the row
          // sum keeps the fp32 values, so the LSE stays exact to fp32)
          s[2 * i] = tf32_round_bits(f2u(e0));
          s[2 * i + 1] = tf32_round_bits(f2u(e1));
        } else {
          s[i] = pack_bf16x2(e0, e1);   // P packed in place: s[i] is already consumed
        }
      }
      if constexpr (C::TF32 && C::BN == 128) {
        tmem_st_x128(tS, s);
      } else if constexpr (C::TF32) {
        tmem_st_x64(tS, s);
      } else {
        if constexpr (C::SEP_P) {
          if (!pv_done) {
            ok = mbar_wait(bar_pvdone(wg), (j - 1) & 1, abort_flag, p.timeout_ns,
                           &g_cpattn_device_error, kErrWaitSoftmax);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
          }
          tmem_st_x64(tmem + lane_base + C::P_COL + wg * (C::BN / 2),
                      *reinterpret_cast<uint32_t(*)[64]>(&s[0]));
        } else {
          tmem_st_x64(tS, *reinterpret_cast<uint32_t(*)[64]>(&s[0]));
        }
      }
      l += (acc[0] + acc[1]) + (acc[2] + acc[3]);
      // the final merge reads the running state through bulk copies: this
      // thread's workspace stores are fenced for them a few key tiles into
      // the last chunk, once those stores have long drained
      const bool ws_ready =
          kPrefetchState && r_eff > 1 && w.c == r_eff - 1 && w.t == min(2, w.nt - 1);
      if (ws_ready) fence_proxy_async_global();
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_p(wg));
        if (ws_ready) mbar_arrive(bar_ws_ready(wg));
      }
      w.next(p);
    }
    if (ok) {
      // (prefetching: the running state's LSE is requested before the final
      // O is awaited)
      const bool merge = r_eff > 1;
      float lse_run = 0.f;
      if (kPrefetchState && merge && row_ok) lse_run = ws_lse_at(p, tile_id * kBM + tile_row);
      ok = mbar_wait(bar_o(wg), 0, abort_flag, p.timeout_ns, &g_cpattn_device_error,
                     kErrWaitSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      // bf16: the running state itself was fetched into shared memory
      const bool pre = kPrefetchState && merge && q_row0 + wg * kBM < p.s_q;
      if (ok && pre) {
        ok = mbar_wait(bar_ws(wg), 0, abort_flag, p.timeout_ns, &g_cpattn_device_error,
                       kErrWaitSoftmax);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        if (!kPrefetchState && merge && row_ok) lse_run = ws_lse_at(p, tile_id * kBM + tile_row);
        tc_fence_after();
        // (the state is read only where the epilogue merges, for rows of an
        // existing query tile: exactly where it was prefetched)
        const uint32_t pre0 = ws_piece(2 * wg, n_tiles), pre1 = ws_piece(2 * wg + 1, n_tiles);
        // the Q tiles are idle once every Q K has completed: each warp
        // stages its 32 output rows there (32 x D x out bytes = 8 KB)
        chunk_epilogue<T, D, kPrefetchState>(p, tO, r_eff - 1, r_eff, m_used, l, b, h, q_row,
                                             row_ok, tile_id, tile_row,
                                             smem + warp * 32 * D * sizeof(T), lse_run, smem,
                                             pre0, pre1);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename T, int D, bool CAUSAL, bool GROUPED>
cudaError_t launch_impl(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                        const AttnParams& p, cudaStream_t stream) {
  using C = Cfg<T, D>;
  auto kernel = attn_fwd_kernel<T, D, CAUSAL, GROUPED>;
  // Once per device and instantiation: the setmaxnreg split assumes exactly
  // kLaunchRegs registers per thread at launch (with fewer, the softmax
  // warpgroups' increase could never be granted: refuse to launch such a
  // build), and the dynamic shared-memory limit is raised.
  static std::atomic<unsigned long long> ready{0};   // bit d: device d is set up
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit == 0 || (ready.load(std::memory_order_acquire) & bit) == 0) {
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, kernel);
    if (e != cudaSuccess) return e;
    if (attr.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    ready.fetch_or(bit, std::memory_order_acq_rel);
  }
  const unsigned q_blocks = (p.s_q + C::NT * kBM - 1) / (C::NT * kBM);
  const dim3 grid = CAUSAL ? dim3(p.heads, p.batch, q_blocks) : dim3(q_blocks, p.heads, p.batch);
  // one CTA per SM is resident (its shared memory and registers fill one)
  AttnParams pl = p;
  pl.resident_ctas = sm_count();
  kernel<<<grid, kThreads, C::SMEM_BYTES, stream>>>(tm_q, tm_k, tm_v, pl);
  return cudaGetLastError();
}

// causal masking and the Ulysses Anything head skip are compiled in only
// where a launch asks for them, so the plain kernel carries neither
template <typename T, int D>
cudaError_t launch_variant(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, const AttnParams& p, cudaStream_t stream) {
  const bool grouped = p.group_count > 0;
  if (p.causal != 0)
    return grouped ? launch_impl<T, D, true, true>(tm_q, tm_k, tm_v, p, stream)
                   : launch_impl<T, D, true, false>(tm_q, tm_k, tm_v, p, stream);
  return grouped ? launch_impl<T, D, false, true>(tm_q, tm_k, tm_v, p, stream)
                 : launch_impl<T, D, false, false>(tm_q, tm_k, tm_v, p, stream);
}

}  // namespace

cudaError_t launch_attention(InDtype dt, int head_dim, const CUtensorMap& tm_q,
                             const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const AttnParams& p, cudaStream_t stream) {
  if (dt == InDtype::BF16 && head_dim == 128)
    return launch_variant<__nv_bfloat16, 128>(tm_q, tm_k, tm_v, p, stream);
  if (dt == InDtype::BF16 && head_dim == 64)
    return launch_variant<__nv_bfloat16, 64>(tm_q, tm_k, tm_v, p, stream);
  if (dt == InDtype::F32 && head_dim == 64)
    return launch_variant<float, 64>(tm_q, tm_k, tm_v, p, stream);
  if (dt == InDtype::F32 && head_dim == 128)
    return launch_variant<float, 128>(tm_q, tm_k, tm_v, p, stream);
  return cudaErrorInvalidValue;
}

int attn_kv_tile_rows(InDtype dt, int head_dim) {
  if (dt == InDtype::F32 && head_dim == 128) return Cfg<float, 128>::BN;
  return dt == InDtype::F32 ? Cfg<float, 64>::BN : Cfg<__nv_bfloat16, 128>::BN;
}

unsigned int* device_error_word() {
  static std::atomic<unsigned int*> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  unsigned int* w = cached[dev].load(std::memory_order_acquire);
  if (w == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_cpattn_device_error) != cudaSuccess) return nullptr;
    w = static_cast<unsigned int*>(ptr);
    cached[dev].store(w, std::memory_order_release);
  }
  return w;
}

cudaError_t read_and_clear_device_error(unsigned int* value, cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(value, g_cpattn_device_error, sizeof(unsigned int));
  if (e != cudaSuccess || *value == 0) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_cpattn_device_error, &zero, sizeof(unsigned int));
}

}  // namespace cpattn
