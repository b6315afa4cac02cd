// FP8 (e4m3) forward pass of exact attention on sm_103a with incoherent
// processing: Q and K are multiplied by one random orthogonal matrix
// diag(signs) H_128 / sqrt(128) (H the Sylvester-Hadamard matrix), which
// leaves Q K^T unchanged but spreads outlier channels, then Q, K and V are
// scaled per (batch, head) so that their largest magnitude maps to 448 and
// rounded to e4m3 (the FlashAttention-3 summary on news.hada.io, sections
// on FP8 and incoherent processing). Both GEMMs run as tcgen05.mma
// kind::f8f6f4 with fp32 accumulation; P is rounded to e4m3 for the P V
// GEMM; the softmax, its conditional rescale and the epilogue are those of
// the bf16 kernel (fa_fwd.cu), with the per-head scales folded into the
// logit scale and into O.
//
//   fp8_rows_kernel<false> : per (batch, head) max |x| of Q M, K M and V.
//   fp8_rows_kernel<true>  : Q M, K M -> e4m3 rows (a quad of lanes per row;
//                       the Hadamard transform is a butterfly, five index
//                       bits inside a lane and two across the quad), and in
//                       the same launch V -> e4m3, transposed to [B, Hkv, d,
//                       keys] so that it is the K-major B operand of P V.
//   fa_fwd8_kernel    : the attention: the warp roles, unit schedule and
//                       TMEM layout of the bf16 forward (d = 128), with
//                       S = Q8 K8^T and O += P8 V8 from shared memory: P of
//                       each stage is staged as an e4m3 tile [128 rows x 128
//                       keys] with the 128-byte swizzle.
#include <cuda_bf16.h>
#include <cmath>

#include "fa_internal.h"
#include "sm103_math.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace fwd8 {

constexpr int kThreads = 512;
constexpr int kMaxSlots = 8;

// Share of exponentials done by the polynomial: one column pair in every
// kPolyEvery goes to the FMA pipes (0 = all on the special-function unit).
#ifndef FA_POLY_EVERY
#define FA_POLY_EVERY 0
#endif
constexpr int kPolyEvery = FA_POLY_EVERY;

// Rescale threshold (log2 units). A row's reference max m, to which O and l
// are scaled, moves to the new row max only when that max exceeds m by more
// than kTau; otherwise the block is exponentiated against the stale m, so
// every unnormalised probability stays below 2^kTau. The result is the same
// for any kTau (O, l and LSE all use the same m); kTau = 0 moves m on every
// growth.
#ifndef FA_RESCALE_TAU
#define FA_RESCALE_TAU 8.0f
#endif
constexpr float kTau = FA_RESCALE_TAU;

template <int D>
struct Cfg {
  static constexpr int kChunks = 1;           // one 128-byte swizzle atom holds a whole e4m3 row of d = 128
  static constexpr int kTileBytes = 128 * D;  // one 128-row e4m3 tile of Q, K, V^T or P
  static constexpr int kSlots = 8;
  static constexpr int kStgBytes = 16384;  // O staging: 4 warps x [32 rows x 64 cols] bf16
  static constexpr int kSmemDyn = (2 + kSlots + 2) * kTileBytes + kStgBytes + 1024;
  static constexpr uint32_t kOCol0 = 256;
};

struct Params {
  __nv_bfloat16* o;
  float* lse;
  // per (batch, head) max |x| of Q M, K M, V (float bits); the e4m3 scale
  // of a tensor is amax / 448 (1 for an all-zero head)
  const unsigned* amax_q;
  const unsigned* amax_k;
  const unsigned* amax_v;
  int B, Hq, Hkv, Nq, Nk;
  int group;
  float scale_log2;  // |scale| * log2(e) (2^-100 for a zero scale)
  uint32_t neg_s;     // 1 for a negative scale: S is computed as (-Q) K^T
  int n_mblocks;
  int n_units;
  // Row-split tail (non-causal): the units [n_full, n_units) of the last,
  // partly filled round run as two work items each, one per 128-row stage,
  // on twice as many CTAs; the work items are the n_full whole units
  // followed by those halves, n_items in all.
  int n_items, n_full;
  // Visible keys of query row i (masked kernels): i + off - wl <= j <=
  // i + off + wr with off = Nk - Nq; a negative bound is no limit. Causal
  // is wl = -1, wr = 0.
  int wl, wr;
  unsigned long long wait_limit_ns;
  int inject;
  unsigned* status;
  unsigned long long* trace;  // optional pipeline trace
};

// Trace points (fa_trace); a step is the CTA's running key-tile counter
// across its units:
//   MMA         0 PV0 issued, 1 PV1 issued, 2 S0(next) issued, 3 S1(next) issued
//   softmax s   4+3s S ready, 5+3s alpha published, 6+3s P stored
//   correction  10+2s alpha seen, 11+2s O released for PV
//   producer    14 K slot free, 15 V slot free
// and, in the last step slot (kernel events): 0 entry, 1 set-up done,
// 2 epilogue start (last unit), 6 teardown start, 7 exit.
constexpr int kEv = kTraceSteps - 1;

struct __align__(8) Ctl {
  uint64_t q_full[2];
  uint64_t q_empty;
  uint64_t kv_full[kMaxSlots];
  uint64_t kv_empty[kMaxSlots];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t alpha_full[2];
  uint64_t o_ready[2];
  uint64_t o_full[2];
  uint64_t stats_full[2];
  uint64_t stats_empty[2];
  uint64_t drain;
  float alpha[2][128];
  float stat_l[2][128];
  float stat_m[2][128];
  uint32_t tmem_base;
  uint32_t abort;
};

struct Unit {
  int b, h, kvh, row0;
  int kb0;    // first key tile of the unit
  int a[2];   // stage s visits key tiles kb0 + a[s] .. kb0 + a[s] + n[s] - 1
  int n[2];
  int nb;     // key tiles the unit loads: max over stages of a[s] + n[s]
  bool rows[2];
  __device__ __forceinline__ bool active(int s, int j) const { return j >= a[s] && j < a[s] + n[s]; }
};

// Window bounds as a kernel sees them: the plain causal kernels (WIN false)
// fix them at compile time (no left bound, right bound 0).
template <bool WIN>
__device__ __forceinline__ int win_l(const Params& p) { return WIN ? p.wl : -1; }
template <bool WIN>
__device__ __forceinline__ int win_r(const Params& p) { return WIN ? p.wr : 0; }

template <bool CAUSAL, bool WIN>
__device__ __forceinline__ Unit decode_unit(const Params& p, int item) {
  Unit x;
  int u = item, half = -1;
  if (!CAUSAL && item >= p.n_full) {
    const int k = item - p.n_full;
    u = p.n_full + (k >> 1);
    half = k & 1;
  }
  const int bh_count = p.B * p.Hq;
  // causal: rounds over all heads, longest units (last query blocks) first;
  // non-causal: all query blocks of one head in a row, so the CTAs that run
  // together share K and V through L2
  int r, bh;
  if (CAUSAL) {
    r = u / bh_count;
    bh = u - r * bh_count;
  } else {
    bh = u / p.n_mblocks;
    r = u - bh * p.n_mblocks;
  }
  const int mb = CAUSAL ? (p.n_mblocks - 1 - r) : r;
  x.b = bh / p.Hq;
  x.h = bh - x.b * p.Hq;
  x.kvh = x.h / p.group;
  x.row0 = mb * 256;
  const int off = p.Nk - p.Nq;
  const int nkb = (p.Nk + 127) >> 7;
  int t0[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int r0 = x.row0 + s * 128;
    x.rows[s] = r0 < p.Nq;
    t0[s] = 0;
    if (!x.rows[s]) {
      x.n[s] = 0;
    } else if (!CAUSAL) {
      x.n[s] = nkb;
    } else {
      // keys seen by any row of the stage: [lo, hi]
      const int rl = min(r0 + 127, p.Nq - 1);
      const int wl = win_l<WIN>(p), wr = win_r<WIN>(p);
      const int lo = wl >= 0 ? max(0, r0 + off - wl) : 0;
      const int hi = wr >= 0 ? min(p.Nk - 1, rl + off + wr) : p.Nk - 1;
      if (hi < lo) {
        x.n[s] = 0;
      } else {
        t0[s] = lo >> 7;
        x.n[s] = (hi >> 7) - t0[s] + 1;
      }
    }
  }
  if (half >= 0) {  // one stage of a row-split unit; the other item has the other rows
    x.n[half ^ 1] = 0;
    x.rows[half ^ 1] = false;
  }
  // stage 1's rows follow stage 0's, so its key range starts and ends no
  // earlier, and (both bounds being >= 0 or absent) leaves no gap after it
  x.kb0 = x.n[0] > 0 ? t0[0] : t0[1];
#pragma unroll
  for (int s = 0; s < 2; ++s) x.a[s] = x.n[s] > 0 ? t0[s] - x.kb0 : 0;
  x.nb = max(x.a[0] + x.n[0], x.a[1] + x.n[1]);
  return x;
}

// Static snake order over rounds of gridDim.x units (longest first when
// causal): CTA c takes unit c in even rounds and G-1-c in odd rounds.
__device__ __forceinline__ int unit_at(int round, int c) {
  const int G = gridDim.x;
  return round * G + ((round & 1) ? (G - 1 - c) : c);
}

// e4m3 scale of a tensor from its per-head max |x| (float bits)
__device__ __forceinline__ float amax_scale(unsigned bits) {
  const float a = __uint_as_float(bits);
  return a > 0.0f ? a * (1.0f / 448.0f) : 1.0f;
}

// two floats to e4m3 (round to nearest even, saturating at +-448); lo in
// bits 0-7, hi in bits 8-15
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// instruction descriptor of kind::f8f6f4 with e4m3 A and B (both K-major),
// fp32 accumulation
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T for e4m3 operands (32 per K step);
// descriptors given by their low words (the high word is kSdescHi)
__device__ __forceinline__ void mma_f8_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "mov.b64 da, {%1, %5};\n\t"
      "mov.b64 db, {%2, %5};\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(kSdescHi)
      : "memory");
}

// sign_i of the incoherent transform: -1 where bit 31 of
// 2654435769 * (i + 1) mod 2^32 is set
__device__ __forceinline__ float had_sign(int i) {
  return ((2654435769u * uint32_t(i + 1)) >> 31) ? -1.0f : 1.0f;
}

// Rows of 128 values are handled by quads of lanes: lane ql = lane & 3 of a
// quad holds elements 32 ql .. 32 ql + 31 of its row. quad_transform
// multiplies the row by diag(signs) H_128 (the 1/sqrt(128) is left to the
// caller): a butterfly over the seven index bits, five inside the lane
// (bit 0 fused with the signs sg[j] = sign_{32 ql + j}) and two across the
// quad.
__device__ __forceinline__ void quad_transform(float (&x)[32], const float (&sg)[32], int ql) {
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float a = x[j] * sg[j];
    x[j] = fmaf(x[j + 1], sg[j + 1], a);
    x[j + 1] = fmaf(-x[j + 1], sg[j + 1], a);
  }
#pragma unroll
  for (int m = 2; m < 32; m <<= 1) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j & m) continue;
      const float a = x[j], c = x[j + m];
      x[j] = a + c;
      x[j + m] = a - c;
    }
  }
#pragma unroll
  for (int m = 1; m < 4; m <<= 1) {
    const float sel = (ql & m) ? -1.0f : 1.0f;  // upper partner: o - x, lower: x + o
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = fmaf(sel, x[j], __shfl_xor_sync(0xffffffffu, x[j], m));
  }
}

__device__ __forceinline__ void load_quad_row(const __nv_bfloat16* row, int ql, bool valid, uint4 (&u)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    u[c] = valid ? reinterpret_cast<const uint4*>(row + ql * 32)[c] : make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ void unpack_quad_row(const uint4 (&u)[4], float (&x)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u[c]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h2[e]);
      x[c * 8 + e * 2] = f.x;
      x[c * 8 + e * 2 + 1] = f.y;
    }
  }
}

// V rounded to e4m3 and transposed to [B, Hkv, 128 (d), Nk_pad (keys)], one
// 128-key tile (kt) of one (batch b, kv head) per call by a 256-thread
// block: lane l of warp w takes keys 4l .. 4l+3 and d = 16w .. 16w+15 (one
// 32-byte sector of each key row), so that each store of the warp writes 128
// contiguous bytes of one d row. Keys past Nk are written as zeros.
__device__ __forceinline__ void quant_v_tile(const __nv_bfloat16* v, int Nk, int Hkv, int Nk_pad, float inv,
                                             uint8_t* vt8, int kt, int kvh, int b) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint4 u[4][2];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int gk = kt * 128 + 4 * lane + j;
    const uint4* src = reinterpret_cast<const uint4*>(v + ((size_t(b) * Nk + gk) * Hkv + kvh) * 128 + warp * 16);
    u[j][0] = gk < Nk ? src[0] : make_uint4(0, 0, 0, 0);
    u[j][1] = gk < Nk ? src[1] : make_uint4(0, 0, 0, 0);
  }
  uint8_t* dst = vt8 + ((size_t(b) * Hkv + kvh) * 128 + warp * 16) * Nk_pad + kt * 128 + 4 * lane;
#pragma unroll
  for (int dd = 0; dd < 16; ++dd) {
    float f[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&u[j][dd >> 3]);
      f[j] = __bfloat162float(h[dd & 7]) * inv;
    }
    *reinterpret_cast<uint32_t*>(dst + size_t(dd) * Nk_pad) = pack_e4m3x2(f[0], f[1]) | (pack_e4m3x2(f[2], f[3]) << 16);
  }
}

constexpr float kInvSqrt128 = 0.08838834764831845f;

// Row pass over Q, K (and V when !QUANT) of one batch (blockIdx.z), tensor
// t = blockIdx.y (0 = Q, 1 = K, 2 = V), rows [B, N, H] of 128 values:
//   !QUANT: per (batch, head) max |x M| (M the incoherent transform when
//           had; V untransformed), gathered per head in shared memory and
//           merged with one atomicMax on the (non-negative) float bits per
//           head and block; the maxima start at zero.
//   QUANT:  x M rounded to e4m3 with its head's scale, [rows x 128] bytes.
// A warp takes 8 rows (a quad each) and loads its next group of rows before
// transforming the current one; the grid strides over the batch's rows.
template <bool QUANT>
__global__ void __launch_bounds__(256, 2) fp8_rows_kernel(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                                       const __nv_bfloat16* v, int Nq, int Nk, int Hq, int Hkv,
                                                       int had, unsigned* amax_q, unsigned* amax_k,
                                                       unsigned* amax_v, uint8_t* q8, uint8_t* k8, int Nk_pad,
                                                       uint8_t* vt8) {
  extern __shared__ float head_sm[];  // QUANT: 1 / (scale sqrt(128)) per head; else max bits per head
  if (QUANT && blockIdx.y == 2) {
    // the V transpose runs in the same launch: blockIdx.y = 2 strides over
    // the (key tile, kv head) tiles of batch blockIdx.z
    const int b = blockIdx.z, nkt = Nk_pad / 128;
    for (int t = blockIdx.x; t < nkt * Hkv; t += gridDim.x) {
      const int kvh = t / nkt, kt = t - kvh * nkt;
      quant_v_tile(v, Nk, Hkv, Nk_pad, 1.0f / amax_scale(amax_v[b * Hkv + kvh]), vt8, kt, kvh, b);
    }
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int ql = lane & 3, quad = lane >> 2;
  const int t = blockIdx.y, b = blockIdx.z;
  const int H = t == 0 ? Hq : Hkv, N = t == 0 ? Nq : Nk;
  const __nv_bfloat16* x_b = (t == 0 ? q : (t == 1 ? k : v)) + size_t(b) * N * H * 128;
  unsigned* amax = (t == 0 ? amax_q : (t == 1 ? amax_k : amax_v)) + b * H;
  uint8_t* x8_b = (t == 0 ? q8 : k8) + size_t(b) * N * H * 128;
  const bool tr = had != 0 && t < 2;
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    if (QUANT) head_sm[h] = (tr ? kInvSqrt128 : 1.0f) / amax_scale(amax[h]);
    else reinterpret_cast<unsigned*>(head_sm)[h] = 0u;
  }
  float sg[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) sg[j] = had_sign(ql * 32 + j);
  __syncthreads();
  const int R = N * H;
  const int step = gridDim.x * nwarps;
  int g = blockIdx.x * nwarps + warp;
  uint4 u[4];
  load_quad_row(x_b + size_t(g * 8 + quad) * 128, ql, g * 8 + quad < R, u);
  for (; g * 8 < R; g += step) {
    const int r = g * 8 + quad, rn = r + step * 8;
    float x[32];
    unpack_quad_row(u, x);
    load_quad_row(x_b + size_t(rn) * 128, ql, rn < R, u);  // the next group's row, in flight meanwhile
    if (tr) quad_transform(x, sg, ql);
    const int h = r % H;
    if (QUANT) {
      const float inv = r < R ? head_sm[h] : 0.0f;
      uint32_t w[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        w[c] = pack_e4m3x2(x[4 * c] * inv, x[4 * c + 1] * inv) |
               (pack_e4m3x2(x[4 * c + 2] * inv, x[4 * c + 3] * inv) << 16);
      if (r < R) {
        uint4* dst = reinterpret_cast<uint4*>(x8_b + size_t(r) * 128 + ql * 32);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    } else {
      float m = 0.0f;
#pragma unroll
      for (int j = 0; j < 32; ++j) m = fmaxf(m, fabsf(x[j]));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      if (tr) m *= kInvSqrt128;
      if (ql == 0 && r < R) atomicMax(reinterpret_cast<unsigned*>(head_sm) + h, __float_as_uint(m));
    }
  }
  if (!QUANT) {
    __syncthreads();
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
      const unsigned bits = reinterpret_cast<const unsigned*>(head_sm)[h];
      if (bits) atomicMax(amax + h, bits);
    }
  }
}

template <int D, bool CAUSAL, bool WIN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Ctl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                               // 2 tiles
  uint8_t* sKV = smem + 2 * C::kTileBytes;          // kSlots tiles: K [keys x d] and V^T [d x keys]
  uint8_t* sP = sKV + C::kSlots * C::kTileBytes;    // 2 tiles: e4m3 P of each stage [rows x keys]
  uint8_t* sStg = sP + 2 * C::kTileBytes;           // O staging

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wg = warp >> 2;
  volatile uint32_t* abort_flag = &ctl.abort;
  const uint64_t LIM = p.wait_limit_ns;
  if (threadIdx.x == 0) trace_stamp(p.trace, kEv, 0);

  if (threadIdx.x == 0) {
    ctl.abort = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl.q_full[s], 1);
      mbar_init(&ctl.s_full[s], 1);
      mbar_init(&ctl.p_full[s], 4);
      mbar_init(&ctl.alpha_full[s], 4);
      mbar_init(&ctl.o_ready[s], 4);
      mbar_init(&ctl.o_full[s], 1);
      mbar_init(&ctl.stats_full[s], 4);
      mbar_init(&ctl.stats_empty[s], 4);
    }
    mbar_init(&ctl.q_empty, 1);
    mbar_init(&ctl.drain, 1);
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(&ctl.kv_full[i], 1);
      mbar_init(&ctl.kv_empty[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(&ctl.tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 12 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  if (threadIdx.x == 0) trace_stamp(p.trace, kEv, 1);

  if (wg <= 1) {
    // ------------------------------------------------------------ softmax
    setmaxnreg_inc<176>();
    const int s = wg;
    const int row = ((warp & 3) << 5) + lane;
    const uint32_t t_s = tmem + (uint32_t(warp & 3) << 21) + uint32_t(s * 128);  // lane quarter + S columns
    uint32_t ph_s = 0, ph_se = 0;
    int blk = 0;  // running key-tile counter (trace only)
    float sl = p.scale_log2;
    bool ok = true;
    for (int rnd = 0; ok; ++rnd) {
      const int u = unit_at(rnd, blockIdx.x);
      if (u >= p.n_items) break;
      const Unit un = decode_unit<CAUSAL, WIN>(p, u);
      const int n = un.n[s];
      const int blk0 = blk;
      blk += un.nb;
      if (n == 0) continue;
      const int rg = un.row0 + s * 128 + row;  // global query row
      sl = p.scale_log2 * amax_scale(p.amax_q[un.b * p.Hq + un.h]) * amax_scale(p.amax_k[un.b * p.Hkv + un.kvh]);
      const int off = p.Nk - p.Nq;
      const int r0 = un.row0 + s * 128, rl = min(r0 + 127, p.Nq - 1);  // the stage's rows
      const int wl = win_l<WIN>(p), wr = win_r<WIN>(p);
      float m_run = -INFINITY, l_run = 0.0f;
      for (int j = 0; j < n; ++j) {
        if (!mbar_wait_bounded(&ctl.s_full[s], ph_s, abort_flag, LIM)) { ok = false; break; }
        ph_s ^= 1;
        if (row == 0) trace_stamp(p.trace, blk0 + j, 4 + 3 * s);
        tc_fence_after();
        uint32_t x[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(t_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&x[c * 32]));
        tmem_wait_ld();
        const int kb = (un.kb0 + un.a[s] + j) * 128;
        // a tile needs masking when it reaches past the keys or crosses a
        // window edge of some row of the stage
        const bool need_mask = (kb + 127 >= p.Nk) ||
                               (CAUSAL && ((wr >= 0 && kb + 127 > r0 + off + wr) || (wl >= 0 && kb < rl + off - wl)));
        if (need_mask) {
          int lim = p.Nk - kb;  // columns [lo_c, lim) of this row are visible
          int lo_c = 0;
          if (CAUSAL && wr >= 0) lim = min(lim, rg + off + wr + 1 - kb);
          if (CAUSAL && wl >= 0) lo_c = rg + off - wl - kb;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim || c < lo_c) x[c] = f2u(-INFINITY);
        }
        float mA = -INFINITY, mB = -INFINITY, mC = -INFINITY, mD = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; c += 8) {
          mA = fmax3(mA, u2f(x[c]), u2f(x[c + 1]));
          mB = fmax3(mB, u2f(x[c + 2]), u2f(x[c + 3]));
          mC = fmax3(mC, u2f(x[c + 4]), u2f(x[c + 5]));
          mD = fmax3(mD, u2f(x[c + 6]), u2f(x[c + 7]));
        }
        const float mx = fmaxf(fmaxf(mA, mB), fmaxf(mC, mD));
        const float m_cand = fmaxf(m_run, mx * sl);
        const float m_new = (m_cand > m_run + kTau) ? m_cand : m_run;
        const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
        const float alpha = ex2_mufu(m_run - m_use);
        ctl.alpha[s][row] = alpha;
        __syncwarp();
        if (row == 0) trace_stamp(p.trace, blk0 + j, 5 + 3 * s);
        if (lane == 0) mbar_arrive(&ctl.alpha_full[s]);

        const uint64_t sl2 = pack2(sl, sl);
        const uint64_t nm2 = pack2(-m_use, -m_use);
        uint64_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;
        uint32_t pk[32];  // e4m3 P, four keys per word
        uint32_t half_lo = 0;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          uint64_t y = ffma2(pack2(u2f(x[2 * c]), u2f(x[2 * c + 1])), sl2, nm2);
          float a, b;
          unpack2(y, a, b);
          if (kPolyEvery > 0 && (c % (kPolyEvery > 0 ? kPolyEvery : 1)) == (kPolyEvery - 1)) {
            exp2_poly_pair(a, b);
          } else {
            a = ex2_mufu(a);
            b = ex2_mufu(b);
          }
          const uint64_t pr = pack2(a, b);
          if ((c & 3) == 0) acc0 = c == 0 ? pr : fadd2(acc0, pr);
          if ((c & 3) == 1) acc1 = c == 1 ? pr : fadd2(acc1, pr);
          if ((c & 3) == 2) acc2 = c == 2 ? pr : fadd2(acc2, pr);
          if ((c & 3) == 3) acc3 = c == 3 ? pr : fadd2(acc3, pr);
          const uint32_t h2 = pack_e4m3x2(a, b);
          if (c & 1) pk[c >> 1] = half_lo | (h2 << 16);
          else half_lo = h2;
        }
        {
          // row r of the stage's P tile: 8 chunks of 16 keys, 128-byte swizzle
          uint8_t* prow = sP + s * C::kTileBytes + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(prow + ((ch ^ (row & 7)) << 4)) =
                make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        }
        const uint64_t acc = fadd2(fadd2(acc0, acc1), fadd2(acc2, acc3));
        float la, lb;
        unpack2(acc, la, lb);
        l_run = fmaf(l_run, alpha, la + lb);
        m_run = m_new;
        fence_proxy_async_smem();  // P is read by the tensor core (async proxy)
        __syncwarp();
        if (row == 0) trace_stamp(p.trace, blk0 + j, 6 + 3 * s);
        if (lane == 0) mbar_arrive(&ctl.p_full[s]);
      }
      if (!ok) break;
      // final row statistics for the epilogue
      if (!mbar_wait_bounded(&ctl.stats_empty[s], ph_se ^ 1, abort_flag, LIM)) { ok = false; break; }
      ph_se ^= 1;
      ctl.stat_l[s][row] = l_run;
      ctl.stat_m[s][row] = m_run;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.stats_full[s]);
    }
  } else if (wg == 2) {
    // ------------------------------------------------ correction + epilogue
    setmaxnreg_dec<80>();
    const int wq = warp & 3;
    const int row = (wq << 5) + lane;
    const uint32_t t_lane = tmem + (uint32_t(wq) << 21);
    uint32_t ph_a[2] = {0, 0}, ph_st[2] = {0, 0}, ph_of[2] = {0, 0};
    int blk = 0;
    bool ok = true;
    for (int rnd = 0; ok; ++rnd) {
      const int u = unit_at(rnd, blockIdx.x);
      if (u >= p.n_items) break;
      const Unit un = decode_unit<CAUSAL, WIN>(p, u);
      const int blk0 = blk;
      blk += un.nb;
      for (int j = 0; j < un.nb && ok; ++j) {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (!un.active(s, j)) continue;
          if (!mbar_wait_bounded(&ctl.alpha_full[s], ph_a[s], abort_flag, LIM)) { ok = false; break; }
          ph_a[s] ^= 1;
          if (row == 0) trace_stamp(p.trace, blk0 + j, 10 + 2 * s);
          const float a = ctl.alpha[s][row];
          if (j > un.a[s] && __any_sync(0xffffffffu, a < 1.0f)) {
            tc_fence_after();
            const uint32_t t_o = t_lane + C::kOCol0 + uint32_t(s * D);
            const uint64_t a2 = pack2(a, a);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t v[32];
              tmem_ld32(t_o + c * 32, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                float lo, hi;
                unpack2(fmul2(pack2(u2f(v[i]), u2f(v[i + 1])), a2), lo, hi);
                v[i] = f2u(lo);
                v[i + 1] = f2u(hi);
              }
              tmem_st32(t_o + c * 32, v);
            }
            tmem_wait_st();
          }
          tc_fence_before();
          __syncwarp();
          if (row == 0) trace_stamp(p.trace, blk0 + j, 11 + 2 * s);
          if (lane == 0) mbar_arrive(&ctl.o_ready[s]);
        }
      }
      if (!ok) break;
      // epilogue: O / l -> bf16, LSE
      if (row == 0) trace_stamp(p.trace, kEv, 2);
#pragma unroll 1
      for (int s = 0; s < 2; ++s) {
        if (!un.rows[s]) continue;
        const int rg = un.row0 + s * 128 + row;
        const bool valid = rg < p.Nq;
        __nv_bfloat16* dst = p.o + ((size_t(un.b) * p.Nq + rg) * p.Hq + un.h) * D;
        float* lse_dst = p.lse + (size_t(un.b) * p.Hq + un.h) * p.Nq + rg;
        if (un.n[s] == 0) {
          if (valid) {
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(dst)[c] = z;
            *lse_dst = -INFINITY;
          }
          continue;
        }
        if (!mbar_wait_bounded(&ctl.stats_full[s], ph_st[s], abort_flag, LIM)) { ok = false; break; }
        ph_st[s] ^= 1;
        const float l = ctl.stat_l[s][row];
        const float m = ctl.stat_m[s][row];
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.stats_empty[s]);
        if (!mbar_wait_bounded(&ctl.o_full[s], ph_of[s], abort_flag, LIM)) { ok = false; break; }
        ph_of[s] ^= 1;
        tc_fence_after();
        const float inv = l > 0.0f ? amax_scale(p.amax_v[un.b * p.Hkv + un.kvh]) / l : 0.0f;
        const uint32_t t_o = t_lane + C::kOCol0 + uint32_t(s * D);
        // each warp stages its 32 rows x 64 columns (bf16, 128-byte swizzle)
        // and writes them with one TMA store; rows past Nq are clipped
        uint8_t* stg = sStg + wq * 4096;
        const int wrow0 = un.row0 + s * 128 + wq * 32;
#pragma unroll 1
        for (int hf = 0; hf < D / 64; ++hf) {
          if (lane == 0) bulk_wait_read_all();  // the previous store has read the buffer
          __syncwarp();
#pragma unroll 1
          for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t v[32];
            tmem_ld32(t_o + hf * 64 + c2 * 32, v);
            tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(u2f(v[2 * i]) * inv, u2f(v[2 * i + 1]) * inv);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              *reinterpret_cast<uint4*>(stg + lane * 128 + (((c2 * 4 + i) ^ (lane & 7)) << 4)) =
                  make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && wrow0 < p.Nq) {
            tma_store_4d(&tmO, stg, hf * 64, un.h, wrow0, un.b);
            bulk_commit();
          }
        }
        if (valid) *lse_dst = l > 0.0f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        tc_fence_before();
      }
    }
    if (lane == 0) bulk_wait_all();  // stores complete (and staging reads done) before the CTA exits
  } else {
    setmaxnreg_dec<80>();
  }
  if (warp == 12) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t kv_it = 0, ph_qe = 0;
      int blk = 0;
      bool first = true, ok = true;
      bool injected = false;
      for (int rnd = 0; ok; ++rnd) {
        const int u = unit_at(rnd, blockIdx.x);
        if (u >= p.n_items) break;
        const Unit un = decode_unit<CAUSAL, WIN>(p, u);
        if (un.nb == 0) continue;
        if (!first) {
          if (!mbar_wait_bounded(&ctl.q_empty, ph_qe, abort_flag, LIM)) { ok = false; break; }
          ph_qe ^= 1;
        }
        first = false;
        for (int s = 0; s < 2; ++s) {
          if (un.n[s] == 0) continue;
          mbar_arrive_expect_tx(&ctl.q_full[s], C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(sQ + s * C::kTileBytes, &tmQ, &ctl.q_full[s], 0, un.h, un.row0 + s * 128, un.b);
        }
        for (int j = 0; j < un.nb && ok; ++j) {
#pragma unroll 1
          for (int t = 0; t < 2; ++t) {
            const uint32_t slot = kv_it % C::kSlots;
            const uint32_t ph = ((kv_it / C::kSlots) & 1) ^ 1;
            if (!mbar_wait_bounded(&ctl.kv_empty[slot], ph, abort_flag, LIM)) { ok = false; break; }
            trace_stamp(p.trace, blk + j, 14 + t);
            ++kv_it;
            if (p.inject == 1 && !injected) {  // test hook: never deliver this tile
              injected = true;
              continue;
            }
            mbar_arrive_expect_tx(&ctl.kv_full[slot], C::kTileBytes);
            if (t == 0)  // K tile [128 keys x d]
              tma_load_4d(sKV + slot * C::kTileBytes, &tmK, &ctl.kv_full[slot], 0, un.kvh, (un.kb0 + j) * 128, un.b);
            else  // V^T tile [d x 128 keys]
              tma_load_4d(sKV + slot * C::kTileBytes, &tmV, &ctl.kv_full[slot], (un.kb0 + j) * 128, 0, un.kvh, un.b);
          }
        }
        blk += un.nb;
      }
      if (*abort_flag) {
        // let copies already in flight land before shared memory is released
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
      }
    }
  } else if (warp == 13) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // a negative scale negates A (Q) in S = Q K^T: bit 13 of the instruction descriptor
      const uint32_t idS = idesc_e4m3_f32(128, 128) | (p.neg_s << 13);
      constexpr uint32_t idPV = idesc_e4m3_f32(128, D);
      const uint32_t sQa = smem_u32(sQ), sKVa = smem_u32(sKV), sPa = smem_u32(sP);
      uint32_t kv_it = 0, ph_q[2] = {0, 0}, ph_p[2] = {0, 0}, ph_o[2] = {0, 0};
      int blk = 0;
      bool ok = true;
      // Tile descriptors are built once; a K step is one add of a constant,
      // so MMAs issue back to back (the tensor core idles otherwise).
      const uint32_t dQ = sdesc_lo(sQa, 16);   // Q tiles, K-major (K = d)
      const uint32_t dK = sdesc_lo(sKVa, 16);  // K and V^T tiles, K-major (K = d, keys)
      const uint32_t dP = sdesc_lo(sPa, 16);   // P tiles, K-major (K = keys)
      auto issue_S = [&](int s, uint32_t kslot) {
        const uint32_t a0 = sdesc_step(dQ, s * C::kTileBytes);
        const uint32_t b0 = sdesc_step(dK, kslot * C::kTileBytes);
        const uint32_t d = tmem + uint32_t(s * 128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // 32 e4m3 values (32 bytes) of d per MMA
          mma_f8_lo(d, sdesc_step(a0, kk * 32), sdesc_step(b0, kk * 32), idS, kk > 0);
      };
      auto issue_PV = [&](int s, uint32_t vslot, bool acc) {
        const uint32_t a0 = sdesc_step(dP, s * C::kTileBytes);
        const uint32_t b0 = sdesc_step(dK, vslot * C::kTileBytes);
        const uint32_t d = tmem + C::kOCol0 + uint32_t(s * D);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // 32 keys per MMA
          mma_f8_lo(d, sdesc_step(a0, kk * 32), sdesc_step(b0, kk * 32), idPV, (acc || kk > 0) ? 1u : 0u);
      };
      auto wait_kv = [&](uint32_t& slot) -> bool {
        slot = kv_it % C::kSlots;
        const bool r = mbar_wait_bounded(&ctl.kv_full[slot], (kv_it / C::kSlots) & 1, abort_flag, LIM);
        ++kv_it;
        return r;
      };
      for (int rnd = 0; ok; ++rnd) {
        const int u = unit_at(rnd, blockIdx.x);
        if (u >= p.n_items) break;
        const Unit un = decode_unit<CAUSAL, WIN>(p, u);
        if (un.nb == 0) continue;
        for (int s = 0; s < 2 && ok; ++s) {
          if (un.n[s] == 0) continue;
          ok = mbar_wait_bounded(&ctl.q_full[s], ph_q[s], abort_flag, LIM);
          ph_q[s] ^= 1;
        }
        uint32_t kslot = 0, vslot = 0;
        if (!ok || !wait_kv(kslot)) { ok = false; break; }
        tc_fence_after();
        for (int s = 0; s < 2; ++s) {
          if (!un.active(s, 0)) continue;
          issue_S(s, kslot);
          mma_commit(&ctl.s_full[s]);
        }
        mma_commit(&ctl.kv_empty[kslot]);
        if (un.nb == 1) mma_commit(&ctl.q_empty);
        for (int j = 0; j < un.nb && ok; ++j) {
          if (!wait_kv(vslot)) { ok = false; break; }
          const bool nxt = j + 1 < un.nb;
          if (nxt && !wait_kv(kslot)) { ok = false; break; }
          const int last_v = un.active(1, j) ? 1 : 0;  // the last stage that reads V_j
          for (int s = 0; s < 2; ++s) {
            if (un.active(s, j)) {
              if (!mbar_wait_bounded(&ctl.p_full[s], ph_p[s], abort_flag, LIM)) { ok = false; break; }
              ph_p[s] ^= 1;
              if (!mbar_wait_bounded(&ctl.o_ready[s], ph_o[s], abort_flag, LIM)) { ok = false; break; }
              ph_o[s] ^= 1;
              tc_fence_after();
              trace_stamp(p.trace, blk + j, s);
              issue_PV(s, vslot, j > un.a[s]);
              if (j == un.a[s] + un.n[s] - 1) mma_commit(&ctl.o_full[s]);
              // V_j is free once the last PV reading it completes: release it
              // before the next S is issued so the refill starts earlier
              if (s == last_v) mma_commit(&ctl.kv_empty[vslot]);
            }
            if (nxt && un.active(s, j + 1)) {  // S of the next tile (a stage's first S when it starts there)
              tc_fence_after();
              trace_stamp(p.trace, blk + j, 2 + s);
              issue_S(s, kslot);
              mma_commit(&ctl.s_full[s]);
            }
          }
          if (!ok) break;
          if (nxt) mma_commit(&ctl.kv_empty[kslot]);
          if (j + 2 == un.nb) mma_commit(&ctl.q_empty);
        }
        blk += un.nb;
      }
      if (*abort_flag) {
        // drain the tensor pipe before TMEM is released
        mma_commit(&ctl.drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&ctl.drain), 0) && globaltimer_ns() - t0 < 100000000ull) {
        }
      }
    }
  }

  // ------------------------------------------------------------- teardown
  if (warp == 8 && lane == 0) trace_stamp(p.trace, kEv, 6);
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 13) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0 && ctl.abort) atomicOr(p.status, kDevTimeout);
  if (threadIdx.x == 0) trace_stamp(p.trace, kEv, 7);
}

// 4-D e4m3 tensor map with a 128-byte swizzle: dims and box innermost first
bool make_u8_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3,
                 uint64_t row_bytes, uint32_t box0, uint32_t box1, uint32_t box2) {
  const uint64_t dims[4] = {d0, d1, d2, d3};
  const uint64_t strides[3] = {row_bytes, row_bytes * d1, row_bytes * d1 * d2};
  const uint32_t box[4] = {box0, box1, box2, 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <bool CAUSAL>
cudaError_t launch_t(const Problem& pb, void* o, float* lse, int incoherent, cudaStream_t stream) {
  constexpr int D = 128;
  using C = Cfg<D>;
  const int Nk_pad = (pb.Nk + 127) / 128 * 128;
  const size_t q8_bytes = size_t(pb.B) * pb.Nq * pb.Hq * D, k8_bytes = size_t(pb.B) * pb.Nk * pb.Hkv * D;
  const size_t vt_bytes = size_t(pb.B) * pb.Hkv * D * Nk_pad;
  const size_t n_amax = size_t(pb.B) * (pb.Hq + 2 * pb.Hkv);
  cudaMemPool_t pool = workspace_pool();
  if (pool == nullptr) return cudaErrorMemoryAllocation;
  void* ws = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&ws, q8_bytes + k8_bytes + vt_bytes + n_amax * 4, pool, stream);
  if (e != cudaSuccess) return e;
  uint8_t* q8 = static_cast<uint8_t*>(ws);
  uint8_t* k8 = q8 + q8_bytes;
  uint8_t* vt8 = k8 + k8_bytes;
  unsigned* amax_q = reinterpret_cast<unsigned*>(vt8 + vt_bytes);
  unsigned* amax_k = amax_q + size_t(pb.B) * pb.Hq;
  unsigned* amax_v = amax_k + size_t(pb.B) * pb.Hkv;
  CUtensorMap mq, mk, mv, mo;
  bool maps = make_u8_map(&mq, q8, D, pb.Hq, pb.Nq, pb.B, D, 128, 1, 128) &&
              make_u8_map(&mk, k8, D, pb.Hkv, pb.Nk, pb.B, D, 128, 1, 128) &&
              make_u8_map(&mv, vt8, pb.Nk, D, pb.Hkv, pb.B, Nk_pad, 128, 128, 1) &&
              make_bshd_map(&mo, o, pb.B, pb.Nq, pb.Hq, D, 32);
  Params p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.amax_q = amax_q;
  p.amax_k = amax_k;
  p.amax_v = amax_v;
  p.B = pb.B;
  p.Hq = pb.Hq;
  p.Hkv = pb.Hkv;
  p.Nq = pb.Nq;
  p.Nk = pb.Nk;
  p.group = pb.Hq / pb.Hkv;
  p.scale_log2 = fabsf(exp_scale_log2(pb.scale));
  p.neg_s = pb.scale < 0.0f ? 1u : 0u;
  p.wl = -1;
  p.wr = CAUSAL ? 0 : -1;
  p.n_mblocks = (pb.Nq + 255) / 256;
  p.n_units = p.n_mblocks * pb.B * pb.Hq;
  const int G = num_sms();
  const int T = p.n_units % G;
  const int n_split = (!CAUSAL && T > 0 && 2 * T <= G && pb.Nq > 128) ? T : 0;
  p.n_full = p.n_units - n_split;
  p.n_items = p.n_full + 2 * n_split;
  const DebugCfg dc = debug_cfg();
  p.wait_limit_ns = dc.wait_limit_ns;
  p.inject = dc.inject;
  p.trace = dc.trace;
  p.status = status_word();
  auto kern = fa_fwd8_kernel<D, CAUSAL, false>;
  if (maps && p.status) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemDyn);
  } else {
    e = maps ? cudaErrorMemoryAllocation : cudaErrorInvalidValue;
  }
  if (e == cudaSuccess) e = cudaMemsetAsync(amax_q, 0, n_amax * 4, stream);
  if (e == cudaSuccess) {
    // about two resident blocks per SM over all (tensor, batch) columns
    const int Hmax = pb.Hq > pb.Hkv ? pb.Hq : pb.Hkv;
    const size_t hs = size_t(Hmax) * 4;
    const int bx_a = (2 * G + 3 * pb.B - 1) / (3 * pb.B), bx_q = (2 * G + 2 * pb.B - 1) / (2 * pb.B);
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(pb.q);
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(pb.k);
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(pb.v);
    fp8_rows_kernel<false><<<dim3(bx_a, 3, pb.B), 256, hs, stream>>>(q, k, v, pb.Nq, pb.Nk, pb.Hq, pb.Hkv, incoherent,
                                                                      amax_q, amax_k, amax_v, q8, k8, Nk_pad, vt8);
    fp8_rows_kernel<true><<<dim3(bx_q, 3, pb.B), 256, hs, stream>>>(q, k, v, pb.Nq, pb.Nk, pb.Hq, pb.Hkv, incoherent,
                                                                     amax_q, amax_k, amax_v, q8, k8, Nk_pad, vt8);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    const int grid = p.n_items < G ? p.n_items : G;
    if (dc.ev_begin) cudaEventRecord(dc.ev_begin, stream);
    kern<<<grid, kThreads, C::kSmemDyn, stream>>>(mq, mk, mv, mo, p);
    e = cudaGetLastError();
    if (dc.ev_end) cudaEventRecord(dc.ev_end, stream);
  }
  const cudaError_t f = cudaFreeAsync(ws, stream);
  return e != cudaSuccess ? e : f;
}

}  // namespace fwd8

cudaError_t launch_fwd8(const Problem& p, void* o, float* lse, int incoherent, cudaStream_t stream) {
  return p.causal ? fwd8::launch_t<true>(p, o, lse, incoherent, stream)
                  : fwd8::launch_t<false>(p, o, lse, incoherent, stream);
}

}  // namespace fa
