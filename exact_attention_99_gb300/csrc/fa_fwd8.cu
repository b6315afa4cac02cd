// FP8 (e4m3) forward pass of exact attention on sm_103a with incoherent
// processing: Q and K are multiplied by one random orthogonal matrix
// diag(signs) H_128 / sqrt(128) (H the Sylvester-Hadamard matrix), which
// leaves Q K^T unchanged but spreads outlier channels, then Q, K and V are
// scaled per (batch, head) by the power of two that maps their largest
// magnitude into (224, 448] and rounded to e4m3 (the FlashAttention-3 summary on news.hada.io, sections
// on FP8 and incoherent processing). Both GEMMs run as tcgen05.mma
// kind::f8f6f4 with fp32 accumulation; P is rounded to e4m3 for the P V
// GEMM; the softmax, its conditional rescale and the epilogue are the
// shared forward pipeline (fa_fwd_pipeline.cuh), with the per-head scales
// folded into the logit scale and into O.
//
//   fp8_rows_kernel<false> : per (batch, head) max |x| of Q M, K M and V.
//   fp8_rows_kernel<true>  : Q M, K M -> e4m3 rows (a quad of lanes per row;
//                       the Hadamard transform is a butterfly, five index
//                       bits inside a lane and two across the quad), and in
//                       the same launch V -> e4m3, transposed to [B, Hkv, d,
//                       keys] so that it is the K-major B operand of P V.
//   fa_fwd8_kernel    : the attention: the shared pipeline with the E4m3
//                       policy below (d = 128): S = Q8 K8^T and O += P8 V8
//                       from shared memory; P of each stage is staged as an
//                       e4m3 tile [128 rows x 128 keys] with the 128-byte
//                       swizzle.
#include <algorithm>

#include "fa_fwd_pipeline.cuh"

namespace fa {
namespace fwd8 {

using fwdp::Params;
using fwdp::Unit;

// e4m3 scale of a tensor from its per-head max |x| (float bits): the
// smallest power of two s with amax / s <= 448, so the largest magnitude maps
// into (224, 448]; 1 for an all-zero head. With amax = m 2^E (m in [1/2, 1))
// and 448 = 0.875 2^9 that is s = 2^(E - 9) when m <= 0.875, else 2^(E - 8).
// Dividing by a power of two is exact, so the e4m3 code of x is the
// round-to-nearest-even of x / s itself, whatever precision computes it.
__device__ __forceinline__ float amax_scale(unsigned bits) {
  const float a = __uint_as_float(bits);
  if (!(a > 0.0f)) return 1.0f;
  int E;
  const float m = frexpf(a, &E);
  return ldexpf(1.0f, m <= 0.875f ? E - 9 : E - 8);
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

// the signs of the 32 elements lane ql of a quad holds, as bits: bit j set
// where sign_{32 ql + j} = -1
__device__ __forceinline__ uint32_t had_sign_bits(int ql) {
  uint32_t bits = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) bits |= (had_sign(ql * 32 + j) < 0.0f ? 1u : 0u) << j;
  return bits;
}

// x with its sign flipped where bit j of `bits` is set (exact)
__device__ __forceinline__ float flip_sign(float x, uint32_t bits, int j) {
  return __uint_as_float(__float_as_uint(x) ^ (((bits >> j) & 1u) << 31));
}

// Rows of 128 values are handled by quads of lanes: lane ql = lane & 3 of a
// quad holds elements 32 ql .. 32 ql + 31 of its row. quad_transform
// multiplies the row by diag(signs) H_128 (the 1/sqrt(128) is left to the
// caller): a butterfly over the seven index bits, five inside the lane
// (bit 0 fused with the signs, `sgn` = had_sign_bits(ql)) and two across
// the quad.
__device__ __forceinline__ void quad_transform(float (&x)[32], uint32_t sgn, int ql) {
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float a = flip_sign(x[j], sgn, j), c = flip_sign(x[j + 1], sgn, j + 1);
    x[j] = a + c;
    x[j + 1] = a - c;
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

// Row pass over Q, K (and V when !QUANT) of one batch (blockIdx.z), rows
// [B, N, H] of 128 values:
//   !QUANT: per (batch, head) max |x M| (M the incoherent transform when
//           had; V untransformed), gathered per head in shared memory and
//           merged with one atomicMax on the (non-negative) float bits per
//           head and block; the maxima start at zero.
//   QUANT:  x M rounded to e4m3 with its head's scale, [rows x 128] bytes;
//           V rounded and transposed by the V blocks.
// Blocks [0, nbq) of a batch take Q, [nbq, nbq + nbk) K and the rest V (the
// host splits them in proportion to the tensors' rows, so that every block
// has about the same bytes to move). A warp takes 8 rows (a quad each)
// and keeps the loads of its next two groups of rows in flight while it
// transforms the current one; each tensor's blocks stride over its rows.
template <bool QUANT>
__global__ void __launch_bounds__(256, 2) fp8_rows_kernel(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                                       const __nv_bfloat16* v, int Nq, int Nk, int Hq, int Hkv,
                                                       int had, unsigned* amax_q, unsigned* amax_k,
                                                       unsigned* amax_v, uint8_t* q8, uint8_t* k8, int Nk_pad,
                                                       uint8_t* vt8, int nbq, int nbk) {
  extern __shared__ float head_sm[];  // QUANT: 1 / (scale sqrt(128)) per head; else max bits per head
  const int bi = blockIdx.x;
  const int t = bi < nbq ? 0 : (bi < nbq + nbk ? 1 : 2);
  const int bx = bi - (t == 0 ? 0 : (t == 1 ? nbq : nbq + nbk));
  const int nbx = t == 0 ? nbq : (t == 1 ? nbk : int(gridDim.x) - nbq - nbk);
  const int b = blockIdx.z;
  if (QUANT && t == 2) {
    // the V blocks stride over the (key tile, kv head) tiles of the batch
    const int nkt = Nk_pad / 128;
    for (int i = bx; i < nkt * Hkv; i += nbx) {
      const int kvh = i / nkt, kt = i - kvh * nkt;
      quant_v_tile(v, Nk, Hkv, Nk_pad, 1.0f / amax_scale(amax_v[b * Hkv + kvh]), vt8, kt, kvh, b);
    }
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int ql = lane & 3, quad = lane >> 2;
  const int H = t == 0 ? Hq : Hkv, N = t == 0 ? Nq : Nk;
  const __nv_bfloat16* x_b = (t == 0 ? q : (t == 1 ? k : v)) + size_t(b) * N * H * 128;
  unsigned* amax = (t == 0 ? amax_q : (t == 1 ? amax_k : amax_v)) + b * H;
  uint8_t* x8_b = (t == 0 ? q8 : k8) + size_t(b) * N * H * 128;
  const bool tr = had != 0 && t < 2;
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    if (QUANT) head_sm[h] = (tr ? kInvSqrt128 : 1.0f) / amax_scale(amax[h]);
    else reinterpret_cast<unsigned*>(head_sm)[h] = 0u;
  }
  const uint32_t sgn = had_sign_bits(ql);
  __syncthreads();
  const int R = N * H;
  const int step = nbx * nwarps;
  int g = bx * nwarps + warp;
  uint4 u[4], un[4];
  load_quad_row(x_b + size_t(g * 8 + quad) * 128, ql, g * 8 + quad < R, u);
  load_quad_row(x_b + size_t((g + step) * 8 + quad) * 128, ql, (g + step) * 8 + quad < R, un);
  for (; g * 8 < R; g += step) {
    const int r = g * 8 + quad, rn = r + 2 * step * 8;
    float x[32];
    unpack_quad_row(u, x);
#pragma unroll
    for (int c = 0; c < 4; ++c) u[c] = un[c];
    load_quad_row(x_b + size_t(rn) * 128, ql, rn < R, un);  // the group after next, in flight meanwhile
    if (tr) quad_transform(x, sgn, ql);
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


// The e4m3 operand policy of the shared forward pipeline (d = 128). A
// 128-row e4m3 tile of d = 128 is one 128-byte swizzle atom deep, so Q, K
// and V^T tiles are 16 KB and the K/V ring holds 8 slots. P cannot stay in
// TMEM (the TMEM operand of the .ts form is the A operand of 16-bit kinds
// only in the layout used here), so the softmax warps write P as e4m3 into
// a swizzled 16 KB shared tile per stage and the P V GEMM reads both
// operands from shared memory.
struct E4m3 {
  static constexpr bool kPair = false;
  static constexpr int D = 128;
  static constexpr int kTileBytes = 128 * D;   // one 128-row e4m3 tile of Q, K or V^T
  static constexpr int kSlotBytes = kTileBytes;  // a K/V ring slot holds one tile
  static constexpr int kSlots = 8;
  static constexpr int kPTileBytes = 128 * 128;  // e4m3 P of one stage [rows x keys]
  static constexpr int kSmemDyn = (2 + kSlots) * kTileBytes + 2 * kPTileBytes + fwdp::kStgBytes + 1024;

  __device__ __forceinline__ static void load_q(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int h, int row,
                                                int b) {
    tma_load_4d(dst, m, bar, 0, h, row, b);
  }
  // K tile [128 keys x d]
  __device__ __forceinline__ static void load_k(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int kvh, int key0,
                                                int b) {
    tma_load_4d(dst, m, bar, 0, kvh, key0, b);
  }
  // V^T tile [d x 128 keys]
  __device__ __forceinline__ static void load_v(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int kvh, int key0,
                                                int b) {
    tma_load_4d(dst, m, bar, key0, 0, kvh, b);
  }

  struct Desc {
    uint32_t q, k, p;  // descriptor low words of tile 0: Q, K (and V^T), P; all K-major
  };
  __device__ __forceinline__ static Desc make_desc(uint32_t sQa, uint32_t sKVa, uint32_t sPa) {
    return Desc{sdesc_lo(sQa, 16), sdesc_lo(sKVa, 16), sdesc_lo(sPa, 16)};
  }
  __host__ __device__ static constexpr uint32_t idesc_s() { return idesc_e4m3_f32(128, 128); }
  __host__ __device__ static constexpr uint32_t idesc_pv() { return idesc_e4m3_f32(128, D); }
  // S[stage s] = Q8_s K8^T: 32 e4m3 values (32 bytes) of d per MMA
  __device__ __forceinline__ static void issue_s(const Desc& dc, uint32_t d, int s, uint32_t kslot, uint32_t idS) {
    const uint32_t a0 = sdesc_step(dc.q, s * kTileBytes);
    const uint32_t b0 = sdesc_step(dc.k, kslot * kTileBytes);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_f8_lo(d, sdesc_step(a0, kk * 32), sdesc_step(b0, kk * 32), idS, kk > 0);
  }
  // O[stage s] (+)= P8_s V8: 32 keys per MMA, both operands in shared memory
  __device__ __forceinline__ static void issue_pv(const Desc& dc, uint32_t d, uint32_t, int s, uint32_t vslot,
                                                  bool acc, uint32_t idPV) {
    const uint32_t a0 = sdesc_step(dc.p, s * kPTileBytes);
    const uint32_t b0 = sdesc_step(dc.k, vslot * kTileBytes);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_f8_lo(d, sdesc_step(a0, kk * 32), sdesc_step(b0, kk * 32), idPV, (acc || kk > 0) ? 1u : 0u);
  }

  struct PK {
    uint32_t w[32];  // e4m3 P of one row, four keys per word
    uint32_t half_lo;
  };
  __device__ __forceinline__ static void pack_p(PK& pk, int c, float a, float b) {
    const uint32_t h2 = pack_e4m3x2(a, b);
    if (c & 1) pk.w[c >> 1] = pk.half_lo | (h2 << 16);
    else pk.half_lo = h2;
  }
  // row r of the stage's P tile: 8 chunks of 16 keys, 128-byte swizzle
  __device__ __forceinline__ static void store_p(const PK& pk, uint32_t, uint8_t* sP_s, int row) {
    uint8_t* prow = sP_s + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
      *reinterpret_cast<uint4*>(prow + ((ch ^ (row & 7)) << 4)) =
          make_uint4(pk.w[4 * ch], pk.w[4 * ch + 1], pk.w[4 * ch + 2], pk.w[4 * ch + 3]);
  }
  __device__ __forceinline__ static void publish_p() { fence_proxy_async_smem(); }  // read by the async proxy
  __device__ __forceinline__ static float logit_scale(const Params& p, const Unit& un) {
    return p.scale_log2 * amax_scale(p.amax_q[un.b * p.Hq + un.h]) * amax_scale(p.amax_k[un.b * p.Hkv + un.kvh]);
  }
  __device__ __forceinline__ static float out_scale(const Params& p, const Unit& un) {
    return amax_scale(p.amax_v[un.b * p.Hkv + un.kvh]);
  }
};

template <bool CAUSAL, int POLY>
__global__ void __launch_bounds__(fwdp::kThreads, 1)
    fa_fwd8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, const Params p) {
  fwdp::fwd_body<E4m3, CAUSAL, false, POLY>(tmQ, tmK, tmV, tmO, p);
}

// 4-D e4m3 tensor map with a 128-byte swizzle: dims and box innermost first
bool make_u8_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3,
                 uint64_t row_bytes, uint32_t box0, uint32_t box1, uint32_t box2) {
  const uint64_t dims[4] = {d0, d1, d2, d3};
  const uint64_t strides[3] = {row_bytes, row_bytes * d1, row_bytes * d1 * d2};
  const uint32_t box[4] = {box0, box1, box2, 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

using KernelFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const Params);

// the exp2 split (one column pair in every `poly` on the FMA polynomial; 0 =
// every exponential on the special-function unit)
template <bool CAUSAL>
KernelFn kernel_for(int poly) {
  switch (poly) {
    case 1: return fa_fwd8_kernel<CAUSAL, 1>;
    case 2: return fa_fwd8_kernel<CAUSAL, 2>;
    case 4: return fa_fwd8_kernel<CAUSAL, 4>;
    case 8: return fa_fwd8_kernel<CAUSAL, 8>;
    default: return fa_fwd8_kernel<CAUSAL, 0>;
  }
}

template <bool CAUSAL>
cudaError_t launch_t(const Problem& pb, void* o, float* lse, int incoherent, cudaStream_t stream) {
  constexpr int D = 128;
  using C = E4m3;
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
  Params p{};
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
  const int G = num_sms();
  fwdp::plan_units(p, pb, CAUSAL, G);
  const DebugCfg dc = debug_cfg();
  p.wait_limit_ns = dc.wait_limit_ns;
  p.inject = dc.inject;
  p.trace = dc.trace;
  p.status = status_word();
  const KernelFn kern = kernel_for<CAUSAL>(dc.poly_every);
  if (maps && p.status) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemDyn);
  } else {
    e = maps ? cudaErrorMemoryAllocation : cudaErrorInvalidValue;
  }
  if (e == cudaSuccess) e = cudaMemsetAsync(amax_q, 0, n_amax * 4, stream);
  if (e == cudaSuccess) {
    // about two resident blocks per SM, split between Q, K and V of each
    // batch element in proportion to their rows (at least one block each)
    const int Hmax = pb.Hq > pb.Hkv ? pb.Hq : pb.Hkv;
    const size_t hs = size_t(Hmax) * 4;
    const int per_b = std::max(3, (2 * G + pb.B - 1) / pb.B);
    const double rq = double(pb.Nq) * pb.Hq, rk = double(pb.Nk) * pb.Hkv, rall = rq + 2.0 * rk;
    const int nbq = std::max(1, int(per_b * rq / rall + 0.5)), nbk = std::max(1, int(per_b * rk / rall + 0.5));
    const int nbv = std::max(1, per_b - nbq - nbk);
    const dim3 grid(unsigned(nbq + nbk + nbv), 1, unsigned(pb.B));
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(pb.q);
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(pb.k);
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(pb.v);
    fp8_rows_kernel<false><<<grid, 256, hs, stream>>>(q, k, v, pb.Nq, pb.Nk, pb.Hq, pb.Hkv, incoherent, amax_q, amax_k,
                                                      amax_v, q8, k8, Nk_pad, vt8, nbq, nbk);
    fp8_rows_kernel<true><<<grid, 256, hs, stream>>>(q, k, v, pb.Nq, pb.Nk, pb.Hq, pb.Hkv, incoherent, amax_q, amax_k,
                                                     amax_v, q8, k8, Nk_pad, vt8, nbq, nbk);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    const int grid = p.n_items < G ? p.n_items : G;
    if (dc.ev_begin) cudaEventRecord(dc.ev_begin, stream);
    kern<<<grid, fwdp::kThreads, C::kSmemDyn, stream>>>(mq, mk, mv, mo, p);
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
