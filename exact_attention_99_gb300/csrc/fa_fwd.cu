// Forward pass of exact attention on sm_103a, bf16 operands (d = 64 or 128).
//
// The pipeline itself (work decomposition, warp roles, online softmax with
// its conditional rescale, epilogue) is fa_fwd_pipeline.cuh; this file gives
// it the bf16 operand policy and launches it:
//   * Q, K, V tiles of [128 rows x d] bf16, loaded by TMA as 64-column
//     atoms with the 128-byte swizzle; K/V ring of 4 slots (d = 128) or 8
//     (d = 64) in shared memory;
//   * S = Q K^T: tcgen05.mma kind::f16, both operands K-major in shared
//     memory, accumulator in TMEM;
//   * P (bf16 pairs) written back over the first 64 columns of its S in
//     TMEM and used from there as the A operand of O += P V (the .ts form),
//     V MN-major from shared memory.
// The method and its Blackwell mapping are described at the top of
// fa_fwd_pipeline.cuh (the post "FlashAttention v1", deep_school #630,
// sections "Тайлинг (Tiling)" and "Онлайн-Softmax"; the FlashAttention-4
// article on smntcn.com).
#include "fa_fwd_pipeline.cuh"

namespace fa {
namespace fwd {

using fwdp::Params;
using fwdp::Unit;

template <int D_>
struct Bf16 {
  static constexpr bool kPair = false;
  static constexpr int D = D_;
  static constexpr int kChunks = D / 64;          // 64-wide swizzle atoms along d
  static constexpr int kTileBytes = 128 * D * 2;  // one 128-row tile of Q, K or V
  static constexpr int kSlotBytes = kTileBytes;   // a K/V ring slot holds one tile
  static constexpr int kSlots = D == 128 ? 4 : 8;
  static constexpr int kPTileBytes = 0;  // P stays in TMEM
  static constexpr int kSmemDyn = (2 + kSlots) * kTileBytes + fwdp::kStgBytes + 1024;

  // L2 policy: Q is read once per unit (evict first); K and V tiles are read
  // by every unit of their head (evict last), which keeps more of them in L2
  // for the causal order's concurrent heads
  __device__ __forceinline__ static void load_q(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int h, int row,
                                                int b) {
    const uint64_t pol = l2_policy_evict_first();
#pragma unroll
    for (int c = 0; c < kChunks; ++c) tma_load_4d_hint(dst + c * 16384, m, bar, c * 64, h, row, b, pol);
  }
  __device__ __forceinline__ static void load_k(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int kvh, int key0,
                                                int b) {
    const uint64_t pol = l2_policy_evict_last();
#pragma unroll
    for (int c = 0; c < kChunks; ++c) tma_load_4d_hint(dst + c * 16384, m, bar, c * 64, kvh, key0, b, pol);
  }
  __device__ __forceinline__ static void load_v(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int kvh, int key0,
                                                int b) {
    load_k(dst, m, bar, kvh, key0, b);
  }

  struct Desc {
    uint32_t q, k, v;  // descriptor low words of tile 0: Q, K K-major; V MN-major
  };
  __device__ __forceinline__ static Desc make_desc(uint32_t sQa, uint32_t sKVa, uint32_t) {
    return Desc{sdesc_lo(sQa, 16), sdesc_lo(sKVa, 16), sdesc_lo(sKVa, 16384)};
  }
  __host__ __device__ static constexpr uint32_t idesc_s() { return idesc_bf16_f32(128, 128, 0, 0); }
  __host__ __device__ static constexpr uint32_t idesc_pv() { return idesc_bf16_f32(128, D, 0, 1); }
  // S[stage s] = Q_s K^T (K = d in steps of 16)
  __device__ __forceinline__ static void issue_s(const Desc& dc, uint32_t d, int s, uint32_t kslot, uint32_t idS) {
    const uint32_t a0 = sdesc_step(dc.q, s * kTileBytes);
    const uint32_t b0 = sdesc_step(dc.k, kslot * kTileBytes);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
      mma_ss_lo(d, sdesc_step(a0, koff), sdesc_step(b0, koff), idS, kk > 0);
    }
  }
  // O[stage s] (+)= P_s V (P in TMEM at a_tmem, K = 128 keys in steps of 16)
  __device__ __forceinline__ static void issue_pv(const Desc& dc, uint32_t d, uint32_t a_tmem, int, uint32_t vslot,
                                                  bool acc, uint32_t idPV) {
    const uint32_t b0 = sdesc_step(dc.v, vslot * kTileBytes);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ts_lo(d, a_tmem + kk * 8, sdesc_step(b0, kk * 2048), idPV, (acc || kk > 0) ? 1u : 0u);
  }

  struct PK {
    uint32_t w[64];  // bf16 pairs of one row of P
  };
  __device__ __forceinline__ static void pack_p(PK& pk, int c, float a, float b) { pk.w[c] = pack_bf16x2(a, b); }
  __device__ __forceinline__ static void store_p(const PK& pk, uint32_t t_s, uint8_t*, int) {
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_st16(t_s + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk.w[c * 16]));
  }
  __device__ __forceinline__ static void publish_p() {
    tmem_wait_st();
    tc_fence_before();
  }
  __device__ __forceinline__ static float logit_scale(const Params& p, const Unit&) { return p.scale_log2; }
  __device__ __forceinline__ static float out_scale(const Params&, const Unit&) { return 1.0f; }
};

// The same operands for a cluster of two CTAs (d = 128): one unit of 512
// query rows, stage s = 256 rows of which this CTA holds 128 (its Q tile);
// each CTA holds half of every K tile (64 keys, 16 KB) and half of every V
// tile (64 of the d columns, 16 KB) in a ring of 8 slots, and the even CTA
// issues M = 256 MMAs (cta_group::2) for both.
struct Bf16Pair {
  static constexpr bool kPair = true;
  static constexpr int D = 128;
  static constexpr int kTileBytes = 128 * D * 2;  // this CTA's 128-row Q tile of a stage
  static constexpr int kSlotBytes = 64 * D * 2;   // half a K tile or half a V tile
  static constexpr int kSlots = 8;
  static constexpr int kPTileBytes = 0;           // P stays in TMEM
  static constexpr int kSmemDyn = 2 * kTileBytes + kSlots * kSlotBytes + fwdp::kStgBytes + 1024;

  // completion counted on the even CTA's barrier (shared::cluster address)
  __device__ __forceinline__ static void load_q(uint8_t* dst, const CUtensorMap* m, uint32_t bar, int h, int row,
                                                int b) {
#pragma unroll
    for (int c = 0; c < 2; ++c) tma_load_4d_pair(dst + c * 16384, m, bar, c * 64, h, row, b);
  }
  // keys key0 + 64 rank .. +63 of the tile, both 64-column atoms of d (2 x 8 KB)
  __device__ __forceinline__ static void load_k(uint8_t* dst, const CUtensorMap* m, uint32_t bar, int kvh, int key0,
                                                int b, uint32_t rank) {
#pragma unroll
    for (int c = 0; c < 2; ++c) tma_load_4d_pair(dst + c * 8192, m, bar, c * 64, kvh, key0 + 64 * int(rank), b);
  }
  // all 128 keys of the tile, d columns 64 rank .. +63 (one 16 KB atom)
  __device__ __forceinline__ static void load_v(uint8_t* dst, const CUtensorMap* m, uint32_t bar, int kvh, int key0,
                                                int b, uint32_t rank) {
    tma_load_4d_pair(dst, m, bar, 64 * int(rank), kvh, key0, b);
  }

  struct Desc {
    uint32_t q, k, v;  // descriptor low words of slot / tile 0: Q, K K-major; V MN-major
  };
  __device__ __forceinline__ static Desc make_desc(uint32_t sQa, uint32_t sKVa, uint32_t) {
    return Desc{sdesc_lo(sQa, 16), sdesc_lo(sKVa, 16), sdesc_lo(sKVa, 16384)};
  }
  __host__ __device__ static constexpr uint32_t idesc_s() { return idesc_bf16_f32(256, 128, 0, 0); }
  __host__ __device__ static constexpr uint32_t idesc_pv() { return idesc_bf16_f32(256, D, 0, 1); }
  // S[stage s] of both CTAs = Q K^T (M = 256, N = 128 keys, K = d in steps of 16)
  __device__ __forceinline__ static void issue_s(const Desc& dc, uint32_t d, int s, uint32_t kslot, uint32_t idS) {
    const uint32_t a0 = sdesc_step(dc.q, s * kTileBytes);
    const uint32_t b0 = sdesc_step(dc.k, kslot * kSlotBytes);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t ka = (kk >> 2) * 16384 + (kk & 3) * 32, kb = (kk >> 2) * 8192 + (kk & 3) * 32;
      mma_ss_lo_pair(d, sdesc_step(a0, ka), sdesc_step(b0, kb), idS, kk > 0);
    }
  }
  // O[stage s] of both CTAs (+)= P V (P in each CTA's TMEM, K = 128 keys)
  __device__ __forceinline__ static void issue_pv(const Desc& dc, uint32_t d, uint32_t a_tmem, int, uint32_t vslot,
                                                  bool acc, uint32_t idPV) {
    const uint32_t b0 = sdesc_step(dc.v, vslot * kSlotBytes);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ts_lo_pair(d, a_tmem + kk * 8, sdesc_step(b0, kk * 2048), idPV, (acc || kk > 0) ? 1u : 0u);
  }

  using PK = typename Bf16<128>::PK;
  __device__ __forceinline__ static void pack_p(PK& pk, int c, float a, float b) { Bf16<128>::pack_p(pk, c, a, b); }
  __device__ __forceinline__ static void store_p(const PK& pk, uint32_t t_s, uint8_t* sp, int row) {
    Bf16<128>::store_p(pk, t_s, sp, row);
  }
  __device__ __forceinline__ static void publish_p() { Bf16<128>::publish_p(); }
  __device__ __forceinline__ static float logit_scale(const Params& p, const Unit& u) {
    return Bf16<128>::logit_scale(p, u);
  }
  __device__ __forceinline__ static float out_scale(const Params& p, const Unit& u) { return Bf16<128>::out_scale(p, u); }
};

template <bool CAUSAL, int POLY>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(fwdp::kThreads, 1)
    fa_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                       const Params p) {
  fwdp::fwd_body<Bf16Pair, CAUSAL, false, POLY>(tmQ, tmK, tmV, tmO, p);
}

template <int D, bool CAUSAL, bool WIN, int POLY>
__global__ void __launch_bounds__(fwdp::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, const Params p) {
  fwdp::fwd_body<Bf16<D>, CAUSAL, WIN, POLY>(tmQ, tmK, tmV, tmO, p);
}

template <int D, bool CAUSAL, bool WIN, int POLY>
cudaError_t launch_t(const Problem& pb, void* o, float* lse, cudaStream_t stream) {
  using K = Bf16<D>;
  CUtensorMap mq, mk, mv, mo;
  if (!make_bshd_map(&mq, pb.q, pb.B, pb.Nq, pb.Hq, D, 128) || !make_bshd_map(&mk, pb.k, pb.B, pb.Nk, pb.Hkv, D, 128) ||
      !make_bshd_map(&mv, pb.v, pb.B, pb.Nk, pb.Hkv, D, 128) || !make_bshd_map(&mo, o, pb.B, pb.Nq, pb.Hq, D, 32))
    return cudaErrorInvalidValue;
  Params p{};
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.B = pb.B;
  p.Hq = pb.Hq;
  p.Hkv = pb.Hkv;
  p.Nq = pb.Nq;
  p.Nk = pb.Nk;
  p.group = pb.Hq / pb.Hkv;
  p.scale_log2 = fabsf(exp_scale_log2(pb.scale));
  p.neg_s = pb.scale < 0.0f ? 1u : 0u;
  p.wl = normalize_window(pb.window_left, pb.Nq, pb.Nk);
  p.wr = pb.causal ? 0 : normalize_window(pb.window_right, pb.Nq, pb.Nk);
  const int G = num_sms();
  fwdp::plan_units(p, pb, CAUSAL, G);
  const DebugCfg dc = debug_cfg();
  p.wait_limit_ns = dc.wait_limit_ns;
  p.inject = dc.inject;
  p.trace = dc.trace;
  p.status = status_word();
  if (!p.status) return cudaErrorMemoryAllocation;
  auto kern = fa_fwd_kernel<D, CAUSAL, WIN, POLY>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, K::kSmemDyn);
  if (e != cudaSuccess) return e;
  const int grid = p.n_items < G ? p.n_items : G;
  if (dc.ev_begin) cudaEventRecord(dc.ev_begin, stream);
  kern<<<grid, fwdp::kThreads, K::kSmemDyn, stream>>>(mq, mk, mv, mo, p);
  e = cudaGetLastError();
  if (dc.ev_end) cudaEventRecord(dc.ev_end, stream);
  return e;
}

// CTA pairs (d = 128, no window): a grid of 2 x (pairs) CTAs in clusters of
// two, units of 512 query rows
template <bool CAUSAL, int POLY>
cudaError_t launch_pair(const Problem& pb, void* o, float* lse, cudaStream_t stream) {
  using K = Bf16Pair;
  constexpr int D = 128;
  CUtensorMap mq, mk, mv, mo;
  if (!make_bshd_map(&mq, pb.q, pb.B, pb.Nq, pb.Hq, D, 128) || !make_bshd_map(&mk, pb.k, pb.B, pb.Nk, pb.Hkv, D, 64) ||
      !make_bshd_map(&mv, pb.v, pb.B, pb.Nk, pb.Hkv, D, 128) || !make_bshd_map(&mo, o, pb.B, pb.Nq, pb.Hq, D, 32))
    return cudaErrorInvalidValue;
  Params p{};
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
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
  const int pairs = num_sms() / 2;
  fwdp::plan_units(p, pb, CAUSAL, pairs, 512);
  const DebugCfg dc = debug_cfg();
  p.wait_limit_ns = dc.wait_limit_ns;
  p.inject = dc.inject;
  p.trace = dc.trace;
  p.status = status_word();
  if (!p.status) return cudaErrorMemoryAllocation;
  auto kern = fa_fwd_pair_kernel<CAUSAL, POLY>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, K::kSmemDyn);
  if (e != cudaSuccess) return e;
  const int grid = 2 * (p.n_items < pairs ? p.n_items : pairs);
  if (dc.ev_begin) cudaEventRecord(dc.ev_begin, stream);
  kern<<<grid, fwdp::kThreads, K::kSmemDyn, stream>>>(mq, mk, mv, mo, p);
  e = cudaGetLastError();
  if (dc.ev_end) cudaEventRecord(dc.ev_end, stream);
  return e;
}

// the exp2 split (one column pair in every `poly` on the FMA polynomial)
// for the unwindowed kernels; 0 = every exponential on the special-function
// unit
template <int D, bool CAUSAL>
cudaError_t launch_poly(const Problem& p, void* o, float* lse, int poly, cudaStream_t stream) {
  switch (poly) {
    case 1: return launch_t<D, CAUSAL, false, 1>(p, o, lse, stream);
    case 2: return launch_t<D, CAUSAL, false, 2>(p, o, lse, stream);
    case 4: return launch_t<D, CAUSAL, false, 4>(p, o, lse, stream);
    case 8: return launch_t<D, CAUSAL, false, 8>(p, o, lse, stream);
    default: return launch_t<D, CAUSAL, false, 0>(p, o, lse, stream);
  }
}

}  // namespace fwd

cudaError_t launch_fwd(const Problem& p, void* o, float* lse, cudaStream_t stream) {
  // three kernels per head dim: no mask, the plain causal mask, any window
  const bool m = p.masked();
  const bool win = m && !p.plain_causal();
  const int poly = debug_cfg().poly_every;
  if (p.d == 128) {
    if (win) return fwd::launch_t<128, true, true, 0>(p, o, lse, stream);
    if (debug_cfg().cta_pairs) return m ? fwd::launch_pair<true, 0>(p, o, lse, stream) : fwd::launch_pair<false, 0>(p, o, lse, stream);
    return m ? fwd::launch_poly<128, true>(p, o, lse, poly, stream)
             : fwd::launch_poly<128, false>(p, o, lse, poly, stream);
  }
  if (win) return fwd::launch_t<64, true, true, 0>(p, o, lse, stream);
  return m ? fwd::launch_poly<64, true>(p, o, lse, poly, stream) : fwd::launch_poly<64, false>(p, o, lse, poly, stream);
}

}  // namespace fa
