// Backward pass of exact attention on sm_103a.
//
// Method: the probabilities are recomputed tile by tile from the saved
// log-sum-exp instead of being stored (the FlashAttention-3 summary on
// news.hada.io, section "Resumo do FlashAttention": tiling and
// recomputation), and the intermediates of the five GEMMs stay in tensor
// memory to cut shared-memory traffic (the FlashAttention-4 article on
// smntcn.com: backward is bound by shared-memory traffic; intermediates are
// kept in the 256 KB of tensor memory per SM).
//
// Gradients of L = sum(dO * O) with P = softmax(scale * Q K^T):
//   dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,  dS = P o (dP - D),
//   dQ = scale * dS K,  dK = scale * dS^T Q.
//
// Kernels:
//   bwd_pre  : D_i and LSE * log2(e) per query row (padded to whole tiles),
//              zero the fp32 dQ accumulator.
//   bwd_main : persistent, one CTA per SM, running work units round robin:
//              a unit is one (batch, kv head, 128-key tile) -- a pair of key
//              tiles (j, n-1-j) when causal, so the units have the same work
//              -- and each tile ("item") loops over the query heads of the GQA
//              group x 128-row query tiles that see it. Near an item's end
//              the next item's K and V are prefetched into L2.
//     warps 0-7  compute: two warps per lane quarter, each thread one key
//                row and 64 of the tile's 128 query columns; P^T =
//                2^(S^T*scale*log2e - LSE*log2e), dS^T = P^T o (dP^T - D)
//     warps 8-11 dQ drain and the dK/dV epilogue. d = 128: dQ leaves TMEM
//                into a shared-memory staging buffer and is added to the fp32
//                accumulator by TMA bulk reductions, and dK/dV leave through
//                the same buffer by TMA stores; d = 64: coalesced fp32
//                reductions.
//     Shared memory: K and V tiles (resident), a 2-slot Q ring, a 1-slot dO
//     ring (its last reader, dV, runs early in each step), the dS^T tile,
//     the dQ staging buffer, LSE/D vectors.
//     warp 12    TMA producer, warp 13 MMA issuer, warps 14-15 idle
//     TMEM: S^T [0,128) with P^T (bf16) over its first 64 columns;
//           dP^T [128,256), reused for dQ once read; dV [256,256+d);
//           dK [256+d, 256+2d).
//     MMA order per query tile i:
//       dP(i), dV(i) += P^T dO, S(i+1), dK(i) += dS^T Q, dQ(i) = dS K
//   bwd_post : dQ = bf16(scale * accumulator) in BSHD (a row-by-row pass for
//              d = 128, a transpose through shared memory for d = 64).
//   The accumulator is fp32, [B*Hq, Nq_pad, d] (d innermost) for d = 128
//   and [B*Hq, d, Nq_pad] (query index innermost) for d = 64.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "sm103_math.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace bwd {

constexpr int kThreads = 512;
constexpr int kPrefetchSteps = 4;  // the next item's K/V go to L2 this many steps before an item ends

template <int D>
struct Cfg {
  static constexpr int kTile = 128 * D * 2;  // K, V, Q or dO tile of 128 rows
  static constexpr int kDsBytes = 128 * 128 * 2;
  static constexpr int kStgBytes = D == 128 ? 32768 : 0;  // dQ staging: 4 warps x 2 boxes of [32 q][32 d] fp32
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTile;
  static constexpr int kOffQ = 2 * kTile;   // 2 slots
  static constexpr int kOffDO = 4 * kTile;  // 1 slot
  static constexpr int kOffDs = 5 * kTile;
  static constexpr int kOffStg = kOffDs + kDsBytes;
  static constexpr int kOffVec = kOffStg + kStgBytes;  // [2 stages][lse2 128 | delta 128] fp32
  static constexpr int kOffCtl = kOffVec + 2 * 2 * 128 * 4;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
};

// A CTA's work: one or two key tiles ("items") of one (batch, kv head),
// each visited against every query tile that sees it, for every query head
// of the group.
struct Item {
  int j;      // key tile
  int i0;     // first query tile that sees it
  int nq;     // query tiles per head
  int h0;     // first query head of the group that the item takes
  int nh;     // query heads it takes: the whole group, or one (a tail piece)
  int tt;     // tail tile index of a piece (its dK/dV are partial sums), else -1
  int steps;  // nh * nq
};
struct Work {
  int b, kvh, n_items;
  Item it[2];
};

// The maps the dQ drain writes through, in one kernel parameter so that one
// base address serves them all: the fp32 dQ accumulator (reductions), dK
// and dV (stores), and the fp32 partial dK/dV of tail pieces (stores).
struct OutMaps {
  CUtensorMap acc, dk, dv;
  CUtensorMap dkv;  // tail pieces: fp32 [B*Hkv*n_tail*group][2][128][D], boxes of 32 rows x 32 d
};

struct Cur {  // a warp's current item, kept in shared memory (see below)
  Item I;
  int b, kvh;
};

struct __align__(8) Ctl {
  uint64_t kv_full;
  uint64_t q_full[2], q_empty[2], do_full, do_empty;
  uint64_t vec_full[2];
  uint64_t vec_empty[2];
  uint64_t kv_empty, acc_empty;
  uint64_t s_full, p_full, dp_full, ds_full, dq_full, dq_empty, acc_full, drain;
  uint32_t tmem_base;
  uint32_t abort;
  Cur cur[kThreads / 32];
};

struct Params {
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* dq_acc;        // fp32: [B*Hq, Nq_pad, D] for D = 128, [B*Hq, D, Nq_pad] for D = 64
  const float* lse2;    // [B*Hq, Nq_pad]: LSE*log2(e), +inf for padded / empty rows
  const float* delta;   // [B*Hq, Nq_pad]
  int B, Hq, Hkv, Nq, Nk, Nq_pad, group, n_ktiles, n_qtiles;
  // causal pairs (see decode): of the n_ktiles / 2 pairs (j, n-1-j) of each
  // head, the last n_split (those nearest the middle, both tiles about half
  // a pair's work) run as two single-tile CTAs each, after every whole pair
  int n_split;
  // GQA tail pieces (d = 128): the single tiles are split further, one unit
  // per query head of the group; such a unit stores its partial dK/dV in
  // its own slot of the fp32 buffer [B*Hkv, n_tail, group, 2 (dV, dK), 128,
  // D], which a last pass sums in a fixed order (so dK, dV stay
  // deterministic). n_tail = 2 * n_split + (n_ktiles & 1) tiles per kv head.
  int head_split, n_tail;
  // work units (a pair or a single key tile of one (batch, kv head)); the
  // CTAs are persistent: CTA c runs units c, c + gridDim.x, ...
  int n_units;
  // masked kernels: key j visible to query row i iff i + off - wl <= j <=
  // i + off + wr (off = Nk - Nq); a negative bound is no limit; causal is
  // wl = -1, wr = 0
  int wl, wr;
  float scale, scale_log2;
  unsigned long long wait_limit_ns;
  unsigned* status;
  unsigned long long* trace;  // optional pipeline trace
};

// Trace points (fa_trace), per query-tile step:
//   MMA      0 dP issued, 1 P ready (dV next), 2 next Q ready (S next), 3 dS ready (dK next), 4 dQ issued
//   compute  5 LSE/D ready, 6 S^T ready, 7 P^T stored, 8 dP^T ready, 9 dS^T stored
//   drain    10 dQ ready, 11 dQ columns released, 12 reductions issued
//   producer 13 Q slot free, 14 dO slot free

// Window bounds as a kernel sees them: the plain causal kernels (WIN false)
// fix them at compile time (no left bound, right bound 0).
template <bool WIN>
__device__ __forceinline__ int win_l(const Params& p) { return WIN ? p.wl : -1; }
template <bool WIN>
__device__ __forceinline__ int win_r(const Params& p) { return WIN ? p.wr : 0; }

template <bool CAUSAL, bool WIN, bool PIECES>
__device__ __forceinline__ Work decode(const Params& p, int unit) {
  Work w;
  int r;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    w.it[k].h0 = 0;
    w.it[k].nh = p.group;
    w.it[k].tt = -1;
  }
  if (CAUSAL && win_l<WIN>(p) < 0) {
    // key tiles j and n-1-j share a CTA: the pair always has n+1 query-tile
    // steps (for Nq = Nk), so all these CTAs carry the same work; heads in a
    // row. After them come single tiles: both tiles of the n_split pairs of
    // each head nearest the middle (pair index n/2 - n_split .. n/2 - 1),
    // then the middle tile when n is odd; each has about half a pair's work
    // and fills what would otherwise be a partly idle last wave of pairs.
    const int half = p.n_ktiles / 2, kept = half - p.n_split;
    const int whole = p.B * p.Hkv * kept;
    if (unit < whole) {
      r = unit / kept;
      const int pr = unit - r * kept;
      w.it[0].j = pr;
      w.it[1].j = p.n_ktiles - 1 - pr;
      w.n_items = 2;
    } else {
      const int hs = PIECES ? p.group : 1;  // units per tail tile
      const int per_head = p.n_tail * hs;
      const int s = unit - whole;
      r = s / per_head;
      const int t = s - r * per_head;
      const int tt = t / hs;  // the query heads of one tile are consecutive units
      const int pr = kept + (tt >> 1);
      w.it[0].j = tt < 2 * p.n_split ? ((tt & 1) ? p.n_ktiles - 1 - pr : pr) : half;
      if (PIECES) {
        w.it[0].h0 = t - tt * hs;
        w.it[0].nh = 1;
        w.it[0].tt = tt;
      }
      w.it[1].j = 0;
      w.n_items = 1;
    }
  } else {
    // all key tiles of one head in a row, so concurrent CTAs share Q, dO and
    // the dQ accumulator in L2 (also for windows with a left bound, where
    // every key tile has about the same number of query tiles)
    r = unit / p.n_ktiles;
    w.it[0].j = unit - r * p.n_ktiles;
    w.it[1].j = 0;
    w.n_items = 1;
  }
  w.b = r / p.Hkv;
  w.kvh = r - w.b * p.Hkv;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    // query rows that see some key of the tile: [lo, hi]
    const int off = p.Nk - p.Nq;
    const int k0 = w.it[k].j * 128, k1 = min(k0 + 127, p.Nk - 1);
    int lo = 0, hi = p.Nq - 1;
    if (CAUSAL && win_r<WIN>(p) >= 0) lo = max(lo, k0 - off - win_r<WIN>(p));
    if (CAUSAL && win_l<WIN>(p) >= 0) hi = min(hi, k1 - off + win_l<WIN>(p));
    int i0 = 0, nq = 0;
    if (lo <= hi && k < w.n_items) {
      i0 = lo >> 7;
      nq = (hi >> 7) - i0 + 1;
    }
    w.it[k].i0 = i0;
    w.it[k].nq = nq;
    w.it[k].steps = nq * w.it[k].nh;
  }
  return w;
}

// (a select, not an indexed load: keeps a Work in registers)
__device__ __forceinline__ Item pick(const Work& w, int k) { return k == 0 ? w.it[0] : w.it[1]; }

// The k-th item of this (persistent) CTA: item k & 1 of unit blockIdx.x +
// (k >> 1) * gridDim.x. Returns 0 past the last unit, 1 when the unit has no
// such item (a single), 2 with I, b, kvh set.
template <bool CAUSAL, bool WIN, bool PIECES>
__device__ __forceinline__ int item_at(const Params& p, int k, Item& I, int& b, int& kvh) {
  const int u = int(blockIdx.x) + (k >> 1) * int(gridDim.x);
  if (u >= p.n_units) return 0;
  const Work w = decode<CAUSAL, WIN, PIECES>(p, u);
  if ((k & 1) >= w.n_items) return 1;
  I = pick(w, k & 1);
  b = w.b;
  kvh = w.kvh;
  return 2;
}

// swizzled (128-byte) byte offset of element (row, col) in a [128 rows x 128
// cols] bf16 tile stored as two 64-column atoms
__device__ __forceinline__ uint32_t sw128_off(int row, int col) {
  const int chunk = col >> 6, c = col & 63;
  return chunk * 16384 + (row >> 3) * 1024 + (row & 7) * 128 + ((((c >> 3) ^ (row & 7))) << 4) + ((c & 7) << 1);
}

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// PIECES: the tail singles are split per query head (d = 128, GQA, paired
// causal); without it no item is a piece and that code is compiled out.
template <int D, bool CAUSAL, bool WIN, bool PIECES>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ OutMaps out, const Params p) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctl& ctl = *reinterpret_cast<Ctl*>(smem + C::kOffCtl);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wg = warp >> 2;
  const uint64_t LIM = p.wait_limit_ns;
  volatile uint32_t* abort_flag = &ctl.abort;

  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzle atoms need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicOr(p.status, kDevTimeout);
    return;
  }
  if (threadIdx.x == 0) {
    ctl.abort = 0;
    mbar_init(&ctl.kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.q_full[i], 1);
      mbar_init(&ctl.q_empty[i], 1);
    }
    mbar_init(&ctl.do_full, 1);
    mbar_init(&ctl.do_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.vec_full[i], 1);
      mbar_init(&ctl.vec_empty[i], 8);
    }
    mbar_init(&ctl.s_full, 1);
    mbar_init(&ctl.p_full, 8);
    mbar_init(&ctl.dp_full, 1);
    mbar_init(&ctl.ds_full, 8);
    mbar_init(&ctl.dq_full, 1);
    mbar_init(&ctl.dq_empty, 4);
    mbar_init(&ctl.acc_full, 1);
    mbar_init(&ctl.kv_empty, 1);
    mbar_init(&ctl.acc_empty, 4);
    mbar_init(&ctl.drain, 1);
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(&ctl.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // (a no-op in plain stream order) the pre-pass's LSE/D rows and zeroed
  // accumulator are read below; then let the dQ conversion launch early
  grid_dep_wait();
  grid_dep_launch();
  const uint32_t tmem = ctl.tmem_base;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sDO = smem + C::kOffDO;
  uint8_t* sDs = smem + C::kOffDs;
  float* sVec = reinterpret_cast<float*>(smem + C::kOffVec);

  if (wg <= 1) {
    // ------------------------------------------------------------ compute
    // Two warps per lane quarter: warp w (0-7) takes key rows of lane
    // quarter w % 4 and query columns [64 h, 64 h + 64) with h = w / 4. P and
    // dS are elementwise given the row's LSE and D, so the halves need no
    // exchange; two warps per SMSP hide each other's latencies.
    // Registers (launch: 512 threads x 128): compute 8 warps x 136, dQ drain
    // 4 x 144, producer / MMA / idle 4 x 96 = 2048 x 32 = the 65536 of the SM.
    setmaxnreg_inc<136>();
    const int row = ((warp & 3) << 5) + lane;  // key row within the tile
    const int c0 = (warp >> 2) * 64;          // first query column of this warp
    const uint32_t t_lane = tmem + (uint32_t(warp & 3) << 21);
    const int off = p.Nk - p.Nq;
    const float sl = p.scale_log2;
    uint32_t ph_s = 0, ph_dp = 0;
    bool ok = true;
    int g = 0;  // step counter across items
    for (int k = 0; ok; ++k) {
      {
        // the item goes to this warp's shared slot: the compute and drain
        // warps have no registers to spare for it
        Item t;
        int tb, tk;
        const int have = item_at<CAUSAL, WIN, PIECES>(p, k, t, tb, tk);
        if (have == 0) break;
        if (have == 1) continue;
        __syncwarp();
        if (lane == 0) ctl.cur[warp] = Cur{t, tb, tk};
        __syncwarp();
      }
      const Item& I = ctl.cur[warp].I;
      const int key = I.j * 128 + row;
      const bool kvalid = key < p.Nk;  // keys past Nk are zero-filled: give them P = 0
      for (int st = 0; st < I.steps && ok; ++st, ++g) {
        const int it = I.i0 + st % I.nq;  // query tile
        const int vs = g & 1;
        const float* lse2 = sVec + vs * 256 + c0;
        const float* dlt = sVec + vs * 256 + 128 + c0;
        if (!mbar_wait_bounded(&ctl.vec_full[vs], (g >> 1) & 1, abort_flag, LIM)) { ok = false; break; }
        if (threadIdx.x == 0) trace_stamp(p.trace, g, 5);
        if (!mbar_wait_bounded(&ctl.s_full, ph_s, abort_flag, LIM)) { ok = false; break; }
        ph_s ^= 1;
        if (threadIdx.x == 0) trace_stamp(p.trace, g, 6);
        tc_fence_after();
        float pv[64];
        {
          uint32_t x[64];
          tmem_ld32(t_lane + C::kColS + c0, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
          tmem_ld32(t_lane + C::kColS + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(lse2 + c);
            const uint64_t y0 = ffma2(pack2(u2f(x[c]), u2f(x[c + 1])), pack2(sl, sl), pack2(-l4.x, -l4.y));
            const uint64_t y1 = ffma2(pack2(u2f(x[c + 2]), u2f(x[c + 3])), pack2(sl, sl), pack2(-l4.z, -l4.w));
            float a0, a1, a2, a3;
            unpack2(y0, a0, a1);
            unpack2(y1, a2, a3);
            pv[c] = ex2_mufu(a0);
            pv[c + 1] = ex2_mufu(a1);
            pv[c + 2] = ex2_mufu(a2);
            pv[c + 3] = ex2_mufu(a3);
          }
        }
        // query row q (column c = q - it*128) sees this key iff
        // key - off - wr <= q <= key - off + wl: mask tiles that cross an edge
        const int wl = win_l<WIN>(p), wr = win_r<WIN>(p);
        const bool need_mask = CAUSAL && ((wr >= 0 && it * 128 < I.j * 128 + 127 - off - wr) ||
                                          (wl >= 0 && it * 128 + 127 > I.j * 128 - off + wl));
        // masking only on diagonal tiles and past-the-end keys, in its own
        // pass so the common case carries no per-element selects; column
        // bounds relative to this warp's first column
        if (need_mask || !kvalid) {
          const int qlim = wr >= 0 ? key - off - wr - it * 128 - c0 : -(1 << 30);  // columns c < qlim are hidden
          const int lim = kvalid ? qlim : 64;
          if (WIN) {
            const int qmax = wl >= 0 ? key - off + wl - it * 128 - c0 : (1 << 30);  // and columns c > qmax
            const int top = kvalid ? qmax : -1;
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c < lim || c > top) pv[c] = 0.0f;
          } else {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c < lim) pv[c] = 0.0f;
          }
        }
        {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(pv[2 * c], pv[2 * c + 1]);
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tmem_st16(t_lane + C::kColS + c0 / 2 + c * 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[c * 16]));
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (threadIdx.x == 0) trace_stamp(p.trace, g, 7);
        if (lane == 0) mbar_arrive(&ctl.p_full);

        // dS^T = P^T o (dP^T - D), 32 columns per TMEM load
        if (!mbar_wait_bounded(&ctl.dp_full, ph_dp, abort_flag, LIM)) { ok = false; break; }
        ph_dp ^= 1;
        if (threadIdx.x == 0) trace_stamp(p.trace, g, 8);
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 64; h += 32) {
          uint32_t gg[32];
          tmem_ld32(t_lane + C::kColDP + c0 + h, gg);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 4; ++u) {  // 8 columns = one 16-byte unit
            const int c = h + u * 8;
            const float4 d0 = *reinterpret_cast<const float4*>(dlt + c);
            const float4 d1 = *reinterpret_cast<const float4*>(dlt + c + 4);
            const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              float s0, s1;
              unpack2(fmul2(pack2(pv[c + e], pv[c + e + 1]),
                            fadd2(pack2(u2f(gg[u * 8 + e]), u2f(gg[u * 8 + e + 1])), pack2(-dd[e], -dd[e + 1]))),
                      s0, s1);
              pk[e >> 1] = pack_bf16x2(s0, s1);
            }
            *reinterpret_cast<uint4*>(sDs + sw128_off(row, c0 + c)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (threadIdx.x == 0) trace_stamp(p.trace, g, 9);
        if (lane == 0) {
          mbar_arrive(&ctl.ds_full);
          mbar_arrive(&ctl.vec_empty[vs]);
        }
      }
    }
  } else if (wg == 2) {
    // ------------------------------------------------ dQ drain + epilogue
    setmaxnreg_inc<144>();
    const int wq = warp & 3;
    const uint32_t t_lane = tmem + (uint32_t(wq) << 21);
    const int lr = (wq << 5) + lane;  // TMEM lane: d index (D=128) or query row (D=64)
    uint32_t ph_dq = 0, nacc = 0;
    bool ok = true;
    int g = 0;
    for (int k = 0; ok; ++k) {
      {
        // the item goes to this warp's shared slot: the compute and drain
        // warps have no registers to spare for it
        Item t;
        int tb, tk;
        const int have = item_at<CAUSAL, WIN, PIECES>(p, k, t, tb, tk);
        if (have == 0) break;
        if (have == 1) continue;
        __syncwarp();
        if (lane == 0) ctl.cur[warp] = Cur{t, tb, tk};
        __syncwarp();
      }
      const Item& I = ctl.cur[warp].I;
      const int& ib = ctl.cur[warp].b;
      const int& ikvh = ctl.cur[warp].kvh;
      for (int st = 0; st < I.steps && ok; ++st, ++g) {
        const int it = I.i0 + st % I.nq;
        const int h = ikvh * p.group + (PIECES ? I.h0 : 0) + st / I.nq;
        if (!mbar_wait_bounded(&ctl.dq_full, ph_dq, abort_flag, LIM)) { ok = false; break; }
        ph_dq ^= 1;
        if (threadIdx.x == 256) trace_stamp(p.trace, g, 10);
        tc_fence_after();
        if (D == 128) {
          uint32_t v[128];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tmem_ld32(t_lane + C::kColDP + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[c * 32]));
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.dq_empty);
          if (threadIdx.x == 256) trace_stamp(p.trace, g, 11);
          // dQ: lane = query row of the tile, column = d. Stage it as
          // 128-byte-swizzled boxes of [32 q rows][32 d] fp32, two boxes per
          // warp and half of d, and add each box into the accumulator with a
          // TMA reduction; the buffer is rewritten once the previous
          // reductions have read it.
          uint8_t* stg = smem + C::kOffStg + wq * 8192;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int b2 = 0; b2 < 2; ++b2) {
              const int db = half * 2 + b2;  // d block of 32
              uint8_t* box = stg + b2 * 4096 + lane * 128;
#pragma unroll
              for (int u = 0; u < 8; ++u)
                *reinterpret_cast<uint4*>(box + ((u ^ (lane & 7)) << 4)) =
                    make_uint4(v[db * 32 + 4 * u], v[db * 32 + 4 * u + 1], v[db * 32 + 4 * u + 2],
                               v[db * 32 + 4 * u + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
              for (int b2 = 0; b2 < 2; ++b2)
                tma_reduce_add_4d(&out.acc, stg + b2 * 4096, (half * 2 + b2) * 32, it * 128 + wq * 32, h, ib);
              bulk_commit();
            }
          }
          if (threadIdx.x == 256) trace_stamp(p.trace, g, 12);
        } else {
          uint32_t v[64];
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tmem_ld32(t_lane + C::kColDP + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[c * 32]));
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.dq_empty);
          // dQ: lane = query row, 64 columns = d; for a fixed d the warp's
          // lanes hit consecutive query rows of the accumulator
          const int q = it * 128 + lr;
          float* dst = p.dq_acc + (size_t(ib) * p.Hq + h) * D * size_t(p.Nq_pad) + q;
#pragma unroll
          for (int c = 0; c < 64; ++c) red_add_f32(dst + size_t(c) * p.Nq_pad, u2f(v[c]));
        }
      }
      if (!ok) break;
      // epilogue of this item: dV, dK rows of its key tile (lane = key row)
      if (I.steps == 0) {
        if (PIECES && I.tt >= 0) continue;  // a tail piece: the last pass writes the tile's zeros
        const int key = I.j * 128 + lr;
        __nv_bfloat16* dv = p.dv + ((size_t(ib) * p.Nk + key) * p.Hkv + ikvh) * D;
        __nv_bfloat16* dk = p.dk + ((size_t(ib) * p.Nk + key) * p.Hkv + ikvh) * D;
        if (key < p.Nk) {
          for (int c = 0; c < D / 8; ++c) {
            reinterpret_cast<uint4*>(dv)[c] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4*>(dk)[c] = make_uint4(0, 0, 0, 0);
          }
        }
        continue;
      }
      if (!mbar_wait_bounded(&ctl.acc_full, nacc & 1, abort_flag, LIM)) { ok = false; break; }
      ++nacc;
      tc_fence_after();
      if (D == 128 && PIECES && I.tt >= 0) {
        // A tail piece (one query head of the group): its dV, then dK, are
        // partial sums, stored in fp32 into the piece's own slot of the tail
        // buffer with TMA stores, staged like dQ as [32 rows][32 d] boxes,
        // two per half of d; a last pass sums the slots of each tile.
        uint8_t* stg = smem + C::kOffStg + wq * 8192;
        const int slot = ((ib * p.Hkv + ikvh) * p.n_tail + I.tt) * p.group + I.h0;
#pragma unroll 1
        for (int t = 0; t < 2; ++t) {
          const uint32_t col = t == 0 ? C::kColDV : C::kColDK;
          const float mul = t == 0 ? 1.0f : p.scale;
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            uint32_t v[64];
            tmem_ld32(t_lane + col + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(t_lane + col + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_wait_ld();
            if (t == 1 && half == 1) {  // the next item's MMAs may overwrite the accumulators
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&ctl.acc_empty);
            }
            if (lane == 0) bulk_wait_read_all();  // earlier reductions and stores have read the quarter
            __syncwarp();
#pragma unroll
            for (int b2 = 0; b2 < 2; ++b2) {
              uint8_t* box = stg + b2 * 4096 + lane * 128;
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int c = b2 * 32 + 4 * u;
                *reinterpret_cast<uint4*>(box + ((u ^ (lane & 7)) << 4)) =
                    make_uint4(f2u(u2f(v[c]) * mul), f2u(u2f(v[c + 1]) * mul), f2u(u2f(v[c + 2]) * mul),
                               f2u(u2f(v[c + 3]) * mul));
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
              for (int b2 = 0; b2 < 2; ++b2)
                tma_store_4d(&out.dkv, stg + b2 * 4096, (half * 2 + b2) * 32, wq * 32, t, slot);
              bulk_commit();
            }
          }
        }
      } else if (D == 128) {
        // Each warp stages its 32 key rows of dV, then of dK, as two
        // 128-byte-swizzled [32 rows][64 d] bf16 boxes in its quarter of the
        // dQ staging buffer and writes them with TMA stores (rows past Nk
        // are clipped): whole-line writes, and the warp is free at once.
        // The accumulators are released as soon as dK is in registers.
        uint8_t* stg = smem + C::kOffStg + wq * 8192;
        const int row0 = I.j * 128 + wq * 32;
#pragma unroll 1
        for (int t = 0; t < 2; ++t) {
          const uint32_t col = t == 0 ? C::kColDV : C::kColDK;
          const float mul = t == 0 ? 1.0f : p.scale;
#pragma unroll 1
          for (int b2 = 0; b2 < 2; ++b2) {  // 64 columns (one box) at a time
            uint32_t v[64];
            tmem_ld32(t_lane + col + b2 * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(t_lane + col + b2 * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_wait_ld();
            if (t == 1 && b2 == 1) {  // the next item's MMAs may overwrite the accumulators
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&ctl.acc_empty);
            }
            if (b2 == 0) {
              if (lane == 0) bulk_wait_read_all();  // earlier reductions and stores have read the quarter
              __syncwarp();
            }
            uint8_t* box = stg + b2 * 4096 + lane * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int c = u * 8;
              *reinterpret_cast<uint4*>(box + ((u ^ (lane & 7)) << 4)) =
                  make_uint4(pack_bf16x2(u2f(v[c]) * mul, u2f(v[c + 1]) * mul),
                             pack_bf16x2(u2f(v[c + 2]) * mul, u2f(v[c + 3]) * mul),
                             pack_bf16x2(u2f(v[c + 4]) * mul, u2f(v[c + 5]) * mul),
                             pack_bf16x2(u2f(v[c + 6]) * mul, u2f(v[c + 7]) * mul));
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < p.Nk) {
            const CUtensorMap* m = t == 0 ? &out.dv : &out.dk;
            tma_store_4d(m, stg, 0, ikvh, row0, ib);
            tma_store_4d(m, stg + 4096, 64, ikvh, row0, ib);
            bulk_commit();
          }
        }
      } else {
        const int key = I.j * 128 + lr;
        const bool valid = key < p.Nk;
#pragma unroll 1
        for (int t = 0; t < 2; ++t) {
          const uint32_t col = t == 0 ? C::kColDV : C::kColDK;
          const float mul = t == 0 ? 1.0f : p.scale;
          __nv_bfloat16* dst = (t == 0 ? p.dv : p.dk) + ((size_t(ib) * p.Nk + key) * p.Hkv + ikvh) * D;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(t_lane + col + c * 32, v);
            tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(u2f(v[2 * i]) * mul, u2f(v[2 * i + 1]) * mul);
            if (valid) {
              uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
        }
        // the accumulators may now be overwritten by the next item
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.acc_empty);
      }
    }
    if (D == 128 && lane == 0) bulk_wait_all();  // the accumulator and dK/dV are written when the kernel ends
  } else {
    setmaxnreg_dec<96>();
  }
  if (warp == 12) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      bool ok = true;
      int g = 0, nkv = 0;
      for (int k = 0; ok; ++k) {
        {
          Item t;
          int tb, tk;
          const int have = item_at<CAUSAL, WIN, PIECES>(p, k, t, tb, tk);
          if (have == 0) break;
          if (have == 1) continue;
          ctl.cur[warp] = Cur{t, tb, tk};  // one thread runs this role
        }
        const Item& I = ctl.cur[warp].I;
        const int& ib = ctl.cur[warp].b;
        const int& ikvh = ctl.cur[warp].kvh;
        if (I.steps == 0) continue;
        if (nkv > 0 && !mbar_wait_bounded(&ctl.kv_empty, (nkv - 1) & 1, abort_flag, LIM)) { ok = false; break; }
        ++nkv;
        mbar_arrive_expect_tx(&ctl.kv_full, 2 * C::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(sK + c * 16384, &tmK, &ctl.kv_full, c * 64, ikvh, I.j * 128, ib);
          tma_load_4d(sV + c * 16384, &tmV, &ctl.kv_full, c * 64, ikvh, I.j * 128, ib);
        }
        for (int st = 0; st < I.steps && ok; ++st, ++g) {
          const int it = I.i0 + st % I.nq;
          const int h = ikvh * p.group + (PIECES ? I.h0 : 0) + st / I.nq;
          const int qs = g & 1;
          if (st == max(0, I.steps - kPrefetchSteps)) {
            // the next item's K and V into L2, so that its loads (issued
            // once this item's last GEMM has read K and V) hit L2
            Item N;
            int nb, nkvh;
            int nh = item_at<CAUSAL, WIN, PIECES>(p, k + 1, N, nb, nkvh);
            if (nh == 1) nh = item_at<CAUSAL, WIN, PIECES>(p, k + 2, N, nb, nkvh);
            if (nh == 2 && N.steps > 0) {
#pragma unroll
              for (int c = 0; c < D / 64; ++c) {
                tma_prefetch_l2_4d(&tmK, c * 64, nkvh, N.j * 128, nb);
                tma_prefetch_l2_4d(&tmV, c * 64, nkvh, N.j * 128, nb);
              }
            }
          }
          if (!mbar_wait_bounded(&ctl.q_empty[qs], ((g >> 1) & 1) ^ 1, abort_flag, LIM)) { ok = false; break; }
          trace_stamp(p.trace, g, 13);
          mbar_arrive_expect_tx(&ctl.q_full[qs], C::kTile);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(sQ + qs * C::kTile + c * 16384, &tmQ, &ctl.q_full[qs], c * 64, h, it * 128, ib);
          // LSE/D rows before dO: the compute warps need them as soon as
          // S is ready, while dO (one slot) waits for the previous dV
          const int vs = g & 1;
          if (!mbar_wait_bounded(&ctl.vec_empty[vs], ((g >> 1) & 1) ^ 1, abort_flag, LIM)) { ok = false; break; }
          mbar_arrive_expect_tx(&ctl.vec_full[vs], 1024);
          const size_t roff = (size_t(ib) * p.Hq + h) * p.Nq_pad + size_t(it) * 128;
          bulk_load(sVec + vs * 256, p.lse2 + roff, 512, &ctl.vec_full[vs]);
          bulk_load(sVec + vs * 256 + 128, p.delta + roff, 512, &ctl.vec_full[vs]);
          if (!mbar_wait_bounded(&ctl.do_empty, (g & 1) ^ 1, abort_flag, LIM)) { ok = false; break; }
          trace_stamp(p.trace, g, 14);
          mbar_arrive_expect_tx(&ctl.do_full, C::kTile);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(sDO + c * 16384, &tmDO, &ctl.do_full, c * 64, h, it * 128, ib);
        }
      }
      if (*abort_flag) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
      }
    }
  } else if (warp == 13) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSS = idesc_bf16_f32(128, 128, 0, 0);     // S^T, dP^T
      constexpr uint32_t idAcc = idesc_bf16_f32(128, D, 0, 1);      // dV, dK
      constexpr uint32_t idDQ = D == 128 ? idesc_bf16_f32(128, 128, 1, 1) : idesc_bf16_f32(128, 64, 1, 1);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ), aDO = smem_u32(sDO),
                     aDs = smem_u32(sDs);
      bool ok = true;
      uint32_t ph_p = 0, ph_ds = 0, ph_dqe = 0;
      int g = 0, nkv = 0;
      // Tile descriptors are built once; a K step is one add of a constant,
      // so MMAs issue back to back (the tensor core idles otherwise).
      const uint32_t kK = sdesc_lo(aK, 16), kV = sdesc_lo(aV, 16), kQ = sdesc_lo(aQ, 16);  // K-major
      const uint32_t kDO = sdesc_lo(aDO, 16), kDs = sdesc_lo(aDs, 16);
      const uint32_t mQ = sdesc_lo(aQ, 16384), mDO = sdesc_lo(aDO, 16384);  // MN-major
      const uint32_t mK = sdesc_lo(aK, 16384), mDs = sdesc_lo(aDs, 16384);
      auto issue_kmajor = [&](uint32_t d_col, uint32_t a0, uint32_t b0) {  // [128 x 128] += A B^T, K = D
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss_lo(tmem + d_col, sdesc_step(a0, ko), sdesc_step(b0, ko), idSS, kk > 0);
        }
      };
      for (int k = 0; ok; ++k) {
        {
          Item t;
          int tb, tk;
          const int have = item_at<CAUSAL, WIN, PIECES>(p, k, t, tb, tk);
          if (have == 0) break;
          if (have == 1) continue;
          ctl.cur[warp] = Cur{t, tb, tk};  // one thread runs this role
        }
        const Item& I = ctl.cur[warp].I;
        if (I.steps == 0) continue;
        ok = mbar_wait_bounded(&ctl.kv_full, nkv & 1, abort_flag, LIM);
        if (ok) ok = mbar_wait_bounded(&ctl.q_full[g & 1], (g >> 1) & 1, abort_flag, LIM);
        if (!ok) break;
        ++nkv;
        tc_fence_after();
        issue_kmajor(C::kColS, kK, sdesc_step(kQ, (g & 1) * C::kTile));  // S^T = K Q^T for the item's first step
        mma_commit(&ctl.s_full);
        for (int st = 0; st < I.steps && ok; ++st, ++g) {
          const uint32_t mQcur = sdesc_step(mQ, (g & 1) * C::kTile);
          if (!mbar_wait_bounded(&ctl.do_full, g & 1, abort_flag, LIM)) { ok = false; break; }
          if (g > 0) {
            if (!mbar_wait_bounded(&ctl.dq_empty, ph_dqe, abort_flag, LIM)) { ok = false; break; }
            ph_dqe ^= 1;
          }
          tc_fence_after();
          trace_stamp(p.trace, g, 0);
          issue_kmajor(C::kColDP, kV, kDO);  // dP^T = V dO^T
          mma_commit(&ctl.dp_full);
          if (!mbar_wait_bounded(&ctl.p_full, ph_p, abort_flag, LIM)) { ok = false; break; }
          ph_p ^= 1;
          // before the first dV of a later item overwrites the accumulators,
          // the previous item's dK/dV must have been read out of TMEM
          if (st == 0 && nkv > 1 && !mbar_wait_bounded(&ctl.acc_empty, (nkv - 2) & 1, abort_flag, LIM)) {
            ok = false;
            break;
          }
          trace_stamp(p.trace, g, 1);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dV += P^T dO   (P^T in TMEM, dO MN-major)
            mma_ts_lo(tmem + C::kColDV, tmem + C::kColS + kk * 8, sdesc_step(mDO, kk * 2048), idAcc,
                   (st > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&ctl.do_empty);
          if (st + 1 < I.steps) {
            const int nx = (g + 1) & 1;
            if (!mbar_wait_bounded(&ctl.q_full[nx], ((g + 1) >> 1) & 1, abort_flag, LIM)) { ok = false; break; }
            trace_stamp(p.trace, g, 2);
            tc_fence_after();
            issue_kmajor(C::kColS, kK, sdesc_step(kQ, nx * C::kTile));  // S^T for the next step
            mma_commit(&ctl.s_full);
          }
          if (!mbar_wait_bounded(&ctl.ds_full, ph_ds, abort_flag, LIM)) { ok = false; break; }
          ph_ds ^= 1;
          trace_stamp(p.trace, g, 3);
          tc_fence_after();
          // dK first, then dQ (issuing dQ first, so that its drain overlaps
          // dK, measured 0.5-1 % slower)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // dK += dS^T Q   (dS^T K-major, Q MN-major)
            const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss_lo(tmem + C::kColDK, sdesc_step(kDs, ko), sdesc_step(mQcur, kk * 2048), idAcc,
                      (st > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&ctl.q_empty[g & 1]);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // dQ = dS K  (both MN-major): lane = query row, column = d
            mma_ss_lo(tmem + C::kColDP, sdesc_step(mDs, kk * 2048), sdesc_step(mK, kk * 2048), idDQ, kk > 0);
          }
          mma_commit(&ctl.dq_full);
          trace_stamp(p.trace, g, 4);
        }
        if (!ok) break;
        mma_commit(&ctl.acc_full);  // dK, dV of this item are complete
        mma_commit(&ctl.kv_empty);  // K, V of this item no longer read
      }
      if (*abort_flag) {
        mma_commit(&ctl.drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&ctl.drain), 0) && globaltimer_ns() - t0 < 100000000ull) {
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 13) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0 && ctl.abort) atomicOr(p.status, kDevTimeout);
}

// D_i = sum_c dO_ic O_ic and LSE * log2(e) per row, written to padded
// [B*Hq, Nq_pad] arrays; padded rows and rows with LSE = -inf get +inf (so
// their probabilities recompute to 0) and D = 0. Also zeroes the fp32 dQ
// accumulator.
// Work is split into groups of 16 consecutive query rows of one (batch,
// head), one group per warp at a time: the warp loads the group's O and dO
// rows (16 bytes per lane per row piece, all loads issued before any is
// used), zeroes an equal share of the dQ accumulator meanwhile, then
// writes the group's 16 LSE/D values as one contiguous run.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* o, const __nv_bfloat16* dout,
                                                      const float* lse, float* lse2, float* delta, float* dq_acc,
                                                      int B, int Hq, int Nq, int Nq_pad, long long zero4) {
  grid_dep_launch();  // the main kernel may start its set-up meanwhile
  constexpr int TPR = D / 8;          // lanes per row, 8 elements (16 bytes) each
  constexpr int RPP = 32 / TPR;       // rows per pass of the warp
  constexpr int kRows = 16;           // rows per group
  constexpr int kPass = kRows / RPP;  // passes per group
  const int lane = threadIdx.x & 31;
  const int part = lane % TPR, sub = lane / TPR;
  const long long warp_id = (1LL * blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = (1LL * gridDim.x * blockDim.x) >> 5;
  const int gq = (Nq + kRows - 1) / kRows;  // groups per (batch, head)
  const long long n_groups = 1LL * B * Hq * gq;
  const long long n4 = zero4;  // the dQ accumulator, in float4
  const long long zc = (n4 + n_groups - 1) / n_groups;  // float4 zeroed per group
  float4* acc4 = reinterpret_cast<float4*>(dq_acc);
  for (long long grp = warp_id; grp < n_groups; grp += n_warps) {
    const long long bh = grp / gq;
    const int q0 = int(grp - bh * gq) * kRows;
    const int b = int(bh / Hq), h = int(bh - 1LL * b * Hq);
    uint4 a[kPass], g[kPass];
#pragma unroll
    for (int i = 0; i < kPass; ++i) {
      const int q = q0 + i * RPP + sub;
      a[i] = g[i] = make_uint4(0, 0, 0, 0);
      if (q < Nq) {
        const size_t off = ((size_t(b) * Nq + q) * Hq + h) * D + part * 8;
        a[i] = *reinterpret_cast<const uint4*>(o + off);
        g[i] = *reinterpret_cast<const uint4*>(dout + off);
      }
    }
    const long long z1 = (grp + 1) * zc < n4 ? (grp + 1) * zc : n4;
    for (long long z = grp * zc + lane; z < z1; z += 32) acc4[z] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float mine = 0.0f;  // lane t < 16: D of the group's row t
#pragma unroll
    for (int i = 0; i < kPass; ++i) {
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[i]);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g[i]);
      float acc = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(a2[e]), fg = __bfloat1622float2(g2[e]);
        acc = fmaf(fa.x, fg.x, acc);
        acc = fmaf(fa.y, fg.y, acc);
      }
#pragma unroll
      for (int m = TPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
      // row i * RPP + r sits in lanes [r * TPR, r * TPR + TPR)
      const float v = __shfl_sync(0xffffffffu, acc, (lane % RPP) * TPR);
      if (lane / RPP == i) mine = v;
    }
    const int q = q0 + lane;
    if (lane < kRows && q < Nq) {
      const size_t dst = size_t(bh) * Nq_pad + q;
      const float l = lse[size_t(bh) * Nq + q];
      lse2[dst] = l == -INFINITY ? INFINITY : l * 1.4426950408889634f;
      delta[dst] = mine;
    }
  }
  // padded rows
  const long long tid = 1LL * blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = 1LL * gridDim.x * blockDim.x;
  const long long pad = 1LL * B * Hq * (Nq_pad - Nq);
  for (long long i = tid; i < pad; i += nthreads) {
    const long long bh = i / (Nq_pad - Nq);
    const int q = Nq + int(i % (Nq_pad - Nq));
    lse2[bh * Nq_pad + q] = INFINITY;
    delta[bh * Nq_pad + q] = 0.0f;
  }
}

// d = 128: dq[b, q, h, :] = bf16(scale * acc[b*Hq + h, q, :]) (the
// accumulator is row-major there), a streaming pass: 16 lanes per row, each
// reading 32 bytes and writing 16, four row pieces per thread in flight.
__global__ void __launch_bounds__(256) bwd_post_rows_kernel(const float* dq_acc, __nv_bfloat16* dq, int B, int Hq,
                                                            int Nq, int Nq_pad, float scale) {
  grid_dep_wait();  // launched while the main kernel may still run
  constexpr int D = 128, TPR = D / 8, U = 4;
  const long long n = 1LL * B * Hq * Nq * TPR;  // 8-element pieces
  const long long tid = 1LL * blockIdx.x * blockDim.x + threadIdx.x;
  const long long nth = 1LL * gridDim.x * blockDim.x;
  for (long long base = tid; base < n; base += U * nth) {
    float4 x[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long idx = base + u * nth;
      if (idx < n) {
        const long long row = idx / TPR;  // (b*Hq + h)*Nq + q
        const int part = int(idx - row * TPR);
        const long long bh = row / Nq;
        const int q = int(row - bh * Nq);
        const float4* src = reinterpret_cast<const float4*>(dq_acc + (size_t(bh) * Nq_pad + q) * D + part * 8);
        x[u][0] = __ldcs(src);
        x[u][1] = __ldcs(src + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long idx = base + u * nth;
      if (idx < n) {
        const long long row = idx / TPR;
        const int part = int(idx - row * TPR);
        const long long bh = row / Nq;
        const int q = int(row - bh * Nq);
        const int b = int(bh / Hq), h = int(bh - 1LL * b * Hq);
        *reinterpret_cast<uint4*>(dq + ((size_t(b) * Nq + q) * Hq + h) * D + part * 8) =
            make_uint4(pack_bf16x2(x[u][0].x * scale, x[u][0].y * scale),
                       pack_bf16x2(x[u][0].z * scale, x[u][0].w * scale),
                       pack_bf16x2(x[u][1].x * scale, x[u][1].y * scale),
                       pack_bf16x2(x[u][1].z * scale, x[u][1].w * scale));
      }
    }
  }
}

// d = 128 tail pieces: dV and dK rows of the tail tiles (their scale already
// applied), the sum over the group's slots [B*Hkv][n_tail][group][2][128][D]
// taken in slot order, to bf16 BSHD, 16 lanes per row; rows past Nk are
// skipped, and a tile that no query row sees (its pieces stored nothing)
// gets zeros. The tile of tail index tt is the one the main kernel's decode
// gives it; wr is the kernel's right window bound (0 when causal).
__global__ void __launch_bounds__(256) bwd_tail_kernel(const float* dkv, __nv_bfloat16* dk, __nv_bfloat16* dv, int B,
                                                       int Hkv, int group, int Nq, int Nk, int wr, int n_ktiles,
                                                       int n_split, int n_tail) {
  grid_dep_wait();  // launched while the kernels before may still run
  constexpr int D = 128, TPR = D / 8;
  const long long n = 1LL * B * Hkv * n_tail * 2 * 128 * TPR;
  const long long tid = 1LL * blockIdx.x * blockDim.x + threadIdx.x;
  const long long nth = 1LL * gridDim.x * blockDim.x;
  for (long long idx = tid; idx < n; idx += nth) {
    const long long row = idx / TPR;  // ((r * n_tail + tt) * 2 + t) * 128 + rr
    const int part = int(idx - row * TPR);
    const int rr = int(row % 128);
    long long x = row / 128;
    const int t = int(x % 2);  // 0: dV, 1: dK
    x /= 2;
    const int tt = int(x % n_tail);
    const long long r = x / n_tail;
    const int b = int(r / Hkv), kvh = int(r - 1LL * b * Hkv);
    const int half = n_ktiles / 2, kept = half - n_split, pr = kept + (tt >> 1);
    const int j = tt < 2 * n_split ? ((tt & 1) ? n_ktiles - 1 - pr : pr) : half;
    const int key = j * 128 + rr;
    if (key >= Nk) continue;
    // the first query row that sees key tile j is past the last one: no pieces ran
    const bool empty = wr >= 0 && j * 128 - (Nk - Nq) - wr > Nq - 1;
    float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (!empty) {
      for (int g = 0; g < group; ++g) {
        const float4* src =
            reinterpret_cast<const float4*>(dkv + ((((r * n_tail + tt) * group + g) * 2 + t) * 128 + rr) * D + part * 8);
        const float4 a = src[0], c = src[1];
        f[0] += a.x; f[1] += a.y; f[2] += a.z; f[3] += a.w;
        f[4] += c.x; f[5] += c.y; f[6] += c.z; f[7] += c.w;
      }
    }
    __nv_bfloat16* dst = (t == 0 ? dv : dk) + ((size_t(b) * Nk + key) * Hkv + kvh) * D + part * 8;
    *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                                pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
  }
}

// d = 64: dq[b, q, h, :] = bf16(scale * acc[b*Hq + h, :, q]), through a shared
// tile: a block takes 64 queries of one (batch, head); each warp reads whole
// 256-byte runs of accumulator rows (one d, 64 q), then every thread writes
// 16-byte pieces of dq rows (16 consecutive threads write one 256-byte row
// for d = 128).
template <int D>
__global__ void __launch_bounds__(256) bwd_post_kernel(const float* dq_acc, __nv_bfloat16* dq, int BH, int Hq, int Nq,
                                                       int Nq_pad, float scale) {
  grid_dep_wait();  // launched while the main kernel may still run
  __shared__ float tile[D][65];
  const int nqt = Nq_pad / 64;
  const int bh = blockIdx.x / nqt, qt = blockIdx.x - bh * nqt;
  if (bh >= BH) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* src = dq_acc + size_t(bh) * D * Nq_pad + qt * 64 + 2 * lane;
  float2 x[D / 8];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) x[i] = *reinterpret_cast<const float2*>(src + size_t(warp + 8 * i) * Nq_pad);
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    tile[warp + 8 * i][2 * lane] = x[i].x;
    tile[warp + 8 * i][2 * lane + 1] = x[i].y;
  }
  __syncthreads();
  const int b = bh / Hq, h = bh - b * Hq;
  constexpr int kD8 = D / 8;
  for (int it = threadIdx.x; it < 64 * kD8; it += 256) {
    const int ql = it / kD8, d8 = (it - ql * kD8) * 8;
    const int q = qt * 64 + ql;
    if (q >= Nq) continue;
    float f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = tile[d8 + e][ql] * scale;
    *reinterpret_cast<uint4*>(dq + ((size_t(b) * Nq + q) * Hq + h) * D + d8) =
        make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
  }
}

// How many key-tile pairs per kv head (those nearest the middle) to run as
// single-tile units, for `heads` (batch, kv head) slices of n key tiles on G
// persistent CTAs, each single split further into `hs` units (one per query
// head of the group, or hs = 1). Model, in units of one such piece (half a
// pair's work for one head): a whole pair takes 2 * hs, a piece 1. Units go
// to CTAs round robin in order (P pairs, then S pieces): with W = P / G and
// T = P mod G, CTA c runs W pairs (one more if c < T) and then the pieces u
// with (P + u) mod G = c. The finish time is the largest CTA's total; the
// smallest split count reaching the least finish time wins.
int split_pairs(int heads, int n, int G, int hs) {
  const int half = n / 2;
  const long long cp = 2LL * hs;
  int best_m = 0;
  long long best_t = -1;
  for (int m = 0; m <= half; ++m) {
    const long long P = 1LL * heads * (half - m), S = 1LL * heads * (2 * m + (n & 1)) * hs;
    const long long W = P / G, T = P % G;
    // CTAs c >= T take pieces at positions c - T, those below T at
    // c - T + G; each takes S / G, plus one at positions below S mod G
    const long long q = S / G, r = S % G;
    long long t = cp * W + q + (r > 0 ? 1 : 0);
    if (T > 0) t = std::max(t, cp * (W + 1) + q + (r > G - T ? 1 : 0));
    if (best_t < 0 || t < best_t) {
      best_t = t;
      best_m = m;
    }
  }
  return best_m;
}

// The causal backward's work split: pairs of key tiles, n_split of them per
// kv head run as single tiles, which for d = 128 with GQA are split once more
// per query head (their dK/dV summed in the fp32 tail accumulator).
struct TailPlan {
  bool paired;
  int n_split, head_split, n_tail;
  size_t dkv_floats;  // size of the tail accumulator
};
TailPlan tail_plan(const Problem& pb) {
  TailPlan t{};
  const int n_ktiles = (pb.Nk + 127) / 128;
  const int wl = normalize_window(pb.window_left, pb.Nq, pb.Nk);
  t.paired = pb.masked() && wl < 0;  // pairs of key tiles only without a left bound
  if (!t.paired) return t;
  const int group = pb.Hq / pb.Hkv;
  t.head_split = (pb.d == 128 && group > 1) ? 1 : 0;
  const int forced = debug_cfg().bwd_split;
  t.n_split = forced >= 0 ? std::min(forced, n_ktiles / 2)
                          : split_pairs(pb.B * pb.Hkv, n_ktiles, num_sms(), t.head_split ? group : 1);
  t.n_tail = 2 * t.n_split + (n_ktiles & 1);
  if (t.head_split && t.n_tail > 0)
    t.dkv_floats = size_t(pb.B) * pb.Hkv * t.n_tail * size_t(group) * 2 * 128 * size_t(pb.d);
  if (t.dkv_floats == 0) t.head_split = 0;
  const size_t base = sizeof(float) * size_t(pb.B) * pb.Hq * ((size_t(pb.Nq) + 127) / 128 * 128) * size_t(pb.d + 2);
  if (t.head_split && pb.ws_cap > 0 && base + sizeof(float) * t.dkv_floats > pb.ws_cap) {
    // the slots do not fit the caller's workspace: whole single tiles, as
    // many as the model wants for them
    if (forced < 0) t.n_split = split_pairs(pb.B * pb.Hkv, n_ktiles, num_sms(), 1);
    t.n_tail = 2 * t.n_split + (n_ktiles & 1);
    t.head_split = 0;
    t.dkv_floats = 0;
  }
  return t;
}

template <int D, bool CAUSAL, bool WIN>
cudaError_t launch_t(const Problem& pb, const void* o, const float* lse, const void* dout, void* dq, void* dk, void* dv,
                     float* ws, cudaStream_t stream) {
  const int Nq_pad = (pb.Nq + 127) / 128 * 128;
  const size_t acc_elems = size_t(pb.B) * pb.Hq * D * Nq_pad;
  const TailPlan tp = tail_plan(pb);
  float* dq_acc = ws;
  float* dkv_acc = ws + acc_elems;  // tail pieces' partial dK/dV (d = 128, GQA), may be empty; not zeroed
  float* lse2 = dkv_acc + tp.dkv_floats;
  float* delta = lse2 + size_t(pb.B) * pb.Hq * Nq_pad;
  {
    // 8 warps a block, one group of 16 query rows per warp at a time; at
    // most 8 blocks per SM, so the blocks are resident together
    const long long groups = 1LL * pb.B * pb.Hq * ((pb.Nq + 15) / 16);
    long long blocks = (groups + 7) / 8;
    const long long maxb = 8LL * num_sms();
    if (blocks > maxb) blocks = maxb;
    bwd_pre_kernel<D><<<unsigned(blocks), 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(o),
                                                             static_cast<const __nv_bfloat16*>(dout), lse, lse2, delta,
                                                             dq_acc, pb.B, pb.Hq, pb.Nq, Nq_pad,
                                                             (long long)(acc_elems / 4));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mq, mk, mv, mdo;
  OutMaps out;  // dK/dV: stores of [32 key rows][64 d] boxes
  if (!make_bshd_map(&mq, pb.q, pb.B, pb.Nq, pb.Hq, D, 128) || !make_bshd_map(&mk, pb.k, pb.B, pb.Nk, pb.Hkv, D, 128) ||
      !make_bshd_map(&mv, pb.v, pb.B, pb.Nk, pb.Hkv, D, 128) ||
      !make_bshd_map(&mdo, dout, pb.B, pb.Nq, pb.Hq, D, 128) || !make_bshd_map(&out.dk, dk, pb.B, pb.Nk, pb.Hkv, D, 32) ||
      !make_bshd_map(&out.dv, dv, pb.B, pb.Nk, pb.Hkv, D, 32))
    return cudaErrorInvalidValue;
  {
    // out.dkv: the tail slots [B*Hkv*n_tail*group][2][128][D] fp32, boxes of
    // 32 rows x 32 d (unused without tail pieces: then a map over the first
    // rows of the dQ accumulator)
    const uint64_t n2 = tp.dkv_floats ? 2 : 1;
    const uint64_t nr = tp.dkv_floats ? uint64_t(pb.B) * pb.Hkv * tp.n_tail * (pb.Hq / pb.Hkv) : 1;
    const uint64_t dims[4] = {uint64_t(D), 128, n2, nr};
    const uint64_t strides[3] = {uint64_t(D) * 4, uint64_t(D) * 128 * 4, uint64_t(D) * 128 * 4 * n2};
    const uint32_t box[4] = {32, 32, 1, 1};
    if (!encode_tiled(&out.dkv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, tp.dkv_floats ? dkv_acc : dq_acc, dims, strides,
                      box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  // out.acc (d = 128): the fp32 accumulator [B, Hq, Nq_pad, D], boxes of 32 q x 32 d
  {
    const uint64_t dims[4] = {uint64_t(D), uint64_t(Nq_pad), uint64_t(pb.Hq), uint64_t(pb.B)};
    const uint64_t strides[3] = {uint64_t(D) * 4, uint64_t(D) * Nq_pad * 4, uint64_t(pb.Hq) * D * Nq_pad * 4};
    const uint32_t box[4] = {32, 32, 1, 1};
    if (!encode_tiled(&out.acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dq_acc, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  Params p;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.dq_acc = dq_acc;
  p.lse2 = lse2;
  p.delta = delta;
  p.B = pb.B;
  p.Hq = pb.Hq;
  p.Hkv = pb.Hkv;
  p.Nq = pb.Nq;
  p.Nk = pb.Nk;
  p.Nq_pad = Nq_pad;
  p.group = pb.Hq / pb.Hkv;
  p.n_ktiles = (pb.Nk + 127) / 128;
  p.n_qtiles = Nq_pad / 128;
  p.scale = pb.scale;
  p.scale_log2 = pb.scale * 1.4426950408889634f;
  p.wl = normalize_window(pb.window_left, pb.Nq, pb.Nk);
  p.wr = pb.causal ? 0 : normalize_window(pb.window_right, pb.Nq, pb.Nk);
  const DebugCfg dc = debug_cfg();
  p.wait_limit_ns = dc.wait_limit_ns;
  p.trace = dc.trace;
  p.status = status_word();
  if (!p.status) return cudaErrorMemoryAllocation;
  using C = Cfg<D>;
  constexpr int smem = C::kOffCtl + int(sizeof(Ctl));
  auto kern = bwd_main_kernel<D, CAUSAL, WIN, false>;
  if constexpr (D == 128 && CAUSAL) {
    if (tp.head_split) kern = bwd_main_kernel<D, CAUSAL, WIN, true>;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const bool paired = tp.paired;  // decode: pairs of key tiles only without a left bound
  p.n_split = tp.n_split;
  p.head_split = tp.head_split;
  p.n_tail = tp.n_tail;
  const long long units =
      paired ? 1LL * pb.B * pb.Hkv * (p.n_ktiles / 2 - p.n_split + 1LL * p.n_tail * (p.head_split ? p.group : 1))
             : 1LL * pb.B * pb.Hkv * p.n_ktiles;
  if (units > (1LL << 31) - 1) return cudaErrorInvalidValue;
  p.n_units = int(units);
  const unsigned grid = unsigned(std::min<long long>(units, num_sms()));  // persistent CTAs, one per SM
  if (dc.ev_begin) cudaEventRecord(dc.ev_begin, stream);
  // The main kernel goes out in plain stream order: launched with
  // programmatic stream serialisation (its CTAs taking SMs as pre-pass
  // blocks retire, then waiting on griddepcontrol) it measured 1 % faster
  // on B4 H16 N2048 but 5 % slower on the 1024-key window. The kernels
  // after it (dQ conversion, tail pass) do use it: they start while the main
  // kernel's last CTAs finish and wait for it.
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  lc.attrs = pdl;
  lc.numAttrs = 0;
  e = cudaLaunchKernelEx(&lc, kern, mq, mk, mv, mdo, out, p);
  if (e != cudaSuccess) return e;
  lc.numAttrs = 1;
  e = cudaGetLastError();
  if (dc.ev_end) cudaEventRecord(dc.ev_end, stream);
  if (e != cudaSuccess) return e;
  if (D == 128) {
    const long long pieces = 1LL * pb.B * pb.Hq * pb.Nq * (D / 8);
    long long blocks = (pieces + 4 * 256 - 1) / (4 * 256);
    if (blocks > 8LL * num_sms()) blocks = 8LL * num_sms();
    lc.gridDim = dim3(unsigned(blocks));
    lc.blockDim = dim3(256);
    lc.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&lc, bwd_post_rows_kernel, dq_acc, static_cast<__nv_bfloat16*>(dq), pb.B, pb.Hq, pb.Nq,
                           Nq_pad, pb.scale);
    if (e != cudaSuccess) return e;
  } else {
    const long long blocks = 1LL * pb.B * pb.Hq * (Nq_pad / 64);
    lc.gridDim = dim3(unsigned(blocks));
    lc.blockDim = dim3(256);
    lc.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&lc, bwd_post_kernel<D>, dq_acc, static_cast<__nv_bfloat16*>(dq), pb.B * pb.Hq, pb.Hq,
                           pb.Nq, Nq_pad, pb.scale);
    if (e != cudaSuccess) return e;
  }
  if (D == 128 && tp.dkv_floats > 0) {  // dK/dV of the tail tiles, from their pieces' sums
    const long long pieces = 1LL * pb.B * pb.Hkv * tp.n_tail * 2 * 128 * (D / 8);
    long long blocks = (pieces + 255) / 256;
    if (blocks > 8LL * num_sms()) blocks = 8LL * num_sms();
    lc.gridDim = dim3(unsigned(blocks));
    lc.blockDim = dim3(256);
    lc.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&lc, bwd_tail_kernel, static_cast<const float*>(dkv_acc), static_cast<__nv_bfloat16*>(dk),
                           static_cast<__nv_bfloat16*>(dv), pb.B, pb.Hkv, p.group, pb.Nq, pb.Nk, p.wr, p.n_ktiles,
                           p.n_split, p.n_tail);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace bwd

int bwd_launch_count(const Problem& p) {
  // pre-pass, main kernel, dQ conversion, and the tail pieces' last pass
  return 3 + (p.d == 128 && bwd::tail_plan(p).dkv_floats > 0 ? 1 : 0);
}

size_t bwd_workspace_bytes(const Problem& p) {
  const size_t Nq_pad = size_t(p.Nq + 127) / 128 * 128;
  // dQ accumulator and LSE/D rows, plus the tail pieces' partial dK/dV
  return sizeof(float) * (size_t(p.B) * p.Hq * Nq_pad * size_t(p.d + 2) + bwd::tail_plan(p).dkv_floats);
}

cudaError_t launch_bwd(const Problem& p, const void* o, const float* lse, const void* dout, void* dq, void* dk,
                       void* dv, float* ws, cudaStream_t stream) {
  if (p.d == 128)
    return !p.masked()        ? bwd::launch_t<128, false, false>(p, o, lse, dout, dq, dk, dv, ws, stream)
           : p.plain_causal() ? bwd::launch_t<128, true, false>(p, o, lse, dout, dq, dk, dv, ws, stream)
                              : bwd::launch_t<128, true, true>(p, o, lse, dout, dq, dk, dv, ws, stream);
  return !p.masked()        ? bwd::launch_t<64, false, false>(p, o, lse, dout, dq, dk, dv, ws, stream)
         : p.plain_causal() ? bwd::launch_t<64, true, false>(p, o, lse, dout, dq, dk, dv, ws, stream)
                            : bwd::launch_t<64, true, true>(p, o, lse, dout, dq, dk, dv, ws, stream);
}

}  // namespace fa

// ---------------------------------------------------------------------------
// Allocation-free backward (fa_bwd_noalloc in fa.h).
//
// fa_bwd asks the stream-ordered allocator for its fp32 workspace on every
// call. Some callers must not allocate device memory at that point: serving
// loops that fix their whole memory plan at start-up and treat any later
// allocation as a failure, and code that runs where the CUDA allocator may
// not be entered at all (for instance inside another allocator's hooks).
// For them the workspace lives in a fixed file-scope device array instead.
// Its address is a device address only on the device side; host code must
// look it up per device with cudaGetSymbolAddress, which is done once per
// device on that device's first call.
namespace fa {
namespace {

static __device__ __align__(256) float g_bwd_noalloc_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES / sizeof(float)];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kNoAllocMaxDevices];

// Device address of this device's scratch array (nullptr on failure).
float* noalloc_scratch() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_bwd_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_noalloc_ptr[dev] = static_cast<float*>(ptr);
  }
  return g_noalloc_ptr[dev];
}

}  // namespace
}  // namespace fa

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk,
                              int d, float scale, int causal, void* stream) {
  const int st = fa::check_bwd_args(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, scale, causal);
  if (st != FA_OK) return st;
  fa::Problem p{q, k, v, B, Hq, Hkv, Nq, Nk, d, scale, causal};
  p.ws_cap = FA_BWD_NOALLOC_SCRATCH_BYTES;  // tail pieces only where their slots fit too
  if (fa::bwd_workspace_bytes(p) > FA_BWD_NOALLOC_SCRATCH_BYTES) return FA_ERR_UNSUPPORTED;
  float* ws = fa::noalloc_scratch();
  if (ws == nullptr) return FA_ERR_LAUNCH;
  // The preprocess kernel zeroes the dQ accumulator and rewrites every LSE/D
  // row it reads, and every tail slot that the last pass reads is stored by
  // this call, so nothing left in the array by an earlier call is used.
  return fa::launch_bwd(p, o, lse, dout, dq, dk, dv, ws, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_LAUNCH;
}
