// The forward attention pipeline shared by the bf16 forward (fa_fwd.cu) and
// the e4m3 forward (fa_fwd8.cu): work decomposition, warp roles, the
// mbarrier protocol, the online softmax with its conditional rescale, and
// the epilogue. What differs between the two operand types (tile sizes,
// loads, where P lives, the GEMM instructions, the per-head scales of the
// e4m3 path) comes from a policy class `K`:
//
//   K::kPair (CTA pairs, below), K::D, K::kTileBytes (a Q tile),
//   K::kSlotBytes (a K/V ring slot), K::kSlots, K::kPTileBytes, K::kSmemDyn
//   K::load_q / load_k / load_v (producer; TMA tile loads onto an mbarrier)
//   K::Desc, K::make_desc, K::idesc_s, K::idesc_pv, K::issue_s, K::issue_pv
//   K::PK, K::pack_p, K::store_p, K::publish_p (softmax -> P for the P V GEMM)
//   K::logit_scale, K::out_scale (per-unit scales)
//
// Method (the post "FlashAttention v1", deep_school #630, sections
// "Тайлинг (Tiling)" and "Онлайн-Softmax"): Q, K and V are cut into tiles
// that are staged on chip; each 128-row query tile meets every visible
// 128-key tile in turn; per row the running max and running sum of
// exponentials are updated and the accumulated output is rescaled when the
// max grows, so the score matrix never leaves the chip and the result equals
// the classical softmax.
//
// Blackwell mapping (the FlashAttention-4 article on smntcn.com describes the
// ingredients: fully asynchronous fifth-generation tensor cores, 256 KB of
// tensor memory per SM for intermediates, warps specialised into data
// movers and MMA issuers, and exp computed partly in software because the
// special-function unit scales slower than the tensor cores):
//
//   CTA = 512 threads, persistent (one per SM), one unit of work = one
//   (batch, query head, 256-row query block) handled as two 128-row stages.
//     warps 0-3   softmax, stage 0      (one thread per query row)
//     warps 4-7   softmax, stage 1
//     warps 8-11  correction + epilogue (rescale O when a row max grows;
//                                        O / l -> bf16 staged in shared
//                                        memory and written by TMA, LSE)
//     warp 12     TMA producer          (Q per unit, K/V ring)
//     warp 13     MMA issuer            (tcgen05.mma, one thread)
//     warps 14-15 idle
//   TMEM (512 columns x 128 lanes, fp32):
//     [0,128)   S of stage 0 (bf16: its first 64 columns are overwritten by
//               P as bf16 pairs, the A operand of O += P V)
//     [128,256) S (/ P) of stage 1
//     [256, 256+d)       O of stage 0
//     [256+d, 256+2d)    O of stage 1
//   MMA issue order per key tile j (stages interleaved so one stage's
//   softmax overlaps the other stage's GEMMs):
//     ... PV0(j), S0(j+1), PV1(j), S1(j+1), PV0(j+1), ...
//   Every mbarrier wait is bounded; on timeout the CTA stops cleanly and
//   the per-device status word records it.
//
// CTA pairs (K::kPair): a cluster of two CTAs runs one unit of 512 query
// rows. Stage s covers 256 consecutive rows, 128 in each CTA (each CTA keeps
// its own softmax, correction and epilogue for its rows), and the even CTA
// alone issues tcgen05.mma with cta_group::2: M = 256 over both CTAs' tensor
// memory, each CTA holding half of each K tile (64 keys) and half of each V
// tile (64 of the d columns) at the same shared-memory offset, so one MMA
// instruction does the work of two and each CTA loads half the K/V bytes.
// The barriers the issuing CTA waits on (Q and K/V loaded, P stored, O
// corrected) count the other CTA's arrivals too; its commits arrive on the
// barriers of both CTAs. Each CTA loads its own tiles (no multicast).
//
// exp2 split: the template argument POLY sends one column pair in every
// POLY of the softmax's exponentials to the fitted polynomial on the FMA
// pipes (exp2_poly_pair) and the rest to ex2.approx on the special-function
// unit; POLY = 0 keeps every exponential on the special-function unit.
#pragma once
#include <cuda_bf16.h>

#include <cmath>

#include "fa_internal.h"
#include "sm103_math.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace fwdp {

constexpr int kThreads = 512;
constexpr int kMaxSlots = 8;
constexpr uint32_t kOCol0 = 256;
constexpr int kStgBytes = 16384;  // O staging: 4 warps x [32 rows x 64 cols] bf16

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

struct Params {
  __nv_bfloat16* o;
  float* lse;
  // e4m3 path only: per (batch, head) max |x| of Q M, K M, V (float bits);
  // the e4m3 scale of a tensor is amax / 448 (1 for an all-zero head)
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

// A unit is a block of query rows of one (batch, head): two stages of 128
// rows (256 rows), or with CTA pairs two stages of 256 rows (512 rows, 128 of
// each stage per CTA). Key ranges are those of a whole stage.
template <bool CAUSAL, bool WIN, bool PAIR = false>
__device__ __forceinline__ Unit decode_unit(const Params& p, int item) {
  constexpr int kStage = PAIR ? 256 : 128;  // query rows per stage
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
  x.row0 = mb * 2 * kStage;
  const int off = p.Nk - p.Nq;
  const int nkb = (p.Nk + 127) >> 7;
  int t0[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int r0 = x.row0 + s * kStage;
    x.rows[s] = r0 < p.Nq;
    t0[s] = 0;
    if (!x.rows[s]) {
      x.n[s] = 0;
    } else if (!CAUSAL) {
      x.n[s] = nkb;
    } else {
      // keys seen by any row of the stage: [lo, hi]
      const int rl = min(r0 + kStage - 1, p.Nq - 1);
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

// Static snake order over rounds of G units (longest first when causal):
// worker c (a CTA, or a CTA pair) takes unit c in even rounds and G-1-c in
// odd rounds.
__device__ __forceinline__ int unit_at(int round, int c, int G) {
  return round * G + ((round & 1) ? (G - 1 - c) : c);
}

// The kernel body; each operand type's translation unit wraps it in its own
// __global__ function (fa_fwd_kernel, fa_fwd8_kernel) launched with
// kThreads threads, one CTA per SM, K::kSmemDyn bytes of dynamic shared
// memory. The tensor maps are the kernel's __grid_constant__ parameters.
template <class K, bool CAUSAL, bool WIN, int POLY>
__device__ __forceinline__ void fwd_body(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                         const CUtensorMap& tmO, const Params& p) {
  constexpr int D = K::D;
  constexpr bool PAIR = K::kPair;
  constexpr int kStage = PAIR ? 256 : 128;  // query rows per stage of a unit
  extern __shared__ uint8_t smem_raw[];
  __shared__ Ctl ctl;  // one per CTA
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                 // 2 tiles
  uint8_t* sKV = smem + 2 * K::kTileBytes;            // kSlots K/V slots
  uint8_t* sP = sKV + K::kSlots * K::kSlotBytes;      // 2 P tiles (none when P stays in TMEM)
  uint8_t* sStg = sP + 2 * K::kPTileBytes;            // O staging

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wg = warp >> 2;
  volatile uint32_t* abort_flag = &ctl.abort;
  const uint64_t LIM = p.wait_limit_ns;
  // CTA pairs: this CTA's rank in the pair (0 issues the MMAs), the worker
  // index and the number of workers of the static schedule
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int worker = PAIR ? int(blockIdx.x >> 1) : int(blockIdx.x);
  const int n_workers = PAIR ? int(gridDim.x >> 1) : int(gridDim.x);
  if (threadIdx.x == 0) trace_stamp(p.trace, kEv, 0);

  if (threadIdx.x == 0) {
    ctl.abort = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl.q_full[s], 1);
      mbar_init(&ctl.s_full[s], 1);
      mbar_init(&ctl.p_full[s], PAIR ? 8 : 4);   // softmax warps of both CTAs of a pair
      mbar_init(&ctl.alpha_full[s], 4);
      mbar_init(&ctl.o_ready[s], PAIR ? 8 : 4);  // correction warps of both CTAs of a pair
      mbar_init(&ctl.o_full[s], 1);
      mbar_init(&ctl.stats_full[s], 4);
      mbar_init(&ctl.stats_empty[s], 4);
    }
    mbar_init(&ctl.q_empty, 1);
    mbar_init(&ctl.drain, 1);
    for (int i = 0; i < K::kSlots; ++i) {
      mbar_init(&ctl.kv_full[i], 1);
      mbar_init(&ctl.kv_empty[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == 13) {
    if constexpr (PAIR) {
      tmem_alloc_pair(&ctl.tmem_base, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&ctl.tmem_base, 512);
      tmem_relinquish();
    }
  }
  if (warp == 12 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  tc_fence_before();
  if constexpr (PAIR) {
    cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrival
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  // arrival on a barrier that the MMA-issuing CTA waits on: local, or from
  // the odd CTA of a pair on the even CTA's barrier (release at cluster
  // scope, so that this CTA's tensor-memory writes are ordered before the
  // MMA that reads them)
  auto arrive_issuer = [&](uint64_t* bar) {
    if (PAIR && rank != 0) {
      mbar_arrive_cluster(mapa_shared(smem_u32(bar), 0));
    } else {
      mbar_arrive(bar);
    }
  };
  if (threadIdx.x == 0) trace_stamp(p.trace, kEv, 1);

  if (wg <= 1) {
    // ------------------------------------------------------------ softmax
    setmaxnreg_inc<176>();
    const int s = wg;
    const int row = ((warp & 3) << 5) + lane;
    const uint32_t t_s = tmem + (uint32_t(warp & 3) << 21) + uint32_t(s * 128);  // lane quarter + S columns
    uint8_t* sP_s = sP + s * K::kPTileBytes;
    uint32_t ph_s = 0, ph_se = 0;
    int blk = 0;  // running key-tile counter (trace only)
    bool ok = true;
    for (int rnd = 0; ok; ++rnd) {
      const int u = unit_at(rnd, worker, n_workers);
      if (u >= p.n_items) break;
      const Unit un = decode_unit<CAUSAL, WIN, PAIR>(p, u);
      const int n = un.n[s];
      const int blk0 = blk;
      blk += un.nb;
      if (n == 0) continue;
      const float sl = K::logit_scale(p, un);
      const int r0 = un.row0 + s * kStage + 128 * int(rank), rl = min(r0 + 127, p.Nq - 1);  // this CTA's rows
      const int rg = r0 + row;  // global query row
      const int off = p.Nk - p.Nq;
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
        typename K::PK pk;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          uint64_t y = ffma2(pack2(u2f(x[2 * c]), u2f(x[2 * c + 1])), sl2, nm2);
          float a, b;
          unpack2(y, a, b);
          if (POLY > 0 && (c % (POLY > 0 ? POLY : 1)) == (POLY - 1)) {
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
          K::pack_p(pk, c, a, b);
        }
        K::store_p(pk, t_s, sP_s, row);
        const uint64_t acc = fadd2(fadd2(acc0, acc1), fadd2(acc2, acc3));
        float la, lb;
        unpack2(acc, la, lb);
        l_run = fmaf(l_run, alpha, la + lb);
        m_run = m_new;
        K::publish_p();
        __syncwarp();
        if (row == 0) trace_stamp(p.trace, blk0 + j, 6 + 3 * s);
        if (lane == 0) arrive_issuer(&ctl.p_full[s]);
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
      const int u = unit_at(rnd, worker, n_workers);
      if (u >= p.n_items) break;
      const Unit un = decode_unit<CAUSAL, WIN, PAIR>(p, u);
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
            const uint32_t t_o = t_lane + kOCol0 + uint32_t(s * D);
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
          if (lane == 0) arrive_issuer(&ctl.o_ready[s]);
        }
      }
      if (!ok) break;
      // epilogue: O / l -> bf16, LSE
      if (row == 0) trace_stamp(p.trace, kEv, 2);
#pragma unroll 1
      for (int s = 0; s < 2; ++s) {
        if (!un.rows[s]) continue;
        const int rg = un.row0 + s * kStage + 128 * int(rank) + row;
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
        const float inv = l > 0.0f ? K::out_scale(p, un) / l : 0.0f;
        const uint32_t t_o = t_lane + kOCol0 + uint32_t(s * D);
        // each warp stages its 32 rows x 64 columns (bf16, 128-byte swizzle)
        // and writes them with one TMA store; rows past Nq are clipped
        uint8_t* stg = sStg + wq * 4096;
        const int wrow0 = un.row0 + s * kStage + 128 * int(rank) + wq * 32;
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
        const int u = unit_at(rnd, worker, n_workers);
        if (u >= p.n_items) break;
        const Unit un = decode_unit<CAUSAL, WIN, PAIR>(p, u);
        if (un.nb == 0) continue;
        if (!first) {
          if (!mbar_wait_bounded(&ctl.q_empty, ph_qe, abort_flag, LIM)) { ok = false; break; }
          ph_qe ^= 1;
        }
        first = false;
        for (int s = 0; s < 2; ++s) {
          if (un.n[s] == 0) continue;
          if constexpr (PAIR) {
            // both CTAs' Q tiles complete on the even CTA's barrier
            if (rank == 0) mbar_arrive_expect_tx(&ctl.q_full[s], 2 * K::kTileBytes);
            K::load_q(sQ + s * K::kTileBytes, &tmQ, mapa_shared(smem_u32(&ctl.q_full[s]), 0), un.h,
                      un.row0 + s * kStage + 128 * int(rank), un.b);
          } else {
            mbar_arrive_expect_tx(&ctl.q_full[s], K::kTileBytes);
            K::load_q(sQ + s * K::kTileBytes, &tmQ, &ctl.q_full[s], un.h, un.row0 + s * kStage, un.b);
          }
        }
        for (int j = 0; j < un.nb && ok; ++j) {
#pragma unroll 1
          for (int t = 0; t < 2; ++t) {
            const uint32_t slot = kv_it % K::kSlots;
            const uint32_t ph = ((kv_it / K::kSlots) & 1) ^ 1;
            if (!mbar_wait_bounded(&ctl.kv_empty[slot], ph, abort_flag, LIM)) { ok = false; break; }
            trace_stamp(p.trace, blk + j, 14 + t);
            ++kv_it;
            if (p.inject == 1 && !injected && rank == 0) {  // test hook: never deliver this tile
              injected = true;
              continue;
            }
            uint8_t* dst = sKV + slot * K::kSlotBytes;
            if constexpr (PAIR) {
              if (rank == 0) mbar_arrive_expect_tx(&ctl.kv_full[slot], 2 * K::kSlotBytes);
              const uint32_t bar = mapa_shared(smem_u32(&ctl.kv_full[slot]), 0);
              if (t == 0)
                K::load_k(dst, &tmK, bar, un.kvh, (un.kb0 + j) * 128, un.b, rank);
              else
                K::load_v(dst, &tmV, bar, un.kvh, (un.kb0 + j) * 128, un.b, rank);
            } else {
              mbar_arrive_expect_tx(&ctl.kv_full[slot], K::kSlotBytes);
              if (t == 0)
                K::load_k(dst, &tmK, &ctl.kv_full[slot], un.kvh, (un.kb0 + j) * 128, un.b);
              else
                K::load_v(dst, &tmV, &ctl.kv_full[slot], un.kvh, (un.kb0 + j) * 128, un.b);
            }
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
    // (with CTA pairs only the even CTA issues, for both)
    if (lane == 0 && rank == 0) {
      // completion of the issued MMAs: on this CTA's barrier, or on the same
      // barrier of both CTAs of a pair
      auto commit = [&](uint64_t* bar) {
        if constexpr (PAIR) {
          mma_commit_pair(bar, 3);
        } else {
          mma_commit(bar);
        }
      };
      // a negative scale negates A (Q) in S = Q K^T: bit 13 of the instruction descriptor
      const uint32_t idS = K::idesc_s() | (p.neg_s << 13);
      constexpr uint32_t idPV = K::idesc_pv();
      uint32_t kv_it = 0, ph_q[2] = {0, 0}, ph_p[2] = {0, 0}, ph_o[2] = {0, 0};
      int blk = 0;
      bool ok = true;
      // Tile descriptors are built once; a K step is one add of a constant,
      // so MMAs issue back to back (the tensor core idles otherwise).
      const typename K::Desc dsc = K::make_desc(smem_u32(sQ), smem_u32(sKV), smem_u32(sP));
      auto wait_kv = [&](uint32_t& slot) -> bool {
        slot = kv_it % K::kSlots;
        const bool r = mbar_wait_bounded(&ctl.kv_full[slot], (kv_it / K::kSlots) & 1, abort_flag, LIM);
        ++kv_it;
        return r;
      };
      for (int rnd = 0; ok; ++rnd) {
        const int u = unit_at(rnd, worker, n_workers);
        if (u >= p.n_items) break;
        const Unit un = decode_unit<CAUSAL, WIN, PAIR>(p, u);
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
          K::issue_s(dsc, tmem + uint32_t(s * 128), s, kslot, idS);
          commit(&ctl.s_full[s]);
        }
        commit(&ctl.kv_empty[kslot]);
        if (un.nb == 1) commit(&ctl.q_empty);
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
              K::issue_pv(dsc, tmem + kOCol0 + uint32_t(s * D), tmem + uint32_t(s * 128), s, vslot, j > un.a[s],
                          idPV);
              if (j == un.a[s] + un.n[s] - 1) commit(&ctl.o_full[s]);
              // V_j is free once the last PV reading it completes: release it
              // before the next S is issued so the refill starts earlier
              if (s == last_v) commit(&ctl.kv_empty[vslot]);
            }
            if (nxt && un.active(s, j + 1)) {  // S of the next tile (a stage's first S when it starts there)
              tc_fence_after();
              trace_stamp(p.trace, blk + j, 2 + s);
              K::issue_s(dsc, tmem + uint32_t(s * 128), s, kslot, idS);
              commit(&ctl.s_full[s]);
            }
          }
          if (!ok) break;
          if (nxt) commit(&ctl.kv_empty[kslot]);
          if (j + 2 == un.nb) commit(&ctl.q_empty);
        }
        blk += un.nb;
      }
      if (*abort_flag) {
        // drain the tensor pipe before TMEM is released
        if constexpr (PAIR) {
          mma_commit_pair(&ctl.drain, 1);
        } else {
          mma_commit(&ctl.drain);
        }
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
  if constexpr (PAIR) {
    cluster_sync_all();  // no CTA of a pair leaves while the other may still reach its memory
  } else {
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 13) {
    if constexpr (PAIR) {
      tmem_dealloc_pair(tmem, 512);
    } else {
      tmem_dealloc(tmem, 512);
    }
  }
  if (threadIdx.x == 0 && ctl.abort) atomicOr(p.status, kDevTimeout);
  if (threadIdx.x == 0) trace_stamp(p.trace, kEv, 7);
}

// Work items of one launch: the unit count and the row-split tail
// (non-causal only; see Params). G is the number of workers (CTAs, or CTA
// pairs with 512-row units).
inline void plan_units(Params& p, const Problem& pb, bool causal, int G, int rows_per_unit = 256) {
  p.n_mblocks = (pb.Nq + rows_per_unit - 1) / rows_per_unit;
  p.n_units = p.n_mblocks * pb.B * pb.Hq;
  // Row-split tail: when the T = n_units mod G units of the last round fit
  // on G CTAs twice over, each runs as two single-stage items (its two
  // 128-row halves). A single-stage item has no second stage to overlap its
  // softmax with, but takes well under a whole unit's time, so the last
  // round ends sooner. Causal units stay whole: their longest-first order
  // already fills the last round with short units.
  const int T = p.n_units % G;
  const int n_split = (!causal && T > 0 && 2 * T <= G && pb.Nq > rows_per_unit / 2) ? T : 0;
  p.n_full = p.n_units - n_split;
  p.n_items = p.n_full + 2 * n_split;
}

}  // namespace fwdp
}  // namespace fa
