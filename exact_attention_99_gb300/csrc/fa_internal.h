// Host-side declarations shared by the translation units of libfa.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Status bits written by kernels into the per-device status word.
constexpr unsigned kDevTimeout = 1u;

struct Problem {
  const void* q;
  const void* k;
  const void* v;
  int B, Hq, Hkv, Nq, Nk, d;
  float scale;
  int causal;
  // sliding window: key j visible to query i iff i + off - window_left <= j
  // <= i + off + window_right (off = Nk - Nq); -1 = no limit on that side
  int window_left = -1, window_right = -1;
  // backward: largest workspace the call may use (0: any); the tail pieces
  // fall back to whole single tiles when their slots would not fit
  size_t ws_cap = 0;
  bool masked() const { return causal || window_left >= 0 || window_right >= 0; }
  // the causal mask and nothing else (window bounds already normalised)
  bool plain_causal() const { return window_left < 0 && (causal || window_right == 0); }
};

struct DebugCfg {
  unsigned long long wait_limit_ns;
  int inject;
  cudaEvent_t ev_begin;  // recorded around the main kernel when set
  cudaEvent_t ev_end;
  unsigned long long* trace;  // optional device trace buffer
  int poly_every;             // forward exp2 split (fa_tune FA_TUNE_EXP2_SPLIT)
  int cta_pairs;              // forward on CTA pairs (fa_tune FA_TUNE_CTA_PAIRS)
  int bwd_split;              // causal backward split count, -1 = model (fa_tune FA_TUNE_BWD_SPLIT)
};
DebugCfg debug_cfg();

// Per-device stream-ordered pool for the backward workspace (nullptr if it
// could not be created).
cudaMemPool_t workspace_pool();

// Device properties cached per device.
int num_sms();

// Per-device status word (device pointer), created on first use.
unsigned* status_word();

// 4-D bf16 tensor map over a BSHD tensor [B, N, H, d]: dims {d, H, N, B},
// box {64, 1, box_rows, 1}, 128-byte swizzle, zero fill out of range.
bool make_bshd_map(CUtensorMap* m, const void* base, int B, int N, int H, int d, int box_rows);

// Any tiled tensor map: rank <= 5, dims innermost first, strides (bytes) of
// dims 1..rank-1, zero fill out of range.
bool encode_tiled(CUtensorMap* m, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                  const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle);

// Window bounds as the kernels take them: negative -> -1 (no limit); a
// bound that reaches past every key (>= Nq + Nk) is no limit either.
int normalize_window(int w, int Nq, int Nk);

// The forward's exponent scale, scale * log2(e). A zero scale (every visible
// key equally weighted) becomes 2^-100: the scaled scores are then 0 to
// within fp32 rounding while a masked score (-inf) still gives probability 0,
// which 0 * -inf would not.
inline float exp_scale_log2(float scale) {
  return scale == 0.0f ? 7.888609052210118e-31f : scale * 1.4426950408889634f;
}

// Launchers. Return a cudaError_t (cudaSuccess on success).
cudaError_t launch_fwd(const Problem& p, void* o, float* lse, cudaStream_t stream);
// FP8 (e4m3) forward, d = 128 only; incoherent != 0 applies the Hadamard
// transform to Q and K before quantisation. Workspace from the pool.
cudaError_t launch_fwd8(const Problem& p, void* o, float* lse, int incoherent, cudaStream_t stream);
// The host-side checks fa_bwd performs (pointers, sizes, device), as one call.
int check_bwd_args(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                   void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                   int causal);

// Backward workspace (fp32 dQ accumulator, padded LSE*log2e and D rows).
size_t bwd_workspace_bytes(const Problem& p);
// kernels fa_bwd launches for p
int bwd_launch_count(const Problem& p);
cudaError_t launch_bwd(const Problem& p, const void* o, const float* lse, const void* dout, void* dq, void* dk,
                       void* dv, float* ws, cudaStream_t stream);
cudaError_t launch_debug_exp2(const float* x, float* y, int n, int mode, cudaStream_t stream);

}  // namespace fa
