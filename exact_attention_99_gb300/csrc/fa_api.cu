// C ABI of libfa: argument validation, per-device state, dispatch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "sm103_math.cuh"
#include "sm103_ptx.cuh"

namespace fa {

// Per-device status word: kernels OR error bits into it; fa_get_status reads
// and clears it. A file-scope __device__ word (one copy per device).
__device__ unsigned g_fa_status;

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;

std::mutex g_mu;
int g_sms[kMaxDevices];
cudaMemPool_t g_pool[kMaxDevices];
// fa_step_host: copy streams per device, kCopyLanes for each direction
// (host to device: even indices, device to host: odd), then one compute
// stream. One lane per direction measured fastest: splitting each copy over
// two streams per direction made the end-to-end step slower (1.44 instead
// of 1.19 ms).
constexpr int kCopyLanes = 1;
cudaStream_t g_copy[kMaxDevices][2 * kCopyLanes + 1];
// fa_step_host: two device buffers per device, used by alternate calls, so
// that a call's input copies can run while the previous call computes. A
// buffer is released (event on the caller's stream) once its call's last
// copy and kernel have finished; the call after next waits for that.
struct StepSlots {
  void* buf[2];
  size_t cap[2];
  cudaEvent_t released[2];
  bool pending[2];
  int next;
};
std::mutex g_step_mu;  // held for a whole fa_step_host enqueue
StepSlots g_step[kMaxDevices];
unsigned* g_status_ptr[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
DebugCfg g_debug = {kDefaultWaitNs, 0, nullptr, nullptr, nullptr, 0, 0, -1};

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// the copy streams of the current device, created on first use
bool copy_streams(cudaStream_t (&out)[2 * kCopyLanes + 1]) {
  const int dev = current_device();
  if (dev < 0) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < 2 * kCopyLanes + 1; ++i) {
    if (g_copy[dev][i] == nullptr && cudaStreamCreateWithFlags(&g_copy[dev][i], cudaStreamNonBlocking) != cudaSuccess) {
      g_copy[dev][i] = nullptr;
      return false;
    }
    out[i] = g_copy[dev][i];
  }
  return true;
}

// Argument checks shared by fa_fwd and fa_bwd (pointers checked by callers).
int check_sizes(int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  // index ranges: sequence coordinates and unit counts stay in int32,
  // tensor strides stay below the tensor-map limit of 2^40 bytes
  if (Nq > (1 << 28) || Nk > (1 << 28)) return FA_ERR_UNSUPPORTED;
  const long long q_elems = 1LL * B * Nq * Hq * d, k_elems = 1LL * B * Nk * Hkv * d;
  if (q_elems * 2 >= (1LL << 40) || k_elems * 2 >= (1LL << 40)) return FA_ERR_UNSUPPORTED;
  if (1LL * B * Hq * ((Nq + 255) / 256) >= (1LL << 30)) return FA_ERR_UNSUPPORTED;
  if (1LL * B * Hkv * ((Nk + 127) / 128) >= (1LL << 30)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

int check_device() {
  const int dev = current_device();
  if (dev < 0) return FA_ERR_NO_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return FA_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return FA_ERR_NO_DEVICE;
  if (major != 10 || minor != 3) return FA_ERR_NO_DEVICE;
  return FA_OK;
}

__global__ void debug_exp2_kernel(const float* x, float* y, int n, int mode) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float a = x[i];
  if (mode == 0) {
    y[i] = ex2_mufu(a);
  } else {
    float b = a;
    exp2_poly_pair(a, b);
    y[i] = a;
  }
}

}  // namespace

int normalize_window(int w, int Nq, int Nk) {
  if (w < 0) return -1;
  if (1LL * w >= 1LL * Nq + Nk) return -1;
  return w;
}


// Stream-ordered pool for the backward workspace, one per device, that
// keeps freed memory for the next call (release threshold = max) instead of
// returning it to the driver at every synchronisation.
cudaMemPool_t workspace_pool() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_pool[dev] == nullptr) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    uint64_t keep = ~0ull;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    g_pool[dev] = pool;
  }
  return g_pool[dev];
}

DebugCfg debug_cfg() {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_debug;
}

int num_sms() {
  const int dev = current_device();
  if (dev < 0) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sms[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 1;
  }
  return g_sms[dev];
}

unsigned* status_word() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_status_ptr[dev];
}

// cuTensorMapEncodeTiled from the driver, looked up once
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      cudaGetLastError();
      return nullptr;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

bool encode_tiled(CUtensorMap* m, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                  const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  return encode(m, dtype, rank, const_cast<void*>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_bshd_map(CUtensorMap* m, const void* base, int B, int N, int H, int d, int box_rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2, (cuuint64_t)N * H * d * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int check_bwd_args(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                   void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                   int causal) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  const int st = check_sizes(B, Hq, Hkv, Nq, Nk, d, scale, causal);
  if (st != FA_OK) return st;
  return check_device();
}

cudaError_t launch_debug_exp2(const float* x, float* y, int n, int mode, cudaStream_t stream) {
  debug_exp2_kernel<<<(n + 255) / 256, 256, 0, stream>>>(x, y, n, mode);
  return cudaGetLastError();
}

}  // namespace fa

using namespace fa;

extern "C" int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                      int Nk, int d, float scale, int causal, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_INVALID_ARG;
  int st = check_sizes(B, Hq, Hkv, Nq, Nk, d, scale, causal);
  if (st != FA_OK) return st;
  st = check_device();
  if (st != FA_OK) return st;
  Problem p{q, k, v, B, Hq, Hkv, Nq, Nk, d, scale, causal};
  return launch_fwd(p, o, lse, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

extern "C" int fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                             int Nq, int Nk, int d, float scale, int window_left, int window_right, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_INVALID_ARG;
  int st = check_sizes(B, Hq, Hkv, Nq, Nk, d, scale, 0);
  if (st != FA_OK) return st;
  st = check_device();
  if (st != FA_OK) return st;
  Problem p{q, k, v, B, Hq, Hkv, Nq, Nk, d, scale, 0};
  p.window_left = normalize_window(window_left, Nq, Nk);
  p.window_right = normalize_window(window_right, Nq, Nk);
  return launch_fwd(p, o, lse, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

extern "C" int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                          int Nq, int Nk, int d, float scale, int causal, int incoherent, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_INVALID_ARG;
  if (incoherent != 0 && incoherent != 1) return FA_ERR_INVALID_ARG;
  int st = check_sizes(B, Hq, Hkv, Nq, Nk, d, scale, causal);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  st = check_device();
  if (st != FA_OK) return st;
  const Problem p{q, k, v, B, Hq, Hkv, Nq, Nk, d, scale, causal};
  const cudaError_t e = launch_fwd8(p, o, lse, incoherent, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorMemoryAllocation) {
    cudaGetLastError();
    return FA_ERR_ALLOC;
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

namespace {
// fa_bwd / fa_bwd_window after their checks: workspace from the pool,
// launch, free, all on the caller's stream
int bwd_pooled(const Problem& p, const void* o, const float* lse, const void* dout, void* dq, void* dk, void* dv,
               void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaMemPool_t pool = workspace_pool();
  void* ws = nullptr;
  if (pool == nullptr || cudaMallocFromPoolAsync(&ws, bwd_workspace_bytes(p), pool, s) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_ALLOC;
  }
  const cudaError_t e = launch_bwd(p, o, lse, dout, dq, dk, dv, static_cast<float*>(ws), s);
  const cudaError_t f = cudaFreeAsync(ws, s);
  if (e != cudaSuccess || f != cudaSuccess) return FA_ERR_LAUNCH;
  return FA_OK;
}
}  // namespace

extern "C" int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                      void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                      int causal, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  int st = check_sizes(B, Hq, Hkv, Nq, Nk, d, scale, causal);
  if (st != FA_OK) return st;
  st = check_device();
  if (st != FA_OK) return st;
  const Problem p{q, k, v, B, Hq, Hkv, Nq, Nk, d, scale, causal};
  return bwd_pooled(p, o, lse, dout, dq, dk, dv, stream);
}

extern "C" int fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk,
                             int d, float scale, int window_left, int window_right, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  int st = check_sizes(B, Hq, Hkv, Nq, Nk, d, scale, 0);
  if (st != FA_OK) return st;
  st = check_device();
  if (st != FA_OK) return st;
  Problem p{q, k, v, B, Hq, Hkv, Nq, Nk, d, scale, 0};
  p.window_left = normalize_window(window_left, Nq, Nk);
  p.window_right = normalize_window(window_right, Nq, Nk);
  return bwd_pooled(p, o, lse, dout, dq, dk, dv, stream);
}

extern "C" int fa_get_status(void* stream) {
  if (check_device() != FA_OK) return FA_ERR_NO_DEVICE;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_LAUNCH;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fa_status, sizeof(v)) != cudaSuccess) return FA_ERR_LAUNCH;
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_LAUNCH;
  return (v & kDevTimeout) ? FA_ERR_TIMEOUT : FA_OK;
}

extern "C" const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_ALLOC: return "FA_ERR_ALLOC";
    case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_NO_DEVICE: return "FA_ERR_NO_DEVICE";
    default: return "FA_ERR_UNKNOWN";
  }
}

extern "C" int fa_debug_set(unsigned long long wait_limit_ns, int inject) {
  if (inject < 0 || inject > 1) return FA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_debug.wait_limit_ns = wait_limit_ns == 0 ? kDefaultWaitNs : wait_limit_ns;
  g_debug.inject = inject;
  return FA_OK;
}

extern "C" int fa_bwd_launches(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal) {
  const int st = check_sizes(B, Hq, Hkv, Nq, Nk, d, 1.0f, causal);
  if (st != FA_OK) return -st;
  const Problem p{nullptr, nullptr, nullptr, B, Hq, Hkv, Nq, Nk, d, 1.0f, causal};
  return bwd_launch_count(p);
}

extern "C" int fa_tune(int knob, int value) {
  if (knob == FA_TUNE_EXP2_SPLIT) {
    if (value != 0 && value != 1 && value != 2 && value != 4 && value != 8) return FA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    g_debug.poly_every = value;
    return FA_OK;
  }
  if (knob == FA_TUNE_CTA_PAIRS) {
    if (value != 0 && value != 1) return FA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    g_debug.cta_pairs = value;
    return FA_OK;
  }
  if (knob == FA_TUNE_BWD_SPLIT) {
    if (value < -1) return FA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    g_debug.bwd_split = value;
    return FA_OK;
  }
  return FA_ERR_INVALID_ARG;
}

extern "C" int fa_profile_events(void* begin, void* end) {
  if ((begin == nullptr) != (end == nullptr)) return FA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_debug.ev_begin = static_cast<cudaEvent_t>(begin);
  g_debug.ev_end = static_cast<cudaEvent_t>(end);
  return FA_OK;
}

extern "C" int fa_trace(void* buf) {
#ifndef FA_ENABLE_TRACE
  if (buf != nullptr) return FA_ERR_UNSUPPORTED;
#endif
  if (buf != nullptr && (reinterpret_cast<uintptr_t>(buf) & 7u) != 0) return FA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_debug.trace = static_cast<unsigned long long*>(buf);
  return FA_OK;
}

extern "C" int fa_debug_exp2(const float* x, float* y, int n, int mode, void* stream) {
  if (!aligned16(x) || !aligned16(y) || n < 0 || (mode != 0 && mode != 1)) return FA_ERR_INVALID_ARG;
  if (n == 0) return FA_OK;
  const int st = check_device();
  if (st != FA_OK) return st;
  return launch_debug_exp2(x, y, n, mode, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

extern "C" int fa_step_host(const void* q, const void* k, const void* v, const void* dout, void* o, float* lse,
                            void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                            int causal, void* stream) {
  if (!q || !k || !v || !dout || !o || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  int st = check_sizes(B, Hq, Hkv, Nq, Nk, d, scale, causal);
  if (st != FA_OK) return st;
  st = check_device();
  if (st != FA_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t cs[2 * kCopyLanes + 1];
  if (!copy_streams(cs)) return FA_ERR_LAUNCH;
  // the kernels run on the library's compute stream: they read and write
  // only the library's buffers, so they wait for their input copies and not
  // for `stream`, which the previous call left waiting for its last copies
  // out; this call's compute then runs while those copies drain
  const cudaStream_t sc = cs[2 * kCopyLanes];
  // Chunks: one batch element each; a batch of one element is cut into two
  // halves of its kv heads (each with its query heads) when Hkv is even.
  // On the device every tensor is stored chunk after chunk, [chunk][rows]
  // [hq or hk heads][d] (LSE [chunk][hq][Nq]), i.e. as a batch of n_chunks
  // elements with hq query and hk kv heads: the same attention problem,
  // since (batch, head) pairs are independent. The forward runs in two
  // launches over halves of the chunks, so that it starts once the first
  // half's inputs are in and the first half's O goes out while the second
  // computes; the backward runs as one launch over all chunks (per-chunk
  // backward launches left the persistent kernel's last round half empty:
  // 6.3 instead of 5.9 ms per call on the causal GQA N16384 step), and its
  // results go out after it.
  const int C = (B == 1 && Hkv % 2 == 0) ? 2 : 1;  // kv-head slices per batch element
  const int hk = Hkv / C, hq = Hq / C;
  const size_t e2 = 2;  // bf16
  const size_t bq = size_t(Nq) * hq * d * e2, bk = size_t(Nk) * hk * d * e2, nl = size_t(hq) * Nq;
  const int n_chunks = B * C;
  const int F = n_chunks >= 2 ? 2 : 1;  // forward launches
  const size_t per = 4 * bq + 4 * bk + nl * 4;
  const int dev = current_device();
  if (dev < 0) return FA_ERR_LAUNCH;
  std::lock_guard<std::mutex> step_lock(g_step_mu);
  StepSlots& slots = g_step[dev];
  const int slot = slots.next;
  slots.next ^= 1;
  if (slots.released[slot] == nullptr &&
      cudaEventCreateWithFlags(&slots.released[slot], cudaEventDisableTiming) != cudaSuccess) {
    slots.released[slot] = nullptr;
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  const size_t need = per * size_t(n_chunks);
  if (slots.cap[slot] < need) {  // grow: wait for the buffer's last user, then reallocate
    if (slots.pending[slot]) cudaEventSynchronize(slots.released[slot]);
    if (slots.buf[slot] != nullptr) cudaFree(slots.buf[slot]);
    slots.buf[slot] = nullptr;
    slots.cap[slot] = 0;
    slots.pending[slot] = false;
    if (cudaMalloc(&slots.buf[slot], need) != cudaSuccess) {
      slots.buf[slot] = nullptr;
      cudaGetLastError();
      return FA_ERR_ALLOC;
    }
    slots.cap[slot] = need;
  }
  void* ws = slots.buf[slot];
  // events, per copy lane: "q, k, v of forward group f in" (f < 2) and
  // "dout in"; then "forward f done" (f < 2) and "backward done"; then one
  // "done" per copy stream and one for the compute stream
  const auto ev_qkv = [](int f, int l) { return size_t(f) * kCopyLanes + l; };
  const auto ev_do = [](int l) { return size_t(2) * kCopyLanes + l; };
  const auto ev_fwd = [](int f) { return size_t(3) * kCopyLanes + f; };
  const size_t ev_bwd = 3 * kCopyLanes + 2, per_c = 3 * kCopyLanes + 3;
  std::vector<cudaEvent_t> ev(per_c + 2 * kCopyLanes + 1, nullptr);
  bool ok = true;
  for (auto& e : ev) ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
  // the copies wait only for the previous user of this buffer (two calls
  // back), not for earlier work on the caller's stream
  if (ok && slots.pending[slot]) {
    for (int i = 0; i < 2 * kCopyLanes && ok; ++i)
      ok = cudaStreamWaitEvent(cs[i], slots.released[slot], 0) == cudaSuccess;
  }
  const auto* hq_ = static_cast<const uint8_t*>(q);
  const auto* hk_ = static_cast<const uint8_t*>(k);
  const auto* hv_ = static_cast<const uint8_t*>(v);
  const auto* hdo = static_cast<const uint8_t*>(dout);
  auto* ho = static_cast<uint8_t*>(o);
  auto* hl = reinterpret_cast<uint8_t*>(lse);
  auto* hdq = static_cast<uint8_t*>(dq);
  auto* hdk = static_cast<uint8_t*>(dk);
  auto* hdv = static_cast<uint8_t*>(dv);
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  // rows x (h heads of d) bf16 between a [rows, H, d] host tensor (starting
  // at head h0) and a contiguous [rows, h, d] device buffer: one 2-D copy
  // (plain 1-D when the slice is the whole row), split in kCopyLanes
  // contiguous pieces of rows over the copy streams of one direction
  auto copy_heads = [&](uint8_t* dev, uint8_t* host, int rows, int H, int h0, int h, cudaMemcpyKind kind,
                        int dir) -> bool {
    const size_t w = size_t(h) * d * e2, pitch = size_t(H) * d * e2;
    const int piece = (rows + kCopyLanes - 1) / kCopyLanes;
    for (int l = 0; l < kCopyLanes; ++l) {
      const int r0 = piece * l;
      if (r0 >= rows) break;
      const int nr = rows - r0 < piece ? rows - r0 : piece;
      uint8_t* hp = host + size_t(r0) * pitch + size_t(h0) * d * e2;
      uint8_t* dp = dev + size_t(r0) * w;
      const cudaError_t e =
          w == pitch ? cudaMemcpyAsync(kind == h2d ? dp : hp, kind == h2d ? hp : dp, w * nr, kind, cs[2 * l + dir])
                     : (kind == h2d ? cudaMemcpy2DAsync(dp, w, hp, pitch, w, nr, kind, cs[2 * l + dir])
                                    : cudaMemcpy2DAsync(hp, pitch, dp, w, w, nr, kind, cs[2 * l + dir]));
      if (e != cudaSuccess) return false;
    }
    return true;
  };
  auto in = [&](uint8_t* dev, const uint8_t* host, int rows, int H, int h0, int h) {
    return copy_heads(dev, const_cast<uint8_t*>(host), rows, H, h0, h, h2d, 0);
  };
  auto out = [&](uint8_t* host, uint8_t* dev, int rows, int H, int h0, int h) {
    return copy_heads(dev, host, rows, H, h0, h, d2h, 1);
  };
  uint8_t* const base = static_cast<uint8_t*>(ws);
  uint8_t *const Rq = base, *const Rdo = Rq + n_chunks * bq, *const Ro = Rdo + n_chunks * bq;
  uint8_t *const Rdq = Ro + n_chunks * bq, *const Rk = Rdq + n_chunks * bq, *const Rv = Rk + n_chunks * bk;
  uint8_t *const Rdk = Rv + n_chunks * bk, *const Rdv = Rdk + n_chunks * bk;
  float* const Rl = reinterpret_cast<float*>(Rdv + n_chunks * bk);
  // chunk c = (batch element b, kv-head slice g): its host offsets
  const auto qoff = [&](int c) { return size_t(c / C) * Nq * Hq * d * e2; };
  const auto koff = [&](int c) { return size_t(c / C) * Nk * Hkv * d * e2; };
  const auto first = [&](int f) { return n_chunks * f / F; };  // first chunk of forward group f
  // inputs: q, k, v of the first forward group, then of the second, then
  // dout (needed by the backward only)
  for (int f = 0; f < F && ok; ++f) {
    for (int c = first(f); c < first(f + 1) && ok; ++c) {
      const int g = c % C;
      ok = in(Rq + c * bq, hq_ + qoff(c), Nq, Hq, g * hq, hq) && in(Rk + c * bk, hk_ + koff(c), Nk, Hkv, g * hk, hk) &&
           in(Rv + c * bk, hv_ + koff(c), Nk, Hkv, g * hk, hk);
    }
    for (int l = 0; l < kCopyLanes && ok; ++l) ok = cudaEventRecord(ev[ev_qkv(f, l)], cs[2 * l]) == cudaSuccess;
  }
  for (int c = 0; c < n_chunks && ok; ++c) ok = in(Rdo + c * bq, hdo + qoff(c), Nq, Hq, (c % C) * hq, hq);
  for (int l = 0; l < kCopyLanes && ok; ++l) ok = cudaEventRecord(ev[ev_do(l)], cs[2 * l]) == cudaSuccess;
  // forward group f on the compute stream; its O and LSE go out while the
  // next group (or the backward) runs. Host LSE [B][Hq][Nq] holds the chunks
  // in chunk order, so a group's LSE is one contiguous copy.
  for (int f = 0; f < F && ok; ++f) {
    const int c0 = first(f), nc = first(f + 1) - c0;
    for (int l = 0; l < kCopyLanes && ok; ++l) ok = cudaStreamWaitEvent(sc, ev[ev_qkv(f, l)], 0) == cudaSuccess;
    if (!ok) break;
    const Problem pf{Rq + c0 * bq, Rk + c0 * bk, Rv + c0 * bk, nc, hq, hk, Nq, Nk, d, scale, causal};
    ok = launch_fwd(pf, Ro + c0 * bq, Rl + c0 * nl, sc) == cudaSuccess &&
         cudaEventRecord(ev[ev_fwd(f)], sc) == cudaSuccess;
    for (int l = 0; l < kCopyLanes && ok; ++l)
      ok = cudaStreamWaitEvent(cs[2 * l + 1], ev[ev_fwd(f)], 0) == cudaSuccess;
    for (int c = c0; c < c0 + nc && ok; ++c) ok = out(ho + qoff(c), Ro + c * bq, Nq, Hq, (c % C) * hq, hq);
    ok = ok && cudaMemcpyAsync(hl + size_t(c0) * nl * 4, Rl + c0 * nl, nc * nl * 4, d2h, cs[1]) == cudaSuccess;
  }
  // the backward over all chunks, then its results out
  for (int l = 0; l < kCopyLanes && ok; ++l) ok = cudaStreamWaitEvent(sc, ev[ev_do(l)], 0) == cudaSuccess;
  if (ok) {
    const Problem pb{Rq, Rk, Rv, n_chunks, hq, hk, Nq, Nk, d, scale, causal};
    ok = bwd_pooled(pb, Ro, Rl, Rdo, Rdq, Rdk, Rdv, sc) == FA_OK && cudaEventRecord(ev[ev_bwd], sc) == cudaSuccess;
  }
  for (int l = 0; l < kCopyLanes && ok; ++l) ok = cudaStreamWaitEvent(cs[2 * l + 1], ev[ev_bwd], 0) == cudaSuccess;
  for (int c = 0; c < n_chunks && ok; ++c) {
    const int g = c % C;
    ok = out(hdq + qoff(c), Rdq + c * bq, Nq, Hq, g * hq, hq) && out(hdk + koff(c), Rdk + c * bk, Nk, Hkv, g * hk, hk) &&
         out(hdv + koff(c), Rdv + c * bk, Nk, Hkv, g * hk, hk);
  }
  // the caller's stream waits for every copy stream and the compute stream,
  // then releases the buffer
  for (int i = 0; i < 2 * kCopyLanes + 1; ++i) {
    cudaEvent_t e = ev[per_c + i];
    if (e != nullptr && cudaEventRecord(e, cs[i]) == cudaSuccess) cudaStreamWaitEvent(s, e, 0);
  }
  const bool released = cudaEventRecord(slots.released[slot], s) == cudaSuccess;
  slots.pending[slot] = released;
  for (auto& e : ev)
    if (e != nullptr) cudaEventDestroy(e);
  if (!ok || !released) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}
