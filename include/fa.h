/*
 * fa.h — C ABI of the exact-attention library for one NVIDIA GB300 (sm_103a).
 *
 * What is computed. Exact scaled-dot-product attention
 *     O = softmax(scale * Q K^T [+ causal mask]) V
 * (the post "FlashAttention v1", deep_school #630, section "Проблема
 * базового attention"), evaluated tile by tile with online softmax so the
 * Nq x Nk score matrix never reaches device memory (same post, sections
 * "Тайлинг (Tiling)" and "Онлайн-Softmax"). The result equals the classical
 * softmax up to floating-point rounding. The backward pass recomputes the
 * probabilities from the saved log-sum-exp instead of storing them (the
 * FlashAttention-3 summary on news.hada.io, section "Resumo do
 * FlashAttention": tiling and recomputation).
 *
 * Conventions shared by every call.
 *   Layout   : contiguous, head dimension innermost ("BSHD").
 *              q, o, dout, dq : [B, Nq, Hq, d]   bf16
 *              k, v, dk, dv   : [B, Nk, Hkv, d]  bf16
 *              lse            : [B, Hq, Nq]      fp32, natural log:
 *                               lse[b,h,i] = ln sum_j exp(scale * q_i . k_j)
 *                               over the keys j visible to row i.
 *   GQA      : query head h reads kv head h / (Hq / Hkv); Hq % Hkv == 0.
 *   Causal   : causal = 1 hides key j from query i when j > i + (Nk - Nq)
 *              (bottom-right alignment; with Nq == Nk this is j > i). A row
 *              that sees no key gets o = 0 and lse = -inf.
 *   Sizes    : B, Hq, Hkv, Nq, Nk >= 1; d in {64, 128}; scale any finite
 *              value (negative: the softmax of the negated scores; zero:
 *              every visible key weighted equally); every element count
 *              and B*Hq*Nq*d fit in int32 indices per the limits checked
 *              below.
 *   Pointers : device pointers owned by the caller, 16-byte aligned. The
 *              library keeps no pointer after a call returns.
 *   Stream   : `stream` is a cudaStream_t (NULL = legacy default stream).
 *              Calls only enqueue work; outputs are valid once the stream
 *              has been synchronised. The calls are not re-entrant on one
 *              stream from several host threads.
 *   Errors   : argument errors are detected on the host before anything is
 *              enqueued and return FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED.
 *              A failed launch returns FA_ERR_LAUNCH. Every wait inside the
 *              kernels is bounded; a wait that runs out stops the kernel and
 *              records FA_ERR_TIMEOUT in a per-device status word that
 *              fa_get_status() returns.
 */
#ifndef FA_H_
#define FA_H_

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, bad scale or flag */
  FA_ERR_UNSUPPORTED = 2, /* valid request this build does not serve (e.g. d not in {64,128}) */
  FA_ERR_ALLOC = 3,       /* device workspace allocation failed */
  FA_ERR_LAUNCH = 4,      /* a CUDA call or kernel launch failed */
  FA_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out (reported by fa_get_status) */
  FA_ERR_NO_DEVICE = 6    /* no usable sm_103 device is current */
} fa_status;

/*
 * fa_fwd — forward pass.
 *   in : q [B,Nq,Hq,d], k [B,Nk,Hkv,d], v [B,Nk,Hkv,d]   (bf16, device)
 *   out: o [B,Nq,Hq,d] (bf16), lse [B,Hq,Nq] (fp32)        (device)
 * Needs no device workspace. All outputs are fully written.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq, int Nk,
           int d, float scale, int causal, void* stream);

/*
 * fa_fwd_window — the forward pass with a sliding-window (local) mask (the
 *   FlashAttention-4 article on smntcn.com names variable and local masks;
 *   the pages do not define them, so this is the causal mask's bottom-right
 *   alignment with two bounds).
 *   Key j is visible to query row i iff
 *       i + off - window_left <= j <= i + off + window_right,  off = Nk - Nq
 *   (the bottom-right alignment of the causal mask); a negative bound, or one
 *   of at least Nq + Nk, means no limit on that side. window_right = 0 with
 *   window_left < 0 is the causal mask; both negative is fa_fwd non-causal.
 *   Rows that see no key get O = 0 and LSE = -inf. Key tiles outside every
 *   row's window are skipped, so the work scales with the window.
 *   Arguments, layouts, ownership and errors otherwise as fa_fwd.
 */
int fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                  int Nk, int d, float scale, int window_left, int window_right, void* stream);

/*
 * fa_fwd_fp8 — the forward pass with e4m3 (FP8) tensor-core GEMMs, d = 128.
 *   Inputs, outputs, layouts and the causal flag as fa_fwd (bf16 q, k, v in,
 *   bf16 o and fp32 lse out). incoherent = 1 first multiplies Q and K along
 *   d by diag(signs) H_128 / sqrt(128) (H the Sylvester-Hadamard matrix;
 *   sign_i = -1 where bit 31 of 2654435769 * (i + 1) mod 2^32 is set), which
 *   leaves Q K^T unchanged and spreads outlier channels; incoherent = 0
 *   skips it. Q (transformed), K (transformed) and V are then divided per
 *   (batch, head) by the smallest power of two that brings their largest
 *   magnitude to at most 448 (into (224, 448]) and rounded to e4m3 (nearest,
 *   ties to even; a division by a power of two is exact, so each code is the
 *   rounding of the exact quotient); P is rounded to e4m3 for the P V GEMM.
 *   The result approximates fa_fwd's: O is the attention of the dequantised
 *   tensors up to the rounding of P. (The FlashAttention-3 summary on
 *   news.hada.io, sections on FP8 and incoherent processing: e4m3 GEMMs,
 *   and a random orthogonal transform that spreads outliers before
 *   quantisation.)
 *   Workspace: the e4m3 copies (B*(Nq*Hq + Nk*Hkv)*128 bytes plus
 *   B*Hkv*128*ceil(Nk/128)*128 for V transposed) and per-head maxima, from
 *   the per-device pool fa_bwd uses, on `stream`.
 *   Errors as fa_fwd; d != 128 returns FA_ERR_UNSUPPORTED; incoherent other
 *   than 0/1 returns FA_ERR_INVALID_ARG.
 */
int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
               int Nk, int d, float scale, int causal, int incoherent, void* stream);

/*
 * fa_bwd — backward pass for L = sum(dout * o).
 *   in : q, k, v, o (bf16), lse (fp32, as written by fa_fwd for the same
 *        inputs), dout [B,Nq,Hq,d] (bf16)
 *   out: dq [B,Nq,Hq,d], dk [B,Nk,Hkv,d], dv [B,Nk,Hkv,d] (bf16), fully written.
 * Allocates its fp32 workspace (dq accumulator, row terms D_i) with the
 * stream-ordered allocator on `stream`, from a memory pool the library keeps
 * per device, and frees it on the same stream; the pool keeps freed memory
 * (up to the largest workspace used so far) for later calls until the
 * process exits. Returns FA_ERR_ALLOC if the allocation fails. GQA gradients of dk/dv are summed over
 * the query heads of each group inside the kernel.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
           void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
           void* stream);

/*
 * fa_bwd_window — the backward pass of fa_fwd_window: the same window
 *   bounds (and the o, lse that fa_fwd_window wrote); key tiles and query
 *   tiles outside every window are skipped. Arguments, layouts, workspace
 *   and errors otherwise as fa_bwd.
 */
int fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                  void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                  int window_left, int window_right, void* stream);

/*
 * fa_step_host — one forward and backward pass on HOST buffers: the
 * end-to-end call for a caller whose tensors live in host memory. The
 * operations are those of fa_fwd followed by fa_bwd (same arguments, layouts
 * and results), with every pointer a host address:
 *   in : q [B,Nq,Hq,d], k, v [B,Nk,Hkv,d], dout [B,Nq,Hq,d] (bf16)
 *   out: o [B,Nq,Hq,d] (bf16), lse [B,Hq,Nq] (fp32), dq, dk, dv (bf16).
 * The batch is processed in chunks and pipelined over library-owned
 * streams (one copy stream each way, one compute stream): a chunk is one
 * batch element, or, for a batch of one element with an even Hkv, one half
 * of its kv heads with their query heads (copied as 2-D slices of the head
 * dimension). The forward runs as two launches over halves of the chunks:
 * the first starts once its half's q, k, v are in, and its O and LSE go
 * out while the second runs; dout is copied in meanwhile. The backward runs
 * as one launch over all chunks, and dq, dk, dv go out after it.
 * The call only enqueues; `stream` is ordered after all of it, so
 * synchronise `stream` before reading the outputs, and keep every host
 * buffer alive (and the inputs unchanged) until then. Nothing of the
 * call waits for earlier work on `stream` (the copies and kernels touch only
 * the host buffers and the library's device buffers): the host inputs must
 * hold their values when the call is made. Consecutive calls therefore
 * overlap: the inputs of one call are copied in while the previous call
 * computes, and its kernels start while the previous call's last results
 * are still being copied out.
 * Page-locked host memory gives asynchronous, full-speed copies; pageable
 * memory works but the copies are staged by the driver.
 * Device memory: two library-owned buffers per device, each a copy of every
 * tensor of the batch (about the size of all inputs and outputs), used by
 * alternate calls and kept (grown to the largest call) until the process
 * exits; a call waits only for the call two before it to release its
 * buffer. Calls from several host threads on one device are serialised
 * while they enqueue. Plus the backward's own workspace from its pool.
 * Errors: a null pointer or a bad size gives FA_ERR_INVALID_ARG /
 * FA_ERR_UNSUPPORTED before anything is enqueued; FA_ERR_ALLOC if the device
 * copy cannot be allocated; FA_ERR_LAUNCH if a copy, launch or event call
 * fails (work already enqueued still completes in order on `stream`).
 */
int fa_step_host(const void* q, const void* k, const void* v, const void* dout, void* o, float* lse, void* dq,
                 void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                 void* stream);

/*
 * fa_bwd_noalloc — the same backward pass as fa_bwd, for callers that may
 * not allocate device memory during the call: serving loops that fix their
 * memory plan at start-up, and code that runs where the CUDA allocator must
 * not be entered. The pages have no counterpart of this call; it only
 * changes where the workspace lives.
 *   Arguments, layouts, results and argument errors are those of fa_bwd.
 *   Workspace: a file-scope device array of FA_BWD_NOALLOC_SCRATCH_BYTES
 *     (64 MiB) inside the library. Every device that loads the library holds
 *     it until the process exits. The call needs
 *       4 * B*Hq*ceil(Nq/128)*128 * (d + 2) bytes of it and returns
 *     FA_ERR_UNSUPPORTED, without enqueuing anything, when that exceeds the
 *     array. The causal GQA backward at d = 128 splits its last round per
 *     query head only where the pieces' fp32 slots (4 * 2 * 128 * d bytes
 *     each) fit in the rest of the array; otherwise that round runs whole
 *     single tiles (same results up to the order of fp32 additions).
 *   No cudaMalloc, cudaFree or other allocating routine is called.
 *   Set-up: the first call on each device looks up the array's device
 *     address on that device (cudaGetSymbolAddress); make that first call
 *     before any stream capture. A failed look-up returns FA_ERR_LAUNCH.
 *   Sharing: all calls on a device share the one array, and it keeps the
 *     last call's contents (the call re-initialises what it reads). Calls
 *     whose work overlaps on the GPU (different streams, no ordering between
 *     them) race on the array and give wrong results; order them.
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (64ull << 20)
/*
 * fa_bwd_launches — how many kernels fa_bwd launches for this problem
 *   (fa_bwd_noalloc: the same, or one fewer where the tail slots would not
 *   fit its array): the pre-pass, the main kernel and the dQ conversion,
 *   plus, for the causal GQA backward at d = 128 whose last round is split
 *   per query head, the pass that sums the pieces' dK/dV. With the split
 *   count of the current fa_tune setting and this GPU's SM count. For
 *   profiling and accounting; returns the count, or minus an fa_status for
 *   sizes fa_bwd would reject.
 */
int fa_bwd_launches(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal);
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                   void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                   int causal, void* stream);

/*
 * fa_get_status — synchronises `stream`, then returns and clears the
 * current device's status word: FA_OK, or FA_ERR_TIMEOUT if any kernel of
 * this library gave up on a bounded wait since the last call. A CUDA error
 * seen while synchronising is returned as FA_ERR_LAUNCH.
 */
int fa_get_status(void* stream);

/* fa_status_string — static, human-readable name of a status code. */
const char* fa_status_string(int status);

/*
 * Test hooks (not for production use).
 * fa_debug_set — wait_limit_ns: per-wait time limit of every kernel (0
 *   restores the default of 2 s). inject: 0 = off; 1 = the forward producer
 *   never issues its first K-tile load, so the consumer's bounded wait must
 *   run out and the kernel must report FA_ERR_TIMEOUT and exit cleanly.
 *   Process-wide; not thread-safe.
 * fa_debug_exp2 — y[i] = 2^x[i] for n device floats, evaluated by the
 *   kernels' own device routine: mode 0 = ex2.approx on the special-function
 *   unit, mode 1 = the fitted polynomial on the FMA pipes.
 */
int fa_debug_set(unsigned long long wait_limit_ns, int inject);

int fa_debug_exp2(const float* x, float* y, int n, int mode, void* stream);

/*
 * fa_tune — process-wide tuning knob, read by every later launch (not
 *   thread-safe). Returns FA_ERR_INVALID_ARG for an unknown knob or value.
 *   FA_TUNE_EXP2_SPLIT: how the forward softmax evaluates its exponentials
 *     (the FlashAttention-4 article on smntcn.com: part of the exponentials
 *     are emulated in software on the FMA pipes because the special-function
 *     unit does not keep up with the tensor cores). value 0 (the default):
 *     every exponential by ex2.approx on the special-function unit; value N
 *     in {1, 2, 4, 8}: one column pair in every N by the fitted degree-3
 *     polynomial on the FMA pipes (relative error below 7.5e-5; N = 1: all
 *     of them), the rest as before. Applies to fa_fwd (both head dims,
 *     causal or not) and fa_fwd_fp8; fa_fwd_window and the backward always
 *     use the special-function unit. Results differ from the default only
 *     by the polynomial's rounding.
 */
#define FA_TUNE_EXP2_SPLIT 1
/*
 *   FA_TUNE_CTA_PAIRS: value 1 runs fa_fwd (d = 128, causal or not; not
 *     fa_fwd_window) on pairs of CTAs: a cluster of two CTAs takes 512
 *     query rows at a time and the even one issues tcgen05.mma with
 *     cta_group::2 (M = 256 over both CTAs' tensor memory), each CTA loading
 *     half of every K and V tile (the FlashAttention-4 article on smntcn.com:
 *     fifth-generation tensor cores and 256 KB of tensor memory per SM; the
 *     pair form halves the MMA instructions and the K/V shared-memory
 *     traffic per flop). value 0 (the default): one CTA per SM. The exp2
 *     split does not apply to the paired kernel. Results are the same up to
 *     the order of floating-point additions.
 */
#define FA_TUNE_CTA_PAIRS 2
/*
 *   FA_TUNE_BWD_SPLIT: the causal backward (no left window bound) runs key
 *     tiles in pairs (j, n-1-j) of equal work; of each kv head's pairs, the
 *     m nearest the middle run as single tiles to fill the last round of
 *     the persistent CTAs, and with grouped-query heads at d = 128 each such
 *     single is split further into one unit per query head, whose dK/dV are
 *     partial sums kept in fp32 and summed in a fixed order by a last pass
 *     (dK, dV stay deterministic). value -1
 *     (the default): m from a model of the round-robin schedule on this
 *     GPU's SM count; value m >= 0: that m (at most n/2). For tests of the
 *     split paths on small shapes; results differ only in the order of
 *     floating-point additions.
 */
#define FA_TUNE_BWD_SPLIT 3
int fa_tune(int knob, int value);

/*
 * fa_profile_events — begin/end are cudaEvent_t handles (or NULL to stop).
 *   While set, fa_fwd records `begin` on its stream right before its kernel
 *   and `end` right after it; fa_bwd does the same around its main
 *   (five-GEMM) kernel, leaving out the preprocess and dQ-convert kernels.
 *   The events are owned by the caller. Process-wide; not thread-safe.
 */
int fa_profile_events(void* begin, void* end);

/*
 * fa_trace — buf: device buffer of FA_TRACE_WORDS uint64 words (or NULL to
 *   stop). While set, the first FA_TRACE_CTAS CTAs of each main kernel write
 *   %globaltimer stamps (ns) at their pipeline hand-off points into
 *   buf[(cta * FA_TRACE_STEPS + step) * FA_TRACE_POINTS + point], for the
 *   first FA_TRACE_STEPS steps of that CTA; a step is one key tile of one
 *   unit (forward) or one query tile (backward). The points are listed in the
 *   kernels' sources. The buffer is owned by the caller; the library only
 *   writes it. Process-wide; not thread-safe. Available only in a library
 *   built with -DFA_ENABLE_TRACE (the build's FA_BUILD_TRACE=1); otherwise a
 *   non-NULL buffer returns FA_ERR_UNSUPPORTED.
 */
#define FA_TRACE_CTAS 4
#define FA_TRACE_STEPS 64
#define FA_TRACE_POINTS 16
#define FA_TRACE_WORDS (FA_TRACE_CTAS * FA_TRACE_STEPS * FA_TRACE_POINTS)
int fa_trace(void* buf);

#ifdef __cplusplus
}
#endif
#endif /* FA_H_ */
