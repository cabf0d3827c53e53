/*
 * dualkv.h -- C ABI of libdualkv.so: DualKV shared-prompt exact attention,
 * forward and backward, on one NVIDIA GB300 (sm_103a).
 *
 * Source of the method: "DualKV: Shared-Prompt Flash Attention for Efficient
 * RL Training with Large Rollouts and Long Contexts", abstract.  A micro-batch
 * holds one shared prompt of P tokens and N response segments; the data
 * pipeline stores the N(P+R) replicated tokens as P + sum_n R_n rows, and
 * each kernel walks, for a query, the prompt's keys and then those of the
 * query's own segment within one launch.  By the paper's account the result
 * is exactly causal attention on the N replicated sequences.
 *
 * Packed layout (all buffers contiguous, device memory unless stated):
 *   row t in [0, P)                 prompt token t, position t
 *   row P + R_offsets[n] + r        response token r of segment n, position P + r
 *   T = P + R_offsets[N] rows in total.
 *   q, out, dout, dq : [T, Hq, D]  bf16
 *   k, v, dk, dv     : [T, Hkv, D] bf16
 *   lse              : [Hq, T]     fp32, natural-log log-sum-exp of each row
 * Attention rule for a query at position p and a key at position p':
 *   the key lies in the prompt or in the query's own segment, p' <= p, and
 *   (window <= 0 or p - p' < window).
 * GQA: q-head h reads kv-head h / (Hq / Hkv).
 *
 * Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is
 * the legacy default stream).  Outputs are fully overwritten, never
 * accumulated.  Results are bitwise deterministic for a given GPU, library
 * build and input.  Inputs must be finite.  Every device pointer must be
 * 16-byte aligned.  The caller owns every buffer it passes; the library owns
 * only a bounded per-layout plan cache (small device arrays, see
 * dualkv_plan_cache_info) and a per-device status word, both freed by
 * dualkv_release().
 *
 * Return codes: DUALKV_OK, or one of the DUALKV_ERR_* values below; on an
 * error no kernel is launched (except DUALKV_ERR_CUDA, which reports a failed
 * launch).  Kernel-side failures do not abort the launch: a bounded wait that
 * timed out, or a work-list entry whose rows fall outside the tensors (the
 * kernels check each entry before using it and skip it), is recorded in the
 * status word and reported by dualkv_check_status().
 */
#ifndef DUALKV_H_
#define DUALKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DUALKV_OK 0
#define DUALKV_ERR_INVALID 1     /* bad sizes, offsets, head counts or head dimension */
#define DUALKV_ERR_ALIGN 2       /* a device pointer is not 16-byte aligned */
#define DUALKV_ERR_WORKSPACE 3   /* workspace missing or smaller than dualkv_bwd_workspace_bytes() */
#define DUALKV_ERR_CUDA 4        /* a CUDA runtime call or kernel launch failed */
#define DUALKV_ERR_DEVICE 5      /* a kernel reported a timeout or bounds violation */
#define DUALKV_ERR_UNSUPPORTED 6 /* valid arguments outside what this library supports */

/*
 * Forward pass (paper abstract: one kernel launch covers both key ranges of a
 * query, the shared prompt and the query's own response).  For every packed
 * query row and q-head:
 * S = scale * q k^T over the allowed keys of the prompt region and then of the
 * row's own segment, online softmax, out = softmax(S) v, lse = log-sum-exp(S).
 *
 *   q, k, v        device, bf16, layouts above (read only)
 *   P >= 0         prompt tokens; N >= 1 segments
 *   R_offsets      HOST int32[N+1], R_offsets[0] = 0, non-decreasing;
 *                  segment n has R_offsets[n+1] - R_offsets[n] >= 0 tokens
 *   Hq, Hkv        Hq % Hkv == 0
 *   D              head dimension: 64, 128 or 512
 *   scale          softmax scale (typically 1/sqrt(D))
 *   window         <= 0: global causal; else sliding window of `window` keys
 *   out            device bf16 [T, Hq, D] (written)
 *   lse            device fp32 [Hq, T] (written)
 */
int dualkv_fwd(const void* q, const void* k, const void* v, int P, int N, const int32_t* R_offsets, int Hq,
               int Hkv, int D, float scale, int window, void* out, float* lse, void* stream);

/*
 * Bytes of device workspace dualkv_bwd needs for this layout: the per-row
 * rowsum(dO * O) and log2-scaled LSE (2 * Hq * T fp32) plus the fp32 partial
 * dK/dV tiles of prompt key tiles whose query walk is split across CTAs; for
 * D = 512 also the bf16 P and dS blocks (2 x 32 KB per visited pair of a
 * 128-row query tile and a 128-key tile), about 32 GB for P=16384, N=16,
 * R=3072, Hq=8.
 * Returns 0 when the arguments are invalid.
 */
size_t dualkv_bwd_workspace_bytes(int P, int N, const int32_t* R_offsets, int Hq, int Hkv, int D, int window);

/*
 * Backward pass (paper abstract: fused backward kernels; the prompt's dK/dV
 * gather the contributions of every segment, since the packed result equals
 * standard attention on the replicated sequences with prompt gradients summed).
 * Runs: preprocess (Delta = rowsum(dout * out)), dK/dV (each key tile walks
 * every query block that attends it in a fixed order: for a prompt key tile the
 * blocks of segments 0..N-1 and then of the prompt, ascending; the group's
 * heads of one block consecutively), a fixed-order reduction of split prompt
 * tiles, and dQ.  For D = 512 the dK/dV and dQ products are formed from bf16
 * P and dS blocks kept in the workspace (see dualkv_bwd_workspace_bytes).
 *
 *   q, k, v, out, lse, dout   as produced for/by dualkv_fwd with the same layout
 *   dq, dk, dv                device bf16, written
 *   workspace                 device, >= dualkv_bwd_workspace_bytes(), 256-byte aligned
 */
int dualkv_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse, const void* dout,
               int P, int N, const int32_t* R_offsets, int Hq, int Hkv, int D, float scale, int window, void* dq,
               void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Head-range variants (paper abstract: the kernels integrate with Ulysses
 * sequence parallelism, which hands each rank a group of heads after its
 * all-to-all; heads never interact inside attention).  Same arguments, layout
 * and results as dualkv_fwd / dualkv_bwd on the full-head tensors, but only
 * kv-heads [kv_head_begin, kv_head_end) and their q-heads
 * [kv_head_begin * G, kv_head_end * G) (G = Hq / Hkv) are computed: out, lse
 * and dq of those q-heads and dk, dv of those kv-heads are written, every
 * other head of every output is left untouched, and only those heads of the
 * inputs are read.  Each head's result is bitwise identical to the one the
 * full call writes, so disjoint ranges may run as separate calls (one per
 * stream, or interleaved with the exchange that brings in each group) and
 * together equal one full call.  Calls on disjoint ranges may overlap on the
 * GPU if each backward call has its own workspace.  The workspace of
 * dualkv_bwd_heads needs at most dualkv_bwd_workspace_bytes() of the full
 * layout.  DUALKV_ERR_INVALID unless 0 <= kv_head_begin < kv_head_end <= Hkv.
 */
int dualkv_fwd_heads(const void* q, const void* k, const void* v, int P, int N, const int32_t* R_offsets, int Hq,
                     int Hkv, int D, float scale, int window, int kv_head_begin, int kv_head_end, void* out,
                     float* lse, void* stream);
int dualkv_bwd_heads(const void* q, const void* k, const void* v, const void* out, const float* lse, const void* dout,
                     int P, int N, const int32_t* R_offsets, int Hq, int Hkv, int D, float scale, int window,
                     int kv_head_begin, int kv_head_end, void* dq, void* dk, void* dv, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * Layer stacks (paper abstract: the method extends to models that interleave
 * sliding-window and global attention layers, with head dimension 512).  A
 * stack of n_layers attention layers over one packed micro-batch: every layer
 * shares the layout (P, N, R_offsets, Hq, Hkv, D, scale) and has its own
 * tensors and its own window (window[l] <= 0: global causal).  The layers run
 * back to back on `stream` in the order given (pass them in reverse order to
 * dualkv_bwd_layers for a model's backward pass); the plan of each distinct
 * window is built once and reused by every layer that has it, and the
 * backward layers share one workspace of at least
 * dualkv_bwd_layers_workspace_bytes() (the largest that any of its windows
 * needs; 0 for invalid input).  q[l], k[l], ... are host arrays of n_layers
 * device pointers, window a host array of n_layers ints.  The results are
 * bitwise those of n_layers dualkv_fwd / dualkv_bwd calls.  Every pointer of
 * every layer is checked before the first layer is launched.
 */
size_t dualkv_bwd_layers_workspace_bytes(int n_layers, const int32_t* window, int P, int N, const int32_t* R_offsets,
                                         int Hq, int Hkv, int D);
int dualkv_fwd_layers(int n_layers, const void* const* q, const void* const* k, const void* const* v,
                      const int32_t* window, int P, int N, const int32_t* R_offsets, int Hq, int Hkv, int D,
                      float scale, void* const* out, float* const* lse, void* stream);
int dualkv_bwd_layers(int n_layers, const void* const* q, const void* const* k, const void* const* v,
                      const void* const* out, const float* const* lse, const void* const* dout, const int32_t* window,
                      int P, int N, const int32_t* R_offsets, int Hq, int Hkv, int D, float scale, void* const* dq,
                      void* const* dk, void* const* dv, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Packing indices (host only, no GPU needed; paper abstract: the pipeline
 * stores N(P+R) replicated tokens as P+NR rows).  All outputs are HOST int32:
 *   seg_id[T]          -1 for prompt rows, else the segment of the row
 *   pos_id[T]          position of the row in its replicated sequence
 *   cu_seqlens_rep[N+1] start of replicated sequence n (length P + R_n)
 *   rep2pack[sum_n (P+R_n)]  packed row of each replicated row
 * Any output pointer may be NULL.  Returns DUALKV_OK or DUALKV_ERR_INVALID.
 */
int dualkv_build_index(int P, int N, const int32_t* R_offsets, int32_t* seg_id, int32_t* pos_id,
                       int32_t* cu_seqlens_rep, int32_t* rep2pack);

/*
 * Per-token tensors between the replicated and the packed layout (paper
 * abstract: with the prompt stored once, the layers around attention also run
 * on P+NR rows; these calls move their activations and gradients between the
 * two layouts).
 *
 * Replicated layout: sequence n is the P prompt rows followed by its R_n
 * response rows; the sequences lie end to end (sequence n starts at row
 * n*P + R_offsets[n]; T_rep = N*P + R_offsets[N] rows).  Packed layout as
 * above (T rows).  A row is row_elems bf16 values (row_elems >= 8, a multiple
 * of 8, i.e. whole 16-byte vectors), rows contiguous, both buffers device
 * memory, 16-byte aligned, owned by the caller, and not overlapping.
 *
 *   dualkv_pack    x_rep[T_rep, row] -> x_packed[T, row]: a prompt row is
 *                  copied from replica 0, a response row from its sequence.
 *   dualkv_unpack  x_packed[T, row] -> x_rep[T_rep, row]: every replica gets
 *                  a copy of the prompt rows (the inverse of pack on tensors
 *                  whose replicas agree).
 *   dualkv_fold    g_rep[T_rep, row] -> g_packed[T, row]: the adjoint of
 *                  unpack, i.e. the gradient of the packed rows.  A prompt row
 *                  is the sum of its N replica rows, accumulated in fp32 in
 *                  replica order n = 0..N-1 and rounded once to bf16; a
 *                  response row is copied.
 *
 * Copies are bit-exact.  Asynchronous on `stream`.  Returns DUALKV_OK,
 * DUALKV_ERR_INVALID (bad layout, row_elems, null or overlapping buffers),
 * DUALKV_ERR_ALIGN or DUALKV_ERR_CUDA.  The first call for a layout uploads
 * R_offsets into a small cached device array (freed by dualkv_release()).
 */
int dualkv_pack(const void* x_rep, void* x_packed, int P, int N, const int32_t* R_offsets, int row_elems,
                void* stream);
int dualkv_unpack(const void* x_packed, void* x_rep, int P, int N, const int32_t* R_offsets, int row_elems,
                  void* stream);
int dualkv_fold(const void* g_rep, void* g_packed, int P, int N, const int32_t* R_offsets, int row_elems,
                void* stream);

/*
 * Token-reduction factor rho = sum_n (P + R_n) / (P + sum_n R_n) (paper
 * abstract: rho = N(P+R)/(P+NR) for equal lengths).  Host only; -1 on invalid input.
 */
double dualkv_rho(int P, int N, const int32_t* R_offsets);

/*
 * Attended (query, key) pairs of one head in the packed layout, each packed
 * query row counted once.  Host only; -1 on invalid input.
 */
int64_t dualkv_pairs(int P, int N, const int32_t* R_offsets, int window);

/*
 * Synchronises `stream`, reads and clears the status word of the current
 * device, and returns DUALKV_OK or DUALKV_ERR_DEVICE (a kernel timed out in
 * a bounded wait or found an index out of range) or DUALKV_ERR_CUDA.
 */
int dualkv_check_status(void* stream);

/* Static, NUL-terminated description of a return code. */
const char* dualkv_error_string(int code);

/*
 * Per-kernel timing for benchmarks.  While enabled (on != 0), every kernel the
 * library launches is bracketed by CUDA events recorded on the caller's
 * stream.  dualkv_profile_read() waits for the recorded events, adds each
 * kernel's elapsed milliseconds and launch count into ms[kind] and
 * launches[kind] for kind = DUALKV_KERNEL_* (arrays of DUALKV_KERNEL_KINDS
 * entries, host memory), and forgets the records.  Returns DUALKV_OK or
 * DUALKV_ERR_CUDA.
 */
#define DUALKV_KERNEL_FWD 0
#define DUALKV_KERNEL_PREP 1
#define DUALKV_KERNEL_DKV 2
#define DUALKV_KERNEL_REDUCE 3
#define DUALKV_KERNEL_DQ 4
#define DUALKV_KERNEL_PACK 5 /* dualkv_pack, dualkv_unpack and dualkv_fold */
#define DUALKV_KERNEL_KINDS 6
int dualkv_profile_enable(int on);
int dualkv_profile_read(double* ms, int64_t* launches);

/*
 * Backward pass that allocates no device memory.  The paper has no counterpart
 * to this entry point: it is here for callers that cannot call cudaMalloc on
 * the call path -- for example a runtime that hands all device memory to its
 * own pool at start-up and fails any later allocation, or a host binding that
 * owns no device allocator and holds only the buffers it was given.
 *
 * Same arguments and results as dualkv_bwd for head dimensions 64 and 128,
 * without the workspace; D = 512 returns DUALKV_ERR_UNSUPPORTED (its bf16 P and
 * dS blocks need gigabytes, far beyond a fixed array).  Delta, the log2-scaled
 * LSE, the split dK/dV partials, the work lists and a status word live in one
 * fixed array of DUALKV_NOALLOC_SCRATCH_BYTES (32 MiB) in the library's device
 * memory, which every GPU that loads the library holds until the process
 * exits.  The first call on a device looks up that array's device address
 * (set-up), so make that first call before any stream capture on the device.
 * A layout whose scratch would exceed the maximum is rejected with
 * DUALKV_ERR_WORKSPACE before anything is launched.  Every call shares the
 * array and leaves its contents behind; the status word is cleared at the
 * start of each call and everything else is fully written before it is read.
 * Calls that overlap on the GPU (different streams, or host threads) race on
 * the array and corrupt each other's results.  The call is synchronous: it
 * returns after its kernels have finished on `stream` (also when it fails
 * after queueing work), with DUALKV_ERR_DEVICE if one of them reported a
 * timed-out wait or an index out of range.
 */
#define DUALKV_NOALLOC_SCRATCH_BYTES 33554432
int dualkv_bwd_noalloc(const void* q, const void* k, const void* v, const void* out, const float* lse,
                       const void* dout, int P, int N, const int32_t* R_offsets, int Hq, int Hkv, int D, float scale,
                       int window, void* dq, void* dk, void* dv, void* stream);

/*
 * Self-test of the kernels' failure path (no counterpart in the paper; it
 * exists so that timeout handling can be tested without faulting a GPU).
 * Launches one CTA of 64 threads that wait, with the same bounded mbarrier
 * wait every kernel uses but a limit of limit_ns nanoseconds (1 ms .. 10 s),
 * on a barrier that nothing completes.  The wait gives up, records a timeout
 * in the status word and the kernel returns; dualkv_check_status() then
 * reports DUALKV_ERR_DEVICE and the context stays usable.  Returns
 * DUALKV_ERR_INVALID for a limit out of range, DUALKV_ERR_CUDA if the launch
 * fails, else DUALKV_OK.
 */
int dualkv_selftest_timeout(uint64_t limit_ns, void* stream);

/*
 * Self-test of the production kernels' failure paths (no counterpart in the
 * paper; it exists so that timeout and range handling can be tested without
 * faulting a GPU).  Runs one kernel on a tiny internal layout (zero inputs,
 * P = 128, two responses of 128, one head, D = 128) with every bounded wait
 * limited to limit_ns nanoseconds (1 ms .. 10 s):
 *   which = 0  the forward kernel; the first K/V tile of every CTA is never
 *              loaded, so the wait for it runs out;
 *   which = 1  the dK/dV kernel; the first query block of its first CTA gets
 *              one barrier arrival too few, so the waits for it run out;
 *   which = 2  the forward kernel given a work list whose first entry lies past
 *              the last row; the kernel's range check skips it;
 *   which = 3  the backward preprocess and dQ kernel given a dQ work list whose
 *              first entry lies past the last row; the preprocess, which checks
 *              that list before the dQ kernel reads it, empties the entry;
 *   which = 4  the head-dimension-512 P / dS pass (same layout with D = 512);
 *              the first K/V tile of every CTA is never loaded.
 * The failure is recorded in the status word; a kernel whose wait ran out
 * drains its copies and tensor-core operations, frees its tensor memory and
 * returns;
 * dualkv_check_status() then reports DUALKV_ERR_DEVICE and the context stays
 * usable.  The call allocates and frees its own small buffers and returns
 * after the kernel has finished on `stream`: DUALKV_OK, DUALKV_ERR_INVALID
 * (which or limit out of range) or DUALKV_ERR_CUDA.
 */
int dualkv_selftest_kernel(int which, uint64_t limit_ns, void* stream);

/*
 * The library keeps the work lists of the 32 most recently used layouts
 * (per layout, window, head dimension and kv-head range) in device memory and
 * evicts the least recently used one beyond that; the memory of evicted plans
 * is pooled and reused, so a training loop whose offsets change every
 * micro-batch neither grows device memory nor allocates on every call.  Plans
 * are uploaded with one asynchronous copy on the caller's stream.  Reports the
 * number of resident plans and the device bytes the cache holds (resident and
 * pooled); either pointer may be NULL.  Returns DUALKV_OK.
 */
int dualkv_plan_cache_info(int* n_plans, int64_t* device_bytes);

/* Frees the plan cache, status words and timing events.  Not safe while launches are pending. */
void dualkv_release(void);

#ifdef __cplusplus
}
#endif

#endif /* DUALKV_H_ */
