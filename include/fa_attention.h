/*
 * fa_attention.h -- C ABI of the exact-attention library for GB300 (sm_103a).
 *
 * What it computes
 * ----------------
 * Exact scaled-dot-product attention, O = softmax(Q K^T * scale + mask) V, the
 * formula of the page "FlashAttention — فلاش أتنشن", section "The problem of
 * standard attention" (there the scale is 1/sqrt(d_k)).  The forward pass is
 * done the way the same page describes in its sections "Tiling and block
 * processing", "Online softmax" and "Fusion of the operations into one CUDA
 * kernel": Q, K, V tiles are staged on chip, each query row keeps a running
 * maximum and a running sum of exponentials, masking is fused, and only the
 * final output (plus one float per row) is written -- no N x N matrix ever
 * reaches device memory.  The parallel split over (batch, head, query block) and
 * over key blocks in the backward pass follows the page "FlashAttention-2 —
 * فلاش أتنشن-2", section "Technical architecture", item 2 ("parallelism").
 *
 * Layout and types (every call)
 * -----------------------------
 *  - Q, K, V, O, dO, dQ, dK, dV: [B, H, N, d] contiguous, d innermost, element
 *    type fp16 or bf16 (`fa_dtype`), all in the same type.
 *  - lse (the per-row logsumexp L): [B, H, N] fp32, natural log of the sum of
 *    exp(scaled, masked scores) of that row.
 *  - d in {64, 128, 256}; N >= 0 (any value: ragged tails are masked); B, H >= 0;
 *    B*H*N == 0 is an empty problem and returns FA_OK without launching work.
 *  - causal != 0 hides key j from query i when j > i (square, top-left
 *    aligned); masked scores are -inf before the softmax.
 *  - Every pointer is a device pointer, 16-byte aligned.
 *
 * Ownership: the caller owns every buffer.  The library allocates no device
 * memory; the backward pass takes a caller-provided workspace whose size
 * `fa_bwd_workspace_size` reports (linear in N).  TMA descriptors are encoded
 * on the host for every call and passed by value to the kernels.
 *
 * Errors: argument errors are detected on the host, return at once and launch
 * nothing.  A failed launch returns FA_ERR_CUDA.  All calls are asynchronous on
 * `stream`; a kernel that gave up on a bounded device-side wait records it in a
 * device error word, which `fa_check_device_status` reports (it synchronizes
 * the stream).  No kernel traps.
 *
 * Threads: calls may come from several host threads on different streams; the
 * device-buffer entry points share no host state between calls but the device
 * error record (one per device: a status check reports, and clears, what any
 * call on that device recorded) and the measurement hook (one per process, not
 * thread-safe).  The host-buffer entry points serialize themselves.
 */
#ifndef FA_ATTENTION_H_
#define FA_ATTENTION_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,    /* null pointer, negative size, scale not finite and > 0, bad enum */
  FA_ERR_UNSUPPORTED = 2,    /* head dim outside {64,128,256}, sizes over the limits, no sm_103a device */
  FA_ERR_MISALIGNED = 3,     /* a pointer is not 16-byte aligned */
  FA_ERR_WORKSPACE = 4,      /* backward workspace missing or smaller than fa_bwd_workspace_size */
  FA_ERR_CUDA = 5,           /* a CUDA runtime/driver call or a launch failed */
  FA_ERR_DEVICE_TIMEOUT = 6, /* a kernel gave up on a bounded wait (see fa_check_device_status) */
  FA_ERR_DEVICE_CHECK = 7    /* debug builds: a device-side bounds, alignment or phase check failed */
} fa_status;

typedef enum { FA_FP16 = 0, FA_BF16 = 1 } fa_dtype;

/* The stream type of the CUDA runtime, spelled without including its headers. */
typedef struct CUstream_st* fa_stream_t;

/*
 * Forward pass: O and L from Q, K, V.
 *   q, k, v : inputs [B,H,N,d] (read only)
 *   o       : output [B,H,N,d], same type as the inputs
 *   lse     : output [B,H,N] fp32, L_i = ln sum_j exp(scale * q_i.k_j) over visible j
 *   scale   : softmax scale, finite and > 0, normally 1/sqrt(d)
 * Computation per page "FlashAttention — فلاش أتنشن", sections "Online softmax"
 * and "Fusion of the operations into one CUDA kernel".
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, fa_dtype dtype, fa_stream_t stream);

/*
 * Forward pass with grouped-query attention and unequal lengths.
 *   q, o : [B, H, N_q, d];  k, v : [B, H_kv, N_k, d];  lse : [B, H, N_q] fp32.
 *   H_kv >= 1 divides H; query head h reads key/value head h / (H / H_kv)
 *   (H_kv = 1 is multi-query attention; MQA support is named on the page
 *   "FlashAttention — فلاش أتنشن", section "FlashAttention-2").
 *   Under causal != 0 the mask is aligned at the bottom right: key j is visible
 *   to query i iff j <= i + (N_k - N_q), so the last query row sees every key.
 *   A query row that sees no key (only when N_q > N_k) gets O = 0, L = -inf.
 *   N_k must be >= 1 when B*H*N_q > 0 (FA_ERR_UNSUPPORTED otherwise).
 * fa_fwd(..., N, ...) is fa_fwd_ex with H_kv = H and N_q = N_k = N.
 */
fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv,
                    int N_q, int N_k, int d, float scale, int causal, fa_dtype dtype, fa_stream_t stream);

/*
 * Bytes of device workspace `fa_bwd` needs: two fp32 row vectors (L log2 e and
 * D = rowsum(dO o O)) whose rows are padded per head to a multiple of 128, each
 * part 256-byte aligned -- 8 bytes per (padded) query row at every head
 * dimension, linear in N.  No kernel keeps a gradient accumulator in device
 * memory.  Returns 0 for invalid or empty sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass: dQ, dK, dV of the loss sum(O o dO), recomputing S and P from
 * Q, K and the forward pass's L (no N x N matrix is stored).  The pages state
 * that the method serves training (page "FlashAttention-2 — فلاش أتنشن-2",
 * section "Performance and efficiency"); the gradients are the chain-rule
 * derivatives of the attention formula:
 *   D_i = sum_c dO_ic O_ic,  P = exp(scale*S - L),  dV = P^T dO,
 *   dS = P o (dO V^T - D),   dQ = scale dS K,       dK = scale dS^T Q.
 *   q,k,v,o,dout : inputs [B,H,N,d] (o is the forward output)
 *   lse          : input [B,H,N] fp32 from fa_fwd
 *   dq,dk,dv     : outputs [B,H,N,d], same type as the inputs
 *   workspace    : device buffer of at least fa_bwd_workspace_size(B,H,N,d)
 *                  bytes, 256-byte aligned; contents need not be initialised
 *                  and are overwritten.
 * Launches, in order on `stream`: the pre-pass (D and L log2 e), then for d =
 * 64 and 128 a key-block-parallel dK/dV kernel and a query-block-parallel dQ
 * kernel, for d = 256 one kernel whose CTAs compute dK (per key block), dV (per
 * key block) or dQ (per query block).  No kernel uses atomics.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                 float scale, int causal, fa_dtype dtype, fa_stream_t stream);

/*
 * Backward pass with grouped-query attention and unequal lengths; shapes as in
 * fa_fwd_ex (dq like q, dk and dv like k).  The gradient of a shared key/value
 * head is the sum over the query heads of its group (computed inside one CTA
 * per key block, without atomics on dK/dV).  The workspace is
 * fa_bwd_workspace_size(B, H, N_q, d) bytes.  With B*H*N_q == 0 no query
 * row exists, so dk and dv are set to zero (cudaMemsetAsync on `stream`).
 * The result is deterministic at every head dimension: one CTA sums each key
 * row of dK, dV and each query row of dQ in a fixed order, so repeated calls
 * give bitwise equal gradients.
 * fa_bwd(..., N, ...) is fa_bwd_ex with H_kv = H and N_q = N_k = N.
 */
fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                    void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int H_kv,
                    int N_q, int N_k, int d, float scale, int causal, fa_dtype dtype, fa_stream_t stream);

/*
 * fa_bwd without a caller-provided workspace, for callers that cannot allocate
 * device memory: code that runs inside another runtime's allocator or memory
 * pool callbacks, hosts that reserved the whole device memory up front for
 * their own pool, or real-time loops where cudaMalloc's implicit device
 * synchronization is not acceptable.  (The attention method itself has no
 * counterpart to this entry point; it only changes where the scratch lives.)
 *
 * Arguments, layout, results and errors are those of fa_bwd, minus the
 * workspace pair.  The scratch (the fp32 row vectors L log2 e and D:
 * fa_bwd_workspace_size(B,H,N,d) bytes) lives in one fixed 32 MiB array in the
 * library's device memory, allocated when the library's device code is loaded
 * and held by every GPU that loads it until the process exits.  Calls whose
 * scratch would exceed 32 MiB (33554432 bytes) return FA_ERR_WORKSPACE and
 * launch nothing: B*H*Npad <= 4,194,304, Npad being N rounded up to a multiple
 * of 128 (with B*H = 1, N up to 4,194,304 rows).
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it, keyed on the device's current CUDA
 * context; make that first call before any stream capture.  After
 * cudaDeviceReset (a new primary context) the next call looks the address up
 * again, as it does the library's device error record.  No call allocates: no
 * cudaMalloc, cudaFree or allocating library routine.  Every call overwrites the whole scratch region
 * it uses before reading it (the D pre-pass writes every row vector, padding
 * rows included), so stale contents from an earlier call never leak into a
 * result.  All calls share the one array: two calls whose kernels overlap on
 * the GPU (different streams, no ordering between them) race on it and give
 * wrong gradients; order them on one stream or with events.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                         int causal, fa_dtype dtype, fa_stream_t stream);

/*
 * Synchronizes `stream`, then reads and clears the device error word of the
 * current device.  FA_OK if no kernel gave up on a wait (and, in a debug build,
 * no device-side check failed) since the last check; otherwise the kind of the
 * first failure: FA_ERR_DEVICE_TIMEOUT or FA_ERR_DEVICE_CHECK.  FA_ERR_CUDA if
 * the synchronization failed.
 */
fa_status fa_check_device_status(fa_stream_t stream);

/*
 * Debug builds (the library compiled with -DFA_DEBUG, `build(debug=True)` of the
 * Python build script: libfa_attention_debug.so) check on the device, before
 * every TMA copy, tensor-memory access and tensor-core product and at every
 * CTA's exit:
 *   - the box origin of each TMA copy: column a multiple of 64 inside the head
 *     dimension, row inside the tensor's rows rounded up to 256, plane inside
 *     the tensor's planes (kinds 1, 2, 3);
 *   - each tensor-memory address and the columns its access spans against the
 *     CTA's 512 allocated columns and 128 lanes (kinds 4, 5);
 *   - each bulk copy of L log2 e and D rows against the workspace's rows (kind 6);
 *   - at CTA exit, that every mbarrier completed the number of phases the
 *     kernel's protocol says (kind 7; only when no wait gave up).
 * A failed check records the error bit 64, the code 0x100 | kind, the CTA and
 * the offending value in the device error record, clamps the access to a safe
 * one and lets the kernel run on (it never traps); fa_check_device_status then
 * returns FA_ERR_DEVICE_CHECK and fa_last_device_error_detail gives the record.
 * This is the stand-in for a memory checker where none can be run.
 *
 * fa_selftest_device_check(kind, stream) makes check `kind` (1..7) fail once on
 * purpose: one thread hands the check a value that breaks its rule and discards
 * the clamped result, so nothing is copied or accessed.  Returns FA_OK
 * (asynchronous on `stream`), FA_ERR_INVALID_ARG for another kind,
 * FA_ERR_UNSUPPORTED in a release build (the checks are compiled out) or on a
 * device other than sm_103, FA_ERR_CUDA if the launch failed.
 */
fa_status fa_selftest_device_check(int kind, fa_stream_t stream);

/*
 * Host-buffer entry points (a runtime convenience; the attention method has no
 * counterpart): the forward pass, or the forward and backward pass, of a
 * problem whose inputs and outputs live in host memory.  The B*H heads are split
 * into `chunks` chunks of consecutive heads (equal chunks, at most 64; with
 * chunks <= 0, middle chunks of about B*H / 4 heads between a first and a last
 * chunk of half that size, which shortens the pipeline's fill and drain);
 * chunk c's host-to-device copies, kernels and device-to-host copies run on
 * three library-owned streams, so copies of one chunk overlap the kernels of
 * another.  Every chunk is an independent problem (B = 1, H = heads of the
 * chunk) computed by fa_fwd_ex / fa_bwd_ex, so the results equal those of the
 * device entry points on the whole problem.
 *   q,k,v,dout      : host inputs [B,H,N,d] (16-bit); dout only for fa_fwd_bwd_host
 *   o,lse,dq,dk,dv  : host outputs, layouts as in fa_fwd / fa_bwd
 *   dev_scratch     : device buffer of at least fa_host_scratch_size(B,H,N,d,bwd)
 *                     bytes, 256-byte aligned, owned by the caller; it holds the
 *                     device copies of every tensor and the backward workspace
 * Multi-head attention with N_q = N_k = N only.  Host buffers should be pinned
 * (page-locked); with pageable memory the copies are correct but do not overlap.
 * The call is asynchronous: all work starts after the work already queued on
 * `stream`, and `stream` waits for its completion, so the outputs are valid once
 * `stream` has been synchronized.  Errors: as fa_fwd / fa_bwd, plus
 * FA_ERR_WORKSPACE for a missing or small scratch; if a chunk fails part-way the
 * call still makes `stream` wait for the copies already issued.  Calls from
 * several host threads are serialized by the library.
 */
size_t fa_host_scratch_size(int B, int H, int N, int d, int with_backward);

/*
 * The chunk plan fa_fwd_host / fa_fwd_bwd_host use for these sizes and `chunks`
 * (a host query; it touches no device): writes the heads of each chunk, in
 * order, to plan[0 .. n-1] when plan is non-null and capacity >= n, and returns
 * n (at most 64).  Every chunk but the last starts at a head h whose first row
 * h*N keeps L 16-byte aligned.  Returns 0 for an empty problem and -1 for
 * negative sizes.
 */
int fa_host_chunk_plan(int B, int H, int N, int chunks, int* plan, int capacity);
fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, void* dev_scratch,
                      size_t scratch_bytes, int B, int H, int N, int d, float scale, int causal, fa_dtype dtype,
                      int chunks, fa_stream_t stream);
fa_status fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dout, void* o, float* lse,
                          void* dq, void* dk, void* dv, void* dev_scratch, size_t scratch_bytes, int B, int H, int N,
                          int d, float scale, int causal, fa_dtype dtype, int chunks, fa_stream_t stream);

/*
 * Heads per group of the CTA order the kernels use (a host query; it touches no
 * device when num_sms > 0).  The main kernels take heads in groups of G, the
 * heaviest blocks first inside a group, so the tiles that concurrently running
 * CTAs read stay in L2.  G is the smallest head count whose group gives each of
 * num_sms SMs at least as much work as the group's longest CTA (nblocks blocks
 * per head, each doing up to nblocks steps; under the causal mask the steps fall
 * to 1), raised until the group's tensors (bytes_per_head each) fill about 48 MB,
 * at most nheads, and then rounded up to a divisor of nheads within a factor of
 * two when there is one.  num_sms <= 0 uses the current device's SM count.
 * Returns -1 for nheads < 1 or nblocks < 0.
 */
int fa_cta_head_group(long long nheads, int nblocks, size_t bytes_per_head, int causal, int num_sms);

/*
 * Failure-detection self-test (a diagnostic; the attention method has no
 * counterpart): launches one thread that waits, through the same bounded wait
 * every kernel of this library uses, on an mbarrier that nothing arrives on, with
 * a limit of limit_us microseconds instead of the kernels' 4 s.  The wait gives
 * up, records code 32 (self-test) in the device error record and the kernel
 * returns; the next fa_check_device_status on `stream` returns
 * FA_ERR_DEVICE_TIMEOUT with that record and clears it, and the context stays
 * usable.  Returns FA_ERR_INVALID_ARG unless 0 < limit_us <= 1000000,
 * FA_ERR_UNSUPPORTED on a device other than sm_103, FA_ERR_CUDA if the launch
 * failed, FA_OK otherwise (asynchronous on `stream`).  Kernels of this library
 * that run between the self-test and that status check see the failure bit and
 * stop early, as after a real timeout.
 */
fa_status fa_selftest_wait_timeout(uint32_t limit_us, fa_stream_t stream);

/* Raw device error word of the last fa_check_device_status (0 = none). */
uint32_t fa_last_device_error_bits(void);

/*
 * The error record behind it: out4[0] the bits, out4[1] the code of the first
 * wait that gave up (1 TMA tile, 2 tensor-core commit, 4 elementwise output,
 * 8 ring slot, 16 warpgroup barrier, 32 self-test; 0x100 | kind for a failed
 * debug-build check), out4[2] that CTA's index,
 * out4[3] its
 * barrier's shared-memory address (for a check: the offending value).  After the first failure every other wait
 * of the grid gives up at once (bit 31), and kernels launched before the next
 * fa_check_device_status stop early: their results are not valid.
 */
void fa_last_device_error_detail(uint32_t* out4);

/*
 * Measurement hook.  fa_profile_begin(n) makes the library record a pair of CUDA
 * events (created and owned by the library) on the launching stream around each
 * of the next n main-kernel launches of fa_fwd / fa_bwd (and their _ex forms):
 * the fused forward kernel, and the backward kernels without the D pre-pass.
 * One fa_fwd call makes one launch; one fa_bwd call makes two for d = 64 and
 * 128 (the dK/dV kernel, then the dQ kernel) and one for d = 256.
 * fa_profile_end waits for those events, writes each launch's time in
 * milliseconds to out_ms[i] and its kind to out_kind[i] (0 forward kernel, 1
 * dK/dV kernel, 2 dQ kernel, 3 the single backward launch of d = 256), in
 * launch order, stops recording and returns the number of entries written (at
 * most max_out), or -1 if the events could not be read.  Returns of
 * fa_profile_begin: FA_OK, FA_ERR_INVALID_ARG (n < 0 or n > 65536), FA_ERR_CUDA
 * (event creation failed).  Not thread-safe: one recording per process.
 */
fa_status fa_profile_begin(int n);
int fa_profile_end(float* out_ms, int* out_kind, int max_out);

/* Human-readable name of a status code (static storage). */
const char* fa_status_string(fa_status s);

/* Library version, (major << 16) | minor. */
uint32_t fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_ATTENTION_H_ */
