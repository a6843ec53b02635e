/*
 * aaren.h -- C ABI of libaaren, a B300 (sm_103a) CUDA library for the
 * numerically stable softmax-attention prefix scan.
 *
 * The operation.  For every head, given a query q in R^d, keys k_1..k_N and
 * values v_1..v_N in R^d, the scan produces every causal prefix output
 *
 *     s_i = q . k_i                       (unscaled; pre-scale q if wanted)
 *     o_t = sum_{i<=t} e^{s_i} v_i / sum_{i<=t} e^{s_i},      t = 1..N,
 *
 * i.e. attention's many-to-many RNN output computed with a parallel prefix
 * scan ("Attention as an RNN" review, "Proposed method": attention as a
 * many-to-one RNN, its many-to-many output via the parallel prefix scan, and
 * a constant-size state updated one token at a time), which is also the
 * streaming running sum of the "Self-attention Does Not Need O(n^2) Memory"
 * review, section 2 "Algorithm" (sums of v_i e^{s_i} and e^{s_i}, divided
 * at the end), evaluated at every prefix.  The scan carries the state
 *
 *     (m, u, w) = (max_i s_i, sum_i e^{s_i - m} v_i, sum_i e^{s_i - m}),
 *
 * the max-subtraction reading of that review's section 3 "Numerical
 * Stability" (whose body the page lacks), combined with the associative
 * operator (m_a,u_a,w_a) (+) (m_b,u_b,w_b) = (M, e^{m_a-M}u_a + e^{m_b-M}u_b,
 * e^{m_a-M}w_a + e^{m_b-M}w_b), M = max(m_a, m_b), identity (-inf, 0, 0).
 * The output is o_t = u_t / w_t of the inclusive prefix state.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never frees or keeps them.  Tensors are dense and row-major with the
 *    last dimension fastest:  q [B,H,d];  K, V, O [B,H,N,d] (each head's
 *    tokens contiguous, in token order);  state m, w [B*H];  u [B*H, d].
 *  - q, K, V, O and u pointers must be 16-byte aligned; m, w 4-byte aligned.
 *  - dtype selects the element types: AAREN_F32 (q, K, V, O float32),
 *    AAREN_BF16 (q, K, V, O bfloat16), AAREN_BF16_F32OUT (q, K, V bfloat16,
 *    O float32).  Arithmetic is float32 throughout; bfloat16 inputs are
 *    widened exactly, bfloat16 outputs are rounded to nearest even.  The state
 *    (m, u, w) is always float32.
 *  - d must be 16, 32, 64 or 128 (else AAREN_ERR_UNSUPPORTED).
 *  - stream is a cudaStream_t (NULL = the legacy default stream).  Every call
 *    is asynchronous and ordered on that stream.  The return value covers
 *    argument checks and the launch; failures on the device (a wait that gave
 *    up) are reported by aaren_check().
 *  - Non-finite inputs are not checked; NaN and Inf propagate.
 */
#ifndef AAREN_H
#define AAREN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    AAREN_OK = 0,
    AAREN_ERR_INVALID = 1,          /* bad argument: null or misaligned pointer,
                                       negative or overflowing size, O aliasing
                                       K or V, partial state triple */
    AAREN_ERR_UNSUPPORTED = 2,      /* d or dtype not built */
    AAREN_ERR_CUDA = 3,             /* a CUDA runtime call failed */
    AAREN_ERR_LOOKBACK_TIMEOUT = 4, /* device: a cross-block carry wait gave up */
    AAREN_ERR_BOUNDS = 5,           /* device, checked build only: an index fell
                                       outside its buffer; the access was skipped */
    AAREN_ERR_LOAD_TIMEOUT = 6,     /* device: a bulk copy into shared memory, or
                                       a hand-off between the warps of a block,
                                       did not complete in time */
    AAREN_ERR_WORKSPACE = 7         /* caller workspace too small or misaligned */
} aaren_status_t;

typedef enum {
    AAREN_F32 = 0,          /* q, K, V, O float32                */
    AAREN_BF16 = 1,         /* q, K, V, O bfloat16               */
    AAREN_BF16_F32OUT = 2   /* q, K, V bfloat16, O float32       */
} aaren_dtype_t;

/*
 * aaren_scan_forward -- many-to-many output of every head, in one pass over
 * K and V ("Attention as an RNN" review, "Proposed method": the many-to-many
 * output by parallel prefix scan).
 *   q  [B,H,d]     query of each head (dtype's input type)
 *   K  [B,H,N,d]   keys          V [B,H,N,d] values   (input type)
 *   O  [B,H,N,d]   output o_t of every prefix, written (output type);
 *                  must not overlap K or V
 * N = 0 (or B*H = 0) is a no-op.  The cross-block carry needs a workspace of
 * aaren_scan_workspace_bytes(B,H,N,d) bytes, taken from the stream-ordered
 * allocator (cudaMallocAsync / cudaFreeAsync on `stream`) for this call.
 * Results are not bitwise reproducible from call to call: a chunk's carry
 * combines whichever predecessors it finds holding only their own aggregate,
 * so the grouping of the combining steps, and the last bits of O, depend on
 * timing.  Every grouping is within the same error bound.
 * A call launches two kernels on `stream`: one that zeroes the workspace's
 * ticket and chunk flags, then the scan, launched as its programmatic
 * dependent (its set-up overlaps the zeroing; it reads nothing before the
 * zeroing has completed).
 * Errors: AAREN_ERR_INVALID, AAREN_ERR_UNSUPPORTED, AAREN_ERR_CUDA.
 */
aaren_status_t aaren_scan_forward(const void *q, const void *K, const void *V,
                                  void *O, int64_t B, int64_t H, int64_t N,
                                  int64_t d, int32_t dtype, void *stream);

/*
 * aaren_scan_forward_ex -- aaren_scan_forward with an optional starting
 * state, an optional final state and an optional caller workspace.
 *   m_in [B*H], u_in [B*H,d], w_in [B*H]   state each head starts from (the
 *        constant-size RNN state: a stream saved by aaren_step or by an
 *        earlier scan continues here); all three NULL = the identity
 *        (-inf, 0, 0).  Read only.
 *   m_out, u_out, w_out  final state (m, u, w) of each head after token N,
 *        written; all three NULL = not written.  With N = 0 the final state
 *        is the starting state.
 *   workspace, workspace_bytes  device scratch for the cross-block carry, at
 *        least aaren_scan_workspace_bytes(B,H,N,d) bytes, 256-byte aligned;
 *        NULL = allocate as aaren_scan_forward does.  Its contents need no
 *        initialisation and are meaningless after the call.  Two calls in
 *        flight at once (on different streams) must not share a workspace.
 * A state triple must be all NULL or all non-NULL (else AAREN_ERR_INVALID).
 * Errors: as aaren_scan_forward, plus AAREN_ERR_WORKSPACE.
 */
aaren_status_t aaren_scan_forward_ex(const void *q, const void *K,
                                     const void *V, void *O, int64_t B,
                                     int64_t H, int64_t N, int64_t d,
                                     int32_t dtype, const float *m_in,
                                     const float *u_in, const float *w_in,
                                     float *m_out, float *u_out, float *w_out,
                                     void *workspace, size_t workspace_bytes,
                                     void *stream);

/* Bytes of workspace aaren_scan_forward_ex needs for this shape (0 when
 * N = 0 or B*H = 0; SIZE_MAX when d is unsupported or the shape overflows). */
size_t aaren_scan_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d);

/*
 * aaren_scan_forward_stats -- aaren_scan_forward that also saves, for every
 * prefix t, the pair (m_t, w_t) of its state: the running maximum of the
 * scores and the rescaled sum of their exponentials, so that
 * log sum_{i<=t} e^{s_i} = m_t + log w_t.  aaren_scan_backward needs them.
 *   stats [B,H,N,2] float32 (m_t, w_t), written; 8-byte aligned.
 * Other arguments, workspace and errors as aaren_scan_forward_ex (no start
 * or final state: a sequence that is differentiated starts empty).
 */
aaren_status_t aaren_scan_forward_stats(const void *q, const void *K,
                                        const void *V, void *O, float *stats,
                                        int64_t B, int64_t H, int64_t N,
                                        int64_t d, int32_t dtype,
                                        void *workspace, size_t workspace_bytes,
                                        void *stream);

/*
 * aaren_scan_backward -- gradients of the many-to-many output: given the
 * upstream gradient dO = dL/dO, computes dL/dq, dL/dK and dL/dV in one pass
 * over K, V, O and dO with O(1) memory per head beyond the inputs (the
 * memory-efficient-attention review reports its method for differentiation
 * as well as inference; the Aaren review calls the RNN form exact and
 * differentiable).  With p_{t,i} = e^{s_i} / sum_{j<=t} e^{s_j}:
 *     dL/dv_i = sum_{t>=i} p_{t,i} g_t,
 *     dL/ds_i = sum_{t>=i} p_{t,i} (g_t . v_i - g_t . o_t),
 *     dL/dq = sum_i dL/ds_i k_i,   dL/dk_i = dL/ds_i q,
 * computed as suffix sums from the last token back, with the forward's
 * per-prefix statistics keeping every weight <= 1.
 *   q [B,H,d], K, V [B,H,N,d]   inputs of the forward (input type)
 *   O, dO [B,H,N,d]   the forward's output and its gradient (output type)
 *   stats [B,H,N,2]   from aaren_scan_forward_stats of the same inputs
 *   dq [B*H,d], dK, dV [B,H,N,d]   gradients, float32, written; they must not
 *        overlap the inputs or each other
 *   workspace, workspace_bytes   at least aaren_backward_workspace_bytes
 *        bytes, 256-byte aligned, or NULL (stream-ordered allocation)
 * N = 0 writes dq = 0.  Errors: AAREN_ERR_INVALID, AAREN_ERR_UNSUPPORTED,
 * AAREN_ERR_CUDA, AAREN_ERR_WORKSPACE; device-side waits that give up are
 * reported by aaren_check().  dL/dq is summed with float32 atomics, so its
 * last bits may differ between runs; so may those of dK and dV, whose
 * cross-block carry combines whichever successors it finds holding only
 * their own aggregate (every grouping is within the same error bound).
 */
aaren_status_t aaren_scan_backward(const void *q, const void *K, const void *V,
                                   const void *O, const void *dO,
                                   const float *stats, float *dq, float *dK,
                                   float *dV, int64_t B, int64_t H, int64_t N,
                                   int64_t d, int32_t dtype, void *workspace,
                                   size_t workspace_bytes, void *stream);

/* Bytes of workspace aaren_scan_backward needs for this shape (0 when N = 0
 * or B*H = 0; SIZE_MAX when d is unsupported or the shape overflows). */
size_t aaren_backward_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d);

/*
 * aaren_scan_reduce -- the many-to-one output: for every head only the last
 * output o_N = sum_{i<=N} e^{s_i} v_i / sum_{i<=N} e^{s_i} and, optionally,
 * the final state (m, u, w); no per-token output is written, so K and V are
 * the only large traffic ("Attention as an RNN" review, "Proposed method":
 * attention as a many-to-one RNN; "Self-attention Does Not Need O(n^2)
 * Memory" review, section 2 "Algorithm": the single-query running sums).
 * Each head's tokens are reduced in independent parts that are combined at
 * the end (the state operator is associative and commutative), so nothing
 * waits on a neighbouring part.
 *   q  [B,H,d], K, V [B,H,N,d]   as for aaren_scan_forward (input type)
 *   o_last [B*H,d]   o_N of each head (output type), written; NULL = not
 *        computed.  Must not overlap K or V.
 *   m_in, u_in, w_in   optional starting state (all NULL = identity), read
 *   m_out, u_out, w_out   optional final state (all NULL = not written)
 *   workspace, workspace_bytes   device scratch of at least
 *        aaren_reduce_workspace_bytes(B,H,N,d) bytes, 256-byte aligned; NULL
 *        = taken from the stream-ordered allocator for this call.  Contents
 *        need no initialisation; calls in flight at once must not share it.
 * At least one of o_last and the final state must be requested.  N = 0:
 * the final state is the starting state, and o_last needs a starting state
 * (the empty prefix has no output).  The result does not depend on the
 * launch shape chosen for the device beyond float32 rounding (parts are
 * combined in token order).
 * Errors: AAREN_ERR_INVALID, AAREN_ERR_UNSUPPORTED, AAREN_ERR_CUDA,
 * AAREN_ERR_WORKSPACE.
 */
aaren_status_t aaren_scan_reduce(const void *q, const void *K, const void *V,
                                 void *o_last, int64_t B, int64_t H,
                                 int64_t N, int64_t d, int32_t dtype,
                                 const float *m_in, const float *u_in,
                                 const float *w_in, float *m_out,
                                 float *u_out, float *w_out, void *workspace,
                                 size_t workspace_bytes, void *stream);

/* Bytes of workspace aaren_scan_reduce needs for this shape (0 when
 * B*H = 0; SIZE_MAX when d is unsupported or the shape overflows). */
size_t aaren_reduce_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d);

/*
 * aaren_state_init -- set n states to the identity (m = -inf, u = 0, w = 0),
 * the state of an empty prefix, before the first aaren_step: the RNN of the
 * "Attention as an RNN" review ("Proposed method") starts from an empty
 * state and takes one token per update; in the running sums of the
 * "Self-attention Does Not Need O(n^2) Memory" review (section 2
 * "Algorithm": v* and s* start at zero) with the maximum of section 3
 * "Numerical Stability" subtracted, the empty prefix has no maximum yet,
 * hence m = -inf.
 *   m [n], u [n,d], w [n]   float32, written.
 * Errors: AAREN_ERR_INVALID, AAREN_ERR_UNSUPPORTED, AAREN_ERR_CUDA.
 */
aaren_status_t aaren_state_init(float *m, float *u, float *w, int64_t n,
                                int64_t d, void *stream);

/*
 * aaren_step -- one token for each of n independent streams: the constant
 * memory RNN update of the "Attention as an RNN" review ("Proposed method":
 * Aaren is updated with new tokens using constant memory):
 *     s = q . k_t;  M = max(m, s);  u = e^{m-M} u + e^{s-M} v_t;
 *     w = e^{m-M} w + e^{s-M};  m = M;  o_t = u / w.
 *   q   [n,d]  query of each stream (input type), read only
 *   m [n], u [n,d], w [n]  float32 state, read and updated in place
 *   k_t [n,d], v_t [n,d]   this step's key and value (input type)
 *   o_t [n,d]  this step's output (output type), written
 * n = 0 is a no-op.  The states must have been set by aaren_state_init, by
 * earlier steps, or by aaren_scan_forward_ex's final state.
 * Errors: AAREN_ERR_INVALID, AAREN_ERR_UNSUPPORTED, AAREN_ERR_CUDA.
 */
aaren_status_t aaren_step(const void *q, float *m, float *u, float *w,
                          const void *k_t, const void *v_t, void *o_t,
                          int64_t n, int64_t d, int32_t dtype, void *stream);

/*
 * aaren_linattn_forward -- causal cos-re-weighted linear attention of every
 * head (LG AI Research blog "[ICLR 2022] Part 1: Efficient Transformer",
 * section "cosFormer"): with Q' = ReLU(Q), K' = ReLU(K),
 *
 *     s_ij = (Q'_i . K'_j) cos(pi/2 * (i - j) / M)
 *     o_i  = sum_{j<=i} s_ij v_j / sum_{j<=i} s_ij      (0 where the sum is 0)
 *
 * computed as a prefix scan whose state is the section's key-first sums
 * split by the cosine sum formula: S^cos = sum_j cos(pi j/2M) K'_j^T v_j,
 * S^sin likewise with sin, z^cos = sum_j cos(pi j/2M) K'_j, z^sin likewise.
 * Positions j are 1-based and continue from pos0 (the position of the token
 * before the first one of this call), so a long sequence can be processed in
 * pieces: pass the previous call's final state and pos0 = tokens so far.
 *   Q, K, V [B,H,N,d]   bfloat16 queries (one per token), keys, values
 *   O       [B,H,N,d]   written: bfloat16 (AAREN_BF16) or float32
 *                        (AAREN_BF16_F32OUT); AAREN_F32 is UNSUPPORTED
 *   d       64 only (else AAREN_ERR_UNSUPPORTED)
 *   M       re-weighting length, finite and > 0 (cosFormer takes the
 *           sequence length; M >= pos0 + N - 1 keeps every weight >= 0)
 *   S_in, z_in    starting state, float32 [B,H,2,64,64] (index 0 = cos, 1 =
 *           sin; row = key coordinate, column = value coordinate) and
 *           [B,H,2,64]; both NULL = the zero state.  16- and 4-byte aligned.
 *   S_out, z_out  final state in the same layout, or both NULL.  May not
 *           alias S_in / z_in of other heads (the same head in place is fine).
 * Arithmetic: float32 accumulation on the tensor cores; every operand the
 * method rounds (the intra-chunk weights, the position-weighted keys, the
 * state) is carried as a bfloat16 pair hi + lo, so the result is float32
 * accurate.  N = 0 copies the starting state to the final state (or zeroes
 * it).  Errors: AAREN_ERR_INVALID for negative sizes, pos0 < 0, M not finite
 * and positive, null / misaligned pointers, one of a state pair missing, O
 * overlapping Q, K or V, N or B*H beyond 2^31 - 129; AAREN_ERR_CUDA when the
 * driver's tensor-map encoder is unavailable or a launch fails; device
 * waits that give up are reported by aaren_check().
 */
aaren_status_t aaren_linattn_forward(const void *Q, const void *K, const void *V, void *O,
                                     int64_t B, int64_t H, int64_t N, int64_t d, double M,
                                     int64_t pos0, int32_t dtype, const float *S_in,
                                     const float *z_in, float *S_out, float *z_out, void *stream);

/*
 * aaren_check -- synchronise `stream`, then report and clear the device
 * status word of the current device (one word per device, shared by every
 * stream and call: a failure on any stream shows up in the next check).
 * Returns AAREN_OK, AAREN_ERR_BOUNDS (checked build), AAREN_ERR_LOAD_TIMEOUT,
 * AAREN_ERR_LOOKBACK_TIMEOUT (in that order when several bits are set) or
 * AAREN_ERR_CUDA (a CUDA error from the synchronisation).
 */
aaren_status_t aaren_check(void *stream);

/* Static, NUL-terminated description of a status code. */
const char *aaren_status_string(int32_t status);

/* Version of this ABI (incremented on any incompatible change). */
int32_t aaren_abi_version(void);

/*
 * aaren_debug_set_fault -- testing hook for the bounded waits.  Every later
 * launch of the scan, the scan with statistics and the backward pass in this
 * process uses these values:
 *   never_publish_chunk  index (head * chunks per head + c, c the chunk of
 *        the head) of a chunk whose carry is never published, so the chunks
 *        that wait on it give up: its successors in the forward scans
 *        (chunks of aaren_scan_chunk_tokens tokens), its predecessors in the
 *        backward pass (chunks of aaren_backward_chunk_tokens tokens);
 *        -1 = none (the default).
 *   wait_limit_ns        how long a device wait lasts before it gives up
 *        (every kernel's waits; the persistent scan's waits inside a block
 *        get 16 times as long); <= 0 restores the default (1 s).
 * Returns AAREN_OK.  Not for production use.
 */
aaren_status_t aaren_debug_set_fault(int64_t never_publish_chunk,
                                     int64_t wait_limit_ns);

/*
 * aaren_debug_drop_arrival -- testing hook for the waits inside a block.
 * Every later launch in this process withholds one arrival on a barrier
 * between the warps of one block, so the warps waiting on it give up with
 * AAREN_ERR_LOAD_TIMEOUT (reported by aaren_check) and the block leaves
 * early, with no copy or tensor-core product still in flight:
 *   - the persistent scan kernel (bfloat16 inputs, and float32 at d = 64):
 *     the first compute warp of chunk `chunk` (numbered as for
 *     aaren_debug_set_fault) does not report its partial aggregate;
 *   - aaren_linattn_forward: in chunk `chunk` of the first thread block
 *     (chunk c of head 0 for c < ceil(N/128)), the weighted keys are never
 *     announced to the warp that issues the tensor-core products.
 * -1 = none (the default).  Returns AAREN_OK.  Not for production use.
 */
aaren_status_t aaren_debug_drop_arrival(int64_t chunk);

/*
 * aaren_checked_build -- 1 in the checked build of this library
 * (libaaren_checked.so, compiled with -DAAREN_CHECKED), 0 otherwise.  In the
 * checked build every kernel tests each extent it computes (rows of a global
 * tensor, a workspace slot, a bulk copy, a shared-memory stage) against its
 * buffer before the access; a violation skips the access and makes
 * aaren_check report AAREN_ERR_BOUNDS.  Results are otherwise identical.
 */
int32_t aaren_checked_build(void);

/*
 * aaren_debug_bounds_probe -- testing hook of the checked build: every later
 * aaren_step adds `offset` to the stream index its bounds check tests (never
 * to an address), so an offset >= n makes every stream's check fail, skip
 * its accesses and report AAREN_ERR_BOUNDS.  No effect in the regular build.
 * 0 = none (the default).  Returns AAREN_OK.  Not for production use.
 */
aaren_status_t aaren_debug_bounds_probe(int64_t offset);

/* Tokens per chunk (one thread block) the scan uses for this d and dtype
 * (0 if unsupported); the chunk index of aaren_debug_set_fault counts these. */
int64_t aaren_scan_chunk_tokens(int64_t d, int32_t dtype);

/* Tokens per chunk of aaren_scan_backward for this d and dtype (0 if
 * unsupported); aaren_debug_set_fault counts these in the backward pass. */
int64_t aaren_backward_chunk_tokens(int64_t d, int32_t dtype);

/*
 * aaren_scan_forward_noalloc -- aaren_scan_forward for callers that must not
 * allocate device memory.  The pages have no counterpart: this is a
 * deployment variant of the same scan.
 *
 * Who needs it: code whose GPU memory is owned by another allocator (a host
 * framework or plugin host that reserves the device and forbids outside
 * cudaMalloc), and latency-critical loops that cannot risk an allocator call,
 * which may block or fail when memory is full or fragmented.  Such callers
 * pass inputs and outputs exactly as for aaren_scan_forward (same arguments,
 * layouts and errors); the scan's cross-block carry workspace then lives in
 * a fixed array of AAREN_NOALLOC_SCRATCH_BYTES inside this library, which
 * every GPU that loads the library keeps until the process exits.
 *
 * Limits and behaviour:
 *  - A problem whose workspace, aaren_scan_workspace_bytes(B,H,N,d), exceeds
 *    AAREN_NOALLOC_SCRATCH_BYTES is rejected with AAREN_ERR_WORKSPACE before
 *    any pointer is read or any CUDA call is made (with d = 128 that is one
 *    to two million tokens over all heads, depending on the dtype's chunk
 *    size; smaller d allow more).  Unsupported d or dtype and negative sizes
 *    are rejected first, as by aaren_scan_forward.
 *  - No cudaMalloc, cudaFree or other allocating call is made.  The part of
 *    the array that must start at zero is cleared on `stream` by every call.
 *  - When the array takes its memory: with CUDA's lazy module loading (the
 *    default) the library's device code, this array included, is loaded on
 *    a device the first time any entry point of this library launches a
 *    kernel or looks up a device symbol there; with eager loading
 *    (CUDA_MODULE_LOADING=EAGER) when the library's module is loaded on that
 *    device's context.  Either way the 16 MiB stay reserved until the
 *    process exits.
 *  - The first call of this entry point on a device looks up the array's
 *    device address and keeps it for the rest of the process (once per
 *    device).  Make that first call before any stream capture.
 *  - Devices with ordinals 0..63 only (AAREN_ERR_CUDA beyond).
 *  - Do not call it on a device after cudaDeviceReset of that device in the
 *    same process: the reset unloads the module, and the kept address would
 *    name memory that no longer holds the array.
 *  - All calls on a device share the one array, which keeps the last call's
 *    contents: calls whose executions overlap on the GPU (different streams
 *    without ordering between them) race and corrupt each other's results.
 *    Order them on one stream, or use aaren_scan_forward_ex with separate
 *    workspaces.
 */
#define AAREN_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

aaren_status_t aaren_scan_forward_noalloc(const void *q, const void *K,
                                          const void *V, void *O, int64_t B,
                                          int64_t H, int64_t N, int64_t d,
                                          int32_t dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* AAREN_H */
