// scan_kernel.cuh -- fused score + chunked prefix scan with a decoupled
// look-back carry: the many-to-many softmax-attention output in one pass over
// K and V.
//
// The method ("Attention as an RNN" review, "Proposed method"): every prefix
// output o_t = sum_{i<=t} e^{s_i} v_i / sum_{i<=t} e^{s_i}, s_i = q . k_i, is
// the inclusive prefix of the associative operator on (m, u, w) (running
// max, rescaled sum of e^s v, rescaled sum of e^s), computed by a parallel
// prefix scan.  The running sums are those of the "Self-attention Does Not
// Need O(n^2) Memory" review, section 2 "Algorithm", kept stable by
// subtracting the running maximum (its section 3, "Numerical Stability").
//
// Work decomposition (one thread block = one chunk of C tokens of one head):
//   1. take a ticket (chunks are processed in ticket order, so every
//      predecessor of a chunk already runs), bulk-copy the chunk's K and V
//      rows (contiguous) into shared memory with one TMA copy each;
//   2. scores: lane t of a warp computes s for token t of its 32-token group
//      (a full dot product over d, reading K with a per-lane rotation so the
//      32 rows hit distinct shared-memory banks);
//   3. each warp reduces its tokens to an aggregate (m, u, w);
//   4. warp 0 combines the warp aggregates into the chunk aggregate,
//      publishes it, walks back over predecessor chunks until it meets an
//      inclusive prefix (decoupled look-back), publishes this chunk's
//      inclusive prefix, and derives each warp's incoming carry;
//   5. each warp rescans its tokens from its carry: the scalar parts
//      (running max, the rescale factor alpha_t and weight beta_t, and w_t)
//      by warp shuffles across tokens, then the d-wide recurrence
//      u_t = alpha_t u_{t-1} + beta_t v_t per lane over the lane's dims,
//      writing o_t = u_t / w_t.
// V stays in shared memory between steps 3 and 5, so HBM sees K and V once
// and O once.  Every wait is bounded: a wait that gives up sets a bit of the
// device status word, poisons this chunk's flag so successors stop waiting,
// and the block returns.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace aaren {

// Flags of a chunk in the look-back workspace (monotone except POISON).
enum : unsigned { FLAG_NONE = 0, FLAG_AGG = 1, FLAG_INC = 2, FLAG_POISON = 3 };

// Waits poll at least this many times before they may give up, so a context
// switch that stalls the whole kernel cannot by itself end a wait.
constexpr unsigned kMinWaitPolls = 256;

struct ScanParams {
    const void *q;
    const void *K;
    const void *V;
    void *O;
    const float *m_in;   // optional starting state per head (all or none)
    const float *u_in;
    const float *w_in;
    float *m_out;        // optional final state per head (all or none)
    float *u_out;
    float *w_out;
    unsigned *ticket;    // workspace: ticket counter (zeroed before launch)
    unsigned *flags;     // workspace: one flag per chunk (zeroed before launch)
    float *states;       // workspace: per chunk [aggregate | inclusive] states
    float2 *stats;       // optional [heads, N]: (m_t, w_t) of every prefix, for a backward pass
    unsigned *status;    // device status word
    int64_t N;
    int64_t heads;           // B * H
    int64_t chunks_per_head;
    int64_t fault_chunk;     // testing: chunk that never publishes (-1 = none)
    int64_t drop_chunk;      // testing: chunk whose compute warp 0 never reports its
                             // aggregate to its group (persistent kernel; -1 = none)
    int64_t wait_limit_ns;
};

// Zeroes the first n16 16-byte words of a scan workspace (the ticket and
// the chunk flags).  The scan after it is launched as its programmatic
// dependent: every block of this kernel lets that launch begin at once, so
// the scan's blocks are placed and set up while the zeroing runs, and the
// scan waits for this kernel's completion (griddepcontrol.wait) before its
// first access to global memory.  This kernel itself is launched in plain
// stream order, after everything before it (an earlier scan on the same
// workspace included) has completed.
__global__ void __launch_bounds__(256) k_zero_ws(uint4 *ws, int64_t n16)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += int64_t(gridDim.x) * blockDim.x)
        ws[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Layout of one state in the workspace and in shared memory:
// [m, w, unused, unused, u_0 .. u_{d-1}] (u 16-byte aligned).
template <int D>
struct StateLayout {
    static constexpr int SS = D + 4;
};

template <int D, typename Tin, int WARPS, int GROUPS>
struct ScanTile {
    static constexpr int C = WARPS * GROUPS * 32;   // tokens per chunk
    static constexpr int SS = StateLayout<D>::SS;
    static constexpr size_t kv_bytes = size_t(C) * D * sizeof(Tin);
    static constexpr size_t q_off = 2 * kv_bytes;
    static constexpr size_t wst_off = q_off + D * sizeof(float);
    static constexpr size_t cst_off = wst_off + size_t(WARPS) * SS * sizeof(float);
    static constexpr size_t coef_off = cst_off + size_t(WARPS) * SS * sizeof(float);
    static constexpr size_t bar_off = coef_off + size_t(WARPS) * 32 * sizeof(float4);
    static constexpr size_t smem_bytes = bar_off + 32;
    static_assert(kv_bytes % 16 == 0 && q_off % 16 == 0 && wst_off % 16 == 0 &&
                      cst_off % 16 == 0 && coef_off % 16 == 0 && bar_off % 8 == 0,
                  "shared-memory regions must stay 16-byte aligned");
};

// Where element j of q lives in shared memory.  The dot product reads q in
// 16-byte pieces matching one 16-byte piece of a key row: for float keys
// piece c holds q[4c..4c+3] (natural order); for bfloat16 keys piece c spans
// q[8c..8c+7], stored as two float4 arrays (q[8c..8c+3] in the first half,
// q[8c+4..8c+7] in the second) so both reads are conflict-free.
template <int D, typename Tin>
__device__ __forceinline__ int q_slot(int j)
{
    if constexpr (sizeof(Tin) == 4) {
        return j;
    } else {
        const int c = j >> 3, e = j & 7;
        return (e < 4) ? c * 4 + e : D / 2 + c * 4 + (e - 4);
    }
}

// Compensated dot-product step (Ogita, Rump & Oishi, "Accurate Sum and Dot
// Product", SIAM J. Sci. Comput. 2005, algorithm Dot2): TwoProduct by FMA and
// TwoSum, errors accumulated in c.  Used for float32 keys, whose scores can be
// large (hundreds) so that plain float32 accumulation would perturb the
// softmax weights.
__device__ __forceinline__ void dot2_step(float &p, float &c, float a, float b)
{
    const float h = __fmul_rn(a, b);
    const float r = __fmaf_rn(a, b, -h);              // a*b = h + r exactly
    const float s = __fadd_rn(p, h);
    const float z = __fsub_rn(s, p);
    const float e = __fadd_rn(__fsub_rn(p, __fsub_rn(s, z)), __fsub_rn(h, z));   // p+h = s+e
    p = s;
    c = __fadd_rn(c, __fadd_rn(e, r));
}

// s = q . k for one key row in shared memory.  The row is read in 16-byte
// pieces starting at piece `lane` (mod the piece count), so the 32 lanes of a
// warp, each on its own row, touch distinct banks.
template <int D, typename Tin>
__device__ __forceinline__ float dot_row(const Tin *krow, const float *qs, int lane)
{
    constexpr int EPC = 16 / int(sizeof(Tin));   // elements per 16-byte piece
    constexpr int NCH = D / EPC;                 // pieces per row (power of two)
    const uint4 *kr = reinterpret_cast<const uint4 *>(krow);
    if constexpr (sizeof(Tin) == 4) {
        const float4 *qa = reinterpret_cast<const float4 *>(qs);
        float p = 0.f, c = 0.f;
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            const int ch = (i + lane) & (NCH - 1);
            const uint4 r = kr[ch];
            const float4 x = qa[ch];
            dot2_step(p, c, x.x, __uint_as_float(r.x));
            dot2_step(p, c, x.y, __uint_as_float(r.y));
            dot2_step(p, c, x.z, __uint_as_float(r.z));
            dot2_step(p, c, x.w, __uint_as_float(r.w));
        }
        return __fadd_rn(p, c);
    } else {
        const float4 *qa = reinterpret_cast<const float4 *>(qs);
        const float4 *qb = reinterpret_cast<const float4 *>(qs + D / 2);
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            const int ch = (i + lane) & (NCH - 1);
            const uint4 r = kr[ch];
            const float4 x = qa[ch];
            const float4 y = qb[ch];
            float k0, k1, k2, k3, k4, k5, k6, k7;
            bf16x2_to_f32(r.x, k0, k1);
            bf16x2_to_f32(r.y, k2, k3);
            bf16x2_to_f32(r.z, k4, k5);
            bf16x2_to_f32(r.w, k6, k7);
            a0 = fmaf(x.x, k0, a0); a1 = fmaf(x.y, k1, a1);
            a2 = fmaf(x.z, k2, a2); a3 = fmaf(x.w, k3, a3);
            a0 = fmaf(y.x, k4, a0); a1 = fmaf(y.y, k5, a1);
            a2 = fmaf(y.z, k6, a2); a3 = fmaf(y.w, k7, a3);
        }
        return (a0 + a1) + (a2 + a3);
    }
}

// s = q . k for one bfloat16 key row in shared memory, lane = token, q in
// shared memory as bfloat16 [D].  Both operands go straight into the float32
// accumulation (mixed-precision FMA, exact products), in four chains.  The
// row and q are read in 16-byte pieces starting at piece `lane` (mod the
// piece count), so the eight rows a quarter-warp reads at a time sit in
// distinct banks for d >= 64.  Every kernel that scores bfloat16 keys this
// way gets bitwise the same score for the same token (lane = token mod 32 in
// all of them).
template <int D>
__device__ __forceinline__ float dot_row_bf16(const __nv_bfloat16 *krow, const __nv_bfloat16 *qsm, int lane)
{
    constexpr int NCH = D / 8;   // 16-byte pieces per row (power of two)
    const uint4 *kr = reinterpret_cast<const uint4 *>(krow);
    const uint4 *qr = reinterpret_cast<const uint4 *>(qsm);
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int ch = (i + lane) & (NCH - 1);
        const uint4 k = kr[ch];
        const uint4 q = qr[ch];
        fma_bf16x2(a0, a1, q.x, k.x);
        fma_bf16x2(a2, a3, q.y, k.y);
        fma_bf16x2(a0, a1, q.z, k.z);
        fma_bf16x2(a2, a3, q.w, k.w);
    }
    return (a0 + a1) + (a2 + a3);
}

// Bounded wait on an mbarrier phase; false when it gave up.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, unsigned parity, int64_t limit_ns)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (unsigned polls = 1;; ++polls) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (polls >= kMinWaitPolls && int64_t(ptx::globaltimer() - t0) > limit_ns) return false;
    }
}

template <int D>
__device__ __forceinline__ void read_state_smem(const float *st, float &m,
                                                float (&u)[VLayout<D>::E], float &w, int lane)
{
    using L = VLayout<D>;
    m = st[0];
    w = st[1];
    if (L::LANES == 32 || lane < L::LANES) {
        load_vals<L::E>(st + 4 + lane * L::E, u);
    } else {
#pragma unroll
        for (int e = 0; e < L::E; ++e) u[e] = 0.f;
    }
}

template <int D>
__device__ __forceinline__ void write_state(float *st, float m, const float (&u)[VLayout<D>::E],
                                            float w, int lane)
{
    using L = VLayout<D>;
    if (lane == 0) {
        st[0] = m;
        st[1] = w;
    }
    if (L::LANES == 32 || lane < L::LANES) store_vals<L::E>(st + 4 + lane * L::E, u);
}

// Set a chunk's flag after this warp's workspace writes: the warp barrier
// orders every lane's writes before lane 0's release store, which makes them
// visible at GPU scope to any reader that acquires the flag.
__device__ __forceinline__ void publish_flag(unsigned *flag, unsigned value, int lane)
{
    __syncwarp();
    if (lane == 0) ptx::st_release(flag, value);
}

// The same, but only while the flag is still FLAG_NONE (an aggregate must
// never replace an inclusive prefix or a poison mark published meanwhile).
__device__ __forceinline__ void publish_agg_if_none(unsigned *flag, int lane)
{
    __syncwarp();
    if (lane == 0) ptx::cas_release(flag, FLAG_NONE, FLAG_AGG);
}

// Bounded wait on an mbarrier phase by spinning on the non-blocking test.
__device__ __forceinline__ bool wait_bar_spin(uint64_t *bar, unsigned parity, int64_t limit_ns)
{
    if (ptx::mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (unsigned polls = 1;; ++polls) {
        if (ptx::mbar_test_wait(bar, parity)) return true;
        if (polls >= kMinWaitPolls && int64_t(ptx::globaltimer() - t0) > limit_ns) return false;
    }
}

// Decoupled look-back (warp 0), 32 predecessors at a time: lane i watches
// chunk j0 - i of the same head.  Once every lane up to the nearest inclusive
// prefix (lane k) has a flag, lanes 0..k are folded in one pass: the scalar
// parts (m_i, w_i) lane-parallel, the d-wide u_i by every lane over its dims.
// x := (window) (+) x, repeated one window further back until an inclusive
// prefix was met.  False when a wait gave up or a predecessor was poisoned.
struct NoHook {
    __device__ void operator()() const {}
};

// `hook` is called (by the whole warp) each time a poll finds a predecessor
// without a published state, before backing off: the caller can do useful
// work there (e.g. publish its own aggregate once it is ready).
template <int D, int BATCH = 8, typename Hook = NoHook>
__device__ bool lookback(const ScanParams &p, int64_t head, int64_t c, float &xm,
                         float (&xu)[VLayout<D>::E], float &xw, int lane, Hook &&hook = Hook())
{
    using L = VLayout<D>;
    constexpr int E = L::E;
    constexpr int SS = StateLayout<D>::SS;
    const int64_t first = head * p.chunks_per_head;   // chunk 0 of this head
    const bool owns = (L::LANES == 32 || lane < L::LANES);
    // every predecessor slot read below lies in [first, first + c), inside the workspace
    if (!AAREN_IN_BOUNDS(p.status, c <= p.chunks_per_head && in_range(first, c, p.heads * p.chunks_per_head)))
        return false;
    for (int64_t j0 = c - 1; j0 >= 0; j0 -= 32) {
        const int64_t j = j0 - lane;
        const bool has = (j >= 0);                       // lanes before chunk 0 act as a stop
        const unsigned *fp = p.flags + first + (has ? j : 0);
        unsigned f = FLAG_INC;
        unsigned inc = 0;
        int k = 31;
        uint64_t t0 = 0;
        unsigned sleep_ns = 32;
        for (unsigned polls = 0;; ++polls) {
            if (has) f = ptx::ld_acquire(fp);
            inc = __ballot_sync(kFull, f == FLAG_INC);
            const unsigned none = __ballot_sync(kFull, f == FLAG_NONE);
            const unsigned poison = __ballot_sync(kFull, f == FLAG_POISON);
            k = inc ? __ffs(inc) - 1 : 31;
            const unsigned upto = (k == 31) ? kFull : ((2u << k) - 1u);   // lanes 0..k
            if (poison & upto) return false;
            if (!(none & upto)) break;
            if (polls == 0) t0 = ptx::globaltimer();
            if (polls >= kMinWaitPolls) {
                int give_up = 0;
                if (lane == 0) give_up = int64_t(ptx::globaltimer() - t0) > p.wait_limit_ns;
                if (__shfl_sync(kFull, give_up, 0)) return false;
            }
            hook();
            __nanosleep(sleep_ns);
            if (sleep_ns < 256) sleep_ns *= 2;
        }
        // scalars of predecessor (lane) i <= k, each read by the lane that saw its flag
        const bool in = has && lane <= k;
        const float *st = p.states + (size_t(first + (has ? j : 0)) * 2 + (f == FLAG_INC ? 1 : 0)) * SS;
        float mi = -INFINITY, wi = 0.f;
        if (in) {
            mi = ptx::ld_relaxed(st);
            wi = ptx::ld_relaxed(st + 1);
        }
        // u of predecessors 0..k, BATCH at a time: a batch's loads are all
        // issued before any is used (one memory round trip per batch, not per
        // predecessor), and the first batch does not wait for the scalars
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
        float ei = 0.f;
        float M = xm;
        for (int i0 = 0; i0 <= k; i0 += BATCH) {
            float v[BATCH][E];
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const int i = i0 + b;
                const unsigned fi = __shfl_sync(kFull, f, i & 31);
                const int64_t ji = j0 - i;
#pragma unroll
                for (int e = 0; e < E; ++e) v[b][e] = 0.f;
                if (owns && i <= k && ji >= 0) {
                    const float *src = p.states + (size_t(first + ji) * 2 + (fi == FLAG_INC ? 1 : 0)) * SS +
                                       4 + lane * E;
                    if constexpr (E == 4) ptx::ld_relaxed4(src, v[b][0], v[b][1], v[b][2], v[b][3]);
                    else if constexpr (E == 2) ptx::ld_relaxed2(src, v[b][0], v[b][1]);
                    else v[b][0] = ptx::ld_relaxed(src);
                }
            }
            if (i0 == 0) {
                M = fmaxf(warp_max(mi), xm);
                ei = in ? exp_rel(mi, M) : 0.f;
            }
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const float ew = __shfl_sync(kFull, ei, (i0 + b) & 31);
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = fmaf(ew, v[b][e], acc[e]);
            }
        }
        const float wsum = warp_sum(ei * wi);
        const float ex = (xm == -INFINITY) ? 0.f : exp_rel(xm, M);
#pragma unroll
        for (int e = 0; e < E; ++e) xu[e] = fmaf(ex, xu[e], acc[e]);
        xw = fmaf(ex, xw, wsum);
        xm = M;
        if (inc != 0) return true;   // lane k held an inclusive prefix (or the head start)
    }
    return true;
}

// Rescan one 32-token group from the running state (rm, u, rw): scalar parts
// across lanes (lane = token), then the d-wide recurrence per lane (lane =
// dims), writing o_t.  FULL = all 32 tokens valid.
template <int D, typename Tin, typename Tout, bool FULL>
__device__ __forceinline__ void rescan_group(float sl, float &rm, float &rw,
                                             float (&u)[VLayout<D>::E], const Tin *vrow,
                                             Tout *orow, float4 *cf, int ntok, int lane,
                                             float2 *strow)
{
    using L = VLayout<D>;
    constexpr int E = L::E;
    // running maximum M_t over the group, seeded with the incoming state's m
    float M = sl;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(kFull, M, off);
        if (lane >= off) M = fmaxf(M, y);
    }
    M = fmaxf(M, rm);
    float Mp = __shfl_up_sync(kFull, M, 1);
    if (lane == 0) Mp = rm;
    const float alpha = exp_rel(Mp, M);                 // rescale of the state carried in
    const float beta = (sl == -INFINITY) ? 0.f : exp_rel(sl, M);   // weight of token t
    // w_t = alpha_t w_{t-1} + beta_t: scan of the affine maps w -> A w + B
    float A = alpha, Bc = beta;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float Ap = __shfl_up_sync(kFull, A, off);
        const float Bp = __shfl_up_sync(kFull, Bc, off);
        if (lane >= off) {
            Bc = fmaf(A, Bp, Bc);
            A *= Ap;
        }
    }
    const float wt = fmaf(A, rw, Bc);
    const float rcp = (sl == -INFINITY) ? 0.f : __frcp_rn(wt);
    if (strow != nullptr && lane < ntok) strow[lane] = make_float2(M, wt);   // this prefix's (m, w)
    cf[lane] = make_float4(alpha, beta, rcp, 0.f);
    __syncwarp();
    rm = __shfl_sync(kFull, M, 31);
    rw = __shfl_sync(kFull, wt, 31);
    const bool owns = (L::LANES == 32 || lane < L::LANES);
    const int n = FULL ? 32 : ntok;
#pragma unroll(FULL ? 32 : 1)
    for (int t = 0; t < n; ++t) {
        const float4 k = cf[t];
        float v[E], o[E];
        if (owns) load_vals<E>(vrow + size_t(t) * D, v);
        if (k.x != 1.0f) {
#pragma unroll
            for (int e = 0; e < E; ++e) u[e] *= k.x;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
            u[e] = fmaf(k.y, owns ? v[e] : 0.f, u[e]);
            o[e] = u[e] * k.z;
        }
        if (owns) store_vals<E>(orow + size_t(t) * D, o);
    }
    __syncwarp();
}

template <int D, typename Tin, typename Tout, int WARPS, int GROUPS>
__global__ void __launch_bounds__(WARPS * 32)
    k_scan_fwd(const ScanParams p)
{
    using L = VLayout<D>;
    using Tile = ScanTile<D, Tin, WARPS, GROUPS>;
    constexpr int E = L::E;
    constexpr int C = Tile::C;
    constexpr int SS = Tile::SS;

    extern __shared__ __align__(128) unsigned char smem[];
    Tin *Ks = reinterpret_cast<Tin *>(smem);
    Tin *Vs = reinterpret_cast<Tin *>(smem + Tile::kv_bytes);
    float *qs = reinterpret_cast<float *>(smem + Tile::q_off);
    float *wst = reinterpret_cast<float *>(smem + Tile::wst_off);   // per-warp aggregates
    float *cst = reinterpret_cast<float *>(smem + Tile::cst_off);   // per-warp carries
    float4 *coef = reinterpret_cast<float4 *>(smem + Tile::coef_off);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Tile::bar_off);
    long long *s_chunk = reinterpret_cast<long long *>(smem + Tile::bar_off + 8);
    int *s_abort = reinterpret_cast<int *>(smem + Tile::bar_off + 16);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // launched as a programmatic dependent of the workspace zeroing: nothing
    // in global memory is touched before that kernel has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) {
        *s_chunk = static_cast<long long>(atomicAdd(p.ticket, 1u));
        *s_abort = 0;
        ptx::mbar_init(bar, 1);
        ptx::fence_barrier_init();
    }
    __syncthreads();
    // tickets interleave the heads (ticket = c * heads + head), so the chunks
    // in flight spread over all heads and their carries progress in parallel;
    // within a head, chunk c - 1 always has an earlier ticket than chunk c
    const int64_t ticket = *s_chunk;
    // one block per chunk: the ticket names a chunk of the launch (uniform)
    if (!AAREN_IN_BOUNDS(p.status, in_range(ticket, 1, p.heads * p.chunks_per_head))) return;
    const int64_t c = ticket / p.heads;
    const int64_t head = ticket - c * p.heads;
    const int64_t chunk = head * p.chunks_per_head + c;   // workspace slot
    const int64_t t0 = c * C;
    const int nvalid = static_cast<int>(p.N - t0 < C ? p.N - t0 : C);
    const int64_t row0 = head * p.N + t0;
    const bool publish = (chunk != p.fault_chunk);
    unsigned *my_flag = p.flags + chunk;
    float *my_state = p.states + size_t(chunk) * 2 * SS;
    // the chunk's rows of K, V, O (and stats) and its slot of the workspace
    const bool rows_ok = AAREN_IN_BOUNDS(p.status, nvalid >= 1 && nvalid <= C && in_range(row0, nvalid, p.heads * p.N) &&
                                                       in_range(chunk, 1, p.heads * p.chunks_per_head) &&
                                                       in_range(head, 1, p.heads));

    // 1. K and V rows of the chunk into shared memory (one bulk copy each)
    if (tid == 0) {
        if (rows_ok) {
            const unsigned bytes = static_cast<unsigned>(nvalid) * D * sizeof(Tin);
            ptx::mbar_arrive_expect_tx(bar, 2 * bytes);
            const uint64_t pol = ptx::policy_evict_first();
            ptx::bulk_g2s(Ks, static_cast<const Tin *>(p.K) + row0 * D, bytes, bar, pol);
            ptx::bulk_g2s(Vs, static_cast<const Tin *>(p.V) + row0 * D, bytes, bar, pol);
        } else {
            ptx::mbar_arrive(bar);   // no copy: the phase completes at once
        }
    }
    if (!rows_ok) {   // uniform: nothing of this chunk is read or written
        wait_bar(bar, 0, p.wait_limit_ns);
        return;
    }
    for (int j = tid; j < D; j += WARPS * 32)
        qs[q_slot<D, Tin>(j)] = to_f32(static_cast<const Tin *>(p.q)[head * D + j]);
    const bool loaded = wait_bar(bar, 0, p.wait_limit_ns);
    if (__syncthreads_or(!loaded)) {
        if (tid == 0) atomicOr(p.status, STATUS_LOAD_TIMEOUT);
        wait_bar(bar, 0, p.wait_limit_ns);   // let copies still in flight land
        if (warp == 0 && publish) publish_flag(my_flag, FLAG_POISON, lane);
        return;
    }

    // 2. scores, lane = token
    float s[GROUPS];
#pragma unroll
    for (int g = 0; g < GROUPS; ++g) {
        const int tok = (warp * GROUPS + g) * 32 + lane;
        s[g] = (tok < nvalid) ? dot_row<D, Tin>(Ks + size_t(tok) * D, qs, lane) : -INFINITY;
    }

    // 3. warp aggregate (m_w, u_w, w_w) relative to the warp's maximum
    {
        float mloc = -INFINITY;
#pragma unroll
        for (int g = 0; g < GROUPS; ++g) mloc = fmaxf(mloc, s[g]);
        const float mw = warp_max(mloc);
        float b[GROUPS];
        float bsum = 0.f;
#pragma unroll
        for (int g = 0; g < GROUPS; ++g) {
            b[g] = (s[g] == -INFINITY) ? 0.f : exp_rel(s[g], mw);
            bsum += b[g];
        }
        const float ww = warp_sum(bsum);
        float u[E];
#pragma unroll
        for (int e = 0; e < E; ++e) u[e] = 0.f;
        const bool owns = (L::LANES == 32 || lane < L::LANES);
#pragma unroll
        for (int g = 0; g < GROUPS; ++g) {
            const int base = (warp * GROUPS + g) * 32;
            if (base >= nvalid) break;
            const Tin *vrow = Vs + size_t(base) * D + lane * E;
            if (base + 32 <= nvalid) {
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const float bt = __shfl_sync(kFull, b[g], t);
                    float v[E];
                    if (owns) load_vals<E>(vrow + size_t(t) * D, v);
#pragma unroll
                    for (int e = 0; e < E; ++e) u[e] = fmaf(bt, owns ? v[e] : 0.f, u[e]);
                }
            } else {
                const int n = nvalid - base;
                for (int t = 0; t < n; ++t) {
                    const float bt = __shfl_sync(kFull, b[g], t);
                    float v[E];
                    if (owns) load_vals<E>(vrow + size_t(t) * D, v);
#pragma unroll
                    for (int e = 0; e < E; ++e) u[e] = fmaf(bt, owns ? v[e] : 0.f, u[e]);
                }
            }
        }
        write_state<D>(wst + warp * SS, mw, u, ww, lane);
    }
    __syncthreads();

    // 4. chunk aggregate, look-back, inclusive prefix, per-warp carries
    if (warp == 0) {
        float am, aw, au[E];
        read_state_smem<D>(wst, am, au, aw, lane);
#pragma unroll
        for (int k = 1; k < WARPS; ++k) {
            float bm, bw, bu[E];
            read_state_smem<D>(wst + k * SS, bm, bu, bw, lane);
            combine_into<E>(am, au, aw, bm, bu, bw);   // b := agg (+) warp k
            am = bm; aw = bw;
#pragma unroll
            for (int e = 0; e < E; ++e) au[e] = bu[e];
        }
        // exclusive prefix of this chunk
        float xm = -INFINITY, xw = 0.f, xu[E];
#pragma unroll
        for (int e = 0; e < E; ++e) xu[e] = 0.f;
        bool ok = true;
        if (c == 0) {
            if (p.m_in != nullptr) {
                xm = p.m_in[head];
                xw = p.w_in[head];
                if (L::LANES == 32 || lane < L::LANES) load_vals<E>(p.u_in + head * D + lane * E, xu);
            }
        } else {
            if (publish) {
                write_state<D>(my_state, am, au, aw, lane);
                publish_flag(my_flag, FLAG_AGG, lane);
            }
            ok = lookback<D>(p, head, c, xm, xu, xw, lane);
        }
        if (ok) {
            float im = am, iw = aw, iu[E];
#pragma unroll
            for (int e = 0; e < E; ++e) iu[e] = au[e];
            combine_into<E>(xm, xu, xw, im, iu, iw);   // inclusive = exclusive (+) aggregate
            if (publish) {
                write_state<D>(my_state + SS, im, iu, iw, lane);
                publish_flag(my_flag, FLAG_INC, lane);
            }
            if (c == p.chunks_per_head - 1 && p.m_out != nullptr) {
                if (lane == 0) {
                    p.m_out[head] = im;
                    p.w_out[head] = iw;
                }
                if (L::LANES == 32 || lane < L::LANES) store_vals<E>(p.u_out + head * D + lane * E, iu);
            }
            // carry into warp k = exclusive (+) aggregates of warps 0..k-1
#pragma unroll
            for (int k = 0; k < WARPS; ++k) {
                write_state<D>(cst + k * SS, xm, xu, xw, lane);
                if (k + 1 < WARPS) {
                    float bm, bw, bu[E];
                    read_state_smem<D>(wst + k * SS, bm, bu, bw, lane);
                    combine_into<E>(xm, xu, xw, bm, bu, bw);
                    xm = bm; xw = bw;
#pragma unroll
                    for (int e = 0; e < E; ++e) xu[e] = bu[e];
                }
            }
        } else {
            if (lane == 0) {
                atomicOr(p.status, STATUS_LOOKBACK_TIMEOUT);
                *s_abort = 1;
            }
            if (publish) publish_flag(my_flag, FLAG_POISON, lane);
        }
    }
    __syncthreads();
    if (*s_abort) return;

    // 5. rescan from the carry and write O
    {
        float rm, rw, u[E];
        read_state_smem<D>(cst + warp * SS, rm, u, rw, lane);
        float4 *cf = coef + warp * 32;
#pragma unroll
        for (int g = 0; g < GROUPS; ++g) {
            const int base = (warp * GROUPS + g) * 32;
            if (base >= nvalid) break;
            const Tin *vrow = Vs + size_t(base) * D + lane * E;
            Tout *orow = static_cast<Tout *>(p.O) + size_t(row0 + base) * D + lane * E;
            if (base + 32 <= nvalid)
                rescan_group<D, Tin, Tout, true>(s[g], rm, rw, u, vrow, orow, cf, 32, lane,
                                                 p.stats ? p.stats + (row0 + base) : nullptr);
            else
                rescan_group<D, Tin, Tout, false>(s[g], rm, rw, u, vrow, orow, cf, nvalid - base,
                                                  lane, p.stats ? p.stats + (row0 + base) : nullptr);
        }
    }
}

}  // namespace aaren
