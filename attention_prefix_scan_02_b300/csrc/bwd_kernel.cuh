// bwd_kernel.cuh -- gradients of the many-to-many output with respect to q,
// K and V, in one pass over K, V, O and dO, with O(1) extra memory per head.
//
// The memory-efficient-attention review reports its method for inference
// and for differentiation (its abstract; section 5.2, whose body the page
// lacks), and the Aaren review calls the RNN form exact and differentiable
// ("Proposed method").  For one head, an upstream gradient g_t = dL/do_t and
// lse_t = log sum_{i<=t} e^{s_i} (so p_{t,i} = e^{s_i - lse_t}):
//
//   dL/dv_i = e^{s_i - lse_i} R_i,   dL/ds_i = e^{s_i - lse_i} (v_i . R_i - D_i),
//   R_i = sum_{t>=i} e^{lse_i - lse_t} g_t,   D_i = sum_{t>=i} e^{lse_i - lse_t} (g_t . o_t),
//   dL/dq = sum_i dL/ds_i k_i,   dL/dk_i = dL/ds_i q.
//
// R and D are suffix sums with weights <= 1 (lse never decreases), i.e. the
// reverse linear recurrence R_i = g_i + e^{lse_i - lse_{i+1}} R_{i+1}.  The
// forward pass saved every prefix's (m_t, w_t), lse_t = m_t + log w_t, so
//   e^{s_i - lse_i} = e^{s_i - m_i} / w_i,
//   e^{lse_a - lse_b} = e^{m_a - m_b} w_a / w_b
// and no absolute exponential appears.
//
// Structure: the forward kernel's chunked scan run backwards.  One block
// handles one chunk of C = 32 WARPS tokens; tickets are handed out from the
// last chunk of each head to the first, interleaved over heads.  A suffix
// state is (m_ref, w_ref, D, R[d]): sums relative to lse at its first token.
// Combining a state L with the state that follows it, Rt:
//   (m_L, w_L, D_L + f D_Rt, R_L + f R_Rt),  f = e^{m_L - m_Rt} w_L / w_Rt  (<= 1),
// and an empty state (w = 0) is the identity.  A chunk publishes its
// aggregate, looks FORWARD over its successors (decoupled look-back, 32 at a
// time) for the suffix that follows it, and publishes its inclusive suffix.
// Within the chunk each warp rescans its 32 rows from the last to the first.
// dL/dq is summed per block, added to a per-head float32 accumulator, and
// the head's last chunk to finish writes it out.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"
#include "scan_kernel.cuh"

namespace aaren {

struct BwdParams {
    const void *q;
    const void *K;
    const void *V;
    const void *O;
    const void *dO;
    const float2 *stats;   // [heads, N]: (m_t, w_t) of every prefix, from the forward
    float *dq;             // [heads, d]      float32
    float *dK;             // [heads, N, d]   float32
    float *dV;             // [heads, N, d]   float32
    float *dq_acc;         // workspace [heads, d] (zeroed before launch)
    unsigned *dq_count;    // workspace [heads]    (zeroed before launch)
    unsigned *ticket;      // workspace
    unsigned *flags;       // workspace: one flag per chunk (zeroed)
    float *states;         // workspace: per chunk [aggregate | inclusive] suffix states
    unsigned *status;
    int64_t N;
    int64_t heads;
    int64_t chunks_per_head;
    int64_t fault_chunk;   // testing: chunk that never publishes its suffix (-1 = none)
    int64_t wait_limit_ns;
};

// A suffix state: reference (m, w) of its first token, D, and this lane's
// E components of R.
template <int E>
struct Suffix {
    float m, w, D;
    float R[E];
};

template <int E>
__device__ __forceinline__ void suffix_empty(Suffix<E> &x)
{
    x.m = -INFINITY;
    x.w = 0.f;
    x.D = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) x.R[e] = 0.f;
}

// e^{lse_a - lse_b} from the two prefixes' (m, w); b follows a, so <= 1.
__device__ __forceinline__ float lse_ratio(float ma, float wa, float mb, float wb)
{
    return exp_rel(ma, mb) * (wa / wb);
}

// x := x (+) y   (y follows x)
template <int E>
__device__ __forceinline__ void suffix_append(Suffix<E> &x, const Suffix<E> &y)
{
    if (y.w == 0.f) return;
    if (x.w == 0.f) {
        x = y;
        return;
    }
    const float f = lse_ratio(x.m, x.w, y.m, y.w);
    x.D = fmaf(f, y.D, x.D);
#pragma unroll
    for (int e = 0; e < E; ++e) x.R[e] = fmaf(f, y.R[e], x.R[e]);
}

// Layout in the workspace and in shared memory: [m, w, D, unused, R_0 .. R_{d-1}].
template <int D>
__device__ __forceinline__ void suffix_store(float *st, const Suffix<VLayout<D>::E> &x, int lane)
{
    using L = VLayout<D>;
    if (lane == 0) {
        st[0] = x.m;
        st[1] = x.w;
        st[2] = x.D;
    }
    if (L::LANES == 32 || lane < L::LANES) store_vals<L::E>(st + 4 + lane * L::E, x.R);
}

template <int D>
__device__ __forceinline__ void suffix_load_smem(const float *st, Suffix<VLayout<D>::E> &x, int lane)
{
    using L = VLayout<D>;
    x.m = st[0];
    x.w = st[1];
    x.D = st[2];
    if (L::LANES == 32 || lane < L::LANES) {
        load_vals<L::E>(st + 4 + lane * L::E, x.R);
    } else {
#pragma unroll
        for (int e = 0; e < L::E; ++e) x.R[e] = 0.f;
    }
}

// Suffix that follows chunk c of `head`: successors c+1, c+2, ... folded,
// 32 chunks per poll (lane i watches chunk j0 + i); a window is folded up to
// its first inclusive suffix (or the end of the head).  False when a wait
// gave up or a successor was poisoned.
template <int D>
__device__ bool lookforward(const BwdParams &p, int64_t head, int64_t c, Suffix<VLayout<D>::E> &x,
                            int lane)
{
    using L = VLayout<D>;
    constexpr int E = L::E;
    constexpr int SS = StateLayout<D>::SS;
    const int64_t first = head * p.chunks_per_head;
    const bool owns = (L::LANES == 32 || lane < L::LANES);
    suffix_empty<E>(x);
    // every successor slot read below lies in (first + c, first + chunks_per_head)
    if (!AAREN_IN_BOUNDS(p.status, c >= 0 && in_range(first, p.chunks_per_head, p.heads * p.chunks_per_head)))
        return false;
    for (int64_t j0 = c + 1; j0 < p.chunks_per_head; j0 += 32) {
        const int64_t j = j0 + lane;
        const bool has = (j < p.chunks_per_head);   // lanes past the end act as a stop
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
            const unsigned upto = (k == 31) ? kFull : ((2u << k) - 1u);
            if (poison & upto) return false;
            if (!(none & upto)) break;
            if (polls == 0) t0 = ptx::globaltimer();
            if (polls >= kMinWaitPolls) {
                int give_up = 0;
                if (lane == 0) give_up = int64_t(ptx::globaltimer() - t0) > p.wait_limit_ns;
                if (__shfl_sync(kFull, give_up, 0)) return false;
            }
            __nanosleep(sleep_ns);
            if (sleep_ns < 256) sleep_ns *= 2;
        }
        // the window's states relative to its first chunk (lane 0, always present)
        const bool in = has && lane <= k;
        const float *st = p.states + (size_t(first + (has ? j : 0)) * 2 + (f == FLAG_INC ? 1 : 0)) * SS;
        float mi = 0.f, wi = 0.f, Di = 0.f;
        if (in) {
            mi = ptx::ld_relaxed(st);
            wi = ptx::ld_relaxed(st + 1);
            Di = ptx::ld_relaxed(st + 2);
        }
        const float m0 = __shfl_sync(kFull, mi, 0);
        const float w0 = __shfl_sync(kFull, wi, 0);
        const float fi = (in && wi != 0.f) ? lse_ratio(m0, w0, mi, wi) : 0.f;
        Suffix<E> win;
        win.m = m0;
        win.w = w0;
        win.D = warp_sum(fi * Di);
#pragma unroll
        for (int e = 0; e < E; ++e) win.R[e] = 0.f;
        for (int i0 = 0; i0 <= k; i0 += 8) {
            float v[8][E];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const int i = i0 + b;
                const unsigned fl = __shfl_sync(kFull, f, i & 31);
                const int64_t ji = j0 + i;
#pragma unroll
                for (int e = 0; e < E; ++e) v[b][e] = 0.f;
                if (owns && i <= k && ji < p.chunks_per_head) {
                    const float *src = p.states + (size_t(first + ji) * 2 + (fl == FLAG_INC ? 1 : 0)) * SS +
                                       4 + lane * E;
                    if constexpr (E == 4) ptx::ld_relaxed4(src, v[b][0], v[b][1], v[b][2], v[b][3]);
                    else if constexpr (E == 2) ptx::ld_relaxed2(src, v[b][0], v[b][1]);
                    else v[b][0] = ptx::ld_relaxed(src);
                }
            }
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const float fb = __shfl_sync(kFull, fi, (i0 + b) & 31);
#pragma unroll
                for (int e = 0; e < E; ++e) win.R[e] = fmaf(fb, v[b][e], win.R[e]);
            }
        }
        suffix_append<E>(x, win);
        if (inc != 0) return true;   // an inclusive suffix (or the end of the head) was reached
    }
    return true;
}

// Rows per block (chunk) of the backward kernel: K, dO and one shared slot
// for O and then V of a chunk fill at most about 64 KB of shared memory.  O
// is read only for the per-token dot products g . o at the start, V only in
// the rescan after the look-forward, so V is copied into O's slot once every
// warp is done with O (the copy overlaps the look-forward).
template <int D, typename Tin, typename Tout>
struct BwdTile {
    static constexpr int OV_ELEM = int(sizeof(Tin)) > int(sizeof(Tout)) ? int(sizeof(Tin)) : int(sizeof(Tout));
    static constexpr int ROW_BYTES = D * (int(sizeof(Tin)) + OV_ELEM + int(sizeof(Tout)));
    static constexpr int WARPS_RAW = 65536 / (32 * ROW_BYTES);
    static constexpr int WARPS = WARPS_RAW < 1 ? 1 : (WARPS_RAW > 4 ? 4 : WARPS_RAW);
    static constexpr int C = 32 * WARPS;
    static constexpr int SS = StateLayout<D>::SS;
    static constexpr size_t in_bytes = size_t(C) * D * sizeof(Tin);
    static constexpr size_t out_bytes = size_t(C) * D * sizeof(Tout);
    static constexpr size_t ov_bytes = size_t(C) * D * OV_ELEM;
    static constexpr size_t k_off = 0;
    static constexpr size_t o_off = k_off + in_bytes;   // O, then V
    static constexpr size_t v_off = o_off;
    static constexpr size_t g_off = o_off + ov_bytes;
    static constexpr size_t wst_off = g_off + out_bytes;                         // [WARPS][SS]
    static constexpr size_t cst_off = wst_off + size_t(WARPS) * SS * sizeof(float);
    static constexpr size_t cf_off = cst_off + size_t(WARPS) * SS * sizeof(float); // [WARPS][32] float4
    static constexpr size_t dq_off = cf_off + size_t(WARPS) * 32 * sizeof(float4);  // [WARPS][D]
    static constexpr size_t q_off = dq_off + size_t(WARPS) * D * sizeof(float);      // [D] float
    static constexpr size_t bar_off = q_off + size_t(D) * sizeof(float);
    static constexpr size_t smem_bytes = bar_off + 32;
    static_assert(in_bytes % 16 == 0 && out_bytes % 16 == 0 && wst_off % 16 == 0 &&
                      cf_off % 16 == 0 && dq_off % 16 == 0 && q_off % 16 == 0 && bar_off % 8 == 0,
                  "shared-memory regions must stay aligned");
};

// x[i] holds this lane's share of row i's dot product (i < 8); returns on
// every lane the full sum over the 32 lanes for row (lane & 7).
template <typename Acc>
__device__ __forceinline__ Acc bwd_transpose_sum8(Acc (&x)[8], int lane)
{
#pragma unroll
    for (int h = 4; h >= 1; h >>= 1) {
        const bool upper = (lane & h) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const Acc send = upper ? x[i] : x[i + h];
            const Acc keep = upper ? x[i + h] : x[i];
            x[i] = keep + __shfl_xor_sync(kFull, send, h);
        }
    }
    Acc y = x[0];
    y += __shfl_xor_sync(kFull, y, 8);
    y += __shfl_xor_sync(kFull, y, 16);
    return y;
}

template <int D, typename Tin, typename Tout>
__global__ void __launch_bounds__(BwdTile<D, Tin, Tout>::WARPS * 32) k_scan_bwd(const BwdParams p)
{
    using L = VLayout<D>;
    using T = BwdTile<D, Tin, Tout>;
    constexpr int E = L::E;
    constexpr int C = T::C;
    constexpr int SS = T::SS;
    constexpr int WARPS = T::WARPS;

    extern __shared__ __align__(128) unsigned char smem[];
    Tin *Ks = reinterpret_cast<Tin *>(smem + T::k_off);
    Tin *Vs = reinterpret_cast<Tin *>(smem + T::v_off);
    Tout *Os = reinterpret_cast<Tout *>(smem + T::o_off);
    Tout *Gs = reinterpret_cast<Tout *>(smem + T::g_off);
    float *wst = reinterpret_cast<float *>(smem + T::wst_off);
    float *cst = reinterpret_cast<float *>(smem + T::cst_off);
    float *dqs = reinterpret_cast<float *>(smem + T::dq_off);
    float *qs = reinterpret_cast<float *>(smem + T::q_off);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + T::bar_off);
    long long *s_ticket = reinterpret_cast<long long *>(smem + T::bar_off + 8);
    int *s_abort = reinterpret_cast<int *>(smem + T::bar_off + 16);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const bool owns = (L::LANES == 32 || lane < L::LANES);

    if (tid == 0) {
        *s_ticket = static_cast<long long>(atomicAdd(p.ticket, 1u));
        *s_abort = 0;
        ptx::mbar_init(bar, 1);
        ptx::fence_barrier_init();
    }
    __syncthreads();
    // tickets run from the last chunk of each head to the first, interleaved
    // over heads: every successor of a chunk holds an earlier ticket
    const int64_t ticket = *s_ticket;
    // one block per chunk: the ticket names a chunk of the launch (uniform)
    if (!AAREN_IN_BOUNDS(p.status, in_range(ticket, 1, p.heads * p.chunks_per_head))) return;
    const int64_t rc = ticket / p.heads;
    const int64_t head = ticket - rc * p.heads;
    const int64_t c = p.chunks_per_head - 1 - rc;
    const int64_t chunk = head * p.chunks_per_head + c;
    const int64_t t0 = c * C;
    const int nvalid = static_cast<int>(p.N - t0 < C ? p.N - t0 : C);
    const int64_t row0 = head * p.N + t0;
    // the chunk's rows of K, V, O, dO, stats, dK and dV, the head's q and dq
    // entries, and the chunk's workspace slot (uniform; on a violation the
    // block reads and writes nothing and publishes nothing)
    if (!AAREN_IN_BOUNDS(p.status, nvalid >= 1 && nvalid <= C && in_range(row0, nvalid, p.heads * p.N) &&
                                       in_range(head, 1, p.heads) &&
                                       in_range(chunk, 1, p.heads * p.chunks_per_head)))
        return;
    unsigned *my_flag = p.flags + chunk;
    const bool publish = (chunk != p.fault_chunk);   // testing hook: a suffix never published
    float *my_state = p.states + size_t(chunk) * 2 * SS;

    // K, O, dO rows of the chunk into shared memory (V follows into O's slot)
    const unsigned bi = static_cast<unsigned>(nvalid) * D * sizeof(Tin);
    if (tid == 0) {
        const unsigned bo = static_cast<unsigned>(nvalid) * D * sizeof(Tout);
        ptx::mbar_arrive_expect_tx(bar, bi + 2 * bo);
        const uint64_t pol = ptx::policy_evict_first();
        ptx::bulk_g2s(Ks, static_cast<const Tin *>(p.K) + row0 * D, bi, bar, pol);
        ptx::bulk_g2s(Os, static_cast<const Tout *>(p.O) + row0 * D, bo, bar, pol);
        ptx::bulk_g2s(Gs, static_cast<const Tout *>(p.dO) + row0 * D, bo, bar, pol);
    }
    // meanwhile: q (lane dims; for float32 keys also in shared memory in the
    // forward kernel's layout) and this lane's token statistics
    if constexpr (sizeof(Tin) == 4) {
        for (int j = tid; j < D; j += WARPS * 32)
            qs[q_slot<D, Tin>(j)] = to_f32(static_cast<const Tin *>(p.q)[head * D + j]);
    } else {   // bfloat16 q as it is stored, for the forward's score function
        for (int j = tid; j < D; j += WARPS * 32)
            reinterpret_cast<Tin *>(qs)[j] = static_cast<const Tin *>(p.q)[head * D + j];
    }
    float qv[E];
    if (owns) {
        load_vals<E>(static_cast<const Tin *>(p.q) + head * D + lane * E, qv);
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) qv[e] = 0.f;
    }
    int nv = nvalid - warp * 32;
    nv = nv < 0 ? 0 : (nv > 32 ? 32 : nv);
    float mt = -INFINITY, wt = 0.f;          // (m, w) of this lane's prefix (token = lane)
    if (lane < nv) {
        const float2 st = p.stats[row0 + warp * 32 + lane];
        mt = st.x;
        wt = st.y;
    }
    const bool loaded = wait_bar(bar, 0, p.wait_limit_ns);
    if (__syncthreads_or(!loaded)) {
        if (tid == 0) atomicOr(p.status, STATUS_LOAD_TIMEOUT);
        wait_bar(bar, 0, p.wait_limit_ns);
        if (warp == 0 && publish) publish_flag(my_flag, FLAG_POISON, lane);
        return;
    }

    // 1. per token (lane = token): score, g . o, weight p = e^{s - lse}
    const Tin *Kw = Ks + size_t(warp) * 32 * D;
    const Tin *Vw = Vs + size_t(warp) * 32 * D;
    const Tout *Ow = Os + size_t(warp) * 32 * D;
    const Tout *Gw = Gs + size_t(warp) * 32 * D;
    // The score is recomputed with the forward kernel's arithmetic (bitwise
    // the same value), so e^{s - m} is consistent with the saved (m, w).
    float s;
    if constexpr (sizeof(Tin) == 4) {
        s = (lane < nv) ? dot_row<D, Tin>(Kw + size_t(lane) * D, qs, lane) : -INFINITY;
    } else {
        s = (lane < nv) ? dot_row_bf16<D>(Kw + size_t(lane) * D, reinterpret_cast<const Tin *>(qs), lane)
                        : -INFINITY;
    }
    // g_t . o_t (both rows from shared memory), and in the same pass the R
    // part of the warp aggregate, sum_t c_t g_t with c_t = e^{lse_0 - lse_t}
    // relative to the warp's first row: the weights need only the saved
    // (m, w), so each g row is read once and the aggregate, which the
    // predecessors' look-forwards wait on, is ready sooner.  Rows past nv
    // are zero and weigh 0.
    const bool valid = lane < nv;
    const float am0 = __shfl_sync(kFull, mt, 0), aw0 = __shfl_sync(kFull, wt, 0);
    const float cw = valid ? lse_ratio(am0, aw0, mt, wt) : 0.f;
    float delta, Ragg[E];
#pragma unroll
    for (int e = 0; e < E; ++e) Ragg[e] = 0.f;
    {
        float x8[8];
        delta = 0.f;
#pragma unroll 1
        for (int quarter = 0; quarter < 4; ++quarter) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = quarter * 8 + i;
                x8[i] = 0.f;
                float gf[E];
#pragma unroll
                for (int e = 0; e < E; ++e) gf[e] = 0.f;
                if (owns && r < nv) {
                    float of[E];
                    load_vals<E>(Gw + size_t(r) * D + lane * E, gf);
                    load_vals<E>(Ow + size_t(r) * D + lane * E, of);
                    float acc = gf[0] * of[0];
#pragma unroll
                    for (int e = 1; e < E; ++e) acc = fmaf(gf[e], of[e], acc);
                    x8[i] = acc;
                }
                const float cr = __shfl_sync(kFull, cw, r);
#pragma unroll
                for (int e = 0; e < E; ++e) Ragg[e] = fmaf(cr, gf[e], Ragg[e]);
            }
            const float sr = bwd_transpose_sum8<float>(x8, lane);
            if ((lane >> 3) == quarter) delta = sr;
        }
    }
    const float pw = valid ? exp_rel(s, mt) / wt : 0.f;

    // 2. warp aggregate: sums relative to lse at the warp's first row
    {
        Suffix<E> a;
        if (nv > 0) {
            a.m = am0;
            a.w = aw0;
            a.D = warp_sum(cw * delta);
#pragma unroll
            for (int e = 0; e < E; ++e) a.R[e] = Ragg[e];
        } else {
            suffix_empty<E>(a);
        }
        suffix_store<D>(wst + warp * SS, a, lane);
    }
    // every warp is done with O: V into its slot, during the look-forward
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0) {
        ptx::mbar_arrive_expect_tx(bar, bi);
        ptx::bulk_g2s(Vs, static_cast<const Tin *>(p.V) + row0 * D, bi, bar, ptx::policy_evict_first());
    }

    // 3. chunk aggregate, look-forward, inclusive suffix, per-warp carries
    if (warp == 0) {
        Suffix<E> agg;
        suffix_empty<E>(agg);
#pragma unroll
        for (int k = 0; k < WARPS; ++k) {
            Suffix<E> b;
            suffix_load_smem<D>(wst + k * SS, b, lane);
            suffix_append<E>(agg, b);
        }
        Suffix<E> x;
        bool ok = true;
        if (c == p.chunks_per_head - 1) {
            suffix_empty<E>(x);
        } else {
            if (publish) {
                suffix_store<D>(my_state, agg, lane);
                publish_flag(my_flag, FLAG_AGG, lane);
            }
            ok = lookforward<D>(p, head, c, x, lane);
        }
        if (ok) {
            Suffix<E> inc = agg;
            suffix_append<E>(inc, x);
            if (publish) {
                suffix_store<D>(my_state + SS, inc, lane);
                publish_flag(my_flag, FLAG_INC, lane);
            }
            // carry into warp k = aggregates of warps k+1.. (+) the suffix after the chunk
            for (int k = WARPS - 1; k >= 0; --k) {
                suffix_store<D>(cst + k * SS, x, lane);
                Suffix<E> b;
                suffix_load_smem<D>(wst + k * SS, b, lane);
                suffix_append<E>(b, x);
                x = b;
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
    // V has landed (a block never leaves with its copy in flight)
    const bool v_loaded = wait_bar(bar, 1, p.wait_limit_ns);
    if (*s_abort) return;
    if (__syncthreads_or(!v_loaded)) {
        if (tid == 0) atomicOr(p.status, STATUS_LOAD_TIMEOUT);
        wait_bar(bar, 1, p.wait_limit_ns);
        return;
    }

    // 4. rescan the warp's rows from the last to the first
    float dsv = 0.f;   // dL/ds of this lane's token
    if (nv > 0) {
        Suffix<E> cy;
        suffix_load_smem<D>(cst + warp * SS, cy, lane);
        // decay from each row to the next (the carry's reference after the last row)
        float mn = __shfl_down_sync(kFull, mt, 1);
        float wn = __shfl_down_sync(kFull, wt, 1);
        if (lane == nv - 1) {
            mn = cy.m;
            wn = cy.w;
        }
        const float fdec = (valid && wn != 0.f) ? lse_ratio(mt, wt, mn, wn) : 0.f;
        // D_i = delta_i + f_i D_{i+1}: a scan of affine maps from the last row back
        float A = valid ? fdec : 1.f, Bv = valid ? delta : 0.f;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float Ap = __shfl_down_sync(kFull, A, off);
            const float Bp = __shfl_down_sync(kFull, Bv, off);
            if (lane + off < 32) {
                Bv = fmaf(A, Bp, Bv);
                A *= Ap;
            }
        }
        const float Dt = fmaf(A, cy.D, Bv);
        // R_i = g_i + f_i R_{i+1} per lane over its dims; dV_i = p_i R_i;
        // v_i . R_i gathered eight rows at a time (lane = token)
        float4 *cf = reinterpret_cast<float4 *>(smem + T::cf_off) + warp * 32;
        cf[lane] = make_float4(fdec, pw, 0.f, 0.f);
        __syncwarp();
        float R[E];
#pragma unroll
        for (int e = 0; e < E; ++e) R[e] = cy.R[e];
        float vR = 0.f;
        float *dVrow = p.dV + size_t(row0 + warp * 32) * D + lane * E;
        const int top = ((nv + 7) / 8) * 8;   // rows [top - 8, top) first
#pragma unroll 1
        for (int b0 = top - 8; b0 >= 0; b0 -= 8) {
            float x8[8];
#pragma unroll
            for (int ii = 7; ii >= 0; --ii) {
                const int r = b0 + ii;
                x8[ii] = 0.f;
                if (r < nv) {
                    const float4 k4 = cf[r];
                    float gf[E], vf[E], dv[E];
                    if (owns) {
                        load_vals<E>(Gw + size_t(r) * D + lane * E, gf);
                        load_vals<E>(Vw + size_t(r) * D + lane * E, vf);
                    } else {
#pragma unroll
                        for (int e = 0; e < E; ++e) gf[e] = vf[e] = 0.f;
                    }
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        R[e] = fmaf(k4.x, R[e], gf[e]);
                        dv[e] = k4.y * R[e];
                        acc = fmaf(vf[e], R[e], acc);
                    }
                    x8[ii] = acc;
                    if (owns) store_vals<E>(dVrow + size_t(r) * D, dv);
                }
            }
            const float sr = bwd_transpose_sum8<float>(x8, lane);
            if ((lane >> 3) == (b0 >> 3)) vR = sr;
        }
        dsv = valid ? pw * (vR - Dt) : 0.f;

        // 5. dL/dk_t = ds_t q, and this warp's share of dL/dq = sum_t ds_t k_t
        float dq[E];
#pragma unroll
        for (int e = 0; e < E; ++e) dq[e] = 0.f;
        float *dKrow = p.dK + size_t(row0 + warp * 32) * D + lane * E;
#pragma unroll 4
        for (int r = 0; r < nv; ++r) {
            const float dr = __shfl_sync(kFull, dsv, r);
            if (owns) {
                float kf[E], dk[E];
                load_vals<E>(Kw + size_t(r) * D + lane * E, kf);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    dk[e] = dr * qv[e];
                    dq[e] = fmaf(dr, kf[e], dq[e]);
                }
                store_vals<E>(dKrow + size_t(r) * D, dk);
            }
        }
        if (owns) store_vals<E>(dqs + warp * D + lane * E, dq);
    } else {
        float z[E];
#pragma unroll
        for (int e = 0; e < E; ++e) z[e] = 0.f;
        if (owns) store_vals<E>(dqs + warp * D + lane * E, z);
    }
    __syncthreads();

    // 6. the block's dL/dq into the head's accumulator; the last chunk writes it
    if (warp == 0) {
        if (owns) {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                float sum = 0.f;
#pragma unroll
                for (int k = 0; k < WARPS; ++k) sum += dqs[k * D + lane * E + e];
                atomicAdd(p.dq_acc + head * D + lane * E + e, sum);
            }
        }
        __threadfence();
        __syncwarp();
        unsigned done = 0;
        if (lane == 0) done = atomicAdd(p.dq_count + head, 1u);
        done = __shfl_sync(kFull, done, 0);
        if (done == static_cast<unsigned>(p.chunks_per_head - 1)) {
            __threadfence();
            if (owns) {
                float out[E];
#pragma unroll
                for (int e = 0; e < E; ++e) out[e] = ptx::ld_relaxed(p.dq_acc + head * D + lane * E + e);
                store_vals<E>(p.dq + head * D + lane * E, out);
            }
        }
    }
}

}  // namespace aaren
