// reduce_kernel.cuh -- the many-to-one form of the softmax-attention
// accumulation: for every head only the last output o_N (and the final state
// (m, u, w)), reading K and V once and writing no per-token output.
//
// The method: attention as a many-to-one RNN ("Attention as an RNN" review,
// "Proposed method": a query attends over all N tokens and yields one
// output), computed as the single-query running sums of the "Self-attention
// Does Not Need O(n^2) Memory" review (section 2, "Algorithm": sums of
// v_i e^{s_i} and e^{s_i}, divided at the end), kept stable by the running
// maximum (its section 3).  The state operator (+) is associative and
// commutative, so a head's tokens can be cut into parts that are reduced
// independently and combined in any grouping: no part waits for another.
//
// Work decomposition: every head is cut into P contiguous parts of `seg`
// tokens; one warp reduces one part, streaming its K and V rows straight
// from global memory into registers (lane l owns dims [E l, E l + E) of
// every row; a row of K or V is one coalesced warp-wide load), eight rows
// per batch with the next batch's loads in flight while the current one is
// reduced:
//   * scores: each lane's E-term share of q . k_t, then a transposed
//     butterfly of shuffles (8 rows at a time);
//   * running state: when the batch's maximum exceeds the running maximum
//     m, u and w are rescaled by e^{m_old - m_new}; then w += sum e^{s - m},
//     u += sum e^{s - m} v (per lane over its dims).
// The warp writes its part's state to the workspace and counts itself in
// the head's arrival counter; the warp that arrives last folds the P part
// states in part order (so the result does not depend on which warp was
// last), applies the optional starting state, and writes o_N = u / w and the
// final state.  Nothing waits on another warp: there is no spin loop.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"
#include "scan_kernel.cuh"

namespace aaren {

constexpr int kReduceWarps = 8;        // warps per block
constexpr int kReduceRows = 8;         // rows per batch
constexpr int kReduceMinSeg = 64;      // shortest part worth a warp

struct ReduceParams {
    const void *q;
    const void *K;
    const void *V;
    void *o_last;          // [heads, d] in the output type, or null
    const float *m_in;     // optional starting state per head (all or none)
    const float *u_in;
    const float *w_in;
    float *m_out;          // optional final state per head (all or none)
    float *u_out;
    float *w_out;
    float *parts;          // workspace: [heads][P] part states of SS floats
    unsigned *counts;      // workspace: [heads] arrivals (zeroed before launch)
    int64_t N;
    int64_t heads;
    int64_t P;             // parts per head
    int64_t seg;           // tokens per part (a multiple of kReduceRows)
    int64_t part_slots;    // part states the workspace holds (checked build)
    unsigned *status;      // device status word (checked build)
};

// Streaming loads (read once: evict first).
__device__ __forceinline__ uint4 ldg_stream_u4(const uint4 *p) { return __ldcs(p); }
__device__ __forceinline__ uint2 ldg_stream_u2(const uint2 *p) { return __ldcs(p); }
__device__ __forceinline__ unsigned ldg_stream_u1(const unsigned *p) { return __ldcs(p); }
__device__ __forceinline__ unsigned ldg_stream_u16(const unsigned short *p) { return __ldcs(p); }

// One row's lane-owned E values of K or V, held in registers.
template <typename Tin, int E>
struct RowRegs;

template <int E>
struct RowRegs<__nv_bfloat16, E> {
    unsigned w[E == 4 ? 2 : 1];
    __device__ __forceinline__ void clear()
    {
#pragma unroll
        for (int k = 0; k < (E == 4 ? 2 : 1); ++k) w[k] = 0u;
    }
    __device__ __forceinline__ void load(const __nv_bfloat16 *p)
    {
        if constexpr (E == 4) {
            const uint2 v = ldg_stream_u2(reinterpret_cast<const uint2 *>(p));
            w[0] = v.x;
            w[1] = v.y;
        } else if constexpr (E == 2) {
            w[0] = ldg_stream_u1(reinterpret_cast<const unsigned *>(p));
        } else {
            w[0] = ldg_stream_u16(reinterpret_cast<const unsigned short *>(p));
        }
    }
    __device__ __forceinline__ void get(float (&f)[E]) const
    {
        if constexpr (E == 4) {
            bf16x2_to_f32(w[0], f[0], f[1]);
            bf16x2_to_f32(w[1], f[2], f[3]);
        } else if constexpr (E == 2) {
            bf16x2_to_f32(w[0], f[0], f[1]);
        } else {
            f[0] = __uint_as_float(w[0] << 16);
        }
    }
};

template <int E>
struct RowRegs<float, E> {
    float v[E];
    __device__ __forceinline__ void clear()
    {
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = 0.f;
    }
    __device__ __forceinline__ void load(const float *p)
    {
        if constexpr (E == 4) {
            const uint4 r = ldg_stream_u4(reinterpret_cast<const uint4 *>(p));
            v[0] = __uint_as_float(r.x);
            v[1] = __uint_as_float(r.y);
            v[2] = __uint_as_float(r.z);
            v[3] = __uint_as_float(r.w);
        } else if constexpr (E == 2) {
            const uint2 r = ldg_stream_u2(reinterpret_cast<const uint2 *>(p));
            v[0] = __uint_as_float(r.x);
            v[1] = __uint_as_float(r.y);
        } else {
            v[0] = __uint_as_float(ldg_stream_u1(reinterpret_cast<const unsigned *>(p)));
        }
    }
    __device__ __forceinline__ void get(float (&f)[E]) const
    {
#pragma unroll
        for (int e = 0; e < E; ++e) f[e] = v[e];
    }
};

// x[i] holds this lane's share of row i's value (i < 8); returns on every
// lane the sum over the 32 lanes for row (lane & 7).  Float and double.
template <typename Acc>
__device__ __forceinline__ Acc transpose_sum8_t(Acc (&x)[8], int lane)
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

// Reduce one batch of up to 8 rows into the running state (m, u, w).
// float32 keys take their score in float64 (products exact, sum rounded
// once to float32), as their scores reach hundreds.
template <typename Tin, int D>
__device__ __forceinline__ void reduce_batch(const RowRegs<Tin, VLayout<D>::E> (&kr)[kReduceRows],
                                             const RowRegs<Tin, VLayout<D>::E> (&vr)[kReduceRows],
                                             int nvb, const float (&qv)[VLayout<D>::E], float &m,
                                             float (&u)[VLayout<D>::E], float &w, int lane)
{
    constexpr int E = VLayout<D>::E;
    float s;
    if constexpr (sizeof(Tin) == 4) {
        double x[kReduceRows];
#pragma unroll
        for (int i = 0; i < kReduceRows; ++i) {
            float kf[E];
            kr[i].get(kf);
            double acc = 0.0;
#pragma unroll
            for (int e = 0; e < E; ++e) acc = fma(double(qv[e]), double(kf[e]), acc);
            x[i] = acc;
        }
        s = static_cast<float>(transpose_sum8_t<double>(x, lane));
    } else {
        float x[kReduceRows];
#pragma unroll
        for (int i = 0; i < kReduceRows; ++i) {
            float kf[E];
            kr[i].get(kf);
            float acc = qv[0] * kf[0];
#pragma unroll
            for (int e = 1; e < E; ++e) acc = fmaf(qv[e], kf[e], acc);
            x[i] = acc;
        }
        s = transpose_sum8_t<float>(x, lane);
    }
    if ((lane & 7) >= nvb) s = -INFINITY;
    // the batch maximum (lanes hold rows lane & 7, four copies each)
    float bm = s;
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 1));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 2));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 4));
    if (bm > m) {   // warp-uniform
        const float a = (m == -INFINITY) ? 0.f : exp_rel(m, bm);
#pragma unroll
        for (int e = 0; e < E; ++e) u[e] *= a;
        w *= a;
        m = bm;
    }
    const float beta = (s == -INFINITY) ? 0.f : exp_rel(s, m);
    float bs = beta;
    bs += __shfl_xor_sync(kFull, bs, 1);
    bs += __shfl_xor_sync(kFull, bs, 2);
    bs += __shfl_xor_sync(kFull, bs, 4);
    w += bs;
#pragma unroll
    for (int i = 0; i < kReduceRows; ++i) {
        const float bi = __shfl_sync(kFull, beta, i);
        float v[E];
        vr[i].get(v);
#pragma unroll
        for (int e = 0; e < E; ++e) u[e] = fmaf(bi, v[e], u[e]);
    }
}

// x := x (+) st_0 (+) ... (+) st_{n-1} for n states of SS floats at `st`
// (written by other warps before they counted themselves in), 32 at a
// time: lane i reads state i's (m, w); every lane reads its dims of u for
// eight states per round trip.
template <int D>
__device__ __forceinline__ void fold_states(const float *st, int64_t n, float &xm,
                                            float (&xu)[VLayout<D>::E], float &xw, int lane)
{
    using L = VLayout<D>;
    constexpr int E = L::E;
    constexpr int SS = StateLayout<D>::SS;
    const bool owns = (L::LANES == 32 || lane < L::LANES);
    for (int64_t i0 = 0; i0 < n; i0 += 32) {
        const int cnt = (n - i0 < 32) ? static_cast<int>(n - i0) : 32;
        float mi = -INFINITY, wi = 0.f;
        if (lane < cnt) {
            mi = ptx::ld_relaxed(st + size_t(i0 + lane) * SS);
            wi = ptx::ld_relaxed(st + size_t(i0 + lane) * SS + 1);
        }
        const float M = fmaxf(warp_max(mi), xm);
        if (M == -INFINITY) continue;   // all identities so far
        const float ei = (mi == -INFINITY) ? 0.f : exp_rel(mi, M);
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
        for (int b0 = 0; b0 < cnt; b0 += 8) {
            float v[8][E];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
#pragma unroll
                for (int e = 0; e < E; ++e) v[b][e] = 0.f;
                if (owns && b0 + b < cnt) {
                    const float *src = st + size_t(i0 + b0 + b) * SS + 4 + lane * E;
                    if constexpr (E == 4) ptx::ld_relaxed4(src, v[b][0], v[b][1], v[b][2], v[b][3]);
                    else if constexpr (E == 2) ptx::ld_relaxed2(src, v[b][0], v[b][1]);
                    else v[b][0] = ptx::ld_relaxed(src);
                }
            }
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const float eb = __shfl_sync(kFull, ei, (b0 + b) & 31);
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = fmaf(eb, v[b][e], acc[e]);
            }
        }
        const float wsum = warp_sum(ei * wi);
        const float ex = (xm == -INFINITY) ? 0.f : exp_rel(xm, M);
#pragma unroll
        for (int e = 0; e < E; ++e) xu[e] = fmaf(ex, xu[e], acc[e]);
        xw = fmaf(ex, xw, wsum);
        xm = M;
    }
}

template <int D, typename Tin, typename Tout>
__global__ void __launch_bounds__(kReduceWarps * 32) k_scan_reduce(const ReduceParams p)
{
    using L = VLayout<D>;
    constexpr int E = L::E;
    constexpr int SS = StateLayout<D>::SS;
    using Row = RowRegs<Tin, E>;

    const int lane = threadIdx.x & 31;
    const int64_t gw = int64_t(blockIdx.x) * kReduceWarps + (threadIdx.x >> 5);
    if (gw >= p.heads * p.P) return;
    const int64_t head = gw / p.P;
    const int64_t part = gw - head * p.P;
    const bool owns = (L::LANES == 32 || lane < L::LANES);
    const int64_t r0 = part * p.seg;
    const int64_t r1 = (r0 + p.seg < p.N) ? r0 + p.seg : p.N;   // r0 may be >= r1 (empty part)
    // the part's rows of K and V, the head's q and counter, the part's slot
    // and the head's parts in the workspace (uniform per warp)
    if (!AAREN_IN_BOUNDS(p.status, in_range(head, 1, p.heads) && in_range(gw, 1, p.part_slots) &&
                                       in_range(head * p.P, p.P, p.part_slots) &&
                                       (r0 >= r1 || in_range(head * p.N + r0, r1 - r0, p.heads * p.N))))
        return;

    float qv[E];
    if (owns) {
        load_vals<E>(static_cast<const Tin *>(p.q) + head * D + lane * E, qv);
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) qv[e] = 0.f;
    }
    const Tin *Kh = static_cast<const Tin *>(p.K) + size_t(head) * p.N * D + lane * E;
    const Tin *Vh = static_cast<const Tin *>(p.V) + size_t(head) * p.N * D + lane * E;

    float m = -INFINITY, w = 0.f, u[E];
#pragma unroll
    for (int e = 0; e < E; ++e) u[e] = 0.f;

    // two register buffers of 8 rows: the next batch loads while this one reduces
    Row ka[kReduceRows], va[kReduceRows], kb[kReduceRows], vb[kReduceRows];
    auto load = [&](Row (&kk)[kReduceRows], Row (&vv)[kReduceRows], int64_t b) {
#pragma unroll
        for (int i = 0; i < kReduceRows; ++i) {
            kk[i].clear();
            vv[i].clear();
            if (owns && b + i < r1) {
                kk[i].load(Kh + size_t(b + i) * D);
                vv[i].load(Vh + size_t(b + i) * D);
            }
        }
    };
    auto valid = [&](int64_t b) -> int {
        const int64_t n = r1 - b;
        return n <= 0 ? 0 : (n >= kReduceRows ? kReduceRows : static_cast<int>(n));
    };
    if (r0 < r1) load(ka, va, r0);
    for (int64_t b = r0; b < r1; b += 2 * kReduceRows) {
        if (b + kReduceRows < r1) load(kb, vb, b + kReduceRows);
        reduce_batch<Tin, D>(ka, va, valid(b), qv, m, u, w, lane);
        if (b + 2 * kReduceRows < r1) load(ka, va, b + 2 * kReduceRows);
        if (b + kReduceRows < r1) reduce_batch<Tin, D>(kb, vb, valid(b + kReduceRows), qv, m, u, w, lane);
    }

    // this part's state to the workspace; the head's last arrival combines
    float *mine = p.parts + size_t(gw) * SS;
    write_state<D>(mine, m, u, w, lane);
    __threadfence();
    __syncwarp();
    unsigned arrived = 0;
    if (lane == 0) arrived = atomicAdd(p.counts + head, 1u);
    arrived = __shfl_sync(kFull, arrived, 0);
    if (arrived != static_cast<unsigned>(p.P - 1)) return;
    __threadfence();

    float xm = -INFINITY, xw = 0.f, xu[E];
#pragma unroll
    for (int e = 0; e < E; ++e) xu[e] = 0.f;
    if (p.m_in != nullptr) {
        xm = p.m_in[head];
        xw = p.w_in[head];
        if (owns) load_vals<E>(p.u_in + head * D + lane * E, xu);
    }
    fold_states<D>(p.parts + size_t(head) * p.P * SS, p.P, xm, xu, xw, lane);
    if (p.m_out != nullptr) {
        if (lane == 0) {
            p.m_out[head] = xm;
            p.w_out[head] = xw;
        }
        if (owns) store_vals<E>(p.u_out + head * D + lane * E, xu);
    }
    if (p.o_last != nullptr && owns) {
        const float r = __frcp_rn(xw);
        float o[E];
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = xu[e] * r;
        store_vals<E>(static_cast<Tout *>(p.o_last) + head * D + lane * E, o);
    }
}

}  // namespace aaren
