// step_kernel.cuh -- the constant-memory one-token update of many independent
// streams ("Attention as an RNN" review, "Proposed method": Aaren is updated
// with each new token in constant memory), and the identity-state fill.
//
// One warp per stream; lanes own E consecutive dims of q, k_t, v_t, u and o_t:
//   s = q . k_t  (warp reduction);  M = max(m, s);
//   u = e^{m-M} u + e^{s-M} v_t;  w = e^{m-M} w + e^{s-M};  m = M;  o_t = u / w.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"

namespace aaren {

struct StepParams {
    const void *q;
    float *m;
    float *u;
    float *w;
    const void *k;
    const void *v;
    void *o;
    int64_t n;
    unsigned *status;     // device status word (checked build)
    int64_t probe;        // testing, checked build: added to the stream index the
                          // bounds check tests (never to an address)
};

template <int D, typename Tin, typename Tout>
__global__ void __launch_bounds__(256) k_step(const StepParams p)
{
    using L = VLayout<D>;
    constexpr int E = L::E;
    // Launched as a programmatic dependent of the kernel before it in the
    // stream (usually the previous step): wait until that kernel has completed
    // and its writes are visible, then let the next step's launch begin, so
    // that launch overlaps this step's work.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int64_t i = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (i >= p.n) return;   // uniform per warp
    // every access below is row i of an [n, ...] tensor
    if (!AAREN_IN_BOUNDS(p.status, in_range(i + p.probe, 1, p.n))) return;
    const bool owns = (L::LANES == 32 || lane < L::LANES);
    const size_t off = size_t(i) * D + lane * E;

    float q[E], k[E], v[E], u[E];
    float part = 0.f;
    if (owns) {
        load_vals<E>(static_cast<const Tin *>(p.q) + off, q);
        load_vals<E>(static_cast<const Tin *>(p.k) + off, k);
        load_vals<E>(static_cast<const Tin *>(p.v) + off, v);
        load_vals<E>(p.u + off, u);
#pragma unroll
        for (int e = 0; e < E; ++e) part = fmaf(q[e], k[e], part);
    }
    const float s = warp_sum(part);
    const float m = p.m[i];
    const float w = p.w[i];
    const float M = fmaxf(m, s);
    const float alpha = exp_rel(m, M);
    const float beta = exp_rel(s, M);
    const float w2 = fmaf(alpha, w, beta);
    const float rcp = __frcp_rn(w2);
    if (owns) {
        float o[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            u[e] = fmaf(beta, v[e], alpha * u[e]);
            o[e] = u[e] * rcp;
        }
        store_vals<E>(p.u + off, u);
        store_vals<E>(static_cast<Tout *>(p.o) + off, o);
    }
    if (lane == 0) {
        p.m[i] = M;
        p.w[i] = w2;
    }
}

// Identity state (-inf, 0, 0) for n streams.
__global__ void k_state_init(float *m, float *u, float *w, int64_t n, int64_t d)
{
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n * d; i += stride) {
        u[i] = 0.f;
        if (i < n) {
            m[i] = -INFINITY;
            w[i] = 0.f;
        }
    }
}

}  // namespace aaren
