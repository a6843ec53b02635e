// common.cuh -- element loads/stores, warp reductions and the associative
// state operator shared by the scan and step kernels.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace aaren {

constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

// Bits of the per-device status word (reported by aaren_check).
enum : unsigned { STATUS_LOOKBACK_TIMEOUT = 1u, STATUS_LOAD_TIMEOUT = 2u, STATUS_BOUNDS = 4u };

// Checked build.  Compiled with -DAAREN_CHECKED, every kernel tests each
// extent it computes (rows of a global tensor, a workspace slot, a bulk copy,
// a shared-memory stage) against its buffer before the access; a violation
// ORs STATUS_BOUNDS into the device status word (reported by aaren_check as
// AAREN_ERR_BOUNDS) and the access is skipped.  In the regular build
// AAREN_IN_BOUNDS is the constant true and the tested expression is never
// evaluated, so the regular kernels carry none of it.
#ifdef AAREN_CHECKED
#define AAREN_IN_BOUNDS(status, cond) (::aaren::bounds_ok((status), (cond)))
#else
#define AAREN_IN_BOUNDS(status, cond) (true)
#endif

__device__ __forceinline__ bool bounds_ok(unsigned *status, bool ok)
{
    if (!ok) atomicOr(status, STATUS_BOUNDS);
    return ok;
}

// [first, first + count) lies inside [0, extent).
__device__ __forceinline__ bool in_range(int64_t first, int64_t count, int64_t extent)
{
    return first >= 0 && count >= 0 && first <= extent && count <= extent - first;
}

// How value dimensions are spread over a warp: LANES lanes own E consecutive
// dims each (d = 16 leaves lanes 16..31 without dims).
template <int D>
struct VLayout {
    static constexpr int LANES = D < 32 ? D : 32;
    static constexpr int E = D / LANES;
    static_assert(E == 1 || E == 2 || E == 4, "d must be 16, 32, 64 or 128");
};

__device__ __forceinline__ void bf16x2_to_f32(unsigned x, float &lo, float &hi)
{
    lo = __uint_as_float(x << 16);          // element at the lower address
    hi = __uint_as_float(x & 0xffff0000u);
}

__device__ __forceinline__ unsigned f32x2_to_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // round to nearest even
    return *reinterpret_cast<unsigned *>(&h);
}

// Packed float32 pairs for the sm_100 family's two-wide float32 FMA and
// multiply (one instruction for two lanes' worth of work): .x in the low
// word.  Rounding is that of the scalar fmaf / multiply, element by element.
__device__ __forceinline__ uint64_t pack2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(uint64_t x, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
}

__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Two bfloat16 products accumulated in float32 with the sm_100 family's
// mixed-precision FMA: lo += a.lo * b.lo, hi += a.hi * b.hi for bfloat16 pairs
// a, b (the element at the lower address in the low half).  A product of two
// bfloat16 values is exact in float32, so each step rounds once, as fmaf
// on the widened values would.
__device__ __forceinline__ void fma_bf16x2(float &lo, float &hi, unsigned a, unsigned b)
{
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\t"
        "mov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.bf16 %1, ah, bh, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(a), "r"(b));
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// E consecutive elements starting at p (p aligned to E elements).
template <int E>
__device__ __forceinline__ void load_vals(const float *p, float (&f)[E])
{
    if constexpr (E == 4) {
        float4 v = *reinterpret_cast<const float4 *>(p);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    } else if constexpr (E == 2) {
        float2 v = *reinterpret_cast<const float2 *>(p);
        f[0] = v.x; f[1] = v.y;
    } else {
        f[0] = *p;
    }
}

template <int E>
__device__ __forceinline__ void load_vals(const __nv_bfloat16 *p, float (&f)[E])
{
    if constexpr (E == 4) {
        uint2 v = *reinterpret_cast<const uint2 *>(p);
        bf16x2_to_f32(v.x, f[0], f[1]);
        bf16x2_to_f32(v.y, f[2], f[3]);
    } else if constexpr (E == 2) {
        unsigned v = *reinterpret_cast<const unsigned *>(p);
        bf16x2_to_f32(v, f[0], f[1]);
    } else {
        unsigned short v = *reinterpret_cast<const unsigned short *>(p);
        f[0] = __uint_as_float(static_cast<unsigned>(v) << 16);
    }
}

template <int E>
__device__ __forceinline__ void store_vals(float *p, const float (&f)[E])
{
    if constexpr (E == 4) {
        *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
    } else if constexpr (E == 2) {
        *reinterpret_cast<float2 *>(p) = make_float2(f[0], f[1]);
    } else {
        *p = f[0];
    }
}

template <int E>
__device__ __forceinline__ void store_vals(__nv_bfloat16 *p, const float (&f)[E])
{
    if constexpr (E == 4) {
        *reinterpret_cast<uint2 *>(p) =
            make_uint2(f32x2_to_bf16x2(f[0], f[1]), f32x2_to_bf16x2(f[2], f[3]));
    } else if constexpr (E == 2) {
        *reinterpret_cast<unsigned *>(p) = f32x2_to_bf16x2(f[0], f[1]);
    } else {
        *p = __float2bfloat16_rn(f[0]);
    }
}

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, off));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
    return x;
}

// e^{x - ref} for x <= ref, exactly 1 when x == ref and 0 when x is -inf.
__device__ __forceinline__ float exp_rel(float x, float ref)
{
    return (x == ref) ? 1.0f : exp2f((x - ref) * kLog2e);
}

// The associative operator on states, lane-parallel over the lane's E dims:
//   b := a (+) b = (M, e^{m_a-M} u_a + e^{m_b-M} u_b, e^{m_a-M} w_a + e^{m_b-M} w_b),
//   M = max(m_a, m_b).  Two identities (-inf, 0, 0) give the identity.
template <int E>
__device__ __forceinline__ void combine_into(float ma, const float (&ua)[E], float wa, float &mb,
                                             float (&ub)[E], float &wb)
{
    const float M = fmaxf(ma, mb);
    if (M == -INFINITY) return;
    const float ea = exp_rel(ma, M);
    const float eb = exp_rel(mb, M);
#pragma unroll
    for (int e = 0; e < E; ++e) ub[e] = fmaf(ea, ua[e], eb * ub[e]);
    wb = fmaf(ea, wa, eb * wb);
    mb = M;
}

}  // namespace aaren
