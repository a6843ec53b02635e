// linattn_kernel.cuh -- causal cos-re-weighted linear attention (cosFormer)
// on the fifth-generation tensor cores.
//
// Per head, with Q' = ReLU(Q), K' = ReLU(K) and theta = pi / (2 M):
//     o_i = sum_{j<=i} s_ij v_j / sum_{j<=i} s_ij,
//     s_ij = (Q'_i . K'_j) cos(theta (i - j))
// (LG AI Research blog "[ICLR 2022] Part 1: Efficient Transformer", section
// "cosFormer": ReLU feature maps, cos re-weighting of the position distance,
// and its split by the cosine sum formula into a cos part and a sin part that
// can be summed key-first).  Positions are 1-based and continue from pos0.
//
// Chunked form (C = 128 tokens, d = 64).  For a chunk starting after position
// t0 (state S^c, S^s [d x d], z^c, z^s [d] summed over all earlier tokens):
//     intra_i = sum_{j in chunk, j<=i} A_ij v_j,  A_ij = (Q'_i . K'_j) cos(theta (i-j))
//     inter_i = cos_i Q'_i S^c + sin_i Q'_i S^s
//     den_i   = sum_j A_ij + cos_i Q'_i . z^c + sin_i Q'_i . z^s
//     o_i     = (intra_i + inter_i) / den_i        (0 where den_i = 0)
// then S^c += sum_j (cos_j K'_j)^T v_j, S^s likewise with sin_j, z the same
// without v.  Four tensor-core products per chunk:
//     MMA1  P     = Q' K'^T                         M=128 N=128 K=64
//     MMA3  inter = Q' [S^c | S^s | z^c z^s]        M=128 N=144 K=64   (S, z as hi + lo)
//     MMA4  dS    = [cos K' | sin K']^T [V | 1]     M=128 N=80  K=128  (weighted K' as hi + lo)
//     MMA2  intra = A [V | 1]                       M=128 N=80  K=128  (A as hi + lo, in tensor memory)
// The ones column appended to V makes MMA4 also produce dz and MMA2 the
// intra-chunk row sums of A; z appended to S makes MMA3 produce Q'_i . z:
// every denominator term comes out of the same products as its numerator.
// Every rounded operand (A, the weighted keys, S, z) is carried as a
// bfloat16 pair hi + lo = x to within 2^-16 relative (hi the truncation, lo
// the rounded remainder), so products are float32-accurate; Q', K' and V are
// exact bfloat16 inputs.
//
// One persistent CTA per SM walks whole heads (h = blockIdx.x, += gridDim.x)
// chunk by chunk (g counts this CTA's chunks).  Roles:
//   warp 0, one thread   tiled TMA loads of Q, K, V (two stages)
//   warp 1, one thread   issues MMA1, then MMA3 and MMA2 in whatever order
//       their inputs arrive (one commit for both)
//   warp 2, one thread   issues MMA4 once the weighted keys are written (a
//       second issuing thread: one thread issues about one MMA per 33 ns
//       for any N up to 128)
//   two row warpgroups (warps 4-7 and 8-11, thread = token row i = TMEM
//       lane; warpgroup hf takes columns 64hf.. of P and dims 32hf.. of O):
//       ReLU of Q and K in place (half of each row each); P -> A (causal
//       mask, cos weight, hi/lo) back into tensor memory, skipping blocks the
//       mask zeroes; o_i from intra, inter and the denominators.  The ReLU of
//       the next chunk runs while MMA2 of this chunk executes.
//   key / state warpgroup (warps 12-15): as token rows, the weighted keys as
//       hi/lo; as state rows (r < 64 cos part, key dim r; r >= 64 sin part)
//       its S row (64 floats) and z entry in registers, dS and dz added after
//       each chunk, S and z published as hi/lo for the next chunk's MMA3, the
//       final state written at the end of a head.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"
#include "scan_kernel.cuh"
#include "tc.cuh"

namespace aaren {
namespace la {

constexpr int C = 128;                     // tokens per chunk
constexpr int D = 64;                      // head dimension (one 128-byte row)
constexpr int kTile = C * D * 2;           // 16 KB: one [128 x 64] bf16 tile
constexpr int kThreads = 512;
constexpr uint32_t kTmemCols = 512;

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr int OFF_STAGE = 0;                // stage s: Q, K, V at s*3*kTile + {0, 1, 2}*kTile
constexpr int OFF_KW = 2 * 3 * kTile;       // weighted K': hi cos, hi sin, lo cos, lo sin
constexpr int OFF_S = OFF_KW + 4 * kTile;   // hi [S^c | S^s | Z] 8 KB each, then lo likewise
constexpr int kSPart = 3 * 8192;
constexpr int OFF_ONES = OFF_S + 2 * kSPart;   // [128 x 64] with column 0 = 1
constexpr int OFF_W = OFF_ONES + kTile;     // W[256]: W[128 + delta] = cos(theta delta), 0 for delta < 0
constexpr int OFF_BAR = OFF_W + 256 * 4;
constexpr int kSmemBytes = OFF_BAR + 128 + 1024;   // + alignment slack

// Tensor-memory columns.
constexpr uint32_t COL_P = 0;      // P (float32), then A as hi/lo pairs: 128 columns
constexpr uint32_t COL_I = 128;    // inter: cos part +0..63, sin part +64..127, Q'.z^c, Q'.z^s at +128, +129
constexpr uint32_t COL_X = 288;    // intra: +0..63, row sum of A at +64
constexpr uint32_t COL_DS = 384;   // dS (lanes: cos rows 0-63, sin rows 64-127), dz at +64

constexpr uint32_t ID_QK = tc::idesc_bf16(128, 128, 0, 0);   // MMA1
constexpr uint32_t ID_QS = tc::idesc_bf16(128, 144, 0, 1);   // MMA3
constexpr uint32_t ID_KV = tc::idesc_bf16(128, 80, 1, 1);    // MMA4
constexpr uint32_t ID_AV = tc::idesc_bf16(128, 80, 0, 1);    // MMA2

struct Params {
    void *O;                    // [BH, N, 64] bf16 or float
    const float *S_in, *z_in;   // [BH, 2, 64, 64], [BH, 2, 64] or null (zero state)
    float *S_out, *z_out;       // same layout or null
    int64_t BH, N, pos0;
    double inv_2M;              // position * inv_2M = angle / pi
    float inv_2Mf;              // the same in single precision
    unsigned *status;
    int64_t wait_limit_ns;
    int64_t drop_chunk;         // testing: chunk (of CTA 0) whose weighted keys are never
                                // announced, so the MMA warp's wait gives up (-1 = none)
};

struct Bars {
    uint64_t full[2], empty[2];   // TMA stages (empty: both row warpgroups and the key warpgroup)
    uint64_t qk[2];               // per stage: ReLU of Q and K done (both row warpgroups): MMA1
    uint64_t kw;                  // weighted keys written: MMA4
    uint64_t sready;              // S, z published: MMA3
    uint64_t aready;              // A in tensor memory (both row warpgroups): MMA2
    uint64_t pfull, dsfull, ofull;   // MMA completion (commit)
    uint64_t tfree;               // inter / intra read (both row warpgroups)
    uint64_t drain, drain4;       // after a give-up: every MMA issued so far (by the MMA warp,
                                  // by the MMA4 warp) has completed
    uint32_t tmem;
    int abort;
};
static_assert(sizeof(Bars) <= 128, "the barriers' shared-memory slot is 128 bytes");

__device__ __forceinline__ uint32_t relu_bf16x2(uint32_t w)
{
    const uint32_t s = (w >> 15) & 0x00010001u;
    return w & ~(s * 0xFFFFu);
}

__device__ __forceinline__ uint32_t bf2_bits(float a, float b)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);   // a in the low half
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Packed float32 pairs (sm_100 family f32x2 arithmetic): .x in the low word.
__device__ __forceinline__ uint64_t f2(float a, float b)
{
    return static_cast<uint64_t>(__float_as_uint(a)) | (static_cast<uint64_t>(__float_as_uint(b)) << 32);
}

__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// pair (a, b) -> hi = the bfloat16 truncations of a and b (their top 16
// bits), lo = bf16x2(a - hi.a, b - hi.b) rounded to nearest: x = hi + lo to
// within 2^-16 relative (the remainder is below 2^-7 |x| and keeps 8 bits).
__device__ __forceinline__ void split2p(uint64_t ab, uint32_t &hi, uint32_t &lo)
{
    const uint32_t ua = static_cast<uint32_t>(ab), ub = static_cast<uint32_t>(ab >> 32);
    hi = __byte_perm(ua, ub, 0x7632);
    const uint64_t r = sub2(ab, (ab & 0xFFFF0000FFFF0000ull));
    lo = bf2_bits(__uint_as_float(static_cast<uint32_t>(r)), __uint_as_float(static_cast<uint32_t>(r >> 32)));
}

__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo)
{
    split2p(f2(a, b), hi, lo);
}

__device__ __forceinline__ bool aborted(const Bars &b) { return *reinterpret_cast<const volatile int *>(&b.abort) != 0; }

// A wait that gives up sets the CTA's abort flag; once it is set every
// further wait returns at once.  Threads never leave a chunk half-way (the
// named barriers inside a chunk would then wait for them forever): they run
// the rest of the chunk without waiting, and each warpgroup leaves its loop
// together at the next chunk boundary (stop_all).
__device__ __forceinline__ bool la_wait(Bars &b, uint64_t *bar, unsigned parity, const Params &p)
{
    if (aborted(b)) return false;
    if (wait_bar(bar, parity, p.wait_limit_ns)) return true;
    atomicOr(p.status, STATUS_LOAD_TIMEOUT);
    *reinterpret_cast<volatile int *>(&b.abort) = 1;
    return false;
}

// True in every thread of the named barrier's group if it is true in any.
__device__ __forceinline__ bool stop_all(unsigned id, bool pred)
{
    unsigned r;
    asm volatile("{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\n"
                 "barrier.red.or.pred q, %2, 128, p;\nselp.u32 %0, 1, 0, q;\n}\n"
                 : "=r"(r) : "r"(static_cast<unsigned>(pred)), "r"(id) : "memory");
    return r != 0;
}

// 32 consecutive outputs of one row (16-byte stores).
__device__ __forceinline__ void store_row32(float *dst, const float (&o)[32])
{
#pragma unroll
    for (int t = 0; t < 32; t += 4)
        *reinterpret_cast<float4 *>(dst + t) = make_float4(o[t], o[t + 1], o[t + 2], o[t + 3]);
}

__device__ __forceinline__ void store_row32(__nv_bfloat16 *dst, const float (&o)[32])
{
#pragma unroll
    for (int t = 0; t < 32; t += 8)
        *reinterpret_cast<uint4 *>(dst + t) =
            make_uint4(bf2_bits(o[t], o[t + 1]), bf2_bits(o[t + 2], o[t + 3]), bf2_bits(o[t + 4], o[t + 5]),
                       bf2_bits(o[t + 6], o[t + 7]));
}

// (cos, sin) of the angle of 1-based position pos: pi/2 * pos / M, with
// inv_2Mf = 1 / (2M) in single precision.  The argument carries at most three
// units in the last place of relative error (the conversion of pos, exact
// below 2^24, inv_2Mf and the product) against one when the product is taken
// in double precision and rounded; either way it is then a float.  The empty
// asm keeps the computation where it is called, off the path that first
// reads the values.
__device__ __forceinline__ void pos_angle(int64_t pos, float inv_2Mf, float &cs, float &sn)
{
    sincospif(static_cast<float>(pos) * inv_2Mf, &sn, &cs);
    asm volatile("" : "+f"(cs), "+f"(sn));
}

// ReLU of half of one 128-byte row (row index r, half hf: slots visited 4hf
// .. 4hf+3) in place.  The 16-byte slots are visited in the order slot = ch ^
// (r % 8), so the eight rows a quarter-warp touches at a time sit in eight
// different bank groups.
__device__ __forceinline__ void relu_half_row(uint8_t *row, int r, int hf)
{
#pragma unroll
    for (int ch = 4 * hf; ch < 4 * hf + 4; ++ch) {
        uint4 *slot = reinterpret_cast<uint4 *>(row) + (ch ^ (r & 7));
        uint4 x = *slot;
        x.x = relu_bf16x2(x.x); x.y = relu_bf16x2(x.y); x.z = relu_bf16x2(x.z); x.w = relu_bf16x2(x.w);
        *slot = x;
    }
}

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
k_linattn(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
          const __grid_constant__ CUtensorMap tv, const Params p)
{
    extern __shared__ uint8_t la_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(la_raw) + 1023) & ~uintptr_t(1023));
    Bars &b = *reinterpret_cast<Bars *>(sm + OFF_BAR);
    const float *Wt = reinterpret_cast<const float *>(sm + OFF_W);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t nc = (p.N + C - 1) / C;
    const int64_t my_heads = (p.BH - blockIdx.x + gridDim.x - 1) / gridDim.x;
    const int64_t total = my_heads * nc;   // chunks of this CTA

    if (tid == 0) {
        ptx::mbar_init(&b.full[0], 1); ptx::mbar_init(&b.full[1], 1);
        ptx::mbar_init(&b.empty[0], 3); ptx::mbar_init(&b.empty[1], 3);
        ptx::mbar_init(&b.qk[0], 2); ptx::mbar_init(&b.qk[1], 2);
        ptx::mbar_init(&b.kw, 1); ptx::mbar_init(&b.sready, 1); ptx::mbar_init(&b.aready, 2);
        ptx::mbar_init(&b.pfull, 1); ptx::mbar_init(&b.dsfull, 1); ptx::mbar_init(&b.ofull, 1);
        ptx::mbar_init(&b.tfree, 2);
        ptx::mbar_init(&b.drain, 1); ptx::mbar_init(&b.drain4, 1);
        b.abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0) tc::tmem_alloc(&b.tmem, kTmemCols);
    // constant operand pieces: the ones column, the zero padding of the z blocks, the weight table
    for (int x = tid; x < kTile / 16; x += kThreads) {
        const int row = x >> 3, ch = x & 7;   // physical 16-byte slot ch of row
        const uint32_t one = (ch == (row & 7)) ? 0x3F80u : 0u;   // logical chunk 0 holds column 0
        reinterpret_cast<uint4 *>(sm + OFF_ONES)[x] = make_uint4(one, 0u, 0u, 0u);
    }
    for (int x = tid; x < 8192 / 16; x += kThreads) {
        reinterpret_cast<uint4 *>(sm + OFF_S + 2 * 8192)[x] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4 *>(sm + OFF_S + kSPart + 2 * 8192)[x] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (tid < 256) {
        float *Ww = reinterpret_cast<float *>(sm + OFF_W);
        Ww[tid] = tid >= C ? static_cast<float>(cospi(static_cast<double>(tid - C) * p.inv_2M)) : 0.f;
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = b.tmem;

    if (warp == 0) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int64_t g = 0;
            for (; g < total; ++g) {
                const int s = static_cast<int>(g & 1);
                if (!la_wait(b, &b.empty[s], static_cast<unsigned>(((g >> 1) & 1) ^ 1), p)) break;
                const int64_t h = blockIdx.x + (g / nc) * gridDim.x, c = g % nc;
                uint8_t *st = sm + OFF_STAGE + s * 3 * kTile;
                const int y = static_cast<int>(c * C), z = static_cast<int>(h);
                // the tile's first row and its head lie inside the tensors
                if (AAREN_IN_BOUNDS(p.status, in_range(h, 1, p.BH) && in_range(c * C, 1, p.N))) {
                    ptx::mbar_arrive_expect_tx(&b.full[s], 3 * kTile);
                    tc::tma_load_3d(st, &tq, 0, y, z, &b.full[s]);
                    tc::tma_load_3d(st + kTile, &tk, 0, y, z, &b.full[s]);
                    tc::tma_load_3d(st + 2 * kTile, &tv, 0, y, z, &b.full[s]);
                } else {
                    ptx::mbar_arrive(&b.full[s]);   // no copy: the fill completes at once
                }
            }
            // let copies still in flight land before the CTA can exit
            for (int64_t k = g - 2 > 0 ? g - 2 : 0; k < g; ++k)
                wait_bar(&b.full[k & 1], static_cast<unsigned>((k >> 1) & 1), p.wait_limit_ns);
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------- MMA issue: warp 1 MMA1, MMA3, MMA2; warp 2 MMA4 ----------------
        // Two issuing threads: one thread issues an MMA about every 33 ns for
        // any N up to 128 (M = 128, K = 16), and MMA4 (the state update) and
        // MMA2 (intra) are both narrow (N = 80), so together they keep the
        // tensor pipe busier.
        // Descriptors of each operand's first K step are built once.  A step
        // of `off` bytes adds off >> 4 to the descriptor's start-address
        // field, which never carries out of it: every shared address here is
        // below 256 KB, so (address >> 4) stays below 2^14.  The products are
        // fully unrolled, so issuing one MMA costs an add and the instruction.
        const uint32_t ones = tc::saddr(sm + OFF_ONES);
        uint64_t dq[2], dk[2], dv[2];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const uint32_t q0 = tc::saddr(sm + OFF_STAGE + s * 3 * kTile);
            dq[s] = tc::sdesc(q0, 16, 1024);
            dk[s] = tc::sdesc(q0 + kTile, 16, 1024);
            dv[s] = tc::sdesc(q0 + 2 * kTile, ones - (q0 + 2 * kTile), 1024);
        }
        if (warp == 2 && lane == 0) {
            // MMA4: dS of chunk g once its weighted keys are written (which
            // the key warpgroup does only after reading the previous dS)
            const uint64_t dkw = tc::sdesc(tc::saddr(sm + OFF_KW), kTile, 1024);
            bool issued = false;
            for (int64_t g = 0; g < total; ++g) {
                const uint64_t bv = (g & 1) ? dv[1] : dv[0];
                if (!la_wait(b, &b.kw, static_cast<unsigned>(g & 1), p)) break;
                tc::fence_after();
#pragma unroll
                for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_ss(tmem + COL_DS, dkw + ((hl * 2 * kTile + kk * 2048) >> 4), bv + 128 * kk, ID_KV,
                                   hl > 0 || kk > 0);
                tc::commit(&b.dsfull);
                issued = true;
            }
            // gave up: let this thread's MMAs finish before tensor memory is freed
            if (aborted(b) && issued) {
                tc::commit(&b.drain4);
                wait_bar(&b.drain4, 0, p.wait_limit_ns);
            }
        } else if (warp == 1 && lane == 0) {
            const uint64_t dsz = tc::sdesc(tc::saddr(sm + OFF_S), 8192, 1024);
            const uint64_t *last = nullptr;   // the latest commit (null: no MMA issued yet)
            for (int64_t g = 0; g < total; ++g) {
                const int s = static_cast<int>(g & 1);
                const unsigned par = static_cast<unsigned>(g & 1), prev = par ^ 1u;
                const uint64_t aq = s ? dq[1] : dq[0], ak = s ? dk[1] : dk[0], bv = s ? dv[1] : dv[0];
                la_wait(b, &b.qk[s], static_cast<unsigned>((g >> 1) & 1), p);
                if (g > 0) la_wait(b, &b.ofull, prev, p);   // MMA2 of the previous chunk has read A
                if (aborted(b)) break;
                tc::fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_ss(tmem + COL_P, aq + 2 * kk, ak + 2 * kk, ID_QK, kk > 0);
                tc::commit(&b.pfull);
                last = &b.pfull;
                // MMA3 (inter) and MMA2 (intra) as their operands come ready,
                // in whatever order that is; one output commit covers both
                bool d3 = false, d2 = false, dO = false, tf = (g == 0), timed_out = false;
                const uint64_t t_start = ptx::globaltimer();
                for (unsigned polls = 0; !dO; ++polls) {
                    bool any = false;
                    if (!tf) tf = ptx::mbar_test_wait(&b.tfree, prev);   // inter / intra of the previous chunk read
                    if (tf && !d3 && ptx::mbar_test_wait(&b.sready, par)) {
                        tc::fence_after();
#pragma unroll
                        for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc::mma_ss(tmem + COL_I, aq + 2 * kk, dsz + ((hl * kSPart + kk * 2048) >> 4), ID_QS,
                                           hl > 0 || kk > 0);
                        d3 = any = true;
                    }
                    if (tf && !d2 && ptx::mbar_test_wait(&b.aready, par)) {
                        tc::fence_after();
#pragma unroll
                        for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk)
                                tc::mma_ts(tmem + COL_X, tmem + COL_P + 32 * (kk >> 1) + 16 * hl + 8 * (kk & 1),
                                           bv + 128 * kk, ID_AV, hl > 0 || kk > 0);
                        d2 = any = true;
                    }
                    if (d2 && d3 && !dO) {   // exactly one output commit per chunk
                        tc::commit(&b.ofull);
                        last = &b.ofull;
                        dO = true;
                    }
                    if (!any) {
                        if (aborted(b) ||
                            (polls >= kMinWaitPolls && int64_t(ptx::globaltimer() - t_start) > p.wait_limit_ns)) {
                            timed_out = true;
                            break;
                        }
                        __nanosleep(32);
                    }
                }
                if (timed_out) {
                    atomicOr(p.status, STATUS_LOAD_TIMEOUT);
                    *reinterpret_cast<volatile int *>(&b.abort) = 1;
                    break;
                }
            }
            // gave up: let every MMA still in flight finish before tensor
            // memory is freed.  A commit covers all earlier MMAs of this
            // thread, including any issued after the last per-chunk commit
            // (a give-up inside the poll loop can leave MMA3 or MMA2 without one).
            if (aborted(b) && last != nullptr) {
                tc::commit(&b.drain);
                wait_bar(&b.drain, 0, p.wait_limit_ns);
            }
        }
    } else if (warp >= 4 && warp < 12) {
        // ---------------- row warpgroups: token rows, half hf of the columns each ----------------
        const int hf = (warp - 4) >> 2;                           // 0: warps 4-7, 1: warps 8-11
        const unsigned nb = 1 + hf;                               // named barrier of this warpgroup
        const int i = (warp & 3) * 32 + lane;                     // token row = TMEM lane
        const bool leader = (warp & 3) == 0 && lane == 0;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        if (total > 0) {
            la_wait(b, &b.full[0], 0, p);
            relu_half_row(sm + OFF_STAGE + i * 128, i, hf);
            relu_half_row(sm + OFF_STAGE + kTile + i * 128, i, hf);
            tc::fence_async_smem();
            ptx::named_bar_sync(nb, 128);
            if (leader) ptx::mbar_arrive(&b.qk[0]);
        }
        int64_t h = blockIdx.x, c = 0;   // head and chunk of chunk g
        for (int64_t g = 0; g < total; ++g) {
            if (stop_all(nb, aborted(b))) break;
            const int s = static_cast<int>(g & 1);
            const unsigned par = static_cast<unsigned>(g & 1);
            float cs, sn;
            pos_angle(p.pos0 + c * C + i + 1, p.inv_2Mf, cs, sn);

            // ---- P -> A on columns 64 hf .. 64 hf + 63: causal mask and cos weight, hi/lo ----
            la_wait(b, &b.pfull, par, p);
            tc::fence_after();
            __syncwarp();
            const float *wrow = Wt + C + i;   // wrow[-j] = weight of column j (0 for j > i)
#pragma unroll 1
            for (int qb = 2 * hf; qb < 2 * hf + 2; ++qb) {
                uint32_t wv[32];
                if (qb > (warp & 3)) {         // every row of this warp is above the block: A = 0
#pragma unroll
                    for (int t = 0; t < 32; ++t) wv[t] = 0u;
                } else {
                    uint32_t pc[32];
                    tc::ld32_async(tmem + lane_base + COL_P + 32 * qb, pc);
                    tc::wait_ld();
#pragma unroll
                    for (int t = 0; t < 32; t += 2) {
                        const int j = 32 * qb + t;
                        const uint64_t pp = static_cast<uint64_t>(pc[t]) | (static_cast<uint64_t>(pc[t + 1]) << 32);
                        split2p(mul2(pp, f2(wrow[-j], wrow[-j - 1])), wv[t >> 1], wv[16 + (t >> 1)]);
                    }
                }
                tc::st32(tmem + lane_base + COL_P + 32 * qb, wv);
            }
            tc::wait_st();
            tc::fence_before();
            ptx::named_bar_sync(nb, 128);
            if (leader) ptx::mbar_arrive(&b.aready);

            // ---- ReLU of the next chunk's Q and K (this half of each row) while MMA2 runs ----
            if (g + 1 < total) {
                const int s1 = static_cast<int>((g + 1) & 1);
                la_wait(b, &b.full[s1], static_cast<unsigned>(((g + 1) >> 1) & 1), p);
                uint8_t *st1 = sm + OFF_STAGE + s1 * 3 * kTile;
                relu_half_row(st1 + i * 128, i, hf);
                relu_half_row(st1 + kTile + i * 128, i, hf);
                tc::fence_async_smem();
                ptx::named_bar_sync(nb, 128);
                if (leader) ptx::mbar_arrive(&b.qk[s1]);
            }

            // ---- o_i on dims 32 hf .. 32 hf + 31:
            //      (intra + cos inter_c + sin inter_s) / (den_intra + cos Q'.z^c + sin Q'.z^s) ----
            la_wait(b, &b.ofull, par, p);
            tc::fence_after();
            __syncwarp();
            {
                const int b0 = 32 * hf;
                uint32_t x[32], ic[32], is[32], d0, d1, z0, z1;
                tc::ld32_async(tmem + lane_base + COL_X + b0, x);
                tc::ld32_async(tmem + lane_base + COL_I + b0, ic);
                tc::ld32_async(tmem + lane_base + COL_I + 64 + b0, is);
                tc::ld2_async(tmem + lane_base + COL_X + 64, d0, d1);
                tc::ld2_async(tmem + lane_base + COL_I + 128, z0, z1);
                tc::wait_ld();
                const float dt = __uint_as_float(d0) + cs * __uint_as_float(z0) + sn * __uint_as_float(z1);
                const float r = dt != 0.f ? __frcp_rn(dt) : 0.f;   // correctly rounded, as 1 / dt
                float o[32];
#pragma unroll
                for (int t = 0; t < 32; ++t)
                    o[t] = (__uint_as_float(x[t]) + cs * __uint_as_float(ic[t]) + sn * __uint_as_float(is[t])) * r;
                const int64_t row = c * C + i;
                if (row < p.N && AAREN_IN_BOUNDS(p.status, in_range(h * p.N + row, 1, p.BH * p.N)))
                    store_row32(reinterpret_cast<Tout *>(p.O) + (h * p.N + row) * D + b0, o);
            }
            tc::fence_before();
            ptx::named_bar_sync(nb, 128);
            if (leader) {
                ptx::mbar_arrive(&b.tfree);
                ptx::mbar_arrive(&b.empty[s]);
            }
            if (++c == nc) {
                c = 0;
                h += gridDim.x;
            }
        }
    } else if (warp >= 12) {
        // ---------------- key / state warpgroup ----------------
        const int r = tid - 384;                 // token row (key work) and state row (dS lane)
        const int half = r >> 6, k = r & 63;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        uint8_t *kw = sm + OFF_KW;
        uint8_t *Sh = sm + OFF_S + half * 8192;   // this row's block (cos or sin part), hi
        uint8_t *Zh = sm + OFF_S + 2 * 8192;      // z block, hi (column 0 = z^c, 1 = z^s)
        float S[64];
        float z = 0.f;
        // the state a head starts from: the caller's, or zero
        auto load_start = [&](int64_t h) {
            if (p.S_in != nullptr && AAREN_IN_BOUNDS(p.status, in_range(h, 1, p.BH))) {
                const float4 *src = reinterpret_cast<const float4 *>(p.S_in + ((h * 2 + half) * 64 + k) * 64);
#pragma unroll
                for (int q4 = 0; q4 < 16; ++q4) {
                    const float4 v = src[q4];
                    S[4 * q4] = v.x; S[4 * q4 + 1] = v.y; S[4 * q4 + 2] = v.z; S[4 * q4 + 3] = v.w;
                }
                z = p.z_in[(h * 2 + half) * 64 + k];
            } else {
#pragma unroll
                for (int t = 0; t < 64; ++t) S[t] = 0.f;
                z = 0.f;
            }
        };
        // S and z of the next chunk's start as hi/lo (the B operand of MMA3)
        auto publish_state = [&]() {
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split2(S[8 * ch + 2 * e], S[8 * ch + 2 * e + 1], hw[e], lw[e]);
                const int off = k * 128 + ((ch ^ (k & 7)) << 4);
                *reinterpret_cast<uint4 *>(Sh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4 *>(Sh + kSPart + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            const __nv_bfloat16 zh = __float2bfloat16_rn(z);
            const __nv_bfloat16 zl = __float2bfloat16_rn(z - __bfloat162float(zh));
            const int off = k * 128 + ((k & 7) << 4) + half * 2;   // row k, column half
            *reinterpret_cast<__nv_bfloat16 *>(Zh + off) = zh;
            *reinterpret_cast<__nv_bfloat16 *>(Zh + kSPart + off) = zl;
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(3, 128);
            if (r == 0) ptx::mbar_arrive(&b.sready);
        };
        if (total > 0) {
            load_start(blockIdx.x);
            publish_state();   // the first chunk's state
        }
        // head and chunk of chunk g, and the angle of this thread's token row
        // in it (the next chunk's is computed while MMA4 runs)
        int64_t h = blockIdx.x, c = 0;
        float cs, sn;
        pos_angle(p.pos0 + r + 1, p.inv_2Mf, cs, sn);
        for (int64_t g = 0; g < total; ++g) {
            if (stop_all(3, aborted(b))) break;
            const int s = static_cast<int>(g & 1);
            const unsigned par = static_cast<unsigned>(g & 1);

            // ---- keys (ReLU'd by the row warpgroups): cos / sin weighted as hi/lo (MMA4);
            //      the previous chunk's MMA4 is done with the buffer (dsfull waited below) ----
            la_wait(b, &b.qk[s], static_cast<unsigned>((g >> 1) & 1), p);
            {
                const uint8_t *krow = sm + OFF_STAGE + s * 3 * kTile + kTile + r * 128;
                const uint64_t c2 = f2(cs, cs), s2 = f2(sn, sn);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const int slot = ch ^ (r & 7);   // conflict-free order, as in relu_half_row
                    const uint4 kx = reinterpret_cast<const uint4 *>(krow)[slot];
                    const uint32_t w4[4] = {kx.x, kx.y, kx.z, kx.w};
                    uint32_t hc[4], lc[4], hs[4], ls[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint64_t x = f2(bf_lo(w4[e]), bf_hi(w4[e]));
                        split2p(mul2(x, c2), hc[e], lc[e]);
                        split2p(mul2(x, s2), hs[e], ls[e]);
                    }
                    const int off = r * 128 + slot * 16;   // same physical slot: same swizzle
                    *reinterpret_cast<uint4 *>(kw + 0 * kTile + off) = make_uint4(hc[0], hc[1], hc[2], hc[3]);
                    *reinterpret_cast<uint4 *>(kw + 1 * kTile + off) = make_uint4(hs[0], hs[1], hs[2], hs[3]);
                    *reinterpret_cast<uint4 *>(kw + 2 * kTile + off) = make_uint4(lc[0], lc[1], lc[2], lc[3]);
                    *reinterpret_cast<uint4 *>(kw + 3 * kTile + off) = make_uint4(ls[0], ls[1], ls[2], ls[3]);
                }
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(3, 128);
            if (r == 0 && !(blockIdx.x == 0 && g == p.drop_chunk)) ptx::mbar_arrive(&b.kw);
            const bool head_end = c == nc - 1;
            {
                const int64_t pos1 = head_end ? 0 : (c + 1) * C;
                pos_angle(p.pos0 + pos1 + r + 1, p.inv_2Mf, cs, sn);   // the next chunk's angle
            }

            // ---- dS, dz of this chunk; then the stage is no longer read here or by MMA4 ----
            la_wait(b, &b.dsfull, par, p);
            tc::fence_after();
            __syncwarp();
            {
                uint32_t dv[32], dz, dz1;
                tc::ld32_async(tmem + lane_base + COL_DS, dv);
                tc::ld2_async(tmem + lane_base + COL_DS + 64, dz, dz1);
                tc::wait_ld();
#pragma unroll
                for (int t = 0; t < 32; ++t) S[t] += __uint_as_float(dv[t]);
                z += __uint_as_float(dz);
                tc::ld32_async(tmem + lane_base + COL_DS + 32, dv);
                tc::wait_ld();
#pragma unroll
                for (int t = 0; t < 32; ++t) S[32 + t] += __uint_as_float(dv[t]);
            }
            if (r == 0) ptx::mbar_arrive(&b.empty[s]);
            if (head_end) {   // end of a head: its final state, then the next head's start
                if (p.S_out != nullptr && !aborted(b) && AAREN_IN_BOUNDS(p.status, in_range(h, 1, p.BH))) {
                    float4 *dst = reinterpret_cast<float4 *>(p.S_out + ((h * 2 + half) * 64 + k) * 64);
#pragma unroll
                    for (int q4 = 0; q4 < 16; ++q4)
                        dst[q4] = make_float4(S[4 * q4], S[4 * q4 + 1], S[4 * q4 + 2], S[4 * q4 + 3]);
                    p.z_out[(h * 2 + half) * 64 + k] = z;
                }
                if (g + 1 < total) load_start(h + gridDim.x);
            }

            // ---- the next chunk's state, once MMA3 of this chunk has read the buffer ----
            if (g + 1 < total) {
                la_wait(b, &b.ofull, par, p);
                publish_state();
            }
            if (head_end) {
                c = 0;
                h += gridDim.x;
            } else {
                ++c;
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc::fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace la
}  // namespace aaren
